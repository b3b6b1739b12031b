"""Counts of what the GPU parity tests compared, printed as one summary line at
the end of a pytest run: tokens compared, near-tie divergences (oracle
decision margin below 1e-3, allowed and counted), trees compared exactly or up
to a near tie, and the largest logit error seen per path."""
from __future__ import annotations

from collections import defaultdict

_counts = defaultdict(int)
_max_abs = defaultdict(float)


def tokens(compared: int, near_ties: int) -> None:
    _counts["tokens"] += int(compared)
    _counts["token_near_ties"] += int(near_ties)


def trees(exact: int, near_tie: int) -> None:
    _counts["trees_exact"] += int(exact)
    _counts["trees_near_tie"] += int(near_tie)


def count(name: str, n: int) -> None:
    _counts[name] += int(n)


def logits(path: str, err: float) -> None:
    _max_abs[path] = max(_max_abs[path], float(err))


def summary() -> str | None:
    if not _counts and not _max_abs:
        return None
    parts = [f"{k} {v}" for k, v in sorted(_counts.items())]
    parts += [f"max|dL| {k} {v:.2e}" for k, v in sorted(_max_abs.items())]
    return "parity: " + ", ".join(parts)
