"""The checked build (libdomino_checked.so: the same kernels compiled with
device-side index checks that report DOMINO_ERR_INDEX instead of touching
memory out of range) gives the regular library's results bit for bit and a
clean status on small chain, batched-chain, tree, statistics-chain and
head-form verification cases."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_matches_and_reports_no_index_error():
    from draft_head_gb300 import build as bld
    if not os.path.exists(bld.LIB_CHECKED):
        bld.build(checked=True)
    env = dict(os.environ, DOMINO_LIB="checked")
    r = subprocess.run([sys.executable, "-m", "tests.checked_cases"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    checked = json.loads(r.stdout.strip().splitlines()[-1])
    from tests.checked_cases import run
    regular = run()
    for key in regular:
        if key.startswith("status"):
            assert checked[key] == 0, f"{key}: checked build reported {checked[key]}"
            assert regular[key] == 0
        else:
            assert checked[key] == regular[key], key
    torch.cuda.synchronize()
