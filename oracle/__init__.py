"""CPU oracle for the Domino drafting hot path (test infrastructure only).

Only tests/, the smoke check and the benchmark's CPU-baseline leg import this
package; the product path never does."""
from .domino_oracle import *  # noqa: F401,F403
