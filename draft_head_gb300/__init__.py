"""GB300-native (sm_103a) Domino drafting hot path.

The compute path is the C-ABI CUDA library libdomino (include/domino.h);
`draft_head_gb300.binding` is its thin ctypes binding and
`draft_head_gb300.synth` draws the seeded synthetic inputs. The binding is
imported lazily so that the input generator works without a built library.
"""
__all__ = ["binding", "synth", "build"]
