"""CPU oracle for Speculative Pipeline Decoding -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp32 numpy implementation of what the CUDA path computes:
ordinary greedy autoregressive decoding of the target decoder
(``oracle.model``) and the SPD cycle with its anchor tables, depth staircase,
draft module, streaming verification and three-step rollback
(``oracle.spd``).  It shares no code with the CUDA path; both take their inputs
from ``spd_inputs``.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
``--impl reference`` legs may import this package.  Nothing in the library
(``speculative_pipeline_decoding_gb300``) imports or calls it.

Parity status: every function is pinned by tests under ``tests/`` that do not
restate it (library routines, closed forms, special cases, brute force).  The
draft module's numerics are pinned only as far as its pieces are (the shared
decoder layer, the FC special case, incremental == full recompute); there are
no trained weights to check its predictions against.
"""
from . import model, spd  # noqa: F401
