"""CPU oracle for the SMC-SD per-step particle update.  TEST INFRASTRUCTURE.

This package is a plain, slow, fp64 restatement of what the hot path computes,
written from the pages that describe the method.  It exists only to check the
CUDA path: the tests under ``tests/``, the ``smoke()`` self-check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it;
nothing in the product path does, and the product fails loudly rather than fall
back to it.  It shares no code, constants or generators with the CUDA path.

Modules:
  philox  Philox4x32-10 and the step's uniforms
  smc     row log-sum-exp, gather, weight increment, bonus token, ESS,
          systematic resampling, token emission (the whole step)
  kv      block-table remap by ancestors and token append with copy-on-write
  sps     single-particle speculative-sampling verify

Pins (tests marked ``not gpu``) tie each function to something other than
itself: published Philox known-answer vectors and an independent library
implementation; scipy's logsumexp; closed forms (draft == target gives zero
weight increments and ESS = N); brute-force enumeration of the SpS output law
(Theorem 1) and of the SMC target on a small bigram model, including the
power-sampling target p^alpha; invariants of systematic resampling and of
reference counting; a shadow KV store that replays copy-on-write pairs.
Parity pinned only by internal consistency: the specific free-stack order and
which particle keeps a shared partial tail block (both are choices the pages
leave open; the invariants pin that the choice is valid, not which one).
"""
from . import philox, smc, kv, sps, errors  # noqa: F401
from .errors import OracleError  # noqa: F401
