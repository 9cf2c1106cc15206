"""Large-sample parity tallies at the serving vocabulary (V = 128256, bf16).

The step's contract for integer outputs: identical to the CPU oracle except
on draws the oracle flags as near ties (the drawn point within 1e-5 of a
cumulative boundary, as a fraction of the total), and such mismatches under
1e-4 of the draws.  A rate of 1e-4 can only be seen over many draws, so each
test here makes at least MIN_DRAWS draws of every kind it covers, on the
serving workload's logits, and asserts for each kind

  * no mismatch outside a flagged near tie (the harness fails on any), and
  * mismatches <= 1e-4 x draws.

Kinds: bonus tokens, resampling ancestors and decisions (the SMC step);
acceptance tests, residual draws and bonus draws (speculative sampling);
draft-sampler draws; and bonus draws inside a top-p nucleus.  The oracle runs
in a spawned process pool (tests/oracle_pool.py), one prompt slice a task.
Each test prints one TALLY line; ``SMCSD_TALLY_LOG`` names a file that also
receives them.
"""
import json
import os

import numpy as np
import pytest
import torch

import smc_speculative_decoding_gb300 as smcsd
from smc_speculative_decoding_gb300.workloads import (WORKLOADS, make_step_inputs,
                                                      to_numpy_logits)

import oracle_pool
from gpu_harness import MISMATCH_RATE, NEAR_TIE, Tally, lockstep, sps_lockstep

pytestmark = pytest.mark.gpu

MIN_DRAWS = 10_000
SERVING = WORKLOADS["batched_serving_v128256"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_speculative_decoding_gb300 import build
    build.build()


def _record(name, tally, kinds):
    line = {"test": name, "lw_checked": tally.lw_checked, "lw_err_max": tally.lw_err_max,
            "kinds": {k: dict(zip(("draws", "flagged", "mismatched"), v))
                      for k, v in sorted(tally.kinds.items())}}
    print("TALLY " + json.dumps(line))
    path = os.environ.get("SMCSD_TALLY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")
    for k in kinds:
        d, f, m = tally.kinds.get(k, (0, 0, 0))
        assert d >= MIN_DRAWS, f"{k}: only {d} draws"
        assert m <= MISMATCH_RATE * d, f"{k}: {m} mismatches in {d} draws"


def test_tally_smc_step_serving(pool):
    """32 prompts x 16 particles, K = 1, 40 steps with KV state: even steps
    never resample (every log-weight is compared, at 2e-3), odd steps always
    do (every ancestor is compared).  20480 bonus draws, 10240 ancestors."""
    w = SERVING.with_(B=32, K=1)
    t = lockstep(w, 40, seed=31, with_kv=True, pool=pool,
                 ess_schedule=lambda step: 0.0 if step % 2 == 0 else 1.0)
    _record("smc_step serving B32 N16 K1 V128256 bf16", t, ["bonus", "ancestors"])
    assert t.lw_checked >= MIN_DRAWS


def test_tally_smc_step_serving_k4_at_each_draft_noise(pool):
    """The serving shape itself (B16 N16 K4), 14 steps at each draft noise
    0.25, 1 and 2 with the workload's threshold ESS < N/2: 10752 bonus draws
    and every resampling decision and ancestor these steps take."""
    total = Tally()
    for sigma in (0.25, 1.0, 2.0):
        w = SERVING.with_(sigma_d=sigma)
        total.merge(lockstep(w, 14, seed=37, with_kv=True, pool=pool))
    _record("smc_step serving B16 N16 K4 V128256 bf16, sigma_d 0.25/1/2", total, ["bonus"])


def test_tally_sps_verify(pool):
    """Speculative sampling on the serving rows, K = 4, 8 calls of 2048
    one-particle prompts with drafted tokens sampled from the draft (about
    three prompts in four reject a drafted token, so about 12000 residual
    draws)."""
    total = Tally()
    w = SERVING.with_(B=2048, N=1, K=4)
    for step in range(8):
        t, _, _ = sps_lockstep(w, seed=41, step=step, pool=pool)
        total.merge(t)
    _record("sps_verify B2048x8 K4 V128256 bf16", total, ["sps_accept", "sps_residual"])


def test_tally_draft_sample(pool):
    """The draft-side sampler over 640 x 16 draft rows of the serving
    workload at alpha 1 and 0.5 (20480 draws)."""
    w = SERVING.with_(B=640, K=1)
    inp = make_step_inputs(w, 43, device="cuda")
    rows = inp["draft"][:, :, 0].contiguous()
    del inp
    rows_np = to_numpy_logits(rows)
    tok = torch.empty(w.B * w.N, dtype=torch.int32, device="cuda")
    tally = Tally()
    for alpha in (1.0, 0.5):
        params = smcsd.make_params(w.B, w.N, 1, w.V, w.dtype, alpha, 0.5, 43, 5)
        ws = smcsd.alloc_workspace(params)
        smcsd.smc_draft_sample(params, rows, 0, tok, ws)
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(ws) == 0
        g = tok.cpu().numpy().reshape(w.B, w.N)
        ref, margin = oracle_pool.draft_sample(pool, rows_np, 0, alpha=alpha, seed=43, step=5,
                                               dtype=w.dtype)
        tally.add(g.size, margin < NEAR_TIE, g != ref, f"draft tokens alpha={alpha}", "draft")
    _record("smc_draft_sample 640x16 rows V128256 bf16", tally, ["draft"])


def test_tally_top_p_bonus(pool):
    """smc_step_ex at top_p = 0.9 on the serving rows (B32 N16 K1, drafted
    tokens each draft row's argmax, so inside the draft's nucleus), 20 steps:
    10240 bonus draws inside the target's nucleus."""
    w = SERVING.with_(B=32, K=1)

    def argmax_tokens(inp, step):
        inp["draft_tokens"].copy_(inp["draft"].float().argmax(-1).to(torch.int32))

    t = lockstep(w, 20, seed=47, with_kv=False, pool=pool, top_p=0.9, tokens_fn=argmax_tokens,
                 temperature=1.0)
    _record("smc_step_ex top_p=0.9 B32 N16 K1 V128256 bf16", t, ["bonus"])
