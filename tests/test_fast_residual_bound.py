"""The error bound behind sps_verify's fp32 residual pass, checked on the CPU.

The fp32 pass ("Accelerating Large Language Model Decoding with Speculative
Sampling", section 4.2, the residual max(0, p - q)) draws a token only when
u R lies farther than 2E from both edges of the token's interval in its
computed CDF. E bounds the distance between that CDF and the exact one at
every prefix. These tests take the pass's arithmetic in numpy float32, step
for step. Each exp2 is given an error of 2 ulp with a random sign, the most
CUDA documents for its approximation. The tests then check three things on
rows shaped like the serving workload's: the bound holds at every prefix,
every draw the margin test accepts is the exact inverse-CDF draw, and most
draws are accepted.

The kernel's constants are restated here from their derivation:
- kArgErr = 2.09 u per unit of |y|: three roundings of y, through 2^y;
- kEx2Err = 2^-21: twice the documented 2-ulp error;
- 64 u for the lane sums, the normaliser divisions and the weights' roundings;
- |cp - cq| S_q for weighing Q by cp.
"""
import numpy as np
import pytest
import torch

from smc_speculative_decoding_gb300.workloads import WORKLOADS, make_step_inputs

U = 2.0 ** -24
K_ARG = 2.09 * U
K_EX2 = 2.0 ** -21
ROUND_UNITS = 64
LANE = 16          # terms in each fp32 lane sum (bf16: 32 logits a thread, two lanes)
F32 = np.float32


def _fma32(a, b, c):
    """fl32(a b + c) for float32 operands: the product is exact in float64."""
    return (a.astype(np.float64) * np.float64(b) + np.float64(c)).astype(F32)


def _fast_probs(x, lse_hi, lse_lo, rng):
    """P^ = 2^y with y = fl(fl(x - L.hi) log2 e - L.lo log2 e), as the pass takes
    it at T = 1, and |y|; 2^y carries a 2-ulp error of random sign."""
    t = (x.astype(F32) - F32(lse_hi)).astype(F32)
    y = _fma32(t, F32(np.log2(np.e)), F32(-F32(lse_lo) * F32(np.log2(np.e))))
    p = np.exp2(y.astype(np.float64)) * (1.0 + rng.choice([-1.0, 1.0], y.shape) * 2.0 ** -22)
    return p.astype(F32), np.abs(y.astype(np.float64))


def _lane_sum(v):
    """Sequential float32 sums of LANE terms, then exact addition (float-float)."""
    v = v.astype(F32)
    pad = (-len(v)) % LANE
    v = np.concatenate([v, np.zeros(pad, F32)]).reshape(-1, LANE)
    acc = np.zeros(v.shape[0], F32)
    for j in range(LANE):
        acc = (acc + v[:, j]).astype(F32)
    return float(acc.astype(np.float64).sum())


def _case(x, y, rng):
    """(E, max prefix error, residual error, computed CDF, exact CDF)."""
    xd, yd = x.astype(np.float64), y.astype(np.float64)
    lp = np.logaddexp.reduce(xd)
    lq = np.logaddexp.reduce(yd)
    # the row kernel's log-sum-exps are right to about 1e-7: perturb them so
    lp_hi = F32(lp * (1 + 1e-7 * rng.standard_normal()))
    lq_hi = F32(lq * (1 + 1e-7 * rng.standard_normal()))
    P, ayp = _fast_probs(x, lp_hi, 0.0, rng)
    Q, ayq = _fast_probs(y, lq_hi, 0.0, rng)
    D = (P - Q).astype(F32)
    sp, sq = _lane_sum(P), _lane_sum(Q)
    bnd = float((P * ayp).sum() + (Q * ayq).sum())
    cp = F32(F32(1.0) / F32(sp))
    dc = float(F32(cp - F32(F32(1.0) / F32(sq))))
    err = 1.05 * (2 * K_ARG * bnd / min(sp, sq) + 4 * K_EX2 + ROUND_UNITS * U
                  + 1.001 * abs(dc) * sq)
    w = (cp * np.maximum(D, F32(0))).astype(F32).astype(np.float64)
    C = np.cumsum(w)
    p = np.exp(xd - lp)
    q = np.exp(yd - lq)
    Ce = np.cumsum(np.maximum(p - q, 0.0))
    return err, float(np.abs(C - Ce).max()), abs(C[-1] - Ce[-1]), C, Ce


def _rows(n_prompts, V, seed):
    w = WORKLOADS["batched_serving_v128256"].with_(B=1, N=n_prompts, V=V)
    inp = make_step_inputs(w, seed)
    t = inp["target"].float().numpy().reshape(-1, w.K + 1, V)
    d = inp["draft"].float().numpy().reshape(-1, w.K, V)
    return [(t[i, j], d[i, j]) for i in range(t.shape[0]) for j in range(w.K)]


def test_bound_holds_at_every_prefix():
    rng = np.random.default_rng(5)
    for x, y in _rows(4, 32000, 11):
        err, worst, rerr, _, _ = _case(x, y, rng)
        assert worst <= err and rerr <= err, (worst, err)
        # and the bound is not vacuous: well under the 1e-5 near-tie margin scale
        assert err < 2e-5


def test_margin_test_never_settles_a_wrong_token():
    rng = np.random.default_rng(7)
    settled = total = 0
    for x, y in _rows(8, 32000, 13):
        err, _, _, C, Ce = _case(x, y, rng)
        R, Re = C[-1], Ce[-1]
        for u in rng.random(16):
            t = u * R
            k = int(np.searchsorted(C, t, side="right"))
            if k >= len(C):
                continue
            before = C[k - 1] if k > 0 else 0.0
            ok = R > 4 * err and t - before > 2 * err and C[k] - t > 2 * err
            total += 1
            if ok:
                settled += 1
                assert k == int(np.searchsorted(Ce, u * Re, side="right"))
    # most draws are settled by the fp32 pass (about four in five on these rows)
    assert settled >= 0.6 * total


@pytest.mark.parametrize("shift", [0.0, 1e-3])
def test_equal_rows_are_never_settled(shift):
    """p == q (up to a tiny shift): the residual is (nearly) empty, so the
    margin test must leave the draw to the float-float pass."""
    rng = np.random.default_rng(3)
    x = _rows(1, 4096, 17)[0][0]
    y = (x.astype(np.float64) + shift).astype(F32)
    y = torch.from_numpy(y).to(torch.bfloat16).float().numpy()
    err, _, _, C, _ = _case(x, y, rng)
    assert not C[-1] > 4 * err
