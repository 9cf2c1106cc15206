"""GPU parity: libsmcsd (through its C ABI) against the CPU oracle.

Every test here runs the CUDA kernels on cuda:0.  Integer outputs (ancestors,
tokens, block tables, reference counts, free stacks, copy-on-write pairs) must
match the oracle exactly, except draws the oracle flags as near ties;
log-weights must match within 1e-4 (fp32 logits) or 2e-3 (bf16 logits).
"""
import numpy as np
import pytest
import torch

import smc_speculative_decoding_gb300 as smcsd
from smc_speculative_decoding_gb300.workloads import (WORKLOADS, Workload, make_step_inputs,
                                                      make_kv_state, to_numpy_logits)
from oracle import smc as osmc, kv as okv

from gpu_harness import lockstep, sps_lockstep, StepRunner, kv_to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_speculative_decoding_gb300 import build
    build.build()


def _report(t, name):
    print(f"{name}: {t.summary()}")


# ---------------------------------------------------------------------------
# smc_step in lockstep with the oracle
# ---------------------------------------------------------------------------
def test_tiny_v64_ten_steps_with_kv():
    t = lockstep(WORKLOADS["tiny_v64"], steps=10)
    _report(t, "tiny")
    assert t.mismatched == 0 and t.lw_checked > 0


def test_tiny_v64_no_resampling_checks_every_weight():
    w = WORKLOADS["tiny_v64"].with_(B=3, N=16)
    t = lockstep(w, steps=6, ess_frac=0.0)
    assert t.mismatched == 0 and t.lw_checked == 6 * w.B * w.N


def test_tiny_v64_always_resample():
    w = WORKLOADS["tiny_v64"].with_(B=4, N=32, sigma_d=2.0)
    t = lockstep(w, steps=6, ess_frac=1.0)
    _report(t, "always-resample")
    assert t.rate_ok()


def test_single_prompt_v32000_bf16():
    t = lockstep(WORKLOADS["single_prompt_v32000"], steps=24)
    _report(t, "single prompt")
    assert t.rate_ok()


def test_power_sampling_alpha4_fp32():
    w = WORKLOADS["power_sampling_v151936"].with_(B=2, N=8)
    t = lockstep(w, steps=2)
    _report(t, "power sampling")
    assert t.rate_ok()


def test_serving_full_size_one_step():
    """B16 N16 K4 V128256 bf16, prefix 2048, the bench's launch configuration."""
    t = lockstep(WORKLOADS["batched_serving_v128256"], steps=1)
    _report(t, "serving")
    assert t.rate_ok()


def test_serving_full_size_every_log_weight(pool):
    """B16 N16 K4 V128256 bf16 with resampling off for two steps, so that
    every one of the B*N log-weights is compared (at 2e-3) after each step."""
    w = WORKLOADS["batched_serving_v128256"]
    t = lockstep(w, steps=2, ess_frac=0.0, pool=pool)
    _report(t, "serving, every log-weight")
    assert t.lw_checked == 2 * w.B * w.N
    assert t.rate_ok()


def test_power_sampling_full_size_every_log_weight(pool):
    """B8 N32 K8 V151936 fp32, alpha = 4, resampling off: every log-weight,
    bonus term lse(4 l) - 4 lse(l) included, compared at 1e-4."""
    w = WORKLOADS["power_sampling_v151936"]
    t = lockstep(w, steps=1, ess_frac=0.0, with_kv=False, pool=pool)
    _report(t, "power sampling, every log-weight")
    assert t.lw_checked == w.B * w.N
    assert t.rate_ok()


@pytest.mark.parametrize("case", ["fused_power_sampling", "tail_n64", "tail_top_p_serving"])
def test_large_staged_kv_state(case, pool):
    """KV tables and pools sized for long episodes, staged in dynamic shared
    memory: 30 to 45 KB on top of the tail's static shared memory, so the
    launch needs the opt-in above 48 KB.  Through the fused epilogue (N = 32)
    and through the separate tail kernel (N = 64, and top-p)."""
    from test_gpu_next import _nucleus_tokens
    if case == "fused_power_sampling":
        w = WORKLOADS["power_sampling_v151936"].with_(B=1)
        t = lockstep(w, steps=2, kv_steps=128, pool=pool)
    elif case == "tail_n64":
        w = WORKLOADS["sweep_v128256"].with_(B=2, N=64, K=8)
        t = lockstep(w, steps=2, kv_steps=32, pool=pool)
    else:
        w = WORKLOADS["batched_serving_v128256"].with_(B=2)
        t = lockstep(w, steps=1, kv_steps=128, pool=pool, top_p=0.95,
                     tokens_fn=_nucleus_tokens(w, 0.95, 1.0, 61))
    _report(t, f"large staged KV ({case})")
    assert t.rate_ok()


@pytest.mark.parametrize("V,dtype", [(1001, "bf16"), (37, "f32"), (8193, "bf16"),
                                     (16392, "bf16"), (4097, "f32"), (1, "f32"), (2, "bf16")])
def test_ragged_and_unaligned_vocab(V, dtype):
    w = Workload(f"ragged_{V}", B=2, N=5, K=2, V=V, dtype=dtype, sigma_t=2.0,
                 top_m=min(5, V), sigma_d=1.0, steps=3, prefix=7, block_size=4)
    t = lockstep(w, steps=3)
    assert t.mismatched == 0


def test_single_particle_single_draft():
    w = Workload("n1k1", B=3, N=1, K=1, V=300, dtype="f32", sigma_t=2.0, top_m=3,
                 sigma_d=1.0, steps=4, prefix=5, block_size=2)
    t = lockstep(w, steps=4)
    assert t.mismatched == 0


def test_max_particles_and_long_draft():
    w = Workload("n256", B=1, N=256, K=9, V=96, dtype="f32", sigma_t=2.0, top_m=4,
                 sigma_d=1.5, steps=3, prefix=20, block_size=8)
    t = lockstep(w, steps=3)
    _report(t, "N=256")
    assert t.rate_ok()


def test_misaligned_base_pointer_takes_scalar_path():
    w = Workload("mis", B=2, N=3, K=2, V=512, dtype="bf16", sigma_t=2.0, top_m=5,
                 sigma_d=1.0, steps=1, prefix=4, block_size=4)
    inp = make_step_inputs(w, 3, device="cuda")
    runner = StepRunner(w, seed=3, with_kv=False)
    shifted = {}
    for key in ("target", "draft"):
        buf = torch.empty(inp[key].numel() + 1, dtype=inp[key].dtype, device="cuda")
        view = buf[1:]
        view.copy_(inp[key].reshape(-1))
        shifted[key] = view
    shifted["draft_tokens"] = inp["draft_tokens"]
    runner.run(shifted, 0)
    torch.cuda.synchronize()
    assert runner.status() == 0
    ref = osmc.smc_step(to_numpy_logits(inp["target"]), to_numpy_logits(inp["draft"]),
                        inp["draft_tokens"].cpu().numpy(), np.zeros((2, 3)),
                        seed=3, step=0, dtype="bf16")
    g = runner.tokens_out.cpu().numpy().reshape(2, 3, 3)
    assert np.array_equal(g, ref["tokens_out"]) or (ref["bonus_margin"] < 1e-5).any()


def test_repeat_call_is_bitwise_deterministic():
    w = WORKLOADS["single_prompt_v32000"].with_(B=2)
    inp = make_step_inputs(w, 5, device="cuda")
    outs = []
    for _ in range(2):
        r = StepRunner(w, seed=5, with_kv=True, steps=2)
        r.run(inp, 0)
        torch.cuda.synchronize()
        outs.append([t.cpu().clone() for t in (r.log_weights, r.tokens_out, r.ancestors, r.ess)]
                    + [v.cpu().clone() for v in r.kv.values()])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_bonus_mismatch_rate_at_v128256(pool):
    """Float-float sampling sums: bonus tokens at V=128256 agree with the
    fp64 oracle except on near ties, and every log-weight within 2e-3;
    resampling is off, so each of the 12 steps compares all 512 weights."""
    w = WORKLOADS["batched_serving_v128256"].with_(K=1, N=16, B=32)
    t = lockstep(w, steps=12, seed=11, with_kv=False, ess_frac=0.0, pool=pool)
    _report(t, "bonus at V=128256")
    assert t.kinds["bonus"][0] == 12 * w.B * w.N
    assert t.lw_checked == 12 * w.B * w.N
    assert t.rate_ok()


# ---------------------------------------------------------------------------
# sps_verify
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("V,dtype,B,K", [(64, "f32", 256, 3), (128256, "bf16", 32, 4),
                                         (1001, "bf16", 64, 2), (151936, "f32", 8, 8)])
def test_sps_verify_matches_oracle(V, dtype, B, K):
    w = Workload("sps", B=B, N=1, K=K, V=V, dtype=dtype, sigma_t=3.0 if V > 64 else 2.0,
                 top_m=50 if V > 64 else 0, sigma_d=1.0, steps=1)
    t, ref, g_n = sps_lockstep(w, seed=2, step=1)
    _report(t, f"sps V={V}")
    assert (ref["n_emitted"] < K + 1).any(), "no rejection exercised"
    assert t.rate_ok()


def test_sps_verify_draft_equals_target_accepts_all():
    w = Workload("sps_eq", B=16, N=1, K=4, V=500, dtype="f32", sigma_t=2.0, top_m=0,
                 sigma_d=0.0, steps=1)
    t, ref, g_n = sps_lockstep(w, seed=4, step=0)
    assert (g_n == 5).all()


def _swapped_pair_drafts(shift):
    """tokens_fn for sps_lockstep: each draft row becomes its target row with
    two logits swapped, a (target probability nearest 3e-5) and b (the
    smallest logit), and every other logit moved by `shift`; every drafted
    token is b, so position 0 rejects almost surely.  The residual then lies
    on a and on the shifted bulk, where p/q is the same for every element and
    within about 1e-4 of 1: the sign of p - q is a close call for every
    element of the bulk, and the residual must still come out exact."""
    def fn(inp, step):
        K = inp["draft"].shape[2]
        tg = inp["target"][:, 0, :K].float()
        logp = torch.log_softmax(tg.double(), dim=-1)
        a = (logp - np.log(3e-5)).abs().argmin(dim=-1, keepdim=True)
        b = tg.argmin(dim=-1, keepdim=True)
        d = tg + shift
        d.scatter_(-1, a, tg.gather(-1, b))
        d.scatter_(-1, b, tg.gather(-1, a))
        inp["draft"][:, 0].copy_(d.to(inp["draft"].dtype))
        inp["draft_tokens"][:, 0].copy_(b.squeeze(-1).to(torch.int32))
    return fn


@pytest.mark.parametrize("dtype,shift", [("bf16", 0.0), ("f32", -1.0), ("f32", 1.0)])
def test_sps_verify_residual_with_a_bulk_of_close_calls(dtype, shift):
    """shift 0: p = q exactly on the bulk (bf16 rows copied), so the sign of
    p - q there is a tie that rounding decides; the bulk's residual is zero
    and the draw must land on a.  shift -1 / +1 (fp32): p/q on the bulk is
    1 + 5e-5 or 1 - 2e-5, so the bulk carries about 60 % of the residual mass,
    or none of it."""
    w = Workload("sps_close", B=32, N=1, K=2, V=128256, dtype=dtype, sigma_t=3.0, top_m=50,
                 sigma_d=1.0, steps=1)
    t, ref, g_n = sps_lockstep(w, seed=6, step=2, tokens_fn=_swapped_pair_drafts(shift))
    _report(t, f"sps close calls {dtype} shift={shift}")
    assert (ref["n_emitted"] == 1).mean() > 0.9, "position 0 should reject"
    assert t.rate_ok()


# ---------------------------------------------------------------------------
# standalone smc_resample and kv_blocktable_remap
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N", [1, 7, 64, 256])
def test_smc_resample_bit_exact_on_identical_weights(N):
    B = 40
    rng = np.random.default_rng(N)
    lw = (rng.normal(0, 1, (B, N)) * rng.uniform(0.1, 4, (B, 1))).astype(np.float32)
    lw[::5, : max(1, N // 3)] = -np.inf
    lw[::5, 0] = 0.0
    params = smcsd.make_params(B, N, 1, 1, "f32", 1.0, 0.7, 123, 9)
    ws = smcsd.alloc_workspace(params)
    d_lw = torch.from_numpy(lw.reshape(-1).copy()).cuda()
    anc = torch.empty(B * N, dtype=torch.int32, device="cuda")
    ess = torch.empty(B, dtype=torch.float32, device="cuda")
    res = torch.empty(B, dtype=torch.int32, device="cuda")
    smcsd.smc_resample(params, d_lw, anc, ess, res, ws)
    torch.cuda.synchronize()
    assert smcsd.smc_device_status(ws) == 0
    g_anc = anc.cpu().numpy().reshape(B, N)
    g_lw = d_lw.cpu().numpy().reshape(B, N)
    for b in range(B):
        r = osmc.resample_prompt(lw[b].astype(np.float64), 0.7, 123, 9, b)
        # the GPU normalises in fp32: decisions agree except within fp32 rounding
        assert abs(ess[b].item() - r["ess"]) <= 1e-5 * r["ess"]
        assert bool(res[b].item()) == r["resampled"] or r["ess_margin"] < 1e-5
        if r["resampled"]:
            ok = (g_anc[b] == r["ancestors"]) | (r["margins"] < 1e-6)
            assert ok.all()
            assert (g_lw[b] == 0).all()
        else:
            assert np.array_equal(g_anc[b], np.arange(N))
            assert np.array_equal(g_lw[b], lw[b])


@pytest.mark.parametrize("prefix,bs,N,T_min", [(10, 4, 12, 0), (32, 16, 12, 0), (0, 8, 12, 0),
                                               (40, 4, 256, 120)])
def test_kv_blocktable_remap_bit_exact(prefix, bs, N, T_min):
    """Small tables take the shared-memory staged path; N*T = 30720 entries
    (last case) exceeds the staging budget and takes the global-scratch path."""
    B, steps, n_app = 3 if N < 100 else 2, 8, 5
    T = max(T_min, (prefix + steps * n_app + bs - 1) // bs + 1)
    P = N * T
    params = smcsd.make_params(B, N, 4, 8, "f32")
    kv = make_kv_state(B, N, prefix, bs, T, P, device="cuda")
    kv_s = smcsd.make_kv(params, kv, bs)
    ws = smcsd.alloc_workspace(params, kv_s)
    rng = np.random.default_rng(prefix + bs)
    for step in range(steps):
        res = (rng.random(B) < 0.7).astype(np.int32)
        anc = np.stack([np.sort(rng.integers(0, N, N)) for _ in range(B)]).astype(np.int32)
        before = kv_to_numpy(kv)
        smcsd.kv_blocktable_remap(params, kv_s, torch.from_numpy(anc.reshape(-1)).cuda(),
                                  torch.from_numpy(res).cuda(), n_app, ws)
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(ws) == 0
        ref = okv.remap_append(before["tables"], before["seq_len"], before["refcount"],
                               before["free_list"], before["free_top"],
                               np.where(res[:, None] == 1, anc, np.arange(N)[None]),
                               res.astype(bool), n_app, bs, P)
        got = kv_to_numpy(kv)
        for key in ("tables", "seq_len", "refcount", "free_top"):
            assert np.array_equal(got[key], ref[key]), key
        for b in range(B):
            top = ref["free_top"][b]
            assert np.array_equal(got["free_list"][b, :top], ref["free_list"][b, :top])
            assert got["n_cow"][b] == len(ref["cow_pairs"][b])
            if ref["cow_pairs"][b]:
                assert np.array_equal(got["cow_pairs"][b, :len(ref["cow_pairs"][b])],
                                      np.array(ref["cow_pairs"][b]))


# ---------------------------------------------------------------------------
# bonus rows with extreme value ranges
# ---------------------------------------------------------------------------
def _bonus_check(w, inp, seed=5):
    """One step (no resampling) and the bonus tokens against the oracle."""
    r = StepRunner(w, seed=seed, with_kv=False, ess_frac=0.0)
    r.run(inp, 0)
    torch.cuda.synchronize()
    assert r.status() == 0
    x = inp["draft_tokens"].cpu().numpy().astype(np.int64)
    ref = osmc.smc_step(to_numpy_logits(inp["target"]), to_numpy_logits(inp["draft"]), x,
                        np.zeros((w.B, w.N)), alpha=w.alpha, ess_frac=0.0, seed=seed, step=0,
                        dtype=w.dtype)
    g = r.tokens_out.cpu().numpy().reshape(w.B, w.N, w.K + 1)[:, :, w.K]
    flagged = ref["bonus_margin"] < 1e-5
    bad = (g != ref["bonus"]) & ~flagged
    assert not bad.any(), (np.argwhere(bad)[:4], g[bad][:4], ref["bonus"][bad][:4])
    lw = r.log_weights.cpu().numpy().reshape(w.B, w.N)
    assert np.abs(lw - ref["log_weights_pre"]).max() <= (2e-3 if w.dtype == "bf16" else 1e-4)
    return g, ref


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("log2_big", [30, 32])
def test_bonus_row_with_huge_max(dtype, log2_big):
    """Bonus rows with two equal maxima of 2^30 or 2^32 in different units,
    everything else O(1): the token is the first maximum iff u < 1/2.  At
    2^32, max - 40 rounds to max, so the streaming kernel flags those units
    and the combine sums them exactly instead."""
    w = WORKLOADS["single_prompt_v32000"].with_(B=2, N=4, K=2, V=40000, dtype=dtype)
    inp = make_step_inputs(w, 21, device="cuda")
    big = 2.0 ** log2_big
    below = 2.0 ** (log2_big - (8 if dtype == "bf16" else 24))  # one step below big
    t = inp["target"]
    t[:, :, w.K, 3000] = big
    t[:, :, w.K, 35000] = big
    t[0, 1, w.K, 17] = big - below
    g, ref = _bonus_check(w, inp)
    assert set(np.unique(g)) <= {3000, 35000}


def test_bonus_row_of_tiny_logits_under_a_large_max():
    """bf16 logits 2^-20 in size against a max of 12: x - max is not a float
    there, and the weights must still sum to the oracle's within tolerance."""
    w = WORKLOADS["single_prompt_v32000"].with_(B=2, N=8, K=2, V=32000)
    inp = make_step_inputs(w, 22, device="cuda")
    t = inp["target"]
    tiny = (torch.randn(t[:, :, w.K].shape, device="cuda") * 2.0 ** -20).to(t.dtype)
    t[:, :, w.K] = tiny
    t[:, :, w.K, 777] = 2.5
    _bonus_check(w, inp)


def test_row_timing_hook_records_the_row_pass_and_changes_nothing():
    w = WORKLOADS["single_prompt_v32000"].with_(B=2)
    inp = make_step_inputs(w, 3, device="cuda")
    plain = StepRunner(w, seed=3, with_kv=True, steps=2)
    plain.run(inp, 0)
    hooked = StepRunner(w, seed=3, with_kv=True, steps=2)
    b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    smcsd.smc_set_row_timing_events(b, e)
    try:
        hooked.run(inp, 0)
    finally:
        smcsd.smc_set_row_timing_events(None, None)
    torch.cuda.synchronize()
    assert b.elapsed_time(e) > 0.0
    assert plain.status() == 0 and hooked.status() == 0
    for name in ("log_weights", "tokens_out", "ancestors", "ess", "resampled"):
        assert torch.equal(getattr(plain, name), getattr(hooked, name)), name
    for key in plain.kv:
        assert torch.equal(plain.kv[key], hooked.kv[key]), key


# ---------------------------------------------------------------------------
# errors: reported through the status word, never a trap
# ---------------------------------------------------------------------------
def _tiny_run(mutate, with_kv=False, kv_mut=None):
    w = WORKLOADS["tiny_v64"].with_(B=2)
    inp = make_step_inputs(w, 1, device="cuda")
    mutate(inp)
    r = StepRunner(w, seed=1, with_kv=with_kv, steps=2)
    if kv_mut:
        kv_mut(r)
    r.run(inp, 0)
    torch.cuda.synchronize()
    return set(smcsd.status_names(r.status()))


def test_status_nonfinite_logit():
    def m(inp):
        inp["target"][0, 1, 2, 7] = float("nan")
    assert "nonfinite" in _tiny_run(m)


def test_status_nonfinite_bonus_row():
    def m(inp):
        inp["target"][1, 0, 3, 0] = float("inf")
    assert "nonfinite" in _tiny_run(m)


def test_status_empty_row():
    def m(inp):
        inp["draft"][0, 0, 1, :] = float("-inf")
    assert "empty_row" in _tiny_run(m)


def test_status_bad_token():
    def m(inp):
        inp["draft_tokens"][1, 2, 0] = 64
    assert "bad_token" in _tiny_run(m)


def test_status_all_zero_weight():
    def kvm(r):
        r.log_weights.fill_(float("-inf"))
    assert "all_zero_weight" in _tiny_run(lambda inp: None, kv_mut=kvm)


def test_status_pool_exhausted():
    def kvm(r):
        r.kv["free_top"].zero_()
    assert "pool_exhausted" in _tiny_run(lambda inp: None, with_kv=True, kv_mut=kvm)


def test_status_table_overflow():
    """Tables sized for one step; the step that outgrows them reports it."""
    w = WORKLOADS["tiny_v64"].with_(B=2)
    r = StepRunner(w, seed=1, with_kv=True, steps=1)
    seen = set()
    for step in range(12):
        r.run(make_step_inputs(w, 1, device="cuda", step=step), step)
        torch.cuda.synchronize()
        seen |= set(smcsd.status_names(r.status()))
        if seen:
            break
    assert seen == {"table_overflow"}


def test_status_bad_block():
    def kvm(r):
        r.kv["tables"][1, 0, 0] = 0  # prompt 0's block in prompt 1's table
        r.log_weights.copy_(torch.tensor([0.0, -50.0, -50.0, -50.0] * 2, device="cuda"))
    bits = _tiny_run(lambda inp: None, with_kv=True, kv_mut=kvm)
    assert "bad_block" in bits


def test_host_side_argument_errors():
    p = smcsd.make_params(1, 300, 3, 64, "f32")
    with pytest.raises(smcsd.SmcError):
        smcsd.smc_workspace_bytes(p)
    p = smcsd.make_params(2, 4, 3, 64, "f32")
    ws = smcsd.alloc_workspace(p)
    z = torch.zeros(2 * 4 * 4 * 64, device="cuda")
    small_ws = ws[: ws.numel() // 2]
    with pytest.raises(smcsd.SmcError):  # sps_verify needs N == 1
        smcsd.sps_verify(p, z[: 2 * 4 * 64], z[: 2 * 3 * 64],
                         torch.zeros(6, dtype=torch.int32, device="cuda"),
                         torch.empty(8, dtype=torch.int32, device="cuda"),
                         torch.empty(2, dtype=torch.int32, device="cuda"), ws)
    with pytest.raises(smcsd.SmcError):
        smcsd.smc_resample(p, torch.zeros(8, device="cuda"),
                           torch.empty(8, dtype=torch.int32, device="cuda"),
                           torch.empty(2, device="cuda"),
                           torch.empty(2, dtype=torch.int32, device="cuda"), small_ws)
