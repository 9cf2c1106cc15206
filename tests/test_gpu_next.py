"""GPU parity of the step's extensions against the CPU oracle: smc_step_ex
(temperature, per-particle log-potentials, top-p nuclei), smc_draft_sample
(the draft-side sampler) and smc_kv_usage (KV-cache accounting).  Same bar as the basic
step: integer outputs exact except draws the oracle flags as near ties, and
no more such mismatches than 1e-4 of the draws (none, below 10^4 draws);
log-weights within 1e-4 (fp32 logits) or 2e-3 (bf16 logits).  The tests
built to put the nucleus boundary on ties of equal logits (tied and
two-valued rows, vocabularies of a few tokens) require only that every
mismatch be flagged: they sample the near-tie cases on purpose."""
import numpy as np
import pytest
import torch

import smc_speculative_decoding_gb300 as smcsd
from smc_speculative_decoding_gb300.workloads import (WORKLOADS, Workload, make_step_inputs,
                                                      to_numpy_logits)
from smc_speculative_decoding_gb300.workloads import torch_dtype
from oracle import smc as osmc, kv as okv

from gpu_harness import lockstep, sps_lockstep, StepRunner, kv_to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_speculative_decoding_gb300 import build
    build.build()


def _potentials(w, seed):
    """A step's log-potentials: N(0, 0.7^2), and -inf on one particle of each
    prompt on odd steps (a violated constraint)."""
    def fn(step):
        g = torch.Generator(device="cuda")
        g.manual_seed(seed * 7919 + step)
        phi = torch.randn(w.B, w.N, generator=g, device="cuda") * 0.7
        if step % 2:
            phi[:, (step // 2) % w.N] = float("-inf")
        return phi.reshape(-1).contiguous()
    return fn


@pytest.mark.parametrize("name,B,temperature", [("tiny_v64", 2, 0.7),
                                                ("single_prompt_v32000", 2, 1.6),
                                                ("power_sampling_v151936", 1, 0.8)])
def test_step_ex_matches_oracle(name, B, temperature):
    w = WORKLOADS[name].with_(B=B)
    steps = 6 if w.V > 1000 else 10
    t = lockstep(w, steps, seed=17, with_kv=True, temperature=temperature,
                 potential_fn=_potentials(w, 17))
    print(f"{name} T={temperature}: {t.summary()}")
    assert t.rate_ok()


def test_step_ex_serving_size_one_step():
    w = WORKLOADS["batched_serving_v128256"].with_(B=4)
    t = lockstep(w, 2, seed=5, with_kv=True, temperature=1.3, potential_fn=_potentials(w, 5))
    print(f"serving T=1.3: {t.summary()}")
    assert t.rate_ok()


def test_step_ex_unaligned_vocab_takes_the_per_chunk_path():
    w = WORKLOADS["single_prompt_v32000"].with_(V=1001, B=3)
    lockstep(w, 4, seed=8, with_kv=False, temperature=0.6, potential_fn=_potentials(w, 8))


def test_step_ex_defaults_equal_smc_step():
    w = WORKLOADS["single_prompt_v32000"].with_(B=2)
    inp = make_step_inputs(w, 4, device="cuda")
    a = StepRunner(w, seed=4, with_kv=True, steps=2)
    b = StepRunner(w, seed=4, with_kv=True, steps=2, temperature=1.0)
    a.run(inp, 0)
    b.run(inp, 0)
    torch.cuda.synchronize()
    for name in ("log_weights", "tokens_out", "ancestors", "ess", "resampled"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    for key in a.kv:
        assert torch.equal(a.kv[key], b.kv[key]), key


@pytest.mark.parametrize("V,dtype,alpha", [(128256, "bf16", 1.0), (128256, "bf16", 0.5),
                                           (151936, "f32", 1.0), (1001, "bf16", 1.0),
                                           (64, "f32", 2.0)])
def test_draft_sample_matches_oracle(V, dtype, alpha):
    w = WORKLOADS["sweep_v128256"].with_(B=8, N=8, K=2, V=V, dtype=dtype)
    draft = make_step_inputs(w, 31, device="cuda")["draft"][:, :, 0].contiguous()
    params = smcsd.make_params(w.B, w.N, w.K, V, dtype, alpha, 0.5, 31, 3)
    ws = smcsd.alloc_workspace(params)
    out = torch.empty(w.B * w.N, dtype=torch.int32, device="cuda")
    draws = mism = flagged = 0
    for position in range(3):
        smcsd.smc_draft_sample(params, draft, position, out, ws)
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(ws, clear=True) == 0
        ref, margin = osmc.draft_sample(to_numpy_logits(draft), position, alpha=alpha, seed=31,
                                        step=3, dtype=dtype)
        g = out.cpu().numpy().reshape(w.B, w.N)
        bad = (g != ref) & (margin >= 1e-5)
        assert not bad.any(), (np.argwhere(bad)[:4], g[bad][:4], ref[bad][:4])
        draws += g.size
        flagged += int((margin < 1e-5).sum())
        mism += int((g != ref).sum())
    print(f"draft sample V={V} {dtype} alpha={alpha}: draws={draws} flagged={flagged} "
          f"mismatched={mism}")
    assert mism <= 1e-4 * draws


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_draft_sample_masked_vocab(dtype):
    """Half of every row masked to -inf (a constrained vocabulary): draws land
    in the unmasked half and match the oracle."""
    w = WORKLOADS["single_prompt_v32000"].with_(B=2, N=8, dtype=dtype)
    draft = make_step_inputs(w, 37, device="cuda")["draft"][:, :, 0].contiguous()
    draft[..., ::2] = float("-inf")
    params = smcsd.make_params(w.B, w.N, w.K, w.V, dtype, 1.0, 0.5, 37, 5)
    ws = smcsd.alloc_workspace(params)
    out = torch.empty(w.B * w.N, dtype=torch.int32, device="cuda")
    smcsd.smc_draft_sample(params, draft, 1, out, ws)
    torch.cuda.synchronize()
    assert smcsd.smc_device_status(ws, clear=True) == 0
    g = out.cpu().numpy().reshape(w.B, w.N)
    assert (g % 2 == 1).all()
    ref, margin = osmc.draft_sample(to_numpy_logits(draft), 1, alpha=1.0, seed=37, step=5,
                                    dtype=dtype)
    assert not ((g != ref) & (margin >= 1e-5)).any()


def test_draft_sample_nonfinite_row_is_reported():
    w = WORKLOADS["tiny_v64"].with_(B=1, N=4)
    draft = make_step_inputs(w, 2, device="cuda")["draft"][:, :, 0].contiguous()
    draft[0, 1, 7] = float("nan")
    params = smcsd.make_params(1, 4, 3, 64, "f32", 1.0, 0.5, 2, 0)
    ws = smcsd.alloc_workspace(params)
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    smcsd.smc_draft_sample(params, draft, 0, out, ws)
    torch.cuda.synchronize()
    # a status bit leaves that call's outputs unspecified; the call still
    # writes a token or -1 for every particle
    assert "nonfinite" in smcsd.status_names(smcsd.smc_device_status(ws, clear=True))
    assert all(-1 <= t < 64 for t in out.tolist())


def test_draft_sample_empty_row_reports_and_returns_minus_one():
    w = WORKLOADS["tiny_v64"].with_(B=1, N=4)
    draft = make_step_inputs(w, 2, device="cuda")["draft"][:, :, 0].contiguous()
    draft[0, 2, :] = float("-inf")
    params = smcsd.make_params(1, 4, 3, 64, "f32", 1.0, 0.5, 2, 0)
    ws = smcsd.alloc_workspace(params)
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    smcsd.smc_draft_sample(params, draft, 0, out, ws)
    torch.cuda.synchronize()
    assert "empty_row" in smcsd.status_names(smcsd.smc_device_status(ws, clear=True))
    assert out[2].item() == -1


def test_kv_usage_matches_oracle():
    w = WORKLOADS["single_prompt_v32000"].with_(B=3, N=8)
    r = StepRunner(w, seed=12, with_kv=True, steps=6)
    params = r.params(0)
    used = torch.empty(w.B, dtype=torch.int32, device="cuda")
    unshared = torch.empty(w.B, dtype=torch.int32, device="cuda")
    for step in range(6):
        r.run(make_step_inputs(w, 12, device="cuda", step=step), step)
        smcsd.smc_kv_usage(params, r.kv_struct, used, unshared)
        torch.cuda.synchronize()
        assert r.status() == 0
        st = kv_to_numpy(r.kv)
        ref_used, ref_unshared = okv.usage(st["tables"], st["seq_len"], w.block_size)
        assert np.array_equal(used.cpu().numpy(), ref_used)
        assert np.array_equal(unshared.cpu().numpy(), ref_unshared)


def _nucleus_tokens(w, top_p, temperature, seed):
    """Replaces each step's drafted tokens by tokens drawn from the draft
    row's renormalised nucleus (computed by the oracle, on the CPU): inputs
    that a top-p draft could have produced."""
    rng = np.random.default_rng(seed)
    s = osmc.temperature_scale(temperature)

    def fn(inp, step):
        d = to_numpy_logits(inp["draft"])
        toks = np.zeros((w.B, w.N, w.K), dtype=np.int32)
        for b in range(w.B):
            for n in range(w.N):
                rows = osmc.widen(d[b, n], w.dtype) * s
                for k in range(w.K):
                    kept, _, _ = osmc.nucleus(rows[k], top_p)
                    pk = np.where(kept, np.exp(rows[k] - rows[k][kept].max()), 0.0)
                    toks[b, n, k] = rng.choice(len(pk), p=pk / pk.sum())
        inp["draft_tokens"].copy_(torch.from_numpy(toks).to(inp["draft_tokens"].device))
    return fn


@pytest.mark.parametrize("name,B,top_p,temperature", [("tiny_v64", 2, 0.8, 1.0),
                                                      ("single_prompt_v32000", 2, 0.9, 1.0),
                                                      ("single_prompt_v32000", 2, 0.5, 0.7)])
def test_step_ex_top_p_matches_oracle(name, B, top_p, temperature):
    w = WORKLOADS[name].with_(B=B)
    steps = 4 if w.V > 1000 else 10
    t = lockstep(w, steps, seed=23, with_kv=True, temperature=temperature, top_p=top_p,
                 tokens_fn=_nucleus_tokens(w, top_p, temperature, 23))
    print(f"{name} top_p={top_p} T={temperature}: {t.summary()}")
    assert t.rate_ok()


@pytest.mark.parametrize("V,top_p", [(32000, 0.9), (151936, 0.8)])
def test_step_ex_top_p_fp32_rows(V, top_p):
    """fp32 logits: the nucleus kernel's first attempt keeps 32-bit values in its
    list (16 a thread) and tests groups of four logits."""
    w = WORKLOADS["single_prompt_v32000"].with_(B=2, N=4, V=V, dtype="f32")
    t = lockstep(w, 2, seed=67, with_kv=False, top_p=top_p,
                 tokens_fn=_nucleus_tokens(w, top_p, 1.0, 67))
    print(f"fp32 V={V} top_p={top_p}: {t.summary()}")
    assert t.rate_ok()


def test_step_ex_top_p_serving_size_and_unaligned():
    w = WORKLOADS["batched_serving_v128256"].with_(B=2, N=8)
    lockstep(w, 2, seed=29, with_kv=True, top_p=0.95,
             tokens_fn=_nucleus_tokens(w, 0.95, 1.0, 29))
    w = WORKLOADS["single_prompt_v32000"].with_(V=1001, B=2)
    lockstep(w, 3, seed=30, with_kv=False, top_p=0.6, tokens_fn=_nucleus_tokens(w, 0.6, 1.0, 30))


@pytest.mark.parametrize("sigma_t,top_m,top_p,sigma_d", [(1.0, 0, 0.9, 1.0), (0.05, 0, 0.5, 1.0),
                                                         (3.0, 50, 0.99, 1.0), (2.0, 0, 0.5, 0.0)])
def test_step_ex_top_p_threshold_below_the_first_attempt(sigma_t, top_m, top_p, sigma_d):
    """Serving-size rows whose nucleus threshold lies below pi = 2^-16 (sigma 1:
    about 2^-18; sigma 0.05: every pi near 1/V; top_p 0.99 on the serving
    logits), so the nucleus kernel's first attempt, which bins only the
    logits above 2^-16, falls short of top_p and the full pass runs.  With
    sigma 2 and top_p 0.5 the threshold lies near 2^-14, inside the first
    attempt, but about 12000 logits of a row lie above 2^-16: some threads'
    slices of the shared-memory list overflow, and the threshold bin's logits
    are read from the row again (draft rows equal to the target rows, so that
    the drafted tokens lie in the target's nucleus at so small a top_p)."""
    w = WORKLOADS["batched_serving_v128256"].with_(B=2, N=4, sigma_t=sigma_t, top_m=top_m,
                                                   sigma_d=sigma_d)
    t = lockstep(w, 2, seed=61, with_kv=False, top_p=top_p,
                 tokens_fn=_nucleus_tokens(w, top_p, 1.0, 61))
    print(f"sigma={sigma_t} top_p={top_p}: draws={t.draws} flagged={t.flagged} "
          f"mismatched={t.mismatched}")
    assert t.rate_ok()


@pytest.mark.parametrize("dtype,V", [("f32", 600_001), ("bf16", 1_100_000)])
def test_step_ex_top_p_long_rows(dtype, V):
    """Rows long enough that a bonus row's runs span several warp reads, and
    fp32 keys that take all three radix digits."""
    w = WORKLOADS["single_prompt_v32000"].with_(B=1, N=2, K=2, V=V, dtype=dtype)
    t = lockstep(w, 1, seed=41, with_kv=False, top_p=0.85,
                 tokens_fn=_nucleus_tokens(w, 0.85, 1.0, 41))
    print(f"{dtype} V={V}: draws={t.draws} flagged={t.flagged} mismatched={t.mismatched}")


def test_step_ex_top_p_tied_logits():
    """Logits rounded to multiples of 1/4, so that the nucleus boundary cuts
    through large groups of equal logits (kept or dropped together)."""
    w = WORKLOADS["single_prompt_v32000"].with_(B=2)
    nucleus_fn = _nucleus_tokens(w, 0.7, 1.0, 43)

    def fn(inp, step):
        for key in ("target", "draft"):
            inp[key].copy_((inp[key].float() * 4).round() / 4)
        nucleus_fn(inp, step)
    t = lockstep(w, 3, seed=43, with_kv=True, top_p=0.7, tokens_fn=fn)
    print(f"tied: draws={t.draws} flagged={t.flagged} mismatched={t.mismatched}")


@pytest.mark.parametrize("top_p", [0.5, 0.9])
def test_step_ex_top_p_threshold_in_a_huge_tie_group(top_p):
    """Two-valued logits (0 and 3): the threshold value is shared by thousands
    of tokens, more than the threshold bin's shared-memory list holds, so the
    rows take the exact radix select over the whole row."""
    w = WORKLOADS["single_prompt_v32000"].with_(B=1, N=4)
    nucleus_fn = _nucleus_tokens(w, top_p, 1.0, 47)

    def fn(inp, step):
        for key in ("target", "draft"):
            inp[key].copy_(torch.where(inp[key].float() > 3.0, 3.0, 0.0))
        nucleus_fn(inp, step)
    t = lockstep(w, 2, seed=47, with_kv=False, top_p=top_p, tokens_fn=fn)
    print(f"two-valued top_p={top_p}: draws={t.draws} flagged={t.flagged} mismatched={t.mismatched}")


@pytest.mark.parametrize("V,dtype", [(1, "f32"), (2, "bf16"), (37, "f32"), (9, "bf16")])
def test_step_ex_top_p_tiny_and_ragged_vocab(V, dtype):
    """Rows of a handful of logits, none a whole 16-byte group: the scalar
    loads, padding and one-group rows of the nucleus kernel."""
    w = Workload(f"topp_{V}", B=2, N=4, K=2, V=V, dtype=dtype, sigma_t=2.0, top_m=min(2, V),
                 sigma_d=1.0, steps=3, prefix=5, block_size=4)
    t = lockstep(w, 3, seed=53, with_kv=True, top_p=0.7,
                 tokens_fn=_nucleus_tokens(w, 0.7, 1.0, 53))
    print(f"top-p V={V} {dtype}: draws={t.draws} flagged={t.flagged} mismatched={t.mismatched}")


def test_step_ex_top_p_draft_outside_nucleus_is_reported():
    w = WORKLOADS["tiny_v64"].with_(B=1)
    inp = make_step_inputs(w, 3, device="cuda")
    d = to_numpy_logits(inp["draft"])[0, 0, 0].astype(np.float64)
    kept, _, _ = osmc.nucleus(d, 0.3)
    inp["draft_tokens"][0, 0, 0] = int(np.flatnonzero(~kept)[0])
    r = StepRunner(w, seed=3, with_kv=False, temperature=1.0)
    r.run(inp, 0, top_p=0.3)
    torch.cuda.synchronize()
    assert "bad_token" in smcsd.status_names(r.status())


# ---------------------------------------------------------------------------
# sps_verify under temperature and top-p
# ---------------------------------------------------------------------------
def _sps_nucleus_tokens(w, top_p, temperature, seed):
    """Drafted tokens drawn from each draft row's tempered nucleus (oracle,
    CPU): inputs that a top-p draft could have produced."""
    rng = np.random.default_rng(seed)
    s = osmc.temperature_scale(temperature)

    def fn(inp, step):
        d = to_numpy_logits(inp["draft"])
        toks = np.zeros((w.B, 1, w.K), dtype=np.int32)
        for b in range(w.B):
            rows = osmc.widen(d[b, 0], w.dtype) * s
            for k in range(w.K):
                kept, _, _ = osmc.nucleus(rows[k], top_p)
                pk = np.where(kept, np.exp(rows[k] - rows[k][kept].max()), 0.0)
                toks[b, 0, k] = rng.choice(len(pk), p=pk / pk.sum())
        inp["draft_tokens"].copy_(torch.from_numpy(toks).to(inp["draft_tokens"].device))
    return fn


@pytest.mark.parametrize("V,dtype,B,K,temperature,top_p", [
    (64, "f32", 128, 3, 0.6, 1.0), (32000, "bf16", 32, 4, 1.3, 1.0),
    (64, "f32", 128, 3, 1.0, 0.8), (32000, "bf16", 32, 4, 0.8, 0.9),
    (1001, "bf16", 48, 2, 0.7, 0.95)])
def test_sps_verify_ex_matches_oracle(V, dtype, B, K, temperature, top_p):
    w = Workload("sps_ex", B=B, N=1, K=K, V=V, dtype=dtype, sigma_t=3.0 if V > 64 else 2.0,
                 top_m=50 if V > 64 else 0, sigma_d=1.0, steps=1)
    fn = _sps_nucleus_tokens(w, top_p, temperature, 17) if top_p < 1.0 else None
    t, ref, g_n = sps_lockstep(w, seed=6, step=2, temperature=temperature, top_p=top_p,
                               tokens_fn=fn)
    print(f"sps_ex V={V} T={temperature} top_p={top_p}: {t.summary()}")
    assert (ref["n_emitted"] < K + 1).any(), "no rejection exercised"
    assert t.rate_ok()


def test_sps_verify_ex_draft_outside_nucleus_is_reported():
    w = Workload("sps_bad", B=4, N=1, K=2, V=64, dtype="f32", sigma_t=2.0, top_m=0,
                 sigma_d=1.0, steps=1)
    inp = make_step_inputs(w, 8, device="cuda")
    d = to_numpy_logits(inp["draft"])[0, 0, 0].astype(np.float64)
    kept, _, _ = osmc.nucleus(d, 0.3)
    inp["draft_tokens"][0, 0, 0] = int(np.flatnonzero(~kept)[0])
    params = smcsd.make_params(4, 1, 2, 64, "f32", 1.0, 0.5, 8, 0)
    ws = smcsd.alloc_workspace(params)
    tok = torch.empty(4 * 3, dtype=torch.int32, device="cuda")
    n = torch.empty(4, dtype=torch.int32, device="cuda")
    smcsd.sps_verify_ex(params, inp["target"], inp["draft"], inp["draft_tokens"], tok, n, ws,
                        top_p=0.3)
    torch.cuda.synchronize()
    assert "bad_token" in smcsd.status_names(smcsd.smc_device_status(ws, clear=True))
