"""Pins of the oracle's reweighting, ESS, systematic resampling and emission (CPU)."""
import itertools

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import smc, philox
from oracle.errors import OracleError, DEV_ALL_ZERO_WEIGHT, DEV_BAD_TOKEN


def _rows(rng, n_rows, v, sigma=2.0):
    return rng.normal(0, sigma, (n_rows, v))


def test_draft_equal_target_gives_zero_increment_and_no_resample():
    rng = np.random.default_rng(0)
    big_b, n, k, v = 2, 8, 3, 64
    target = rng.normal(0, 2, (big_b, n, k + 1, v))
    draft = target[:, :, :k].copy()
    toks = rng.integers(0, v, (big_b, n, k))
    lw = np.zeros((big_b, n))
    out = smc.smc_step(target, draft, toks, lw, alpha=1.0, ess_frac=0.5, seed=0, step=0)
    assert np.array_equal(out["delta"], np.zeros((big_b, n)))
    assert np.allclose(out["ess"], n, rtol=0, atol=1e-12)
    assert not out["resampled"].any()
    assert np.array_equal(out["ancestors"], np.tile(np.arange(n), (big_b, 1)))
    assert np.array_equal(out["tokens_out"][:, :, :k], toks)
    assert np.array_equal(out["tokens_out"][:, :, k], out["bonus"])


@pytest.mark.parametrize("alpha", [1.0, 4.0, 0.5])
def test_importance_weight_expectation_closed_form(alpha):
    """E_q[exp(delta)] = prod_{k<=K} sum_v p_k(v)^alpha (= 1 when alpha = 1).

    Enumerates every draft x in V^K with probability prod q_k(x_k); catches a
    swapped p/q, a wrong sign, a dropped alpha or a wrong bonus term.
    """
    rng = np.random.default_rng(int(alpha * 7))
    k, v = 3, 5
    target = _rows(rng, k + 1, v)
    draft = _rows(rng, k, v)
    logq = draft - logsumexp(draft, axis=1, keepdims=True)
    total = 0.0
    for x in itertools.product(range(v), repeat=k):
        s = smc.score_particle(target, draft, np.array(x), alpha)
        total += np.exp(sum(logq[i, x[i]] for i in range(k)) + s["delta"])
    logp = target - logsumexp(target, axis=1, keepdims=True)
    expect = np.prod(np.exp(logsumexp(alpha * logp, axis=1)))
    assert abs(total - expect) < 1e-12 * expect


def test_score_rejects_bad_token():
    rng = np.random.default_rng(1)
    with pytest.raises(OracleError) as e:
        smc.score_particle(_rows(rng, 3, 8), _rows(rng, 2, 8), np.array([1, 8]), 1.0)
    assert e.value.kind == DEV_BAD_TOKEN


def test_normalise_invariants():
    rng = np.random.default_rng(2)
    for _ in range(200):
        n = int(rng.integers(1, 65))
        lw = rng.normal(0, rng.uniform(0.01, 30), n)
        if rng.random() < 0.2:
            lw[rng.integers(0, n, max(1, n // 3))] = -np.inf
            lw[0] = 0.0
        w, ess = smc.normalise(lw)
        assert abs(w.sum() - 1) < 1e-12
        assert 1 - 1e-12 <= ess <= n + 1e-9
    w, ess = smc.normalise(np.full(16, -3.5))
    assert abs(ess - 16) < 1e-12
    w, ess = smc.normalise(np.array([0.0, -np.inf, -np.inf]))
    assert ess == 1.0 and w[0] == 1.0


def test_normalise_rejects_all_zero_weights():
    with pytest.raises(OracleError) as e:
        smc.normalise(np.full(4, -np.inf))
    assert e.value.kind == DEV_ALL_ZERO_WEIGHT


def test_systematic_offspring_counts_are_floor_or_ceil():
    rng = np.random.default_rng(3)
    for _ in range(500):
        n = int(rng.integers(1, 65))
        w = rng.dirichlet(np.full(n, rng.uniform(0.05, 3)))
        u0 = rng.random()
        a, _ = smc.systematic_resample(w, u0)
        assert np.all(np.diff(a) >= 0) and a.min() >= 0 and a.max() < n
        counts = np.bincount(a, minlength=n)
        assert np.all(counts >= np.floor(n * w - 1e-9))
        assert np.all(counts <= np.ceil(n * w + 1e-9))
        assert counts.sum() == n


def test_systematic_expected_offspring_is_n_w():
    """Averaged over u0 on a fine lattice, offspring counts equal N*w."""
    rng = np.random.default_rng(4)
    n = 7
    w = rng.dirichlet(np.ones(n))
    grid = (np.arange(4096) + 0.5) / 4096
    mean = np.mean([np.bincount(smc.systematic_resample(w, u)[0], minlength=n)
                    for u in grid], axis=0)
    assert np.allclose(mean, n * w, atol=n / 4096 * 2)


def test_resample_threshold_is_strict_and_resets_weights():
    n = 4
    # weights 1/2, 1/6, 1/6, 1/6: ESS = 1 / (1/4 + 3/36) = 3
    lw = np.log(np.array([3.0, 1.0, 1.0, 1.0]))
    r = smc.resample_prompt(lw, 0.74, seed=0, step=0, b=0)
    assert abs(r["ess"] - 3.0) < 1e-12 and not r["resampled"]
    assert np.array_equal(r["log_weights_out"], lw)
    # ESS exactly at the threshold: equal weights give ESS = N, tau = 1 keeps them
    r = smc.resample_prompt(np.zeros(8), 1.0, seed=0, step=0, b=0)
    assert abs(r["ess"] - 8) < 1e-12
    r = smc.resample_prompt(lw, 0.76, seed=0, step=0, b=0)
    assert r["resampled"] and np.array_equal(r["log_weights_out"], np.zeros(n))
    u0 = philox.uniform(0, 0, 0, 0, philox.RESAMPLE)
    assert np.array_equal(r["ancestors"], smc.systematic_resample(r["weights"], u0)[0])


def test_step_emits_k_plus_one_tokens_of_the_ancestor():
    rng = np.random.default_rng(5)
    big_b, n, k, v = 3, 6, 4, 32
    target = rng.normal(0, 3, (big_b, n, k + 1, v))
    draft = target[:, :, :k] + rng.normal(0, 2, (big_b, n, k, v))
    toks = rng.integers(0, v, (big_b, n, k))
    lw = rng.normal(0, 3, (big_b, n))
    out = smc.smc_step(target, draft, toks, lw, alpha=1.0, ess_frac=1.0, seed=9, step=4)
    assert out["resampled"].all()  # ESS < N whenever weights are unequal
    assert out["tokens_out"].shape == (big_b, n, k + 1)
    for b in range(big_b):
        for i in range(n):
            a = out["ancestors"][b, i]
            assert list(out["tokens_out"][b, i]) == list(toks[b, a]) + [out["bonus"][b, a]]
    assert np.array_equal(out["log_weights"], np.zeros((big_b, n)))
    assert np.allclose(out["log_weights_pre"], lw + out["delta"])


def test_prompt_offset_slices_equal_the_whole_batch():
    """The oracle on a batch equals the oracle on its prompt slices with
    prompt_offset set, for the step, the verify and the draft sampler: only
    the random streams depend on a prompt's number, and the offset keeps them."""
    from smc_speculative_decoding_gb300.workloads import Workload, make_step_inputs, \
        to_numpy_logits
    from oracle import sps as osps
    w = Workload("slices", B=5, N=3, K=2, V=40, dtype="f32", sigma_t=2.0, top_m=3,
                 sigma_d=1.5)
    inp = make_step_inputs(w, 9)
    t, d = to_numpy_logits(inp["target"]), to_numpy_logits(inp["draft"])
    x = inp["draft_tokens"].numpy().astype(np.int64)
    lw = np.random.default_rng(2).normal(0, 1, (w.B, w.N))
    whole = smc.smc_step(t, d, x, lw, ess_frac=0.9, seed=4, step=3)
    for b0, b1 in ((0, 2), (2, 3), (3, 5)):
        part = smc.smc_step(t[b0:b1], d[b0:b1], x[b0:b1], lw[b0:b1], ess_frac=0.9, seed=4,
                            step=3, prompt_offset=b0)
        for key in ("bonus", "ancestors", "tokens_out", "ess", "resampled"):
            assert np.array_equal(part[key], whole[key][b0:b1]), key
    assert whole["resampled"].any() and not whole["resampled"].all()
    one = t[:, 0]  # [B, K+1, V] as one-particle prompts
    sw = osps.sps_verify(one, d[:, 0], x[:, 0], seed=4, step=3)
    sp = osps.sps_verify(one[1:4], d[1:4, 0], x[1:4, 0], seed=4, step=3, prompt_offset=1)
    assert np.array_equal(sp["tokens_out"], sw["tokens_out"][1:4])
    dw, _ = smc.draft_sample(d[:, :, 0], 1, seed=4, step=3)
    dp, _ = smc.draft_sample(d[2:, :, 0], 1, seed=4, step=3, prompt_offset=2)
    assert np.array_equal(dp, dw[2:])
    # a wrong offset changes the draws
    moved = smc.smc_step(t[2:5], d[2:5], x[2:5], lw[2:5], ess_frac=0.9, seed=4, step=3)
    assert not np.array_equal(moved["bonus"], whole["bonus"][2:5])
