"""System-level pin of the oracle's SMC-SD step on an enumerable bigram model.

"Faster LLM Inference via Sequential Monte Carlo" (section 3, theoretical
contributions) states that SMC-SD is an approximate sampler whose L1 bias falls
as O(1/sqrt(N)) and whose L2 bias and MSE fall as O(1/N), and that the same
machinery samples unnormalised targets such as p^alpha (power sampling).

Here the target and draft are bigram models over V=6 tokens, so the exact law
of a 6-token continuation, proportional to prod_t P(y_t | y_{t-1})^alpha, can
be enumerated.  Two SMC-SD steps with K=2 drafted tokens (3 emitted tokens per
step) are run with the oracle for N particles; the weighted particle estimate
of E[f] must converge to the exact value with an error slope near -1/2 in
log-log.  The estimate is the pair of marginal laws of the 3rd and the 6th
token (the bonus token of each step), and its error is the L1 distance to
the exact marginals.  Planting a wrong weight (on the CPU, in the oracle) must break it.
"""
import itertools

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle.smc as osmc

V, K, STEPS, CTX0 = 6, 2, 2, 0
LENGTH = STEPS * (K + 1)


def _models(seed=0):
    rng = np.random.default_rng(seed)
    lp = rng.normal(0, 1.5, (V, V))
    lq = lp + rng.normal(0, 1.0, (V, V))
    logp = lp - logsumexp(lp, axis=1, keepdims=True)
    logq = lq - logsumexp(lq, axis=1, keepdims=True)
    return logp, logq


def _f(seqs):
    """One-hots of y_3 and of y_6 side by side: two 6-cell marginal laws."""
    eye = np.eye(V)
    return np.concatenate([eye[seqs[..., K]], eye[seqs[..., -1]]], axis=-1)


def _exact(logp, alpha):
    seqs = np.array(list(itertools.product(range(V), repeat=LENGTH)))
    prev = np.concatenate([np.full((len(seqs), 1), CTX0), seqs[:, :-1]], axis=1)
    logw = alpha * logp[prev, seqs].sum(axis=1)
    w = np.exp(logw - logsumexp(logw))
    return np.sum(w[:, None] * _f(seqs), axis=0)


def _run_smc(logp, logq, alpha, n_part, runs, seed):
    rng = np.random.default_rng(seed)
    seqs = np.zeros((runs, n_part, 0), dtype=np.int64)
    ctx = np.full((runs, n_part), CTX0)
    lw = np.zeros((runs, n_part))
    for step in range(STEPS):
        x = np.zeros((runs, n_part, K), dtype=np.int64)
        c = ctx.copy()
        for k in range(K):
            cum = np.cumsum(np.exp(logq[c]), axis=-1)
            x[:, :, k] = np.minimum((cum < rng.random((runs, n_part, 1))).sum(-1), V - 1)
            c = x[:, :, k]
        prevs = np.concatenate([ctx[..., None], x], axis=-1)  # contexts of rows 0..K
        target = logp[prevs]                                   # [runs, N, K+1, V]
        draft = logq[prevs[..., :K]]                           # [runs, N, K, V]
        out = osmc.smc_step(target, draft, x, lw, alpha=alpha, ess_frac=0.5,
                            seed=seed, step=step)
        a = out["ancestors"]
        seqs = np.concatenate([np.take_along_axis(seqs, a[..., None], axis=1),
                               out["tokens_out"]], axis=-1)
        ctx = seqs[:, :, -1]
        lw = out["log_weights"]
    w = np.exp(lw - logsumexp(lw, axis=1, keepdims=True))
    return np.sum(w[..., None] * _f(seqs), axis=1)


def _errors(alpha, ns, runs=64, seed=1):
    logp, logq = _models()
    truth = _exact(logp, alpha)
    # L1 distance between the weighted-particle law and the exact law, per run
    return np.array([np.mean(np.abs(_run_smc(logp, logq, alpha, n, runs, seed + n)
                                    - truth).sum(axis=-1)) for n in ns])


def _bias(alpha, n_part, runs=64, seed=3):
    """L1 distance between the run-averaged estimate and the exact law."""
    logp, logq = _models()
    est = _run_smc(logp, logq, alpha, n_part, runs, seed)
    return float(np.abs(est.mean(axis=0) - _exact(logp, alpha)).sum())


NS = (4, 16, 64, 256)


@pytest.mark.parametrize("alpha", [1.0, 4.0])
def test_weighted_particles_converge_at_root_n(alpha):
    err = _errors(alpha, NS)
    slope = np.polyfit(np.log(NS), np.log(err), 1)[0]
    assert -0.8 < slope < -0.3, (slope, err)
    assert err[-1] < 0.7


def test_planted_wrong_bonus_weight_is_detected(monkeypatch):
    """Dropping the power-sampling bonus term leaves a bias the pin catches."""
    good = _bias(4.0, 256)
    orig = osmc.score_particle

    def no_bonus_term(target_rows, draft_rows, tokens, alpha):
        s = orig(target_rows, draft_rows, tokens, alpha)
        s["delta"] -= s["lse_alpha"] - alpha * s["lse_p"][-1]
        return s

    monkeypatch.setattr(osmc, "score_particle", no_bonus_term)
    bad = _bias(4.0, 256)
    assert bad > 3 * good, (good, bad)


def test_planted_swapped_ratio_is_detected(monkeypatch):
    """Using q/p instead of p/q as the importance ratio is caught."""
    good = _bias(1.0, 256)
    orig = osmc.score_particle

    def swapped(target_rows, draft_rows, tokens, alpha):
        s = orig(target_rows, draft_rows, tokens, alpha)
        s["delta"] = -s["delta"]
        return s

    monkeypatch.setattr(osmc, "score_particle", swapped)
    bad = _bias(1.0, 256)
    assert bad > 3 * good, (good, bad)
