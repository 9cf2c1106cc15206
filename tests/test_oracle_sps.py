"""Pins of the oracle's speculative-sampling verify (CPU only).

Theorem 1 of speculative sampling: every emitted token follows the target
distribution of its position.  The stopping law follows from the acceptance
rule: position k accepts with probability beta_k = sum_v min(p_k(v), q_k(v)).
"""
import numpy as np
import pytest
from scipy.special import logsumexp
from scipy.stats import chisquare

from oracle import sps, smc

V, K = 8, 3
GRID = (np.arange(2 ** 16) + 0.5) / 2 ** 16   # midpoints of a fine u lattice


def _rows(seed):
    rng = np.random.default_rng(seed)
    target = rng.normal(0, 1.5, (K + 1, V))
    draft = target[:K] + rng.normal(0, 1.0, (K, V))
    p = np.exp(target - logsumexp(target, axis=1, keepdims=True))
    q = np.exp(draft - logsumexp(draft, axis=1, keepdims=True))
    return target, draft, p, q


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_theorem1_each_position_follows_target(seed):
    """Enumerate drafted tokens exactly; integrate each uniform over a lattice."""
    target, draft, p, q = _rows(seed)
    for k in range(K):
        res_tok, _ = smc.inverse_cdf(sps.residual_weights(target[k], draft[k]), GRID)
        res_law = np.bincount(res_tok, minlength=V) / len(GRID)
        law = np.zeros(V)
        for x in range(V):
            acc = np.mean(GRID < sps.accept_ratio(target[k], draft[k], x))
            law[x] += q[k, x] * acc
            law += q[k, x] * (1 - acc) * res_law
        assert np.abs(law - p[k]).max() < 4 * V / len(GRID)
    bonus_tok, _ = smc.inverse_cdf(smc.bonus_weights(target[K], 1.0), GRID)
    assert np.abs(np.bincount(bonus_tok, minlength=V) / len(GRID) - p[K]).max() < 2 / len(GRID)


def test_verify_one_control_flow():
    target, draft, p, q = _rows(3)
    x = np.array([1, 2, 3])
    ones = [1 - 2 ** -24] * K
    zeros = [0.0] * K
    # u = 0 accepts every drafted token (ratio > 0): K+1 tokens, last from the bonus row
    out, _, _ = sps.verify_one(target, draft, x, zeros, zeros, 0.0)
    assert out[:K] == list(x) and len(out) == K + 1
    assert out[K] == smc.inverse_cdf(smc.bonus_weights(target[K], 1.0), 0.0)[0]
    # u -> 1 rejects the first drafted token whose ratio is below 1
    ratios = [sps.accept_ratio(target[k], draft[k], x[k]) for k in range(K)]
    out, _, _ = sps.verify_one(target, draft, x, ones, [0.5] * K, 0.0)
    j = next((k for k in range(K) if ratios[k] < 1 - 2 ** -24), None)
    if j is None:
        assert len(out) == K + 1
    else:
        assert out[:j] == list(x[:j]) and len(out) == j + 1
        assert out[j] == smc.inverse_cdf(sps.residual_weights(target[j], draft[j]), 0.5)[0]


def test_residual_falls_back_to_target_when_empty():
    row = np.random.default_rng(0).normal(size=V)
    w = sps.residual_weights(row, row.copy())
    assert np.allclose(w, np.exp(row - logsumexp(row)))


def test_philox_driven_verify_matches_laws():
    """3*10^4 prompts with drafts x ~ q: first-token law = p_0, stopping law closed form."""
    target, draft, p, q = _rows(4)
    n_prompts = 30000
    rng = np.random.default_rng(99)
    toks = np.stack([rng.choice(V, size=n_prompts, p=q[k]) for k in range(K)], axis=1)
    t = np.broadcast_to(target, (n_prompts, K + 1, V))
    d = np.broadcast_to(draft, (n_prompts, K, V))
    out = sps.sps_verify(t, d, toks, seed=5, step=2)
    first = out["tokens_out"][:, 0]
    counts = np.bincount(first, minlength=V)
    assert chisquare(counts, p[0] * n_prompts).pvalue > 1e-4
    beta = np.minimum(p[:K], q).sum(axis=1)
    law_n = [np.prod(beta[:j]) * (1 - beta[j]) for j in range(K)] + [np.prod(beta)]
    obs_n = np.bincount(out["n_emitted"] - 1, minlength=K + 1)
    assert chisquare(obs_n, np.array(law_n) * n_prompts).pvalue > 1e-4
    # padding past the emitted tokens
    for b in range(200):
        assert (out["tokens_out"][b, out["n_emitted"][b]:] == -1).all()
