"""Pins of the oracle's per-row reductions and samplers (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest
import torch
from scipy.special import logsumexp
from scipy.stats import chisquare

from oracle import smc, philox
from oracle.errors import OracleError, DEV_NONFINITE, DEV_EMPTY_ROW


def test_widen_bf16_matches_torch_on_every_pattern():
    bits = np.arange(2 ** 16, dtype=np.uint16)
    with np.errstate(invalid="ignore"):  # the NaN patterns, signalling ones included
        ours = smc.widen(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[np.isinf(ref)], ref[np.isinf(ref)])


def test_widen_f32_exact():
    x = np.random.default_rng(0).normal(size=1000).astype(np.float32)
    assert np.array_equal(smc.widen(x, "f32"), x.astype(np.float64))


@pytest.mark.parametrize("v", [1, 7, 64, 32000])
def test_row_logsumexp_matches_scipy(v):
    rng = np.random.default_rng(v)
    row = rng.normal(0, 3, v)
    if v > 4:
        row[rng.integers(0, v, v // 4)] = -np.inf  # masked tokens are allowed
    assert abs(smc.row_logsumexp(row) - logsumexp(row)) < 1e-12 * max(1, abs(logsumexp(row)))


def test_row_logsumexp_shift_invariance_and_uniform_closed_form():
    row = np.zeros(1000)
    assert abs(smc.row_logsumexp(row) - np.log(1000)) < 1e-13
    r = np.random.default_rng(3).normal(size=50)
    assert abs(smc.row_logsumexp(r + 123.25) - (smc.row_logsumexp(r) + 123.25)) < 1e-12


@pytest.mark.parametrize("bad,kind", [(np.nan, DEV_NONFINITE), (np.inf, DEV_NONFINITE)])
def test_row_logsumexp_rejects_nonfinite(bad, kind):
    row = np.zeros(10)
    row[4] = bad
    with pytest.raises(OracleError) as e:
        smc.row_logsumexp(row)
    assert e.value.kind == kind


def test_row_logsumexp_rejects_empty_row():
    with pytest.raises(OracleError) as e:
        smc.row_logsumexp(np.full(5, -np.inf))
    assert e.value.kind == DEV_EMPTY_ROW


def _first_exceeding_exact(weights, k):
    """Exact rational inverse CDF for u = k/2^24: first v with C_v > u*S."""
    u = Fraction(k, 2 ** 24)
    total = sum(Fraction(w) for w in weights)
    acc = Fraction(0)
    for v, w in enumerate(weights):
        acc += Fraction(w)
        if acc > u * total:
            return v
    raise AssertionError("u >= 1")


def test_inverse_cdf_matches_exact_rational_arithmetic():
    rng = np.random.default_rng(5)
    for trial in range(40):
        v = int(rng.integers(1, 9))
        weights = rng.integers(0, 6, v).astype(np.float64)
        if weights.sum() == 0:
            weights[-1] = 1.0
        for k in rng.integers(0, 2 ** 24, 50):
            got, _ = smc.inverse_cdf(weights, k / 2 ** 24)
            assert got == _first_exceeding_exact(weights, int(k))


def test_inverse_cdf_skips_zero_weight_tokens_and_edges():
    w = np.array([0.0, 1.0, 0.0, 0.0, 3.0, 0.0])
    assert smc.inverse_cdf(w, 0.0)[0] == 1
    assert smc.inverse_cdf(w, 0.2499)[0] == 1
    assert smc.inverse_cdf(w, 0.25)[0] == 4  # strict: C_v must exceed u*S
    assert smc.inverse_cdf(w, 1 - 2 ** -24)[0] == 4


@pytest.mark.parametrize("alpha", [1.0, 4.0, 0.5])
def test_bonus_sampler_histogram_matches_softmax(alpha):
    """10^6 Philox-keyed draws from softmax(alpha*l) on V=64 pass chi-square."""
    rng = np.random.default_rng(int(alpha * 10))
    row = rng.normal(0, 2, 64)
    p = np.exp(alpha * row - logsumexp(alpha * row))
    u = philox.uniform_np(0, 0, np.arange(10 ** 6), 3, philox.BONUS)
    toks, _ = smc.inverse_cdf(smc.bonus_weights(row, alpha), u)
    counts = np.bincount(toks, minlength=64)
    keep = p * 1e6 > 20
    obs, exp = counts[keep], p[keep] * 1e6
    if (~keep).any():
        obs = np.append(obs, counts[~keep].sum())
        exp = np.append(exp, p[~keep].sum() * 1e6)
    exp *= obs.sum() / exp.sum()
    assert chisquare(obs, exp).pvalue > 1e-4


def test_near_tie_margin_definition():
    w = np.array([1.0, 1.0, 2.0])
    _, m = smc.inverse_cdf(w, 0.5 + 1e-7)  # just above the boundary C_1 = 2 of S = 4
    assert abs(m - 1e-7) < 1e-12
