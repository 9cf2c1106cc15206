"""Pins of the oracle's extensions beyond the basic step (CPU): temperature,
per-particle log-potentials, top-p nuclei, the draft-side sampler and KV-usage
accounting."""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax
from scipy.stats import chisquare

from oracle import smc, kv
from oracle.errors import OracleError, DEV_ALL_ZERO_WEIGHT


def _inputs(rng, big_b=2, n=8, k=3, v=32, sigma=2.0, noise=1.0):
    target = rng.normal(0, sigma, (big_b, n, k + 1, v))
    draft = target[:, :, :k] + rng.normal(0, noise, (big_b, n, k, v))
    toks = rng.integers(0, v, (big_b, n, k))
    return target, draft, toks


# ---------------------------------------------------------------------------
# temperature
# ---------------------------------------------------------------------------
def test_temperature_divides_the_logits():
    """Logits scaled by 4 at temperature 4 are the logits themselves at
    temperature 1 (1/4 is exact in fp32): every output is identical.  Catches
    a temperature that multiplies instead of dividing."""
    rng = np.random.default_rng(3)
    target, draft, toks = _inputs(rng)
    lw = rng.normal(0, 1, (2, 8))
    plain = smc.smc_step(target, draft, toks, lw, ess_frac=0.9, seed=5, step=2)
    hot = smc.smc_step(4.0 * target, 4.0 * draft, toks, lw, ess_frac=0.9, seed=5, step=2,
                       temperature=4.0)
    for key in ("delta", "ess", "ancestors", "bonus", "tokens_out", "log_weights"):
        assert np.array_equal(plain[key], hot[key]), key


@pytest.mark.parametrize("temperature", [0.5, 2.0])
def test_tempered_weight_increment_closed_form(temperature):
    """delta = sum_k log p_T(x_k) - log q_T(x_k) with p_T = softmax(l / T),
    from scipy's log-softmax of the scaled rows."""
    rng = np.random.default_rng(11)
    target, draft, toks = _inputs(rng, big_b=1, n=4)
    out = smc.smc_step(target, draft, toks, np.zeros((1, 4)), temperature=temperature)
    s = smc.temperature_scale(temperature)
    for n in range(4):
        lp = target[0, n, :3] * s - logsumexp(target[0, n, :3] * s, axis=1, keepdims=True)
        lq = draft[0, n] * s - logsumexp(draft[0, n] * s, axis=1, keepdims=True)
        expect = sum(lp[k, toks[0, n, k]] - lq[k, toks[0, n, k]] for k in range(3))
        assert abs(out["delta"][0, n] - expect) < 1e-12


def test_draft_equal_target_stays_unweighted_at_any_temperature():
    rng = np.random.default_rng(2)
    target, _, toks = _inputs(rng)
    out = smc.smc_step(target, target[:, :, :3].copy(), toks, np.zeros((2, 8)), temperature=0.3)
    assert np.array_equal(out["delta"], np.zeros((2, 8)))
    assert not out["resampled"].any()


def test_temperature_must_be_positive():
    rng = np.random.default_rng(2)
    target, draft, toks = _inputs(rng)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(ValueError):
            smc.smc_step(target, draft, toks, np.zeros((2, 8)), temperature=bad)


# ---------------------------------------------------------------------------
# log-potentials
# ---------------------------------------------------------------------------
def test_constant_potential_changes_no_normalised_quantity():
    rng = np.random.default_rng(4)
    target, draft, toks = _inputs(rng)
    lw = rng.normal(0, 1, (2, 8))
    a = smc.smc_step(target, draft, toks, lw, ess_frac=0.9, seed=1, step=3)
    b = smc.smc_step(target, draft, toks, lw, ess_frac=0.9, seed=1, step=3,
                     log_potential=np.full((2, 8), -7.5))
    assert np.allclose(a["ess"], b["ess"], rtol=1e-12, atol=0)
    assert np.array_equal(a["ancestors"], b["ancestors"])
    assert np.allclose(b["log_weights_pre"] - a["log_weights_pre"], -7.5, atol=1e-12)


def test_potential_alone_sets_the_weights_closed_form():
    """With draft == target the increment is the potential alone, so
    ESS = (sum e^phi)^2 / sum e^(2 phi)."""
    rng = np.random.default_rng(5)
    target, _, toks = _inputs(rng)
    phi = rng.normal(0, 1.5, (2, 8))
    out = smc.smc_step(target, target[:, :, :3].copy(), toks, np.zeros((2, 8)),
                       log_potential=phi, ess_frac=0.0)
    w = np.exp(phi)
    assert np.allclose(out["ess"], w.sum(1) ** 2 / (w ** 2).sum(1), rtol=1e-12, atol=0)


def test_minus_infinity_potential_removes_a_particle():
    """A particle with potential -inf (a violated constraint) weighs 0: it is
    never an ancestor when the prompt resamples."""
    rng = np.random.default_rng(6)
    target, draft, toks = _inputs(rng)
    phi = np.zeros((2, 8))
    phi[:, 0] = -np.inf
    phi[1, 5] = -np.inf
    for step in range(20):
        out = smc.smc_step(target, draft, toks, np.zeros((2, 8)), log_potential=phi,
                           ess_frac=1.01, seed=9, step=step)
        assert out["resampled"].all()
        assert not (out["ancestors"][0] == 0).any()
        assert not np.isin(out["ancestors"][1], [0, 5]).any()


def test_all_minus_infinity_potentials_are_an_error():
    rng = np.random.default_rng(7)
    target, draft, toks = _inputs(rng)
    with pytest.raises(OracleError) as e:
        smc.smc_step(target, draft, toks, np.zeros((2, 8)), log_potential=np.full((2, 8), -np.inf))
    assert e.value.kind == DEV_ALL_ZERO_WEIGHT


# ---------------------------------------------------------------------------
# draft-side sampler
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("alpha", [1.0, 0.5])
def test_draft_sample_follows_the_tempered_softmax(alpha):
    """Over 40000 (seed, step) draws, token counts of one row match
    softmax(alpha * l) by a chi-square test."""
    rng = np.random.default_rng(8)
    v = 12
    row = rng.normal(0, 1.5, v)
    logits = np.broadcast_to(row, (1, 1, v))
    counts = np.zeros(v)
    for seed in range(200):
        for step in range(200):
            t, _ = smc.draft_sample(logits, position=2, alpha=alpha, seed=seed, step=step)
            counts[t[0, 0]] += 1
    p = softmax(alpha * row)
    assert chisquare(counts, p * counts.sum()).pvalue > 1e-4


def test_draft_sample_positions_draw_independently_and_masks_hold():
    """-inf logits are never drawn; different positions use different
    uniforms (so whole-row samples differ across positions)."""
    rng = np.random.default_rng(9)
    draft = rng.normal(0, 1.0, (3, 5, 40))
    draft[:, :, ::3] = -np.inf
    toks = np.stack([smc.draft_sample(draft, position=k, seed=4, step=1)[0] for k in range(4)])
    assert (toks % 3 != 0).all()
    assert not all(np.array_equal(toks[0], toks[k]) for k in range(1, 4))


# ---------------------------------------------------------------------------
# KV usage
# ---------------------------------------------------------------------------
def _state(big_b, n, prefix, bs, t_len, pool):
    tables = np.full((big_b, n, t_len), -1, dtype=np.int64)
    refcount = np.zeros(big_b * pool, dtype=np.int64)
    free_list = np.zeros((big_b, pool), dtype=np.int64)
    free_top = np.zeros(big_b, dtype=np.int64)
    nb = -(-prefix // bs)
    for b in range(big_b):
        tables[b, :, :nb] = np.arange(b * pool, b * pool + nb)
        refcount[b * pool: b * pool + nb] = n
        free = np.arange(b * pool + pool - 1, b * pool + nb - 1, -1)
        free_list[b, :len(free)] = free
        free_top[b] = len(free)
    seq_len = np.full((big_b, n), prefix, dtype=np.int64)
    return tables, seq_len, refcount, free_list, free_top


def test_usage_of_a_shared_prefix():
    tables, seq_len, *_ = _state(2, 8, 40, 16, 10, 81)
    used, unshared = kv.usage(tables, seq_len, 16)
    assert list(used) == [3, 3] and list(unshared) == [24, 24]


def test_usage_counts_the_blocks_with_live_references():
    """After remaps with resampling and appends, used blocks are exactly the
    pool blocks whose reference count is positive."""
    rng = np.random.default_rng(10)
    big_b, n, bs, t_len = 2, 6, 4, 12
    pool = n * t_len + 1
    tables, seq_len, refcount, free_list, free_top = _state(big_b, n, 6, bs, t_len, pool)
    for step in range(5):
        anc = rng.integers(0, n, (big_b, n))
        res = rng.random(big_b) < 0.7
        out = kv.remap_append(tables, seq_len, refcount, free_list, free_top, anc, res, 3, bs,
                              pool)
        assert all(not e for e in out["errors"])
        tables, seq_len, refcount = out["tables"], out["seq_len"], out["refcount"]
        free_list, free_top = out["free_list"], out["free_top"]
        used, unshared = kv.usage(tables, seq_len, bs)
        for b in range(big_b):
            assert used[b] == int((np.asarray(refcount[b * pool:(b + 1) * pool]) > 0).sum())
            assert unshared[b] == sum(-(-int(seq_len[b][i]) // bs) for i in range(n))
            assert used[b] <= unshared[b]


# ---------------------------------------------------------------------------
# top-p (nucleus)
# ---------------------------------------------------------------------------
def _nucleus_by_sorting(row, top_p):
    """Independent restatement: sort tokens by probability, walk down in
    groups of equal logit, keep a group while the mass before it is below
    top_p."""
    pi = softmax(row)
    order = np.argsort(-row, kind="stable")
    kept = np.zeros(len(row), dtype=bool)
    before = 0.0
    i = 0
    while i < len(order):
        j = i
        while j < len(order) and row[order[j]] == row[order[i]]:
            j += 1
        if before >= top_p:
            break
        kept[order[i:j]] = True
        before += pi[order[i:j]].sum()
        i = j
    return kept


@pytest.mark.parametrize("top_p", [0.3, 0.8, 0.95])
def test_nucleus_matches_sorting(top_p):
    rng = np.random.default_rng(int(top_p * 100))
    for _ in range(40):
        row = np.round(rng.normal(0, 2, 50) * 4) / 4  # coarse values: many ties
        kept, log_z, _ = smc.nucleus(row, top_p)
        assert np.array_equal(kept, _nucleus_by_sorting(row, top_p))
        assert abs(log_z - np.log(softmax(row)[kept].sum())) < 1e-12


def test_tiny_top_p_keeps_only_the_most_likely_tokens():
    row = np.array([0.5, 2.0, -1.0, 2.0, 1.9])
    kept, log_z, _ = smc.nucleus(row, 1e-6)
    assert list(np.flatnonzero(kept)) == [1, 3]
    assert abs(log_z - np.log(2 * softmax(row)[1])) < 1e-12


def test_top_p_weight_expectation_closed_form():
    """E_{x ~ q_top}[exp(delta)] = prod_k p_top,k(S_q,k): with both sides
    truncated to nuclei, the weights average to the target nucleus mass that
    the draft's nucleus covers.  Enumerates V^K."""
    import itertools
    rng = np.random.default_rng(12)
    k, v, top_p = 2, 6, 0.8
    target = rng.normal(0, 1.5, (k + 1, v))
    draft = rng.normal(0, 1.5, (k, v))
    total = 0.0
    q_sets = [smc.nucleus(draft[i], top_p)[0] for i in range(k)]
    for x in itertools.product(range(v), repeat=k):
        if not all(q_sets[i][x[i]] for i in range(k)):
            continue
        s = smc.score_particle_topp(target, draft, np.array(x), top_p)
        logq = sum(draft[i, x[i]] - s["lse_q"][i] for i in range(k))
        total += np.exp(logq + s["delta"])
    expect = 1.0
    for i in range(k):
        kept_p, log_zp, _ = smc.nucleus(target[i], top_p)
        pt = np.where(kept_p, softmax(target[i]), 0.0) / np.exp(log_zp)
        expect *= pt[q_sets[i]].sum()
    assert abs(total - expect) < 1e-12


def test_top_p_step_bonus_stays_in_the_nucleus_and_bad_drafts_raise():
    rng = np.random.default_rng(13)
    target, draft, _ = _inputs(rng, big_b=1, n=6, k=2, v=40)
    toks = np.zeros((1, 6, 2), dtype=np.int64)
    for n in range(6):
        for i in range(2):
            toks[0, n, i] = int(np.argmax(draft[0, n, i]))  # always in q's nucleus
    out = smc.smc_step(target, draft, toks, np.zeros((1, 6)), top_p=0.7, seed=3, step=1)
    for n in range(6):
        kept, _, _ = smc.nucleus(target[0, n, 2], 0.7)
        assert kept[out["bonus"][0, n]]
    toks[0, 0, 1] = int(np.argmin(draft[0, 0, 1]))
    with pytest.raises(OracleError):
        smc.smc_step(target, draft, toks, np.zeros((1, 6)), top_p=0.7)


# ---------------------------------------------------------------------------
# speculative-sampling verify under temperature and top-p
# ---------------------------------------------------------------------------
from oracle import sps  # noqa: E402
from oracle.errors import DEV_BAD_TOKEN  # noqa: E402

SPS_GRID = (np.arange(2 ** 16) + 0.5) / 2 ** 16   # midpoints of a fine u lattice


def _tempered_nucleus(row, temperature, top_p):
    """softmax(row / T) restricted to its nucleus (found by sorting) and
    renormalised: an independent restatement."""
    z = row * float(np.float32(1.0) / np.float32(temperature))
    kept = _nucleus_by_sorting(z, top_p)
    p = np.where(kept, softmax(z), 0.0)
    return p / p.sum()


@pytest.mark.parametrize("temperature,top_p", [(0.7, 0.8), (1.5, 0.6), (1.0, 0.95)])
def test_sps_tempered_nucleus_theorem1(temperature, top_p):
    """Every emitted token follows the tempered nucleus of the target.  For
    one position, verify_one_logprobs is run with every drafted token x of
    the draft's nucleus and with uniforms on a lattice: the acceptance rate
    of x and the law of the residual draw give the law of the emitted token,
    sum_x q_top(x) [acc(x) 1{v = x} + (1 - acc(x)) res(v)], which must be
    p_top (Theorem 1 applied to the restricted distributions).  Catches a
    ratio or residual taken on the unrestricted p or q, or a nucleus that is
    not renormalised."""
    rng = np.random.default_rng(int(temperature * 10 + top_p * 100))
    V = 8
    grid = (np.arange(4096) + 0.5) / 4096
    target = np.round(rng.normal(0, 1.5, (2, V)) * 8) / 8
    draft = np.round((target[:1] + rng.normal(0, 1.0, (1, V))) * 8) / 8
    scale = smc.temperature_scale(temperature)
    logp, _ = sps.tempered_logprobs(target, scale, top_p)
    logq, _ = sps.tempered_logprobs(draft, scale, top_p)
    p = _tempered_nucleus(target[0], temperature, top_p)
    q = _tempered_nucleus(draft[0], temperature, top_p)
    assert np.allclose(np.exp(logp[0]), p, atol=1e-12)
    assert np.allclose(np.exp(logq[0]), q, atol=1e-12)

    def run(x, u, u2):
        return sps.verify_one_logprobs(logp, logq, [x], [u], [u2], 0.5)[0]
    law = np.zeros(V)
    res = None
    for x in np.flatnonzero(q > 0):
        acc = np.mean([len(run(x, u, 0.5)) == 2 for u in grid])
        if acc < 1 and res is None:
            u_rej = 1 - 2 ** -24                       # rejects whenever p/q < 1
            res = np.bincount([run(x, u_rej, u2)[0] for u2 in grid], minlength=V) / len(grid)
        law[x] += q[x] * acc
        if acc < 1:
            law += q[x] * (1 - acc) * res
    assert np.abs(law - p).max() < 3 * V / len(grid), (law, p)


def test_sps_temperature_divides_the_logits():
    """Rows scaled by 4 at temperature 4 give exactly the outputs of the
    plain verify on the rows themselves (1/4 is exact in fp32)."""
    rng = np.random.default_rng(11)
    B, K, V = 40, 3, 16
    target = rng.normal(0, 2, (B, K + 1, V))
    draft = target[:, :K] + rng.normal(0, 1, (B, K, V))
    toks = rng.integers(0, V, (B, K))
    plain = sps.sps_verify(target, draft, toks, seed=3, step=4)
    hot = sps.sps_verify(4.0 * target, 4.0 * draft, toks, seed=3, step=4, temperature=4.0)
    assert (plain["n_emitted"] < K + 1).any()
    assert np.array_equal(plain["tokens_out"], hot["tokens_out"])
    assert np.array_equal(plain["n_emitted"], hot["n_emitted"])


def test_sps_top_p_bonus_inside_nucleus_and_bad_draft_raises():
    rng = np.random.default_rng(5)
    B, K, V = 60, 2, 32
    target = rng.normal(0, 2, (B, K + 1, V))
    draft = target[:, :K] + rng.normal(0, 0.3, (B, K, V))
    scale = smc.temperature_scale(1.0)
    # drafted tokens: each draft row's argmax, always inside its nucleus
    toks = draft.argmax(-1)
    out = sps.sps_verify(target, draft, toks, seed=1, step=0, top_p=0.5)
    assert (out["n_emitted"] < K + 1).any() and (out["n_emitted"] == K + 1).any()
    for b in range(B):
        n = out["n_emitted"][b]
        last = out["tokens_out"][b, n - 1]
        # a bonus draw, or a residual draw (zero outside the target's nucleus)
        assert _nucleus_by_sorting(target[b, n - 1] * scale, 0.5)[last]
    bad = toks.copy()
    b0 = 0
    kept_q = _nucleus_by_sorting(draft[b0, 0], 0.5)
    bad[b0, 0] = int(np.flatnonzero(~kept_q)[0])
    with pytest.raises(OracleError) as e:
        sps.sps_verify(target[:1], draft[:1], bad[:1], seed=1, step=0, top_p=0.5)
    assert e.value.kind == DEV_BAD_TOKEN
