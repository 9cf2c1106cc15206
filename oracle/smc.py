"""SMC-SD per-step particle update, written out plainly in fp64 (CPU oracle).

Test infrastructure: part of the CPU oracle (see ``oracle/__init__.py``).

Follows the step as "Faster LLM Inference via Sequential Monte Carlo" states it
(gist.science explainer, zh: section 2 "核心流程" and "系统优化设计"; es:
"Resumen Técnico", section 2 "Metodología: SMC-SD"):

  * Extend: the draft model extends each of N particles by K tokens (input
    here: drafted tokens and the draft logits they were drawn from).
  * Score & Bonus: one batched target pass scores the K drafted tokens of every
    particle and yields one extra bonus token per particle (target row K).
  * Reweight: each particle's importance weight is updated by the ratio of
    target to draft probability of its drafted tokens.
  * Resample: the effective sample size is computed; when it falls below a
    threshold, particles are resampled by weight.  Every step emits exactly
    K+1 tokens per particle; there is no truncation.

The power-sampling generalisation (section 3 "通用性扩展": the target may be an
unnormalised distribution such as p^alpha) enters as ``alpha``.

Readings of steps the pages leave open (each one is listed with its reason in
the design notes of the repository):
  * weight increment: sum_k alpha*log p(x_k) - log q(x_k); for alpha != 1 the
    bonus token, drawn from the locally normalised p^alpha, contributes
    log sum_v p_v^alpha = lse(alpha*l) - alpha*lse(l); for alpha == 1 it
    contributes nothing;
  * ESS = 1 / sum_n w_n^2 over normalised weights; resample iff ESS < tau*N;
  * resampling is systematic, with one uniform per (prompt, step);
  * after resampling all log-weights are reset to 0;
  * the bonus token is sampled per pre-resampling particle and gathered
    through the ancestor indices;
  * sampling is inverse-CDF in vocabulary order: the smallest v whose
    inclusive cumulative weight exceeds u times the total.

Everything is computed in fp64 from exactly widened inputs, one row at a time,
with no blocking or reordering beyond numpy's own reductions.
"""
import numpy as np

from . import philox
from .errors import (OracleError, DEV_BAD_TOKEN, DEV_NONFINITE, DEV_EMPTY_ROW,
                     DEV_ALL_ZERO_WEIGHT)

#: a draw is flagged as a near tie when u*S lies closer than this fraction of
#: S to either edge of the selected cumulative interval
NEAR_TIE = 1e-5


# --------------------------------------------------------------------------
# inputs
# --------------------------------------------------------------------------
def widen(logits, dtype):
    """Widen stored logits exactly to fp64.

    ``dtype`` is "f32" (any float array) or "bf16" (an array of raw uint16
    bfloat16 bit patterns: a bfloat16 is the upper half of an IEEE fp32).
    """
    if dtype == "bf16":
        bits = np.asarray(logits).view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(logits, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# per-row vocabulary reductions (Score & Bonus)
# --------------------------------------------------------------------------
def row_logsumexp(row):
    """log sum_v exp(l_v) of one logit row, with the max taken out first."""
    if np.isnan(row).any() or np.isposinf(row).any():
        raise OracleError(DEV_NONFINITE, "row holds NaN or +inf")
    m = np.max(row)
    if m == -np.inf:
        raise OracleError(DEV_EMPTY_ROW, "every logit of the row is -inf")
    return m + np.log(np.sum(np.exp(row - m)))


def inverse_cdf(weights, u):
    """Inverse-CDF draw in vocabulary order from non-negative ``weights``.

    Returns (v, margin) with v the smallest index whose inclusive cumulative
    weight exceeds u * total, and margin the distance of u * total to the
    nearer edge of v's interval, as a fraction of the total.  ``u`` may be an
    array, in which case both results are arrays.
    """
    c = np.cumsum(weights)
    total = c[-1]
    if not total > 0:
        raise OracleError(DEV_EMPTY_ROW, "no positive weight to sample from")
    u_arr = np.atleast_1d(np.asarray(u, dtype=np.float64))
    target = u_arr * total
    v = np.searchsorted(c, target, side="right")
    # u < 1 keeps target < total, so v < len(c); rounding cannot push it past.
    last = int(np.flatnonzero(weights > 0)[-1])
    v = np.minimum(v, last)
    lo = np.where(v > 0, c[np.maximum(v - 1, 0)], 0.0)
    hi = c[v]
    margin = np.minimum(np.abs(target - lo), np.abs(hi - target)) / total
    if np.ndim(u) == 0:
        return int(v[0]), float(margin[0])
    return v.astype(np.int64), margin


def bonus_weights(row, alpha):
    """Unnormalised softmax(alpha * l) of the bonus row: exp(alpha*(l - max l))."""
    m = np.max(row)
    return np.exp(alpha * (row - m))


# --------------------------------------------------------------------------
# Resample: normalisation, ESS, systematic resampling
# --------------------------------------------------------------------------
def normalise(log_weights):
    """Normalised weights and ESS = 1/sum w^2 of one prompt's N log-weights."""
    lw = np.asarray(log_weights, dtype=np.float64)
    if np.isnan(lw).any() or np.isposinf(lw).any():
        raise OracleError(DEV_NONFINITE, "log-weight is NaN or +inf")
    m = np.max(lw)
    if m == -np.inf:
        raise OracleError(DEV_ALL_ZERO_WEIGHT, "every particle has weight 0")
    big_l = m + np.log(np.sum(np.exp(lw - m)))
    w = np.exp(lw - big_l)
    ess = 1.0 / np.sum(w * w)
    return w, ess


def systematic_resample(w, u0):
    """Ancestors a_i = min{j : C_j > (u0 + i)/N}, C the inclusive prefix of w.

    Returns (ancestors, margins) where margins[i] is the distance of
    (u0 + i)/N to the nearer edge of [C_{a_i - 1}, C_{a_i}).  The ancestor is
    clamped to N-1 should rounding leave (u0 + i)/N at or above C_{N-1}.
    """
    n = len(w)
    c = np.cumsum(w)
    pts = (u0 + np.arange(n, dtype=np.float64)) / n
    a = np.minimum(np.searchsorted(c, pts, side="right"), n - 1)
    lo = np.where(a > 0, c[np.maximum(a - 1, 0)], 0.0)
    hi = c[a]
    margins = np.minimum(np.abs(pts - lo), np.abs(hi - pts))
    return a.astype(np.int64), margins


def resample_prompt(log_weights, ess_frac, seed, step, b):
    """Normalise, compute ESS and, if ESS < ess_frac*N, resample one prompt.

    Returns dict(ancestors, ess, resampled, log_weights_out, margins,
    ess_margin).  Log-weights are reset to 0 after resampling.
    """
    n = len(log_weights)
    w, ess = normalise(log_weights)
    thresh = float(np.float32(ess_frac)) * n
    resampled = bool(ess < thresh)
    if resampled:
        u0 = philox.uniform(seed, step, b, 0, philox.RESAMPLE)
        anc, margins = systematic_resample(w, u0)
        lw_out = np.zeros(n)
    else:
        anc = np.arange(n, dtype=np.int64)
        margins = np.full(n, np.inf)
        lw_out = np.asarray(log_weights, dtype=np.float64).copy()
    return dict(ancestors=anc, ess=ess, resampled=resampled,
                log_weights_out=lw_out, weights=w, margins=margins,
                ess_margin=abs(ess - thresh) / n)


# --------------------------------------------------------------------------
# the whole step
# --------------------------------------------------------------------------
def score_particle(target_rows, draft_rows, tokens, alpha):
    """Row statistics and the weight increment of one particle.

    target_rows: [K+1, V] fp64, draft_rows: [K, V] fp64, tokens: [K] ints.
    Returns dict(lse_p[K+1], g_p[K], lse_q[K], g_q[K], lse_alpha, delta).
    """
    k_drafts = draft_rows.shape[0]
    v_size = target_rows.shape[1]
    lse_p = np.array([row_logsumexp(r) for r in target_rows])
    lse_q = np.array([row_logsumexp(r) for r in draft_rows])
    tokens = np.asarray(tokens, dtype=np.int64)
    if (tokens < 0).any() or (tokens >= v_size).any():
        raise OracleError(DEV_BAD_TOKEN, "drafted token outside [0, V)")
    g_p = target_rows[np.arange(k_drafts), tokens]
    g_q = draft_rows[np.arange(k_drafts), tokens]
    delta = np.sum(alpha * (g_p - lse_p[:k_drafts]) - (g_q - lse_q))
    lse_alpha = row_logsumexp(alpha * target_rows[k_drafts])
    if alpha != 1.0:
        delta += lse_alpha - alpha * lse_p[k_drafts]
    return dict(lse_p=lse_p, g_p=g_p, lse_q=lse_q, g_q=g_q,
                lse_alpha=lse_alpha, delta=delta)


def nucleus(row, top_p, scale=1.0):
    """The top-p (nucleus) set of one row of logits.

    With pi = softmax(scale * row), token v is kept iff the probability mass
    of the tokens strictly more likely than v is below top_p; tokens of equal
    logit are kept or dropped together (so the set does not depend on an
    order among ties).  Returns (kept mask, log of the kept mass, margin): the
    margin is the distance of top_p from the nearest value that mass-above
    takes, so a draw is flagged as a near tie when it is small.
    """
    row = np.asarray(row, dtype=np.float64)
    z = scale * row
    finite = np.isfinite(z)
    m = np.max(z[finite])
    pi = np.where(finite, np.exp(z - m), 0.0)
    pi = pi / np.sum(pi)
    vals, inv = np.unique(row[finite], return_inverse=True)   # distinct logits, ascending
    mass = np.bincount(inv, weights=pi[finite], minlength=len(vals))
    vals, mass = vals[::-1], mass[::-1]                          # descending
    above = np.concatenate([[0.0], np.cumsum(mass)[:-1]])   # mass strictly above each value
    keep_vals = above < top_p
    thresh = vals[keep_vals][-1]
    kept = finite & (row >= thresh)
    margin = float(np.min(np.abs(np.concatenate([above, [np.sum(mass)]]) - top_p)))
    return kept, float(np.log(np.sum(pi[kept]))), margin


def score_particle_topp(target_rows, draft_rows, tokens, top_p):
    """score_particle (alpha = 1) with p and q restricted to their nuclei.

    Rows are the already scaled (tempered) logits.  lse_p / lse_q become the
    log-normalisers of the renormalised nuclei (lse + log kept mass), g_p is
    -inf for a token outside the target's nucleus, and a token outside the
    draft's nucleus raises (bad token).  Also returns the bonus row's kept
    mask and the smallest nucleus margin over the particle's rows.
    """
    k_drafts = draft_rows.shape[0]
    v_size = target_rows.shape[1]
    tokens = np.asarray(tokens, dtype=np.int64)
    if (tokens < 0).any() or (tokens >= v_size).any():
        raise OracleError(DEV_BAD_TOKEN, "drafted token outside [0, V)")
    lse_p = np.zeros(k_drafts + 1)
    lse_q = np.zeros(k_drafts)
    g_p = np.zeros(k_drafts)
    g_q = np.zeros(k_drafts)
    margin = np.inf
    bonus_kept = None
    for k in range(k_drafts + 1):
        kept, log_z, mg = nucleus(target_rows[k], top_p)
        margin = min(margin, mg)
        lse_p[k] = row_logsumexp(target_rows[k]) + log_z
        if k == k_drafts:
            bonus_kept = kept
        else:
            g_p[k] = target_rows[k, tokens[k]] if kept[tokens[k]] else -np.inf
    for k in range(k_drafts):
        kept, log_z, mg = nucleus(draft_rows[k], top_p)
        margin = min(margin, mg)
        if not kept[tokens[k]]:
            raise OracleError(DEV_BAD_TOKEN, "drafted token outside the draft's nucleus")
        lse_q[k] = row_logsumexp(draft_rows[k]) + log_z
        g_q[k] = draft_rows[k, tokens[k]]
    delta = np.sum((g_p - lse_p[:k_drafts]) - (g_q - lse_q))
    return dict(lse_p=lse_p, g_p=g_p, lse_q=lse_q, g_q=g_q, lse_alpha=lse_p[k_drafts],
                delta=delta, bonus_kept=bonus_kept, margin=margin)


def temperature_scale(temperature):
    """The multiplier 1/T that a temperature T applies to every logit.

    The pages fix no precision for it; it is taken as the fp32 rounding of
    1/T computed from the fp32 value of T, the value a caller passing T as a
    float arrives at, and is then applied exactly (in fp64) to the logits.
    """
    t32 = np.float32(temperature)
    if not (np.isfinite(t32) and t32 > 0):
        raise ValueError("temperature must be positive and finite")
    return float(np.float32(np.float32(1.0) / t32))


def effective_alpha(alpha, temperature=1.0):
    """The exponent of the bonus distribution softmax(alpha * l / T), taken
    as the fp32 product of alpha and the temperature's multiplier."""
    return float(np.float32(np.float32(alpha) * np.float32(temperature_scale(temperature))))


def smc_step(target, draft, draft_tokens, log_weights, *, alpha=1.0,
             ess_frac=0.5, seed=0, step=0, dtype=None, temperature=1.0,
             log_potential=None, top_p=1.0, prompt_offset=0):
    """One SMC-SD step over B prompts x N particles (no KV state).

    target: [B, N, K+1, V], draft: [B, N, K, V], either already fp64 or, when
    ``dtype`` is given, stored logits that are widened one particle at a time
    (see ``widen``); draft_tokens: [B, N, K] ints, log_weights: [B, N].

    temperature T: p and q are softmax(l / T) before they are scored or
    sampled; the drafted tokens are taken to come from the tempered draft.
    log_potential: optional [B, N] per-particle log-potential increment of
    this step (for example a log reward ratio, or -inf for a particle that
    breaks a constraint), added to the weight increment.  Both settings are
    extensions the pages name without fixing (the SMC page's section 3 on
    unnormalised targets such as rewards and constraints; the SpS notes'
    evaluation at nucleus and temperature settings).
    top_p < 1 (alpha must be 1): p and q are each restricted to their nucleus
    (see ``nucleus``) and renormalised, after the temperature; the bonus is
    drawn from the target's nucleus.  A drafted token outside the draft's
    nucleus could not have been drawn and is an error (bad token); one
    outside the target's nucleus gives the particle weight 0.  The returned
    dict then also holds topp_margin[B, N]: the smallest nucleus margin of the
    particle's rows.

    prompt_offset: the batch is prompts prompt_offset .. prompt_offset+B-1
    of a larger one; only the random streams depend on it (prompt b draws
    with the stream numbers of prompt prompt_offset + b), so a batch can be
    checked in slices.

    Returns a dict with
      delta[B,N], log_weights_pre[B,N] (after reweighting), log_weights[B,N]
      (after the optional reset), ess[B], resampled[B], ancestors[B,N],
      bonus[B,N] (per pre-resampling particle), tokens_out[B,N,K+1],
      bonus_margin[B,N], resample_margin[B,N], ess_margin[B], and the row
      statistics lse_p, g_p, lse_q, g_q, lse_alpha.
    """
    alpha = float(np.float32(alpha))
    scale = temperature_scale(temperature)
    bonus_alpha = effective_alpha(alpha, temperature)
    top_p = float(np.float32(top_p))
    if not 0.0 < top_p <= 1.0:
        raise ValueError("top_p must be in (0, 1]")
    use_topp = top_p < 1.0
    if use_topp and alpha != 1.0:
        raise ValueError("top_p < 1 needs alpha == 1")
    big_b, n_part, k1, v_size = target.shape
    k_drafts = k1 - 1
    draft_tokens = np.asarray(draft_tokens, dtype=np.int64)
    out = dict(
        lse_p=np.zeros((big_b, n_part, k1)), g_p=np.zeros((big_b, n_part, k_drafts)),
        lse_q=np.zeros((big_b, n_part, k_drafts)), g_q=np.zeros((big_b, n_part, k_drafts)),
        lse_alpha=np.zeros((big_b, n_part)), delta=np.zeros((big_b, n_part)),
        bonus=np.zeros((big_b, n_part), dtype=np.int64),
        bonus_margin=np.zeros((big_b, n_part)), topp_margin=np.full((big_b, n_part), np.inf))
    for b in range(big_b):
        for n in range(n_part):
            t_rows = widen(target[b, n], dtype) if dtype else target[b, n]
            d_rows = widen(draft[b, n], dtype) if dtype else draft[b, n]
            if scale != 1.0:
                t_rows = np.asarray(t_rows, dtype=np.float64) * scale
                d_rows = np.asarray(d_rows, dtype=np.float64) * scale
            u = philox.uniform(seed, step, (prompt_offset + b) * n_part + n, k_drafts,
                               philox.BONUS)
            raw = widen(target[b, n, k_drafts], dtype) if dtype else target[b, n, k_drafts]
            if use_topp:
                s = score_particle_topp(t_rows, d_rows, draft_tokens[b, n], top_p)
                out["topp_margin"][b, n] = s["margin"]
                w = np.where(s["bonus_kept"], bonus_weights(raw, bonus_alpha), 0.0)
            else:
                s = score_particle(t_rows, d_rows, draft_tokens[b, n], alpha)
                w = bonus_weights(raw, bonus_alpha)
            for key in ("lse_p", "g_p", "lse_q", "g_q", "lse_alpha", "delta"):
                out[key][b, n] = s[key]
            tok, margin = inverse_cdf(w, u)
            out["bonus"][b, n] = tok
            out["bonus_margin"][b, n] = margin
    if log_potential is not None:
        out["delta"] = out["delta"] + np.asarray(log_potential, dtype=np.float64)
    lw_pre = np.asarray(log_weights, dtype=np.float64) + out["delta"]
    out["log_weights_pre"] = lw_pre
    out["log_weights"] = np.zeros((big_b, n_part))
    out["ess"] = np.zeros(big_b)
    out["resampled"] = np.zeros(big_b, dtype=bool)
    out["ancestors"] = np.zeros((big_b, n_part), dtype=np.int64)
    out["resample_margin"] = np.zeros((big_b, n_part))
    out["ess_margin"] = np.zeros(big_b)
    out["tokens_out"] = np.zeros((big_b, n_part, k1), dtype=np.int64)
    for b in range(big_b):
        r = resample_prompt(lw_pre[b], ess_frac, seed, step, prompt_offset + b)
        out["log_weights"][b] = r["log_weights_out"]
        out["ess"][b] = r["ess"]
        out["resampled"][b] = r["resampled"]
        out["ancestors"][b] = r["ancestors"]
        out["resample_margin"][b] = r["margins"]
        out["ess_margin"][b] = r["ess_margin"]
        a = r["ancestors"]
        out["tokens_out"][b, :, :k_drafts] = draft_tokens[b, a]
        out["tokens_out"][b, :, k_drafts] = out["bonus"][b, a]
    return out


# --------------------------------------------------------------------------
# the extend-side draft sampler
# --------------------------------------------------------------------------
def draft_sample(draft, position, *, alpha=1.0, seed=0, step=0, dtype=None, prompt_offset=0):
    """One drafted token per particle: x ~ softmax(alpha * l) of draft row
    [B, N, V], by inverse CDF in vocabulary order with the uniform of
    (seed, step, particle b*N+n, position, DRAFT).

    The SMC page's Extend stage has the draft model extend every particle by
    K tokens; this is the sampling half of one of those K positions.  alpha
    is the inverse temperature of the draft (1: sample q itself).
    prompt_offset shifts the stream numbers as in ``smc_step``.
    Returns (tokens[B, N], margins[B, N]).
    """
    alpha = float(np.float32(alpha))
    big_b, n_part, v_size = draft.shape
    toks = np.zeros((big_b, n_part), dtype=np.int64)
    margins = np.zeros((big_b, n_part))
    for b in range(big_b):
        for n in range(n_part):
            row = widen(draft[b, n], dtype) if dtype else np.asarray(draft[b, n], np.float64)
            u = philox.uniform(seed, step, (prompt_offset + b) * n_part + n, position,
                               philox.DRAFT)
            toks[b, n], margins[b, n] = inverse_cdf(bonus_weights(row, alpha), u)
    return toks, margins
