"""Single-particle speculative-sampling verify (CPU oracle, fp64).

Test infrastructure: part of the CPU oracle (see ``oracle/__init__.py``).

"Accelerating Large Language Model Decoding with Speculative Sampling" (blog
notes, sections 1 "Introduction" and 4.2 "Modified Rejection Sampling"): the
draft model proposes K tokens, the target scores them in parallel, and a
modified rejection sampling accepts or resamples each drafted token so that the
output follows the target distribution (Theorem 1, cited under section 6).
The notes do not restate the rule; the plain form of it is taken:

  * drafted token x_k is accepted iff u_k < p_k(x_k) / q_k(x_k), u_k uniform,
    which accepts with probability min(1, p/q);
  * at the first rejection j, one token is drawn from the residual
    max(0, p_j - q_j), normalised, and the step ends with j+1 tokens;
  * if all K are accepted, one bonus token is drawn from target row K and the
    step ends with K+1 tokens;
  * should the residual have no positive mass (only through rounding when
    p_j == q_j), the token is drawn from p_j instead.

With a temperature T and a top-p threshold (the settings under which the
notes evaluate the method, section 6), p and q are first replaced by
softmax(l / T) restricted to their top-p nuclei and renormalised (the same
reading as the SMC step's, ``smc.nucleus``); the rule above then runs on
those distributions unchanged, so Theorem 1 holds for the tempered nucleus
of the target.  A drafted token outside the draft's nucleus could not have
been drawn and is reported.
"""
import numpy as np

from . import philox
from .smc import (row_logsumexp, inverse_cdf, bonus_weights, widen, nucleus,
                  temperature_scale)
from .errors import OracleError, DEV_BAD_TOKEN


def accept_ratio(target_row, draft_row, token):
    """p(x)/q(x) of one drafted token, from fp64 log-probabilities."""
    lse_p = row_logsumexp(target_row)
    lse_q = row_logsumexp(draft_row)
    return np.exp((target_row[token] - lse_p) - (draft_row[token] - lse_q))


def residual_weights(target_row, draft_row):
    """max(0, p - q) over the vocabulary, falling back to p if it has no mass."""
    p = np.exp(target_row - row_logsumexp(target_row))
    q = np.exp(draft_row - row_logsumexp(draft_row))
    r = np.maximum(p - q, 0.0)
    if not np.sum(r) > 0:
        return p
    return r


def verify_one(target_rows, draft_rows, tokens, u_accept, u_residual, u_bonus):
    """Verify one prompt with the uniforms given explicitly.

    target_rows [K+1, V], draft_rows [K, V] (fp64), tokens [K];
    u_accept[k], u_residual[k] for k < K, u_bonus scalar.
    Returns (emitted tokens list, accept margins, final-draw margin).
    """
    k_drafts, v_size = draft_rows.shape
    out = []
    accept_margins = []
    for k in range(k_drafts):
        x = int(tokens[k])
        if not 0 <= x < v_size:
            raise OracleError(DEV_BAD_TOKEN, "drafted token outside [0, V)")
        r = accept_ratio(target_rows[k], draft_rows[k], x)
        accept_margins.append(abs(u_accept[k] - r))
        if u_accept[k] < r:
            out.append(x)
            continue
        y, margin = inverse_cdf(residual_weights(target_rows[k], draft_rows[k]), u_residual[k])
        out.append(int(y))
        return out, accept_margins, margin
    y, margin = inverse_cdf(bonus_weights(target_rows[k_drafts], 1.0), u_bonus)
    out.append(int(y))
    return out, accept_margins, margin


def tempered_logprobs(rows, scale, top_p):
    """log of softmax(scale * row) restricted to the row's top-p nucleus and
    renormalised, -inf outside it, for each row of ``rows`` [R, V] (fp64; the
    product with an fp32 scale is exact).  Returns (log-probs [R, V], the
    smallest nucleus margin over the rows; inf without a nucleus)."""
    z = scale * np.asarray(rows, dtype=np.float64)
    out = np.empty_like(z)
    margin = np.inf
    for r in range(z.shape[0]):
        lse = row_logsumexp(z[r])
        if top_p < 1.0:
            kept, log_z, mg = nucleus(z[r], top_p)
            margin = min(margin, mg)
            out[r] = np.where(kept, z[r] - lse - log_z, -np.inf)
        else:
            out[r] = z[r] - lse
    return out, margin


def verify_one_logprobs(logp, logq, tokens, u_accept, u_residual, u_bonus):
    """verify_one on given log-probability rows: logp [K+1, V] and logq [K, V]
    (-inf outside a nucleus).  A drafted token with q = 0 could not have been
    drawn from q and is reported.  Same results as verify_one."""
    k_drafts, v_size = logq.shape
    out = []
    accept_margins = []
    for k in range(k_drafts):
        x = int(tokens[k])
        if not 0 <= x < v_size:
            raise OracleError(DEV_BAD_TOKEN, "drafted token outside [0, V)")
        if logq[k, x] == -np.inf:
            raise OracleError(DEV_BAD_TOKEN, "drafted token outside the draft's nucleus")
        r = np.exp(logp[k, x] - logq[k, x])
        accept_margins.append(abs(u_accept[k] - r))
        if u_accept[k] < r:
            out.append(x)
            continue
        p = np.exp(logp[k])
        w = np.maximum(p - np.exp(logq[k]), 0.0)
        if not np.sum(w) > 0:
            w = p
        y, margin = inverse_cdf(w, u_residual[k])
        out.append(int(y))
        return out, accept_margins, margin
    last = logp[k_drafts]
    y, margin = inverse_cdf(np.exp(last - np.max(last)), u_bonus)
    out.append(int(y))
    return out, accept_margins, margin


def sps_verify(target, draft, draft_tokens, *, seed=0, step=0, dtype=None, temperature=1.0,
               top_p=1.0, prompt_offset=0):
    """Verify B independent prompts (N = 1 particle each).

    target [B, K+1, V], draft [B, K, V] fp64 (or stored logits widened per
    prompt when ``dtype`` is given, see ``smc.widen``), draft_tokens [B, K].
    Uniforms: ACCEPT and RESIDUAL keyed by (step, b, k), BONUS by (step, b, K).
    With temperature != 1 or top_p < 1, p and q are the tempered nuclei
    (``tempered_logprobs``).  prompt_offset: the batch is prompts
    prompt_offset .. prompt_offset+B-1 of a larger one (the uniforms use those
    prompt numbers).
    Returns dict(tokens_out [B, K+1] padded with -1, n_emitted [B],
    accept_margin [B, K] (inf where not tested), final_margin [B], and with
    top_p < 1 topp_margin [B], each prompt's smallest nucleus margin).
    """
    plain = temperature == 1.0 and top_p == 1.0
    scale = temperature_scale(temperature)
    big_b, k1, _ = target.shape
    k_drafts = k1 - 1
    tokens_out = np.full((big_b, k1), -1, dtype=np.int64)
    n_emitted = np.zeros(big_b, dtype=np.int64)
    accept_margin = np.full((big_b, k_drafts), np.inf)
    final_margin = np.zeros(big_b)
    topp_margin = np.full(big_b, np.inf)
    for b in range(big_b):
        pb = prompt_offset + b
        ua = [philox.uniform(seed, step, pb, k, philox.ACCEPT) for k in range(k_drafts)]
        ur = [philox.uniform(seed, step, pb, k, philox.RESIDUAL) for k in range(k_drafts)]
        ub = philox.uniform(seed, step, pb, k_drafts, philox.BONUS)
        t_rows = widen(target[b], dtype) if dtype else target[b]
        d_rows = widen(draft[b], dtype) if dtype else draft[b]
        if plain:
            toks, margins, fm = verify_one(t_rows, d_rows, draft_tokens[b], ua, ur, ub)
        else:
            logp, mp = tempered_logprobs(t_rows, scale, top_p)
            logq, mq = tempered_logprobs(d_rows, scale, top_p)
            topp_margin[b] = min(mp, mq)
            toks, margins, fm = verify_one_logprobs(logp, logq, draft_tokens[b], ua, ur, ub)
        tokens_out[b, :len(toks)] = toks
        n_emitted[b] = len(toks)
        accept_margin[b, :len(margins)] = margins
        final_margin[b] = fm
    res = dict(tokens_out=tokens_out, n_emitted=n_emitted,
               accept_margin=accept_margin, final_margin=final_margin)
    if top_p < 1.0:
        res["topp_margin"] = topp_margin
    return res
