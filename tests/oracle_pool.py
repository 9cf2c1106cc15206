"""Oracle calls spread over a process pool, for the large-sample parity tallies.

Test infrastructure.  A batch of prompts is cut into slices; each slice goes
to one worker, which runs the CPU oracle on it with ``prompt_offset`` set to
the slice's first prompt, so every random stream is the one the whole batch
would use.  The results are concatenated along the prompt axis.  This module
imports only numpy and the oracle, so spawned workers start quickly.
"""
import numpy as np

from oracle import smc as osmc, sps as osps

STEP_KEYS = ("ess", "ess_margin", "resampled", "resample_margin", "ancestors",
             "log_weights_pre", "bonus", "bonus_margin", "topp_margin")


def _step_slice(args):
    b0, target, draft, x, lw, phi, kw = args
    r = osmc.smc_step(target, draft, x, lw, prompt_offset=b0, log_potential=phi, **kw)
    return {k: r[k] for k in STEP_KEYS if k in r}


def _sps_slice(args):
    b0, target, draft, x, kw = args
    return osps.sps_verify(target, draft, x, prompt_offset=b0, **kw)


def _draft_slice(args):
    b0, rows, position, kw = args
    return osmc.draft_sample(rows, position, prompt_offset=b0, **kw)


def _concat(parts):
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def smc_step(pool, target, draft, x, lw, per_task=1, **kw):
    """oracle.smc.smc_step over [B, ...] inputs, ``per_task`` prompts a task."""
    B = target.shape[0]
    phi = kw.pop("log_potential", None)
    tasks = [(b, target[b:b + per_task], draft[b:b + per_task], x[b:b + per_task],
              lw[b:b + per_task], None if phi is None else phi[b:b + per_task], kw)
             for b in range(0, B, per_task)]
    return _concat(pool.map(_step_slice, tasks))


def sps_verify(pool, target, draft, x, per_task=32, **kw):
    """oracle.sps.sps_verify over [B, ...] inputs, ``per_task`` prompts a task."""
    B = target.shape[0]
    tasks = [(b, target[b:b + per_task], draft[b:b + per_task], x[b:b + per_task], kw)
             for b in range(0, B, per_task)]
    return _concat(pool.map(_sps_slice, tasks))


def draft_sample(pool, rows, position, per_task=16, **kw):
    """oracle.smc.draft_sample over rows [B, N, V]; returns (tokens, margins)."""
    B = rows.shape[0]
    tasks = [(b, rows[b:b + per_task], position, kw) for b in range(0, B, per_task)]
    parts = pool.map(_draft_slice, tasks)
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))
