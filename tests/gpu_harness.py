"""Lockstep parity harness: the CUDA path against the CPU oracle.

Each step feeds the same seeded inputs (drawn by the workloads module on the
GPU) to libsmcsd (through the Python binding of its C ABI) and to the oracle,
compares every output, then carries the GPU's state (log-weights, KV tables)
into the next step for both sides.  Integer outputs must match exactly except
for draws the oracle flags as near ties (the drawn point lies within
``tie`` = 1e-5 of a cumulative boundary, as a fraction of the total); those
are counted per kind of draw, and the mismatch rate of each kind is bounded
by MISMATCH_RATE.
"""
from dataclasses import dataclass, field

import numpy as np
import torch

import smc_speculative_decoding_gb300 as smcsd
from smc_speculative_decoding_gb300.workloads import (make_step_inputs, make_kv_state,
                                                      to_numpy_logits)
from oracle import smc as osmc, kv as okv, sps as osps

LW_TOL = {"f32": 1e-4, "bf16": 2e-3}
NEAR_TIE = 1e-5          # |u*S - C| / S below this flags a draw as a near tie
MISMATCH_RATE = 1e-4     # flagged mismatches allowed per draw, for each kind


@dataclass
class Tally:
    draws: int = 0          # draws compared (all kinds)
    flagged: int = 0        # of which the oracle flags as near ties
    mismatched: int = 0     # of which GPU and oracle differ (all must be flagged)
    lw_checked: int = 0     # log-weights compared
    lw_err_max: float = 0.0  # largest |GPU - oracle| among them
    kinds: dict = field(default_factory=dict)  # kind -> [draws, flagged, mismatched]

    def add(self, n, flagged_mask, mismatch_mask, what, kind="other"):
        flagged_mask = np.asarray(flagged_mask, dtype=bool)
        mismatch_mask = np.asarray(mismatch_mask, dtype=bool)
        bad = mismatch_mask & ~flagged_mask
        assert not bad.any(), f"{what}: {int(bad.sum())} unflagged mismatches at {np.argwhere(bad)[:5].tolist()}"
        f, m = int(flagged_mask.sum()), int(mismatch_mask.sum())
        self.draws += int(n)
        self.flagged += f
        self.mismatched += m
        k = self.kinds.setdefault(kind, [0, 0, 0])
        k[0] += int(n)
        k[1] += f
        k[2] += m

    def merge(self, other):
        self.draws += other.draws
        self.flagged += other.flagged
        self.mismatched += other.mismatched
        self.lw_checked += other.lw_checked
        self.lw_err_max = max(self.lw_err_max, other.lw_err_max)
        for kind, v in other.kinds.items():
            k = self.kinds.setdefault(kind, [0, 0, 0])
            for i in range(3):
                k[i] += v[i]

    def rate_ok(self):
        """Every kind's mismatches within MISMATCH_RATE of its draws (so no
        mismatch at all below 1/MISMATCH_RATE draws)."""
        return all(m <= MISMATCH_RATE * d for d, _, m in self.kinds.values())

    def summary(self):
        kinds = " ".join(f"{k}={d}/{f}/{m}" for k, (d, f, m) in sorted(self.kinds.items()))
        return (f"draws={self.draws} flagged={self.flagged} mismatched={self.mismatched} "
                f"lw_checked={self.lw_checked} lw_err_max={self.lw_err_max:.3g} "
                f"[kind=draws/flagged/mismatched: {kinds}]")


def kv_to_numpy(kv):
    return {k: v.detach().cpu().numpy().astype(np.int64) for k, v in kv.items()}


class StepRunner:
    """Owns the device state of one workload run through smc_step."""

    def __init__(self, w, seed=0, device="cuda", with_kv=True, steps=None, ess_frac=None,
                 temperature=None):
        self.w = w
        self.seed = seed
        self.temperature = temperature  # None: plain smc_step; else smc_step_ex
        self.device = device
        self.ess_frac = w.ess_frac if ess_frac is None else ess_frac
        B, N, K = w.B, w.N, w.K
        self.log_weights = torch.zeros(B * N, dtype=torch.float32, device=device)
        self.tokens_out = torch.empty(B * N * (K + 1), dtype=torch.int32, device=device)
        self.ancestors = torch.empty(B * N, dtype=torch.int32, device=device)
        self.ess = torch.empty(B, dtype=torch.float32, device=device)
        self.resampled = torch.empty(B, dtype=torch.int32, device=device)
        self.kv = None
        self.kv_struct = None
        params = self.params(0)
        if with_kv:
            T, P = w.kv_dims(steps)
            self.T, self.P = T, P
            self.kv = make_kv_state(B, N, w.prefix, w.block_size, T, P, device=device)
            self.kv_struct = smcsd.make_kv(params, self.kv, w.block_size)
        self.workspace = smcsd.alloc_workspace(params, self.kv_struct, device=device)

    def params(self, step):
        w = self.w
        return smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, self.ess_frac,
                                 self.seed, step)

    def run(self, inputs, step, log_potential=None, top_p=1.0):
        if self.temperature is None and log_potential is None and top_p == 1.0:
            smcsd.smc_step(self.params(step), inputs["target"], inputs["draft"],
                           inputs["draft_tokens"], self.log_weights, self.tokens_out,
                           self.ancestors, self.ess, self.resampled, kv=self.kv_struct,
                           workspace=self.workspace)
        else:
            smcsd.smc_step_ex(self.params(step), inputs["target"], inputs["draft"],
                              inputs["draft_tokens"], self.log_weights, self.tokens_out,
                              self.ancestors, self.ess, self.resampled, kv=self.kv_struct,
                              workspace=self.workspace,
                              temperature=1.0 if self.temperature is None else self.temperature,
                              log_potential=log_potential, top_p=top_p)

    def status(self):
        return smcsd.smc_device_status(self.workspace, clear=True)


def lockstep(w, steps, seed=0, with_kv=True, ess_frac=None, tie=NEAR_TIE, resample_tie=NEAR_TIE,
             lw_init=None, temperature=None, potential_fn=None, top_p=1.0, tokens_fn=None,
             pool=None, ess_schedule=None, kv_steps=None):
    """Run `steps` steps on GPU and oracle; return the Tally.  temperature and
    potential_fn(step) -> [B, N] fp32 CUDA tensor (or None) select smc_step_ex.
    pool: a process pool for the oracle (oracle_pool), else it runs here.
    ess_schedule(step) -> the ESS fraction of that step (else ess_frac).
    kv_steps: size the KV tables and pool for this many steps (else `steps`)."""
    runner = StepRunner(w, seed=seed, with_kv=with_kv, steps=kv_steps or steps,
                        ess_frac=ess_frac, temperature=temperature)
    if lw_init is not None:
        runner.log_weights.copy_(torch.as_tensor(lw_init, dtype=torch.float32).reshape(-1))
    B, N, K = w.B, w.N, w.K
    tally = Tally()
    for step in range(steps):
        if ess_schedule is not None:
            runner.ess_frac = ess_schedule(step)
        inp = make_step_inputs(w, seed, device="cuda", step=step)
        if tokens_fn is not None:
            tokens_fn(inp, step)
        lw_in = runner.log_weights.cpu().numpy().reshape(B, N).astype(np.float64)
        kv_in = kv_to_numpy(runner.kv) if with_kv else None
        phi = potential_fn(step) if potential_fn is not None else None
        runner.run(inp, step, log_potential=phi, top_p=top_p)
        torch.cuda.synchronize()
        bits = runner.status()
        assert bits == 0, f"device status {smcsd.status_names(bits)}"
        g_lw = runner.log_weights.cpu().numpy().reshape(B, N).astype(np.float64)
        g_tok = runner.tokens_out.cpu().numpy().reshape(B, N, K + 1)
        g_anc = runner.ancestors.cpu().numpy().reshape(B, N)
        g_ess = runner.ess.cpu().numpy().astype(np.float64)
        g_res = runner.resampled.cpu().numpy().astype(bool)

        x = inp["draft_tokens"].cpu().numpy().astype(np.int64)
        kw = dict(alpha=w.alpha, ess_frac=runner.ess_frac, seed=seed, step=step, dtype=w.dtype,
                  temperature=1.0 if temperature is None else temperature,
                  log_potential=None if phi is None else
                  phi.cpu().numpy().reshape(B, N).astype(np.float64), top_p=top_p)
        tgt, dft = to_numpy_logits(inp["target"]), to_numpy_logits(inp["draft"])
        del inp
        if pool is None:
            ref = osmc.smc_step(tgt, dft, x, lw_in, **kw)
        else:
            import oracle_pool
            ref = oracle_pool.smc_step(pool, tgt, dft, x, lw_in, **kw)
        check_step(w, ref, x, g_lw, g_tok, g_anc, g_ess, g_res, tally, tie, resample_tie)
        if with_kv:
            check_kv(w, runner, kv_in, g_anc, g_res)
    return tally


def check_step(w, ref, x, g_lw, g_tok, g_anc, g_ess, g_res, tally, tie, resample_tie):
    B, N, K = w.B, w.N, w.K
    tol = LW_TOL[w.dtype]
    # a top-p nucleus whose boundary lies within 1e-5 of top_p may differ by
    # one group of tied logits: such a particle's weight, and its prompt's
    # resampling, are compared as near ties
    tp = ref["topp_margin"] < NEAR_TIE if "topp_margin" in ref else np.zeros((B, N), dtype=bool)
    # ESS and the resampling decision
    ess_ok = np.isclose(g_ess, ref["ess"], rtol=1e-4, atol=0)
    assert (ess_ok | tp.any(1)).all(), (g_ess, ref["ess"])
    ess_flag = (ref["ess_margin"] < NEAR_TIE) | tp.any(1)
    tally.add(B, ess_flag, g_res != ref["resampled"], "resample decision", "ess_decision")
    for b in range(B):
        if g_res[b] != ref["resampled"][b]:
            continue
        if g_res[b]:
            flag = (ref["resample_margin"][b] < resample_tie) | tp[b].any()
            tally.add(N, flag, g_anc[b] != ref["ancestors"][b], f"ancestors of prompt {b}",
                      "ancestors")
            assert np.array_equal(g_lw[b], np.zeros(N))
        else:
            assert np.array_equal(g_anc[b], np.arange(N))
            r = ref["log_weights_pre"][b]
            dead = np.isneginf(r)  # weight 0: a -inf increment (potential or masked token)
            same = ~tp[b]
            assert np.array_equal(np.isneginf(g_lw[b])[same], dead[same]), "-inf log-weights differ"
            live = same & ~dead
            err = np.abs(g_lw[b][live] - r[live])
            assert err.size == 0 or err.max() <= tol, f"log-weights off by {err.max()} (tol {tol})"
            tally.lw_checked += int(err.size)
            if err.size:
                tally.lw_err_max = max(tally.lw_err_max, float(err.max()))
            n_tp = int(tp[b].sum())
            tally.add(n_tp, np.ones(n_tp, bool), np.zeros(n_tp, bool), "nucleus near ties",
                      "nucleus")
        # tokens: drafted tokens of the GPU's ancestor, bonus of that ancestor
        a = g_anc[b]
        assert np.array_equal(g_tok[b, :, :K], x[b, a]), "drafted tokens not gathered by ancestor"
        flag = (ref["bonus_margin"][b, a] < tie) | tp[b, a]
        tally.add(N, flag, g_tok[b, :, K] != ref["bonus"][b, a], f"bonus tokens of prompt {b}",
                  "bonus")


def check_kv(w, runner, kv_in, g_anc, g_res):
    ref = okv.remap_append(kv_in["tables"], kv_in["seq_len"], kv_in["refcount"],
                           kv_in["free_list"], kv_in["free_top"], g_anc, g_res, w.K + 1,
                           w.block_size, runner.P)
    assert all(not e for e in ref["errors"]), ref["errors"]
    got = kv_to_numpy(runner.kv)
    for key in ("tables", "seq_len", "refcount", "free_top"):
        assert np.array_equal(got[key], ref[key]), f"KV {key} differs"
    for b in range(w.B):
        top = ref["free_top"][b]
        assert np.array_equal(got["free_list"][b, :top], ref["free_list"][b, :top]), "free stack differs"
        pairs = ref["cow_pairs"][b]
        assert got["n_cow"][b] == len(pairs)
        if pairs:
            assert np.array_equal(got["cow_pairs"][b, :len(pairs)], np.array(pairs)), "cow pairs differ"


def sps_lockstep(w, seed=0, step=0, tie=NEAR_TIE, temperature=1.0, top_p=1.0, tokens_fn=None,
                 pool=None):
    """One sps_verify call (N = 1) against the oracle; returns the Tally.
    temperature != 1 or top_p < 1 goes through sps_verify_ex; tokens_fn(inp,
    step) may replace the drafted tokens first.  Kinds: sps_accept (one draw
    per acceptance test the oracle made), sps_residual and sps_bonus (the
    final draw after a rejection, or after K acceptances)."""
    assert w.N == 1
    B, K = w.B, w.K
    inp = make_step_inputs(w, seed, device="cuda", step=step)
    if tokens_fn is not None:
        tokens_fn(inp, step)
    params = smcsd.make_params(B, 1, K, w.V, w.dtype, 1.0, 0.5, seed, step)
    ws = smcsd.alloc_workspace(params)
    tokens_out = torch.empty(B * (K + 1), dtype=torch.int32, device="cuda")
    n_emitted = torch.empty(B, dtype=torch.int32, device="cuda")
    if temperature == 1.0 and top_p == 1.0:
        smcsd.sps_verify(params, inp["target"], inp["draft"], inp["draft_tokens"], tokens_out,
                         n_emitted, ws)
    else:
        smcsd.sps_verify_ex(params, inp["target"], inp["draft"], inp["draft_tokens"], tokens_out,
                            n_emitted, ws, temperature=temperature, top_p=top_p)
    torch.cuda.synchronize()
    bits = smcsd.smc_device_status(ws, clear=True)
    assert bits == 0, smcsd.status_names(bits)
    g_tok = tokens_out.cpu().numpy().reshape(B, K + 1)
    g_n = n_emitted.cpu().numpy()
    x = inp["draft_tokens"].cpu().numpy().reshape(B, K).astype(np.int64)
    tgt = to_numpy_logits(inp["target"]).reshape(B, K + 1, w.V)
    dft = to_numpy_logits(inp["draft"]).reshape(B, K, w.V)
    del inp
    kw = dict(seed=seed, step=step, dtype=w.dtype, temperature=temperature, top_p=top_p)
    if pool is None:
        ref = osps.sps_verify(tgt, dft, x, **kw)
    else:
        import oracle_pool
        ref = oracle_pool.sps_verify(pool, tgt, dft, x, **kw)
    # a nucleus boundary within 1e-5 of top_p flags the whole prompt
    tp = ref["topp_margin"] < NEAR_TIE if "topp_margin" in ref else np.zeros(B, dtype=bool)
    tally = Tally()
    for b in range(B):
        n_ref = ref["n_emitted"][b]
        margins = ref["accept_margin"][b]
        test_flags = (margins[np.isfinite(margins)] < tie) | tp[b]
        acc_flag = bool(test_flags.any())
        miss = np.zeros(test_flags.size, bool)
        if g_n[b] != n_ref:
            # the count differs: one acceptance test went the other way, which
            # must be a flagged one
            miss[int(np.argmax(test_flags)) if acc_flag else 0] = True
            tally.add(test_flags.size, test_flags, miss, f"accepted count of prompt {b}",
                      "sps_accept")
            continue
        tally.add(test_flags.size, test_flags, miss, f"acceptance tests of prompt {b}",
                  "sps_accept")
        kind = "sps_residual" if n_ref <= K else "sps_bonus"
        if tp[b]:
            tally.add(1, [True], [not np.array_equal(g_tok[b], ref["tokens_out"][b])],
                      f"prompt {b} (nucleus near tie)", kind)
            continue
        assert np.array_equal(g_tok[b, :n_ref - 1], ref["tokens_out"][b, :n_ref - 1])
        assert (g_tok[b, n_ref:] == -1).all()
        flag = acc_flag or ref["final_margin"][b] < tie
        tally.add(1, [flag], [g_tok[b, n_ref - 1] != ref["tokens_out"][b, n_ref - 1]],
                  f"final token of prompt {b}", kind)
    return tally, ref, g_n
