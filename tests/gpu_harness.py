"""Lockstep parity harness: the CUDA path against the CPU oracle.

Each step feeds the same seeded inputs (drawn by the workloads module on the
GPU) to libsmcsd (through the Python binding of its C ABI) and to the oracle,
compares every output, then carries the GPU's state (log-weights, KV tables)
into the next step for both sides.  Integer outputs must match exactly except
for draws the oracle flags as near ties (the drawn point lies within
``tie`` of a cumulative boundary); those are counted.
"""
from dataclasses import dataclass, field

import numpy as np
import torch

import smc_speculative_decoding_gb300 as smcsd
from smc_speculative_decoding_gb300.workloads import (make_step_inputs, make_kv_state,
                                                      to_numpy_logits)
from oracle import smc as osmc, kv as okv, sps as osps

LW_TOL = {"f32": 1e-4, "bf16": 2e-3}


@dataclass
class Tally:
    draws: int = 0          # bonus / residual / resampling draws compared
    flagged: int = 0        # of which the oracle flags as near ties
    mismatched: int = 0     # of which GPU and oracle differ (all must be flagged)
    notes: list = field(default_factory=list)

    def add(self, n, flagged_mask, mismatch_mask, what):
        flagged_mask = np.asarray(flagged_mask, dtype=bool)
        mismatch_mask = np.asarray(mismatch_mask, dtype=bool)
        self.draws += int(n)
        self.flagged += int(flagged_mask.sum())
        self.mismatched += int(mismatch_mask.sum())
        bad = mismatch_mask & ~flagged_mask
        assert not bad.any(), f"{what}: {int(bad.sum())} unflagged mismatches at {np.argwhere(bad)[:5].tolist()}"


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


def lockstep(w, steps, seed=0, with_kv=True, ess_frac=None, tie=1e-5, resample_tie=1e-4,
             lw_init=None, temperature=None, potential_fn=None, top_p=1.0, tokens_fn=None):
    """Run `steps` steps on GPU and oracle; return the Tally.  temperature and
    potential_fn(step) -> [B, N] fp32 CUDA tensor (or None) select smc_step_ex."""
    runner = StepRunner(w, seed=seed, with_kv=with_kv, steps=steps, ess_frac=ess_frac,
                        temperature=temperature)
    if lw_init is not None:
        runner.log_weights.copy_(torch.as_tensor(lw_init, dtype=torch.float32).reshape(-1))
    B, N, K = w.B, w.N, w.K
    tally = Tally()
    for step in range(steps):
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
        ref = osmc.smc_step(to_numpy_logits(inp["target"]), to_numpy_logits(inp["draft"]), x,
                            lw_in, alpha=w.alpha, ess_frac=runner.ess_frac, seed=seed,
                            step=step, dtype=w.dtype,
                            temperature=1.0 if temperature is None else temperature,
                            log_potential=None if phi is None else
                            phi.cpu().numpy().reshape(B, N).astype(np.float64), top_p=top_p)
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
    tp = ref["topp_margin"] < 1e-5 if "topp_margin" in ref else np.zeros((B, N), dtype=bool)
    # ESS and the resampling decision
    ess_ok = np.isclose(g_ess, ref["ess"], rtol=1e-3, atol=0)
    assert (ess_ok | tp.any(1)).all(), (g_ess, ref["ess"])
    ess_flag = (ref["ess_margin"] < 1e-4) | tp.any(1)
    tally.add(B, ess_flag, g_res != ref["resampled"], "resample decision")
    for b in range(B):
        if g_res[b] != ref["resampled"][b]:
            continue
        if g_res[b]:
            flag = (ref["resample_margin"][b] < resample_tie) | tp[b].any()
            tally.add(N, flag, g_anc[b] != ref["ancestors"][b], f"ancestors of prompt {b}")
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
            tally.add(int(tp[b].sum()), np.ones(int(tp[b].sum()), bool),
                      np.zeros(int(tp[b].sum()), bool), "nucleus near ties")
        # tokens: drafted tokens of the GPU's ancestor, bonus of that ancestor
        a = g_anc[b]
        assert np.array_equal(g_tok[b, :, :K], x[b, a]), "drafted tokens not gathered by ancestor"
        flag = (ref["bonus_margin"][b, a] < tie) | tp[b, a]
        tally.add(N, flag, g_tok[b, :, K] != ref["bonus"][b, a], f"bonus tokens of prompt {b}")


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


def sps_lockstep(w, seed=0, step=0, tie=1e-5, temperature=1.0, top_p=1.0, tokens_fn=None):
    """One sps_verify call (N = 1) against the oracle; returns the Tally.
    temperature != 1 or top_p < 1 goes through sps_verify_ex; tokens_fn(inp,
    step) may replace the drafted tokens first."""
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
    ref = osps.sps_verify(to_numpy_logits(inp["target"]).reshape(B, K + 1, w.V),
                          to_numpy_logits(inp["draft"]).reshape(B, K, w.V), x,
                          seed=seed, step=step, dtype=w.dtype, temperature=temperature,
                          top_p=top_p)
    # a nucleus boundary within 1e-5 of top_p flags the whole prompt
    tp = ref["topp_margin"] < 1e-5 if "topp_margin" in ref else np.zeros(B, dtype=bool)
    tally = Tally()
    for b in range(B):
        n_ref = ref["n_emitted"][b]
        acc_flag = (ref["accept_margin"][b] < tie).any() or tp[b]
        if g_n[b] != n_ref:
            tally.add(1, [acc_flag], [True], f"accepted count of prompt {b}")
            continue
        if tp[b]:
            tally.add(1, [True], [not np.array_equal(g_tok[b], ref["tokens_out"][b])],
                      f"prompt {b} (nucleus near tie)")
            continue
        assert np.array_equal(g_tok[b, :n_ref - 1], ref["tokens_out"][b, :n_ref - 1])
        assert (g_tok[b, n_ref:] == -1).all()
        flag = acc_flag or ref["final_margin"][b] < tie
        tally.add(1, [flag], [g_tok[b, n_ref - 1] != ref["tokens_out"][b, n_ref - 1]],
                  f"final token of prompt {b}")
    return tally, ref, g_n
