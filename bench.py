"""Throughput of the SMC-SD per-step particle update on GB300.

One step = one smc_step call over the batched-serving workload (16 prompts x
16 particles, K = 4 drafted tokens, V = 128256, bf16 logits, KV block tables
with a 2048-token shared prefix): every logit row's log-sum-exp and drafted
token gather, the bonus-token draw, the importance-weight update, ESS,
systematic resampling when ESS < N/2, token emission and the block-table
remap.  The metric is particle-tokens per second (B*N*(K+1) tokens per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): prompts are independent, so every rank
runs its own 16 prompts (weak scaling, no collective on the data path); the
timed region is bracketed by barriers and the slowest rank's time is used.

Inputs are resident in HBM before timing; each step reads 591 MB of logits,
more than the 129 MB L2, from a ring of two distinct step inputs, so no step
finds its logits in L2.  The KV state and weights are reset every 128 steps
(the workload's episode length), outside the timed region.

Besides the headline line's own numbers, the JSON carries:
  * ``extensions``: the draft sampler, smc_step_ex (temperature, potentials,
    top-p), sps_verify on the serving rows with sampled and with argmax
    drafts, and the KV-cache saving over a 128-step serving episode;
  * ``workloads``: every other workload the method is described on (power
    sampling, the serving draft-noise sweep, the single-prompt latency case,
    the batch-32 (N, K) sweep), each timed the same way, with its row-pass and
    whole-step roofline fractions and the oracle timed on a sample of it;
  * ``parity_sample``: the headline's first steps checked against the CPU
    oracle (part of the oracle leg), with flagged and mismatched draw counts.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SMC step particle-tokens/s at V=128256 bf16; % of GB300 HBM roofline"
WORKLOAD = "batched_serving_v128256"
KERNEL = "row_stream_kernel"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "row_stream_kernel_batched_serving_v128256.md")
KERNEL_SOURCES = ["smc_step.cu", "step_args.cuh", "row_common.cuh", "device_common.cuh",
                  "exp2_table.cuh"]
L2_BYTES = 129 * 2 ** 20
RING_MIN_BYTES = 4 * L2_BYTES   # a ring of distinct step inputs at least this large


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--sigma-d", type=float, default=None, help="draft noise override")
    ap.add_argument("--episode", type=int, default=128, help="steps between KV resets")
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--row-steps", type=int, default=256,
                    help="steps of the separate row-pass timing run")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work budget of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the secondary measurements of the step's extensions")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads (power sampling, sweeps, latency case)")
    ap.add_argument("--sweep", choices=["full", "corners", "none"], default="full",
                    help="points of the batch-32 (N, K) sweep to time")
    return ap.parse_args()


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def input_seed(rank):
    """Each rank draws its own prompts: the path shards by prompt, so the
    ranks share nothing and the per-GPU work is fixed (weak scaling)."""
    return 1000 + rank


def workload(args):
    from smc_speculative_decoding_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.sigma_d is not None:
        w = w.with_(sigma_d=args.sigma_d)
    return w


def logit_bytes(w):
    return w.B * w.N * (2 * w.K + 1) * w.V * w.bytes_per_logit


def algorithmic_bytes(w, T, resampled_prompts):
    """Bytes one step must move: every logit once, the particle state, and the
    block tables of prompts that resampled (read + write)."""
    particle = w.B * w.N * (4 * w.K        # drafted tokens read
                            + 8             # log-weight read + write
                            + 4 * (w.K + 1)  # emitted tokens
                            + 4)            # ancestor
    tables = resampled_prompts * w.N * (T * 4 * 2 + 8)
    return logit_bytes(w) + particle + tables


def kernels_per_step(w):
    """Kernels one plain smc_step launches: the streaming row pass, the
    per-particle epilogue and the per-prompt tail when a row's bytes are a
    multiple of 16; else the per-chunk row kernel and the tail."""
    return 3 if (w.V * w.bytes_per_logit) % 16 == 0 else 2


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "smc_speculative_decoding_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    text = open(PROFILE_SUMMARY).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != kernel_hash():
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        load = [float(r[1]) for r in rows if float(r[3]) > 200.0] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(float(r[3]) for r in rows)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class StepBench:
    """Device state of smc_step on one workload: a ring of distinct step
    inputs (at least RING_MIN_BYTES, so no step finds its logits in L2), the
    particle outputs and, with KV tables, the paged KV state of an episode."""

    def __init__(self, smcsd, w, dev, seed, episode, with_kv=True, ring_min=RING_MIN_BYTES):
        from smc_speculative_decoding_gb300.workloads import make_step_inputs, make_kv_state
        self.smcsd, self.w, self.dev, self.episode = smcsd, w, dev, episode
        n_ring = max(2, math.ceil(ring_min / logit_bytes(w)))
        self.ring = [make_step_inputs(w, seed, device=dev, step=s) for s in range(n_ring)]
        self.T, self.P = w.kv_dims(episode)
        p0 = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 0, 0)
        self.kv0 = self.kv = self.kv_s = None
        if with_kv:
            self.kv0 = make_kv_state(w.B, w.N, w.prefix, w.block_size, self.T, self.P, device=dev)
            self.kv = {k: v.clone() for k, v in self.kv0.items()}
            self.kv_s = smcsd.make_kv(p0, self.kv, w.block_size)
        self.ws = smcsd.alloc_workspace(p0, self.kv_s, device=dev)
        self.lw = torch.zeros(w.B * w.N, device=dev)
        self.tok = torch.empty(w.B * w.N * (w.K + 1), dtype=torch.int32, device=dev)
        self.anc = torch.empty(w.B * w.N, dtype=torch.int32, device=dev)
        self.ess = torch.empty(w.B, device=dev)
        self.res = torch.empty(w.B, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()

    def reset(self):
        if self.kv is not None:
            for k in self.kv:
                self.kv[k].copy_(self.kv0[k])
        self.lw.zero_()

    def step(self, s):
        """One smc_step; s is the global step counter (the Philox counter)."""
        w, inp = self.w, self.ring[s % len(self.ring)]
        p = self.smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 0, s)
        self.smcsd.smc_step(p, inp["target"], inp["draft"], inp["draft_tokens"], self.lw,
                            self.tok, self.anc, self.ess, self.res, kv=self.kv_s,
                            workspace=self.ws, stream=self.stream)

    def time_steps(self, n_steps, s0):
        """Episodes of `episode` steps, the state reset between them (untimed).
        Each episode is bracketed by one pair of CUDA events with nothing in
        between but the steps: an event recorded between two steps would
        delay the second one's launch (it ends the programmatic overlap of
        one step's tail with the next one's start).  The library's step clock
        stamps every step's start on the device; consecutive stamps within an
        episode give the per-step periods.  Returns (total ms, per-step ms)."""
        total, per, done = 0.0, [], 0
        stamps = torch.zeros(self.episode + 8, dtype=torch.int64, device=self.dev)
        counter = torch.zeros(1, dtype=torch.int32, device=self.dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        while done < n_steps:
            self.reset()
            counter.zero_()
            n = min(self.episode, n_steps - done)
            self.smcsd.smc_set_step_clock(stamps, counter)
            e0.record(self.stream)
            for i in range(n):
                self.step(s0 + done + i)
            e1.record(self.stream)
            self.smcsd.smc_set_step_clock(None)
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1)
            st = stamps[:n].cpu().numpy().astype(np.float64)
            per += list(np.diff(st) / 1e6)
            done += n
        return total, per

    def time_rows(self, n_steps, s0):
        """The same steps again with the library's row-timing hook recording
        CUDA events around the streaming row kernel; also keeps each step's
        ESS and resampling flags (copied on the device, outside any timing).
        Returns (row ms per step, ess [n, B], resampled [n, B])."""
        w = self.w
        ess_buf = torch.empty(n_steps, w.B, device=self.dev)
        res_buf = torch.empty(n_steps, w.B, dtype=torch.int32, device=self.dev)
        row_ms, done = [], 0
        while done < n_steps:
            self.reset()
            n = min(self.episode, n_steps - done)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            for i in range(n):
                self.smcsd.smc_set_row_timing_events(*evs[i])
                self.step(s0 + done + i)
                ess_buf[done + i].copy_(self.ess)
                res_buf[done + i].copy_(self.res)
            self.smcsd.smc_set_row_timing_events(None, None)
            torch.cuda.synchronize()
            row_ms += [b.elapsed_time(e) for b, e in evs]
            done += n
        return row_ms, ess_buf.cpu().numpy(), res_buf.cpu().numpy()

    def status(self):
        return self.smcsd.smc_device_status(self.ws, clear=True)


def step_figures(w, total_ms, per_ms, n_steps, row_ms, ess, res, T, peak, world=1):
    """The numbers of one workload's timing: throughput, per-step spread, the
    row pass against the HBM peak, the whole step against it."""
    ms = total_ms / n_steps
    resampled = float(res.sum()) / max(1, res.shape[0])
    row_launch_ms = float(np.mean(row_ms))
    row_gbs = logit_bytes(w) / (row_launch_ms / 1e3) / 1e9
    step_bytes = algorithmic_bytes(w, T, resampled)
    step_gbs = step_bytes / (ms / 1e3) / 1e9
    return {
        "ms_per_step": ms, "ms_per_step_median": float(np.median(per_ms)),
        "ms_per_step_min": float(np.min(per_ms)),
        "particle_tokens_per_s": w.particle_tokens * n_steps * world / (total_ms / 1e3),
        "steps_per_s": n_steps * world / (total_ms / 1e3),
        "row_pass": {"ms": row_launch_ms, "gbs": row_gbs, "frac": row_gbs / peak,
                     "bytes": logit_bytes(w)},
        "step": {"gbs": step_gbs, "frac": step_gbs / peak, "bytes": step_bytes},
        "resampled_prompts_per_step": resampled, "mean_ess": float(np.mean(ess)),
        "mean_ess_over_n": float(np.mean(ess)) / w.N,
    }


def run_ours(args, world, rank, local):
    import smc_speculative_decoding_gb300 as smcsd
    from smc_speculative_decoding_gb300 import build

    build.build()
    dev = f"cuda:{local}"
    w = workload(args)
    sb = StepBench(smcsd, w, dev, input_seed(rank), args.episode, ring_min=0)

    # the clock sampler starts first, so that the timed steps follow the
    # warm-up with no idle gap (an idle GPU drops its clocks, and the first
    # step after a pause then runs several times slower)
    clocks = ClockSampler(local)
    clocks.start()
    sb.reset()
    for s in range(args.warmup):
        sb.step(s)
        if (s + 1) % args.episode == 0:
            sb.reset()
    assert sb.status() == 0  # synchronises

    # timed region: episodes of `episode` steps, KV reset between them (untimed)
    barrier(world)
    torch.cuda.synchronize()
    total_ms, per_ms = sb.time_steps(args.steps, args.warmup)
    barrier(world)
    torch.cuda.synchronize()
    clk = clocks.stop()
    bits = sb.status()
    if bits:
        raise RuntimeError(f"device status during timing: {smcsd.status_names(bits)}")
    total_ms = max_over_ranks(total_ms, world)

    # the row pass alone: a second run of the same steps with the library's
    # row-timing hook recording CUDA events around the streaming kernel
    n_rows_steps = min(args.steps, args.row_steps)
    row_ms, ess, res = sb.time_rows(n_rows_steps, args.warmup)
    assert sb.status() == 0
    row_launch_ms = max_over_ranks(float(np.mean(row_ms)), world)
    peak, peak_kind = measured_peak()
    fig = step_figures(w, total_ms, per_ms, args.steps, [row_launch_ms], ess, res, sb.T, peak,
                       world)
    row_bytes = logit_bytes(w)
    achieved = row_bytes / (row_launch_ms / 1e3) / 1e9

    out = {
        "metric": METRIC, "value": fig["particle_tokens_per_s"], "unit": "particle-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "ms_per_step_median": fig["ms_per_step_median"], "ms_per_step_min": fig["ms_per_step_min"],
        "step_timing": (f"one CUDA event pair around each {args.episode}-step episode (KV reset "
                        "between episodes, untimed); median and min are step periods from the "
                        "library's device step clock (smc_set_step_clock), which puts nothing "
                        "between steps"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "K": w.K, "V": w.V,
                   "logits": w.dtype, "sigma_t": w.sigma_t, "top_m": w.top_m,
                   "sigma_d": w.sigma_d, "alpha": w.alpha, "ess_frac": w.ess_frac,
                   "prefix": w.prefix, "block_size": w.block_size, "episode_steps": args.episode,
                   "parallelism": f"prompt-sharded x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: 591 MB of logits per step from a ring of "
                         "2 distinct steps (129 MB L2)"},
        "steps_per_s": fig["steps_per_s"],
        "resampled_prompts_per_step": fig["resampled_prompts_per_step"],
        "mean_ess": fig["mean_ess"], "mean_ess_over_n": fig["mean_ess_over_n"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "kernel": KERNEL, "algorithmic_bytes_per_launch": row_bytes,
                     "avg_launch_ms": row_launch_ms,
                     "launch_timing": f"CUDA events around the row pass (library hook), "
                                      f"{len(row_ms)} steps after the timed region",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "step_roofline": {"achieved": fig["step"]["gbs"], "frac": fig["step"]["frac"],
                          "unit": "GB/s", "algorithmic_bytes_per_step": fig["step"]["bytes"],
                          "avg_step_ms": total_ms / args.steps,
                          "kernels": ["row_stream_kernel", "particle_kernel", "prompt_kernel"]
                          if kernels_per_step(w) == 3 else
                          ["step_rows_kernel", "tail_kernel"]},
        "gpu_launches": kernels_per_step(w) * args.steps,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["_parity_inputs"] = gpu_parity_sample(sb, n_steps=2, s0=args.warmup + args.steps)
    del sb
    torch.cuda.empty_cache()
    if not args.no_e2e:
        out["e2e"] = run_e2e(args, w, dev, smcsd, world)
    if not args.no_extras:
        out["extensions"] = run_extensions(w, dev, smcsd)
    if not args.no_workloads and rank == 0:
        out["workloads"] = run_workloads(args, dev, smcsd, peak, with_cpu=not args.no_cpu_baseline)
    return out


def gpu_parity_sample(sb, n_steps, s0):
    """The headline's first steps of a fresh episode, with each step's inputs
    and the GPU's state before and after, copied to the host for the oracle
    leg to check (the oracle runs in cpu_baseline, not here)."""
    w = sb.w
    sb.reset()
    samples = []
    for i in range(n_steps):
        inp = sb.ring[(s0 + i) % len(sb.ring)]
        lw_in = sb.lw.cpu().numpy().reshape(w.B, w.N).astype(np.float64)
        sb.step(s0 + i)
        torch.cuda.synchronize()
        samples.append(dict(
            step=s0 + i, lw_in=lw_in,
            target=inp["target"].cpu(), draft=inp["draft"].cpu(),
            x=inp["draft_tokens"].cpu().numpy().astype(np.int64),
            lw=sb.lw.cpu().numpy().reshape(w.B, w.N).astype(np.float64),
            tok=sb.tok.cpu().numpy().reshape(w.B, w.N, w.K + 1),
            anc=sb.anc.cpu().numpy().reshape(w.B, w.N),
            ess=sb.ess.cpu().numpy().astype(np.float64),
            res=sb.res.cpu().numpy().astype(bool)))
    assert sb.status() == 0
    return samples


def run_extensions(w, dev, smcsd, reps=50):
    """Secondary measurements on the headline workload's rows: the draft-side
    sampler, smc_step_ex at temperature 0.8 with log-potentials and at top-p
    0.9, sps_verify on the same rows, and the KV-cache saving of an episode."""
    from smc_speculative_decoding_gb300.workloads import make_step_inputs, make_kv_state
    peak = measured_peak()[0]
    res = {}
    ring = [make_step_inputs(w, 1000, device=dev, step=s) for s in range(2)]
    params = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, 1.0, w.ess_frac, 0, 0)
    ws = smcsd.alloc_workspace(params)
    rows = ring[0]["draft"][:, :, 0].contiguous()
    tok = torch.empty(w.B * w.N, dtype=torch.int32, device=dev)
    for _ in range(5):
        smcsd.smc_draft_sample(params, rows, 0, tok, ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 256 MB > L2
    ms = []
    for r in range(reps):
        flush.zero_()
        e0.record()
        smcsd.smc_draft_sample(params, rows, r % w.K, tok, ws)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    bytes_call = w.B * w.N * w.V * w.bytes_per_logit
    iso = float(np.median(ms))
    # back to back over the K draft positions of both ring steps (8 x 66 MB of
    # distinct rows, more than L2), as a drafting loop issues them: each
    # call's row pass streams beside the previous call's row combine
    sets = [r["draft"][:, :, k].contiguous() for r in ring for k in range(w.K)]
    torch.cuda.synchronize()
    n_b2b = 64
    e0.record()
    for r in range(n_b2b):
        smcsd.smc_draft_sample(params, sets[r % len(sets)], r % w.K, tok, ws)
    e1.record()
    torch.cuda.synchronize()
    med = e0.elapsed_time(e1) / n_b2b
    res["draft_sample"] = {"rows": w.B * w.N, "V": w.V, "ms_per_call": med,
                           "tokens_per_s": w.B * w.N / (med / 1e3),
                           "achieved_gbs": bytes_call / (med / 1e3) / 1e9,
                           "frac_of_hbm_peak": bytes_call / (med / 1e3) / 1e9 / peak,
                           "calls": f"{n_b2b} back to back over {len(sets)} distinct row sets "
                                    f"({len(sets) * bytes_call / 1e6:.0f} MB, more than L2)",
                           "ms_per_call_isolated": iso,
                           "isolated": "one call at a time, a 256 MB buffer written between "
                                       "calls (median of 50)"}
    del rows, flush, sets
    T, P = w.kv_dims(64)
    kv0 = make_kv_state(w.B, w.N, w.prefix, w.block_size, T, P, device=dev)
    kv = {k: v.clone() for k, v in kv0.items()}
    kv_s = smcsd.make_kv(params, kv, w.block_size)
    ws2 = smcsd.alloc_workspace(params, kv_s)
    lw = torch.zeros(w.B * w.N, device=dev)
    outs = dict(tok=torch.empty(w.B * w.N * (w.K + 1), dtype=torch.int32, device=dev),
                anc=torch.empty(w.B * w.N, dtype=torch.int32, device=dev),
                ess=torch.empty(w.B, device=dev), res=torch.empty(w.B, dtype=torch.int32, device=dev))
    phi = torch.zeros(w.B * w.N, device=dev)

    def reset():
        for k in kv:
            kv[k].copy_(kv0[k])
        lw.zero_()

    def ex_steps(n, s0, ring_, **kw):
        for s in range(n):
            p = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 0, s0 + s)
            r = ring_[s % 2]
            smcsd.smc_step_ex(p, r["target"], r["draft"], r["draft_tokens"], lw, outs["tok"],
                              outs["anc"], outs["ess"], outs["res"], kv=kv_s, workspace=ws2, **kw)

    def timed(n, ring_, **kw):
        reset()
        ex_steps(3, 0, ring_, **kw)
        torch.cuda.synchronize()
        e0.record()
        ex_steps(n, 3, ring_, **kw)
        e1.record()
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(ws2, clear=True) == 0
        return e0.elapsed_time(e1) / n

    ms_step = timed(48, ring, temperature=0.8, log_potential=phi)
    res["step_ex_temperature_potential"] = {"ms_per_step": ms_step,
                                            "particle_tokens_per_s": w.particle_tokens / (ms_step / 1e3),
                                            "temperature": 0.8, "steps": 48}
    # top-p 0.9: drafted tokens are each draft row's argmax, always inside its nucleus
    ring_tp = [dict(r, draft_tokens=r["draft"].float().argmax(-1).to(torch.int32).contiguous())
               for r in ring]
    ms_tp = timed(16, ring_tp, top_p=0.9)
    res["step_ex_top_p"] = {"ms_per_step": ms_tp, "top_p": 0.9, "steps": 16,
                            "particle_tokens_per_s": w.particle_tokens / (ms_tp / 1e3),
                            "note": "the nucleus kernel reads every row once more from HBM "
                                    "and again from L2 (mass bins, then the threshold bin)"}
    # speculative-sampling verify on the same rows, one particle per prompt
    # (B*N prompts): drafted tokens sampled from the draft rows (the
    # workload's own, as speculative sampling draws them), and each draft
    # row's argmax (few rejections); then under temperature 0.8 and top-p 0.9
    nb = w.B * w.N
    ps = smcsd.make_params(nb, 1, w.K, w.V, w.dtype, 1.0, 0.5, 0, 0)
    ws3 = smcsd.alloc_workspace(ps)
    s_tok = torch.empty(nb * (w.K + 1), dtype=torch.int32, device=dev)
    s_n = torch.empty(nb, dtype=torch.int32, device=dev)
    bytes_call = nb * (2 * w.K + 1) * w.V * w.bytes_per_logit

    def sps_time(ring_, **kw):
        views = [(r["target"].view(nb, w.K + 1, w.V), r["draft"].view(nb, w.K, w.V),
                  r["draft_tokens"].view(nb, w.K)) for r in ring_]
        fn = smcsd.sps_verify_ex if kw else smcsd.sps_verify
        for s in range(3):
            fn(ps, *views[s % 2], s_tok, s_n, ws3, **kw)
        torch.cuda.synchronize()
        n_sps = 16
        e0.record()
        for s in range(n_sps):
            fn(ps, *views[s % 2], s_tok, s_n, ws3, **kw)
        e1.record()
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(ws3, clear=True) == 0
        m = e0.elapsed_time(e1) / n_sps
        em = int(s_n.sum().item())
        return {"prompts": nb, "ms_per_call": m, "tokens_per_s_last_call": em / (m / 1e3),
                "rejected_prompts_last_call": int((s_n <= w.K).sum().item()),
                "achieved_gbs": bytes_call / (m / 1e3) / 1e9,
                "frac_of_hbm_peak": bytes_call / (m / 1e3) / 1e9 / peak,
                "bytes": "every row once; a rejected prompt's rows p_j and q_j again"}

    res["sps_verify"] = dict(sps_time(ring), drafts="sampled from the draft rows")
    res["sps_verify_argmax_drafts"] = dict(sps_time(ring_tp), drafts="each draft row's argmax")
    r2 = sps_time(ring_tp, temperature=0.8, top_p=0.9)
    res["sps_verify_ex_top_p"] = {k: r2[k] for k in ("prompts", "ms_per_call",
                                                      "tokens_per_s_last_call")}
    res["sps_verify_ex_top_p"].update(temperature=0.8, top_p=0.9, drafts="argmax")
    del ring_tp
    res["kv_saving"] = kv_saving_episode(w, dev, smcsd, ring)
    return res


def kv_saving_episode(w, dev, smcsd, ring, steps=128):
    """The KV cache of one serving episode: every step appends K+1 tokens,
    resampling shares blocks by pointer; smc_kv_usage after each step gives
    the blocks in use and the blocks N unshared copies would hold."""
    from smc_speculative_decoding_gb300.workloads import make_kv_state
    T, P = w.kv_dims(steps)
    params = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 0, 0)
    kv = make_kv_state(w.B, w.N, w.prefix, w.block_size, T, P, device=dev)
    kv_s = smcsd.make_kv(params, kv, w.block_size)
    ws = smcsd.alloc_workspace(params, kv_s)
    lw = torch.zeros(w.B * w.N, device=dev)
    tok = torch.empty(w.B * w.N * (w.K + 1), dtype=torch.int32, device=dev)
    anc = torch.empty(w.B * w.N, dtype=torch.int32, device=dev)
    ess = torch.empty(w.B, device=dev)
    res = torch.empty(w.B, dtype=torch.int32, device=dev)
    used = torch.empty(steps, w.B, dtype=torch.int32, device=dev)
    unshared = torch.empty(steps, w.B, dtype=torch.int32, device=dev)
    for s in range(steps):
        p = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 0, s)
        r = ring[s % len(ring)]
        smcsd.smc_step(p, r["target"], r["draft"], r["draft_tokens"], lw, tok, anc, ess, res,
                       kv=kv_s, workspace=ws)
        smcsd.smc_kv_usage(params, kv_s, used[s], unshared[s])
    torch.cuda.synchronize()
    assert smcsd.smc_device_status(ws) == 0
    u = used.cpu().numpy().sum(1).astype(np.float64)
    x = unshared.cpu().numpy().sum(1).astype(np.float64)
    saving = 1.0 - u / x
    return {"steps": steps, "prefix": w.prefix, "block_size": w.block_size,
            "used_blocks_final": int(u[-1]), "unshared_blocks_final": int(x[-1]),
            "saving_final": float(saving[-1]), "saving_mean": float(saving.mean()),
            "saving_first_step": float(saving[0]),
            "context": "the pages report 72.3 % less KV cache for SMC-SD on their models; "
                       "this is the same ratio on synthetic logits"}


def run_workloads(args, dev, smcsd, peak, with_cpu):
    """Every other workload of the method, timed like the headline: power
    sampling (alpha = 4), the serving draft-noise sweep, the single-prompt
    latency case and the batch-32 (N, K) sweep."""
    from smc_speculative_decoding_gb300.workloads import (WORKLOADS, SERVING_SIGMAS, SWEEP_N,
                                                          SWEEP_K)
    out = {}
    cases = [("power_sampling_v151936", WORKLOADS["power_sampling_v151936"], 16)]
    for sig in SERVING_SIGMAS:
        if sig != WORKLOADS[WORKLOAD].sigma_d:
            cases.append((f"batched_serving_v128256_sigma_d{sig:g}",
                          WORKLOADS[WORKLOAD].with_(sigma_d=sig), 16))
    cases.append(("single_prompt_v32000", WORKLOADS["single_prompt_v32000"], 64))
    if args.sweep != "none":
        pts = [(n, k) for n in SWEEP_N for k in SWEEP_K]
        if args.sweep == "corners":
            pts = [(1, 2), (8, 4), (64, 8)]
        for n, k in pts:
            cases.append((f"sweep_v128256_N{n}_K{k}", WORKLOADS["sweep_v128256"].with_(N=n, K=k), 12))
    for name, w, n_steps in cases:
        sb = StepBench(smcsd, w, dev, 1000, max(128, n_steps))
        sb.reset()
        for s in range(3):
            sb.step(s)
        torch.cuda.synchronize()
        total, per = sb.time_steps(n_steps, 3)
        assert sb.status() == 0
        row_ms, ess, res = sb.time_rows(min(n_steps, 8), 3)
        fig = step_figures(w, total, per, n_steps, row_ms, ess, res, sb.T, peak)
        fig["config"] = {"B": w.B, "N": w.N, "K": w.K, "V": w.V, "logits": w.dtype,
                         "alpha": w.alpha, "sigma_d": w.sigma_d, "prefix": w.prefix,
                         "steps": n_steps, "ring_inputs": len(sb.ring),
                         "ring_bytes": len(sb.ring) * logit_bytes(w)}
        fig["us_per_step"] = 1e3 * fig["ms_per_step"]
        fig["gpu_launches_per_step"] = kernels_per_step(w)
        del sb
        torch.cuda.empty_cache()
        if with_cpu:
            n, el = oracle_prompt_steps(w, 0.5 if name.startswith("sweep") else 2.0, max_steps=2)
            fig["cpu_baseline"] = {"value": n * w.N * (w.K + 1) / el, "unit": "particle-tokens/s",
                                   "cores": 1, "kind": "oracle",
                                   "sample": f"{n} prompt-steps of 1 x {w.N} particles, "
                                             f"{2 * w.K + 1} rows of V={w.V}, in {el:.2f} s"}
        out[name] = fig
    return out


def run_e2e(args, w, dev, smcsd, world):
    """Same metric through the public API with host buffers: every step copies
    its logits and drafted tokens from pinned host memory and reads the emitted
    tokens and weights back, inside the timed region.  The copy of step s+1's
    inputs runs on a second stream into the other half of a double buffer while
    step s computes, as a serving loop whose inputs arrive from the host would
    overlap them."""
    from smc_speculative_decoding_gb300.workloads import make_step_inputs, make_kv_state
    T, P = w.kv_dims(args.episode)
    host = []
    for s in range(2):
        inp = make_step_inputs(w, 2000, device=dev, step=s)
        host.append({k: v.cpu().pin_memory() for k, v in inp.items()})
        del inp
    d_in = [{k: torch.empty_like(v, device=dev) for k, v in host[0].items()} for _ in range(2)]
    kv0 = make_kv_state(w.B, w.N, w.prefix, w.block_size, T, P, device=dev)
    kv = {k: v.clone() for k, v in kv0.items()}
    p0 = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 0, 0)
    kv_s = smcsd.make_kv(p0, kv, w.block_size)
    ws = smcsd.alloc_workspace(p0, kv_s, device=dev)
    lw = torch.zeros(w.B * w.N, device=dev)
    tok = torch.empty(w.B * w.N * (w.K + 1), dtype=torch.int32, device=dev)
    anc = torch.empty(w.B * w.N, dtype=torch.int32, device=dev)
    ess = torch.empty(w.B, device=dev)
    res = torch.empty(w.B, dtype=torch.int32, device=dev)
    h_tok = torch.empty(tok.shape, dtype=torch.int32).pin_memory()
    h_lw = torch.empty(lw.shape, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    # the copies go out as N_COPY slices on as many streams, so that several
    # copy engines carry them
    n_copy = 4
    copy_streams = [torch.cuda.Stream() for _ in range(n_copy)]
    n_steps = min(args.e2e_steps, args.steps)
    h2d = sum(v.numel() * v.element_size() for v in host[0].values())
    d2h = h_tok.numel() * 4 + h_lw.numel() * 4
    copied = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]

    def upload(s):
        # step s's inputs into buffer s % 2, once the step that used it last is
        # done: slice j of every tensor on copy stream j
        b = s % 2
        for j, cs in enumerate(copy_streams):
            cs.wait_event(consumed[b])
            with torch.cuda.stream(cs):
                for k in d_in[b]:
                    dst, src = d_in[b][k].view(-1), host[s % 2][k].view(-1)
                    lo, hi = dst.numel() * j // n_copy, dst.numel() * (j + 1) // n_copy
                    if hi > lo:
                        dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
            copied[b][j].record(cs)

    def run(s0, n):
        for b in range(2):
            consumed[b].record(stream)
        upload(s0)
        for s in range(s0, s0 + n):
            if s + 1 < s0 + n:
                upload(s + 1)
            b = s % 2
            for ev in copied[b]:
                stream.wait_event(ev)
            p = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 0, s)
            smcsd.smc_step(p, d_in[b]["target"], d_in[b]["draft"], d_in[b]["draft_tokens"], lw,
                           tok, anc, ess, res, kv=kv_s, workspace=ws, stream=stream)
            consumed[b].record(stream)
            h_tok.copy_(tok, non_blocking=True)
            h_lw.copy_(lw, non_blocking=True)

    run(0, 3)
    torch.cuda.synchronize()
    for k in kv:
        kv[k].copy_(kv0[k])
    lw.zero_()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(0, n_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    return {"value": w.particle_tokens * n_steps * world / (ms / 1e3), "unit": "particle-tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_steps,
            "ms_per_step": ms / n_steps,
            "overlap": f"step s+1's H2D copy, as {n_copy} slices on {n_copy} streams, during "
                       "step s (double buffer)",
            "h2d_gbs": h2d * n_steps / (ms / 1e3) / 1e9}


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline of our line)
# ---------------------------------------------------------------------------
def oracle_prompt_steps(w, budget_s, max_steps=None, seed=3000):
    """Runs the fp64 oracle on one prompt at a time (N particles, full rows,
    weights, resampling and KV remap) until `budget_s` seconds or
    `max_steps` prompt-steps; returns (prompt_steps, seconds)."""
    from smc_speculative_decoding_gb300.workloads import make_step_inputs, make_kv_state, \
        to_numpy_logits
    from oracle import smc as osmc, kv as okv
    w1 = w.with_(B=1)
    T, P = w1.kv_dims(128)
    inputs = []
    for s in range(2):
        inp = make_step_inputs(w1, seed, device="cpu", step=s)
        inputs.append((to_numpy_logits(inp["target"]), to_numpy_logits(inp["draft"]),
                       inp["draft_tokens"].numpy().astype(np.int64)))
    kv = {k: v.numpy().astype(np.int64) for k, v in
          make_kv_state(1, w1.N, w1.prefix, w1.block_size, T, P).items()}
    lw = np.zeros((1, w1.N))
    done = 0
    t0 = time.perf_counter()
    while True:
        tgt, dft, x = inputs[done % 2]
        r = osmc.smc_step(tgt, dft, x, lw, alpha=w1.alpha, ess_frac=w1.ess_frac, seed=0,
                          step=done, dtype=w1.dtype)
        k2 = okv.remap_append(kv["tables"], kv["seq_len"], kv["refcount"], kv["free_list"],
                              kv["free_top"], r["ancestors"], r["resampled"], w1.K + 1,
                              w1.block_size, P)
        kv = {k: k2[k] for k in ("tables", "seq_len", "refcount", "free_list", "free_top")}
        lw = r["log_weights"]
        done += 1
        if done % 100 == 0:
            kv = {k: v.numpy().astype(np.int64) for k, v in
                  make_kv_state(1, w1.N, w1.prefix, w1.block_size, T, P).items()}
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps is not None and done >= max_steps):
            return done, el


def _oracle_worker(args):
    """One process of the all-cores oracle timing: its own prompt stream."""
    w, budget_s, seed = args
    return oracle_prompt_steps(w, budget_s, seed=seed)


def oracle_all_cores(w, budget_s):
    """The same oracle on every host core at once, one independent prompt
    stream per process (prompts share nothing); a spawned pool, since this
    process already holds a CUDA context."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    try:
        with mp.get_context("spawn").Pool(cores) as pool:
            res = pool.map(_oracle_worker, [(w, budget_s, 3000 + i) for i in range(cores)])
    except Exception as e:  # no pool on this host: report why
        return {"value": None, "cores": cores, "error": str(e)[:200]}
    n = sum(r[0] for r in res)
    el = max(r[1] for r in res)
    return {"value": n * w.N * (w.K + 1) / el, "unit": "particle-tokens/s", "cores": cores,
            "sample": f"{n} prompt-steps over {cores} processes in {el:.1f} s"}


def oracle_parity(w, samples):
    """The oracle on the GPU's parity sample (inputs and the GPU's incoming
    log-weights, step by step): draws compared, flagged as near ties
    (|u S - C| < 1e-5 S), mismatched; log-weights compared where no
    resampling reset them."""
    from smc_speculative_decoding_gb300.workloads import to_numpy_logits
    from oracle import smc as osmc
    tol = 2e-3 if w.dtype == "bf16" else 1e-4
    c = {"prompt_steps": 0, "draws": 0, "flagged": 0, "mismatched": 0, "unflagged_mismatched": 0,
         "lw_checked": 0, "lw_err_max": 0.0, "lw_out_of_tolerance": 0}
    t0 = time.perf_counter()
    for smp in samples:
        tgt, dft = to_numpy_logits(smp["target"]), to_numpy_logits(smp["draft"])
        r = osmc.smc_step(tgt, dft, smp["x"], smp["lw_in"], alpha=w.alpha, ess_frac=w.ess_frac,
                          seed=0, step=smp["step"], dtype=w.dtype)
        c["prompt_steps"] += w.B

        def add(n, flag, miss):
            c["draws"] += int(n)
            c["flagged"] += int(np.sum(flag))
            c["mismatched"] += int(np.sum(miss))
            c["unflagged_mismatched"] += int(np.sum(miss & ~flag))
        add(w.B, r["ess_margin"] < 1e-5, smp["res"] != r["resampled"])
        for b in range(w.B):
            if smp["res"][b] != r["resampled"][b]:
                continue
            a = smp["anc"][b]
            if smp["res"][b]:
                add(w.N, r["resample_margin"][b] < 1e-5, a != r["ancestors"][b])
            else:
                err = np.abs(smp["lw"][b] - r["log_weights_pre"][b])
                c["lw_checked"] += w.N
                c["lw_err_max"] = max(c["lw_err_max"], float(err.max()))
                c["lw_out_of_tolerance"] += int((err > tol).sum())
            add(w.N, r["bonus_margin"][b, a] < 1e-5, smp["tok"][b, :, w.K] != r["bonus"][b, a])
    c["oracle_seconds"] = time.perf_counter() - t0
    return c


def cpu_baseline(w, budget_s, parity_samples=None):
    n, el = oracle_prompt_steps(w, budget_s)
    out = {"value": n * w.N * (w.K + 1) / el, "unit": "particle-tokens/s", "cores": 1,
           "kind": "oracle",
           "sample": f"{n} prompt-steps of {w.name} (1 prompt x {w.N} particles x "
                     f"{2 * w.K + 1} rows of V={w.V}, tail and KV remap) in {el:.1f} s, "
                     f"numpy fp64, single thread",
           "all_cores": oracle_all_cores(w, budget_s)}
    if parity_samples:
        out["parity_sample"] = oracle_parity(w, parity_samples)
    return out


def run_reference(args, world, rank):
    """The oracle timed on host cores, as the reference arm: each step is a
    bounded sample of the workload (one prompt of 16), the whole run kept to a
    few minutes."""
    w = workload(args)
    budget = 150.0
    # warm-up sample steps
    oracle_prompt_steps(w, 5.0, max_steps=max(1, min(args.warmup, 3)))
    n, el = oracle_prompt_steps(w, budget, max_steps=args.steps)
    value = n * w.N * (w.K + 1) / el
    sample = (f"{n} of {args.steps} steps timed (time budget {budget:.0f} s); each step one "
              f"prompt of {w.B} ({w.N} particles x {2 * w.K + 1} rows of V={w.V}, weights, "
              f"resampling, KV remap), numpy fp64, single thread")
    return {"metric": METRIC, "value": value, "unit": "particle-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / n * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "N": w.N, "K": w.K, "V": w.V,
                       "logits": w.dtype, "sigma_d": w.sigma_d, "prefix": w.prefix},
            "cpu_baseline": {"value": value, "unit": "particle-tokens/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "particle-tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, world, rank)), flush=True)
        return 0
    world, rank, local = dist_setup(args.gpus)
    out = run_ours(args, world, rank, local)
    samples = out.pop("_parity_inputs", None)
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(workload(args), args.cpu_seconds, samples)
            out["parity_sample"] = out["cpu_baseline"].pop("parity_sample", None)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
