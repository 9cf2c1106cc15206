"""Checkpoint and resume: 5 steps, the state saved to a file and loaded into
fresh buffers, then 5 more steps, equal 10 straight steps bit for bit.

The step's state is what the caller holds: the log-weights, the paged KV
state (tables, token counts, reference counts, free stacks) and the step
counter, which keys every random draw (Philox counter word 0).  The library
keeps nothing between calls (its workspace is scratch whose counters every
call leaves at zero), so a resumed run is the same run.  Checked on the GPU
through the C ABI, and for the CPU oracle itself.
"""
import numpy as np
import pytest
import torch

from smc_speculative_decoding_gb300.workloads import WORKLOADS, make_step_inputs, make_kv_state, \
    to_numpy_logits

KV_KEYS = ("tables", "seq_len", "refcount", "free_list", "free_top")


def _gpu_runner(w, dev):
    import smc_speculative_decoding_gb300 as smcsd
    T, P = w.kv_dims(10)
    kv = make_kv_state(w.B, w.N, w.prefix, w.block_size, T, P, device=dev)
    p0 = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 5, 0)
    kv_s = smcsd.make_kv(p0, kv, w.block_size)
    st = dict(kv=kv, kv_s=kv_s, ws=smcsd.alloc_workspace(p0, kv_s, device=dev),
              lw=torch.zeros(w.B * w.N, device=dev),
              tok=torch.empty(w.B * w.N * (w.K + 1), dtype=torch.int32, device=dev),
              anc=torch.empty(w.B * w.N, dtype=torch.int32, device=dev),
              ess=torch.empty(w.B, device=dev), res=torch.empty(w.B, dtype=torch.int32, device=dev))
    return st


def _gpu_steps(w, st, steps, inputs):
    import smc_speculative_decoding_gb300 as smcsd
    outs = []
    for s in steps:
        inp = inputs[s]
        p = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 5, s)
        smcsd.smc_step(p, inp["target"], inp["draft"], inp["draft_tokens"], st["lw"], st["tok"],
                       st["anc"], st["ess"], st["res"], kv=st["kv_s"], workspace=st["ws"])
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(st["ws"], clear=True) == 0
        outs.append({k: st[k].cpu().clone() for k in ("lw", "tok", "anc", "ess", "res")})
    return outs


@pytest.mark.gpu
def test_resume_on_the_gpu_is_bit_exact(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_speculative_decoding_gb300 import build
    build.build()
    w = WORKLOADS["single_prompt_v32000"].with_(B=3, sigma_d=2.0)
    dev = "cuda"
    inputs = [make_step_inputs(w, 5, device=dev, step=s) for s in range(10)]
    straight = _gpu_runner(w, dev)
    ref = _gpu_steps(w, straight, range(10), inputs)
    assert any(o["res"].any() for o in ref), "no step resampled"

    first = _gpu_runner(w, dev)
    _gpu_steps(w, first, range(5), inputs)
    path = tmp_path / "state.npz"
    np.savez(path, lw=first["lw"].cpu().numpy(), step=5,
             **{k: first["kv"][k].cpu().numpy() for k in KV_KEYS})
    del first
    torch.cuda.synchronize()

    loaded = np.load(path)
    resumed = _gpu_runner(w, dev)  # fresh buffers and a fresh workspace
    resumed["lw"].copy_(torch.from_numpy(loaded["lw"]))
    for k in KV_KEYS:
        resumed["kv"][k].copy_(torch.from_numpy(loaded[k]))
    s0 = int(loaded["step"])
    got = _gpu_steps(w, resumed, range(s0, 10), inputs)
    for a, b in zip(ref[5:], got):
        for k in a:
            assert torch.equal(a[k], b[k]), k
    for k in KV_KEYS:
        assert torch.equal(straight["kv"][k], resumed["kv"][k]), k


def test_resume_of_the_oracle_is_bit_exact(tmp_path):
    from oracle import smc as osmc, kv as okv
    w = WORKLOADS["tiny_v64"].with_(B=2, N=8, sigma_d=1.5)
    T, P = w.kv_dims(10)
    inputs = []
    for s in range(10):
        inp = make_step_inputs(w, 6, step=s)
        inputs.append((to_numpy_logits(inp["target"]), to_numpy_logits(inp["draft"]),
                       inp["draft_tokens"].numpy().astype(np.int64)))

    def fresh():
        kv = {k: v.numpy().astype(np.int64) for k, v in
              make_kv_state(w.B, w.N, w.prefix, w.block_size, T, P).items()}
        return {"lw": np.zeros((w.B, w.N)), **{k: kv[k] for k in KV_KEYS}}

    def run(state, steps):
        outs = []
        for s in steps:
            tgt, dft, x = inputs[s]
            r = osmc.smc_step(tgt, dft, x, state["lw"], alpha=w.alpha, ess_frac=w.ess_frac,
                              seed=6, step=s, dtype=w.dtype)
            k2 = okv.remap_append(state["tables"], state["seq_len"], state["refcount"],
                                  state["free_list"], state["free_top"], r["ancestors"],
                                  r["resampled"], w.K + 1, w.block_size, P)
            state.update({k: k2[k] for k in KV_KEYS}, lw=r["log_weights"])
            outs.append((r["tokens_out"], r["ancestors"], r["log_weights"]))
        return outs

    straight = fresh()
    ref = run(straight, range(10))
    first = fresh()
    run(first, range(5))
    np.savez(tmp_path / "o.npz", step=5, **first)
    loaded = dict(np.load(tmp_path / "o.npz"))
    s0 = int(loaded.pop("step"))
    resumed = {k: v.copy() for k, v in loaded.items()}
    got = run(resumed, range(s0, 10))
    for a, b in zip(ref[5:], got):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
    for k in KV_KEYS:
        assert np.array_equal(straight[k], resumed[k]), k
