"""smc_step_noalloc: the step without a caller workspace.

Some callers cannot allocate device memory themselves (for example a plugin
inside a serving runtime whose allocator owns the GPU's memory), so they have
no workspace to pass; smc_step_noalloc runs the same step on a fixed scratch
array inside the library.  These tests call it through the C ABI and check,
on two calls in a row (state carried from the first into the second), that
it produces what smc_step produces with a workspace of its own, within the
parity tolerances used elsewhere (log-weights 1e-4 for fp32 logits, 2e-3 for
bf16; integer outputs exact).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import smc_speculative_decoding_gb300 as smcsd
from smc_speculative_decoding_gb300 import binding
from smc_speculative_decoding_gb300.workloads import WORKLOADS, make_step_inputs, make_kv_state

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-3}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_speculative_decoding_gb300 import build
    build.build()


def _state(w, dev, steps):
    T, P = w.kv_dims(steps)
    kv = make_kv_state(w.B, w.N, w.prefix, w.block_size, T, P, device=dev)
    outs = dict(lw=torch.zeros(w.B * w.N, device=dev),
                tok=torch.empty(w.B * w.N * (w.K + 1), dtype=torch.int32, device=dev),
                anc=torch.empty(w.B * w.N, dtype=torch.int32, device=dev),
                ess=torch.empty(w.B, device=dev),
                res=torch.empty(w.B, dtype=torch.int32, device=dev))
    return kv, outs


@pytest.mark.parametrize("name,B", [("tiny_v64", 3), ("single_prompt_v32000", 2),
                                    ("batched_serving_v128256", 16)])
def test_noalloc_matches_workspace_entry_point(name, B):
    """Two calls in a row; the serving shape (16 prompts x 16 particles, K 4,
    V 128256) is the library's main use and must fit the fixed array."""
    w = WORKLOADS[name].with_(B=B)
    dev = "cuda"
    kv_a, out_a = _state(w, dev, 2)
    kv_b, out_b = _state(w, dev, 2)
    p0 = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 7, 0)
    kv_sa = smcsd.make_kv(p0, kv_a, w.block_size)
    kv_sb = smcsd.make_kv(p0, kv_b, w.block_size)
    assert smcsd.smc_workspace_bytes(p0, kv_sa) <= (8 << 20), "shape does not fit the array"
    ws = smcsd.alloc_workspace(p0, kv_sa, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for step in range(2):  # two calls in a row, state carried forward
        inp = make_step_inputs(w, 7, device=dev, step=step)
        p = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, w.alpha, w.ess_frac, 7, step)
        smcsd.smc_step(p, inp["target"], inp["draft"], inp["draft_tokens"], out_a["lw"],
                       out_a["tok"], out_a["anc"], out_a["ess"], out_a["res"], kv=kv_sa,
                       workspace=ws)
        binding.smc_step_noalloc(p, inp["target"], inp["draft"], inp["draft_tokens"],
                                 out_b["lw"], out_b["tok"], out_b["anc"], out_b["ess"],
                                 out_b["res"], status, kv=kv_sb)
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(ws, clear=True) == 0
        assert status.item() == 0
        for key in ("tok", "anc", "res"):
            assert torch.equal(out_a[key], out_b[key]), key
        assert (out_a["lw"] - out_b["lw"]).abs().max().item() <= TOL[w.dtype]
        assert np.allclose(out_a["ess"].cpu().numpy(), out_b["ess"].cpu().numpy(), rtol=1e-5)
        for key in kv_a:
            assert torch.equal(kv_a[key], kv_b[key]), key


@pytest.mark.parametrize("B,N,K,V,dtype", [(64, 256, 16, 1 << 20, "bf16"),
                                            (128, 16, 4, 128256, "bf16"),
                                            (8, 256, 8, 151936, "f32")])
def test_noalloc_rejects_shapes_beyond_its_array(B, N, K, V, dtype):
    """Shapes whose workspace exceeds the fixed array are refused with
    SMC_ERR_WORKSPACE before anything is launched (the pointers below are
    never touched)."""
    lib = binding.lib()
    fn = lib.smc_step_noalloc
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(binding.smc_params)] + [ctypes.c_void_p] * 8 + \
        [ctypes.POINTER(binding.smc_kv), ctypes.c_void_p, ctypes.c_void_p]
    big = smcsd.make_params(B, N, K, V, dtype)
    assert smcsd.smc_workspace_bytes(big) > (8 << 20)
    fake = ctypes.c_void_p(0x1000)
    rc = fn(ctypes.byref(big), *[fake] * 8, None, fake, None)
    assert rc == -3, smcsd.smc_strerror(rc)
