"""Thin Python binding of libsmcsd.so (include/smcsd.h), by ctypes.

Argument marshalling only: every function checks that the tensors it is given
are CUDA, contiguous and of the expected dtype and size, passes their device
pointers and the caller's stream to the C entry point of the same name, and
raises ``SmcError`` on a non-zero return.  All arithmetic runs in the
library's kernels; there is no CPU path.  PyTorch supplies device memory and
streams only.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsmcsd.so")

SMC_F32, SMC_BF16 = 0, 1

# device status bits (smcsd.h)
DEV_BITS = {
    0x01: "bad_token", 0x02: "nonfinite", 0x04: "empty_row", 0x08: "all_zero_weight",
    0x10: "pool_exhausted", 0x20: "table_overflow", 0x40: "bad_block", 0x80: "timeout",
}


class SmcError(RuntimeError):
    """A non-zero return code of a libsmcsd entry point."""

    def __init__(self, fn, code, text):
        super().__init__(f"{fn} returned {code}: {text}")
        self.code = code


class smc_params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
                ("V", ctypes.c_int32), ("dtype", ctypes.c_int32), ("alpha", ctypes.c_float),
                ("ess_frac", ctypes.c_float), ("seed", ctypes.c_uint64), ("step", ctypes.c_uint32)]


class smc_kv(ctypes.Structure):
    _fields_ = [("tables", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
                ("refcount", ctypes.c_void_p), ("free_list", ctypes.c_void_p),
                ("free_top", ctypes.c_void_p), ("cow_pairs", ctypes.c_void_p),
                ("n_cow", ctypes.c_void_p), ("T", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("P", ctypes.c_int32)]


class smc_step_opts(ctypes.Structure):
    _fields_ = [("log_potential", ctypes.c_void_p), ("temperature", ctypes.c_float),
                ("top_p", ctypes.c_float), ("reserved", ctypes.c_int32 * 2)]


_lib = None

_SIGS = {
    "smc_abi_version": (ctypes.c_int32, []),
    "smc_strerror": (ctypes.c_char_p, [ctypes.c_int32]),
    "smc_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(smc_params), ctypes.POINTER(smc_kv)]),
    "smc_workspace_init": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "smc_device_status": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]),
    "smc_step": (ctypes.c_int32, [ctypes.POINTER(smc_params)] + [ctypes.c_void_p] * 8 +
                 [ctypes.POINTER(smc_kv), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "smc_resample": (ctypes.c_int32, [ctypes.POINTER(smc_params)] + [ctypes.c_void_p] * 4 +
                     [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "kv_blocktable_remap": (ctypes.c_int32, [ctypes.POINTER(smc_params), ctypes.POINTER(smc_kv),
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "sps_verify": (ctypes.c_int32, [ctypes.POINTER(smc_params)] + [ctypes.c_void_p] * 5 +
                   [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "sps_verify_ex": (ctypes.c_int32, [ctypes.POINTER(smc_params)] + [ctypes.c_void_p] * 5 +
                      [ctypes.POINTER(smc_step_opts), ctypes.c_void_p, ctypes.c_size_t,
                       ctypes.c_void_p]),
    "smc_set_row_timing_events": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_void_p]),
    "smc_set_step_clock": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]),
    "smc_selftest_bounded_wait": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.c_void_p]),
    "smc_step_ex": (ctypes.c_int32, [ctypes.POINTER(smc_params), ctypes.POINTER(smc_step_opts)] +
                    [ctypes.c_void_p] * 8 +
                    [ctypes.POINTER(smc_kv), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "smc_draft_sample": (ctypes.c_int32, [ctypes.POINTER(smc_params), ctypes.c_void_p,
                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.c_void_p]),
    "smc_kv_usage": (ctypes.c_int32, [ctypes.POINTER(smc_params), ctypes.POINTER(smc_kv),
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
}


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m smc_speculative_decoding_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(fn, rc):
    if rc != 0:
        raise SmcError(fn, rc, lib().smc_strerror(rc).decode())


def _ptr(t, name, dtype=None, numel=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_params(B, N, K, V, dtype="bf16", alpha=1.0, ess_frac=0.5, seed=0, step=0):
    """smc_params for a shape; dtype is "bf16"/"f32" or a torch dtype."""
    if dtype in ("bf16", torch.bfloat16):
        code = SMC_BF16
    elif dtype in ("f32", torch.float32):
        code = SMC_F32
    else:
        raise ValueError(f"unsupported dtype {dtype!r}")
    return smc_params(int(B), int(N), int(K), int(V), code, float(alpha), float(ess_frac),
                      int(seed), int(step) & 0xFFFFFFFF)


_KV_KEYS = ("tables", "seq_len", "refcount", "free_list", "free_top", "cow_pairs", "n_cow")


def make_kv(params, kv, block_size):
    """smc_kv over a dict of int32 CUDA tensors (see workloads.make_kv_state)."""
    B, N = params.B, params.N
    T = kv["tables"].shape[-1]
    P = kv["free_list"].shape[-1]
    sizes = dict(tables=B * N * T, seq_len=B * N, refcount=B * P, free_list=B * P,
                 free_top=B, cow_pairs=B * N * 2, n_cow=B)
    ptrs = {k: _ptr(kv[k], f"kv[{k!r}]", torch.int32, sizes[k]) for k in _KV_KEYS}
    return smc_kv(*(ptrs[k] for k in _KV_KEYS), int(T), int(block_size), int(P))


def smc_abi_version():
    return lib().smc_abi_version()


def smc_strerror(code):
    return lib().smc_strerror(int(code)).decode()


def smc_workspace_bytes(params, kv=None):
    n = lib().smc_workspace_bytes(ctypes.byref(params), ctypes.byref(kv) if kv is not None else None)
    if n == 0:
        raise SmcError("smc_workspace_bytes", -1, "invalid shape")
    return n


def alloc_workspace(params, kv=None, device="cuda"):
    """A zero-filled workspace tensor of smc_workspace_bytes() bytes."""
    return torch.zeros(smc_workspace_bytes(params, kv), dtype=torch.uint8, device=device)


def smc_workspace_init(workspace, stream=None):
    _check("smc_workspace_init", lib().smc_workspace_init(
        _ptr(workspace, "workspace"), workspace.numel(), _stream(stream)))


def smc_device_status(workspace, clear=False, stream=None):
    """Device status bits of a workspace (synchronises the stream)."""
    out = ctypes.c_int32(0)
    _check("smc_device_status", lib().smc_device_status(
        _ptr(workspace, "workspace"), int(bool(clear)), ctypes.byref(out), _stream(stream)))
    return out.value


def smc_set_row_timing_events(rows_begin=None, rows_end=None):
    """Record two torch.cuda.Event objects (created with enable_timing=True)
    around the row pass of every later step; None, None turns it off.

    The events are recorded once here, on the current stream, so that torch
    creates them and treats them as recorded; the library records them
    again, around the row pass, at every later step."""
    def handle(ev):
        if ev is None:
            return None
        if not isinstance(ev, torch.cuda.Event):
            raise TypeError("expected a torch.cuda.Event")
        ev.record()
        return ctypes.c_void_p(ev.cuda_event)
    _check("smc_set_row_timing_events",
           lib().smc_set_row_timing_events(handle(rows_begin), handle(rows_end)))


def smc_set_step_clock(stamps=None, counter=None):
    """Device-side step clock: `stamps` (int64 CUDA tensor) receives the GPU
    timer (ns) as each later step's row pass starts, at index counter[0]++
    (`counter`: int32 CUDA tensor of one element, zeroed by the caller).
    None turns it off."""
    if stamps is None:
        _check("smc_set_step_clock", lib().smc_set_step_clock(None, None, 0))
        return
    if not (stamps.is_cuda and stamps.dtype == torch.int64 and counter is not None
            and counter.is_cuda and counter.dtype == torch.int32 and counter.numel() >= 1):
        raise TypeError("stamps: int64 CUDA tensor; counter: int32 CUDA tensor")
    _check("smc_set_step_clock",
           lib().smc_set_step_clock(ctypes.c_void_p(stamps.data_ptr()),
                                    ctypes.c_void_p(counter.data_ptr()), stamps.numel()))


def smc_selftest_bounded_wait(workspace, kind, poll_limit=1000, stream=None):
    """Run one of the library's bounded waits (kind 0: counter, 1: mbarrier)
    against a condition nothing satisfies; it raises the timeout status bit
    in `workspace` (a zeroed uint8 CUDA tensor of at least 8 bytes)."""
    _check("smc_selftest_bounded_wait",
           lib().smc_selftest_bounded_wait(ctypes.c_void_p(workspace.data_ptr()),
                                           workspace.numel() * workspace.element_size(),
                                           kind, poll_limit, _stream(stream)))


def status_names(bits):
    return [name for bit, name in DEV_BITS.items() if bits & bit]


def _logit_dtype(params):
    return torch.bfloat16 if params.dtype == SMC_BF16 else torch.float32


def smc_step(params, target_logits, draft_logits, draft_tokens, log_weights, tokens_out,
             ancestors, ess, resampled, kv=None, workspace=None, stream=None):
    B, N, K, V = params.B, params.N, params.K, params.V
    ld = _logit_dtype(params)
    args = [
        _ptr(target_logits, "target_logits", ld, B * N * (K + 1) * V),
        _ptr(draft_logits, "draft_logits", ld, B * N * K * V),
        _ptr(draft_tokens, "draft_tokens", torch.int32, B * N * K),
        _ptr(log_weights, "log_weights", torch.float32, B * N),
        _ptr(tokens_out, "tokens_out", torch.int32, B * N * (K + 1)),
        _ptr(ancestors, "ancestors", torch.int32, B * N),
        _ptr(ess, "ess", torch.float32, B),
        _ptr(resampled, "resampled", torch.int32, B),
    ]
    _check("smc_step", lib().smc_step(
        ctypes.byref(params), *args, ctypes.byref(kv) if kv is not None else None,
        _ptr(workspace, "workspace"), workspace.numel(), _stream(stream)))


def smc_step_ex(params, target_logits, draft_logits, draft_tokens, log_weights, tokens_out,
                ancestors, ess, resampled, kv=None, workspace=None, stream=None,
                temperature=1.0, log_potential=None, top_p=1.0):
    """smc_step with a temperature, a top-p nucleus and an optional [B, N]
    fp32 CUDA tensor of per-particle log-potential increments (smc_step_ex in
    smcsd.h)."""
    B, N, K, V = params.B, params.N, params.K, params.V
    ld = _logit_dtype(params)
    opts = smc_step_opts(
        _ptr(log_potential, "log_potential", torch.float32, B * N) if log_potential is not None
        else None, float(temperature), float(top_p))
    args = [
        _ptr(target_logits, "target_logits", ld, B * N * (K + 1) * V),
        _ptr(draft_logits, "draft_logits", ld, B * N * K * V),
        _ptr(draft_tokens, "draft_tokens", torch.int32, B * N * K),
        _ptr(log_weights, "log_weights", torch.float32, B * N),
        _ptr(tokens_out, "tokens_out", torch.int32, B * N * (K + 1)),
        _ptr(ancestors, "ancestors", torch.int32, B * N),
        _ptr(ess, "ess", torch.float32, B),
        _ptr(resampled, "resampled", torch.int32, B),
    ]
    _check("smc_step_ex", lib().smc_step_ex(
        ctypes.byref(params), ctypes.byref(opts), *args,
        ctypes.byref(kv) if kv is not None else None,
        _ptr(workspace, "workspace"), workspace.numel(), _stream(stream)))


def smc_draft_sample(params, draft_logits, position, tokens_out, workspace, stream=None):
    """One token per particle from softmax(alpha * l) of draft_logits [B, N, V]."""
    B, N, V = params.B, params.N, params.V
    _check("smc_draft_sample", lib().smc_draft_sample(
        ctypes.byref(params), _ptr(draft_logits, "draft_logits", _logit_dtype(params), B * N * V),
        int(position), _ptr(tokens_out, "tokens_out", torch.int32, B * N),
        _ptr(workspace, "workspace"), workspace.numel(), _stream(stream)))


def smc_kv_usage(params, kv, used_blocks, unshared_blocks, stream=None):
    """Per prompt: blocks in use with sharing, and blocks unshared copies would hold."""
    B = params.B
    _check("smc_kv_usage", lib().smc_kv_usage(
        ctypes.byref(params), ctypes.byref(kv), _ptr(used_blocks, "used_blocks", torch.int32, B),
        _ptr(unshared_blocks, "unshared_blocks", torch.int32, B), _stream(stream)))


def smc_resample(params, log_weights, ancestors, ess, resampled, workspace, stream=None):
    B, N = params.B, params.N
    _check("smc_resample", lib().smc_resample(
        ctypes.byref(params), _ptr(log_weights, "log_weights", torch.float32, B * N),
        _ptr(ancestors, "ancestors", torch.int32, B * N), _ptr(ess, "ess", torch.float32, B),
        _ptr(resampled, "resampled", torch.int32, B), _ptr(workspace, "workspace"),
        workspace.numel(), _stream(stream)))


def kv_blocktable_remap(params, kv, ancestors, resampled, n_append, workspace, stream=None):
    B, N = params.B, params.N
    _check("kv_blocktable_remap", lib().kv_blocktable_remap(
        ctypes.byref(params), ctypes.byref(kv), _ptr(ancestors, "ancestors", torch.int32, B * N),
        _ptr(resampled, "resampled", torch.int32, B), int(n_append),
        _ptr(workspace, "workspace"), workspace.numel(), _stream(stream)))


def sps_verify(params, target_logits, draft_logits, draft_tokens, tokens_out, n_emitted,
               workspace, stream=None):
    B, K, V = params.B, params.K, params.V
    ld = _logit_dtype(params)
    _check("sps_verify", lib().sps_verify(
        ctypes.byref(params), _ptr(target_logits, "target_logits", ld, B * (K + 1) * V),
        _ptr(draft_logits, "draft_logits", ld, B * K * V),
        _ptr(draft_tokens, "draft_tokens", torch.int32, B * K),
        _ptr(tokens_out, "tokens_out", torch.int32, B * (K + 1)),
        _ptr(n_emitted, "n_emitted", torch.int32, B),
        _ptr(workspace, "workspace"), workspace.numel(), _stream(stream)))


def sps_verify_ex(params, target_logits, draft_logits, draft_tokens, tokens_out, n_emitted,
                  workspace, stream=None, temperature=1.0, top_p=1.0):
    """sps_verify under a temperature and a top-p nucleus (sps_verify_ex in
    smcsd.h)."""
    B, K, V = params.B, params.K, params.V
    ld = _logit_dtype(params)
    opts = smc_step_opts(None, float(temperature), float(top_p))
    _check("sps_verify_ex", lib().sps_verify_ex(
        ctypes.byref(params), _ptr(target_logits, "target_logits", ld, B * (K + 1) * V),
        _ptr(draft_logits, "draft_logits", ld, B * K * V),
        _ptr(draft_tokens, "draft_tokens", torch.int32, B * K),
        _ptr(tokens_out, "tokens_out", torch.int32, B * (K + 1)),
        _ptr(n_emitted, "n_emitted", torch.int32, B), ctypes.byref(opts),
        _ptr(workspace, "workspace"), workspace.numel(), _stream(stream)))


def smc_step_noalloc(params, target_logits, draft_logits, draft_tokens, log_weights, tokens_out,
                     ancestors, ess, resampled, status_bits, kv=None, stream=None):
    """smc_step without a caller workspace: the library's own fixed scratch
    array is used (see smc_step_noalloc in smcsd.h).  status_bits is a CUDA
    int32 tensor of one element that receives this call's device status."""
    fn = lib().smc_step_noalloc
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(smc_params)] + [ctypes.c_void_p] * 8 + \
        [ctypes.POINTER(smc_kv), ctypes.c_void_p, ctypes.c_void_p]
    B, N, K, V = params.B, params.N, params.K, params.V
    ld = _logit_dtype(params)
    args = [
        _ptr(target_logits, "target_logits", ld, B * N * (K + 1) * V),
        _ptr(draft_logits, "draft_logits", ld, B * N * K * V),
        _ptr(draft_tokens, "draft_tokens", torch.int32, B * N * K),
        _ptr(log_weights, "log_weights", torch.float32, B * N),
        _ptr(tokens_out, "tokens_out", torch.int32, B * N * (K + 1)),
        _ptr(ancestors, "ancestors", torch.int32, B * N),
        _ptr(ess, "ess", torch.float32, B),
        _ptr(resampled, "resampled", torch.int32, B),
    ]
    _check("smc_step_noalloc", fn(ctypes.byref(params), *args,
                                  ctypes.byref(kv) if kv is not None else None,
                                  _ptr(status_bits, "status_bits", torch.int32, 1),
                                  _stream(stream)))
