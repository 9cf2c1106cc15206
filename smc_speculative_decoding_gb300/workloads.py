"""Seeded synthetic inputs for the SMC-SD step: logits, drafted tokens, KV state.

This module holds no arithmetic of the step itself: it draws Gaussian logits,
adds a rank-based peak, perturbs them into draft logits, draws drafted tokens
with ``torch.multinomial`` and lays out an initial paged KV state.  Both the
CUDA path and the CPU oracle are fed from here, so neither generates its own
inputs.

Logit recipe (the workloads the method is described on use Llama- and
Qwen-family vocabularies; no model or dataset is involved here):
  * target logits l ~ N(0, sigma_t^2), i.i.d. per row;
  * the top-M entries of each row (by value) get +boost / r, r = 1..M the rank;
  * draft logits = target logits of the same position + N(0, sigma_d^2);
  * rows are cast to the storage dtype (bf16 rounds to nearest even);
  * drafted token x_k ~ softmax(stored draft row k), drawn by torch.multinomial.
Every row is independent: positions, particles and steps do not condition on
one another.
"""
from dataclasses import dataclass, replace
import math

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """Shape and generator parameters of one synthetic workload."""
    name: str
    B: int               # prompts
    N: int               # particles per prompt
    K: int               # drafted tokens per particle per step
    V: int               # vocabulary size
    dtype: str           # "f32" or "bf16" storage of the logits
    sigma_t: float       # std of target logits
    top_m: int           # size of the rank-boosted peak (0: none)
    sigma_d: float       # std of the draft perturbation
    alpha: float = 1.0   # power-sampling exponent of the target
    ess_frac: float = 0.5
    steps: int = 10
    prefix: int = 16     # shared prompt tokens held in the KV tables
    block_size: int = 16
    boost: float = 4.0

    @property
    def rows(self):
        """Logit rows read per step: B*N*(2K+1)."""
        return self.B * self.N * (2 * self.K + 1)

    @property
    def bytes_per_logit(self):
        return 2 if self.dtype == "bf16" else 4

    @property
    def particle_tokens(self):
        """Tokens emitted per step: B*N*(K+1)."""
        return self.B * self.N * (self.K + 1)

    def kv_dims(self, steps=None):
        """(T, P): table length per particle and pool blocks per prompt that
        hold the prefix plus ``steps`` appends of K+1 tokens with no sharing."""
        steps = self.steps if steps is None else steps
        t_len = math.ceil((self.prefix + steps * (self.K + 1)) / self.block_size) + 1
        return t_len, self.N * t_len + 1

    def with_(self, **kw):
        return replace(self, **kw)


#: the workloads, named by what they are
WORKLOADS = {
    "tiny_v64": Workload("tiny_v64", B=1, N=4, K=3, V=64, dtype="f32", sigma_t=2.0,
                         top_m=0, sigma_d=0.5, steps=10, prefix=16),
    "single_prompt_v32000": Workload("single_prompt_v32000", B=1, N=8, K=4, V=32000,
                                     dtype="bf16", sigma_t=3.0, top_m=50, sigma_d=1.0,
                                     steps=256, prefix=512),
    "batched_serving_v128256": Workload("batched_serving_v128256", B=16, N=16, K=4,
                                        V=128256, dtype="bf16", sigma_t=3.0, top_m=50,
                                        sigma_d=1.0, steps=128, prefix=2048),
    "power_sampling_v151936": Workload("power_sampling_v151936", B=8, N=32, K=8,
                                       V=151936, dtype="f32", sigma_t=2.5, top_m=100,
                                       sigma_d=0.75, alpha=4.0, steps=64, prefix=512),
    "sweep_v128256": Workload("sweep_v128256", B=32, N=8, K=4, V=128256, dtype="bf16",
                              sigma_t=3.0, top_m=50, sigma_d=1.0, steps=32, prefix=512),
}

#: draft-noise levels of the serving sweep and the (N, K) grid of the sweep
SERVING_SIGMAS = (0.25, 1.0, 2.0)
SWEEP_N = (1, 2, 4, 8, 16, 32, 64)
SWEEP_K = (2, 4, 8)


def torch_dtype(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def _peaked_gaussian(shape, sigma, top_m, boost, gen, device):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * sigma
    if top_m:
        _, idx = x.topk(top_m, dim=-1)
        bump = boost / torch.arange(1, top_m + 1, device=device, dtype=torch.float32)
        x.scatter_add_(-1, idx, bump.expand(idx.shape).contiguous())
    return x


def make_logits(w, seed, device="cpu", step=0):
    """Target [B,N,K+1,V] and draft [B,N,K,V] logits in the storage dtype."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 1_000_003 + int(step))
    shape_t = (w.B, w.N, w.K + 1, w.V)
    target = _peaked_gaussian(shape_t, w.sigma_t, w.top_m, w.boost, gen, device)
    noise = torch.randn((w.B, w.N, w.K, w.V), generator=gen, device=device,
                        dtype=torch.float32)
    draft = target[:, :, :w.K] + w.sigma_d * noise
    del noise
    dt = torch_dtype(w.dtype)
    return target.to(dt).contiguous(), draft.to(dt).contiguous(), gen


def draw_tokens(draft, gen, rows_per_call=256):
    """x ~ softmax(draft row) for every draft row, by torch.multinomial."""
    big_b, n_part, k_drafts, v_size = draft.shape
    flat = draft.reshape(-1, v_size)
    out = torch.empty(flat.shape[0], dtype=torch.int64, device=draft.device)
    for s in range(0, flat.shape[0], rows_per_call):
        probs = torch.softmax(flat[s:s + rows_per_call].float(), dim=-1)
        out[s:s + rows_per_call] = torch.multinomial(probs, 1, generator=gen).squeeze(1)
    return out.reshape(big_b, n_part, k_drafts).to(torch.int32)


def make_step_inputs(w, seed, device="cpu", step=0):
    """dict(target, draft, draft_tokens) for one step of workload ``w``."""
    target, draft, gen = make_logits(w, seed, device, step)
    tokens = draw_tokens(draft, gen)
    return dict(target=target, draft=draft, draft_tokens=tokens)


def make_kv_state(B, N, prefix, block_size, T, P, device="cpu"):
    """Initial paged KV state: every particle of a prompt shares the prefix.

    tables [B,N,T] (-1 past the used blocks), seq_len [B,N], refcount [B*P],
    free_list [B,P] (prompt b's free ids, the lowest id on top), free_top [B],
    cow_pairs [B,N,2], n_cow [B]; all int32.
    """
    nb = (prefix + block_size - 1) // block_size
    if nb > T or nb > P:
        raise ValueError("prefix does not fit the table or the pool")
    tables = torch.full((B, N, T), -1, dtype=torch.int32)
    refcount = torch.zeros(B * P, dtype=torch.int32)
    free_list = torch.zeros((B, P), dtype=torch.int32)
    free_top = torch.zeros(B, dtype=torch.int32)
    for b in range(B):
        ids = torch.arange(b * P, b * P + nb, dtype=torch.int32)
        tables[b, :, :nb] = ids
        refcount[b * P: b * P + nb] = N
        free = torch.arange(b * P + P - 1, b * P + nb - 1, -1, dtype=torch.int32)
        free_list[b, :free.numel()] = free
        free_top[b] = free.numel()
    seq_len = torch.full((B, N), prefix, dtype=torch.int32)
    cow_pairs = torch.full((B, N, 2), -1, dtype=torch.int32)
    n_cow = torch.zeros(B, dtype=torch.int32)
    state = dict(tables=tables, seq_len=seq_len, refcount=refcount, free_list=free_list,
                 free_top=free_top, cow_pairs=cow_pairs, n_cow=n_cow)
    return {k: v.to(device) for k, v in state.items()}


def bf16_bits(t):
    """Raw uint16 bit patterns of a bfloat16 tensor, as a numpy array."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_numpy_logits(t):
    """Stored logits as numpy: uint16 bit patterns for bf16, float32 otherwise."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().float().numpy()
