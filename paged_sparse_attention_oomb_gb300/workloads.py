"""Named workloads and the seeded synthetic input generator.

This module holds sizes and random numbers only -- none of the method's
arithmetic -- so that both the CUDA path and the CPU oracle can be fed the
same stored tensors.

Recipe (one ``torch.Generator`` seeded with ``seed``, drawn in this order):

1. page centroids ``[N, Hkv, D] ~ N(0, 0.5^2)``;
2. keys, page block by page block (``PAGE_BLOCK`` pages at a time):
   centroid + ``N(0, 1)`` noise, then rounded to the storage dtype;
3. values ``[N, Hkv, P, D] ~ N(0, 1)``, same page blocks;
4. queries ``[C, Hq, D] ~ N(0, 1)``;
5. output gradients ``[C, Hq, D] ~ N(0, 1)``;
6. if the workload shuffles its page table: ``randperm(N)`` (logical page ->
   physical slot), otherwise the identity.

Values are drawn in fp32 and rounded once (round-to-nearest-even) to the
storage dtype.  Pools are stored by physical slot: the key of logical page l
lives in slot ``page_table[l]``.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

PAGE_BLOCK = 2048


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "bf16" or "fp32"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    context: int          # tokens in the paged cache (= num_pages * page_size)
    page_size: int
    chunk_len: int
    top_k: int            # pages kept per (chunk, KV head); >= candidates means all
    shuffled: bool = False
    chunk_start: int = -1  # -1: the last chunk of the context

    @property
    def num_pages(self):
        return self.context // self.page_size

    @property
    def start(self):
        return self.context - self.chunk_len if self.chunk_start < 0 else self.chunk_start

    @property
    def num_candidates(self):
        return self.start // self.page_size

    @property
    def n_sel(self):
        return min(self.top_k, self.num_candidates)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def with_(self, **kw):
        return replace(self, **kw)


# The five workloads of the method's evaluation ladder: a tiny fp32 check and
# Qwen2.5-7B-shaped attention (28 query heads, 4 KV heads, head_dim 128) at
# 32K, 256K, 1M and 4M tokens of context.
WORKLOADS = {
    "tiny_fp32_ctx1k": Workload("tiny_fp32_ctx1k", "fp32", 2, 1, 64, 1024, 16, 128, 8),
    "qwen7b_dense_ctx32k": Workload("qwen7b_dense_ctx32k", "bf16", 28, 4, 128, 32768, 64,
                                    4096, 1 << 30),
    "qwen7b_ctx256k_k64": Workload("qwen7b_ctx256k_k64", "bf16", 28, 4, 128, 262144, 64,
                                   4096, 64),
    "qwen7b_ctx1m_k128": Workload("qwen7b_ctx1m_k128", "bf16", 28, 4, 128, 1048576, 64,
                                  4096, 128, shuffled=True),
    "qwen7b_ctx4m_k128": Workload("qwen7b_ctx4m_k128", "bf16", 28, 4, 128, 4194304, 128,
                                  8192, 128, shuffled=True),
}


@dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor           # [C, Hq, D]
    k_pool: torch.Tensor      # [N, Hkv, P, D] by physical slot
    v_pool: torch.Tensor
    do: torch.Tensor          # [C, Hq, D]
    page_table: torch.Tensor  # int32 [N]
    extra: dict = field(default_factory=dict)


def make_inputs(wl: Workload, seed: int = 0, device="cpu") -> Inputs:
    """Draw the synthetic tensors of ``wl`` on ``device`` (see module recipe)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    n, hkv, p, d = wl.num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim
    dt = wl.torch_dtype
    cent = torch.randn((n, hkv, d), generator=gen, device=dev) * 0.5
    k_logical = torch.empty((n, hkv, p, d), dtype=dt, device=dev)
    for b0 in range(0, n, PAGE_BLOCK):
        b1 = min(n, b0 + PAGE_BLOCK)
        noise = torch.randn((b1 - b0, hkv, p, d), generator=gen, device=dev)
        k_logical[b0:b1] = (noise + cent[b0:b1, :, None, :]).to(dt)
        del noise
    del cent
    v_logical = torch.empty((n, hkv, p, d), dtype=dt, device=dev)
    for b0 in range(0, n, PAGE_BLOCK):
        b1 = min(n, b0 + PAGE_BLOCK)
        v_logical[b0:b1] = torch.randn((b1 - b0, hkv, p, d), generator=gen, device=dev).to(dt)
    q = torch.randn((wl.chunk_len, wl.num_q_heads, d), generator=gen, device=dev).to(dt)
    do = torch.randn((wl.chunk_len, wl.num_q_heads, d), generator=gen, device=dev).to(dt)
    if wl.shuffled:
        pt = torch.randperm(n, generator=gen, device=dev).to(torch.int32)
        # place logical page l at slot pt[l]
        k_pool = torch.empty_like(k_logical)
        v_pool = torch.empty_like(v_logical)
        idx = pt.long()
        k_pool.index_copy_(0, idx, k_logical)
        del k_logical
        v_pool.index_copy_(0, idx, v_logical)
        del v_logical
    else:
        pt = torch.arange(n, dtype=torch.int32, device=dev)
        k_pool, v_pool = k_logical, v_logical
    return Inputs(wl, q.contiguous(), k_pool, v_pool, do.contiguous(), pt)


def to_numpy64(t: torch.Tensor):
    """Exact widening of a stored tensor to a float64 (or int64) host array."""
    t = t.detach().to("cpu")
    if t.is_floating_point():
        return t.to(torch.float64).numpy()
    return t.to(torch.int64).numpy()
