"""Seeded synthetic inputs for paged-KV decode attention.

This module only draws random tensors and lays them out as a paged cache; it
holds none of the attention arithmetic.  Both the CUDA path and the float64
oracle consume what it returns, so it imports neither.

Layouts follow the FlashInfer ``xqa`` API page: q [B, q_seq_len, Hq, D];
caches [num_pages, page_size, Hkv, D] (NHD) or [num_pages, Hkv, page_size, D]
(HND); page_table int32 [B, pages_per_seq] shared by K and V; seq_lens uint32
[B]; sinks fp32 [Hkv, Hq / Hkv]; mask uint16 [B, q_seq_len,
((q_seq_len + 31) // 32) * 2], bit-packed into little-endian 32-bit words.

Pool recipe: the pool holds exactly the pages the sequences need (or a fixed
pool size), a seeded permutation assigns them, and table entries past a
sequence's last page point at arbitrary valid pages.  With ``poison=True``
every pool page no sequence uses and every slot past seq_len in a sequence's
last page holds NaN, so a kernel that reads masked data shows NaN instead of
faulting.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

E4M3_NAN_BITS = 0x7F


@dataclasses.dataclass
class Case:
    name: str
    q: torch.Tensor  # [B, q_seq_len, Hq, D]
    k_cache: torch.Tensor
    v_cache: torch.Tensor  # the same tensor object as k_cache for the MLA variant
    page_table: torch.Tensor  # int32 [B, pages_per_seq]
    seq_lens: torch.Tensor  # int32 storage of uint32 lengths, [B]
    num_kv_heads: int
    page_size: int
    kv_layout: str
    q_seq_len: int = 1
    v_head_dim: Optional[int] = None
    sinks: Optional[torch.Tensor] = None
    mask: Optional[torch.Tensor] = None  # int16 storage of uint16 words
    q_scale: float = 1.0
    kv_scale: float = 1.0
    softmax_scale: Optional[float] = None
    sliding_win_size: int = 0
    rcp_out_scale: float = 1.0
    mla: bool = False

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def num_q_heads(self):
        return self.q.shape[2]

    @property
    def head_dim(self):
        return self.q.shape[3]

    @property
    def dv(self):
        return self.head_dim if self.v_head_dim is None else self.v_head_dim

    def kwargs(self):
        """Keyword arguments shared by the oracle and the CUDA binding."""
        return dict(num_kv_heads=self.num_kv_heads, page_size=self.page_size,
                    kv_layout=self.kv_layout, v_head_dim=self.v_head_dim, sinks=self.sinks,
                    q_scale=self.q_scale, kv_scale=self.kv_scale,
                    softmax_scale=self.softmax_scale, sliding_win_size=self.sliding_win_size,
                    rcp_out_scale=self.rcp_out_scale, mask=self.mask)

    def to(self, device):
        out = dataclasses.replace(self)
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            if isinstance(v, torch.Tensor):
                setattr(out, f.name, v.to(device))
        if self.v_cache is self.k_cache:
            out.v_cache = out.k_cache
        return out

    def visible_tokens(self):
        """Tokens a query row of each sequence reads, summed over the batch
        (the window bounds them when one is set)."""
        lens = self.seq_lens.to(torch.int64).cpu()
        if self.sliding_win_size > 0:
            lens = torch.clamp(lens, max=self.sliding_win_size + self.q_seq_len - 1)
        return int(lens.sum())

    def kv_bytes(self):
        """Algorithmic KV bytes: every visible token's K row and V row once
        (the MLA latent row once, since V is its prefix)."""
        elt = self.k_cache.element_size()
        per_tok = self.head_dim * elt * self.num_kv_heads * (1 if self.mla else 2)
        return self.visible_tokens() * per_tok

    def q_bytes(self):
        return self.q.numel() * self.q.element_size()


def _randn(shape, gen, device, chunk=1 << 27):
    """N(0,1) float32 drawn in bounded chunks (keeps peak memory small)."""
    out = torch.empty(shape, dtype=torch.float32, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        flat[s:s + n] = torch.randn(n, generator=gen, device=device)
    return out


def _randn_as(shape, dtype, gen, device, divisor=1.0, chunk=1 << 26):
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        x = torch.randn(n, generator=gen, device=device)
        if divisor != 1.0:
            x = x / divisor
        flat[s:s + n] = x.to(dtype)
    return out


def pack_mask(allowed):
    """Bit-pack a boolean [B, q_seq_len, q_seq_len] "query i may see new token
    j" array into uint16 words (returned as int16 storage): bit j % 32 of the
    little-endian 32-bit word j // 32, each word split into two uint16."""
    allowed = torch.as_tensor(allowed, dtype=torch.bool)
    B, qs, _ = allowed.shape
    nwords = (qs + 31) // 32
    w32 = torch.zeros((B, qs, nwords), dtype=torch.int64)
    for j in range(qs):
        w32[..., j // 32] |= allowed[..., j].to(torch.int64) << (j % 32)
    m16 = torch.stack([w32 & 0xFFFF, (w32 >> 16) & 0xFFFF], dim=-1).reshape(B, qs, 2 * nwords)
    return torch.where(m16 >= 0x8000, m16 - 0x10000, m16).to(torch.int16)


def causal_spec_mask(batch, q_seq_len, device="cpu"):
    """Lower-triangular speculative mask: query token i sees new tokens 0..i."""
    tri = torch.ones(q_seq_len, q_seq_len, dtype=torch.bool).tril()
    return pack_mask(tri.expand(batch, q_seq_len, q_seq_len)).to(device)


def full_spec_mask(batch, q_seq_len, device="cpu"):
    """All-ones speculative mask: every new token visible to every query."""
    return pack_mask(torch.ones(batch, q_seq_len, q_seq_len, dtype=torch.bool)).to(device)


def make_case(*, batch, num_q_heads, num_kv_heads, head_dim, page_size, seq_lens,
              kv_layout="NHD", q_dtype=torch.bfloat16, kv_dtype=None, q_seq_len=1,
              v_head_dim=None, mla=False, q_scale=1.0, kv_scale=1.0, kv_divisor=1.0, q_divisor=1.0,
              softmax_scale=None, sinks=False, sliding_win_size=0, mask=None,
              rcp_out_scale=1.0, pool_pages=None, pages_per_seq=None, seed=0,
              device="cpu", poison=True, q_mult=1.0, name="case"):
    """Build one seeded problem.  seq_lens: list of ints.  mask: None,
    "causal" or "full".  kv_divisor: K/V drawn as N(0,1)/kv_divisor before the
    cast to kv_dtype (the fp8 recipe uses 1/kv_scale); q_divisor likewise for
    q (an e4m3 query is drawn as N(0,1)/q_scale)."""
    kv_dtype = q_dtype if kv_dtype is None else kv_dtype
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    hkv = 1 if mla else num_kv_heads
    lens = [int(x) for x in seq_lens]
    npages_seq = [max(0, math.ceil(L / page_size)) for L in lens]
    pps = pages_per_seq if pages_per_seq is not None else max(1, max(npages_seq))
    if max(npages_seq) > pps:
        raise ValueError("pages_per_seq too small for seq_lens")
    need = sum(npages_seq)
    num_pages = max(need, 1) if pool_pages is None else int(pool_pages)
    if num_pages < need:
        raise ValueError("pool too small")
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed + 7919))
    filler = torch.randint(0, num_pages, (batch, pps),
                           generator=torch.Generator().manual_seed(seed + 104729))
    table = filler.to(torch.int32).clone()
    off = 0
    for b, n in enumerate(npages_seq):
        table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n

    q = _randn_as((batch, q_seq_len, num_q_heads, head_dim), q_dtype, gen, device, divisor=q_divisor)
    if q_mult != 1.0:
        q = (q.float() * q_mult).to(q_dtype)
    if kv_layout.upper() == "NHD":
        shape = (num_pages, page_size, hkv, head_dim)
    else:
        shape = (num_pages, hkv, page_size, head_dim)
    k_cache = _randn_as(shape, kv_dtype, gen, device, divisor=kv_divisor)
    v_cache = k_cache if mla else _randn_as(shape, kv_dtype, gen, device, divisor=kv_divisor)

    if poison:
        used = torch.zeros(num_pages, dtype=torch.bool)
        used[perm[:need]] = True
        caches = [k_cache] if mla else [k_cache, v_cache]
        for c in caches:
            nan_fill(c, torch.nonzero(~used).flatten().to(device), None, kv_layout)
            for b, L in enumerate(lens):
                if L % page_size and npages_seq[b] > 0:
                    last = int(table[b, npages_seq[b] - 1])
                    nan_fill(c, torch.tensor([last], device=device), L % page_size, kv_layout)

    sink_t = None
    if sinks:
        sink_t = _randn((hkv, num_q_heads // hkv), gen, device)
    mask_t = None
    if mask == "causal":
        mask_t = causal_spec_mask(batch, q_seq_len, device)
    elif mask == "full":
        mask_t = full_spec_mask(batch, q_seq_len, device)
    return Case(name=name, q=q, k_cache=k_cache, v_cache=v_cache, page_table=table.to(device),
                seq_lens=torch.tensor(lens, dtype=torch.int32, device=device),
                num_kv_heads=hkv, page_size=page_size, kv_layout=kv_layout.upper(),
                q_seq_len=q_seq_len, v_head_dim=v_head_dim, sinks=sink_t, mask=mask_t,
                q_scale=q_scale, kv_scale=kv_scale, softmax_scale=softmax_scale,
                sliding_win_size=sliding_win_size, rcp_out_scale=rcp_out_scale, mla=mla)


def nan_fill(cache, pages, from_slot, layout):
    """Write NaN into whole pages (from_slot None) or their slots >= from_slot."""
    if pages.numel() == 0:
        return
    if cache.dtype == torch.float8_e4m3fn:
        view = cache.view(torch.uint8)
        val = E4M3_NAN_BITS
    else:
        view = cache
        val = float("nan")
    s = 0 if from_slot is None else from_slot
    for p in pages.tolist():
        if layout.upper() == "NHD":
            view[p, s:] = val
        else:
            view[p, :, s:] = val


# ---------------------------------------------------------------------------
# The five named workloads (seed = workload index).

def _uniform_lens(lo, hi, batch, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (batch,), generator=g).tolist()


WORKLOADS = {
    1: "tiny GQA decode (B2 Hq8 Hkv2 D128 ps16 L{37,100} NHD bf16)",
    2: "Llama-3-8B-shaped decode (B64 Hq32 Hkv8 D128 ps64 L~U[1024,8192] HND bf16)",
    3: "fp8 KV long-context decode (B128 Hq64 Hkv8 D128 ps32 L=32768 NHD e4m3 kv_scale=0.05)",
    4: "sliding-window + sinks + speculative decode (B32 Hq64 Hkv8 D64 ps16 "
       "L~U[2048,16384] W128 q_seq_len4 causal mask NHD bf16)",
    5: "MLA latent decode (B64 Hq128 latent 576/512 ps64 L~U[4096,32768] bf16)",
}
# The e4m3 variant of workload 5: the same shapes and lengths with an e4m3
# latent cache and an e4m3 query (vLLM Kimi-K3 MultiHeadLatentAttention page:
# an fp8 cache takes an fp8 query), both drawn as N(0,1)/scale with
# q_scale = kv_scale = 0.05 (the fp8 recipe of workload 3).
WORKLOAD_5_E4M3 = ("MLA latent decode, e4m3 latent cache and query (B64 Hq128 latent 576/512 ps64 "
                   "L~U[4096,32768] q_scale=kv_scale=0.05)")


LARGE_GROUP = ("speculative decode on a large group (B64 Hq128 Hkv8 D128 ps64 L~U[1024,8192] HND bf16, "
               "q_seq_len4 causal mask: 64 query rows per kv head)")


def large_group_workload(device="cpu", poison=True, batch=None):
    """The Llama-3-8B-shaped cache (workload 2's lengths and pool) with four
    speculative tokens and a group of 16 query heads per kv head: 64 rows per
    kv head, the tile the grouped-query kernel's warp row groups serve in one
    pass over the pages."""
    B = 64
    lens = _uniform_lens(1024, 8192, B, 2)[: batch or B]
    return make_case(batch=len(lens), num_q_heads=128, num_kv_heads=8, head_dim=128, page_size=64,
                     seq_lens=lens, kv_layout="HND", q_seq_len=4, mask="causal",
                     pages_per_seq=8192 // 64, seed=12, device=device, poison=poison,
                     name="large_group_spec")


def workload(idx, device="cpu", poison=True, batch=None, kv_dtype=None):
    """The named workload idx (1..5); `batch` truncates B for smaller runs
    while keeping every other size.  kv_dtype=torch.float8_e4m3fn with idx 5
    gives its e4m3 variant (e4m3 latent cache and query)."""
    if kv_dtype is not None and not (idx == 5 and kv_dtype == torch.float8_e4m3fn):
        raise ValueError("only workload 5 has a kv_dtype variant (torch.float8_e4m3fn)")
    seed = idx
    if idx == 1:
        # 16-page pool, seq0 takes 3 pages and seq1 takes 7.
        return make_case(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                         seq_lens=[37, 100], kv_layout="NHD", pool_pages=16, seed=seed,
                         device=device, poison=poison, name="tiny_gqa")
    if idx == 2:
        B = 64
        lens = _uniform_lens(1024, 8192, B, seed)[: batch or B]
        return make_case(batch=len(lens), num_q_heads=32, num_kv_heads=8, head_dim=128,
                         page_size=64, seq_lens=lens, kv_layout="HND",
                         pages_per_seq=8192 // 64, seed=seed, device=device, poison=poison,
                         name="llama3_8b_decode")
    if idx == 3:
        B = batch or 128
        return make_case(batch=B, num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=32,
                         seq_lens=[32768] * B, kv_layout="NHD", q_dtype=torch.bfloat16,
                         kv_dtype=torch.float8_e4m3fn, kv_scale=0.05, kv_divisor=0.05,
                         q_scale=1.0, pages_per_seq=32768 // 32, seed=seed, device=device,
                         poison=poison, name="fp8_long_context")
    if idx == 4:
        B = 32
        lens = _uniform_lens(2048, 16384, B, seed)[: batch or B]
        return make_case(batch=len(lens), num_q_heads=64, num_kv_heads=8, head_dim=64,
                         page_size=16, seq_lens=lens, kv_layout="NHD", q_seq_len=4,
                         sinks=True, sliding_win_size=128, mask="causal",
                         pages_per_seq=16384 // 16, seed=seed, device=device, poison=poison,
                         name="window_sinks_spec")
    if idx == 5:
        B = 64
        lens = _uniform_lens(4096, 32768, B, seed)[: batch or B]
        f8 = kv_dtype == torch.float8_e4m3fn
        dt = torch.float8_e4m3fn if f8 else torch.bfloat16
        scale = 0.05 if f8 else 1.0
        return make_case(batch=len(lens), num_q_heads=128, num_kv_heads=1, head_dim=576,
                         v_head_dim=512, mla=True, page_size=64, seq_lens=lens,
                         kv_layout="NHD", softmax_scale=(128 + 64) ** -0.5, q_dtype=dt,
                         kv_dtype=dt, q_scale=scale, kv_scale=scale, q_divisor=scale,
                         kv_divisor=scale, pages_per_seq=32768 // 64, seed=seed, device=device,
                         poison=poison, name="mla_latent_decode_e4m3" if f8 else "mla_latent_decode")
    raise ValueError(f"unknown workload {idx}")
