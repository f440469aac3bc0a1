"""Float64 CPU oracle for paged-KV decode attention.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline and reference legs are the only callers.  The product path (the
CUDA library and its binding in ``paged_kv_decode_20_gb300``) never imports
this package, and this package never imports that one.

The arithmetic lives in ``xqa_oracle.c`` (plain C loops in double precision,
OpenMP over output rows); this module only compiles it with gcc, marshals
CPU tensors and calls it.  Semantics follow the FlashInfer ``xqa`` API page
(parameter list and shape-inference note) and, for the MLA latent variant, the
vLLM Kimi-K3 MultiHeadLatentAttention page (``head_size``, ``scale`` and the
``forward_mqa`` call): see the header of ``xqa_oracle.c``.
"""

from __future__ import annotations

import ctypes
import hashlib
import math
import os
import platform
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "xqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_xqa.so")
_lock = threading.Lock()
_lib = None

# element codes of the oracle's own C entry point
_F16, _BF16, _E4M3 = 0, 1, 2
_DTYPE_CODE = {torch.float16: _F16, torch.bfloat16: _BF16, torch.float8_e4m3fn: _E4M3}


_GCC = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11"]


def _digest() -> str:
    """SHA-256 of the source, the compiler flags and the host machine."""
    h = hashlib.sha256()
    with open(_SRC, "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(_GCC).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile xqa_oracle.c into a shared library (gcc, -O2, OpenMP); rebuilt
    whenever the source's content (not its modification time) changes."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    digest, stamp = _digest(), _LIB_PATH + ".sha256"
    current = os.path.exists(_LIB_PATH) and os.path.exists(stamp) and open(stamp).read().strip() == digest
    if force or not current:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(_GCC + ["-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
        with open(stamp + f".{os.getpid()}.tmp", "w") as fh:
            fh.write(digest + "\n")
        os.replace(stamp + f".{os.getpid()}.tmp", stamp)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_xqa_attention.restype = ctypes.c_int
            lib.oracle_xqa_attention.argtypes = [
                ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_void_p, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ]
            lib.oracle_merge_attn_states.restype = None
            lib.oracle_merge_attn_states.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 4 + [
                ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_encode_e4m3.restype = ctypes.c_uint32
            lib.oracle_encode_e4m3.argtypes = [ctypes.c_double]
            lib.oracle_decode.restype = ctypes.c_double
            lib.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
            _lib = lib
    return _lib


def decode(dtype: torch.dtype, bits: int) -> float:
    """Decode one element from its bit pattern, as the oracle does."""
    return _load().oracle_decode(_DTYPE_CODE[dtype], bits)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _cpu_contig(t, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        t = torch.as_tensor(np.asarray(t))
    t = t.detach().to("cpu")
    if dtype is not None and t.dtype != dtype:
        t = t.to(dtype)
    return t.contiguous()


def xqa_attention(q, k_cache, v_cache, page_table, seq_lens, *, num_kv_heads, page_size,
                  kv_layout="NHD", v_head_dim=None, sinks=None, q_scale=1.0, kv_scale=1.0,
                  softmax_scale=None, sliding_win_size=0, rcp_out_scale=1.0, q_seq_len=None,
                  mask=None, units=None, threads=0, return_lse=False):
    """Exact float64 paged decode attention.

    q: [B, q_seq_len, Hq, D] (or [B, Hq, D]) fp16/bf16, or float8_e4m3fn (the
    fp8 query an fp8 latent cache takes; decoded like the cache).  k_cache, v_cache:
    [num_pages, page_size, Hkv, D] (NHD) or [num_pages, Hkv, page_size, D]
    (HND), fp16/bf16/float8_e4m3fn; for the MLA variant pass the same latent
    cache twice and v_head_dim < D.  page_table: int32 [B, pages_per_seq].
    seq_lens: [B] (uint32 semantics).  softmax_scale None means 1/sqrt(D).
    units: optional flat row ids (b * q_seq_len + i) * Hq + h; the result is
    then [len(units), Dv], otherwise [B, q_seq_len, Hq, Dv].  float64 tensor.
    return_lse: also return each row's log-sum-exp (natural log of the
    normaliser the output was divided by, sink included; -inf for an empty
    row), shaped [len(units)] or [B, q_seq_len, Hq].
    """
    q = _cpu_contig(q)
    if q.dim() == 3:
        q = q.unsqueeze(1)
    B, qs, Hq, D = q.shape
    if q_seq_len is not None and q_seq_len != qs:
        raise ValueError(f"q has {qs} query tokens per sequence, q_seq_len={q_seq_len}")
    k_cache = _cpu_contig(k_cache)
    v_cache = k_cache if v_cache is None else _cpu_contig(v_cache)
    if k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must share one dtype")
    if k_cache.shape[-1] != D:
        raise ValueError("cache head_dim differs from q head_dim")
    Dv = D if v_head_dim is None else int(v_head_dim)
    page_table = _cpu_contig(page_table, torch.int32)
    seq_lens = _cpu_contig(seq_lens).to(torch.int64).to(torch.int32)  # uint32 bits
    sinks = _cpu_contig(sinks, torch.float32)
    mask = _cpu_contig(mask)
    if mask is not None:
        mask = mask.view(torch.int16) if mask.dtype == torch.uint16 else mask.to(torch.int16)
        words = ((qs + 31) // 32) * 2
        if tuple(mask.shape) != (B, qs, words):
            raise ValueError(f"mask must be [{B}, {qs}, {words}], got {tuple(mask.shape)}")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    layout_hnd = {"NHD": 0, "HND": 1}[kv_layout.upper()]
    q_bits = q.view(torch.uint8) if q.dtype == torch.float8_e4m3fn else q.view(torch.int16)
    kv_code = _DTYPE_CODE[k_cache.dtype]
    k_bits = k_cache.view(torch.uint8) if kv_code == _E4M3 else k_cache.view(torch.int16)
    v_bits = v_cache.view(torch.uint8) if kv_code == _E4M3 else v_cache.view(torch.int16)
    if units is not None:
        units = _cpu_contig(units, torch.int64)
        out = torch.empty((units.numel(), Dv), dtype=torch.float64)
        lse = torch.empty((units.numel(),), dtype=torch.float64)
        n_units = units.numel()
    else:
        out = torch.empty((B, qs, Hq, Dv), dtype=torch.float64)
        lse = torch.empty((B, qs, Hq), dtype=torch.float64)
        n_units = 0
    rc = _load().oracle_xqa_attention(
        _ptr(q_bits), _DTYPE_CODE[q.dtype], _ptr(k_bits), _ptr(v_bits), kv_code, layout_hnd,
        k_cache.shape[0], _ptr(page_table), page_table.shape[1], _ptr(seq_lens), B, Hq,
        int(num_kv_heads), D, Dv, int(page_size), qs, _ptr(sinks), float(q_scale),
        float(kv_scale), float(softmax_scale), int(sliding_win_size), float(rcp_out_scale),
        _ptr(mask), _ptr(units), n_units, _ptr(out), _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return (out, lse) if return_lse else out


def merge_attn_states(prefix_out, prefix_lse, suffix_out, suffix_lse, n_with_prefix=None):
    """merge_attn_states (Kimi-K3 MultiHeadLatentAttention page, prefill with
    chunked context) in float64: outputs [T, H, D] with log-sum-exps [T, H];
    rows t >= n_with_prefix take the suffix unchanged.  Returns (out, lse)."""
    po = _cpu_contig(prefix_out, torch.float64)
    so = _cpu_contig(suffix_out, torch.float64)
    pl = _cpu_contig(prefix_lse, torch.float64)
    sl = _cpu_contig(suffix_lse, torch.float64)
    T, H, D = so.shape
    if tuple(po.shape) != (T, H, D) or tuple(pl.shape) != (T, H) or tuple(sl.shape) != (T, H):
        raise ValueError("outputs must be [T, H, D] and lse [T, H]")
    n = T if n_with_prefix is None else int(n_with_prefix)
    out = torch.empty((T, H, D), dtype=torch.float64)
    lse = torch.empty((T, H), dtype=torch.float64)
    _load().oracle_merge_attn_states(_ptr(po), _ptr(pl), _ptr(so), _ptr(sl), T, H, D, n, _ptr(out),
                                     _ptr(lse))
    return out, lse


def encode_e4m3(x) -> torch.Tensor:
    """OCP E4M3FN codes (uint8) of float64 values: round to nearest even,
    saturating at +-448 (the oracle's rounding of an fp8 output)."""
    x = _cpu_contig(x, torch.float64).reshape(-1)
    enc = _load().oracle_encode_e4m3
    return torch.tensor([enc(float(v)) for v in x.tolist()], dtype=torch.uint8)


def unit_ids(batch_idx, q_idx, head_idx, q_seq_len, num_q_heads):
    """Flat row ids understood by ``xqa_attention(units=...)``."""
    b = torch.as_tensor(batch_idx, dtype=torch.int64)
    i = torch.as_tensor(q_idx, dtype=torch.int64)
    h = torch.as_tensor(head_idx, dtype=torch.int64)
    return (b * q_seq_len + i) * num_q_heads + h


def rope_pairs(x, cos, sin):
    """GPT-J (non-neox) rotary embedding of the last dim of x: element pairs
    (2i, 2i+1) rotate by angle i (Kimi-K3 MultiHeadLatentAttention page,
    `get_rope(..., is_neox_style=False)`): out_2i = x_2i cos_i - x_2i+1 sin_i,
    out_2i+1 = x_2i+1 cos_i + x_2i sin_i.  cos, sin broadcast over the pairs."""
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = torch.empty_like(x)
    out[..., 0::2] = x0 * cos - x1 * sin
    out[..., 1::2] = x1 * cos + x0 * sin
    return out


def mla_decode_prep(ql_nope, q_pe, kv_c, k_pe, positions, cos_sin_cache, slot_mapping, kv_cache):
    """The fused decode query-concat + latent cache insert (Kimi-K3
    MultiHeadLatentAttention page, `_decode_concat_cache`), in float64.

    ql_nope [T, H, Lr], q_pe [T, H, R], kv_c [T, Lr], k_pe [T, R]; positions
    [T] (None: no rotation); cos_sin_cache fp32 [max_pos, R] holding cos then
    sin of the R/2 angles; slot_mapping [T] (a negative slot is skipped);
    kv_cache [num_slots, Lr + R] (any float dtype, not modified).

    Returns (q [T, H, Lr + R] float64, cache float64 copy of kv_cache with the
    rows [kv_c | rope(k_pe)] written at their slots)."""
    ql = _cpu_contig(ql_nope).to(torch.float64)
    qp = _cpu_contig(q_pe).to(torch.float64)
    kc = _cpu_contig(kv_c).to(torch.float64)
    kp = _cpu_contig(k_pe).to(torch.float64)
    cache = _cpu_contig(kv_cache).to(torch.float64).clone()
    T, H, Lr = ql.shape
    R = qp.shape[-1]
    q = torch.empty((T, H, Lr + R), dtype=torch.float64)
    for t in range(T):
        if positions is None:
            c, s = torch.ones(R // 2, dtype=torch.float64), torch.zeros(R // 2, dtype=torch.float64)
        else:
            row = _cpu_contig(cos_sin_cache)[int(positions[t])].to(torch.float64)
            c, s = row[: R // 2], row[R // 2:]
        q[t, :, :Lr] = ql[t]
        q[t, :, Lr:] = rope_pairs(qp[t], c, s)
        slot = int(slot_mapping[t])
        if slot >= 0:
            cache[slot, :Lr] = kc[t]
            cache[slot, Lr:] = rope_pairs(kp[t], c, s)
    return q, cache


def mla_decode_prep_e4m3(ql_nope, q_pe, kv_c, k_pe, positions, cos_sin_cache, slot_mapping, kv_cache,
                         q_scale_inv, cache_scale_inv):
    """The fused decode prep for a plain per-tensor fp8 latent cache (Kimi-K3
    MultiHeadLatentAttention page, `_decode_concat_cache`: an fp8 cache takes
    an fp8 query, quantised with q_scale_inv, the inserted latent row with
    cache_scale_inv).  The float64 values of ``mla_decode_prep`` times the
    inverse scale, encoded as E4M3 (``encode_e4m3``: nearest even, saturated
    at +-448).  kv_cache: uint8 codes [num_slots, Lr + R] (not modified).

    Returns (q codes uint8 [T, H, Lr + R], cache codes uint8 with the rows
    written at their slots)."""
    codes = _cpu_contig(kv_cache).view(torch.uint8).reshape(-1, kv_cache.shape[-1])
    q64, cache64 = mla_decode_prep(ql_nope, q_pe, kv_c, k_pe, positions, cos_sin_cache, slot_mapping,
                                   torch.zeros(codes.shape, dtype=torch.float64))
    T, H, W = q64.shape
    q_codes = encode_e4m3(q64 * float(q_scale_inv)).reshape(T, H, W)
    out = codes.clone()
    for t in range(T):
        slot = int(slot_mapping[t])
        if slot >= 0:
            out[slot] = encode_e4m3(cache64[slot] * float(cache_scale_inv))
    return q_codes, out
