"""ctypes binding of the C ABI in include/xqa.h (argument marshalling only).

Every step of the computation runs in the CUDA library ``libxqa_gb300.so``;
this module turns torch tensors into pointers, sizes and a stream handle, and
raises on a non-OK status.  There is no fallback: if the library is missing
or cannot load, the import of this module's entry points raises.

``xqa`` follows the argument list of FlashInfer's ``flashinfer.xqa.xqa``
(API page; beam_width fixed to 1) with one addition, ``softmax_scale``
(default 1/sqrt(head_dim)); ``xqa_mla`` is the MLA latent variant (Kimi-K3
MultiHeadLatentAttention page, ``forward_mqa``).
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libxqa_gb300.so")

XQA_OK, XQA_ERR_INVALID_ARG, XQA_ERR_UNSUPPORTED, XQA_ERR_WORKSPACE_TOO_SMALL, XQA_ERR_CUDA = range(5)
XQA_F16, XQA_BF16, XQA_E4M3 = 0, 1, 2
XQA_NHD, XQA_HND = 0, 1
_DTYPES = {torch.float16: XQA_F16, torch.bfloat16: XQA_BF16, torch.float8_e4m3fn: XQA_E4M3}


class XqaParams(ctypes.Structure):
    """Mirror of ``struct xqa_params`` (field order and types as in xqa.h)."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("q_dtype", ctypes.c_int),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("kv_dtype", ctypes.c_int),
        ("kv_layout", ctypes.c_int),
        ("num_pages", ctypes.c_int64),
        ("page_table", ctypes.c_void_p),
        ("pages_per_seq", ctypes.c_int32),
        ("seq_lens", ctypes.c_void_p),
        ("output", ctypes.c_void_p),
        ("out_dtype", ctypes.c_int),
        ("batch_size", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("q_seq_len", ctypes.c_int32),
        ("sinks", ctypes.c_void_p),
        ("q_scale", ctypes.c_float),
        ("kv_scale", ctypes.c_float),
        ("q_scale_dev", ctypes.c_void_p),
        ("kv_scale_dev", ctypes.c_void_p),
        ("softmax_scale", ctypes.c_float),
        ("sliding_win_size", ctypes.c_int32),
        ("rcp_out_scale", ctypes.c_float),
        ("mask", ctypes.c_void_p),
        ("sm_count", ctypes.c_int32),
        ("enable_pdl", ctypes.c_int32),
        ("error_word", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
    ]


class XqaMergeParams(ctypes.Structure):
    """Mirror of ``struct xqa_merge_params``."""

    _fields_ = [
        ("output", ctypes.c_void_p),
        ("prefix_output", ctypes.c_void_p),
        ("suffix_output", ctypes.c_void_p),
        ("dtype", ctypes.c_int),
        ("output_lse", ctypes.c_void_p),
        ("prefix_lse", ctypes.c_void_p),
        ("suffix_lse", ctypes.c_void_p),
        ("num_tokens", ctypes.c_int64),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("tokens_with_prefix", ctypes.c_int64),
        ("out_stride_token", ctypes.c_int64),
        ("out_stride_head", ctypes.c_int64),
        ("prefix_stride_token", ctypes.c_int64),
        ("prefix_stride_head", ctypes.c_int64),
        ("suffix_stride_token", ctypes.c_int64),
        ("suffix_stride_head", ctypes.c_int64),
        ("lse_stride_token", ctypes.c_int64),
        ("lse_stride_head", ctypes.c_int64),
    ]


class XqaMlaPrepParams(ctypes.Structure):
    """Mirror of ``struct xqa_mla_prep_params``."""

    _fields_ = [
        ("ql_nope", ctypes.c_void_p),
        ("ql_stride_token", ctypes.c_int64),
        ("ql_stride_head", ctypes.c_int64),
        ("q_pe", ctypes.c_void_p),
        ("qpe_stride_token", ctypes.c_int64),
        ("qpe_stride_head", ctypes.c_int64),
        ("kv_c", ctypes.c_void_p),
        ("kvc_stride_token", ctypes.c_int64),
        ("k_pe", ctypes.c_void_p),
        ("kpe_stride_token", ctypes.c_int64),
        ("positions", ctypes.c_void_p),
        ("cos_sin_cache", ctypes.c_void_p),
        ("max_position", ctypes.c_int64),
        ("slot_mapping", ctypes.c_void_p),
        ("kv_cache", ctypes.c_void_p),
        ("num_slots", ctypes.c_int64),
        ("q_out", ctypes.c_void_p),
        ("num_tokens", ctypes.c_int64),
        ("num_heads", ctypes.c_int32),
        ("kv_lora_rank", ctypes.c_int32),
        ("rope_dim", ctypes.c_int32),
        ("error_word", ctypes.c_void_p),
        ("fp8", ctypes.c_int32),
        ("q_scale_inv", ctypes.c_void_p),
        ("cache_scale_inv", ctypes.c_void_p),
    ]


EXPORTS = ["xqa_workspace_size", "xqa_semaphore_count", "xqa_decode", "xqa_mla_workspace_size",
           "xqa_mla_semaphore_count", "xqa_mla_decode", "xqa_decode_noalloc", "xqa_merge_attn_states", "xqa_mla_decode_prep",
           "xqa_read_bandwidth_probe", "xqa_status_string", "xqa_last_error"]

_lock = threading.Lock()
_lib = None


class XqaError(RuntimeError):
    def __init__(self, status, detail):
        self.status = status
        super().__init__(f"{status_name(status)}: {detail}")


def load(path: str = LIB_PATH):
    """Load libxqa_gb300.so (raises OSError if it is missing or broken)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise OSError(f"{path} is missing: build it with paged_kv_decode_20_gb300.build")
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER(XqaParams)
            lib.xqa_workspace_size.argtypes = [P, ctypes.c_int]
            lib.xqa_workspace_size.restype = ctypes.c_size_t
            lib.xqa_semaphore_count.argtypes = [P]
            lib.xqa_semaphore_count.restype = ctypes.c_size_t
            lib.xqa_decode.argtypes = [P, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                       ctypes.c_void_p]
            lib.xqa_decode.restype = ctypes.c_int
            lib.xqa_mla_workspace_size.argtypes = [P, ctypes.c_int, ctypes.c_int]
            lib.xqa_mla_workspace_size.restype = ctypes.c_size_t
            lib.xqa_mla_semaphore_count.argtypes = [P, ctypes.c_int]
            lib.xqa_mla_semaphore_count.restype = ctypes.c_size_t
            lib.xqa_mla_decode.argtypes = [P, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.c_void_p, ctypes.c_void_p]
            lib.xqa_mla_decode.restype = ctypes.c_int
            lib.xqa_merge_attn_states.argtypes = [ctypes.POINTER(XqaMergeParams), ctypes.c_void_p]
            lib.xqa_merge_attn_states.restype = ctypes.c_int
            lib.xqa_mla_decode_prep.argtypes = [ctypes.POINTER(XqaMlaPrepParams), ctypes.c_void_p]
            lib.xqa_mla_decode_prep.restype = ctypes.c_int
            lib.xqa_read_bandwidth_probe.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int,
                                                     ctypes.c_void_p]
            lib.xqa_read_bandwidth_probe.restype = ctypes.c_int
            lib.xqa_status_string.argtypes = [ctypes.c_int]
            lib.xqa_status_string.restype = ctypes.c_char_p
            lib.xqa_last_error.argtypes = []
            lib.xqa_last_error.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_name(status: int) -> str:
    return load().xqa_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("every tensor argument must live on a CUDA device")
    return t.data_ptr()


def _q_view(q, q_seq_len):
    """q as [B, q_seq_len, Hq, D]: accepts [B, Hq, D], [B, q_seq_len, Hq, D]
    or [B, 1, q_seq_len, Hq, D] (beam width 1)."""
    if q.dim() == 3:
        q = q.unsqueeze(1)
    elif q.dim() == 5:
        if q.shape[1] != 1:
            raise ValueError("only beam_width 1 is supported")
        q = q[:, 0]
    if q.dim() != 4:
        raise ValueError(f"q must be 3-, 4- or 5-dimensional, got {tuple(q.shape)}")
    if q.shape[1] != q_seq_len:
        raise ValueError(f"q carries {q.shape[1]} tokens per sequence but q_seq_len={q_seq_len}")
    return q


def make_params(q, k_cache, v_cache, page_table, seq_lens, output, *, num_kv_heads, page_size,
                sinks=None, q_scale=1.0, kv_scale=1.0, sliding_win_size=0, kv_layout="NHD",
                sm_count=None, enable_pdl=None, rcp_out_scale=1.0, q_seq_len=1, mask=None,
                softmax_scale=None, error_word=None, lse=None):
    """Build the C parameter struct; shapes are inferred as the API page
    states (B from q, Hq from q.shape[-2], D from q.shape[-1], dtypes from q
    and k_cache, max_seq_len = page_table.shape[-1] * page_size)."""
    q4 = _q_view(q, q_seq_len)
    for name, t in (("q", q4), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("page_table", page_table), ("seq_lens", seq_lens), ("output", output)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q4.dtype not in _DTYPES or k_cache.dtype not in _DTYPES:
        raise ValueError("unsupported dtype")
    if page_table.dtype != torch.int32:
        raise ValueError("page_table must be int32")
    if seq_lens.dtype not in (torch.int32, torch.uint32):
        raise ValueError("seq_lens must be uint32 (int32 storage accepted)")
    if seq_lens.numel() != q4.shape[0]:
        raise ValueError("seq_lens must hold one length per sequence (beam width 1)")
    if sinks is not None and (sinks.dtype != torch.float32 or not sinks.is_contiguous()):
        raise ValueError("sinks must be contiguous float32 [num_kv_heads, head_group_ratio]")
    if sinks is not None and sinks.numel() != q4.shape[2]:
        raise ValueError("sinks must hold num_kv_heads * head_group_ratio values")
    if mask is not None:
        words = ((q_seq_len + 31) // 32) * 2
        if tuple(mask.shape) != (q4.shape[0], q_seq_len, words) or mask.element_size() != 2:
            raise ValueError(f"mask must be 16-bit [{q4.shape[0]}, {q_seq_len}, {words}]")
        if not mask.is_contiguous():
            raise ValueError("mask must be contiguous")
    if lse is not None:
        if lse.dtype != torch.float32 or tuple(lse.shape) != tuple(q4.shape[:3]) or not lse.is_contiguous():
            raise ValueError(f"lse must be contiguous float32 {tuple(q4.shape[:3])}")
    p = XqaParams()
    keep = [q4, k_cache, v_cache, page_table, seq_lens, output, sinks, mask, error_word, lse]
    p.q = _ptr(q4)
    p.q_dtype = _DTYPES[q4.dtype]
    p.k_cache = _ptr(k_cache)
    p.v_cache = _ptr(v_cache)
    p.kv_dtype = _DTYPES[k_cache.dtype]
    if v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache must share one dtype")
    layout = kv_layout.upper()
    if layout not in ("NHD", "HND"):
        raise ValueError("kv_layout must be NHD or HND")
    p.kv_layout = XQA_NHD if layout == "NHD" else XQA_HND
    p.num_pages = k_cache.shape[0]
    p.page_table = _ptr(page_table)
    p.pages_per_seq = page_table.shape[-1]
    p.seq_lens = _ptr(seq_lens)
    p.output = _ptr(output)
    p.out_dtype = _DTYPES.get(output.dtype, -1)
    p.batch_size = q4.shape[0]
    p.num_q_heads = q4.shape[-2]
    p.num_kv_heads = int(num_kv_heads)
    p.head_dim = q4.shape[-1]
    p.page_size = int(page_size)
    p.q_seq_len = int(q_seq_len)
    p.sinks = _ptr(sinks)
    if isinstance(q_scale, torch.Tensor):
        qs_t = q_scale.to(torch.float32).contiguous()
        keep.append(qs_t)
        p.q_scale, p.q_scale_dev = 1.0, _ptr(qs_t)
    else:
        p.q_scale = float(q_scale)
    if isinstance(kv_scale, torch.Tensor):
        kvs_t = kv_scale.to(torch.float32).contiguous()
        keep.append(kvs_t)
        p.kv_scale, p.kv_scale_dev = 1.0, _ptr(kvs_t)
    else:
        p.kv_scale = float(kv_scale)
    p.softmax_scale = 0.0 if softmax_scale is None else float(softmax_scale)
    p.sliding_win_size = int(sliding_win_size)
    p.rcp_out_scale = float(rcp_out_scale)
    p.mask = _ptr(mask)
    p.sm_count = 0 if sm_count is None else int(sm_count)
    p.enable_pdl = 1 if enable_pdl is None else int(bool(enable_pdl))
    p.error_word = _ptr(error_word)
    p.lse = _ptr(lse)
    # the struct holds raw pointers: keep every tensor it names alive with it
    p._keep = keep
    return p


def _check(status):
    if status != XQA_OK:
        raise XqaError(status, load().xqa_last_error().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def xqa_workspace_size(params: XqaParams, sm_count: int = 0) -> int:
    n = load().xqa_workspace_size(ctypes.byref(params), int(sm_count))
    if n == ctypes.c_size_t(-1).value:
        raise XqaError(XQA_ERR_INVALID_ARG, load().xqa_last_error().decode())
    return n


def xqa_semaphore_count(params: XqaParams) -> int:
    n = load().xqa_semaphore_count(ctypes.byref(params))
    if n == ctypes.c_size_t(-1).value:
        raise XqaError(XQA_ERR_INVALID_ARG, load().xqa_last_error().decode())
    return n


def xqa_mla_workspace_size(params: XqaParams, v_head_dim: int, sm_count: int = 0) -> int:
    n = load().xqa_mla_workspace_size(ctypes.byref(params), int(v_head_dim), int(sm_count))
    if n == ctypes.c_size_t(-1).value:
        raise XqaError(XQA_ERR_UNSUPPORTED, load().xqa_last_error().decode())
    return n


def xqa_mla_semaphore_count(params: XqaParams, v_head_dim: int) -> int:
    n = load().xqa_mla_semaphore_count(ctypes.byref(params), int(v_head_dim))
    if n == ctypes.c_size_t(-1).value:
        raise XqaError(XQA_ERR_UNSUPPORTED, load().xqa_last_error().decode())
    return n


def _check_semaphores(semaphores, count):
    """The C ABI takes the semaphores as a bare pointer: a tensor shorter than
    the count the sizing query returns is refused here, before the launch.
    (Parameters the sizing query rejects are left to the call's own status.)"""
    try:
        needed = count()
    except XqaError:
        return
    if semaphores is not None and needed > 0 and semaphores.numel() * semaphores.element_size() < 4 * needed:
        raise XqaError(XQA_ERR_WORKSPACE_TOO_SMALL,
                       f"semaphores hold {semaphores.numel() * semaphores.element_size() // 4} uint32, "
                       f"{needed} needed")


def xqa_decode(params: XqaParams, workspace, semaphores, stream=None, check_semaphores=True):
    """Launch through the C ABI.  workspace: uint8 CUDA tensor or None.
    check_semaphores=False skips the size check (a caller that sized the
    buffer with xqa_semaphore_count for these parameters)."""
    if check_semaphores:
        _check_semaphores(semaphores, lambda: xqa_semaphore_count(params))
    ws_ptr = None if workspace is None else _ptr(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().xqa_decode(ctypes.byref(params), ws_ptr, ws_bytes, _ptr(semaphores),
                             _stream(stream)))


def xqa_mla_decode(params: XqaParams, v_head_dim, workspace, semaphores, stream=None, check_semaphores=True):
    if check_semaphores:
        _check_semaphores(semaphores, lambda: xqa_mla_semaphore_count(params, v_head_dim))
    ws_ptr = None if workspace is None else _ptr(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().xqa_mla_decode(ctypes.byref(params), int(v_head_dim), ws_ptr, ws_bytes,
                                 _ptr(semaphores), _stream(stream)))


def xqa(q, k_cache, v_cache, page_table, seq_lens, output, workspace_buffer, semaphores,
        num_kv_heads, page_size, sinks=None, q_scale=1.0, kv_scale=1.0, sliding_win_size=0,
        kv_layout="NHD", sm_count=None, enable_pdl=None, rcp_out_scale=1.0, q_seq_len=1,
        mask=None, softmax_scale=None, error_word=None, lse=None, stream=None):
    """Paged decode attention with the XQA API page's argument list; writes
    ``output`` in place (and, when given, each row's log-sum-exp into ``lse``,
    float32 [B, q_seq_len, Hq]).  workspace_buffer: uint8, at least
    ``xqa_workspace_size`` bytes; semaphores: uint32/int32, zeroed, at least
    ``xqa_semaphore_count`` entries (left zeroed)."""
    p = make_params(q, k_cache, v_cache, page_table, seq_lens, output, num_kv_heads=num_kv_heads,
                    page_size=page_size, sinks=sinks, q_scale=q_scale, kv_scale=kv_scale,
                    sliding_win_size=sliding_win_size, kv_layout=kv_layout, sm_count=sm_count,
                    enable_pdl=enable_pdl, rcp_out_scale=rcp_out_scale, q_seq_len=q_seq_len,
                    mask=mask, softmax_scale=softmax_scale, error_word=error_word, lse=lse)
    xqa_decode(p, workspace_buffer, semaphores, stream)


def xqa_mla(q, kv_cache, page_table, seq_lens, output, workspace_buffer, semaphores, page_size,
            v_head_dim, softmax_scale, kv_layout="NHD", q_scale=1.0, kv_scale=1.0,
            sm_count=None, rcp_out_scale=1.0, error_word=None, lse=None, stream=None):
    """MLA latent decode: q [B, Hq, Lr + rope] (absorbed), one latent kv head
    ``kv_cache`` [num_pages, page_size, 1, Lr + rope]; output [B, Hq, Lr]."""
    q_seq_len = 1 if q.dim() == 3 else q.shape[1]
    p = make_params(q, kv_cache, kv_cache, page_table, seq_lens, output, num_kv_heads=1,
                    page_size=page_size, q_scale=q_scale, kv_scale=kv_scale, kv_layout=kv_layout,
                    sm_count=sm_count, rcp_out_scale=rcp_out_scale, q_seq_len=q_seq_len,
                    softmax_scale=softmax_scale, error_word=error_word, lse=lse)
    xqa_mla_decode(p, v_head_dim, workspace_buffer, semaphores, stream)


def read_bandwidth_probe(buf, sink, stream=None):
    """One launch of the library's read-only streaming kernel over the bytes
    of `buf` (a contiguous CUDA tensor, a multiple of 16 bytes); `sink` is an
    int32 CUDA tensor of at least one word per CTA (4 per SM).  A
    measurement aid beside the decode path, not part of it."""
    if not (buf.is_cuda and sink.is_cuda and buf.is_contiguous() and sink.dtype == torch.int32):
        raise ValueError("buf: contiguous CUDA tensor; sink: int32 CUDA tensor")
    _check(load().xqa_read_bandwidth_probe(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                                           sink.numel(), _stream(stream)))


def merge_attn_states(output, prefix_output, prefix_lse, suffix_output, suffix_lse,
                      tokens_with_prefix=None, output_lse=None, stream=None):
    """merge_attn_states (Kimi-K3 MultiHeadLatentAttention page, prefill with
    chunked context) through the C ABI.  Outputs are [T, H, D] fp16/bf16 views
    with a contiguous last dim (a prefix wider than D may be a slice); lse
    tensors are float32 [T, H] sharing one stride pattern.  Rows of tokens
    t >= tokens_with_prefix (default T) take the suffix unchanged."""
    T, H, D = suffix_output.shape
    for name, t in (("output", output), ("prefix_output", prefix_output)):
        if tuple(t.shape) != (T, H, D):
            raise ValueError(f"{name} must be [{T}, {H}, {D}]")
    for t in (output, prefix_output, suffix_output):
        if t.stride(-1) != 1 or t.dtype != suffix_output.dtype:
            raise ValueError("outputs must share one dtype and have a contiguous last dim")
    lses = [x for x in (prefix_lse, suffix_lse, output_lse) if x is not None]
    for x in lses:
        if x.dtype != torch.float32 or tuple(x.shape) != (T, H) or x.stride() != suffix_lse.stride():
            raise ValueError(f"lse tensors must be float32 [{T}, {H}] with identical strides")
    if suffix_output.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("merge works on fp16 or bf16 outputs")
    p = XqaMergeParams()
    p.output, p.prefix_output, p.suffix_output = _ptr(output), _ptr(prefix_output), _ptr(suffix_output)
    p.dtype = _DTYPES[suffix_output.dtype]
    p.output_lse, p.prefix_lse, p.suffix_lse = _ptr(output_lse), _ptr(prefix_lse), _ptr(suffix_lse)
    p.num_tokens, p.num_heads, p.head_dim = T, H, D
    p.tokens_with_prefix = T if tokens_with_prefix is None else int(tokens_with_prefix)
    p.out_stride_token, p.out_stride_head = output.stride(0), output.stride(1)
    p.prefix_stride_token, p.prefix_stride_head = prefix_output.stride(0), prefix_output.stride(1)
    p.suffix_stride_token, p.suffix_stride_head = suffix_output.stride(0), suffix_output.stride(1)
    p.lse_stride_token, p.lse_stride_head = suffix_lse.stride(0), suffix_lse.stride(1)
    _check(load().xqa_merge_attn_states(ctypes.byref(p), _stream(stream)))


def mla_decode_prep(ql_nope, q_pe, kv_c, k_pe, positions, cos_sin_cache, slot_mapping, kv_cache,
                    q_out=None, error_word=None, q_scale_inv=None, cache_scale_inv=None, stream=None):
    """Fused MLA decode prep through the C ABI (Kimi-K3 MultiHeadLatentAttention
    page, `_decode_concat_cache`): returns q_out [T, H, Lr + R] = [ql_nope |
    rope(q_pe)] and writes [kv_c | rope(k_pe)] into kv_cache at slot_mapping.
    bf16 inputs with a contiguous last dim; kv_cache [num_pages, page_size,
    (1,) Lr + R] contiguous; positions and slot_mapping int64 [T].  An e4m3
    kv_cache (the page's plain fp8 cache) takes the fp8 path: q_out and the
    inserted rows are e4m3 of the values times q_scale_inv / cache_scale_inv
    (fp32 device scalars, required then)."""
    T, H, Lr = ql_nope.shape
    R = q_pe.shape[-1]
    kc = kv_c.reshape(T, Lr)
    kp = k_pe.reshape(T, R)
    for name, t in (("ql_nope", ql_nope), ("q_pe", q_pe), ("kv_c", kc), ("k_pe", kp)):
        if t.dtype != torch.bfloat16 or t.stride(-1) != 1:
            raise ValueError(f"{name} must be bf16 with a contiguous last dim")
    fp8 = kv_cache.dtype == torch.float8_e4m3fn
    if kv_cache.dtype not in (torch.bfloat16, torch.float8_e4m3fn) or not kv_cache.is_contiguous() \
            or kv_cache.shape[-1] != Lr + R:
        raise ValueError(f"kv_cache must be contiguous bf16 or e4m3 with rows of {Lr + R}")
    scales = []
    if fp8:
        for name, t in (("q_scale_inv", q_scale_inv), ("cache_scale_inv", cache_scale_inv)):
            if t is None or t.dtype != torch.float32 or t.numel() != 1:
                raise ValueError(f"the e4m3 prep needs {name} as a one-element float32 device tensor")
            scales.append(t.contiguous())
    for name, t in (("slot_mapping", slot_mapping), ("positions", positions)):
        if t is not None and (t.dtype != torch.int64 or not t.is_contiguous() or t.numel() != T):
            raise ValueError(f"{name} must be contiguous int64 [{T}]")
    if cos_sin_cache is not None and (cos_sin_cache.dtype != torch.float32 or not cos_sin_cache.is_contiguous()
                                      or cos_sin_cache.shape[-1] != R):
        raise ValueError(f"cos_sin_cache must be contiguous fp32 [max_position, {R}]")
    if q_out is None:
        q_out = torch.empty((T, H, Lr + R), dtype=kv_cache.dtype, device=ql_nope.device)
    if q_out.dtype != kv_cache.dtype:
        raise ValueError("q_out takes the cache's dtype")
    p = XqaMlaPrepParams()
    p.ql_nope, p.ql_stride_token, p.ql_stride_head = _ptr(ql_nope), ql_nope.stride(0), ql_nope.stride(1)
    p.q_pe, p.qpe_stride_token, p.qpe_stride_head = _ptr(q_pe), q_pe.stride(0), q_pe.stride(1)
    p.kv_c, p.kvc_stride_token = _ptr(kc), kc.stride(0)
    p.k_pe, p.kpe_stride_token = _ptr(kp), kp.stride(0)
    p.positions = _ptr(positions)
    p.cos_sin_cache = _ptr(cos_sin_cache)
    p.max_position = 0 if cos_sin_cache is None else cos_sin_cache.shape[0]
    p.slot_mapping = _ptr(slot_mapping)
    p.kv_cache = _ptr(kv_cache)
    p.num_slots = kv_cache.numel() // (Lr + R)
    p.q_out = _ptr(q_out)
    p.num_tokens, p.num_heads, p.kv_lora_rank, p.rope_dim = T, H, Lr, R
    p.error_word = _ptr(error_word)
    p.fp8 = 1 if fp8 else 0
    if fp8:
        p.q_scale_inv, p.cache_scale_inv = _ptr(scales[0]), _ptr(scales[1])
    _check(load().xqa_mla_decode_prep(ctypes.byref(p), _stream(stream)))
    return q_out
