"""GPU parity of the per-row log-sum-exp output (grouped-query and MLA
kernels) and of merge_attn_states, through the C ABI, against the float64
oracle on identical seeded inputs.

Tolerances follow from the arithmetic:

- lse: the kernels sum P after rounding it to bf16/f16. That rounding is
  relative 2^-9 per weight and unbiased, so the normaliser's relative error stays
  far below 1e-3. The lse bound is 3e-3 absolute.
- merge: fp32 weights, and one rounding of the result to 16 bits (2^-8 relative
  for bf16, 2^-11 for f16).
- chunked end to end: the decode tolerance, 1e-2 max-abs, plus the output's
  own rounding to bf16 where rcp_out_scale makes outputs large.
"""

import math

import pytest
import torch

import oracle
from paged_kv_decode_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LSE_TOL = 3e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_20_gb300 import build as B
    B.build()


def gpu_with_lse(case, **kw):
    from paged_kv_decode_20_gb300.runner import Decoder
    dec = Decoder(case.to("cuda"), lse=True, **kw)
    dec.lse.fill_(float("nan"))
    out = dec.run()
    torch.cuda.synchronize()
    assert dec.error_bits() == 0
    return out.cpu(), dec.lse.cpu()


def oracle_with_lse(c):
    return oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens,
                                return_lse=True, **c.kwargs())


def check_lse(got, ref):
    fin = torch.isfinite(ref)
    assert torch.equal(torch.isneginf(got), torch.isneginf(ref)), "-inf rows differ"
    err = (got.to(torch.float64)[fin] - ref[fin]).abs().max().item() if fin.any() else 0.0
    assert err <= LSE_TOL, f"lse max abs {err:.3e}"


LSE_CASES = [
    dict(batch=3, num_q_heads=16, num_kv_heads=2, head_dim=128, page_size=16,
         seq_lens=[1, 300, 2000]),
    dict(batch=2, num_q_heads=16, num_kv_heads=4, head_dim=64, page_size=32, seq_lens=[0, 500],
         q_seq_len=3, mask="causal", sinks=True, sliding_win_size=90),
    dict(batch=2, num_q_heads=8, num_kv_heads=1, head_dim=128, page_size=64, seq_lens=[700, 64],
         kv_dtype=torch.float8_e4m3fn, kv_scale=0.5, kv_divisor=0.5, q_scale=1.2),
    dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, seq_lens=[5, 77],
         q_mult=8.0, sinks=True, rcp_out_scale=2.0),
]


@pytest.mark.parametrize("sm_count", [1, 0, 10000])
@pytest.mark.parametrize("k", range(len(LSE_CASES)))
def test_gqa_lse_matches_oracle(k, sm_count):
    c = W.make_case(seed=60 + k, **LSE_CASES[k])
    out, lse = gpu_with_lse(c, sm_count=sm_count or None)
    ref_out, ref_lse = oracle_with_lse(c)
    tol = 3e-2 if c.k_cache.dtype == torch.float8_e4m3fn else 1e-2
    # the decode tolerance plus the output's own rounding to bf16 (half an ulp,
    # 2^-9 relative), which rcp_out_scale = 2 on a peaked row pushes past 1e-2
    err = (out.to(torch.float64) - ref_out).abs() - 2.0 ** -9 * ref_out.abs()
    assert err.max().item() <= tol
    check_lse(lse, ref_lse)


@pytest.mark.parametrize("sm_count", [2, 0])
def test_mla_lse_matches_oracle(sm_count):
    c = W.make_case(batch=2, num_q_heads=128, num_kv_heads=1, head_dim=576, v_head_dim=512,
                    mla=True, page_size=64, seq_lens=[3000, 77], kv_layout="NHD",
                    softmax_scale=(128 + 64) ** -0.5, sinks=True, seed=71)
    out, lse = gpu_with_lse(c, sm_count=sm_count or None)
    ref_out, ref_lse = oracle_with_lse(c)
    assert (out.to(torch.float64) - ref_out).abs().max().item() <= 1e-2
    check_lse(lse, ref_lse)


def _as_cuda16(x, dtype):
    return x.to(dtype).cuda()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_merge_matches_oracle_with_strided_prefix_and_partial_prefix(dtype):
    from paged_kv_decode_20_gb300 import xqa as X
    g = torch.Generator().manual_seed(7)
    T, H, D, wide = 37, 5, 512, 576
    pre_wide = torch.randn(T, H, wide, generator=g)
    suf = torch.randn(T, H, D, generator=g)
    pl = torch.randn(T, H, generator=g) * 3
    sl = torch.randn(T, H, generator=g) * 3
    pl[0, :2] = -math.inf
    pl[1, 0] = sl[1, 0] = -math.inf
    n_pre = 30
    pre_g = _as_cuda16(pre_wide, dtype)[..., :D]  # a slice: token stride 5 * 576
    suf_g = _as_cuda16(suf, dtype)
    out_g = torch.full((T, H, D), float("nan"), dtype=dtype, device="cuda")
    lse_g = torch.full((T, H), float("nan"), device="cuda")
    X.merge_attn_states(out_g, pre_g, pl.cuda(), suf_g, sl.cuda(), tokens_with_prefix=n_pre,
                        output_lse=lse_g)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.merge_attn_states(pre_g.cpu().to(torch.float64), pl.to(torch.float64),
                                            suf_g.cpu().to(torch.float64), sl.to(torch.float64),
                                            n_with_prefix=n_pre)
    got = out_g.cpu()
    # rows without a prefix, and rows whose prefix saw no key, are the suffix bit for bit
    assert torch.equal(got[n_pre:], suf_g.cpu()[n_pre:])
    assert torch.equal(got[0, :2], suf_g.cpu()[0, :2])
    assert torch.equal(got[1, 0], torch.zeros(D, dtype=dtype))
    rel = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11
    err = (got.to(torch.float64) - ref).abs()
    assert (err <= rel * ref.abs() + 1e-6).all(), f"max err {err.max().item():.3e}"
    gl = lse_g.cpu().to(torch.float64)
    assert torch.isneginf(gl[1, 0]) and torch.isneginf(ref_lse[1, 0])
    fin = torch.isfinite(ref_lse)
    assert (gl[fin] - ref_lse[fin]).abs().max().item() <= 1e-5 * (1 + ref_lse[fin].abs().max().item())


def _split(c, prefix_pages):
    ps = c.page_size
    pre = W.Case(**{**c.__dict__})
    pre.seq_lens = torch.clamp(c.seq_lens.to(torch.int64), max=prefix_pages * ps).to(torch.int32)
    pre.sinks = None  # the sink counts once, on the suffix side
    suf = W.Case(**{**c.__dict__})
    suf.page_table = torch.roll(c.page_table, -prefix_pages, dims=1).contiguous()
    suf.seq_lens = (c.seq_lens.to(torch.int64) - pre.seq_lens.to(torch.int64)).to(torch.int32)
    return pre, suf


@pytest.mark.parametrize("mla", [False, True])
def test_chunked_decode_then_merge_equals_full_attention(mla):
    """Attention over a prefix of the pages and over the rest, each with its
    log-sum-exp, merged on the GPU, equals attention over all pages."""
    from paged_kv_decode_20_gb300 import xqa as X
    if mla:
        c = W.make_case(batch=2, num_q_heads=128, num_kv_heads=1, head_dim=576, v_head_dim=512,
                        mla=True, page_size=64, seq_lens=[1500, 700], kv_layout="NHD",
                        softmax_scale=(128 + 64) ** -0.5, sinks=True, seed=81, pages_per_seq=32)
        prefix_pages = 8
    else:
        c = W.make_case(batch=3, num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=32,
                        seq_lens=[900, 300, 2000], sinks=True, seed=82, pages_per_seq=80)
        prefix_pages = 6
    pre, suf = _split(c, prefix_pages)
    po, plse = gpu_with_lse(pre)
    so, slse = gpu_with_lse(suf)
    B, qs, Hq, Dv = so.shape
    out = torch.empty((B * qs, Hq, Dv), dtype=so.dtype, device="cuda")
    X.merge_attn_states(out, po.cuda().reshape(B * qs, Hq, Dv), plse.cuda().reshape(B * qs, Hq),
                        so.cuda().reshape(B * qs, Hq, Dv), slse.cuda().reshape(B * qs, Hq))
    torch.cuda.synchronize()
    ref = oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens, **c.kwargs())
    err = (out.cpu().to(torch.float64).reshape(ref.shape) - ref).abs().max().item()
    assert err <= 1e-2, f"max abs {err:.3e}"


# ---------------------------------------------------------------- fp8 output
def _code_order(codes):
    """E4M3 codes as integers that increase with the value (sign-magnitude to
    a monotone scale), so neighbouring representable values differ by 1."""
    c = codes.to(torch.int32)
    mag = c & 0x7F
    return torch.where(c & 0x80 != 0, -mag, mag)


@pytest.mark.parametrize("split", [1, 0])
def test_fp8_output_codes_match_oracle_rounding(split):
    """Output dtype float8_e4m3fn with an fp8 cache (the API page's output
    "matches kv"), scaled by rcp_out_scale.  The kernel rounds its fp32 result,
    the oracle its float64 one, so a code may differ by one step where the
    value sits near a rounding boundary; most codes agree exactly."""
    c = W.make_case(batch=3, num_q_heads=16, num_kv_heads=2, head_dim=128, page_size=32,
                    seq_lens=[40, 700, 2500], kv_dtype=torch.float8_e4m3fn, kv_scale=0.5,
                    kv_divisor=0.5, rcp_out_scale=37.0, sinks=True, seed=91)
    from paged_kv_decode_20_gb300.runner import Decoder
    dec = Decoder(c.to("cuda"), sm_count=10000 if split else None, out_dtype=torch.float8_e4m3fn)
    out = dec.run()
    torch.cuda.synchronize()
    assert dec.error_bits() == 0
    got = out.cpu().view(torch.uint8).reshape(-1)
    ref = oracle.encode_e4m3(oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table,
                                                  c.seq_lens, **c.kwargs()))
    d = (_code_order(got) - _code_order(ref)).abs()
    assert d.max().item() <= 1, f"codes differ by {d.max().item()} steps"
    assert (d == 0).float().mean().item() >= 0.9
    # values past 448 saturate instead of becoming NaN
    c.rcp_out_scale = 1.0e4
    dec = Decoder(c.to("cuda"), out_dtype=torch.float8_e4m3fn)
    vals = dec.run().cpu().view(torch.uint8)
    torch.cuda.synchronize()
    assert not ((vals & 0x7F) == 0x7F).any(), "NaN codes in a saturated output"
