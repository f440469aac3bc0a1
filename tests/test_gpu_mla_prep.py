"""GPU parity of the fused MLA decode prep (query concat with RoPE, latent
cache insert at slot_mapping) through the C ABI against the float64 oracle.

Copied parts (ql_nope, kv_c) must match bit for bit. The rotated parts may
differ by one bf16 step, because the GPU rotates in fp32 and the oracle in
float64 before both round to bf16: at most 2^-8 relative plus 1e-6. Slots
that receive no row keep their bits.
"""

import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_20_gb300 import build as B
    B.build()


def table(max_pos, R, base=10000.0):
    inv = base ** (-torch.arange(0, R, 2, dtype=torch.float64) / R)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cat([ang.cos(), ang.sin()], dim=1).to(torch.float32)


def close_bf16(got, ref):
    got = got.to(torch.float64)
    return bool(((got - ref).abs() <= 2.0 ** -8 * ref.abs() + 1e-6).all())


@pytest.mark.parametrize("with_rope", [True, False])
def test_prep_matches_oracle(with_rope):
    from paged_kv_decode_20_gb300 import xqa as X
    g = torch.Generator().manual_seed(5)
    T, H, Lr, R, ps, pages, P = 9, 128, 512, 64, 64, 6, 5000
    q_full = torch.randn(T, H, Lr + 64, generator=g).to(torch.bfloat16)  # ql_nope is a slice of it
    q_pe = torch.randn(T, H, R, generator=g).to(torch.bfloat16)
    kv_c = torch.randn(T, Lr, generator=g).to(torch.bfloat16)
    k_pe = torch.randn(T, 1, R, generator=g).to(torch.bfloat16)
    cache = torch.randn(pages, ps, 1, Lr + R, generator=g).to(torch.bfloat16)
    pos = torch.randint(0, P, (T,), generator=g)
    pos[3] = P + 7  # out of the table: not rotated, flagged
    slots = torch.randperm(pages * ps, generator=g)[:T]
    slots[2] = -1   # a padding token
    cs = table(P, R)
    dev = "cuda"
    ql_g = q_full.to(dev)[..., :Lr]
    cache_g = cache.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    q_out = X.mla_decode_prep(ql_g, q_pe.to(dev), kv_c.to(dev), k_pe.to(dev),
                              pos.to(dev) if with_rope else None, cs.to(dev), slots.to(dev), cache_g,
                              error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == (1 if with_rope else 0)
    pos_ref = pos.clone()
    pos_ref[3] = 0  # row 0 of the table is the identity rotation
    q_ref, cache_ref = oracle.mla_decode_prep(q_full[..., :Lr], q_pe, kv_c, k_pe.reshape(T, R),
                                              pos_ref if with_rope else None, cs, slots,
                                              cache.reshape(pages * ps, Lr + R))
    qg = q_out.cpu()
    assert torch.equal(qg[..., :Lr], q_full[..., :Lr])
    assert close_bf16(qg[..., Lr:], q_ref[..., Lr:])
    cg = cache_g.cpu().reshape(pages * ps, Lr + R)
    hit = slots[slots >= 0]
    miss = torch.ones(pages * ps, dtype=torch.bool)
    miss[hit] = False
    assert torch.equal(cg[miss], cache.reshape(pages * ps, Lr + R)[miss])
    assert torch.equal(cg[hit, :Lr], cache_ref[hit, :Lr].to(torch.bfloat16))
    assert close_bf16(cg[hit, Lr:], cache_ref[hit, Lr:])


def codes_close(got, ref):
    """e4m3 codes: the GPU scales in fp32 and the oracle in float64 before both
    round, so a code may sit one step away at a rounding boundary: every
    decoded value within one e4m3 spacing of the oracle's, 99 % identical."""
    g = got.view(torch.float8_e4m3fn).to(torch.float64)
    r = ref.view(torch.float8_e4m3fn).to(torch.float64)
    spacing = torch.clamp(2.0 ** (torch.floor(torch.log2(r.abs().clamp_min(2.0 ** -6))) - 3), min=2.0 ** -9)
    near = bool(((g - r).abs() <= spacing).all())
    same = (got == ref).to(torch.float64).mean().item()
    return near and same >= 0.99


@pytest.mark.parametrize("with_rope", [True, False])
def test_prep_e4m3_matches_oracle_codes(with_rope):
    """The plain per-tensor fp8 cache: the query and the inserted latent rows
    come out as e4m3 of the values times q_scale_inv / cache_scale_inv."""
    from paged_kv_decode_20_gb300 import xqa as X
    g = torch.Generator().manual_seed(6)
    T, H, Lr, R, ps, pages, P = 9, 128, 512, 64, 64, 6, 5000
    ql = torch.randn(T, H, Lr, generator=g).to(torch.bfloat16)
    q_pe = torch.randn(T, H, R, generator=g).to(torch.bfloat16)
    kv_c = torch.randn(T, Lr, generator=g).to(torch.bfloat16)
    k_pe = torch.randn(T, R, generator=g).to(torch.bfloat16)
    cache = torch.randint(0, 126, (pages, ps, 1, Lr + R), generator=g).to(torch.uint8)
    pos = torch.randint(0, P, (T,), generator=g)
    slots = torch.randperm(pages * ps, generator=g)[:T]
    slots[4] = -1
    cs = table(P, R)
    q_inv, c_inv = 20.0, 16.0
    dev = "cuda"
    cache_g = cache.to(dev).view(torch.float8_e4m3fn)
    q_out = X.mla_decode_prep(ql.to(dev), q_pe.to(dev), kv_c.to(dev), k_pe.to(dev),
                              pos.to(dev) if with_rope else None, cs.to(dev), slots.to(dev), cache_g,
                              q_scale_inv=torch.tensor([q_inv], device=dev),
                              cache_scale_inv=torch.tensor([c_inv], device=dev))
    torch.cuda.synchronize()
    assert q_out.dtype == torch.float8_e4m3fn
    q_ref, c_ref = oracle.mla_decode_prep_e4m3(ql, q_pe, kv_c, k_pe, pos if with_rope else None, cs, slots,
                                               cache.reshape(pages * ps, Lr + R), q_inv, c_inv)
    assert codes_close(q_out.cpu().view(torch.uint8), q_ref)
    cg = cache_g.cpu().view(torch.uint8).reshape(pages * ps, Lr + R)
    hit = slots[slots >= 0]
    miss = torch.ones(pages * ps, dtype=torch.bool)
    miss[hit] = False
    assert torch.equal(cg[miss], cache.reshape(pages * ps, Lr + R)[miss])
    assert codes_close(cg[hit], c_ref[hit])


def test_prep_then_decode_e4m3_step():
    """One fp8 decode step: the prep quantises this step's query and inserts
    its latent row, then the MLA decode attends with the e4m3 query over the
    e4m3 cache (dequantised by q_scale = 1 / q_scale_inv, kv_scale = 1 /
    cache_scale_inv); checked against the oracle on the same codes."""
    from paged_kv_decode_20_gb300 import xqa as X
    from paged_kv_decode_20_gb300 import workloads as W
    B, H, Lr, R = 3, 128, 512, 64
    q_scale, kv_scale = 0.05, 0.05
    c = W.make_case(batch=B, num_q_heads=H, num_kv_heads=1, head_dim=Lr + R, v_head_dim=Lr, mla=True,
                    page_size=64, seq_lens=[300, 1000, 65], kv_layout="NHD", q_dtype=torch.float8_e4m3fn,
                    kv_dtype=torch.float8_e4m3fn, q_scale=q_scale, kv_scale=kv_scale, q_divisor=q_scale,
                    kv_divisor=kv_scale, softmax_scale=(128 + 64) ** -0.5, seed=31, poison=False)
    g = torch.Generator().manual_seed(32)
    ql = torch.randn(B, H, Lr, generator=g).to(torch.bfloat16)
    q_pe = torch.randn(B, H, R, generator=g).to(torch.bfloat16)
    kv_c = torch.randn(B, Lr, generator=g).to(torch.bfloat16)
    k_pe = torch.randn(B, R, generator=g).to(torch.bfloat16)
    cs = table(4096, R)
    # this step's token is the last of each sequence
    lens = c.seq_lens.to(torch.int64)
    pos = lens - 1
    slots = torch.stack([c.page_table[b, int(pos[b]) // 64].to(torch.int64) * 64 + int(pos[b]) % 64
                         for b in range(B)])
    dev = "cuda"
    cache_g = c.k_cache.to(dev)
    q8 = X.mla_decode_prep(ql.to(dev), q_pe.to(dev), kv_c.to(dev), k_pe.to(dev), pos.to(dev), cs.to(dev),
                           slots.to(dev), cache_g, q_scale_inv=torch.tensor([1 / q_scale], device=dev),
                           cache_scale_inv=torch.tensor([1 / kv_scale], device=dev))
    out = torch.empty((B, 1, H, Lr), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(1 << 26, dtype=torch.uint8, device=dev)
    sems = torch.zeros(2 * B + 2, dtype=torch.int32, device=dev)
    X.xqa_mla(q8.view(B, 1, H, Lr + R), cache_g, c.page_table.to(dev), c.seq_lens.to(dev), out, ws, sems,
              page_size=64, v_head_dim=Lr, softmax_scale=(128 + 64) ** -0.5, q_scale=q_scale, kv_scale=kv_scale)
    torch.cuda.synchronize()
    cache_cpu = cache_g.cpu()
    ref = oracle.xqa_attention(q8.cpu().view(B, 1, H, Lr + R), cache_cpu, cache_cpu, c.page_table, c.seq_lens,
                               **c.kwargs())
    assert (out.cpu().to(torch.float64) - ref).abs().max().item() <= 3e-2
