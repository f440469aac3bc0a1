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
