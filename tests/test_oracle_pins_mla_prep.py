"""Pins of the oracle's fused MLA decode prep (query concat with RoPE on
q_pe, latent cache insert at slot_mapping):

- The RoPE is checked against complex multiplication by e^(i * pos * theta)
  in torch.complex128, a different route than the oracle's pair arithmetic.
- The insert is checked by writing the rows by hand.
- Untouched slots keep their bits.
"""

import math

import torch

import oracle


def cos_sin_table(max_pos, R, base=10000.0):
    inv = base ** (-torch.arange(0, R, 2, dtype=torch.float64) / R)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cat([ang.cos(), ang.sin()], dim=1).to(torch.float32), ang


def test_rope_equals_complex_rotation():
    g = torch.Generator().manual_seed(1)
    R, P = 64, 100
    table, ang = cos_sin_table(P, R)
    x = torch.randn(7, 5, R, generator=g, dtype=torch.float64)
    pos = torch.randint(0, P, (7,), generator=g)
    for t in range(7):
        row = table[pos[t]].to(torch.float64)
        got = oracle.rope_pairs(x[t], row[: R // 2], row[R // 2:])
        z = torch.complex(x[t, :, 0::2], x[t, :, 1::2])
        phase = torch.complex(row[: R // 2], row[R // 2:])  # e^(i * angle) from the same fp32 table
        zr = z * phase
        want = torch.stack([zr.real, zr.imag], dim=-1).reshape(5, R)
        torch.testing.assert_close(got, want, rtol=1e-14, atol=1e-14)
        # and the table itself is e^(i * pos * theta) to fp32 precision
        torch.testing.assert_close(phase, torch.exp(1j * ang[pos[t]]), rtol=0, atol=1e-6)


def test_position_zero_is_identity_and_rotation_keeps_pair_norms():
    g = torch.Generator().manual_seed(2)
    R = 64
    table, _ = cos_sin_table(10, R)
    x = torch.randn(3, R, generator=g, dtype=torch.float64)
    row0 = table[0].to(torch.float64)
    torch.testing.assert_close(oracle.rope_pairs(x, row0[:32], row0[32:]), x)
    row = table[7].to(torch.float64)
    y = oracle.rope_pairs(x, row[:32], row[32:])
    torch.testing.assert_close(y[:, 0::2] ** 2 + y[:, 1::2] ** 2, x[:, 0::2] ** 2 + x[:, 1::2] ** 2,
                               rtol=1e-6, atol=1e-12)


def test_prep_concat_and_insert_by_hand():
    g = torch.Generator().manual_seed(3)
    T, H, Lr, R, slots = 5, 4, 16, 8, 40
    ql = torch.randn(T, H, Lr, generator=g).to(torch.bfloat16)
    qp = torch.randn(T, H, R, generator=g).to(torch.bfloat16)
    kc = torch.randn(T, Lr, generator=g).to(torch.bfloat16)
    kp = torch.randn(T, R, generator=g).to(torch.bfloat16)
    cache = torch.randn(slots, Lr + R, generator=g).to(torch.bfloat16)
    table, _ = cos_sin_table(64, R)
    pos = torch.tensor([0, 3, 9, 63, 5])
    slot = torch.tensor([7, -1, 0, 39, 12])
    q, c2 = oracle.mla_decode_prep(ql, qp, kc, kp, pos, table, slot, cache)
    torch.testing.assert_close(q[..., :Lr], ql.to(torch.float64))
    untouched = [s for s in range(slots) if s not in (7, 0, 39, 12)]
    assert torch.equal(c2[untouched], cache.to(torch.float64)[untouched])
    for t in range(T):
        row = table[pos[t]].to(torch.float64)
        c, s = row[: R // 2], row[R // 2:]
        x = qp[t].to(torch.float64)
        want = torch.empty_like(x)
        want[:, 0::2] = x[:, 0::2] * c - x[:, 1::2] * s
        want[:, 1::2] = x[:, 1::2] * c + x[:, 0::2] * s
        torch.testing.assert_close(q[t, :, Lr:], want)
        if slot[t] >= 0:
            torch.testing.assert_close(c2[slot[t], :Lr], kc[t].to(torch.float64))
            k = kp[t].to(torch.float64)
            kw = torch.empty_like(k)
            kw[0::2] = k[0::2] * c - k[1::2] * s
            kw[1::2] = k[1::2] * c + k[0::2] * s
            torch.testing.assert_close(c2[slot[t], Lr:], kw)


def _prep_inputs(seed, T=5, H=3, Lr=16, R=8, slots_n=40):
    g = torch.Generator().manual_seed(seed)
    ql = torch.randn(T, H, Lr, generator=g).to(torch.bfloat16)
    qp = torch.randn(T, H, R, generator=g).to(torch.bfloat16)
    kc = torch.randn(T, Lr, generator=g).to(torch.bfloat16)
    kp = torch.randn(T, R, generator=g).to(torch.bfloat16)
    table, _ = cos_sin_table(64, R)
    pos = torch.randint(0, 64, (T,), generator=g)
    slots = torch.randperm(slots_n, generator=g)[:T]
    slots[1] = -1
    return ql, qp, kc, kp, pos, table, slots


def test_e4m3_prep_is_torch_cast_of_the_scaled_values():
    """The fp8 prep's codes equal torch's float8_e4m3fn cast (nearest even) of
    the float64 prep values times the inverse scales (all inside +-448 here);
    untouched slots and the padding token's keep their codes."""
    ql, qp, kc, kp, pos, table, slots = _prep_inputs(3)
    g = torch.Generator().manual_seed(4)
    cache = torch.randint(0, 256, (40, 24), generator=g).to(torch.uint8)
    cache[cache == 0x7F] = 0  # no NaN codes in the untouched rows (compared with equal)
    q_inv, c_inv = 20.0, 12.5
    q_codes, c_codes = oracle.mla_decode_prep_e4m3(ql, qp, kc, kp, pos, table, slots, cache, q_inv, c_inv)
    q64, c64 = oracle.mla_decode_prep(ql, qp, kc, kp, pos, table, slots, torch.zeros(40, 24))
    assert (q64 * q_inv).abs().max() < 448 and (c64 * c_inv).abs().max() < 448
    want_q = (q64 * q_inv).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(q_codes, want_q)
    hit = slots[slots >= 0]
    want_c = cache.clone()
    want_c[hit] = (c64[hit] * c_inv).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(c_codes, want_c)


def test_e4m3_prep_saturates_beyond_448():
    """Out of range the prep saturates to +-448 (the reading for the fp8
    output and the fp8 prep; torch's cast gives NaN there instead)."""
    ql, qp, kc, kp, pos, table, slots = _prep_inputs(5)
    cache = torch.zeros(40, 24, dtype=torch.uint8)
    q_codes, c_codes = oracle.mla_decode_prep_e4m3(ql, qp, kc, kp, pos, table, slots, cache, 1e4, 1e4)
    q64, _ = oracle.mla_decode_prep(ql, qp, kc, kp, pos, table, slots, torch.zeros(40, 24))
    big = (q64 * 1e4).abs() > 464
    assert big.any()
    dec = q_codes.view(torch.float8_e4m3fn).to(torch.float64)
    assert torch.equal(dec[big].abs(), torch.full_like(dec[big], 448.0))
    assert torch.equal(torch.sign(dec[big]), torch.sign(q64[big]))
