"""Pins for the float64 oracle, independent of the oracle itself.

Each test checks the oracle against something it does not share code with:
a library routine (torch's dtype decodes, CPU ``scaled_dot_product_attention``
on pages gathered by tensor indexing), a closed form, an invariant, or a hand
worked example.  Semantics: FlashInfer ``xqa`` API page (parameter list and
the shape-inference note); MLA variant: vLLM Kimi-K3 MultiHeadLatentAttention
page (``head_size``, ``scale``, ``process_weights_after_loading`` absorption,
``forward_mqa`` call).
"""

import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_decode_20_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# element decodes

def test_decode_e4m3_every_code_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64)
    got = torch.tensor([oracle.decode(torch.float8_e4m3fn, c) for c in range(256)],
                       dtype=torch.float64)
    assert torch.equal(torch.isnan(ref), torch.isnan(got))
    ok = ~torch.isnan(ref)
    assert torch.equal(ref[ok], got[ok])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_16bit_every_code_matches_torch(dtype):
    codes = torch.arange(65536, dtype=torch.int32)
    ref = codes.to(torch.int16).view(dtype).to(torch.float64)
    got = torch.tensor([oracle.decode(dtype, c) for c in range(65536)], dtype=torch.float64)
    assert torch.equal(torch.isnan(ref), torch.isnan(got))
    ok = ~torch.isnan(ref)
    assert torch.equal(ref[ok], got[ok])


def test_decode_e4m3_spec_table():
    for line in open(os.path.join(GOLDEN, "e4m3_codes.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, val = line.split()
        got = oracle.decode(torch.float8_e4m3fn, int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


# ---------------------------------------------------------------------------
# hand-worked example

def _two_key_case(sink=None, rcp=1.0):
    # D = 2: q = [1, 0]; page 0 slot 0: k=[0,0], v=[1,0]; slot 1: k=[1,0], v=[0,1]
    q = torch.tensor([[[[1.0, 0.0]]]], dtype=torch.bfloat16)
    k = torch.zeros((1, 16, 1, 2), dtype=torch.bfloat16)
    v = torch.zeros((1, 16, 1, 2), dtype=torch.bfloat16)
    k[0, 1, 0, 0] = 1.0
    v[0, 0, 0, 0] = 1.0
    v[0, 1, 0, 1] = 1.0
    sinks = None if sink is None else torch.tensor([[sink]], dtype=torch.float32)
    return oracle.xqa_attention(q, k, v, torch.zeros((1, 1), dtype=torch.int32),
                                torch.tensor([2], dtype=torch.int32), num_kv_heads=1,
                                page_size=16, softmax_scale=math.log(3.0), sinks=sinks,
                                rcp_out_scale=rcp)[0, 0, 0]


def test_two_key_worked_example():
    rows = {}
    for line in open(os.path.join(GOLDEN, "two_key_worked_example.txt")):
        line = line.split("#")[0].strip()
        if line:
            name, a, b = line.split()
            rows[name] = (float(a), float(b))
    got = {"no_sink": _two_key_case(), "sink_ln2": _two_key_case(sink=math.log(2.0)),
           "rcp_out_2": _two_key_case(rcp=2.0)}
    for name, (a, b) in rows.items():
        # the sink is fp32, so ln 2 carries ~1e-8 relative rounding
        assert got[name].tolist() == pytest.approx([a, b], rel=1e-7, abs=1e-12), name


# ---------------------------------------------------------------------------
# brute force: dense attention by a separate route (tensor indexing + SDPA)

def _bits_allowed(mask_words, b, i, j):
    words = mask_words[b, i].to(torch.int64) & 0xFFFF
    w32 = int(words[2 * (j // 32)]) | (int(words[2 * (j // 32) + 1]) << 16)
    return (w32 >> (j % 32)) & 1 == 1


def dense_reference(c: W.Case):
    """Float64 attention of every row via torch SDPA over pages gathered by
    indexing.  Sinks become one extra key per query row whose logit equals the
    sink and whose value is zero."""
    B, qs, Hq, D = c.q.shape
    Hkv, ps, Dv = c.num_kv_heads, c.page_size, c.dv
    G = Hq // Hkv
    scale = (c.softmax_scale if c.softmax_scale is not None else D ** -0.5) * c.q_scale * c.kv_scale
    out = torch.zeros((B, qs, Hq, Dv), dtype=torch.float64)
    for b in range(B):
        L = int(c.seq_lens[b])
        npg = -(-L // ps)
        idx = c.page_table[b, :npg].long()
        kc = c.k_cache[idx].to(torch.float64)
        vc = c.v_cache[idx].to(torch.float64)
        if c.kv_layout == "HND":
            kc, vc = kc.transpose(1, 2), vc.transpose(1, 2)
        K = kc.reshape(npg * ps, Hkv, D)[:L].repeat_interleave(G, dim=1).transpose(0, 1)
        V = vc.reshape(npg * ps, Hkv, D)[:L, :, :Dv].repeat_interleave(G, dim=1).transpose(0, 1)
        Q = c.q[b].to(torch.float64).transpose(0, 1)  # [Hq, qs, D]
        allowed = torch.ones((qs, L), dtype=torch.bool)
        for i in range(qs):
            p = L - qs + i
            for t in range(L):
                if c.sliding_win_size and not (t > p - c.sliding_win_size):
                    allowed[i, t] = False
                if c.mask is not None and t >= L - qs and not _bits_allowed(c.mask, b, i, t - (L - qs)):
                    allowed[i, t] = False
        allowed = allowed.unsqueeze(0).expand(Hq, qs, L)
        if c.sinks is not None:
            sig = c.sinks.to(torch.float64).reshape(Hq)  # h = kvh * G + g
            ks = Q * (sig[:, None, None] / (scale * (Q * Q).sum(-1, keepdim=True)))
            K = torch.cat([K, ks], dim=1)
            V = torch.cat([V, torch.zeros((Hq, qs, Dv), dtype=torch.float64)], dim=1)
            eye = torch.eye(qs, dtype=torch.bool).unsqueeze(0).expand(Hq, qs, qs)
            allowed = torch.cat([allowed, eye], dim=2)
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=allowed, scale=scale)
        out[b] = (o * (c.kv_scale * c.rcp_out_scale)).transpose(0, 1)
    return out


def _run(c: W.Case, **over):
    kw = c.kwargs()
    kw.update(over)
    return oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens, **kw)


SMALL = [
    dict(name="gqa_nhd_bf16", batch=3, num_q_heads=8, num_kv_heads=2, head_dim=16, page_size=16,
         seq_lens=[1, 17, 40], kv_layout="NHD"),
    dict(name="gqa_hnd_f16", batch=2, num_q_heads=6, num_kv_heads=3, head_dim=8, page_size=32,
         seq_lens=[33, 64], kv_layout="HND", q_dtype=torch.float16),
    dict(name="fp8_scales", batch=2, num_q_heads=4, num_kv_heads=1, head_dim=16, page_size=16,
         seq_lens=[20, 31], kv_layout="NHD", kv_dtype=torch.float8_e4m3fn, kv_scale=0.25,
         kv_divisor=0.25, q_scale=1.5, rcp_out_scale=0.5),
    dict(name="window_sinks_spec", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8,
         page_size=16, seq_lens=[30, 45], kv_layout="NHD", q_seq_len=3, sinks=True,
         sliding_win_size=7, mask="causal"),
    dict(name="spec_nomask_hnd", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8,
         page_size=16, seq_lens=[5, 19], kv_layout="HND", q_seq_len=4),
    dict(name="mla_like", batch=2, num_q_heads=4, num_kv_heads=1, head_dim=24, v_head_dim=16,
         mla=True, page_size=16, seq_lens=[18, 40], kv_layout="NHD", softmax_scale=0.2),
    dict(name="peaked", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=16, page_size=16,
         seq_lens=[9, 23], kv_layout="NHD", q_mult=8.0, sinks=True),
    # an e4m3 query against an e4m3 latent cache (the fp8 MLA decode), both scaled
    dict(name="mla_e4m3_query", batch=2, num_q_heads=4, num_kv_heads=1, head_dim=24, v_head_dim=16,
         mla=True, page_size=16, seq_lens=[18, 40], kv_layout="NHD", softmax_scale=0.2,
         q_dtype=torch.float8_e4m3fn, kv_dtype=torch.float8_e4m3fn, q_scale=0.25, kv_scale=0.125,
         q_divisor=0.25, kv_divisor=0.125, sinks=True),
]


@pytest.mark.parametrize("spec", SMALL, ids=[s["name"] for s in SMALL])
def test_oracle_matches_dense_sdpa(spec):
    c = W.make_case(seed=11, **spec)
    got = _run(c)
    ref = dense_reference(c)
    assert not torch.isnan(got).any()
    torch.testing.assert_close(got, ref, rtol=1e-10, atol=1e-12)


def test_row_subset_matches_full():
    c = W.make_case(seed=3, **SMALL[3])
    full = _run(c)
    B, qs, Hq, _ = c.q.shape
    units = torch.tensor([0, 5, 17, B * qs * Hq - 1])
    sub = _run(c, units=units)
    assert torch.equal(sub, full.reshape(-1, full.shape[-1])[units])


# ---------------------------------------------------------------------------
# invariants and special cases

def test_page_permutation_invariance():
    c = W.make_case(seed=5, **SMALL[0])
    base = _run(c)
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(c.k_cache.shape[0], generator=g)  # new slot of old page p: perm[p]
    k2 = torch.empty_like(c.k_cache)
    v2 = torch.empty_like(c.v_cache)
    k2[perm] = c.k_cache
    v2[perm] = c.v_cache
    t2 = perm[c.page_table.long()].to(torch.int32)
    got = oracle.xqa_attention(c.q, k2, v2, t2, c.seq_lens, **c.kwargs())
    assert torch.equal(got, base)


def test_nhd_hnd_same_logical_data():
    c = W.make_case(seed=6, **SMALL[0])
    got = _run(c)
    k_h = c.k_cache.transpose(1, 2).contiguous()
    v_h = c.v_cache.transpose(1, 2).contiguous()
    kw = c.kwargs()
    kw["kv_layout"] = "HND"
    got_h = oracle.xqa_attention(c.q, k_h, v_h, c.page_table, c.seq_lens, **kw)
    assert torch.equal(got, got_h)


def test_seq_len_one_returns_v0_and_sink_closed_form():
    c = W.make_case(name="one", batch=1, num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=16,
                    seq_lens=[1], seed=8, kv_scale=0.5, rcp_out_scale=3.0, sinks=True)
    v0 = c.v_cache[c.page_table[0, 0], 0, 0].to(torch.float64)
    nosink = _run(c, sinks=None)[0, 0]
    for h in range(2):
        torch.testing.assert_close(nosink[h], v0 * 0.5 * 3.0, rtol=1e-15, atol=0)
    k0 = c.k_cache[c.page_table[0, 0], 0, 0].to(torch.float64)
    with_sink = _run(c)[0, 0]
    for h in range(2):
        s0 = float((c.q[0, 0, h].to(torch.float64) * k0).sum()) * 8 ** -0.5 * 0.5
        sig = float(c.sinks[0, h])
        torch.testing.assert_close(with_sink[h], v0 * 1.5 / (1 + math.exp(sig - s0)),
                                   rtol=1e-12, atol=1e-15)


def test_identical_keys_return_mean_of_visible_values():
    c = W.make_case(name="same", batch=1, num_q_heads=2, num_kv_heads=1, head_dim=8,
                    page_size=16, seq_lens=[37], seed=9, sliding_win_size=10, poison=False)
    c.k_cache[:] = c.k_cache[c.page_table[0, 0], 3, 0]
    got = _run(c)[0, 0]
    rows = []
    for t in range(37 - 10, 37):
        rows.append(c.v_cache[c.page_table[0, t // 16], t % 16, 0].to(torch.float64))
    mean = torch.stack(rows).mean(0)
    for h in range(2):
        torch.testing.assert_close(got[h], mean, rtol=1e-12, atol=1e-14)


def test_window_large_is_no_window_and_window_one_is_own_value():
    c = W.make_case(seed=10, **SMALL[0])
    torch.testing.assert_close(_run(c, sliding_win_size=1000), _run(c), rtol=0, atol=0)
    got = _run(c, sliding_win_size=1)
    for b in range(c.batch):
        L = int(c.seq_lens[b])
        t = L - 1
        for h in range(c.num_q_heads):
            kvh = h // (c.num_q_heads // c.num_kv_heads)
            v = c.v_cache[c.page_table[b, t // 16], t % 16, kvh].to(torch.float64)
            torch.testing.assert_close(got[b, 0, h], v, rtol=1e-15, atol=0)


def test_causal_spec_equals_single_token_calls():
    n = 4
    c = W.make_case(name="spec", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8,
                    page_size=16, seq_lens=[21, 50], q_seq_len=n, mask="causal", seed=12,
                    sinks=True, sliding_win_size=9)
    got = _run(c)
    for i in range(n):
        lens = c.seq_lens - n + 1 + i
        single = oracle.xqa_attention(c.q[:, i:i + 1].contiguous(), c.k_cache, c.v_cache,
                                      c.page_table, lens, num_kv_heads=2, page_size=16,
                                      sinks=c.sinks, sliding_win_size=9)
        torch.testing.assert_close(got[:, i], single[:, 0], rtol=0, atol=0)


def test_full_mask_equals_no_mask():
    c = W.make_case(name="full", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8,
                    page_size=16, seq_lens=[21, 50], q_seq_len=3, mask="full", seed=13)
    torch.testing.assert_close(_run(c), _run(c, mask=None), rtol=0, atol=0)


def test_scales_compose_as_logit_product_and_value_factor():
    c = W.make_case(seed=14, **SMALL[0])
    base = _run(c, softmax_scale=0.3)
    torch.testing.assert_close(_run(c, q_scale=2.0, softmax_scale=0.15), base,
                               rtol=1e-13, atol=1e-15)
    # kv_scale multiplies the logits and the values
    torch.testing.assert_close(_run(c, kv_scale=4.0, softmax_scale=0.075), base * 4.0,
                               rtol=1e-13, atol=1e-15)
    torch.testing.assert_close(_run(c, softmax_scale=0.3, rcp_out_scale=0.25), base * 0.25,
                               rtol=1e-15, atol=0)


def test_gqa_equals_mha_with_repeated_kv_heads():
    c = W.make_case(seed=15, **SMALL[0])  # Hq 8, Hkv 2
    got = _run(c)
    G = 4
    k_rep = c.k_cache.repeat_interleave(G, dim=2).contiguous()
    v_rep = c.v_cache.repeat_interleave(G, dim=2).contiguous()
    mha = oracle.xqa_attention(c.q, k_rep, v_rep, c.page_table, c.seq_lens, num_kv_heads=8,
                               page_size=16)
    torch.testing.assert_close(got, mha, rtol=0, atol=0)


def test_empty_visible_set_gives_zero_and_sink_only_gives_zero():
    c = W.make_case(name="empty", batch=2, num_q_heads=2, num_kv_heads=1, head_dim=8,
                    page_size=16, seq_lens=[0, 5], seed=16, sinks=True)
    got = _run(c)
    assert torch.equal(got[0], torch.zeros_like(got[0]))
    assert torch.isfinite(got[1]).all() and got[1].abs().sum() > 0


def test_sink_scales_output_by_closed_form_factor():
    # out_sink = out_nosink * S / (S + e^sigma), S = sum_t e^{s_t}
    c = W.make_case(seed=17, **SMALL[0])
    c.sinks = torch.full((2, 4), 0.7, dtype=torch.float32)
    with_sink = _run(c)
    nosink = _run(c, sinks=None)
    scale = 16 ** -0.5
    for b in range(c.batch):
        L = int(c.seq_lens[b])
        for h in range(c.num_q_heads):
            kvh = h // 4
            s = []
            for t in range(L):
                k = c.k_cache[c.page_table[b, t // 16], t % 16, kvh].to(torch.float64)
                s.append(float((c.q[b, 0, h].to(torch.float64) * k).sum()) * scale)
            S = sum(math.exp(x) for x in s)
            sig = float(c.sinks[0, 0])  # the fp32 value of 0.7
            torch.testing.assert_close(with_sink[b, 0, h], nosink[b, 0, h] * S / (S + math.exp(sig)),
                                       rtol=1e-12, atol=1e-15)


def test_rejects_sequence_longer_than_table():
    c = W.make_case(seed=18, **SMALL[0])
    bad = c.seq_lens.clone()
    bad[0] = c.page_table.shape[1] * 16 + 1
    with pytest.raises(ValueError):
        oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, bad, **c.kwargs())


# ---------------------------------------------------------------------------
# MLA latent variant: the absorption identity

def test_mla_absorbed_latent_attention_equals_unabsorbed_mha():
    """Kimi-K3 MLA page, process_weights_after_loading / _attention: with
    W_UK_T (N, P, Lr) and W_UV (N, Lr, V), attention of ql = q_nope W_UK_T
    concatenated with q_pe against the latent rows [c | k_pe] (V = c, the
    first Lr dims), followed by W_UV, equals plain attention with
    k = [W_UK c | k_pe], v = W_UV^T c.  Small integers keep every bf16 input
    exact, so the comparison is in float64."""
    g = torch.Generator().manual_seed(21)
    N, P, Lr, R, Vd, T = 3, 4, 8, 2, 5, 37
    ri = lambda *s: torch.randint(-2, 3, s, generator=g).to(torch.float64)
    W_UK_T, W_UV = ri(N, P, Lr), ri(N, Lr, Vd)
    c_lat, k_pe = ri(T, Lr), ri(T, R)
    q_nope, q_pe = ri(N, P), ri(N, R)
    scale = 0.05
    # unabsorbed: per head n
    k_nope = torch.einsum("npl,tl->ntp", W_UK_T, c_lat)
    K = torch.cat([k_nope, k_pe.expand(N, T, R)], dim=-1)
    V = torch.einsum("nlv,tl->ntv", W_UV, c_lat)
    Qf = torch.cat([q_nope, q_pe], dim=-1).unsqueeze(1)
    ref = F.scaled_dot_product_attention(Qf, K, V, scale=scale)[:, 0]  # [N, Vd]
    # absorbed: one latent head of width Lr + R, paged
    ql = torch.einsum("np,npl->nl", q_nope, W_UK_T)
    mqa_q = torch.cat([ql, q_pe], dim=-1).to(torch.bfloat16)
    assert torch.equal(mqa_q.to(torch.float64), torch.cat([ql, q_pe], -1))
    ps = 16
    npg = -(-T // ps)
    rows = torch.zeros((npg * ps, Lr + R), dtype=torch.float64)
    rows[:T] = torch.cat([c_lat, k_pe], dim=-1)
    order = torch.tensor([2, 0, 1])  # logical page j lives in physical page order[j]
    cache = torch.zeros((npg, ps, 1, Lr + R), dtype=torch.bfloat16)
    cache[order] = rows.reshape(npg, ps, 1, Lr + R).to(torch.bfloat16)
    latent = oracle.xqa_attention(mqa_q.reshape(1, 1, N, Lr + R), cache, cache,
                                  order.reshape(1, npg).to(torch.int32),
                                  torch.tensor([T], dtype=torch.int32), num_kv_heads=1,
                                  page_size=ps, v_head_dim=Lr, softmax_scale=scale)[0, 0]
    got = torch.einsum("nl,nlv->nv", latent, W_UV)
    torch.testing.assert_close(got, ref, rtol=1e-12, atol=1e-12)
