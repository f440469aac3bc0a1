"""Pins of the oracle's log-sum-exp output, its merge_attn_states and its fp8
(E4M3FN) output rounding against things other than the oracle itself:

- The log-sum-exp equals torch.logsumexp over logits gathered by dense
  indexing. The sink is one more logit.
- Merging the results over a prefix and a suffix of the keys equals attention
  over all keys, computed by torch's scaled_dot_product_attention.
- The E4M3 encoding equals torch's round-to-nearest-even cast wherever that
  cast is finite, and saturates at +-448 beyond.
"""

import math

import pytest
import torch

import oracle
from paged_kv_decode_20_gb300 import workloads as W

from test_oracle_pins import SMALL, _bits_allowed, dense_reference


def dense_lse(c: W.Case):
    """Natural-log log-sum-exp of every row's visible logits (plus the sink),
    from K gathered by page indexing and an einsum."""
    B, qs, Hq, D = c.q.shape
    Hkv, ps = c.num_kv_heads, c.page_size
    G = Hq // Hkv
    scale = (c.softmax_scale if c.softmax_scale is not None else D ** -0.5) * c.q_scale * c.kv_scale
    out = torch.empty((B, qs, Hq), dtype=torch.float64)
    for b in range(B):
        L = int(c.seq_lens[b])
        npg = -(-L // ps)
        kc = c.k_cache[c.page_table[b, :npg].long()].to(torch.float64)
        if c.kv_layout == "HND":
            kc = kc.transpose(1, 2)
        K = kc.reshape(npg * ps, Hkv, D)[:L]
        for i in range(qs):
            p = L - qs + i
            for h in range(Hq):
                s = torch.einsum("d,td->t", c.q[b, i, h].to(torch.float64), K[:, h // G]) * scale
                keep = torch.ones(L, dtype=torch.bool)
                for t in range(L):
                    if c.sliding_win_size and not (t > p - c.sliding_win_size):
                        keep[t] = False
                    if c.mask is not None and t >= L - qs and not _bits_allowed(c.mask, b, i, t - (L - qs)):
                        keep[t] = False
                vals = s[keep]
                if c.sinks is not None:
                    vals = torch.cat([vals, c.sinks.reshape(-1)[h:h + 1].to(torch.float64)])
                out[b, i, h] = torch.logsumexp(vals, 0) if vals.numel() else -math.inf
    return out


@pytest.mark.parametrize("spec", SMALL, ids=[s["name"] for s in SMALL])
def test_lse_matches_dense_logsumexp(spec):
    c = W.make_case(seed=21, **spec)
    kw = c.kwargs()
    _, lse = oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens,
                                  return_lse=True, **kw)
    torch.testing.assert_close(lse, dense_lse(c), rtol=1e-12, atol=1e-12)


def test_lse_of_empty_row_is_minus_inf_and_sink_only_row_is_the_sink():
    c = W.make_case(batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=16,
                    seq_lens=[0, 5], sinks=True, seed=4)
    _, lse = oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens,
                                  return_lse=True, **c.kwargs())
    torch.testing.assert_close(lse[0, 0], c.sinks.reshape(-1).to(torch.float64))
    c.sinks = None
    _, lse = oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens,
                                  return_lse=True, **c.kwargs())
    assert torch.isneginf(lse[0]).all() and torch.isfinite(lse[1]).all()


def _split_case(c: W.Case, prefix_pages):
    """The same problem over the first prefix_pages pages of every sequence
    (prefix) and over the rest (suffix: the page table shifted, lengths
    reduced).  Only valid without window, mask and speculative tokens, where
    key positions do not matter."""
    ps = c.page_size
    pre = W.Case(**{**c.__dict__})
    pre.seq_lens = torch.clamp(c.seq_lens.to(torch.int64), max=prefix_pages * ps).to(torch.int32)
    pre.sinks = None  # the sink counts once: on the suffix side
    suf = W.Case(**{**c.__dict__})
    suf.page_table = torch.roll(c.page_table, -prefix_pages, dims=1).contiguous()
    suf.seq_lens = (c.seq_lens.to(torch.int64) - pre.seq_lens.to(torch.int64)).to(torch.int32)
    return pre, suf


@pytest.mark.parametrize("sinks", [False, True])
def test_merge_of_prefix_and_suffix_equals_full_attention(sinks):
    c = W.make_case(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=16, page_size=16,
                    seq_lens=[70, 40, 100], sinks=sinks, seed=31, pages_per_seq=8)
    pre, suf = _split_case(c, prefix_pages=2)
    outs = []
    for part in (pre, suf):
        o, l = oracle.xqa_attention(part.q, part.k_cache, part.v_cache, part.page_table,
                                    part.seq_lens, return_lse=True, **part.kwargs())
        B, qs, Hq, Dv = o.shape
        outs.append((o.reshape(B * qs, Hq, Dv), l.reshape(B * qs, Hq)))
    merged, _ = oracle.merge_attn_states(outs[0][0], outs[0][1], outs[1][0], outs[1][1])
    ref = dense_reference(c)
    torch.testing.assert_close(merged, ref.reshape(merged.shape), rtol=1e-10, atol=1e-12)


def test_merge_lse_is_logaddexp_and_rows_past_the_prefix_take_the_suffix():
    g = torch.Generator().manual_seed(5)
    T, H, D = 6, 3, 4
    po, so = torch.randn(T, H, D, generator=g, dtype=torch.float64), torch.randn(T, H, D, generator=g,
                                                                                dtype=torch.float64)
    pl, sl = torch.randn(T, H, generator=g, dtype=torch.float64), torch.randn(T, H, generator=g,
                                                                            dtype=torch.float64)
    pl[0, 0] = -math.inf            # an empty prefix: the suffix alone
    pl[1, 1] = sl[1, 1] = -math.inf  # both empty: zeros and -inf
    out, lse = oracle.merge_attn_states(po, pl, so, sl, n_with_prefix=4)
    torch.testing.assert_close(out[4:], so[4:])
    torch.testing.assert_close(lse[4:], sl[4:])
    torch.testing.assert_close(out[0, 0], so[0, 0])
    assert torch.equal(out[1, 1], torch.zeros(D, dtype=torch.float64)) and torch.isneginf(lse[1, 1])
    keep = torch.ones(T, H, dtype=torch.bool)
    keep[1, 1] = False
    keep[4:] = False
    torch.testing.assert_close(lse[keep], torch.logaddexp(pl, sl)[keep])
    w = torch.exp(pl - lse)[..., None]
    torch.testing.assert_close(out[:4][keep[:4]], (w * po + torch.exp(sl - lse)[..., None] * so)[:4][keep[:4]])


def test_encode_e4m3_matches_torch_cast_in_range_and_saturates():
    g = torch.Generator().manual_seed(9)
    x = torch.cat([torch.randn(4000, generator=g, dtype=torch.float64) * s for s in (0.003, 0.1, 3, 90)])
    # every code's value and every midpoint between neighbours (ties to even)
    codes = torch.arange(0, 127, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64)
    x = torch.cat([x, vals, (vals[1:] + vals[:-1]) / 2, -vals])
    x = x[x.abs() <= 448]
    want = x.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(oracle.encode_e4m3(x), want)
    big = torch.tensor([449.0, 464.0, 1e6, -500.0], dtype=torch.float64)
    assert oracle.encode_e4m3(big).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
