"""Randomised parity: seeded draws over the whole argument space of the decode
call (dtypes, head dims, group sizes, speculative rows, page sizes, layouts,
lengths, windows, sinks, masks, scales, split counts) against the float64
oracle, so that combinations the named sweeps do not cross are covered too.

Each case is drawn from its own seed; the test id spells the draw out, so a
failing case can be rebuilt from its id alone.  Tolerances are those of the
named parity tests: max-abs 1e-2 (16-bit K/V) or 3e-2 (fp8 K/V) beyond the
output's own rounding, and a relative-L2 bound of 1e-2; each draw runs again
returning the log-sum-exp (max-abs 3e-3, -inf rows alike), which must leave
the output bit for bit unchanged.
"""

import random

import pytest
import torch

import oracle
from paged_kv_decode_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu

F8 = torch.float8_e4m3fn
LSE_TOL = 3e-3  # natural-log units, as the named log-sum-exp tests
DT = {"bf16": torch.bfloat16, "f16": torch.float16, "e4m3": F8}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_20_gb300 import build as B
    B.build()


def gqa_draw(seed):
    r = random.Random(seed)
    kv = r.choice(["bf16", "f16", "e4m3", "e4m3"])
    q = r.choice(["bf16", "f16"]) if kv == "e4m3" else kv
    d = 128 if kv == "e4m3" else r.choice([64, 128])
    hkv = r.choice([1, 2, 3, 4])
    g = r.choice([1, 2, 3, 4, 5, 8, 12, 16, 32, 64])
    qs = r.choice([1, 1, 1, 2, 3, 4, 5, 8])
    while g * qs > 256:
        qs = max(1, qs // 2)
    ps = r.choice([16, 32, 64, 128])
    lens = []
    for _ in range(r.choice([1, 2, 3, 4])):
        kind = r.random()
        if kind < 0.1:
            lens.append(0)
        elif kind < 0.3:
            lens.append(r.choice([qs, qs + 1, ps, ps + 1, 2 * ps - 1]))
        elif kind < 0.45:
            lens.append(r.randint(900, 5000))
        else:
            lens.append(r.randint(qs, 900))
    return dict(kv=kv, q=q, d=d, hkv=hkv, g=g, qs=qs, ps=ps, lens=lens,
                layout=r.choice(["NHD", "HND"]),
                win=r.choice([0, 0, 1, r.randint(2, 400)]),
                sinks=r.random() < 0.4,
                mask=("causal" if qs > 1 and r.random() < 0.7 else None),
                q_scale=round(r.uniform(0.5, 2.0), 3),
                kv_scale=(0.05 if kv == "e4m3" else round(r.uniform(0.5, 1.5), 3)),
                rcp_out=r.choice([1.0, 1.0, 0.5]),
                sm=r.choice([None, None, 1, 7, 40, 10000]))


def mla_draw(seed):
    r = random.Random(seed)
    kv = r.choice(["bf16", "e4m3"])
    heads = r.choice([8, 16, 24, 32, 64, 128])
    qs = r.choice([1, 1, 2, 3])
    while heads * qs > 128:
        qs -= 1
    lens = [r.choice([0, 1, r.randint(2, 300), r.randint(300, 2500)]) for _ in range(r.choice([1, 2, 3]))]
    lens = [L if L == 0 else max(L, qs) for L in lens]
    return dict(kv=kv, heads=heads, qs=qs, ps=r.choice([16, 32, 64, 128]), lens=lens,
                win=r.choice([0, 0, r.randint(1, 600)]), sinks=r.random() < 0.4,
                mask=("causal" if qs > 1 and r.random() < 0.7 else None),
                rcp_out=r.choice([1.0, 0.5]), sm=r.choice([None, 2, 40, 1000]))


def _id(d):
    return ",".join(f"{k}={v}" for k, v in d.items()).replace(" ", "")


GQA_SEEDS = list(range(1000, 1096))
MLA_SEEDS = list(range(2000, 2024))
GQA_CASES = [(s, gqa_draw(s)) for s in GQA_SEEDS]
MLA_CASES = [(s, mla_draw(s)) for s in MLA_SEEDS]


def run_and_compare(c, tol, sm):
    """tol bounds the decode's error; on top of it each output element keeps
    its own rounding to the 16-bit output type (half an ulp: 2^-9 of |out|
    for bf16, 2^-11 for f16), which alone passes 1e-2 once |out| >= 4."""
    from paged_kv_decode_20_gb300.runner import Decoder
    kw = {} if sm is None else {"sm_count": sm}
    dec = Decoder(c.to("cuda"), **kw)
    outs = []
    for _ in range(2):
        dec.output.fill_(float("nan"))
        outs.append(dec.run().clone())
    torch.cuda.synchronize()
    assert dec.error_bits() == 0, f"error word {dec.error_bits()}"
    assert int(dec.semaphores.abs().sum()) == 0, "semaphores must be left zeroed"
    assert torch.equal(outs[0], outs[1]), "repeat calls must agree bit for bit"
    got = outs[0].cpu().to(torch.float64)
    ref = oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens, **c.kwargs())
    assert not torch.isnan(got).any(), "NaN in output"
    half_ulp = 2.0 ** -9 if outs[0].dtype == torch.bfloat16 else 2.0 ** -11
    err = ((got - ref).abs() - half_ulp * ref.abs()).max().item()
    l2 = ((got - ref).norm() / ref.norm().clamp_min(1e-30)).item()
    assert err <= tol, f"max abs error {err:.3e} > {tol}"
    assert l2 <= 1e-2, f"relative L2 error {l2:.3e}"
    # the same draw with the log-sum-exp returned: the output must not change
    dec2 = Decoder(c.to("cuda"), lse=True, **kw)
    dec2.lse.fill_(float("nan"))
    out2 = dec2.run().clone()
    torch.cuda.synchronize()
    assert dec2.error_bits() == 0
    assert torch.equal(out2, outs[0]), "the log-sum-exp output changed the attention output"
    _, ref_lse = oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens, return_lse=True,
                                      **c.kwargs())
    got_lse = dec2.lse.cpu()
    assert torch.equal(torch.isneginf(got_lse), torch.isneginf(ref_lse)), "-inf rows differ"
    fin = torch.isfinite(ref_lse)
    if fin.any():
        lerr = (got_lse.to(torch.float64)[fin] - ref_lse[fin]).abs().max().item()
        assert lerr <= LSE_TOL, f"lse max abs {lerr:.3e}"


@pytest.mark.parametrize("seed,d", GQA_CASES, ids=[_id(d) for _, d in GQA_CASES])
def test_gqa_random_draw(seed, d):
    f8 = d["kv"] == "e4m3"
    c = W.make_case(batch=len(d["lens"]), num_q_heads=d["hkv"] * d["g"], num_kv_heads=d["hkv"],
                    head_dim=d["d"], page_size=d["ps"], seq_lens=d["lens"], kv_layout=d["layout"],
                    q_dtype=DT[d["q"]], kv_dtype=DT[d["kv"]], q_seq_len=d["qs"], sinks=d["sinks"],
                    sliding_win_size=d["win"], mask=d["mask"], q_scale=d["q_scale"],
                    kv_scale=d["kv_scale"], kv_divisor=d["kv_scale"] if f8 else 1.0,
                    rcp_out_scale=d["rcp_out"], seed=seed)
    run_and_compare(c, 3e-2 if f8 else 1e-2, d["sm"])


@pytest.mark.parametrize("seed,d", MLA_CASES, ids=[_id(d) for _, d in MLA_CASES])
def test_mla_random_draw(seed, d):
    f8 = d["kv"] == "e4m3"
    extra = dict(q_dtype=F8, kv_dtype=F8, q_scale=0.05, kv_scale=0.05, q_divisor=0.05,
                 kv_divisor=0.05) if f8 else {}
    c = W.make_case(batch=len(d["lens"]), num_q_heads=d["heads"], num_kv_heads=1, head_dim=576,
                    v_head_dim=512, mla=True, page_size=d["ps"], seq_lens=d["lens"], kv_layout="NHD",
                    q_seq_len=d["qs"], softmax_scale=(128 + 64) ** -0.5, sinks=d["sinks"],
                    sliding_win_size=d["win"], mask=d["mask"], rcp_out_scale=d["rcp_out"], seed=seed,
                    **extra)
    run_and_compare(c, 3e-2 if f8 else 1e-2, d["sm"])
