"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
identical seeded inputs, element by element.

Tolerances: max-abs 1e-2 for 16-bit K/V and 3e-2 for fp8 K/V (bf16/fp16
output), plus a relative-L2 bound of 1e-2 so that small-magnitude outputs
(flat softmax over thousands of keys) are still held to the arithmetic's
precision: P is rounded to 16 bits before the P.V product (relative error
<= 2^-8 per weight for bf16) and the output is rounded to 16 bits once.
"""

import pytest
import torch

import oracle
from paged_kv_decode_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_16 = 1e-2
TOL_FP8 = 3e-2
REL_L2 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_20_gb300 import build as B
    B.build()


def run_gpu(case_cpu, runs=2, **kw):
    from paged_kv_decode_20_gb300.runner import Decoder
    dec = Decoder(case_cpu.to("cuda"), **kw)
    outs = []
    for _ in range(runs):
        dec.output.fill_(float("nan"))
        outs.append(dec.run().clone())
    torch.cuda.synchronize()
    assert int(dec.semaphores.abs().sum()) == 0, "semaphores must be left zeroed"
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "repeat calls must agree bit for bit"
    return outs[0].cpu(), dec


def compare(got, ref, tol, rel=REL_L2):
    got = got.to(torch.float64)
    assert not torch.isnan(got).any(), "NaN in output"
    err = (got - ref).abs().max().item()
    l2 = ((got - ref).norm() / ref.norm().clamp_min(1e-30)).item()
    assert err <= tol, f"max abs error {err:.3e} > {tol}"
    assert l2 <= rel, f"relative L2 error {l2:.3e} > {rel}"
    return err, l2


def oracle_full(c, **over):
    kw = c.kwargs()
    kw.update(over)
    return oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens, **kw)


def check(case, tol=None, **kw):
    tol = tol if tol is not None else (TOL_FP8 if case.k_cache.dtype == torch.float8_e4m3fn else TOL_16)
    got, dec = run_gpu(case, **kw)
    assert dec.error_bits() == 0
    return compare(got, oracle_full(case), tol)


# ---------------------------------------------------------------- named workloads, reduced batch

def test_tiny_gqa_workload():
    check(W.workload(1))


def test_llama3_8b_workload_first_sequences():
    check(W.workload(2, batch=3))


def test_fp8_long_context_workload_one_sequence():
    check(W.workload(3, batch=1))


def test_window_sinks_spec_workload_first_sequences():
    check(W.workload(4, batch=4))


# ---------------------------------------------------------------- sweeps

SWEEP = []
for dt in ("bf16", "f16", "e4m3"):
    for ps in (16, 32, 64, 128):
        for layout in ("NHD", "HND"):
            SWEEP.append((dt, ps, layout))


@pytest.mark.parametrize("dt,ps,layout", SWEEP, ids=[f"{a}-ps{b}-{c}" for a, b, c in SWEEP])
def test_dtype_page_layout_sweep(dt, ps, layout):
    q_dtype = torch.float16 if dt == "f16" else torch.bfloat16
    kv_dtype = torch.float8_e4m3fn if dt == "e4m3" else q_dtype
    extra = dict(kv_scale=0.5, kv_divisor=0.5) if dt == "e4m3" else {}
    c = W.make_case(batch=3, num_q_heads=16, num_kv_heads=2, head_dim=128, page_size=ps,
                    seq_lens=[1, ps * 3 + 5, 700], kv_layout=layout, q_dtype=q_dtype,
                    kv_dtype=kv_dtype, seed=ps + len(layout), **extra)
    check(c)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32])
def test_group_sizes_d128(G):
    c = W.make_case(batch=2, num_q_heads=2 * G, num_kv_heads=2, head_dim=128, page_size=32,
                    seq_lens=[300, 77], seed=G)
    check(c)


@pytest.mark.parametrize("G,qs", [(4, 1), (8, 2), (16, 2), (8, 4), (16, 4)])
def test_group_and_spec_rows_d64(G, qs):
    c = W.make_case(batch=2, num_q_heads=2 * G, num_kv_heads=2, head_dim=64, page_size=16,
                    seq_lens=[200, 45], q_seq_len=qs, mask="causal" if qs > 1 else None,
                    sinks=True, seed=10 * G + qs)
    check(c)


# Large grouped tiles (speculative tokens x a large GQA group): up to 64 rows per
# kv head run as one CTA per (sequence, kv head, split) whose four consumer
# warps split the rows (warp row groups), so each KV page is read once; 128
# rows take two such row groups.
LARGE = [(8, 4, torch.bfloat16), (16, 2, torch.bfloat16), (16, 4, torch.bfloat16), (32, 2, torch.float16),
         (32, 4, torch.bfloat16), (8, 4, torch.float8_e4m3fn), (16, 4, torch.float8_e4m3fn),
         (24, 1, torch.bfloat16)]


@pytest.mark.parametrize("G,qs,kv", LARGE, ids=[f"G{g}-qs{q}-{str(k).split('.')[-1]}" for g, q, k in LARGE])
def test_large_group_tiles_d128(G, qs, kv):
    f8 = kv == torch.float8_e4m3fn
    extra = dict(kv_scale=0.25, kv_divisor=0.25) if f8 else {}
    c = W.make_case(batch=3, num_q_heads=2 * G, num_kv_heads=2, head_dim=128, page_size=32 if qs % 2 else 64,
                    seq_lens=[900, 37, 2500], q_seq_len=qs, mask="causal" if qs > 1 else None, sinks=True,
                    kv_layout="HND" if G % 16 else "NHD", q_dtype=torch.float16 if kv == torch.float16 else
                    torch.bfloat16, kv_dtype=kv, seed=100 * G + qs, **extra)
    check(c, tol=TOL_FP8 if f8 else TOL_16)


@pytest.mark.parametrize("sm_count", [1, 30, 10000])
def test_large_group_tiles_split_counts(sm_count):
    c = W.make_case(batch=2, num_q_heads=64, num_kv_heads=4, head_dim=128, page_size=16,
                    seq_lens=[3000, 130], q_seq_len=4, mask="causal", sinks=True, sliding_win_size=700,
                    seed=77)
    check(c, sm_count=sm_count)



@pytest.mark.parametrize("sm_count", [1, 3, 7])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_large_group_persistent_ctas_walk_many_units(sm_count, layout):
    """More unsplit tensor-core units than CTA slots: resident CTAs take the
    units in turn (here 20 units on 1, 3 or 7 CTAs), with empty and
    one-token sequences, a window, sinks, a spec mask and two row groups per
    kv head (144 rows: 128 + 16)."""
    c = W.make_case(batch=5, num_q_heads=96, num_kv_heads=2, head_dim=128, page_size=32,
                    seq_lens=[0, 700, 3, 300, 129], q_seq_len=3, mask="causal", sinks=True,
                    sliding_win_size=200, kv_layout=layout, seed=91)
    check(c, sm_count=sm_count)


@pytest.mark.parametrize("G,qs", [(16, 4), (32, 4), (64, 1)])
def test_large_group_tiles_d64(G, qs):
    c = W.make_case(batch=2, num_q_heads=2 * G, num_kv_heads=2, head_dim=64, page_size=16,
                    seq_lens=[600, 45], q_seq_len=qs, mask="causal" if qs > 1 else None,
                    sinks=True, seed=7 * G + qs)
    check(c)


def test_f16_query_with_fp8_cache():
    c = W.make_case(batch=2, num_q_heads=8, num_kv_heads=1, head_dim=128, page_size=64,
                    seq_lens=[513, 1000], q_dtype=torch.float16, kv_dtype=torch.float8_e4m3fn,
                    kv_scale=0.05, kv_divisor=0.05, q_scale=0.7, seed=31)
    check(c)


def test_bf16_query_far_outside_f16_range_with_fp8_cache():
    # The fp8 path feeds an f16 MMA; a power-of-two rescale keeps q exact.
    c = W.make_case(batch=1, num_q_heads=8, num_kv_heads=1, head_dim=128, page_size=32,
                    seq_lens=[257], kv_dtype=torch.float8_e4m3fn, q_mult=1.0e6,
                    softmax_scale=1.0e-7, seed=32)
    check(c)


def test_scales_sinks_window_mask_and_rcp_out():
    c = W.make_case(batch=3, num_q_heads=16, num_kv_heads=4, head_dim=64, page_size=16,
                    seq_lens=[40, 129, 500], q_seq_len=3, mask="causal", sinks=True,
                    sliding_win_size=37, q_scale=1.3, kv_scale=0.8, rcp_out_scale=2.0, seed=33)
    check(c)


def test_spec_without_mask_and_full_mask():
    c = W.make_case(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                    seq_lens=[50, 90], q_seq_len=4, seed=34)
    check(c)
    c.mask = W.full_spec_mask(2, 4)
    check(c)


def test_device_scale_tensors_match_host_scales():
    from paged_kv_decode_20_gb300 import xqa as X
    c = W.make_case(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64,
                    seq_lens=[300, 700], kv_dtype=torch.float8_e4m3fn, kv_scale=0.25,
                    kv_divisor=0.25, q_scale=1.5, seed=35).to("cuda")
    ref = oracle_full(c.to("cpu"))
    out = torch.empty((2, 1, 8, 128), dtype=torch.bfloat16, device="cuda")
    p = X.make_params(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens, out, num_kv_heads=2,
                      page_size=64, q_scale=torch.tensor([1.5], device="cuda"),
                      kv_scale=torch.tensor([0.25], device="cuda"))
    ws = torch.zeros(max(X.xqa_workspace_size(p), 16), dtype=torch.uint8, device="cuda")
    sem = torch.zeros(X.xqa_semaphore_count(p), dtype=torch.int32, device="cuda")
    X.xqa_decode(p, ws, sem)
    torch.cuda.synchronize()
    compare(out.cpu(), ref, TOL_FP8)


def test_peaked_softmax():
    c = W.make_case(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                    seq_lens=[33, 400], q_mult=8.0, seed=36)
    check(c)


# ---------------------------------------------------------------- edge cases

def test_empty_sequence_gives_zeros_and_length_one_gives_v0():
    c = W.make_case(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                    seq_lens=[0, 1, 16], sinks=True, seed=40)
    got, _ = run_gpu(c)
    assert torch.equal(got[0], torch.zeros_like(got[0]))
    compare(got, oracle_full(c), TOL_16)


def test_window_of_one_and_window_past_the_start():
    c = W.make_case(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=32,
                    seq_lens=[70, 1000], sliding_win_size=1, seed=41)
    check(c)
    c.sliding_win_size = 5000
    check(c)


@pytest.mark.parametrize("sm_count", [1, 20, 10000])
def test_split_counts_agree(sm_count):
    c = W.make_case(batch=2, num_q_heads=8, num_kv_heads=1, head_dim=128, page_size=16,
                    seq_lens=[4000, 9], pages_per_seq=256, seed=42)
    check(c, sm_count=sm_count)


def test_long_table_full_length_sequences():
    c = W.make_case(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=128,
                    seq_lens=[128 * 40, 128 * 40], seed=43)
    check(c)


def test_length_above_table_is_clamped_and_flagged():
    c = W.make_case(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                    seq_lens=[64, 30], pages_per_seq=4, seed=44, poison=False)
    ref = oracle_full(c)
    c.seq_lens[0] = 1000  # beyond pages_per_seq * page_size = 64
    got, dec = run_gpu(c)
    assert dec.error_bits() & 1
    compare(got, ref, TOL_16)


def test_page_index_out_of_range_reads_zeros_and_is_flagged():
    c = W.make_case(batch=1, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                    seq_lens=[48], seed=45, poison=False)
    c.page_table[0, 1] = 1 << 20  # page 1 of 3 points outside the pool
    kz = c.k_cache.clone()
    vz = c.v_cache.clone()
    got, dec = run_gpu(c)
    assert dec.error_bits() & 1
    # the oracle sees the same problem with that page's rows as zeros
    zero_page = torch.zeros((1,) + tuple(c.k_cache.shape[1:]), dtype=c.k_cache.dtype)
    k2 = torch.cat([kz, zero_page])
    v2 = torch.cat([vz, zero_page])
    t2 = c.page_table.clone()
    t2[0, 1] = c.k_cache.shape[0]
    ref = oracle.xqa_attention(c.q, k2, v2, t2, c.seq_lens, **c.kwargs())
    compare(got, ref, TOL_16)


def test_nan_poison_outside_the_sequence_never_leaks():
    # every unused page and every slot past seq_len holds NaN
    c = W.make_case(batch=4, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64,
                    seq_lens=[1, 63, 65, 130], pool_pages=40, seed=46, poison=True)
    check(c)
