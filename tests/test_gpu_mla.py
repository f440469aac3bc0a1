"""GPU parity of the MLA latent decode kernel (one 576-wide latent kv head, V =
its first 512 elements; vLLM Kimi-K3 MultiHeadLatentAttention page) against
the float64 oracle on identical seeded inputs.  Tolerance: max-abs 1e-2 (bf16
cache) or 3e-2 (e4m3 cache and query, the fp8 bound) and relative L2 1e-2
(bf16 output; P rounded to bf16, or to f16 against the widened e4m3 V)."""

import pytest
import torch

import oracle
from paged_kv_decode_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-2
SCALE = (128 + 64) ** -0.5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_20_gb300 import build as B
    B.build()


F8 = torch.float8_e4m3fn
TOL_F8 = 3e-2


def mla_case(lens, ps=64, seed=0, heads=128, qs=1, dtype=torch.bfloat16, **kw):
    if dtype == F8:
        # e4m3 latent cache and query drawn as N(0,1)/scale (the fp8 recipe)
        kw = dict(dict(q_dtype=F8, kv_dtype=F8, q_scale=0.05, kv_scale=0.05, q_divisor=0.05,
                       kv_divisor=0.05), **kw)
    return W.make_case(batch=len(lens), num_q_heads=heads, num_kv_heads=1, head_dim=576,
                       v_head_dim=512, mla=True, page_size=ps, seq_lens=lens, kv_layout="NHD",
                       q_seq_len=qs, softmax_scale=SCALE, seed=seed, **kw)


def run_and_compare(c, tol=TOL, runs=2, out_round=False, **kw):
    from paged_kv_decode_20_gb300.runner import Decoder
    dec = Decoder(c.to("cuda"), **kw)
    outs = []
    for _ in range(runs):
        dec.output.fill_(float("nan"))
        outs.append(dec.run().clone())
    torch.cuda.synchronize()
    assert dec.error_bits() == 0, f"error word {dec.error_bits()}"
    assert int(dec.semaphores.abs().sum()) == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    got = outs[0].cpu().to(torch.float64)
    ref = oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens, **c.kwargs())
    assert not torch.isnan(got).any()
    d = (got - ref).abs()
    if out_round:
        # the output's own rounding to bf16 (half an ulp, 2^-9 relative) on top of
        # the decode bound: peaked rows of short sequences reach |out| ~ 3.5
        d = d - 2.0 ** -9 * ref.abs()
    err = d.max().item()
    l2 = ((got - ref).norm() / ref.norm().clamp_min(1e-30)).item()
    assert err <= tol, f"max abs {err:.3e}"
    assert l2 <= 1e-2, f"rel L2 {l2:.3e}"
    return err, l2


def test_mla_workload_first_sequences():
    run_and_compare(W.workload(5, batch=2))


@pytest.mark.parametrize("ps", [16, 32, 64, 128])
def test_mla_page_sizes(ps):
    run_and_compare(mla_case([1, 63, 64, 65, 700], ps=ps, seed=ps))


@pytest.mark.parametrize("sm_count", [2, 40, 1000])
def test_mla_split_counts(sm_count):
    run_and_compare(mla_case([5000, 130], seed=3), sm_count=sm_count)


def test_mla_peaked_rows_force_rescales():
    run_and_compare(mla_case([3000, 77], seed=4, q_mult=4.0))


def test_mla_sinks_window_and_spec_tokens():
    c = mla_case([900, 300], seed=5, heads=64, qs=2, sinks=True, sliding_win_size=200,
                 mask="causal")
    run_and_compare(c)


def test_mla_empty_and_nan_poison():
    c = mla_case([0, 1, 129], seed=6, pool_pages=12, poison=True)
    run_and_compare(c)


def test_mla_persistent_clusters_loop_over_many_sequences():
    """Few persistent clusters (sm_count 8 -> 4 clusters) each run dozens of
    sequences one after another, re-arming their barriers per piece; the
    lengths mix empty, one-token, page-boundary and multi-page sequences so that
    slices start and end inside sequences."""
    g = torch.Generator().manual_seed(11)
    lens = torch.randint(0, 400, (60,), generator=g).tolist()
    lens[:6] = [0, 1, 63, 64, 65, 0]
    run_and_compare(mla_case(lens, ps=32, seed=12), sm_count=8)


def test_mla_large_batch_takes_fixed_splits():
    """Batches above 256 sequences launch one cluster per (sequence, split)
    instead of persistent clusters."""
    g = torch.Generator().manual_seed(13)
    lens = torch.randint(1, 160, (260,), generator=g).tolist()
    run_and_compare(mla_case(lens, ps=64, seed=14), runs=1, out_round=True)


# ---------------------------------------------------------------- padded query rows
@pytest.mark.parametrize("heads,qs", [(16, 1), (32, 1), (64, 1), (32, 2), (24, 3)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, F8], ids=["bf16", "e4m3"])
def test_mla_fewer_than_128_query_rows(heads, qs, dtype):
    """Tensor-parallel shards of the heads (num_local_heads = num_heads / tp)
    run as a 128-row tile whose rows past heads x q_seq_len are padding: never
    stored, no lse written (checked by NaN-filled outputs and lse)."""
    from paged_kv_decode_20_gb300.runner import Decoder
    c = mla_case([700, 65, 2000], seed=20 + heads + qs, heads=heads, qs=qs, dtype=dtype, sinks=True,
                 mask="causal" if qs > 1 else None)
    run_and_compare(c, tol=TOL_F8 if dtype == F8 else TOL)
    dec = Decoder(c.to("cuda"), lse=True)
    dec.lse.fill_(float("nan"))
    dec.run()
    _, ref_lse = oracle.xqa_attention(c.q, c.k_cache, c.v_cache, c.page_table, c.seq_lens,
                                      return_lse=True, **c.kwargs())
    torch.cuda.synchronize()
    assert (dec.lse.cpu().double() - ref_lse).abs().max().item() <= 3e-3


# ---------------------------------------------------------------- e4m3 latent cache and query
def test_mla_e4m3_workload_first_sequences():
    run_and_compare(W.workload(5, batch=2, kv_dtype=F8), tol=TOL_F8)


@pytest.mark.parametrize("ps", [16, 32, 64, 128])
def test_mla_e4m3_page_sizes(ps):
    run_and_compare(mla_case([1, 63, 64, 65, 700], ps=ps, seed=40 + ps, dtype=F8), tol=TOL_F8)


@pytest.mark.parametrize("sm_count", [2, 40, 1000])
def test_mla_e4m3_split_counts(sm_count):
    run_and_compare(mla_case([5000, 130], seed=43, dtype=F8), tol=TOL_F8, sm_count=sm_count)


def test_mla_e4m3_peaked_rows_force_rescales():
    # (q x 2.5 keeps the e4m3 query inside its finite range: |q| <= ~250)
    run_and_compare(mla_case([3000, 77], seed=44, dtype=F8, q_mult=2.5), tol=TOL_F8, out_round=True)


def test_mla_e4m3_sinks_window_and_spec_tokens():
    c = mla_case([900, 300], seed=45, heads=64, qs=2, dtype=F8, sinks=True, sliding_win_size=200,
                 mask="causal")
    run_and_compare(c, tol=TOL_F8)


def test_mla_e4m3_empty_and_nan_poison():
    c = mla_case([0, 1, 129], seed=46, pool_pages=12, poison=True, dtype=F8)
    run_and_compare(c, tol=TOL_F8)


def test_mla_e4m3_scales_from_device_and_output_scale():
    """q_scale and kv_scale as device scalars, rcp_out_scale != 1."""
    from paged_kv_decode_20_gb300 import xqa as X
    c = mla_case([1500, 40], seed=47, dtype=F8, rcp_out_scale=0.5).to("cuda")
    out = torch.empty((2, 1, 128, 512), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(1 << 26, dtype=torch.uint8, device="cuda")
    sems = torch.zeros(2 * 2 + 2, dtype=torch.int32, device="cuda")
    X.xqa_mla(c.q, c.k_cache, c.page_table, c.seq_lens, out, ws, sems, page_size=64, v_head_dim=512,
              softmax_scale=SCALE, q_scale=torch.tensor([0.05], device="cuda"),
              kv_scale=torch.tensor([0.05], device="cuda"), rcp_out_scale=0.5)
    torch.cuda.synchronize()
    cc = c.to("cpu")
    ref = oracle.xqa_attention(cc.q, cc.k_cache, cc.v_cache, cc.page_table, cc.seq_lens, **cc.kwargs())
    assert (out.cpu().double() - ref).abs().max().item() <= TOL_F8


def test_mla_e4m3_persistent_clusters_loop_over_many_sequences():
    g = torch.Generator().manual_seed(48)
    lens = torch.randint(0, 400, (60,), generator=g).tolist()
    lens[:6] = [0, 1, 63, 64, 65, 0]
    run_and_compare(mla_case(lens, ps=32, seed=49, dtype=F8), tol=TOL_F8, sm_count=8)


def test_mla_e4m3_large_batch_takes_fixed_splits():
    g = torch.Generator().manual_seed(50)
    lens = torch.randint(1, 160, (260,), generator=g).tolist()
    run_and_compare(mla_case(lens, ps=64, seed=51, dtype=F8), tol=TOL_F8, runs=1, out_round=True)


# ---------------------------------------------------------------- fixed splits with merges
@pytest.mark.parametrize("dtype", [torch.bfloat16, F8], ids=["bf16", "e4m3"])
def test_mla_large_batch_with_splits(dtype):
    """Above 256 sequences each sequence takes a fixed number of splits; a large
    SM count asks for two per sequence here, so the merge kernel reads the
    partials at slots [sequence][split].  Six sequences are checked against
    the oracle (first, middle, last)."""
    from paged_kv_decode_20_gb300.runner import Decoder
    g = torch.Generator().manual_seed(60)
    lens = torch.randint(1500, 2600, (260,), generator=g).tolist()
    c = mla_case(lens, ps=64, seed=61, dtype=dtype)
    dec = Decoder(c.to("cuda"), sm_count=1000)
    dec.output.fill_(float("nan"))
    got = dec.run().clone()
    torch.cuda.synchronize()
    assert dec.error_bits() == 0
    assert int(dec.semaphores.abs().sum()) == 0
    sel = [0, 1, 2, 130, 258, 259]
    # (CPU indexing of e4m3 tensors goes through their bytes)
    q = c.q.view(torch.uint8)[sel].view(F8) if c.q.dtype == F8 else c.q[sel]
    ref = oracle.xqa_attention(q, c.k_cache, c.v_cache, c.page_table[sel], c.seq_lens[sel], **c.kwargs())
    gs = got.cpu().to(torch.float64)[sel]
    d = (gs - ref).abs() - 2.0 ** -9 * ref.abs()
    assert d.max().item() <= (TOL_F8 if dtype == F8 else TOL)
    assert ((gs - ref).norm() / ref.norm()).item() <= 1e-2
