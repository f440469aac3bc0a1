"""Parity at the named workloads' full sizes, in the launch configuration the
bench times (same generator, same Decoder, same split plan), on sampled
output rows: the oracle computes the sampled rows one by one from a compacted
copy of the sampled sequences' pages (plain data movement: index_select of the
pages and a renumbered page table)."""

import pytest
import torch

import oracle
from paged_kv_decode_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_20_gb300 import build as B
    B.build()


def compact(case, batch_idx):
    """CPU problem holding only the listed sequences and their pages."""
    ps = case.page_size
    lens = case.seq_lens.to(torch.int64).cpu()[batch_idx]
    npg = [(-(-int(L) // ps)) for L in lens]
    pps = max(1, max(npg))
    table = case.page_table.cpu()[batch_idx]
    used = torch.cat([table[j, :n] for j, n in enumerate(npg)]).to(torch.int64)
    uniq, inv = torch.unique(used, return_inverse=True)
    new_table = torch.zeros((len(batch_idx), pps), dtype=torch.int32)
    off = 0
    for j, n in enumerate(npg):
        new_table[j, :n] = inv[off:off + n].to(torch.int32)
        off += n
    idx = uniq.to(case.k_cache.device)
    k = case.k_cache.index_select(0, idx).cpu()
    v = k if case.mla else case.v_cache.index_select(0, idx).cpu()
    c = W.Case(name=case.name, q=case.q[batch_idx].cpu(), k_cache=k, v_cache=v,
               page_table=new_table, seq_lens=lens.to(torch.int32), num_kv_heads=case.num_kv_heads,
               page_size=ps, kv_layout=case.kv_layout, q_seq_len=case.q_seq_len,
               v_head_dim=case.v_head_dim,
               sinks=None if case.sinks is None else case.sinks.cpu(),
               mask=None if case.mask is None else case.mask[batch_idx].cpu(),
               q_scale=case.q_scale, kv_scale=case.kv_scale, softmax_scale=case.softmax_scale,
               sliding_win_size=case.sliding_win_size, rcp_out_scale=case.rcp_out_scale,
               mla=case.mla)
    return c


@pytest.mark.parametrize("idx,tol", [(2, 1e-2), (3, 3e-2), (4, 1e-2), (5, 1e-2), ("large_group", 1e-2)])
def test_full_size_sampled_rows(idx, tol):
    from paged_kv_decode_20_gb300.runner import Decoder
    if idx == "large_group":  # (its shortest sequences run as two splits on the tensor-core kernel)
        case = W.large_group_workload(device="cuda", poison=False)
    else:
        case = W.workload(idx, device="cuda", poison=False)
    dec = Decoder(case)
    out = dec.run()
    torch.cuda.synchronize()
    assert dec.error_bits() == 0
    B, qs, Hq, _ = case.q.shape
    lens = case.seq_lens.to(torch.int64).cpu()
    g = torch.Generator().manual_seed(100 + (idx if isinstance(idx, int) else 9))
    picks = {0, B - 1, int(lens.argmin()), int(lens.argmax())}
    picks |= set(torch.randint(0, B, (2,), generator=g).tolist())
    batch_idx = sorted(picks)
    small = compact(case, batch_idx)
    heads = sorted({0, Hq - 1, Hq // 2} | set(torch.randint(0, Hq, (3,), generator=g).tolist()))
    units, got = [], []
    out_cpu = out.cpu()
    for j, b in enumerate(batch_idx):
        for i in range(qs):
            for h in heads:
                units.append((j * qs + i) * Hq + h)
                got.append(out_cpu[b, i, h])
    ref = oracle.xqa_attention(small.q, small.k_cache, small.v_cache, small.page_table,
                               small.seq_lens, units=torch.tensor(units), **small.kwargs())
    got = torch.stack(got).to(torch.float64)
    assert not torch.isnan(got).any()
    err = (got - ref).abs().max().item()
    l2 = ((got - ref).norm() / ref.norm()).item()
    assert err <= tol, f"workload {idx}: max abs {err:.3e}"
    assert l2 <= 1e-2, f"workload {idx}: rel L2 {l2:.3e}"
