"""The host's split plan on the measured workload shapes, and the read-only
bandwidth probe (a measurement aid beside the decode path)."""
import ctypes

import pytest
import torch

from paged_kv_decode_20_gb300 import xqa as X

pytestmark = pytest.mark.gpu


def params(**over):
    """A parameter block with fake (never dereferenced) pointers: the plan
    reads only sizes."""
    p = X.XqaParams()
    p.q = p.k_cache = p.v_cache = p.page_table = p.seq_lens = p.output = 0x10000
    p.q_dtype = p.kv_dtype = p.out_dtype = X.XQA_BF16
    p.kv_layout = X.XQA_HND
    p.num_pages = 1 << 16
    p.q_scale = p.kv_scale = p.rcp_out_scale = 1.0
    p.q_seq_len = 1
    for k, v in over.items():
        setattr(p, k, v)
    return p


def splits(lib, p, rows, sm_count=152):
    """Splits per (sequence, kv head) that the workspace size implies."""
    ws = lib.xqa_workspace_size(ctypes.byref(p), sm_count)
    assert ws != ctypes.c_size_t(-1).value, lib.xqa_last_error()
    units = p.batch_size * p.num_kv_heads
    per_split = units * rows * (p.head_dim + 4) * 4
    return 1 if ws == 0 else ws // per_split


@pytest.fixture(scope="module")
def lib():
    return X.load()


def test_split_plan_on_the_measured_shapes(lib):
    # Llama-3-8B-shaped decode (B64 Hq32 Hkv8, 8192-token bound): one split
    w2 = params(batch_size=64, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64, pages_per_seq=128)
    assert splits(lib, w2, 16) == 1
    # fp8 long context (B128 Hq64 Hkv8, 32768 tokens): two splits fill the last wave
    w3 = params(batch_size=128, num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=32, pages_per_seq=1024,
                kv_dtype=X.XQA_E4M3, kv_layout=X.XQA_NHD)
    assert splits(lib, w3, 16) == 2
    # one 32768-token sequence: enough splits for about one CTA per SM
    b1 = params(batch_size=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64, pages_per_seq=512)
    assert 12 <= splits(lib, b1, 16) <= 38


def test_read_probe_streams_a_buffer():
    buf = torch.ones(64 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(4096, dtype=torch.int32, device="cuda")
    X.read_bandwidth_probe(buf, sink)
    torch.cuda.synchronize()
    # the sink is written only when a CTA's folded word equals a fixed
    # constant; all-ones data folds to zero
    assert int(sink.abs().sum()) == 0


def test_single_long_sequence_runs_many_splits_and_matches_the_oracle():
    """One 32768-token sequence: the plan splits it across about one CTA per
    SM (the last CTA of each kv head merges the partials); every row against
    the oracle."""
    import oracle
    from paged_kv_decode_20_gb300 import workloads as W
    from paged_kv_decode_20_gb300.runner import Decoder
    c = W.make_case(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64, seq_lens=[32768],
                    kv_layout="HND", pages_per_seq=512, seed=61, device="cuda", poison=False)
    dec = Decoder(c)
    assert dec.workspace.numel() > 16  # split partials in use
    out = dec.run()
    torch.cuda.synchronize()
    assert dec.error_bits() == 0
    assert int(dec.semaphores.abs().sum()) == 0
    cc = c.to("cpu")
    ref = oracle.xqa_attention(cc.q, cc.k_cache, cc.v_cache, cc.page_table, cc.seq_lens, **cc.kwargs())
    got = out.cpu().to(torch.float64)
    assert (got - ref).abs().max().item() <= 1e-2
    assert ((got - ref).norm() / ref.norm()).item() <= 1e-2
