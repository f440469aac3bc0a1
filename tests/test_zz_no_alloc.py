"""xqa_decode_noalloc against xqa_decode and against the float64 oracle.

xqa_decode_noalloc serves callers that may not allocate device memory where
they run decode attention (a runtime that has reserved the GPU's memory for its
own KV-cache pool, or code whose allocator is owned elsewhere): it takes its
split workspace and tickets from a scratch array built into the library.  The
test calls it through the C ABI twice in a row -- the second call finds the
first call's leftovers in the shared array -- and checks both outputs against
the ordinary entry point with caller-provided buffers and against the oracle,
within the tolerance the parity tests use.  This file is collected last on
purpose.
"""

import ctypes

import pytest
import torch

from paged_kv_decode_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_16 = 1e-2
TOL_FP8 = 3e-2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_20_gb300 import build as B
    from paged_kv_decode_20_gb300 import xqa as X
    B.build()
    lib = X.load()
    lib.xqa_decode_noalloc.argtypes = [ctypes.POINTER(X.XqaParams), ctypes.c_void_p]
    lib.xqa_decode_noalloc.restype = ctypes.c_int
    return lib


CASES = [
    ("llama3_8b_first_8_sequences", lambda: W.workload(2, batch=8), TOL_16),
    ("fp8_two_sequences", lambda: W.workload(3, batch=2), TOL_FP8),
    ("window_sinks_spec", lambda: W.workload(4, batch=4), TOL_16),
]


@pytest.mark.parametrize("name,make,tol", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_caller_buffers_twice(lib, name, make, tol):
    from paged_kv_decode_20_gb300 import xqa as X
    from paged_kv_decode_20_gb300.runner import Decoder
    import oracle
    cpu_case = make()
    exact = oracle.xqa_attention(cpu_case.q, cpu_case.k_cache, cpu_case.v_cache, cpu_case.page_table,
                                 cpu_case.seq_lens, **cpu_case.kwargs())
    case = cpu_case.to("cuda")
    ref_dec = Decoder(case)
    ref = ref_dec.run().clone()
    out = torch.empty_like(ref)
    kw = case.kwargs()
    kw.pop("v_head_dim")
    p = X.make_params(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, out,
                      q_seq_len=case.q_seq_len, **kw)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out.fill_(float("nan"))
        st = lib.xqa_decode_noalloc(ctypes.byref(p), stream)
        assert st == X.XQA_OK, lib.xqa_last_error().decode()
        torch.cuda.synchronize()
        assert not torch.isnan(out).any()
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= tol, f"{name}: max abs difference {err:.3e}"
        err_o = (out.cpu().to(torch.float64) - exact).abs().max().item()
        assert err_o <= tol, f"{name}: max abs error against the oracle {err_o:.3e}"


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    from paged_kv_decode_20_gb300 import xqa as X
    # A long-context batch whose split workspace exceeds the built-in 64 MiB;
    # rejected on the host, so the (small) tensors are never read.
    B, pps = 4096, 4096
    q = torch.zeros((B, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((16, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((B, pps), dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    p = X.make_params(q, cache, cache, table, lens, out, num_kv_heads=8, page_size=16)
    need = X.xqa_workspace_size(p)
    assert need > (64 << 20) or X.xqa_semaphore_count(p) > (16 << 10)
    st = lib.xqa_decode_noalloc(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == X.XQA_ERR_WORKSPACE_TOO_SMALL
    assert "scratch" in lib.xqa_last_error().decode()
