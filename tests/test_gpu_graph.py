"""The decode calls record into a CUDA graph and replay bit for bit: they
make no host synchronisation, allocation or blocking call while the stream
is captured, so a serving loop can replay a whole decode step as one graph
(CUDA graphs in place of a tracing compiler)."""

import pytest
import torch

from paged_kv_decode_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_20_gb300 import build as B
    B.build()


@pytest.mark.parametrize("idx", [1, 4, 5])
def test_decode_replays_from_a_cuda_graph(idx):
    from paged_kv_decode_20_gb300.runner import Decoder
    case = W.workload(idx, device="cuda", poison=False, batch=4 if idx == 5 else None)
    dec = Decoder(case, lse=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dec.run(s)  # warm: the first call looks up driver entry points
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = dec.output.clone()
    eager_lse = dec.lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dec.run(s)
    dec.output.fill_(float("nan"))
    dec.lse.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(dec.output, eager)
    assert torch.equal(dec.lse, eager_lse)
    assert dec.error_bits() == 0
    assert int(dec.semaphores.abs().sum()) == 0
