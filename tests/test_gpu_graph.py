"""CUDA graphs (the stage page's graph-capture paragraph): encode and decode
captured once into a graph and launched repeatedly with new input contents;
every launch's stream is byte-identical to the oracle's for that input and
decodes back to it. Capture on a stream without scratch is refused."""
import numpy as np
import pytest

from gpu_util import lib

pytestmark = pytest.mark.gpu


def _inputs(n, k):
    import synth
    x = synth.generate(2)
    # different slices of the plane, one with a run and one all zero
    for j in range(k):
        y = x[j * 3_000_000: j * 3_000_000 + n].copy()
        if j == 2:
            y[100_000: 400_000] = 7
        if j == 3:
            y[:] = 0
        yield y


@pytest.mark.parametrize("window", [32, 64])
def test_graph_launches_repeat(orc, window):
    import torch
    g = lib()
    n, ws, cs = (2 << 20) + 12, 4, 2048
    s = torch.cuda.Stream()
    d_in = torch.zeros(n, dtype=torch.uint8, device="cuda")
    cap = g.gpulz_compress_bound(n, ws, cs)
    out = torch.zeros(cap, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    y = torch.zeros(n, dtype=torch.uint8, device="cuda")

    def calls():
        if window == 32:
            assert g.gpulz_compress(d_in, n, ws, cs, 0, out, cap, nb, s) == g.GPULZ_OK
        else:
            assert g.gpulz_compress_window(d_in, n, ws, cs, 0, window, out, cap, nb, s) == g.GPULZ_OK
        assert g.gpulz_decompress(out, y, n, s) == g.GPULZ_OK

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls()  # a direct call first: the stream's scratch exists before capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        calls()
    for x in _inputs(n, 5):
        with torch.cuda.stream(s):
            d_in.copy_(torch.from_numpy(x))
            graph.replay()
        s.synchronize()
        assert g.gpulz_device_status(s) == g.GPULZ_OK
        got = out[: int(nb.item())].cpu().numpy()
        ref = orc.compress(x, ws, cs, 0, window=window)
        assert np.array_equal(got, ref)
        assert np.array_equal(y.cpu().numpy(), x)
    # a direct call on the same stream after the graph launches is still right
    x = next(_inputs(n, 1))
    with torch.cuda.stream(s):
        d_in.copy_(torch.from_numpy(x))
        calls()
    s.synchronize()
    assert np.array_equal(out[: int(nb.item())].cpu().numpy(), orc.compress(x, ws, cs, 0, window=window))


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")  # nothing was captured, by design
def test_capture_without_scratch_is_refused():
    import torch
    g = lib()
    s = torch.cuda.Stream()  # never used directly: no scratch
    n = 1 << 20
    d_in = torch.zeros(n, dtype=torch.uint8, device="cuda")
    cap = g.gpulz_compress_bound(n, 4, 2048)
    out = torch.zeros(cap, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    graph = torch.cuda.CUDAGraph()
    codes = []
    with torch.cuda.graph(graph, stream=s):
        codes.append(g.gpulz_compress(d_in, n, 4, 2048, 0, out, cap, nb, s))
    assert codes == [g.GPULZ_ERR_INVALID_ARG]
