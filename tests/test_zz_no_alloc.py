"""gpulz_compress_noalloc: the encode entry point for callers that cannot
allocate device memory (a framework's caching allocator already holds it, a
latency-critical path cannot take cudaMalloc's implicit synchronisation, or a
plug-in host forbids allocations). Its scratch is a fixed array inside the
library and its kernel is the single-pass form of the encoder (blocks placed
by look-back over per-chunk entries, its own level-1 verification), so the
tests check, through the C ABI, that its streams equal the oracle's byte for
byte (this is integer work) on every geometry and both levels, that two calls
in a row give exactly what gpulz_compress gives (the array's leftovers from
the first call do not leak into the second), and that inputs beyond the fixed
limit are refused. The file is named to run last; it also passes when run on
its own."""
import functools

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

GEOMS = [(ws, cs) for ws in (1, 2, 4) for cs in (1024, 2048, 4096)]


def _stream_of(g, fn, d_in, n, ws, cs, lvl):
    import torch
    cap = g.gpulz_compress_bound(n, ws, cs)
    out = torch.full((max(cap, 4),), 0xAB, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert fn(d_in, n, ws, cs, lvl, out, cap, nb) == g.GPULZ_OK
    torch.cuda.synchronize()
    assert int(nb.item()) <= cap   # a wait that gave up would read as SIZE_MAX
    return out[: int(nb.item())].cpu().numpy()


@functools.lru_cache(maxsize=1)
def _plane():
    import synth
    return synth.generate(2)


def _dev(x):
    import torch
    t = torch.zeros(max(x.size, 1), dtype=torch.uint8, device="cuda")
    if x.size:
        t[: x.size] = torch.from_numpy(np.ascontiguousarray(x))
    return t


@pytest.mark.parametrize("ws,cs", GEOMS)
@pytest.mark.parametrize("lvl", [0, 1])
def test_noalloc_matches_oracle_every_geometry(orc, ws, cs, lvl):
    import lz77_family_coder_gb300 as g
    from test_gpu_parity import _edge_inputs
    g.load()
    cases = list(_edge_inputs(ws, cs, ws * 7 + cs + lvl))
    # a plane slice, and one with more chunks than the persistent grid has CTAs
    plane = _plane()
    cases.append(("plane_slice", plane[: (1 << 20) + 4099]))
    cases.append(("plane_many_chunks", plane[: min(plane.size, 4000 * cs + 17)]))
    for name, x in cases:
        ref = orc.compress_threads(x, ws, cs, lvl, threads=16)
        d = _dev(x)
        for call in range(2):                       # two calls in a row
            got = _stream_of(g, g.gpulz_compress_noalloc, d, x.size, ws, cs, lvl)
            assert np.array_equal(got, ref), (name, call)


@pytest.mark.parametrize("lvl", [0, 1])
def test_noalloc_matches_compress_twice(lvl):
    import torch
    import lz77_family_coder_gb300 as g
    import synth
    g.load()
    x = synth.generate(2)[: 7 * (1 << 20) + 13]        # ~7 MB of plane codes, ragged tail
    y = synth.generate(1)                               # a second, different input
    dx = torch.from_numpy(x).cuda()
    dy = torch.from_numpy(y).cuda()
    ref_x = _stream_of(g, g.gpulz_compress, dx, x.size, 4, 2048, lvl)
    ref_y = _stream_of(g, g.gpulz_compress, dy, y.size, 4, 2048, lvl)
    assert g.gpulz_device_status() == g.GPULZ_OK
    # two calls in a row: a large one, then a smaller one over the same array
    got_x = _stream_of(g, g.gpulz_compress_noalloc, dx, x.size, 4, 2048, lvl)
    got_y = _stream_of(g, g.gpulz_compress_noalloc, dy, y.size, 4, 2048, lvl)
    assert np.array_equal(got_x, ref_x)
    assert np.array_equal(got_y, ref_y)
    # and the stream decodes back to the input
    out = torch.from_numpy(got_y).cuda()
    dec = g.decompress(out, y.size)
    assert g.gpulz_device_status() == g.GPULZ_OK
    assert np.array_equal(dec.cpu().numpy(), y)


def test_noalloc_refuses_inputs_beyond_its_limit():
    import torch
    import lz77_family_coder_gb300 as g
    g.load()
    d = torch.zeros(16, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    too_big = 65536 * 1024 + 1                         # 65537 chunks at chunk_size 1024
    st = g.gpulz_compress_noalloc(d, too_big, 4, 1024, 0, d, 16, nb)
    assert st == g.GPULZ_ERR_INVALID_ARG
