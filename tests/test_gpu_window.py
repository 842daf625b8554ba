"""GPU parity of the wider near window (the window-width study of the GPULZ
stage page's match-search section): for windows of 33, 48 and 64 elements the
CUDA stream is byte-identical to the oracle's with the same window, on edge
cases over every geometry (periods only a wide window sees among them) and on
the plane workload at full size; every stream decodes back to its input."""
import numpy as np
import pytest

from gpu_util import lib, to_dev
from test_gpu_parity import GEOMS, _edge_inputs

pytestmark = pytest.mark.gpu

WINDOWS = (33, 48, 64)


def gpu_compress_window(x, ws, cs, window):
    g = lib()
    d = to_dev(x)
    out, nb = g.compress(d[:x.size] if x.size else d, ws, cs, 0, window=window)
    st = g.gpulz_device_status()
    assert st == g.GPULZ_OK, g.gpulz_status_string(st)
    return out[: int(nb.item())].cpu().numpy()


def gpu_decompress(s, n):
    g = lib()
    y = g.decompress(to_dev(s), n)
    assert g.gpulz_device_status() == g.GPULZ_OK
    return y.cpu().numpy()


def _check(orc, x, ws, cs, window, ref=None):
    if ref is None:
        ref = orc.compress(x, ws, cs, 0, window=window)
    got = gpu_compress_window(x, ws, cs, window)
    if not np.array_equal(got, ref):
        n = min(got.size, ref.size)
        diff = np.nonzero(got[:n] != ref[:n])[0]
        raise AssertionError("window %d stream differs: sizes %d vs %d, first diff at byte %d"
                             % (window, got.size, ref.size, int(diff[0]) if diff.size else n))
    assert np.array_equal(gpu_decompress(got, x.size), x)


def _wide_periods(ws, cs, seed):
    """Periods only a window wider than 32 sees, with and without breaks."""
    rng = np.random.default_rng(seed)
    E = cs // ws
    for p in (33, 40, 47, 48, 49, 63, 64, 65):
        base = rng.integers(0, 2**32, p, dtype=np.uint64).astype(np.uint32)
        w = np.tile(base, (3 * E) // p + 2)[:3 * E]
        yield "period_%d" % p, w.view(np.uint8)[:3 * cs].copy()
        b = w.view(np.uint8)[:3 * cs].copy()
        b[rng.integers(0, b.size, 12)] ^= 0x5A
        yield "period_%d_broken" % p, b


@pytest.mark.parametrize("ws,cs", GEOMS)
@pytest.mark.parametrize("window", WINDOWS)
def test_window_edge_cases(orc, ws, cs, window):
    inputs = list(_edge_inputs(ws, cs, ws * 131 + cs + window))
    inputs += list(_wide_periods(ws, cs, ws * 17 + cs + window))
    for name, x in inputs:
        try:
            _check(orc, x, ws, cs, window)
        except AssertionError as e:
            raise AssertionError("%s: %s" % (name, e))


@pytest.mark.parametrize("window", [48, 64])
def test_window_plane_full_size(orc, window):
    import synth
    cfg = synth.CONFIGS[2]
    x = synth.generate(2)
    ref = orc.compress_threads(x, cfg.word_size, cfg.chunk_size, 0, threads=16, window=window)
    _check(orc, x, cfg.word_size, cfg.chunk_size, window, ref=ref)


def test_window_32_is_the_default_stream(orc):
    import synth
    x = synth.generate(2)[: 3 << 20]
    assert np.array_equal(gpu_compress_window(x, 4, 2048, 32),
                          orc.compress(x, 4, 2048, 0))


def test_window_sparse_workload(orc):
    import synth
    x = synth.generate(7)[: 16 << 20]
    _check(orc, x, 2, 2048, 64)
