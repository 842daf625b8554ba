"""GPU parity: the CUDA stream must be byte-identical to the oracle's, and the
CUDA decode byte-identical to the input, on every workload at full size and on
edge cases over every supported geometry and both match levels."""
import numpy as np
import pytest

import goldens
import streamcheck
from gpu_util import gpu_compress, gpu_decompress, lib, to_dev

pytestmark = pytest.mark.gpu

GEOMS = [(ws, cs) for ws in (1, 2, 4) for cs in (1024, 2048, 4096)]


def _check(orc, x, ws, cs, lvl):
    ref = orc.compress_threads(x, ws, cs, lvl, threads=16)
    got = gpu_compress(x, ws, cs, lvl)
    if not np.array_equal(got, ref):
        n = min(got.size, ref.size)
        diff = np.nonzero(got[:n] != ref[:n])[0]
        first = int(diff[0]) if diff.size else n
        raise AssertionError("stream differs: sizes %d vs %d, first diff at byte %d"
                             % (got.size, ref.size, first))
    y = gpu_decompress(got, x.size)
    assert np.array_equal(y, x)
    return got


# ---------------------------------------------------------------------------
# the seven workloads at full size
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg_id", [1, 2, 3, 4, 5, 6, 7])
def test_workload_full_size(orc, cfg_id):
    import synth
    cfg = synth.CONFIGS[cfg_id]
    x = synth.generate(cfg_id)
    s = _check(orc, x, cfg.word_size, cfg.chunk_size, cfg.match_level)
    # the oracle decodes the CUDA stream too (cross-decode)
    assert np.array_equal(orc.decompress(s, x.size), x)


def test_gpu_decodes_oracle_stream_other_level(orc):
    import synth
    x = synth.generate(2)
    for lvl in (0, 1):
        s = orc.compress_threads(x, 4, 2048, lvl, threads=16)
        assert np.array_equal(gpu_decompress(s, x.size), x)


# ---------------------------------------------------------------------------
# edge cases: every geometry x level
# ---------------------------------------------------------------------------
def _edge_inputs(ws, cs, seed):
    rng = np.random.default_rng(seed)
    E = cs // ws
    yield "empty", np.zeros(0, np.uint8)
    yield "one_byte", np.array([7], np.uint8)
    yield "not_word_multiple", rng.integers(0, 3, 5 * ws + 1).astype(np.uint8)
    yield "one_chunk", rng.integers(0, 4, cs).astype(np.uint8)
    yield "tail_one_element", rng.integers(0, 4, 3 * cs + ws).astype(np.uint8)
    yield "all_zero", np.zeros(5 * cs + 17, np.uint8)
    yield "random_raw", rng.integers(0, 256, 4 * cs + 3).astype(np.uint8)
    yield "constant", np.full(6 * cs - 1, 0xA5, np.uint8)
    for p in (1, 3, 32, 33, 100, 255, 256):
        base = rng.integers(0, 2**32, p, dtype=np.uint64).astype(np.uint32)
        w = np.tile(base, (3 * E) // p + 2)[:3 * E]
        yield "period_%d" % p, w.view(np.uint8)[:3 * cs]
    # mixed chunk kinds in one stream: zero, raw, compressible, zero, tail
    parts = [np.zeros(cs, np.uint8), rng.integers(0, 256, cs).astype(np.uint8),
             rng.integers(0, 3, cs).astype(np.uint8), np.zeros(cs, np.uint8),
             rng.integers(0, 5, cs // 3).astype(np.uint8)]
    yield "mixed_kinds", np.concatenate(parts)
    # sparse: mostly zero chunks
    sp = np.zeros(40 * cs, np.uint8)
    sp[rng.integers(0, sp.size, 30)] = rng.integers(1, 255, 30).astype(np.uint8)
    yield "sparse", sp


@pytest.mark.parametrize("ws,cs", GEOMS)
@pytest.mark.parametrize("lvl", [0, 1])
def test_edge_cases(orc, ws, cs, lvl):
    for name, x in _edge_inputs(ws, cs, ws * 31 + cs + lvl):
        try:
            s = _check(orc, x, ws, cs, lvl)
            streamcheck.check_invariants(s, x.size)
        except AssertionError as e:
            raise AssertionError("%s: %s" % (name, e))


@pytest.mark.parametrize("ws,cs", GEOMS)
@pytest.mark.parametrize("lvl", [0, 1])
def test_plane_sample_all_geometries(orc, ws, cs, lvl):
    """A 2 MiB slice of the 1800x3600 plane's codes under every geometry."""
    import synth
    x = synth.generate(2)[: (1 << 21) + 4099]
    _check(orc, x, ws, cs, lvl)


@pytest.mark.parametrize("case", goldens.load_all(), ids=lambda c: c["name"])
def test_golden_streams_on_gpu(case):
    for lvl in case["levels"]:
        for window in case["windows"]:
            s = gpu_compress(case["x"], case["ws"], case["cs"], lvl, window=window)
            assert np.array_equal(s, case["stream"]), (lvl, window)
    assert np.array_equal(gpu_decompress(case["stream"], case["x"].size), case["x"])


def test_unaligned_input_pointer(orc):
    import synth
    g = lib()
    x = synth.generate(1)[:100000]
    d = to_dev(x, pad=16)
    import torch
    buf = torch.zeros(x.size + 1, dtype=torch.uint8, device="cuda")
    buf[1:] = d[:x.size]
    out, nb = g.compress(buf[1:], 4, 2048, 1)
    assert g.gpulz_device_status() == g.GPULZ_OK
    got = out[: int(nb.item())].cpu().numpy()
    assert np.array_equal(got, orc.compress(x, 4, 2048, 1))
