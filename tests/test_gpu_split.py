"""GPU parity of split mode: the four ports (meta, literals, lengths, offsets)
byte-identical to the oracle's, the split decode byte-identical to the input
(from the oracle's ports and from the GPU's), on workloads and on edge cases
over every geometry and both levels; corrupt or short ports are reported, and
nothing is written past a port's capacity."""
import numpy as np
import pytest

from gpu_util import lib, to_dev
from test_gpu_parity import GEOMS, _edge_inputs

pytestmark = pytest.mark.gpu

PORTS = ("meta", "literals", "lengths", "offsets")


def gpu_split(x, ws, cs, lvl):
    g = lib()
    d = to_dev(x)
    ports, pb = g.compress_split(d[:x.size] if x.size else d, ws, cs, lvl)
    assert g.gpulz_device_status() == g.GPULZ_OK
    n = [int(v) for v in pb.cpu().numpy()]
    return [p[:k].cpu().numpy() for p, k in zip(ports, n)]


def gpu_unsplit(ports, n, expect=0):
    g = lib()
    import torch
    dev = [to_dev(p) if p.size else None for p in ports]
    out = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    st = g.gpulz_decompress_split(*dev, [p.size for p in ports], out, n)
    assert st == g.GPULZ_OK
    dst = g.gpulz_device_status()
    assert dst == expect, g.gpulz_status_string(dst)
    return out[:n].cpu().numpy()


def _check(orc, x, ws, cs, lvl):
    ref = orc.compress_split(x, ws, cs, lvl)
    got = gpu_split(x, ws, cs, lvl)
    for name, r, o in zip(PORTS, ref, got):
        if not np.array_equal(o, r):
            n = min(o.size, r.size)
            diff = np.nonzero(o[:n] != r[:n])[0]
            raise AssertionError("%s port differs: sizes %d vs %d, first diff %s"
                                 % (name, o.size, r.size, diff[0] if diff.size else n))
    assert np.array_equal(gpu_unsplit(got, x.size), x)
    return got


@pytest.mark.parametrize("cfg_id", [1, 2, 3, 5, 6, 7])
def test_split_workloads(orc, cfg_id):
    import synth
    cfg = synth.CONFIGS[cfg_id]
    x = synth.generate(cfg_id)
    if x.size > (48 << 20):
        x = x[: 48 << 20]  # the oracle's split encode is single-threaded
    _check(orc, x, cfg.word_size, cfg.chunk_size, cfg.match_level)


def test_split_volume_slice(orc):
    import synth
    x = synth.generate(4)[: 64 << 20]
    _check(orc, x, 4, 4096, 1)


@pytest.mark.parametrize("ws,cs", GEOMS)
@pytest.mark.parametrize("lvl", [0, 1])
def test_split_edge_cases(orc, ws, cs, lvl):
    for name, x in _edge_inputs(ws, cs, ws * 17 + cs + lvl):
        try:
            _check(orc, x, ws, cs, lvl)
        except AssertionError as e:
            raise AssertionError("%s: %s" % (name, e))


def test_split_decode_of_oracle_ports_both_levels(orc):
    import synth
    x = synth.generate(2)[: 3 << 20]
    for lvl in (0, 1):
        ports = orc.compress_split(x, 4, 2048, lvl)
        assert np.array_equal(gpu_unsplit(ports, x.size), x)


def test_split_corrupt_or_short_ports_reported(orc):
    import synth
    g = lib()
    x = synth.generate(1)
    ports = orc.compress_split(x, 4, 2048, 1)
    # each port one byte short: the header totals no longer fit
    for k in range(4):
        if ports[k].size == 0:
            continue
        cut = [p.copy() for p in ports]
        cut[k] = cut[k][:-1]
        gpu_unsplit(cut, x.size, expect=g.GPULZ_ERR_CORRUPT)
    # a chunk entry that claims more matches than items
    bad = [p.copy() for p in ports]
    bad[0][48 + 4:48 + 8] = np.frombuffer(np.uint32(100000).tobytes(), np.uint8)
    gpu_unsplit(bad, x.size, expect=g.GPULZ_ERR_CORRUPT)
    # wrong original size
    gpu_unsplit(ports, x.size + 1, expect=g.GPULZ_ERR_SIZE_MISMATCH)


def test_split_capacity_contained(orc):
    import torch
    import synth
    g = lib()
    x = synth.generate(1)
    ref = orc.compress_split(x, 4, 2048, 0)
    st, bounds = g.gpulz_split_bounds(x.size, 4, 2048)
    assert st == g.GPULZ_OK
    for k in range(4):
        cap = [b for b in bounds]
        cap[k] = max(ref[k].size // 2, 1)
        bufs = [torch.full((b + 64,), 0x5C, dtype=torch.uint8, device="cuda") for b in bounds]
        pb = torch.zeros(4, dtype=torch.int64, device="cuda")
        assert g.gpulz_compress_split(to_dev(x), x.size, 4, 2048, 0, *bufs, cap, pb) == g.GPULZ_OK
        assert g.gpulz_device_status() == g.GPULZ_ERR_CAPACITY
        assert [int(v) for v in pb.cpu().numpy()] == [r.size for r in ref]
        o = bufs[k].cpu().numpy()
        assert (o[cap[k]:] == 0x5C).all(), k
