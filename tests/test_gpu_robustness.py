"""GPU robustness through the C ABI: capacity overflow containment, corrupt or
truncated streams, size mismatch, concurrent streams, repeated calls (including
the scratch epoch wrap) and dirty output memory. Every fault here is made on the
host (a short capacity, edited stream bytes); nothing traps or hangs the GPU."""
import numpy as np
import pytest

from gpu_util import gpu_compress, lib, to_dev

pytestmark = pytest.mark.gpu

CANARY = 0x5C


def _workload(n=600000, seed=3):
    import synth
    return synth.generate(2)[:n]


def test_capacity_too_small_writes_nothing_past_capacity(orc):
    import torch
    g = lib()
    x = _workload()
    ref = orc.compress(x, 4, 2048, 0)
    for cap in (0, 16, 31, 32, 33, 1000, ref.size // 2 + 1, ref.size - 1):
        d_in = to_dev(x)
        out = torch.full((ref.size + 64,), CANARY, dtype=torch.uint8, device="cuda")
        nb = torch.zeros(1, dtype=torch.int64, device="cuda")
        st = g.gpulz_compress(d_in, x.size, 4, 2048, 0, out, cap, nb)
        assert st == g.GPULZ_OK
        assert g.gpulz_device_status() == g.GPULZ_ERR_CAPACITY
        assert int(nb.item()) == ref.size
        o = out.cpu().numpy()
        assert (o[cap:] == CANARY).all(), cap
        w = cap & ~3
        assert np.array_equal(o[:w], ref[:w]), cap
    # exact capacity succeeds
    out = torch.full((ref.size + 64,), CANARY, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert g.gpulz_compress(to_dev(x), x.size, 4, 2048, 0, out, ref.size, nb) == g.GPULZ_OK
    assert g.gpulz_device_status() == g.GPULZ_OK
    o = out.cpu().numpy()
    assert np.array_equal(o[:ref.size], ref) and (o[ref.size:] == CANARY).all()


def _decode_raw(stream: np.ndarray, n: int, in_bytes=None):
    import torch
    g = lib()
    d_s = to_dev(stream)
    out = torch.full((n + 64,), CANARY, dtype=torch.uint8, device="cuda")
    st = g.gpulz_decompress_bounded(d_s, stream.size if in_bytes is None else in_bytes, out, n)
    assert st == g.GPULZ_OK
    return g.gpulz_device_status(), out.cpu().numpy()


def test_truncated_and_bad_header(orc):
    g = lib()
    x = _workload()
    s = orc.compress(x, 4, 2048, 1)
    st, o = _decode_raw(s, x.size, in_bytes=s.size - 4)
    assert st == g.GPULZ_ERR_CORRUPT and (o == CANARY).all()
    st, o = _decode_raw(s[:20], x.size)
    assert st == g.GPULZ_ERR_CORRUPT and (o == CANARY).all()
    for byte in (0, 4, 6, 7, 8, 12):
        bad = s.copy()
        bad[byte] ^= 0x10
        st, o = _decode_raw(bad, x.size)
        assert st == g.GPULZ_ERR_CORRUPT and (o == CANARY).all(), byte
    st, o = _decode_raw(s, x.size - 1)
    assert st == g.GPULZ_ERR_SIZE_MISMATCH and (o == CANARY).all()


def test_corrupt_table_and_blocks_stay_in_bounds(orc):
    g = lib()
    x = _workload()
    s = orc.compress(x, 4, 2048, 0)
    n_chunks = s[12:16].view(np.uint32)[0]
    rng = np.random.default_rng(5)
    for trial in range(40):
        bad = s.copy()
        if trial < 20:
            c = int(rng.integers(0, n_chunks))
            off = 32 + 8 * c + int(rng.integers(0, 8))
            bad[off] ^= np.uint8(1 << int(rng.integers(0, 8)))
        else:
            body0 = 32 + 8 * int(n_chunks)
            for _ in range(8):
                k = int(rng.integers(body0, s.size))
                bad[k] ^= np.uint8(rng.integers(1, 256))
        st, o = _decode_raw(bad, x.size)
        assert st in (g.GPULZ_OK, g.GPULZ_ERR_CORRUPT), trial
        assert (o[x.size:] == CANARY).all(), trial
        if trial < 20:
            assert st == g.GPULZ_ERR_CORRUPT or np.array_equal(o[:x.size], x)


def test_concurrent_streams_match_serial(orc):
    import torch
    g = lib()
    import synth
    xs = [synth.generate(2)[k * 3000000: (k + 1) * 3000000 - 7 * k] for k in range(4)]
    refs = [orc.compress(x, 4, 2048, k % 2) for k, x in enumerate(xs)]
    streams = [torch.cuda.Stream() for _ in xs]
    ins = [to_dev(x) for x in xs]
    torch.cuda.synchronize()
    outs = []
    for k, (x, d, st) in enumerate(zip(xs, ins, streams)):
        with torch.cuda.stream(st):
            out, nb = g.compress(d[:x.size], 4, 2048, k % 2, stream=st)
            y = torch.empty(x.size, dtype=torch.uint8, device="cuda")
            assert g.gpulz_decompress(out, y, x.size, st) == g.GPULZ_OK
            outs.append((out, nb, y))
    for k, st in enumerate(streams):
        assert g.gpulz_device_status(st) == g.GPULZ_OK
        out, nb, y = outs[k]
        assert np.array_equal(out[: int(nb.item())].cpu().numpy(), refs[k])
        assert np.array_equal(y.cpu().numpy(), xs[k])


def test_repeated_calls_and_epoch_wrap(orc):
    """More calls on one stream than the 16-bit scratch epoch holds: results
    stay identical across the wrap (which clears tickets and descriptors)."""
    import torch
    g = lib()
    x = _workload(n=3 * 2048 + 100)
    ref = orc.compress(x, 4, 2048, 1)
    d = to_dev(x)
    out = torch.empty(g.gpulz_compress_bound(x.size, 4, 2048), dtype=torch.uint8, device="cuda")
    nb = torch.empty(1, dtype=torch.int64, device="cuda")
    y = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    checks = {1, 2, 299, 32767, 32768, 32769, 65535, 65536, 65537, 66000}
    for k in range(1, 66001):
        out.fill_(0xFF) if k in checks else None
        assert g.gpulz_compress(d, x.size, 4, 2048, 1, out, out.numel(), nb) == g.GPULZ_OK
        if k in checks:
            assert g.gpulz_device_status() == g.GPULZ_OK
            assert np.array_equal(out[: int(nb.item())].cpu().numpy(), ref), k
            assert g.gpulz_decompress(out, y, x.size) == g.GPULZ_OK
            assert g.gpulz_device_status() == g.GPULZ_OK
            assert np.array_equal(y.cpu().numpy(), x), k


def test_dirty_output_memory(orc):
    """Padding and every written byte are defined: garbage in the output buffer
    never leaks into the stream."""
    import torch
    g = lib()
    x = _workload()
    ref = orc.compress(x, 4, 2048, 0)
    for fill in (0x00, 0xFF, 0x5A):
        d = to_dev(x)
        out = torch.full((ref.size + 100,), fill, dtype=torch.uint8, device="cuda")
        nb = torch.empty(1, dtype=torch.int64, device="cuda")
        assert g.gpulz_compress(d, x.size, 4, 2048, 0, out, out.numel(), nb) == g.GPULZ_OK
        assert g.gpulz_device_status() == g.GPULZ_OK
        assert np.array_equal(out[: ref.size].cpu().numpy(), ref)


def test_kernel_events_hook_brackets_the_main_kernels(orc):
    """The measurement hook records the caller's events around the encode and
    decode kernels: both pairs complete with a positive elapsed time inside
    the whole call's, the results are unchanged, and clearing the hook stops
    further records."""
    import torch
    g = lib()
    x = _workload()
    ref = orc.compress(x, 4, 2048, 0)
    d_in = to_dev(x)
    cap = g.gpulz_compress_bound(x.size, 4, 2048)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    y = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record()  # creates the events
    torch.cuda.synchronize()
    ev[0].record()
    assert g.gpulz_set_kernel_events(ev[1], ev[2]) == g.GPULZ_OK
    assert g.gpulz_compress(d_in, x.size, 4, 2048, 0, out, cap, nb) == g.GPULZ_OK
    assert g.gpulz_set_kernel_events(ev[3], ev[4]) == g.GPULZ_OK
    assert g.gpulz_decompress(out, y, x.size) == g.GPULZ_OK
    assert g.gpulz_set_kernel_events(None, None) == g.GPULZ_OK
    ev[5].record()
    torch.cuda.synchronize()
    assert g.gpulz_device_status() == g.GPULZ_OK
    n = int(nb.item())
    assert np.array_equal(out[:n].cpu().numpy(), ref)
    assert np.array_equal(y.cpu().numpy(), x)
    t_enc = ev[1].elapsed_time(ev[2])
    t_dec = ev[3].elapsed_time(ev[4])
    t_all = ev[0].elapsed_time(ev[5])
    assert 0 < t_enc < t_all and 0 < t_dec < t_all
    assert t_enc + t_dec <= t_all
    # cleared: a further call leaves the events where they were
    stamp = ev[1].elapsed_time(ev[2])
    assert g.gpulz_compress(d_in, x.size, 4, 2048, 0, out, cap, nb) == g.GPULZ_OK
    torch.cuda.synchronize()
    assert ev[1].elapsed_time(ev[2]) == stamp


# ---------------------------------------------------------------------------
# bounded device waits: a look-back whose predecessor never publishes gives up
# after its limit, records the timeout and returns (the context stays usable)
# ---------------------------------------------------------------------------
def _desc(epoch, kind, value):
    return (epoch << 48) | (kind << 46) | value


def test_bounded_lookback_wait_times_out(orc):
    import time
    import torch
    g = lib()
    n, idx, ep = 100, 99, 7
    arr = np.array([_desc(ep, 2 if k == 0 else 1, k + 1) for k in range(n)], np.uint64)
    pre = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    assert g.gpulz_device_status() == g.GPULZ_OK
    # control: every predecessor published -> exact prefix, no timeout
    d = torch.from_numpy(arr.view(np.int64).copy()).cuda()
    assert g.gpulz_test_lookback(d, idx, 5, ep, 20_000_000, pre) == g.GPULZ_OK
    assert g.gpulz_device_status() == g.GPULZ_OK
    total = sum(range(1, idx + 1))
    assert int(pre.item()) == total
    after = d.cpu().numpy().view(np.uint64)
    assert np.array_equal(after[:idx], arr[:idx])
    assert int(after[idx]) == _desc(ep, 2, total + 5)
    # entry 37 carries another call's epoch: it is never published for this one
    bad = arr.copy()
    bad[37] = _desc(ep - 1, 1, 38)
    d = torch.from_numpy(bad.view(np.int64).copy()).cuda()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert g.gpulz_test_lookback(d, idx, 5, ep, 20_000_000, pre) == g.GPULZ_OK
    st = g.gpulz_device_status()
    dt = time.perf_counter() - t0
    assert st == g.GPULZ_ERR_TIMEOUT
    assert 0.02 <= dt < 5.0, dt
    after = d.cpu().numpy().view(np.uint64)
    assert np.array_equal(after[:idx], bad[:idx])      # nothing below idx was written
    assert (int(after[idx]) >> 46) == (ep << 2) | 2     # idx published (inclusive, partial)
    assert g.gpulz_device_status() == g.GPULZ_OK        # the status was read and cleared
    # the context is still usable
    x = _workload(200000)
    assert np.array_equal(gpu_compress(x, 4, 2048, 1), orc.compress(x, 4, 2048, 1))


# ---------------------------------------------------------------------------
# scratch lifetime: per-stream scratch is given back by gpulz_release_scratch
# ---------------------------------------------------------------------------
def test_release_scratch_returns_memory():
    import torch
    g = lib()
    n, cs = 512 << 20, 4096
    d_in = torch.zeros(n, dtype=torch.uint8, device="cuda")
    streams = [torch.cuda.Stream() for _ in range(8)]
    outs = [torch.empty(2 << 20, dtype=torch.uint8, device="cuda") for _ in streams]
    nbs = [torch.zeros(1, dtype=torch.int64, device="cuda") for _ in streams]
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for s, o, nb in zip(streams, outs, nbs):
        assert g.gpulz_compress(d_in, n, 4, cs, 0, o, o.numel(), nb, s) == g.GPULZ_OK
    torch.cuda.synchronize()
    held = free0 - torch.cuda.mem_get_info()[0]
    assert held >= 8 * n * 0.9, held                      # a slot area per stream
    for s, nb in zip(streams, nbs):
        assert g.gpulz_device_status(s) == g.GPULZ_OK
        assert int(nb.item()) == 32 + 8 * (n // cs)       # all-zero chunks
        assert g.gpulz_release_scratch(s) == g.GPULZ_OK
        assert g.gpulz_release_scratch(s) == g.GPULZ_OK   # nothing left: a no-op
    torch.cuda.synchronize()
    left = free0 - torch.cuda.mem_get_info()[0]
    assert left < (64 << 20), left
    # a released stream allocates afresh on its next call
    s, o, nb = streams[0], outs[0], nbs[0]
    assert g.gpulz_compress(d_in[:1 << 20], 1 << 20, 4, cs, 1, o, o.numel(), nb, s) == g.GPULZ_OK
    assert g.gpulz_device_status(s) == g.GPULZ_OK
    assert int(nb.item()) == 32 + 8 * ((1 << 20) // cs)
    assert g.gpulz_release_scratch(s) == g.GPULZ_OK
