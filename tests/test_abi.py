"""CPU-only checks of the C ABI library: it loads, exports every entry point that
include/gpulz.h declares, and its host-only functions and argument checks work
without a GPU (no compute call is made here)."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    import lz77_family_coder_gb300 as g
    g.build()
    g.load()
    return g


def declared_functions():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(gpulz_\w+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(g):
    names = declared_functions()
    assert {"gpulz_compress", "gpulz_decompress", "gpulz_release_scratch",
            "gpulz_test_lookback"} <= set(names)
    lib = g.load()
    for n in names:
        assert hasattr(lib, n), n


def test_compress_bound(g):
    for ws in (1, 2, 4):
        for cs in (1024, 2048, 4096):
            for n in (0, 1, cs, cs + 1, 25920000):
                chunks = -(-n // cs)
                assert g.gpulz_compress_bound(n, ws, cs) == 32 + chunks * (8 + cs)
    assert g.gpulz_compress_bound(100, 3, 2048) == 0
    assert g.gpulz_compress_bound(100, 4, 1000) == 0


def test_stream_info_parses_oracle_header(g, orc):
    x = (np.arange(50000) % 7).astype(np.uint8)
    s = orc.compress(x, 2, 1024, 1)
    st, orig, total, ws, cs = g.gpulz_stream_info(bytes(s[:32]))
    assert (st, orig, total, ws, cs) == (0, x.size, s.size, 2, 1024)
    bad = bytearray(s[:32])
    bad[0] ^= 0xFF
    assert g.gpulz_stream_info(bytes(bad))[0] == g.GPULZ_ERR_CORRUPT
    assert g.gpulz_stream_info(bytes(s[:16]))[0] == g.GPULZ_ERR_INVALID_ARG


def test_invalid_arguments_rejected_before_any_launch(g):
    P = 1 << 20  # a fake, aligned address: never dereferenced on these paths
    assert g.gpulz_compress(P, 100, 3, 2048, 0, P, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_compress(P, 100, 4, 3000, 0, P, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_compress(P, 100, 4, 2048, 2, P, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_compress(0, 100, 4, 2048, 0, P, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_compress(P, 100, 4, 2048, 0, 0, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_compress(P, 100, 4, 2048, 0, P + 2, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_compress(P, 100, 4, 2048, 0, P, 1000, P + 4, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_decompress(0, P, 100, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_decompress(P + 1, P, 100, 0) == g.GPULZ_ERR_INVALID_ARG
    # near window: 32..64, and above 32 only at level 0
    for window, lvl in ((31, 0), (65, 0), (0, 0), (48, 1), (64, 1)):
        assert (g.gpulz_compress_window(P, 100, 4, 2048, lvl, window, P, 1000, P, 0)
                == g.GPULZ_ERR_INVALID_ARG), (window, lvl)
    assert g.gpulz_compress_window(P, 100, 3, 2048, 0, 48, P, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG


def test_status_strings(g):
    for code in range(7):
        assert g.gpulz_status_string(code)


def test_kernel_events_hook_arguments(g):
    """Both events or neither: a half-set hook is refused, clearing is fine."""
    assert g.gpulz_set_kernel_events(1 << 20, None) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_set_kernel_events(None, 1 << 20) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_set_kernel_events(None, None) == g.GPULZ_OK


def test_release_and_test_hook_arguments(g):
    """Releasing a stream that holds no scratch is a no-op; the look-back test
    hook refuses bad arguments before touching the GPU."""
    P = 1 << 20
    assert g.gpulz_release_scratch(0) == g.GPULZ_OK
    assert g.gpulz_test_lookback(0, 3, 1, 5, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_test_lookback(P, 3, 1, 5, 1000, 0, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_test_lookback(P, 3, 1, 0, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_test_lookback(P, 3, 1, 65536, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert g.gpulz_test_lookback(P + 4, 3, 1, 5, 1000, P, 0) == g.GPULZ_ERR_INVALID_ARG
    assert (g.gpulz_test_lookback(P, 3, 1, 5, 200 * 1000 * 1000 + 1, P, 0)
            == g.GPULZ_ERR_INVALID_ARG)
