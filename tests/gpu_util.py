"""Helpers for the GPU tests: every call goes through the C ABI (libgpulz.so)."""
from __future__ import annotations

import numpy as np


def lib():
    import lz77_family_coder_gb300 as g
    g.load()
    return g


def to_dev(x: np.ndarray, pad: int = 0):
    import torch
    t = torch.zeros(x.size + pad, dtype=torch.uint8, device="cuda")
    if x.size:
        t[:x.size] = torch.from_numpy(np.ascontiguousarray(x))
    return t


def gpu_compress(x: np.ndarray, ws: int, cs: int, lvl: int, stream=None,
                 window: int = 32) -> np.ndarray:
    """Compress host bytes on the GPU; returns the stream bytes (host)."""
    import torch
    g = lib()
    d_in = to_dev(x)
    out, nbytes = g.compress(d_in[:x.size] if x.size else d_in, ws, cs, lvl, stream=stream,
                             window=window)
    st = g.gpulz_device_status(stream)
    assert st == g.GPULZ_OK, g.gpulz_status_string(st)
    n = int(nbytes.item())
    return out[:n].cpu().numpy()


def gpu_decompress(stream_bytes: np.ndarray, n: int, stream=None, expect=0) -> np.ndarray:
    g = lib()
    d_s = to_dev(stream_bytes)
    y = g.decompress(d_s, n, stream=stream, in_bytes=stream_bytes.size)
    st = g.gpulz_device_status(stream)
    assert st == expect, g.gpulz_status_string(st)
    return y.cpu().numpy()
