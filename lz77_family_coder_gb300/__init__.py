"""GB300-native GPULZ chunked LZSS coder: thin Python binding of libgpulz.so.

The functions named ``gpulz_*`` mirror the C ABI in ``include/gpulz.h`` one to
one and only marshal arguments (torch tensors or raw device pointers, CUDA
stream handles). Every step of encode and decode runs in the library's CUDA
kernels; there is no fallback: if the library is missing, importing the
binding's functions raises.

``compress`` / ``decompress`` are conveniences that allocate the output with
torch (device memory is torch's job here) and call the same entry points.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "GPULZ_OK", "GPULZ_ERR_INVALID_ARG", "GPULZ_ERR_CAPACITY", "GPULZ_ERR_CORRUPT",
    "GPULZ_ERR_TIMEOUT", "GPULZ_ERR_CUDA", "GPULZ_ERR_SIZE_MISMATCH", "GpulzError",
    "library_path", "load", "build", "gpulz_compress", "gpulz_compress_window",
    "gpulz_compress_noalloc", "gpulz_decompress",
    "gpulz_decompress_bounded", "gpulz_compress_bound", "gpulz_stream_info",
    "gpulz_device_status", "gpulz_set_kernel_events", "gpulz_status_string", "compress",
    "decompress", "gpulz_split_bounds", "gpulz_compress_split", "gpulz_decompress_split",
    "compress_split", "decompress_split", "gpulz_release_scratch", "gpulz_test_lookback",
]

GPULZ_OK = 0
GPULZ_ERR_INVALID_ARG = 1
GPULZ_ERR_CAPACITY = 2
GPULZ_ERR_CORRUPT = 3
GPULZ_ERR_TIMEOUT = 4
GPULZ_ERR_CUDA = 5
GPULZ_ERR_SIZE_MISMATCH = 6

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libgpulz.so")
_lib = None


class GpulzError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what or "gpulz", _status_name(status), status))


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False, verbose: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force, verbose=verbose)


def load():
    """Load libgpulz.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("libgpulz.so is missing (%s); build it with "
                           "lz77_family_coder_gb300.build()" % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.gpulz_compress.argtypes = [vp, sz, i32, i32, i32, vp, sz, vp, vp]
    lib.gpulz_compress.restype = i32
    lib.gpulz_compress_window.argtypes = [vp, sz, i32, i32, i32, i32, vp, sz, vp, vp]
    lib.gpulz_compress_window.restype = i32
    lib.gpulz_compress_noalloc.argtypes = [vp, sz, i32, i32, i32, vp, sz, vp, vp]
    lib.gpulz_compress_noalloc.restype = i32
    lib.gpulz_decompress.argtypes = [vp, vp, sz, vp]
    lib.gpulz_decompress.restype = i32
    lib.gpulz_decompress_bounded.argtypes = [vp, sz, vp, sz, vp]
    lib.gpulz_decompress_bounded.restype = i32
    lib.gpulz_compress_bound.argtypes = [sz, i32, i32]
    lib.gpulz_compress_bound.restype = sz
    lib.gpulz_stream_info.argtypes = [vp, sz, ctypes.POINTER(sz), ctypes.POINTER(sz),
                                      ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.gpulz_stream_info.restype = i32
    lib.gpulz_device_status.argtypes = [vp]
    lib.gpulz_device_status.restype = i32
    szp = ctypes.POINTER(sz)
    lib.gpulz_split_bounds.argtypes = [sz, i32, i32, szp]
    lib.gpulz_split_bounds.restype = i32
    lib.gpulz_compress_split.argtypes = [vp, sz, i32, i32, i32, vp, vp, vp, vp, szp, vp, vp]
    lib.gpulz_compress_split.restype = i32
    lib.gpulz_decompress_split.argtypes = [vp, vp, vp, vp, szp, vp, sz, vp]
    lib.gpulz_decompress_split.restype = i32
    lib.gpulz_set_kernel_events.argtypes = [vp, vp]
    lib.gpulz_set_kernel_events.restype = i32
    lib.gpulz_status_string.argtypes = [i32]
    lib.gpulz_status_string.restype = ctypes.c_char_p
    lib.gpulz_release_scratch.argtypes = [vp]
    lib.gpulz_release_scratch.restype = i32
    lib.gpulz_test_lookback.argtypes = [vp, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint32,
                                        ctypes.c_uint64, vp, vp]
    lib.gpulz_test_lookback.restype = i32
    _lib = lib
    return lib


def _status_name(status: int) -> str:
    try:
        return load().gpulz_status_string(status).decode()
    except Exception:  # noqa: BLE001 - message only
        return "status"


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ---- the C ABI, one to one ----
def gpulz_compress(d_in, n_bytes, word_size, chunk_size, match_level, d_out, capacity,
                   d_out_bytes, stream=None) -> int:
    return load().gpulz_compress(_ptr(d_in), n_bytes, word_size, chunk_size, match_level,
                                 _ptr(d_out), capacity, _ptr(d_out_bytes), _stream(stream))


def gpulz_compress_window(d_in, n_bytes, word_size, chunk_size, match_level, window, d_out,
                          capacity, d_out_bytes, stream=None) -> int:
    return load().gpulz_compress_window(_ptr(d_in), n_bytes, word_size, chunk_size, match_level,
                                        window, _ptr(d_out), capacity, _ptr(d_out_bytes),
                                        _stream(stream))


def gpulz_compress_noalloc(d_in, n_bytes, word_size, chunk_size, match_level, d_out, capacity,
                           d_out_bytes, stream=None) -> int:
    """gpulz_compress for callers that cannot allocate (fixed in-library scratch)."""
    return load().gpulz_compress_noalloc(_ptr(d_in), n_bytes, word_size, chunk_size, match_level,
                                         _ptr(d_out), capacity, _ptr(d_out_bytes),
                                         _stream(stream))


def gpulz_decompress(d_in, d_out, n_bytes, stream=None) -> int:
    return load().gpulz_decompress(_ptr(d_in), _ptr(d_out), n_bytes, _stream(stream))


def gpulz_decompress_bounded(d_in, in_bytes, d_out, n_bytes, stream=None) -> int:
    return load().gpulz_decompress_bounded(_ptr(d_in), in_bytes, _ptr(d_out), n_bytes,
                                           _stream(stream))


def gpulz_compress_bound(n_bytes, word_size, chunk_size) -> int:
    return load().gpulz_compress_bound(n_bytes, word_size, chunk_size)


def gpulz_stream_info(h_header: bytes):
    """Returns (status, orig_bytes, stream_bytes, word_size, chunk_size)."""
    buf = ctypes.create_string_buffer(bytes(h_header), len(h_header))
    o, s = ctypes.c_size_t(), ctypes.c_size_t()
    w, c = ctypes.c_int(), ctypes.c_int()
    st = load().gpulz_stream_info(ctypes.cast(buf, ctypes.c_void_p), len(h_header),
                                  ctypes.byref(o), ctypes.byref(s), ctypes.byref(w),
                                  ctypes.byref(c))
    return st, o.value, s.value, w.value, c.value


def gpulz_device_status(stream=None) -> int:
    return load().gpulz_device_status(_stream(stream))


def gpulz_split_bounds(n_bytes, word_size, chunk_size):
    """Returns (status, [meta, literals, lengths, offsets] byte bounds)."""
    b = (ctypes.c_size_t * 4)()
    st = load().gpulz_split_bounds(n_bytes, word_size, chunk_size, b)
    return st, [int(v) for v in b]


def gpulz_compress_split(d_in, n_bytes, word_size, chunk_size, match_level, d_meta, d_literals,
                         d_lengths, d_offsets, capacity, d_port_bytes, stream=None) -> int:
    cap = (ctypes.c_size_t * 4)(*[int(v) for v in capacity])
    return load().gpulz_compress_split(_ptr(d_in), n_bytes, word_size, chunk_size, match_level,
                                       _ptr(d_meta), _ptr(d_literals), _ptr(d_lengths),
                                       _ptr(d_offsets), cap, _ptr(d_port_bytes), _stream(stream))


def gpulz_decompress_split(d_meta, d_literals, d_lengths, d_offsets, port_bytes, d_out, n_bytes,
                           stream=None) -> int:
    pb = (ctypes.c_size_t * 4)(*[int(v) for v in port_bytes])
    return load().gpulz_decompress_split(_ptr(d_meta), _ptr(d_literals), _ptr(d_lengths),
                                         _ptr(d_offsets), pb, _ptr(d_out), n_bytes,
                                         _stream(stream))


def gpulz_set_kernel_events(start, stop) -> int:
    """Measurement hook: bracket the encode/decode kernel of the following calls
    from this thread with two CUDA events (torch.cuda.Event, raw handles or
    None to clear)."""
    def handle(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    return load().gpulz_set_kernel_events(handle(start), handle(stop))


def gpulz_status_string(status: int) -> str:
    return load().gpulz_status_string(status).decode()


def gpulz_release_scratch(stream=None) -> int:
    return load().gpulz_release_scratch(_stream(stream))


def gpulz_test_lookback(d_desc, idx, value, epoch, limit_ns, d_prefix, stream=None) -> int:
    """Test hook (include/gpulz_testing.h): the library's bounded look-back on a
    caller-made descriptor array."""
    return load().gpulz_test_lookback(_ptr(d_desc), idx, value, epoch, limit_ns, _ptr(d_prefix),
                                      _stream(stream))


# ---- conveniences (torch allocates, the library computes) ----
def compress(x, word_size: int, chunk_size: int, match_level: int, stream=None, out=None,
             out_bytes=None, window: int = 32):
    """Encode a contiguous CUDA tensor's bytes. Returns (out, out_bytes) tensors:
    ``out`` has compress-bound capacity; ``out_bytes`` (int64, 1 element) holds
    the stream length on the device (no host synchronisation). ``window`` is
    the exact near window in elements (32..64; above 32, level 0 only)."""
    import torch
    n = x.numel() * x.element_size()
    cap = gpulz_compress_bound(n, word_size, chunk_size)
    if cap == 0:
        raise GpulzError(GPULZ_ERR_INVALID_ARG, "compress")
    if out is None:
        out = torch.empty(cap, dtype=torch.uint8, device=x.device)
    if out_bytes is None:
        out_bytes = torch.empty(1, dtype=torch.int64, device=x.device)
    if window == 32:
        st = gpulz_compress(x if n else None, n, word_size, chunk_size, match_level, out,
                            out.numel(), out_bytes, stream)
    else:
        st = gpulz_compress_window(x if n else None, n, word_size, chunk_size, match_level,
                                   window, out, out.numel(), out_bytes, stream)
    if st != GPULZ_OK:
        raise GpulzError(st, "gpulz_compress")
    return out, out_bytes


def compress_split(x, word_size: int, chunk_size: int, match_level: int, stream=None):
    """Split-mode encode of a contiguous CUDA tensor's bytes. Returns
    ([meta, literals, lengths, offsets] tensors at their bounds, port_bytes)
    where port_bytes (int64, 4 elements, on the device) holds the lengths."""
    import torch
    n = x.numel() * x.element_size()
    st, bounds = gpulz_split_bounds(n, word_size, chunk_size)
    if st != GPULZ_OK:
        raise GpulzError(st, "gpulz_split_bounds")
    ports = [torch.empty(max(b, 4), dtype=torch.uint8, device=x.device) for b in bounds]
    port_bytes = torch.empty(4, dtype=torch.int64, device=x.device)
    st = gpulz_compress_split(x if n else None, n, word_size, chunk_size, match_level, *ports,
                              [p.numel() for p in ports], port_bytes, stream)
    if st != GPULZ_OK:
        raise GpulzError(st, "gpulz_compress_split")
    return ports, port_bytes


def decompress_split(ports, port_bytes, n_bytes: int, stream=None, out=None):
    """Split-mode decode of four CUDA tensors (meta, literals, lengths,
    offsets) with port_bytes[k] valid bytes each (host ints)."""
    import torch
    if out is None:
        out = torch.empty(max(n_bytes, 1), dtype=torch.uint8, device=ports[0].device)
    st = gpulz_decompress_split(*[p if p is not None and p.numel() else None for p in ports],
                                port_bytes, out, n_bytes, stream)
    if st != GPULZ_OK:
        raise GpulzError(st, "gpulz_decompress_split")
    return out[:n_bytes]


def decompress(stream_buf, n_bytes: int, stream=None, out=None, in_bytes: int | None = None):
    """Decode a GPULZ stream held in a CUDA tensor into n_bytes (uint8 tensor)."""
    import torch
    if out is None:
        out = torch.empty(max(n_bytes, 1), dtype=torch.uint8, device=stream_buf.device)
    if in_bytes is None:
        in_bytes = stream_buf.numel() * stream_buf.element_size()
    st = gpulz_decompress_bounded(stream_buf, in_bytes, out, n_bytes, stream)
    if st != GPULZ_OK:
        raise GpulzError(st, "gpulz_decompress")
    return out[:n_bytes]
