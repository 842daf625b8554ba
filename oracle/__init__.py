"""GPULZ oracle: plain sequential CPU encoder/decoder (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may use this package. It shares no code with the CUDA
library; the C source it loads is ``oracle/gpulz_oracle.c``.

The functions here only marshal numpy arrays into that C code. The method
itself (GPULZ stage documentation of FZGPUModules: chunking, exact near-window
longest match, hashed level-1 candidates over 8 sub-blocks, greedy parse,
flag bitmap + packed items, raw fallback, zero-chunk sentinel) lives in the C
file, step by step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gpulz_oracle.c")
_HDR = os.path.join(_HERE, "gpulz_oracle.h")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libgpulz_oracle.so")

ERR_INVALID_ARG = -1
ERR_CAPACITY = -2
ERR_CORRUPT = -3

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable flags only)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    fresh = os.path.exists(_LIB) and all(
        os.path.getmtime(_LIB) >= os.path.getmtime(p) for p in (_SRC, _HDR))
    if fresh and not force:
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-fPIC", "-shared",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        lib.orc_valid_geometry.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.orc_valid_geometry.restype = ctypes.c_int
        lib.orc_min_match_len.argtypes = [ctypes.c_int]
        lib.orc_min_match_len.restype = ctypes.c_int
        lib.orc_hash_bits.argtypes = [ctypes.c_int]
        lib.orc_hash_bits.restype = ctypes.c_uint32
        lib.orc_hash.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        lib.orc_hash.restype = ctypes.c_uint32
        lib.orc_compress_bound.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int]
        lib.orc_compress_bound.restype = ctypes.c_uint64
        lib.orc_near_matches.argtypes = [u32p, ctypes.c_int, u8p, u8p]
        lib.orc_near_matches.restype = None
        lib.orc_near_matches_w.argtypes = [u32p, ctypes.c_int, ctypes.c_int, u8p, u8p]
        lib.orc_near_matches_w.restype = None
        lib.orc_level1_matches.argtypes = [u32p, ctypes.c_int, u8p, u8p]
        lib.orc_level1_matches.restype = None
        lib.orc_encode_chunk.argtypes = [u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p,
                                         u32p, u32p]
        lib.orc_encode_chunk.restype = ctypes.c_uint32
        lib.orc_compress.argtypes = [u8p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, u8p, ctypes.c_uint64]
        lib.orc_compress.restype = ctypes.c_int64
        lib.orc_compress_w.argtypes = [u8p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, u8p, ctypes.c_uint64]
        lib.orc_compress_w.restype = ctypes.c_int64
        lib.orc_decompress.argtypes = [u8p, ctypes.c_uint64, u8p, ctypes.c_uint64]
        lib.orc_decompress.restype = ctypes.c_int
        lib.orc_encode_chunk_range.argtypes = [u8p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                               u8p, u32p, u32p]
        lib.orc_encode_chunk_range.restype = None
        lib.orc_encode_chunk_range_w.argtypes = [u8p, ctypes.c_uint64, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_uint64, ctypes.c_uint64, u8p, u32p,
                                                 u32p]
        lib.orc_encode_chunk_range_w.restype = None
        u64p = ctypes.POINTER(ctypes.c_uint64)
        lib.orc_decode_chunk_range.argtypes = [u8p, ctypes.c_uint64, u64p, u8p, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_uint64]
        lib.orc_decode_chunk_range.restype = ctypes.c_int
        lib.orc_split_bounds.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, u64p]
        lib.orc_split_bounds.restype = None
        lib.orc_compress_split.argtypes = [u8p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, u8p, u8p, u8p, u8p, u64p]
        lib.orc_compress_split.restype = ctypes.c_int
        lib.orc_decompress_split.argtypes = [u8p, u8p, u8p, u8p, u64p, u8p, ctypes.c_uint64]
        lib.orc_decompress_split.restype = ctypes.c_int
        _lib = lib
        return lib


def _u8(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _u32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32))


def _as_bytes(data) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(data))
    return a.view(np.uint8).reshape(-1)


def min_match_len(word_size: int) -> int:
    return _load().orc_min_match_len(word_size)


def hash_bits(elems: int) -> int:
    return _load().orc_hash_bits(elems)


def hash2(k0: int, k1: int, bits: int) -> int:
    return _load().orc_hash(k0 & 0xFFFFFFFF, k1 & 0xFFFFFFFF, bits)


def compress_bound(n_bytes: int, word_size: int, chunk_size: int) -> int:
    return _load().orc_compress_bound(n_bytes, word_size, chunk_size)


def near_matches(words, window: int = 32) -> tuple[np.ndarray, np.ndarray]:
    """Level-0 (length, offset) for every position of one chunk of words, over
    a near window of `window` elements (32 by default; up to 64)."""
    w = np.ascontiguousarray(np.asarray(words, dtype=np.uint32))
    ln = np.zeros(w.size, np.uint8)
    of = np.zeros(w.size, np.uint8)
    if window == 32:
        _load().orc_near_matches(_u32(w), w.size, _u8(ln), _u8(of))
    else:
        _load().orc_near_matches_w(_u32(w), w.size, window, _u8(ln), _u8(of))
    return ln, of


def level1_matches(words) -> tuple[np.ndarray, np.ndarray]:
    """Level-1 (length, offset): near window combined with hashed candidates."""
    w = np.ascontiguousarray(np.asarray(words, dtype=np.uint32))
    ln, of = near_matches(w)
    _load().orc_level1_matches(_u32(w), w.size, _u8(ln), _u8(of))
    return ln, of


def encode_chunk(chunk, word_size: int, chunk_size: int, match_level: int):
    """Encode one zero-padded chunk. Returns (block bytes, entry_items, entry_data)."""
    c = np.zeros(chunk_size, np.uint8)
    b = _as_bytes(chunk)
    c[:b.size] = b
    out = np.zeros(chunk_size, np.uint8)
    items = np.zeros(1, np.uint32)
    dbytes = np.zeros(1, np.uint32)
    n = _load().orc_encode_chunk(_u8(c), word_size, chunk_size, match_level, _u8(out),
                                 _u32(items), _u32(dbytes))
    return out[:n].copy(), int(items[0]), int(dbytes[0])


def compress(data, word_size: int, chunk_size: int, match_level: int,
             window: int = 32) -> np.ndarray:
    """Whole-stream encode; returns the stream as a uint8 array. `window` is
    the near window in elements (32 by default, up to 64)."""
    src = _as_bytes(data)
    cap = compress_bound(src.size, word_size, chunk_size)
    out = np.zeros(cap, np.uint8)
    n = _load().orc_compress_w(_u8(src), src.size, word_size, chunk_size, match_level, window,
                               _u8(out), cap)
    if n < 0:
        raise ValueError("oracle compress failed with code %d" % n)
    return out[:n].copy()


def decompress(stream, n_bytes: int) -> np.ndarray:
    """Whole-stream decode; raises ValueError on a corrupt stream."""
    s = _as_bytes(stream)
    out = np.zeros(max(n_bytes, 1), np.uint8)
    rc = _load().orc_decompress(_u8(s), s.size, _u8(out), n_bytes)
    if rc != 0:
        raise ValueError("oracle decompress failed with code %d" % rc)
    return out[:n_bytes]


PORTS = ("meta", "literals", "lengths", "offsets")


def split_bounds(n_bytes: int, word_size: int, chunk_size: int) -> list[int]:
    """Upper bounds on the four split-mode ports' byte lengths."""
    b = np.zeros(4, np.uint64)
    _load().orc_split_bounds(n_bytes, word_size, chunk_size,
                             b.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
    return [int(v) for v in b]


def compress_split(data, word_size: int, chunk_size: int, match_level: int) -> list[np.ndarray]:
    """Split-mode encode; returns the four ports (meta, literals, lengths,
    offsets) as uint8 arrays."""
    src = _as_bytes(data)
    bounds = split_bounds(src.size, word_size, chunk_size)
    ports = [np.zeros(max(b, 1), np.uint8) for b in bounds]
    sizes = np.zeros(4, np.uint64)
    rc = _load().orc_compress_split(_u8(src), src.size, word_size, chunk_size, match_level,
                                    *[_u8(p) for p in ports],
                                    sizes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
    if rc != 0:
        raise ValueError("oracle split compress failed with code %d" % rc)
    return [p[:int(n)].copy() for p, n in zip(ports, sizes)]


def decompress_split_status(ports, n_bytes: int):
    """Split-mode decode; returns (status, output)."""
    ps = [_as_bytes(p) for p in ports]
    bufs = [p if p.size else np.zeros(1, np.uint8) for p in ps]
    lens = np.array([p.size for p in ps], np.uint64)
    out = np.zeros(max(n_bytes, 1), np.uint8)
    rc = _load().orc_decompress_split(*[_u8(b) for b in bufs],
                                      lens.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                      _u8(out), n_bytes)
    return rc, out[:n_bytes]


def decompress_split(ports, n_bytes: int) -> np.ndarray:
    """Split-mode decode; raises ValueError on corrupt ports."""
    rc, out = decompress_split_status(ports, n_bytes)
    if rc != 0:
        raise ValueError("oracle split decompress failed with code %d" % rc)
    return out


def decompress_status(stream, n_bytes: int) -> int:
    """Decode and return the oracle's status code only (0 = ok)."""
    s = _as_bytes(stream)
    out = np.zeros(max(n_bytes, 1), np.uint8)
    return _load().orc_decompress(_u8(s), s.size, _u8(out), n_bytes)


def compress_threads(data, word_size: int, chunk_size: int, match_level: int,
                     threads: int, window: int = 32) -> np.ndarray:
    """The same oracle chunk encoder spread over host threads by chunk range.

    Chunks are independent, so concatenating the per-chunk blocks in chunk
    order gives exactly the stream ``compress`` returns. ctypes releases the
    GIL during each call, so the ranges run concurrently.
    """
    src = _as_bytes(data)
    n = src.size
    chunks = (n + chunk_size - 1) // chunk_size
    blocks = np.zeros(max(chunks, 1) * chunk_size, np.uint8)
    sizes = np.zeros(max(chunks, 1), np.uint32)
    entries = np.zeros(max(chunks, 1) * 2, np.uint32)
    lib = _load()
    threads = max(1, min(threads, max(chunks, 1)))
    bounds = [chunks * t // threads for t in range(threads + 1)]

    def run(t):
        lib.orc_encode_chunk_range_w(_u8(src), n, word_size, chunk_size, match_level, window,
                                     bounds[t], bounds[t + 1], _u8(blocks), _u32(sizes),
                                     _u32(entries))

    pool = [threading.Thread(target=run, args=(t,)) for t in range(threads)]
    for th in pool:
        th.start()
    for th in pool:
        th.join()
    body = [blocks[c * chunk_size: c * chunk_size + int(sizes[c])] for c in range(chunks)]
    total = 32 + 8 * chunks + int(sizes[:chunks].sum(dtype=np.uint64))
    header = np.zeros(32, np.uint8)
    hv = header.view(np.uint32)
    hv[0] = 0x5A4C5047
    header[4] = 1
    header[5] = 0
    header[6] = word_size
    header[7] = 0
    hv[2] = chunk_size
    hv[3] = chunks
    header.view(np.uint64)[2] = n
    header.view(np.uint64)[3] = total
    table = entries[:2 * chunks].view(np.uint8)
    return np.concatenate([header, table] + body) if chunks else header


def decompress_threads(stream, n_bytes: int, threads: int) -> np.ndarray:
    """The oracle decoder spread over host threads by chunk range.

    Block offsets come from the size table (each block's size follows from its
    entry); every range is then decoded by the same sequential replay as
    ``decompress``."""
    s = _as_bytes(stream)
    hdr = s[:32]
    chunk_size = int(hdr[8:12].view(np.uint32)[0])
    chunks = int(hdr[12:16].view(np.uint32)[0])
    ent = s[32:32 + 8 * chunks].view(np.uint32).reshape(-1, 2).astype(np.uint64)
    items, dbytes = ent[:, 0], ent[:, 1]
    raw = items == 0x80000000
    zero = (items == 0) & (dbytes == 0)
    blk = 4 * ((items + 31) // 32) + ((dbytes + 3) & ~np.uint64(3))
    blk = np.where(raw, np.uint64(chunk_size), np.where(zero, np.uint64(0), blk))
    offs = np.zeros(max(chunks, 1), np.uint64)
    if chunks:
        offs[:chunks] = 32 + 8 * chunks + np.concatenate([[0], np.cumsum(blk)[:-1]]).astype(
            np.uint64)
    out = np.zeros(max(n_bytes, 1), np.uint8)
    lib = _load()
    threads = max(1, min(threads, max(chunks, 1)))
    bounds = [chunks * t // threads for t in range(threads + 1)]
    rcs = [0] * threads
    optr = offs.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64))

    def run(t):
        rcs[t] = lib.orc_decode_chunk_range(_u8(s), s.size, optr, _u8(out), n_bytes, bounds[t],
                                            bounds[t + 1])

    pool = [threading.Thread(target=run, args=(t,)) for t in range(threads)]
    for th in pool:
        th.start()
    for th in pool:
        th.join()
    if any(rcs):
        raise ValueError("oracle decompress failed with code %d" % min(rcs))
    return out[:n_bytes]
