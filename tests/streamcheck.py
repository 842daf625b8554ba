"""Independent Python reader of the GPULZ stream (format v1), for checking invariants.

Written from the format definition, not from the oracle or the CUDA code:

* header, 32 bytes, little-endian: u32 magic 0x5A4C5047 ("GPLZ"), u16 version
  1, u8 word_size, u8 reserved 0, u32 chunk_size, u32 n_chunks, u64
  orig_bytes, u64 stream_bytes;
* size table: n_chunks entries {u32 n_items | RAW<<31, u32 data_bytes};
  zero chunk = {0, 0}; raw chunk = {RAW, chunk_size};
* blocks in chunk order: normal = flag words u32[ceil(n_items/32)] (bit j of
  word j/32, LSB first, 1 = match) then the packed items (literal = word_size
  bytes, match = u8 length, u8 offset), zero padded to a multiple of 4;
  raw = chunk_size bytes of the zero-padded chunk; zero chunk = nothing.
"""
from __future__ import annotations

import struct

import numpy as np

MAGIC = 0x5A4C5047
RAW = 0x80000000


def min_match_len(ws: int) -> int:
    # smallest length whose literal bytes exceed the 2-byte token
    return {1: 3, 2: 2, 4: 1}[ws]


def parse(stream) -> dict:
    s = bytes(np.asarray(stream, dtype=np.uint8))
    magic, ver, ws, rsv, cs, nch, orig, total = struct.unpack_from("<IHBBIIQQ", s, 0)
    assert magic == MAGIC and ver == 1 and rsv == 0
    assert total == len(s), (total, len(s))
    pos = 32 + 8 * nch
    chunks = []
    for c in range(nch):
        items, dbytes = struct.unpack_from("<II", s, 32 + 8 * c)
        if items == 0 and dbytes == 0:
            chunks.append(dict(kind="zero", items=[], block=b""))
            continue
        if items == RAW:
            assert dbytes == cs
            chunks.append(dict(kind="raw", block=s[pos:pos + cs]))
            pos += cs
            continue
        assert items & RAW == 0 and items >= 1
        fwords = (items + 31) // 32
        flags = struct.unpack_from("<%dI" % fwords, s, pos)
        data = s[pos + 4 * fwords: pos + 4 * fwords + dbytes]
        pad = s[pos + 4 * fwords + dbytes: pos + 4 * fwords + ((dbytes + 3) & ~3)]
        toks = []
        b = 0
        for j in range(items):
            if (flags[j // 32] >> (j % 32)) & 1:
                toks.append(("M", data[b], data[b + 1]))
                b += 2
            else:
                toks.append(("L", data[b:b + ws]))
                b += ws
        blk = 4 * fwords + ((dbytes + 3) & ~3)
        chunks.append(dict(kind="lz", items=toks, flags=flags, dbytes=dbytes, data_used=b,
                           pad=pad, block=s[pos:pos + blk], fwords=fwords, n_items=items))
        pos += blk
    return dict(ws=ws, cs=cs, n_chunks=nch, orig=orig, total=total, end=pos, chunks=chunks)


def check_invariants(stream, n_bytes: int | None = None) -> dict:
    """Assert every structural invariant of a stream; return the parsed form."""
    p = parse(stream)
    ws, cs = p["ws"], p["cs"]
    E = cs // ws
    lmin = min_match_len(ws)
    if n_bytes is not None:
        assert p["orig"] == n_bytes
    assert p["n_chunks"] == (p["orig"] + cs - 1) // cs
    assert p["end"] == p["total"]
    for ch in p["chunks"]:
        if ch["kind"] != "lz":
            continue
        q = 0
        nm = nl = 0
        for t in ch["items"]:
            if t[0] == "M":
                ln, off = t[1], t[2]
                assert 1 <= ln <= 255 and ln >= lmin
                assert 1 <= off <= min(255, q)
                q += ln
                nm += 1
            else:
                q += 1
                nl += 1
        assert q == E, (q, E)
        assert ch["dbytes"] == ws * nl + 2 * nm == ch["data_used"]
        # match flags beyond the last item are zero; popcount == number of matches
        pop = sum(bin(f).count("1") for f in ch["flags"])
        assert pop == nm
        assert all(v == 0 for v in ch["pad"])
        assert len(ch["block"]) < cs
    return p


def replay(p: dict) -> np.ndarray:
    """Decode a parsed stream by sequential replay (independent of the oracle)."""
    ws, cs = p["ws"], p["cs"]
    out = bytearray()
    for ch in p["chunks"]:
        if ch["kind"] == "zero":
            buf = bytearray(cs)
        elif ch["kind"] == "raw":
            buf = bytearray(ch["block"])
        else:
            buf = bytearray()
            for t in ch["items"]:
                if t[0] == "L":
                    buf += t[1]
                else:
                    ln, off = t[1], t[2]
                    for _ in range(ln):
                        start = len(buf) - off * ws
                        buf += buf[start:start + ws]
        out += buf
    return np.frombuffer(bytes(out[:p["orig"]]), np.uint8)
