"""Pins of the oracle's split mode (four ports: meta, literals, lengths,
offsets) against the single-stream form, which the other oracle tests pin.
Split mode carries the same items; re-interleaving its ports by the flag
bitmaps, written out here from the two formats' definitions, must give the
single stream byte for byte."""
import struct

import numpy as np
import pytest

RAW = 0x80000000


def v1_from_split(ports):
    """The single stream, rebuilt from the four ports."""
    meta, lits, lens, offs = (bytes(p) for p in ports)
    magic, ver, ws, res, cs, C, orig, mbytes, nlit, nmat = struct.unpack_from("<IHBBIIQQQQ", meta, 0)
    assert (magic, ver, res) == (0x5A4C5047, 2, 0)
    flag_at = 48 + 8 * C
    li = mi = 0
    entries, blocks = [], []
    for c in range(C):
        items, m = struct.unpack_from("<II", meta, 48 + 8 * c)
        if items == 0 and m == 0:
            entries.append((0, 0))
            blocks.append(b"")
        elif items == RAW:
            assert m == 0
            entries.append((RAW, cs))
            blocks.append(lits[li:li + cs])
            li += cs
        else:
            fw = (items + 31) // 32
            flags = meta[flag_at:flag_at + 4 * fw]
            flag_at += 4 * fw
            words = struct.unpack("<%dI" % fw, flags)
            data = bytearray()
            seen = 0
            for j in range(items):
                if (words[j // 32] >> (j % 32)) & 1:
                    data += bytes([lens[mi], offs[mi]])
                    mi += 1
                    seen += 1
                else:
                    data += lits[li:li + ws]
                    li += ws
            assert seen == m
            entries.append((items, len(data)))
            blocks.append(flags + bytes(data) + b"\0" * (-len(data) % 4))
    assert (flag_at, li, mi) == (mbytes, nlit, nmat)
    assert (len(meta), len(lits), len(lens), len(offs)) == (mbytes, nlit, nmat, nmat)
    body = b"".join(blocks)
    total = 32 + 8 * C + len(body)
    head = struct.pack("<IHBBIIQQ", 0x5A4C5047, 1, ws, 0, cs, C, orig, total)
    table = b"".join(struct.pack("<II", *e) for e in entries)
    return np.frombuffer(head + table + body, np.uint8)


_CACHE = []


def _inputs():
    if not _CACHE:
        _CACHE.extend(_make_inputs())
    return _CACHE


def _make_inputs():
    import synth
    rng = np.random.default_rng(31)
    tiny = synth.generate(1)  # 256x256 Lorenzo codes, u32
    yield "plane", tiny[:40000]
    yield "bytes", (tiny.view(np.uint32)[:24000] & 0xFF).astype(np.uint8)
    yield "random", rng.integers(0, 256, 9000, dtype=np.uint8)        # raw chunks
    z = np.zeros(12000, np.uint8)
    z[5000:5100] = 7
    yield "mostly_zero", z                                            # zero chunks
    yield "short", rng.integers(0, 4, 777, dtype=np.uint8)            # ragged tail
    yield "empty", np.zeros(0, np.uint8)


@pytest.mark.parametrize("ws", [1, 2, 4])
@pytest.mark.parametrize("cs", [1024, 2048, 4096])
@pytest.mark.parametrize("lvl", [0, 1])
def test_split_ports_reinterleave_to_the_single_stream(orc, ws, cs, lvl):
    for name, x in _inputs():
        ports = orc.compress_split(x, ws, cs, lvl)
        assert np.array_equal(v1_from_split(ports), orc.compress(x, ws, cs, lvl)), name


def test_split_round_trip_and_bounds(orc):
    for name, x in _inputs():
        for ws, cs, lvl in ((4, 2048, 0), (1, 4096, 1), (2, 1024, 1)):
            ports = orc.compress_split(x, ws, cs, lvl)
            bounds = orc.split_bounds(x.size, ws, cs)
            assert all(p.size <= b for p, b in zip(ports, bounds)), name
            assert np.array_equal(orc.decompress_split(ports, x.size), x), name


def test_split_literals_keep_the_word_alphabet(orc):
    """Literal words appear in the literals port exactly as in the input: for
    an input with no repeats at all every chunk is raw and the port is the
    input itself (zero padded to whole chunks)."""
    rng = np.random.default_rng(5)
    x = rng.permutation(np.arange(2048, dtype=np.uint32)).view(np.uint8)  # 4 whole chunks
    meta, lits, lens, offs = orc.compress_split(x, 4, 2048, 1)
    assert np.array_equal(lits, x)
    assert lens.size == 0 and offs.size == 0


def test_split_corrupt_ports_rejected(orc):
    import synth
    x = synth.generate(1)[:40000]
    ports = orc.compress_split(x, 4, 2048, 0)
    assert orc.decompress_split_status(ports, x.size)[0] == 0
    for k in range(4):
        if ports[k].size == 0:
            continue
        cut = [p.copy() for p in ports]
        cut[k] = cut[k][:-1]
        assert orc.decompress_split_status(cut, x.size)[0] != 0, k
    bad = [p.copy() for p in ports]
    bad[0][4] = 1  # version 1 is the single-stream form
    assert orc.decompress_split_status(bad, x.size)[0] != 0
    assert orc.decompress_split_status(ports, x.size + 1)[0] != 0
