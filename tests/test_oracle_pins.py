"""Pins of the CPU oracle against facts fixed outside itself.

Each check is chosen so that a plausible slip in the oracle (a wrong window
bound, a dropped AND, a farthest-instead-of-nearest offset, a table that
admits the current sub-block, min instead of max in a bucket, an off-by-one
cap, a flipped flag polarity, a wrong raw threshold) fails at least one:

* brute-force longest match on tiny inputs (exhaustive over a 2-symbol
  alphabet, random over small alphabets);
* closed forms: constant chunk, period-p chunk (p <= 32) at level 0, period-40
  chunk at level 1 (only the hashed table can see it, and only from earlier
  sub-blocks, keeping the most recent position), zero chunk, incompressible
  chunk;
* hand-derived golden streams (tests/golden/), among them a level-1 chunk
  whose bytes depend on a bucket collision (hash, table size, max rule), the
  word-size-2 minimum match length from both sides and the raw threshold from
  both sides; the bucket hash worked out by hand for four table sizes;
* structural invariants and an independent replay decoder on every stream;
* round trip through the oracle's own decoder, both levels, all geometries.
"""
import itertools
import os

import numpy as np
import pytest

import goldens
import streamcheck


# ----------------------------------------------------------------------------
# brute force longest match over the near window
# ----------------------------------------------------------------------------
def brute_near(w, window=32):
    """Direct definition: for each i, the longest run w[i+k] == w[i+k-o] over
    1 <= o <= min(window, i), capped at min(255, E - i); the smallest o wins
    ties."""
    E = len(w)
    L = np.zeros(E, np.uint8)
    O = np.zeros(E, np.uint8)
    for i in range(E):
        cap = min(255, E - i)
        best, bo = 0, 0
        for o in range(1, min(window, i) + 1):
            k = 0
            while k < cap and w[i + k] == w[i + k - o]:
                k += 1
            if k > best:
                best, bo = k, o
        L[i], O[i] = best, bo
    return L, O


def test_near_exhaustive_binary_len10(orc):
    for bits in itertools.product((0, 1), repeat=10):
        w = np.array(bits, np.uint32) + 7
        L, O = orc.near_matches(w)
        bl, bo = brute_near(list(w))
        assert np.array_equal(L, bl) and np.array_equal(O, bo), bits


@pytest.mark.parametrize("alphabet,E", [(2, 40), (3, 64), (4, 64), (3, 300), (40, 96)])
def test_near_random_small_alphabet(orc, alphabet, E):
    rng = np.random.default_rng(1000 + alphabet * 7 + E)
    for _ in range(20):
        w = rng.integers(0, alphabet, E).astype(np.uint32) * 0x01010101
        L, O = orc.near_matches(w)
        bl, bo = brute_near(list(w))
        assert np.array_equal(L, bl)
        assert np.array_equal(O, bo)


def test_near_window_is_32(orc):
    # period 32 is seen, period 33 is not
    base = goldens.distinct_u32(33)
    for p, expect in ((32, True), (33, False)):
        w = np.tile(base[:p], 600 // p + 1)[:600]
        L, _ = orc.near_matches(w)
        assert bool(L[p:].any()) is expect
        assert not L[:p].any()


# ----------------------------------------------------------------------------
# the window-width study (match-search section: 32, 48 and 64 elements)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("window", [1, 17, 33, 48, 63, 64])
def test_near_random_small_alphabet_window(orc, window):
    rng = np.random.default_rng(4000 + window)
    for E in (70, 200):
        for alphabet in (2, 5, 60):
            w = rng.integers(0, alphabet, E).astype(np.uint32) * 0x01010101
            L, O = orc.near_matches(w, window)
            bl, bo = brute_near(list(w), window)
            assert np.array_equal(L, bl) and np.array_equal(O, bo), (E, alphabet)


@pytest.mark.parametrize("window", [48, 64])
def test_near_window_bound(orc, window):
    # period `window` is seen, period `window + 1` is not
    base = goldens.distinct_u32(window + 1)
    for p, expect in ((window, True), (window + 1, False)):
        w = np.tile(base[:p], 1200 // p + 1)[:1200]
        L, O = orc.near_matches(w, window)
        assert bool(L[p:].any()) is expect
        assert not L[:p].any()
        if expect:
            assert (O[p:] == p).all()


@pytest.mark.parametrize("p", [33, 40, 48, 64])
def test_period_p_wide_window_closed_form(orc, p):
    # the level-0 closed form of a period-p chunk holds for p up to the window
    E = 512
    w = np.tile(goldens.distinct_u32(p), E // p + 1)[:E]
    s = orc.compress(w.view(np.uint8), 4, 2048, 0, window=64)
    toks = streamcheck.parse(s)["chunks"][0]["items"]
    n_match = -(-(E - p) // 255)
    assert [t[0] for t in toks] == ["L"] * p + ["M"] * n_match
    assert [t[1] for t in toks[p:]] == [255] * (n_match - 1) + [E - p - 255 * (n_match - 1)]
    assert all(t[2] == p for t in toks[p:])
    # a 32-element window sees none of it
    s32 = orc.compress(w.view(np.uint8), 4, 2048, 0)
    assert s32[32 + 8:].size >= 2048


@pytest.mark.parametrize("ws,cs", [(4, 2048), (2, 1024), (1, 4096)])
def test_window_streams_valid(orc, ws, cs):
    import synth
    x = synth.generate(2)[: 300_000 + 5]
    s32 = orc.compress(x, ws, cs, 0)
    assert np.array_equal(orc.compress(x, ws, cs, 0, window=32), s32)
    for window in (48, 64):
        s = orc.compress(x, ws, cs, 0, window=window)
        p = streamcheck.check_invariants(s, x.size)
        offs = [t[2] for ch in p["chunks"] for t in ch["items"] if t[0] == "M"]
        assert max(offs) <= window
        assert np.array_equal(streamcheck.replay(p), x)
        assert np.array_equal(orc.decompress(s, x.size), x)


def test_window_ratio_climbs_on_plane(orc):
    # the pages report the level-0 ratio climbing with the window (32 -> 48 -> 64);
    # on the plane workload the streams shrink in the same order
    import synth
    x = synth.generate(2)[: 1 << 21]
    sizes = [orc.compress(x, 4, 2048, 0, window=w).size for w in (32, 48, 64)]
    assert sizes[0] > sizes[1] > sizes[2]


def test_near_length_cap_and_chunk_end(orc):
    w = np.full(512, 5, np.uint32)
    L, O = orc.near_matches(w)
    assert L[0] == 0 and L[1] == 255 and O[1] == 1
    assert L[256] == 255 and L[300] == 212 and L[511] == 1
    assert (O[1:] == 1).all()


# ----------------------------------------------------------------------------
# closed forms through the whole-chunk encoder
# ----------------------------------------------------------------------------
def test_constant_chunk_both_levels(orc):
    x = np.full(512, 0x01020304, np.uint32).view(np.uint8)
    for lvl in (0, 1):
        blk, items, dbytes = orc.encode_chunk(x, 4, 2048, lvl)
        assert (items, dbytes) == (4, 10)
        assert blk.size == 16
        flags = blk[:4].view(np.uint32)[0]
        assert flags == 0b1110
        assert list(blk[4:16]) == [4, 3, 2, 1, 255, 1, 255, 1, 1, 1, 0, 0]


@pytest.mark.parametrize("p", [1, 2, 7, 16, 31, 32])
def test_period_p_level0_closed_form(orc, p):
    E = 512
    w = np.tile(goldens.distinct_u32(p), E // p + 1)[:E]
    blk, items, dbytes = orc.encode_chunk(w.view(np.uint8), 4, 2048, 0)
    n_match = -(-(E - p) // 255)
    assert items == p + n_match
    assert dbytes == 4 * p + 2 * n_match
    parsed = streamcheck.parse(_one_chunk_stream(orc, w.view(np.uint8), 4, 2048, 0))
    toks = parsed["chunks"][0]["items"]
    assert [t[0] for t in toks] == ["L"] * p + ["M"] * n_match
    lens = [t[1] for t in toks[p:]]
    assert lens == [255] * (n_match - 1) + [E - p - 255 * (n_match - 1)]
    assert all(t[2] == p for t in toks[p:])


def _collision_free_period(orc, P, E, seed):
    """P distinct random words whose P cyclic two-word keys hash to distinct
    buckets, so every hashed lookup of a periodic chunk is unambiguous."""
    bits = orc.hash_bits(E)
    rng = np.random.default_rng(seed)
    while True:
        base = rng.integers(1, 2**32, P, dtype=np.uint64).astype(np.uint32)
        if len(set(base.tolist())) < P:
            continue
        keys = {orc.hash2(int(base[j]), int(base[(j + 1) % P]), bits) for j in range(P)}
        if len(keys) == P:
            return base


def test_period40_level1_closed_form(orc):
    """Period 40 > 32: the near window sees nothing. Level 1 finds a candidate
    at position i only for sources in earlier sub-blocks (of 64 positions), and
    the bucket keeps the most recent (largest) position:
      i = 0..63   : sub-block 0 looks up an empty table -> 64 literals
      i = 64      : most recent key position in [0, 64) is 24 -> (255, 40)
      i = 319     : sub-block 4, table holds [0, 256): most recent of
                    39, 79, ..., 239 is 239 -> offset 80, length 512-319 = 193.
    """
    E, P = 512, 40
    base = _collision_free_period(orc, P, E, 4040)
    w = np.tile(base, E // P + 1)[:E]
    x = w.view(np.uint8)
    blk0, items0, d0 = orc.encode_chunk(x, 4, 2048, 0)
    assert items0 == 0x80000000 and d0 == 2048          # level 0: raw
    blk, items, dbytes = orc.encode_chunk(x, 4, 2048, 1)
    assert items == 66 and dbytes == 64 * 4 + 4
    assert blk.size == 12 + 260
    fl = blk[:12].view(np.uint32)
    assert list(fl) == [0, 0, 0b11]
    data = blk[12:]
    assert np.array_equal(data[:256].view(np.uint32), w[:64])
    assert list(data[256:260]) == [255, 40, 193, 80]


def test_level1_never_worse_than_level0_and_valid(orc):
    rng = np.random.default_rng(7)
    for E in (256, 512, 1024):
        for alphabet in (3, 50, 1000):
            w = rng.integers(0, alphabet, E).astype(np.uint32)
            L0, O0 = orc.near_matches(w)
            L1, O1 = orc.level1_matches(w)
            assert (L1 >= L0).all()
            for i in range(E):
                if L1[i]:
                    o, ln = int(O1[i]), int(L1[i])
                    assert 1 <= o <= min(255, i)
                    assert np.array_equal(w[i:i + ln], w[i - o:i - o + ln])
                    if L1[i] == L0[i]:
                        assert O1[i] == O0[i]


def test_level1_table_definition_tiny(orc):
    """Declarative form of the sub-block rule on small chunks: the candidate for
    i in sub-block s is the largest p < s*E/8 (p+1 < E) whose two-word key
    hashes to i's bucket; it counts only if it verifies and i - p <= 255."""
    rng = np.random.default_rng(11)
    for E in (256, 512):
        bits = orc.hash_bits(E)
        for alphabet in (2, 4, 9):
            w = rng.integers(0, alphabet, E).astype(np.uint32)
            L0, O0 = orc.near_matches(w)
            L1, O1 = orc.level1_matches(w)
            h = [orc.hash2(int(w[p]), int(w[p + 1]), bits) for p in range(E - 1)]
            sb = E // 8
            for i in range(E - 1):
                s = i // sb
                cands = [p for p in range(0, s * sb) if p + 1 < E and h[p] == h[i]]
                el, eo = int(L0[i]), int(O0[i])
                if cands:
                    p = max(cands)
                    d = i - p
                    if 1 <= d <= 255:
                        k = 0
                        cap = min(255, E - i)
                        while k < cap and w[i + k] == w[p + k]:
                            k += 1
                        if k > el or (k == el and k > 0 and d < eo):
                            el, eo = k, d
                assert (L1[i], O1[i]) == (el, eo), (E, alphabet, i)


def _hash_table_rows():
    rows = []
    with open(os.path.join(goldens.GOLDEN_DIR, "level1_hash_values.tab")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(v, 0) for v in line.split()])
    return rows


def test_level1_hash_values(orc):
    """The bucket of a two-word key and the table size against values worked
    out by hand from the documented formula (tests/golden/level1_hash_values.tab):
    a slip in either multiplier, the xor, the shift or log2(2E) changes a row."""
    rows = _hash_table_rows()
    assert len(rows) >= 20
    for E, B, k0, k1, p0, p1, x, h in rows:
        # the row's own arithmetic (guards the table against a typo)
        assert p0 ^ p1 == x and x >> (32 - B) == h
        assert orc.hash_bits(E) == B, (E, B)
        assert orc.hash2(k0, k1, B) == h, (E, k0, k1)


def test_min_match_len_each_word_size(orc):
    """A token (2 bytes) is taken only when its literals would take more: the
    shortest match is 3, 2 and 1 elements for word sizes 1, 2 and 4 (the
    abcab, lmin_ws2 and constant goldens show each one in a stream)."""
    assert [orc.min_match_len(ws) for ws in (1, 2, 4)] == [3, 2, 1]


def _one_chunk_stream(orc, x, ws, cs, lvl):
    return orc.compress(x, ws, cs, lvl)


def test_zero_chunk_sentinel_and_raw(orc):
    g = [c for c in goldens.load_all() if c["name"].startswith("zero_then")][0]
    s = orc.compress(g["x"], 4, 1024, 0)
    assert np.array_equal(s, g["stream"])


# ----------------------------------------------------------------------------
# golden streams
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("case", goldens.load_all(), ids=lambda c: c["name"])
def test_golden_streams(orc, case):
    for lvl in case["levels"]:
        for window in case["windows"]:
            s = orc.compress(case["x"], case["ws"], case["cs"], lvl, window=window)
            assert np.array_equal(s, case["stream"]), (lvl, window)
    y = orc.decompress(case["stream"], case["x"].size)
    assert np.array_equal(y, case["x"])
    p = streamcheck.check_invariants(case["stream"], case["x"].size)
    assert np.array_equal(streamcheck.replay(p), case["x"])


# ----------------------------------------------------------------------------
# invariants + round trip
# ----------------------------------------------------------------------------
GEOMS = [(ws, cs) for ws in (1, 2, 4) for cs in (1024, 2048, 4096)]


@pytest.mark.parametrize("ws,cs", GEOMS)
@pytest.mark.parametrize("lvl", [0, 1])
def test_round_trip_and_invariants_random(orc, ws, cs, lvl):
    rng = np.random.default_rng(ws * 100 + cs + lvl)
    for n in (0, 1, 3, cs - 1, cs, cs + 1, 3 * cs + 5, 7 * cs + 2):
        kind = rng.integers(0, 4)
        if kind == 0:
            x = rng.integers(0, 4, n).astype(np.uint8)
        elif kind == 1:
            x = rng.integers(0, 256, n).astype(np.uint8)
        elif kind == 2:
            x = np.zeros(n, np.uint8)
            if n:
                x[rng.integers(0, n, n // 50 + 1)] = 3
        else:
            x = (np.arange(n) // 7 % 5).astype(np.uint8)
        s = orc.compress(x, ws, cs, lvl)
        p = streamcheck.check_invariants(s, n)
        assert np.array_equal(streamcheck.replay(p), x)
        assert np.array_equal(orc.decompress(s, n), x)
        assert s.size <= orc.compress_bound(n, ws, cs)


@pytest.mark.parametrize("cfg_id", [1])
@pytest.mark.parametrize("lvl", [0, 1])
def test_round_trip_tiny_workload(orc, cfg_id, lvl):
    import synth
    cfg = synth.CONFIGS[cfg_id]
    x = synth.generate(cfg_id)
    s = orc.compress(x, cfg.word_size, cfg.chunk_size, lvl)
    p = streamcheck.check_invariants(s, x.size)
    assert np.array_equal(orc.decompress(s, x.size), x)
    assert np.array_equal(streamcheck.replay(p), x)


def test_sparse_workload_zero_chunks(orc):
    # the zero-chunk sentinel at workload scale: a chunk is coded {0, 0} exactly
    # when its bytes are all zero, and the other chunks replay to the input
    import synth
    cfg = synth.CONFIGS[7]
    x = synth.generate(7)[: 4 << 20]
    s = orc.compress(x, cfg.word_size, cfg.chunk_size, cfg.match_level)
    p = streamcheck.check_invariants(s, x.size)
    cs = cfg.chunk_size
    zero = [not x[i: i + cs].any() for i in range(0, x.size, cs)]
    assert [ch["kind"] == "zero" for ch in p["chunks"]] == zero
    assert 0.3 < sum(zero) / len(zero) < 1.0
    assert np.array_equal(streamcheck.replay(p), x)


def test_u16_workload_codes():
    # word_size 2 workload: Lorenzo codes centred on the radius, within u16
    import synth
    cfg = synth.CONFIGS[6]
    assert (cfg.word_size, cfg.dtype, cfg.radius) == (2, "u16", 32768)
    v = synth.generate(6)[: 1 << 20].view(np.uint16)
    assert abs(int(np.median(v)) - cfg.radius) <= 2


def test_levels_decode_identically_plane(orc):
    import synth
    x = synth.generate(2)[: 1 << 21]
    s0 = orc.compress(x, 4, 2048, 0)
    s1 = orc.compress(x, 4, 2048, 1)
    assert s1.size <= s0.size
    assert np.array_equal(orc.decompress(s0, x.size), x)
    assert np.array_equal(orc.decompress(s1, x.size), x)


def test_threaded_oracle_matches_sequential(orc):
    import synth
    x = synth.generate(1)
    for lvl in (0, 1):
        a = orc.compress(x, 4, 2048, lvl)
        b = orc.compress_threads(x, 4, 2048, lvl, threads=4)
        assert np.array_equal(a, b)
        assert np.array_equal(orc.decompress_threads(a, x.size, threads=3), x)
    z = np.zeros(3 * 1024 + 5, np.uint8)
    s = orc.compress(z, 1, 1024, 1)
    assert np.array_equal(orc.decompress_threads(s, z.size, threads=2), z)


# ----------------------------------------------------------------------------
# decoder rejects corrupt streams
# ----------------------------------------------------------------------------
def test_oracle_decoder_rejects_corruption(orc):
    import synth
    x = synth.generate(1)[:20000]
    s = orc.compress(x, 4, 2048, 0)
    assert orc.decompress_status(s, x.size) == 0
    assert orc.decompress_status(s[:-4], x.size) != 0          # truncated
    assert orc.decompress_status(s, x.size + 1) != 0           # wrong n
    bad = s.copy()
    bad[0] ^= 1                                               # magic
    assert orc.decompress_status(bad, x.size) != 0
    bad = s.copy()
    bad[32 + 4] ^= 0x40                                        # data_bytes of chunk 0
    assert orc.decompress_status(bad, x.size) != 0


def test_level1_changes_only_to_far_and_longer(orc):
    """The near search is exact over offsets 1..32 with the same caps (255 and
    the chunk end) and nearest-offset ties, so a hashed candidate can replace
    the level-0 result only with an offset above 32 and a strictly longer run.
    Checked on inputs with many near and far repeats."""
    rng = np.random.default_rng(23)
    changed = 0
    for E in (256, 512, 1024, 4096):
        for alphabet in (2, 3, 8, 64):
            base = rng.integers(0, alphabet, 48).astype(np.uint32)
            w = np.tile(base, E // 48 + 1)[:E].copy()
            flip = rng.random(E) < 0.05
            w[flip] = rng.integers(0, alphabet, int(flip.sum()))
            L0, O0 = orc.near_matches(w)
            L1, O1 = orc.level1_matches(w)
            diff = (L1 != L0) | (O1 != O0)
            changed += int(diff.sum())
            assert (O1[diff] > 32).all()
            assert (L1[diff] > L0[diff]).all()
    assert changed > 0
