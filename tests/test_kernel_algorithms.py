"""Models of the encode kernel's parallel algorithms, checked on CPU against
the definitions they must reproduce exactly (GPULZ stage page, match-search
section and provenance paragraph):

* the segment-parallel greedy parse with its fixpoint and exact-entry frontier
  equals the sequential greedy parse;
* the register AND-chain search (per-thread triangle, lockstep continuation,
  four- and one-segment skips under the 255 cap) equals the longest match over
  the near window, nearest offset on ties;
* the far pass for windows of 33..64 elements (masks for offsets 33..64, the
  same chain search, merge keeping the near run on ties) equals the longest
  match over the whole window.

These are statements about the algorithms the kernel implements, written in
plain Python from the kernel's step list; the CUDA code itself is checked
against the oracle by the GPU parity tests.
"""
import numpy as np
import pytest

MAXLEN = 255


# ----------------------------------------------------------------------------
# definitions
# ----------------------------------------------------------------------------
def longest_matches(v, window):
    """Longest run v[i+k] == v[i+k-o] over 1 <= o <= min(window, i), capped at
    min(255, E - i); nearest offset on ties. Returns (len, off) arrays."""
    E = len(v)
    best = np.zeros(E, np.int64)
    boff = np.zeros(E, np.int64)
    for o in range(1, window + 1):
        if o >= E:
            break
        eq = np.zeros(E + 1, bool)
        eq[o:E] = v[o:] == v[:-o]
        run = np.zeros(E + 1, np.int64)
        for i in range(E - 1, -1, -1):
            run[i] = run[i + 1] + 1 if eq[i] else 0
        r = np.minimum(run[:E], np.minimum(MAXLEN, E - np.arange(E)))
        better = r > best
        best[better] = r[better]
        boff[better] = o
    return best, np.where(best > 0, boff, 0)


def serial_parse(step):
    path, p = set(), 0
    while p < len(step):
        path.add(p)
        p += int(step[p])
    return path


# ----------------------------------------------------------------------------
# models of the kernel steps
# ----------------------------------------------------------------------------
def masks(v, K=0, far_mask=0xFFFFFFFF):
    """Bit o-1 of m[i] set iff v[i] == v[i-K-o], 1 <= o <= 32, i-K-o >= 0."""
    E = len(v)
    m = [0] * E
    for i in range(E):
        mm = 0
        for o in range(1, 33):
            j = i - K - o
            if j >= 0 and v[i] == v[j]:
                mm |= 1 << (o - 1)
        m[i] = mm & far_mask
    return m


def and_chains(m, E, SEGP):
    """Per position (length, nearest offset bit) from the masks, as each thread
    computes them: the triangle inside its segment, then the continuation of
    the chains alive at the segment end, with whole-segment skips."""
    sa = []
    for t in range(E // SEGP):
        a = 0xFFFFFFFF
        for p in range(SEGP):
            a &= m[t * SEGP + p]
        sa.append(a)
    out = []
    for t in range(E // SEGP):
        seg_a = t * SEGP
        cc = [m[seg_a + p] for p in range(SEGP)]
        L = [1 if c else 0 for c in cc]
        alive = [c != 0 for c in cc]
        for k in range(1, SEGP):
            for p in range(SEGP - k):
                if alive[p]:
                    x = cc[p] & m[seg_a + p + k]
                    if x:
                        cc[p], L[p] = x, L[p] + 1
                    else:
                        alive[p] = False
        live = alive[:]  # chains alive at the segment end
        st = 0
        while any(live) and seg_a + SEGP + st < E:
            q0 = seg_a + SEGP + st
            if all(live) or st >= SEGP:
                j = q0 // SEGP
                p0 = live.index(True)
                room = MAXLEN - (SEGP - p0 + st)
                take, s = 0, 0
                if room > 4 * SEGP and q0 + 4 * SEGP <= E:
                    s = sa[j] & sa[j + 1] & sa[j + 2] & sa[j + 3]
                    if all(not live[p] or cc[p] & s for p in range(SEGP)):
                        take = 4 * SEGP
                if not take and room > SEGP:
                    s = sa[j]
                    if all(not live[p] or cc[p] & s for p in range(SEGP)):
                        take = SEGP
                if take:
                    for p in range(SEGP):
                        if live[p]:
                            cc[p] &= s
                            L[p] += take
                    st += take
                    continue
            for k in range(SEGP):
                if not any(live):
                    break
                om = m[q0 + k]
                nxt = [False] * SEGP
                for p in range(SEGP):
                    if live[p] and cc[p] & om:
                        cc[p] &= om
                        nxt[p] = True
                        L[p] += 1
                over = SEGP + st + 1 - MAXLEN
                if over >= 0:
                    for p in range(min(over, SEGP - 1) + 1):
                        nxt[p] = False
                live = nxt
                st += 1
        for p in range(SEGP):
            out.append((L[p], (cc[p] & -cc[p]).bit_length() if L[p] else 0))
    return out


def segment_parse(step, SEGP, frontier_from=2, stop_on_exits=True):
    """Greedy parse by per-segment walks and fixpoint rounds, with the
    exact-entry frontier from round `frontier_from` on. The rounds end once a
    round changed no segment's exit (`stop_on_exits`, the kernel's rule: every
    entry then equals the exit before it, the fixpoint) or, the slower rule,
    no segment's entry. Returns (path, rounds)."""
    E = len(step)
    nthr = E // SEGP

    def walk(t, e):
        p, path = e, set()
        while p < (t + 1) * SEGP:
            path.add(p)
            p += int(step[p])
        return p, path

    exits, paths, cur = [], [], []
    for t in range(nthr):
        x, pa = walk(t, t * SEGP)
        exits.append(x)
        paths.append(pa)
        cur.append(t * SEGP)
    fr = [(0, exits[0]), None]
    rnd = 0
    while True:
        use = rnd >= frontier_from
        fb = rnd & 1
        fk, fx = fr[fb] if use else (nthr, 0)
        new, changed, wrote = list(exits), False, False
        for t in range(nthr):
            prev = 0 if t == 0 else exits[t - 1]
            reached = use and t > fk and t * SEGP <= fx
            if reached:
                prev = fx
            if prev != cur[t]:
                changed, cur[t] = True, prev
                if prev >= (t + 1) * SEGP:
                    new[t], paths[t] = prev, set()
                else:
                    new[t], paths[t] = walk(t, prev)
            if use and reached and fx < (t + 1) * SEGP:
                fr[fb ^ 1], wrote = (t, new[t]), True
        if use and not wrote:
            fr[fb ^ 1] = fr[fb]
        exit_changed = new != exits
        exits = new
        rnd += 1
        if not (exit_changed if stop_on_exits else changed):
            return set().union(*paths), rnd


def and_chains_zeroed(m, E, SEGP):
    """The same chains in the representation the kernel steps them in: a
    chain's running AND is left at 0 once it dies (so a step needs no liveness
    test: AND, and where the result is nonzero keep it and set the survivor
    bit), the last nonzero value is kept aside for the offset, the lengths are
    counted from the survivor bits, and a chain reaching the cap is zeroed."""
    sa = []
    for t in range(E // SEGP):
        a = 0xFFFFFFFF
        for p in range(SEGP):
            a &= m[t * SEGP + p]
        sa.append(a)
    out = []
    for t in range(E // SEGP):
        seg_a = t * SEGP
        cc = [m[seg_a + p] for p in range(SEGP)]
        keep = cc[:]
        A = sum(1 << p for p in range(SEGP) if cc[p])
        L = [(A >> p) & 1 for p in range(SEGP)]
        P = A & (1 << (SEGP - 1))
        for k in range(1, SEGP):
            act = A & ((1 << (SEGP - k)) - 1)
            if not act:
                break
            An = 0
            for p in range(SEGP - k):  # no liveness test: dead chains hold 0
                cc[p] &= m[seg_a + p + k]
                if cc[p]:
                    keep[p] = cc[p]
                    An |= 1 << p
            for p in range(SEGP):
                L[p] += (An >> p) & 1
            P |= An & (1 << (SEGP - 1 - k))
            A = An
        A2, st = P, 0
        while A2 and seg_a + SEGP + st < E:
            q0 = seg_a + SEGP + st
            if A2 == (1 << SEGP) - 1 or st >= SEGP:
                j = q0 // SEGP
                p0 = (A2 & -A2).bit_length() - 1
                room = MAXLEN - (SEGP - p0 + st)
                take, s = 0, 0
                live = [(A2 >> p) & 1 for p in range(SEGP)]
                if room > 4 * SEGP and q0 + 4 * SEGP <= E:
                    s = sa[j] & sa[j + 1] & sa[j + 2] & sa[j + 3]
                    if all(not live[p] or cc[p] & s for p in range(SEGP)):
                        take = 4 * SEGP
                if not take and room > SEGP:
                    s = sa[j]
                    if all(not live[p] or cc[p] & s for p in range(SEGP)):
                        take = SEGP
                if take:
                    for p in range(SEGP):
                        cc[p] &= s  # dead chains stay 0
                        if live[p]:
                            keep[p] = cc[p]
                            L[p] += take
                    st += take
                    continue
            for k in range(SEGP):
                if not A2:
                    break
                om = m[q0 + k]
                An = 0
                for p in range(SEGP):
                    cc[p] &= om
                    if cc[p]:
                        keep[p] = cc[p]
                        An |= 1 << p
                for p in range(SEGP):
                    L[p] += (An >> p) & 1
                over = SEGP + st + 1 - MAXLEN
                if over >= 0:
                    lim = min(over, SEGP - 1)
                    An &= ~((2 << lim) - 1)
                    for p in range(lim + 1):
                        cc[p] = 0
                A2 = An
                st += 1
        for p in range(SEGP):
            out.append((L[p], (keep[p] & -keep[p]).bit_length()))
    return out


# ----------------------------------------------------------------------------
# inputs
# ----------------------------------------------------------------------------
def _chunks(seed, E):
    rng = np.random.default_rng(seed)
    yield "constant", np.full(E, 7)
    yield "period3", np.tile(rng.integers(0, 9, 3), E)[:E]
    yield "period40", np.tile(rng.integers(0, 1000, 40), E)[:E]
    yield "period57_broken", np.where(rng.random(E) < 0.01, 99, np.tile(rng.integers(0, 50, 57), E)[:E])
    yield "small_alphabet", rng.integers(0, 3, E)
    yield "sparse", np.where(rng.random(E) < 0.03, rng.integers(1, 4, E), 0)
    runs = np.zeros(E, np.int64)
    p = 0
    while p < E:
        n = int(rng.integers(1, 400))
        runs[p:p + n] = rng.integers(0, 3) if rng.random() < 0.5 else rng.integers(0, 4, min(n, E - p))
        p += n
    yield "run_mix", runs
    # short periods with a few breaks, and long runs with short bursts: chains
    # of one thread then die at different steps, so the cap is approached at
    # every phase of the skips
    for k in range(4):
        base = rng.integers(0, 4, int(rng.integers(1, 6)))
        w = np.tile(base, E)[:E].copy()
        nb = int(rng.integers(1, 6))
        w[rng.integers(0, E, nb)] = rng.integers(0, 6, nb)
        yield "period_breaks_%d" % k, w
        w = np.full(E, 1)
        for _ in range(int(rng.integers(1, 5))):
            a = int(rng.integers(0, E))
            w[a:a + int(rng.integers(1, 6))] = rng.integers(0, 3)
        yield "run_bursts_%d" % k, w
    # one long run entered at many phases relative to the segments and the cap
    for ph in (1, 3, 5, 9, 13, 17, 23, 29, 31):
        w = np.full(E, 5)
        w[:ph] = np.arange(ph) + 100
        w[ph + 300: ph + 301] = 99
        yield "run_phase_%d" % ph, w


# ----------------------------------------------------------------------------
# checks
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("E,SEGP", [(256, 8), (512, 8)])
def test_and_chains_with_skips_equal_longest_match(E, SEGP):
    for name, v in _chunks(E + SEGP, E):
        got = and_chains(masks(v), E, SEGP)
        L, O = longest_matches(v, 32)
        assert got == list(zip(L.tolist(), O.tolist())), name


@pytest.mark.parametrize("E,SEGP", [(256, 8), (512, 8), (1024, 16)])
def test_zeroed_chains_equal_longest_match(E, SEGP):
    # the kernel's representation of the chains gives the same lengths and
    # nearest offsets as brute force
    for name, v in _chunks(E + 3 * SEGP, E):
        got = and_chains_zeroed(masks(v), E, SEGP)
        L, O = longest_matches(v, 32)
        assert got == list(zip(L.tolist(), O.tolist())), name


@pytest.mark.parametrize("window", [33, 48, 64])
def test_far_pass_merge_equals_wide_window(window):
    E, SEGP = 512, 8
    far_mask = 0xFFFFFFFF if window == 64 else (1 << (window - 32)) - 1
    for name, v in _chunks(window, E):
        near = and_chains(masks(v), E, SEGP)
        far = and_chains(masks(v, 32, far_mask), E, SEGP)
        got = [(l2, o2 + 32) if l2 > l1 else (l1, o1) for (l1, o1), (l2, o2) in zip(near, far)]
        L, O = longest_matches(v, window)
        assert got == list(zip(L.tolist(), O.tolist())), name


def test_segment_parse_equals_serial_parse():
    rng = np.random.default_rng(77)
    for trial in range(120):
        SEGP = (8, 16)[trial % 2]
        E = (256, 512, 1024)[trial % 3] if SEGP == 8 else 4096
        dens = rng.random()
        step = np.ones(E, np.int64)
        for j in range(E):
            if rng.random() < dens:
                step[j] = rng.integers(1, 256) if rng.random() < 0.3 else rng.integers(1, 12)
            step[j] = min(step[j], E - j)
        ref = serial_parse(step)
        for start in (0, 2, 10 ** 9):  # frontier from the start, from round 3, never
            for stop_on_exits in (True, False):
                got, _ = segment_parse(step, SEGP, start, stop_on_exits)
                assert got == ref, (trial, start, stop_on_exits)


def test_frontier_bounds_rounds_on_long_runs():
    # a chunk of long matches: without the frontier the rounds grow with the
    # number of segments a match spans; with it they stay few
    E, SEGP = 1024, 8
    v = np.zeros(E, np.int64)
    v[[0, 300, 301, 700]] = [1, 2, 3, 4]
    L, _ = longest_matches(v, 32)
    step = np.where(L >= 2, L, 1)
    _, plain = segment_parse(step, SEGP, 10 ** 9)
    path, fast = segment_parse(step, SEGP, 2)
    assert path == serial_parse(step)
    assert plain > 30 and fast <= 10


def test_step_byte_tricks():
    # the parse's step bytes, built four at a time from the run-length bytes:
    # step = len where len >= Lmin (a match), else 1 (a literal); the match
    # bits gathered by one multiply. Lmin is 1, 2, 3 for word sizes 4, 2, 1.
    rng = np.random.default_rng(5)
    lens = np.concatenate([rng.integers(0, 256, (20000, 4)),
                           rng.choice([0, 1, 2, 3, 4, 127, 128, 129, 130, 131, 255], (20000, 4))])
    M = 0xFFFFFFFF
    for row in lens.tolist():
        t = row[0] | row[1] << 8 | row[2] << 16 | row[3] << 24
        for ws, lmin in ((4, 1), (2, 2)):
            u = t & 0xFEFEFEFE if ws == 2 else t
            z = ~(((u & 0x7F7F7F7F) + 0x7F7F7F7F) | u | 0x7F7F7F7F) & M
            T = t | (z >> 7)
            mt = ((((~z & M) >> 7) & 0x01010101) * 0x01020408 & M) >> 24
            for k in range(4):
                assert (T >> 8 * k) & 0xFF == (row[k] if row[k] >= lmin else 1)
                assert (mt >> k) & 1 == (row[k] >= lmin)
        f = ((((t | 0x80808080) - 0x03030303) & M) | t) & 0x80808080
        keep = (f >> 7) * 0xFF & M
        T = (t & keep) | (~keep & 0x01010101 & M)
        mt = ((((f >> 7) & 0x01010101) * 0x01020408) & M) >> 24
        for k in range(4):
            assert (T >> 8 * k) & 0xFF == (row[k] if row[k] >= 3 else 1)
            assert (mt >> k) & 1 == (row[k] >= 3)
