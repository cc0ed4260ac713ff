"""Pins for the CPU oracle: each checks the oracle against something other than
itself -- a closed form, a library routine (numpy reflect padding, numpy /
scipy convolution), a hand-worked example, a brute-force per-output loop or an
invariant.  Each pin is a function of an ``oracle.Oracle`` that raises
AssertionError when the oracle disagrees, so the same pins run against the real
oracle (all must hold) and against builds with a planted mistake (at least one
must fail for every plant).

Definition pinned (integer motion blur, reading A):
  V[y][x] = (sum_k t_k F[mirror(y+k-2)][x] + 2^(bpc-1)) >> bpc     (vertical first,
  B[y][x] = (sum_k t_k V[y][mirror(x+k-2)] + 2^15) >> 16            ADR-1392 Decision 4)
  t = (3571, 16004, 26386, 16004, 3571); mirror: i<0 -> -i, i>=n -> 2n-i-2.
"""
from __future__ import annotations

import numpy as np

T = (3571, 16004, 26386, 16004, 3571)
assert sum(T) == 65536


def _dt(bpc):
    return np.uint8 if bpc == 8 else np.uint16


def reflect_index(i: int, n: int) -> int:
    """Mirror index by a library routine: numpy's 'reflect' padding (reflection
    about the edge sample, the edge not repeated)."""
    padded = np.pad(np.arange(n), 2, mode="reflect")
    return int(padded[i + 2])


def conv1d_reflect(x: np.ndarray, taps=T) -> np.ndarray:
    """sum_k t_k x[mirror(i+k-2)] for every i, with numpy padding + convolution
    (int64; the taps are symmetric so correlation == convolution)."""
    p = np.pad(np.asarray(x, dtype=np.int64), 2, mode="reflect")
    return np.convolve(p, np.asarray(taps, dtype=np.int64), mode="valid")


# --------------------------------------------------------------------------- pins

def pin_mirror(o):
    for n in range(3, 13):
        for i in range(-2, n + 2):
            assert o.mirror(i, n) == reflect_index(i, n), (i, n)


def pin_constant_frames(o):
    """A constant frame c blurs to exactly c * 2^(16-bpc): the vertical pass gives
    (65536 c + 2^(bpc-1)) >> bpc = c 2^(16-bpc) and the horizontal pass keeps it."""
    for bpc in (8, 10, 12, 16):
        for (w, h) in ((3, 3), (7, 5), (17, 4)):
            for c in (0, 1, (1 << bpc) // 3, (1 << bpc) - 1):
                f = np.full((h, w), c, dtype=_dt(bpc))
                b = o.blur(f, bpc)
                assert np.all(b == (c << (16 - bpc))), (bpc, w, h, c)


def pin_two_constant_sad_and_score(o):
    """Two constant frames: SAD = |c1-c2| 2^(16-bpc) w h; the 8-bit score is
    exactly |c1-c2| (and a quarter of it at 10 bits)."""
    for bpc, pairs in ((8, ((0, 255), (17, 3), (100, 100))), (10, ((0, 1023), (500, 20)))):
        w, h = 9, 6
        seq = np.stack([np.full((h, w), c, _dt(bpc)) for c in pairs[0]] +
                       [np.full((h, w), c, _dt(bpc)) for c in pairs[1]])
        sad = o.motion_sad_sequence(seq, bpc)
        c = [pairs[0][0], pairs[0][1], pairs[1][0], pairs[1][1]]
        for i in range(1, 4):
            assert int(sad[i]) == abs(c[i] - c[i - 1]) * (1 << (16 - bpc)) * w * h
        score, _ = o.scores(sad, w, h)
        for i in range(1, 4):
            assert score[i] == abs(c[i] - c[i - 1]) / (1 << (bpc - 8))


def pin_impulse_interior(o):
    """Impulse v at (y0, x0) far enough from every edge that no mirrored tap
    reaches it (3 <= y0 <= h-4, likewise x0): B is the outer form
    ((v t_{2+dy} + 2^(bpc-1)) >> bpc) t_{2+dx} + 2^15) >> 16 in the 5x5 window,
    zero elsewhere."""
    for bpc, v in ((8, 255), (8, 1), (10, 1023), (10, 37), (16, 65535)):
        h, w = 11, 13
        for (y0, x0) in ((5, 6), (3, 3), (7, 9)):
            f = np.zeros((h, w), _dt(bpc))
            f[y0, x0] = v
            exp = np.zeros((h, w), np.int64)
            for dy in range(-2, 3):
                vert = (v * T[2 + dy] + (1 << (bpc - 1))) >> bpc
                for dx in range(-2, 3):
                    exp[y0 + dy, x0 + dx] = (vert * T[2 + dx] + 32768) >> 16
            assert np.array_equal(o.blur(f, bpc).astype(np.int64), exp), (bpc, v, y0, x0)


def pin_hand_worked_6x6(o):
    """Hand-worked 8-bit example: 6x6, cur is zero except cur[2][2] = 255.

    Centre: vertical (255*26386 + 128) >> 8 = (6728430 + 128) >> 8 = 26283;
            horizontal (26283*26386 + 32768) >> 16 = (693503238 + 32768) >> 16 = 10582.
    Corner: row 0 takes t0 through mirror(-2) = 2 and t4 at row 2, so the vertical
            value is (255*(3571+3571) + 128) >> 8 = (1821210 + 128) >> 8 = 7114;
            column 0 likewise folds t0 and t4 onto column 2:
            (7114*7142 + 32768) >> 16 = (50808188 + 32768) >> 16 = 775.
    Last row/column: mirror never reaches row/column 2 from y = 5, so B = 0 there.
    """
    f = np.zeros((6, 6), np.uint8)
    f[2, 2] = 255
    b = o.blur(f, 8).astype(np.int64)
    assert b[2, 2] == 10582
    assert b[0, 0] == 775
    assert np.all(b[5, :] == 0) and np.all(b[:, 5] == 0)
    # full matrix: fold the taps through numpy's reflect padding
    eff = np.zeros(6, np.int64)
    for y in range(6):
        eff[y] = sum(T[k] for k in range(5) if reflect_index(y + k - 2, 6) == 2)
    vert = (255 * eff + 128) >> 8
    exp = (np.outer(vert, eff) + 32768) >> 16
    assert np.array_equal(b, exp)
    assert o.sad(b, np.zeros((6, 6), np.uint16)) == int(exp.sum())
    # corner impulse: the top-left 3x3 mirrors the centre 3x3's lower-right quadrant
    g = np.zeros((6, 6), np.uint8)
    g[0, 0] = 255
    bc = o.blur(g, 8).astype(np.int64)
    assert bc[0, 0] == 10582 and bc[0, 1] == b[2, 3] and bc[2, 2] == b[4, 4]
    assert np.all(bc[3:, :] == 0) and np.all(bc[:, 3:] == 0)


def pin_row_constant(o):
    """F[y][x] = g(y): the horizontal pass of a constant row returns it exactly,
    so B[y][x] = (conv_reflect(g)[y] + 2^(bpc-1)) >> bpc for every x."""
    rng = np.random.default_rng(11)
    for bpc in (8, 10, 16):
        for (w, h) in ((3, 3), (5, 9), (12, 31)):
            g = rng.integers(0, 1 << bpc, size=h)
            f = np.repeat(g[:, None], w, axis=1).astype(_dt(bpc))
            exp = (conv1d_reflect(g) + (1 << (bpc - 1))) >> bpc
            b = o.blur(f, bpc).astype(np.int64)
            assert np.array_equal(b, np.repeat(exp[:, None], w, axis=1)), (bpc, w, h)


def pin_column_constant(o):
    """F[y][x] = f(x): the vertical pass gives f(x) 2^(16-bpc) exactly, so
    B[y][x] = (conv_reflect(f 2^(16-bpc))[x] + 2^15) >> 16 for every y."""
    rng = np.random.default_rng(12)
    for bpc in (8, 10, 16):
        for (w, h) in ((3, 3), (9, 5), (33, 4)):
            fx = rng.integers(0, 1 << bpc, size=w)
            f = np.repeat(fx[None, :], h, axis=0).astype(_dt(bpc))
            exp = (conv1d_reflect(fx << (16 - bpc)) + 32768) >> 16
            b = o.blur(f, bpc).astype(np.int64)
            assert np.array_equal(b, np.repeat(exp[None, :], h, axis=0)), (bpc, w, h)


def pin_scipy_separable(o):
    """General frames against scipy.ndimage.correlate1d in mirror mode (float64,
    exact below 2^53), vertical first with floor shifts."""
    from scipy import ndimage
    rng = np.random.default_rng(13)
    taps = np.asarray(T, dtype=np.float64)
    for bpc in (8, 10, 12, 16):
        for (w, h) in ((3, 3), (4, 7), (16, 9), (37, 23), (64, 48)):
            f = rng.integers(0, 1 << bpc, size=(h, w)).astype(_dt(bpc))
            s = ndimage.correlate1d(f.astype(np.float64), taps, axis=0, mode="mirror")
            v = (s.astype(np.int64) + (1 << (bpc - 1))) >> bpc
            s2 = ndimage.correlate1d(v.astype(np.float64), taps, axis=1, mode="mirror")
            exp = (s2.astype(np.int64) + 32768) >> 16
            assert np.array_equal(o.blur(f, bpc).astype(np.int64), exp), (bpc, w, h)


def _mirror_fold(i: int, n: int) -> int:
    # the same reflection written as a fold: (n-1) - |(n-1) - |i||
    return (n - 1) - abs((n - 1) - abs(i))


def brute_force_blur(f: np.ndarray, bpc: int) -> np.ndarray:
    """Per-output 25-MAC loop: for each output and each horizontal tap the
    vertical value is recomputed from scratch (the form ADR-1392 says the
    separable kernel must reproduce)."""
    h, w = f.shape
    out = np.zeros((h, w), np.int64)
    fl = f.astype(np.int64).tolist()
    for y in range(h):
        for x in range(w):
            acc = 32768
            for j in range(5):
                xx = _mirror_fold(x + j - 2, w)
                col = (1 << (bpc - 1))
                for k in range(5):
                    col += T[k] * fl[_mirror_fold(y + k - 2, h)][xx]
                acc += T[j] * (col >> bpc)
            out[y, x] = acc >> 16
    return out


def pin_brute_force_tiny(o):
    rng = np.random.default_rng(14)
    for bpc in (8, 10):
        for h in range(3, 10):
            for w in range(3, 10):
                f = rng.integers(0, 1 << bpc, size=(h, w)).astype(_dt(bpc))
                assert np.array_equal(o.blur(f, bpc).astype(np.int64),
                                      brute_force_blur(f, bpc)), (bpc, w, h)


def pin_sad_invariants(o):
    """SAD(a,a) = 0, SAD(a,b) = SAD(b,a), triangle inequality, and SAD equals the
    numpy sum of |a - b|."""
    rng = np.random.default_rng(15)
    for _ in range(10):
        a, b, c = (rng.integers(0, 65536, size=(7, 19)).astype(np.uint16) for _ in range(3))
        ab, ba = o.sad(a, b), o.sad(b, a)
        assert o.sad(a, a) == 0 and ab == ba
        assert o.sad(a, c) <= ab + o.sad(b, c)
        assert ab == int(np.abs(a.astype(np.int64) - b.astype(np.int64)).sum())


def pin_sequence(o):
    """SAD[0] = 0 and SAD[i] = sum |blur(F_i) - blur(F_{i-1})| (numpy sum)."""
    rng = np.random.default_rng(16)
    for bpc in (8, 10):
        seq = rng.integers(0, 1 << bpc, size=(5, 13, 21)).astype(_dt(bpc))
        sad = o.motion_sad_sequence(seq, bpc)
        assert sad[0] == 0
        for i in range(1, 5):
            d = o.blur(seq[i], bpc).astype(np.int64) - o.blur(seq[i - 1], bpc).astype(np.int64)
            assert int(sad[i]) == int(np.abs(d).sum())
        # symmetric in time: the reversed sequence has the same SADs, reversed
        rev = o.motion_sad_sequence(np.ascontiguousarray(seq[::-1]), bpc)
        assert np.array_equal(rev[1:], sad[1:][::-1])


def pin_sse(o):
    """SSE = k^2 N for dist = ref + k (no clipping); SSE(a,a) = 0; random planes
    equal the numpy int64 sum of squares, including 16-bit extremes."""
    rng = np.random.default_rng(17)
    for bpc in (8, 10, 16):
        hi = (1 << bpc) - 1
        for (w, h) in ((3, 3), (33, 17), (64, 48)):
            ref = rng.integers(0, hi - 9, size=(h, w)).astype(_dt(bpc))
            for k in (0, 1, 9):
                dist = (ref.astype(np.int64) + k).astype(_dt(bpc))
                assert o.sse(ref, dist, bpc) == k * k * w * h
                assert o.sse(dist, ref, bpc) == k * k * w * h
            a = rng.integers(0, hi + 1, size=(h, w)).astype(_dt(bpc))
            b = rng.integers(0, hi + 1, size=(h, w)).astype(_dt(bpc))
            e = a.astype(np.int64) - b.astype(np.int64)
            assert o.sse(a, b, bpc) == int((e * e).sum())
        full = np.full((5, 7), hi, _dt(bpc))
        zero = np.zeros((5, 7), _dt(bpc))
        assert o.sse(full, zero, bpc) == hi * hi * 35


def pin_scores(o):
    """score = SAD/256/(w h) in double; motion2_i = min(score_i, score_{i+1}),
    motion2_0 = 0 (score_0 = 0), motion2_{n-1} = score_{n-1}."""
    sad = np.array([0, 256 * 35 * 3, 256 * 35, 256 * 35 * 7], dtype=np.uint64)
    s, m2 = o.scores(sad, 7, 5)
    assert list(s) == [0.0, 3.0, 1.0, 7.0]
    assert list(m2) == [0.0, 1.0, 1.0, 7.0]
    s, m2 = o.scores(sad, 7, 5, next_score=2.0)
    assert list(m2) == [0.0, 1.0, 1.0, 2.0]
    # the division order is (SAD / 256) / (w h); /256 is exact in binary
    sad = np.array([0, 72587], dtype=np.uint64)
    s, _ = o.scores(sad, 6, 6)
    assert s[1] == (72587 / 256.0) / 36.0


# ------------------------------------------------------------------ moment sums
# ADR-1392 Decision 6: four accumulators per pair -- sum ref, sum dist, sum ref^2,
# sum dist^2 -- exact 64-bit integers (Context).

def pin_moment_closed_forms(o):
    """Constant planes c1 (ref), c2 (dist): sums c N and squares c^2 N.  A column
    ramp ref[y][x] = x (x < 2^bpc): sum = h w(w-1)/2, squares = h (w-1)w(2w-1)/6."""
    for bpc in (8, 10, 16):
        hi = (1 << bpc) - 1
        for (w, h) in ((1, 1), (3, 3), (17, 5), (64, 48)):
            n = w * h
            for c1, c2 in ((0, hi), (hi, hi), (7, 3)):
                r = np.full((h, w), c1, _dt(bpc))
                d = np.full((h, w), c2, _dt(bpc))
                assert list(o.moment_sums(r, d, bpc)) == [c1 * n, c2 * n, c1 * c1 * n, c2 * c2 * n]
        w, h = min(200, hi + 1), 7
        ramp = np.repeat(np.arange(w)[None, :], h, axis=0).astype(_dt(bpc))
        zero = np.zeros((h, w), _dt(bpc))
        s = o.moment_sums(ramp, zero, bpc)
        assert int(s[0]) == h * w * (w - 1) // 2 and int(s[1]) == 0
        assert int(s[2]) == h * (w - 1) * w * (2 * w - 1) // 6 and int(s[3]) == 0


def pin_moment_numpy(o):
    """Random planes (and a strided view) against numpy's uint64 sums."""
    rng = np.random.default_rng(21)
    for bpc in (8, 10, 16):
        for (w, h) in ((3, 3), (33, 17), (129, 40)):
            big = rng.integers(0, 1 << bpc, size=(2, h, w + 9)).astype(_dt(bpc))
            r, d = big[0][:, 4:4 + w], big[1][:, 2:2 + w]
            r64, d64 = r.astype(np.uint64), d.astype(np.uint64)
            exp = [r64.sum(), d64.sum(), (r64 * r64).sum(), (d64 * d64).sum()]
            assert [int(x) for x in o.moment_sums(r, d, bpc)] == [int(x) for x in exp], (bpc, w, h)


def pin_moments_from_sums(o):
    """The moments are the sums over the sample count, in double."""
    sums = np.array([[35 * 3, 35 * 200, 35 * 9, 35 * 40000], [1, 2, 3, 4]], np.uint64)
    m = o.moments(sums, 7, 5)
    assert list(m[0]) == [3.0, 200.0, 9.0, 40000.0]
    assert list(m[1]) == [1 / 35, 2 / 35, 3 / 35, 4 / 35]


# ------------------------------------------------------------------- motion_v2
# ADR-1392 Decision 4: stage prev - cur, vertical 5-tap pass rounded >> bpc, then
# the horizontal taps rounded >> 16; a right shift of a negative sum floors.

def pin_v2_equal_and_constant_frames(o):
    """prev == cur blurs to 0.  Constant prev c1, cur c2: the difference d = c1-c2
    is constant, the vertical pass gives floor((65536 d + 2^(bpc-1)) / 2^bpc) =
    d 2^(16-bpc) exactly (also for d < 0) and the horizontal pass keeps it, so
    SAD = |d| 2^(16-bpc) w h."""
    rng = np.random.default_rng(22)
    for bpc in (8, 10, 16):
        hi = (1 << bpc) - 1
        for (w, h) in ((3, 3), (11, 7)):
            f = rng.integers(0, hi + 1, size=(h, w)).astype(_dt(bpc))
            assert np.all(o.blur_diff(f, f, bpc) == 0)
            for c1, c2 in ((0, hi), (hi, 0), (5, 9), (9, 5)):
                p = np.full((h, w), c1, _dt(bpc))
                c = np.full((h, w), c2, _dt(bpc))
                d = c1 - c2
                assert np.all(o.blur_diff(p, c, bpc) == d * (1 << (16 - bpc))), (bpc, c1, c2)
                sad = o.motion_v2_sequence(np.stack([p, c]), bpc)
                assert int(sad[0]) == 0 and int(sad[1]) == abs(d) * (1 << (16 - bpc)) * w * h


def pin_v2_nonnegative_is_blur(o):
    """Where prev >= cur everywhere the difference is a valid frame and every sum
    is non-negative, so the difference blur equals the (separately pinned) blur
    of the frame prev - cur."""
    rng = np.random.default_rng(23)
    for bpc in (8, 10, 16):
        hi = (1 << bpc) - 1
        for (w, h) in ((3, 3), (8, 5), (40, 19)):
            cur = rng.integers(0, hi // 2, size=(h, w))
            prev = cur + rng.integers(0, hi // 2, size=(h, w))
            diff = (prev - cur).astype(_dt(bpc))
            got = o.blur_diff(prev.astype(_dt(bpc)), cur.astype(_dt(bpc)), bpc)
            assert np.array_equal(got.astype(np.int64), o.blur(diff, bpc).astype(np.int64)), (bpc, w, h)


def pin_v2_floor_impulse(o):
    """Impulse difference at an interior point, worked by hand for prev = 0 and
    cur = 128 there (8-bit), i.e. d = -128:
      row y0-2: -128*3571 + 128 = -456960 = -1785 * 256 exactly, so V = -1785
                (the blur of +128 gives (457088 + 128) >> 8 = 1786: the floor of
                a negative sum is not the negated positive result);
      row y0-1: -128*16004 + 128 = -2048384, / 256 = -8001.5, floor -8002;
      row y0:   -128*26386 + 128 = -3377280, / 256 = -13192.5, floor -13193;
      centre:   -13193*26386 + 32768 = -348077730, / 65536 = -5311.24, floor -5312.
    Every other output is 0; the 5x5 window is the outer form
    floor((floor((d t_{2+dy} + 2^(bpc-1)) / 2^bpc) t_{2+dx} + 2^15) / 2^16).
    The SAD of an impulse is not symmetric in time: d = +32 gives 8194 and
    d = -32 gives 8188 (the outer form summed)."""
    h, w, y0, x0 = 11, 13, 5, 6
    p = np.zeros((h, w), np.uint8)
    c = np.zeros((h, w), np.uint8)
    c[y0, x0] = 128
    b = o.blur_diff(p, c, 8).astype(np.int64)
    assert b[y0, x0] == -5312
    assert b[y0 - 2, x0] == (-1785 * 26386 + 32768) // 65536
    for bpc, d in ((8, -128), (8, 128), (8, -255), (10, -1023), (10, 37), (16, -65535), (16, 65535)):
        p = np.zeros((h, w), _dt(bpc))
        c = np.zeros((h, w), _dt(bpc))
        if d >= 0:
            p[y0, x0] = d
        else:
            c[y0, x0] = -d
        exp = np.zeros((h, w), np.int64)
        for dy in range(-2, 3):
            vert = (d * T[2 + dy] + (1 << (bpc - 1))) // (1 << bpc)
            for dx in range(-2, 3):
                exp[y0 + dy, x0 + dx] = (vert * T[2 + dx] + 32768) // 65536
        assert np.array_equal(o.blur_diff(p, c, bpc).astype(np.int64), exp), (bpc, d)
    imp = np.zeros((h, w), np.uint8)
    imp[y0, x0] = 32
    zero = np.zeros((h, w), np.uint8)
    assert int(o.motion_v2_sequence(np.stack([imp, zero]), 8)[1]) == 8194
    assert int(o.motion_v2_sequence(np.stack([zero, imp]), 8)[1]) == 8188


def brute_force_blur_diff(p: np.ndarray, c: np.ndarray, bpc: int) -> np.ndarray:
    """Per-output 25-MAC loop over the signed difference with floor division
    (Python's // floors), the vertical value recomputed for every horizontal tap."""
    h, w = p.shape
    dl = (p.astype(np.int64) - c.astype(np.int64)).tolist()
    out = np.zeros((h, w), np.int64)
    for y in range(h):
        for x in range(w):
            acc = 32768
            for j in range(5):
                xx = _mirror_fold(x + j - 2, w)
                col = 1 << (bpc - 1)
                for k in range(5):
                    col += T[k] * dl[_mirror_fold(y + k - 2, h)][xx]
                acc += T[j] * (col // (1 << bpc))
            out[y, x] = acc // 65536
    return out


def pin_v2_brute_force_tiny(o):
    rng = np.random.default_rng(24)
    for bpc in (8, 10, 16):
        for h in range(3, 9):
            for w in range(3, 9):
                p = rng.integers(0, 1 << bpc, size=(h, w)).astype(_dt(bpc))
                c = rng.integers(0, 1 << bpc, size=(h, w)).astype(_dt(bpc))
                assert np.array_equal(o.blur_diff(p, c, bpc).astype(np.int64),
                                      brute_force_blur_diff(p, c, bpc)), (bpc, w, h)


def pin_v2_sequence(o):
    """SAD[0] = 0 and SAD[i] = sum |blur_diff(F_{i-1}, F_i)| (numpy sum)."""
    rng = np.random.default_rng(25)
    for bpc in (8, 10):
        seq = rng.integers(0, 1 << bpc, size=(5, 9, 14)).astype(_dt(bpc))
        sad = o.motion_v2_sequence(seq, bpc)
        assert sad[0] == 0
        for i in range(1, 5):
            assert int(sad[i]) == int(np.abs(o.blur_diff(seq[i - 1], seq[i], bpc).astype(np.int64)).sum())


ALL_PINS = [pin_mirror, pin_constant_frames, pin_two_constant_sad_and_score,
            pin_impulse_interior, pin_hand_worked_6x6, pin_row_constant,
            pin_column_constant, pin_scipy_separable, pin_brute_force_tiny,
            pin_sad_invariants, pin_sequence, pin_sse, pin_scores,
            pin_moment_closed_forms, pin_moment_numpy, pin_moments_from_sums,
            pin_v2_equal_and_constant_frames, pin_v2_nonnegative_is_blur,
            pin_v2_floor_impulse, pin_v2_brute_force_tiny, pin_v2_sequence]
