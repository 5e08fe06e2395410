"""Pins of the oracle's FFN stages: closed forms, brute force, invariants and
library special cases, each chosen so a plausible slip (a dropped term, a
swapped operand, a transposed scale, an off-by-one row) fails one of them."""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from oracle import (bf16_decode, bf16_encode, combine, e4m3_decode, e4m3_encode,
                    gemm_block_scaled, gemm_contig, gemm_masked, permute, quant_1x128,
                    quant_128x128, swiglu, swiglu_quant)

RNG = np.random.default_rng(1234)
FLOOR_SCALE = np.float32(np.float32(1e-4) / np.float32(448.0))


def _bf16(x):
    return bf16_decode(bf16_encode(x)).astype(np.float32)


# ----------------------------------------------------------------------------- quant
def test_quant_zero_block_uses_floor_scale():
    x = np.zeros((3, 256), np.float32)
    x[1, 128:] = RNG.standard_normal(128)
    q, s = quant_1x128(x)
    assert s.shape == (2, 3)
    assert s[0, 0] == FLOOR_SCALE and s[1, 0] == FLOOR_SCALE and s[0, 1] == FLOOR_SCALE
    assert (q[0] == 0).all() and (q[1, :128] == 0).all()


def test_quant_amax_maps_to_448():
    x = _bf16(RNG.standard_normal((4, 384)))
    x[2, 130] = 9.0
    x[3, 300] = -9.0
    q, s = quant_1x128(x)
    assert q[2, 130] == 0x7E and q[3, 300] == 0xFE
    assert s[1, 2] == np.float32(np.float32(9.0) / np.float32(448.0))
    # every block holds its own max |x| -> exactly one code of magnitude 0x7E per block
    assert ((q.reshape(4, 3, 128) & 0x7F) == 0x7E).any(axis=2).all()


def test_quant_power_of_two_scale_is_exact():
    # amax = 448 * 2^-5 -> s = 2^-5 exactly; inputs on the E4M3 grid times 2^-5
    # must come back bit-exactly.
    codes = RNG.integers(0, 0x7F, size=(2, 256)).astype(np.uint8) | (RNG.integers(0, 2, (2, 256)) << 7).astype(np.uint8)
    codes[:, 0] = 0x7E
    codes[:, 128] = 0xFE
    x = (e4m3_decode(codes) * 2.0 ** -5).astype(np.float32)
    q, s = quant_1x128(x)
    assert (s == np.float32(2.0 ** -5)).all()
    assert np.array_equal(e4m3_decode(q), e4m3_decode(codes))


def test_quant_error_bound_and_layout():
    M, K = 37, 640
    x = _bf16(RNG.standard_normal((M, K)) * np.exp(RNG.uniform(-6, 6, (M, 1))))
    q, s = quant_1x128(x)
    assert s.shape == (K // 128, M)
    # scale layout: s[kb, m] is row m's block kb
    amax = np.abs(x.reshape(M, K // 128, 128)).max(axis=2)
    assert np.array_equal(s, (np.maximum(amax, np.float32(1e-4)) / np.float32(448)).astype(np.float32).T)
    deq = e4m3_decode(q) * np.repeat(s.T, 128, axis=1)
    err = np.abs(deq - x)
    # half an E4M3 ulp: 2^-4 relative for normals, 2^-10 * s absolute below 2^-6 * s
    bound = np.maximum(np.abs(x) * 2.0 ** -4, np.repeat(s.T, 128, axis=1) * 2.0 ** -10) * (1 + 1e-6)
    assert (err <= bound).all()


def _smallest_pow2_exponent(a: float) -> int:
    """Brute force with exact rationals: the smallest e with a <= 448 * 2^e."""
    from fractions import Fraction
    fa = Fraction(float(a))
    e = -200
    while fa > 448 * Fraction(2) ** e:
        e += 1
    return e


def test_ue8m0_scale_is_the_smallest_power_of_two():
    # amax over a wide exponent range, with the exact boundaries 448 * 2^j and
    # their float32 neighbours, the 1e-4 floor and values below it
    j = np.arange(-30, 40)
    edges = (448.0 * np.exp2(j)).astype(np.float32)
    amax = np.concatenate([edges, np.nextafter(edges, np.float32(np.inf)),
                           np.nextafter(edges, np.float32(0)),
                           np.exp2(RNG.uniform(-30, 40, 300)).astype(np.float32),
                           np.float32([0.0, 1e-30, 1e-4, 2e-4])])
    x = np.zeros((amax.size, 128), np.float32)
    x[:, 5] = amax
    x[:, 9] = -amax / 2
    q, s, byte = oracle.quant_1x128_ue8m0(x)
    for r, a in enumerate(amax):
        e = _smallest_pow2_exponent(max(float(a), float(np.float32(1e-4))))
        assert s[0, r] == np.float32(2.0 ** e), (a, s[0, r], e)
        assert int(byte[0, r]) == e + 127
    # the block maximum never saturates and lands in the top binade of E4M3
    big = amax >= np.float32(1e-4)
    top = e4m3_decode(q[big, 5])
    assert (top <= 448.0).all() and (top >= 224.0).all()


def test_quant_non_finite_inputs():
    # A reading for inputs the pages never mention: NaN elements take no part in
    # the block maximum (IEEE maxNum, as a hardware fmax reduction) and encode to
    # the NaN code 0x7F; a block of NaNs has maximum 0 (floor scale); an infinite
    # element gives s = inf (UE8M0 byte 0xFF), so the finite elements of its block
    # become signed zeros and the infinite one NaN (inf / inf).
    x = np.zeros((4, 256), np.float32)
    x[0, :128] = _bf16(RNG.standard_normal(128))
    x[0, 7] = np.nan
    x[1, :128] = np.nan
    x[2, :128] = _bf16(RNG.standard_normal(128))
    x[2, 5], x[2, 6], x[2, 8] = np.inf, -3.0, 2.5
    x[3, 200], x[3, 201], x[3, 202] = -np.inf, 1.0, -1.0
    clean = x[0].copy()
    clean[7] = 0.0
    floors = {quant_1x128: FLOOR_SCALE, oracle.quant_1x128_ue8m0: np.float32(2.0 ** -22)}
    for fn, floor in floors.items():
        res = fn(x)
        q, s = res[0], res[1]
        qc, sc = fn(clean[None])[:2]
        assert s[0, 0] == sc[0, 0] and np.isfinite(s[0, 0])
        assert q[0, 7] == 0x7F and np.array_equal(np.delete(q[0, :128], 7), np.delete(qc[0, :128], 7))
        assert s[0, 1] == floor and (q[1, :128] == 0x7F).all()
        assert np.isinf(s[0, 2]) and q[2, 5] == 0x7F and q[2, 6] == 0x80 and q[2, 8] == 0x00
        assert np.isinf(s[1, 3]) and q[3, 200] == 0x7F and q[3, 201] == 0x00 and q[3, 202] == 0x80
        assert np.isfinite(s[1, 2]) and np.isfinite(s[0, 3])   # the other blocks are unaffected
    byte = oracle.quant_1x128_ue8m0(x)[2]
    assert byte[0, 2] == 255 and byte[1, 3] == 255 and byte[0, 1] == 127 - 22
    # a 128x128 weight tile: the same rules over the tile
    w = np.zeros((128, 256), np.float32)
    w[3, 3], w[9, 10] = np.nan, -2.0
    w[100, 200] = np.inf
    qw, sw = quant_128x128(w)
    assert sw[0, 0] == np.float32(np.float32(2.0) / np.float32(448.0)) and qw[3, 3] == 0x7F
    assert qw[9, 10] == 0xFE and np.isinf(sw[0, 1]) and qw[100, 200] == 0x7F
    _, swe, bwe = oracle.quant_128x128_ue8m0(w)
    assert swe[0, 0] == np.float32(2.0 ** -7) and bwe[0, 1] == 255


def test_ue8m0_codes_are_the_bruteforce_encoding_of_x_over_s():
    # blocks whose maximum is 448 * 2^j: s = 2^j exactly and every element's code
    # is the brute-force nearest E4M3 of x / 2^j
    allv = bf16_decode(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    vals = allv[np.isfinite(allv) & (np.abs(allv) <= 448.0)].astype(np.float32)
    for jexp in (-9, 0, 5):
        scale = np.float32(2.0 ** jexp)
        v = vals * scale
        nb = -(-v.size // 127)
        blocks = np.zeros((nb, 128), np.float32)
        blocks[:, 0] = np.float32(448.0) * scale
        flat = np.zeros(nb * 127, np.float32)
        flat[:v.size] = v
        blocks[:, 1:] = flat.reshape(nb, 127)
        q, s, _ = oracle.quant_1x128_ue8m0(blocks)
        assert (s == scale).all()
        ref = oracle.e4m3_encode_bruteforce(blocks.astype(np.float64) / float(scale))
        assert np.array_equal(q, ref)
        assert (q[:, 0] == 0x7E).all()


def test_ue8m0_against_fp32_scales():
    # the power-of-two scale is the fp32 scale rounded up to a power of two
    # (never below it, less than twice it), and both dequantise within the
    # E4M3 rounding bound of x: half a step, 2^-4 relative for normal codes,
    # 2^-10 * s absolute below the normal range
    x = (RNG.standard_normal((64, 1024)) * np.exp2(RNG.integers(-6, 6, (64, 1))) ).astype(np.float32)
    x = bf16_decode(bf16_encode(x)).astype(np.float32)
    q32, s32 = quant_1x128(x)
    q8, s8, _ = oracle.quant_1x128_ue8m0(x)
    assert (s8 >= s32).all() and (s8 < 2 * s32).all()
    for q, s in ((q32, s32), (q8, s8)):
        sc = np.repeat(s.T, 128, axis=1).astype(np.float64)
        deq = e4m3_decode(q) * sc
        err = np.abs(deq - x)
        assert (err <= np.abs(x) * 2.0 ** -4 + sc * 2.0 ** -10 + 1e-30).all()


def test_ue8m0_weight_tiles():
    # 128x128 tiles with UE8M0 scales: each tile's scale is the smallest power
    # of two for its own maximum (brute force), tiles are independent, and the
    # codes are the brute-force encoding of w / s
    w = (RNG.standard_normal((256, 384)) * np.exp2(RNG.integers(-8, 8, (2, 1, 3, 1)))
         .repeat(128, 1).reshape(2, 128, 3, 1).repeat(128, 3).reshape(256, 384)).astype(np.float32)
    q, s, byte = oracle.quant_128x128_ue8m0(w)
    for nb in range(2):
        for kb in range(3):
            tile = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            e = _smallest_pow2_exponent(max(float(np.abs(tile).max()), float(np.float32(1e-4))))
            assert s[nb, kb] == np.float32(2.0 ** e) and int(byte[nb, kb]) == e + 127
            ref = oracle.e4m3_encode_bruteforce(tile.astype(np.float64) / 2.0 ** e)
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128], ref)


def test_ue8m0_gemm_within_tolerance_of_the_fp32_scale_gemm():
    # tolerance-only parity between the two readings of the input scales: the
    # block-scaled GEMM with UE8M0 activation scales stays as close to the exact
    # float64 product as the fp32-scale one, up to the factor the coarser
    # scale grid allows (a power of two wastes under one bit of E4M3 range)
    rng = np.random.default_rng(99)
    x = (rng.standard_normal((96, 512)) * np.exp2(rng.integers(-3, 4, (96, 4))).repeat(128, 1)).astype(np.float32)
    x = bf16_decode(bf16_encode(x)).astype(np.float32)
    w = bf16_decode(bf16_encode(rng.standard_normal((256, 512)) / np.sqrt(512))).astype(np.float32)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    qb, sb = quant_128x128(w)
    qa32, sa32 = quant_1x128(x)
    qa8, sa8, _ = oracle.quant_1x128_ue8m0(x)
    rel = lambda y: np.sqrt(np.mean((y - exact) ** 2) / np.mean(exact ** 2))
    e32 = rel(gemm_block_scaled(qa32, sa32, qb, sb))
    e8 = rel(gemm_block_scaled(qa8, sa8, qb, sb))
    assert 0 < e32 < 0.05 and 0 < e8 < 0.05
    assert e8 < 2.0 * e32
    # the two readings differ by quantisation noise, far beyond the bf16-level
    # GEMM tolerance: parity between them is at this level only
    d8, d32 = gemm_block_scaled(qa8, sa8, qb, sb), gemm_block_scaled(qa32, sa32, qb, sb)
    assert 0 < np.sqrt(np.mean((d8 - d32) ** 2) / np.mean(d32 ** 2)) < e8 + e32


def test_quant_128x128_tiles_are_independent():
    w = _bf16(RNG.standard_normal((256, 384)) * 0.05)
    q, s = quant_128x128(w)
    assert s.shape == (2, 3)
    w2 = w.copy()
    w2[130, 260] = 7.0                       # tile (1, 2)
    q2, s2 = quant_128x128(w2)
    changed = s2 != s
    assert changed[1, 2] and changed.sum() == 1
    assert q2[130, 260] == 0x7E
    assert np.array_equal(q2[:128], q[:128]) and np.array_equal(q2[:, :256], q[:, :256])
    # tile amax definition
    tiles = np.abs(w.reshape(2, 128, 3, 128)).max(axis=(1, 3))
    assert np.array_equal(s, (np.maximum(tiles, np.float32(1e-4)) / np.float32(448)).astype(np.float32))


# ----------------------------------------------------------------------------- permute
def _permute_bruteforce(ids, eb, E, layout, max_m, align=128):
    T, k = ids.shape
    per = {e: [] for e in range(E)}
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j]) - eb
            if 0 <= e < E:
                per[e].append(t * k + j)
    dst = [-1] * (T * k)
    if layout == "masked":
        for e in range(E):
            for r, i in enumerate(per[e]):
                if r < max_m:
                    dst[i] = e * max_m + r
        return [min(len(per[e]), max_m) for e in range(E)], dst
    row = 0
    for e in range(E):
        for r, i in enumerate(per[e]):
            dst[i] = row + r
        row += -(-len(per[e]) // align) * align
    return [len(per[e]) for e in range(E)], dst


@pytest.mark.parametrize("layout", ["masked", "contig"])
def test_permute_matches_bruteforce(layout):
    for trial in range(5):
        T, k, E, eb = 50, 3, 5, 2
        ids = RNG.integers(0, 9, (T, k)).astype(np.int32)
        max_m = 16
        p = permute(ids, eb, E, layout, max_m=max_m, align=8)
        counts, dst = _permute_bruteforce(ids, eb, E, layout, max_m, align=8)
        assert list(p["counts"]) == counts
        assert list(p["dst_row"]) == dst


def test_permute_invariants_and_gather():
    T, k, E, K = 40, 2, 4, 256
    ids = np.stack([RNG.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    q = RNG.integers(0, 256, (T, K)).astype(np.uint8)
    s = RNG.random((K // 128, T)).astype(np.float32)
    for layout in ("masked", "contig"):
        p = permute(ids, 0, E, layout, max_m=64, q=q, s=s)
        assert p["counts"].sum() == T * k                     # all assignments local
        dst, src = p["dst_row"], p["row_src"]
        assert (src[dst] == np.arange(T * k)).all()            # mutually inverse
        assert (np.sort(dst) == np.sort(np.nonzero(src >= 0)[0])).all()
        for i in range(T * k):
            assert np.array_equal(p["q"][dst[i]], q[i // k])
        if layout == "masked":
            for i in range(T * k):
                e, r = divmod(dst[i], 64)
                assert np.array_equal(p["s"][e, :, r], s[:, i // k])
        else:
            assert (p["offsets"] % 128 == 0).all()
            assert np.array_equal(p["s"][:, dst], s[:, np.arange(T * k) // k])
            mi = p["m_indices"]
            for e in range(E):
                seg = mi[p["offsets"][e]:p["offsets"][e + 1]]
                assert (seg[:p["counts"][e]] == e).all() and (seg[p["counts"][e]:] == -1).all()


def test_permute_masked_overflow_and_nonlocal():
    ids = np.array([[0, 5], [0, 1], [0, 7], [0, 1]], np.int32)  # expert 0 gets 4 > max_m=2
    p = permute(ids, 0, 2, "masked", max_m=2)
    assert p["overflow"] and list(p["counts"]) == [2, 2] and list(p["raw_counts"]) == [4, 2]
    assert list(p["dst_row"]) == [0, -1, 1, 2, -1, -1, -1, 3]


# ----------------------------------------------------------------------------- GEMM
def _rand_codes(shape):
    c = RNG.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3A                              # no NaN codes
    return c


def test_gemm_integer_exact_closed_form():
    # integers in [-16, 16] are exact in E4M3; with unit scales the result is the
    # integer matmul.
    M, N, K = 19, 256, 384
    a = RNG.integers(-16, 17, (M, K))
    b = RNG.integers(-16, 17, (N, K))
    qa, qb = e4m3_encode(a.astype(np.float64)), e4m3_encode(b.astype(np.float64))
    assert np.array_equal(e4m3_decode(qa), a)
    D = gemm_block_scaled(qa, np.ones((K // 128, M), np.float32), qb, np.ones((N // 128, K // 128), np.float32))
    assert np.array_equal(D, (a @ b.T).astype(np.float64))


def test_gemm_bruteforce_triple_loop():
    M, N, K = 3, 256, 256
    qa, qb = _rand_codes((M, K)), _rand_codes((N, K))
    sa = RNG.random((K // 128, M)).astype(np.float32) + 0.5
    sb = RNG.random((N // 128, K // 128)).astype(np.float32) + 0.5
    D = gemm_block_scaled(qa, sa, qb, sb)
    A, B = e4m3_decode(qa), e4m3_decode(qb)
    for m in range(M):
        for n in range(0, N, 37):
            ref = 0.0
            for k in range(K):
                ref += float(sa[k // 128, m]) * float(sb[n // 128, k // 128]) * A[m, k] * B[n, k]
            assert abs(D[m, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_gemm_matches_dequantised_matmul():
    M, N, K = 33, 384, 512                                   # KB != NB != M/128: transposes show
    qa, qb = _rand_codes((M, K)), _rand_codes((N, K))
    sa = (RNG.random((K // 128, M)) * 4).astype(np.float32)
    sb = (RNG.random((N // 128, K // 128)) * 4).astype(np.float32)
    D = gemm_block_scaled(qa, sa, qb, sb)
    A = e4m3_decode(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    B = e4m3_decode(qb) * np.kron(sb.astype(np.float64), np.ones((128, 128)))
    ref = A @ B.T
    assert np.allclose(D, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gemm_masked_and_contig_wrappers():
    E, max_m, N, K = 3, 8, 128, 256
    qa, qb = _rand_codes((E, max_m, K)), _rand_codes((E, N, K))
    sa = RNG.random((E, K // 128, max_m)).astype(np.float32)
    sb = RNG.random((E, N // 128, K // 128)).astype(np.float32)
    counts = np.array([8, 0, 3])
    D, valid = gemm_masked(qa, sa, qb, sb, counts)
    assert valid.sum() == 11 and not valid[1].any() and valid[2, :3].all() and not valid[2, 3:].any()
    ref = bf16_encode(gemm_block_scaled(qa[2, :3], sa[2][:, :3], qb[2], sb[2]))
    assert np.array_equal(D[2, :3], ref)
    # contiguous: same rows laid out with padding to 8
    offsets = np.array([0, 8, 8, 16])
    mi = np.array([0] * 8 + [2] * 3 + [-1] * 5)
    qa_c = np.concatenate([qa[0], qa[2]])
    sa_c = np.concatenate([sa[0], sa[2]], axis=1)
    Dc, vc = gemm_contig(qa_c, sa_c, qb, sb, offsets, mi)
    assert np.array_equal(Dc[:8], D[0]) and np.array_equal(Dc[8:11], D[2, :3]) and vc.sum() == 11


# ----------------------------------------------------------------------------- SwiGLU
def test_swiglu_matches_scipy_expit_and_gate_up_order():
    rows, I = 5, 256
    y = _bf16(RNG.standard_normal((rows, 2 * I)) * 3)
    bits = bf16_encode(y.astype(np.float64))
    h = swiglu(bits)
    g, u = y[:, :I].astype(np.float64), y[:, I:].astype(np.float64)
    assert np.array_equal(h, (g * expit(g) * u).astype(np.float32)) or \
        np.max(np.abs(h - g * expit(g) * u) / (np.abs(g * expit(g) * u) + 1e-30)) < 2 ** -23
    # order: gate first.  silu(30) * 1 ~ 30, silu(1) * 30 ~ 21.9
    t = bf16_encode(np.array([[30.0, 1.0]]))
    assert abs(swiglu(t)[0, 0] - 30.0) < 1e-6
    t = bf16_encode(np.array([[0.0, 5.0, -3.0, 0.0]]))
    assert list(swiglu(t)[0]) == [0.0, 0.0]


def test_swiglu_quant_is_quant_of_swiglu():
    y = bf16_encode(RNG.standard_normal((6, 512)))
    q, s = swiglu_quant(y)
    q2, s2 = quant_1x128(swiglu(y))
    assert np.array_equal(q, q2) and np.array_equal(s, s2) and s.shape == (2, 6)


# ----------------------------------------------------------------------------- combine
def test_combine_constant_rows_and_weights_sum_to_one():
    T, k, H = 16, 4, 256
    w = RNG.random((T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    c = _bf16(RNG.standard_normal(H))
    y2 = np.tile(bf16_encode(c.astype(np.float64)), (T * k, 1))
    dst = RNG.permutation(T * k)
    out = combine(y2, dst, w)
    assert np.array_equal(bf16_decode(out), np.tile(c, (T, 1)).astype(np.float64)) or \
        np.abs(bf16_decode(out) - c).max() <= 2 ** -8 * np.abs(c).max()


def test_combine_single_choice_is_a_gather_and_skips_dropped():
    T, H = 10, 128
    y2 = bf16_encode(RNG.standard_normal((20, H)))
    dst = RNG.permutation(20)[:T]
    out = combine(y2, dst, np.ones((T, 1), np.float32))
    assert np.array_equal(out, y2[dst])
    dst2 = dst.copy()
    dst2[3] = -1
    out2 = combine(y2, dst2, np.ones((T, 1), np.float32))
    assert (bf16_decode(out2[3]) == 0).all() and np.array_equal(out2[4:], y2[dst[4:]])


def test_combine_bruteforce():
    T, k, H = 6, 3, 128
    y2 = bf16_encode(RNG.standard_normal((T * k + 2, H)))
    dst = RNG.permutation(T * k + 2)[:T * k]
    dst[4] = -1
    w = RNG.random((T, k)).astype(np.float32)
    out = bf16_decode(combine(y2, dst, w))
    Y = bf16_decode(y2)
    for t in range(T):
        ref = np.zeros(H)
        for j in range(k):
            if dst[t * k + j] >= 0:
                ref += float(w[t, j]) * Y[dst[t * k + j]]
        assert np.array_equal(out[t], bf16_decode(bf16_encode(ref)))


def test_combine_shared_row_and_accumulate():
    # the shared expert's row at weight 1 equals one more routing slot of weight
    # 1 (same float64 steps); accumulating into an output adds its values; with
    # no slot and no shared row, accumulation leaves the output as it was; brute
    # force on a small case
    T, k, H, rows = 6, 3, 16, 10
    y = bf16_encode(RNG.standard_normal((rows, H)))
    sh = bf16_encode(RNG.standard_normal((T, H)))
    old = bf16_encode(RNG.standard_normal((T, H)))
    dst = RNG.integers(-1, rows, (T, k))
    w = RNG.uniform(0, 1, (T, k)).astype(np.float32)
    y_ext = np.concatenate([y, sh])
    dst_ext = np.concatenate([dst, rows + np.arange(T)[:, None]], axis=1)
    w_ext = np.concatenate([w, np.ones((T, 1), np.float32)], axis=1)
    assert np.array_equal(combine(y, dst.reshape(-1), w, shared_bits=sh),
                          combine(y_ext, dst_ext.reshape(-1), w_ext))
    none = -np.ones((T, k), np.int64)
    assert np.array_equal(combine(y, none.reshape(-1), w, out_bits=old), old)
    got = bf16_decode(combine(y, dst.reshape(-1), w, shared_bits=sh, out_bits=old))
    yd, sd, od = bf16_decode(y), bf16_decode(sh), bf16_decode(old)
    for t in range(T):
        for h in range(H):
            acc = od[t, h]
            for j in range(k):
                if dst[t, j] >= 0:
                    acc += float(w[t, j]) * yd[dst[t, j], h]
            acc += sd[t, h]
            assert got[t, h] == bf16_decode(bf16_encode(np.array([acc])))[0]


# ----------------------------------------------------------------------------- UE8M0 packing
# The packed layouts are pinned against the two placement rules measured on the
# tensor cores (not against their own formula):
#  copy rule: a 32 x 16-byte shared-memory source goes to TMEM lanes i, 32+i,
#    64+i, 96+i, columns 0..3 (row i -> its 4 words); with a core-matrix stride
#    of 0 the 8-row core matrix repeats, so lane i takes source row i % 8;
#  read rule: the MMA takes row m of A from lane m, column m // 32, and column n
#    of B from lane n % 32, column n // 32; the scale-factor id picks the byte.
def _tmem_after_copy(src_words, repeat8=False):
    """[128 lanes, 4 columns] after one copy of a 512-byte (or 128-byte) source."""
    w = np.asarray(src_words, np.uint32).reshape(-1, 4)
    return np.array([w[(lane % 32) % 8] if repeat8 else w[lane % 32] for lane in range(128)])


def test_ue8m0_act_packing_meets_the_tensor_core_placement():
    rng = np.random.default_rng(3)
    for G, rows, KB in ((128, 128, 8), (300, 900, 5), (16, 64, 2)):
        groups = -(-rows // G)
        e = rng.integers(-30, 30, (groups, KB, G))
        s = np.exp2(e.astype(np.float64)).astype(np.float32)
        words = oracle.pack_ue8m0_act(s, G, rows)
        KG, NC = -(-KB // 4), -(-G // 128)
        assert words.size == groups * KG * NC * 128
        for grp in range(groups):
            for g in range(KG):
                for c in range(NC):
                    chunk = words[((grp * KG + g) * NC + c) * 128:((grp * KG + g) * NC + c + 1) * 128]
                    tm = _tmem_after_copy(chunk)
                    for m in range(128):
                        r = c * 128 + m                     # row of the group
                        word = int(tm[m, m // 32])          # what the MMA reads for row m
                        for sf_id in range(4):
                            kb = 4 * g + sf_id
                            byte = (word >> (8 * sf_id)) & 0xFF
                            if r < G and grp * G + r < rows and kb < KB:
                                assert byte == e[grp, kb, r] + 127
                            else:
                                assert byte == 0x7F


def test_ue8m0_weight_packing_meets_the_tensor_core_placement():
    rng = np.random.default_rng(4)
    E, NB, KB = 3, 2, 6
    e = rng.integers(-20, 20, (E, NB, KB))
    words = oracle.pack_ue8m0_weight(np.exp2(e.astype(np.float64)).astype(np.float32))
    KG = -(-KB // 4)
    assert words.size == E * NB * KG * 32
    for ex in range(E):
        for g in range(KG):
            # a 256-column tile: block 0's record to columns 0..3, block 1's to 4..7
            cols = np.concatenate([_tmem_after_copy(words[((ex * NB + nb) * KG + g) * 32:
                                                          ((ex * NB + nb) * KG + g + 1) * 32], repeat8=True)
                                   for nb in range(NB)], axis=1)
            for n in range(NB * 128):
                word = int(cols[n % 32, n // 32])
                for sf_id in range(4):
                    kb = 4 * g + sf_id
                    byte = (word >> (8 * sf_id)) & 0xFF
                    assert byte == (e[ex, n // 128, kb] + 127 if kb < KB else 0x7F)
