"""The stages of the routed-expert FP8 FFN, written as plain definitions
(test infrastructure only).

Array conventions (all numpy):

* FP8 tensors are uint8 E4M3 codes; bf16 tensors are uint16 bit patterns.
* Activation scales are "packed" MN-major: ``s[kb, m]`` is the fp32 scale of
  row ``m``'s 128-column block ``kb`` (one contiguous fp32 vector per k-block,
  the layout a TMA-fed GEMM epilogue reads).  Masked layout: ``s[e, kb, m]``.
* Weights are stored K-major, ``w[e, n, k]``; their scales are ``sw[e, nb, kb]``
  for the 128x128 block (nb, kb).  W13 stacks the gate rows [0, I) above the
  up rows [I, 2I) (a reading: the problem statement names W1 and W3 but not
  their order in one operand).

Citations: the FP8 GEMM with quantised and packed input scales is the
DeepGEMM bullet of "Deploying DeepSeek on GB200 NVL72 with PD and Large Scale
EP (Part I)", section "Implementation details"; the two grouped layouts are the
prefill/decode grouped-GEMM pair of "Deploying DeepSeek with PD Disaggregation
and Large-Scale Expert Parallelism on 96 H100 GPUs", section "DeepGEMM
integration".  The formulas below are this library's problem statement; the
readings taken where it is silent are named where they apply.
"""
from __future__ import annotations

import numpy as np

from .fp8 import E4M3_MAX, bf16_decode, bf16_encode, e4m3_decode, e4m3_encode

BLOCK = 128
# Reading: the pages give no formula for the scale; amax/448 is plain FP8-max
# scaling and the floor keeps all-zero blocks finite.
SCALE_FLOOR = np.float32(1e-4)


def _block_amax(blocks: np.ndarray, axis) -> np.ndarray:
    """max |x| over a block (exact in float32).  A reading for non-finite inputs,
    which the pages never mention: NaN elements take no part in the maximum
    (IEEE maxNum, what a hardware fmax reduction does), so a block whose
    elements are all NaN has maximum 0; an infinite element makes it inf."""
    with np.errstate(invalid="ignore"):
        a = np.fmax.reduce(np.abs(blocks), axis=axis)
    return np.where(np.isnan(a), np.float32(0.0), a).astype(np.float32)


def _block_scale(amax_f32: np.ndarray) -> np.ndarray:
    """s = float32(max(amax, 1e-4) / 448): one correctly rounded float32 division
    (an infinite maximum gives s = inf, and then x / s is 0 or NaN)."""
    a = np.fmax(amax_f32.astype(np.float32), SCALE_FLOOR)
    return (a / np.float32(E4M3_MAX)).astype(np.float32)


def quant_1x128(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-row 1x128 E4M3 quantisation.

    x: [M, K] float32 values (bf16 inputs decoded exactly), K % 128 == 0.
    Per row m and 128-column block kb: amax = max |x| (exact in float32);
    s = fp32(max(amax, 1e-4) / 448); q = e4m3(fp32(x / s)) -- a float32
    division, correctly rounded (a reading: divide, not multiply by 1/s).
    Returns q [M, K] uint8 and s [K/128, M] float32 (MN-major).
    """
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % BLOCK == 0
    blocks = x.reshape(M, K // BLOCK, BLOCK)
    amax = _block_amax(blocks, 2)                            # [M, KB]
    s = _block_scale(amax)                                   # [M, KB]
    with np.errstate(invalid="ignore"):
        y = (blocks / s[:, :, None]).astype(np.float32)      # float32 IEEE division
    q = e4m3_encode(y.astype(np.float64)).reshape(M, K)
    return q, np.ascontiguousarray(s.T)


def _block_scale_ue8m0(amax_f32: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Power-of-two scale of the other reading of "packed" input scales (UE8M0:
    an unsigned 8-bit exponent, s = 2^(byte - 127)): the smallest power of two
    s with max(amax, 1e-4) / s <= 448, i.e. s = 2^ceil(log2(max(amax, 1e-4) / 448)).
    The exponent is found by exact comparisons of a against 448 * 2^e (both
    exact in float64), not by a rounded logarithm.  An infinite maximum has no
    such power of two: it gives s = inf and the byte 0xFF (the all-ones UE8M0
    exponent), so that x / s is 0 or NaN as with the float32 scale.
    Returns (s float32, byte uint8)."""
    a = np.fmax(amax_f32.astype(np.float32), SCALE_FLOOR).astype(np.float64)
    inf = np.isinf(a)
    a = np.where(inf, 1.0, a)
    e = np.ceil(np.log2(a / E4M3_MAX)).astype(np.int64)          # estimate, then make exact
    e = np.where(a > E4M3_MAX * np.exp2(e.astype(np.float64)), e + 1, e)
    e = np.where(a <= E4M3_MAX * np.exp2((e - 1).astype(np.float64)), e - 1, e)
    s = np.where(inf, np.inf, np.exp2(e.astype(np.float64))).astype(np.float32)
    return s, np.where(inf, 255, e + 127).astype(np.uint8)


def quant_1x128_ue8m0(x) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """1x128 E4M3 quantisation with power-of-two (UE8M0) block scales -- the
    alternative reading of the DeepGEMM bullet's "packing of the input scales"
    (the hardware block-scaled MMA consumes such scales).  Per row and block:
    s = _block_scale_ue8m0(amax); q = e4m3(x / s), the quotient exact (a division
    by a power of two).  Returns q [M, K] uint8, s [K/128, M] float32 and the
    UE8M0 bytes [K/128, M] uint8 (s = 2^(byte - 127))."""
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % BLOCK == 0
    blocks = x.reshape(M, K // BLOCK, BLOCK)
    amax = _block_amax(blocks, 2)
    s, byte = _block_scale_ue8m0(amax)
    with np.errstate(invalid="ignore"):
        y = blocks.astype(np.float64) / s[:, :, None].astype(np.float64)   # exact
    q = e4m3_encode(y).reshape(M, K)
    return q, np.ascontiguousarray(s.T), np.ascontiguousarray(byte.T)


def quant_128x128(w) -> tuple[np.ndarray, np.ndarray]:
    """128x128 block E4M3 quantisation of a K-major weight [N, K] (float32 values):
    the same rule as ``quant_1x128`` with amax over the whole tile.
    Returns q [N, K] uint8 and s [N/128, K/128] float32."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert N % BLOCK == 0 and K % BLOCK == 0
    tiles = w.reshape(N // BLOCK, BLOCK, K // BLOCK, BLOCK)
    amax = _block_amax(tiles, (1, 3))                       # [NB, KB]
    s = _block_scale(amax)
    with np.errstate(invalid="ignore"):
        y = (tiles / s[:, None, :, None]).astype(np.float32)
    q = e4m3_encode(y.astype(np.float64)).reshape(N, K)
    return q, s


def quant_128x128_ue8m0(w) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """128x128 block E4M3 quantisation of a K-major weight [N, K] with power-of-two
    (UE8M0) tile scales: the rule of ``quant_1x128_ue8m0`` with amax over the
    whole tile.  Returns q [N, K] uint8, s [N/128, K/128] float32 (2^e) and the
    bytes e + 127 [N/128, K/128] uint8."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert N % BLOCK == 0 and K % BLOCK == 0
    tiles = w.reshape(N // BLOCK, BLOCK, K // BLOCK, BLOCK)
    amax = _block_amax(tiles, (1, 3))                       # [NB, KB]
    s, byte = _block_scale_ue8m0(amax)
    with np.errstate(invalid="ignore"):
        y = tiles.astype(np.float64) / s[:, None, :, None].astype(np.float64)   # exact
    q = e4m3_encode(y).reshape(N, K)
    return q, s, byte


def permute(topk_ids, expert_begin: int, E: int, layout: str, max_m: int = 0,
            align: int = BLOCK, q=None, s=None) -> dict:
    """Route token-order assignments into the grouped layout of the local experts.

    Assignment i = t*k + j goes to local expert e = topk_ids[t, j] - expert_begin
    when 0 <= e < E.  Within an expert the rows keep ascending i (a reading: the
    pages fix no order; ascending assignment index makes it deterministic).

    masked: expert e owns rows [e*max_m, (e+1)*max_m); if more than max_m
      assignments arrive, the first max_m are kept, the rest get dst_row = -1,
      and ``overflow`` is set (a reading: clamp and report).  counts = kept rows.
    contig: expert segments follow each other, each padded to a multiple of
      ``align``; offsets[e] is the first row of segment e, m_indices[row] is the
      expert owning a real row and -1 on padding.
    row_src[row] = i for every real row, -1 elsewhere; dst_row[i] = row, or -1
    for non-local or dropped assignments.

    With q [T, K] and s [K/128, T] given, the FP8 rows and their scales are
    gathered too: masked -> q_out [E*max_m, K], s_out [E, K/128, max_m];
    contig -> q_out [rows, K], s_out [K/128, rows].  Rows without a source
    stay zero here; the library leaves them untouched.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    lists = [np.nonzero(flat == expert_begin + e)[0] for e in range(E)]
    raw = np.array([len(l) for l in lists], dtype=np.int64)
    dst_row = np.full(T * k, -1, dtype=np.int64)
    out = dict(raw_counts=raw)
    if layout == "masked":
        counts = np.minimum(raw, max_m)
        rows = E * max_m
        row_src = np.full(rows, -1, dtype=np.int64)
        for e, l in enumerate(lists):
            kept = l[:max_m]
            dst_row[kept] = e * max_m + np.arange(len(kept))
            row_src[e * max_m: e * max_m + len(kept)] = kept
        out.update(counts=counts, overflow=bool((raw > max_m).any()))
    elif layout == "contig":
        seg = (raw + align - 1) // align * align
        offsets = np.concatenate([[0], np.cumsum(seg)]).astype(np.int64)
        rows = int(offsets[-1])
        row_src = np.full(rows, -1, dtype=np.int64)
        m_indices = np.full(rows, -1, dtype=np.int64)
        for e, l in enumerate(lists):
            dst_row[l] = offsets[e] + np.arange(len(l))
            row_src[offsets[e]: offsets[e] + len(l)] = l
            m_indices[offsets[e]: offsets[e] + len(l)] = e
        out.update(counts=raw.copy(), offsets=offsets, m_indices=m_indices, overflow=False)
    else:
        raise ValueError(layout)
    out.update(dst_row=dst_row, row_src=row_src, rows=rows)
    if q is not None:
        q = np.asarray(q)
        s = np.asarray(s)
        KB = q.shape[1] // BLOCK
        q_out = np.zeros((rows, q.shape[1]), dtype=np.uint8)
        valid = row_src >= 0
        tok = row_src[valid] // k
        q_out[valid] = q[tok]
        if layout == "masked":
            s_flat = np.zeros((KB, rows), dtype=np.float32)
            s_flat[:, valid] = s[:, tok]
            s_out = np.ascontiguousarray(s_flat.reshape(KB, E, max_m).transpose(1, 0, 2))
        else:
            s_out = np.zeros((KB, rows), dtype=np.float32)
            s_out[:, valid] = s[:, tok]
        out.update(q=q_out, s=s_out)
    return out


def gemm_block_scaled(qa, sa, qb, sb) -> np.ndarray:
    """D = sum over k-blocks kb of sa[kb, m] * sb[n // 128, kb] * sum_{k in kb} qa[m,k] qb[n,k]
    with exact E4M3 decode and float64 accumulation.

    qa [M, K] uint8, sa [K/128, M] float32; qb [N, K] uint8, sb [N/128, K/128]
    float32.  Returns float64 [M, N] (not yet rounded to bf16)."""
    A = e4m3_decode(qa)
    B = e4m3_decode(qb)
    M, K = A.shape
    N = B.shape[0]
    sa = np.asarray(sa, dtype=np.float64)
    sb = np.asarray(sb, dtype=np.float64)
    D = np.zeros((M, N), dtype=np.float64)
    for kb in range(K // BLOCK):
        cols = slice(kb * BLOCK, (kb + 1) * BLOCK)
        partial = A[:, cols] @ B[:, cols].T                   # exact: 8-bit products, 128 terms
        scale = sa[kb, :][:, None] * np.repeat(sb[:, kb], BLOCK)[None, :]
        D += scale * partial
    return D


def gemm_masked(qa, sa, qb, sb, counts) -> tuple[np.ndarray, np.ndarray]:
    """Masked grouped GEMM: for each expert e, rows [0, counts[e]) of
    qa[e] ([max_m, K]) times expert e's weights.  qa [E, max_m, K],
    sa [E, K/128, max_m], qb [E, N, K], sb [E, N/128, K/128].
    Returns (D bf16 bits [E, max_m, N], valid [E, max_m]); rows past the count
    are not produced (the library leaves them untouched)."""
    E, max_m, K = qa.shape
    N = qb.shape[1]
    D = np.zeros((E, max_m, N), dtype=np.uint16)
    valid = np.zeros((E, max_m), dtype=bool)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        D[e, :c] = bf16_encode(gemm_block_scaled(qa[e, :c], sa[e][:, :c], qb[e], sb[e]))
        valid[e, :c] = True
    return D, valid


def gemm_contig(qa, sa, qb, sb, offsets, m_indices) -> tuple[np.ndarray, np.ndarray]:
    """Contiguous grouped GEMM: rows [offsets[e], offsets[e+1]) belong to expert
    e; a row with m_indices == -1 is padding and is not produced.
    qa [rows, K], sa [K/128, rows]; returns (D bf16 bits [rows, N], valid [rows])."""
    rows, K = qa.shape
    N = qb.shape[1]
    D = np.zeros((rows, N), dtype=np.uint16)
    m_indices = np.asarray(m_indices)
    valid = m_indices >= 0
    for e in range(len(offsets) - 1):
        r = np.nonzero(m_indices[offsets[e]:offsets[e + 1]] == e)[0] + offsets[e]
        if len(r) == 0:
            continue
        D[r] = bf16_encode(gemm_block_scaled(qa[r], sa[:, r], qb[e], sb[e]))
    return D, valid


def swiglu(y1_bits) -> np.ndarray:
    """h = silu(g) * u with g = Y1[:, :I] (gate) and u = Y1[:, I:] (up), computed
    in float64 from the bf16 inputs and rounded once to float32 (a reading: h is
    not rounded to bf16 before it is requantised)."""
    y = bf16_decode(y1_bits)
    I = y.shape[1] // 2
    g, u = y[:, :I], y[:, I:]
    with np.errstate(over="ignore"):
        h = g / (1.0 + np.exp(-g)) * u
    return h.astype(np.float32)


def swiglu_quant(y1_bits, ue8m0: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """SwiGLU followed by the 1x128 E4M3 quantisation of ``quant_1x128`` (or, with
    ``ue8m0``, of ``quant_1x128_ue8m0``: power-of-two scales, returned as floats)."""
    if ue8m0:
        q, s, _ = quant_1x128_ue8m0(swiglu(y1_bits))
        return q, s
    return quant_1x128(swiglu(y1_bits))


def combine(y2_bits, dst_row, topk_w, shared_bits=None, out_bits=None) -> np.ndarray:
    """out[t] = bf16( a[t] + sum_j w[t, j] * Y2[dst_row[t*k + j]] + shared[t] ), float64
    accumulation, assignments with dst_row == -1 skipped.  y2_bits [rows, H] -> [T, H]
    bf16 bits.  Optional terms: ``shared_bits`` [T, H], the output of a shared
    expert every token uses at weight 1 (added, not renormalised with the top-k
    weights -- a reading); ``out_bits`` [T, H], the current output to add to
    (a = 0 without it)."""
    w = np.asarray(topk_w, dtype=np.float64)
    T, k = w.shape
    y = bf16_decode(y2_bits)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    if out_bits is not None:
        out += bf16_decode(out_bits)
    dst = np.asarray(dst_row).reshape(T, k)
    for j in range(k):
        ok = dst[:, j] >= 0
        out[ok] += w[ok, j][:, None] * y[dst[ok, j]]
    if shared_bits is not None:
        out += bf16_decode(shared_bits)
    return bf16_encode(out)


def ffn_chain(x_bits, topk_ids, topk_w, expert_begin, E, layout, max_m,
              w13_q, w13_s, w2_q, w2_s, align: int = BLOCK, ue8m0: bool = False) -> dict:
    """The whole path: quant -> permute -> GEMM1 (W13) -> SwiGLU+quant -> GEMM2 (W2)
    -> combine.  Weights are pre-quantised: w13_q [E, 2I, H], w13_s [E, 2I/128, H/128],
    w2_q [E, H, I], w2_s [E, H/128, I/128].  With ``ue8m0`` both activation
    quantisations take power-of-two scales (the other reading of the packed
    input scales; the weights are then expected from quant_128x128_ue8m0, their
    scales as floats 2^e).  Returns every intermediate."""
    x = bf16_decode(x_bits).astype(np.float32)
    q, s = quant_1x128_ue8m0(x)[:2] if ue8m0 else quant_1x128(x)
    p = permute(topk_ids, expert_begin, E, layout, max_m, align, q=q, s=s)
    if layout == "masked":
        A1 = p["q"].reshape(E, max_m, -1)
        y1, valid = gemm_masked(A1, p["s"], w13_q, w13_s, p["counts"])
        y1f = y1.reshape(E * max_m, -1)
        vflat = valid.reshape(-1)
        q2 = np.zeros((E * max_m, y1f.shape[1] // 2), dtype=np.uint8)
        s2 = np.zeros((y1f.shape[1] // 2 // BLOCK, E * max_m), dtype=np.float32)
        qq, ss = swiglu_quant(y1f[vflat], ue8m0)
        q2[vflat], s2[:, vflat] = qq, ss
        s2m = np.ascontiguousarray(s2.reshape(-1, E, max_m).transpose(1, 0, 2))
        y2, _ = gemm_masked(q2.reshape(E, max_m, -1), s2m, w2_q, w2_s, p["counts"])
        y2f = y2.reshape(E * max_m, -1)
    else:
        y1f, vflat = gemm_contig(p["q"], p["s"], w13_q, w13_s, p["offsets"], p["m_indices"])
        q2 = np.zeros((p["rows"], y1f.shape[1] // 2), dtype=np.uint8)
        s2 = np.zeros((y1f.shape[1] // 2 // BLOCK, p["rows"]), dtype=np.float32)
        qq, ss = swiglu_quant(y1f[vflat], ue8m0)
        q2[vflat], s2[:, vflat] = qq, ss
        s2m = s2
        y2f, _ = gemm_contig(q2, s2, w2_q, w2_s, p["offsets"], p["m_indices"])
    out = combine(y2f, p["dst_row"], topk_w)
    return dict(q=q, s=s, perm=p, y1=y1f, valid=vflat, q2=q2, s2=s2m, y2=y2f, out=out)


# ----------------------------------------------------------------------------
# The packed UE8M0 scale layouts of the block-scaled GEMM (the reading of the
# DeepGEMM bullet's "packing of the input scales" in which four exponent bytes
# share a 32-bit word).  Pure layout: no arithmetic on the scales.
# ----------------------------------------------------------------------------
def _ue8m0_bytes(s) -> np.ndarray:
    """Exponent bytes of power-of-two float32 scales (e + 127 for 2^e; 0xFF for inf)."""
    return ((np.asarray(s, dtype=np.float32).view(np.uint32) >> 23) & 0xFF).astype(np.uint8)


def pack_ue8m0_act(s, G: int, rows: int) -> np.ndarray:
    """Power-of-two activation scales in the grouped layout s[(grp*KB + kb)*G + r]
    (flattened; groups of G rows, the first ``rows`` rows existing) -> packed words.

    Group grp, k-group g (k-blocks 4g..4g+3), 128-row chunk c, row i of the
    chunk: word ((grp*KG + g)*NC + c)*128 + 4*(i % 32) + i // 32, whose byte b
    is the exponent byte of k-block 4g + b (0x7F where there is no such row or
    k-block).  KG = ceil(KB/4), NC = ceil(G/128).  Returns uint32 [words]."""
    s = np.asarray(s, dtype=np.float32).reshape(-1)
    groups = -(-rows // G) if rows else 0
    KB = s.size // (groups * G) if groups else 0
    KG, NC = -(-KB // 4), -(-G // 128)
    byte = np.full((groups, KG * 4, NC * 128), 0x7F, np.uint8)       # [grp, kb, row of group]
    b = _ue8m0_bytes(s).reshape(groups, KB, G)
    for grp in range(groups):
        n = min(G, rows - grp * G)
        byte[grp, :KB, :n] = b[grp, :, :n]
    words = np.zeros((groups, KG, NC, 128), np.uint32)
    i = np.arange(128)
    pos = 4 * (i % 32) + i // 32
    for grp in range(groups):
        for g in range(KG):
            for c in range(NC):
                w = np.zeros(128, np.uint32)
                for bb in range(4):
                    w |= byte[grp, 4 * g + bb, c * 128:(c + 1) * 128].astype(np.uint32) << np.uint32(8 * bb)
                words[grp, g, c, pos] = w
    return words.reshape(-1)


def pack_ue8m0_weight(s) -> np.ndarray:
    """Power-of-two weight scales [E, NB, KB] -> 32 copies per (e, nb, g) of the
    word whose byte b is the exponent byte of k-block 4g + b (0x7F past KB).
    Returns uint32 [E*NB*KG*32]."""
    b = _ue8m0_bytes(s)
    E, NB, KB = b.shape
    KG = -(-KB // 4)
    full = np.full((E, NB, KG * 4), 0x7F, np.uint8)
    full[:, :, :KB] = b
    quad = full.reshape(E, NB, KG, 4).astype(np.uint32)
    w = quad[..., 0] | (quad[..., 1] << 8) | (quad[..., 2] << 16) | (quad[..., 3] << 24)
    return np.repeat(w[..., None], 32, axis=3).reshape(-1)
