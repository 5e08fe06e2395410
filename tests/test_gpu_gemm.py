"""Parity of the grouped FP8 GEMMs with the oracle.

* integer-exact closed form: integer operands in [-16, 16] (exact in E4M3) with
  unit scales give an exact integer result, so the bf16 output must be
  bf16(exact integer) bit for bit;
* the acceptance bound |err| <= 2^-7 |ref| + 1e-3 rms(ref) against the oracle
  on random codes and scales, on the configs' shapes (several tiles, ragged
  tails, a half-width last N tile, empty experts);
* rows the layout marks unused keep their sentinel;
* a stalled pipeline (test-only flag) reports MOE_ERR_TIMEOUT and the library
  keeps working afterwards."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_common import (SENTINEL_BF16, Guarded, activations_bits, bits, check_tol, from_bits,
                              oracle_weights, rand_codes, routing, to_dev, u8)

pytestmark = pytest.mark.gpu


def _masked(lib, A, sA, B, sB, counts, flags=0, expected_m=0):
    E, max_m, K = A.shape
    N = B.shape[1]
    g = Guarded((E, max_m, N), torch.bfloat16, SENTINEL_BF16)
    err = lib.new_error_word()
    lib.moe_gemm_fp8_masked(to_dev(A), to_dev(sA), to_dev(B), to_dev(sB),
                            to_dev(np.asarray(counts, np.int32)), g.t, expected_m=expected_m,
                            flags=flags, err=err)
    status, _ = lib.moe_read_device_status(err)
    assert g.intact(), "a store landed past the end of D"
    return bits(g.t), status


def _contig(lib, A, sA, B, sB, offsets, m_indices, flags=0):
    M_cap, K = A.shape
    N = B.shape[1]
    g = Guarded((M_cap, N), torch.bfloat16, SENTINEL_BF16)
    err = lib.new_error_word()
    lib.moe_gemm_fp8_contig(to_dev(A), to_dev(sA), to_dev(B), to_dev(sB),
                            to_dev(np.asarray(offsets, np.int32)), to_dev(np.asarray(m_indices, np.int32)),
                            g.t, flags=flags, err=err)
    status, _ = lib.moe_read_device_status(err)
    assert g.intact(), "a store landed past the end of D"
    return bits(g.t), status


def _check_masked(got, ref, valid, what):
    check_tol(got[valid], ref[valid], what)
    assert (got[~valid] == SENTINEL_BF16).all(), f"{what}: rows past the count were written"


# (flags, expected_m): the tokens-as-M kernel, and the weights-as-M kernel with
# each token-tile width (64 / 128 / 256 columns)
MASKED_KERNELS = [(0x1, 0), (0x2, 16), (0x2, 100), (0x2, 200)]
MASKED_IDS = ["tokens_m", "weights_m64", "weights_m128", "weights_m256"]


@pytest.mark.parametrize("flags,hint", MASKED_KERNELS, ids=MASKED_IDS)
def test_gemm_integer_exact_masked(lib, flags, hint):
    rng = np.random.default_rng(11)
    E, max_m, N, K = 3, 256, 384, 512                 # N = 1.5 tiles of 256: half last tile
    counts = [256, 0, 77]
    a = rng.integers(-16, 17, (E, max_m, K))
    b = rng.integers(-16, 17, (E, N, K))
    A, B = oracle.e4m3_encode(a.astype(np.float64)), oracle.e4m3_encode(b.astype(np.float64))
    sA = np.ones((E, K // 128, max_m), np.float32)
    sB = np.ones((E, N // 128, K // 128), np.float32)
    got, st = _masked(lib, A, sA, B, sB, counts, flags=flags, expected_m=hint)
    assert st == 0
    for e in range(E):
        c = counts[e]
        exact = (a[e, :c] @ b[e].T).astype(np.float64)
        assert np.array_equal(got[e, :c], oracle.bf16_encode(exact)), f"expert {e}"
        assert (got[e, c:] == SENTINEL_BF16).all()


def test_gemm_integer_exact_contig(lib):
    rng = np.random.default_rng(12)
    N, K = 256, 384
    seg = [130, 0, 300]
    offsets = [0, 256, 256, 640]
    M_cap = 768
    mi = -np.ones(M_cap, np.int64)
    mi[0:130] = 0
    mi[256:556] = 2
    a = rng.integers(-16, 17, (M_cap, K))
    b = rng.integers(-16, 17, (3, N, K))
    A, B = oracle.e4m3_encode(a.astype(np.float64)), oracle.e4m3_encode(b.astype(np.float64))
    sA = np.ones((K // 128, M_cap), np.float32)
    sB = np.ones((3, N // 128, K // 128), np.float32)
    got, st = _contig(lib, A, sA, B, sB, offsets, mi)
    assert st == 0
    for e, (lo, n) in enumerate([(0, 130), (256, 0), (256, 300)]):
        if n:
            exact = (a[lo:lo + n] @ b[e].T).astype(np.float64)
            assert np.array_equal(got[lo:lo + n], oracle.bf16_encode(exact)), f"expert {e}"
    assert (got[mi < 0] == SENTINEL_BF16).all()


@pytest.mark.parametrize("flags,hint", MASKED_KERNELS, ids=MASKED_IDS)
def test_gemm_masked_random_scales(lib, flags, hint):
    rng = np.random.default_rng(13)
    E, max_m, N, K = 4, 384, 640, 1024
    counts = [1, 383, 0, 129]
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA = np.exp(rng.uniform(-8, 2, (E, K // 128, max_m))).astype(np.float32)
    sB = np.exp(rng.uniform(-8, 2, (E, N // 128, K // 128))).astype(np.float32)
    got, st = _masked(lib, A, sA, B, sB, counts, flags=flags, expected_m=hint)
    assert st == 0
    ref, valid = oracle.gemm_masked(A, sA, B, sB, counts)
    _check_masked(got, ref, valid, "masked random")


def test_gemm_contig_random_scales(lib):
    rng = np.random.default_rng(14)
    N, K = 384, 768
    seg = [5, 260, 0, 128, 1]
    offsets = [0]
    for c in seg:
        offsets.append(offsets[-1] + -(-c // 128) * 128)
    M_cap = offsets[-1] + 256
    mi = -np.ones(M_cap, np.int64)
    for e, c in enumerate(seg):
        mi[offsets[e]:offsets[e] + c] = e
    A, B = rand_codes(rng, (M_cap, K)), rand_codes(rng, (len(seg), N, K))
    sA = np.exp(rng.uniform(-6, 2, (K // 128, M_cap))).astype(np.float32)
    sB = np.exp(rng.uniform(-6, 2, (len(seg), N // 128, K // 128))).astype(np.float32)
    got, st = _contig(lib, A, sA, B, sB, offsets, mi)
    assert st == 0
    ref, valid = oracle.gemm_contig(A, sA, B, sB, offsets, mi)
    check_tol(got[valid], ref[valid], "contig random")
    assert (got[~valid] == SENTINEL_BF16).all()


@pytest.mark.parametrize("flags,hint", MASKED_KERNELS[:2], ids=MASKED_IDS[:2])
def test_gemm_masked_count_above_max_m_is_clamped(lib, flags, hint):
    rng = np.random.default_rng(15)
    E, max_m, N, K = 2, 128, 256, 256
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA = np.ones((E, K // 128, max_m), np.float32)
    sB = np.ones((E, N // 128, K // 128), np.float32)
    got, st = _masked(lib, A, sA, B, sB, [500, 3], flags=flags, expected_m=hint)
    assert st == lib.MOE_ERR_OVERFLOW
    ref, valid = oracle.gemm_masked(A, sA, B, sB, [128, 3])
    _check_masked(got, ref, valid, "clamped")


def _decode_gemm_inputs(cfg_name, which):
    """Oracle-quantised activations in the masked layout for a decode config."""
    cfg = synth.get_config(cfg_name)
    r = routing(cfg_name)
    K = cfg.H if which == "w13" else cfg.I
    xb = activations_bits(cfg_name, r["T"]) if which == "w13" else None
    if which == "w13":
        q, s = oracle.quant_1x128(oracle.bf16_decode(xb).astype(np.float32))
    else:  # a synthetic SwiGLU output of the right scale, quantised by the oracle
        h = np.random.default_rng(7).standard_normal((r["T"], K)).astype(np.float32) * 0.05
        q, s = oracle.quant_1x128(h)
    p = oracle.permute(r["topk_ids"], r["expert_begin"], cfg.E, "masked", cfg.max_m, q=q, s=s)
    return cfg, p["q"].reshape(cfg.E, cfg.max_m, K), p["s"], p["counts"]


@pytest.mark.parametrize("flags", [0, 0x1, 0x9], ids=["default", "tokens_m", "tokens_m_pair"])
@pytest.mark.parametrize("which", ["w13", "w2"])
def test_gemm_masked_decode_full_size(lib, which, flags):
    cfg, A, sA, counts = _decode_gemm_inputs("c2", which)
    Bq, Bs = oracle_weights("c2", which, tuple(range(cfg.E)))
    got, st = _masked(lib, A, sA, Bq, Bs, counts, flags=flags,
                      expected_m=int(np.ceil(counts.sum() / (counts > 0).sum())))
    assert st == 0
    ref, valid = oracle.gemm_masked(A, sA, Bq, Bs, counts)
    _check_masked(got, ref, valid, f"c2 {which}")


@pytest.mark.parametrize("flags", [0, 0x8], ids=["single", "pair"])
def test_gemm_contig_prefill_sampled_rows(lib, flags):
    cfg = synth.get_config("c3")
    r = routing("c3")
    T = r["T"]
    xb = activations_bits("c3", T)
    # the GPU quantises all rows (bit-exact with the oracle per test_gpu_quant)
    x = from_bits(xb)
    q = torch.empty((T, cfg.H), dtype=torch.uint8, device="cuda")
    s = torch.empty((cfg.H // 128, T), dtype=torch.float32, device="cuda")
    lib.moe_quant_fp8(x, q, s)
    cap = lib.moe_contig_rows_bound(T, cfg.E)
    A = torch.empty((cap, cfg.H), dtype=torch.uint8, device="cuda")
    sA = torch.empty((cfg.H // 128, cap), dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
    mi = torch.empty(cap, dtype=torch.int32, device="cuda")
    row_src = torch.empty(cap, dtype=torch.int32, device="cuda")
    dst = torch.empty(T, dtype=torch.int32, device="cuda")
    lib.moe_permute(q, s, to_dev(r["topk_ids"]), 0, cfg.E, 1, 0, A, sA, counts, offsets, mi,
                    row_src, dst, rows_capacity=cap)
    experts = tuple(range(cfg.E))
    Bq, Bs = oracle_weights("c3", "w13", experts)
    D = torch.full((cap, 2 * cfg.I), SENTINEL_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    lib.moe_gemm_fp8_contig(A, sA, to_dev(Bq), to_dev(Bs), offsets, mi, D, flags=flags)
    torch.cuda.synchronize()
    got = bits(D)
    off = offsets.cpu().numpy()
    mi_h = mi.cpu().numpy()
    # oracle on sampled rows: every tile edge of every expert plus random rows
    rng = np.random.default_rng(9)
    rows = []
    for e in range(cfg.E):
        lo, c = off[e], int(r["split"][e])
        for rr in (0, 1, 127, 128, c - 1, c // 2):
            if 0 <= rr < c:
                rows.append(lo + rr)
        rows += list(lo + rng.integers(0, c, 6))
    rows = np.unique(np.array(rows))
    rs_h = row_src.cpu().numpy()
    for e in range(cfg.E):
        sel = rows[mi_h[rows] == e]
        if len(sel) == 0:
            continue
        tok = rs_h[sel]                       # k = 1: assignment index = token
        xq, xs = oracle.quant_1x128(oracle.bf16_decode(xb[tok]).astype(np.float32))
        ref = oracle.bf16_encode(oracle.gemm_block_scaled(xq, xs, Bq[e], Bs[e]))
        check_tol(got[sel], ref, f"c3 expert {e}")
    assert (got[mi_h < 0] == SENTINEL_BF16).all()


@pytest.mark.parametrize("case", ["past_capacity", "negative", "unaligned", "decreasing"])
@pytest.mark.parametrize("flags", [0, 0x8], ids=["single", "pair"])
def test_gemm_contig_segment_outside_capacity_is_skipped(lib, case, flags):
    # offsets that put a segment outside [0, M_capacity) (or off the 128-row grid)
    # must not be read or written: the segment is skipped, MOE_DEV_BAD_INDEX is
    # set, the good segments are still computed, and nothing lands past D
    rng = np.random.default_rng(17)
    N, K, M_cap = 256, 256, 384
    offsets = {"past_capacity": [0, 128, M_cap + 128], "negative": [-128, 128, 384],
               "unaligned": [0, 64, 384], "decreasing": [0, 128, 0]}[case]
    good = {"past_capacity": [0], "negative": [1], "unaligned": [], "decreasing": [0]}[case]
    mi = -np.ones(M_cap, np.int64)
    mi[0:100] = 0
    mi[128:384] = 1
    A, B = rand_codes(rng, (M_cap, K)), rand_codes(rng, (2, N, K))
    sA = np.exp(rng.uniform(-4, 1, (K // 128, M_cap))).astype(np.float32)
    sB = np.exp(rng.uniform(-4, 1, (2, N // 128, K // 128))).astype(np.float32)
    got, st = _contig(lib, A, sA, B, sB, offsets, mi, flags=flags)
    assert st == lib.MOE_ERR_BAD_INDEX
    written = np.zeros(M_cap, bool)
    for e in good:
        lo = offsets[e]
        rows = np.nonzero(mi[lo:offsets[e + 1]] == e)[0] + lo
        ref = oracle.bf16_encode(oracle.gemm_block_scaled(A[rows], sA[:, rows], B[e], sB[e]))
        check_tol(got[rows], ref, f"{case} expert {e}")
        written[rows] = True
    assert (got[~written] == SENTINEL_BF16).all(), "a skipped segment was written"


def test_gemm_stall_reports_timeout_and_recovers(lib):
    rng = np.random.default_rng(16)
    E, max_m, N, K = 1, 128, 256, 256
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA = np.ones((E, K // 128, max_m), np.float32)
    sB = np.ones((E, N // 128, K // 128), np.float32)
    for kernel in (lib.MOE_GEMM_FORCE_TOKENS_M, lib.MOE_GEMM_FORCE_WEIGHTS_M,
                   lib.MOE_GEMM_FORCE_TOKENS_M | lib.MOE_GEMM_CTA_PAIR):
        got, st = _masked(lib, A, sA, B, sB, [5], flags=lib.MOE_GEMM_DEBUG_STALL | kernel)
        assert st == lib.MOE_ERR_TIMEOUT
        assert (got == SENTINEL_BF16).all()
    got, st = _masked(lib, A, sA, B, sB, [5])
    assert st == 0
    ref, valid = oracle.gemm_masked(A, sA, B, sB, [5])
    _check_masked(got, ref, valid, "after timeout")


# ---------------------------------------------------------------- CTA pairs
# The pair kernel (MOE_GEMM_CTA_PAIR) cuts an expert's rows into 256-row blocks;
# the cases below give experts an odd number of 128-row blocks (a pair block
# that runs into the next expert's rows or past the buffer), a ragged count,
# an empty expert, and more than one 256-column tile.

def test_gemm_pair_integer_exact_masked(lib):
    rng = np.random.default_rng(31)
    E, max_m, N, K = 3, 384, 512, 512
    counts = [384, 0, 77]
    a = rng.integers(-16, 17, (E, max_m, K))
    b = rng.integers(-16, 17, (E, N, K))
    A, B = oracle.e4m3_encode(a.astype(np.float64)), oracle.e4m3_encode(b.astype(np.float64))
    sA = np.ones((E, K // 128, max_m), np.float32)
    sB = np.ones((E, N // 128, K // 128), np.float32)
    got, st = _masked(lib, A, sA, B, sB, counts, flags=lib.MOE_GEMM_FORCE_TOKENS_M | lib.MOE_GEMM_CTA_PAIR)
    assert st == 0
    for e in range(E):
        c = counts[e]
        exact = (a[e, :c] @ b[e].T).astype(np.float64)
        assert np.array_equal(got[e, :c], oracle.bf16_encode(exact)), f"expert {e}"
        assert (got[e, c:] == SENTINEL_BF16).all()


def _pair_contig_layout(seg):
    offsets = [0]
    for c in seg:
        offsets.append(offsets[-1] + -(-c // 128) * 128)
    M_cap = offsets[-1]
    mi = -np.ones(M_cap, np.int64)
    for e, c in enumerate(seg):
        mi[offsets[e]:offsets[e] + c] = e
    return offsets, M_cap, mi


def test_gemm_pair_integer_exact_contig(lib):
    rng = np.random.default_rng(32)
    N, K = 256, 384
    seg = [130, 0, 300, 128, 1]             # 2, 0, 3, 1, 1 row blocks of 128
    offsets, M_cap, mi = _pair_contig_layout(seg)
    a = rng.integers(-16, 17, (M_cap, K))
    b = rng.integers(-16, 17, (len(seg), N, K))
    A, B = oracle.e4m3_encode(a.astype(np.float64)), oracle.e4m3_encode(b.astype(np.float64))
    sA = np.ones((K // 128, M_cap), np.float32)
    sB = np.ones((len(seg), N // 128, K // 128), np.float32)
    got, st = _contig(lib, A, sA, B, sB, offsets, mi, flags=lib.MOE_GEMM_CTA_PAIR)
    assert st == 0
    for e, c in enumerate(seg):
        lo = offsets[e]
        if c:
            exact = (a[lo:lo + c] @ b[e].T).astype(np.float64)
            assert np.array_equal(got[lo:lo + c], oracle.bf16_encode(exact)), f"expert {e}"
    assert (got[mi < 0] == SENTINEL_BF16).all()


def test_gemm_pair_random_scales(lib):
    rng = np.random.default_rng(33)
    N, K = 768, 1024
    seg = [5, 260, 0, 640, 1]
    offsets, M_cap, mi = _pair_contig_layout(seg)
    A, B = rand_codes(rng, (M_cap, K)), rand_codes(rng, (len(seg), N, K))
    sA = np.exp(rng.uniform(-6, 2, (K // 128, M_cap))).astype(np.float32)
    sB = np.exp(rng.uniform(-6, 2, (len(seg), N // 128, K // 128))).astype(np.float32)
    got, st = _contig(lib, A, sA, B, sB, offsets, mi, flags=lib.MOE_GEMM_CTA_PAIR)
    assert st == 0
    ref, valid = oracle.gemm_contig(A, sA, B, sB, offsets, mi)
    check_tol(got[valid], ref[valid], "pair contig random")
    assert (got[~valid] == SENTINEL_BF16).all()
    # masked layout, counts around the 256-row pair block
    E, max_m = 4, 640
    counts = [1, 256, 0, 513]
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA = np.exp(rng.uniform(-8, 2, (E, K // 128, max_m))).astype(np.float32)
    sB = np.exp(rng.uniform(-8, 2, (E, N // 128, K // 128))).astype(np.float32)
    got, st = _masked(lib, A, sA, B, sB, counts, flags=lib.MOE_GEMM_FORCE_TOKENS_M | lib.MOE_GEMM_CTA_PAIR)
    assert st == 0
    ref, valid = oracle.gemm_masked(A, sA, B, sB, counts)
    _check_masked(got, ref, valid, "pair masked random")


@pytest.mark.parametrize("K", [256, 640])
@pytest.mark.parametrize("flags,hint", MASKED_KERNELS, ids=MASKED_IDS)
def test_gemm_early_weights_flag_is_bit_identical_masked(lib, flags, hint, K):
    """MOE_GEMM_EARLY_WEIGHTS (counts complete before the previous kernel) only
    moves the schedule and the first stages' weight copies ahead of the grid
    dependency wait: the result is the same bits.  K = 256 spreads the early
    stages over several tiles, K = 640 keeps them in one."""
    rng = np.random.default_rng(17)
    E, max_m, N = 3, 256, 384
    counts = [200, 0, 77]
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA = np.exp(rng.uniform(-6, 2, (E, K // 128, max_m))).astype(np.float32)
    sB = np.exp(rng.uniform(-6, 2, (E, N // 128, K // 128))).astype(np.float32)
    ref, st0 = _masked(lib, A, sA, B, sB, counts, flags=flags, expected_m=hint)
    got, st1 = _masked(lib, A, sA, B, sB, counts, flags=flags | lib.MOE_GEMM_EARLY_WEIGHTS, expected_m=hint)
    assert st0 == 0 and st1 == 0
    assert np.array_equal(got, ref)


def test_gemm_early_weights_flag_is_bit_identical_contig(lib):
    rng = np.random.default_rng(18)
    N, K, M_cap = 384, 384, 768
    offsets = [0, 256, 256, 640]
    mi = -np.ones(M_cap, np.int64)
    mi[0:130] = 0
    mi[256:556] = 2
    A, B = rand_codes(rng, (M_cap, K)), rand_codes(rng, (3, N, K))
    sA = np.exp(rng.uniform(-6, 2, (K // 128, M_cap))).astype(np.float32)
    sB = np.exp(rng.uniform(-6, 2, (3, N // 128, K // 128))).astype(np.float32)
    ref, st0 = _contig(lib, A, sA, B, sB, offsets, mi)
    got, st1 = _contig(lib, A, sA, B, sB, offsets, mi, flags=lib.MOE_GEMM_EARLY_WEIGHTS)
    assert st0 == 0 and st1 == 0
    assert np.array_equal(got, ref)
