"""Parity of the block-scaled (UE8M0) grouped GEMM with the oracle.

The scales are powers of two packed four k-blocks per word (the layouts of
moe_fp8.h, written here by the oracle's packers) and applied by the tensor
cores.  Checks:
* the library's packers equal the oracle's bit for bit;
* integer-exact products: integer operands in [-4, 4] with power-of-two scales
  varying per row, k-block and weight block keep every partial sum exact in
  fp32, so the bf16 output must equal bf16(exact) bit for bit -- a misplaced
  scale byte (wrong row, k-block or weight block) changes the result;
* random codes and scales at the acceptance bound, full-size decode and prefill
  shapes, ragged and empty experts, a half-width last N tile;
* rows past a count / padding rows keep their sentinel, nothing is written past
  D (guard band), and a stalled pipeline reports MOE_ERR_TIMEOUT."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_common import (SENTINEL_BF16, Guarded, activations_bits, bits, check_tol, rand_codes, routing,
                              to_dev)

pytestmark = pytest.mark.gpu


def _pow2(rng, shape, lo, hi):
    return np.exp2(rng.integers(lo, hi + 1, shape).astype(np.float64)).astype(np.float32)


def _sfa_masked(sA):
    """Oracle-packed words of masked scales sA [E, KB, max_m] (groups of max_m rows)."""
    E, _, max_m = sA.shape
    return oracle.pack_ue8m0_act(sA, max_m, E * max_m)


def _sfa_contig(sA, ld):
    """Oracle-packed words of contiguous scales sA [KB, ld] (one group of ld rows)."""
    return oracle.pack_ue8m0_act(sA, ld, ld)


def _i32(words):
    return to_dev(np.ascontiguousarray(words).view(np.int32))


def _masked(lib, A, sA, B, sB, counts, flags=0, hint=0):
    E, max_m, K = A.shape
    N = B.shape[1]
    g = Guarded((E, max_m, N), torch.bfloat16, SENTINEL_BF16)
    err = lib.new_error_word()
    lib.moe_gemm_fp8_masked_ue8m0(to_dev(A), _i32(_sfa_masked(sA)), to_dev(B), _i32(oracle.pack_ue8m0_weight(sB)),
                                  to_dev(np.asarray(counts, np.int32)), g.t, expected_m=hint, flags=flags, err=err)
    st, _ = lib.moe_read_device_status(err)
    assert g.intact(), "a store landed past the end of D"
    return bits(g.t), st


def _contig(lib, A, sA, B, sB, offsets, mi, flags=0):
    M_cap, K = A.shape
    N = B.shape[1]
    g = Guarded((M_cap, N), torch.bfloat16, SENTINEL_BF16)
    err = lib.new_error_word()
    lib.moe_gemm_fp8_contig_ue8m0(to_dev(A), _i32(_sfa_contig(sA, M_cap)), M_cap, to_dev(B),
                                  _i32(oracle.pack_ue8m0_weight(sB)), to_dev(np.asarray(offsets, np.int32)),
                                  to_dev(np.asarray(mi, np.int32)), g.t, flags=flags, err=err)
    st, _ = lib.moe_read_device_status(err)
    assert g.intact(), "a store landed past the end of D"
    return bits(g.t), st


def test_pack_kernels_equal_the_oracle(lib):
    rng = np.random.default_rng(40)
    for groups, G, K in ((3, 300, 1024), (1, 256, 640), (257, 128, 7168), (4, 16, 256)):
        s = _pow2(rng, (groups, K // 128, G), -25, 25)
        s[0, 0, 0] = np.inf
        n = lib.moe_ue8m0_act_words(groups, G, K)
        out = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        lib.moe_pack_ue8m0_act(to_dev(s), groups, G, groups * G, K, out)
        torch.cuda.synchronize()
        ref = oracle.pack_ue8m0_act(s, G, groups * G)
        assert n == ref.size and np.array_equal(out.cpu().numpy().view(np.uint32), ref), (groups, G, K)
    for E, N, K in ((3, 384, 1024), (2, 4096, 7168), (1, 7168, 2048)):
        s = _pow2(rng, (E, N // 128, K // 128), -25, 25)
        n = lib.moe_ue8m0_weight_words(E, N, K)
        out = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        lib.moe_pack_ue8m0_weight(to_dev(s), out, K)
        torch.cuda.synchronize()
        ref = oracle.pack_ue8m0_weight(s)
        assert n == ref.size and np.array_equal(out.cpu().numpy().view(np.uint32), ref), (E, N, K)


# (flags, hint): the tokens-as-M kernel, and the weights-as-M kernel with
# 64- and 128-column token tiles
KERNELS = [(0x1, 0), (0x2, 16), (0x2, 100)]
KERNEL_IDS = ["tokens_m", "weights_m64", "weights_m128"]


@pytest.mark.parametrize("flags,hint", KERNELS, ids=KERNEL_IDS)
def test_integer_exact_masked(lib, flags, hint):
    rng = np.random.default_rng(41)
    E, max_m, N, K = 3, 256, 384, 1024             # N = 1.5 tiles: a half-width last tile; 2 k-groups
    counts = [256, 0, 77]
    a = rng.integers(-4, 5, (E, max_m, K))
    b = rng.integers(-4, 5, (E, N, K))
    A, B = oracle.e4m3_encode(a.astype(np.float64)), oracle.e4m3_encode(b.astype(np.float64))
    sA = _pow2(rng, (E, K // 128, max_m), -2, 2)
    sB = _pow2(rng, (E, N // 128, K // 128), -2, 2)
    got, st = _masked(lib, A, sA, B, sB, counts, flags, hint)
    assert st == 0
    ref, valid = oracle.gemm_masked(A, sA, B, sB, counts)
    assert np.array_equal(got[valid], ref[valid]), "not bit-exact"
    assert (got[~valid] == SENTINEL_BF16).all(), "rows past a count were written"


def test_integer_exact_contig(lib):
    rng = np.random.default_rng(42)
    N, K = 256, 768                                # 6 k-blocks: a part-filled last k-group
    seg = [130, 0, 300, 128, 1]
    offsets = [0]
    for c in seg:
        offsets.append(offsets[-1] + -(-c // 128) * 128)
    M_cap = offsets[-1] + 128
    mi = -np.ones(M_cap, np.int64)
    for e, c in enumerate(seg):
        mi[offsets[e]:offsets[e] + c] = e
    a = rng.integers(-4, 5, (M_cap, K))
    b = rng.integers(-4, 5, (len(seg), N, K))
    A, B = oracle.e4m3_encode(a.astype(np.float64)), oracle.e4m3_encode(b.astype(np.float64))
    sA = _pow2(rng, (K // 128, M_cap), -2, 2)
    sB = _pow2(rng, (len(seg), N // 128, K // 128), -2, 2)
    got, st = _contig(lib, A, sA, B, sB, offsets, mi)
    assert st == 0
    ref, valid = oracle.gemm_contig(A, sA, B, sB, offsets, mi)
    assert np.array_equal(got[valid], ref[valid]), "not bit-exact"
    assert (got[~valid] == SENTINEL_BF16).all()


@pytest.mark.parametrize("flags,hint", KERNELS, ids=KERNEL_IDS)
def test_random_codes_and_scales_masked(lib, flags, hint):
    rng = np.random.default_rng(43)
    E, max_m, N, K = 4, 384, 640, 1024
    counts = [1, 383, 0, 129]
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA = _pow2(rng, (E, K // 128, max_m), -12, 3)
    sB = _pow2(rng, (E, N // 128, K // 128), -12, 3)
    got, st = _masked(lib, A, sA, B, sB, counts, flags, hint)
    assert st == 0
    ref, valid = oracle.gemm_masked(A, sA, B, sB, counts)
    check_tol(got[valid], ref[valid], "ue8m0 masked random")
    assert (got[~valid] == SENTINEL_BF16).all()


def test_decode_full_size(lib):
    # the EP72-like decode GEMM1 and GEMM2 with UE8M0-quantised activations and
    # weights (oracle quantisation, oracle packing)
    cfg = synth.get_config("c2")
    r = routing("c2")
    for which, K, N in (("w13", cfg.H, 2 * cfg.I), ("w2", cfg.I, cfg.H)):
        if which == "w13":
            x = oracle.bf16_decode(activations_bits("c2", r["T"])).astype(np.float32)
        else:
            x = np.random.default_rng(7).standard_normal((r["T"], K)).astype(np.float32) * 0.05
        q, s, _ = oracle.quant_1x128_ue8m0(x)
        p = oracle.permute(r["topk_ids"], r["expert_begin"], cfg.E, "masked", cfg.max_m, q=q, s=s)
        wq, ws = [], []
        for e in range(cfg.E):
            w = oracle.bf16_decode(bits(synth.make_expert_weights(cfg, which, e, device="cuda"))).astype(np.float32)
            a, b, _ = oracle.quant_128x128_ue8m0(w)
            wq.append(a)
            ws.append(b)
        A = p["q"].reshape(cfg.E, cfg.max_m, K)
        got, st = _masked(lib, A, p["s"], np.stack(wq), np.stack(ws), p["counts"])
        assert st == 0
        ref, valid = oracle.gemm_masked(A, p["s"], np.stack(wq), np.stack(ws), p["counts"])
        check_tol(got[valid], ref[valid], f"ue8m0 c2 {which}")
        assert (got[~valid] == SENTINEL_BF16).all()


def test_prefill_contig_sampled_rows(lib):
    # prefill GEMM1 shape (9 experts, 32768 rows, N 4096, K 7168) on random codes
    # with power-of-two scales; the oracle on tile-edge and random rows
    cfg = synth.get_config("c3")
    split = synth.make_routing(cfg)["split"]
    offsets = [0]
    for c in split:
        offsets.append(offsets[-1] + -(-int(c) // 128) * 128)
    M_cap = offsets[-1]
    mi = -np.ones(M_cap, np.int64)
    for e, c in enumerate(split):
        mi[offsets[e]:offsets[e] + c] = e
    rng = np.random.default_rng(44)
    N, K = 2 * cfg.I, cfg.H
    A = rand_codes(rng, (M_cap, K))
    B = rand_codes(rng, (cfg.E, N, K))
    sA = _pow2(rng, (K // 128, M_cap), -10, 0)
    sB = _pow2(rng, (cfg.E, N // 128, K // 128), -12, -4)
    got, st = _contig(lib, A, sA, B, sB, offsets, mi)
    assert st == 0
    rows = []
    for e, c in enumerate(split):
        for rr in (0, 1, 127, 128, int(c) - 1, int(c) // 2):
            if 0 <= rr < c:
                rows.append(offsets[e] + rr)
    rows = np.unique(np.array(rows + list(rng.choice(np.nonzero(mi >= 0)[0], 40, replace=False))))
    for e in range(cfg.E):
        sel = rows[mi[rows] == e]
        if len(sel):
            ref = oracle.bf16_encode(oracle.gemm_block_scaled(A[sel], sA[:, sel], B[e], sB[e]))
            check_tol(got[sel], ref, f"ue8m0 c3 expert {e}")
    assert (got[mi < 0] == SENTINEL_BF16).all()


def test_stall_reports_timeout_and_recovers(lib):
    rng = np.random.default_rng(45)
    E, max_m, N, K = 1, 128, 256, 512
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA = np.ones((E, K // 128, max_m), np.float32)
    sB = np.ones((E, N // 128, K // 128), np.float32)
    for kernel in (lib.MOE_GEMM_FORCE_TOKENS_M, lib.MOE_GEMM_FORCE_WEIGHTS_M):
        got, st = _masked(lib, A, sA, B, sB, [5], flags=lib.MOE_GEMM_DEBUG_STALL | kernel)
        assert st == lib.MOE_ERR_TIMEOUT
        assert (got == SENTINEL_BF16).all()
    got, st = _masked(lib, A, sA, B, sB, [5])
    assert st == 0
    ref, valid = oracle.gemm_masked(A, sA, B, sB, [5])
    check_tol(got[valid], ref[valid], "after timeout")


def test_all_experts_decode_shape_weights_m(lib):
    # the all-experts decode GEMM1 shape with a few rows per expert (16 experts
    # of the 257, counts 0..3, max_m 128): the weights-as-M kernel streams each
    # expert's weights once; random codes with power-of-two scales
    rng = np.random.default_rng(46)
    E, max_m, N, K = 16, 128, 4096, 7168
    counts = rng.integers(0, 4, E)
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA = _pow2(rng, (E, K // 128, max_m), -10, 0)
    sB = _pow2(rng, (E, N // 128, K // 128), -12, -4)
    got, st = _masked(lib, A, sA, B, sB, counts, hint=2)
    assert st == 0
    ref, valid = oracle.gemm_masked(A, sA, B, sB, counts)
    check_tol(got[valid], ref[valid], "ue8m0 all-experts shape")
    assert (got[~valid] == SENTINEL_BF16).all()


@pytest.mark.parametrize("K", [256, 640])
@pytest.mark.parametrize("flags,hint", KERNELS, ids=KERNEL_IDS)
def test_early_weights_flag_is_bit_identical_masked(lib, flags, hint, K):
    """MOE_GEMM_EARLY_WEIGHTS (counts complete before the previous kernel) only
    moves the schedule and the first stages' weight copies ahead of the grid
    dependency wait: the result is the same bits.  K = 256 spreads the early
    stages over several tiles, K = 640 keeps them in one."""
    rng = np.random.default_rng(47)
    E, max_m, N = 3, 256, 384
    counts = [200, 0, 77]
    A, B = rand_codes(rng, (E, max_m, K)), rand_codes(rng, (E, N, K))
    sA, sB = _pow2(rng, (E, K // 128, max_m), -6, 2), _pow2(rng, (E, N // 128, K // 128), -6, 2)
    ref, st0 = _masked(lib, A, sA, B, sB, counts, flags=flags, hint=hint)
    got, st1 = _masked(lib, A, sA, B, sB, counts, flags=flags | lib.MOE_GEMM_EARLY_WEIGHTS, hint=hint)
    assert st0 == 0 and st1 == 0
    assert np.array_equal(got, ref)


def test_early_weights_flag_is_bit_identical_contig(lib):
    rng = np.random.default_rng(48)
    N, K, M_cap = 384, 384, 768
    offsets = [0, 256, 256, 640]
    mi = -np.ones(M_cap, np.int64)
    mi[0:130] = 0
    mi[256:556] = 2
    A, B = rand_codes(rng, (M_cap, K)), rand_codes(rng, (3, N, K))
    sA, sB = _pow2(rng, (K // 128, M_cap), -6, 2), _pow2(rng, (3, N // 128, K // 128), -6, 2)
    ref, st0 = _contig(lib, A, sA, B, sB, offsets, mi)
    got, st1 = _contig(lib, A, sA, B, sB, offsets, mi, flags=lib.MOE_GEMM_EARLY_WEIGHTS)
    assert st0 == 0 and st1 == 0
    assert np.array_equal(got, ref)
