"""Parity of moe_swiglu_quant and moe_combine with the oracle.

SwiGLU: the GPU's expf is not correctly rounded, so h may differ from the
oracle's float64-then-float32 value by a few float32 ulps.  Acceptance: scales
within 4 ulp; an FP8 code may differ only by one step, only where the oracle's
value of h/s lies within 2^-19 (relative) of the rounding midpoint between
the two codes (or the scale moved), and on fewer than 1e-4 of the codes.
Combine: the acceptance bound; k=1 at weight 1 is a pure gather (bit-exact);
constant expert rows come back unchanged; dropped entries are skipped."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_common import (Guarded, f32_bits, SENTINEL_BF16, SENTINEL_F32, SENTINEL_U8, bits, check_swiglu,
                              check_tol, from_bits, to_dev, u8)

pytestmark = pytest.mark.gpu


def _y1(rows, I, seed, scale=2.0):
    z = synth.counter_normal(rows * 2 * I, seed, 77, device="cuda") * scale
    return bits(z.to(torch.bfloat16).reshape(rows, 2 * I))


def test_swiglu_quant_masked_rows(lib):
    E, max_m, I = 3, 64, 256
    counts = np.array([64, 0, 17], np.int32)
    y1 = _y1(E * max_m, I, 1)
    gq = Guarded((E * max_m, I), torch.uint8, SENTINEL_U8)
    gs = Guarded((E, I // 128, max_m), torch.float32, f32_bits(SENTINEL_F32))
    q, s = gq.t, gs.t
    lib.moe_swiglu_quant(from_bits(y1), q, s, counts=to_dev(counts), max_m=max_m)
    torch.cuda.synchronize()
    assert gq.intact() and gs.intact(), "SwiGLU wrote past the end of an output"
    qh, sh = u8(q), s.cpu().numpy()
    valid = np.concatenate([np.arange(max_m) < c for c in counts])
    sflat = sh.transpose(1, 0, 2).reshape(I // 128, -1)
    check_swiglu(qh, sflat[:, valid], y1, valid)
    assert (qh[~valid] == SENTINEL_U8).all() and (sflat[:, ~valid] == SENTINEL_F32).all()


def test_swiglu_quant_masked_counts_clamped_and_many_experts(lib):
    # a count above max_m covers the whole slot range, a negative count none;
    # 300 experts, most of them empty, exercise the expert search over the
    # counts prefix (rows of the nonempty ones land in the right slots)
    max_m, I = 32, 256
    counts = np.zeros(300, np.int32)
    counts[[0, 1, 2, 150, 298, 299]] = [100, -5, 7, 32, 1, 19]
    E = counts.size
    y1 = _y1(E * max_m, I, 6)
    gq = Guarded((E * max_m, I), torch.uint8, SENTINEL_U8)
    gs = Guarded((E, I // 128, max_m), torch.float32, f32_bits(SENTINEL_F32))
    q, s = gq.t, gs.t
    lib.moe_swiglu_quant(from_bits(y1), q, s, counts=to_dev(counts), max_m=max_m)
    torch.cuda.synchronize()
    assert gq.intact() and gs.intact(), "SwiGLU wrote past the end of an output"
    qh, sh = u8(q), s.cpu().numpy()
    kept = np.clip(counts, 0, max_m)
    valid = np.concatenate([np.arange(max_m) < c for c in kept])
    sflat = sh.transpose(1, 0, 2).reshape(I // 128, -1)
    check_swiglu(qh, sflat[:, valid], y1, valid)
    assert (qh[~valid] == SENTINEL_U8).all() and (sflat[:, ~valid] == SENTINEL_F32).all()


def test_swiglu_quant_contig_selection_and_full_width(lib):
    rows, I = 512, 2048
    mi = np.full(rows, -1, np.int32)
    mi[:200] = 0
    mi[256:300] = 1
    y1 = _y1(rows, I, 2, scale=3.0)
    gq = Guarded((rows, I), torch.uint8, SENTINEL_U8)
    gs = Guarded((I // 128, rows), torch.float32, f32_bits(SENTINEL_F32))
    q, s = gq.t, gs.t
    lib.moe_swiglu_quant(from_bits(y1), q, s, m_indices=to_dev(mi), s_ld=rows)
    torch.cuda.synchronize()
    assert gq.intact() and gs.intact(), "SwiGLU wrote past the end of an output"
    qh, sh = u8(q), s.cpu().numpy()
    valid = mi >= 0
    check_swiglu(qh, sh[:, valid], y1, valid)
    assert (qh[~valid] == SENTINEL_U8).all() and (sh[:, ~valid] == SENTINEL_F32).all()


def _combine(lib, y2_bits, dst, w):
    T, k = w.shape
    g = Guarded((T, y2_bits.shape[1]), torch.bfloat16, SENTINEL_BF16)
    err = lib.new_error_word()
    lib.moe_combine(from_bits(y2_bits), to_dev(dst.astype(np.int32)), to_dev(w.astype(np.float32)), g.t, err=err)
    st, _ = lib.moe_read_device_status(err)
    assert g.intact(), "combine wrote past the end of out"
    return bits(g.t), st


def test_combine_matches_oracle_decode_routing(lib):
    cfg = synth.get_config("c4")
    r = synth.make_routing(cfg)
    p = oracle.permute(r["topk_ids"], r["expert_begin"], cfg.E, "masked", cfg.max_m)
    H = 1024
    y2 = _y1(cfg.E * cfg.max_m, H // 2, 3)
    got, st = _combine(lib, y2, p["dst_row"], r["topk_w"])
    assert st == 0
    check_tol(got, oracle.combine(y2, p["dst_row"], r["topk_w"]), "combine c4 routing")


def test_combine_gather_and_constant_rows_and_dropped(lib):
    rng = np.random.default_rng(4)
    H = 7168
    y2 = _y1(40, H // 2, 4)
    dst = rng.permutation(40)[:25]
    got, st = _combine(lib, y2, dst, np.ones((25, 1), np.float32))
    assert st == 0 and np.array_equal(got, y2[dst])
    # constant rows, weights summing to one
    c = oracle.bf16_encode(rng.standard_normal(H))
    yc = np.tile(c, (32, 1))
    w = rng.random((8, 4)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    got, st = _combine(lib, yc, rng.permutation(32), w)
    assert np.array_equal(got, np.tile(c, (8, 1)))
    # dropped entries; a token with none gets zeros
    dst2 = np.array([0, -1, -1, -1, 5, 6], np.int64)
    w2 = np.full((3, 2), 0.5, np.float32)
    got, st = _combine(lib, y2, dst2, w2)
    assert np.array_equal(got, oracle.combine(y2, dst2, w2))
    assert (oracle.bf16_decode(got[1]) == 0).all()


def test_combine_bad_row_index_is_reported(lib):
    y2 = _y1(8, 64, 5)
    dst = np.array([0, 9, 3, 2], np.int64)             # 9 >= 8 rows
    got, st = _combine(lib, y2, dst, np.full((2, 2), 0.5, np.float32))
    assert st == lib.MOE_ERR_BAD_INDEX
    ok = dst.copy()
    ok[1] = -1
    assert np.array_equal(got, oracle.combine(y2, ok, np.full((2, 2), 0.5, np.float32)))


@pytest.mark.parametrize("T", [40, 1000], ids=["latency_shape", "wave_shape"])
def test_combine_shared_row_and_accumulate(lib, T):
    # the shared expert's row (weight 1, added after the slots) gives the same
    # bits as routing it as one more slot of weight 1; ACCUMULATE adds to the
    # output's current values; both against the oracle, with guard bands
    rng = np.random.default_rng(6)
    k, H, rows = 8, 7168, 300
    y2 = _y1(rows, H // 2, 6)
    sh = _y1(T, H // 2, 7)
    dst = rng.integers(-1, rows, (T, k)).astype(np.int64)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    g = Guarded((T, H), torch.bfloat16, SENTINEL_BF16)
    lib.moe_combine(from_bits(y2), to_dev(dst.reshape(-1).astype(np.int32)), to_dev(w), g.t, shared=from_bits(sh))
    torch.cuda.synchronize()
    assert g.intact()
    got = bits(g.t)
    check_tol(got, oracle.combine(y2, dst.reshape(-1), w, shared_bits=sh), "combine + shared")
    y_ext = np.concatenate([y2, sh])
    dst_ext = np.concatenate([dst, rows + np.arange(T)[:, None]], axis=1)
    w_ext = np.concatenate([w, np.ones((T, 1), np.float32)], axis=1)
    ext, st = _combine(lib, y_ext, dst_ext.reshape(-1), w_ext)
    assert st == 0 and np.array_equal(got, ext)
    # accumulate on top of an existing output (synthetic values; shared row included)
    old = _y1(T, H // 2, 8)
    g.t.copy_(from_bits(old))
    lib.moe_combine(from_bits(y2), to_dev(dst.reshape(-1).astype(np.int32)), to_dev(w), g.t, shared=from_bits(sh),
                    flags=lib.MOE_COMBINE_ACCUMULATE)
    torch.cuda.synchronize()
    assert g.intact()
    check_tol(bits(g.t), oracle.combine(y2, dst.reshape(-1), w, shared_bits=sh, out_bits=old), "accumulate")
    # no slots and no shared row: the output is left as it was
    none = to_dev(np.full(T * k, -1, np.int32))
    before = bits(g.t).copy()
    lib.moe_combine(from_bits(y2), none, to_dev(w), g.t, flags=lib.MOE_COMBINE_ACCUMULATE)
    torch.cuda.synchronize()
    assert np.array_equal(bits(g.t), before)
