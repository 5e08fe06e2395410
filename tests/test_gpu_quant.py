"""Parity of the quantisation kernels with the oracle: bit-exact FP8 bytes and
scales (the GPU divides with IEEE float32 like the definition)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_common import (SENTINEL_F32, SENTINEL_U8, activations_bits, bits, from_bits,
                              oracle_weights, to_dev, u8)

pytestmark = pytest.mark.gpu


def _gpu_quant(lib, xbits, s_ld=None):
    M, K = xbits.shape
    x = from_bits(xbits)
    s_ld = s_ld or max(4, (M + 3) // 4 * 4)
    q = torch.full((M, K), SENTINEL_U8, dtype=torch.uint8, device="cuda")
    s = torch.full((K // 128, s_ld), SENTINEL_F32, dtype=torch.float32, device="cuda")
    lib.moe_quant_fp8(x, q, s, s_ld)
    torch.cuda.synchronize()
    return u8(q), s.cpu().numpy()


def _assert_quant_equal(lib, xbits):
    q, s = _gpu_quant(lib, xbits)
    rq, rs = oracle.quant_1x128(oracle.bf16_decode(xbits).astype(np.float32))
    M = xbits.shape[0]
    assert np.array_equal(s[:, :M], rs), "scales differ"
    assert (s[:, M:] == SENTINEL_F32).all(), "scale padding columns were written"
    mism = np.nonzero(q != rq)
    assert mism[0].size == 0, f"{mism[0].size} codes differ, first at {mism[0][0]},{mism[1][0]}"


def test_quant_tiny_config_bitexact(lib):
    _assert_quant_equal(lib, activations_bits("c1", 64))


def test_quant_every_bf16_value(lib):
    # Every finite bf16 value with |v| <= 448 (the range a block can hold once its
    # amax is 448), 127 per block next to a 448 that pins s = 1, so q = e4m3(v).
    allv = oracle.bf16_decode(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    keep = np.isfinite(allv) & (np.abs(allv) <= 448.0)
    vals = np.arange(65536, dtype=np.uint32).astype(np.uint16)[keep]
    n_blocks = -(-vals.size // 127)
    blocks = np.full((n_blocks, 128), 0, dtype=np.uint16)
    blocks[:, 0] = oracle.bf16_encode(np.array([448.0]))[0]
    flat = blocks[:, 1:].reshape(-1)
    flat[:vals.size] = vals
    blocks[:, 1:] = flat.reshape(n_blocks, 127)
    rows = -(-n_blocks // 4)
    xb = np.zeros((rows * 4, 128), dtype=np.uint16)
    xb[:n_blocks] = blocks
    xb = xb.reshape(rows, 512)
    q, s = _gpu_quant(lib, xb)
    assert (s[:, :n_blocks // 4] == 1.0).all()
    ref = oracle.e4m3_encode(oracle.bf16_decode(xb))
    assert np.array_equal(q, ref)


def test_quant_division_every_bf16_under_many_scales(lib):
    # The quotient x / s must be the correctly rounded float32 division for every
    # scale: 48 block maxima spread over the exponent range with random
    # mantissas give 48 scales s = fp32(amax / 448); each block pairs its
    # maximum with every finite bf16 value of smaller magnitude, both signs.
    rng = np.random.default_rng(41)
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    allv = oracle.bf16_decode(allbits)
    fin = np.isfinite(allv)
    exps = rng.integers(-20, 100, 48)
    mants = rng.integers(0, 128, 48)
    mants[:4] = [0, 127, 64, 1]
    blocks = []
    for e, m in zip(exps, mants):
        amax_bits = np.uint16(((int(e) + 127) << 7) | int(m))
        amax = float(oracle.bf16_decode(np.array([amax_bits]))[0])
        vals = allbits[fin & (np.abs(allv) <= amax)]
        nb = -(-vals.size // 127)
        b = np.zeros((nb, 128), np.uint16)
        b[:, 0] = amax_bits
        flat = np.zeros(nb * 127, np.uint16)
        flat[:vals.size] = vals
        b[:, 1:] = flat.reshape(nb, 127)
        blocks.append(b)
    blocks = np.concatenate(blocks)
    pad = (-blocks.shape[0]) % 4
    blocks = np.concatenate([blocks, np.zeros((pad, 128), np.uint16)])
    xb = blocks.reshape(-1, 512)
    _assert_quant_equal(lib, xb)


def test_quant_scale_every_bf16_block_maximum(lib):
    # s = fp32(max(amax, 1e-4) / 448) for every finite bf16 magnitude as a
    # block's maximum (with its negative in the block too): scales and codes
    # bit-exact against the oracle's float32 division.
    allbits = np.arange(0x7F80, dtype=np.uint32).astype(np.uint16)      # +0 .. max finite
    nb = allbits.size
    blocks = np.zeros((nb + (-nb) % 4, 128), np.uint16)
    blocks[:nb, 0] = allbits
    blocks[:nb, 1] = allbits | 0x8000
    blocks[:nb, 2] = allbits >> 1
    _assert_quant_equal(lib, blocks.reshape(-1, 512))


def test_quant_edge_cases(lib):
    rng = np.random.default_rng(5)
    M, K = 37, 384                     # M not a multiple of 4, three blocks
    x = rng.standard_normal((M, K))
    x[0] = 0.0                          # all-zero row: floor scale, zero codes
    x[1, :128] = -0.0                   # negative zeros keep their sign
    x[2] *= 1e-30                       # below the floor: amax < 1e-4
    x[3] *= 1e4                         # large values
    x[4, 5] = 3.0e38                    # near the bf16 maximum
    x[5, :] = 2.0 ** -20                # constant block
    x[6, 130] = -7.0                    # negative amax
    xb = oracle.bf16_encode(x)
    _assert_quant_equal(lib, xb)
    q, s = _gpu_quant(lib, xb)
    assert (q[0] == 0).all() and (q[1, :128] == 0x80).all()
    assert q[6, 130] == 0xFE


def test_quant_decode_batch_full_size(lib):
    r = synth.make_routing(synth.get_config("c4"))
    _assert_quant_equal(lib, activations_bits("c4", r["T"]))


def test_quant_prefill_outliers_sample(lib):
    # the prefill activations carry 1% outliers at 20x
    _assert_quant_equal(lib, activations_bits("c3", 1000))


def test_weight_quant_bitexact(lib):
    cfg = synth.get_config("c1")
    w = torch.stack([synth.make_expert_weights(cfg, "w13", e, device="cuda") for e in range(cfg.E)])
    q = torch.empty(w.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty((cfg.E, w.shape[1] // 128, w.shape[2] // 128), dtype=torch.float32, device="cuda")
    lib.moe_quant_weight_fp8(w, q, s)
    rq, rs = oracle_weights("c1", "w13", tuple(range(cfg.E)))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(u8(q), rq)


def test_weight_quant_full_size_expert(lib):
    cfg = synth.get_config("c2")
    w = synth.make_expert_weights(cfg, "w2", 1, device="cuda")[None]
    q = torch.empty(w.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty((1, cfg.H // 128, cfg.I // 128), dtype=torch.float32, device="cuda")
    lib.moe_quant_weight_fp8(w, q, s)
    rq, rs = oracle_weights("c2", "w2", (1,))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(u8(q), rq)


def _gpu_quant_ue8m0(lib, xbits, s_ld=None):
    M, K = xbits.shape
    x = from_bits(xbits)
    s_ld = s_ld or max(4, (M + 3) // 4 * 4)
    q = torch.full((M, K), SENTINEL_U8, dtype=torch.uint8, device="cuda")
    s = torch.full((K // 128, s_ld), SENTINEL_F32, dtype=torch.float32, device="cuda")
    e8 = torch.full((K // 128, s_ld), 0xA5, dtype=torch.uint8, device="cuda")
    lib.moe_quant_fp8_ue8m0(x, q, s, e8, s_ld)
    torch.cuda.synchronize()
    return u8(q), s.cpu().numpy(), e8.cpu().numpy()


def _assert_ue8m0_equal(lib, xbits):
    q, s, e8 = _gpu_quant_ue8m0(lib, xbits)
    rq, rs, rb = oracle.quant_1x128_ue8m0(oracle.bf16_decode(xbits).astype(np.float32))
    M = xbits.shape[0]
    assert np.array_equal(s[:, :M], rs), "scales differ"
    assert np.array_equal(e8[:, :M], rb), "scale bytes differ"
    assert (s[:, M:] == SENTINEL_F32).all() and (e8[:, M:] == 0xA5).all(), "padding columns written"
    mism = np.nonzero(q != rq)
    assert mism[0].size == 0, f"{mism[0].size} codes differ, first at {mism[0][0]},{mism[1][0]}"


def test_quant_ue8m0_configs_bitexact(lib):
    # power-of-two (UE8M0) block scales: codes, scales and exponent bytes equal
    # the oracle's on the tiny config and a prefill sample with 20x outliers
    _assert_ue8m0_equal(lib, activations_bits("c1", 64))
    _assert_ue8m0_equal(lib, activations_bits("c3", 600))


def test_quant_ue8m0_every_bf16_value_under_three_scales(lib):
    # blocks whose maximum is 448 * 2^j hold every finite bf16 magnitude <= 448
    # scaled by 2^j (both signs): s = 2^j and q = e4m3(x / 2^j) exactly
    allv = oracle.bf16_decode(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    vals = allv[np.isfinite(allv) & (np.abs(allv) <= 448.0)]
    for j in (-9, 0, 5):
        v = oracle.bf16_encode(vals * 2.0 ** j)
        nb = -(-v.size // 127)
        blocks = np.zeros((nb + (-nb) % 4, 128), np.uint16)
        blocks[:nb, 0] = oracle.bf16_encode(np.array([448.0 * 2.0 ** j]))[0]
        flat = np.zeros(nb * 127, np.uint16)
        flat[:v.size] = v
        blocks[:nb, 1:] = flat.reshape(nb, 127)
        _assert_ue8m0_equal(lib, blocks.reshape(-1, 512))


def test_quant_ue8m0_edge_cases(lib):
    rng = np.random.default_rng(8)
    M, K = 21, 384
    x = rng.standard_normal((M, K))
    x[0] = 0.0                          # all zero: floor scale 2^-22, zero codes
    x[1, :128] = -0.0
    x[2] *= 1e-30                       # below the floor
    x[3] *= 1e4
    x[4, 5] = 3.0e38                    # near the bf16 maximum: s = 2^120
    x[5, :] = 2.0 ** -20
    x[6, 130] = -7.0
    x[7, 256:] = 448.0                  # exactly 448: s = 1
    x[8, 256:] = 448.0 * (1 + 2 ** -7)  # just above: s = 2
    _assert_ue8m0_equal(lib, oracle.bf16_encode(x))
    q, s, e8 = _gpu_quant_ue8m0(lib, oracle.bf16_encode(x))
    assert s[0, 0] == np.float32(2.0 ** -22) and e8[0, 0] == 105
    assert s[2, 7] == 1.0 and s[2, 8] == 2.0


def test_quant_non_finite_inputs(lib):
    # NaN elements are left out of the block maximum and encode to 0x7F; a block
    # of NaNs takes the floor scale; an infinite element makes the block's scale
    # inf (UE8M0 byte 0xFF): finite elements become signed zeros, the infinite
    # one NaN.  Both scale readings, bit for bit against the oracle.
    rng = np.random.default_rng(9)
    M, K = 9, 384
    x = rng.standard_normal((M, K))
    x[0, 7] = np.nan
    x[1, :128] = np.nan
    x[2, 5] = np.inf
    x[3, 200] = -np.inf
    x[4, 130:140] = np.nan
    x[4, 300] = np.inf
    x[5, 256:] = -np.inf
    xb = oracle.bf16_encode(x)
    xb[6, 10] = 0xFFC0                  # NaNs with the sign bit set encode to 0x7F too
    xb[6, 140] = 0xFF81
    _assert_quant_equal(lib, xb)
    _assert_ue8m0_equal(lib, xb)
    q, s = _gpu_quant(lib, xb)
    assert q[0, 7] == 0x7F and (q[1, :128] == 0x7F).all() and np.isinf(s[0, 2])
    assert q[6, 10] == 0x7F and q[6, 140] == 0x7F
    _, _, e8 = _gpu_quant_ue8m0(lib, xb)
    assert e8[0, 2] == 255 and e8[1, 3] == 255 and e8[2, 5] == 255


def test_quant_flag_selects_power_of_two_scales(lib):
    # moe_quant_fp8 with MOE_QUANT_UE8M0 writes what moe_quant_fp8_ue8m0 writes
    xb = activations_bits("c3", 64)
    x = from_bits(xb)
    q = torch.full((64, xb.shape[1]), SENTINEL_U8, dtype=torch.uint8, device="cuda")
    s = torch.full((xb.shape[1] // 128, 64), SENTINEL_F32, dtype=torch.float32, device="cuda")
    lib.moe_quant_fp8(x, q, s, flags=lib.MOE_QUANT_UE8M0)
    torch.cuda.synchronize()
    rq, rs, _ = oracle.quant_1x128_ue8m0(oracle.bf16_decode(xb).astype(np.float32))
    assert np.array_equal(u8(q), rq) and np.array_equal(s.cpu().numpy(), rs)


def test_weight_quant_ue8m0_bitexact(lib):
    # power-of-two tile scales: codes, scales and exponent bytes equal the
    # oracle's for every expert of the tiny config and one full-size W2 expert
    for name, which, experts in (("c1", "w13", range(4)), ("c1", "w2", range(4)), ("c2", "w2", (1,))):
        cfg = synth.get_config(name)
        for e in experts:
            wb = synth.make_expert_weights(cfg, which, e, device="cuda")
            N, K = wb.shape
            q = torch.full((1, N, K), SENTINEL_U8, dtype=torch.uint8, device="cuda")
            s = torch.full((1, N // 128, K // 128), SENTINEL_F32, dtype=torch.float32, device="cuda")
            e8 = torch.full((1, N // 128, K // 128), 0xA5, dtype=torch.uint8, device="cuda")
            lib.moe_quant_weight_fp8_ue8m0(wb[None], q, s, e8)
            torch.cuda.synchronize()
            rq, rs, rb = oracle.quant_128x128_ue8m0(oracle.bf16_decode(bits(wb)).astype(np.float32))
            assert np.array_equal(u8(q)[0], rq), (name, which, e)
            assert np.array_equal(s.cpu().numpy()[0], rs) and np.array_equal(e8.cpu().numpy()[0], rb)
