"""Helpers shared by the GPU parity tests: tensor <-> oracle conversions, the
acceptance tolerance, sentinels, and cached oracle-quantised expert weights.

Inputs always come from ``synth`` (the seeded generator); expected values
always come from ``oracle``.  Nothing here feeds a CUDA result to the oracle."""
from __future__ import annotations

import functools
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import synth

# Acceptance bound for floating-point outputs (GEMM, FFN, combine):
#   |gpu - ref| <= 2^-7 * |ref| + 1e-3 * rms(ref), elementwise.
REL_TOL = 2.0 ** -7
RMS_TOL = 1e-3

SENTINEL_U8 = 0xA5
SENTINEL_BF16 = 0x7E57          # a finite bf16 (~7.1e37) no output takes
SENTINEL_F32 = -12345.0


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 numpy bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def check_tol(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = ""):
    """Assert the acceptance bound between a GPU bf16 result and the oracle's."""
    got = oracle.bf16_decode(got_bits)
    ref = oracle.bf16_decode(ref_bits)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite GPU output"
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    bound = REL_TOL * np.abs(ref) + RMS_TOL * rms
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu {got[i]!r} ref {ref[i]!r} bound {bound[i]!r}")
    return float((err / np.maximum(bound, 1e-30)).max()) if err.size else 0.0


# End to end, an FP8 requantisation sits between the two GEMMs: a one-ulp bf16
# difference in Y1 (fp32 vs float64 accumulation) or a few-ulp float32
# difference in h (expf) can flip one E4M3 code of h, which moves that routed
# row's output by one E4M3 step of one term.  Stage-fed checks hold every stage
# to the strict bound.  End to end, at most CHAIN_FRAC of the outputs may leave
# the strict bound, and every output must stay within the strict bound plus
# the largest effect one such flip per routed row can have (computed by the
# oracle alone, see flip_bound).
CHAIN_FRAC = 1e-3


def e4m3_flip_step(q2: np.ndarray, s2_cols: np.ndarray) -> np.ndarray:
    """Per element of h: the larger gap from its E4M3 code to a neighbouring
    code, times the element's block scale (s2_cols: the scale of each column)."""
    mag = (q2 & 0x7F).astype(np.int64)
    here = oracle.e4m3_decode(mag.astype(np.uint8))
    up = np.abs(oracle.e4m3_decode(np.minimum(mag + 1, 0x7E).astype(np.uint8)) - here)
    dn = np.abs(here - oracle.e4m3_decode(np.maximum(mag - 1, 0).astype(np.uint8)))
    return np.maximum(up, dn) * s2_cols


def w2_colmax(w2q_e: np.ndarray, w2s_e: np.ndarray) -> np.ndarray:
    """max_i |W2[n, i]| of one expert's dequantised W2, per output column n."""
    return np.abs(oracle.e4m3_decode(w2q_e) * np.repeat(np.repeat(w2s_e, 128, 0), 128, 1)).max(axis=1)


def flip_bound(ref: dict, topk_w: np.ndarray, w2q: np.ndarray, w2s: np.ndarray) -> np.ndarray:
    """Oracle-side bound [T, H] on how far one E4M3 flip of h per routed row can
    move each output: sum_j w_j * max_i(step(q2[r_j, i]) * s2[r_j, i]) * max_i |W2[e_j][n, i]|,
    with step the larger gap to a neighbouring code and W2 dequantised."""
    rows_valid = ref["valid"]
    q2 = ref["q2"]
    I = q2.shape[1]
    KB2 = I // 128
    s2 = ref["s2"]
    if s2.ndim == 3:                                     # masked [E, KB, max_m] -> [KB, rows]
        s2 = s2.transpose(1, 0, 2).reshape(KB2, -1)
    step = e4m3_flip_step(q2, np.repeat(s2.T, 128, axis=1))          # [rows, I]
    rowflip = np.where(rows_valid, step.max(axis=1), 0.0)             # [rows]
    E = w2q.shape[0]
    colmax = np.stack([w2_colmax(w2q[e], w2s[e]) for e in range(E)])  # [E, H]
    dst = ref["perm"]["dst_row"].reshape(topk_w.shape)
    T, k = topk_w.shape
    rows_per_e = rows_valid.size // E if ref["perm"].get("offsets") is None else None
    out = np.zeros((T, colmax.shape[1]))
    for j in range(k):
        d = dst[:, j]
        ok = d >= 0
        if rows_per_e is not None:
            e_of = d // rows_per_e
        else:
            e_of = ref["perm"]["m_indices"][np.maximum(d, 0)]
        out[ok] += (topk_w[ok, j] * rowflip[d[ok]])[:, None] * colmax[e_of[ok]]
    return out


def check_tol_chain(got_bits: np.ndarray, ref_bits: np.ndarray, extra: np.ndarray, what: str = ""):
    got = oracle.bf16_decode(got_bits)
    ref = oracle.bf16_decode(ref_bits)
    assert np.isfinite(got).all(), f"{what}: non-finite GPU output"
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    strict_b = REL_TOL * np.abs(ref) + RMS_TOL * rms
    strict = err > strict_b
    beyond = err > strict_b + extra
    frac = strict.mean()
    if beyond.any():
        i = np.unravel_index(np.argmax(err - strict_b - extra), err.shape)
        raise AssertionError(f"{what}: {beyond.sum()} outputs beyond the one-flip bound; worst at {i}: "
                             f"gpu {got[i]!r} ref {ref[i]!r} strict {strict_b[i]!r} flip {extra[i]!r}")
    assert frac <= CHAIN_FRAC, f"{what}: {frac:.2e} of outputs outside the strict bound"
    return frac


def check_swiglu(q, s, y1_bits, valid_rows, ref_q=None, ref_s=None):
    """SwiGLU+quant acceptance: scales within 4 float32 ulp; an FP8 code may
    differ only by one step, only where the oracle's h/s lies within 2^-19
    (relative) of the rounding midpoint between the two codes (or the scale
    moved), and on fewer than 1e-4 of the codes."""
    if ref_q is None:
        ref_q, ref_s = oracle.swiglu_quant(y1_bits[valid_rows])
    gq = q[valid_rows]
    ulp = np.spacing(ref_s.astype(np.float32))
    assert (np.abs(s.astype(np.float64) - ref_s) <= 4 * ulp).all(), "scales beyond 4 ulp"
    mism = np.nonzero(gq != ref_q)
    frac = mism[0].size / max(ref_q.size, 1)
    assert frac < 1e-4, f"code mismatch fraction {frac}"
    if mism[0].size:
        h = oracle.swiglu(y1_bits[valid_rows])
        for r, c in zip(*mism):
            a, b = int(gq[r, c]), int(ref_q[r, c])
            assert (a & 0x80) == (b & 0x80) and abs((a & 0x7F) - (b & 0x7F)) == 1, (r, c, a, b)
            v = float(h[r, c]) / float(ref_s[c // 128, r])
            mid = (abs(oracle.e4m3_decode(np.uint8(a))) + abs(oracle.e4m3_decode(np.uint8(b)))) / 2
            near = abs(abs(v) - mid) <= 2.0 ** -19 * mid
            assert near or s[c // 128, r] != ref_s[c // 128, r], (r, c, a, b, v, mid)
    return frac


def rand_codes(rng, shape) -> np.ndarray:
    """Random E4M3 codes with NaN codes replaced (finite operands only)."""
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3A
    return c


def gen_device():
    return "cuda" if torch.cuda.is_available() else "cpu"


def expert_bf16(cfg, which, e, device=None) -> torch.Tensor:
    return synth.make_expert_weights(cfg, which, e, device=device or gen_device())


def _oracle_quant_expert(args):
    cfg, which, e = args
    w = oracle.bf16_decode(bits(expert_bf16(cfg, which, e))).astype(np.float32)
    return oracle.quant_128x128(w)


@functools.lru_cache(maxsize=16)
def oracle_weights(cfg_name: str, which: str, experts: tuple) -> tuple[np.ndarray, np.ndarray]:
    """Oracle-quantised weights of the listed experts: (q [n, N, K], s [n, N/128, K/128])."""
    cfg = synth.get_config(cfg_name)
    with ThreadPoolExecutor(max_workers=16) as ex:
        res = list(ex.map(_oracle_quant_expert, [(cfg, which, e) for e in experts]))
    return np.stack([r[0] for r in res]), np.stack([r[1] for r in res])


def routing(cfg_name: str) -> dict:
    return synth.make_routing(synth.get_config(cfg_name))


def activations_bits(cfg_name: str, T: int) -> np.ndarray:
    return bits(synth.make_activations(synth.get_config(cfg_name), T, device=gen_device()))
