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


# Guard bands: compute-sanitizer is not available, so an output buffer is carved
# from the front of a larger allocation whose tail holds a sentinel pattern; a
# store past the end of the buffer changes the tail.
GUARD_BYTES = 64 * 1024
_INT_OF = {1: torch.uint8, 2: torch.int16, 4: torch.int32}


class Guarded:
    """A device tensor of `shape`/`dtype` filled with the bit pattern `fill`
    (an int, the element's bits), followed in memory by GUARD_BYTES bytes of
    the same pattern.  `t` is the tensor; `intact()` checks the band."""

    def __init__(self, shape, dtype, fill, device="cuda"):
        n = int(np.prod(shape))
        size = torch.empty((), dtype=dtype).element_size()
        idt = _INT_OF[size]
        guard = GUARD_BYTES // size
        u = int(fill) & ((1 << (8 * size)) - 1)           # the element's bits
        fill = u - (1 << (8 * size)) if size > 1 and u >= (1 << (8 * size - 1)) else u
        self.buf = torch.full((n + guard,), fill, dtype=idt, device=device)
        self.n, self.fill = n, fill
        self.t = self.buf[:n].view(dtype).view(shape)

    def intact(self) -> bool:
        tail = self.buf[self.n:]
        return bool((tail == self.fill).all().item())


def f32_bits(v: float) -> int:
    return int(np.float32(v).view(np.uint32))


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
# With power-of-two (UE8M0) scales a block's scale is up to twice the fp32
# scale, so one E4M3 flip of h moves an output up to twice as far and up to
# twice as many outputs leave the strict bound; the one-flip bound itself is
# unchanged (computed from the oracle's own q2 and s2).
CHAIN_FRAC_UE8M0 = 2e-3


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


def flip_bound(ref: dict, topk_w: np.ndarray, w2q, w2s) -> np.ndarray:
    """Oracle-side bound [T, H] on how far one E4M3 flip of h per routed row can
    move each output: sum_j w_j * max_i(step(q2[r_j, i]) * s2[r_j, i]) * max_i |W2[e_j][n, i]|,
    with step the larger gap to a neighbouring code and W2 dequantised.
    w2q / w2s: per-expert weights, indexable by local expert id (arrays or
    dicts holding at least the experts that own rows)."""
    rows_valid = ref["valid"]
    q2 = ref["q2"]
    I = q2.shape[1]
    KB2 = I // 128
    s2 = ref["s2"]
    if s2.ndim == 3:                                     # masked [E, KB, max_m] -> [KB, rows]
        s2 = s2.transpose(1, 0, 2).reshape(KB2, -1)
    step = e4m3_flip_step(q2, np.repeat(s2.T, 128, axis=1))          # [rows, I]
    rowflip = np.where(rows_valid, step.max(axis=1), 0.0)             # [rows]
    perm = ref["perm"]
    rows = rows_valid.size
    if perm.get("offsets") is None:                      # masked: E blocks of max_m rows
        owner = np.arange(rows) // (rows // len(perm["counts"]))
    else:
        owner = np.asarray(perm["m_indices"])
    experts = [int(e) for e in np.unique(owner[rows_valid])]
    with ThreadPoolExecutor(max_workers=16) as ex:
        colmax = dict(zip(experts, ex.map(lambda e: w2_colmax(w2q[e], w2s[e]), experts)))
    dst = perm["dst_row"].reshape(topk_w.shape)
    T, k = topk_w.shape
    H = next(iter(colmax.values())).shape[0] if colmax else 0
    out = np.zeros((T, H))
    for j in range(k):
        d = dst[:, j]
        ok = d >= 0
        e_of = np.where(ok, owner[np.maximum(d, 0)], -1)
        for e in np.unique(e_of[ok]):
            sel = e_of == e
            out[sel] += (topk_w[sel, j] * rowflip[d[sel]])[:, None] * colmax[int(e)]
    return out


def check_tol_chain(got_bits: np.ndarray, ref_bits: np.ndarray, extra: np.ndarray, what: str = "",
                    max_frac: float = CHAIN_FRAC):
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
    assert frac <= max_frac, f"{what}: {frac:.2e} of outputs outside the strict bound"
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


def oracle_chain_chunked(x_bits, topk_ids, topk_w, expert_begin, E, layout, max_m,
                         w13_q, w13_s, w2_q, w2_s, chunk=1024, workers=16, ue8m0=False) -> dict:
    """``oracle.ffn_chain`` computed row chunk by row chunk in a thread pool, for
    the full-size configs (the weights may be dicts holding only the experts
    that own rows: no other expert's weights are read).  It calls only the
    oracle's own stage functions and
    returns the same dict, bit for bit: every stage is row-independent (the
    quantisations are per row, each GEMM row depends on that row alone, and a
    128-term sum of E4M3 products is exact in float64 whatever the summation
    order, so the row count of a GEMM call cannot change a row's result).  The
    permutation and the combine run once, as in ffn_chain.  Pinned against
    ffn_chain on the tiny configs in tests/test_oracle_chain.py."""
    T, H = x_bits.shape
    I = (w2_q[next(iter(w2_q))] if isinstance(w2_q, dict) else w2_q[0]).shape[1]
    pool = ThreadPoolExecutor(max_workers=workers)
    try:
        spans = [(a, min(a + chunk, T)) for a in range(0, T, chunk)]
        quant = (lambda v: oracle.quant_1x128_ue8m0(v)[:2]) if ue8m0 else oracle.quant_1x128
        parts = list(pool.map(lambda sp: quant(oracle.bf16_decode(x_bits[sp[0]:sp[1]]).astype(np.float32)), spans))
        q = np.concatenate([a for a, _ in parts]) if parts else np.zeros((0, H), np.uint8)
        s = np.concatenate([b for _, b in parts], axis=1) if parts else np.zeros((H // 128, 0), np.float32)
        p = oracle.permute(topk_ids, expert_begin, E, layout, max_m, q=q, s=s)
        rows = p["rows"]
        if layout == "masked":
            sA = p["s"].transpose(1, 0, 2).reshape(H // 128, rows)
            owner = np.repeat(np.arange(E), max_m)
            valid = (np.arange(rows) % max_m) < np.repeat(p["counts"], max_m)
        else:
            sA = p["s"]
            owner = p["m_indices"]
            valid = owner >= 0
        tasks = []
        for e in range(E):
            r = np.nonzero(valid & (owner == e))[0]
            tasks += [(e, r[a:a + chunk]) for a in range(0, len(r), chunk)]

        def run(task):
            e, r = task
            y1 = oracle.bf16_encode(oracle.gemm_block_scaled(p["q"][r], sA[:, r], w13_q[e], w13_s[e]))
            q2, s2 = oracle.swiglu_quant(y1, ue8m0)
            y2 = oracle.bf16_encode(oracle.gemm_block_scaled(q2, s2, w2_q[e], w2_s[e]))
            return r, y1, q2, s2, y2

        y1 = np.zeros((rows, 2 * I), np.uint16)
        q2 = np.zeros((rows, I), np.uint8)
        s2 = np.zeros((I // 128, rows), np.float32)
        y2 = np.zeros((rows, H), np.uint16)
        for r, a, b, c, d in pool.map(run, tasks):
            y1[r], q2[r], s2[:, r], y2[r] = a, b, c, d
    finally:
        pool.shutdown()
    out = oracle.combine(y2, p["dst_row"], topk_w)
    if layout == "masked":
        s2 = np.ascontiguousarray(s2.reshape(I // 128, E, max_m).transpose(1, 0, 2))
    return dict(q=q, s=s, perm=p, y1=y1, valid=valid, q2=q2, s2=s2, y2=y2, out=out)


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
