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
