"""CPU oracle for the routed-expert FP8 MoE FFN -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct statement of what the hot path computes,
in numpy with float64 accumulation.  Only the tests, the smoke check and the
benchmark's CPU-baseline / reference legs may import it; the library itself
never does, and this package imports nothing from the library (no shared
kernels, tables, constants or helpers).

What the pages fix, and where the rest comes from:

* "Deploying DeepSeek on GB200 NVL72 with PD and Large Scale EP (Part I)",
  section "Implementation details", DeepGEMM bullet: an FP8 GEMM library whose
  API adds quantisation and packing of the input scales, running on UMMA.
* "Deploying DeepSeek with PD Disaggregation and Large-Scale Expert
  Parallelism on 96 H100 GPUs", section "DeepGEMM integration": two grouped-GEMM
  functions for MoE, one for prefill (paired with DeepEP normal dispatch) and
  one for decode (paired with the CUDA-Graph-compatible low-latency dispatch,
  section "Expert parallelism based on DeepEP", mode table).
* The pages do not state the arithmetic.  This library's problem statement
  fixes it: per-token 1x128 E4M3 activation quantisation with fp32 scales,
  128x128 block-scaled E4M3 weights, a contiguous (prefill) and a masked
  (decode) grouped layout, SwiGLU with FP8 requantisation, a second grouped
  GEMM and a top-k-weighted combine.  Every point where that statement is
  silent is a named reading in the function that takes it.

Modules: ``fp8`` (E4M3 and bf16 codecs), ``ffn`` (the stages and their chain).
Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, brute force, library special cases, invariants).
"""
from .fp8 import (bf16_decode, bf16_encode, e4m3_decode, e4m3_encode,
                  e4m3_encode_bruteforce, E4M3_MAX)
from .ffn import (quant_1x128, quant_1x128_ue8m0, quant_128x128, quant_128x128_ue8m0, permute,
                  gemm_block_scaled,
                  gemm_masked, gemm_contig, swiglu, swiglu_quant, combine,
                  ffn_chain, SCALE_FLOOR, pack_ue8m0_act, pack_ue8m0_weight)

__all__ = [
    "bf16_decode", "bf16_encode", "e4m3_decode", "e4m3_encode", "e4m3_encode_bruteforce",
    "E4M3_MAX", "quant_1x128", "quant_1x128_ue8m0", "quant_128x128", "quant_128x128_ue8m0", "permute",
    "gemm_block_scaled",
    "gemm_masked", "gemm_contig", "swiglu", "swiglu_quant", "combine", "ffn_chain",
    "SCALE_FLOOR", "pack_ue8m0_act", "pack_ue8m0_weight",
]
