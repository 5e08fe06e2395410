"""Python binding of libmoe_fp8.so, the GB300 (sm_103a) routed-expert FP8 MoE FFN.

Argument marshalling only: every step runs in the library's CUDA kernels;
PyTorch supplies device memory and the current stream.  Each function has the
name of the C entry point it calls (see include/moe_fp8.h for the definitions,
layouts and error rules).  A non-zero status raises ``MoeError``.

The library is built in-tree by ``fp8_grouped_expert_x128_gb300/_build.py``
(``__graft_entry__.build()`` does it).  Importing this package without the
built library raises ImportError: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_fp8.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python fp8_grouped_expert_x128_gb300/_build.py` "
        "(the CUDA library is the only implementation; there is no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------- constants
MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_OVERFLOW = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_BAD_INDEX = -6
MOE_DEV_OVERFLOW, MOE_DEV_TIMEOUT, MOE_DEV_BAD_INDEX = 0x1, 0x2, 0x4
MOE_LAYOUT_MASKED, MOE_LAYOUT_CONTIG = 0, 1
MOE_GEMM_DEFAULT = 0
MOE_GEMM_FORCE_TOKENS_M = 0x1
MOE_GEMM_FORCE_WEIGHTS_M = 0x2
MOE_FFN_FUSE_SWIGLU = 0x4
MOE_GEMM_CTA_PAIR = 0x8
MOE_FFN_UE8M0 = 0x10
MOE_GEMM_EARLY_WEIGHTS = 0x20
MOE_GEMM_DEBUG_STALL = 0x100
MOE_QUANT_UE8M0 = 0x1
MOE_COMBINE_ACCUMULATE = 0x1

EXPORTED = [
    "moe_status_string", "moe_version", "moe_read_device_status", "moe_quant_fp8",
    "moe_quant_weight_fp8", "moe_contig_rows_bound", "moe_permute", "moe_gemm_fp8_contig",
    "moe_gemm_fp8_masked", "moe_gemm_fp8_masked_variant", "moe_swiglu_quant", "moe_combine", "moe_ffn_workspace_size", "moe_ffn",
    "moe_ffn_noalloc", "moe_ffn_noalloc_capacity", "moe_ffn_kernel_count", "moe_quant_fp8_ue8m0",
    "moe_ue8m0_scale", "moe_quant_weight_fp8_ue8m0", "moe_ue8m0_act_words", "moe_ue8m0_weight_words",
    "moe_pack_ue8m0_act", "moe_pack_ue8m0_weight", "moe_gemm_fp8_contig_ue8m0", "moe_gemm_fp8_masked_ue8m0",
]

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


class moe_ffn_desc(ctypes.Structure):
    _fields_ = [
        ("T", _I64), ("H", _I32), ("I", _I32), ("k", _I32), ("expert_begin", _I32), ("E", _I32),
        ("layout", _I32), ("max_m", _I32), ("expected_m", _I32), ("gemm_flags", _I32),
        ("x", _P), ("topk_ids", _P), ("topk_w", _P), ("w13", _P), ("w13_s", _P), ("w2", _P),
        ("w2_s", _P), ("out", _P), ("err", _P), ("stage_events", _P), ("w13_sf", _P), ("w2_sf", _P),
    ]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_sig("moe_status_string", ctypes.c_char_p, [ctypes.c_int])
_sig("moe_version", ctypes.c_int, [])
_sig("moe_read_device_status", ctypes.c_int,
     [_P, _P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(_I32)])
_sig("moe_quant_fp8", ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _I32, _P, _P])
_sig("moe_quant_fp8_ue8m0", ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _I64, _P, _P])
_sig("moe_ue8m0_scale", ctypes.c_float, [ctypes.c_float, ctypes.POINTER(ctypes.c_uint8)])
_sig("moe_quant_weight_fp8", ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P])
_sig("moe_quant_weight_fp8_ue8m0", ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _P])
_sig("moe_contig_rows_bound", _I64, [_I64, _I32])
_sig("moe_permute", ctypes.c_int,
     [_P, _P, _I64, _P, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _I64, _P, _P, _P, _P,
      _P, _I64, _P, _P])
_sig("moe_gemm_fp8_contig", ctypes.c_int,
     [_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _P, _I64, _I32, _P, _P])
_sig("moe_gemm_fp8_masked", ctypes.c_int,
     [_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I32, _P, _P])
_sig("moe_gemm_fp8_masked_variant", ctypes.c_int, [_I32, _I32, _I32])
_sig("moe_swiglu_quant", ctypes.c_int, [_P, _I64, _I32, _P, _I32, _P, _P, _P, _I64, _I32, _P, _P])
_sig("moe_combine", ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _I32, _I32, _P, _I64, _I32, _P, _I64, _P, _P])
_sig("moe_ue8m0_act_words", _I64, [_I64, _I64, _I64])
_sig("moe_ue8m0_weight_words", _I64, [_I64, _I64, _I64])
_sig("moe_pack_ue8m0_act", ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P])
_sig("moe_pack_ue8m0_weight", ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P])
_sig("moe_gemm_fp8_contig_ue8m0", ctypes.c_int,
     [_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _P, _I64, _I32, _P, _P])
_sig("moe_gemm_fp8_masked_ue8m0", ctypes.c_int,
     [_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I32, _P, _P])
_sig("moe_ffn_workspace_size", ctypes.c_size_t, [ctypes.POINTER(moe_ffn_desc)])
_sig("moe_ffn_kernel_count", ctypes.c_int, [ctypes.POINTER(moe_ffn_desc)])
_sig("moe_ffn", ctypes.c_int, [ctypes.POINTER(moe_ffn_desc), _P, ctypes.c_size_t, _P])
_sig("moe_ffn_noalloc", ctypes.c_int, [ctypes.POINTER(moe_ffn_desc), _P])
_sig("moe_ffn_noalloc_capacity", ctypes.c_size_t, [])


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} ({status})")


def moe_status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()


def moe_version() -> int:
    return _lib.moe_version()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _dev(t, dtype=None, name="tensor"):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")


_U8 = (torch.uint8, torch.float8_e4m3fn)


def _u8(t):
    return t.view(torch.uint8) if t is not None and t.dtype == torch.float8_e4m3fn else t


def new_error_word(device=None) -> torch.Tensor:
    """A zeroed device int32 word for the library's device-side error bits."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def moe_read_device_status(err: torch.Tensor, stream=None) -> tuple[int, int]:
    """Synchronise, read and clear the device error word -> (status, raw bits)."""
    st = ctypes.c_int(0)
    bits = _I32(0)
    _check(_lib.moe_read_device_status(_ptr(err), _stream(stream), ctypes.byref(st),
                                       ctypes.byref(bits)), "moe_read_device_status")
    return st.value, bits.value


def moe_contig_rows_bound(assignments: int, E: int) -> int:
    return int(_lib.moe_contig_rows_bound(assignments, E))


def moe_quant_fp8(x, q, s, s_ld=None, flags=0, err=None, stream=None):
    """a1: x bf16 [M, K] -> q uint8 [M, K], s fp32 [K/128, s_ld] (s[kb, m]);
    flags = MOE_QUANT_UE8M0 for power-of-two scales."""
    _dev(x, torch.bfloat16, "x"); _dev(q, _U8, "q"); _dev(s, torch.float32, "s")
    M, K = x.shape
    s_ld = s.shape[-1] if s_ld is None else s_ld
    _check(_lib.moe_quant_fp8(_ptr(x), M, K, x.stride(0), _ptr(_u8(q)), q.stride(0), _ptr(s), s_ld,
                              flags, _ptr(err), _stream(stream)), "moe_quant_fp8")
    return q, s


def moe_quant_fp8_ue8m0(x, q, s, e8=None, s_ld=None, err=None, stream=None):
    """a1 with power-of-two block scales: s fp32 [K/128, s_ld] holds 2^e, e8 uint8
    (optional, same shape) holds e + 127."""
    _dev(x, torch.bfloat16, "x"); _dev(q, _U8, "q"); _dev(s, torch.float32, "s"); _dev(e8, _U8, "e8")
    M, K = x.shape
    s_ld = s.shape[-1] if s_ld is None else s_ld
    _check(_lib.moe_quant_fp8_ue8m0(_ptr(x), M, K, x.stride(0), _ptr(_u8(q)), q.stride(0), _ptr(s),
                                    _ptr(e8), s_ld, _ptr(err), _stream(stream)), "moe_quant_fp8_ue8m0")
    return q, s


def moe_ue8m0_scale(amax: float) -> tuple[float, int]:
    """The UE8M0 block-scale rule for one block maximum (host): (2^e, e + 127)."""
    b = ctypes.c_uint8(0)
    s = float(_lib.moe_ue8m0_scale(ctypes.c_float(amax), ctypes.byref(b)))
    return s, int(b.value)


def moe_quant_weight_fp8(w, q, s, stream=None):
    """a3: w bf16 [E, N, K] -> q uint8 [E, N, K], s fp32 [E, N/128, K/128]."""
    _dev(w, torch.bfloat16, "w"); _dev(q, _U8, "q"); _dev(s, torch.float32, "s")
    E, N, K = w.shape
    assert w.is_contiguous() and q.is_contiguous() and s.is_contiguous()
    _check(_lib.moe_quant_weight_fp8(_ptr(w), E, N, K, _ptr(_u8(q)), _ptr(s), _stream(stream)),
           "moe_quant_weight_fp8")
    return q, s


def moe_quant_weight_fp8_ue8m0(w, q, s, e8=None, stream=None):
    """a3 with power-of-two tile scales: s fp32 [E, N/128, K/128] holds 2^e, e8
    uint8 (optional, same shape) holds e + 127."""
    _dev(w, torch.bfloat16, "w"); _dev(q, _U8, "q"); _dev(s, torch.float32, "s"); _dev(e8, _U8, "e8")
    E, N, K = w.shape
    assert w.is_contiguous() and q.is_contiguous() and s.is_contiguous()
    _check(_lib.moe_quant_weight_fp8_ue8m0(_ptr(w), E, N, K, _ptr(_u8(q)), _ptr(s), _ptr(e8), _stream(stream)),
           "moe_quant_weight_fp8_ue8m0")
    return q, s


def moe_permute(q, s, topk_ids, expert_begin, E, layout, max_m, q_out, s_out, counts, offsets,
                m_indices, row_src, dst_row, rows_capacity=0, s_ld=None, s_out_ld=None, err=None,
                stream=None):
    """a2: token-order q/s -> grouped layout.  See moe_fp8.h for the layouts."""
    T, H = q.shape
    k = topk_ids.shape[1]
    s_ld = s.shape[-1] if s_ld is None else s_ld
    if s_out_ld is None:
        s_out_ld = s_out.shape[-1] if layout == MOE_LAYOUT_CONTIG else max_m
    _check(_lib.moe_permute(_ptr(_u8(q)), _ptr(s), s_ld, _ptr(topk_ids), T, H, k, expert_begin, E,
                            layout, max_m, _ptr(_u8(q_out)), _ptr(s_out), s_out_ld, _ptr(counts),
                            _ptr(offsets), _ptr(m_indices), _ptr(row_src), _ptr(dst_row),
                            rows_capacity, _ptr(err), _stream(stream)), "moe_permute")


def moe_gemm_fp8_contig(A, sA, B, sB, offsets, m_indices, D, sA_ld=None, flags=0, err=None,
                        stream=None):
    """a4/a6, contiguous layout: A [M_cap, K], sA [K/128, sA_ld], B [E, N, K], D [M_cap, N]."""
    E, N, K = B.shape
    M_cap = A.shape[0]
    sA_ld = sA.shape[-1] if sA_ld is None else sA_ld
    _check(_lib.moe_gemm_fp8_contig(_ptr(_u8(A)), A.stride(0), _ptr(sA), sA_ld, _ptr(_u8(B)),
                                    _ptr(sB), _ptr(offsets), _ptr(m_indices), M_cap, E, N, K,
                                    _ptr(D), D.stride(0), flags, _ptr(err), _stream(stream)),
           "moe_gemm_fp8_contig")
    return D


def moe_gemm_fp8_masked(A, sA, B, sB, counts, D, expected_m=0, flags=0, err=None, stream=None):
    """a4/a6, masked layout: A [E, max_m, K], sA [E, K/128, max_m], D [E, max_m, N]."""
    E, max_m, K = A.shape
    N = B.shape[1]
    _check(_lib.moe_gemm_fp8_masked(_ptr(_u8(A)), _ptr(sA), _ptr(_u8(B)), _ptr(sB), _ptr(counts),
                                    E, max_m, N, K, expected_m, _ptr(D), flags, _ptr(err),
                                    _stream(stream)), "moe_gemm_fp8_masked")
    return D


def moe_gemm_fp8_masked_variant(max_m: int, expected_m: int = 0, flags: int = 0) -> int:
    """0 = tokens-as-M kernel; 64/128/256 = weights-as-M token-tile width."""
    return int(_lib.moe_gemm_fp8_masked_variant(max_m, expected_m, flags))


def moe_ue8m0_act_words(groups: int, G: int, K: int) -> int:
    return int(_lib.moe_ue8m0_act_words(groups, G, K))


def moe_ue8m0_weight_words(E: int, N: int, K: int) -> int:
    return int(_lib.moe_ue8m0_weight_words(E, N, K))


def moe_pack_ue8m0_act(s, groups, G, rows, K, sfA, stream=None):
    """Power-of-two fp32 scales in the grouped layout (groups of G rows) -> packed
    UE8M0 words sfA (int32 tensor of moe_ue8m0_act_words(groups, G, K) words)."""
    _dev(s, torch.float32, "s"); _dev(sfA, torch.int32, "sfA")
    _check(_lib.moe_pack_ue8m0_act(_ptr(s), groups, G, rows, K, _ptr(sfA), _stream(stream)), "moe_pack_ue8m0_act")
    return sfA


def moe_pack_ue8m0_weight(s, sfB, K, stream=None):
    """Power-of-two fp32 weight scales [E, N/128, K/128] -> packed records sfB."""
    _dev(s, torch.float32, "s"); _dev(sfB, torch.int32, "sfB")
    E, NB, _ = s.shape
    _check(_lib.moe_pack_ue8m0_weight(_ptr(s), E, NB * 128, K, _ptr(sfB), _stream(stream)), "moe_pack_ue8m0_weight")
    return sfB


def moe_gemm_fp8_contig_ue8m0(A, sfA, sfA_ld, B, sfB, offsets, m_indices, D, flags=0, err=None, stream=None):
    """a4/a6 with packed UE8M0 scales, contiguous layout."""
    E, N, K = B.shape
    _check(_lib.moe_gemm_fp8_contig_ue8m0(_ptr(_u8(A)), A.stride(0), _ptr(sfA), sfA_ld, _ptr(_u8(B)), _ptr(sfB),
                                          _ptr(offsets), _ptr(m_indices), A.shape[0], E, N, K, _ptr(D),
                                          D.stride(0), flags, _ptr(err), _stream(stream)), "moe_gemm_fp8_contig_ue8m0")
    return D


def moe_gemm_fp8_masked_ue8m0(A, sfA, B, sfB, counts, D, expected_m=0, flags=0, err=None, stream=None):
    """a4/a6 with packed UE8M0 scales, masked layout: A [E, max_m, K], D [E, max_m, N]."""
    E, max_m, K = A.shape
    N = B.shape[1]
    _check(_lib.moe_gemm_fp8_masked_ue8m0(_ptr(_u8(A)), _ptr(sfA), _ptr(_u8(B)), _ptr(sfB), _ptr(counts), E, max_m,
                                          N, K, expected_m, _ptr(D), flags, _ptr(err), _stream(stream)),
           "moe_gemm_fp8_masked_ue8m0")
    return D


def moe_swiglu_quant(Y1, q, s, counts=None, max_m=0, m_indices=None, s_ld=0, flags=0, err=None,
                     stream=None):
    """a5: Y1 bf16 [rows, 2I] -> q uint8 [rows, I] + scales (groups of max_m rows when
    ``counts`` is given, else one group of ``s_ld`` rows selected by ``m_indices``);
    flags = MOE_QUANT_UE8M0 for power-of-two scales."""
    two_i = Y1.shape[-1]
    rows = Y1.numel() // two_i
    _check(_lib.moe_swiglu_quant(_ptr(Y1), rows, two_i // 2, _ptr(counts), max_m, _ptr(m_indices),
                                 _ptr(_u8(q)), _ptr(s), s_ld, flags, _ptr(err), _stream(stream)),
           "moe_swiglu_quant")


def moe_combine(Y2, dst_row, topk_w, out, shared=None, flags=0, err=None, stream=None):
    """a7: out[t] = bf16((out[t] if ACCUMULATE) + sum_j w[t,j] * Y2[dst_row[t*k+j]] + shared[t]);
    Y2 viewed as [rows, H]; shared (optional) bf16 [T, H]."""
    H = Y2.shape[-1]
    rows = Y2.numel() // H
    T, k = topk_w.shape
    _dev(shared, torch.bfloat16, "shared")
    _check(_lib.moe_combine(_ptr(Y2), H, rows, _ptr(dst_row), _ptr(topk_w), T, k, H, _ptr(shared),
                            shared.stride(0) if shared is not None else 0, flags, _ptr(out),
                            out.stride(0), _ptr(err), _stream(stream)), "moe_combine")
    return out


def make_ffn_desc(x, topk_ids, topk_w, w13, w13_s, w2, w2_s, out, expert_begin, E, layout,
                  max_m=0, expected_m=0, gemm_flags=0, err=None, stage_events=None, w13_sf=None, w2_sf=None):
    T, H = x.shape
    I = w2.shape[2]
    d = moe_ffn_desc(T=T, H=H, I=I, k=topk_ids.shape[1], expert_begin=expert_begin, E=E,
                     layout=layout, max_m=max_m, expected_m=expected_m, gemm_flags=gemm_flags,
                     x=x.data_ptr(), topk_ids=topk_ids.data_ptr(), topk_w=topk_w.data_ptr(),
                     w13=_u8(w13).data_ptr(), w13_s=w13_s.data_ptr() if w13_s is not None else None,
                     w2=_u8(w2).data_ptr(),
                     w2_s=w2_s.data_ptr() if w2_s is not None else None, out=out.data_ptr(),
                     err=err.data_ptr() if err is not None else None, stage_events=None,
                     w13_sf=w13_sf.data_ptr() if w13_sf is not None else None,
                     w2_sf=w2_sf.data_ptr() if w2_sf is not None else None)
    if stage_events is not None:
        if len(stage_events) != 7:
            raise ValueError("stage_events needs 7 events")
        for ev in stage_events:
            if not ev.cuda_event:          # torch creates the CUDA event on first record
                ev.record()
        arr = (ctypes.c_void_p * len(stage_events))(*[ev.cuda_event for ev in stage_events])
        d._events_keepalive = arr
        d.stage_events = ctypes.cast(arr, ctypes.c_void_p)
    return d


def moe_ffn_kernel_count(desc: moe_ffn_desc) -> int:
    """Kernels one moe_ffn call with `desc` launches (host-only)."""
    n = int(_lib.moe_ffn_kernel_count(ctypes.byref(desc)))
    _check(n if n < 0 else MOE_OK, "moe_ffn_kernel_count")
    return n


def moe_ffn_workspace_size(desc: moe_ffn_desc) -> int:
    return int(_lib.moe_ffn_workspace_size(ctypes.byref(desc)))


def moe_ffn(desc: moe_ffn_desc, workspace: torch.Tensor, stream=None):
    """a8: the whole FFN on one stream; ``workspace`` is a uint8 device tensor of at
    least moe_ffn_workspace_size(desc) bytes, 256-byte aligned."""
    _check(_lib.moe_ffn(ctypes.byref(desc), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_ffn")


def moe_ffn_noalloc(desc: moe_ffn_desc, stream=None):
    """a8 without a workspace argument: the intermediates live in the library's
    fixed device scratch (moe_ffn_noalloc_capacity() bytes, shared by all calls;
    calls that overlap on the GPU race).  For callers that cannot allocate."""
    _check(_lib.moe_ffn_noalloc(ctypes.byref(desc), _stream(stream)), "moe_ffn_noalloc")


def moe_ffn_noalloc_capacity() -> int:
    return int(_lib.moe_ffn_noalloc_capacity())


def alloc_workspace(desc: moe_ffn_desc, device=None) -> torch.Tensor:
    n = moe_ffn_workspace_size(desc)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_ffn_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")
