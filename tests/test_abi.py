"""The C-ABI library: it builds, loads without a GPU, exports every entry point
include/moe_fp8.h declares, and rejects bad arguments on the host before any
CUDA call (no compute is attempted here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def so():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path), path


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_hot_path(so):
    names = _declared_functions()
    for required in ("moe_quant_fp8", "moe_permute", "moe_gemm_fp8_contig", "moe_gemm_fp8_masked",
                     "moe_swiglu_quant", "moe_combine", "moe_ffn", "moe_ffn_workspace_size",
                     "moe_read_device_status", "moe_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(so):
    lib, path = so
    missing = [n for n in sorted(_declared_functions()) if not hasattr(lib, n)]
    assert not missing, missing
    import fp8_grouped_expert_x128_gb300 as moe
    assert set(moe.EXPORTED) <= _declared_functions()


def test_status_strings_and_version(so):
    import fp8_grouped_expert_x128_gb300 as moe
    assert moe.moe_status_string(0) == "MOE_OK"
    assert moe.moe_status_string(-5) == "MOE_ERR_TIMEOUT"
    assert moe.moe_status_string(12345) == "MOE_ERR_UNKNOWN"
    assert moe.moe_version() >= 200


def test_host_side_argument_validation(so):
    lib, _ = so
    lib.moe_quant_fp8.restype = ctypes.c_int
    i64, p = ctypes.c_int64, ctypes.c_void_p
    # K not a multiple of 128 -> rejected before any CUDA call
    i32 = ctypes.c_int32
    rc = lib.moe_quant_fp8(p(16), i64(4), i64(100), i64(100), p(16), i64(100), p(16), i64(4), i32(0), None, None)
    assert rc == -1
    # null pointers
    rc = lib.moe_quant_fp8(None, i64(4), i64(128), i64(128), None, i64(128), None, i64(4), i32(0), None, None)
    assert rc == -1
    # misaligned pointer
    rc = lib.moe_quant_fp8(p(18), i64(4), i64(128), i64(128), p(16), i64(128), p(16), i64(4), i32(0), None, None)
    assert rc == -1
    # unknown flag bits
    rc = lib.moe_quant_fp8(p(16), i64(4), i64(128), i64(128), p(16), i64(128), p(16), i64(4), i32(0x6), None, None)
    assert rc == -1
    # empty input is a no-op
    rc = lib.moe_quant_fp8(None, i64(0), i64(128), i64(128), None, i64(128), None, i64(0), i32(0), None, None)
    assert rc == 0
    lib.moe_combine.restype = ctypes.c_int
    # unknown combine flag bits; a misaligned shared row pointer
    rc = lib.moe_combine(p(16), i64(256), i64(8), p(16), p(16), i64(4), i32(2), i32(256), None, i64(0), i32(2),
                         p(16), i64(256), None, None)
    assert rc == -1
    rc = lib.moe_combine(p(16), i64(256), i64(8), p(16), p(16), i64(4), i32(2), i32(256), p(18), i64(256), i32(0),
                         p(16), i64(256), None, None)
    assert rc == -1
    lib.moe_gemm_fp8_masked.restype = ctypes.c_int
    rc = lib.moe_gemm_fp8_masked(p(16), p(16), p(16), p(16), p(16), i32(4), i32(128), i32(200),
                                 i32(256), i32(0), p(16), i32(0), None, None)
    assert rc == -1                                   # N % 128 != 0
    rc = lib.moe_permute(p(16), p(16), i64(4), p(16), i64(4), ctypes.c_int32(256), ctypes.c_int32(2),
                         i32(0), i32(2000), i32(0), i32(128), p(16), p(16), i64(128), p(16), None,
                         None, p(16), p(16), i64(0), None, None)
    assert rc == -1                                   # E above the 1024 limit


def test_contig_bound_and_workspace_plan(so):
    import fp8_grouped_expert_x128_gb300 as moe
    assert moe.moe_contig_rows_bound(0, 4) == 3 * 128
    assert moe.moe_contig_rows_bound(32768, 9) == (32768 + 9 * 127) // 128 * 128
    d = moe.moe_ffn_desc(T=64, H=256, I=128, k=2, expert_begin=0, E=4, layout=0, max_m=128)
    ws = moe.moe_ffn_workspace_size(d)
    rows = 4 * 128
    assert ws >= rows * 256 + rows * 256 * 2 + rows * 128 + rows * 256 * 2
    assert ws % 256 == 0
    d.H = 200
    assert moe.moe_ffn_workspace_size(d) == 0         # invalid descriptor


def test_register_split_kernels_compile_to_the_launch_budget(tmp_path):
    """The GEMM kernels that hand registers between warpgroups with setmaxnreg
    are only safe when they launch with exactly the register count the split
    was computed for: weights-as-M<256> and the three tokens-as-M kernels, 384
    threads, 128*40 + 256*232 = 384*168.  Compile gemm.cu and read ptxas's
    register report (the library also re-checks at launch)."""
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = os.path.join(ROOT, "fp8_grouped_expert_x128_gb300", "csrc", "gemm.cu")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-Xptxas", "-v",
                        "-c", src, "-o", str(tmp_path / "g.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    report = {}
    current = None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            current = m.group(1)
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            report[current] = int(m.group(1))
        m = re.search(r"(\d+) bytes spill stores", line)
        if m and current and "gemm" in current:
            # a few bytes of spill are tolerated; the register split exists to
            # keep the 128 fp32 accumulators out of local memory
            assert int(m.group(1)) <= 64, f"{current} spills {m.group(1)} bytes"
    tok = [k for k in report if "tokens_m" in k]
    wm = [k for k in report if "weights_m_kernelILi256" in k]
    assert len(tok) == 3 and len(wm) == 1      # tokens-as-M plain, fused SwiGLU, CTA pair; weights-as-M<256>
    for k in tok + wm:
        assert report[k] == 168, (k, report[k])


def test_masked_gemm_dispatch_is_host_logic(so):
    # the masked GEMM's kernel choice is made on the host from (max_m, count
    # hint, flags) alone: weights-as-M for a few rows per expert, tile width by
    # the hint; tokens-as-M otherwise; the force flags override
    import fp8_grouped_expert_x128_gb300 as moe
    v = moe.moe_gemm_fp8_masked_variant
    assert v(128, 2) == 64 and v(128, 32) == 64           # all-experts decode
    assert v(1024, 134) == 0 and v(2048, 1024) == 0        # EP decode: tokens-as-M
    assert v(1024, 0) == 0                                 # no hint: max_m decides
    assert v(16, 0) == 64                                  # ... a tiny max_m is the hint
    assert v(128, 2, moe.MOE_GEMM_FORCE_TOKENS_M) == 0
    assert v(1024, 40, moe.MOE_GEMM_FORCE_WEIGHTS_M) == 64
    assert v(1024, 100, moe.MOE_GEMM_FORCE_WEIGHTS_M) == 128
    assert v(1024, 200, moe.MOE_GEMM_FORCE_WEIGHTS_M) == 256
    assert v(1000, 200, moe.MOE_GEMM_FORCE_WEIGHTS_M) == moe.MOE_ERR_UNSUPPORTED   # max_m % 16
    assert v(1000, 2) == 0                                 # weights-as-M needs max_m % 16 == 0


def test_ue8m0_scale_rule_matches_the_oracle(so):
    # the library's power-of-two block-scale rule (the code the UE8M0 quant
    # kernel runs, compiled for the host here) against the oracle's, bit for
    # bit: exact boundaries 448 * 2^j, their float32 neighbours, random maxima,
    # the floor and below it, the bf16 maximum
    import numpy as np
    import fp8_grouped_expert_x128_gb300 as moe
    from oracle.ffn import _block_scale_ue8m0
    rng = np.random.default_rng(7)
    edges = (448.0 * np.exp2(np.arange(-30, 120))).astype(np.float32)
    amax = np.concatenate([edges, np.nextafter(edges, np.float32(np.inf)), np.nextafter(edges, np.float32(0)),
                           np.exp2(rng.uniform(-40, 127, 2000)).astype(np.float32),
                           np.float32([0.0, 1e-30, 1e-4, 2e-4, 3.3895314e38])])
    amax = np.concatenate([amax[np.isfinite(amax)], np.float32([np.inf, np.nan])])
    ref_s, ref_b = _block_scale_ue8m0(amax)
    for a, rs, rb in zip(amax, ref_s, ref_b):
        s, b = moe.moe_ue8m0_scale(float(a))
        assert np.float32(s) == rs and b == int(rb), (a, s, b, rs, rb)
    assert moe.moe_ue8m0_scale(float("inf")) == (float("inf"), 0xFF)


def test_binding_constants_equal_the_header(so):
    """Every MOE_* value the Python binding names is the header's #define."""
    import fp8_grouped_expert_x128_gb300 as lib
    text = open(os.path.join(ROOT, "include", "moe_fp8.h")).read()
    defines = {m.group(1): int(m.group(2), 0)
               for m in re.finditer(r"^#define\s+(MOE_\w+)\s+\(?(-?(?:0x[0-9a-fA-F]+|\d+))\)?", text, flags=re.M)}
    named = [n for n in dir(lib) if n.startswith("MOE_") and isinstance(getattr(lib, n), int)]
    assert len(named) >= 10
    for n in named:
        assert n in defines, f"{n} is not in the header"
        assert getattr(lib, n) == defines[n], n
    for flag in ("MOE_GEMM_EARLY_WEIGHTS", "MOE_FFN_UE8M0", "MOE_QUANT_UE8M0", "MOE_COMBINE_ACCUMULATE"):
        assert flag in named


def test_empty_batch_launches_nothing(so):
    """T = 0 is a valid empty batch: host-only, the plan launches no kernel and
    the token I/O may be empty tensors (null pointers)."""
    import torch
    import fp8_grouped_expert_x128_gb300 as moe
    E, H, I, k = 4, 256, 128, 2
    x = torch.empty((0, H), dtype=torch.bfloat16)
    ids = torch.empty((0, k), dtype=torch.int32)
    w = torch.empty((0, k), dtype=torch.float32)
    w13 = torch.zeros((E, 2 * I, H), dtype=torch.uint8)
    w2 = torch.zeros((E, H, I), dtype=torch.uint8)
    s13 = torch.ones((E, 2 * I // 128, H // 128))
    s2 = torch.ones((E, H // 128, I // 128))
    out = torch.empty((0, H), dtype=torch.bfloat16)
    for layout in (moe.MOE_LAYOUT_MASKED, moe.MOE_LAYOUT_CONTIG):
        d = moe.make_ffn_desc(x, ids, w, w13, s13, w2, s2, out, 0, E, layout, max_m=128)
        assert moe.moe_ffn_kernel_count(d) == 0
        assert moe.moe_ffn_workspace_size(d) > 0
