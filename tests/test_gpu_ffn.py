"""End-to-end parity of moe_ffn with the oracle chain on every config, plus the
stage-fed check: each GPU stage fed the oracle's previous-stage output and
compared with the oracle's own next stage.

Every routed row and every token of every config is compared (the tiny masked
config, the EP72-like and 48-GPU-domain decode configs, the all-experts layer
at T = 64 and at T = 1, 4, 16, and the prefill contiguous config).  The oracle
chain is computed on row chunks in threads (bit for bit ffn_chain, see
tests/gpu_common.py); output buffers carry guard bands."""
import dataclasses

import numpy as np
import pytest
import torch

from bench import build_workload, make_desc
from tests.gpu_common import (SENTINEL_BF16, SENTINEL_F32, SENTINEL_U8, Guarded, bits, check_swiglu,
                              check_tol, check_tol_chain, f32_bits, flip_bound, from_bits,
                              oracle_chain_chunked, oracle_weights, to_dev, u8)

pytestmark = pytest.mark.gpu


def _gpu_ffn(lib, wl):
    T, H = wl["T"], wl["cfg"].H
    out = torch.full((T, H), 0x7E57, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    err = lib.new_error_word()
    desc = make_desc(wl, out, err=err)
    ws = lib.alloc_workspace(desc)
    lib.moe_ffn(desc, ws)
    st, _ = lib.moe_read_device_status(err)
    return bits(out), st


_ORACLE_CACHE = {}


def _oracle_full(name, wl):
    """The oracle chain on every row of a config (row-chunked and threaded, bit
    for bit ffn_chain) and the oracle-quantised weights of the experts that own
    rows (dicts keyed by local expert); cached per config for this module."""
    if name not in _ORACLE_CACHE:
        cfg = wl["cfg"]
        r = wl["routing"]
        ids = r["topk_ids"].reshape(-1) - r["expert_begin"]
        active = tuple(sorted({int(e) for e in ids if 0 <= e < cfg.E}))
        W = []
        for which in ("w13", "w2"):
            q, s = oracle_weights(name, which, active)
            W += [dict(zip(active, q)), dict(zip(active, s))]
        ref = oracle_chain_chunked(bits(wl["x"]), r["topk_ids"], r["topk_w"], r["expert_begin"], cfg.E,
                                   cfg.layout, cfg.max_m, *W)
        _ORACLE_CACHE[name] = (ref, tuple(W))
    return _ORACLE_CACHE[name]


def _dev_weights(Wq: dict, Ws: dict, E: int):
    """Device copies [E, N, K] / [E, N/128, K/128] of the oracle-quantised weights;
    experts without rows hold zeros (no kernel reads them)."""
    e0 = next(iter(Wq))
    q = torch.zeros((E,) + Wq[e0].shape, dtype=torch.uint8, device="cuda")
    s = torch.zeros((E,) + Ws[e0].shape, dtype=torch.float32, device="cuda")
    for e in Wq:
        q[e].copy_(torch.from_numpy(Wq[e]))
        s[e].copy_(torch.from_numpy(Ws[e]))
    return q, s


def test_ffn_tiny_config_end_to_end(lib):
    wl = build_workload("c1")
    got, st = _gpu_ffn(lib, wl)
    assert st == 0
    ref, _ = _oracle_full("c1", wl)
    check_tol(got, ref["out"], "c1 ffn")


def _stage_fed(lib, name):
    """Each GPU stage fed the oracle's previous-stage output, compared with the
    oracle's own next stage at the stage's acceptance rule, on every routed row
    (GEMMs at the strict bound, SwiGLU+quant at its relaxed rule, combine strict)."""
    wl = build_workload(name)
    cfg = wl["cfg"]
    ref, (w13q, w13s, w2q, w2s) = _oracle_full(name, wl)
    E, M, I, H = cfg.E, cfg.max_m, cfg.I, cfg.H
    p = ref["perm"]
    v = ref["valid"]
    rows = p["rows"]
    masked = cfg.layout == "masked"
    hint = wl["expected_m"]
    if masked:
        counts = to_dev(p["counts"].astype(np.int32))

        def gemm(A, sA, Bq, Bs, N, K):
            g = Guarded((E, M, N), torch.bfloat16, SENTINEL_BF16)
            lib.moe_gemm_fp8_masked(to_dev(A.reshape(E, M, K)), to_dev(sA), *_dev_weights(Bq, Bs, E), counts, g.t,
                                    expected_m=hint)
            torch.cuda.synchronize()
            assert g.intact(), f"{name}: GEMM wrote past D"
            return bits(g.t).reshape(rows, N)
    else:
        offsets = to_dev(p["offsets"].astype(np.int32))
        mi = to_dev(p["m_indices"].astype(np.int32))

        def gemm(A, sA, Bq, Bs, N, K):
            g = Guarded((rows, N), torch.bfloat16, SENTINEL_BF16)
            lib.moe_gemm_fp8_contig(to_dev(A), to_dev(sA), *_dev_weights(Bq, Bs, E), offsets, mi, g.t)
            torch.cuda.synchronize()
            assert g.intact(), f"{name}: GEMM wrote past D"
            return bits(g.t)
    # GEMM1 on the oracle's permuted activations
    y1 = gemm(p["q"], p["s"], w13q, w13s, 2 * I, H)
    check_tol(y1[v], ref["y1"][v], f"{name} stage GEMM1")
    assert (y1[~v] == SENTINEL_BF16).all(), f"{name}: GEMM1 wrote rows past a count / padding"
    del y1
    # SwiGLU+quant on the oracle's GEMM1 output (the relaxed SwiGLU rule)
    gq = Guarded((rows, I), torch.uint8, SENTINEL_U8)
    gs = Guarded((E, I // 128, M) if masked else (I // 128, rows), torch.float32, f32_bits(SENTINEL_F32))
    if masked:
        lib.moe_swiglu_quant(from_bits(ref["y1"]), gq.t, gs.t, counts=counts, max_m=M)
    else:
        lib.moe_swiglu_quant(from_bits(ref["y1"]), gq.t, gs.t, m_indices=mi, s_ld=rows)
    torch.cuda.synchronize()
    assert gq.intact() and gs.intact(), f"{name}: SwiGLU wrote past its outputs"
    s2 = gs.t.cpu().numpy()
    s2f = s2.transpose(1, 0, 2).reshape(I // 128, -1) if masked else s2
    r2f = ref["s2"].transpose(1, 0, 2).reshape(I // 128, -1) if masked else ref["s2"]
    q2 = u8(gq.t)
    check_swiglu(q2, s2f[:, v], ref["y1"], v, ref_q=ref["q2"][v], ref_s=r2f[:, v])
    assert (q2[~v] == SENTINEL_U8).all() and (s2f[:, ~v] == SENTINEL_F32).all()
    # GEMM2 on the oracle's requantised activations
    y2 = gemm(ref["q2"], ref["s2"], w2q, w2s, H, I)
    check_tol(y2[v], ref["y2"][v], f"{name} stage GEMM2")
    assert (y2[~v] == SENTINEL_BF16).all(), f"{name}: GEMM2 wrote rows past a count / padding"
    del y2
    # combine on the oracle's GEMM2 output
    go = Guarded((wl["T"], H), torch.bfloat16, SENTINEL_BF16)
    lib.moe_combine(from_bits(ref["y2"]), to_dev(p["dst_row"].astype(np.int32)), wl["topk_w"], go.t)
    torch.cuda.synchronize()
    assert go.intact(), f"{name}: combine wrote past out"
    check_tol(bits(go.t), ref["out"], f"{name} stage combine")


@pytest.mark.parametrize("name", ["c1", "c2", "c4", "c5", "c3"])
def test_ffn_stage_fed(lib, name):
    _stage_fed(lib, name)


@pytest.mark.parametrize("name", ["c2", "c4", "c5", "c5t1", "c5t4", "c5t16", "c3"])
def test_ffn_end_to_end_every_token(lib, name):
    # every token of every config against the oracle chain under the chain rule:
    # the decode configs (the status must report an overflow exactly when the
    # oracle's permutation drops rows), the all-experts layer (T = 64, and the
    # latency regime T = 1, 4, 16: ~9-110 active experts with 1-2 rows each,
    # weights-as-M) and the prefill layout (32768 tokens, contiguous, one slot
    # per token: GEMM2 writes the output rows itself)
    wl = build_workload(name)
    got, st = _gpu_ffn(lib, wl)
    ref, (_, _, w2q, w2s) = _oracle_full(name, wl)
    assert st == (lib.MOE_ERR_OVERFLOW if ref["perm"]["overflow"] else lib.MOE_OK)
    check_tol_chain(got, ref["out"], flip_bound(ref, wl["routing"]["topk_w"], w2q, w2s), f"{name} ffn")


@pytest.mark.parametrize("name,fuse", [("c1", False), ("c2", False), ("c3", False), ("c2", True), ("c3", True),
                                       ("c5t1", False), ("c1_overflow", False), ("c4_overflow", False),
                                       ("c3_ragged", False)])
def test_ffn_equals_the_stage_entry_points(lib, name, fuse):
    """moe_ffn fuses quantisation into the permute (and, with MOE_FFN_FUSE_SWIGLU,
    SwiGLU + requantisation into the tokens-as-M GEMM1 epilogue); its output must
    be bit-identical to the public stage calls made one by one (quant, permute,
    GEMM1, SwiGLU+quant, GEMM2, combine).  The index pass differs by batch size
    inside moe_ffn (inside the quant-scatter kernel for c1 / c5t1, one CTA for c2,
    many CTAs for c3 / c4) and is the one-CTA kernel in moe_permute.
    c1_overflow / c4_overflow: max_m cut to 16 / 1024, so experts overflow and
    the ranks past max_m are dropped the same way on both paths.  c3_ragged: the
    first 30000 prefill tokens, so the last 4096-assignment chunk of the
    many-CTA index pass is partly empty."""
    overflow = name.endswith("_overflow")
    wl = build_workload(name.split("_")[0] if overflow or name.endswith("_ragged") else name)
    if overflow:
        wl["cfg"] = dataclasses.replace(wl["cfg"], max_m=16 if name.startswith("c1") else 1024)
    if name.endswith("_ragged"):
        T = 30000
        wl.update(x=wl["x"][:T], topk_ids=wl["topk_ids"][:T], topk_w=wl["topk_w"][:T], T=T)
    cfg = wl["cfg"]
    if fuse:
        wl["gemm_flags"] = lib.MOE_FFN_FUSE_SWIGLU
    got, st = _gpu_ffn(lib, wl)
    assert st == (lib.MOE_ERR_OVERFLOW if overflow else lib.MOE_OK)
    T, H, I, E, k = wl["T"], cfg.H, cfg.I, cfg.E, wl["k"]
    dev = "cuda"
    q = torch.empty((T, H), dtype=torch.uint8, device=dev)
    Tp = (T + 3) // 4 * 4
    s = torch.empty((H // 128, Tp), dtype=torch.float32, device=dev)
    lib.moe_quant_fp8(wl["x"], q, s, Tp)
    masked = wl["layout"] == lib.MOE_LAYOUT_MASKED
    rows = E * cfg.max_m if masked else lib.moe_contig_rows_bound(T * k, E)
    A1 = torch.empty((rows, H), dtype=torch.uint8, device=dev)
    sA1 = torch.empty((E, H // 128, cfg.max_m) if masked else (H // 128, rows), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    mi = torch.empty(rows, dtype=torch.int32, device=dev)
    row_src = torch.empty(rows, dtype=torch.int32, device=dev)
    dst = torch.empty(T * k, dtype=torch.int32, device=dev)
    lib.moe_permute(q, s, wl["topk_ids"], wl["routing"]["expert_begin"], E, wl["layout"], cfg.max_m,
                    A1, sA1, counts, offsets, mi, row_src, dst, rows_capacity=0 if masked else rows, s_ld=Tp)
    Y1 = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device=dev)
    A2 = torch.empty((rows, I), dtype=torch.uint8, device=dev)
    sA2 = torch.empty((E, I // 128, cfg.max_m) if masked else (I // 128, rows), dtype=torch.float32, device=dev)
    Y2 = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
    if masked:
        M = cfg.max_m
        lib.moe_gemm_fp8_masked(A1.view(E, M, H), sA1, wl["w13"], wl["w13_s"], counts, Y1.view(E, M, 2 * I),
                                expected_m=wl["expected_m"])
        lib.moe_swiglu_quant(Y1, A2, sA2, counts=counts, max_m=M)
        lib.moe_gemm_fp8_masked(A2.view(E, M, I), sA2, wl["w2"], wl["w2_s"], counts, Y2.view(E, M, H),
                                expected_m=wl["expected_m"])
    else:
        lib.moe_gemm_fp8_contig(A1, sA1, wl["w13"], wl["w13_s"], offsets, mi, Y1)
        lib.moe_swiglu_quant(Y1, A2, sA2, m_indices=mi, s_ld=rows)
        lib.moe_gemm_fp8_contig(A2, sA2, wl["w2"], wl["w2_s"], offsets, mi, Y2)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    lib.moe_combine(Y2, dst, wl["topk_w"], out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), got)


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c5t4"])
def test_ffn_host_buffers_equal_device_buffers(lib, name):
    # x, the routing and out in mapped page-locked host memory: the kernels read
    # and write them in place across the host link; the bytes of out equal the
    # device-buffer call's (c3 covers the single-slot path: out rows written by
    # GEMM2's epilogue, zero rows by the quant-scatter pass)
    wl = build_workload(name)
    ref, st = _gpu_ffn(lib, wl)
    T, H = wl["T"], wl["cfg"].H
    x_h = wl["x"].cpu().pin_memory()
    ids_h = wl["topk_ids"].cpu().pin_memory()
    w_h = wl["topk_w"].cpu().pin_memory()
    out_h = torch.full((T, H), 0x7E57, dtype=torch.int16).pin_memory().view(torch.bfloat16)
    err = lib.new_error_word()
    desc = make_desc(wl, out_h, err=err, x=x_h, ids=ids_h, w=w_h)
    ws = lib.alloc_workspace(desc)
    lib.moe_ffn(desc, ws)
    torch.cuda.synchronize()
    st_h, _ = lib.moe_read_device_status(err)
    assert st_h == st
    assert np.array_equal(bits(out_h), ref)


def test_ffn_refuses_pageable_host_buffers(lib):
    # pageable host memory is not mapped for the GPU: refused before any launch
    wl = build_workload("c1")
    T, H = wl["T"], wl["cfg"].H
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    for which in ("x", "out"):
        x = wl["x"].cpu() if which == "x" else wl["x"]
        o = torch.empty((T, H), dtype=torch.bfloat16) if which == "out" else out
        desc = make_desc(wl, o, x=x)
        ws = lib.alloc_workspace(desc)
        with pytest.raises(lib.MoeError) as ei:
            lib.moe_ffn(desc, ws)
        assert ei.value.status == lib.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("reading", ["fp32", "ue8m0"])
@pytest.mark.parametrize("layout", ["masked", "contig"])
@pytest.mark.parametrize("case", ["no_tokens", "no_local_slot"])
def test_ffn_degenerate_batches(lib, case, layout, reading):
    """The degenerate batches of the method, through moe_ffn on the tiny config
    in both layouts and both scale readings: no tokens at all (T = 0, empty
    token tensors whose pointers are null: the call succeeds, launches nothing
    and writes nothing), and tokens none of whose slots is local (every output
    row is the empty combine, +0.0, and no expert runs)."""
    wl = build_workload("c1", ue8m0=reading == "ue8m0")
    if layout == "contig":
        wl["cfg"] = dataclasses.replace(wl["cfg"], layout="contig")
        wl["layout"] = lib.MOE_LAYOUT_CONTIG
    H, E = wl["cfg"].H, wl["cfg"].E
    ids = wl["topk_ids"]
    if case == "no_local_slot":
        ids = (ids - wl["routing"]["expert_begin"]) % E + wl["routing"]["expert_begin"] + E   # all remote
    T = 0 if case == "no_tokens" else wl["T"]
    g = Guarded((T, H), torch.bfloat16, SENTINEL_BF16)
    err = lib.new_error_word()
    desc = make_desc(wl, g.t, err=err, x=wl["x"][:T], ids=ids[:T], w=wl["topk_w"][:T])
    ws = lib.alloc_workspace(desc)
    if T == 0:
        assert lib.moe_ffn_kernel_count(desc) == 0
    lib.moe_ffn(desc, ws)
    st, _ = lib.moe_read_device_status(err)
    assert st == lib.MOE_OK
    assert g.intact(), "moe_ffn wrote past out"
    if T:
        assert (bits(g.t) == 0).all(), "a token with no local slot must come out +0.0"


@pytest.mark.parametrize("name,expected", [("c1", 5), ("c5t1", 5), ("c5", 5), ("c2", 6), ("c4", 7), ("c3", 6)])
def test_ffn_kernel_count(lib, name, expected):
    """The kernels one moe_ffn call launches (what bench.py reports per step):
    small masked batches run the index pass inside the quant-scatter kernel,
    mid-sized ones as one kernel, large ones (c3, c4) as two; one slot per
    token (c3) folds the combine into GEMM2's epilogue."""
    wl = build_workload(name)
    T, H = wl["T"], wl["cfg"].H
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    assert lib.moe_ffn_kernel_count(make_desc(wl, out)) == expected
