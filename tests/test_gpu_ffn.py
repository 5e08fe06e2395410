"""End-to-end parity of moe_ffn with the oracle chain on the configs, plus the
stage-fed check: each GPU stage fed the oracle's previous-stage output and
compared with the oracle's own next stage.

Configs: the tiny masked config in full; the EP72-like and 48-GPU-domain
decode configs in full (every routed row); the all-experts decode layer and the
prefill (contiguous) config on sampled tokens, each sampled token's output
computed by the oracle alone from x, its routing and its experts' weights."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from bench import build_workload, make_desc
from tests.gpu_common import (bits, check_swiglu, check_tol, check_tol_chain, e4m3_flip_step,
                              flip_bound, from_bits, oracle_weights, to_dev, u8, w2_colmax)

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


def _oracle_full(name, wl):
    cfg = wl["cfg"]
    r = wl["routing"]
    e_all = tuple(range(cfg.E))
    w13q, w13s = oracle_weights(name, "w13", e_all)
    w2q, w2s = oracle_weights(name, "w2", e_all)
    return oracle.ffn_chain(bits(wl["x"]), r["topk_ids"], r["topk_w"], r["expert_begin"], cfg.E,
                            cfg.layout, cfg.max_m, w13q, w13s, w2q, w2s), (w13q, w13s, w2q, w2s)


def _oracle_tokens(name, wl, tokens):
    """The oracle chain restricted to `tokens` (rows are independent), and the
    end-to-end allowance of one E4M3 flip of h per routed row (as flip_bound)."""
    cfg = wl["cfg"]
    r = wl["routing"]
    xb = bits(wl["x"])[tokens]
    q, s = oracle.quant_1x128(oracle.bf16_decode(xb).astype(np.float32))
    ids = r["topk_ids"][tokens] - r["expert_begin"]
    need = tuple(sorted({int(e) for e in ids.reshape(-1) if 0 <= e < cfg.E}))
    w13q, w13s = oracle_weights(name, "w13", need)
    w2q, w2s = oracle_weights(name, "w2", need)
    slot = {e: i for i, e in enumerate(need)}
    colmax = {}
    out, extra = [], []
    for i, t in enumerate(tokens):
        y2, w = [], []
        flip = np.zeros(cfg.H)
        for j in range(r["k"]):
            e = int(r["topk_ids"][t, j]) - r["expert_begin"]
            if not 0 <= e < cfg.E:
                continue
            n = slot[e]
            y1 = oracle.bf16_encode(oracle.gemm_block_scaled(q[i:i + 1], s[:, i:i + 1], w13q[n], w13s[n]))
            q2, s2 = oracle.swiglu_quant(y1)
            y2.append(oracle.bf16_encode(oracle.gemm_block_scaled(q2, s2, w2q[n], w2s[n]))[0])
            w.append(float(r["topk_w"][t, j]))
            if n not in colmax:
                colmax[n] = w2_colmax(w2q[n], w2s[n])
            rowflip = e4m3_flip_step(q2[0], np.repeat(s2[:, 0], 128)).max()
            flip += w[-1] * rowflip * colmax[n]
        out.append(oracle.combine(np.stack(y2), np.arange(len(w)), np.array([w], np.float32))[0])
        extra.append(flip)
    return np.stack(out), np.stack(extra)


def test_ffn_tiny_config_end_to_end(lib):
    wl = build_workload("c1")
    got, st = _gpu_ffn(lib, wl)
    assert st == 0
    ref, _ = _oracle_full("c1", wl)
    check_tol(got, ref["out"], "c1 ffn")


def _stage_fed(lib, name):
    """Each GPU stage fed the oracle's previous-stage output, compared with the
    oracle's own next stage at the stage's acceptance rule."""
    wl = build_workload(name)
    cfg = wl["cfg"]
    ref, (w13q, w13s, w2q, w2s) = _oracle_full(name, wl)
    E, M, I, H = cfg.E, cfg.max_m, cfg.I, cfg.H
    counts = to_dev(ref["perm"]["counts"].astype(np.int32))
    hint = wl["expected_m"]
    v = ref["valid"]
    # GEMM1 on the oracle's permuted activations
    y1 = torch.empty((E, M, 2 * I), dtype=torch.bfloat16, device="cuda")
    lib.moe_gemm_fp8_masked(to_dev(ref["perm"]["q"].reshape(E, M, H)), to_dev(ref["perm"]["s"]),
                            to_dev(w13q), to_dev(w13s), counts, y1, expected_m=hint)
    check_tol(bits(y1).reshape(E * M, -1)[v], ref["y1"][v], f"{name} stage GEMM1")
    # SwiGLU+quant on the oracle's GEMM1 output (the relaxed SwiGLU rule)
    q2 = torch.empty((E * M, I), dtype=torch.uint8, device="cuda")
    s2 = torch.empty((E, I // 128, M), dtype=torch.float32, device="cuda")
    lib.moe_swiglu_quant(from_bits(ref["y1"]), q2, s2, counts=counts, max_m=M)
    torch.cuda.synchronize()
    s2f = s2.cpu().numpy().transpose(1, 0, 2).reshape(I // 128, -1)
    r2f = ref["s2"].transpose(1, 0, 2).reshape(I // 128, -1)
    check_swiglu(u8(q2), s2f[:, v], ref["y1"], v, ref_q=ref["q2"][v], ref_s=r2f[:, v])
    # GEMM2 on the oracle's requantised activations
    y2 = torch.empty((E, M, H), dtype=torch.bfloat16, device="cuda")
    lib.moe_gemm_fp8_masked(to_dev(ref["q2"].reshape(E, M, I)), to_dev(ref["s2"]), to_dev(w2q),
                            to_dev(w2s), counts, y2, expected_m=hint)
    check_tol(bits(y2).reshape(E * M, -1)[v], ref["y2"][v], f"{name} stage GEMM2")
    # combine on the oracle's GEMM2 output
    out = torch.empty((wl["T"], H), dtype=torch.bfloat16, device="cuda")
    lib.moe_combine(from_bits(ref["y2"]), to_dev(ref["perm"]["dst_row"].astype(np.int32)),
                    wl["topk_w"], out)
    check_tol(bits(out), ref["out"], f"{name} stage combine")


@pytest.mark.parametrize("name", ["c1", "c2", "c4"])
def test_ffn_stage_fed(lib, name):
    _stage_fed(lib, name)


@pytest.mark.parametrize("name", ["c2", "c4"])
def test_ffn_decode_configs_end_to_end(lib, name):
    wl = build_workload(name)
    got, st = _gpu_ffn(lib, wl)
    assert st in (0, lib.MOE_ERR_OVERFLOW)
    ref, (_, _, w2q, w2s) = _oracle_full(name, wl)
    assert (st == lib.MOE_ERR_OVERFLOW) == bool(ref["perm"]["overflow"])
    check_tol_chain(got, ref["out"], flip_bound(ref, wl["routing"]["topk_w"], w2q, w2s), f"{name} ffn")


def test_ffn_all_experts_layer_sampled_tokens(lib):
    wl = build_workload("c5")
    got, st = _gpu_ffn(lib, wl)
    assert st == 0
    tokens = [0, 63]
    ref, extra = _oracle_tokens("c5", wl, tokens)
    check_tol_chain(got[tokens], ref, extra, "c5 ffn tokens")
    assert np.isfinite(oracle.bf16_decode(got)).all()


@pytest.mark.parametrize("name", ["c5t1", "c5t4", "c5t16"])
def test_ffn_all_experts_small_batch(lib, name):
    # the latency regime of the all-experts layer: 1-16 tokens, ~9-100 active
    # experts, 1-2 rows each (weights-as-M with 16-wide token tiles)
    wl = build_workload(name)
    got, st = _gpu_ffn(lib, wl)
    assert st == 0
    T = wl["T"]
    tokens = sorted({0, T - 1})
    ref, extra = _oracle_tokens(name, wl, tokens)
    check_tol_chain(got[tokens], ref, extra, f"{name} ffn tokens")
    assert np.isfinite(oracle.bf16_decode(got)).all()


def test_ffn_prefill_contiguous_sampled_tokens(lib):
    wl = build_workload("c3")
    got, st = _gpu_ffn(lib, wl)
    assert st == 0
    r = wl["routing"]
    rng = np.random.default_rng(21)
    tokens = []
    for e in range(wl["cfg"].E):                 # a few tokens of every expert
        tokens += list(rng.choice(np.nonzero(r["topk_ids"][:, 0] == e)[0], 3, replace=False))
    tokens = sorted(tokens)
    ref, extra = _oracle_tokens("c3", wl, tokens)
    check_tol_chain(got[tokens], ref, extra, "c3 ffn tokens")


@pytest.mark.parametrize("name,fuse", [("c1", False), ("c2", False), ("c3", False), ("c2", True), ("c3", True),
                                       ("c5t1", False), ("c1_overflow", False)])
def test_ffn_equals_the_stage_entry_points(lib, name, fuse):
    """moe_ffn fuses quantisation into the permute (and, with MOE_FFN_FUSE_SWIGLU,
    SwiGLU + requantisation into the tokens-as-M GEMM1 epilogue); its output must
    be bit-identical to the public stage calls made one by one (quant, permute,
    GEMM1, SwiGLU+quant, GEMM2, combine).
    c1_overflow: the tiny config with 16 slots per expert, so every expert
    overflows and the ranks past max_m are dropped the same way on both paths."""
    overflow = name == "c1_overflow"
    wl = build_workload("c1" if overflow else name)
    if overflow:
        wl["cfg"] = dataclasses.replace(wl["cfg"], max_m=16)
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
