"""The FFN with the power-of-two (UE8M0) reading of the packed scales end to
end (moe_ffn with MOE_FFN_UE8M0): both activation quantisations take
power-of-two scales written in the packed layout, the weights carry
power-of-two tile scales, and both GEMMs are block-scaled on the tensor cores.

* against the oracle chain with the same reading (ffn_chain(..., ue8m0=True)):
  the tiny config at the strict bound, every token of the decode and prefill
  configs under the chain rule (one requantisation flip per routed row, up to
  2e-3 of the outputs past the strict bound: a power-of-two scale is up to
  twice the fp32 one), backed by strict stage-fed chains on c2 and c3;
* bit for bit against the public stage calls made one by one (quant with
  MOE_QUANT_UE8M0, permute, pack, block-scaled GEMM1, SwiGLU+quant with
  MOE_QUANT_UE8M0, pack, block-scaled GEMM2, combine)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from bench import build_workload, make_desc
from tests.gpu_common import (CHAIN_FRAC_UE8M0, SENTINEL_BF16, SENTINEL_F32, SENTINEL_U8, Guarded, bits,
                              check_swiglu, check_tol, check_tol_chain, f32_bits, flip_bound, from_bits,
                              oracle_chain_chunked, to_dev, u8)

pytestmark = pytest.mark.gpu


def _gpu_ffn(lib, wl):
    T, H = wl["T"], wl["cfg"].H
    out = torch.full((T, H), 0x7E57, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    err = lib.new_error_word()
    desc = make_desc(wl, out, err=err)
    lib.moe_ffn(desc, lib.alloc_workspace(desc))
    st, _ = lib.moe_read_device_status(err)
    return bits(out), st


_CACHE = {}


def _oracle(name, wl):
    """The UE8M0 oracle chain on every row, with UE8M0 oracle-quantised weights
    of the experts that own rows."""
    cfg = wl["cfg"]
    r = wl["routing"]
    ids = r["topk_ids"].reshape(-1) - r["expert_begin"]
    active = sorted({int(e) for e in ids if 0 <= e < cfg.E})
    W = [{}, {}, {}, {}]
    for e in active:
        for i, which in enumerate(("w13", "w2")):
            w = oracle.bf16_decode(bits(synth.make_expert_weights(cfg, which, e, device="cuda"))).astype(np.float32)
            q, s, _ = oracle.quant_128x128_ue8m0(w)
            W[2 * i][e], W[2 * i + 1][e] = q, s
    ref = oracle_chain_chunked(bits(wl["x"]), r["topk_ids"], r["topk_w"], r["expert_begin"], cfg.E, cfg.layout,
                               cfg.max_m, *W, ue8m0=True)
    return ref, W


def _oracle_cached(name, wl):
    if name not in _CACHE:
        _CACHE[name] = _oracle(name, wl)
    return _CACHE[name]


def test_ue8m0_ffn_tiny_config_strict(lib):
    wl = build_workload("c1", ue8m0=True)
    got, st = _gpu_ffn(lib, wl)
    assert st == 0
    ref, _ = _oracle("c1", wl)
    check_tol(got, ref["out"], "c1 ue8m0 ffn")


@pytest.mark.parametrize("name", ["c2", "c4", "c3", "c5t4"])
def test_ue8m0_ffn_every_token(lib, name):
    wl = build_workload(name, ue8m0=True)
    got, st = _gpu_ffn(lib, wl)
    ref, W = _oracle_cached(name, wl)
    assert st == (lib.MOE_ERR_OVERFLOW if ref["perm"]["overflow"] else lib.MOE_OK)
    check_tol_chain(got, ref["out"], flip_bound(ref, wl["routing"]["topk_w"], W[2], W[3]), f"{name} ue8m0 ffn",
                    max_frac=CHAIN_FRAC_UE8M0)


@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_ue8m0_ffn_equals_the_stage_entry_points(lib, name):
    wl = build_workload(name, ue8m0=True)
    got, st = _gpu_ffn(lib, wl)
    assert st == 0
    cfg = wl["cfg"]
    T, H, I, E, k = wl["T"], cfg.H, cfg.I, cfg.E, wl["k"]
    dev = "cuda"
    Tp = (T + 3) // 4 * 4
    q = torch.empty((T, H), dtype=torch.uint8, device=dev)
    s = torch.empty((H // 128, Tp), dtype=torch.float32, device=dev)
    lib.moe_quant_fp8(wl["x"], q, s, Tp, flags=lib.MOE_QUANT_UE8M0)
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
    groups, G = (E, cfg.max_m) if masked else (1, rows)

    def pack(sA, K):
        sf = torch.empty(lib.moe_ue8m0_act_words(groups, G, K), dtype=torch.int32, device=dev)
        lib.moe_pack_ue8m0_act(sA, groups, G, groups * G, K, sf)
        return sf

    Y1 = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device=dev)
    A2 = torch.empty((rows, I), dtype=torch.uint8, device=dev)
    sA2 = torch.empty((E, I // 128, cfg.max_m) if masked else (I // 128, rows), dtype=torch.float32, device=dev)
    Y2 = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
    if masked:
        M = cfg.max_m
        lib.moe_gemm_fp8_masked_ue8m0(A1.view(E, M, H), pack(sA1, H), wl["w13"], wl["w13_sf"], counts,
                                      Y1.view(E, M, 2 * I))
        lib.moe_swiglu_quant(Y1, A2, sA2, counts=counts, max_m=M, flags=lib.MOE_QUANT_UE8M0)
        lib.moe_gemm_fp8_masked_ue8m0(A2.view(E, M, I), pack(sA2, I), wl["w2"], wl["w2_sf"], counts, Y2.view(E, M, H))
    else:
        lib.moe_gemm_fp8_contig_ue8m0(A1, pack(sA1, H), rows, wl["w13"], wl["w13_sf"], offsets, mi, Y1)
        lib.moe_swiglu_quant(Y1, A2, sA2, m_indices=mi, s_ld=rows, flags=lib.MOE_QUANT_UE8M0)
        lib.moe_gemm_fp8_contig_ue8m0(A2, pack(sA2, I), rows, wl["w2"], wl["w2_sf"], offsets, mi, Y2)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    lib.moe_combine(Y2, dst, wl["topk_w"], out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), got)


def test_ue8m0_swiglu_quant_matches_the_oracle(lib):
    # the power-of-two SwiGLU requantisation alone: scales exact powers of two,
    # codes under the relaxed SwiGLU rule (GPU expf) against the oracle
    from tests.gpu_common import check_swiglu, from_bits, u8
    rows, I = 300, 2048
    y1 = bits((synth.counter_normal(rows * 2 * I, 5, 77, device="cuda") * 2.0).to(torch.bfloat16).reshape(rows, 2 * I))
    q = torch.empty((rows, I), dtype=torch.uint8, device="cuda")
    s = torch.empty((I // 128, rows), dtype=torch.float32, device="cuda")
    lib.moe_swiglu_quant(from_bits(y1), q, s, s_ld=rows, flags=lib.MOE_QUANT_UE8M0)
    torch.cuda.synchronize()
    ref_q, ref_s = oracle.swiglu_quant(y1, ue8m0=True)
    sh = s.cpu().numpy()
    assert (np.log2(sh) == np.round(np.log2(sh))).all()
    check_swiglu(u8(q), sh, y1, np.ones(rows, bool), ref_q=ref_q, ref_s=ref_s)


def _dev_w(Wq, Ws, E, K):
    """Device weights [E, N, K] and their packed records (oracle-packed) from the
    oracle's per-expert dicts; experts without rows are zero (never read)."""
    e0 = next(iter(Wq))
    q = torch.zeros((E,) + Wq[e0].shape, dtype=torch.uint8, device="cuda")
    s = np.ones((E,) + Ws[e0].shape, np.float32)
    for e in Wq:
        q[e].copy_(torch.from_numpy(Wq[e]))
        s[e] = Ws[e]
    return q, to_dev(oracle.pack_ue8m0_weight(s).view(np.int32))


@pytest.mark.parametrize("name", ["c2", "c3"])
def test_ue8m0_ffn_stage_fed(lib, name):
    """Each block-scaled stage fed the oracle's previous stage (scales packed by
    the oracle's packers) on every routed row: GEMMs and combine at the strict
    bound, SwiGLU+quant at its rule."""
    wl = build_workload(name, ue8m0=True)
    cfg = wl["cfg"]
    ref, W = _oracle_cached(name, wl)
    E, M, I, H = cfg.E, cfg.max_m, cfg.I, cfg.H
    p, v = ref["perm"], ref["valid"]
    rows = p["rows"]
    masked = cfg.layout == "masked"
    groups, G = (E, M) if masked else (1, rows)
    w13, w13_sf = _dev_w(W[0], W[1], E, H)
    w2, w2_sf = _dev_w(W[2], W[3], E, I)

    def sfa(s):
        return to_dev(oracle.pack_ue8m0_act(s, G, groups * G).view(np.int32))

    def gemm(A, s, B, sf, N, K):
        if masked:
            g = Guarded((E, M, N), torch.bfloat16, SENTINEL_BF16)
            lib.moe_gemm_fp8_masked_ue8m0(to_dev(A.reshape(E, M, K)), sfa(s), B, sf,
                                          to_dev(p["counts"].astype(np.int32)), g.t, expected_m=wl["expected_m"])
        else:
            g = Guarded((rows, N), torch.bfloat16, SENTINEL_BF16)
            lib.moe_gemm_fp8_contig_ue8m0(to_dev(A), sfa(s), rows, B, sf, to_dev(p["offsets"].astype(np.int32)),
                                          to_dev(p["m_indices"].astype(np.int32)), g.t)
        torch.cuda.synchronize()
        assert g.intact()
        return bits(g.t).reshape(rows, N)

    y1 = gemm(p["q"], p["s"], w13, w13_sf, 2 * I, H)
    check_tol(y1[v], ref["y1"][v], f"{name} ue8m0 stage GEMM1")
    assert (y1[~v] == SENTINEL_BF16).all()
    del y1
    gq = Guarded((rows, I), torch.uint8, SENTINEL_U8)
    gs = Guarded((E, I // 128, M) if masked else (I // 128, rows), torch.float32, f32_bits(SENTINEL_F32))
    if masked:
        lib.moe_swiglu_quant(from_bits(ref["y1"]), gq.t, gs.t, counts=to_dev(p["counts"].astype(np.int32)), max_m=M,
                             flags=lib.MOE_QUANT_UE8M0)
    else:
        lib.moe_swiglu_quant(from_bits(ref["y1"]), gq.t, gs.t, m_indices=to_dev(p["m_indices"].astype(np.int32)),
                             s_ld=rows, flags=lib.MOE_QUANT_UE8M0)
    torch.cuda.synchronize()
    assert gq.intact() and gs.intact()
    s2 = gs.t.cpu().numpy()
    s2f = s2.transpose(1, 0, 2).reshape(I // 128, -1) if masked else s2
    r2f = ref["s2"].transpose(1, 0, 2).reshape(I // 128, -1) if masked else ref["s2"]
    check_swiglu(u8(gq.t), s2f[:, v], ref["y1"], v, ref_q=ref["q2"][v], ref_s=r2f[:, v])
    y2 = gemm(ref["q2"], ref["s2"], w2, w2_sf, H, I)
    check_tol(y2[v], ref["y2"][v], f"{name} ue8m0 stage GEMM2")
    assert (y2[~v] == SENTINEL_BF16).all()
    del y2
    go = Guarded((wl["T"], H), torch.bfloat16, SENTINEL_BF16)
    lib.moe_combine(from_bits(ref["y2"]), to_dev(p["dst_row"].astype(np.int32)), wl["topk_w"], go.t)
    torch.cuda.synchronize()
    assert go.intact()
    check_tol(bits(go.t), ref["out"], f"{name} ue8m0 stage combine")
