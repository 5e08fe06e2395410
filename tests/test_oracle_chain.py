"""Pins of the oracle's whole chain on the tiny masked config and on a tiny
contiguous config with ragged segments: against an unquantised float64 FFN
(the quantisation error must stay small and a swapped gate/up or a dropped
combine weight must not), against a per-token restatement of the chain (rows
are independent, so routing each token alone through the block-scaled GEMMs
must give the chain's output bit for bit -- this pins the permutation, the
gathers and the scatter of both layouts), and against the stored digest
written by tests/golden/make_golden.py."""
import dataclasses
import os

import numpy as np

import oracle
import synth
from tests.golden.make_golden import _bits, c1_oracle_outputs, digest_lines

HERE = os.path.dirname(os.path.abspath(__file__))


def _ideal_ffn(cfg, r, swap=False, drop_weights=False):
    """The FFN in float64 on the unquantised bf16 weights and activations."""
    x = oracle.bf16_decode(_bits(synth.make_activations(cfg, r["T"])))
    out = np.zeros_like(x)
    I = cfg.I
    for t in range(r["T"]):
        for j in range(r["k"]):
            e = int(r["topk_ids"][t, j]) - r["expert_begin"]
            if not 0 <= e < cfg.E:
                continue
            w13 = oracle.bf16_decode(_bits(synth.make_expert_weights(cfg, "w13", e)))
            w2 = oracle.bf16_decode(_bits(synth.make_expert_weights(cfg, "w2", e)))
            y = w13 @ x[t]
            g, u = (y[I:], y[:I]) if swap else (y[:I], y[I:])
            h = g / (1 + np.exp(-g)) * u
            w = 1.0 if drop_weights else float(r["topk_w"][t, j])
            out[t] += w * (w2 @ h)
    return out


def test_chain_close_to_unquantised_ffn():
    cfg = synth.get_config("c1")
    r = synth.make_routing(cfg)
    res = c1_oracle_outputs()
    got = oracle.bf16_decode(res["out"])
    ref = _ideal_ffn(cfg, r)
    rel = np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))
    assert rel < 0.08, rel                                   # FP8 quantisation noise only
    for kw in (dict(swap=True), dict(drop_weights=True)):
        wrong = _ideal_ffn(cfg, r, **kw)
        assert np.sqrt(np.mean((got - wrong) ** 2) / np.mean(wrong ** 2)) > 4 * rel


def test_chain_routing_invariants():
    cfg = synth.get_config("c1")
    r = synth.make_routing(cfg)
    res = c1_oracle_outputs()
    assert res["perm"]["counts"].sum() == r["T"] * r["k"]
    assert np.allclose(r["topk_w"].sum(axis=1), 1.0, atol=1e-6)


def test_chain_matches_stored_digest():
    with open(os.path.join(HERE, "golden", "c1_oracle.txt")) as f:
        stored = [l.rstrip("\n") for l in f if not l.startswith("#")]
    assert digest_lines(c1_oracle_outputs()) == stored


def _contig_case():
    """E = 3 experts, hidden 256, intermediate 128, T = 150 tokens, top-2 over the
    three experts with a skewed draw, so the segments are ragged (one of them
    longer than 128 rows, none a multiple of 128)."""
    cfg = dataclasses.replace(synth.get_config("c1"), E=3, layout="contig", max_m=0)
    rng = np.random.default_rng(77)
    T, k = 150, 2
    ids = np.stack([rng.permutation(3)[:k] for _ in range(T)]).astype(np.int32)
    ids[:110, 0] = 1                                    # expert 1 gets most tokens
    ids[:110, 1] = np.where(ids[:110, 1] == 1, 2, ids[:110, 1])
    w = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    r = dict(topk_ids=ids, topk_w=w, T=T, k=k, expert_begin=0)
    return cfg, r


def _quantised_weights(cfg, ue8m0=False):
    quant = (lambda w: oracle.quant_128x128_ue8m0(w)[:2]) if ue8m0 else oracle.quant_128x128
    w13q, w13s, w2q, w2s = [], [], [], []
    for e in range(cfg.E):
        w13 = oracle.bf16_decode(_bits(synth.make_expert_weights(cfg, "w13", e)))
        w2 = oracle.bf16_decode(_bits(synth.make_expert_weights(cfg, "w2", e)))
        q, s = quant(w13.astype(np.float32)); w13q.append(q); w13s.append(s)
        q, s = quant(w2.astype(np.float32)); w2q.append(q); w2s.append(s)
    return np.stack(w13q), np.stack(w13s), np.stack(w2q), np.stack(w2s)


def _per_token(xb, r, E, W, ue8m0=False):
    """Each token alone: quantise its row, and for each of its local slots in
    order run GEMM1 -> SwiGLU+quant -> GEMM2 on that one row; combine."""
    w13q, w13s, w2q, w2s = W
    quant = (lambda v: oracle.quant_1x128_ue8m0(v)[:2]) if ue8m0 else oracle.quant_1x128
    out = []
    for t in range(r["T"]):
        q, s = quant(oracle.bf16_decode(xb[t:t + 1]).astype(np.float32))
        y2, w = [], []
        for j in range(r["k"]):
            e = int(r["topk_ids"][t, j]) - r["expert_begin"]
            if not 0 <= e < E:
                continue
            y1 = oracle.bf16_encode(oracle.gemm_block_scaled(q, s, w13q[e], w13s[e]))
            q2, s2 = oracle.swiglu_quant(y1, ue8m0)
            y2.append(oracle.bf16_encode(oracle.gemm_block_scaled(q2, s2, w2q[e], w2s[e]))[0])
            w.append(float(r["topk_w"][t, j]))
        out.append(oracle.combine(np.stack(y2), np.arange(len(w)), np.array([w], np.float32))[0]
                   if y2 else np.zeros(xb.shape[1], np.uint16))
    return np.stack(out)


def test_contig_chain_layout_and_close_to_unquantised_ffn():
    cfg, r = _contig_case()
    xb = _bits(synth.make_activations(cfg, r["T"]))
    W = _quantised_weights(cfg)
    res = oracle.ffn_chain(xb, r["topk_ids"], r["topk_w"], 0, cfg.E, "contig", 0, *W)
    p = res["perm"]
    counts = np.array([(r["topk_ids"] == e).sum() for e in range(cfg.E)])
    assert (counts % 128 != 0).all() and counts.max() > 128       # ragged segments
    assert np.array_equal(p["counts"], counts) and counts.sum() == r["T"] * r["k"]
    assert np.array_equal(np.diff(p["offsets"]), (counts + 127) // 128 * 128)
    assert (res["valid"] == (p["m_indices"] >= 0)).all() and res["valid"].sum() == counts.sum()
    got = oracle.bf16_decode(res["out"])
    ref = _ideal_ffn(cfg, r)
    rel = np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))
    assert rel < 0.08, rel
    for kw in (dict(swap=True), dict(drop_weights=True)):
        wrong = _ideal_ffn(cfg, r, **kw)
        assert np.sqrt(np.mean((got - wrong) ** 2) / np.mean(wrong ** 2)) > 4 * rel
    assert np.array_equal(res["out"], _per_token(xb, r, cfg.E, W))


def test_masked_chain_equals_the_per_token_restatement():
    cfg = synth.get_config("c1")
    r = synth.make_routing(cfg)
    xb = _bits(synth.make_activations(cfg, r["T"]))
    res = c1_oracle_outputs()
    assert np.array_equal(res["out"], _per_token(xb, r, cfg.E, _quantised_weights(cfg)))


def test_chunked_chain_equals_ffn_chain():
    # the row-chunked, threaded restatement the full-size GPU tests use for their
    # expected values gives ffn_chain's every stage bit for bit, in both layouts,
    # with chunks smaller than an expert's rows
    from tests.gpu_common import oracle_chain_chunked
    cfg, r = _contig_case()
    xb = _bits(synth.make_activations(cfg, r["T"]))
    W = _quantised_weights(cfg)
    c1 = synth.get_config("c1")
    r1 = synth.make_routing(c1)
    cases = [(xb, r, cfg.E, "contig", 0, W),
             (_bits(synth.make_activations(c1, r1["T"])), r1, c1.E, "masked", c1.max_m, _quantised_weights(c1))]
    for xbits, rr, E, layout, max_m, WW in cases:
        ref = oracle.ffn_chain(xbits, rr["topk_ids"], rr["topk_w"], rr["expert_begin"], E, layout, max_m, *WW)
        got = oracle_chain_chunked(xbits, rr["topk_ids"], rr["topk_w"], rr["expert_begin"], E, layout, max_m,
                                   *WW, chunk=24, workers=4)
        for key in ("q", "s", "y1", "valid", "q2", "s2", "y2", "out"):
            assert np.array_equal(got[key], ref[key]), (layout, key)


def test_ue8m0_chain_close_to_unquantised_ffn_and_per_token():
    # the chain with power-of-two scales everywhere (activations, requantised h
    # and weight tiles): as close to the unquantised FFN as the fp32-scale chain
    # (FP8 noise only), far from it with a gate/up swap or dropped weights, bit
    # for bit the per-token restatement, and the chunked harness's result
    from tests.gpu_common import oracle_chain_chunked
    cfg, r = _contig_case()
    xb = _bits(synth.make_activations(cfg, r["T"]))
    W = _quantised_weights(cfg, ue8m0=True)
    res = oracle.ffn_chain(xb, r["topk_ids"], r["topk_w"], 0, cfg.E, "contig", 0, *W, ue8m0=True)
    ref32 = oracle.ffn_chain(xb, r["topk_ids"], r["topk_w"], 0, cfg.E, "contig", 0, *_quantised_weights(cfg))
    got = oracle.bf16_decode(res["out"])
    ideal = _ideal_ffn(cfg, r)
    rel = np.sqrt(np.mean((got - ideal) ** 2) / np.mean(ideal ** 2))
    rel32 = np.sqrt(np.mean((oracle.bf16_decode(ref32["out"]) - ideal) ** 2) / np.mean(ideal ** 2))
    assert rel < 0.08 and rel < 1.5 * rel32, (rel, rel32)
    for kw in (dict(swap=True), dict(drop_weights=True)):
        wrong = _ideal_ffn(cfg, r, **kw)
        assert np.sqrt(np.mean((got - wrong) ** 2) / np.mean(wrong ** 2)) > 4 * rel
    assert (np.log2(res["s"]) == np.round(np.log2(res["s"]))).all()        # powers of two
    assert (np.log2(res["s2"][:, res["valid"]]) == np.round(np.log2(res["s2"][:, res["valid"]]))).all()
    assert np.array_equal(res["out"], _per_token(xb, r, cfg.E, W, ue8m0=True))
    ch = oracle_chain_chunked(xb, r["topk_ids"], r["topk_w"], 0, cfg.E, "contig", 0, *W, chunk=24, workers=4,
                              ue8m0=True)
    for key in ("q", "s", "y1", "q2", "s2", "y2", "out"):
        assert np.array_equal(ch[key], res[key]), key
