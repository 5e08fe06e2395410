"""Pins of the oracle's whole chain on the tiny masked config: against an
unquantised float64 FFN (the quantisation error must stay small and a swapped
gate/up or a dropped combine weight must not), and against the stored digest
written by tests/golden/make_golden.py."""
import os

import numpy as np

import oracle
import synth
from tests.golden.make_golden import _bits, c1_oracle_outputs, digest_lines

HERE = os.path.dirname(os.path.abspath(__file__))


def _ideal_ffn(cfg, r, swap=False, drop_weights=False):
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
