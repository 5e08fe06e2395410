"""Writes tests/golden/c1_oracle.txt from the CPU oracle alone.

The tiny masked config (E=4, hidden 256, intermediate 128, T=64, top-2) is run
through ``oracle.ffn_chain`` on the seeded synthetic inputs, and the SHA-256 of
every stage's output plus a few sampled values are stored as text.  Nothing
here touches the CUDA library; rerun it only when a change to the oracle's
arithmetic has been justified by the definitions it follows.

    python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth   # noqa: E402


def _bits(t):
    """bf16 torch tensor -> uint16 bit patterns (the oracle's bf16 carrier)."""
    return t.contiguous().view(torch.int16).numpy().astype(np.uint16)


def c1_oracle_outputs():
    cfg = synth.get_config("c1")
    r = synth.make_routing(cfg)
    xb = _bits(synth.make_activations(cfg, r["T"]))
    w13q, w13s, w2q, w2s = [], [], [], []
    for e in range(cfg.E):
        w13 = oracle.bf16_decode(_bits(synth.make_expert_weights(cfg, "w13", e)))
        w2 = oracle.bf16_decode(_bits(synth.make_expert_weights(cfg, "w2", e)))
        q, s = oracle.quant_128x128(w13.astype(np.float32)); w13q.append(q); w13s.append(s)
        q, s = oracle.quant_128x128(w2.astype(np.float32)); w2q.append(q); w2s.append(s)
    res = oracle.ffn_chain(xb, r["topk_ids"], r["topk_w"], r["expert_begin"], cfg.E, cfg.layout,
                           cfg.max_m, np.stack(w13q), np.stack(w13s), np.stack(w2q), np.stack(w2s))
    return res


def digest_lines(res):
    lines = []
    for key in ("q", "s", "y1", "q2", "s2", "y2", "out"):
        a = np.ascontiguousarray(res[key])
        lines.append(f"sha256 {key} {a.dtype} {'x'.join(map(str, a.shape))} "
                     f"{hashlib.sha256(a.tobytes()).hexdigest()}")
    out = oracle.bf16_decode(res["out"])
    for t, h in [(0, 0), (5, 17), (31, 200), (63, 255)]:
        lines.append(f"out[{t},{h}] {out[t, h]!r}")
    lines.append(f"counts {' '.join(map(str, res['perm']['counts']))}")
    return lines


if __name__ == "__main__":
    lines = digest_lines(c1_oracle_outputs())
    with open(os.path.join(HERE, "c1_oracle.txt"), "w") as f:
        f.write("# CPU-oracle digest of the tiny masked config; written by make_golden.py\n")
        f.write("\n".join(lines) + "\n")
    print("\n".join(lines))
