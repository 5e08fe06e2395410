"""The seeded input generator: slices regenerate alone, statistics are sane,
routing follows the configs' recipes."""
import numpy as np
import torch

import synth


def test_counter_normal_slices_and_stats():
    z = synth.counter_normal(1 << 20, 7, 3)
    assert torch.equal(synth.counter_normal(1000, 7, 3, offset=5000), z[5000:6000])
    assert abs(z.mean().item()) < 5e-3 and abs(z.std().item() - 1) < 5e-3
    assert z.abs().max().item() <= 6.0
    other = synth.counter_normal(1 << 10, 7, 4)
    assert not torch.equal(other, z[:1 << 10])


def test_expert_weight_rows_regenerate_alone():
    cfg = synth.get_config("c1")
    full = synth.make_expert_weights(cfg, "w13", 2)
    part = synth.make_expert_weights(cfg, "w13", 2, row0=128, rows=64)
    assert torch.equal(full[128:192], part)
    assert full.dtype == torch.bfloat16 and full.shape == (2 * cfg.I, cfg.H)
    assert abs(full.float().std().item() * np.sqrt(cfg.H) - 1) < 0.02


def test_outliers_fraction():
    cfg = synth.get_config("c3")
    x = synth.make_activations(cfg, 64).float()
    frac = (x.abs() > 6.5).float().mean().item()        # |N(0,1)| <= 6 by construction
    assert 0.005 < frac < 0.015


def test_routing_recipes():
    c1 = synth.make_routing(synth.get_config("c1"))
    assert c1["topk_ids"].shape == (64, 2) and np.allclose(c1["topk_w"].sum(1), 1, atol=1e-6)
    c3 = synth.make_routing(synth.get_config("c3"))
    assert list(c3["split"]) == [12600, 5878, 3763, 2742, 2145, 1755, 1482, 1279, 1124]
    assert np.bincount(c3["topk_ids"][:, 0]).tolist() == list(c3["split"])
    c5 = synth.make_routing(synth.get_config("c5"))
    assert c5["topk_ids"].shape == (64, 9) and (c5["topk_ids"][:, 8] == 256).all()
    assert (c5["topk_w"][:, 8] == 1).all() and np.allclose(c5["topk_w"][:, :8].sum(1), 1, atol=1e-6)
    for name, T in (("c5t1", 1), ("c5t4", 4), ("c5t16", 16)):
        r = synth.make_routing(synth.get_config(name))
        assert r["topk_ids"].shape == (T, 9) and (r["topk_ids"][:, 8] == 256).all()
        counts = np.bincount(r["topk_ids"].reshape(-1), minlength=257)
        assert counts.max() <= synth.get_config(name).max_m
    for name in ("c2", "c4"):
        cfg = synth.get_config(name)
        r = synth.make_routing(cfg)
        ids = r["topk_ids"]
        assert ids.shape[1] == 8 and all(len(set(row)) == 8 for row in ids)
        local = (ids >= r["expert_begin"]) & (ids < r["expert_begin"] + cfg.E)
        assert local.any(axis=1).all()
        assert r["raw_counts"].sum() == local.sum()
