"""Parity of moe_permute with the oracle: counts, offsets, row maps and the
gathered FP8 rows/scales bit-exact; rows with no source keep their sentinel."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_common import SENTINEL_F32, SENTINEL_U8, Guarded, f32_bits, to_dev, u8

pytestmark = pytest.mark.gpu


def _run(lib, ids, expert_begin, E, layout, max_m, H=256, seed=0):
    rng = np.random.default_rng(seed)
    T, k = ids.shape
    q = rng.integers(0, 256, (T, H)).astype(np.uint8)
    T_pad = max(4, (T + 3) // 4 * 4)
    s = np.full((H // 128, T_pad), -1.0, np.float32)
    s[:, :T] = rng.random((H // 128, T)).astype(np.float32)
    dev = "cuda"
    # every output carries a guard band: nothing may be written past its end
    if layout == lib.MOE_LAYOUT_MASKED:
        rows = E * max_m
        gs = Guarded((E, H // 128, max_m), torch.float32, f32_bits(SENTINEL_F32))
        cap = 0
    else:
        cap = lib.moe_contig_rows_bound(T * k, E) + 128
        rows = cap
        gs = Guarded((H // 128, cap), torch.float32, f32_bits(SENTINEL_F32))
    gq = Guarded((rows, H), torch.uint8, SENTINEL_U8)
    outs = [Guarded((n,), torch.int32, -7) for n in (E, E + 1, max(rows, 1), rows, T * k)]
    counts, offsets, m_ind, row_src, dst = [g.t for g in outs]
    s_out, q_out = gs.t, gq.t
    err = lib.new_error_word()
    lib.moe_permute(to_dev(q), to_dev(s), to_dev(ids.astype(np.int32)), expert_begin, E, layout,
                    max_m, q_out, s_out, counts, offsets, m_ind, row_src, dst, rows_capacity=cap,
                    err=err)
    status, raw = lib.moe_read_device_status(err)
    assert all(g.intact() for g in [gs, gq] + outs), "permute wrote past the end of an output"
    ref = oracle.permute(ids, expert_begin, E, "masked" if layout == 0 else "contig", max_m,
                         q=q, s=s[:, :T])
    got = dict(counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(),
               m_indices=m_ind.cpu().numpy(), row_src=row_src.cpu().numpy(),
               dst_row=dst.cpu().numpy(), q=u8(q_out), s=s_out.cpu().numpy(), status=status)
    return got, ref


def _check(lib, got, ref, layout, E, max_m):
    assert np.array_equal(got["counts"], ref["counts"])
    assert np.array_equal(got["dst_row"], ref["dst_row"])
    valid = ref["row_src"] >= 0
    n = ref["rows"]
    assert np.array_equal(got["row_src"][:n], ref["row_src"])
    assert np.array_equal(got["q"][:n][valid], ref["q"][valid])
    assert (got["q"][:n][~valid] == SENTINEL_U8).all(), "rows without a source were written"
    if layout == lib.MOE_LAYOUT_MASKED:
        gs = got["s"].transpose(1, 0, 2).reshape(got["s"].shape[1], -1)
        rs = ref["s"].transpose(1, 0, 2).reshape(ref["s"].shape[1], -1)
        assert np.array_equal(gs[:, valid], rs[:, valid])
        assert (gs[:, ~valid] == SENTINEL_F32).all()
        assert got["status"] == (lib.MOE_ERR_OVERFLOW if ref["overflow"] else 0)
    else:
        assert np.array_equal(got["offsets"], ref["offsets"])
        assert np.array_equal(got["m_indices"][:n], ref["m_indices"])
        assert (got["m_indices"][n:] == -1).all() and (got["row_src"][n:] == -1).all()
        assert np.array_equal(got["s"][:, :n][:, valid], ref["s"][:, valid])
        assert (got["s"][:, :n][:, ~valid] == SENTINEL_F32).all()
        assert got["status"] == 0


@pytest.mark.parametrize("layout", [0, 1])
def test_permute_tiny_config(lib, layout):
    r = synth.make_routing(synth.get_config("c1"))
    got, ref = _run(lib, r["topk_ids"], 0, 4, layout, 128)
    _check(lib, got, ref, layout, 4, 128)


def test_permute_decode_config_with_remote_experts(lib):
    cfg = synth.get_config("c4")
    r = synth.make_routing(cfg)
    got, ref = _run(lib, r["topk_ids"], r["expert_begin"], cfg.E, 0, cfg.max_m, H=512)
    _check(lib, got, ref, 0, cfg.E, cfg.max_m)
    assert got["counts"].sum() == r["raw_counts"].sum()


def test_permute_all_experts_config(lib):
    cfg = synth.get_config("c5")
    r = synth.make_routing(cfg)
    got, ref = _run(lib, r["topk_ids"], 0, cfg.E, 0, cfg.max_m, H=7168)
    _check(lib, got, ref, 0, cfg.E, cfg.max_m)
    assert got["counts"][256] == 64 and got["counts"].sum() == 64 * 9


def test_permute_prefill_contiguous(lib):
    cfg = synth.get_config("c3")
    r = synth.make_routing(cfg)
    got, ref = _run(lib, r["topk_ids"], 0, cfg.E, 1, 0, H=256)
    _check(lib, got, ref, 1, cfg.E, 0)
    assert list(got["counts"]) == list(r["split"])


def test_permute_masked_overflow_clamps_and_reports(lib):
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 3, (300, 2)).astype(np.int32)   # ~200 per expert > max_m=64
    got, ref = _run(lib, ids, 0, 3, 0, 64)
    assert ref["overflow"]
    _check(lib, got, ref, 0, 3, 64)
    assert (got["counts"] == 64).all()


def test_permute_empty_and_ragged(lib):
    ids = np.array([[5, 6]], np.int32)                      # no local expert at all
    for layout in (0, 1):
        got, ref = _run(lib, ids, 0, 4, layout, 16)
        _check(lib, got, ref, layout, 4, 16)
        assert (got["counts"] == 0).all() and (got["dst_row"] == -1).all()
