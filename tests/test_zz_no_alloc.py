"""moe_ffn_noalloc: the FFN for callers that cannot allocate device memory
(runtimes that own all device memory, code running under stream capture,
loops that must not touch the allocator).  It keeps the intermediates in the
library's fixed device scratch instead of a caller workspace.

Checked through the C ABI against moe_ffn with a fresh caller workspace, on
two calls in a row with different workloads: the scratch keeps the previous
call's contents, so the first call leaves values in it that the second call
would not write (other activations, other routing, two experts that the second
call fills left empty), and the second call's output must still equal moe_ffn's
bit for bit (same kernels, same inputs).  A descriptor too large for the scratch
must be refused before any launch.  Collected last on purpose: a failure here
leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

from bench import build_workload, make_desc
from tests.gpu_common import SENTINEL_BF16, bits

pytestmark = pytest.mark.gpu


def _noalloc(lib, desc):
    return lib._lib.moe_ffn_noalloc(ctypes.byref(desc), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _sentinel_out(wl):
    T, H = wl["T"], wl["cfg"].H
    return torch.full((T, H), SENTINEL_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def _ffn_fresh_workspace(lib, wl, err):
    """moe_ffn with a newly allocated caller workspace (filled with 0xFF bytes)."""
    out = _sentinel_out(wl)
    desc = make_desc(wl, out, err=err)
    ws = lib.alloc_workspace(desc)
    ws.fill_(0xFF)
    lib.moe_ffn(desc, ws)
    st, _ = lib.moe_read_device_status(err)
    assert st == lib.MOE_OK
    return bits(out).copy()


def _other_workload(wl):
    """The tiny config's shapes with other inputs: x negated and every token
    routed to experts 0 and 1 (experts 2 and 3 empty)."""
    other = dict(wl)
    other["x"] = -wl["x"]
    ids = torch.zeros_like(wl["topk_ids"])
    ids[:, 1] = 1
    other["topk_ids"] = ids
    return other


def test_noalloc_matches_workspace_entry_point_twice(lib):
    c1 = build_workload("c1")
    other = _other_workload(c1)
    err = lib.new_error_word()
    assert lib.moe_ffn_workspace_size(make_desc(c1, _sentinel_out(c1))) <= lib.moe_ffn_noalloc_capacity()
    refs = [_ffn_fresh_workspace(lib, wl, err) for wl in (other, c1)]
    assert not np.array_equal(refs[0], refs[1])
    for call, (wl, ref) in enumerate(zip((other, c1), refs)):
        out = _sentinel_out(wl)
        rc = _noalloc(lib, make_desc(wl, out, err=err))
        assert rc == lib.MOE_OK, lib.moe_status_string(rc)
        st, _ = lib.moe_read_device_status(err)
        assert st == lib.MOE_OK
        assert np.array_equal(bits(out), ref), f"noalloc call {call} differs from moe_ffn"


def test_noalloc_refuses_a_workspace_beyond_its_scratch(lib):
    wl = build_workload("c1")
    out = torch.empty((wl["T"], wl["cfg"].H), dtype=torch.bfloat16, device="cuda")
    d = make_desc(wl, out)
    d.max_m = 1 << 20                                   # E * max_m rows far past 64 MiB
    assert lib.moe_ffn_workspace_size(d) > lib.moe_ffn_noalloc_capacity()
    assert _noalloc(lib, d) == lib.MOE_ERR_UNSUPPORTED
