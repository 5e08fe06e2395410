"""moe_ffn_noalloc: the FFN for callers that cannot allocate device memory
(runtimes that own all device memory, code running under stream capture,
loops that must not touch the allocator).  It keeps the intermediates in the
library's fixed device scratch instead of a caller workspace.

Checked through the C ABI against moe_ffn with a caller workspace, on two
calls in a row (the scratch keeps the previous call's contents, so the second
call must not depend on them), at the tolerance the other GPU tests use; and a
descriptor too large for the scratch must be refused before any launch.
Collected last on purpose: a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

from bench import build_workload, make_desc
from tests.gpu_common import bits, check_tol

pytestmark = pytest.mark.gpu


def _noalloc(lib, desc):
    return lib._lib.moe_ffn_noalloc(ctypes.byref(desc), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice(lib):
    wl = build_workload("c1")
    T, H = wl["T"], wl["cfg"].H
    ref_out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    err = lib.new_error_word()
    desc = make_desc(wl, ref_out, err=err)
    assert lib.moe_ffn_workspace_size(desc) <= lib.moe_ffn_noalloc_capacity()
    lib.moe_ffn(desc, lib.alloc_workspace(desc))
    st, _ = lib.moe_read_device_status(err)
    assert st == 0
    ref = bits(ref_out).copy()
    for call in range(2):
        out = torch.full((T, H), 0x7E57, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        d = make_desc(wl, out, err=err)
        rc = _noalloc(lib, d)
        assert rc == 0, lib.moe_status_string(rc)
        st, _ = lib.moe_read_device_status(err)
        assert st == 0
        check_tol(bits(out), ref, f"noalloc call {call}")


def test_noalloc_refuses_a_workspace_beyond_its_scratch(lib):
    wl = build_workload("c1")
    out = torch.empty((wl["T"], wl["cfg"].H), dtype=torch.bfloat16, device="cuda")
    d = make_desc(wl, out)
    d.max_m = 1 << 20                                   # E * max_m rows far past 64 MiB
    assert lib.moe_ffn_workspace_size(d) > lib.moe_ffn_noalloc_capacity()
    assert _noalloc(lib, d) == lib.MOE_ERR_UNSUPPORTED
