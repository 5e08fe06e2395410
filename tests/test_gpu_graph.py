"""moe_ffn is graph-capturable: no host synchronisation and no allocation
inside, counts stay on the device.  Capture the decode step once, replay it on
new inputs copied into the same buffers, and compare with eager calls."""
import numpy as np
import pytest
import torch

from bench import build_workload, make_desc
from tests.gpu_common import bits

pytestmark = pytest.mark.gpu


def test_ffn_captured_in_cuda_graph_matches_eager(lib):
    wl = build_workload("c1")
    T, H = wl["T"], wl["cfg"].H
    out = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    err = lib.new_error_word()
    x_buf = wl["x"].clone()
    desc = make_desc(wl, out, err=err, x=x_buf)
    ws = lib.alloc_workspace(desc)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lib.moe_ffn(desc, ws)                         # warm-up (tensor-map encoder, attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lib.moe_ffn(desc, ws)
    for trial in range(3):
        x_new = wl["x"] * (1.0 + 0.5 * trial)
        x_buf.copy_(x_new)
        g.replay()
        torch.cuda.synchronize()
        got = bits(out).copy()
        lib.moe_ffn(desc, ws)                         # eager on the same inputs
        torch.cuda.synchronize()
        assert np.array_equal(got, bits(out)), f"replay {trial} differs from eager"
    st, _ = lib.moe_read_device_status(err)
    assert st == 0
