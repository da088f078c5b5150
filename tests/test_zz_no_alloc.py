"""moe_route_noalloc: routing for callers that cannot allocate device memory
when they call the router (an engine plugin that gets only its input and
output buffers, code where allocating CUDA calls are not allowed).  It must
give the same results as moe_route with a workspace.

The check runs two calls in a row through the C ABI -- the second on a
smaller batch, so a stale histogram left in the shared scratch by the first
call would show up -- and compares each with moe_route on the same inputs:
indices, gates and counts must be identical (same kernels, same order of
arithmetic).  This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from moe_inputs import generate, get_config

pytestmark = pytest.mark.gpu


def _via_abi(moe, fn_name, cfg, u, E, b, with_ws):
    sh = moe.make_shape(cfg.T, cfg.d, cfg.n_routed, cfg.top_k, cfg.n_shared,
                        cfg.d_ff, cfg.dtype)
    idx = torch.full((cfg.T, cfg.top_k), -3, dtype=torch.int32, device="cuda")
    gate = torch.full((cfg.T, cfg.top_k), -1.0, device="cuda")
    counts = torch.full((cfg.n_routed,), -3, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    args = [ctypes.byref(sh), P(u.data_ptr()), P(E.data_ptr()),
            P(b.data_ptr()), P(idx.data_ptr()), P(gate.data_ptr()),
            P(counts.data_ptr())]
    if with_ws:
        ws = torch.empty(moe.workspace_size(sh), dtype=torch.uint8,
                         device="cuda")
        args += [P(ws.data_ptr()), ctypes.c_size_t(ws.numel())]
    st = getattr(moe.LIB, fn_name)(*args, stream)
    assert st == 0, moe.LIB.moe_last_error_detail()
    moe.get_device_error()
    return idx.cpu().numpy(), gate.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("name,T_first,T_second", [("mid", 2000, 300),
                                                   ("tiny", 500, 70)])
def test_route_noalloc_matches_route(name, T_first, T_second):
    import mixture_experts_layer_gemms_b300 as moe
    for T in (T_first, T_second):
        cfg = get_config(name).with_(T=T)
        t = generate(cfg, "cpu", experts=False)
        u, E, b = (t[k].cuda() for k in ("u", "E", "b"))
        ref = _via_abi(moe, "moe_route", cfg, u, E, b, with_ws=True)
        got = _via_abi(moe, "moe_route_noalloc", cfg, u, E, b, with_ws=False)
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_array_equal(got[1], ref[1])
        np.testing.assert_array_equal(got[2], ref[2])
        assert got[2].sum() == T * cfg.top_k


def test_route_noalloc_rejects_oversize():
    import mixture_experts_layer_gemms_b300 as moe
    cfg = get_config("mid").with_(T=200_000, n_routed=256, top_k=8)
    sh = moe.make_shape(cfg.T, cfg.d, cfg.n_routed, cfg.top_k, cfg.n_shared,
                        cfg.d_ff, cfg.dtype)
    P = ctypes.c_void_p
    # never dereferenced: the size check refuses the call before any launch
    st = moe.LIB.moe_route_noalloc(ctypes.byref(sh), P(256), P(512), P(768),
                                   P(1024), P(1280), P(1536), None)
    assert st == 2
    assert b"static scratch" in moe.LIB.moe_last_error_detail()
