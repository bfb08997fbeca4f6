"""ra_attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (for example code inside a host runtime that owns all of the GPU's
memory, or plain-C callers without an allocator).  It must give the same
gradients as ra_attn_bwd with a caller workspace, call after call, although
its scratch array keeps the previous call's contents.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_flash_ra_gb300 as ra
import oracle
from workloads import Workload, make_inputs

GRAD_TOL = 1e-2  # relative L2, the bar of the other gradient tests


def _rel(a, b):
    a = a.detach().double().cpu().numpy()
    b = b.detach().double().cpu().numpy()
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_twice():
    from block_sparse_flash_ra_gb300 import _build
    _build.build()
    w = Workload("noalloc", B=1, L=1024, Hq=4, Hkv=2, D=128, n_shards=2, sinks=True,
                 soft_cap=20.0, backward=True, seed=41)
    inp = make_inputs(w)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    p = ra.make_params(d["q"], d["k"], scale=w.scale, causal=True, soft_cap=w.soft_cap,
                       n_virtual_shards=2, sinks=d["sinks"])
    mask = ra.build_mask(p)
    out, lse = ra.forward(p, d["q"], d["k"], d["v"], mask)
    ref = ra.backward(p, d["q"], d["k"], d["v"], out, lse, d["dout"], mask)
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    exact = oracle.attn_bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["dout"]),
                            scale=w.scale, soft_cap=w.soft_cap, causal=True,
                            sinks=f64(inp["sinks"]))[:4]
    for call in range(2):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (d["q"], d["k"], d["v"]))
        dsinks = torch.full((w.Hq,), float("nan"), dtype=torch.float32, device="cuda")
        ra.ra_attn_bwd_noalloc(p, d["q"], d["k"], d["v"], out, lse, d["dout"], mask, dq, dk, dv,
                               dsinks)
        torch.cuda.synchronize()
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2]),
                                ("dsinks", dsinks, ref[3])):
            err = _rel(got, want)
            assert err <= GRAD_TOL, (call, name, err)
        # and against the fp64 oracle, at the same bar
        for name, got, want in (("dq", dq, exact[0]), ("dk", dk, exact[1]), ("dv", dv, exact[2]),
                                ("dsinks", dsinks, exact[3])):
            err = _rel(got, torch.from_numpy(want))
            assert err <= GRAD_TOL, (call, name, "oracle", err)
    assert ra.ra_get_device_status() == ra.RA_OK


@pytest.mark.gpu
def test_noalloc_rejects_problems_larger_than_its_scratch():
    # a real block map (the arguments are checked before the size), tensor
    # pointers that are never used: the size check refuses the call before
    # anything is launched
    from block_sparse_flash_ra_gb300 import _build
    _build.build()
    L = ra.lib()
    cap = ra.ra_attn_bwd_noalloc_max_workspace()
    # 64 heads x 65536 rows of Delta alone need 16 MiB > the built-in scratch
    p = ra.RaAttnParams(1, 65536, 65536, 64, 8, 128, ra.RA_BF16, 0.08, 0.0, 1, 0, 1, -1)
    assert L.ra_attn_bwd_workspace_size(ctypes.byref(p)) > cap
    m = ra.build_mask(p)
    rc = L.ra_attn_bwd_noalloc(ctypes.byref(p), 256, 256, 256, 256, 256, 256, ctypes.byref(m),
                               256, 256, 256, None, None)
    assert rc == ra.RA_ERR_WORKSPACE
    assert "scratch" in ra.ra_last_error()
    torch.cuda.synchronize()


def test_noalloc_reports_the_same_errors_as_the_workspace_backward():
    # argument checks only (they run before any CUDA call): the no-workspace
    # entry point returns exactly the code ra_attn_bwd returns
    from block_sparse_flash_ra_gb300 import _build
    _build.build()
    L = ra.lib()
    ws = (ctypes.c_uint8 * 256)()
    cases = {
        # a sequence longer than 2^20 tokens: RA_ERR_UNSUPPORTED, even though
        # its workspace would also exceed the built-in scratch
        "too_long": (ra.RaAttnParams(1, 1 << 21, 1 << 21, 4, 2, 128, ra.RA_BF16, 0.08, 0.0, 1, 0,
                                     1, -1), 256, ra.RA_ERR_UNSUPPORTED),
        # a NULL tensor pointer
        "null_ptr": (ra.RaAttnParams(1, 256, 256, 4, 2, 128, ra.RA_BF16, 0.08, 0.0, 1, 0, 1, -1),
                     None, ra.RA_ERR_INVALID_ARG),
        # a block map that was never built
        "empty_mask": (ra.RaAttnParams(1, 256, 256, 4, 2, 128, ra.RA_BF16, 0.08, 0.0, 1, 0, 1, -1),
                       256, ra.RA_ERR_INVALID_ARG),
    }
    for name, (p, ptr, code) in cases.items():
        m = ra.RaBlockMask()
        a = L.ra_attn_bwd(ctypes.byref(p), ptr, 256, 256, 256, 256, 256, ctypes.byref(m), 256, 256,
                          256, None, ctypes.addressof(ws), 256, None)
        msg_a = ra.ra_last_error()
        b = L.ra_attn_bwd_noalloc(ctypes.byref(p), ptr, 256, 256, 256, 256, 256, ctypes.byref(m),
                                  256, 256, 256, None, None)
        msg_b = ra.ra_last_error()
        assert a == b == code, (name, a, b, msg_a, msg_b)
        assert msg_a == msg_b, name
