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
    assert ra.ra_get_device_status() == ra.RA_OK


def test_noalloc_rejects_problems_larger_than_its_scratch():
    # argument check only: runs before any CUDA call, so it needs no GPU
    from block_sparse_flash_ra_gb300 import _build
    _build.build()
    L = ra.lib()
    cap = ra.ra_attn_bwd_noalloc_max_workspace()
    # 64 heads x 65536 rows of Delta alone need 16 MiB > the built-in scratch
    p = ra.RaAttnParams(1, 65536, 65536, 64, 8, 128, ra.RA_BF16, 0.08, 0.0, 1, 0, 1, -1)
    assert L.ra_attn_bwd_workspace_size(ctypes.byref(p)) > cap
    m = ra.RaBlockMask()
    rc = L.ra_attn_bwd_noalloc(ctypes.byref(p), 256, 256, 256, 256, 256, 256, ctypes.byref(m),
                               256, 256, 256, None, None)
    assert rc == ra.RA_ERR_WORKSPACE
    assert "scratch" in ra.ra_last_error()
