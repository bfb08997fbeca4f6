"""Failure detection without a GPU fault: every in-kernel wait of the library
is bounded.  A wait that can never complete gives up after its limit, the
kernel records RA_ERR_TIMEOUT in the device status word and returns, the host
reads the status, and the context keeps working for the next call."""
import ctypes

import pytest
import torch

import block_sparse_flash_ra_gb300 as ra
import oracle
from workloads import Workload, make_inputs


def test_selftest_argument_check_needs_no_gpu():
    from block_sparse_flash_ra_gb300 import _build
    _build.build()
    assert ra.lib().ra_selftest_wait_timeout(1000, None, None) == ra.RA_ERR_INVALID_ARG
    assert "gave_up" in ra.ra_last_error()


@pytest.mark.gpu
def test_wait_that_never_completes_times_out_and_context_survives():
    from block_sparse_flash_ra_gb300 import _build
    _build.build()
    assert ra.ra_get_device_status() == ra.RA_OK          # clean start
    gave_up = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ra.ra_selftest_wait_timeout(2_000_000, gave_up)        # 2 ms limit
    assert ra.ra_get_device_status() == ra.RA_ERR_TIMEOUT
    assert int(gave_up.item()) == 1
    assert ra.ra_get_device_status() == ra.RA_OK          # reading resets the word
    # the context is still usable: a small forward matches the oracle
    w = Workload("after_timeout", B=1, L=512, Hq=2, Hkv=1, D=128, n_shards=2, seed=77)
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    p = ra.make_params(d["q"], d["k"], scale=w.scale, causal=True, n_virtual_shards=2)
    out, lse = ra.forward(p, d["q"], d["k"], d["v"], ra.build_mask(p))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attn_fwd_ring(*(inp[k].double().numpy() for k in ("q", "k", "v")),
                                        scale=w.scale, causal=True, n_shards=2)
    assert abs(out.double().cpu().numpy() - o_ref).max() <= 2e-2
    assert abs(lse.double().cpu().numpy() - l_ref).max() <= 1e-3
    assert ra.ra_get_device_status() == ra.RA_OK
