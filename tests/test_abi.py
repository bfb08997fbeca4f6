"""The C-ABI library builds, loads and exports every entry point of
include/ra.h; host-side argument validation rejects bad calls synchronously
without touching a GPU."""
import ctypes
import os
import re

import pytest

import block_sparse_flash_ra_gb300 as ra
from block_sparse_flash_ra_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return ra.lib()


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"RA_API\s+[^;(]*?\b(ra_\w+)\s*\(", txt)
    return names


def test_header_declares_the_boundary():
    names = set(_declared())
    for n in ("ra_build_block_mask", "ra_attn_fwd", "ra_merge_out_lse", "ra_attn_bwd",
              "ra_permute_tokens", "ra_unpermute_tokens"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in _declared():
        assert hasattr(L, n), n


def _params(**kw):
    d = dict(B=1, Lq=256, Lkv=256, Hq=4, Hkv=2, D=128, dtype=ra.RA_BF16, scale=0.125,
             soft_cap=0.0, causal=1, is_mqa=0, n_virtual_shards=2, pad_segment_id=-1)
    d.update(kw)
    return ra.RaAttnParams(**d)


@pytest.mark.parametrize("bad", [
    dict(Hq=3, Hkv=2), dict(is_mqa=1, Hkv=2), dict(Lq=200), dict(Lq=384, n_virtual_shards=2),
    dict(n_virtual_shards=0), dict(B=0), dict(dtype=7), dict(scale=0.0),
    dict(local_mask=256),  # a local mask needs causal == 0
    dict(block_q_dkv=32),  # the dK/dV stage's grids: 128 (default) or 64 query rows
])
def test_invalid_params_rejected(L, bad):
    p = _params(**bad)
    assert L.ra_block_mask_bytes(ctypes.byref(p)) == 0
    m = ra.RaBlockMask()
    rc = L.ra_attn_fwd(ctypes.byref(p), 16, 16, 16, ctypes.byref(m), 16, 16, None, 0, None)
    assert rc == ra.RA_ERR_INVALID_ARG
    assert ra.ra_last_error()


def test_backward_grid_of_64_rows_needs_d128(L):
    p = _params(D=64, block_q_dkv=64)
    assert L.ra_block_mask_bytes(ctypes.byref(p)) == 0
    assert "block_q_dkv" in ra.ra_last_error()
    assert L.ra_block_mask_bytes(ctypes.byref(_params(block_q_dkv=64))) > 0


def test_segments_must_come_in_pairs(L):
    p = _params(q_seg=256)
    assert L.ra_block_mask_bytes(ctypes.byref(p)) == 0
    assert "seg" in ra.ra_last_error()


def test_mask_from_other_params_rejected(L):
    p = _params()
    m = ra.RaBlockMask(16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 2, 2, 2, 48, 12345)
    rc = L.ra_attn_fwd(ctypes.byref(p), 16, 16, 16, ctypes.byref(m), 16, 16, None, 0, None)
    assert rc == ra.RA_ERR_INVALID_ARG
    assert "mask" in ra.ra_last_error()


def test_null_tensor_rejected(L):
    p = _params()
    m = ra.RaBlockMask()
    rc = L.ra_attn_fwd(ctypes.byref(p), None, 16, 16, ctypes.byref(m), 16, 16, None, 0, None)
    assert rc == ra.RA_ERR_INVALID_ARG


def test_mask_bytes_cover_every_array(L):
    p = _params(B=2, Lq=512, Lkv=1024, n_virtual_shards=1)
    n = L.ra_block_mask_bytes(ctypes.byref(p))
    nq, nk = 4, 8
    cap = 4 * 2 * (nq + nk)  # partial mask blocks: 4 B (nq + nk) slots of 2 KB, twice
    need = 2 * nq * nk + 4 * (2 * nq + 2 * nq * nk + 2 * nk + 2 * nk * nq + 2 * nq + 2 * nk
                              + 2 * nq * 2  # fwd_shard: N + 1 = 2 offsets per row
                              + 2 * nq * 2 + 2 * nk + 1) + 2 * cap * 128 * 16
    assert n >= need


def test_permute_validation(L):
    assert L.ra_permute_tokens(16, 4096, 1, 10, 4, 4, None) == ra.RA_ERR_INVALID_ARG  # 10 % 8
    assert L.ra_permute_tokens(16, 32, 1, 16, 4, 2, None) == ra.RA_ERR_INVALID_ARG    # overlap
    assert L.ra_unpermute_tokens(None, 4096, 1, 16, 4, 2, None) == ra.RA_ERR_INVALID_ARG


def test_merge_validation(L):
    assert L.ra_merge_out_lse(16, 16, 4096, 16, 1, 1, 1, 6, None) == ra.RA_ERR_INVALID_ARG
    assert L.ra_merge_out_lse(16, 16, 32, 16, 1, 4, 1, 8, None) == ra.RA_ERR_INVALID_ARG


def test_bwd_needs_workspace_and_dsinks(L):
    p = _params(sinks=4096)
    m = ra.RaBlockMask()
    rc = L.ra_attn_bwd(ctypes.byref(p), 16, 16, 16, 16, 16, 16, ctypes.byref(m), 16, 16, 16,
                       None, None, 0, None)
    assert rc == ra.RA_ERR_INVALID_ARG  # dsinks NULL with sinks
    assert L.ra_attn_bwd_workspace_size(ctypes.byref(_params())) >= 4 * 4 * 256


def test_version(L):
    assert "sm_103a" in ra.ra_version()


def test_ring_step_validation(L):
    # checks that come before any device work, for both dtypes
    for dt in (ra.RA_BF16, ra.RA_FP32):
        m = ra.RaBlockMask()
        p2 = _params(dtype=dt)  # two virtual shards: a ring step takes one chunk
        assert L.ra_attn_fwd_step(ctypes.byref(p2), 16, 16, 16, ctypes.byref(m), 0, 16, 16, None,
                                  None) == ra.RA_ERR_INVALID_ARG
        assert "n_virtual_shards" in ra.ra_last_error()
        p1 = _params(dtype=dt, n_virtual_shards=1)
        assert L.ra_attn_fwd_step(ctypes.byref(p1), 16, 16, 16, ctypes.byref(m), 8, 16, 16, None,
                                  None) == ra.RA_ERR_INVALID_ARG  # unknown flag
        assert L.ra_attn_fwd_step(ctypes.byref(p1), 16, 16, 16, ctypes.byref(m), 0, None, 16, None,
                                  None) == ra.RA_ERR_INVALID_ARG  # no running output
        assert L.ra_attn_bwd_step(ctypes.byref(p2), 16, 16, 16, 16, ctypes.byref(m), 16, 16, 16,
                                  4096, 1 << 20, None) == ra.RA_ERR_INVALID_ARG
        assert L.ra_attn_bwd_step(ctypes.byref(p1), 16, 16, 16, 16, None, 16, 16, 16, 4096,
                                  1 << 20, None) == ra.RA_ERR_INVALID_ARG  # no mask
