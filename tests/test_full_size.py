"""Parity at the full sizes of the benchmark workloads, in the launch
configuration bench.py times (zigzag permutation of the inputs, block map,
forward, backward, unpermutation of the outputs), on sampled outputs that the
fp64 oracle computes one row range at a time.

Sampling stays exact: the oracle restricted to a set of query rows gives
their O, lse and dq exactly, and it gives dk / dv of a key row exactly when
every query row that can see that key lies inside the set (the last rows of a
causal sequence, or the rows of one whole document).  Bars as in the small
parity tests: O max-abs 2e-2, lse max-abs 1e-3, gradients relative L2 1e-2.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_flash_ra_gb300 as ra
import oracle
from workloads import PAD_SEGMENT_ID, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, GRAD_TOL = 2e-2, 1e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_sparse_flash_ra_gb300 import _build
    _build.build()
    yield
    torch.cuda.synchronize()
    assert ra.ra_get_device_status() == ra.RA_OK


def f64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def i32(t):
    return None if t is None else t.detach().cpu().numpy().astype(np.int32)


def rel_l2(a, b):
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def run_gpu(w, inp):
    """The bench pipeline on the device; outputs back in original token order."""
    N = w.n_shards
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    if w.zigzag:
        for key in ("q", "k", "v", "dout", "q_pos", "kv_pos", "q_seg", "kv_seg"):
            if d[key] is not None:
                d[key] = ra.permute(d[key], N)
    p = ra.make_params(d["q"], d["k"], scale=w.scale, causal=w.causal, soft_cap=w.soft_cap,
                       n_virtual_shards=N, is_mqa=w.is_mqa, q_pos=d["q_pos"],
                       kv_pos=d["kv_pos"], q_seg=d["q_seg"], kv_seg=d["kv_seg"],
                       sinks=d["sinks"], pad_segment_id=PAD_SEGMENT_ID,
                       local_mask=d["local_mask"])
    m = ra.build_mask(p)
    out, lse = ra.forward(p, d["q"], d["k"], d["v"], m)
    grads = dsinks = None
    if w.backward:
        dq, dk, dv, dsinks = ra.backward(p, d["q"], d["k"], d["v"], out, lse, d["dout"], m)
        grads = (dq, dk, dv)
    if w.zigzag:
        out = ra.unpermute(out, N)
        # lse is (B, H, L): unpermute along L through a (B, L, H) view
        lse = ra.unpermute(lse.transpose(1, 2).contiguous(), N).transpose(1, 2)
        if grads is not None:
            grads = tuple(ra.unpermute(g, N) for g in grads)
    torch.cuda.synchronize()
    assert ra.ra_get_device_status() == ra.RA_OK
    res = dict(out=f64(out), lse=f64(lse))
    if grads is not None:
        res.update(dq=f64(grads[0]), dk=f64(grads[1]), dv=f64(grads[2]), dsinks=f64(dsinks))
    return res


def oracle_kw(w, inp):
    return dict(scale=w.scale, soft_cap=w.soft_cap or None, causal=w.causal,
                q_pos=i32(inp["q_pos"]), kv_pos=i32(inp["kv_pos"]),
                q_seg=i32(inp["q_seg"]), kv_seg=i32(inp["kv_seg"]),
                sinks=f64(inp["sinks"]), pad_segment_id=PAD_SEGMENT_ID,
                local_mask=None if inp["local_mask"] is None else inp["local_mask"].numpy())


def check_rows(got, w, q, k, v, kw, heads, rows):
    o_ref, l_ref = oracle.attn_fwd(q, k, v, heads=heads, rows=rows, **kw)
    hs, rs = slice(*heads), slice(*rows)
    o, l = got["out"][:, rs, hs], got["lse"][:, hs, rs]
    o_r, l_r = o_ref[:, rs, hs], l_ref[:, hs, rs]
    fin = np.isfinite(l_r)
    assert np.array_equal(np.isfinite(l), fin), (w.name, heads, rows)
    if fin.any():
        assert np.max(np.abs(l[fin] - l_r[fin])) <= LSE_TOL, (w.name, heads, rows)
    assert np.max(np.abs(o - o_r)) <= O_TOL, (w.name, heads, rows)


FWD = ["gqa8k", "mqa32k", "packed16k", "long64k", "gqa32k", "local8k"]


@pytest.mark.parametrize("name", FWD)
def test_full_size_forward_sampled_rows(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    got = run_gpu(w, inp)
    q, k, v = f64(inp["q"]), f64(inp["k"]), f64(inp["v"])
    kw = oracle_kw(w, inp)
    L, H = w.L, w.Hq
    for heads in ((0, 1), (H - 1, H)):
        for rows in ((0, 24), (L // 2 - 12, L // 2 + 12), (L - 24, L)):
            check_rows(got, w, q, k, v, kw, heads, rows)


def _grad_rows(w, inp):
    """Query rows R such that every query row seeing a key in R lies in R,
    with the batch those keys are exact for."""
    if w.packed_docs:
        # the last whole document of batch 0 (segment isolation)
        seg = inp["q_seg"][0].numpy()
        body = seg[seg != PAD_SEGMENT_ID]
        last = body[-1]
        idx = np.nonzero(seg == last)[0]
        lo, hi = int(idx[0]), int(idx[-1]) + 1
        if hi - lo > 1024:  # keep the oracle call short: a tail of the document
            lo = hi - 1024
            # a causal tail of one document only sees keys inside it, and
            # its keys are only seen from inside it
        return (lo, hi), 0
    return (w.L - 128, w.L), None


BWD = ["packed16k", "long64k", "gqa32k", "local8k", "mqa32k"]

# Workloads whose longest dK/dV columns are checked too: under causal masking
# keys 0..127 are seen by every query row, so their dk / dv sum the most
# tiles (every query tile of the sequence, times the heads of the group).
DEEP = ("gqa32k", "long64k")


def _check_deep_columns(w, got, q, k, v, do, kw):
    """dk / dv of the first 128 keys of kv head 0 (original order) against the
    oracle over every query row of the heads of that group: the oracle
    restricted to those keys gives their sums exactly."""
    G = w.Hq // w.Hkv
    _, dk, dv, _, _, _ = oracle.attn_bwd(q, k, v, do, heads=(0, G), keys=(0, 128), **kw)
    assert rel_l2(got["dk"][:, 0:128, 0:1], dk[:, 0:128, 0:1]) <= GRAD_TOL, w.name
    assert rel_l2(got["dv"][:, 0:128, 0:1], dv[:, 0:128, 0:1]) <= GRAD_TOL, w.name


def _check_dsinks(w, q, k, v, do, kw, heads):
    """dsinks of `heads`, which sums exp(sink - lse) Delta over every query row:
    the oracle over all rows of those heads (keys restricted to the last 128,
    which does not change dsinks and keeps the pair loop short)."""
    L = w.L
    _, _, _, ds, _, _ = oracle.attn_bwd(q, k, v, do, heads=heads, keys=(L - 128, L), **kw)
    return ds[heads[0]:heads[1]]


@pytest.mark.parametrize("name", BWD)
def test_full_size_backward_sampled_rows(name):
    w = WORKLOADS[name]
    if not w.backward:
        # a forward-only configuration: its backward drawn with a dO (the
        # shapes, cap, sinks and permutation of the configuration)
        w = w.scaled(backward=True)
    inp = make_inputs(w)
    got = run_gpu(w, inp)
    q, k, v, do = f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["dout"])
    kw = oracle_kw(w, inp)
    G = w.Hq // w.Hkv
    heads = (0, G)  # every query head of kv head 0
    hs = slice(*heads)
    if w.local_window:
        # keys at local index < 128 of every shard are seen only by query rows
        # at local index < 128 + window, in every shard: sum the oracle over
        # those row ranges (each restricted call adds its rows' contributions)
        ls = w.L // w.n_shards
        span = 128 + w.local_window
        dk = dv = 0.0
        for s in range(w.n_shards):
            rows = (s * ls, s * ls + span)
            dq_s, dk_s, dv_s, _, _, _ = oracle.attn_bwd(q, k, v, do, heads=heads, rows=rows, **kw)
            rs = slice(*rows)
            assert rel_l2(got["dq"][:, rs, hs], dq_s[:, rs, hs]) <= GRAD_TOL
            dk = dk + dk_s
            dv = dv + dv_s
        keys = np.concatenate([np.arange(s * ls, s * ls + 128) for s in range(w.n_shards)])
        assert rel_l2(got["dk"][:, keys, 0:1], dk[:, keys, 0:1]) <= GRAD_TOL
        assert rel_l2(got["dv"][:, keys, 0:1], dv[:, keys, 0:1]) <= GRAD_TOL
        return
    rows, batch = _grad_rows(w, inp)
    dq, dk, dv, _, _, _ = oracle.attn_bwd(q, k, v, do, heads=heads, rows=rows, **kw)
    rs = slice(*rows)
    bs = slice(None) if batch is None else slice(batch, batch + 1)
    assert rel_l2(got["dq"][:, rs, hs], dq[:, rs, hs]) <= GRAD_TOL
    assert rel_l2(got["dk"][bs, rs, 0:1], dk[bs, rs, 0:1]) <= GRAD_TOL
    assert rel_l2(got["dv"][bs, rs, 0:1], dv[bs, rs, 0:1]) <= GRAD_TOL
    if name in DEEP:
        _check_deep_columns(w, got, q, k, v, do, kw)
    if w.sinks:
        # dsinks of the first and the last query head, each over all 32K rows
        for hh in ((0, 1), (w.Hq - 1, w.Hq)):
            want = _check_dsinks(w, q, k, v, do, kw, hh)
            assert rel_l2(got["dsinks"][hh[0]:hh[1]], want) <= GRAD_TOL, (name, hh)


def test_full_size_block_map_and_permutation_bit_exact():
    # the benchmark workload: 32K tokens, zigzag over 8 shards
    w = WORKLOADS["gqa32k"]
    N, L = w.n_shards, w.L
    pos = torch.arange(L, dtype=torch.int32).unsqueeze(0)
    dpos = ra.permute(pos.cuda(), N)
    assert np.array_equal(dpos.cpu().numpy(), oracle.permute(pos.numpy(), N))
    q = torch.zeros(1, L, 1, 64, dtype=torch.bfloat16, device="cuda")
    p = ra.make_params(q, q, scale=1.0, causal=True, n_virtual_shards=N, q_pos=dpos,
                       kv_pos=dpos)
    m = ra.build_mask(p)
    torch.cuda.synchronize()
    hp = oracle.permute(pos.numpy(), N)
    ref = oracle.block_mask(1, L, L, causal=True, q_pos=hp, kv_pos=hp)
    nq = nk = L // 128
    buf = m._buf

    def dev_arr(ptr, n, dtype):
        off = ptr - buf.data_ptr()
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return buf[off:off + nbytes].view(dtype).cpu().numpy()

    got = dict(tile_class=dev_arr(m.tile_class, nq * nk, torch.uint8),
               fwd_cnt=dev_arr(m.fwd_cnt, nq, torch.int32),
               fwd_idx=dev_arr(m.fwd_idx, nq * nk, torch.int32),
               bwd_cnt=dev_arr(m.bwd_cnt, nk, torch.int32),
               bwd_idx=dev_arr(m.bwd_idx, nk * nq, torch.int32),
               fwd_order=dev_arr(m.fwd_order, nq, torch.int32),
               bwd_order=dev_arr(m.bwd_order, nk, torch.int32))
    for key, val in got.items():
        assert np.array_equal(val.reshape(-1), np.asarray(ref[key]).reshape(-1)), key


def test_maximum_sequence_length_forward_sampled_rows():
    # the longest sequence the library accepts (2^20 tokens), one head, D = 64
    L = 1 << 20
    g = torch.Generator().manual_seed(71)
    q, k, v = (torch.randn((1, L, 1, 64), generator=g).to(torch.bfloat16) for _ in range(3))
    dq_, dk_, dv_ = q.cuda(), k.cuda(), v.cuda()
    scale = 0.125
    p = ra.make_params(dq_, dk_, scale=scale, causal=True, n_virtual_shards=2)
    m = ra.build_mask(p)
    out, lse = ra.forward(p, dq_, dk_, dv_, m)
    torch.cuda.synchronize()
    assert ra.ra_get_device_status() == ra.RA_OK
    o, l = f64(out), f64(lse)
    q64, k64, v64 = f64(q), f64(k), f64(v)
    for rows in ((0, 16), (L // 2 - 8, L // 2 + 8), (L - 16, L)):
        o_ref, l_ref = oracle.attn_fwd(q64, k64, v64, scale=scale, causal=True, rows=rows)
        rs = slice(*rows)
        assert np.max(np.abs(l[:, :, rs] - l_ref[:, :, rs])) <= LSE_TOL, rows
        assert np.max(np.abs(o[:, rs] - o_ref[:, rs])) <= O_TOL, rows
    # the next admissible length above the limit is refused
    p2 = ra.RaAttnParams(1, L + 256, L + 256, 1, 1, 64, ra.RA_BF16, scale, 0.0, 1, 0, 2, -1)
    assert ra.lib().ra_block_mask_bytes(ctypes.byref(p2)) == 0
