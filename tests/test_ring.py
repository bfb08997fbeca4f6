"""The ring run step by step through the C ABI (ra_attn_fwd_step,
ra_attn_bwd_prep, ra_attn_bwd_step, ra_cast_from_f32, ra_add_f32), against
the fp64 oracle: N virtual devices on one GPU, and two processes that pass
their chunks over gloo (host memory), each running its device's steps on the
GPU -- every kernel call is a one-GPU call and no kernel waits on another.

Bars as in the other parity tests: O max-abs 2e-2, lse max-abs 1e-3,
gradients relative L2 1e-2.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import block_sparse_flash_ra_gb300 as ra
import oracle
from block_sparse_flash_ra_gb300 import ring
from workloads import PAD_SEGMENT_ID, Workload, make_inputs, random_structure

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


CASES = {
    "causal_gqa_n4": dict(w=Workload("r1", 1, 512, 4, 2, 128, n_shards=4, backward=True, seed=61)),
    "mqa_sinks_cap20_zigzag_n2": dict(w=Workload("r2", 1, 512, 4, 1, 128, n_shards=2, zigzag=True,
                                                 soft_cap=20.0, sinks=True, is_mqa=True,
                                                 backward=True, seed=62)),
    "segments_padding_noncausal_b2_n2": dict(w=Workload("r3", 2, 512, 4, 2, 128, causal=False,
                                                        n_shards=2, backward=True, seed=63),
                                             segs=True),
    "d64_causal_n2_sinks": dict(w=Workload("r4", 1, 256, 2, 2, 64, n_shards=2, sinks=True,
                                           backward=True, seed=64)),
    "causal_n8_one_tile_each": dict(w=Workload("r5", 1, 1024, 2, 1, 128, n_shards=8,
                                               backward=True, seed=65)),
    # fp32 inputs: the tiny workload's shapes (B1 Hq=Hkv=2 L256 D64, 2 shards)
    # and a GQA one with sinks, soft cap and zigzag; the forward keeps fp32
    # logits (tf32 hi / lo products), so it is held to the fp32 bars
    "tiny_fp32_n2": dict(w=Workload("r6", 1, 256, 2, 2, 64, dtype="fp32", n_shards=2,
                                    backward=True, seed=0), f32=True),
    "fp32_gqa_sinks_cap20_zigzag_n4": dict(w=Workload("r7", 1, 1024, 4, 2, 128, dtype="fp32",
                                                      n_shards=4, zigzag=True, soft_cap=20.0,
                                                      sinks=True, backward=True, seed=67),
                                           f32=True),
}

# fp32 forward bars (as for ra_attn_fwd on fp32 inputs): lse and O well inside
# what a bf16 rounding of q and k would allow
F32_LSE_TOL, F32_O_TOL = 1e-4, 4e-3


def _prepare(case):
    """Device inputs of a case in the ring's token order, and the oracle kwargs."""
    w = case["w"]
    inp = make_inputs(w)
    N, L = w.n_shards, w.L
    seg = pos = None
    if case.get("segs"):
        seg, _ = random_structure(torch.Generator().manual_seed(w.seed), w.B, L, n_docs_max=3,
                                  pad_max=40)
    if w.zigzag:
        perm = oracle.permute(np.arange(L)[None], N)[0]
        for key in ("q", "k", "v", "dout"):
            inp[key] = inp[key][:, perm].contiguous()
        pos = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(perm, (w.B, L))).astype(np.int32))
    d = {key: (t.cuda() if isinstance(t, torch.Tensor) else t) for key, t in inp.items()}
    kw = dict(scale=w.scale, causal=w.causal, soft_cap=w.soft_cap, is_mqa=w.is_mqa,
              sinks=d["sinks"], pad_segment_id=PAD_SEGMENT_ID)
    geo = dict(q_pos=None if pos is None else pos.cuda(), kv_pos=None if pos is None else pos.cuda(),
               q_seg=None if seg is None else seg.cuda(), kv_seg=None if seg is None else seg.cuda())
    okw = dict(scale=w.scale, causal=w.causal, soft_cap=w.soft_cap or None, sinks=f64(inp["sinks"]),
               q_pos=i32(pos), kv_pos=i32(pos), q_seg=i32(seg), kv_seg=i32(seg),
               pad_segment_id=PAD_SEGMENT_ID)
    return w, inp, d, kw, geo, okw


def _compare(w, inp, okw, out, lse, grads, f32=False):
    q, k, v, do = (f64(inp[key]) for key in ("q", "k", "v", "dout"))
    o_ref, l_ref = oracle.attn_fwd(q, k, v, **okw)
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.max(np.abs(lse[fin] - l_ref[fin])) <= (F32_LSE_TOL if f32 else LSE_TOL)
    assert np.max(np.abs(out - o_ref)) <= (F32_O_TOL if f32 else O_TOL)
    dq, dk, dv, ds, _, _ = oracle.attn_bwd(q, k, v, do, **okw)
    for name, got, ref in (("dq", grads[0], dq), ("dk", grads[1], dk), ("dv", grads[2], dv)):
        assert rel_l2(got, ref) <= GRAD_TOL, name
    if ds is not None:
        assert rel_l2(grads[3], ds) <= GRAD_TOL, "dsinks"


@pytest.mark.parametrize("name", list(CASES))
def test_ring_steps_on_virtual_devices_match_oracle(name):
    w, inp, d, kw, geo, okw = _prepare(CASES[name])
    N = w.n_shards
    outs, lses = ring.ring_forward_local(d["q"], d["k"], d["v"], N, **geo, **kw)
    dqs, dks, dvs, dsinks = ring.ring_backward_local(d["q"], d["k"], d["v"], outs, lses, d["dout"],
                                                     N, **geo, **kw)
    torch.cuda.synchronize()
    assert ra.ra_get_device_status() == ra.RA_OK
    for t in list(outs) + list(dqs) + list(dks) + list(dvs):
        assert t.dtype == w.torch_dtype  # results in the input dtype
    out = np.concatenate([f64(o) for o in outs], 1)
    lse = np.concatenate([f64(x) for x in lses], 2)
    grads = (np.concatenate([f64(x) for x in dqs], 1), np.concatenate([f64(x) for x in dks], 1),
             np.concatenate([f64(x) for x in dvs], 1), f64(dsinks))
    _compare(w, inp, okw, out, lse, grads, CASES[name].get("f32", False))


@pytest.mark.parametrize("name", ["mqa_sinks_cap20_zigzag_n2", "fp32_gqa_sinks_cap20_zigzag_n4"])
def test_ring_step_forward_equals_the_fused_ring(name):
    # the same ring, once step by step and once in the single-launch forward
    # (ra_attn_fwd over N virtual shards): both are the pages' ring; they
    # differ only in rounding
    w, inp, d, kw, geo, okw = _prepare(CASES[name])
    N = w.n_shards
    outs, lses = ring.ring_forward_local(d["q"], d["k"], d["v"], N, **geo, **kw)
    p = ra.make_params(d["q"], d["k"], scale=w.scale, causal=True, soft_cap=w.soft_cap,
                       n_virtual_shards=N, is_mqa=w.is_mqa, q_pos=geo["q_pos"],
                       kv_pos=geo["kv_pos"], sinks=d["sinks"])
    out_f, lse_f = ra.forward(p, d["q"], d["k"], d["v"], ra.build_mask(p))
    torch.cuda.synchronize()
    out = np.concatenate([f64(o) for o in outs], 1)
    lse = np.concatenate([f64(x) for x in lses], 2)
    f32 = CASES[name].get("f32", False)
    assert np.max(np.abs(out - f64(out_f))) <= (F32_O_TOL if f32 else O_TOL)
    assert np.max(np.abs(lse - f64(lse_f))) <= (F32_LSE_TOL if f32 else LSE_TOL)


def test_step_with_an_empty_chunk_and_sinks_keeps_the_running_pair():
    # a chunk that no query row can see (causal, the chunk lies after every
    # query) with the sink flag: the partial is (0, sink); without it the
    # running pair must come back unchanged
    g = torch.Generator().manual_seed(66)
    B, L, H, D = 1, 256, 2, 128
    q, k, v = (torch.randn(B, L, H, D, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    sinks = torch.randn(H, generator=g).cuda()
    qpos = torch.arange(L, dtype=torch.int32)[None].cuda()
    kpos = (qpos + L).contiguous()
    p = ra.make_params(q, k, scale=0.1, causal=True, q_pos=qpos, kv_pos=kpos, sinks=sinks)
    m = ra.build_mask(p)
    o_run = torch.randn(B, L, H, D, generator=g).cuda()
    l_run = torch.randn(B, H, L, generator=g).cuda()
    o0, l0 = o_run.clone(), l_run.clone()
    ra.ra_attn_fwd_step(p, q, k, v, m, 0, o_run, l_run)
    torch.cuda.synchronize()
    assert torch.equal(o_run, o0) and torch.equal(l_run, l0)
    ra.ra_attn_fwd_step(p, q, k, v, m, ra.RA_STEP_SINKS, o_run, l_run)
    torch.cuda.synchronize()
    ro, rl = oracle.merge(f64(o0), f64(l0), np.zeros((B, L, H, D)),
                          np.broadcast_to(f64(sinks)[None, :, None], (B, H, L)).copy())
    assert np.max(np.abs(f64(l_run) - rl)) <= 1e-5
    assert np.max(np.abs(f64(o_run) - ro)) <= 1e-5


def test_step_arguments_are_checked():
    q = torch.zeros(1, 256, 2, 128, dtype=torch.bfloat16, device="cuda")
    p = ra.make_params(q, q, scale=0.1, causal=True, n_virtual_shards=2)
    m = ra.build_mask(p)
    o = torch.zeros(1, 256, 2, 128, device="cuda")
    lse = torch.zeros(1, 2, 256, device="cuda")
    with pytest.raises(ra.RaError) as e:
        ra.ra_attn_fwd_step(p, q, q, q, m, 0, o, lse)  # a step takes one chunk
    assert e.value.code == ra.RA_ERR_INVALID_ARG
    p1 = ra.make_params(q, q, scale=0.1, causal=True)
    m1 = ra.build_mask(p1)
    with pytest.raises(ra.RaError):
        ra.ra_attn_fwd_step(p1, q, q, q, m1, 8, o, lse)  # unknown flag
    with pytest.raises(ra.RaError):
        ra.ra_attn_fwd_step(p1, q, q, q, m1, 0, None, lse)
    # fp32: the optional output may not share memory with the running output
    q32 = torch.zeros(1, 256, 2, 128, device="cuda")
    p32 = ra.make_params(q32, q32, scale=0.1, causal=True)
    m32 = ra.build_mask(p32)
    with pytest.raises(ra.RaError) as e:
        ra.ra_attn_fwd_step(p32, q32, q32, q32, m32, ra.RA_STEP_FIRST, o, lse, o)
    assert e.value.code == ra.RA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert ra.ra_get_device_status() == ra.RA_OK


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, resq):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        torch.cuda.set_device(0)
        w, inp, d, kw, geo, okw = _prepare(CASES["mqa_sinks_cap20_zigzag_n2"])
        Ls = w.L // ws
        sl = slice(rank * Ls, (rank + 1) * Ls)
        mine = {key: d[key][:, sl].contiguous() for key in ("q", "k", "v", "dout")}
        pos = geo["q_pos"][:, sl].contiguous()
        comm = ring.DistComm()
        out, lse = ring.run_dist(ring.forward_device(mine["q"], mine["k"], mine["v"],
                                                     device_idx=rank, n_devices=ws, q_pos=pos,
                                                     kv_pos=pos, **kw), comm)
        dq, dk, dv, ds = ring.run_dist(ring.backward_device(
            mine["q"], mine["k"], mine["v"], out, lse, mine["dout"], device_idx=rank,
            n_devices=ws, q_pos=pos, kv_pos=pos, **kw), comm)
        ds = comm.all_reduce_sum(ds)
        torch.cuda.synchronize()
        status = ra.ra_get_device_status()
        resq.put((rank, status, f64(out), f64(lse), f64(dq), f64(dk), f64(dv), f64(ds)))
    finally:
        dist.destroy_process_group()


def test_two_processes_exchange_chunks_over_gloo():
    ctx = mp.get_context("spawn")
    resq = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, resq)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((resq.get(timeout=300) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(r[1] == ra.RA_OK for r in res)
    w, inp, d, kw, geo, okw = _prepare(CASES["mqa_sinks_cap20_zigzag_n2"])
    out = np.concatenate([r[2] for r in res], 1)
    lse = np.concatenate([r[3] for r in res], 2)
    grads = (np.concatenate([r[4] for r in res], 1), np.concatenate([r[5] for r in res], 1),
             np.concatenate([r[6] for r in res], 1), res[0][7])
    np.testing.assert_array_equal(res[0][7], res[1][7])
    _compare(w, inp, okw, out, lse, grads)
