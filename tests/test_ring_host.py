"""The host side of the ring (block_sparse_flash_ra_gb300/ring.py) on the CPU.

The ring's schedule -- device d holds chunk (d - t) mod N at step t, the
sinks only at step 0, dk / dv travelling with their chunk and home after N
shifts, the dsinks psum -- runs here with fp64 step operations built on the
oracle (the plain attention of a chunk and the pages' merge) and a numpy
restatement of a chunk's gradient with the final lse.  The assembled result
must equal the oracle's plain attention and exact gradient over the whole
sequence.  Two cases run the ring as two gloo ranks exchanging chunks
through torch.distributed, one as virtual devices in one process.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from block_sparse_flash_ra_gb300 import RA_STEP_FIRST, RA_STEP_SINKS, ring
from tests import brute


def _np(t):
    return None if t is None else t.detach().cpu().numpy()


class OracleOps:
    """The ring's per-step work in fp64 on the CPU."""

    @staticmethod
    def _kw(cfg, chunk):
        return dict(scale=cfg["scale"], soft_cap=cfg["soft_cap"] or None, causal=cfg["causal"],
                    q_pos=_np(cfg["q_pos"]), kv_pos=_np(chunk["kv_pos"]), q_seg=_np(cfg["q_seg"]),
                    kv_seg=_np(chunk["kv_seg"]), pad_segment_id=cfg["pad_segment_id"])

    def fwd_step(self, q, chunk, cfg, flags, out_run, lse_run, out):
        sinks = _np(cfg["sinks"]) if flags & RA_STEP_SINKS else None
        o_s, l_s = oracle.attn_fwd(_np(q), _np(chunk["k"]), _np(chunk["v"]), sinks=sinks,
                                   **self._kw(cfg, chunk))
        if flags & RA_STEP_FIRST:
            o_run, l_run = np.zeros(o_s.shape), np.full(l_s.shape, -np.inf)
        else:
            o_run, l_run = _np(out_run).astype(np.float64), _np(lse_run).astype(np.float64)
        o, l = oracle.merge(o_run, l_run, o_s, l_s)
        out_run.copy_(torch.from_numpy(o))
        lse_run.copy_(torch.from_numpy(l))
        if out is not None:
            out.copy_(torch.from_numpy(o))

    def bwd_prep(self, q, chunk, cfg, out, lse, dout):
        delta = np.einsum("bihd,bihd->bhi", _np(dout).astype(np.float64), _np(out).astype(np.float64))
        ws = dict(delta=delta, lse=_np(lse).astype(np.float64))
        dsinks = None
        if cfg["sinks"] is not None:
            s = _np(cfg["sinks"]).astype(np.float64)
            with np.errstate(over="ignore"):
                w = np.where(np.isfinite(ws["lse"]), np.exp(s[None, :, None] - ws["lse"]), 0.0)
            dsinks = torch.from_numpy(-(w * delta).sum(axis=(0, 2)))
        return ws, dsinks

    def bwd_step(self, q, chunk, cfg, dout, ws, dq_acc):
        kw = self._kw(cfg, chunk)
        dq, dk, dv = brute.chunk_grads(_np(q), _np(chunk["k"]), _np(chunk["v"]), _np(dout),
                                       ws["lse"], ws["delta"], scale=kw["scale"],
                                       soft_cap=kw["soft_cap"], causal=kw["causal"],
                                       q_pos=kw["q_pos"], kv_pos=kw["kv_pos"], q_seg=kw["q_seg"],
                                       kv_seg=kw["kv_seg"], pad=kw["pad_segment_id"])
        dq_acc += torch.from_numpy(dq).to(dq_acc.dtype)
        chunk["dk"] += torch.from_numpy(dk).to(chunk["dk"].dtype)
        chunk["dv"] += torch.from_numpy(dv).to(chunk["dv"].dtype)

    def cast(self, acc, like):
        return acc.to(like.dtype)

    def add(self, acc, x):
        acc += x


CASE = dict(B=1, L=64, Hq=4, Hkv=2, D=8)


def _inputs(seed, *, B, L, Hq, Hkv, D, segs=False):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, L, Hq, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, L, Hkv, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, L, Hkv, D, generator=g, dtype=torch.float64)
    do = torch.randn(B, L, Hq, D, generator=g, dtype=torch.float64)
    sinks = torch.randn(Hq, generator=g, dtype=torch.float64)
    seg = None
    if segs:
        seg = torch.zeros(B, L, dtype=torch.int32)
        seg[:, L // 3:] = 1
        seg[:, L - 5:] = -1
    return q, k, v, do, sinks, seg


def _check(out, lse, grads, q, k, v, do, kw):
    o_ref, l_ref = oracle.attn_fwd(_np(q), _np(k), _np(v), **kw)
    np.testing.assert_allclose(_np(out), o_ref, atol=1e-5)
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(_np(lse)), fin)
    np.testing.assert_allclose(_np(lse)[fin], l_ref[fin], atol=1e-5)
    dq, dk, dv, ds, _, _ = oracle.attn_bwd(_np(q), _np(k), _np(v), _np(do), **kw)
    np.testing.assert_allclose(_np(grads[0]), dq, atol=1e-5)
    np.testing.assert_allclose(_np(grads[1]), dk, atol=1e-5)
    np.testing.assert_allclose(_np(grads[2]), dv, atol=1e-5)
    if ds is not None:
        np.testing.assert_allclose(_np(grads[3]), ds, atol=1e-5)


@pytest.mark.parametrize("n", [1, 2, 4])
@pytest.mark.parametrize("case", ["causal_sinks_cap", "segments_noncausal", "zigzag_positions"])
def test_local_ring_schedule_matches_oracle(n, case):
    q, k, v, do, sinks, seg = _inputs(3 + n, segs=case == "segments_noncausal", **CASE)
    L = CASE["L"]
    kw = dict(scale=0.3, causal=case != "segments_noncausal",
              soft_cap=2.0 if case == "causal_sinks_cap" else 0.0,
              sinks=sinks if case == "causal_sinks_cap" else None)
    pos = None
    if case == "zigzag_positions":
        perm = oracle.permute(np.arange(L)[None], n)[0]       # the permuted token order
        q, k, v, do = (t[:, perm].contiguous() for t in (q, k, v, do))
        pos = torch.from_numpy(perm.astype(np.int32))[None].contiguous()
    ops = OracleOps()
    outs, lses = ring.ring_forward_local(q, k, v, n, ops=ops, q_pos=pos, kv_pos=pos, q_seg=seg,
                                         kv_seg=seg, **kw)
    dqs, dks, dvs, dsinks = ring.ring_backward_local(q, k, v, outs, lses, do, n, ops=ops,
                                                     q_pos=pos, kv_pos=pos, q_seg=seg,
                                                     kv_seg=seg, **kw)
    out, lse = torch.cat(outs, 1), torch.cat(lses, 2)
    grads = (torch.cat(dqs, 1), torch.cat(dks, 1), torch.cat(dvs, 1), dsinks)
    okw = dict(scale=kw["scale"], causal=kw["causal"], soft_cap=kw["soft_cap"] or None,
               sinks=_np(kw["sinks"]), q_seg=_np(seg), kv_seg=_np(seg), q_pos=_np(pos),
               kv_pos=_np(pos))
    _check(out, lse, grads, q, k, v, do, okw)


def test_ring_sources_follow_the_pages_order():
    # device d holds the chunk of source (d - t) mod N at step t: the chunk
    # dicts carry their kv positions, so the schedule can be read off them
    n, Ls = 4, 4
    k = torch.zeros(1, n * Ls, 1, 1)
    pos = torch.arange(n * Ls, dtype=torch.int32)[None]
    seen = {d: [] for d in range(n)}

    class Spy(OracleOps):
        def __init__(self, d):
            self.d = d

        def fwd_step(self, q, chunk, cfg, flags, out_run, lse_run, out):
            seen[self.d].append((int(chunk["kv_pos"][0, 0]) // Ls, flags))

    shards = ring._shards
    gens = [ring.forward_device(shards(k, n)[d], shards(k, n)[d], shards(k, n)[d], device_idx=d,
                                n_devices=n, scale=1.0, causal=True, q_pos=shards(pos, n)[d],
                                kv_pos=shards(pos, n)[d], sinks=torch.zeros(1), ops=Spy(d))
            for d in range(n)]
    ring.run_local(gens)
    for d in range(n):
        assert [s for s, _ in seen[d]] == [oracle.ring_source(d, t, n) for t in range(n)]
        assert [f for _, f in seen[d]] == [RA_STEP_FIRST | RA_STEP_SINKS] + [0] * (n - 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, resq):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        q, k, v, do, sinks, _ = _inputs(11, **CASE)
        n = ws
        Ls = CASE["L"] // n
        sl = slice(rank * Ls, (rank + 1) * Ls)
        mine = [t[:, sl].contiguous() for t in (q, k, v, do)]
        kw = dict(scale=0.3, causal=True, soft_cap=2.0, sinks=sinks, ops=OracleOps())
        comm = ring.DistComm()
        out, lse = ring.run_dist(ring.forward_device(*mine[:3], device_idx=rank, n_devices=n, **kw),
                                 comm)
        dq, dk, dv, ds = ring.run_dist(
            ring.backward_device(*mine[:3], out, lse, mine[3], device_idx=rank, n_devices=n, **kw),
            comm)
        ds = comm.all_reduce_sum(ds)
        resq.put((rank, out.numpy(), lse.numpy(), dq.numpy(), dk.numpy(), dv.numpy(), ds.numpy()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_the_ring():
    ctx = mp.get_context("spawn")
    resq = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, resq)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((resq.get(timeout=180) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    q, k, v, do, sinks, _ = _inputs(11, **CASE)
    cat = lambda i, ax: torch.from_numpy(np.concatenate([r[i] for r in res], ax))  # noqa: E731
    out, lse = cat(1, 1), cat(2, 2)
    grads = (cat(3, 1), cat(4, 1), cat(5, 1), torch.from_numpy(res[0][6]))
    np.testing.assert_array_equal(res[0][6], res[1][6])  # the psum reached both ranks
    okw = dict(scale=0.3, causal=True, soft_cap=2.0, sinks=_np(sinks))
    _check(out, lse, grads, q, k, v, do, okw)
