"""The ring of devices around the per-step entry points, driven by the host.

"ejKernel ring_attention._ring_splash" module source:

* ``_ring_attention_forward`` -- device ``d`` keeps its query shard; at step
  ``t`` it holds the key/value chunk of source ``(d - t) mod N`` (the initial
  source is its own index, each step's chunk comes from device ``d - 1``: the
  ``ppermute`` to ``(i + 1) mod N``), computes that chunk's partial
  ``(out, lse)`` -- the sinks only at step 0 -- and merges it into the running
  pair with ``_update_out_and_lse``; the result is cast to the query dtype.
* ``_ring_attention_backward`` -- with the final ``out`` and ``lse``, each step
  adds the pair's gradients to ``dq`` (kept locally) and to ``dk`` / ``dv``
  accumulators that travel with their chunk; after ``N`` shifts every chunk
  is back home with its complete ``dk`` / ``dv``; ``dsinks`` is summed over
  the ring (``psum``); the gradients are cast to the input dtypes.

Every step runs in the library's kernels (``ra_attn_fwd_step``,
``ra_attn_bwd_prep``, ``ra_attn_bwd_step``, ``ra_cast_from_f32``,
``ra_add_f32``).  The host only schedules them and moves chunks:

* each device's work is a generator that yields the chunk it holds after a
  step and is sent the chunk of its left neighbour;
* ``run_local`` drives ``N`` virtual devices on one GPU (a shift is a
  rotation of references, nothing is copied);
* ``run_dist`` drives this rank's device in a ``torch.distributed`` process
  group: a shift sends every tensor of the chunk to ``rank + 1`` and receives
  ``rank - 1``'s into local buffers (device tensors over NCCL; over gloo the
  tensors are staged through host memory), and ``dsinks`` is all-reduced.

Positions: the causal rule compares positions that travel with the tokens.
When none are given, device ``d``'s rows get their global indices
``d * L_local + i``, which is the pages' per-step offset
``device_idx * q_len - kv_src * kv_len``.
"""
from __future__ import annotations

import torch

from . import (RA_BF16, RA_FP32, RA_STEP_FIRST, RA_STEP_SINKS, build_mask, make_params,
               ra_add_f32, ra_attn_bwd_prep, ra_attn_bwd_step, ra_attn_bwd_workspace_size,
               ra_attn_fwd_step, ra_cast_from_f32)

_CHUNK_KEYS = ("k", "v", "kv_pos", "kv_seg", "dk", "dv")


def _dtype_code(t):
    return RA_BF16 if t.dtype == torch.bfloat16 else RA_FP32


def _global_positions(B, n, device_idx, device):
    """Rows of device ``device_idx`` of a sequence split into shards of ``n``."""
    ar = torch.arange(device_idx * n, (device_idx + 1) * n, dtype=torch.int32, device=device)
    return ar.unsqueeze(0).repeat(B, 1).contiguous()


class KernelOps:
    """The ring's per-step work on this library's kernels (the default)."""

    @staticmethod
    def _params(q, chunk, cfg):
        return make_params(q, chunk["k"], scale=cfg["scale"], causal=cfg["causal"],
                           soft_cap=cfg["soft_cap"], n_virtual_shards=1, is_mqa=cfg["is_mqa"],
                           pad_segment_id=cfg["pad_segment_id"], q_pos=cfg["q_pos"],
                           kv_pos=chunk["kv_pos"], q_seg=cfg["q_seg"], kv_seg=chunk["kv_seg"],
                           sinks=cfg["sinks"])

    def fwd_step(self, q, chunk, cfg, flags, out_run, lse_run, out):
        p = self._params(q, chunk, cfg)
        ra_attn_fwd_step(p, q, chunk["k"], chunk["v"], build_mask(p), flags, out_run, lse_run, out)

    def bwd_prep(self, q, chunk, cfg, out, lse, dout):
        p = self._params(q, chunk, cfg)
        ws = torch.empty(ra_attn_bwd_workspace_size(p), dtype=torch.uint8, device=q.device)
        dsinks = (torch.empty(q.shape[2], dtype=torch.float32, device=q.device)
                  if cfg["sinks"] is not None else None)
        ra_attn_bwd_prep(p, out, lse, dout, dsinks, ws)
        return ws, dsinks

    def bwd_step(self, q, chunk, cfg, dout, ws, dq_acc):
        p = self._params(q, chunk, cfg)
        ra_attn_bwd_step(p, q, chunk["k"], chunk["v"], dout, build_mask(p), dq_acc, chunk["dk"],
                         chunk["dv"], ws)

    def cast(self, acc, like):
        dst = torch.empty_like(like)
        ra_cast_from_f32(acc, dst, acc.numel(), _dtype_code(dst))
        return dst

    def add(self, acc, x):
        ra_add_f32(acc, x, acc.numel())


def forward_device(q, k, v, *, device_idx, n_devices, scale, causal=False, soft_cap=0.0,
                   is_mqa=False, q_pos=None, kv_pos=None, q_seg=None, kv_seg=None, sinks=None,
                   pad_segment_id=-1, ops=None):
    """Device ``device_idx``'s forward as a generator (see the module notes).

    q (B, Lq, Hq, D), k / v (B, Lkv, Hkv, D): this device's shards (bf16 or
    fp32, contiguous).  Yields its chunk dict after each step but the last and is
    sent the left neighbour's; returns (out in q's dtype, lse fp32)."""
    ops = ops or KernelOps()
    B, Lq, Hq, D = q.shape
    if causal and q_pos is None:
        q_pos = _global_positions(B, Lq, device_idx, q.device)
        kv_pos = _global_positions(B, k.shape[1], device_idx, q.device)
    cfg = dict(scale=scale, causal=causal, soft_cap=soft_cap, is_mqa=is_mqa,
               pad_segment_id=pad_segment_id, q_pos=q_pos, q_seg=q_seg, sinks=sinks)
    out_run = torch.empty((B, Lq, Hq, D), dtype=torch.float32, device=q.device)
    lse_run = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    out = torch.empty_like(q)
    chunk = dict(k=k, v=v, kv_pos=kv_pos, kv_seg=kv_seg)
    for t in range(n_devices):
        flags = RA_STEP_FIRST if t == 0 else 0
        if t == 0 and sinks is not None:
            flags |= RA_STEP_SINKS
        last = t == n_devices - 1
        ops.fwd_step(q, chunk, cfg, flags, out_run, lse_run, out if last else None)
        if not last:
            chunk = yield chunk
    return out, lse_run


def backward_device(q, k, v, out, lse, dout, *, device_idx, n_devices, scale, causal=False,
                    soft_cap=0.0, is_mqa=False, q_pos=None, kv_pos=None, q_seg=None,
                    kv_seg=None, sinks=None, pad_segment_id=-1, ops=None):
    """Device ``device_idx``'s backward as a generator: yields its chunk (with
    the travelling dk / dv accumulators) after every step -- the last shift
    brings each chunk home -- and returns (dq, dk, dv, dsinks_local) with the
    grads in the input dtypes and dsinks_local this device's fp32 part of the
    sum (None without sinks)."""
    ops = ops or KernelOps()
    B, Lq, Hq, D = q.shape
    if causal and q_pos is None:
        q_pos = _global_positions(B, Lq, device_idx, q.device)
        kv_pos = _global_positions(B, k.shape[1], device_idx, q.device)
    cfg = dict(scale=scale, causal=causal, soft_cap=soft_cap, is_mqa=is_mqa,
               pad_segment_id=pad_segment_id, q_pos=q_pos, q_seg=q_seg, sinks=sinks)
    chunk = dict(k=k, v=v, kv_pos=kv_pos, kv_seg=kv_seg,
                 dk=torch.zeros(k.shape, dtype=torch.float32, device=q.device),
                 dv=torch.zeros(v.shape, dtype=torch.float32, device=q.device))
    # Delta, -lse * log2 e and this device's dsinks, once: they depend only on
    # the local rows
    ws, dsinks = ops.bwd_prep(q, chunk, cfg, out, lse, dout)
    dq_acc = torch.zeros(q.shape, dtype=torch.float32, device=q.device)
    for _ in range(n_devices):
        ops.bwd_step(q, chunk, cfg, dout, ws, dq_acc)
        chunk = yield chunk
    return ops.cast(dq_acc, q), ops.cast(chunk["dk"], k), ops.cast(chunk["dv"], v), dsinks


def _advance(gen, value, first):
    """One resumption of a device generator: (yielded chunk, None) or (None, result)."""
    try:
        return (next(gen) if first else gen.send(value)), None
    except StopIteration as stop:
        return None, stop.value


def run_local(gens):
    """Drive N device generators on one GPU in lockstep: after every step the
    chunk of device d - 1 becomes device d's (a rotation, no copy)."""
    n = len(gens)
    state = [_advance(g, None, True) for g in gens]
    while state[0][1] is None and state[0][0] is not None:
        chunks = [s[0] for s in state]
        state = [_advance(g, chunks[(d - 1) % n], False) for d, g in enumerate(gens)]
    return [s[1] for s in state]


class DistComm:
    """Point-to-point shift to the next rank of a torch.distributed group.

    Over NCCL the chunk's device tensors are sent as they are; over gloo they
    are staged through host memory.  Tensors arrive in new local buffers."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.size = dist.get_world_size(group)
        self.host = dist.get_backend(group) == "gloo"

    def shift(self, chunk):
        dist = self.dist
        nxt, prv = (self.rank + 1) % self.size, (self.rank - 1) % self.size
        ops, recv = [], {}
        for key in _CHUNK_KEYS:
            t = chunk.get(key)
            if t is None:
                continue
            src = t.cpu() if self.host else t
            buf = torch.empty_like(src)
            ops.append(dist.P2POp(dist.isend, src.contiguous(), nxt, self.group))
            ops.append(dist.P2POp(dist.irecv, buf, prv, self.group))
            recv[key] = (buf, t.device)
        for req in dist.batch_isend_irecv(ops):
            req.wait()
        out = dict(chunk)
        for key, (buf, dev) in recv.items():
            out[key] = buf.to(dev) if self.host else buf
        return out

    def all_reduce_sum(self, t):
        if t is None:
            return None
        x = t.cpu() if self.host else t
        self.dist.all_reduce(x, op=self.dist.ReduceOp.SUM, group=self.group)
        return x.to(t.device) if self.host else x


def run_dist(gen, comm):
    """Drive this rank's device generator; every yield is a shift."""
    chunk, result = _advance(gen, None, True)
    while result is None and chunk is not None:
        chunk, result = _advance(gen, comm.shift(chunk), False)
    return result


# ------------------------------------------------------------------ helpers
def _shards(x, n):
    """Contiguous per-device shards of axis 1 of x (B, L, ...), or None."""
    if x is None:
        return [None] * n
    s = x.shape[1] // n
    return [x[:, d * s:(d + 1) * s].contiguous() for d in range(n)]


def ring_forward_local(q, k, v, n_devices, **kw):
    """The ring over ``n_devices`` virtual devices on this GPU.  q, k, v and
    the optional positions / segment ids cover the whole (possibly permuted)
    sequence; device d holds rows [d L / N, (d + 1) L / N).  Returns the
    per-device lists (out, lse)."""
    qs, ks, vs = _shards(q, n_devices), _shards(k, n_devices), _shards(v, n_devices)
    pos = {key: _shards(kw.pop(key, None), n_devices) for key in ("q_pos", "kv_pos", "q_seg", "kv_seg")}
    gens = [forward_device(qs[d], ks[d], vs[d], device_idx=d, n_devices=n_devices,
                           **{key: pos[key][d] for key in pos}, **kw)
            for d in range(n_devices)]
    res = run_local(gens)
    return [r[0] for r in res], [r[1] for r in res]


def ring_backward_local(q, k, v, outs, lses, dout, n_devices, **kw):
    """Backward of ``ring_forward_local``: per-device lists (dq, dk, dv) and
    dsinks summed over the virtual devices (the pages' psum)."""
    qs, ks, vs = _shards(q, n_devices), _shards(k, n_devices), _shards(v, n_devices)
    dos = _shards(dout, n_devices)
    pos = {key: _shards(kw.pop(key, None), n_devices) for key in ("q_pos", "kv_pos", "q_seg", "kv_seg")}
    gens = [backward_device(qs[d], ks[d], vs[d], outs[d], lses[d], dos[d], device_idx=d,
                            n_devices=n_devices, **{key: pos[key][d] for key in pos}, **kw)
            for d in range(n_devices)]
    res = run_local(gens)
    dsinks = res[0][3]
    ops = kw.get("ops") or KernelOps()
    for r in res[1:]:
        if dsinks is not None:
            ops.add(dsinks, r[3])
    return [r[0] for r in res], [r[1] for r in res], [r[2] for r in res], dsinks
