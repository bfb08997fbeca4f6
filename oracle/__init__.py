"""fp64 CPU oracle for block-sparse masked attention with the ring (out, lse) merge.

TEST INFRASTRUCTURE ONLY.  The product library never imports, links or calls
anything here; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` do.  The arithmetic lives in ``ra_oracle.c`` (plain C,
fp64, OpenMP over rows); this module compiles it with gcc and marshals numpy
arrays.  Every function follows a section of the pages:

* ``attn_fwd``        -- the plain definition of masked attention with segment
  ids, positions, causal mask, sinks and soft cap (Kvax "Flash Attention for
  JAX": ``flash_attention`` arguments; ejKernel ``_ring_splash`` module:
  ``_ring_attention_forward`` for sinks and ``logits_soft_cap``).
* ``attn_fwd_ring``   -- the same, computed literally as the ring loop of
  ``_ring_attention_forward`` over N virtual devices, each chunk merged by
  ``_update_out_and_lse``.
* ``merge``           -- ``_update_out_and_lse`` elementwise.
* ``attn_bwd``        -- the exact gradient (summed per chunk as in
  ``_ring_attention_backward``; dsinks summed over all rows).
* ``block_mask``      -- tile classification on the 128 x 128 grid and the
  per-row / per-column tile lists (``MaskInfo`` in ``make_ring_attention``;
  Kvax ``create_attention_mask``).
* ``permute`` / ``unpermute`` -- the zigzag token permutation (Kvax context
  parallelism: permute tokens, unpermute outputs).

Parity status of each function (what pins it) is listed in the tests:
``tests/test_oracle_pins.py``.  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ra_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libra_oracle.so")
_lock = threading.Lock()
_lib = None

TILE = 128


class _Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Lq", ctypes.c_int), ("Lkv", ctypes.c_int),
        ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("scale", ctypes.c_double), ("soft_cap", ctypes.c_double),
        ("causal", ctypes.c_int), ("pad_segment_id", ctypes.c_int),
        ("q_pos", ctypes.c_void_p), ("kv_pos", ctypes.c_void_p),
        ("q_seg", ctypes.c_void_p), ("kv_seg", ctypes.c_void_p),
        ("sinks", ctypes.c_void_p), ("local_mask", ctypes.c_void_p),
        ("lq_s", ctypes.c_int), ("lk_s", ctypes.c_int),
    ]


def build(force: bool = False) -> str:
    """Compile ra_oracle.c into oracle/_lib/libra_oracle.so (gcc, -fopenmp)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Params)
            vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.ora_attn_fwd.argtypes = [P, vp, vp, vp, vp, vp, ci, ci, ci, ci]
            lib.ora_attn_fwd_ring.argtypes = [P, ci, vp, vp, vp, vp, vp, ci, ci]
            lib.ora_attn_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci,
                                        ci, ci]
            lib.ora_merge.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci]
            lib.ora_merge.restype = None
            lib.ora_block_mask.argtypes = [P, vp, vp, vp, vp, vp, vp, vp]
            lib.ora_block_mask_sized.argtypes = [P, ci, ci, vp, vp, vp, vp, vp, vp, vp]
            lib.ora_permute.argtypes = [vp, vp, ci, ci, sz, ci, ci]
            lib.ora_zigzag_source.argtypes = [ci, ci, ci]
            lib.ora_ring_source.argtypes = [ci, ci, ci]
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle may use."""
    return int(_load().ora_num_threads())


def last_threads() -> int:
    """Threads that ran work in the last attn_fwd / attn_bwd call."""
    return int(_load().ora_last_threads())


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _local(mask, Lq, Lkv):
    """A local (per-device) 2-D mask as contiguous uint8, with its shape (R-local)."""
    if mask is None:
        return None, 1, 1
    m = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
    lq_s, lk_s = m.shape
    if Lq % lq_s or Lkv % lk_s:
        raise ValueError("the local mask's shape must divide (Lq, Lkv)")
    return m, int(lq_s), int(lk_s)


class _Call:
    """Holds the numpy buffers referenced by one params struct alive."""

    def __init__(self, q, k, v, *, scale, soft_cap=None, causal=False, q_pos=None,
                 kv_pos=None, q_seg=None, kv_seg=None, sinks=None, pad_segment_id=-1,
                 local_mask=None):
        self.q, self.k, self.v = _f64(q), _f64(k), _f64(v)
        B, Lq, Hq, D = self.q.shape
        _, Lkv, Hkv, _ = self.k.shape
        self.q_pos, self.kv_pos = _i32(q_pos), _i32(kv_pos)
        self.q_seg, self.kv_seg = _i32(q_seg), _i32(kv_seg)
        self.sinks = None if sinks is None else _f64(sinks)
        self.local_mask, lq_s, lk_s = _local(local_mask, Lq, Lkv)
        self.p = _Params(B, Lq, Lkv, Hq, Hkv, D, float(scale),
                         float(soft_cap) if soft_cap else 0.0, int(bool(causal)),
                         int(pad_segment_id), _ptr(self.q_pos), _ptr(self.kv_pos),
                         _ptr(self.q_seg), _ptr(self.kv_seg), _ptr(self.sinks),
                         _ptr(self.local_mask), lq_s, lk_s)
        self.shape = (B, Lq, Lkv, Hq, Hkv, D)


def attn_fwd(q, k, v, *, scale, heads=None, rows=None, **kw):
    """Plain definition.  q [B,Lq,Hq,D], k/v [B,Lkv,Hkv,D] -> (out [B,Lq,Hq,D], lse [B,Hq,Lq]).

    ``heads=(lo, hi)`` / ``rows=(lo, hi)`` restrict the computation to those
    query heads / query rows; the other outputs are left at zero / -inf.
    """
    c = _Call(q, k, v, scale=scale, **kw)
    B, Lq, Lkv, Hq, Hkv, D = c.shape
    out = np.zeros((B, Lq, Hq, D))
    lse = np.full((B, Hq, Lq), -np.inf)
    lo, hi = heads if heads else (0, 0)
    rlo, rhi = rows if rows else (0, 0)
    rc = _load().ora_attn_fwd(ctypes.byref(c.p), _ptr(c.q), _ptr(c.k), _ptr(c.v),
                              _ptr(out), _ptr(lse), lo, hi, rlo, rhi)
    if rc:
        raise ValueError(f"ora_attn_fwd failed ({rc})")
    return out, lse


def attn_fwd_ring(q, k, v, *, scale, n_shards, heads=None, **kw):
    """Ring mode over ``n_shards`` virtual devices with the pages' merge."""
    c = _Call(q, k, v, scale=scale, **kw)
    B, Lq, Lkv, Hq, Hkv, D = c.shape
    out = np.zeros((B, Lq, Hq, D))
    lse = np.full((B, Hq, Lq), -np.inf)
    lo, hi = heads if heads else (0, 0)
    rc = _load().ora_attn_fwd_ring(ctypes.byref(c.p), int(n_shards), _ptr(c.q), _ptr(c.k),
                                   _ptr(c.v), _ptr(out), _ptr(lse), lo, hi)
    if rc:
        raise ValueError(f"ora_attn_fwd_ring failed ({rc})")
    return out, lse


def attn_bwd(q, k, v, dout, *, scale, heads=None, rows=None, keys=None, **kw):
    """Exact gradient -> (dq, dk, dv, dsinks or None, out, lse).

    ``heads`` / ``rows`` / ``keys`` restrict the sums to the contributions of
    pairs with a query head, query row and key row in those ranges (dq of
    other rows and dk / dv of other keys stay 0; dsinks sums the rows of the
    row range)."""
    c = _Call(q, k, v, scale=scale, **kw)
    B, Lq, Lkv, Hq, Hkv, D = c.shape
    do = _f64(dout)
    dq = np.zeros((B, Lq, Hq, D))
    dk = np.zeros((B, Lkv, Hkv, D))
    dv = np.zeros((B, Lkv, Hkv, D))
    ds = np.zeros(Hq) if c.sinks is not None else None
    out = np.zeros((B, Lq, Hq, D))
    lse = np.full((B, Hq, Lq), -np.inf)
    lo, hi = heads if heads else (0, 0)
    rlo, rhi = rows if rows else (0, 0)
    klo, khi = keys if keys else (0, 0)
    rc = _load().ora_attn_bwd(ctypes.byref(c.p), _ptr(c.q), _ptr(c.k), _ptr(c.v), _ptr(do),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ds), _ptr(out), _ptr(lse),
                              lo, hi, rlo, rhi, klo, khi)
    if rc:
        raise ValueError(f"ora_attn_bwd failed ({rc})")
    return dq, dk, dv, ds, out, lse


def merge(out, lse, block_out, block_lse):
    """``_update_out_and_lse`` on out [B,L,H,D], lse [B,H,L]; returns new arrays."""
    o = _f64(out).copy()
    l = _f64(lse).copy()
    bo, bl = _f64(block_out), _f64(block_lse)
    B, L, H, D = o.shape
    _load().ora_merge(_ptr(o), _ptr(l), _ptr(bo), _ptr(bl), B, L, H, D)
    return o, l


def block_mask(B, Lq, Lkv, *, causal, q_pos=None, kv_pos=None, q_seg=None, kv_seg=None,
               pad_segment_id=-1, local_mask=None, block_q=TILE, block_kv=TILE):
    """Tile classes (0 empty, 1 partial, 2 full) and tile lists, see ra_oracle.c,
    on a grid of block_q query rows x block_kv key rows (128 x 128 by default)."""
    q_pos, kv_pos, q_seg, kv_seg = map(_i32, (q_pos, kv_pos, q_seg, kv_seg))
    lm, lq_s, lk_s = _local(local_mask, Lq, Lkv)
    p = _Params(B, Lq, Lkv, 1, 1, 1, 1.0, 0.0, int(bool(causal)), int(pad_segment_id),
                _ptr(q_pos), _ptr(kv_pos), _ptr(q_seg), _ptr(kv_seg), None, _ptr(lm), lq_s, lk_s)
    nq, nk = Lq // block_q, Lkv // block_kv
    cls = np.zeros((B, nq, nk), np.uint8)
    fcnt = np.zeros(B * nq, np.int32)
    fidx = np.zeros((B * nq, nk), np.int32)
    bcnt = np.zeros(B * nk, np.int32)
    bidx = np.zeros((B * nk, nq), np.int32)
    ford = np.zeros(B * nq, np.int32)
    bord = np.zeros(B * nk, np.int32)
    rc = _load().ora_block_mask_sized(ctypes.byref(p), int(block_q), int(block_kv), _ptr(cls),
                                      _ptr(fcnt), _ptr(fidx), _ptr(bcnt), _ptr(bidx), _ptr(ford),
                                      _ptr(bord))
    if rc:
        raise ValueError(f"ora_block_mask failed ({rc})")
    return dict(tile_class=cls, fwd_cnt=fcnt, fwd_idx=fidx, bwd_cnt=bcnt, bwd_idx=bidx,
                fwd_order=ford, bwd_order=bord)


def _perm(x, n, inverse):
    a = np.ascontiguousarray(x)
    B, L = a.shape[0], a.shape[1]
    row_bytes = a.itemsize * int(np.prod(a.shape[2:], dtype=np.int64))
    out = np.empty_like(a)
    rc = _load().ora_permute(_ptr(a), _ptr(out), B, L, row_bytes, int(n), int(inverse))
    if rc:
        raise ValueError(f"ora_permute failed ({rc})")
    return out


def permute(x, n_shards):
    """Zigzag permutation of axis 1 of x [B, L, ...] (any dtype, bitwise)."""
    return _perm(x, n_shards, 0)


def unpermute(x, n_shards):
    """Inverse of ``permute``."""
    return _perm(x, n_shards, 1)


def ring_source(device, step, n_shards):
    """Key/value shard held by virtual ``device`` at ring ``step``."""
    return int(_load().ora_ring_source(int(device), int(step), int(n_shards)))


def zigzag_source(L, n_shards, p):
    """Source index (original order) of permuted row p."""
    return int(_load().ora_zigzag_source(int(L), int(n_shards), int(p)))
