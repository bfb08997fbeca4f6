"""Block-sparse masked flash attention with the ring (out, lse) merge, for GB300.

A thin ctypes binding over ``libra_gb300.so`` (the C ABI of ``include/ra.h``).
Every function named ``ra_*`` here has the same name, arguments and meaning
as its C counterpart and only marshals arguments: torch tensors become device
pointers, ``stream=None`` becomes the current torch CUDA stream.  All work
runs in the library's CUDA kernels; there is no fallback: if the library has
not been built, every call raises.

The helpers at the bottom (``make_params``, ``build_mask``, ``forward``,
``backward``, ``permute``, ``unpermute``) allocate outputs with torch and
call the same entry points.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "RA_OK", "RA_ERR_INVALID_ARG", "RA_ERR_UNSUPPORTED", "RA_ERR_CUDA", "RA_ERR_WORKSPACE",
    "RA_ERR_TIMEOUT", "RA_BF16", "RA_FP32", "RA_TILE", "RaError", "RaAttnParams", "RaBlockMask",
    "lib", "ra_last_error", "ra_version", "ra_set_wait_timeout_ns", "ra_block_mask_bytes",
    "ra_build_block_mask", "ra_attn_fwd_workspace_size", "ra_attn_fwd", "ra_merge_out_lse",
    "ra_attn_bwd_workspace_size", "ra_attn_bwd", "ra_attn_bwd_prep", "ra_attn_bwd_dkdv",
    "ra_attn_bwd_dq", "ra_attn_bwd_noalloc", "ra_attn_bwd_noalloc_max_workspace",
    "ra_permute_tokens", "ra_unpermute_tokens", "RA_STEP_SINKS", "RA_STEP_FIRST",
    "ra_attn_fwd_step", "ra_attn_bwd_step", "ra_cast_from_f32", "ra_add_f32",
    "ra_get_device_status", "ra_launch_count", "ra_selftest_wait_timeout", "make_params", "build_mask", "forward", "backward", "permute",
    "unpermute",
]

RA_OK = 0
RA_ERR_INVALID_ARG = -1
RA_ERR_UNSUPPORTED = -2
RA_ERR_CUDA = -3
RA_ERR_WORKSPACE = -4
RA_ERR_TIMEOUT = -5
RA_BF16 = 0
RA_FP32 = 1
RA_TILE = 128
RA_STEP_SINKS = 1
RA_STEP_FIRST = 2

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libra_gb300.so")


class RaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class RaAttnParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Lq", ctypes.c_int), ("Lkv", ctypes.c_int),
        ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("dtype", ctypes.c_int), ("scale", ctypes.c_float), ("soft_cap", ctypes.c_float),
        ("causal", ctypes.c_int), ("is_mqa", ctypes.c_int), ("n_virtual_shards", ctypes.c_int),
        ("pad_segment_id", ctypes.c_int),
        ("q_pos", ctypes.c_void_p), ("kv_pos", ctypes.c_void_p),
        ("q_seg", ctypes.c_void_p), ("kv_seg", ctypes.c_void_p),
        ("sinks", ctypes.c_void_p), ("local_mask", ctypes.c_void_p),
        ("block_q_dkv", ctypes.c_int),
    ]


class RaBlockMask(ctypes.Structure):
    _fields_ = [
        ("tile_class", ctypes.c_void_p), ("fwd_cnt", ctypes.c_void_p),
        ("fwd_idx", ctypes.c_void_p), ("bwd_cnt", ctypes.c_void_p),
        ("bwd_idx", ctypes.c_void_p), ("fwd_order", ctypes.c_void_p),
        ("bwd_order", ctypes.c_void_p), ("fwd_shard", ctypes.c_void_p),
        ("part_fwd", ctypes.c_void_p), ("part_bwd", ctypes.c_void_p),
        ("part_rows", ctypes.c_void_p), ("part_cols", ctypes.c_void_p),
        ("n_part", ctypes.c_void_p), ("dkv_class", ctypes.c_void_p), ("dkv_cnt", ctypes.c_void_p),
        ("dkv_idx", ctypes.c_void_p), ("dkv_slot", ctypes.c_void_p), ("dkv_order", ctypes.c_void_p),
        ("B", ctypes.c_int), ("nq", ctypes.c_int),
        ("nk", ctypes.c_int), ("n_shards", ctypes.c_int), ("part_cap", ctypes.c_int),
        ("key", ctypes.c_uint64),
    ]


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.POINTER(RaAttnParams)
            M = ctypes.POINTER(RaBlockMask)
            vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.ra_last_error.restype = ctypes.c_char_p
            L.ra_version.restype = ctypes.c_char_p
            L.ra_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
            L.ra_set_wait_timeout_ns.restype = None
            L.ra_block_mask_bytes.argtypes = [P]
            L.ra_block_mask_bytes.restype = sz
            L.ra_build_block_mask.argtypes = [P, vp, sz, M, vp]
            L.ra_attn_fwd_workspace_size.argtypes = [P]
            L.ra_attn_fwd_workspace_size.restype = sz
            L.ra_attn_fwd.argtypes = [P, vp, vp, vp, M, vp, vp, vp, sz, vp]
            L.ra_merge_out_lse.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, vp]
            L.ra_attn_bwd_workspace_size.argtypes = [P]
            L.ra_attn_bwd_workspace_size.restype = sz
            L.ra_attn_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, M, vp, vp, vp, vp, vp, sz, vp]
            L.ra_attn_bwd_prep.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
            L.ra_attn_bwd_dkdv.argtypes = [P, vp, vp, vp, vp, M, vp, vp, vp, sz, vp]
            L.ra_attn_bwd_dq.argtypes = [P, vp, vp, vp, vp, M, vp, vp, sz, vp]
            L.ra_permute_tokens.argtypes = [vp, vp, ci, ci, sz, ci, vp]
            L.ra_unpermute_tokens.argtypes = [vp, vp, ci, ci, sz, ci, vp]
            L.ra_attn_bwd_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, M, vp, vp, vp, vp, vp]
            L.ra_attn_fwd_step.argtypes = [P, vp, vp, vp, M, ci, vp, vp, vp, vp]
            L.ra_attn_bwd_step.argtypes = [P, vp, vp, vp, vp, M, vp, vp, vp, vp, sz, vp]
            L.ra_cast_from_f32.argtypes = [vp, vp, sz, ci, vp]
            L.ra_add_f32.argtypes = [vp, vp, sz, vp]
            L.ra_attn_bwd_noalloc_max_workspace.restype = sz
            L.ra_get_device_status.argtypes = [vp]
            L.ra_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp, vp]
            L.ra_launch_count.restype = ctypes.c_uint64
            _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int):
    if rc != RA_OK:
        raise RaError(rc, ra_last_error())


# ------------------------------------------------------------- C entry points
def ra_last_error() -> str:
    return lib().ra_last_error().decode()


def ra_version() -> str:
    return lib().ra_version().decode()


def ra_set_wait_timeout_ns(ns: int) -> None:
    lib().ra_set_wait_timeout_ns(int(ns))


def ra_block_mask_bytes(params: RaAttnParams) -> int:
    n = lib().ra_block_mask_bytes(ctypes.byref(params))
    if n == 0:
        raise RaError(RA_ERR_INVALID_ARG, ra_last_error())
    return int(n)


def ra_build_block_mask(params, buf, mask: RaBlockMask | None = None, stream=None) -> RaBlockMask:
    m = mask if mask is not None else RaBlockMask()
    nbytes = buf.numel() * buf.element_size()
    _check(lib().ra_build_block_mask(ctypes.byref(params), _ptr(buf), nbytes, ctypes.byref(m),
                                     _stream(stream)))
    m._buf = buf  # keep the device buffer alive with the struct
    return m


def ra_attn_fwd_workspace_size(params) -> int:
    return int(lib().ra_attn_fwd_workspace_size(ctypes.byref(params)))


def ra_attn_fwd(params, q, k, v, mask, out, lse, ws=None, stream=None) -> None:
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().ra_attn_fwd(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), ctypes.byref(mask),
                             _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)))


def ra_merge_out_lse(out, lse, block_out, block_lse, B, L, H, D, stream=None) -> None:
    _check(lib().ra_merge_out_lse(_ptr(out), _ptr(lse), _ptr(block_out), _ptr(block_lse),
                                  B, L, H, D, _stream(stream)))


def ra_attn_bwd_workspace_size(params) -> int:
    return int(lib().ra_attn_bwd_workspace_size(ctypes.byref(params)))


def ra_attn_bwd(params, q, k, v, out, lse, dout, mask, dq, dk, dv, dsinks, ws, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().ra_attn_bwd(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                             _ptr(lse), _ptr(dout), ctypes.byref(mask), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(dsinks), _ptr(ws), ws_bytes, _stream(stream)))


def ra_attn_bwd_noalloc(params, q, k, v, out, lse, dout, mask, dq, dk, dv, dsinks, stream=None):
    """ra_attn_bwd with the library's built-in scratch instead of a workspace."""
    _check(lib().ra_attn_bwd_noalloc(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                     _ptr(lse), _ptr(dout), ctypes.byref(mask), _ptr(dq), _ptr(dk),
                                     _ptr(dv), _ptr(dsinks), _stream(stream)))


def ra_attn_bwd_noalloc_max_workspace() -> int:
    return int(lib().ra_attn_bwd_noalloc_max_workspace())


def _wsb(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def ra_attn_bwd_prep(params, out, lse, dout, dsinks, ws, stream=None):
    _check(lib().ra_attn_bwd_prep(ctypes.byref(params), _ptr(out), _ptr(lse), _ptr(dout),
                                  _ptr(dsinks), _ptr(ws), _wsb(ws), _stream(stream)))


def ra_attn_bwd_dkdv(params, q, k, v, dout, mask, dk, dv, ws, stream=None):
    _check(lib().ra_attn_bwd_dkdv(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                  ctypes.byref(mask), _ptr(dk), _ptr(dv), _ptr(ws), _wsb(ws),
                                  _stream(stream)))


def ra_attn_bwd_dq(params, q, k, v, dout, mask, dq, ws, stream=None):
    _check(lib().ra_attn_bwd_dq(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                ctypes.byref(mask), _ptr(dq), _ptr(ws), _wsb(ws), _stream(stream)))


def ra_attn_fwd_step(params, q, k, v, mask, flags, out_run, lse_run, out=None, stream=None):
    """One ring step of the forward: merge the chunk (k, v) into (out_run, lse_run)."""
    _check(lib().ra_attn_fwd_step(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v),
                                  ctypes.byref(mask), int(flags), _ptr(out_run), _ptr(lse_run),
                                  _ptr(out), _stream(stream)))


def ra_attn_bwd_step(params, q, k, v, dout, mask, dq_acc, dk_acc, dv_acc, ws, stream=None):
    """One ring step of the backward: += the pair's gradients into fp32 accumulators."""
    _check(lib().ra_attn_bwd_step(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                  ctypes.byref(mask), _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc),
                                  _ptr(ws), _wsb(ws), _stream(stream)))


def ra_cast_from_f32(inp, out, n, dtype, stream=None) -> None:
    _check(lib().ra_cast_from_f32(_ptr(inp), _ptr(out), int(n), int(dtype), _stream(stream)))


def ra_add_f32(acc, x, n, stream=None) -> None:
    _check(lib().ra_add_f32(_ptr(acc), _ptr(x), int(n), _stream(stream)))


def ra_permute_tokens(inp, out, B, L, row_bytes, n_shards, stream=None) -> None:
    _check(lib().ra_permute_tokens(_ptr(inp), _ptr(out), B, L, row_bytes, n_shards,
                                   _stream(stream)))


def ra_unpermute_tokens(inp, out, B, L, row_bytes, n_shards, stream=None) -> None:
    _check(lib().ra_unpermute_tokens(_ptr(inp), _ptr(out), B, L, row_bytes, n_shards,
                                     _stream(stream)))


def ra_launch_count() -> int:
    return int(lib().ra_launch_count())


def ra_get_device_status(stream=None) -> int:
    return int(lib().ra_get_device_status(_stream(stream)))


def ra_selftest_wait_timeout(timeout_ns, gave_up, stream=None) -> None:
    """One in-kernel wait that can never complete gives up after timeout_ns;
    ``gave_up`` is a device int32 tensor of one element."""
    _check(lib().ra_selftest_wait_timeout(int(timeout_ns), _ptr(gave_up), _stream(stream)))


# ------------------------------------------------------------- helpers
_DT = {torch.bfloat16: RA_BF16, torch.float32: RA_FP32}


def make_params(q, k, *, scale, causal=False, soft_cap=0.0, n_virtual_shards=1, is_mqa=False,
                pad_segment_id=-1, q_pos=None, kv_pos=None, q_seg=None, kv_seg=None,
                sinks=None, local_mask=None, block_q_dkv=0) -> RaAttnParams:
    """Params for q (B,Lq,Hq,D) and k (B,Lkv,Hkv,D) tensors; keeps the
    position / segment / sink / local-mask tensors referenced by the struct
    alive.  ``local_mask``: (Lq/N, Lkv/N) uint8 device tensor (non-causal only).
    ``block_q_dkv``: 0 / 128, or 64 for the dK/dV stage's own 64-row grid."""
    B, Lq, Hq, D = q.shape
    Lkv, Hkv = k.shape[1], k.shape[2]
    if q.dtype not in _DT:
        raise TypeError(f"unsupported dtype {q.dtype}")
    p = RaAttnParams(B, Lq, Lkv, Hq, Hkv, D, _DT[q.dtype], float(scale),
                     float(soft_cap or 0.0), int(bool(causal)), int(bool(is_mqa)),
                     int(n_virtual_shards), int(pad_segment_id), _ptr(q_pos), _ptr(kv_pos),
                     _ptr(q_seg), _ptr(kv_seg), _ptr(sinks), _ptr(local_mask), int(block_q_dkv))
    p._keep = (q_pos, kv_pos, q_seg, kv_seg, sinks, local_mask)
    return p


def build_mask(params, device=None, stream=None) -> RaBlockMask:
    n = ra_block_mask_bytes(params)
    buf = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    return ra_build_block_mask(params, buf, stream=stream)


def forward(params, q, k, v, mask, stream=None, workspace=True):
    """Forward; with ``workspace`` the optional fp32 workspace that lets the
    library run two query heads per CTA is allocated (when it applies)."""
    B, Lq, Hq, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    n = ra_attn_fwd_workspace_size(params) if workspace else 0
    ws = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    ra_attn_fwd(params, q, k, v, mask, out, lse, ws=ws, stream=stream)
    return out, lse


def backward(params, q, k, v, out, lse, dout, mask, stream=None):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dsinks = (torch.empty(q.shape[2], dtype=torch.float32, device=q.device)
              if params.sinks else None)
    ws = torch.empty(ra_attn_bwd_workspace_size(params), dtype=torch.uint8, device=q.device)
    ra_attn_bwd(params, q, k, v, out, lse, dout, mask, dq, dk, dv, dsinks, ws, stream=stream)
    return dq, dk, dv, dsinks


def _rows(x):
    B, L = x.shape[0], x.shape[1]
    return B, L, x[0, 0].numel() * x.element_size()


def permute(x, n_shards, stream=None):
    """Zigzag permutation of axis 1 of a contiguous (B, L, ...) tensor."""
    x = x.contiguous()
    out = torch.empty_like(x)
    B, L, rb = _rows(x)
    ra_permute_tokens(x, out, B, L, rb, n_shards, stream=stream)
    return out


def unpermute(x, n_shards, stream=None):
    x = x.contiguous()
    out = torch.empty_like(x)
    B, L, rb = _rows(x)
    ra_unpermute_tokens(x, out, B, L, rb, n_shards, stream=stream)
    return out
