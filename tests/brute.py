"""Brute-force masked attention in vectorised numpy fp64, for tiny inputs.

An independent restatement used only to pin the C oracle: it materialises the
whole (B, H, Lq, Lkv) logit tensor, sets invisible pairs to -inf, appends the
sink as one more logit column, and takes scipy's logsumexp.  Shares no code
with ``oracle/``.
"""
import numpy as np
from scipy.special import logsumexp


def visibility(B, Lq, Lkv, *, causal, q_pos=None, kv_pos=None, q_seg=None, kv_seg=None, pad=-1,
               local_mask=None):
    qp = np.broadcast_to(np.arange(Lq), (B, Lq)) if q_pos is None else np.asarray(q_pos)
    kp = np.broadcast_to(np.arange(Lkv), (B, Lkv)) if kv_pos is None else np.asarray(kv_pos)
    qs = np.zeros((B, Lq), np.int64) if q_seg is None else np.asarray(q_seg, np.int64)
    ks = np.zeros((B, Lkv), np.int64) if kv_seg is None else np.asarray(kv_seg, np.int64)
    vis = (qs[:, :, None] == ks[:, None, :]) & (qs[:, :, None] != pad)
    if causal:
        vis &= qp[:, :, None] >= kp[:, None, :]
    if local_mask is not None:
        # the per-device mask repeated over every (query shard, kv shard) block
        lm = np.asarray(local_mask) != 0
        vis &= np.tile(lm, (Lq // lm.shape[0], Lkv // lm.shape[1]))[None]
    return vis  # [B, Lq, Lkv]


def attention(q, k, v, *, scale, soft_cap=None, causal=False, q_pos=None, kv_pos=None,
              q_seg=None, kv_seg=None, sinks=None, pad=-1, local_mask=None):
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    B, Lq, Hq, D = q.shape
    Lkv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    kk = np.repeat(k, G, axis=2)
    vv = np.repeat(v, G, axis=2)
    s = scale * np.einsum("bihd,bjhd->bhij", q, kk)
    if soft_cap:
        s = soft_cap * np.tanh(s / soft_cap)
    vis = visibility(B, Lq, Lkv, causal=causal, q_pos=q_pos, kv_pos=kv_pos, q_seg=q_seg,
                     kv_seg=kv_seg, pad=pad, local_mask=local_mask)
    s = np.where(vis[:, None], s, -np.inf)
    if sinks is not None:
        col = np.broadcast_to(np.asarray(sinks, np.float64)[None, :, None, None], (B, Hq, Lq, 1))
        s_all = np.concatenate([s, col], axis=-1)
    else:
        s_all = s
    with np.errstate(invalid="ignore", divide="ignore"):
        lse = logsumexp(s_all, axis=-1)                 # [B, H, Lq]
        p = np.exp(s - lse[..., None])
    p = np.where(np.isfinite(lse)[..., None], p, 0.0)
    out = np.einsum("bhij,bjhd->bihd", p, vv)
    return out, lse


def chunk_grads(q, k, v, dout, lse, delta, *, scale, soft_cap=None, causal=False, q_pos=None,
                kv_pos=None, q_seg=None, kv_seg=None, pad=-1):
    """Gradient contributions of one (query rows, key chunk) pair with the
    FINAL lse of the query rows and Delta = <dO, O> (B, H, Lq): returns
    (dq, dk, dv) of this pair, dk / dv summed over the query heads of a kv
    head."""
    q, k, v, dout = (np.asarray(a, np.float64) for a in (q, k, v, dout))
    B, Lq, Hq, D = q.shape
    Lkv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    kk = np.repeat(k, G, axis=2)
    vv = np.repeat(v, G, axis=2)
    raw = scale * np.einsum("bihd,bjhd->bhij", q, kk)
    s = soft_cap * np.tanh(raw / soft_cap) if soft_cap else raw
    vis = visibility(B, Lq, Lkv, causal=causal, q_pos=q_pos, kv_pos=kv_pos, q_seg=q_seg,
                     kv_seg=kv_seg, pad=pad)[:, None]
    lse = np.asarray(lse, np.float64)
    fin = np.isfinite(lse)[..., None]
    with np.errstate(invalid="ignore", over="ignore"):
        p = np.where(vis & fin, np.exp(s - np.where(fin, lse[..., None], 0.0)), 0.0)
    dp = np.einsum("bihd,bjhd->bhij", dout, vv)
    ds = p * (dp - np.asarray(delta, np.float64)[..., None])
    if soft_cap:
        ds = ds * (1.0 - (s / soft_cap) ** 2)
    dq = scale * np.einsum("bhij,bjhd->bihd", ds, kk)
    dk_h = scale * np.einsum("bhij,bihd->bjhd", ds, q)
    dv_h = np.einsum("bhij,bihd->bjhd", p, dout)
    dk = dk_h.reshape(B, Lkv, Hkv, G, D).sum(axis=3)
    dv = dv_h.reshape(B, Lkv, Hkv, G, D).sum(axis=3)
    return dq, dk, dv
