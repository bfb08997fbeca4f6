"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no attention arithmetic: it only draws random tensors and
builds segment ids / positions from random document lengths.  Both the CUDA
path (tests, bench) and the fp64 oracle consume its output; each side then
applies its own permutation, masking and attention.

Recipe (all on a seeded torch CPU generator, fp32 N(0,1) drawn in the order
q, k, v, dO, sinks, document lengths, then cast to the workload dtype):

* ``tiny``      B1 Hq=Hkv=2 L256 D64 fp32, causal, one segment, 2 shards, seed 0.
* ``gqa8k``     B1 Hq32 Hkv8 L8192 D128 bf16, causal, one segment, 4 shards.
* ``packed16k`` B2 Hq=Hkv=16 L16384 D128 bf16; document lengths uniform in
  [128, 4096] (inclusive) fill each row, the last document truncated, segment
  ids 0, 1, 2, ... per row, positions restart at 0 in each document; the last
  L // 20 tokens of each row are padding (segment id -1, position 0); causal
  within a segment; dO drawn; one shard.
* ``mqa32k``    B1 Hq32 Hkv1 (MQA) L32768 D128 bf16, causal, soft cap 50,
  sinks N(0,1) per head, 8 shards, zigzag permutation.
* ``long64k``   B1 Hq8 Hkv2 L65536 D128 bf16, causal, 8 shards, zigzag, dO.
* ``gqa32k``    B1 Hq32 Hkv8 L32768 D128 bf16, causal, 8 shards, zigzag, dO --
  the 32K causal GQA workload the throughput target is quoted on.
* ``local8k``   B1 Hq32 Hkv8 L8192 D128 bf16, non-causal, 4 shards, dO, with
  the per-shard local mask of the non-causal ring: a band |i - j| < 512 in
  local (within-shard) coordinates, applied to every shard pair.

The seed of a named workload is its index in the list above.  Positions are
always produced in the original token order; a permuted run permutes them
together with the tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

PAD_SEGMENT_ID = -1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    dtype: str = "bf16"          # "bf16" | "fp32"
    causal: bool = True
    n_shards: int = 1
    zigzag: bool = False
    soft_cap: float = 0.0
    sinks: bool = False
    is_mqa: bool = False
    packed_docs: bool = False    # segment ids / positions from random documents
    doc_len: tuple = (128, 4096)
    pad_frac_den: int = 20       # last L // pad_frac_den tokens are padding
    backward: bool = False
    local_window: int = 0        # > 0: per-shard local band mask |i - j| < window (non-causal)
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def scaled(self, **kw) -> "Workload":
        """Same structure at other sizes (used for small parity cases)."""
        return replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 1, 256, 2, 2, 64, dtype="fp32", n_shards=2, seed=0),
        Workload("gqa8k", 1, 8192, 32, 8, 128, n_shards=4, seed=1),
        Workload("packed16k", 2, 16384, 16, 16, 128, packed_docs=True, backward=True,
                 n_shards=1, seed=2),
        Workload("mqa32k", 1, 32768, 32, 1, 128, n_shards=8, zigzag=True, soft_cap=50.0,
                 sinks=True, is_mqa=True, seed=3),
        Workload("long64k", 1, 65536, 8, 2, 128, n_shards=8, zigzag=True, backward=True,
                 seed=4),
        Workload("gqa32k", 1, 32768, 32, 8, 128, n_shards=8, zigzag=True, backward=True,
                 seed=5),
        Workload("local8k", 1, 8192, 32, 8, 128, causal=False, n_shards=4, local_window=512,
                 backward=True, seed=6),
    ]
}


def _documents(gen, B, L, lo, hi, pad_tokens):
    """Segment ids and positions from random document lengths (original order)."""
    seg = torch.full((B, L), PAD_SEGMENT_ID, dtype=torch.int32)
    pos = torch.zeros((B, L), dtype=torch.int32)
    body = L - pad_tokens
    for b in range(B):
        start, sid = 0, 0
        while start < body:
            n = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
            n = min(n, body - start)
            seg[b, start:start + n] = sid
            pos[b, start:start + n] = torch.arange(n, dtype=torch.int32)
            start += n
            sid += 1
    return seg, pos


def make_inputs(w: Workload, *, device="cpu", with_dout=None):
    """Inputs of workload ``w`` in original token order.

    Returns a dict: q [B,L,Hq,D], k/v [B,L,Hkv,D], dout [B,L,Hq,D] (if the
    workload has a backward or ``with_dout``), sinks [Hq] fp32 or None,
    q_pos / kv_pos / q_seg / kv_seg [B,L] int32 or None (None = sequential
    positions, one segment).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(w.seed))
    dt = w.torch_dtype
    Hkv = 1 if w.is_mqa else w.Hkv
    q = torch.randn((w.B, w.L, w.Hq, w.D), generator=gen, dtype=torch.float32)
    k = torch.randn((w.B, w.L, Hkv, w.D), generator=gen, dtype=torch.float32)
    v = torch.randn((w.B, w.L, Hkv, w.D), generator=gen, dtype=torch.float32)
    need_do = w.backward if with_dout is None else with_dout
    dout = (torch.randn((w.B, w.L, w.Hq, w.D), generator=gen, dtype=torch.float32)
            if need_do else None)
    sinks = torch.randn((w.Hq,), generator=gen, dtype=torch.float32) if w.sinks else None
    q_pos = kv_pos = q_seg = kv_seg = None
    if w.packed_docs:
        seg, pos = _documents(gen, w.B, w.L, w.doc_len[0], w.doc_len[1],
                              w.L // w.pad_frac_den)
        q_seg, kv_seg, q_pos, kv_pos = seg, seg.clone(), pos, pos.clone()
    elif w.zigzag:
        # explicit positions so that they can travel with the permuted tokens
        ar = torch.arange(w.L, dtype=torch.int32).unsqueeze(0).repeat(w.B, 1)
        q_pos, kv_pos = ar, ar.clone()
    local_mask = None
    if w.local_window:
        # the non-causal ring's per-shard mask: a band in local coordinates
        ls = w.L // w.n_shards
        i = torch.arange(ls).unsqueeze(1)
        j = torch.arange(ls).unsqueeze(0)
        local_mask = ((i - j).abs() < w.local_window).to(torch.uint8)
    out = dict(q=q.to(dt), k=k.to(dt), v=v.to(dt),
               dout=None if dout is None else dout.to(dt), sinks=sinks,
               q_pos=q_pos, kv_pos=kv_pos, q_seg=q_seg, kv_seg=kv_seg, local_mask=local_mask)
    if device != "cpu":
        out = {n: (t.to(device) if isinstance(t, torch.Tensor) else t) for n, t in out.items()}
    return out


def random_structure(gen: torch.Generator, B: int, L: int, *, n_docs_max=4, pad_max=0,
                     shuffle_positions=False):
    """Small random segment / padding / position layouts for parity edge cases.

    Documents of random length fill each row, a random number (< pad_max) of
    trailing tokens are padding, positions restart per document; with
    ``shuffle_positions`` the positions inside each row are a random
    permutation instead (exercising arbitrary position orders).
    """
    seg = torch.full((B, L), PAD_SEGMENT_ID, dtype=torch.int32)
    pos = torch.zeros((B, L), dtype=torch.int32)
    for b in range(B):
        pad = int(torch.randint(0, pad_max + 1, (1,), generator=gen).item()) if pad_max else 0
        body = L - pad
        n_docs = int(torch.randint(1, n_docs_max + 1, (1,), generator=gen).item())
        cuts = sorted(torch.randperm(max(body - 1, 1), generator=gen)[:n_docs - 1].tolist())
        edges = [0] + [c + 1 for c in cuts] + [body]
        for sid, (a, e) in enumerate(zip(edges[:-1], edges[1:])):
            seg[b, a:e] = sid
            pos[b, a:e] = torch.arange(e - a, dtype=torch.int32)
        if shuffle_positions:
            pos[b] = torch.randperm(L, generator=gen).to(torch.int32)
    return seg, pos
