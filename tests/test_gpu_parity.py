"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Bars: block map and permutations bit-exact; forward O max-abs <= 2e-2 and
lse max-abs <= 1e-3 (rows whose lse is -inf must be -inf on both sides);
gradients dq, dk, dv, dsinks relative L2 <= 1e-2 per tensor.
"""
import math

import numpy as np
import pytest
import torch

import block_sparse_flash_ra_gb300 as ra
import oracle
from tests.brute import visibility
from workloads import WORKLOADS, Workload, make_inputs, random_structure

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


def check_fwd(out, lse, o_ref, l_ref):
    o, l = f64(out), f64(lse)
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(l), fin), "rows with nothing visible differ"
    assert np.all(l[~fin] == l_ref[~fin])
    if fin.any():
        assert np.max(np.abs(l[fin] - l_ref[fin])) <= LSE_TOL
    assert np.max(np.abs(o - o_ref)) <= O_TOL


def rel_l2(a, b):
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def host_permute(t, n):
    """The oracle's zigzag permutation of a CPU tensor (bitwise, any dtype)."""
    if t.dtype == torch.bfloat16:
        return torch.from_numpy(oracle.permute(t.view(torch.int16).numpy(), n)).view(torch.bfloat16)
    return torch.from_numpy(oracle.permute(t.numpy(), n))


class Case:
    """One problem, with inputs on both sides in the (possibly permuted) order."""

    def __init__(self, w: Workload, *, structure=None, seed_struct=0, dout=False,
                 overrides=None, block_q_dkv=0):
        self.w = w
        inp = make_inputs(w, with_dout=dout)
        if structure is not None:
            g = torch.Generator().manual_seed(seed_struct)
            seg, pos = random_structure(g, w.B, w.L, **structure)
            inp.update(q_seg=seg, kv_seg=seg.clone(), q_pos=pos, kv_pos=pos.clone())
        if overrides:
            inp.update(overrides)
        self.inp = inp
        N = w.n_shards
        dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        host = dict(inp)
        if w.zigzag:
            for key in ("q", "k", "v", "dout", "q_pos", "kv_pos", "q_seg", "kv_seg"):
                if dev[key] is not None:
                    dev[key] = ra.permute(dev[key], N)
                    host[key] = host_permute(host[key], N)
        self.dev, self.host = dev, host
        lm = inp.get("local_mask")
        self.params = ra.make_params(
            dev["q"], dev["k"], scale=w.scale, causal=w.causal, soft_cap=w.soft_cap,
            n_virtual_shards=N, is_mqa=w.is_mqa, q_pos=dev["q_pos"], kv_pos=dev["kv_pos"],
            q_seg=dev["q_seg"], kv_seg=dev["kv_seg"], sinks=dev["sinks"],
            local_mask=dev.get("local_mask"), block_q_dkv=block_q_dkv)
        self.okw = dict(scale=w.scale, soft_cap=w.soft_cap or None, causal=w.causal,
                        q_pos=i32(host["q_pos"]), kv_pos=i32(host["kv_pos"]),
                        q_seg=i32(host["q_seg"]), kv_seg=i32(host["kv_seg"]),
                        sinks=f64(host["sinks"]),
                        local_mask=None if lm is None else lm.numpy())

    def mask(self):
        return ra.build_mask(self.params)

    def gpu_fwd(self, workspace=True):
        m = self.mask()
        d = self.dev
        return ra.forward(self.params, d["q"], d["k"], d["v"], m, workspace=workspace) + (m,)

    def oracle_fwd(self, ring=True):
        h = self.host
        if ring:
            return oracle.attn_fwd_ring(f64(h["q"]), f64(h["k"]), f64(h["v"]),
                                        n_shards=self.w.n_shards, **self.okw)
        return oracle.attn_fwd(f64(h["q"]), f64(h["k"]), f64(h["v"]), **self.okw)


def W(**kw):
    base = dict(name="t", B=1, L=1024, Hq=4, Hkv=2, D=128, n_shards=2, seed=11)
    base.update(kw)
    return Workload(**base)


FWD_CASES = {
    "tiny_fp32": WORKLOADS["tiny"],
    "causal_n1": W(n_shards=1),
    "causal_n4": W(n_shards=4, seed=12),
    "causal_n8_one_tile_per_shard": W(n_shards=8, seed=13),
    "gqa_noncausal": W(causal=False, Hq=8, Hkv=2, seed=14),
    "mqa_sinks_cap50_zigzag": W(Hq=4, Hkv=1, is_mqa=True, sinks=True, soft_cap=50.0,
                                zigzag=True, n_shards=2, seed=15),
    "sinks_cap5": W(sinks=True, soft_cap=5.0, seed=16),
    # |s * scale| / cap mostly in [1/8, 1/4): the degree-7 tanh series
    "cap20": W(soft_cap=20.0, seed=21),
    "d64": W(D=64, seed=17),
    "d64_cap50_sinks": W(D=64, soft_cap=50.0, sinks=True, seed=22),
    "d64_fp32": W(D=64, dtype="fp32", seed=18, L=512),
    "d128_fp32_gqa_sinks_cap20_zigzag": W(dtype="fp32", Hq=4, Hkv=2, sinks=True, soft_cap=20.0,
                                          zigzag=True, n_shards=4, L=512, seed=61),
    "d128_fp32_noncausal_b2_n3": W(dtype="fp32", causal=False, B=2, Hq=2, Hkv=1, L=384,
                                   n_shards=3, seed=62),
    "zigzag_n4": W(zigzag=True, n_shards=4, seed=19),
    "b2_gqa": W(B=2, Hq=6, Hkv=3, seed=20, L=768, n_shards=3),
}


# workspace: with it, D = 128 problems whose kv heads serve an even number of
# query heads run the two-heads-per-CTA forward; without it, one head per CTA
@pytest.mark.parametrize("workspace", [True, False], ids=["ws", "no_ws"])
@pytest.mark.parametrize("name", list(FWD_CASES))
def test_forward_matches_oracle(name, workspace):
    c = Case(FWD_CASES[name])
    out, lse, _ = c.gpu_fwd(workspace)
    torch.cuda.synchronize()
    o_ref, l_ref = c.oracle_fwd()
    check_fwd(out, lse, o_ref, l_ref)


STRUCT_CASES = {
    "packed_docs_pad": (W(B=2, seed=21), dict(n_docs_max=5, pad_max=300)),
    "packed_docs_pad_sinks": (W(B=2, seed=22, sinks=True), dict(n_docs_max=4, pad_max=400)),
    "shuffled_positions": (W(seed=23, L=512, n_shards=1), dict(n_docs_max=1, shuffle_positions=True)),
    # more partial tiles than stored blocks: tiles past the capacity are
    # masked from positions and segments
    "shuffled_positions_past_block_capacity": (W(seed=26, L=2048, Hq=2, Hkv=1, n_shards=2),
                                               dict(n_docs_max=2, shuffle_positions=True)),
    "noncausal_segments": (W(causal=False, seed=24), dict(n_docs_max=6, pad_max=50)),
    "fp32_packed_docs_pad": (W(B=2, seed=63, dtype="fp32", L=512, sinks=True),
                             dict(n_docs_max=4, pad_max=100)),
}


# fp32 inputs run on the tensor cores with the logits from three tf32 products
# (q and k split into hi and lo parts), so lse stays near fp32 accuracy; P and
# V enter the output product in tf32 (relative 2^-11 per term)
F32_LSE_TOL, F32_O_TOL = 1e-4, 4e-3


@pytest.mark.parametrize("name", [n for n in FWD_CASES if "fp32" in n])
def test_fp32_forward_keeps_fp32_logits(name):
    c = Case(FWD_CASES[name])
    out, lse, _ = c.gpu_fwd()
    torch.cuda.synchronize()
    o_ref, l_ref = c.oracle_fwd()
    l, fin = f64(lse), np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.max(np.abs(l[fin] - l_ref[fin])) <= F32_LSE_TOL
    assert np.max(np.abs(f64(out) - o_ref)) <= F32_O_TOL


@pytest.mark.parametrize("workspace", [True, False], ids=["ws", "no_ws"])
@pytest.mark.parametrize("name", list(STRUCT_CASES))
def test_forward_structured_matches_oracle(name, workspace):
    w, st = STRUCT_CASES[name]
    c = Case(w, structure=st, seed_struct=7)
    out, lse, _ = c.gpu_fwd(workspace)
    torch.cuda.synchronize()
    o_ref, l_ref = c.oracle_fwd()
    check_fwd(out, lse, o_ref, l_ref)


def test_forward_all_padding_rows_and_empty_tiles():
    # the last 256 tokens are padding: two whole query tiles with no visible
    # key (lse = sink, out = 0), and padding rows inside a partial tile
    w = W(B=1, L=1024, n_shards=2, sinks=True, seed=25)
    g = torch.Generator().manual_seed(3)
    seg, pos = random_structure(g, 1, 1024, n_docs_max=3)
    seg[:, -300:] = -1
    c = Case(w, overrides=dict(q_seg=seg, kv_seg=seg.clone(), q_pos=pos, kv_pos=pos.clone()))
    out, lse, _ = c.gpu_fwd()
    torch.cuda.synchronize()
    o_ref, l_ref = c.oracle_fwd()
    check_fwd(out, lse, o_ref, l_ref)
    assert torch.all(out[:, -300:] == 0)


# ------------------------------------------------------------ block map
def _dev_arr(m, ptr, n, dtype):
    buf = m._buf
    off = ptr - buf.data_ptr()
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return buf[off:off + nbytes].view(dtype).cpu().numpy()


def _pack_rows(block):
    """(128, 128) bool -> (128, 4) uint32, bit z of word w = column 32w + z."""
    return np.packbits(block, axis=1, bitorder="little").view("<u4")


def check_partial_blocks(m, cls, vis, n_shards):
    """The partial mask blocks against the dense visibility (bit-exact):
    numbering in row and column order, per-shard first numbers, and the bits
    of every numbered tile below the capacity."""
    B, nq, nk = cls.shape
    cap = m.part_cap
    assert cap == 4 * B * (nq + nk)
    part = [(b, qt, kt) for b in range(B) for qt in range(nq) for kt in range(nk)
            if cls[b, qt, kt] == 1]
    assert int(_dev_arr(m, m.n_part, 1, torch.int32)[0]) == len(part)
    tk = nk // n_shards
    pf = _dev_arr(m, m.part_fwd, B * nq * (n_shards + 1), torch.int32).reshape(B * nq, -1)
    pb = _dev_arr(m, m.part_bwd, B * nk, torch.int32)
    want_f = np.zeros_like(pf)
    for r in range(B * nq):
        b, qt = divmod(r, nq)
        before = sum(1 for t in part if (t[0], t[1]) < (b, qt))
        for s_ in range(n_shards + 1):
            want_f[r, s_] = before + sum(1 for t in part if (t[0], t[1]) == (b, qt)
                                         and t[2] < s_ * tk)
    assert np.array_equal(pf, want_f)
    colpart = sorted(part, key=lambda t: (t[0], t[2], t[1]))
    want_b = [sum(1 for t in colpart if (t[0], t[2]) < divmod(c, nk)) for c in range(B * nk)]
    assert pb.tolist() == want_b
    rows = _dev_arr(m, m.part_rows, cap * 128 * 4, torch.int32).view("<u4").reshape(cap, 128, 4)
    cols = _dev_arr(m, m.part_cols, cap * 128 * 4, torch.int32).view("<u4").reshape(cap, 128, 4)
    for order, got, transpose in ((part, rows, False), (colpart, cols, True)):
        for slot, (b, qt, kt) in enumerate(order[:cap]):
            blk = vis[b, qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128]
            assert np.array_equal(got[slot], _pack_rows(blk.T if transpose else blk)), (slot, b, qt, kt)
    return len(part)


def check_dkv_map(m, B, L, cls128, **okw):
    """The backward's grid (64 query rows x 128 kv rows) against the oracle's
    map on that grid: classes, column counts and lists, the column order, and
    for each listed block its parent's column-order partial number."""
    ref = oracle.block_mask(B, L, L, block_q=64, block_kv=128, **okw)
    nq, nk = L // 128, L // 128
    got = dict(tile_class=_dev_arr(m, m.dkv_class, B * 2 * nq * nk, torch.uint8),
               bwd_cnt=_dev_arr(m, m.dkv_cnt, B * nk, torch.int32),
               bwd_idx=_dev_arr(m, m.dkv_idx, B * nk * 2 * nq, torch.int32),
               bwd_order=_dev_arr(m, m.dkv_order, B * nk, torch.int32))
    for key, val in got.items():
        assert np.array_equal(val.reshape(-1), np.asarray(ref[key]).reshape(-1)), key
    # parents' numbers: PARTIAL 128 x 128 tiles numbered by column (b*nk+kt),
    # then query tile, over the whole map
    slot = _dev_arr(m, m.dkv_slot, B * nk * 2 * nq, torch.int32).reshape(B * nk, 2 * nq)
    idx = np.asarray(ref["bwd_idx"]).reshape(B * nk, 2 * nq)
    cols = cls128.transpose(0, 2, 1).reshape(B * nk, nq)
    number, n = {}, 0
    for c in range(B * nk):
        for qt in range(nq):
            if cols[c, qt] == 1:
                number[(c, qt)] = n
                n += 1
    for c in range(B * nk):
        for e, qb in enumerate(idx[c]):
            if qb < 0:
                assert slot[c, e] == -1
                continue
            assert slot[c, e] == number.get((c, qb // 2), -1), (c, e)


@pytest.mark.parametrize("seed", range(5))
def test_block_mask_bit_exact(seed):
    g = torch.Generator().manual_seed(seed)
    B, L = 2, 1024 + 128 * seed
    seg, pos = random_structure(g, B, L, n_docs_max=1 + 2 * seed, pad_max=150 * seed,
                                shuffle_positions=(seed == 4))
    causal = seed != 3
    n_shards = (4, 3, 5, 11, 6)[seed]  # divides nq = 8 + seed
    q = torch.zeros(B, L, 1, 128, dtype=torch.bfloat16, device="cuda")
    dseg, dpos = seg.cuda(), pos.cuda()
    p = ra.make_params(q, q, scale=1.0, causal=causal, q_pos=dpos, kv_pos=dpos, q_seg=dseg,
                       kv_seg=dseg, n_virtual_shards=n_shards, block_q_dkv=64)
    m = ra.build_mask(p)
    torch.cuda.synchronize()
    ref = oracle.block_mask(B, L, L, causal=causal, q_pos=pos.numpy(), kv_pos=pos.numpy(),
                            q_seg=seg.numpy(), kv_seg=seg.numpy())
    nq = nk = L // 128

    buf = m._buf

    def dev_arr(ptr, n, dtype):
        off = ptr - buf.data_ptr()
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return buf[off:off + nbytes].view(dtype).cpu().numpy()

    got = dict(tile_class=dev_arr(m.tile_class, B * nq * nk, torch.uint8),
               fwd_cnt=dev_arr(m.fwd_cnt, B * nq, torch.int32),
               fwd_idx=dev_arr(m.fwd_idx, B * nq * nk, torch.int32),
               bwd_cnt=dev_arr(m.bwd_cnt, B * nk, torch.int32),
               bwd_idx=dev_arr(m.bwd_idx, B * nk * nq, torch.int32),
               fwd_order=dev_arr(m.fwd_order, B * nq, torch.int32),
               bwd_order=dev_arr(m.bwd_order, B * nk, torch.int32))
    for key, val in got.items():
        assert np.array_equal(val.reshape(-1), np.asarray(ref[key]).reshape(-1)), key
    # shard offsets: entry s of a row counts the oracle's listed tiles below s*nk/N
    shard = dev_arr(m.fwd_shard, B * nq * (n_shards + 1), torch.int32).reshape(B * nq, -1)
    idx = np.asarray(ref["fwd_idx"]).reshape(B * nq, nk)
    tk = nk // n_shards
    for r in range(B * nq):
        listed = idx[r][idx[r] >= 0]
        want = [int(np.sum(listed < s_ * tk)) for s_ in range(n_shards + 1)]
        assert shard[r].tolist() == want, r
    vis = visibility(B, L, L, causal=causal, q_pos=pos.numpy(), kv_pos=pos.numpy(),
                     q_seg=seg.numpy(), kv_seg=seg.numpy())
    check_partial_blocks(m, np.asarray(ref["tile_class"]).reshape(B, nq, nk), vis, n_shards)
    check_dkv_map(m, B, L, np.asarray(ref["tile_class"]).reshape(B, nq, nk), causal=causal,
                  q_pos=pos.numpy(), kv_pos=pos.numpy(), q_seg=seg.numpy(), kv_seg=seg.numpy())


def test_block_mask_partial_blocks_past_capacity():
    # shuffled positions: all 256 tiles partial, blocks for the first 128 only
    g = torch.Generator().manual_seed(4)
    B, L, N = 1, 2048, 2
    seg, pos = random_structure(g, B, L, n_docs_max=2, shuffle_positions=True)
    q = torch.zeros(B, L, 1, 128, dtype=torch.bfloat16, device="cuda")
    dseg, dpos = seg.cuda(), pos.cuda()
    p = ra.make_params(q, q, scale=1.0, causal=True, q_pos=dpos, kv_pos=dpos, q_seg=dseg,
                       kv_seg=dseg, n_virtual_shards=N, block_q_dkv=64)
    m = ra.build_mask(p)
    torch.cuda.synchronize()
    ref = oracle.block_mask(B, L, L, causal=True, q_pos=pos.numpy(), kv_pos=pos.numpy(),
                            q_seg=seg.numpy(), kv_seg=seg.numpy())
    vis = visibility(B, L, L, causal=True, q_pos=pos.numpy(), kv_pos=pos.numpy(),
                     q_seg=seg.numpy(), kv_seg=seg.numpy())
    nq = L // 128
    n_part = check_partial_blocks(m, np.asarray(ref["tile_class"]).reshape(B, nq, nq), vis, N)
    assert n_part > m.part_cap
    # the backward grid's classes of parents past the capacity come from
    # positions and segments: exact all the same
    check_dkv_map(m, B, L, np.asarray(ref["tile_class"]).reshape(B, nq, nq), causal=True,
                  q_pos=pos.numpy(), kv_pos=pos.numpy(), q_seg=seg.numpy(), kv_seg=seg.numpy())


def test_block_mask_sequential_positions_bit_exact():
    # no position / segment arrays: positions are the token indices
    B, L = 1, 2048
    q = torch.zeros(B, L, 1, 64, dtype=torch.bfloat16, device="cuda")
    for causal in (True, False):
        p = ra.make_params(q, q, scale=1.0, causal=causal, n_virtual_shards=4)
        m = ra.build_mask(p)
        off = m.tile_class - m._buf.data_ptr()
        cls = m._buf[off:off + B * 16 * 16].cpu().numpy()
        ref = oracle.block_mask(B, L, L, causal=causal)
        assert np.array_equal(cls, ref["tile_class"].reshape(-1))


# ------------------------------------------------------------ permutation
@pytest.mark.parametrize("dtype,inner", [(torch.bfloat16, (4, 64)), (torch.int32, ()),
                                         (torch.float32, (3,)), (torch.uint8, (5,))])
@pytest.mark.parametrize("n", [1, 2, 8])
def test_permute_bit_exact(dtype, inner, n):
    B, L = 2, 256
    g = torch.Generator().manual_seed(n)
    x = (torch.randn((B, L) + inner, generator=g) * 50).to(dtype)
    y = ra.permute(x.cuda(), n)
    src = x.view(torch.int16) if dtype == torch.bfloat16 else x
    ref = oracle.permute(src.numpy(), n)
    got = y.cpu().view(torch.int16) if dtype == torch.bfloat16 else y.cpu()
    assert np.array_equal(got.numpy(), ref)
    back = ra.unpermute(y, n)
    assert torch.equal(back.cpu(), x)


# ------------------------------------------------------------ merge
@pytest.mark.parametrize("D", [128, 64, 8, 4, 200, 132])
def test_merge_matches_oracle(D):
    g = torch.Generator().manual_seed(5)
    B, L, H = 2, 301, 3
    o = torch.randn(B, L, H, D, generator=g)
    bo = torch.randn(B, L, H, D, generator=g)
    l = torch.randn(B, H, L, generator=g) * 3
    bl = torch.randn(B, H, L, generator=g) * 3
    l[0, 0, :7] = -math.inf      # first merge: take the block
    bl[1, 2, 5:9] = -math.inf    # empty block: no change
    l[1, 1, 3] = bl[1, 1, 3] = -math.inf
    ro, rl = oracle.merge(o.double().numpy(), l.double().numpy(), bo.double().numpy(),
                          bl.double().numpy())
    do, dl = o.cuda(), l.cuda()
    ra.ra_merge_out_lse(do, dl, bo.cuda(), bl.cuda(), B, L, H, D)
    torch.cuda.synchronize()
    dl = dl.cpu().double().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(dl), fin)
    assert np.max(np.abs(dl[fin] - rl[fin])) < 1e-5
    assert np.max(np.abs(do.cpu().double().numpy() - ro)) < 1e-5


def test_merge_extreme_lse_gaps():
    # lse gaps of +-80 (sigmoid ~ e^-80 or 1 - e^-80, softplus ~ e^-80 or 80),
    # a -inf block after a finite running lse (a shard with nothing visible
    # for the row), and both -inf: O and lse must follow the oracle's update
    g = torch.Generator().manual_seed(9)
    B, L, H, D = 1, 64, 2, 128
    o = torch.randn(B, L, H, D, generator=g)
    bo = torch.randn(B, L, H, D, generator=g)
    l = torch.randn(B, H, L, generator=g)
    bl = l.clone()
    bl[:, :, 0:16] += 80.0
    bl[:, :, 16:32] -= 80.0
    bl[:, :, 32:40] = -math.inf
    bl[:, :, 40:48] += 30.0
    bl[:, :, 48:56] -= 30.0
    l[:, :, 56:60] = -math.inf
    l[:, :, 60:64] = bl[:, :, 60:64] = -math.inf
    ro, rl = oracle.merge(o.double().numpy(), l.double().numpy(), bo.double().numpy(),
                          bl.double().numpy())
    do, dl = o.cuda(), l.cuda()
    ra.ra_merge_out_lse(do, dl, bo.cuda(), bl.cuda(), B, L, H, D)
    torch.cuda.synchronize()
    dl = dl.cpu().double().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(dl), fin)
    assert np.max(np.abs(dl[fin] - rl[fin])) <= 1e-5 * np.maximum(1.0, np.abs(rl[fin])).max()
    got_o = do.cpu().double().numpy()
    assert not np.isnan(got_o).any()
    assert np.max(np.abs(got_o - ro)) < 1e-5


# ------------------------------------------------------------ backward
BWD_CASES = {
    "causal_gqa": W(Hq=4, Hkv=2, L=512, seed=31, n_shards=2),
    "mqa_sinks_cap": W(Hq=4, Hkv=1, is_mqa=True, sinks=True, soft_cap=5.0, L=512, seed=32),
    "noncausal": W(causal=False, L=512, seed=33),
    "d64_zigzag": W(D=64, L=512, zigzag=True, n_shards=2, seed=34),
    "mqa_sinks_cap50": W(Hq=4, Hkv=1, is_mqa=True, sinks=True, soft_cap=50.0, L=512, seed=37),
    "cap20": W(Hq=4, Hkv=2, soft_cap=20.0, L=512, seed=39),
    "d64_cap20_sinks": W(D=64, Hq=4, Hkv=2, soft_cap=20.0, sinks=True, L=512, seed=40),
    "ragged_n5_b2": W(B=2, Hq=6, Hkv=2, L=640, n_shards=5, seed=38),
    # fp32 inputs: the gradient kernels read bf16 copies (rounded once) and
    # accumulate into fp32 dq, dk, dv; Delta and dsinks come from fp32 out, dO
    "tiny_fp32": WORKLOADS["tiny"].scaled(backward=True),
    "fp32_gqa_sinks_cap20_zigzag": W(dtype="fp32", Hq=4, Hkv=2, sinks=True, soft_cap=20.0, L=512,
                                     zigzag=True, seed=42),
    "fp32_mqa_d64": W(dtype="fp32", D=64, Hq=4, Hkv=1, is_mqa=True, L=512, n_shards=4, seed=43),
}


def _check_bwd(c, grads):
    h = c.host
    dq, dk, dv, ds, _, _ = oracle.attn_bwd(f64(h["q"]), f64(h["k"]), f64(h["v"]), f64(h["dout"]),
                                           **c.okw)
    for name, got, ref in (("dq", grads[0], dq), ("dk", grads[1], dk), ("dv", grads[2], dv)):
        err = rel_l2(f64(got), ref)
        assert err <= GRAD_TOL, (name, err)
    if ds is not None:
        err = rel_l2(f64(grads[3]), ds)
        assert err <= GRAD_TOL, ("dsinks", err)


# block_q_dkv = 64: the dK/dV stage on the backward's own grid (64 query rows
# x 128 kv rows; D = 128 only)
@pytest.mark.parametrize("block_q_dkv", [0, 64], ids=["dkv128", "dkv64"])
@pytest.mark.parametrize("name", list(BWD_CASES))
def test_backward_matches_oracle(name, block_q_dkv):
    if block_q_dkv == 64 and BWD_CASES[name].D != 128:
        pytest.skip("the 64-row dK/dV grid serves D = 128")
    c = Case(BWD_CASES[name], dout=True, block_q_dkv=block_q_dkv)
    out, lse, m = c.gpu_fwd()
    d = c.dev
    grads = ra.backward(c.params, d["q"], d["k"], d["v"], out, lse, d["dout"], m)
    torch.cuda.synchronize()
    _check_bwd(c, grads)


# Query and key lengths that differ: each virtual device holds Lq/N query rows
# and Lkv/N key rows.  "suffix": the queries are the last Lq positions of the
# key sequence (explicit positions), so causal rows see a prefix of keys.
UNEQUAL = {
    "lkv2x_noncausal_n2": dict(Lq=512, Lkv=1024, causal=False, N=2, seed=71),
    "lkv2x_causal_suffix_n4_sinks": dict(Lq=512, Lkv=1024, causal=True, N=4, seed=72, suffix=True,
                                         sinks=True),
    "lq2x_causal_n2_cap20": dict(Lq=1024, Lkv=512, causal=True, N=2, seed=73, cap=20.0),
    "lkv3x_gqa_d64_n1": dict(Lq=256, Lkv=768, causal=False, N=1, seed=74, D=64, Hq=6),
}


@pytest.mark.parametrize("name", list(UNEQUAL))
def test_unequal_lengths_match_oracle(name):
    cfg = UNEQUAL[name]
    g = torch.Generator().manual_seed(cfg["seed"])
    B, Hq, Hkv, D = 1, cfg.get("Hq", 4), 2, cfg.get("D", 128)
    Lq, Lkv, N = cfg["Lq"], cfg["Lkv"], cfg["N"]
    q, do = (torch.randn(B, Lq, Hq, D, generator=g).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn(B, Lkv, Hkv, D, generator=g).to(torch.bfloat16) for _ in range(2))
    q_pos = kv_pos = None
    if cfg.get("suffix"):
        q_pos = (torch.arange(Lq, dtype=torch.int32) + (Lkv - Lq)).expand(B, Lq).contiguous()
        kv_pos = torch.arange(Lkv, dtype=torch.int32).expand(B, Lkv).contiguous()
    sinks = torch.randn(Hq, generator=g) if cfg.get("sinks") else None
    cu = lambda t: None if t is None else t.cuda()  # noqa: E731
    dq_, dk_, dv_, ddo = cu(q), cu(k), cu(v), cu(do)
    p = ra.make_params(dq_, dk_, scale=D ** -0.5, causal=cfg["causal"], soft_cap=cfg.get("cap", 0.0),
                       n_virtual_shards=N, q_pos=cu(q_pos), kv_pos=cu(kv_pos), sinks=cu(sinks))
    m = ra.build_mask(p)
    out, lse = ra.forward(p, dq_, dk_, dv_, m)
    grads = ra.backward(p, dq_, dk_, dv_, out, lse, ddo, m)
    torch.cuda.synchronize()
    okw = dict(scale=D ** -0.5, soft_cap=cfg.get("cap"), causal=cfg["causal"], q_pos=i32(q_pos),
               kv_pos=i32(kv_pos), sinks=f64(sinks))
    o_ref, l_ref = oracle.attn_fwd_ring(f64(q), f64(k), f64(v), n_shards=N, **okw)
    check_fwd(out, lse, o_ref, l_ref)
    dq, dk, dv, ds, _, _ = oracle.attn_bwd(f64(q), f64(k), f64(v), f64(do), **okw)
    for nm, got, ref in (("dq", grads[0], dq), ("dk", grads[1], dk), ("dv", grads[2], dv)):
        assert rel_l2(f64(got), ref) <= GRAD_TOL, nm
    if ds is not None:
        assert rel_l2(f64(grads[3]), ds) <= GRAD_TOL


def test_backward_packed_docs_with_padding():
    c = Case(W(B=2, L=768, Hq=2, Hkv=2, seed=35, n_shards=3, sinks=True), dout=True,
             structure=dict(n_docs_max=4, pad_max=200), seed_struct=9)
    out, lse, m = c.gpu_fwd()
    d = c.dev
    grads = ra.backward(c.params, d["q"], d["k"], d["v"], out, lse, d["dout"], m)
    torch.cuda.synchronize()
    _check_bwd(c, grads)


def test_backward_past_partial_block_capacity():
    # shuffled positions make (nearly) every tile partial: 256 tiles, 128 blocks
    c = Case(W(B=1, L=2048, Hq=2, Hkv=1, seed=39, n_shards=2), dout=True,
             structure=dict(n_docs_max=2, shuffle_positions=True), seed_struct=4)
    out, lse, m = c.gpu_fwd()
    assert int(_dev_arr(m, m.n_part, 1, torch.int32)[0]) > m.part_cap
    d = c.dev
    grads = ra.backward(c.params, d["q"], d["k"], d["v"], out, lse, d["dout"], m)
    torch.cuda.synchronize()
    _check_bwd(c, grads)


def test_backward_padding_rows_inside_a_tile_without_sinks():
    # rows 700..767 are padding: nothing visible, lse = -inf, and they share
    # the last 128-row tile with document rows, so that tile is partial for
    # them (no sink keeps their lse finite here)
    B, L = 1, 768
    seg = torch.zeros((B, L), dtype=torch.int32)
    seg[:, 700:] = -1
    pos = torch.arange(L, dtype=torch.int32).unsqueeze(0).clone()
    c = Case(W(B=B, L=L, Hq=2, Hkv=1, seed=36, n_shards=3), dout=True,
             overrides=dict(q_seg=seg, kv_seg=seg.clone(), q_pos=pos, kv_pos=pos.clone()))
    out, lse, m = c.gpu_fwd()
    d = c.dev
    grads = ra.backward(c.params, d["q"], d["k"], d["v"], out, lse, d["dout"], m)
    torch.cuda.synchronize()
    for g in grads[:3]:
        assert torch.isfinite(g).all()
    _check_bwd(c, grads)


# ------------------------------------------- the non-causal ring's local mask
def _local_mask(seed, ls, window=None, density=0.9):
    """(ls, ls) uint8: a band |i - j| < window (if given) with random holes."""
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand((ls, ls), generator=g) < density)
    if window is not None:
        i = torch.arange(ls)[:, None]
        j = torch.arange(ls)[None, :]
        m &= (i - j).abs() < window
    return m.to(torch.uint8)


LOCAL_CASES = {
    "n2_band": (W(causal=False, n_shards=2, seed=51), dict(window=200)),
    "n4_random_segments": (W(causal=False, n_shards=4, seed=52), dict(density=0.6, segs=True)),
    "mqa_sinks_cap": (W(causal=False, Hq=4, Hkv=1, is_mqa=True, sinks=True, soft_cap=30.0,
                        n_shards=2, seed=53), dict(window=300, density=0.95)),
    "d64": (W(causal=False, D=64, n_shards=2, seed=54), dict(window=64)),
    "fp32": (W(causal=False, D=64, dtype="fp32", L=512, n_shards=2, seed=55), dict(window=100)),
    # one shard: the mask covers the whole (Lq, Lkv) grid (a dense 2-D mask)
    "n1_dense_random": (W(causal=False, n_shards=1, seed=56, L=1536), dict(density=0.3)),
}


def _local_case(name, dout=False):
    w, spec = LOCAL_CASES[name]
    spec = dict(spec)
    segs = spec.pop("segs", False)
    lm = _local_mask(w.seed, w.L // w.n_shards, **spec)
    kw = dict(overrides=dict(local_mask=lm), dout=dout)
    if segs:
        kw.update(structure=dict(n_docs_max=3, pad_max=100), seed_struct=w.seed)
    return Case(w, **kw)


@pytest.mark.parametrize("name", list(LOCAL_CASES))
def test_local_mask_forward_matches_oracle(name):
    c = _local_case(name)
    out, lse, _ = c.gpu_fwd()
    torch.cuda.synchronize()
    o_ref, l_ref = c.oracle_fwd()
    check_fwd(out, lse, o_ref, l_ref)


@pytest.mark.parametrize("name", ["n2_band", "n4_random_segments", "mqa_sinks_cap",
                                  "n1_dense_random"])
def test_local_mask_backward_matches_oracle(name):
    c = _local_case(name, dout=True)
    out, lse, m = c.gpu_fwd()
    d = c.dev
    grads = ra.backward(c.params, d["q"], d["k"], d["v"], out, lse, d["dout"], m)
    torch.cuda.synchronize()
    _check_bwd(c, grads)


def test_local_mask_block_map_bit_exact():
    g = torch.Generator().manual_seed(9)
    B, L, N = 2, 1024, 4
    seg, pos = random_structure(g, B, L, n_docs_max=3, pad_max=150)
    lm = _local_mask(3, L // N, window=180, density=0.97)
    q = torch.zeros(B, L, 1, 128, dtype=torch.bfloat16, device="cuda")
    dseg, dlm = seg.cuda(), lm.cuda()
    p = ra.make_params(q, q, scale=1.0, causal=False, q_seg=dseg, kv_seg=dseg,
                       n_virtual_shards=N, local_mask=dlm, block_q_dkv=64)
    m = ra.build_mask(p)
    torch.cuda.synchronize()
    ref = oracle.block_mask(B, L, L, causal=False, q_seg=seg.numpy(), kv_seg=seg.numpy(),
                            local_mask=lm.numpy())
    nq = nk = L // 128
    buf = m._buf
    off = m.tile_class - buf.data_ptr()
    got = buf[off:off + B * nq * nk].cpu().numpy()
    assert np.array_equal(got, ref["tile_class"].reshape(-1))
    assert (got == 0).any() and (got == 1).any()  # the band leaves empty and partial tiles
    vis = visibility(B, L, L, causal=False, q_seg=seg.numpy(), kv_seg=seg.numpy(),
                     local_mask=lm.numpy())
    check_partial_blocks(m, got.reshape(B, nq, nk), vis, N)
    check_dkv_map(m, B, L, got.reshape(B, nq, nk), causal=False, q_seg=seg.numpy(),
                  kv_seg=seg.numpy(), local_mask=lm.numpy())
