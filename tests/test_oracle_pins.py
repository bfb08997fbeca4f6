"""Pins of the fp64 oracle to things other than itself (CPU only).

* hand-derived worked examples (tests/golden/worked_examples.json);
* brute force on tiny inputs (tests/brute.py, vectorised numpy + scipy);
* a library special case (torch scaled_dot_product_attention, fp64, CPU);
* invariants the method must satisfy (ring == plain, segment isolation,
  padding rows, sink adds to the denominator only, MQA == MHA with repeated
  keys, constant V, causal row 0, large cap -> no cap);
* central finite differences of the forward for the backward;
* per-pair brute force for the block map, index formula tables for the
  zigzag permutation.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests import brute
from workloads import random_structure

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
_ENV = {"log": math.log, "exp": math.exp, "tanh": math.tanh, "inf": math.inf}


def ev(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, _ENV))
    if isinstance(x, list):
        return [ev(y) for y in x]
    return float(x)


def _arr(x, shape=None):
    a = np.array(ev(x), dtype=np.float64)
    return a.reshape(shape) if shape is not None else a


def _tiny(ex):
    L = len(ex["q"])
    D = len(ex["q"][0])
    q = _arr(ex["q"]).reshape(1, L, 1, D)
    k = _arr(ex["k"]).reshape(1, L, 1, D)
    v = _arr(ex["v"]).reshape(1, L, 1, D)
    kw = dict(scale=ev(ex["scale"]), causal=ex.get("causal", False))
    if "soft_cap" in ex:
        kw["soft_cap"] = ev(ex["soft_cap"])
    if "sinks" in ex:
        kw["sinks"] = _arr(ex["sinks"])
    if "q_seg" in ex:
        kw["q_seg"] = np.array([ex["q_seg"]], np.int32)
        kw["kv_seg"] = np.array([ex["kv_seg"]], np.int32)
    return q, k, v, kw


# ---------------------------------------------------------------- golden
@pytest.mark.parametrize("ex", GOLD["attention"], ids=lambda e: e["name"])
def test_golden_attention(ex):
    q, k, v, kw = _tiny(ex)
    L = q.shape[1]
    if "n_shards" in ex:
        out, lse = oracle.attn_fwd_ring(q, k, v, n_shards=ex["n_shards"], **kw)
    else:
        out, lse = oracle.attn_fwd(q, k, v, **kw)
    np.testing.assert_allclose(out.reshape(L, -1), _arr(ex["out"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(L), _arr(ex["lse"]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("ex", GOLD["gradients"], ids=lambda e: e["name"])
def test_golden_gradients(ex):
    q, k, v, kw = _tiny(ex)
    L = q.shape[1]
    do = _arr(ex["dout"]).reshape(q.shape)
    dq, dk, dv, ds, _, _ = oracle.attn_bwd(q, k, v, do, **kw)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        if name in ex:
            np.testing.assert_allclose(got.reshape(L, -1), _arr(ex[name]), atol=1e-12)
    if "dsinks" in ex:
        np.testing.assert_allclose(ds, _arr(ex["dsinks"]), atol=1e-12)


@pytest.mark.parametrize("ex", GOLD["merge"], ids=lambda e: e["name"])
def test_golden_merge(ex):
    o = np.full((1, 1, 1, 1), ev(ex["out"]))
    l = np.full((1, 1, 1), ev(ex["lse"]))
    bo = np.full((1, 1, 1, 1), ev(ex["block_out"]))
    bl = np.full((1, 1, 1), ev(ex["block_lse"]))
    no, nl = oracle.merge(o, l, bo, bl)
    assert abs(no.item() - ev(ex["new_out"])) < 1e-12
    assert nl.item() == ev(ex["new_lse"]) or abs(nl.item() - ev(ex["new_lse"])) < 1e-12


@pytest.mark.parametrize("ex", GOLD["zigzag"], ids=lambda e: f"L{e['L']}n{e['n_shards']}")
def test_golden_zigzag(ex):
    L, n = ex["L"], ex["n_shards"]
    src = [oracle.zigzag_source(L, n, p) for p in range(L)]
    assert src == ex["source"]
    x = np.arange(L, dtype=np.int32).reshape(1, L)
    assert oracle.permute(x, n)[0].tolist() == ex["source"]


@pytest.mark.parametrize("ex", GOLD["block_mask"], ids=lambda e: f"causal{e['causal']}")
def test_golden_block_mask(ex):
    L = ex["L"]
    seg = None
    if "seg_first" in ex:
        seg = np.full((1, L), -1, np.int32)
        seg[0, :ex["seg_first"]] = 0
    m = oracle.block_mask(1, L, L, causal=ex["causal"], q_seg=seg, kv_seg=seg)
    for key in ("tile_class", "fwd_cnt", "fwd_idx", "bwd_cnt", "bwd_idx", "fwd_order", "bwd_order"):
        assert np.array_equal(np.asarray(m[key]).reshape(-1), np.asarray(ex[key]).reshape(-1)), key


# ------------------------------------------------------------ brute force
def _case(seed, *, B=2, L=96, Hq=4, Hkv=2, D=16, causal=True, segs=False, pad=0, sinks=False,
          cap=0.0, shuffle=False):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, L, Hq, D, generator=g, dtype=torch.float64).numpy()
    k = torch.randn(B, L, Hkv, D, generator=g, dtype=torch.float64).numpy()
    v = torch.randn(B, L, Hkv, D, generator=g, dtype=torch.float64).numpy()
    kw = dict(scale=1.0 / math.sqrt(D), causal=causal)
    if segs or pad or shuffle:
        seg, pos = random_structure(g, B, L, n_docs_max=3 if segs else 1, pad_max=pad,
                                    shuffle_positions=shuffle)
        kw.update(q_seg=seg.numpy(), kv_seg=seg.numpy(), q_pos=pos.numpy(), kv_pos=pos.numpy())
    if sinks:
        kw["sinks"] = torch.randn(Hq, generator=g, dtype=torch.float64).numpy()
    if cap:
        kw["soft_cap"] = cap
    return q, k, v, kw


CASES = [
    dict(),
    dict(causal=False),
    dict(segs=True),
    dict(segs=True, pad=20),
    dict(sinks=True),
    dict(cap=1.5),
    dict(segs=True, pad=12, sinks=True, cap=2.0),
    dict(Hq=4, Hkv=1),
    dict(Hq=3, Hkv=3, causal=False, shuffle=True),
    dict(L=64, shuffle=True, segs=True, sinks=True),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_fwd_equals_bruteforce(ci):
    q, k, v, kw = _case(100 + ci, **CASES[ci])
    o1, l1 = oracle.attn_fwd(q, k, v, **kw)
    o2, l2 = brute.attention(q, k, v, **kw)
    assert np.array_equal(np.isfinite(l1), np.isfinite(l2))
    f = np.isfinite(l2)
    np.testing.assert_allclose(l1[f], l2[f], atol=1e-12, rtol=0)
    np.testing.assert_allclose(o1, o2, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_equals_torch_sdpa(causal):
    q, k, v, kw = _case(7, B=2, L=80, Hq=2, Hkv=2, D=8, causal=causal, segs=True, pad=10)
    out, _ = oracle.attn_fwd(q, k, v, **kw)
    vis = brute.visibility(2, 80, 80, causal=causal, q_pos=kw.get("q_pos"), kv_pos=kw.get("kv_pos"),
                           q_seg=kw.get("q_seg"), kv_seg=kw.get("kv_seg"))
    qt, kt, vt = (torch.from_numpy(a).transpose(1, 2) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(vis)[:, None], scale=kw["scale"])
    ref = ref.transpose(1, 2).numpy()
    rows = vis.any(-1)  # rows with nothing visible are NaN in the library routine
    np.testing.assert_allclose(out[rows], ref[rows], atol=1e-12, rtol=0)
    assert np.all(out[~rows] == 0)


# ------------------------------------------------------------- invariants
@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("ci", [0, 3, 6, 7])
def test_ring_equals_plain(n, ci):
    case = dict(CASES[ci])
    case["L"] = 128
    q, k, v, kw = _case(200 + ci, **case)
    o1, l1 = oracle.attn_fwd(q, k, v, **kw)
    o2, l2 = oracle.attn_fwd_ring(q, k, v, n_shards=n, **kw)
    assert np.array_equal(np.isfinite(l1), np.isfinite(l2))
    f = np.isfinite(l1)
    np.testing.assert_allclose(l2[f], l1[f], atol=1e-12, rtol=0)
    np.testing.assert_allclose(o2, o1, atol=1e-12, rtol=0)


def test_merge_closed_form():
    g = np.random.default_rng(3)
    B, L, H, D = 2, 5, 3, 4
    o, bo = g.normal(size=(B, L, H, D)), g.normal(size=(B, L, H, D))
    l, bl = g.normal(size=(B, H, L)) * 3, g.normal(size=(B, H, L)) * 3
    no, nl = oracle.merge(o, l, bo, bl)
    np.testing.assert_allclose(nl, np.logaddexp(l, bl), atol=1e-13)
    wa = np.exp(l - nl).transpose(0, 2, 1)[..., None]
    wb = np.exp(bl - nl).transpose(0, 2, 1)[..., None]
    np.testing.assert_allclose(no, wa * o + wb * bo, atol=1e-13)


def test_merge_split_keys_equals_unsplit():
    """Partials over disjoint key sets merged by the update equal attention over all keys."""
    q, k, v, kw = _case(11, B=1, L=96, Hq=2, Hkv=2, D=8, causal=False)
    full_o, full_l = oracle.attn_fwd(q, k, v, **kw)
    rng = np.random.default_rng(0)
    part = rng.integers(0, 3, size=96)
    run_o, run_l = np.zeros_like(full_o), np.full_like(full_l, -np.inf)
    for c in range(3):
        seg_k = np.where(part == c, 0, 5).astype(np.int32)[None]
        seg_q = np.zeros((1, 96), np.int32)
        bo, bl = oracle.attn_fwd(q, k, v, q_seg=seg_q, kv_seg=seg_k, **kw)
        run_o, run_l = oracle.merge(run_o, run_l, bo, bl)
    np.testing.assert_allclose(run_l, full_l, atol=1e-12)
    np.testing.assert_allclose(run_o, full_o, atol=1e-12)


def test_causal_row0_and_constant_v():
    q, k, v, kw = _case(5, B=1, L=64, Hq=2, Hkv=2, D=8)
    out, lse = oracle.attn_fwd(q, k, v, **kw)
    np.testing.assert_allclose(out[0, 0], v[0, 0], atol=1e-14)
    s00 = kw["scale"] * np.sum(q[0, 0] * k[0, 0], axis=-1)
    np.testing.assert_allclose(lse[0, :, 0], s00, atol=1e-14)
    vc = np.full_like(v, 0.7)
    out, _ = oracle.attn_fwd(q, k, vc, **kw)
    np.testing.assert_allclose(out, 0.7, atol=1e-13)


def test_segment_isolation_and_padding_rows():
    q, k, v, kw = _case(9, B=2, L=96, segs=True, pad=16)
    o1, l1 = oracle.attn_fwd(q, k, v, **kw)
    seg = kw["q_seg"]
    # perturb keys / values of every segment except the one of row (b, i)
    for b, i in [(0, 5), (1, 40), (0, 70)]:
        if seg[b, i] == -1:
            continue
        other = seg[b] != seg[b, i]
        k2, v2 = k.copy(), v.copy()
        k2[b, other] += 3.0
        v2[b, other] -= 5.0
        o2, l2 = oracle.attn_fwd(q, k2, v2, **kw)
        assert np.array_equal(o1[b, i], o2[b, i])
        assert np.array_equal(l1[b, :, i], l2[b, :, i])
    pad_rows = seg == -1
    assert pad_rows.any()
    assert np.all(o1[pad_rows] == 0)
    assert np.all(np.isneginf(l1.transpose(0, 2, 1)[pad_rows]))
    kw["sinks"] = np.array([0.3, -0.2, 1.1, 0.0])
    o3, l3 = oracle.attn_fwd(q, k, v, **kw)
    assert np.all(o3[pad_rows] == 0)
    np.testing.assert_allclose(l3.transpose(0, 2, 1)[pad_rows],
                               np.broadcast_to(kw["sinks"], l3.transpose(0, 2, 1)[pad_rows].shape))


def test_sink_adds_to_denominator_only():
    q, k, v, kw = _case(13, B=2, L=64, segs=True)
    o0, l0 = oracle.attn_fwd(q, k, v, **kw)
    sinks = np.array([0.5, -1.0, 2.0, 0.0])
    o1, l1 = oracle.attn_fwd(q, k, v, sinks=sinks, **kw)
    ls = np.logaddexp(l0, sinks[None, :, None])
    np.testing.assert_allclose(l1, ls, atol=1e-12)
    ratio = np.exp(l0 - l1).transpose(0, 2, 1)[..., None]
    np.testing.assert_allclose(o1, o0 * ratio, atol=1e-12)


def test_mqa_gqa_equal_mha_with_repeated_kv():
    q, k, v, kw = _case(17, B=1, L=64, Hq=4, Hkv=1, D=8, sinks=True, cap=3.0)
    o1, l1 = oracle.attn_fwd(q, k, v, **kw)
    o2, l2 = oracle.attn_fwd(q, np.repeat(k, 4, 2), np.repeat(v, 4, 2), **kw)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
    q, k, v, kw = _case(19, B=1, L=64, Hq=4, Hkv=2, D=8, segs=True)
    do = np.random.default_rng(1).normal(size=q.shape)
    g1 = oracle.attn_bwd(q, k, v, do, **kw)
    kr, vr = np.repeat(k, 2, 2), np.repeat(v, 2, 2)
    g2 = oracle.attn_bwd(q, kr, vr, do, **kw)
    np.testing.assert_allclose(g1[0], g2[0], atol=1e-12)
    for a, b in ((g1[1], g2[1]), (g1[2], g2[2])):
        np.testing.assert_allclose(a, b.reshape(1, 64, 2, 2, 8).sum(3), atol=1e-12)


def test_large_cap_approaches_uncapped():
    q, k, v, kw = _case(23, B=1, L=64)
    o0, l0 = oracle.attn_fwd(q, k, v, **kw)
    o1, l1 = oracle.attn_fwd(q, k, v, soft_cap=1e6, **kw)
    np.testing.assert_allclose(o1, o0, atol=1e-9)
    np.testing.assert_allclose(l1, l0, atol=1e-9)


# ------------------------------------------------------- finite differences
@pytest.mark.parametrize("ci", [0, 1, 3, 6, 7])
def test_bwd_central_differences(ci):
    case = dict(CASES[ci])
    case.update(B=1, L=24, D=4)
    q, k, v, kw = _case(300 + ci, **case)
    do = np.random.default_rng(ci).normal(size=q.shape)
    dq, dk, dv, ds, _, _ = oracle.attn_bwd(q, k, v, do, **kw)

    def loss(q_, k_, v_, sinks_=None):
        kk = dict(kw)
        if sinks_ is not None:
            kk["sinks"] = sinks_
        o, _ = oracle.attn_fwd(q_, k_, v_, **kk)
        return float(np.sum(o * do))

    rng = np.random.default_rng(1000 + ci)
    h = 1e-5
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            ap, am = arr.copy(), arr.copy()
            ap[idx] += h
            am[idx] -= h
            args_p = {"q": (ap, k, v), "k": (q, ap, v), "v": (q, k, ap)}[name]
            args_m = {"q": (am, k, v), "k": (q, am, v), "v": (q, k, am)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])
    if "sinks" in kw:
        for hh in range(q.shape[2]):
            sp, sm = kw["sinks"].copy(), kw["sinks"].copy()
            sp[hh] += h
            sm[hh] -= h
            fd = (loss(q, k, v, sp) - loss(q, k, v, sm)) / (2 * h)
            assert abs(fd - ds[hh]) <= 1e-6 * max(1.0, abs(fd))


# ------------------------------------------------------------ block map
def _brute_map(B, L, **kw):
    vis = brute.visibility(B, L, L, **kw)
    n = L // 128
    cnt = vis.reshape(B, n, 128, n, 128).sum(axis=(2, 4))
    cls = np.where(cnt == 0, 0, np.where(cnt == 128 * 128, 2, 1)).astype(np.uint8)
    return cls


@pytest.mark.parametrize("seed", range(4))
def test_block_mask_bruteforce(seed):
    g = torch.Generator().manual_seed(seed)
    B, L = 2, 512
    seg, pos = random_structure(g, B, L, n_docs_max=5, pad_max=200, shuffle_positions=seed == 3)
    kw = dict(causal=seed != 2, q_pos=pos.numpy(), kv_pos=pos.numpy(), q_seg=seg.numpy(),
              kv_seg=seg.numpy())
    m = oracle.block_mask(B, L, L, **kw)
    cls = _brute_map(B, L, **kw)
    assert np.array_equal(m["tile_class"], cls)
    n = L // 128
    flat = cls.reshape(B * n, n)
    for r in range(B * n):
        nz = np.nonzero(flat[r])[0]
        assert m["fwd_cnt"][r] == len(nz)
        assert np.array_equal(m["fwd_idx"][r][:len(nz)], nz)
        assert np.all(m["fwd_idx"][r][len(nz):] == -1)
    colcls = cls.transpose(0, 2, 1).reshape(B * n, n)
    for c in range(B * n):
        nz = np.nonzero(colcls[c])[0]
        assert m["bwd_cnt"][c] == len(nz)
        assert np.array_equal(m["bwd_idx"][c][:len(nz)], nz)
    ford = np.lexsort((np.arange(B * n), -m["fwd_cnt"]))
    bord = np.lexsort((np.arange(B * n), -m["bwd_cnt"]))
    assert np.array_equal(m["fwd_order"], ford)
    assert np.array_equal(m["bwd_order"], bord)


@pytest.mark.parametrize("bq,bk", [(64, 128), (128, 64), (64, 64), (32, 128)])
def test_block_mask_other_block_sizes_bruteforce(bq, bk):
    # the backward's own grid (the dkv MaskInfo of make_ring_attention on
    # (block_q_dkv, block_kv_dkv)): classes from per-pair counts, lists, orders
    g = torch.Generator().manual_seed(bq + bk)
    B, L = 2, 512
    seg, pos = random_structure(g, B, L, n_docs_max=5, pad_max=150)
    kw = dict(causal=True, q_pos=pos.numpy(), kv_pos=pos.numpy(), q_seg=seg.numpy(),
              kv_seg=seg.numpy())
    m = oracle.block_mask(B, L, L, block_q=bq, block_kv=bk, **kw)
    vis = brute.visibility(B, L, L, **kw)
    nq, nk = L // bq, L // bk
    cnt = vis.reshape(B, nq, bq, nk, bk).sum(axis=(2, 4))
    cls = np.where(cnt == 0, 0, np.where(cnt == bq * bk, 2, 1)).astype(np.uint8)
    assert np.array_equal(m["tile_class"], cls)
    colcls = cls.transpose(0, 2, 1).reshape(B * nk, nq)
    for c in range(B * nk):
        nz = np.nonzero(colcls[c])[0]
        assert m["bwd_cnt"][c] == len(nz)
        assert np.array_equal(m["bwd_idx"][c][:len(nz)], nz)
        assert np.all(m["bwd_idx"][c][len(nz):] == -1)
    rowcls = cls.reshape(B * nq, nk)
    for r in range(B * nq):
        assert m["fwd_cnt"][r] == np.count_nonzero(rowcls[r])
    assert np.array_equal(m["bwd_order"], np.lexsort((np.arange(B * nk), -m["bwd_cnt"])))
    # halving the query blocks splits each 128-row class: a 128 x bk block is
    # EMPTY iff both halves are, FULL iff both are
    if (bq, bk) == (64, 128):
        m128 = oracle.block_mask(B, L, L, **kw)["tile_class"]
        halves = cls.reshape(B, nq // 2, 2, nk)
        assert np.array_equal(m128 == 0, np.all(halves == 0, axis=2))
        assert np.array_equal(m128 == 2, np.all(halves == 2, axis=2))


# ------------------------------------------------------------ permutation
@pytest.mark.parametrize("dtype", [np.uint8, np.int32, np.float32, np.float64])
@pytest.mark.parametrize("n", [1, 2, 8])
def test_permute_roundtrip_and_formula(dtype, n):
    L = 64
    rng = np.random.default_rng(n)
    x = (rng.normal(size=(3, L, 5)) * 100).astype(dtype)
    y = oracle.permute(x, n)
    assert np.array_equal(oracle.unpermute(y, n), x)
    c = L // (2 * n)
    for p in range(L):
        d, r = divmod(p, L // n)
        src = d * c + r if r < c else (2 * n - 1 - d) * c + (r - c)
        assert np.array_equal(y[:, p], x[:, src])


@pytest.mark.parametrize("ex", GOLD["ring_order"], ids=lambda e: f"n{e['n_shards']}")
def test_golden_ring_order(ex):
    n = ex["n_shards"]
    got = [[oracle.ring_source(d, t, n) for t in range(n)] for d in range(n)]
    assert got == ex["source"]


def test_row_and_head_restriction_equals_full():
    """Restricted runs (used to sample large workloads) agree with the full oracle on
    the rows / heads they compute, and the row contributions add up to the full gradient."""
    q, k, v, kw = _case(41, B=1, L=96, Hq=4, Hkv=2, D=8, segs=True, sinks=True, cap=2.0)
    o, l = oracle.attn_fwd(q, k, v, **kw)
    o2, l2 = oracle.attn_fwd(q, k, v, heads=(1, 3), rows=(17, 60), **kw)
    np.testing.assert_array_equal(o2[:, 17:60, 1:3], o[:, 17:60, 1:3])
    np.testing.assert_array_equal(l2[:, 1:3, 17:60], l[:, 1:3, 17:60])
    assert np.all(o2[:, :17] == 0) and np.all(np.isneginf(l2[:, 0]))
    do = np.random.default_rng(2).normal(size=q.shape)
    full = oracle.attn_bwd(q, k, v, do, **kw)
    parts = [oracle.attn_bwd(q, k, v, do, rows=r, heads=hh, **kw)
             for r in ((0, 50), (50, 96)) for hh in ((0, 1), (1, 4))]
    for t in range(4):
        np.testing.assert_allclose(sum(pp[t] for pp in parts), full[t], atol=1e-12)
    # key ranges split the pair sums the same way (dsinks, a sum over rows, is
    # the same in every key-restricted call)
    kparts = [oracle.attn_bwd(q, k, v, do, keys=kr, **kw) for kr in ((0, 40), (40, 96))]
    for t in range(3):
        np.testing.assert_allclose(sum(pp[t] for pp in kparts), full[t], atol=1e-12)
    np.testing.assert_array_equal(kparts[0][3], full[3])
    assert np.all(kparts[0][1][:, 40:] == 0) and np.all(kparts[1][2][:, :40] == 0)


# ------------------------------------------------- local mask (non-causal ring)
def _local_mask(seed, ls, lk=None, density=0.5):
    rng = np.random.default_rng(seed)
    lk = ls if lk is None else lk
    return (rng.random((ls, lk)) < density).astype(np.uint8)


LOCAL_CASES = [
    dict(n=2),
    dict(n=4, segs=True, pad=10),
    dict(n=2, sinks=True, cap=2.0),
    dict(n=3, Hq=4, Hkv=1),
    dict(n=1, segs=True),
]


@pytest.mark.parametrize("ci", range(len(LOCAL_CASES)))
def test_local_mask_equals_bruteforce_and_ring(ci):
    case = dict(LOCAL_CASES[ci])
    n = case.pop("n")
    case.setdefault("L", 96)
    q, k, v, kw = _case(500 + ci, causal=False, **case)
    lm = _local_mask(ci, case["L"] // n)
    kw["local_mask"] = lm
    o1, l1 = oracle.attn_fwd(q, k, v, **kw)
    o2, l2 = brute.attention(q, k, v, **kw)
    assert np.array_equal(np.isfinite(l1), np.isfinite(l2))
    f = np.isfinite(l2)
    np.testing.assert_allclose(l1[f], l2[f], atol=1e-12, rtol=0)
    np.testing.assert_allclose(o1, o2, atol=1e-12, rtol=0)
    # the ring over n shards with the mask applied at every step == plain
    o3, l3 = oracle.attn_fwd_ring(q, k, v, n_shards=n, **kw)
    np.testing.assert_allclose(l3[f], l1[f], atol=1e-12, rtol=0)
    np.testing.assert_allclose(o3, o1, atol=1e-12, rtol=0)


def test_local_mask_special_cases():
    q, k, v, kw = _case(601, L=64, causal=False)
    # an all-ones local mask is no mask at all
    ones = np.ones((32, 32), np.uint8)
    o0, l0 = oracle.attn_fwd(q, k, v, **kw)
    o1, l1 = oracle.attn_fwd(q, k, v, local_mask=ones, **kw)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    # one shard with a lower-triangular local mask is the causal mask
    tri = np.tril(np.ones((64, 64), np.uint8))
    o2, l2 = oracle.attn_fwd(q, k, v, local_mask=tri, **kw)
    kc = dict(kw, causal=True)
    o3, l3 = oracle.attn_fwd(q, k, v, **kc)
    assert np.array_equal(o2, o3) and np.array_equal(l2, l3)
    # with two shards the triangle repeats per block: query row 40 (local
    # row 8 of shard 1) sees keys 0..8 of shard 0 and 32..40 of shard 1
    tri2 = np.tril(np.ones((32, 32), np.uint8))
    vis = brute.visibility(1, 64, 64, causal=False, local_mask=tri2)[0]
    assert np.nonzero(vis[40])[0].tolist() == list(range(0, 9)) + list(range(32, 41))


def test_local_mask_gradients_central_differences():
    q, k, v, kw = _case(602, B=1, L=24, D=4, causal=False, sinks=True)
    kw["local_mask"] = _local_mask(7, 12)
    do = np.random.default_rng(5).normal(size=q.shape)
    dq, dk, dv, ds, _, _ = oracle.attn_bwd(q, k, v, do, **kw)

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd(q_, k_, v_, **kw)
        return float(np.sum(o * do))

    rng = np.random.default_rng(9)
    h = 1e-5
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(10):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            ap, am = arr.copy(), arr.copy()
            ap[idx] += h
            am[idx] -= h
            args_p = {"q": (ap, k, v), "k": (q, ap, v), "v": (q, k, ap)}[name]
            args_m = {"q": (am, k, v), "k": (q, am, v), "v": (q, k, am)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


@pytest.mark.parametrize("n", [1, 2, 4])
def test_local_mask_block_map_bruteforce(n):
    g = torch.Generator().manual_seed(40 + n)
    B, L = 2, 512
    seg, pos = random_structure(g, B, L, n_docs_max=3, pad_max=100)
    ls = L // n
    # banded local mask (a sliding window) with a random hole pattern
    i = np.arange(ls)[:, None]
    j = np.arange(ls)[None, :]
    lm = ((np.abs(i - j) < 150) & (_local_mask(n, ls, density=0.97) != 0)).astype(np.uint8)
    kw = dict(causal=False, q_pos=pos.numpy(), kv_pos=pos.numpy(), q_seg=seg.numpy(),
              kv_seg=seg.numpy(), local_mask=lm)
    m = oracle.block_mask(B, L, L, **kw)
    assert np.array_equal(m["tile_class"], _brute_map(B, L, **kw))
