"""Throughput of block-sparse masked attention with the virtual-ring LSE merge.

One step is one pass of the whole hot path over one batch of synthetic input:
zigzag-permute q, k, v, dO and positions -> build the block map -> forward
(ring over N virtual shards, fused merge) -> unpermute out and lse ->
backward (Delta/dsinks, dK/dV, dQ) -> unpermute dq, dk, dv.

Metric: masked-attention TFLOP/s counted over non-empty 128 x 128 tiles
(4 * 128 * 128 * D per tile and query head forward, x3.5 forward+backward),
and its fraction of the dense bf16 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload gqa32k] [--no-cpu-baseline] [--no-e2e]

With N > 1 (launched by torchrun) every rank runs its own batch on its own
GPU (weak scaling, no collective on the data path); the step time is the
max over ranks.  ``--impl reference`` times the fp64 CPU oracle on the host
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "masked-attention TFLOP/s fwd and fwd+bwd (unmasked tiles) and % BF16 tensor peak"
UNIT = "TFLOP/s"

# DRAM traffic per launch of each kernel from an ncu capture (bytes), keyed by
# (workload, kernel), with the hash of the sources the kernel is compiled from
# (_src_hash); a changed source, or another workload, reports null.
TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one launch, ncu on the gqa32k bench step
    ("gqa32k", "fwd2_tc_kernel"): (0.671e9 + 0.572e9, "36db991536e00879"),
    ("gqa32k", "bwd_dkdv_kernel"): (1.695e9 + 0.120e9, "f4257c54327ebfb9"),
    ("gqa32k", "bwd_dq_kernel"): (0.715e9 + 0.242e9, "f4257c54327ebfb9"),
}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _src_hash(name):
    """sha256 (first 16 hex) of a kernel source and the headers it includes."""
    csrc = os.path.join(ROOT, "block_sparse_flash_ra_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in (name, "ra_sched.cuh", "ra_device.cuh", "ra_internal.h")]
    files.append(os.path.join(ROOT, "include", "ra.h"))
    h = hashlib.sha256()
    try:
        for f in files:
            with open(f, "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return h.hexdigest()[:16]


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---- multi-rank logic (weak scaling: every rank runs its own batch of the
# workload, the data path has no collective; only the timing is reduced)
def rank_workload(w, rank):
    """The batch rank `rank` processes: same shapes, its own input seed."""
    return w.scaled(seed=w.seed + rank, backward=True)


def max_over_ranks(x, ws_):
    """Max of a per-rank float over all ranks (the slowest rank's time)."""
    if ws_ <= 1:
        return float(x)
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank, ms_max, ws_):
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return flops_per_rank * ws_ / (ms_max * 1e-3) / 1e12


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.dev = device
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.sel = str(device)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm
class Pipeline:
    """Device buffers and the hot-path step of one workload on one GPU."""

    def __init__(self, w, seed_offset=0):
        import block_sparse_flash_ra_gb300 as ra
        self.ra = ra
        self.w = w
        inp = make_inputs(rank_workload(w, seed_offset), with_dout=True)
        self.host = inp
        self.dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        N, B, L = w.n_shards, w.B, w.L
        d = self.dev
        self.perm = {k: torch.empty_like(d[k]) for k in ("q", "k", "v", "dout")}
        for k in ("q_pos", "kv_pos", "q_seg", "kv_seg"):
            self.perm[k] = torch.empty_like(d[k]) if d[k] is not None else None
        self.out = torch.empty_like(d["q"])
        self.lse = torch.empty((B, w.Hq, L), dtype=torch.float32, device="cuda")
        self.dq, self.dk, self.dv = (torch.empty_like(d[k]) for k in ("q", "k", "v"))
        self.final = {k: torch.empty_like(getattr(self, k)) for k in ("out", "lse", "dq", "dk", "dv")}
        self.dsinks = torch.empty(w.Hq, dtype=torch.float32, device="cuda") if d["sinks"] is not None else None
        src = self.perm if w.zigzag else d
        self.params = ra.make_params(
            d["q"], d["k"], scale=w.scale, causal=w.causal, soft_cap=w.soft_cap, n_virtual_shards=N,
            is_mqa=w.is_mqa, q_pos=src["q_pos"], kv_pos=src["kv_pos"], q_seg=src["q_seg"],
            kv_seg=src["kv_seg"], sinks=d["sinks"], local_mask=d["local_mask"])
        self.mask_buf = torch.empty(ra.ra_block_mask_bytes(self.params), dtype=torch.uint8, device="cuda")
        self.ws = torch.empty(ra.ra_attn_bwd_workspace_size(self.params), dtype=torch.uint8, device="cuda")
        n_fws = ra.ra_attn_fwd_workspace_size(self.params)
        self.fws = torch.empty(n_fws, dtype=torch.uint8, device="cuda") if n_fws else None
        self.mask = ra.RaBlockMask()
        self.names = ["permute", "mask", "fwd", "unpermute_fwd", "bwd_prep", "bwd_dkdv", "bwd_dq",
                      "unpermute_bwd"]
        # count non-empty tiles once (host read, outside any timed region)
        self._prepare_inputs()
        ra.ra_build_block_mask(self.params, self.mask_buf, self.mask)
        torch.cuda.synchronize()
        nq = L // 128
        off = self.mask.fwd_cnt - self.mask_buf.data_ptr()
        cnt = self.mask_buf[off:off + 4 * B * nq].view(torch.int32).cpu().numpy()
        self.tiles = int(cnt.sum()) * w.Hq           # non-empty (q tile, kv tile, head) triples
        self.f_fwd = float(self.tiles) * 4 * 128 * 128 * w.D
        self.f_fwd_bwd = 3.5 * self.f_fwd

    def _prepare_inputs(self):
        ra, w, d, p = self.ra, self.w, self.dev, self.perm
        N, B, L = w.n_shards, w.B, w.L
        if not w.zigzag:
            for k in ("q", "k", "v", "dout"):
                p[k] = d[k]
            return
        for k in ("q", "k", "v", "dout"):
            t = d[k]
            ra.ra_permute_tokens(t, p[k], B, L, t[0, 0].numel() * t.element_size(), N)
        for k in ("q_pos", "kv_pos", "q_seg", "kv_seg"):
            if d[k] is not None:
                ra.ra_permute_tokens(d[k], p[k], B, L, 4, N)

    def step(self, ev=None):
        """One pass of the hot path; ev: dict name -> (start, end) CUDA events."""
        ra, w, p = self.ra, self.w, self.perm
        N, B, L, H = w.n_shards, w.B, w.L, w.Hq

        def mark(name, i):
            if ev is not None:
                ev[name][i].record()

        mark("permute", 0)
        self._prepare_inputs()
        mark("permute", 1)
        mark("mask", 0)
        ra.ra_build_block_mask(self.params, self.mask_buf, self.mask)
        mark("mask", 1)
        mark("fwd", 0)
        ra.ra_attn_fwd(self.params, p["q"], p["k"], p["v"], self.mask, self.out, self.lse, ws=self.fws)
        mark("fwd", 1)
        mark("unpermute_fwd", 0)
        if w.zigzag:
            ra.ra_unpermute_tokens(self.out, self.final["out"], B, L, H * w.D * 2, N)
            ra.ra_unpermute_tokens(self.lse, self.final["lse"], B * H, L, 4, N)
        mark("unpermute_fwd", 1)
        mark("bwd_prep", 0)
        ra.ra_attn_bwd_prep(self.params, self.out, self.lse, p["dout"], self.dsinks, self.ws)
        mark("bwd_prep", 1)
        mark("bwd_dkdv", 0)
        ra.ra_attn_bwd_dkdv(self.params, p["q"], p["k"], p["v"], p["dout"], self.mask,
                            self.dk, self.dv, self.ws)
        mark("bwd_dkdv", 1)
        mark("bwd_dq", 0)
        ra.ra_attn_bwd_dq(self.params, p["q"], p["k"], p["v"], p["dout"], self.mask,
                          self.dq, self.ws)
        mark("bwd_dq", 1)
        mark("unpermute_bwd", 0)
        if w.zigzag:
            for k in ("dq", "dk", "dv"):
                t = getattr(self, k)
                ra.ra_unpermute_tokens(t, self.final[k], B, L, t[0, 0].numel() * 2, N)
        mark("unpermute_bwd", 1)




def time_merge(w, reps=10):
    """Mean time of one standalone ra_merge_out_lse over the workload's (B, L,
    Hq, D) fp32 output and (B, Hq, L) lse -- the ring update as its own call --
    with inputs larger than L2, after 3 untimed calls."""
    import block_sparse_flash_ra_gb300 as ra
    B, L, H, D = w.B, w.L, w.Hq, w.D
    g = torch.Generator(device="cuda").manual_seed(7)
    out = torch.randn((B, L, H, D), device="cuda", generator=g)
    bout = torch.randn((B, L, H, D), device="cuda", generator=g)
    lse = torch.randn((B, H, L), device="cuda", generator=g)
    blse = torch.randn((B, H, L), device="cuda", generator=g)
    for _ in range(3):
        ra.ra_merge_out_lse(out, lse, bout, blse, B, L, H, D)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(reps):
        ra.ra_merge_out_lse(out, lse, bout, blse, B, L, H, D)
    e.record()
    torch.cuda.synchronize()
    nbytes = 3 * out.numel() * 4 + 3 * lse.numel() * 4  # out read + written, block_out read; same for lse
    return s.elapsed_time(e) / reps, nbytes


def hbm_kernels(pipe, per, peaks, peak_kind):
    """Achieved bandwidth of the memory-bound stages of the step (algorithmic
    bytes over their CUDA-event time) and of the standalone merge call,
    against the measured HBM copy bandwidth."""
    w, d = pipe.w, pipe.dev
    tb = lambda t: 0 if t is None else t.numel() * t.element_size()  # noqa: E731
    pos = sum(tb(d[k]) for k in ("q_pos", "kv_pos", "q_seg", "kv_seg"))
    stages = {
        # every token row of q, k, v, dO (and positions / segments) read and written once
        "permute": (per["permute"], 2 * (sum(tb(d[k]) for k in ("q", "k", "v", "dout")) + pos))
        if w.zigzag else None,
        "unpermute_fwd": (per["unpermute_fwd"], 2 * (tb(pipe.out) + tb(pipe.lse))) if w.zigzag else None,
        "unpermute_bwd": (per["unpermute_bwd"], 2 * (tb(pipe.dq) + tb(pipe.dk) + tb(pipe.dv)))
        if w.zigzag else None,
        # O and dO read, lse read, Delta and -lse*log2 e written
        "bwd_prep": (per["bwd_prep"], tb(pipe.out) + tb(pipe.dev["dout"]) + 3 * tb(pipe.lse)),
        # positions and segments read, one class byte per tile written (lists and
        # orders add a few MB): kilobytes to megabytes, so the stage is launch-bound
        "mask": (per["mask"], pos + w.B * (w.L // 128) ** 2),
    }
    mm, mb = time_merge(w)
    stages["merge_out_lse"] = (mm, mb)
    hbm = peaks["hbm_gbs"]
    r = {"peak_gbs": hbm, "peak_kind": f"hbm_gbs ({peak_kind})"}
    for k, v in stages.items():
        if v is None:
            continue
        ms, nb = v
        gbs = nb / (ms * 1e-3) / 1e9
        r[k] = {"ms": round(ms, 4), "bytes": int(nb), "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4)}
    return r


def run_ours(args, w, ws_, rank, local):
    import block_sparse_flash_ra_gb300 as ra
    torch.cuda.set_device(local)
    pipe = Pipeline(w, seed_offset=rank)
    K, W = args.steps, args.warmup
    for _ in range(W):
        pipe.step()
    torch.cuda.synchronize()
    if ra.ra_get_device_status() != ra.RA_OK:
        raise RuntimeError("device status after warm-up: " + ra.ra_last_error())
    ev = {n: [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
          for n in pipe.names}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws_ > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    n0 = ra.ra_launch_count()
    with Clocks(local) as clk:
        t_wall = time.perf_counter()
        start.record()
        for i in range(K):
            pipe.step({n: ev[n][i] for n in pipe.names})
        end.record()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    launches = ra.ra_launch_count() - n0
    if ws_ > 1:
        torch.distributed.barrier()
    ms_total = start.elapsed_time(end)
    per = {n: sum(ev[n][i][0].elapsed_time(ev[n][i][1]) for i in range(K)) / K for n in pipe.names}
    if ra.ra_get_device_status() != ra.RA_OK:
        raise RuntimeError("device status after timing: " + ra.ra_last_error())
    ms_step = max_over_ranks(ms_total / K, ws_)

    # end to end through the C ABI with host buffers: H2D inputs, step, D2H results
    e2e = None
    if not args.no_e2e:
        # as many steps as the device-timed loop: the first upload and the last
        # download, which nothing overlaps, weigh 1/K of the region
        e2e = run_e2e(pipe, max(3, K), ws_, rank)

    peaks, peak_kind = _peaks()
    tf = lambda flops, ms: flops / (ms * 1e-3) / 1e12  # noqa: E731
    bwd_ms = per["bwd_prep"] + per["bwd_dkdv"] + per["bwd_dq"]
    # the forward runs two query heads per CTA when it has its workspace
    fwd_name, fwd_src = (("fwd2_tc_kernel", "k_attn_fwd2_tc.cu") if pipe.fws is not None
                         else ("fwd_tc_kernel", "k_attn_fwd_tc.cu"))
    kern = {
        fwd_name: (per["fwd"], pipe.f_fwd, fwd_src),
        "bwd_dkdv_kernel": (per["bwd_dkdv"], 2.0 * pipe.f_fwd, "k_attn_bwd_tc.cu"),
        "bwd_dq_kernel": (per["bwd_dq"], 1.5 * pipe.f_fwd, "k_attn_bwd_tc.cu"),
    }
    dom = max(kern, key=lambda k: kern[k][0])
    d_ms, d_flops, d_src = kern[dom]
    achieved = tf(d_flops, d_ms)
    # the timed region is well under a second (K steps of tens of ms), so the
    # kernels are held to the burst peak, not the seconds-long sustained one
    peak = peaks["bf16_tflops"]
    # the backward as the method counts it: F_bwd = 2.5 F_fwd (five tile
    # products against the forward's two) over the dK/dV and dQ kernels' time,
    # whatever products the kernels recompute
    bwd_alg = tf(2.5 * pipe.f_fwd, per["bwd_dkdv"] + per["bwd_dq"])
    tr = TRAFFIC.get((w.name, dom))
    traffic = tr[0] if tr and tr[1] == _src_hash(d_src) else None
    value = job_tflops(pipe.f_fwd_bwd, ms_step, ws_)
    fwd_tf = tf(pipe.f_fwd, per["fwd"])
    fb_tf = tf(pipe.f_fwd_bwd, per["fwd"] + bwd_ms)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws_, "steps": K,
        "warmup": W, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B * ws_, "B_per_gpu": w.B, "L": w.L, "Hq": w.Hq,
                   "Hkv": w.Hkv, "D": w.D, "causal": w.causal, "n_virtual_shards": w.n_shards,
                   "zigzag": w.zigzag, "soft_cap": w.soft_cap, "sinks": w.sinks,
                   "parallelism": f"dp{ws_}" if ws_ > 1 else "single",
                   "l2": "no flush; inputs larger than L2 (q+k+v+dO = "
                         f"{sum(pipe.dev[k].numel() * pipe.dev[k].element_size() for k in ('q', 'k', 'v', 'dout')) / 1e6:.0f} MB > 129 MB)",
                   "flops_fwd_per_step": pipe.f_fwd, "flops_fwd_bwd_per_step": pipe.f_fwd_bwd,
                   "nonempty_tile_heads": pipe.tiles},
        "fwd_tflops": round(fwd_tf, 2),
        "fwd_pct_peak": round(100 * fwd_tf / peaks["bf16_tflops"], 2),
        "fwd_bwd_kernel_tflops": round(fb_tf, 2),
        "fwd_bwd_pct_peak": round(100 * fb_tf / peaks["bf16_tflops"], 2),
        "pct_peak_of": f"bf16_tflops {peaks['bf16_tflops']} ({peak_kind})",
        "ms_per_stage": {n: round(v, 4) for n, v in per.items()},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "peak_kind": f"bf16_tflops burst ({peak_kind}): the timed region is "
                                  f"{K * ms_step / 1e3:.2f} s, not a seconds-long run",
                     "counted": "products the kernel issues (the dK/dV kernel's four per tile "
                                "are all algorithmic)",
                     "algorithmic": {
                         fwd_name: {"achieved": round(fwd_tf, 2),
                                           "frac": round(fwd_tf / peak, 4),
                                           "flops": "F_fwd = 4*128*128*D per non-empty tile-head"},
                         "backward": {"achieved": round(bwd_alg, 2), "frac": round(bwd_alg / peak, 4),
                                      "flops": "F_bwd = 2.5 F_fwd over the dK/dV + dQ kernels' time"},
                     }},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "wall_s_timed": round(t_wall, 3),
    }
    if e2e is not None:
        line["e2e"] = e2e
    line["hbm_kernels"] = hbm_kernels(pipe, per, peaks, peak_kind)
    return line, pipe


def run_e2e(pipe, K, ws_, rank=0):
    """End to end through the C ABI with host buffers: every step copies its
    inputs host -> device (pinned), runs the hot path and copies O, lse, dq,
    dk, dv back.  Two sets of device buffers and separate copy streams let
    step i+1's input copy and step i-1's result copy overlap step i's
    compute, as a serving loop would; each step still moves its own bytes."""
    w = pipe.w
    pipes = [pipe, Pipeline(w, seed_offset=rank)]
    host_in = {k: pipe.host[k].pin_memory() for k in ("q", "k", "v", "dout")}
    for k in ("q_pos", "kv_pos", "q_seg", "kv_seg"):
        if pipe.host[k] is not None:
            host_in[k] = pipe.host[k].pin_memory()
    host_out = [{k: torch.empty(pp.final[k].shape, dtype=pp.final[k].dtype, pin_memory=True)
                 for k in ("out", "lse", "dq", "dk", "dv")} for pp in pipes]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    comp, up, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    computed = [torch.cuda.Event() for _ in pipes]   # step done on buffer set j
    fetched = [torch.cuda.Event() for _ in pipes]    # its results copied out
    used = [False, False]

    def one(i):
        j = i % 2
        pp = pipes[j]
        src = pp.final if w.zigzag else {"out": pp.out, "lse": pp.lse, "dq": pp.dq,
                                         "dk": pp.dk, "dv": pp.dv}
        loaded = torch.cuda.Event()
        with torch.cuda.stream(up):
            if used[j]:
                up.wait_event(computed[j])     # the previous step on this set read its inputs
            for k, t in host_in.items():
                pp.dev[k].copy_(t, non_blocking=True)
            loaded.record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(loaded)
            if used[j]:
                comp.wait_event(fetched[j])    # its results are out before they are overwritten
            pp.step()
            computed[j].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[j])
            for k, t in host_out[j].items():
                t.copy_(src[k], non_blocking=True)
            fetched[j].record(down)
        used[j] = True

    one(0)
    one(1)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws_ > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(torch.cuda.current_device()) as clk:
        s.record(up)
        for i in range(K):
            one(i)
        # the region ends when the last results are on the host
        for st in (up, comp):
            down.wait_stream(st)
        e.record(down)
        torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e) / K, ws_)
    v = job_tflops(pipe.f_fwd_bwd, ms, ws_)
    return {"value": round(v, 2), "unit": UNIT, "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": K,
            "overlap": "input copy of step i+1 and result copy of step i-1 overlap step i",
            "clocks": clk.summary()}


# ---------------------------------------------------------------- oracle
def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_sample(w, rows):
    """fp64 oracle forward + backward on a bounded sample of the workload: the
    first query head of every kv group (Hkv heads, with their kv heads) and
    query rows [L - rows, L), in the original token order (the ring order
    changes rounding only).  Returns (seconds, counted flops, heads, threads
    that ran work)."""
    import oracle
    inp = make_inputs(w.scaled(backward=True), with_dout=True)
    G = w.Hq // w.Hkv
    f = lambda t: None if t is None else t.to(torch.float64).numpy()  # noqa: E731
    i = lambda t: None if t is None else t.numpy()  # noqa: E731
    sl = lambda t: None if t is None else t[:, :, ::G].contiguous()  # noqa: E731
    kw = dict(scale=w.scale, soft_cap=w.soft_cap or None, causal=w.causal, q_pos=i(inp["q_pos"]),
              kv_pos=i(inp["kv_pos"]), q_seg=i(inp["q_seg"]), kv_seg=i(inp["kv_seg"]),
              sinks=None if inp["sinks"] is None else f(inp["sinks"][::G]),
              local_mask=i(inp["local_mask"]))
    q, do = f(sl(inp["q"])), f(sl(inp["dout"]))
    k, v = f(inp["k"]), f(inp["v"])
    r0 = w.L - rows
    m = oracle.block_mask(w.B, w.L, w.L, causal=w.causal, q_pos=kw["q_pos"], kv_pos=kw["kv_pos"],
                          q_seg=kw["q_seg"], kv_seg=kw["kv_seg"], local_mask=kw["local_mask"])
    nq = w.L // 128
    tiles = int(sum(m["fwd_cnt"][b * nq + qt] for b in range(w.B) for qt in range(r0 // 128, nq)))
    flops = 3.5 * tiles * w.Hkv * 4 * 128 * 128 * w.D
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, rows=(r0, w.L), **kw)
    used = oracle.last_threads()
    oracle.attn_bwd(q, k, v, do, rows=(r0, w.L), **kw)
    used = max(used, oracle.last_threads())
    return time.perf_counter() - t0, flops, w.Hkv, used


def cpu_baseline(w, rows):
    import oracle
    oracle.build()
    secs, flops, heads, used = _oracle_sample(w, rows)
    return {"value": round(flops / secs / 1e12, 6), "unit": UNIT, "cores": used,
            "kind": "oracle",
            "sample": f"{w.name}: {heads} of {w.Hq} query heads (one per kv group), query rows "
                      f"[{w.L - rows}, {w.L}) of {w.L}, batch {w.B}; fp64 forward (threads over "
                      f"blocks of query rows) + backward (threads over blocks of query rows, then "
                      f"of keys), {secs:.2f} s for {flops:.3e} counted flops; {used} of "
                      f"{oracle.num_threads()} host threads ran work"}


def run_reference(args, w):
    import oracle
    oracle.build()
    rows = args.ref_rows
    for _ in range(args.warmup):
        _oracle_sample(w, rows)
    times, flops, heads, cores = [], 0.0, 0, 1
    for _ in range(args.steps):
        s, flops, heads, used = _oracle_sample(w, rows)
        times.append(s)
        cores = max(cores, used)
    sec = sum(times) / len(times)
    v = flops / sec / 1e12
    sample = (f"{w.name}: {heads} of {w.Hq} query heads (one per kv group), query rows "
              f"[{w.L - rows}, {w.L}) of {w.L}, fp64 forward + backward per step")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": w.B, "L": w.L, "Hq": w.Hq,
                                            "Hkv": w.Hkv, "D": w.D, "sample_rows": rows},
            "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa32k", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=512,
                    help="query rows of the oracle sample for cpu_baseline")
    ap.add_argument("--ref-rows", type=int, default=128,
                    help="query rows of the oracle sample per reference step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    ws_, rank, local = _dist()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return

    if ws_ > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    from block_sparse_flash_ra_gb300 import _build
    if rank == 0 or ws_ == 1:
        _build.build()
    if ws_ > 1:
        torch.distributed.barrier()
    line, _ = run_ours(args, w, ws_, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and ws_ == 1:
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_rows)
        print(json.dumps(line), flush=True)
    if ws_ > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
