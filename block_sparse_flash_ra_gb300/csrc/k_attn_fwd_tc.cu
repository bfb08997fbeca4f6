// k_attn_fwd_tc.cu -- block-sparse flash attention forward on the 5th-gen
// tensor cores (tcgen05 + TMEM, TMA-fed), with the ring (out, lse) merge
// fused into the epilogue of every virtual shard.
//
// What it computes ("ejKernel ring_attention._ring_splash" module source,
// _ring_attention_forward and _update_out_and_lse; Kvax "Flash Attention for
// JAX", flash_attention): for each (b, h, 128-row query tile) on virtual
// device d, the KV shards are visited in ring order s = (d - t) mod N; inside
// a shard the non-empty 128-row KV tiles of the block map are processed with
// an online softmax (S = Q K^T on tensor cores, scale, soft cap, mask of
// partial tiles, P = exp2(S - m) in bf16, O_acc += P V on tensor cores); at
// the shard's end the partial (O_s = O_acc / l, lse_s) -- with the sink in
// the denominator at t = 0 -- is merged into the running (O_run, lse_run) by
// the sigmoid/softplus update.  Output is bf16, lse fp32.
//
// Design (one CTA per SM, persistent, longest-row-first static schedule):
//   warps 0-7   softmax in two warpgroups that split the 128 columns of each
//               S row; the two threads of a query row exchange their row
//               maxima through shared memory (warp w may only touch TMEM
//               lanes 32(w%4)..+31).  At a shard's end they post their row
//               sums and the row max and go straight on to the next shard.
//   warps 8-11  correction warpgroup: the shard-end work of the ring --
//               normalise the shard's O_acc, add the sink (t = 0), merge it
//               into O_run with the sigmoid/softplus update, and at the
//               unit's end store bf16 O and lse -- one query row per thread,
//               overlapped with the softmax of the next shard's tiles
//   warp 12     TMA producer: Q once per work unit, K and V tiles into rings
//               of shared-memory stages (2 for K, 3 for V at D = 128)
//   warp 13     TMEM allocator and MMA issuer (the whole warp runs the issue
//               loop; one elected lane issues each product)
//   warps 14-15 no role (with warps 12-13 they form the warpgroup that hands
//               registers to the softmax warpgroups through setmaxnreg)
// TMEM (512 columns x 128 lanes, fp32):
//   [0,128)   S buffer 0   (P of the tile, bf16, overwrites columns [0,32)
//                           and [64,96): each half over columns it has read)
//   [128,256) S buffer 1
//   [256,256+D)      O_acc  shard accumulator
//   [256+D,256+2D)   O_run  running merged output of the ring
// MMA issue order per tile g: S(g) = Q K(g)^T, then O_acc += P(g-1) V(g-1),
// so the softmax of tile g overlaps the PV product of tile g-1.  The first PV
// product of a shard overwrites O_acc, so it waits until the correction
// warpgroup has read the previous shard's O_acc.  The O_acc rescale after a
// row-max increase is lazy (only when the max grows by more than 2^8) and
// waits for the previous PV product.
#include <math.h>

#include "ra_sched.cuh"

namespace ra {
namespace {

template <int D>
struct FwdCfg {
    static constexpr int kTileBytes = kTile * D * 2; // one 128-row bf16 tile
    // K tiles are consumed at once by S = Q K^T; V tiles wait for the softmax,
    // so the V ring is the deeper one
    static constexpr int kKStages = (D == 128) ? 2 : 3;
    static constexpr int kVStages = (D == 128) ? 3 : 4;
    static constexpr int kMaxStages = kVStages;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kTileBytes;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
    static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 5 + 1 + 4 + 2 + 2;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // row max exchange [2 tiles][2 halves][128], then the shard-end posts of
    // the softmax: row sums [2 slots][2 halves][128] and row max [2 slots][128]
    static constexpr int kXOff = kMiscOff + 16;
    static constexpr int kStatLOff = kXOff + 2 * 2 * 128 * 4;
    static constexpr int kStatMOff = kStatLOff + 2 * 2 * 128 * 4;
    static constexpr int kSmemUsed = kStatMOff + 2 * 128 * 4;
    static constexpr int kSmem = kSmemUsed + 1024; // slack for 1024-byte alignment
    static_assert(kSmem <= 232448, "forward shared memory exceeds the 227 KB per-block limit");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 256;
    static constexpr uint32_t kColRun = 256 + D;
    static constexpr uint32_t kIdescQK = idesc_bf16(128, 128, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16(128, D, false, true);
};

struct Bars {
    uint64_t *q_full, *q_empty, *k_full, *k_empty, *v_full, *v_empty, *s_full, *p_full, *pv_done,
        *drain, *xsync, *stat_full, *o_full, *o_empty;
};

template <int D>
__device__ __forceinline__ Bars carve_bars(uint8_t *smem)
{
    using C = FwdCfg<D>;
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    Bars r;
    r.q_full = b;
    r.q_empty = b + 1;
    r.k_full = b + 2;
    r.k_empty = r.k_full + C::kKStages;
    r.v_full = r.k_empty + C::kKStages;
    r.v_empty = r.v_full + C::kVStages;
    r.s_full = r.v_empty + C::kVStages;
    r.p_full = r.s_full + 2;
    r.pv_done = r.p_full + 2;
    r.drain = r.pv_done + 1;
    r.xsync = r.drain + 1;
    r.stat_full = r.xsync + 4; // [2]: shard-end posts of the softmax, per slot
    r.o_full = r.stat_full + 2; // a shard's last PV product has completed
    r.o_empty = r.o_full + 1;   // the correction warps have read O_acc
    return r;
}

// Work unit u -> (row id b*nq+qt from the longest-first order, head h).
struct Unit {
    int b, qt, h, row, cnt, dev;
    const int32_t *list;
    const int32_t *shard; // N+1 offsets into list: where each KV shard's tiles begin
    const int32_t *pfwd;  // N+1 row-order numbers of the first partial tile of each shard
};

__device__ __forceinline__ Unit unit_of(const Problem &p, int u)
{
    Unit x;
    x.row = p.fwd_order[u / p.Hq];
    x.h = u % p.Hq;
    x.b = x.row / p.nq;
    x.qt = x.row - x.b * p.nq;
    x.cnt = p.fwd_cnt[x.row];
    x.dev = x.qt / p.tq;
    x.list = p.fwd_idx + (size_t)x.row * p.nk;
    x.shard = p.fwd_shard + (size_t)x.row * (p.N + 1);
    x.pfwd = p.part_fwd + (size_t)x.row * (p.N + 1);
    return x;
}

// Range [lo, hi) of the unit's tile list that lies in KV shard `src`.
__device__ __forceinline__ void shard_range(const Problem &p, const Unit &x, int src, int &lo,
                                            int &hi)
{
    lo = x.shard[src];
    hi = x.shard[src + 1];
}

constexpr int kSoftmaxThreads = 256; // warps 0-7
constexpr int kCorrWarp0 = 8;        // warps 8-11
constexpr int kCorrThreads = 128;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kFwdThreads = 512;
// setmaxnreg split: 256 x 184 + 128 x 64 + 128 x 80 = 65536 = 512 x 128, the
// block's registers at launch (the kernel is built for 128 per thread; the
// launcher checks that count before the first launch)
constexpr int kLaunchRegs = 128;
constexpr uint32_t kSoftmaxRegs = 184;
constexpr uint32_t kCorrRegs = 64;
constexpr uint32_t kSideRegs = 80;
static_assert(256 * kSoftmaxRegs + 128 * kCorrRegs + 128 * kSideRegs <= kFwdThreads * kLaunchRegs,
              "register split exceeds the block's launch registers");

// Correction-warp work of one unit in ring-step mode (ra_attn_fwd_step):
// the chunk's partial (O_s, lse_s) -- (0, -inf) for an empty chunk, with the
// sink in the denominator when `sink_here` -- merged by the pages' update
// (_update_out_and_lse) into the running pair (p.run_out, p.run_lse) of this
// thread's query row, read from global memory (unless p.step_first: then the
// running pair is (0, -inf)) and written back; the bf16 `out`, if given, gets
// the merged row too.  O_s passes through TMEM columns [kColRun, +D) (idle in
// this mode), so that O_acc is released to the next unit as soon as it has
// been read.  Returns false when a wait gave up.
template <int D, typename WaitAll>
__device__ __forceinline__ bool step_merge(const Problem &p, const Unit &x, int row, int qi,
                                           uint32_t lane_base, const Bars &bars, const float *stat_l,
                                           const float *stat_m, uint32_t &nshard, uint32_t &n_of,
                                           bool sink_here, float sink2, __nv_bfloat16 *out,
                                           WaitAll &wait_all)
{
    using C = FwdCfg<D>;
    const size_t ro = (((size_t)x.b * p.Lq + qi) * p.Hq + x.h) * D;
    float *lrun = p.run_lse + ((size_t)x.b * p.Hq + x.h) * p.Lq + qi;
    const bool nonempty = x.cnt > 0; // uniform over the CTA
    float lse_s = sink_here ? sink2 * kLn2 : -INFINITY;
    if (nonempty) {
        const int slot = nshard & 1;
        if (!wait_all(bars.stat_full + slot, (nshard >> 1) & 1)) return false;
        ++nshard;
        float l = stat_l[slot * 256 + row] + stat_l[slot * 256 + 128 + row];
        const float m_ref = stat_m[slot * 128 + row];
        if (!wait_all(bars.o_full, n_of++ & 1)) return false;
        tc_fence_after();
        float m_fin = m_ref, fac = 1.f;
        if (sink_here) {
            m_fin = fmaxf(m_ref, sink2);
            fac = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_fin);
            l = l * fac + ex2_approx(sink2 - m_fin);
        }
        float inv = 0.f;
        if (l > 0.f) {
            lse_s = (m_fin + lg2_approx(l)) * kLn2;
            inv = fac * rcp_approx(l);
        } else {
            lse_s = -INFINITY;
        }
        // O_s = O_acc / l into the idle O_run columns; then O_acc is free
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
            float a[16];
            tmem_ld16(lane_base + C::kColO + c * 16, a);
            tmem_ld_wait();
            if (c == D / 16 - 1) {
                tc_fence_before();
                mbar_arrive(bars.o_empty);
            }
            uint32_t w16[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w16[j] = __float_as_uint(a[j] * inv);
            tmem_st16(lane_base + C::kColRun + c * 16, w16);
        }
        tmem_st_wait();
    }
    const float lse_in = p.step_first ? -INFINITY : *lrun;
    const bool first = lse_in == -INFINITY;
    const float w = first ? 1.f : sigmoid_fast(lse_s - lse_in);
    float *grow = p.run_out + ro;
    __nv_bfloat16 *orow = out ? out + ro : nullptr;
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
        float os[16];
        if (nonempty) {
            tmem_ld16(lane_base + C::kColRun + c * 16, os);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) os[j] = 0.f;
        }
        float4 *g4 = reinterpret_cast<float4 *>(grow + c * 16);
        float nv[16];
        if (first) {
#pragma unroll
            for (int j = 0; j < 16; ++j) nv[j] = os[j];
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 cv = g4[k];
                nv[4 * k + 0] = cv.x - w * (cv.x - os[4 * k + 0]);
                nv[4 * k + 1] = cv.y - w * (cv.y - os[4 * k + 1]);
                nv[4 * k + 2] = cv.z - w * (cv.z - os[4 * k + 2]);
                nv[4 * k + 3] = cv.w - w * (cv.w - os[4 * k + 3]);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            g4[k] = make_float4(nv[4 * k + 0], nv[4 * k + 1], nv[4 * k + 2], nv[4 * k + 3]);
        if (orow) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 16);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                uint4 v;
                v.x = pack_bf16x2(nv[8 * k + 0], nv[8 * k + 1]);
                v.y = pack_bf16x2(nv[8 * k + 2], nv[8 * k + 3]);
                v.z = pack_bf16x2(nv[8 * k + 4], nv[8 * k + 5]);
                v.w = pack_bf16x2(nv[8 * k + 6], nv[8 * k + 7]);
                dst[k] = v;
            }
        }
    }
    *lrun = first ? lse_s : lse_in + softplus_fast(lse_s - lse_in);
    return true;
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, Problem p,
                  __nv_bfloat16 *__restrict__ out, float *__restrict__ lse)
{
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const Bars bars = carve_bars<D>(smem);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
    const WaitCtx ctx{abort_flag, p.status, p.timeout_ns};
    float *stat_l = reinterpret_cast<float *>(smem + C::kStatLOff); // [2 slots][2 halves][128]
    float *stat_m = reinterpret_cast<float *>(smem + C::kStatMOff); // [2 slots][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = p.B * p.nq * p.Hq;
    const int G = gridDim.x;

    if (threadIdx.x == 0) {
        mbar_init(bars.q_full, 1);
        mbar_init(bars.q_empty, 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(bars.k_full + s, 1);
            mbar_init(bars.k_empty + s, 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(bars.v_full + s, 1);
            mbar_init(bars.v_empty + s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bars.s_full + s, 1);
            mbar_init(bars.p_full + s, kSoftmaxThreads);
            mbar_init(bars.stat_full + s, kSoftmaxThreads);
        }
        mbar_init(bars.pv_done, 1);
        mbar_init(bars.drain, 1);
        for (int q4 = 0; q4 < 4; ++q4) mbar_init(bars.xsync + q4, 64);
        mbar_init(bars.o_full, 1);
        mbar_init(bars.o_empty, kCorrThreads);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_holder, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp >= kProducerWarp) {
        regs_shrink<kSideRegs>();
        if (warp == kProducerWarp) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                uint32_t g = 0, uq = 0;
                uint32_t k_issued[C::kMaxStages] = {}, v_issued[C::kMaxStages] = {};
                bool ok = true;
                for (int r = 0; ok && r * G < U; ++r) {
                    const int u = unit_index(r, blockIdx.x, G);
                    if (u >= U) continue;
                    const Unit x = unit_of(p, u);
                    if (x.cnt == 0) continue;
                    if (!(ok = mbar_wait(bars.q_empty, (uq & 1) ^ 1, ctx))) break;
                    mbar_expect_tx(bars.q_full, C::kTileBytes);
                    for (int hb = 0; hb < D / 64; ++hb)
                        tma_load_4d(smem + C::kQOff + hb * 16384, &tm_q, bars.q_full, hb * 64, x.h,
                                    x.qt * kTile, x.b);
                    ++uq;
                    const int g_kv = x.h / p.G;
                    for (int t = 0; ok && t < p.N; ++t) {
                        int lo, hi;
                        shard_range(p, x, (x.dev - t + p.N) % p.N, lo, hi);
                        for (int e = lo; e < hi; ++e) {
                            const int kt = x.list[e];
                            const int sk = g % C::kKStages;
                            if (!(ok = mbar_wait(bars.k_empty + sk, ((g / C::kKStages) & 1) ^ 1, ctx))) break;
                            mbar_expect_tx(bars.k_full + sk, C::kTileBytes);
                            for (int hb = 0; hb < D / 64; ++hb)
                                tma_load_4d(smem + C::kKOff + sk * C::kTileBytes + hb * 16384, &tm_k,
                                            bars.k_full + sk, hb * 64, g_kv, kt * kTile, x.b);
                            ++k_issued[sk];
                            const int sv = g % C::kVStages;
                            if (!(ok = mbar_wait(bars.v_empty + sv, ((g / C::kVStages) & 1) ^ 1, ctx))) break;
                            mbar_expect_tx(bars.v_full + sv, C::kTileBytes);
                            for (int hb = 0; hb < D / 64; ++hb)
                                tma_load_4d(smem + C::kVOff + sv * C::kTileBytes + hb * 16384, &tm_v,
                                            bars.v_full + sv, hb * 64, g_kv, kt * kTile, x.b);
                            ++v_issued[sv];
                            ++g;
                        }
                    }
                }
                if (!ok) {
                    // let the copies already issued land before the CTA exits
                    for (int s = 0; s < C::kKStages; ++s)
                        if (k_issued[s]) wait_drain(bars.k_full + s, (k_issued[s] - 1) & 1, kDrainNs);
                    for (int s = 0; s < C::kVStages; ++s)
                        if (v_issued[s]) wait_drain(bars.v_full + s, (v_issued[s] - 1) & 1, kDrainNs);
                    if (uq) wait_drain(bars.q_full, (uq - 1) & 1, kDrainNs);
                }
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA issuer
            // The whole warp runs the issue loop, converged: every lane waits on
            // the barriers, and one lane, chosen by elect.sync, issues each
            // product and commit.
            {
                auto wait_w = [&](uint64_t *bar, uint32_t parity) -> bool {
                    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
                };
                // descriptors are built once per operand; an offset o adds o / 16
                const uint64_t qd = sdesc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
                const uint64_t kd0 = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
                const uint64_t vd0 = sdesc_sw128(smem_u32(smem + C::kVOff), 16384, 1024);
                constexpr uint32_t kStageStep = C::kTileBytes >> 4;
                uint32_t g = 0, uq = 0, n_oe = 0;
                bool have_prev = false, prev_first = false, prev_last = false;
                uint32_t prev_g = 0;
                bool ok = true;
                // PV product of tile pg; `first` / `last`: the tile opens / closes its shard
                auto issue_pv = [&](uint32_t pg, bool first, bool last) -> bool {
                    const int sb = pg & 1;
                    if (!wait_w(bars.p_full + sb, (pg >> 1) & 1)) return false;
                    const int st = pg % C::kVStages;
                    if (!wait_w(bars.v_full + st, (pg / C::kVStages) & 1)) return false;
                    // the shard's first product overwrites O_acc: the correction
                    // warps must have read the previous shard's
                    if (first && !wait_w(bars.o_empty, (n_oe++ & 1) ^ 1)) return false;
                    tc_fence_after();
                    const uint64_t vd = vd0 + (uint64_t)(st * kStageStep);
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk) {
                        const uint64_t bdesc = vd + (uint32_t)((kk * 2048) >> 4);
                        // P of kv rows 16kk..16kk+15: the half of warps 0-3 (kk < 4) sits
                        // in columns [0,32) of the S buffer, the other half in [64,96)
                        const uint32_t acol = sb * 128 + kk * 8 + (kk >= 4 ? 32 : 0);
                        mma_ts_w(tmem + C::kColO, tmem + acol, bdesc, C::kIdescPV,
                               (kk > 0 || !first) ? 1u : 0u);
                    }
                    tc_commit_w(bars.v_empty + st);
                    tc_commit_w(bars.pv_done);
                    if (last) tc_commit_w(bars.o_full);
                    return true;
                };
                for (int r = 0; ok && r * G < U; ++r) {
                    const int u = unit_index(r, blockIdx.x, G);
                    if (u >= U) continue;
                    const Unit x = unit_of(p, u);
                    if (x.cnt == 0) continue;
                    if (!(ok = wait_w(bars.q_full, uq & 1))) break;
                    tc_fence_after();
                    ++uq;
                    int done = 0;
                    for (int t = 0; ok && t < p.N; ++t) {
                        int lo, hi;
                        shard_range(p, x, (x.dev - t + p.N) % p.N, lo, hi);
                        for (int e = lo; e < hi; ++e) {
                            const int st = g % C::kKStages;
                            if (!(ok = wait_w(bars.k_full + st, (g / C::kKStages) & 1))) break;
                            tc_fence_after();
                            const int sb = g & 1;
                            const uint64_t kd = kd0 + (uint64_t)(st * kStageStep);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                                mma_ss_w(tmem + sb * 128, qd + o, kd + o, C::kIdescQK, kk > 0 ? 1u : 0u);
                            }
                            tc_commit_w(bars.k_empty + st);
                            tc_commit_w(bars.s_full + sb);
                            if (++done == x.cnt) tc_commit_w(bars.q_empty);
                            if (have_prev && !(ok = issue_pv(prev_g, prev_first, prev_last))) break;
                            have_prev = true;
                            prev_g = g;
                            prev_first = (e == lo);
                            prev_last = (e == hi - 1);
                            ++g;
                        }
                    }
                }
                if (ok && have_prev) ok = issue_pv(prev_g, prev_first, prev_last);
                // all issued MMAs must finish before TMEM is released
                tc_commit_w(bars.drain);
                wait_drain(bars.drain, 0, kDrainNs);
            }
        }
    } else if (warp >= kCorrWarp0) {
        regs_shrink<kCorrRegs>();
        // ------------------------------------------------------------ correction
        // Thread t owns query row t = TMEM lane t.  Per non-empty shard of a
        // unit, in ring order: wait for the softmax's row sums and row max and
        // for the shard's last PV product, form (O_s, lse_s) -- the sink in
        // the denominator at t = 0 -- and merge it into (O_run, lse_run) by
        // the sigmoid/softplus update (the unit's last non-empty shard stores
        // the merged row straight to the bf16 output); then the unit's lse.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t nshard = 0, n_of = 0;
        bool ok = true;
        auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
        };
        for (int r = 0; ok && r * G < U; ++r) {
            const int u = unit_index(r, blockIdx.x, G);
            if (u >= U) continue;
            const Unit x = unit_of(p, u);
            const int qi = x.qt * kTile + row;
            __nv_bfloat16 *orow = out + (((size_t)x.b * p.Lq + qi) * p.Hq + x.h) * D;
            float *lrow = lse + ((size_t)x.b * p.Hq + x.h) * p.Lq + qi;
            const bool has_sink = p.sinks != nullptr;
            const float sink2 = has_sink ? p.sinks[x.h] * kLog2e : 0.f;
            if (p.run_out) {
                // one ring step: merge this chunk's partial into the running
                // pair in global memory (one shard per unit, N == 1)
                if (!(ok = step_merge<D>(p, x, row, qi, lane_base, bars, stat_l, stat_m, nshard, n_of,
                                         has_sink && p.step_sink, sink2, out, wait_all)))
                    break;
                continue;
            }
            float lse_run = -INFINITY;
            bool orun_set = false;    // uniform: O_run columns hold this unit's data
            bool out_written = false; // uniform: the last merge stored the output itself
            int tiles_done = 0;
            if (x.cnt > 0) {
                for (int t = 0; ok && t < p.N; ++t) {
                    const int src = (x.dev - t + p.N) % p.N;
                    int lo, hi;
                    shard_range(p, x, src, lo, hi);
                    const bool sink_here = has_sink && t == 0;
                    if (lo == hi) {
                        // empty shard: partial is (0, -inf), or (0, sink) at t = 0
                        if (sink_here) {
                            const float ls = sink2 * kLn2;
                            lse_run = (lse_run == -INFINITY) ? ls : lse_run + softplus_fast(ls - lse_run);
                        }
                        continue;
                    }
                    tiles_done += hi - lo;
                    // the unit's last non-empty shard merges straight into the bf16 output
                    const bool last = tiles_done == x.cnt;
                    const int slot = nshard & 1;
                    if (!(ok = wait_all(bars.stat_full + slot, (nshard >> 1) & 1))) break;
                    ++nshard;
                    float l = stat_l[slot * 256 + row] + stat_l[slot * 256 + 128 + row];
                    const float m_ref = stat_m[slot * 128 + row];
                    if (!(ok = wait_all(bars.o_full, n_of++ & 1))) break;
                    tc_fence_after();
                    float m_fin = m_ref, fac = 1.f;
                    if (sink_here) {
                        m_fin = fmaxf(m_ref, sink2);
                        fac = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_fin);
                        l = l * fac + ex2_approx(sink2 - m_fin);
                    }
                    float lse_s, inv;
                    if (l > 0.f) {
                        lse_s = (m_fin + lg2_approx(l)) * kLn2;
                        inv = fac * rcp_approx(l);
                    } else {
                        lse_s = -INFINITY;
                        inv = 0.f;
                    }
                    const bool first = (lse_run == -INFINITY);
                    const float w = first ? 1.f : sigmoid_fast(lse_s - lse_run);
#pragma unroll
                    for (int c = 0; c < D / 16; ++c) {
                        float a[16], cur[16];
                        tmem_ld16(lane_base + C::kColO + c * 16, a);
                        if (orun_set) tmem_ld16(lane_base + C::kColRun + c * 16, cur);
                        tmem_ld_wait();
                        if (c == D / 16 - 1) {
                            // every column of O_acc is in registers: the next
                            // shard's first PV product may overwrite it
                            tc_fence_before();
                            mbar_arrive(bars.o_empty);
                        }
                        float nv[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float os = a[j] * inv;
                            const float cv = orun_set ? cur[j] : 0.f;
                            nv[j] = first ? os : cv - w * (cv - os);
                        }
                        if (last) {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 16);
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                uint4 v;
                                v.x = pack_bf16x2(nv[8 * k + 0], nv[8 * k + 1]);
                                v.y = pack_bf16x2(nv[8 * k + 2], nv[8 * k + 3]);
                                v.z = pack_bf16x2(nv[8 * k + 4], nv[8 * k + 5]);
                                v.w = pack_bf16x2(nv[8 * k + 6], nv[8 * k + 7]);
                                dst[k] = v;
                            }
                        } else {
                            uint32_t nw[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) nw[j] = __float_as_uint(nv[j]);
                            tmem_st16(lane_base + C::kColRun + c * 16, nw);
                        }
                    }
                    if (!last) tmem_st_wait();
                    out_written = last;
                    lse_run = first ? lse_s : lse_run + softplus_fast(lse_s - lse_run);
                    orun_set = true;
                }
                if (!ok) break;
            } else if (has_sink) {
                lse_run = sink2 * kLn2;
            }
            // ---- epilogue: O_run -> bf16 (unless the last merge stored it), lse
            if (out_written) {
            } else if (orun_set) {
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    float a[16];
                    tmem_ld16(lane_base + C::kColRun + c * 16, a);
                    tmem_ld_wait();
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 16);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        uint4 v;
                        v.x = pack_bf16x2(a[8 * k + 0], a[8 * k + 1]);
                        v.y = pack_bf16x2(a[8 * k + 2], a[8 * k + 3]);
                        v.z = pack_bf16x2(a[8 * k + 4], a[8 * k + 5]);
                        v.w = pack_bf16x2(a[8 * k + 6], a[8 * k + 7]);
                        dst[k] = v;
                    }
                }
            } else {
                uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
                for (int k = 0; k < D / 8; ++k) dst[k] = make_uint4(0, 0, 0, 0);
            }
            *lrow = lse_run;
        }
    } else {
        regs_grow<kSoftmaxRegs>();
        // ------------------------------------------------------------ softmax
        // Two warpgroups split the 128 S columns of every query row: warps
        // 0-3 take columns 0-63, warps 4-7 columns 64-127.  Warp w may only
        // touch TMEM lanes 32*(w%4)..+31, so thread t of both groups owns
        // query row 32*(w%4) + lane.  Row maxima are exchanged between the
        // two threads of a row through shared memory.
        const int wg = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int c0 = wg * 64;                 // first S column of this half
        constexpr int kOH = D / 2;              // O columns of this half
        const uint32_t o_col = wg * kOH;
        float *xmax = reinterpret_cast<float *>(smem + C::kXOff);   // [2 slots][2 halves][128]
        const float scale2 = p.scale * kLog2e;
        const float cap = p.soft_cap;
        const float cap2 = cap * kLog2e;
        const float scale_over_cap = cap > 0.f ? p.scale / cap : 0.f;
        const float a_mul = cap > 0.f ? 1.f : scale2; // log2-unit logit = s * a_mul
        uint32_t g = 0, pv_seen = 0, nshard = 0;
        bool ok = true;
        // waits of the softmax warps are made warp-uniform, so that no warp
        // reaches a .sync.aligned tcgen05 instruction with some lanes gone
        auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
        };
        auto wait_pv_upto = [&](uint32_t n) -> bool {
            while (pv_seen < n) {
                if (!wait_all(bars.pv_done, pv_seen & 1)) return false;
                ++pv_seen;
            }
            return true;
        };
        // the two threads of a row meet at mbarrier xsync[quarter] (64
        // arrivals per phase); unlike a named barrier its wait is bounded, so
        // a group whose partner aborted gives up too
        uint32_t xph = 0;
        auto pair_sync = [&]() -> bool {
            mbar_arrive(bars.xsync + quarter);
            return wait_all(bars.xsync + quarter, (xph++) & 1);
        };
        for (int r = 0; ok && r * G < U; ++r) {
            const int u = unit_index(r, blockIdx.x, G);
            if (u >= U) continue;
            const Unit x = unit_of(p, u);
            if (x.cnt == 0) continue;
            const int qi = x.qt * kTile + row;
            const int my_pos = p.q_pos ? p.q_pos[(size_t)x.b * p.Lq + qi] : qi;
            const int my_seg = p.q_seg ? p.q_seg[(size_t)x.b * p.Lq + qi] : 0;
            const bool my_pad = p.q_seg && my_seg == p.pad_id;
            const uint8_t *crow = p.tile_class + (size_t)x.row * p.nk;
            for (int t = 0; ok && t < p.N; ++t) {
                const int src = (x.dev - t + p.N) % p.N;
                int lo, hi;
                shard_range(p, x, src, lo, hi);
                if (lo == hi) continue; // the correction warps account for the empty shard
                int pslot = x.pfwd[src]; // number of the shard's first partial tile
                float m_ref = -INFINITY, l = 0.f;
                // the next tile's id and class are fetched one tile ahead
                int kt_next = x.list[lo];
                uint8_t cls_next = crow[kt_next];
                for (int e = lo; ok && e < hi; ++e) {
                    const int kt = kt_next;
                    const bool partial = cls_next == RA_TILE_PARTIAL;
                    if (e + 1 < hi) {
                        kt_next = x.list[e + 1];
                        cls_next = crow[kt_next];
                    }
                    const int sb = g & 1;
                    uint32_t vis0 = ~0u, vis1 = ~0u;
                    if (partial) {
                        // visibility of kv columns kt*128 + c0 .. +63 for this row
                        const uint2 vb = row_bits(p, pslot++, row, wg, x.b, kt * kTile + c0, qi,
                                                  my_seg, my_pad, my_pos);
                        vis0 = vb.x;
                        vis1 = vb.y;
                    }
                    if (!(ok = wait_all(bars.s_full + sb, (g >> 1) & 1))) break;
                    tc_fence_after();
                    float s[64];
                    tmem_ld32(lane_base + sb * 128 + c0, s);
                    tmem_ld32(lane_base + sb * 128 + c0 + 32, s + 32);
                    tmem_ld_wait();
                    // with a soft cap the logits are formed here in log2 units;
                    // without one s stays raw and the scale rides in the exponent
                    if (cap > 0.f) {
                        // max |s| in four independent chains (one serial chain of max3 would
                        // put 32 dependent instructions on the softmax's path)
                        float xa4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int j = 0; j < 64; j += 8)
                            for (int k = 0; k < 4; ++k) xa4[k] = max3(xa4[k], fabsf(s[j + 2 * k]), fabsf(s[j + 2 * k + 1]));
                        const float xa = fmaxf(fmaxf(xa4[0], xa4[1]), fmaxf(xa4[2], xa4[3]));
                        if (__all_sync(0xffffffffu, xa * scale_over_cap < kTanhTiny)) {
                            // cap * log2 e * (x - x^3/3), x = s * scale / cap, as
                            // s * (A + B s^2): three instructions per pair of logits
                            const float kk = scale_over_cap;
                            const float2 A = make_float2(cap2 * kk, cap2 * kk);
                            const float2 B = make_float2(cap2 * kTanhC3 * kk * kk * kk,
                                                         cap2 * kTanhC3 * kk * kk * kk);
#pragma unroll
                            for (int j = 0; j < 64; j += 2) {
                                const float2 v = make_float2(s[j], s[j + 1]);
                                const float2 rr = fmul2(v, ffma2(fmul2(v, v), B, A));
                                s[j] = rr.x;
                                s[j + 1] = rr.y;
                            }
                        } else if (__all_sync(0xffffffffu, xa * scale_over_cap < kTanhSmall)) {
                            // cap * log2 e * tanh(x), x = s / cap * scale, on the FMA pipe:
                            // x * (d1 + x^2 (d3 + x^2 (d5 + x^2 d7))), d = cap2 * c
                            const float2 k2 = make_float2(scale_over_cap, scale_over_cap);
                            const float2 d7 = make_float2(cap2 * kTanhC7, cap2 * kTanhC7);
                            const float2 d5 = make_float2(cap2 * kTanhC5, cap2 * kTanhC5);
                            const float2 d3 = make_float2(cap2 * kTanhC3, cap2 * kTanhC3);
                            const float2 d1 = make_float2(cap2, cap2);
#pragma unroll
                            for (int j = 0; j < 64; j += 2) {
                                const float2 xx = fmul2(make_float2(s[j], s[j + 1]), k2);
                                const float2 x2 = fmul2(xx, xx);
                                float2 pp = ffma2(x2, d7, d5);
                                pp = ffma2(x2, pp, d3);
                                pp = ffma2(x2, pp, d1);
                                const float2 rr = fmul2(xx, pp);
                                s[j] = rr.x;
                                s[j + 1] = rr.y;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 64; ++j) s[j] = cap2 * tanh_fast(s[j] * scale_over_cap);
                        }
                    }
                    if (partial) {
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            if (!(((j < 32 ? vis0 : vis1) >> (j & 31)) & 1u)) s[j] = -INFINITY;
                    }
                    float mx[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        mx[k] = max3(s[k], s[k + 8], s[k + 16]);
                        mx[k] = max3(mx[k], s[k + 24], s[k + 32]);
                        mx[k] = max3(mx[k], s[k + 40], s[k + 48]);
                        mx[k] = fmaxf(mx[k], s[k + 56]);
                    }
                    // a_mul > 0, so scaling commutes with the max
                    float tmax = a_mul * max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]),
                                              fmaxf(mx[6], mx[7]));
                    float *xm = xmax + (g & 1) * 256;
                    xm[wg * 128 + row] = tmax;
                    if (!(ok = pair_sync())) break;
                    tmax = fmaxf(tmax, xm[(wg ^ 1) * 128 + row]);
                    const float m_new = fmaxf(m_ref, tmax);
                    const bool need = (m_ref != -INFINITY) && (m_new > m_ref + 8.f);
                    if (m_ref == -INFINITY) m_ref = m_new;
                    if (__any_sync(0xffffffffu, need)) {
                        // rescale this half of O_acc: the previous PV product must be complete
                        if (!(ok = wait_pv_upto(g))) break;
                        tc_fence_after();
                        const float f = need ? ex2_approx(m_ref - m_new) : 1.f;
                        if (need) {
                            l *= f;
                            m_ref = m_new;
                        }
#pragma unroll
                        for (int c = 0; c < kOH / 32; ++c) {
                            float o[32];
                            tmem_ld32(lane_base + C::kColO + o_col + c * 32, o);
                            tmem_ld_wait();
                            uint32_t w32[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) w32[j] = __float_as_uint(o[j] * f);
                            tmem_st32(lane_base + C::kColO + o_col + c * 32, w32);
                        }
                        tmem_st_wait();
                    }
                    const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                    // p = 2^(s * a_mul - m), two lanes per instruction
                    const float2 am2 = make_float2(a_mul, a_mul);
                    const float2 nm2 = make_float2(-m_use, -m_use);
                    float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                    make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    uint32_t pk[32];
#pragma unroll
                    for (int j = 0; j < 64; j += 2) {
                        const float2 x2 = ffma2(make_float2(s[j], s[j + 1]), am2, nm2);
                        const float2 e2 = make_float2(ex2_approx(x2.x), ex2_approx(x2.y));
                        ls[(j >> 1) & 3] = fadd2(ls[(j >> 1) & 3], e2);
                        pk[j >> 1] = pack_bf16x2(e2.x, e2.y);
                    }
                    const float2 l01 = fadd2(ls[0], ls[1]), l23 = fadd2(ls[2], ls[3]);
                    const float2 l03 = fadd2(l01, l23);
                    l += l03.x + l03.y;
                    // P of this half: columns [64*wg, 64*wg + 32) of the S buffer,
                    // which this half has already read
                    tmem_st32(lane_base + sb * 128 + c0, pk);
                    tmem_st_wait();
                    // PV(g-1) must be complete before P(g) is published
                    if (!(ok = wait_pv_upto(g))) break;
                    tc_fence_before();
                    mbar_arrive(bars.p_full + sb);
                    ++g;
                }
                if (!ok) break;
                // ---- shard end: post this half's row sum and the row max (the
                // same in both halves) for the correction warps; no wait here
                const int slot = nshard & 1;
                ++nshard;
                stat_l[slot * 256 + wg * 128 + row] = l;
                if (wg == 0) stat_m[slot * 128 + row] = m_ref;
                mbar_arrive(bars.stat_full + slot);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

} // namespace

int fwd_tc_smem_bytes(int D)
{
    return D == 64 ? FwdCfg<64>::kSmem : FwdCfg<128>::kSmem;
}

cudaError_t fwd_tc_set_attributes(int D)
{
    const void *fn = D == 64 ? reinterpret_cast<const void *>(fwd_tc_kernel<64>)
                             : reinterpret_cast<const void *>(fwd_tc_kernel<128>);
    // the setmaxnreg split draws on the registers the block is launched with:
    // refuse to run a build that gives each thread fewer than it assumes
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                D == 64 ? FwdCfg<64>::kSmem : FwdCfg<128>::kSmem);
}

cudaError_t launch_fwd_tc(const Problem &p, const void *tm_q, const void *tm_k, const void *tm_v,
                          void *out, float *lse, int num_sms, cudaStream_t s)
{
    const int U = p.B * p.nq * p.Hq;
    const int grid = U < num_sms ? U : num_sms;
    const CUtensorMap &q = *static_cast<const CUtensorMap *>(tm_q);
    const CUtensorMap &k = *static_cast<const CUtensorMap *>(tm_k);
    const CUtensorMap &v = *static_cast<const CUtensorMap *>(tm_v);
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(out);
    if (p.D == 64)
        fwd_tc_kernel<64><<<grid, kFwdThreads, FwdCfg<64>::kSmem, s>>>(q, k, v, p, o, lse);
    else
        fwd_tc_kernel<128><<<grid, kFwdThreads, FwdCfg<128>::kSmem, s>>>(q, k, v, p, o, lse);
    return cudaGetLastError();
}

} // namespace ra
