// k_attn_bwd_tc.cu -- block-sparse flash attention backward on tcgen05 tensor
// cores ("ejKernel ring_attention._ring_splash" module source,
// _ring_attention_backward: per chunk the gradient is taken with the FINAL
// out and lse, dq accumulates locally, dk/dv accumulate with their chunk,
// everything in fp32 and cast back at the end).  Summing over every
// non-empty tile of every chunk gives, with P = exp(s - lse) on visible
// pairs and Delta = <dO, O> (from the preprocessing kernel, which also
// stores -lse * log2 e so that P = 2^(s * scale * log2 e - lse * log2 e) is
// one fused multiply-add per logit):
//   dV_j = sum_i P_ij dO_i                      dP_ij = <dO_i, V_j>
//   dS_ij = P_ij (dP_ij - Delta_i) (1 - tanh^2)  (tanh term only with a cap)
//   dK_j = scale sum_i dS_ij Q_i                dQ_i = scale sum_j dS_ij K_j
// dK / dV are summed over the query heads of a kv head (GQA / MQA).
//
// Two persistent kernels, both without atomics (deterministic):
//   dkdv: one work unit per (b, kv head, 128-row kv tile); it walks the G
//         query heads and the non-empty query tiles of its block-map column.
//         Thread t owns kv row t = TMEM lane t.  TMEM: S^T [0,128),
//         dP^T [128,256), dV [256,256+D), dK [256+D,256+2D).  P^T and dS^T
//         (bf16) overwrite the first halves of S^T and dP^T and feed the
//         dV += P^T dO and dK += dS^T Q products straight from TMEM.
//   dq:   one work unit per (b, q head, 128-row query tile); it walks the
//         non-empty kv tiles of its block-map row.  Thread t owns query row
//         t.  TMEM: S [0,128), dP of even tiles [128,256), dQ [256,256+D),
//         dP of odd tiles [384,512); dS (bf16) overwrites its dP and feeds
//         dQ += dS K from TMEM.
// The dkdv kernel recomputes S and dP per tile and the dq kernel recomputes
// them again: 7 tile products instead of 5, in exchange for no fp32 atomics.
#include <math.h>
#include <type_traits>

#include "ra_sched.cuh"

namespace ra {
namespace {

constexpr uint32_t kIdescT = idesc_bf16(128, 128, false, false); // S^T / dP^T / S / dP

// Warps 0-7: the softmax-gradient work in two warpgroups, each over 64 of the
// 128 tile columns; warp 8: TMA producer; warp 9: TMEM owner and MMA issuer;
// warps 10-11: no role (with warps 8-9 they form the warpgroup that gives
// registers to the softmax warpgroups through setmaxnreg).
// The bf16 operand (P^T, dS^T or dS) each group writes back to TMEM lands on
// columns [0,32) (group 0) or [64,96) (group 1) of the fp32 tile it read,
// so the 16-row K chunks kk of the next MMA sit at column 8*kk + 32*(kk>=4).
constexpr int kSoftmaxThreads = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kBwdThreads = 384;
// setmaxnreg split: 256 x 176 + 128 x 152 = 64512 = 384 x 168, the block's
// registers at launch (the kernels are built for 168 per thread, the most a
// 384-thread block can have: three warps share each sub-partition's 16K;
// the launcher checks the count before the first launch).  The issuing warps
// then have room to spare: spills there slow every product the CTA issues.
constexpr int kBwdLaunchRegs = 168;
constexpr uint32_t kBwdSoftmaxRegs = 176;
constexpr uint32_t kBwdSideRegs = 152;
static_assert(256 * kBwdSoftmaxRegs + 128 * kBwdSideRegs <= kBwdThreads * kBwdLaunchRegs,
              "register split exceeds the block's launch registers");

// ====================================================================== dkdv
template <int D>
struct DkdvCfg {
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kStageBytes = 2 * kTileBytes + 1024; // Q, dO, nlse2[128], delta[128]
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTileBytes;
    static constexpr int kStageOff = 2 * kTileBytes;
    static constexpr int kStages = 2;
    static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
    static constexpr int kNumBars = 2 + 2 * kStages + 6;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // at least 120 KB so that one CTA (which takes all 512 TMEM columns)
    // occupies an SM on its own
    static constexpr int kSmem = (kMiscOff + 16 + 1024) > 122880 ? (kMiscOff + 16 + 1024) : 122880;
    static_assert(kSmem <= 232448, "dK/dV shared memory exceeds the 227 KB per-block limit");
    static constexpr uint32_t kColDP = 128, kColDV = 256, kColDK = 256 + D;
    static constexpr uint32_t kIdescAcc = idesc_bf16(128, D, false, true);
};

struct DkdvBars {
    uint64_t *kv_full, *kv_empty, *st_full, *st_empty, *s_full, *dp_full, *p_ready, *ds_ready,
        *acc_ready, *drain;
};

template <int D>
__device__ __forceinline__ DkdvBars dkdv_bars(uint8_t *smem)
{
    using C = DkdvCfg<D>;
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    DkdvBars r;
    r.kv_full = b;
    r.kv_empty = b + 1;
    r.st_full = b + 2;
    r.st_empty = r.st_full + C::kStages;
    r.s_full = r.st_empty + C::kStages;
    r.dp_full = r.s_full + 1;
    r.p_ready = r.dp_full + 1;
    r.ds_ready = r.p_ready + 1;
    r.acc_ready = r.ds_ready + 1;
    r.drain = r.acc_ready + 1;
    return r;
}

// dK/dV work unit: (kv tile column, kv head, chunk of its query heads); the
// gc query heads h0 .. h0+gc-1 of the chunk are walked over the column.
struct ColUnit {
    int b, kt, hkv, col, cnt, chunk, h0, gc;
    const int32_t *list; // q tiles of the column
};

__device__ __forceinline__ ColUnit col_unit(const Problem &p, int u)
{
    ColUnit x;
    // waves of two kv heads: all columns (longest first) of kv heads 2w and
    // 2w + 1 before the next pair, so that the Q / dO rows read at a time
    // belong to 2 G query heads (when a wave holds at least three units per
    // CTA; smaller waves would leave CTAs on the same few tiles at once)
    int hpw = (p.Hkv % 2 == 0) ? 2 : 1;
    if (p.B * p.nk * hpw * p.hsplit < 3 * (int)gridDim.x) hpw = p.Hkv;
    const int per = hpw * p.hsplit;
    const int wave_units = p.B * p.nk * per;
    const int w = u / wave_units;
    const int rr = u - w * wave_units;
    x.col = p.bwd_order[rr / per];
    const int r = rr - (rr / per) * per;
    x.hkv = w * hpw + r / p.hsplit;
    x.chunk = r - (r / p.hsplit) * p.hsplit;
    x.gc = p.G / p.hsplit;
    x.h0 = x.hkv * p.G + x.chunk * x.gc;
    x.b = x.col / p.nk;
    x.kt = x.col - x.b * p.nk;
    x.cnt = p.bwd_cnt[x.col];
    x.list = p.bwd_idx + (size_t)x.col * p.nq;
    return x;
}

// CAP: soft cap on (compiled per choice, so that neither form carries the
// other's code)
template <int D, bool CAP>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    Problem p, const float *__restrict__ nlse2, const float *__restrict__ delta,
                    __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv)
{
    using C = DkdvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const DkdvBars bars = dkdv_bars<D>(smem);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
    const WaitCtx ctx{abort_flag, p.status, p.timeout_ns};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = p.B * p.nk * p.Hkv * p.hsplit;
    const int Gd = gridDim.x;

    if (threadIdx.x == 0) {
        mbar_init(bars.kv_full, 1);
        mbar_init(bars.kv_empty, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bars.st_full + s, 1);
            mbar_init(bars.st_empty + s, 1);
        }
        mbar_init(bars.s_full, 1);
        mbar_init(bars.dp_full, 1);
        mbar_init(bars.p_ready, kSoftmaxThreads);
        mbar_init(bars.ds_ready, kSoftmaxThreads);
        mbar_init(bars.acc_ready, 1);
        mbar_init(bars.drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp >= kProducerWarp) {
        regs_shrink<kBwdSideRegs>();
        if (warp == kProducerWarp) {
            // ---------------------------------------------------------- producer
            if (lane == 0) {
                uint32_t n = 0, uk = 0;
                uint32_t st_issued[C::kStages] = {};
                bool ok = true;
                for (int r = 0; ok && r * Gd < U; ++r) {
                    const int u = unit_index(r, blockIdx.x, Gd);
                    if (u >= U) continue;
                    const ColUnit x = col_unit(p, u);
                    if (x.cnt == 0) continue;
                    if (!(ok = mbar_wait(bars.kv_empty, (uk & 1) ^ 1, ctx))) break;
                    mbar_expect_tx(bars.kv_full, 2 * C::kTileBytes);
                    for (int hb = 0; hb < D / 64; ++hb) {
                        tma_load_4d(smem + C::kKOff + hb * 16384, &tm_k, bars.kv_full, hb * 64, x.hkv,
                                    x.kt * kTile, x.b);
                        tma_load_4d(smem + C::kVOff + hb * 16384, &tm_v, bars.kv_full, hb * 64, x.hkv,
                                    x.kt * kTile, x.b);
                    }
                    ++uk;
                    for (int gi = 0; ok && gi < x.gc; ++gi) {
                        const int h = x.h0 + gi;
                        for (int e = 0; e < x.cnt; ++e) {
                            const int qt = x.list[e];
                            const int st = n % C::kStages;
                            if (!(ok = mbar_wait(bars.st_empty + st, ((n / C::kStages) & 1) ^ 1, ctx))) break;
                            uint8_t *sb = smem + C::kStageOff + st * C::kStageBytes;
                            mbar_expect_tx(bars.st_full + st, 2 * C::kTileBytes + 1024);
                            for (int hb = 0; hb < D / 64; ++hb) {
                                tma_load_4d(sb + hb * 16384, &tm_q, bars.st_full + st, hb * 64, h,
                                            qt * kTile, x.b);
                                tma_load_4d(sb + C::kTileBytes + hb * 16384, &tm_do, bars.st_full + st,
                                            hb * 64, h, qt * kTile, x.b);
                            }
                            const size_t li = ((size_t)x.b * p.Hq + h) * p.Lq + (size_t)qt * kTile;
                            bulk_load(sb + 2 * C::kTileBytes, nlse2 + li, 512, bars.st_full + st);
                            bulk_load(sb + 2 * C::kTileBytes + 512, delta + li, 512, bars.st_full + st);
                            ++st_issued[st];
                            ++n;
                        }
                    }
                }
                if (!ok) {
                    for (int s = 0; s < C::kStages; ++s)
                        if (st_issued[s]) wait_drain(bars.st_full + s, (st_issued[s] - 1) & 1, kDrainNs);
                    if (uk) wait_drain(bars.kv_full, (uk - 1) & 1, kDrainNs);
                }
            }
        } else if (warp == kMmaWarp) {
            // ---------------------------------------------------------- MMA issuer
            // The whole warp runs the issue loop, converged: every lane waits on
            // the barriers, and one lane, chosen by elect.sync, issues each
            // product, copy and commit.
            {
                auto wait_w = [&](uint64_t *bar, uint32_t parity) -> bool {
                    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
                };
                const uint32_t k_base = smem_u32(smem + C::kKOff);
                const uint32_t v_base = smem_u32(smem + C::kVOff);
                uint32_t n = 0, uk = 0;
                bool ok = true;
                auto stage_base = [&](uint32_t step) {
                    return smem_u32(smem + C::kStageOff + (step % C::kStages) * C::kStageBytes);
                };
                auto wait_stage = [&](uint32_t step) -> bool {
                    if (!wait_w(bars.st_full + step % C::kStages, (step / C::kStages) & 1)) return false;
                    tc_fence_after();
                    return true;
                };
                // S^T = K Q^T into columns [0,128)
                // descriptors are built once per operand; an offset o adds o / 16
                const uint64_t kd = sdesc_sw128(k_base, 16, 1024), vd = sdesc_sw128(v_base, 16, 1024);
                auto issue_s = [&](uint32_t q_base) {
                    const uint64_t qd = sdesc_sw128(q_base, 16, 1024);
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        mma_ss_w(tmem, kd + o, qd + o, kIdescT, kk > 0 ? 1u : 0u);
                    }
                    tc_commit_w(bars.s_full);
                };
                // dP^T = V dO^T into columns [128,256)
                auto issue_dp = [&](uint32_t do_base) {
                    const uint64_t dd = sdesc_sw128(do_base, 16, 1024);
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        mma_ss_w(tmem + C::kColDP, vd + o, dd + o, kIdescT, kk > 0 ? 1u : 0u);
                    }
                    tc_commit_w(bars.dp_full);
                };
                // Issue order per step n (each product overlaps a softmax phase):
                //   dP(n) | phase A(n);  dV(n), S(n+1) | phase B(n);
                //   dK(n), dP(n+1) | phase A(n+1).
                // S(n+1) may overwrite P^T(n) once dV(n) is issued (MMAs run in
                // order); dP(n+1) may overwrite dS^T(n) once dK(n) is issued.
                for (int r = 0; ok && r * Gd < U; ++r) {
                    const int u = unit_index(r, blockIdx.x, Gd);
                    if (u >= U) continue;
                    const ColUnit x = col_unit(p, u);
                    if (x.cnt == 0) continue;
                    if (!(ok = wait_w(bars.kv_full, uk & 1))) break;
                    tc_fence_after();
                    ++uk;
                    const int steps = x.gc * x.cnt;
                    if (!(ok = wait_stage(n))) break;
                    issue_s(stage_base(n));
                    for (int i = 0; i < steps; ++i, ++n) {
                        const uint32_t q_base = stage_base(n);
                        const uint32_t do_base = q_base + C::kTileBytes;
                        issue_dp(do_base);
                        // dV += P^T dO   (A = P^T from TMEM, B = dO as a K=q x N=D MN-major tile)
                        if (!(ok = wait_w(bars.p_ready, n & 1))) break;
                        tc_fence_after();
                        const uint64_t dmn = sdesc_sw128(do_base, 16384, 1024);
    #pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ts_w(tmem + C::kColDV, tmem + kk * 8 + (kk >= 4 ? 32 : 0),
                                   dmn + (uint32_t)((kk * 2048) >> 4), C::kIdescAcc,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                        if (i + 1 < steps) {
                            if (!(ok = wait_stage(n + 1))) break;
                            issue_s(stage_base(n + 1));
                        }
                        // dK += dS^T Q
                        if (!(ok = wait_w(bars.ds_ready, n & 1))) break;
                        tc_fence_after();
                        const uint64_t qmn = sdesc_sw128(q_base, 16384, 1024);
    #pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ts_w(tmem + C::kColDK, tmem + C::kColDP + kk * 8 + (kk >= 4 ? 32 : 0),
                                   qmn + (uint32_t)((kk * 2048) >> 4), C::kIdescAcc,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                        tc_commit_w(bars.st_empty + n % C::kStages);
                    }
                    if (!ok) break;
                    tc_commit_w(bars.kv_empty);
                    tc_commit_w(bars.acc_ready);
                }
                tc_commit_w(bars.drain);
                wait_drain(bars.drain, 0, kDrainNs);
            }
        }
    } else {
        regs_grow<kBwdSoftmaxRegs>();
        // ---------------------------------------------------------- softmax-grad
        // Warps 0-7 in two warpgroups: group wg handles query columns
        // 64*wg..64*wg+63 (and D/2 columns of dK, dV) of kv row 32*(w%4)+lane.
        const int wg = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane; // kv row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int c0 = wg * 64;
        // head split: the chunk's scaled dK and dV go to fp32 partials
        const bool split = p.hsplit > 1;
        float *part_k = p.dkv_part;
        float *part_v = split ? p.dkv_part + (size_t)p.hsplit * p.B * p.Lkv * p.Hkv * D : nullptr;
        constexpr int kOH = D / 2;
        const uint32_t o_col = wg * kOH;
        const float scale2 = p.scale * kLog2e;
        const float cap = CAP ? p.soft_cap : 0.f;
        const float cap2 = cap * kLog2e;
        const float scale_over_cap = cap > 0.f ? p.scale / cap : 0.f;
        uint32_t n = 0, ua = 0;
        bool ok = true;
        auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
        };
        for (int r = 0; ok && r * Gd < U; ++r) {
            const int u = unit_index(r, blockIdx.x, Gd);
            if (u >= U) continue;
            const ColUnit x = col_unit(p, u);
            const int kj = x.kt * kTile + row;
            const size_t orow = (((size_t)x.b * p.Lkv + kj) * p.Hkv + x.hkv) * D + o_col;
            // this chunk's slice of the partials: (hsplit, B, Lkv, Hkv, D)
            const size_t prow = (size_t)x.chunk * p.B * p.Lkv * p.Hkv * D + orow;
            if (x.cnt > 0) {
                const int my_pos = p.kv_pos ? p.kv_pos[(size_t)x.b * p.Lkv + kj] : kj;
                const int my_seg = p.kv_seg ? p.kv_seg[(size_t)x.b * p.Lkv + kj] : 0;
                const int steps = x.gc * x.cnt;
                // column-order number of the next partial tile (restarts with each head)
                const int pbase = p.part_bwd[x.col];
                int pslot = pbase;
                for (int i = 0; i < steps; ++i, ++n) {
                    const int e = i % x.cnt;
                    if (e == 0) pslot = pbase;
                    const int qt = x.list[e];
                    const int st = n % C::kStages;
                    const float *lse_s = reinterpret_cast<const float *>(
                        smem + C::kStageOff + st * C::kStageBytes + 2 * C::kTileBytes) + c0;
                    const float *dl_s = lse_s + 128;
                    const bool partial =
                        p.tile_class[((size_t)x.b * p.nq + qt) * p.nk + x.kt] == RA_TILE_PARTIAL;
                    // ---- visibility bits of this half's 64 query columns (partial tiles only)
                    uint32_t vis[2] = {~0u, ~0u};
                    if (partial) {
                        const uint2 vb = col_bits(p, pslot++, row, wg, x.b, qt * kTile + c0, kj, my_seg,
                                                  my_pos);
                        vis[0] = vb.x;
                        vis[1] = vb.y;
                    }
                    if (!(ok = wait_all(bars.s_full, n & 1))) break;
                    tc_fence_after();
                    // ---- P^T (bf16 -> TMEM) and Pc = P * (1 - tanh^2) kept packed
                    uint32_t pc[32];
                    {
                        float s[64];
                        tmem_ld32(lane_base + c0, s);
                        tmem_ld32(lane_base + c0 + 32, s + 32);
                        tmem_ld_wait();
                        const float4 *l4 = reinterpret_cast<const float4 *>(lse_s);
                        uint32_t pk[32];
                        if (CAP) {
                            // max |s| in four independent chains (one serial chain of max3 would
                            // put 32 dependent instructions on the softmax's path)
                            float xa4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int j = 0; j < 64; j += 8)
                                for (int k = 0; k < 4; ++k) xa4[k] = max3(xa4[k], fabsf(s[j + 2 * k]), fabsf(s[j + 2 * k + 1]));
                            const float xa = fmaxf(fmaxf(xa4[0], xa4[1]), fmaxf(xa4[2], xa4[3]));
                            const bool tiny = __all_sync(0xffffffffu, xa * scale_over_cap < kTanhTiny) != 0;
                            if (tiny || __all_sync(0xffffffffu, xa * scale_over_cap < kTanhSmall)) {
                                // tanh by its odd Taylor series on the FMA pipe, two lanes
                                // per instruction: t = x (1 + x^2 (c3 + x^2 (c5 + x^2 c7))),
                                // or t = x (1 + c3 x^2) when every |x| < 1/8
                                const float2 k2 = make_float2(scale_over_cap, scale_over_cap);
                                const float2 c7 = make_float2(kTanhC7, kTanhC7);
                                const float2 c5 = make_float2(kTanhC5, kTanhC5);
                                const float2 c3 = make_float2(kTanhC3, kTanhC3);
                                const float2 one = make_float2(1.f, 1.f);
                                const float2 cc = make_float2(cap2, cap2);
                                auto run = [&](auto tiny_c) {
                                    constexpr bool kTiny = decltype(tiny_c)::value;
#pragma unroll
                                    for (int j = 0; j < 64; j += 4) {
                                        const float4 lv = l4[j >> 2];
                                        const float2 la[2] = {make_float2(lv.x, lv.y), make_float2(lv.z, lv.w)};
#pragma unroll
                                        for (int h = 0; h < 2; ++h) {
                                            const int c = j + 2 * h;
                                            const float2 x = fmul2(make_float2(s[c], s[c + 1]), k2);
                                            const float2 x2 = fmul2(x, x);
                                            float2 pp;
                                            if (kTiny) {
                                                pp = ffma2(x2, c3, one);
                                            } else {
                                                pp = ffma2(x2, c7, c5);
                                                pp = ffma2(x2, pp, c3);
                                                pp = ffma2(x2, pp, one);
                                            }
                                            const float2 t = fmul2(x, pp);
                                            const float2 a = ffma2(cc, t, la[h]);
                                            float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                                            if (partial) {
                                                e.x = ((vis[c >> 5] >> (c & 31)) & 1u) ? e.x : 0.f;
                                                e.y = ((vis[(c + 1) >> 5] >> ((c + 1) & 31)) & 1u) ? e.y : 0.f;
                                            }
                                            const float2 cr = fmul2(e, fsub2(one, fmul2(t, t)));
                                            pk[c >> 1] = pack_bf16x2(e.x, e.y);
                                            pc[c >> 1] = pack_bf16x2(cr.x, cr.y);
                                        }
                                    }
                                };
                                if (tiny) run(std::true_type{});
                                else run(std::false_type{});
                            } else {
#pragma unroll
                                for (int j = 0; j < 64; j += 4) {
                                    const float4 lv = l4[j >> 2];
                                    const float la[4] = {lv.x, lv.y, lv.z, lv.w};
                                    float pr[4], cr[4];
#pragma unroll
                                    for (int z = 0; z < 4; ++z) {
                                        const int c = j + z;
                                        const float t = tanh_fast(s[c] * scale_over_cap);
                                        float e = ex2_approx(fmaf(cap2, t, la[z]));
                                        e = ((vis[c >> 5] >> (c & 31)) & 1u) ? e : 0.f;
                                        pr[z] = e;
                                        cr[z] = e * (1.f - t * t);
                                    }
                                    pk[j >> 1] = pack_bf16x2(pr[0], pr[1]);
                                    pk[(j >> 1) + 1] = pack_bf16x2(pr[2], pr[3]);
                                    pc[j >> 1] = pack_bf16x2(cr[0], cr[1]);
                                    pc[(j >> 1) + 1] = pack_bf16x2(cr[2], cr[3]);
                                }
                            }
                        } else {
                            // masked logits -> -inf, so that 2^(...) = 0 below
                            if (partial) {
#pragma unroll
                                for (int c = 0; c < 64; ++c)
                                    if (!((vis[c >> 5] >> (c & 31)) & 1u)) s[c] = -INFINITY;
                            }
                            // P = 2^(s * scale * log2 e + nlse2), two lanes per instruction
                            const float2 sc2 = make_float2(scale2, scale2);
#pragma unroll
                            for (int j = 0; j < 64; j += 4) {
                                const float4 lv = l4[j >> 2];
                                const float2 x0 = ffma2(make_float2(s[j], s[j + 1]), sc2, make_float2(lv.x, lv.y));
                                const float2 x1 = ffma2(make_float2(s[j + 2], s[j + 3]), sc2, make_float2(lv.z, lv.w));
                                pk[j >> 1] = pack_bf16x2(ex2_approx(x0.x), ex2_approx(x0.y));
                                pk[(j >> 1) + 1] = pack_bf16x2(ex2_approx(x1.x), ex2_approx(x1.y));
                                pc[j >> 1] = pk[j >> 1];
                                pc[(j >> 1) + 1] = pk[(j >> 1) + 1];
                            }
                        }
                        // this half's P^T over the S^T columns it has just read
                        tmem_st32(lane_base + c0, pk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bars.p_ready);
                    // ---- dS^T = Pc (dP^T - Delta)
                    if (!(ok = wait_all(bars.dp_full, n & 1))) break;
                    tc_fence_after();
                    {
                        float dpv[64];
                        tmem_ld32(lane_base + C::kColDP + c0, dpv);
                        tmem_ld32(lane_base + C::kColDP + c0 + 32, dpv + 32);
                        tmem_ld_wait();
                        const float4 *d4 = reinterpret_cast<const float4 *>(dl_s);
                        uint32_t dk2[32];
                        // (dP - Delta) rounded to bf16, times the bf16 Pc, two lanes per
                        // instruction
#pragma unroll
                        for (int j = 0; j < 64; j += 4) {
                            const float4 dl = d4[j >> 2];
                            const float2 r0 = fsub2(make_float2(dpv[j], dpv[j + 1]), make_float2(dl.x, dl.y));
                            const float2 r1 = fsub2(make_float2(dpv[j + 2], dpv[j + 3]), make_float2(dl.z, dl.w));
                            dk2[j >> 1] = mul_bf16x2(pc[j >> 1], pack_bf16x2(r0.x, r0.y));
                            dk2[(j >> 1) + 1] = mul_bf16x2(pc[(j >> 1) + 1], pack_bf16x2(r1.x, r1.y));
                        }
                        tmem_st32(lane_base + C::kColDP + c0, dk2);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bars.ds_ready);
                }
                if (!ok) break;
                // ---- epilogue: this half of dV and scale * dK -> bf16 (or, with
                // a head split, the chunk's fp32 partials)
                if (!(ok = wait_all(bars.acc_ready, ua & 1))) break;
                ++ua;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kOH / 32; ++c) {
                    float a[32], bk[32];
                    tmem_ld32(lane_base + C::kColDV + o_col + c * 32, a);
                    tmem_ld32(lane_base + C::kColDK + o_col + c * 32, bk);
                    tmem_ld_wait();
                    if (p.acc_dk) {
                        // ring step: add to the chunk's travelling fp32 accumulators
                        float4 *ak4 = reinterpret_cast<float4 *>(p.acc_dk + orow + c * 32);
                        float4 *av4 = reinterpret_cast<float4 *>(p.acc_dv + orow + c * 32);
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4) {
                            float4 tk = ak4[k4], tv = av4[k4];
                            tk.x += p.scale * bk[4 * k4];
                            tk.y += p.scale * bk[4 * k4 + 1];
                            tk.z += p.scale * bk[4 * k4 + 2];
                            tk.w += p.scale * bk[4 * k4 + 3];
                            tv.x += a[4 * k4];
                            tv.y += a[4 * k4 + 1];
                            tv.z += a[4 * k4 + 2];
                            tv.w += a[4 * k4 + 3];
                            ak4[k4] = tk;
                            av4[k4] = tv;
                        }
                        continue;
                    }
                    if (split) {
                        float4 *pk4 = reinterpret_cast<float4 *>(part_k + prow + c * 32);
                        float4 *pv4 = reinterpret_cast<float4 *>(part_v + prow + c * 32);
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4) {
                            pv4[k4] = make_float4(a[4 * k4], a[4 * k4 + 1], a[4 * k4 + 2], a[4 * k4 + 3]);
                            pk4[k4] = make_float4(p.scale * bk[4 * k4], p.scale * bk[4 * k4 + 1],
                                                  p.scale * bk[4 * k4 + 2], p.scale * bk[4 * k4 + 3]);
                        }
                        continue;
                    }
                    uint4 *dvp = reinterpret_cast<uint4 *>(dv + orow + c * 32);
                    uint4 *dkp = reinterpret_cast<uint4 *>(dk + orow + c * 32);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        uint4 v, w;
                        v.x = pack_bf16x2(a[8 * k4 + 0], a[8 * k4 + 1]);
                        v.y = pack_bf16x2(a[8 * k4 + 2], a[8 * k4 + 3]);
                        v.z = pack_bf16x2(a[8 * k4 + 4], a[8 * k4 + 5]);
                        v.w = pack_bf16x2(a[8 * k4 + 6], a[8 * k4 + 7]);
                        w.x = pack_bf16x2(p.scale * bk[8 * k4 + 0], p.scale * bk[8 * k4 + 1]);
                        w.y = pack_bf16x2(p.scale * bk[8 * k4 + 2], p.scale * bk[8 * k4 + 3]);
                        w.z = pack_bf16x2(p.scale * bk[8 * k4 + 4], p.scale * bk[8 * k4 + 5]);
                        w.w = pack_bf16x2(p.scale * bk[8 * k4 + 6], p.scale * bk[8 * k4 + 7]);
                        dvp[k4] = v;
                        dkp[k4] = w;
                    }
                }
            } else if (p.acc_dk) {
                // ring step: a column with nothing visible adds nothing
            } else if (split) {
                float4 *pk4 = reinterpret_cast<float4 *>(part_k + prow);
                float4 *pv4 = reinterpret_cast<float4 *>(part_v + prow);
                for (int k4 = 0; k4 < kOH / 4; ++k4) {
                    pk4[k4] = make_float4(0.f, 0.f, 0.f, 0.f);
                    pv4[k4] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            } else {
                uint4 *dvp = reinterpret_cast<uint4 *>(dv + orow);
                uint4 *dkp = reinterpret_cast<uint4 *>(dk + orow);
                for (int k4 = 0; k4 < kOH / 8; ++k4) {
                    dvp[k4] = make_uint4(0, 0, 0, 0);
                    dkp[k4] = make_uint4(0, 0, 0, 0);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ====================================================================== dq
template <int D>
struct DqCfg {
    static constexpr int kTileBytes = kTile * D * 2;
    // Q and dO of a unit land in shared memory by TMA and are copied into
    // TMEM once (tcgen05.cp), where they are the A operands of S = Q K^T and
    // dP = dO V^T for the whole unit; their shared-memory tiles are then free
    // for the next unit's.  A K tile is held from S(g) to dQ(g), a V tile
    // only until dP(g).
    static constexpr int kQOff = 0;
    static constexpr int kDoOff = kTileBytes;
    static constexpr int kKOff = 2 * kTileBytes;
    static constexpr int kKStages = 3;
    static constexpr int kVStages = 2;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
    static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 7;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmem = (kMiscOff + 16 + 1024) > 122880 ? (kMiscOff + 16 + 1024) : 122880;
    static_assert(kSmem <= 232448, "dQ shared memory exceeds the 227 KB per-block limit");
    // TMEM: S, dP (dS written over it), dQ, and the unit's Q and dO rows as
    // packed bf16 pairs (D / 2 columns each)
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
    static constexpr uint32_t kColQA = 384, kColDOA = 384 + D / 2;
    static constexpr uint32_t kIdescAcc = idesc_bf16(128, D, false, true);
};

struct DqBars {
    uint64_t *q_full, *q_empty, *k_full, *k_empty, *v_full, *v_empty, *s_full, *dp_full, *s_free,
        *ds_ready, *acc_ready, *drain;
};

template <int D>
__device__ __forceinline__ DqBars dq_bars(uint8_t *smem)
{
    using C = DqCfg<D>;
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    DqBars r;
    r.q_full = b;
    r.q_empty = b + 1;
    r.k_full = b + 2;
    r.k_empty = r.k_full + C::kKStages;
    r.v_full = r.k_empty + C::kKStages;
    r.v_empty = r.v_full + C::kVStages;
    r.s_full = r.v_empty + C::kVStages;
    r.dp_full = r.s_full + 1;
    r.s_free = r.dp_full + 1;
    r.ds_ready = r.s_free + 1;
    r.acc_ready = r.ds_ready + 1;
    r.drain = r.acc_ready + 1;
    return r;
}

struct RowUnit {
    int b, qt, h, row, cnt;
    const int32_t *list;
};

__device__ __forceinline__ RowUnit row_unit(const Problem &p, int u)
{
    RowUnit x;
    // waves of the query heads of two kv heads: all rows (longest first) of
    // those 2 G heads before the next, so that the K / V rows read at a time
    // belong to two kv heads (when a wave holds at least three units per CTA;
    // smaller waves would leave CTAs on the same few tiles at once)
    int hpw = (p.Hkv % 2 == 0) ? 2 * p.G : p.G;
    if (p.B * p.nq * hpw < 3 * (int)gridDim.x) hpw = p.Hq;
    const int wave_units = p.B * p.nq * hpw;
    const int w = u / wave_units;
    const int rr = u - w * wave_units;
    x.row = p.fwd_order[rr / hpw];
    x.h = w * hpw + (rr - (rr / hpw) * hpw);
    x.b = x.row / p.nq;
    x.qt = x.row - x.b * p.nq;
    x.cnt = p.fwd_cnt[x.row];
    x.list = p.fwd_idx + (size_t)x.row * p.nk;
    return x;
}

template <int D, bool CAP>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  Problem p, const float *__restrict__ nlse2, const float *__restrict__ delta,
                  __nv_bfloat16 *__restrict__ dq)
{
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const DqBars bars = dq_bars<D>(smem);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
    const WaitCtx ctx{abort_flag, p.status, p.timeout_ns};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = p.B * p.nq * p.Hq;
    const int Gd = gridDim.x;

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
        mbar_init(bars.s_full, 1);
        mbar_init(bars.s_free, kSoftmaxThreads);
        mbar_init(bars.dp_full, 1);
        mbar_init(bars.ds_ready, kSoftmaxThreads);
        mbar_init(bars.acc_ready, 1);
        mbar_init(bars.drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp >= kProducerWarp) {
        regs_shrink<kBwdSideRegs>();
        if (warp == kProducerWarp) {
            // ---------------------------------------------------------- producer
            if (lane == 0) {
                uint32_t g = 0, uq = 0;
                uint32_t k_issued[C::kKStages] = {}, v_issued[C::kVStages] = {};
                bool ok = true;
                for (int r = 0; ok && r * Gd < U; ++r) {
                    const int u = unit_index(r, blockIdx.x, Gd);
                    if (u >= U) continue;
                    const RowUnit x = row_unit(p, u);
                    if (x.cnt == 0) continue;
                    if (!(ok = mbar_wait(bars.q_empty, (uq & 1) ^ 1, ctx))) break;
                    mbar_expect_tx(bars.q_full, 2 * C::kTileBytes);
                    for (int hb = 0; hb < D / 64; ++hb) {
                        tma_load_4d(smem + C::kQOff + hb * 16384, &tm_q, bars.q_full, hb * 64, x.h,
                                    x.qt * kTile, x.b);
                        tma_load_4d(smem + C::kDoOff + hb * 16384, &tm_do, bars.q_full, hb * 64, x.h,
                                    x.qt * kTile, x.b);
                    }
                    ++uq;
                    const int g_kv = x.h / p.G;
                    for (int e = 0; e < x.cnt; ++e) {
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
                if (!ok) {
                    for (int s = 0; s < C::kKStages; ++s)
                        if (k_issued[s]) wait_drain(bars.k_full + s, (k_issued[s] - 1) & 1, kDrainNs);
                    for (int s = 0; s < C::kVStages; ++s)
                        if (v_issued[s]) wait_drain(bars.v_full + s, (v_issued[s] - 1) & 1, kDrainNs);
                    if (uq) wait_drain(bars.q_full, (uq - 1) & 1, kDrainNs);
                }
            }
        } else if (warp == kMmaWarp) {
            // ---------------------------------------------------------- MMA issuer
            // The whole warp runs the issue loop, converged: every lane waits on
            // the barriers, and one lane, chosen by elect.sync, issues each
            // product, copy and commit.
            {
                auto wait_w = [&](uint64_t *bar, uint32_t parity) -> bool {
                    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
                };
                const uint32_t k_base = smem_u32(smem + C::kKOff);
                const uint32_t v_base = smem_u32(smem + C::kVOff);
                const uint64_t qd = sdesc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
                const uint64_t dod = sdesc_sw128(smem_u32(smem + C::kDoOff), 16, 1024);
                uint32_t g = 0, uq = 0;
                bool ok = true;
                // S = Q K^T of tile t into columns [0,128): A = the unit's Q rows
                // from TMEM (16-column K chunk kk at column 8 kk), B = the K tile
                // descriptors are built once per operand; an offset o adds o / 16
                auto issue_s = [&](uint32_t t) -> bool {
                    if (!wait_w(bars.k_full + t % C::kKStages, (t / C::kKStages) & 1)) return false;
                    tc_fence_after();
                    const uint64_t kd = sdesc_sw128(k_base + (t % C::kKStages) * C::kTileBytes, 16, 1024);
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        mma_ts_w(tmem + C::kColS, tmem + C::kColQA + kk * 8, kd + o, kIdescT, kk > 0 ? 1u : 0u);
                    }
                    tc_commit_w(bars.s_full);
                    return true;
                };
                // dP = dO V^T of tile t into [128,256); V's stage is free after it
                auto issue_dp = [&](uint32_t t) -> bool {
                    if (!wait_w(bars.v_full + t % C::kVStages, (t / C::kVStages) & 1)) return false;
                    tc_fence_after();
                    const uint64_t vd = sdesc_sw128(v_base + (t % C::kVStages) * C::kTileBytes, 16, 1024);
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        mma_ts_w(tmem + C::kColDP, tmem + C::kColDOA + kk * 8, vd + o, kIdescT, kk > 0 ? 1u : 0u);
                    }
                    tc_commit_w(bars.dp_full);
                    tc_commit_w(bars.v_empty + t % C::kVStages);
                    return true;
                };
                // Issue order per tile g: S(g+1) as soon as phase A(g) has read S(g);
                // dQ(g) once phase B(g) has written dS(g) over dP(g); then dP(g+1),
                // which the in-order pipe runs after dQ(g) has read dS(g).  Every
                // product takes its A operand from TMEM, so the shared-memory
                // traffic per product is the one B tile.
                for (int r = 0; ok && r * Gd < U; ++r) {
                    const int u = unit_index(r, blockIdx.x, Gd);
                    if (u >= U) continue;
                    const RowUnit x = row_unit(p, u);
                    if (x.cnt == 0) continue;
                    // this unit's Q and dO tiles into TMEM, 16 columns of the head
                    // dimension per copy, at the K-chunk offsets the products use.
                    // No product still reads the previous unit's: its last dP had
                    // completed before its last phase B began.
                    if (!(ok = wait_w(bars.q_full, uq & 1))) break;
                    tc_fence_after();
                    ++uq;
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        tmem_cp_128x256b_w(tmem + C::kColQA + kk * 8, qd + o);
                        tmem_cp_128x256b_w(tmem + C::kColDOA + kk * 8, dod + o);
                    }
                    tc_commit_w(bars.q_empty); // the tiles' shared memory is free once the copies are done
                    if (!(ok = issue_s(g))) break;
                    if (!(ok = issue_dp(g))) break;
                    for (int e = 0; e < x.cnt; ++e, ++g) {
                        if (!(ok = wait_w(bars.s_free, g & 1))) break;
                        if (e + 1 < x.cnt && !(ok = issue_s(g + 1))) break;
                        // dQ += dS K   (A = dS from TMEM, B = K as a K=kv x N=D MN-major tile)
                        if (!(ok = wait_w(bars.ds_ready, g & 1))) break;
                        tc_fence_after();
                        const int sk = g % C::kKStages;
                        const uint64_t kmn = sdesc_sw128(k_base + sk * C::kTileBytes, 16384, 1024);
    #pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ts_w(tmem + C::kColDQ, tmem + C::kColDP + kk * 8 + (kk >= 4 ? 32 : 0),
                                   kmn + (uint32_t)((kk * 2048) >> 4), C::kIdescAcc,
                                   (e > 0 || kk > 0) ? 1u : 0u);
                        tc_commit_w(bars.k_empty + sk);
                        if (e + 1 < x.cnt && !(ok = issue_dp(g + 1))) break;
                    }
                    if (!ok) break;
                    tc_commit_w(bars.acc_ready);
                }
                tc_commit_w(bars.drain);
                wait_drain(bars.drain, 0, kDrainNs);
            }
        }
    } else {
        regs_grow<kBwdSoftmaxRegs>();
        // ---------------------------------------------------------- softmax-grad
        // Warps 0-7 in two warpgroups: group wg handles kv columns
        // 64*wg..64*wg+63 (and D/2 columns of dQ) of query row 32*(w%4)+lane.
        const int wg = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int c0 = wg * 64;
        constexpr int kOH = D / 2;
        const uint32_t o_col = wg * kOH;
        const float scale2 = p.scale * kLog2e;
        const float cap = CAP ? p.soft_cap : 0.f;
        const float cap2 = cap * kLog2e;
        const float scale_over_cap = cap > 0.f ? p.scale / cap : 0.f;
        uint32_t g = 0, ua = 0;
        bool ok = true;
        auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
        };
        for (int r = 0; ok && r * Gd < U; ++r) {
            const int u = unit_index(r, blockIdx.x, Gd);
            if (u >= U) continue;
            const RowUnit x = row_unit(p, u);
            const int qi = x.qt * kTile + row;
            __nv_bfloat16 *qrow = dq + (((size_t)x.b * p.Lq + qi) * p.Hq + x.h) * D + o_col;
            if (x.cnt > 0) {
                const size_t li = ((size_t)x.b * p.Hq + x.h) * p.Lq + qi;
                // exponent offset -lse * log2 e (0 for a row with nothing visible:
                // it only meets partial tiles, where the mask zeroes every P)
                const float nl2 = nlse2[li];
                const float dl = delta[li];
                const int my_pos = p.q_pos ? p.q_pos[(size_t)x.b * p.Lq + qi] : qi;
                const int my_seg = p.q_seg ? p.q_seg[(size_t)x.b * p.Lq + qi] : 0;
                const bool my_pad = p.q_seg && my_seg == p.pad_id;
                const uint8_t *crow = p.tile_class + (size_t)x.row * p.nk;
                // row-order number of the next partial tile
                int pslot = p.part_fwd[(size_t)x.row * (p.N + 1)];
                for (int e = 0; e < x.cnt; ++e, ++g) {
                    const int kt = x.list[e];
                    const bool partial = crow[kt] == RA_TILE_PARTIAL;
                    uint32_t vis[2] = {~0u, ~0u};
                    if (partial) {
                        const uint2 vb = row_bits(p, pslot++, row, wg, x.b, kt * kTile + c0, qi, my_seg,
                                                  my_pad, my_pos);
                        vis[0] = vb.x;
                        vis[1] = vb.y;
                    }
                    if (!(ok = wait_all(bars.s_full, g & 1))) break;
                    tc_fence_after();
                    // ---- phase A: Pc = P * (1 - tanh^2) in fp32 registers (P from S)
                    float pf[64];
                    {
                        float s[64];
                        tmem_ld32(lane_base + c0, s);
                        tmem_ld32(lane_base + c0 + 32, s + 32);
                        tmem_ld_wait();
                        if (CAP) {
                            // max |s| in four independent chains (one serial chain of max3 would
                            // put 32 dependent instructions on the softmax's path)
                            float xa4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int j = 0; j < 64; j += 8)
                                for (int k = 0; k < 4; ++k) xa4[k] = max3(xa4[k], fabsf(s[j + 2 * k]), fabsf(s[j + 2 * k + 1]));
                            const float xa = fmaxf(fmaxf(xa4[0], xa4[1]), fmaxf(xa4[2], xa4[3]));
                            const bool tiny = __all_sync(0xffffffffu, xa * scale_over_cap < kTanhTiny) != 0;
                            if (tiny || __all_sync(0xffffffffu, xa * scale_over_cap < kTanhSmall)) {
                                // tanh by its odd Taylor series on the FMA pipe, two lanes
                                // per instruction: t = x (1 + x^2 (c3 + x^2 (c5 + x^2 c7))),
                                // or t = x (1 + c3 x^2) when every |x| < 1/8
                                const float2 k2 = make_float2(scale_over_cap, scale_over_cap);
                                const float2 c7 = make_float2(kTanhC7, kTanhC7);
                                const float2 c5 = make_float2(kTanhC5, kTanhC5);
                                const float2 c3 = make_float2(kTanhC3, kTanhC3);
                                const float2 one = make_float2(1.f, 1.f);
                                const float2 cc = make_float2(cap2, cap2);
                                const float2 nl22 = make_float2(nl2, nl2);
                                auto run = [&](auto tiny_c) {
                                    constexpr bool kTiny = decltype(tiny_c)::value;
#pragma unroll
                                    for (int c = 0; c < 64; c += 2) {
                                        const float2 x = fmul2(make_float2(s[c], s[c + 1]), k2);
                                        const float2 x2 = fmul2(x, x);
                                        float2 pp;
                                        if (kTiny) {
                                            pp = ffma2(x2, c3, one);
                                        } else {
                                            pp = ffma2(x2, c7, c5);
                                            pp = ffma2(x2, pp, c3);
                                            pp = ffma2(x2, pp, one);
                                        }
                                        const float2 t = fmul2(x, pp);
                                        const float2 a = ffma2(cc, t, nl22);
                                        float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                                        if (partial) {
                                            e.x = ((vis[c >> 5] >> (c & 31)) & 1u) ? e.x : 0.f;
                                            e.y = ((vis[(c + 1) >> 5] >> ((c + 1) & 31)) & 1u) ? e.y : 0.f;
                                        }
                                        const float2 cv = fmul2(e, fsub2(one, fmul2(t, t)));
                                        pf[c] = cv.x;
                                        pf[c + 1] = cv.y;
                                    }
                                };
                                if (tiny) run(std::true_type{});
                                else run(std::false_type{});
                            } else {
#pragma unroll
                                for (int j = 0; j < 64; j += 2) {
                                    float cv[2];
#pragma unroll
                                    for (int z = 0; z < 2; ++z) {
                                        const int c = j + z;
                                        const float t = tanh_fast(s[c] * scale_over_cap);
                                        float e = ex2_approx(fmaf(cap2, t, nl2));
                                        e = ((vis[c >> 5] >> (c & 31)) & 1u) ? e : 0.f;
                                        cv[z] = e * (1.f - t * t);
                                    }
                                    pf[j] = cv[0];
                                    pf[j + 1] = cv[1];
                                }
                            }
                        } else {
                            // masked logits -> -inf, so that 2^(...) = 0 below
                            if (partial) {
#pragma unroll
                                for (int c = 0; c < 64; ++c)
                                    if (!((vis[c >> 5] >> (c & 31)) & 1u)) s[c] = -INFINITY;
                            }
                            const float2 sc2 = make_float2(scale2, scale2);
                            const float2 nl22 = make_float2(nl2, nl2);
#pragma unroll
                            for (int j = 0; j < 64; j += 2) {
                                const float2 x2 = ffma2(make_float2(s[j], s[j + 1]), sc2, nl22);
                                pf[j] = ex2_approx(x2.x);
                                pf[j + 1] = ex2_approx(x2.y);
                            }
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(bars.s_free);
                    // ---- phase B: dS = Pc (dP - Delta), written over this half's dP columns
                    const uint32_t dpc = C::kColDP;
                    if (!(ok = wait_all(bars.dp_full, g & 1))) break;
                    tc_fence_after();
                    {
                        float dpv[64];
                        tmem_ld32(lane_base + dpc + c0, dpv);
                        tmem_ld32(lane_base + dpc + c0 + 32, dpv + 32);
                        tmem_ld_wait();
                        uint32_t pk[32];
                        const float2 dl2 = make_float2(dl, dl);
#pragma unroll
                        for (int j = 0; j < 64; j += 2) {
                            const float2 r = fmul2(make_float2(pf[j], pf[j + 1]),
                                                   fsub2(make_float2(dpv[j], dpv[j + 1]), dl2));
                            pk[j >> 1] = pack_bf16x2(r.x, r.y);
                        }
                        tmem_st32(lane_base + dpc + c0, pk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bars.ds_ready);
                }
                if (!ok) break;
                if (!(ok = wait_all(bars.acc_ready, ua & 1))) break;
                ++ua;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kOH / 32; ++c) {
                    float a[32];
                    tmem_ld32(lane_base + C::kColDQ + o_col + c * 32, a);
                    tmem_ld_wait();
                    if (p.acc_dq) {
                        // ring step: add to the local fp32 dq accumulator
                        float4 *aq4 = reinterpret_cast<float4 *>(
                            p.acc_dq + (((size_t)x.b * p.Lq + qi) * p.Hq + x.h) * D + o_col + c * 32);
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4) {
                            float4 t = aq4[k4];
                            t.x += p.scale * a[4 * k4];
                            t.y += p.scale * a[4 * k4 + 1];
                            t.z += p.scale * a[4 * k4 + 2];
                            t.w += p.scale * a[4 * k4 + 3];
                            aq4[k4] = t;
                        }
                        continue;
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(qrow + c * 32);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        uint4 v;
                        v.x = pack_bf16x2(p.scale * a[8 * k4 + 0], p.scale * a[8 * k4 + 1]);
                        v.y = pack_bf16x2(p.scale * a[8 * k4 + 2], p.scale * a[8 * k4 + 3]);
                        v.z = pack_bf16x2(p.scale * a[8 * k4 + 4], p.scale * a[8 * k4 + 5]);
                        v.w = pack_bf16x2(p.scale * a[8 * k4 + 6], p.scale * a[8 * k4 + 7]);
                        dst[k4] = v;
                    }
                }
            } else if (!p.acc_dq) {
                uint4 *dst = reinterpret_cast<uint4 *>(qrow);
                for (int k4 = 0; k4 < kOH / 8; ++k4) dst[k4] = make_uint4(0, 0, 0, 0);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// dk, dv = sum over the hsplit chunks of the fp32 partials, as bf16; one
// thread per 4 elements (n = B*Lkv*Hkv*D).
__global__ void __launch_bounds__(256) dkv_reduce_kernel(const float *__restrict__ part, int hsplit,
                                                         size_t n, __nv_bfloat16 *__restrict__ dk,
                                                         __nv_bfloat16 *__restrict__ dv)
{
    const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= n) return;
    float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
    for (int c = 0; c < hsplit; ++c) {
        const float4 a = *reinterpret_cast<const float4 *>(part + (size_t)c * n + i);
        const float4 b = *reinterpret_cast<const float4 *>(part + (size_t)(hsplit + c) * n + i);
        sk = make_float4(sk.x + a.x, sk.y + a.y, sk.z + a.z, sk.w + a.w);
        sv = make_float4(sv.x + b.x, sv.y + b.y, sv.z + b.z, sv.w + b.w);
    }
    *reinterpret_cast<uint2 *>(dk + i) = make_uint2(pack_bf16x2(sk.x, sk.y), pack_bf16x2(sk.z, sk.w));
    *reinterpret_cast<uint2 *>(dv + i) = make_uint2(pack_bf16x2(sv.x, sv.y), pack_bf16x2(sv.z, sv.w));
}

} // namespace

int bwd_dkdv_smem_bytes(int D) { return D == 64 ? DkdvCfg<64>::kSmem : DkdvCfg<128>::kSmem; }
int bwd_dq_smem_bytes(int D) { return D == 64 ? DqCfg<64>::kSmem : DqCfg<128>::kSmem; }

template <int D>
cudaError_t bwd_set_attributes_d()
{
    const void *fns[4] = {(const void *)bwd_dkdv_kernel<D, false>, (const void *)bwd_dkdv_kernel<D, true>,
                          (const void *)bwd_dq_kernel<D, false>, (const void *)bwd_dq_kernel<D, true>};
    const int smem[4] = {DkdvCfg<D>::kSmem, DkdvCfg<D>::kSmem, DqCfg<D>::kSmem, DqCfg<D>::kSmem};
    for (int i = 0; i < 4; ++i) {
        // the setmaxnreg split draws on the registers the block is launched
        // with: refuse a build that gives each thread fewer than it assumes
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fns[i]);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < kBwdLaunchRegs) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, smem[i]);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t bwd_tc_set_attributes(int D)
{
    return D == 64 ? bwd_set_attributes_d<64>() : bwd_set_attributes_d<128>();
}

template <int D>
void launch_dkdv_d(const Problem &p, int grid, const CUtensorMap &q, const CUtensorMap &k,
                   const CUtensorMap &v, const CUtensorMap &d, const float *nlse2,
                   const float *delta, __nv_bfloat16 *gk, __nv_bfloat16 *gv, cudaStream_t s)
{
    if (p.soft_cap > 0.f)
        bwd_dkdv_kernel<D, true><<<grid, kBwdThreads, DkdvCfg<D>::kSmem, s>>>(q, k, v, d, p, nlse2, delta, gk, gv);
    else
        bwd_dkdv_kernel<D, false><<<grid, kBwdThreads, DkdvCfg<D>::kSmem, s>>>(q, k, v, d, p, nlse2, delta, gk, gv);
}

template <int D>
void launch_dq_d(const Problem &p, int grid, const CUtensorMap &q, const CUtensorMap &k,
                 const CUtensorMap &v, const CUtensorMap &d, const float *nlse2, const float *delta,
                 __nv_bfloat16 *gq, cudaStream_t s)
{
    if (p.soft_cap > 0.f)
        bwd_dq_kernel<D, true><<<grid, kBwdThreads, DqCfg<D>::kSmem, s>>>(q, k, v, d, p, nlse2, delta, gq);
    else
        bwd_dq_kernel<D, false><<<grid, kBwdThreads, DqCfg<D>::kSmem, s>>>(q, k, v, d, p, nlse2, delta, gq);
}

cudaError_t launch_bwd_dkdv_tc(const Problem &p, const void *tm_q, const void *tm_k,
                               const void *tm_v, const void *tm_do, const float *nlse2,
                               const float *delta, void *dk, void *dv, int num_sms,
                               cudaStream_t s)
{
    const int U = p.B * p.nk * p.Hkv * p.hsplit;
    const int grid = U < num_sms ? U : num_sms;
    const CUtensorMap &q = *static_cast<const CUtensorMap *>(tm_q);
    const CUtensorMap &k = *static_cast<const CUtensorMap *>(tm_k);
    const CUtensorMap &v = *static_cast<const CUtensorMap *>(tm_v);
    const CUtensorMap &d = *static_cast<const CUtensorMap *>(tm_do);
    __nv_bfloat16 *gk = static_cast<__nv_bfloat16 *>(dk), *gv = static_cast<__nv_bfloat16 *>(dv);
    if (p.D == 64)
        launch_dkdv_d<64>(p, grid, q, k, v, d, nlse2, delta, gk, gv, s);
    else
        launch_dkdv_d<128>(p, grid, q, k, v, d, nlse2, delta, gk, gv, s);
    if (p.hsplit > 1) {
        const size_t n = (size_t)p.B * p.Lkv * p.Hkv * p.D;
        const unsigned blocks = (unsigned)((n / 4 + 255) / 256);
        dkv_reduce_kernel<<<blocks, 256, 0, s>>>(p.dkv_part, p.hsplit, n, gk, gv);
    }
    return cudaGetLastError();
}

cudaError_t launch_dkv_reduce(const Problem &p, void *dk, void *dv, cudaStream_t s)
{
    const size_t n = (size_t)p.B * p.Lkv * p.Hkv * p.D;
    const unsigned blocks = (unsigned)((n / 4 + 255) / 256);
    dkv_reduce_kernel<<<blocks, 256, 0, s>>>(p.dkv_part, p.hsplit, n, static_cast<__nv_bfloat16 *>(dk),
                                             static_cast<__nv_bfloat16 *>(dv));
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq_tc(const Problem &p, const void *tm_q, const void *tm_k,
                             const void *tm_v, const void *tm_do, const float *nlse2,
                             const float *delta, void *dq, int num_sms, cudaStream_t s)
{
    const int U = p.B * p.nq * p.Hq;
    const int grid = U < num_sms ? U : num_sms;
    const CUtensorMap &q = *static_cast<const CUtensorMap *>(tm_q);
    const CUtensorMap &k = *static_cast<const CUtensorMap *>(tm_k);
    const CUtensorMap &v = *static_cast<const CUtensorMap *>(tm_v);
    const CUtensorMap &d = *static_cast<const CUtensorMap *>(tm_do);
    __nv_bfloat16 *gq = static_cast<__nv_bfloat16 *>(dq);
    if (p.D == 64)
        launch_dq_d<64>(p, grid, q, k, v, d, nlse2, delta, gq, s);
    else
        launch_dq_d<128>(p, grid, q, k, v, d, nlse2, delta, gq, s);
    return cudaGetLastError();
}

} // namespace ra
