// k_attn_bwd64_tc.cu -- the dK/dV stage of the backward on its own tile shape:
// 128 kv rows x 64 query rows per step (block_kv_dkv = 128, block_q_dkv = 64,
// "ejKernel ring_attention._ring_splash" module source, make_ring_attention
// with block_sizes.has_backward_blocks), walking the dkv block map of that
// grid (ra_block_mask dkv_*), for D = 128.
//
// What it computes is the dK/dV part of _ring_attention_backward's gradient
// (the final out and lse, Delta = <dO, O>):
//   dV_j = sum_i P_ij dO_i          dK_j = scale sum_i dS_ij Q_i
//   P = exp(s - lse), dS = P (dP - Delta) (1 - tanh^2 with a soft cap)
// summed over the query heads of a kv head (GQA / MQA).
//
// Design (one CTA per SM, persistent, one unit per (b, kv head, kv tile,
// chunk of query heads), longest column first):
//   warps 0-3  softmax-gradient of the even steps, warps 4-7 of the odd
//              steps: thread t owns kv row t and all 64 query columns of its
//              step.  The two warpgroups work on consecutive steps at once,
//              so one's exponent phase overlaps the other's waits.
//   warp 8     TMA producer: K, V once per unit; Q, dO (64-row blocks),
//              -lse*log2 e and Delta per step into a 4-stage ring
//   warp 9     TMEM owner and MMA issuer
//   warps 10-11 no role (setmaxnreg donors)
// TMEM: S^T of even / odd steps [0,64) / [64,128), dP^T [128,192) /
// [192,256), dV [256,384), dK [384,512).  P^T and dS^T (bf16) overwrite the
// first 32 columns of their fp32 buffers and feed dV += P^T dO and
// dK += dS^T Q from TMEM.  Issue order per step n: dV(n), dK(n), then S^T and
// dP^T of step n + 2 into the buffers step n has just released -- the products
// of step n + 1 were issued a step earlier, so its warpgroup never waits for
// step n's.
#include <math.h>
#include <type_traits>

#include "ra_sched.cuh"

namespace ra {
namespace {

constexpr int kQB = 64;                     // query rows per step
constexpr int kD64 = 128;                   // head dim served
constexpr int kBlk = kQB * kD64 * 2;        // one 64-row bf16 block (16 KB)
constexpr int kKvTile = kTile * kD64 * 2;   // one 128-row bf16 tile (32 KB)
constexpr int kStages64 = 4;
constexpr int kThreads64 = 384;
constexpr int kProducer64 = 8;
constexpr int kMma64 = 9;
// setmaxnreg split as the other backward kernels: 176 for the softmax-gradient
// warpgroups, 152 for the producer / MMA warpgroup, over 168 at launch
constexpr int kLaunchRegs64 = 168;
constexpr uint32_t kSoftRegs64 = 176;
constexpr uint32_t kSideRegs64 = 152;
static_assert(256 * kSoftRegs64 + 128 * kSideRegs64 <= kThreads64 * kLaunchRegs64,
              "register split exceeds the block's launch registers");

struct Cfg64 {
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKvTile;
    static constexpr int kStageBytes = 2 * kBlk + 1024; // Q, dO, nlse2[64], delta[64], padding
    static constexpr int kStageOff = 2 * kKvTile;
    static constexpr int kBarOff = kStageOff + kStages64 * kStageBytes;
    // kv_full, kv_empty, st_full[4], st_empty[4], s_full[2], dp_full[2],
    // p_ready[2], ds_ready[2], acc_ready, drain
    static constexpr int kNumBars = 2 + 2 * kStages64 + 8 + 2;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmem = kMiscOff + 16 + 1024;
    static_assert(kSmem <= 232448, "dK/dV shared memory exceeds the 227 KB per-block limit");
    static constexpr uint32_t kColDP = 128, kColDV = 256, kColDK = 384;
    static constexpr uint32_t kIdescT = idesc_bf16(128, kQB, false, false); // S^T, dP^T
    static constexpr uint32_t kIdescAcc = idesc_bf16(128, kD64, false, true); // dV, dK
};

struct Bars64 {
    uint64_t *kv_full, *kv_empty, *st_full, *st_empty, *s_full, *dp_full, *p_ready, *ds_ready,
        *acc_ready, *drain;
};

__device__ __forceinline__ Bars64 bars64(uint8_t *smem)
{
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + Cfg64::kBarOff);
    Bars64 r;
    r.kv_full = b;
    r.kv_empty = b + 1;
    r.st_full = b + 2;
    r.st_empty = r.st_full + kStages64;
    r.s_full = r.st_empty + kStages64; // [buffer]
    r.dp_full = r.s_full + 2;
    r.p_ready = r.dp_full + 2;
    r.ds_ready = r.p_ready + 2;
    r.acc_ready = r.ds_ready + 2;
    r.drain = r.acc_ready + 1;
    return r;
}

// Work unit: (kv tile column, kv head, chunk of its query heads) over the
// column's non-empty 64-row query blocks.
struct Col64 {
    int b, kt, hkv, col, cnt, chunk, h0, gc;
    const int32_t *list, *slot;
};

__device__ __forceinline__ Col64 col64_of(const Problem &p, int u)
{
    Col64 x;
    const int per = p.Hkv * p.hsplit;
    x.col = p.dkv_order[u / per];
    const int r = u - (u / per) * per;
    x.hkv = r / p.hsplit;
    x.chunk = r - x.hkv * p.hsplit;
    x.gc = p.G / p.hsplit;
    x.h0 = x.hkv * p.G + x.chunk * x.gc;
    x.b = x.col / p.nk;
    x.kt = x.col - x.b * p.nk;
    x.cnt = p.dkv_cnt[x.col];
    x.list = p.dkv_idx + (size_t)x.col * 2 * p.nq;
    x.slot = p.dkv_slot + (size_t)x.col * 2 * p.nq;
    return x;
}

template <bool CAP>
__global__ void __launch_bounds__(kThreads64, 1)
    bwd_dkdv64_kernel(const __grid_constant__ CUtensorMap tm_q64, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do64,
                      Problem p, const float *__restrict__ nlse2, const float *__restrict__ delta,
                      __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv)
{
    using C = Cfg64;
    constexpr int D = kD64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const Bars64 bars = bars64(smem);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
    const WaitCtx ctx{abort_flag, p.status, p.timeout_ns};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = p.B * p.nk * p.Hkv * p.hsplit;
    const int Gd = gridDim.x;

    if (threadIdx.x == 0) {
        mbar_init(bars.kv_full, 1);
        mbar_init(bars.kv_empty, 1);
        for (int s = 0; s < kStages64; ++s) {
            mbar_init(bars.st_full + s, 1);
            mbar_init(bars.st_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.s_full + b, 1);
            mbar_init(bars.dp_full + b, 1);
            mbar_init(bars.p_ready + b, 128);
            mbar_init(bars.ds_ready + b, 128);
        }
        mbar_init(bars.acc_ready, 1);
        mbar_init(bars.drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMma64) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    if (warp == kProducer64 && lane == 0) {
        prefetch_tmap(&tm_q64);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do64);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp >= kProducer64) {
        regs_shrink<kSideRegs64>();
        if (warp == kProducer64 && lane == 0) {
            // ---------------------------------------------------------- producer
            uint32_t n = 0, uk = 0;
            uint32_t st_issued[kStages64] = {};
            bool ok = true;
            for (int r = 0; ok && r * Gd < U; ++r) {
                const int u = unit_index(r, blockIdx.x, Gd);
                if (u >= U) continue;
                const Col64 x = col64_of(p, u);
                if (x.cnt == 0) continue;
                if (!(ok = mbar_wait(bars.kv_empty, (uk & 1) ^ 1, ctx))) break;
                mbar_expect_tx(bars.kv_full, 2 * kKvTile);
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
                        const int qb = x.list[e];
                        const int st = n % kStages64;
                        if (!(ok = mbar_wait(bars.st_empty + st, ((n / kStages64) & 1) ^ 1, ctx))) break;
                        uint8_t *sb = smem + C::kStageOff + st * C::kStageBytes;
                        mbar_expect_tx(bars.st_full + st, 2 * kBlk + 512);
                        for (int hb = 0; hb < D / 64; ++hb) {
                            tma_load_4d(sb + hb * 8192, &tm_q64, bars.st_full + st, hb * 64, h,
                                        qb * kQB, x.b);
                            tma_load_4d(sb + kBlk + hb * 8192, &tm_do64, bars.st_full + st, hb * 64, h,
                                        qb * kQB, x.b);
                        }
                        const size_t li = ((size_t)x.b * p.Hq + h) * p.Lq + (size_t)qb * kQB;
                        bulk_load(sb + 2 * kBlk, nlse2 + li, 256, bars.st_full + st);
                        bulk_load(sb + 2 * kBlk + 256, delta + li, 256, bars.st_full + st);
                        ++st_issued[st];
                        ++n;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < kStages64; ++s)
                    if (st_issued[s]) wait_drain(bars.st_full + s, (st_issued[s] - 1) & 1, kDrainNs);
                if (uk) wait_drain(bars.kv_full, (uk - 1) & 1, kDrainNs);
            }
        } else if (warp == kMma64) {
            // ---------------------------------------------------------- MMA issuer
            // The whole warp runs the issue loop, converged: every lane waits on
            // the barriers, and one lane, chosen by elect.sync, issues each
            // product and commit.
            auto wait_w = [&](uint64_t *bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
            };
            // descriptors built once per operand; an offset o adds o / 16
            const uint64_t kd = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
            const uint64_t vd = sdesc_sw128(smem_u32(smem + C::kVOff), 16, 1024);
            const uint32_t stage0 = smem_u32(smem + C::kStageOff);
            uint32_t n = 0, uk = 0;
            bool ok = true;
            auto wait_stage = [&](uint32_t step) -> bool {
                if (!wait_w(bars.st_full + step % kStages64, (step / kStages64) & 1)) return false;
                tc_fence_after();
                return true;
            };
            // S^T = K Q^T and dP^T = V dO^T of a step into its buffer pair
            auto issue_sdp = [&](uint32_t step) {
                const uint32_t sb = stage0 + (step % kStages64) * C::kStageBytes;
                const uint64_t qd = sdesc_sw128(sb, 16, 1024), dd = sdesc_sw128(sb + kBlk, 16, 1024);
                const uint32_t buf = step & 1;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                    mma_ss_w(tmem + buf * 64, kd + oa, qd + ob, C::kIdescT, kk > 0 ? 1u : 0u);
                }
                tc_commit_w(bars.s_full + buf);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                    mma_ss_w(tmem + C::kColDP + buf * 64, vd + oa, dd + ob, C::kIdescT, kk > 0 ? 1u : 0u);
                }
                tc_commit_w(bars.dp_full + buf);
            };
            for (int r = 0; ok && r * Gd < U; ++r) {
                const int u = unit_index(r, blockIdx.x, Gd);
                if (u >= U) continue;
                const Col64 x = col64_of(p, u);
                if (x.cnt == 0) continue;
                if (!(ok = wait_w(bars.kv_full, uk & 1))) break;
                tc_fence_after();
                ++uk;
                const int steps = x.gc * x.cnt;
                for (int j = 0; ok && j < 2 && j < steps; ++j) {
                    if (!(ok = wait_stage(n + j))) break;
                    issue_sdp(n + j);
                }
                for (int i = 0; ok && i < steps; ++i, ++n) {
                    const uint32_t buf = n & 1, ph = (n >> 1) & 1;
                    const uint32_t sb = stage0 + (n % kStages64) * C::kStageBytes;
                    // dV += P^T dO   (A = P^T from TMEM, B = dO as a K=q x N=D MN-major block)
                    if (!(ok = wait_w(bars.p_ready + buf, ph))) break;
                    tc_fence_after();
                    const uint64_t dmn = sdesc_sw128(sb + kBlk, 8192, 1024);
#pragma unroll
                    for (int kk = 0; kk < kQB / 16; ++kk)
                        mma_ts_w(tmem + C::kColDV, tmem + buf * 64 + kk * 8,
                               dmn + (uint32_t)((kk * 2048) >> 4), C::kIdescAcc,
                               (i > 0 || kk > 0) ? 1u : 0u);
                    // dK += dS^T Q
                    if (!(ok = wait_w(bars.ds_ready + buf, ph))) break;
                    tc_fence_after();
                    const uint64_t qmn = sdesc_sw128(sb, 8192, 1024);
#pragma unroll
                    for (int kk = 0; kk < kQB / 16; ++kk)
                        mma_ts_w(tmem + C::kColDK, tmem + C::kColDP + buf * 64 + kk * 8,
                               qmn + (uint32_t)((kk * 2048) >> 4), C::kIdescAcc,
                               (i > 0 || kk > 0) ? 1u : 0u);
                    tc_commit_w(bars.st_empty + n % kStages64);
                    // the next products of this buffer pair: step n + 2
                    if (i + 2 < steps) {
                        if (!(ok = wait_stage(n + 2))) break;
                        issue_sdp(n + 2);
                    }
                }
                if (!ok) break;
                tc_commit_w(bars.kv_empty);
                tc_commit_w(bars.acc_ready);
            }
            tc_commit_w(bars.drain);
            wait_drain(bars.drain, 0, kDrainNs);
        }
    } else {
        regs_grow<kSoftRegs64>();
        // ---------------------------------------------------------- softmax-grad
        // Warpgroup wb takes the steps n with n % 2 == wb; thread t owns kv
        // row 32*(w%4)+lane and the 64 query columns of its step, and D/2
        // columns of dK, dV in the epilogue.
        const int wb = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool split = p.hsplit > 1;
        float *part_k = p.dkv_part;
        float *part_v = split ? p.dkv_part + (size_t)p.hsplit * p.B * p.Lkv * p.Hkv * D : nullptr;
        constexpr int kOH = D / 2;
        const uint32_t o_col = wb * kOH;
        const float scale2 = p.scale * kLog2e;
        const float cap = CAP ? p.soft_cap : 0.f;
        const float cap2 = cap * kLog2e;
        const float scale_over_cap = cap > 0.f ? p.scale / cap : 0.f;
        const uint32_t col_s = wb * 64, col_dp = C::kColDP + wb * 64;
        uint32_t n = 0, ua = 0;
        bool ok = true;
        auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx)) != 0;
        };
        for (int r = 0; ok && r * Gd < U; ++r) {
            const int u = unit_index(r, blockIdx.x, Gd);
            if (u >= U) continue;
            const Col64 x = col64_of(p, u);
            const int kj = x.kt * kTile + row;
            const size_t orow = (((size_t)x.b * p.Lkv + kj) * p.Hkv + x.hkv) * D + o_col;
            const size_t prow = (size_t)x.chunk * p.B * p.Lkv * p.Hkv * D + orow;
            if (x.cnt > 0) {
                const int my_pos = p.kv_pos ? p.kv_pos[(size_t)x.b * p.Lkv + kj] : kj;
                const int my_seg = p.kv_seg ? p.kv_seg[(size_t)x.b * p.Lkv + kj] : 0;
                const int steps = x.gc * x.cnt;
                for (int i = 0; i < steps; ++i, ++n) {
                    if ((n & 1) != (uint32_t)wb) continue;
                    const int e = i % x.cnt;
                    const int qb = x.list[e];
                    const int st = n % kStages64;
                    const uint32_t ph = (n >> 1) & 1;
                    const float *lse_s = reinterpret_cast<const float *>(
                        smem + C::kStageOff + st * C::kStageBytes + 2 * kBlk);
                    const float *dl_s = lse_s + kQB;
                    const bool partial =
                        p.dkv_class[((size_t)x.b * 2 * p.nq + qb) * p.nk + x.kt] == RA_TILE_PARTIAL;
                    // ---- visibility of the step's 64 query columns (partial blocks only):
                    // words 2h, 2h+1 of the parent tile's stored column bits
                    uint32_t vis[2] = {~0u, ~0u};
                    if (partial) {
                        const uint2 vb = col_bits(p, x.slot[e], row, qb & 1, x.b, qb * kQB, kj, my_seg,
                                                  my_pos);
                        vis[0] = vb.x;
                        vis[1] = vb.y;
                    }
                    if (!(ok = wait_all(bars.s_full + wb, ph))) break;
                    tc_fence_after();
                    // ---- P^T (bf16 -> TMEM) and Pc = P * (1 - tanh^2) kept packed
                    uint32_t pc[32];
                    {
                        float s[64];
                        tmem_ld32(lane_base + col_s, s);
                        tmem_ld32(lane_base + col_s + 32, s + 32);
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
                                // per instruction
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
                                            const float2 xx = fmul2(make_float2(s[c], s[c + 1]), k2);
                                            const float2 x2 = fmul2(xx, xx);
                                            float2 pp;
                                            if (kTiny) {
                                                pp = ffma2(x2, c3, one);
                                            } else {
                                                pp = ffma2(x2, c7, c5);
                                                pp = ffma2(x2, pp, c3);
                                                pp = ffma2(x2, pp, one);
                                            }
                                            const float2 t = fmul2(xx, pp);
                                            const float2 a = ffma2(cc, t, la[h]);
                                            float2 ev = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                                            if (partial) {
                                                ev.x = ((vis[c >> 5] >> (c & 31)) & 1u) ? ev.x : 0.f;
                                                ev.y = ((vis[(c + 1) >> 5] >> ((c + 1) & 31)) & 1u) ? ev.y : 0.f;
                                            }
                                            const float2 cr = fmul2(ev, fsub2(one, fmul2(t, t)));
                                            pk[c >> 1] = pack_bf16x2(ev.x, ev.y);
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
                                        float ev = ex2_approx(fmaf(cap2, t, la[z]));
                                        ev = ((vis[c >> 5] >> (c & 31)) & 1u) ? ev : 0.f;
                                        pr[z] = ev;
                                        cr[z] = ev * (1.f - t * t);
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
                        // P^T over the S^T columns just read
                        tmem_st32(lane_base + col_s, pk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bars.p_ready + wb);
                    // ---- dS^T = Pc (dP^T - Delta)
                    if (!(ok = wait_all(bars.dp_full + wb, ph))) break;
                    tc_fence_after();
                    {
                        float dpv[64];
                        tmem_ld32(lane_base + col_dp, dpv);
                        tmem_ld32(lane_base + col_dp + 32, dpv + 32);
                        tmem_ld_wait();
                        const float4 *d4 = reinterpret_cast<const float4 *>(dl_s);
                        uint32_t dk2[32];
#pragma unroll
                        for (int j = 0; j < 64; j += 4) {
                            const float4 dl = d4[j >> 2];
                            const float2 r0 = fsub2(make_float2(dpv[j], dpv[j + 1]), make_float2(dl.x, dl.y));
                            const float2 r1 = fsub2(make_float2(dpv[j + 2], dpv[j + 3]), make_float2(dl.z, dl.w));
                            dk2[j >> 1] = mul_bf16x2(pc[j >> 1], pack_bf16x2(r0.x, r0.y));
                            dk2[(j >> 1) + 1] = mul_bf16x2(pc[(j >> 1) + 1], pack_bf16x2(r1.x, r1.y));
                        }
                        tmem_st32(lane_base + col_dp, dk2);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bars.ds_ready + wb);
                }
                if (!ok) break;
                // ---- epilogue: this warpgroup's half of dV and scale * dK -> bf16
                // (a head split: the chunk's fp32 partials; ring steps and fp32
                // inputs: added to the fp32 accumulators)
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
                        uint4 v4, w4;
                        v4.x = pack_bf16x2(a[8 * k4 + 0], a[8 * k4 + 1]);
                        v4.y = pack_bf16x2(a[8 * k4 + 2], a[8 * k4 + 3]);
                        v4.z = pack_bf16x2(a[8 * k4 + 4], a[8 * k4 + 5]);
                        v4.w = pack_bf16x2(a[8 * k4 + 6], a[8 * k4 + 7]);
                        w4.x = pack_bf16x2(p.scale * bk[8 * k4 + 0], p.scale * bk[8 * k4 + 1]);
                        w4.y = pack_bf16x2(p.scale * bk[8 * k4 + 2], p.scale * bk[8 * k4 + 3]);
                        w4.z = pack_bf16x2(p.scale * bk[8 * k4 + 4], p.scale * bk[8 * k4 + 5]);
                        w4.w = pack_bf16x2(p.scale * bk[8 * k4 + 6], p.scale * bk[8 * k4 + 7]);
                        dvp[k4] = v4;
                        dkp[k4] = w4;
                    }
                }
            } else if (p.acc_dk) {
                // a column with nothing visible adds nothing
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
    if (warp == kMma64) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

} // namespace

cudaError_t bwd_dkdv64_set_attributes()
{
    const void *fns[2] = {(const void *)bwd_dkdv64_kernel<false>, (const void *)bwd_dkdv64_kernel<true>};
    for (const void *fn : fns) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < kLaunchRegs64) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg64::kSmem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_bwd_dkdv64_tc(const Problem &p, const void *tm_q64, const void *tm_k,
                                 const void *tm_v, const void *tm_do64, const float *nlse2,
                                 const float *delta, void *dk, void *dv, int num_sms,
                                 cudaStream_t s)
{
    const int U = p.B * p.nk * p.Hkv * p.hsplit;
    const int grid = U < num_sms ? U : num_sms;
    const CUtensorMap &q = *static_cast<const CUtensorMap *>(tm_q64);
    const CUtensorMap &k = *static_cast<const CUtensorMap *>(tm_k);
    const CUtensorMap &v = *static_cast<const CUtensorMap *>(tm_v);
    const CUtensorMap &d = *static_cast<const CUtensorMap *>(tm_do64);
    __nv_bfloat16 *gk = static_cast<__nv_bfloat16 *>(dk), *gv = static_cast<__nv_bfloat16 *>(dv);
    if (p.soft_cap > 0.f)
        bwd_dkdv64_kernel<true><<<grid, kThreads64, Cfg64::kSmem, s>>>(q, k, v, d, p, nlse2, delta, gk, gv);
    else
        bwd_dkdv64_kernel<false><<<grid, kThreads64, Cfg64::kSmem, s>>>(q, k, v, d, p, nlse2, delta, gk, gv);
    return cudaGetLastError();
}

} // namespace ra
