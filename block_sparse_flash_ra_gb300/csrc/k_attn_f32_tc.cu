// k_attn_f32_tc.cu -- forward for RA_FP32 inputs on the tcgen05 tensor cores.
//
// Same schedule as the bf16 forward ("ejKernel ring_attention._ring_splash"
// module source, _ring_attention_forward): per query tile the virtual shards
// are visited in ring order s = (d - t) mod N, empty tiles are skipped from
// the block map, the sink enters on step 0 only, and each shard's normalised
// partial is merged into the running (out, lse) by _update_out_and_lse.
//
// Precision.  The logits decide lse, which is held to 1e-3: one tf32
// rounding of q and k (relative 2^-11 each) moves a logit of this scale by
// a few 1e-4 and the largest of many rows past that bound.  So each fp32
// operand x is split into x_hi = x with its low 13 mantissa bits cleared
// (exact in tf32) and x_lo = x - x_hi (exact in fp32, |x_lo| < 2^-10 |x|),
// and S = Q_hi K_hi^T + Q_hi K_lo^T + Q_lo K_hi^T: three kind::tf32 products
// whose omitted and rounded terms are ~2^-20 relative.  P and V enter the
// output product once each in tf32 (relative 2^-11 per term, far inside the
// output's bound); the softmax, the row sums and the merge run in fp32.
//
// grid (nq, Hq, B), 128 threads: thread t owns query row qt*128 + t, TMEM
// lane t.  Thread 0 issues the products; every step waits for them (a
// correctness path for small problems, not a pipelined one).  Shared
// memory, two 64 KB regions with 128-byte swizzled, K-major tiles:
//   A: Q_hi | Q_lo of one 64-column pass of the head dimension, then P
//   B: K_hi | K_lo of the same pass, then V^T (D rows x 128 keys)
// TMEM: S [0,128), the tile's P V [128,128+D), the running output
// O_run [256,256+D).
//
// Ring step (p.run_out set, one key/value chunk): the running pair starts
// from run_out / run_lse (unless step_first, then (0, -inf)), the sinks count
// only with step_sink, and the merged pair goes back to run_out / run_lse --
// and to `out` as well when it is given (the last step's result in the query
// dtype, which here is fp32).
#include <math.h>

#include "ra_sched.cuh"

namespace ra {
namespace {

constexpr int kRegion = 65536;
constexpr int kF32Smem = 2 * kRegion + 1024 /* kpos, kseg */ + 64 /* barrier, tmem, flag */ + 1024;

// instruction descriptor of kind::tf32: tf32 A and B (format 2), fp32 D,
// both operands K-major
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// generic-proxy stores to shared memory -> visible to the tensor cores
__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// byte offset of element (r, c) of a K-major operand whose rows hold 32
// fp32 per 128-byte swizzled line; column block c / 32 of a `rows`-row
// operand lies rows * 128 bytes after the previous one
__device__ __forceinline__ uint32_t sw_off(int r, int c, int rows)
{
    return (uint32_t)((c >> 5) * rows * 128 + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + (c & 3) * 4);
}

__device__ __forceinline__ float tf32_hi(float x)
{
    return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

template <int D>
__global__ void __launch_bounds__(128, 1) fwd_f32tc_kernel(Problem p, const float *__restrict__ q,
                                                           const float *__restrict__ k,
                                                           const float *__restrict__ v,
                                                           float *__restrict__ out,
                                                           float *__restrict__ lse)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *regA = smem, *regB = smem + kRegion;
    int *kpos = reinterpret_cast<int *>(smem + 2 * kRegion);
    int *kseg = kpos + kTile;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 2 * kRegion + 1024);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bar + 2);
    const WaitCtx ctx{abort_flag, p.status, p.timeout_ns};

    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x, warp = t >> 5;
    if (t == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    constexpr uint32_t kColS = 0, kColPV = 128, kColRun = 256;
    const uint32_t sA = smem_u32(regA), sB = smem_u32(regB);

    const int i = qt * kTile + t;
    const int g = h / p.G;
    const int row_id = b * p.nq + qt;
    const int cnt = p.fwd_cnt[row_id];
    const int32_t *list = p.fwd_idx + (size_t)row_id * p.nk;
    const int dev = qt / p.tq;
    const float *qrow = q + (((size_t)b * p.Lq + i) * p.Hq + h) * D;
    const int my_pos = p.q_pos ? p.q_pos[(size_t)b * p.Lq + i] : i;
    const int my_seg = p.q_seg ? p.q_seg[(size_t)b * p.Lq + i] : 0;
    const bool my_pad = p.q_seg && my_seg == p.pad_id;
    const float scale2 = p.scale * kLog2e;
    const float cap = p.soft_cap;

    uint32_t phase = 0;
    bool ok = true;
    // every product issued so far has completed (thread 0 commits, all wait)
    auto sync_mma = [&]() -> bool {
        if (t == 0) tc_commit(bar);
        const bool r = __syncthreads_and(mbar_wait(bar, phase, ctx) ? 1 : 0) != 0;
        phase ^= 1;
        tc_fence_after();
        return r;
    };

    const bool stepm = p.run_out != nullptr;
    const size_t row_off = (((size_t)b * p.Lq + i) * p.Hq + h) * D;
    float lse_run = -INFINITY;
    bool orun_set = false; // O_run holds real data (else logically zero)
    if (stepm && !p.step_first) {
        // the running pair of the ring so far
        lse_run = p.run_lse[((size_t)b * p.Hq + h) * p.Lq + i];
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t run[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) run[c] = __float_as_uint(p.run_out[row_off + c0 + c]);
            tmem_st32(lane_base + kColRun + c0, run);
        }
        tmem_st_wait();
        orun_set = true;
    }
    for (int step = 0; ok && step < p.N; ++step) {
        const int src = (dev - step + p.N) % p.N;
        const int lo_kt = src * p.tk, hi_kt = lo_kt + p.tk;
        float m = -INFINITY, l = 0.f;
        float o[D];
#pragma unroll
        for (int d = 0; d < D; ++d) o[d] = 0.f;
        bool any_tile = false;
        for (int e = 0; ok && e < cnt; ++e) {
            const int kt = list[e];
            if (kt < lo_kt || kt >= hi_kt) continue;
            any_tile = true;
            const bool partial = p.tile_class[(size_t)row_id * p.nk + kt] == RA_TILE_PARTIAL;
            const int j = kt * kTile + t; // the key row this thread stages
            const float *krow = k + (((size_t)b * p.Lkv + j) * p.Hkv + g) * D;
            const float *vrow = v + (((size_t)b * p.Lkv + j) * p.Hkv + g) * D;
            kpos[t] = p.kv_pos ? p.kv_pos[(size_t)b * p.Lkv + j] : j;
            kseg[t] = p.kv_seg ? p.kv_seg[(size_t)b * p.Lkv + j] : 0;
            // ---- S = Q K^T in passes of 64 head-dim columns, three products each
            for (int pass = 0; pass < D / 64; ++pass) {
                for (int c = 0; c < 64; ++c) {
                    const float xq = qrow[pass * 64 + c], xk = krow[pass * 64 + c];
                    const float qh = tf32_hi(xq), kh = tf32_hi(xk);
                    const uint32_t o_ = sw_off(t, c, kTile);
                    *reinterpret_cast<float *>(regA + o_) = qh;
                    *reinterpret_cast<float *>(regA + 32768 + o_) = xq - qh;
                    *reinterpret_cast<float *>(regB + o_) = kh;
                    *reinterpret_cast<float *>(regB + 32768 + o_) = xk - kh;
                }
                fence_async_smem();
                __syncthreads();
                if (t == 0) {
                    tc_fence_after();
                    const uint64_t qh_d = sdesc_sw128(sA, 16, 1024), ql_d = sdesc_sw128(sA + 32768, 16, 1024);
                    const uint64_t kh_d = sdesc_sw128(sB, 16, 1024), kl_d = sdesc_sw128(sB + 32768, 16, 1024);
                    const uint64_t a_[3] = {qh_d, qh_d, ql_d}, b_[3] = {kh_d, kl_d, kh_d};
                    for (int pr = 0; pr < 3; ++pr)
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = ((kk & 3) * 32 + (kk >> 2) * 16384) >> 4;
                            mma_tf32_ss(tmem + kColS, a_[pr] + off, b_[pr] + off, idesc_tf32(128, 128),
                                        (pass > 0 || pr > 0 || kk > 0) ? 1u : 0u);
                        }
                }
                if (!(ok = sync_mma())) break; // the regions are free again
            }
            if (!ok) break;
            // ---- online softmax over the tile: max first, then P into region A
            float x2[kTile];
            float mt = -INFINITY;
            for (int c0 = 0; c0 < kTile; c0 += 32) {
                float s[32];
                tmem_ld32(lane_base + kColS + c0, s);
                tmem_ld_wait();
                for (int c = 0; c < 32; ++c) {
                    const int jj = c0 + c;
                    bool vis = true;
                    if (partial) {
                        vis = (kseg[jj] == my_seg) && !my_pad;
                        if (p.causal) vis = vis && (my_pos >= kpos[jj]);
                        if (p.local_mask)
                            vis = vis && p.local_mask[(size_t)(i % p.lq_s) * p.lk_s +
                                                      (kt * kTile + jj) % p.lk_s] != 0;
                    }
                    const float y = cap > 0.f ? cap * kLog2e * tanhf(s[c] * p.scale / cap) : s[c] * scale2;
                    x2[jj] = vis ? y : -INFINITY;
                    mt = fmaxf(mt, x2[jj]);
                }
            }
            const float m_new = fmaxf(m, mt);
            const float f = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
            float lt = 0.f;
            for (int jj = 0; jj < kTile; ++jj) {
                const float pj = (x2[jj] == -INFINITY) ? 0.f : exp2f(x2[jj] - m_new);
                lt += pj;
                *reinterpret_cast<float *>(regA + sw_off(t, jj, kTile)) = pj;
            }
            // V^T: this thread's key row t becomes column t of the D x 128 operand
            for (int d = 0; d < D; ++d)
                *reinterpret_cast<float *>(regB + sw_off(d, t, D)) = vrow[d];
            fence_async_smem();
            __syncthreads();
            if (t == 0) {
                tc_fence_after();
                const uint64_t pd = sdesc_sw128(sA, 16, 1024), vd = sdesc_sw128(sB, 16, 1024);
                for (int kk = 0; kk < kTile / 8; ++kk)
                    mma_tf32_ss(tmem + kColPV, pd + (((kk & 3) * 32 + (kk >> 2) * 16384) >> 4),
                                vd + (((kk & 3) * 32 + (kk >> 2) * D * 128) >> 4), idesc_tf32(128, D),
                                kk > 0 ? 1u : 0u);
            }
            if (!(ok = sync_mma())) break;
            for (int c0 = 0; c0 < D; c0 += 32) {
                float pv[32];
                tmem_ld32(lane_base + kColPV + c0, pv);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c0 + c] = o[c0 + c] * f + pv[c];
            }
            l = l * f + lt;
            m = m_new;
            tc_fence_before();
            __syncthreads(); // P V read from TMEM before the next tile's products
            tc_fence_after();
        }
        if (!ok) break;
        const bool sink_here = (step == 0) && p.sinks && (!stepm || p.step_sink);
        if (!any_tile && !sink_here) continue; // partial (0, -inf): merge is a no-op
        if (sink_here) {
            const float s2 = p.sinks[h] * kLog2e;
            if (s2 > m) {
                const float fs = (m == -INFINITY) ? 0.f : exp2f(m - s2);
                l *= fs;
#pragma unroll
                for (int d = 0; d < D; ++d) o[d] *= fs;
                m = s2;
            }
            l += exp2f(s2 - m);
        }
        float lse_s, inv;
        if (l > 0.f) {
            lse_s = (m + log2f(l)) * kLn2;
            inv = 1.f / l;
        } else {
            lse_s = -INFINITY;
            inv = 0.f;
        }
        // _update_out_and_lse into O_run (TMEM lane t)
        const bool first = (lse_run == -INFINITY);
        const float x = lse_s - lse_run;
        const float w = first ? 1.f : (x >= 0.f ? 1.f / (1.f + expf(-x)) : expf(x) / (1.f + expf(x)));
        for (int c0 = 0; c0 < D; c0 += 32) {
            float run[32];
            tmem_ld32(lane_base + kColRun + c0, run);
            tmem_ld_wait();
            uint32_t nw[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float blk = o[c0 + c] * inv;
                const float cur = (orun_set && !first) ? run[c] : 0.f;
                nw[c] = __float_as_uint(first ? blk : cur - w * (cur - blk));
            }
            tmem_st32(lane_base + kColRun + c0, nw);
        }
        tmem_st_wait();
        lse_run = first ? lse_s : lse_run + (fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
        orun_set = true;
    }
    // a wait that gave up leaves the last commit pending: let it land (bounded)
    // before the TMEM it writes is freed
    if (!ok && t == 0) wait_drain(bar, phase ^ 1, kDrainNs);
    if (ok) {
        float *dst = out ? out + row_off : nullptr;
        float *dst_run = stepm ? p.run_out + row_off : nullptr;
        for (int c0 = 0; c0 < D; c0 += 32) {
            float run[32];
            tmem_ld32(lane_base + kColRun + c0, run);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float val = orun_set ? run[c] : 0.f;
                if (dst) dst[c0 + c] = val;
                if (dst_run) dst_run[c0 + c] = val;
            }
        }
        lse[((size_t)b * p.Hq + h) * p.Lq + i] = lse_run;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

} // namespace

cudaError_t f32tc_set_attributes(int D)
{
    if (D == 64)
        return cudaFuncSetAttribute(fwd_f32tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kF32Smem);
    return cudaFuncSetAttribute(fwd_f32tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kF32Smem);
}

cudaError_t launch_fwd_f32_tc(const Problem &p, const float *q, const float *k, const float *v,
                              float *out, float *lse, cudaStream_t s)
{
    const dim3 grid(p.nq, p.Hq, p.B);
    if (p.D == 64)
        fwd_f32tc_kernel<64><<<grid, 128, kF32Smem, s>>>(p, q, k, v, out, lse);
    else
        fwd_f32tc_kernel<128><<<grid, 128, kF32Smem, s>>>(p, q, k, v, out, lse);
    return cudaGetLastError();
}

} // namespace ra
