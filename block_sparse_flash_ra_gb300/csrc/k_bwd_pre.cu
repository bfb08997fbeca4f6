// k_bwd_pre.cu -- backward preprocessing ("ejKernel ring_attention._ring_splash"
// module source, _ring_attention_backward: dO widened to fp32, dsinks
// accumulated and summed over the ring):
//   Delta[b, h, i] = <dO[b, i, h, :], O[b, i, h, :]>           (fp32)
//   dsinks[h]      = - sum_{b, i} exp(sink_h - lse[b, h, i]) * Delta[b, h, i]
// and, for the gradient kernels, nlse2[b, h, i] = -lse * log2(e): the
// exponent offset of P = 2^(s * scale * log2 e + nlse2).  A row with nothing
// visible (lse = -inf) gets 0 instead of +inf; all its entries are masked, so
// its P stays 0 and no inf - inf can arise.
// The dsinks sum is taken in two deterministic passes over Delta and lse:
// per-(b, head, q-tile) partials, then one block per head.  HBM-bound: reads
// O and dO once.
#include <cuda_bf16.h>

#include "ra_internal.h"

namespace ra {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x)
{
    return x;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}

// Delta and nlse2 of any dtype and D: grid (Hq, nq, B), 128 threads, warp w
// handles rows w, w+4, ... of one head's query tile.
template <typename T>
__global__ void __launch_bounds__(128) bwd_pre_kernel(Problem p, const T *__restrict__ out,
                                                      const T *__restrict__ dout,
                                                      const float *__restrict__ lse,
                                                      float *__restrict__ delta,
                                                      float *__restrict__ nlse2)
{
    const int h = blockIdx.x, qt = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int r = wid; r < kTile; r += 4) {
        const int i = qt * kTile + r;
        const size_t row = (((size_t)b * p.Lq + i) * p.Hq + h) * p.D;
        float acc = 0.f;
        for (int d = lane; d < p.D; d += 32) acc += to_f(out[row + d]) * to_f(dout[row + d]);
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        const size_t li = ((size_t)b * p.Hq + h) * p.Lq + i;
        if (lane == 0) {
            delta[li] = acc;
            const float l = lse[li];
            nlse2[li] = (l == -INFINITY) ? 0.f : -l * 1.4426950408889634f;
        }
    }
}

// The same for bf16 rows, one warp per token (b, i): the token's Hq rows of O
// and of dO are each one contiguous stretch of Hq * D bf16, streamed in
// 16-byte chunks with kU chunks of each tensor in flight per lane; D/8
// adjacent lanes hold one head's row and reduce it with shuffles.  8 tokens
// per block of 256 threads.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_bf16_kernel(Problem p, const __nv_bfloat16 *__restrict__ out,
                                                           const __nv_bfloat16 *__restrict__ dout,
                                                           const float *__restrict__ lse,
                                                           float *__restrict__ delta,
                                                           float *__restrict__ nlse2)
{
    constexpr int kLanes = D / 8; // lanes per head row
    constexpr int kU = 4;
    const int lane = threadIdx.x & 31;
    const long long toks = (long long)p.B * p.Lq;
    const long long t = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= toks) return;
    const int b = (int)(t / p.Lq), i = (int)(t - (long long)b * p.Lq);
    const int n16 = p.Hq * kLanes;
    const uint4 *o16 = reinterpret_cast<const uint4 *>(out) + t * n16;
    const uint4 *g16 = reinterpret_cast<const uint4 *>(dout) + t * n16;
    const size_t lrow = (size_t)b * p.Hq * p.Lq + i; // head h at lrow + h * Lq
    for (int f0 = 0; f0 < n16; f0 += 32 * kU) {
        uint4 o[kU], g[kU];
        float lv[kU]; // the head's lse, loaded by the lane that stores its row
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int f = f0 + u * 32 + lane;
            lv[u] = 0.f;
            if (f < n16) {
                o[u] = __ldg(o16 + f);
                g[u] = __ldg(g16 + f);
                if (f % kLanes == 0) lv[u] = lse[lrow + (size_t)(f / kLanes) * p.Lq];
            } else {
                o[u] = make_uint4(0u, 0u, 0u, 0u);
                g[u] = o[u];
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const uint32_t ow[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
            const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc = fmaf(__uint_as_float(ow[j] << 16), __uint_as_float(gw[j] << 16), acc);
                acc = fmaf(__uint_as_float(ow[j] & 0xffff0000u), __uint_as_float(gw[j] & 0xffff0000u), acc);
            }
#pragma unroll
            for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const int f = f0 + u * 32 + lane;
            if (f < n16 && f % kLanes == 0) {
                const size_t li = lrow + (size_t)(f / kLanes) * p.Lq;
                delta[li] = acc;
                nlse2[li] = (lv[u] == -INFINITY) ? 0.f : -lv[u] * 1.4426950408889634f;
            }
        }
    }
}

// dsinks partial sums, one warp per (b, head, query tile): the tile's 128
// rows of Delta and lse (contiguous in the (B, Hq, Lq) layout) in float4,
// part[h][b][qt] = sum over the rows of exp(sink_h - lse) * Delta.
__global__ void __launch_bounds__(32) dsink_part_kernel(Problem p, const float *__restrict__ lse,
                                                        const float *__restrict__ delta,
                                                        float *__restrict__ part)
{
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x;
    const float sink = p.sinks[h];
    const size_t base = ((size_t)b * p.Hq + h) * p.Lq + (size_t)qt * kTile;
    const float4 l4 = reinterpret_cast<const float4 *>(lse + base)[lane];
    const float4 d4 = reinterpret_cast<const float4 *>(delta + base)[lane];
    const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
    float ds = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (lv[j] != -INFINITY) ds += __expf(sink - lv[j]) * dv[j];
    for (int off = 16; off > 0; off >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, off);
    if (lane == 0) part[(size_t)h * p.B * p.nq + (size_t)b * p.nq + qt] = ds;
}

// one block per head: dsinks[h] = -sum of its partials (fixed order)
__global__ void __launch_bounds__(256) dsink_reduce_kernel(const float *part, int n, float *dsinks)
{
    const int h = blockIdx.x;
    float s = 0.f;
    for (int i = threadIdx.x; i < n; i += 256) s += part[(size_t)h * n + i];
    __shared__ float w[256];
    w[threadIdx.x] = s;
    __syncthreads();
    for (int k = 128; k > 0; k >>= 1) {
        if ((int)threadIdx.x < k) w[threadIdx.x] += w[threadIdx.x + k];
        __syncthreads();
    }
    if (threadIdx.x == 0) dsinks[h] = -w[0];
}

} // namespace

cudaError_t launch_bwd_pre(const Problem &p, const void *out, const void *dout, int dtype,
                           const float *lse, float *delta, float *nlse2, float *dsink_part,
                           float *dsinks, cudaStream_t s)
{
    const dim3 grid(p.Hq, p.nq, p.B);
    const __nv_bfloat16 *ob = static_cast<const __nv_bfloat16 *>(out);
    const __nv_bfloat16 *gb = static_cast<const __nv_bfloat16 *>(dout);
    const unsigned tok_blocks = (unsigned)(((long long)p.B * p.Lq + 7) / 8);
    if (dtype == RA_BF16 && p.D == 128)
        bwd_pre_bf16_kernel<128><<<tok_blocks, 256, 0, s>>>(p, ob, gb, lse, delta, nlse2);
    else if (dtype == RA_BF16 && p.D == 64)
        bwd_pre_bf16_kernel<64><<<tok_blocks, 256, 0, s>>>(p, ob, gb, lse, delta, nlse2);
    else if (dtype == RA_BF16)
        bwd_pre_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(p, ob, gb, lse, delta, nlse2);
    else
        bwd_pre_kernel<float><<<grid, 128, 0, s>>>(p, static_cast<const float *>(out),
                                                   static_cast<const float *>(dout), lse, delta,
                                                   nlse2);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !p.sinks) return e;
    dsink_part_kernel<<<dim3(p.nq, p.Hq, p.B), 32, 0, s>>>(p, lse, delta, dsink_part);
    dsink_reduce_kernel<<<p.Hq, 256, 0, s>>>(dsink_part, p.B * p.nq, dsinks);
    return cudaGetLastError();
}

} // namespace ra
