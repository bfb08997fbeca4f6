// k_bwd_pre.cu -- backward preprocessing ("ejKernel ring_attention._ring_splash"
// module source, _ring_attention_backward: dO widened to fp32, dsinks
// accumulated and summed over the ring):
//   Delta[b, h, i] = <dO[b, i, h, :], O[b, i, h, :]>           (fp32)
//   dsinks[h]      = - sum_{b, i} exp(sink_h - lse[b, h, i]) * Delta[b, h, i]
// and, for the gradient kernels, nlse2[b, h, i] = -lse * log2(e): the
// exponent offset of P = 2^(s * scale * log2 e + nlse2).  A row with nothing
// visible (lse = -inf) gets 0 instead of +inf; all its entries are masked, so
// its P stays 0 and no inf - inf can arise.
// The dsinks sum is taken in two deterministic passes: per-(b, q-tile)
// partials, then one block per head.  HBM-bound: reads O and dO once.
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

// grid (nq, Hq, B), 128 threads: warp w handles rows w, w+4, ... of the tile.
template <typename T>
__global__ void __launch_bounds__(128) bwd_pre_kernel(Problem p, const T *__restrict__ out,
                                                      const T *__restrict__ dout,
                                                      const float *__restrict__ lse,
                                                      float *__restrict__ delta,
                                                      float *__restrict__ nlse2,
                                                      float *__restrict__ dsink_part)
{
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const float sink = p.sinks ? p.sinks[h] : 0.f;
    float ds = 0.f;
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
            if (p.sinks && l != -INFINITY) ds += __expf(sink - l) * acc;
        }
    }
    if (p.sinks) {
        __shared__ float w[4];
        if (lane == 0) w[wid] = ds;
        __syncthreads();
        if (threadIdx.x == 0)
            dsink_part[(size_t)h * p.B * p.nq + (size_t)b * p.nq + qt] = w[0] + w[1] + w[2] + w[3];
    }
}

// The same for bf16 rows, with 16-byte loads: D/8 lanes share a row (each
// lane 8 elements of O and of dO), so a warp covers 256/D rows at a time and
// keeps kRowsInFlight of those groups' loads in flight.  grid (nq, Hq, B),
// 128 threads.
template <int D>
__global__ void __launch_bounds__(128) bwd_pre_bf16_kernel(Problem p, const __nv_bfloat16 *__restrict__ out,
                                                           const __nv_bfloat16 *__restrict__ dout,
                                                           const float *__restrict__ lse,
                                                           float *__restrict__ delta,
                                                           float *__restrict__ nlse2,
                                                           float *__restrict__ dsink_part)
{
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    constexpr int kRowsPerPass = 4 * kRowsPerWarp; // 4 warps
    constexpr int kRowsInFlight = 4;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int sub = lane / kLanesPerRow, part = lane % kLanesPerRow;
    const float sink = p.sinks ? p.sinks[h] : 0.f;
    float ds = 0.f;
    for (int r0 = wid * kRowsPerWarp + sub; r0 < kTile; r0 += kRowsPerPass * kRowsInFlight) {
        uint4 o[kRowsInFlight], g[kRowsInFlight];
#pragma unroll
        for (int k = 0; k < kRowsInFlight; ++k) {
            const int r = r0 + k * kRowsPerPass;
            if (r < kTile) {
                const size_t row = (((size_t)b * p.Lq + qt * kTile + r) * p.Hq + h) * D;
                o[k] = __ldg(reinterpret_cast<const uint4 *>(out + row) + part);
                g[k] = __ldg(reinterpret_cast<const uint4 *>(dout + row) + part);
            }
        }
#pragma unroll
        for (int k = 0; k < kRowsInFlight; ++k) {
            const int r = r0 + k * kRowsPerPass;
            const uint32_t ow[4] = {o[k].x, o[k].y, o[k].z, o[k].w};
            const uint32_t gw[4] = {g[k].x, g[k].y, g[k].z, g[k].w};
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc = fmaf(__uint_as_float(ow[j] << 16), __uint_as_float(gw[j] << 16), acc);
                acc = fmaf(__uint_as_float(ow[j] & 0xffff0000u), __uint_as_float(gw[j] & 0xffff0000u), acc);
            }
#pragma unroll
            for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (r < kTile && part == 0) {
                const size_t li = ((size_t)b * p.Hq + h) * p.Lq + qt * kTile + r;
                delta[li] = acc;
                const float l = lse[li];
                nlse2[li] = (l == -INFINITY) ? 0.f : -l * 1.4426950408889634f;
                if (p.sinks && l != -INFINITY) ds += __expf(sink - l) * acc;
            }
        }
    }
    if (p.sinks) {
        // lanes with part == 0 hold partial sums; the rest hold 0
        for (int off = 16; off > 0; off >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, off);
        __shared__ float w[4];
        if (lane == 0) w[wid] = ds;
        __syncthreads();
        if (threadIdx.x == 0)
            dsink_part[(size_t)h * p.B * p.nq + (size_t)b * p.nq + qt] = w[0] + w[1] + w[2] + w[3];
    }
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
    const dim3 grid(p.nq, p.Hq, p.B);
    const __nv_bfloat16 *ob = static_cast<const __nv_bfloat16 *>(out);
    const __nv_bfloat16 *gb = static_cast<const __nv_bfloat16 *>(dout);
    if (dtype == RA_BF16 && p.D == 128)
        bwd_pre_bf16_kernel<128><<<grid, 128, 0, s>>>(p, ob, gb, lse, delta, nlse2, dsink_part);
    else if (dtype == RA_BF16 && p.D == 64)
        bwd_pre_bf16_kernel<64><<<grid, 128, 0, s>>>(p, ob, gb, lse, delta, nlse2, dsink_part);
    else if (dtype == RA_BF16)
        bwd_pre_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(p, ob, gb, lse, delta, nlse2, dsink_part);
    else
        bwd_pre_kernel<float><<<grid, 128, 0, s>>>(p, static_cast<const float *>(out),
                                                   static_cast<const float *>(dout), lse, delta,
                                                   nlse2, dsink_part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !p.sinks) return e;
    dsink_reduce_kernel<<<p.Hq, 256, 0, s>>>(dsink_part, p.B * p.nq, dsinks);
    return cudaGetLastError();
}

} // namespace ra
