// k_merge.cu -- the pages' running-state update, elementwise over rows
// ("ejKernel ring_attention._ring_splash" module source, _update_out_and_lse):
//   first (lse == -inf): take the block;
//   else w = sigmoid(block_lse - lse), out -= w * (out - block_out),
//        lse += softplus(block_lse - lse).
// HBM-bound: per (b, l, h) row it reads 2*D*4 + 8 bytes and writes D*4 + 4.
#include "ra_internal.h"

namespace ra {
namespace {

__device__ __forceinline__ float sigmoid_stable(float x)
{
    if (x >= 0.f) return 1.f / (1.f + __expf(-x));
    const float e = __expf(x);
    return e / (1.f + e);
}

__device__ __forceinline__ float softplus_stable(float x)
{
    return fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x)));
}

// One (b, l, h) row: the new (out, lse) from the running pair and the block's.
// `first` (running lse = -inf) takes the block as is, whatever out holds.
__device__ __forceinline__ float4 merge4(float4 o, float4 bo, bool first, float w)
{
    if (first) return bo;
    o.x -= w * (o.x - bo.x);
    o.y -= w * (o.y - bo.y);
    o.z -= w * (o.z - bo.z);
    o.w -= w * (o.w - bo.w);
    return o;
}

// One warp per token (b, l): the token's H rows of out and block_out are one
// contiguous stretch of H * D floats, which the warp streams in float4 with U
// loads of each tensor in flight per lane (all the token's rows are adjacent,
// so the warps of the GPU sweep memory in order).  First pass: the new out
// from the old lse values; second pass, after every lane has read them: lane
// h writes the new lse of head h.  D4 = D / 4 as a compile-time constant for
// the usual head sizes (0: taken from the argument).
template <int D4C, int U>
__global__ void __launch_bounds__(256) merge_tok_kernel(float *__restrict__ out, float *__restrict__ lse,
                                                        const float *__restrict__ bout,
                                                        const float *__restrict__ blse, int B, int L,
                                                        int H, int D4a)
{
    const int D4 = D4C ? D4C : D4a;
    const int lane = threadIdx.x & 31;
    const long long toks = (long long)B * L;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const int n4 = H * D4;
    for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < toks;
         t += warps) {
        const int b = (int)(t / L), l = (int)(t - (long long)b * L);
        float4 *o4 = reinterpret_cast<float4 *>(out) + t * n4;
        const float4 *b4 = reinterpret_cast<const float4 *>(bout) + t * n4;
        const float *lse_b = lse + (size_t)b * H * L + l;   // head h at lse_b[h * L]
        const float *blse_b = blse + (size_t)b * H * L + l;
        for (int f0 = 0; f0 < n4; f0 += 32 * U) {
            float4 o[U], bo[U];
            float lo[U], lb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int f = f0 + u * 32 + lane;
                if (f < n4) {
                    const int h = f / D4;
                    lo[u] = lse_b[(size_t)h * L];
                    lb[u] = blse_b[(size_t)h * L];
                    o[u] = o4[f];
                    bo[u] = b4[f];
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int f = f0 + u * 32 + lane;
                if (f >= n4) continue;
                const bool first = (lo[u] == -INFINITY);
                o4[f] = merge4(o[u], bo[u], first, first ? 1.f : sigmoid_stable(lb[u] - lo[u]));
            }
        }
        __syncwarp(); // every lane has read the old lse values
        float *lse_w = lse + (size_t)b * H * L + l;
        for (int h = lane; h < H; h += 32) {
            const float lo = lse_w[(size_t)h * L], lb = blse_b[(size_t)h * L];
            lse_w[(size_t)h * L] = (lo == -INFINITY) ? lb : lo + softplus_stable(lb - lo);
        }
    }
}

} // namespace

cudaError_t launch_merge(float *out, float *lse, const float *bout, const float *blse, int B,
                         int L, int H, int D, cudaStream_t s)
{
    // one warp per token, 8 tokens per block, up to ~64 blocks per SM of a
    // 152-SM GPU (a grid-stride loop covers the rest)
    const long long toks = (long long)B * L;
    long long blocks = (toks + 7) / 8;
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    if (blocks < 1) blocks = 1;
    const unsigned g = (unsigned)blocks;
    if (D == 128)
        merge_tok_kernel<32, 4><<<g, 256, 0, s>>>(out, lse, bout, blse, B, L, H, 32);
    else if (D == 64)
        merge_tok_kernel<16, 4><<<g, 256, 0, s>>>(out, lse, bout, blse, B, L, H, 16);
    else
        merge_tok_kernel<0, 4><<<g, 256, 0, s>>>(out, lse, bout, blse, B, L, H, D / 4);
    return cudaGetLastError();
}

} // namespace ra
