// k_merge.cu -- the pages' running-state update, elementwise over rows
// ("ejKernel ring_attention._ring_splash" module source, _update_out_and_lse):
//   first (lse == -inf): take the block;
//   else w = sigmoid(block_lse - lse), out -= w * (out - block_out),
//        lse += softplus(block_lse - lse).
// One warp per (b, l, h) row; HBM-bound: per row it reads 2*D*4 + 8 bytes and
// writes D*4 + 4 bytes.
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

__global__ void __launch_bounds__(256) merge_kernel(float *__restrict__ out, float *__restrict__ lse,
                                                    const float *__restrict__ bout,
                                                    const float *__restrict__ blse, int B, int L,
                                                    int H, int D)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long rows = (long long)B * L * H;
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        // row r = (b, l, h) of out; lse index (b, h, l)
        const int h = (int)(r % H);
        const long long bl = r / H;
        const int l = (int)(bl % L);
        const int b = (int)(bl / L);
        const long long li = ((long long)b * H + h) * L + l;
        const float lo = lse[li];
        const float lb = blse[li];
        const bool first = (lo == -INFINITY);
        const float w = first ? 1.f : sigmoid_stable(lb - lo);
        float4 *o4 = reinterpret_cast<float4 *>(out + r * D);
        const float4 *b4 = reinterpret_cast<const float4 *>(bout + r * D);
        for (int c = lane; c < D / 4; c += 32) {
            const float4 bo = b4[c];
            float4 o;
            if (first) {
                o = bo;
            } else {
                o = o4[c];
                o.x -= w * (o.x - bo.x);
                o.y -= w * (o.y - bo.y);
                o.z -= w * (o.z - bo.z);
                o.w -= w * (o.w - bo.w);
            }
            o4[c] = o;
        }
        if (lane == 0) lse[li] = first ? lb : lo + softplus_stable(lb - lo);
    }
}

} // namespace

cudaError_t launch_merge(float *out, float *lse, const float *bout, const float *blse, int B,
                         int L, int H, int D, cudaStream_t s)
{
    const long long rows = (long long)B * L * H;
    long long blocks = (rows + 7) / 8;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    if (blocks < 1) blocks = 1;
    merge_kernel<<<(unsigned)blocks, 256, 0, s>>>(out, lse, bout, blse, B, L, H, D);
    return cudaGetLastError();
}

} // namespace ra
