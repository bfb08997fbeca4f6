// k_ring.cu -- elementwise kernels of the ring's end ("ejKernel
// ring_attention._ring_splash" module source, _ring_attention_backward):
// the casts of the fp32 accumulators dq, dk, dv to the input dtype, and the
// sum of per-device dsinks (its psum over the ring) when several virtual
// devices share one GPU.  HBM-bound: 16-byte loads, grid-stride loops.
#include <cuda_bf16.h>

#include "ra_device.cuh"

namespace ra {
namespace {

// out[i] = bf16(in[i]); n4 float4 groups, then the tail
__global__ void __launch_bounds__(256) cast_bf16_kernel(const float *__restrict__ in,
                                                        __nv_bfloat16 *__restrict__ out, size_t n)
{
    const size_t n4 = n / 4;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 v = reinterpret_cast<const float4 *>(in)[i];
        reinterpret_cast<uint2 *>(out)[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
    if (blockIdx.x == 0 && threadIdx.x < n - n4 * 4) {
        const size_t i = n4 * 4 + threadIdx.x;
        out[i] = __float2bfloat16_rn(in[i]);
    }
}

__global__ void __launch_bounds__(256) copy_f32_kernel(const float *__restrict__ in,
                                                       float *__restrict__ out, size_t n)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) out[i] = in[i];
}

__global__ void __launch_bounds__(256) add_f32_kernel(float *__restrict__ acc,
                                                      const float *__restrict__ x, size_t n)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) acc[i] += x[i];
}

unsigned grid_for(size_t work)
{
    size_t b = (work + 255) / 256;
    if (b > 152 * 32) b = 152 * 32;
    return b < 1 ? 1u : (unsigned)b;
}

} // namespace

cudaError_t launch_cast_from_f32(const float *in, void *out, size_t n, int dtype, cudaStream_t s)
{
    if (dtype == RA_BF16)
        cast_bf16_kernel<<<grid_for(n / 4 + 1), 256, 0, s>>>(in, static_cast<__nv_bfloat16 *>(out), n);
    else
        copy_f32_kernel<<<grid_for(n), 256, 0, s>>>(in, static_cast<float *>(out), n);
    return cudaGetLastError();
}

cudaError_t launch_add_f32(float *acc, const float *x, size_t n, cudaStream_t s)
{
    add_f32_kernel<<<grid_for(n), 256, 0, s>>>(acc, x, n);
    return cudaGetLastError();
}

} // namespace ra
