// k_permute.cu -- zigzag token permutation along the sequence axis (Kvax
// "Flash Attention for JAX", context parallelism: permute tokens for load
// balance, unpermute outputs).  Bitwise copy of whole token rows; HBM-bound:
// each launch reads and writes B * L * row_bytes bytes once.
#include "ra_internal.h"

namespace ra {
namespace {

// Original index of permuted row p: 2N chunks of c = L/(2N) rows, virtual
// device d = p / (L/N) holds chunk d then chunk 2N-1-d.
__device__ __forceinline__ int zigzag_source(int p, int per, int c, int n)
{
    const int d = p / per;
    const int r = p - d * per;
    return r < c ? d * c + r : (2 * n - 1 - d) * c + (r - c);
}

template <typename V>
__global__ void __launch_bounds__(256) permute_kernel(const V *__restrict__ in, V *__restrict__ out,
                                                      int B, int L, long long vec_per_row, int n,
                                                      int inverse)
{
    const int per = L / n, c = L / (2 * n);
    const long long total = (long long)B * L * vec_per_row;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long row = e / vec_per_row;
        const long long col = e - row * vec_per_row;
        const int b = (int)(row / L);
        const int p = (int)(row - (long long)b * L);
        const int s = zigzag_source(p, per, c, n);
        const long long dst = inverse ? s : p;
        const long long src = inverse ? p : s;
        out[((long long)b * L + dst) * vec_per_row + col] =
            in[((long long)b * L + src) * vec_per_row + col];
    }
}

// Rows of at least 256 bytes: one warp per row (the source row is computed
// once per row), each lane copying 16-byte chunks with four in flight.
__global__ void __launch_bounds__(256) permute_rows_kernel(const uint4 *__restrict__ in,
                                                           uint4 *__restrict__ out, int B, int L,
                                                           int vec_per_row, int n, int inverse)
{
    const int per = L / n, c = L / (2 * n);
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)B * L;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += warps) {
        const int b = (int)(row / L);
        const int p = (int)(row - (long long)b * L);
        const int sidx = zigzag_source(p, per, c, n);
        const long long dst = (long long)b * L + (inverse ? sidx : p);
        const long long src = (long long)b * L + (inverse ? p : sidx);
        const uint4 *ip = in + src * vec_per_row;
        uint4 *op = out + dst * vec_per_row;
        for (int k0 = lane; k0 < vec_per_row; k0 += 4 * 32) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (k0 + 32 * u < vec_per_row) v[u] = __ldg(ip + k0 + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (k0 + 32 * u < vec_per_row) op[k0 + 32 * u] = v[u];
        }
    }
}

template <typename V>
cudaError_t run(const void *in, void *out, int B, int L, size_t row_bytes, int n, int inverse,
                cudaStream_t s)
{
    const long long vpr = (long long)(row_bytes / sizeof(V));
    const long long total = (long long)B * L * vpr;
    long long blocks = (total + 255) / 256;
    if (blocks > 152LL * 32) blocks = 152LL * 32;
    if (blocks < 1) blocks = 1;
    permute_kernel<V><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const V *>(in),
                                                       static_cast<V *>(out), B, L, vpr, n,
                                                       inverse);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_permute(const void *in, void *out, int B, int L, size_t row_bytes, int n,
                           int inverse, cudaStream_t s)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out);
    if (row_bytes % 16 == 0 && a % 16 == 0 && row_bytes >= 256 && row_bytes / 16 <= 0x7fffffff) {
        const long long rows = (long long)B * L;
        long long blocks = (rows + 7) / 8; // 8 warps per block, one row each
        if (blocks > 152LL * 16) blocks = 152LL * 16;
        permute_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4 *>(in),
                                                             static_cast<uint4 *>(out), B, L,
                                                             (int)(row_bytes / 16), n, inverse);
        return cudaGetLastError();
    }
    if (row_bytes % 16 == 0 && a % 16 == 0) return run<uint4>(in, out, B, L, row_bytes, n, inverse, s);
    if (row_bytes % 8 == 0 && a % 8 == 0) return run<uint2>(in, out, B, L, row_bytes, n, inverse, s);
    if (row_bytes % 4 == 0 && a % 4 == 0) return run<uint32_t>(in, out, B, L, row_bytes, n, inverse, s);
    if (row_bytes % 2 == 0 && a % 2 == 0) return run<uint16_t>(in, out, B, L, row_bytes, n, inverse, s);
    return run<uint8_t>(in, out, B, L, row_bytes, n, inverse, s);
}

} // namespace ra
