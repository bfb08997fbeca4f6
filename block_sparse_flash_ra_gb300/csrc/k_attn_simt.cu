// k_attn_simt.cu -- fp32 forward on the CUDA cores, for RA_FP32 inputs.
//
// Same schedule as the tensor-core forward ("ejKernel ring_attention.
// _ring_splash" module source, _ring_attention_forward): per query tile the
// virtual shards are visited in ring order s = (d - t) mod N, empty tiles are
// skipped from the block map, the sink enters on step 0 only, and each
// shard's normalised partial is merged into the running (out, lse) by
// _update_out_and_lse.  fp32 inputs stay fp32 here because tf32 rounding of
// q and k (2^-11) moves lse by up to ~1e-3, the bound the results are held to.
//
// grid (nq, Hq, B), 128 threads; thread t owns query row qt*128 + t.  K and V
// tiles are staged in shared memory (fp32), the running output in shared
// memory transposed ([D][128]) so that thread t's column accesses are
// conflict-free; q and the shard accumulator live in registers.
#include <math.h>

#include "ra_device.cuh"

namespace ra {
namespace {

template <int D>
__global__ void __launch_bounds__(128) fwd_simt_kernel(Problem p, const float *__restrict__ q,
                                                       const float *__restrict__ k,
                                                       const float *__restrict__ v,
                                                       float *__restrict__ out,
                                                       float *__restrict__ lse)
{
    extern __shared__ float sm[];
    float *Ks = sm;                 // [128][D]
    float *Vs = Ks + kTile * D;     // [128][D]
    float *Orun = Vs + kTile * D;   // [D][128]
    int *kpos = reinterpret_cast<int *>(Orun + D * kTile);
    int *kseg = kpos + kTile;

    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int i = qt * kTile + t;
    const int g = h / p.G;
    const int row_id = b * p.nq + qt;
    const int cnt = p.fwd_cnt[row_id];
    const int32_t *list = p.fwd_idx + (size_t)row_id * p.nk;
    const int dev = qt / p.tq;

    float qr[D];
    {
        const float *src = q + (((size_t)b * p.Lq + i) * p.Hq + h) * D;
        for (int d = 0; d < D; ++d) qr[d] = src[d];
    }
    const int my_pos = p.q_pos ? p.q_pos[(size_t)b * p.Lq + i] : i;
    const int my_seg = p.q_seg ? p.q_seg[(size_t)b * p.Lq + i] : 0;
    const bool my_pad = p.q_seg && my_seg == p.pad_id;
    const float scale2 = p.scale * kLog2e;
    const float cap = p.soft_cap;

    float lse_run = -INFINITY;
    bool orun_set = false; // O_run holds real data (else logically zero)
    for (int d = 0; d < D; ++d) Orun[d * kTile + t] = 0.f;

    for (int step = 0; step < p.N; ++step) {
        const int src = (dev - step + p.N) % p.N;
        const int lo_kt = src * p.tk, hi_kt = lo_kt + p.tk;
        float m = -INFINITY, l = 0.f;
        float o[D];
        for (int d = 0; d < D; ++d) o[d] = 0.f;
        bool any_tile = false;
        for (int e = 0; e < cnt; ++e) {
            const int kt = list[e];
            if (kt < lo_kt || kt >= hi_kt) continue;
            any_tile = true;
            const bool partial = p.tile_class[(size_t)row_id * p.nk + kt] == RA_TILE_PARTIAL;
            __syncthreads();
            for (int x = t; x < kTile * D; x += 128) {
                const int r = x / D, d = x % D;
                const size_t gi = (((size_t)b * p.Lkv + kt * kTile + r) * p.Hkv + g) * D + d;
                Ks[x] = k[gi];
                Vs[x] = v[gi];
            }
            {
                const int j = kt * kTile + t;
                kpos[t] = p.kv_pos ? p.kv_pos[(size_t)b * p.Lkv + j] : j;
                kseg[t] = p.kv_seg ? p.kv_seg[(size_t)b * p.Lkv + j] : 0;
            }
            __syncthreads();
            for (int j = 0; j < kTile; ++j) {
                if (partial) {
                    bool vis = (kseg[j] == my_seg) && !my_pad;
                    if (p.causal) vis = vis && (my_pos >= kpos[j]);
                    if (p.local_mask)
                        vis = vis && p.local_mask[(size_t)(i % p.lq_s) * p.lk_s +
                                                  (kt * kTile + j) % p.lk_s] != 0;
                    if (!vis) continue;
                }
                float acc = 0.f;
                for (int d = 0; d < D; ++d) acc = fmaf(qr[d], Ks[j * D + d], acc);
                float x2;
                if (cap > 0.f)
                    x2 = cap * kLog2e * tanhf(acc * p.scale / cap);
                else
                    x2 = acc * scale2;
                if (x2 > m) {
                    const float f = exp2f(m - x2);
                    l *= f;
                    for (int d = 0; d < D; ++d) o[d] *= f;
                    m = x2;
                }
                const float pj = exp2f(x2 - m);
                l += pj;
                for (int d = 0; d < D; ++d) o[d] = fmaf(pj, Vs[j * D + d], o[d]);
            }
        }
        const bool sink_here = (step == 0) && p.sinks;
        if (!any_tile && !sink_here) continue; // partial (0, -inf): merge is a no-op
        if (sink_here) {
            const float s2 = p.sinks[h] * kLog2e;
            if (s2 > m) {
                const float f = exp2f(m - s2);
                l *= f;
                for (int d = 0; d < D; ++d) o[d] *= f;
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
        // _update_out_and_lse
        if (lse_run == -INFINITY) {
            for (int d = 0; d < D; ++d) Orun[d * kTile + t] = o[d] * inv;
            lse_run = lse_s;
        } else {
            const float x = lse_s - lse_run;
            const float w = x >= 0.f ? 1.f / (1.f + expf(-x)) : expf(x) / (1.f + expf(x));
            for (int d = 0; d < D; ++d) {
                const float cur = orun_set ? Orun[d * kTile + t] : 0.f;
                Orun[d * kTile + t] = cur - w * (cur - o[d] * inv);
            }
            lse_run = lse_run + (fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
        }
        orun_set = true;
    }
    float *dst = out + (((size_t)b * p.Lq + i) * p.Hq + h) * D;
    for (int d = 0; d < D; ++d) dst[d] = Orun[d * kTile + t];
    lse[((size_t)b * p.Hq + h) * p.Lq + i] = lse_run;
}

template <int D>
int simt_smem()
{
    return (3 * kTile * D) * 4 + 2 * kTile * 4;
}

} // namespace

cudaError_t simt_set_attributes(int D)
{
    if (D == 64)
        return cudaFuncSetAttribute(fwd_simt_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    simt_smem<64>());
    return cudaFuncSetAttribute(fwd_simt_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                simt_smem<128>());
}

cudaError_t launch_fwd_simt_f32(const Problem &p, const float *q, const float *k, const float *v,
                                float *out, float *lse, cudaStream_t s)
{
    const dim3 grid(p.nq, p.Hq, p.B);
    if (p.D == 64)
        fwd_simt_kernel<64><<<grid, 128, simt_smem<64>(), s>>>(p, q, k, v, out, lse);
    else
        fwd_simt_kernel<128><<<grid, 128, simt_smem<128>(), s>>>(p, q, k, v, out, lse);
    return cudaGetLastError();
}

} // namespace ra
