// ra_sched.cuh -- work-unit scheduling helpers shared by the persistent
// tensor-core kernels: snake round-robin over a longest-first unit order,
// bounded drain waits and the scalar merge math.
#pragma once

#include "ra_device.cuh"

namespace ra {

// Snake order over rounds of G units: round r gives CTA c the unit r*G + c
// (even r) or r*G + G-1-c (odd r).
__device__ __forceinline__ int unit_index(int round, int cta, int G)
{
    return round * G + ((round & 1) ? (G - 1 - cta) : cta);
}

// The non-causal ring's per-shard mask (Problem::local_mask) on partial
// tiles.  Row form: bit c of bits[c / 32] is set iff query row qi may see kv
// column j0 + c, i.e. local_mask[qi mod lq_s][(j0 + c) mod lk_s] != 0; j0 is a
// multiple of 64 and shards are whole tiles, so the 64 bytes are contiguous
// and 16-byte aligned.
__device__ __forceinline__ void local_row_bits(const Problem &p, int qi, int j0, uint32_t bits[2])
{
    const uint4 *m4 = reinterpret_cast<const uint4 *>(
        p.local_mask + (size_t)(qi % p.lq_s) * p.lk_s + (j0 % p.lk_s));
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        uint32_t b = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 v = __ldg(m4 + 2 * w + h);
            const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    b |= (((words[k] >> (8 * z)) & 0xffu) ? 1u : 0u) << (16 * h + 4 * k + z);
        }
        bits[w] = b;
    }
}

// Column form: bit c set iff query row q0 + c may see kv row kj (q0 a
// multiple of 64).
__device__ __forceinline__ void local_col_bits(const Problem &p, int q0, int kj, uint32_t bits[2])
{
    const uint8_t *m = p.local_mask + (size_t)(q0 % p.lq_s) * p.lk_s + (kj % p.lk_s);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        uint32_t b = 0;
#pragma unroll 8
        for (int c = 0; c < 32; ++c)
            b |= (__ldg(m + (size_t)(32 * w + c) * p.lk_s) ? 1u : 0u) << c;
        bits[w] = b;
    }
}

// Visibility bits of one 64-column half of a PARTIAL tile, in the two forms
// the kernels need.  A tile numbered below Problem::part_cap reads the block
// the block map stored (one 8-byte load); a tile past it re-derives the bits
// from positions, segments and the local mask.  The row form's derivation is
// a call kept out of line, so that the rarely taken path stays out of the
// forward's hot loop (measured faster there); the dK/dV kernel measured
// slightly faster with the column form inlined.
//
// Row form: bit c of word c / 32 is set iff query row qi sees kv row k0 + c
// (k0 = kt * 128 + 64 * half).
static __device__ __noinline__ uint2 row_bits_derived(const Problem p, int b, int k0, int qi, int q_seg,
                                               int q_pad, int q_pos)
{
    const int32_t *kp = p.kv_pos ? p.kv_pos + (size_t)b * p.Lkv + k0 : nullptr;
    const int32_t *ks = p.kv_seg ? p.kv_seg + (size_t)b * p.Lkv + k0 : nullptr;
    uint32_t bits[2] = {0u, 0u};
    for (int c = 0; c < 64; ++c) {
        const int pos = kp ? __ldg(kp + c) : k0 + c;
        const int seg = ks ? __ldg(ks + c) : 0;
        bool v = seg == q_seg && !q_pad;
        if (p.causal) v = v && q_pos >= pos;
        if (v) bits[c >> 5] |= 1u << (c & 31);
    }
    if (p.local_mask) {
        uint32_t lb[2];
        local_row_bits(p, qi, k0, lb);
        bits[0] &= lb[0];
        bits[1] &= lb[1];
    }
    return make_uint2(bits[0], bits[1]);
}

__device__ __forceinline__ uint2 row_bits(const Problem &p, int slot, int row, int half, int b,
                                          int k0, int qi, int q_seg, bool q_pad, int q_pos)
{
    if (slot < p.part_cap)
        return __ldg(reinterpret_cast<const uint2 *>(p.part_rows + ((size_t)slot * kTile + row) * 4) +
                     half);
    return row_bits_derived(p, b, k0, qi, q_seg, q_pad ? 1 : 0, q_pos);
}

// Column form: bit c of word c / 32 is set iff query row q0 + c sees kv row
// kj (q0 = qt * 128 + 64 * half).
__device__ __forceinline__ uint2 col_bits_derived(const Problem &p, int b, int q0, int kj, int kv_seg,
                                                  int kv_pos)
{
    const int32_t *qp = p.q_pos ? p.q_pos + (size_t)b * p.Lq + q0 : nullptr;
    const int32_t *qs = p.q_seg ? p.q_seg + (size_t)b * p.Lq + q0 : nullptr;
    uint32_t bits[2] = {0u, 0u};
    for (int c = 0; c < 64; ++c) {
        const int pos = qp ? __ldg(qp + c) : q0 + c;
        const int seg = qs ? __ldg(qs + c) : 0;
        bool v = seg == kv_seg && !(qs && seg == p.pad_id);
        if (p.causal) v = v && pos >= kv_pos;
        if (v) bits[c >> 5] |= 1u << (c & 31);
    }
    if (p.local_mask) {
        uint32_t lb[2];
        local_col_bits(p, q0, kj, lb);
        bits[0] &= lb[0];
        bits[1] &= lb[1];
    }
    return make_uint2(bits[0], bits[1]);
}

__device__ __forceinline__ uint2 col_bits(const Problem &p, int slot, int row, int half, int b,
                                          int q0, int kj, int kv_seg, int kv_pos)
{
    if (slot < p.part_cap)
        return __ldg(reinterpret_cast<const uint2 *>(p.part_cols + ((size_t)slot * kTile + row) * 4) +
                     half);
    return col_bits_derived(p, b, q0, kj, kv_seg, kv_pos);
}

// Wait used only while tearing down after an abort: bounded, ignores the
// abort flag.
__device__ __forceinline__ bool wait_drain(uint64_t *bar, uint32_t parity, uint64_t ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > ns) return false;
    }
    return true;
}

// sigmoid and softplus of the ring merge (_update_out_and_lse) from the
// approximate base-2 exponent, logarithm and reciprocal instructions
// (relative errors near 2^-22): sigmoid(x) = 1 / (1 + 2^(-x log2 e)),
// softplus(x) = max(x, 0) + ln 2 * log2(1 + 2^(-|x| log2 e)).  Both give 0
// at x = -inf and no NaN at +-inf.
__device__ __forceinline__ float sigmoid_fast(float x)
{
    return rcp_approx(1.f + ex2_approx(-x * kLog2e));
}

__device__ __forceinline__ float softplus_fast(float x)
{
    return fmaxf(x, 0.f) + kLn2 * lg2_approx(1.f + ex2_approx(-fabsf(x) * kLog2e));
}

constexpr uint64_t kDrainNs = 100000000ull; // 100 ms

} // namespace ra
