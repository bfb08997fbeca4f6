// k_mask.cu -- block map on the 128 x 128 tile grid: the counterpart of the
// pages' MaskInfo ("ejKernel ring_attention._ring_splash" module source,
// make_ring_attention: forward and dkv mask infos) and of Kvax
// create_attention_mask (block-wise mask from positions and segment ids,
// padding-only blocks skipped).  Integer work, bit-exact:
//   class(qt, kt) = EMPTY if no pair is visible, FULL if all are, else PARTIAL
// with visible(i, j) = same non-padding segment && (!causal || q_pos >= kv_pos).
//
// 1. tile_summary: per 128-row tile, min / max segment id and position over
//    the non-padding rows and the padding count.
// 2. classify_rows: one block per (b, qt).  Tiles whose class follows
//    exactly from the summaries (disjoint segment ranges; one common segment,
//    where the causal predicate reduces to comparing position ranges) are
//    classified from them, the rest pair by pair.  With the non-causal ring's
//    local mask, each 128 x 128 block of the mask is classified once first;
//    a tile is then empty if either class is, takes the mask's class where
//    every pair passes the other rules, and is counted pair by pair only
//    where both are partial.  The block then
//    compacts the non-empty kt of its row into fwd_idx and records where the
//    tiles of each KV shard begin in that list (fwd_shard).
//    It also counts the row's PARTIAL tiles per KV shard.
// 3. columns: one block per (b, kt) compacts the non-empty qt into bwd_idx
//    and counts the column's PARTIAL tiles.
// 4. order: stable counting sort of rows (columns) by descending count.
// 5. part_scan: exclusive prefix sums of the partial counts give every
//    PARTIAL tile a number in row order and one in column order.
// 6. part_rows / part_cols: the partial mask blocks (the pages' MaskInfo
//    partial_mask_blocks): the 128 x 128 visibility bits of each numbered
//    tile below the capacity, row-major by row-order number and transposed by
//    column-order number.
#include "ra_internal.h"

namespace ra {
namespace {

struct TileSum {
    int seg_min, seg_max, pos_min, pos_max, npad;
};

__device__ __forceinline__ int seg_at(const int32_t *seg, int b, int L, int i)
{
    return seg ? seg[(size_t)b * L + i] : 0;
}
__device__ __forceinline__ int pos_at(const int32_t *pos, int b, int L, int i)
{
    return pos ? pos[(size_t)b * L + i] : i;
}

// grid (ntiles, B), 128 threads: thread i looks at row tile*128 + i.
__global__ void __launch_bounds__(128) tile_summary_kernel(const int32_t *seg, const int32_t *pos,
                                                           int L, int pad_id, TileSum *out)
{
    const int b = blockIdx.y, t = blockIdx.x, i = t * kTile + threadIdx.x;
    const int s = seg_at(seg, b, L, i);
    const int p = pos_at(pos, b, L, i);
    const bool pad = seg && (s == pad_id);
    int smin = pad ? INT_MAX : s, smax = pad ? INT_MIN : s;
    int pmin = pad ? INT_MAX : p, pmax = pad ? INT_MIN : p;
    int npad = pad ? 1 : 0;
    for (int o = 16; o > 0; o >>= 1) {
        smin = min(smin, __shfl_xor_sync(0xffffffffu, smin, o));
        smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
        pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
        npad += __shfl_xor_sync(0xffffffffu, npad, o);
    }
    __shared__ TileSum w[4];
    if ((threadIdx.x & 31) == 0) w[threadIdx.x >> 5] = TileSum{smin, smax, pmin, pmax, npad};
    __syncthreads();
    if (threadIdx.x == 0) {
        TileSum r = w[0];
        for (int k = 1; k < 4; ++k) {
            r.seg_min = min(r.seg_min, w[k].seg_min);
            r.seg_max = max(r.seg_max, w[k].seg_max);
            r.pos_min = min(r.pos_min, w[k].pos_min);
            r.pos_max = max(r.pos_max, w[k].pos_max);
            r.npad += w[k].npad;
        }
        out[(size_t)b * gridDim.x + t] = r;
    }
}

// Class from the summaries when it is exact, else -1 (count pairs).
__device__ __forceinline__ int classify_fast(const TileSum &q, const TileSum &k, int causal)
{
    if (q.npad == kTile || k.npad == kTile) return RA_TILE_EMPTY;
    if (q.seg_max < k.seg_min || k.seg_max < q.seg_min) return RA_TILE_EMPTY;
    const bool one = q.seg_min == q.seg_max && k.seg_min == k.seg_max && q.seg_min == k.seg_min;
    if (!one) return -1;
    const bool nopad = (q.npad == 0 && k.npad == 0);
    if (!causal) return nopad ? RA_TILE_FULL : RA_TILE_PARTIAL;
    if (q.pos_max < k.pos_min) return RA_TILE_EMPTY;
    if (q.pos_min >= k.pos_max) return nopad ? RA_TILE_FULL : RA_TILE_PARTIAL;
    return RA_TILE_PARTIAL;
}

constexpr int kCls = 256; // threads of classify / column kernels

// grid (tq, tk): class of one 128 x 128 block of the non-causal ring's local
// mask (lq_s x lk_s bytes, nonzero = visible); the mask repeats over every
// shard pair, so tile (qt, kt) sees local block (qt mod tq, kt mod tk).
__global__ void __launch_bounds__(kCls) local_tile_kernel(const uint8_t *__restrict__ m, int lk_s,
                                                          int tk, uint8_t *__restrict__ lcls)
{
    const int lt = blockIdx.x, kt = blockIdx.y;
    int cnt = 0;
    // 128 rows of 128 bytes = 8 uint4 per row
    for (int e = threadIdx.x; e < kTile * 8; e += kCls) {
        const int i = e >> 3, c16 = e & 7;
        const uint4 v = *reinterpret_cast<const uint4 *>(
            m + (size_t)(lt * kTile + i) * lk_s + (size_t)kt * kTile + c16 * 16);
        // __vcmpne4 gives 0xff in every nonzero byte
        cnt += (__popc(__vcmpne4(v.x, 0u)) + __popc(__vcmpne4(v.y, 0u)) +
                __popc(__vcmpne4(v.z, 0u)) + __popc(__vcmpne4(v.w, 0u))) >> 3;
    }
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    __shared__ int red[kCls / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
        int t = 0;
        for (int w = 0; w < kCls / 32; ++w) t += red[w];
        lcls[(size_t)lt * tk + kt] =
            (uint8_t)(t == 0 ? RA_TILE_EMPTY : (t == kTile * kTile ? RA_TILE_FULL : RA_TILE_PARTIAL));
    }
}

// grid (nq, B)
__global__ void __launch_bounds__(kCls) classify_rows_kernel(Problem p, const TileSum *qsum,
                                                             const TileSum *ksum,
                                                             const uint8_t *lcls, uint8_t *cls,
                                                             int32_t *fwd_cnt, int32_t *fwd_idx,
                                                             int32_t *fwd_shard, int32_t *part_fwd)
{
    const int b = blockIdx.y, qt = blockIdx.x, nk = p.nk;
    // partial tiles per KV shard, counted into entries 1..N
    int32_t *prow = part_fwd + ((size_t)b * p.nq + qt) * (p.N + 1);
    for (int sh = threadIdx.x; sh <= p.N; sh += kCls) prow[sh] = 0;
    __shared__ int q_seg_s[kTile], q_pos_s[kTile], k_seg_s[kTile], k_pos_s[kTile];
    __shared__ int slow[1024];
    __shared__ int nslow, red[kCls / 32], base;
    const TileSum qs = qsum[(size_t)b * p.nq + qt];
    uint8_t *crow = cls + ((size_t)b * p.nq + qt) * nk;
    int32_t *irow = fwd_idx + ((size_t)b * p.nq + qt) * nk;
    if (threadIdx.x < kTile) {
        const int i = qt * kTile + threadIdx.x;
        q_seg_s[threadIdx.x] = seg_at(p.q_seg, b, p.Lq, i);
        q_pos_s[threadIdx.x] = pos_at(p.q_pos, b, p.Lq, i);
    }
    if (threadIdx.x == 0) base = 0;
    for (int k0 = 0; k0 < nk; k0 += 1024) {
        const int kend = min(nk, k0 + 1024);
        if (threadIdx.x == 0) nslow = 0;
        __syncthreads();
        for (int kt = k0 + threadIdx.x; kt < kend; kt += kCls) {
            int c = classify_fast(qs, ksum[(size_t)b * nk + kt], p.causal);
            if (p.local_mask && c != RA_TILE_EMPTY) {
                // the local mask can only remove pairs
                const int lc = lcls[(size_t)(qt % p.tq) * p.tk + (kt % p.tk)];
                if (lc == RA_TILE_EMPTY) c = RA_TILE_EMPTY;
                else if (c == RA_TILE_FULL) c = lc; // every pair passes the other rules
                else if (lc != RA_TILE_FULL) c = -1; // both partial (or unknown): count pairs
            }
            if (c < 0) {
                slow[atomicAdd(&nslow, 1)] = kt;
            } else {
                crow[kt] = (uint8_t)c;
            }
        }
        __syncthreads();
        const int ns = nslow;
        for (int si = 0; si < ns; ++si) {
            const int kt = slow[si];
            if (threadIdx.x < kTile) {
                const int j = kt * kTile + threadIdx.x;
                k_seg_s[threadIdx.x] = seg_at(p.kv_seg, b, p.Lkv, j);
                k_pos_s[threadIdx.x] = pos_at(p.kv_pos, b, p.Lkv, j);
            }
            __syncthreads();
            int cnt = 0;
            for (int e = threadIdx.x; e < kTile * kTile; e += kCls) {
                const int i = e >> 7, j = e & (kTile - 1);
                const int sq = q_seg_s[i];
                bool vis = (sq == k_seg_s[j]) && !(p.q_seg && sq == p.pad_id);
                if (p.causal) vis = vis && (q_pos_s[i] >= k_pos_s[j]);
                if (p.local_mask)
                    vis = vis && p.local_mask[(size_t)((qt * kTile + i) % p.lq_s) * p.lk_s +
                                              (kt * kTile + j) % p.lk_s] != 0;
                cnt += vis ? 1 : 0;
            }
            for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
            if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
            __syncthreads();
            if (threadIdx.x == 0) {
                int t = 0;
                for (int w = 0; w < kCls / 32; ++w) t += red[w];
                crow[kt] = (uint8_t)(t == 0 ? RA_TILE_EMPTY
                                            : (t == kTile * kTile ? RA_TILE_FULL : RA_TILE_PARTIAL));
            }
            __syncthreads();
        }
        __syncthreads();
        // compact non-empty kt of this chunk, in ascending order
        for (int kk = k0; kk < kend; kk += kCls) {
            const int kt = kk + threadIdx.x;
            const bool ne = kt < kend && crow[kt] != RA_TILE_EMPTY;
            const unsigned m = __ballot_sync(0xffffffffu, ne);
            const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
            if (lane == 0) red[wid] = __popc(m);
            __syncthreads();
            int off = base;
            for (int w = 0; w < wid; ++w) off += red[w];
            if (ne) {
                irow[off + __popc(m & ((1u << lane) - 1u))] = kt;
                if (crow[kt] == RA_TILE_PARTIAL) atomicAdd(&prow[1 + kt / p.tk], 1);
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                int t = 0;
                for (int w = 0; w < kCls / 32; ++w) t += red[w];
                base += t;
            }
            __syncthreads();
        }
    }
    __syncthreads();
    const int cnt = base;
    for (int r = cnt + threadIdx.x; r < nk; r += kCls) irow[r] = -1;
    if (threadIdx.x == 0) fwd_cnt[(size_t)b * p.nq + qt] = cnt;
    // shard s of the ring covers kt in [s*tk, (s+1)*tk): its first list
    // position is the number of listed tiles below s*tk (the compacted row
    // is visible to the whole block after the barrier above)
    int32_t *srow = fwd_shard + ((size_t)b * p.nq + qt) * (p.N + 1);
    for (int sh = threadIdx.x; sh <= p.N; sh += kCls) {
        const int key = sh * p.tk;
        int lo = 0, hi = cnt;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (irow[mid] < key) lo = mid + 1;
            else hi = mid;
        }
        srow[sh] = lo;
    }
    // prow[s] = partial tiles of the row before shard s (row-local; the
    // global row offset is added by part_scan)
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int s0 = 1; s0 <= p.N; s0 += 32) {
            const int sh = s0 + lane;
            int v = sh <= p.N ? prow[sh] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            if (sh <= p.N) prow[sh] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
}

// grid (nk, B): column compaction
__global__ void __launch_bounds__(kCls) columns_kernel(const uint8_t *cls, int nq, int nk,
                                                       int32_t *bwd_cnt, int32_t *bwd_idx,
                                                       int32_t *part_bwd)
{
    const int b = blockIdx.y, kt = blockIdx.x;
    __shared__ int red[kCls / 32], base, npart;
    if (threadIdx.x == 0) npart = 0;
    int mine = 0; // partial tiles seen by this thread
    if (threadIdx.x == 0) base = 0;
    __syncthreads();
    int32_t *col = bwd_idx + ((size_t)b * nk + kt) * nq;
    for (int q0 = 0; q0 < nq; q0 += kCls) {
        const int qt = q0 + threadIdx.x;
        const uint8_t c = qt < nq ? cls[((size_t)b * nq + qt) * nk + kt] : (uint8_t)RA_TILE_EMPTY;
        const bool ne = c != RA_TILE_EMPTY;
        mine += c == RA_TILE_PARTIAL ? 1 : 0;
        const unsigned m = __ballot_sync(0xffffffffu, ne);
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
        if (lane == 0) red[wid] = __popc(m);
        __syncthreads();
        int off = base;
        for (int w = 0; w < wid; ++w) off += red[w];
        if (ne) col[off + __popc(m & ((1u << lane) - 1u))] = qt;
        __syncthreads();
        if (threadIdx.x == 0) {
            int t = 0;
            for (int w = 0; w < kCls / 32; ++w) t += red[w];
            base += t;
        }
        __syncthreads();
    }
    const int cnt = base;
    for (int r = cnt + threadIdx.x; r < nq; r += kCls) col[r] = -1;
    if (threadIdx.x == 0) bwd_cnt[(size_t)b * nk + kt] = cnt;
    if (mine) atomicAdd(&npart, mine);
    __syncthreads();
    // column-local count; part_scan turns it into the column's first number
    if (threadIdx.x == 0) part_bwd[(size_t)b * nk + kt] = npart;
}

// Block 0: exclusive prefix over rows of their partial counts, added to
// every per-shard entry of the row (entry N held the row's own total), and
// the grand total into n_part.  Block 1: exclusive prefix over columns.
__global__ void __launch_bounds__(1024) part_scan_kernel(int32_t *part_fwd, int rows, int n1,
                                                         int32_t *part_bwd, int cols,
                                                         int32_t *n_part)
{
    __shared__ int part[1024];
    const bool by_rows = blockIdx.x == 0;
    const int R = by_rows ? rows : cols;
    const int per = (R + 1023) / 1024;
    const int lo = min(R, (int)threadIdx.x * per), hi = min(R, lo + per);
    int sum = 0;
    for (int r = lo; r < hi; ++r)
        sum += by_rows ? part_fwd[(size_t)r * n1 + n1 - 1] : part_bwd[r];
    part[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int t = 0; t < 1024; ++t) {
            const int v = part[t];
            part[t] = run;
            run += v;
        }
        if (by_rows) *n_part = run;
    }
    __syncthreads();
    int run = part[threadIdx.x];
    for (int r = lo; r < hi; ++r) {
        if (by_rows) {
            int32_t *e = part_fwd + (size_t)r * n1;
            const int total = e[n1 - 1];
            for (int k = 0; k < n1; ++k) e[k] += run;
            run += total;
        } else {
            const int v = part_bwd[r];
            part_bwd[r] = run;
            run += v;
        }
    }
}

// Gathers, in list order, the PARTIAL tiles among entries e0 .. e0+127 of a
// tile list into `plist`; returns how many (block-uniform).  128 threads.
__device__ __forceinline__ int gather_partial(const int32_t *list, int cnt, int e0,
                                              const uint8_t *cls, size_t cls_base, size_t cls_stride,
                                              int *plist, int *wcnt)
{
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int e = e0 + t;
    const int id = e < cnt ? list[e] : -1;
    const bool pt = id >= 0 && cls[cls_base + (size_t)id * cls_stride] == RA_TILE_PARTIAL;
    const unsigned m = __ballot_sync(0xffffffffu, pt);
    if (lane == 0) wcnt[wid] = __popc(m);
    __syncthreads();
    int off = 0;
    for (int w = 0; w < wid; ++w) off += wcnt[w];
    if (pt) plist[off + __popc(m & ((1u << lane) - 1u))] = id;
    const int n = wcnt[0] + wcnt[1] + wcnt[2] + wcnt[3];
    __syncthreads();
    return n;
}

// grid (nq, B), 128 threads: thread i writes row i of the row-major block of
// each PARTIAL tile of query-tile row (b, qt) numbered below the capacity.
__global__ void __launch_bounds__(128) part_rows_kernel(Problem p, const uint8_t *cls,
                                                        const int32_t *fwd_cnt,
                                                        const int32_t *fwd_idx,
                                                        const int32_t *part_fwd, uint32_t *out)
{
    const int b = blockIdx.y, qt = blockIdx.x, i = threadIdx.x;
    const size_t row = (size_t)b * p.nq + qt;
    int slot = part_fwd[row * (p.N + 1)];
    if (slot >= p.part_cap || part_fwd[row * (p.N + 1) + p.N] == slot) return;
    __shared__ int k_seg_s[kTile], k_pos_s[kTile], plist[kTile], wcnt[4];
    const int qi = qt * kTile + i;
    const int my_seg = seg_at(p.q_seg, b, p.Lq, qi);
    const int my_pos = pos_at(p.q_pos, b, p.Lq, qi);
    const bool my_pad = p.q_seg && my_seg == p.pad_id;
    const int cnt = fwd_cnt[row];
    const int32_t *list = fwd_idx + row * p.nk;
    for (int e0 = 0; e0 < cnt && slot < p.part_cap; e0 += kTile) {
        const int n = gather_partial(list, cnt, e0, cls, row * p.nk, 1, plist, wcnt);
        for (int t = 0; t < n && slot < p.part_cap; ++t, ++slot) {
            const int kt = plist[t];
            k_seg_s[i] = seg_at(p.kv_seg, b, p.Lkv, kt * kTile + i);
            k_pos_s[i] = pos_at(p.kv_pos, b, p.Lkv, kt * kTile + i);
            __syncthreads();
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t bits = 0;
#pragma unroll 8
                for (int z = 0; z < 32; ++z) {
                    const int j = 32 * k + z;
                    bool v = k_seg_s[j] == my_seg && !my_pad;
                    if (p.causal) v = v && my_pos >= k_pos_s[j];
                    bits |= (v ? 1u : 0u) << z;
                }
                w[k] = bits;
            }
            if (p.local_mask) {
                const uint8_t *lm = p.local_mask + (size_t)(qi % p.lq_s) * p.lk_s + (kt * kTile) % p.lk_s;
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll 8
                    for (int z = 0; z < 32; ++z)
                        if (!lm[32 * k + z]) w[k] &= ~(1u << z);
            }
            reinterpret_cast<uint4 *>(out)[(size_t)slot * kTile + i] = make_uint4(w[0], w[1], w[2], w[3]);
            __syncthreads();
        }
    }
}

// grid (nk, B), 128 threads: thread j writes row j (kv row) of the
// transposed block of each PARTIAL tile of key-tile column (b, kt) numbered
// below the capacity.
__global__ void __launch_bounds__(128) part_cols_kernel(Problem p, const uint8_t *cls,
                                                        const int32_t *bwd_cnt,
                                                        const int32_t *bwd_idx,
                                                        const int32_t *part_bwd, uint32_t *out)
{
    const int b = blockIdx.y, kt = blockIdx.x, j = threadIdx.x;
    const size_t col = (size_t)b * p.nk + kt;
    int slot = part_bwd[col];
    if (slot >= p.part_cap) return;
    __shared__ int q_seg_s[kTile], q_pos_s[kTile], plist[kTile], wcnt[4];
    const int kj = kt * kTile + j;
    const int my_seg = seg_at(p.kv_seg, b, p.Lkv, kj);
    const int my_pos = pos_at(p.kv_pos, b, p.Lkv, kj);
    const int cnt = bwd_cnt[col];
    const int32_t *list = bwd_idx + col * p.nq;
    for (int e0 = 0; e0 < cnt && slot < p.part_cap; e0 += kTile) {
        const int n = gather_partial(list, cnt, e0, cls, (size_t)b * p.nq * p.nk + kt, p.nk, plist,
                                     wcnt);
        for (int t = 0; t < n && slot < p.part_cap; ++t, ++slot) {
            const int qt = plist[t];
            q_seg_s[j] = seg_at(p.q_seg, b, p.Lq, qt * kTile + j);
            q_pos_s[j] = pos_at(p.q_pos, b, p.Lq, qt * kTile + j);
            __syncthreads();
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t bits = 0;
#pragma unroll 8
                for (int z = 0; z < 32; ++z) {
                    const int i = 32 * k + z;
                    const int sq = q_seg_s[i];
                    bool v = sq == my_seg && !(p.q_seg && sq == p.pad_id);
                    if (p.causal) v = v && q_pos_s[i] >= my_pos;
                    bits |= (v ? 1u : 0u) << z;
                }
                w[k] = bits;
            }
            if (p.local_mask) {
                const uint8_t *lm = p.local_mask + (size_t)((qt * kTile) % p.lq_s) * p.lk_s + kj % p.lk_s;
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll 8
                    for (int z = 0; z < 32; ++z)
                        if (!lm[(size_t)(32 * k + z) * p.lk_s]) w[k] &= ~(1u << z);
            }
            reinterpret_cast<uint4 *>(out)[(size_t)slot * kTile + j] = make_uint4(w[0], w[1], w[2], w[3]);
            __syncthreads();
        }
    }
}

// Stable counting sort of ids 0..R-1 by descending cnt[id] (ties by id).
// One block of 1024 threads; hist needs (maxc + 1) ints of dynamic smem.
__global__ void __launch_bounds__(1024) order_kernel(const int32_t *cnt, int R, int maxc,
                                                     int32_t *order)
{
    extern __shared__ int hist[]; // [maxc + 1], then [1024] partials
    int *part = hist + maxc + 1;
    const int nb = maxc + 1;
    for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < R; i += blockDim.x) atomicAdd(&hist[maxc - cnt[i]], 1);
    __syncthreads();
    // exclusive scan of hist (key = maxc - cnt ascending == cnt descending)
    const int per = (nb + blockDim.x - 1) / blockDim.x;
    const int lo = threadIdx.x * per, hi = min(nb, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += hist[i];
    part[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int t = 0; t < (int)blockDim.x; ++t) {
            const int v = part[t];
            part[t] = run;
            run += v;
        }
    }
    __syncthreads();
    int run = part[threadIdx.x];
    for (int i = lo; i < hi; ++i) {
        const int v = hist[i];
        hist[i] = run;
        run += v;
    }
    __syncthreads();
    // stable scatter by warp 0, 32 ids at a time in id order
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        for (int i0 = 0; i0 < R; i0 += 32) {
            const int id = i0 + lane;
            const bool act = id < R;
            const int key = act ? maxc - cnt[id] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const int leader = __ffs(peers) - 1;
            int start = 0;
            if (act && lane == leader) {
                start = hist[key];
                hist[key] = start + __popc(peers);
            }
            start = __shfl_sync(0xffffffffu, start, leader);
            if (act) order[start + __popc(peers & ((1u << lane) - 1u))] = id;
            __syncwarp();
        }
    }
}

} // namespace

size_t mask_scratch_ints(int B, int nq, int nk, int N)
{
    const size_t local_tiles = (size_t)(nq / N) * (nk / N); // one byte each
    return (size_t)B * (nq + nk) * (sizeof(TileSum) / sizeof(int32_t)) + (local_tiles + 3) / 4;
}

int mask_part_cap(int B, int nq, int nk)
{
    return 4 * B * (nq + nk);
}

cudaError_t launch_mask_build(const Problem &pin, const ra_block_mask &m, int32_t *scratch,
                              cudaStream_t s)
{
    Problem p = pin;
    p.part_cap = m.part_cap;
    uint8_t *cls = m.tile_class;
    TileSum *qsum = reinterpret_cast<TileSum *>(scratch);
    TileSum *ksum = qsum + (size_t)p.B * p.nq;
    uint8_t *lcls = reinterpret_cast<uint8_t *>(ksum + (size_t)p.B * p.nk);
    tile_summary_kernel<<<dim3(p.nq, p.B), 128, 0, s>>>(p.q_seg, p.q_pos, p.Lq, p.pad_id, qsum);
    tile_summary_kernel<<<dim3(p.nk, p.B), 128, 0, s>>>(p.kv_seg, p.kv_pos, p.Lkv, p.pad_id, ksum);
    if (p.local_mask)
        local_tile_kernel<<<dim3(p.tq, p.tk), kCls, 0, s>>>(p.local_mask, p.lk_s, p.tk, lcls);
    classify_rows_kernel<<<dim3(p.nq, p.B), kCls, 0, s>>>(p, qsum, ksum, lcls, cls, m.fwd_cnt,
                                                          m.fwd_idx, m.fwd_shard, m.part_fwd);
    columns_kernel<<<dim3(p.nk, p.B), kCls, 0, s>>>(cls, p.nq, p.nk, m.bwd_cnt, m.bwd_idx,
                                                    m.part_bwd);
    const size_t sm_f = sizeof(int) * ((size_t)p.nk + 1 + 1024);
    const size_t sm_b = sizeof(int) * ((size_t)p.nq + 1 + 1024);
    order_kernel<<<1, 1024, sm_f, s>>>(m.fwd_cnt, p.B * p.nq, p.nk, m.fwd_order);
    order_kernel<<<1, 1024, sm_b, s>>>(m.bwd_cnt, p.B * p.nk, p.nq, m.bwd_order);
    part_scan_kernel<<<2, 1024, 0, s>>>(m.part_fwd, p.B * p.nq, p.N + 1, m.part_bwd, p.B * p.nk,
                                        m.n_part);
    part_rows_kernel<<<dim3(p.nq, p.B), kTile, 0, s>>>(p, cls, m.fwd_cnt, m.fwd_idx, m.part_fwd,
                                                       m.part_rows);
    part_cols_kernel<<<dim3(p.nk, p.B), kTile, 0, s>>>(p, cls, m.bwd_cnt, m.bwd_idx, m.part_bwd,
                                                       m.part_cols);
    return cudaGetLastError();
}

} // namespace ra
