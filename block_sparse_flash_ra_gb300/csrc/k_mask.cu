// k_mask.cu -- block map on the 128 x 128 tile grid: the counterpart of the
// pages' MaskInfo ("ejKernel ring_attention._ring_splash" module source,
// make_ring_attention: forward and dkv mask infos) and of Kvax
// create_attention_mask (block-wise mask from positions and segment ids,
// padding-only blocks skipped).  Integer work, bit-exact:
//   class(qt, kt) = EMPTY if no pair is visible, FULL if all are, else PARTIAL
// with visible(i, j) = same non-padding segment && (!causal || q_pos >= kv_pos).
//
// 1. tile_summary: per 128-row tile, the padding count, the segment id range
//    and, for up to four distinct segments, each one's position range.
// 2. classify_rows: one block per (b, qt).  Tiles whose class follows
//    exactly from the summaries (every segment of both tiles summarised, or
//    disjoint segment ranges) are classified from them, the rest (tiles with
//    more than four segments) pair by pair.  With the non-causal ring's
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
// 6. part_list / part_bits: the partial mask blocks (the pages' MaskInfo
//    partial_mask_blocks): each row and column lists its numbered tiles, then
//    one block per number writes the 128 x 128 visibility bits of the tile of
//    that row-order number (row-major) and of that column-order number
//    (transposed), for the numbers below the capacity.
#include "ra_sched.cuh"

namespace ra {
namespace {

// Per 128-row tile: the padding count, the range of segment ids, and for up
// to kMaxSeg distinct non-padding segments the id and the position range of
// the tile's tokens in it (nseg = kMaxSeg + 1: more segments than that).
constexpr int kMaxSeg = 4;
struct TileSum {
    int nseg, npad, seg_min, seg_max;
    int seg[kMaxSeg], pmin[kMaxSeg], pmax[kMaxSeg];
};

__device__ __forceinline__ int seg_at(const int32_t *seg, int b, int L, int i)
{
    return seg ? seg[(size_t)b * L + i] : 0;
}
__device__ __forceinline__ int pos_at(const int32_t *pos, int b, int L, int i)
{
    return pos ? pos[(size_t)b * L + i] : i;
}

// One side (query or key rows) of the summaries: blockIdx.x = tile, thread i
// looks at row tile*128 + i.
__device__ __forceinline__ void tile_summary(const int32_t *seg, const int32_t *pos, int L, int pad_id,
                                             TileSum *out)
{
    const int b = blockIdx.y, t = blockIdx.x, i = t * kTile + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int s = seg_at(seg, b, L, i);
    const int p = pos_at(pos, b, L, i);
    const bool pad = seg && (s == pad_id);
    // lanes of one segment (padding is a group of its own)
    const unsigned long long key = pad ? (1ull << 32) : (unsigned long long)(uint32_t)s;
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    int mn = p, mx = p;
    for (int l = 0; l < 32; ++l) {
        const int v = __shfl_sync(0xffffffffu, p, l);
        if ((grp >> l) & 1u) {
            mn = min(mn, v);
            mx = max(mx, v);
        }
    }
    const bool leader = lane == __ffs(grp) - 1;
    __shared__ TileSum ts;
    if (threadIdx.x == 0) {
        ts.nseg = 0;
        ts.npad = 0;
        ts.seg_min = INT_MAX;
        ts.seg_max = INT_MIN;
    }
    __syncthreads();
    if (pad && leader) atomicAdd(&ts.npad, __popc(grp));
    if (!pad && leader) {
        atomicMin(&ts.seg_min, s);
        atomicMax(&ts.seg_max, s);
    }
    // group leaders merge their segment into the table one at a time
    for (int w = 0; w < 4; ++w) {
        if (warp == w) {
            for (int l = 0; l < 32; ++l) {
                if (lane == l && leader && !pad) {
                    const int n = ts.nseg;
                    const int m = min(n, kMaxSeg);
                    int k = 0;
                    while (k < m && ts.seg[k] != s) ++k;
                    if (k < m) {
                        ts.pmin[k] = min(ts.pmin[k], mn);
                        ts.pmax[k] = max(ts.pmax[k], mx);
                    } else if (n < kMaxSeg) {
                        ts.seg[n] = s;
                        ts.pmin[n] = mn;
                        ts.pmax[n] = mx;
                        ts.nseg = n + 1;
                    } else {
                        ts.nseg = kMaxSeg + 1;
                    }
                }
                __syncwarp();
            }
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) out[(size_t)b * gridDim.x + t] = ts;
}

// grid (max(nq, nk), B, 2), 128 threads: z = 0 summarises the query-row
// tiles, z = 1 the key-row tiles (blocks past a side's tile count return).
__global__ void __launch_bounds__(128) tile_summary_kernel(const int32_t *q_seg, const int32_t *q_pos,
                                                           int Lq, const int32_t *kv_seg,
                                                           const int32_t *kv_pos, int Lkv, int pad_id,
                                                           TileSum *qsum, TileSum *ksum)
{
    const bool q_side = blockIdx.z == 0;
    const int L = q_side ? Lq : Lkv;
    if ((int)blockIdx.x >= L / kTile) return;
    if (q_side) tile_summary(q_seg, q_pos, Lq, pad_id, qsum);
    else tile_summary(kv_seg, kv_pos, Lkv, pad_id, ksum);
}

// Class from the summaries when it is exact, else -1 (count pairs).  With
// every segment of both tiles summarised the class is exact: some pair is
// visible iff a common segment has a query position >= a key position
// (always, without causal); all pairs are iff both tiles hold one and the
// same segment, no padding, and (causal) the smallest query position is >=
// the largest key position.
__device__ __forceinline__ int classify_fast(const TileSum &q, const TileSum &k, int causal)
{
    if (q.nseg == 0 || k.nseg == 0) return RA_TILE_EMPTY; // all padding
    if (q.seg_max < k.seg_min || k.seg_max < q.seg_min) return RA_TILE_EMPTY;
    if (q.nseg > kMaxSeg || k.nseg > kMaxSeg) return -1;
    bool vis = false;
#pragma unroll
    for (int a = 0; a < kMaxSeg; ++a)
#pragma unroll
        for (int c = 0; c < kMaxSeg; ++c)
            if (a < q.nseg && c < k.nseg && q.seg[a] == k.seg[c] && (!causal || q.pmax[a] >= k.pmin[c]))
                vis = true;
    if (!vis) return RA_TILE_EMPTY;
    if (q.nseg == 1 && k.nseg == 1 && q.npad == 0 && k.npad == 0 &&
        (!causal || q.pmin[0] >= k.pmax[0]))
        return RA_TILE_FULL;
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
        // Quick pass: thread t tests kv column t mod 128 of a slow tile against
        // query rows t/128 + 16k (k < 8), one pair in eight; a visible and a
        // hidden pair among them make the tile PARTIAL without counting (the
        // usual case: tiles cut by a document boundary).  The next tile's kv
        // entries are fetched one tile ahead.
        const int cj = threadIdx.x & (kTile - 1), r0 = threadIdx.x >> 7;
        int ks_next = 0, kp_next = 0;
        if (ns > 0) {
            ks_next = seg_at(p.kv_seg, b, p.Lkv, slow[0] * kTile + cj);
            kp_next = pos_at(p.kv_pos, b, p.Lkv, slow[0] * kTile + cj);
        }
        for (int si = 0; si < ns; ++si) {
            const int kt = slow[si];
            const int ksg = ks_next, kps = kp_next;
            if (si + 1 < ns) {
                ks_next = seg_at(p.kv_seg, b, p.Lkv, slow[si + 1] * kTile + cj);
                kp_next = pos_at(p.kv_pos, b, p.Lkv, slow[si + 1] * kTile + cj);
            }
            bool seen_vis = false, seen_hid = false;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = r0 + 16 * k;
                const int sq = q_seg_s[i];
                bool vis = (sq == ksg) && !(p.q_seg && sq == p.pad_id);
                if (p.causal) vis = vis && (q_pos_s[i] >= kps);
                if (p.local_mask)
                    vis = vis && p.local_mask[(size_t)((qt * kTile + i) % p.lq_s) * p.lk_s +
                                              (kt * kTile + cj) % p.lk_s] != 0;
                seen_vis |= vis;
                seen_hid |= !vis;
            }
            const int any_vis = __syncthreads_or(seen_vis ? 1 : 0);
            const int any_hid = __syncthreads_or(seen_hid ? 1 : 0);
            if (any_vis && any_hid) {
                if (threadIdx.x == 0) crow[kt] = (uint8_t)RA_TILE_PARTIAL;
                continue;
            }
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

// Exclusive prefix sum of one value per thread over a block of 1024 threads
// (warp shuffles, then the 32 warp totals); `total` gets the block sum.
// `wsum` is 32 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int *wsum, int &total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += t;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = wsum[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        wsum[lane] = w; // inclusive over warps
    }
    __syncthreads();
    total = wsum[31];
    const int r = (wid > 0 ? wsum[wid - 1] : 0) + x - v;
    __syncthreads(); // wsum may be reused by the caller
    return r;
}

// Stable counting sort of ids 0..R-1 by descending cnt[id] (ties by id).
// One block of 1024 threads; hist needs (maxc + 1) ints of dynamic smem.
__device__ __forceinline__ void order_block(const int32_t *cnt, int R, int maxc, int32_t *order)
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
    int total;
    int run = block_exclusive_scan(sum, part, total);
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

__global__ void __launch_bounds__(1024) order_kernel(const int32_t *cnt, int R, int maxc,
                                                     int32_t *order)
{
    order_block(cnt, R, maxc, order);
}

// by_rows: exclusive prefix over rows of their partial counts, added to
// every per-shard entry of the row (entry N held the row's own total), and
// the grand total into n_part; else: exclusive prefix over columns.
__device__ __forceinline__ void part_scan_block(bool by_rows, int32_t *part_fwd, int rows, int n1,
                                                int32_t *part_bwd, int cols, int32_t *n_part)
{
    __shared__ int wsum[32];
    const int R = by_rows ? rows : cols;
    const int per = (R + 1023) / 1024;
    const int lo = min(R, (int)threadIdx.x * per), hi = min(R, lo + per);
    int sum = 0;
    for (int r = lo; r < hi; ++r)
        sum += by_rows ? part_fwd[(size_t)r * n1 + n1 - 1] : part_bwd[r];
    int total;
    int run = block_exclusive_scan(sum, wsum, total);
    if (by_rows && threadIdx.x == 0) *n_part = total;
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

// The row and column orders and the partial-tile numbering, which all read
// only the classified map: 4 blocks of 1024 threads, block 0 the row order
// (fwd_order), 1 the column order (bwd_order), 2 and 3 the row and column
// scans of the partial counts.  Dynamic smem: the larger histogram.
__global__ void __launch_bounds__(1024) orders_scans_kernel(const ra_block_mask m, int B, int nq, int nk,
                                                            int n1)
{
    switch (blockIdx.x) {
    case 0: order_block(m.fwd_cnt, B * nq, nk, m.fwd_order); break;
    case 1: order_block(m.bwd_cnt, B * nk, nq, m.bwd_order); break;
    case 2: part_scan_block(true, m.part_fwd, B * nq, n1, m.part_bwd, B * nk, m.n_part); break;
    default: part_scan_block(false, m.part_fwd, B * nq, n1, m.part_bwd, B * nk, m.n_part); break;
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

// grid (max(nq, nk), B, 2), 128 threads: block (x, b, 0) lists, in row
// order, the PARTIAL tiles of query-tile row (b, x) numbered below the
// capacity as (row id, kt); block (x, b, 1) lists those of key-tile column
// (b, x) in column order as (column id, qt).
__global__ void __launch_bounds__(128) part_list_kernel(Problem p, const uint8_t *cls,
                                                        const int32_t *fwd_cnt,
                                                        const int32_t *fwd_idx,
                                                        const int32_t *part_fwd,
                                                        const int32_t *bwd_cnt,
                                                        const int32_t *bwd_idx,
                                                        const int32_t *part_bwd, int2 *rows_list,
                                                        int2 *cols_list)
{
    const int b = blockIdx.y, x = blockIdx.x;
    const bool by_rows = blockIdx.z == 0;
    if (x >= (by_rows ? p.nq : p.nk)) return;
    __shared__ int plist[kTile], wcnt[4];
    const size_t id = (size_t)b * (by_rows ? p.nq : p.nk) + x;
    int slot = by_rows ? part_fwd[id * (p.N + 1)] : part_bwd[id];
    if (slot >= p.part_cap) return;
    const int cnt = by_rows ? fwd_cnt[id] : bwd_cnt[id];
    const int32_t *list = by_rows ? fwd_idx + id * p.nk : bwd_idx + id * p.nq;
    const size_t cls_base = by_rows ? id * p.nk : (size_t)b * p.nq * p.nk + x;
    const size_t cls_stride = by_rows ? 1 : p.nk;
    int2 *out = by_rows ? rows_list : cols_list;
    for (int e0 = 0; e0 < cnt && slot < p.part_cap; e0 += kTile) {
        const int n = gather_partial(list, cnt, e0, cls, cls_base, cls_stride, plist, wcnt);
        if ((int)threadIdx.x < n && slot + (int)threadIdx.x < p.part_cap)
            out[slot + threadIdx.x] = make_int2((int)id, plist[threadIdx.x]);
        slot += n;
        __syncthreads(); // plist is rewritten by the next chunk
    }
}

// Visibility word k (columns 32k..32k+31) of one row against 128 staged
// columns: bit z set iff column 32k + z is visible.
__device__ __forceinline__ uint32_t vis_word(int k, int seg, bool pad, int pos, const int *seg_s,
                                             const int *pos_s, bool row_is_query, int causal,
                                             bool q_seg_present, int pad_id)
{
    uint32_t bits = 0;
#pragma unroll 8
    for (int z = 0; z < 32; ++z) {
        const int j = 32 * k + z;
        bool v;
        if (row_is_query) {
            v = seg_s[j] == seg && !pad;
            if (causal) v = v && pos >= pos_s[j];
        } else {
            const int sq = seg_s[j];
            v = sq == seg && !(q_seg_present && sq == pad_id);
            if (causal) v = v && pos_s[j] >= pos;
        }
        bits |= (v ? 1u : 0u) << z;
    }
    return bits;
}

// grid (part_cap), 128 threads: block i writes the row-major bits of the
// i-th tile in row order and the transposed bits of the i-th tile in column
// order (when they exist).
__global__ void __launch_bounds__(128) part_bits_kernel(Problem p, const int32_t *n_part,
                                                        const int2 *rows_list,
                                                        const int2 *cols_list, uint32_t *rows_out,
                                                        uint32_t *cols_out)
{
    const int i = blockIdx.x, t = threadIdx.x;
    if (i >= min(*n_part, p.part_cap)) return;
    __shared__ int seg_s[kTile], pos_s[kTile];
    // ---- row-major block: thread t = query row t of the tile
    {
        const int2 e = rows_list[i];
        const int b = e.x / p.nq, qt = e.x - b * p.nq, kt = e.y;
        seg_s[t] = seg_at(p.kv_seg, b, p.Lkv, kt * kTile + t);
        pos_s[t] = pos_at(p.kv_pos, b, p.Lkv, kt * kTile + t);
        const int qi = qt * kTile + t;
        const int seg = seg_at(p.q_seg, b, p.Lq, qi);
        const int pos = pos_at(p.q_pos, b, p.Lq, qi);
        const bool pad = p.q_seg && seg == p.pad_id;
        __syncthreads();
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = vis_word(k, seg, pad, pos, seg_s, pos_s, true, p.causal, p.q_seg != nullptr, p.pad_id);
        if (p.local_mask) {
            const uint8_t *lm = p.local_mask + (size_t)(qi % p.lq_s) * p.lk_s + (kt * kTile) % p.lk_s;
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll 8
                for (int z = 0; z < 32; ++z)
                    if (!lm[32 * k + z]) w[k] &= ~(1u << z);
        }
        reinterpret_cast<uint4 *>(rows_out)[(size_t)i * kTile + t] = make_uint4(w[0], w[1], w[2], w[3]);
        __syncthreads(); // seg_s / pos_s are restaged below
    }
    // ---- transposed block: thread t = kv row t of the tile
    {
        const int2 e = cols_list[i];
        const int b = e.x / p.nk, kt = e.x - b * p.nk, qt = e.y;
        seg_s[t] = seg_at(p.q_seg, b, p.Lq, qt * kTile + t);
        pos_s[t] = pos_at(p.q_pos, b, p.Lq, qt * kTile + t);
        const int kj = kt * kTile + t;
        const int seg = seg_at(p.kv_seg, b, p.Lkv, kj);
        const int pos = pos_at(p.kv_pos, b, p.Lkv, kj);
        __syncthreads();
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = vis_word(k, seg, false, pos, seg_s, pos_s, false, p.causal, p.q_seg != nullptr, p.pad_id);
        if (p.local_mask) {
            const uint8_t *lm = p.local_mask + (size_t)((qt * kTile) % p.lq_s) * p.lk_s + kj % p.lk_s;
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll 8
                for (int z = 0; z < 32; ++z)
                    if (!lm[(size_t)(32 * k + z) * p.lk_s]) w[k] &= ~(1u << z);
        }
        reinterpret_cast<uint4 *>(cols_out)[(size_t)i * kTile + t] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

} // namespace

// The backward's grid of 64 query rows x 128 kv rows, one CTA per kv-tile
// column (thread j = kv row j).  Each non-empty 128 x 128 tile of the column
// gives its two 64-row halves: a FULL tile two FULL blocks; a PARTIAL tile
// is split by counting the visible pairs of each half from its stored column
// bits (or, past the block capacity, from positions and segments), so the
// classes are exact.  Lists keep ascending block order; each entry carries
// its parent's column-order partial number (-1 for FULL parents).
__global__ void __launch_bounds__(kTile) dkv_columns_kernel(Problem p, const uint8_t *cls,
                                                            const int32_t *bwd_cnt,
                                                            const int32_t *bwd_idx,
                                                            const int32_t *part_bwd,
                                                            const uint32_t *part_cols,
                                                            uint8_t *dkv_class, int32_t *dkv_cnt,
                                                            int32_t *dkv_idx, int32_t *dkv_slot)
{
    const int b = blockIdx.y, kt = blockIdx.x, j = threadIdx.x;
    const int nq2 = 2 * p.nq;
    const int col = b * p.nk + kt;
    __shared__ int red[kTile / 32];
    for (int qb = j; qb < nq2; qb += kTile)
        dkv_class[((size_t)b * nq2 + qb) * p.nk + kt] = RA_TILE_EMPTY;
    __syncthreads();
    const int kj = kt * kTile + j;
    const int kv_pos = p.kv_pos ? p.kv_pos[(size_t)b * p.Lkv + kj] : kj;
    const int kv_seg = p.kv_seg ? p.kv_seg[(size_t)b * p.Lkv + kj] : 0;
    const int cnt = bwd_cnt[col];
    const int32_t *list = bwd_idx + (size_t)col * p.nq;
    int32_t *oidx = dkv_idx + (size_t)col * nq2;
    int32_t *oslot = dkv_slot + (size_t)col * nq2;
    int slot = part_bwd[col], n = 0; // uniform over the CTA
    for (int e = 0; e < cnt; ++e) {
        const int qt = list[e];
        const uint8_t c = cls[((size_t)b * p.nq + qt) * p.nk + kt];
        uint8_t half_cls[2];
        int s = -1;
        if (c == RA_TILE_FULL) {
            half_cls[0] = half_cls[1] = RA_TILE_FULL;
        } else {
            s = slot++;
            for (int h = 0; h < 2; ++h) {
                uint2 bits;
                if (s < p.part_cap)
                    bits = reinterpret_cast<const uint2 *>(part_cols + ((size_t)s * kTile + j) * 4)[h];
                else
                    bits = col_bits_derived(p, b, qt * kTile + 64 * h, kj, kv_seg, kv_pos);
                int v = __popc(bits.x) + __popc(bits.y);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if ((j & 31) == 0) red[j >> 5] = v;
                __syncthreads();
                const int tot = red[0] + red[1] + red[2] + red[3];
                __syncthreads();
                half_cls[h] = tot == 0 ? RA_TILE_EMPTY
                                       : (tot == 64 * kTile ? RA_TILE_FULL : RA_TILE_PARTIAL);
            }
        }
        for (int h = 0; h < 2; ++h) {
            if (half_cls[h] == RA_TILE_EMPTY) continue;
            if (j == 0) {
                dkv_class[((size_t)b * nq2 + 2 * qt + h) * p.nk + kt] = half_cls[h];
                oidx[n] = 2 * qt + h;
                oslot[n] = s;
            }
            ++n;
        }
    }
    for (int r = n + j; r < nq2; r += kTile) {
        oidx[r] = -1;
        oslot[r] = -1;
    }
    if (j == 0) dkv_cnt[col] = n;
}

size_t mask_scratch_ints(int B, int nq, int nk, int N)
{
    const size_t local_tiles = (size_t)(nq / N) * (nk / N); // one byte each
    // tile summaries, local classes, and the two lists of numbered partial
    // tiles (an int2 per number) -- the lists first, for their alignment
    return (size_t)4 * mask_part_cap(B, nq, nk) +
           (size_t)B * (nq + nk) * (sizeof(TileSum) / sizeof(int32_t)) + (local_tiles + 3) / 4;
}

int mask_part_cap(int B, int nq, int nk)
{
    return 4 * B * (nq + nk);
}

cudaError_t launch_mask_build(const Problem &pin, const ra_block_mask &m, int32_t *scratch,
                              bool dkv_grid, cudaStream_t s)
{
    Problem p = pin;
    p.part_cap = m.part_cap;
    uint8_t *cls = m.tile_class;
    int2 *rows_list = reinterpret_cast<int2 *>(scratch);
    int2 *cols_list = rows_list + m.part_cap;
    TileSum *qsum = reinterpret_cast<TileSum *>(cols_list + m.part_cap);
    TileSum *ksum = qsum + (size_t)p.B * p.nq;
    uint8_t *lcls = reinterpret_cast<uint8_t *>(ksum + (size_t)p.B * p.nk);
    tile_summary_kernel<<<dim3(max(p.nq, p.nk), p.B, 2), 128, 0, s>>>(
        p.q_seg, p.q_pos, p.Lq, p.kv_seg, p.kv_pos, p.Lkv, p.pad_id, qsum, ksum);
    if (p.local_mask)
        local_tile_kernel<<<dim3(p.tq, p.tk), kCls, 0, s>>>(p.local_mask, p.lk_s, p.tk, lcls);
    classify_rows_kernel<<<dim3(p.nq, p.B), kCls, 0, s>>>(p, qsum, ksum, lcls, cls, m.fwd_cnt,
                                                          m.fwd_idx, m.fwd_shard, m.part_fwd);
    columns_kernel<<<dim3(p.nk, p.B), kCls, 0, s>>>(cls, p.nq, p.nk, m.bwd_cnt, m.bwd_idx,
                                                    m.part_bwd);
    // histograms of nk + 1 (rows) or nq + 1 (columns) counts: at most 8193
    // ints for 2^20 tokens, 37 KB with the partials, under the default limit
    const size_t sm_o = sizeof(int) * ((size_t)max(p.nq, p.nk) + 1 + 1024);
    orders_scans_kernel<<<4, 1024, sm_o, s>>>(m, p.B, p.nq, p.nk, p.N + 1);
    part_list_kernel<<<dim3(max(p.nq, p.nk), p.B, 2), kTile, 0, s>>>(
        p, cls, m.fwd_cnt, m.fwd_idx, m.part_fwd, m.bwd_cnt, m.bwd_idx, m.part_bwd, rows_list,
        cols_list);
    part_bits_kernel<<<m.part_cap, kTile, 0, s>>>(p, m.n_part, rows_list, cols_list, m.part_rows,
                                                 m.part_cols);
    if (!dkv_grid) return cudaGetLastError();
    dkv_columns_kernel<<<dim3(p.nk, p.B), kTile, 0, s>>>(p, cls, m.bwd_cnt, m.bwd_idx, m.part_bwd,
                                                         m.part_cols, m.dkv_class, m.dkv_cnt,
                                                         m.dkv_idx, m.dkv_slot);
    const size_t sm_d = sizeof(int) * ((size_t)2 * p.nq + 1 + 1024);
    if (sm_d > 48 * 1024) {
        // long sequences: the histogram of the 64-row grid's counts needs more
        // than the default dynamic shared memory (2^20 tokens: 69 KB)
        const cudaError_t e = cudaFuncSetAttribute(order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)sm_d);
        if (e != cudaSuccess) return e;
    }
    order_kernel<<<1, 1024, sm_d, s>>>(m.dkv_cnt, p.B * p.nk, 2 * p.nq, m.dkv_order);
    return cudaGetLastError();
}

} // namespace ra
