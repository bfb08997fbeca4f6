/*
 * ra.h -- C ABI of block-sparse masked flash attention with the ring
 * (out, lse) merge, for NVIDIA GB300 (sm_103a).
 *
 * What is computed (sources are named by page title and section):
 *   - "ejKernel ring_attention._ring_splash" module source:
 *       _update_out_and_lse      the sigmoid/softplus merge of a chunk's
 *                                partial (out, lse) into the running pair;
 *       _ring_attention_forward  the ring loop: step t of virtual device d
 *                                attends to the key/value chunk of source
 *                                (d - t) mod N, sinks only on step 0, soft cap;
 *       _ring_attention_backward dq accumulated locally, dk/dv travelling with
 *                                their chunk, dsinks summed over the ring;
 *       make_ring_attention      MaskInfo block metadata for forward and dkv.
 *   - "Kvax: Flash Attention for JAX":
 *       flash_attention          (batch, seq, heads, head_dim) layout,
 *                                positions, segment ids, PADDING_SEGMENT_ID,
 *                                scale, GQA via num_kv_heads;
 *       create_attention_mask    block-wise mask from positions and segments,
 *                                padding-only blocks skipped;
 *       context parallelism      permute tokens for load balance, unpermute
 *                                outputs.
 *
 * Semantics, for each batch b, query head h (kv head g = h / (Hq / Hkv)):
 *   visible(i, j) = q_seg[i] == kv_seg[j] && q_seg[i] != pad_segment_id
 *                   && (!causal || q_pos[i] >= kv_pos[j])
 *   s_ij   = scale * <q_i, k_j>;  if soft_cap > 0: s_ij = soft_cap * tanh(s_ij / soft_cap)
 *   lse_i  = log( sum_{visible j} exp(s_ij) + (sinks ? exp(sinks[h]) : 0) )
 *   out_i  = sum_{visible j} exp(s_ij - lse_i) v_j
 *   Invisible pairs are excluded; a row with nothing visible and no sink has
 *   out = 0, lse = -inf.  The forward walks the KV sequence as N virtual ring
 *   shards and merges each shard's partial into the running pair with the
 *   pages' update, which equals the formula above up to rounding.
 *
 * Conventions
 *   - Every pointer argument is a DEVICE pointer on the current CUDA device
 *     unless stated otherwise; the caller owns every buffer.  The library
 *     never allocates memory and keeps no state besides a per-device cache of
 *     device properties and kernel attributes.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous; argument errors are reported synchronously.
 *   - Layouts are dense, row-major: q, out, dout, dq (B, Lq, Hq, D);
 *     k, v, dk, dv (B, Lkv, Hkv, D); lse (B, Hq, Lq) fp32;
 *     positions / segment ids (B, L) int32; sinks (Hq) fp32.
 *   - Tiles are 128 x 128 tokens: Lq and Lkv must be multiples of
 *     128 * n_virtual_shards.
 *   - Device pointers handed to the attention calls must be 16-byte aligned.
 *   - Return value: RA_OK or a negative RA_ERR_* code; ra_last_error() gives
 *     a thread-local message for the last failing call of this thread.
 */
#ifndef RA_H
#define RA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RA_API __attribute__((visibility("default")))
#else
#define RA_API
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *ra_stream_t;

enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = -1, /* bad shape, pointer, alignment or mask */
    RA_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. D not in {64,128}) */
    RA_ERR_CUDA = -3,        /* a CUDA runtime call failed */
    RA_ERR_WORKSPACE = -4,   /* workspace missing or smaller than required */
    RA_ERR_TIMEOUT = -5      /* a kernel's bounded wait ran out (device status) */
};

enum { RA_BF16 = 0, RA_FP32 = 1 };
enum { RA_TILE_EMPTY = 0, RA_TILE_PARTIAL = 1, RA_TILE_FULL = 2 };
#define RA_TILE 128

/*
 * Problem description shared by every attention call.
 *   B, Lq, Lkv, Hq, Hkv, D  sizes; D in {64, 128}; Hq % Hkv == 0.
 *   dtype            RA_BF16 or RA_FP32: element type of q, k, v, out, dout,
 *                    dq, dk, dv.  Accumulation is always fp32.
 *   scale            multiplies <q, k> before the cap (Kvax `scale`).
 *   soft_cap         > 0 applies cap * tanh(s / cap); <= 0 disables it
 *                    (_ring_splash `logits_soft_cap`).
 *   causal           1: a pair is visible only if q_pos >= kv_pos.
 *   is_mqa           1: one kv head shared by all query heads (requires
 *                    Hkv == 1); _ring_splash `is_mqa`.
 *   n_virtual_shards N >= 1 ring shards of Lq / N query and Lkv / N key rows.
 *   pad_segment_id   segment id that marks padding (Kvax PADDING_SEGMENT_ID;
 *                    this library's reading: -1).  Padding is never visible.
 *   q_pos, kv_pos    (B, L) int32 positions, or NULL for the token's index in
 *                    the sequence as passed (after any permutation).
 *   q_seg, kv_seg    (B, L) int32 segment ids, or NULL for a single segment
 *                    without padding.  Both or neither.
 *   sinks            (Hq) fp32 sink logits, counted once per row in the
 *                    denominator only, or NULL.
 *   local_mask       (Lq/N, Lkv/N) uint8, nonzero = visible, or NULL: the
 *                    2-D mask of _ring_splash make_ring_attention, which the
 *                    non-causal ring applies at every ring step, so pair
 *                    (i, j) also needs local_mask[i mod Lq/N][j mod Lkv/N].
 *                    Only with causal == 0 (the pages' causal ring replaces
 *                    the mask; the combination is rejected here).  16-byte
 *                    aligned; owned by the caller, read by the block-map
 *                    build and by the attention kernels on partial tiles.
 *   block_q_dkv      query rows per step of the backward's dK/dV stage: 0 or
 *                    128 (the default: 128 x 128 tiles, the forward's grid)
 *                    or 64 (the backward's own grid of 64 query rows x 128
 *                    kv rows, _ring_splash make_ring_attention's
 *                    block_q_dkv with has_backward_blocks; D = 128 only).
 *                    The block map then also carries the dkv_* arrays.
 */
typedef struct {
    int B, Lq, Lkv, Hq, Hkv, D;
    int dtype;
    float scale;
    float soft_cap;
    int causal;
    int is_mqa;
    int n_virtual_shards;
    int pad_segment_id;
    const int32_t *q_pos;
    const int32_t *kv_pos;
    const int32_t *q_seg;
    const int32_t *kv_seg;
    const float *sinks;
    const uint8_t *local_mask;
    int block_q_dkv;
} ra_attn_params;

/*
 * Block map on the 128 x 128 tile grid (nq = Lq / 128, nk = Lkv / 128),
 * the counterpart of the pages' MaskInfo.  All arrays live in one caller
 * buffer carved by ra_build_block_mask.
 *   tile_class  (B, nq, nk) uint8: RA_TILE_EMPTY / PARTIAL / FULL.
 *   fwd_cnt     (B*nq) non-empty tiles in each query-tile row.
 *   fwd_idx     (B*nq, nk) their kt, ascending, padded with -1.
 *   bwd_cnt     (B*nk) non-empty tiles in each key-tile column.
 *   bwd_idx     (B*nk, nq) their qt, ascending, padded with -1.
 *   fwd_order   (B*nq) row ids b*nq+qt by descending fwd_cnt, ties by id
 *               (the longest-first schedule of the forward).
 *   bwd_order   (B*nk) column ids b*nk+kt, same rule (backward schedule).
 *   fwd_shard   (B*nq, N+1) with N = n_virtual_shards: entry s of a row is
 *               the position in its fwd_idx row of the first tile with
 *               kt >= s*nk/N, so KV shard s owns fwd_idx[fwd_shard[s] ..
 *               fwd_shard[s+1]) (entry N = fwd_cnt).  The forward walks a
 *               row's shards in ring order through these offsets.
 * Partial mask blocks (the pages' MaskInfo partial_mask_blocks): the
 * visibility bits of PARTIAL tiles, stored once per tile and shared by every
 * head, so the attention kernels mask a partial tile with one 8-byte load per
 * thread instead of re-deriving it from positions and segments.  PARTIAL
 * tiles are numbered twice: in row order (by b*nq+qt, then kt ascending) and
 * in column order (by b*nk+kt, then qt ascending); the first part_cap of each
 * numbering have a block, the rest are masked from positions and segments.
 *   part_fwd    (B*nq, N+1): entry s of a row is the row-order number of the
 *               first PARTIAL tile at or after fwd_idx position fwd_shard[s]
 *               of that row (entry 0: the row's first, entry N: one past its
 *               last).
 *   part_bwd    (B*nk): column-order number of each column's first PARTIAL
 *               tile.
 *   part_rows   (part_cap, 128, 4) uint32, row-order: bit z of word w of row i
 *               is set iff query row qt*128+i sees kv row kt*128+32w+z.
 *   part_cols   (part_cap, 128, 4) uint32, column-order: bit z of word w of
 *               row j is set iff query row qt*128+32w+z sees kv row kt*128+j.
 *   n_part      (1) int32: PARTIAL tiles in the map (blocks stored:
 *               min(n_part, part_cap)).
 * The backward's own grid (make_ring_attention's dkv MaskInfo with
 * block_sizes.has_backward_blocks; Kvax create_attention_mask's backward
 * mask): blocks of 64 query rows x 128 kv rows, which the dK/dV stage walks
 * when params.block_q_dkv == 64 (filled only then):
 *   dkv_class   (B, 2*nq, nk) uint8: EMPTY / PARTIAL / FULL of each block.
 *   dkv_cnt     (B*nk) non-empty 64-row query blocks of each kv-tile column.
 *   dkv_idx     (B*nk, 2*nq) their 64-row block index, ascending, -1 padded.
 *   dkv_slot    (B*nk, 2*nq) for each listed block, the column-order number
 *               of its 128 x 128 parent when that is PARTIAL (the parent's
 *               stored bits give the block's visibility), -1 when FULL.
 *   dkv_order   (B*nk) column ids by descending dkv_cnt, ties by id.
 *   part_cap    4 * B * (nq + nk).
 *   key         fingerprint of the ra_attn_params fields the map depends on;
 *               attention calls reject a map built for other params.
 */
typedef struct {
    uint8_t *tile_class;
    int32_t *fwd_cnt;
    int32_t *fwd_idx;
    int32_t *bwd_cnt;
    int32_t *bwd_idx;
    int32_t *fwd_order;
    int32_t *bwd_order;
    int32_t *fwd_shard;
    int32_t *part_fwd;
    int32_t *part_bwd;
    uint32_t *part_rows;
    uint32_t *part_cols;
    int32_t *n_part;
    uint8_t *dkv_class;
    int32_t *dkv_cnt;
    int32_t *dkv_idx;
    int32_t *dkv_slot;
    int32_t *dkv_order;
    int B, nq, nk, n_shards, part_cap;
    uint64_t key;
} ra_block_mask;

/* Thread-local message of the last failing call on this thread ("" if none). */
RA_API const char *ra_last_error(void);

/* Library version string. */
RA_API const char *ra_version(void);

/*
 * Bytes of the device buffer ra_build_block_mask needs for params `p`
 * (0 if `p` is invalid; ra_last_error says why).
 */
RA_API size_t ra_block_mask_bytes(const ra_attn_params *p);

/*
 * Classifies every 128 x 128 tile from positions and segment ids and builds
 * the tile lists and schedules (make_ring_attention's forward and dkv
 * MaskInfo; Kvax create_attention_mask with padding-only tiles skipped).
 * Result is bit-exact: a tile is EMPTY iff no pair is visible, FULL iff all
 * 128*128 pairs are, PARTIAL otherwise; the partial mask blocks hold the
 * exact visibility bits of the PARTIAL tiles they cover.
 *   buf, buf_bytes  device buffer of at least ra_block_mask_bytes(p) bytes,
 *                   256-byte aligned; owned by the caller and must outlive
 *                   every call that uses `out`.
 *   out             host struct filled with device pointers into `buf`.
 * Errors: RA_ERR_INVALID_ARG (params, null pointers), RA_ERR_WORKSPACE
 * (buffer too small or misaligned), RA_ERR_CUDA.
 */
RA_API int ra_build_block_mask(const ra_attn_params *p, void *buf, size_t buf_bytes,
                               ra_block_mask *out, ra_stream_t stream);

/* Workspace bytes of ra_attn_fwd: 0 when the forward keeps its running state
 * on chip; for bf16 inputs with D = 128 and an even number of query heads
 * per kv head (GQA, MQA) the forward runs two query heads per CTA and keeps
 * their running ring outputs in this fp32 workspace (one fixed-size slot per
 * CTA, about 40 MiB whatever the problem size).  Passing a smaller workspace
 * (or none) is allowed: the forward then runs one head per CTA. */
RA_API size_t ra_attn_fwd_workspace_size(const ra_attn_params *p);

/*
 * Forward (_ring_attention_forward on N virtual shards, one launch).
 *   q (B,Lq,Hq,D), k, v (B,Lkv,Hkv,D) in p->dtype;  mask from
 *   ra_build_block_mask for the same params;  out (B,Lq,Hq,D) in p->dtype;
 *   lse (B,Hq,Lq) fp32 natural-log (-inf for rows with nothing visible).
 *   For each query tile the shards are visited in ring order
 *   s = (d - t) mod N (d = the tile's own shard, t = 0..N-1), empty tiles are
 *   skipped, the sink enters at t = 0 only, and each shard's partial is merged
 *   into the running (out, lse) by the sigmoid/softplus update.
 *   ws, ws_bytes: optional workspace (ra_attn_fwd_workspace_size, 256-byte
 *   aligned), see above; results are the same either way up to rounding.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA.
 */
RA_API int ra_attn_fwd(const ra_attn_params *p, const void *q, const void *k, const void *v,
                       const ra_block_mask *mask, void *out, float *lse, void *ws,
                       size_t ws_bytes, ra_stream_t stream);

/*
 * _update_out_and_lse, elementwise and in place:
 *   out (B,L,H,D) fp32, lse (B,H,L) fp32 running pair;
 *   block_out, block_lse the chunk's partial, same layouts.
 *   Where lse == -inf the block is taken as is; otherwise
 *   w = sigmoid(block_lse - lse), out -= w * (out - block_out),
 *   lse += softplus(block_lse - lse).
 *   out / block_out must not overlap and must be 16-byte aligned;
 *   D % 4 == 0.
 * Errors: RA_ERR_INVALID_ARG (NULL, sizes, alignment, overlap), RA_ERR_CUDA.
 */
RA_API int ra_merge_out_lse(float *out, float *lse, const float *block_out,
                            const float *block_lse, int B, int L, int H, int D,
                            ra_stream_t stream);

/* Workspace bytes of ra_attn_bwd: per-row Delta = <dO, O> and per-row
 * -lse * log2(e) (fp32, B*Hq*Lq each), per-tile partial sums of dsinks, and,
 * when the kv tiles times kv heads are few (B * Lkv/128 * Hkv < 608, e.g.
 * MQA), fp32 partial dK and dV of each chunk of query heads (2 * hs * B * Lkv
 * * Hkv * D floats, hs = the number of chunks, a power of two dividing
 * Hq/Hkv): the dK/dV stage then splits each kv head's query heads over hs
 * work units, so that the units spread evenly over the SMs, and sums the
 * partials afterwards.  For fp32 inputs: no split, and bf16 copies of q, k,
 * v and dout (2 bytes per element) in front. */
RA_API size_t ra_attn_bwd_workspace_size(const ra_attn_params *p);

/*
 * Backward (_ring_attention_backward): the exact gradient of ra_attn_fwd's
 * output, computed with the final out and lse.
 *   q, k, v, out, dout in p->dtype (bf16, or fp32: Delta and dsinks are then
 *   formed from the fp32 out and dout, the tensor-core products read bf16
 *   copies of q, k, v and dout made in the workspace -- each input rounded to
 *   bf16 once -- and the gradients accumulate in fp32 straight into dq, dk,
 *   dv); lse from ra_attn_fwd;
 *   dq (B,Lq,Hq,D), dk, dv (B,Lkv,Hkv,D) in p->dtype, overwritten (dk, dv
 *   summed over the query heads that share a kv head);
 *   dsinks (Hq) fp32, overwritten, summed over batch and all rows; may be
 *   NULL only when p->sinks is NULL.
 *   ws: at least ra_attn_bwd_workspace_size(p) bytes, 256-byte aligned.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_WORKSPACE, RA_ERR_CUDA.
 */
RA_API int ra_attn_bwd(const ra_attn_params *p, const void *q, const void *k, const void *v,
                       const void *out, const float *lse, const void *dout,
                       const ra_block_mask *mask, void *dq, void *dk, void *dv, float *dsinks,
                       void *ws, size_t ws_bytes, ra_stream_t stream);

/*
 * The three stages ra_attn_bwd runs, for callers that schedule or time them
 * one by one.  Arguments mean what they mean for ra_attn_bwd and obey the
 * same rules; the stages communicate through `ws`, so for one problem they
 * must run in this order on one stream (or be ordered by the caller):
 *   ra_attn_bwd_prep  Delta = rowsum(dO * O) and -lse * log2(e) into ws,
 *                     and dsinks (if sinks);
 *   ra_attn_bwd_dkdv  dk, dv (one work unit per kv head and 128-row kv tile);
 *   ra_attn_bwd_dq    dq     (one work unit per query head and query tile).
 * dkdv and dq read lse and Delta only through ws.  These two stages take
 * bf16 inputs only (RA_ERR_UNSUPPORTED for fp32); ra_attn_bwd and
 * ra_attn_bwd_prep take both (fp32: Delta and dsinks from the fp32 out and
 * dout, as ra_attn_bwd forms them).
 */
RA_API int ra_attn_bwd_prep(const ra_attn_params *p, const void *out, const float *lse,
                            const void *dout, float *dsinks, void *ws, size_t ws_bytes,
                            ra_stream_t stream);
RA_API int ra_attn_bwd_dkdv(const ra_attn_params *p, const void *q, const void *k, const void *v,
                            const void *dout, const ra_block_mask *mask, void *dk, void *dv,
                            void *ws, size_t ws_bytes, ra_stream_t stream);
RA_API int ra_attn_bwd_dq(const ra_attn_params *p, const void *q, const void *k, const void *v,
                          const void *dout, const ra_block_mask *mask, void *dq, void *ws,
                          size_t ws_bytes, ra_stream_t stream);

/*
 * ra_attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory themselves (code running inside a host runtime that owns all
 * of the GPU's memory, or plain-C callers with no allocator at hand).  The
 * pages have no counterpart of this call; it is a convenience of this
 * library.
 *   Same arguments, results and errors as ra_attn_bwd, minus ws / ws_bytes.
 *   The workspace comes from a fixed array of ra_attn_bwd_noalloc_max_workspace()
 *   bytes (8 MiB) in the library's device memory, held by every GPU that loads
 *   the library until the process exits.  Problems whose
 *   workspace exceeds it fail with RA_ERR_WORKSPACE (roughly B * Hq * Lq
 *   above one million query rows; this call never splits the query heads of
 *   the dK/dV stage, so it needs no dK/dV partials); use ra_attn_bwd then.
 *   Nothing is allocated: no cudaMalloc / cudaFree is ever called.
 *   The first call on a device looks up the array's device address on that
 *   device (a synchronous runtime query); make that first call before any
 *   stream capture begins.  The address is kept for the life of the process:
 *   after a cudaDeviceReset (or on another context of the same device) it is
 *   stale, so this call is not supported once the device has been reset.
 *   All calls share the one array and it keeps the last call's contents.
 *   Calls whose GPU work overlaps in time (different streams, different
 *   threads, without ordering between them) race on it and give wrong
 *   results: order them on one stream.
 */
RA_API int ra_attn_bwd_noalloc(const ra_attn_params *p, const void *q, const void *k,
                               const void *v, const void *out, const float *lse,
                               const void *dout, const ra_block_mask *mask, void *dq, void *dk,
                               void *dv, float *dsinks, ra_stream_t stream);
RA_API size_t ra_attn_bwd_noalloc_max_workspace(void);

/*
 * One step of the ring, for callers that run the ring themselves -- one
 * query shard per GPU, key/value chunks passed from device to device
 * ("ejKernel ring_attention._ring_splash" module source,
 * _ring_attention_forward: the loop body; _ring_attention_backward: the
 * scan body).  The params describe the step's pair: Lq = the local query
 * rows, Lkv = the rows of the key/value chunk this step holds, and
 * n_virtual_shards = 1; positions and segment ids of the chunk travel with
 * it (kv_pos / kv_seg), so that the causal rule q_pos >= kv_pos is the pages'
 * per-step offset device_idx * q_len - kv_src * kv_len when the positions are
 * the tokens' global indices.  The block map is built for these params.
 */
enum { RA_STEP_SINKS = 1, RA_STEP_FIRST = 2 };

/*
 * Forward step: the chunk's partial (out, lse) -- with the sinks in the
 * denominator when flags has RA_STEP_SINKS (the pages: step 0 only) -- merged
 * by _update_out_and_lse into the running pair.
 *   q (B,Lq,Hq,D), k, v (B,Lkv,Hkv,D) in p->dtype (bf16, or fp32: then the
 *   products are those of ra_attn_fwd for fp32): the local queries and the
 *   chunk.
 *   out_run (B,Lq,Hq,D) fp32 and lse_run (B,Hq,Lq) fp32: the running pair,
 *   read and written in place; with RA_STEP_FIRST they are not read and the
 *   running pair is taken as (0, -inf) (the pages' initial state).
 *   out: NULL, or (B,Lq,Hq,D) in p->dtype, not overlapping out_run, that also
 *   receives the merged output (the final cast to the query dtype after the
 *   last step).
 * lse_run ends as the natural-log lse of the rows over every chunk merged so
 * far (-inf for rows with nothing visible).
 * Errors: RA_ERR_INVALID_ARG (n_virtual_shards != 1, flags, pointers, mask,
 * out overlapping out_run), RA_ERR_UNSUPPORTED (D), RA_ERR_CUDA.
 */
RA_API int ra_attn_fwd_step(const ra_attn_params *p, const void *q, const void *k, const void *v,
                            const ra_block_mask *mask, int flags, float *out_run, float *lse_run,
                            void *out, ra_stream_t stream);

/*
 * Backward step: the gradient contributions of the pair (local queries, this
 * chunk), computed with the FINAL out and lse, added to fp32 accumulators:
 *   dq_acc (B,Lq,Hq,D) += this chunk's part of dq (the local accumulator);
 *   dk_acc, dv_acc (B,Lkv,Hkv,D) += the local queries' part of the chunk's
 *   dk, dv (the accumulators that travel with the chunk).
 * ws: the workspace ra_attn_bwd_prep filled for the same local rows (Delta,
 * -lse * log2 e); run ra_attn_bwd_prep once per backward, before the steps
 * (it also gives this device's dsinks, whose sum over the devices is the
 * pages' psum).  The query heads of a kv head are never split here.  With
 * fp32 inputs the step also writes bf16 copies of q, k, v, dout into the
 * front of ws, a part ra_attn_bwd_prep does not use (so steps sharing one ws
 * must be ordered, as the ring orders them anyway).
 * Errors: as ra_attn_bwd.
 */
RA_API int ra_attn_bwd_step(const ra_attn_params *p, const void *q, const void *k, const void *v,
                            const void *dout, const ra_block_mask *mask, float *dq_acc,
                            float *dk_acc, float *dv_acc, void *ws, size_t ws_bytes,
                            ra_stream_t stream);

/*
 * The ring's last elementwise steps (_ring_attention_backward: the casts of
 * dq, dk, dv "to input dtypes"; the psum of dsinks).
 *   ra_cast_from_f32: out[i] = in[i] in `dtype` (RA_BF16: round to nearest
 *   even; RA_FP32: a copy), n elements, buffers 16-byte aligned and disjoint.
 *   ra_add_f32: acc[i] += x[i], n floats (the sum of per-device dsinks when
 *   several ring devices share one GPU).
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_CUDA.
 */
RA_API int ra_cast_from_f32(const float *in, void *out, size_t n, int dtype, ra_stream_t stream);
RA_API int ra_add_f32(float *acc, const float *x, size_t n, ra_stream_t stream);

/*
 * Zigzag load-balancing permutation along the sequence (Kvax context
 * parallelism).  The sequence of L rows is split into 2N chunks of L/(2N);
 * virtual device d holds chunk d followed by chunk 2N-1-d, so permuted row
 * p = d*(L/N) + r comes from row d*c + r if r < c, else (2N-1-d)*c + r - c,
 * with c = L/(2N).
 *   in, out      (B, L, row_bytes) device buffers, must not overlap.
 *   row_bytes    bytes per token row (any element type; copied bitwise).
 * ra_unpermute_tokens applies the inverse.
 * Errors: RA_ERR_INVALID_ARG (L % (2N) != 0, in == out, null), RA_ERR_CUDA.
 */
RA_API int ra_permute_tokens(const void *in, void *out, int B, int L, size_t row_bytes,
                             int n_shards, ra_stream_t stream);
RA_API int ra_unpermute_tokens(const void *in, void *out, int B, int L, size_t row_bytes,
                               int n_shards, ra_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: RA_OK, or RA_ERR_TIMEOUT if a kernel gave up a bounded wait.
 * The library caches, per device, the device address of this word and the
 * kernels' attributes on first use; resetting the device (cudaDeviceReset)
 * after the library's first call on it is not supported.
 */
RA_API int ra_get_device_status(ra_stream_t stream);

/* Number of CUDA kernels this library has launched in this process (all
 * devices, all threads); lets callers count the library's launches in a
 * region without a profiler. */
RA_API uint64_t ra_launch_count(void);

/* Upper bound, in nanoseconds, of any single in-kernel wait (default 2e9).
 * Applies to launches made after the call, from any thread. */
RA_API void ra_set_wait_timeout_ns(uint64_t ns);

/*
 * Failure-detection self-test: launches one block whose single in-kernel
 * wait can never complete (an mbarrier nothing arrives at).  The wait gives
 * up after timeout_ns (0 = the current ra_set_wait_timeout_ns limit), exactly
 * as the waits of the attention kernels do, and records the timeout in the
 * device status word; the kernel then returns and the context stays usable.
 *   gave_up: device int, set to 1 when the wait gave up (0 otherwise).
 * Read the outcome with ra_get_device_status (RA_ERR_TIMEOUT expected).
 * Errors: RA_ERR_INVALID_ARG (gave_up NULL), RA_ERR_CUDA.
 */
RA_API int ra_selftest_wait_timeout(uint64_t timeout_ns, int *gave_up, ra_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RA_H */
