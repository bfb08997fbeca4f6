// ra_internal.h -- declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ra.h"

namespace ra {

constexpr int kTile = RA_TILE;            // canonical tile edge (tokens)
constexpr int RA_STATUS_TIMEOUT = 1;      // device status word value on a timed-out wait

// Everything a kernel needs to know about the problem, in device-friendly form.
struct Problem {
    int B, Lq, Lkv, Hq, Hkv, G, D;
    int nq, nk;          // tiles along q and kv
    int N;               // virtual ring shards
    int tq, tk;          // tiles per shard along q and kv
    float scale;
    float soft_cap;      // 0 = none
    int causal;
    int pad_id;
    const int32_t *q_pos, *kv_pos, *q_seg, *kv_seg;
    const float *sinks;
    const uint8_t *local_mask; // (lq_s, lk_s) per-shard mask of the non-causal ring, or NULL
    int lq_s, lk_s;            // Lq / N, Lkv / N
    // block map
    const uint8_t *tile_class;
    const int32_t *fwd_cnt, *fwd_idx, *bwd_cnt, *bwd_idx, *fwd_order, *bwd_order;
    const int32_t *fwd_shard; // (B*nq, N+1) first fwd_idx position of each KV shard
    // partial mask blocks: bits of PARTIAL tiles, numbered in row order
    // (part_fwd: first number at each shard start of a row) and in column
    // order (part_bwd: first number of each column); numbers >= part_cap have
    // no block and are masked from positions and segments
    const int32_t *part_fwd, *part_bwd;
    const uint32_t *part_rows, *part_cols; // (part_cap, 128, 4) words each
    int part_cap;
    // the backward's grid of 64 query rows x 128 kv rows: classes, per-column
    // lists of non-empty 64-row blocks with their parents' partial numbers,
    // and the longest-first column order
    const uint8_t *dkv_class;
    const int32_t *dkv_cnt, *dkv_idx, *dkv_slot, *dkv_order;
    // dK/dV schedule: each kv head's G query heads are split into hsplit
    // chunks of units; with hsplit > 1 each chunk stores its scaled dK and
    // dV as fp32 partials (dkv_part: dK then dV, each (hsplit, B, Lkv, Hkv, D))
    // that a reduction sums into dk, dv
    int hsplit;
    float *dkv_part;
    // one ring step (ra_attn_fwd_step / ra_attn_bwd_step): a single KV chunk
    // (N == 1) whose results are merged into, or added to, fp32 state in
    // global memory instead of being written as the final outputs.
    //   forward: run_out (B, Lq, Hq, D) and run_lse (B, Hq, Lq) are the
    //   running pair (read unless step_first, then written); step_sink counts
    //   the sinks in this step; the `out` of the launch (bf16, or fp32 for
    //   fp32 inputs), if not NULL, receives the merged result (the last
    //   step's cast).
    //   backward: acc_dq (B, Lq, Hq, D), acc_dk / acc_dv (B, Lkv, Hkv, D)
    //   receive += of the step's scaled gradients (hsplit == 1).
    float *run_out, *run_lse;
    int step_sink, step_first;
    float *acc_dq, *acc_dk, *acc_dv;
    // failure reporting
    int *status;
    uint64_t timeout_ns;
};

// ---- launchers (each returns cudaError_t of its launch) -------------------
cudaError_t launch_permute(const void *in, void *out, int B, int L, size_t row_bytes, int n,
                           int inverse, cudaStream_t s);
// Builds every array of `m` (device pointers) from the problem's positions,
// segments and local mask; `scratch` holds mask_scratch_ints() ints.
// Launches kMaskBuildKernels kernels, one more with a local mask.
cudaError_t launch_mask_build(const Problem &p, const ra_block_mask &m, int32_t *scratch,
                              bool dkv_grid, cudaStream_t s);
// kernels of a build; two more with the backward's 64-row grid (dkv_grid)
constexpr int kMaskBuildKernels = 6;
size_t mask_scratch_ints(int B, int nq, int nk, int N);
// slots of partial mask blocks in a map of B x nq x nk tiles
int mask_part_cap(int B, int nq, int nk);
cudaError_t launch_merge(float *out, float *lse, const float *bout, const float *blse, int B,
                         int L, int H, int D, cudaStream_t s);
// fp32 inputs: the forward on the tensor cores (kind::tf32, the logits from
// three hi / lo products); a ring step when p.run_out is set (out may then be
// NULL)
cudaError_t launch_fwd_f32_tc(const Problem &p, const float *q, const float *k, const float *v,
                              float *out, float *lse, cudaStream_t s);
cudaError_t launch_fwd_tc(const Problem &p, const void *tm_q, const void *tm_k, const void *tm_v,
                          void *out, float *lse, int num_sms, cudaStream_t s);
// The two-heads-per-CTA forward (D = 128, an even number of query heads per
// kv head): its workspace bytes, whether it serves a problem, attributes and
// launch (ws: fwd2_ws_bytes() bytes, 256-byte aligned).
size_t fwd2_ws_bytes();
bool fwd2_supported(const Problem &p);
cudaError_t fwd2_set_attributes();
cudaError_t launch_fwd2_tc(const Problem &p, const void *tm_q, const void *tm_k, const void *tm_v,
                           void *out, float *lse, float *ws, int num_sms, cudaStream_t s);
cudaError_t launch_bwd_pre(const Problem &p, const void *out, const void *dout, int dtype,
                           const float *lse, float *delta, float *nlse2, float *dsink_part,
                           float *dsinks, cudaStream_t s);
cudaError_t launch_bwd_dkdv_tc(const Problem &p, const void *tm_q, const void *tm_k,
                               const void *tm_v, const void *tm_do, const float *nlse2,
                               const float *delta, void *dk, void *dv, int num_sms,
                               cudaStream_t s);
// dK/dV on the backward's own grid (64 query rows per step, D = 128), and
// the sum of the head split's fp32 partials into dk, dv (hsplit > 1)
cudaError_t bwd_dkdv64_set_attributes();
cudaError_t launch_bwd_dkdv64_tc(const Problem &p, const void *tm_q64, const void *tm_k,
                                 const void *tm_v, const void *tm_do64, const float *nlse2,
                                 const float *delta, void *dk, void *dv, int num_sms,
                                 cudaStream_t s);
cudaError_t launch_dkv_reduce(const Problem &p, void *dk, void *dv, cudaStream_t s);
cudaError_t launch_bwd_dq_tc(const Problem &p, const void *tm_q, const void *tm_k,
                             const void *tm_v, const void *tm_do, const float *nlse2,
                             const float *delta, void *dq, int num_sms, cudaStream_t s);

// fp32 -> bf16 (or a copy for fp32) of n elements; acc += x over n floats
cudaError_t launch_cast_from_f32(const float *in, void *out, size_t n, int dtype, cudaStream_t s);
cudaError_t launch_add_f32(float *acc, const float *x, size_t n, cudaStream_t s);

cudaError_t launch_wait_selftest(int *status, uint64_t timeout_ns, int *gave_up, cudaStream_t s);

// dynamic shared memory the tensor-core kernels request (for attribute setup)
int fwd_tc_smem_bytes(int D);
int bwd_dkdv_smem_bytes(int D);
int bwd_dq_smem_bytes(int D);
cudaError_t fwd_tc_set_attributes(int D);
cudaError_t bwd_tc_set_attributes(int D);
cudaError_t f32tc_set_attributes(int D);

// ra_attn_bwd with the dK/dV head split allowed or not (without it the
// workspace needs only bwd_ws_min_bytes).
int bwd_all(const ra_attn_params *p, const void *q, const void *k, const void *v,
            const void *out, const float *lse, const void *dout, const ra_block_mask *mask,
            void *dq, void *dk, void *dv, float *dsinks, void *ws, size_t ws_bytes,
            ra_stream_t stream, bool allow_split);
size_t bwd_ws_min_bytes(const ra_attn_params *p);
// Every argument check of ra_attn_bwd except those of the workspace, with
// the same error codes and messages (RA_OK when the arguments are valid).
int bwd_all_validate(const ra_attn_params *p, const void *q, const void *k, const void *v,
                     const void *out, const float *lse, const void *dout,
                     const ra_block_mask *mask, const void *dq, const void *dk, const void *dv,
                     const float *dsinks);

// Records `msg` as this thread's last error message and returns `code`.
int set_last_error(int code, const char *msg);

} // namespace ra
