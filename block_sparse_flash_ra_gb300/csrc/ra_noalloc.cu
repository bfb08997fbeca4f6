// ra_noalloc.cu -- ra_attn_bwd_noalloc: the backward for callers that cannot
// allocate device memory for a workspace.
//
// Some callers of this library have no way to hand it a workspace: for
// example code embedded in a host runtime that owns and pre-reserves all of
// the GPU's memory, or plain-C callers with no allocator of their own.  For
// them this entry point runs the same backward kernels as ra_attn_bwd, with
// the workspace (per-row Delta and the dsinks partial sums) taken from a
// fixed-size array in the library's own device memory instead of a buffer
// passed by the caller.  It never calls cudaMalloc or cudaFree.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  Host code sees
// only a host-side stand-in for its name, so the device address is looked up
// with cudaGetSymbolAddress once per device, with that device current.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "ra_internal.h"

namespace ra {
namespace {

// 8 MiB: enough for B * Hq * Lq up to about one million query rows (8 bytes
// per row: Delta and -lse * log2 e), with room for the dsinks partial sums.
constexpr size_t kScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
void *g_scratch_addr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of g_bwd_scratch on the current device (set up on first use).
int scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_last_error(RA_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDev) return set_last_error(RA_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
        if (e != cudaSuccess || !ptr)
            return set_last_error(RA_ERR_CUDA, "cudaGetSymbolAddress of the backward scratch failed");
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return RA_OK;
}

} // namespace
} // namespace ra

extern "C" {

RA_API size_t ra_attn_bwd_noalloc_max_workspace(void) { return ra::kScratchBytes; }

RA_API int ra_attn_bwd_noalloc(const ra_attn_params *p, const void *q, const void *k,
                               const void *v, const void *out, const float *lse,
                               const void *dout, const ra_block_mask *mask, void *dq, void *dk,
                               void *dv, float *dsinks, ra_stream_t stream)
{
    // the arguments are checked exactly as ra_attn_bwd checks them (same codes),
    // before the problem's size is compared with the built-in scratch
    int rc = ra::bwd_all_validate(p, q, k, v, out, lse, dout, mask, dq, dk, dv, dsinks);
    if (rc) return rc;
    // the built-in scratch serves the schedule without a dK/dV head split
    const size_t need = ra::bwd_ws_min_bytes(p);
    if (need > ra::kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "ra_attn_bwd_noalloc: this problem needs %zu bytes of workspace, more than the "
                 "%zu bytes of built-in scratch; use ra_attn_bwd with a caller workspace",
                 need, ra::kScratchBytes);
        return ra::set_last_error(RA_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    rc = ra::scratch_address(&scratch);
    if (rc) return rc;
    // Every value the backward reads from its workspace is written earlier in
    // the same call, so nothing in the scratch has to start at zero.
    return ra::bwd_all(p, q, k, v, out, lse, dout, mask, dq, dk, dv, dsinks, scratch,
                       ra::kScratchBytes, stream, false);
}

} // extern "C"
