// ra_api.cu -- the C ABI declared in include/ra.h: argument validation,
// per-device property cache, TMA descriptor encoding and kernel dispatch.
// No allocation anywhere: every buffer comes from the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ra_internal.h"

namespace ra {

// Device-side status word (one per device that loads the library).
__device__ int g_status;

namespace {

thread_local char t_err[512] = "";

int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<uint64_t> g_launches{0};

void count(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

constexpr int kMaxDevices = 64;
struct DevCache {
    bool ready = false;
    int num_sms = 0;
    int *status = nullptr;
    bool attr_fwd64 = false, attr_fwd128 = false, attr_bwd64 = false, attr_bwd128 = false,
         attr_f32tc64 = false, attr_f32tc128 = false, attr_fwd2 = false, attr_dkdv64 = false;
};
DevCache g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int device_cache(DevCache **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DevCache &c = g_dev[dev];
    if (!c.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10)
            return fail(RA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                        dev, major, minor);
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&c.status), g_status);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        c.ready = true;
    }
    *out = &c;
    return RA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_params(const ra_attn_params *p)
{
    if (!p) return fail(RA_ERR_INVALID_ARG, "params is NULL");
    if (p->B <= 0 || p->Lq <= 0 || p->Lkv <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0)
        return fail(RA_ERR_INVALID_ARG, "sizes must be positive (B=%d Lq=%d Lkv=%d Hq=%d Hkv=%d D=%d)",
                    p->B, p->Lq, p->Lkv, p->Hq, p->Hkv, p->D);
    if (p->Hq % p->Hkv)
        return fail(RA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", p->Hq, p->Hkv);
    if (p->is_mqa && p->Hkv != 1)
        return fail(RA_ERR_INVALID_ARG, "is_mqa requires Hkv == 1 (got %d)", p->Hkv);
    if (p->n_virtual_shards < 1)
        return fail(RA_ERR_INVALID_ARG, "n_virtual_shards must be >= 1");
    const int N = p->n_virtual_shards;
    if (p->Lq % (RA_TILE * N) || p->Lkv % (RA_TILE * N))
        return fail(RA_ERR_INVALID_ARG,
                    "Lq (%d) and Lkv (%d) must be multiples of 128 * n_virtual_shards (%d)", p->Lq,
                    p->Lkv, RA_TILE * N);
    if ((long long)p->Lq > (1 << 20) || (long long)p->Lkv > (1 << 20))
        return fail(RA_ERR_UNSUPPORTED, "sequence lengths above 2^20 are not supported");
    if (p->dtype != RA_BF16 && p->dtype != RA_FP32)
        return fail(RA_ERR_INVALID_ARG, "dtype must be RA_BF16 or RA_FP32");
    if (!(p->scale > 0.f) || !(p->scale < 1e30f))
        return fail(RA_ERR_INVALID_ARG, "scale must be positive and finite");
    if ((p->q_seg == nullptr) != (p->kv_seg == nullptr))
        return fail(RA_ERR_INVALID_ARG, "q_seg and kv_seg must both be given or both be NULL");
    if (p->local_mask && p->causal)
        return fail(RA_ERR_INVALID_ARG, "local_mask is only defined for causal == 0 (the causal ring "
                                        "replaces the mask)");
    if (p->block_q_dkv != 0 && p->block_q_dkv != 64 && p->block_q_dkv != RA_TILE)
        return fail(RA_ERR_INVALID_ARG, "block_q_dkv must be 0, 64 or 128 (got %d)", p->block_q_dkv);
    if (p->block_q_dkv == 64 && p->D != 128)
        return fail(RA_ERR_UNSUPPORTED, "block_q_dkv = 64 is implemented for D = 128");
    const void *ptrs[6] = {p->q_pos, p->kv_pos, p->q_seg, p->kv_seg, p->sinks, p->local_mask};
    for (const void *x : ptrs)
        if (x && !aligned16(x))
            return fail(RA_ERR_INVALID_ARG,
                        "positions, segment ids, sinks and local_mask must be 16-byte aligned");
    return RA_OK;
}

uint64_t mix(uint64_t h, uint64_t v)
{
    h ^= v + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    return h;
}

// Fingerprint of the parameters a block map depends on.
uint64_t mask_key(const ra_attn_params *p)
{
    uint64_t h = 0x243f6a8885a308d3ull;
    h = mix(h, (uint64_t)p->B);
    h = mix(h, (uint64_t)p->Lq);
    h = mix(h, (uint64_t)p->Lkv);
    h = mix(h, (uint64_t)p->causal);
    h = mix(h, (uint64_t)p->n_virtual_shards);
    h = mix(h, (uint64_t)(uint32_t)p->pad_segment_id);
    h = mix(h, reinterpret_cast<uintptr_t>(p->q_pos));
    h = mix(h, reinterpret_cast<uintptr_t>(p->kv_pos));
    h = mix(h, reinterpret_cast<uintptr_t>(p->q_seg));
    h = mix(h, reinterpret_cast<uintptr_t>(p->kv_seg));
    h = mix(h, reinterpret_cast<uintptr_t>(p->local_mask));
    h = mix(h, (uint64_t)(p->block_q_dkv == 64 ? 64 : RA_TILE));
    return h;
}

struct MaskLayout {
    size_t cls, fwd_cnt, fwd_idx, bwd_cnt, bwd_idx, fwd_order, bwd_order, fwd_shard, part_fwd,
        part_bwd, part_rows, part_cols, n_part, dkv_class, dkv_cnt, dkv_idx, dkv_slot, dkv_order,
        scratch, total;
};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Query-head chunks of each dK/dV work unit: halved until the units number
// at least kDkdvTargetUnits (four per SM of a 152-SM GPU; a fixed figure, so
// that the workspace size does not depend on the device) or the group cannot
// be split further.  Few kv tiles and kv heads (MQA) otherwise leave too few
// units, each long, for an even spread over the SMs.
constexpr long kDkdvTargetUnits = 608;

int dkdv_head_split(const ra_attn_params *p)
{
    const long units = (long)p->B * (p->Lkv / RA_TILE) * p->Hkv;
    const int G = p->Hq / p->Hkv;
    int hs = 1;
    while (units * hs < kDkdvTargetUnits && G % (2 * hs) == 0) hs *= 2;
    return hs;
}

// Backward workspace: Delta and -lse*log2 e per row, dsinks partials per
// (b, head, q tile), and with a head split the fp32 dK / dV partials.
// bf16 copies of q, k, v and dout that the fp32 backward's tensor-core
// kernels read (fp32 inputs are rounded to bf16 once, in a prologue).
size_t bwd_f32_copy_bytes(const ra_attn_params *p)
{
    const size_t nq = (size_t)p->B * p->Lq * p->Hq * p->D, nk = (size_t)p->B * p->Lkv * p->Hkv * p->D;
    return 2 * up256(nq * 2) + 2 * up256(nk * 2);
}

size_t bwd_ws_bytes(const ra_attn_params *p, bool allow_split)
{
    const size_t rows = (size_t)p->B * p->Hq * p->Lq;
    const size_t part = (size_t)p->Hq * p->B * (p->Lq / RA_TILE);
    size_t n = 2 * up256(rows * 4) + up256(part * 4);
    // fp32 inputs: the gradients accumulate straight into the fp32 outputs,
    // so the query heads are never split; the bf16 copies come first
    if (p->dtype == RA_FP32) return bwd_f32_copy_bytes(p) + n;
    const int hs = allow_split ? dkdv_head_split(p) : 1;
    if (hs > 1) n += up256(2 * (size_t)hs * p->B * p->Lkv * p->Hkv * p->D * 4);
    return n;
}

MaskLayout mask_layout(const ra_attn_params *p)
{
    const size_t B = p->B, nq = p->Lq / RA_TILE, nk = p->Lkv / RA_TILE;
    MaskLayout m;
    size_t o = 0;
    m.cls = o;       o += up256(B * nq * nk);
    m.fwd_cnt = o;   o += up256(4 * B * nq);
    m.fwd_idx = o;   o += up256(4 * B * nq * nk);
    m.bwd_cnt = o;   o += up256(4 * B * nk);
    m.bwd_idx = o;   o += up256(4 * B * nk * nq);
    m.fwd_order = o; o += up256(4 * B * nq);
    m.bwd_order = o; o += up256(4 * B * nk);
    m.fwd_shard = o; o += up256(4 * B * nq * ((size_t)p->n_virtual_shards + 1));
    m.part_fwd = o;  o += up256(4 * B * nq * ((size_t)p->n_virtual_shards + 1));
    m.part_bwd = o;  o += up256(4 * B * nk);
    const size_t cap = (size_t)mask_part_cap((int)B, (int)nq, (int)nk);
    m.part_rows = o; o += up256(cap * RA_TILE * 16);
    m.part_cols = o; o += up256(cap * RA_TILE * 16);
    m.n_part = o;    o += 256;
    m.dkv_class = o; o += up256(B * 2 * nq * nk);
    m.dkv_cnt = o;   o += up256(4 * B * nk);
    m.dkv_idx = o;   o += up256(4 * B * nk * 2 * nq);
    m.dkv_slot = o;  o += up256(4 * B * nk * 2 * nq);
    m.dkv_order = o; o += up256(4 * B * nk);
    m.scratch = o;   o += up256(4 * mask_scratch_ints((int)B, (int)nq, (int)nk, p->n_virtual_shards));
    m.total = o;
    return m;
}

Problem make_problem(const ra_attn_params *p, const ra_block_mask *m, int *status)
{
    Problem x{};
    x.B = p->B;
    x.Lq = p->Lq;
    x.Lkv = p->Lkv;
    x.Hq = p->Hq;
    x.Hkv = p->Hkv;
    x.G = p->Hq / p->Hkv;
    x.D = p->D;
    x.nq = p->Lq / RA_TILE;
    x.nk = p->Lkv / RA_TILE;
    x.N = p->n_virtual_shards;
    x.tq = x.nq / x.N;
    x.tk = x.nk / x.N;
    x.scale = p->scale;
    x.soft_cap = p->soft_cap > 0.f ? p->soft_cap : 0.f;
    x.causal = p->causal ? 1 : 0;
    x.pad_id = p->pad_segment_id;
    x.q_pos = p->q_pos;
    x.kv_pos = p->kv_pos;
    x.q_seg = p->q_seg;
    x.kv_seg = p->kv_seg;
    x.sinks = p->sinks;
    x.local_mask = p->local_mask;
    x.lq_s = p->Lq / p->n_virtual_shards;
    x.lk_s = p->Lkv / p->n_virtual_shards;
    if (m) {
        x.tile_class = m->tile_class;
        x.fwd_cnt = m->fwd_cnt;
        x.fwd_idx = m->fwd_idx;
        x.bwd_cnt = m->bwd_cnt;
        x.bwd_idx = m->bwd_idx;
        x.fwd_order = m->fwd_order;
        x.bwd_order = m->bwd_order;
        x.fwd_shard = m->fwd_shard;
        x.part_fwd = m->part_fwd;
        x.part_bwd = m->part_bwd;
        x.part_rows = m->part_rows;
        x.part_cols = m->part_cols;
        x.part_cap = m->part_cap;
        x.dkv_class = m->dkv_class;
        x.dkv_cnt = m->dkv_cnt;
        x.dkv_idx = m->dkv_idx;
        x.dkv_slot = m->dkv_slot;
        x.dkv_order = m->dkv_order;
    }
    x.hsplit = 1;
    x.dkv_part = nullptr;
    x.run_out = x.run_lse = nullptr;
    x.step_sink = x.step_first = 0;
    x.acc_dq = x.acc_dk = x.acc_dv = nullptr;
    x.status = status;
    x.timeout_ns = g_timeout_ns.load();
    return x;
}

int check_mask(const ra_attn_params *p, const ra_block_mask *m)
{
    if (!m) return fail(RA_ERR_INVALID_ARG, "mask is NULL");
    if (!m->tile_class || !m->fwd_cnt || !m->fwd_idx || !m->bwd_cnt || !m->bwd_idx ||
        !m->fwd_order || !m->bwd_order || !m->fwd_shard || !m->part_fwd || !m->part_bwd ||
        !m->part_rows || !m->part_cols || !m->n_part || !m->dkv_class || !m->dkv_cnt ||
        !m->dkv_idx || !m->dkv_slot || !m->dkv_order)
        return fail(RA_ERR_INVALID_ARG, "mask has NULL arrays (not built?)");
    if (m->B != p->B || m->nq != p->Lq / RA_TILE || m->nk != p->Lkv / RA_TILE ||
        m->n_shards != p->n_virtual_shards || m->key != mask_key(p) ||
        m->part_cap != mask_part_cap(p->B, p->Lq / RA_TILE, p->Lkv / RA_TILE))
        return fail(RA_ERR_INVALID_ARG, "mask was built for other params (sizes, causal, shards, "
                                        "padding id or pos/seg arrays)");
    return RA_OK;
}

// 4-D TMA descriptor over a (B, L, H, D) bf16 tensor, box (64, 1, rows, 1),
// 128-byte swizzle: one box is `rows` token rows (128, or 64 for the dK/dV
// stage's query blocks) x 64 head-dim elements.
int encode_rows(CUtensorMap *map, const void *base, int B, int L, int H, int D, int rows = RA_TILE)
{
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                   (cuuint64_t)L * H * D * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return RA_OK;
}

} // namespace

int set_last_error(int code, const char *msg) { return fail(code, "%s", msg); }

} // namespace ra

using namespace ra;

extern "C" {

RA_API const char *ra_last_error(void) { return t_err; }

RA_API const char *ra_version(void) { return "ra-gb300 0.1 (sm_103a)"; }

RA_API void ra_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

RA_API uint64_t ra_launch_count(void) { return g_launches.load(); }

RA_API size_t ra_block_mask_bytes(const ra_attn_params *p)
{
    if (check_params(p) != RA_OK) return 0;
    return mask_layout(p).total;
}

RA_API int ra_build_block_mask(const ra_attn_params *p, void *buf, size_t buf_bytes,
                               ra_block_mask *out, ra_stream_t stream)
{
    int rc = check_params(p);
    if (rc) return rc;
    if (!out) return fail(RA_ERR_INVALID_ARG, "out is NULL");
    if (!buf) return fail(RA_ERR_INVALID_ARG, "buf is NULL");
    const MaskLayout L = mask_layout(p);
    if (buf_bytes < L.total)
        return fail(RA_ERR_WORKSPACE, "mask buffer has %zu bytes, needs %zu", buf_bytes, L.total);
    if (reinterpret_cast<uintptr_t>(buf) & 255u)
        return fail(RA_ERR_WORKSPACE, "mask buffer must be 256-byte aligned");
    DevCache *dc = nullptr;
    if ((rc = device_cache(&dc))) return rc;
    uint8_t *b = static_cast<uint8_t *>(buf);
    ra_block_mask m;
    m.tile_class = b + L.cls;
    m.fwd_cnt = reinterpret_cast<int32_t *>(b + L.fwd_cnt);
    m.fwd_idx = reinterpret_cast<int32_t *>(b + L.fwd_idx);
    m.bwd_cnt = reinterpret_cast<int32_t *>(b + L.bwd_cnt);
    m.bwd_idx = reinterpret_cast<int32_t *>(b + L.bwd_idx);
    m.fwd_order = reinterpret_cast<int32_t *>(b + L.fwd_order);
    m.bwd_order = reinterpret_cast<int32_t *>(b + L.bwd_order);
    m.fwd_shard = reinterpret_cast<int32_t *>(b + L.fwd_shard);
    m.part_fwd = reinterpret_cast<int32_t *>(b + L.part_fwd);
    m.part_bwd = reinterpret_cast<int32_t *>(b + L.part_bwd);
    m.part_rows = reinterpret_cast<uint32_t *>(b + L.part_rows);
    m.part_cols = reinterpret_cast<uint32_t *>(b + L.part_cols);
    m.n_part = reinterpret_cast<int32_t *>(b + L.n_part);
    m.dkv_class = b + L.dkv_class;
    m.dkv_cnt = reinterpret_cast<int32_t *>(b + L.dkv_cnt);
    m.dkv_idx = reinterpret_cast<int32_t *>(b + L.dkv_idx);
    m.dkv_slot = reinterpret_cast<int32_t *>(b + L.dkv_slot);
    m.dkv_order = reinterpret_cast<int32_t *>(b + L.dkv_order);
    m.B = p->B;
    m.nq = p->Lq / RA_TILE;
    m.nk = p->Lkv / RA_TILE;
    m.n_shards = p->n_virtual_shards;
    m.part_cap = mask_part_cap(m.B, m.nq, m.nk);
    m.key = mask_key(p);
    const Problem pr = make_problem(p, nullptr, dc->status);
    const bool dkv = p->block_q_dkv == 64;
    cudaError_t e = launch_mask_build(pr, m, reinterpret_cast<int32_t *>(b + L.scratch), dkv,
                                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "mask build launch");
    count(kMaskBuildKernels + (p->local_mask ? 1 : 0) + (dkv ? 2 : 0));
    *out = m;
    return RA_OK;
}

RA_API size_t ra_attn_fwd_workspace_size(const ra_attn_params *p)
{
    if (check_params(p) != RA_OK) return 0;
    const Problem pr = make_problem(p, nullptr, nullptr);
    return (p->dtype == RA_BF16 && fwd2_supported(pr)) ? fwd2_ws_bytes() : 0;
}

RA_API int ra_attn_fwd(const ra_attn_params *p, const void *q, const void *k, const void *v,
                       const ra_block_mask *mask, void *out, float *lse, void *ws,
                       size_t ws_bytes, ra_stream_t stream)
{
    (void)ws;
    (void)ws_bytes;
    int rc = check_params(p);
    if (rc) return rc;
    if (!q || !k || !v || !out || !lse) return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return fail(RA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    if ((rc = check_mask(p, mask))) return rc;
    if (p->D != 64 && p->D != 128) return fail(RA_ERR_UNSUPPORTED, "D must be 64 or 128 (got %d)", p->D);
    DevCache *dc = nullptr;
    if ((rc = device_cache(&dc))) return rc;
    const Problem pr = make_problem(p, mask, dc->status);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p->dtype == RA_FP32) {
        bool &done = p->D == 64 ? dc->attr_f32tc64 : dc->attr_f32tc128;
        if (!done) {
            if ((e = f32tc_set_attributes(p->D)) != cudaSuccess) return cuda_fail(e, "fp32 forward attributes");
            done = true;
        }
        e = launch_fwd_f32_tc(pr, static_cast<const float *>(q), static_cast<const float *>(k),
                              static_cast<const float *>(v), static_cast<float *>(out), lse, s);
        if (e != cudaSuccess) return cuda_fail(e, "forward (fp32) launch");
        count(1);
        return RA_OK;
    }
    alignas(64) CUtensorMap tq, tk, tv;
    if ((rc = encode_rows(&tq, q, p->B, p->Lq, p->Hq, p->D))) return rc;
    if ((rc = encode_rows(&tk, k, p->B, p->Lkv, p->Hkv, p->D))) return rc;
    if ((rc = encode_rows(&tv, v, p->B, p->Lkv, p->Hkv, p->D))) return rc;
    // two query heads per CTA when the problem allows it and the caller gave
    // the workspace for their running outputs; else one head per CTA
    if (fwd2_supported(pr) && ws && ws_bytes >= fwd2_ws_bytes() &&
        (reinterpret_cast<uintptr_t>(ws) & 255u) == 0) {
        if (!dc->attr_fwd2) {
            if ((e = fwd2_set_attributes()) != cudaSuccess) return cuda_fail(e, "forward attributes");
            dc->attr_fwd2 = true;
        }
        e = launch_fwd2_tc(pr, &tq, &tk, &tv, out, lse, static_cast<float *>(ws), dc->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e, "forward launch");
        count(1);
        return RA_OK;
    }
    bool &done = p->D == 64 ? dc->attr_fwd64 : dc->attr_fwd128;
    if (!done) {
        if ((e = fwd_tc_set_attributes(p->D)) != cudaSuccess) return cuda_fail(e, "forward attributes");
        done = true;
    }
    e = launch_fwd_tc(pr, &tq, &tk, &tv, out, lse, dc->num_sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    count(1);
    return RA_OK;
}

RA_API int ra_attn_fwd_step(const ra_attn_params *p, const void *q, const void *k, const void *v,
                            const ra_block_mask *mask, int flags, float *out_run, float *lse_run,
                            void *out, ra_stream_t stream)
{
    int rc = check_params(p);
    if (rc) return rc;
    if (p->n_virtual_shards != 1)
        return fail(RA_ERR_INVALID_ARG, "a ring step takes one key/value chunk: n_virtual_shards "
                                        "must be 1 (got %d)", p->n_virtual_shards);
    if (flags & ~(RA_STEP_SINKS | RA_STEP_FIRST)) return fail(RA_ERR_INVALID_ARG, "unknown step flags");
    if (!q || !k || !v || !out_run || !lse_run) return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out_run) ||
        !aligned16(lse_run) || (out && !aligned16(out)))
        return fail(RA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    if ((rc = check_mask(p, mask))) return rc;
    if (p->D != 64 && p->D != 128) return fail(RA_ERR_UNSUPPORTED, "D must be 64 or 128 (got %d)", p->D);
    if (out) {
        const size_t nrun = (size_t)p->B * p->Lq * p->Hq * p->D * 4;
        const size_t nout = nrun / (p->dtype == RA_BF16 ? 2 : 1);
        const uintptr_t a = reinterpret_cast<uintptr_t>(out), r = reinterpret_cast<uintptr_t>(out_run);
        if (a < r + nrun && r < a + nout) return fail(RA_ERR_INVALID_ARG, "out overlaps out_run");
    }
    DevCache *dc = nullptr;
    if ((rc = device_cache(&dc))) return rc;
    Problem pr = make_problem(p, mask, dc->status);
    pr.run_out = out_run;
    pr.run_lse = lse_run;
    pr.step_sink = (flags & RA_STEP_SINKS) ? 1 : 0;
    pr.step_first = (flags & RA_STEP_FIRST) ? 1 : 0;
    cudaError_t e;
    if (p->dtype == RA_FP32) {
        bool &done = p->D == 64 ? dc->attr_f32tc64 : dc->attr_f32tc128;
        if (!done) {
            if ((e = f32tc_set_attributes(p->D)) != cudaSuccess) return cuda_fail(e, "fp32 forward attributes");
            done = true;
        }
        e = launch_fwd_f32_tc(pr, static_cast<const float *>(q), static_cast<const float *>(k),
                              static_cast<const float *>(v), static_cast<float *>(out), lse_run,
                              reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "forward step (fp32) launch");
        count(1);
        return RA_OK;
    }
    bool &done = p->D == 64 ? dc->attr_fwd64 : dc->attr_fwd128;
    if (!done) {
        if ((e = fwd_tc_set_attributes(p->D)) != cudaSuccess) return cuda_fail(e, "forward attributes");
        done = true;
    }
    alignas(64) CUtensorMap tq, tk, tv;
    if ((rc = encode_rows(&tq, q, p->B, p->Lq, p->Hq, p->D))) return rc;
    if ((rc = encode_rows(&tk, k, p->B, p->Lkv, p->Hkv, p->D))) return rc;
    if ((rc = encode_rows(&tv, v, p->B, p->Lkv, p->Hkv, p->D))) return rc;
    e = launch_fwd_tc(pr, &tq, &tk, &tv, out, lse_run, dc->num_sms,
                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "forward step launch");
    count(1);
    return RA_OK;
}

RA_API int ra_cast_from_f32(const float *in, void *out, size_t n, int dtype, ra_stream_t stream)
{
    if (!in || !out) return fail(RA_ERR_INVALID_ARG, "NULL pointer");
    if (n == 0) return fail(RA_ERR_INVALID_ARG, "n must be positive");
    if (dtype != RA_BF16 && dtype != RA_FP32) return fail(RA_ERR_INVALID_ARG, "dtype must be RA_BF16 or RA_FP32");
    if (!aligned16(in) || !aligned16(out)) return fail(RA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    const size_t ob = n * (dtype == RA_BF16 ? 2 : 4);
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    if (a < b + ob && b < a + n * 4) return fail(RA_ERR_INVALID_ARG, "in and out overlap");
    cudaError_t e = launch_cast_from_f32(in, out, n, dtype, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cast launch");
    count(1);
    return RA_OK;
}

RA_API int ra_add_f32(float *acc, const float *x, size_t n, ra_stream_t stream)
{
    if (!acc || !x) return fail(RA_ERR_INVALID_ARG, "NULL pointer");
    if (n == 0) return fail(RA_ERR_INVALID_ARG, "n must be positive");
    const uintptr_t a = reinterpret_cast<uintptr_t>(acc), b = reinterpret_cast<uintptr_t>(x);
    if (a != b && a < b + n * 4 && b < a + n * 4) return fail(RA_ERR_INVALID_ARG, "acc and x overlap");
    cudaError_t e = launch_add_f32(acc, x, n, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "add launch");
    count(1);
    return RA_OK;
}

RA_API int ra_merge_out_lse(float *out, float *lse, const float *block_out, const float *block_lse,
                            int B, int L, int H, int D, ra_stream_t stream)
{
    if (!out || !lse || !block_out || !block_lse) return fail(RA_ERR_INVALID_ARG, "NULL pointer");
    if (B <= 0 || L <= 0 || H <= 0 || D <= 0 || D % 4)
        return fail(RA_ERR_INVALID_ARG, "sizes must be positive and D a multiple of 4");
    if (!aligned16(out) || !aligned16(block_out))
        return fail(RA_ERR_INVALID_ARG, "out and block_out must be 16-byte aligned");
    const size_t n = (size_t)B * L * H * D;
    const uintptr_t a = reinterpret_cast<uintptr_t>(out), bb = reinterpret_cast<uintptr_t>(block_out);
    if (a < bb + n * 4 && bb < a + n * 4) return fail(RA_ERR_INVALID_ARG, "out and block_out overlap");
    cudaError_t e = launch_merge(out, lse, block_out, block_lse, B, L, H, D,
                                 reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    count(1);
    return RA_OK;
}

RA_API size_t ra_attn_bwd_workspace_size(const ra_attn_params *p)
{
    if (check_params(p) != RA_OK) return 0;
    return bwd_ws_bytes(p, true);
}

} // extern "C"

namespace ra {
namespace {

enum BwdStage { kPrep = 1, kDkdv = 2, kDq = 4 };

// Backward workspace: Delta rows, the rows' -lse * log2 e, dsinks partials,
// and the dK / dV partials of a head split (hsplit > 1).
struct BwdWs {
    float *delta, *nlse2, *part, *dkv_part;
    int hsplit;
};

} // namespace

// Checks of the backward entry points that do not involve the workspace:
// params, tensor pointers, the mask, D and dtype.
int bwd_validate(const ra_attn_params *p, const void *const *ptrs, int nptrs,
                 const ra_block_mask *mask, bool allow_fp32 = false)
{
    int rc = check_params(p);
    if (rc) return rc;
    for (int i = 0; i < nptrs; ++i) {
        if (!ptrs[i]) return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
        if (!aligned16(ptrs[i])) return fail(RA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    }
    if (mask && (rc = check_mask(p, mask))) return rc;
    if (p->D != 64 && p->D != 128) return fail(RA_ERR_UNSUPPORTED, "D must be 64 or 128 (got %d)", p->D);
    if (p->dtype != RA_BF16 && !allow_fp32)
        return fail(RA_ERR_UNSUPPORTED, "this backward stage is implemented for bf16 inputs "
                                        "(ra_attn_bwd takes fp32 too)");
    return RA_OK;
}

int bwd_all_validate(const ra_attn_params *p, const void *q, const void *k, const void *v,
                     const void *out, const float *lse, const void *dout,
                     const ra_block_mask *mask, const void *dq, const void *dk, const void *dv,
                     const float *dsinks)
{
    if (!mask) return fail(RA_ERR_INVALID_ARG, "mask is NULL");
    if (p && p->sinks && !dsinks) return fail(RA_ERR_INVALID_ARG, "dsinks is NULL but sinks are given");
    const void *ptrs[9] = {q, k, v, out, lse, dout, dq, dk, dv};
    return bwd_validate(p, ptrs, 9, mask, true);
}

namespace {

// Shared checks of the backward entry points; on success fills the device
// cache and the workspace split.
int bwd_common(const ra_attn_params *p, const void *const *ptrs, int nptrs,
               const ra_block_mask *mask, void *ws, size_t ws_bytes, DevCache **dc, BwdWs *w,
               bool allow_split = true, bool allow_fp32 = false)
{
    int rc = bwd_validate(p, ptrs, nptrs, mask, allow_fp32);
    if (rc) return rc;
    const size_t need = bwd_ws_bytes(p, allow_split);
    if (!ws || ws_bytes < need)
        return fail(RA_ERR_WORKSPACE, "backward workspace has %zu bytes, needs %zu", ws_bytes, need);
    if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return fail(RA_ERR_WORKSPACE, "backward workspace must be 256-byte aligned");
    if ((rc = device_cache(dc))) return rc;
    const size_t rows_bytes = up256((size_t)p->B * p->Hq * p->Lq * 4);
    uint8_t *b = static_cast<uint8_t *>(ws) + (p->dtype == RA_FP32 ? bwd_f32_copy_bytes(p) : 0);
    w->delta = reinterpret_cast<float *>(b);
    w->nlse2 = reinterpret_cast<float *>(b + rows_bytes);
    w->part = reinterpret_cast<float *>(b + 2 * rows_bytes);
    w->hsplit = (allow_split && p->dtype != RA_FP32) ? dkdv_head_split(p) : 1;
    const size_t part_bytes = up256((size_t)p->Hq * p->B * (p->Lq / RA_TILE) * 4);
    w->dkv_part = w->hsplit > 1 ? reinterpret_cast<float *>(b + 2 * rows_bytes + part_bytes) : nullptr;
    return RA_OK;
}

// fp32 inputs of the backward: bf16 copies of q, k, v, dout in the front of
// ws (bwd_f32_copy_bytes of it), each rounded to nearest once; out16 gets
// the copies' addresses in that order
int bwd_f32_copies(const ra_attn_params *p, const void *q, const void *k, const void *v,
                   const void *dout, void *ws, const void **out16, cudaStream_t s)
{
    const size_t nq = (size_t)p->B * p->Lq * p->Hq * p->D, nk = (size_t)p->B * p->Lkv * p->Hkv * p->D;
    uint8_t *cb = static_cast<uint8_t *>(ws);
    void *q16 = cb, *do16 = cb + up256(nq * 2), *k16 = cb + 2 * up256(nq * 2),
         *v16 = cb + 2 * up256(nq * 2) + up256(nk * 2);
    const struct { const void *src; void *dst; size_t n; } casts[4] = {
        {q, q16, nq}, {dout, do16, nq}, {k, k16, nk}, {v, v16, nk}};
    for (const auto &c : casts) {
        cudaError_t e = launch_cast_from_f32(static_cast<const float *>(c.src), c.dst, c.n, RA_BF16, s);
        if (e != cudaSuccess) return cuda_fail(e, "fp32 -> bf16 cast launch");
        count(1);
    }
    out16[0] = q16, out16[1] = k16, out16[2] = v16, out16[3] = do16;
    return RA_OK;
}

int bwd_tc_kernels(const ra_attn_params *p, DevCache *dc, const Problem &pr, int stages,
                   const void *q, const void *k, const void *v, const void *dout,
                   const BwdWs &w, void *dq, void *dk, void *dv, cudaStream_t s)
{
    cudaError_t e;
    bool &done = p->D == 64 ? dc->attr_bwd64 : dc->attr_bwd128;
    if (!done) {
        if ((e = bwd_tc_set_attributes(p->D)) != cudaSuccess) return cuda_fail(e, "backward attributes");
        done = true;
    }
    int rc;
    alignas(64) CUtensorMap tq, tk, tv, tdo;
    if ((rc = encode_rows(&tq, q, p->B, p->Lq, p->Hq, p->D))) return rc;
    if ((rc = encode_rows(&tk, k, p->B, p->Lkv, p->Hkv, p->D))) return rc;
    if ((rc = encode_rows(&tv, v, p->B, p->Lkv, p->Hkv, p->D))) return rc;
    if ((rc = encode_rows(&tdo, dout, p->B, p->Lq, p->Hq, p->D))) return rc;
    if (stages & kDkdv) {
        Problem ps = pr;
        ps.hsplit = w.hsplit;
        ps.dkv_part = w.dkv_part;
        if (p->block_q_dkv == 64) {
            // the backward's own tile shape: 64 query rows per step
            if (!dc->attr_dkdv64) {
                if ((e = bwd_dkdv64_set_attributes()) != cudaSuccess)
                    return cuda_fail(e, "backward dK/dV attributes");
                dc->attr_dkdv64 = true;
            }
            alignas(64) CUtensorMap tq64, tdo64;
            if ((rc = encode_rows(&tq64, q, p->B, p->Lq, p->Hq, p->D, 64))) return rc;
            if ((rc = encode_rows(&tdo64, dout, p->B, p->Lq, p->Hq, p->D, 64))) return rc;
            e = launch_bwd_dkdv64_tc(ps, &tq64, &tk, &tv, &tdo64, w.nlse2, w.delta, dk, dv,
                                     dc->num_sms, s);
            if (e == cudaSuccess && w.hsplit > 1) e = launch_dkv_reduce(ps, dk, dv, s);
        } else {
            e = launch_bwd_dkdv_tc(ps, &tq, &tk, &tv, &tdo, w.nlse2, w.delta, dk, dv, dc->num_sms, s);
        }
        if (e != cudaSuccess) return cuda_fail(e, "backward dK/dV launch");
        count(w.hsplit > 1 ? 2 : 1);
    }
    if (stages & kDq) {
        e = launch_bwd_dq_tc(pr, &tq, &tk, &tv, &tdo, w.nlse2, w.delta, dq, dc->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e, "backward dQ launch");
        count(1);
    }
    return RA_OK;
}

} // namespace
} // namespace ra

extern "C" {

RA_API int ra_attn_bwd_prep(const ra_attn_params *p, const void *out, const float *lse,
                            const void *dout, float *dsinks, void *ws, size_t ws_bytes,
                            ra_stream_t stream)
{
    const void *ptrs[3] = {out, lse, dout};
    DevCache *dc = nullptr;
    BwdWs w{};
    // fp32 out / dout too: the ring's prep (Delta and dsinks in fp32)
    int rc = bwd_common(p, ptrs, 3, nullptr, ws, ws_bytes, &dc, &w, true, true);
    if (rc) return rc;
    if (p->sinks && !dsinks) return fail(RA_ERR_INVALID_ARG, "dsinks is NULL but sinks are given");
    const Problem pr = make_problem(p, nullptr, dc->status);
    cudaError_t e = launch_bwd_pre(pr, out, dout, p->dtype, lse, w.delta, w.nlse2, w.part, dsinks,
                                   reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "backward preprocessing launch");
    count(p->sinks ? 3 : 1);
    return RA_OK;
}

RA_API int ra_attn_bwd_dkdv(const ra_attn_params *p, const void *q, const void *k, const void *v,
                            const void *dout, const ra_block_mask *mask, void *dk, void *dv,
                            void *ws, size_t ws_bytes, ra_stream_t stream)
{
    if (!mask) return fail(RA_ERR_INVALID_ARG, "mask is NULL");
    const void *ptrs[6] = {q, k, v, dout, dk, dv};
    DevCache *dc = nullptr;
    BwdWs w{};
    int rc = bwd_common(p, ptrs, 6, mask, ws, ws_bytes, &dc, &w);
    if (rc) return rc;
    const Problem pr = make_problem(p, mask, dc->status);
    return bwd_tc_kernels(p, dc, pr, kDkdv, q, k, v, dout, w, nullptr, dk, dv,
                          reinterpret_cast<cudaStream_t>(stream));
}

RA_API int ra_attn_bwd_dq(const ra_attn_params *p, const void *q, const void *k, const void *v,
                          const void *dout, const ra_block_mask *mask, void *dq, void *ws,
                          size_t ws_bytes, ra_stream_t stream)
{
    if (!mask) return fail(RA_ERR_INVALID_ARG, "mask is NULL");
    const void *ptrs[5] = {q, k, v, dout, dq};
    DevCache *dc = nullptr;
    BwdWs w{};
    int rc = bwd_common(p, ptrs, 5, mask, ws, ws_bytes, &dc, &w);
    if (rc) return rc;
    const Problem pr = make_problem(p, mask, dc->status);
    return bwd_tc_kernels(p, dc, pr, kDq, q, k, v, dout, w, dq, nullptr, nullptr,
                          reinterpret_cast<cudaStream_t>(stream));
}

RA_API int ra_attn_bwd_step(const ra_attn_params *p, const void *q, const void *k, const void *v,
                            const void *dout, const ra_block_mask *mask, float *dq_acc,
                            float *dk_acc, float *dv_acc, void *ws, size_t ws_bytes,
                            ra_stream_t stream)
{
    if (!mask) return fail(RA_ERR_INVALID_ARG, "mask is NULL");
    if (p && p->n_virtual_shards != 1)
        return fail(RA_ERR_INVALID_ARG, "a ring step takes one key/value chunk: n_virtual_shards "
                                        "must be 1 (got %d)", p->n_virtual_shards);
    const void *ptrs[7] = {q, k, v, dout, dq_acc, dk_acc, dv_acc};
    DevCache *dc = nullptr;
    BwdWs w{};
    int rc = bwd_common(p, ptrs, 7, mask, ws, ws_bytes, &dc, &w, false, true);
    if (rc) return rc;
    Problem pr = make_problem(p, mask, dc->status);
    pr.acc_dq = dq_acc;
    pr.acc_dk = dk_acc;
    pr.acc_dv = dv_acc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (p->dtype == RA_FP32) {
        // the products read bf16 copies of this step's q, k, v, dout, made in
        // the front of ws (the part ra_attn_bwd_prep leaves alone)
        const void *c16[4];
        if ((rc = bwd_f32_copies(p, q, k, v, dout, ws, c16, s))) return rc;
        q = c16[0], k = c16[1], v = c16[2], dout = c16[3];
    }
    // the gradient kernels never write their bf16 outputs in this mode
    return bwd_tc_kernels(p, dc, pr, kDkdv | kDq, q, k, v, dout, w, dq_acc, dk_acc, dv_acc, s);
}

RA_API int ra_attn_bwd(const ra_attn_params *p, const void *q, const void *k, const void *v,
                       const void *out, const float *lse, const void *dout,
                       const ra_block_mask *mask, void *dq, void *dk, void *dv, float *dsinks,
                       void *ws, size_t ws_bytes, ra_stream_t stream)
{
    return ra::bwd_all(p, q, k, v, out, lse, dout, mask, dq, dk, dv, dsinks, ws, ws_bytes, stream,
                       true);
}

} // extern "C"

namespace ra {

int bwd_all(const ra_attn_params *p, const void *q, const void *k, const void *v,
            const void *out, const float *lse, const void *dout, const ra_block_mask *mask,
            void *dq, void *dk, void *dv, float *dsinks, void *ws, size_t ws_bytes,
            ra_stream_t stream, bool allow_split)
{
    int rc = bwd_all_validate(p, q, k, v, out, lse, dout, mask, dq, dk, dv, dsinks);
    if (rc) return rc;
    const void *ptrs[9] = {q, k, v, out, lse, dout, dq, dk, dv};
    DevCache *dc = nullptr;
    BwdWs w{};
    rc = bwd_common(p, ptrs, 9, mask, ws, ws_bytes, &dc, &w, allow_split, true);
    if (rc) return rc;
    Problem pr = make_problem(p, mask, dc->status);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_bwd_pre(pr, out, dout, p->dtype, lse, w.delta, w.nlse2, w.part, dsinks, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward preprocessing launch");
    count(p->sinks ? 3 : 1);
    if (p->dtype == RA_BF16)
        return bwd_tc_kernels(p, dc, pr, kDkdv | kDq, q, k, v, dout, w, dq, dk, dv, s);
    // fp32 inputs: Delta and dsinks above come from the fp32 out / dout; the
    // tensor-core kernels read bf16 copies of q, k, v, dout made here and add
    // their fp32 gradients into dq, dk, dv, zeroed first
    const void *c16[4];
    if ((rc = bwd_f32_copies(p, q, k, v, dout, ws, c16, s))) return rc;
    const size_t nq = (size_t)p->B * p->Lq * p->Hq * p->D, nk = (size_t)p->B * p->Lkv * p->Hkv * p->D;
    const struct { void *dst; size_t n; } zero[3] = {{dq, nq}, {dk, nk}, {dv, nk}};
    for (const auto &z : zero)
        if ((e = cudaMemsetAsync(z.dst, 0, z.n * 4, s)) != cudaSuccess) return cuda_fail(e, "gradient zeroing");
    pr.acc_dq = static_cast<float *>(dq);
    pr.acc_dk = static_cast<float *>(dk);
    pr.acc_dv = static_cast<float *>(dv);
    return bwd_tc_kernels(p, dc, pr, kDkdv | kDq, c16[0], c16[1], c16[2], c16[3], w, dq, dk, dv, s);
}

size_t bwd_ws_min_bytes(const ra_attn_params *p) { return bwd_ws_bytes(p, false); }

} // namespace ra

extern "C" {

RA_API int ra_permute_tokens(const void *in, void *out, int B, int L, size_t row_bytes,
                             int n_shards, ra_stream_t stream)
{
    if (!in || !out) return fail(RA_ERR_INVALID_ARG, "NULL pointer");
    if (B <= 0 || L <= 0 || row_bytes == 0 || n_shards <= 0)
        return fail(RA_ERR_INVALID_ARG, "sizes must be positive");
    if (L % (2 * n_shards)) return fail(RA_ERR_INVALID_ARG, "L (%d) must be a multiple of 2 * n_shards", L);
    const size_t n = (size_t)B * L * row_bytes;
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    if (a < b + n && b < a + n) return fail(RA_ERR_INVALID_ARG, "in and out overlap (out-of-place only)");
    cudaError_t e = launch_permute(in, out, B, L, row_bytes, n_shards, 0,
                                   reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "permute launch");
    count(1);
    return RA_OK;
}

RA_API int ra_unpermute_tokens(const void *in, void *out, int B, int L, size_t row_bytes,
                               int n_shards, ra_stream_t stream)
{
    if (!in || !out) return fail(RA_ERR_INVALID_ARG, "NULL pointer");
    if (B <= 0 || L <= 0 || row_bytes == 0 || n_shards <= 0)
        return fail(RA_ERR_INVALID_ARG, "sizes must be positive");
    if (L % (2 * n_shards)) return fail(RA_ERR_INVALID_ARG, "L (%d) must be a multiple of 2 * n_shards", L);
    const size_t n = (size_t)B * L * row_bytes;
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    if (a < b + n && b < a + n) return fail(RA_ERR_INVALID_ARG, "in and out overlap (out-of-place only)");
    cudaError_t e = launch_permute(in, out, B, L, row_bytes, n_shards, 1,
                                   reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "unpermute launch");
    count(1);
    return RA_OK;
}

RA_API int ra_selftest_wait_timeout(uint64_t timeout_ns, int *gave_up, ra_stream_t stream)
{
    if (!gave_up) return fail(RA_ERR_INVALID_ARG, "gave_up is NULL");
    DevCache *dc = nullptr;
    int rc = device_cache(&dc);
    if (rc) return rc;
    const uint64_t ns = timeout_ns ? timeout_ns : g_timeout_ns.load();
    cudaError_t e = launch_wait_selftest(dc->status, ns, gave_up, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    count(1);
    return RA_OK;
}

RA_API int ra_get_device_status(ra_stream_t stream)
{
    DevCache *dc = nullptr;
    int rc = device_cache(&dc);
    if (rc) return rc;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int v = 0;
    e = cudaMemcpy(&v, dc->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    const int zero = 0;
    e = cudaMemcpy(dc->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    if (v == RA_STATUS_TIMEOUT) return fail(RA_ERR_TIMEOUT, "a kernel wait timed out");
    return RA_OK;
}

} // extern "C"
