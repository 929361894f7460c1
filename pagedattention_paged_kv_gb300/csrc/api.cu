// api.cu -- the extern "C" entry points of libpagedkv.so (declared in
// include/pagedkv.h): argument checks, launch planning, TMA descriptors, launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <atomic>

#include "../../include/pagedkv.h"
#include "paged_decode.cuh"
#include "paged_prefill.cuh"
#include "paged_varlen.cuh"

namespace pkv {
cudaError_t launch_reshape_and_cache(void *k_cache, void *v_cache, const void *k, const void *v,
                                     const int64_t *slot_mapping, int64_t num_tokens,
                                     int64_t num_slots, int row_bytes, int num_sms, int *err,
                                     cudaStream_t stream);
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *pairs, int64_t num_pairs,
                               int64_t num_blocks, int64_t block_bytes, int num_sms, int *err,
                               cudaStream_t stream);
cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, int num_sms, cudaStream_t stream);
cudaError_t launch_reshape_and_cache_fp8(void *k_cache, void *v_cache, const void *k, const void *v,
                                         const int64_t *slot_mapping, int64_t num_tokens,
                                         int64_t num_slots, int row_elems, float k_scale,
                                         float v_scale, int num_sms, int *err, cudaStream_t stream);
}

// The device error word (one per device that loads the library).
__device__ int g_pkv_device_error;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kBlockSize = 16;
constexpr int kMaxDecodeItems = 8192;

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;
    int *err = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];

// Limit of a kernel's pipeline waits (pkv_set_wait_limit_ns); read at each launch.
std::atomic<uint64_t> g_wait_ns{pkv::kWaitTimeoutNs};
// Split-K of the decode rows (pkv_set_decode_split); read at each launch.
std::atomic<int> g_decode_split{1};

// Measured GB300 rates behind the varlen grid split (paged_varlen.cu).  A decode CTA that
// shares the GPU with prefill CTAs streams ~83 GB/s of bf16 K/V (~42 GB/s of FP8 codes);
// alone, a few decode CTAs reach ~95-105 (~48) GB/s each.  The whole decode saturates near
// 5.9 TB/s; a prefill CTA sustains ~7.8 TFLOP/s of causal attention.  On the 512-token
// chunk + 127 decodes step these rates put the split at the measured optimum (32 of 152
// CTAs decode, with a bf16 or an FP8 cache).
constexpr float kDecodeBytesPerUsSm = 83e3f;
constexpr float kDecodeBytesPerUsSmFp8 = 42e3f;
constexpr float kDecodeBytesPerUsGpu = 5.9e6f;
constexpr float kPrefillFlopPerUsSm = 7.8e6f;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device facts, looked up once per device with that device current.
int device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PKV_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
            return PKV_ERR_CUDA;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err), g_pkv_device_error) !=
            cudaSuccess)
            return PKV_ERR_CUDA;
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return PKV_ERR_CUDA;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return PKV_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Tensor map over a KV cache [num_blocks][16][num_kv_heads][head_dim] with its
// dimensions listed as (column in a 64-wide chunk, token, head, chunk, block): the
// strides are not in memory order, which lets one box of 16 tokens x box_heads heads x
// 64 columns land in shared memory as [head][token][64] -- every head's 16 rows
// contiguous, so the 128-byte swizzle spreads an 8-token ldmatrix over all banks.  One
// box moves box_heads * 2 KiB; a block's K (or V) for box_heads heads takes
// head_dim / 64 boxes.
// With an FP8 cache (fp8 = true) an element is one byte, so a 128-byte chunk holds 128
// columns: head_dim 128 is one chunk and one box per block row.
int encode_cache_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int block_size,
                     int num_kv_heads, int head_dim, int box_heads, bool fp8 = false) {
    const int elem = fp8 ? 1 : 2;
    const int cw = 128 / elem;  // columns per 128-byte chunk
    const cuuint64_t row = (cuuint64_t)num_kv_heads * head_dim * elem;  // bytes per token
    cuuint64_t dims[5] = {(cuuint64_t)cw, (cuuint64_t)block_size, (cuuint64_t)num_kv_heads,
                          (cuuint64_t)(head_dim / cw), (cuuint64_t)num_blocks};
    cuuint64_t strides[4] = {row, (cuuint64_t)head_dim * elem, 128, row * block_size};
    // a box is one 16-token slice of a block (block sizes >= 16) or one whole 8-token block
    const cuuint32_t box_tokens = block_size < 16 ? (cuuint32_t)block_size : 16u;
    cuuint32_t box[5] = {(cuuint32_t)cw, box_tokens, (cuuint32_t)box_heads, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                          const_cast<void *>(cache), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// Tensor map over q [total_q][num_heads][head_dim] for the chunked-prefill tiles: one
// box is `tokens` consecutive query rows x the `group` heads of one KV head x 64
// columns, landing in shared memory as [token][head][64] (row = token * group + head),
// 128-byte swizzled -- the K-major A operand of the tensor-core MMA.
int encode_q_map(CUtensorMap *map, const void *q, int total_q, int num_heads, int head_dim,
                 int group, int tokens) {
    cuuint64_t dims[4] = {64, (cuuint64_t)(head_dim / 64), (cuuint64_t)num_heads,
                          (cuuint64_t)total_q};
    cuuint64_t strides[3] = {128, (cuuint64_t)head_dim * 2, (cuuint64_t)num_heads * head_dim * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)group, (cuuint32_t)tokens};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// ---- decode planning -------------------------------------------------------
struct DecodePlan {
    int group, warps_per_head, heads_per_cta, head_tiles, items, stage_bytes, num_stages, grid;
    size_t smem;
    size_t off_jobs, off_ml, off_o, bytes;
};

int plan_decode(int num_seqs, int num_heads, int num_kv_heads, int head_dim, const DeviceInfo &d,
                DecodePlan *p, int elem_bytes = 2) {
    p->group = num_heads / num_kv_heads;
    p->warps_per_head = (p->group + 15) / 16;
    if (p->warps_per_head > 8) return PKV_ERR_UNSUPPORTED;
    int ht = 1;
    for (int c = 1; c <= num_kv_heads; ++c)
        if (num_kv_heads % c == 0 && c * p->warps_per_head <= 8) ht = c;
    p->heads_per_cta = ht;
    p->head_tiles = num_kv_heads / ht;
    p->items = num_seqs * p->head_tiles;
    if (p->items > kMaxDecodeItems) return PKV_ERR_UNSUPPORTED;
    p->stage_bytes = ht * head_dim * kBlockSize * elem_bytes;
    const size_t fixed = pkv::decode_smem_bytes(0, 0, p->items);
    const int budget = d.smem_optin;
    int nst = (int)((budget - (int64_t)fixed) / (p->stage_bytes + 16));
    // 6 bf16 stages (192 KiB in flight): deeper rings measured no faster; an FP8 ring
    // keeps the same bytes in flight with twice the stages
    const int cap = elem_bytes == 1 ? 12 : 6;
    if (nst > cap) nst = cap;
    if (nst < 2) return PKV_ERR_UNSUPPORTED;
    p->num_stages = nst;
    p->smem = pkv::decode_smem_bytes(p->stage_bytes, nst, p->items);
    p->grid = d.sms < 256 ? d.sms : 256;  // the merge kernels hold <= 256 parts per item
    const size_t rows = (size_t)ht * p->group;
    p->off_jobs = 0;
    p->off_ml = round_up(sizeof(pkv::MergeJob) * (size_t)p->grid, 256);
    p->off_o = p->off_ml + round_up(2 * (size_t)p->grid * rows * 8, 256);
    p->bytes = p->off_o + round_up(2 * (size_t)p->grid * rows * head_dim * 4, 256);
    return PKV_OK;
}

int check_common(int num_seqs, int max_blocks_per_seq, int num_heads, int num_kv_heads,
                 int head_dim, int block_size, int64_t num_blocks, int dtype) {
    if (num_seqs < 0 || max_blocks_per_seq < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    // decode: pool blocks of 8, 16, 32 or 64 tokens (prefill rows need 16, checked there)
    if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64)
        return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_blocks * block_size > (int64_t)UINT32_MAX) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * max_blocks_per_seq * num_kv_heads > (int64_t)INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// The decode kernel's tensor maps and arguments for the sequences selected by
// `query_start_loc` (all if null).
int prepare_decode(pkv::DecodeArgs &a, CUtensorMap &kmap, CUtensorMap &vmap, void *out, const void *q,
                   const int32_t *query_start_loc, int total_q, const void *k_cache,
                   const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                   int num_seqs, int max_blocks_per_seq, int num_heads, int num_kv_heads,
                   int head_dim, int64_t num_blocks, float scale, uint8_t *ws, size_t ws_bytes,
                   const DeviceInfo &d, const DecodePlan &p, int block_size, bool fp8, float k_scale,
                   float v_scale, const void *k_new, const void *v_new) {
    if (ws_bytes < p.bytes || !ws) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(ws, 256)) return PKV_ERR_INVALID_ARG;
    const int box_heads = block_size < kBlockSize ? 1 : p.heads_per_cta;
    int st = encode_cache_map(&kmap, k_cache, num_blocks, block_size, num_kv_heads, head_dim, box_heads,
                              fp8);
    if (st == PKV_OK)
        st = encode_cache_map(&vmap, v_cache, num_blocks, block_size, num_kv_heads, head_dim, box_heads,
                              fp8);
    if (st != PKV_OK) return st;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start_loc = query_start_loc;
    a.total_q = total_q;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.block_size = block_size;
    a.num_heads = num_heads;
    a.group = p.group;
    a.heads_per_cta = p.heads_per_cta;
    a.head_tiles = p.head_tiles;
    a.warps_per_head = p.warps_per_head;
    a.num_stages = p.num_stages;
    a.grid = p.grid;
    a.min_blocks_per_cta = 2;
    a.num_blocks = num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f * k_scale;
    a.v_scale = v_scale;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache_w = const_cast<void *>(k_cache);
    a.v_cache_w = const_cast<void *>(v_cache);
    a.k_scale_q = k_scale;
    a.v_scale_q = v_scale;
    a.ws_jobs = reinterpret_cast<pkv::MergeJob *>(ws + p.off_jobs);
    a.ws_ml = reinterpret_cast<float2 *>(ws + p.off_ml);
    a.ws_o = reinterpret_cast<float *>(ws + p.off_o);
    a.err = d.err;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    a.whole_items = g_decode_split.load(std::memory_order_relaxed) ? 0 : 1;
    return PKV_OK;
}

// Runs the decode kernel (and its merge) on the sequences selected by `query_start_loc`
// (all if null).
int run_decode(void *out, const void *q, const int32_t *query_start_loc, int total_q,
               const void *k_cache,
               const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
               int num_seqs, int max_blocks_per_seq, int num_heads, int num_kv_heads,
               int head_dim, int64_t num_blocks, float scale, uint8_t *ws, size_t ws_bytes,
               const DeviceInfo &d, const DecodePlan &p, cudaStream_t stream, int block_size,
               bool fp8 = false, float k_scale = 1.f, float v_scale = 1.f, const void *k_new = nullptr,
               const void *v_new = nullptr) {
    pkv::DecodeArgs a;
    CUtensorMap kmap, vmap;
    const int st = prepare_decode(a, kmap, vmap, out, q, query_start_loc, total_q, k_cache, v_cache,
                                  block_tables, context_lens, num_seqs, max_blocks_per_seq, num_heads,
                                  num_kv_heads, head_dim, num_blocks, scale, ws, ws_bytes, d, p, block_size,
                                  fp8, k_scale, v_scale, k_new, v_new);
    if (st != PKV_OK) return st;
    return pkv::launch_paged_decode(head_dim, fp8, kmap, vmap, a, p.smem, stream) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

}  // namespace

extern "C" const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_OOM: return "out of blocks";
        case PKV_ERR_DEVICE_DATA: return "invalid device data";
        case PKV_ERR_STATIC_SCRATCH_LIMIT: return "sizes exceed the static scratch limit";
        default: return "unknown status";
    }
}

extern "C" int pkv_get_device_error(void *stream) {
    DeviceInfo *d = nullptr;
    int st = device_info(&d);
    if (st != PKV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaMemcpyAsync(&h, d->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaMemsetAsync(d->err, 0, sizeof(int), s) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    return h;
}

extern "C" void pkv_set_decode_split(int enabled) {
    g_decode_split.store(enabled ? 1 : 0, std::memory_order_relaxed);
}

extern "C" void pkv_set_wait_limit_ns(uint64_t limit_ns) {
    g_wait_ns.store(limit_ns == 0 ? pkv::kWaitTimeoutNs : limit_ns, std::memory_order_relaxed);
}

extern "C" int pkv_reshape_and_cache(void *k_cache, void *v_cache, const void *k, const void *v,
                                     const int64_t *slot_mapping, int64_t num_tokens,
                                     int64_t num_blocks, int block_size, int num_kv_heads,
                                     int head_dim, int dtype, void *stream) {
    if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_cache || !v_cache || !k || !v || !slot_mapping) return PKV_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
    if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k, 16) || !aligned(v, 16) ||
        !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    int st = device_info(&d);
    if (st != PKV_OK) return st;
    cudaError_t e = pkv::launch_reshape_and_cache(k_cache, v_cache, k, v, slot_mapping, num_tokens,
                                                  num_blocks * block_size, (int)row_bytes, d->sms,
                                                  d->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_reshape_and_cache_fp8(void *k_cache, void *v_cache, const void *k, const void *v,
                                         const int64_t *slot_mapping, int64_t num_tokens,
                                         int64_t num_blocks, int block_size, int num_kv_heads,
                                         int head_dim, float k_scale, float v_scale, void *stream) {
    if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_cache || !v_cache || !k || !v || !slot_mapping) return PKV_ERR_INVALID_ARG;
    const int64_t row_elems = (int64_t)num_kv_heads * head_dim;
    if (row_elems % 16 != 0 || row_elems > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k, 16) || !aligned(v, 16) ||
        !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    int st = device_info(&d);
    if (st != PKV_OK) return st;
    cudaError_t e = pkv::launch_reshape_and_cache_fp8(k_cache, v_cache, k, v, slot_mapping, num_tokens,
                                                      num_blocks * block_size, (int)row_elems, k_scale,
                                                      v_scale, d->sms, d->err,
                                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *block_pairs,
                               int64_t num_pairs, int64_t num_blocks, int block_size, int num_kv_heads,
                               int head_dim, int dtype, void *stream) {
    if (num_pairs < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_DTYPE_BF16 && dtype != PKV_DTYPE_FP8_E4M3) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_INVALID_ARG;
    const int64_t block_bytes =
        (int64_t)block_size * num_kv_heads * head_dim * (dtype == PKV_DTYPE_BF16 ? 2 : 1);
    if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 4))
        return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    int st = device_info(&d);
    if (st != PKV_OK) return st;
    cudaError_t e = pkv::launch_copy_blocks(k_cache, v_cache, block_pairs, num_pairs, num_blocks, block_bytes,
                                            d->sms, d->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Host <-> device copies of a step's buffers, done by the SMs when the host side is
// page-locked memory mapped into the device's address space (transfer.cu); other host
// memory goes through cudaMemcpyAsync.  See pagedkv.h.
static int step_copy(void *dst, const void *src, size_t bytes, void *stream, bool to_device) {
    if (bytes == 0) return PKV_OK;
    if (!dst || !src) return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    int st = device_info(&d);
    if (st != PKV_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const void *host = to_device ? src : dst;
    const void *devp = to_device ? dst : src;
    cudaPointerAttributes da, ha;
    if (cudaPointerGetAttributes(&da, devp) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_INVALID_ARG;
    }
    if (da.type != cudaMemoryTypeDevice || da.device != dev) return PKV_ERR_INVALID_ARG;
    bool mapped = false;
    if (cudaPointerGetAttributes(&ha, host) == cudaSuccess) {
        mapped = ha.type == cudaMemoryTypeHost && ha.devicePointer != nullptr;
    } else {
        cudaGetLastError();
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!mapped) {
        return cudaMemcpyAsync(dst, src, bytes, to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost, s) ==
                       cudaSuccess
                   ? PKV_OK
                   : PKV_ERR_CUDA;
    }
    void *hdev = ha.devicePointer;  // the host buffer's address in the device's space
    cudaError_t e = to_device ? pkv::launch_copy(dst, hdev, (int64_t)bytes, d->sms, s)
                              : pkv::launch_copy(hdev, src, (int64_t)bytes, d->sms, s);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_copy_to_device(void *dst, const void *src, size_t bytes, void *stream) {
    return step_copy(dst, src, bytes, stream, true);
}

extern "C" int pkv_copy_to_host(void *dst, const void *src, size_t bytes, void *stream) {
    return step_copy(dst, src, bytes, stream, false);
}

extern "C" size_t pkv_workspace_size(int op, int num_seqs, int total_q_tokens, int num_heads,
                                     int num_kv_heads, int head_dim, int block_size) {
    if (check_common(num_seqs, 0, num_heads, num_kv_heads, head_dim, block_size, 0,
                     PKV_DTYPE_BF16) != PKV_OK)
        return 0;
    DeviceInfo *d = nullptr;
    if (device_info(&d) != PKV_OK) return 0;
    DecodePlan p;
    if (plan_decode(num_seqs, num_heads, num_kv_heads, head_dim, *d, &p) != PKV_OK) return 0;
    if (op == PKV_OP_DECODE) return p.bytes;
    if (op != PKV_OP_VARLEN || total_q_tokens < 0) return 0;
    pkv::PrefillPlan pp;
    if (pkv::plan_prefill(num_seqs, num_heads, num_kv_heads, head_dim, d->sms, d->smem_optin,
                          &pp) != PKV_OK)
        return round_up(p.bytes, 256);  // decode rows only (prefill rows unsupported)
    return round_up(p.bytes, 256) + pp.ws_bytes;
}

extern "C" int pkv_paged_attention_decode(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, int num_seqs,
                                          int max_blocks_per_seq, int num_heads, int num_kv_heads,
                                          int head_dim, int block_size, int64_t num_blocks,
                                          float scale, int dtype, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    int st = check_common(num_seqs, max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, dtype);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16))
        return PKV_ERR_INVALID_ARG;
    if (num_blocks == 0 || max_blocks_per_seq == 0) return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    st = device_info(&d);
    if (st != PKV_OK) return st;
    DecodePlan p;
    st = plan_decode(num_seqs, num_heads, num_kv_heads, head_dim, *d, &p);
    if (st != PKV_OK) return st;
    return run_decode(out, q, nullptr, num_seqs, k_cache, v_cache, block_tables, context_lens, num_seqs,
                      max_blocks_per_seq, num_heads, num_kv_heads, head_dim, num_blocks, scale,
                      static_cast<uint8_t *>(workspace), workspace_bytes, *d, p,
                      static_cast<cudaStream_t>(stream), block_size);
}

extern "C" int pkv_paged_attention_decode_fp8(void *out, const void *q, const void *k_cache,
                                              const void *v_cache, const int32_t *block_tables,
                                              const int32_t *context_lens, int num_seqs,
                                              int max_blocks_per_seq, int num_heads, int num_kv_heads,
                                              int head_dim, int block_size, int64_t num_blocks,
                                              float scale, float k_scale, float v_scale,
                                              void *workspace, size_t workspace_bytes, void *stream) {
    int st = check_common(num_seqs, max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, PKV_DTYPE_BF16);
    if (st != PKV_OK) return st;
    if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16))
        return PKV_ERR_INVALID_ARG;
    if (num_blocks == 0 || max_blocks_per_seq == 0) return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    st = device_info(&d);
    if (st != PKV_OK) return st;
    DecodePlan p;
    st = plan_decode(num_seqs, num_heads, num_kv_heads, head_dim, *d, &p, 1);
    if (st != PKV_OK) return st;
    return run_decode(out, q, nullptr, num_seqs, k_cache, v_cache, block_tables, context_lens, num_seqs,
                      max_blocks_per_seq, num_heads, num_kv_heads, head_dim, num_blocks, scale,
                      static_cast<uint8_t *>(workspace), workspace_bytes, *d, p,
                      static_cast<cudaStream_t>(stream), block_size, true, k_scale, v_scale);
}

// Decode with the step's KV write fused in (bf16 or FP8 cache); see pagedkv.h.
static int decode_kvwrite(void *out, const void *q, const void *k_new, const void *v_new, void *k_cache,
                          void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                          int num_seqs, int max_blocks_per_seq, int num_heads, int num_kv_heads,
                          int head_dim, int block_size, int64_t num_blocks, float scale, bool fp8,
                          float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                          void *stream) {
    int st = check_common(num_seqs, max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, PKV_DTYPE_BF16);
    if (st != PKV_OK) return st;
    if (fp8) {
        if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
        if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY)
            return PKV_ERR_INVALID_ARG;
    }
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_new || !v_new || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(k_new, 16) || !aligned(v_new, 16))
        return PKV_ERR_INVALID_ARG;
    if (num_blocks == 0 || max_blocks_per_seq == 0) return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    st = device_info(&d);
    if (st != PKV_OK) return st;
    DecodePlan p;
    st = plan_decode(num_seqs, num_heads, num_kv_heads, head_dim, *d, &p, fp8 ? 1 : 2);
    if (st != PKV_OK) return st;
    return run_decode(out, q, nullptr, num_seqs, k_cache, v_cache, block_tables, context_lens, num_seqs,
                      max_blocks_per_seq, num_heads, num_kv_heads, head_dim, num_blocks, scale,
                      static_cast<uint8_t *>(workspace), workspace_bytes, *d, p,
                      static_cast<cudaStream_t>(stream), block_size, fp8, fp8 ? k_scale : 1.f,
                      fp8 ? v_scale : 1.f, k_new, v_new);
}

extern "C" int pkv_paged_attention_decode_kvwrite(void *out, const void *q, const void *k_new,
                                                  const void *v_new, void *k_cache, void *v_cache,
                                                  const int32_t *block_tables, const int32_t *context_lens,
                                                  int num_seqs, int max_blocks_per_seq, int num_heads,
                                                  int num_kv_heads, int head_dim, int block_size,
                                                  int64_t num_blocks, float scale, int dtype,
                                                  void *workspace, size_t workspace_bytes, void *stream) {
    if (dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    return decode_kvwrite(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, num_seqs,
                          max_blocks_per_seq, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          scale, false, 1.f, 1.f, workspace, workspace_bytes, stream);
}

extern "C" int pkv_paged_attention_decode_kvwrite_fp8(void *out, const void *q, const void *k_new,
                                                      const void *v_new, void *k_cache, void *v_cache,
                                                      const int32_t *block_tables,
                                                      const int32_t *context_lens, int num_seqs,
                                                      int max_blocks_per_seq, int num_heads,
                                                      int num_kv_heads, int head_dim, int block_size,
                                                      int64_t num_blocks, float scale, float k_scale,
                                                      float v_scale, void *workspace,
                                                      size_t workspace_bytes, void *stream) {
    return decode_kvwrite(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, num_seqs,
                          max_blocks_per_seq, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          scale, true, k_scale, v_scale, workspace, workspace_bytes, stream);
}

// Varlen batch (bf16 or FP8 cache): decode rows through the decode kernel, prefill
// rows through the chunked-prefill kernel; see pagedkv.h.
static int varlen(void *out, const void *q, const int32_t *query_start_loc, const void *k_cache,
                  const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                  int num_seqs, int total_q_tokens, int max_q_len, int max_blocks_per_seq,
                  int num_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                  float scale, int causal, int dtype, bool fp8, float k_scale, float v_scale,
                  void *workspace, size_t workspace_bytes, void *stream) {
    int st = check_common(num_seqs, max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, dtype);
    if (st != PKV_OK) return st;
    if (fp8) {
        if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
        if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY)
            return PKV_ERR_INVALID_ARG;
    }
    if (total_q_tokens < 0 || max_q_len < 0) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q_tokens == 0) return PKV_OK;
    if (!out || !q || !query_start_loc || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16))
        return PKV_ERR_INVALID_ARG;
    if (num_blocks == 0 || max_blocks_per_seq == 0) return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    st = device_info(&d);
    if (st != PKV_OK) return st;
    DecodePlan p;
    st = plan_decode(num_seqs, num_heads, num_kv_heads, head_dim, *d, &p, fp8 ? 1 : 2);
    if (st != PKV_OK) return st;
    pkv::PrefillPlan pp;
    const bool prefill_rows = max_q_len >= 2;
    if (prefill_rows && block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
    if (prefill_rows) {
        st = pkv::plan_prefill(num_seqs, num_heads, num_kv_heads, head_dim, d->sms, d->smem_optin,
                               &pp, fp8);
        if (st != PKV_OK) return st;
    }
    const size_t need = round_up(p.bytes, 256) + (prefill_rows ? pp.ws_bytes : 0);
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE_TOO_SMALL;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!prefill_rows)  // single-token rows only: the decode kernel
        return run_decode(out, q, query_start_loc, total_q_tokens, k_cache, v_cache, block_tables,
                          context_lens, num_seqs, max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                          num_blocks, scale, ws, p.bytes, *d, p, s, block_size, fp8, k_scale, v_scale);
    // Decode rows and prefill chunks: one launch whose CTAs split between the two
    // (paged_varlen.cu); the decode side skips sequences with q_len != 1, the prefill
    // side those with q_len < 2.
    pkv::DecodeArgs ad;
    CUtensorMap dkmap, dvmap;
    st = prepare_decode(ad, dkmap, dvmap, out, q, query_start_loc, total_q_tokens, k_cache, v_cache,
                        block_tables, context_lens, num_seqs, max_blocks_per_seq, num_heads, num_kv_heads,
                        head_dim, num_blocks, scale, ws, p.bytes, *d, p, block_size, fp8, k_scale, v_scale,
                        nullptr, nullptr);
    if (st != PKV_OK) return st;
    CUtensorMap qmap, kmap, vmap;
    // one box per tile half
    st = encode_q_map(&qmap, q, total_q_tokens, num_heads, head_dim, pp.group, pp.tokens_per_tile / 2);
    if (st == PKV_OK)
        st = encode_cache_map(&kmap, k_cache, num_blocks, kBlockSize, num_kv_heads, head_dim, 1, fp8);
    if (st == PKV_OK)
        st = encode_cache_map(&vmap, v_cache, num_blocks, kBlockSize, num_kv_heads, head_dim, 1, fp8);
    if (st != PKV_OK) return st;
    pkv::PrefillArgs a;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.query_start_loc = query_start_loc;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.total_q = total_q_tokens;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = pp.group;
    a.tokens_per_tile = pp.tokens_per_tile;
    a.grid = pp.grid;
    a.num_stages = pp.num_stages;
    a.num_stages8 = pp.num_stages8;
    a.causal = causal != 0;
    a.num_blocks = num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);  // FP8: K = code x k_scale
    a.v_scale = fp8 ? v_scale : 1.f;
    uint8_t *pws = ws + round_up(p.bytes, 256);
    a.ws_jobs = reinterpret_cast<pkv::MergeJob *>(pws + pp.off_jobs);
    a.ws_ml = reinterpret_cast<float2 *>(pws + pp.off_ml);
    a.ws_o = reinterpret_cast<float *>(pws + pp.off_o);
    a.max_seqs = num_seqs;
    a.err = d->err;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    // unit costs for the grid split
    const float dec_unit_bytes = (float)kBlockSize * p.heads_per_cta * head_dim * (fp8 ? 1 : 2) * 2;
    const float pre_unit_flops = 4.f * head_dim * kBlockSize * pp.rows;
    pkv::VarlenSplit sp;
    sp.dec_sm_us = dec_unit_bytes / (fp8 ? kDecodeBytesPerUsSmFp8 : kDecodeBytesPerUsSm);
    sp.dec_gpu_us = dec_unit_bytes / kDecodeBytesPerUsGpu;
    sp.pre_sm_us = pre_unit_flops / kPrefillFlopPerUsSm;
    const size_t smem = p.smem > pp.smem ? p.smem : pp.smem;
    if (smem > (size_t)d->smem_optin || p.grid != pp.grid) return PKV_ERR_UNSUPPORTED;
    return pkv::launch_paged_varlen(head_dim, fp8, dkmap, dvmap, ad, qmap, kmap, vmap, a, pp, sp, smem, s) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

extern "C" int pkv_paged_attention_varlen(void *out, const void *q, const int32_t *query_start_loc,
                                          const void *k_cache, const void *v_cache,
                                          const int32_t *block_tables,
                                          const int32_t *context_lens, int num_seqs,
                                          int total_q_tokens, int max_q_len,
                                          int max_blocks_per_seq, int num_heads, int num_kv_heads,
                                          int head_dim, int block_size, int64_t num_blocks,
                                          float scale, int causal, int dtype, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    return varlen(out, q, query_start_loc, k_cache, v_cache, block_tables, context_lens, num_seqs,
                  total_q_tokens, max_q_len, max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                  block_size, num_blocks, scale, causal, dtype, false, 1.f, 1.f, workspace,
                  workspace_bytes, stream);
}

extern "C" int pkv_paged_attention_varlen_fp8(void *out, const void *q, const int32_t *query_start_loc,
                                              const void *k_cache, const void *v_cache,
                                              const int32_t *block_tables,
                                              const int32_t *context_lens, int num_seqs,
                                              int total_q_tokens, int max_q_len,
                                              int max_blocks_per_seq, int num_heads,
                                              int num_kv_heads, int head_dim, int block_size,
                                              int64_t num_blocks, float scale, int causal,
                                              float k_scale, float v_scale, void *workspace,
                                              size_t workspace_bytes, void *stream) {
    return varlen(out, q, query_start_loc, k_cache, v_cache, block_tables, context_lens, num_seqs,
                  total_q_tokens, max_q_len, max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                  block_size, num_blocks, scale, causal, PKV_DTYPE_BF16, true, k_scale, v_scale,
                  workspace, workspace_bytes, stream);
}

// ---- decode with the library's own scratch array (no workspace, no allocation) ----
//
// For callers that may not allocate device memory on the path that runs attention
// (see pkv_paged_attention_decode_static in pagedkv.h): the scratch lives in this
// fixed-size array of the library's device image instead of a caller buffer.

static __device__ __align__(256) unsigned char g_pkv_static_scratch[PKV_STATIC_SCRATCH_BYTES];

namespace {
void *g_static_scratch[kMaxDevices];

// Device address of g_pkv_static_scratch on the current device.  Host code only sees a
// host-side stand-in under the array's name, so the address has to be looked up (once
// per device, with that device current) before a kernel may be given it.
int static_scratch_address(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_static_scratch[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_static_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_static_scratch[dev] = p;
    }
    *ptr = g_static_scratch[dev];
    return PKV_OK;
}
}  // namespace

extern "C" int pkv_paged_attention_decode_static(void *out, const void *q, const void *k_cache,
                                                 const void *v_cache, const int32_t *block_tables,
                                                 const int32_t *context_lens, int num_seqs,
                                                 int max_blocks_per_seq, int num_heads,
                                                 int num_kv_heads, int head_dim, int block_size,
                                                 int64_t num_blocks, float scale, int dtype,
                                                 void *stream) {
    int st = check_common(num_seqs, max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, dtype);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16))
        return PKV_ERR_INVALID_ARG;
    if (num_blocks == 0 || max_blocks_per_seq == 0) return PKV_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    st = device_info(&d);
    if (st != PKV_OK) return st;
    DecodePlan p;
    st = plan_decode(num_seqs, num_heads, num_kv_heads, head_dim, *d, &p);
    if (st != PKV_OK) return st;
    if (p.bytes > PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_STATIC_SCRATCH_LIMIT;
    void *scratch = nullptr;
    st = static_scratch_address(&scratch);
    if (st != PKV_OK) return st;
    // Every byte the kernels read from the scratch is written earlier in the same call.
    return run_decode(out, q, nullptr, num_seqs, k_cache, v_cache, block_tables, context_lens,
                      num_seqs, max_blocks_per_seq, num_heads, num_kv_heads, head_dim, num_blocks,
                      scale, static_cast<uint8_t *>(scratch), PKV_STATIC_SCRATCH_BYTES, *d, p,
                      static_cast<cudaStream_t>(stream), block_size);
}
