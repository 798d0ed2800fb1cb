// gqa_capi.cu -- the extern "C" entry points of include/gqa_decode.h: argument
// validation, TMA descriptor encoding and dispatch to the kernels.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "gqa_internal.h"

namespace gqa {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count per device, asked of the runtime once per device.
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {};
std::mutex g_sms_mutex;

int num_sms_of(int device) {
    if (device < 0 && cudaGetDevice(&device) != cudaSuccess) return -1;
    if (device < kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_sms_mutex);
        if (g_sms[device] > 0) return g_sms[device];
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return -1;
    if (device < kMaxDevices && n > 0) {
        std::lock_guard<std::mutex> lock(g_sms_mutex);
        g_sms[device] = n;
    }
    return n;
}

// Checks shared by append and decode.
int check_cache(const gqa_kv_cache_t* c) {
    if (!c || !c->k || !c->v) return GQA_ERR_INVALID;
    if (c->block_size != GQA_BLOCK_SIZE) return GQA_ERR_UNSUPPORTED;
    if (c->num_blocks <= 0 || c->num_blocks > 0x7fffffffLL || c->num_kv_heads <= 0)
        return GQA_ERR_INVALID;
    if (c->head_dim != 64 && c->head_dim != 128) return GQA_ERR_UNSUPPORTED;
    const int bits = dtype_bits(c->dtype);
    if (bits == 0) return GQA_ERR_INVALID;
    if (c->stride_block <= 0 || c->stride_head <= 0 || c->stride_token < c->head_dim)
        return GQA_ERR_INVALID;
    if ((c->stride_block * bits) % 128 || (c->stride_head * bits) % 128 || (c->stride_token * bits) % 128)
        return GQA_ERR_INVALID;
    if (!aligned16(c->k) || !aligned16(c->v)) return GQA_ERR_INVALID;
    if (dtype_coded(c->dtype)) {
        if (!c->k_scale || !c->v_scale) return GQA_ERR_INVALID;
        if (!aligned16(c->k_scale) || !aligned16(c->v_scale)) return GQA_ERR_INVALID;
    }
    return GQA_OK;
}

// The appends of a GQA_DTYPE_I4_KC cache also need the residual rows.
int check_residual(const gqa_kv_cache_t* c, int batch) {
    if (c->dtype != GQA_DTYPE_I4_KC) return GQA_OK;
    if (!c->k_residual || !aligned16(c->k_residual) || c->residual_rows < batch) return GQA_ERR_INVALID;
    return GQA_OK;
}

// Tensor maps already encoded, keyed by everything an encoding reads (the
// base address, the cache's shape, strides and element type, the box and the
// swizzle): a serving loop calls with the same cache every step, and encoding
// costs more host time than the launch. A map depends only on its key, so an
// entry stays right even if the memory behind it is freed and reused.
struct MapKey {
    const void* base;
    long long num_blocks, stride_block, stride_head, stride_token;
    int num_kv_heads, head_dim, dtype, box_inner, swizzle_bytes, form;
    bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    int perm[3];
};
constexpr int kMapCacheSize = 32;
MapEntry g_maps[kMapCacheSize];
int g_maps_used = 0, g_maps_next = 0;
std::mutex g_maps_mutex;

MapKey map_key(const gqa_kv_cache_t& c, const void* base, int box_inner, int swizzle_bytes, int form) {
    MapKey k;
    std::memset(&k, 0, sizeof(k));   // padding bytes take part in the comparison
    k.base = base;
    k.num_blocks = c.num_blocks;
    k.stride_block = c.stride_block;
    k.stride_head = c.stride_head;
    k.stride_token = c.stride_token;
    k.num_kv_heads = c.num_kv_heads;
    k.head_dim = c.head_dim;
    k.dtype = c.dtype;
    k.box_inner = box_inner;
    k.swizzle_bytes = swizzle_bytes;
    k.form = form;
    return k;
}

bool cached_map(const MapKey& k, CUtensorMap* map, int* perm, int nperm) {
    std::lock_guard<std::mutex> lock(g_maps_mutex);
    for (int i = 0; i < g_maps_used; ++i) {
        if (g_maps[i].key == k) {
            *map = g_maps[i].map;
            for (int j = 0; j < nperm; ++j) perm[j] = g_maps[i].perm[j];
            return true;
        }
    }
    return false;
}

void remember_map(const MapKey& k, const CUtensorMap& map, const int* perm, int nperm) {
    std::lock_guard<std::mutex> lock(g_maps_mutex);
    MapEntry& e = g_maps[g_maps_next];
    e.key = k;
    e.map = map;
    for (int j = 0; j < 3; ++j) e.perm[j] = j < nperm ? perm[j] : 0;
    g_maps_next = (g_maps_next + 1) % kMapCacheSize;
    g_maps_used = std::max(g_maps_used, g_maps_next == 0 ? kMapCacheSize : g_maps_next);
}

bool encode_cache_map_uncached(CUtensorMap* map, const gqa_kv_cache_t& c, const void* base, int box_inner,
                               int swizzle_bytes, int perm[3]);
bool encode_page_map_uncached(CUtensorMap* map, const gqa_kv_cache_t& c, const void* base, int perm[2]);

}  // namespace

// SM count of a device (-1: the current one), remembered per device; the
// prefill sizes its persistent grid with it.
int device_sms(int device) { return num_sms_of(device); }

// 3-D tensor map over a prefill's fp32 output [tokens, num_heads, 128]: boxes of
// 16 columns x min(G, 32) heads x 32 / min(G, 32) tokens, 64-byte swizzle (one
// warp's 32 output rows, 16 columns at a time). `tokens` bounds the rows; the
// kernel stores only rows it owns.
bool encode_out_map(CUtensorMap* map, void* out, int num_heads, int G, long long tokens) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc || tokens <= 0) return false;
    const int bh = G < 32 ? G : 32;
    cuuint64_t gdim[3] = {128, (cuuint64_t)num_heads, (cuuint64_t)tokens};
    cuuint64_t gstride[2] = {128 * 4, (cuuint64_t)num_heads * 128 * 4};
    cuuint32_t box[3] = {16, (cuuint32_t)bh, (cuuint32_t)(32 / bh)};
    cuuint32_t estride[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_cache_map(CUtensorMap* map, const gqa_kv_cache_t& c, const void* base, int box_inner,
                      int swizzle_bytes, int perm[3]) {
    const MapKey k = map_key(c, base, box_inner, swizzle_bytes, 0);
    if (cached_map(k, map, perm, 3)) return true;
    if (!encode_cache_map_uncached(map, c, base, box_inner, swizzle_bytes, perm)) return false;
    remember_map(k, *map, perm, 3);
    return true;
}

bool encode_page_map(CUtensorMap* map, const gqa_kv_cache_t& c, const void* base, int perm[2]) {
    const MapKey k = map_key(c, base, 64, 128, 1);
    if (cached_map(k, map, perm, 2)) return true;
    if (!encode_page_map_uncached(map, c, base, perm)) return false;
    remember_map(k, *map, perm, 2);
    return true;
}

namespace {

bool encode_cache_map_uncached(CUtensorMap* map, const gqa_kv_cache_t& c, const void* base, int box_inner,
                               int swizzle_bytes, int perm[3]) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    CUtensorMapDataType dt;
    switch (c.dtype) {
        case GQA_DTYPE_F32: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; break;
        case GQA_DTYPE_F16: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; break;
        case GQA_DTYPE_BF16: dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; break;
        default: dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; break;   // one-byte codes
    }
    // outer axes: 0 slot, 1 kv-head, 2 block; sort by stride. A 4-bit cache is
    // described as one-byte elements (d/2 per row).
    const long long stride[3] = {c.stride_token, c.stride_head, c.stride_block};
    const long long extent[3] = {GQA_BLOCK_SIZE, c.num_kv_heads, c.num_blocks};
    int order[3] = {0, 1, 2};
    std::stable_sort(order, order + 3, [&](int x, int y) { return stride[x] < stride[y]; });
    const bool i4 = dtype_bits(c.dtype) == 4;
    cuuint64_t gdim[4] = {(cuuint64_t)(i4 ? c.head_dim / 2 : c.head_dim), 0, 0, 0};
    cuuint64_t gstride[3];
    cuuint32_t box[4] = {(cuuint32_t)box_inner, 1, 1, 1};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    for (int i = 0; i < 3; ++i) {
        perm[i] = order[i];
        gdim[i + 1] = (cuuint64_t)extent[order[i]];
        gstride[i] = (cuuint64_t)dtype_bytes(c.dtype, stride[order[i]]);
        if (order[i] == 0) box[i + 1] = GQA_BLOCK_SIZE;
    }
    const CUresult r = enc(map, dt, 4, const_cast<void*>(base), gdim, gstride, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                           : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                 : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Whole 16-token pages of 128-element 16-bit rows in one box: dims (64
// elements, 16 slots, 2 row halves, then the kv-head and block axes by
// stride), box (64, 16, 2, 1, 1), 128-byte swizzle, so that a page lands as
// [half][slot][128 B]. perm[i] names dim 3 + i: 1 kv-head, 2 block.
bool encode_page_map_uncached(CUtensorMap* map, const gqa_kv_cache_t& c, const void* base, int perm[2]) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc || c.head_dim != 128 || dtype_bits(c.dtype) != 16) return false;
    const CUtensorMapDataType dt =
        c.dtype == GQA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const long long stride[2] = {c.stride_head, c.stride_block};
    const long long extent[2] = {c.num_kv_heads, c.num_blocks};
    const int o0 = stride[0] <= stride[1] ? 0 : 1, o1 = 1 - o0;
    cuuint64_t gdim[5] = {64, GQA_BLOCK_SIZE, 2, (cuuint64_t)extent[o0], (cuuint64_t)extent[o1]};
    cuuint64_t gstride[4] = {(cuuint64_t)dtype_bytes(c.dtype, c.stride_token), 128,
                             (cuuint64_t)dtype_bytes(c.dtype, stride[o0]),
                             (cuuint64_t)dtype_bytes(c.dtype, stride[o1])};
    cuuint32_t box[5] = {64, GQA_BLOCK_SIZE, 2, 1, 1};
    cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    perm[0] = o0 + 1;
    perm[1] = o1 + 1;
    const CUresult r = enc(map, dt, 5, const_cast<void*>(base), gdim, gstride, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

}  // namespace gqa

using namespace gqa;

extern "C" {

const char* gqa_status_string(int status) {
    switch (status) {
        case GQA_OK: return "ok";
        case GQA_ERR_INVALID: return "invalid argument";
        case GQA_ERR_UNSUPPORTED: return "unsupported configuration";
        case GQA_ERR_WORKSPACE: return "workspace missing or too small";
        case GQA_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int gqa_version(void) { return 300; }

int64_t gqa_kv_pool_elements(int64_t num_blocks, int32_t num_kv_heads, int32_t head_dim) {
    if (num_blocks < 0 || num_kv_heads < 0 || head_dim < 0) return -1;
    return 2 * num_blocks * (int64_t)num_kv_heads * GQA_BLOCK_SIZE * (int64_t)head_dim;
}

int gqa_kv_append(const gqa_kv_cache_t* cache, const void* k_new, const void* v_new,
                  int32_t new_dtype, const int32_t* block_tables, int32_t max_blocks_per_seq,
                  const int32_t* positions, int32_t batch, int32_t tokens_per_seq, int32_t* err_flag,
                  void* stream) {
    int st = check_cache(cache);
    if (st != GQA_OK) return st;
    if (batch < 0 || max_blocks_per_seq <= 0 || tokens_per_seq < 0) return GQA_ERR_INVALID;
    const int T = std::max(1, (int)tokens_per_seq);
    if ((long long)batch * T * cache->num_kv_heads >= 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;
    if (batch == 0) return GQA_OK;
    if (!k_new || !v_new || !block_tables || !positions) return GQA_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new)) return GQA_ERR_INVALID;
    if ((long long)max_blocks_per_seq * GQA_BLOCK_SIZE > 0x7fffffffLL) return GQA_ERR_INVALID;
    if (dtype_coded(cache->dtype)) {
        if (new_dtype != GQA_DTYPE_F32 && new_dtype != GQA_DTYPE_F16 && new_dtype != GQA_DTYPE_BF16)
            return GQA_ERR_UNSUPPORTED;
    } else if (new_dtype != cache->dtype) {
        return GQA_ERR_UNSUPPORTED;
    }
    if ((st = check_residual(cache, batch)) != GQA_OK) return st;
    const cudaError_t e = launch_kv_append(*cache, k_new, v_new, new_dtype, block_tables,
                                           max_blocks_per_seq, positions, batch, T, nullptr, err_flag,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

int gqa_kv_append_varlen(const gqa_kv_cache_t* cache, const void* k_new, const void* v_new,
                         int32_t new_dtype, const int32_t* token_start, int32_t max_new_tokens,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* positions, int32_t batch, int32_t* err_flag, void* stream) {
    int st = check_cache(cache);
    if (st != GQA_OK) return st;
    if (batch < 0 || max_blocks_per_seq <= 0 || max_new_tokens < 0) return GQA_ERR_INVALID;
    if ((long long)batch * max_new_tokens * cache->num_kv_heads >= 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;
    if (batch == 0 || max_new_tokens == 0) return GQA_OK;
    if (!k_new || !v_new || !token_start || !block_tables || !positions) return GQA_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new)) return GQA_ERR_INVALID;
    if ((long long)max_blocks_per_seq * GQA_BLOCK_SIZE > 0x7fffffffLL) return GQA_ERR_INVALID;
    if (dtype_coded(cache->dtype)) {
        if (new_dtype != GQA_DTYPE_F32 && new_dtype != GQA_DTYPE_F16 && new_dtype != GQA_DTYPE_BF16)
            return GQA_ERR_UNSUPPORTED;
    } else if (new_dtype != cache->dtype) {
        return GQA_ERR_UNSUPPORTED;
    }
    if ((st = check_residual(cache, batch)) != GQA_OK) return st;
    const cudaError_t e = launch_kv_append(*cache, k_new, v_new, new_dtype, block_tables,
                                           max_blocks_per_seq, positions, batch, max_new_tokens,
                                           token_start, err_flag, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

int gqa_prefill(const gqa_kv_cache_t* cache, const void* q, int32_t q_dtype, int32_t num_heads,
                const int32_t* q_start, int32_t max_new_tokens, const int32_t* block_tables,
                int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch, float scale,
                int32_t sliding_window, void* out, int32_t out_dtype, int32_t kernel, int32_t* err_flag,
                void* stream) {
    int st = check_cache(cache);
    if (kernel < 0 || kernel > GQA_PREFILL_TCGEN05_PAIRED) return GQA_ERR_INVALID;
    if (st != GQA_OK) return st;
    if (batch < 0 || num_heads <= 0 || max_blocks_per_seq <= 0 || max_new_tokens < 0 || sliding_window < 0)
        return GQA_ERR_INVALID;
    if (num_heads % cache->num_kv_heads) return GQA_ERR_INVALID;
    if (cache->dtype != GQA_DTYPE_BF16 && cache->dtype != GQA_DTYPE_F16) return GQA_ERR_UNSUPPORTED;
    if (q_dtype != cache->dtype) return GQA_ERR_UNSUPPORTED;
    if (out_dtype != GQA_DTYPE_F32 && out_dtype != GQA_DTYPE_BF16 && out_dtype != GQA_DTYPE_F16)
        return GQA_ERR_UNSUPPORTED;
    if (batch > 65535 || cache->num_kv_heads > 65535) return GQA_ERR_UNSUPPORTED;   // grid y, z
    if (!std::isfinite(scale)) return GQA_ERR_INVALID;
    if (batch == 0 || max_new_tokens == 0) return GQA_OK;
    if (!q || !q_start || !block_tables || !context_lens || !out) return GQA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(out)) return GQA_ERR_INVALID;
    PrefillLaunch L;
    L.cache = cache;
    L.q = q;
    L.num_heads = num_heads;
    L.q_start = q_start;
    L.max_new_tokens = max_new_tokens;
    L.block_tables = block_tables;
    L.max_blocks = max_blocks_per_seq;
    L.context_lens = context_lens;
    L.batch = batch;
    L.scale = scale;
    L.window = sliding_window;
    L.out = out;
    L.out_dtype = out_dtype;
    L.kernel = kernel;
    L.err = err_flag;
    L.stream = static_cast<cudaStream_t>(stream);
    return launch_prefill(L);
}

size_t gqa_decode_workspace_size(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t tokens_per_seq, int32_t device) {
    if (batch < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    if (tokens_per_seq < 0 || tokens_per_seq > kMaxGroup) return 0;
    const int sms = num_sms_of(device);
    if (sms <= 0) return 0;
    return decode_workspace_bytes(batch, num_heads, num_kv_heads, head_dim, tokens_per_seq, sms);
}

int gqa_decode(const gqa_kv_cache_t* cache, const void* q, int32_t q_dtype, int32_t num_heads,
               const int32_t* block_tables, int32_t max_blocks_per_seq,
               const int32_t* context_lens, int32_t batch, float scale, void* out,
               int32_t out_dtype, void* workspace, size_t workspace_bytes,
               const gqa_decode_opts_t* opts, int32_t* err_flag, void* stream) {
    int st = check_cache(cache);
    if (st != GQA_OK) return st;
    if (batch < 0 || num_heads <= 0 || max_blocks_per_seq <= 0) return GQA_ERR_INVALID;
    if (num_heads % cache->num_kv_heads) return GQA_ERR_INVALID;
    const int T = opts ? opts->tokens_per_seq : 0;
    const int window = opts ? opts->sliding_window : 0;
    if (T < 0 || window < 0) return GQA_ERR_INVALID;
    if ((long long)(num_heads / cache->num_kv_heads) * std::max(1, T) > kMaxGroup) return GQA_ERR_UNSUPPORTED;
    if ((long long)batch * std::max(1, T) * num_heads >= 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;
    if (batch > kMaxBatch) return GQA_ERR_UNSUPPORTED;
    if ((long long)batch * cache->num_kv_heads * max_blocks_per_seq >= 0x7fffffffLL)
        return GQA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return GQA_ERR_INVALID;
    if (batch == 0) return GQA_OK;
    if (!q || !block_tables || !context_lens || !out) return GQA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(out)) return GQA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GQA_ERR_INVALID;
    if (out_dtype != GQA_DTYPE_F32 && out_dtype != GQA_DTYPE_BF16 && out_dtype != GQA_DTYPE_F16)
        return GQA_ERR_UNSUPPORTED;
    const int cd = cache->dtype;
    const bool q_ok = dtype_coded(cd) ? (q_dtype == GQA_DTYPE_BF16 || q_dtype == GQA_DTYPE_F16)
                                           : (q_dtype == cd);
    if (!q_ok) return GQA_ERR_UNSUPPORTED;
    int kernel = opts ? opts->kernel : 0;
    if (kernel < 0 || kernel > 2) return GQA_ERR_INVALID;
    if (opts && (opts->row_layout < 0 || opts->row_layout > 2)) return GQA_ERR_INVALID;
    const int sms = num_sms_of(-1);
    if (sms <= 0) return GQA_ERR_CUDA;

    DecodeLaunch L;
    L.cache = cache;
    L.q = q;
    L.q_dtype = q_dtype;
    L.num_heads = num_heads;
    L.block_tables = block_tables;
    L.max_blocks = max_blocks_per_seq;
    L.context_lens = context_lens;
    L.batch = batch;
    L.scale = scale;
    L.out = out;
    L.out_dtype = out_dtype;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.tokens_per_seq = std::max(1, T);
    L.window = window;
    L.kernel = kernel;
    L.max_warps = opts ? std::max(0, opts->max_warps) : 0;
    L.min_blocks_per_warp = opts ? std::max(0, opts->min_blocks_per_warp) : 0;
    L.row_layout = opts ? opts->row_layout : 0;
    L.ev_begin = opts ? static_cast<cudaEvent_t>(opts->event_main_begin) : nullptr;
    L.ev_end = opts ? static_cast<cudaEvent_t>(opts->event_main_end) : nullptr;
    L.err = err_flag;
    L.stream = static_cast<cudaStream_t>(stream);
    return launch_decode(L, sms);
}

}  // extern "C"
