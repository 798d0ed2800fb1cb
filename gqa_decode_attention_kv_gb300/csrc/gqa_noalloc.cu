// gqa_noalloc.cu -- gqa_decode for callers that cannot allocate device memory:
// the split-KV scratch lives in a fixed array compiled into the library.
#include <mutex>

#include "gqa_internal.h"

namespace {

// The scratch every gqa_decode_noalloc call uses (held by each GPU that loads
// the library until exit). 256-byte aligned, as gqa_decode requires.
static __device__ __align__(256) uint8_t g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" GQA_API int gqa_decode_noalloc(const gqa_kv_cache_t* cache, const void* q,
                                          int32_t q_dtype, int32_t num_heads,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t batch, float scale,
                                          void* out, int32_t out_dtype,
                                          const gqa_decode_opts_t* opts, int32_t* err_flag,
                                          void* stream) {
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return GQA_ERR_CUDA;
    return gqa_decode(cache, q, q_dtype, num_heads, block_tables, max_blocks_per_seq, context_lens,
                      batch, scale, out, out_dtype, scratch, GQA_NOALLOC_SCRATCH_BYTES, opts,
                      err_flag, stream);
}
