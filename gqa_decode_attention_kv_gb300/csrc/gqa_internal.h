// gqa_internal.h -- declarations shared between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gqa_decode.h"

namespace gqa {

inline int dtype_bits(int dt) {
    switch (dt) {
        case GQA_DTYPE_F32: return 32;
        case GQA_DTYPE_F16: return 16;
        case GQA_DTYPE_BF16: return 16;
        case GQA_DTYPE_I8: return 8;
        case GQA_DTYPE_FP8_E4M3: return 8;
        case GQA_DTYPE_I4: return 4;
        case GQA_DTYPE_I4_KC: return 4;
        default: return 0;
    }
}
// Bytes of n elements of a cache dtype (n even for 4-bit elements).
inline long long dtype_bytes(int dt, long long n) { return n * dtype_bits(dt) / 8; }

// Code caches (8- or 4-bit codes) with fp16 scales: per (token, kv-head), or
// for the K of GQA_DTYPE_I4_KC per (block, kv-head, channel).
inline bool dtype_coded(int dt) {
    return dt == GQA_DTYPE_I8 || dt == GQA_DTYPE_FP8_E4M3 || dt == GQA_DTYPE_I4 || dt == GQA_DTYPE_I4_KC;
}

// Which split-KV kernel runs.
enum KernelKind { kKernelMma = 1, kKernelFma = 2 };

// Fixed part of the decode workspace (header ints) before the block prefix.
constexpr int kWsHeaderInts = 64;
// Upper bound on decode warps per SM used for sizing the workspace.
constexpr int kMaxWarpsPerSm = 64;
constexpr int kMaxBatch = 8191;
constexpr int kMaxGroup = 64;   // query heads per KV head the kernels serve

// token_start: NULL (every sequence appends tokens_per_seq tokens, rows
// b*T + i of k_new) or [batch+1] row offsets (sequence b appends rows
// token_start[b] .. token_start[b+1]-1, at most tokens_per_seq of them).
cudaError_t launch_kv_append(const gqa_kv_cache_t& c, const void* k_new, const void* v_new,
                             int new_dtype, const int32_t* block_tables, int max_blocks,
                             const int32_t* positions, int batch, int tokens_per_seq,
                             const int32_t* token_start, int32_t* err, cudaStream_t stream);

struct PrefillLaunch {
    const gqa_kv_cache_t* cache;
    const void* q;
    int num_heads;
    const int32_t* q_start;
    int max_new_tokens;
    const int32_t* block_tables;
    int max_blocks;
    const int32_t* context_lens;
    int batch;
    float scale;
    int window;
    void* out;
    int out_dtype;
    int kernel;                 // GQA_PREFILL_* (0 = tcgen05)
    int32_t* err;
    cudaStream_t stream;
};

// Validated launch; returns a gqa_status_t.
int launch_prefill(const PrefillLaunch& L);

struct DecodeLaunch {
    const gqa_kv_cache_t* cache;
    const void* q;
    int q_dtype;
    int num_heads;
    const int32_t* block_tables;
    int max_blocks;
    const int32_t* context_lens;
    int batch;
    float scale;
    void* out;
    int out_dtype;
    void* workspace;
    size_t workspace_bytes;
    int tokens_per_seq;         // T >= 1 queries per sequence (q, out: [B, T, H, d])
    int window;                 // sliding window in tokens, 0 = full attention
    int kernel;                 // KernelKind
    int max_warps;              // 0 = fill the GPU
    int min_blocks_per_warp;
    int row_layout;             // 0 auto, 1 virtual heads, 2 shared ring (G*T > 8)
    cudaEvent_t ev_begin, ev_end;
    int32_t* err;
    cudaStream_t stream;
};

// Resident CTAs per SM of kernel fn with `threads` threads and `smem` bytes of
// dynamic shared memory on the current device (its shared-memory limit set to
// smem on the way); asked of the runtime once per (device, kernel, size) and
// remembered. 0 if the kernel cannot launch so.
int ctas_per_sm(const void* fn, int threads, int smem);

// Bytes of workspace for a shape (T query tokens per sequence) given the
// device's SM count.
size_t decode_workspace_bytes(int batch, int num_heads, int num_kv_heads, int head_dim, int tokens_per_seq,
                              int num_sms);

// Validated launch; returns a gqa_status_t.
int launch_decode(const DecodeLaunch& L, int num_sms);

// 4-D tensor map over one cache tensor. Dim 0 is the head dimension d; dims
// 1..3 are the slot (16), kv-head (K) and block (num_blocks) axes sorted by
// increasing stride, and perm[i] names which of them (0 slot, 1 head, 2 block)
// map dim i+1 is. The box is box_inner elements by 16 slots; swizzle_bytes is
// 0 (none), 64 or 128. Returns false if the driver rejects the description.
bool encode_cache_map(CUtensorMap* map, const gqa_kv_cache_t& c, const void* base,
                      int box_inner, int swizzle_bytes, int perm[3]);

// 5-D tensor map whose box is one whole 16-token page of a 16-bit cache with
// head_dim 128, landed as [half][slot][128 B] with the 128-byte swizzle (the
// layout of two 64-element boxes of encode_cache_map); perm: dims 3 and 4 ->
// 1 kv-head, 2 block. Returns false for other caches.
bool encode_page_map(CUtensorMap* map, const gqa_kv_cache_t& c, const void* base, int perm[2]);

}  // namespace gqa
