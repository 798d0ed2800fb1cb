/*
 * gqa_decode.h -- C ABI of the GB300 (sm_103a) grouped-query decode-attention
 * library over a paged KV cache.
 *
 * One autoregressive decode step of grouped-query attention: each of the H
 * query heads of the new token attends to the shared K/V head of its group,
 * g = h / (H/K), over the whole cached context ("分组查询注意力 (GQA)",
 * 技术原理 steps 1-4 and the attention equation
 * softmax(Q_group K_g^T / sqrt(d_k)) V_g). The cache is paged: fixed blocks of
 * 16 tokens, addressed per sequence through a block table
 * ("LLM 推理性能优化实战", section 8.2; block_size 16 from the KV-cache essay's
 * padding paragraph).
 *
 * Conventions for every call:
 *  - Pointers named "device" are CUDA device pointers owned by the caller; the
 *    library never frees or keeps them. Structs passed by pointer are host
 *    memory and are read during the call only.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). All GPU work
 *    is enqueued on it; no call synchronises the host with the device, and no
 *    call allocates device memory.
 *  - Host-detectable argument errors return a non-zero gqa_status_t before any
 *    launch. Data-dependent faults found on the device (a block-table entry
 *    outside [0, num_blocks), a context length outside [0, max_blocks*16], an
 *    append position out of range) never trap: the offending unit is skipped
 *    and a GQA_DEVERR_* bit is OR-ed into *err_flag (a device int32, may be
 *    NULL). Outputs of a sequence that raised a device error are unspecified.
 *  - Tensor layouts are row-major with the innermost index last.
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GQA_API __attribute__((visibility("default")))
#else
#define GQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
typedef enum {
    GQA_DTYPE_F32 = 0,
    GQA_DTYPE_F16 = 1,
    GQA_DTYPE_BF16 = 2,
    GQA_DTYPE_I8 = 3,         /* cache only: int8 codes + one fp16 scale per (token, kv-head) */
    GQA_DTYPE_FP8_E4M3 = 4,   /* cache only: e4m3 codes (max 448) + one fp16 scale per (token, kv-head) */
    GQA_DTYPE_I4 = 5,         /* cache only: 4-bit codes in [-7, 7], two per byte + one fp16 scale
                                 per (token, kv-head) */
    GQA_DTYPE_I4_KC = 6       /* cache only: 4-bit codes as GQA_DTYPE_I4; K with one fp16 scale per
                                 (block, kv-head, channel), V with one per (token, kv-head) */
} gqa_dtype_t;

/* Return codes. */
typedef enum {
    GQA_OK = 0,
    GQA_ERR_INVALID = 1,      /* null pointer, bad size or stride, misaligned address */
    GQA_ERR_UNSUPPORTED = 2,  /* well-formed but not built: head_dim, group size, dtype mix */
    GQA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than gqa_decode_workspace_size */
    GQA_ERR_CUDA = 4          /* a CUDA runtime call or a kernel launch failed */
} gqa_status_t;

/* Device-side error bits OR-ed into *err_flag. */
#define GQA_DEVERR_BLOCK_INDEX 1   /* block-table entry outside [0, num_blocks) */
#define GQA_DEVERR_CONTEXT_LEN 2   /* context length < 0 or > max_blocks_per_seq * 16 */
#define GQA_DEVERR_POSITION    4   /* append position < 0 or >= max_blocks_per_seq * 16 */
#define GQA_DEVERR_TIMEOUT     8   /* a bounded wait for an asynchronous copy expired */

#define GQA_BLOCK_SIZE 16

/*
 * A paged KV cache. Token t (slot t % 16) of kv-head g in physical block p
 * starts at element  p*stride_block + g*stride_head + (t % 16)*stride_token
 * of `k` (and of `v`). The default pool layout [num_blocks, K, 16, d] has
 * stride_block = K*16*d, stride_head = 16*d, stride_token = d (one 16 x d tile
 * per (block, kv-head), contiguous). A contiguous un-paged cache
 * [B, S_pad, K, d] is the same thing with stride_block = 16*K*d,
 * stride_head = d, stride_token = K*d and the identity block table
 * table[b][j] = b*(S_pad/16) + j.
 *
 * For the coded caches (GQA_DTYPE_I8, GQA_DTYPE_FP8_E4M3, GQA_DTYPE_I4),
 * k_scale / v_scale hold one fp16 scale per (block, kv-head, slot) as
 * [num_blocks, K, 16]; the cached value is code * scale (an int8 or int4
 * code, or the value of an e4m3 code). Other dtypes leave them NULL. An I4
 * element is half a byte: elements 2j and 2j+1 of a row share byte j, 2j in
 * the low nibble, each a two's-complement 4-bit code; strides still count
 * elements (byte offset = element offset / 2).
 *
 * GQA_DTYPE_I4_KC is the KIVI-style cache ("LLM 推理性能优化实战" section 15.5:
 * K quantised per channel, V per token, both to INT4). V is stored as for
 * GQA_DTYPE_I4. K keeps one fp16 scale per channel for each (block, kv-head):
 * k_scale is [num_blocks, K, head_dim], and the cached K of slot t, channel i
 * is code[t][i] * k_scale[p][g][i]. The scales of a block cover the tokens it
 * holds: the append re-quantises a block, per channel, over all its tokens
 * each time tokens join it (symmetric: s_i = fp16(max_t |k[t][i]| / 7),
 * code = clamp(rint(k / s_i), -7, 7)). To do so without compounding rounding
 * it keeps the unquantised K of every sequence's unfinished block in
 * k_residual: fp32 [residual_rows, K, 16, head_dim], row b serving the
 * sequence an append call passes as batch row b (a caller that moves a
 * sequence to another row moves its residual row with it). Only the appends
 * read or write k_residual; decode reads codes and scales alone.
 *
 * Requirements: block_size == 16; head_dim in {64, 128}; k, v, k_scale,
 * v_scale 16-byte aligned; every stride times the element size a multiple of
 * 16 bytes; stride_token >= head_dim.
 */
typedef struct {
    void   *k;                /* device */
    void   *v;                /* device */
    void   *k_scale;          /* device, fp16 [num_blocks, K, 16], coded caches only */
    void   *v_scale;          /* device, fp16 [num_blocks, K, 16], coded caches only */
    int64_t num_blocks;
    int32_t num_kv_heads;     /* K */
    int32_t block_size;       /* must be 16 */
    int32_t head_dim;         /* d */
    int32_t dtype;            /* gqa_dtype_t */
    int64_t stride_block;     /* elements */
    int64_t stride_head;      /* elements */
    int64_t stride_token;     /* elements */
    void   *k_residual;       /* device, fp32 [residual_rows, K, 16, d], GQA_DTYPE_I4_KC only */
    int32_t residual_rows;    /* rows of k_residual (>= the batch of every append) */
    int32_t reserved;         /* zero */
} gqa_kv_cache_t;

/*
 * Options of gqa_decode. NULL, or a zero-filled struct, gives the plain decode
 * step: one new token per sequence, full attention, automatic kernel choice.
 *  tokens_per_seq  T >= 1 new tokens (queries) per sequence, causal among
 *                  themselves (speculative verification, "LLM 推理性能优化实战"
 *                  section 14.2; chunked prefill next to decode, section 11.7).
 *                  0 means 1. q and out become [batch, T, num_heads, head_dim].
 *  sliding_window  W > 0: every query attends only the last W positions up to
 *                  and including its own (sliding-window attention, section
 *                  6.4.1); 0 = full attention. Blocks wholly before a query's
 *                  window are never read, so their table entries may hold
 *                  anything (a caller may recycle those blocks).
 */
typedef struct {
    int32_t tokens_per_seq;       /* 0 or 1: one new token per sequence */
    int32_t sliding_window;       /* 0: full attention */
    int32_t kernel;               /* 0 auto, 1 tensor-core (mma.sync) kernel, 2 CUDA-core kernel */
    int32_t max_warps;            /* 0 = fill the GPU; > 0 caps the split-KV workers, i.e. KV splits */
    int32_t min_blocks_per_warp;  /* 0 = default (4): smallest KV range one warp takes */
    int32_t row_layout;           /* more than 8 query rows per kv-head (G*T > 8): 0 auto
                                     (2 where that kernel exists, else 1), 1 every 8 rows
                                     stream the tiles on their own (the re-reads hit L2),
                                     2 the warps of a CTA share each tile */
    void   *event_main_begin;     /* optional cudaEvent_t recorded just before the split-KV kernel */
    void   *event_main_end;       /* optional cudaEvent_t recorded just after it */
} gqa_decode_opts_t;

/* Human-readable name of a gqa_status_t. Never NULL. */
GQA_API const char *gqa_status_string(int status);

/* Library ABI version (major*10000 + minor*100 + patch). */
GQA_API int gqa_version(void);

/*
 * Elements of K and V together that a pool of num_blocks 16-token blocks holds:
 * 2 * num_blocks * num_kv_heads * 16 * head_dim. The closed form of
 * "分组查询注意力 (GQA)", 关键参数 item 2 (2*K*d_k per token per layer) and
 * "LLM 推理性能优化实战", section 6.1, sized by the allocator. Returns -1 on a
 * negative argument. Host only; needs no GPU.
 */
GQA_API int64_t gqa_kv_pool_elements(int64_t num_blocks, int32_t num_kv_heads, int32_t head_dim);

/*
 * Paged KV append: write the T new tokens of every sequence into the cache.
 * For each b < batch, i < T and kv-head g < K, with pos = positions[b] + i:
 *   block = block_tables[b*max_blocks_per_seq + pos/16], slot = pos % 16,
 *   K[block, g, slot, :] = k_new[b, i, g, :],  V[...] = v_new[b, i, g, :].
 * (The write of one token's K and V per step, "LLM 推理性能优化实战" sections
 * 5.3-5.4; the block table of section 8.2.)
 *
 *  k_new, v_new   device, [batch, T, K, head_dim] of new_dtype, 16-byte aligned.
 *                 For F32/F16/BF16 caches new_dtype must equal the cache dtype
 *                 and the copy is bit-exact. For an I8 cache new_dtype is F32,
 *                 F16 or BF16 and each (token, kv-head) row is quantised on the
 *                 device: amax = max|x| (fp32); s = fp16_rne(min(amax/127, 65504));
 *                 code = s == 0 ? 0 : clamp(rint(x/s), -127, 127) with IEEE fp32
 *                 division (symmetric int8, "LLM 推理性能优化实战" sections 15.1,
 *                 15.2, 15.5). For an I4 cache likewise with
 *                 s = fp16_rne(min(amax/7, 65504)), code = clamp(rint(x/s), -7, 7)
 *                 (the INT4 KV option of section 15.5), two codes per byte.
 *                 For an FP8_E4M3 cache likewise with
 *                 s = fp16_rne(min(amax/448, 65504)) and code = e4m3 of x/s,
 *                 rounded to nearest even and saturated to +-448 (the FP8 option
 *                 of section 15.5). The scale goes to k_scale / v_scale.
 *                 For an I4_KC cache V is quantised as for I4, and every block
 *                 the new tokens reach is re-quantised per channel over all
 *                 the tokens it then holds (codes of its older slots included),
 *                 the older tokens' K read from k_residual row b; the new
 *                 tokens' K of a block left unfinished is kept there.
 *                 k_residual must be non-NULL, 16-byte aligned, with
 *                 residual_rows >= batch; sequences of one call must not
 *                 share a block.
 *  block_tables   device int32 [batch, max_blocks_per_seq].
 *  positions      device int32 [batch]: position of the first new token, i.e.
 *                 the context length BEFORE the append. Not modified; the
 *                 caller advances its context lengths by T.
 *  tokens_per_seq T >= 1 (0 means 1).
 *  err_flag       device int32 or NULL (GQA_DEVERR_POSITION / _BLOCK_INDEX).
 *                 A token whose position or block is out of range is skipped
 *                 (for an I4_KC cache: an out-of-range position skips the
 *                 sequence's whole append, an out-of-range block that block).
 */
GQA_API int gqa_kv_append(const gqa_kv_cache_t *cache, const void *k_new, const void *v_new,
                  int32_t new_dtype, const int32_t *block_tables,
                  int32_t max_blocks_per_seq, const int32_t *positions, int32_t batch,
                  int32_t tokens_per_seq, int32_t *err_flag, void *stream);

/*
 * Paged KV append with a different number of new tokens per sequence (a batch
 * of prompts, or chunks of them): sequence b writes rows token_start[b] ..
 * token_start[b+1]-1 of k_new / v_new ([total, K, head_dim], 16-byte aligned)
 * at positions positions[b], positions[b]+1, ... Quantisation and exactness as
 * gqa_kv_append ("LLM 推理性能优化实战" section 5.3.1: prefill writes every new
 * token's K and V at increasing positions).
 *  token_start    device int32 [batch+1], non-decreasing.
 *  max_new_tokens host bound on token_start[b+1] - token_start[b]; a sequence
 *                 with more (or a negative count) is skipped and flagged
 *                 (GQA_DEVERR_POSITION).
 */
GQA_API int gqa_kv_append_varlen(const gqa_kv_cache_t *cache, const void *k_new, const void *v_new,
                  int32_t new_dtype, const int32_t *token_start, int32_t max_new_tokens,
                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                  const int32_t *positions, int32_t batch, int32_t *err_flag, void *stream);

/*
 * Paged prefill attention: the n_b = q_start[b+1] - q_start[b] new tokens of
 * sequence b, at positions context_lens[b] - n_b .. context_lens[b] - 1, each
 * attend causally to the sequence's cache (their own K/V already appended, e.g.
 * by gqa_kv_append_varlen) -- the same per-query definition as gqa_decode with
 * T = n_b, for prompts of any length ("LLM 推理性能优化实战" sections 9.2-9.4:
 * FlashAttention's tiled Q x KV with the online softmax, reading the paged cache
 * block by block). With sliding_window W > 0 each query attends only its last W
 * positions. No workspace: every (query tile, kv-head, sequence) is one CTA.
 *
 *  q              device [total new tokens, num_heads, head_dim], rows of
 *                 sequence b from q_start[b]; the cache dtype (BF16 or F16 caches).
 *  q_start        device int32 [batch+1], non-decreasing.
 *  max_new_tokens host bound on every n_b (sizes the grid); a sequence with a
 *                 larger or negative n_b, or context_lens[b] < n_b, or
 *                 context_lens[b] > max_blocks_per_seq*16, is skipped and flagged
 *                 (GQA_DEVERR_CONTEXT_LEN); its output rows are not written.
 *  out            device [total new tokens, num_heads, head_dim] of out_dtype.
 *  kernel         GQA_PREFILL_AUTO: GQA_PREFILL_TCGEN05_WIDE for head_dim 128,
 *                 else GQA_PREFILL_TCGEN05. GQA_PREFILL_TCGEN05_WIDE (head_dim
 *                 128 only): one CTA per SM, two 128-row query tiles sharing
 *                 64-token K/V chunks on the 5th-generation tensor cores, all
 *                 512 tensor-memory columns. GQA_PREFILL_TCGEN05_PAIRED (head_dim
 *                 128 only): the same with one query tile per CTA and two CTAs
 *                 per SM. GQA_PREFILL_TCGEN05: 128-row query tiles, 32-token
 *                 chunks, two CTAs per SM. GQA_PREFILL_MMA_SYNC: 64-row tiles on
 *                 warp-level mma.sync. The forms other than AUTO's choice are the
 *                 measured alternatives.
 *  Limits: BF16/F16 caches; head_dim 64 or 128; batch and K <= 65535.
 */
#define GQA_PREFILL_AUTO 0
#define GQA_PREFILL_TCGEN05 1
#define GQA_PREFILL_MMA_SYNC 2
#define GQA_PREFILL_TCGEN05_WIDE 3
#define GQA_PREFILL_TCGEN05_PAIRED 4
GQA_API int gqa_prefill(const gqa_kv_cache_t *cache, const void *q, int32_t q_dtype, int32_t num_heads,
                const int32_t *q_start, int32_t max_new_tokens, const int32_t *block_tables,
                int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch, float scale,
                int32_t sliding_window, void *out, int32_t out_dtype, int32_t kernel, int32_t *err_flag,
                void *stream);

/*
 * Bytes of device workspace gqa_decode needs for this shape (tokens_per_seq as
 * in gqa_decode_opts_t, 0 meaning 1) on `device` (-1 = the current device).
 * Returns 0 on bad arguments. The bound covers every kernel choice, window and
 * context-length mix of this shape.
 */
GQA_API size_t gqa_decode_workspace_size(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t tokens_per_seq, int32_t device);

/*
 * Grouped-query decode attention over the paged cache:
 *   out[b, h, :] = sum_t softmax_t(scale * q[b,h,:] . K[b, t, g]) V[b, t, g],
 *   g = h / (num_heads / K), t in [0, context_lens[b]),
 * where K[b, t, g] is read through block_tables as in gqa_kv_append. With
 * T = opts->tokens_per_seq > 1 the queries q[b, i] (i < T) sit at positions
 * context_lens[b] - T + i and query i attends t <= context_lens[b] - T + i
 * (a query at a negative position gets a zero row); with W =
 * opts->sliding_window > 0 only t > (its position) - W.
 * The KV range of each (sequence, kv-head) is split across warps
 * (split-KV flash decoding, "LLM 推理性能优化实战" section 10.2); each split
 * keeps a running (max, sum, weighted V) state (online softmax, section 9.2)
 * and a second kernel merges the splits with their log-sum-exp weights
 * ("global max and sum" reduction of section 10.2). An empty context
 * (length 0) yields a zero output row.
 *
 *  q              device [batch, T, num_heads, head_dim]; BF16 for a BF16 cache,
 *                 F16 for F16, F32 for F32, BF16 or F16 for a coded cache.
 *  block_tables   device int32 [batch, max_blocks_per_seq].
 *  context_lens   device int32 [batch], lengths AFTER the append (the T new
 *                 tokens included), each in [0, max_blocks_per_seq*16].
 *  scale          softmax scale (1/sqrt(head_dim) for standard attention).
 *  out            device [batch, T, num_heads, head_dim] of out_dtype (F32,
 *                 BF16 or F16); 16-byte aligned.
 *  workspace      device, >= gqa_decode_workspace_size(...) bytes, 256-byte
 *                 aligned, zero-filled before its first use (one word of it, the
 *                 run-time work counter, must start at zero; every call leaves it
 *                 at zero again, a call failing with GQA_ERR_CUDA after its first
 *                 kernel was queued by a reset queued on the stream). Otherwise
 *                 clobbered by each call. Calls that
 *                 share a workspace must not overlap on the GPU.
 *  opts           NULL or options (gqa_decode_opts_t).
 *  Limits: num_heads % K == 0; T * num_heads / K <= 64 query rows per kv-head;
 *  sliding_window >= 0; batch <= 8191; batch * K * max_blocks_per_seq < 2^31
 *  (above 8 rows per kv-head on a kernel without a shared-ring form, times the
 *  number of 8-row groups).
 */
GQA_API int gqa_decode(const gqa_kv_cache_t *cache, const void *q, int32_t q_dtype,
               int32_t num_heads, const int32_t *block_tables, int32_t max_blocks_per_seq,
               const int32_t *context_lens, int32_t batch, float scale, void *out,
               int32_t out_dtype, void *workspace, size_t workspace_bytes,
               const gqa_decode_opts_t *opts, int32_t *err_flag, void *stream);

/*
 * gqa_decode without a caller-supplied workspace. The pages have no
 * counterpart for this call; it exists for callers that cannot allocate device
 * memory: a plugin running inside a host engine whose device allocator it does
 * not own, or a runtime that plans every device byte before serving starts and
 * forbids allocation in the decode loop. Such callers can still pass their
 * inputs and outputs, but have nowhere to put the split-KV partial results.
 *
 * The scratch lives in one fixed array of GQA_NOALLOC_SCRATCH_BYTES compiled
 * into the library; every GPU that loads the library holds it until the
 * process exits. Arguments and results are those of gqa_decode minus the
 * workspace. This call allocates nothing (no cudaMalloc, no library allocator).
 *  - Returns GQA_ERR_WORKSPACE when the shape needs more scratch than the array
 *    holds (the five workloads of the benchmark need under 48 MiB).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture on the device.
 *  - Every call shares the one array and it keeps the last call's contents.
 *    The one word that must start at zero does: the array is zero when the
 *    library loads and every call leaves that word at zero (a call that fails
 *    with GQA_ERR_CUDA after its first kernel was queued also queues a reset
 *    of that word on the stream). Calls whose GPU
 *    work overlaps -- different streams, or different host threads -- race on
 *    it; serialise them.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

GQA_API int gqa_decode_noalloc(const gqa_kv_cache_t *cache, const void *q, int32_t q_dtype,
                               int32_t num_heads, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens,
                               int32_t batch, float scale, void *out, int32_t out_dtype,
                               const gqa_decode_opts_t *opts, int32_t *err_flag, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H */
