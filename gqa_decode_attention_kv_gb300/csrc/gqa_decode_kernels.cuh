// gqa_decode_kernels.cuh -- the split-KV decode kernel and the combine kernel
// as templates, with the host-side variant table. Included by gqa_decode.cu
// (the one-token, full-attention flavour and the combine kernels) and by
// gqa_decode_general.cu (the flavour for several queries per sequence or a
// sliding window), so the two sets of instantiations compile in parallel.
//
// Split-KV grouped-query decode attention over a paged cache.
//
// What is computed (per sequence b, query head h, group g = h / G, G = H/K):
//   out[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . K[b,t,g,:]) V[b,t,g,:]
// ("分组查询注意力 (GQA)", 技术原理 steps 2-4 and its attention equation).
// With T new tokens per sequence (speculative verification / chunked prefill,
// "LLM 推理性能优化实战" sections 14.2 and 11.7) query i of sequence b sits at
// position L_b - T + i and attends positions up to its own; with a sliding
// window W (section 6.4.1) only the last W of those. Every (sequence, kv-head)
// pair then serves G*T query rows (row = i*G + head-in-group), all reading the
// same K/V tiles: T widens the MMA N dimension exactly like a larger group.
//
// How (GB300 design):
//  * Work unit = one 16-token cache block of one (sequence, kv-head) pair. All
//    units are laid out in (b, g, block) order and cut into equal contiguous
//    ranges, one per warp of a single resident wave (persistent, stream-K
//    style). A pair that straddles ranges becomes several KV splits
//    (Flash-Decoding, "LLM 推理性能优化实战" section 10.2); the cut is found on
//    the device from context_lens, so no host synchronisation is needed.
//  * Each warp streams its blocks through a private ring of shared-memory
//    stages filled by TMA (cp.async.bulk.tensor, 4-D tensor map over the
//    paged pool, mbarrier completion). The block table is consulted per unit;
//    each K/V tile is read from HBM exactly once and serves all G query heads
//    of its group (the group broadcast of the GQA page's 下游 section).
//  * Tensor-core kernel: scores S^T[16 tokens x 8 heads] = K_tile Q^T and the
//    update O^T[d x 8 heads] += V_tile^T P^T with mma.sync m16n8k16 (bf16 or
//    f16 in, fp32 accumulate). P is split into a high and a low 16-bit part
//    so the product keeps ~16 significant bits. Online softmax in fp32 with
//    the running (m, l, o) state of "LLM 推理性能优化实战" section 9.2; the
//    rescale is skipped while the block maximum stays within 2^kRescaleSlack
//    of the running one (o and l share the stale maximum, so o/l is exact).
//  * CUDA-core kernel: same pipeline, one token at a time with fp32 FMAs and
//    warp-shuffle reductions; used for fp32 caches and as the measured
//    alternative to the tensor-core kernel.
//  * A second kernel merges the splits of each pair with their log-sum-exp
//    weights: M = max m_s, L = sum l_s 2^(m_s-M), o = sum o_s 2^(m_s-M) / L
//    (the "global max and sum" reduction of section 10.2), in base 2.
#pragma once

#include <algorithm>
#include <type_traits>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {
namespace dec {

constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
    const void* q;
    const __half* k_scale;
    const __half* v_scale;
    const int32_t* block_tables;
    const int32_t* context_lens;
    void* out;
    int32_t* err;
    int32_t* ws_hdr;     // the Partition: [0] R, [1] U, [2] Rs, [3] Cz, [4] P, [5] cpw
    unsigned long long* ws_ctr;   // next dynamic chunk; zero between calls
    int32_t* ws_pref;    // [B+1] exclusive prefix of blocks per sequence
    float2* ws_ml;       // [slots][RS] (running max m in log2 units, running sum l)
    float* ws_o;         // [slots][RS][D] un-normalised partial outputs
    long long num_blocks;
    int B, H, K, G, max_blocks, out_dtype, q_dtype, P, min_units;
    int T;               // new tokens (queries) per sequence
    int GT;              // query rows per (sequence, kv-head) pair: G * T
    int window;          // sliding window in tokens; 0 = full attention
    // Unit space: Kv = K * NRG heads per sequence. NRG > 1 splits a pair's GT
    // rows into groups of 8 ("virtual kv-heads" gv = g * NRG + group), each an
    // independent unit stream that re-reads the pair's tiles (from L2, since
    // the groups of a pair are adjacent in unit order). RS = rows per split
    // slot of the workspace (GT, or 8 with NRG > 1).
    int Kv, NRG, RS;
    int map_perm[3];     // tensor-map dims 1..3 -> 0 slot, 1 kv-head, 2 block
    int page_box;        // 16-bit caches, d = 128: the maps are page maps (one copy per tile)
    int page_perm[2];    // page-map dims 3, 4 -> 1 kv-head, 2 block
    int max_tail_chunks; // pooled chunks per worker range (0 = static partition only)
    float scale_log2;    // scale * log2(e)
};

// Warps per CTA and shared-memory ring bytes per warp of the split-KV kernel
// (overridable at build time for tuning sweeps).
#ifndef GQA_WARPS_PER_CTA
#define GQA_WARPS_PER_CTA 4
#endif
#ifndef GQA_RING_BYTES_PER_WARP
#define GQA_RING_BYTES_PER_WARP 16384
#endif
// CTAs per SM the narrow int8 tensor-core kernel is compiled to fit (registers).
#ifndef GQA_MIN_CTAS_PER_SM_I8
#define GQA_MIN_CTAS_PER_SM_I8 3
#endif
// The one-token INT4 tensor-core kernel (per-token scales) fits 128 registers
// without spilling, so it runs 4 CTAs (16 warps) per SM, with a ring of five
// 2.5 KB stages per warp so that four CTAs fit in shared memory. Measured on
// the B=128 ragged INT4 workload: 2852 against 2647 GB/s at 3 CTAs and six
// stages; four stages 2807. int8, FP8 and the KIVI-style cache spill at 128.
#ifndef GQA_MIN_CTAS_PER_SM_I4
#define GQA_MIN_CTAS_PER_SM_I4 4
#endif
#ifndef GQA_RING_BYTES_PER_WARP_I4
#define GQA_RING_BYTES_PER_WARP_I4 12800
#endif
// Ring bytes of a CTA whose warps share one ring (groups of more than 8 heads).
// Measured on the T = 4, G = 16 and G = 64 workloads at 12 warps per SM with
// the copy warp: 32 KB (four bf16 stages) beats 24 KB by 2-4% and ties 40 KB;
// 16 KB loses 5%.
#ifndef GQA_SHARED_RING_BYTES
#define GQA_SHARED_RING_BYTES 32768
#endif
// Warps per SM the tensor-core shared-ring kernels are compiled to fit
// (registers), copy warps included: 12 (168 registers, no next-pair query
// prefetch) beat the unconstrained 244 registers by 19-23% on the T = 4 and
// G = 16 workloads before the copy warp; 14 and 16 spill and lose 40%; with
// the copy warp, 9 (three CTAs of three warps) loses 15% to 12.
#ifndef GQA_SHARED_MIN_WARPS_PER_SM
#define GQA_SHARED_MIN_WARPS_PER_SM 12
#endif

// Tail balancing: about 1/8 of every worker's range, in at most kMaxTailChunks
// chunks of at least kMinChunk blocks, is pooled and taken at run time by
// whichever worker finishes its own part first.
#ifndef GQA_MAX_TAIL_CHUNKS
#define GQA_MAX_TAIL_CHUNKS 4
#endif
constexpr int kMaxTailChunks = GQA_MAX_TAIL_CHUNKS;
constexpr int kMinChunk = 4;

constexpr int kHeadsPerWarp = 8;   // query heads one warp serves (the MMA N dimension)

// kHeadWarps == 1: every warp is an independent split-KV worker with its own
// ring and serves all (<= 8) heads of its group. kHeadWarps > 1: the CTA is one
// worker; its kHeadWarps warps take 8 heads each of a larger group and share
// one ring, so each K/V tile is still loaded once for the whole group. One more
// warp only issues the copies: refilling a slot costs the issuing warp ~1000
// cycles a block, which a row warp would add to the group's pace while the
// others waited (measured; with eight row warps the ninth caps registers at 168
// and still wins).
template <int kKind, typename T, int D, int kHeadWarps = 1, bool kGeneral = false>
struct Cfg {
    // kGen: T > 1 queries per sequence or a sliding window (per-row ranges);
    // false compiles the one-token, full-attention step with no range logic.
    static constexpr bool kGen = kGeneral;
    static constexpr bool kI8 = std::is_same<T, int8_t>::value;
    static constexpr bool kFp8 = std::is_same<T, __nv_fp8_e4m3>::value;
    static constexpr bool kKc = std::is_same<T, int4kc>::value;   // K scales per channel
    static constexpr bool kI4 = std::is_same<T, int4x2>::value || kKc;
    static constexpr bool kCoded = kI8 || kFp8 || kI4;   // codes with fp16 scales
    static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    static constexpr int kEs = sizeof(T);                           // bytes per copied element
    static constexpr int kRowBytes = kI4 ? D / 2 : D * kEs;          // one token's row
    static constexpr int kTile = 16 * kRowBytes;                    // one (block, head) tile
    // fp16 scales after the two tiles: 16 k + 16 v, or (KIVI-style) D k + 16 v
    static constexpr int kScaleBytes = kKc ? 2 * D + 32 : kCoded ? 64 : 0;
    static constexpr int kVsOff = kKc ? 2 * D : 32;                 // v scales within them
    // 128-byte swizzled boxes for the tensor-core kernel; a 4-bit tile (64-byte
    // rows) takes the 64-byte swizzle (16-byte chunk ^= (row >> 1) & 3), which
    // spreads its V reads over twice the banks. The CUDA-core kernel reads rows
    // whole and needs none.
    static constexpr bool kSwizzle = (kKind == kKernelMma) && !kI4;
    static constexpr int kSwizzleBytes = kKind != kKernelMma ? 0 : kI4 ? 64 : 128;
    static constexpr int kStageAlign = kSwizzleBytes == 128 ? 1024 : kSwizzleBytes == 64 ? 512 : 128;
    static constexpr int kStage = ((2 * kTile + kScaleBytes + kStageAlign - 1) / kStageAlign) * kStageAlign;
    static constexpr int kNw = kHeadWarps;
    // The coded-cache kernels are issue-bound: the pool's bookkeeping costs
    // them more than the tail it removes (measured on int8), so they keep the
    // static partition.
    static constexpr int kTailChunks = kCoded ? 0 : kMaxTailChunks;
    // CTAs per SM the register budget is cut for. The code-cache kernels are
    // bound by issue and latency and gain from 12 warps per SM (16 for the
    // one-token INT4 kernel); the bf16/f16 kernels would spill at that budget
    // and keep 8 (all measured).
    static constexpr bool kCopyWarp = kHeadWarps >= 2 && kKind == kKernelMma;   // a warp that only issues copies
    static constexpr int kWarps = kHeadWarps == 1 ? GQA_WARPS_PER_CTA : kHeadWarps + (kCopyWarp ? 1 : 0);
    static constexpr bool kNarrowI4 =                // the one-token INT4 kernel with per-token scales
        kI4 && !kKc && !kGen && kHeadWarps == 1 && kKind == kKernelMma && D == 128;
    static constexpr int kMinCtas =
        kNarrowI4 ? GQA_MIN_CTAS_PER_SM_I4
        : (kHeadWarps == 1 && kKind == kKernelMma && D == 128) ? (kCoded ? GQA_MIN_CTAS_PER_SM_I8 : 2)
        : (kHeadWarps > 1 && kKind == kKernelMma) ? std::max(1, GQA_SHARED_MIN_WARPS_PER_SM / kWarps)
                                                  : 1;
    // Load the next pair's query fragments while the current pair runs (16
    // registers). A worker meets a new pair once every few hundred blocks on
    // the benchmark workloads, so kernels short of registers load them when
    // the pair starts instead.
    static constexpr bool kPrefetchQ =
        !(kCoded && kMinCtas >= 4) && !(kHeadWarps > 1 && kWarps * kMinCtas >= 12);
    static constexpr int kRings = kHeadWarps == 1 ? kWarps : 1;
    static constexpr int kStages = std::max(
        2, std::min(8, (kNarrowI4 ? GQA_RING_BYTES_PER_WARP_I4
                        : kHeadWarps == 1 ? GQA_RING_BYTES_PER_WARP : GQA_SHARED_RING_BYTES) / kStage));
    static constexpr int kBoxInner = kSwizzle ? 128 / kEs : kRowBytes / kEs;   // elements per box row
    static constexpr int kNumBox = kSwizzle ? kRowBytes / 128 : 1;
    static constexpr int kBoxBytes = 16 * kBoxInner * kEs;
    static constexpr uint32_t kTxBytes = 2 * kTile + kScaleBytes;
    // log2 of how far the block maximum may exceed the running maximum before
    // the state is rescaled (0 = always exact). The int8 path folds the V
    // scale into the fp16 P operand, so it keeps P <= 1.
    static constexpr float kRescaleSlack = kCoded ? 0.f : 8.f;
    static constexpr int kMt = D / 16;                              // m-tiles of the P.V product
    static constexpr int kRuns = D / 64;                            // 8-dim output runs per head
    static constexpr int kDpl = D / 32;                             // CUDA-core kernel: dims per lane
    static constexpr int kLaneBytes = kRowBytes / 32;               // ... and their bytes
};

// Dynamic shared memory layout shared by host and device.
template <class C>
struct Smem {
    static constexpr int kRing = C::kRings * C::kStages * C::kStage;
    static constexpr int kBars = kRing;                                   // "full", 8 B per stage
    static constexpr int kEmpty = kBars + C::kRings * C::kStages * 8;     // "empty" (shared ring)
    static constexpr int kMeta = kEmpty + C::kStages * 8;                 // 4 ints per stage
    static constexpr int kScan = kMeta + C::kRings * C::kStages * 16;     // 64 ints
    static constexpr int kLens = kScan + 64 * 4;                          // B ints, then B+1 prefix
    static int bytes(int B) { return 1024 + kLens + (2 * B + 1) * 4; }
};

// ------------------------------------------------------------------ prologue

// First position any query row of a length-L sequence attends (the window of
// its first new token), and the block holding it.
template <bool kGen>
__device__ __forceinline__ int attend_lo(const DecodeArgs& a, int L) {
    if constexpr (!kGen) return 0;
    else return a.window > 0 ? max(0, L - a.T + 1 - a.window) : 0;
}
template <bool kGen>
__device__ __forceinline__ int first_block(const DecodeArgs& a, int L) {
    return attend_lo<kGen>(a, L) / kBlock;
}

// Row rr (0 .. GT-1) of pair (b, g) -> its row of q and out ([B, T, H, d]).
template <bool kGen>
__device__ __forceinline__ long long q_row(const DecodeArgs& a, int b, int g, int rr) {
    if constexpr (!kGen) {
        return (long long)b * a.H + (long long)g * a.G + rr;
    } else {
        const int i = rr / a.G, hh = rr - i * a.G;
        return ((long long)b * a.T + i) * a.H + (long long)g * a.G + hh;
    }
}

// Attended positions [lo, hi) of row rr in a length-L sequence (rows past GT,
// the padding of a warp's 8 columns, get the last query's range).
__device__ __forceinline__ void row_range(const DecodeArgs& a, int L, int rr, int& lo, int& hi) {
    const int i = min(rr / a.G, a.T - 1);
    hi = L - a.T + i + 1;
    lo = a.window > 0 ? max(0, hi - a.window) : 0;
}


// Validated lengths into lens_s and the prefix pref[0..B] (pref[0] = 0) of the
// blocks each sequence's query rows attend.
template <bool kGen>
__device__ void block_prefix(const DecodeArgs& a, int* lens_s, int* pref, int* tmp) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, wid = tid >> 5;
    const int nw = nthr >> 5;
    const int maxtok = a.max_blocks * kBlock;
    int carry = 0;
    for (int base = 0; base < a.B; base += nthr) {
        const int i = base + tid;
        int L = 0;
        if (i < a.B) {
            L = a.context_lens[i];
            if (L < 0 || L > maxtok) {
                if (blockIdx.x == 0) flag_error(a.err, GQA_DEVERR_CONTEXT_LEN);
                L = 0;
            }
            lens_s[i] = L;
        }
        int x = (L + kBlock - 1) / kBlock - first_block<kGen>(a, L);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) tmp[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int t = lane < nw ? tmp[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, t, o);
                if (lane >= o) t += y;
            }
            tmp[32 + lane] = t;
        }
        __syncthreads();
        if (i < a.B) pref[i + 1] = carry + (wid ? tmp[32 + wid - 1] : 0) + x;
        carry += tmp[32 + nw - 1];
        __syncthreads();
    }
    if (tid == 0) pref[0] = 0;
    __syncthreads();
}

// Unit u -> (b, g, j): the largest b with K*pref[b] <= u, then the head and block.
__device__ __forceinline__ void locate(int u, const int* pref, int B, int K, int& b, int& g,
                                       int& j) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (K * pref[mid] <= u) lo = mid;
        else hi = mid;
    }
    const int nb = pref[lo + 1] - pref[lo];
    const int rem = u - K * pref[lo];
    b = lo;
    g = rem / nb;
    j = rem - g * nb;
}

// The pair after (b, g) in unit order (skipping empty sequences); b = B if none.
__device__ __forceinline__ void next_pair(const int* pref, int B, int K, int& b, int& g) {
    if (g + 1 < K) {
        ++g;
        return;
    }
    g = 0;
    ++b;
    while (b < B && pref[b + 1] == pref[b]) ++b;
}

// ------------------------------------------------------------------ loads

template <typename T, int N>
__device__ __forceinline__ void lds_row_as_float(uint32_t addr, float (&v)[N]) {
    if constexpr (std::is_same<T, float>::value) {
        if constexpr (N == 4) {
            const uint4 x = lds128(addr);
            v[0] = __uint_as_float(x.x); v[1] = __uint_as_float(x.y);
            v[2] = __uint_as_float(x.z); v[3] = __uint_as_float(x.w);
        } else {
            const uint2 x = lds64(addr);
            v[0] = __uint_as_float(x.x); v[1] = __uint_as_float(x.y);
        }
    } else if constexpr (std::is_same<T, __nv_fp8_e4m3>::value) {
        uint32_t w;
        if constexpr (N == 4) {
            w = lds32(addr);
        } else {
            unsigned short h;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr));
            w = h;
        }
#pragma unroll
        for (int e = 0; e < N; e += 2) {
            const float2 f = unpack2<false>(e4m3x2_to_f16x2(w >> (8 * e)));
            v[e] = f.x;
            v[e + 1] = f.y;
        }
    } else if constexpr (std::is_same<T, int4x2>::value || std::is_same<T, int4kc>::value) {
        // N 4-bit codes in N/2 bytes, element 2j in the low nibble
        uint32_t w;
        if constexpr (N == 4) {
            unsigned short h;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr));
            w = h;
        } else {
            unsigned short h;
            asm volatile("ld.shared.u8 %0, [%1];" : "=h"(h) : "r"(addr));
            w = h;
        }
#pragma unroll
        for (int e = 0; e < N; ++e) v[e] = (float)((int)(((w >> (4 * e)) & 0xFu) ^ 8u) - 8);
    } else if constexpr (std::is_same<T, int8_t>::value) {
        uint32_t w;
        if constexpr (N == 4) {
            w = lds32(addr);
        } else {
            unsigned short h;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr));
            w = h;
        }
#pragma unroll
        for (int e = 0; e < N; ++e) v[e] = (float)(int8_t)((w >> (8 * e)) & 0xff);
    } else {
        constexpr bool bf = std::is_same<T, __nv_bfloat16>::value;
        if constexpr (N == 4) {
            const uint2 x = lds64(addr);
            const float2 a = unpack2<bf>(x.x), b = unpack2<bf>(x.y);
            v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        } else {
            const float2 a = unpack2<bf>(lds32(addr));
            v[0] = a.x; v[1] = a.y;
        }
    }
}

__device__ __forceinline__ float load_q_float(const void* q, int q_dtype, long long i) {
    if (q_dtype == GQA_DTYPE_F32) return static_cast<const float*>(q)[i];
    if (q_dtype == GQA_DTYPE_F16) return __half2float(static_cast<const __half*>(q)[i]);
    return __bfloat162float(static_cast<const __nv_bfloat16*>(q)[i]);
}

__device__ __forceinline__ uint4 ldg128(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    const float2 f = unpack2<true>(w);
    return pack2<false>(f.x, f.y);
}

// Store 8 consecutive output floats (scaled) in the output dtype.
__device__ __forceinline__ void store8(void* out, int out_dtype, long long idx, const float (&v)[8],
                                       float mul) {
    if (out_dtype == GQA_DTYPE_F32) {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
        p[0] = make_float4(v[0] * mul, v[1] * mul, v[2] * mul, v[3] * mul);
        p[1] = make_float4(v[4] * mul, v[5] * mul, v[6] * mul, v[7] * mul);
    } else {
        uint4 w;
        if (out_dtype == GQA_DTYPE_BF16) {
            w.x = pack2<true>(v[0] * mul, v[1] * mul); w.y = pack2<true>(v[2] * mul, v[3] * mul);
            w.z = pack2<true>(v[4] * mul, v[5] * mul); w.w = pack2<true>(v[6] * mul, v[7] * mul);
        } else {
            w.x = pack2<false>(v[0] * mul, v[1] * mul); w.y = pack2<false>(v[2] * mul, v[3] * mul);
            w.z = pack2<false>(v[4] * mul, v[5] * mul); w.w = pack2<false>(v[6] * mul, v[7] * mul);
        }
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + idx) = w;
    }
}

__device__ __forceinline__ void store1(void* out, int out_dtype, long long idx, float v) {
    if (out_dtype == GQA_DTYPE_F32) static_cast<float*>(out)[idx] = v;
    else if (out_dtype == GQA_DTYPE_BF16) static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else static_cast<__half*>(out)[idx] = __float2half_rn(v);
}

// ------------------------------------------------------------------ tensor-core state

template <class C, int D>
struct MmaState {
    float m[2], l[2];          // heads 2c, 2c+1 of the group (log2 units)
    float acc[C::kMt][4];      // O^T fragments: rows = dims, cols = heads 2c, 2c+1
    uint2 qf[D / 16];          // Q^T B-fragments of the current pair, one per 16-dim k-step
    uint2 qn[C::kPrefetchQ ? D / 16 : 1];   // prefetched fragments of the next pair

    __device__ __forceinline__ void reset() {
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int j = 0; j < C::kMt; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    }
};

// Everything one block needs from shared memory, gathered before any math so
// the ring slot can be refilled while the block is being computed.
template <class C, int D>
struct MmaFrags {
    // bf16/f16: A fragments of K per k-step; int8/fp8: raw code quads; int4:
    // k[0] / k[1] = the 16 code bytes of tokens r / r+8 at byte 16c
    uint32_t k[D / 16][4];
    // bf16/f16: A fragments of V^T per m-tile; int8/fp8: raw rows of 4 tokens;
    // int4: v[i][0..1] = 8 code bytes (dims 16r..16r+15) of token i
    uint32_t v[C::kMt][4];
    float ks_r, ks_r8, vs_r, vs_r8;   // int8 scales of tokens r and r+8
    // KIVI-style K: the fp16 channel scales of dims 32c .. 32c+31 (8 per word)
    uint4 kc[C::kKc ? 4 : 1];
};

// Q fragments (B operand of the score MMA) of query head g*G + r; zero for
// padded heads r >= G. k-step t covers dims 16t..16t+15:
//  bf16/f16: .x = dims 16t + 2c, +1;     .y = dims 16t + 2c + 8, +9  (standard layout)
//  int8:     .x = dims 16t + 4c, +1;     .y = dims 16t + 4c + 2, +3  (matches the code quads)
template <class C, int D>
__device__ __forceinline__ void load_q_frags(const DecodeArgs& a, int b, int g, int hbase, int r,
                                             int c, uint2 (&qf)[D / 16]) {
    r += hbase;
    if (r >= a.GT || b >= a.B) {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) qf[i] = make_uint2(0, 0);
        return;
    }
    const uint16_t* base = static_cast<const uint16_t*>(a.q) + q_row<C::kGen>(a, b, g, r) * D;
    if constexpr (C::kI4) {
        // 4-bit K: lane c holds dims 32c .. 32c+31 of its tokens; k-step 2u+h
        // takes dims 32c + 8u + 2h + {0, 4} (.x) and + {1, 5} (.y)
        static_assert(D == 128, "the 4-bit tensor-core path reads 64-byte rows");
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint4 raw = __ldg(reinterpret_cast<const uint4*>(base + 32 * c + 8 * u));
            if (a.q_dtype == GQA_DTYPE_BF16) {
                raw.x = bf16x2_to_f16x2(raw.x);
                raw.y = bf16x2_to_f16x2(raw.y);
                raw.z = bf16x2_to_f16x2(raw.z);
                raw.w = bf16x2_to_f16x2(raw.w);
            }
            qf[2 * u].x = __byte_perm(raw.x, raw.z, 0x5410);       // dims +0, +4
            qf[2 * u].y = __byte_perm(raw.x, raw.z, 0x7632);       // dims +1, +5
            qf[2 * u + 1].x = __byte_perm(raw.y, raw.w, 0x5410);   // dims +2, +6
            qf[2 * u + 1].y = __byte_perm(raw.y, raw.w, 0x7632);   // dims +3, +7
        }
        return;
    }
#pragma unroll
    for (int t = 0; t < D / 16; ++t) {
        if constexpr (!C::kCoded) {
            qf[t].x = __ldg(reinterpret_cast<const uint32_t*>(base + 16 * t + 2 * c));
            qf[t].y = __ldg(reinterpret_cast<const uint32_t*>(base + 16 * t + 2 * c + 8));
        } else {
            uint2 raw = __ldg(reinterpret_cast<const uint2*>(base + 16 * t + 4 * c));
            if (a.q_dtype == GQA_DTYPE_BF16) {
                raw.x = bf16x2_to_f16x2(raw.x);
                raw.y = bf16x2_to_f16x2(raw.y);
            }
            qf[t] = raw;
        }
    }
}

// Output dim of accumulator row (j, rh): row r + 8*rh of m-tile j.
template <class C, int D>
__device__ __forceinline__ int acc_dim(int j, int rh, int r) {
    if constexpr (C::kCoded) return 16 * r + 2 * j + rh;
    else return 16 * j + r + 8 * rh;
}

template <bool kBf16>
__device__ __forceinline__ void mma_t(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                      uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (kBf16) mma_bf16(d, a0, a1, a2, a3, b0, b1);
    else mma_f16(d, a0, a1, a2, a3, b0, b1);
}


// Gather one block's operands from shared memory (all reads of the slot).
template <class C, int D>
__device__ __forceinline__ void mma_load(MmaFrags<C, D>& f, uint32_t stage, int lane, int r, int c) {
    const uint32_t sk = stage, sv = stage + C::kTile;
    const int mi = lane >> 3, rr = lane & 7;
    if constexpr (!C::kCoded) {
        // K: matrices (toks 0-7 | 8-15) x (dims 16t..+7 | +8..+15) = a0, a1, a2, a3
#pragma unroll
        for (int t = 0; t < D / 16; ++t)
            ldsm_x4(swz(sk, rr + 8 * (mi & 1), 2 * t + (mi >> 1)), f.k[t]);
        // V^T: transposed matrices (dims 16j..+7 | +8..+15) x (toks 0-7 | 8-15)
#pragma unroll
        for (int j = 0; j < C::kMt; ++j)
            ldsm_x4_t(swz(sv, rr + 8 * (mi >> 1), 2 * j + (mi & 1)), f.v[j]);
    } else if constexpr (C::kI4) {
        // K: 16 bytes (32 codes) of tokens r and r+8 at chunk c; V: 8 bytes
        // (dims 16r..16r+15) of tokens 2c, 2c+1, 2c+8, 2c+9. 64-byte rows with
        // the 64-byte swizzle (chunk ^ (row >> 1) & 3): K touches each bank once
        // per phase, V twice.
        const uint32_t kx = (uint32_t)((c ^ (r >> 1)) & 3) * 16;         // rows r, r+8 alike
        const uint4 k0 = lds128(sk + r * C::kRowBytes + kx);
        const uint4 k1 = lds128(sk + (r + 8) * C::kRowBytes + kx);
        f.k[0][0] = k0.x; f.k[0][1] = k0.y; f.k[0][2] = k0.z; f.k[0][3] = k0.w;
        f.k[1][0] = k1.x; f.k[1][1] = k1.y; f.k[1][2] = k1.z; f.k[1][3] = k1.w;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tok = 2 * c + (i & 1) + 8 * (i >> 1);
            const uint2 w = lds64(sv + tok * C::kRowBytes + 16 * ((r >> 1) ^ ((tok >> 1) & 3)) + 8 * (r & 1));
            f.v[i][0] = w.x;
            f.v[i][1] = w.y;
        }
    } else {
        // K codes: x4 number t holds chunks 2t (a0/a1) and 2t+1 (a2/a3), 16 codes each
#pragma unroll
        for (int t = 0; t < D / 32; ++t)
            ldsm_x4(swz(sk, rr + 8 * (mi & 1), 2 * t + (mi >> 1)), f.k[t]);
        // V codes: dims 16r..16r+15 of tokens 2c, 2c+1, 2c+8, 2c+9
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tok = 2 * c + (i & 1) + 8 * (i >> 1);
            const uint4 raw = lds128(swz(sv, tok, r));
            f.v[i][0] = raw.x; f.v[i][1] = raw.y; f.v[i][2] = raw.z; f.v[i][3] = raw.w;
        }
    }
    if constexpr (C::kCoded) {
        const uint32_t sc = stage + 2 * C::kTile;
        unsigned short h2, h3;
        if constexpr (C::kKc) {
            // lanes of one c read the same 64 bytes (a broadcast); the four c
            // cover 256 distinct bytes
#pragma unroll
            for (int u = 0; u < 4; ++u) f.kc[u] = lds128(sc + 64 * c + 16 * u);
            f.ks_r = f.ks_r8 = 1.f;
        } else {
            unsigned short h0, h1;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h0) : "r"(sc + 2 * r));
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h1) : "r"(sc + 2 * (r + 8)));
            f.ks_r = __half2float(__ushort_as_half(h0));
            f.ks_r8 = __half2float(__ushort_as_half(h1));
        }
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h2) : "r"(sc + C::kVsOff + 2 * r));
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h3) : "r"(sc + C::kVsOff + 2 * (r + 8)));
        f.vs_r = __half2float(__ushort_as_half(h2));
        f.vs_r8 = __half2float(__ushort_as_half(h3));
    }
}

// Which tokens of a block the two query rows of a lane (2c, 2c+1) attend:
// lo <= token < hi, block-relative. `partial` is false when every row of the
// pair attends the whole block (the masks are then skipped, and the block lies
// wholly inside the sequence).
struct BlockMask {
    bool partial;
    int lo0, hi0, lo1, hi1;
};

// One 16-token block on the tensor cores, from gathered operands. nvalid
// counts the block's tokens inside the sequence; slots past it hold arbitrary
// bits and are zeroed or masked.
template <class C, int D>
__device__ __forceinline__ void mma_compute(MmaState<C, D>& st, MmaFrags<C, D>& f, int nvalid,
                                            const BlockMask& bm, int r, int c, float scale_log2) {
    constexpr bool kB = C::kBf16;            // P and V operand type: bf16, else f16

    // ---- scores: S^T[tok][head] = K_tile . Q^T (two accumulators halve the chain)
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (!C::kCoded) {
#pragma unroll
        for (int t = 0; t < D / 16; ++t) {
            if (t & 1) mma_t<kB>(sb, f.k[t][0], f.k[t][1], f.k[t][2], f.k[t][3], st.qf[t].x, st.qf[t].y);
            else mma_t<kB>(sa, f.k[t][0], f.k[t][1], f.k[t][2], f.k[t][3], st.qf[t].x, st.qf[t].y);
        }
    } else if constexpr (C::kI4) {
        // word u of tokens r / r+8: bytes 4u..4u+3 = dims 32c + 8u + 0..7;
        // lo/hi nibbles of bytes 0,2 feed k-step 2u, of bytes 1,3 k-step 2u+1
        if constexpr (C::kKc) {
            // The per-channel K scales fold into q: q_i * s_i has at most 22
            // significant bits (11 x 11), so it is carried exactly as an f16
            // high part (the rounded product) plus an f16 low part (the
            // product minus the high part, one rounding), each with its own
            // MMA. Scales are permuted like the q fragments: (+0, +4), (+1, +5),
            // (+2, +6), (+3, +7).
            float sc_[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
            constexpr uint32_t kNeg = 0x80008000u;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w = f.k[0][u], w8 = f.k[1][u];
                const uint4 sc = f.kc[u];
                const uint32_t s0 = __byte_perm(sc.x, sc.z, 0x5410), s1 = __byte_perm(sc.x, sc.z, 0x7632);
                const uint32_t s2 = __byte_perm(sc.y, sc.w, 0x5410), s3 = __byte_perm(sc.y, sc.w, 0x7632);
                const uint32_t q0 = st.qf[2 * u].x, q1 = st.qf[2 * u].y;
                const uint32_t q2 = st.qf[2 * u + 1].x, q3 = st.qf[2 * u + 1].y;
                const uint32_t h0 = hmul2_u32(q0, s0), h1 = hmul2_u32(q1, s1);
                const uint32_t h2 = hmul2_u32(q2, s2), h3 = hmul2_u32(q3, s3);
                const uint32_t l0 = hfma2_u32(q0, s0, h0 ^ kNeg), l1 = hfma2_u32(q1, s1, h1 ^ kNeg);
                const uint32_t l2 = hfma2_u32(q2, s2, h2 ^ kNeg), l3 = hfma2_u32(q3, s3, h3 ^ kNeg);
                const uint32_t a0 = i4_lo_pair(w), a1 = i4_lo_pair(w8), a2 = i4_hi_pair(w), a3 = i4_hi_pair(w8);
                const uint32_t c0 = i4_lo_pair(w >> 8), c1 = i4_lo_pair(w8 >> 8);
                const uint32_t c2 = i4_hi_pair(w >> 8), c3 = i4_hi_pair(w8 >> 8);
                mma_f16(sa, a0, a1, a2, a3, h0, h1);
                mma_f16(sb, c0, c1, c2, c3, h2, h3);
                mma_f16(sc_, a0, a1, a2, a3, l0, l1);
                mma_f16(sd, c0, c1, c2, c3, l2, l3);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sa[e] += sc_[e];
                sb[e] += sd[e];
            }
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w = f.k[0][u], w8 = f.k[1][u];
                mma_f16(sa, i4_lo_pair(w), i4_lo_pair(w8), i4_hi_pair(w), i4_hi_pair(w8),
                        st.qf[2 * u].x, st.qf[2 * u].y);
                mma_f16(sb, i4_lo_pair(w >> 8), i4_lo_pair(w8 >> 8), i4_hi_pair(w >> 8), i4_hi_pair(w8 >> 8),
                        st.qf[2 * u + 1].x, st.qf[2 * u + 1].y);
            }
        }
    } else {
#pragma unroll
        for (int t = 0; t < D / 32; ++t) {
            uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
            if constexpr (C::kFp8) {
                // widened as 2^-8 x (integer ops; 256 goes into the K scale)
                l0 = e4m3x2_to_f16x2_scaled(f.k[t][0], 0u, 0x9180u);   // elements 0, 1
                h0 = e4m3x2_to_f16x2_scaled(f.k[t][0], 0u, 0xB3A2u);   // elements 2, 3
                l1 = e4m3x2_to_f16x2_scaled(f.k[t][1], 0u, 0x9180u);
                h1 = e4m3x2_to_f16x2_scaled(f.k[t][1], 0u, 0xB3A2u);
                l2 = e4m3x2_to_f16x2_scaled(f.k[t][2], 0u, 0x9180u);
                h2 = e4m3x2_to_f16x2_scaled(f.k[t][2], 0u, 0xB3A2u);
                l3 = e4m3x2_to_f16x2_scaled(f.k[t][3], 0u, 0x9180u);
                h3 = e4m3x2_to_f16x2_scaled(f.k[t][3], 0u, 0xB3A2u);
            } else {
                i8x4_to_f16x4(f.k[t][0], l0, h0);
                i8x4_to_f16x4(f.k[t][1], l1, h1);
                i8x4_to_f16x4(f.k[t][2], l2, h2);
                i8x4_to_f16x4(f.k[t][3], l3, h3);
            }
            mma_f16(sa, l0, l1, h0, h1, st.qf[2 * t].x, st.qf[2 * t].y);
            mma_f16(sb, l2, l3, h2, h3, st.qf[2 * t + 1].x, st.qf[2 * t + 1].y);
        }
    }
    // fragment: [0] = (tok r, head 2c), [1] = (tok r, head 2c+1), [2]/[3] = tok r+8
    float kr = scale_log2, kr8 = scale_log2, vr_s = 1.f, vr8_s = 1.f;
    if constexpr (C::kCoded) {
        const float kfix = C::kFp8 ? 256.f : 1.f;
        kr = f.ks_r * (kfix * scale_log2);
        kr8 = f.ks_r8 * (kfix * scale_log2);
        vr_s = f.vs_r;
        vr8_s = f.vs_r8;
    }
    float s0 = (sa[0] + sb[0]) * kr, s1 = (sa[1] + sb[1]) * kr;
    float s2 = (sa[2] + sb[2]) * kr8, s3 = (sa[3] + sb[3]) * kr8;
    if constexpr (!C::kGen) {
        if (r >= nvalid) { s0 = -INFINITY; s1 = -INFINITY; vr_s = 0.f; }
        if (r + 8 >= nvalid) { s2 = -INFINITY; s3 = -INFINITY; vr8_s = 0.f; }
    } else if (bm.partial) {
        if (r >= nvalid) vr_s = 0.f;
        if (r + 8 >= nvalid) vr8_s = 0.f;
        if (r < bm.lo0 || r >= bm.hi0) s0 = -INFINITY;
        if (r < bm.lo1 || r >= bm.hi1) s1 = -INFINITY;
        if (r + 8 < bm.lo0 || r + 8 >= bm.hi0) s2 = -INFINITY;
        if (r + 8 < bm.lo1 || r + 8 >= bm.hi1) s3 = -INFINITY;
    }

    // ---- online softmax (per head, over the 16 tokens of this block)
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
    }
    const bool up0 = mx0 > st.m[0] + C::kRescaleSlack, up1 = mx1 > st.m[1] + C::kRescaleSlack;
    if (__any_sync(kFull, up0 || up1)) {
        const float n0 = up0 ? mx0 : st.m[0], n1 = up1 ? mx1 : st.m[1];
        const float a0 = up0 ? fast_exp2(st.m[0] - n0) : 1.f;
        const float a1 = up1 ? fast_exp2(st.m[1] - n1) : 1.f;
        st.m[0] = n0; st.m[1] = n1;
        st.l[0] *= a0; st.l[1] *= a1;
#pragma unroll
        for (int j = 0; j < C::kMt; ++j) {
            st.acc[j][0] *= a0; st.acc[j][1] *= a1; st.acc[j][2] *= a0; st.acc[j][3] *= a1;
        }
    }
    // a row that has attended nothing yet keeps m = -inf (only after masked
    // blocks); its p must be 0, not NaN
    float mu0 = st.m[0], mu1 = st.m[1];
    if constexpr (C::kGen) {
        if (bm.partial) {
            if (mu0 == -INFINITY) mu0 = 0.f;
            if (mu1 == -INFINITY) mu1 = 0.f;
        }
    }
    const float p0 = fast_exp2(s0 - mu0), p1 = fast_exp2(s1 - mu1);
    const float p2 = fast_exp2(s2 - mu0), p3 = fast_exp2(s3 - mu1);
    st.l[0] += p0 + p2;
    st.l[1] += p1 + p3;

    // ---- P -> 16-bit high + low parts, transposed to the B layout of P.V
    const float w0 = p0 * vr_s, w1 = p1 * vr_s, w2 = p2 * vr8_s, w3 = p3 * vr8_s;
    const uint32_t hr = pack2<kB>(w0, w1), hr8 = pack2<kB>(w2, w3);
    const float2 fr = unpack2<kB>(hr), fr8 = unpack2<kB>(hr8);
    const uint32_t lr = pack2<kB>(w0 - fr.x, w1 - fr.y), lr8 = pack2<kB>(w2 - fr8.x, w3 - fr8.y);
    // hr holds (token r; heads 2c, 2c+1), hr8 the same for token r+8: an 8x8
    // token x head matrix each, whose transposes are exactly the B fragments
    // (tokens 2c, 2c+1 | 2c+8, 2c+9; head r) of P^T
    const uint32_t bh0 = movmatrix_t(hr), bh1 = movmatrix_t(hr8);
    const uint32_t bl0 = movmatrix_t(lr), bl1 = movmatrix_t(lr8);

    // ---- O^T[dim][head] += V^T . P^T (high part, then low part)
    if constexpr (!C::kCoded) {
        if (nvalid < kBlock) {
            // zero V of tokens past the end: the slots hold arbitrary (even NaN) bits
            const uint32_t m01 = (2 * c < nvalid ? 0x0000ffffu : 0u) | (2 * c + 1 < nvalid ? 0xffff0000u : 0u);
            const uint32_t m89 = (2 * c + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * c + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
            for (int j = 0; j < C::kMt; ++j) {
                f.v[j][0] &= m01; f.v[j][1] &= m01; f.v[j][2] &= m89; f.v[j][3] &= m89;
            }
        }
#pragma unroll
        for (int j = 0; j < C::kMt; ++j) {
            mma_t<kB>(st.acc[j], f.v[j][0], f.v[j][1], f.v[j][2], f.v[j][3], bh0, bh1);
            mma_t<kB>(st.acc[j], f.v[j][0], f.v[j][1], f.v[j][2], f.v[j][3], bl0, bl1);
        }
    } else {
        // f.v[i][w] holds dims 16r + 4w .. +3 (one byte each) of token i in
        // {2c, 2c+1, 2c+8, 2c+9}. Tokens past the end hold arbitrary codes.
        if (nvalid < kBlock) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = 2 * c + (i & 1) + 8 * (i >> 1);
                if (tok >= nvalid) f.v[i][0] = f.v[i][1] = f.v[i][2] = f.v[i][3] = 0u;
            }
        }
        if constexpr (C::kFp8) {
            // pair (x.b[k], y.b[k]) straight from the two tokens' words, with
            // the sign bytes, then widened as 2^-8 x (undone at the flush)
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t s0 = e ? 0xE6A2u : 0xC480u, s1 = e ? 0xF7B3u : 0xD591u;
                    const uint32_t a0 = e4m3x2_to_f16x2_scaled(f.v[0][wd], f.v[1][wd], s0);
                    const uint32_t a1 = e4m3x2_to_f16x2_scaled(f.v[0][wd], f.v[1][wd], s1);
                    const uint32_t a2 = e4m3x2_to_f16x2_scaled(f.v[2][wd], f.v[3][wd], s0);
                    const uint32_t a3 = e4m3x2_to_f16x2_scaled(f.v[2][wd], f.v[3][wd], s1);
                    const int j = 2 * wd + e;
                    mma_f16(st.acc[j], a0, a1, a2, a3, bh0, bh1);
                    mma_f16(st.acc[j], a0, a1, a2, a3, bl0, bl1);
                }
            }
            return;
        }
        if constexpr (C::kI4) {
            // byte j of a token's 8 bytes holds dims 16r + 2j (low nibble, row r
            // of m-tile j) and 16r + 2j + 1 (high nibble, row r+8). Pair the bytes
            // of tokens (2c, 2c+1) and (2c+8, 2c+9): (x.bj, x.bj+1, y.bj, y.bj+1).
#pragma unroll
            for (int wd = 0; wd < 2; ++wd) {
                const uint32_t t0 = __byte_perm(f.v[0][wd], f.v[1][wd], 0x5410);
                const uint32_t t1 = __byte_perm(f.v[0][wd], f.v[1][wd], 0x7632);
                const uint32_t u0 = __byte_perm(f.v[2][wd], f.v[3][wd], 0x5410);
                const uint32_t u1 = __byte_perm(f.v[2][wd], f.v[3][wd], 0x7632);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t tx = (e < 2 ? t0 : t1) >> (8 * (e & 1));
                    const uint32_t ux = (e < 2 ? u0 : u1) >> (8 * (e & 1));
                    const uint32_t a0 = i4_lo_pair(tx), a1 = i4_hi_pair(tx);
                    const uint32_t a2 = i4_lo_pair(ux), a3 = i4_hi_pair(ux);
                    const int j = 4 * wd + e;
                    mma_f16(st.acc[j], a0, a1, a2, a3, bh0, bh1);
                    mma_f16(st.acc[j], a0, a1, a2, a3, bl0, bl1);
                }
            }
            return;
        }
        // A fragment of m-tile j = 2w + e (dims 16r + 4w + 2e, +1) for the token
        // pair (x, y): interleave the two tokens' bytes, then widen each byte to
        // f16 exactly (1024 + (code ^ 0x80) - 1152).
        const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
        auto widen = [&](uint32_t t, uint32_t sel) -> uint32_t {
            const uint32_t hv = __byte_perm(t, 0x64646464u, sel);
            __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&hv), bias);
            return as_u32(h);
        };
        const uint32_t flip = 0x80808080u;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            const uint32_t x0 = f.v[0][wd] ^ flip, y0 = f.v[1][wd] ^ flip;
            const uint32_t x1 = f.v[2][wd] ^ flip, y1 = f.v[3][wd] ^ flip;
            // bytes (x.b0, y.b0, x.b1, y.b1) and (x.b2, y.b2, x.b3, y.b3)
            const uint32_t lo0 = __byte_perm(x0, y0, 0x5140), hi0 = __byte_perm(x0, y0, 0x7362);
            const uint32_t lo1 = __byte_perm(x1, y1, 0x5140), hi1 = __byte_perm(x1, y1, 0x7362);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t t0 = e ? hi0 : lo0, t1 = e ? hi1 : lo1;
                // rows r (dim 4wd + 2e) and r+8 (dim 4wd + 2e + 1): tokens (2c, 2c+1)
                const uint32_t a0 = widen(t0, 0x4140), a1 = widen(t0, 0x4342);
                const uint32_t a2 = widen(t1, 0x4140), a3 = widen(t1, 0x4342);
                const int j = 2 * wd + e;
                mma_f16(st.acc[j], a0, a1, a2, a3, bh0, bh1);
                mma_f16(st.acc[j], a0, a1, a2, a3, bl0, bl1);
            }
        }
    }
}

// Write the state of unit-space pair (b, gv): final output if this warp saw the
// whole pair, else a partial (o, m, l) into split slot (b*Kv + gv) + segment w,
// rows counted from row0 (the slot's first row).
template <class C, int D>
__device__ __forceinline__ void mma_flush(const DecodeArgs& a, MmaState<C, D>& st, int b, int gv,
                                          int hbase, int row0, bool whole, int w, int r, int c) {
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, o);
        l1 += __shfl_xor_sync(kFull, l1, o);
    }
    const long long slot = (long long)b * a.Kv + gv + w;
    const int g = gv / a.NRG;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int hh = hbase + 2 * c + e;               // row of the pair
        if (hh >= a.GT) continue;
        const float lsum = e ? l1 : l0;
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const long long obase = whole ? q_row<C::kGen>(a, b, g, hh) * D : (slot * a.RS + hh - row0) * D;
#pragma unroll
        for (int j = 0; j < C::kMt; ++j) {
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const int dim = acc_dim<C, D>(j, rh, r);
                const float v = st.acc[j][e + 2 * rh] * (C::kFp8 ? 256.f : 1.f);
                if (whole) store1(a.out, a.out_dtype, obase + dim, v * inv);
                else a.ws_o[obase + dim] = v;
            }
        }
        if (!whole && r == 0) a.ws_ml[slot * a.RS + hh - row0] = make_float2(st.m[e], lsum);
    }
}

// ------------------------------------------------------------------ CUDA-core state

template <class C, int D>
struct FmaState {
    static constexpr int kN = C::kDpl;
    float m[kHeadsPerWarp], l[kHeadsPerWarp];
    float acc[kHeadsPerWarp][kN];
    float q[kHeadsPerWarp][kN];

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int h = 0; h < kHeadsPerWarp; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < kN; ++i) acc[h][i] = 0.f;
        }
    }
};

template <class C, int D>
__device__ __forceinline__ void fma_load_q(const DecodeArgs& a, FmaState<C, D>& st, int b, int g,
                                           int hbase, int lane) {
#pragma unroll
    for (int h = 0; h < kHeadsPerWarp; ++h) {
        const bool live = hbase + h < a.GT && b < a.B;
        const long long row = live ? q_row<C::kGen>(a, b, g, hbase + h) : 0;
#pragma unroll
        for (int i = 0; i < C::kDpl; ++i)
            st.q[h][i] = live ? load_q_float(a.q, a.q_dtype, row * D + lane * C::kDpl + i) : 0.f;
    }
}

// One block, token by token: fp32 FMAs, butterfly reductions, per-token online softmax.
template <class C, int D, typename T>
__device__ __forceinline__ void fma_block(const DecodeArgs& a, FmaState<C, D>& st, uint32_t stage,
                                          int nvalid, bool partial, int bpos, int len, int hbase,
                                          int lane) {
    constexpr int kN = C::kDpl;
    const uint32_t sk = stage, sv = stage + C::kTile;
    const int G = a.GT - hbase;                  // rows of this warp: hbase .. hbase+7
    float kcs[kN];                               // KIVI-style K: this lane's channel scales
    if constexpr (C::kKc) lds_row_as_float<__half, kN>(stage + 2 * C::kTile + 2 * kN * lane, kcs);
    for (int t = 0; t < nvalid; ++t) {
        float kf[kN], vf[kN];
        lds_row_as_float<T, kN>(sk + t * C::kRowBytes + lane * C::kLaneBytes, kf);
        lds_row_as_float<T, kN>(sv + t * C::kRowBytes + lane * C::kLaneBytes, vf);
        float ksc = a.scale_log2, vsc = 1.f;
        if constexpr (C::kCoded) {
            unsigned short hv;
            if constexpr (C::kKc) {
#pragma unroll
                for (int i = 0; i < kN; ++i) kf[i] *= kcs[i];          // exact: code * fp16
            } else {
                unsigned short hk;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(hk) : "r"(stage + 2 * C::kTile + 2 * t));
                ksc *= __half2float(__ushort_as_half(hk));
            }
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(hv) : "r"(stage + 2 * C::kTile + C::kVsOff + 2 * t));
            vsc = __half2float(__ushort_as_half(hv));
        }
#pragma unroll
        for (int h = 0; h < kHeadsPerWarp; ++h) {
            if (h >= G) break;
            if constexpr (C::kGen) {
                if (partial) {                   // row outside its attended range?
                    int lo, hi;
                    row_range(a, len, hbase + h, lo, hi);
                    if (bpos + t < lo || bpos + t >= hi) continue;
                }
            }
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < kN; ++i) dot = fmaf(st.q[h][i], kf[i], dot);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);
            const float s = dot * ksc;
            const float mn = fmaxf(st.m[h], s);
            const float al = fast_exp2(st.m[h] - mn);
            const float p = fast_exp2(s - mn);
            st.l[h] = st.l[h] * al + p;
            const float pv = p * vsc;
#pragma unroll
            for (int i = 0; i < kN; ++i) st.acc[h][i] = fmaf(st.acc[h][i], al, pv * vf[i]);
            st.m[h] = mn;
        }
    }
}

template <class C, int D>
__device__ __forceinline__ void fma_flush(const DecodeArgs& a, FmaState<C, D>& st, int b, int gv,
                                          int hbase, int row0, bool whole, int w, int lane) {
    const long long slot = (long long)b * a.Kv + gv + w;
    const int g = gv / a.NRG;
#pragma unroll
    for (int h = 0; h < kHeadsPerWarp; ++h) {
        const int hh = hbase + h;                // row of the pair
        if (hh >= a.GT) break;
        const float inv = st.l[h] > 0.f ? 1.f / st.l[h] : 0.f;
        const long long obase = whole ? q_row<C::kGen>(a, b, g, hh) * D : (slot * a.RS + hh - row0) * D;
#pragma unroll
        for (int i = 0; i < C::kDpl; ++i) {
            const int dim = lane * C::kDpl + i;
            if (whole) store1(a.out, a.out_dtype, obase + dim, st.acc[h][i] * inv);
            else a.ws_o[obase + dim] = st.acc[h][i];
        }
        if (!whole && lane == 0) a.ws_ml[slot * a.RS + hh - row0] = make_float2(st.m[h], st.l[h]);
    }
}

// ------------------------------------------------------------------ the split-KV kernel

// Slot metadata the producer writes before a slot's barrier completes.
enum SlotKind : int { kSlotData = 0, kSlotSkip = 1, kSlotEnd = 2 };

// The partition of the U units, identical on every CTA and in the combine.
// Worker w's range is [w*R, min(U, (w+1)*R)); its first Rs units are its own
// (static segment), the remaining cpw chunks of Cz units go to a pool. Segment
// index of worker w's static part is w*(1+cpw), of its chunk i w*(1+cpw)+1+i:
// indices grow with unit position, so a split slot (b*K + g) + segment is unique
// and every pair's pieces are the consecutive segments that cover it.
struct Partition {
    int U, R, Rs, Cz, cpw, P;
    __device__ __forceinline__ int segment_of(int u) const {
        const int w = u / R, off = u - w * R;
        return w * (1 + cpw) + (off < Rs ? 0 : 1 + (off - Rs) / Cz);
    }
};

__device__ __forceinline__ Partition make_partition(const DecodeArgs& a, int U) {
    Partition pt;
    pt.U = U;
    pt.P = max(a.P, 1);
    pt.R = max((U + pt.P - 1) / pt.P, a.min_units);
    pt.Cz = max(kMinChunk, (pt.R + 31) / 32);
    pt.cpw = min(a.max_tail_chunks, pt.R / (8 * pt.Cz));
    pt.Rs = pt.R - pt.cpw * pt.Cz;
    return pt;
}

template <int kKind, typename T, int D, int kHeadWarps, bool kGen>
__global__ void __launch_bounds__(Cfg<kKind, T, D, kHeadWarps, kGen>::kWarps * 32,
                                  Cfg<kKind, T, D, kHeadWarps, kGen>::kMinCtas)
split_kv_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const DecodeArgs a) {
    using C = Cfg<kKind, T, D, kHeadWarps, kGen>;
    using S = Smem<C>;
    constexpr bool kShared = kHeadWarps > 1;     // one ring, one worker per CTA
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);
    int* tmp = reinterpret_cast<int*>(gbase + S::kScan);
    int* lens_s = reinterpret_cast<int*>(gbase + S::kLens);
    int* pref = lens_s + a.B;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    launch_dependents();                       // the combine kernel may take its place now
    grid_dependency_wait();                    // inputs may come from the previous kernel
    block_prefix<kGen>(a, lens_s, pref, tmp);
    const Partition pt = make_partition(a, a.Kv * pref[a.B]);
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i <= a.B; i += blockDim.x) a.ws_pref[i] = pref[i];
        if (threadIdx.x == 0) {
            a.ws_hdr[0] = pt.R;
            a.ws_hdr[1] = pt.U;
            a.ws_hdr[2] = pt.Rs;
            a.ws_hdr[3] = pt.Cz;
            a.ws_hdr[4] = pt.P;
            a.ws_hdr[5] = pt.cpw;
        }
    }
    if (pt.U == 0) return;                     // uniform: every row is empty (combine zeroes them)

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int w = kShared ? (int)blockIdx.x : (int)blockIdx.x * C::kWarps + warp;   // worker
    // first query row this warp serves: fixed per warp when the CTA's warps
    // share a pair, else set per pair from its row group
    int hbase = kShared ? warp * kHeadsPerWarp : 0;
    if (w >= pt.P) return;                     // uniform per worker (grid is sized to P)
    const long long sl = (long long)w * pt.R;
    const int st_lo = (int)min((long long)pt.U, sl);
    const int st_hi = (int)min((long long)pt.U, sl + pt.Rs);

    const int ring_id = kShared ? 0 : warp;
    const uint32_t ring = sbase + ring_id * C::kStages * C::kStage;
    const uint32_t bar0 = sbase + S::kBars + ring_id * C::kStages * 8;
    const uint32_t ebar0 = sbase + S::kEmpty;
    volatile int* meta = reinterpret_cast<volatile int*>(gbase + S::kMeta) + ring_id * C::kStages * 4;
    // the warp that issues this ring's copies: each warp its own, else warp 0,
    // or the copy warp (warp kHeadWarps) that does nothing else
    const bool producer = !kShared || warp == (C::kCopyWarp ? kHeadWarps : 0);
    if (kShared) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < C::kStages; ++s) {
                mbar_init(bar0 + 8 * s, 1);
                mbar_init(ebar0 + 8 * s, kHeadWarps);
            }
            fence_mbar_init();
        }
        __syncthreads();                       // every warp of this CTA reached here (same worker)
    } else {
        if (lane == 0) {
            for (int s = 0; s < C::kStages; ++s) mbar_init(bar0 + 8 * s, 1);
            fence_mbar_init();
        }
        __syncwarp();
    }
    // K/V tiles are read once: evict them first. The 32-byte scale rows of a
    // (block, kv-head) share L2 lines with the other heads' rows, which other
    // workers read later; keep those lines (all scales are ~1.6% of the pool).
    const uint64_t pol = l2_policy_evict_first();
    const uint64_t pol_keep = C::kCoded ? l2_policy_evict_last() : pol;

    // ---- producer: segments (static range first, then pooled chunks) and copies
    // The pool is asked for the next chunk kLookahead units before the current
    // segment runs out, and that chunk's block-table entries are fetched as soon
    // as its id is known, so switching segments costs no round trip.
    constexpr int kLookahead = 2;
    const unsigned long long pool = (unsigned long long)pt.P * pt.cpw;
    int iss_u = 0, iss_hi = 0, iss_seg = -1, n_issued = 0;
    int nxt_lo = 0, nxt_hi = 0, nxt_seg = -1;
    bool iss_done = false, nxt_ok = false, pend_out = false, exhausted = pool == 0;
    unsigned long long pend = 0;                           // lane 0: in-flight pool ticket
    int win_base = -(1 << 30), win_phys = -1, win_g = 0;   // lane l: unit win_base + l
    auto refill = [&](int base) {
        win_base = base;
        const int u = base + lane;
        win_phys = -1;
        win_g = 0;
        if (u < pt.U) {
            int b, g, j;
            locate(u, pref, a.B, a.Kv, b, g, j);
            const int ph = a.block_tables[(long long)b * a.max_blocks + first_block<C::kGen>(a, lens_s[b]) + j];
            if (ph < 0 || ph >= a.num_blocks) flag_error(a.err, GQA_DEVERR_BLOCK_INDEX);
            else win_phys = ph;
            win_g = g / a.NRG;                 // the real kv-head
        }
    };
    auto request = [&]() {
        if (pend_out || exhausted) return;
        if (lane == 0) pend = atomicAdd(a.ws_ctr, 1ull);
        pend_out = true;
    };
    auto resolve = [&]() {                 // the in-flight ticket -> the next segment
        while (pend_out) {
            const unsigned long long cidx = __shfl_sync(kFull, pend, 0);
            pend_out = false;
            if (cidx >= pool) {
                exhausted = true;
                return;
            }
            const int wc = (int)(cidx % pt.P), ic = (int)(cidx / pt.P);
            const long long lo = (long long)wc * pt.R + pt.Rs + (long long)ic * pt.Cz;
            if (lo >= pt.U) {              // a chunk past the last unit: take another
                request();
                continue;
            }
            nxt_lo = (int)lo;
            nxt_hi = (int)min((long long)pt.U, lo + pt.Cz);
            nxt_seg = wc * (1 + pt.cpw) + 1 + ic;
            nxt_ok = true;
        }
    };
    if (producer) {
        if (st_lo < st_hi) {
            iss_u = st_lo;
            iss_hi = st_hi;
            iss_seg = w * (1 + pt.cpw);
            if (iss_hi - iss_u <= kLookahead) request();
        } else {
            request();
        }
    }
    // Fill ring slot s with the next unit of this worker, or with the end marker.
    auto issue_next = [&](int s) {
        if (iss_done) return;
        const uint32_t bar = bar0 + 8 * s;
        ++n_issued;
        if (iss_u >= iss_hi) {
            if (!nxt_ok) {
                request();
                resolve();
            }
            if (!nxt_ok) {
                iss_done = true;
                if (lane == 0) {
                    meta[4 * s] = kSlotEnd;
                    mbar_arrive(bar);
                }
                return;
            }
            iss_u = nxt_lo;
            iss_hi = nxt_hi;
            iss_seg = nxt_seg;
            nxt_ok = false;
            if (iss_hi - iss_u <= kLookahead) request();
        }
        const int u = iss_u++;
        // pooled chunks can lie before this worker's own range: refill on any jump
        if (u < win_base || u - win_base >= 32) refill(u);
        const int ph = __shfl_sync(kFull, win_phys, u - win_base);
        const int gg = __shfl_sync(kFull, win_g, u - win_base);
        if (lane == 0) {
            meta[4 * s + 1] = u;
            meta[4 * s + 2] = iss_seg;
            meta[4 * s + 3] = iss_hi;
            if (ph >= 0) {
                const uint32_t dst = ring + s * C::kStage;
                auto coord = [&](int which) { return which == 0 ? 0 : (which == 1 ? gg : ph); };
                const int y = coord(a.map_perm[0]), z = coord(a.map_perm[1]), ww = coord(a.map_perm[2]);
                meta[4 * s] = kSlotData;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, C::kTxBytes);
                if (C::kNumBox == 2 && a.page_box) {
                    // one copy per tile: the page map lands both 64-element halves
                    const int p3 = coord(a.page_perm[0]), p4 = coord(a.page_perm[1]);
                    tma_load_5d(dst, &kmap, 0, 0, 0, p3, p4, bar, pol);
                    tma_load_5d(dst + C::kTile, &vmap, 0, 0, 0, p3, p4, bar, pol);
                } else {
#pragma unroll
                    for (int x = 0; x < C::kNumBox; ++x)
                        tma_load_4d(dst + x * C::kBoxBytes, &kmap, x * C::kBoxInner, y, z, ww, bar, pol);
#pragma unroll
                    for (int x = 0; x < C::kNumBox; ++x)
                        tma_load_4d(dst + C::kTile + x * C::kBoxBytes, &vmap, x * C::kBoxInner, y, z, ww, bar, pol);
                }
                if constexpr (C::kCoded) {
                    const long long si = ((long long)ph * a.K + gg) * kBlock;
                    if constexpr (C::kKc)   // whole 256-byte rows of their own: read once
                        bulk_load(dst + 2 * C::kTile, a.k_scale + ((long long)ph * a.K + gg) * D, 2 * D, bar, pol);
                    else
                        bulk_load(dst + 2 * C::kTile, a.k_scale + si, 32, bar, pol_keep);
                    bulk_load(dst + 2 * C::kTile + C::kVsOff, a.v_scale + si, 32, bar, pol_keep);
                }
            } else {
                meta[4 * s] = kSlotSkip;
                mbar_arrive(bar);
            }
        }
        if (iss_hi - iss_u == kLookahead) request();
        if (iss_u == iss_hi) {             // segment issued: learn the next one, prefetch its table
            resolve();
            if (nxt_ok) refill(nxt_lo);
        }
    };
    // Bounded waits whose verdict is warp-uniform, so a timeout never splits a warp.
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(kFull, mbar_wait(bar, parity));
    };
    auto bail = [&](int k) {
        // A copy (or a peer warp) did not arrive in time: report, let this ring's
        // in-flight copies land, leave.
        if (lane == 0) flag_error(a.err, GQA_DEVERR_TIMEOUT);
        if (producer)
            for (int q = k; q < n_issued; ++q)
                mbar_wait(bar0 + 8 * (q % C::kStages), (uint32_t)(q / C::kStages) & 1u, kWaitLimitNs / 4);
    };
    // Hand slot s (use k, just read) back; the producer refills it.
    auto release_and_refill = [&](int k, int s) -> bool {
        __syncwarp();
        if (kShared && lane == 0) mbar_arrive(ebar0 + 8 * s);
        if (producer && !iss_done) {
            if (kShared && !wait_all(ebar0 + 8 * s, (uint32_t)(k / C::kStages) & 1u)) return false;
            issue_next(s);
        }
        return true;
    };

    if (producer)
        for (int s = 0; s < C::kStages; ++s) issue_next(s);
    if (C::kCopyWarp && producer) {
        // refill each slot once every row warp has released it, in use order;
        // the last fill is the end marker, after which the row warps finish alone
        for (int k = 0; !iss_done; ++k) {
            const int s = k % C::kStages;
            if (!wait_all(ebar0 + 8 * s, (uint32_t)(k / C::kStages) & 1u)) {
                bail(k);
                return;
            }
            issue_next(s);
        }
        return;
    }

    // ---- consumer: walk the units as they arrive
    const int r = lane >> 2, c = lane & 3;
    using State = typename std::conditional<kKind == kKernelMma, MmaState<C, D>, FmaState<C, D>>::type;
    State st;
    int cb = 0, cg = 0, cj = 0, cnb = 1, clen = 0, first_j = 0, cu_pair = 0;
    int nb_b = 0, nb_g = 0, next_u = -1;
    // Blocks cj in [cjf_lo, cjf_lo + cjf_n) of the current pair are attended
    // whole by every row (all rows attend positions [max(0, L - W), L - T + 1));
    // the others need masks.
    int cjf_lo = 0, cjf_n = 0;
    auto pair_ranges = [&]() {
        if constexpr (!C::kGen) return;
        const int c0 = first_block<C::kGen>(a, clen) * kBlock;
        const int flo = a.window > 0 ? max(0, clen - a.window) : 0;
        const int fhi = clen - a.T + 1;
        cjf_lo = (max(0, flo - c0) + kBlock - 1) / kBlock;
        const int cjf_hi = fhi - c0 >= kBlock ? (fhi - c0 - kBlock) / kBlock : -1;
        cjf_n = max(0, cjf_hi - cjf_lo + 1);
    };

    for (int k = 0;; ++k) {
        const int s = k % C::kStages;
        // every lane observes the phase, which acquires the TMA writes and the metadata
        if (!wait_all(bar0 + 8 * s, (uint32_t)(k / C::kStages) & 1u)) {
            bail(k);
            return;
        }
        const int kind = meta[4 * s];
        if (kind == kSlotEnd) break;
        const int u = meta[4 * s + 1], seg = meta[4 * s + 2], seg_end = meta[4 * s + 3];
        if (u != next_u) {
            // first unit of a segment: find its pair and load that pair's queries
            locate(u, pref, a.B, a.Kv, cb, cg, cj);
            if (!kShared) hbase = (cg % a.NRG) * kHeadsPerWarp;
            cnb = pref[cb + 1] - pref[cb];
            clen = lens_s[cb];
            pair_ranges();
            first_j = cj;
            cu_pair = a.Kv * pref[cb] + cg * cnb;
            st.reset();
            nb_b = cb;
            nb_g = cg;
            next_pair(pref, a.B, a.Kv, nb_b, nb_g);
            if constexpr (kKind == kKernelMma) {
                load_q_frags<C, D>(a, cb, cg / a.NRG, hbase, r, c, st.qf);
                if constexpr (C::kPrefetchQ) {
                    if (cu_pair + cnb < seg_end)
                        load_q_frags<C, D>(a, nb_b, nb_g / a.NRG,
                                           kShared ? hbase : (nb_g % a.NRG) * kHeadsPerWarp, r, c, st.qn);
                }
            } else {
                fma_load_q<C, D>(a, st, cb, cg / a.NRG, hbase, lane);
            }
        }
        bool partial;
        int bpos, nvalid;                         // block position, its tokens inside the sequence
        if constexpr (!C::kGen) {
            bpos = kBlock * cj;
            nvalid = min((int)kBlock, clen - bpos);
            partial = nvalid < kBlock;
        } else {
            partial = (unsigned)(cj - cjf_lo) >= (unsigned)cjf_n;
            bpos = 0;
            nvalid = kBlock;
            if (partial) {
                bpos = (first_block<C::kGen>(a, clen) + cj) * kBlock;
                nvalid = min((int)kBlock, clen - bpos);
            }
        }
        const bool unit_ok = kind == kSlotData;
        if constexpr (kKind == kKernelMma) {
            // read the whole slot, hand it back to TMA, then compute from registers
            MmaFrags<C, D> fr;
            if (unit_ok) mma_load<C, D>(fr, ring + s * C::kStage, lane, r, c);
            if (!release_and_refill(k, s)) {
                bail(k + 1);
                return;
            }
            BlockMask bm{partial, 0, 0, 0, 0};
            if (C::kGen && partial) {
                row_range(a, clen, hbase + 2 * c, bm.lo0, bm.hi0);
                row_range(a, clen, hbase + 2 * c + 1, bm.lo1, bm.hi1);
                bm.lo0 -= bpos; bm.hi0 -= bpos; bm.lo1 -= bpos; bm.hi1 -= bpos;
            }
            if (unit_ok) mma_compute<C, D>(st, fr, nvalid, bm, r, c, a.scale_log2);
        } else {
            if (unit_ok) fma_block<C, D, T>(a, st, ring + s * C::kStage, nvalid, partial, bpos, clen, hbase, lane);
            if (!release_and_refill(k, s)) {
                bail(k + 1);
                return;
            }
        }

        const bool last_of_pair = (cj == cnb - 1);
        const bool last_of_seg = (u == seg_end - 1);
        next_u = u + 1;
        if (last_of_pair || last_of_seg) {
            const bool whole = (first_j == 0) && last_of_pair;
            const int row0 = kShared ? 0 : hbase;
            if constexpr (kKind == kKernelMma) mma_flush<C, D>(a, st, cb, cg, hbase, row0, whole, seg, r, c);
            else fma_flush<C, D>(a, st, cb, cg, hbase, row0, whole, seg, lane);
            if (last_of_seg) {
                next_u = -1;                   // the next unit starts a new segment
                continue;
            }
            cb = nb_b;
            cg = nb_g;
            if (!kShared) hbase = (cg % a.NRG) * kHeadsPerWarp;
            cj = 0;
            first_j = 0;
            cnb = pref[cb + 1] - pref[cb];
            clen = lens_s[cb];
            pair_ranges();
            cu_pair = a.Kv * pref[cb] + cg * cnb;
            st.reset();
            next_pair(pref, a.B, a.Kv, nb_b, nb_g);
            if constexpr (kKind == kKernelMma) {
                if constexpr (C::kPrefetchQ) {
#pragma unroll
                    for (int q = 0; q < D / 16; ++q) st.qf[q] = st.qn[q];
                    if (cu_pair + cnb < seg_end)
                        load_q_frags<C, D>(a, nb_b, nb_g / a.NRG,
                                           kShared ? hbase : (nb_g % a.NRG) * kHeadsPerWarp, r, c, st.qn);
                } else {
                    load_q_frags<C, D>(a, cb, cg / a.NRG, hbase, r, c, st.qf);
                }
            } else {
                fma_load_q<C, D>(a, st, cb, cg / a.NRG, hbase, lane);
            }
        } else {
            ++cj;
        }
    }
}

// ------------------------------------------------------------------ combine

// Merge the splits of each (sequence, new token, query head) row; zero rows
// of empty sequences. kRowWarps warps share a row (each takes an even share of its splits;
// they meet in shared memory); a CTA holds kRows rows. CTA 0 also rewinds the run-time
// work counter for the next call (every split-KV CTA has finished by now).
template <int D, int kRowWarps, int kRows>
__global__ void __launch_bounds__(kRowWarps * kRows * 32) combine_kernel(const DecodeArgs a) {
    static_assert(kRowWarps == 1 || kRows == 1, "rows of several warps need a CTA each");
    __shared__ float s_red[kRowWarps];
    __shared__ float s_acc[kRowWarps > 1 ? kRowWarps : 1][kRowWarps > 1 ? D : 1];
    __shared__ float s_l[kRowWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = warp % kRowWarps;
    const int bh = (int)blockIdx.x * kRows + warp / kRowWarps;   // rows < 2^31 (host-checked)
    launch_dependents();
    grid_dependency_wait();                    // the split-KV kernel's partials
    if (blockIdx.x == 0 && tid == 0) *a.ws_ctr = 0ull;
    const int TH = a.T * a.H;
    if (bh >= a.B * TH) return;
    const int b = bh / TH, ih = bh - b * TH;                          // ih = i * H + h
    const int i = ih / a.H, h = ih - i * a.H, g = h / a.G;
    const int rr = i * a.G + (h - g * a.G);                           // row of the pair
    const int rg = a.NRG > 1 ? rr / kHeadsPerWarp : 0;                // its row group
    const int gv = g * a.NRG + rg;                                    // unit-space head
    const int hh = rr - rg * kHeadsPerWarp;                           // row in the slot
    const long long orow = (long long)bh * D;                         // out is [B, T, H, d]
    const int p0 = a.ws_pref[b];
    const int nb = a.ws_pref[b + 1] - p0;
    if (nb == 0) {
        for (int i = sub * 32 + lane; i < D; i += kRowWarps * 32) store1(a.out, a.out_dtype, orow + i, 0.f);
        return;
    }
    Partition pt;
    pt.R = a.ws_hdr[0];
    pt.U = a.ws_hdr[1];
    pt.Rs = a.ws_hdr[2];
    pt.Cz = a.ws_hdr[3];
    pt.P = a.ws_hdr[4];
    pt.cpw = a.ws_hdr[5];
    const int u0 = a.Kv * p0 + gv * nb;
    const int s0 = pt.segment_of(u0), s1 = pt.segment_of(u0 + nb - 1);
    if (s0 == s1) return;                      // one segment held the whole pair and wrote it
    const long long first = (long long)b * a.Kv + gv + s0;   // slot of the first piece
    const int n = s1 - s0 + 1;

    // One pass over the pieces. Each warp takes an even share of them (in
    // chunks of 32 when the share is larger): lane j loads piece j's (m, l), the
    // warp keeps a running maximum Mw and rescales what it holds when Mw grows,
    // then every lane gathers its dims of the chunk's partial vectors with
    // independent loads, 8 in flight. The warps of a row meet in shared memory,
    // where each share is rescaled from its Mw to the row's maximum. Pieces that
    // saw only skipped blocks hold m = -inf and o = 0 and weigh 0.
    const int per = (n + kRowWarps - 1) / kRowWarps;
    const int lo = min(n, sub * per), hi = min(n, lo + per);
    const bool has_dims = 4 * lane < D;
    const long long step = (long long)a.RS * D;
    float Mw = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = lo; base < hi; base += 32) {
        const int p = base + lane;
        float2 ml = make_float2(-INFINITY, 0.f);
        if (p < hi) ml = __ldcg(&a.ws_ml[(first + p) * a.RS + hh]);
        float mc = ml.x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kFull, mc, o));
        const float Mn = fmaxf(Mw, mc);
        if (Mn == -INFINITY) continue;         // warp-uniform: nothing seen yet
        const float sc = fast_exp2(Mw - Mn);   // 0 while Mw = -inf, 1 if unchanged
        acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
        L *= sc;
        Mw = Mn;
        const float e = fast_exp2(ml.x - Mw);
        L += ml.y * e;
        const int cnt = min(32, hi - base);
        const float* op = a.ws_o + ((first + base) * a.RS + hh) * D + 4 * lane;
        for (int j0 = 0; j0 < cnt; j0 += 8) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                const float ej = __shfl_sync(kFull, e, j & 31);
                if (j < cnt && has_dims) {
                    const float4 o = __ldcg(reinterpret_cast<const float4*>(op + j * step));
                    acc.x += o.x * ej; acc.y += o.y * ej; acc.z += o.z * ej; acc.w += o.w * ej;
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
    if constexpr (kRowWarps > 1) {
        if (has_dims) {
            s_acc[sub][4 * lane + 0] = acc.x;
            s_acc[sub][4 * lane + 1] = acc.y;
            s_acc[sub][4 * lane + 2] = acc.z;
            s_acc[sub][4 * lane + 3] = acc.w;
        }
        if (lane == 0) {
            s_red[sub] = Mw;
            s_l[sub] = L;
        }
        __syncthreads();
        float M = s_red[0];
#pragma unroll
        for (int w = 1; w < kRowWarps; ++w) M = fmaxf(M, s_red[w]);
        auto share_scale = [&](int w) {        // a share with no pieces weighs 0
            return s_red[w] == -INFINITY ? 0.f : fast_exp2(s_red[w] - M);
        };
        float Lt = 0.f;
#pragma unroll
        for (int w = 0; w < kRowWarps; ++w) Lt += s_l[w] * share_scale(w);
        const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
        for (int i = tid; i < D; i += blockDim.x) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kRowWarps; ++w) v += s_acc[w][i] * share_scale(w);
            store1(a.out, a.out_dtype, orow + i, v * inv);
        }
    } else {
        const float inv = L > 0.f ? 1.f / L : 0.f;
        if (has_dims) {
            store1(a.out, a.out_dtype, orow + 4 * lane + 0, acc.x * inv);
            store1(a.out, a.out_dtype, orow + 4 * lane + 1, acc.y * inv);
            store1(a.out, a.out_dtype, orow + 4 * lane + 2, acc.z * inv);
            store1(a.out, a.out_dtype, orow + 4 * lane + 3, acc.w * inv);
        }
    }
}

// ------------------------------------------------------------------ host side

struct Variant {
    const void* fn;
    int tail_chunks;     // pooled chunks per worker range
    int warps;           // threads / 32
    int workers_per_cta; // split-KV workers per CTA
    int box_inner;       // elements per TMA box row
    int swizzle_bytes;   // TMA swizzle of the tiles: 0, 64 or 128
    int (*smem)(int);
};

template <int kKind, typename T, int D, int NW, bool kGen>
Variant make_variant() {
    using C = Cfg<kKind, T, D, NW, kGen>;
    return Variant{reinterpret_cast<const void*>(&split_kv_kernel<kKind, T, D, NW, kGen>), C::kTailChunks, C::kWarps,
                   NW == 1 ? C::kWarps : 1, C::kBoxInner, C::kSwizzleBytes, &Smem<C>::bytes};
}

template <int kKind, typename T, int D, bool kGen>
Variant pick_width(int nw) {
    if (nw == 1) return make_variant<kKind, T, D, 1, kGen>();
    if (nw == 2) return make_variant<kKind, T, D, 2, kGen>();
    if (nw == 4) return make_variant<kKind, T, D, 4, kGen>();
    return make_variant<kKind, T, D, 8, kGen>();
}

template <typename T, int D, bool kGen>
bool pick_kind(int kind, int nw, Variant& v) {
    if (kind == kKernelMma) {
        if constexpr (std::is_same<T, float>::value ||
                      ((std::is_same<T, int8_t>::value || std::is_same<T, __nv_fp8_e4m3>::value ||
                        std::is_same<T, int4x2>::value || std::is_same<T, int4kc>::value) && D != 128)) {
            return false;
        } else {
            v = pick_width<kKernelMma, T, D, kGen>(nw);
            return true;
        }
    }
    if constexpr (std::is_same<T, float>::value) {
        v = pick_width<kKernelFma, T, D, kGen>(nw);
        return true;
    } else {
        // the CUDA-core kernel serves fp32 caches, and <= 8-head groups of the others
        if (nw > 1) return false;
        v = make_variant<kKernelFma, T, D, 1, kGen>();
        return true;
    }
}

template <typename T, bool kGen>
bool pick_dim(int kind, int d, int nw, Variant& v) {
    if (d == 64) return pick_kind<T, 64, kGen>(kind, nw, v);
    if (d == 128) return pick_kind<T, 128, kGen>(kind, nw, v);
    return false;
}

// The split-KV kernel for a cache dtype, kernel kind, head_dim and warps per
// pair, in its plain (one token, full attention) or general flavour.
template <bool kGen>
bool pick_variant(int dtype, int kind, int d, int nw, Variant& v) {
    switch (dtype) {
        case GQA_DTYPE_F32: return pick_dim<float, kGen>(kind, d, nw, v);
        case GQA_DTYPE_F16: return pick_dim<__half, kGen>(kind, d, nw, v);
        case GQA_DTYPE_BF16: return pick_dim<__nv_bfloat16, kGen>(kind, d, nw, v);
        case GQA_DTYPE_I8: return pick_dim<int8_t, kGen>(kind, d, nw, v);
        case GQA_DTYPE_FP8_E4M3: return pick_dim<__nv_fp8_e4m3, kGen>(kind, d, nw, v);
        case GQA_DTYPE_I4: return pick_dim<int4x2, kGen>(kind, d, nw, v);
        case GQA_DTYPE_I4_KC: return pick_dim<int4kc, kGen>(kind, d, nw, v);
        default: return false;
    }
}

// Defined in gqa_decode.cu (plain) and gqa_decode_general.cu (general).
bool pick_plain(int dtype, int kind, int d, int nw, Variant& v);
bool pick_general(int dtype, int kind, int d, int nw, Variant& v);

}  // namespace dec
}  // namespace gqa
