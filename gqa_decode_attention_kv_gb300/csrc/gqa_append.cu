// gqa_append.cu -- paged KV append: the K and V of every new token of every
// (sequence, kv-head) go to slot pos % 16 of block block_tables[b][pos / 16]
// ("LLM 推理性能优化实战", sections 5.3-5.4 and 8.2). One warp per
// (sequence, new token, kv-head) writes both rows, so K and V of a token leave
// together.
// For an int8, int4 or FP8 (e4m3) cache each row is quantised on the way (one
// fp16 scale per (token, kv-head); sections 15.1, 15.2 and 15.5 of that page).
// The KIVI-style 4-bit cache (section 15.5: K per channel, V per token) takes
// one warp per (sequence, kv-head) instead: every block the new tokens reach is
// re-quantised channel by channel over all the tokens it then holds.
#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

struct AppendArgs {
    void* k_cache;
    void* v_cache;
    __half* k_scale;
    __half* v_scale;
    const void* k_new;
    const void* v_new;
    const int32_t* block_tables;
    const int32_t* positions;
    const int32_t* token_start;   // NULL, or [batch+1] row offsets of k_new/v_new
    float* k_residual;            // KIVI-style cache: fp32 [rows, K, 16, d]
    int32_t* err;
    long long num_blocks;
    long long sb, sh, st;   // element strides of the cache
    int batch, T, K, d, max_blocks, es;
};

constexpr int kWarpsPerCta = 4;

// Warp `row` of the grid -> (b, i, g): sequence, new token, kv-head, and the
// source row of k_new/v_new; false when sequence b has fewer than i+1 tokens.
__device__ __forceinline__ bool row_of(const AppendArgs& a, long long row, int& b, int& i, int& g,
                                       long long& src_row) {
    g = (int)(row % a.K);
    const long long bi = row / a.K;
    i = (int)(bi % a.T);
    b = (int)(bi / a.T);
    if (a.token_start == nullptr) {
        src_row = row;
        return true;
    }
    const int t0 = a.token_start[b], n = a.token_start[b + 1] - t0;
    if (n < 0 || n > a.T) {
        if (i == 0 && g == 0 && (threadIdx.x & 31) == 0) flag_error(a.err, GQA_DEVERR_POSITION);
        return false;
    }
    src_row = ((long long)t0 + i) * a.K + g;
    return i < n;
}

// Resolve (b, token position, g) -> element offset of the destination row, or -1
// after flagging.
__device__ __forceinline__ long long dest_offset(const AppendArgs& a, int b, int pos, int g, int lane) {
    if (pos < 0 || pos >= a.max_blocks * kBlock) {
        if (lane == 0 && g == 0) flag_error(a.err, GQA_DEVERR_POSITION);
        return -1;
    }
    const int phys = a.block_tables[(long long)b * a.max_blocks + pos / kBlock];
    if (phys < 0 || phys >= a.num_blocks) {
        if (lane == 0 && g == 0) flag_error(a.err, GQA_DEVERR_BLOCK_INDEX);
        return -1;
    }
    return (long long)phys * a.sb + (long long)g * a.sh + (long long)(pos % kBlock) * a.st;
}

// Bit-exact copy for f32/f16/bf16 caches, 16 bytes per lane step.
__global__ void __launch_bounds__(kWarpsPerCta * 32) append_copy_kernel(const AppendArgs a) {
    grid_dependency_wait();
    launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (row >= (long long)a.batch * a.T * a.K) return;
    int b, i, g;
    long long srow;
    if (!row_of(a, row, b, i, g, srow)) return;
    const long long off = dest_offset(a, b, a.positions[b] + i, g, lane);
    if (off < 0) return;
    const int row_bytes = a.d * a.es;
    const int nvec = row_bytes / 16;                 // 16-byte vectors per row
    const long long src = srow * row_bytes;          // k_new/v_new rows of [*, K, d]
    for (int x = lane; x < 2 * nvec; x += 32) {
        const bool is_v = x >= nvec;
        const int vi = is_v ? x - nvec : x;
        const uint8_t* s = static_cast<const uint8_t*>(is_v ? a.v_new : a.k_new) + src + vi * 16;
        uint8_t* dptr = static_cast<uint8_t*>(is_v ? a.v_cache : a.k_cache) + off * a.es + vi * 16;
        *reinterpret_cast<uint4*>(dptr) = *reinterpret_cast<const uint4*>(s);
    }
}

template <typename In>
__device__ __forceinline__ float load_as_float(const void* p, long long i) {
    if constexpr (sizeof(In) == 4) return static_cast<const float*>(p)[i];
    else if constexpr (std::is_same<In, __half>::value) return __half2float(static_cast<const __half*>(p)[i]);
    else return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// Code formats of the quantising append.
enum CodeKind : int { kCodeI8 = 0, kCodeFp8 = 1, kCodeI4 = 2 };

// Quantise one row of d values held EPL per lane; writes codes and the scale.
// kFp8: e4m3 codes, s = amax/448, nearest-even with saturation to +-448;
// kI8: int8 codes, s = amax/127, rint with ties to even, clamped to +-127;
// kI4: the same with 7, two codes per byte (element 2j in the low nibble).
// dst is the row's first byte.
template <typename In, int EPL, int kCode>
__device__ __forceinline__ void quantise_row(const void* src, long long src_off, uint8_t* dst,
                                             __half* scale_dst, int lane) {
    constexpr bool kFp8 = kCode == kCodeFp8;
    constexpr float kQmax = kCode == kCodeI4 ? 7.0f : 127.0f;
    float x[EPL];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        x[e] = load_as_float<In>(src, src_off + lane * EPL + e);
        amax = fmaxf(amax, fabsf(x[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    float s32 = __fdiv_rn(amax, kFp8 ? 448.0f : kQmax);
    s32 = fminf(s32, 65504.0f);
    const __half sh = __float2half_rn(s32);
    const float sf = __half2float(sh);
    uint8_t codes[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        uint8_t q = 0;
        if (sf != 0.f) {
            const float t = __fdiv_rn(x[e], sf);
            if constexpr (kFp8) {
                q = (uint8_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
            } else {
                const int qm = (int)kQmax;
                q = (uint8_t)(int8_t)max(-qm, min(qm, __float2int_rn(t)));
            }
        }
        codes[e] = q;
    }
    if constexpr (kCode == kCodeI4) {
        // EPL (even) codes -> EPL/2 bytes at byte lane*EPL/2
#pragma unroll
        for (int e = 0; e < EPL; e += 2)
            dst[lane * (EPL / 2) + e / 2] = (uint8_t)((codes[e] & 0xF) | ((codes[e + 1] & 0xF) << 4));
    } else if constexpr (EPL % 4 == 0) {
#pragma unroll
        for (int w = 0; w < EPL / 4; ++w)
            reinterpret_cast<uint32_t*>(dst + lane * EPL)[w] =
                (uint32_t)codes[4 * w] | ((uint32_t)codes[4 * w + 1] << 8) |
                ((uint32_t)codes[4 * w + 2] << 16) | ((uint32_t)codes[4 * w + 3] << 24);
    } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) dst[lane * EPL + e] = codes[e];
    }
    if (lane == 0) *scale_dst = sh;
}

template <typename In, int EPL, int kCode>
__global__ void __launch_bounds__(kWarpsPerCta * 32) append_quant_kernel(const AppendArgs a) {
    grid_dependency_wait();
    launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (row >= (long long)a.batch * a.T * a.K) return;
    int b, i, g;
    long long srow;
    if (!row_of(a, row, b, i, g, srow)) return;
    const int pos = a.positions[b] + i;
    const long long off = dest_offset(a, b, pos, g, lane);
    if (off < 0) return;
    const int phys = a.block_tables[(long long)b * a.max_blocks + pos / kBlock];
    const long long sidx = ((long long)phys * a.K + g) * kBlock + pos % kBlock;
    const long long src = srow * a.d;
    const long long boff = kCode == kCodeI4 ? off / 2 : off;      // element -> byte offset
    quantise_row<In, EPL, kCode>(a.k_new, src, static_cast<uint8_t*>(a.k_cache) + boff, a.k_scale + sidx, lane);
    quantise_row<In, EPL, kCode>(a.v_new, src, static_cast<uint8_t*>(a.v_cache) + boff, a.v_scale + sidx, lane);
}

// KIVI-style cache, one warp per (sequence b, kv-head g); lane l owns the EPL
// channels EPL*l .. EPL*l+EPL-1, so a channel's amax, scale and codes stay in
// one lane and the slice of a residual row a lane reads is the slice it
// writes. The n new tokens of b sit at positions p0 .. p0+n-1. Each block
// they reach is taken whole: its slots before p0 from the residual row, the
// rest from k_new; per channel over its tend present tokens s_i =
// fp16(amax_i / 7) and code = clamp(rint(x / s_i), -7, 7) (fp32 IEEE
// division); codes of every present slot and the d scales are written, and
// the new rows of a block left unfinished go to the residual. V rows are
// quantised per token.
template <typename In, int EPL>
__global__ void __launch_bounds__(kWarpsPerCta * 32) append_kc_kernel(const AppendArgs a) {
    grid_dependency_wait();
    launch_dependents();
    constexpr int D = 32 * EPL;
    const int lane = threadIdx.x & 31;
    const long long pair = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (pair >= (long long)a.batch * a.K) return;
    const int b = (int)(pair / a.K), g = (int)(pair % a.K);
    const bool reporter = g == 0 && lane == 0;
    int n = a.T;
    long long t0 = (long long)b * a.T;                   // first source token of b
    if (a.token_start != nullptr) {
        t0 = a.token_start[b];
        n = a.token_start[b + 1] - (int)t0;
        if (n < 0 || n > a.T) {
            if (reporter) flag_error(a.err, GQA_DEVERR_POSITION);
            return;
        }
    }
    if (n == 0) return;
    const int p0 = a.positions[b];
    if (p0 < 0 || (long long)p0 + n > (long long)a.max_blocks * kBlock) {
        if (reporter) flag_error(a.err, GQA_DEVERR_POSITION);
        return;
    }
    float* res = a.k_residual + ((long long)b * a.K + g) * kBlock * D + lane * EPL;
    const int jb_end = (p0 + n - 1) / kBlock;
    for (int jb = p0 / kBlock; jb <= jb_end; ++jb) {
        const int first = jb * kBlock;
        const int tend = min((int)kBlock, p0 + n - first);
        const int ph = a.block_tables[(long long)b * a.max_blocks + jb];
        if (ph < 0 || ph >= a.num_blocks) {
            if (reporter) flag_error(a.err, GQA_DEVERR_BLOCK_INDEX);
            continue;
        }
        float x[kBlock][EPL];
        float amax[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) amax[e] = 0.f;
#pragma unroll
        for (int t = 0; t < kBlock; ++t) {
            if (t >= tend) break;
            const int p = first + t;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                x[t][e] = p < p0 ? res[t * D + e]
                                 : load_as_float<In>(a.k_new, ((t0 + p - p0) * a.K + g) * D + lane * EPL + e);
                amax[e] = fmaxf(amax[e], fabsf(x[t][e]));
            }
        }
        float sf[EPL];
        uint16_t sbits[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const __half sh = __float2half_rn(fminf(__fdiv_rn(amax[e], 7.0f), 65504.0f));
            sf[e] = __half2float(sh);
            sbits[e] = __half_as_ushort(sh);
        }
        __half* ks = a.k_scale + ((long long)ph * a.K + g) * D + lane * EPL;
        if constexpr (EPL == 4)
            *reinterpret_cast<uint2*>(ks) = make_uint2(sbits[0] | ((uint32_t)sbits[1] << 16),
                                                       sbits[2] | ((uint32_t)sbits[3] << 16));
        else
            *reinterpret_cast<uint32_t*>(ks) = sbits[0] | ((uint32_t)sbits[1] << 16);
        uint8_t* kb = static_cast<uint8_t*>(a.k_cache) + ((long long)ph * a.sb + (long long)g * a.sh) / 2 +
                      lane * (EPL / 2);
#pragma unroll
        for (int t = 0; t < kBlock; ++t) {
            if (t >= tend) break;
            uint32_t packed = 0;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const int q = sf[e] != 0.f ? max(-7, min(7, __float2int_rn(__fdiv_rn(x[t][e], sf[e])))) : 0;
                packed |= (uint32_t)(q & 0xF) << (4 * e);
            }
            uint8_t* row = kb + (long long)t * (a.st / 2);
            if constexpr (EPL == 4) *reinterpret_cast<uint16_t*>(row) = (uint16_t)packed;
            else *row = (uint8_t)packed;
            if (tend < kBlock && first + t >= p0) {       // the block stays unfinished: keep the row
#pragma unroll
                for (int e = 0; e < EPL; ++e) res[t * D + e] = x[t][e];
            }
        }
    }
    // V: per-token scale, the whole warp per row
    for (int i = 0; i < n; ++i) {
        const int pos = p0 + i;
        const int ph = a.block_tables[(long long)b * a.max_blocks + pos / kBlock];
        if (ph < 0 || ph >= a.num_blocks) continue;                        // flagged above
        const long long off = (long long)ph * a.sb + (long long)g * a.sh + (long long)(pos % kBlock) * a.st;
        quantise_row<In, EPL, kCodeI4>(a.v_new, ((t0 + i) * a.K + g) * D,
                                       static_cast<uint8_t*>(a.v_cache) + off / 2,
                                       a.v_scale + ((long long)ph * a.K + g) * kBlock + pos % kBlock, lane);
    }
}

template <int EPL>
const void* kc_kernel(int new_dtype) {
    switch (new_dtype) {
        case GQA_DTYPE_F32: return reinterpret_cast<const void*>(&append_kc_kernel<float, EPL>);
        case GQA_DTYPE_F16: return reinterpret_cast<const void*>(&append_kc_kernel<__half, EPL>);
        default: return reinterpret_cast<const void*>(&append_kc_kernel<__nv_bfloat16, EPL>);
    }
}

template <int kCode>
const void* quant_kernel(int new_dtype, bool d64) {
    switch (new_dtype) {
        case GQA_DTYPE_F32:
            return d64 ? reinterpret_cast<const void*>(&append_quant_kernel<float, 2, kCode>)
                       : reinterpret_cast<const void*>(&append_quant_kernel<float, 4, kCode>);
        case GQA_DTYPE_F16:
            return d64 ? reinterpret_cast<const void*>(&append_quant_kernel<__half, 2, kCode>)
                       : reinterpret_cast<const void*>(&append_quant_kernel<__half, 4, kCode>);
        default:
            return d64 ? reinterpret_cast<const void*>(&append_quant_kernel<__nv_bfloat16, 2, kCode>)
                       : reinterpret_cast<const void*>(&append_quant_kernel<__nv_bfloat16, 4, kCode>);
    }
}

}  // namespace

cudaError_t launch_kv_append(const gqa_kv_cache_t& c, const void* k_new, const void* v_new,
                             int new_dtype, const int32_t* block_tables, int max_blocks,
                             const int32_t* positions, int batch, int tokens_per_seq,
                             const int32_t* token_start, int32_t* err, cudaStream_t stream) {
    AppendArgs a;
    a.k_cache = c.k;
    a.v_cache = c.v;
    a.k_scale = static_cast<__half*>(c.k_scale);
    a.v_scale = static_cast<__half*>(c.v_scale);
    a.k_new = k_new;
    a.v_new = v_new;
    a.block_tables = block_tables;
    a.positions = positions;
    a.token_start = token_start;
    a.k_residual = static_cast<float*>(c.k_residual);
    a.err = err;
    a.num_blocks = c.num_blocks;
    a.sb = c.stride_block;
    a.sh = c.stride_head;
    a.st = c.stride_token;
    a.batch = batch;
    a.T = tokens_per_seq;
    a.K = c.num_kv_heads;
    a.d = c.head_dim;
    a.max_blocks = max_blocks;
    a.es = dtype_bits(c.dtype) / 8;             // bytes per element of the copy path
    const long long warps = (long long)batch * tokens_per_seq * c.num_kv_heads;
    int grid = (int)((warps + kWarpsPerCta - 1) / kWarpsPerCta);
    if (grid == 0) return cudaSuccess;
    const void* fn;
    if (c.dtype == GQA_DTYPE_I4_KC) {
        // one warp per (sequence, kv-head) instead of per row
        fn = a.d == 64 ? kc_kernel<2>(new_dtype) : kc_kernel<4>(new_dtype);
        grid = (int)(((long long)batch * c.num_kv_heads + kWarpsPerCta - 1) / kWarpsPerCta);
    } else if (c.dtype == GQA_DTYPE_I8) fn = quant_kernel<kCodeI8>(new_dtype, a.d == 64);
    else if (c.dtype == GQA_DTYPE_FP8_E4M3) fn = quant_kernel<kCodeFp8>(new_dtype, a.d == 64);
    else if (c.dtype == GQA_DTYPE_I4) fn = quant_kernel<kCodeI4>(new_dtype, a.d == 64);
    else fn = reinterpret_cast<const void*>(&append_copy_kernel);
    // programmatic serialisation: the kernel waits on the device for its predecessor
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kWarpsPerCta * 32);
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    void* args[] = {&a};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace gqa
