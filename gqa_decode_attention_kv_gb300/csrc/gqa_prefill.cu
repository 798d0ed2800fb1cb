// gqa_prefill.cu -- paged prefill attention: the n_b new tokens of every
// sequence attend, causally, to its whole paged cache (the new tokens'
// K/V already appended), "LLM 推理性能优化实战" sections 9.2-9.4: the query
// tile stays on chip while K/V blocks stream through it (FlashAttention-2
// ordering), the cache is read block by block through the block table, and
// the softmax is the online (m, l, o) recurrence of section 9.2.
//
// One CTA = one (query tile, kv-head g, sequence b). A tile holds 64 query
// rows, row = new token * G + head in group, so every K/V tile serves all G
// heads of the group (the GQA broadcast). Each warp owns 16 rows:
//   S[16 rows x 16 tokens] = Q K^T   (mma.sync m16n8k16, A = Q from registers,
//                                     B = K tile by ldmatrix)
//   O[16 rows x d]        += P V     (A = P straight from the S accumulators,
//                                     split in a high and a low 16-bit part;
//                                     B = V tile by ldmatrix.trans)
// K/V tiles arrive by TMA (4-D tensor map over the pool, 128-byte swizzle)
// in a ring of stages shared by the CTA's warps (full/empty mbarriers), one
// thread issuing. Tiles run heaviest first (the last query tiles of a
// sequence attend the most blocks).
#include <algorithm>
#include <type_traits>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

constexpr int kPfWarps = 4;                  // warps per CTA, 16 query rows each
constexpr int kPfRows = 16 * kPfWarps;       // query rows per tile
constexpr int kPfStages = 4;                 // ring stages (one 16-token block each)
constexpr float kLog2eP = 1.4426950408889634f;

struct PrefillArgs {
    const void* q;              // [total new tokens, H, D]
    const int32_t* q_start;     // [B + 1] first new-token row of each sequence
    const int32_t* block_tables;
    const int32_t* context_lens;  // [B], new tokens included
    void* out;                  // [total new tokens, H, D]
    int32_t* err;
    long long num_blocks;
    int B, H, K, G, max_blocks, out_dtype, tiles_per_seq, max_new, window;
    int map_perm[3];
    float scale_log2;
};

template <typename T, int D>
struct PfCfg {
    static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    static constexpr int kTile = 16 * D * 2;          // one (block, kv-head) tile of K or V
    static constexpr int kStage = 2 * kTile;          // K then V
    static constexpr int kNumBox = D * 2 / 128;       // 128-byte swizzled boxes per tile
    static constexpr int kBoxBytes = 16 * 128;
    static constexpr int kKs = D / 16;                // k-steps of Q.K^T
    static constexpr int kNd = D / 8;                 // n-tiles (8 dims) of P.V
    static constexpr int kSmem = 1024 + kPfStages * kStage + 16 * kPfStages + 16 * kPfStages;
};

template <bool kBf16>
__device__ __forceinline__ void mma_p(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                      uint32_t b0, uint32_t b1) {
    if constexpr (kBf16) mma_bf16(d, a0, a1, a2, a3, b0, b1);
    else mma_f16(d, a0, a1, a2, a3, b0, b1);
}

__device__ __forceinline__ void store2(void* out, int dt, long long idx, float x, float y) {
    if (dt == GQA_DTYPE_F32) {
        *reinterpret_cast<float2*>(static_cast<float*>(out) + idx) = make_float2(x, y);
    } else if (dt == GQA_DTYPE_BF16) {
        *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(out) + idx) = pack2<true>(x, y);
    } else {
        *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(out) + idx) = pack2<false>(x, y);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kPfWarps * 32)
prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const PrefillArgs a) {
    using C = PfCfg<T, D>;
    constexpr bool kB = C::kBf16;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (ring - raw);
    const uint32_t full0 = ring + kPfStages * C::kStage;
    const uint32_t empty0 = full0 + 8 * kPfStages;
    volatile int* skip_s = reinterpret_cast<volatile int*>(gbase + kPfStages * C::kStage + 16 * kPfStages);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, c = lane & 3;
    const int tile = a.tiles_per_seq - 1 - (int)blockIdx.x;    // heaviest first
    const int g = blockIdx.y, b = blockIdx.z;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    grid_dependency_wait();                    // the append before us wrote the new K/V
    launch_dependents();

    const int q0 = a.q_start[b];
    const int n = a.q_start[b + 1] - q0;
    const int L = a.context_lens[b];
    if (n < 0 || n > a.max_new || L < n || L > a.max_blocks * kBlock) {
        if (tile == 0 && g == 0 && threadIdx.x == 0) flag_error(a.err, GQA_DEVERR_CONTEXT_LEN);
        return;                                // uniform per CTA
    }
    const int rows = n * a.G;
    const int row0 = tile * kPfRows;
    if (row0 >= rows) return;                  // uniform per CTA
    const int base_pos = L - n;                // position of new token 0

    // blocks this tile attends: from the window start of its first row to the
    // block holding its last row's position
    const int tok_lo = row0 / a.G, tok_hi = min(rows - 1, row0 + kPfRows - 1) / a.G;
    const int att_lo = a.window > 0 ? max(0, base_pos + tok_lo - a.window + 1) : 0;
    const int jb_lo = att_lo / kBlock;
    const int jb_hi = (base_pos + tok_hi + kBlock) / kBlock;
    const int nblk = jb_hi - jb_lo;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kPfWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // ---- this warp's rows: wrow0 + r and wrow0 + r + 8
    const int wrow0 = row0 + warp * 16;
    const int rr0 = wrow0 + r, rr1 = wrow0 + r + 8;
    const bool live0 = rr0 < rows, live1 = rr1 < rows;
    const int tk0 = live0 ? rr0 / a.G : 0, tk1 = live1 ? rr1 / a.G : 0;
    // attended positions [lo, hi) of each row (empty for rows past the tile)
    const int hi0 = live0 ? base_pos + tk0 + 1 : 0, hi1 = live1 ? base_pos + tk1 + 1 : 0;
    const int lo0 = a.window > 0 ? hi0 - a.window : 0, lo1 = a.window > 0 ? hi1 - a.window : 0;
    // the warp's positions: a block inside [wlo_all, whi_all) needs no mask
    const int wtk_lo = min(wrow0, rows - 1) / a.G, wtk_hi = min(wrow0 + 15, rows - 1) / a.G;
    const bool warp_full_rows = wrow0 + 15 < rows;
    const int whi_all = base_pos + wtk_lo + 1;                               // min over rows of hi
    const int wlo_all = a.window > 0 ? base_pos + wtk_hi + 1 - a.window : 0;  // max over rows of lo

    // Q fragments (A operand, row-major 16 x 16 per k-step)
    uint32_t qf[C::kKs][4];
    {
        const uint16_t* qb = static_cast<const uint16_t*>(a.q);
        const long long ra = live0 ? ((long long)(q0 + tk0) * a.H + (long long)g * a.G + (rr0 - tk0 * a.G)) * D : -1;
        const long long rb = live1 ? ((long long)(q0 + tk1) * a.H + (long long)g * a.G + (rr1 - tk1 * a.G)) * D : -1;
#pragma unroll
        for (int ks = 0; ks < C::kKs; ++ks) {
            const int d0 = 16 * ks + 2 * c;
            qf[ks][0] = ra >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(qb + ra + d0)) : 0u;
            qf[ks][1] = rb >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(qb + rb + d0)) : 0u;
            qf[ks][2] = ra >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(qb + ra + d0 + 8)) : 0u;
            qf[ks][3] = rb >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(qb + rb + d0 + 8)) : 0u;
        }
    }

    float acc[C::kNd][4];
#pragma unroll
    for (int i = 0; i < C::kNd; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // ---- producer (warp 0): lane l holds the table entry of block win_base + l
    const uint64_t pol = l2_policy_evict_last();   // every query tile of the sequence re-reads these
    int win_base = -(1 << 30), win_phys = -1;
    auto issue = [&](int it) {                 // warp 0 only (warp-uniform)
        const int j = jb_lo + it;
        if (j - win_base >= 32 || j < win_base) {
            win_base = j;
            const int jj = j + lane;
            win_phys = -1;
            if (jj < jb_hi) {
                const int ph = a.block_tables[(long long)b * a.max_blocks + jj];
                if (ph < 0 || ph >= a.num_blocks) flag_error(a.err, GQA_DEVERR_BLOCK_INDEX);
                else win_phys = ph;
            }
        }
        const int ph = __shfl_sync(kFull, win_phys, j - win_base);
        if (lane == 0) {
            const int s = it % kPfStages;
            const uint32_t bar = full0 + 8 * s;
            if (ph < 0) {
                skip_s[s] = 1;
                mbar_arrive(bar);
            } else {
                skip_s[s] = 0;
                auto coord = [&](int which) { return which == 0 ? 0 : (which == 1 ? g : ph); };
                const int y = coord(a.map_perm[0]), z = coord(a.map_perm[1]), w = coord(a.map_perm[2]);
                const uint32_t dst = ring + s * C::kStage;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, 2 * C::kTile);
#pragma unroll
                for (int x = 0; x < C::kNumBox; ++x)
                    tma_load_4d(dst + x * C::kBoxBytes, &kmap, x * 64, y, z, w, bar, pol);
#pragma unroll
                for (int x = 0; x < C::kNumBox; ++x)
                    tma_load_4d(dst + C::kTile + x * C::kBoxBytes, &vmap, x * 64, y, z, w, bar, pol);
            }
        }
    };
    auto wait_all = [&](uint32_t bar, uint32_t parity) { return __all_sync(kFull, mbar_wait(bar, parity)); };
    int n_issued = 0;
    if (warp == 0)
        for (; n_issued < min(kPfStages, nblk); ++n_issued) issue(n_issued);

    const int mi = lane >> 3, rq = lane & 7;
    for (int it = 0; it < nblk; ++it) {
        const int s = it % kPfStages;
        const uint32_t par = (uint32_t)(it / kPfStages) & 1u;
        if (!wait_all(full0 + 8 * s, par)) {
            // a copy did not land in time: report, let this CTA's copies land, leave
            if (lane == 0) flag_error(a.err, GQA_DEVERR_TIMEOUT);
            if (warp == 0)
                for (int q = it; q < n_issued; ++q)
                    mbar_wait(full0 + 8 * (q % kPfStages), (uint32_t)(q / kPfStages) & 1u, kWaitLimitNs / 4);
            return;
        }
        const int j = jb_lo + it;
        const int bpos = j * kBlock;
        if (!skip_s[s]) {
            const uint32_t sk = ring + s * C::kStage, sv = sk + C::kTile;
            // ---- S = Q K^T for tokens 0-7 (sa) and 8-15 (sb)
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < C::kKs; ++ks) {
                uint32_t kb[4];
                ldsm_x4(swz(sk, rq + 8 * (mi >> 1), 2 * ks + (mi & 1)), kb);
                mma_p<kB>(sa, qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], kb[0], kb[1]);
                mma_p<kB>(sb, qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], kb[2], kb[3]);
            }
            // element e of row x: token bpos + 8*(e/2 ... ) -- sa[0..1] row r tokens 2c, 2c+1;
            // sa[2..3] row r+8; sb the same for tokens 8 + 2c, 8 + 2c + 1
            float s_[8] = {sa[0], sa[1], sb[0], sb[1], sa[2], sa[3], sb[2], sb[3]};
#pragma unroll
            for (int e = 0; e < 8; ++e) s_[e] *= a.scale_log2;
            const bool full = warp_full_rows && bpos >= wlo_all && bpos + kBlock <= whi_all;
            if (!full) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int tp = bpos + 2 * c + (e & 1) + 8 * ((e >> 1) & 1);
                    const bool row1 = e >= 4;
                    const int lo = row1 ? lo1 : lo0, hi = row1 ? hi1 : hi0;
                    if (tp < lo || tp >= hi) s_[e] = -INFINITY;
                }
            }
            // ---- online softmax per row (rows r: e 0..3, r+8: e 4..7)
            float mx0 = fmaxf(fmaxf(s_[0], s_[1]), fmaxf(s_[2], s_[3]));
            float mx1 = fmaxf(fmaxf(s_[4], s_[5]), fmaxf(s_[6], s_[7]));
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
            }
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            // rows that have attended nothing yet keep -inf: use 0 so p = 0, not NaN
            const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
            const float al0 = fast_exp2(m0 - u0), al1 = fast_exp2(m1 - u1);
            m0 = n0;
            m1 = n1;
            float p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) p[e] = fast_exp2(s_[e] - (e < 4 ? u0 : u1));
            l0 = l0 * al0 + (p[0] + p[1] + p[2] + p[3]);
            l1 = l1 * al1 + (p[4] + p[5] + p[6] + p[7]);
#pragma unroll
            for (int i = 0; i < C::kNd; ++i) {
                acc[i][0] *= al0; acc[i][1] *= al0; acc[i][2] *= al1; acc[i][3] *= al1;
            }
            // ---- P (A operand: rows r / r+8, tokens 2c.. / 2c+8..) high and low parts
            uint32_t ph[4], pl[4];
            const int order[4][2] = {{0, 1}, {4, 5}, {2, 3}, {6, 7}};   // a0 a1 a2 a3
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = p[order[q][0]], y = p[order[q][1]];
                ph[q] = pack2<kB>(x, y);
                const float2 f = unpack2<kB>(ph[q]);
                pl[q] = pack2<kB>(x - f.x, y - f.y);
            }
            // ---- O += P V; tokens past the sequence hold arbitrary bits: zero them
            const bool tail = bpos + kBlock > L;
            const uint32_t m01 = (bpos + 2 * c < L ? 0x0000ffffu : 0u) | (bpos + 2 * c + 1 < L ? 0xffff0000u : 0u);
            const uint32_t m89 = (bpos + 2 * c + 8 < L ? 0x0000ffffu : 0u) | (bpos + 2 * c + 9 < L ? 0xffff0000u : 0u);
#pragma unroll
            for (int pp = 0; pp < C::kNd / 2; ++pp) {
                uint32_t vb[4];
                ldsm_x4_t(swz(sv, rq + 8 * (mi & 1), 2 * pp + (mi >> 1)), vb);
                if (tail) {
                    vb[0] &= m01; vb[1] &= m89; vb[2] &= m01; vb[3] &= m89;
                }
                mma_p<kB>(acc[2 * pp], ph[0], ph[1], ph[2], ph[3], vb[0], vb[1]);
                mma_p<kB>(acc[2 * pp], pl[0], pl[1], pl[2], pl[3], vb[0], vb[1]);
                mma_p<kB>(acc[2 * pp + 1], ph[0], ph[1], ph[2], ph[3], vb[2], vb[3]);
                mma_p<kB>(acc[2 * pp + 1], pl[0], pl[1], pl[2], pl[3], vb[2], vb[3]);
            }
        }
        // ---- hand the stage back; warp 0 refills it once every warp has
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (warp == 0 && n_issued < nblk) {
            if (!wait_all(empty0 + 8 * s, par)) {
                if (lane == 0) flag_error(a.err, GQA_DEVERR_TIMEOUT);
                for (int q = it + 1; q < n_issued; ++q)
                    mbar_wait(full0 + 8 * (q % kPfStages), (uint32_t)(q / kPfStages) & 1u, kWaitLimitNs / 4);
                return;
            }
            issue(n_issued);
            ++n_issued;
        }
    }

    // ---- normalise and store rows r and r+8
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, o);
        l1 += __shfl_xor_sync(kFull, l1, o);
    }
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const long long oa = live0 ? ((long long)(q0 + tk0) * a.H + (long long)g * a.G + (rr0 - tk0 * a.G)) * D : -1;
    const long long ob = live1 ? ((long long)(q0 + tk1) * a.H + (long long)g * a.G + (rr1 - tk1 * a.G)) * D : -1;
#pragma unroll
    for (int i = 0; i < C::kNd; ++i) {
        const int dim = 8 * i + 2 * c;
        if (oa >= 0) store2(a.out, a.out_dtype, oa + dim, acc[i][0] * inv0, acc[i][1] * inv0);
        if (ob >= 0) store2(a.out, a.out_dtype, ob + dim, acc[i][2] * inv1, acc[i][3] * inv1);
    }
}

template <typename T, int D>
const void* prefill_fn() {
    return reinterpret_cast<const void*>(&prefill_kernel<T, D>);
}

}  // namespace

int launch_prefill(const PrefillLaunch& L) {
    const gqa_kv_cache_t& c = *L.cache;
    const int D = c.head_dim, K = c.num_kv_heads, G = L.num_heads / K;
    const void* fn = nullptr;
    int smem = 0;
    if (c.dtype == GQA_DTYPE_BF16) {
        fn = D == 64 ? prefill_fn<__nv_bfloat16, 64>() : prefill_fn<__nv_bfloat16, 128>();
        smem = D == 64 ? PfCfg<__nv_bfloat16, 64>::kSmem : PfCfg<__nv_bfloat16, 128>::kSmem;
    } else if (c.dtype == GQA_DTYPE_F16) {
        fn = D == 64 ? prefill_fn<__half, 64>() : prefill_fn<__half, 128>();
        smem = D == 64 ? PfCfg<__half, 64>::kSmem : PfCfg<__half, 128>::kSmem;
    } else {
        return GQA_ERR_UNSUPPORTED;
    }
    CUtensorMap kmap, vmap;
    int perm[3];
    if (!encode_cache_map(&kmap, c, c.k, 64, true, perm) || !encode_cache_map(&vmap, c, c.v, 64, true, perm))
        return GQA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GQA_ERR_CUDA;

    PrefillArgs a;
    a.q = L.q;
    a.q_start = L.q_start;
    a.block_tables = L.block_tables;
    a.context_lens = L.context_lens;
    a.out = L.out;
    a.err = L.err;
    a.num_blocks = c.num_blocks;
    a.B = L.batch;
    a.H = L.num_heads;
    a.K = K;
    a.G = G;
    a.max_blocks = L.max_blocks;
    a.out_dtype = L.out_dtype;
    a.max_new = L.max_new_tokens;
    a.tiles_per_seq = (int)(((long long)L.max_new_tokens * G + kPfRows - 1) / kPfRows);
    a.window = L.window;
    a.map_perm[0] = perm[0];
    a.map_perm[1] = perm[1];
    a.map_perm[2] = perm[2];
    a.scale_log2 = L.scale * kLog2eP;
    if (a.tiles_per_seq == 0) return GQA_OK;

    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.tiles_per_seq, (unsigned)K, (unsigned)L.batch);
    cfg.blockDim = dim3(kPfWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    void* args[] = {&kmap, &vmap, &a};
    return cudaLaunchKernelExC(&cfg, fn, args) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
