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
#include <cstring>
#include <type_traits>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

// Bulk tensor store of a shared-memory box to global through `map`, in this
// thread's bulk group; then the group's commit, and the waits for its reads of
// shared memory (the box may be rewritten) or for its completion.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

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
    int page_perm[2];           // tcgen05 kernel, d = 128: dims 3, 4 of the V page map
    int out_tma;                // 64-token tcgen05 forms: the output map is valid (fp32 out, G | 32 or 32 | G)
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

// Four consecutive outputs of a row.
__device__ __forceinline__ void store4(void* out, int dt, long long idx, float4 v) {
    if (dt == GQA_DTYPE_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = v;
    } else if (dt == GQA_DTYPE_BF16) {
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) =
            make_uint2(pack2<true>(v.x, v.y), pack2<true>(v.z, v.w));
    } else {
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) =
            make_uint2(pack2<false>(v.x, v.y), pack2<false>(v.z, v.w));
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

// ============================================================================
// The same prefill on the 5th-generation tensor cores (tcgen05.mma, fp32
// accumulators in tensor memory). One CTA = 128 query rows (the MMA M; one
// tensor-memory lane per row) of one (kv-head, sequence); the KV range goes by
// in chunks of 32 tokens (2 paged blocks):
//   S[128 x 32]  = Q[128 x d] K_chunk^T     A = Q from tensor memory (each row
//                                            thread writes its own), B = the
//                                            K-major 128-byte-swizzled K tile
//   softmax      one thread per row: tcgen05.ld of its 32 scores, mask, online
//                (m, l) with the lazy rescale; P as a high and a low 16-bit
//                part written to tensor memory with tcgen05.st
//   O[128 x d]  += P_hi V + P_lo V          A = P from tensor memory, B = the
//                                            V tiles read MN-major
// Tensor memory (256 columns): two 32-column S buffers, Q (d/2 columns), O (d).
// Warp roles: warps 0-3 own the 128 rows (Q, softmax, epilogue); warp 4 issues
// every MMA; warp 5 issues the K copies and warp 6 the V copies, so that K runs
// ahead of the P.V products (the copy engine takes ~100 ns a box). A K page is
// two 2 KB boxes (128-byte swizzle rows are half a row); a V page is one 4 KB
// box through a 5-D map that splits the row into two halves.
// The warps meet only on mbarriers: tcgen05.commit -> "S(c) done" and "P(c).V(c)
// done", each softmax warp -> "P(c) ready" and once "Q stored", TMA -> "K/V stage
// full", and a per-slot barrier that publishes which blocks of a chunk exist.
// Every per-chunk barrier comes in four copies taken in turn by chunk, so that
// no waiter can fall two phases behind one (a parity wait cannot tell those
// apart). P(c) is written over the S(c) it comes from (a row's scores are all
// in registers by then), so S(c+1) and P(c-1).V(c-1) run on the tensor cores
// while the softmax works on S(c): the MMA warp issues S(c+1) into P(c-1)'s
// buffer once P(c-1).V(c-1) has read it, before it waits for P(c). K and V have
// four shared stages each: K(c+4) loads once S(c) has read K(c), V(c+4) once
// P(c).V(c) has read V(c). The epilogue writes whole output rows through the
// idle shared stages. Two CTAs share an SM (~100 KB of shared memory and 256
// tensor-memory columns each).

constexpr int kTcRows = 128;                 // query rows per CTA = M = TMEM lanes
constexpr int kTcThreads = kTcRows + 96;     // + the MMA warp and the K and V copy warps
constexpr int kTcChunk = 32;                 // KV tokens per step = N of S = K of P.V
constexpr int kTcBlocks = kTcChunk / kBlock;
constexpr int kTcBufs = 4;                   // K and V stages, per-chunk barrier copies: c & 3
constexpr int kTcMasks = 8;                  // block-mask slots: chunk c uses c & 7
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColBuf = kTcChunk;       // S buffer b at columns [32b, 32b+32): S(c) in buffer
constexpr uint32_t kColPl = kTcChunk / 2;    // c & 1, then P(c) over it: high part +0, low part +16
constexpr uint32_t kColQ = 2 * kColBuf;      // Q: d 16-bit values per row, two per column
constexpr uint32_t kColO = 128;              // O: d fp32 columns
static_assert(kColQ + 64 <= kColO && kColO + 128 <= kTmemCols, "S, Q and O share the CTA's tensor-memory columns");
constexpr float kTcSlack = 8.f;              // log2 headroom before (m, l, O) are rescaled

template <typename T, int D>
struct TcCfg {
    static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    static constexpr int kHalves = D / 64;                      // 128-byte column halves of a row
    static constexpr int kQ = kTcRows * D * 2;                  // Q-sized area: epilogue staging
    static constexpr int kKc = kTcChunk * D * 2;                // K chunk: 32 rows per half
    static constexpr int kVb = kBlock * D * 2;                  // one block's V tile
    static constexpr int kVc = kTcBlocks * kVb;                 // V chunk
    static constexpr int kOffK = kQ, kOffV = kOffK + kTcBufs * kKc, kOffBar = kOffV + kTcBufs * kVc;
    static constexpr int kSmem = 1024 + kOffBar + 512;
    static_assert(4 * 32 * (D + 4) * 4 <= kOffBar, "the epilogue stages 4 warps x 32 padded rows below the barriers");
    static constexpr uint32_t kIdescS = mma_idesc_f16(kTcRows, kTcChunk, kBf16, false, false);
    static constexpr uint32_t kIdescO = mma_idesc_f16(kTcRows, D, kBf16, false, true);
};

// D[tmem] (+)= A[tmem] * B[smem], issued by one thread.
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 2)
prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const PrefillArgs a) {
    using C = TcCfg<T, D>;
    constexpr bool kB = C::kBf16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t* gb = smem_raw + (sb - raw);
    const uint32_t sK = sb + C::kOffK, sV = sb + C::kOffV;   // the Q stage only stages the epilogue
    // barriers (8 B each), every per-chunk one in four copies taken in turn by
    // chunk, so that no waiter can fall two phases behind one (event c is
    // completion c >> 2 of copy c & 3): K stage, V stage, "S(c) done", "P(c).V(c)
    // done", "P(c) ready"; then mask slots 0..7 (c & 7), the TMEM address and the
    // 8 block masks
    const uint32_t bar0 = sb + C::kOffBar;
    const uint32_t bar_q = bar0 + 224;         // "Q is in tensor memory": one arrival per softmax warp
    const uint32_t tslot = bar0 + 232;
    volatile uint32_t* cmask = reinterpret_cast<volatile uint32_t*>(gb + C::kOffBar + 236);   // [8]
    auto bar_k = [&](int c) { return bar0 + 8 * (c & 3); };
    auto bar_v = [&](int c) { return bar0 + 32 + 8 * (c & 3); };
    auto bar_s = [&](int c) { return bar0 + 64 + 8 * (c & 3); };
    auto bar_o = [&](int c) { return bar0 + 96 + 8 * (c & 3); };
    auto bar_p = [&](int c) { return bar0 + 128 + 8 * (c & 3); };
    auto bar_m = [&](int c) { return bar0 + 160 + 8 * (c & 7); };
    auto par4 = [](int c) { return (uint32_t)(c >> 2) & 1u; };
    auto par8 = [](int c) { return (uint32_t)(c >> 3) & 1u; };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool softmax = warp < 4, mma_warp = warp == 4, loader = warp >= 5;
    const int tile = a.tiles_per_seq - 1 - (int)blockIdx.x;    // heaviest first
    const int g = blockIdx.y, b = blockIdx.z;
    if (tid == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    grid_dependency_wait();
    launch_dependents();

    const int q0 = a.q_start[b];
    const int n = a.q_start[b + 1] - q0;
    const int L = a.context_lens[b];
    if (n < 0 || n > a.max_new || L < n || L > a.max_blocks * kBlock) {
        if (tile == 0 && g == 0 && tid == 0) flag_error(a.err, GQA_DEVERR_CONTEXT_LEN);
        return;                                // uniform per CTA, before any allocation
    }
    const int rows = n * a.G;
    const int row0 = tile * kTcRows;
    if (row0 >= rows) return;
    const int base_pos = L - n;
    const int tok_lo = row0 / a.G, tok_hi = min(rows - 1, row0 + kTcRows - 1) / a.G;
    const int att_lo = a.window > 0 ? max(0, base_pos + tok_lo - a.window + 1) : 0;
    const int jb_lo = att_lo / kBlock;
    const int jb_hi = (base_pos + tok_hi + kBlock) / kBlock;
    const int nchunks = (jb_hi - jb_lo + kTcBlocks - 1) / kTcBlocks;

    // ---- this thread's row (softmax warps) and the positions it attends, [lo, hi)
    const int rr = row0 + (softmax ? tid : 0);
    const bool live = softmax && rr < rows;
    const int tk = live ? rr / a.G : 0;
    const int hi = live ? base_pos + tk + 1 : 0;
    const int lo = a.window > 0 ? hi - a.window : 0;

    // This thread's Q row (rows past the prompt are zero), loaded now and
    // written to its tensor-memory lane once the columns are allocated: the S
    // products then read Q from tensor memory, not from shared memory.
    uint4 qv[D / 8];
    if (softmax) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                          ((long long)(q0 + tk) * a.H + (long long)g * a.G + (rr - tk * a.G)) * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) qv[i] = live ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid == 0) {
        for (int i = 0; i < 4 * kTcBufs; ++i) mbar_init(bar0 + 8 * i, 1);   // K, V, S done, P.V done
        for (int i = 0; i < kTcBufs; ++i) mbar_init(bar_p(i), 4);         // one arrival per softmax warp
        for (int i = 0; i < kTcMasks; ++i) mbar_init(bar_m(i), 1);
        mbar_init(bar_q, 4);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gb + (tslot - sb));
    bool ok = true;
    if (softmax) {
        const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16) + kColQ;
#pragma unroll
        for (int u = 0; u < D / 32; ++u) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w[4 * i] = qv[4 * u + i].x; w[4 * i + 1] = qv[4 * u + i].y;
                w[4 * i + 2] = qv[4 * u + i].z; w[4 * i + 3] = qv[4 * u + i].w;
            }
            tmem_st16(t_row + 16 * u, w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_q);
    }

    if (loader) {
        // ================================================== copy warps: 5 = K, 6 = V
        const bool k_warp = warp == 5;
        const uint64_t pol = l2_policy_evict_last();   // every query tile of the sequence re-reads them
        int win_base = -(1 << 30), win_phys = -1;
        int k_issued = 0, v_issued = 0;
        auto issue_kv = [&](int c, bool is_k) {
            int ph[kTcBlocks];
#pragma unroll
            for (int q = 0; q < kTcBlocks; ++q) {
                const int j = jb_lo + kTcBlocks * c + q;
                if (j - win_base >= 32 || j < win_base) {
                    win_base = j;
                    const int jj = j + lane;
                    win_phys = -1;
                    if (jj < jb_hi) {
                        const int p = a.block_tables[(long long)b * a.max_blocks + jj];
                        if (p < 0 || p >= a.num_blocks) flag_error(a.err, GQA_DEVERR_BLOCK_INDEX);
                        else win_phys = p;
                    }
                }
                ph[q] = __shfl_sync(kFull, win_phys, j - win_base);
                if (j >= jb_hi) ph[q] = -1;
            }
            const uint32_t bar = is_k ? bar_k(c) : bar_v(c);
            if (lane == 0) {
                uint32_t mask = 0;
                int nval = 0;
#pragma unroll
                for (int q = 0; q < kTcBlocks; ++q)
                    if (ph[q] >= 0) mask |= 1u << q, ++nval;
                if (is_k) {
                    cmask[c & (kTcMasks - 1)] = mask;
                    mbar_arrive(bar_m(c));     // publishes the mask (release)
                }
                mbar_arrive_expect_tx(bar, (uint32_t)(nval * C::kVb));
            }
            fence_proxy_async_smem();          // earlier generic writes to the stage come first
            __syncwarp();
            // one lane per (block, half) box
            if (!is_k && C::kHalves == 2) {
                // V: one box per page (the page map lands it as [half][slot][128 B])
                if (lane < kTcBlocks) {
                    int pq = ph[0];
#pragma unroll
                    for (int i = 1; i < kTcBlocks; ++i)
                        if (lane == i) pq = ph[i];
                    if (pq >= 0) {
                        auto coord = [&](int which) { return which == 1 ? g : pq; };
                        tma_load_5d(sV + (c & 3) * C::kVc + lane * C::kVb, &vmap, 0, 0, 0,
                                    coord(a.page_perm[0]), coord(a.page_perm[1]), bar, pol);
                    }
                }
            } else if (lane < kTcBlocks * C::kHalves) {
                const int q = lane / C::kHalves, h = lane % C::kHalves;
                int pq = ph[0];
#pragma unroll
                for (int i = 1; i < kTcBlocks; ++i)
                    if (q == i) pq = ph[i];
                if (pq >= 0) {
                    auto coord = [&](int which) { return which == 0 ? 0 : (which == 1 ? g : pq); };
                    const int y = coord(a.map_perm[0]), z = coord(a.map_perm[1]), w = coord(a.map_perm[2]);
                    const uint32_t base = is_k ? sK + (c & 3) * C::kKc : sV + (c & 3) * C::kVc;
                    const uint32_t dst = is_k ? base + h * (kTcChunk * 128) + q * (kBlock * 128)
                                              : base + q * C::kVb + h * (kBlock * 128);
                    tma_load_4d(dst, is_k ? &kmap : &vmap, h * 64, y, z, w, bar, pol);
                }
            }
            if (is_k) ++k_issued;
            else ++v_issued;
        };
        for (int c = 0; c < min(nchunks, kTcBufs); ++c) issue_kv(c, k_warp);
        for (int c = 0; c + kTcBufs < nchunks && ok; ++c) {
            // S(c) has read K(c): its stage takes K(c+4); P(c).V(c) has read V(c):
            // its stage takes V(c+4). Each tensor has its own warp, so that K runs
            // ahead of the P.V products.
            ok = __all_sync(kFull, mbar_wait(k_warp ? bar_s(c) : bar_o(c), par4(c)));
            if (!ok) break;
            issue_kv(c + kTcBufs, k_warp);
        }
        if (!ok && lane == 0) {
            // let this CTA's copies land before the shared memory goes
            flag_error(a.err, GQA_DEVERR_TIMEOUT);
            for (int c = max(0, k_issued - kTcBufs); c < k_issued; ++c) mbar_wait(bar_k(c), par4(c), kWaitLimitNs / 4);
            for (int c = max(0, v_issued - kTcBufs); c < v_issued; ++c) mbar_wait(bar_v(c), par4(c), kWaitLimitNs / 4);
        }
    } else if (mma_warp) {
        // ================================================== MMA warp
        auto issue_s = [&](int c) {            // S(c) = Q K(c)^T into buffer c & 1, Q from tensor memory
            const uint32_t kb = sK + (c & 3) * C::kKc;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t bd = smem_desc_sw128(kb + (ks >> 2) * (kTcChunk * 128) + (ks & 3) * 32, 16, 1024);
                tc_mma_f16_ta(tmem + (c & 1) * kColBuf, tmem + kColQ + 8 * ks, bd, C::kIdescS, ks > 0);
            }
        };
        int s_issued = 0, o_issued = 0;        // events committed (for the failure path)
        if (lane == 0) {
            ok = mbar_wait(bar_q, 0u) && mbar_wait(bar_k(0), par4(0));
            tc_fence_after();
            if (ok) issue_s(0);
            tc_commit(bar_s(0));               // S(0) done
            ++s_issued;
        }
        ok = __shfl_sync(kFull, ok, 0);
        for (int c = 0; c < nchunks && ok; ++c) {
            // S(c+1) first, so that it is ready when the softmax finishes S(c):
            // it goes over P(c-1), once P(c-1).V(c-1) has read it
            if (lane == 0 && c + 1 < nchunks) {
                bool w = c == 0 || mbar_wait(bar_o(c - 1), par4(c - 1));
                w = w && mbar_wait(bar_k(c + 1), par4(c + 1));
                tc_fence_after();
                if (w) issue_s(c + 1);
                tc_commit(bar_s(c + 1));
                ++s_issued;
                ok = w;
            }
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok) break;
            // P(c) written over S(c), V(c) rows zeroed by the softmax warps
            ok = __all_sync(kFull, mbar_wait(bar_p(c), par4(c)));
            if (!ok) break;
            if (lane == 0) {
                tc_fence_after();
                bool w = mbar_wait(bar_v(c), par4(c));
                if (w) {
                    const uint32_t vb = sV + (c & 3) * C::kVc;
                    const uint32_t pb = tmem + (c & 1) * kColBuf;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int jl = 0; jl < kTcBlocks; ++jl)
                            tc_mma_f16_ta(tmem + kColO, pb + (part ? kColPl : 0) + 8 * jl,
                                          smem_desc_sw128(vb + jl * C::kVb, kBlock * 128, 1024), C::kIdescO,
                                          !(c == 0 && part == 0 && jl == 0));
                    }
                }
                tc_commit(bar_o(c));           // P(c).V(c) done
                ++o_issued;
                ok = w;
            }
            ok = __shfl_sync(kFull, ok, 0);
        }
        if (!ok && lane == 0) {
            // let this CTA's MMAs land before the tensor memory goes, each
            // barrier's events in order
            flag_error(a.err, GQA_DEVERR_TIMEOUT);
            for (int k = max(0, s_issued - kTcBufs); k < s_issued; ++k) mbar_wait(bar_s(k), par4(k), kWaitLimitNs / 4);
            for (int k = max(0, o_issued - kTcBufs); k < o_issued; ++k) mbar_wait(bar_o(k), par4(k), kWaitLimitNs / 4);
        }
    } else {
        // ================================================== softmax warps: one row per thread
        const uint32_t t_lane = tmem + ((uint32_t)(32 * warp) << 16);
        float m = -INFINITY, l = 0.f;
        int c = 0;
        for (; c < nchunks; ++c) {
            ok = __all_sync(kFull, mbar_wait(bar_s(c), par4(c)));   // S(c) done
            ok = ok && __all_sync(kFull, mbar_wait(bar_m(c), par8(c)));
            if (!ok) break;
            tc_fence_after();
            const int cpos = (jb_lo + kTcBlocks * c) * kBlock;
            const uint32_t bm = cmask[c & (kTcMasks - 1)];
            const uint32_t t_buf = t_lane + (uint32_t)(c & 1) * kColBuf;
            float sv[kTcChunk];
            {
                uint32_t r[kTcChunk / 16][16];
#pragma unroll
                for (int u = 0; u < kTcChunk / 16; ++u) tmem_ld16(t_buf + 16 * u, r[u]);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < kTcChunk / 16; ++u)
#pragma unroll
                    for (int j = 0; j < 16; ++j) sv[16 * u + j] = __uint_as_float(r[u][j]) * a.scale_log2;
            }
            const bool whole = bm == (1u << kTcBlocks) - 1u && cpos >= lo && cpos + kTcChunk <= hi;
            if (!whole) {
#pragma unroll
                for (int j = 0; j < kTcChunk; ++j) {
                    const int pos = cpos + j;
                    if (!((bm >> (j / kBlock)) & 1u) || pos < lo || pos >= hi) sv[j] = -INFINITY;
                }
            }
            float mx4[4] = {sv[0], sv[1], sv[2], sv[3]};      // short chains
#pragma unroll
            for (int j = 4; j < kTcChunk; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], sv[j]);
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            // lazy rescale: keep the stale maximum while the new one stays within 2^slack
            const bool old_live = m != -INFINITY;
            const bool resc = mx > m + kTcSlack;
            float alpha = 1.f;
            if (resc) {
                alpha = old_live ? fast_exp2(m - mx) : 0.f;
                m = mx;
            }
            l *= alpha;
            if (c > 0 && __any_sync(kFull, resc && old_live)) {       // O holds earlier chunks: scale it
                // once P(c-1).V(c-1) has landed in it
                ok = __all_sync(kFull, mbar_wait(bar_o(c - 1), par4(c - 1)));
                if (!ok) break;
                tc_fence_after();
                const float f = (resc && old_live) ? alpha : 1.f;
#pragma unroll
                for (int q = 0; q < D / 16; ++q) {
                    uint32_t r16[16];
                    tmem_ld16(t_lane + kColO + 16 * q, r16);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) r16[j] = __float_as_uint(__uint_as_float(r16[j]) * f);
                    tmem_st16(t_lane + kColO + 16 * q, r16);
                }
            }
            const float mu = m == -INFINITY ? 0.f : m;    // a row with nothing attended yet: p = 0
            float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int hq = 0; hq < kTcChunk / 32; ++hq) {   // 32 tokens -> 16 packed columns each
                uint32_t ph16[16], pl16[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float x = fast_exp2(sv[32 * hq + 2 * e] - mu), y = fast_exp2(sv[32 * hq + 2 * e + 1] - mu);
                    ps4[e & 3] += x + y;
                    ph16[e] = pack2<kB>(x, y);
                    const float2 f = unpack2<kB>(ph16[e]);
                    pl16[e] = pack2<kB>(x - f.x, y - f.y);
                }
                tmem_st16(t_buf + 16 * hq, ph16);              // over this row's S(c)
                tmem_st16(t_buf + kColPl + 16 * hq, pl16);
            }
            tmem_wait_st();
            l += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
            // V rows of tokens outside the sequence or of missing blocks hold arbitrary bits
            if (bm != (1u << kTcBlocks) - 1u || cpos + kTcChunk > L) {
                ok = __all_sync(kFull, mbar_wait(bar_v(c), par4(c)));
                const uint32_t vb = sV + (c & 3) * C::kVc;
                for (int i = tid; i < kTcChunk * C::kHalves * 8; i += kTcRows) {
                    const int t = i / (C::kHalves * 8), h = (i / 8) % C::kHalves, ck = i % 8;
                    if (((bm >> (t / kBlock)) & 1u) && cpos + t < L) continue;
                    sts128(vb + (t / kBlock) * C::kVb + h * (kBlock * 128) + (t % kBlock) * 128 + ck * 16,
                           make_uint4(0u, 0u, 0u, 0u));
                }
                fence_proxy_async_smem();      // zeroed V visible to the tensor core (the
                                               // producer reads it after every warp's arrival)
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p(c));
            if (!ok) break;
        }
        // ---- wait for the last MMAs, then normalise and store this row
        // the last P.V (P(n-5).V(n-5), the previous event on its barrier, landed
        // before S(n-1) was issued)
        if (ok) ok = __all_sync(kFull, mbar_wait(bar_o(nchunks - 1), par4(nchunks - 1)));
        tc_fence_after();
        if (ok) {
            // This warp's 32 rows leave through shared memory (the staging area
            // and the K/V stages are idle now: every copy has landed and every
            // MMA is done),
            // so that each store writes whole rows: one lane per 4 dims of a row.
            const float inv = l > 0.f ? 1.f / l : 0.f;
            constexpr int kRowF = D + 4;       // padded row: 16-byte stores stay conflict-free
            float* stage = reinterpret_cast<float*>(gb) + warp * 32 * kRowF;
#pragma unroll
            for (int q = 0; q < D / 16; ++q) {
                uint32_t r16[16];
                tmem_ld16(t_lane + kColO + 16 * q, r16);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4*>(stage + lane * kRowF + 16 * q + j) =
                        make_float4(__uint_as_float(r16[j]) * inv, __uint_as_float(r16[j + 1]) * inv,
                                    __uint_as_float(r16[j + 2]) * inv, __uint_as_float(r16[j + 3]) * inv);
            }
            __syncwarp();
            int tkr = (row0 + 32 * warp) / a.G, hr = (row0 + 32 * warp) - tkr * a.G;   // token, head of row r
            for (int r = 0; r < 32; ++r) {
                if (row0 + 32 * warp + r >= rows) break;
                if (4 * lane < D) {
                    const long long orow = ((long long)(q0 + tkr) * a.H + (long long)g * a.G + hr) * D;
                    store4(a.out, a.out_dtype, orow + 4 * lane,
                           *reinterpret_cast<const float4*>(stage + r * kRowF + 4 * lane));
                }
                if (++hr == a.G) {
                    hr = 0;
                    ++tkr;
                }
            }
        } else if (lane == 0) {
            flag_error(a.err, GQA_DEVERR_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ============================================================================
// Wide form of the tcgen05 prefill (head_dim 128): one CTA per SM holds two
// 128-row query tiles of one (kv-head, sequence) -- 256 consecutive rows --
// that both read every K/V chunk of 64 tokens (4 paged blocks), so K/V tiles
// are copied once per 256 rows and each S product is 128 x 64. The SM's 512
// tensor-memory columns hold, per tile t, two S buffers at columns 256t and
// 256t + 64 (S(c) in buffer c & 1, P(c) written over it) and O at 256t + 128:
//   S_t(c) = Q_t K(c)^T     A = Q_t from shared memory (K-major, 128-byte swizzle)
//   softmax of tile t       one thread per row: its 64 scores in registers in
//                           one tensor-memory round trip; P as a high and a low
//                           16-bit part over the same columns
//   O_t   += P_t(c) V(c)    A = P from tensor memory, B = V pages MN-major
// Each tile has its own MMA warp, which issues S_t(0..1) and then per chunk
// PV_t(c), S_t(c+2). Products into different accumulators are not ordered by
// issue alone, so S_t(c+2) goes over P_t(c) only once PV_t(c)'s commit says it
// has read it; S_t(c+1) is then ready when tile t's softmax finishes chunk c
// (it was issued one chunk earlier). A single issuing thread gets about one
// tcgen05.mma per ~100 cycles through, whatever the shape; M=128 products of
// N <= 128 finish faster than that, so one issuer per tile doubles the rate at
// which the SM's tensor core is fed. Warps 0-3 own tile 0's rows, 4-7 tile
// 1's, 8 and 9 issue tile 0's and tile 1's MMAs, 10 copies K and 11 copies V
// (four 16 KB stages each). Per-chunk barriers (stages, S done, P ready, P.V done)
// come in four copies taken in turn by chunk and the block masks in eight, so
// that no parity wait can fall two phases behind (as in the 32-token kernel).
// 16-byte cp.async into shared memory; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Packed fp32 pairs (one 64-bit register pair): add, subtract and multiply
// both halves in one instruction, each half rounded to nearest like the scalar
// operation; and the three-input maximum. They halve the softmax's arithmetic
// instruction count per score.
__device__ __forceinline__ uint64_t f2_make(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

constexpr int kW2Chunk = 64;                     // KV tokens per chunk: N of S, K of P.V
constexpr int kW2Blocks = kW2Chunk / kBlock;
constexpr int kW2Bufs = 4;                       // per-chunk barrier copies (c & 3)
constexpr uint32_t kW2ColTile = 256;             // tile t: S buffers at 256t, 256t + 64
constexpr uint32_t kW2ColO = 128;                //         O at 256t + 128

// kTiles query tiles of 128 rows per CTA. Two tiles: one CTA per SM (512
// tensor-memory columns, four K and four V stages). One tile: two CTAs per SM
// (256 columns, two stages each, ~108 KB of shared memory). Either way the CTAs
// are persistent: each walks its share of the (query tile, kv-head, sequence)
// items, and the next item's Q load and first S products run while the softmax
// warps store the last item's output.
template <int kTiles>
struct W2Cfg {
    static constexpr int D = 128;
    static constexpr int kRows = kTiles * kTcRows;       // query rows per CTA
    static constexpr int kSoftWarps = 4 * kTiles;
    static constexpr int kThreads = kRows + 32 * kTiles + 64;   // + an MMA warp per tile, K and V copy warps
    static constexpr int kStages = kTiles == 2 ? 4 : 2;  // K and V stages
    static constexpr int kCtasPerSm = kTiles == 2 ? 1 : 2;
    static constexpr uint32_t kTmemCols = 256u * kTiles;
    static constexpr int kQt = kTcRows * D * 2;          // one Q tile: 2 halves x 128 rows x 128 B
    static constexpr int kKc = kW2Chunk * D * 2;         // K chunk: 2 halves x 64 rows x 128 B
    static constexpr int kVb = kBlock * D * 2;           // one V page
    static constexpr int kVc = kW2Blocks * kVb;          // V chunk
    static constexpr int kStgRowF = 20;                  // output staging: 16 columns + 4 pad per row
    static constexpr int kOffQ = 0, kOffK = kTiles * kQt, kOffV = kOffK + kStages * kKc,
                         kOffStg = kOffV + kStages * kVc, kOffBar = kOffStg + kSoftWarps * 32 * kStgRowF * 4;
    static constexpr int kSmem = 1024 + kOffBar + 512;
    static_assert(kSmem * kCtasPerSm <= 227 * 1024, "CTAs per SM fit the shared memory");
};

template <typename T, int kTiles>
__global__ void __launch_bounds__(W2Cfg<kTiles>::kThreads, W2Cfg<kTiles>::kCtasPerSm)
prefill_tc2_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap omap, const PrefillArgs a) {
    using C = W2Cfg<kTiles>;
    constexpr int kS = C::kStages;
    constexpr int D = C::D;
    constexpr bool kB = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdescS = mma_idesc_f16(kTcRows, kW2Chunk, kB, false, false);
    constexpr uint32_t kIdescO = mma_idesc_f16(kTcRows, D, kB, false, true);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t* gb = smem_raw + (sb - raw);
    const uint32_t sQ = sb + C::kOffQ, sK = sb + C::kOffK, sV = sb + C::kOffV;
    // barriers, 8 B each: K stages, V stages (stage G % kS), then per tile t
    // "S_t(G) done", "P_t(G).V(G) done", "P_t(G) ready" (copy G & 3); then the
    // block-mask slots (G & 7), the TMEM address, the masks and per tile "Q_t
    // stored". G counts the CTA's chunks across its items.
    const uint32_t bar0 = sb + C::kOffBar;
    auto stage = [](int c) { return c % kS; };
    auto par_st = [](int c) { return (uint32_t)(c / kS) & 1u; };
    auto bar_k = [&](int c) { return bar0 + 8 * stage(c); };
    auto bar_v = [&](int c) { return bar0 + 32 + 8 * stage(c); };
    auto bar_s = [&](int t, int c) { return bar0 + 64 + 96 * t + 8 * (c & 3); };
    auto bar_o = [&](int t, int c) { return bar0 + 96 + 96 * t + 8 * (c & 3); };
    auto bar_p = [&](int t, int c) { return bar0 + 128 + 96 * t + 8 * (c & 3); };
    auto bar_m = [&](int c) { return bar0 + 256 + 8 * (c & 7); };
    auto bar_q = [&](int t) { return bar0 + 320 + 8 * t; };
    const uint32_t tslot = bar0 + 336;
    volatile uint32_t* cmask = reinterpret_cast<volatile uint32_t*>(gb + C::kOffBar + 344);   // [8]
    auto par4 = [](int c) { return (uint32_t)(c >> 2) & 1u; };
    auto par8 = [](int c) { return (uint32_t)(c >> 3) & 1u; };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool softmax = warp < C::kSoftWarps, loader = warp >= C::kSoftWarps + kTiles;
    const bool mma_warp = !softmax && !loader;
    const int tt = warp >> 2;                                   // softmax warps: their tile
    if (tid == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        if (a.out_tma) prefetch_tensormap(&omap);
    }

    // ---- the CTA's items: (query tile, kv-head, sequence). The (kv-head,
    // sequence) groups go in sets of about eight rounds' worth of items, so that
    // only a set's K/V need to stay in L2; within a set the heaviest tiles come
    // first. (Sets of three rounds read K/V once but lose ~7% to the load
    // imbalance at each set's end; eight rounds lose ~1%.) Items are dealt to the CTAs in snake order (round r goes left
    // to right when r is even, right to left when odd) so each CTA's total stays
    // close to the others'.
    struct Item {
        int g, b, q0, n, L, rows, row0, base_pos, jb_lo, jb_hi, nchunks;
    };
    const int tps = a.tiles_per_seq, n_groups = a.K * a.B;
    const int n_items = tps * n_groups;
    const int P = (int)gridDim.x, j = (int)blockIdx.x;
    const int gps = min(n_groups, max(1, (8 * P + tps - 1) / tps));   // groups per set: ~8 rounds of items
    auto item_at = [&](int i, Item& it) -> bool {    // false: nothing to do
        const int set = i / (gps * tps), w = i - set * gps * tps;
        const int g0 = set * gps, gn = min(gps, n_groups - g0);
        const int level = w / gn, grp = g0 + (w - level * gn);
        it.b = grp / a.K;
        it.g = grp - it.b * a.K;
        const int tile = tps - 1 - level;
        it.q0 = a.q_start[it.b];
        it.n = a.q_start[it.b + 1] - it.q0;
        it.L = a.context_lens[it.b];
        if (it.n < 0 || it.n > a.max_new || it.L < it.n || it.L > a.max_blocks * kBlock) {
            if (tile == 0 && it.g == 0 && tid == 0) flag_error(a.err, GQA_DEVERR_CONTEXT_LEN);
            return false;
        }
        it.rows = it.n * a.G;
        it.row0 = tile * C::kRows;
        if (it.row0 >= it.rows) return false;
        it.base_pos = it.L - it.n;
        const int tok_lo = it.row0 / a.G, tok_hi = min(it.rows - 1, it.row0 + C::kRows - 1) / a.G;
        const int att_lo = a.window > 0 ? max(0, it.base_pos + tok_lo - a.window + 1) : 0;
        it.jb_lo = att_lo / kBlock;
        it.jb_hi = (it.base_pos + tok_hi + kBlock) / kBlock;
        it.nchunks = (it.jb_hi - it.jb_lo + kW2Blocks - 1) / kW2Blocks;
        return true;
    };
    auto next_item = [&](int& r, Item& it) -> bool {  // the next valid item from round r on
        for (;;) {
            const int base = r * P;
            if (base >= n_items) return false;
            const int i = base + ((r & 1) ? P - 1 - j : j);
            ++r;
            if (i < n_items && item_at(i, it)) return true;
        }
    };

    grid_dependency_wait();
    launch_dependents();
    if (tid == 0) {
        for (int i = 0; i < kS; ++i) {
            mbar_init(bar_k(i), 1);            // K, V stages
            mbar_init(bar_v(i), 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            for (int i = 0; i < kW2Bufs; ++i) {
                mbar_init(bar_s(t, i), 1);
                mbar_init(bar_o(t, i), 1);
                mbar_init(bar_p(t, i), 4);     // one arrival per softmax warp of the tile
            }
            mbar_init(bar_q(t), 4);
        }
        for (int i = 0; i < 8; ++i) mbar_init(bar_m(i), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gb + (tslot - sb));
    bool ok = true;
    int round = 0;
    Item it;
    bool have = next_item(round, it);

    if (loader) {
        // ================================================== copy warps: K, then V
        const bool k_warp = warp == C::kSoftWarps + kTiles;
        const uint64_t pol = l2_policy_evict_last();   // every query tile of the sequence re-reads them
        int issued = 0, gc = 0;
        while (have && ok) {
            int win_base = -(1 << 30), win_phys = -1;
            for (int c = 0; c < it.nchunks && ok; ++c) {
                const int G = gc + c;
                if (G >= kS) {
                    // K(G) once every tile's S(G-kS) has read K(G-kS); V(G) once
                    // every tile's P(G-kS).V(G-kS) has read V(G-kS)
                    bool w = true;
#pragma unroll
                    for (int t = 0; t < kTiles; ++t)
                        w = w && mbar_wait(k_warp ? bar_s(t, G - kS) : bar_o(t, G - kS), par4(G - kS));
                    ok = __all_sync(kFull, w);
                    if (!ok) break;
                }
                int ph[kW2Blocks];
#pragma unroll
                for (int q = 0; q < kW2Blocks; ++q) {
                    const int jb = it.jb_lo + kW2Blocks * c + q;
                    if (jb - win_base >= 32 || jb < win_base) {
                        win_base = jb;
                        const int jj = jb + lane;
                        win_phys = -1;
                        if (jj < it.jb_hi) {
                            const int p = a.block_tables[(long long)it.b * a.max_blocks + jj];
                            if (p < 0 || p >= a.num_blocks) flag_error(a.err, GQA_DEVERR_BLOCK_INDEX);
                            else win_phys = p;
                        }
                    }
                    ph[q] = __shfl_sync(kFull, win_phys, jb - win_base);
                    if (jb >= it.jb_hi) ph[q] = -1;
                }
                const uint32_t bar = k_warp ? bar_k(G) : bar_v(G);
                if (lane == 0) {
                    uint32_t mask = 0;
                    int nval = 0;
#pragma unroll
                    for (int q = 0; q < kW2Blocks; ++q)
                        if (ph[q] >= 0) mask |= 1u << q, ++nval;
                    if (k_warp) {
                        cmask[G & 7] = mask;
                        mbar_arrive(bar_m(G));     // publishes the mask (release)
                    }
                    mbar_arrive_expect_tx(bar, (uint32_t)(nval * C::kVb));
                }
                fence_proxy_async_smem();          // earlier generic writes to the stage come first
                __syncwarp();
                if (!k_warp) {
                    // V: one box per page (the page map lands it as [half][slot][128 B])
                    if (lane < kW2Blocks) {
                        int pq = ph[0];
#pragma unroll
                        for (int i = 1; i < kW2Blocks; ++i)
                            if (lane == i) pq = ph[i];
                        if (pq >= 0) {
                            auto coord = [&](int which) { return which == 1 ? it.g : pq; };
                            tma_load_5d(sV + stage(G) * C::kVc + lane * C::kVb, &vmap, 0, 0, 0,
                                        coord(a.page_perm[0]), coord(a.page_perm[1]), bar, pol);
                        }
                    }
                } else if (lane < 2 * kW2Blocks) {
                    // K: one lane per (block, 64-element half) box
                    const int q = lane >> 1, h = lane & 1;
                    int pq = ph[0];
#pragma unroll
                    for (int i = 1; i < kW2Blocks; ++i)
                        if (q == i) pq = ph[i];
                    if (pq >= 0) {
                        auto coord = [&](int which) { return which == 0 ? 0 : (which == 1 ? it.g : pq); };
                        const int y = coord(a.map_perm[0]), z = coord(a.map_perm[1]), w = coord(a.map_perm[2]);
                        tma_load_4d(sK + stage(G) * C::kKc + h * (kW2Chunk * 128) + q * (kBlock * 128), &kmap,
                                    h * 64, y, z, w, bar, pol);
                    }
                }
                ++issued;
            }
            gc += it.nchunks;
            have = next_item(round, it);
        }
        if (!ok && lane == 0) {
            // let this CTA's copies land before the shared memory goes
            flag_error(a.err, GQA_DEVERR_TIMEOUT);
            for (int c = max(0, issued - kS); c < issued; ++c)
                mbar_wait(k_warp ? bar_k(c) : bar_v(c), par_st(c), kWaitLimitNs / 4);
        }
    } else if (mma_warp) {
        // ================================================== MMA warps: one per tile (one lane issues)
        const int t = warp - C::kSoftWarps;
        if (lane == 0) {
            auto issue_s = [&](int G) {            // S_t(G) = Q_t K(G)^T into buffer G & 1
                const uint32_t kb = sK + stage(G) * C::kKc, qb = sQ + t * C::kQt;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t ad = smem_desc_sw128(qb + (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(kb + (ks >> 2) * (kW2Chunk * 128) + (ks & 3) * 32, 16, 1024);
                    tc_mma_f16(tmem + kW2ColTile * t + kW2Chunk * (G & 1), ad, bd, kIdescS, ks > 0);
                }
            };
            auto issue_pv = [&](int G, bool first) {   // O_t (+)= P_t(G) V(G), high part then low part per block
                const uint32_t vb = sV + stage(G) * C::kVc, pb = tmem + kW2ColTile * t + kW2Chunk * (G & 1);
#pragma unroll
                for (int jl = 0; jl < kW2Blocks; ++jl)
#pragma unroll
                    for (int part = 0; part < 2; ++part)
                        tc_mma_f16_ta(tmem + kW2ColTile * t + kW2ColO, pb + 16 * jl + 8 * part,
                                      smem_desc_sw128(vb + jl * C::kVb, kBlock * 128, 1024), kIdescO,
                                      !(first && jl == 0 && part == 0));
            };
            int s_done = 0, o_done = 0, gc = 0, qi = 0;   // commits issued (failure path), chunks, items
            while (have && ok) {
                // Q_t of this item stored; the previous item's last P.V done, so
                // both S buffers are free (its commit covers every earlier product)
                ok = mbar_wait(bar_q(t), (uint32_t)qi & 1u);
                ++qi;
                if (ok && gc > 0) ok = mbar_wait(bar_o(t, gc - 1), par4(gc - 1));
                for (int c = 0; c < min(it.nchunks, 2) && ok; ++c) {
                    ok = mbar_wait(bar_k(gc + c), par_st(gc + c));
                    tc_fence_after();
                    if (!ok) break;
                    issue_s(gc + c);
                    tc_commit(bar_s(t, gc + c));
                    ++s_done;
                }
                for (int c = 0; c < it.nchunks && ok; ++c) {
                    const int G = gc + c;
                    // P_t(G) written over S_t(G); V(G) rows of missing tokens zeroed by tile t's softmax
                    ok = mbar_wait(bar_p(t, G), par4(G)) && mbar_wait(bar_v(G), par_st(G));
                    tc_fence_after();
                    if (!ok) break;
                    issue_pv(G, c == 0);
                    tc_commit(bar_o(t, G));
                    ++o_done;
                    if (c + 2 < it.nchunks) {
                        // S_t(G+2) overwrites P_t(G): wait until PV_t(G) has read it
                        ok = mbar_wait(bar_o(t, G), par4(G)) && mbar_wait(bar_k(G + 2), par_st(G + 2));
                        tc_fence_after();
                        if (!ok) break;
                        issue_s(G + 2);
                        tc_commit(bar_s(t, G + 2));
                        ++s_done;
                    }
                }
                gc += it.nchunks;
                if (ok) have = next_item(round, it);
            }
            if (!ok) {
                // let this tile's MMAs land before the tensor memory goes, each
                // barrier's events in order
                flag_error(a.err, GQA_DEVERR_TIMEOUT);
                for (int k = max(0, s_done - kW2Bufs); k < s_done; ++k)
                    mbar_wait(bar_s(t, k), par4(k), kWaitLimitNs / 4);
                for (int k = max(0, o_done - kW2Bufs); k < o_done; ++k)
                    mbar_wait(bar_o(t, k), par4(k), kWaitLimitNs / 4);
            }
        }
        __syncwarp();
    } else {
        // ================================================== softmax warps: one row per thread
        const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kW2ColTile * tt;
        const uint32_t t_o = t_lane + kW2ColO;
        const uint32_t qt = sQ + tt * C::kQt;
        float* stg = reinterpret_cast<float*>(gb + C::kOffStg) + (warp * 32) * C::kStgRowF;
        // This warp's 32 Q rows of item x into its tile's swizzled K-major
        // layout by cp.async (16 lanes per row, 16 bytes each; rows past the
        // prompt are zero-filled), then "Q_t stored" once they have landed.
        auto load_q = [&](const Item& x) {
            constexpr int kLanesPerRow = D / 8, kRowsPerStep = 32 / kLanesPerRow, kSteps = 32 / kRowsPerStep;
            const int c16 = lane % kLanesPerRow;
            const int rl0 = 32 * (warp & 3) + lane / kLanesPerRow;
            const int rq0 = x.row0 + 128 * tt + rl0;
            int tq = rq0 / a.G, hq = rq0 - tq * a.G;
#pragma unroll
            for (int i = 0; i < kSteps; ++i) {
                const int rl = rl0 + i * kRowsPerStep, rq = rq0 + i * kRowsPerStep;
                const bool in = rq < x.rows;
                const long long src = in ? ((long long)(x.q0 + tq) * a.H + (long long)x.g * a.G + hq) * D + 8 * c16 : 0;
                cp_async16(qt + (c16 >> 3) * (kTcRows * 128) + rl * 128 + (((c16 & 7) ^ (rl & 7)) << 4),
                           static_cast<const uint16_t*>(a.q) + src, in ? 16u : 0u);
                hq += kRowsPerStep;
                while (hq >= a.G) {
                    hq -= a.G;
                    ++tq;
                }
            }
        };
        auto q_stored = [&]() {
            cp_async_wait_all();
            fence_proxy_async_smem();          // Q visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q(tt));
        };
        if (have) {
            load_q(it);
            q_stored();
        }
        int gc = 0;
        while (have && ok) {
            Item nx;
            int round_nx = round;
            const bool have_nx = next_item(round_nx, nx);
            // ---- this thread's row and the positions it attends, [lo, hi)
            const int rr = it.row0 + tid;      // tid = 128 t + row of tile t
            const bool live = rr < it.rows;
            const int tk = live ? rr / a.G : 0;
            const int hi = live ? it.base_pos + tk + 1 : 0;
            const int lo = a.window > 0 ? hi - a.window : 0;
            float m = -INFINITY, l = 0.f;
            for (int c = 0; c < it.nchunks; ++c) {
                const int G = gc + c;
                ok = __all_sync(kFull, mbar_wait(bar_s(tt, G), par4(G)));   // S_t(G) done
                ok = ok && __all_sync(kFull, mbar_wait(bar_m(G), par8(G)));
                if (!ok) break;
                tc_fence_after();
                const int cpos = (it.jb_lo + kW2Blocks * c) * kBlock;
                const uint32_t bm = cmask[G & 7];
                const uint32_t t_buf = t_lane + kW2Chunk * (G & 1);
                float sv[kW2Chunk];
                {
                    uint32_t r[kW2Chunk / 16][16];
#pragma unroll
                    for (int u = 0; u < kW2Chunk / 16; ++u) tmem_ld16(t_buf + 16 * u, r[u]);
                    tmem_wait_ld();
                    const uint64_t sc2 = f2_make(a.scale_log2, a.scale_log2);
#pragma unroll
                    for (int u = 0; u < kW2Chunk / 16; ++u)
#pragma unroll
                        for (int q = 0; q < 16; q += 2) {
                            const float2 v = f2_split(f2_mul(f2_make(__uint_as_float(r[u][q]), __uint_as_float(r[u][q + 1])), sc2));
                            sv[16 * u + q] = v.x;
                            sv[16 * u + q + 1] = v.y;
                        }
                }
                // the item's last S_t is in registers, and with it every S_t of the
                // item is done: Q_t's buffer is free for the next item's rows
                if (c == it.nchunks - 1 && have_nx) load_q(nx);
                const bool whole = bm == (1u << kW2Blocks) - 1u && cpos >= lo && cpos + kW2Chunk <= hi;
                if (!whole) {
#pragma unroll
                    for (int q = 0; q < kW2Chunk; ++q) {
                        const int pos = cpos + q;
                        if (!((bm >> (q / kBlock)) & 1u) || pos < lo || pos >= hi) sv[q] = -INFINITY;
                    }
                }
                float mx4[4];                                     // four short chains of 3-input maxima
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float v = fmaxf(sv[16 * k], sv[16 * k + 15]);
#pragma unroll
                    for (int i = 1; i < 15; i += 2) v = fmax3(v, sv[16 * k + i], sv[16 * k + i + 1]);
                    mx4[k] = v;
                }
                const float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
                // lazy rescale: keep the stale maximum while the new one stays within 2^slack
                const bool old_live = m != -INFINITY;
                const bool resc = mx > m + kTcSlack;
                float alpha = 1.f;
                if (resc) {
                    alpha = old_live ? fast_exp2(m - mx) : 0.f;
                    m = mx;
                }
                l *= alpha;
                if (c > 0 && __any_sync(kFull, resc && old_live)) {       // O holds earlier chunks: scale it
                    // once P_t(G-1).V(G-1) has landed in it
                    ok = __all_sync(kFull, mbar_wait(bar_o(tt, G - 1), par4(G - 1)));
                    if (!ok) break;
                    tc_fence_after();
                    const float f = (resc && old_live) ? alpha : 1.f;
#pragma unroll
                    for (int q = 0; q < D / 16; ++q) {
                        uint32_t r16[16];
                        tmem_ld16(t_o + 16 * q, r16);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; ++k) r16[k] = __float_as_uint(__uint_as_float(r16[k]) * f);
                        tmem_st16(t_o + 16 * q, r16);
                    }
                }
                const float mu = m == -INFINITY ? 0.f : m;    // a row with nothing attended yet: p = 0
                const uint64_t mu2 = f2_make(mu, mu);
                uint64_t ps2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
                // P over S: block jl's 16 tokens to columns [16jl, 16jl+16) of the
                // buffer, 8 high then 8 low columns
#pragma unroll
                for (int jl = 0; jl < kW2Blocks; ++jl) {
                    uint32_t w16[16];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 d = f2_split(f2_sub(f2_make(sv[16 * jl + 2 * e], sv[16 * jl + 2 * e + 1]), mu2));
                        const float x = fast_exp2(d.x), y = fast_exp2(d.y);
                        const uint64_t xy = f2_make(x, y);
                        ps2[e & 1] = f2_add(ps2[e & 1], xy);
                        w16[e] = pack2<kB>(x, y);
                        const float2 f = unpack2<kB>(w16[e]);
                        const float2 r = f2_split(f2_sub(xy, f2_make(f.x, f.y)));
                        w16[8 + e] = pack2<kB>(r.x, r.y);
                    }
                    tmem_st16(t_buf + 16 * jl, w16);
                }
                tmem_wait_st();
                {
                    const float2 p0 = f2_split(ps2[0]), p1 = f2_split(ps2[1]);
                    l += (p0.x + p1.x) + (p0.y + p1.y);
                }
                // V rows of tokens outside the sequence or of missing blocks hold
                // arbitrary bits: each tile zeroes them before its P(G) is ready (its
                // MMA warp issues P_t(G).V(G) only then); both tiles write the same zeros
                if (bm != (1u << kW2Blocks) - 1u || cpos + kW2Chunk > it.L) {
                    ok = __all_sync(kFull, mbar_wait(bar_v(G), par_st(G)));
                    const uint32_t vb = sV + stage(G) * C::kVc;
                    for (int i = tid & (kTcRows - 1); i < kW2Chunk * 2 * 8; i += kTcRows) {
                        const int tk2 = i / 16, h = (i / 8) % 2, ck = i % 8;
                        if (((bm >> (tk2 / kBlock)) & 1u) && cpos + tk2 < it.L) continue;
                        sts128(vb + (tk2 / kBlock) * C::kVb + h * (kBlock * 128) + (tk2 % kBlock) * 128 + ck * 16,
                               make_uint4(0u, 0u, 0u, 0u));
                    }
                    fence_proxy_async_smem();      // zeroed V visible to the tensor core
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p(tt, G));
                if (!ok) break;
            }
            if (!ok) break;
            // the next item's Q_t has landed: its MMA warp may start on it
            if (have_nx) q_stored();
            // ---- wait for this tile's last P.V (the copy's newest event; the one
            // before it, four chunks back, was done before S_t(last) was issued),
            // then normalise and store, 16 columns at a time through this warp's
            // staging rows: by TMA, or with 64-byte row pieces, eight rows per
            // store instruction, where a row is past the prompt or the output is
            // not fp32
            const int G_last = gc + it.nchunks - 1;
            ok = __all_sync(kFull, mbar_wait(bar_o(tt, G_last), par4(G_last)));
            if (!ok) break;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int wr0 = it.row0 + 32 * warp;  // this warp's first row (tile 1 = warps 4-7)
            if (a.out_tma && wr0 + 32 <= it.rows) {
                // every row of the warp is live: the 32 rows are (32/G tokens x G
                // heads) or (1 token x 32 heads), one box of the output map per 16
                // columns, stored by TMA from this warp's staging (unpadded rows,
                // 16-byte chunk j of row r at chunk j ^ ((r >> 1) & 3): the map's
                // 64-byte swizzle) while the warp goes on
                const uint32_t sst = smem_addr(stg);
                const int tq = wr0 / a.G, hq = wr0 - tq * a.G;
#pragma unroll
                for (int q = 0; q < D / 16; ++q) {
                    uint32_t r16[16];
                    tmem_ld16(t_o + 16 * q, r16);
                    tmem_wait_ld();
                    if (lane == 0) bulk_wait_read();        // the previous box has been read out
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        sts128(sst + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4),
                               make_uint4(__float_as_uint(__uint_as_float(r16[4 * k]) * inv),
                                          __float_as_uint(__uint_as_float(r16[4 * k + 1]) * inv),
                                          __float_as_uint(__uint_as_float(r16[4 * k + 2]) * inv),
                                          __float_as_uint(__uint_as_float(r16[4 * k + 3]) * inv)));
                    fence_proxy_async_smem();               // the box visible to the TMA unit
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&omap, sst, 16 * q, it.g * a.G + hq, it.q0 + tq);
                        bulk_commit();
                    }
                }
                if (lane == 0) bulk_wait_read();            // staging free for the next item
                __syncwarp();
            } else {
                long long orow[4];
                bool orow_ok[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int rw = wr0 + 8 * k + (lane >> 2);
                    const int tkr = rw / a.G, hr = rw - tkr * a.G;
                    orow_ok[k] = rw < it.rows;
                    orow[k] = ((long long)(it.q0 + tkr) * a.H + (long long)it.g * a.G + hr) * D + 4 * (lane & 3);
                }
#pragma unroll
                for (int q = 0; q < D / 16; ++q) {
                    uint32_t r16[16];
                    tmem_ld16(t_o + 16 * q, r16);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; k += 4)
                        *reinterpret_cast<float4*>(stg + lane * C::kStgRowF + k) =
                            make_float4(__uint_as_float(r16[k]) * inv, __uint_as_float(r16[k + 1]) * inv,
                                        __uint_as_float(r16[k + 2]) * inv, __uint_as_float(r16[k + 3]) * inv);
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (orow_ok[k])
                            store4(a.out, a.out_dtype, orow[k] + 16 * q,
                                   *reinterpret_cast<const float4*>(stg + (8 * k + (lane >> 2)) * C::kStgRowF + 4 * (lane & 3)));
                    __syncwarp();
                }
            }
            gc += it.nchunks;
            it = nx;
            round = round_nx;
            have = have_nx;
        }
        if (!ok && lane == 0) flag_error(a.err, GQA_DEVERR_TIMEOUT);
        cp_async_wait_all();                   // nothing of this warp's still lands in shared memory
        if (lane == 0) bulk_wait_all();        // its output stores are done
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

template <typename T, int kTiles>
const void* prefill_tc2_fn() {
    return reinterpret_cast<const void*>(&prefill_tc2_kernel<T, kTiles>);
}

template <typename T, int D>
const void* prefill_tc_fn() {
    return reinterpret_cast<const void*>(&prefill_tc_kernel<T, D>);
}

template <typename T, int D>
const void* prefill_fn() {
    return reinterpret_cast<const void*>(&prefill_kernel<T, D>);
}

}  // namespace

int device_sms(int device);   // gqa_capi.cu
bool encode_out_map(CUtensorMap* map, void* out, int num_heads, int G, long long tokens);   // gqa_capi.cu

int launch_prefill(const PrefillLaunch& L) {
    const gqa_kv_cache_t& c = *L.cache;
    const int D = c.head_dim, K = c.num_kv_heads, G = L.num_heads / K;
    const bool tc = L.kernel != GQA_PREFILL_MMA_SYNC;
    // the 64-token-chunk tcgen05 forms serve head_dim 128: two query tiles per
    // CTA (one CTA per SM) or one (two CTAs per SM)
    const bool wide2 = tc && D == 128 && (L.kernel == GQA_PREFILL_AUTO || L.kernel == GQA_PREFILL_TCGEN05_WIDE);
    const bool wide1 = tc && D == 128 && L.kernel == GQA_PREFILL_TCGEN05_PAIRED;
    const bool wide = wide1 || wide2;
    const int rows_per_cta = wide2 ? W2Cfg<2>::kRows : wide1 ? W2Cfg<1>::kRows : tc ? kTcRows : kPfRows;
    const void* fn = nullptr;
    int smem = 0;
    if (wide) {
        if (c.dtype != GQA_DTYPE_BF16 && c.dtype != GQA_DTYPE_F16) return GQA_ERR_UNSUPPORTED;
        const bool bf = c.dtype == GQA_DTYPE_BF16;
        fn = wide2 ? (bf ? prefill_tc2_fn<__nv_bfloat16, 2>() : prefill_tc2_fn<__half, 2>())
                   : (bf ? prefill_tc2_fn<__nv_bfloat16, 1>() : prefill_tc2_fn<__half, 1>());
        smem = wide2 ? W2Cfg<2>::kSmem : W2Cfg<1>::kSmem;
    } else if (c.dtype == GQA_DTYPE_BF16) {
        if (tc) {
            fn = D == 64 ? prefill_tc_fn<__nv_bfloat16, 64>() : prefill_tc_fn<__nv_bfloat16, 128>();
            smem = D == 64 ? TcCfg<__nv_bfloat16, 64>::kSmem : TcCfg<__nv_bfloat16, 128>::kSmem;
        } else {
            fn = D == 64 ? prefill_fn<__nv_bfloat16, 64>() : prefill_fn<__nv_bfloat16, 128>();
            smem = D == 64 ? PfCfg<__nv_bfloat16, 64>::kSmem : PfCfg<__nv_bfloat16, 128>::kSmem;
        }
    } else if (c.dtype == GQA_DTYPE_F16) {
        if (tc) {
            fn = D == 64 ? prefill_tc_fn<__half, 64>() : prefill_tc_fn<__half, 128>();
            smem = D == 64 ? TcCfg<__half, 64>::kSmem : TcCfg<__half, 128>::kSmem;
        } else {
            fn = D == 64 ? prefill_fn<__half, 64>() : prefill_fn<__half, 128>();
            smem = D == 64 ? PfCfg<__half, 64>::kSmem : PfCfg<__half, 128>::kSmem;
        }
    } else {
        return GQA_ERR_UNSUPPORTED;
    }
    CUtensorMap kmap, vmap;
    int perm[3];
    if (!encode_cache_map(&kmap, c, c.k, 64, 128, perm) || !encode_cache_map(&vmap, c, c.v, 64, 128, perm))
        return GQA_ERR_UNSUPPORTED;
    int page_perm[2] = {1, 2};
    if (tc && D == 128 && !encode_page_map(&vmap, c, c.v, page_perm))   // V a page per box
        return GQA_ERR_UNSUPPORTED;
    const int threads = wide2 ? W2Cfg<2>::kThreads : wide1 ? W2Cfg<1>::kThreads : tc ? kTcThreads : kPfWarps * 32;
    if (ctas_per_sm(fn, threads, smem) < 1) return GQA_ERR_CUDA;

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
    a.tiles_per_seq = (int)(((long long)L.max_new_tokens * G + rows_per_cta - 1) / rows_per_cta);
    a.window = L.window;
    a.map_perm[0] = perm[0];
    a.map_perm[1] = perm[1];
    a.map_perm[2] = perm[2];
    a.page_perm[0] = page_perm[0];
    a.page_perm[1] = page_perm[1];
    a.scale_log2 = L.scale * kLog2eP;
    if (a.tiles_per_seq == 0) return GQA_OK;
    // the 64-token forms store whole-live warps' output by TMA: fp32 out, a
    // warp's 32 rows a box of (32/G tokens x G heads) or (1 token x 32 heads)
    CUtensorMap omap;
    memset(&omap, 0, sizeof(omap));
    a.out_tma = 0;
    if (wide && L.out_dtype == GQA_DTYPE_F32 && (32 % G == 0 || G % 32 == 0))
        a.out_tma = encode_out_map(&omap, L.out, L.num_heads, G, (long long)L.max_new_tokens * L.batch) ? 1 : 0;

    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    if (wide) {
        // persistent CTAs: as many as fit at once, each walking its items
        const long long items = (long long)a.tiles_per_seq * K * L.batch;
        const int sms = device_sms(-1);
        if (items > INT32_MAX || sms <= 0) return GQA_ERR_UNSUPPORTED;
        const long long fit = (long long)sms * (wide2 ? W2Cfg<2>::kCtasPerSm : W2Cfg<1>::kCtasPerSm);
        cfg.gridDim = dim3((unsigned)(items < fit ? items : fit));
    } else {
        cfg.gridDim = dim3((unsigned)a.tiles_per_seq, (unsigned)K, (unsigned)L.batch);
    }
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    void* args[] = {&kmap, &vmap, &a};
    void* args_w[] = {&kmap, &vmap, &omap, &a};
    return cudaLaunchKernelExC(&cfg, fn, wide ? args_w : args) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
