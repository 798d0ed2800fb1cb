// gqa_device.cuh -- device helpers shared by the decode and append kernels:
// inline PTX for mbarriers, TMA (cp.async.bulk.tensor / cp.async.bulk),
// warp-level bf16/f16 tensor-core MMA, exp2 and small packing routines.
// sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gqa_decode.h"

namespace gqa {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kBlock = 16;                       // tokens per cache block
// Longest a warp waits for one asynchronous copy before it gives up, sets
// GQA_DEVERR_TIMEOUT and leaves (a copy never takes this long unless the
// hardware is wedged).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void flag_error(int32_t* err, int bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- dependent launch

// Wait until the grid this one depends on (previous kernel in the stream) has
// completed and its memory is visible. A no-op without programmatic launch.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel in the stream be scheduled now (it still waits for this
// grid's completion before it reads anything).
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false after the time limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 4-D tiled tensor copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
        : "memory");
}

// 5-D tiled tensor copy global -> shared (a whole page through a page map).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, int v, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v), "r"(bar), "l"(policy)
        : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- shared loads

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Four 8x8 b16 matrices; lanes 8i..8i+7 give the row addresses of matrix i.
// Register i holds matrix i's fragment: row lane/4, elements 2(lane%4), +1.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Same, transposed: register i holds column lane/4, rows 2(lane%4), +1 of matrix i.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// Address of 16-byte chunk `chunk` of row `tok` in a tile written by TMA with
// 128-byte swizzle (2 KB boxes of 16 rows x 128 B; chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(uint32_t tile, int tok, int chunk) {
    return tile + (uint32_t)(chunk >> 3) * 2048u + (uint32_t)tok * 128u +
           ((uint32_t)((chunk & 7) ^ (tok & 7)) << 4);
}

// ---------------------------------------------------------------- math

// 2^x on the SFU (ex2.approx; -inf -> +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// D += A(16x16, row) * B(16x8, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ uint32_t as_u32(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }

// Two floats -> packed 16-bit pair (lo in bits 0..15), round to nearest even.
template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (kBf16) return as_u32(__floats2bfloat162_rn(lo, hi));
    else return as_u32(__floats2half2_rn(lo, hi));
}

// Packed 16-bit pair -> the two floats (exact).
template <bool kBf16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
    if constexpr (kBf16) {
        return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    } else {
        __half2 h = *reinterpret_cast<__half2*>(&v);
        return __half22float2(h);
    }
}

// Four int8 codes (one 32-bit word, byte i = element i) -> two packed f16 pairs,
// exact: each byte is biased to u = x + 128, placed as the mantissa of
// 1024 + u (fp16 0x6400 | u), and 1152 is subtracted.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t t = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(t, 0x64646464u, 0x4140);   // bytes 0,1
    const uint32_t b = __byte_perm(t, 0x64646464u, 0x4342);   // bytes 2,3
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = as_u32(ha);
    hi = as_u32(hb);
}

// Two e4m3 codes (16 bits, element 0 in the low byte) -> f16 pair, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xffffu), __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Element tag of a 4-bit cache: one byte holds two codes (element 2j in the
// low nibble). Only its size (1) and identity are used.
struct int4x2 {
    uint8_t v;
};
// The same codes with K scaled per (block, kv-head, channel) (KIVI-style).
struct int4kc {
    uint8_t v;
};

// Lane-wise product of two f16 pairs, rounded to nearest.
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Lane-wise a*b + c of f16 pairs with one rounding.
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// d = b ? (a ^ c) : c, bit by bit (one LOP3): with b a mask and c holding the
// bits to flip under the mask and the bits to set elsewhere.
__device__ __forceinline__ uint32_t lop3_select_xor(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two signed 4-bit codes -> f16 pair, exactly. From the low nibbles of bytes 0
// and 2 of w: each becomes the fp16 1024 + (code ^ 8) = 1032 + code (nibble
// under the exponent of 1024), then 1032 is subtracted.
__device__ __forceinline__ uint32_t i4_lo_pair(uint32_t w) {
    uint32_t h = lop3_select_xor(w, 0x000F000Fu, 0x64086408u);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
    return *reinterpret_cast<const uint32_t*>(&r);
}
// The same from the high nibbles of bytes 0 and 2: 1024 + 16*(code ^ 8) =
// 1152 + 16*code, so code = x/16 - 72 (one exact fma).
__device__ __forceinline__ uint32_t i4_hi_pair(uint32_t w) {
    uint32_t h = lop3_select_xor(w, 0x00F000F0u, 0x64806480u);
    const __half2 m = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));   // 1/16
    const __half2 c = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));   // -72
    const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&h), m, c);
    return *reinterpret_cast<const uint32_t*>(&r);
}

// Transpose of an 8x8 matrix of 16-bit values held one register per lane in
// the mma fragment layout (lane l: row l / 4, columns 2 (l % 4) and +1): lane l
// gets row l / 4 of the transpose, columns 2 (l % 4) and +1 (warp-collective).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Byte permute with the PTX selector semantics: a selector nibble with bit 3
// set writes the sign of the chosen byte replicated over all 8 bits.
__device__ __forceinline__ uint32_t prmt(uint32_t x, uint32_t y, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(y), "r"(sel));
    return r;
}

// Two e4m3 codes -> f16 pair holding 2^-8 times their values, exactly, with
// integer ops only. e4m3 is s.eeee.mmm with bias 7, f16 is s.eeeee.m(10) with
// bias 15: moving the seven exponent+mantissa bits up by 7 gives an f16 whose
// exponent is 8 smaller, for normal and subnormal codes alike (the largest
// code, 448, becomes 1.75; the smallest subnormal, 2^-9, becomes 2^-17).
// `sel` picks the two codes into bytes 0 and 2 of the halves, with their
// sign bytes (selector nibble | 8) in bytes 1 and 3; after the shift bit 15 of
// each half holds the sign and the mask clears what spilled past it.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t x, uint32_t y, uint32_t sel) {
    return (prmt(x, y, sel) << 7) & 0xBF80BF80u;
}

// ---------------------------------------------------------------- tcgen05 / TMEM

// Tensor-memory allocation of `cols` columns (a power of two >= 32) by one
// whole warp; the address lands in shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets, the fixed 0b001 at bits 46-48, 128-byte swizzle (mode 2, bits 61-63).
// K-major tiles: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO); an
// MN-major tile: 64-element MN atoms LBO apart, 8 K-rows SBO apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16 with fp32 accumulation: A/B element type
// (0 f16, 1 bf16), major-ness of A and B (1 = MN-major), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t mma_idesc_f16(int M, int N, bool bf16, bool a_mn, bool b_mn) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Arrive on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

}  // namespace gqa
