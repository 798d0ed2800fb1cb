// hbm_read_probe.cu -- the HBM read ceiling the decode kernels are held
// against: a pure read stream of a buffer larger than L2, in the two forms the
// library's kernels use to move data, each reduced to an XOR so the loads
// cannot be dropped.
//
//  * bulk: every warp streams consecutive chunks of the buffer through its own
//    ring of shared-memory stages with 1-D bulk copies (cp.async.bulk), one
//    mbarrier per stage, as the split-KV kernel streams its K/V tiles.
//  * ldg:  16-byte non-coherent vector loads, grid-strided.
//
// Built as its own small library (libhbm_probe.so), loaded only by the
// benchmark; the decode library does not contain it.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool try_wait_parity(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits at most one second; false on expiry.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
    if (try_wait_parity(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 1000000000ull)
        if (try_wait_parity(bar, parity)) return true;
    return false;
}

constexpr unsigned long long kTimeoutFlag = 1ull << 40;

// Warp w of the grid reads chunks [w*per, min((w+1)*per, nchunks)) of CH bytes.
template <int S, int CH>
__global__ void __launch_bounds__(128) bulk_read_kernel(const uint8_t* __restrict__ p, size_t nchunks,
                                                        unsigned long long* sink) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[4][S];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + (size_t)warp * S * CH;
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&bars[warp][0]);
    const uint32_t ring0 = (uint32_t)__cvta_generic_to_shared(ring);
    if (lane == 0) {
        for (int s = 0; s < S; ++s) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8 * s));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const size_t W = (size_t)gridDim.x * 4, gw = (size_t)blockIdx.x * 4 + warp;
    const size_t per = (nchunks + W - 1) / W;
    const size_t c0 = gw * per, c1 = c0 + per < nchunks ? c0 + per : nchunks;
    if (c0 >= c1) return;
    const size_t n = c1 - c0;
    auto issue = [&](size_t k, int s) {
        if (lane == 0) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar0 + 8 * s), "r"(CH)
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    ring0 + s * CH),
                "l"(p + (c0 + k) * CH), "r"(CH), "r"(bar0 + 8 * s)
                : "memory");
        }
    };
    const int first = n < (size_t)S ? (int)n : S;
    for (int s = 0; s < first; ++s) issue(s, s);
    uint32_t acc = 0;
    for (size_t k = 0; k < n; ++k) {
        const int s = (int)(k % S);
        const uint32_t ph = (uint32_t)((k / S) & 1);
        if (!wait_bounded(bar0 + 8 * s, ph)) {
            if (lane == 0) atomicAdd(sink, kTimeoutFlag);
            // let this warp's other copies in flight land (bounded) before leaving
            for (size_t j = k + 1; j < k + S && j < n; ++j)
                wait_bounded(bar0 + 8 * (int)(j % S), (uint32_t)((j / S) & 1));
            return;
        }
        uint32_t x, y, z, w;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x), "=r"(y), "=r"(z), "=r"(w)
                     : "r"(ring0 + s * CH + lane * 16)
                     : "memory");
        acc ^= x ^ y ^ z ^ w;
        __syncwarp();
        if (k + S < n) issue(k + S, s);
    }
    if (acc == 0x9e3779b9u) atomicAdd(sink, 1ull);
}

__global__ void ldg_read_kernel(const uint4* __restrict__ p, size_t n, unsigned long long* sink) {
    uint32_t acc = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
#pragma unroll 8
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint4 v = __ldg(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == 0x9e3779b9u) atomicAdd(sink, 1ull);
}

template <int S, int CH>
int launch_bulk(const void* buf, size_t bytes, unsigned long long* sink, int ctas_per_sm, int sms,
                cudaStream_t st) {
    const int smem = 4 * S * CH;
    auto fn = bulk_read_kernel<S, CH>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -3;
    fn<<<sms * ctas_per_sm, 128, smem, st>>>(static_cast<const uint8_t*>(buf), bytes / CH, sink);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace

// Reads `bytes` of `buf` once (`form` 0..2: bulk copies in 8 KB chunks with 2
// or 3 stages per warp, or 4 KB chunks with 4 stages; 3: 16-byte loads) on
// `stream`. buf must be 16-byte aligned and bytes a multiple of 8192; sink is
// one device word, zeroed by the caller, that stays below 2^40 unless a wait
// timed out. Returns 0, -1 on a bad argument, -3 on a launch error.
extern "C" __attribute__((visibility("default"))) int hbm_read_probe(const void* buf, size_t bytes,
                                                                     unsigned long long* sink, int form,
                                                                     int ctas_per_sm, void* stream) {
    if (!buf || !sink || (reinterpret_cast<uintptr_t>(buf) & 15u) || bytes == 0 || bytes % 8192 ||
        ctas_per_sm < 1 || ctas_per_sm > 16)
        return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -3;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (form) {
        case 0: return launch_bulk<2, 8192>(buf, bytes, sink, ctas_per_sm, sms, st);
        case 1: return launch_bulk<3, 8192>(buf, bytes, sink, ctas_per_sm, sms, st);
        case 2: return launch_bulk<4, 4096>(buf, bytes, sink, ctas_per_sm, sms, st);
        case 3:
            ldg_read_kernel<<<sms * ctas_per_sm, 256, 0, st>>>(static_cast<const uint4*>(buf), bytes / 16, sink);
            return cudaGetLastError() == cudaSuccess ? 0 : -3;
        default: return -1;
    }
}
