// gqa_decode.cu -- host side of the split-KV decode: kernel choice, workspace
// layout, partition sizing and the launches (kernels in gqa_decode_kernels.cuh).
// Instantiates the one-token, full-attention kernels and the combine kernels.
#include <mutex>

#include "gqa_decode_kernels.cuh"

namespace gqa {
namespace dec {

bool pick_plain(int dtype, int kind, int d, int nw, Variant& v) {
    return pick_variant<false>(dtype, kind, d, nw, v);
}

}  // namespace dec

// Resident CTAs per SM of a kernel at a dynamic shared-memory size, asked of
// the runtime once per (device, kernel, size) and remembered: a decode step
// asks on every call. The kernel's shared-memory limit is raised to the
// largest size asked for so far on the device (a limit set for one size
// serves every smaller one).
namespace {
struct OccEntry {
    int device;
    const void* fn;
    int smem, threads, per_sm;
};
struct LimitEntry {
    int device;
    const void* fn;
    int smem;
};
constexpr int kOccCacheSize = 128;
OccEntry g_occ[kOccCacheSize];
LimitEntry g_limit[kOccCacheSize];
int g_occ_used = 0, g_occ_next = 0, g_limit_used = 0;
std::mutex g_occ_mutex;

// Raises fn's dynamic shared-memory limit to at least smem; g_occ_mutex held.
bool ensure_limit(int dev, const void* fn, int smem) {
    for (int i = 0; i < g_limit_used; ++i) {
        LimitEntry& e = g_limit[i];
        if (e.device == dev && e.fn == fn) {
            if (e.smem >= smem) return true;
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
                return false;
            e.smem = smem;
            return true;
        }
    }
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
    if (g_limit_used < kOccCacheSize) g_limit[g_limit_used++] = LimitEntry{dev, fn, smem};
    return true;
}
}  // namespace

int ctas_per_sm(const void* fn, int threads, int smem) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    if (!ensure_limit(dev, fn, smem)) return 0;
    for (int i = 0; i < g_occ_used; ++i) {
        const OccEntry& e = g_occ[i];
        if (e.device == dev && e.fn == fn && e.smem == smem && e.threads == threads) return e.per_sm;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess) return 0;
    g_occ[g_occ_next] = OccEntry{dev, fn, smem, threads, per_sm};
    g_occ_next = (g_occ_next + 1) % kOccCacheSize;
    g_occ_used = std::max(g_occ_used, g_occ_next == 0 ? kOccCacheSize : g_occ_next);
    return per_sm;
}

namespace {

using namespace dec;

struct WsLayout {
    size_t hdr, pref, ml, o, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split slots: one per (pair, segment) overlap, at most pairs + segments. A
// worker's range has R <= max(ceil(B*K*max_blocks / P), min_units) units and at
// most min(kMaxTailChunks, R / 32) pooled chunks (make_partition); max_blocks
// <= 0 means unknown.
long long max_slots(int B, int K, int P, int max_blocks, int min_units, int tail_chunks) {
    int cpw = tail_chunks;
    if (max_blocks > 0) {
        const long long u_max = (long long)B * K * max_blocks;
        const long long r_max = std::max<long long>((u_max + P - 1) / P, min_units);
        cpw = (int)std::min<long long>(tail_chunks, r_max / (8 * kMinChunk));
    }
    return (long long)B * K + (long long)P * (1 + cpw);
}

WsLayout ws_layout(int B, int K, int rows, int D, long long slots) {
    WsLayout w;
    w.hdr = 0;
    w.pref = align256(kWsHeaderInts * 4);
    w.ml = w.pref + align256((size_t)(B + 1) * 4);
    w.o = w.ml + align256((size_t)slots * rows * 8);
    w.total = w.o + align256((size_t)slots * rows * D * 4);
    return w;
}

// Split-KV workers one launch uses for variant v at this batch (occupancy of a
// single resident wave); 0 if the variant cannot launch.
int workers_of(const Variant& v, int batch, int num_sms) {
    return num_sms * ctas_per_sm(v.fn, v.warps * 32, v.smem(batch)) * v.workers_per_cta;
}

}  // namespace

// Warps that share one pair's tiles for GT query rows per pair (8 rows each).
int warps_for_rows(int GT) { return GT <= 8 ? 1 : GT <= 16 ? 2 : GT <= 32 ? 4 : 8; }
int row_groups(int GT) { return (GT + kHeadsPerWarp - 1) / kHeadsPerWarp; }


// The largest workspace any kernel choice needs for this shape: workers are
// taken from the occupancy of every variant that can serve (G*T, head_dim), in
// both the shared-ring and the virtual-head layout.
size_t decode_workspace_bytes(int batch, int num_heads, int num_kv_heads, int head_dim, int tokens_per_seq,
                              int num_sms) {
    const int GT = num_heads / num_kv_heads * std::max(1, tokens_per_seq);
    const int nw = warps_for_rows(GT);
    int P = 0;
    for (int kind : {kKernelMma, kKernelFma}) {
        for (int dt : {GQA_DTYPE_F32, GQA_DTYPE_F16, GQA_DTYPE_BF16, GQA_DTYPE_I8, GQA_DTYPE_FP8_E4M3,
                       GQA_DTYPE_I4, GQA_DTYPE_I4_KC}) {
            for (int w : {1, nw}) {
                Variant v{};
                if (pick_plain(dt, kind, head_dim, w, v)) P = std::max(P, workers_of(v, batch, num_sms));
                if (pick_general(dt, kind, head_dim, w, v)) P = std::max(P, workers_of(v, batch, num_sms));
            }
        }
    }
    if (P == 0) P = num_sms * kMaxWarpsPerSm;             // no occupancy answer: the hard bound
    size_t bytes = ws_layout(batch, num_kv_heads, GT, head_dim,
                             max_slots(batch, num_kv_heads, P, 0, 0, kMaxTailChunks)).total;
    if (GT > kHeadsPerWarp) {
        const int Kv = num_kv_heads * row_groups(GT);
        bytes = std::max(bytes, ws_layout(batch, Kv, kHeadsPerWarp, head_dim,
                                          max_slots(batch, Kv, P, 0, 0, kMaxTailChunks)).total);
    }
    return bytes;
}

int launch_decode(const DecodeLaunch& L, int num_sms) {
    const gqa_kv_cache_t& c = *L.cache;
    const int D = c.head_dim, K = c.num_kv_heads, G = L.num_heads / K;
    const int T = std::max(1, L.tokens_per_seq), GT = G * T;
    int kind = L.kernel;
    if (kind == 0) kind = (c.dtype == GQA_DTYPE_F32 || (dtype_coded(c.dtype) && D != 128)) ? kKernelFma : kKernelMma;
    Variant v{};
    const bool general = T > 1 || L.window > 0;
    auto pick = [&](int warps) {
        return general ? pick_general(c.dtype, kind, D, warps, v) : pick_plain(c.dtype, kind, D, warps, v);
    };
    // More than 8 rows: by default the CTA's warps share each tile (measured
    // faster than 8-row unit streams at 16, 32 and 64 rows: the per-block
    // latency, not the worker count, bounds these shapes); unit streams where
    // no shared-ring kernel exists or when asked for. (Virtual heads multiply
    // the unit count, which must stay below 2^31.)
    int nrg = 1;
    bool ok = false;
    if (GT <= kHeadsPerWarp) {
        ok = pick(1);
    } else {
        const int groups = row_groups(GT);
        const bool virt_fits = (long long)L.batch * K * groups * L.max_blocks < 0x7fffffffLL;
        const bool want_virt = L.row_layout == 1;
        if (virt_fits && want_virt && pick(1)) {
            ok = true;
            nrg = groups;
        } else if (pick(warps_for_rows(GT))) {
            ok = true;
        } else if (virt_fits && pick(1)) {
            ok = true;
            nrg = groups;
        }
    }
    if (!ok) return GQA_ERR_UNSUPPORTED;
    const int Kv = K * nrg, RS = nrg > 1 ? kHeadsPerWarp : GT;

    CUtensorMap kmap, vmap;
    int perm[3];
    if (!encode_cache_map(&kmap, c, c.k, v.box_inner, v.swizzle_bytes, perm) ||
        !encode_cache_map(&vmap, c, c.v, v.box_inner, v.swizzle_bytes, perm))
        return GQA_ERR_UNSUPPORTED;
    // 16-bit tiles of 128-element rows come two 64-element boxes at a time
    // through the maps above; a page map moves the whole tile in one copy
    int page_perm[2] = {1, 2};
    bool page_box = false;
    if (dtype_bits(c.dtype) == 16 && D == 128 && v.box_inner == 64 && v.swizzle_bytes == 128) {
        CUtensorMap kp, vp;
        if (encode_page_map(&kp, c, c.k, page_perm) && encode_page_map(&vp, c, c.v, page_perm)) {
            kmap = kp;
            vmap = vp;
            page_box = true;
        }
    }

    const int smem = v.smem(L.batch);
    const int workers = workers_of(v, L.batch, num_sms);
    if (workers < 1) return GQA_ERR_UNSUPPORTED;
    int grid = workers / v.workers_per_cta;
    cudaError_t e;
    if (L.max_warps > 0)
        grid = std::min(grid, std::max(1, (L.max_warps + v.workers_per_cta - 1) / v.workers_per_cta));
    const int P = grid * v.workers_per_cta;   // split-KV workers (KV splits per pass)

    const int min_units = L.min_blocks_per_warp > 0 ? L.min_blocks_per_warp : 4;
    const WsLayout wl =
        ws_layout(L.batch, Kv, RS, D, max_slots(L.batch, Kv, P, L.max_blocks, min_units, v.tail_chunks));
    if (L.workspace == nullptr || L.workspace_bytes < wl.total) return GQA_ERR_WORKSPACE;

    DecodeArgs a;
    a.q = L.q;
    a.k_scale = static_cast<const __half*>(c.k_scale);
    a.v_scale = static_cast<const __half*>(c.v_scale);
    a.block_tables = L.block_tables;
    a.context_lens = L.context_lens;
    a.out = L.out;
    a.err = L.err;
    uint8_t* ws = static_cast<uint8_t*>(L.workspace);
    a.ws_hdr = reinterpret_cast<int32_t*>(ws + wl.hdr);
    a.ws_ctr = reinterpret_cast<unsigned long long*>(ws + wl.hdr + 32 * sizeof(int32_t));
    a.ws_pref = reinterpret_cast<int32_t*>(ws + wl.pref);
    a.ws_ml = reinterpret_cast<float2*>(ws + wl.ml);
    a.ws_o = reinterpret_cast<float*>(ws + wl.o);
    a.num_blocks = c.num_blocks;
    a.B = L.batch;
    a.H = L.num_heads;
    a.K = K;
    a.G = G;
    a.T = T;
    a.GT = GT;
    a.Kv = Kv;
    a.NRG = nrg;
    a.RS = RS;
    a.window = L.window;
    a.max_blocks = L.max_blocks;
    a.out_dtype = L.out_dtype;
    a.q_dtype = L.q_dtype;
    a.P = P;
    a.map_perm[0] = perm[0];
    a.map_perm[1] = perm[1];
    a.map_perm[2] = perm[2];
    a.page_box = page_box ? 1 : 0;
    a.page_perm[0] = page_perm[0];
    a.page_perm[1] = page_perm[1];
    a.min_units = min_units;
    a.max_tail_chunks = v.tail_chunks;
    a.scale_log2 = L.scale * kLog2e;

    // Both kernels go out with programmatic stream serialisation: each may be
    // scheduled while its predecessor drains and waits on the device
    // (griddepcontrol.wait) before it reads any input. Timing events split the
    // chain, so with events the launches are plain.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    const bool timed = L.ev_begin || L.ev_end;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(v.warps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = timed ? 0 : 1;
    if (L.ev_begin && cudaEventRecord(L.ev_begin, L.stream) != cudaSuccess) return GQA_ERR_CUDA;
    void* args[] = {&kmap, &vmap, &a};
    e = cudaLaunchKernelExC(&cfg, v.fn, args);
    if (e != cudaSuccess) return GQA_ERR_CUDA;
    // From here the split-KV kernel has advanced the pool's ticket counter,
    // which only the combine rewinds: a failure before the combine is queued
    // rewinds it on the stream instead, so the next call on this workspace
    // starts from zero.
    auto fail_after_split = [&]() {
        cudaMemsetAsync(a.ws_ctr, 0, sizeof(unsigned long long), L.stream);
        return GQA_ERR_CUDA;
    };
    if (L.ev_end && cudaEventRecord(L.ev_end, L.stream) != cudaSuccess) return fail_after_split();

    // Combine width from the expected pieces per row (about 1.5 workers' worth
    // of segments per pair when lengths are even).
    const long long pairs = (long long)L.batch * Kv;
    const long long est = (3LL * P) / (2 * pairs) + 1;
    const void* cfn;
    int rows_per_cta, cthreads;
    if (est <= 8) {
        cfn = D == 64 ? reinterpret_cast<const void*>(&combine_kernel<64, 1, 8>)
                      : reinterpret_cast<const void*>(&combine_kernel<128, 1, 8>);
        rows_per_cta = 8;
        cthreads = 256;
    } else if (est <= 64) {
        cfn = D == 64 ? reinterpret_cast<const void*>(&combine_kernel<64, 8, 1>)
                      : reinterpret_cast<const void*>(&combine_kernel<128, 8, 1>);
        rows_per_cta = 1;
        cthreads = 256;
    } else {
        cfn = D == 64 ? reinterpret_cast<const void*>(&combine_kernel<64, 32, 1>)
                      : reinterpret_cast<const void*>(&combine_kernel<128, 32, 1>);
        rows_per_cta = 1;
        cthreads = 1024;
    }
    const long long rows = (long long)L.batch * T * L.num_heads;
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3((unsigned)((rows + rows_per_cta - 1) / rows_per_cta));
    ccfg.blockDim = dim3(cthreads);
    ccfg.stream = L.stream;
    ccfg.attrs = pdl;
    ccfg.numAttrs = timed ? 0 : 1;
    void* cargs[] = {&a};
    if (cudaLaunchKernelExC(&ccfg, cfn, cargs) != cudaSuccess) return fail_after_split();
    return GQA_OK;
}

}  // namespace gqa
