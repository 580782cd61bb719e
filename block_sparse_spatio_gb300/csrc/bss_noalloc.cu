// bss_noalloc.cu -- a tile-map build that allocates no device memory.
//
// bss_build_tile_map allocates its scratch (one class byte per tile, one
// counter per q tile) and the map itself with cudaMalloc, and synchronizes.
// Some callers cannot do that: a framework whose caching allocator owns all of
// the device memory and enforces its own limit (a stray cudaMalloc can fail or
// fragment the pool), or a latency-critical loop where cudaMalloc / cudaFree
// would synchronize the device.  They pass their own output buffers to
// bss_build_tile_map_csr_noalloc; the scratch lives in the fixed-size
// __device__ array below, which every GPU that loads this library holds until
// the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "bss_internal.h"

namespace bss {
namespace {

constexpr size_t kNoallocScratchBytes = static_cast<size_t>(BSS_NOALLOC_SCRATCH_BYTES);

// Scratch shared by every call: [class byte per tile | pad to 256 | int32 per q tile].
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
uint8_t* g_scratch_dev[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  Host code only
// holds a stand-in for the array's name, so the address is looked up once per
// device, with that device current, in the context then current (the device's
// primary context for runtime-API callers); it stays valid for that context's
// lifetime.
bss_status scratch_address(uint8_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(BSS_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mutex);
    if (g_scratch_dev[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_check(e, "cudaGetSymbolAddress(tile-map scratch)");
        g_scratch_dev[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_scratch_dev[dev];
    return BSS_OK;
}

// Exclusive prefix sum of the per-q-tile counts into row_ptr[0..nq], one block.
__global__ void __launch_bounds__(1024) row_ptr_scan_kernel(const int32_t* __restrict__ cnt, int32_t* __restrict__ row_ptr,
                                                            int32_t nq) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int32_t base = 0; base < nq; base += 1024) {
        const int32_t i = base + tid;
        const int32_t v = i < nq ? cnt[i] : 0;
        int32_t x = v;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int32_t w = warp_sums[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;  // inclusive sums of the warps
        }
        __syncthreads();
        const int32_t incl = x + (wid > 0 ? warp_sums[wid - 1] : 0) + carry;
        if (i < nq) row_ptr[i] = incl - v;
        __syncthreads();
        if (tid == 1023) carry = incl;
        __syncthreads();
    }
    if (tid == 0) row_ptr[nq] = carry;
}

}  // namespace
}  // namespace bss

extern "C" bss_status bss_build_tile_map_csr_noalloc(const bss_mask_params* params, int32_t kind, int32_t BQ,
                                                     int32_t BKV, int32_t* row_ptr, int32_t* entries,
                                                     int64_t entries_capacity, int64_t* stats, cudaStream_t stream) {
    using namespace bss;
    clear_error();
    bss_status st = check_mask_params(params);
    if (st != BSS_OK) return st;
    if (kind != 0 && kind != 1) return set_error(BSS_ERR_INVALID_ARG, "kind must be 0 or 1");
    if (BQ < 16 || BQ > 65536 || BKV < 16 || BKV > 65536)
        return set_error(BSS_ERR_INVALID_ARG, "BQ and BKV must lie in [16, 65536] (got %d, %d)", BQ, BKV);
    if (row_ptr == nullptr || entries == nullptr || stats == nullptr)
        return set_error(BSS_ERR_INVALID_ARG, "NULL output buffer");
    if ((reinterpret_cast<uintptr_t>(row_ptr) & 3u) || (reinterpret_cast<uintptr_t>(entries) & 3u) ||
        (reinterpret_cast<uintptr_t>(stats) & 7u))
        return set_error(BSS_ERR_INVALID_ARG, "misaligned output buffer");
    Geom g;
    g.F = params->F;
    g.S = params->Hs * params->Ws;
    g.N = g.F * g.S;
    g.wf = params->spatial_frame_window;
    g.ws = params->temporal_raster_window;
    g.S_pad = ((g.S + BKV - 1) / BKV) * BKV;
    const int32_t code = kind == 0 ? MASK_SPATIAL : (params->temporal_permuted ? MASK_TEMPORAL_VIRT : MASK_TEMPORAL_FHW);
    const int64_t nq = (static_cast<int64_t>(g.N) + BQ - 1) / BQ;
    int64_t ncols = 0, nkv = 0;
    tile_map_geometry(g, code, BKV, &ncols, &nkv);
    const int64_t ntiles = nq * nkv;
    const int64_t cnt_offset = (ntiles + 255) / 256 * 256;
    const int64_t need = cnt_offset + nq * static_cast<int64_t>(sizeof(int32_t));
    if (need > static_cast<int64_t>(kNoallocScratchBytes))
        return set_error(BSS_ERR_UNSUPPORTED,
                         "tile map of %lld x %lld tiles needs %lld scratch bytes, the fixed scratch holds %lld",
                         (long long)nq, (long long)nkv, (long long)need, (long long)kNoallocScratchBytes);
    if (ntiles > 0x7FFFFFFF) return set_error(BSS_ERR_UNSUPPORTED, "too many tiles");
    if (entries_capacity < ntiles)
        return set_error(BSS_ERR_INVALID_ARG, "entries_capacity %lld < q tiles x kv tiles = %lld",
                         (long long)entries_capacity, (long long)ntiles);
    uint8_t* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != BSS_OK) return st;
    uint8_t* cls = scratch;
    int32_t* cnt = reinterpret_cast<int32_t*>(scratch + cnt_offset);
    // the scratch keeps the previous call's contents: counters restart at zero
    if ((st = cuda_check(cudaMemsetAsync(cnt, 0, sizeof(int32_t) * nq, stream), "clear q-tile counters")) != BSS_OK)
        return st;
    if ((st = cuda_check(cudaMemsetAsync(stats, 0, sizeof(int64_t) * BSS_STAT_COUNT, stream), "clear stats")) !=
        BSS_OK)
        return st;
    st = launch_tile_classify(g, code, params->rounding, BQ, BKV, static_cast<int32_t>(nq), static_cast<int32_t>(nkv),
                              cls, cnt, reinterpret_cast<unsigned long long*>(stats), stream);
    if (st != BSS_OK) return st;
    // rounded maps of permuted temporal heads: the sink copies of kept band keys
    // (the column bitmasks are not needed for the CSR)
    st = launch_tile_dedup(g, code, params->rounding, BQ, BKV, static_cast<int32_t>(nq), static_cast<int32_t>(nkv), cls,
                           cnt, reinterpret_cast<unsigned long long*>(stats), nullptr, stream);
    if (st != BSS_OK) return st;
    row_ptr_scan_kernel<<<1, 1024, 0, stream>>>(cnt, row_ptr, static_cast<int32_t>(nq));
    if ((st = cuda_check(cudaGetLastError(), "row_ptr scan launch")) != BSS_OK) return st;
    return launch_tile_compact(static_cast<int32_t>(nq), static_cast<int32_t>(nkv), cls, row_ptr, entries, stream);
}
