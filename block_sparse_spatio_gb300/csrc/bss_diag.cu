// bss_diag.cu -- one-tile self-test of the tcgen05 / TMA building blocks used
// by the attention kernel (same descriptor helpers, same TMEM layout).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "bss_diag.h"
#include "bss_internal.h"
#include "bss_ptx.cuh"

namespace bss {
namespace {

struct DiagArgs {
    CUtensorMap tm_a, tm_b, tm_v;
    const uint16_t* P;
    float* S;
    float* O;
    int* status;
};

template <int D>
__global__ void __launch_bounds__(128, 1) diag_kernel(const __grid_constant__ DiagArgs args) {
    constexpr uint32_t kTile = 128 * D * 2;
    constexpr int kChunks = D / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kTile;
    uint8_t* sV = smem + 2 * kTile;
    uint64_t* bar_load = reinterpret_cast<uint64_t*>(smem + 3 * kTile);
    uint64_t* bar_mma = bar_load + 1;
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
    const int warp = threadIdx.x >> 5;
    const int r = threadIdx.x;
    if (r == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    bool ok = true;
    if (r == 0) {
        mbar_arrive_expect_tx(bar_load, 3 * kTile);
        for (int c = 0; c < kChunks; ++c) {
            tma_load_3d(sA + c * kChunkBytesSw128, &args.tm_a, c * 64, 0, 0, bar_load);
            tma_load_3d(sB + c * kChunkBytesSw128, &args.tm_b, c * 64, 0, 0, bar_load);
            tma_load_3d(sV + c * kChunkBytesSw128, &args.tm_v, c * 64, 0, 0, bar_load);
        }
    }
    // P row r -> TMEM columns [384, 448) of lane r, bf16 pairs, low half = even column
    {
        uint32_t pk[64];
        const uint32_t* prow = reinterpret_cast<const uint32_t*>(args.P + r * 128);
#pragma unroll
        for (int i = 0; i < 64; ++i) pk[i] = prow[i];
        BSS_TMEM_ST32(tmem + lane_base + 384, (pk + 0));
        BSS_TMEM_ST32(tmem + lane_base + 384 + 32, (pk + 32));
        tmem_wait_st();
    }
    ok = mbar_wait(bar_load, 0, args.status);
    tc_fence_before();
    __syncthreads();
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (r == 0 && ok) {
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);
        const uint32_t a = smem_u32(sA), b = smem_u32(sB), v = smem_u32(sV);
        for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + 0, desc_kmajor_sw128(a, kk), desc_kmajor_sw128(b, kk), idesc_qk, kk > 0);
        for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + 256, tmem + 384 + kk * 8, desc_mnmajor_sw128(v, kk), idesc_pv, kk > 0);
        tc_commit(bar_mma);
    }
    if (ok) ok = mbar_wait(bar_mma, 0, args.status);
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (ok) {
        tc_fence_after();
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t s[32];
            BSS_TMEM_LD32(tmem + lane_base + cc * 32, s);
            tmem_wait_ld();
            for (int i = 0; i < 32; ++i) args.S[r * 128 + cc * 32 + i] = __uint_as_float(s[i]);
        }
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            BSS_TMEM_LD32(tmem + lane_base + 256 + cc * 32, o);
            tmem_wait_ld();
            for (int i = 0; i < 32; ++i) args.O[r * D + cc * 32 + i] = __uint_as_float(o[i]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
bss_status diag_launch(const void* A, const void* B, const void* P, const void* V, float* S, float* O,
                       cudaStream_t stream) {
    DiagArgs args;
    memset(&args, 0, sizeof(args));
    const uint64_t rs = D * 2;
    bss_status st;
    if ((st = encode_tmap_3d(&args.tm_a, A, D, 128, 1, rs, rs * 128, 64, 128)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_b, B, D, 128, 1, rs, rs * 128, 64, 128)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_v, V, D, 128, 1, rs, rs * 128, 64, 128)) != BSS_OK) return st;
    args.P = static_cast<const uint16_t*>(P);
    args.S = S;
    args.O = O;
    args.status = device_status_ptr();
    if (args.status == nullptr) return set_error(BSS_ERR_CUDA, "cannot resolve the device status word");
    const uint32_t smem = 3 * 128 * D * 2 + 64 + 1024;
    cudaError_t e = cudaFuncSetAttribute(diag_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(diag)");
    diag_kernel<D><<<1, 128, smem, stream>>>(args);
    return cuda_check(cudaGetLastError(), "diag launch");
}

}  // namespace
}  // namespace bss

extern "C" bss_status bss_diag_mma_tile(const void* A, const void* B, const void* P, const void* V, float* S,
                                        float* O, int32_t d, cudaStream_t stream) {
    using namespace bss;
    if (!A || !B || !P || !V || !S || !O) return set_error(BSS_ERR_INVALID_ARG, "NULL pointer");
    const void* ptrs[6] = {A, B, P, V, S, O};
    for (const void* p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return set_error(BSS_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (d == 128) return diag_launch<128>(A, B, P, V, S, O, stream);
    if (d == 64) return diag_launch<64>(A, B, P, V, S, O, stream);
    return set_error(BSS_ERR_UNSUPPORTED, "d must be 64 or 128");
}

namespace bss {
namespace {
// An mbarrier with one expected arrival that never comes: the bounded wait
// must give up, record BSS_ERR_TIMEOUT and return.
__global__ void wait_timeout_kernel(uint64_t limit_ns, int64_t* waited_ns, int* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        const bool ok = mbar_wait(&bar, 0, status, limit_ns);
        const uint64_t t1 = global_timer_ns();
        if (waited_ns != nullptr) *waited_ns = ok ? -1 : static_cast<int64_t>(t1 - t0);
    }
}
}  // namespace
}  // namespace bss

extern "C" bss_status bss_diag_wait_timeout(int64_t limit_ns, int64_t* waited_ns, cudaStream_t stream) {
    using namespace bss;
    if (limit_ns < 1000 || limit_ns > 1000000000ll) return set_error(BSS_ERR_INVALID_ARG, "limit_ns out of range");
    if (waited_ns != nullptr && (reinterpret_cast<uintptr_t>(waited_ns) & 7u))
        return set_error(BSS_ERR_INVALID_ARG, "waited_ns must be 8-byte aligned");
    int* status = device_status_ptr();
    if (status == nullptr) return set_error(BSS_ERR_CUDA, "cannot resolve the device status word");
    wait_timeout_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(limit_ns), waited_ns, status);
    return cuda_check(cudaGetLastError(), "wait timeout launch");
}
