// bss_permute.cu -- flag-driven (F,H,W) <-> (H,W,F) token permutation.
//
// Blog "Accelerating Spatio-Temporal Attention for Video Diffusion on TPUs",
// section "Arrange tokens for efficient temporal access" (Figure 9): permuting
// frame-major tokens to temporal-major order puts the same spatial position of
// consecutive frames next to each other; section "Support dynamic routing with
// fixed tensor shapes": a per-head boolean selects the layout, shapes stay
// fixed, and the same flags restore the original order afterwards.
//
// HBM-bound gather: every destination row (d bf16 = 128 or 256 contiguous
// bytes) is read from its source row with 16-byte vector loads; consecutive
// threads cover consecutive 16-byte pieces of consecutive destination rows, so
// both the reads (whole rows) and the writes are fully coalesced.
#include <cuda_runtime.h>

#include <cstdint>

#include "bss_internal.h"

namespace bss {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

template <int VEC_PER_ROW, int UNROLL>
__global__ void __launch_bounds__(256) permute_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                      const uint8_t* __restrict__ flags, int64_t H, int64_t F,
                                                      int64_t S, int inverse) {
    const int64_t N = F * S;
    const int64_t total = H * N * VEC_PER_ROW;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i < total; i += stride * UNROLL) {
        uint4 v[UNROLL];
        int64_t dst[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t idx = i + u * stride;
            dst[u] = -1;
            if (idx < total) {
                const int64_t row = idx / VEC_PER_ROW;
                const int64_t piece = idx - row * VEC_PER_ROW;
                const int64_t h = row / N;
                const int64_t x = row - h * N;  // destination token
                int64_t src = x;
                if (flags != nullptr && flags[h]) {
                    if (!inverse) {  // destination x = s*F + f  <-  source f*S + s
                        const int64_t s = x / F, f = x - s * F;
                        src = f * S + s;
                    } else {  // destination x = f*S + s  <-  source s*F + f
                        const int64_t f = x / S, s = x - f * S;
                        src = s * F + f;
                    }
                }
                v[u] = ld_stream(in + (h * N + src) * VEC_PER_ROW + piece);
                dst[u] = idx;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (dst[u] >= 0) st_stream(out + dst[u], v[u]);
    }
}

}  // namespace

bss_status launch_permute(const void* in, void* out, const uint8_t* flags, int32_t H, int32_t F, int32_t S,
                          int32_t d, int32_t inverse, cudaStream_t stream) {
    const int64_t N = static_cast<int64_t>(F) * S;
    const int threads = 256;
    const int64_t blocks = static_cast<int64_t>(num_sms()) * 8;
    const int64_t total_vec = static_cast<int64_t>(H) * N * (d * 2 / 16);
    if (total_vec == 0) return BSS_OK;
    const int64_t need = (total_vec + threads - 1) / threads;
    const unsigned grid = static_cast<unsigned>(need < blocks ? need : blocks);
    const uint4* src = static_cast<const uint4*>(in);
    uint4* dst = static_cast<uint4*>(out);
    if (d == 128) {
        permute_kernel<16, 4><<<grid, threads, 0, stream>>>(src, dst, flags, H, F, S, inverse);
    } else if (d == 64) {
        permute_kernel<8, 4><<<grid, threads, 0, stream>>>(src, dst, flags, H, F, S, inverse);
    } else {
        return set_error(BSS_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", d);
    }
    return cuda_check(cudaGetLastError(), "permute launch");
}

}  // namespace bss
