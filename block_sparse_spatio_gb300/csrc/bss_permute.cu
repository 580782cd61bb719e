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
#include <cstring>

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

// blockIdx.y = head; block x covers (256 / VEC_PER_ROW) * UNROLL consecutive
// destination rows in one pass (no grid-stride loop: timed back to back, this
// grid ran 12% faster than a one-wave grid whose blocks loop).  A thread moves one
// 16-byte piece of UNROLL rows, 256 / VEC_PER_ROW rows apart; the source row
// index (one 32-bit division per row) is the only arithmetic.
// blockIdx.z picks one of up to kMaxTensors (in, out) pairs permuted by the
// same flags in one launch (the step's Q, K and V).
struct Tensors {
    const uint4* in[kMaxPermuteTensors];
    uint4* out[kMaxPermuteTensors];
};

template <int VEC_PER_ROW, int UNROLL>
__global__ void __launch_bounds__(256) permute_kernel(const __grid_constant__ Tensors t,
                                                      const uint8_t* __restrict__ flags, uint32_t N, uint32_t F,
                                                      uint32_t S, int inverse, int only_flagged) {
    constexpr uint32_t kRowsPerBlock = 256 / VEC_PER_ROW;
    const uint32_t h = blockIdx.y;
    const bool perm = flags != nullptr && flags[h] != 0;
    if (only_flagged && !perm) return;  // the head's rows stay as they are in `out`
    const uint4* src_h = t.in[blockIdx.z] + static_cast<size_t>(h) * N * VEC_PER_ROW;
    uint4* dst_h = t.out[blockIdx.z] + static_cast<size_t>(h) * N * VEC_PER_ROW;
    const uint32_t piece = threadIdx.x % VEC_PER_ROW;
    const uint32_t row0 = blockIdx.x * (kRowsPerBlock * UNROLL) + threadIdx.x / VEC_PER_ROW;
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const uint32_t x = row0 + u * kRowsPerBlock;  // destination row
        if (x < N) {
            uint32_t src = x;
            if (perm) {
                if (!inverse) {  // destination x = s*F + f  <-  source f*S + s
                    const uint32_t sp = x / F, f = x - sp * F;
                    src = f * S + sp;
                } else {  // destination x = f*S + s  <-  source s*F + f
                    const uint32_t f = x / S, sp = x - f * S;
                    src = sp * F + f;
                }
            }
            v[u] = ld_stream(src_h + static_cast<size_t>(src) * VEC_PER_ROW + piece);
        }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const uint32_t x = row0 + u * kRowsPerBlock;
        if (x < N) st_stream(dst_h + static_cast<size_t>(x) * VEC_PER_ROW + piece, v[u]);
    }
}

}  // namespace

bss_status launch_permute(const void* in, void* out, const uint8_t* flags, int32_t H, int32_t F, int32_t S,
                          int32_t d, int32_t inverse, int32_t only_flagged, cudaStream_t stream) {
    const void* ins[1] = {in};
    void* outs[1] = {out};
    return launch_permute_multi(ins, outs, 1, flags, H, F, S, d, inverse, only_flagged, stream);
}

bss_status launch_permute_multi(const void* const* in, void* const* out, int32_t count, const uint8_t* flags,
                                int32_t H, int32_t F, int32_t S, int32_t d, int32_t inverse, int32_t only_flagged,
                                cudaStream_t stream) {
    const int64_t N = static_cast<int64_t>(F) * S;
    if (N == 0 || H == 0 || count == 0) return BSS_OK;
    if (count < 0 || count > kMaxPermuteTensors)
        return set_error(BSS_ERR_INVALID_ARG, "between 1 and %d tensors per launch", kMaxPermuteTensors);
    if (N > 0xFFFFFFFFll / 16) return set_error(BSS_ERR_UNSUPPORTED, "too many tokens per head");
    if (H > 65535) return set_error(BSS_ERR_UNSUPPORTED, "too many heads (at most 65535)");
    const int threads = 256;
    const int vec = d * 2 / 16;
    constexpr int kUnroll = 4;
    const int64_t rows_per_block = threads / vec;
    const int64_t bx = (N + rows_per_block * kUnroll - 1) / (rows_per_block * kUnroll);
    const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(H), static_cast<unsigned>(count));
    Tensors t;
    memset(&t, 0, sizeof(t));
    for (int i = 0; i < count; ++i) {
        t.in[i] = static_cast<const uint4*>(in[i]);
        t.out[i] = static_cast<uint4*>(out[i]);
    }
    if (d == 128) {
        permute_kernel<16, kUnroll><<<grid, threads, 0, stream>>>(t, flags, static_cast<uint32_t>(N), F, S, inverse,
                                                                 only_flagged);
    } else if (d == 64) {
        permute_kernel<8, kUnroll><<<grid, threads, 0, stream>>>(t, flags, static_cast<uint32_t>(N), F, S, inverse,
                                                                only_flagged);
    } else {
        return set_error(BSS_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", d);
    }
    return cuda_check(cudaGetLastError(), "permute launch");
}

}  // namespace bss
