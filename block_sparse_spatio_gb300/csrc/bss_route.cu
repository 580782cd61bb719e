// bss_route.cu -- per-head routing from sampled queries.
//
// Blog "Accelerating Spatio-Temporal Attention for Video Diffusion on TPUs",
// section "Speeding up attention": Sparse VideoGen profiles the heads at
// inference time by sampling a small number of queries, computing their
// attention outputs under dense, spatial and temporal attention, and routing
// each head to the sparse mask whose output deviates least from the dense one
// (Figure 8: the routing step produces one boolean flag per head).
//
// Reading: the deviation is the squared L2 distance between the masked and the
// dense outputs, summed over the sampled rows and channels; a head is temporal
// iff its temporal deviation is strictly smaller (ties stay spatial).  Masks are
// evaluated in (F,H,W) order (routing runs before the permutation).
//
// Kernel: one CTA of 512 threads per (head, block of kRows sampled rows).  Pass
// 1 finds each row's maximum logit under the three masks; pass 2 forms the
// exponentials of a 512-key chunk (one key per thread) in shared memory and
// accumulates the three outputs per channel (128 channels x 4 key groups),
// reading each V row of the chunk coalesced.  fp32 throughout, exact two-pass
// softmax.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bss_internal.h"
#include "bss_ptx.cuh"

namespace bss {
namespace {

constexpr int kRows = 4;       // sampled rows per CTA
constexpr int kThreads = 512;  // keys per chunk in passes 1 and 2
constexpr int kGroups = 4;     // key groups per channel in the accumulation (kThreads / 128)

struct RouteArgs {
    const __nv_bfloat16* Q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    const int32_t* rows;
    float* errors;  // [H][2]: spatial, temporal
    int* status;
    int32_t R, N, F, S, wf, ws;
    float c;  // softmax scale * log2(e)
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D>
__device__ __forceinline__ void dots(const __nv_bfloat16* krow, const float (*qs)[D], float (&s)[kRows]) {
#pragma unroll
    for (int r = 0; r < kRows; ++r) s[r] = 0.0f;
    const uint4* k4 = reinterpret_cast<const uint4*>(krow);
#pragma unroll 4
    for (int v = 0; v < D / 8; ++v) {
        const uint4 w = __ldg(k4 + v);
        const float k8[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                             bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int e = 0; e < 8; ++e) s[r] = fmaf(qs[r][8 * v + e], k8[e], s[r]);
    }
}

// block-wide max / sum of NV values per thread (kThreads threads)
template <int NV, bool MAX>
__device__ void block_reduce(float (&v)[NV], float* scratch /* [NV][kThreads / 32] */) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        float x = v[i];
        for (int o = 16; o > 0; o >>= 1) {
            const float y = __shfl_xor_sync(0xFFFFFFFFu, x, o);
            x = MAX ? fmaxf(x, y) : x + y;
        }
        if (lane == 0) scratch[i * (kThreads / 32) + wid] = x;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        float x = scratch[i * (kThreads / 32)];
        for (int w = 1; w < kThreads / 32; ++w) {
            const float y = scratch[i * (kThreads / 32) + w];
            x = MAX ? fmaxf(x, y) : x + y;
        }
        v[i] = x;
    }
    __syncthreads();
}

template <int D>
__global__ void __launch_bounds__(kThreads) route_kernel(const RouteArgs a) {
    __shared__ float qs[kRows][D];
    __shared__ int fq[kRows], sq[kRows], valid[kRows], rowix[kRows];
    __shared__ float ps[3][kRows][kThreads];
    __shared__ float red[3 * kRows * (kThreads / 32)];
    const int h = blockIdx.y;
    const int r0 = blockIdx.x * kRows;
    const int t = threadIdx.x;
    const size_t head = static_cast<size_t>(h) * a.N * D;
    if (t < kRows) {
        int row = r0 + t < a.R ? a.rows[r0 + t] : -1;
        if (r0 + t < a.R && (row < 0 || row >= a.N)) {
            record_status(a.status, BSS_ERR_INVALID_ARG);  // sampled row outside [0, N)
            row = -1;
        }
        valid[t] = row >= 0;
        row = row < 0 ? 0 : row;
        fq[t] = row / a.S;
        sq[t] = row % a.S;
        rowix[t] = row;
    }
    __syncthreads();
    for (int i = t; i < kRows * D; i += kThreads) {
        const int r = i / D, e = i % D;
        qs[r][e] = __bfloat162float(a.Q[head + static_cast<size_t>(rowix[r]) * D + e]);
    }
    __syncthreads();

    // mask m: 0 dense, 1 spatial, 2 temporal
    auto keep = [&](int m, int r, int fk, int sk) -> bool {
        if (m == 0) return true;
        if (fk == 0) return true;  // first-frame sink
        if (m == 1) return abs(fk - fq[r]) <= a.wf;
        return abs(sk - sq[r]) <= a.ws;
    };

    // ---- pass 1: maximum logit per (mask, row)
    float mx[3 * kRows];
#pragma unroll
    for (int i = 0; i < 3 * kRows; ++i) mx[i] = -INFINITY;
    for (int k0 = 0; k0 < a.N; k0 += kThreads) {
        const int k = k0 + t;
        if (k < a.N) {
            float s[kRows];
            dots<D>(a.K + head + static_cast<size_t>(k) * D, qs, s);
            const int fk = k / a.S, sk = k - fk * a.S;
#pragma unroll
            for (int r = 0; r < kRows; ++r)
#pragma unroll
                for (int m = 0; m < 3; ++m)
                    if (keep(m, r, fk, sk)) mx[m * kRows + r] = fmaxf(mx[m * kRows + r], s[r] * a.c);
        }
    }
    block_reduce<3 * kRows, true>(mx, red);

    // ---- pass 2: exponentials of a chunk, then per-channel accumulation
    float o[3 * kRows], l[3 * kRows];
#pragma unroll
    for (int i = 0; i < 3 * kRows; ++i) o[i] = l[i] = 0.0f;
    for (int k0 = 0; k0 < a.N; k0 += kThreads) {
        const int k = k0 + t;
        float s[kRows];
        if (k < a.N) {
            dots<D>(a.K + head + static_cast<size_t>(k) * D, qs, s);
            const int fk = k / a.S, sk = k - fk * a.S;
#pragma unroll
            for (int r = 0; r < kRows; ++r)
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    const float p = keep(m, r, fk, sk) ? ex2_approx(s[r] * a.c - mx[m * kRows + r]) : 0.0f;
                    ps[m][r][t] = p;
                    l[m * kRows + r] += p;
                }
        } else {
#pragma unroll
            for (int r = 0; r < kRows; ++r)
#pragma unroll
                for (int m = 0; m < 3; ++m) ps[m][r][t] = 0.0f;
        }
        __syncthreads();
        const int ch = t % 128, grp = t / 128;
        if (ch < D) {
            const int kn = a.N - k0 < kThreads ? a.N - k0 : kThreads;
            for (int j = grp; j < kn; j += kGroups) {
                const float v = __bfloat162float(a.V[head + static_cast<size_t>(k0 + j) * D + ch]);
#pragma unroll
                for (int m = 0; m < 3; ++m)
#pragma unroll
                    for (int r = 0; r < kRows; ++r) o[m * kRows + r] = fmaf(ps[m][r][j], v, o[m * kRows + r]);
            }
        }
        __syncthreads();
    }
    block_reduce<3 * kRows, false>(l, red);
    // combine the key groups' partial outputs per channel
    __shared__ float og[kGroups][3 * kRows][128];
    {
        const int ch = t % 128, grp = t / 128;
#pragma unroll
        for (int i = 0; i < 3 * kRows; ++i) og[grp][i][ch] = o[i];
        __syncthreads();
        if (grp == 0) {
#pragma unroll
            for (int i = 0; i < 3 * kRows; ++i) o[i] = og[0][i][ch] + og[1][i][ch] + og[2][i][ch] + og[3][i][ch];
        }
        __syncthreads();
    }

    // ---- deviations from the dense output, summed over rows and channels
    float dev[2] = {0.0f, 0.0f};
    if (t < D) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            if (!valid[r]) continue;
            const float od = o[r] / l[r];
            const float os = o[kRows + r] / l[kRows + r];
            const float ot = o[2 * kRows + r] / l[2 * kRows + r];
            dev[0] += (os - od) * (os - od);
            dev[1] += (ot - od) * (ot - od);
        }
    }
    block_reduce<2, false>(dev, red);
    if (t == 0) {
        atomicAdd(a.errors + 2 * h + 0, dev[0]);
        atomicAdd(a.errors + 2 * h + 1, dev[1]);
    }
}

__global__ void route_flags_kernel(const float* __restrict__ errors, uint8_t* __restrict__ flags, int H) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h < H) flags[h] = errors[2 * h + 1] < errors[2 * h + 0] ? 1 : 0;
}

}  // namespace
}  // namespace bss

extern "C" bss_status bss_route_heads(const void* Q, const void* K, const void* V, int32_t H,
                                      const bss_mask_params* params, const int32_t* rows, int32_t R,
                                      uint8_t* head_is_temporal, float* errors, cudaStream_t stream) {
    using namespace bss;
    bss_status st = check_mask_params(params);
    if (st != BSS_OK) return st;
    if (!Q || !K || !V || !rows || !head_is_temporal || !errors) return set_error(BSS_ERR_INVALID_ARG, "NULL pointer");
    if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V)) & 15u)
        return set_error(BSS_ERR_INVALID_ARG, "Q, K, V must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(rows) | reinterpret_cast<uintptr_t>(errors)) & 3u)
        return set_error(BSS_ERR_INVALID_ARG, "rows and errors must be 4-byte aligned");
    if (H <= 0 || H > 65535) return set_error(BSS_ERR_INVALID_ARG, "H must lie in [1, 65535]");
    if (R <= 0) return set_error(BSS_ERR_INVALID_ARG, "R must be positive");
    RouteArgs a;
    a.Q = static_cast<const __nv_bfloat16*>(Q);
    a.K = static_cast<const __nv_bfloat16*>(K);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.rows = rows;
    a.errors = errors;
    a.status = device_status_ptr();
    if (a.status == nullptr) return set_error(BSS_ERR_CUDA, "cannot resolve the device status word");
    a.R = R;
    a.S = params->Hs * params->Ws;
    a.F = params->F;
    a.N = a.F * a.S;
    a.wf = params->spatial_frame_window;
    a.ws = params->temporal_raster_window;
    a.c = 1.4426950408889634f / sqrtf(static_cast<float>(params->head_dim));
    if ((st = cuda_check(cudaMemsetAsync(errors, 0, sizeof(float) * 2 * H, stream), "clear errors")) != BSS_OK)
        return st;
    const dim3 grid((R + kRows - 1) / kRows, H);
    if (params->head_dim == 128)
        route_kernel<128><<<grid, kThreads, 0, stream>>>(a);
    else
        route_kernel<64><<<grid, kThreads, 0, stream>>>(a);
    if ((st = cuda_check(cudaGetLastError(), "route launch")) != BSS_OK) return st;
    route_flags_kernel<<<(H + 127) / 128, 128, 0, stream>>>(errors, head_is_temporal, H);
    return cuda_check(cudaGetLastError(), "route flags launch");
}
