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
// GB300 form: routing is dense attention of the sampled rows under three
// masks, so it runs on the tensor cores in the block-sparse attention kernel's
// routing mode.  The sampled query rows are gathered three times into
// [H][3R][d] (rows [mR, (m+1)R) for mask m: dense, spatial, temporal), so that
// one work item holds every mask's copy of its rows (64 sampled rows: 192 of
// the 256 rows of a two-half item, instead of three one-half items each half
// padding); one launch computes, for every head, the three outputs of those
// rows over every kv tile (each row evaluates its own mask's predicate at its
// own token), with the kv range split so that the launch fills the GPU; each
// split writes its normalised fp32 output and log-sum-exp.  Two
// small kernels follow: one CTA per (sampled row, head) merges the splits
// through their log-sum-exps and sums the row's squared deviations over the
// channels; one CTA per head adds up its rows in a fixed order and sets the
// flag.  (A single merge kernel with one CTA per head took 0.15 ms, 40% of the
// routing time: ten CTAs walking dependent loads.)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "bss_internal.h"
#include "bss_ptx.cuh"

namespace bss {
namespace {

constexpr int kDevThreads = 256;

// Qs[h][m * R + r] = Q[h][rows[r]] for the three masks m (16 bytes per thread);
// a row outside [0, N) is recorded in the status word and replaced by token 0
// (its deviation is skipped)
__global__ void gather_rows_kernel(const uint4* __restrict__ Q, uint4* __restrict__ Qs,
                                   const int32_t* __restrict__ rows, int R, int N, int vec, int* status) {
    const int r = blockIdx.x, h = blockIdx.y;
    int t = __ldg(rows + r);
    if (t < 0 || t >= N) {
        if (threadIdx.x == 0) record_status(status, BSS_ERR_INVALID_ARG);
        t = 0;
    }
    for (int v = threadIdx.x; v < vec; v += blockDim.x) {
        const uint4 x = __ldg(Q + (static_cast<size_t>(h) * N + t) * vec + v);
#pragma unroll
        for (int m = 0; m < 3; ++m) Qs[(static_cast<size_t>(h) * 3 * R + m * R + r) * vec + v] = x;
    }
}

// One CTA per (sampled row, head), one thread per channel: merge the kv splits
// of the dense (m = 0), spatial (1) and temporal (2) outputs of the row,
// O = sum_p O_p exp(LSE_p - LSE) / sum_p exp(LSE_p - LSE), and write the row's
// squared deviations of the masked outputs from the dense one, summed over
// channels, to partial[h][r][0..1] (zero for a row outside [0, N)).  The split
// weights of the row are computed once into shared memory (3 * splits floats
// of dynamic shared memory); each thread then loads its channel of every split
// (the three masks' loads of a split together) and sums them in split order.
template <int D>
__global__ void __launch_bounds__(D) route_merge_kernel(const float* __restrict__ o_f32,
                                                        const float* __restrict__ lse_f32,
                                                        const int32_t* __restrict__ rows, float* __restrict__ partial,
                                                        int H, int R, int N, int splits) {
    extern __shared__ float s_w[];  // [3][splits]: LSE, then weight of each split
    __shared__ float s_mx[3];
    const int r = blockIdx.x, h = blockIdx.y, ch = threadIdx.x;
    const int t = __ldg(rows + r);
    float dev[2] = {0.0f, 0.0f};
    if (t >= 0 && t < N) {
        for (int i = ch; i < 3 * splits; i += D) {
            const int m = i / splits, p = i - m * splits;
            s_w[i] = __ldg(lse_f32 + ((static_cast<int64_t>(m) * H + h) * R + r) * splits + p);
        }
        __syncthreads();
        if (ch < 3) {
            float mx = -INFINITY;
            for (int p = 0; p < splits; ++p) mx = fmaxf(mx, s_w[ch * splits + p]);
            s_mx[ch] = mx;
        }
        __syncthreads();
        for (int i = ch; i < 3 * splits; i += D) {
            const float lp = s_w[i];
            s_w[i] = lp == -INFINITY ? 0.0f : expf(lp - s_mx[i / splits]);
        }
        __syncthreads();
        // the row's splits are contiguous ([3H][R][splits][D]); the three masks'
        // loads of a split are issued together
        const float* src[3];
        float wsum[3] = {0.0f, 0.0f, 0.0f}, acc[3] = {0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int m = 0; m < 3; ++m) src[m] = o_f32 + ((static_cast<int64_t>(m) * H + h) * R + r) * splits * D + ch;
#pragma unroll 4
        for (int p = 0; p < splits; ++p) {
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                const float w = s_w[m * splits + p];
                wsum[m] += w;
                acc[m] += w * __ldg(src[m] + static_cast<int64_t>(p) * D);
            }
        }
        float o[3];
#pragma unroll
        for (int m = 0; m < 3; ++m) o[m] = wsum[m] > 0.0f ? acc[m] / wsum[m] : 0.0f;
        dev[0] = (o[1] - o[0]) * (o[1] - o[0]);
        dev[1] = (o[2] - o[0]) * (o[2] - o[0]);
    }
    __shared__ float red[2][D / 32];
    const int lane = ch & 31, wid = ch >> 5;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float x = dev[k];
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
        if (lane == 0) red[k][wid] = x;
    }
    __syncthreads();
    if (ch < 2) {
        float x = 0.0f;
        for (int w = 0; w < D / 32; ++w) x += red[ch][w];
        partial[(static_cast<int64_t>(h) * R + r) * 2 + ch] = x;
    }
}

// One CTA per head: sum the rows' squared deviations in a fixed order (so the
// result does not depend on scheduling) and route the head to the mask whose
// output deviates less from the dense one.
__global__ void __launch_bounds__(kDevThreads) route_flags_kernel(const float* __restrict__ partial,
                                                                  float* __restrict__ errors,
                                                                  uint8_t* __restrict__ flags, int R) {
    const int h = blockIdx.x;
    float dev[2] = {0.0f, 0.0f};
    for (int r = threadIdx.x; r < R; r += kDevThreads) {
        dev[0] += __ldg(partial + (static_cast<int64_t>(h) * R + r) * 2 + 0);
        dev[1] += __ldg(partial + (static_cast<int64_t>(h) * R + r) * 2 + 1);
    }
    __shared__ float red[2][kDevThreads / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float x = dev[k];
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
        if (lane == 0) red[k][wid] = x;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float e0 = 0.0f, e1 = 0.0f;
        for (int w = 0; w < kDevThreads / 32; ++w) {
            e0 += red[0][w];
            e1 += red[1][w];
        }
        errors[2 * h + 0] = e0;
        errors[2 * h + 1] = e1;
        flags[h] = e1 < e0 ? 1 : 0;
    }
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
    if (R <= 0 || R > 65535) return set_error(BSS_ERR_INVALID_ARG, "R must lie in [1, 65535]");
    const int d = params->head_dim;
    const int S = params->Hs * params->Ws;
    const int N = params->F * S;
    // the 3R virtual rows of a head (its sampled rows once per mask) in 256-row
    // items, or one 128-row half when they fit in it
    const int rows3 = 3 * R;
    const int bq = rows3 <= 128 ? 128 : attention_block_q();
    const int nq = (rows3 + bq - 1) / bq;
    const int nkv = (N + attention_block_kv() - 1) / attention_block_kv();
    // kv splits: enough CTAs for one wave of the GPU
    const int64_t base = static_cast<int64_t>(H) * nq;
    int splits = static_cast<int>(num_sms() / base);
    splits = splits < 1 ? 1 : (splits > nkv ? nkv : splits);
    if (base * splits > 0x7FFFFFFFll) return set_error(BSS_ERR_UNSUPPORTED, "too many routing work items");
    // scratch, stream-ordered: gathered rows, per-split outputs and LSEs
    const size_t q_bytes = static_cast<size_t>(H) * rows3 * d * 2;
    const size_t o_bytes = static_cast<size_t>(splits) * 3 * H * R * d * 4;
    const size_t l_bytes = static_cast<size_t>(splits) * 3 * H * R * 4;
    const size_t p_bytes = static_cast<size_t>(H) * R * 2 * 4;
    uint8_t* scratch = nullptr;
    if ((st = cuda_check(cudaMallocAsync(reinterpret_cast<void**>(&scratch), q_bytes + o_bytes + l_bytes + p_bytes + 512, stream),
                         "routing scratch")) != BSS_OK)
        return st;
    void* qs = scratch;
    float* o32 = reinterpret_cast<float*>(scratch + ((q_bytes + 255) & ~size_t(255)));
    float* l32 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(o32) + o_bytes);
    float* partial = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(l32) + l_bytes);
    int* status = device_status_ptr();
    if (status == nullptr) st = set_error(BSS_ERR_CUDA, "cannot resolve the device status word");
    if (st == BSS_OK) {
        gather_rows_kernel<<<dim3(R, H), 32, 0, stream>>>(static_cast<const uint4*>(Q), static_cast<uint4*>(qs), rows,
                                                          R, N, d / 8, status);
        st = cuda_check(cudaGetLastError(), "routing gather launch");
    }
    if (st == BSS_OK) {
        AttnLaunch a;
        memset(&a, 0, sizeof(a));
        a.Q = qs;
        a.K = K;
        a.V = V;
        a.O = qs;
        a.H = H;
        a.N = N;
        a.d = d;
        a.F = params->F;
        a.S = S;
        a.S_pad = S;
        a.wf = params->spatial_frame_window;
        a.ws = params->temporal_raster_window;
        a.nq = nq;
        a.route = 1;
        a.bq = bq;
        a.Nq = R;
        a.splits = splits;
        a.qmap = rows;
        a.o_f32 = o32;
        a.lse_f32 = l32;
        st = launch_attention(a, stream);
    }
    if (st == BSS_OK) {
        if (d == 128)
            route_merge_kernel<128><<<dim3(R, H), 128, 3 * splits * sizeof(float), stream>>>(o32, l32, rows, partial,
                                                                                              H, R, N, splits);
        else
            route_merge_kernel<64><<<dim3(R, H), 64, 3 * splits * sizeof(float), stream>>>(o32, l32, rows, partial,
                                                                                            H, R, N, splits);
        st = cuda_check(cudaGetLastError(), "routing merge launch");
    }
    if (st == BSS_OK) {
        route_flags_kernel<<<H, kDevThreads, 0, stream>>>(partial, errors, head_is_temporal, R);
        st = cuda_check(cudaGetLastError(), "routing flags launch");
    }
    const bss_status fst = cuda_check(cudaFreeAsync(scratch, stream), "routing scratch free");
    return st != BSS_OK ? st : fst;
}
