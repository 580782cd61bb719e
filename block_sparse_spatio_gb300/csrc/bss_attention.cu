// bss_attention.cu -- block-sparse flash attention for sm_103a.
//
// Method: blog "Accelerating Spatio-Temporal Attention for Video Diffusion on
// TPUs".  Attention is computed tile by tile, Q[i1:i2] K[j1:j2]^T, with running
// softmax statistics (section "Logical sparsity is not physical sparsity");
// the kernel visits only the non-skipped kv tiles listed for its q tile, runs
// full tiles with no mask at all and evaluates the coordinate predicate only on
// boundary tiles (section "Avoid intra-tile masking when there is nothing to
// mask"), or only the padding predicate on padding tiles of a tile-aligned
// mask (section "Align the sparse mask with final execution").
//
// GB300 design (one CTA per (head, 128-row q tile), 256 threads):
//   warp 0      TMA producer: Q once, then K and V tiles of the list into a
//               KV_STAGES-deep ring (128-byte swizzled, 64-column boxes).
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//               S_j = Q K_j^T into one of two TMEM S buffers, then
//               O += P_{j-1} V_{j-1} with P read from TMEM.
//   warps 4..7  softmax: one thread per query row (= TMEM lane).  Reads S,
//               masks boundary / padding tiles, keeps the running max with a
//               lazy rescale (O and l are rescaled only when the max grows by
//               more than 2^8), writes bf16 P to TMEM, and finally normalises O
//               and stores it with a TMA store; LSE is written directly.
// Every mbarrier wait is bounded; on a timeout the status word is set and all
// roles unwind to a common exit that frees TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "bss_internal.h"
#include "bss_ptx.cuh"

namespace bss {
namespace {

constexpr int kBQ = 128;
constexpr int kBKV = 128;
constexpr int kThreads = 256;
constexpr int kStages = 2;
// TMEM columns: two S buffers, O, two P buffers (bf16 packed two per column)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;  // P buffer b at kColP + 64 * b
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when max grows by > 256x

struct AttnArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_o, tm_ks, tm_vs;
    const int32_t* row_ptr[2];
    const int32_t* entries[2];
    const int32_t* order[2];
    const uint8_t* flags;
    float* lse;
    int* status;
    int32_t code[2];
    int32_t H, N, nq, F, S, S_pad, wf, ws, dense, nkv_dense;
    float scale_log2;
};

template <int D>
struct Smem {
    static constexpr uint32_t kTile = kBQ * D * 2;  // bytes of one 128-row bf16 tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kTile;
    static constexpr uint32_t kV = kTile * (1 + kStages);
    static constexpr uint32_t kBar = kTile * (1 + 2 * kStages);
    static constexpr uint32_t kNumBars = 1 + 3 * kStages + 2 + 2 + 2 + 2 + 1;
    static constexpr uint32_t kBytes = kBar + kNumBars * 8 + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

__device__ __forceinline__ uint32_t bits_range(int lo, int hi) {  // 0 <= lo < hi <= 32
    const uint32_t h = hi >= 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u);
    return h & ~((1u << lo) - 1u);
}

// OR the columns of [lo, hi) that fall inside the tile starting at column c0.
__device__ __forceinline__ void add_interval(uint32_t (&bits)[4], int lo, int hi, int c0) {
    int l = lo - c0, h = hi - c0;
    l = l < 0 ? 0 : l;
    h = h > kBKV ? kBKV : h;
    if (h <= l) return;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        int lw = l - 32 * w, hw = h - 32 * w;
        lw = lw < 0 ? 0 : lw;
        hw = hw > 32 ? 32 : hw;
        if (hw > lw) bits[w] |= bits_range(lw, hw);
    }
}

// Per-row constants of the coordinate predicate.
struct RowPred {
    int lo, hi;  // spatial: band columns; temporal: raster band [a, b)
};

__device__ __forceinline__ RowPred row_pred(const AttnArgs& a, int code, int q) {
    RowPred r{0, 0};
    if (code == MASK_SPATIAL) {
        const int f = q / a.S;
        const int f0 = f - a.wf < 0 ? 0 : f - a.wf;
        const int f1 = f + a.wf > a.F - 1 ? a.F - 1 : f + a.wf;
        r.lo = f0 * a.S;
        r.hi = (f1 + 1) * a.S;
    } else if (code == MASK_TEMPORAL_VIRT || code == MASK_TEMPORAL_FHW) {
        const int s = code == MASK_TEMPORAL_VIRT ? q / a.F : q % a.S;
        r.lo = s - a.ws < 0 ? 0 : s - a.ws;
        r.hi = (s + a.ws > a.S - 1 ? a.S - 1 : s + a.ws) + 1;
    }
    return r;
}

// Retained-column bitmask of one row over the tile starting at column c0.
//   boundary tile: the coordinate predicate (all masks are unions of <= 3
//   intervals except the striped (F,H,W) temporal mask, one interval per frame);
//   padding tile: the real-column predicate only.
__device__ __forceinline__ void tile_bits(uint32_t (&bits)[4], const AttnArgs& a, int code, int cls, int c0,
                                          const RowPred& rp) {
    bits[0] = bits[1] = bits[2] = bits[3] = 0u;
    if (cls == BSS_CLASS_PAD) {
        if (code == MASK_TEMPORAL_VIRT) {
            add_interval(bits, 0, a.S, c0);
            add_interval(bits, a.S_pad, a.S_pad + a.N, c0);
        } else {
            add_interval(bits, 0, a.N, c0);
        }
        return;
    }
    if (code == MASK_SPATIAL) {
        add_interval(bits, 0, a.S, c0);  // first-frame sink
        add_interval(bits, rp.lo, rp.hi, c0);
    } else if (code == MASK_TEMPORAL_VIRT) {
        add_interval(bits, 0, rp.lo, c0);  // sink keys the band misses
        add_interval(bits, rp.hi, a.S, c0);
        add_interval(bits, a.S_pad + rp.lo * a.F, a.S_pad + rp.hi * a.F, c0);
    } else if (code == MASK_TEMPORAL_FHW) {
        add_interval(bits, 0, a.S, c0);  // frame 0 entirely
        int f_lo = c0 / a.S;
        f_lo = f_lo < 1 ? 1 : f_lo;
        int f_hi = (c0 + kBKV - 1) / a.S;
        f_hi = f_hi > a.F - 1 ? a.F - 1 : f_hi;
        for (int f = f_lo; f <= f_hi; ++f) add_interval(bits, f * a.S + rp.lo, f * a.S + rp.hi, c0);
    } else {
        add_interval(bits, 0, a.N, c0);
    }
}

__device__ __forceinline__ uint32_t entry_at(const AttnArgs& a, const int32_t* ents, int j) {
    if (a.dense) {
        const uint32_t cls = (j == a.nkv_dense - 1 && (a.N % kBKV) != 0) ? BSS_CLASS_PAD : BSS_CLASS_FULL;
        return static_cast<uint32_t>(j) | (cls << BSS_CLASS_SHIFT);
    }
    return static_cast<uint32_t>(__ldg(ents + j));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnArgs args) {
    using L = Smem<D>;
    constexpr int kChunks = D / 64;          // 64-column (128-byte) swizzle atoms per row
    constexpr uint32_t kChunkBytes = kBQ * 128;  // one 64-column box of 128 rows

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + L::kQ;
    uint8_t* sK = smem + L::kK;
    uint8_t* sV = smem + L::kV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* bar_q = bars;
    uint64_t* bar_k = bars + 1;
    uint64_t* bar_v = bars + 1 + kStages;
    uint64_t* bar_kv_empty = bars + 1 + 2 * kStages;
    uint64_t* bar_s_full = bars + 1 + 3 * kStages;
    uint64_t* bar_s_free = bar_s_full + 2;
    uint64_t* bar_p_full = bar_s_free + 2;   // [2]: P of tile j in buffer j & 1
    uint64_t* bar_o_done = bar_p_full + 2;   // [2]: PV of tile j committed to j & 1
    uint64_t* bar_mma_done = bar_o_done + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma_done + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int* status = args.status;

    // ---- work item: (head, q tile); heads in order, q tiles longest first
    const int item = blockIdx.x;
    const int h = item / args.nq;
    const int local = item - h * args.nq;
    int kind = 0;
    if (!args.dense && args.flags != nullptr) kind = args.flags[h] ? 1 : 0;
    const int code = args.dense ? static_cast<int>(MASK_DENSE) : args.code[kind];
    int qt, n;
    const int32_t* ents = nullptr;
    if (args.dense) {
        qt = local;
        n = args.nkv_dense;
    } else {
        qt = __ldg(args.order[kind] + local);
        const int rb = __ldg(args.row_ptr[kind] + qt);
        n = __ldg(args.row_ptr[kind] + qt + 1) - rb;
        ents = args.entries[kind] + rb;
    }

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_k + s, 1);
            mbar_init(bar_v + s, 1);
            mbar_init(bar_kv_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_s_full + b, 1);
            mbar_init(bar_s_free + b, 128);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_p_full + b, 128);
            mbar_init(bar_o_done + b, 1);
        }
        mbar_init(bar_mma_done, 1);
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // =========================== TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&args.tm_q);
            tma_prefetch_desc(&args.tm_k);
            tma_prefetch_desc(&args.tm_v);
            mbar_arrive_expect_tx(bar_q, L::kTile);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) tma_load_3d(sQ + c * kChunkBytes, &args.tm_q, c * 64, qt * kBQ, h, bar_q);
            bool ok = true;
            int j = 0;
            for (; j < n; ++j) {
                const int st = j % kStages;
                if (j >= kStages) ok = mbar_wait(bar_kv_empty + st, ((j / kStages) - 1) & 1, status);
                if (!ok) break;
                const uint32_t e = entry_at(args, ents, j);
                const int col0 = static_cast<int>(e & BSS_TILE_INDEX_MASK) * kBKV;
                const CUtensorMap* mk = &args.tm_k;
                const CUtensorMap* mv = &args.tm_v;
                int row = col0;
                if (code == MASK_TEMPORAL_VIRT) {
                    if (col0 < args.S_pad) {
                        mk = &args.tm_ks;  // frame-0 keys: every F-th permuted row
                        mv = &args.tm_vs;
                    } else {
                        row = col0 - args.S_pad;
                    }
                }
                mbar_arrive_expect_tx(bar_k + st, L::kTile);
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    tma_load_3d(sK + st * L::kTile + c * kChunkBytes, mk, c * 64, row, h, bar_k + st);
                mbar_arrive_expect_tx(bar_v + st, L::kTile);
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    tma_load_3d(sV + st * L::kTile + c * kChunkBytes, mv, c * 64, row, h, bar_v + st);
            }
            // drain: no copy may still be landing in shared memory at exit
            mbar_wait(bar_q, 0, status);
            for (int jj = (j - kStages > 0 ? j - kStages : 0); jj < j; ++jj) {
                const int st = jj % kStages;
                mbar_wait(bar_k + st, (jj / kStages) & 1, status);
                mbar_wait(bar_v + st, (jj / kStages) & 1, status);
            }
        }
    } else if (warp == 1) {
        // =========================== MMA issuer (one thread)
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBQ, kBKV, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBQ, D, 1);
            bool ok = n > 0 ? mbar_wait(bar_q, 0, status) : true;
            const uint32_t q_base = smem_u32(sQ);
            for (int j = 0; ok && j <= n; ++j) {
                if (j < n) {
                    const int st = j % kStages;
                    const int b = j & 1;
                    ok = mbar_wait(bar_k + st, (j / kStages) & 1, status);
                    if (ok && j >= 2) ok = mbar_wait(bar_s_free + b, ((j >> 1) - 1) & 1, status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t k_base = smem_u32(sK + st * L::kTile);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_ss(tmem + kColS0 + b * kBKV, desc_kmajor_sw128(q_base, kk),
                                desc_kmajor_sw128(k_base, kk), idesc_qk, kk > 0 ? 1u : 0u);
                    tc_commit(bar_s_full + b);
                }
                if (j >= 1) {
                    const int jp = j - 1;
                    const int st = jp % kStages;
                    ok = mbar_wait(bar_v + st, (jp / kStages) & 1, status);
                    if (ok) ok = mbar_wait(bar_p_full + (jp & 1), (jp >> 1) & 1, status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t v_base = smem_u32(sV + st * L::kTile);
#pragma unroll
                    for (int kk = 0; kk < kBKV / 16; ++kk)
                        umma_ts(tmem + kColO, tmem + kColP + (jp & 1) * 64 + kk * 8, desc_mnmajor_sw128(v_base, kk),
                                idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_kv_empty + st);
                    tc_commit(bar_o_done + (jp & 1));
                }
            }
            tc_commit(bar_mma_done);
            mbar_wait(bar_mma_done, 0, status);
        }
    } else if (warp >= 4) {
        // =========================== softmax + epilogue (one thread per row)
        const int r = threadIdx.x - 128;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int q = qt * kBQ + r;
        const RowPred rp = row_pred(args, code, q);
        const float c = args.scale_log2;
        float m = -INFINITY;
        float l = 0.0f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int b = j & 1;
            const uint32_t e = entry_at(args, ents, j);
            const int cls = static_cast<int>(e >> BSS_CLASS_SHIFT);
            const int c0 = static_cast<int>(e & BSS_TILE_INDEX_MASK) * kBKV;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_s_full + b, (j >> 1) & 1, status));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[128];
            BSS_TMEM_LD32(tmem + lane_base + kColS0 + b * kBKV + 0, (sr + 0));
            BSS_TMEM_LD32(tmem + lane_base + kColS0 + b * kBKV + 32, (sr + 32));
            BSS_TMEM_LD32(tmem + lane_base + kColS0 + b * kBKV + 64, (sr + 64));
            BSS_TMEM_LD32(tmem + lane_base + kColS0 + b * kBKV + 96, (sr + 96));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar_s_free + b);
            float x[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(sr[i]);
            if (cls != BSS_CLASS_FULL) {
                uint32_t bits[4];
                tile_bits(bits, args, code, cls, c0, rp);
#pragma unroll
                for (int i = 0; i < 128; ++i) x[i] = ((bits[i >> 5] >> (i & 31)) & 1u) ? x[i] : -INFINITY;
            }
            // row max with 8 independent chains, then a tree
            float mx[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) mx[t] = x[t];
#pragma unroll
            for (int i = 8; i < 128; ++i) mx[i & 7] = fmaxf(mx[i & 7], x[i]);
            const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            const float tmax_s = tmax * c;
            const float m_new = (tmax_s > m + kRescaleThreshold) ? tmax_s : m;
            const float alpha = (m_new == m) ? 1.0f : ex2_approx(m - m_new);
            const float mref = (m_new == -INFINITY) ? 0.0f : m_new;
            float sm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 8 independent partial sums
            uint32_t pk[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const float p0 = ex2_approx(fmaf(x[2 * i], c, -mref));
                const float p1 = ex2_approx(fmaf(x[2 * i + 1], c, -mref));
                sm[(2 * i) & 7] += p0;
                sm[(2 * i + 1) & 7] += p1;
                pk[i] = pack_bf16x2(p0, p1);
            }
            const float sum = ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
            // O is rescaled only when some row's reference max moved; that needs
            // every earlier PV to have landed.
            if (j >= 1 && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o_done + ((j - 1) & 1), ((j - 1) >> 1) & 1, status));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    BSS_TMEM_LD32(tmem + lane_base + kColO + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    BSS_TMEM_ST32(tmem + lane_base + kColO + cc * 32, o);
                }
            }
            // P buffer b was last read by the PV of tile j - 2
            if (j >= 2) {
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o_done + b, ((j - 2) >> 1) & 1, status));
                if (!ok) break;
                tc_fence_after();
            }
            l = l * alpha + sum;
            m = m_new;
            BSS_TMEM_ST32(tmem + lane_base + kColP + b * 64 + 0, (pk + 0));
            BSS_TMEM_ST32(tmem + lane_base + kColP + b * 64 + 32, (pk + 32));
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_p_full + b);
        }
        // ---- epilogue: O / l -> bf16 -> swizzled staging (reuses the Q tile) -> TMA store
        if (ok && n > 0)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o_done + ((n - 1) & 1), ((n - 1) >> 1) & 1, status));
        if (ok) {
            tc_fence_after();
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                if (n > 0) {
                    BSS_TMEM_LD32(tmem + lane_base + kColO + cc * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                // columns [32cc, 32cc+32) = 16-byte units 4*(cc%2) .. +3 of 64-column chunk cc/2
                uint8_t* chunk = sQ + (cc >> 1) * kChunkBytes + r * 128;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int unit = (cc & 1) * 4 + u;
                    uint4 v = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    *reinterpret_cast<uint4*>(chunk + ((unit ^ (r & 7)) << 4)) = v;
                }
            }
            if (args.lse != nullptr && q < args.N) {
                const float lse = l > 0.0f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
                args.lse[static_cast<int64_t>(h) * args.N + q] = lse;
            }
            fence_proxy_async_smem();
        }
        named_barrier_sync(1, 128);
        if (r == 0 && ok) {
#pragma unroll
            for (int cc = 0; cc < kChunks; ++cc) tma_store_3d(&args.tm_o, sQ + cc * kChunkBytes, cc * 64, qt * kBQ, h);
            tma_store_commit();
            tma_store_wait_read_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
bss_status launch_d(const AttnLaunch& a, cudaStream_t stream) {
    AttnArgs args;
    memset(&args, 0, sizeof(args));
    const uint64_t rs = static_cast<uint64_t>(a.d) * 2;
    const uint64_t hs = rs * static_cast<uint64_t>(a.N);
    bss_status st;
    if ((st = encode_tmap_3d(&args.tm_q, a.Q, a.d, a.N, a.H, rs, hs, 64, kBQ)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_k, a.K, a.d, a.N, a.H, rs, hs, 64, kBKV)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_v, a.V, a.d, a.N, a.H, rs, hs, 64, kBKV)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_o, a.O, a.d, a.N, a.H, rs, hs, 64, kBQ)) != BSS_OK) return st;
    // frame-0 keys of a (H,W,F)-permuted head: row s of this view is permuted row s*F
    if ((st = encode_tmap_3d(&args.tm_ks, a.K, a.d, a.S, a.H, rs * a.F, hs, 64, kBKV)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_vs, a.V, a.d, a.S, a.H, rs * a.F, hs, 64, kBKV)) != BSS_OK) return st;
    for (int k = 0; k < 2; ++k) {
        args.row_ptr[k] = a.row_ptr[k];
        args.entries[k] = a.entries[k];
        args.order[k] = a.order[k];
        args.code[k] = a.code[k];
    }
    args.flags = a.flags;
    args.lse = a.lse;
    args.status = device_status_ptr();
    if (args.status == nullptr) return set_error(BSS_ERR_CUDA, "cannot resolve the device status word");
    args.H = a.H;
    args.N = a.N;
    args.nq = a.nq;
    args.F = a.F;
    args.S = a.S;
    args.S_pad = a.S_pad;
    args.wf = a.wf;
    args.ws = a.ws;
    args.dense = a.dense;
    args.nkv_dense = (a.N + kBKV - 1) / kBKV;
    const float scale = a.softmax_scale > 0.0f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(a.d));
    args.scale_log2 = scale * 1.4426950408889634f;

    const uint32_t smem = Smem<D>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(attention)");
    const int64_t items = static_cast<int64_t>(a.H) * a.nq;
    if (items <= 0) return BSS_OK;
    if (items > 0x7FFFFFFF) return set_error(BSS_ERR_UNSUPPORTED, "too many work items");
    attn_fwd_kernel<D><<<static_cast<unsigned>(items), kThreads, smem, stream>>>(args);
    return cuda_check(cudaGetLastError(), "attention launch");
}

}  // namespace

bss_status launch_attention(const AttnLaunch& a, cudaStream_t stream) {
    if (a.d == 128) return launch_d<128>(a, stream);
    if (a.d == 64) return launch_d<64>(a, stream);
    return set_error(BSS_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", a.d);
}

}  // namespace bss
