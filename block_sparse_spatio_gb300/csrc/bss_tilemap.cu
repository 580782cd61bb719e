// bss_tilemap.cu -- tile classification and CSR compaction on the GPU.
//
// Blog "Accelerating Spatio-Temporal Attention for Video Diffusion on TPUs":
// tiles are full (every pair retained, no mask), boundary (mixed, elementwise
// mask) or skipped (nothing retained), section "Logical sparsity is not
// physical sparsity"; with tile-aligned rounding a tile is kept or dropped as
// a whole and only padding is masked, section "Align the sparse mask with
// final execution" (this library keeps a tile iff at least half of its real
// pairs are retained).  Mode 2 reproduces the blog's naive traversal (B1):
// tiles are skipped or visited, and every visited tile evaluates the mask.
//
// Counting uses the closed-form interval structure of each query row's
// retained set (at most three intervals, or one per frame for the striped
// (F,H,W) temporal predicate) intersected with the tile's columns, so the cost
// per tile is O(BQ), independent of BKV.
//
// Tile-aligned maps of permuted temporal heads are rounded in the virtual key
// space, where the frame-0 key at raster v has two columns: sink column v and
// band column S_pad + v*F.  The rounded result is attention over the set of
// physical pairs that the kept tiles cover, so a kept sink tile then drops the
// columns whose band twin lies in a kept tile of the same q tile (class
// COLUMNS, with a per-column bitmask that is the same for every row; SKIP when
// no real column is left).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#include "bss_internal.h"

namespace bss {
namespace {

enum : uint8_t { CLS_FULL = 0, CLS_BOUNDARY = 1, CLS_PAD = 2, CLS_COLUMNS = 3, CLS_SKIP = 4 };

// statistics slot counting the tiles of a class
__host__ __device__ constexpr int stat_of_class(uint8_t k) {
    return k == CLS_SKIP ? BSS_STAT_SKIP : (k == CLS_COLUMNS ? BSS_STAT_COLUMNS : k);
}
static_assert(CLS_FULL == BSS_CLASS_FULL && CLS_BOUNDARY == BSS_CLASS_BOUNDARY && CLS_PAD == BSS_CLASS_PAD &&
                  CLS_COLUMNS == BSS_CLASS_COLUMNS,
              "tile classes are the entry class codes");

struct TmArgs {
    int64_t F, S, N, wf, ws, S_pad;
    int32_t code, rounding, BQ, BKV, nq, nkv;
};

__device__ __forceinline__ int64_t overlap(int64_t lo, int64_t hi, int64_t c0, int64_t c1) {
    lo = lo > c0 ? lo : c0;
    hi = hi < c1 ? hi : c1;
    return hi > lo ? hi - lo : 0;
}

// retained real keys of layout query q among columns [c0, c1)
__device__ int64_t row_count(const TmArgs& g, int64_t q, int64_t c0, int64_t c1) {
    if (g.code == MASK_SPATIAL) {
        const int64_t f = q / g.S;
        const int64_t lo = (f - g.wf > 0 ? f - g.wf : 0) * g.S;
        const int64_t hi = ((f + g.wf < g.F - 1 ? f + g.wf : g.F - 1) + 1) * g.S;
        if (lo <= g.S) return overlap(0, hi, c0, c1);  // band touches the sink frame
        return overlap(0, g.S, c0, c1) + overlap(lo, hi, c0, c1);
    }
    if (g.code == MASK_TEMPORAL_VIRT) {
        const int64_t s = q / g.F;
        const int64_t a = s - g.ws > 0 ? s - g.ws : 0;
        const int64_t b = (s + g.ws < g.S - 1 ? s + g.ws : g.S - 1) + 1;
        return overlap(0, a, c0, c1) + overlap(b, g.S, c0, c1) +
               overlap(g.S_pad + a * g.F, g.S_pad + b * g.F, c0, c1);
    }
    if (g.code == MASK_TEMPORAL_FHW) {
        const int64_t s = q % g.S;
        const int64_t a = s - g.ws > 0 ? s - g.ws : 0;
        const int64_t b = (s + g.ws < g.S - 1 ? s + g.ws : g.S - 1) + 1;
        int64_t cnt = overlap(0, g.S, c0, c1);
        int64_t f_lo = c0 / g.S;
        f_lo = f_lo < 1 ? 1 : f_lo;
        int64_t f_hi = (c1 - 1) / g.S;
        f_hi = f_hi > g.F - 1 ? g.F - 1 : f_hi;
        for (int64_t f = f_lo; f <= f_hi; ++f) cnt += overlap(f * g.S + a, f * g.S + b, c0, c1);
        return cnt;
    }
    return overlap(0, g.N, c0, c1);  // dense
}

__device__ __forceinline__ int64_t real_cols(const TmArgs& g, int64_t c0, int64_t c1) {
    if (g.code == MASK_TEMPORAL_VIRT) return overlap(0, g.S, c0, c1) + overlap(g.S_pad, g.S_pad + g.N, c0, c1);
    return overlap(0, g.N, c0, c1);
}

// One thread per tile: count, classify, accumulate statistics and per-row
// non-skipped counts.  stats: full, boundary, pad, skip, retained, exact retained.
__global__ void classify_kernel(TmArgs g, uint8_t* __restrict__ cls, int32_t* __restrict__ row_cnt,
                                unsigned long long* __restrict__ stats) {
    __shared__ unsigned long long s_stats[BSS_STAT_COUNT];
    if (threadIdx.x < BSS_STAT_COUNT) s_stats[threadIdx.x] = 0ull;
    __syncthreads();
    const int64_t ntiles = static_cast<int64_t>(g.nq) * g.nkv;
    unsigned long long loc[BSS_STAT_COUNT] = {0, 0, 0, 0, 0, 0, 0};
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < ntiles;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t I = t / g.nkv, J = t - I * g.nkv;
        const int64_t c0 = J * g.BKV, c1 = c0 + g.BKV;
        const int64_t q0 = I * g.BQ;
        const int64_t q1 = (q0 + g.BQ < g.N) ? q0 + g.BQ : g.N;
        int64_t c = 0;
        for (int64_t q = q0; q < q1; ++q) c += row_count(g, q, c0, c1);
        const int64_t rr = q1 - q0;
        const int64_t rc = real_cols(g, c0, c1);
        uint8_t k;
        int64_t retained;
        if (g.rounding == 0) {
            k = c == 0 ? CLS_SKIP : ((rc == g.BKV && c == rr * g.BKV) ? CLS_FULL : CLS_BOUNDARY);
            retained = c;
        } else if (g.rounding == 2) {  // every visited tile evaluates the exact mask
            k = c == 0 ? CLS_SKIP : CLS_BOUNDARY;
            retained = c;
        } else {
            const int64_t area = rr * rc;
            const bool kept = area > 0 && 2 * c >= area;
            k = kept ? (rc < g.BKV ? CLS_PAD : CLS_FULL) : CLS_SKIP;
            retained = kept ? area : 0;
        }
        cls[t] = k;
        loc[stat_of_class(k)] += 1;
        loc[BSS_STAT_RETAINED] += static_cast<unsigned long long>(retained);
        loc[BSS_STAT_EXACT_RETAINED] += static_cast<unsigned long long>(c);
        if (k != CLS_SKIP) atomicAdd(row_cnt + I, 1);
    }
#pragma unroll
    for (int i = 0; i < BSS_STAT_COUNT; ++i) {
        unsigned long long v = loc[i];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xFFFFFFFFu, v, o);
        if ((threadIdx.x & 31) == 0 && v) atomicAdd(s_stats + i, v);
    }
    __syncthreads();
    if (threadIdx.x < BSS_STAT_COUNT && s_stats[threadIdx.x]) atomicAdd(stats + threadIdx.x, s_stats[threadIdx.x]);
}

// Rounded maps of permuted temporal heads: one thread per (q tile I, sink tile
// J).  A kept sink tile drops every real column v whose band twin (column
// S_pad + v*F) lies in a kept tile of row I; statistics and row counts follow.
// Only sink tiles are written and only band tiles are read, so the threads of a
// row do not race.  colmask (may be NULL) receives the retained real columns of
// every (I, J), nwords words of 32 columns each, row-major over [nq][nsink].
__global__ void dedup_sink_kernel(TmArgs g, uint8_t* __restrict__ cls, int32_t* __restrict__ row_cnt,
                                  unsigned long long* __restrict__ stats, uint32_t* __restrict__ colmask,
                                  int nwords) {
    const int64_t nsink = g.S_pad / g.BKV;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= static_cast<int64_t>(g.nq) * nsink) return;
    const int64_t I = t / nsink, J = t - I * nsink;
    uint8_t* row = cls + I * g.nkv;
    const uint8_t k = row[J];
    uint32_t* mask = colmask != nullptr ? colmask + t * nwords : nullptr;
    int64_t real = 0, dropped = 0;
    for (int w = 0; w < nwords; ++w) {
        uint32_t bits = 0u;
        if (k != CLS_SKIP) {
            for (int b = 0; b < 32; ++b) {
                const int64_t col = static_cast<int64_t>(w) * 32 + b;
                const int64_t v = J * g.BKV + col;
                if (col >= g.BKV || v >= g.S) break;
                ++real;
                const int64_t twin = g.S_pad + v * g.F;
                if (row[twin / g.BKV] != CLS_SKIP)
                    ++dropped;
                else
                    bits |= 1u << b;
            }
        }
        if (mask != nullptr) mask[w] = bits;
    }
    if (dropped == 0) return;
    const int64_t rr = (I + 1) * g.BQ <= g.N ? g.BQ : g.N - I * g.BQ;
    // unsigned wrap-around: adding 2^64 - x subtracts x
    atomicAdd(stats + BSS_STAT_RETAINED, static_cast<unsigned long long>(-(rr * dropped)));
    atomicAdd(stats + stat_of_class(k), ~0ull);
    if (dropped == real) {
        row[J] = CLS_SKIP;
        atomicAdd(stats + BSS_STAT_SKIP, 1ull);
        atomicAdd(row_cnt + I, -1);
    } else {
        row[J] = CLS_COLUMNS;
        atomicAdd(stats + BSS_STAT_COLUMNS, 1ull);
    }
}

// One warp per q-tile row: write its non-skipped tiles in ascending kv order.
__global__ void compact_kernel(TmArgs g, const uint8_t* __restrict__ cls, const int32_t* __restrict__ row_ptr,
                               int32_t* __restrict__ entries) {
    const int warps_per_block = blockDim.x >> 5;
    const int64_t I = static_cast<int64_t>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (I >= g.nq) return;
    int32_t out = row_ptr[I];
    const uint8_t* row = cls + I * g.nkv;
    for (int32_t j0 = 0; j0 < g.nkv; j0 += 32) {
        const int32_t j = j0 + lane;
        const uint8_t k = j < g.nkv ? row[j] : CLS_SKIP;
        const unsigned keep = __ballot_sync(0xFFFFFFFFu, k != CLS_SKIP);
        if (k != CLS_SKIP) {
            const int pos = __popc(keep & ((1u << lane) - 1u));
            entries[out + pos] = j | (static_cast<int32_t>(k) << BSS_CLASS_SHIFT);
        }
        out += __popc(keep);
    }
}

}  // namespace

void tile_map_geometry(const Geom& geo, int32_t code, int32_t BKV, int64_t* ncols, int64_t* nkv) {
    *ncols = code == MASK_TEMPORAL_VIRT ? static_cast<int64_t>(geo.S_pad) + geo.N : geo.N;
    *nkv = (*ncols + BKV - 1) / BKV;
}

bss_status launch_tile_classify(const Geom& geo, int32_t code, int32_t rounding, int32_t BQ, int32_t BKV, int32_t nq,
                                int32_t nkv, uint8_t* cls, int32_t* row_cnt, unsigned long long* stats,
                                cudaStream_t stream) {
    TmArgs g;
    g.F = geo.F;
    g.S = geo.S;
    g.N = geo.N;
    g.wf = geo.wf;
    g.ws = geo.ws;
    g.S_pad = geo.S_pad;
    g.code = code;
    g.rounding = rounding;
    g.BQ = BQ;
    g.BKV = BKV;
    g.nq = nq;
    g.nkv = nkv;
    const int64_t ntiles = static_cast<int64_t>(nq) * nkv;
    const int threads = 256;
    int64_t blocks = (ntiles + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    classify_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(g, cls, row_cnt, stats);
    return cuda_check(cudaGetLastError(), "classify launch");
}

bool tile_map_needs_dedup(int32_t code, int32_t rounding) { return code == MASK_TEMPORAL_VIRT && rounding == 1; }

bss_status launch_tile_dedup(const Geom& geo, int32_t code, int32_t rounding, int32_t BQ, int32_t BKV, int32_t nq,
                             int32_t nkv, uint8_t* cls, int32_t* row_cnt, unsigned long long* stats, uint32_t* colmask,
                             cudaStream_t stream) {
    if (!tile_map_needs_dedup(code, rounding)) return BSS_OK;
    TmArgs g;
    memset(&g, 0, sizeof(g));
    g.F = geo.F;
    g.S = geo.S;
    g.N = geo.N;
    g.S_pad = geo.S_pad;
    g.code = code;
    g.rounding = rounding;
    g.BQ = BQ;
    g.BKV = BKV;
    g.nq = nq;
    g.nkv = nkv;
    const int64_t n = static_cast<int64_t>(nq) * (geo.S_pad / BKV);
    if (n <= 0) return BSS_OK;
    const int threads = 128;
    dedup_sink_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, stream>>>(
        g, cls, row_cnt, stats, colmask, tile_colmask_words(BKV));
    return cuda_check(cudaGetLastError(), "sink dedup launch");
}

bss_status launch_tile_compact(int32_t nq, int32_t nkv, const uint8_t* cls, const int32_t* row_ptr, int32_t* entries,
                               cudaStream_t stream) {
    TmArgs g;
    memset(&g, 0, sizeof(g));
    g.nq = nq;
    g.nkv = nkv;
    const int threads = 256;
    const int64_t blocks = (static_cast<int64_t>(nq) + (threads / 32) - 1) / (threads / 32);
    if (blocks <= 0) return BSS_OK;
    compact_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(g, cls, row_ptr, entries);
    return cuda_check(cudaGetLastError(), "compact launch");
}

bss_status build_kind_map(const Geom& geo, int32_t code, int32_t rounding, int32_t BQ, int32_t BKV, int32_t nq,
                          KindMap* km, cudaStream_t stream) {
    TmArgs g;
    g.F = geo.F;
    g.S = geo.S;
    g.N = geo.N;
    g.wf = geo.wf;
    g.ws = geo.ws;
    g.S_pad = geo.S_pad;
    g.code = code;
    g.rounding = rounding;
    g.BQ = BQ;
    g.BKV = BKV;
    g.nq = nq;
    const int64_t ncols = code == MASK_TEMPORAL_VIRT ? static_cast<int64_t>(geo.S_pad) + geo.N : geo.N;
    const int64_t nkv = (ncols + BKV - 1) / BKV;
    if (nkv > BSS_TILE_INDEX_MASK) return set_error(BSS_ERR_UNSUPPORTED, "too many kv tiles");
    g.nkv = static_cast<int32_t>(nkv);
    km->code = code;
    km->nkv = g.nkv;
    km->ncols = static_cast<int32_t>(ncols);

    const int64_t ntiles = static_cast<int64_t>(nq) * nkv;
    uint8_t* d_cls = nullptr;
    int32_t* d_cnt = nullptr;
    unsigned long long* d_stats = nullptr;
    bss_status st = BSS_OK;
    std::vector<int32_t> cnt(nq), row_ptr(nq + 1);
    unsigned long long hstats[BSS_STAT_COUNT];
    int64_t nnz = 0;
    if (cudaMalloc(&d_cls, ntiles > 0 ? ntiles : 1) != cudaSuccess || cudaMalloc(&d_cnt, sizeof(int32_t) * nq) != cudaSuccess ||
        cudaMalloc(&d_stats, sizeof(unsigned long long) * BSS_STAT_COUNT) != cudaSuccess) {
        (void)cudaGetLastError();
        st = set_error(BSS_ERR_OOM, "tile map scratch allocation failed");
        goto done;
    }
    if ((st = cuda_check(cudaMemsetAsync(d_cnt, 0, sizeof(int32_t) * nq, stream), "memset")) != BSS_OK) goto done;
    if ((st = cuda_check(cudaMemsetAsync(d_stats, 0, sizeof(unsigned long long) * BSS_STAT_COUNT, stream),
                         "memset")) != BSS_OK)
        goto done;
    {
        const int threads = 256;
        int64_t blocks = (ntiles + threads - 1) / threads;
        const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        classify_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(g, d_cls, d_cnt, d_stats);
        if ((st = cuda_check(cudaGetLastError(), "classify launch")) != BSS_OK) goto done;
    }
    if (tile_map_needs_dedup(code, rounding)) {
        // the kernel reads the column bitmasks of maps it can run (64- or 128-key tiles)
        km->nsink = geo.S_pad / BKV;
        if (BKV == 64 || BKV == 128) {
            const size_t bytes = sizeof(uint32_t) * static_cast<size_t>(nq) * km->nsink * tile_colmask_words(BKV);
            if (cudaMalloc(&km->d_colmask, bytes > 0 ? bytes : 4) != cudaSuccess) {
                (void)cudaGetLastError();
                st = set_error(BSS_ERR_OOM, "tile map column-mask allocation failed");
                goto done;
            }
        }
        if ((st = launch_tile_dedup(geo, code, rounding, BQ, BKV, nq, g.nkv, d_cls, d_cnt, d_stats, km->d_colmask,
                                    stream)) != BSS_OK)
            goto done;
    }
    if ((st = cuda_check(cudaMemcpyAsync(cnt.data(), d_cnt, sizeof(int32_t) * nq, cudaMemcpyDeviceToHost, stream),
                         "copy counts")) != BSS_OK)
        goto done;
    if ((st = cuda_check(cudaMemcpyAsync(hstats, d_stats, sizeof(hstats), cudaMemcpyDeviceToHost, stream),
                         "copy stats")) != BSS_OK)
        goto done;
    if ((st = cuda_check(cudaStreamSynchronize(stream), "tile map classify")) != BSS_OK) goto done;
    row_ptr[0] = 0;
    for (int32_t i = 0; i < nq; ++i) {
        nnz += cnt[i];
        if (nnz > 0x7FFFFFFF) {
            st = set_error(BSS_ERR_UNSUPPORTED, "tile map has more than 2^31 entries");
            goto done;
        }
        row_ptr[i + 1] = static_cast<int32_t>(nnz);
    }
    km->nnz = nnz;
    for (int i = 0; i < BSS_STAT_COUNT; ++i) km->stats[i] = static_cast<int64_t>(hstats[i]);
    {
        // longest-first processing order of q tiles (stable on ties)
        std::vector<int32_t> order(nq);
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return cnt[a] > cnt[b]; });
        if (cudaMalloc(&km->d_row_ptr, sizeof(int32_t) * (nq + 1)) != cudaSuccess ||
            cudaMalloc(&km->d_entries, sizeof(int32_t) * (nnz > 0 ? nnz : 1)) != cudaSuccess ||
            cudaMalloc(&km->d_order, sizeof(int32_t) * (nq > 0 ? nq : 1)) != cudaSuccess) {
            (void)cudaGetLastError();
            st = set_error(BSS_ERR_OOM, "tile map allocation failed");
            goto done;
        }
        if ((st = cuda_check(cudaMemcpyAsync(km->d_row_ptr, row_ptr.data(), sizeof(int32_t) * (nq + 1),
                                             cudaMemcpyHostToDevice, stream),
                             "copy row_ptr")) != BSS_OK)
            goto done;
        if ((st = cuda_check(cudaMemcpyAsync(km->d_order, order.data(), sizeof(int32_t) * nq, cudaMemcpyHostToDevice,
                                             stream),
                             "copy order")) != BSS_OK)
            goto done;
        const int threads = 256;
        const int64_t blocks = (static_cast<int64_t>(nq) + (threads / 32) - 1) / (threads / 32);
        if (blocks > 0) {
            compact_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(g, d_cls, km->d_row_ptr,
                                                                                 km->d_entries);
            if ((st = cuda_check(cudaGetLastError(), "compact launch")) != BSS_OK) goto done;
        }
        if ((st = cuda_check(cudaStreamSynchronize(stream), "tile map compaction")) != BSS_OK) goto done;
    }
done:
    if (d_cls) cudaFree(d_cls);
    if (d_cnt) cudaFree(d_cnt);
    if (d_stats) cudaFree(d_stats);
    return st;
}

}  // namespace bss
