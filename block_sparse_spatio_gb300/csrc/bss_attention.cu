// bss_attention.cu -- block-sparse flash attention for sm_103a.
//
// Method: blog "Accelerating Spatio-Temporal Attention for Video Diffusion on
// TPUs".  Attention is computed tile by tile, Q[i1:i2] K[j1:j2]^T, with running
// softmax statistics (section "Logical sparsity is not physical sparsity");
// the kernel visits only the non-skipped kv tiles listed for its q tile, runs
// full tiles with no mask at all and evaluates the coordinate predicate only on
// boundary tiles (section "Avoid intra-tile masking when there is nothing to
// mask"), or only the padding predicate on padding tiles of a tile-aligned
// mask (section "Align the sparse mask with final execution"); a tile-aligned
// map of permuted temporal heads also masks, in some sink-segment tiles, the
// frame-0 keys that a kept band tile of the same q tile already holds (a
// per-column bitmask from the map, the same for every row).
//
// GB300 design.  One CTA per (head, 256-row q tile), 384 threads.  The q tile
// is two 128-row halves that share every K/V tile brought into shared memory
// (half the L2 -> SM bytes and TMA operations per FLOP of 128-row tiles) and
// whose softmaxes alternate with each other's MMAs.  A one-half instance
// (128-row tiles, 256 threads, S double-buffered in TMEM) serves 128-row maps,
// and 64-key instances (BKV = 64: S_h of 64 columns, P_h over its first 32, K
// and V stages of 64 rows, a row's tile mask in two words) serve maps with
// 64-key tiles.  The text below describes the default 128-key tiles.
//   warp 0       TMA producer: Q (both halves) once, then K and V tiles of the
//                list into separate kStages-deep rings (128-byte swizzled,
//                64-column boxes).
//   warp 1       TMEM allocator and single-thread tcgen05.mma issuer; it
//                waits with the suspending try_wait, which leaves the issue
//                slots of its SM sub-partition to the softmax warps there.
//                TMEM: S_h (128 fp32 columns) and O_h (D columns) per half h;
//                the bf16 P_h is written over the first 64 columns of S_h.
//                Issue order  S_1(j) PV_0(j) S_0(j+1) PV_1(j) S_1(j+1) ...
//                gives each half's softmax one full MMA tile of time.
//   warps 4..7   softmax of half 0, warps 8..11 softmax of half 1: one thread
//                per query row (= TMEM lane).  Reads S, masks boundary /
//                padding tiles, keeps a reference max with a lazy rescale (a
//                tile is exponentiated against the reference and kept unless a
//                row's sum of P over the tile exceeds 2^16; only then are the
//                max, O and l moved), writes bf16 P to TMEM; finally
//                normalises O, stores it with a TMA store (or, for a permuted
//                temporal head whose permutation the stores undo, row by row
//                to the rows' (F,H,W) positions) and writes the LSE.
// With two halves, warpgroup 0 (warps 0..3) runs at 72 registers a thread and
// the softmax warpgroups at 208 (setmaxnreg), so that the softmax keeps a
// tile's P in registers without spilling.
// tcgen05.mma operations issued by one thread execute in issue order, so an S
// that overwrites P_h is issued after the PV that reads it.  Every mbarrier
// wait is bounded; on a timeout the status word is set and all roles unwind to
// a common exit that frees TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "bss_internal.h"
#include "bss_ptx.cuh"

namespace bss {
namespace {

constexpr int kBQ = 256;        // query rows per CTA of the default shape (two halves of 128)
constexpr int kHalf = 128;      // rows per half = MMA M
constexpr int kBKV = 128;       // key columns per tile of the default shape = MMA N of S
// threads per CTA: producer, MMA and two spare warps, plus four softmax warps
// per 128-row half
template <int HALVES>
constexpr int threads_for() { return 128 * (1 + HALVES); }
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S_h at kColS + 128 h (P_h over its first 64 columns)
constexpr uint32_t kColO = 256;  // O_h at kColO + 128 h
// Lazy rescale.  The fast path exponentiates a tile against the row's reference
// max and keeps the result unless the row's sum of P over the tile exceeds 2^16
// (then no P exceeds 2^16: bf16 P and the fp32 O and l stay far from overflow).
// Checking the sum, which the row needs anyway, instead of a tile max saves one
// instruction per pair of scores.  A tile that fails the check holds a P above
// 2^9, so the general path, which moves the reference when the tile max is more
// than 2^8 above it, always moves it there.
constexpr float kRescaleThreshold = 8.0f;  // log2 units (general path)
constexpr float kSumLimit = 65536.0f;      // fast path

// Register split of the two-half CTA (384 threads launched at 168 registers a
// thread = 64,512): warpgroup 0 (producer, MMA and the two spare warps) gives
// registers back, the two softmax warpgroups take them, so that the softmax
// keeps a whole tile of P in registers without spilling.  setmaxnreg.inc waits
// until enough registers are free, so the split must fit in the launch's
// allocation: 128 * 72 + 256 * 208 = 62,464 <= 64,512; per SM sub-partition
// (one warp of each warpgroup) 72 + 2 * 208 = 488 <= 512 registers a lane.
constexpr uint32_t kRegsControl = 72;
constexpr uint32_t kRegsSoftmax = 208;
constexpr uint32_t kRegsAtLaunch = 168;  // 65,536 / 384 rounded down to a multiple of 8
static_assert(kRegsAtLaunch * 384 <= 65536, "launch allocation");
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= 384 * kRegsAtLaunch,
              "register split exceeds the launch allocation");
static_assert(kRegsControl + 2 * kRegsSoftmax <= 512, "register split exceeds an SM sub-partition");

struct AttnArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_o, tm_ks, tm_vs;
    CUtensorMap tm_qt, tm_kt, tm_vt, tm_ot;  // heads with flag 1 (= the maps above unless split buffers)
    const uint16_t *q_rows, *k_rows, *v_rows;  // Q, K, V as bf16 bits (fused permutation: row gathers)
    uint16_t* o_rows;                 // O as bf16 bits (fused permutation: row-wise stores)
    const int32_t* qmap;              // routing: token index of each query row (mask predicate)
    float* o_f32;                     // routing: [3H][Nq][splits][D] normalised fp32 outputs
    float* lse_f32;                   // routing: [3H][Nq][splits] natural-log LSE
    const int32_t* row_ptr[2];
    const int32_t* entries[2];
    const int32_t* order[2];
    const uint32_t* colmask[2];  // column bitmasks of BSS_CLASS_COLUMNS tiles, [nq][nsink][BKV/32]
    const uint8_t* flags;
    float* lse;
    int* status;
    int32_t code[2];
    int32_t nsink;
    int32_t H, N, nq, F, S, S_pad, wf, ws, dense, nkv_dense;
    int32_t fused;  // 0: none, 1: permutation in loads and stores, 2: in the O stores only
    int32_t route, Nq, splits;  // routing mode: query rows per head, kv splits
    float scale_log2;
};

// Fused permutation: the threads of warps 2 and 3 gather the permuted rows of
// a temporal head's Q and band K / V tiles with 16-byte cp.async copies.
constexpr int kGatherThreads = 64;
constexpr int kGatherThread0 = 64;  // first thread of warp 2

// One 128-row tile of permuted rows p0 .. p0+127 of a head whose (F,H,W) rows
// start at g (already offset by this thread's 16-byte unit): permuted row
// p = s*F + f is row f*S + s of g; rows past the end of the sequence repeat the
// last row (they are padding: query rows are never stored, key columns are
// masked with P = 0).  Thread (unit, rsub) copies unit `unit` of rows rsub,
// rsub + RPR, ... into the 128-byte swizzled layout of a tiled TMA load with
// 64-column boxes: 64-column chunk unit / 8 (chunks chunk_bytes apart), row r
// at r * 128, 16-byte unit (unit % 8) ^ (r % 8).  Consecutive lanes copy
// consecutive units of a row, so a warp instruction reads whole rows.
template <int D, int RPR>
__device__ __forceinline__ void gather_tile(uint32_t sbase, const uint16_t* g, int p0, int rsub, int unit,
                                            const AttnArgs& a) {
    const uint32_t base = sbase + static_cast<uint32_t>(unit >> 3) * kChunkBytesSw128;
    const uint32_t u = static_cast<uint32_t>(unit & 7);
    int p = p0 + rsub;
    int s = p / a.F, f = p - s * a.F;
#pragma unroll 4
    for (int r = rsub; r < kHalf; r += RPR) {
        const int row = p < a.N ? f * a.S + s : a.N - 1;
        cp_async_16(base + static_cast<uint32_t>(r) * 128u + ((u ^ static_cast<uint32_t>(r & 7)) << 4),
                    g + static_cast<size_t>(row) * D);
        p += RPR;
        f += RPR;
        while (f >= a.F) {
            f -= a.F;
            ++s;
        }
    }
}

template <int D, int HALVES = 2, int BKV = kBKV>
struct Smem {
    static constexpr uint32_t kTile = kHalf * D * 2;   // bytes of one 128-row bf16 tile (a q half)
    static constexpr uint32_t kTileKV = BKV * D * 2;   // bytes of one K or V tile
    static constexpr uint32_t kChunkKV = BKV * 128u;  // one 64-column (128-byte) chunk of a K or V tile
    static constexpr uint32_t kQ = 0;                  // the q halves
    static constexpr uint32_t kK = HALVES * kTile;
    static constexpr uint32_t kV = kK + kStages * kTileKV;
    static constexpr uint32_t kBar = kV + kStages * kTileKV;
    // q, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[2], p_full[2], o_done[2], mma_done
    static constexpr uint32_t kNumBars = 1 + 4 * kStages + 2 + 2 + 2 + 1;
    static constexpr uint32_t kBytes = kBar + kNumBars * 8 + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

__device__ __forceinline__ uint32_t bits_range(int lo, int hi) {  // 0 <= lo < hi <= 32
    const uint32_t h = hi >= 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u);
    return h & ~((1u << lo) - 1u);
}

// OR the columns of [lo, hi) that fall inside the tile of NW * 32 columns
// starting at column c0.
template <int NW>
__device__ __forceinline__ void add_interval(uint32_t (&bits)[NW], int lo, int hi, int c0) {
    int l = lo - c0, h = hi - c0;
    l = l < 0 ? 0 : l;
    h = h > NW * 32 ? NW * 32 : h;
    if (h <= l) return;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
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
//   padding tile: the real-column predicate only;
//   column-set tile: the map's bitmask of the tile.
template <int NW>
__device__ __forceinline__ void tile_bits(uint32_t (&bits)[NW], const AttnArgs& a, int code, int cls, int c0,
                                          const RowPred& rp, int kind, int qt) {
#pragma unroll
    for (int w = 0; w < NW; ++w) bits[w] = 0u;
    if (cls >= BSS_CLASS_PAD) {
        if (cls == BSS_CLASS_COLUMNS) {
            const uint32_t* m = a.colmask[kind] + (static_cast<int64_t>(qt) * a.nsink + c0 / (NW * 32)) * NW;
#pragma unroll
            for (int w = 0; w < NW; ++w) bits[w] = __ldg(m + w);
            return;
        }
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
        int f_hi = (c0 + NW * 32 - 1) / a.S;
        f_hi = f_hi > a.F - 1 ? a.F - 1 : f_hi;
        for (int f = f_lo; f <= f_hi; ++f) add_interval(bits, f * a.S + rp.lo, f * a.S + rp.hi, c0);
    } else {
        add_interval(bits, 0, a.N, c0);
    }
}

// j-th kv tile of the work item: from the tile map, or every tile from j0 on
// (dense control and routing: FULL, PAD for a ragged last tile; BOUNDARY for a
// masked routing kind, whose rows are scattered sampled queries)
template <bool ROUTE, int BKV = kBKV>
__device__ __forceinline__ uint32_t entry_at(const AttnArgs& a, const int32_t* ents, int j, int code, int j0) {
    if constexpr (ROUTE) {
        const int t = j0 + j;
        uint32_t cls = (t == a.nkv_dense - 1 && (a.N % BKV) != 0) ? BSS_CLASS_PAD : BSS_CLASS_FULL;
        if (code != MASK_DENSE) cls = BSS_CLASS_BOUNDARY;
        return static_cast<uint32_t>(t) | (cls << BSS_CLASS_SHIFT);
    } else {
        if (a.dense) {
            const uint32_t cls = (j == a.nkv_dense - 1 && (a.N % BKV) != 0) ? BSS_CLASS_PAD : BSS_CLASS_FULL;
            return static_cast<uint32_t>(j) | (cls << BSS_CLASS_SHIFT);
        }
        return static_cast<uint32_t>(__ldg(ents + j));
    }
}

template <int D, bool ROUTE, int HALVES, int BKV = kBKV>
__global__ void __launch_bounds__(threads_for<HALVES>(), 1) attn_fwd_kernel(const __grid_constant__ AttnArgs args) {
    static_assert(HALVES == 1 || HALVES == 2, "one or two 128-row halves per CTA");
    static_assert(BKV == 64 || BKV == 128, "kv tiles of 64 or 128 keys");
    using L = Smem<D, HALVES, BKV>;
    constexpr int kNW = BKV / 32;  // 32-column chunks of a kv tile (words of its row bitmask)
    constexpr int kBQt = HALVES * kHalf;  // query rows per CTA
    constexpr int kChunks = D / 64;  // 64-column (128-byte) swizzle atoms per row

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + L::kQ;
    uint8_t* sK = smem + L::kK;
    uint8_t* sV = smem + L::kV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* bar_q = bars;
    uint64_t* bar_k_full = bars + 1;
    uint64_t* bar_v_full = bar_k_full + kStages;
    uint64_t* bar_k_empty = bar_v_full + kStages;
    uint64_t* bar_v_empty = bar_k_empty + kStages;
    uint64_t* bar_s_full = bar_v_empty + kStages;  // [2] per half
    uint64_t* bar_p_full = bar_s_full + 2;         // [2] per half
    uint64_t* bar_o_done = bar_p_full + 2;         // [2] per half
    uint64_t* bar_mma_done = bar_o_done + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma_done + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int* status = args.status;

    // ---- work item: (head, q tile); heads in order, q tiles longest first.
    // Routing: (head, q tile, kv split) over the head's 3 * Nq virtual query rows
    // (its sampled rows once for each mask: dense, spatial, temporal in (F,H,W)
    // order), every kv tile of the split; each row decodes its own mask.
    const int item = blockIdx.x;
    int h, vh = 0, split = 0, j0 = 0, code;
    bool tbuf = false;  // head with flag 1: its tensors come from the temporal-head buffers
    int qt, n;
    const int32_t* ents = nullptr;
    if constexpr (ROUTE) {
        h = item / (args.nq * args.splits);
        const int rem = item - h * args.nq * args.splits;
        qt = rem / args.splits;
        split = rem - qt * args.splits;
        // the item's rows mix the three masks, so every tile is masked row by row
        // (a masked kind here makes every entry BOUNDARY; rows use their own kind)
        code = static_cast<int>(MASK_SPATIAL);
        j0 = static_cast<int>(static_cast<int64_t>(split) * args.nkv_dense / args.splits);
        n = static_cast<int>(static_cast<int64_t>(split + 1) * args.nkv_dense / args.splits) - j0;
    } else {
        h = item / args.nq;
        const int local = item - h * args.nq;
        int kind = 0;
        if (!args.dense && args.flags != nullptr) kind = args.flags[h] ? 1 : 0;
        tbuf = kind == 1;
        code = args.dense ? static_cast<int>(MASK_DENSE) : args.code[kind];
        if (args.dense) {
            qt = local;
            n = args.nkv_dense;
        } else {
            qt = __ldg(args.order[kind] + local);
            const int rb = __ldg(args.row_ptr[kind] + qt);
            n = __ldg(args.row_ptr[kind] + qt + 1) - rb;
            ents = args.entries[kind] + rb;
        }
    }

    // temporal head whose (H,W,F) permutation is applied by the loads and stores
    // (fused mode 1), or by the output stores only (mode 2: Q, K, V come permuted,
    // O rows go straight to their (F,H,W) positions)
    const bool gather = BKV == 128 && !ROUTE && args.fused == 1 && code == MASK_TEMPORAL_VIRT;
    const bool scatter = gather || (!ROUTE && args.fused == 2 && code == MASK_TEMPORAL_VIRT);
    // a stage filled by the gathering threads completes with one arrival of each
    const uint32_t fill_arrivals = gather ? kGatherThreads : 1;

    if (threadIdx.x == 0) {
        mbar_init(bar_q, fill_arrivals);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_k_full + s, fill_arrivals);
            mbar_init(bar_v_full + s, fill_arrivals);
            mbar_init(bar_k_empty + s, 1);
            mbar_init(bar_v_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_s_full + b, 1);
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

    if (warp < 4) {
        // warpgroup 0: TMA producer, MMA issuer, two spare warps
        if constexpr (HALVES == 2) setmaxnreg_dec<kRegsControl>();
        if (gather && (warp == 2 || warp == 3)) {
            // =========================== gather producer, fused permutation: the 64
            // threads of warps 2-3 copy Q and every band K / V tile row by row
            // (gather_tile) with cp.async; each thread waits for its own copies,
            // makes them visible to the tensor cores' (async) proxy and arrives on
            // the fill's barrier (64 arrivals a fill), one fill behind the copies
            // it issues, so that one fill's copies are in flight while the next is
            // issued.  Measured for 10 temporal heads at 75.6K: 11.6 ms, the same
            // as asynchronous arrivals (cp.async.mbarrier.arrive) with the proxy
            // fence in the MMA issuer, which slowed the kernel's other paths, and
            // faster than two fills in flight (13.8 ms).  Sink tiles (frame-0
            // keys, contiguous in (F,H,W) order) are one box load each (thread 0
            // arms the barrier, the others arrive); the fill still pending is
            // completed before one, because the producer may then wait for a stage
            // that only that fill's consumption frees.
            constexpr int kUnits = D / 8;  // 16-byte units per row
            constexpr int kRPR = kGatherThreads / kUnits;
            const int t = static_cast<int>(threadIdx.x) - kGatherThread0;
            const int unit = t % kUnits, rsub = t / kUnits;
            const size_t head_off = static_cast<size_t>(h) * args.N * D + static_cast<size_t>(unit) * 8;
            const uint16_t* gq = args.q_rows + head_off;
            const uint16_t* gk = args.k_rows + head_off;
            const uint16_t* gv = args.v_rows + head_off;
            uint64_t* pending = nullptr;
            auto complete_pending = [&](bool keep_newest) {
                if (pending == nullptr) return;
                if (keep_newest)
                    cp_async_wait_group<1>();
                else
                    cp_async_wait_group<0>();
                fence_proxy_async_smem();
                mbar_arrive(pending);
                pending = nullptr;
            };
            auto close_fill = [&](uint64_t* bar) {  // after issuing a gathered fill
                cp_async_commit();
                complete_pending(true);
                pending = bar;
            };
            if (t == 0) {
                tma_prefetch_desc(&args.tm_ks);
                tma_prefetch_desc(&args.tm_vs);
            }
#pragma unroll
            for (int hh = 0; hh < HALVES; ++hh)
                gather_tile<D, kRPR>(smem_u32(sQ + hh * L::kTile), gq, qt * kBQt + hh * kHalf, rsub, unit, args);
            close_fill(bar_q);
            bool ok = true;
            int jk = 0, jv = 0;
            for (; jv < n; ++jv) {
                const int st = jv % kStages;
                const uint32_t e = entry_at<ROUTE, BKV>(args, ents, jv, code, j0);
                const int col0 = static_cast<int>(e & BSS_TILE_INDEX_MASK) * BKV;
                const bool sink = col0 < args.S_pad;
                if (sink) complete_pending(false);
                if (jv >= kStages) {
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_k_empty + st, ((jv / kStages) - 1) & 1, status));
                    // the tensor cores' reads of the stage come before these writes
                    fence_proxy_async_smem();
                }
                if (!ok) break;
                if (sink) {
                    if (t == 0) {
                        mbar_arrive_expect_tx(bar_k_full + st, L::kTileKV);
#pragma unroll
                        for (int c = 0; c < kChunks; ++c)
                            tma_load_3d(sK + st * L::kTileKV + c * L::kChunkKV, &args.tm_ks, c * 64, col0, h,
                                        bar_k_full + st);
                    } else {
                        mbar_arrive(bar_k_full + st);
                    }
                } else {
                    gather_tile<D, kRPR>(smem_u32(sK + st * L::kTileKV), gk, col0 - args.S_pad, rsub, unit, args);
                    close_fill(bar_k_full + st);
                }
                jk = jv + 1;
                if (jv >= kStages) {
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_v_empty + st, ((jv / kStages) - 1) & 1, status));
                    fence_proxy_async_smem();
                }
                if (!ok) break;
                if (sink) {
                    if (t == 0) {
                        mbar_arrive_expect_tx(bar_v_full + st, L::kTileKV);
#pragma unroll
                        for (int c = 0; c < kChunks; ++c)
                            tma_load_3d(sV + st * L::kTileKV + c * L::kChunkKV, &args.tm_vs, c * 64, col0, h,
                                        bar_v_full + st);
                    } else {
                        mbar_arrive(bar_v_full + st);
                    }
                } else {
                    gather_tile<D, kRPR>(smem_u32(sV + st * L::kTileKV), gv, col0 - args.S_pad, rsub, unit, args);
                    close_fill(bar_v_full + st);
                }
            }
            // no copy may still be landing in shared memory at exit
            complete_pending(false);
            cp_async_wait_group<0>();
            if (t == 0) {
                mbar_wait(bar_q, 0, status);
                for (int jj = (jk - kStages > 0 ? jk - kStages : 0); jj < jk; ++jj)
                    mbar_wait(bar_k_full + jj % kStages, (jj / kStages) & 1, status);
                for (int jj = (jv - kStages > 0 ? jv - kStages : 0); jj < jv; ++jj)
                    mbar_wait(bar_v_full + jj % kStages, (jj / kStages) & 1, status);
            }
        } else if (warp == 0 && !gather) {
            // =========================== TMA producer
            if (lane == 0) {
                const CUtensorMap* mq = tbuf ? &args.tm_qt : &args.tm_q;
                const CUtensorMap* mk0 = tbuf ? &args.tm_kt : &args.tm_k;
                const CUtensorMap* mv0 = tbuf ? &args.tm_vt : &args.tm_v;
                tma_prefetch_desc(mq);
                tma_prefetch_desc(mk0);
                tma_prefetch_desc(mv0);
                mbar_arrive_expect_tx(bar_q, HALVES * L::kTile);
#pragma unroll
                for (int hh = 0; hh < HALVES; ++hh)
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_3d(sQ + hh * L::kTile + c * kChunkBytesSw128, mq, c * 64, qt * kBQt + hh * kHalf,
                                    h, bar_q);
                bool ok = true;
                int jk = 0, jv = 0;  // K tiles and V tiles issued
                for (; jv < n; ++jv) {
                    const int st = jv % kStages;
                    const uint32_t e = entry_at<ROUTE, BKV>(args, ents, jv, code, j0);
                    const int col0 = static_cast<int>(e & BSS_TILE_INDEX_MASK) * BKV;
                    const CUtensorMap* mk = mk0;
                    const CUtensorMap* mv = mv0;
                    int row = col0;
                    if (code == MASK_TEMPORAL_VIRT) {
                        if (col0 < args.S_pad) {
                            mk = &args.tm_ks;  // frame-0 keys: every F-th permuted row
                            mv = &args.tm_vs;
                        } else {
                            row = col0 - args.S_pad;
                        }
                    }
                    if (jv >= kStages) ok = mbar_wait(bar_k_empty + st, ((jv / kStages) - 1) & 1, status);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar_k_full + st, L::kTileKV);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_3d(sK + st * L::kTileKV + c * L::kChunkKV, mk, c * 64, row, h, bar_k_full + st);
                    jk = jv + 1;
                    if (jv >= kStages) ok = mbar_wait(bar_v_empty + st, ((jv / kStages) - 1) & 1, status);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar_v_full + st, L::kTileKV);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_3d(sV + st * L::kTileKV + c * L::kChunkKV, mv, c * 64, row, h, bar_v_full + st);
                }
                // drain: no copy may still be landing in shared memory at exit
                mbar_wait(bar_q, 0, status);
                for (int jj = (jk - kStages > 0 ? jk - kStages : 0); jj < jk; ++jj)
                    mbar_wait(bar_k_full + jj % kStages, (jj / kStages) & 1, status);
                for (int jj = (jv - kStages > 0 ? jv - kStages : 0); jj < jv; ++jj)
                    mbar_wait(bar_v_full + jj % kStages, (jj / kStages) & 1, status);
            }
        } else if (warp == 1) {
            // =========================== MMA issuer: the whole warp runs the loop (so
            // descriptors stay warp-uniform), one elected lane issues and commits.
            if (n > 0) {
                constexpr uint32_t idesc_qk = idesc_bf16_f32(kHalf, BKV, 0);
                constexpr uint32_t idesc_pv = idesc_bf16_f32(kHalf, D, 1);
                const bool leader = elect_one();
                // base descriptors; K step kk adds (kk / 4) * 16 KiB + (kk % 4) * 32 bytes
                // (K-major) or kk * 2 KiB (MN-major) to the start-address field (>> 4)
                const uint64_t dq0 = desc_kmajor_sw128(smem_u32(sQ), 0);
                const uint64_t dq1 = desc_kmajor_sw128(smem_u32(sQ + L::kTile), 0);
                const uint64_t dk0 = desc_kmajor_sw128(smem_u32(sK), 0, L::kChunkKV);
                const uint64_t dv0 = desc_mnmajor_sw128(smem_u32(sV), 0, L::kChunkKV);
                constexpr uint64_t kStageStep = L::kTileKV >> 4;  // one K or V stage
                auto kstep = [](int kk) -> uint64_t {  // Q: 128-row chunks
                    return static_cast<uint64_t>((kk >> 2) * (kChunkBytesSw128 >> 4) + (kk & 3) * 2);
                };
                auto kstep_kv = [](int kk) -> uint64_t {  // K: BKV-row chunks
                    return static_cast<uint64_t>((kk >> 2) * (L::kChunkKV >> 4) + (kk & 3) * 2);
                };
                auto issue_s = [&](uint32_t d_col, uint64_t dq, uint64_t dk) {
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            umma_ss(tmem + d_col, dq + kstep(kk), dk + kstep_kv(kk), idesc_qk, kk > 0 ? 1u : 0u);
                    }
                };
                auto issue_pv = [&](uint32_t d_col, uint32_t p_col, uint64_t dv, bool acc) {
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < BKV / 16; ++kk)
                            umma_ts(tmem + d_col, tmem + p_col + kk * 8, dv + static_cast<uint64_t>(kk * 128), idesc_pv,
                                    (acc || kk > 0) ? 1u : 0u);
                    }
                };
                auto commit = [&](uint64_t* bar) {
                    if (leader) tc_commit(bar);
                };

                bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_q, 0, status));
                if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_k_full, 0, status));
                if constexpr (HALVES == 1) {
                    // one half: S in two TMEM buffers (columns 0 / 128 by tile parity), so
                    // S(j+1) is issued before PV(j) and overlaps the softmax of tile j;
                    // the P-ready barrier is double-buffered the same way
                    if (ok) {
                        tc_fence_after();
                        issue_s(kColS, dq0, dk0);
                        commit(bar_s_full + 0);
                        commit(bar_k_empty + 0);
                    }
                    for (int j = 0; ok && j < n; ++j) {
                        const int st = j % kStages;
                        if (j + 1 < n) {
                            const int st1 = (j + 1) % kStages;
                            ok = __all_sync(0xFFFFFFFFu,
                                            mbar_wait(bar_k_full + st1, ((j + 1) / kStages) & 1, status));
                            if (!ok) break;
                            tc_fence_after();
                            issue_s(kColS + 128 * ((j + 1) & 1), dq0, dk0 + st1 * kStageStep);
                            commit(bar_s_full + ((j + 1) & 1));
                            commit(bar_k_empty + st1);
                        }
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_v_full + st, (j / kStages) & 1, status));
                        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_p_full + (j & 1), (j >> 1) & 1, status));
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(kColO, kColS + 128 * (j & 1), dv0 + st * kStageStep, j > 0);
                        commit(bar_o_done + 0);
                        commit(bar_v_empty + st);
                    }
                } else {
                    if (ok) {
                        tc_fence_after();
                        issue_s(kColS, dq0, dk0);
                        commit(bar_s_full + 0);
                    }
                    for (int j = 0; ok && j < n; ++j) {
                        const int st = j % kStages;
                        const uint64_t dk = dk0 + st * kStageStep;
                        const uint64_t dv = dv0 + st * kStageStep;
                        // S_1(j): K_j is resident (waited before S_0(j))
                        issue_s(kColS + 128, dq1, dk);
                        commit(bar_s_full + 1);
                        commit(bar_k_empty + st);  // K_j is free once S_0(j) and S_1(j) complete
                        // PV_0(j)
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_v_full + st, (j / kStages) & 1, status));
                        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_p_full + 0, j & 1, status));
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(kColO, kColS, dv, j > 0);
                        commit(bar_o_done + 0);
                        // S_0(j+1)
                        if (j + 1 < n) {
                            const int st1 = (j + 1) % kStages;
                            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_k_full + st1, ((j + 1) / kStages) & 1, status));
                            if (!ok) break;
                            tc_fence_after();
                            issue_s(kColS, dq0, dk0 + st1 * kStageStep);
                            commit(bar_s_full + 0);
                        }
                        // PV_1(j)
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_p_full + 1, j & 1, status));
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(kColO + 128, kColS + 128, dv, j > 0);
                        commit(bar_o_done + 1);
                        commit(bar_v_empty + st);
                    }
                }
                commit(bar_mma_done);
                mbar_wait(bar_mma_done, 0, status);
            }
        }
    } else {
        if constexpr (HALVES == 2) setmaxnreg_inc<kRegsSoftmax>();
        // =========================== softmax + epilogue (one thread per row)
        const int hf = (warp - 4) >> 2;  // half
        const int r = threadIdx.x - 128 - hf * 128;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        // S of this half (two halves), or S buffer 0 of the single half, whose
        // tile j uses buffer j % 2
        const uint32_t t_s0 = tmem + lane_base + kColS + hf * 128;
        const uint32_t t_o = tmem + lane_base + kColO + hf * 128;
        const int q = qt * kBQt + hf * kHalf + r;
        // mask predicate row: the query itself, or (routing) the sampled token of
        // virtual row q = mask * Nq + sampled row, under that mask; the padding
        // rows past 3 * Nq repeat the last one and are not stored
        int qo = q;
        int rcode = code;
        int rr = q;
        if constexpr (ROUTE) {
            int mk = q / args.Nq;
            mk = mk > 2 ? 2 : mk;
            rr = q - mk * args.Nq;
            rr = rr >= args.Nq ? args.Nq - 1 : rr;
            vh = mk * args.H + h;
            rcode = mk == 0 ? static_cast<int>(MASK_DENSE)
                            : (mk == 1 ? static_cast<int>(MASK_SPATIAL) : static_cast<int>(MASK_TEMPORAL_FHW));
            qo = __ldg(args.qmap + rr);
            qo = qo < 0 ? 0 : (qo >= args.N ? args.N - 1 : qo);
        }
        const RowPred rp = row_pred(args, rcode, qo);
        // output row of this query: its own index, or its (F,H,W) position when the
        // kernel applies the permutation
        const int orow = (scatter && q < args.N) ? (q % args.F) * args.S + q / args.F : q;
        const float c = args.scale_log2;
        float m = -INFINITY;
        if constexpr (ROUTE) {
            // The sampled token's own key is retained by all three masks, so its
            // score is at most the row's maximum.  The reference starts there (log2
            // units): every tile can take the single pass from the first one on,
            // and only terms more than 2^126 below the row's maximum can underflow;
            // a tile whose sum of P passes kSumLimit moves the reference up as
            // usual.  Starting from -inf instead sent a warp through the two-pass
            // path at each of its rows' first retained key in the kv split (a
            // temporal row's band starts at a different tile for every row).
            const int qv = q < 3 * args.Nq ? q : 3 * args.Nq - 1;
            const uint4* qr =
                reinterpret_cast<const uint4*>(args.q_rows + (static_cast<int64_t>(h) * 3 * args.Nq + qv) * D);
            const uint4* kr = reinterpret_cast<const uint4*>(args.k_rows + (static_cast<int64_t>(h) * args.N + qo) * D);
            float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll 4
            for (int u = 0; u < D / 8; ++u) {
                const uint4 x = __ldg(qr + u), y = __ldg(kr + u);
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc0 = fmaf(__uint_as_float(xs[k] << 16), __uint_as_float(ys[k] << 16), acc0);
                    acc1 = fmaf(__uint_as_float(xs[k] & 0xFFFF0000u), __uint_as_float(ys[k] & 0xFFFF0000u), acc1);
                }
            }
            m = (acc0 + acc1) * c;
        }
        float l = 0.0f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const uint32_t e = entry_at<ROUTE, BKV>(args, ents, j, code, j0);
            const int cls = static_cast<int>(e >> BSS_CLASS_SHIFT);
            const int c0 = static_cast<int>(e & BSS_TILE_INDEX_MASK) * BKV;
            // one half: the four softmax warps start every tile together.  S(j+1) is
            // issued before PV(j), so without this a warp could run a tile ahead of
            // another; the outputs then came out wrong when rows rescaled O after
            // their first tile (found with keys whose magnitude grows along the
            // sequence), so the warps are kept in step.
            if constexpr (HALVES == 1) named_barrier_sync(3, 128);
            const uint32_t t_s = HALVES == 2 ? t_s0 : t_s0 + 128 * (j & 1);
            if constexpr (HALVES == 2)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_s_full + hf, j & 1, status));
            else
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_s_full + (j & 1), (j >> 1) & 1, status));
            if (!ok) break;
            tc_fence_after();
            // ---- fast path: every row of the warp already has a finite reference
            // max.  One pass: exponentiate against the current reference (FULL tiles
            // without any mask, boundary / padding tiles through their bitmask); the
            // result is kept unless some row's sum of P exceeds kSumLimit (then the
            // tile is redone on the general path).
            bool done = false;
            // one pass over the row's BKV scores; MASKED applies the tile's
            // retained-column bitmask (boundary / padding tiles; a 64-key tile uses
            // the first two words: the parameter has a fixed size because nvcc 13.0
            // crashes on a generic lambda taking an array of a template-dependent
            // size by reference)
            auto single_pass = [&](auto masked_tag, const uint32_t (&bits)[4]) -> bool {
                constexpr bool MASKED = decltype(masked_tag)::value;
                uint32_t pk[BKV / 2];
                uint64_t s2a = 0ull, s2b = 0ull;  // packed partial sums (two chains)
                const uint64_t c2 = f2_pack(c, c);
                // routing lets a row without a reference max (m = -inf) through when
                // none of its columns is retained: exp2(-inf - 0) = 0 for all of them
                const float mref = (ROUTE && m == -INFINITY) ? 0.0f : m;
                const uint64_t nm2 = f2_pack(-mref, -mref);
                // the row's 128 scores in one wait, so that the scheduler has 64
                // independent pairs to interleave with the exponentials (measured:
                // 1.9% faster than a wait per 32-column chunk)
                uint32_t sb[kNW][32];
#pragma unroll
                for (int cc = 0; cc < kNW; ++cc) BSS_TMEM_LD32(t_s + 32 * cc, sb[cc]);
                tmem_wait_ld();
#pragma unroll
                for (int cc = 0; cc < kNW; ++cc) {
                    const uint32_t (&sr)[32] = sb[cc];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float x0 = __uint_as_float(sr[2 * i]), x1 = __uint_as_float(sr[2 * i + 1]);
                        if (MASKED) {
                            x0 = ((bits[cc] >> (2 * i)) & 1u) ? x0 : -INFINITY;
                            x1 = ((bits[cc] >> (2 * i + 1)) & 1u) ? x1 : -INFINITY;
                        }
                        float y0, y1;
                        f2_unpack(f2_fma(f2_pack(x0, x1), c2, nm2), y0, y1);
                        const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
                        const uint64_t pp = f2_pack(p0, p1);
                        if (i & 1)
                            s2b = f2_add(s2b, pp);
                        else
                            s2a = f2_add(s2a, pp);
                        pk[16 * cc + i] = pack_bf16x2(p0, p1);
                    }
                }
                float a0, a1, b0, b1;
                f2_unpack(s2a, a0, a1);
                f2_unpack(s2b, b0, b1);
                const float tsum = (a0 + a1) + (b0 + b1);
                if (__any_sync(0xFFFFFFFFu, tsum > kSumLimit)) return false;
                l += tsum;
                // P in 16-column stores (measured: 1.6% faster than 32-column ones,
                // 1% slower with 8-column ones)
#pragma unroll
                for (int q4 = 0; q4 < kNW; ++q4) BSS_TMEM_ST16(t_s + 16 * q4, (pk + 16 * q4));
                return true;
            };
            if (__all_sync(0xFFFFFFFFu, m != -INFINITY)) {
                if (cls == BSS_CLASS_FULL) {
                    const uint32_t none[4] = {0u, 0u, 0u, 0u};
                    done = single_pass(std::integral_constant<bool, false>(), none);
                } else {
                    uint32_t bits[4];
                    tile_bits<kNW>(*reinterpret_cast<uint32_t(*)[kNW]>(bits), args, rcode, cls, c0, rp, tbuf ? 1 : 0, qt);
                    done = single_pass(std::integral_constant<bool, true>(), bits);
                }
            } else if constexpr (ROUTE) {
                // routing: a kv split often holds no retained key of some sampled rows
                // (a spatial window of other frames), whose reference max then stays
                // -inf for the whole split.  A masked tile takes the single pass when
                // every such row has no retained column in it (its P is 0), instead of
                // sending the whole warp to the two-pass path on every tile.
                if (cls != BSS_CLASS_FULL) {
                    uint32_t bits[4];
                    tile_bits<kNW>(*reinterpret_cast<uint32_t(*)[kNW]>(bits), args, rcode, cls, c0, rp, tbuf ? 1 : 0, qt);
                    uint32_t any = 0u;
#pragma unroll
                    for (int w = 0; w < kNW; ++w) any |= bits[w];
                    if (__all_sync(0xFFFFFFFFu, m != -INFINITY || any == 0u))
                        done = single_pass(std::integral_constant<bool, true>(), bits);
                }
            }
            if (!done) {
                // ---- general path: masking (boundary / padding tiles), first tile of
                // a row, or a reference max that must move.  Pass 1 finds the row max,
                // pass 2 exponentiates and writes P chunk by chunk.
                uint32_t bits[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
                if (cls != BSS_CLASS_FULL)
                    tile_bits<kNW>(*reinterpret_cast<uint32_t(*)[kNW]>(bits), args, rcode, cls, c0, rp, tbuf ? 1 : 0, qt);
                float mx[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) mx[t] = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < kNW; ++cc) {
                    uint32_t sr[32];
                    BSS_TMEM_LD32(t_s + 32 * cc, sr);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float v = ((bits[cc] >> i) & 1u) ? __uint_as_float(sr[i]) : -INFINITY;
                        mx[i & 7] = fmaxf(mx[i & 7], v);
                    }
                }
                const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                const float tmax_s = tmax * c;
                const float m_new = (tmax_s > m + kRescaleThreshold) ? tmax_s : m;
                const float alpha = (m_new == m) ? 1.0f : ex2_approx(m - m_new);
                const float mref = (m_new == -INFINITY) ? 0.0f : m_new;
                // O_h is rescaled only when some row's reference max moved.  With two
                // halves PV_h(j-1) was issued before S_h(j), so it has completed and
                // the wait only orders; with one half S(j) was issued before PV(j-1)
                // and the wait is real.
                if (j >= 1 && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o_done + hf, (j - 1) & 1, status));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        BSS_TMEM_LD32(t_o + cc * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        BSS_TMEM_ST32(t_o + cc * 32, o);
                    }
                }
                // P = exp2(s * scale * log2 e - m) as bf16 pairs, written over the first
                // 64 S columns; 32-column chunk cc lands in columns [16cc, 16cc+16),
                // which chunks <= cc have already been read from.
                float sm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int cc = 0; cc < kNW; ++cc) {
                    uint32_t sr[32];
                    BSS_TMEM_LD32(t_s + 32 * cc, sr);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float x0 = ((bits[cc] >> (2 * i)) & 1u) ? __uint_as_float(sr[2 * i]) : -INFINITY;
                        const float x1 =
                            ((bits[cc] >> (2 * i + 1)) & 1u) ? __uint_as_float(sr[2 * i + 1]) : -INFINITY;
                        const float p0 = ex2_approx(fmaf(x0, c, -mref));
                        const float p1 = ex2_approx(fmaf(x1, c, -mref));
                        sm[(2 * i) & 7] += p0;
                        sm[(2 * i + 1) & 7] += p1;
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    BSS_TMEM_ST16(t_s + 16 * cc, pk);
                }
                const float sum = ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
                l = l * alpha + sum;
                m = m_new;
            }
            tmem_wait_st();
            tc_fence_before();
            // P ready: one barrier per half, or (one half) per tile parity, since a
            // warp may start tile j+1 (its S is issued before PV(j)) while another
            // is still in tile j; it cannot start tile j+2, whose S waits for PV(j)
            mbar_arrive(bar_p_full + (HALVES == 2 ? hf : (j & 1)));
        }
        // ---- epilogue: O / l -> bf16 -> swizzled staging (reuses this half's Q) -> TMA store
        uint8_t* stage = sQ + hf * L::kTile;
        if (ok && n > 0) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o_done + hf, (n - 1) & 1, status));
        // a q tile with no kv tiles (a rounded mask can drop all of them) computes
        // nothing, but its Q load was issued: let it land before the staging
        // buffer, which is this half's Q, is overwritten with the zero rows
        if (ok && n == 0) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_q, 0, status));
        if (ok) {
            tc_fence_after();
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                if (n > 0) {
                    BSS_TMEM_LD32(t_o + cc * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                if constexpr (ROUTE) {
                    // routing: normalised fp32 row of this split
                    if (q < 3 * args.Nq) {
                        float4* dst = reinterpret_cast<float4*>(
                                          args.o_f32 +
                                          ((static_cast<int64_t>(vh) * args.Nq + rr) * args.splits + split) * D) +
                                      cc * 8;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            dst[u] = make_float4(__uint_as_float(o[4 * u]) * inv_l, __uint_as_float(o[4 * u + 1]) * inv_l,
                                                 __uint_as_float(o[4 * u + 2]) * inv_l,
                                                 __uint_as_float(o[4 * u + 3]) * inv_l);
                    }
                } else if (scatter) {
                    // permutation applied by the store: the row goes straight to its
                    // (F,H,W) position
                    if (q < args.N) {
                        uint4* dst = reinterpret_cast<uint4*>(args.o_rows + (static_cast<int64_t>(h) * args.N + orow) * D) +
                                     cc * 4;
#pragma unroll
                        for (int u = 0; u < 4; ++u) dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                } else {
                    // columns [32cc, 32cc+32) = 16-byte units 4*(cc%2) .. +3 of 64-column chunk cc/2
                    uint8_t* chunk = stage + (cc >> 1) * kChunkBytesSw128 + r * 128;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int unit = (cc & 1) * 4 + u;
                        *reinterpret_cast<uint4*>(chunk + ((unit ^ (r & 7)) << 4)) =
                            make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                }
            }
            if constexpr (ROUTE) {
                if (q < 3 * args.Nq) {
                    const float lse = l > 0.0f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
                    args.lse_f32[(static_cast<int64_t>(vh) * args.Nq + rr) * args.splits + split] = lse;
                }
            } else if (args.lse != nullptr && q < args.N) {
                const float lse = l > 0.0f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
                // fused mode: LSE in (F,H,W) order like O; otherwise in layout order
                args.lse[static_cast<int64_t>(h) * args.N + (gather ? orow : q)] = lse;
            }
            fence_proxy_async_smem();
        }
        named_barrier_sync(1 + hf, 128);
        const int row0 = qt * kBQt + hf * kHalf;
        if (r == 0 && ok && row0 < args.N && !scatter && !ROUTE) {
#pragma unroll
            for (int cc = 0; cc < kChunks; ++cc)
                tma_store_3d(tbuf ? &args.tm_ot : &args.tm_o, stage + cc * kChunkBytesSw128, cc * 64, row0, h);
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
    // query rows per head: N, or in routing mode the sampled rows once for each
    // of the three masks
    const int64_t nq_rows = a.route ? 3ll * a.Nq : a.N;
    // keys per kv tile: the map's BKV (routing and the dense control use 128;
    // the fused permutation needs a 128-key map)
    const int bkv = (a.route || a.dense || a.bkv == 0) ? kBKV : a.bkv;
    if (bkv != 64 && bkv != kBKV) return set_error(BSS_ERR_UNSUPPORTED, "kv tile of %d keys", bkv);
    if (a.fused == 1 && bkv != kBKV)
        return set_error(BSS_ERR_UNSUPPORTED, "the fused permutation needs %d-key tiles", kBKV);
    if ((st = encode_tmap_3d(&args.tm_q, a.Q, a.d, nq_rows, a.H, rs, rs * nq_rows, 64, kHalf)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_k, a.K, a.d, a.N, a.H, rs, hs, 64, bkv)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_v, a.V, a.d, a.N, a.H, rs, hs, 64, bkv)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_o, a.route ? a.Q : a.O, a.d, nq_rows, a.H, rs, rs * nq_rows, 64, kHalf)) !=
        BSS_OK)
        return st;
    // frame-0 keys of a temporal head: row s of this view is key (f = 0, s), which
    // is permuted row s*F of a permuted tensor, or row s of an (F,H,W) tensor
    const uint64_t sink_rs = a.fused == 1 ? rs : rs * a.F;
    // heads with flag 1: split buffers if given
    const void* Qt = a.Qt ? a.Qt : a.Q;
    const void* Kt = a.Kt ? a.Kt : a.K;
    const void* Vt = a.Vt ? a.Vt : a.V;
    void* Ot = a.Ot ? a.Ot : (a.route ? const_cast<void*>(a.Q) : a.O);
    if ((st = encode_tmap_3d(&args.tm_qt, Qt, a.d, nq_rows, a.H, rs, rs * nq_rows, 64, kHalf)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_kt, Kt, a.d, a.N, a.H, rs, hs, 64, bkv)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_vt, Vt, a.d, a.N, a.H, rs, hs, 64, bkv)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_ot, Ot, a.d, nq_rows, a.H, rs, rs * nq_rows, 64, kHalf)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_ks, Kt, a.d, a.S, a.H, sink_rs, hs, 64, bkv)) != BSS_OK) return st;
    if ((st = encode_tmap_3d(&args.tm_vs, Vt, a.d, a.S, a.H, sink_rs, hs, 64, bkv)) != BSS_OK) return st;
    if (a.fused == 1 && static_cast<uint64_t>(a.H) * static_cast<uint64_t>(a.N) > 0x7FFFFFFFull)
        return set_error(BSS_ERR_UNSUPPORTED, "H*N too large for the fused permutation");
    args.q_rows = static_cast<const uint16_t*>(a.Q);
    args.k_rows = static_cast<const uint16_t*>(a.K);
    args.v_rows = static_cast<const uint16_t*>(a.V);
    args.o_rows = static_cast<uint16_t*>(a.O);
    args.fused = a.fused;
    args.route = a.route;
    args.qmap = a.qmap;
    args.o_f32 = a.o_f32;
    args.lse_f32 = a.lse_f32;
    args.Nq = a.Nq;
    args.splits = a.route ? a.splits : 1;
    for (int k = 0; k < 2; ++k) {
        args.row_ptr[k] = a.row_ptr[k];
        args.entries[k] = a.entries[k];
        args.order[k] = a.order[k];
        args.colmask[k] = a.colmask[k];
        args.code[k] = a.code[k];
    }
    args.nsink = a.nsink;
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

    // one or two 128-row q halves per CTA: the map's BQ, or the routing call's
    // choice (the dense control uses two)
    const int halves = a.dense ? 2 : a.bq / kHalf;
    if (halves != 1 && halves != 2) return set_error(BSS_ERR_UNSUPPORTED, "query tile of %d rows", a.bq);
    uint32_t smem;
    void (*kernel)(AttnArgs);
    if (bkv == 64) {  // the tile-shape comparison's 64-key tiles (not in routing)
        smem = halves == 2 ? Smem<D, 2, 64>::kAlloc : Smem<D, 1, 64>::kAlloc;
        kernel = halves == 2 ? attn_fwd_kernel<D, false, 2, 64> : attn_fwd_kernel<D, false, 1, 64>;
    } else {
        smem = halves == 2 ? Smem<D, 2>::kAlloc : Smem<D, 1>::kAlloc;
        kernel = a.route ? (halves == 2 ? attn_fwd_kernel<D, true, 2> : attn_fwd_kernel<D, true, 1>)
                         : (halves == 2 ? attn_fwd_kernel<D, false, 2> : attn_fwd_kernel<D, false, 1>);
    }
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(attention)");
    const int64_t items = static_cast<int64_t>(a.H) * a.nq * (a.route ? a.splits : 1);
    if (items <= 0) return BSS_OK;
    if (items > 0x7FFFFFFF) return set_error(BSS_ERR_UNSUPPORTED, "too many work items");
    const int threads = halves == 2 ? threads_for<2>() : threads_for<1>();
    kernel<<<static_cast<unsigned>(items), threads, smem, stream>>>(args);
    return cuda_check(cudaGetLastError(), "attention launch");
}

}  // namespace

int attention_block_q() { return kBQ; }
bool attention_supports_block_q(int bq) { return bq == kHalf || bq == 2 * kHalf; }
int attention_block_kv() { return kBKV; }
bool attention_supports_block_kv(int bkv) { return bkv == 64 || bkv == kBKV; }

bss_status launch_attention(const AttnLaunch& a, cudaStream_t stream) {
    if (a.d == 128) return launch_d<128>(a, stream);
    if (a.d == 64) return launch_d<64>(a, stream);
    return set_error(BSS_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", a.d);
}

}  // namespace bss
