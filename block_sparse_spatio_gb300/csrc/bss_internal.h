// bss_internal.h -- host-side structures shared by the library's translation
// units (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime_api.h>

#include <cstdint>

#include "bss.h"

struct bss_tile_map_s;

namespace bss {

constexpr uint64_t kMapMagic = 0x6273735f6d617031ull;  // "bss_map1"

// Mask code used inside kernels: which coordinate predicate a head evaluates.
enum MaskCode : int32_t {
    MASK_SPATIAL = 0,        // frame band + sink, (F,H,W) columns
    MASK_TEMPORAL_VIRT = 1,  // raster band, (H,W,F) rows, sink segment + band columns
    MASK_TEMPORAL_FHW = 2,   // raster band evaluated in (F,H,W) order (striped)
    MASK_DENSE = 3           // every real pair
};

struct KindMap {
    int32_t code;     // MaskCode of this kind
    int32_t nkv;      // kv tiles
    int32_t ncols;    // key columns (N, or S_pad + N)
    int64_t nnz;      // CSR entries
    int32_t* d_row_ptr = nullptr;  // [nq + 1]
    int32_t* d_entries = nullptr;  // [nnz]
    int32_t* d_order = nullptr;    // [nq] q tiles, most entries first
    // rounded maps of permuted temporal heads: retained real columns of every
    // (q tile, sink tile), tile_colmask_words(BKV) words each, [nq][nsink]
    // (BSS_CLASS_COLUMNS entries read theirs); NULL otherwise
    uint32_t* d_colmask = nullptr;
    int32_t nsink = 0;  // sink-segment tiles (S_pad / BKV) of such a map
    int64_t stats[BSS_STAT_COUNT] = {0, 0, 0, 0, 0, 0, 0};
};

// 32-column words of a kv tile's column bitmask
constexpr int tile_colmask_words(int BKV) { return (BKV + 31) / 32; }

struct Geom {
    int32_t F, S, N, wf, ws, S_pad;
};

// tile-map builder (bss_tilemap.cu)
bss_status build_kind_map(const Geom& g, int32_t code, int32_t rounding, int32_t BQ, int32_t BKV, int32_t nq,
                          KindMap* km, cudaStream_t stream);

// the tile-map kernels on caller-provided buffers (bss_tilemap.cu)
void tile_map_geometry(const Geom& geo, int32_t code, int32_t BKV, int64_t* ncols, int64_t* nkv);
bss_status launch_tile_classify(const Geom& geo, int32_t code, int32_t rounding, int32_t BQ, int32_t BKV, int32_t nq,
                                int32_t nkv, uint8_t* cls, int32_t* row_cnt, unsigned long long* stats,
                                cudaStream_t stream);
bss_status launch_tile_compact(int32_t nq, int32_t nkv, const uint8_t* cls, const int32_t* row_ptr, int32_t* entries,
                               cudaStream_t stream);
// rounded maps of permuted temporal heads: drop sink columns whose band twin is
// kept (no-op for other maps); colmask may be NULL
bool tile_map_needs_dedup(int32_t code, int32_t rounding);
bss_status launch_tile_dedup(const Geom& geo, int32_t code, int32_t rounding, int32_t BQ, int32_t BKV, int32_t nq,
                             int32_t nkv, uint8_t* cls, int32_t* row_cnt, unsigned long long* stats, uint32_t* colmask,
                             cudaStream_t stream);

// permutation kernel launch (bss_permute.cu)
// only_flagged: heads whose flag is 0 are not touched (else they are copied)
bss_status launch_permute(const void* in, void* out, const uint8_t* flags, int32_t H, int32_t F, int32_t S,
                          int32_t d, int32_t inverse, int32_t only_flagged, cudaStream_t stream);
// the same for `count` (in, out) pairs in one launch
constexpr int kMaxPermuteTensors = 3;
bss_status launch_permute_multi(const void* const* in, void* const* out, int32_t count, const uint8_t* flags,
                                int32_t H, int32_t F, int32_t S, int32_t d, int32_t inverse, int32_t only_flagged,
                                cudaStream_t stream);

// attention launch (bss_attention.cu)
struct AttnLaunch {
    const void *Q, *K, *V;
    void* O;
    float* lse;
    const uint8_t* flags;
    int32_t H, N, d, F, S, S_pad, wf, ws;
    int32_t code[2];  // mask code of kind 0 / kind 1
    int32_t dense;
    int32_t nq;
    const int32_t* row_ptr[2];
    const int32_t* entries[2];
    const int32_t* order[2];
    const uint32_t* colmask[2];  // per kind: column bitmasks of BSS_CLASS_COLUMNS tiles (or NULL)
    int32_t nsink;               // sink-segment tiles per q tile in colmask
    float softmax_scale;
    // 1: Q, K, V, O and lse are in (F,H,W) token order for every head; the
    // temporal kind's (H,W,F) permutation is applied by the kernel's loads and
    // stores instead of separate permute passes.  2: temporal heads' Q, K, V come
    // permuted (Qt, Kt, Vt) and only their O rows are written straight to their
    // (F,H,W) positions in O (lse stays in layout order).
    int32_t fused;
    // routing mode: 3 x H output heads (dense, spatial, temporal in (F,H,W)
    // order) over Nq sampled query rows per head whose tokens are qmap[r]; Q
    // holds each head's rows once per mask ([H][3 Nq][d], mask-major); every kv
    // tile, split into `splits` ranges; normalised fp32 O and LSE per split
    int32_t route, Nq, splits;
    int32_t bq;   // query rows per CTA: the map's BQ (128 or 256)
    int32_t bkv;  // keys per kv tile: the map's BKV (64 or 128; 0 = 128)
    // split buffers: heads with flag 1 read Qt, Kt, Vt and write Ot (NULL: Q, K, V, O)
    const void *Qt, *Kt, *Vt;
    void* Ot;
    const int32_t* qmap;
    float* o_f32;
    float* lse_f32;
};
bss_status launch_attention(const AttnLaunch& a, cudaStream_t stream);
int attention_block_q();   // query rows per attention tile of the default shape (the map's BQ)
bool attention_supports_block_q(int bq);  // 128 (one MMA half per CTA) or 256 (two)
int attention_block_kv();  // key columns per attention tile of routing and the dense control
bool attention_supports_block_kv(int bkv);  // 64 or 128 for a map-driven call

// helpers (bss_api.cu)
bss_status set_error(bss_status st, const char* fmt, ...);
void clear_error();  // empties the calling thread's last-error message
bool tile_map_is_live(const bss_tile_map_s* m);  // a handle bss_build_tile_map returned and not destroyed
bss_status cuda_check(cudaError_t e, const char* what);
int* device_status_ptr();  // per-device status word (device address)
bss_status encode_tmap_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t heads,
                          uint64_t row_stride_bytes, uint64_t head_stride_bytes, uint32_t box_inner,
                          uint32_t box_rows);
int num_sms();
bss_status check_mask_params(const bss_mask_params* p);  // validation shared by the entry points

}  // namespace bss

struct bss_tile_map_s {
    uint64_t magic;
    bss_mask_params p;
    int32_t BQ, BKV, nq, device;
    bss::Geom g;
    bss::KindMap kind[2];
};
