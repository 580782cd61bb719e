// bss_api.cu -- the extern "C" entry points declared in include/bss.h:
// argument validation, tile-map handle ownership, TMA descriptor encoding and
// the per-device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_set>

#include "bss_internal.h"

namespace {

__device__ int g_device_status;  // first device-side error since the last read (0 = none)

thread_local char t_last_error[512] = "";

std::mutex g_mutex;
std::unordered_set<const void*> g_live_maps;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool map_is_live(const bss_tile_map m) {
    std::lock_guard<std::mutex> lk(g_mutex);
    return m != nullptr && g_live_maps.count(m) != 0 && m->magic == bss::kMapMagic;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bss_status validate_params(const bss_mask_params* p) {
    using bss::set_error;
    if (p == nullptr) return set_error(BSS_ERR_INVALID_ARG, "params is NULL");
    if (p->F <= 0 || p->Hs <= 0 || p->Ws <= 0)
        return set_error(BSS_ERR_INVALID_ARG, "F, Hs, Ws must be positive (got %d, %d, %d)", p->F, p->Hs, p->Ws);
    const int64_t S = static_cast<int64_t>(p->Hs) * p->Ws;
    const int64_t N = S * p->F;
    if (N > (int64_t(1) << 30)) return set_error(BSS_ERR_UNSUPPORTED, "N = %lld tokens is too large", (long long)N);
    if (p->head_dim != 64 && p->head_dim != 128)
        return set_error(BSS_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", p->head_dim);
    if (p->spatial_frame_window < 0 || p->temporal_raster_window < 0)
        return set_error(BSS_ERR_INVALID_ARG, "mask windows must be >= 0");
    if (p->sink_frames != 1) return set_error(BSS_ERR_UNSUPPORTED, "sink_frames must be 1 (got %d)", p->sink_frames);
    if (p->temporal_permuted != 0 && p->temporal_permuted != 1)
        return set_error(BSS_ERR_INVALID_ARG, "temporal_permuted must be 0 or 1");
    if (p->rounding < 0 || p->rounding > 2) return set_error(BSS_ERR_INVALID_ARG, "rounding must be 0, 1 or 2");
    return BSS_OK;
}

void free_kind(bss::KindMap& k) {
    if (k.d_row_ptr) cudaFree(k.d_row_ptr);
    if (k.d_entries) cudaFree(k.d_entries);
    if (k.d_order) cudaFree(k.d_order);
    if (k.d_colmask) cudaFree(k.d_colmask);
    k.d_row_ptr = k.d_entries = k.d_order = nullptr;
    k.d_colmask = nullptr;
}

}  // namespace

namespace bss {

bss_status set_error(bss_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return st;
}

void clear_error() { t_last_error[0] = '\0'; }

bool tile_map_is_live(const bss_tile_map_s* m) { return map_is_live(const_cast<bss_tile_map>(m)); }

bss_status cuda_check(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return BSS_OK;
    return set_error(e == cudaErrorMemoryAllocation ? BSS_ERR_OOM : BSS_ERR_CUDA, "%s: %s", what,
                     cudaGetErrorString(e));
}

int* device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mutex);
    if (g_status_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

namespace {
bss_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000* out) {
    std::lock_guard<std::mutex> lk(g_mutex);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return set_error(BSS_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return BSS_OK;
}
}  // namespace

bss_status encode_tmap_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t heads,
                          uint64_t row_stride_bytes, uint64_t head_stride_bytes, uint32_t box_inner,
                          uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    bss_status st = encode_fn(&enc);
    if (st != BSS_OK) return st;
    cuuint64_t dims[3] = {inner, rows, heads};
    cuuint64_t strides[2] = {row_stride_bytes, head_stride_bytes};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(BSS_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return BSS_OK;
}

bss_status check_mask_params(const bss_mask_params* p) { return validate_params(p); }

}  // namespace bss

extern "C" {

int32_t bss_version(void) { return 100; }

const char* bss_status_string(bss_status s) {
    switch (s) {
        case BSS_OK: return "BSS_OK";
        case BSS_ERR_INVALID_ARG: return "BSS_ERR_INVALID_ARG";
        case BSS_ERR_UNSUPPORTED: return "BSS_ERR_UNSUPPORTED";
        case BSS_ERR_CUDA: return "BSS_ERR_CUDA";
        case BSS_ERR_TIMEOUT: return "BSS_ERR_TIMEOUT";
        case BSS_ERR_OOM: return "BSS_ERR_OOM";
    }
    return "BSS_ERR_UNKNOWN";
}

const char* bss_last_error_message(void) { return t_last_error; }

bss_status bss_build_tile_map(const bss_mask_params* params, int32_t BQ, int32_t BKV, bss_tile_map* out,
                              cudaStream_t stream) {
    using namespace bss;
    t_last_error[0] = '\0';
    if (out == nullptr) return set_error(BSS_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    bss_status st = validate_params(params);
    if (st != BSS_OK) return st;
    if (BQ < 16 || BQ > 65536 || BKV < 16 || BKV > 65536)
        return set_error(BSS_ERR_INVALID_ARG, "BQ and BKV must lie in [16, 65536] (got %d, %d)", BQ, BKV);
    bss_tile_map m = new (std::nothrow) bss_tile_map_s();
    if (m == nullptr) return set_error(BSS_ERR_OOM, "host allocation failed");
    m->magic = kMapMagic;
    m->p = *params;
    m->BQ = BQ;
    m->BKV = BKV;
    cudaGetDevice(&m->device);
    m->g.F = params->F;
    m->g.S = params->Hs * params->Ws;
    m->g.N = m->g.F * m->g.S;
    m->g.wf = params->spatial_frame_window;
    m->g.ws = params->temporal_raster_window;
    m->g.S_pad = ((m->g.S + BKV - 1) / BKV) * BKV;
    m->nq = (m->g.N + BQ - 1) / BQ;
    const int32_t tcode = params->temporal_permuted ? MASK_TEMPORAL_VIRT : MASK_TEMPORAL_FHW;
    st = build_kind_map(m->g, MASK_SPATIAL, params->rounding, BQ, BKV, m->nq, &m->kind[0], stream);
    if (st == BSS_OK) st = build_kind_map(m->g, tcode, params->rounding, BQ, BKV, m->nq, &m->kind[1], stream);
    if (st != BSS_OK) {
        free_kind(m->kind[0]);
        free_kind(m->kind[1]);
        delete m;
        return st;
    }
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        g_live_maps.insert(m);
    }
    *out = m;
    return BSS_OK;
}

bss_status bss_tile_map_stats(bss_tile_map map, int32_t kind, int64_t* out) {
    using namespace bss;
    if (!map_is_live(map)) return set_error(BSS_ERR_INVALID_ARG, "invalid or destroyed tile map");
    if (kind != 0 && kind != 1) return set_error(BSS_ERR_INVALID_ARG, "kind must be 0 or 1");
    if (out == nullptr) return set_error(BSS_ERR_INVALID_ARG, "out is NULL");
    for (int i = 0; i < BSS_STAT_COUNT; ++i) out[i] = map->kind[kind].stats[i];
    return BSS_OK;
}

bss_status bss_tile_map_dims(bss_tile_map map, int32_t kind, int32_t* out) {
    using namespace bss;
    if (!map_is_live(map)) return set_error(BSS_ERR_INVALID_ARG, "invalid or destroyed tile map");
    if (kind != 0 && kind != 1) return set_error(BSS_ERR_INVALID_ARG, "kind must be 0 or 1");
    if (out == nullptr) return set_error(BSS_ERR_INVALID_ARG, "out is NULL");
    out[0] = map->nq;
    out[1] = map->kind[kind].nkv;
    out[2] = static_cast<int32_t>(map->kind[kind].nnz);
    out[3] = map->kind[kind].ncols;
    return BSS_OK;
}

bss_status bss_tile_map_copy_csr(bss_tile_map map, int32_t kind, int32_t* row_ptr, int32_t* entries) {
    using namespace bss;
    if (!map_is_live(map)) return set_error(BSS_ERR_INVALID_ARG, "invalid or destroyed tile map");
    if (kind != 0 && kind != 1) return set_error(BSS_ERR_INVALID_ARG, "kind must be 0 or 1");
    if (row_ptr == nullptr || entries == nullptr) return set_error(BSS_ERR_INVALID_ARG, "NULL output buffer");
    const KindMap& k = map->kind[kind];
    bss_status st = cuda_check(
        cudaMemcpy(row_ptr, k.d_row_ptr, sizeof(int32_t) * (map->nq + 1), cudaMemcpyDeviceToHost), "copy row_ptr");
    if (st != BSS_OK) return st;
    if (k.nnz > 0)
        st = cuda_check(cudaMemcpy(entries, k.d_entries, sizeof(int32_t) * k.nnz, cudaMemcpyDeviceToHost),
                        "copy entries");
    return st;
}

void bss_destroy_tile_map(bss_tile_map map) {
    if (map == nullptr) return;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        if (g_live_maps.erase(map) == 0) return;
    }
    free_kind(map->kind[0]);
    free_kind(map->kind[1]);
    map->magic = 0;
    delete map;
}

namespace {
bss_status permute_impl(const void* in, void* out, const uint8_t* head_is_temporal, int32_t H,
                        const bss_mask_params* params, int32_t inverse, int32_t only_flagged, cudaStream_t stream) {
    using namespace bss;
    t_last_error[0] = '\0';
    bss_status st = validate_params(params);
    if (st != BSS_OK) return st;
    if (in == nullptr || out == nullptr) return set_error(BSS_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(in) || !aligned16(out)) return set_error(BSS_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    if (H <= 0) return set_error(BSS_ERR_INVALID_ARG, "H must be positive");
    if (inverse != 0 && inverse != 1) return set_error(BSS_ERR_INVALID_ARG, "inverse must be 0 or 1");
    if (only_flagged && head_is_temporal == nullptr)
        return set_error(BSS_ERR_INVALID_ARG, "head_is_temporal is NULL (no head to permute)");
    const int64_t S = static_cast<int64_t>(params->Hs) * params->Ws;
    const int64_t bytes = static_cast<int64_t>(H) * S * params->F * params->head_dim * 2;
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    if (a < b + static_cast<uintptr_t>(bytes) && b < a + static_cast<uintptr_t>(bytes))
        return set_error(BSS_ERR_INVALID_ARG, "in and out overlap");
    return launch_permute(in, out, head_is_temporal, H, params->F, static_cast<int32_t>(S), params->head_dim,
                          inverse, only_flagged, stream);
}
}  // namespace

bss_status bss_permute(const void* in, void* out, const uint8_t* head_is_temporal, int32_t H,
                       const bss_mask_params* params, int32_t inverse, cudaStream_t stream) {
    return permute_impl(in, out, head_is_temporal, H, params, inverse, 0, stream);
}

bss_status bss_permute_flagged(const void* in, void* out, const uint8_t* head_is_temporal, int32_t H,
                               const bss_mask_params* params, int32_t inverse, cudaStream_t stream) {
    return permute_impl(in, out, head_is_temporal, H, params, inverse, 1, stream);
}

bss_status bss_permute_flagged_multi(const void* const* in, void* const* out, int32_t count,
                                     const uint8_t* head_is_temporal, int32_t H, const bss_mask_params* params,
                                     int32_t inverse, cudaStream_t stream) {
    using namespace bss;
    t_last_error[0] = '\0';
    bss_status st = validate_params(params);
    if (st != BSS_OK) return st;
    if (in == nullptr || out == nullptr) return set_error(BSS_ERR_INVALID_ARG, "NULL tensor array");
    if (count < 1 || count > kMaxPermuteTensors)
        return set_error(BSS_ERR_INVALID_ARG, "count must lie in [1, %d]", kMaxPermuteTensors);
    if (H <= 0) return set_error(BSS_ERR_INVALID_ARG, "H must be positive");
    if (inverse != 0 && inverse != 1) return set_error(BSS_ERR_INVALID_ARG, "inverse must be 0 or 1");
    if (head_is_temporal == nullptr) return set_error(BSS_ERR_INVALID_ARG, "head_is_temporal is NULL (no head to permute)");
    const int64_t S = static_cast<int64_t>(params->Hs) * params->Ws;
    const uintptr_t bytes = static_cast<uintptr_t>(static_cast<int64_t>(H) * S * params->F * params->head_dim * 2);
    for (int i = 0; i < count; ++i) {
        if (in[i] == nullptr || out[i] == nullptr) return set_error(BSS_ERR_INVALID_ARG, "NULL tensor");
        if (!aligned16(in[i]) || !aligned16(out[i])) return set_error(BSS_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    }
    // no output may overlap an input or another output
    for (int i = 0; i < count; ++i) {
        const uintptr_t b = reinterpret_cast<uintptr_t>(out[i]);
        for (int j = 0; j < count; ++j) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(in[j]);
            if (a < b + bytes && b < a + bytes) return set_error(BSS_ERR_INVALID_ARG, "an output overlaps an input");
            const uintptr_t c = reinterpret_cast<uintptr_t>(out[j]);
            if (j != i && c < b + bytes && b < c + bytes) return set_error(BSS_ERR_INVALID_ARG, "outputs overlap");
        }
    }
    return launch_permute_multi(in, out, count, head_is_temporal, H, params->F, static_cast<int32_t>(S),
                                params->head_dim, inverse, 1, stream);
}

namespace {
bss_status sparse_attention_impl(const void* Q, const void* K, const void* V, void* O, float* lse, bss_tile_map map,
                                 const uint8_t* head_is_temporal, int32_t H, float softmax_scale, int32_t fused,
                                 cudaStream_t stream, const void* Qt = nullptr, const void* Kt = nullptr,
                                 const void* Vt = nullptr, void* Ot = nullptr) {
    using namespace bss;
    t_last_error[0] = '\0';
    if (!map_is_live(map)) return set_error(BSS_ERR_INVALID_ARG, "invalid or destroyed tile map");
    if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr)
        return set_error(BSS_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return set_error(BSS_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    if (H <= 0) return set_error(BSS_ERR_INVALID_ARG, "H must be positive");
    if (!attention_supports_block_q(map->BQ) || !attention_supports_block_kv(map->BKV))
        return set_error(BSS_ERR_UNSUPPORTED,
                         "attention needs a map built with BQ = 128 or 256 and BKV = 64 or 128 (got %d x %d)",
                         map->BQ, map->BKV);
    if (!std::isfinite(softmax_scale)) return set_error(BSS_ERR_INVALID_ARG, "softmax_scale is not finite");
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev != map->device) return set_error(BSS_ERR_INVALID_ARG, "tile map belongs to device %d", map->device);
    AttnLaunch a;
    memset(&a, 0, sizeof(a));
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.lse = lse;
    a.flags = head_is_temporal;
    a.H = H;
    a.N = map->g.N;
    a.d = map->p.head_dim;
    a.F = map->g.F;
    a.S = map->g.S;
    a.S_pad = map->g.S_pad;
    a.wf = map->g.wf;
    a.ws = map->g.ws;
    a.dense = 0;
    a.nq = map->nq;
    for (int k = 0; k < 2; ++k) {
        a.code[k] = map->kind[k].code;
        a.row_ptr[k] = map->kind[k].d_row_ptr;
        a.entries[k] = map->kind[k].d_entries;
        a.order[k] = map->kind[k].d_order;
        a.colmask[k] = map->kind[k].d_colmask;
        if (map->kind[k].d_colmask != nullptr) a.nsink = map->kind[k].nsink;
    }
    a.softmax_scale = softmax_scale;
    a.fused = fused;
    a.bq = map->BQ;
    a.bkv = map->BKV;
    a.Qt = Qt;
    a.Kt = Kt;
    a.Vt = Vt;
    a.Ot = Ot;
    return launch_attention(a, stream);
}
}  // namespace

bss_status bss_sparse_attention(const void* Q, const void* K, const void* V, void* O, float* lse,
                                bss_tile_map map, const uint8_t* head_is_temporal, int32_t H, float softmax_scale,
                                cudaStream_t stream) {
    return sparse_attention_impl(Q, K, V, O, lse, map, head_is_temporal, H, softmax_scale, 0, stream);
}

bss_status bss_sparse_attention_split(const void* Q, const void* K, const void* V, void* O, const void* Qt,
                                      const void* Kt, const void* Vt, void* Ot, float* lse, bss_tile_map map,
                                      const uint8_t* head_is_temporal, int32_t H, float softmax_scale,
                                      cudaStream_t stream) {
    using namespace bss;
    if (Qt == nullptr || Kt == nullptr || Vt == nullptr)
        return set_error(BSS_ERR_INVALID_ARG, "NULL temporal-head tensor");
    if (!aligned16(Qt) || !aligned16(Kt) || !aligned16(Vt) || (Ot != nullptr && !aligned16(Ot)))
        return set_error(BSS_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    // Ot == NULL: the temporal heads' O rows are written straight to O in (F,H,W) order
    return sparse_attention_impl(Q, K, V, O, lse, map, head_is_temporal, H, softmax_scale, Ot == nullptr ? 2 : 0,
                                 stream, Qt, Kt, Vt, Ot);
}

bss_status bss_sparse_attention_fused(const void* Q, const void* K, const void* V, void* O, float* lse,
                                      bss_tile_map map, const uint8_t* head_is_temporal, int32_t H,
                                      float softmax_scale, cudaStream_t stream) {
    return sparse_attention_impl(Q, K, V, O, lse, map, head_is_temporal, H, softmax_scale, 1, stream);
}

bss_status bss_dense_attention(const void* Q, const void* K, const void* V, void* O, float* lse, int32_t H,
                               int32_t N, int32_t d, float softmax_scale, cudaStream_t stream) {
    using namespace bss;
    t_last_error[0] = '\0';
    if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr)
        return set_error(BSS_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return set_error(BSS_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    if (H <= 0 || N <= 0) return set_error(BSS_ERR_INVALID_ARG, "H and N must be positive");
    if (N > (1 << 30)) return set_error(BSS_ERR_UNSUPPORTED, "N too large");
    if (d != 64 && d != 128) return set_error(BSS_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", d);
    if (!std::isfinite(softmax_scale)) return set_error(BSS_ERR_INVALID_ARG, "softmax_scale is not finite");
    AttnLaunch a;
    memset(&a, 0, sizeof(a));
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.lse = lse;
    a.H = H;
    a.N = N;
    a.d = d;
    a.F = 1;
    a.S = N;
    a.S_pad = N;
    a.dense = 1;
    a.nq = (N + attention_block_q() - 1) / attention_block_q();
    a.code[0] = a.code[1] = MASK_DENSE;
    a.softmax_scale = softmax_scale;
    return launch_attention(a, stream);
}

bss_status bss_get_device_status(cudaStream_t stream) {
    using namespace bss;
    bss_status st = cuda_check(cudaStreamSynchronize(stream), "stream synchronize");
    if (st != BSS_OK) return st;
    int* p = device_status_ptr();
    if (p == nullptr) return set_error(BSS_ERR_CUDA, "cannot resolve the device status word");
    int v = 0;
    st = cuda_check(cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost), "read status");
    if (st != BSS_OK) return st;
    if (v != 0) {
        const int zero = 0;
        st = cuda_check(cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice), "clear status");
        if (st != BSS_OK) return st;
    }
    return static_cast<bss_status>(v);
}

}  // extern "C"
