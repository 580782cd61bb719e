// bss_step.cu -- the per-layer path as library calls.
//
// Blog "Accelerating Spatio-Temporal Attention for Video Diffusion on TPUs",
// Figure 8 and section "Support dynamic routing with fixed tensor shapes": per
// layer, the routing flags pick each head's mask, the temporal heads' tokens
// are permuted to (H,W,F) order, block-sparse attention runs, and the same
// flags restore the token order.
//
// bss_attention_step chains that path on device buffers: the temporal heads'
// Q, K, V are permuted into caller workspaces (one launch for the three) and
// the split attention reads
// the spatial heads in place and stores every temporal head's O row straight
// to its (F,H,W) row.  bss_attention_step_host runs the same chain from pinned
// host buffers: a library-owned workspace holds `depth` device buffer sets and
// two copy streams, and every call copies its inputs in, computes and copies O
// out in groups of heads (heads are independent), so that a group's kernels
// start while the next group is still being copied and the copies of one call
// overlap the kernels of the previous one.  Odd groups compute on a second
// stream, so a group's launches can start on the SMs that the previous group's
// attention leaves idle at its end.  Every copy is one cudaMemcpyAsync; events
// order the four streams.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>

#include "bss_internal.h"

namespace {

constexpr uint64_t kWsMagic = 0x6273735f73746570ull;  // "bss_step"
constexpr int kMaxDepth = 8;

struct StepSet {
    void *Q = nullptr, *K = nullptr, *V = nullptr, *O = nullptr, *Qp = nullptr, *Kp = nullptr, *Vp = nullptr;
    uint8_t* flags = nullptr;
    cudaEvent_t free_ev = nullptr;  // the set's previous call is done (kernels and D2H copy)
    bool used = false;
    std::vector<cudaEvent_t> ready, done;  // per head group: inputs copied / outputs computed
};

std::mutex g_ws_mutex;
std::unordered_set<const void*> g_live_ws;

}  // namespace

struct bss_step_workspace_s {
    uint64_t magic;
    int32_t H, N, d, F, S, device, depth, group, ngroups, next;
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    // odd head groups run on this stream, even ones on the caller's, so that a
    // group's kernels can start while the previous group's attention drains
    cudaStream_t compute2 = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::vector<StepSet> sets;
};

namespace {

bool ws_is_live(const bss_step_workspace w) {
    std::lock_guard<std::mutex> lk(g_ws_mutex);
    return w != nullptr && g_live_ws.count(w) != 0 && w->magic == kWsMagic;
}

void free_workspace(bss_step_workspace w) {
    if (w->copy_in) cudaStreamSynchronize(w->copy_in);
    if (w->copy_out) cudaStreamSynchronize(w->copy_out);
    if (w->compute2) cudaStreamSynchronize(w->compute2);
    for (StepSet& s : w->sets) {
        if (s.free_ev) cudaEventSynchronize(s.free_ev);
        for (void* p : {s.Q, s.K, s.V, s.O, s.Qp, s.Kp, s.Vp})
            if (p) cudaFree(p);
        if (s.flags) cudaFree(s.flags);
        if (s.free_ev) cudaEventDestroy(s.free_ev);
        for (cudaEvent_t e : s.ready)
            if (e) cudaEventDestroy(e);
        for (cudaEvent_t e : s.done)
            if (e) cudaEventDestroy(e);
    }
    if (w->copy_in) cudaStreamDestroy(w->copy_in);
    if (w->copy_out) cudaStreamDestroy(w->copy_out);
    if (w->compute2) cudaStreamDestroy(w->compute2);
    if (w->fork) cudaEventDestroy(w->fork);
    if (w->join) cudaEventDestroy(w->join);
    w->magic = 0;
    delete w;
}

// The step on device buffers, with no argument checks of its own beyond the
// calls it makes (each validates its arguments before launching).
bss_status step_device(const void* Q, const void* K, const void* V, void* O, float* lse, bss_tile_map map,
                       const uint8_t* flags, int32_t H, void* Qp, void* Kp, void* Vp, cudaStream_t stream) {
    // no flags (every head spatial), or temporal heads kept in (F,H,W) order:
    // nothing to permute
    if (flags == nullptr || !map->p.temporal_permuted)
        return bss_sparse_attention(Q, K, V, O, lse, map, flags, H, 0.0f, stream);
    const void* in[3] = {Q, K, V};
    void* out[3] = {Qp, Kp, Vp};
    const bss_status st = bss_permute_flagged_multi(in, out, 3, flags, H, &map->p, 0, stream);
    if (st != BSS_OK) return st;
    return bss_sparse_attention_split(Q, K, V, O, Qp, Kp, Vp, nullptr, lse, map, flags, H, 0.0f, stream);
}

}  // namespace

extern "C" {

bss_status bss_attention_step(const void* Q, const void* K, const void* V, void* O, float* lse, bss_tile_map map,
                              const uint8_t* head_is_temporal, int32_t H, void* Qp, void* Kp, void* Vp,
                              cudaStream_t stream) {
    using namespace bss;
    clear_error();
    if (!tile_map_is_live(map)) return set_error(BSS_ERR_INVALID_ARG, "invalid or destroyed tile map");
    if (map->p.temporal_permuted && head_is_temporal != nullptr && (Qp == nullptr || Kp == nullptr || Vp == nullptr))
        return set_error(BSS_ERR_INVALID_ARG, "the permuted layout needs the Qp, Kp, Vp workspaces");
    return step_device(Q, K, V, O, lse, map, head_is_temporal, H, Qp, Kp, Vp, stream);
}

bss_status bss_step_workspace_create(const bss_mask_params* params, int32_t H, int32_t depth,
                                     int32_t heads_per_group, bss_step_workspace* out) {
    using namespace bss;
    clear_error();
    if (out == nullptr) return set_error(BSS_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    bss_status st = check_mask_params(params);
    if (st != BSS_OK) return st;
    if (H <= 0) return set_error(BSS_ERR_INVALID_ARG, "H must be positive");
    if (depth < 1 || depth > kMaxDepth) return set_error(BSS_ERR_INVALID_ARG, "depth must lie in [1, %d]", kMaxDepth);
    if (heads_per_group < 1 || heads_per_group > H)
        return set_error(BSS_ERR_INVALID_ARG, "heads_per_group must lie in [1, H]");
    bss_step_workspace w = new (std::nothrow) bss_step_workspace_s();
    if (w == nullptr) return set_error(BSS_ERR_OOM, "host allocation failed");
    w->magic = kWsMagic;
    w->H = H;
    w->F = params->F;
    w->S = params->Hs * params->Ws;
    w->N = w->F * w->S;
    w->d = params->head_dim;
    w->depth = depth;
    w->group = heads_per_group;
    w->ngroups = (H + heads_per_group - 1) / heads_per_group;
    w->next = 0;
    cudaGetDevice(&w->device);
    const size_t bytes = static_cast<size_t>(H) * w->N * w->d * 2;
    auto fail = [&](bss_status s) {
        free_workspace(w);
        return s;
    };
    if (cudaStreamCreateWithFlags(&w->copy_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&w->copy_out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&w->compute2, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&w->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&w->join, cudaEventDisableTiming) != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(set_error(BSS_ERR_CUDA, "stream or event creation failed"));
    }
    w->sets.resize(depth);
    for (StepSet& s : w->sets) {
        for (void** p : {&s.Q, &s.K, &s.V, &s.O, &s.Qp, &s.Kp, &s.Vp}) {
            if (cudaMalloc(p, bytes) != cudaSuccess) {
                (void)cudaGetLastError();
                *p = nullptr;
                return fail(set_error(BSS_ERR_OOM, "step workspace allocation of %zu bytes failed", bytes));
            }
        }
        if (cudaMalloc(&s.flags, static_cast<size_t>(H)) != cudaSuccess) {
            (void)cudaGetLastError();
            s.flags = nullptr;
            return fail(set_error(BSS_ERR_OOM, "step workspace allocation failed"));
        }
        s.ready.assign(w->ngroups, nullptr);
        s.done.assign(w->ngroups, nullptr);
        bool ok = cudaEventCreateWithFlags(&s.free_ev, cudaEventDisableTiming) == cudaSuccess;
        for (int g = 0; ok && g < w->ngroups; ++g)
            ok = cudaEventCreateWithFlags(&s.ready[g], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&s.done[g], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            (void)cudaGetLastError();
            return fail(set_error(BSS_ERR_CUDA, "event creation failed"));
        }
    }
    {
        std::lock_guard<std::mutex> lk(g_ws_mutex);
        g_live_ws.insert(w);
    }
    *out = w;
    return BSS_OK;
}

void bss_step_workspace_destroy(bss_step_workspace ws) {
    if (ws == nullptr) return;
    {
        std::lock_guard<std::mutex> lk(g_ws_mutex);
        if (g_live_ws.erase(ws) == 0) return;
    }
    free_workspace(ws);
}

bss_status bss_step_workspace_wait_stream(bss_step_workspace ws, cudaStream_t stream) {
    using namespace bss;
    clear_error();
    if (!ws_is_live(ws)) return set_error(BSS_ERR_INVALID_ARG, "invalid or destroyed step workspace");
    cudaEvent_t e = nullptr;
    bss_status st = cuda_check(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "event");
    if (st != BSS_OK) return st;
    st = cuda_check(cudaEventRecord(e, stream), "event record");
    if (st == BSS_OK) st = cuda_check(cudaStreamWaitEvent(ws->copy_in, e, 0), "copy-in wait");
    if (st == BSS_OK) st = cuda_check(cudaStreamWaitEvent(ws->copy_out, e, 0), "copy-out wait");
    cudaEventDestroy(e);  // released once the waits it orders have been resolved
    return st;
}

bss_status bss_attention_step_host(const void* hQ, const void* hK, const void* hV, void* hO,
                                   const uint8_t* h_head_is_temporal, bss_tile_map map, bss_step_workspace ws,
                                   cudaEvent_t done, cudaStream_t stream) {
    using namespace bss;
    clear_error();
    if (!ws_is_live(ws)) return set_error(BSS_ERR_INVALID_ARG, "invalid or destroyed step workspace");
    if (!tile_map_is_live(map)) return set_error(BSS_ERR_INVALID_ARG, "invalid or destroyed tile map");
    if (hQ == nullptr || hK == nullptr || hV == nullptr || hO == nullptr || h_head_is_temporal == nullptr)
        return set_error(BSS_ERR_INVALID_ARG, "NULL host buffer");
    if (map->g.N != ws->N || map->p.head_dim != ws->d || map->g.F != ws->F)
        return set_error(BSS_ERR_INVALID_ARG, "the tile map's geometry differs from the workspace's");
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev != ws->device || dev != map->device)
        return set_error(BSS_ERR_INVALID_ARG, "workspace or tile map belongs to another device");
    StepSet& s = ws->sets[ws->next];
    const size_t row_bytes = static_cast<size_t>(ws->N) * ws->d * 2;  // one head of one tensor
    bss_status st;
    // A failure after the first enqueue leaves earlier groups' copies and
    // kernels in flight on this set: order them before the caller's later work
    // and before the set's next use, as a successful call would (the message of
    // the failure is kept: these calls do not set the error text).
    auto settle = [&](bss_status failed) {
        if (ws->ngroups > 1 && cudaEventRecord(ws->join, ws->compute2) == cudaSuccess)
            cudaStreamWaitEvent(stream, ws->join, 0);
        if (cudaEventRecord(ws->fork, stream) == cudaSuccess) cudaStreamWaitEvent(ws->copy_out, ws->fork, 0);
        if (cudaEventRecord(s.free_ev, ws->copy_out) == cudaSuccess) s.used = true;
        ws->next = (ws->next + 1) % ws->depth;
        return failed;
    };
#define BSS_TRY(call, what)                                              \
    do {                                                                 \
        if ((st = cuda_check((call), what)) != BSS_OK) return settle(st); \
    } while (0)
    // the set's previous call must be done with it: its kernels read Q, K, V and
    // its D2H copy reads O
    if (s.used && (st = cuda_check(cudaStreamWaitEvent(ws->copy_in, s.free_ev, 0), "wait for the buffer set")) !=
                      BSS_OK)
        return st;
    // the second compute stream starts after the caller's work so far
    if (ws->ngroups > 1) {
        BSS_TRY(cudaEventRecord(ws->fork, stream), "record fork");
        BSS_TRY(cudaStreamWaitEvent(ws->compute2, ws->fork, 0), "fork the second compute stream");
    }
    BSS_TRY(cudaMemcpyAsync(s.flags, h_head_is_temporal, static_cast<size_t>(ws->H), cudaMemcpyHostToDevice,
                            ws->copy_in),
            "copy flags");
    for (int g = 0; g < ws->ngroups; ++g) {
        const int h0 = g * ws->group;
        const int h1 = h0 + ws->group < ws->H ? h0 + ws->group : ws->H;
        const size_t off = static_cast<size_t>(h0) * row_bytes;
        const size_t n = static_cast<size_t>(h1 - h0) * row_bytes;
        auto at = [off](const void* base) { return static_cast<const uint8_t*>(base) + off; };
        auto at_mut = [off](void* base) { return static_cast<uint8_t*>(base) + off; };
        BSS_TRY(cudaMemcpyAsync(at_mut(s.Q), at(hQ), n, cudaMemcpyHostToDevice, ws->copy_in), "copy Q in");
        BSS_TRY(cudaMemcpyAsync(at_mut(s.K), at(hK), n, cudaMemcpyHostToDevice, ws->copy_in), "copy K in");
        BSS_TRY(cudaMemcpyAsync(at_mut(s.V), at(hV), n, cudaMemcpyHostToDevice, ws->copy_in), "copy V in");
        BSS_TRY(cudaEventRecord(s.ready[g], ws->copy_in), "record inputs ready");
        cudaStream_t cs = (g & 1) ? ws->compute2 : stream;
        BSS_TRY(cudaStreamWaitEvent(cs, s.ready[g], 0), "wait for inputs");
        if ((st = step_device(at(s.Q), at(s.K), at(s.V), at_mut(s.O), nullptr, map, s.flags + h0, h1 - h0,
                              at_mut(s.Qp), at_mut(s.Kp), at_mut(s.Vp), cs)) != BSS_OK)
            return settle(st);
        BSS_TRY(cudaEventRecord(s.done[g], cs), "record outputs done");
        BSS_TRY(cudaStreamWaitEvent(ws->copy_out, s.done[g], 0), "wait for outputs");
        BSS_TRY(cudaMemcpyAsync(at_mut(hO), at(s.O), n, cudaMemcpyDeviceToHost, ws->copy_out), "copy O out");
    }
    // the caller's stream is ordered after every group's kernels
    if (ws->ngroups > 1) {
        BSS_TRY(cudaEventRecord(ws->join, ws->compute2), "record join");
        BSS_TRY(cudaStreamWaitEvent(stream, ws->join, 0), "join the second compute stream");
    }
    BSS_TRY(cudaEventRecord(s.free_ev, ws->copy_out), "record set free");
    if (done != nullptr) BSS_TRY(cudaEventRecord(done, ws->copy_out), "record done");
#undef BSS_TRY
    s.used = true;
    ws->next = (ws->next + 1) % ws->depth;
    return BSS_OK;
}

}  // extern "C"
