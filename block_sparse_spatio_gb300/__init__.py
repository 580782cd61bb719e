"""Python binding of the block-sparse spatio-temporal attention library.

Argument marshalling only: every step runs in the CUDA library ``libbss.so``
(C ABI in ``include/bss.h``).  PyTorch supplies device memory and the current
stream.  There is no CPU or PyTorch fallback: if the library is missing or was
not built for this GPU, every call raises.

Method: blog "Accelerating Spatio-Temporal Attention for Video Diffusion on
TPUs" (Google Developers) -- per-head spatial / temporal block-sparse
attention with full / boundary / skipped tiles, optional tile-aligned rounding,
and the (F,H,W) <-> (H,W,F) token permutation for temporal heads.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbss.so")

KIND_SPATIAL, KIND_TEMPORAL = 0, 1
CLASS_FULL, CLASS_BOUNDARY, CLASS_PAD, CLASS_COLUMNS = 0, 1, 2, 3
ATTN_BQ, ATTN_BKV = 256, 128   # default tile shape of bss_sparse_attention's map
ATTN_BQ_SUPPORTED = (128, 256)  # query rows per tile it runs (one or two 128-row MMA halves)
ATTN_BKV_SUPPORTED = (64, 128)  # keys per tile it runs (routing, dense control and fused permutation: 128)
CLASS_SHIFT = 30
TILE_INDEX_MASK = (1 << 30) - 1
STAT_NAMES = ("full", "boundary", "pad", "skip", "retained_pairs", "exact_retained_pairs", "columns")
STATUS_NAMES = {0: "BSS_OK", 1: "BSS_ERR_INVALID_ARG", 2: "BSS_ERR_UNSUPPORTED", 3: "BSS_ERR_CUDA",
                4: "BSS_ERR_TIMEOUT", 5: "BSS_ERR_OOM"}

_lib = None


class BssError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _MaskParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("F", "Hs", "Ws", "head_dim", "spatial_frame_window",
                                               "temporal_raster_window", "sink_frames", "temporal_permuted",
                                               "rounding")]


@dataclass(frozen=True)
class MaskParams:
    """Video geometry and mask windows (see ``bss_mask_params`` in include/bss.h)."""
    F: int
    Hs: int
    Ws: int
    head_dim: int
    spatial_frame_window: int
    temporal_raster_window: int
    sink_frames: int = 1
    temporal_permuted: int = 1
    rounding: int = 0

    @property
    def S(self) -> int:
        return self.Hs * self.Ws

    @property
    def N(self) -> int:
        return self.F * self.S

    def c(self) -> _MaskParams:
        return _MaskParams(self.F, self.Hs, self.Ws, self.head_dim, self.spatial_frame_window,
                           self.temporal_raster_window, self.sink_frames, self.temporal_permuted, self.rounding)


EXPORTED = ("bss_build_tile_map", "bss_tile_map_stats", "bss_tile_map_dims", "bss_tile_map_copy_csr",
            "bss_destroy_tile_map", "bss_permute", "bss_sparse_attention", "bss_dense_attention",
            "bss_get_device_status", "bss_status_string", "bss_last_error_message", "bss_version",
            "bss_diag_mma_tile", "bss_build_tile_map_csr_noalloc", "bss_route_heads",
            "bss_sparse_attention_fused", "bss_permute_flagged", "bss_sparse_attention_split",
            "bss_diag_wait_timeout", "bss_attention_step", "bss_step_workspace_create",
            "bss_step_workspace_destroy", "bss_step_workspace_wait_stream", "bss_attention_step_host",
            "bss_permute_flagged_multi")


def load(path: str | None = None):
    """Load libbss.so (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m block_sparse_spatio_gb300.build`")
    lib = ctypes.CDLL(path)
    p, i32, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int
    MP = ctypes.POINTER(_MaskParams)
    lib.bss_build_tile_map.argtypes = [MP, i32, i32, ctypes.POINTER(p), p]
    lib.bss_build_tile_map.restype = st
    lib.bss_tile_map_stats.argtypes = [p, i32, ctypes.POINTER(ctypes.c_int64)]
    lib.bss_tile_map_stats.restype = st
    lib.bss_tile_map_dims.argtypes = [p, i32, ctypes.POINTER(ctypes.c_int32)]
    lib.bss_tile_map_dims.restype = st
    lib.bss_tile_map_copy_csr.argtypes = [p, i32, p, p]
    lib.bss_tile_map_copy_csr.restype = st
    lib.bss_destroy_tile_map.argtypes = [p]
    lib.bss_destroy_tile_map.restype = None
    lib.bss_permute.argtypes = [p, p, p, i32, MP, i32, p]
    lib.bss_permute.restype = st
    lib.bss_sparse_attention.argtypes = [p, p, p, p, p, p, p, i32, ctypes.c_float, p]
    lib.bss_sparse_attention.restype = st
    lib.bss_sparse_attention_fused.argtypes = [p, p, p, p, p, p, p, i32, ctypes.c_float, p]
    lib.bss_sparse_attention_fused.restype = st
    lib.bss_sparse_attention_split.argtypes = [p, p, p, p, p, p, p, p, p, p, p, i32, ctypes.c_float, p]
    lib.bss_sparse_attention_split.restype = st
    lib.bss_permute_flagged.argtypes = [p, p, p, i32, MP, i32, p]
    lib.bss_permute_flagged.restype = st
    lib.bss_diag_wait_timeout.argtypes = [ctypes.c_int64, p, p]
    lib.bss_diag_wait_timeout.restype = st
    lib.bss_dense_attention.argtypes = [p, p, p, p, p, i32, i32, i32, ctypes.c_float, p]
    lib.bss_dense_attention.restype = st
    lib.bss_get_device_status.argtypes = [p]
    lib.bss_get_device_status.restype = st
    lib.bss_status_string.argtypes = [st]
    lib.bss_status_string.restype = ctypes.c_char_p
    lib.bss_last_error_message.argtypes = []
    lib.bss_last_error_message.restype = ctypes.c_char_p
    lib.bss_version.argtypes = []
    lib.bss_version.restype = i32
    lib.bss_diag_mma_tile.argtypes = [p, p, p, p, p, p, i32, p]
    lib.bss_diag_mma_tile.restype = st
    lib.bss_build_tile_map_csr_noalloc.argtypes = [MP, i32, i32, i32, p, p, ctypes.c_int64, p, p]
    lib.bss_build_tile_map_csr_noalloc.restype = st
    lib.bss_route_heads.argtypes = [p, p, p, i32, MP, p, i32, p, p, p]
    lib.bss_route_heads.restype = st
    lib.bss_permute_flagged_multi.argtypes = [ctypes.POINTER(p), ctypes.POINTER(p), i32, p, i32, MP, i32, p]
    lib.bss_permute_flagged_multi.restype = st
    lib.bss_attention_step.argtypes = [p, p, p, p, p, p, p, i32, p, p, p, p]
    lib.bss_attention_step.restype = st
    lib.bss_step_workspace_create.argtypes = [MP, i32, i32, i32, ctypes.POINTER(p)]
    lib.bss_step_workspace_create.restype = st
    lib.bss_step_workspace_destroy.argtypes = [p]
    lib.bss_step_workspace_destroy.restype = None
    lib.bss_step_workspace_wait_stream.argtypes = [p, p]
    lib.bss_step_workspace_wait_stream.restype = st
    lib.bss_attention_step_host.argtypes = [p, p, p, p, p, p, p, p, p]
    lib.bss_attention_step_host.restype = st
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise BssError(status, load().bss_last_error_message().decode())


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev_tensor(t, name, dtype=None):
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _check_shapes(tile_map, lse, *named):
    """Every tensor [H][N][d] of the map's geometry (same H), lse [H][N]: a
    map built for another geometry is refused before any launch."""
    p = tile_map.params
    N, d = p.F * p.Hs * p.Ws, p.head_dim
    H = named[0][0].shape[0]
    for t, n in named:
        if tuple(t.shape) != (H, N, d):
            raise ValueError(f"{n} has shape {tuple(t.shape)}, the tile map wants ({H}, {N}, {d})")
    if lse is not None and tuple(lse.shape) != (H, N):
        raise ValueError(f"lse has shape {tuple(lse.shape)}, the tile map wants ({H}, {N})")
    return H


class TileMap:
    """Owning wrapper of a ``bss_tile_map`` handle."""

    def __init__(self, handle: ctypes.c_void_p, params: MaskParams, BQ: int, BKV: int):
        self._h = handle
        self.params, self.BQ, self.BKV = params, BQ, BKV

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("tile map destroyed")
        return self._h

    def stats(self, kind: int) -> dict:
        return tile_map_stats(self, kind)

    def dims(self, kind: int):
        return tile_map_dims(self, kind)

    def csr(self, kind: int):
        return tile_map_copy_csr(self, kind)

    def destroy(self):
        if self._h is not None and _lib is not None:
            _lib.bss_destroy_tile_map(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()


def build_tile_map(params: MaskParams, BQ: int = ATTN_BQ, BKV: int = ATTN_BKV, stream=None) -> TileMap:
    lib = load()
    h = ctypes.c_void_p()
    mp = params.c()
    _check(lib.bss_build_tile_map(ctypes.byref(mp), BQ, BKV, ctypes.byref(h), _stream(stream)))
    return TileMap(h, params, BQ, BKV)


def _raw_handle(m):
    return m.handle if isinstance(m, TileMap) else m


def tile_map_stats(m, kind: int) -> dict:
    out = (ctypes.c_int64 * len(STAT_NAMES))()
    _check(load().bss_tile_map_stats(_raw_handle(m), kind, out))
    return dict(zip(STAT_NAMES, [int(x) for x in out]))


def tile_map_dims(m, kind: int):
    out = (ctypes.c_int32 * 4)()
    _check(load().bss_tile_map_dims(_raw_handle(m), kind, out))
    return tuple(int(x) for x in out)  # nq, nkv, nnz, ncols


def tile_map_copy_csr(m, kind: int):
    nq, nkv, nnz, ncols = tile_map_dims(m, kind)
    row_ptr = np.zeros(nq + 1, dtype=np.int32)
    entries = np.zeros(max(nnz, 1), dtype=np.int32)
    _check(load().bss_tile_map_copy_csr(_raw_handle(m), kind, row_ptr.ctypes.data, entries.ctypes.data))
    return row_ptr, entries[:nnz]


def destroy_tile_map(m):
    if isinstance(m, TileMap):
        m.destroy()
    else:
        load().bss_destroy_tile_map(m)


def permute(x, out, head_is_temporal, params: MaskParams, inverse: bool = False, stream=None,
            only_flagged: bool = False):
    """out <- per-head (F,H,W) -> (H,W,F) permutation of x (inverse=True: back).
    Heads with flag 0 are copied, or left untouched with ``only_flagged``."""
    import torch
    _dev_tensor(x, "x", torch.bfloat16)
    _dev_tensor(out, "out", torch.bfloat16)
    _dev_tensor(head_is_temporal, "head_is_temporal", torch.uint8)
    fn = load().bss_permute_flagged if only_flagged else load().bss_permute
    _check(fn(_ptr(x), _ptr(out), _ptr(head_is_temporal), x.shape[0], ctypes.byref(params.c()), int(bool(inverse)),
              _stream(stream)))
    return out


def permute_flagged_multi(xs, outs, head_is_temporal, params: MaskParams, inverse: bool = False, stream=None):
    """outs[i] <- the flagged heads of xs[i] permuted, 1 to 3 tensors in one launch
    (heads with flag 0 are left untouched in outs)."""
    import torch
    if len(xs) != len(outs) or not 1 <= len(xs) <= 3:
        raise ValueError("1 to 3 (input, output) pairs")
    for i, (x, o) in enumerate(zip(xs, outs)):
        _dev_tensor(x, f"xs[{i}]", torch.bfloat16)
        _dev_tensor(o, f"outs[{i}]", torch.bfloat16)
        if x.shape != xs[0].shape or o.shape != xs[0].shape:
            raise ValueError("every tensor must have the same shape")
    _dev_tensor(head_is_temporal, "head_is_temporal", torch.uint8)
    n = len(xs)
    ins = (ctypes.c_void_p * n)(*[x.data_ptr() for x in xs])
    ous = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    _check(load().bss_permute_flagged_multi(ins, ous, n, _ptr(head_is_temporal), xs[0].shape[0],
                                            ctypes.byref(params.c()), int(bool(inverse)), _stream(stream)))
    return outs


def sparse_attention(Q, K, V, O, tile_map: TileMap, head_is_temporal=None, lse=None, softmax_scale: float = 0.0,
                     stream=None):
    """O <- block-sparse attention of [H][N][d] bf16 Q, K, V (temporal heads pre-permuted)."""
    import torch
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (O, "O")):
        _dev_tensor(t, n, torch.bfloat16)
    _dev_tensor(head_is_temporal, "head_is_temporal", torch.uint8)
    _dev_tensor(lse, "lse", torch.float32)
    _check_shapes(tile_map, lse, (Q, "Q"), (K, "K"), (V, "V"), (O, "O"))
    _check(load().bss_sparse_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), tile_map.handle,
                                       _ptr(head_is_temporal), Q.shape[0], float(softmax_scale), _stream(stream)))
    return O


def sparse_attention_split(Q, K, V, O, Qt, Kt, Vt, Ot, tile_map: TileMap, head_is_temporal, lse=None,
                           softmax_scale: float = 0.0, stream=None):
    """Block-sparse attention with spatial heads in Q, K, V -> O and temporal
    heads (flag 1) in the permuted buffers Qt, Kt, Vt -> Ot.  Ot=None writes the
    temporal heads' output rows straight to O in (F,H,W) order (no inverse
    permutation needed)."""
    import torch
    named = [(Q, "Q"), (K, "K"), (V, "V"), (O, "O"), (Qt, "Qt"), (Kt, "Kt"), (Vt, "Vt")]
    if Ot is not None:
        named.append((Ot, "Ot"))
    for t, n in named:
        _dev_tensor(t, n, torch.bfloat16)
    _dev_tensor(head_is_temporal, "head_is_temporal", torch.uint8)
    _dev_tensor(lse, "lse", torch.float32)
    _check_shapes(tile_map, lse, *named)
    _check(load().bss_sparse_attention_split(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(Qt), _ptr(Kt), _ptr(Vt),
                                             _ptr(Ot), _ptr(lse), tile_map.handle, _ptr(head_is_temporal),
                                             Q.shape[0], float(softmax_scale), _stream(stream)))
    return O


def sparse_attention_fused(Q, K, V, O, tile_map: TileMap, head_is_temporal=None, lse=None,
                           softmax_scale: float = 0.0, stream=None):
    """O <- block-sparse attention of [H][N][d] bf16 Q, K, V, all heads in (F,H,W)
    order: the temporal heads' permutation is applied inside the kernel."""
    import torch
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (O, "O")):
        _dev_tensor(t, n, torch.bfloat16)
    _dev_tensor(head_is_temporal, "head_is_temporal", torch.uint8)
    _dev_tensor(lse, "lse", torch.float32)
    _check_shapes(tile_map, lse, (Q, "Q"), (K, "K"), (V, "V"), (O, "O"))
    _check(load().bss_sparse_attention_fused(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), tile_map.handle,
                                             _ptr(head_is_temporal), Q.shape[0], float(softmax_scale),
                                             _stream(stream)))
    return O


def dense_attention(Q, K, V, O, lse=None, softmax_scale: float = 0.0, stream=None):
    """O <- dense attention of [H][N][d] bf16 Q, K, V (the control)."""
    import torch
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (O, "O")):
        _dev_tensor(t, n, torch.bfloat16)
    _dev_tensor(lse, "lse", torch.float32)
    H, N, d = Q.shape
    _check(load().bss_dense_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), H, N, d, float(softmax_scale),
                                      _stream(stream)))
    return O


def get_device_status(stream=None) -> int:
    """Synchronize and return (and clear) the device status word; 0 = OK."""
    return int(load().bss_get_device_status(_stream(stream)))


def status_string(status: int) -> str:
    return load().bss_status_string(status).decode()


def diag_wait_timeout(limit_ns: int, waited_ns=None, stream=None):
    """Run a bounded wait that nothing completes (see include/bss_diag.h); the
    device status word then holds BSS_ERR_TIMEOUT."""
    import torch
    _dev_tensor(waited_ns, "waited_ns", torch.int64)
    _check(load().bss_diag_wait_timeout(int(limit_ns), _ptr(waited_ns), _stream(stream)))


def diag_mma_tile(A, B, P, V, S, O, stream=None):
    """One-tile tensor-core self-test: S = A B^T, O = P V (see include/bss_diag.h)."""
    _check(load().bss_diag_mma_tile(_ptr(A), _ptr(B), _ptr(P), _ptr(V), _ptr(S), _ptr(O), A.shape[1],
                                    _stream(stream)))
    return S, O


def noalloc_map_dims(params: MaskParams, kind: int, BQ: int = ATTN_BQ, BKV: int = ATTN_BKV):
    """(nq, nkv) of the map bss_build_tile_map_csr_noalloc writes for one kind."""
    N, S = params.N, params.S
    ncols = (-(-S // BKV) * BKV + N) if (kind == KIND_TEMPORAL and params.temporal_permuted) else N
    return -(-N // BQ), -(-ncols // BKV)


def build_tile_map_csr_noalloc(params: MaskParams, kind: int, row_ptr, entries, stats, BQ: int = ATTN_BQ,
                               BKV: int = ATTN_BKV, stream=None):
    """Allocation-free CSR build of one kind into caller-owned device buffers
    (int32 row_ptr[nq + 1], int32 entries[>= nq * nkv], int64 stats[len(STAT_NAMES)])."""
    import torch
    _dev_tensor(row_ptr, "row_ptr", torch.int32)
    _dev_tensor(entries, "entries", torch.int32)
    _dev_tensor(stats, "stats", torch.int64)
    _check(load().bss_build_tile_map_csr_noalloc(ctypes.byref(params.c()), kind, BQ, BKV, _ptr(row_ptr),
                                                  _ptr(entries), entries.numel(), _ptr(stats), _stream(stream)))
    return row_ptr, entries, stats


def route_heads(Q, K, V, params: MaskParams, rows, head_is_temporal, errors, stream=None):
    """Per-head routing from sampled query rows (int32 device tensor of (F,H,W)
    token indices): writes head_is_temporal (uint8[H]) and errors (float32[H][2]:
    spatial and temporal deviation from the dense output)."""
    import torch
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _dev_tensor(t, n, torch.bfloat16)
    _dev_tensor(rows, "rows", torch.int32)
    _dev_tensor(head_is_temporal, "head_is_temporal", torch.uint8)
    _dev_tensor(errors, "errors", torch.float32)
    _check(load().bss_route_heads(_ptr(Q), _ptr(K), _ptr(V), Q.shape[0], ctypes.byref(params.c()), _ptr(rows),
                                  rows.numel(), _ptr(head_is_temporal), _ptr(errors), _stream(stream)))
    return head_is_temporal, errors


def attention_step(Q, K, V, O, tile_map: TileMap, head_is_temporal, Qp, Kp, Vp, lse=None, stream=None):
    """The per-layer path of the blog's Figure 8 on one GPU (``bss_attention_step``):
    permute the temporal heads' Q, K, V to (H,W,F) into the workspaces Qp, Kp,
    Vp, run block-sparse attention, and store their O rows back in (F,H,W)
    order.  Q, K, V, O are in (F,H,W) order; Qp, Kp, Vp may be None when no
    head is permuted (no flags, or a map with temporal_permuted = 0).  lse, if
    given, is in each head's own layout."""
    import torch
    named = [(Q, "Q"), (K, "K"), (V, "V"), (O, "O")] + [(t, n) for t, n in ((Qp, "Qp"), (Kp, "Kp"), (Vp, "Vp"))
                                                          if t is not None]
    for t, n in named:
        _dev_tensor(t, n, torch.bfloat16)
    _dev_tensor(head_is_temporal, "head_is_temporal", torch.uint8)
    _dev_tensor(lse, "lse", torch.float32)
    _check_shapes(tile_map, lse, *named)
    _check(load().bss_attention_step(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), tile_map.handle,
                                     _ptr(head_is_temporal), Q.shape[0], _ptr(Qp), _ptr(Kp), _ptr(Vp),
                                     _stream(stream)))
    return O


class StepWorkspace:
    """Owning wrapper of a ``bss_step_workspace`` (device buffer sets, copy
    streams and events of ``attention_step_host``)."""

    def __init__(self, handle, params: MaskParams, H: int, depth: int, heads_per_group: int):
        self._h = handle
        self.params, self.H, self.depth, self.heads_per_group = params, H, depth, heads_per_group

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("step workspace destroyed")
        return self._h

    def wait_stream(self, stream=None):
        """Order the workspace's copy streams after the work enqueued on ``stream``."""
        _check(load().bss_step_workspace_wait_stream(self.handle, _stream(stream)))

    def destroy(self):
        if self._h is not None and _lib is not None:
            _lib.bss_step_workspace_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()


def step_workspace(params: MaskParams, H: int, depth: int = 3, heads_per_group: int = 2) -> StepWorkspace:
    """Workspace of ``attention_step_host`` (``bss_step_workspace_create``).

    depth buffer sets used in turn: with three (the default) the host-to-device
    copy of a call can start while the device-to-host copy of the call two back
    is still running; measured with two, steps were 2.4% slower (6.00 vs 5.86
    ms on the mixed 75.6K workload, against 5.78 ms for the kernels alone).
    heads_per_group heads are copied in and computed together: two (the
    default) cost nothing when the host link keeps up and shorten the step when
    it does not (6.07 ms per step against 7.22 ms for one group of all ten
    heads on a box whose host-to-device copies slowed down now and then);
    single-head groups were slower (7.2-7.4 ms: ten small attention launches,
    each with its own tail)."""
    h = ctypes.c_void_p()
    mp = params.c()
    _check(load().bss_step_workspace_create(ctypes.byref(mp), H, depth, heads_per_group, ctypes.byref(h)))
    return StepWorkspace(h, params, H, depth, heads_per_group)


def _host_tensor(t, name, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def attention_step_host(hQ, hK, hV, hO, tile_map: TileMap, head_is_temporal, workspace: StepWorkspace, stream=None):
    """The per-layer path from HOST buffers (``bss_attention_step_host``): H2D
    copies of Q, K, V, the ``attention_step`` kernels and the D2H copy of O,
    pipelined over groups of heads on the workspace's copy streams and
    ``stream`` (default: current).  hQ, hK, hV, hO: CPU bf16 [H][N][d], pinned
    for overlap; head_is_temporal: CPU uint8[H].  Returns a CUDA event that
    completes when hO is written; until then the host buffers must stay alive
    (the copies read and write them asynchronously) and the inputs unchanged."""
    import torch
    for t, n in ((hQ, "hQ"), (hK, "hK"), (hV, "hV"), (hO, "hO")):
        _host_tensor(t, n, torch.bfloat16)
    _host_tensor(head_is_temporal, "head_is_temporal", torch.uint8)
    p = tile_map.params
    shape = (workspace.H, p.N, p.head_dim)
    for t, n in ((hQ, "hQ"), (hK, "hK"), (hV, "hV"), (hO, "hO")):
        if tuple(t.shape) != shape:
            raise ValueError(f"{n} has shape {tuple(t.shape)}, the workspace and map want {shape}")
    if tuple(head_is_temporal.shape) != (workspace.H,):
        raise ValueError(f"head_is_temporal must have {workspace.H} entries")
    done = torch.cuda.Event()
    done.record()  # creates the event; the library records it again after the D2H copy
    _check(load().bss_attention_step_host(_ptr(hQ), _ptr(hK), _ptr(hV), _ptr(hO), _ptr(head_is_temporal),
                                          tile_map.handle, workspace.handle, ctypes.c_void_p(done.cuda_event),
                                          _stream(stream)))
    return done
