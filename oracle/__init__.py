"""fp64 CPU oracle for block-sparse spatio-temporal attention.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product package
(``block_sparse_spatio_gb300``) never does, and the two share no code.

Source: "Accelerating Spatio-Temporal Attention for Video Diffusion on TPUs"
(Google Developers blog).  The arithmetic lives in ``bss_oracle.c`` (plain C,
fp64, one query/key pair at a time); this module only marshals numpy arrays.

Mask kinds (oracle codes):
  SPATIAL = 0            frame band + first-frame sink, (F,H,W) layout
  TEMPORAL_PERMUTED = 1  raster band across frames + sink, (H,W,F) layout,
                         keys in a virtual space: a sink segment of S_pad
                         columns (S rounded up to BKV) in front of the N
                         permuted rows
  TEMPORAL_FHW = 2       same retained set evaluated in (F,H,W) order
  DENSE = 3              every pair retained

Parity status: every function here is pinned by ``tests/test_oracle.py``
(brute-force dense masked softmax over explicit N x N matrices, closed-form
counts, the hand-derived Tiny tile map, the permutation round trip and hand
values, Q = 0 coverage, poison invariance; the tile-aligned mask against the
set of physical pairs its kept tiles cover, built from token multiplicities;
routing against constructed heads whose closer mask is known and against
all-covering windows, where both deviations vanish).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

SPATIAL, TEMPORAL_PERMUTED, TEMPORAL_FHW, DENSE = 0, 1, 2, 3
FULL, BOUNDARY, PAD, COLUMNS, SKIP = 0, 1, 2, 3, 4
CLASS_SHIFT = 30

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bss_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", _LIB_PATH, "-lm"]
        subprocess.check_call(cmd)
    return _LIB_PATH


class _Geom(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("F", "S", "N", "wf", "ws", "sink_frames", "S_pad")]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.orc_perm_index.restype = i64
        lib.orc_perm_index.argtypes = [i64, i64, i64]
        lib.orc_unperm_index.restype = i64
        lib.orc_unperm_index.argtypes = [i64, i64, i64]
        lib.orc_permute.restype = None
        lib.orc_permute.argtypes = [p, p, i64, i64, i64, i64, p, ctypes.c_int]
        lib.orc_retained.restype = ctypes.c_int
        lib.orc_retained.argtypes = [ctypes.c_int, ctypes.POINTER(_Geom), i64, i64]
        lib.orc_num_cols.restype = i64
        lib.orc_num_cols.argtypes = [ctypes.c_int, ctypes.POINTER(_Geom)]
        lib.orc_classify.restype = None
        lib.orc_classify.argtypes = [ctypes.c_int, ctypes.POINTER(_Geom), i64, i64, ctypes.c_int,
                                     i64, i64, p, p]
        lib.orc_attention.restype = None
        lib.orc_attention.argtypes = [p, p, p, i64, ctypes.c_int, ctypes.POINTER(_Geom), ctypes.c_double,
                                      p, i64, i64, p, i64, p, p]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_set_num_threads.restype = None
        lib.orc_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on."""
    _load().orc_set_num_threads(int(n))


class Geometry:
    """Video token geometry plus mask windows.

    F frames of Hs x Ws latent patches; S = Hs*Ws; N = F*S.  ``wf`` is the
    spatial frame window, ``ws`` the temporal raster window, ``bkv`` fixes the
    sink-segment padding of the temporal virtual key space."""

    def __init__(self, F, Hs, Ws, wf=0, ws=0, sink_frames=1, bkv=128):
        self.F, self.Hs, self.Ws = int(F), int(Hs), int(Ws)
        self.S = self.Hs * self.Ws
        self.N = self.F * self.S
        self.wf, self.ws, self.sink_frames = int(wf), int(ws), int(sink_frames)
        self.bkv = int(bkv)
        self.S_pad = -(-self.S // self.bkv) * self.bkv

    def c(self) -> _Geom:
        return _Geom(self.F, self.S, self.N, self.wf, self.ws, self.sink_frames, self.S_pad)

    def with_bkv(self, bkv):
        return Geometry(self.F, self.Hs, self.Ws, self.wf, self.ws, self.sink_frames, bkv)


def perm_index(t, F, S):
    return int(_load().orc_perm_index(int(t), int(F), int(S)))


def unperm_index(p, F, S):
    return int(_load().orc_unperm_index(int(p), int(F), int(S)))


def permute(x: np.ndarray, F: int, S: int, flags, inverse: bool = False) -> np.ndarray:
    """Per-head (F,H,W) <-> (H,W,F) permutation of a [H][N][d] uint16 (bf16 bits) array."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    H, N, d = x.shape
    assert N == F * S
    fl = np.ascontiguousarray(np.asarray(flags, dtype=np.uint8).reshape(H))
    out = np.empty_like(x)
    _load().orc_permute(x.ctypes.data, out.ctypes.data, H, F, S, d, fl.ctypes.data, int(bool(inverse)))
    return out


def retained(kind: int, g: Geometry, q: int, k: int) -> int:
    gc = g.c()
    return int(_load().orc_retained(kind, ctypes.byref(gc), int(q), int(k)))


def num_cols(kind: int, g: Geometry) -> int:
    gc = g.c()
    return int(_load().orc_num_cols(kind, ctypes.byref(gc)))


def classify(kind: int, g: Geometry, BQ: int, BKV: int, rounding, qt0: int = 0, qt1: int | None = None):
    """Per-tile retained real-pair counts and classes for q-tile rows [qt0, qt1).
    rounding: 0 exact, 1 tile-aligned, 2 exact mask in every visited tile.
    Rounded permuted-temporal rows mark a kept sink tile COLUMNS (or SKIP) when
    some (or all) of its frame-0 keys also sit in a kept band tile of the row."""
    g = g.with_bkv(BKV)
    nq = -(-g.N // BQ)
    if qt1 is None:
        qt1 = nq
    nkv = -(-num_cols(kind, g) // BKV)
    counts = np.zeros((qt1 - qt0, nkv), dtype=np.int64)
    cls = np.zeros((qt1 - qt0, nkv), dtype=np.int8)
    gc = g.c()
    _load().orc_classify(kind, ctypes.byref(gc), BQ, BKV, int(rounding), qt0, qt1,
                         counts.ctypes.data, cls.ctypes.data)
    return counts, cls


def tile_map(kind: int, g: Geometry, BQ: int, BKV: int, rounding: bool, qt0: int = 0, qt1: int | None = None):
    """CSR tile map (ascending kv index per q-tile, class in bits 30..31) plus statistics.

    Returns (row_ptr int32 [rows+1], entries int32, stats dict).  ``retained_pairs``
    is the exact retained count for the exact mask, and for the rounded mask the
    number of distinct physical (query, key) pairs the kept tiles cover: every
    real row of a q tile sees the same keys, those read by the real columns of
    its kept tiles, each physical key once."""
    gg = g.with_bkv(BKV)
    counts, cls = classify(kind, gg, BQ, BKV, rounding, qt0, qt1)
    rows, nkv = cls.shape
    row_ptr = np.zeros(rows + 1, dtype=np.int64)
    ents = []
    for i in range(rows):
        js = np.nonzero(cls[i] != SKIP)[0]
        ents.append((js.astype(np.int64) | (cls[i, js].astype(np.int64) << CLASS_SHIFT)))
        row_ptr[i + 1] = row_ptr[i] + js.size
    entries = np.concatenate(ents) if ents else np.zeros(0, np.int64)
    # real key columns, for the rounded retained-pair count
    ncols = num_cols(kind, gg)
    k = np.arange(nkv * BKV, dtype=np.int64)
    if kind == TEMPORAL_PERMUTED:
        col_real = ((k < gg.S_pad) & (k < gg.S)) | ((k >= gg.S_pad) & (k - gg.S_pad < gg.N))
    else:
        col_real = k < gg.N
    q0 = qt0 if qt0 else 0
    real_rows = np.array([min(BQ, max(0, gg.N - (q0 + i) * BQ)) for i in range(rows)], dtype=np.int64)
    kept = cls != SKIP
    if rounding == 1:
        keys = key_rows(kind, gg)
        retained_pairs = 0
        for i in range(rows):
            cols = np.repeat(kept[i], BKV)[: ncols] & col_real[: ncols]
            retained_pairs += int(real_rows[i]) * int(np.unique(keys[cols]).size)
    else:
        retained_pairs = int(counts.sum())
    stats = {
        "full": int((cls == FULL).sum()),
        "boundary": int((cls == BOUNDARY).sum()),
        "pad": int((cls == PAD).sum()),
        "skip": int((cls == SKIP).sum()),
        "retained_pairs": retained_pairs,
        "exact_retained_pairs": int(counts.sum()),
        "columns": int((cls == COLUMNS).sum()),
        "ncols": ncols,
    }
    return row_ptr.astype(np.int32), entries.astype(np.uint32).view(np.int32), stats


def key_rows(kind: int, g: Geometry) -> np.ndarray:
    """Physical row of the head's layout tensor that each key column reads: for
    the permuted temporal kind, sink column v is the frame-0 key at raster v
    (permuted row v*F) and band column S_pad + p is permuted row p; otherwise
    column k is row k.  Padding columns map to row 0 (never read)."""
    ncols = num_cols(kind, g)
    k = np.arange(ncols, dtype=np.int64)
    if kind != TEMPORAL_PERMUTED:
        return k
    return np.where(k < g.S_pad, np.where(k < g.S, k * g.F, 0), k - g.S_pad)


def _layout_kind(kind: int, g: Geometry):
    """(uses_permuted_layout) for an oracle mask kind."""
    return kind == TEMPORAL_PERMUTED


def attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, kind: int, g: Geometry, rows=None,
              rounding=0, BQ: int = 128, BKV: int = 128, scale: float | None = None):
    """fp64 masked attention of ONE head.

    Q, K, V: [N][d] uint16 (bf16 bits) in the ORIGINAL (F,H,W) token order.
    rows: original token indices to evaluate (default: all).
    Returns (O [len(rows)][d] float64, lse [len(rows)] float64), rows in the order given.
    For the temporal-permuted kind the head is permuted (H,W,F) first, attention
    runs over the virtual key space, and the rows are read back in (F,H,W) order.
    A rounded mask keeps, for every row of a q tile, the physical keys read by
    the real columns of the tile's kept tiles, each key once."""
    lib = _load()
    Q = np.ascontiguousarray(Q, dtype=np.uint16)
    K = np.ascontiguousarray(K, dtype=np.uint16)
    V = np.ascontiguousarray(V, dtype=np.uint16)
    N, d = Q.shape
    g = g.with_bkv(BKV)
    assert N == g.N
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if rows is None:
        rows = np.arange(N, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    if _layout_kind(kind, g):
        one = np.ones(1, np.uint8)
        Qp = permute(Q[None], g.F, g.S, one)[0]
        Kp = permute(K[None], g.F, g.S, one)[0]
        Vp = permute(V[None], g.F, g.S, one)[0]
        lrows = np.array([perm_index(t, g.F, g.S) for t in rows], dtype=np.int64)
    else:
        Qp, Kp, Vp, lrows = Q, K, V, rows
    kept_ptr = None
    kept = None
    if rounding == 1:  # only the tile-aligned mask changes the retained set
        nq = -(-N // BQ)
        nkv = -(-num_cols(kind, g) // BKV)
        kept = np.zeros((nq, nkv), dtype=np.int8)
        for qt in sorted(set((lrows // BQ).tolist())):
            _, cls = classify(kind, g, BQ, BKV, True, qt, qt + 1)
            kept[qt] = (cls[0] != SKIP)
        kept_ptr = kept.ctypes.data
    O = np.zeros((rows.size, d), dtype=np.float64)
    lse = np.zeros(rows.size, dtype=np.float64)
    gc = g.c()
    lib.orc_attention(Qp.ctypes.data, Kp.ctypes.data, Vp.ctypes.data, d, kind, ctypes.byref(gc),
                      float(scale), kept_ptr, BQ, BKV, lrows.ctypes.data, rows.size,
                      O.ctypes.data, lse.ctypes.data)
    return O, lse


def route(Q: np.ndarray, K: np.ndarray, V: np.ndarray, g: Geometry, rows):
    """Per-head routing from sampled queries, fp64 (blog section "Speeding up
    attention": compare each sampled query's spatial and temporal outputs with
    its dense output and pick the mask that deviates least).  Deviation = squared
    L2 distance to the dense output summed over rows and channels; temporal iff
    strictly smaller.  Q, K, V: [H][N][d] uint16 (bf16 bits), (F,H,W) order.
    Returns (flags uint8[H], errors float64[H][2])."""
    H = Q.shape[0]
    errors = np.zeros((H, 2), dtype=np.float64)
    for h in range(H):
        Od, _ = attention(Q[h], K[h], V[h], DENSE, g, rows=rows)
        Os, _ = attention(Q[h], K[h], V[h], SPATIAL, g, rows=rows)
        Ot, _ = attention(Q[h], K[h], V[h], TEMPORAL_FHW, g, rows=rows)
        errors[h, 0] = float(((Os - Od) ** 2).sum())
        errors[h, 1] = float(((Ot - Od) ** 2).sum())
    flags = (errors[:, 1] < errors[:, 0]).astype(np.uint8)
    return flags, errors
