"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle on the same seeded bf16 inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

# Parity bar for O (bf16 output, fp32 accumulation) on N(0,1) inputs:
# max |dO| <= 1e-2 and mean |dO| <= 1e-3; plus rel-L2 <= 1e-2 and |dLSE| <= 1e-3
# because |O| is only ~1e-2 when the softmax spreads over thousands of keys.
MAX_ABS, MEAN_ABS, REL_L2, LSE_ABS = 1e-2, 1e-3, 1e-2, 1e-3


def oracle_kind(flag: int, temporal_permuted: int) -> int:
    if not flag:
        return oracle.SPATIAL
    return oracle.TEMPORAL_PERMUTED if temporal_permuted else oracle.TEMPORAL_FHW


def run_gpu(bss, q, k, v, flags, params, want_lse=True, dense=False, BQ=None, BKV=None):
    """(F,H,W)-order CPU bf16 q, k, v -> (O [H][N][d] float32 CPU in (F,H,W) order,
    lse [H][N] float32 CPU in (F,H,W) order, tile map stats)."""
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in (q, k, v))
    H, N, d = Q.shape
    O = torch.empty_like(Q)
    lse = torch.empty(H, N, dtype=torch.float32, device=dev) if want_lse else None
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    stats = None
    if dense:
        bss.dense_attention(Q, K, V, O, lse=lse)
    else:
        ws = [torch.empty_like(Q) for _ in range(3)]
        with bss.build_tile_map(params, BQ=BQ or bss.ATTN_BQ, BKV=BKV or bss.ATTN_BKV) as tm:
            bss.attention_step(Q, K, V, O, tm, fl, *ws, lse=lse)
            stats = (tm.stats(0), tm.stats(1))
            torch.cuda.synchronize()
    st = bss.get_device_status()
    assert st == 0, bss.status_string(st)
    torch.cuda.synchronize()
    out = O.float().cpu()
    lse_c = None
    if want_lse:
        lse_c = lse.cpu()
        if params is not None and params.temporal_permuted and not dense:
            F, S = params.F, params.S
            t = torch.arange(N)
            p = (t % S) * F + t // S          # layout position of original token t
            for h in range(H):
                if flags[h]:
                    lse_c[h] = lse_c[h][p]
    return out, lse_c, stats


def oracle_rows(q, k, v, h, kind, g, rows, rounding, dense=False, BQ=None, BKV=None):
    """Oracle rows; a rounded mask is rounded on the attention kernel's tile grid."""
    import block_sparse_spatio_gb300 as bss
    b = W.bf16_bits
    if dense:
        kind = oracle.DENSE
    return oracle.attention(b(q[h]), b(k[h]), b(v[h]), kind, g, rows=rows, rounding=bool(rounding),
                            BQ=BQ or bss.ATTN_BQ, BKV=BKV or bss.ATTN_BKV)


def compare(out_rows: np.ndarray, lse_rows, Oref: np.ndarray, lref: np.ndarray, what: str):
    d = np.abs(out_rows.astype(np.float64) - Oref)
    maxe, meane = float(d.max()), float(d.mean())
    rel = float(np.linalg.norm(out_rows - Oref) / max(np.linalg.norm(Oref), 1e-30))
    msg = f"{what}: max {maxe:.3e} mean {meane:.3e} relL2 {rel:.3e}"
    assert maxe <= MAX_ABS, msg
    assert meane <= MEAN_ABS, msg
    assert rel <= REL_L2, msg
    if lse_rows is not None:
        fin = np.isfinite(lref)
        assert np.array_equal(np.isfinite(lse_rows), fin), what + ": -inf rows differ"
        if fin.any():
            le = float(np.abs(lse_rows[fin] - lref[fin]).max())
            assert le <= LSE_ABS, f"{what}: max |dLSE| {le:.3e}"
    return maxe, meane, rel


def rounded_row_counts(kind: int, g, BQ: int, BKV: int, qt0: int = 0, qt1=None):
    """Distinct keys kept by each LAYOUT query row of q tiles [qt0, qt1) under the
    tile-aligned mask, from the oracle's brute-force tile classes: every real row
    of a q tile keeps the physical keys that the real columns of its kept tiles
    read, each key once.  Returns an int64 array over the rows of those tiles
    (padding rows past N dropped)."""
    gg = g.with_bkv(BKV)
    _, cls = oracle.classify(kind, gg, BQ, BKV, 1, qt0, qt1)
    keys = oracle.key_rows(kind, gg)
    ncols = keys.size
    k = np.arange(ncols)
    real = ((k < gg.S) | (k >= gg.S_pad)) if kind == oracle.TEMPORAL_PERMUTED else np.ones(ncols, bool)
    per_tile = np.array([np.unique(keys[np.repeat(c != oracle.SKIP, BKV)[:ncols] & real]).size for c in cls],
                        dtype=np.int64)
    rows = np.repeat(per_tile, BQ)
    return rows[: max(0, min(rows.size, gg.N - qt0 * BQ))]


def exact_row_counts(kind: int, F: int, S: int, wf: int, ws: int):
    """Closed-form retained keys of every query token t = f*S + s in (F,H,W)
    order: spatial S*(frames in the band + the sink frame when outside it),
    temporal F*b + (S - b) with b the raster positions in the band."""
    t = np.arange(F * S, dtype=np.int64)
    f, s = t // S, t % S
    if kind == oracle.SPATIAL:
        return S * (np.minimum(f + wf, F - 1) - np.maximum(f - wf, 0) + 1 + (f > wf))
    b = np.minimum(s + ws, S - 1) - np.maximum(s - ws, 0) + 1
    return F * b + (S - b)


def fhw_of_layout(values: np.ndarray, F: int, S: int) -> np.ndarray:
    """Reorder per-row values of a permuted (H,W,F) head to (F,H,W) token order."""
    t = np.arange(F * S)
    return values[(t % S) * F + t // S]
