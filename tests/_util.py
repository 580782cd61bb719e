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
        ws = [torch.empty_like(Q) for _ in range(4)]
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
