"""Exact coverage at the sizes the benchmark runs: which keys every row sees.

With Q = 0 every retained key gets weight exp(0) = 1, so exp(LSE_i) is the
number of keys row i keeps: an exact, per-row pin of the mask (blog, section
"Logical sparsity is not physical sparsity": excluded pairs carry no weight;
section "Align the sparse mask with final execution": the rounded mask keeps
whole tiles).  Exact masks are checked against closed-form per-row counts,
tile-aligned masks against the distinct keys of the oracle's kept tiles.  The
poison test puts huge keys and values at excluded positions of interior q tiles
and requires the outputs there to stay bit for bit the same."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import exact_row_counts, fhw_of_layout, rounded_row_counts


def _zero_query_step(bss, wl, tperm, rounding, H=None, seed=None, BQ=None, BKV=None):
    """Run the step with Q = 0 and seeded K, V on the device; LSE per head in
    (F,H,W) token order (float64, CPU)."""
    dev = torch.device("cuda")
    H = wl.H if H is None else H
    g = torch.Generator(device=dev).manual_seed(wl.index + 500 if seed is None else seed)
    K = torch.randn(H, wl.N, wl.d, generator=g, device=dev).to(torch.bfloat16)
    V = torch.randn(H, wl.N, wl.d, generator=g, device=dev).to(torch.bfloat16)
    Q = torch.zeros_like(K)
    flags = wl.head_flags()[:H]
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    O = torch.empty_like(Q)
    lse = torch.empty(H, wl.N, device=dev)
    ws = [torch.empty_like(Q) for _ in range(3)]
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=tperm, rounding=rounding)
    with bss.build_tile_map(p, BQ=BQ or bss.ATTN_BQ, BKV=BKV or bss.ATTN_BKV) as tm:
        bss.attention_step(Q, K, V, O, tm, fl, *ws, lse=lse)
        torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    out = lse.double().cpu().numpy()
    for h in range(H):
        if flags[h] and tperm:
            out[h] = fhw_of_layout(out[h], wl.F, wl.S)
    return flags, out


def _counts_of(lse_row):
    return np.rint(np.exp(lse_row)).astype(np.int64)


@pytest.mark.gpu
@pytest.mark.parametrize("case", [("mixed_75600tok_10h_d128", 1), ("mixed_75600tok_10h_d128", 0),
                                  ("p1440_302400tok_10h_d128", 1)], ids=["mixed75k_hwf", "mixed75k_fhw", "p1440"])
def test_exact_mask_coverage_every_row_every_head(bss, case):
    name, tperm = case
    wl = W.BY_NAME[name]
    flags, lse = _zero_query_step(bss, wl, tperm, 0)
    want = {k: exact_row_counts(k, wl.F, wl.S, wl.wf, wl.ws) for k in (oracle.SPATIAL, oracle.TEMPORAL_FHW)}
    for h, fl in enumerate(flags):
        exp = want[oracle.TEMPORAL_FHW if fl else oracle.SPATIAL]
        got = _counts_of(lse[h])
        bad = np.nonzero(got != exp)[0]
        assert bad.size == 0, f"{name} head {h}: {bad.size} rows differ, first {bad[:8]}"


@pytest.mark.gpu
@pytest.mark.parametrize("tile", [(128, 128), (256, 64), (128, 64)], ids=lambda t: f"{t[0]}x{t[1]}")
def test_exact_mask_coverage_every_row_other_tiles_75k(bss, tile):
    # the other kernel instances (one 128-row half per CTA, 64-key tiles) at the
    # benchmark's size, both head kinds, every row
    wl = W.MIXED_75K
    BQ, BKV = tile
    flags, lse = _zero_query_step(bss, wl, 1, 0, BQ=BQ, BKV=BKV)
    want = {k: exact_row_counts(k, wl.F, wl.S, wl.wf, wl.ws) for k in (oracle.SPATIAL, oracle.TEMPORAL_FHW)}
    for h, fl in enumerate(flags):
        got = _counts_of(lse[h])
        bad = np.nonzero(got != want[oracle.TEMPORAL_FHW if fl else oracle.SPATIAL])[0]
        assert bad.size == 0, f"{tile} head {h}: {bad.size} rows differ, first {bad[:8]}"


@pytest.mark.gpu
def test_dense_control_coverage_every_row(bss):
    # Q = 0: every row of the dense control keeps all N keys, also through the
    # ragged last kv tile (75,600 = 590 x 128 + 80)
    wl = W.MIXED_75K
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(17)
    K = torch.randn(wl.H, wl.N, wl.d, generator=g, device=dev).to(torch.bfloat16)
    V = torch.randn(wl.H, wl.N, wl.d, generator=g, device=dev).to(torch.bfloat16)
    Q = torch.zeros_like(K)
    O = torch.empty_like(Q)
    lse = torch.empty(wl.H, wl.N, device=dev)
    bss.dense_attention(Q, K, V, O, lse=lse)
    torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    got = _counts_of(lse.double().cpu().numpy())
    assert np.all(got == wl.N), np.nonzero(got != wl.N)


@pytest.mark.gpu
@pytest.mark.parametrize("BQ", [128, 256])
@pytest.mark.parametrize("BKV", [128, 64])
def test_rounded_mask_coverage_small_is_distinct_keys(bss, BQ, BKV):
    wl = W.SMALL
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(91)
    K = torch.randn(2, wl.N, wl.d, generator=g, device=dev).to(torch.bfloat16)
    V = torch.randn(2, wl.N, wl.d, generator=g, device=dev).to(torch.bfloat16)
    Q = torch.zeros_like(K)
    fl = torch.tensor([0, 1], dtype=torch.uint8, device=dev)
    O = torch.empty_like(Q)
    lse = torch.empty(2, wl.N, device=dev)
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=1, rounding=1)
    with bss.build_tile_map(p, BQ=BQ, BKV=BKV) as tm:
        assert tm.stats(1)["columns"] > 0  # sink tiles that lose their band twins
        bss.attention_step(Q, K, V, O, tm, fl, *[torch.empty_like(Q) for _ in range(3)], lse=lse)
        torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    go = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws)
    got = lse.double().cpu().numpy()
    want0 = rounded_row_counts(oracle.SPATIAL, go, BQ, BKV)
    want1 = rounded_row_counts(oracle.TEMPORAL_PERMUTED, go, BQ, BKV)   # layout order
    np.testing.assert_array_equal(_counts_of(got[0]), want0)
    np.testing.assert_array_equal(_counts_of(got[1]), want1)


@pytest.mark.gpu
def test_rounded_mask_coverage_75k_every_row(bss):
    # temporal heads permuted, tile-aligned: every row's key count equals the
    # distinct keys of its q tile's kept tiles (no frame-0 key counted twice)
    wl = W.MIXED_75K
    flags, lse = _zero_query_step(bss, wl, 1, 1)
    go = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws)
    want = {0: rounded_row_counts(oracle.SPATIAL, go, bss.ATTN_BQ, bss.ATTN_BKV),
            1: fhw_of_layout(rounded_row_counts(oracle.TEMPORAL_PERMUTED, go, bss.ATTN_BQ, bss.ATTN_BKV),
                             wl.F, wl.S)}
    for h, fl in enumerate(flags):
        got = _counts_of(lse[h])
        bad = np.nonzero(got != want[fl])[0]
        assert bad.size == 0, f"head {h}: {bad.size} rows differ, first {bad[:8]}"


@pytest.mark.gpu
def test_rounded_mask_coverage_1440p(bss):
    # 302.4K tokens, tile-aligned: all rows of a q tile keep the same keys; the
    # count of sampled q tiles equals the distinct keys of the oracle's kept
    # tiles, and the counts sum to the map's retained pairs
    wl = W.P1440_302K
    flags, lse = _zero_query_step(bss, wl, 1, 1)
    go = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws)
    BQ = bss.ATTN_BQ
    nq = -(-wl.N // BQ)
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=1, rounding=1)
    with bss.build_tile_map(p) as tm:
        retained = (tm.stats(0)["retained_pairs"], tm.stats(1)["retained_pairs"])
    sample = sorted({0, 1, nq // 3, nq // 2, (2 * nq) // 3, nq - 2, nq - 1})
    seen = set()
    for h, fl in enumerate(flags):
        if fl in seen:
            continue
        seen.add(fl)
        got = _counts_of(lse[h])
        if fl:
            t = np.arange(wl.N)
            layout = np.empty_like(got)
            layout[(t % wl.S) * wl.F + t // wl.S] = got   # back to (H,W,F) rows
            got = layout
        pad = np.full(nq * BQ, -1, np.int64)
        pad[: wl.N] = got
        per_tile = pad.reshape(nq, BQ)
        for i in range(nq):
            row = per_tile[i][per_tile[i] >= 0]
            assert np.all(row == row[0]), f"head {h} q tile {i}: rows see different key counts"
        assert int(got.sum()) == retained[fl], f"head {h}"
        kind = oracle.TEMPORAL_PERMUTED if fl else oracle.SPATIAL
        for i in sample:
            want = rounded_row_counts(kind, go, BQ, bss.ATTN_BKV, i, i + 1)
            assert per_tile[i][0] == want[0], f"head {h} q tile {i}: {per_tile[i][0]} != {want[0]}"
    assert seen == {0, 1}


@pytest.mark.gpu
def test_poisoned_excluded_keys_interior_q_tiles_75k(bss):
    # Interior q tiles of the 75.6K geometry (of 296 at 256 rows): a spatial
    # head's queries of frame 10 keep frames 0 and 7..13; a temporal head's
    # queries at raster 1800..1899 keep rasters 1188..2511 of every frame plus
    # frame 0.  Huge keys and values everywhere else must not change their rows.
    wl = W.MIXED_75K
    F, S, N, d = wl.F, wl.S, wl.N, wl.d
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(2024)
    Q, K, V = (torch.randn(2, N, d, generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
    fl = torch.tensor([0, 1], dtype=torch.uint8, device=dev)
    p = bss.MaskParams(F, wl.Hs, wl.Ws, d, wl.wf, wl.ws, temporal_permuted=1, rounding=0)
    t = torch.arange(N, device=dev)
    f, s = t // S, t % S
    far0 = ((f >= 1) & (f <= 6)) | (f >= 14)
    far1 = (f >= 1) & ((s < 1188) | (s > 2511))
    rows0 = torch.nonzero(f == 10).flatten()
    rows1 = torch.nonzero((s >= 1800) & (s < 1900)).flatten()
    qt0 = set((rows0 // 256).tolist())
    qt1 = set((((rows1 % S) * F + rows1 // S) // 256).tolist())
    assert min(qt0) > 100 and max(qt0) < 200 and min(qt1) > 100 and max(qt1) < 200
    outs = []
    with bss.build_tile_map(p) as tm:
        for poison in (False, True):
            K2, V2 = K.clone(), V.clone()
            if poison:
                K2[0, far0] = 1.0e4
                V2[0, far0] = -1.0e4
                K2[1, far1] = -1.0e4
                V2[1, far1] = 1.0e4
            O = torch.empty_like(Q)
            lse = torch.empty(2, N, device=dev)
            bss.attention_step(Q, K2, V2, O, tm, fl, *[torch.empty_like(Q) for _ in range(3)], lse=lse)
            torch.cuda.synchronize()
            assert bss.get_device_status() == 0
            outs.append((O, lse))
    (O1, l1), (O2, l2) = outs
    assert torch.equal(O1[0, rows0].view(torch.int16), O2[0, rows0].view(torch.int16))
    assert torch.equal(O1[1, rows1].view(torch.int16), O2[1, rows1].view(torch.int16))
    perm1 = (rows1 % S) * F + rows1 // S   # LSE of a permuted head is in layout order
    assert torch.equal(l1[0, rows0].view(torch.int32), l2[0, rows0].view(torch.int32))
    assert torch.equal(l1[1, perm1].view(torch.int32), l2[1, perm1].view(torch.int32))
    # the poison is visible to rows that keep those keys
    seen = torch.nonzero(f == 3).flatten()
    assert not torch.equal(O1[0, seen], O2[0, seen])
