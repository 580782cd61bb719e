"""GPU tile maps (closed-form interval counting) against the oracle's brute-force
classifier: CSR and statistics must match bit for bit."""
import numpy as np
import pytest

import oracle
import workloads as W

GEOMS = [  # name, F, Hs, Ws, wf, ws, head_dim, BQ, BKV
    ("tiny64", 4, 8, 8, 1, 10, 64, 64, 64),
    ("tiny128", 4, 8, 8, 1, 10, 64, 128, 128),
    ("ragged_s63", 5, 7, 9, 1, 5, 64, 64, 64),
    ("ragged_s130", 3, 10, 13, 0, 20, 128, 128, 128),
    ("small", 8, 16, 24, 2, 40, 128, 128, 128),
    ("small_odd_tiles", 8, 16, 24, 2, 40, 128, 96, 160),
]


def check_map(bss, tm, kind_code, g, BQ, BKV, rounding, qtiles=None):
    kind = 0 if kind_code == oracle.SPATIAL else 1
    row_ptr, entries = tm.csr(kind)
    nq, nkv, nnz, ncols = tm.dims(kind)
    assert ncols == oracle.num_cols(kind_code, g.with_bkv(BKV))
    if qtiles is None:
        orp, oent, ost = oracle.tile_map(kind_code, g, BQ, BKV, rounding)
        assert np.array_equal(row_ptr, orp)
        assert np.array_equal(entries, oent)
        st = tm.stats(kind)
        for key in ("full", "boundary", "pad", "skip", "retained_pairs", "exact_retained_pairs", "columns"):
            assert st[key] == ost[key], key
        return st
    for qt in qtiles:
        orp, oent, _ = oracle.tile_map(kind_code, g, BQ, BKV, rounding, qt, qt + 1)
        seg = entries[row_ptr[qt]:row_ptr[qt + 1]]
        assert np.array_equal(seg, oent), f"q tile {qt}"
    return tm.stats(kind)


@pytest.mark.gpu
@pytest.mark.parametrize("geo", GEOMS, ids=[x[0] for x in GEOMS])
@pytest.mark.parametrize("rounding", [0, 1, 2])
@pytest.mark.parametrize("tperm", [1, 0])
def test_tile_map_bit_exact_small(bss, geo, rounding, tperm):
    name, F, Hs, Ws, wf, ws, d, BQ, BKV = geo
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=rounding)
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=BKV)
    with bss.build_tile_map(p, BQ, BKV) as tm:
        check_map(bss, tm, oracle.SPATIAL, g, BQ, BKV, rounding)
        check_map(bss, tm, oracle.TEMPORAL_PERMUTED if tperm else oracle.TEMPORAL_FHW, g, BQ, BKV, rounding)


@pytest.mark.gpu
def test_tile_map_tiny_golden(bss):
    w = W.TINY
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    with bss.build_tile_map(p, 64, 64) as tm:
        row_ptr, entries = tm.csr(0)
        assert row_ptr.tolist() == [0, 2, 5, 9, 12]
        assert (entries & 0x3FFFFFFF).tolist() == [0, 1, 0, 1, 2, 0, 1, 2, 3, 0, 2, 3]
        assert ((entries.view(np.uint32) >> 30) == 0).all()
        st = tm.stats(0)
        assert (st["full"], st["boundary"], st["skip"], st["retained_pairs"]) == (12, 0, 4, 49152)


@pytest.mark.gpu
def test_tile_map_destroy_is_idempotent_and_blocks_use(bss):
    w = W.TINY
    tm = bss.build_tile_map(bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws), 64, 64)
    assert tm.dims(0)[0] == 4
    bss.destroy_tile_map(tm)
    bss.destroy_tile_map(tm)  # a second destroy is a no-op
    with pytest.raises(ValueError):
        tm.stats(0)


def closed_form_spatial(F, S, wf):
    return S * S * sum(min(f + wf, F - 1) - max(f - wf, 0) + 1 + (1 if f > wf else 0) for f in range(F))


def closed_form_temporal(F, S, ws):
    tot = 0
    for s in range(S):
        b = min(s + ws, S - 1) - max(s - ws, 0) + 1
        tot += F * b + (S - b)
    return F * tot


@pytest.mark.gpu
@pytest.mark.parametrize("wl", [W.SPATIAL_75K, W.MIXED_75K, W.P1440_302K], ids=lambda w: w.name)
@pytest.mark.parametrize("tperm", [1, 0])
def test_tile_map_full_size_sampled(bss, wl, tperm):
    g = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws, bkv=128)
    for rounding in (0, 1):
        p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=tperm, rounding=rounding)
        with bss.build_tile_map(p, 128, 128) as tm:
            nq = tm.dims(0)[0]
            qts = sorted({0, 1, nq // 3, nq // 2, nq - 2, nq - 1})
            st0 = check_map(bss, tm, oracle.SPATIAL, g, 128, 128, rounding, qts)
            st1 = check_map(bss, tm, oracle.TEMPORAL_PERMUTED if tperm else oracle.TEMPORAL_FHW, g, 128, 128,
                            rounding, qts)
            assert st0["exact_retained_pairs"] == closed_form_spatial(wl.F, wl.S, wl.wf)
            assert st1["exact_retained_pairs"] == closed_form_temporal(wl.F, wl.S, wl.ws)
            for st, kd in ((st0, 0), (st1, 1)):
                nq_, nkv, nnz, _ = tm.dims(kd)
                assert st["full"] + st["boundary"] + st["pad"] + st["columns"] + st["skip"] == nq_ * nkv
                assert st["full"] + st["boundary"] + st["pad"] + st["columns"] == nnz
                if rounding == 0:
                    assert st["retained_pairs"] == st["exact_retained_pairs"]
                    assert st["pad"] == 0


@pytest.mark.gpu
def test_tile_map_pages_tile_shape_sampled(bss):
    # the blog's reference tiles (3328 query rows x 1536 key columns) at 75.6K tokens
    wl = W.SPATIAL_75K
    g = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws, bkv=1536)
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=1, rounding=0)
    with bss.build_tile_map(p, 3328, 1536) as tm:
        nq = tm.dims(0)[0]
        assert nq == 23
        check_map(bss, tm, oracle.SPATIAL, g, 3328, 1536, 0, [0, nq - 1])
        assert tm.stats(0)["exact_retained_pairs"] == closed_form_spatial(wl.F, wl.S, wl.wf)


@pytest.mark.gpu
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("tperm", [1, 0])
def test_tile_map_whole_75k_matches_oracle(bss, rounding, tperm):
    # every q tile of the map the attention kernel runs at 75.6K tokens (256 x 128
    # tiles) against the oracle's brute-force classifier, CSR and statistics
    wl = W.MIXED_75K
    BQ, BKV = 256, 128
    g = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws, bkv=BKV)
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=tperm, rounding=rounding)
    with bss.build_tile_map(p, BQ, BKV) as tm:
        if tperm:
            check_map(bss, tm, oracle.SPATIAL, g, BQ, BKV, rounding)
        st = check_map(bss, tm, oracle.TEMPORAL_PERMUTED if tperm else oracle.TEMPORAL_FHW, g, BQ, BKV, rounding)
    if rounding == 1 and tperm:
        assert st["columns"] > 0
