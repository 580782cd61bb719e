"""Pins for the fp64 oracle, each independent of the oracle's own code.

The oracle (oracle/bss_oracle.c) decodes coordinates with div/mod and tests one
pair at a time.  The pins below rebuild the masks from meshgrid coordinates as
explicit N x N boolean matrices, count tiles with numpy reshapes, and run a
textbook float64 masked softmax through torch -- so a dropped sink term, a wrong
window sign or index, a transposed operand or a wrong tile rule in the oracle
fails at least one of them.  Mask definitions: blog "Accelerating
Spatio-Temporal Attention for Video Diffusion on TPUs" (Figure 3; sections
"Logical sparsity is not physical sparsity", "Align the sparse mask with final
execution", "Arrange tokens for efficient temporal access").
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import DENSE, SPATIAL, TEMPORAL_FHW, TEMPORAL_PERMUTED

HERE = os.path.dirname(os.path.abspath(__file__))

# (name, F, Hs, Ws, wf, ws, BQ, BKV): Tiny and Small from the workloads, plus
# two ragged geometries (N and S not multiples of the tile) to exercise padding.
GEOMS = [
    ("tiny", 4, 8, 8, 1, 10, 64, 64),
    ("ragged_s63", 5, 7, 9, 1, 5, 64, 64),
    ("ragged_s130", 3, 10, 13, 0, 20, 128, 128),
    ("small", 8, 16, 24, 2, 40, 128, 128),
]


# ----------------------------------------------------------------------------
# independent reconstructions (no div/mod, explicit matrices)
# ----------------------------------------------------------------------------
def coords(F, Hs, Ws):
    """Frame index and raster index of every token in (F,H,W) order, via meshgrid."""
    f, h, w = np.meshgrid(np.arange(F), np.arange(Hs), np.arange(Ws), indexing="ij")
    return f.ravel(), (h * Ws + w).ravel()


def phys_mask(kind, F, Hs, Ws, wf, ws):
    """Explicit N x N retained matrix over physical tokens in (F,H,W) order."""
    f, s = coords(F, Hs, Ws)
    sink = np.broadcast_to(f[None, :] == 0, (f.size, f.size))
    if kind == SPATIAL:
        band = np.abs(f[:, None] - f[None, :]) <= wf
    elif kind == DENSE:
        return np.ones((f.size, f.size), bool)
    else:
        band = np.abs(s[:, None] - s[None, :]) <= ws
    return band | sink


def perm_tokens(F, S):
    """Position p of the (H,W,F) order holds original token perm_tokens[p]."""
    return (np.arange(F)[None, :] * S + np.arange(S)[:, None]).ravel()


def layout_mask(kind, F, Hs, Ws, wf, ws, BKV):
    """Retained matrix in the kernel's layout: rows are layout queries, columns
    the layout's key columns, plus the physical token each column reads and a
    real-column flag.  For temporal (H,W,F) heads the key columns are a sink
    segment (frame-0 key at raster v, v < S, padded to a BKV multiple) followed
    by the N permuted rows; a frame-0 key counts in the band when the band
    covers it and in the sink segment otherwise."""
    S = Hs * Ws
    N = F * S
    if kind != TEMPORAL_PERMUTED:
        M = phys_mask(SPATIAL if kind == SPATIAL else (DENSE if kind == DENSE else TEMPORAL_FHW), F, Hs, Ws, wf, ws)
        return M, np.arange(N), np.ones(N, bool), np.arange(N)
    pt = perm_tokens(F, S)
    f, s = coords(F, Hs, Ws)
    sq = s[pt]                       # raster of each permuted query
    S_pad = -(-S // BKV) * BKV
    band_cols = np.abs(sq[:, None] - s[pt][None, :]) <= ws
    sink_raster = np.arange(S_pad)
    sink_cols = (np.abs(sq[:, None] - sink_raster[None, :]) > ws) & (sink_raster[None, :] < S)
    M = np.concatenate([sink_cols, band_cols], axis=1)
    col_tok = np.concatenate([np.where(sink_raster < S, sink_raster, 0), pt])   # frame-0 token at raster v is token v
    col_real = np.concatenate([sink_raster < S, np.ones(N, bool)])
    return M, col_tok, col_real, pt


def tile_classes(M, col_real, BQ, BKV, rounding, col_tok=None):
    """Tile counts and classes by numpy reshapes of the layout matrix.  With
    ``col_tok`` (rounded masks), a kept sink-segment column whose physical token
    is also read by another kept column of the same q tile is dropped: a kept
    tile left with none of its real columns is SKIP, with some COLUMNS."""
    N, C = M.shape
    nq, nkv = -(-N // BQ), -(-C // BKV)
    Mp = np.zeros((nq * BQ, nkv * BKV), bool)
    Mp[:N, :C] = M
    cr = np.zeros(nkv * BKV, bool)
    cr[:C] = col_real
    counts = Mp.reshape(nq, BQ, nkv, BKV).sum(axis=(1, 3))
    real_rows = np.minimum(BQ, N - np.arange(nq) * BQ)
    real_cols = cr.reshape(nkv, BKV).sum(1)
    area = np.outer(real_rows, real_cols)
    cls = np.full((nq, nkv), oracle.SKIP, np.int8)
    if rounding == 2:  # naive traversal: every visited tile masks
        cls[counts > 0] = oracle.BOUNDARY
    elif rounding:
        kept = (area > 0) & (2 * counts >= area)
        cls[kept] = oracle.FULL
        cls[kept & (real_cols[None, :] < BKV)] = oracle.PAD
        if col_tok is not None:
            # how many kept real columns of q tile i read each token
            kc = np.repeat(kept, BKV, axis=1)[:, :C] & col_real[None, :]
            mult = token_counts(kc, col_tok, col_real, N)
            S_pad = C - N
            for i in range(nq):
                for j in range(S_pad // BKV):
                    if not kept[i, j]:
                        continue
                    cols = np.arange(j * BKV, (j + 1) * BKV)
                    cols = cols[col_real[cols]]
                    dropped = mult[i, col_tok[cols]] >= 2
                    if dropped.all():
                        cls[i, j] = oracle.SKIP
                    elif dropped.any():
                        cls[i, j] = oracle.COLUMNS
    else:
        cls[counts > 0] = oracle.BOUNDARY
        full = (counts == real_rows[:, None] * BKV) & (real_cols[None, :] == BKV) & (counts > 0)
        cls[full] = oracle.FULL
    return counts, cls


def token_counts(keep, col_tok, col_real, N):
    """R x N counts: how many real columns c with keep[:, c] read each token."""
    out = np.zeros((keep.shape[0], N), np.int64)
    for c in np.nonzero(col_real)[0]:
        out[:, col_tok[c]] += keep[:, c]
    return out


def rounded_phys_mask(kind, F, Hs, Ws, wf, ws, BQ, BKV):
    """Rounded mask as an explicit matrix over PHYSICAL tokens: rows are layout
    queries, columns the N tokens in (F,H,W) order; a pair is retained iff some
    real column of a kept tile of the query's q tile reads that token (a set:
    a token read through two columns is one pair)."""
    M, col_tok, col_real, pt = layout_mask(kind, F, Hs, Ws, wf, ws, BKV)
    N = M.shape[0]
    counts, _ = tile_classes(M, col_real, BQ, BKV, 0)
    real_rows = np.minimum(BQ, N - np.arange(counts.shape[0]) * BQ)
    cr = np.zeros(counts.shape[1] * BKV, bool)
    cr[: col_real.size] = col_real
    area = np.outer(real_rows, cr.reshape(-1, BKV).sum(1))
    kept = (area > 0) & (2 * counts >= area)
    keep = np.repeat(np.repeat(kept, BQ, 0), BKV, 1)[:N, : M.shape[1]] & col_real[None, :]
    P = token_counts(keep, col_tok, col_real, N) > 0
    return P, pt


def torch_attention(Qf, Kf, Vf, mask, scale):
    """Textbook float64 masked softmax attention (rows with no key excluded by caller)."""
    s = (Qf @ Kf.T) * scale
    s = s.masked_fill(~mask, float("-inf"))
    return torch.softmax(s, dim=-1) @ Vf, torch.logsumexp(s, dim=-1)


def rand_head(N, d, seed):
    q, k, v = W.qkv(W.SMALL, H=1, N=N, d=d, seed=seed)
    return q[0], k[0], v[0]


def bits(x):
    return W.bf16_bits(x)


def geom(F, Hs, Ws, wf, ws, BKV):
    return oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=BKV)


KINDS = [SPATIAL, TEMPORAL_PERMUTED, TEMPORAL_FHW]


# ----------------------------------------------------------------------------
# permutation
# ----------------------------------------------------------------------------
def test_permutation_hand_values_small():
    # Small geometry F=8, S=16*24=384: token (f=1, s=0) -> p = 0*8 + 1 = 1,
    # token (f=0, s=1) -> p = 1*8 + 0 = 8 (Figure 9: same position across frames adjacent)
    F, S = 8, 384
    assert oracle.perm_index(1 * S + 0, F, S) == 1
    assert oracle.perm_index(0 * S + 1, F, S) == 8
    assert oracle.unperm_index(8, F, S) == 1
    pt = perm_tokens(F, S)
    assert all(oracle.perm_index(int(pt[p]), F, S) == p for p in range(0, F * S, 37))


def test_permutation_round_trip_and_flags():
    F, Hs, Ws, d = 5, 7, 9, 16
    S = Hs * Ws
    x = np.random.default_rng(0).integers(0, 65535, size=(3, F * S, d), dtype=np.uint16)
    flags = [1, 0, 1]
    y = oracle.permute(x, F, S, flags)
    assert np.array_equal(y[1], x[1])                      # spatial head keeps its order
    pt = perm_tokens(F, S)
    assert np.array_equal(y[0], x[0][pt])                  # temporal head gathered (H,W,F)
    z = oracle.permute(y, F, S, flags, inverse=True)
    assert np.array_equal(z, x)                            # bit-exact round trip


def test_permutation_makes_temporal_band_contiguous():
    # after the permutation a temporal query's band keys form one contiguous run
    F, Hs, Ws, ws = 6, 5, 7, 4
    S = Hs * Ws
    M, col_tok, col_real, pt = layout_mask(TEMPORAL_PERMUTED, F, Hs, Ws, 0, ws, 64)
    S_pad = M.shape[1] - F * S
    for q in range(0, F * S, 11):
        band = np.nonzero(M[q, S_pad:])[0]
        assert band.size and np.all(np.diff(band) == 1)


# ----------------------------------------------------------------------------
# predicate and tile classification
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("g", GEOMS, ids=[g[0] for g in GEOMS])
@pytest.mark.parametrize("kind", KINDS)
def test_retained_predicate_matches_explicit_matrix(g, kind):
    name, F, Hs, Ws, wf, ws, BQ, BKV = g
    M, col_tok, col_real, pt = layout_mask(kind, F, Hs, Ws, wf, ws, BKV)
    gg = geom(F, Hs, Ws, wf, ws, BKV)
    rng = np.random.default_rng(1)
    for q in rng.integers(0, M.shape[0], 12):
        row = np.array([oracle.retained(kind, gg, int(q), k) for k in range(M.shape[1])], bool)
        assert np.array_equal(row, M[q])


@pytest.mark.parametrize("g", GEOMS, ids=[g[0] for g in GEOMS])
def test_temporal_virtual_space_counts_each_key_once(g):
    # the union of the sink and band copies equals the physical temporal mask, no duplicates
    name, F, Hs, Ws, wf, ws, BQ, BKV = g
    M, col_tok, col_real, pt = layout_mask(TEMPORAL_PERMUTED, F, Hs, Ws, wf, ws, BKV)
    P = phys_mask(TEMPORAL_FHW, F, Hs, Ws, wf, ws)
    for q in range(0, M.shape[0], 7):
        toks = col_tok[M[q] & col_real]
        assert len(set(toks.tolist())) == toks.size
        assert np.array_equal(np.sort(toks), np.nonzero(P[pt[q]])[0])


@pytest.mark.parametrize("g", GEOMS, ids=[g[0] for g in GEOMS])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("rounding", [0, 1, 2])
def test_classify_matches_numpy_tiling(g, kind, rounding):
    name, F, Hs, Ws, wf, ws, BQ, BKV = g
    M, col_tok, col_real, pt = layout_mask(kind, F, Hs, Ws, wf, ws, BKV)
    counts_np, cls_np = tile_classes(M, col_real, BQ, BKV, rounding, col_tok if rounding == 1 else None)
    counts, cls = oracle.classify(kind, geom(F, Hs, Ws, wf, ws, BKV), BQ, BKV, rounding)
    assert np.array_equal(counts, counts_np)
    assert np.array_equal(cls, cls_np)
    row_ptr, entries, stats = oracle.tile_map(kind, geom(F, Hs, Ws, wf, ws, BKV), BQ, BKV, rounding)
    e = entries.view(np.uint32)
    for i in range(cls.shape[0]):
        seg = e[row_ptr[i]:row_ptr[i + 1]]
        js = seg & ((1 << 30) - 1)
        assert np.all(np.diff(js.astype(np.int64)) > 0)            # ascending kv index
        assert np.array_equal(js, np.nonzero(cls_np[i] != oracle.SKIP)[0])
        assert np.array_equal(seg >> 30, cls_np[i][js])


def test_tiny_tile_map_golden():
    expect = {}
    with open(os.path.join(HERE, "golden", "tiny_tile_map.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            qt, rest = line.split(":")
            expect[int(qt)] = [(int(tok[:-1]), {"F": 0, "B": 1, "P": 2}[tok[-1]]) for tok in rest.split()]
    w = W.TINY
    for rounding in (0, 1):
        row_ptr, entries, stats = oracle.tile_map(SPATIAL, geom(w.F, w.Hs, w.Ws, w.wf, w.ws, w.BKV),
                                                  w.BQ, w.BKV, rounding)
        e = entries.view(np.uint32)
        for qt, ents in expect.items():
            seg = e[row_ptr[qt]:row_ptr[qt + 1]]
            assert [(int(x & 0x3FFFFFFF), int(x >> 30)) for x in seg] == ents
        assert (stats["full"], stats["boundary"], stats["skip"]) == (12, 0, 4)
        assert stats["retained_pairs"] == 49152


# ----------------------------------------------------------------------------
# closed-form retained-pair counts
# ----------------------------------------------------------------------------
def closed_form_spatial(F, S, wf):
    return S * S * sum(min(f + wf, F - 1) - max(f - wf, 0) + 1 + (1 if f > wf else 0) for f in range(F))


def closed_form_temporal(F, S, ws):
    tot = 0
    for s in range(S):
        b = min(s + ws, S - 1) - max(s - ws, 0) + 1
        tot += F * b + (S - b)
    return F * tot


def closed_form_row(kind, F, S, wf, ws, t):
    """Retained keys of one query, (F,H,W) token t."""
    f, s = t // S, t % S
    if kind == SPATIAL:
        return S * (min(f + wf, F - 1) - max(f - wf, 0) + 1 + (1 if f > wf else 0))
    b = min(s + ws, S - 1) - max(s - ws, 0) + 1
    return F * b + (S - b)


@pytest.mark.parametrize("g", GEOMS, ids=[g[0] for g in GEOMS])
def test_retained_counts_closed_form(g):
    name, F, Hs, Ws, wf, ws, BQ, BKV = g
    S = Hs * Ws
    gg = geom(F, Hs, Ws, wf, ws, BKV)
    _, _, st = oracle.tile_map(SPATIAL, gg, BQ, BKV, 0)
    assert st["retained_pairs"] == closed_form_spatial(F, S, wf)
    for kind in (TEMPORAL_PERMUTED, TEMPORAL_FHW):
        _, _, st = oracle.tile_map(kind, gg, BQ, BKV, 0)
        assert st["retained_pairs"] == closed_form_temporal(F, S, ws)


def test_closed_forms_at_workload_sizes():
    # values of the closed forms for the workloads (derived, not printed by the pages)
    assert closed_form_spatial(4, 64, 1) == 49152
    assert closed_form_spatial(8, 384, 2) == 5750784
    assert closed_form_temporal(8, 384, 40) == 2829632
    assert closed_form_spatial(21, 3600, 3) == 1969920000
    assert closed_form_temporal(21, 3600, 612) == 1966794480


@pytest.mark.parametrize("kind", [SPATIAL, TEMPORAL_PERMUTED])
def test_classify_rows_at_75k_match_closed_form(kind):
    # sampled q-tile rows of the full 75.6K geometry: the oracle's brute-force
    # tile counts summed over a q-tile equal the closed-form per-query counts
    w = W.MIXED_75K
    gg = geom(w.F, w.Hs, w.Ws, w.wf, w.ws, 128)
    N, S, F = w.N, w.S, w.F
    for qt in (0, 300, N // 128):
        counts, _ = oracle.classify(kind, gg, 128, 128, 0, qt, qt + 1)
        rows = range(qt * 128, min(N, qt * 128 + 128))
        if kind == TEMPORAL_PERMUTED:
            toks = [oracle.unperm_index(p, F, S) for p in rows]
        else:
            toks = list(rows)
        assert counts.sum() == sum(closed_form_row(kind, F, S, w.wf, w.ws, t) for t in toks)


# ----------------------------------------------------------------------------
# attention values
# ----------------------------------------------------------------------------
def _oracle_vs_torch(name, F, Hs, Ws, wf, ws, BQ, BKV, kind, rounding, d=64, seed=5):
    S = Hs * Ws
    N = F * S
    q, k, v = rand_head(N, d, seed)
    gg = geom(F, Hs, Ws, wf, ws, BKV)
    O, lse = oracle.attention(bits(q), bits(k), bits(v), kind, gg, rounding=rounding, BQ=BQ, BKV=BKV)
    M, col_tok, col_real, pt = layout_mask(kind, F, Hs, Ws, wf, ws, BKV)
    Qf, Kf, Vf = q.double(), k.double(), v.double()
    if rounding:
        # rows in layout order, keys the physical tokens of the explicit rounded matrix
        P, pt = rounded_phys_mask(kind, F, Hs, Ws, wf, ws, BQ, BKV)
        Ol, lsel = torch_attention(Qf[pt], Kf, Vf, torch.from_numpy(P), 1.0 / np.sqrt(d))
    else:
        # rows in layout order, keys through the column -> token map
        Ol, lsel = torch_attention(Qf[pt], Kf[col_tok], Vf[col_tok], torch.from_numpy(M), 1.0 / np.sqrt(d))
    Oref = torch.empty_like(Ol)
    lref = torch.empty_like(lsel)
    Oref[pt] = Ol
    lref[pt] = lsel
    np.testing.assert_allclose(O, Oref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("g", GEOMS, ids=[g[0] for g in GEOMS])
@pytest.mark.parametrize("kind", KINDS)
def test_attention_exact_mask_vs_bruteforce(g, kind):
    _oracle_vs_torch(*g, kind=kind, rounding=0)


@pytest.mark.parametrize("g", GEOMS, ids=[g[0] for g in GEOMS])
@pytest.mark.parametrize("kind", KINDS)
def test_attention_rounded_mask_vs_bruteforce(g, kind):
    _oracle_vs_torch(*g, kind=kind, rounding=1)


@pytest.mark.parametrize("BQ", [128, 256])
def test_rounded_mask_rows_left_empty_give_zero_and_minus_infinity(BQ):
    # One raster position and 130 frames: a spatial row keeps 6 of 128 keys in its
    # tiles, so rounding drops all tiles of the first q tile (and at BQ = 256 every
    # tile); an empty row's output is 0 and its LSE -inf, the rest is the textbook
    # softmax over the kept tiles.
    F, Hs, Ws, wf, ws, BKV, d = 130, 1, 1, 2, 0, 128, 64
    N = F
    q, k, v = rand_head(N, d, 12)
    gg = geom(F, Hs, Ws, wf, ws, BKV)
    O, lse = oracle.attention(bits(q), bits(k), bits(v), SPATIAL, gg, rounding=True, BQ=BQ, BKV=BKV)
    M, col_tok, col_real, pt = layout_mask(SPATIAL, F, Hs, Ws, wf, ws, BKV)
    _, cls = tile_classes(M, col_real, BQ, BKV, 1)
    keep = np.repeat(np.repeat(cls != oracle.SKIP, BQ, 0), BKV, 1)[:N, :N]
    M = keep & col_real[None, :]
    empty = ~M.any(axis=1)
    assert empty[:128].all() and empty.all() == (BQ == 256)
    assert np.all(O[empty] == 0.0) and np.all(np.isneginf(lse[empty]))
    live = ~empty
    if live.any():
        Qf, Kf, Vf = q.double(), k.double(), v.double()
        Ol, ll = torch_attention(Qf[live], Kf, Vf, torch.from_numpy(M[live]), 1.0 / np.sqrt(d))
        np.testing.assert_allclose(O[live], Ol.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[live], ll.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("g", GEOMS, ids=[g[0] for g in GEOMS])
@pytest.mark.parametrize("kind", KINDS)
def test_rounded_mask_is_a_set_of_physical_pairs(g, kind):
    # Rounded masks (section "Align the sparse mask with final execution") keep
    # whole tiles; the result is attention over the SET of physical pairs they
    # cover.  Q = 0 gives every retained key weight 1, so exp(LSE) is the number
    # of distinct keys of the row, and the map's retained-pair count is the
    # explicit physical matrix's sum.
    name, F, Hs, Ws, wf, ws, BQ, BKV = g
    N = F * Hs * Ws
    _, k, v = rand_head(N, 64, 3)
    q = torch.zeros_like(k)
    gg = geom(F, Hs, Ws, wf, ws, BKV)
    O, lse = oracle.attention(bits(q), bits(k), bits(v), kind, gg, rounding=True, BQ=BQ, BKV=BKV)
    P, pt = rounded_phys_mask(kind, F, Hs, Ws, wf, ws, BQ, BKV)
    Pt = np.zeros_like(P)
    Pt[pt] = P                                   # rows back in (F,H,W) order
    cnt = Pt.sum(1)
    live = cnt > 0
    np.testing.assert_array_equal(np.rint(np.exp(lse[live])).astype(np.int64), cnt[live])
    assert np.all(np.isneginf(lse[~live]))
    mean = (Pt[live].astype(np.float64) @ v.double().numpy()) / cnt[live][:, None]
    np.testing.assert_allclose(O[live], mean, rtol=0, atol=1e-12)
    _, _, st = oracle.tile_map(kind, gg, BQ, BKV, 1)
    assert st["retained_pairs"] == int(P.sum())


def test_rounded_temporal_small_drops_sink_twins():
    # Small's rounded temporal map keeps frame-0 keys both as sink columns and
    # inside kept band tiles; those sink tiles must lose the twin columns (else
    # a key carries double weight), and the kept tiles still cover the same set.
    w = W.SMALL
    gg = geom(w.F, w.Hs, w.Ws, w.wf, w.ws, 128)
    _, _, st = oracle.tile_map(TEMPORAL_PERMUTED, gg, 128, 128, 1)
    assert st["columns"] > 0
    M, col_tok, col_real, pt = layout_mask(TEMPORAL_PERMUTED, w.F, w.Hs, w.Ws, w.wf, w.ws, 128)
    counts, _ = tile_classes(M, col_real, 128, 128, 0)
    real_rows = np.minimum(128, w.N - np.arange(counts.shape[0]) * 128)
    cr = np.zeros(counts.shape[1] * 128, bool)
    cr[: col_real.size] = col_real
    area = np.outer(real_rows, cr.reshape(-1, 128).sum(1))
    kept = (area > 0) & (2 * counts >= area)
    keep = np.repeat(np.repeat(kept, 128, 0), 128, 1)[: w.N, : M.shape[1]] & col_real[None, :]
    multiset = int(keep.sum())
    P, _ = rounded_phys_mask(TEMPORAL_PERMUTED, w.F, w.Hs, w.Ws, w.wf, w.ws, 128, 128)
    assert st["retained_pairs"] == int(P.sum()) < multiset


def test_attention_d128_small_rows_subset():
    w = W.SMALL
    q, k, v = W.qkv(w)
    rows = W.sample_rows(w.N, 40, seed=3)
    for h, kind in ((0, SPATIAL), (1, TEMPORAL_PERMUTED)):
        gg = geom(w.F, w.Hs, w.Ws, w.wf, w.ws, 128)
        O, lse = oracle.attention(bits(q[h]), bits(k[h]), bits(v[h]), kind, gg, rows=rows)
        M = phys_mask(SPATIAL if kind == SPATIAL else TEMPORAL_FHW, w.F, w.Hs, w.Ws, w.wf, w.ws)
        Oref, lref = torch_attention(q[h].double()[rows], k[h].double(), v[h].double(),
                                     torch.from_numpy(M[rows]), 1.0 / np.sqrt(w.d))
        np.testing.assert_allclose(O, Oref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lref.numpy(), rtol=0, atol=1e-12)


def test_all_retained_mask_equals_dense_and_sdpa():
    F, Hs, Ws, d = 5, 7, 9, 64
    S, N = Hs * Ws, 5 * 63
    q, k, v = rand_head(N, d, 9)
    gg = geom(F, Hs, Ws, F - 1, S - 1, 64)
    Od, ld = oracle.attention(bits(q), bits(k), bits(v), DENSE, gg, BQ=64, BKV=64)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double()[None], k.double()[None], v.double()[None])[0]
    np.testing.assert_allclose(Od, ref.numpy(), rtol=0, atol=1e-12)
    for kind in KINDS:
        O, l = oracle.attention(bits(q), bits(k), bits(v), kind, gg, BQ=64, BKV=64)
        np.testing.assert_allclose(O, Od, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, ld, rtol=0, atol=1e-12)


@pytest.mark.parametrize("kind", KINDS)
def test_zero_query_gives_mean_and_log_count(kind):
    # Q = 0: every retained weight is exp(0) = 1, so O = mean of V over the
    # retained keys and lse = ln |R| exactly
    name, F, Hs, Ws, wf, ws, BQ, BKV = GEOMS[1]
    N = F * Hs * Ws
    _, k, v = rand_head(N, 64, 2)
    q = torch.zeros_like(k)
    gg = geom(F, Hs, Ws, wf, ws, BKV)
    O, lse = oracle.attention(bits(q), bits(k), bits(v), kind, gg, BQ=BQ, BKV=BKV)
    M = phys_mask(SPATIAL if kind == SPATIAL else TEMPORAL_FHW, F, Hs, Ws, wf, ws)
    cnt = M.sum(1)
    np.testing.assert_array_equal(np.rint(np.exp(lse)).astype(np.int64), cnt)
    mean = (M.astype(np.float64) @ v.double().numpy()) / cnt[:, None]
    np.testing.assert_allclose(O, mean, rtol=0, atol=1e-12)


def test_poisoned_excluded_keys_do_not_change_output():
    # spatial head of Small: queries of frame 7 keep frames {0, 5, 6, 7}; poisoning
    # K/V of frames 1..4 with large finite values must leave their outputs unchanged
    w = W.SMALL
    q, k, v = (x[0] for x in W.qkv(w))
    S = w.S
    rows = list(range(7 * S, 7 * S + S, 5))
    gg = geom(w.F, w.Hs, w.Ws, w.wf, w.ws, 128)
    O1, l1 = oracle.attention(bits(q), bits(k), bits(v), SPATIAL, gg, rows=rows)
    k2, v2 = k.clone(), v.clone()
    k2[S:5 * S] = 1.0e4
    v2[S:5 * S] = -1.0e4
    O2, l2 = oracle.attention(bits(q), bits(k2), bits(v2), SPATIAL, gg, rows=rows)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)
    # and the poison is visible to a query that does retain those frames
    O3, _ = oracle.attention(bits(q), bits(k2), bits(v2), SPATIAL, gg, rows=[2 * S])
    O4, _ = oracle.attention(bits(q), bits(k), bits(v), SPATIAL, gg, rows=[2 * S])
    assert not np.allclose(O3, O4)


def test_small_tile_stats_regression():
    # regression pin written by tests/golden/make_golden.py (calls only oracle/)
    import json
    with open(os.path.join(HERE, "golden", "small_tile_stats.json")) as fh:
        gold = json.load(fh)
    w = W.SMALL
    gg = geom(w.F, w.Hs, w.Ws, w.wf, w.ws, 128)
    for key, (kind, rounding) in {"spatial_exact": (SPATIAL, 0), "temporal_permuted_exact": (TEMPORAL_PERMUTED, 0),
                                  "temporal_fhw_exact": (TEMPORAL_FHW, 0), "spatial_rounded": (SPATIAL, 1),
                                  "temporal_permuted_rounded": (TEMPORAL_PERMUTED, 1)}.items():
        _, _, st = oracle.tile_map(kind, gg, 128, 128, rounding)
        st.pop("ncols")
        assert st == gold[key], key


# ----------------------------------------------------------------------------
# routing (blog section "Speeding up attention")
# ----------------------------------------------------------------------------
def _structured_heads(F, Hs, Ws, d, seed):
    """Two heads of constructed data: head 0 attends within its own frame (every
    key of frame f points along a frame-specific direction shared by that
    frame's queries), head 1 attends to its own raster position across frames
    (keys at raster s share a direction with queries at s)."""
    g = torch.Generator().manual_seed(seed)
    S, N = Hs * Ws, F * Hs * Ws
    f = torch.arange(N) // S
    s = torch.arange(N) % S
    noise = 0.05
    fdir = torch.randn(F, d, generator=g)
    sdir = torch.randn(S, d, generator=g)
    Q = torch.empty(2, N, d)
    K = torch.empty(2, N, d)
    Q[0] = 3.0 * fdir[f] + noise * torch.randn(N, d, generator=g)
    K[0] = fdir[f] + noise * torch.randn(N, d, generator=g)
    Q[1] = 3.0 * sdir[s] + noise * torch.randn(N, d, generator=g)
    K[1] = sdir[s] + noise * torch.randn(N, d, generator=g)
    V = torch.randn(2, N, d, generator=g)
    return Q.bfloat16(), K.bfloat16(), V.bfloat16()


def test_route_picks_the_mask_that_matches_the_attention_structure():
    F, Hs, Ws, d = 6, 6, 8, 64
    q, k, v = _structured_heads(F, Hs, Ws, d, 3)
    gg = geom(F, Hs, Ws, 1, 2, 64)
    rows = list(range(0, F * Hs * Ws, 7))
    flags, err = oracle.route(bits(q), bits(k), bits(v), gg, rows)
    assert flags.tolist() == [0, 1]
    assert err[0, 0] < err[0, 1] and err[1, 1] < err[1, 0]


def test_route_windows_covering_everything_give_zero_deviation():
    F, Hs, Ws, d = 5, 7, 9, 64
    S, N = Hs * Ws, F * Hs * Ws
    q, k, v = W.qkv(W.SMALL, H=1, N=N, d=d, seed=4)
    rows = [0, 17, N - 1]
    _, err = oracle.route(bits(q), bits(k), bits(v), geom(F, Hs, Ws, 1, S - 1, 64), rows)
    assert err[0, 1] == 0.0 and err[0, 0] > 0.0       # temporal mask = dense
    flags, err = oracle.route(bits(q), bits(k), bits(v), geom(F, Hs, Ws, F - 1, 3, 64), rows)
    assert err[0, 0] == 0.0 and err[0, 1] > 0.0 and flags[0] == 0  # spatial mask = dense
