"""GPU block-sparse attention against the fp64 oracle.

Bar (floating point): max |dO| <= 1e-2, mean |dO| <= 1e-3, rel-L2 <= 1e-2 and
|dLSE| <= 1e-3 on N(0,1) inputs; the coverage (Q = 0) and poison tests pin
which keys each row sees exactly."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import compare, oracle_kind, oracle_rows, run_gpu

SMALL_CASES = [  # name, F, Hs, Ws, d, wf, ws, flags
    ("tiny", 4, 8, 8, 64, 1, 10, [0]),
    ("small", 8, 16, 24, 128, 2, 40, [0, 1]),
    ("ragged_s63_d64", 5, 7, 9, 64, 1, 5, [1, 0]),
    ("ragged_s130_d128", 3, 10, 13, 128, 0, 20, [1, 1, 0]),
    ("ragged_s130_d64", 3, 10, 13, 64, 1, 200, [0, 1]),
    # degenerate geometries: one token, one frame, one raster position, fewer
    # tokens than a tile, zero-width windows (a row keeps its own frame / raster
    # position and frame 0)
    ("one_token", 1, 1, 1, 64, 0, 0, [0, 1]),
    ("one_frame_s300", 1, 12, 25, 128, 0, 3, [1, 0]),
    ("one_position_f130", 130, 1, 1, 128, 2, 0, [1, 0]),
    ("n100_below_a_tile", 4, 5, 5, 128, 1, 2, [1, 0]),
    ("windows_zero", 3, 10, 13, 128, 0, 0, [1, 0]),
]


def _inputs(H, N, d, seed):
    w = W.SMALL
    return W.qkv(w, H=H, N=N, d=d, seed=seed)


@pytest.mark.gpu
@pytest.mark.parametrize("case", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
@pytest.mark.parametrize("rounding", [0, 1, 2])
@pytest.mark.parametrize("tperm", [1, 0])
def test_attention_matches_oracle_all_rows(bss, case, rounding, tperm):
    name, F, Hs, Ws, d, wf, ws, flags = case
    N = F * Hs * Ws
    q, k, v = _inputs(len(flags), N, d, seed=len(name))
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=rounding)
    out, lse, stats = run_gpu(bss, q, k, v, flags, p)
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=128)
    for h, fl in enumerate(flags):
        kind = oracle_kind(fl, tperm)
        Oref, lref = oracle_rows(q, k, v, h, kind, g, None, rounding == 1)
        compare(out[h].numpy(), lse[h].numpy(), Oref, lref, f"{name} head {h} kind {kind} rounding {rounding}")


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(2, 3072, 128), (1, 315, 64), (3, 390, 128), (1, 130, 64)])
def test_dense_matches_oracle(bss, shape):
    H, N, d = shape
    q, k, v = _inputs(H, N, d, seed=N)
    out, lse, _ = run_gpu(bss, q, k, v, [0] * H, None, dense=True)
    g = oracle.Geometry(1, 1, N)
    for h in range(H):
        Oref, lref = oracle.attention(W.bf16_bits(q[h]), W.bf16_bits(k[h]), W.bf16_bits(v[h]), oracle.DENSE, g)
        compare(out[h].numpy(), lse[h].numpy(), Oref, lref, f"dense {shape} head {h}")


def _row_counts(kind, F, S, wf, ws):
    t = np.arange(F * S)
    f, s = t // S, t % S
    if kind == oracle.SPATIAL:
        return S * (np.minimum(f + wf, F - 1) - np.maximum(f - wf, 0) + 1 + (f > wf))
    b = np.minimum(s + ws, S - 1) - np.maximum(s - ws, 0) + 1
    return F * b + (S - b)


@pytest.mark.gpu
@pytest.mark.parametrize("tperm", [1, 0])
def test_zero_query_coverage_is_exact(bss, tperm):
    # Q = 0: every retained key has weight 1, so exp(LSE) = |R_i| exactly and
    # O = mean of V over R_i -- this pins the set of keys each row sees.
    F, Hs, Ws, d, wf, ws = 8, 16, 24, 128, 2, 40
    S, N = Hs * Ws, F * Hs * Ws
    flags = [0, 1]
    q, k, v = _inputs(2, N, d, seed=77)
    q = torch.zeros_like(q)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=0)
    out, lse, _ = run_gpu(bss, q, k, v, flags, p)
    for h, fl in enumerate(flags):
        kind = oracle.SPATIAL if fl == 0 else oracle.TEMPORAL_FHW
        cnt = _row_counts(kind, F, S, wf, ws)
        got = np.rint(np.exp(lse[h].numpy().astype(np.float64))).astype(np.int64)
        assert np.array_equal(got, cnt), f"head {h}: {np.nonzero(got != cnt)[0][:10]}"


@pytest.mark.gpu
@pytest.mark.parametrize("tperm", [1, 0])
def test_poisoned_excluded_keys_leave_output_bit_identical(bss, tperm):
    F, Hs, Ws, d, wf, ws = 8, 16, 24, 128, 2, 40
    S, N = Hs * Ws, F * Hs * Ws
    flags = [0, 1]
    q, k, v = _inputs(2, N, d, seed=78)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=0)
    out1, lse1, _ = run_gpu(bss, q, k, v, flags, p)
    k2, v2 = k.clone(), v.clone()
    # spatial head 0: frames 1..4 are excluded for queries of frame 7
    k2[0, S:5 * S] = 1.0e4
    v2[0, S:5 * S] = -1.0e4
    # temporal head 1: raster >= 200 of frames >= 1 is excluded for queries with raster <= 40
    t = torch.arange(N)
    far = ((t % S) >= 200) & ((t // S) >= 1)
    k2[1, far] = -1.0e4
    v2[1, far] = 1.0e4
    out2, lse2, _ = run_gpu(bss, q, k2, v2, flags, p)
    rows0 = torch.arange(7 * S, 8 * S)
    rows1 = torch.nonzero((t % S) <= 40).flatten()
    assert torch.equal(out1[0, rows0], out2[0, rows0])
    assert torch.equal(lse1[0, rows0], lse2[0, rows0])
    assert torch.equal(out1[1, rows1], out2[1, rows1])
    assert torch.equal(lse1[1, rows1], lse2[1, rows1])
    assert not torch.equal(out1[0, :S], out2[0, :S])  # frame-0 queries do see frames 1..2


@pytest.mark.gpu
@pytest.mark.parametrize("path", ["step", "bq128", "fused"])
def test_rounded_mask_with_empty_q_tiles_gives_zero_rows(bss, path):
    # One raster position, 130 frames: a spatial row keeps 6 keys, so the rounded
    # mask drops every tile of the spatial heads at BQ = 256 and all but the
    # 2 x 2 tile of the last two frames at BQ = 128; rows of a q tile with an
    # empty list get O = 0, LSE = -inf.  The temporal head keeps every frame.
    # Q is large, so a Q row leaking into the output (the zero rows are staged
    # in Q's shared-memory buffer) would show; the launch is repeated because
    # such a leak depends on timing.
    F, Hs, Ws, d, wf, ws = 130, 1, 1, 128, 2, 0
    N = F
    flags = [0, 1, 0]
    q, k, v = _inputs(3, N, d, seed=81)
    q[0] = 100.0
    q[2] = -60.0
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=1, rounding=1)
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=128)
    BQ = 128 if path == "bq128" else bss.ATTN_BQ
    ref = {h: oracle_rows(q, k, v, h, oracle_kind(flags[h], 1), g, None, True, BQ=BQ) for h in range(3)}
    empty = {h: np.isneginf(ref[h][1]) for h in (0, 2)}
    assert all(e[:128].all() for e in empty.values())  # the first q tile has an empty list
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in (q, k, v))
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    ws_ = [torch.empty_like(Q) for _ in range(3)]
    with bss.build_tile_map(p, BQ=BQ) as tm:
        for it in range(10):
            O = torch.full_like(Q, 3.0)
            lse = torch.zeros(3, N, device=dev)
            if path == "fused":
                bss.sparse_attention_fused(Q, K, V, O, tm, fl, lse=lse)
            else:
                bss.attention_step(Q, K, V, O, tm, fl, *ws_, lse=lse)
            torch.cuda.synchronize()
            assert bss.get_device_status() == 0
            for h in (0, 2):
                e = torch.from_numpy(empty[h])
                assert torch.count_nonzero(O[h].cpu()[e]).item() == 0, f"launch {it} head {h}: O is not zero"
                assert torch.all(torch.isneginf(lse[h].cpu()[e])), f"launch {it} head {h}: LSE is not -inf"
    for h in range(3):
        lrow = lse[h].cpu()  # one raster position: the permutation is the identity
        compare(O[h].float().cpu().numpy(), lrow.numpy(), ref[h][0], ref[h][1], f"{path} head {h}")


def _full_size(bss, wl, tperm, rounding, heads, nrows, tile_stride=1):
    dev = torch.device("cuda")
    Q, K, V = W.qkv_device(wl, dev)
    flags = wl.head_flags()
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=tperm, rounding=rounding)
    O = torch.empty_like(Q)
    lse = torch.empty(wl.H, wl.N, device=dev)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    ws_ = [torch.empty_like(Q) for _ in range(3)]
    with bss.build_tile_map(p) as tm:
        bss.attention_step(Q, K, V, O, tm, fl, *ws_, lse=lse)
        torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    g = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws, bkv=128)
    sampled = W.sample_rows(wl.N, nrows, seed=wl.index)
    # plus one row of every tile_stride-th q tile of the head's layout (the
    # oracle classifies the q tile of every row of a rounded mask)
    BQ = bss.ATTN_BQ
    nq = -(-wl.N // BQ)
    tiles = np.unique(np.append(np.arange(0, nq, tile_stride), nq - 1))
    off = np.random.default_rng(wl.index).integers(0, BQ, tiles.size)
    lay = np.minimum(tiles * BQ + off, wl.N - 1)
    for h in heads:
        kind = oracle_kind(flags[h], tperm)
        per_tile = lay
        if flags[h] and tperm:   # layout row p = s*F + f is token f*S + s
            per_tile = (lay % wl.F) * wl.S + lay // wl.F
        rows = sorted(set(sampled) | set(int(r) for r in per_tile))
        qh, kh, vh = (x[h].cpu() for x in (Q, K, V))
        Oref, lref = oracle.attention(W.bf16_bits(qh), W.bf16_bits(kh), W.bf16_bits(vh), kind, g, rows=rows,
                                      rounding=bool(rounding), BQ=bss.ATTN_BQ, BKV=bss.ATTN_BKV)
        lrow = lse[h].cpu()
        if flags[h] and tperm:
            lrow = lrow[[(r % wl.S) * wl.F + r // wl.S for r in rows]]
        else:
            lrow = lrow[rows]
        compare(O[h, rows].float().cpu().numpy(), lrow.numpy(), Oref, lref,
                f"{wl.name} head {h} kind {kind} rounding {rounding}")


@pytest.mark.gpu
@pytest.mark.parametrize("rounding", [0, 1])
def test_full_size_spatial_75k_sampled(bss, rounding):
    _full_size(bss, W.SPATIAL_75K, 1, rounding, heads=[0, 4, 9], nrows=24)


@pytest.mark.gpu
@pytest.mark.parametrize("tperm", [1, 0])
def test_full_size_mixed_75k_sampled(bss, tperm):
    wl = W.MIXED_75K
    fl = wl.head_flags()
    heads = [fl.index(0), fl.index(1), len(fl) - 1 - fl[::-1].index(1)]
    _full_size(bss, wl, tperm, 0, heads=heads, nrows=24)


@pytest.mark.gpu
def test_full_size_1440p_302k_rounded_sampled(bss):
    wl = W.P1440_302K
    fl = wl.head_flags()
    _full_size(bss, wl, 1, 1, heads=[fl.index(0), fl.index(1)], nrows=12, tile_stride=16)


@pytest.mark.gpu
def test_full_size_1440p_dense_control_sampled(bss):
    # the dense control at the size the benchmark times it: 10 heads x 302,400
    # tokens, 2,363 kv tiles per row with a ragged last one
    wl = W.P1440_302K
    dev = torch.device("cuda")
    Q, K, V = W.qkv_device(wl, dev)
    O = torch.empty_like(Q)
    lse = torch.empty(wl.H, wl.N, device=dev)
    bss.dense_attention(Q, K, V, O, lse=lse)
    torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    g = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws, bkv=128)
    rows = W.sample_rows(wl.N, 12, seed=wl.index + 1)
    for h in (0, wl.H - 1):
        qh, kh, vh = (x[h].cpu() for x in (Q, K, V))
        Oref, lref = oracle.attention(W.bf16_bits(qh), W.bf16_bits(kh), W.bf16_bits(vh), oracle.DENSE, g, rows=rows)
        compare(O[h, rows].float().cpu().numpy(), lse[h, rows].cpu().numpy(), Oref, lref,
                f"{wl.name} dense head {h}")


@pytest.mark.gpu
@pytest.mark.parametrize("geom", [(8, 16, 24, 128), (3, 10, 13, 64), (5, 7, 9, 128)], ids=["small", "ragged_d64", "ragged_d128"])
def test_all_covering_windows_equal_dense_bit_for_bit(bss, geom):
    # spatial with wf >= F-1 and the (F,H,W) temporal mask with ws >= S-1 retain
    # every pair, visit every kv tile in ascending order and mask only the
    # padding columns: the same arithmetic as the dense control
    F, Hs, Ws, d = geom
    S, N = Hs * Ws, F * Hs * Ws
    q, k, v = _inputs(2, N, d, seed=N + 3)
    dense, dlse, _ = run_gpu(bss, q, k, v, [0, 0], None, dense=True)
    p = bss.MaskParams(F, Hs, Ws, d, F - 1, S - 1, temporal_permuted=0, rounding=0)
    out, lse, _ = run_gpu(bss, q, k, v, [0, 1], p)
    assert torch.equal(out.view(torch.int32), dense.view(torch.int32))
    assert torch.equal(lse.view(torch.int32), dlse.view(torch.int32))


@pytest.mark.gpu
@pytest.mark.parametrize("wl_name", ["small_3072tok_2h_d128", "mixed_75600tok_10h_d128"])
def test_split_step_equals_full_permutation_step(bss, wl_name):
    # temporal heads permuted alone + split attention == every head permuted (spatial
    # heads copied) + one-buffer attention, bit for bit, O and LSE
    import workloads as W
    wl = W.BY_NAME[wl_name]
    dev = torch.device("cuda")
    Q, K, V = W.qkv_device(wl, dev)
    H = Q.shape[0]
    flags = wl.head_flags()
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=1, rounding=0)
    O1, O2 = torch.empty_like(Q), torch.empty_like(Q)
    l1 = torch.empty(H, wl.N, device=dev)
    l2 = torch.empty(H, wl.N, device=dev)
    ws = [torch.empty_like(Q) for _ in range(3)]
    with bss.build_tile_map(p) as tm:
        bss.attention_step(Q, K, V, O1, tm, fl, *ws, lse=l1)
        Qp, Kp, Vp, Op = (torch.empty_like(Q) for _ in range(4))
        bss.permute(Q, Qp, fl, p, False)
        bss.permute(K, Kp, fl, p, False)
        bss.permute(V, Vp, fl, p, False)
        bss.sparse_attention(Qp, Kp, Vp, Op, tm, fl, lse=l2)
        bss.permute(Op, O2, fl, p, True)
        # the split call with an explicit Ot, then the inverse permute of Ot (the
        # step stores the temporal heads' rows in (F,H,W) order itself, Ot = None)
        O3, Ot = torch.empty_like(Q), torch.empty_like(Q)
        l3 = torch.empty(H, wl.N, device=dev)
        bss.permute(Q, Qp, fl, p, False, only_flagged=True)
        bss.permute(K, Kp, fl, p, False, only_flagged=True)
        bss.permute(V, Vp, fl, p, False, only_flagged=True)
        bss.sparse_attention_split(Q, K, V, O3, Qp, Kp, Vp, Ot, tm, fl, lse=l3)
        bss.permute(Ot, O3, fl, p, True, only_flagged=True)
        torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    assert torch.equal(O3.view(torch.int16), O1.view(torch.int16))
    assert torch.equal(l3.view(torch.int32), l1.view(torch.int32))
