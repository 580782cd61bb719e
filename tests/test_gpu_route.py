"""GPU per-head routing against the fp64 oracle (deviations and flags)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from test_oracle import _structured_heads


def _run(bss, q, k, v, p, rows):
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in (q, k, v))
    R = torch.tensor(rows, dtype=torch.int32, device=dev)
    flags = torch.empty(q.shape[0], dtype=torch.uint8, device=dev)
    err = torch.empty(q.shape[0], 2, dtype=torch.float32, device=dev)
    bss.route_heads(Q, K, V, p, R, flags, err)
    torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    return flags.cpu().numpy(), err.cpu().numpy()


@pytest.mark.gpu
def test_route_structured_heads(bss):
    F, Hs, Ws, d = 6, 6, 8, 64
    q, k, v = _structured_heads(F, Hs, Ws, d, 3)
    p = bss.MaskParams(F, Hs, Ws, d, 1, 2)
    rows = list(range(0, F * Hs * Ws, 7))
    flags, err = _run(bss, q, k, v, p, rows)
    oflags, oerr = oracle.route(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v),
                                oracle.Geometry(F, Hs, Ws, wf=1, ws=2), rows)
    assert flags.tolist() == oflags.tolist() == [0, 1]
    np.testing.assert_allclose(err, oerr, rtol=2e-3, atol=1e-6)


@pytest.mark.gpu
@pytest.mark.parametrize("wl", [W.SMALL, W.MIXED_75K], ids=lambda w: w.name)
@pytest.mark.parametrize("R", [24, 43, 64])
def test_route_random_heads_match_oracle(bss, wl, R):
    # 24 sampled rows: the three masks' 72 copies fit one 128-row half; 43: 129
    # copies, one past a half, so a two-half item with 127 padding rows; 64 (the
    # benchmark's count): 192 copies in one two-half item
    H = 4
    q, k, v = W.qkv(wl, H=H, seed=11)
    rows = W.sample_rows(wl.N, R, seed=5)
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws)
    flags, err = _run(bss, q, k, v, p, rows)
    oflags, oerr = oracle.route(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v),
                                oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws), rows)
    np.testing.assert_allclose(err, oerr, rtol=5e-3, atol=1e-7)
    clear = np.abs(oerr[:, 0] - oerr[:, 1]) > 1e-2 * np.maximum(oerr[:, 0], oerr[:, 1])
    assert np.array_equal(flags[clear], oflags[clear])


@pytest.mark.gpu
@pytest.mark.parametrize("d", [128, 64])
def test_route_more_rows_than_one_query_tile_and_ragged_geometry(bss, d):
    # 300 sampled rows, 900 copies for the three masks: four 256-row items, the
    # last one ragged; N = 390 is not a multiple of the 128-key tile (padding
    # columns in the last kv tile)
    F, Hs, Ws, wf, ws = 3, 10, 13, 0, 20
    N = F * Hs * Ws
    q, k, v = W.qkv(W.SMALL, H=3, N=N, d=d, seed=31)
    g = torch.Generator().manual_seed(7)
    rows = torch.randint(0, N, (300,), generator=g).tolist()
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws)
    flags, err = _run(bss, q, k, v, p, rows)
    oflags, oerr = oracle.route(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v),
                                oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws), rows)
    np.testing.assert_allclose(err, oerr, rtol=5e-3, atol=1e-7)
    clear = np.abs(oerr[:, 0] - oerr[:, 1]) > 1e-2 * np.maximum(oerr[:, 0], oerr[:, 1])
    assert np.array_equal(flags[clear], oflags[clear])


@pytest.mark.gpu
def test_route_rows_outside_the_sequence_are_skipped_and_recorded(bss):
    wl = W.SMALL
    q, k, v = W.qkv(wl, H=2, seed=12)
    good = W.sample_rows(wl.N, 20, seed=6)
    rows = good[:5] + [-3] + good[5:] + [wl.N + 4]
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws)
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in (q, k, v))
    R = torch.tensor(rows, dtype=torch.int32, device=dev)
    flags = torch.empty(2, dtype=torch.uint8, device=dev)
    err = torch.empty(2, 2, dtype=torch.float32, device=dev)
    bss.route_heads(Q, K, V, p, R, flags, err)
    torch.cuda.synchronize()
    assert bss.status_string(bss.get_device_status()) == "BSS_ERR_INVALID_ARG"
    assert bss.get_device_status() == 0  # reading clears the word
    _, oerr = oracle.route(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v),
                           oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws), good)
    np.testing.assert_allclose(err.cpu().numpy(), oerr, rtol=5e-3, atol=1e-7)
