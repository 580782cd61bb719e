"""Seeded random small geometries: the tile map bit for bit and the attention
step (all rows, both layouts of the temporal mask, all three traversal modes,
both query-tile heights) against the fp64 oracle; the fused permutation against
the step bit for bit; routing against the oracle's routing.  The geometries are
drawn from a fixed seed, so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import compare, oracle_kind, oracle_rows, run_gpu
from test_gpu_tilemap import check_map


def _cases(count=48, seed=2026):
    g = torch.Generator().manual_seed(seed)

    def r(lo, hi):  # inclusive
        return int(torch.randint(lo, hi + 1, (1,), generator=g))

    out = []
    for i in range(count):
        F, Hs, Ws = r(1, 9), r(1, 14), r(1, 17)
        while F * Hs * Ws > 3000:
            F = max(1, F - 1)
            Hs = max(1, Hs - 1)
        S = Hs * Ws
        wf, ws = r(0, F), r(0, S)
        d = 64 if r(0, 1) == 0 else 128
        H = r(1, 3)
        flags = [r(0, 1) for _ in range(H)]
        out.append((f"c{i:02d}_F{F}_H{Hs}_W{Ws}_wf{wf}_ws{ws}_d{d}", F, Hs, Ws, wf, ws, d, flags,
                    r(0, 2), r(0, 1), 128 if r(0, 1) else 256))
    return out


CASES = _cases()


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_random_geometry_matches_oracle(bss, case):
    name, F, Hs, Ws, wf, ws, d, flags, rounding, tperm, BQ = case
    N = F * Hs * Ws
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=rounding)
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=128)
    with bss.build_tile_map(p, BQ, 128) as tm:
        check_map(bss, tm, oracle.SPATIAL, g, BQ, 128, rounding)
        check_map(bss, tm, oracle.TEMPORAL_PERMUTED if tperm else oracle.TEMPORAL_FHW, g, BQ, 128, rounding)
    q, k, v = W.qkv(W.SMALL, H=len(flags), N=N, d=d, seed=len(name) + N)
    out, lse, _ = run_gpu(bss, q, k, v, flags, p, BQ=BQ)
    for h, fl in enumerate(flags):
        Oref, lref = oracle_rows(q, k, v, h, oracle_kind(fl, tperm), g, None, rounding == 1, BQ=BQ)
        compare(out[h].numpy(), lse[h].numpy(), Oref, lref, f"{name} head {h} rounding {rounding} BQ {BQ}")


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_random_geometry_fused_equals_step(bss, case):
    # the permutation applied by the kernel's loads and stores gives the same bits
    # as the permute -> attention step (LSE compared in (F,H,W) order)
    name, F, Hs, Ws, wf, ws, d, flags, rounding, tperm, BQ = case
    N = F * Hs * Ws
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=rounding)
    q, k, v = W.qkv(W.SMALL, H=len(flags), N=N, d=d, seed=len(name) + N)
    out, lse, _ = run_gpu(bss, q, k, v, flags, p, BQ=BQ)
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in (q, k, v))
    O = torch.empty_like(Q)
    L = torch.empty(len(flags), N, dtype=torch.float32, device=dev)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    with bss.build_tile_map(p, BQ, 128) as tm:
        bss.sparse_attention_fused(Q, K, V, O, tm, fl, lse=L)
        torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    assert torch.equal(O.float().cpu().view(torch.int32), out.view(torch.int32)), name
    assert torch.equal(L.cpu().view(torch.int32), lse.view(torch.int32)), name


ROUTE_CASES = CASES[:16]


@pytest.mark.gpu
@pytest.mark.parametrize("case", ROUTE_CASES, ids=[c[0] for c in ROUTE_CASES])
def test_random_geometry_routing_matches_oracle(bss, case):
    name, F, Hs, Ws, wf, ws, d, flags, _, _, _ = case
    N = F * Hs * Ws
    H = len(flags)
    g = torch.Generator().manual_seed(N + H)
    R = int(torch.randint(1, 301, (1,), generator=g))
    rows = torch.randint(0, N, (R,), generator=g).tolist()
    q, k, v = W.qkv(W.SMALL, H=H, N=N, d=d, seed=len(name) + 7)
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in (q, k, v))
    fl = torch.empty(H, dtype=torch.uint8, device=dev)
    err = torch.empty(H, 2, dtype=torch.float32, device=dev)
    bss.route_heads(Q, K, V, bss.MaskParams(F, Hs, Ws, d, wf, ws), torch.tensor(rows, dtype=torch.int32, device=dev),
                    fl, err)
    torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    oflags, oerr = oracle.route(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v),
                                oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws), rows)
    e = err.cpu().numpy()
    np.testing.assert_allclose(e, oerr, rtol=5e-3, atol=1e-6)
    clear = np.abs(oerr[:, 0] - oerr[:, 1]) > 1e-2 * np.maximum(oerr[:, 0], oerr[:, 1])
    assert np.array_equal(fl.cpu().numpy()[clear], oflags[clear])
