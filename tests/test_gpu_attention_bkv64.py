"""Attention on 64-key tiles (the tile-shape comparison's BKV axis) against the
fp64 oracle: all rows of the small geometries, every traversal mode and both
layouts of the temporal mask, at both query-tile heights; a rounded mask is
rounded on the 64-key grid."""
import pytest
import torch

import oracle
import workloads as W
from _util import compare, oracle_kind, oracle_rows, run_gpu
from test_gpu_attention import SMALL_CASES


@pytest.mark.gpu
@pytest.mark.parametrize("case", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
@pytest.mark.parametrize("rounding", [0, 1, 2])
@pytest.mark.parametrize("tperm", [1, 0])
@pytest.mark.parametrize("BQ", [256, 128])
def test_bkv64_matches_oracle(bss, case, rounding, tperm, BQ):
    name, F, Hs, Ws, d, wf, ws, flags = case
    N = F * Hs * Ws
    q, k, v = W.qkv(W.SMALL, H=len(flags), N=N, d=d, seed=len(name) + 3)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=rounding)
    out, lse, _ = run_gpu(bss, q, k, v, flags, p, BQ=BQ, BKV=64)
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=64)
    for h, fl in enumerate(flags):
        Oref, lref = oracle_rows(q, k, v, h, oracle_kind(fl, tperm), g, None, rounding == 1, BQ=BQ, BKV=64)
        compare(out[h].numpy(), lse[h].numpy(), Oref, lref, f"{name} head {h} rounding {rounding} BQ {BQ} BKV 64")


@pytest.mark.gpu
def test_bkv64_rescales_after_the_first_tile(bss):
    # keys growing along the sequence force O rescales on later tiles
    F, Hs, Ws, d, wf, ws, flags = 8, 16, 24, 128, 2, 40, [1, 0]
    N = F * Hs * Ws
    q, k, v = W.qkv(W.SMALL, H=2, N=N, d=d, seed=93)
    ramp = (1.0 + 7.0 * torch.arange(N, dtype=torch.float32) / N).view(1, N, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=1, rounding=0)
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=64)
    for BQ in (256, 128):
        out, lse, _ = run_gpu(bss, q, k, v, flags, p, BQ=BQ, BKV=64)
        for h, fl in enumerate(flags):
            Oref, lref = oracle_rows(q, k, v, h, oracle_kind(fl, 1), g, None, False, BQ=BQ, BKV=64)
            tol = 2.0 ** -8 * abs(Oref).max() + 1e-2
            assert abs(out[h].numpy() - Oref).max() <= tol
            assert abs(lse[h].numpy() - lref).max() <= 1e-3


@pytest.mark.gpu
def test_bkv64_full_size_mixed_sampled(bss):
    wl = W.MIXED_75K
    dev = torch.device("cuda")
    Q, K, V = W.qkv_device(wl, dev)
    flags = wl.head_flags()
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=1, rounding=0)
    O = torch.empty_like(Q)
    lse = torch.empty(wl.H, wl.N, device=dev)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    ws_ = [torch.empty_like(Q) for _ in range(3)]
    with bss.build_tile_map(p, 256, 64) as tm:
        bss.attention_step(Q, K, V, O, tm, fl, *ws_, lse=lse)
        torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    g = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws, bkv=64)
    rows = W.sample_rows(wl.N, 12, seed=wl.index + 60)
    for h in (flags.index(1), flags.index(0)):
        qh, kh, vh = (x[h].cpu() for x in (Q, K, V))
        Oref, lref = oracle.attention(W.bf16_bits(qh), W.bf16_bits(kh), W.bf16_bits(vh), oracle_kind(flags[h], 1), g,
                                      rows=rows, BQ=256, BKV=64)
        lrow = lse[h].cpu()
        if flags[h]:
            lrow = lrow[[(r % wl.S) * wl.F + r // wl.S for r in rows]]
        else:
            lrow = lrow[rows]
        compare(O[h, rows].float().cpu().numpy(), lrow.numpy(), Oref, lref, f"bkv64 mixed head {h}")


@pytest.mark.gpu
def test_fused_permutation_refuses_a_64_key_map(bss):
    # the 4-row gathers of the fused permutation fill 128-key tiles only: a map
    # with 64-key tiles is refused on the host, before any launch, and the
    # output is left untouched
    wl = W.SMALL
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in W.qkv(wl))
    O = torch.full_like(Q, 7.0)
    fl = torch.tensor(wl.head_flags(), dtype=torch.uint8, device=dev)
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=1, rounding=0)
    with bss.build_tile_map(p, BKV=64) as tm:
        with pytest.raises(bss.BssError) as err:
            bss.sparse_attention_fused(Q, K, V, O, tm, fl)
    assert err.value.status == 2  # BSS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    assert bool((O == 7.0).all())
