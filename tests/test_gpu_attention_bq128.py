"""Attention on 128-row query tiles (one MMA half per CTA, S double-buffered in
tensor memory) against the fp64 oracle; for exact masks it must equal the
256-row kernel bit for bit (each row sees its retained keys in the same order;
the extra tiles of a 256-row tile are fully masked for it and add exact zeros)."""
import numpy as np
import pytest
import torch

import oracle
from _util import compare, oracle_kind, oracle_rows, run_gpu
from test_gpu_attention import SMALL_CASES, _inputs


@pytest.mark.gpu
@pytest.mark.parametrize("case", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
@pytest.mark.parametrize("rounding", [0, 1, 2])
@pytest.mark.parametrize("tperm", [1, 0])
def test_bq128_matches_oracle_and_bq256(bss, case, rounding, tperm):
    name, F, Hs, Ws, d, wf, ws, flags = case
    N = F * Hs * Ws
    q, k, v = _inputs(len(flags), N, d, seed=len(name) + 40)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=rounding)
    out, lse, _ = run_gpu(bss, q, k, v, flags, p, BQ=128)
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=128)
    for h, fl in enumerate(flags):
        Oref, lref = oracle_rows(q, k, v, h, oracle_kind(fl, tperm), g, None, rounding == 1, BQ=128)
        compare(out[h].numpy(), lse[h].numpy(), Oref, lref, f"BQ=128 {name} head {h} rounding {rounding}")
    if rounding != 1:
        out2, lse2, _ = run_gpu(bss, q, k, v, flags, p, BQ=256)
        assert torch.equal(out.view(torch.int32), out2.view(torch.int32)), f"{name}: O differs from BQ=256"
        assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32)), f"{name}: LSE differs from BQ=256"


@pytest.mark.gpu
@pytest.mark.parametrize("tperm", [1, 0])
def test_bq128_rescales_after_the_first_tile(bss, tperm):
    # keys grow along the sequence, so each row's maximum keeps growing past the
    # lazy-rescale threshold on later tiles, at different tiles for different
    # rows and warps (the warps of a 128-row CTA then run tiles apart)
    F, Hs, Ws, d, wf, ws, flags = 8, 16, 24, 128, 2, 40, [0, 1]
    N = F * Hs * Ws
    q, k, v = _inputs(2, N, d, seed=91)
    ramp = (1.0 + 7.0 * torch.arange(N, dtype=torch.float32) / N).view(1, N, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=tperm, rounding=0)
    out, lse, _ = run_gpu(bss, q, k, v, flags, p, BQ=128)
    out2, lse2, _ = run_gpu(bss, q, k, v, flags, p, BQ=256)
    assert torch.equal(out.view(torch.int32), out2.view(torch.int32))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    # |O| reaches ~4 here, so the absolute bar scales with it: bf16 output
    # rounding alone is up to |O| * 2^-8; relative L2 and LSE keep their bars
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=128)
    for h, fl in enumerate(flags):
        Oref, lref = oracle_rows(q, k, v, h, oracle_kind(fl, tperm), g, None, False, BQ=128)
        o = out[h].numpy().astype(np.float64)
        assert np.all(np.abs(o - Oref) <= 2.0 ** -8 * np.abs(Oref) + 1e-2), f"head {h}"
        assert np.linalg.norm(o - Oref) / np.linalg.norm(Oref) <= 1e-2
        assert np.abs(lse[h].numpy() - lref).max() <= 1e-3
