"""Attention with the token permutation fused into the kernel.

bss_sparse_attention_fused reads every head in (F,H,W) order and applies a
temporal head's (H,W,F) permutation in its loads and stores.  The tile map,
masks and arithmetic are those of the explicit path (permute -> attention ->
unpermute), so the outputs must be bit-identical to it; they are also compared
with the fp64 oracle directly."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import compare, oracle_kind, oracle_rows, run_gpu

CASES = [  # name, F, Hs, Ws, d, wf, ws, flags
    ("small", 8, 16, 24, 128, 2, 40, [0, 1]),
    ("ragged_s63_d64", 5, 7, 9, 64, 1, 5, [1, 0]),
    ("ragged_s130_d128", 3, 10, 13, 128, 0, 20, [1, 1, 0]),
    ("ragged_s130_d64", 3, 10, 13, 64, 1, 200, [0, 1]),
    ("frames1", 1, 20, 30, 128, 0, 7, [1, 0]),
    ("s1_frames300", 300, 1, 1, 128, 5, 0, [1, 0, 1]),
]


def run_fused(bss, q, k, v, flags, params):
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in (q, k, v))
    H, N, _ = Q.shape
    O = torch.empty_like(Q)
    lse = torch.empty(H, N, dtype=torch.float32, device=dev)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    with bss.build_tile_map(params) as tm:
        bss.sparse_attention_fused(Q, K, V, O, tm, fl, lse=lse)
        torch.cuda.synchronize()
    st = bss.get_device_status()
    assert st == 0, bss.status_string(st)
    return O.float().cpu(), lse.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("rounding", [0, 1, 2])
def test_fused_bit_identical_to_explicit_and_matches_oracle(bss, case, rounding):
    name, F, Hs, Ws, d, wf, ws, flags = case
    N = F * Hs * Ws
    q, k, v = W.qkv(W.SMALL, H=len(flags), N=N, d=d, seed=100 + len(name))
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=1, rounding=rounding)
    o_ref, lse_ref, _ = run_gpu(bss, q, k, v, flags, p)
    o_f, lse_f = run_fused(bss, q, k, v, flags, p)
    assert torch.equal(o_f.view(torch.int32), o_ref.view(torch.int32)), f"{name}: O differs from the explicit path"
    assert torch.equal(lse_f.view(torch.int32), lse_ref.view(torch.int32)), f"{name}: LSE differs"
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=128)
    for h, fl in enumerate(flags):
        Oref, lref = oracle_rows(q, k, v, h, oracle_kind(fl, 1), g, None, rounding == 1)
        compare(o_f[h].numpy(), lse_f[h].numpy(), Oref, lref, f"fused {name} head {h} rounding {rounding}")


@pytest.mark.gpu
def test_fused_bit_identical_with_rescales_after_the_first_tile(bss):
    # keys growing along the sequence force O rescales on later tiles
    F, Hs, Ws, d, wf, ws, flags = 8, 16, 24, 128, 2, 40, [1, 0]
    N = F * Hs * Ws
    q, k, v = W.qkv(W.SMALL, H=2, N=N, d=d, seed=92)
    ramp = (1.0 + 7.0 * torch.arange(N, dtype=torch.float32) / N).view(1, N, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=1, rounding=0)
    o_ref, lse_ref, _ = run_gpu(bss, q, k, v, flags, p)
    o_f, lse_f = run_fused(bss, q, k, v, flags, p)
    assert torch.equal(o_f.view(torch.int32), o_ref.view(torch.int32))
    assert torch.equal(lse_f.view(torch.int32), lse_ref.view(torch.int32))


@pytest.mark.gpu
def test_fused_zero_query_coverage_is_exact(bss):
    # Q = 0: exp(LSE) counts the keys each row sees (frame-0 sink + raster band)
    F, Hs, Ws, d, wf, ws = 8, 16, 24, 128, 2, 40
    S, N = Hs * Ws, F * Hs * Ws
    q, k, v = W.qkv(W.SMALL, H=2, N=N, d=d, seed=79)
    q = torch.zeros_like(q)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, temporal_permuted=1, rounding=0)
    _, lse = run_fused(bss, q, k, v, [1, 1], p)
    s = np.arange(N) % S
    b = np.minimum(s + ws, S - 1) - np.maximum(s - ws, 0) + 1
    cnt = F * b + (S - b)
    for h in range(2):
        got = np.rint(np.exp(lse[h].numpy().astype(np.float64))).astype(np.int64)
        assert np.array_equal(got, cnt), f"head {h}: {np.nonzero(got != cnt)[0][:10]}"


def _full_size_equal(bss, wl, rounding, nrows, heads_checked):
    dev = torch.device("cuda")
    Q, K, V = W.qkv_device(wl, dev)
    flags = wl.head_flags()
    p = bss.MaskParams(wl.F, wl.Hs, wl.Ws, wl.d, wl.wf, wl.ws, temporal_permuted=1, rounding=rounding)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    O1, O2 = torch.empty_like(Q), torch.empty_like(Q)
    l1 = torch.empty(wl.H, wl.N, device=dev)
    l2 = torch.empty(wl.H, wl.N, device=dev)
    ws_ = [torch.empty_like(Q) for _ in range(3)]
    with bss.build_tile_map(p) as tm:
        bss.attention_step(Q, K, V, O1, tm, fl, *ws_, lse=l1)
        bss.sparse_attention_fused(Q, K, V, O2, tm, fl, lse=l2)
        torch.cuda.synchronize()
    del ws_
    assert bss.get_device_status() == 0
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    # the explicit path's LSE is in layout order; bring temporal heads back to (F,H,W)
    t = torch.arange(wl.N, device=dev)
    pos = (t % wl.S) * wl.F + t // wl.S
    for h in range(wl.H):
        ref = l1[h][pos] if flags[h] else l1[h]
        assert torch.equal(ref.view(torch.int32), l2[h].view(torch.int32)), f"head {h}: LSE differs"
    g = oracle.Geometry(wl.F, wl.Hs, wl.Ws, wf=wl.wf, ws=wl.ws, bkv=128)
    rows = W.sample_rows(wl.N, nrows, seed=wl.index + 50)
    for h in heads_checked:
        qh, kh, vh = (x[h].cpu() for x in (Q, K, V))
        Oref, lref = oracle.attention(W.bf16_bits(qh), W.bf16_bits(kh), W.bf16_bits(vh), oracle_kind(flags[h], 1), g,
                                      rows=rows, rounding=bool(rounding), BQ=bss.ATTN_BQ, BKV=bss.ATTN_BKV)
        compare(O2[h, rows].float().cpu().numpy(), l2[h, rows].cpu().numpy(), Oref, lref,
                f"fused {wl.name} head {h}")


@pytest.mark.gpu
def test_fused_full_size_mixed_75k(bss):
    wl = W.MIXED_75K
    fl = wl.head_flags()
    _full_size_equal(bss, wl, 0, 16, [fl.index(1), fl.index(0)])


@pytest.mark.gpu
def test_fused_full_size_1440p_302k_rounded(bss):
    wl = W.P1440_302K
    _full_size_equal(bss, wl, 1, 8, [wl.head_flags().index(1)])
