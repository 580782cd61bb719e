"""GPU flag-driven permutation against the oracle's scalar permutation (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

CASES = [  # F, Hs, Ws, d, flags
    (8, 16, 24, 128, [0, 1]),
    (5, 7, 9, 64, [1, 0, 1]),
    (3, 10, 13, 128, [1, 1]),
    (1, 1, 1, 64, [1, 0]),      # one token
    (1, 12, 25, 128, [1]),      # one frame: the permutation is the identity
    (130, 1, 1, 128, [0, 1]),   # one raster position: the identity too
    (4, 5, 5, 64, [1]),         # fewer rows than one thread block covers
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_permute_bit_exact(bss, case):
    F, Hs, Ws, d, flags = case
    S = Hs * Ws
    N = F * S
    x = torch.randint(-32768, 32767, (len(flags), N, d), dtype=torch.int16,
                      generator=torch.Generator().manual_seed(3))
    xb = x.view(torch.bfloat16)
    p = bss.MaskParams(F, Hs, Ws, d, 1, 1)
    dev = torch.device("cuda")
    X = xb.to(dev)
    Y = torch.empty_like(X)
    Z = torch.empty_like(X)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    bss.permute(X, Y, fl, p, inverse=False)
    bss.permute(Y, Z, fl, p, inverse=True)
    torch.cuda.synchronize()
    xn = x.numpy().view(np.uint16)
    ref = oracle.permute(xn, F, S, flags)
    assert np.array_equal(Y.cpu().view(torch.int16).numpy().view(np.uint16), ref)
    assert np.array_equal(Z.cpu().view(torch.int16).numpy().view(np.uint16), xn)
    refinv = oracle.permute(xn, F, S, flags, inverse=True)
    bss.permute(X, Y, fl, p, inverse=True)
    torch.cuda.synchronize()
    assert np.array_equal(Y.cpu().view(torch.int16).numpy().view(np.uint16), refinv)


@pytest.mark.gpu
def test_permute_full_size_round_trip_and_samples(bss):
    w = W.MIXED_75K
    flags = w.head_flags()
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(5)
    X = torch.randn(w.H, w.N, w.d, device=dev, generator=g).bfloat16()
    Y = torch.empty_like(X)
    Z = torch.empty_like(X)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    bss.permute(X, Y, fl, p)
    bss.permute(Y, Z, fl, p, inverse=True)
    torch.cuda.synchronize()
    assert torch.equal(X.view(torch.int16), Z.view(torch.int16))
    rng = np.random.default_rng(0)
    for h in range(w.H):
        for t in rng.integers(0, w.N, 50):
            dst = oracle.perm_index(int(t), w.F, w.S) if flags[h] else int(t)
            assert torch.equal(Y[h, dst].view(torch.int16), X[h, int(t)].view(torch.int16))


@pytest.mark.gpu
def test_permute_flagged_touches_only_flagged_heads(bss):
    w = W.SMALL
    H = 4
    x, _, _ = W.qkv(w, H=H, seed=5)
    flags = [1, 0, 0, 1]
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    dev = torch.device("cuda")
    xd = x.to(dev)
    out = torch.full_like(xd, 7.0)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    bss.permute(xd, out, fl, p, False, only_flagged=True)
    torch.cuda.synchronize()
    o = out.cpu()
    ref = oracle.permute(W.bf16_bits(x), w.F, w.S, flags)
    for h in range(H):
        if flags[h]:
            assert np.array_equal(o[h].view(torch.int16).numpy().view(np.uint16), ref[h])
        else:
            assert torch.all(o[h] == 7.0)
    back = torch.full_like(xd, 7.0)
    bss.permute(out, back, fl, p, True, only_flagged=True)
    torch.cuda.synchronize()
    b = back.cpu()
    for h in range(H):
        if flags[h]:
            assert torch.equal(b[h].view(torch.int16), x[h].view(torch.int16))
        else:
            assert torch.all(b[h] == 7.0)


@pytest.mark.gpu
def test_permute_full_size_bit_exact_every_row(bss):
    # all 10 heads x 75,600 rows of the mixed workload, forward and inverse, and
    # the flagged-only form the step uses, against the oracle's scalar permutation
    w = W.MIXED_75K
    flags = w.head_flags()
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(6)
    X = torch.randint(-32768, 32767, (w.H, w.N, w.d), dtype=torch.int16, device=dev, generator=g)
    Xb = X.view(torch.bfloat16)
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    xn = X.cpu().numpy().view(np.uint16)
    for inverse in (False, True):
        Y = torch.empty_like(Xb)
        bss.permute(Xb, Y, fl, p, inverse=inverse)
        Yf = torch.zeros_like(Xb)
        bss.permute(Xb, Yf, fl, p, inverse=inverse, only_flagged=True)
        torch.cuda.synchronize()
        ref = oracle.permute(xn, w.F, w.S, flags, inverse=inverse)
        assert np.array_equal(Y.cpu().view(torch.int16).numpy().view(np.uint16), ref)
        yf = Yf.cpu().view(torch.int16).numpy().view(np.uint16)
        for h in range(w.H):
            if flags[h]:
                assert np.array_equal(yf[h], ref[h]), f"head {h}"
            else:
                assert not yf[h].any(), f"head {h} was written"


@pytest.mark.gpu
def test_permute_flagged_multi_equals_three_single_launches(bss):
    # one launch for Q, K and V (the step's) is bit for bit three flagged launches;
    # unflagged heads of every output keep their bytes
    w = W.SMALL
    H = 4
    flags = [1, 0, 1, 1]
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    dev = torch.device("cuda")
    xs = [t.to(dev) for t in W.qkv(w, H=H, seed=8)]
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    for inverse in (False, True):
        one = [torch.full_like(xs[0], 7.0) for _ in range(3)]
        bss.permute_flagged_multi(xs, one, fl, p, inverse)
        ref = [torch.full_like(xs[0], 7.0) for _ in range(3)]
        for x, r in zip(xs, ref):
            bss.permute(x, r, fl, p, inverse, only_flagged=True)
        torch.cuda.synchronize()
        for a, b in zip(one, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.all(one[1][1] == 7.0)
    for n in (1, 2):
        outs = [torch.empty_like(xs[0]) for _ in range(n)]
        bss.permute_flagged_multi(xs[:n], outs, fl, p)
    torch.cuda.synchronize()
    with pytest.raises(bss.BssError):   # an output overlapping an input
        bss.permute_flagged_multi(xs, [xs[1], one[1], one[2]], fl, p)
