"""Guard bands around every output: each output is a view inside a larger buffer
whose bands before and after hold a sentinel; after the kernels the bands must
be unchanged (no write outside the output, e.g. by a clipped TMA store of the
ragged last tile or a row-wise store)."""
import pytest
import torch

import workloads as W

G = 4096  # guard elements on each side (a multiple of 16 bytes for every dtype)


def guarded(shape, dtype, fill, dev):
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + 2 * G,), fill, dtype=dtype, device=dev)
    return buf, buf[G:G + n].view(*shape)


def intact(buf, fill):
    return bool(torch.all(buf[:G] == fill)) and bool(torch.all(buf[-G:] == fill))


GEOMS = [(5, 7, 9, 64, 1, 5, [1, 0]), (3, 10, 13, 128, 0, 20, [1, 1, 0]), (1, 1, 1, 64, 0, 0, [1, 0]),
         (4, 5, 5, 128, 1, 2, [0, 1])]


@pytest.mark.gpu
@pytest.mark.parametrize("geom", GEOMS, ids=["s63_d64", "s130_d128", "one_token", "n100"])
@pytest.mark.parametrize("path", ["step", "explicit", "fused", "dense", "bq128"])
def test_attention_writes_only_its_outputs(bss, geom, path):
    F, Hs, Ws, d, wf, ws, flags = geom
    N, H = F * Hs * Ws, len(flags)
    dev = torch.device("cuda")
    q, k, v = W.qkv(W.SMALL, H=H, N=N, d=d, seed=71)
    Q, K, V = (x.to(dev) for x in (q, k, v))
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    sent = -7.0
    obuf, O = guarded((H, N, d), torch.bfloat16, sent, dev)
    lbuf, L = guarded((H, N), torch.float32, sent, dev)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws)
    if path == "dense":
        bss.dense_attention(Q, K, V, O, lse=L)
    else:
        with bss.build_tile_map(p, BQ=128 if path == "bq128" else bss.ATTN_BQ) as tm:
            wsp = [torch.empty_like(Q) for _ in range(3)]
            if path in ("step", "bq128"):
                bss.attention_step(Q, K, V, O, tm, fl, *wsp, lse=L)
            elif path == "explicit":
                Qp, Kp, Vp = wsp
                bss.permute(Q, Qp, fl, p, False)
                bss.permute(K, Kp, fl, p, False)
                bss.permute(V, Vp, fl, p, False)
                bss.sparse_attention(Qp, Kp, Vp, O, tm, fl, lse=L)
            else:
                bss.sparse_attention_fused(Q, K, V, O, tm, fl, lse=L)
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    assert intact(obuf, sent) and intact(lbuf, sent)
    assert torch.isfinite(O.float()).all()


@pytest.mark.gpu
@pytest.mark.parametrize("only_flagged", [False, True])
def test_permute_writes_only_its_output(bss, only_flagged):
    F, Hs, Ws, d = 3, 10, 13, 128
    N = F * Hs * Ws
    dev = torch.device("cuda")
    x = torch.randn(3, N, d, device=dev).to(torch.bfloat16)
    fl = torch.tensor([1, 0, 1], dtype=torch.uint8, device=dev)
    sent = 5.0
    buf, out = guarded((3, N, d), torch.bfloat16, sent, dev)
    p = bss.MaskParams(F, Hs, Ws, d, 1, 1)
    bss.permute(x, out, fl, p, False, only_flagged=only_flagged)
    torch.cuda.synchronize()
    assert intact(buf, sent)
    if only_flagged:
        assert torch.all(out[1] == sent)  # the unflagged head was not touched


@pytest.mark.gpu
def test_routing_writes_only_its_outputs(bss):
    w = W.SMALL
    dev = torch.device("cuda")
    q, k, v = W.qkv(w, H=2, seed=72)
    Q, K, V = (x.to(dev) for x in (q, k, v))
    rows = torch.tensor(W.sample_rows(w.N, 40, seed=3), dtype=torch.int32, device=dev)
    fbuf, flags = guarded((2,), torch.uint8, 9, dev)
    ebuf, err = guarded((2, 2), torch.float32, -3.0, dev)
    bss.route_heads(Q, K, V, bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws), rows, flags, err)
    torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    assert intact(fbuf, 9) and intact(ebuf, -3.0)
    assert set(flags.cpu().tolist()) <= {0, 1}


@pytest.mark.gpu
@pytest.mark.parametrize("geom", GEOMS, ids=["s63_d64", "s130_d128", "one_token", "n100"])
@pytest.mark.parametrize("rounding", [0, 1])
def test_step_writes_only_its_output_and_workspaces(bss, geom, rounding):
    # bss_attention_step writes O and the temporal heads' rows of the three
    # permutation workspaces (one launch), nothing around them; tile-aligned
    # maps include column-masked sink tiles where the geometry has them
    F, Hs, Ws, d, wf, ws, flags = geom
    N, H = F * Hs * Ws, len(flags)
    dev = torch.device("cuda")
    q, k, v = W.qkv(W.SMALL, H=H, N=N, d=d, seed=73)
    Q, K, V = (x.to(dev) for x in (q, k, v))
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    sent = -7.0
    obuf, O = guarded((H, N, d), torch.bfloat16, sent, dev)
    wbufs = [guarded((H, N, d), torch.bfloat16, sent, dev) for _ in range(3)]
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws, rounding=rounding)
    with bss.build_tile_map(p) as tm:
        bss.attention_step(Q, K, V, O, tm, fl, *[w[1] for w in wbufs])
        torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    assert intact(obuf, sent)
    for buf, wsp in wbufs:
        assert intact(buf, sent)
        for h, f in enumerate(flags):
            if not f:
                assert torch.all(wsp[h] == sent)  # spatial heads are never copied
    assert torch.isfinite(O.float()).all()


@pytest.mark.gpu
def test_multi_permute_writes_only_its_outputs(bss):
    F, Hs, Ws, d = 3, 10, 13, 128
    N = F * Hs * Ws
    dev = torch.device("cuda")
    xs = [torch.randn(3, N, d, device=dev).to(torch.bfloat16) for _ in range(3)]
    fl = torch.tensor([1, 0, 1], dtype=torch.uint8, device=dev)
    sent = 5.0
    outs = [guarded((3, N, d), torch.bfloat16, sent, dev) for _ in range(3)]
    p = bss.MaskParams(F, Hs, Ws, d, 1, 1)
    for inverse in (False, True):
        bss.permute_flagged_multi(xs, [o[1] for o in outs], fl, p, inverse)
        torch.cuda.synchronize()
        for buf, out in outs:
            assert intact(buf, sent)
            assert torch.all(out[1] == sent)
