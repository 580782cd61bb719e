"""The pipelined host-buffer step (bss_attention_step_host, through the C ABI)
gives the same O as the device step, also when consecutive calls overlap (the
workspace's buffer sets used in turn, each reused once its previous call is
done)."""
import pytest
import torch

import workloads as W


@pytest.mark.gpu
@pytest.mark.parametrize("hpc", [1, 2, 3, 5])
@pytest.mark.parametrize("pinned", [False, True])
@pytest.mark.parametrize("depth", [1, 2, 3])
def test_host_steps_match_device_step(bss, hpc, pinned, depth):
    w = W.SMALL
    H = 5
    flags = torch.tensor([0, 1, 1, 0, 1], dtype=torch.uint8)
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    dev = torch.device("cuda")
    calls = 5  # more calls than buffer sets: every set is reused
    inputs = [W.qkv(w, H=H, seed=21 + c) for c in range(calls)]
    with bss.build_tile_map(p) as tm:
        fl = flags.to(dev)
        expect = []
        for q, k, v in inputs:
            Q, K, V = (x.to(dev) for x in (q, k, v))
            O = torch.empty_like(Q)
            ws = [torch.empty_like(Q) for _ in range(3)]
            bss.attention_step(Q, K, V, O, tm, fl, *ws)
            expect.append(O.cpu())
        pin = (lambda x: x.pin_memory()) if pinned else (lambda x: x.clone())  # pageable copies work too
        hosts = [tuple(pin(x) for x in qkv) for qkv in inputs]
        outs = [pin(torch.empty_like(inputs[0][0])) for _ in range(calls)]
        wsp = bss.step_workspace(p, H, depth=depth, heads_per_group=hpc)
        hfl = pin(flags)
        events = [bss.attention_step_host(*hosts[c], outs[c], tm, hfl, wsp) for c in range(calls)]
        for e in events:
            e.synchronize()
        torch.cuda.synchronize()
        assert bss.get_device_status() == 0
        for c in range(calls):
            assert torch.equal(outs[c].view(torch.int16), expect[c].view(torch.int16)), f"call {c}"
        wsp.destroy()


@pytest.mark.gpu
def test_host_step_rejects_mismatched_buffers_before_any_work(bss):
    w = W.SMALL
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    hq = torch.zeros(2, w.N, w.d, dtype=torch.bfloat16).pin_memory()
    ho = torch.full_like(hq, 5.0)
    flags = torch.tensor([0, 1], dtype=torch.uint8)
    with bss.build_tile_map(p) as tm, bss.step_workspace(p, 2) as wsp:
        with pytest.raises(ValueError):  # shape of another H
            bss.attention_step_host(hq[:1], hq[:1], hq[:1], ho[:1], tm, flags[:1], wsp)
        other = bss.MaskParams(w.F, w.Hs, w.Ws + 8, w.d, w.wf, w.ws)
        with bss.build_tile_map(other) as tm2, pytest.raises(ValueError):  # geometry
            bss.attention_step_host(hq, hq, hq, ho, tm2, flags, wsp)
        lib = bss.load()
        import ctypes
        rc = lib.bss_attention_step_host(ctypes.c_void_p(hq.data_ptr()), ctypes.c_void_p(hq.data_ptr()),
                                         ctypes.c_void_p(hq.data_ptr()), ctypes.c_void_p(ho.data_ptr()),
                                         None, tm.handle, wsp.handle, None, None)
        assert rc == 1 and b"NULL" in lib.bss_last_error_message()
        torch.cuda.synchronize()
        assert bool((ho == 5.0).all())
    with pytest.raises(bss.BssError):
        bss.step_workspace(p, 2, depth=9)


@pytest.mark.gpu
def test_head_local_path_on_one_rank_is_the_attention_step(bss):
    from block_sparse_spatio_gb300.head_local import head_local_attention, make_attention_step
    w = W.SMALL
    q, k, v = W.qkv(w, H=4, seed=33)
    dev = torch.device("cuda")
    Q, K, V = (x.to(dev) for x in (q, k, v))
    fl = torch.tensor([1, 0, 1, 0], dtype=torch.uint8, device=dev)
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    with bss.build_tile_map(p) as tm:
        O = head_local_attention(Q, K, V, fl, make_attention_step(tm, 4, w.N, w.d, dev)).clone()
        O2 = torch.empty_like(Q)
        ws = [torch.empty_like(Q) for _ in range(3)]
        bss.attention_step(Q, K, V, O2, tm, fl, *ws)
        torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    assert torch.equal(O.view(torch.int16), O2.view(torch.int16))


@pytest.mark.gpu
def test_host_steps_at_full_size_match_device_step(bss):
    # the configuration the benchmark's end-to-end leg times: mixed 75.6K tokens x
    # 10 heads, the default workspace (three sets) and head groups (two heads),
    # four consecutive calls with different inputs, so that copies and kernels
    # of neighbouring calls overlap and a set is reused
    w = W.MIXED_75K
    dev = torch.device("cuda")
    flags = torch.tensor(w.head_flags(), dtype=torch.uint8)
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    calls = 4
    with bss.build_tile_map(p) as tm:
        fl = flags.to(dev)
        ws = [torch.empty(w.H, w.N, w.d, dtype=torch.bfloat16, device=dev) for _ in range(3)]
        hosts, expect = [], []
        for c in range(calls):
            Q, K, V = W.qkv_device(w, dev, seed=500 + c)
            O = torch.empty_like(Q)
            bss.attention_step(Q, K, V, O, tm, fl, *ws)
            expect.append(O.cpu())
            hosts.append(tuple(x.cpu().pin_memory() for x in (Q, K, V)))
            del Q, K, V, O
        outs = [torch.empty(w.H, w.N, w.d, dtype=torch.bfloat16).pin_memory() for _ in range(calls)]
        wsp = bss.step_workspace(p, w.H)
        hfl = flags.pin_memory()
        events = [bss.attention_step_host(*hosts[c], outs[c], tm, hfl, wsp) for c in range(calls)]
        for e in events:
            e.synchronize()
        torch.cuda.synchronize()
        assert bss.get_device_status() == 0
        for c in range(calls):
            assert torch.equal(outs[c].view(torch.int16), expect[c].view(torch.int16)), f"call {c}"
        wsp.destroy()


@pytest.mark.gpu
def test_device_step_without_flags_or_permutation_is_plain_attention(bss):
    # bss_attention_step falls back to one sparse-attention launch when nothing
    # is permuted: no flags (every head spatial), or a map that keeps temporal
    # heads in (F,H,W) order; bit for bit the direct call in both cases, and the
    # host-buffer step on such a map gives the same O
    w = W.SMALL
    H = 3
    dev = torch.device("cuda")
    q, k, v = W.qkv(w, H=H, seed=41)
    Q, K, V = (x.to(dev) for x in (q, k, v))
    for tperm, flags in ((1, None), (0, [1, 0, 1])):
        p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=tperm)
        fl = None if flags is None else torch.tensor(flags, dtype=torch.uint8, device=dev)
        with bss.build_tile_map(p) as tm:
            O1, O2 = torch.empty_like(Q), torch.empty_like(Q)
            l1 = torch.empty(H, w.N, device=dev)
            l2 = torch.empty(H, w.N, device=dev)
            bss.attention_step(Q, K, V, O1, tm, fl, None, None, None, lse=l1)
            bss.sparse_attention(Q, K, V, O2, tm, fl, lse=l2)
            torch.cuda.synchronize()
            assert bss.get_device_status() == 0
            assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
            assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
            if flags is not None:
                with bss.step_workspace(p, H, depth=2, heads_per_group=2) as wsp:
                    hq, hk, hv = (x.pin_memory() for x in (q, k, v))
                    ho = torch.empty_like(hq).pin_memory()
                    e = bss.attention_step_host(hq, hk, hv, ho, tm, torch.tensor(flags, dtype=torch.uint8), wsp)
                    e.synchronize()
                    torch.cuda.synchronize()
                assert torch.equal(ho.view(torch.int16), O1.cpu().view(torch.int16))
