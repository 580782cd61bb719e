"""The pipelined host-buffer step gives the same O as the device step."""
import pytest
import torch

import workloads as W


@pytest.mark.gpu
@pytest.mark.parametrize("hpc", [1, 2, 3])
def test_host_step_matches_device_step(bss, hpc):
    w = W.SMALL
    H = 5
    q, k, v = W.qkv(w, H=H, seed=21)
    flags = torch.tensor([0, 1, 1, 0, 1], dtype=torch.uint8)
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws)
    dev = torch.device("cuda")
    with bss.build_tile_map(p) as tm:
        fl = flags.to(dev)
        Q, K, V = (x.to(dev) for x in (q, k, v))
        O = torch.empty_like(Q)
        ws = [torch.empty_like(Q) for _ in range(4)]
        bss.attention_step(Q, K, V, O, tm, fl, *ws)
        hq, hk, hv = (x.pin_memory() for x in (q, k, v))
        ho = torch.empty_like(q).pin_memory()
        wsp = bss.step_workspace(H, w.N, w.d, dev)
        bss.attention_step_host(hq, hk, hv, ho, tm, fl, wsp, heads_per_chunk=hpc)
        torch.cuda.synchronize()
        assert bss.get_device_status() == 0
        assert torch.equal(ho.view(torch.int16), O.cpu().view(torch.int16))
