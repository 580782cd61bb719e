"""Failure detection without a GPU fault: a bounded device wait that nothing
completes records BSS_ERR_TIMEOUT, the kernel returns, the host reads the
status, and the context keeps running the attention kernel correctly."""
import pytest
import torch

import oracle
from _util import compare, oracle_kind, oracle_rows, run_gpu
from test_gpu_attention import _inputs


@pytest.mark.gpu
def test_bounded_wait_times_out_and_the_context_stays_usable(bss):
    dev = torch.device("cuda")
    assert bss.get_device_status() == 0
    waited = torch.zeros(1, dtype=torch.int64, device=dev)
    bss.diag_wait_timeout(5_000_000, waited)  # 5 ms
    torch.cuda.synchronize()
    assert bss.status_string(bss.get_device_status()) == "BSS_ERR_TIMEOUT"
    assert bss.get_device_status() == 0  # reading clears the word
    w = int(waited.item())
    assert 5_000_000 <= w < 500_000_000, w
    # the same context still computes attention correctly
    F, Hs, Ws, d, wf, ws, flags = 5, 7, 9, 64, 1, 5, [1, 0]
    q, k, v = _inputs(2, F * Hs * Ws, d, seed=61)
    p = bss.MaskParams(F, Hs, Ws, d, wf, ws)
    out, lse, _ = run_gpu(bss, q, k, v, flags, p)
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=128)
    for h, fl in enumerate(flags):
        Oref, lref = oracle_rows(q, k, v, h, oracle_kind(fl, 1), g, None, False)
        compare(out[h].numpy(), lse[h].numpy(), Oref, lref, f"after timeout, head {h}")


@pytest.mark.gpu
def test_a_map_of_another_geometry_is_refused_before_any_launch(bss):
    dev = torch.device("cuda")
    F, Hs, Ws, d = 5, 7, 9, 64
    q, k, v = _inputs(2, F * Hs * Ws, d, seed=62)
    Q, K, V = (x.to(dev) for x in (q, k, v))
    O = torch.zeros_like(Q)
    fl = torch.tensor([0, 1], dtype=torch.uint8, device=dev)
    other = bss.MaskParams(F + 1, Hs, Ws, d, 1, 5)  # one more frame
    with bss.build_tile_map(other) as tm:
        with pytest.raises(ValueError):
            bss.sparse_attention(Q, K, V, O, tm, fl)
        with pytest.raises(ValueError):
            bss.sparse_attention_fused(Q, K, V, O, tm, fl)
    torch.cuda.synchronize()
    assert torch.all(O == 0)
    assert bss.get_device_status() == 0
