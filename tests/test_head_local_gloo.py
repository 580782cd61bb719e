"""Head-local layout (blog section "Perform layout transformations on local
heads"): the two all-to-all exchanges around the per-head path, run with two
gloo ranks on the CPU.  The per-head step is a stand-in that needs every token
of a head, then the oracle's exact attention."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _full_inputs(H, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(H, N, d, generator=g) for _ in range(3)]


def _mixing_step(Qh, Kh, Vh, flags):
    # depends on the whole sequence of each head (a mean over all tokens) and on its flag
    f = flags.to(torch.float32).view(-1, 1, 1)
    return Qh * (1.0 + f) + Kh.mean(dim=1, keepdim=True) - Vh[:, :1, :]


def _oracle_step(geom):
    import oracle
    import workloads as W
    F, Hs, Ws, wf, ws = geom
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws)

    def step(Qh, Kh, Vh, flags):
        out = []
        for h in range(Qh.shape[0]):
            kind = oracle.TEMPORAL_FHW if int(flags[h]) else oracle.SPATIAL
            b = [W.bf16_bits(x[h].to(torch.bfloat16)) for x in (Qh, Kh, Vh)]
            o, _ = oracle.attention(*b, kind, g)
            out.append(torch.from_numpy(o.astype(np.float32)))
        return torch.stack(out)
    return step


def _rank_main(rank, world, port, case, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from block_sparse_spatio_gb300.head_local import head_local_attention
    H, N, d, flags, geom = case
    Qf, Kf, Vf = _full_inputs(H, N, d, seed=9)
    if geom is not None:  # bf16-representable inputs for the oracle step
        Qf, Kf, Vf = (x.to(torch.bfloat16).to(torch.float32) for x in (Qf, Kf, Vf))
    n = N // world
    shard = slice(rank * n, (rank + 1) * n)
    fl = torch.tensor(flags, dtype=torch.uint8)
    step = _mixing_step if geom is None else _oracle_step(geom)
    O = head_local_attention(Qf[:, shard].contiguous(), Kf[:, shard].contiguous(), Vf[:, shard].contiguous(), fl,
                             step)
    expect = step(Qf, Kf, Vf, fl)[:, shard]
    out[rank] = bool(torch.equal(O, expect))
    dist.barrier()
    dist.destroy_process_group()


def _run(case, world=2):
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, case, out), nprocs=world, join=True)
        return dict(out)


def test_exchanges_give_each_rank_whole_heads_and_return_its_tokens():
    res = _run((4, 12, 8, [0, 1, 1, 0], None))
    assert res == {0: True, 1: True}


def test_head_local_path_equals_unsplit_attention_oracle():
    # Small geometry: F=4, 6 x 8 latent, head 0 spatial (window 1), head 1 temporal (window 5)
    F, Hs, Ws = 4, 6, 8
    res = _run((2, F * Hs * Ws, 16, [0, 1], (F, Hs, Ws, 1, 5)))
    assert res == {0: True, 1: True}
