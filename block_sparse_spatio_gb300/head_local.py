"""Head-local layout for sequence-parallel inference.

Blog "Accelerating Spatio-Temporal Attention for Video Diffusion on TPUs",
section "Perform layout transformations on local heads": with the sequence
split over P devices, each device first holds every head for 1/P of the
tokens; one all-to-all exchange gives each device H/P heads with the whole
sequence (the head-local layout).  The per-head routing flags travel with
their heads; the permutation to (H,W,F) order, the sparse attention and the
inverse permutation run there, where every token a head needs is local; a
second all-to-all returns the outputs to the sequence-split layout.

The exchanges use ``torch.distributed.all_to_all_single`` (NCCL between GPUs);
the per-head work is the library's own kernels (``attention_step``).  Sending
needs no packing: the local [H][N/P][d] tensor is already ordered by
destination rank (heads r*H/P .. (r+1)*H/P - 1 go to rank r).  Receiving
transposes (source rank, head) into [H/P][N][d].
"""
from __future__ import annotations


def _exchange_to_heads(x, world: int, group):
    """[H][N/P][d] (all heads, this rank's tokens) -> [H/P][N][d] (this rank's
    heads, all tokens, token blocks in source-rank order)."""
    import torch
    import torch.distributed as dist
    H, n, d = x.shape
    recv = torch.empty_like(x)  # [P (source rank)][H/P][N/P][d]
    dist.all_to_all_single(recv, x.contiguous(), group=group)
    return recv.view(world, H // world, n, d).transpose(0, 1).reshape(H // world, world * n, d)


def _exchange_to_tokens(y, world: int, group):
    """[H/P][N][d] (this rank's heads) -> [H][N/P][d] (all heads, this rank's tokens)."""
    import torch
    import torch.distributed as dist
    hl, N, d = y.shape
    n = N // world
    send = y.view(hl, world, n, d).transpose(0, 1).contiguous()  # [P (destination)][H/P][N/P][d]
    recv = torch.empty_like(send)  # [P (source rank = head group)][H/P][N/P][d]
    dist.all_to_all_single(recv, send, group=group)
    return recv.view(world * hl, n, d)


def head_local_attention(Q, K, V, head_is_temporal, step, group=None):
    """Sequence-split attention through the head-local layout.

    Q, K, V: [H][N/P][d] bf16, this rank's contiguous 1/P of the (F,H,W)-ordered
    tokens for every head (rank r holds tokens r*N/P .. (r+1)*N/P - 1).
    head_is_temporal: uint8[H] routing flags, the same on every rank.
    step(Qh, Kh, Vh, flags_h) -> Oh: the per-head path on the local heads
    ([H/P][N][d] in, [H/P][N][d] out), e.g. ``attention_step`` with its map and
    workspaces bound.  H and N must be multiples of the group size.
    Returns O: [H][N/P][d], this rank's tokens of every head."""
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    H = Q.shape[0]
    if H % world:
        raise ValueError(f"{H} heads do not split over {world} ranks")
    if world == 1:
        return step(Q, K, V, head_is_temporal)
    hl = H // world
    Qh, Kh, Vh = (_exchange_to_heads(x, world, group) for x in (Q, K, V))
    Oh = step(Qh, Kh, Vh, head_is_temporal[rank * hl:(rank + 1) * hl])
    return _exchange_to_tokens(Oh, world, group)


def make_attention_step(tile_map, heads_local: int, N: int, d: int, device=None):
    """A ``step`` for ``head_local_attention``: the library's permute -> sparse
    attention path (``attention_step``) on the local heads, with its workspaces
    allocated once ([H/P][N][d] bf16 each)."""
    import torch

    from . import attention_step
    device = device or torch.device("cuda")
    ws = [torch.empty(heads_local, N, d, dtype=torch.bfloat16, device=device) for _ in range(4)]

    def step(Qh, Kh, Vh, flags):
        Oh = ws[3]
        attention_step(Qh, Kh, Vh, Oh, tile_map, flags, ws[0], ws[1], ws[2])
        return Oh

    return step
