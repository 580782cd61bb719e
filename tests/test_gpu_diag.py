"""One-tile tensor-core self-test (TMA + swizzled shared memory + tcgen05.mma
with shared-memory and tensor-memory operands), against float64 matmuls."""
import pytest
import torch


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_mma_tile_matches_matmul(bss, d):
    g = torch.Generator().manual_seed(100 + d)
    A = torch.randn(128, d, generator=g).bfloat16()
    B = torch.randn(128, d, generator=g).bfloat16()
    V = torch.randn(128, d, generator=g).bfloat16()
    P = torch.rand(128, 128, generator=g).bfloat16()
    dev = torch.device("cuda")
    S = torch.full((128, 128), float("nan"), device=dev)
    O = torch.full((128, d), float("nan"), device=dev)
    bss.diag_mma_tile(A.to(dev), B.to(dev), P.to(dev), V.to(dev), S, O)
    assert bss.get_device_status() == 0
    Sref = A.double() @ B.double().T
    Oref = P.double() @ V.double()
    es = (S.double().cpu() - Sref).abs().max().item()
    eo = (O.double().cpu() - Oref).abs().max().item()
    assert es < 1e-3, f"S = A B^T wrong: max err {es}"
    assert eo < 1e-3, f"O = P V wrong: max err {eo}"
