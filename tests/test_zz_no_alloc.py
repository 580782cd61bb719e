"""The allocation-free tile-map build, checked against the allocating one.

bss_build_tile_map_csr_noalloc is for callers that cannot allocate device
memory themselves -- a framework whose caching allocator owns the GPU's memory
and enforces its own limit, or a latency-critical loop where cudaMalloc /
cudaFree would synchronize the device.  It keeps its scratch in a fixed
__device__ array that every call shares, so this test makes two calls in a row
(a large map, then smaller ones of other kinds and modes) through the C ABI
and compares each (the first made through the C ABI, the others through the
Python binding), bit for bit, with what bss_build_tile_map produces; and it
checks that refused calls write nothing.  It lives in its own file so that
pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

CALLS = [  # (workload, kind, temporal_permuted, rounding, BQ, BKV)
    (W.MIXED_75K, 1, 1, 0, 256, 128),
    (W.SMALL, 0, 1, 1, 128, 128),
    (W.SMALL, 1, 1, 1, 256, 128),   # tile-aligned permuted temporal: sink tiles lose their band twins
    (W.SMALL, 1, 0, 2, 256, 128),   # every visited tile masked, temporal heads in (F,H,W) order
    (W.MIXED_75K, 0, 1, 2, 128, 64),
]


@pytest.mark.gpu
def test_noalloc_tile_map_matches_allocating_build_on_two_calls_in_a_row(bss):
    lib = bss.load()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    for w, kind, tperm, rounding, BQ, BKV in CALLS:
        p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=tperm, rounding=rounding)
        nq, nkv = bss.noalloc_map_dims(p, kind, BQ, BKV)
        row_ptr = torch.full((nq + 1,), -7, dtype=torch.int32, device=dev)
        entries = torch.full((nq * nkv,), -7, dtype=torch.int32, device=dev)
        stats = torch.full((len(bss.STAT_NAMES),), -7, dtype=torch.int64, device=dev)
        if w is W.SMALL:  # through the Python binding
            bss.build_tile_map_csr_noalloc(p, kind, row_ptr, entries, stats, BQ, BKV, stream=stream)
        else:  # straight through the C ABI
            mp = p.c()
            st = lib.bss_build_tile_map_csr_noalloc(ctypes.byref(mp), kind, BQ, BKV,
                                                    ctypes.c_void_p(row_ptr.data_ptr()),
                                                    ctypes.c_void_p(entries.data_ptr()), entries.numel(),
                                                    ctypes.c_void_p(stats.data_ptr()),
                                                    ctypes.c_void_p(stream.cuda_stream))
            assert st == 0, lib.bss_last_error_message()
        torch.cuda.synchronize()
        assert bss.get_device_status() == 0
        with bss.build_tile_map(p, BQ, BKV) as tm:
            ref_ptr, ref_ent = tm.csr(kind)
            ref_stats = tm.stats(kind)
        got_ptr = row_ptr.cpu().numpy()
        assert np.array_equal(got_ptr, ref_ptr)
        nnz = int(got_ptr[-1])
        assert np.array_equal(entries[:nnz].cpu().numpy(), ref_ent)
        assert stats.cpu().tolist() == [ref_stats[k] for k in bss.STAT_NAMES]
        assert lib.bss_last_error_message() == b""


@pytest.mark.gpu
def test_noalloc_rejections_leave_the_outputs_untouched(bss):
    # each refused call returns its status before any launch: the sentinel-filled
    # device buffers keep every byte, and a later good call clears the message
    lib = bss.load()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    w = W.SMALL
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=1, rounding=1)
    nq, nkv = bss.noalloc_map_dims(p, 1, 256, 128)
    row_ptr = torch.full((nq + 2,), -7, dtype=torch.int32, device=dev)
    entries = torch.full((nq * nkv + 1,), -7, dtype=torch.int32, device=dev)
    stats = torch.full((len(bss.STAT_NAMES) + 1,), -7, dtype=torch.int64, device=dev)
    ptr = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)  # noqa: E731
    mp = p.c()
    big = bss.MaskParams(21, 180, 320, 128, 3, 2450, temporal_permuted=1, rounding=1).c()
    s = ctypes.c_void_p(stream.cuda_stream)
    cases = [
        (ctypes.byref(big), 1, 128, 128, ptr(row_ptr), ptr(entries), 1 << 40, ptr(stats), 2),  # too large
        (ctypes.byref(mp), 1, 256, 128, ptr(row_ptr), ptr(entries), nq * nkv - 1, ptr(stats), 1),  # capacity
        (ctypes.byref(mp), 1, 256, 128, ptr(row_ptr, 2), ptr(entries), nq * nkv, ptr(stats), 1),  # misaligned
        (ctypes.byref(mp), 1, 256, 128, ptr(row_ptr), ptr(entries, 1), nq * nkv, ptr(stats), 1),
        (ctypes.byref(mp), 1, 256, 128, ptr(row_ptr), ptr(entries), nq * nkv, ptr(stats, 4), 1),
        (ctypes.byref(mp), 1, 256, 128, None, ptr(entries), nq * nkv, ptr(stats), 1),            # NULL
        (ctypes.byref(mp), 3, 256, 128, ptr(row_ptr), ptr(entries), nq * nkv, ptr(stats), 1),    # kind
        (ctypes.byref(mp), 1, 8, 128, ptr(row_ptr), ptr(entries), nq * nkv, ptr(stats), 1),      # tile size
    ]
    for i, (*args, want) in enumerate(cases):
        assert lib.bss_build_tile_map_csr_noalloc(*args, s) == want, f"case {i}"
        assert lib.bss_last_error_message() != b"", f"case {i}"
        torch.cuda.synchronize()
        assert bool((row_ptr == -7).all()) and bool((entries == -7).all()) and bool((stats == -7).all()), \
            f"case {i} wrote its outputs"
    assert lib.bss_build_tile_map_csr_noalloc(ctypes.byref(mp), 1, 256, 128, ptr(row_ptr), ptr(entries),
                                              nq * nkv, ptr(stats), s) == 0
    assert lib.bss_last_error_message() == b""
    torch.cuda.synchronize()
    assert bss.get_device_status() == 0
    assert int(row_ptr[nq + 1]) == -7 and int(stats[-1]) == -7   # nothing past the declared sizes
