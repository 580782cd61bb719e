"""The allocation-free tile-map build, checked against the allocating one.

bss_build_tile_map_csr_noalloc is for callers that cannot allocate device
memory themselves -- a framework whose caching allocator owns the GPU's memory
and enforces its own limit, or a latency-critical loop where cudaMalloc /
cudaFree would synchronize the device.  It keeps its scratch in a fixed
__device__ array that every call shares, so this test makes two calls in a row
(a large map, then a smaller one of a different kind) through the C ABI and
compares each (the first made through the C ABI, the second through the
Python binding), bit for bit, with what bss_build_tile_map produces.  It lives in
its own file so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

CALLS = [  # (workload, kind, temporal_permuted, rounding, BQ, BKV)
    (W.MIXED_75K, 1, 1, 0, 256, 128),
    (W.SMALL, 0, 1, 1, 128, 128),
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
        stats = torch.full((6,), -7, dtype=torch.int64, device=dev)
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
