"""The SMLA_DEBUG build (libsmla_debug.so): the same C ABI and kernels with device-side
bounds checks of every computed shared-memory address (the explicit shared loads
and stores of the converters, the softmax and the epilogue) and of every gathered
row, reported as SMLA_ERR_INTERNAL in that library's device status word, the access
skipped, no trap.

A correct kernel never trips them, and the checks do not touch the arithmetic: on
every shape here the debug build's status word stays 0 and its out and lse are
bit-identical to the release build's."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_mla_decode_03_gb300 import _lib, make_params
from sparse_mla_decode_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _decode(lib, q, kv, idx, num_splits):
    B, H = q.shape[0], q.shape[1]
    p = make_params(B, H, idx.shape[1], kv.shape[0], kv.stride(0))
    need = ctypes.c_size_t()
    assert lib.smla_workspace_size(ctypes.byref(p), num_splits, ctypes.byref(need)) == 0
    ws = torch.empty(max(need.value, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, H, 448), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    vp = ctypes.c_void_p
    st = lib.sparse_mla_decode(vp(q.data_ptr()), vp(kv.data_ptr()), vp(idx.data_ptr()),
                               vp(out.data_ptr()), vp(lse.data_ptr()), ctypes.byref(p),
                               num_splits, vp(ws.data_ptr()), need.value,
                               vp(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def _status(lib):
    v = ctypes.c_int32()
    assert lib.smla_device_status(ctypes.byref(v), 1) == 0
    return v.value


@pytest.mark.parametrize("H,B,k,S", [(64, 3, 700, 0), (64, 2, 512, 1), (16, 4, 900, 0),
                                     (16, 2, 300, 3), (32, 2, 640, 0), (128, 1, 256, 2)])
def test_debug_build_matches_release_and_reports_nothing(H, B, k, S):
    rel, dbg = _lib.load(), _lib.load_debug()
    w = W.Workload("dbg", B, H, k, 4096, "uniform", seed=900 + H + B)
    L = W.seq_lengths(w)
    kv = W.make_cache(w, L, device="cuda")
    q = W.make_q(w, device="cuda")
    idx_np = W.make_indices(w, L)
    idx_np[-1, k // 3:] = -1                      # a query with masked slots
    idx = torch.as_tensor(idx_np, device="cuda")
    _status(rel)
    _status(dbg)
    out_r, lse_r = _decode(rel, q, kv, idx, S)
    out_d, lse_d = _decode(dbg, q, kv, idx, S)
    assert _status(dbg) == 0
    assert _status(rel) == 0
    assert torch.equal(out_r.view(torch.int16), out_d.view(torch.int16))
    assert np.array_equal(lse_r.numpy().view(np.int32), lse_d.numpy().view(np.int32))
