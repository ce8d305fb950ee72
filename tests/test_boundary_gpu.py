"""The C ABI's error paths and stream/graph behaviour on a GPU."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_mla_decode_03_gb300 import (SmlaError, make_params, smla_default_num_splits,
                                        smla_workspace_size, sparse_mla_decode)
from sparse_mla_decode_03_gb300 import _lib
from sparse_mla_decode_03_gb300 import workloads as W

from _helpers import assert_lse_close, assert_out_close, oracle_decode, small_case

pytestmark = pytest.mark.gpu


def _raw_decode(q, kv, idx, out, lse, p, S, ws, ws_bytes):
    lib = _lib.load()
    vp = ctypes.c_void_p
    return lib.sparse_mla_decode(vp(q), vp(kv), vp(idx), vp(out), vp(lse), ctypes.byref(p), S,
                                 vp(ws), ws_bytes, vp(torch.cuda.current_stream().cuda_stream))


def test_error_statuses():
    w, kv, q, idx_np = small_case(2, 64, 300, 64, seed=1)
    idx = torch.as_tensor(idx_np, device="cuda")
    out = torch.empty((2, 64, 448), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 64), dtype=torch.float32, device="cuda")
    p = make_params(2, 64, 64, kv.shape[0], 584)
    need = smla_workspace_size(p, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = [q.data_ptr(), kv.data_ptr(), idx.data_ptr(), out.data_ptr(), lse.data_ptr()]
    assert _raw_decode(*args, p, 0, ws.data_ptr(), need) == 0
    assert _raw_decode(*args, p, 0, ws.data_ptr(), need - 1) == _lib.SMLA_ERR_WORKSPACE_TOO_SMALL
    assert _raw_decode(0, *args[1:], p, 0, ws.data_ptr(), need) == _lib.SMLA_ERR_INVALID_ARG
    assert _raw_decode(args[0] + 2, *args[1:], p, 0, ws.data_ptr(), need) == _lib.SMLA_ERR_INVALID_ARG
    assert _raw_decode(*args, p, 0, ws.data_ptr() + 16, need) == _lib.SMLA_ERR_INVALID_ARG
    assert _raw_decode(*args, p, 1000, ws.data_ptr(), need) == _lib.SMLA_ERR_INVALID_ARG
    bad = make_params(2, 48, 64, kv.shape[0], 584)
    assert _raw_decode(*args, bad, 0, ws.data_ptr(), need) == _lib.SMLA_ERR_UNSUPPORTED_SHAPE
    bad = make_params(2, 64, 64, kv.shape[0], 580)
    assert _raw_decode(*args, bad, 0, ws.data_ptr(), need) == _lib.SMLA_ERR_INVALID_ARG
    with pytest.raises(SmlaError):
        sparse_mla_decode(q, kv, idx, num_splits=999)
    torch.cuda.synchronize()


def test_default_plan_fills_the_device():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = make_params(32, 64, 2048, 1 << 21, 584)
    S = smla_default_num_splits(p)
    assert 1 <= S <= 128 and 32 * S <= 2 * sms


def test_side_stream_and_graph_replay():
    w, kv, q, idx_np = small_case(4, 64, 3000, 700, seed=3)
    idx = torch.as_tensor(idx_np, device="cuda")
    ro, rl = oracle_decode(q, kv, idx_np)
    s = torch.cuda.Stream()
    out = torch.empty((4, 64, 448), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((4, 64), dtype=torch.float32, device="cuda")
    p = make_params(4, 64, 700, kv.shape[0], 584)
    ws = torch.empty(smla_workspace_size(p, 0), dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(s):
        sparse_mla_decode(q, kv, idx, out=out, lse=lse, workspace=ws)
    s.synchronize()
    assert_out_close(out.float().cpu().numpy(), ro)
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sparse_mla_decode(q, kv, idx, out=out, lse=lse, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert_lse_close(lse.cpu().numpy(), rl)
