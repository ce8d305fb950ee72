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


def test_plan_reports_the_on_chip_merge():
    """The batch-32 / 64-head / top-2048 plan (4 splits) runs as one clustered launch;
    more than 8 splits use the split + combine kernels."""
    from sparse_mla_decode_03_gb300 import smla_decode_plan
    p = make_params(32, 64, 2048, 32 * 65536, 584)
    S, fused = smla_decode_plan(p, 0)
    assert S == smla_default_num_splits(p)
    assert fused and S <= 8
    assert smla_decode_plan(p, 16) == (16, False)
    assert smla_decode_plan(make_params(4, 16, 512, 4 * 16384, 584), 3) == (3, True)


@pytest.mark.parametrize("H,S", [(64, 1), (64, 4), (32, 3), (16, 8), (128, 2)])
def test_on_chip_merge_matches_split_and_combine(H, S):
    """sparse_mla_decode with the merge on chip equals the split kernel followed by the
    combine kernel on the same inputs, and both equal the oracle."""
    from sparse_mla_decode_03_gb300 import (smla_decode_plan, sparse_mla_combine,
                                            sparse_mla_decode_split)
    B, k = 3, 700
    w, kv, q, idx_np = small_case(B, H, 4000, k, seed=H + S)
    idx_np[1, 300:] = -1
    idx_np[2, :] = -1                        # an empty query
    idx = torch.as_tensor(idx_np, device="cuda")
    p = make_params(B, H, k, kv.shape[0], 584)
    assert smla_decode_plan(p, S) == (S, True)
    out_f, lse_f = sparse_mla_decode(q, kv, idx, num_splits=S)
    o_part, lse_part = sparse_mla_decode_split(q, kv, idx, S)
    out_u, lse_u = sparse_mla_combine(o_part, lse_part)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_decode(q, kv, idx_np)
    assert_out_close(out_f.float().cpu().numpy(), ref_out)
    assert_lse_close(lse_f.cpu().numpy(), ref_lse)
    assert_out_close(out_f.float().cpu().numpy(), out_u.float().cpu().numpy().astype(np.float64))
    assert np.all(out_f[2].float().cpu().numpy() == 0) and np.all(np.isneginf(lse_f[2].cpu().numpy()))


@pytest.mark.parametrize("S", [4, 12])   # merged on chip / split + combine kernels
def test_back_to_back_calls_keep_stream_order(S):
    """Programmatic launch lets a call start while the previous kernel ends: each call
    waits for it before touching memory.  A chain of calls sharing one workspace, each
    reading a q written by the kernel just before it, must give bit for bit the
    results of separate, synchronised calls."""
    w, kv, q, idx_np = small_case(8, 64, 5000, 1000, seed=11)
    idx = torch.as_tensor(idx_np, device="cuda")
    p = make_params(8, 64, 1000, kv.shape[0], 584)
    ws = torch.empty(smla_workspace_size(p, S), dtype=torch.uint8, device="cuda")
    qs = [q * (1.0 + 0.25 * i) for i in range(4)]
    ref = []
    for qi in qs:
        o, l = sparse_mla_decode(qi, kv, idx, num_splits=S, workspace=ws)
        torch.cuda.synchronize()
        ref.append((o.clone(), l.clone()))
    outs = [torch.empty((8, 64, 448), dtype=torch.bfloat16, device="cuda") for _ in qs]
    lses = [torch.empty((8, 64), dtype=torch.float32, device="cuda") for _ in qs]
    q_in = torch.empty_like(q)
    for chained in (True, False):
        for _ in range(3):
            for o in outs:
                o.zero_()
            for i, qi in enumerate(qs):
                if chained:
                    q_in.copy_(qi)   # a kernel right before the call writes its input
                # otherwise the calls follow each other directly, sharing the workspace
                sparse_mla_decode(q_in if chained else qi, kv, idx, out=outs[i], lse=lses[i],
                                  num_splits=S, workspace=ws)
            torch.cuda.synchronize()
            for i in range(len(qs)):
                assert torch.equal(outs[i], ref[i][0])
                assert torch.equal(lses[i], ref[i][1])


@pytest.mark.parametrize("capture", [False, True])
def test_pipelined_host_copies_over_three_streams(capture):
    """The serving pattern the bench's end-to-end leg uses: inputs copied from pinned
    host memory on one stream, decode on another, results copied back on a third,
    three rotating device buffer sets, optionally captured in a CUDA graph.  Every
    step's host result must equal a separate synchronous call bit for bit."""
    w, kv, q, idx_np = small_case(4, 64, 3000, 700, seed=21)
    idx = torch.as_tensor(idx_np, device="cuda")
    p = make_params(4, 64, 700, kv.shape[0], 584)
    S = smla_default_num_splits(p)
    ws = torch.empty(smla_workspace_size(p, S), dtype=torch.uint8, device="cuda")
    n_src, NB, n = 5, 3, 15
    qs = [q * (1.0 + 0.125 * i) for i in range(n_src)]
    ref = []
    for qi in qs:
        o, l = sparse_mla_decode(qi, kv, idx, num_splits=S, workspace=ws)
        torch.cuda.synchronize()
        ref.append((o.cpu(), l.cpu()))
    q_h = [x.cpu().pin_memory() for x in qs]
    idx_h = idx.cpu().pin_memory()
    q_d = [torch.empty_like(q) for _ in range(NB)]
    idx_d = [torch.empty_like(idx) for _ in range(NB)]
    out_d = [torch.empty((4, 64, 448), dtype=torch.bfloat16, device="cuda") for _ in range(NB)]
    lse_d = [torch.empty((4, 64), dtype=torch.float32, device="cuda") for _ in range(NB)]
    out_h = [torch.empty((4, 64, 448), dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    lse_h = [torch.empty((4, 64), dtype=torch.float32).pin_memory() for _ in range(n)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(NB)]
    ev_dec = [torch.cuda.Event() for _ in range(NB)]
    ev_res = [torch.cuda.Event() for _ in range(NB)]

    def steps(cs, chained):
        for i in range(n):
            k = i % NB
            if chained or i >= NB:
                s_in.wait_event(ev_dec[k])
            with torch.cuda.stream(s_in):
                q_d[k].copy_(q_h[i % n_src], non_blocking=True)
                idx_d[k].copy_(idx_h, non_blocking=True)
            ev_in[k].record(s_in)
            cs.wait_event(ev_in[k])
            if chained or i >= NB:
                cs.wait_event(ev_res[k])
            sparse_mla_decode(q_d[k], kv, idx_d[k], out=out_d[k], lse=lse_d[k], num_splits=S,
                              workspace=ws, stream=cs)
            ev_dec[k].record(cs)
            s_out.wait_event(ev_dec[k])
            with torch.cuda.stream(s_out):
                out_h[i].copy_(out_d[k], non_blocking=True)
                lse_h[i].copy_(lse_d[k], non_blocking=True)
            ev_res[k].record(s_out)

    if capture:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            s_in.wait_stream(cs)
            s_out.wait_stream(cs)
            steps(cs, chained=False)
            cs.wait_stream(s_in)
            cs.wait_stream(s_out)
        for h in out_h:
            h.zero_()
        g.replay()
    else:
        steps(torch.cuda.current_stream(), chained=True)
    torch.cuda.synchronize()
    for i in range(n):
        assert torch.equal(out_h[i], ref[i % n_src][0])
        assert torch.equal(lse_h[i], ref[i % n_src][1])
