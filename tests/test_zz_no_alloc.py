"""sparse_mla_decode_noalloc: the decode step for callers that cannot allocate device
memory (a host framework that owns every device allocation, or a serving loop that
must not call cudaMalloc because it can synchronise the device and fail under
memory pressure).  The split partials live in the library's own 16 MiB scratch, so
the call takes no workspace.

The test calls the new C entry point directly through ctypes, twice in a row with
different inputs, and checks each result against sparse_mla_decode with a
caller-provided workspace, within the parity tolerances the other GPU tests use.
It runs last (file name) and passes alone or after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_mla_decode_03_gb300 import _lib, make_params, sparse_mla_decode
from sparse_mla_decode_03_gb300 import workloads as W

from _helpers import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


def _noalloc(q, kv, idx, out, lse, num_splits=0):
    lib = _lib.load()
    p = make_params(q.shape[0], q.shape[1], idx.shape[1], kv.shape[0], kv.stride(0))
    vp = ctypes.c_void_p
    return lib.sparse_mla_decode_noalloc(vp(q.data_ptr()), vp(kv.data_ptr()), vp(idx.data_ptr()),
                                         vp(out.data_ptr()), vp(lse.data_ptr()), ctypes.byref(p),
                                         num_splits, vp(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_path_on_two_calls():
    w = W.Workload("noalloc", 8, 64, 1000, 20000, "uniform", outlier_frac=0.0, seed=77)
    L = W.seq_lengths(w)
    kv = W.make_cache(w, L, device="cuda")
    q = W.make_q(w, device="cuda")
    out = torch.empty((8, 64, 448), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((8, 64), dtype=torch.float32, device="cuda")
    for variant in (0, 1):                       # two calls in a row, different index sets
        idx_np = W.make_indices(w, L, variant=variant)
        idx_np[variant, 700:] = -1               # a ragged query in each call
        idx = torch.as_tensor(idx_np, device="cuda")
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        assert _noalloc(q, kv, idx, out, lse) == 0
        ref_out, ref_lse = sparse_mla_decode(q, kv, idx)
        torch.cuda.synchronize()
        assert_out_close(out.float().cpu().numpy(), ref_out.float().cpu().numpy().astype(np.float64))
        assert_lse_close(lse.cpu().numpy(), ref_lse.cpu().numpy().astype(np.float64))


def test_noalloc_rejects_problems_beyond_its_scratch():
    q = torch.zeros((128, 128, 512), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((16, 584), dtype=torch.uint8, device="cuda")
    idx = torch.zeros((128, 64), dtype=torch.int32, device="cuda")
    out = torch.empty((128, 128, 448), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    # 128 x 128 heads x 448 fp32 partials = 28 MiB even with one split
    assert _noalloc(q, kv, idx, out, lse) == _lib.SMLA_ERR_SCRATCH_TOO_SMALL
    assert _noalloc(q, kv, idx, out, lse, num_splits=2) == _lib.SMLA_ERR_SCRATCH_TOO_SMALL


def test_noalloc_lowers_the_split_count_until_the_partials_fit():
    """When the default plan's partials exceed the 16 MiB scratch but fewer splits fit,
    the call takes the largest split count that fits; its result is then bit for bit
    that of sparse_mla_decode with that split count and a caller workspace."""
    from sparse_mla_decode_03_gb300 import smla_default_num_splits, smla_workspace_size
    limit = 16 << 20
    rows_per_seq = 4096
    for B, H, k in [(19, 64, 2048), (25, 64, 2048), (37, 64, 2048), (49, 64, 2048),
                    (37, 128, 2048), (26, 128, 4096)]:
        p = make_params(B, H, k, B * rows_per_seq, 584)
        S0 = smla_default_num_splits(p)
        if smla_workspace_size(p, S0) > limit and smla_workspace_size(p, 1) <= limit:
            break
    else:
        pytest.fail("no candidate shape whose default plan exceeds the scratch")
    S = S0
    while S > 1 and smla_workspace_size(p, S) > limit:
        S -= 1
    assert 1 <= S < S0
    w = W.Workload("noalloc_fit", B, H, k, rows_per_seq, "uniform", seed=78)
    L = W.seq_lengths(w)
    kv = W.make_cache(w, L, device="cuda")
    q = W.make_q(w, device="cuda")
    idx = torch.as_tensor(W.make_indices(w, L), device="cuda")
    out = torch.empty((B, H, 448), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    assert _noalloc(q, kv, idx, out, lse) == 0
    ref_out, ref_lse = sparse_mla_decode(q, kv, idx, num_splits=S)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
