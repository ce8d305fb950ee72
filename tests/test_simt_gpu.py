"""The per-head fp32 SIMT form of the decode step (the pages' pre-MMA kernel style),
checked against the oracle through the C ABI, and against the tensor-core path."""
import numpy as np
import pytest
import torch

from sparse_mla_decode_03_gb300 import sparse_mla_decode, sparse_mla_decode_simt, smla_device_status

from _helpers import assert_lse_close, assert_out_close, oracle_decode, small_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,k", [(16, 1), (16, 300), (64, 17), (64, 129), (128, 64)])
def test_simt_matches_oracle(H, k):
    B = 2
    w, kv, q, idx_np = small_case(B, H, 2000, k, seed=300 + H + k)
    if k > 20:
        idx_np[1, k // 3: k // 2] = -1           # a masked run inside the list
    idx = torch.as_tensor(idx_np, device="cuda")
    out, lse = sparse_mla_decode_simt(q, kv, idx)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_decode(q, kv, idx_np)
    assert_out_close(out.float().cpu().numpy(), ref_out)
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_simt_empty_query_and_agreement_with_mma_path():
    B, H, k = 3, 64, 400
    w, kv, q, idx_np = small_case(B, H, 3000, k, seed=311)
    idx_np[2, :] = -1
    idx = torch.as_tensor(idx_np, device="cuda")
    out_s, lse_s = sparse_mla_decode_simt(q, kv, idx)
    out_m, lse_m = sparse_mla_decode(q, kv, idx)
    torch.cuda.synchronize()
    assert np.all(out_s[2].float().cpu().numpy() == 0)
    assert np.all(np.isneginf(lse_s[2].cpu().numpy()))
    assert_out_close(out_s.float().cpu().numpy(), out_m.float().cpu().numpy().astype(np.float64))
    assert_lse_close(lse_s.cpu().numpy(), lse_m.cpu().numpy().astype(np.float64))


def test_simt_reports_out_of_range_index():
    w, kv, q, idx_np = small_case(1, 16, 500, 32, seed=312)
    idx_np[0, 5] = kv.shape[0] + 10
    smla_device_status(clear=True)
    out, lse = sparse_mla_decode_simt(q, kv, torch.as_tensor(idx_np, device="cuda"))
    assert smla_device_status(clear=True) == -7
    idx_np[0, 5] = -1
    ref_out, ref_lse = oracle_decode(q, kv, idx_np)
    assert_out_close(out.float().cpu().numpy(), ref_out)
