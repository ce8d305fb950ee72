"""Decode over a paged cache (block table -> pool rows) through the C ABI.

The pool is the flat cache of the other tests with its pages shuffled; the block
tables undo the shuffle, so the paged call must equal the flat call on the matching
row ids, and the oracle."""
import numpy as np
import pytest
import torch

from sparse_mla_decode_03_gb300 import (smla_device_status, sparse_mla_decode,
                                        sparse_mla_decode_paged)
from sparse_mla_decode_03_gb300 import workloads as W

from _helpers import assert_lse_close, assert_out_close, oracle_decode, small_case

pytestmark = pytest.mark.gpu


def _paged(B, H, n_rows, k, page, seed):
    """Flat case + the same rows as a shuffled page pool with block tables."""
    w, kv, q, idx = small_case(B, H, n_rows, k, seed=seed)
    assert n_rows % page == 0
    n_pages = kv.shape[0] // page
    rng = np.random.default_rng(seed)
    perm = rng.permutation(n_pages)              # pool page p holds flat page perm[p]
    where = np.empty(n_pages, dtype=np.int64)    # flat page -> pool page
    where[perm] = np.arange(n_pages)
    pool = kv.view(n_pages, page, -1)[torch.as_tensor(perm, device=kv.device)].reshape(kv.shape)
    pages_per_seq = n_rows // page
    table = np.stack([where[b * pages_per_seq:(b + 1) * pages_per_seq] for b in range(B)])
    logical = np.where(idx >= 0, idx - (np.arange(B)[:, None] * n_rows), -1)
    return w, kv, q, idx, pool.contiguous(), table.astype(np.int32), logical.astype(np.int32)


@pytest.mark.parametrize("H,k,page", [(64, 300, 16), (16, 129, 64), (128, 64, 1)])
def test_paged_equals_flat_and_oracle(H, k, page):
    B, n_rows = 3, 2048
    w, kv, q, idx, pool, table, logical = _paged(B, H, n_rows, k, page, seed=400 + H + page)
    logical[1, 10:40] = -1
    idx = idx.copy()
    idx[1, 10:40] = -1
    out_p, lse_p = sparse_mla_decode_paged(q, pool, torch.as_tensor(table, device="cuda"), page,
                                           torch.as_tensor(logical, device="cuda"))
    out_f, lse_f = sparse_mla_decode(q, kv, torch.as_tensor(idx, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_f) and torch.equal(lse_p, lse_f)
    ref_out, ref_lse = oracle_decode(q, kv, idx)
    assert_out_close(out_p.float().cpu().numpy(), ref_out)
    assert_lse_close(lse_p.cpu().numpy(), ref_lse)


def test_unmapped_pages_and_positions_past_the_table():
    B, H, n_rows, k, page = 2, 64, 1024, 200, 32
    w, kv, q, idx, pool, table, logical = _paged(B, H, n_rows, k, page, seed=431)
    table[0, 3] = -1                               # an unmapped page: its positions masked
    idx = idx.copy()
    on_page3 = (logical[0] // page) == 3
    idx[0, on_page3 & (logical[0] >= 0)] = -1
    smla_device_status(clear=True)
    out_p, lse_p = sparse_mla_decode_paged(q, pool, torch.as_tensor(table, device="cuda"), page,
                                           torch.as_tensor(logical, device="cuda"))
    assert smla_device_status(clear=True) == 0
    ref_out, ref_lse = oracle_decode(q, kv, idx)
    assert_out_close(out_p.float().cpu().numpy(), ref_out)
    assert_lse_close(lse_p.cpu().numpy(), ref_lse)
    # a position past the block table is masked and reported
    logical2 = logical.copy()
    logical2[1, 0] = table.shape[1] * page + 5
    idx2 = idx.copy()
    idx2[1, 0] = -1
    out2, lse2 = sparse_mla_decode_paged(q, pool, torch.as_tensor(table, device="cuda"), page,
                                         torch.as_tensor(logical2, device="cuda"))
    assert smla_device_status(clear=True) == -7
    ref_out2, ref_lse2 = oracle_decode(q, kv, idx2)
    assert_out_close(out2.float().cpu().numpy(), ref_out2)
