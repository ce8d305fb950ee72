"""Element-wise parity of the CUDA path (through the C ABI) with the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle.mla_oracle as O
from sparse_mla_decode_03_gb300 import (sparse_mla_combine, sparse_mla_decode,
                                        sparse_mla_decode_split, smla_device_status)
from sparse_mla_decode_03_gb300 import workloads as W

from _helpers import (SCALE, assert_lse_close, assert_out_close, oracle_decode,
                      oracle_deviation, oracle_split, small_case)

pytestmark = pytest.mark.gpu


def _run(q, kv, idx_np, **kw):
    idx = torch.as_tensor(np.ascontiguousarray(idx_np), dtype=torch.int32, device="cuda")
    out, lse = sparse_mla_decode(q, kv, idx, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


# ---------------------------------------------------------------------------
# small shapes: several tiles, ragged tails, every head count
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H", [16, 32, 64, 128])
@pytest.mark.parametrize("k", [1, 17, 128, 129, 300])
def test_decode_small(H, k):
    w, kv, q, idx = small_case(2, H, 700, k, seed=100 + H + k)
    out, lse = _run(q, kv, idx)
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("S", [1, 2, 3, 7])
def test_split_partials_match_oracle(S):
    w, kv, q, idx = small_case(3, 64, 900, 333, seed=7)
    idx[1, 40:200] = -1
    o_part, lse_part = sparse_mla_decode_split(q, kv, torch.as_tensor(idx, device="cuda"), S)
    torch.cuda.synchronize()
    ro, rl = oracle_split(q, kv, idx, S)
    assert_out_close(o_part.cpu().numpy(), ro)
    assert_lse_close(lse_part.cpu().numpy(), rl)


@pytest.mark.parametrize("S", [1, 2, 5, 16])
def test_explicit_splits_same_result(S):
    w, kv, q, idx = small_case(2, 64, 4000, 1000, seed=8)
    out, lse = _run(q, kv, idx, num_splits=S)
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_masked_slots_and_empty_queries():
    w, kv, q, idx = small_case(4, 64, 600, 256, seed=9)
    idx = idx.copy()
    idx[0, ::3] = -1                 # interleaved
    idx[1, 100:] = -1                # tail
    idx[2, :] = -1                   # nothing valid
    idx[3, :130] = -1                # whole first tile masked
    out, lse = _run(q, kv, idx, num_splits=2)
    ro, rl = oracle_decode(q, kv, idx)
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_minus_one_padding_equals_shorter_list():
    w, kv, q, idx = small_case(2, 64, 800, 200, seed=10)
    short = idx[:, :150]
    padded = np.concatenate([short, -np.ones((2, 250), np.int32)], axis=1)
    o1, l1 = _run(q, kv, short)
    o2, l2 = _run(q, kv, padded)
    ro, rl = oracle_decode(q, kv, short)
    assert_out_close(o1, ro)
    assert_out_close(o2, ro)
    assert_lse_close(l2, rl)


def test_permutation_changes_nothing_beyond_tolerance():
    w, kv, q, idx = small_case(2, 64, 3000, 1024, seed=11)
    perm = idx[:, np.random.default_rng(0).permutation(idx.shape[1])]
    o1, l1 = _run(q, kv, idx)
    o2, l2 = _run(q, kv, perm)
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(o1, ro)
    assert_out_close(o2, ro)
    assert np.max(np.abs(o1 - o2)) <= 2e-2


def test_pad_byte_ff_and_outliers():
    w, kv, q, idx = small_case(2, 64, 1000, 512, seed=12, outliers=0.01, pad_byte=0xFF)
    out, lse = _run(q, kv, idx)
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out, ro, strict_abs=False, D=oracle_deviation(q, kv, idx))
    assert_lse_close(lse, rl)


def test_dense_top_k_covers_every_row():
    w, kv, q, _ = small_case(1, 64, 512, 512, seed=13)
    idx = np.random.default_rng(1).permutation(512)[None].astype(np.int32)
    out, lse = _run(q, kv, idx)
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_single_row_closed_form():
    """k = 1: the output is the dequantised row itself (exact in bf16)."""
    w, kv, q, _ = small_case(1, 64, 64, 1, seed=14)
    idx = np.array([[37]], np.int32)
    out, lse = _run(q, kv, idx)
    nope, _ = O.dequantize_rows(kv[37:38].cpu().numpy())
    assert np.array_equal(out[0], np.broadcast_to(nope[0], out[0].shape))


def test_kv_row_stride_larger_than_row():
    w, kv, q, idx = small_case(2, 64, 500, 200, seed=15)
    wide = torch.zeros((kv.shape[0], 640), dtype=torch.uint8, device="cuda")
    wide[:, :584] = kv
    wide[:, 584:] = 0xFF
    out, lse = _run(q, wide, idx)
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def _padded_cache(kv, stride):
    wide = torch.full((kv.shape[0], stride), 0xFF, dtype=torch.uint8, device="cuda")
    wide[:, :584] = kv
    return wide


@pytest.mark.parametrize("H", [64, 16])
@pytest.mark.parametrize("stride,n", [(584, 501), (584, 500), (584, 2), (584, 1), (600, 333),
                                      (592, 257), (640, 3)])
def test_rows_at_the_cache_edges(stride, n, H):
    """The first and last rows of the cache, of both parities, under each row stride the
    gather treats differently (a multiple of 16 bytes or 8 past one, odd and even row
    counts): the last row of an odd-sized cache ends exactly at the cache's end."""
    w, kv, q0, _ = small_case(1, H, n, 1, seed=stride + n + H)     # a cache of n rows
    q = torch.cat([q0, small_case(1, H, 1, 1, seed=stride + n + H + 1)[2]])
    assert kv.shape[0] == n
    rng = np.random.default_rng(n)
    k = min(n, 150)
    rest = [r for r in rng.permutation(n).tolist() if r not in (0, n - 1)]
    row0 = ([0, n - 1] if n > 1 else [0]) + rest[: k - min(n, 2)]
    idx = np.full((2, k), -1, np.int32)
    idx[0] = rng.permutation(np.array(row0, np.int32))
    idx[1, -1] = n - 1                      # one valid slot: the last row, in the last block
    out, lse = _run(q, _padded_cache(kv, stride), idx)
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("offset,stride", [(16, 584), (48, 584), (16, 592)])
def test_cache_view_at_a_16_byte_offset(offset, stride):
    """A cache that starts 16 or 48 bytes into its allocation (16-byte aligned, as the
    ABI requires, but not 256): the row maps and the odd-row map's shifted base are
    then not at an allocation boundary."""
    w, kv, q, idx = small_case(2, 64, 333, 150, seed=offset + stride)
    n = kv.shape[0]
    buf = torch.full((offset + n * stride,), 0xFF, dtype=torch.uint8, device="cuda")
    view = buf[offset:].view(n, stride)
    view[:, :584] = kv
    assert view.data_ptr() % 16 == 0 and view.data_ptr() % 256 != 0
    idx = idx.copy()
    idx[0, :2] = [0, n - 1]          # first and last rows of the view
    out, lse = _run(q, view, idx)
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("pattern", ["even", "odd", "one_odd", "alternating", "three_even"])
def test_gather_groups_by_row_parity(pattern):
    """Blocks whose rows are all of one parity, or split 63 / 1, 61 / 3 or evenly:
    every way the gather's groups of four can be filled and padded."""
    w, kv, q, _ = small_case(2, 64, 2048, 1, seed=77)
    n = kv.shape[0]
    rng = np.random.default_rng(5)
    ev, od = rng.permutation(np.arange(0, n, 2)), rng.permutation(np.arange(1, n, 2))
    k = 320
    if pattern == "even":
        row = ev[:k]
    elif pattern == "odd":
        row = od[:k]
    elif pattern == "one_odd":          # per block of 64: 63 even, 1 odd
        row = np.concatenate([np.concatenate([ev[63 * b:63 * b + 63], od[b:b + 1]]) for b in range(5)])
    elif pattern == "three_even":       # per block: 3 even, 61 odd
        row = np.concatenate([np.concatenate([od[61 * b:61 * b + 61], ev[3 * b:3 * b + 3]]) for b in range(5)])
    else:
        row = np.stack([ev[:k // 2], od[:k // 2]], axis=1).reshape(-1)
    idx = np.stack([row, row[::-1]]).astype(np.int32)
    out, lse = _run(q, kv, idx, num_splits=1)        # blocks = slots 64b .. 64b + 63
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_deterministic():
    w, kv, q, idx = small_case(4, 64, 5000, 2048, seed=16)
    o1, l1 = _run(q, kv, idx)
    o2, l2 = _run(q, kv, idx)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_index_out_of_range_is_skipped_and_reported():
    w, kv, q, idx = small_case(1, 64, 300, 100, seed=17)
    smla_device_status(clear=True)
    bad = idx.copy()
    bad[0, 5] = kv.shape[0] + 10
    out, lse = _run(q, kv, bad)
    assert smla_device_status(clear=True) == -7
    masked = bad.copy()
    masked[0, 5] = -1
    ro, rl = oracle_decode(q, kv, masked)
    assert_out_close(out, ro)
    assert smla_device_status() == 0


# ---------------------------------------------------------------------------
# combine kernel against the oracle merge
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("S", [1, 2, 3, 6, 9, 33, 200])
def test_combine_matches_oracle(S):
    g = torch.Generator(device="cuda").manual_seed(S)
    B, H = 3, 16
    o = torch.randn((B, H, S, 448), generator=g, device="cuda")
    l = torch.randn((B, H, S), generator=g, device="cuda") * 5
    l[0, 0, :] = -float("inf")
    if S > 1:
        l[1, 2, 0] = -float("inf")
    out, lse = sparse_mla_combine(o, l)
    torch.cuda.synchronize()
    ro, rl = O.combine(o.double().cpu().numpy(), l.double().cpu().numpy())
    # random N(0,1) partials reach |o| ~ 4, where bf16's half-ulp alone is 0.0156
    assert_out_close(out.float().cpu().numpy(), ro, strict_abs=False)
    assert_lse_close(lse.cpu().numpy(), rl)


# ---------------------------------------------------------------------------
# the five workload shapes, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("key", ["c1", "c2", "c3", "c4", "c5"])
def test_workload_parity(key):
    w = W.WORKLOADS[key]
    L = W.seq_lengths(w)
    kv = W.make_cache(w, L, device="cuda")
    q = W.make_q(w, device="cuda")
    idx = W.make_indices(w, L)
    out, lse = _run(q, kv, idx)
    queries = range(w.batch)        # every query of every workload
    ro, rl = oracle_decode(q, kv, idx, queries=queries)
    sel = list(queries)
    if w.outlier_frac == 0:
        assert_out_close(out[sel], ro)
    else:
        D = oracle_deviation(q, kv, idx, queries=queries)
        assert_out_close(out[sel], ro, strict_abs=False, D=D)
    assert_lse_close(lse[sel], rl)
    del kv
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# the largest accepted top-k: every row of a 65536-row sequence selected
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("S", [0, 8])   # default plan (split + combine kernels) / cluster merge
def test_maximum_topk_every_row(S):
    w, kv, q, idx_np = small_case(1, 64, 65536, 65536, seed=31)
    assert idx_np.shape == (1, 65536) and np.array_equal(np.sort(idx_np[0]), np.arange(65536))
    out, lse = _run(q, kv, idx_np, num_splits=S)
    ro, rl = oracle_decode(q, kv, idx_np)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
    assert smla_device_status() == 0
