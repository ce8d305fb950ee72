"""Sanity of the seeded input generators (shapes, index laws, row bytes)."""
import numpy as np
import torch

from sparse_mla_decode_03_gb300 import workloads as W


def test_index_laws():
    for key in ("c1", "c2", "c3"):
        w = W.WORKLOADS[key]
        L = W.seq_lengths(w)
        idx = W.make_indices(w, L)
        assert idx.shape == (w.batch, w.topk) and idx.dtype == np.int32
        bases = W.seq_bases(L)
        for b in range(w.batch):
            pos = idx[b].astype(np.int64) - bases[b]
            assert len(set(pos.tolist())) == w.topk
            assert pos.min() >= 0 and pos.max() < L[b]
            if w.index_law == "recent_half":
                assert (pos >= L[b] - 4096).sum() >= w.topk // 2
    # a second variant is a different draw
    w = W.WORKLOADS["c2"]
    L = W.seq_lengths(w)
    assert not np.array_equal(W.make_indices(w, L, 0), W.make_indices(w, L, 1))


def test_ragged_tail_is_minus_one():
    w = W.Workload("r", 6, 4, 2048, 0, "ragged", ragged_lo=100, ragged_hi=3000, seed=9)
    L = W.seq_lengths(w)
    idx = W.make_indices(w, L)
    bases = W.seq_bases(L)
    for b in range(w.batch):
        n = min(2048, int(L[b]))
        assert np.all(idx[b, n:] == -1)
        pos = idx[b, :n].astype(np.int64) - bases[b]
        assert len(set(pos.tolist())) == n and pos.min() >= 0 and pos.max() < L[b]


def test_rows_well_formed():
    w = W.Workload("t", 2, 4, 64, 300, "uniform", outlier_frac=0.01, seed=3)
    kv = W.make_cache(w, W.seq_lengths(w), pad_byte=0xAB)
    assert kv.shape == (600, 584) and kv.dtype == torch.uint8
    s = kv[:, 448:455]
    assert int(s.min()) >= 1 and int(s.max()) <= 254
    assert torch.all(kv[:, 455] == 0xAB)
    fp8 = kv[:, :448]
    assert not torch.any((fp8 & 0x7F) == 0x7F)          # no NaN pattern
    q = W.make_q(w)
    assert q.shape == (2, 4, 512) and q.dtype == torch.bfloat16
