"""Branches of the online softmax that random workloads do not reach.

The kernel raises its running max lazily: only when a score passes it by 2^15 (in
log2 units) does it take the exact block max and rescale O and the denominator in
tensor memory.  With N(0, 1) data the first block sets a max that later blocks never
pass by that much, so these tests build scores that grow along the index list by
tens of nats (the query's rope times a growing multiple of it in each row's rope),
which makes many blocks raise the max, on one split so the state runs through all
blocks.  They also cover a first block whose only valid tokens are its second half
(one softmax thread of a head sees none), and fully masked blocks between valid ones.
Both softmax forms run: 64 heads (Q in tensor memory) and 16 heads (Q in shared
memory).  Each result is compared with the float64 oracle."""
import numpy as np
import pytest
import torch

from sparse_mla_decode_03_gb300 import smla_device_status, sparse_mla_decode
from sparse_mla_decode_03_gb300 import workloads as W

import oracle.mla_oracle as O

from _helpers import SCALE, assert_lse_close, assert_out_close, oracle_decode

LAZY_HEADROOM_LOG2 = 15.0   # the kernel raises its running max past this headroom


def _raises(q, kv, idx_row) -> int:
    """How many times a running max started at the first valid token's block would
    be passed by more than the headroom (head 0, log2 units, 64-token blocks)."""
    rows = kv.cpu().numpy()
    kn, kr = O.dequantize_rows(rows)
    qf = q[0, 0].float().numpy().astype(np.float64)
    s = SCALE * (kn @ qf[:448] + kr @ qf[448:]) / np.log(2.0)
    m, n = None, 0
    for b0 in range(0, len(idx_row), 64):
        blk = [int(i) for i in idx_row[b0:b0 + 64] if i >= 0]
        if not blk:
            continue
        bm = s[blk].max()
        if m is None:
            m = bm
        elif bm > m + LAZY_HEADROOM_LOG2:
            m, n = bm, n + 1
    return n


pytestmark = pytest.mark.gpu


def _rows_with_growing_scores(n: int, q_rope: np.ndarray, lo: float, hi: float, seed: int):
    """n cache rows: nope from the workload recipe; rope of row t = a_t * q_rope with
    a_t chosen so that the head-0 score of row t (scaled) rises linearly lo..hi."""
    w = W.Workload("grow", 1, 64, 64, n, "uniform", seed=seed)
    L = W.seq_lengths(w)
    kv = W.make_cache(w, L, device="cpu").numpy().copy()
    norm2 = float(np.dot(q_rope, q_rope))
    for t in range(n):
        a = (lo + (hi - lo) * t / (n - 1)) / (SCALE * norm2)
        rope = torch.as_tensor(a * q_rope, dtype=torch.float32).to(torch.bfloat16)
        kv[t, W.ROPE_OFF:] = rope.view(torch.uint8).numpy()
    return kv


def _query(H: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((1, H, 512), generator=g) * 0.05        # small nope part
    q[0, :, 448:] = torch.randn((64,), generator=g)          # one rope direction, all heads
    return q.to(torch.bfloat16)


@pytest.mark.parametrize("H", [64, 16])
@pytest.mark.parametrize("order", ["rising", "falling"])
def test_running_max_raised_many_times(H, order):
    q = _query(H, seed=31 + H)
    q_rope = q[0, 0, 448:].float().numpy().astype(np.float64)
    n = 1024
    kv = torch.as_tensor(_rows_with_growing_scores(n, q_rope, -20.0, 60.0, seed=7), device="cuda")
    idx = np.arange(n, dtype=np.int32)
    if order == "falling":
        idx = idx[::-1].copy()
    idx = idx[None]
    # rising scores make the running max be raised (O rescaled) several times
    assert _raises(q, kv, idx[0]) >= (4 if order == "rising" else 0)
    smla_device_status(clear=True)
    out, lse = sparse_mla_decode(q.cuda(), kv, torch.as_tensor(idx, device="cuda"), num_splits=1)
    torch.cuda.synchronize()
    assert smla_device_status() == 0
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out.float().cpu().numpy(), ro)
    assert_lse_close(lse.cpu().numpy(), rl)


@pytest.mark.parametrize("H", [64, 16])
def test_first_valid_tokens_in_second_half_and_masked_blocks(H):
    q = _query(H, seed=41 + H)
    q_rope = q[0, 0, 448:].float().numpy().astype(np.float64)
    n = 640
    kv = torch.as_tensor(_rows_with_growing_scores(n, q_rope, -5.0, 40.0, seed=8), device="cuda")
    idx = np.arange(n, dtype=np.int32)
    idx[:32] = -1            # block 0: tokens 0..31 masked, 32..63 valid
    idx[64:192] = -1         # blocks 1 and 2 fully masked
    idx[400:464] = -1        # another fully masked block, after valid ones
    idx = idx[None]
    assert _raises(q, kv, idx[0]) >= 2
    smla_device_status(clear=True)
    out, lse = sparse_mla_decode(q.cuda(), kv, torch.as_tensor(idx, device="cuda"), num_splits=1)
    torch.cuda.synchronize()
    assert smla_device_status() == 0
    ro, rl = oracle_decode(q, kv, idx)
    assert_out_close(out.float().cpu().numpy(), ro)
    assert_lse_close(lse.cpu().numpy(), rl)
