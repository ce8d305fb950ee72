"""What an FP8 score path (block-scaled e4m3 QK, the next step after the f16 kernel)
would do to the results: q rounded to e4m3 with one UE8M0 scale per 32 values, the
format "The Power-of-Two Trap: Debugging a Triton MMA Kernel on Blackwell GPUs"
(sections "3. The Scale Indexing Complication" and "Input Knowledge Required")
uses for the cache, applied to the query.

Measured on the float64 oracle (`attend`) over synthetic workload rows:
  - one e4m3 copy of q moves the LSE by more than the 1e-3 parity bound;
  - a hi/lo pair of e4m3 copies (the low one quantising the residual with its own
    block scales) reproduces the bf16 q, so the scores are unchanged.
These pin the precision argument recorded for the FP8 variant; no kernel runs."""
import numpy as np
import torch

import oracle.mla_oracle as O
from sparse_mla_decode_03_gb300 import workloads as W


def _e4m3(x: np.ndarray) -> np.ndarray:
    t = torch.as_tensor(np.clip(x, -448.0, 448.0), dtype=torch.float32)
    return t.to(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def _quant_blocks(q: np.ndarray, blk: int = 32) -> np.ndarray:
    """e4m3 with a UE8M0 scale 2^ceil(log2(amax / 448)) per block of 32 values."""
    qb = q.reshape(*q.shape[:-1], -1, blk)
    amax = np.abs(qb).max(-1, keepdims=True)
    sc = np.exp2(np.ceil(np.log2(np.maximum(amax, 1e-300) / 448.0)))
    return (_e4m3(qb / sc) * sc).reshape(q.shape)


def _case(heads: int, seed: int):
    w = W.Workload("fp8q", 1, heads, 1024, 8192, "uniform", seed=seed)
    L = W.seq_lengths(w)
    kv = W.make_cache(w, L, device="cpu")
    q = W.make_q(w, device="cpu")[0].float().numpy().astype(np.float64)
    idx = W.make_indices(w, L)
    rows, remap = W.compact_rows(kv, idx)
    kn, kr = O.dequantize_rows(rows[remap[0]])
    return q, kn, kr, w.softmax_scale


def test_one_e4m3_copy_of_q_breaks_the_lse_bound():
    worst = 0.0
    for heads, seed in ((16, 11), (64, 12)):
        q, kn, kr, scale = _case(heads, seed)
        _, ref_l = O.attend(q, kn, kr, scale)
        _, l = O.attend(_quant_blocks(q), kn, kr, scale)
        worst = max(worst, np.abs(l - ref_l).max())
    assert worst > 1e-3, worst


def test_hi_lo_pair_of_e4m3_copies_reproduces_q():
    for heads, seed in ((16, 11), (64, 12)):
        q, kn, kr, scale = _case(heads, seed)
        hi = _quant_blocks(q)
        lo = _quant_blocks(q - hi)
        assert np.abs(hi + lo - q).max() <= 1e-6 * np.abs(q).max()
        ref_o, ref_l = O.attend(q, kn, kr, scale)
        o, l = O.attend(hi + lo, kn, kr, scale)
        assert np.abs(l - ref_l).max() < 1e-6
        assert np.abs(o - ref_o).max() < 1e-6
