"""CPU float64 oracle for sparse Multi-head Latent Attention (MLA) decode.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this module: only the tests, the smoke check and the benchmark's CPU-baseline leg
do.  It shares no code, constants or tables with the CUDA path.

What it computes (the plain definition of the method, written out step by step):

The pages describe sparse MLA decode in which every query head of one decode
token attends over the same top-k selected KV-cache rows ("The Moment of
Compilation: When a Triton Kernel Meets Its Constraints", section "The Context: A
Kernel Optimization Campaign": one shared read of the KV rows for all heads, scores
for all heads as one batched product).  Each row holds a 448-wide FP8 "nope" part
with per-64-column UE8M0 scales and a 64-wide bf16 "rope" part ("The Power-of-Two
Trap: Debugging a Triton MMA Kernel on Blackwell GPUs", sections "3. The Scale
Indexing Complication" and "Input Knowledge Required").  For query b and head h:

    k_nope[t, c] = e4m3(row_t[c]) * 2**(row_t[448 + c // 64] - 127)      c < 448
    k_rope[t, j] = bf16(row_t[456 + 2j : 458 + 2j])                       j < 64
    s[t]  = scale * (q[h, :448] . k_nope[t] + q[h, 448:] . k_rope[t])
    lse   = log(sum_t exp(s[t]))                       (natural log)
    out   = sum_t exp(s[t] - lse) * k_nope[t]          (448 wide: only the nope
                                                         part is the value vector)

over the set of valid (index >= 0) top-k positions of query b.  With no valid
position, out = 0 and lse = -inf.  The 448 -> 512 zero padding the pages use
("2. The Padding Strategy") changes nothing in this definition: padded columns are
zero in both operands and the pad scale byte never takes part.

Readings taken where the pages are silent (all listed in the design notes):
row byte order as above; UE8M0 = 2**(byte - 127) with 0xFF = NaN (OCP MX); V is the
dequantised nope part; the natural-log LSE is of the *scaled* scores; split-K
partials merge by the standard log-sum-exp weighting.

Parity pins: every function here is checked in tests/test_oracle_pins.py against
something other than itself (library decoders, dense softmax attention written
with torch ops, closed forms, brute force on tiny inputs, invariances).
"""
from __future__ import annotations

import math

import numpy as np

# Row layout (the oracle's own copy; see the module docstring).
NOPE_DIM = 448
ROPE_DIM = 64
GROUP_COLS = 64
NUM_GROUPS = NOPE_DIM // GROUP_COLS      # 7
SCALE_BYTE0 = 448
PAD_BYTE = 455
ROPE_BYTE0 = 456
ROW_END = 584


# ---------------------------------------------------------------------------
# Element decoders
# ---------------------------------------------------------------------------
def e4m3_to_float(byte: int) -> float:
    """Value of one OCP FP8 E4M3 ("fn": finite, no infinities) byte.

    Sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.  Exponent 0 is
    subnormal (2**-6 * m/8); the pattern S.1111.111 is NaN; there is no infinity.
    The pages name the format FP8 ("Input Knowledge Required", item 3)."""
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m / 8.0, -6)
    return s * math.ldexp(1.0 + m / 8.0, e - 7)


E4M3_TABLE = np.array([e4m3_to_float(b) for b in range(256)], dtype=np.float64)


def ue8m0_to_float(byte: int) -> float:
    """Value of one UE8M0 scale byte: 2**(byte - 127); 0xFF is NaN (OCP MX E8M0).

    "Input Knowledge Required", item 3, of "The Power-of-Two Trap": unsigned
    exponent-only scale bytes shared by a group of 64 columns."""
    if byte == 0xFF:
        return math.nan
    return math.ldexp(1.0, byte - 127)


UE8M0_TABLE = np.array([ue8m0_to_float(b) for b in range(256)], dtype=np.float64)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact: bf16 is the top half of f32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Row dequantisation
# ---------------------------------------------------------------------------
def dequantize_rows(rows: np.ndarray):
    """Packed rows uint8 [n, >=584] -> (k_nope [n, 448], k_rope [n, 64]) float64.

    Column c of the nope part uses the scale byte of group c // 64 ("3. The Scale
    Indexing Complication": 7 groups of 64 columns plus one padding byte).  The
    padding byte at offset 455 is never read."""
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    fp8 = E4M3_TABLE[rows[:, :NOPE_DIM]]                                   # [n, 448]
    scales = UE8M0_TABLE[rows[:, SCALE_BYTE0:SCALE_BYTE0 + NUM_GROUPS]]    # [n, 7]
    group_of_col = np.arange(NOPE_DIM) // GROUP_COLS                       # [448]
    k_nope = fp8 * scales[:, group_of_col]
    rope_bytes = np.ascontiguousarray(rows[:, ROPE_BYTE0:ROW_END])          # [n, 128]
    rope_bits = rope_bytes.view("<u2").reshape(n, ROPE_DIM)
    k_rope = bf16_bits_to_float(rope_bits)
    return k_nope, k_rope


# ---------------------------------------------------------------------------
# Attention over one set of rows
# ---------------------------------------------------------------------------
def attend(q: np.ndarray, k_nope: np.ndarray, k_rope: np.ndarray, scale: float):
    """Exact softmax attention of H query heads over n rows, in float64.

    q [H, 512] (448 nope | 64 rope), k_nope [n, 448], k_rope [n, 64].
    Returns out [H, 448] and lse [H] (natural log of the sum of exp(scaled scores)).
    n == 0 gives out = 0, lse = -inf."""
    q = np.asarray(q, dtype=np.float64)
    H = q.shape[0]
    n = k_nope.shape[0]
    if n == 0:
        return np.zeros((H, NOPE_DIM)), np.full(H, -np.inf)
    # scores for all heads against all rows: one batched product
    s = scale * (q[:, :NOPE_DIM] @ k_nope.T + q[:, NOPE_DIM:] @ k_rope.T)   # [H, n]
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    l = w.sum(axis=1, keepdims=True)
    lse = (m + np.log(l))[:, 0]
    out = (w / l) @ k_nope                                                  # V = nope
    return out, lse


def _valid_rows(kv: np.ndarray, idx_row: np.ndarray) -> np.ndarray:
    sel = np.asarray(idx_row, dtype=np.int64)
    sel = sel[sel >= 0]
    return kv[sel]


def sparse_mla_decode(q_bits: np.ndarray, kv: np.ndarray, indices: np.ndarray,
                      scale: float):
    """Whole decode step.

    q_bits  uint16 [B, H, 512]   bf16 bit patterns of the queries
    kv      uint8  [R, >=584]    packed cache rows
    indices int    [B, k]        row ids into kv, < 0 = masked (shared by all heads)
    Returns out float64 [B, H, 448], lse float64 [B, H]."""
    q = bf16_bits_to_float(q_bits)
    B, H, _ = q.shape
    out = np.zeros((B, H, NOPE_DIM))
    lse = np.zeros((B, H))
    for b in range(B):
        k_nope, k_rope = dequantize_rows(_valid_rows(kv, indices[b]))
        out[b], lse[b] = attend(q[b], k_nope, k_rope, scale)
    return out, lse


def weighted_deviation(q_bits: np.ndarray, kv: np.ndarray, indices: np.ndarray,
                       scale: float) -> np.ndarray:
    """D[b, h, c] = sum_t w_t |k_nope[t, c] - out[b, h, c]|, w_t = exp(s_t - lse).

    Not part of the method: it sizes the forward error of any implementation that
    rounds the attention weights to a p-bit format before the weighted sum.  With
    each weight perturbed by a relative eps_t and renormalised, the output moves by
    sum_t w_t eps_t (k_nope[t] - out), so |error| <= max|eps| * D to first order."""
    q = bf16_bits_to_float(q_bits)
    B, H, _ = q.shape
    D = np.zeros((B, H, NOPE_DIM))
    for b in range(B):
        k_nope, k_rope = dequantize_rows(_valid_rows(kv, indices[b]))
        if k_nope.shape[0] == 0:
            continue
        s = scale * (q[b, :, :NOPE_DIM] @ k_nope.T + q[b, :, NOPE_DIM:] @ k_rope.T)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        out = w @ k_nope
        D[b] = np.einsum("ht,htc->hc", w, np.abs(k_nope[None, :, :] - out[:, None, :]))
    return D


# ---------------------------------------------------------------------------
# Split-K over the top-k positions, and the merge of partials
# ---------------------------------------------------------------------------
def split_ranges(topk: int, num_splits: int):
    """Positions [t0, t1) of each split: the top-k list is cut into 16-token
    granules and split s takes granules [s*G // S, (s+1)*G // S), G = ceil(topk/16).
    A split may be empty when S > G."""
    G = (topk + 15) // 16
    res = []
    for s in range(num_splits):
        g0 = (s * G) // num_splits
        g1 = ((s + 1) * G) // num_splits
        res.append((min(16 * g0, topk), min(16 * g1, topk)))
    return res


def split_partials(q_bits, kv, indices, scale, num_splits):
    """Per-split normalised partials: o_part [B, H, S, 448], lse_part [B, H, S].

    Split s attends only over positions split_ranges(k, S)[s] of each index list
    (the split-K partition of "The 80KB Mystery: Resolving Contradictory Evidence in
    Triton Kernel Optimization", section "The Context: Optimizing Attention on
    Blackwell")."""
    q = bf16_bits_to_float(q_bits)
    B, H, _ = q.shape
    k = indices.shape[1]
    o = np.zeros((B, H, num_splits, NOPE_DIM))
    l = np.zeros((B, H, num_splits))
    for b in range(B):
        for s, (t0, t1) in enumerate(split_ranges(k, num_splits)):
            k_nope, k_rope = dequantize_rows(_valid_rows(kv, indices[b, t0:t1]))
            o[b, :, s], l[b, :, s] = attend(q[b], k_nope, k_rope, scale)
    return o, l


def combine(o_part: np.ndarray, lse_part: np.ndarray):
    """Merge split partials: lse = log sum_s exp(lse_s); out = sum_s exp(lse_s - lse) o_s.

    Splits with lse_s = -inf carry no weight; if every split is empty the result
    is out = 0, lse = -inf."""
    o_part = np.asarray(o_part, dtype=np.float64)
    lse_part = np.asarray(lse_part, dtype=np.float64)
    m = lse_part.max(axis=-1, keepdims=True)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_part), np.exp(lse_part - m_safe), 0.0)
    tot = w.sum(axis=-1, keepdims=True)
    lse = np.where(finite, m_safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)[..., 0]
    wn = np.where(tot > 0, w / np.where(tot > 0, tot, 1.0), 0.0)
    out = (wn[..., None] * o_part).sum(axis=-2)
    return out, lse
