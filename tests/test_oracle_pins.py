"""Pins for the CPU float64 oracle: each check compares the oracle with something
other than itself -- a library decoder, dense softmax attention written with torch
ops, a closed form, a brute-force scalar loop or an invariance the method must
have.  A planted-mistake section shows the pins catch plausible errors."""
import math

import numpy as np
import pytest
import torch

import oracle.mla_oracle as O
from sparse_mla_decode_03_gb300 import workloads as W

SCALE = 1.0 / math.sqrt(512)


# ---------------------------------------------------------------------------
# helpers: a tiny synthetic cache and an independent torch reference
# ---------------------------------------------------------------------------
def tiny_inputs(B=2, H=4, n_rows=256, k=None, seed=0, pad_byte=0, outliers=0.0):
    w = W.Workload("tiny", B, H, k or n_rows, n_rows, "uniform", outlier_frac=outliers,
                   seed=seed)
    lengths = W.seq_lengths(w)
    kv = W.make_cache(w, lengths, device="cpu", pad_byte=pad_byte)
    q = W.make_q(w, device="cpu")
    return w, kv.numpy(), W.bf16_bits(q), q


def torch_reference(q_bf16: torch.Tensor, kv_u8: torch.Tensor, idx: np.ndarray, scale: float,
                    pad_to_512: bool = False):
    """Dense softmax attention over the selected rows, written with torch ops only
    (torch's own fp8 / bf16 decoders, torch.softmax, torch.logsumexp)."""
    q = q_bf16.to(torch.float64)
    B, H, _ = q.shape
    outs, lses = [], []
    for b in range(B):
        sel = torch.as_tensor(idx[b][idx[b] >= 0], dtype=torch.long)
        rows = kv_u8[sel]
        fp8 = rows[:, :448].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
        ex = rows[:, 448:455].to(torch.int64) - 127
        scale_cols = torch.repeat_interleave(ex, 64, dim=1)
        nope = torch.ldexp(fp8, scale_cols.to(torch.float64))
        rope = rows[:, 456:584].contiguous().view(torch.bfloat16).to(torch.float64)
        qn, qr = q[b, :, :448], q[b, :, 448:]
        if pad_to_512:
            z = torch.zeros(nope.shape[0], 64, dtype=torch.float64)
            nope_p = torch.cat([nope, z], 1)
            qn = torch.cat([qn, torch.zeros(H, 64, dtype=torch.float64)], 1)
        else:
            nope_p = nope
        s = scale * (torch.einsum("hc,tc->ht", qn, nope_p) + torch.einsum("hc,tc->ht", qr, rope))
        if s.shape[1] == 0:
            outs.append(torch.zeros(H, 448, dtype=torch.float64))
            lses.append(torch.full((H,), -math.inf, dtype=torch.float64))
            continue
        p = torch.softmax(s, dim=1)
        outs.append(p @ nope)
        lses.append(torch.logsumexp(s, dim=1))
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


def perm_indices(B, n_rows, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(n_rows, size=k, replace=False) for _ in range(B)]).astype(np.int64)


# ---------------------------------------------------------------------------
# element decoders
# ---------------------------------------------------------------------------
def test_e4m3_table_matches_torch_decoder():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.E4M3_TABLE
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], ours[fin])


def test_e4m3_spec_values():
    # closed forms from the E4M3 bit definition
    assert O.e4m3_to_float(0x00) == 0.0
    assert O.e4m3_to_float(0x01) == 2.0 ** -9          # smallest subnormal
    assert O.e4m3_to_float(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert O.e4m3_to_float(0x08) == 2.0 ** -6          # smallest normal
    assert O.e4m3_to_float(0x38) == 1.0
    assert O.e4m3_to_float(0x7E) == 448.0              # largest finite
    assert O.e4m3_to_float(0xFE) == -448.0
    assert math.isnan(O.e4m3_to_float(0x7F)) and math.isnan(O.e4m3_to_float(0xFF))
    assert O.e4m3_to_float(0x80) == 0.0 and math.copysign(1, O.e4m3_to_float(0x80)) == -1


def test_ue8m0_table():
    for b in range(255):
        assert O.UE8M0_TABLE[b] == math.ldexp(1.0, b - 127)
    assert math.isnan(O.UE8M0_TABLE[255])
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        fin = ~np.isnan(ref)
        assert np.array_equal(np.isnan(ref), np.isnan(O.UE8M0_TABLE))
        assert np.array_equal(ref[fin], O.UE8M0_TABLE[fin])


def test_bf16_decoder_matches_torch():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_bits_to_float(bits), x.to(torch.float64).numpy())


# ---------------------------------------------------------------------------
# row dequantisation
# ---------------------------------------------------------------------------
def test_dequant_roundtrip_within_e4m3_bound():
    """Quantise known values with the cache writer, dequantise with the oracle: the
    error must stay inside e4m3 round-to-nearest bounds for *each* group's own
    scale (a wrong group index or offset blows the bound)."""
    g = torch.Generator().manual_seed(11)
    n = 512
    x = torch.randn(n, 448, generator=g)
    # give each group a very different magnitude so group mix-ups are visible
    mags = torch.tensor([1e-3, 1.0, 30.0, 1e-2, 500.0, 0.25, 7.0]).repeat_interleave(64)
    x = x * mags
    packed = W._quantise_block(x, pad_byte=0).numpy()
    rows = np.zeros((n, 584), np.uint8)
    rows[:, :456] = packed
    rope = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    rows[:, 456:] = rope.view(torch.uint8).numpy().reshape(n, 128)
    nope, rp = O.dequantize_rows(rows)
    xs = x.double().numpy()
    scale = np.repeat(np.ldexp(1.0, rows[:, 448:455].astype(np.int64) - 127), 64, axis=1)
    bound = np.maximum(2.0 ** -4 * np.abs(xs), 2.0 ** -10 * scale) * (1 + 1e-12)
    assert np.all(np.abs(nope - xs) <= bound)
    assert np.array_equal(rp, rope.double().numpy())


def test_pad_byte_never_used():
    rows = np.random.default_rng(5).integers(0, 256, size=(64, 584), dtype=np.uint8)
    rows[:, :448] = np.where((rows[:, :448] & 0x7F) == 0x7F, 0x7E, rows[:, :448])  # no NaN
    rows[:, 456:] = 0x3F                                                          # finite rope
    rows[:, 448:455] = np.clip(rows[:, 448:455], 100, 140)
    a = rows.copy(); a[:, 455] = 0
    b = rows.copy(); b[:, 455] = 0xFF
    na, ra = O.dequantize_rows(a)
    nb, rb = O.dequantize_rows(b)
    assert np.array_equal(na, nb) and np.array_equal(ra, rb)


# ---------------------------------------------------------------------------
# attention: dense equivalence and invariances
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("outliers", [0.0, 0.01])
def test_dense_equivalence(outliers):
    """top-k covering every cached token == dense softmax attention (torch)."""
    B, H, n = 2, 4, 256
    w, kv, qbits, q = tiny_inputs(B, H, n, seed=21, outliers=outliers)
    # each query covers its own sequence's rows, all of them, in random order
    idx = np.stack([b * n + np.random.default_rng(b).permutation(n) for b in range(B)])
    out, lse = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    ro, rl = torch_reference(q, torch.from_numpy(kv), idx, SCALE)
    assert np.max(np.abs(out - ro)) < 1e-12 * max(1.0, np.max(np.abs(ro)))
    assert np.max(np.abs(lse - rl)) < 1e-12


def test_permutation_invariance():
    B, H, n, k = 1, 8, 300, 97
    w, kv, qbits, q = tiny_inputs(B, H, n, seed=4)
    idx = perm_indices(B, n, k, 9)
    o1, l1 = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    idx2 = idx[:, np.random.default_rng(1).permutation(k)]
    o2, l2 = O.sparse_mla_decode(qbits, kv, idx2, SCALE)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def test_minus_one_padding_equals_shorter_list():
    B, H, n, m = 1, 4, 200, 37
    w, kv, qbits, q = tiny_inputs(B, H, n, seed=6)
    short = perm_indices(B, n, m, 2)
    padded = np.concatenate([short, -np.ones((B, 90), np.int64)], axis=1)
    inter = np.full((B, 2 * m + 5), -1, np.int64)
    inter[:, 1::2][:, :m] = short
    o1, l1 = O.sparse_mla_decode(qbits, kv, short, SCALE)
    o2, l2 = O.sparse_mla_decode(qbits, kv, padded, SCALE)
    o3, l3 = O.sparse_mla_decode(qbits, kv, inter, SCALE)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.max(np.abs(o1 - o3)) < 1e-12 and np.max(np.abs(l1 - l3)) < 1e-12


def test_zero_padding_448_to_512_changes_nothing():
    """Appending 64 zero columns to q_nope and k_nope (and a 0xFF pad scale byte)
    leaves scores and outputs unchanged ("2. The Padding Strategy")."""
    B, H, n = 1, 4, 128
    w, kv, qbits, q = tiny_inputs(B, H, n, seed=8, pad_byte=0xFF)
    idx = perm_indices(B, n, n, 3)
    out, lse = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    ro, rl = torch_reference(q, torch.from_numpy(kv), idx, SCALE, pad_to_512=True)
    assert np.max(np.abs(out - ro)) < 1e-12 and np.max(np.abs(lse - rl)) < 1e-12


def test_all_masked_gives_zero_and_neg_inf():
    w, kv, qbits, q = tiny_inputs(2, 4, 64, seed=1)
    idx = -np.ones((2, 32), np.int64)
    out, lse = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def _scores_by_hand(qv, nope, rope, scale):
    return scale * (float(np.dot(qv[:448], nope)) + float(np.dot(qv[448:], rope)))


def test_closed_form_single_row():
    w, kv, qbits, q = tiny_inputs(1, 3, 64, seed=2)
    idx = np.array([[17]])
    out, lse = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    nope, rope = O.dequantize_rows(kv[[17]])
    qf = q.to(torch.float64).numpy()[0]
    for h in range(3):
        assert np.array_equal(out[0, h], nope[0])
        assert abs(lse[0, h] - _scores_by_hand(qf[h], nope[0], rope[0], SCALE)) < 1e-12


def test_closed_form_two_rows_sigmoid():
    w, kv, qbits, q = tiny_inputs(1, 2, 64, seed=3)
    idx = np.array([[5, 40]])
    out, lse = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    nope, rope = O.dequantize_rows(kv[[5, 40]])
    qf = q.to(torch.float64).numpy()[0]
    for h in range(2):
        s1 = _scores_by_hand(qf[h], nope[0], rope[0], SCALE)
        s2 = _scores_by_hand(qf[h], nope[1], rope[1], SCALE)
        a = 1.0 / (1.0 + math.exp(s2 - s1))
        assert np.max(np.abs(out[0, h] - (a * nope[0] + (1 - a) * nope[1]))) < 1e-12
        big = max(s1, s2)
        assert abs(lse[0, h] - (big + math.log(math.exp(s1 - big) + math.exp(s2 - big)))) < 1e-12


def test_weighted_deviation_closed_forms():
    """Two rows: D = 2 w1 w2 |v1 - v2|; identical rows: D = 0."""
    w, kv, qbits, q = tiny_inputs(1, 2, 64, seed=3)
    idx = np.array([[5, 40]])
    D = O.weighted_deviation(qbits, kv, idx, SCALE)
    nope, rope = O.dequantize_rows(kv[[5, 40]])
    qf = q.to(torch.float64).numpy()[0]
    for h in range(2):
        s1 = _scores_by_hand(qf[h], nope[0], rope[0], SCALE)
        s2 = _scores_by_hand(qf[h], nope[1], rope[1], SCALE)
        a = 1.0 / (1.0 + math.exp(s2 - s1))
        assert np.max(np.abs(D[0, h] - 2 * a * (1 - a) * np.abs(nope[0] - nope[1]))) < 1e-12
    kv2 = np.repeat(kv[[3]], 20, axis=0)
    assert np.all(O.weighted_deviation(qbits, kv2, np.arange(20)[None], SCALE) < 1e-12)


def test_closed_form_zero_query_is_mean():
    w, kv, _, _ = tiny_inputs(1, 2, 100, seed=4)
    qbits = np.zeros((1, 2, 512), np.uint16)
    idx = perm_indices(1, 100, 60, 4)
    out, lse = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    nope, _ = O.dequantize_rows(kv[idx[0]])
    assert np.max(np.abs(out[0] - nope.mean(0))) < 1e-12
    assert np.max(np.abs(lse - math.log(60))) < 1e-12


def test_closed_form_identical_rows():
    w, kv, qbits, q = tiny_inputs(1, 4, 16, seed=5)
    kv2 = np.repeat(kv[[3]], 50, axis=0)
    idx = np.arange(50)[None]
    out, lse = O.sparse_mla_decode(qbits, kv2, idx, SCALE)
    nope, rope = O.dequantize_rows(kv2[:1])
    qf = q.to(torch.float64).numpy()[0]
    for h in range(4):
        assert np.max(np.abs(out[0, h] - nope[0])) < 1e-12
        s = _scores_by_hand(qf[h], nope[0], rope[0], SCALE)
        assert abs(lse[0, h] - (s + math.log(50))) < 1e-12


def test_brute_force_tiny():
    """B=1, H=2, k=3: scalar loops from the definition, element values decoded by
    torch (not by the oracle's tables)."""
    w, kv, qbits, q = tiny_inputs(1, 2, 32, seed=7)
    idx = np.array([[9, 2, 30]])
    out, lse = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    qf = q.to(torch.float64)[0]
    for h in range(2):
        scores, vals = [], []
        for r in idx[0]:
            row = torch.from_numpy(kv[r])
            acc = 0.0
            nope = []
            for c in range(448):
                v = float(row[c:c + 1].view(torch.float8_e4m3fn).to(torch.float64))
                v *= 2.0 ** (int(row[448 + c // 64]) - 127)
                nope.append(v)
                acc += float(qf[h, c]) * v
            for j in range(64):
                v = float(row[456 + 2 * j:458 + 2 * j].view(torch.bfloat16).to(torch.float64))
                acc += float(qf[h, 448 + j]) * v
            scores.append(acc * SCALE)
            vals.append(nope)
        mx = max(scores)
        den = sum(math.exp(s - mx) for s in scores)
        exp_lse = mx + math.log(den)
        exp_out = [sum(math.exp(scores[i] - exp_lse) * vals[i][c] for i in range(3)) for c in range(448)]
        assert abs(lse[0, h] - exp_lse) < 1e-12
        assert np.max(np.abs(out[0, h] - np.array(exp_out))) < 1e-12


# ---------------------------------------------------------------------------
# split-K partials and their merge
# ---------------------------------------------------------------------------
def test_split_ranges_partition():
    for k in (1, 15, 16, 17, 128, 2048, 2047):
        for S in (1, 2, 3, 7, 16, 19, 200):
            r = O.split_ranges(k, S)
            assert r[0][0] == 0 and r[-1][1] == k
            for (a0, a1), (b0, b1) in zip(r, r[1:]):
                assert a1 == b0 and a0 <= a1
            for a0, a1 in r:
                assert a0 % 16 == 0 and (a1 % 16 == 0 or a1 == k)


@pytest.mark.parametrize("S", [1, 2, 7, 16])
def test_split_invariance(S):
    B, H, n, k = 2, 4, 400, 256
    w, kv, qbits, q = tiny_inputs(B, H, n, seed=12)
    idx = perm_indices(B, n, k, 5)
    idx[1, 16:48] = -1                       # an all-masked stretch (a whole split at S=16)
    ref_o, ref_l = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    op, lp = O.split_partials(qbits, kv, idx, SCALE, S)
    o, l = O.combine(op, lp)
    assert np.max(np.abs(o - ref_o)) < 1e-12 and np.max(np.abs(l - ref_l)) < 1e-12
    if S == 16:
        assert np.all(np.isneginf(lp[1, :, 1])) and np.all(op[1, :, 1] == 0)


def test_combine_closed_forms():
    o = np.random.default_rng(0).standard_normal((3, 2, 448))
    lse = np.array([[0.5, 0.5]] * 3)
    out, l = O.combine(o, lse)
    assert np.max(np.abs(out - o.mean(1))) < 1e-15 and np.max(np.abs(l - (0.5 + math.log(2)))) < 1e-15
    lse2 = np.array([[-np.inf, 1.25]] * 3)
    out2, l2 = O.combine(o, lse2)
    assert np.array_equal(out2, o[:, 1]) and np.all(l2 == 1.25)
    out3, l3 = O.combine(o, np.full((3, 2), -np.inf))
    assert np.all(out3 == 0) and np.all(np.isneginf(l3))


# ---------------------------------------------------------------------------
# planted mistakes: each must make a pin fail
# ---------------------------------------------------------------------------
def _dense_pin_passes():
    B, H, n = 1, 4, 128
    w, kv, qbits, q = tiny_inputs(B, H, n, seed=31, outliers=0.01)
    idx = np.arange(n)[None]
    try:
        out, lse = O.sparse_mla_decode(qbits, kv, idx, SCALE)
    except Exception:
        return False
    ro, rl = torch_reference(q, torch.from_numpy(kv), idx, SCALE)
    return bool(np.max(np.abs(out - ro)) < 1e-9 and np.max(np.abs(lse - rl)) < 1e-9)


def test_planted_mistakes_are_caught(monkeypatch):
    assert _dense_pin_passes()
    # 1) wrong scale group (off by one)
    orig = O.dequantize_rows

    def wrong_group(rows):
        rows = np.asarray(rows, np.uint8).copy()
        rows[:, 448:455] = np.roll(rows[:, 448:455], 1, axis=1)
        return orig(rows)
    monkeypatch.setattr(O, "dequantize_rows", wrong_group)
    assert not _dense_pin_passes()
    monkeypatch.setattr(O, "dequantize_rows", orig)
    # 2) rope term dropped
    orig_attend = O.attend
    monkeypatch.setattr(O, "attend", lambda q, kn, kr, s: orig_attend(q, kn, kr * 0, s))
    assert not _dense_pin_passes()
    monkeypatch.setattr(O, "attend", orig_attend)
    # 3) rope read one bf16 element off
    monkeypatch.setattr(O, "ROPE_BYTE0", 458)
    monkeypatch.setattr(O, "ROW_END", 586)
    with np.errstate(all="ignore"):
        assert not _dense_pin_passes()
    monkeypatch.setattr(O, "ROPE_BYTE0", 456)
    monkeypatch.setattr(O, "ROW_END", 584)
    # 4) base-2 instead of natural LSE
    monkeypatch.setattr(O.np, "log", np.log2)
    assert not _dense_pin_passes()
    monkeypatch.undo()
    assert _dense_pin_passes()
