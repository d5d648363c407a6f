"""Pins for the CPU oracle: brute force, closed forms, invariants and the
figures the pages print.  None of these compares the oracle with itself.

Sources (web pages on multi-LoRA serving):
  [Guide]    "Multi-LoRA batching and adapter paging"
  [Concepts] "Serving Many LoRA Adapters"
  [Handbook] "Serving multiple LoRAs: segmented matrix multiplies and adapter scheduling"
  [Blog]     "Serving many LoRA adapters" (blog.ecitis.org)
"""
import json
import os

import numpy as np
import pytest

from oracle import lora_ref as O
from lora_serving_device_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# brute force: the layer's definition with explicit scalar loops, tiny shapes
# ----------------------------------------------------------------------------

def brute_force_y(x, W0, A, B, scale, ids):
    T, d_in = x.shape
    d_out = W0.shape[1]
    n_slots, _, r = A.shape
    y = [[0.0] * d_out for _ in range(T)]
    for t in range(T):
        a = int(ids[t])
        v = [0.0] * r
        if 0 <= a < n_slots:
            for q in range(r):
                acc = 0.0
                for k in range(d_in):
                    acc += float(x[t, k]) * float(A[a, k, q])
                v[q] = float(scale[a]) * acc
        for n in range(d_out):
            acc = 0.0
            for k in range(d_in):
                acc += float(x[t, k]) * float(W0[k, n])
            if 0 <= a < n_slots:
                for q in range(r):
                    acc += v[q] * float(B[a, q, n])
            y[t][n] = acc
    return np.array(y)


def _tiny(seed, T=7, d_in=12, d_out=10, r=3, n_slots=4, invalid=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d_in))
    W0 = rng.standard_normal((d_in, d_out))
    A = rng.standard_normal((n_slots, d_in, r))
    B = rng.standard_normal((n_slots, r, d_out))
    scale = rng.uniform(0.5, 3.0, n_slots)
    ids = rng.integers(-1, n_slots, T)
    if invalid:
        ids[0] = n_slots          # out of range -> base only
        ids[-1] = -3              # below -1 -> base only
    return x, W0, A, B, scale, ids


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    x, W0, A, B, s, ids = _tiny(seed, T=1 + seed, d_in=4 + 2 * seed, d_out=3 + seed,
                                r=1 + seed % 4, n_slots=1 + seed % 5)
    ref = brute_force_y(x, W0, A, B, s, ids)
    for fn in (O.lora_linear, O.lora_linear_gathered, O.lora_linear_segmented):
        np.testing.assert_allclose(fn(x, W0, A, B, s, ids), ref, rtol=1e-12, atol=1e-12)


def test_shrink_expand_brute_force():
    x, W0, A, B, s, ids = _tiny(11)
    v = O.shrink(x, A, s, ids)
    for t in range(x.shape[0]):
        a = ids[t]
        for q in range(A.shape[2]):
            want = 0.0
            if 0 <= a < A.shape[0]:
                want = s[a] * sum(x[t, k] * A[a, k, q] for k in range(x.shape[1]))
            assert abs(v[t, q] - want) <= 1e-12 * (1 + abs(want))
    d = O.expand(v, B, ids)
    base = brute_force_y(x, W0, A, B, s, np.full_like(ids, -1))
    full = brute_force_y(x, W0, A, B, s, ids)
    np.testing.assert_allclose(d, full - base, rtol=1e-10, atol=1e-10)


def test_brute_force_catches_planted_mistakes():
    """The brute-force pin separates the oracle from plausible mistakes: a
    dropped or doubled scale, A/B of the wrong adapter, -1 read as the last
    adapter (negative indexing), the base term dropped."""
    x, W0, A, B, s, ids = _tiny(3, T=8, invalid=False)
    ids[2] = -1
    ref = brute_force_y(x, W0, A, B, s, ids)
    good = O.lora_linear(x, W0, A, B, s, ids)
    np.testing.assert_allclose(good, ref, rtol=1e-12, atol=1e-12)
    mutants = {
        "scale dropped": O.lora_linear(x, W0, A, B, np.ones_like(s), ids),
        "scale doubled": O.lora_linear(x, W0, A, B, 2 * s, ids),
        "adapter off by one": O.lora_linear(x, W0, np.roll(A, 1, 0), np.roll(B, 1, 0), np.roll(s, 1), ids),
        "-1 read as last adapter": O.lora_linear(x, W0, A, B, s, np.where(ids < 0, A.shape[0] - 1, ids)),
        "base dropped": O.lora_linear(x, 0 * W0, A, B, s, ids),
    }
    for name, y in mutants.items():
        assert not np.allclose(y, ref, rtol=1e-6, atol=1e-6), name


# ----------------------------------------------------------------------------
# closed forms and invariants the pages state
# ----------------------------------------------------------------------------

def test_merge_equivalence():
    """[Blog, "Merge or keep separate"]: W' = W0 + (alpha/r) B A gives the same
    output as the unmerged path; in row-vector form x (W0 + s A B)."""
    x, W0, A, B, s, _ = _tiny(5, T=9, d_in=20, d_out=14, r=4, n_slots=3, invalid=False)
    for a in range(3):
        ids = np.full(x.shape[0], a)
        Wm = O.merge(W0, A[a], B[a], s[a])
        np.testing.assert_allclose(O.lora_linear(x, W0, A, B, s, ids), x @ Wm, rtol=1e-12, atol=1e-12)


def test_base_only_rows_and_zero_B():
    """Id -1 rows ([Blog, "Replay": "req C -> base only"]) and adapters with
    B = 0 both give exactly x W0 ([Blog, "Low-rank structure and additivity"]:
    the base output does not depend on the adapter)."""
    x, W0, A, B, s, ids = _tiny(6, invalid=False)
    base = x @ W0
    y = O.lora_linear(x, W0, A, B, s, np.full_like(ids, -1))
    np.testing.assert_array_equal(y, base)
    y0 = O.lora_linear(x, W0, A, np.zeros_like(B), s, ids)
    np.testing.assert_allclose(y0, base, rtol=0, atol=1e-13)


def test_permutation_invariance():
    """Additivity ([Blog, "Low-rank structure and additivity"]): each row's
    output depends only on its own input and adapter, so shuffling the batch
    (rows with their ids) shuffles the output identically."""
    x, W0, A, B, s, ids = _tiny(7, T=16)
    y = O.lora_linear(x, W0, A, B, s, ids)
    p = np.random.default_rng(1).permutation(x.shape[0])
    np.testing.assert_allclose(O.lora_linear(x[p], W0, A, B, s, ids[p]), y[p], rtol=1e-13, atol=1e-13)


def test_one_hot_rows_closed_form():
    """x_t = e_k picks row k: y_t = W0[k] + s A[a][k] B[a]."""
    _, W0, A, B, s, _ = _tiny(8, invalid=False)
    d_in = W0.shape[0]
    x = np.eye(d_in)
    for a in (-1, 0, 2):
        y = O.lora_linear(x, W0, A, B, s, np.full(d_in, a))
        want = W0 + (s[a] * (A[a] @ B[a]) if a >= 0 else 0.0)
        np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)


def test_rank_padding_exact():
    """Zero-padding an adapter to the pool rank leaves the result unchanged
    ([Concepts, "When It Falls Down"]; [Handbook, Exercise 2])."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((5, 24))
    W0 = rng.standard_normal((24, 18))
    A = rng.standard_normal((24, 8))
    B = rng.standard_normal((8, 18))
    Ap, Bp = O.pad_rank(A, B, 64)
    ids = np.zeros(5, int)
    y8 = O.lora_linear(x, W0, A[None], B[None], [2.0], ids)
    y64 = O.lora_linear(x, W0, Ap[None], Bp[None], [2.0], ids)
    np.testing.assert_allclose(y64, y8, rtol=1e-13, atol=1e-13)
    # the padded pass does r_pad/r times the adapter arithmetic: rank 4 in a
    # rank-64 batch pays 16x ([Concepts, "When It Falls Down"])
    f = _gold("printed_figures.json")["rank_padding_penalty"]
    assert f["r_max"] // f["r_small"] == f["penalty"]


def test_ragged_brute_force_and_padding():
    """Adapters at their own ranks: scalar loops over each adapter's own rank
    give the same y, and so does the pool zero-padded to the largest rank
    ([Concepts, "When It Falls Down"]; [Blog, "Batching across different
    adapters"])."""
    rng = np.random.default_rng(21)
    T, d_in, d_out = 9, 11, 7
    ranks = [1, 4, 2, 6, 3]
    x = rng.standard_normal((T, d_in))
    W0 = rng.standard_normal((d_in, d_out))
    A = [rng.standard_normal((d_in, r)) for r in ranks]
    B = [rng.standard_normal((r, d_out)) for r in ranks]
    s = rng.uniform(0.5, 3.0, len(ranks))
    ids = rng.integers(-1, len(ranks), T)
    ids[0], ids[1] = len(ranks), -4           # read as base only
    want = np.zeros((T, d_out))
    for t in range(T):
        a = int(ids[t])
        for n in range(d_out):
            acc = sum(x[t, k] * W0[k, n] for k in range(d_in))
            if 0 <= a < len(ranks):
                for q in range(ranks[a]):
                    vq = s[a] * sum(x[t, k] * A[a][k, q] for k in range(d_in))
                    acc += vq * B[a][q, n]
            want[t, n] = acc
    got = O.lora_linear_ragged(x, W0, A, B, s, ids)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    r_pad = max(ranks)
    Ap = np.stack([O.pad_rank(A[a], B[a], r_pad)[0] for a in range(len(ranks))])
    Bp = np.stack([O.pad_rank(A[a], B[a], r_pad)[1] for a in range(len(ranks))])
    np.testing.assert_allclose(O.lora_linear(x, W0, Ap, Bp, s, ids), want, rtol=1e-12,
                               atol=1e-12)
    # a plausible mistake: every adapter cut to the smallest rank
    cut = O.lora_linear_ragged(x, W0, [a[:, :1] for a in A], [b[:1] for b in B], s, ids)
    assert not np.allclose(cut, want, rtol=1e-6, atol=1e-6)


def test_bf16_round_closed_forms():
    """Ties to even at the 8-bit significand, and agreement with rounding
    x / ulp(x) half to even in float64 for normal numbers."""
    one = 1.0
    cases = {one: one, one + 2.0 ** -8: one, one + 3 * 2.0 ** -8: one + 2.0 ** -6,
             one + 2.0 ** -8 + 2.0 ** -20: one + 2.0 ** -7, -(one + 2.0 ** -8): -one,
             0.0: 0.0, 3.0: 3.0, 2.0 ** -100: 2.0 ** -100}
    got = O.bf16_round(np.array(list(cases), np.float32))
    assert got.tolist() == list(cases.values())
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4000) * 10.0 ** rng.uniform(-6, 6, 4000)).astype(np.float32)
    xd = x.astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(xd))) - 7)
    want = np.round(xd / ulp) * ulp             # numpy rounds half to even
    np.testing.assert_array_equal(O.bf16_round(x), want)


def _codebook():
    return O.bf16_round(np.array(W.nf4_like_codebook(), np.float32))


def test_quantize_4bit_recovers_exact_codes():
    """Weights built as absmax * codebook[code], each block holding a +-1
    entry, quantise back to those codes and scales exactly; scales that vary
    along both axes catch blocks taken along the wrong axis."""
    cb = _codebook()
    assert cb.size == 16 and np.unique(cb).size == 16 and cb.min() == -1 and cb.max() == 1
    rng = np.random.default_rng(8)
    d_in, d_out = 256, 40
    codes = rng.integers(0, 16, (d_in, d_out)).astype(np.uint8)
    codes[::64] = 15                                  # codebook[15] = +1 in every block
    s = O.bf16_round(rng.uniform(0.01, 0.2, (d_in // 64, d_out)).astype(np.float32))
    Wt = (cb[codes] * np.repeat(s, 64, axis=0)).astype(np.float32)
    got_c, got_s = O.quantize_4bit(Wt, cb)
    np.testing.assert_array_equal(got_c, codes)
    np.testing.assert_array_equal(got_s, s)
    np.testing.assert_array_equal(O.dequantize_4bit(got_c, got_s, cb), O.bf16_round(Wt))
    # blocks along the other axis give other scales
    wrong = np.abs(Wt.reshape(d_in, d_out // 8, 8)).max(axis=2)
    assert wrong.shape != got_s.shape or not np.array_equal(wrong, got_s)


def test_quantize_4bit_brute_force():
    """Scalar loops over a tiny matrix with a zero block, in fp32 scalars."""
    cb = _codebook().astype(np.float32)
    rng = np.random.default_rng(12)
    d_in, d_out = 128, 6
    Wt = O.bf16_round(rng.standard_normal((d_in, d_out)).astype(np.float32) * 0.02)
    Wt[64:, 2] = 0.0
    Wt = Wt.astype(np.float32)
    codes, absmax = O.quantize_4bit(Wt, cb)
    for b in range(d_in // 64):
        for n in range(d_out):
            m = np.float32(0.0)
            for k in range(64):
                m = max(m, np.float32(abs(Wt[64 * b + k, n])))
            assert absmax[b, n] == m
            for k in range(64):
                v = np.float32(Wt[64 * b + k, n]) / m if m > 0 else np.float32(0.0)
                dists = [abs(np.float32(v) - cb[c]) for c in range(16)]
                assert codes[64 * b + k, n] == int(np.argmin(dists))
    assert np.all(codes[64:, 2] == int(np.argmin(np.abs(cb))))


def test_dequantize_4bit_error_bound_and_packing():
    """|w - deq(w)| is at most half the widest codebook gap times absmax plus
    one bf16 rounding; the packing keeps k contiguous per column."""
    cb = _codebook()
    rng = np.random.default_rng(13)
    Wt = O.bf16_round(rng.standard_normal((192, 64)).astype(np.float32) * 0.02)
    codes, absmax = O.quantize_4bit(Wt, cb)
    deq = O.dequantize_4bit(codes, absmax, cb)
    gap = np.max(np.diff(np.sort(cb)))
    s = np.repeat(absmax.astype(np.float64), 64, axis=0)
    assert np.all(np.abs(Wt - deq) <= s * gap / 2 * (1 + 1e-6) + np.abs(deq) * 2.0 ** -8)
    assert np.max(np.abs(Wt - deq)) > 0
    packed = O.pack_4bit(codes)
    assert packed.shape == (64, 96)
    np.testing.assert_array_equal(packed & 15, codes[0::2, :].T)
    np.testing.assert_array_equal(packed >> 4, codes[1::2, :].T)
    assert packed[5, 7] == codes[14, 5] | (codes[15, 5] << 4)
    # one value worked by hand: code 3 at scale 0.5
    c3 = np.zeros((64, 2), np.uint8)
    c3[0, 1] = 3
    d = O.dequantize_4bit(c3, np.array([[1.0, 0.5]], np.float32), cb)
    assert d[0, 1] == O.bf16_round(np.float32(cb[3]) * np.float32(0.5))[()]


# ----------------------------------------------------------------------------
# the pages' printed figures
# ----------------------------------------------------------------------------

def test_toy_counts_and_segments_golden():
    """[Handbook] toy batch: 53 rows, 6 requests, 4 segments; perm / seg_off
    hand-derived (tests/golden/toy_segments.json)."""
    g = _gold("toy_segments.json")
    w = W.toy_mixed_batch()
    assert w.T == g["rows"] == 53
    assert len(w.req_lengths) == g["requests"] == 6
    seg = O.build_segments(w.slot_ids, w.n_slots)
    assert seg["n_seg"] == g["segments"] == 4
    assert seg["seg_slot"].tolist() == g["seg_slot"]
    assert seg["seg_off"].tolist() == g["seg_off"]
    assert np.diff(seg["seg_off"]).tolist() == g["seg_counts"]
    assert seg["perm"].tolist() == g["perm"]


def test_toy_three_forms_agree():
    """[Handbook]: BGMV and SGMV both match the per-request computation (the
    toy checks this in fp32 at atol 1e-5; in fp64 they agree to rounding)."""
    w = W.toy_mixed_batch()
    ref = O.lora_linear_per_request(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.req_lengths, w.req_slots)
    for fn in (O.lora_linear, O.lora_linear_gathered, O.lora_linear_segmented):
        np.testing.assert_allclose(fn(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids), ref,
                                   rtol=0, atol=1e-12)


def _segments_by_definition(ids, n_slots):
    """Counting-sort definition in plain Python: for each bin in ascending order
    (base-only bin first), the token indices holding it, in index order."""
    ids = [int(i) if 0 <= i < n_slots else -1 for i in ids]
    perm, seg_slot, seg_off = [], [], []
    for b in [-1] + list(range(n_slots)):
        members = [t for t, a in enumerate(ids) if a == b]
        if b >= 0 and members:
            seg_slot.append(b)
            seg_off.append(len(perm))
        perm.extend(members)
    seg_off.append(len(ids))
    return perm, seg_slot, seg_off


@pytest.mark.parametrize("seed", range(8))
def test_segments_by_definition(seed):
    rng = np.random.default_rng(100 + seed)
    n_slots = int(rng.integers(1, 12))
    T = int(rng.integers(0, 40))
    ids = rng.integers(-3, n_slots + 3, T)
    seg = O.build_segments(ids, n_slots)
    perm, seg_slot, seg_off = _segments_by_definition(ids, n_slots)
    assert seg["perm"].tolist() == perm
    assert seg["seg_slot"].tolist() == seg_slot
    assert seg["seg_off"].tolist() == seg_off
    assert seg["n_seg"] == len(seg_slot)


def test_param_count_figure():
    """[Blog, "Low-rank structure and additivity"]: d = k = 4096, r = 16 gives
    131k adapter parameters against 16.8M, about 0.8%."""
    f = _gold("printed_figures.json")["param_count"]
    n = O.lora_param_count(f["d"], f["k"], f["r"])
    assert n == 131072
    assert round(n / 1000) == round(f["lora_params_approx"] / 1000)
    dense = f["d"] * f["k"]
    assert round(dense / 1e5) == round(f["dense_params_approx"] / 1e5)
    assert abs(n / dense - f["fraction_approx"]) < 0.0005


def test_adapter_size_figures():
    """[Handbook] ~80 MB per adapter for an 8B base at rank 16 over the 7
    projections (8 GB keeps ~100); [Guide] 40 MB per hot adapter (10 GB keeps
    ~250), which is the same model at rank 8."""
    f = _gold("printed_figures.json")
    proj = [tuple(p) for p in f["decoder_8b_shape"]["projections"]]
    layers = f["decoder_8b_shape"]["layers"]
    b16 = O.adapter_bytes(proj, 16, layers)
    b8 = O.adapter_bytes(proj, 8, layers)
    assert b16 == 80 * 2 ** 20 and b8 == 40 * 2 ** 20
    assert abs(b16 / 1e6 - f["adapter_size_r16"]["approx_mb"]) / 80 < 0.06
    assert round(f["adapter_size_r16"]["budget_gb"] * 1e9 / (b16 * 1.0) / 10) * 10 == 100 or \
        abs(f["adapter_size_r16"]["budget_gb"] * 1e9 / b16 - 100) < 5
    assert abs(f["adapter_size_hot"]["budget_gb"] * 1e9 / (f["adapter_size_hot"]["approx_mb"] * 1e6)
               - f["adapter_size_hot"]["resident_approx"]) < 1e-9


def test_bf16_unit_roundoff_is_two_to_minus_eight():
    """The per-element parity bound uses 2^-8 as bf16's unit roundoff: one
    round-to-nearest-even to bf16 (8 significand bits) moves a value by at
    most 2^-8 / (1 + 2^-8) of its magnitude, reached by the tie just above a
    power of two.  A sweep of every fp32 significand pattern in one binade,
    at two scales, never exceeds it, and the tie attains it."""
    bound = 2.0 ** -8 / (1 + 2.0 ** -8)
    for scale in (1.0, 2.0 ** -30):
        # all 2^23 fp32 values in [1, 2), scaled (exact in fp32)
        bits = np.arange(0x3F800000, 0x40000000, dtype=np.uint32)
        x = bits.view(np.float32).astype(np.float64) * scale
        rel = np.abs(O.bf16_round(x.astype(np.float32)) - x) / x
        assert rel.max() <= bound * (1 + 1e-12)
        assert rel.max() >= bound * (1 - 1e-6)
    tie = np.float32(1 + 2.0 ** -8)
    assert O.bf16_round(np.array([tie]))[0] == 1.0
    assert abs((1.0 - float(tie)) / float(tie)) == pytest.approx(bound, rel=1e-12)
