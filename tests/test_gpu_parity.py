"""Parity of the CUDA path (through the C ABI) with the CPU fp64 oracle.

Integer outputs (segments) must match bit for bit; floating-point outputs
must meet the bar in tests/tolerances.py, for y and for the adapter delta.
Shapes span several tiles with ragged tails, every supported rank, empty and
single-token batches, invalid ids, and the full-size workloads.
"""
import numpy as np
import pytest

from oracle import lora_ref as O
from lora_serving_device_gb300 import workloads as W

from tests.gpu_util import DeviceCase, dev, host, torch_mod
from tests.tolerances import check_close, check_close_bf16_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from lora_serving_device_gb300 import build, lora
    build.build()
    lora.load()
    return lora


def _ws(L, n=1 << 16):
    torch = torch_mod()
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


# ------------------------------------------------------------ segment builder
SEG_CASES = [
    ("toy", lambda: (W.toy_mixed_batch().slot_ids, 8)),
    ("decode", lambda: (W.decode_ids(2), 256)),
    ("prefill", lambda: (np.repeat(np.array(W.prefill_ids()[1], np.int32),
                                   np.array(W.prefill_ids()[0])), 64)),
    ("sweep", lambda: (W.sweep_ids(256, 64), 1024)),
    ("empty", lambda: (np.zeros(0, np.int32), 5)),
    ("one", lambda: (np.array([3], np.int32), 5)),
    ("all_base", lambda: (np.full(100, -1, np.int32), 7)),
    ("one_slot", lambda: (np.zeros(300, np.int32), 1)),
    ("invalid", lambda: (W.random_case(3, 500, 8, 8, 8, 40, invalid=9).slot_ids, 40)),
    ("max_tokens_16k", lambda: (np.random.default_rng(5).integers(-1, 64, 16432).astype(np.int32), 64)),
    ("max_slots", lambda: (np.random.default_rng(6).integers(-1, 16384, 5000).astype(np.int32), 16384)),
    ("many_tokens", lambda: (np.random.default_rng(7).integers(-1, 1024, 70000).astype(np.int32), 1024)),
]


@pytest.mark.parametrize("name,make", SEG_CASES, ids=[c[0] for c in SEG_CASES])
def test_segments_bit_exact(L, name, make):
    torch = torch_mod()
    ids, n_slots = make()
    ids = np.asarray(ids, np.int32)
    ws = _ws(L)
    perm, seg_slot, seg_off, n_seg = L.build_segments_t(dev(ids), n_slots, ws)
    torch.cuda.synchronize()
    ref = O.build_segments(ids, n_slots)
    n = int(n_seg.item())
    assert n == ref["n_seg"]
    assert perm.cpu().numpy().tolist() == ref["perm"].tolist()
    assert seg_slot.cpu().numpy()[:n].tolist() == ref["seg_slot"].tolist()
    assert seg_off.cpu().numpy()[:n + 1].tolist() == ref["seg_off"].tolist()
    err = L.get_error_t(ws)
    bad = np.any((ids < -1) | (ids >= n_slots))
    assert bool(err & L.DEVERR_BAD_SLOT) == bool(bad)


# ------------------------------------------------------------ BGMV / SGMV
GATHER_CASES = [
    # T, d_in, d_out, r, n_slots, dtype
    (1, 64, 64, 16, 3, "bf16"),
    (37, 200, 136, 8, 5, "bf16"),
    (64, 512, 264, 16, 9, "bf16"),
    (130, 256, 520, 32, 4, "bf16"),
    (70, 136, 200, 64, 6, "bf16"),
    (45, 128, 1032, 128, 3, "bf16"),
    # several 128-token SGMV items per segment, ragged d_in tail
    (700, 4096, 72, 64, 9, "bf16"),
    (300, 1000, 64, 128, 5, "bf16"),
    # many full 128-token items whose rows are consecutive (y moved by TMA in
    # the SGMV expand), a ragged last column tile
    (640, 256, 1032, 64, 4, "bf16"),
    (384, 512, 264, 128, 3, "bf16"),
    (53, 256, 256, 16, 8, "f32"),
    (90, 96, 72, 64, 4, "f32"),
]


def _v_input(T, r, ksplit, seed):
    # a seeded synthetic v_partial (input of the expand tests)
    rng = np.random.default_rng([7000, seed, T, r])
    return (rng.standard_normal((ksplit, T, r)) * 0.5).astype(np.float32)


@pytest.mark.parametrize("case", GATHER_CASES, ids=[str(c) for c in GATHER_CASES])
@pytest.mark.parametrize("form", ["bgmv", "sgmv"])
def test_shrink_matches_oracle(L, case, form):
    torch = torch_mod()
    T, d_in, d_out, r, n_slots, dt = case
    w = W.random_case(11 + T, T, d_in, d_out, r, n_slots, runs=(form == "sgmv"),
                      bf16=(dt == "bf16"))
    d = DeviceCase(w)
    ws = _ws(L)
    ref = O.shrink(w.x, w.A_pool, w.scale, w.slot_ids)
    for ksplit in (1, 3):
        if form == "bgmv":
            vp = L.bgmv_shrink_t(d.x, d.A, d.ids, d.scale, ksplit, ws)
        else:
            segs = L.build_segments_t(d.ids, n_slots, ws)
            vp = L.sgmv_shrink_t(d.x, d.A, segs, d.scale, ksplit, ws)
        torch.cuda.synchronize()
        v = host(vp).sum(axis=0)
        check_close(v, ref, f"{form} shrink ksplit={ksplit}")


@pytest.mark.parametrize("case", GATHER_CASES, ids=[str(c) for c in GATHER_CASES])
@pytest.mark.parametrize("form", ["bgmv", "sgmv"])
def test_expand_matches_oracle(L, case, form):
    torch = torch_mod()
    T, d_in, d_out, r, n_slots, dt = case
    w = W.random_case(23 + T, T, d_in, d_out, r, n_slots, runs=(form == "sgmv"),
                      bf16=(dt == "bf16"))
    d = DeviceCase(w)
    ws = _ws(L)
    ksplit = 2
    vp = _v_input(T, r, ksplit, 1)
    v = vp.astype(np.float64).sum(axis=0)
    y0 = (np.random.default_rng([7001, T]).standard_normal((T, d_out)) * 0.1).astype(np.float32)
    if dt == "bf16":
        y0 = W.bf16_round(y0)
    y = dev(y0, dt)
    if form == "bgmv":
        L.bgmv_expand_t(dev(vp, "f32"), d.B, d.ids, y, ws)
    else:
        segs = L.build_segments_t(d.ids, n_slots, ws)
        L.sgmv_expand_t(dev(vp, "f32"), d.B, segs, y, ws)
    torch.cuda.synchronize()
    delta_ref = O.expand(v, w.B_pool, w.slot_ids)
    got = host(y)
    check_close(got, y0 + delta_ref, f"{form} expand y")
    # base-only rows untouched, bit for bit
    base_rows = ~((w.slot_ids >= 0) & (w.slot_ids < n_slots))
    np.testing.assert_array_equal(got[base_rows], y0[base_rows].astype(np.float64))
    # delta alone, measured where it is large enough to resolve
    if dt == "f32":
        check_close(got - y0, delta_ref, f"{form} expand delta")


# SGMV expand items whose token rows are not consecutive in y (every token its
# own adapter draw): full 128-token items and ragged ones move y row by row
SCATTERED_EXPAND_CASES = [(600, 264, 64, 3), (1000, 1032, 64, 5), (300, 520, 128, 2),
                          (160, 136, 64, 1)]


@pytest.mark.parametrize("T,d_out,r,n_slots", SCATTERED_EXPAND_CASES,
                         ids=[str(c) for c in SCATTERED_EXPAND_CASES])
def test_sgmv_expand_scattered_rows(L, T, d_out, r, n_slots):
    torch = torch_mod()
    w = W.random_case(31 + T, T, 64, d_out, r, n_slots, runs=False)
    d = DeviceCase(w)
    ws = _ws(L)
    vp = _v_input(T, r, 2, 3)
    y0 = W.bf16_round((np.random.default_rng([7002, T]).standard_normal((T, d_out)) * 0.1)
                      .astype(np.float32))
    y = dev(y0, "bf16")
    segs = L.build_segments_t(d.ids, n_slots, ws)
    L.sgmv_expand_t(dev(vp, "f32"), d.B, segs, y, ws)
    torch.cuda.synchronize()
    got = host(y)
    check_close(got, y0 + O.expand(vp.astype(np.float64).sum(axis=0), w.B_pool, w.slot_ids),
                "scattered SGMV expand y")
    base_rows = ~((w.slot_ids >= 0) & (w.slot_ids < n_slots))
    np.testing.assert_array_equal(got[base_rows], y0[base_rows].astype(np.float64))
    assert L.get_error_t(ws) == 0


def _run_tail_ids(T, layout, seed):
    """Slot ids with, per slot, a run of consecutive rows and a number of
    scattered rows after it: layout = [(slot, run start, run length, n
    scattered)]; every other row is base-only."""
    rng = np.random.default_rng([7003, seed])
    ids = np.full(T, -1, np.int32)
    for slot, start, n_run, _ in layout:
        ids[start:start + n_run] = slot
    for slot, start, n_run, n_sc in layout:
        free = np.flatnonzero(ids[start + n_run:] == -1) + start + n_run
        ids[rng.choice(free, size=n_sc, replace=False)] = slot
    return ids


# SGMV expand items that start with a run of consecutive rows and end with
# scattered ones (a prefill request's last item joined by decode tokens of
# the same adapter): runs of 22 / 100 rows with 16 / 1 later rows move the
# run by TMA; 17 later rows, or a run shorter than 16, move row by row
RUN_TAIL_LAYOUT = [(0, 0, 150, 16), (1, 160, 40, 17), (2, 210, 15, 3), (3, 240, 100, 1)]


@pytest.mark.parametrize("d_out,r", [(264, 64), (1032, 128)])
def test_sgmv_expand_run_and_tail_items(L, d_out, r):
    torch = torch_mod()
    T, n_slots = 700, 4
    ids = _run_tail_ids(T, RUN_TAIL_LAYOUT, d_out)
    rng = np.random.default_rng([7004, d_out])
    B = W.bf16_round((rng.standard_normal((n_slots, r, d_out)) * 0.02).astype(np.float32))
    vp = _v_input(T, r, 2, 4)
    y0 = W.bf16_round((rng.standard_normal((T, d_out)) * 0.1).astype(np.float32))
    y = dev(y0, "bf16")
    ws = _ws(L)
    segs = L.build_segments_t(dev(ids), n_slots, ws)
    L.sgmv_expand_t(dev(vp, "f32"), dev(B, "bf16"), segs, y, ws)
    torch.cuda.synchronize()
    got = host(y)
    check_close(got, y0 + O.expand(vp.astype(np.float64).sum(axis=0), B, ids),
                "run + tail SGMV expand y")
    np.testing.assert_array_equal(got[ids < 0], y0[ids < 0].astype(np.float64))
    assert L.get_error_t(ws) == 0


# SGMV shrink on the same layouts and on more runs with scattered rows after
# them (a segment's last chunk mixes a run with later rows and is gathered:
# 22 + 16, 40 + 17, 15 + 3, 100 + 1, 100 + 20, 17 + 111, 127 + 1, 62 + 3 in a
# 193-token segment, 16 + 14, 112 + 2, 50 + 5; the other chunks are
# consecutive rows, moved by TMA); the shrink numbers every last chunk first;
# d_in with and without a ragged last K-block
SHRINK_RUN_TAIL_LAYOUTS = [RUN_TAIL_LAYOUT,
                           [(0, 0, 100, 20), (1, 130, 16, 112), (2, 300, 127, 1),
                            (3, 450, 60, 0)],
                           [(0, 0, 190, 3), (1, 200, 16, 14), (2, 300, 112, 2),
                            (3, 450, 50, 5)]]


@pytest.mark.parametrize("layout", [0, 1, 2])
@pytest.mark.parametrize("d_in,r", [(520, 64), (1032, 128), (1024, 64), (512, 128)])
def test_sgmv_shrink_run_and_tail_items(L, d_in, r, layout):
    torch = torch_mod()
    T, n_slots = 700, 4
    ids = _run_tail_ids(T, SHRINK_RUN_TAIL_LAYOUTS[layout], d_in)
    rng = np.random.default_rng([7007, d_in])
    A = W.bf16_round((rng.standard_normal((n_slots, d_in, r)) / np.sqrt(d_in)).astype(np.float32))
    x = W.bf16_round(rng.standard_normal((T, d_in)).astype(np.float32))
    scale = rng.uniform(0.5, 2.5, n_slots).astype(np.float32)
    ws = _ws(L)
    segs = L.build_segments_t(dev(ids), n_slots, ws)
    ref = O.shrink(x, A, scale, ids)
    for ksplit in (1, 4):
        vp = L.sgmv_shrink_t(dev(x, "bf16"), dev(A, "bf16"), segs, dev(scale, "f32"), ksplit, ws)
        torch.cuda.synchronize()
        check_close(host(vp).sum(axis=0), ref, f"run + tail SGMV shrink ksplit={ksplit}")
    assert L.get_error_t(ws) == 0


def _short_segment_ids(T, n_single, seed):
    """Slot ids for segments of at most 16 tokens (which the rank-64 SGMV
    expand serves two to a CTA): n_single one-token segments, one segment of 5
    tokens and one of 17 (not paired), the rest base-only, shuffled."""
    rng = np.random.default_rng([7005, seed])
    ids = np.full(T, -1, np.int32)
    pos = rng.permutation(T)
    k = 0
    for slot in range(n_single):
        ids[pos[k]] = slot
        k += 1
    for slot, n in ((n_single, 5), (n_single + 1, 17)):
        ids[pos[k:k + n]] = slot
        k += n
    return ids


# an odd and an even number of short segments; a ragged last column tile
@pytest.mark.parametrize("n_single,d_out", [(30, 1032), (21, 264)])
def test_sgmv_expand_short_segments_in_pairs(L, n_single, d_out):
    torch = torch_mod()
    T, r, n_slots = 80, 64, n_single + 2
    ids = _short_segment_ids(T, n_single, n_single)
    rng = np.random.default_rng([7006, n_single])
    B = W.bf16_round((rng.standard_normal((n_slots, r, d_out)) * 0.02).astype(np.float32))
    vp = _v_input(T, r, 1, 5)
    y0 = W.bf16_round((rng.standard_normal((T, d_out)) * 0.1).astype(np.float32))
    y = dev(y0, "bf16")
    ws = _ws(L)
    segs = L.build_segments_t(dev(ids), n_slots, ws)
    L.sgmv_expand_t(dev(vp, "f32"), dev(B, "bf16"), segs, y, ws)
    torch.cuda.synchronize()
    got = host(y)
    check_close(got, y0 + O.expand(vp.astype(np.float64).sum(axis=0), B, ids),
                "short-segment SGMV expand y")
    np.testing.assert_array_equal(got[ids < 0], y0[ids < 0].astype(np.float64))
    assert L.get_error_t(ws) == 0


# ------------------------------------------------------------ fused layer
FUSED_CASES = [
    # T, d_in, d_out, r, n_slots : decode tiles (T <= 256) and prefill tiles
    (1, 64, 128, 16, 3),
    (5, 200, 136, 8, 7),
    (32, 1000, 264, 16, 12),
    (33, 256, 384, 32, 5),
    (64, 512, 1024, 16, 40),
    (100, 128, 520, 64, 9),
    (128, 384, 256, 128, 4),
    (200, 256, 264, 128, 6),
    (96, 320, 392, 8, 21),
    # adapter clusters of 2 and 4 CTAs with ragged d_in / d_out slices
    (7, 1032, 600, 32, 4),
    (48, 2056, 2120, 16, 9),
    (16, 2048, 2048, 128, 5),
    (200, 640, 136, 16, 30),
    (256, 256, 512, 64, 70),
    # 65..256 tokens: the merge grouped by adapter (items of <= 8 tokens of
    # one id): rank 32, one adapter for every token, ids nearly all distinct
    (160, 1032, 600, 32, 11),
    (200, 256, 264, 16, 1),
    (220, 512, 1024, 8, 1000),
    (65, 4096, 1032, 64, 3),
    # more adapter clusters than fit beside the decode GEMM: the persistent
    # merge (adapter terms through the workspace), ragged column slices
    (256, 2056, 4104, 16, 50),
    (240, 1024, 2056, 64, 30),
    (257, 192, 264, 16, 11),
    (300, 520, 512, 32, 6),
    (517, 136, 776, 64, 13),
    (1000, 256, 1288, 16, 50),
]


@pytest.mark.parametrize("case", FUSED_CASES, ids=[str(c) for c in FUSED_CASES])
def test_fused_matches_oracle(L, case):
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    for runs in (False, True):
        w = W.random_case(100 + T + int(runs), T, d_in, d_out, r, n_slots, runs=runs)
        d = DeviceCase(w)
        y, ws = d.fused()
        torch.cuda.synchronize()
        ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
        check_close_bf16_out(host(y), ref, f"y runs={runs}")
        assert L.get_error_t(ws) == 0
        # the adapter path alone (W0 = 0), so bf16 rounding of the base term
        # cannot hide an error in it
        d0 = DeviceCase(w, W0_zero=True)
        y0, _ = d0.fused()
        torch.cuda.synchronize()
        base = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, np.full(T, -1))
        check_close_bf16_out(host(y0), ref - base, f"delta runs={runs}")


@pytest.mark.parametrize("T,d_in,d_out", [(90, 256, 264), (250, 1024, 4104)])
def test_fused_invalid_ids_are_base_only_and_flagged(L, T, d_in, d_out):
    torch = torch_mod()
    w = W.random_case(501, T, d_in, d_out, 16, 10, invalid=7)
    d = DeviceCase(w)
    y, ws = d.fused()
    torch.cuda.synchronize()
    ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
    check_close_bf16_out(host(y), ref, f"y with invalid ids, T={T}")
    assert L.get_error_t(ws) & L.DEVERR_BAD_SLOT
    assert L.get_error_t(ws) == 0          # cleared by the read


def test_fused_all_base_and_zero_B(L):
    torch = torch_mod()
    w = W.random_case(502, 48, 256, 136, 16, 4)
    w.slot_ids[:] = -1
    d = DeviceCase(w)
    y, _ = d.fused()
    torch.cuda.synchronize()
    check_close(host(y), O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids), "all base")
    w2 = W.random_case(503, 48, 256, 136, 16, 4)
    w2.B_pool[:] = 0
    d2 = DeviceCase(w2)
    y2, _ = d2.fused()
    torch.cuda.synchronize()
    base = O.lora_linear(w2.x, w2.W0, w2.A_pool, w2.B_pool, w2.scale, np.full(48, -1))
    check_close(host(y2), base, "B = 0")


def test_fused_deterministic_and_graph_capturable(L):
    torch = torch_mod()
    w = W.random_case(504, 64, 1024, 1024, 16, 20)
    d = DeviceCase(w)
    y1, ws = d.fused()
    y2, _ = d.fused(ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    y3 = torch.empty_like(y1)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.fused(ws=ws, y=y3)     # warm-up on the capture stream
        with torch.cuda.graph(g, stream=s):
            d.fused(ws=ws, y=y3)
    torch.cuda.current_stream().wait_stream(s)
    y3.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1, y3)


# ------------------------------------------------------------ the workloads
def test_toy_mixed_batch_fp32(L):
    torch = torch_mod()
    w = W.toy_mixed_batch()
    d = DeviceCase(w)
    y, ws = d.fused()
    torch.cuda.synchronize()
    ref = O.lora_linear_per_request(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.req_lengths, w.req_slots)
    check_close(host(y), ref, "toy y")
    # fp32 storage: the toy page checks allclose at atol 1e-5
    assert np.max(np.abs(host(y) - ref)) < 1e-4


def test_decode_bgmv_full(L):
    torch = torch_mod()
    w = W.decode_bgmv()
    d = DeviceCase(w)
    y, ws = d.fused()
    torch.cuda.synchronize()
    ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
    check_close(host(y), ref, "decode y")
    assert L.get_error_t(ws) == 0
    # standalone BGMV shrink + expand on the same batch
    wsb = _ws(L)
    vp = L.bgmv_shrink_t(d.x, d.A, d.ids, d.scale, 16, wsb)
    yb = dev(np.zeros((w.T, w.d_out), np.float32), "bf16")
    L.bgmv_expand_t(vp, d.B, d.ids, yb, wsb)
    torch.cuda.synchronize()
    base = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, np.full(w.T, -1))
    check_close_bf16_out(host(yb), ref - base, "decode BGMV delta")
    d0 = DeviceCase(w, W0_zero=True)
    y0, _ = d0.fused()
    torch.cuda.synchronize()
    check_close_bf16_out(host(y0), ref - base, "decode fused delta")


def test_prefill_sgmv_full(L):
    torch = torch_mod()
    w = W.prefill_sgmv()
    d = DeviceCase(w)
    y, ws = d.fused()
    torch.cuda.synchronize()
    ref = O.lora_linear_per_request(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.req_lengths, w.req_slots)
    check_close(host(y), ref, "prefill y")
    assert L.get_error_t(ws) == 0
    # standalone SGMV shrink + expand on the same batch (delta only)
    wsb = _ws(L)
    segs = L.build_segments_t(d.ids, w.n_slots, wsb)
    vp = L.sgmv_shrink_t(d.x, d.A, segs, d.scale, 2, wsb)
    yb = dev(np.zeros((w.T, w.d_out), np.float32), "bf16")
    L.sgmv_expand_t(vp, d.B, segs, yb, wsb)
    torch.cuda.synchronize()
    base = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, np.full(w.T, -1))
    delta = ref - base
    check_close_bf16_out(host(yb), delta, "prefill SGMV delta")


# more 128 x 256 output tiles than SMs: each CTA walks several tiles with two
# accumulators in tensor memory (632 tiles: up to five per CTA)
PERSIST_CASES = [(1000, 200, 20008, 16, True), (700, 1032, 12296, 64, False),
                 # 256 x 256 tiles with four rank-8 units per LoRA stage (B rows
                 # past the stage's units zero-filled) and with rank 128
                 (1024, 136, 19456, 8, False), (600, 264, 30000, 128, True)]


@pytest.mark.parametrize("T,d_in,d_out,r,runs", PERSIST_CASES, ids=[str(c) for c in PERSIST_CASES])
def test_prefill_many_tiles(L, T, d_in, d_out, r, runs):
    """Runs of adapters (or every token its own draw), whole tiles with no
    adapter and ragged token, column and d_in tails, with and without the
    base term."""
    torch = torch_mod()
    w = W.random_case(1200 + T, T, d_in, d_out, r, 24, runs=runs)
    w.slot_ids[128:400] = -1
    w.slot_ids[-40:] = -1
    for W0_zero in (False, True):
        d = DeviceCase(w, W0_zero=W0_zero)
        y, ws = d.fused()
        torch.cuda.synchronize()
        W0 = np.zeros_like(w.W0) if W0_zero else w.W0
        ref = O.lora_linear(w.x, W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
        if W0_zero:
            check_close_bf16_out(host(y), ref, "many-tile delta")
        else:
            check_close(host(y), ref, "many-tile y")
        assert L.get_error_t(ws) == 0
        del d, y, ws


# prefill batches at rank 64 / 128: the tensor-core shrink folds its d_in
# splits into one partial; d_in 520 at split 4 leaves the last split empty,
# d_in 264 runs at split 2
FOLD_CASES = [(300, 520, 264, 64), (1100, 1032, 1032, 128), (700, 264, 520, 64)]


@pytest.mark.parametrize("T,d_in,d_out,r", FOLD_CASES, ids=[str(c) for c in FOLD_CASES])
def test_prefill_shrink_fold(L, T, d_in, d_out, r):
    """The CTA of each shrink item that finishes last sums the splits in
    split order, counted on words of the workspace that the segment build
    zeroes: a workspace that starts as 0xFF bytes (error word aside) must
    give the oracle's result, and a second call the same bits."""
    torch = torch_mod()
    w = W.random_case(1300 + T, T, d_in, d_out, r, 24, runs=True)
    w.slot_ids[40:90] = -1
    ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, w.n_slots)
    ws.fill_(255)
    ws[:16] = 0
    for W0_zero in (False, True):
        d = DeviceCase(w, W0_zero=W0_zero)
        y1, _ = d.fused(ws=ws)
        y2, _ = d.fused(ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2)
        W0 = np.zeros_like(w.W0) if W0_zero else w.W0
        ref = O.lora_linear(w.x, W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
        check_close_bf16_out(host(y1), ref, f"folded shrink, W0 zero={W0_zero}")
        assert L.get_error_t(ws) == 0
        if not W0_zero:
            # replays of a captured call: the counters are zeroed by the
            # captured segment build on every replay
            y3 = torch.empty_like(y1)
            g = torch.cuda.CUDAGraph()
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                d.fused(ws=ws, y=y3)
                with torch.cuda.graph(g, stream=st):
                    d.fused(ws=ws, y=y3)
            torch.cuda.current_stream().wait_stream(st)
            for _ in range(2):
                y3.zero_()
                g.replay()
                torch.cuda.synchronize()
                assert torch.equal(y1, y3)
            assert L.get_error_t(ws) == 0
            del g, y3
        del d, y1, y2


# the folded shrink at the edges of the prefill path: one token above the
# decode sizes, one adapter for every token (16 chunks of one segment, split
# 4), ids outside the pool (flagged, base-only), and a batch with no adapter
# at all (no work item; the GEMM alone)
FOLD_EDGE_CASES = [("T=257", 257, 512, 264, 64, 3, 0, False),
                   ("one adapter", 2000, 1024, 520, 128, 1, 0, False),
                   ("invalid ids", 600, 512, 1032, 64, 12, 9, False),
                   ("all base-only", 300, 512, 264, 64, 4, 0, True)]


@pytest.mark.parametrize("name,T,d_in,d_out,r,n_slots,invalid,all_base", FOLD_EDGE_CASES,
                         ids=[c[0] for c in FOLD_EDGE_CASES])
def test_prefill_fold_edge_cases(L, name, T, d_in, d_out, r, n_slots, invalid, all_base):
    torch = torch_mod()
    w = W.random_case(1400 + T, T, d_in, d_out, r, n_slots, base_frac=0.0 if n_slots == 1 else 0.15,
                      runs=n_slots > 1, invalid=invalid)
    if all_base:
        w.slot_ids[:] = -1
    for W0_zero in (False, True):
        d = DeviceCase(w, W0_zero=W0_zero)
        y, ws = d.fused()
        torch.cuda.synchronize()
        W0 = np.zeros_like(w.W0) if W0_zero else w.W0
        ref = O.lora_linear(w.x, W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
        if all_base and W0_zero:
            np.testing.assert_array_equal(host(y), 0.0)
        elif W0_zero:
            check_close_bf16_out(host(y), ref, f"{name} delta")
        else:
            check_close(host(y), ref, f"{name} y")
        err = L.get_error_t(ws)
        assert (err & L.DEVERR_BAD_SLOT) if invalid else err == 0
        del d, y, ws


# the prefill GEMM's 256 x 256 tiles with one tile row far heavier in LoRA
# stages (40 one-token adapters at the batch's end, after long runs): the
# kernel moves that row's tiles to CTAs without a tile in the walk's last,
# partial round.  T 1100 over 76 column tiles: 380 tiles, 76 in the last
# round; T 1024: 304 tiles, none
@pytest.mark.parametrize("T", [1100, 1024])
def test_prefill_heavy_tile_row(L, T):
    torch = torch_mod()
    d_in, d_out, r, n_slots = 136, 256 * 76, 64, 48
    w = W.random_case(1500 + T, T, d_in, d_out, r, n_slots, base_frac=0.0)
    ids = np.repeat(np.arange(5, dtype=np.int32), -(-(T - 40) // 5))[:T - 40]
    w.slot_ids[:] = np.concatenate([ids, np.arange(8, 48, dtype=np.int32)])
    for W0_zero in (False, True):
        d = DeviceCase(w, W0_zero=W0_zero)
        y, ws = d.fused()
        torch.cuda.synchronize()
        W0 = np.zeros_like(w.W0) if W0_zero else w.W0
        ref = O.lora_linear(w.x, W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
        check_close_bf16_out(host(y), ref, f"heavy row {'delta' if W0_zero else 'y'} T={T}")
        assert L.get_error_t(ws) == 0
        del d, y, ws


@pytest.mark.parametrize("T,k", W.SWEEP_POINTS)
def test_diversity_sweep_point(L, T, k):
    torch = torch_mod()
    w = W.diversity_sweep(T, k, only_used_slots=True)
    d = DeviceCase(w)
    y, ws = d.fused()
    torch.cuda.synchronize()
    ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
    check_close(host(y), ref, f"sweep T={T} k={k}")
    assert L.get_error_t(ws) == 0


STACK_CHECK = [(0, p) for p in range(7)] + [(31, p) for p in range(7)] + [(13, 4), (22, 6)]


@pytest.mark.parametrize("layer,proj", STACK_CHECK)
def test_stack_8b_projection(L, layer, proj):
    torch = torch_mod()
    from lora_serving_device_gb300 import lora as Lm
    ranks = W.stack_ranks()
    ids = W.stack_ids()
    t = W.stack_layer_device(layer, proj, ranks=ranks)
    _, d_in, d_out = W.STACK_PROJECTIONS[proj]
    n_slots, r = 250, 64
    ws = Lm.workspace(Lm.OP_LINEAR_FUSED, 256, d_in, d_out, r, n_slots)
    scale = torch.full((n_slots,), W.SCALE, dtype=torch.float32, device="cuda")
    ids_d = torch.from_numpy(ids).cuda()
    y = Lm.linear_fused_t(t["x"], t["W0"], t["A_pool"], t["B_pool"], ids_d, scale, ws)
    torch.cuda.synchronize()
    used = np.unique(ids[ids >= 0])
    A = np.zeros((n_slots, d_in, r))
    B = np.zeros((n_slots, r, d_out))
    A[used] = host(t["A_pool"][torch.from_numpy(used).cuda()])
    B[used] = host(t["B_pool"][torch.from_numpy(used).cuda()])
    for j in used:   # rank padding really is zero
        assert np.all(A[j][:, ranks[j]:] == 0) and np.all(B[j][ranks[j]:] == 0)
    lengths, slots = W.stack_requests()
    ref = O.lora_linear_per_request(host(t["x"]), host(t["W0"]), A, B,
                                    np.full(n_slots, W.SCALE), lengths, slots)
    check_close(host(y), ref, f"stack layer {layer} proj {proj}")


# ------------------------------------------------- building-block entry points
BLOCK_CASES = [(1, 64, 128, 16, 3), (40, 512, 264, 16, 20), (64, 1024, 1024, 64, 9),
               (130, 256, 520, 8, 33), (256, 320, 392, 128, 5), (300, 256, 512, 32, 7)]


@pytest.mark.parametrize("case", BLOCK_CASES, ids=[str(c) for c in BLOCK_CASES])
def test_bgmv_delta_matches_oracle(L, case):
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    w = W.random_case(700 + T, T, d_in, d_out, r, n_slots)
    d = DeviceCase(w)
    ws = _ws(L)
    vp = _v_input(T, r, 3, 2)
    delta = torch.full((T, d_out), 7.0, dtype=torch.float32, device="cuda")
    L.bgmv_delta_t(dev(vp, "f32"), d.B, d.ids, ws, delta=delta)
    torch.cuda.synchronize()
    ref = O.expand(vp.astype(np.float64).sum(axis=0), w.B_pool, w.slot_ids)
    got = host(delta)
    valid = (w.slot_ids >= 0) & (w.slot_ids < n_slots)
    check_close(got[valid], ref[valid], "bgmv delta (fp32 out)", rel_fro=1e-5, max_rms=1e-4)
    assert np.all(got[~valid] == 7.0)          # base-only rows not written


ADAPTER_CASES = BLOCK_CASES + [(7, 1032, 600, 32, 4), (48, 2056, 2120, 16, 9),
                               (16, 2048, 2048, 128, 5), (64, 4096, 4096, 16, 256)]


@pytest.mark.parametrize("case", ADAPTER_CASES, ids=[str(c) for c in ADAPTER_CASES])
def test_bgmv_adapter_matches_oracle(L, case):
    """The one-launch adapter term (shrink, cluster sum, expand) against the
    oracle's shrink then expand.  Nothing is rounded to bf16 on this path:
    bf16 inputs, fp32 products and sums, fp32 out, so the bar is the fp32
    accumulation error of a d_in-long and an r-long dot product."""
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    w = W.random_case(730 + T, T, d_in, d_out, r, n_slots, invalid=1)
    d = DeviceCase(w)
    ws = _ws(L)
    delta = torch.full((T, d_out), 7.0, dtype=torch.float32, device="cuda")
    L.bgmv_adapter_t(d.x, d.A, d.B, d.ids, d.scale, ws, delta=delta)
    torch.cuda.synchronize()
    ref = O.expand(O.shrink(w.x, w.A_pool, w.scale, w.slot_ids), w.B_pool, w.slot_ids)
    got = host(delta)
    valid = (w.slot_ids >= 0) & (w.slot_ids < n_slots)
    check_close(got[valid], ref[valid], "bgmv adapter term (fp32 out)", rel_fro=2e-5,
                max_rms=2e-4)
    assert np.all(got[~valid] == 7.0)          # base-only rows not written
    assert L.get_error_t(ws) & L.DEVERR_BAD_SLOT
    # deterministic: the cluster sums its partials in a fixed order
    delta2 = torch.full((T, d_out), 7.0, dtype=torch.float32, device="cuda")
    L.bgmv_adapter_t(d.x, d.A, d.B, d.ids, d.scale, ws, delta=delta2)
    torch.cuda.synchronize()
    assert torch.equal(delta, delta2)


SPLITK_CASES = [(1, 64, 128, 1), (5, 200, 136, 2), (40, 1000, 264, 3), (64, 4096, 4096, 4),
                (64, 4096, 4096, 21), (100, 512, 520, 4), (256, 4096, 4096, 2), (300, 256, 512, 2),
                (64, 4096, 4096, 22), (40, 1000, 264, 6),
                # split 0: the split the fused layer uses
                (64, 4096, 4096, 0), (256, 4096, 4096, 0), (100, 4096, 4096, 0),
                (48, 2056, 2120, 0), (7, 1032, 600, 0), (256, 4096, 1024, 0), (1, 16384, 128, 0)]


@pytest.mark.parametrize("case", SPLITK_CASES, ids=[str(c) for c in SPLITK_CASES])
def test_base_gemm_splitk_matches_oracle(L, case):
    """The split-K tensor-core base product: the S fp32 partials must add up
    to x W0.  Nothing is rounded to bf16 on this path (bf16 inputs, fp32
    products and sums), so the bar is the fp32 accumulation error of a
    d_in-long dot product.  Every partial is written (no stale values)."""
    torch = torch_mod()
    T, d_in, d_out, ks = case
    S = ks if ks > 0 else L.lora_decode_split(T, d_in, d_out)
    w = W.random_case(710 + T + S, T, d_in, d_out, 8, 2)
    d = DeviceCase(w)
    ws = _ws(L)
    partial = torch.full((S, T, d_out), float("nan"), dtype=torch.float32, device="cuda")
    L.base_gemm_splitk_t(d.x, d.W0, ws, ksplit=ks, partial=partial)
    torch.cuda.synchronize()
    got = host(partial)
    assert np.all(np.isfinite(got))
    ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, np.full(T, -1))
    check_close(got.astype(np.float64).sum(axis=0), ref, "sum of split-K partials",
                rel_fro=2e-5, max_rms=2e-4)
    if S > 1 and d_in >= 1024:      # the splits really are partial sums over d_in
        assert not np.allclose(got[0], ref, rtol=1e-2, atol=1e-2)


@pytest.mark.parametrize("case", BLOCK_CASES, ids=[str(c) for c in BLOCK_CASES])
def test_bgmv_adapter_merge_matches_oracle(L, case):
    """y = (sum of given fp32 partials) + adapter term, every row written,
    one bf16 rounding; base-only and invalid ids get the partials only."""
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    w = W.random_case(740 + T, T, d_in, d_out, r, n_slots, invalid=1)
    d = DeviceCase(w)
    ws = _ws(L)
    S = 3
    part = (np.random.default_rng([7003, T]).standard_normal((S, T, d_out)) * 0.3).astype(np.float32)
    y = torch.full((T, d_out), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.bgmv_adapter_merge_t(d.x, d.A, d.B, d.ids, d.scale, dev(part, "f32"), ws, y=y)
    torch.cuda.synchronize()
    ref = part.astype(np.float64).sum(axis=0) + O.expand(
        O.shrink(w.x, w.A_pool, w.scale, w.slot_ids), w.B_pool, w.slot_ids)
    check_close_bf16_out(host(y), ref, "partials + adapter term")
    assert L.get_error_t(ws) & L.DEVERR_BAD_SLOT


@pytest.mark.parametrize("case", BLOCK_CASES, ids=[str(c) for c in BLOCK_CASES])
def test_base_gemm_expand_matches_oracle(L, case):
    """The tensor-core fold of the expand (LoRA K-blocks), given a shrink
    output, on decode and prefill tile shapes."""
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    w = W.random_case(720 + T, T, d_in, d_out, r, n_slots, runs=True)
    d = DeviceCase(w)
    ws = _ws(L)
    vp = _v_input(T, r, 2, 3)
    y = L.base_gemm_expand_t(d.x, d.W0, d.B, d.ids, dev(vp, "f32"), ws)
    torch.cuda.synchronize()
    base = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, np.full(T, -1))
    ref = base + O.expand(vp.astype(np.float64).sum(axis=0), w.B_pool, w.slot_ids)
    check_close_bf16_out(host(y), ref, "base GEMM + folded expand")
    d0 = DeviceCase(w, W0_zero=True)
    y0 = L.base_gemm_expand_t(d0.x, d0.W0, d0.B, d0.ids, dev(vp, "f32"), ws)
    torch.cuda.synchronize()
    check_close_bf16_out(host(y0), ref - base, "folded expand alone")


# more 256 x 256 tiles than two waves, v given as three partials: the wide
# prefill GEMM's LoRA stages sum the partials while building V; and the 128 x
# 256 persistent form
GEMM_EXPAND_WIDE = [(1000, 200, 20008, 16, 24), (1024, 136, 19456, 8, 30),
                    (700, 1032, 12296, 64, 24)]


@pytest.mark.parametrize("case", GEMM_EXPAND_WIDE, ids=[str(c) for c in GEMM_EXPAND_WIDE])
def test_base_gemm_expand_many_tiles(L, case):
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    w = W.random_case(780 + T, T, d_in, d_out, r, n_slots, runs=True)
    w.slot_ids[128:400] = -1
    d = DeviceCase(w)
    ws = _ws(L)
    vp = _v_input(T, r, 3, 4)
    y = L.base_gemm_expand_t(d.x, d.W0, d.B, d.ids, dev(vp, "f32"), ws)
    torch.cuda.synchronize()
    base = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, np.full(T, -1))
    ref = base + O.expand(vp.astype(np.float64).sum(axis=0), w.B_pool, w.slot_ids)
    check_close(host(y), ref, "many-tile base GEMM + folded expand")
    assert L.get_error_t(ws) == 0
    d0 = DeviceCase(w, W0_zero=True)
    y0 = L.base_gemm_expand_t(d0.x, d0.W0, d0.B, d0.ids, dev(vp, "f32"), ws)
    torch.cuda.synchronize()
    check_close_bf16_out(host(y0), ref - base, "many-tile folded expand alone")


# ------------------------------------------------------------- slot upload
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_slot_upload_then_layer_matches_oracle(L, dt):
    """A rank-8 adapter uploaded from pinned host memory into slot 3 of a
    rank-16 pool: the slot holds it zero-padded (bit-exact copy), the other
    slots are untouched, and the layer over tokens that use the slot matches
    the oracle (decode and prefill paths for bf16)."""
    torch = torch_mod()
    n_slots, d_in, d_out, r, r_a, slot, s = 6, 256, 264, 16, 8, 3, 1.75
    w = W.random_case(760, 300, d_in, d_out, r, n_slots, runs=True, bf16=(dt == "bf16"))
    d = DeviceCase(w)
    rng = np.random.default_rng([7004])
    A_a = (rng.standard_normal((d_in, r_a)) / 16).astype(np.float32)
    B_a = (rng.standard_normal((r_a, d_out)) * 0.02).astype(np.float32)
    if dt == "bf16":
        A_a, B_a = W.bf16_round(A_a), W.bf16_round(B_a)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    A_h = torch.from_numpy(A_a).to(tdt).pin_memory()
    B_h = torch.from_numpy(B_a).to(tdt).pin_memory()
    A_before, B_before = host(d.A).copy(), host(d.B).copy()
    L.slot_upload_t(d.A, d.B, d.scale, slot, A_h, B_h, s)
    torch.cuda.synchronize()
    A_after, B_after = host(d.A), host(d.B)
    assert np.array_equal(A_after[slot, :, :r_a], A_a) and not A_after[slot, :, r_a:].any()
    assert np.array_equal(B_after[slot, :r_a, :], B_a) and not B_after[slot, r_a:, :].any()
    others = [i for i in range(n_slots) if i != slot]
    assert np.array_equal(A_after[others], A_before[others])
    assert np.array_equal(B_after[others], B_before[others])
    assert float(d.scale[slot].item()) == s
    A_pool, B_pool, scale = w.A_pool.copy(), w.B_pool.copy(), w.scale.copy()
    A_pool[slot] = 0
    B_pool[slot] = 0
    A_pool[slot, :, :r_a] = A_a
    B_pool[slot, :r_a, :] = B_a
    scale[slot] = s
    ids = w.slot_ids.copy()
    ids[::3] = slot                                     # a third of the rows use the slot
    for T in (64, 300) if dt == "bf16" else (53,):
        ids_t = torch.from_numpy(ids[:T].astype(np.int32)).cuda()
        ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots)
        y = L.linear_fused_t(d.x[:T].contiguous(), d.W0, d.A, d.B, ids_t, d.scale, ws)
        torch.cuda.synchronize()
        ref = O.lora_linear(w.x[:T], w.W0, A_pool, B_pool, scale, ids[:T])
        check_close(host(y), ref, f"layer after upload, T={T}")
