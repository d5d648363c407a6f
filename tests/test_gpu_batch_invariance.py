"""Batch-composition invariance of the decode adapter term on the GPU.

The one-launch adapter term and its merge form (the last kernel of the decode
layer) gather each token's own adapter ([Handbook], "Not merging the weights,
computing in batches": the batched forms compute every row with its own
adapter, whatever the other rows hold).  So, whatever mix of ids a batch has:
- every run length of equal ids, base-only rows and invalid ids included,
  meets the oracle bar;
- a token's output does not depend on the other tokens of the batch:
  permuting the batch permutes the output bit for bit, and a token whose
  batch-mates are all base-only gives the same bits as in the full batch.
"""
import numpy as np
import pytest

from oracle import lora_ref as O
from lora_serving_device_gb300 import workloads as W

from tests.gpu_util import DeviceCase, dev, host, torch_mod
from tests.tolerances import check_close, check_close_bf16_out

pytestmark = pytest.mark.gpu

# tokens per adapter: single tokens, short runs and long runs
RUN_LENGTHS = (1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 13, 16, 17, 31)


@pytest.fixture(scope="module")
def L():
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from lora_serving_device_gb300 import build, lora
    build.build()
    lora.load()
    return lora


def grouped_ids(T, n_slots, seed, n_base=9, n_invalid=3):
    """T ids in which adapter j (distinct slots) gets RUN_LENGTHS[j] tokens,
    cycling, plus n_base base-only rows and n_invalid invalid ids, shuffled."""
    rng = np.random.default_rng([seed, 41])
    ids = []
    slots = rng.permutation(n_slots)
    j = 0
    while len(ids) < T - n_base - n_invalid:
        m = RUN_LENGTHS[j % len(RUN_LENGTHS)]
        ids += [int(slots[j % n_slots])] * m
        j += 1
    ids = ids[:T - n_base - n_invalid] + [-1] * n_base + [n_slots, -5, 1 << 30][:n_invalid]
    return rng.permutation(np.array(ids, dtype=np.int32))


def case_with_ids(seed, T, d_in, d_out, r, n_slots, ids):
    w = W.random_case(seed, T, d_in, d_out, r, n_slots)
    w.slot_ids = ids.astype(np.int32)
    return w


ITEM_CASES = [(257, 520, 1032, 16, 40), (200, 1024, 2056, 64, 30), (64, 4096, 4096, 16, 20),
              (256, 264, 136, 128, 25), (96, 2048, 4104, 32, 12)]


@pytest.mark.parametrize("case", ITEM_CASES, ids=[str(c) for c in ITEM_CASES])
def test_adapter_term_every_run_length(L, case):
    """Delta and merge forms against the oracle on ids with runs of every
    length (the scan runs over more than 256 ids at T = 257)."""
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    w = case_with_ids(1200 + T, T, d_in, d_out, r, n_slots, grouped_ids(T, n_slots, T))
    d = DeviceCase(w)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    delta = torch.full((T, d_out), 7.0, dtype=torch.float32, device="cuda")
    L.bgmv_adapter_t(d.x, d.A, d.B, d.ids, d.scale, ws, delta=delta)
    torch.cuda.synchronize()
    term = O.expand(O.shrink(w.x, w.A_pool, w.scale, w.slot_ids), w.B_pool, w.slot_ids)
    ids = w.slot_ids
    valid = (ids >= 0) & (ids < n_slots)
    got = host(delta)
    check_close(got[valid], term[valid], "adapter term, every run length", rel_fro=2e-5,
                max_rms=2e-4)
    assert np.all(got[~valid] == 7.0)
    assert L.get_error_t(ws) & L.DEVERR_BAD_SLOT

    S = 3
    part = (np.random.default_rng([7013, T]).standard_normal((S, T, d_out)) * 0.3).astype(np.float32)
    y = torch.full((T, d_out), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.bgmv_adapter_merge_t(d.x, d.A, d.B, d.ids, d.scale, dev(part, "f32"), ws, y=y)
    torch.cuda.synchronize()
    check_close_bf16_out(host(y), part.astype(np.float64).sum(axis=0) + term,
                         "partials + adapter term, every run length")


@pytest.mark.parametrize("case", ITEM_CASES, ids=[str(c) for c in ITEM_CASES])
def test_adapter_term_independent_of_grouping(L, case):
    """Permuting the batch permutes the adapter term and the merged y bit for
    bit, and a token whose batch-mates are all made base-only (same T, so the
    same cluster split of d_in) gives the same bits as in the full batch."""
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    w = case_with_ids(1300 + T, T, d_in, d_out, r, n_slots, grouped_ids(T, n_slots, T + 1))
    d = DeviceCase(w)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    S = 2
    part = torch.from_numpy(
        (np.random.default_rng([7014, T]).standard_normal((S, T, d_out)) * 0.3).astype(np.float32)
    ).cuda()

    def run(x, ids, p):
        delta = torch.zeros((x.shape[0], d_out), dtype=torch.float32, device="cuda")
        L.bgmv_adapter_t(x, d.A, d.B, ids, d.scale, ws, delta=delta)
        y = torch.empty((x.shape[0], d_out), dtype=torch.bfloat16, device="cuda")
        L.bgmv_adapter_merge_t(x, d.A, d.B, ids, d.scale, p, ws, y=y)
        torch.cuda.synchronize()
        return delta, y

    delta, y = run(d.x, d.ids, part)
    perm = torch.from_numpy(np.random.default_rng([T, 5]).permutation(T)).cuda()
    delta_p, y_p = run(d.x[perm].contiguous(), d.ids[perm].contiguous(),
                       part[:, perm].contiguous())
    assert torch.equal(delta_p, delta[perm])
    assert torch.equal(y_p.view(torch.int16), y[perm].view(torch.int16))
    # tokens of the longest runs, alone in the batch
    ids = w.slot_ids
    vals, counts = np.unique(ids[(ids >= 0) & (ids < n_slots)], return_counts=True)
    for a in vals[np.argsort(-counts)][:2]:
        for t in np.nonzero(ids == a)[0][[0, -1]]:
            t = int(t)
            lone = np.full(T, -1, np.int32)
            lone[t] = a
            d1, y1 = run(d.x, torch.from_numpy(lone).cuda(), part)
            assert torch.equal(d1[t], delta[t]), (a, t)
            assert torch.equal(y1[t].view(torch.int16), y[t].view(torch.int16)), (a, t)


@pytest.mark.parametrize("T", [1, 5, 64, 256])
def test_fused_layer_one_adapter_for_all(L, T):
    """Every token on one adapter (the longest possible runs) through the
    decode chain of the fused layer, and all base-only."""
    torch = torch_mod()
    d_in, d_out, r, n_slots = 1024, 2056, 16, 6
    for ids in (np.full(T, 4, np.int32), np.full(T, -1, np.int32)):
        w = case_with_ids(1400 + T, T, d_in, d_out, r, n_slots, ids)
        d = DeviceCase(w)
        y, ws = d.fused()
        torch.cuda.synchronize()
        ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
        check_close_bf16_out(host(y), ref, f"fused layer, ids all {ids[0]}")
        assert L.get_error_t(ws) == 0


def test_ragged_every_run_length_and_lone_tokens(L):
    """Ragged-rank pool: each token runs at its slot's rank; the layer meets
    the bar on every run length, and a token whose batch-mates are all
    base-only gives the same adapter term bits as in the full batch."""
    torch = torch_mod()
    T, d_in, d_out, n_slots = 200, 1032, 1032, 24
    ranks_set = np.array([8, 16, 32, 64, 128])
    rng = np.random.default_rng(1500)
    ranks = [int(v) for v in rng.choice(ranks_set, size=n_slots)]
    w = case_with_ids(1500, T, d_in, d_out, 128, n_slots, grouped_ids(T, n_slots, 77))
    A_list = [w.A_pool[a][:, :rk] for a, rk in enumerate(ranks)]
    B_list = [w.B_pool[a][:rk] for a, rk in enumerate(ranks)]
    pool = L.RaggedPool([dev(a) for a in A_list], [dev(b) for b in B_list])
    x = dev(w.x)
    W0 = dev(w.W0)
    idt = torch.from_numpy(w.slot_ids).cuda()
    scale = torch.from_numpy(w.scale.astype(np.float32)).cuda()
    ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, pool.r_max, n_slots)
    y = L.linear_fused_ragged_t(x, W0, pool, idt, scale, ws)
    torch.cuda.synchronize()
    ref = O.lora_linear_ragged(w.x, w.W0, A_list, B_list, w.scale, w.slot_ids)
    check_close_bf16_out(host(y), ref, "ragged layer, every run length")
    assert L.get_error_t(ws) & L.DEVERR_BAD_SLOT
    ws2 = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    delta = L.bgmv_adapter_ragged_t(x, pool, idt, scale, ws2)
    torch.cuda.synchronize()
    ids = w.slot_ids
    for t in np.nonzero((ids >= 0) & (ids < n_slots))[0][::23]:
        t = int(t)
        lone = np.full(T, -1, np.int32)
        lone[t] = ids[t]
        d1 = L.bgmv_adapter_ragged_t(x, pool, torch.from_numpy(lone).cuda(), scale, ws2)
        torch.cuda.synchronize()
        assert torch.equal(d1[t], delta[t]), t
