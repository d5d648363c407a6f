"""Ragged-rank adapter pools on the GPU against the CPU fp64 oracle.

Each adapter keeps its own rank (stored at the next of 8, 16, 32, 64, 128)
instead of the pool's largest ([Concepts, "When It Falls Down"]; [Blog,
"Batching across different adapters"]).  The oracle evaluates every adapter
at its own rank (lora_linear_ragged).  Pool entries that would read outside
the pools are flagged and read as base-only.
"""
import numpy as np
import pytest

from oracle import lora_ref as O
from lora_serving_device_gb300 import workloads as W

from tests.gpu_util import dev, host, torch_mod
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


# T, d_in, d_out, n_slots, ranks drawn per slot
RAGGED_CASES = [
    (1, 64, 128, 3, (8,)),
    (5, 200, 136, 7, (8, 16, 24, 64)),
    (33, 256, 384, 5, (8, 128, 40)),
    (64, 512, 1024, 40, (8, 16, 64)),
    (7, 1032, 600, 4, (16, 32)),
    (48, 2056, 2120, 9, (8, 16, 64, 128)),
    (200, 640, 136, 30, (8, 16, 32, 64, 128)),
    (256, 1024, 4096, 20, (8, 16, 64)),
    # larger batches run as 256-token chunks
    (300, 256, 384, 10, (8, 16, 64)),
    (700, 520, 264, 25, (8, 32, 128)),
]


class RaggedCase:
    """A seeded case whose slot a has rank ranks[a]: the oracle's per-adapter
    lists and the device's packed pool."""

    def __init__(self, L, seed, T, d_in, d_out, n_slots, rank_set, invalid=0, W0_zero=False):
        torch = torch_mod()
        r_pad = max(rank_set)
        w = W.random_case(seed, T, d_in, d_out, r_pad, n_slots, invalid=invalid)
        rng = np.random.default_rng([seed, 17])
        self.ranks = [int(r) for r in rng.choice(np.array(rank_set), size=n_slots)]
        self.w = w
        self.A_list = [w.A_pool[a][:, :r] for a, r in enumerate(self.ranks)]
        self.B_list = [w.B_pool[a][:r] for a, r in enumerate(self.ranks)]
        self.x = dev(w.x)
        self.W0 = dev(np.zeros_like(w.W0) if W0_zero else w.W0)
        self.ids = torch.from_numpy(w.slot_ids.astype(np.int32)).cuda()
        self.scale = torch.from_numpy(w.scale.astype(np.float32)).cuda()
        self.pool = L.RaggedPool([dev(a) for a in self.A_list], [dev(b) for b in self.B_list])
        self.W0_host = np.zeros_like(w.W0) if W0_zero else w.W0

    def ref(self, ids=None):
        w = self.w
        return O.lora_linear_ragged(w.x, self.W0_host, self.A_list, self.B_list, w.scale,
                                    w.slot_ids if ids is None else ids)


@pytest.mark.parametrize("case", RAGGED_CASES, ids=[str(c) for c in RAGGED_CASES])
def test_fused_ragged_matches_oracle(L, case):
    torch = torch_mod()
    T, d_in, d_out, n_slots, rank_set = case
    for W0_zero in (False, True):
        c = RaggedCase(L, 900 + T, T, d_in, d_out, n_slots, rank_set, W0_zero=W0_zero)
        ws = L.workspace(L.OP_LINEAR_FUSED, min(T, 256), d_in, d_out, c.pool.r_max, n_slots)
        y = L.linear_fused_ragged_t(c.x, c.W0, c.pool, c.ids, c.scale, ws)
        torch.cuda.synchronize()
        ref = c.ref()
        if W0_zero:   # the adapter term alone: base rounding cannot hide an error in it
            check_close_bf16_out(host(y), ref, "ragged delta")
        else:
            check_close_bf16_out(host(y), ref, "ragged y")
        assert L.get_error_t(ws) == 0


@pytest.mark.parametrize("case", RAGGED_CASES[:6], ids=[str(c) for c in RAGGED_CASES[:6]])
def test_bgmv_adapter_ragged_matches_oracle(L, case):
    """The fp32 adapter term over a ragged pool (nothing rounded to bf16 on
    this path, so the bar is fp32 accumulation)."""
    torch = torch_mod()
    T, d_in, d_out, n_slots, rank_set = case
    c = RaggedCase(L, 950 + T, T, d_in, d_out, n_slots, rank_set, invalid=1, W0_zero=True)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    delta = torch.full((T, d_out), 7.0, dtype=torch.float32, device="cuda")
    L.bgmv_adapter_ragged_t(c.x, c.pool, c.ids, c.scale, ws, delta=delta)
    torch.cuda.synchronize()
    ids = c.w.slot_ids
    valid = (ids >= 0) & (ids < n_slots)
    got = host(delta)
    check_close(got[valid], c.ref()[valid], "ragged adapter term", rel_fro=2e-5, max_rms=2e-4)
    assert np.all(got[~valid] == 7.0)
    assert L.get_error_t(ws) == L.DEVERR_BAD_SLOT


def test_ragged_bad_entries_are_flagged_and_base_only(L):
    """Table entries that would read outside the pools or break row alignment
    are not read: the error word says so and those tokens get the base term."""
    torch = torch_mod()
    T, d_in, d_out, n_slots = 96, 256, 264, 8
    c = RaggedCase(L, 971, T, d_in, d_out, n_slots, (8, 16, 64))
    ids = np.arange(T, dtype=np.int32) % n_slots
    c.ids = torch.from_numpy(ids).cuda()
    rank = c.pool.rank.clone()
    a_off = c.pool.a_off.clone()
    b_off = c.pool.b_off.clone()
    bad = {1: "rank", 2: "a_off", 3: "b_off", 4: "a_end", 5: "r_max"}
    c.pool.rank[1] = 12                                   # not a stored rank class
    c.pool.a_off[2] += 4                                  # rows not 16-byte aligned
    c.pool.b_off[3] = c.pool.B_flat.numel()               # starts at the pool's end
    c.pool.a_off[4] = c.pool.A_flat.numel() - 8           # runs past the pool's end
    c.pool.rank[5] = 128                                  # above r_max (the pool's 64)
    ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, c.pool.r_max, n_slots)
    y = L.linear_fused_ragged_t(c.x, c.W0, c.pool, c.ids, c.scale, ws)
    torch.cuda.synchronize()
    ref_ids = np.where(np.isin(ids, list(bad)), -1, ids)
    check_close_bf16_out(host(y), c.ref(ref_ids), "ragged y with bad entries")
    assert L.get_error_t(ws) == L.DEVERR_BAD_RANK
    c.pool.rank.copy_(rank)
    c.pool.a_off.copy_(a_off)
    c.pool.b_off.copy_(b_off)


def test_ragged_stack_projection(L):
    """Two projections of the 8B-shaped stack with its adapters at their own
    ranks (8, 16 or 64) against the oracle."""
    torch = torch_mod()
    ranks = W.stack_ranks()
    ids = W.stack_ids()
    n_slots = 250
    ids_d = torch.from_numpy(ids).cuda()
    scale = torch.full((n_slots,), W.SCALE, dtype=torch.float32, device="cuda")
    used = np.unique(ids[ids >= 0])
    for layer, proj in ((0, 0), (7, 6)):
        t = W.stack_layer_device(layer, proj, ranks=ranks)
        _, d_in, d_out = W.STACK_PROJECTIONS[proj]
        pool = L.RaggedPool.from_padded(t["A_pool"], t["B_pool"], ranks)
        ws = L.workspace(L.OP_LINEAR_FUSED, 256, d_in, d_out, pool.r_max, n_slots)
        y = L.linear_fused_ragged_t(t["x"], t["W0"], pool, ids_d, scale, ws)
        torch.cuda.synchronize()
        A_list = [None] * n_slots      # slots no token uses are never read
        B_list = [None] * n_slots
        for j in used:
            A_list[j] = host(t["A_pool"][int(j)][:, :ranks[j]])
            B_list[j] = host(t["B_pool"][int(j)][:ranks[j]])
        ref = O.lora_linear_ragged(host(t["x"]), host(t["W0"]), A_list, B_list,
                                   np.full(n_slots, W.SCALE), ids)
        check_close(host(y), ref, f"ragged stack layer {layer} proj {proj}")
        assert L.get_error_t(ws) == 0
        del t, pool
        torch.cuda.empty_cache()


# prefill route (T > 256 with a workspace for it): the batch's adapters copied
# into a dense pool at r_max, then the prefill path; T, d_in, d_out, n_slots, ranks
RAGGED_PREFILL_CASES = [
    (300, 256, 384, 10, (8, 16, 64)),
    (700, 520, 264, 25, (8, 32, 128)),
    (1000, 1024, 4104, 40, (8, 16, 64)),
    (513, 264, 520, 600, (16, 64)),             # more slots than tokens: n_c = T
    (4096, 512, 5120, 12, (8, 16, 64)),         # enough 256 x 256 tiles for the wide form
]


@pytest.mark.parametrize("case", RAGGED_PREFILL_CASES, ids=[str(c) for c in RAGGED_PREFILL_CASES])
def test_fused_ragged_prefill_route_matches_oracle(L, case):
    """With the ragged layer's own workspace, batches above 256 tokens read W0
    once through the prefill path over a compact padded copy of their
    adapters; the result must still be the per-rank oracle's."""
    torch = torch_mod()
    T, d_in, d_out, n_slots, rank_set = case
    for W0_zero in (False, True):
        c = RaggedCase(L, 1600 + T, T, d_in, d_out, n_slots, rank_set, W0_zero=W0_zero)
        ws = L.workspace(L.OP_LINEAR_FUSED_RAGGED, T, d_in, d_out, c.pool.r_max, n_slots)
        y = L.linear_fused_ragged_t(c.x, c.W0, c.pool, c.ids, c.scale, ws)
        torch.cuda.synchronize()
        what = "ragged prefill route delta" if W0_zero else "ragged prefill route y"
        check_close_bf16_out(host(y), c.ref(), what)
        assert L.get_error_t(ws) == 0


def test_ragged_prefill_route_bad_entries_and_ids(L):
    """On the prefill route, slots with bad table entries are copied as zeros
    (their tokens get the base term, BAD_RANK raised) and ids outside
    [-1, n_slots) are base-only (BAD_SLOT raised)."""
    torch = torch_mod()
    T, d_in, d_out, n_slots = 600, 256, 264, 8
    c = RaggedCase(L, 1701, T, d_in, d_out, n_slots, (8, 16, 64))
    ids = (np.arange(T, dtype=np.int32) * 7) % n_slots
    ids[::50] = -1
    ids[3::97] = n_slots + 3                              # invalid ids
    c.ids = torch.from_numpy(ids).cuda()
    saved = (c.pool.rank.clone(), c.pool.a_off.clone())
    c.pool.rank[1] = 12                                   # not a stored rank class
    c.pool.a_off[2] = c.pool.A_flat.numel() - 8           # runs past the pool's end
    ws = L.workspace(L.OP_LINEAR_FUSED_RAGGED, T, d_in, d_out, c.pool.r_max, n_slots)
    y = L.linear_fused_ragged_t(c.x, c.W0, c.pool, c.ids, c.scale, ws)
    torch.cuda.synchronize()
    ref_ids = np.where(np.isin(ids, [1, 2]) | (ids >= n_slots), -1, ids)
    check_close_bf16_out(host(y), c.ref(ref_ids), "ragged prefill route, bad entries and ids")
    assert L.get_error_t(ws) == L.DEVERR_BAD_RANK | L.DEVERR_BAD_SLOT
    c.pool.rank.copy_(saved[0])
    c.pool.a_off.copy_(saved[1])


@pytest.mark.parametrize("ids_kind", ["all_base", "one_slot", "257_mixed"])
def test_ragged_prefill_route_edges(L, ids_kind):
    """The prefill route's edges: every token base-only (no segment, nothing
    copied), every token on one slot, and the smallest batch that takes the
    route (257 tokens), each against the oracle."""
    torch = torch_mod()
    d_in, d_out, n_slots = 264, 520, 6
    T = 257 if ids_kind == "257_mixed" else 300
    c = RaggedCase(L, 1750 + len(ids_kind), T, d_in, d_out, n_slots, (8, 16, 32, 64, 128))
    if ids_kind == "all_base":
        ids = np.full(T, -1, np.int32)
    elif ids_kind == "one_slot":
        ids = np.full(T, 3, np.int32)
    else:
        ids = c.w.slot_ids.copy()
    c.ids = torch.from_numpy(ids).cuda()
    ws = L.workspace(L.OP_LINEAR_FUSED_RAGGED, T, d_in, d_out, c.pool.r_max, n_slots)
    y = L.linear_fused_ragged_t(c.x, c.W0, c.pool, c.ids, c.scale, ws)
    torch.cuda.synchronize()
    check_close_bf16_out(host(y), c.ref(ids), f"ragged prefill route, {ids_kind}")
    assert L.get_error_t(ws) == 0
