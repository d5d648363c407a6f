"""Seeded synthetic inputs for the multi-LoRA batched linear layer.

This module only DRAWS inputs. It holds none of the layer's arithmetic, so the
CPU oracle (``oracle/``) and the CUDA path can both be fed from it without
sharing any of the method's code.

Sources, cited below by short name (web pages on multi-LoRA serving):
  [Handbook] "Serving multiple LoRAs: segmented matrix multiplies and adapter
             scheduling" (anrans.github.io, ai-infra-handbooks)
  [Blog]     "Serving many LoRA adapters" (blog.ecitis.org)
  [Concepts] "Serving Many LoRA Adapters" (praveentn.live)

Workloads (every one is seeded; workload c draws from streams keyed on 1000 + c):
  1 toy_mixed_batch  -- [Handbook, "Not merging the weights, computing in
                        batches"]: 256->256, rank 16, 8 adapters, requests of
                        lengths [1,1,37,1,12,1] on adapters [3,5,3,0,7,5]; fp32.
  2 decode_bgmv      -- 4096->4096, rank 16, 256 slots, 64 one-token requests,
                        ids Zipf(1.1) over the pool, 8 rows base-only; bf16.
  3 prefill_sgmv     -- 4096->14336, rank 64, 64 slots, 16 prefill requests of
                        lengths U[64,1024] on 16 distinct adapters + 48 decode
                        tokens on uniform adapters; bf16.
  4 diversity_sweep  -- 4096->4096, rank 16, 1024 slots, T tokens spread evenly
                        over k distinct adapters; bf16.
  5 stack_8b         -- 32 layers x 7 projections of an 8B-shaped decoder,
                        250 slots with ranks {8,16,64} zero-padded to 64,
                        T=256 (4x48 prefill + 64 decode), Zipf(1.1), 10% of
                        the requests base-only; bf16.  Its weights (~94 GB)
                        are drawn on the device, see ``stack_layer_device``.

Init for workloads 2-5: W0 ~ N(0, 0.02), A ~ N(0, 1/sqrt(4096)) (std 1/64),
B ~ N(0, 0.02), x ~ N(0, 1), scale alpha/r = 2 for every slot.  N(0, s) is read
as standard deviation s.  bf16 inputs are drawn in fp32 and rounded to the
nearest bf16 (ties to even) here, so both sides see identical values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 1000

# stream ids inside one workload's seed
_S_IDS, _S_X, _S_W0, _S_A, _S_B, _S_RANK = 0, 1, 2, 3, 4, 5

W0_STD = 0.02
A_STD = 1.0 / 64.0
B_STD = 0.02
SCALE = 2.0

# The 7 adapted projections of an 8B-shaped decoder layer: (name, d_in, d_out)
STACK_PROJECTIONS = (
    ("q", 4096, 4096),
    ("k", 4096, 1024),
    ("v", 4096, 1024),
    ("o", 4096, 4096),
    ("gate", 4096, 14336),
    ("up", 4096, 14336),
    ("down", 14336, 4096),
)
STACK_LAYERS = 32


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 value (ties to even); returns fp32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The uint16 bit patterns of already bf16-representable fp32 values."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _rng(key, *stream):
    return np.random.default_rng([SEED_BASE + key if isinstance(key, int) else key, *stream])


def zipf_probs(n_slots: int, s: float = 1.1) -> np.ndarray:
    """Truncated Zipf over slots 0..n_slots-1: p(j) proportional to (j+1)^-s."""
    w = (np.arange(n_slots, dtype=np.float64) + 1.0) ** (-s)
    return w / w.sum()


@dataclass
class Workload:
    name: str
    dtype: str                 # "bf16" or "f32": the arithmetic type of the inputs
    T: int
    d_in: int
    d_out: int
    r: int
    n_slots: int
    x: np.ndarray              # [T, d_in] fp32 (bf16-representable for bf16)
    W0: np.ndarray             # [d_in, d_out]
    A_pool: np.ndarray         # [n_slots, d_in, r]
    B_pool: np.ndarray         # [n_slots, r, d_out]
    scale: np.ndarray          # [n_slots] fp32 (alpha/r travels with the adapter)
    slot_ids: np.ndarray       # [T] int32, -1 = base only
    req_lengths: list = field(default_factory=list)
    req_slots: list = field(default_factory=list)
    meta: dict = field(default_factory=dict)

    @property
    def distinct(self) -> int:
        ids = self.slot_ids
        return int(np.unique(ids[(ids >= 0) & (ids < self.n_slots)]).size)


def _normal(rng, shape, std, dtype_bf16: bool) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return bf16_round(a) if dtype_bf16 else a


def nf4_like_codebook():
    """A 16-entry 4-bit codebook of normal-float kind: levels at quantiles of
    N(0, 1) (8 above zero, 7 below, and an exact zero), scaled so the
    extremes are -1 and +1, rounded to bf16 (returned as float32).  The
    pages name QLoRA-style 4-bit bases without listing levels; this is one
    codebook of that family, an input like the weights."""
    from statistics import NormalDist
    nd = NormalDist()
    p_top = 0.97
    pos = [nd.inv_cdf(0.5 + (p_top - 0.5) * i / 8) for i in range(1, 9)]
    neg = [-nd.inv_cdf(0.5 + (p_top - 0.5) * i / 7) for i in range(1, 8)]
    top = pos[-1]
    vals = sorted([v / top for v in neg] + [0.0] + [v / top for v in pos])
    vals[0], vals[-1] = -1.0, 1.0
    return bf16_round(np.array(vals, np.float32))


def pack_nibbles(codes):
    """Byte layout of a 4-bit matrix [d_in, d_out] -> [d_out, d_in / 2] uint8,
    k contiguous per column: byte i of row n holds rows 2i (low nibble) and
    2i + 1 (high nibble) of column n."""
    c = np.ascontiguousarray(np.asarray(codes, np.uint8).T)
    return (c[:, 0::2] | (c[:, 1::2] << np.uint8(4))).astype(np.uint8)


def random_4bit_base(seed, d_in, d_out):
    """Seeded 4-bit base inputs: codes uniform over 0..15 and bf16 block
    scales in [0.005, 0.05] (absmax [d_in / 64, d_out])."""
    rng = np.random.default_rng([SEED_BASE, 41, seed])
    codes = rng.integers(0, 16, (d_in, d_out)).astype(np.uint8)
    absmax = bf16_round(rng.uniform(0.005, 0.05, (d_in // 64, d_out)).astype(np.float32))
    return codes, absmax


def make_pools(key, n_slots, d_in, d_out, r, slots=None, bf16=True,
               a_std=A_STD, b_std=B_STD, ranks=None):
    """Adapter pools, drawn slot by slot from per-slot streams.

    ``slots`` limits the draw to the listed slots (the others stay zero); a
    slot's values do not depend on which other slots were drawn.  ``ranks``
    (per slot) zero-pads A columns and B rows at and beyond the slot's rank.
    """
    A = np.zeros((n_slots, d_in, r), np.float32)
    B = np.zeros((n_slots, r, d_out), np.float32)
    todo = range(n_slots) if slots is None else sorted(set(int(s) for s in slots))
    for j in todo:
        A[j] = _normal(_rng(key, _S_A, j), (d_in, r), a_std, bf16)
        B[j] = _normal(_rng(key, _S_B, j), (r, d_out), b_std, bf16)
        if ranks is not None and ranks[j] < r:
            A[j, :, ranks[j]:] = 0.0
            B[j, ranks[j]:, :] = 0.0
    return A, B


def _requests_to_ids(lengths, slots):
    return np.repeat(np.asarray(slots, np.int32), np.asarray(lengths, np.int64)).astype(np.int32)


def toy_mixed_batch() -> Workload:
    """Workload 1: the toy mixed batch of [Handbook, "Not merging the weights,
    computing in batches"] (its shapes and distributions; our own seed)."""
    key = 1
    d_in = d_out = 256
    r, n_slots = 16, 8
    lengths = [1, 1, 37, 1, 12, 1]
    slots = [3, 5, 3, 0, 7, 5]
    T = sum(lengths)
    W0 = _normal(_rng(key, _S_W0), (d_in, d_out), 1.0 / 16.0, False)
    A, B = make_pools(key, n_slots, d_in, d_out, r, bf16=False, a_std=1.0 / 16.0, b_std=0.25)
    x = _normal(_rng(key, _S_X), (T, d_in), 1.0, False)
    return Workload("toy_mixed_batch", "f32", T, d_in, d_out, r, n_slots, x, W0, A, B,
                    np.full(n_slots, SCALE, np.float32), _requests_to_ids(lengths, slots),
                    list(lengths), list(slots), {"config": 1})


def decode_ids(key, T=64, n_slots=256, n_base=8):
    rng = _rng(key, _S_IDS)
    base_pos = rng.choice(T, size=n_base, replace=False)
    ids = rng.choice(n_slots, size=T, p=zipf_probs(n_slots)).astype(np.int32)
    ids[base_pos] = -1
    return ids


def decode_bgmv(with_weights=True) -> Workload:
    """Workload 2: one q_proj-shaped decode layer, 64 one-token requests."""
    key = 2
    T, d_in, d_out, r, n_slots = 64, 4096, 4096, 16, 256
    ids = decode_ids(key, T, n_slots, 8)
    return _dense(key, "decode_bgmv", T, d_in, d_out, r, n_slots, ids,
                  [1] * T, ids.tolist(), with_weights)


def prefill_ids(key=3, n_slots=64):
    rng = _rng(key, _S_IDS)
    pre_slots = rng.choice(n_slots, size=16, replace=False).astype(np.int32)
    pre_len = rng.integers(64, 1025, size=16)
    dec_slots = rng.integers(0, n_slots, size=48).astype(np.int32)
    lengths = pre_len.tolist() + [1] * 48
    slots = pre_slots.tolist() + dec_slots.tolist()
    return lengths, slots


def prefill_sgmv(with_weights=True) -> Workload:
    """Workload 3: gate/up-shaped prefill layer, mixed prefill + decode batch."""
    key = 3
    d_in, d_out, r, n_slots = 4096, 14336, 64, 64
    lengths, slots = prefill_ids(key, n_slots)
    ids = _requests_to_ids(lengths, slots)
    return _dense(key, "prefill_sgmv", int(ids.size), d_in, d_out, r, n_slots, ids,
                  lengths, slots, with_weights)


def sweep_ids(T, k, n_slots=1024):
    """Workload 4 ids: k distinct slots, exactly T/k tokens each, shuffled."""
    if T % k:
        raise ValueError("T must be a multiple of k")
    rng = _rng(4, _S_IDS, T, k)
    chosen = rng.choice(n_slots, size=k, replace=False).astype(np.int32)
    ids = chosen[np.arange(T) % k]
    return ids[rng.permutation(T)].astype(np.int32)


SWEEP_POINTS = tuple([(32, k) for k in (1, 2, 4, 8, 16, 32)] +
                     [(256, k) for k in (1, 2, 4, 8, 16, 32, 64, 128, 256)])


def diversity_sweep(T, k, with_weights=True, only_used_slots=False) -> Workload:
    """Workload 4: one 4096->4096 rank-16 layer over a 1024-slot pool."""
    key = 4
    d_in, d_out, r, n_slots = 4096, 4096, 16, 1024
    ids = sweep_ids(T, k, n_slots)
    w = _dense(key, f"diversity_sweep_T{T}_k{k}", T, d_in, d_out, r, n_slots, ids,
               [1] * T, ids.tolist(), with_weights,
               pool_slots=(np.unique(ids) if only_used_slots else None),
               x_stream=(T, k))
    w.meta.update({"T": T, "k": k})
    return w


def _dense(key, name, T, d_in, d_out, r, n_slots, ids, lengths, slots, with_weights,
           pool_slots=None, x_stream=()):
    if with_weights:
        W0 = _normal(_rng(key, _S_W0), (d_in, d_out), W0_STD, True)
        A, B = make_pools(key, n_slots, d_in, d_out, r, slots=pool_slots)
    else:
        W0 = np.zeros((0, 0), np.float32)
        A = np.zeros((0, 0, 0), np.float32)
        B = np.zeros((0, 0, 0), np.float32)
    x = _normal(_rng(key, _S_X, *x_stream), (T, d_in), 1.0, True)
    return Workload(name, "bf16", T, d_in, d_out, r, n_slots, x, W0, A, B,
                    np.full(n_slots, SCALE, np.float32), ids.astype(np.int32),
                    list(lengths), list(slots), {"config": key})


def random_case(seed, T, d_in, d_out, r, n_slots, base_frac=0.15, runs=False,
                bf16=True, invalid=0) -> Workload:
    """A generic seeded case for tile-edge parity tests: ids uniform over the
    pool (or as runs of equal ids when ``runs``), a fraction base-only, and
    ``invalid`` ids outside [-1, n_slots) planted at random positions.  The
    init follows the decode workload (A std 1/sqrt(d_in), so x A ~ N(0, 1);
    W0 and B std 0.02) with a per-slot scale drawn from U[0.5, 2.5]."""
    key = ("case", seed)
    rng = np.random.default_rng([SEED_BASE, 99, seed])
    if runs:
        lengths, slots = [], []
        left = T
        while left > 0:
            n = int(min(left, rng.integers(1, max(2, T // 3) + 1)))
            lengths.append(n)
            slots.append(int(rng.integers(0, n_slots)))
            left -= n
        ids = _requests_to_ids(lengths, slots)
    else:
        ids = rng.integers(0, n_slots, size=T).astype(np.int32)
    nb = int(round(base_frac * T))
    if nb:
        ids[rng.choice(T, size=nb, replace=False)] = -1
    if invalid:
        pos = rng.choice(T, size=invalid, replace=False)
        bad = np.array([n_slots, n_slots + 7, -2, -100, 1 << 30], np.int32)
        ids[pos] = bad[np.arange(invalid) % bad.size]
    std_scale = 1.0
    W0 = _normal(np.random.default_rng([SEED_BASE, 99, seed, 2]), (d_in, d_out), W0_STD, bf16)
    A = np.stack([_normal(np.random.default_rng([SEED_BASE, 99, seed, 3, j]), (d_in, r),
                          std_scale / np.sqrt(d_in), bf16) for j in range(n_slots)]) \
        if n_slots else np.zeros((0, d_in, r), np.float32)
    B = np.stack([_normal(np.random.default_rng([SEED_BASE, 99, seed, 4, j]), (r, d_out),
                          B_STD, bf16) for j in range(n_slots)]) \
        if n_slots else np.zeros((0, r, d_out), np.float32)
    x = _normal(np.random.default_rng([SEED_BASE, 99, seed, 1]), (T, d_in), 1.0, bf16)
    scale = (np.random.default_rng([SEED_BASE, 99, seed, 6]).uniform(0.5, 2.5, n_slots)
             .astype(np.float32))
    return Workload(f"case{seed}", "bf16" if bf16 else "f32", T, d_in, d_out, r, n_slots,
                    x, W0, A, B, scale, ids, [], [], {"seed": seed})


# ---------------------------------------------------------------------------
# Workload 5: the 8B-shaped stack.  Ids and ranks are drawn on the host; the
# ~94 GB of weights are drawn on the device with torch's seeded generator and
# the parts a parity check needs are copied back to the host.
# ---------------------------------------------------------------------------

def stack_requests(n_slots=250):
    """Request layout of workload 5: 4 prefill requests of 48 tokens, then 64
    one-token decode requests; round(0.1 * 68) = 7 requests are base-only."""
    rng = _rng(5, _S_IDS)
    n_req = 4 + 64
    lengths = [48] * 4 + [1] * 64
    slots = rng.choice(n_slots, size=n_req, p=zipf_probs(n_slots)).astype(np.int32)
    slots[rng.choice(n_req, size=7, replace=False)] = -1
    return lengths, slots.tolist()


def stack_ranks(n_slots=250):
    """Per-adapter ranks of workload 5, uniform over {8, 16, 64}."""
    return _rng(5, _S_RANK).choice(np.array([8, 16, 64]), size=n_slots).astype(np.int32)


def stack_ids(n_slots=250):
    lengths, slots = stack_requests(n_slots)
    return _requests_to_ids(lengths, slots)


def stack_layer_device(layer: int, proj: int, device="cuda", n_slots=250, r_pad=64,
                       ranks=None, want=("x", "W0", "A", "B")):
    """Draw one (layer, projection) of workload 5 on the device as bf16 tensors.

    Returns a dict with x [256, d_in], W0 [d_in, d_out], A_pool
    [n_slots, d_in, 64], B_pool [n_slots, 64, d_out], all torch.bfloat16 on
    ``device``; A columns and B rows at and beyond each slot's rank are zero.
    """
    import torch
    _, d_in, d_out = STACK_PROJECTIONS[proj]
    if ranks is None:
        ranks = stack_ranks(n_slots)
    g = torch.Generator(device=device)
    out = {}
    base = (SEED_BASE + 5) * 100000 + layer * 100 + proj * 10

    def draw(tag, shape, std):
        g.manual_seed(base + tag)
        t = torch.empty(shape, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=g)
        return t.to(torch.bfloat16)

    if "x" in want:
        out["x"] = draw(1, (256, d_in), 1.0)
    if "W0" in want:
        out["W0"] = draw(2, (d_in, d_out), W0_STD)
    rk = torch.as_tensor(ranks, device=device, dtype=torch.int32)
    if "A" in want:
        A = torch.empty((n_slots, d_in, r_pad), dtype=torch.bfloat16, device=device)
        for j0 in range(0, n_slots, 25):
            j1 = min(n_slots, j0 + 25)
            A[j0:j1] = _draw_chunk(g, base, 3, j0, (j1 - j0, d_in, r_pad), A_STD, device)
        mask = (torch.arange(r_pad, device=device)[None, :] < rk[:, None]).to(torch.bfloat16)
        A.mul_(mask[:, None, :])
        out["A_pool"] = A
    if "B" in want:
        B = torch.empty((n_slots, r_pad, d_out), dtype=torch.bfloat16, device=device)
        for j0 in range(0, n_slots, 25):
            j1 = min(n_slots, j0 + 25)
            B[j0:j1] = _draw_chunk(g, base, 4, j0, (j1 - j0, r_pad, d_out), B_STD, device)
        mask = (torch.arange(r_pad, device=device)[None, :] < rk[:, None]).to(torch.bfloat16)
        B.mul_(mask[:, :, None])
        out["B_pool"] = B
    return out


def _draw_chunk(g, base, tag, j0, shape, std, device):
    import torch
    g.manual_seed(base * 1000 + tag * 300 + j0)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t.to(torch.bfloat16)
