"""CPU fp64 oracle for the multi-LoRA batched linear layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
baseline leg of the benchmark may import this module.  The product path (the
CUDA library and its Python binding) never calls it and shares no code with it.

Sources, cited below by short name (web pages on multi-LoRA serving):
  [Guide]    "Multi-LoRA batching and adapter paging" (guide.dupenodi.dev)
  [Concepts] "Serving Many LoRA Adapters" (praveentn.live)
  [Handbook] "Serving multiple LoRAs: segmented matrix multiplies and adapter
             scheduling" (anrans.github.io, ai-infra-handbooks)
  [Blog]     "Serving many LoRA adapters" (blog.ecitis.org)

What the layer computes (row-vector form, [Handbook, "Not merging the weights,
computing in batches"]): for token t with adapter a_t,

    y_t = x_t W0 + s_{a_t} * (x_t A_{a_t}) B_{a_t}

with W0 [d_in, d_out], A_a [d_in, r], B_a [r, d_out] and s_a = alpha/r, the
scale that travels with the adapter ([Blog, "Correctness across tenants"]).
A token with id -1 gets the base term only ([Blog, "Replay" figure: "req C ->
base only"]).  Ids outside [-1, n_slots) are read as base-only as well (the
GPU path flags them in its error word).

Readings taken where the pages are silent or disagree (each listed in the
design notes):
  * the row-vector convention above ([Handbook]); [Blog, "Low-rank structure
    and additivity"] writes the same map in column-vector form;
  * the scale is applied to the shrink output, v = s (x A); mathematically the
    same as s ((x A) B);
  * segments come from a STABLE sort of the ids ([Handbook] toy script uses a
    stable argsort), -1 rows sort first and form no segment, seg_slot lists the
    ids >= 0 present in ascending order.

All arithmetic here is float64 on the (already bf16-rounded) inputs.  Every
function is pinned by tests against brute force, closed forms, invariants and
the pages' printed figures; none is pinned against itself.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def valid_ids(slot_ids, n_slots):
    """Ids as the layer reads them: anything outside [0, n_slots) -> -1."""
    ids = np.asarray(slot_ids, dtype=np.int64).copy()
    ids[(ids < 0) | (ids >= n_slots)] = -1
    return ids


def requests_from_ids(slot_ids):
    """Split a token id array into requests: maximal runs of equal ids."""
    ids = np.asarray(slot_ids)
    lengths, slots = [], []
    t = 0
    while t < ids.size:
        u = t
        while u < ids.size and ids[u] == ids[t]:
            u += 1
        lengths.append(u - t)
        slots.append(int(ids[t]))
        t = u
    return lengths, slots


def lora_linear_per_request(x, W0, A_pool, B_pool, scale, req_lengths, req_slots):
    """The layer evaluated request by request, one dense product per request.

    This is the naive form that both [Concepts, "Punica: The Segmented
    Gather-Scatter Kernel"] (its per-request pseudocode) and [Handbook, "Not
    merging the weights, computing in batches"] (its per-request reference)
    use as ground truth: base term for the request's rows, then, when the
    request has an adapter, the scaled low-rank correction (x A) B.
    """
    x, W0 = _f64(x), _f64(W0)
    n_slots = A_pool.shape[0]
    rows = []
    start = 0
    for a, n in zip(req_slots, req_lengths):
        xi = x[start:start + n]
        yi = xi @ W0
        if 0 <= a < n_slots:
            xa = xi @ _f64(A_pool[a])                  # shrink to rank r
            yi = yi + float(scale[a]) * (xa @ _f64(B_pool[a]))   # expand, add
        rows.append(yi)
        start += n
    if not rows:
        return np.zeros((0, W0.shape[1]))
    return np.concatenate(rows, axis=0)


def lora_linear(x, W0, A_pool, B_pool, scale, slot_ids):
    """Reference output y [T, d_out] for per-token ids (requests = runs)."""
    ids = valid_ids(slot_ids, A_pool.shape[0])
    lengths, slots = requests_from_ids(ids)
    return lora_linear_per_request(x, W0, A_pool, B_pool, scale, lengths, slots)


def lora_linear_gathered(x, W0, A_pool, B_pool, scale, slot_ids):
    """BGMV form ([Handbook], BGMV bullet): every token gathers its own
    adapter's A and B by index and does a matrix-vector product."""
    x, W0 = _f64(x), _f64(W0)
    ids = valid_ids(slot_ids, A_pool.shape[0])
    y = x @ W0
    has = ids >= 0
    if has.any():
        a = ids[has]
        At = _f64(A_pool)[a]                          # [n, d_in, r] gathered
        Bt = _f64(B_pool)[a]                          # [n, r, d_out] gathered
        v = np.einsum("tk,tkr->tr", x[has], At) * _f64(scale)[a][:, None]
        y[has] += np.einsum("tr,trn->tn", v, Bt)
    return y


def lora_linear_ragged(x, W0, A_list, B_list, scale, slot_ids):
    """The layer over adapters of different ranks, each kept at its own rank
    (no padding to the largest): A_list[a] [d_in, r_a], B_list[a] [r_a, d_out].
    [Blog, "Batching across different adapters"]: mixed ranks are served by
    ragged indexing or by padding; [Concepts, "When It Falls Down"] and
    [Handbook, Exercise 2]: padding changes the cost, not the result.  Per
    token: y_t = x_t W0 + s_a (x_t A_a) B_a, base only for ids outside
    [0, len(A_list))."""
    x, W0 = _f64(x), _f64(W0)
    ids = valid_ids(slot_ids, len(A_list))
    y = x @ W0
    for t in range(x.shape[0]):
        a = ids[t]
        if a >= 0:
            v = float(scale[a]) * (x[t] @ _f64(A_list[a]))     # shrink to rank r_a
            y[t] += v @ _f64(B_list[a])                        # expand, add
    return y


# ----------------------------------------------------------------------------
# 4-bit base matrix ([Concepts, "When It Falls Down"]: QLoRA-style 4-bit base
# models next to bf16 adapters).  The pages name the style, not the format;
# the reading taken: a 16-entry codebook scaled per block of 64 consecutive
# d_in rows of a column by the block's absolute maximum; a weight's code is
# the entry nearest weight / absmax; the dequantised weight is
# codebook[code] * absmax rounded once to bf16, the type of the adapter path.
# ----------------------------------------------------------------------------
Q4_BLOCK = 64


def bf16_round(a):
    """Nearest bf16 value of each fp32 value (ties to even), as float64."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def quantize_4bit(W, codebook):
    """codes [d_in, d_out] (0..15) and absmax [d_in / 64, d_out] of W.

    absmax: the largest |w| of each block; code: the entry of the codebook
    nearest w / absmax, the quotient and the distances in fp32 (ties go to
    the lower code); a block of zeros takes the entry nearest 0."""
    W = np.asarray(W, dtype=np.float32)
    cb = np.asarray(codebook, dtype=np.float32)
    d_in, d_out = W.shape
    blocks = W.reshape(d_in // Q4_BLOCK, Q4_BLOCK, d_out)
    absmax = np.abs(blocks).max(axis=1)
    safe = np.where(absmax > 0, absmax, np.float32(1.0)).astype(np.float32)
    v = np.where(absmax[:, None, :] > 0, blocks / safe[:, None, :], np.float32(0.0))
    v = v.astype(np.float32)
    best = np.abs(v - cb[0])
    codes = np.zeros(v.shape, np.uint8)
    for c in range(1, cb.size):
        d = np.abs(v - cb[c])
        better = d < best
        codes[better] = c
        best = np.where(better, d, best)
    return codes.reshape(d_in, d_out), absmax


def dequantize_4bit(codes, absmax, codebook):
    """deq[k, n] = bf16(codebook[codes[k, n]] * absmax[k // 64, n]) (fp32 product)."""
    cb = np.asarray(codebook, dtype=np.float32)
    s = np.repeat(np.asarray(absmax, dtype=np.float32), Q4_BLOCK, axis=0)
    return bf16_round(cb[np.asarray(codes)] * s)


def pack_4bit(codes):
    """The stored code matrix [d_out, d_in / 2] of codes [d_in, d_out]: byte i
    of row n holds rows 2i (low nibble) and 2i + 1 (high nibble) of column n."""
    c = np.asarray(codes, dtype=np.uint8).T
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def build_segments(slot_ids, n_slots):
    """SGMV segments ([Handbook], SGMV bullet and its toy script): stable sort
    of the tokens by id, then runs of equal ids.

    Returns perm [T] (token indices in sorted order; base-only and invalid
    tokens first), seg_slot [n_seg] (ids >= 0 present, ascending), seg_off
    [n_seg + 1] (segment j is perm[seg_off[j]:seg_off[j+1]]; seg_off[n_seg] = T)
    and n_seg.
    """
    ids = valid_ids(slot_ids, n_slots)
    T = ids.size
    perm = np.argsort(ids, kind="stable").astype(np.int32)
    sorted_ids = ids[perm]
    seg_slot, seg_off = [], []
    p = 0
    while p < T:
        q = p
        while q < T and sorted_ids[q] == sorted_ids[p]:
            q += 1
        if sorted_ids[p] >= 0:
            seg_slot.append(int(sorted_ids[p]))
            seg_off.append(p)
        p = q
    seg_off.append(T)
    return {
        "perm": perm,
        "seg_slot": np.asarray(seg_slot, np.int32),
        "seg_off": np.asarray(seg_off, np.int32),
        "n_seg": len(seg_slot),
    }


def lora_linear_segmented(x, W0, A_pool, B_pool, scale, slot_ids):
    """SGMV form: base product once for all rows; the adapter term computed
    segment by segment on the sorted rows, then scattered back to token order
    ([Handbook], SGMV toy; [Blog, "Replay"]: segmented gather, grouped GEMM,
    scatter add)."""
    x, W0 = _f64(x), _f64(W0)
    seg = build_segments(slot_ids, A_pool.shape[0])
    y = x @ W0
    perm, off = seg["perm"], seg["seg_off"]
    for j, a in enumerate(seg["seg_slot"]):
        rows = perm[off[j]:off[j + 1]]
        xs = x[rows]
        y[rows] += float(scale[a]) * ((xs @ _f64(A_pool[a])) @ _f64(B_pool[a]))
    return y


def shrink(x, A_pool, scale, slot_ids):
    """Shrink step: v_t = s_{a_t} x_t A_{a_t} (rank-r), zero for base-only."""
    x = _f64(x)
    ids = valid_ids(slot_ids, A_pool.shape[0])
    v = np.zeros((x.shape[0], A_pool.shape[2]))
    for t in range(x.shape[0]):
        a = ids[t]
        if a >= 0:
            v[t] = float(scale[a]) * (x[t] @ _f64(A_pool[a]))
    return v


def expand(v, B_pool, slot_ids):
    """Expand step: the adapter term v_t B_{a_t}, zero for base-only rows."""
    v = _f64(v)
    ids = valid_ids(slot_ids, B_pool.shape[0])
    out = np.zeros((v.shape[0], B_pool.shape[2]))
    for t in range(v.shape[0]):
        a = ids[t]
        if a >= 0:
            out[t] = v[t] @ _f64(B_pool[a])
    return out


def merge(W0, A, B, s):
    """Merged weight W' = W0 + s A B ([Blog, "Merge or keep separate"];
    [Handbook] self-test answer on merging)."""
    return _f64(W0) + float(s) * (_f64(A) @ _f64(B))


def lora_param_count(d, k, r):
    """Adapter parameters of one d x k layer at rank r: r (d + k)
    ([Blog, "Low-rank structure and additivity"], the Rank property)."""
    return r * (d + k)


def adapter_bytes(projections, r, layers, bytes_per_param=2):
    """Bytes of one adapter over ``layers`` layers of the given (d_in, d_out)
    projections ([Handbook, "Scheduling the adapters"] tier table)."""
    return layers * sum(lora_param_count(di, do, r) for di, do in projections) * bytes_per_param


def pad_rank(A, B, r_pad):
    """Zero-pad one adapter to rank r_pad: extra A columns and B rows are 0
    ([Concepts, "When It Falls Down"]; [Handbook, Exercise 2])."""
    A, B = _f64(A), _f64(B)
    d_in, r = A.shape
    Ap = np.zeros((d_in, r_pad))
    Bp = np.zeros((r_pad, B.shape[1]))
    Ap[:, :r] = A
    Bp[:r, :] = B
    return Ap, Bp
