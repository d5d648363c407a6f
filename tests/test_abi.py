"""The C-ABI library: it loads, exports every symbol include/lora.h declares,
and its host-side validation answers without a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora.h")


@pytest.fixture(scope="module")
def L():
    from lora_serving_device_gb300 import build, lora
    build.build()
    lora.load()
    return lora


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("lora_build_segments", "lora_bgmv_shrink", "lora_bgmv_expand", "lora_sgmv_shrink",
              "lora_sgmv_expand", "lora_linear_fused", "lora_base_gemm_expand",
              "lora_bgmv_delta", "lora_bgmv_adapter", "lora_bgmv_adapter_merge",
              "lora_base_gemm_splitk", "lora_decode_split", "lora_slot_upload",
              "lora_workspace_bytes", "lora_get_error",
              "lora_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    lib = ctypes.CDLL(L.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(L.EXPORTS) == set(declared_functions())


def test_status_strings(L):
    for code, name in L.STATUS_NAMES.items():
        assert L.lora_status_string(code).startswith(name)


def test_workspace_sizes(L):
    assert L.lora_workspace_bytes(L.OP_BGMV_SHRINK, 64, 4096, 4096, 16, 256) == 16
    n = L.lora_workspace_bytes(L.OP_LINEAR_FUSED, 64, 4096, 4096, 16, 256)
    # error word + perm/segments + split fp32 partials of the shrink
    assert n >= 16 + 64 * 4 + 64 * 4 * 16 and n % 256 == 0
    assert L.lora_workspace_bytes(L.OP_LINEAR_FUSED, 0, 4096, 4096, 16, 256) >= 16


FAKE = 0x10000  # aligned, never dereferenced: validation rejects first


def _fused(L, **kw):
    a = dict(x=FAKE, W0=FAKE, A=FAKE, B=FAKE, ids=FAKE, scale=None, y=FAKE + 4096, T=8, d_in=64,
             d_out=64, r=16, n_slots=4, dt=L.DTYPE_BF16, ws=FAKE + 8192, ws_bytes=1 << 20,
             stream=None)
    a.update(kw)
    return L.lora_linear_fused(a["x"], a["W0"], a["A"], a["B"], a["ids"], a["scale"], a["y"],
                               a["T"], a["d_in"], a["d_out"], a["r"], a["n_slots"], a["dt"],
                               a["ws"], a["ws_bytes"], a["stream"])


def test_validation_paths(L):
    assert _fused(L, T=-1) == 1                      # INVALID_ARG
    assert _fused(L, r=12) == 2                      # SHAPE: rank
    assert _fused(L, d_in=60) == 2                   # SHAPE: multiple of 8
    assert _fused(L, d_out=0) == 2
    assert _fused(L, n_slots=0) == 2
    assert _fused(L, n_slots=L.MAX_SLOTS + 1) == 2
    assert _fused(L, T=L.MAX_TOKENS + 1) == 2
    assert _fused(L, dt=7) == 3                      # DTYPE
    assert _fused(L, x=None) == 1
    assert _fused(L, W0=FAKE + 2) == 1               # misaligned
    assert _fused(L, y=FAKE) == 1                    # x and y alias
    assert _fused(L, ws=None) == 4                   # WORKSPACE
    assert _fused(L, ws_bytes=16) == 4
    assert _fused(L, ws=FAKE + 8) == 4               # misaligned workspace
    ws = FAKE + 8192
    assert L.lora_bgmv_shrink(FAKE, FAKE, FAKE, None, FAKE, 4, 64, 16, 4, 0, 0, ws, 16, None) == 2
    assert L.lora_bgmv_shrink(FAKE, FAKE, FAKE, None, FAKE, 4, 64, 16, 4, 65, 0, ws, 16, None) == 2
    assert L.lora_bgmv_expand(FAKE, 1, FAKE, None, FAKE, 4, 16, 64, 4, 0, ws, 16, None) == 1
    assert L.lora_sgmv_shrink(FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, 4, 64, 16, 4, 1, 0,
                              ws, 16, None) == 1
    assert L.lora_sgmv_expand(FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 16, 64, 4, 0, ws, 8,
                              None) == 4
    assert L.lora_build_segments(FAKE, 4, 0, FAKE, FAKE, FAKE, FAKE, ws, 16, None) == 2
    assert L.lora_build_segments(FAKE, -2, 4, FAKE, FAKE, FAKE, FAKE, ws, 16, None) == 1
    st, _ = L.lora_get_error(None, None)
    assert st == 1
    # decode building blocks: bf16 only, ksplit within the 64-row blocks of
    # d_in; ksplit 0 (the fused layer's split) only for T <= 256
    assert L.lora_base_gemm_splitk(FAKE, FAKE, FAKE, 4, 4096, 4096, 1, L.DTYPE_F32, ws, 16,
                                   None) == 3
    assert L.lora_base_gemm_splitk(FAKE, FAKE, FAKE, 4, 4096, 4096, -1, 0, ws, 16, None) == 2
    assert L.lora_base_gemm_splitk(FAKE, FAKE, FAKE, 4, 128, 4096, 3, 0, ws, 16, None) == 2
    assert L.lora_base_gemm_splitk(FAKE, FAKE, FAKE, 257, 128, 4096, 0, 0, ws, 16, None) == 2
    assert L.lora_base_gemm_splitk(FAKE, FAKE, None, 4, 4096, 4096, 2, 0, ws, 16, None) == 1
    # the wait-timeout diagnostic: shapes and limit checked before anything runs
    assert L.lora_debug_gemm_wait_timeout(FAKE, FAKE, FAKE, 0, 64, 128, 100, ws, 16, None) == 2
    assert L.lora_debug_gemm_wait_timeout(FAKE, FAKE, FAKE, 4, 64, 128, 0, ws, 16, None) == 1
    assert L.lora_debug_gemm_wait_timeout(FAKE, FAKE, FAKE, 4, 64, 128, 2000001, ws, 16,
                                          None) == 1
    assert L.lora_debug_gemm_wait_timeout(FAKE, FAKE, None, 4, 64, 128, 100, ws, 16, None) == 1
    assert L.lora_bgmv_adapter(FAKE, FAKE, FAKE, FAKE, None, FAKE, 70000, 64, 64, 16, 4, 0, ws,
                               16, None) == 2
    assert L.lora_bgmv_adapter_merge(FAKE, FAKE, FAKE, FAKE, None, FAKE, 2, FAKE, 4, 64, 64, 16,
                                     4, 0, ws, 16, None) == 1        # x and y alias
    assert L.lora_bgmv_adapter_merge(FAKE, FAKE, FAKE, FAKE, None, FAKE, 65, FAKE + 4096, 4, 64,
                                     64, 16, 4, 0, ws, 16, None) == 2


def test_slot_upload_validation(L):
    up = L.lora_slot_upload
    # (A_pool, B_pool, scale, slot, A_host, B_host, s, d_in, d_out, r, r_a, n_slots, dt, stream)
    assert up(FAKE, FAKE, None, 4, FAKE, FAKE, 2.0, 64, 64, 16, 8, 4, 0, None) == 2    # slot
    assert up(FAKE, FAKE, None, -1, FAKE, FAKE, 2.0, 64, 64, 16, 8, 4, 0, None) == 2
    assert up(FAKE, FAKE, None, 0, FAKE, FAKE, 2.0, 64, 64, 16, 17, 4, 0, None) == 2   # r_a > r
    assert up(FAKE, FAKE, None, 0, FAKE, FAKE, 2.0, 64, 64, 16, 0, 4, 0, None) == 2
    assert up(FAKE, FAKE, None, 0, FAKE, FAKE, 2.0, 64, 64, 12, 8, 4, 0, None) == 2    # rank
    assert up(FAKE, FAKE, None, 0, None, FAKE, 2.0, 64, 64, 16, 8, 4, 0, None) == 1    # null
    assert up(FAKE + 2, FAKE, None, 0, FAKE, FAKE, 2.0, 64, 64, 16, 8, 4, 0, None) == 1
    assert up(FAKE, FAKE, None, 0, FAKE, FAKE, 2.0, 64, 64, 16, 8, 4, 7, None) == 3    # dtype


def test_ragged_validation(L):
    WS, NW = FAKE + 8192, 1 << 20

    def fused(T=64, x=FAKE, y=FAKE + 4096, A=FAKE, a_elems=1 << 20, r_max=64, dt=0, d_in=64):
        # (x, W0, A, B, a_off, b_off, rank, a_elems, b_elems, r_max, ids, scale, y,
        #  T, d_in, d_out, n_slots, dt, ws, ws_bytes, stream)
        return L.lora_linear_fused_ragged(x, FAKE, A, FAKE, FAKE, FAKE, FAKE, a_elems, 1 << 20,
                                          r_max, FAKE, None, y, T, d_in, 64, 4, dt, WS, NW, None)

    def delta(T=64, r_max=64):
        return L.lora_bgmv_adapter_ragged(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, 1 << 20,
                                          r_max, FAKE, None, FAKE + 4096, T, 64, 64, 4, 0, WS,
                                          NW, None)

    assert fused(T=(1 << 20) + 1) == 2  # more than LORA_MAX_TOKENS
    assert fused(r_max=48) == 2        # r_max is one of 8 .. 128
    assert fused(r_max=256) == 2
    assert fused(d_in=60) == 2
    assert fused(dt=1) == 3            # bf16 only
    assert fused(A=None) == 1
    assert fused(A=FAKE + 2) == 1      # 16-byte aligned pools
    assert fused(a_elems=-1) == 1
    assert fused(x=FAKE + 4096) == 1   # x == y
    assert fused(T=0) == 0             # empty batch: nothing launched
    assert delta(T=65536) == 2
    assert delta(r_max=12) == 2
    assert delta(T=0) == 0


def test_4bit_validation(L):
    WS, NW = FAKE + 8192, 1 << 20
    q = L.lora_quantize_base_4bit
    # (W0, codebook, W0q, absmax, d_in, d_out, stream)
    assert q(FAKE, FAKE, FAKE, FAKE, 96, 64, None) == 2      # d_in not a multiple of 64
    assert q(FAKE, FAKE, FAKE, FAKE, 128, 48, None) == 2     # d_out not a multiple of 32
    assert q(None, FAKE, FAKE, FAKE, 128, 64, None) == 1
    assert q(FAKE, FAKE, FAKE + 8, FAKE, 128, 64, None) == 1
    g = L.lora_base_gemm_4bit_splitk
    # (x, W0q, absmax, codebook, partial, T, d_in, d_out, ksplit, ws, ws_bytes, stream)
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 128, 64, 3, WS, NW, None) == 2   # ksplit > blocks
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 128, 64, 0, WS, NW, None) == 2
    assert g(FAKE, FAKE, FAKE, None, FAKE, 8, 128, 64, 1, WS, NW, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 128, 64, 2, WS, NW, None) == 0   # empty batch
    f = L.lora_linear_fused_4bit
    # (x, W0q, absmax, codebook, A, B, ids, scale, y, T, d_in, d_out, r, n_slots, ws, ..)
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE + 4096, (1 << 20) + 1, 128, 64,
             16, 4, WS, NW, None) == 2                                   # > LORA_MAX_TOKENS
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE + 4096, 8, 128, 64, 12, 4,
             WS, NW, None) == 2                                          # rank
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 8, 128, 64, 16, 4,
             WS, NW, None) == 1                                          # x == y
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE + 4096, 8, 128, 64, 16, 4,
             WS, 16, None) == 4                                          # workspace


def test_ragged_rank_class():
    from lora_serving_device_gb300 import lora as Lb
    assert [Lb.ragged_rank_class(r) for r in (1, 4, 8, 9, 16, 24, 33, 64, 65, 128)] == \
        [8, 8, 8, 16, 16, 32, 64, 64, 128, 128]
    with pytest.raises(ValueError):
        Lb.ragged_rank_class(129)


def test_ragged_pool_layout_on_cpu():
    """The packed layout: each slot at its rank class, offsets contiguous and 16-byte
    aligned, the padding zero, and the padded pool recovered exactly."""
    import numpy as np
    import torch
    from lora_serving_device_gb300 import lora as Lb
    rng = np.random.default_rng(5)
    d_in, d_out, ranks = 24, 40, [8, 4, 64, 16, 24]
    A = [torch.from_numpy(rng.standard_normal((d_in, r)).astype(np.float32)) for r in ranks]
    B = [torch.from_numpy(rng.standard_normal((r, d_out)).astype(np.float32)) for r in ranks]
    p = Lb.RaggedPool(A, B, device="cpu")
    cls = [8, 8, 64, 16, 32]
    assert p.ranks == cls and p.r_max == 64
    assert p.a_off.tolist() == list(np.cumsum([0] + [d_in * c for c in cls[:-1]]))
    assert p.b_off.tolist() == list(np.cumsum([0] + [c * d_out for c in cls[:-1]]))
    assert all(o % 8 == 0 for o in p.a_off.tolist() + p.b_off.tolist())
    assert p.A_flat.numel() == d_in * sum(cls) and p.B_flat.numel() == d_out * sum(cls)
    for a, (r, c) in enumerate(zip(ranks, cls)):
        Aa = p.A_flat[p.a_off[a]:p.a_off[a] + d_in * c].view(d_in, c)
        Ba = p.B_flat[p.b_off[a]:p.b_off[a] + c * d_out].view(c, d_out)
        assert torch.equal(Aa[:, :r], A[a]) and not Aa[:, r:].any()
        assert torch.equal(Ba[:r], B[a]) and not Ba[r:].any()
    # from_padded keeps the first ranks[a] columns / rows of a padded pool
    Ap = torch.zeros(len(ranks), d_in, 64)
    Bp = torch.zeros(len(ranks), 64, d_out)
    for a, r in enumerate(ranks):
        Ap[a, :, :r] = A[a]
        Bp[a, :r] = B[a]
    q = Lb.RaggedPool.from_padded(Ap, Bp, ranks)
    assert torch.equal(q.A_flat, p.A_flat) and torch.equal(q.B_flat, p.B_flat)


def test_decode_split_is_a_function_of_the_shapes(L):
    assert L.lora_decode_split(64, 4096, 4096) == 4       # 32 column tiles x 4 = 128 CTAs
    assert L.lora_decode_split(256, 4096, 4096) == 4      # one 256-token tile
    assert L.lora_decode_split(100, 4096, 4096) == 4      # one 128-token tile
    assert L.lora_decode_split(256, 4096, 1024) == 19     # 8 column tiles x 19
    assert L.lora_decode_split(256, 14336, 4096) == 4
    assert L.lora_decode_split(1, 64, 128) == 1           # one K block
    assert L.lora_decode_split(1, 16384, 128) == 64       # capped at LORA_MAX_KSPLIT
    assert L.lora_decode_split(0, 4096, 4096) == 0
    assert L.lora_decode_split(257, 4096, 4096) == 0
    assert L.lora_decode_split(64, 60, 4096) == 0


def test_empty_batch_is_a_no_op(L):
    # T = 0 validates and launches nothing, so it succeeds even without a GPU
    assert _fused(L, T=0) == 0
    assert L.lora_bgmv_shrink(FAKE, FAKE, FAKE, None, FAKE, 0, 64, 16, 4, 1, 0, FAKE + 8192, 16,
                              None) == 0


def test_no_gpu_reports_cuda_error_without_crashing(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fused(L) in (5, 6)   # LORA_ERR_CUDA / LORA_ERR_DEVICE, nothing launched


def test_4bit_workspace_holds_the_dequantised_base_above_256_tokens(L):
    """Up to 256 tokens the 4-bit layer runs the decode chain (the fused
    layer's workspace); above, its workspace also holds W0 in bf16."""
    for T, d_in, d_out, r, n in [(64, 4096, 4096, 16, 256), (256, 512, 1024, 64, 9),
                                 (300, 256, 512, 16, 8), (9081, 4096, 14336, 64, 64)]:
        fused = L.lora_workspace_bytes(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n)
        q4 = L.lora_workspace_bytes(L.OP_LINEAR_FUSED_4BIT, T, d_in, d_out, r, n)
        if T <= 256:
            assert q4 == fused
        else:
            assert q4 == -(-fused // 256) * 256 + d_in * d_out * 2


def test_ragged_workspace_holds_a_compact_pool_above_256_tokens(L):
    """Up to 256 tokens the ragged layer runs the decode chain (the fused
    layer's workspace); above, its prefill route lays out lora_linear_fused's
    prefill workspace over n_c = min(T, n_slots) compact slots, then the
    compact ids, scales and the padded pool A_c / B_c."""
    rup = lambda v: -(-v // 256) * 256
    for T, d_in, d_out, r, n in [(64, 4096, 4096, 16, 256), (256, 512, 1024, 64, 9),
                                 (300, 256, 512, 16, 8), (9081, 4096, 14336, 64, 64),
                                 (700, 520, 264, 128, 2000)]:
        rag = L.lora_workspace_bytes(L.OP_LINEAR_FUSED_RAGGED, T, d_in, d_out, r, n)
        if T <= 256:
            assert rag == L.lora_workspace_bytes(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n)
            continue
        n_c = min(T, n)
        o = rup(L.lora_workspace_bytes(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_c))
        o = rup(o + T * 4 + n_c * 4)
        o = rup(o + n_c * d_in * r * 2)
        assert rag == rup(o + n_c * r * d_out * 2)
    assert L.lora_workspace_bytes(L.OP_LINEAR_FUSED_RAGGED, 300, 256, 512, 24, 8) == 16  # bad rank


def test_debug_build_exports_every_declared_symbol(L):
    """liblora_debug.so (-DLORA_DEBUG) is the same boundary with device bounds
    checks; its error bit is declared beside the others."""
    from lora_serving_device_gb300 import build
    path = build.build(debug=True)
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    with open(os.path.join(ROOT, "include", "lora.h")) as f:
        assert "#define LORA_DEVERR_BOUNDS 0x8u" in f.read()
    assert L.DEVERR_BOUNDS == 0x8
