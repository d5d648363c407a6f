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
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", src)))


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
    # decode building blocks: bf16 only, ksplit within the d_in blocks
    assert L.lora_base_gemm_splitk(FAKE, FAKE, FAKE, 4, 4096, 4096, 1, L.DTYPE_F32, ws, 16,
                                   None) == 3
    assert L.lora_base_gemm_splitk(FAKE, FAKE, FAKE, 4, 4096, 4096, 0, 0, ws, 16, None) == 2
    assert L.lora_base_gemm_splitk(FAKE, FAKE, FAKE, 4, 128, 4096, 2, 0, ws, 16, None) == 2
    assert L.lora_base_gemm_splitk(FAKE, FAKE, None, 4, 4096, 4096, 2, 0, ws, 16, None) == 1
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


def test_decode_split_is_a_function_of_the_shapes(L):
    assert L.lora_decode_split(64, 4096, 4096) == 4       # 32 column tiles x 4 = 128 CTAs
    assert L.lora_decode_split(256, 4096, 4096) == 4      # one 256-token tile
    assert L.lora_decode_split(100, 4096, 4096) == 4      # one 128-token tile
    assert L.lora_decode_split(1, 64, 128) == 1           # one K block
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
