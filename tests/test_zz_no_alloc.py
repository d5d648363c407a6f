"""lora_linear_fused_noalloc: the fused layer for callers that cannot
allocate device memory (their framework's allocator owns the GPU memory, or
they run where allocation is not allowed).  It keeps its scratch in a fixed
array inside the library instead of a caller workspace.

Its output must match the regular lora_linear_fused, within the parity bar
the other tests use, on two calls in a row (the second call reuses the array
the first one left behind), and the CPU oracle.  This file is collected last
on purpose.
"""
import numpy as np
import pytest

from oracle import lora_ref as O
from lora_serving_device_gb300 import workloads as W
from tests.tolerances import check_close, check_close_bf16_out


@pytest.fixture(scope="module")
def L():
    from lora_serving_device_gb300 import build, lora
    build.build()
    lora.load()
    return lora


def test_oversized_batch_is_refused_before_any_work(L):
    # rank 128 x 64 splits of 1M tokens needs far more than the fixed array
    st = L.lora_linear_fused_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, None, 0x20000,
                                     1 << 20, 4096, 4096, 128, 64, L.DTYPE_BF16, None)
    assert st == 4  # LORA_ERR_WORKSPACE
    assert L.lora_workspace_bytes(L.OP_LINEAR_FUSED, 1 << 20, 4096, 4096, 128, 64) > \
        L.NOALLOC_SCRATCH_BYTES


def test_realistic_decode_shape_over_the_limit_is_refused(L):
    # a 256-token decode batch on a gate/up projection (4096 -> 14336): its
    # split-K fp32 partials alone are tens of MB, beyond the fixed array
    need = L.lora_workspace_bytes(L.OP_LINEAR_FUSED, 256, 4096, 14336, 64, 250)
    assert need > L.NOALLOC_SCRATCH_BYTES
    st = L.lora_linear_fused_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, None, 0x20000,
                                     256, 4096, 14336, 64, 250, L.DTYPE_BF16, None)
    assert st == 4  # LORA_ERR_WORKSPACE


@pytest.mark.gpu
def test_invalid_arguments_are_refused_before_any_work(L):
    # x and y alias: refused by the argument checks, before the shared
    # array's error word is cleared (the pointers are never dereferenced; a
    # GPU is needed only for the array's address lookup that comes first)
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    st = L.lora_linear_fused_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, None, 0x10000,
                                     64, 4096, 4096, 16, 256, L.DTYPE_BF16, None)
    assert st == 1  # LORA_ERR_INVALID_ARG
    st = L.lora_linear_fused_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, None, 0x60000,
                                     64, 4096, 4096, 12, 256, L.DTYPE_BF16, None)
    assert st == 2  # LORA_ERR_SHAPE (rank 12)


def _noalloc(L, d, w, out):
    import torch
    st = L.lora_linear_fused_noalloc(d.x.data_ptr(), d.W0.data_ptr(), d.A.data_ptr(),
                                     d.B.data_ptr(), d.ids.data_ptr(), d.scale.data_ptr(),
                                     out.data_ptr(), w.T, w.d_in, w.d_out, w.r, w.n_slots,
                                     L.DTYPE_BF16 if w.dtype == "bf16" else L.DTYPE_F32,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == 0, L.lora_status_string(st)
    torch.cuda.synchronize()


@pytest.mark.gpu
def test_noalloc_matches_fused_on_two_calls_in_a_row(L):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tests.gpu_util import DeviceCase, host

    cases = [W.random_case(901, 64, 512, 1024, 16, 40),             # decode path
             W.random_case(902, 300, 256, 520, 64, 9, runs=True),   # prefill path
             W.random_case(903, 64, 512, 1024, 16, 40, invalid=5),  # sets a device error bit
             W.random_case(904, 64, 512, 1024, 16, 40),             # a clean call after it
             W.toy_mixed_batch()]                                   # fp32 storage
    for w in cases:
        d = DeviceCase(w)
        want, _ = d.fused()
        ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
        for call in range(2):
            got = torch.empty_like(want)
            got.fill_(float("nan"))
            _noalloc(L, d, w, got)
            check_close(host(got), host(want), f"noalloc vs fused, T={w.T}, call {call}")
            if w.dtype == "bf16":
                check_close_bf16_out(host(got), ref, f"noalloc vs oracle, T={w.T}, call {call}")
            else:
                check_close(host(got), ref, f"noalloc vs oracle, T={w.T}, call {call}")
