"""lora_linear_fused_noalloc: the fused layer for callers that cannot
allocate device memory (their framework's allocator owns the GPU memory, or
they run where allocation is not allowed).  It keeps its scratch in a fixed
array inside the library instead of a caller workspace.

Its output must match the regular lora_linear_fused, within the parity bar
the other tests use, on two calls in a row (the second call reuses the array
the first one left behind).  This file is collected last on purpose.
"""
import numpy as np
import pytest

from lora_serving_device_gb300 import workloads as W
from tests.tolerances import check_close


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


@pytest.mark.gpu
def test_noalloc_matches_fused_on_two_calls_in_a_row(L):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tests.gpu_util import DeviceCase, host

    cases = [W.random_case(901, 64, 512, 1024, 16, 40),             # decode path
             W.random_case(902, 300, 256, 520, 64, 9, runs=True)]   # prefill path
    for w in cases:
        d = DeviceCase(w)
        want, _ = d.fused()
        got = torch.empty_like(want)
        got.fill_(float("nan"))
        st = L.lora_linear_fused_noalloc(d.x.data_ptr(), d.W0.data_ptr(), d.A.data_ptr(),
                                         d.B.data_ptr(), d.ids.data_ptr(), d.scale.data_ptr(),
                                         got.data_ptr(), w.T, w.d_in, w.d_out, w.r, w.n_slots,
                                         L.DTYPE_BF16, torch.cuda.current_stream().cuda_stream)
        assert st == 0, L.lora_status_string(st)
        torch.cuda.synchronize()
        check_close(host(got), host(want), f"noalloc vs fused, T={w.T}")
