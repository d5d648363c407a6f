"""The failure path of the tensor-core kernels, made to run on purpose.

Every on-chip wait in the library's kernels is bounded.  When one gives up,
the kernel must set LORA_DEVERR_TIMEOUT in the workspace error word, skip its
output, free its tensor memory and return, so the device stays usable.  The
diagnostic entry point lora_debug_gemm_wait_timeout runs the decode GEMM with
its producer held back (nothing ever arrives on the barrier its MMA issuer
waits for) and a wait limit of a millisecond.  Nothing faults or hangs: the
wait simply runs out.  The test then runs ordinary layers on the same device;
had the timed-out kernel kept its tensor memory, their allocation could not
complete.
"""
import numpy as np
import pytest

from oracle import lora_ref as O
from lora_serving_device_gb300 import workloads as W

from tests.gpu_util import DeviceCase, host, torch_mod
from tests.tolerances import check_close

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


def _held_gemm(L, T, d_in, d_out, wait_us):
    torch = torch_mod()
    w = W.random_case(930 + T, T, d_in, d_out, 16, 4)
    d = DeviceCase(w)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    partial = torch.full((1, T, d_out), 3.0, dtype=torch.float32, device="cuda")
    st = L.lora_debug_gemm_wait_timeout(d.x.data_ptr(), d.W0.data_ptr(), partial.data_ptr(), T,
                                        d_in, d_out, wait_us, ws.data_ptr(), ws.numel(),
                                        torch.cuda.current_stream().cuda_stream)
    assert st == 0, L.lora_status_string(st)
    torch.cuda.synchronize()
    return L.get_error_t(ws), partial


@pytest.mark.parametrize("shape", [(8, 256, 256), (64, 4096, 4096), (256, 1024, 512)])
def test_bounded_wait_runs_out_and_reports_timeout(L, shape):
    torch = torch_mod()
    T, d_in, d_out = shape
    err, partial = _held_gemm(L, T, d_in, d_out, 1000)
    assert err & L.DEVERR_TIMEOUT, f"error word {err:#x}"
    assert not err & ~L.DEVERR_TIMEOUT
    # the kernel gave up before its epilogue: the output is untouched
    assert torch.all(partial == 3.0)


def test_device_is_usable_after_timeouts(L):
    """Timed-out kernels on every SM, then ordinary layers (decode chain and
    prefill GEMM, both tensor-memory users) still match the oracle."""
    torch = torch_mod()
    for _ in range(2):
        err, _ = _held_gemm(L, 64, 4096, 4096, 500)    # 32 CTAs, one per column tile
        assert err & L.DEVERR_TIMEOUT
        for w in (W.random_case(941, 64, 512, 1024, 16, 40),
                  W.random_case(942, 300, 256, 520, 64, 9, runs=True)):
            d = DeviceCase(w)
            y, ws = d.fused()
            torch.cuda.synchronize()
            assert L.get_error_t(ws) == 0
            ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
            check_close(host(y), ref, f"layer after a timeout, T={w.T}")
