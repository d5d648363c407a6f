"""The bounds-checking debug build of the library (liblora_debug.so, built with
-DLORA_DEBUG): indices that one kernel hands to another (segment offsets and
slots, perm rows) are checked on the device, and one outside its buffer sets
LORA_DEVERR_BOUNDS and is replaced by an in-range index.

The checks run in a fresh process (the binding holds one library per
process).  There the debug build must give the oracle's results with no
bounds bit on the usual paths, and must raise the bit, with every access
still inside its buffers, when a perm entry it is handed is out of range.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker():
    import torch
    from oracle import lora_ref as O
    from lora_serving_device_gb300 import lora as L, workloads as W
    from tests.gpu_util import DeviceCase, dev, host
    from tests.tolerances import check_close, check_close_bf16_out

    L.load(L.LIB_DEBUG_PATH)
    # segments bit-exact, no bounds bit
    ids = np.random.default_rng(3).integers(-1, 40, 700).astype(np.int32)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    perm, seg_slot, seg_off, n_seg = L.build_segments_t(dev(ids), 40, ws)
    torch.cuda.synchronize()
    ref = O.build_segments(ids, 40)
    assert perm.cpu().numpy().tolist() == ref["perm"].tolist()
    assert L.get_error_t(ws) == 0
    # the fused layer: decode chain, prefill path (tensor-core SGMV), fp32
    for w in (W.random_case(11, 64, 512, 1024, 16, 40), W.random_case(12, 700, 256, 520, 64, 9, runs=True),
              W.random_case(13, 300, 256, 264, 16, 11, runs=True), W.toy_mixed_batch()):
        d = DeviceCase(w)
        y, wsf = d.fused()
        torch.cuda.synchronize()
        assert L.get_error_t(wsf) == 0, w.T
        ref = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)
        (check_close if w.dtype == "f32" else check_close_bf16_out)(host(y), ref, f"debug T={w.T}")
    # standalone SGMV shrink and expand on CUDA cores (rank 16) and tensor cores (rank 64)
    for r in (16, 64):
        w = W.random_case(20 + r, 400, 512, 520, r, 7, runs=True)
        d = DeviceCase(w)
        segs = L.build_segments_t(d.ids, w.n_slots, ws)
        vp = L.sgmv_shrink_t(d.x, d.A, segs, d.scale, 2, ws)
        yb = dev(np.zeros((w.T, w.d_out), np.float32), "bf16")
        L.sgmv_expand_t(vp, d.B, segs, yb, ws)
        torch.cuda.synchronize()
        assert L.get_error_t(ws) == 0, r
        delta = O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids) - \
            O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, np.full(w.T, -1))
        check_close_bf16_out(host(yb), delta, f"debug SGMV r={r}")
        # a perm entry out of range: the CUDA-core expand replaces it and
        # raises the bounds bit (only with the debug build)
        if r == 16:
            bad = segs[0].clone()
            bad[int(segs[2][0].item())] = w.T + 5   # the first token of the first segment
            torch.cuda.synchronize()
            L.sgmv_expand_t(vp, d.B, (bad, segs[1], segs[2], segs[3]), yb, ws)
            torch.cuda.synchronize()
            assert L.get_error_t(ws) & L.DEVERR_BOUNDS
    print("debug build ok")


def test_debug_build_checks_indices_without_faulting():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from lora_serving_device_gb300 import build
    build.build(debug=True)
    r = subprocess.run([sys.executable, "-c", "import tests.test_gpu_debug_build as t; t._worker()"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build ok" in r.stdout
