"""Parity bars shared by the GPU tests.

Floating point: per output tensor, relative Frobenius error <= 5e-3 and
max |err| <= 2e-2 * rms(reference), both for y and for the LoRA delta
y - x W0 (the delta is ~8x smaller than the base term under the decode init,
so a broken adapter path could hide inside y's budget).  Integer / index
outputs: bit-exact.
"""
import numpy as np

REL_FRO = 5e-3
MAX_RMS = 2e-2


def check_close(got, ref, what="y", rel_fro=REL_FRO, max_rms=MAX_RMS):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    if ref.size == 0:
        return {"rel_fro": 0.0, "max_over_rms": 0.0}
    err = got - ref
    nref = np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref * ref))
    rel = float(np.linalg.norm(err) / nref) if nref > 0 else float(np.linalg.norm(err))
    mx = float(np.max(np.abs(err)) / rms) if rms > 0 else float(np.max(np.abs(err)))
    assert rel <= rel_fro, f"{what}: rel Frobenius error {rel:.3e} > {rel_fro}"
    assert mx <= max_rms, f"{what}: max|err|/rms {mx:.3e} > {max_rms}"
    return {"rel_fro": rel, "max_over_rms": mx}
