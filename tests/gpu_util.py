"""Helpers for the GPU parity tests: upload seeded inputs, run the C-ABI
path, fetch results.  Inputs come from the seeded generators; expected
values come only from the CPU oracle."""
import numpy as np

from lora_serving_device_gb300 import workloads as W


def torch_mod():
    import torch
    return torch


def dev(a, dtype="bf16", device="cuda"):
    torch = torch_mod()
    a = np.ascontiguousarray(a)
    if a.dtype in (np.int32, np.int64):
        return torch.from_numpy(a.astype(np.int32)).to(device)
    if dtype == "bf16":
        return torch.from_numpy(W.bf16_bits(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a.astype(np.float32)).to(device)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


class DeviceCase:
    """Device copies of one Workload's tensors."""

    def __init__(self, w, device="cuda", W0_zero=False):
        torch = torch_mod()
        self.w = w
        dt = w.dtype
        self.dt = dt
        self.x = dev(w.x, dt, device)
        self.W0 = dev(np.zeros_like(w.W0) if W0_zero else w.W0, dt, device)
        self.A = dev(w.A_pool, dt, device)
        self.B = dev(w.B_pool, dt, device)
        self.scale = torch.from_numpy(w.scale.astype(np.float32)).to(device)
        self.ids = torch.from_numpy(w.slot_ids.astype(np.int32)).to(device)

    def fused(self, ws=None, y=None):
        from lora_serving_device_gb300 import lora as L
        w = self.w
        if ws is None:
            ws = L.workspace(L.OP_LINEAR_FUSED, w.T, w.d_in, w.d_out, w.r, w.n_slots)
        y = L.linear_fused_t(self.x, self.W0, self.A, self.B, self.ids, self.scale, ws, y=y)
        return y, ws
