"""The 4-bit base path on the GPU against the CPU fp64 oracle.

[Concepts, "When It Falls Down"]: QLoRA-style 4-bit base models served next
to bf16 adapters, the base weights passing through dequantisation.  The
quantiser's codes and scales must match the oracle's bit for bit (both take
the nearest-code decision on the same fp32 quotient); the GEMM and the layer
are compared with the oracle's dequantised matrix in fp64.
"""
import numpy as np
import pytest

from oracle import lora_ref as O
from lora_serving_device_gb300 import workloads as W

from tests.gpu_util import DeviceCase, dev, host, torch_mod
from tests.tolerances import check_close, check_close_bf16_out

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


def _cb():
    return W.nf4_like_codebook()


def _dev_base(L, codes, absmax, cb):
    torch = torch_mod()
    return L.Base4bit(torch.from_numpy(W.pack_nibbles(codes)).cuda(), dev(absmax), dev(cb))


def _ws(n=1 << 16):
    torch = torch_mod()
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("shape", [(64, 32), (192, 160), (1024, 4096), (4096, 4096)])
def test_quantize_base_4bit_bit_exact(L, shape):
    torch = torch_mod()
    d_in, d_out = shape
    rng = np.random.default_rng([5, d_in, d_out])
    Wt = W.bf16_round(rng.standard_normal((d_in, d_out)).astype(np.float32) * np.float32(0.02))
    Wt[:64, : min(d_out, 32)] = 0.0                     # all-zero blocks
    Wt[64 % d_in, 1] = -Wt[64 % d_in, 1] * 3            # a block whose absmax is negative-signed
    Wt = W.bf16_round(Wt)                               # the device copy is bf16
    cb = _cb()
    base = L.Base4bit.quantize(dev(Wt), dev(cb))
    torch.cuda.synchronize()
    codes, absmax = O.quantize_4bit(Wt, cb)
    np.testing.assert_array_equal(base.W0q.cpu().numpy(), O.pack_4bit(codes))
    np.testing.assert_array_equal(host(base.absmax), absmax.astype(np.float64))


Q4_SPLITK_CASES = [(1, 64, 128, 1), (5, 192, 160, 2), (40, 1024, 288, 3), (64, 4096, 4096, 4),
                   (64, 4096, 4096, 17), (100, 512, 544, 8), (256, 4096, 4096, 4),
                   (300, 256, 512, 2)]


@pytest.mark.parametrize("case", Q4_SPLITK_CASES, ids=[str(c) for c in Q4_SPLITK_CASES])
def test_base_gemm_4bit_splitk_matches_oracle(L, case):
    """The split-K product over the dequantised 4-bit base: bf16 operands,
    fp32 products and sums, so the bar is fp32 accumulation error."""
    torch = torch_mod()
    T, d_in, d_out, S = case
    codes, absmax = W.random_4bit_base(T + S, d_in, d_out)
    cb = _cb()
    x = W.bf16_round(np.random.default_rng([7, T, d_in]).standard_normal((T, d_in))
                     .astype(np.float32))
    base = _dev_base(L, codes, absmax, cb)
    ws = _ws()
    partial = torch.full((S, T, d_out), 9.0, dtype=torch.float32, device="cuda")
    L.base_gemm_4bit_splitk_t(dev(x), base, ws, ksplit=S, partial=partial)
    torch.cuda.synchronize()
    ref = x.astype(np.float64) @ O.dequantize_4bit(codes, absmax, cb)
    check_close(host(partial).sum(axis=0), ref, "4-bit split-K product", rel_fro=2e-5,
                max_rms=2e-4)
    assert L.get_error_t(ws) == 0


Q4_FUSED_CASES = [(1, 64, 128, 16, 3), (5, 192, 160, 8, 7), (33, 256, 384, 32, 5),
                  (64, 512, 1024, 16, 40), (7, 1024, 608, 32, 4), (48, 2048, 2112, 16, 9),
                  (200, 640, 160, 16, 30), (256, 256, 512, 64, 70),
                  # larger batches: W0 dequantised into the workspace, then the
                  # prefill path (many 256 x 256 tiles; a half 64-column block)
                  (300, 256, 512, 16, 8), (700, 192, 160, 8, 7), (2000, 1024, 2048, 64, 12),
                  (400, 256, 96, 16, 5)]


@pytest.mark.parametrize("case", Q4_FUSED_CASES, ids=[str(c) for c in Q4_FUSED_CASES])
def test_fused_4bit_matches_oracle(L, case):
    torch = torch_mod()
    T, d_in, d_out, r, n_slots = case
    w = W.random_case(820 + T, T, d_in, d_out, r, n_slots)
    codes, absmax = W.random_4bit_base(900 + T, d_in, d_out)
    cb = _cb()
    d = DeviceCase(w)
    for zero_base in (False, True):
        am = np.zeros_like(absmax) if zero_base else absmax
        base = _dev_base(L, codes, am, cb)
        ws = L.workspace(L.OP_LINEAR_FUSED_4BIT, T, d_in, d_out, r, n_slots)
        y = L.linear_fused_4bit_t(d.x, base, d.A, d.B, d.ids, d.scale, ws)
        torch.cuda.synchronize()
        ref = O.lora_linear(w.x, O.dequantize_4bit(codes, am, cb), w.A_pool, w.B_pool, w.scale,
                            w.slot_ids)
        # zero scales: the adapter term alone, which base rounding cannot hide
        check_close_bf16_out(host(y), ref, f"4-bit layer y zero_base={zero_base}")
        assert L.get_error_t(ws) == 0


def test_fused_4bit_decode_layer_full_size(L):
    """The 4096 -> 4096 rank-16 decode layer (64 tokens, 256 slots, Zipf ids,
    8 base-only rows) with W0 ~ N(0, 0.02) quantised by the oracle."""
    torch = torch_mod()
    w = W.decode_bgmv()
    cb = _cb()
    codes, absmax = O.quantize_4bit(w.W0, cb)
    d = DeviceCase(w)
    base = _dev_base(L, codes, absmax, cb)
    ws = L.workspace(L.OP_LINEAR_FUSED_4BIT, w.T, w.d_in, w.d_out, w.r, w.n_slots)
    y = L.linear_fused_4bit_t(d.x, base, d.A, d.B, d.ids, d.scale, ws)
    torch.cuda.synchronize()
    ref = O.lora_linear(w.x, O.dequantize_4bit(codes, absmax, cb), w.A_pool, w.B_pool, w.scale,
                        w.slot_ids)
    check_close_bf16_out(host(y), ref, "4-bit decode layer")
    assert L.get_error_t(ws) == 0
    # the library's quantiser gives the same base
    q = L.Base4bit.quantize(d.W0, dev(cb))
    torch.cuda.synchronize()
    assert torch.equal(q.W0q, base.W0q) and torch.equal(q.absmax, base.absmax)
