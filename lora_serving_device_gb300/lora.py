"""ctypes binding of liblora.so (C ABI in include/lora.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  The raw functions keep the C names and take integer device
pointers; the ``*_t`` helpers take torch tensors (device memory and streams
come from PyTorch) and raise ``LoraError`` on a non-OK status.  There is no
fallback: if the library is missing or the device is not sm_103, calls fail.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblora.so")
# the same library built with -DLORA_DEBUG (bounds checks that set LORA_DEVERR_BOUNDS)
LIB_DEBUG_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblora_debug.so")

# status codes / enums mirrored from include/lora.h
LORA_OK = 0
STATUS_NAMES = {0: "LORA_OK", 1: "LORA_ERR_INVALID_ARG", 2: "LORA_ERR_SHAPE", 3: "LORA_ERR_DTYPE",
                4: "LORA_ERR_WORKSPACE", 5: "LORA_ERR_CUDA", 6: "LORA_ERR_DEVICE"}
DTYPE_BF16, DTYPE_F32 = 0, 1
OP_BUILD_SEGMENTS, OP_BGMV_SHRINK, OP_BGMV_EXPAND = 0, 1, 2
OP_SGMV_SHRINK, OP_SGMV_EXPAND, OP_LINEAR_FUSED, OP_BASE_GEMM_EXPAND = 3, 4, 5, 6
OP_LINEAR_FUSED_4BIT = 7
OP_LINEAR_FUSED_RAGGED = 8
DEVERR_BAD_SLOT, DEVERR_TIMEOUT, DEVERR_BAD_RANK, DEVERR_BOUNDS = 0x1, 0x2, 0x4, 0x8
RAGGED_RANKS = (8, 16, 32, 64, 128)
MAX_SLOTS, MAX_TOKENS, MAX_KSPLIT = 16384, 1 << 20, 64
NOALLOC_SCRATCH_BYTES = 8 << 20

EXPORTS = ("lora_workspace_bytes", "lora_build_segments", "lora_bgmv_shrink", "lora_bgmv_expand",
           "lora_sgmv_shrink", "lora_sgmv_expand", "lora_linear_fused", "lora_base_gemm_expand",
           "lora_linear_fused_noalloc", "lora_bgmv_delta", "lora_bgmv_adapter",
           "lora_bgmv_adapter_merge", "lora_base_gemm_splitk", "lora_decode_split",
           "lora_slot_upload", "lora_bgmv_adapter_ragged", "lora_linear_fused_ragged",
           "lora_quantize_base_4bit", "lora_base_gemm_4bit_splitk", "lora_linear_fused_4bit",
           "lora_debug_gemm_wait_timeout", "lora_get_error", "lora_status_string")


class LoraError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int32
_Z = ctypes.c_size_t
_L = ctypes.c_int64

_SIGS = {
    "lora_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I]),
    "lora_build_segments": (_I, [_P, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "lora_bgmv_shrink": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_bgmv_expand": (_I, [_P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_sgmv_shrink": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_sgmv_expand": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_linear_fused": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_base_gemm_expand": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_linear_fused_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "lora_bgmv_delta": (_I, [_P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_bgmv_adapter": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_bgmv_adapter_merge": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P,
                                     _Z, _P]),
    "lora_base_gemm_splitk": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_decode_split": (_I, [_I, _I, _I]),
    "lora_slot_upload": (_I, [_P, _P, _P, _I, _P, _P, ctypes.c_float, _I, _I, _I, _I, _I, _I,
                              _P]),
    "lora_bgmv_adapter_ragged": (_I, [_P, _P, _P, _P, _P, _P, _L, _L, _I, _P, _P, _P, _I, _I, _I,
                                      _I, _I, _P, _Z, _P]),
    "lora_linear_fused_ragged": (_I, [_P, _P, _P, _P, _P, _P, _P, _L, _L, _I, _P, _P, _P, _I, _I,
                                      _I, _I, _I, _P, _Z, _P]),
    "lora_quantize_base_4bit": (_I, [_P, _P, _P, _P, _I, _I, _P]),
    "lora_base_gemm_4bit_splitk": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_linear_fused_4bit": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P,
                                    _Z, _P]),
    "lora_debug_gemm_wait_timeout": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "lora_get_error": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "lora_status_string": (ctypes.c_char_p, [_I]),
}


def load(path: str = LIB_PATH):
    """Load liblora.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m lora_serving_device_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _call(name, *args):
    return getattr(load(), name)(*args)


# ----------------------------------------------------------------- raw C names
def lora_workspace_bytes(op, T, d_in, d_out, r, n_slots):
    return _call("lora_workspace_bytes", op, T, d_in, d_out, r, n_slots)


def lora_build_segments(slot_ids, T, n_slots, perm, seg_slot, seg_off, n_seg, ws, ws_bytes, stream):
    return _call("lora_build_segments", slot_ids, T, n_slots, perm, seg_slot, seg_off, n_seg, ws,
                 ws_bytes, stream)


def lora_bgmv_shrink(x, A_pool, slot_ids, scale, v_partial, T, d_in, r, n_slots, ksplit, dt, ws,
                     ws_bytes, stream):
    return _call("lora_bgmv_shrink", x, A_pool, slot_ids, scale, v_partial, T, d_in, r, n_slots,
                 ksplit, dt, ws, ws_bytes, stream)


def lora_bgmv_expand(v_partial, ksplit, B_pool, slot_ids, y, T, r, d_out, n_slots, dt, ws,
                     ws_bytes, stream):
    return _call("lora_bgmv_expand", v_partial, ksplit, B_pool, slot_ids, y, T, r, d_out, n_slots,
                 dt, ws, ws_bytes, stream)


def lora_sgmv_shrink(x, A_pool, perm, seg_slot, seg_off, n_seg, scale, v_partial, T, d_in, r,
                     n_slots, ksplit, dt, ws, ws_bytes, stream):
    return _call("lora_sgmv_shrink", x, A_pool, perm, seg_slot, seg_off, n_seg, scale, v_partial,
                 T, d_in, r, n_slots, ksplit, dt, ws, ws_bytes, stream)


def lora_sgmv_expand(v_partial, ksplit, B_pool, perm, seg_slot, seg_off, n_seg, y, T, r, d_out,
                     n_slots, dt, ws, ws_bytes, stream):
    return _call("lora_sgmv_expand", v_partial, ksplit, B_pool, perm, seg_slot, seg_off, n_seg, y,
                 T, r, d_out, n_slots, dt, ws, ws_bytes, stream)


def lora_linear_fused(x, W0, A_pool, B_pool, slot_ids, scale, y, T, d_in, d_out, r, n_slots, dt,
                      ws, ws_bytes, stream):
    return _call("lora_linear_fused", x, W0, A_pool, B_pool, slot_ids, scale, y, T, d_in, d_out, r,
                 n_slots, dt, ws, ws_bytes, stream)


def lora_base_gemm_expand(x, W0, B_pool, slot_ids, v_partial, ksplit, y, T, d_in, d_out, r,
                          n_slots, dt, ws, ws_bytes, stream):
    return _call("lora_base_gemm_expand", x, W0, B_pool, slot_ids, v_partial, ksplit, y, T, d_in,
                 d_out, r, n_slots, dt, ws, ws_bytes, stream)


def lora_linear_fused_noalloc(x, W0, A_pool, B_pool, slot_ids, scale, y, T, d_in, d_out, r,
                              n_slots, dt, stream):
    return _call("lora_linear_fused_noalloc", x, W0, A_pool, B_pool, slot_ids, scale, y, T, d_in,
                 d_out, r, n_slots, dt, stream)


def lora_bgmv_delta(v_partial, ksplit, B_pool, slot_ids, delta, T, r, d_out, n_slots, dt, ws,
                    ws_bytes, stream):
    return _call("lora_bgmv_delta", v_partial, ksplit, B_pool, slot_ids, delta, T, r, d_out,
                 n_slots, dt, ws, ws_bytes, stream)


def lora_bgmv_adapter(x, A_pool, B_pool, slot_ids, scale, delta, T, d_in, d_out, r, n_slots, dt,
                      ws, ws_bytes, stream):
    return _call("lora_bgmv_adapter", x, A_pool, B_pool, slot_ids, scale, delta, T, d_in, d_out, r,
                 n_slots, dt, ws, ws_bytes, stream)


def lora_bgmv_adapter_merge(x, A_pool, B_pool, slot_ids, scale, partial, ksplit, y, T, d_in,
                            d_out, r, n_slots, dt, ws, ws_bytes, stream):
    return _call("lora_bgmv_adapter_merge", x, A_pool, B_pool, slot_ids, scale, partial, ksplit, y,
                 T, d_in, d_out, r, n_slots, dt, ws, ws_bytes, stream)


def lora_base_gemm_splitk(x, W0, partial, T, d_in, d_out, ksplit, dt, ws, ws_bytes, stream):
    return _call("lora_base_gemm_splitk", x, W0, partial, T, d_in, d_out, ksplit, dt, ws, ws_bytes,
                 stream)


def lora_decode_split(T, d_in, d_out):
    return _call("lora_decode_split", T, d_in, d_out)


def lora_debug_gemm_wait_timeout(x, W0, partial, T, d_in, d_out, wait_us, ws, ws_bytes, stream):
    return _call("lora_debug_gemm_wait_timeout", x, W0, partial, T, d_in, d_out, wait_us, ws,
                 ws_bytes, stream)


def lora_slot_upload(A_pool, B_pool, scale, slot, A_host, B_host, s, d_in, d_out, r, r_a, n_slots,
                     dt, stream):
    return _call("lora_slot_upload", A_pool, B_pool, scale, slot, A_host, B_host, s, d_in, d_out, r,
                 r_a, n_slots, dt, stream)


def lora_bgmv_adapter_ragged(x, A_flat, B_flat, a_off, b_off, rank, a_elems, b_elems, r_max,
                             slot_ids, scale, delta, T, d_in, d_out, n_slots, dt, ws, ws_bytes,
                             stream):
    return _call("lora_bgmv_adapter_ragged", x, A_flat, B_flat, a_off, b_off, rank, a_elems,
                 b_elems, r_max, slot_ids, scale, delta, T, d_in, d_out, n_slots, dt, ws, ws_bytes,
                 stream)


def lora_linear_fused_ragged(x, W0, A_flat, B_flat, a_off, b_off, rank, a_elems, b_elems, r_max,
                             slot_ids, scale, y, T, d_in, d_out, n_slots, dt, ws, ws_bytes, stream):
    return _call("lora_linear_fused_ragged", x, W0, A_flat, B_flat, a_off, b_off, rank, a_elems,
                 b_elems, r_max, slot_ids, scale, y, T, d_in, d_out, n_slots, dt, ws, ws_bytes,
                 stream)


def lora_quantize_base_4bit(W0, codebook, W0q, absmax, d_in, d_out, stream):
    return _call("lora_quantize_base_4bit", W0, codebook, W0q, absmax, d_in, d_out, stream)


def lora_base_gemm_4bit_splitk(x, W0q, absmax, codebook, partial, T, d_in, d_out, ksplit, ws,
                               ws_bytes, stream):
    return _call("lora_base_gemm_4bit_splitk", x, W0q, absmax, codebook, partial, T, d_in, d_out,
                 ksplit, ws, ws_bytes, stream)


def lora_linear_fused_4bit(x, W0q, absmax, codebook, A_pool, B_pool, slot_ids, scale, y, T, d_in,
                           d_out, r, n_slots, ws, ws_bytes, stream):
    return _call("lora_linear_fused_4bit", x, W0q, absmax, codebook, A_pool, B_pool, slot_ids,
                 scale, y, T, d_in, d_out, r, n_slots, ws, ws_bytes, stream)


def lora_get_error(ws, stream):
    out = ctypes.c_int32(0)
    st = _call("lora_get_error", ws, stream, ctypes.byref(out))
    return st, out.value


def lora_status_string(status):
    return _call("lora_status_string", status).decode()


# ----------------------------------------------------------- torch helpers
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dt(t):
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def check(status, what):
    if status != LORA_OK:
        raise LoraError(status, what)


def workspace(op, T, d_in, d_out, r, n_slots, device="cuda"):
    """A zero-filled workspace tensor for `op` (uint8, 256-byte aligned)."""
    import torch
    n = lora_workspace_bytes(op, T, d_in, d_out, r, n_slots)
    return torch.zeros(max(int(n), 16), dtype=torch.uint8, device=device)


def build_segments_t(slot_ids, n_slots, ws, stream=None):
    import torch
    T = slot_ids.numel()
    cap = max(1, min(T, n_slots))
    dev = slot_ids.device
    perm = torch.empty(max(T, 1), dtype=torch.int32, device=dev)
    seg_slot = torch.empty(cap, dtype=torch.int32, device=dev)
    seg_off = torch.empty(cap + 1, dtype=torch.int32, device=dev)
    n_seg = torch.empty(1, dtype=torch.int32, device=dev)
    check(lora_build_segments(_ptr(slot_ids), T, n_slots, _ptr(perm), _ptr(seg_slot),
                              _ptr(seg_off), _ptr(n_seg), _ptr(ws), ws.numel(), _stream(stream)),
          "lora_build_segments")
    return perm[:T], seg_slot, seg_off, n_seg


def bgmv_shrink_t(x, A_pool, slot_ids, scale, ksplit, ws, v_partial=None, stream=None):
    import torch
    T, d_in = x.shape
    n_slots, _, r = A_pool.shape
    if v_partial is None:
        v_partial = torch.empty((ksplit, T, r), dtype=torch.float32, device=x.device)
    check(lora_bgmv_shrink(_ptr(x), _ptr(A_pool), _ptr(slot_ids), _ptr(scale), _ptr(v_partial), T,
                           d_in, r, n_slots, ksplit, _dt(x), _ptr(ws), ws.numel(), _stream(stream)),
          "lora_bgmv_shrink")
    return v_partial


def bgmv_expand_t(v_partial, B_pool, slot_ids, y, ws, stream=None):
    ksplit, T, r = v_partial.shape
    n_slots, _, d_out = B_pool.shape
    check(lora_bgmv_expand(_ptr(v_partial), ksplit, _ptr(B_pool), _ptr(slot_ids), _ptr(y), T, r,
                           d_out, n_slots, _dt(y), _ptr(ws), ws.numel(), _stream(stream)),
          "lora_bgmv_expand")
    return y


def sgmv_shrink_t(x, A_pool, segs, scale, ksplit, ws, v_partial=None, stream=None):
    import torch
    perm, seg_slot, seg_off, n_seg = segs
    T, d_in = x.shape
    n_slots, _, r = A_pool.shape
    if v_partial is None:
        v_partial = torch.empty((ksplit, T, r), dtype=torch.float32, device=x.device)
    check(lora_sgmv_shrink(_ptr(x), _ptr(A_pool), _ptr(perm), _ptr(seg_slot), _ptr(seg_off),
                           _ptr(n_seg), _ptr(scale), _ptr(v_partial), T, d_in, r, n_slots, ksplit,
                           _dt(x), _ptr(ws), ws.numel(), _stream(stream)), "lora_sgmv_shrink")
    return v_partial


def sgmv_expand_t(v_partial, B_pool, segs, y, ws, stream=None):
    perm, seg_slot, seg_off, n_seg = segs
    ksplit, T, r = v_partial.shape
    n_slots, _, d_out = B_pool.shape
    check(lora_sgmv_expand(_ptr(v_partial), ksplit, _ptr(B_pool), _ptr(perm), _ptr(seg_slot),
                           _ptr(seg_off), _ptr(n_seg), _ptr(y), T, r, d_out, n_slots, _dt(y),
                           _ptr(ws), ws.numel(), _stream(stream)), "lora_sgmv_expand")
    return y


def linear_fused_t(x, W0, A_pool, B_pool, slot_ids, scale, ws, y=None, stream=None):
    """y = x W0 + s (x A) B for the batch; allocates y if not given."""
    import torch
    T, d_in = x.shape
    d_out = W0.shape[1]
    n_slots, _, r = A_pool.shape
    if y is None:
        y = torch.empty((T, d_out), dtype=x.dtype, device=x.device)
    check(lora_linear_fused(_ptr(x), _ptr(W0), _ptr(A_pool), _ptr(B_pool), _ptr(slot_ids),
                            _ptr(scale), _ptr(y), T, d_in, d_out, r, n_slots, _dt(x), _ptr(ws),
                            ws.numel(), _stream(stream)), "lora_linear_fused")
    return y


def base_gemm_expand_t(x, W0, B_pool, slot_ids, v_partial, ws, y=None, stream=None):
    """y = x W0 + (sum of v_partial) B_a, overwriting y (allocated if None)."""
    import torch
    T, d_in = x.shape
    d_out = W0.shape[1]
    n_slots, r, _ = B_pool.shape
    if y is None:
        y = torch.empty((T, d_out), dtype=x.dtype, device=x.device)
    check(lora_base_gemm_expand(_ptr(x), _ptr(W0), _ptr(B_pool), _ptr(slot_ids), _ptr(v_partial),
                                v_partial.shape[0], _ptr(y), T, d_in, d_out, r, n_slots, _dt(x),
                                _ptr(ws), ws.numel(), _stream(stream)), "lora_base_gemm_expand")
    return y


def bgmv_delta_t(v_partial, B_pool, slot_ids, ws, delta=None, stream=None):
    """fp32 adapter term delta[t] = v[t] B[a_t] (rows of base-only tokens untouched)."""
    import torch
    ksplit, T, r = v_partial.shape
    n_slots, _, d_out = B_pool.shape
    if delta is None:
        delta = torch.zeros((T, d_out), dtype=torch.float32, device=v_partial.device)
    check(lora_bgmv_delta(_ptr(v_partial), ksplit, _ptr(B_pool), _ptr(slot_ids), _ptr(delta), T, r,
                          d_out, n_slots, _dt(B_pool), _ptr(ws), ws.numel(), _stream(stream)),
          "lora_bgmv_delta")
    return delta


def bgmv_adapter_t(x, A_pool, B_pool, slot_ids, scale, ws, delta=None, stream=None):
    """fp32 adapter term delta[t] = s_a (x[t] A_a) B_a in one launch (rows of base-only
    tokens untouched)."""
    import torch
    T, d_in = x.shape
    n_slots, r, d_out = B_pool.shape
    if delta is None:
        delta = torch.zeros((T, d_out), dtype=torch.float32, device=x.device)
    check(lora_bgmv_adapter(_ptr(x), _ptr(A_pool), _ptr(B_pool), _ptr(slot_ids), _ptr(scale),
                            _ptr(delta), T, d_in, d_out, r, n_slots, _dt(x), _ptr(ws), ws.numel(),
                            _stream(stream)),
          "lora_bgmv_adapter")
    return delta


def slot_upload_t(A_pool, B_pool, scale, slot, A_host, B_host, s, stream=None):
    """Upload one adapter (host tensors A [d_in, r_a], B [r_a, d_out], pinned for overlap)
    into pool slot `slot`, zero-padded to the pool rank; scale[slot] = s."""
    n_slots, d_in, r = A_pool.shape
    d_out = B_pool.shape[2]
    r_a = A_host.shape[1]
    assert A_host.is_contiguous() and B_host.is_contiguous() and B_host.shape == (r_a, d_out)
    check(lora_slot_upload(_ptr(A_pool), _ptr(B_pool), _ptr(scale), slot, _ptr(A_host),
                           _ptr(B_host), float(s), d_in, d_out, r, r_a, n_slots, _dt(A_pool),
                           _stream(stream)),
          "lora_slot_upload")


def base_gemm_splitk_t(x, W0, ws, ksplit=None, partial=None, stream=None):
    """fp32 split-K base product partial[s] = x[:, K_s] W0[K_s, :].  ksplit
    None or 0: the split the fused layer uses (T <= 256; lora_decode_split
    slots); >= 1: that many equal splits of d_in for every column tile."""
    import torch
    T, d_in = x.shape
    d_out = W0.shape[1]
    if ksplit is None:
        ksplit = 0 if 1 <= T <= 256 else 1
    S = lora_decode_split(T, d_in, d_out) if ksplit == 0 else ksplit
    if partial is None:
        partial = torch.empty((max(S, 1), T, d_out), dtype=torch.float32, device=x.device)
    check(lora_base_gemm_splitk(_ptr(x), _ptr(W0), _ptr(partial), T, d_in, d_out, ksplit, _dt(x),
                                _ptr(ws), ws.numel(), _stream(stream)),
          "lora_base_gemm_splitk")
    return partial


def bgmv_adapter_merge_t(x, A_pool, B_pool, slot_ids, scale, partial, ws, y=None, stream=None):
    """y = sum_s partial[s] + s_a (x A_a) B_a, overwriting every row of y."""
    import torch
    T, d_in = x.shape
    n_slots, r, d_out = B_pool.shape
    if y is None:
        y = torch.empty((T, d_out), dtype=x.dtype, device=x.device)
    check(lora_bgmv_adapter_merge(_ptr(x), _ptr(A_pool), _ptr(B_pool), _ptr(slot_ids),
                                  _ptr(scale), _ptr(partial), partial.shape[0], _ptr(y), T, d_in,
                                  d_out, r, n_slots, _dt(x), _ptr(ws), ws.numel(),
                                  _stream(stream)),
          "lora_bgmv_adapter_merge")
    return y


def ragged_rank_class(r):
    """The stored rank of a rank-r adapter in a ragged pool: the next of 8, 16, 32, 64, 128."""
    for c in RAGGED_RANKS:
        if r <= c:
            return c
    raise ValueError(f"rank {r} > {RAGGED_RANKS[-1]}")


class RaggedPool:
    """A ragged-rank adapter pool on the device: slot a keeps A_a [d_in, rank[a]] at
    A_flat[a_off[a]:] and B_a [rank[a], d_out] at B_flat[b_off[a]:], each at its own
    rank (zero-padded only up to the next of 8, 16, 32, 64, 128)."""

    def __init__(self, A_list, B_list, device="cuda", dtype=None):
        """A_list[a] [d_in, r_a], B_list[a] [r_a, d_out] (torch tensors, any device)."""
        import torch
        if len(A_list) != len(B_list) or not A_list:
            raise ValueError("need one A and one B per slot")
        self.n_slots = len(A_list)
        self.d_in = int(A_list[0].shape[0])
        self.d_out = int(B_list[0].shape[1])
        dtype = dtype or A_list[0].dtype
        ranks = [ragged_rank_class(int(a.shape[1])) for a in A_list]
        a_off, b_off, a_n, b_n = [], [], 0, 0
        for rc in ranks:
            a_off.append(a_n)
            b_off.append(b_n)
            a_n += self.d_in * rc
            b_n += rc * self.d_out
        self.A_flat = torch.zeros(a_n, dtype=dtype, device=device)
        self.B_flat = torch.zeros(b_n, dtype=dtype, device=device)
        for a, (A, B, rc) in enumerate(zip(A_list, B_list, ranks)):
            r_a = int(A.shape[1])
            if A.shape[0] != self.d_in or tuple(B.shape) != (r_a, self.d_out):
                raise ValueError(f"slot {a}: shapes {tuple(A.shape)} / {tuple(B.shape)}")
            self.A_flat[a_off[a]:a_off[a] + self.d_in * rc].view(self.d_in, rc)[:, :r_a] = A
            self.B_flat[b_off[a]:b_off[a] + rc * self.d_out].view(rc, self.d_out)[:r_a] = B
        self.ranks = ranks
        self.r_max = max(ranks)
        self.a_off = torch.tensor(a_off, dtype=torch.int64, device=device)
        self.b_off = torch.tensor(b_off, dtype=torch.int64, device=device)
        self.rank = torch.tensor(ranks, dtype=torch.int32, device=device)

    @classmethod
    def from_padded(cls, A_pool, B_pool, ranks):
        """The ragged pool of a zero-padded one: slot a keeps its first ranks[a] columns of A
        and rows of B (the rest must be zero for the two to give the same layer)."""
        return cls([A_pool[a, :, :int(r)] for a, r in enumerate(ranks)],
                   [B_pool[a, :int(r), :] for a, r in enumerate(ranks)], device=A_pool.device)

    @property
    def nbytes(self):
        return (self.A_flat.numel() + self.B_flat.numel()) * self.A_flat.element_size()


def bgmv_adapter_ragged_t(x, pool, slot_ids, scale, ws, delta=None, stream=None):
    """bgmv_adapter_t over a RaggedPool."""
    import torch
    T, d_in = x.shape
    if delta is None:
        delta = torch.zeros((T, pool.d_out), dtype=torch.float32, device=x.device)
    check(lora_bgmv_adapter_ragged(_ptr(x), _ptr(pool.A_flat), _ptr(pool.B_flat),
                                   _ptr(pool.a_off), _ptr(pool.b_off), _ptr(pool.rank),
                                   pool.A_flat.numel(), pool.B_flat.numel(), pool.r_max,
                                   _ptr(slot_ids), _ptr(scale), _ptr(delta), T, d_in, pool.d_out,
                                   pool.n_slots, _dt(x), _ptr(ws), ws.numel(), _stream(stream)),
          "lora_bgmv_adapter_ragged")
    return delta


def linear_fused_ragged_t(x, W0, pool, slot_ids, scale, ws, y=None, stream=None):
    """linear_fused_t over a RaggedPool (bf16).  With ws = workspace(OP_LINEAR_FUSED_RAGGED,
    T, ...) batches above 256 tokens take the prefill route (the batch's adapters copied
    into a dense pool at rank r_max in ws, then the prefill path); with a workspace for
    256 tokens (OP_LINEAR_FUSED) they run as 256-token chunks of the decode path."""
    import torch
    T, d_in = x.shape
    d_out = W0.shape[1]
    if y is None:
        y = torch.empty((T, d_out), dtype=x.dtype, device=x.device)
    check(lora_linear_fused_ragged(_ptr(x), _ptr(W0), _ptr(pool.A_flat), _ptr(pool.B_flat),
                                   _ptr(pool.a_off), _ptr(pool.b_off), _ptr(pool.rank),
                                   pool.A_flat.numel(), pool.B_flat.numel(), pool.r_max,
                                   _ptr(slot_ids), _ptr(scale), _ptr(y), T, d_in, d_out,
                                   pool.n_slots, _dt(x), _ptr(ws), ws.numel(), _stream(stream)),
          "lora_linear_fused_ragged")
    return y


class Base4bit:
    """A 4-bit base matrix on the device: codes W0q [d_out, d_in / 2] uint8 (k contiguous
    per column, row 2i in the low nibble of byte i), absmax [d_in / 64, d_out] bf16,
    codebook [16] bf16."""

    def __init__(self, W0q, absmax, codebook):
        self.W0q, self.absmax, self.codebook = W0q, absmax, codebook
        self.d_out = int(W0q.shape[0])
        self.d_in = int(W0q.shape[1]) * 2

    @classmethod
    def quantize(cls, W0, codebook, stream=None):
        """Quantise a bf16 W0 [d_in, d_out] with the library's kernel."""
        import torch
        d_in, d_out = W0.shape
        W0q = torch.empty((d_out, d_in // 2), dtype=torch.uint8, device=W0.device)
        absmax = torch.empty((d_in // 64, d_out), dtype=torch.bfloat16, device=W0.device)
        check(lora_quantize_base_4bit(_ptr(W0), _ptr(codebook), _ptr(W0q), _ptr(absmax), d_in,
                                      d_out, _stream(stream)), "lora_quantize_base_4bit")
        return cls(W0q, absmax, codebook)

    @property
    def nbytes(self):
        return self.W0q.numel() + self.absmax.numel() * 2


def base_gemm_4bit_splitk_t(x, base, ws, ksplit=None, partial=None, stream=None):
    """fp32 split-K product partial[s] = x[:, K_s] deq(W0)[K_s, :] of a Base4bit."""
    import torch
    T, d_in = x.shape
    if ksplit is None:
        ksplit = lora_decode_split(T, d_in, base.d_out) or 1
    if partial is None:
        partial = torch.empty((ksplit, T, base.d_out), dtype=torch.float32, device=x.device)
    check(lora_base_gemm_4bit_splitk(_ptr(x), _ptr(base.W0q), _ptr(base.absmax),
                                     _ptr(base.codebook), _ptr(partial), T, d_in, base.d_out,
                                     ksplit, _ptr(ws), ws.numel(), _stream(stream)),
          "lora_base_gemm_4bit_splitk")
    return partial


def linear_fused_4bit_t(x, base, A_pool, B_pool, slot_ids, scale, ws, y=None, stream=None):
    """y = x deq(W0) + s (x A) B over a Base4bit (bf16).  ws: workspace(OP_LINEAR_FUSED_4BIT,
    T, ...); above 256 tokens it holds a dequantised copy of W0 for the prefill path."""
    import torch
    T, d_in = x.shape
    n_slots, _, r = A_pool.shape
    if y is None:
        y = torch.empty((T, base.d_out), dtype=x.dtype, device=x.device)
    check(lora_linear_fused_4bit(_ptr(x), _ptr(base.W0q), _ptr(base.absmax), _ptr(base.codebook),
                                 _ptr(A_pool), _ptr(B_pool), _ptr(slot_ids), _ptr(scale), _ptr(y),
                                 T, d_in, base.d_out, r, n_slots, _ptr(ws), ws.numel(),
                                 _stream(stream)),
          "lora_linear_fused_4bit")
    return y


def get_error_t(ws, stream=None):
    st, err = lora_get_error(_ptr(ws), _stream(stream))
    check(st, "lora_get_error")
    return err
