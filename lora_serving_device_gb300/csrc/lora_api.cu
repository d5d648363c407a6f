// C-ABI entry points of liblora.so (declared in include/lora.h): argument
// validation, workspace carving and kernel enqueueing.  Nothing here
// allocates device memory or synchronises, except lora_get_error.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "lora.h"

namespace lora {
namespace {

constexpr int kMaxDevices = 64;
constexpr int32_t kMaxDim = 1 << 20;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool rank_ok(int32_t r) { return r == 8 || r == 16 || r == 32 || r == 64 || r == 128; }
bool dim_ok(int32_t d) { return d >= 8 && d % 8 == 0 && d <= kMaxDim; }
bool tokens_ok(int32_t T) { return T <= LORA_MAX_TOKENS; }
bool slots_ok(int32_t n) { return n >= 1 && n <= LORA_MAX_SLOTS; }
bool dtype_ok(lora_dtype_t dt) { return dt == LORA_DTYPE_BF16 || dt == LORA_DTYPE_F32; }
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr size_t kErrBytes = 16;
// Batches up to this many tokens take the BGMV shrink inside lora_linear_fused
// (one token per request in decode: "Serving multiple LoRAs ...", BGMV
// bullet); larger ones take the segment builder and the SGMV shrink.
constexpr int32_t kDecodeTokens = 256;

struct FusedWs {
  uint32_t* err;
  int32_t* perm;
  int32_t* seg_slot;
  int32_t* seg_off;
  int32_t* n_seg;
  int32_t* fold;   // counters of the shrink's split fold (prefill-sized batches only)
  int n_fold;
  float* vpart;
  float* partial;  // fp32 [S, T, d_out] split-K base product (decode-sized batches only)
  int ksplit;
  int split;       // S of the decode GEMM
  size_t bytes;
};

// Workspace of lora_linear_fused: error word, segment arrays, shrink
// partials, and for decode-sized batches the split-K fp32 base product.
FusedWs fused_ws_layout(void* ws, int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                        int32_t n_slots) {
  FusedWs w;
  const size_t cap = static_cast<size_t>(T < n_slots ? T : n_slots);
  uint8_t* base = static_cast<uint8_t*>(ws);
  size_t o = kErrBytes;
  const size_t o_perm = o;
  o += static_cast<size_t>(T) * 4;
  const size_t o_slot = o;
  o += cap * 4;
  const size_t o_off = o;
  o += (cap + 1) * 4;
  const size_t o_nseg = o;
  o += 4;
  const size_t o_fold = o;
  w.n_fold = T > kDecodeTokens ? sgmv_shrink_tc_items(T, n_slots) : 0;
  o += static_cast<size_t>(w.n_fold) * 4;
  o = round_up(o, 256);
  const size_t o_v = o;
  // The shrink split, the prefill tile form and the decode split are chosen
  // for a 152-SM GB300 (kDecodeScheduleCtas), not the current device, so
  // that the workspace size and every result bit are the same on every
  // device; any split is correct with every form.
  // At rank 64 / 128 the tensor-core shrink folds its splits into one
  // partial (bf16), so the GEMM's LoRA stages read v once.
  constexpr int kSms = kDecodeScheduleCtas;
  w.ksplit = T <= kDecodeTokens                          ? decode_shrink_ksplit(T, d_in)
              : sgmv_shrink_tc_supported(r)               ? fold_shrink_ksplit(T, d_in, n_slots, kSms)
              : fused_wide_tiles(T, d_out, n_slots, kSms) ? 1
                                                          : fused_shrink_ksplit(T, d_in, n_slots, kSms);
  o += static_cast<size_t>(w.ksplit) * T * r * 4;
  o = round_up(o, 256);
  const size_t o_d = o;
  // the split-K base product, S x T x d_out floats.  For T <= 256 there is
  // one token tile, so S does not depend on T: the ragged and 4-bit layers,
  // which run longer batches in chunks of at most 256 tokens, fit every
  // chunk in the region laid out for min(T, 256)
  size_t partial_rows = 0;
  w.split = 0;
  if (T <= kDecodeTokens) {
    w.split = decode_gemm_split(T, d_in, d_out);
    partial_rows = static_cast<size_t>(w.split) * T;
  }
  o += partial_rows * d_out * 4;
  w.bytes = round_up(o, 256);
  w.err = reinterpret_cast<uint32_t*>(base);
  w.perm = reinterpret_cast<int32_t*>(base + o_perm);
  w.seg_slot = reinterpret_cast<int32_t*>(base + o_slot);
  w.seg_off = reinterpret_cast<int32_t*>(base + o_off);
  w.n_seg = reinterpret_cast<int32_t*>(base + o_nseg);
  w.fold = w.n_fold > 0 ? reinterpret_cast<int32_t*>(base + o_fold) : nullptr;
  w.vpart = reinterpret_cast<float*>(base + o_v);
  w.partial = T <= kDecodeTokens ? reinterpret_cast<float*>(base + o_d) : nullptr;
  return w;
}

// Workspace of lora_linear_fused_4bit: T <= 256, the decode chain's layout;
// larger batches, the prefill layout followed by a bf16 copy of W0 [d_in,
// d_out] (the dequantised base the prefill GEMM reads).  `wd` gets that copy.
size_t q4_ws_bytes(void* ws, int32_t T, int32_t d_in, int32_t d_out, int32_t r, int32_t n_slots,
                   FusedWs* w, void** wd) {
  *w = fused_ws_layout(ws, T, d_in, d_out, r, n_slots);
  if (T <= kDecodeTokens) {
    *wd = nullptr;
    return w->bytes;
  }
  const size_t o = round_up(w->bytes, 256);
  *wd = static_cast<uint8_t*>(ws) + o;
  return o + static_cast<size_t>(d_in) * d_out * 2;
}

// Workspace of lora_linear_fused_ragged's prefill route (T > 256): the
// prefill layout of lora_linear_fused over a compact pool of n_c = min(T,
// n_slots) slots at rank r_max, then the compact ids [T], scales [n_c] and
// pool, A_c [n_c, d_in, r_max] and B_c [n_c, r_max, d_out] bf16.  The
// layout's segment arrays first hold the segments of the batch's own ids
// (at most n_c of them), which the compact pool is built from.
struct RaggedWs {
  FusedWs w;
  int32_t n_c;
  int32_t* ids_c;
  float* scale_c;
  void* A_c;
  void* B_c;
  size_t bytes;
};

RaggedWs ragged_ws_layout(void* ws, int32_t T, int32_t d_in, int32_t d_out, int32_t r_max,
                          int32_t n_slots) {
  RaggedWs rw;
  rw.n_c = T < n_slots ? T : n_slots;
  rw.w = fused_ws_layout(ws, T, d_in, d_out, r_max, rw.n_c);
  uint8_t* base = static_cast<uint8_t*>(ws);
  size_t o = round_up(rw.w.bytes, 256);
  rw.ids_c = reinterpret_cast<int32_t*>(base + o);
  o += static_cast<size_t>(T) * 4;
  rw.scale_c = reinterpret_cast<float*>(base + o);
  o = round_up(o + static_cast<size_t>(rw.n_c) * 4, 256);
  rw.A_c = base + o;
  o = round_up(o + static_cast<size_t>(rw.n_c) * d_in * r_max * 2, 256);
  rw.B_c = base + o;
  o += static_cast<size_t>(rw.n_c) * r_max * d_out * 2;
  rw.bytes = round_up(o, 256);
  return rw;
}

lora_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

// The library is built for sm_103a only.
lora_status_t check_device(DeviceInfo* out) {
  return device_info(out) == cudaSuccess
             ? ((out->cc_major == 10 && out->cc_minor == 3) ? LORA_OK : LORA_ERR_DEVICE)
             : LORA_ERR_CUDA;
}

// SGMV shrink: tensor cores for bf16 pools of rank 64 / 128 (there it is a
// GEMM the CUDA cores cannot feed), the CUDA-core kernel otherwise.
cudaError_t sgmv_shrink_any(const void* x, const void* A, const int32_t* perm,
                            const int32_t* seg_slot, const int32_t* seg_off, const int32_t* n_seg,
                            const float* scale, float* vpart, int T, int d_in, int r, int n_slots,
                            int ksplit, lora_dtype_t dt, uint32_t* err, cudaStream_t st, bool pdl,
                            const DeviceInfo& dev, int32_t* fold = nullptr,
                            int* v_parts = nullptr) {
  if (dt == LORA_DTYPE_BF16 && sgmv_shrink_tc_supported(r) && tensor_map_available()) {
    if (v_parts != nullptr) *v_parts = fold != nullptr ? 1 : ksplit;
    return launch_sgmv_shrink_tc(x, A, perm, seg_slot, seg_off, n_seg, scale, vpart, T, d_in, r,
                                 n_slots, ksplit, fold, err, st, pdl, dev);
  }
  if (v_parts != nullptr) *v_parts = ksplit;
  return launch_sgmv_shrink(x, A, perm, seg_slot, seg_off, n_seg, scale, vpart, T, d_in, r,
                            n_slots, ksplit, dt, err, st, pdl);
}

// SGMV expand: tensor cores for bf16 pools of rank 64 / 128, the CUDA-core
// kernel otherwise.
cudaError_t sgmv_expand_any(const float* vpart, int ksplit, const void* B, const int32_t* perm,
                            const int32_t* seg_slot, const int32_t* seg_off, const int32_t* n_seg,
                            void* y, int T, int r, int d_out, int n_slots, lora_dtype_t dt,
                            uint32_t* err, cudaStream_t st, const DeviceInfo& dev) {
  if (dt == LORA_DTYPE_BF16 && sgmv_expand_tc_supported(r) && tensor_map_available())
    return launch_sgmv_expand_tc(vpart, ksplit, B, perm, seg_slot, seg_off, n_seg, y, T, r, d_out,
                                 n_slots, err, st, dev);
  return launch_sgmv_expand(vpart, ksplit, B, perm, seg_slot, seg_off, n_seg, y, T, r, d_out,
                            n_slots, dt, err, st);
}

lora_status_t check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || !aligned16(ws) || ws_bytes < need) return LORA_ERR_WORKSPACE;
  return LORA_OK;
}

// 4-bit base shapes: whole 64-row scale blocks, 16-byte code rows.
bool q4_dims_ok(int32_t d_in, int32_t d_out) {
  return dim_ok(d_in) && dim_ok(d_out) && d_in % 64 == 0 && d_out % 32 == 0;
}

// Shared argument checks of the two ragged entry points.
lora_status_t ragged_args(const void* x, const void* A_flat, const void* B_flat,
                          const int64_t* a_off, const int64_t* b_off, const int32_t* rank,
                          int64_t a_elems, int64_t b_elems, int32_t r_max,
                          const int32_t* slot_ids, const void* out, int32_t T, int32_t T_max,
                          int32_t d_in, int32_t d_out, int32_t n_slots, lora_dtype_t dt) {
  if (T < 0 || a_elems < 0 || b_elems < 0) return LORA_ERR_INVALID_ARG;
  if (dt != LORA_DTYPE_BF16) return LORA_ERR_DTYPE;
  if (T > T_max || !dim_ok(d_in) || !dim_ok(d_out) || !rank_ok(r_max) ||
      !slots_ok(n_slots))
    return LORA_ERR_SHAPE;
  if (x == nullptr || A_flat == nullptr || B_flat == nullptr || a_off == nullptr ||
      b_off == nullptr || rank == nullptr || slot_ids == nullptr || out == nullptr ||
      !aligned16(x) || !aligned16(A_flat) || !aligned16(B_flat) || !aligned16(out))
    return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

}  // namespace

cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.device != dev) {
    DeviceInfo n;
    n.device = dev;
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    n.num_sms = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
    n.cc_major = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
    n.cc_minor = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    n.max_smem_optin = static_cast<size_t>(v);
    d = n;
  }
  *out = d;
  return cudaSuccess;
}

}  // namespace lora

using namespace lora;

extern "C" {

size_t lora_workspace_bytes(int32_t op, int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                            int32_t n_slots) {
  (void)d_out;
  if (op == LORA_OP_LINEAR_FUSED) {
    if (T < 0 || !rank_ok(r) || !slots_ok(n_slots) || d_in < 8 || d_out < 0) return kErrBytes;
    return fused_ws_layout(nullptr, T, d_in, d_out, r, n_slots).bytes;
  }
  if (op == LORA_OP_LINEAR_FUSED_4BIT) {
    if (T < 0 || !rank_ok(r) || !slots_ok(n_slots) || d_in < 8 || d_out < 0) return kErrBytes;
    FusedWs w;
    void* wd;
    return q4_ws_bytes(nullptr, T, d_in, d_out, r, n_slots, &w, &wd);
  }
  if (op == LORA_OP_LINEAR_FUSED_RAGGED) {
    if (T < 0 || !rank_ok(r) || !slots_ok(n_slots) || d_in < 8 || d_out < 0) return kErrBytes;
    if (T <= kDecodeTokens) return fused_ws_layout(nullptr, T, d_in, d_out, r, n_slots).bytes;
    return ragged_ws_layout(nullptr, T, d_in, d_out, r, n_slots).bytes;
  }
  return kErrBytes;
}

const char* lora_status_string(lora_status_t s) {
  switch (s) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG: null or misaligned pointer, or negative size";
    case LORA_ERR_SHAPE: return "LORA_ERR_SHAPE: unsupported dimension";
    case LORA_ERR_DTYPE: return "LORA_ERR_DTYPE: unknown dtype";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA: a CUDA call or kernel launch failed";
    case LORA_ERR_DEVICE: return "LORA_ERR_DEVICE: current device is not sm_103";
  }
  return "LORA_ERR_UNKNOWN";
}

lora_status_t lora_build_segments(const int32_t* slot_ids, int32_t T, int32_t n_slots,
                                  int32_t* perm, int32_t* seg_slot, int32_t* seg_off,
                                  int32_t* n_seg, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!tokens_ok(T) || !slots_ok(n_slots)) return LORA_ERR_SHAPE;
  if ((T > 0 && (slot_ids == nullptr || perm == nullptr || seg_slot == nullptr)) ||
      seg_off == nullptr || n_seg == nullptr)
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  return from_cuda(launch_build_segments(slot_ids, T, n_slots, perm, seg_slot, seg_off, n_seg,
                                         static_cast<uint32_t*>(ws),
                                         static_cast<cudaStream_t>(stream)));
}

lora_status_t lora_bgmv_shrink(const void* x, const void* A_pool, const int32_t* slot_ids,
                               const float* scale, float* v_partial, int32_t T, int32_t d_in,
                               int32_t r, int32_t n_slots, int32_t ksplit, lora_dtype_t dt,
                               void* ws, size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!dtype_ok(dt)) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || !dim_ok(d_in) || !rank_ok(r) || !slots_ok(n_slots) || ksplit < 1 ||
      ksplit > LORA_MAX_KSPLIT)
    return LORA_ERR_SHAPE;
  if (x == nullptr || A_pool == nullptr || slot_ids == nullptr || v_partial == nullptr ||
      !aligned16(x) || !aligned16(A_pool) || !aligned16(v_partial))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  return from_cuda(launch_bgmv_shrink(x, A_pool, slot_ids, scale, v_partial, T, d_in, r, n_slots,
                                      ksplit, dt, static_cast<uint32_t*>(ws),
                                      static_cast<cudaStream_t>(stream)));
}

lora_status_t lora_bgmv_expand(const float* v_partial, int32_t ksplit, const void* B_pool,
                               const int32_t* slot_ids, void* y, int32_t T, int32_t r,
                               int32_t d_out, int32_t n_slots, lora_dtype_t dt, void* ws,
                               size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!dtype_ok(dt)) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || !dim_ok(d_out) || !rank_ok(r) || !slots_ok(n_slots) || ksplit < 1 ||
      ksplit > LORA_MAX_KSPLIT)
    return LORA_ERR_SHAPE;
  if (v_partial == nullptr || B_pool == nullptr || slot_ids == nullptr || y == nullptr ||
      !aligned16(v_partial) || !aligned16(B_pool) || !aligned16(y))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  return from_cuda(launch_bgmv_expand(v_partial, ksplit, B_pool, slot_ids, y, T, r, d_out,
                                      n_slots, dt, static_cast<uint32_t*>(ws),
                                      static_cast<cudaStream_t>(stream)));
}

lora_status_t lora_sgmv_shrink(const void* x, const void* A_pool, const int32_t* perm,
                               const int32_t* seg_slot, const int32_t* seg_off,
                               const int32_t* n_seg, const float* scale, float* v_partial,
                               int32_t T, int32_t d_in, int32_t r, int32_t n_slots,
                               int32_t ksplit, lora_dtype_t dt, void* ws, size_t ws_bytes,
                               void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!dtype_ok(dt)) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || !dim_ok(d_in) || !rank_ok(r) || !slots_ok(n_slots) || ksplit < 1 ||
      ksplit > LORA_MAX_KSPLIT)
    return LORA_ERR_SHAPE;
  if (x == nullptr || A_pool == nullptr || perm == nullptr || seg_slot == nullptr ||
      seg_off == nullptr || n_seg == nullptr || v_partial == nullptr || !aligned16(x) ||
      !aligned16(A_pool) || !aligned16(v_partial))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  return from_cuda(sgmv_shrink_any(x, A_pool, perm, seg_slot, seg_off, n_seg, scale, v_partial,
                                   T, d_in, r, n_slots, ksplit, dt, static_cast<uint32_t*>(ws),
                                   static_cast<cudaStream_t>(stream), false, dev));
}

lora_status_t lora_sgmv_expand(const float* v_partial, int32_t ksplit, const void* B_pool,
                               const int32_t* perm, const int32_t* seg_slot,
                               const int32_t* seg_off, const int32_t* n_seg, void* y, int32_t T,
                               int32_t r, int32_t d_out, int32_t n_slots, lora_dtype_t dt,
                               void* ws, size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!dtype_ok(dt)) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || !dim_ok(d_out) || !rank_ok(r) || !slots_ok(n_slots) || ksplit < 1 ||
      ksplit > LORA_MAX_KSPLIT)
    return LORA_ERR_SHAPE;
  if (v_partial == nullptr || B_pool == nullptr || perm == nullptr || seg_slot == nullptr ||
      seg_off == nullptr || n_seg == nullptr || y == nullptr || !aligned16(v_partial) ||
      !aligned16(B_pool) || !aligned16(y))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  return from_cuda(sgmv_expand_any(v_partial, ksplit, B_pool, perm, seg_slot, seg_off, n_seg, y,
                                   T, r, d_out, n_slots, dt, static_cast<uint32_t*>(ws),
                                   static_cast<cudaStream_t>(stream), dev));
}

lora_status_t lora_linear_fused(const void* x, const void* W0, const void* A_pool,
                                const void* B_pool, const int32_t* slot_ids, const float* scale,
                                void* y, int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                                int32_t n_slots, lora_dtype_t dt, void* ws, size_t ws_bytes,
                                void* stream) {
  return linear_fused_impl(x, W0, A_pool, B_pool, slot_ids, scale, y, T, d_in, d_out, r, n_slots,
                           dt, ws, ws_bytes, stream, false);
}

}  // extern "C"

namespace lora {

// Segments, then the segment-grouped shrink (SGMV) into w.vpart: the first
// two kernels of the prefill path (the GEMM follows as their dependent).
// *v_parts gets the number of partials the GEMM sums: 1 where the
// tensor-core shrink folds its splits (the segment build zeroes its
// counters), w.ksplit otherwise.
cudaError_t prefill_adapter_shrink(const void* x, const void* A_pool, const int32_t* slot_ids,
                                   const float* scale, int32_t T, int32_t d_in, int32_t r,
                                   int32_t n_slots, lora_dtype_t dt, const FusedWs& w,
                                   cudaStream_t st, const DeviceInfo& dev, int* v_parts) {
  int32_t* fold = w.ksplit > 1 ? w.fold : nullptr;
  cudaError_t e = launch_build_segments(slot_ids, T, n_slots, w.perm, w.seg_slot, w.seg_off,
                                        w.n_seg, w.err, st, fold, w.n_fold);
  if (e != cudaSuccess) return e;
  return sgmv_shrink_any(x, A_pool, w.perm, w.seg_slot, w.seg_off, w.n_seg, scale, w.vpart, T,
                         d_in, r, n_slots, w.ksplit, dt, w.err, st, true, dev, fold, v_parts);
}

lora_status_t linear_fused_impl(const void* x, const void* W0, const void* A_pool,
                                const void* B_pool, const int32_t* slot_ids, const float* scale,
                                void* y, int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                                int32_t n_slots, lora_dtype_t dt, void* ws, size_t ws_bytes,
                                void* stream, bool clear_error_word) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!dtype_ok(dt)) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || !dim_ok(d_in) || !dim_ok(d_out) || !rank_ok(r) || !slots_ok(n_slots))
    return LORA_ERR_SHAPE;
  if (x == nullptr || W0 == nullptr || A_pool == nullptr || B_pool == nullptr ||
      slot_ids == nullptr || y == nullptr || !aligned16(x) || !aligned16(W0) ||
      !aligned16(A_pool) || !aligned16(B_pool) || !aligned16(y))
    return LORA_ERR_INVALID_ARG;
  if (x == y) return LORA_ERR_INVALID_ARG;
  const FusedWs w = fused_ws_layout(ws, T, d_in, d_out, r, n_slots);
  lora_status_t s = check_ws(ws, ws_bytes, w.bytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  if (dt == LORA_DTYPE_BF16 && !tensor_map_available()) return LORA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  // every argument has been checked: only now may the error word be cleared
  if (clear_error_word && cudaMemsetAsync(w.err, 0, kErrBytes, st) != cudaSuccess)
    return LORA_ERR_CUDA;
  const bool decode = T <= kDecodeTokens;
  if (decode && dt == LORA_DTYPE_BF16) {
    // decode-sized bf16 batch: the split-K base GEMM, then one kernel that
    // computes the per-token (BGMV, no sort) adapter term while the GEMM
    // streams W0 and, once the GEMM is done, sums its partials, adds the
    // term and stores y.  Both are programmatic dependents: the GEMM
    // streams W0 while the previous kernel in the stream finishes and reads
    // x only after it has.
    const int S = decode_gemm_split(T, d_in, d_out);
    e = launch_decode_gemm(x, W0, w.partial, T, d_in, d_out, 0, w.err, true, st, dev);
    if (e != cudaSuccess) return LORA_ERR_CUDA;
    return from_cuda(launch_bgmv_adapter_merge(x, A_pool, B_pool, slot_ids, scale, w.partial, S,
                                               y, T, d_in, d_out, r, n_slots, w.err, true, st));
  }
  int v_parts = w.ksplit;
  if (decode) {
    // decode-sized fp32 batch: per-token BGMV shrink, then the CUDA-core layer
    e = launch_bgmv_shrink(x, A_pool, slot_ids, scale, w.vpart, T, d_in, r, n_slots, w.ksplit,
                           dt, w.err, st);
  } else {
    // prefill-sized batch: segments, then the segment-grouped shrink (SGMV)
    e = prefill_adapter_shrink(x, A_pool, slot_ids, scale, T, d_in, r, n_slots, dt, w, st, dev,
                               &v_parts);
  }
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  if (dt == LORA_DTYPE_BF16)
    e = launch_fused_tc(x, W0, B_pool, slot_ids, w.vpart, v_parts, y, T, d_in, d_out, r, n_slots,
                        w.err, st, dev);
  else
    e = launch_fused_f32(static_cast<const float*>(x), static_cast<const float*>(W0),
                         static_cast<const float*>(B_pool), slot_ids, w.vpart, v_parts,
                         static_cast<float*>(y), T, d_in, d_out, r, n_slots, w.err, st);
  return from_cuda(e);
}

}  // namespace lora

extern "C" {

lora_status_t lora_base_gemm_expand(const void* x, const void* W0, const void* B_pool,
                                    const int32_t* slot_ids, const float* v_partial,
                                    int32_t ksplit, void* y, int32_t T, int32_t d_in,
                                    int32_t d_out, int32_t r, int32_t n_slots, lora_dtype_t dt,
                                    void* ws, size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!dtype_ok(dt)) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || !dim_ok(d_in) || !dim_ok(d_out) || !rank_ok(r) || !slots_ok(n_slots) ||
      ksplit < 1 || ksplit > LORA_MAX_KSPLIT)
    return LORA_ERR_SHAPE;
  if (x == nullptr || W0 == nullptr || B_pool == nullptr || slot_ids == nullptr ||
      v_partial == nullptr || y == nullptr || !aligned16(x) || !aligned16(W0) ||
      !aligned16(B_pool) || !aligned16(v_partial) || !aligned16(y) || x == y)
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  if (dt == LORA_DTYPE_BF16 && !tensor_map_available()) return LORA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = static_cast<uint32_t*>(ws);
  cudaError_t e;
  if (dt == LORA_DTYPE_BF16)
    e = launch_fused_tc(x, W0, B_pool, slot_ids, v_partial, ksplit, y, T, d_in, d_out, r,
                        n_slots, err, st, dev);
  else
    e = launch_fused_f32(static_cast<const float*>(x), static_cast<const float*>(W0),
                         static_cast<const float*>(B_pool), slot_ids, v_partial, ksplit,
                         static_cast<float*>(y), T, d_in, d_out, r, n_slots, err, st);
  return from_cuda(e);
}

lora_status_t lora_bgmv_delta(const float* v_partial, int32_t ksplit, const void* B_pool,
                              const int32_t* slot_ids, float* delta, int32_t T, int32_t r,
                              int32_t d_out, int32_t n_slots, lora_dtype_t dt, void* ws,
                              size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (dt != LORA_DTYPE_BF16) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || !dim_ok(d_out) || !rank_ok(r) || !slots_ok(n_slots) || ksplit < 1 ||
      ksplit > LORA_MAX_KSPLIT)
    return LORA_ERR_SHAPE;
  if (v_partial == nullptr || B_pool == nullptr || slot_ids == nullptr || delta == nullptr ||
      !aligned16(v_partial) || !aligned16(B_pool) || !aligned16(delta))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  return from_cuda(launch_bgmv_delta(v_partial, ksplit, B_pool, slot_ids, delta, T, r, d_out,
                                     n_slots, static_cast<uint32_t*>(ws),
                                     static_cast<cudaStream_t>(stream), false));
}

lora_status_t lora_bgmv_adapter(const void* x, const void* A_pool, const void* B_pool,
                                const int32_t* slot_ids, const float* scale, float* delta,
                                int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                                int32_t n_slots, lora_dtype_t dt, void* ws, size_t ws_bytes,
                                void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (dt != LORA_DTYPE_BF16) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || T > 65535 || !dim_ok(d_in) || !dim_ok(d_out) || !rank_ok(r) ||
      !slots_ok(n_slots))
    return LORA_ERR_SHAPE;
  if (x == nullptr || A_pool == nullptr || B_pool == nullptr || slot_ids == nullptr ||
      delta == nullptr || !aligned16(x) || !aligned16(A_pool) || !aligned16(B_pool) ||
      !aligned16(delta))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  return from_cuda(launch_bgmv_adapter(x, A_pool, B_pool, slot_ids, scale, delta, T, d_in, d_out,
                                       r, n_slots, static_cast<uint32_t*>(ws),
                                       static_cast<cudaStream_t>(stream)));
}

lora_status_t lora_bgmv_adapter_ragged(const void* x, const void* A_flat, const void* B_flat,
                                       const int64_t* a_off, const int64_t* b_off,
                                       const int32_t* rank, int64_t a_elems, int64_t b_elems,
                                       int32_t r_max, const int32_t* slot_ids,
                                       const float* scale, float* delta, int32_t T,
                                       int32_t d_in, int32_t d_out, int32_t n_slots,
                                       lora_dtype_t dt, void* ws, size_t ws_bytes, void* stream) {
  lora_status_t s = ragged_args(x, A_flat, B_flat, a_off, b_off, rank, a_elems, b_elems, r_max,
                                slot_ids, delta, T, 65535, d_in, d_out, n_slots, dt);
  if (s != LORA_OK) return s;
  if ((s = check_ws(ws, ws_bytes, kErrBytes)) != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  const RaggedPool rp{a_off, b_off, rank, a_elems, b_elems, r_max};
  return from_cuda(launch_bgmv_adapter_ragged(x, A_flat, B_flat, rp, slot_ids, scale, delta, T,
                                              d_in, d_out, n_slots, static_cast<uint32_t*>(ws),
                                              static_cast<cudaStream_t>(stream)));
}

lora_status_t lora_linear_fused_ragged(const void* x, const void* W0, const void* A_flat,
                                       const void* B_flat, const int64_t* a_off,
                                       const int64_t* b_off, const int32_t* rank,
                                       int64_t a_elems, int64_t b_elems, int32_t r_max,
                                       const int32_t* slot_ids, const float* scale, void* y,
                                       int32_t T, int32_t d_in, int32_t d_out, int32_t n_slots,
                                       lora_dtype_t dt, void* ws, size_t ws_bytes, void* stream) {
  lora_status_t s = ragged_args(x, A_flat, B_flat, a_off, b_off, rank, a_elems, b_elems, r_max,
                                slot_ids, y, T, LORA_MAX_TOKENS, d_in, d_out, n_slots, dt);
  if (s != LORA_OK) return s;
  if (W0 == nullptr || !aligned16(W0) || x == y) return LORA_ERR_INVALID_ARG;
  // above 256 tokens a workspace that holds the prefill route's layout takes
  // that route (it can be smaller than the chunked route's, which holds the
  // split-K partials); any other workspace must hold the chunked route's
  const RaggedWs rw = ragged_ws_layout(ws, T, d_in, d_out, r_max, n_slots);
  const bool prefill = T > kDecodeTokens && check_ws(ws, ws_bytes, rw.bytes) == LORA_OK;
  const FusedWs w = fused_ws_layout(ws, T < kDecodeTokens ? T : kDecodeTokens, d_in, d_out, r_max,
                                    n_slots);
  if (!prefill && (s = check_ws(ws, ws_bytes, w.bytes)) != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  if (!tensor_map_available()) return LORA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const RaggedPool rp{a_off, b_off, rank, a_elems, b_elems, r_max};
  if (prefill) {
    // prefill route: the batch's adapters into a dense pool at rank r_max in
    // the workspace, then lora_linear_fused's prefill path over it (segments,
    // SGMV shrink, the base GEMM with the expand in its accumulator)
    const FusedWs& wp = rw.w;
    cudaError_t e = launch_build_segments(slot_ids, T, n_slots, wp.perm, wp.seg_slot, wp.seg_off,
                                          wp.n_seg, wp.err, st);
    if (e == cudaSuccess)
      e = launch_ragged_compact(A_flat, B_flat, rp, scale, wp.seg_slot, wp.n_seg, rw.n_c, n_slots,
                                rw.A_c, rw.B_c, rw.scale_c, d_in, d_out, wp.err, st);
    if (e == cudaSuccess)
      e = launch_ragged_remap(slot_ids, wp.seg_slot, wp.n_seg, rw.ids_c, T, n_slots, wp.err, st);
    int v_parts = wp.ksplit;
    if (e == cudaSuccess)
      e = prefill_adapter_shrink(x, rw.A_c, rw.ids_c, rw.scale_c, T, d_in, r_max, rw.n_c,
                                 LORA_DTYPE_BF16, wp, st, dev, &v_parts);
    if (e == cudaSuccess)
      e = launch_fused_tc(x, W0, rw.B_c, rw.ids_c, wp.vpart, v_parts, y, T, d_in, d_out, r_max,
                          rw.n_c, wp.err, st, dev);
    return from_cuda(e);
  }
  // the decode chain of lora_linear_fused with the ragged merge kernel, over
  // chunks of at most 256 tokens (the GEMM of each chunk starts while the
  // previous chunk's merge runs)
  for (int c0 = 0; c0 < T; c0 += kDecodeTokens) {
    const int Tc = T - c0 < kDecodeTokens ? T - c0 : kDecodeTokens;
    const int S = decode_gemm_split(Tc, d_in, d_out);
    const uint16_t* xc = static_cast<const uint16_t*>(x) + static_cast<size_t>(c0) * d_in;  // bf16
    uint16_t* yc = static_cast<uint16_t*>(y) + static_cast<size_t>(c0) * d_out;
    cudaError_t e = launch_decode_gemm(xc, W0, w.partial, Tc, d_in, d_out, 0, w.err, true, st, dev);
    if (e != cudaSuccess) return LORA_ERR_CUDA;
    e = launch_bgmv_adapter_ragged_merge(xc, A_flat, B_flat, rp, slot_ids + c0, scale, w.partial,
                                         S, yc, Tc, d_in, d_out, n_slots, w.err, true, st);
    if (e != cudaSuccess) return LORA_ERR_CUDA;
  }
  return LORA_OK;
}

lora_status_t lora_quantize_base_4bit(const void* W0, const void* codebook, void* W0q,
                                      void* absmax, int32_t d_in, int32_t d_out, void* stream) {
  if (!q4_dims_ok(d_in, d_out)) return LORA_ERR_SHAPE;
  if (W0 == nullptr || codebook == nullptr || W0q == nullptr || absmax == nullptr ||
      !aligned16(W0) || !aligned16(W0q) || !aligned16(absmax))
    return LORA_ERR_INVALID_ARG;
  DeviceInfo dev;
  lora_status_t s = check_device(&dev);
  if (s != LORA_OK) return s;
  return from_cuda(launch_quantize_q4(W0, codebook, W0q, absmax, d_in, d_out,
                                      static_cast<cudaStream_t>(stream)));
}

lora_status_t lora_base_gemm_4bit_splitk(const void* x, const void* W0q, const void* absmax,
                                         const void* codebook, float* partial, int32_t T,
                                         int32_t d_in, int32_t d_out, int32_t ksplit, void* ws,
                                         size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!tokens_ok(T) || !q4_dims_ok(d_in, d_out) || ksplit < 1 ||
      ksplit > decode_q4_max_split(d_in))
    return LORA_ERR_SHAPE;
  if (x == nullptr || W0q == nullptr || absmax == nullptr || codebook == nullptr ||
      partial == nullptr || !aligned16(x) || !aligned16(W0q) || !aligned16(absmax) ||
      !aligned16(partial))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  if (!tensor_map_available()) return LORA_ERR_CUDA;
  return from_cuda(launch_decode_q4(x, W0q, absmax, codebook, partial, T, d_in, d_out, ksplit,
                                    static_cast<uint32_t*>(ws), false,
                                    static_cast<cudaStream_t>(stream), dev));
}

lora_status_t lora_linear_fused_4bit(const void* x, const void* W0q, const void* absmax,
                                     const void* codebook, const void* A_pool,
                                     const void* B_pool, const int32_t* slot_ids,
                                     const float* scale, void* y, int32_t T, int32_t d_in,
                                     int32_t d_out, int32_t r, int32_t n_slots, void* ws,
                                     size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (!tokens_ok(T) || !q4_dims_ok(d_in, d_out) || !rank_ok(r) || !slots_ok(n_slots))
    return LORA_ERR_SHAPE;
  if (x == nullptr || W0q == nullptr || absmax == nullptr || codebook == nullptr ||
      A_pool == nullptr || B_pool == nullptr || slot_ids == nullptr || y == nullptr ||
      !aligned16(x) || !aligned16(W0q) || !aligned16(absmax) || !aligned16(A_pool) ||
      !aligned16(B_pool) || !aligned16(y) || x == y)
    return LORA_ERR_INVALID_ARG;
  FusedWs w;
  void* wd = nullptr;
  lora_status_t s = check_ws(ws, ws_bytes, q4_ws_bytes(ws, T, d_in, d_out, r, n_slots, &w, &wd));
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  if (!tensor_map_available()) return LORA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (T <= kDecodeTokens) {
    // the decode chain of lora_linear_fused with the 4-bit base GEMM (split
    // evenly over d_in, the same number of ranges for every column tile)
    const int S = decode_uniform_split(T, d_in, d_out);
    e = launch_decode_q4(x, W0q, absmax, codebook, w.partial, T, d_in, d_out, S, w.err, true, st,
                         dev);
    if (e != cudaSuccess) return LORA_ERR_CUDA;
    return from_cuda(launch_bgmv_adapter_merge(x, A_pool, B_pool, slot_ids, scale, w.partial, S,
                                               y, T, d_in, d_out, r, n_slots, w.err, true, st));
  }
  // larger batches: W0 dequantised once into the workspace (each weight
  // rounded to bf16 once, as the decode GEMM feeds its MMAs), then the bf16
  // prefill path over it, so W0 is streamed once, not once per 256 tokens
  e = launch_dequantize_q4(W0q, absmax, codebook, wd, d_in, d_out, st);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  int v_parts = w.ksplit;
  e = prefill_adapter_shrink(x, A_pool, slot_ids, scale, T, d_in, r, n_slots, LORA_DTYPE_BF16, w,
                             st, dev, &v_parts);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  return from_cuda(launch_fused_tc(x, wd, B_pool, slot_ids, w.vpart, v_parts, y, T, d_in, d_out,
                                   r, n_slots, w.err, st, dev));
}

lora_status_t lora_base_gemm_splitk(const void* x, const void* W0, float* partial, int32_t T,
                                    int32_t d_in, int32_t d_out, int32_t ksplit, lora_dtype_t dt,
                                    void* ws, size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (dt != LORA_DTYPE_BF16) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || !dim_ok(d_in) || !dim_ok(d_out) || ksplit < 0 ||
      ksplit > decode_gemm_max_split(T, d_in) || (ksplit == 0 && T > kDecodeTokens))
    return LORA_ERR_SHAPE;
  if (x == nullptr || W0 == nullptr || partial == nullptr || !aligned16(x) || !aligned16(W0) ||
      !aligned16(partial))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  if (!tensor_map_available()) return LORA_ERR_CUDA;
  return from_cuda(launch_decode_gemm(x, W0, partial, T, d_in, d_out, ksplit,
                                      static_cast<uint32_t*>(ws), false,
                                      static_cast<cudaStream_t>(stream), dev));
}

lora_status_t lora_debug_gemm_wait_timeout(const void* x, const void* W0, float* partial,
                                           int32_t T, int32_t d_in, int32_t d_out,
                                           int32_t wait_us, void* ws, size_t ws_bytes,
                                           void* stream) {
  if (T < 1 || T > kDecodeTokens || !dim_ok(d_in) || !dim_ok(d_out)) return LORA_ERR_SHAPE;
  if (wait_us < 1 || wait_us > 2000000) return LORA_ERR_INVALID_ARG;
  if (x == nullptr || W0 == nullptr || partial == nullptr || !aligned16(x) || !aligned16(W0) ||
      !aligned16(partial))
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  if (!tensor_map_available()) return LORA_ERR_CUDA;
  return from_cuda(launch_decode_gemm_held(x, W0, partial, T, d_in, d_out,
                                           static_cast<uint64_t>(wait_us) * 1000ull,
                                           static_cast<uint32_t*>(ws),
                                           static_cast<cudaStream_t>(stream), dev));
}

lora_status_t lora_bgmv_adapter_merge(const void* x, const void* A_pool, const void* B_pool,
                                      const int32_t* slot_ids, const float* scale,
                                      const float* partial, int32_t ksplit, void* y, int32_t T,
                                      int32_t d_in, int32_t d_out, int32_t r, int32_t n_slots,
                                      lora_dtype_t dt, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if (dt != LORA_DTYPE_BF16) return LORA_ERR_DTYPE;
  if (!tokens_ok(T) || T > 65535 || !dim_ok(d_in) || !dim_ok(d_out) || !rank_ok(r) ||
      !slots_ok(n_slots) || ksplit < 1 || ksplit > LORA_MAX_KSPLIT)
    return LORA_ERR_SHAPE;
  if (x == nullptr || A_pool == nullptr || B_pool == nullptr || slot_ids == nullptr ||
      partial == nullptr || y == nullptr || !aligned16(x) || !aligned16(A_pool) ||
      !aligned16(B_pool) || !aligned16(partial) || !aligned16(y) || x == y)
    return LORA_ERR_INVALID_ARG;
  lora_status_t s = check_ws(ws, ws_bytes, kErrBytes);
  if (s != LORA_OK) return s;
  if (T == 0) return LORA_OK;
  DeviceInfo dev;
  if ((s = check_device(&dev)) != LORA_OK) return s;
  return from_cuda(launch_bgmv_adapter_merge(x, A_pool, B_pool, slot_ids, scale, partial, ksplit,
                                             y, T, d_in, d_out, r, n_slots,
                                             static_cast<uint32_t*>(ws), false,
                                             static_cast<cudaStream_t>(stream)));
}

int32_t lora_decode_split(int32_t T, int32_t d_in, int32_t d_out) {
  if (T < 1 || T > kDecodeTokens || !dim_ok(d_in) || !dim_ok(d_out)) return 0;
  return decode_gemm_split(T, d_in, d_out);
}

lora_status_t lora_slot_upload(void* A_pool, void* B_pool, float* scale, int32_t slot,
                               const void* A_host, const void* B_host, float s, int32_t d_in,
                               int32_t d_out, int32_t r, int32_t r_a, int32_t n_slots,
                               lora_dtype_t dt, void* stream) {
  if (!dtype_ok(dt)) return LORA_ERR_DTYPE;
  if (!dim_ok(d_in) || !dim_ok(d_out) || !rank_ok(r) || !slots_ok(n_slots) || slot < 0 ||
      slot >= n_slots || r_a < 1 || r_a > r)
    return LORA_ERR_SHAPE;
  if (A_pool == nullptr || B_pool == nullptr || A_host == nullptr || B_host == nullptr ||
      !aligned16(A_pool) || !aligned16(B_pool))
    return LORA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t es = dt == LORA_DTYPE_BF16 ? 2 : 4;
  uint8_t* A = static_cast<uint8_t*>(A_pool) + static_cast<size_t>(slot) * d_in * r * es;
  uint8_t* B = static_cast<uint8_t*>(B_pool) + static_cast<size_t>(slot) * r * d_out * es;
  // A: d_in rows of r_a values into rows of r values, then zero the padding
  if (cudaMemcpy2DAsync(A, r * es, A_host, r_a * es, r_a * es, d_in, cudaMemcpyHostToDevice,
                        st) != cudaSuccess)
    return LORA_ERR_CUDA;
  if (r_a < r && cudaMemset2DAsync(A + r_a * es, r * es, 0, (r - r_a) * es, d_in, st) != cudaSuccess)
    return LORA_ERR_CUDA;
  // B: r_a contiguous rows, then zero rows up to r
  if (cudaMemcpyAsync(B, B_host, static_cast<size_t>(r_a) * d_out * es, cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return LORA_ERR_CUDA;
  if (r_a < r && cudaMemsetAsync(B + static_cast<size_t>(r_a) * d_out * es, 0,
                                 static_cast<size_t>(r - r_a) * d_out * es, st) != cudaSuccess)
    return LORA_ERR_CUDA;
  if (scale != nullptr) return from_cuda(launch_set_scale(scale, slot, s, st));
  return LORA_OK;
}

lora_status_t lora_get_error(void* ws, void* stream, int32_t* device_err) {
  if (ws == nullptr || device_err == nullptr || !aligned16(ws)) return LORA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
  if (cudaMemcpyAsync(&host, ws, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return LORA_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(host), st) != cudaSuccess) return LORA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
  *device_err = static_cast<int32_t>(host);
  return LORA_OK;
}

}  // extern "C"
