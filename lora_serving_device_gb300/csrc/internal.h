// Internal launcher interface between the C-ABI entry points (lora_api.cu)
// and the kernel translation units.  Launchers assume validated arguments.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "lora.h"

namespace lora {

// Per-device facts the launchers need (cached after the first query).
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  size_t max_smem_optin = 0;
};
cudaError_t device_info(DeviceInfo* out);

// Segment builder: one CTA, see k_segments.cu.  It also zeroes the n_zero
// words at `zero` (the counters of the shrink's split fold), if given.
cudaError_t launch_build_segments(const int32_t* ids, int T, int n_slots, int32_t* perm,
                                  int32_t* seg_slot, int32_t* seg_off, int32_t* n_seg,
                                  uint32_t* err, cudaStream_t st, int32_t* zero = nullptr,
                                  int n_zero = 0);

// Gather kernels (CUDA cores), see k_gather.cu.
cudaError_t launch_bgmv_shrink(const void* x, const void* A, const int32_t* ids,
                               const float* scale, float* vpart, int T, int d_in, int r,
                               int n_slots, int ksplit, lora_dtype_t dt, uint32_t* err,
                               cudaStream_t st);
cudaError_t launch_bgmv_expand(const float* vpart, int ksplit, const void* B, const int32_t* ids,
                               void* y, int T, int r, int d_out, int n_slots, lora_dtype_t dt,
                               uint32_t* err, cudaStream_t st);
// `pdl` launches the shrink as a programmatic dependent of the previous
// kernel on the stream (used inside lora_linear_fused).
cudaError_t launch_sgmv_shrink(const void* x, const void* A, const int32_t* perm,
                               const int32_t* seg_slot, const int32_t* seg_off,
                               const int32_t* n_seg, const float* scale, float* vpart, int T,
                               int d_in, int r, int n_slots, int ksplit, lora_dtype_t dt,
                               uint32_t* err, cudaStream_t st, bool pdl);
cudaError_t launch_sgmv_expand(const float* vpart, int ksplit, const void* B, const int32_t* perm,
                               const int32_t* seg_slot, const int32_t* seg_off,
                               const int32_t* n_seg, void* y, int T, int r, int d_out,
                               int n_slots, lora_dtype_t dt, uint32_t* err, cudaStream_t st);

// scale[slot] = s, one thread (the scale upload of lora_slot_upload).
cudaError_t launch_set_scale(float* scale, int slot, float s, cudaStream_t st);
// Upper bound on SGMV work items (segment x token-chunk pairs) for a batch.
int sgmv_max_items(int T, int n_slots);
// ksplit the fused path uses for its shrink (SGMV / BGMV form).
int fused_shrink_ksplit(int T, int d_in, int n_slots, int num_sms);
// True when the fused prefill GEMM takes 256 x 256 tiles (k_fused_tc.cu).
bool fused_wide_tiles(int T, int d_out, int n_slots, int num_sms);
// ksplit of the tensor-core shrink when it folds its splits into one
// partial (the prefill path at rank 64 / 128), see k_sgmv_tc.cu.
int fold_shrink_ksplit(int T, int d_in, int n_slots, int num_sms);
int decode_shrink_ksplit(int T, int d_in);

// Base GEMM + expand-in-accumulator kernel, bf16 (tcgen05), see k_fused_tc.cu.
cudaError_t launch_fused_tc(const void* x, const void* W0, const void* B, const int32_t* ids,
                            const float* vpart, int v_ksplit, void* y, int T,
                            int d_in, int d_out, int r, int n_slots, uint32_t* err,
                            cudaStream_t st, const DeviceInfo& dev);
// The whole BGMV adapter term of a decode-sized bf16 batch in one launch
// (shrink, cluster sum of the rank-r partials, expand), see k_adapter.cu.
// One cluster of adapter_cluster_size(T, d_in, d_out, ragged) CTAs per token.
//  - launch_bgmv_adapter: fp32 into delta [T, d_out]; rows of base-only
//    tokens are not written.
//  - launch_bgmv_adapter_merge: y = sum of the S fp32 partials [S, T, d_out]
//    of the decode GEMM + the adapter term, bf16, every row written.  `pdl`:
//    launch as a programmatic dependent of that GEMM (it waits for it before
//    reading the partials).
int adapter_cluster_size(int T, int d_in, int d_out, bool ragged);
cudaError_t launch_bgmv_adapter(const void* x, const void* A, const void* B, const int32_t* ids,
                                const float* scale, float* delta, int T, int d_in, int d_out,
                                int r, int n_slots, uint32_t* err, cudaStream_t st);
cudaError_t launch_bgmv_adapter_merge(const void* x, const void* A, const void* B,
                                      const int32_t* ids, const float* scale,
                                      const float* partial, int S, void* y, int T, int d_in,
                                      int d_out, int r, int n_slots, uint32_t* err, bool pdl,
                                      cudaStream_t st);
// Ragged adapter pool: slot a holds A_a [d_in, rank[a]] at A + a_off[a] and
// B_a [rank[a], d_out] at B + b_off[a] (bf16 elements, row-major); a_elems /
// b_elems are the pools' lengths, r_max <= 128 the largest rank allowed.
struct RaggedPool {
  const int64_t* a_off;
  const int64_t* b_off;
  const int32_t* rank;
  int64_t a_elems, b_elems;
  int r_max;
};
// The two forms above over a ragged pool; a slot whose entry is out of range
// sets LORA_DEVERR_BAD_RANK and its rows are treated as base-only.
cudaError_t launch_bgmv_adapter_ragged(const void* x, const void* A, const void* B,
                                       const RaggedPool& rp, const int32_t* ids,
                                       const float* scale, float* delta, int T, int d_in,
                                       int d_out, int n_slots, uint32_t* err, cudaStream_t st);
cudaError_t launch_bgmv_adapter_ragged_merge(const void* x, const void* A, const void* B,
                                             const RaggedPool& rp, const int32_t* ids,
                                             const float* scale, const float* partial, int S,
                                             void* y, int T, int d_in, int d_out, int n_slots,
                                             uint32_t* err, bool pdl, cudaStream_t st);
// The prefill route of the ragged layer, see k_ragged_compact.cu.  Given the
// segments of the batch's ids (seg_slot / n_seg from the segment builder):
//  - launch_ragged_compact: segment j's adapter into compact slot j of a
//    dense bf16 pool at rank rp.r_max (A_c [n_c, d_in, r_max], B_c [n_c,
//    r_max, d_out], zero-padded; scale_c [n_c]); n_c >= the segment count;
//  - launch_ragged_remap: ids_c[t] = the compact slot of token t, or -1.
cudaError_t launch_ragged_compact(const void* A, const void* B, const RaggedPool& rp,
                                  const float* scale, const int32_t* seg_slot,
                                  const int32_t* n_seg, int n_c, int n_slots, void* A_c,
                                  void* B_c, float* scale_c, int d_in, int d_out, uint32_t* err,
                                  cudaStream_t st);
cudaError_t launch_ragged_remap(const int32_t* ids, const int32_t* seg_slot, const int32_t* n_seg,
                                int32_t* ids_c, int T, int n_slots, uint32_t* err,
                                cudaStream_t st);
// BGMV expand into an fp32 term: delta[t, :] = (sum_s vpart[s, t, :]) B[a_t]
// for tokens with a valid id (other rows untouched); bf16 B.  `pdl`: launch
// as a programmatic dependent of the shrink just before.
cudaError_t launch_bgmv_delta(const float* vpart, int ksplit, const void* B, const int32_t* ids,
                              float* delta, int T, int r, int d_out, int n_slots, uint32_t* err,
                              cudaStream_t st, bool pdl);
// Same contract for fp32 storage on CUDA cores, see k_fused_simt.cu.
cudaError_t launch_fused_f32(const float* x, const float* W0, const float* B, const int32_t* ids,
                             const float* vpart, int v_ksplit, float* y, int T, int d_in,
                             int d_out, int r, int n_slots, uint32_t* err, cudaStream_t st);

// Whether cuTensorMapEncodeTiled could be resolved (needed for bf16 fused).
bool tensor_map_available();
// 2-D bf16 tensor map with 128-byte swizzle: `inner` contiguous elements per
// row, `outer` rows `row_elems` apart, box box_inner x box_outer; elements
// outside the tensor read as zero.
bool encode_tensor_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_elems, uint32_t box_inner, uint32_t box_outer);
// 3-D bf16 tensor map with 128-byte swizzle: dims d0 (contiguous) x d1 x
// d2, box box0 x box1 x 1; elements outside the tensor read as zero.
bool encode_tensor_map_bf16_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                               uint64_t d2, uint32_t box0, uint32_t box1);
// SGMV shrink on tensor cores (bf16, r in {64, 128}), see k_sgmv_tc.cu; the
// same contract as launch_sgmv_shrink.  With `fold` (sgmv_shrink_tc_items
// zeroed words) and ksplit > 1, split 0 of vpart ends as the sum of all
// splits (in split order); the other splits hold their own partials.
bool sgmv_shrink_tc_supported(int r);
int sgmv_shrink_tc_items(int T, int n_slots);
cudaError_t launch_sgmv_shrink_tc(const void* x, const void* A, const int32_t* perm,
                                  const int32_t* seg_slot, const int32_t* seg_off,
                                  const int32_t* n_seg, const float* scale, float* vpart, int T,
                                  int d_in, int r, int n_slots, int ksplit, int32_t* fold,
                                  uint32_t* err, cudaStream_t st, bool pdl,
                                  const DeviceInfo& dev);
// SGMV expand on tensor cores (bf16, r in {64, 128}), see k_sgmv_tc.cu; the
// same contract as launch_sgmv_expand.
bool sgmv_expand_tc_supported(int r);
cudaError_t launch_sgmv_expand_tc(const float* vpart, int ksplit, const void* B,
                                  const int32_t* perm, const int32_t* seg_slot,
                                  const int32_t* seg_off, const int32_t* n_seg, void* y, int T,
                                  int r, int d_out, int n_slots, uint32_t* err, cudaStream_t st,
                                  const DeviceInfo& dev);
// 3-D fp32 tensor map without swizzle: dims d0 (contiguous) x d1 x d2,
// box box0 x box1 x 1; elements outside the tensor are not stored.
bool encode_tensor_map_f32_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                              uint64_t d2, uint32_t box0, uint32_t box1);
// 2-D tensor map without swizzle over 1-byte (uint8) or 2-byte (bf16)
// elements: `inner` contiguous elements per row, `outer` rows `row_bytes`
// apart, box box_inner x box_outer; elements outside read as zero.
bool encode_tensor_map_plain_2d(CUtensorMap* m, const void* base, int elem_bytes, uint64_t inner,
                                uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                                uint32_t box_outer);
// 2-D uint8 tensor map with 128-byte swizzle (box_inner <= 128 bytes).
bool encode_tensor_map_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// Decode-sized base GEMM over a 4-bit base (codes [d_out, d_in / 2] bytes,
// bf16 absmax [d_in / 64, d_out], bf16 codebook [16]), split over d_in into S
// fp32 partials like launch_decode_gemm, see k_decode_q4.cu.  d_in % 64 == 0,
// d_out % 32 == 0, 1 <= S <= decode_q4_max_split(d_in).
int decode_q4_max_split(int d_in);
cudaError_t launch_decode_q4(const void* x, const void* Wq, const void* absmax,
                             const void* codebook, float* partial, int T, int d_in, int d_out,
                             int S, uint32_t* err, bool pdl, cudaStream_t st,
                             const DeviceInfo& dev);
// 4-bit codes and absmax -> bf16 W [d_in, d_out], each weight rounded once
// (see k_decode_q4.cu); d_in % 64 == 0, d_out % 32 == 0.
cudaError_t launch_dequantize_q4(const void* Wq, const void* absmax, const void* codebook,
                                 void* W, int d_in, int d_out, cudaStream_t st);
// bf16 W0 [d_in, d_out] -> 4-bit codes and bf16 absmax (see k_decode_q4.cu).
cudaError_t launch_quantize_q4(const void* W0, const void* codebook, void* Wq, void* absmax,
                               int d_in, int d_out, cudaStream_t st);
// The fused layer's decode split is laid out for a 152-SM GB300
// (kDecodeScheduleCtas CTAs at most), not for the current device, so that
// the order of the fp32 additions (and so every result bit) and the
// workspace size are the same on every device.
constexpr int kDecodeScheduleCtas = 152;

// Decode-sized base GEMM split over d_in into S fp32 partials
// partial[z, t, :] = x[t, K_z] W0[K_z, :] (K_z: contiguous ranges of whole
// 64*KSUB-row blocks), see k_decode_tc.cu.  ksplit 0 takes
// decode_gemm_split.  `pdl`: launch as a programmatic dependent (W0 is
// prefetched before the wait, x after).  decode_gemm_split: the S the fused
// layer uses, tiles x S ~ kDecodeScheduleCtas (a function of the shapes
// only); decode_uniform_split: the 4-bit GEMM's split (the same rule);
// decode_gemm_max_split: the largest S the kernel takes.
int decode_gemm_split(int T, int d_in, int d_out);
int decode_gemm_max_split(int T, int d_in);
int decode_uniform_split(int T, int d_in, int d_out);
cudaError_t launch_decode_gemm(const void* x, const void* W0, float* partial, int T, int d_in,
                               int d_out, int ksplit, uint32_t* err, bool pdl, cudaStream_t st,
                               const DeviceInfo& dev);
// Diagnostic form for tests of the failure path: the same kernel (ksplit 1)
// with its TMA producer held back, so nothing ever arrives on the barrier
// the MMA issuer waits on, and every bounded wait gives up after wait_ns.
// The kernel raises LORA_DEVERR_TIMEOUT, skips its output, frees its
// tensor memory and returns.
cudaError_t launch_decode_gemm_held(const void* x, const void* W0, float* partial, int T,
                                    int d_in, int d_out, uint64_t wait_ns, uint32_t* err,
                                    cudaStream_t st, const DeviceInfo& dev);

// lora_linear_fused with one option: clear_error_word clears the
// workspace's error word on the stream once every argument has passed
// validation, right before the layer's kernels (lora_linear_fused_noalloc,
// whose workspace is a shared array inside the library, uses it).
lora_status_t linear_fused_impl(const void* x, const void* W0, const void* A_pool,
                                const void* B_pool, const int32_t* slot_ids, const float* scale,
                                void* y, int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                                int32_t n_slots, lora_dtype_t dt, void* ws, size_t ws_bytes,
                                void* stream, bool clear_error_word);

}  // namespace lora
