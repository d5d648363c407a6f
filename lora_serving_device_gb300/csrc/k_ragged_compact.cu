// The prefill route of the ragged-rank layer: the adapters a batch uses,
// copied out of the ragged pool into a small dense pool at one rank, so that
// the prefill path of the padded layer (segments, SGMV shrink, base GEMM with
// the expand in its accumulator) runs over them.  ("Serving many LoRA
// adapters", section "Batching across different adapters": mixed ranks are
// served either by ragged indexing or by padding to a common rank.  Decode
// batches take the ragged indexing, where a token's cost is its own rank;
// prefill batches are bound by the base GEMM's tensor pipe, where the padded
// LoRA K-blocks of a tile cost a few percent of its MMAs, so they take the
// padding, but only for the adapters present and in a copy that lives for
// one call.)
//
// Inputs: the segments of the batch's slot ids (bins of valid slots in
// increasing slot order, from the segment builder).  Segment j is compact
// slot j:
//   A_c[j] [d_in, r_max]   = A_a with columns rank[a] .. r_max-1 zero
//   B_c[j] [r_max, d_out]  = B_a with rows rank[a] .. r_max-1 zero
//   scale_c[j]             = scale[a]
//   ids_c[t]               = j for a token of slot a = seg_slot[j], -1 for
//                            base-only and invalid ids
// A slot whose table entry breaks the pool's rules is copied as zeros (its
// tokens get no adapter term, as in the ragged merge kernel) and raises
// LORA_DEVERR_BAD_RANK; an id outside [-1, n_slots) raises
// LORA_DEVERR_BAD_SLOT.
#include "common.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kCompactThreads = 256;

__global__ void __launch_bounds__(kCompactThreads)
    ragged_compact_kernel(const bf16* __restrict__ A, const bf16* __restrict__ B,
                          const int64_t* __restrict__ a_off, const int64_t* __restrict__ b_off,
                          const int32_t* __restrict__ rank, int64_t a_elems, int64_t b_elems,
                          int r_max, const float* __restrict__ scale,
                          const int32_t* __restrict__ seg_slot, const int32_t* __restrict__ n_seg,
                          int n_slots, bf16* __restrict__ A_c, bf16* __restrict__ B_c,
                          float* __restrict__ scale_c, int d_in, int d_out, uint32_t* err) {
  const int j = blockIdx.x;
  if (j >= *n_seg) return;  // fewer adapters in the batch than compact slots
  const int a = checked_index(seg_slot[j], n_slots, err);
  int ra = rank[a];
  const int64_t ao = a_off[a], bo = b_off[a];
  const bool ok = (ra == 8 || ra == 16 || ra == 32 || ra == 64 || ra == 128) && ra <= r_max &&
                  ao >= 0 && bo >= 0 && ao % 8 == 0 && bo % 8 == 0 &&
                  ao <= a_elems - static_cast<int64_t>(d_in) * ra &&
                  bo <= b_elems - static_cast<int64_t>(ra) * d_out;
  const bool first = blockIdx.y == 0 && threadIdx.x == 0;
  if (!ok) {
    if (first) flag_error(err, LORA_DEVERR_BAD_RANK);
    ra = 0;  // nothing of the entry is read: the slot is all zeros
  }
  if (first) scale_c[j] = scale ? scale[a] : 1.f;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const int64_t stride = static_cast<int64_t>(gridDim.y) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x;
  // A: d_in rows of r_max elements (16-byte chunks); chunk q of row k comes
  // from A_a's row k when q < rank / 8
  {
    const int qa = r_max / 8, qs = ra / 8;
    const int64_t n = static_cast<int64_t>(d_in) * qa;
    const uint4* src = reinterpret_cast<const uint4*>(A + (ok ? ao : 0));
    uint4* dst = reinterpret_cast<uint4*>(A_c + static_cast<size_t>(j) * d_in * r_max);
    for (int64_t i = i0; i < n; i += stride) {
      const int64_t k = i / qa;
      const int q = static_cast<int>(i - k * qa);
      dst[i] = q < qs ? src[k * qs + q] : zero;
    }
  }
  // B: r_max rows of d_out elements; rows below rank are B_a's rows, in order
  {
    const int qb = d_out / 8;
    const int64_t n = static_cast<int64_t>(r_max) * qb;
    const int64_t n_src = static_cast<int64_t>(ra) * qb;
    const uint4* src = reinterpret_cast<const uint4*>(B + (ok ? bo : 0));
    uint4* dst = reinterpret_cast<uint4*>(B_c + static_cast<size_t>(j) * r_max * d_out);
    for (int64_t i = i0; i < n; i += stride) dst[i] = i < n_src ? src[i] : zero;
  }
}

// ids_c[t]: the segment (compact slot) of token t's slot, found by binary
// search over the increasing seg_slot; -1 for base-only and invalid ids.
__global__ void __launch_bounds__(kCompactThreads)
    ragged_remap_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ seg_slot,
                        const int32_t* __restrict__ n_seg, int32_t* __restrict__ ids_c, int T,
                        int n_slots, uint32_t* err) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int a = ids[t];
  int c = -1;
  if (slot_valid(a, n_slots)) {
    // a valid id has a segment, so n_seg >= 1 and the search ends on it
    int lo = 0, hi = *n_seg - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (seg_slot[mid] < a) lo = mid + 1;
      else hi = mid;
    }
    c = lo;
  } else if (a != -1) {
    flag_error(err, LORA_DEVERR_BAD_SLOT);
  }
  ids_c[t] = c;
}

}  // namespace

cudaError_t launch_ragged_compact(const void* A, const void* B, const RaggedPool& rp,
                                  const float* scale, const int32_t* seg_slot,
                                  const int32_t* n_seg, int n_c, int n_slots, void* A_c,
                                  void* B_c, float* scale_c, int d_in, int d_out, uint32_t* err,
                                  cudaStream_t st) {
  if (n_c <= 0) return cudaSuccess;
  // a few CTAs per adapter: one adapter is up to (d_in + d_out) x 128 x 2
  // bytes (4.7 MB at 4096 + 14336)
  const int64_t chunks = (static_cast<int64_t>(d_in) + d_out) * rp.r_max / 8;
  int gy = static_cast<int>((chunks + 4 * kCompactThreads - 1) / (4 * kCompactThreads));
  if (gy < 1) gy = 1;
  if (gy > 64) gy = 64;
  ragged_compact_kernel<<<dim3(n_c, gy), kCompactThreads, 0, st>>>(
      static_cast<const bf16*>(A), static_cast<const bf16*>(B), rp.a_off, rp.b_off, rp.rank,
      rp.a_elems, rp.b_elems, rp.r_max, scale, seg_slot, n_seg, n_slots,
      static_cast<bf16*>(A_c), static_cast<bf16*>(B_c), scale_c, d_in, d_out, err);
  return cudaGetLastError();
}

cudaError_t launch_ragged_remap(const int32_t* ids, const int32_t* seg_slot, const int32_t* n_seg,
                                int32_t* ids_c, int T, int n_slots, uint32_t* err,
                                cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  ragged_remap_kernel<<<(T + kCompactThreads - 1) / kCompactThreads, kCompactThreads, 0, st>>>(
      ids, seg_slot, n_seg, ids_c, T, n_slots, err);
  return cudaGetLastError();
}

}  // namespace lora
