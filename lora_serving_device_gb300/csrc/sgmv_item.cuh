// SGMV work items ("Serving multiple LoRAs: segmented matrix multiplies and
// adapter scheduling", SGMV bullet: tokens are visited segment by segment).
// Shared by the CUDA-core and the tensor-core SGMV kernels.
#pragma once

#include "common.cuh"

namespace lora {

// Work item `item` -> (slot, first and one-past-last position in perm).
// Items enumerate each segment's kChunk-token chunks in segment order.  The
// whole block cooperates: every thread counts the chunks of a contiguous run of
// segments, a block-wide exclusive scan gives each run its first item, and
// the one thread whose run holds `item` writes the answer to shared memory.
// Every thread must call it; the result is valid after it returns.
template <int kChunk>
__device__ __forceinline__ void sgmv_item(int item, const int32_t* seg_slot,
                                          const int32_t* seg_off, int nseg, int* s_a, int* s_p0,
                                          int* s_p1) {
  __shared__ int warp_sum[33];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  if (tid == 0) *s_a = -1;
  const int per = (nseg + nt - 1) / nt;
  const int j0 = min(nseg, tid * per), j1 = min(nseg, j0 + per);
  int c = 0;
  for (int j = j0; j < j1; ++j)
    c += (ld_dep(seg_off + j + 1) - ld_dep(seg_off + j) + kChunk - 1) / kChunk;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nwarps ? warp_sum[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sum[lane] = wi - w;
  }
  __syncthreads();
  const int first = warp_sum[warp] + incl - c;
  if (item >= first && item < first + c) {
    int x = item - first;
    for (int j = j0; j < j1; ++j) {
      const int o0 = ld_dep(seg_off + j), o1 = ld_dep(seg_off + j + 1);
      const int cj = (o1 - o0 + kChunk - 1) / kChunk;
      if (x < cj) {
        *s_a = ld_dep(seg_slot + j);
        *s_p0 = o0 + x * kChunk;
        *s_p1 = min(o1, *s_p0 + kChunk);
        break;
      }
      x -= cj;
    }
  }
  __syncthreads();
}

}  // namespace lora
