// Segment builder: a stable counting sort of the tokens by adapter slot.
//
// SGMV groups the tokens that use the same adapter so that each group is one
// small matrix product ("Serving multiple LoRAs: segmented matrix multiplies
// and adapter scheduling", SGMV bullet; its toy script groups the tokens with
// a stable sort of the ids and run-length counts).  Here the sort is a
// counting sort in one CTA, which is exactly a stable sort for integer keys:
//
//   bins:   bin 0 = base-only (id -1, and any id outside [-1, n_slots)),
//           bin a+1 = slot a.
//   1. the tokens are cut into P contiguous partitions (one warp each) and
//      every partition builds its own histogram in shared memory;
//   2. for each bin, an exclusive prefix over the partitions (in token order)
//      plus a block-wide exclusive scan over the bins gives every
//      (partition, bin) its first output position;
//   3. every warp walks its partition in token order, 32 tokens at a time;
//      __match_any_sync ranks equal bins inside the 32 tokens by lane order.
// Token order is preserved inside every bin, so the result equals a stable
// argsort bit for bit.  Then the non-empty bins >= 1 are compacted into the
// segment list.
#include "common.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kThreads = 1024;
constexpr size_t kSmemBudget = 200 * 1024;

// In-place exclusive scan of a[0..n) by the whole block; returns the total.
__device__ int block_exclusive_scan(int* a, int n, int* warp_tmp /* >= 33 */) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int chunk = (n + nt - 1) / nt;
  const int b0 = min(n, tid * chunk), b1 = min(n, b0 + chunk);
  int s = 0;
  for (int i = b0; i < b1; ++i) s += a[i];
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = (lane < (nt >> 5)) ? warp_tmp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_tmp[lane] = wi - w;
    if (lane == 31) warp_tmp[32] = wi;
  }
  __syncthreads();
  int run = warp_tmp[warp] + incl - s;
  for (int i = b0; i < b1; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  const int total = warp_tmp[32];
  __syncthreads();
  return total;
}

__device__ __forceinline__ int bin_of(int id, int n_slots) { return slot_valid(id, n_slots) ? id + 1 : 0; }

__global__ void __launch_bounds__(kThreads)
    build_segments_kernel(const int32_t* __restrict__ ids, int T, int n_slots, int P,
                          int32_t* __restrict__ perm, int32_t* __restrict__ seg_slot,
                          int32_t* __restrict__ seg_off, int32_t* __restrict__ n_seg_out,
                          uint32_t* err, int32_t* __restrict__ zero, int n_zero) {
  extern __shared__ int32_t sm[];
  __shared__ int warp_tmp[33];
  __shared__ int bad;
  const int nb = n_slots + 1;
  int32_t* cnt = sm;              // [P][nb]: per-partition histogram -> offsets
  int32_t* start = sm + P * nb;   // [nb + 1]: per-bin totals -> first positions
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < P * nb + nb + 1; i += blockDim.x) sm[i] = 0;
  for (int i = tid; i < n_zero; i += blockDim.x) zero[i] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();

  const int per = (T + P - 1) / P;
  if (warp < P) {
    const int t0 = warp * per, t1 = min(T, t0 + per);
    int32_t* c = cnt + warp * nb;
    for (int t = t0 + lane; t < t1; t += 32) {
      const int id = ids[t];
      if (id < -1 || id >= n_slots) bad = 1;
      atomicAdd(&c[bin_of(id, n_slots)], 1);
    }
  }
  __syncthreads();

  for (int b = tid; b < nb; b += blockDim.x) {
    int run = 0;
    for (int p = 0; p < P; ++p) {
      const int v = cnt[p * nb + b];
      cnt[p * nb + b] = run;
      run += v;
    }
    start[b] = run;
  }
  __syncthreads();
  block_exclusive_scan(start, nb, warp_tmp);

  if (warp < P) {
    const int t0 = warp * per, t1 = min(T, t0 + per);
    int32_t* c = cnt + warp * nb;
    const unsigned lt = (1u << lane) - 1u;
    for (int base = t0; base < t1; base += 32) {
      const int t = base + lane;
      const int b = (t < t1) ? bin_of(ids[t], n_slots) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, b);
      const int rank = __popc(peers & lt);
      const int pos = (b >= 0) ? start[b] + c[b] + rank : 0;
      __syncwarp();
      if (b >= 0 && rank == 0) c[b] += __popc(peers);
      __syncwarp();
      if (b >= 0) perm[checked_index(pos, T, err)] = t;
    }
  }
  __syncthreads();

  if (tid == 0) start[nb] = T;
  __syncthreads();
  int32_t* flag = cnt;  // partition offsets are no longer needed
  for (int b = tid; b < nb; b += blockDim.x) flag[b] = (b >= 1 && start[b + 1] > start[b]) ? 1 : 0;
  __syncthreads();
  const int nseg = block_exclusive_scan(flag, nb, warp_tmp);
  for (int b = 1 + tid; b < nb; b += blockDim.x) {
    if (start[b + 1] > start[b]) {
      const int j = flag[b];
      seg_slot[j] = b - 1;
      seg_off[j] = start[b];
    }
  }
  if (tid == 0) {
    seg_off[nseg] = T;
    *n_seg_out = nseg;
    if (bad) flag_error(err, LORA_DEVERR_BAD_SLOT);
  }
}

}  // namespace

cudaError_t launch_build_segments(const int32_t* ids, int T, int n_slots, int32_t* perm,
                                  int32_t* seg_slot, int32_t* seg_off, int32_t* n_seg,
                                  uint32_t* err, cudaStream_t st, int32_t* zero, int n_zero) {
  const size_t nb = static_cast<size_t>(n_slots) + 1;
  // partitions: as many warps as the shared-memory budget allows, but no
  // more than one per 32 tokens
  size_t p_smem = kSmemBudget / (4 * nb);
  p_smem = (p_smem > 1) ? p_smem - 1 : 1;
  int P = static_cast<int>(p_smem < 32 ? p_smem : 32);
  const int p_tok = (T + 31) / 32;
  if (P > p_tok) P = p_tok;
  if (P < 1) P = 1;
  const size_t smem = (static_cast<size_t>(P) * nb + nb + 1) * sizeof(int32_t);
  cudaError_t e = cudaFuncSetAttribute(build_segments_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBudget + 4 * 1024));
  if (e != cudaSuccess) return e;
  build_segments_kernel<<<1, kThreads, smem, st>>>(ids, T, n_slots, P, perm, seg_slot, seg_off,
                                                   n_seg, err, zero, zero != nullptr ? n_zero : 0);
  return cudaGetLastError();
}

}  // namespace lora
