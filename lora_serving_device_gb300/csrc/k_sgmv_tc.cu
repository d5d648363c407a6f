// SGMV shrink on tcgen05 tensor cores, for bf16 pools of rank 64 or 128
// ("Serving multiple LoRAs: segmented matrix multiplies and adapter
// scheduling", SGMV bullet: the tokens of one adapter's segment are
// multiplied by that adapter's factor as one small matrix product):
//
//   v_partial[s, t, :] = scale[a] * x[t, K_s] A[a][K_s, :]
//
// for the tokens t of one segment (adapter a), in chunks of 128 tokens,
// and the s-th 64-aligned range K_s of d_in.  At rank 64 and prefill sizes
// this is 4.8 GFLOP against ~100 MB, so on CUDA cores it is bound by FMAs;
// here it is a GEMM with M = 128 tokens (x rows gathered through perm,
// K-major), N = r (A[a] rows, MN-major) and K = d_in.
//
// When the item's tokens are consecutive rows of x (one prefill request),
// one thread brings each K-block of x and of A[a] by TMA.  Otherwise warps
// 0-3 gather the x rows with 16-byte cp.async into the 128-byte-swizzled
// K-major layout and one of their threads brings A[a]'s K-block by TMA.
// Warps 0-3 then run the epilogue (TMEM -> registers -> v_partial rows,
// scaled).  Warp 4 allocates TMEM and
// issues the MMAs.  Rows of base-only tokens are written as zeros by the
// first item's CTA.  Every wait is bounded; on timeout the kernel raises
// LORA_DEVERR_TIMEOUT and returns.
//
// SGMV expand on tensor cores (same page, same bullet; the expand is added
// to the base output):  y[t, :] += (sum_s v_partial[s, t, :]) B[a]  for the
// tokens of one segment, y bf16, read and written once.  At rank 64 over a
// prefill batch this is 16.7 GFLOP against ~0.6 GB, again beyond the CUDA
// cores.  A work item (128 tokens of one segment; at rank 64 also two short
// segments together) writes its V rows once into tensor memory, as bf16
// hi + lo halves (v = hi + lo keeps ~16 mantissa bits), then sweeps a group
// of 64-column half-tiles of d_out: B[a] by TMA through a ring fed by its own
// warp, MMAs of both halves into one of several TMEM accumulators, and an
// epilogue in which every warp moves its own rows of y (details at the
// expand's code below).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int kThreads = 160;  // warps 0-3: gather + epilogue, warp 4: MMA
constexpr int kTok = 128;      // tokens per work item (the MMA's M)
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ST ring stages: ST = 4 at rank 64 (~96 KiB, two CTAs per SM) or 3 (~72 KiB,
// three CTAs per SM, so more CTAs' start-up and drain overlap).  Grids of
// more than one wave at two CTAs per SM take the shallower ring.
template <int R, int ST>
struct ShrinkLayout {
  static constexpr uint32_t kX = kTok * 128;            // one 64-wide K block of x
  static constexpr uint32_t kA = (R / 64) * 8192;       // R columns x 64 K rows of A[a]
  static constexpr uint32_t kStage = kX + kA;
  static constexpr int kStages = ST;
  static constexpr int kLag = kStages - 1;              // cp.async groups in flight
  static constexpr uint32_t kBars = kStages * kStage;
  static constexpr uint32_t kTotal = kBars + (2 * kStages + 1) * 8 + 16;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = ptx::mbar_wait_bounded(bar, parity, abort, kWaitLimitNs) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Work items of the shrink: every segment's last 128-token chunk first, in
// segment order, then the other chunks.  A segment's last chunk is where
// decode tokens of the same adapter join a prefill request's rows, the
// items whose rows are gathered and take longest; numbering them first
// starts them first.  Every thread must call it; the result is valid after
// it returns (slot -1: no such item).
__device__ __forceinline__ void shrink_item(int item, const int32_t* seg_slot,
                                            const int32_t* seg_off, int nseg, int* s_a, int* s_p0,
                                            int* s_p1) {
  __shared__ int warp_sum[33];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  if (tid == 0) *s_a = -1;
  if (item < nseg) {  // segment `item`'s last chunk: one thread looks it up
    if (tid == 0) {
      const int o0 = ld_dep(seg_off + item), o1 = ld_dep(seg_off + item + 1);
      *s_a = ld_dep(seg_slot + item);
      *s_p0 = o0 + (o1 - o0 - 1) / kTok * kTok;
      *s_p1 = o1;
    }
    __syncthreads();
    return;
  }
  // the other chunks: every thread counts a run of segments, a block-wide
  // exclusive scan places the runs
  const int x0 = item - nseg;
  const int per = (nseg + nt - 1) / nt;
  const int j0 = min(nseg, tid * per), j1 = min(nseg, j0 + per);
  int c = 0;
  for (int j = j0; j < j1; ++j)
    c += (ld_dep(seg_off + j + 1) - ld_dep(seg_off + j) + kTok - 1) / kTok - 1;
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
  if (x0 >= first && x0 < first + c) {
    int x = x0 - first;
    for (int j = j0; j < j1; ++j) {
      const int o0 = ld_dep(seg_off + j), o1 = ld_dep(seg_off + j + 1);
      const int cj = (o1 - o0 + kTok - 1) / kTok - 1;
      if (x < cj) {
        *s_a = ld_dep(seg_slot + j);
        *s_p0 = o0 + x * kTok;
        *s_p1 = *s_p0 + kTok;
        break;
      }
      x -= cj;
    }
  }
  __syncthreads();
}

// Folds the d_in splits of one shrink item into split 0.  Every CTA of the
// item (one per split, blockIdx.y) counts itself on fold[item] after its
// partial rows are written; the CTA that counts last adds the other splits'
// rows to split 0's, in split order, so the sum does not depend on which
// CTA finishes last.  No CTA waits for another.  Every thread of the CTA
// calls it.
template <int R>
__device__ __forceinline__ void fold_splits(int32_t* fold, float* vpart, const int32_t* perm,
                                            int p0, int n_tok, int T, uint32_t* err) {
  __shared__ int s_rows[kTok];
  __shared__ int s_last;
  __threadfence();  // this CTA's rows before its count
  __syncthreads();
  if (threadIdx.x == 0)
    s_last = atomicAdd(fold + blockIdx.x, 1) == static_cast<int>(gridDim.y) - 1 ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < n_tok; i += blockDim.x) s_rows[i] = perm_row(perm, p0 + i, T, err);
  __syncthreads();
  constexpr int kQ = R / 4;  // float4 per row
  constexpr int kU = 4;      // float4 per thread per pass
  constexpr int kS = 4;      // splits loaded per round trip
  const int ks = gridDim.y, n = n_tok * kQ, nt = blockDim.x;
  const size_t plane = static_cast<size_t>(T) * R;
  for (int e0 = threadIdx.x; e0 < n; e0 += kU * nt) {
    float* p[kU];
    float4 acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * nt;
      p[u] = e < n ? vpart + static_cast<size_t>(s_rows[e / kQ]) * R + (e % kQ) * 4 : nullptr;
      acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int s0 = 0; s0 < ks; s0 += kS) {
      float4 v[kS][kU];
#pragma unroll
      for (int j = 0; j < kS; ++j)
#pragma unroll
        for (int u = 0; u < kU; ++u)
          v[j][u] = p[u] != nullptr && s0 + j < ks
                        ? __ldcg(reinterpret_cast<const float4*>(p[u] + (s0 + j) * plane))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < kS; ++j)
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (s0 + j < ks) {
            acc[u].x += v[j][u].x;
            acc[u].y += v[j][u].y;
            acc[u].z += v[j][u].z;
            acc[u].w += v[j][u].w;
          }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (p[u] != nullptr) *reinterpret_cast<float4*>(p[u]) = acc[u];
  }
}

template <int R, int ST>
__global__ void __launch_bounds__(kThreads, ST == 3 && R == 64 ? 3 : 2)
    sgmv_shrink_tc_kernel(const __grid_constant__ CUtensorMap tm_a,
                          const __grid_constant__ CUtensorMap tm_x, const bf16* x,
                          const int32_t* perm, const int32_t* seg_slot, const int32_t* seg_off,
                          const int32_t* n_seg, const float* scale, float* vpart, int T,
                          int d_in, int n_slots, int kchunk, int32_t* fold, uint32_t* err) {
  using Lay = ShrinkLayout<R, ST>;
  constexpr int S = Lay::kStages;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, R, false, true);
  __shared__ int s_a, s_p0, s_p1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBars);
  uint64_t* empty = full + S;
  uint64_t* accum = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort_f = reinterpret_cast<volatile int*>(accum + 1) + 1;

  pdl_launch_dependents();  // the base GEMM may start streaming W0 now
  pdl_wait();               // the segments are written by the previous kernel
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, s = blockIdx.y;
  const int nseg = ld_dep(n_seg);
  if (blockIdx.x == 0) {  // rows of base-only tokens are zero
    const int nbase = ld_dep(seg_off);
    for (int e = tid; e < nbase * R; e += kThreads)
      vpart[(static_cast<size_t>(s) * T + perm_row(perm, e / R, T, err)) * R + (e % R)] = 0.f;
  }
  shrink_item(blockIdx.x, seg_slot, seg_off, nseg, &s_a, &s_p0, &s_p1);
  if (s_a < 0) return;  // no such item (uniform over the CTA)
  const int a = checked_index(s_a, n_slots, err);
  const int p0 = s_p0, n_tok = s_p1 - s_p0;
  const int k0 = s * kchunk, k1 = min(d_in, k0 + kchunk);
  const int n_it = k1 > k0 ? (k1 - k0 + 63) / 64 : 0;
  const bool folds = fold != nullptr && gridDim.y > 1;
  if (n_it == 0) {  // an empty split of d_in still writes its (zero) rows
    for (int e = tid; e < n_tok * R; e += kThreads)
      vpart[(static_cast<size_t>(s) * T + perm_row(perm, p0 + e / R, T, err)) * R + (e % R)] = 0.f;
    if (folds) fold_splits<R>(fold, vpart, perm, p0, n_tok, T, err);
    return;
  }
  // perm is ascending within a segment, so the item's rows are consecutive
  // in x exactly when the first and last are n_tok - 1 apart
  const int row0 = perm_row(perm, p0, T, err);
  const bool contig = perm_row(perm, p0 + n_tok - 1, T, err) - row0 == n_tok - 1;

  if (warp == 4) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_a);
      ptx::prefetch_tmap(&tm_x);
      for (int i = 0; i < S; ++i) {
        // TMA only: one arrival; gather: every gathering thread + the TMA's
        ptx::mbar_init(&full[i], contig ? 1 : 4 * 32 + 1);
        ptx::mbar_init(&empty[i], 1);
      }
      ptx::mbar_init(accum, 1);
      *abort_f = 0;
      ptx::fence_mbar_init();
    }
    __syncwarp();
    ptx::tmem_alloc(tmem_slot, R);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4 && contig) {
    // ---------------- TMA producer (consecutive rows) ---------------------
    if (tid == 0) {
      for (int it = 0; it < n_it; ++it) {
        const int st = it % S;
        const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
        if (!ptx::mbar_wait_bounded(&empty[st], ph ^ 1u, abort_f, kWaitLimitNs)) break;
        uint8_t* X = smem + static_cast<size_t>(st) * Lay::kStage;
        const int kb = k0 + it * 64;
        ptx::mbar_arrive_expect_tx(&full[st], Lay::kStage);
        ptx::tma_load_2d(X, &tm_x, &full[st], kb, row0);
#pragma unroll
        for (int h = 0; h < R / 64; ++h)
          ptx::tma_load_3d(X + Lay::kX + h * 8192, &tm_a, &full[st], 64 * h, kb, a);
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------- gather producer ------------------------------------
    // thread -> 16-byte chunk c of rows (tid >> 3) + 16 q, q = 0..7
    const int c = tid & 7;
    int rowtok[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = (tid >> 3) + 16 * q;
      rowtok[q] = i < n_tok ? perm_row(perm, p0 + i, T, err) : -1;
    }
    bool ok = true;
    int it = 0;
    for (; it < n_it; ++it) {
      const int st = it % S;
      const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
      if (!warp_wait(&empty[st], ph ^ 1u, abort_f)) {
        ok = false;
        break;
      }
      uint8_t* X = smem + static_cast<size_t>(st) * Lay::kStage;
      const int kb = k0 + it * 64;
      if (tid == 0) {
        ptx::mbar_arrive_expect_tx(&full[st], Lay::kA);
#pragma unroll
        for (int h = 0; h < R / 64; ++h)
          ptx::tma_load_3d(X + Lay::kX + h * 8192, &tm_a, &full[st], 64 * h, kb, a);
      }
      const int col = kb + c * 8;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = (tid >> 3) + 16 * q;
        if (rowtok[q] >= 0) {
          const bool in = col < k1;
          const bf16* src = x + (in ? static_cast<size_t>(rowtok[q]) * d_in + col : 0);
          cp_async16(X + i * 128 + ((c ^ (i & 7)) << 4), src, in ? 16u : 0u);
        }
      }
      cp_async_commit();
      if (it >= Lay::kLag) {
        cp_async_wait<Lay::kLag>();
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&full[(it - Lay::kLag) % S]);
      }
    }
    cp_async_wait<0>();
    ptx::fence_proxy_async_smem();
    // the stages whose gather is complete but not yet signalled
    for (int j = (it > Lay::kLag ? it - Lay::kLag : 0); j < it; ++j) ptx::mbar_arrive(&full[j % S]);
    (void)ok;
  } else if (lane == 0) {
    // ---------------- MMA issuer -----------------------------------------
    for (int it = 0; it < n_it; ++it) {
      const int st = it % S;
      const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
      if (!ptx::mbar_wait_bounded(&full[st], ph, abort_f, kWaitLimitNs)) break;
      ptx::tc_fence_after();
      const uint32_t xa = ptx::smem_u32(smem + static_cast<size_t>(st) * Lay::kStage);
      const uint32_t aa = xa + Lay::kX;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // x: K-major, 16 elements = 32 bytes per step; A[a]: MN-major, 16
        // K-rows = 2048 bytes per step, 64-column boxes 8 KiB apart
        const uint64_t xd = ptx::sdesc_sw128(xa + kk * 32, 16, 1024);
        const uint64_t ad = ptx::sdesc_sw128(aa + kk * 2048, 8192, 1024);
        ptx::mma_bf16(tmem, xd, ad, kIdesc, (it > 0 || kk > 0) ? 1u : 0u);
      }
      ptx::mma_commit(&empty[st]);
    }
    ptx::mma_commit(accum);
  }

  if (warp < 4) {
    // ---------------- epilogue: TMEM row i = token perm[p0 + i] ------------
    const bool acc_ok = warp_wait(accum, 0, abort_f) && !*abort_f;
    if (acc_ok) {
      ptx::tc_fence_after();
      const int i = warp * 32 + lane;
      const float sc = scale ? scale[a] : 1.f;
      float* out = i < n_tok ? vpart + (static_cast<size_t>(s) * T + perm_row(perm, p0 + i, T, err)) * R
                             : nullptr;
      const uint32_t tq = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < R; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld16(tq + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
        ptx::tmem_ld16(tq + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
        ptx::tmem_ld_wait();
        if (out != nullptr) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(out + c0)[j] =
                make_float4(__uint_as_float(v[4 * j]) * sc, __uint_as_float(v[4 * j + 1]) * sc,
                            __uint_as_float(v[4 * j + 2]) * sc, __uint_as_float(v[4 * j + 3]) * sc);
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, R);
  }
  if (tid == 0 && *abort_f) flag_error(err, LORA_DEVERR_TIMEOUT);
  if (folds) fold_splits<R>(fold, vpart, perm, p0, n_tok, T, err);
}

template <int R, int ST>
cudaError_t launch_r(const CUtensorMap& tm, const CUtensorMap& tm_x, const bf16* x,
                     const int32_t* perm,
                     const int32_t* seg_slot, const int32_t* seg_off, const int32_t* n_seg,
                     const float* scale, float* vpart, int T, int d_in, int n_slots, int ksplit,
                     int32_t* fold, uint32_t* err, cudaStream_t st, bool pdl,
                     const DeviceInfo& dev) {
  using Lay = ShrinkLayout<R, ST>;
  const size_t smem = Lay::kTotal + 1024;
  if (smem > dev.max_smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = sgmv_shrink_tc_kernel<R, ST>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int per = (d_in + ksplit - 1) / ksplit;
  const int kchunk = (per + 63) / 64 * 64;
  const int items = sgmv_shrink_tc_items(T, n_slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items > 0 ? items : 1, ksplit);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tm, tm_x, x, perm, seg_slot, seg_off, n_seg, scale, vpart,
                            T, d_in, n_slots, kchunk, fold, err);
}

// ------------------------------------------------------------ expand
// y[rows of an item, the CTA's columns] += V B[a], V = the item's v rows
// summed over the d_in splits.  V sits in tensor memory as the MMAs' A
// operand, as bf16 hi + lo halves (hi = v rounded to bf16, lo = the rest
// rounded), so the product keeps v's fp32 precision.  The CTA walks its
// column tiles in 64-column half-tiles: one group of MMAs (N = 64) per
// half-tile into one of kNAcc 64-column accumulators (three at rank 64, so
// the MMAs run two half-tiles ahead of the epilogue), B[a] through a ring of
// half-tile boxes, y through kYBuf half-tile buffers.
constexpr int kXN = 128;      // d_out columns per tile
constexpr int kXGroup = 10;   // d_out tiles per CTA (20 half-tiles)
constexpr int kXGroupFull = 14;  // per CTA of a full item (28 half-tiles)
constexpr int kYBuf = 4;      // y half-tile buffers
constexpr int kYPitch = 144;  // bytes per token row moved by its own bulk copy
constexpr int kMinRun = 16;   // shortest run of consecutive rows moved by TMA
constexpr int kMaxTail = 16;  // most rows after such a run
constexpr int kPairTok = 16;  // segments this short share an item, two by two
constexpr int kXThreads = 192;  // warps 0-3: epilogue, warp 4: MMA, warp 5: B[a] loads
constexpr uint32_t kAccCols = 64;  // one accumulator: 64 fp32 columns
constexpr uint32_t kYWarp = 32 * 128;  // one warp's 32 rows of a TMA box buffer

// Work items of the expand.  Segments of more than kPairTok tokens give one
// item per 128-token chunk, in segment order; after them, every two
// consecutive segments of at most kPairTok tokens (decode tokens of adapters
// no prefill request uses) share one item, so that a CTA's sweep over its
// columns serves both.  With pairs off, every segment is chunked.  The whole
// block cooperates (each thread counts a run of segments, two block-wide
// scans place the runs); every thread must call it, and the result is valid
// after it returns.  The expand is not launched early, so the segments,
// written by an earlier kernel of the stream, are read through the cached
// read-only path.  it[0..2] = slot, first and one-past-last position in
// perm of the first part; it[3..5] the same for the second part (slot -1:
// none); it[0] = -1: no such item.
__device__ __forceinline__ void expand_item(int item, bool pairs, const int32_t* seg_slot,
                                            const int32_t* seg_off, int nseg, int* it) {
  __shared__ int ws_big[33], ws_small[33], tot[2];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  if (tid < 6) it[tid] = -1;
  const int per = (nseg + nt - 1) / nt;
  const int j0 = min(nseg, tid * per), j1 = min(nseg, j0 + per);
  int cb = 0, cs = 0;  // this run's big chunks and small segments
  for (int j = j0; j < j1; ++j) {
    const int n = __ldg(seg_off + j + 1) - __ldg(seg_off + j);
    if (pairs && n <= kPairTok) ++cs;
    else cb += (n + kTok - 1) / kTok;
  }
  int ib = cb, is = cs;  // inclusive scans within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int vb = __shfl_up_sync(0xffffffffu, ib, o), vs = __shfl_up_sync(0xffffffffu, is, o);
    if (lane >= o) { ib += vb; is += vs; }
  }
  if (lane == 31) { ws_big[warp] = ib; ws_small[warp] = is; }
  __syncthreads();
  if (warp == 0) {
    const int wb = lane < nwarps ? ws_big[lane] : 0, wsm = lane < nwarps ? ws_small[lane] : 0;
    int xb = wb, xs = wsm;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vb = __shfl_up_sync(0xffffffffu, xb, o), vs = __shfl_up_sync(0xffffffffu, xs, o);
      if (lane >= o) { xb += vb; xs += vs; }
    }
    ws_big[lane] = xb - wb;
    ws_small[lane] = xs - wsm;
    if (lane == 31) { tot[0] = xb; tot[1] = xs; }
  }
  __syncthreads();
  const int fb = ws_big[warp] + ib - cb;    // this run's first big chunk
  const int fs = ws_small[warp] + is - cs;  // and first small segment
  const int n_big = tot[0];
  if (item < n_big) {
    if (item >= fb && item < fb + cb) {
      int x = item - fb;
      for (int j = j0; j < j1; ++j) {
        const int o0 = __ldg(seg_off + j), o1 = __ldg(seg_off + j + 1);
        if (pairs && o1 - o0 <= kPairTok) continue;
        const int cj = (o1 - o0 + kTok - 1) / kTok;
        if (x < cj) {
          it[0] = __ldg(seg_slot + j);
          it[1] = o0 + x * kTok;
          it[2] = min(o1, it[1] + kTok);
          break;
        }
        x -= cj;
      }
    }
  } else {
    // small segments 2 q and 2 q + 1; the thread holding each writes its part
    const int q = item - n_big;
    for (int part = 0; part < 2; ++part) {
      const int k = 2 * q + part;
      if (k < fs || k >= fs + cs) continue;
      int x = k - fs;
      for (int j = j0; j < j1; ++j) {
        const int o0 = __ldg(seg_off + j), o1 = __ldg(seg_off + j + 1);
        if (o1 - o0 > kPairTok) continue;
        if (x == 0) {
          it[3 * part] = __ldg(seg_slot + j);
          it[3 * part + 1] = o0;
          it[3 * part + 2] = o1;
          break;
        }
        --x;
      }
    }
  }
  __syncthreads();
}

template <int R>
struct ExpandLayout {
  // B[a] ring: half-tile boxes of 64 columns x R rows (128-byte swizzle);
  // two CTAs per SM fit with four rank-64 boxes or two rank-128 ones
  static constexpr int kBRing = R == 64 ? 4 : 2;
  static constexpr uint32_t kBBox = R * 128;
  // y buffers of one half-tile (128 token rows x 64 columns).  Rows of a run
  // of consecutive y rows arrive by TMA with the 128-byte swizzle, row i at
  // i * 128 (the whole buffer head for a full item); the rows after a ragged
  // run (its tail) follow at kTail, kYPitch apart; an item moved row by row
  // has row i at i * kYPitch.
  static constexpr uint32_t kYHalf = kTok * 128;
  static constexpr uint32_t kTail = kYHalf;
  static constexpr uint32_t kYBufBytes =
      ((kTail + kMaxTail * kYPitch > kTok * kYPitch ? kTail + kMaxTail * kYPitch : kTok * kYPitch) +
       1023) / 1024 * 1024;
  static constexpr uint32_t kYOff = kBRing * kBBox;  // a multiple of 1024
  static constexpr uint32_t kBars = kYOff + kYBuf * kYBufBytes;
  // a pair's second B box sits in y buffer bs past its at most 2 kPairTok
  // rows (pairs are formed at rank 64 only)
  static constexpr uint32_t kPairB = 8192;
  static_assert(R != 64 || (2 * kPairTok * kYPitch <= kPairB && kPairB + kBBox <= kYBufBytes &&
                            kPairB % 1024 == 0 && kYBuf == kBRing),
                "pair B boxes in the y buffers");
  // tensor memory: kNAcc accumulators, then V hi (R / 2 columns of bf16
  // pairs) and V lo, in 256 columns
  static constexpr int kNAcc = R == 64 ? 3 : 2;
  static constexpr uint32_t kVCol = kNAcc * kAccCols;
  // b_full[kBRing], b_empty[kBRing], t_full[kNAcc], t_empty[kNAcc],
  // y_full[4 warps][kYBuf], TMEM slot, abort
  static constexpr int kNBar = 2 * kBRing + 2 * kNAcc + 4 * kYBuf;
  static constexpr uint32_t kTotal = kBars + kNBar * 8 + 16;
  static constexpr uint32_t kTmemCols = 256;
  static_assert(kVCol + R <= kTmemCols, "tensor memory");
};

// At most 128 registers a thread: measured, the kernel ran 6-20% slower on
// the prefill workload's full items in every build that used 155-168.
template <int R>
__global__ void __maxnreg__(128)
    sgmv_expand_tc_kernel(const __grid_constant__ CUtensorMap tm_b,
                          const __grid_constant__ CUtensorMap tm_y, const float* vpart, int ksplit,
                          const int32_t* perm, const int32_t* seg_slot, const int32_t* seg_off,
                          const int32_t* n_seg, bf16* y, int T, int d_out, uint32_t* err) {
  using Lay = ExpandLayout<R>;
  constexpr int kBRing = Lay::kBRing;
  constexpr int kNAcc = Lay::kNAcc;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 64, false, true);
  __shared__ int s_it[6];

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* b_full = reinterpret_cast<uint64_t*>(smem + Lay::kBars);
  uint64_t* b_empty = b_full + kBRing;
  uint64_t* t_full = b_empty + kBRing;
  uint64_t* t_empty = t_full + kNAcc;
  uint64_t* y_full = t_empty + kNAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(y_full + 4 * kYBuf);
  volatile int* abort_f = reinterpret_cast<volatile int*>(y_full + 4 * kYBuf) + 1;
  uint8_t* ybase = smem + Lay::kYOff;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // rank 64 pairs short segments (two copies of V and two accumulators fit
  // in tensor memory; at rank 128 they do not)
  const int nseg = ld_dep(n_seg);
  // every segment adds at most one chunk beyond T / 128 (pairs only merge
  // items), so CTAs past that bound hold no item and leave before the lookup
  if (static_cast<int>(blockIdx.x) >= (T + kTok - 1) / kTok + nseg) return;
  expand_item(blockIdx.x, R == 64, seg_slot, seg_off, nseg, s_it);
  if (s_it[0] < 0) return;  // no such item (uniform over the CTA)
  // B[a] and B[a2] arrive by TMA, which reads nothing outside the pool
  const int a = s_it[0], p0 = s_it[1], n1 = s_it[2] - s_it[1];
  const bool pair = s_it[3] >= 0;
  const int a2 = pair ? s_it[3] : a, p0b = s_it[4], n2 = pair ? s_it[5] - s_it[4] : 0;
  const int n_tok = n1 + n2;  // rows 0 .. n1 - 1 are the first part's tokens
  // accumulators, B ring depth (a pair takes two slots per half-tile) and
  // V's columns for this CTA
  const int nacc = pair ? 2 : kNAcc;
  const int bdepth = kBRing;
  const uint32_t vcol = pair ? 2 * kAccCols : Lay::kVCol, vcol2 = 2 * kAccCols + R;
  const int n_tiles_all = (d_out + kXN - 1) / kXN;
  if (static_cast<int>(blockIdx.y) * kXGroup >= n_tiles_all) return;

  // y moves in half-tiles in one of three ways, each epilogue warp moving
  // its own 32 rows.  The tokens of an item sit in increasing row order, so
  // the rows that are consecutive in y from its first one (a prefill request,
  // or its last item) are a prefix of n_run rows.
  //  - kFull (n_run = 128): a warp's rows of each half-tile are one 32-row
  //    TMA box, loaded, updated in place and stored back.
  //  - kRun (n_run >= kMinRun, at most kMaxTail rows after it): the run
  //    arrives as 32-row boxes (rows past it are read, never written), every
  //    tail row by its own bulk copy.
  //  - kRows (any other item, and every pair): every row arrives by its own
  //    bulk copy, issued by the epilogue thread that owns the row.
  // In kRun and kRows each thread stores its own row from registers, so a
  // buffer is free once it has been read and loads run kYBuf half-tiles
  // ahead; in kFull a buffer is free once the warp's TMA store has read it,
  // and loads run kYBuf - 1 ahead.
  enum { kFull, kRun, kRows };
  const int row0 = perm_row_plain(perm, p0, T, err);
  const int my_row = tid < n1      ? perm_row_plain(perm, p0 + tid, T, err)
                     : tid < n_tok ? perm_row_plain(perm, p0b + tid - n1, T, err)
                                   : -1;
  // the rows consecutive in y from the first (barrier: the rows are known)
  const int n_run = __syncthreads_count(tid < n_tok && my_row - row0 == tid);
  const int n_tail = n_tok - n_run;
  const int mode = pair ? kRows
                   : n_run == kTok ? kFull
                   : (n_run >= kMinRun && n_tail <= kMaxTail ? kRun : kRows);
  // column tiles of this CTA: a full item's CTA sweeps kXGroupFull of them
  // (fewer start-ups for the items that stream the most y; blockIdx.y past
  // its groups leaves), any other item's kXGroup.  Both were swept on a
  // 9081-token prefill batch at 4096 -> 14336 (full 10-16, other 7-14).
  const int grp = mode == kFull ? kXGroupFull : kXGroup;
  const int j0 = blockIdx.y * grp;
  const int nt = min(grp, n_tiles_all - j0);
  if (nt <= 0) return;  // uniform over the CTA; nothing is allocated yet
  const int n_half = 2 * nt;  // half-tiles of this CTA
  if (tid == 4 * 32) {
    ptx::prefetch_tmap(&tm_b);
    ptx::prefetch_tmap(&tm_y);
    for (int i = 0; i < kBRing; ++i) {
      ptx::mbar_init(&b_full[i], 1);
      ptx::mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kNAcc; ++i) {
      ptx::mbar_init(&t_full[i], 1);
      ptx::mbar_init(&t_empty[i], 4 * 32);
    }
    for (int i = 0; i < 4 * kYBuf; ++i) ptx::mbar_init(&y_full[i], 1);
    *abort_f = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 4) {
    __syncwarp();
    ptx::tmem_alloc(tmem_slot, Lay::kTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();  // the barriers are initialised and tensor memory is allocated
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool tail_row = mode == kRun && tid >= n_run && tid < n_tok;

  auto hcol = [&](int hj) { return j0 * kXN + 64 * hj; };
  auto ybuf = [&](int hj) { return ybase + (hj % kYBuf) * Lay::kYBufBytes; };
  // the bytes of one row inside half-tile hj moved by a bulk copy (columns
  // past d_out are not moved; d_out is a multiple of 8, so this is a
  // multiple of 16)
  auto row_bytes = [&](int hj) {
    const int c = d_out - hcol(hj);
    return static_cast<uint32_t>(c <= 0 ? 0 : (c < 64 ? c : 64) * 2);
  };
  // Each epilogue warp moves its own 32 rows of every half-tile (rows 32 w ..
  // 32 w + 31 of the item, 4 KiB at 4096 w of a TMA box buffer) and waits on
  // its own barrier per buffer, so the four warps never wait for each other.
  auto ybar = [&](int w, int hj) { return &y_full[w * kYBuf + hj % kYBuf]; };
  // lane 0 of warp w: the TMA part of the warp's rows of half-tile hj and the
  // byte count of its phase (bulk-copied rows may land before it is set)
  auto issue_y = [&](int w, int hj) {
    uint64_t* bar = ybar(w, hj);
    const int nr = min(32, n_tok - 32 * w);                   // the warp's rows
    const int nrun = mode == kRows ? 0 : max(0, min(32, n_run - 32 * w));  // of them by TMA
    uint32_t bytes = static_cast<uint32_t>(nr - nrun) * row_bytes(hj);
    if (nrun > 0) bytes += kYWarp;
    ptx::mbar_arrive_expect_tx(bar, bytes);
    if (nrun > 0)
      ptx::tma_load_2d(ybuf(hj) + w * kYWarp, &tm_y, bar, hcol(hj), row0 + 32 * w);
  };
  // the epilogue thread of row tid: its own bulk copy of half-tile hj
  auto issue_y_own = [&](int hj) {
    const uint32_t nb = row_bytes(hj);
    if (nb == 0) return;
    uint8_t* dst = nullptr;
    if (mode == kRows && tid < n_tok) dst = ybuf(hj) + tid * kYPitch;
    if (tail_row) dst = ybuf(hj) + Lay::kTail + (tid - n_run) * kYPitch;
    if (dst)
      ptx::bulk_load(dst, y + static_cast<size_t>(my_row) * d_out + hcol(hj), nb, ybar(tid >> 5, hj));
  };
  // B[a][:, half-tile hj] into ring slot bs = hj % bdepth; a pair's B[a2] box
  // goes to the part of y buffer bs that its 32 rows leave free (slots and
  // phases are stepped as counters in the loops: the accumulator count is
  // not a compile-time constant)
  auto bslot = [&](int bs, int part) {
    return part == 0 ? smem + bs * Lay::kBBox : ybase + bs * Lay::kYBufBytes + Lay::kPairB;
  };
  auto issue_b = [&](int hj, int bs) {
    ptx::mbar_arrive_expect_tx(&b_full[bs], (pair ? 2u : 1u) * Lay::kBBox);
    ptx::tma_load_3d(bslot(bs, 0), &tm_b, &b_full[bs], hcol(hj), 0, a);
    if (pair) ptx::tma_load_3d(bslot(bs, 1), &tm_b, &b_full[bs], hcol(hj), 0, a2);
  };
  // step a ring slot and its phase bit
  auto step = [](int& slot, uint32_t& phase, int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  };

  if (warp == 5) {
    if (lane == 0) {
      for (int hj = 0; hj < bdepth && hj < n_half; ++hj) issue_b(hj, hj);
    }
    __syncwarp();
  } else if (warp < 4) {
    if (warp * 32 < n_tok) {  // uniform over the warp
      for (int hj = 0; hj < kYBuf && hj < n_half; ++hj) {
        if (lane == 0) issue_y(warp, hj);
        issue_y_own(hj);
      }
    }
    // V rows into tensor memory: row i = token perm[p0 + i], summed over the
    // d_in splits in order (32 values of two splits per round of loads),
    // split into bf16 hi + lo, two K elements per 32-bit column.  The store
    // is collective over the warp: a warp with any row stores all 32 lanes
    // (rows past the item hold zeros; their accumulator rows are never read).
    // Plain loads: this kernel is not launched early, so stream order makes
    // v visible.
    if (warp * 32 < n_tok) {  // uniform over the warp
      const bool own = tid < n_tok;
      const float* vrow = vpart + static_cast<size_t>(own ? my_row : 0) * R;
      const size_t split = static_cast<size_t>(T) * R;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
      // f (32 values of the row, summed over the splits) -> V hi and lo.  A
      // pair keeps two copies of V, each with only its own part's rows (zeros
      // elsewhere), so one accumulator sums V1 B[a] + V2 B[a2] row by row.
      auto store_v = [&](int q0, const float (&f)[32]) {
        uint32_t hp[16], lp[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float h0 = __bfloat162float(__float2bfloat16_rn(f[2 * m]));
          const float h1 = __bfloat162float(__float2bfloat16_rn(f[2 * m + 1]));
          hp[m] = pack_bf16x2(h0, h1);
          lp[m] = pack_bf16x2(f[2 * m] - h0, f[2 * m + 1] - h1);
        }
        const uint32_t keep = !pair || tid < n1 ? ~0u : 0u;
#pragma unroll
        for (int m = 0; m < 16; ++m) { hp[m] &= keep; lp[m] &= keep; }
        ptx::tmem_st16(lane_base + vcol + q0 / 2, hp);
        ptx::tmem_st16(lane_base + vcol + R / 2 + q0 / 2, lp);
        if (pair) {
          // the rows of the first part are zero here, the others kept
          ptx::tmem_st_wait();
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const float h0 = __bfloat162float(__float2bfloat16_rn(f[2 * m]));
            const float h1 = __bfloat162float(__float2bfloat16_rn(f[2 * m + 1]));
            hp[m] = tid >= n1 ? pack_bf16x2(h0, h1) : 0u;
            lp[m] = tid >= n1 ? pack_bf16x2(f[2 * m] - h0, f[2 * m + 1] - h1) : 0u;
          }
          ptx::tmem_st16(lane_base + vcol2 + q0 / 2, hp);
          ptx::tmem_st16(lane_base + vcol2 + R / 2 + q0 / 2, lp);
        }
      };
      if (R == 64 && ksplit == 1) {
        // rank 64, one split: the whole row in one round of loads, nothing to add
        float4 u[R / 4];
        if (own) {
          const float4* pa = reinterpret_cast<const float4*>(vrow);
#pragma unroll
          for (int k = 0; k < R / 4; ++k) u[k] = pa[k];
        } else {
#pragma unroll
          for (int k = 0; k < R / 4; ++k) u[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q0 = 0; q0 < R; q0 += 32) {
          float f[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 w = u[q0 / 4 + k];
            f[4 * k] = w.x; f[4 * k + 1] = w.y; f[4 * k + 2] = w.z; f[4 * k + 3] = w.w;
          }
          store_v(q0, f);
        }
      } else {
        // 32 values of the row from two splits per round of loads (a whole
        // row of two splits per round needs ~168 registers, and the kernel
        // runs slower above 128)
#pragma unroll 1
        for (int q0 = 0; q0 < R; q0 += 32) {
          float f[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) f[k] = 0.f;
          for (int sp = 0; own && sp < ksplit; sp += 2) {
            const bool two = sp + 1 < ksplit;
            const float4* pa = reinterpret_cast<const float4*>(vrow + sp * split + q0);
            float4 u[8], w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) u[k] = pa[k];
            if (two) {
              const float4* pb = reinterpret_cast<const float4*>(vrow + (sp + 1) * split + q0);
#pragma unroll
              for (int k = 0; k < 8; ++k) w[k] = pb[k];
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              f[4 * k] += u[k].x; f[4 * k + 1] += u[k].y; f[4 * k + 2] += u[k].z; f[4 * k + 3] += u[k].w;
            }
            if (two) {
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                f[4 * k] += w[k].x; f[4 * k + 1] += w[k].y; f[4 * k + 2] += w[k].z; f[4 * k + 3] += w[k].w;
              }
            }
          }
          store_v(q0, f);
        }
      }
      ptx::tmem_st_wait();
    }
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();

  if (warp == 4) {
    // ---------------- MMA issuer -----------------------------------------
    if (lane == 0) {
      int bs = 0, ts = 0;  // B slot and accumulator of half-tile hj
      uint32_t bph = 0, tph = 0;
      for (int hj = 0; hj < n_half; ++hj, step(bs, bph, bdepth), step(ts, tph, nacc)) {
        if (!ptx::mbar_wait_bounded(&b_full[bs], bph, abort_f, kWaitLimitNs)) break;
        if (!ptx::mbar_wait_bounded(&t_empty[ts], tph ^ 1u, abort_f, kWaitLimitNs)) break;
        ptx::tc_fence_after();
        const uint32_t acc = tmem + static_cast<uint32_t>(ts) * kAccCols;
        for (int part = 0; part < (pair ? 2 : 1); ++part) {
          const uint32_t bb = ptx::smem_u32(bslot(bs, part));
          const uint32_t vc = part ? vcol2 : vcol;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int kk = 0; kk < R / 16; ++kk) {
              // A: V hi or lo, 16 K elements = 8 columns per step; B:
              // MN-major, 16 K rows = 2048 bytes per step
              const uint32_t va = tmem + vc + half * (R / 2) + kk * 8;
              const uint64_t bd = ptx::sdesc_sw128(bb + kk * 2048, Lay::kBBox, 1024);
              ptx::mma_bf16_ta(acc, va, bd, kIdesc, (part > 0 || half > 0 || kk > 0) ? 1u : 0u);
            }
          }
        }
        ptx::mma_commit(&b_empty[bs]);
        ptx::mma_commit(&t_full[ts]);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- B[a] loads: a slot takes half-tile hj + bdepth once
    // the MMAs of half-tile hj are done ------------------------------------
    if (lane == 0) {
      int bs = 0;
      uint32_t bph = 0;
      for (int hj = 0; hj + bdepth < n_half; ++hj, step(bs, bph, bdepth)) {
        if (!ptx::mbar_wait_bounded(&b_empty[bs], bph, abort_f, kWaitLimitNs)) break;
        issue_b(hj + bdepth, bs);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: y half-tiles += accumulator rows -----------
    // TMEM lane = token row i of the tile; thread i reads its row of each
    // half-tile from the buffer and adds its accumulator row.  kFull writes
    // the sum back in place for one TMA store of the half-tile; the other
    // modes store the row straight from registers (16 bytes per store).
    // Every epilogue thread passes the same waits and named barriers, aborted
    // or not.  A warp waits only on its own y barriers, and the accumulator
    // barriers keep every warp within kNAcc half-tiles of the slowest, so no
    // phase can complete twice before a thread has waited on it.
    const int i = warp * 32 + lane;
    const bool own = i < n_tok;
    const bool rows = warp * 32 < n_tok;  // this warp has rows (uniform)
    const uint32_t tq = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bf16* const yrow = own ? y + static_cast<size_t>(my_row) * d_out : nullptr;
    // this thread's row of a buffer: swizzled rows of a TMA box, else
    // kYPitch-apart rows of bulk copies
    const bool swz = mode == kFull || (mode == kRun && i < n_run);
    const uint32_t row_off = swz ? static_cast<uint32_t>(i) * 128
                           : (mode == kRun ? Lay::kTail + static_cast<uint32_t>(i - n_run) * kYPitch
                                           : static_cast<uint32_t>(i) * kYPitch);
    bool ok = true;
    int ts = 0;  // accumulator of half-tile hj, and its phase
    uint32_t tph = 0;
#pragma unroll 1
    for (int hj = 0; hj < n_half; ++hj, step(ts, tph, nacc)) {
      ok = ok && warp_wait(&t_full[ts], tph, abort_f);
      if (ok) ptx::tc_fence_after();
      if (rows)
        ok = ok && warp_wait(ybar(warp, hj), static_cast<uint32_t>(hj / kYBuf) & 1u, abort_f);
      uint8_t* const buf = ybuf(hj);
      uint8_t* const yb = buf + row_off;
      const uint32_t acc = tq + static_cast<uint32_t>(ts) * kAccCols;
      // the accumulator is free once its last columns are in registers: the
      // MMAs of half-tile hj + kNAcc may start while these are added
      bool freed = false;
      auto free_acc = [&]() {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&t_empty[ts]);
        freed = true;
      };
      if (ok && mode == kFull) {
        // in place, 32 columns at a time, for the TMA store
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld16(acc + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
          ptx::tmem_ld16(acc + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
          ptx::tmem_ld_wait();
          if (c0 == 32) free_acc();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4* p = reinterpret_cast<uint4*>(yb + ((((c0 >> 3) + q) ^ (i & 7)) << 4));
            const uint4 w = *p;
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              f[2 * e] = bf16_lo(u[e]) + __uint_as_float(v[8 * q + 2 * e]);
              f[2 * e + 1] = bf16_hi(u[e]) + __uint_as_float(v[8 * q + 2 * e + 1]);
            }
            *p = pack8_bf16(f);
          }
        }
      } else if (ok && rows) {
        // 32 columns at a time: the row's chunks read, then the sums stored
        // from registers
        const int col = hcol(hj);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint4 yv[4];
          if (own) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int ch = (c0 >> 3) + q;
              yv[q] = *reinterpret_cast<const uint4*>(yb + ((swz ? ch ^ (i & 7) : ch) << 4));
            }
          }
          uint32_t v[32];
          ptx::tmem_ld16(acc + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
          ptx::tmem_ld16(acc + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
          ptx::tmem_ld_wait();
          if (c0 == 32) free_acc();
          if (own) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t u[4] = {yv[q].x, yv[q].y, yv[q].z, yv[q].w};
              float f[8];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                f[2 * e] = bf16_lo(u[e]) + __uint_as_float(v[8 * q + 2 * e]);
                f[2 * e + 1] = bf16_hi(u[e]) + __uint_as_float(v[8 * q + 2 * e + 1]);
              }
              if (col + c0 + 8 * q < d_out)  // d_out is a multiple of 8
                *reinterpret_cast<uint4*>(yrow + col + c0 + 8 * q) = pack8_bf16(f);
            }
          }
        }
      }
      if (!freed) free_acc();  // (a warp without rows, or aborted)
      if (rows && ok) {
        if (mode == kFull) {
          // lane 0 stores the warp's 32 rows; once its store before that has
          // read the buffer, that buffer takes the load of half-tile
          // hj + kYBuf - 1
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && !*abort_f) {
            ptx::tma_store_2d(&tm_y, buf + warp * kYWarp, hcol(hj), row0 + 32 * warp);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read<1>();
            if (hj >= 1 && hj + kYBuf - 1 < n_half) issue_y(warp, hj + kYBuf - 1);
          }
        } else if (hj + kYBuf < n_half) {
          // every row of the warp has been read: its part of the buffer
          // takes half-tile hj + kYBuf
          __syncwarp();
          if (lane == 0) issue_y(warp, hj + kYBuf);
          issue_y_own(hj + kYBuf);
        }
      }
      __syncwarp();
    }
    if (mode == kFull && lane == 0 && rows) ptx::bulk_wait_group_read_all();  // buffers outlive stores
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Lay::kTmemCols);
  }
  if (tid == 0 && *abort_f) flag_error(err, LORA_DEVERR_TIMEOUT);
}

template <int R>
cudaError_t launch_expand_r(const CUtensorMap& tm, const CUtensorMap& tm_y, const float* vpart,
                            int ksplit, const int32_t* perm, const int32_t* seg_slot,
                            const int32_t* seg_off, const int32_t* n_seg, bf16* y, int T,
                            int d_out, int n_slots, uint32_t* err, cudaStream_t st,
                            const DeviceInfo& dev) {
  using Lay = ExpandLayout<R>;
  // at least 80 KB, so that at most two CTAs share an SM and their 2 x 256
  // tensor-memory columns fit
  size_t smem = Lay::kTotal + 1024;
  if (smem < 80 * 1024) smem = 80 * 1024;
  if (smem > dev.max_smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = sgmv_expand_tc_kernel<R>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int cap = T < n_slots ? T : n_slots;
  const int items = (T + kTok - 1) / kTok + cap;
  const int groups = ((d_out + kXN - 1) / kXN + kXGroup - 1) / kXGroup;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items > 0 ? items : 1, groups);
  cfg.blockDim = dim3(kXThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, tm, tm_y, vpart, ksplit, perm, seg_slot, seg_off, n_seg,
                            y, T, d_out, err);
}

}  // namespace

bool sgmv_shrink_tc_supported(int r) { return r == 64 || r == 128; }

int sgmv_shrink_tc_items(int T, int n_slots) {
  // the chunks of 128 tokens, plus at most one more per segment
  const int cap = T < n_slots ? T : n_slots;
  return (T + kTok - 1) / kTok + cap;
}

int fold_shrink_ksplit(int T, int d_in, int n_slots, int num_sms) {
  // about three CTAs per SM (the ring the shrink takes above two per SM),
  // expected real items ~ chunks + half the segment bound; at most four
  // splits, which the fold loads in one round trip
  const int cap = T < n_slots ? T : n_slots;
  const int est = (T + kTok - 1) / kTok + (cap + 1) / 2;
  int ks = (3 * num_sms + est - 1) / (est > 0 ? est : 1);
  const int kmax = d_in / 128 > 0 ? d_in / 128 : 1;
  if (ks > 4) ks = 4;
  if (ks > kmax) ks = kmax;
  if (ks < 1) ks = 1;
  return ks;
}
bool sgmv_expand_tc_supported(int r) { return r == 64 || r == 128; }

cudaError_t launch_sgmv_expand_tc(const float* vpart, int ksplit, const void* B,
                                  const int32_t* perm, const int32_t* seg_slot,
                                  const int32_t* seg_off, const int32_t* n_seg, void* y, int T,
                                  int r, int d_out, int n_slots, uint32_t* err, cudaStream_t st,
                                  const DeviceInfo& dev) {
  if (T <= 0) return cudaSuccess;
  CUtensorMap tm, tm_y;
  // B_pool as [n_slots][r][d_out]: 64 columns x r rows per box; y [T][d_out]:
  // 64 columns x 32 rows (one epilogue warp's rows) per box, 128-byte swizzle
  if (!encode_tensor_map_bf16_3d(&tm, B, d_out, r, n_slots, 64, r) ||
      !encode_tensor_map_bf16(&tm_y, y, d_out, T, d_out, 64, 32))
    return cudaErrorInvalidValue;
  bf16* ye = static_cast<bf16*>(y);
  if (r == 64)
    return launch_expand_r<64>(tm, tm_y, vpart, ksplit, perm, seg_slot, seg_off, n_seg, ye, T,
                               d_out, n_slots, err, st, dev);
  if (r == 128)
    return launch_expand_r<128>(tm, tm_y, vpart, ksplit, perm, seg_slot, seg_off, n_seg, ye, T,
                                d_out, n_slots, err, st, dev);
  return cudaErrorInvalidValue;
}

cudaError_t launch_sgmv_shrink_tc(const void* x, const void* A, const int32_t* perm,
                                  const int32_t* seg_slot, const int32_t* seg_off,
                                  const int32_t* n_seg, const float* scale, float* vpart, int T,
                                  int d_in, int r, int n_slots, int ksplit, int32_t* fold,
                                  uint32_t* err, cudaStream_t st, bool pdl,
                                  const DeviceInfo& dev) {
  if (T <= 0) return cudaSuccess;
  CUtensorMap tm, tm_x;
  // A_pool as [n_slots][d_in][r]: 64 columns x 64 K rows per box; rows past
  // d_in read as zero.  x: 64 columns x 128 rows per box
  if (!encode_tensor_map_bf16_3d(&tm, A, r, d_in, n_slots, 64, 64) ||
      !encode_tensor_map_bf16(&tm_x, x, d_in, T, d_in, 64, kTok))
    return cudaErrorInvalidValue;
  const bf16* xe = static_cast<const bf16*>(x);
  // more than one wave at two CTAs per SM: the shallower ring, three per SM
  // (prefill workload: 33.3 -> 29.2 us at split 4, 35.7 -> 32.1 us at split
  // 8; at split 2, one wave, the deeper ring stays ahead: 38.0 against 38.7)
  const int cap = T < n_slots ? T : n_slots;
  const long long ctas = static_cast<long long>((T + kTok - 1) / kTok + cap) * ksplit;
  const bool wide = ctas > 2ll * dev.num_sms;
  if (r == 64 && wide)
    return launch_r<64, 3>(tm, tm_x, xe, perm, seg_slot, seg_off, n_seg, scale, vpart, T, d_in,
                           n_slots, ksplit, fold, err, st, pdl, dev);
  if (r == 64)
    return launch_r<64, 4>(tm, tm_x, xe, perm, seg_slot, seg_off, n_seg, scale, vpart, T, d_in,
                           n_slots, ksplit, fold, err, st, pdl, dev);
  if (r == 128)
    return launch_r<128, 3>(tm, tm_x, xe, perm, seg_slot, seg_off, n_seg, scale, vpart, T, d_in,
                            n_slots, ksplit, fold, err, st, pdl, dev);
  return cudaErrorInvalidValue;
}

}  // namespace lora
