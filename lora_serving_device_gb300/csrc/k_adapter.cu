// The whole adapter term of a decode-sized batch in one launch:
// delta[t, :] = s_a * (x[t, :] A_a) B_a for every token t with a valid
// adapter a = ids[t] ("Serving multiple LoRAs: segmented matrix multiplies
// and adapter scheduling", BGMV bullet: each token gathers its own adapter's
// factors; the shrink to rank r comes first, then the expand).  The fp32
// result is added by the decode base GEMM in its epilogue, so y is stored
// once.
//
// One thread-block cluster of C CTAs per token.  CTA c shrinks the c-th
// slice of d_in (x[t, K_c] A_a[K_c, :], the slice of A_a read once), the C
// rank-r partials are summed through distributed shared memory in a fixed
// order (deterministic, no atomics), and CTA c then expands the c-th slice
// of the d_out columns.  B_a rows for the first columns are requested before
// the shrink, so their latency overlaps it.  Launched first in the decode
// chain, it lets the base GEMM start streaming W0 at once (programmatic
// launch); it uses under 1 KiB of shared memory so its CTAs fit beside a
// base-GEMM CTA on one SM.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int kAdThreads = 256;
constexpr int kAdWarps = kAdThreads / 32;

template <int R>
__global__ void __launch_bounds__(kAdThreads)
    bgmv_adapter_kernel(const bf16* __restrict__ x, const bf16* __restrict__ A,
                        const bf16* __restrict__ B, const int32_t* __restrict__ ids,
                        const float* __restrict__ scale, float* __restrict__ delta, int T,
                        int d_in, int d_out, int n_slots, int kc, int nc, uint32_t* err) {
  constexpr int QC = R / 8;             // 8-wide column chunks of an A row
  constexpr int KL = kAdThreads / QC;   // threads along d_in
  constexpr int H = 2;                  // threads sharing one 8-column group of the expand
  constexpr int RH = R / H;             // B rows per thread
  constexpr int kPre = RH < 8 ? RH : 8; // B rows requested before the shrink
  static_assert(R % 8 == 0 && QC <= 32, "rank");
  __shared__ float red[kAdWarps][R];
  __shared__ float pv[R];  // this CTA's partial, read by the whole cluster
  __shared__ float vs[R];  // the token's full shrink output, scaled

  pdl_launch_dependents();  // the base GEMM may start streaming W0 now
  const int c = static_cast<int>(ptx::cluster_ctarank());
  const int C = static_cast<int>(gridDim.x);
  const int t = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int id = ids[t];
  if (!slot_valid(id, n_slots)) {
    // every CTA of the cluster reads the same id and leaves here together
    if (tid == 0 && c == 0 && id != -1) flag_error(err, LORA_DEVERR_BAD_SLOT);
    return;
  }

  // ---- first B rows of this thread's first column group (independent of v)
  const int h = tid % H;
  const int n_begin = c * nc, n_end = min(d_out, n_begin + nc);
  const bf16* Ba = B + static_cast<size_t>(id) * R * d_out;
  const int g0 = n_begin + (tid / H) * 8;
  uint4 bpre[kPre];
  if (g0 < n_end) {
#pragma unroll
    for (int j = 0; j < kPre; ++j)
      bpre[j] = *reinterpret_cast<const uint4*>(Ba + static_cast<size_t>(h * RH + j) * d_out + g0);
  }

  // ---- shrink of this CTA's d_in slice
  const int qc = tid % QC, kl = tid / QC;
  const int k_begin = c * kc, k_end = min(d_in, k_begin + kc);
  const bf16* Aa = A + static_cast<size_t>(id) * d_in * R + qc * 8;
  const bf16* xt = x + static_cast<size_t>(t) * d_in;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
  for (int k = k_begin + kl * 8; k < k_end; k += KL * 8) {
    float xv[8];
    load8(xt + k, xv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a[8];
      load8(Aa + static_cast<size_t>(k + j) * R, a);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(xv[j], a[q], acc[q]);
    }
  }
  // lanes sharing a column chunk sit QC apart in the warp
#pragma unroll
  for (int o = QC; o < 32; o <<= 1) {
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
  }
  if (lane < QC) {
#pragma unroll
    for (int q = 0; q < 8; ++q) red[warp][lane * 8 + q] = acc[q];
  }
  __syncthreads();
  if (tid < R) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kAdWarps; ++w) a += red[w][tid];
    pv[tid] = a;
  }

  // ---- sum the C partials in rank order; every CTA gets the same v
  ptx::cluster_arrive_release();
  ptx::cluster_wait_acquire();
  if (tid < R) {
    const uint32_t local = ptx::smem_u32(&pv[tid]);
    float a = 0.f;
    for (int src = 0; src < C; ++src) {
      float v;
      asm volatile("ld.shared::cluster.f32 %0, [%1];"
                   : "=f"(v)
                   : "r"(ptx::mapa_shared(local, static_cast<uint32_t>(src))));
      a += v;
    }
    vs[tid] = a * (scale ? scale[id] : 1.f);
  }
  __syncthreads();
  // done reading the peers' partials; a CTA leaves only after every peer is
  ptx::cluster_arrive_relaxed();

  // ---- expand this CTA's columns: thread pair (g, h) covers 8 columns, h
  // takes half of the R rows, and the halves are added with one shuffle.
  // The trip count is the same for every thread (the shuffle needs the
  // whole warp).
  constexpr int kStride = (kAdThreads / H) * 8;
#pragma unroll 1
  for (int base = n_begin; base < n_end; base += kStride) {
    const int g = base + (tid / H) * 8;
    const bool on = g < n_end;
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (on) {
#pragma unroll
      for (int j = 0; j < RH; ++j) {
        const uint4 w = (base == n_begin && j < kPre)
                            ? bpre[j]
                            : *reinterpret_cast<const uint4*>(
                                  Ba + static_cast<size_t>(h * RH + j) * d_out + g);
        const float vq = vs[h * RH + j];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[2 * e] = fmaf(vq, bf16_lo(u[e]), o[2 * e]);
          o[2 * e + 1] = fmaf(vq, bf16_hi(u[e]), o[2 * e + 1]);
        }
      }
    }
    if (H == 2) {
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] += __shfl_xor_sync(0xffffffffu, o[e], 1);
    }
    if (on && h == 0) store8(delta + static_cast<size_t>(t) * d_out + g, o);
  }
  ptx::cluster_wait_acquire();
}

}  // namespace

int adapter_cluster_size(int d_in, int d_out) {
  const int m = d_in < d_out ? d_in : d_out;
  if (m >= 2048) return 4;
  if (m >= 512) return 2;
  return 1;
}

cudaError_t launch_bgmv_adapter(const void* x, const void* A, const void* B, const int32_t* ids,
                                const float* scale, float* delta, int T, int d_in, int d_out,
                                int r, int n_slots, uint32_t* err, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (T > 65535) return cudaErrorInvalidValue;
  const int C = adapter_cluster_size(d_in, d_out);
  const int kc = ((d_in + 8 * C - 1) / (8 * C)) * 8;
  const int nc = ((d_out + 8 * C - 1) / (8 * C)) * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, T);
  cfg.blockDim = dim3(kAdThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bf16* xe = static_cast<const bf16*>(x);
  const bf16* Ae = static_cast<const bf16*>(A);
  const bf16* Be = static_cast<const bf16*>(B);
#define LORA_ADAPTER_CASE(RR)                                                                   \
  case RR:                                                                                      \
    return cudaLaunchKernelEx(&cfg, bgmv_adapter_kernel<RR>, xe, Ae, Be, ids, scale, delta, T, \
                              d_in, d_out, n_slots, kc, nc, err);
  switch (r) {
    LORA_ADAPTER_CASE(8)
    LORA_ADAPTER_CASE(16)
    LORA_ADAPTER_CASE(32)
    LORA_ADAPTER_CASE(64)
    LORA_ADAPTER_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef LORA_ADAPTER_CASE
}

}  // namespace lora
