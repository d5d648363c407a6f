// The whole layer for fp32 storage on CUDA cores: y = x W0 + v B_a, where
// v is the (already scaled) shrink output given as split partial sums.
// fp32 storage exists for small checks (the toy mixed batch of "Serving
// multiple LoRAs: segmented matrix multiplies and adapter scheduling" is
// fp32); bf16 layers go through the tensor-core kernel in k_fused_tc.cu.
#include "common.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kBM = 32, kBN = 64, kBK = 32;

__global__ void __launch_bounds__(256)
    fused_f32_kernel(const float* __restrict__ x, const float* __restrict__ W0,
                     const float* __restrict__ B, const int32_t* __restrict__ ids,
                     const float* vpart, int v_ksplit, float* __restrict__ y, int T,
                     int d_in, int d_out, int r, int n_slots, uint32_t* err) {
  __shared__ float xs[kBM][kBK + 1];
  __shared__ float ws[kBK][kBN];
  pdl_wait();
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  for (int k0 = 0; k0 < d_in; k0 += kBK) {
    for (int e = tid; e < kBM * kBK; e += 256) {
      const int i = e / kBK, k = e % kBK;
      xs[i][k] = (m0 + i < T && k0 + k < d_in) ? x[static_cast<size_t>(m0 + i) * d_in + k0 + k] : 0.f;
    }
    for (int e = tid; e < kBK * kBN; e += 256) {
      const int k = e / kBN, n = e % kBN;
      ws[k][n] = (k0 + k < d_in && n0 + n < d_out) ? W0[static_cast<size_t>(k0 + k) * d_out + n0 + n] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < kBK; ++k) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float xv = xs[ty * 2 + i][k];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv, ws[k][tx * 4 + j], acc[i][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = m0 + ty * 2 + i;
    if (t >= T) continue;
    const int id = ids[t];
    if (slot_valid(id, n_slots)) {
      for (int q = 0; q < r; ++q) {
        float vq = 0.f;
        for (int s = 0; s < v_ksplit; ++s) {
          const float* vp = vpart + (static_cast<size_t>(s) * T + t) * r + q;
          float v;
          asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(vp) : "memory");
          vq += v;
        }
        const float* Bq = B + (static_cast<size_t>(id) * r + q) * d_out;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx * 4 + j;
          if (n < d_out) acc[i][j] = fmaf(vq, Bq[n], acc[i][j]);
        }
      }
    } else if (id != -1 && blockIdx.x == 0 && tx == 0) {
      flag_error(err, LORA_DEVERR_BAD_SLOT);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < d_out) y[static_cast<size_t>(t) * d_out + n] = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_fused_f32(const float* x, const float* W0, const float* B, const int32_t* ids,
                             const float* vpart, int v_ksplit, float* y, int T, int d_in,
                             int d_out, int r, int n_slots, uint32_t* err, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((d_out + kBN - 1) / kBN, (T + kBM - 1) / kBM);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_f32_kernel, x, W0, B, ids, vpart, v_ksplit, y, T, d_in,
                            d_out, r, n_slots, err);
}

}  // namespace lora
