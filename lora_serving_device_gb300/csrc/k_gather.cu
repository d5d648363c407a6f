// Shrink and expand kernels on CUDA cores.
//
// BGMV ("Serving multiple LoRAs: segmented matrix multiplies and adapter
// scheduling", BGMV bullet): every token gathers its own adapter's A / B by
// index; one CTA per (token, d_in split) for the shrink and per (token,
// 1024-column chunk) for the expand.  Tokens that share an adapter read the
// same A / B lines, which L2 serves after the first read.
//
// SGMV (same page, SGMV bullet; "Serving Many LoRA Adapters", section
// "Punica: The Segmented Gather-Scatter Kernel"): tokens are visited segment
// by segment (the output of the segment builder); one CTA owns a work item =
// (segment, chunk of up to 64 of its tokens) and reads that adapter's A / B
// slice once for all of them, keeping 4 tokens in registers per pass.
//
// Shrink output is fp32 split over d_in into ksplit ranges (deterministic
// partial sums, no atomics): v_partial[s, t, :] = s_a * x[t, K_s] A_a[K_s, :].
// Expand sums the partials on load and adds v B_a into y with one rounding.
// Inside every CTA the d_in range is spread over lanes in 8-element groups
// (16-byte loads of bf16) and folded with warp shuffles.
#include "common.cuh"
#include "internal.h"
#include "sgmv_item.cuh"

namespace lora {
namespace {

constexpr int kSgTokens = 64;   // tokens per SGMV work item

template <int R>
struct RankLayout {
  static constexpr int QC = R / 8;            // 8-wide column chunks of an A row
  static constexpr int KLW = 32 / QC;         // lanes of one warp along d_in
  static_assert(R % 8 == 0 && QC <= 32, "rank");
};

// Sum the 8 accumulators over the lanes of a warp that share a column chunk.
template <int QC>
__device__ __forceinline__ void fold_klanes(float (&acc)[8]) {
#pragma unroll
  for (int o = QC; o < 32; o <<= 1) {
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], o);
  }
}

// ------------------------------------------------------------------- BGMV
template <typename E, int R>
__global__ void __launch_bounds__(128)
    bgmv_shrink_kernel(const E* __restrict__ x, const E* __restrict__ A,
                       const int32_t* __restrict__ ids, const float* __restrict__ scale,
                       float* __restrict__ vpart, int T, int d_in, int n_slots, int kchunk,
                       uint32_t* err) {
  using RL = RankLayout<R>;
  constexpr int KL = 128 / RL::QC;   // lanes of the block along d_in
  __shared__ float red[4][R];
  pdl_launch_dependents();  // the base GEMM may start streaming W0 now
  const int t = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
  const int id = ids[t];
  float* out = vpart + (static_cast<size_t>(s) * T + t) * R;
  if (!slot_valid(id, n_slots)) {
    for (int q = tid; q < R; q += 128) out[q] = 0.f;
    if (tid == 0 && s == 0 && id != -1) flag_error(err, LORA_DEVERR_BAD_SLOT);
    return;
  }
  const int qc = tid % RL::QC, kl = tid / RL::QC;
  const int k0 = s * kchunk, k1 = min(d_in, k0 + kchunk);
  const E* Aa = A + static_cast<size_t>(id) * d_in * R + qc * 8;
  const E* xt = x + static_cast<size_t>(t) * d_in;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int k = k0 + kl * 8; k < k1; k += KL * 8) {
    float xv[8];
    load8(xt + k, xv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a[8];
      load8(Aa + static_cast<size_t>(k + j) * R, a);
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = fmaf(xv[j], a[c], acc[c]);
    }
  }
  fold_klanes<RL::QC>(acc);
  const int warp = tid >> 5, lane = tid & 31;
  if (lane < RL::QC) {
#pragma unroll
    for (int c = 0; c < 8; ++c) red[warp][lane * 8 + c] = acc[c];
  }
  __syncthreads();
  const float sc = scale ? scale[id] : 1.f;
  for (int q = tid; q < R; q += 128) out[q] = (red[0][q] + red[1][q] + red[2][q] + red[3][q]) * sc;
}

template <typename E, int R>
__global__ void __launch_bounds__(128)
    bgmv_expand_kernel(const float* __restrict__ vpart, int ksplit, const E* __restrict__ B,
                       const int32_t* __restrict__ ids, E* __restrict__ y, int T, int d_out,
                       int n_slots, uint32_t* err) {
  __shared__ float vs[R];
  const int t = blockIdx.x;
  const int id = ids[t];
  if (!slot_valid(id, n_slots)) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && id != -1) flag_error(err, LORA_DEVERR_BAD_SLOT);
    return;
  }
  for (int q = threadIdx.x; q < R; q += 128) {
    float a = 0.f;
    for (int s = 0; s < ksplit; ++s) a += vpart[(static_cast<size_t>(s) * T + t) * R + q];
    vs[q] = a;
  }
  __syncthreads();
  const int n = (blockIdx.y * 128 + threadIdx.x) * 8;
  if (n >= d_out) return;
  const E* Bp = B + static_cast<size_t>(id) * R * d_out + n;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int q = 0; q < R; ++q) {
    float b[8];
    load8(Bp + static_cast<size_t>(q) * d_out, b);
    const float vq = vs[q];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = fmaf(vq, b[c], acc[c]);
  }
  E* yp = y + static_cast<size_t>(t) * d_out + n;
  float yv[8];
  load8(yp, yv);
#pragma unroll
  for (int c = 0; c < 8; ++c) yv[c] += acc[c];
  store8(yp, yv);
}

// BGMV expand into an fp32 adapter term, delta[t, :] = v[t, :] B[a_t], for
// the fused decode path: it runs while the base GEMM streams W0 (launched as
// a programmatic dependent of the shrink, and itself letting the GEMM start)
// and the GEMM adds it in its epilogue.  Rows of base-only tokens are not
// written.  One CTA per (token, 1024 columns).
template <int R>
__global__ void __launch_bounds__(128)
    bgmv_delta_kernel(const float* vpart, int ksplit, const bf16* __restrict__ B,
                      const int32_t* __restrict__ ids, float* __restrict__ delta, int T,
                      int d_out, int n_slots, uint32_t* err) {
  constexpr int kGroups = 128 / R;  // threads summing the partials of one column q
  __shared__ float part[128];
  __shared__ float vs[R];
  pdl_launch_dependents();
  // every CTA waits, so that this grid completing implies the shrink completed
  pdl_wait();  // v is written by the shrink kernel launched just before
  const int t = blockIdx.x;
  const int id = ids[t];
  if (!slot_valid(id, n_slots)) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && id != -1) flag_error(err, LORA_DEVERR_BAD_SLOT);
    return;
  }
  const int n = (blockIdx.y * 128 + threadIdx.x) * 8;
  const bool on = n < d_out;
  const bf16* Bp = B + static_cast<size_t>(id) * R * d_out + (on ? n : 0);
  // the first batch of B rows (independent of v) is loaded before the v sum
  // so the two latencies overlap; B stays packed bf16 until the FMA
  constexpr int kBatch = R < 32 ? R : 32;
  uint4 braw[kBatch];
  if (on) {
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      braw[j] = *reinterpret_cast<const uint4*>(Bp + static_cast<size_t>(j) * d_out);
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  {
    const int q = threadIdx.x % R, g = threadIdx.x / R;
    float a = 0.f;
    for (int s = g; s < ksplit; s += kGroups) {
      const float* vp = vpart + (static_cast<size_t>(s) * T + t) * R + q;
      float v;
      asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(vp) : "memory");
      a += v;
    }
    part[threadIdx.x] = a;
  }
  __syncthreads();
  if (threadIdx.x < R) {
    float a = 0.f;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) a += part[g * R + threadIdx.x];
    vs[threadIdx.x] = a;
  }
  __syncthreads();
  if (!on) return;
#pragma unroll 1
  for (int q0 = 0; q0 < R; q0 += kBatch) {
    if (q0 > 0) {
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        braw[j] = *reinterpret_cast<const uint4*>(Bp + static_cast<size_t>(q0 + j) * d_out);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float vq = vs[q0 + j];
      const uint32_t w4[4] = {braw[j].x, braw[j].y, braw[j].z, braw[j].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[2 * c] = fmaf(vq, bf16_lo(w4[c]), acc[2 * c]);
        acc[2 * c + 1] = fmaf(vq, bf16_hi(w4[c]), acc[2 * c + 1]);
      }
    }
  }
  store8(delta + static_cast<size_t>(t) * d_out + n, acc);
}

// ------------------------------------------------------------------- SGMV

template <typename E, int R>
__global__ void __launch_bounds__(256)
    sgmv_shrink_kernel(const E* __restrict__ x, const E* __restrict__ A, const int32_t* perm,
                       const int32_t* seg_slot, const int32_t* seg_off, const int32_t* n_seg,
                       const float* __restrict__ scale, float* __restrict__ vpart, int T,
                       int d_in, int n_slots, int kchunk, uint32_t* err) {
  using RL = RankLayout<R>;
  __shared__ int s_a, s_p0, s_p1;
  pdl_launch_dependents();  // the base GEMM may start streaming W0 now
  pdl_wait();               // the segments are written by the previous kernel
  const int tid = threadIdx.x, s = blockIdx.y;
  const int nseg = ld_dep(n_seg);
  if (blockIdx.x == 0) {    // rows of base-only tokens are zero
    const int nbase = ld_dep(seg_off);
    for (int e = tid; e < nbase * R; e += 256)
      vpart[(static_cast<size_t>(s) * T + perm_row(perm, e / R, T, err)) * R + (e % R)] = 0.f;
  }
  sgmv_item<kSgTokens>(blockIdx.x, seg_slot, seg_off, nseg, &s_a, &s_p0, &s_p1);
  if (s_a < 0) return;
  const int a = checked_index(s_a, n_slots, err);
  const int p0 = s_p0, p1 = s_p1;
  const int warp = tid >> 5, lane = tid & 31;
  const int qc = lane % RL::QC, kl = lane / RL::QC;
  const int k0 = s * kchunk, k1 = min(d_in, k0 + kchunk);
  const E* Aa = A + static_cast<size_t>(a) * d_in * R + qc * 8;
  const float sc = scale ? scale[a] : 1.f;
  for (int pb = p0 + warp * 4; pb < p1; pb += 32) {
    const int nt = min(4, p1 - pb);
    int tok[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) tok[u] = perm_row(perm, pb + ((u < nt) ? u : 0), T, err);
    float acc[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[u][c] = 0.f;
    for (int k = k0 + kl * 8; k < k1; k += RL::KLW * 8) {
      float xv[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) load8(x + static_cast<size_t>(tok[u]) * d_in + k, xv[u]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float av[8];
        load8(Aa + static_cast<size_t>(k + j) * R, av);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[u][c] = fmaf(xv[u][j], av[c], acc[u][c]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) fold_klanes<RL::QC>(acc[u]);
    if (kl == 0) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (u < nt) {
          float* o = vpart + (static_cast<size_t>(s) * T + tok[u]) * R + qc * 8;
          float f[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) f[c] = acc[u][c] * sc;
          store8(o, f);
        }
      }
    }
  }
}

template <typename E, int R>
__global__ void __launch_bounds__(256)
    sgmv_expand_kernel(const float* __restrict__ vpart, int ksplit, const E* __restrict__ B,
                       const int32_t* perm, const int32_t* seg_slot, const int32_t* seg_off,
                       const int32_t* n_seg, E* __restrict__ y, int T, int d_out, int n_slots,
                       uint32_t* err) {
  __shared__ float vs[kSgTokens][R];
  __shared__ int s_tok[kSgTokens];
  __shared__ int s_a, s_p0, s_p1;
  const int tid = threadIdx.x;
  sgmv_item<kSgTokens>(blockIdx.x, seg_slot, seg_off, ld_dep(n_seg), &s_a, &s_p0, &s_p1);
  if (s_a < 0) return;
  const int a = checked_index(s_a, n_slots, err);
  const int p0 = s_p0, L = s_p1 - s_p0;
  for (int e = tid; e < L * R; e += 256) {
    const int i = e / R, q = e % R;
    const int t = perm_row(perm, p0 + i, T, err);
    float acc = 0.f;
    for (int s = 0; s < ksplit; ++s) acc += vpart[(static_cast<size_t>(s) * T + t) * R + q];
    vs[i][q] = acc;
    if (q == 0) s_tok[i] = t;
  }
  __syncthreads();
  const int n = (blockIdx.y * 256 + tid) * 8;
  if (n >= d_out) return;
  const E* Bp = B + static_cast<size_t>(a) * R * d_out + n;
  for (int i0 = 0; i0 < L; i0 += 4) {
    float acc[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[u][c] = 0.f;
#pragma unroll 2
    for (int q = 0; q < R; ++q) {
      float b[8];
      load8(Bp + static_cast<size_t>(q) * d_out, b);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float vq = (i0 + u < L) ? vs[i0 + u][q] : 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[u][c] = fmaf(vq, b[c], acc[u][c]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (i0 + u < L) {
        E* yp = y + static_cast<size_t>(s_tok[i0 + u]) * d_out + n;
        float yv[8];
        load8(yp, yv);
#pragma unroll
        for (int c = 0; c < 8; ++c) yv[c] += acc[u][c];
        store8(yp, yv);
      }
    }
  }
}

int kchunk_for(int d_in, int ksplit) {
  const int per = (d_in + ksplit - 1) / ksplit;
  return (per + 7) / 8 * 8;
}

template <typename E>
cudaError_t bgmv_shrink_t(const void* x, const void* A, const int32_t* ids, const float* scale,
                          float* vpart, int T, int d_in, int r, int n_slots, int ksplit,
                          uint32_t* err, cudaStream_t st) {
  const dim3 grid(T, ksplit);
  const int kc = kchunk_for(d_in, ksplit);
  const E* xe = static_cast<const E*>(x);
  const E* Ae = static_cast<const E*>(A);
  switch (r) {
    case 8: bgmv_shrink_kernel<E, 8><<<grid, 128, 0, st>>>(xe, Ae, ids, scale, vpart, T, d_in, n_slots, kc, err); break;
    case 16: bgmv_shrink_kernel<E, 16><<<grid, 128, 0, st>>>(xe, Ae, ids, scale, vpart, T, d_in, n_slots, kc, err); break;
    case 32: bgmv_shrink_kernel<E, 32><<<grid, 128, 0, st>>>(xe, Ae, ids, scale, vpart, T, d_in, n_slots, kc, err); break;
    case 64: bgmv_shrink_kernel<E, 64><<<grid, 128, 0, st>>>(xe, Ae, ids, scale, vpart, T, d_in, n_slots, kc, err); break;
    case 128: bgmv_shrink_kernel<E, 128><<<grid, 128, 0, st>>>(xe, Ae, ids, scale, vpart, T, d_in, n_slots, kc, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename E>
cudaError_t bgmv_expand_t(const float* vpart, int ksplit, const void* B, const int32_t* ids,
                          void* y, int T, int r, int d_out, int n_slots, uint32_t* err,
                          cudaStream_t st) {
  const dim3 grid(T, (d_out + 1023) / 1024);
  const E* Be = static_cast<const E*>(B);
  E* ye = static_cast<E*>(y);
  switch (r) {
    case 8: bgmv_expand_kernel<E, 8><<<grid, 128, 0, st>>>(vpart, ksplit, Be, ids, ye, T, d_out, n_slots, err); break;
    case 16: bgmv_expand_kernel<E, 16><<<grid, 128, 0, st>>>(vpart, ksplit, Be, ids, ye, T, d_out, n_slots, err); break;
    case 32: bgmv_expand_kernel<E, 32><<<grid, 128, 0, st>>>(vpart, ksplit, Be, ids, ye, T, d_out, n_slots, err); break;
    case 64: bgmv_expand_kernel<E, 64><<<grid, 128, 0, st>>>(vpart, ksplit, Be, ids, ye, T, d_out, n_slots, err); break;
    case 128: bgmv_expand_kernel<E, 128><<<grid, 128, 0, st>>>(vpart, ksplit, Be, ids, ye, T, d_out, n_slots, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename K, typename... Args>
cudaError_t launch_maybe_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t st, bool pdl,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename E>
cudaError_t sgmv_shrink_t(const void* x, const void* A, const int32_t* perm,
                          const int32_t* seg_slot, const int32_t* seg_off, const int32_t* n_seg,
                          const float* scale, float* vpart, int T, int d_in, int r, int n_slots,
                          int ksplit, uint32_t* err, cudaStream_t st, bool pdl) {
  const dim3 grid(sgmv_max_items(T, n_slots), ksplit);
  const int kc = kchunk_for(d_in, ksplit);
  const E* xe = static_cast<const E*>(x);
  const E* Ae = static_cast<const E*>(A);
#define LORA_SGMV_SHRINK_CASE(RR)                                                              \
  case RR:                                                                                     \
    return launch_maybe_pdl(sgmv_shrink_kernel<E, RR>, grid, dim3(256), st, pdl, xe, Ae, perm, \
                            seg_slot, seg_off, n_seg, scale, vpart, T, d_in, n_slots, kc, err);
  switch (r) {
    LORA_SGMV_SHRINK_CASE(8)
    LORA_SGMV_SHRINK_CASE(16)
    LORA_SGMV_SHRINK_CASE(32)
    LORA_SGMV_SHRINK_CASE(64)
    LORA_SGMV_SHRINK_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef LORA_SGMV_SHRINK_CASE
}

template <typename E>
cudaError_t sgmv_expand_t(const float* vpart, int ksplit, const void* B, const int32_t* perm,
                          const int32_t* seg_slot, const int32_t* seg_off, const int32_t* n_seg,
                          void* y, int T, int r, int d_out, int n_slots, uint32_t* err,
                          cudaStream_t st) {
  const dim3 grid(sgmv_max_items(T, n_slots), (d_out + 2047) / 2048);
  const E* Be = static_cast<const E*>(B);
  E* ye = static_cast<E*>(y);
  switch (r) {
    case 8: sgmv_expand_kernel<E, 8><<<grid, 256, 0, st>>>(vpart, ksplit, Be, perm, seg_slot, seg_off, n_seg, ye, T, d_out, n_slots, err); break;
    case 16: sgmv_expand_kernel<E, 16><<<grid, 256, 0, st>>>(vpart, ksplit, Be, perm, seg_slot, seg_off, n_seg, ye, T, d_out, n_slots, err); break;
    case 32: sgmv_expand_kernel<E, 32><<<grid, 256, 0, st>>>(vpart, ksplit, Be, perm, seg_slot, seg_off, n_seg, ye, T, d_out, n_slots, err); break;
    case 64: sgmv_expand_kernel<E, 64><<<grid, 256, 0, st>>>(vpart, ksplit, Be, perm, seg_slot, seg_off, n_seg, ye, T, d_out, n_slots, err); break;
    case 128: sgmv_expand_kernel<E, 128><<<grid, 256, 0, st>>>(vpart, ksplit, Be, perm, seg_slot, seg_off, n_seg, ye, T, d_out, n_slots, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

namespace {
__global__ void set_scale_kernel(float* scale, int slot, float s) { scale[slot] = s; }
}  // namespace

cudaError_t launch_set_scale(float* scale, int slot, float s, cudaStream_t st) {
  set_scale_kernel<<<1, 1, 0, st>>>(scale, slot, s);
  return cudaGetLastError();
}

int sgmv_max_items(int T, int n_slots) {
  const int cap = T < n_slots ? T : n_slots;
  const int items = (T + kSgTokens - 1) / kSgTokens + cap;
  return items > 0 ? items : 1;
}

int decode_shrink_ksplit(int T, int d_in) {
  // ~256 CTAs of the per-token shrink, each over at least 512 of d_in
  int ks = (256 + T - 1) / (T > 0 ? T : 1);
  const int kmax = d_in / 512 > 0 ? d_in / 512 : 1;
  if (ks > 16) ks = 16;
  if (ks > kmax) ks = kmax;
  return ks < 1 ? 1 : ks;
}

int fused_shrink_ksplit(int T, int d_in, int n_slots, int num_sms) {
  // enough (work item x split) CTAs to cover the GPU about twice; expected
  // real items ~ chunks + half the segment bound
  const int cap = T < n_slots ? T : n_slots;
  const int est = (T + kSgTokens - 1) / kSgTokens + (cap + 1) / 2;
  int ks = (2 * num_sms + est - 1) / (est > 0 ? est : 1);
  const int kmax = d_in / 128 > 0 ? d_in / 128 : 1;
  if (ks > 16) ks = 16;
  if (ks > kmax) ks = kmax;
  if (ks < 1) ks = 1;
  return ks;
}

cudaError_t launch_bgmv_shrink(const void* x, const void* A, const int32_t* ids,
                               const float* scale, float* vpart, int T, int d_in, int r,
                               int n_slots, int ksplit, lora_dtype_t dt, uint32_t* err,
                               cudaStream_t st) {
  return dt == LORA_DTYPE_BF16
             ? bgmv_shrink_t<bf16>(x, A, ids, scale, vpart, T, d_in, r, n_slots, ksplit, err, st)
             : bgmv_shrink_t<float>(x, A, ids, scale, vpart, T, d_in, r, n_slots, ksplit, err, st);
}

cudaError_t launch_bgmv_expand(const float* vpart, int ksplit, const void* B, const int32_t* ids,
                               void* y, int T, int r, int d_out, int n_slots, lora_dtype_t dt,
                               uint32_t* err, cudaStream_t st) {
  return dt == LORA_DTYPE_BF16
             ? bgmv_expand_t<bf16>(vpart, ksplit, B, ids, y, T, r, d_out, n_slots, err, st)
             : bgmv_expand_t<float>(vpart, ksplit, B, ids, y, T, r, d_out, n_slots, err, st);
}

cudaError_t launch_bgmv_delta(const float* vpart, int ksplit, const void* B, const int32_t* ids,
                              float* delta, int T, int r, int d_out, int n_slots, uint32_t* err,
                              cudaStream_t st, bool pdl) {
  const dim3 grid(T, (d_out + 1023) / 1024);
  const bf16* Be = static_cast<const bf16*>(B);
#define LORA_DELTA_CASE(RR)                                                                   \
  case RR:                                                                                    \
    return launch_maybe_pdl(bgmv_delta_kernel<RR>, grid, dim3(128), st, pdl, vpart, ksplit, Be, \
                            ids, delta, T, d_out, n_slots, err);
  switch (r) {
    LORA_DELTA_CASE(8)
    LORA_DELTA_CASE(16)
    LORA_DELTA_CASE(32)
    LORA_DELTA_CASE(64)
    LORA_DELTA_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef LORA_DELTA_CASE
}

cudaError_t launch_sgmv_shrink(const void* x, const void* A, const int32_t* perm,
                               const int32_t* seg_slot, const int32_t* seg_off,
                               const int32_t* n_seg, const float* scale, float* vpart, int T,
                               int d_in, int r, int n_slots, int ksplit, lora_dtype_t dt,
                               uint32_t* err, cudaStream_t st, bool pdl) {
  return dt == LORA_DTYPE_BF16
             ? sgmv_shrink_t<bf16>(x, A, perm, seg_slot, seg_off, n_seg, scale, vpart, T, d_in,
                                   r, n_slots, ksplit, err, st, pdl)
             : sgmv_shrink_t<float>(x, A, perm, seg_slot, seg_off, n_seg, scale, vpart, T, d_in,
                                    r, n_slots, ksplit, err, st, pdl);
}

cudaError_t launch_sgmv_expand(const float* vpart, int ksplit, const void* B, const int32_t* perm,
                               const int32_t* seg_slot, const int32_t* seg_off,
                               const int32_t* n_seg, void* y, int T, int r, int d_out,
                               int n_slots, lora_dtype_t dt, uint32_t* err, cudaStream_t st) {
  return dt == LORA_DTYPE_BF16
             ? sgmv_expand_t<bf16>(vpart, ksplit, B, perm, seg_slot, seg_off, n_seg, y, T, r,
                                   d_out, n_slots, err, st)
             : sgmv_expand_t<float>(vpart, ksplit, B, perm, seg_slot, seg_off, n_seg, y, T, r,
                                    d_out, n_slots, err, st);
}

}  // namespace lora
