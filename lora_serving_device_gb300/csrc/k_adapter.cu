// The BGMV adapter term of a decode-sized batch in one launch
// ("Serving multiple LoRAs: segmented matrix multiplies and adapter
// scheduling", BGMV bullet: each token gathers its own adapter's factors;
// the shrink to rank r comes first, then the expand):
//   delta[t, :] = s_a * (x[t, :] A_a) B_a          a = ids[t] valid
// and, in its merge form, the last kernel of the decode layer:
//   y[t, :] = sum_z partial[z, t, :] + delta[t, :]  (delta = 0 for base-only t)
// where partial holds the split-K fp32 base product x W0 of the decode GEMM,
// so y is stored once ("Multi-LoRA batching and adapter paging", section
// "Walking through a batch": the base product once for all rows, then each
// row's adapter term).
//
// One thread-block cluster of C CTAs per token.  CTA c shrinks the c-th
// slice of d_in (x[t, K_c] A_a[K_c, :], the slice of A_a read once), the C
// rank-r partials are summed through distributed shared memory in rank
// order (deterministic, no atomics), and CTA c expands the c-th slice of
// the d_out columns into registers.  B_a rows of the first columns are
// requested before the shrink, so their latency overlaps it.
//
// The merge form is launched as a programmatic dependent of the decode GEMM:
// it starts while the GEMM still streams W0 (its CTAs need little shared
// memory and fit beside a GEMM CTA), computes the adapter term, and only
// then waits for the GEMM grid and reads its partials.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int kAdThreads = 256;
constexpr int kAdWarps = kAdThreads / 32;
constexpr int kPairs = kAdThreads / 2;     // thread pairs along the columns
constexpr int kGroupCols = 8;              // columns of one thread pair
constexpr int kStride = kPairs * kGroupCols;
constexpr int kKeepGroups = 2;             // column groups held across the wait

template <int R>
struct AdapterShape {
  static constexpr int QC = R / 8;             // 8-wide column chunks of an A row
  static constexpr int KL = kAdThreads / QC;   // threads along d_in
  static constexpr int RH = R / 2;             // B rows per thread of a pair
  static constexpr int kPre = RH < 8 ? RH : 8; // B rows requested before the shrink
  static_assert(R % 8 == 0 && QC <= 32, "rank");
};

// Adapter term of the 8 columns [g, g+8) for thread h of the pair: thread h
// takes B rows [h*R/2, (h+1)*R/2), the halves are added with one shuffle, so
// both threads of the pair end with all 8 values.  Every thread of the warp
// must call it (the shuffle); `on` says whether g is inside the slice.  With
// PRE the first rows come from `pre` (loaded earlier) instead of memory.
template <int R, bool PRE>
__device__ __forceinline__ void expand_group(const bf16* Ba, const float* vs, int d_out, int g,
                                             int h, bool on,
                                             const uint4 (&pre)[AdapterShape<R>::kPre],
                                             float (&o)[8]) {
  using SH = AdapterShape<R>;
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
  if (on) {
#pragma unroll
    for (int j = 0; j < SH::RH; ++j) {
      const int row = h * SH::RH + j;
      const uint4 w = (PRE && j < SH::kPre)
                          ? pre[j < SH::kPre ? j : 0]
                          : *reinterpret_cast<const uint4*>(Ba + static_cast<size_t>(row) * d_out + g);
      const float vq = vs[row];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[2 * e] = fmaf(vq, bf16_lo(u[e]), o[2 * e]);
        o[2 * e + 1] = fmaf(vq, bf16_hi(u[e]), o[2 * e + 1]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] += __shfl_xor_sync(0xffffffffu, o[e], 1);
}

// Output of one column group: thread h of the pair owns columns
// [g + 4h, g + 4h + 4).  Delta form: the fp32 adapter term.  Merge form: the
// S partials of the base product (written by the grid this one waited for)
// plus the adapter term, rounded once to bf16.
template <bool MERGE>
__device__ __forceinline__ void store_group(const float (&o)[8], int g, int h, int t, int d_out,
                                            const float* partial, int S, int T, void* out) {
  const int n = g + 4 * h;
  // (selects, not o[4 * h + k]: a runtime index would put o in local memory)
  float f[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) f[k] = h ? o[4 + k] : o[k];
  if (MERGE) {
    // the partials' loads go out together, then they are added in split order
    constexpr int kBatch = 8;
    for (int z0 = 0; z0 < S; z0 += kBatch) {
      float4 pz[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (z0 + u < S) pz[u] = ld_dep_f4(partial + (static_cast<size_t>(z0 + u) * T + t) * d_out + n);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (z0 + u < S) {
          f[0] += pz[u].x;
          f[1] += pz[u].y;
          f[2] += pz[u].z;
          f[3] += pz[u].w;
        }
      }
    }
    uint2 pk;
    pk.x = pack_bf16x2(f[0], f[1]);
    pk.y = pack_bf16x2(f[2], f[3]);
    *reinterpret_cast<uint2*>(static_cast<bf16*>(out) + static_cast<size_t>(t) * d_out + n) = pk;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + static_cast<size_t>(t) * d_out + n) =
        make_float4(f[0], f[1], f[2], f[3]);
  }
}

// Shared-memory scratch of one CTA, sized for the largest rank it serves.
template <int RM>
struct AdapterSmem {
  float red[kAdWarps * RM];  // per-warp column sums of the shrink
  float pv[RM];              // this CTA's partial, read by the whole cluster
  float vs[RM];              // the token's full shrink output, scaled
};

// One token's adapter term at rank R (the whole cluster runs the same R:
// every CTA reads the same id).  Aa / Ba point at the token's A [d_in, R]
// and B [R, d_out] (row-major), `s` is its scale.  `valid` false: base-only
// row (merge form: partials only).  Every CTA of the cluster takes the same
// branches.
template <int R, bool MERGE, int RM>
__device__ __forceinline__ void adapter_token(const bf16* __restrict__ x, const bf16* Aa,
                                              const bf16* Ba, float s, bool valid,
                                              const float* partial, int S, void* out, int T,
                                              int d_in, int d_out, int kc, int nc,
                                              AdapterSmem<RM>& sm) {
  using SH = AdapterShape<R>;
  const int c = static_cast<int>(ptx::cluster_ctarank());
  const int C = static_cast<int>(gridDim.x);
  const int t = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = tid & 1, pair = tid >> 1;
  const int n_begin = c * nc, n_end = min(d_out, n_begin + nc);
  float keep[kKeepGroups][8];
#pragma unroll
  for (int i = 0; i < kKeepGroups; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) keep[i][e] = 0.f;

  if (valid) {
    // ---- first B rows of this thread's first column group (independent of v)
    const int g0 = n_begin + pair * kGroupCols;
    uint4 bpre[SH::kPre];
    if (g0 < n_end) {
#pragma unroll
      for (int j = 0; j < SH::kPre; ++j)
        bpre[j] = *reinterpret_cast<const uint4*>(Ba + static_cast<size_t>(h * SH::RH + j) * d_out + g0);
    }

    // ---- shrink of this CTA's d_in slice
    const int qc = tid % SH::QC, kl = tid / SH::QC;
    const int k_begin = c * kc, k_end = min(d_in, k_begin + kc);
    const bf16* Ac = Aa + qc * 8;
    const bf16* xt = x + static_cast<size_t>(t) * d_in;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int k = k_begin + kl * 8; k < k_end; k += SH::KL * 8) {
      float xv[8];
      load8(xt + k, xv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float a[8];
        load8(Ac + static_cast<size_t>(k + j) * R, a);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(xv[j], a[q], acc[q]);
      }
    }
    // lanes sharing a column chunk sit QC apart in the warp
#pragma unroll
    for (int o = SH::QC; o < 32; o <<= 1) {
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
    }
    if (lane < SH::QC) {
#pragma unroll
      for (int q = 0; q < 8; ++q) sm.red[warp * R + lane * 8 + q] = acc[q];
    }
    __syncthreads();
    if (tid < R) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kAdWarps; ++w) a += sm.red[w * R + tid];
      sm.pv[tid] = a;
    }

    // ---- sum the C partials in rank order; every CTA gets the same v
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
    if (tid < R) {
      // the C remote reads go out together, then they are added in rank order
      const uint32_t local = ptx::smem_u32(&sm.pv[tid]);
      float pr[8];
#pragma unroll
      for (int src = 0; src < 8; ++src) {
        if (src < C)
          asm volatile("ld.shared::cluster.f32 %0, [%1];"
                       : "=f"(pr[src])
                       : "r"(ptx::mapa_shared(local, static_cast<uint32_t>(src))));
      }
      float a = 0.f;
#pragma unroll
      for (int src = 0; src < 8; ++src)
        if (src < C) a += pr[src];
      sm.vs[tid] = a * s;
    }
    __syncthreads();
    // done reading the peers' partials; a CTA leaves only after every peer is
    ptx::cluster_arrive_relaxed();

    // ---- expand the first column groups into registers
    if (n_begin < n_end)  // uniform over the CTA
      expand_group<R, true>(Ba, sm.vs, d_out, g0, h, g0 < n_end, bpre, keep[0]);
#pragma unroll
    for (int i = 1; i < kKeepGroups; ++i) {
      const int base = n_begin + i * kStride;
      if (base < n_end) {  // uniform over the CTA
        const int g = base + pair * kGroupCols;
        expand_group<R, false>(Ba, sm.vs, d_out, g, h, g < n_end, bpre, keep[i]);
      }
    }
  }

  // ---- outputs.  Merge form: wait for the decode GEMM (its partials)
  if (MERGE) pdl_wait();
#pragma unroll
  for (int i = 0; i < kKeepGroups; ++i) {
    const int g = n_begin + i * kStride + pair * kGroupCols;
    if (g < n_end) store_group<MERGE>(keep[i], g, h, t, d_out, partial, S, T, out);
  }
  // columns beyond the kept groups (slices wider than kKeepGroups * kStride)
#pragma unroll 1
  for (int base = n_begin + kKeepGroups * kStride; base < n_end; base += kStride) {
    const int g = base + pair * kGroupCols;
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid) {
      uint4 none[AdapterShape<R>::kPre];  // not read: PRE is false
      expand_group<R, false>(Ba, sm.vs, d_out, g, h, g < n_end, none, o);
    }
    if (g < n_end) store_group<MERGE>(o, g, h, t, d_out, partial, S, T, out);
  }
  if (valid) ptx::cluster_wait_acquire();
}

// Padded pool: A [n_slots, d_in, R], B [n_slots, R, d_out].  MINB is the
// resident-CTA count the registers are budgeted for: 4 (64 registers, so
// three CTAs fit beside a decode-GEMM CTA) or 3 (80 registers).  Ranks 64
// and 128 always take 80: at 64 they spill and run slower.
template <int R, bool MERGE, int MINB>
__global__ void __launch_bounds__(kAdThreads, MINB)
    bgmv_adapter_kernel(const bf16* __restrict__ x, const bf16* __restrict__ A,
                        const bf16* __restrict__ B, const int32_t* __restrict__ ids,
                        const float* __restrict__ scale, const float* partial, int S,
                        void* out, int T, int d_in, int d_out, int n_slots, int kc, int nc,
                        uint32_t* err) {
  __shared__ AdapterSmem<R> sm;
  pdl_launch_dependents();
  const int c = static_cast<int>(ptx::cluster_ctarank());
  const int id = ids[blockIdx.y];
  // every CTA of the cluster reads the same id, so `valid` and everything it
  // guards (the cluster barriers included) is uniform over the cluster
  const bool valid = slot_valid(id, n_slots);
  if (!valid && id != -1 && threadIdx.x == 0 && c == 0) flag_error(err, LORA_DEVERR_BAD_SLOT);
  if (!MERGE && !valid) return;  // delta form: base-only rows are not written
  const int a = valid ? id : 0;
  adapter_token<R, MERGE, R>(x, A + static_cast<size_t>(a) * d_in * R,
                             B + static_cast<size_t>(a) * R * d_out,
                             valid && scale ? scale[id] : 1.f, valid, partial, S, out, T, d_in,
                             d_out, kc, nc, sm);
}

// Ragged pool: slot a holds A_a [d_in, rank[a]] at A + a_off[a] and B_a
// [rank[a], d_out] at B + b_off[a] (elements), rank[a] in {8, 16, 32, 64,
// 128}.  Each token runs the body of its own adapter's rank, so a rank-8
// adapter costs a rank-8 pass, not one at the pool's largest rank.  (Ranks
// between these are stored zero-padded to the next one: per-row rank checks
// inside the body would cost registers and load batching.)  Compiled for 64
// registers: the rank-64 and -128 bodies spill a little, but more resident
// CTAs pay for it on the mixed-rank pools measured.
template <bool MERGE>
__global__ void __launch_bounds__(kAdThreads, 4)
    bgmv_adapter_ragged_kernel(const bf16* __restrict__ x, const bf16* __restrict__ A,
                               const bf16* __restrict__ B, const int64_t* __restrict__ a_off,
                               const int64_t* __restrict__ b_off,
                               const int32_t* __restrict__ rank, int64_t a_elems,
                               int64_t b_elems, int r_max, const int32_t* __restrict__ ids,
                               const float* __restrict__ scale, const float* partial, int S,
                               void* out, int T, int d_in, int d_out, int n_slots, int kc,
                               int nc, uint32_t* err) {
  __shared__ AdapterSmem<128> sm;
  pdl_launch_dependents();
  const int c = static_cast<int>(ptx::cluster_ctarank());
  const int id = ids[blockIdx.y];
  const bool first = threadIdx.x == 0 && c == 0;
  bool valid = slot_valid(id, n_slots);
  if (!valid && id != -1 && first) flag_error(err, LORA_DEVERR_BAD_SLOT);
  int ra = 0;
  int64_t ao = 0, bo = 0;
  if (valid) {
    // the slot's table entry; one that would read outside the pools or break
    // the 16-byte alignment of the rows is flagged and the row is base-only
    ra = rank[id];
    ao = a_off[id];
    bo = b_off[id];
    const bool ok = (ra == 8 || ra == 16 || ra == 32 || ra == 64 || ra == 128) &&
                    ra <= r_max && ao >= 0 && bo >= 0 &&
                    ao % 8 == 0 && bo % 8 == 0 &&
                    ao <= a_elems - static_cast<int64_t>(d_in) * ra &&
                    bo <= b_elems - static_cast<int64_t>(ra) * d_out;
    if (!ok) {
      if (first) flag_error(err, LORA_DEVERR_BAD_RANK);
      valid = false;
    }
  }
  if (!MERGE && !valid) return;
  const bf16* Aa = A + ao;
  const bf16* Ba = B + bo;
  const float s = valid && scale ? scale[id] : 1.f;
#define LORA_RAGGED_CLASS(RR)                                                                  \
  adapter_token<RR, MERGE, 128>(x, Aa, Ba, s, valid, partial, S, out, T, d_in, d_out, kc, nc, sm)
  // uniform over the cluster: every CTA read the same table entry
  if (!valid || ra == 8) LORA_RAGGED_CLASS(8);
  else if (ra == 16) LORA_RAGGED_CLASS(16);
  else if (ra == 32) LORA_RAGGED_CLASS(32);
  else if (ra == 64) LORA_RAGGED_CLASS(64);
  else LORA_RAGGED_CLASS(128);
#undef LORA_RAGGED_CLASS
}

struct AdapterLaunch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  int kc, nc;
};

// One cluster of C CTAs per token, C = adapter_cluster_size(T, d_in, d_out, ragged).
void adapter_launch_config(AdapterLaunch& L, int T, int d_in, int d_out, bool ragged, bool pdl,
                           cudaStream_t st) {
  const int C = adapter_cluster_size(T, d_in, d_out, ragged);
  L.kc = ((d_in + 8 * C - 1) / (8 * C)) * 8;
  L.nc = ((d_out + 8 * C - 1) / (8 * C)) * 8;
  L.cfg = cudaLaunchConfig_t{};
  L.cfg.gridDim = dim3(C, T);
  L.cfg.blockDim = dim3(kAdThreads);
  L.cfg.dynamicSmemBytes = 0;
  L.cfg.stream = st;
  L.attr[0].id = cudaLaunchAttributeClusterDimension;
  L.attr[0].val.clusterDim.x = C;
  L.attr[0].val.clusterDim.y = 1;
  L.attr[0].val.clusterDim.z = 1;
  L.attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  L.attr[1].val.programmaticStreamSerializationAllowed = 1;
  L.cfg.attrs = L.attr;
  L.cfg.numAttrs = pdl ? 2 : 1;
}

template <bool MERGE>
cudaError_t launch_adapter_form(const void* x, const void* A, const void* B, const int32_t* ids,
                                const float* scale, const float* partial, int S, void* out,
                                int T, int d_in, int d_out, int r, int n_slots, uint32_t* err,
                                bool pdl, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (T > 65535) return cudaErrorInvalidValue;
  AdapterLaunch L;
  adapter_launch_config(L, T, d_in, d_out, false, pdl, st);
  const bf16* xe = static_cast<const bf16*>(x);
  const bf16* Ae = static_cast<const bf16*>(A);
  const bf16* Be = static_cast<const bf16*>(B);
  // ranks up to 32: 64 registers for up to 64 tokens and from 256 on, 80 in
  // between (measured per batch size on 4096 x 4096 layers)
  const bool lean = T <= 64 || T >= 256;
#define LORA_ADAPTER_CASE(RR, MB)                                                              \
  return cudaLaunchKernelEx(&L.cfg, bgmv_adapter_kernel<RR, MERGE, MB>, xe, Ae, Be, ids,      \
                            scale, partial, S, out, T, d_in, d_out, n_slots, L.kc, L.nc, err)
  switch (r) {
    case 8:
      if (lean) LORA_ADAPTER_CASE(8, 4);
      LORA_ADAPTER_CASE(8, 3);
    case 16:
      if (lean) LORA_ADAPTER_CASE(16, 4);
      LORA_ADAPTER_CASE(16, 3);
    case 32:
      if (lean) LORA_ADAPTER_CASE(32, 4);
      LORA_ADAPTER_CASE(32, 3);
    case 64: LORA_ADAPTER_CASE(64, 3);
    case 128: LORA_ADAPTER_CASE(128, 3);
    default: return cudaErrorInvalidValue;
  }
#undef LORA_ADAPTER_CASE
}

template <bool MERGE>
cudaError_t launch_ragged_form(const void* x, const void* A, const void* B, const RaggedPool& rp,
                               const int32_t* ids, const float* scale, const float* partial,
                               int S, void* out, int T, int d_in, int d_out, int n_slots,
                               uint32_t* err, bool pdl, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (T > 65535 || rp.r_max < 8 || rp.r_max > 128) return cudaErrorInvalidValue;
  AdapterLaunch L;
  adapter_launch_config(L, T, d_in, d_out, true, pdl, st);
  return cudaLaunchKernelEx(&L.cfg, bgmv_adapter_ragged_kernel<MERGE>,
                            static_cast<const bf16*>(x), static_cast<const bf16*>(A),
                            static_cast<const bf16*>(B), rp.a_off, rp.b_off, rp.rank,
                            rp.a_elems, rp.b_elems, rp.r_max, ids, scale, partial, S, out, T,
                            d_in, d_out, n_slots, L.kc, L.nc, err);
}

}  // namespace

int adapter_cluster_size(int T, int d_in, int d_out, bool ragged) {
  // up to 4 CTAs per token on wide layers (the shrink's A slice and the
  // expand's B slice per CTA stay small) while the grid stays within ~256
  // CTAs, so all of them fit on the GPU beside the decode GEMM; at least
  // enough that each CTA keeps its columns in registers; at most the
  // portable cluster size of 8.  A ragged pool keeps up to 4 CTAs per token
  // at any T: its high-rank tokens are the long ones, and shorter per-CTA
  // slices measured faster there (for a padded rank-16 pool at 256 tokens,
  // slower)
  const int m = d_in < d_out ? d_in : d_out;
  int C = m >= 2048 ? 4 : (m >= 512 ? 2 : 1);
  int cap = T > 0 && T < 256 ? 256 / T : 1;
  if (ragged && cap < 4) cap = 4;
  if (C > cap) C = cap;
  const int by_cols = (d_out + kKeepGroups * kStride - 1) / (kKeepGroups * kStride);
  if (C < by_cols) C = by_cols;
  return C > 8 ? 8 : C;
}

cudaError_t launch_bgmv_adapter(const void* x, const void* A, const void* B, const int32_t* ids,
                                const float* scale, float* delta, int T, int d_in, int d_out,
                                int r, int n_slots, uint32_t* err, cudaStream_t st) {
  return launch_adapter_form<false>(x, A, B, ids, scale, nullptr, 0, delta, T, d_in, d_out, r,
                                    n_slots, err, false, st);
}

cudaError_t launch_bgmv_adapter_merge(const void* x, const void* A, const void* B,
                                      const int32_t* ids, const float* scale,
                                      const float* partial, int S, void* y, int T, int d_in,
                                      int d_out, int r, int n_slots, uint32_t* err, bool pdl,
                                      cudaStream_t st) {
  return launch_adapter_form<true>(x, A, B, ids, scale, partial, S, y, T, d_in, d_out, r,
                                   n_slots, err, pdl, st);
}

cudaError_t launch_bgmv_adapter_ragged(const void* x, const void* A, const void* B,
                                       const RaggedPool& rp, const int32_t* ids,
                                       const float* scale, float* delta, int T, int d_in,
                                       int d_out, int n_slots, uint32_t* err, cudaStream_t st) {
  return launch_ragged_form<false>(x, A, B, rp, ids, scale, nullptr, 0, delta, T, d_in, d_out,
                                   n_slots, err, false, st);
}

cudaError_t launch_bgmv_adapter_ragged_merge(const void* x, const void* A, const void* B,
                                             const RaggedPool& rp, const int32_t* ids,
                                             const float* scale, const float* partial, int S,
                                             void* y, int T, int d_in, int d_out, int n_slots,
                                             uint32_t* err, bool pdl, cudaStream_t st) {
  return launch_ragged_form<true>(x, A, B, rp, ids, scale, partial, S, y, T, d_in, d_out,
                                  n_slots, err, pdl, st);
}

}  // namespace lora
