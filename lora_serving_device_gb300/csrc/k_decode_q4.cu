// The decode-sized base product with a 4-bit base matrix, split over d_in
// ("Serving Many LoRA Adapters", section "When It Falls Down": 4-bit base
// models in the QLoRA style next to bf16 adapters, the base weights passing
// through dequantisation while the adapter path stays in bf16):
//   partial[z, t, :] = x[t, K_z] deq(W0)[K_z, :]        z = 0 .. S-1
//   deq(W0)[k, n] = bf16( codebook[code[n, k]] * absmax[k / 64, n] )
// Storage: codes [d_out, d_in / 2] bytes, k contiguous per output column
// (rows 2i and 2i + 1 of column n in the low and high nibble of byte i of
// its row, the [out, in] orientation of a QLoRA weight), absmax
// [d_in / 64, d_out] bf16 (one scale per 64 consecutive rows of a column),
// codebook [16] bf16.  The product is rounded once to bf16 (the MMA's
// operand type); the bf16 adapter term is added by the merge kernel exactly
// as for a bf16 base.
//
// Same "swap AB" shape as the bf16 decode GEMM (MMA M = 128 d_out columns,
// N = the token tile), but the dequantised base tile never touches shared
// memory: each dequantising thread owns one output column, reads that
// column's 32 code bytes of a 64-row K block from the staged codes, maps each byte to
// its two codebook values with a table replicated per lane (no bank
// conflicts), applies the block's scale with one bf16x2 FMA per pair, and
// writes the 32 bf16 pairs into its own tensor-memory lane.  The MMA reads
// A (the dequantised W0 tile, row n in lane n) from tensor memory and B (x)
// from shared memory.
//   warp 0      TMA producer: codes and scales of 4 K blocks per stage
//               (128-byte swizzled box of 128 columns), x per K block (the
//               first code stages go out before the wait for the
//               predecessor grid, x after it)
//   warp 1      MMA issuer (and TMEM allocator)
//   warps 2-17  dequantise in four groups of four warps; warp w serves TMEM
//               lanes 32 (w % 4) .. + 31, group g the g-th K block of each
//               code stage (enough warps in flight to hide the table loads'
//               latency); warps 2-5 then drain the fp32 accumulator.
// Every on-chip wait is bounded in time; on timeout the kernel raises
// LORA_DEVERR_TIMEOUT and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int kQGroups = 4;                       // dequantising groups of 4 warps
constexpr int kQDqWarps = 4 * kQGroups;
constexpr int kQThreads = 64 + 32 * kQDqWarps;     // + the producer and MMA warps
constexpr int kQSB = 2;   // TMEM buffers of dequantised A, one code stage (4 K blocks, 128 columns) each
constexpr uint32_t kQLutBytes = 256 * 32 * 4;
constexpr uint32_t kQStage = 128 * 128 + 1024;  // codes of 4 K blocks x 128 columns + scales
constexpr uint64_t kQWaitNs = 2000000000ull;

struct Q4Params {
  int T, d_in, d_out;
  int n_blk;     // 64-row K blocks over d_in
  int xs, qs;    // x ring and code ring depths
  const uint16_t* codebook;
  uint32_t* err;
};

// Shared memory: [x ring][code ring][table][barriers][misc].  The fp32
// partial tile is staged over the drained rings at the end.
template <int BT>
struct Q4Layout {
  static constexpr uint32_t kX = BT * 128;             // x: BT tokens x 64 K, K-major, swizzled
  static constexpr uint32_t kOutBytes = BT * 128 * 4;  // fp32 partial tile, token-major
  static constexpr int kTmemCols = 512;  // the accumulator, then the kQSB stage buffers
  static __host__ __device__ uint32_t qring(int xs) { return xs * kX; }
  static __host__ __device__ uint32_t lut(int xs, int qs) {
    const uint32_t rings = xs * kX + qs * kQStage;
    return rings > kOutBytes ? rings : ((kOutBytes + 1023u) & ~1023u);
  }
  static __host__ __device__ uint32_t bars(int xs, int qs) { return lut(xs, qs) + kQLutBytes; }
  // x_full[xs], q_full[qs], q_empty[qs], dq_full[kQSB], dq_empty[kQSB], accum
  static __host__ __device__ uint32_t misc(int xs, int qs) {
    return bars(xs, qs) + (xs + 2 * qs + 2 * kQSB + 1) * 8;
  }
  static __host__ __device__ uint32_t total(int xs, int qs) { return misc(xs, qs) + 16; }
};

__device__ __forceinline__ bool q4_warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = ptx::mbar_wait_bounded(bar, parity, abort, kQWaitNs) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
__device__ __forceinline__ void q4_named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void q4_named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// two bf16 products, each rounded once (a * b + (-0) is exact before rounding)
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}

template <int BT>
__global__ void __launch_bounds__(kQThreads, 1)
    decode_q4_kernel(const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_s,
                     const __grid_constant__ CUtensorMap tm_p, const Q4Params p) {
  using Lay = Q4Layout<BT>;
  constexpr int kTmemCols = Lay::kTmemCols;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, BT, false, false);
  static_assert(BT % 16 == 0 && BT >= 32 && BT <= 256, "token tile");
  static_assert(BT + kQSB * 128 <= kTmemCols && kQGroups == 4, "TMEM columns; one group per K block");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* qring = smem + Lay::qring(p.xs);
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + Lay::lut(p.xs, p.qs));
  uint64_t* x_full = reinterpret_cast<uint64_t*>(smem + Lay::bars(p.xs, p.qs));
  uint64_t* q_full = x_full + p.xs;
  uint64_t* q_empty = q_full + p.qs;
  uint64_t* dq_full = q_empty + p.qs;
  uint64_t* dq_empty = dq_full + kQSB;
  uint64_t* accum_full = dq_empty + kQSB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::misc(p.xs, p.qs));
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + Lay::misc(p.xs, p.qs) + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * 128, t0 = blockIdx.y * BT;
  const int S = static_cast<int>(gridDim.z), z = static_cast<int>(blockIdx.z);
  const int kb0 = z * p.n_blk / S;
  const int kb1 = (z + 1) * p.n_blk / S;
  const int n_it = kb1 - kb0;              // 64-row K blocks of this CTA
  const int n_q = (n_it + 3) / 4;          // code stages (4 K blocks each)

  // ---- prologue: warp 0 initialises the barriers, warp 1 allocates TMEM
  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_q);
      ptx::prefetch_tmap(&tm_s);
      ptx::prefetch_tmap(&tm_x);
      ptx::prefetch_tmap(&tm_p);
      for (int i = 0; i < p.xs; ++i) ptx::mbar_init(&x_full[i], 1);
      for (int i = 0; i < p.qs; ++i) {
        ptx::mbar_init(&q_full[i], 1);
        ptx::mbar_init(&q_empty[i], kQDqWarps);  // every dequantising warp releases it
      }
      for (int i = 0; i < kQSB; ++i) {
        ptx::mbar_init(&dq_full[i], kQDqWarps);  // every dequantising warp fills its part
        ptx::mbar_init(&dq_empty[i], 1);
      }
      ptx::mbar_init(accum_full, 1);
      *abort_f = 0;
      ptx::fence_mbar_init();
    }
    __syncwarp();
    q4_named_arrive(2, kQThreads);
  } else {
    q4_named_sync(2, kQThreads);
    if (warp == 1) {
      ptx::tmem_alloc(tmem_slot, kTmemCols);
      ptx::tmem_relinquish();
      ptx::tc_fence_before();
      q4_named_arrive(3, kQThreads - 32);
    } else {
      q4_named_sync(3, kQThreads - 32);
    }
    ptx::tc_fence_after();
  }
  const uint32_t tmem = warp == 0 ? 0u : *tmem_slot;
  const uint32_t a_tmem = tmem + BT;  // the kQSB stage buffers follow the accumulator

  if (warp == 0) {
    // ---------------- producer -------------------------------------------
    // codes and scales of the first ring's worth of stages go out before the
    // wait for the predecessor grid (weights: no kernel of the layer writes
    // them), x after it
    auto load_q = [&](int iq) {
      uint8_t* st = qring + static_cast<size_t>(iq % p.qs) * kQStage;
      ptx::mbar_arrive_expect_tx(&q_full[iq % p.qs], 128 * 128 + 4 * 128 * 2);
      ptx::tma_load_2d(st, &tm_q, &q_full[iq % p.qs], (kb0 + 4 * iq) * 32, n0);
      ptx::tma_load_2d(st + 128 * 128, &tm_s, &q_full[iq % p.qs], n0, kb0 + 4 * iq);
    };
    const int q_pre = n_q < p.qs ? n_q : p.qs;
    if (lane == 0)
      for (int iq = 0; iq < q_pre; ++iq) load_q(iq);
    pdl_wait();               // x may be written by the predecessor grid
    pdl_launch_dependents();  // the next kernel of the chain may start
    int iq_next = q_pre;
    for (int it = 0; it < n_it; ++it) {
      const int s = it % p.xs;
      // the slot's previous tile, x of block b = it - xs, is free once the MMAs
      // of b's code stage completed: the commit that frees that stage's TMEM
      // buffer (phase (b / 4) / kQSB of dq_empty[(b / 4) % kQSB]; with xs <= 8
      // that barrier cannot have moved two phases past it)
      if (it >= p.xs) {
        const int sq = (it - p.xs) / 4;
        if (!q4_warp_wait(&dq_empty[sq % kQSB], static_cast<uint32_t>(sq / kQSB) & 1u, abort_f))
          break;
      }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&x_full[s], Lay::kX);
        ptx::tma_load_2d(smem + static_cast<size_t>(s) * Lay::kX, &tm_x, &x_full[s],
                         (kb0 + it) * 64, t0);
      }
      // one more code stage once the dequantisers released its slot
      if (iq_next < n_q && it % 4 == 3) {
        const int qsl = iq_next % p.qs;
        if (!q4_warp_wait(&q_empty[qsl], (static_cast<uint32_t>(iq_next / p.qs) & 1u) ^ 1u,
                          abort_f))
          break;
        if (lane == 0) load_q(iq_next);
        ++iq_next;
      }
      __syncwarp();
    }
    // code stages not yet issued (short x ring)
    for (; iq_next < n_q; ++iq_next) {
      const int qsl = iq_next % p.qs;
      if (!q4_warp_wait(&q_empty[qsl], (static_cast<uint32_t>(iq_next / p.qs) & 1u) ^ 1u,
                        abort_f))
        break;
      if (lane == 0) load_q(iq_next);
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer -----------------------------------------
    if (lane == 0) {
      bool live = true;
      for (int iq = 0; iq < n_q && live; ++iq) {
        const int sb = iq % kQSB;
        if (!ptx::mbar_wait_bounded(&dq_full[sb], static_cast<uint32_t>(iq / kQSB) & 1u, abort_f,
                                    kQWaitNs))
          break;
        ptx::tc_fence_after();
        for (int j = 0; j < 4 && 4 * iq + j < n_it; ++j) {
          const int it = 4 * iq + j, s = it % p.xs;
          if (!ptx::mbar_wait_bounded(&x_full[s], static_cast<uint32_t>(it / p.xs) & 1u, abort_f,
                                      kQWaitNs)) {
            live = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t xa = ptx::smem_u32(smem + static_cast<size_t>(s) * Lay::kX);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A: 16 K elements = 8 TMEM columns per step; x: K-major, 32 bytes per step
            const uint64_t xd = ptx::sdesc_sw128(xa + kk * 32, 16, 1024);
            ptx::mma_bf16_ta(tmem, a_tmem + sb * 128 + j * 32 + kk * 8, xd, kIdesc,
                             (it > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (live) ptx::mma_commit(&dq_empty[sb]);  // frees stage buffer sb and its x slots
      }
      ptx::mma_commit(accum_full);
    }
    __syncwarp();
  } else {
    // ---------------- dequantisation (warps 2 .. 2 + kQDqWarps) ------------
    // warp w owns TMEM lanes 32 (w % 4) .. + 31 = tile columns; group g =
    // (w - 2) / 4 takes K block g of each code stage, so four groups keep
    // enough warps in flight to hide the table loads' latency
    const int q = warp & 3, grp = (warp - 2) >> 2;
    const int m = q * 32 + lane;
    {
      // code byte v -> (codebook[v & 15], codebook[v >> 4]) as bf16x2, one
      // copy per lane: entry v of lane l at word 32 v + l; lane e holds
      // codebook[e % 16] and the others read it by shuffle
      const uint32_t cbr = __ldg(p.codebook + (lane & 15));
      const int dt = tid - 64;
      constexpr int kPer = 256 * 32 / (32 * kQDqWarps);
#pragma unroll 4
      for (int j = 0; j < kPer; ++j) {
        const int i = dt + 32 * kQDqWarps * j, v = i >> 5;
        const uint32_t lo = __shfl_sync(0xffffffffu, cbr, v & 15);
        const uint32_t hi = __shfl_sync(0xffffffffu, cbr, v >> 4);
        lut[i] = lo | (hi << 16);
      }
    }
    q4_named_sync(4, 32 * kQDqWarps);
    const uint32_t* lut_l = lut + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int sw = m & 7;  // the 128-byte swizzle of this thread's code row
    bool ok = true;
#pragma unroll 1
    for (int iq = 0; iq < n_q && ok; ++iq) {
      const int qsl = iq % p.qs;
      ok = ptx::mbar_wait_bounded(&q_full[qsl], static_cast<uint32_t>(iq / p.qs) & 1u, abort_f,
                                  kQWaitNs);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint8_t* st = qring + static_cast<size_t>(qsl) * kQStage;
      {
        const int j = grp;           // K block within the stage
        const int it = 4 * iq + j;   // K block of the CTA
        const int sb = iq % kQSB;
        uint32_t v[32];
        if (it < n_it) {             // warp-uniform
          const uint4 lo = *reinterpret_cast<const uint4*>(st + m * 128 + (((2 * j) ^ sw) << 4));
          const uint4 hi = *reinterpret_cast<const uint4*>(st + m * 128 + (((2 * j + 1) ^ sw) << 4));
          const uint32_t s = *reinterpret_cast<const uint16_t*>(st + 128 * 128 + j * 256 + m * 2);
          const uint32_t s2 = s | (s << 16);
          const uint32_t w8[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
#pragma unroll
            for (int bb = 0; bb < 4; ++bb)
              v[4 * e + bb] = bf16x2_mul(lut_l[((w8[e] >> (8 * bb)) & 0xffu) * 32], s2);
          }
        }
        // the buffer is free once the MMAs of the stage two back completed
        ok = q4_warp_wait(&dq_empty[sb], (static_cast<uint32_t>(iq / kQSB) & 1u) ^ 1u, abort_f);
        if (!ok) break;
        if (it < n_it) {
          ptx::tc_fence_after();
          ptx::tmem_st32(a_tmem + lane_base + sb * 128 + j * 32, v);
          ptx::tmem_st_wait();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&dq_full[sb]);  // every warp, block or not
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&q_empty[qsl]);  // this warp is done with the stage
    }

    if (warp < 6) {
      // ------------- epilogue warps 2-5: TMEM -> fp32 partial tile --------
      // as in the bf16 decode GEMM: TMEM lane = column, TMEM column = token;
      // staged token-major at the start of the drained rings, then one 3-D
      // TMA store into partial [S][T][d_out] (clipped at T and d_out)
      const bool acc_ok = q4_warp_wait(accum_full, 0, abort_f) && n_it > 0 && !*abort_f;
      float* stage_out = reinterpret_cast<float*>(smem);
      if (acc_ok) {
        ptx::tc_fence_after();
        const uint32_t tq = tmem + lane_base;
        constexpr int kCols = BT < 64 ? BT : 64;
#pragma unroll 1
        for (int c0 = 0; c0 < BT; c0 += kCols) {
          uint32_t r[kCols];
#pragma unroll
          for (int jj = 0; jj < kCols / 16; ++jj)
            ptx::tmem_ld16(tq + c0 + 16 * jj, *reinterpret_cast<uint32_t(*)[16]>(r + 16 * jj));
          ptx::tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < kCols; ++jj) stage_out[(c0 + jj) * 128 + m] = __uint_as_float(r[jj]);
        }
        ptx::fence_proxy_async_smem();
      }
      q4_named_sync(1, 128);
      if (tid == 64 && acc_ok) {
        ptx::tma_store_3d(&tm_p, stage_out, n0, t0, z);
        ptx::bulk_commit_group();
        ptx::bulk_wait_group_read_all();
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_f) flag_error(p.err, LORA_DEVERR_TIMEOUT);
}

template <int BT>
cudaError_t launch_q4_variant(const CUtensorMap& tm_x, const CUtensorMap& tm_q,
                              const CUtensorMap& tm_s, const CUtensorMap& tm_p, Q4Params prm,
                              int tiles_n, int tiles_t, int S, bool pdl, cudaStream_t st,
                              const DeviceInfo& dev) {
  using Lay = Q4Layout<BT>;
  // x ring: about 64 KB of x; code ring: as deep as the rest allows (<= 8)
  // x slots are recycled a code stage (4 K blocks) at a time through the
  // dq_empty barriers, so the ring must hold a whole stage (4 <= xs <= 8; see
  // the producer)
  int xs = static_cast<int>(65536 / Lay::kX);
  if (xs < 4) xs = 4;
  if (xs > 8) xs = 8;
  int qs = 0;
  for (int s = 8; s >= 2; --s) {
    if (Lay::total(xs, s) + 1024 <= dev.max_smem_optin) {
      qs = s;
      break;
    }
  }
  if (qs == 0) return cudaErrorInvalidConfiguration;
  prm.xs = xs;
  prm.qs = qs;
  const size_t smem = Lay::total(xs, qs) + 1024;
  auto kern = decode_q4_kernel<BT>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, tiles_t, S);
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_q, tm_s, tm_p, prm);
}

// ---------------------------------------------------------------- quantiser
// One thread per (64-row block b, column n): the block's absmax, then each
// weight's nearest codebook entry after division by it (ties to the lower
// code; an all-zero block divides nothing and takes the entry nearest 0).
// Quotient and distances are IEEE fp32 (round to nearest), so the codes are
// reproducible bit for bit.  The thread writes the block's 32 code bytes of
// its column (row n of the code matrix) with two 16-byte stores.
__global__ void quantize_q4_kernel(const bf16* __restrict__ W, const uint16_t* __restrict__ cb,
                                   uint8_t* __restrict__ Wq, uint16_t* __restrict__ absmax,
                                   int d_in, int d_out) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(d_in / 64) * d_out) return;
  const int b = static_cast<int>(idx / d_out), n = static_cast<int>(idx % d_out);
  float cbf[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) cbf[e] = __uint_as_float(static_cast<uint32_t>(cb[e]) << 16);
  const uint16_t* Wb = reinterpret_cast<const uint16_t*>(W) + static_cast<size_t>(b) * 64 * d_out + n;
  float mx = 0.f;
  for (int k = 0; k < 64; ++k)
    mx = fmaxf(mx, fabsf(__uint_as_float(static_cast<uint32_t>(Wb[static_cast<size_t>(k) * d_out]) << 16)));
  // the maximum is a bf16 value, so storing its upper half is exact
  absmax[static_cast<size_t>(b) * d_out + n] = static_cast<uint16_t>(__float_as_uint(mx) >> 16);
  // row k of the block: nibble k % 8 of word k / 8 (byte k / 2, nibble k % 2)
  uint32_t packed[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    uint32_t word = 0;
#pragma unroll 2
    for (int kk = 0; kk < 8; ++kk) {
      const int k = 8 * g + kk;
      const float w =
          __uint_as_float(static_cast<uint32_t>(Wb[static_cast<size_t>(k) * d_out]) << 16);
      const float v = mx > 0.f ? __fdiv_rn(w, mx) : 0.f;
      uint32_t best = 0;
      float bd = fabsf(__fsub_rn(v, cbf[0]));
#pragma unroll
      for (int e = 1; e < 16; ++e) {
        const float dd = fabsf(__fsub_rn(v, cbf[e]));
        if (dd < bd) {
          bd = dd;
          best = static_cast<uint32_t>(e);
        }
      }
      word |= best << (4 * kk);
    }
    packed[g] = word;
  }
  uint4* dst = reinterpret_cast<uint4*>(Wq + static_cast<size_t>(n) * (d_in / 2) + static_cast<size_t>(b) * 32);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
}

}  // namespace

int decode_q4_max_split(int d_in) {
  const int n_blk = d_in / 64;
  return n_blk < LORA_MAX_KSPLIT ? n_blk : LORA_MAX_KSPLIT;
}

cudaError_t launch_decode_q4(const void* x, const void* Wq, const void* absmax,
                             const void* codebook, float* partial, int T, int d_in, int d_out,
                             int S, uint32_t* err, bool pdl, cudaStream_t st,
                             const DeviceInfo& dev) {
  if (T <= 0) return cudaSuccess;
  if (d_in % 64 != 0 || d_out % 32 != 0) return cudaErrorInvalidValue;
  const int BT = T <= 32 ? 32 : (T <= 64 ? 64 : (T <= 128 ? 128 : 256));
  const int tiles_n = (d_out + 127) / 128;
  const int tiles_t = (T + BT - 1) / BT;
  const int n_blk = d_in / 64;
  if (S < 1 || S > n_blk || tiles_t > 65535) return cudaErrorInvalidValue;

  CUtensorMap tm_x, tm_q, tm_s, tm_p;
  if (!encode_tensor_map_bf16(&tm_x, x, d_in, T, d_in, 64, BT) ||
      !encode_tensor_map_u8_sw128(&tm_q, Wq, d_in / 2, d_out, d_in / 2, 128, 128) ||
      !encode_tensor_map_plain_2d(&tm_s, absmax, 2, d_out, d_in / 64,
                                  static_cast<uint64_t>(d_out) * 2, 128, 4) ||
      !encode_tensor_map_f32_3d(&tm_p, partial, d_out, T, S, 128, BT))
    return cudaErrorInvalidValue;
  Q4Params prm;
  prm.T = T;
  prm.d_in = d_in;
  prm.d_out = d_out;
  prm.n_blk = n_blk;
  prm.xs = prm.qs = 0;
  prm.codebook = static_cast<const uint16_t*>(codebook);
  prm.err = err;
  if (BT == 32) return launch_q4_variant<32>(tm_x, tm_q, tm_s, tm_p, prm, tiles_n, tiles_t, S, pdl, st, dev);
  if (BT == 64) return launch_q4_variant<64>(tm_x, tm_q, tm_s, tm_p, prm, tiles_n, tiles_t, S, pdl, st, dev);
  if (BT == 128) return launch_q4_variant<128>(tm_x, tm_q, tm_s, tm_p, prm, tiles_n, tiles_t, S, pdl, st, dev);
  return launch_q4_variant<256>(tm_x, tm_q, tm_s, tm_p, prm, tiles_n, tiles_t, S, pdl, st, dev);
}

// ---------------------------------------------------------------- dequantiser
// The inverse for batches above 256 tokens, which take the bf16 prefill path
// over a dequantised copy of W0: W [d_in, d_out] bf16, W[k, n] =
// bf16(codebook[code[n, k]] * absmax[k / 64, n]), the product of two bf16
// values exact in fp32 and rounded once (the same values the 4-bit decode
// GEMM feeds its MMAs).  One 64-row x 64-column block per CTA: each of 128
// threads reads 32 codes of one column with one 16-byte load, the block is
// transposed through shared memory and written as 64 rows of 128 bytes.
__global__ void __launch_bounds__(256)
    dequantize_q4_kernel(const uint8_t* __restrict__ Wq, const uint16_t* __restrict__ absmax,
                         const uint16_t* __restrict__ cb, uint16_t* __restrict__ W, int d_in,
                         int d_out) {
  __shared__ __align__(16) uint16_t tile[64][64 + 8];  // [k][n], rows 144 bytes apart
  __shared__ float cbf[16];
  const int n0 = blockIdx.x * 64, k0 = blockIdx.y * 64;
  if (threadIdx.x < 16) cbf[threadIdx.x] = __uint_as_float(static_cast<uint32_t>(cb[threadIdx.x]) << 16);
  __syncthreads();
  if (threadIdx.x < 128) {
    const int c = threadIdx.x >> 1, hh = threadIdx.x & 1;
    const int n = n0 + c;
    if (n < d_out) {
      const uint4 q = *reinterpret_cast<const uint4*>(Wq + static_cast<size_t>(n) * (d_in / 2) +
                                                      k0 / 2 + 16 * hh);
      const float sf =
          __uint_as_float(static_cast<uint32_t>(absmax[static_cast<size_t>(k0 / 64) * d_out + n]) << 16);
      const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const uint32_t byte = (w4[e] >> (8 * bb)) & 0xffu;
          const int k = 32 * hh + 2 * (4 * e + bb);  // low nibble: row k, high: row k + 1
          const __nv_bfloat16 lo = __float2bfloat16_rn(cbf[byte & 15u] * sf);
          const __nv_bfloat16 hi = __float2bfloat16_rn(cbf[byte >> 4] * sf);
          tile[k][c] = *reinterpret_cast<const uint16_t*>(&lo);
          tile[k + 1][c] = *reinterpret_cast<const uint16_t*>(&hi);
        }
      }
    }
  }
  __syncthreads();
  // 64 rows x 64 columns out: thread j writes 16 columns of row j / 4
  const int row = threadIdx.x >> 2, qq = threadIdx.x & 3;
  const int k = k0 + row, n = n0 + 16 * qq;
  if (k < d_in && n < d_out) {
    const uint4* src = reinterpret_cast<const uint4*>(&tile[row][16 * qq]);
    uint4* dst = reinterpret_cast<uint4*>(W + static_cast<size_t>(k) * d_out + n);
    dst[0] = src[0];
    dst[1] = src[1];
  }
}

cudaError_t launch_dequantize_q4(const void* Wq, const void* absmax, const void* codebook,
                                 void* W, int d_in, int d_out, cudaStream_t st) {
  if (d_in % 64 != 0 || d_out % 32 != 0) return cudaErrorInvalidValue;
  const dim3 grid((d_out + 63) / 64, d_in / 64);
  dequantize_q4_kernel<<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(Wq),
                                             static_cast<const uint16_t*>(absmax),
                                             static_cast<const uint16_t*>(codebook),
                                             static_cast<uint16_t*>(W), d_in, d_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_q4(const void* W0, const void* codebook, void* Wq, void* absmax,
                               int d_in, int d_out, cudaStream_t st) {
  if (d_in % 64 != 0 || d_out % 32 != 0) return cudaErrorInvalidValue;
  const long long n = static_cast<long long>(d_in / 64) * d_out;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  quantize_q4_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      static_cast<const bf16*>(W0), static_cast<const uint16_t*>(codebook),
      static_cast<uint8_t*>(Wq), static_cast<uint16_t*>(absmax), d_in, d_out);
  return cudaGetLastError();
}

}  // namespace lora
