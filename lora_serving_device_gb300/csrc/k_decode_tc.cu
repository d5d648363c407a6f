// The decode-sized base product on tcgen05 tensor cores, split over d_in:
//   partial[z, t, :] = x[t, K_z] W0[K_z, :]        z = 0 .. S-1
// where K_0 .. K_{S-1} are contiguous ranges of d_in.  The kernel that runs
// next in the decode chain (the BGMV adapter kernel) sums the S fp32
// partials, adds the adapter term and stores y once ("Multi-LoRA batching
// and adapter paging", section "Walking through a batch": the base matrix is
// read once for the whole batch and each row gets its own adapter term).
//
// Shape: "swap AB".  The MMA's M = 128 d_out columns of W0 (A operand,
// MN-major, W0 stays [d_in, d_out] row-major), N = the token tile (B operand
// = x, K-major), so the skinny token dimension is the MMA's N.  Decode is
// bound by streaming W0 from HBM, and each SM's share of it arrives at the
// rate its bytes in flight allow: each pipeline stage carries KSUB 64-row K
// blocks, W0 arrives as two 64-column x (64*KSUB)-row TMA boxes per stage,
// and the ring takes all the shared memory there is.
//
// The split is over CTAs, not clusters: each CTA stages its partial tile
// from tensor memory in the drained ring, stores it with one TMA tensor
// store (into L2) and exits, so nothing in it waits on another CTA.  It is
// launched as a programmatic dependent: the producer fills the ring with W0
// (which no earlier kernel of the layer writes) before it waits for the
// predecessor grid, then loads x, which the predecessor may have written.
// So the W0 stream of this layer overlaps the tail of the previous kernel.
// The x blocks of those first stages are prefetched into L2 before the wait
// as well, so that their loads after it are L2 hits.
//
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM
// allocator), warps 2-5 = epilogue.  Every on-chip wait is bounded in time;
// on timeout the kernel raises LORA_DEVERR_TIMEOUT and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int kThreads = 192;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct DecParams {
  int T, d_in, d_out;
  int n_blk;          // K blocks of 64*KSUB rows over d_in
  int stages;         // ring depth
  uint64_t wait_ns;   // limit of every bounded wait
  int hold_producer;  // diagnostic: the producer issues no load at all
  uint32_t* err;
};

template <int BT, int KSUB>
struct DecLayout {
  static constexpr uint32_t kXSub = BT * 128;               // one 64-wide K block of x
  static constexpr uint32_t kXBytes = KSUB * kXSub;
  static constexpr uint32_t kWBox = 64 * KSUB * 128;         // 64 columns x 64*KSUB rows
  static constexpr uint32_t kStage = kXBytes + 2 * kWBox;
  static constexpr uint32_t kOutBytes = BT * 128 * 4;       // fp32 partial tile, token-major
  static __host__ __device__ uint32_t bars(int stages) { return stages * kStage; }
  // full[stages], empty[stages], accum_full
  static __host__ __device__ uint32_t misc(int stages) { return bars(stages) + (2 * stages + 1) * 8; }
  static __host__ __device__ uint32_t total(int stages) { return misc(stages) + 16; }
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = ptx::mbar_wait_bounded(bar, parity, abort, limit) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int BT, int KSUB>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_p, const DecParams p) {
  using Lay = DecLayout<BT, KSUB>;
  constexpr int kTmemCols = BT < 32 ? 32 : BT;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, BT, true, false);
  static_assert(BT % 16 == 0 && BT >= 32 && BT <= 256, "token tile");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::bars(p.stages));
  uint64_t* empty = full + p.stages;
  uint64_t* accum_full = empty + p.stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::misc(p.stages));
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + Lay::misc(p.stages) + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * 128, t0 = blockIdx.y * BT;
  const int S = static_cast<int>(gridDim.z), z = static_cast<int>(blockIdx.z);

  // ---- prologue: warp 0 initialises the barriers and starts streaming;
  // the others wait for that (named barrier 2); warp 1 allocates TMEM and
  // hands the address to the epilogue warps (named barrier 3)
  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_w);
      ptx::prefetch_tmap(&tm_x);
      ptx::prefetch_tmap(&tm_p);
      for (int i = 0; i < p.stages; ++i) {
        ptx::mbar_init(&full[i], 1);
        ptx::mbar_init(&empty[i], 1);
      }
      ptx::mbar_init(accum_full, 1);
      *abort_f = 0;
      ptx::fence_mbar_init();
    }
    __syncwarp();
    named_arrive(2, kThreads);
  } else {
    named_sync(2, kThreads);
    if (warp == 1) {
      ptx::tmem_alloc(tmem_slot, kTmemCols);
      ptx::tmem_relinquish();
      ptx::tc_fence_before();
      named_arrive(3, kThreads - 32);
    } else {
      named_sync(3, kThreads - 32);
    }
    ptx::tc_fence_after();
  }
  const uint32_t tmem = warp == 0 ? 0u : *tmem_slot;
  const int kb0 = z * p.n_blk / S;
  const int kb1 = (z + 1) * p.n_blk / S;
  const int n_it = kb1 - kb0;

  if (warp == 0) {
    // ---------------- producer -------------------------------------------
    // W0 of the first ring's worth of stages goes out before the wait for
    // the predecessor grid; x of those stages right after it
    // (held back: nothing is issued, so every consumer's bounded wait runs out)
    const int pre = p.hold_producer ? 0 : (n_it < p.stages ? n_it : p.stages);
    if (lane == 0) {
      for (int it = 0; it < pre; ++it) {
        uint8_t* Wr = smem + static_cast<size_t>(it) * Lay::kStage + Lay::kXBytes;
        const int k0 = (kb0 + it) * 64 * KSUB;
        ptx::mbar_arrive_expect_tx(&full[it], Lay::kStage);
#pragma unroll
        for (int h = 0; h < 2; ++h) ptx::tma_load_2d(Wr + h * Lay::kWBox, &tm_w, &full[it], n0 + 64 * h, k0);
      }
    }
    // x of the ring's first stages into L2 before the wait (the blocks the
    // loads right after it fetch): a prefetch moves no data into this SM,
    // and those loads read what the predecessor wrote.  One CTA in eight
    // column tiles of a split issues it.  A short K range (at most two
    // rings' worth) has the x of all its stages prefetched; on longer ones
    // the prefetches would queue ahead of the ring's own loads.
    if (lane == 0 && !p.hold_producer && blockIdx.x % 8 == 0) {
      const int n_pf = n_it <= 2 * p.stages ? n_it : pre;
      for (int it = 0; it < n_pf; ++it) {
        const int k0 = (kb0 + it) * 64 * KSUB;
#pragma unroll
        for (int j = 0; j < KSUB; ++j)
          if (k0 + 64 * j < p.d_in) ptx::tma_prefetch_l2_2d(&tm_x, k0 + 64 * j, t0);
      }
    }
    // every CTA waits, so this grid completing implies its predecessors did
    pdl_wait();
    pdl_launch_dependents();  // x is ready: the next kernel of the chain may start
    if (lane == 0) {
      for (int it = 0; it < pre; ++it) {
        uint8_t* X = smem + static_cast<size_t>(it) * Lay::kStage;
        const int k0 = (kb0 + it) * 64 * KSUB;
#pragma unroll
        for (int j = 0; j < KSUB; ++j) ptx::tma_load_2d(X + j * Lay::kXSub, &tm_x, &full[it], k0 + 64 * j, t0);
      }
    }
    __syncwarp();
    for (int it = pre; !p.hold_producer && it < n_it; ++it) {
      const int st = it % p.stages;
      const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
      if (!warp_wait(&empty[st], ph ^ 1u, abort_f, p.wait_ns)) break;
      if (lane == 0) {
        uint8_t* X = smem + static_cast<size_t>(st) * Lay::kStage;
        uint8_t* Wr = X + Lay::kXBytes;
        const int k0 = (kb0 + it) * 64 * KSUB;
        ptx::mbar_arrive_expect_tx(&full[st], Lay::kStage);
#pragma unroll
        for (int h = 0; h < 2; ++h) ptx::tma_load_2d(Wr + h * Lay::kWBox, &tm_w, &full[st], n0 + 64 * h, k0);
#pragma unroll
        for (int j = 0; j < KSUB; ++j) ptx::tma_load_2d(X + j * Lay::kXSub, &tm_x, &full[st], k0 + 64 * j, t0);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer -----------------------------------------
    if (lane == 0) {
      for (int it = 0; it < n_it; ++it) {
        const int st = it % p.stages;
        const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
        if (!ptx::mbar_wait_bounded(&full[st], ph, abort_f, p.wait_ns)) break;
        ptx::tc_fence_after();
        const uint32_t xa = ptx::smem_u32(smem + static_cast<size_t>(st) * Lay::kStage);
        const uint32_t wa = xa + Lay::kXBytes;
#pragma unroll
        for (int j = 0; j < KSUB; ++j) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // x: K-major, 128-byte swizzle; 16 elements = 32 bytes per step
            const uint64_t xd = ptx::sdesc_sw128(xa + j * Lay::kXSub + kk * 32, 16, 1024);
            // W0: MN-major, 128-byte swizzle; 16 K-rows = 2048 bytes per step;
            // the two 64-column boxes are kWBox apart (LBO), 8-row groups 1 KiB (SBO)
            const uint64_t wd = ptx::sdesc_sw128(wa + (j * 64 + kk * 16) * 128, Lay::kWBox, 1024);
            ptx::mma_bf16(tmem, wd, xd, kIdesc, (it > 0 || j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        ptx::mma_commit(&empty[st]);
      }
      ptx::mma_commit(accum_full);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps: TMEM -> fp32 partial tile ----------
    // TMEM lane = d_out column of the tile, TMEM column = token.  The tile is
    // staged token-major ([BT][128] fp32) at the start of the ring, which the
    // MMAs have finished reading: for each token a warp writes 32 consecutive
    // floats (no bank conflicts).  One thread then stores it with a 3-D TMA
    // store into partial [S][T][d_out]; rows past T and columns past d_out
    // are clipped by the tensor bounds.
    const int etid = tid - 64;
    const bool acc_ok = warp_wait(accum_full, 0, abort_f, p.wait_ns) && n_it > 0 && !*abort_f;
    float* stage_out = reinterpret_cast<float*>(smem);
    if (acc_ok) {
      ptx::tc_fence_after();
      const int q = warp & 3;
      const int nl = q * 32 + lane;
      const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
      constexpr int kCols = BT < 64 ? BT : 64;  // TMEM loads in flight before one wait
#pragma unroll 1
      for (int c0 = 0; c0 < BT; c0 += kCols) {
        uint32_t v[kCols];
#pragma unroll
        for (int j = 0; j < kCols / 16; ++j)
          ptx::tmem_ld16(tq + c0 + 16 * j, *reinterpret_cast<uint32_t(*)[16]>(v + 16 * j));
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kCols; ++j) stage_out[(c0 + j) * 128 + nl] = __uint_as_float(v[j]);
      }
      ptx::fence_proxy_async_smem();
    }
    named_sync(1, kThreads - 64);
    if (etid == 0 && acc_ok) {
      ptx::tma_store_3d(&tm_p, stage_out, n0, t0, z);
      ptx::bulk_commit_group();
      ptx::bulk_wait_group_read_all();  // the staging area must outlive the read
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

template <int BT, int KSUB>
cudaError_t launch_decode_variant(const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                                  const CUtensorMap& tm_p, DecParams prm, int tiles_n,
                                  int tiles_t, int S, bool pdl, cudaStream_t st,
                                  const DeviceInfo& dev) {
  using Lay = DecLayout<BT, KSUB>;
  int stages = 0;
  for (int s = 6; s >= 2; --s) {
    if (Lay::total(s) + 1024 <= dev.max_smem_optin) {
      stages = s;
      break;
    }
  }
  // the drained ring must hold the staged fp32 partial tile
  if (stages == 0 || Lay::kOutBytes > stages * Lay::kStage) return cudaErrorInvalidConfiguration;
  prm.stages = stages;
  const size_t smem = Lay::total(stages) + 1024;
  auto kern = decode_gemm_kernel<BT, KSUB>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, tiles_t, S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_w, tm_p, prm);
}

// token tile and K-block depth per decode batch size
int decode_bt(int T) { return T <= 32 ? 32 : (T <= 64 ? 64 : (T <= 128 ? 128 : 256)); }
int decode_ksub(int BT) { return BT <= 64 ? 3 : (BT == 128 ? 2 : 1); }
int decode_blocks(int T, int d_in) {
  const int rows = 64 * decode_ksub(decode_bt(T > 0 ? T : 1));
  return (d_in + rows - 1) / rows;
}

}  // namespace

int decode_gemm_split(int T, int d_in, int d_out) {
  // one CTA per SM of a 152-SM GB300: (d_out/128 column tiles) x (token
  // tiles) x S; at most one split per K block and LORA_MAX_KSPLIT splits
  const int BT = decode_bt(T > 0 ? T : 1);
  const int tiles = ((d_out + 127) / 128) * ((T + BT - 1) / BT);
  int S = kDecodeScheduleCtas / (tiles > 0 ? tiles : 1);
  const int smax = decode_gemm_max_split(T, d_in);
  if (S > smax) S = smax;
  return S < 1 ? 1 : S;
}

int decode_gemm_max_split(int T, int d_in) {
  const int n_blk = decode_blocks(T, d_in);
  return n_blk < LORA_MAX_KSPLIT ? n_blk : LORA_MAX_KSPLIT;
}

namespace {

cudaError_t launch_decode_common(const void* x, const void* W0, float* partial, int T, int d_in,
                                 int d_out, int S, uint64_t wait_ns, int hold, uint32_t* err,
                                 bool pdl, cudaStream_t st, const DeviceInfo& dev) {
  if (T <= 0) return cudaSuccess;
  const int BT = decode_bt(T);
  const int ksub = decode_ksub(BT);
  const int tiles_n = (d_out + 127) / 128;
  const int tiles_t = (T + BT - 1) / BT;
  const int n_blk = decode_blocks(T, d_in);
  if (S < 1 || S > n_blk || tiles_t > 65535) return cudaErrorInvalidValue;

  CUtensorMap tm_x, tm_w, tm_p;
  if (!encode_tensor_map_bf16(&tm_x, x, d_in, T, d_in, 64, BT) ||
      !encode_tensor_map_bf16(&tm_w, W0, d_out, d_in, d_out, 64, 64 * ksub) ||
      !encode_tensor_map_f32_3d(&tm_p, partial, d_out, T, S, 128, BT))
    return cudaErrorInvalidValue;
  DecParams prm;
  prm.T = T;
  prm.d_in = d_in;
  prm.d_out = d_out;
  prm.n_blk = n_blk;
  prm.stages = 0;
  prm.wait_ns = wait_ns;
  prm.hold_producer = hold;
  prm.err = err;
  if (BT == 32)
    return launch_decode_variant<32, 3>(tm_x, tm_w, tm_p, prm, tiles_n, tiles_t, S, pdl, st, dev);
  if (BT == 64)
    return launch_decode_variant<64, 3>(tm_x, tm_w, tm_p, prm, tiles_n, tiles_t, S, pdl, st, dev);
  if (BT == 128)
    return launch_decode_variant<128, 2>(tm_x, tm_w, tm_p, prm, tiles_n, tiles_t, S, pdl, st, dev);
  return launch_decode_variant<256, 1>(tm_x, tm_w, tm_p, prm, tiles_n, tiles_t, S, pdl, st, dev);
}

}  // namespace

cudaError_t launch_decode_gemm(const void* x, const void* W0, float* partial, int T, int d_in,
                               int d_out, int ksplit, uint32_t* err, bool pdl, cudaStream_t st,
                               const DeviceInfo& dev) {
  const int S = ksplit >= 1 ? ksplit : decode_gemm_split(T, d_in, d_out);
  return launch_decode_common(x, W0, partial, T, d_in, d_out, S, kWaitLimitNs, 0, err, pdl, st,
                              dev);
}

cudaError_t launch_decode_gemm_held(const void* x, const void* W0, float* partial, int T,
                                    int d_in, int d_out, uint64_t wait_ns, uint32_t* err,
                                    cudaStream_t st, const DeviceInfo& dev) {
  return launch_decode_common(x, W0, partial, T, d_in, d_out, 1, wait_ns, 1, err, false, st, dev);
}

int decode_uniform_split(int T, int d_in, int d_out) { return decode_gemm_split(T, d_in, d_out); }

}  // namespace lora
