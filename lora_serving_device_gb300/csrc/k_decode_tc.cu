// The decode-sized base product (T <= 256 tokens) on tcgen05 tensor cores,
// with the adapter term -- a ready fp32 [T, d_out] tensor written by the
// BGMV expand running concurrently -- added in the epilogue so y is stored
// once ("Multi-LoRA batching and adapter paging", section "Walking through a
// batch": the base matrix is read once for the whole batch and each row gets
// its own adapter term; "Serving multiple LoRAs ...": the expand is added
// directly to the base output).
//
// Shape: "swap AB".  The MMA's M = 128 d_out columns of W0 (A operand,
// MN-major, W0 stays [d_in, d_out] row-major), N = the token tile (B operand
// = x, K-major), so the skinny token dimension is the MMA's N.  Decode is
// bound by streaming W0 from HBM; what matters is how many bytes each SM
// keeps in flight, and that depends on the size of each TMA box rather than
// on the depth of the ring.  So each pipeline stage carries KSUB 64-row K
// blocks and W0 arrives as two 64-column x (64*KSUB)-row boxes per stage.
//
// d_in is split over a thread-block cluster of S CTAs (S a power of two,
// <= 8); rank z owns d_out rows [z*128/S, (z+1)*128/S) of the tile.  Each
// CTA moves its fp32 partial tile from tensor memory into shared memory
// (its own rows straight into slot z of its receive buffer, the others into
// a staging area that reuses the drained pipeline ring), then sends each
// owner its rows with one bulk shared-memory copy per peer, counted in bytes
// on the owner's receive mbarrier.  The owner sums the S slots, adds the
// adapter term and stores its rows of y.
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
constexpr int kEpiThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct DecParams {
  int T, d_in, d_out, n_slots;
  int n_stage;  // K stages over d_in: ceil(d_in / (64 * KSUB))
  int stages;   // ring depth
  const int32_t* ids;
  const float* delta;  // fp32 [T, d_out] adapter term, or null (base only)
  bf16* y;
  uint32_t* err;
};

template <int BT, int KSUB>
struct DecLayout {
  static constexpr uint32_t kXSub = BT * 128;               // one 64-wide K block of x
  static constexpr uint32_t kXBytes = KSUB * kXSub;
  static constexpr uint32_t kWBox = 64 * KSUB * 128;         // 64 columns x 64*KSUB rows
  static constexpr uint32_t kStage = kXBytes + 2 * kWBox;
  static constexpr uint32_t kRb = 128 * BT * 4;              // receive buffer: S slots
  // the fp32 partial tile is staged in the (drained) ring before it is sent
  static_assert(kRb <= kStage, "staging must fit in one pipeline stage");
  static __host__ __device__ uint32_t rb(int stages) { return stages * kStage; }
  static __host__ __device__ uint32_t tok(int stages) { return rb(stages) + kRb; }
  static __host__ __device__ uint32_t bars(int stages) { return tok(stages) + BT * 4; }
  // full[stages], empty[stages], accum_full, rx_full
  static __host__ __device__ uint32_t misc(int stages) { return bars(stages) + (2 * stages + 2) * 8; }
  static __host__ __device__ uint32_t total(int stages) { return misc(stages) + 16; }
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = ptx::mbar_wait_bounded(bar, parity, abort, kWaitLimitNs) ? 1 : 0;
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
                       const __grid_constant__ CUtensorMap tm_w, const DecParams p) {
  using Lay = DecLayout<BT, KSUB>;
  constexpr int kTmemCols = BT < 32 ? 32 : BT;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, BT, true, false);
  static_assert(BT % 16 == 0 && BT >= 32 && BT <= 128, "token tile");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  int* tok = reinterpret_cast<int*>(smem + Lay::tok(p.stages));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::bars(p.stages));
  uint64_t* empty = full + p.stages;
  uint64_t* accum_full = empty + p.stages;
  uint64_t* rx_full = accum_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::misc(p.stages));
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + Lay::misc(p.stages) + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * 128, t0 = blockIdx.y * BT;
  const int S = static_cast<int>(gridDim.z), z = static_cast<int>(blockIdx.z);
  const int rows_own = 128 / S;
  const uint32_t slot_bytes = static_cast<uint32_t>(rows_own * BT * 4);

  // ---- prologue: warp 0 initialises the barriers and starts streaming;
  // the others wait for that (named barrier 2); warp 1 allocates TMEM and
  // hands the address to the epilogue warps (named barrier 3).  Peers send
  // into this CTA only after phase A of the cluster barrier, which every
  // thread arrives at once the receive mbarrier is initialised.
  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_w);
      ptx::prefetch_tmap(&tm_x);
      for (int i = 0; i < p.stages; ++i) {
        ptx::mbar_init(&full[i], 1);
        ptx::mbar_init(&empty[i], 1);
      }
      ptx::mbar_init(accum_full, 1);
      ptx::mbar_init(rx_full, 1);
      *abort_f = 0;
      ptx::fence_mbar_init();
      // the S-1 peers' slots complete phase 0 of rx_full
      if (S > 1) ptx::mbar_arrive_expect_tx(rx_full, static_cast<uint32_t>(S - 1) * slot_bytes);
    }
    __syncwarp();
    if (S > 1) ptx::cluster_arrive_release();
    named_arrive(2, kThreads);
  } else {
    named_sync(2, kThreads);
    if (S > 1) ptx::cluster_arrive_relaxed();
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
  const int kb0 = static_cast<int>(static_cast<long long>(z) * p.n_stage / S);
  const int kb1 = static_cast<int>(static_cast<long long>(z + 1) * p.n_stage / S);

  if (warp == 0) {
    // ---------------- producer -------------------------------------------
    for (int it = 0; it < kb1 - kb0; ++it) {
      const int st = it % p.stages;
      const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
      if (!warp_wait(&empty[st], ph ^ 1u, abort_f)) break;
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
      for (int it = 0; it < kb1 - kb0; ++it) {
        const int st = it % p.stages;
        const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
        if (!ptx::mbar_wait_bounded(&full[st], ph, abort_f, kWaitLimitNs)) break;
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
    // ---------------- epilogue warps -------------------------------------
    const int etid = tid - 64;
    bool bad = false;
    for (int i = etid; i < BT; i += kEpiThreads) {
      const int t = t0 + i;
      int u = -1;
      if (t < p.T) {
        const int id = p.ids[t];
        if (slot_valid(id, p.n_slots)) u = 0;
        else if (id != -1) bad = true;
      }
      tok[i] = u;
    }
    if (bad && blockIdx.x == 0 && z == 0) flag_error(p.err, LORA_DEVERR_BAD_SLOT);
    const bool acc_ok = warp_wait(accum_full, 0, abort_f);
    if (acc_ok) {
      ptx::tc_fence_after();
      // TMEM lane = d_out row n of the tile, column = token.  Row n belongs
      // to rank n / (128/S): this rank's own rows go to its receive slot z,
      // the others to the staging area, rank-major so each peer's rows are
      // one contiguous block.  Rows are BT fp32 (token-contiguous) and the
      // 16-byte chunks of row n are XOR-swizzled by n & 7, so the 32 lanes'
      // vector stores spread over all banks.
      const int q = warp & 3;
      const int n = q * 32 + lane;
      const int owner = n / rows_own, n_loc = n - owner * rows_own;
      float* row = owner == z
          ? reinterpret_cast<float*>(smem + Lay::rb(p.stages)) + (z * rows_own + n_loc) * BT
          : reinterpret_cast<float*>(smem) + n * BT;
      const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BT; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld16(tq + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
        ptx::tmem_ld16(tq + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int chunk = ((c0 >> 2) + j) ^ (n & 7);
          *reinterpret_cast<float4*>(row + chunk * 4) =
              make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                          __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
      }
      ptx::fence_proxy_async_smem();  // the bulk copies read the staging area
    }
    named_sync(1, kEpiThreads);
    if (S > 1) {
      ptx::cluster_wait_acquire();  // phase A: every peer's rx_full is initialised
      if (acc_ok && etid < S && etid != z) {
        const uint32_t src = ptx::smem_u32(smem) + static_cast<uint32_t>(etid) * slot_bytes;
        const uint32_t dst_local = ptx::smem_u32(smem + Lay::rb(p.stages)) +
                                   static_cast<uint32_t>(z) * slot_bytes;
        ptx::bulk_copy_to_cluster(ptx::mapa_shared(dst_local, static_cast<uint32_t>(etid)), src,
                                  slot_bytes,
                                  ptx::mapa_shared(ptx::smem_u32(rx_full), static_cast<uint32_t>(etid)));
      }
    }
  }

  // ---- reduction of the S slots of this rank's rows, store y -------------
  if (S > 1 && warp < 2) ptx::cluster_wait_acquire();  // phase A (epilogue warps did it)
  // this rank owns d_out rows [z * 128/S, (z+1) * 128/S) of the tile; the
  // adapter-term loads (L2) are issued before the receive wait so they
  // overlap it
  const int groups = rows_own / 8;
  const int rows_tok = min(BT, p.T - t0);
  const int n_items = rows_tok * groups;
  constexpr int kMaxItems = (BT * 16 + kThreads - 1) / kThreads;  // S = 1: 16 groups
  float dl[kMaxItems][8];
  // every CTA waits, so that this grid completing implies its predecessors
  // completed; the adapter term is written by the kernel launched just before.
  // Rows of base-only tokens are loaded too (they are in bounds) and dropped
  // in the sum, so this does not wait for the token table.
  pdl_wait();
  if (p.delta != nullptr) {
#pragma unroll
    for (int u = 0; u < kMaxItems; ++u) {
      const int e = tid + u * kThreads;
      const int g = e / (rows_tok > 0 ? rows_tok : 1), t = e - g * rows_tok;
      const int n = n0 + z * rows_own + g * 8;
      if (e < n_items && n < p.d_out)
        load8_dep(p.delta + static_cast<size_t>(t0 + t) * p.d_out + n, dl[u]);
    }
  }
  __syncthreads();  // the token table and slot z, written by the epilogue warps
  bool rx_ok = true;
  if (S > 1) {
    rx_ok = ptx::mbar_wait_bounded(rx_full, 0, abort_f, kWaitLimitNs);
    __syncwarp();
    // phase B: this CTA has received every peer's slot, so the peers'
    // staging areas have been read; a CTA leaves only after phase B
    ptx::cluster_arrive_relaxed();
  }
  if (rx_ok && !*abort_f) {
    const float* rb = reinterpret_cast<const float*>(smem + Lay::rb(p.stages));
#pragma unroll
    for (int u = 0; u < kMaxItems; ++u) {
      const int e = tid + u * kThreads;
      if (e >= n_items) break;
      const int g = e / rows_tok, t = e - g * rows_tok;
      const int n = n0 + z * rows_own + g * 8;
      if (n >= p.d_out) continue;
      float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int src = 0; src < S; ++src) {
        const float* blk = rb + (src * rows_own + g * 8) * BT;
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] += blk[j * BT + ((((t >> 2) ^ j) << 2) | (t & 3))];
      }
      if (p.delta != nullptr && tok[t] >= 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] += dl[u][j];
      }
      store8(p.y + static_cast<size_t>(t0 + t) * p.d_out + n, f);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_f) flag_error(p.err, LORA_DEVERR_TIMEOUT);
  if (S > 1) ptx::cluster_wait_acquire();  // phase B
}

template <int BT, int KSUB>
cudaError_t launch_decode_variant(const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                                  DecParams prm, int tiles_n, int tiles_t, int S,
                                  cudaStream_t st, const DeviceInfo& dev) {
  using Lay = DecLayout<BT, KSUB>;
  int stages = 0;
  for (int s = 4; s >= 2; --s) {
    if (Lay::total(s) + 1024 <= dev.max_smem_optin) {
      stages = s;
      break;
    }
  }
  if (stages == 0) return cudaErrorInvalidConfiguration;
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
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = S;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_w, prm);
}

}  // namespace

cudaError_t launch_decode_tc(const void* x, const void* W0, const int32_t* ids,
                             const float* delta, void* y, int T, int d_in, int d_out, int n_slots,
                             uint32_t* err, cudaStream_t st, const DeviceInfo& dev) {
  // token tile: 32 / 64 / 128 tokens; above 128, 128-token tiles
  const int BT = T <= 32 ? 32 : (T <= 64 ? 64 : 128);
  const int ksub = BT <= 64 ? 4 : 2;
  const int tiles_n = (d_out + 127) / 128;
  const int tiles_t = (T + BT - 1) / BT;
  const int n_stage = (d_in + 64 * ksub - 1) / (64 * ksub);
  int S = dev.num_sms / (tiles_n * tiles_t);
  if (S > 8) S = 8;
  if (S > n_stage) S = n_stage;
  int S2 = 1;
  while (S2 * 2 <= S) S2 *= 2;

  CUtensorMap tm_x, tm_w;
  if (!encode_tensor_map_bf16(&tm_x, x, d_in, T, d_in, 64, BT) ||
      !encode_tensor_map_bf16(&tm_w, W0, d_out, d_in, d_out, 64, 64 * ksub))
    return cudaErrorInvalidValue;
  DecParams prm;
  prm.T = T;
  prm.d_in = d_in;
  prm.d_out = d_out;
  prm.n_slots = n_slots;
  prm.n_stage = n_stage;
  prm.stages = 0;
  prm.ids = ids;
  prm.delta = delta;
  prm.y = static_cast<bf16*>(y);
  prm.err = err;
  if (BT == 32) return launch_decode_variant<32, 4>(tm_x, tm_w, prm, tiles_n, tiles_t, S2, st, dev);
  if (BT == 64) return launch_decode_variant<64, 4>(tm_x, tm_w, prm, tiles_n, tiles_t, S2, st, dev);
  return launch_decode_variant<128, 2>(tm_x, tm_w, prm, tiles_n, tiles_t, S2, st, dev);
}

}  // namespace lora
