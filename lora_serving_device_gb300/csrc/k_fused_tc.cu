// The base product of the multi-LoRA layer on tcgen05 tensor cores, with the
// adapter expand folded into the same accumulator so y is written once.
//
// What it computes, for one output tile (a d_out range x a token range):
//
//   acc  = x[tokens, :] W0[:, cols]                       (base K-blocks)
//   acc += sum over the distinct adapters a in the tile of
//          V_a[tokens, :] B_a[:, cols]                    (LoRA K-blocks)
//   y    = bf16(acc)
//
// where V_a holds the (scaled) shrink output v of the tile's tokens that use
// adapter a and zeros in every other row.  This is the additivity of the
// adapter term ("Serving many LoRA adapters", blog.ecitis.org, section
// "Low-rank structure and additivity"): the base output does not depend on
// the adapter, so one shared GEMM serves every row, and each row's low-rank
// correction is extra accumulation on top ("Multi-LoRA batching and adapter
// paging", section "Walking through a batch"; the expand is "added directly
// to the base output", "Serving multiple LoRAs ...", after its toy script).
// Concatenating the adapters along K, [x | V_a1 | V_a2 ...] x [W0 ; B_a1 ;
// B_a2 ...], turns the gathered expand into ordinary K-blocks of the same
// MMA pipeline: one 64-row K-block holds 64 / r adapters (r <= 64).
//
// Tile: MMA M = 128 tokens (A = x, K-major), N = 256 d_out columns (B = W0,
// MN-major); this is the prefill-sized path (more than 256 tokens).  d_in
// is split over a cluster of S CTAs when there are fewer tiles than SMs; the
// S fp32 partial tiles, staged in each CTA's drained ring, are summed
// through distributed shared memory.  Both operands arrive by TMA with
// 128-byte swizzle; the accumulator lives in
// tensor memory; one thread issues the MMAs.  Warp roles: warp 0 = TMA
// producer (also builds the masked V operand of the LoRA K-blocks), warp 1 =
// MMA issuer (and TMEM allocator), warps 2-5 = epilogue (load v during the
// main loop, then TMEM -> shared -> global).  Every on-chip wait is bounded
// in time; on timeout the kernel raises LORA_DEVERR_TIMEOUT and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int kBK = 64;           // K elements per stage: one 128-byte swizzle row of bf16
constexpr int kThreads = 192;     // 6 warps
constexpr int kEpiThreads = 128;  // warps 2..5
constexpr int kRedPad = 4;        // fp32 padding per staged accumulator row
constexpr int kPanel = 8;         // column tiles per L2 panel of the tile order
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s; the longest legitimate wait is ~ms

struct TcParams {
  int T, d_in, d_out, r, n_slots;
  int n_kblk;    // base stages: ceil(d_in / (64 * KS))
  int stages;
  int box_rows;  // rows of one B_pool TMA box: min(r, 32)
  int lg_box;    // log2(box_rows)
  int lg_upa;    // log2(r / box_rows)
  int v_ksplit;
  const int32_t* ids;
  const float* vpart;
  bf16* y;
  uint32_t* err;
};

struct SmemLayout {
  uint32_t x_sub, x_bytes, w_box, stage_bytes, stages_total;
  uint32_t vt, tok, uniq, bitmap, bars, misc, total;
};

// Offsets from a 1024-byte aligned base (the 128-byte swizzle repeats every
// 8 rows = 1024 bytes, and TMA / MMA agree on it only from such a base).
// A base stage carries KS 64-deep K blocks: KS x boxes of 64 x BT and BN/64
// W0 boxes of 64 columns x 64*KS rows (taller boxes move more bytes per TMA
// operation).  A LoRA stage uses the first K block only.
template <int BT, int BN, int KS>
__host__ __device__ inline SmemLayout smem_layout(int stages, int r, int n_slots) {
  SmemLayout L;
  L.x_sub = BT * 128;
  L.x_bytes = KS * L.x_sub;
  L.w_box = KS * 8192;
  L.stage_bytes = L.x_bytes + (BN / 64) * L.w_box;
  L.stages_total = static_cast<uint32_t>(stages) * L.stage_bytes;
  uint32_t o = L.stages_total;
  L.vt = o;
  o += BT * r * 4;
  o = (o + 15u) & ~15u;
  L.tok = o;
  o += BT * 4;
  L.uniq = o;
  o += BT * 4;
  L.bitmap = o;
  o += ((n_slots + 31) / 32) * 4;
  o = (o + 7u) & ~7u;
  L.bars = o;
  o += (3 * stages + 2) * 8;  // full, empty, accum_full, vt_ready, lora_built
  L.misc = o;
  // TMEM address, adapter count, abort flag, LoRA stages posted; per ring slot
  // (16 at most) its K blocks and whether it is a LoRA stage; the ring slot of
  // each posted LoRA stage (a 16-entry mailbox)
  o += 112;
  L.total = o;
  return L;
}

// One elected lane waits; the result is broadcast so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = ptx::mbar_wait_bounded(bar, parity, abort, kWaitLimitNs) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Named barriers (barrier 0 is __syncthreads): 1 = the four epilogue warps,
// 2 = barrier init done, 3 = TMEM address published.
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int BT, int BN, int KS>
__global__ void __launch_bounds__(kThreads, 1)
    fused_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_y,
                    const TcParams p) {
  constexpr int kUmmaN = BN;
  constexpr int kTmemCols = kUmmaN < 32 ? 32 : kUmmaN;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, kUmmaN, false, true);
  constexpr int kRedLd = BN + kRedPad;   // staged accumulator: [token][d_out column]
  constexpr int kWBoxes = BN / 64;
  static_assert(BT == 128, "MMA M is 128 tokens");
  static_assert(kUmmaN % 16 == 0 && kUmmaN >= 16 && kUmmaN <= 256, "MMA N");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const SmemLayout L = smem_layout<BT, BN, KS>(p.stages, p.r, p.n_slots);
  float* vt = reinterpret_cast<float*>(smem + L.vt);
  int* tok = reinterpret_cast<int*>(smem + L.tok);
  int* uniq = reinterpret_cast<int*>(smem + L.uniq);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L.bitmap);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + p.stages;
  uint64_t* accum_full = empty + p.stages;
  uint64_t* vt_ready = accum_full + 1;
  uint64_t* lora_built = vt_ready + 1;  // [stages]: the epilogue warps built the V operand
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  int* n_uniq_s = reinterpret_cast<int*>(smem + L.misc + 4);
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + L.misc + 8);
  volatile int* lora_posted = reinterpret_cast<volatile int*>(smem + L.misc + 12);
  uint8_t* stage_kblocks = smem + L.misc + 16;  // K blocks the stage in each ring slot holds
  uint8_t* stage_lora = smem + L.misc + 32;     // 1: the slot holds a LoRA stage
  int* lora_mailbox = reinterpret_cast<int*>(smem + L.misc + 48);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // tile order: panels of kPanel column tiles; within a panel the column
  // tile varies fastest, so the CTAs resident at one time share a W0 panel
  // (16 MiB at d_in = 4096) and a band of x rows, and both stay in L2
  const int tiles_n = (p.d_out + BN - 1) / BN, tiles_t = (p.T + BT - 1) / BT;
  const int lin = static_cast<int>(blockIdx.x);
  const int g = lin / (kPanel * tiles_t);
  const int gn = min(kPanel, tiles_n - g * kPanel);
  const int rem = lin - g * kPanel * tiles_t;
  const int tile_n = g * kPanel + rem % gn, tile_t = rem / gn;
  const int n0 = tile_n * BN, t0 = tile_t * BT;
  const int S = static_cast<int>(gridDim.z), z = static_cast<int>(blockIdx.z);

  // ---- prologue: warp 0 initialises the barriers and starts the TMA stream
  // at once; the other warps wait for the barriers (named barrier 2), warp 1
  // allocates TMEM and hands its address to the epilogue warps (barrier 3).
  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_x);
      ptx::prefetch_tmap(&tm_w);
      ptx::prefetch_tmap(&tm_b);
      for (int i = 0; i < p.stages; ++i) {
        ptx::mbar_init(&full[i], 1);
        ptx::mbar_init(&empty[i], 1);
      }
      ptx::mbar_init(accum_full, 1);
      ptx::mbar_init(vt_ready, kEpiThreads);
      for (int i = 0; i < p.stages; ++i) ptx::mbar_init(&lora_built[i], kEpiThreads / 32);
      *abort_f = 0;
      *lora_posted = 0;
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
  const int upa = p.r >> p.lg_box;       // TMA boxes per adapter (r / min(r, 32))
  const int G = (kBK / 2) >> p.lg_box;   // boxes per LoRA K-block (each used twice)
  const int kb0 = static_cast<int>(static_cast<long long>(z) * p.n_kblk / S);
  const int kb1 = static_cast<int>(static_cast<long long>(z + 1) * p.n_kblk / S);
  const int nbase = kb1 - kb0;
  // LoRA K-blocks of this CTA; known once the epilogue warps published the
  // tile's adapter list (vt_ready)
  auto lora_groups = [&](int* U_out) {
    const int U = *n_uniq_s * upa;
    *U_out = U;
    const int n_groups = (U + G - 1) / G;
    return (z < n_groups) ? (n_groups - z + S - 1) / S : 0;
  };

  if (warp == 0) {
    // ---------------- producer -------------------------------------------
    // Base K-blocks stream W0 / x by TMA.  LoRA K-blocks (see the top of this
    // file) are slotted in between them as soon as the epilogue warps have
    // published the tile's adapters and v, so their B loads overlap the W0
    // stream; the MMA issuer consumes stages in ring order whatever they hold.
    int it = 0;
    bool ok = true;
    bool lora_known = false;
    int U = 0, my_groups = 0, gi = 0;
    auto issue_base = [&](int kb, int st) {
      uint8_t* X = smem + static_cast<size_t>(st) * L.stage_bytes;
      uint8_t* Wr = X + L.x_bytes;
      if (lane == 0) {
        stage_kblocks[st] = KS;
        stage_lora[st] = 0;
        ptx::mbar_arrive_expect_tx(&full[st], L.stage_bytes);
#pragma unroll
        for (int j = 0; j < KS; ++j)
          ptx::tma_load_2d(X + j * L.x_sub, &tm_x, &full[st], (kb * KS + j) * kBK, t0);
#pragma unroll
        for (int h = 0; h < kWBoxes; ++h)
          ptx::tma_load_2d(Wr + h * L.w_box, &tm_w, &full[st], n0 + 64 * h, kb * KS * kBK);
      }
      __syncwarp();
    };
    auto issue_lora = [&](int g, int st) {
      // the epilogue warps build this stage's masked V operand (and zero the
      // W rows B leaves empty); the producer only posts the slot and loads
      // the B rows, so the base stream is not held up
      uint8_t* X = smem + static_cast<size_t>(st) * L.stage_bytes;
      uint8_t* Wr = X + L.x_bytes;
      const int u_first = (z + g * S) * G;
      const int n_units = min(G, U - u_first);
      if (lane == 0) {
        stage_kblocks[st] = 1;
        stage_lora[st] = 1;
        lora_mailbox[g & 15] = st;
        __threadfence_block();
        *lora_posted = g + 1;
        ptx::mbar_arrive_expect_tx(
            &full[st], static_cast<uint32_t>(2 * n_units * p.box_rows * 128 * kWBoxes));
      }
      __syncwarp();
      // one B box per lane: (unit, 64-column box, hi/lo copy)
      if (lane < 2 * n_units * kWBoxes) {
        const int u = lane / (2 * kWBoxes), rem = lane % (2 * kWBoxes);
        const int hb = rem >> 1, half = rem & 1;
        const int wv = u_first + u;
        const int a = uniq[wv >> p.lg_upa];
        const int qb = (wv & (upa - 1)) << p.lg_box;
        ptx::tma_load_2d(Wr + hb * L.w_box + (half * (kBK / 2) + u * p.box_rows) * 128, &tm_b,
                         &full[st], n0 + 64 * hb, a * p.r + qb);
      }
      __syncwarp();
    };
    auto next_slot = [&](int* st) {
      *st = it % p.stages;
      const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
      return warp_wait(&empty[*st], ph ^ 1u, abort_f);
    };
    for (int b = 0; b < nbase && ok; ++b) {
      int st;
      if (!(ok = next_slot(&st))) break;
      issue_base(kb0 + b, st);
      ++it;
      if (!lora_known) {
        int ready = 0;
        if (lane == 0) ready = ptx::mbar_test_wait(vt_ready, 0) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          lora_known = true;
          my_groups = lora_groups(&U);
        }
      }
      if (lora_known && gi < my_groups) {
        if (!(ok = next_slot(&st))) break;
        issue_lora(gi++, st);
        ++it;
      }
    }
    if (ok && !lora_known && warp_wait(vt_ready, 0, abort_f)) {
      lora_known = true;
      my_groups = lora_groups(&U);
    }
    while (ok && lora_known && gi < my_groups) {
      int st;
      if (!(ok = next_slot(&st))) break;
      issue_lora(gi++, st);
      ++it;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer -----------------------------------------
    if (lane == 0) {
      uint32_t lora_par = 0;  // bit s: phase parity of lora_built[s]
      auto consume = [&](int it) {
        const int st = it % p.stages;
        const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
        if (!ptx::mbar_wait_bounded(&full[st], ph, abort_f, kWaitLimitNs)) return false;
        if (stage_lora[st]) {  // written by the producer before its arrive
          if (!ptx::mbar_wait_bounded(&lora_built[st], (lora_par >> st) & 1u, abort_f,
                                      kWaitLimitNs))
            return false;
          lora_par ^= 1u << st;
        }
        ptx::tc_fence_after();
        const uint32_t xa = ptx::smem_u32(smem + static_cast<size_t>(st) * L.stage_bytes);
        const uint32_t wa = xa + L.x_bytes;
        const int nkb = stage_kblocks[st];  // written by the producer before its arrive
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          if (j >= nkb) break;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // K-major x / V: advance 16 elements = 32 bytes inside the swizzle row
            const uint64_t xd = ptx::sdesc_sw128(xa + j * L.x_sub + kk * 32, 16, 1024);
            // MN-major W0 / B: advance 16 K-rows = 2048 bytes; the 64-column
            // boxes are w_box apart (LBO), 8-row groups 1 KiB apart (SBO)
            const uint64_t wd = ptx::sdesc_sw128(wa + (j * kBK + kk * 16) * 128, L.w_box, 1024);
            const uint32_t accum = (it > 0 || j > 0 || kk > 0) ? 1u : 0u;
            ptx::mma_bf16(tmem, xd, wd, kIdesc, accum);
          }
        }
        ptx::mma_commit(&empty[st]);
        return true;
      };
      int it = 0;
      bool ok = true;
      for (; it < nbase && ok; ++it) ok = consume(it);
      if (ok && ptx::mbar_wait_bounded(vt_ready, 0, abort_f, kWaitLimitNs)) {
        int U;
        const int my_groups = lora_groups(&U);
        for (int gi = 0; gi < my_groups && ok; ++gi, ++it) ok = consume(it);
      }
      ptx::mma_commit(accum_full);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps -------------------------------------
    const int etid = tid - 64;
    const int n_words = (p.n_slots + 31) >> 5;
    // the tile's slot ids and its distinct adapters (ascending slot order),
    // built while the main loop streams W0
    bool bad = false;
    for (int i = etid; i < BT; i += kEpiThreads) {
      const int t = t0 + i;
      int sl = -1;
      if (t < p.T) {
        const int id = p.ids[t];
        if (slot_valid(id, p.n_slots)) sl = id;
        else if (id != -1) bad = true;
      }
      tok[i] = sl;
    }
    for (int wd = etid; wd < n_words; wd += kEpiThreads) bitmap[wd] = 0u;
    if (bad && tile_n == 0 && z == 0) flag_error(p.err, LORA_DEVERR_BAD_SLOT);
    epi_sync();
    for (int i = etid; i < BT; i += kEpiThreads) {
      const int sl = tok[i];
      if (sl >= 0) atomicOr(&bitmap[sl >> 5], 1u << (sl & 31));
    }
    epi_sync();
    if (warp == 2) {
      const int per = (n_words + 31) / 32;
      const int w0 = min(n_words, lane * per), w1 = min(n_words, w0 + per);
      int cnt = 0;
      for (int wd = w0; wd < w1; ++wd) cnt += __popc(bitmap[wd]);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int off = incl - cnt;
      for (int wd = w0; wd < w1; ++wd) {
        uint32_t m = bitmap[wd];
        while (m) {
          const int b = __ffs(m) - 1;
          m &= m - 1;
          uniq[off++] = wd * 32 + b;
        }
      }
      if (lane == 31) *n_uniq_s = incl;
    }
    epi_sync();
    const int n_uniq = *n_uniq_s;
    // tok[i] becomes the index of token i's adapter in uniq (-1: none)
    for (int i = etid; i < BT; i += kEpiThreads) {
      const int sl = tok[i];
      int u = -1;
      if (sl >= 0) {
        int lo = 0, hi = n_uniq - 1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (uniq[mid] < sl) lo = mid + 1;
          else hi = mid;
        }
        u = lo;
      }
      tok[i] = u;
    }
    pdl_wait();  // v is written by the shrink kernel launched just before
    if (n_uniq > 0) {
      const int qcn = p.r / 8;
      for (int e = etid; e < BT * qcn; e += kEpiThreads) {
        const int i = e / qcn, qc = e % qcn;
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (t0 + i < p.T && tok[i] >= 0) {
          const int t = t0 + i;
          for (int s = 0; s < p.v_ksplit; ++s) {
            float g[8];
            load8_dep(p.vpart + (static_cast<size_t>(s) * p.T + t) * p.r + qc * 8, g);
#pragma unroll
            for (int c = 0; c < 8; ++c) f[c] += g[c];
          }
        }
        store8(vt + i * p.r + qc * 8, f);
      }
    }
    epi_sync();
    ptx::mbar_arrive(vt_ready);
    {
      // this CTA's LoRA stages, in the order the producer posts their ring
      // slots: one token row per thread writes its 8 chunks of the masked V
      // operand (K-major, 128-byte swizzle): v = hi + lo with hi = bf16(v),
      // lo = bf16(v - hi); K rows [0, 32) carry hi parts, [32, 64) lo parts,
      // each against its own copy of the B rows; rows of tokens on other
      // adapters are zero
      int U;
      const int my_groups = lora_groups(&U);
      const int i = etid;  // BT == kEpiThreads
      for (int g2 = 0; g2 < my_groups; ++g2) {
        if (etid == 0) {
          const uint64_t tw = ptx::globaltimer_ns();
          while (*lora_posted <= g2) {
            if (*abort_f) break;
            if (ptx::globaltimer_ns() - tw > kWaitLimitNs) {
              *abort_f = 1;
              break;
            }
          }
          __threadfence_block();
        }
        epi_sync();
        if (*abort_f) break;
        const int st = lora_mailbox[g2 & 15];
        uint8_t* X = smem + static_cast<size_t>(st) * L.stage_bytes;
        uint8_t* Wr = X + L.x_bytes;
        const int u_first = (z + g2 * S) * G;
        const int n_units = min(G, U - u_first);
        const int tv = tok[i];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int kq = (c & 3) << 3;
          const int wu = kq >> p.lg_box;
          uint4 val = make_uint4(0u, 0u, 0u, 0u);
          if (wu < n_units && tv >= 0) {
            const int w = u_first + wu;
            if ((w >> p.lg_upa) == tv) {
              const int q0 = ((w & (upa - 1)) << p.lg_box) + (kq & (p.box_rows - 1));
              float f[8], h[8], l[8];
              load8(vt + i * p.r + q0, f);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                h[q] = __bfloat162float(__float2bfloat16_rn(f[q]));
                l[q] = f[q] - h[q];
              }
              val = pack8_bf16(c >= 4 ? l : h);
            }
          }
          *reinterpret_cast<uint4*>(X + i * 128 + ((c ^ (i & 7)) << 4)) = val;
        }
        const int used = n_units << p.lg_box;  // K rows of W per half that B fills
        if (used < kBK / 2) {
          const int per_half = (kBK / 2 - used) * 8;
          for (int e = etid; e < 2 * per_half * kWBoxes; e += kEpiThreads) {
            const int hb = e / (2 * per_half), rem = e % (2 * per_half);
            const int half = rem / per_half, rr = rem % per_half;
            *reinterpret_cast<uint4*>(Wr + hb * L.w_box + (half * (kBK / 2) + used + rr / 8) * 128 +
                                      (rr % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&lora_built[st]);
      }
    }
    const bool acc_ok = warp_wait(accum_full, 0, abort_f);
    if (acc_ok && S == 1) {
      // no split: each thread rounds its token row to bf16 straight from
      // TMEM into a 128-byte-swizzled tile in the drained ring (64-column
      // boxes of 128 rows), and four TMA stores write y (clipped at T, d_out)
      ptx::tc_fence_after();
      const int q = warp & 3;
      const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
      const int i = q * 32 + lane;
#pragma unroll 1
      for (int h = 0; h < kUmmaN / 64; ++h) {
        uint8_t* box = smem + h * (BT * 128);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t v[16];
          ptx::tmem_ld16(tq + h * 64 + c0, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int ch = (c0 >> 3) + u;  // 16-byte chunk of the 128-byte row
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1]));
            pk.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3]));
            pk.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5]));
            pk.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7]));
            *reinterpret_cast<uint4*>(box + i * 128 + ((ch ^ (i & 7)) << 4)) = pk;
          }
        }
      }
      ptx::fence_proxy_async_smem();
      epi_sync();
      if (etid == 0) {
#pragma unroll
        for (int h = 0; h < kUmmaN / 64; ++h)
          if (n0 + 64 * h < p.d_out) ptx::tma_store_2d(&tm_y, smem + h * (BT * 128), n0 + 64 * h, t0);
        ptx::bulk_commit_group();
        ptx::bulk_wait_group_read_all();  // the tile must outlive the read
      }
    } else if (acc_ok) {
      ptx::tc_fence_after();
      const int q = warp & 3;  // TMEM lanes 32q..32q+31 belong to this warp
      const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
      // the fp32 tile is staged token-major in the drained ring for the
      // split-K reduction
      float* red = reinterpret_cast<float*>(smem);
#pragma unroll 1
      for (int c0 = 0; c0 < kUmmaN; c0 += 16) {
        uint32_t v[16];
        ptx::tmem_ld16(tq + c0, v);
        ptx::tmem_ld_wait();
        const int i = q * 32 + lane;  // TMEM lane = token, column = d_out column
        float4* dst = reinterpret_cast<float4*>(red + i * kRedLd + c0);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                               __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
      }
    }
  }

  // ---- split-K reduction, store y ------------------------------------------
  if (S > 1) ptx::cluster_sync();
  else __syncthreads();
  if (!*abort_f) {
    const int rows = min(BT, p.T - t0);
    const int rb0 = static_cast<int>(static_cast<long long>(z) * rows / S);
    const int rb1 = static_cast<int>(static_cast<long long>(z + 1) * rows / S);
    constexpr int kChunks = BN / 8;
    const uint32_t red_s = ptx::smem_u32(smem);
    const int n_items = S == 1 ? 0 : (rb1 - rb0) * kChunks;
    // two output chunks per pass: every load of both is issued before any sum
    for (int e0 = tid; e0 < n_items; e0 += 2 * kThreads) {
      float4 va[2][8], vb[2][8];
      int ii[2], nn[2];
      bool on[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = e0 + u * kThreads;
        ii[u] = rb0 + e / kChunks;
        nn[u] = n0 + (e % kChunks) * 8;
        on[u] = e < n_items && nn[u] < p.d_out;
        if (on[u]) {
          const uint32_t off = static_cast<uint32_t>((ii[u] * kRedLd + (nn[u] - n0)) * 4);
#pragma unroll
          for (int rk = 0; rk < 8; ++rk) {
            if (rk < S) {
              const uint32_t ra =
                  S > 1 ? ptx::mapa_shared(red_s + off, static_cast<uint32_t>(rk)) : red_s + off;
              va[u][rk] = ptx::ld_dsmem_f4(ra);
              vb[u][rk] = ptx::ld_dsmem_f4(ra + 16);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (!on[u]) continue;
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int rk = 0; rk < 8; ++rk) {
          if (rk < S) {
            f[0] += va[u][rk].x; f[1] += va[u][rk].y; f[2] += va[u][rk].z; f[3] += va[u][rk].w;
            f[4] += vb[u][rk].x; f[5] += vb[u][rk].y; f[6] += vb[u][rk].z; f[7] += vb[u][rk].w;
          }
        }
        store8(p.y + static_cast<size_t>(t0 + ii[u]) * p.d_out + nn[u], f);
      }
    }
  }
  if (S > 1) ptx::cluster_sync();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_f) flag_error(p.err, LORA_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------- persistent form
// The same tile computation for unsplit tiles (S = 1), one CTA per SM looping
// over tiles: two accumulators in tensor memory, so the epilogue warps drain
// tile k - 1 (bf16 through a 16 KB swizzled box and TMA stores) while the MMA
// issuer already accumulates tile k, and the ring, the LoRA-stage mailbox and
// every barrier phase run on across tiles.  The per-tile prologue (TMEM
// allocation, barrier set-up, the first loads) and epilogue are paid once or
// hidden behind the next tile's main loop.
struct PersistLayout {
  uint32_t x_sub, x_bytes, w_box, stage_bytes;
  uint32_t tok, uniq, bitmap, ybox, bars, misc, total;
};

template <int BT, int BN, int KS>
__host__ __device__ inline PersistLayout persist_layout(int stages, int n_slots) {
  PersistLayout L;
  L.x_sub = BT * 128;
  L.x_bytes = KS * L.x_sub;
  L.w_box = KS * 8192;
  L.stage_bytes = L.x_bytes + (BN / 64) * L.w_box;
  uint32_t o = static_cast<uint32_t>(stages) * L.stage_bytes;
  L.ybox = o;  // one 64-column bf16 box of the tile, 128-byte swizzle
  o += BT * 128;
  // v rows are read from the shrink's partials when a LoRA stage is built
  L.tok = o;
  o += BT * 4;
  L.uniq = o;
  o += BT * 4;
  L.bitmap = o;
  o += ((n_slots + 31) / 32) * 4;
  o = (o + 7u) & ~7u;
  L.bars = o;
  // full, empty, lora_built per stage; one unused; acc_full[2]; acc_empty[2]
  o += (3 * stages + 5) * 8;
  L.misc = o;
  o += 160;  // as the one-tile kernel, then per-tile LoRA group and unit counts (4 tiles), vt_seq
  L.total = o;
  return L;
}

struct PersistParams {
  TcParams t;
  int tiles_n, tiles_tp, n_tiles;  // tiles_tp: rows of tiles along the tokens
};

template <int BT, int BN, int KS>
__global__ void __launch_bounds__(kThreads, 1)
    fused_tc_persistent_kernel(const __grid_constant__ CUtensorMap tm_x,
                               const __grid_constant__ CUtensorMap tm_w,
                               const __grid_constant__ CUtensorMap tm_b,
                               const __grid_constant__ CUtensorMap tm_y, const PersistParams pp) {
  const TcParams& p = pp.t;
  constexpr int kUmmaN = BN;
  constexpr int kTmemCols = 2 * BN;  // two accumulators
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, kUmmaN, false, true);
  constexpr int kWBoxes = BN / 64;
  static_assert(BT == 128 && BN == 256, "persistent tile: 128 tokens x 256 columns");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const PersistLayout L = persist_layout<BT, BN, KS>(p.stages, p.n_slots);
  int* tok = reinterpret_cast<int*>(smem + L.tok);
  int* uniq = reinterpret_cast<int*>(smem + L.uniq);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L.bitmap);
  uint8_t* ybox = smem + L.ybox;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + p.stages;
  uint64_t* lora_built = empty + p.stages;
  uint64_t* acc_full = lora_built + p.stages + 1;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  int* n_uniq_s = reinterpret_cast<int*>(smem + L.misc + 4);
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + L.misc + 8);
  volatile int* lora_posted = reinterpret_cast<volatile int*>(smem + L.misc + 12);
  uint8_t* stage_kblocks = smem + L.misc + 16;
  uint8_t* stage_lora = smem + L.misc + 32;
  int* lora_mailbox = reinterpret_cast<int*>(smem + L.misc + 48);
  // per tile (k & 3): its LoRA groups and units, written by the epilogue warps
  // before they publish tile k (vt_seq).  Entry k & 3 is rewritten for tile
  // k + 4 only after tile k + 2's accumulator is full, so after the producer
  // (which reads tile k's counts before it loads tile k + 1) and the MMA
  // issuer have read it; two entries would not be enough when a tile without
  // adapters lets the epilogue warps run ahead
  int* tile_groups = reinterpret_cast<int*>(smem + L.misc + 112);
  int* tile_units = tile_groups + 4;
  // tiles whose adapter list and counts are published (monotonic: unlike a
  // barrier's phase parity it cannot alias when the epilogue warps run a tile
  // ahead of the producer or the MMA issuer)
  volatile int* vt_seq = reinterpret_cast<volatile int*>(tile_groups + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // tile lin -> (n0, t0) in the panel order of the one-tile kernel
  auto tile_origin = [&](int lin, int* n0, int* t0) {
    const int g = lin / (kPanel * pp.tiles_tp);
    const int gn = min(kPanel, pp.tiles_n - g * kPanel);
    const int rem = lin - g * kPanel * pp.tiles_tp;
    *n0 = (g * kPanel + rem % gn) * BN;
    *t0 = (rem / gn) * BT;
  };
  const int first_tile = static_cast<int>(blockIdx.x), tile_step = static_cast<int>(gridDim.x);

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_x);
      ptx::prefetch_tmap(&tm_w);
      ptx::prefetch_tmap(&tm_b);
      ptx::prefetch_tmap(&tm_y);
      for (int i = 0; i < p.stages; ++i) {
        ptx::mbar_init(&full[i], 1);
        ptx::mbar_init(&empty[i], 1);
        ptx::mbar_init(&lora_built[i], kEpiThreads / 32);
      }
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(&acc_full[i], 1);
        ptx::mbar_init(&acc_empty[i], kEpiThreads / 32);
      }
      *abort_f = 0;
      *lora_posted = 0;
      *vt_seq = 0;
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
  const int upa = p.r >> p.lg_box;
  const int G = (kBK / 2) >> p.lg_box;
  const int nbase = p.n_kblk;
  // one thread waits (bounded) until tile k is published
  auto seq_wait = [&](int k) {
    const uint64_t tw = ptx::globaltimer_ns();
    while (*vt_seq <= k) {
      if (*abort_f) return false;
      if (ptx::globaltimer_ns() - tw > kWaitLimitNs) {
        *abort_f = 1;
        return false;
      }
    }
    __threadfence_block();
    return true;
  };

  if (warp == 0) {
    // ---------------- producer -------------------------------------------
    int it = 0, g_run = 0;  // ring position; LoRA stages posted so far
    bool ok = true;
    // a tile's LoRA stages follow this base stage (the same place in every
    // tile)
    const int ins = nbase > 1 ? 1 : 0;
    for (int lin = first_tile, k = 0; lin < pp.n_tiles && ok; lin += tile_step, ++k) {
      int n0, t0;
      tile_origin(lin, &n0, &t0);
      int U = 0, my_groups = 0, gi = 0;
      auto next_slot = [&](int* st) {
        *st = it % p.stages;
        const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
        return warp_wait(&empty[*st], ph ^ 1u, abort_f);
      };
      auto issue_lora = [&](int st) {
        uint8_t* Wr = smem + static_cast<size_t>(st) * L.stage_bytes + L.x_bytes;
        const int u_first = gi * G;
        const int n_units = min(G, U - u_first);
        // the B rows' coordinates are read from the tile's adapter list before
        // the stage is posted: once the epilogue warps have built the tile's
        // last LoRA stage they may rewrite the list for the next tile
        const bool loads = lane < 2 * n_units * kWBoxes;
        int a = 0, hb = 0, half = 0, u = 0, qb = 0;
        if (loads) {
          u = lane / (2 * kWBoxes);
          const int rem = lane % (2 * kWBoxes);
          hb = rem >> 1;
          half = rem & 1;
          const int wv = u_first + u;
          a = uniq[wv >> p.lg_upa];
          qb = (wv & (upa - 1)) << p.lg_box;
        }
        __syncwarp();
        if (lane == 0) {
          stage_kblocks[st] = 1;
          stage_lora[st] = 1;
          lora_mailbox[g_run & 15] = st;
          __threadfence_block();
          *lora_posted = g_run + 1;
          ptx::mbar_arrive_expect_tx(
              &full[st], static_cast<uint32_t>(2 * n_units * p.box_rows * 128 * kWBoxes));
        }
        __syncwarp();
        if (loads)
          ptx::tma_load_2d(Wr + hb * L.w_box + (half * (kBK / 2) + u * p.box_rows) * 128, &tm_b,
                           &full[st], n0 + 64 * hb, a * p.r + qb);
        __syncwarp();
        ++gi;
        ++g_run;
      };
      for (int b = 0; b < nbase && ok; ++b) {
        int st;
        if (!(ok = next_slot(&st))) break;
        uint8_t* X = smem + static_cast<size_t>(st) * L.stage_bytes;
        if (lane == 0) {
          stage_kblocks[st] = KS;
          stage_lora[st] = 0;
          ptx::mbar_arrive_expect_tx(&full[st], L.stage_bytes);
#pragma unroll
          for (int j = 0; j < KS; ++j)
            ptx::tma_load_2d(X + j * L.x_sub, &tm_x, &full[st], (b * KS + j) * kBK, t0);
#pragma unroll
          for (int h = 0; h < kWBoxes; ++h)
            ptx::tma_load_2d(X + L.x_bytes + h * L.w_box, &tm_w, &full[st], n0 + 64 * h,
                             b * KS * kBK);
        }
        __syncwarp();
        ++it;
        if (b == ins) {
          int got = 0, cu = 0, cg = 0;
          if (lane == 0 && seq_wait(k)) {
            got = 1;
            cu = tile_units[k & 3];
            cg = tile_groups[k & 3];
          }
          ok = __shfl_sync(0xffffffffu, got, 0) != 0;
          U = __shfl_sync(0xffffffffu, cu, 0);
          my_groups = __shfl_sync(0xffffffffu, cg, 0);
          while (ok && gi < my_groups) {
            if (!(ok = next_slot(&st))) break;
            issue_lora(st);
            ++it;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer -----------------------------------------
    if (lane == 0) {
      uint32_t lora_par = 0;
      int it = 0;
      bool ok = true;
      for (int lin = first_tile, k = 0; lin < pp.n_tiles && ok; lin += tile_step, ++k) {
        const int b = k & 1;
        // the epilogue has drained this accumulator (tile k - 2)
        if (!ptx::mbar_wait_bounded(&acc_empty[b], (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u,
                                    abort_f, kWaitLimitNs))
          break;
        ptx::tc_fence_after();
        const uint32_t acc = tmem + static_cast<uint32_t>(b * BN);
        int local = 0;  // stages of this tile consumed so far
        auto consume = [&]() {
          const int st = it % p.stages;
          const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
          if (!ptx::mbar_wait_bounded(&full[st], ph, abort_f, kWaitLimitNs)) return false;
          if (stage_lora[st]) {
            if (!ptx::mbar_wait_bounded(&lora_built[st], (lora_par >> st) & 1u, abort_f,
                                        kWaitLimitNs))
              return false;
            lora_par ^= 1u << st;
          }
          ptx::tc_fence_after();
          const uint32_t xa = ptx::smem_u32(smem + static_cast<size_t>(st) * L.stage_bytes);
          const uint32_t wa = xa + L.x_bytes;
          const int nkb = stage_kblocks[st];
#pragma unroll
          for (int j = 0; j < KS; ++j) {
            if (j >= nkb) break;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint64_t xd = ptx::sdesc_sw128(xa + j * L.x_sub + kk * 32, 16, 1024);
              const uint64_t wd =
                  ptx::sdesc_sw128(wa + (j * kBK + kk * 16) * 128, L.w_box, 1024);
              ptx::mma_bf16(acc, xd, wd, kIdesc, (local > 0 || j > 0 || kk > 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit(&empty[st]);
          ++it;
          ++local;
          return true;
        };
        // the tile's stages: nbase base stages with its LoRA stages among them
        for (int s = 0; s < nbase && ok; ++s) ok = consume();
        if (ok && seq_wait(k)) {
          const int my_groups = tile_groups[k & 3];
          for (int g = 0; g < my_groups && ok; ++g) ok = consume();
        } else {
          ok = false;
        }
        ptx::mma_commit(&acc_full[b]);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps -------------------------------------
    const int etid = tid - 64;
    const int n_words = (p.n_slots + 31) >> 5;
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int i = q * 32 + lane;  // this thread's token row of the tile (== etid here)
    int g_run = 0;                // LoRA stages built so far
    // drain accumulator b of tile kk into y.  Every epilogue thread runs the
    // same sequence of named barriers whatever happens: after an abort the
    // work is skipped, never the barriers (waits then return at once)
    auto drain = [&](int kk, int n0, int t0) {
      const int b = kk & 1;
      warp_wait(&acc_full[b], static_cast<uint32_t>(kk >> 1) & 1u, abort_f);
      ptx::tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < kUmmaN / 64; ++h) {
        // the staging box is free once the previous TMA store has read it
        if (etid == 0) ptx::bulk_wait_group_read_all();
        epi_sync();
        // warp-uniform: the TMEM loads are warp-collective
        const bool live = __shfl_sync(0xffffffffu, *abort_f == 0 ? 1 : 0, 0) != 0;
        if (live) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 16) {
            uint32_t v[16];
            ptx::tmem_ld16(tmem + lane_base + b * BN + h * 64 + c0, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int ch = (c0 >> 3) + u;
              uint4 pk;
              pk.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1]));
              pk.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3]));
              pk.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5]));
              pk.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7]));
              *reinterpret_cast<uint4*>(ybox + i * 128 + ((ch ^ (i & 7)) << 4)) = pk;
            }
          }
        }
        ptx::fence_proxy_async_smem();
        epi_sync();
        if (etid == 0 && live) {
          if (n0 + 64 * h < p.d_out) ptx::tma_store_2d(&tm_y, ybox, n0 + 64 * h, t0);
          ptx::bulk_commit_group();
        }
      }
      // every TMEM load of this accumulator has completed (tmem_ld_wait)
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[b]);
    };
    int k = 0;
    int prev_n0 = 0, prev_t0 = 0;
    for (int lin = first_tile; lin < pp.n_tiles; lin += tile_step, ++k) {
      int n0, t0;
      tile_origin(lin, &n0, &t0);
      // ---- this tile's adapters (while the previous tile still streams)
      bool bad = false;
      {
        const int t = t0 + i;
        int sl = -1;
        if (t < p.T) {
          const int id = p.ids[t];
          if (slot_valid(id, p.n_slots)) sl = id;
          else if (id != -1) bad = true;
        }
        tok[i] = sl;
      }
      for (int wd = etid; wd < n_words; wd += kEpiThreads) bitmap[wd] = 0u;
      if (bad && n0 == 0) flag_error(p.err, LORA_DEVERR_BAD_SLOT);
      epi_sync();
      if (tok[i] >= 0) atomicOr(&bitmap[tok[i] >> 5], 1u << (tok[i] & 31));
      epi_sync();
      if (warp == 2) {
        const int per = (n_words + 31) / 32;
        const int w0 = min(n_words, lane * per), w1 = min(n_words, w0 + per);
        int cnt = 0;
        for (int wd = w0; wd < w1; ++wd) cnt += __popc(bitmap[wd]);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int vv = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += vv;
        }
        int off = incl - cnt;
        for (int wd = w0; wd < w1; ++wd) {
          uint32_t m = bitmap[wd];
          while (m) {
            const int bb = __ffs(m) - 1;
            m &= m - 1;
            uniq[off++] = wd * 32 + bb;
          }
        }
        if (lane == 31) *n_uniq_s = incl;
      }
      epi_sync();
      const int n_uniq = *n_uniq_s;
      {
        const int sl = tok[i];
        int u = -1;
        if (sl >= 0) {
          int lo = 0, hi = n_uniq - 1;
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (uniq[mid] < sl) lo = mid + 1;
            else hi = mid;
          }
          u = lo;
        }
        tok[i] = u;
      }
      if (k == 0) pdl_wait();  // v is written by the shrink kernel launched just before
      const int U = n_uniq * upa;
      const int my_groups = (U + G - 1) / G;
      if (etid == 0) {
        tile_units[k & 3] = U;
        tile_groups[k & 3] = my_groups;
      }
      epi_sync();
      if (etid == 0) {
        __threadfence_block();
        *vt_seq = k + 1;  // tile k published
      }
      // ---- this tile's LoRA stages, as the producer posts them early in the
      // tile (the other accumulator, tile k - 1, waits meanwhile)
      for (int g2 = 0; g2 < my_groups; ++g2, ++g_run) {
        if (etid == 0) {
          const uint64_t tw = ptx::globaltimer_ns();
          while (*lora_posted <= g_run) {
            if (*abort_f) break;
            if (ptx::globaltimer_ns() - tw > kWaitLimitNs) {
              *abort_f = 1;
              break;
            }
          }
          __threadfence_block();
        }
        epi_sync();
        if (__shfl_sync(0xffffffffu, *abort_f == 0 ? 1 : 0, 0)) {
          const int st = lora_mailbox[g_run & 15];
          uint8_t* X = smem + static_cast<size_t>(st) * L.stage_bytes;
          uint8_t* Wr = X + L.x_bytes;
          const int u_first = g2 * G;
          const int n_units = min(G, U - u_first);
          const int tv = tok[i];
          // v[t, q0 .. q0+8) for each 8-column chunk of the stage's first half,
          // summed over the shrink's d_in splits (this thread's row only: the
          // values come from L2, with every load issued before any is used)
          const size_t row = static_cast<size_t>(t0 + i) * p.r;
          const size_t split = static_cast<size_t>(p.T) * p.r;
          int q0[4];
          float f[4][8];
#pragma unroll
          for (int cq = 0; cq < 4; ++cq) {
            const int kq = cq << 3;
            const int wu = kq >> p.lg_box;
            const int w = u_first + wu;
            q0[cq] = (wu < n_units && tv >= 0 && (w >> p.lg_upa) == tv)
                         ? ((w & (upa - 1)) << p.lg_box) + (kq & (p.box_rows - 1))
                         : -1;
#pragma unroll
            for (int c = 0; c < 8; ++c) f[cq][c] = 0.f;
          }
          for (int s0 = 0; s0 < p.v_ksplit; ++s0) {
            float g[4][8];
#pragma unroll
            for (int cq = 0; cq < 4; ++cq)
              if (q0[cq] >= 0) load8_dep(p.vpart + s0 * split + row + q0[cq], g[cq]);
#pragma unroll
            for (int cq = 0; cq < 4; ++cq)
              if (q0[cq] >= 0)
#pragma unroll
                for (int c = 0; c < 8; ++c) f[cq][c] += g[cq][c];
          }
#pragma unroll
          for (int cq = 0; cq < 4; ++cq) {
            float hh[8], ll[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              hh[c] = __bfloat162float(__float2bfloat16_rn(f[cq][c]));
              ll[c] = f[cq][c] - hh[c];
            }
            // a chunk with no matching unit is all zeros (f stayed 0)
            *reinterpret_cast<uint4*>(X + i * 128 + ((cq ^ (i & 7)) << 4)) = pack8_bf16(hh);
            *reinterpret_cast<uint4*>(X + i * 128 + (((cq + 4) ^ (i & 7)) << 4)) = pack8_bf16(ll);
          }
          const int used = n_units << p.lg_box;
          if (used < kBK / 2) {
            // B rows past the stage's units: no TMA writes them
            const int per_half = (kBK / 2 - used) * 8;
            for (int e = etid; e < 2 * per_half * kWBoxes; e += kEpiThreads) {
              const int hb = e / (2 * per_half), rem = e % (2 * per_half);
              const int half = rem / per_half, rr = rem % per_half;
              *reinterpret_cast<uint4*>(Wr + hb * L.w_box + (half * (kBK / 2) + used + rr / 8) * 128 +
                                        (rr % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&lora_built[st]);
        }
      }
      // ---- the previous tile's accumulator, while this tile streams
      if (k > 0) drain(k - 1, prev_n0, prev_t0);
      prev_n0 = n0;
      prev_t0 = t0;
    }
    // the last tile
    if (k > 0) drain(k - 1, prev_n0, prev_t0);
    if (etid == 0) ptx::bulk_wait_group_read_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_f) flag_error(p.err, LORA_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------- wide form
// Persistent walk over tiles of 256 tokens x 256 columns.  Each 64-deep
// stage brings x for the tile's two 128-token halves (32 KB) and one W0 slab
// (32 KB), and the two M = 128 MMAs of a 16-deep step share the W0 operand.
// An SM then takes in 64 KB of operands per 8.4 MFLOP instead of the 96 KB of
// a 128 x 256 tile, and that intake, not the tensor pipe, is what bounds the
// narrower tile's main loop (at the same L2 hit rate; a CTA pair that shared
// each W0 box, tried before, cut L2 reads without speeding it up).  The two accumulators fill
// all 512 TMEM columns, so a tile is drained before the next one starts; eight
// epilogue warps (two per TMEM lane quarter, one per 128-column half), each
// with its own 4 KB store box, keep that drain short.
constexpr int kWideThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kWideEpi = 256;

__device__ __forceinline__ void wide_epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWideEpi) : "memory");
}

struct WideLayout {
  uint32_t x_sub, w_off, w_box, stage_bytes;
  uint32_t ybox, tok, uniq, bitmap, bars, misc, total;
};

__host__ __device__ inline WideLayout wide_layout(int stages, int n_slots) {
  WideLayout L;
  L.x_sub = 128 * 128;  // 128 tokens x 64 K of bf16, 128-byte swizzle
  L.w_off = 2 * L.x_sub;
  L.w_box = kBK * 128;  // 64 K rows x 64 columns
  L.stage_bytes = L.w_off + 4 * L.w_box;
  uint32_t o = static_cast<uint32_t>(stages) * L.stage_bytes;
  L.ybox = o;  // per epilogue warp: 32 rows x 64 columns of bf16
  o += 8 * 4096;
  L.tok = o;  // int16 per token of the tile
  o += 256 * 2;
  L.uniq = o;  // int16 per distinct adapter of the tile
  o += 256 * 2;
  L.bitmap = o;
  o += ((n_slots + 31) / 32) * 4;
  o = (o + 7u) & ~7u;
  L.bars = o;  // full, empty, lora_built per stage; acc_full; acc_empty
  o += (3 * stages + 2) * 8;
  L.misc = o;
  o += 160;
  L.total = o;
  return L;
}

__global__ void __launch_bounds__(kWideThreads, 1)
    fused_tc_wide_kernel(const __grid_constant__ CUtensorMap tm_x,
                         const __grid_constant__ CUtensorMap tm_w,
                         const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_y, const PersistParams pp) {
  const TcParams& p = pp.t;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 256, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const WideLayout L = wide_layout(p.stages, p.n_slots);
  int16_t* tok = reinterpret_cast<int16_t*>(smem + L.tok);
  int16_t* uniq = reinterpret_cast<int16_t*>(smem + L.uniq);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L.bitmap);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + p.stages;
  uint64_t* lora_built = empty + p.stages;
  uint64_t* acc_full = lora_built + p.stages;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  int* n_uniq_s = reinterpret_cast<int*>(smem + L.misc + 4);
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + L.misc + 8);
  volatile int* lora_posted = reinterpret_cast<volatile int*>(smem + L.misc + 12);
  uint8_t* stage_lora = smem + L.misc + 32;
  int* lora_mailbox = reinterpret_cast<int*>(smem + L.misc + 48);
  // per tile (k & 3): LoRA groups and units; entry k & 3 is rewritten for
  // tile k + 4 only after tile k + 3's LoRA stages were posted and tile
  // k + 2's accumulators drained, so after the producer and the MMA issuer
  // have read it
  int* tile_groups = reinterpret_cast<int*>(smem + L.misc + 112);
  int* tile_units = tile_groups + 4;
  volatile int* vt_seq = reinterpret_cast<volatile int*>(tile_groups + 8);  // tiles published

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int first_tile = static_cast<int>(blockIdx.x), tile_step = static_cast<int>(gridDim.x);
  // Tile order.  CTA b takes positions b, b + gridDim.x, ...; the first
  // `extra` CTAs also take one of the last, partial round.  A tile row far
  // heavier in LoRA stages than the others (many adapter runs, as where a
  // mixed batch's decode tokens sit) is placed at positions [extra, extra +
  // tiles_n), on CTAs without a tile in that last round; every other tile
  // keeps the panel order (kPanel column tiles per panel).
  int heavy = -1;
  auto tile_origin = [&](int lin, int* n0, int* t0) {
    if (heavy >= 0) {
      const int extra = pp.n_tiles % tile_step;
      if (lin >= extra && lin < extra + pp.tiles_n) {
        *n0 = (lin - extra) * 256;
        *t0 = heavy * 256;
        return;
      }
      const int j = lin < extra ? lin : lin - pp.tiles_n;  // among the other rows' tiles
      const int rows = pp.tiles_tp - 1;
      const int g = j / (kPanel * rows);
      const int gn = min(kPanel, pp.tiles_n - g * kPanel);
      const int rem = j - g * kPanel * rows;
      const int row = rem / gn;
      *n0 = (g * kPanel + rem % gn) * 256;
      *t0 = (row < heavy ? row : row + 1) * 256;
      return;
    }
    const int g = lin / (kPanel * pp.tiles_tp);
    const int gn = min(kPanel, pp.tiles_n - g * kPanel);
    const int rem = lin - g * kPanel * pp.tiles_tp;
    *n0 = (g * kPanel + rem % gn) * 256;
    *t0 = (rem / gn) * 256;
  };

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_x);
      ptx::prefetch_tmap(&tm_w);
      ptx::prefetch_tmap(&tm_b);
      ptx::prefetch_tmap(&tm_y);
      for (int i = 0; i < p.stages; ++i) {
        ptx::mbar_init(&full[i], 1);
        ptx::mbar_init(&empty[i], 1);
        ptx::mbar_init(&lora_built[i], kWideEpi / 32);
      }
      ptx::mbar_init(acc_full, 1);
      ptx::mbar_init(acc_empty, kWideEpi / 32);
      *abort_f = 0;
      *lora_posted = 0;
      *vt_seq = 0;
      ptx::fence_mbar_init();
    }
    __syncwarp();
    named_arrive(2, kWideThreads);
  } else {
    named_sync(2, kWideThreads);
    if (warp == 1) {
      ptx::tmem_alloc(tmem_slot, 512);
      ptx::tmem_relinquish();
      ptx::tc_fence_before();
      named_arrive(3, kWideThreads - 32);
    } else {
      named_sync(3, kWideThreads - 32);
    }
    ptx::tc_fence_after();
  }
  {
    // adapter runs per tile row, counted by the whole CTA in the store boxes
    // (unused until the first drain); ids were written before the kernel
    // ahead of this one started, so they are read before its wait
    int* row_runs = reinterpret_cast<int*>(smem + L.ybox);
    volatile int* heavy_s = reinterpret_cast<volatile int*>(smem + L.misc + 152);
    for (int i = tid; i < pp.tiles_tp; i += kWideThreads) row_runs[i] = 0;
    __syncthreads();
#pragma unroll 8
    for (int t = tid; t < p.T; t += kWideThreads) {
      const int id = p.ids[t];
      const int prev = (t & 255) ? p.ids[t - 1] : -1;
      if (slot_valid(id, p.n_slots) && id != prev) atomicAdd(&row_runs[t >> 8], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int best = -1, most = 0, total = 0;
      for (int i = 0; i < pp.tiles_tp; ++i) {
        total += row_runs[i];
        if (row_runs[i] > most) {
          most = row_runs[i];
          best = i;
        }
      }
      // at least 8 runs and four times the other rows' average, and room
      // for its tiles beside the CTAs of the last round
      const int extra = pp.n_tiles % tile_step;
      const bool move = best >= 0 && pp.tiles_tp > 1 && pp.n_tiles > tile_step &&
                        extra + pp.tiles_n <= tile_step && most >= 8 &&
                        most * (pp.tiles_tp - 1) >= 4 * (total - most);
      *heavy_s = move ? best : -1;
    }
    __syncthreads();
    heavy = *heavy_s;
  }
  const uint32_t tmem = warp == 0 ? 0u : *tmem_slot;
  const int upa = p.r >> p.lg_box;
  const int G = (kBK / 2) >> p.lg_box;
  const int nbase = p.n_kblk;
  auto seq_wait = [&](int k) {
    const uint64_t tw = ptx::globaltimer_ns();
    while (*vt_seq <= k) {
      if (*abort_f) return false;
      if (ptx::globaltimer_ns() - tw > kWaitLimitNs) {
        *abort_f = 1;
        return false;
      }
    }
    __threadfence_block();
    return true;
  };

  if (warp == 0) {
    // ---------------- producer -------------------------------------------
    int it = 0, g_run = 0;
    bool ok = true;
    // a tile's LoRA stages start after its second base stage and are spread
    // over the next `span` base stages, so that their B loads and V builds
    // overlap base-stage MMAs; the last is posted about eight stages before
    // the tile ends, which leaves the epilogue warps time to publish the next
    // tile's adapters
    const int ins = nbase > 1 ? 1 : nbase - 1;
    const int span = nbase - ins - 8 > 1 ? nbase - ins - 8 : 1;
    for (int lin = first_tile, k = 0; lin < pp.n_tiles && ok; lin += tile_step, ++k) {
      int n0, t0;
      tile_origin(lin, &n0, &t0);
      int U = 0, my_groups = 0, gi = 0;
      auto next_slot = [&](int* st) {
        *st = it % p.stages;
        const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
        return warp_wait(&empty[*st], ph ^ 1u, abort_f);
      };
      auto issue_lora = [&](int st) {
        uint8_t* Wr = smem + static_cast<size_t>(st) * L.stage_bytes + L.w_off;
        const int u_first = gi * G;
        const int n_units = min(G, U - u_first);
        const bool loads = lane < 2 * n_units * 4;
        int a = 0, hb = 0, half = 0, u = 0, qb = 0;
        if (loads) {
          u = lane >> 3;
          hb = (lane & 7) >> 1;
          half = lane & 1;
          const int wv = u_first + u;
          a = uniq[wv >> p.lg_upa];
          qb = (wv & (upa - 1)) << p.lg_box;
        }
        __syncwarp();
        if (lane == 0) {
          stage_lora[st] = 1;
          lora_mailbox[g_run & 15] = st;
          __threadfence_block();
          *lora_posted = g_run + 1;
          ptx::mbar_arrive_expect_tx(&full[st],
                                     static_cast<uint32_t>(2 * n_units * p.box_rows * 128 * 4));
        }
        __syncwarp();
        if (loads)
          ptx::tma_load_2d(Wr + hb * L.w_box + (half * (kBK / 2) + u * p.box_rows) * 128, &tm_b,
                           &full[st], n0 + 64 * hb, a * p.r + qb);
        __syncwarp();
        ++gi;
        ++g_run;
      };
      for (int b = 0; b < nbase && ok; ++b) {
        int st;
        if (!(ok = next_slot(&st))) break;
        uint8_t* X = smem + static_cast<size_t>(st) * L.stage_bytes;
        if (lane == 0) {
          stage_lora[st] = 0;
          ptx::mbar_arrive_expect_tx(&full[st], L.stage_bytes);
          ptx::tma_load_2d(X, &tm_x, &full[st], b * kBK, t0);
          ptx::tma_load_2d(X + L.x_sub, &tm_x, &full[st], b * kBK, t0 + 128);
#pragma unroll
          for (int h = 0; h < 4; ++h)
            ptx::tma_load_2d(X + L.w_off + h * L.w_box, &tm_w, &full[st], n0 + 64 * h, b * kBK);
        }
        __syncwarp();
        ++it;
        if (b == ins) {
          int got = 0, cu = 0, cg = 0;
          if (lane == 0 && seq_wait(k)) {
            got = 1;
            cu = tile_units[k & 3];
            cg = tile_groups[k & 3];
          }
          ok = __shfl_sync(0xffffffffu, got, 0) != 0;
          U = __shfl_sync(0xffffffffu, cu, 0);
          my_groups = __shfl_sync(0xffffffffu, cg, 0);
        }
        if (b >= ins) {
          // groups due after base stage b: ceil((b - ins + 1) * groups / span)
          const int due = min(my_groups, ((b - ins + 1) * my_groups + span - 1) / span);
          while (ok && gi < due) {
            if (!(ok = next_slot(&st))) break;
            issue_lora(st);
            ++it;
          }
        }
      }
      while (ok && gi < my_groups) {
        int st;
        if (!(ok = next_slot(&st))) break;
        issue_lora(st);
        ++it;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer -----------------------------------------
    if (lane == 0) {
      uint32_t lora_par = 0;
      int it = 0;
      bool ok = true;
      for (int lin = first_tile, k = 0; lin < pp.n_tiles && ok; lin += tile_step, ++k) {
        // both accumulators drained (tile k - 1)
        if (!ptx::mbar_wait_bounded(acc_empty, (static_cast<uint32_t>(k) & 1u) ^ 1u, abort_f,
                                    kWaitLimitNs))
          break;
        ptx::tc_fence_after();
        int local = 0;
        auto consume = [&]() {
          const int st = it % p.stages;
          const uint32_t ph = static_cast<uint32_t>(it / p.stages) & 1u;
          if (!ptx::mbar_wait_bounded(&full[st], ph, abort_f, kWaitLimitNs)) return false;
          if (stage_lora[st]) {
            if (!ptx::mbar_wait_bounded(&lora_built[st], (lora_par >> st) & 1u, abort_f,
                                        kWaitLimitNs))
              return false;
            lora_par ^= 1u << st;
          }
          ptx::tc_fence_after();
          const uint32_t xa = ptx::smem_u32(smem + static_cast<size_t>(st) * L.stage_bytes);
          const uint32_t wa = xa + L.w_off;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t wd = ptx::sdesc_sw128(wa + kk * 16 * 128, L.w_box, 1024);
            const uint64_t x0 = ptx::sdesc_sw128(xa + kk * 32, 16, 1024);
            const uint64_t x1 = ptx::sdesc_sw128(xa + L.x_sub + kk * 32, 16, 1024);
            const uint32_t acc_in = (local > 0 || kk > 0) ? 1u : 0u;
            ptx::mma_bf16(tmem, x0, wd, kIdesc, acc_in);
            ptx::mma_bf16(tmem + 256u, x1, wd, kIdesc, acc_in);
          }
          ptx::mma_commit(&empty[st]);
          ++it;
          ++local;
          return true;
        };
        for (int s = 0; s < nbase && ok; ++s) ok = consume();
        if (ok && seq_wait(k)) {
          const int my_groups = tile_groups[k & 3];
          for (int g = 0; g < my_groups && ok; ++g) ok = consume();
        } else {
          ok = false;
        }
        ptx::mma_commit(acc_full);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps -------------------------------------
    const int etid = tid - 64;
    const int ew = warp - 2;
    const int n_words = (p.n_slots + 31) >> 5;
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const int c = ew >> 2;    // column half it drains; V half it builds
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int i = q * 32 + lane;  // row within a 128-token half
    const int rr = c * 128 + i;   // this thread's token row of the tile
    uint8_t* mybox = smem + L.ybox + ew * 4096;
    int g_run = 0;
    // Both accumulators of tile kk: this warp's 32 rows of each, its 128
    // columns, through its own box.  Every epilogue thread passes the same
    // named barriers whatever happens (only work is skipped after an abort).
    auto drain = [&](int kk, int n0, int t0) {
      warp_wait(acc_full, static_cast<uint32_t>(kk) & 1u, abort_f);
      ptx::tc_fence_after();
      const bool live = __shfl_sync(0xffffffffu, *abort_f == 0 ? 1 : 0, 0) != 0;
#pragma unroll 1
      for (int a = 0; a < 2; ++a) {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          if (lane == 0) ptx::bulk_wait_group_read_all();  // the box is free again
          __syncwarp();
          if (live) {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
              uint32_t v[16];
              ptx::tmem_ld16(tmem + lane_base + a * 256 + c * 128 + h * 64 + c0, v);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int ch = (c0 >> 3) + u;
                uint4 pk;
                pk.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1]));
                pk.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3]));
                pk.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5]));
                pk.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7]));
                *reinterpret_cast<uint4*>(mybox + lane * 128 + ((ch ^ (lane & 7)) << 4)) = pk;
              }
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && live) {
            const int col = n0 + c * 128 + h * 64, row = t0 + a * 128 + q * 32;
            if (col < p.d_out && row < p.T) ptx::tma_store_2d(&tm_y, mybox, col, row);
            ptx::bulk_commit_group();
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(acc_empty);
    };
    int k = 0;
    int prev_n0 = 0, prev_t0 = 0;
    for (int lin = first_tile; lin < pp.n_tiles; lin += tile_step, ++k) {
      int n0, t0;
      tile_origin(lin, &n0, &t0);
      // ---- this tile's adapters (while the previous tile still streams)
      bool bad = false;
      {
        const int t = t0 + rr;
        int sl = -1;
        if (t < p.T) {
          const int id = p.ids[t];
          if (slot_valid(id, p.n_slots)) sl = id;
          else if (id != -1) bad = true;
        }
        tok[rr] = static_cast<int16_t>(sl);
      }
      for (int wd = etid; wd < n_words; wd += kWideEpi) bitmap[wd] = 0u;
      if (bad && n0 == 0) flag_error(p.err, LORA_DEVERR_BAD_SLOT);
      wide_epi_sync();
      if (tok[rr] >= 0) atomicOr(&bitmap[tok[rr] >> 5], 1u << (tok[rr] & 31));
      wide_epi_sync();
      if (warp == 2) {
        const int per = (n_words + 31) / 32;
        const int w0 = min(n_words, lane * per), w1 = min(n_words, w0 + per);
        int cnt = 0;
        for (int wd = w0; wd < w1; ++wd) cnt += __popc(bitmap[wd]);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int vv = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += vv;
        }
        int off = incl - cnt;
        for (int wd = w0; wd < w1; ++wd) {
          uint32_t m = bitmap[wd];
          while (m) {
            const int bb = __ffs(m) - 1;
            m &= m - 1;
            uniq[off++] = static_cast<int16_t>(wd * 32 + bb);
          }
        }
        if (lane == 31) *n_uniq_s = incl;
      }
      wide_epi_sync();
      const int n_uniq = *n_uniq_s;
      {
        const int sl = tok[rr];
        int u = -1;
        if (sl >= 0) {
          int lo = 0, hi = n_uniq - 1;
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (uniq[mid] < sl) lo = mid + 1;
            else hi = mid;
          }
          u = lo;
        }
        tok[rr] = static_cast<int16_t>(u);
      }
      if (k == 0) pdl_wait();  // v is written by the shrink kernel launched just before
      const int U = n_uniq * upa;
      const int my_groups = (U + G - 1) / G;
      if (etid == 0) {
        tile_units[k & 3] = U;
        tile_groups[k & 3] = my_groups;
      }
      wide_epi_sync();
      if (etid == 0) {
        __threadfence_block();
        *vt_seq = k + 1;
      }
      // ---- the previous tile's accumulators: the MMA issuer waits for them
      if (k > 0) drain(k - 1, prev_n0, prev_t0);
      // ---- this tile's LoRA stages.  This thread's units are those of its
      // token's adapter tv (units tv * upa .. tv * upa + upa - 1).  Its v
      // values for the next stage that holds one of them are loaded ahead
      // (f): the first at the tile's start, each next one as soon as the
      // last is written.
      const int tv = tok[rr];
      const float* vrow = p.vpart + static_cast<size_t>(t0 + rr) * p.r;
      // chunk cq of stage g: this thread's rank offset in v, or -1
      auto chunk_q0 = [&](int g, int cq) {
        const int kq = cq << 3;
        const int wu = kq >> p.lg_box;
        const int w = g * G + wu;
        return (tv >= 0 && wu < min(G, U - g * G) && (w >> p.lg_upa) == tv)
                   ? ((w & (upa - 1)) << p.lg_box) + (kq & (p.box_rows - 1))
                   : -1;
      };
      float f[4][8];
      int next_part = 0, next_g = -1;  // the stage f is loaded for
      auto load_next = [&]() {
        next_g = -1;
        if (tv < 0 || next_part >= upa) return;
        next_g = (tv * upa + next_part) / G;
        ++next_part;
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) {
          const int q0 = chunk_q0(next_g, cq);
          if (q0 >= 0) load8_dep(vrow + q0, f[cq]);
        }
      };
      load_next();
      for (int g2 = 0; g2 < my_groups; ++g2, ++g_run) {
        if (etid == 0) {
          const uint64_t tw = ptx::globaltimer_ns();
          while (*lora_posted <= g_run) {
            if (*abort_f) break;
            if (ptx::globaltimer_ns() - tw > kWaitLimitNs) {
              *abort_f = 1;
              break;
            }
          }
          __threadfence_block();
        }
        wide_epi_sync();
        if (__shfl_sync(0xffffffffu, *abort_f == 0 ? 1 : 0, 0)) {
          const int st = lora_mailbox[g_run & 15];
          uint8_t* X = smem + static_cast<size_t>(st) * L.stage_bytes;
          uint8_t* Wr = X + L.w_off;
          uint8_t* Xh = X + c * L.x_sub;  // this thread's V half
          const int n_units = min(G, U - g2 * G);
          const bool mine = g2 == next_g;
#pragma unroll
          for (int cq = 0; cq < 4; ++cq) {
            const bool use = mine && chunk_q0(g2, cq) >= 0;
            float hh[8], ll[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float v = use ? f[cq][e] : 0.f;
              hh[e] = __bfloat162float(__float2bfloat16_rn(v));
              ll[e] = v - hh[e];
            }
            *reinterpret_cast<uint4*>(Xh + i * 128 + ((cq ^ (i & 7)) << 4)) = pack8_bf16(hh);
            *reinterpret_cast<uint4*>(Xh + i * 128 + (((cq + 4) ^ (i & 7)) << 4)) = pack8_bf16(ll);
          }
          if (mine) load_next();
          const int used = n_units << p.lg_box;
          if (used < kBK / 2) {
            const int per_half = (kBK / 2 - used) * 8;
            for (int e = etid; e < 2 * per_half * 4; e += kWideEpi) {
              const int hb = e / (2 * per_half), rem = e % (2 * per_half);
              const int half = rem / per_half, r2 = rem % per_half;
              *reinterpret_cast<uint4*>(Wr + hb * L.w_box + (half * (kBK / 2) + used + r2 / 8) * 128 +
                                        (r2 % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&lora_built[st]);
        }
      }
      prev_n0 = n0;
      prev_t0 = t0;
    }
    if (k > 0) drain(k - 1, prev_n0, prev_t0);
    if (lane == 0) ptx::bulk_wait_group_read_all();  // this warp's own stores
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  if (tid == 0 && *abort_f) flag_error(p.err, LORA_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void resolve_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// rows `row_elems` apart; box = box_inner x box_outer, 128-byte swizzle,
// out-of-range elements read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_elems,
              uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_elems * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Deepest pipeline that fits next to the v tile and bookkeeping, and that
// can hold the staged fp32 accumulator afterwards (0: none fits).
template <int BT, int BN, int KS>
int pick_stages(const TcParams& prm, size_t cap) {
  const size_t red_bytes = static_cast<size_t>(BT) * (BN + kRedPad) * 4;
  for (int s = 8; s >= 2; --s) {
    const SmemLayout L = smem_layout<BT, BN, KS>(s, prm.r, prm.n_slots);
    if (L.total + 1024 <= cap && L.stages_total >= red_bytes) return s;
  }
  return 0;
}

template <int BT, int BN, int KS>
cudaError_t launch_variant(const void* x, const void* W0, const void* B, TcParams prm,
                           int tiles_n, int tiles_t, int S, cudaStream_t st,
                           const DeviceInfo& dev) {
  const int stages = pick_stages<BT, BN, KS>(prm, dev.max_smem_optin);
  if (stages == 0) return cudaErrorInvalidConfiguration;
  prm.stages = stages;
  const SmemLayout L = smem_layout<BT, BN, KS>(stages, prm.r, prm.n_slots);
  const size_t smem = L.total + 1024;

  CUtensorMap tm_x, tm_w, tm_b, tm_y;
  if (!make_map(&tm_x, x, prm.d_in, prm.T, prm.d_in, kBK, BT) ||
      !make_map(&tm_w, W0, prm.d_out, prm.d_in, prm.d_out, 64, KS * kBK) ||
      !make_map(&tm_b, B, prm.d_out, static_cast<uint64_t>(prm.n_slots) * prm.r, prm.d_out, 64,
                prm.box_rows) ||
      !make_map(&tm_y, prm.y, prm.d_out, prm.T, prm.d_out, 64, BT))
    return cudaErrorInvalidValue;

  auto kern = fused_tc_kernel<BT, BN, KS>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n * tiles_t, 1, S);
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
  return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_w, tm_b, tm_y, prm);
}

template <int BT, int BN, int KS>
cudaError_t launch_persistent(const void* x, const void* W0, const void* B, TcParams prm,
                              int tiles_n, int tiles_t, cudaStream_t st, const DeviceInfo& dev) {
  int stages = 0;
  for (int s = 8; s >= (KS == 2 ? 2 : 3); --s) {
    const PersistLayout L = persist_layout<BT, BN, KS>(s, prm.n_slots);
    if (L.total + 1024 <= dev.max_smem_optin) {
      stages = s;
      break;
    }
  }
  if (stages == 0) return cudaErrorInvalidConfiguration;
  prm.stages = stages;
  const PersistLayout L = persist_layout<BT, BN, KS>(stages, prm.n_slots);
  const size_t smem = L.total + 1024;

  CUtensorMap tm_x, tm_w, tm_b, tm_y;
  if (!make_map(&tm_x, x, prm.d_in, prm.T, prm.d_in, kBK, BT) ||
      !make_map(&tm_w, W0, prm.d_out, prm.d_in, prm.d_out, 64, KS * kBK) ||
      !make_map(&tm_b, B, prm.d_out, static_cast<uint64_t>(prm.n_slots) * prm.r, prm.d_out, 64,
                prm.box_rows) ||
      !make_map(&tm_y, prm.y, prm.d_out, prm.T, prm.d_out, 64, BT))
    return cudaErrorInvalidValue;
  auto kern = fused_tc_persistent_kernel<BT, BN, KS>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  PersistParams pp;
  pp.t = prm;
  pp.tiles_n = tiles_n;
  pp.tiles_tp = tiles_t;
  pp.n_tiles = tiles_n * tiles_t;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pp.n_tiles < dev.num_sms ? pp.n_tiles : dev.num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_w, tm_b, tm_y, pp);
}

cudaError_t launch_wide(const void* x, const void* W0, const void* B, TcParams prm,
                       int tiles_n, cudaStream_t st, const DeviceInfo& dev) {
  if (prm.n_slots > 32767) return cudaErrorInvalidConfiguration;  // int16 slot lists
  if (prm.v_ksplit != 1) return cudaErrorInvalidConfiguration;    // one v partial
  int stages = 0;
  for (int s = 4; s >= 2; --s) {
    if (wide_layout(s, prm.n_slots).total + 1024 <= dev.max_smem_optin) {
      stages = s;
      break;
    }
  }
  if (stages == 0) return cudaErrorInvalidConfiguration;
  prm.stages = stages;
  prm.n_kblk = (prm.d_in + kBK - 1) / kBK;
  const size_t smem = wide_layout(stages, prm.n_slots).total + 1024;
  CUtensorMap tm_x, tm_w, tm_b, tm_y;
  if (!make_map(&tm_x, x, prm.d_in, prm.T, prm.d_in, kBK, 128) ||
      !make_map(&tm_w, W0, prm.d_out, prm.d_in, prm.d_out, 64, kBK) ||
      !make_map(&tm_b, B, prm.d_out, static_cast<uint64_t>(prm.n_slots) * prm.r, prm.d_out, 64,
                prm.box_rows) ||
      !make_map(&tm_y, prm.y, prm.d_out, prm.T, prm.d_out, 64, 32))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fused_tc_wide_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  PersistParams pp;
  pp.t = prm;
  pp.tiles_n = tiles_n;
  pp.tiles_tp = (prm.T + 255) / 256;
  pp.n_tiles = tiles_n * pp.tiles_tp;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pp.n_tiles < dev.num_sms ? pp.n_tiles : dev.num_sms);
  cfg.blockDim = dim3(kWideThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_tc_wide_kernel, tm_x, tm_w, tm_b, tm_y, pp);
}

}  // namespace

bool encode_tensor_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_elems, uint32_t box_inner, uint32_t box_outer) {
  resolve_encode();
  return g_encode != nullptr && make_map(m, base, inner, outer, row_elems, box_inner, box_outer);
}

bool encode_tensor_map_bf16_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                               uint64_t d2, uint32_t box0, uint32_t box1) {
  resolve_encode();
  if (g_encode == nullptr) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_f32_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                              uint64_t d2, uint32_t box0, uint32_t box1) {
  resolve_encode();
  if (g_encode == nullptr) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_plain_2d(CUtensorMap* m, const void* base, int elem_bytes, uint64_t inner,
                                uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                                uint32_t box_outer) {
  resolve_encode();
  if (g_encode == nullptr || (elem_bytes != 1 && elem_bytes != 2)) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  resolve_encode();
  if (g_encode == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool fused_wide_tiles(int T, int d_out, int n_slots, int num_sms) {
  // at least two waves of 256 x 256 tiles; int16 slot lists
  return T > 256 && n_slots <= 32767 &&
         static_cast<long long>((d_out + 255) / 256) * ((T + 255) / 256) >= 2LL * num_sms;
}

bool tensor_map_available() {
  resolve_encode();
  return g_encode != nullptr;
}

cudaError_t launch_fused_tc(const void* x, const void* W0, const void* B, const int32_t* ids,
                            const float* vpart, int v_ksplit, void* y, int T,
                            int d_in, int d_out, int r, int n_slots, uint32_t* err,
                            cudaStream_t st, const DeviceInfo& dev) {
  resolve_encode();
  if (g_encode == nullptr) return cudaErrorNotSupported;
  TcParams prm;
  prm.T = T;
  prm.d_in = d_in;
  prm.d_out = d_out;
  prm.r = r;
  prm.n_slots = n_slots;
  // two 64-deep K blocks per base stage when the ring still holds two such
  // stages next to the v tile (rank <= 64); one otherwise
  const int KS = pick_stages<128, 256, 2>(prm, dev.max_smem_optin) > 0 ? 2 : 1;
  prm.n_kblk = (d_in + KS * kBK - 1) / (KS * kBK);
  prm.stages = 0;
  prm.box_rows = r < 32 ? r : 32;
  prm.lg_box = 31 - __builtin_clz(static_cast<unsigned>(prm.box_rows));
  prm.lg_upa = 31 - __builtin_clz(static_cast<unsigned>(r / prm.box_rows));
  prm.v_ksplit = v_ksplit;
  prm.ids = ids;
  prm.vpart = vpart;
  prm.y = static_cast<bf16*>(y);
  prm.err = err;

  // split-K cluster size: as many CTAs per tile as fill the SMs, at most 8,
  // a power of two
  auto pick_split = [&](int tiles) {
    int S = dev.num_sms / (tiles > 0 ? tiles : 1);
    if (S > 8) S = 8;
    if (S > prm.n_kblk) S = prm.n_kblk;
    int p2 = 1;
    while (p2 * 2 <= S) p2 *= 2;
    return p2;
  };
  const int tiles_n = (d_out + 255) / 256;
  const int tiles_t = (T + 127) / 128;
  const int S = pick_split(tiles_n * tiles_t);
  if (S == 1) {
    // more tiles than SMs: a persistent form, one CTA per SM walking tiles
    // (v rows come from L2 when a LoRA stage is built).  With at least two
    // waves of 256 x 256 tiles, the wide form: two M = 128 MMAs per step
    // share each W0 stage, and their two accumulators fill tensor memory.
    // Otherwise 128 x 256 tiles with two accumulators, so the drain of one
    // tile overlaps the next tile's main loop.
    cudaError_t e = cudaErrorInvalidConfiguration;
    if (fused_wide_tiles(T, d_out, n_slots, dev.num_sms))
      e = launch_wide(x, W0, B, prm, tiles_n, st, dev);
    if (e != cudaErrorInvalidConfiguration) return e;
    TcParams pp = prm;
    pp.n_kblk = (d_in + 2 * kBK - 1) / (2 * kBK);
    e = launch_persistent<128, 256, 2>(x, W0, B, pp, tiles_n, tiles_t, st, dev);
    if (e != cudaErrorInvalidConfiguration) return e;
  }
  if (KS == 2) return launch_variant<128, 256, 2>(x, W0, B, prm, tiles_n, tiles_t, S, st, dev);
  return launch_variant<128, 256, 1>(x, W0, B, prm, tiles_n, tiles_t, S, st, dev);
}

}  // namespace lora
