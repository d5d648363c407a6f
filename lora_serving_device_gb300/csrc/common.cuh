// Device helpers shared by the liblora kernels: 8-element vector loads and
// stores for bf16 / fp32 storage, and the sticky device error word.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "lora.h"

namespace lora {

using bf16 = __nv_bfloat16;

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ void load8(const bf16* p, float f[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ void load8(const float* p, float f[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// fp32 -> bf16 with round-to-nearest-even (CUDA's conversion intrinsic).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8_bf16(const float f[8]) {
  uint4 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  u.z = pack_bf16x2(f[4], f[5]);
  u.w = pack_bf16x2(f[6], f[7]);
  return u;
}

__device__ __forceinline__ void store8(bf16* p, const float f[8]) {
  *reinterpret_cast<uint4*>(p) = pack8_bf16(f);
}

__device__ __forceinline__ void store8(float* p, const float f[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// Loads of data written by the kernel this one depends on through a
// programmatic (early) launch.  Such data is not read-only for this kernel's
// lifetime, so it must not go through __restrict__ / non-coherent loads; an
// asm volatile L2 load also cannot be hoisted above griddepcontrol.wait.
__device__ __forceinline__ int ld_dep(const int32_t* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dep_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void load8_dep(const float* p, float f[8]) {
  const float4 a = ld_dep_f4(p), b = ld_dep_f4(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bits) {
  if (err != nullptr) atomicOr(err, bits);
}

__device__ __forceinline__ bool slot_valid(int id, int n_slots) { return id >= 0 && id < n_slots; }

// Indices that come from data one kernel hands to another (the segment
// builder's perm and segment offsets and slots).  In a debug build
// (-DLORA_DEBUG) an index outside [0, n) raises LORA_DEVERR_BOUNDS and is
// replaced by 0, so no access leaves its buffer; the release build uses the
// index as it is.
#ifdef LORA_DEBUG
__device__ __forceinline__ int checked_index(int i, int n, uint32_t* err) {
  if (i >= 0 && i < n) return i;
  flag_error(err, LORA_DEVERR_BOUNDS);
  return 0;
}
#else
__device__ __forceinline__ int checked_index(int i, int, uint32_t*) { return i; }
#endif
// perm[idx] of a batch of T tokens, written by the grid this one depends on
// (ld_dep) or by an earlier kernel of the stream (plain load).
__device__ __forceinline__ int perm_row(const int32_t* perm, int idx, int T, uint32_t* err) {
  return checked_index(ld_dep(perm + checked_index(idx, T, err)), T, err);
}
__device__ __forceinline__ int perm_row_plain(const int32_t* perm, int idx, int T, uint32_t* err) {
  return checked_index(perm[checked_index(idx, T, err)], T, err);
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible (no-op without the attribute);
// allow the next dependent grid to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace lora
