// common.cuh — device helpers shared by the H2O kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace h2o {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Elements of T in one 16-byte vector.
template <typename T> struct VecN;
template <> struct VecN<float> { static constexpr int N = 4; };
template <> struct VecN<__nv_bfloat16> { static constexpr int N = 8; };

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16-byte loads through the read-only path (data written by earlier launches).
__device__ __forceinline__ uint4 ld_nc16(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
// 16-byte loads through L2 only (data other CTAs of this launch may write).
__device__ __forceinline__ uint4 ld_cg16(const void *p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <typename T> struct Unpack;
template <> struct Unpack<float> {
  __device__ __forceinline__ static void run(const uint4 &v, float *x) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
};
template <> struct Unpack<__nv_bfloat16> {
  __device__ __forceinline__ static void run(const uint4 &v, float *x) {
    x[0] = bf16lo(v.x); x[1] = bf16hi(v.x); x[2] = bf16lo(v.y); x[3] = bf16hi(v.y);
    x[4] = bf16lo(v.z); x[5] = bf16hi(v.z); x[6] = bf16lo(v.w); x[7] = bf16hi(v.w);
  }
};

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Ranking key of the cache entry at position `pos` once the query at position
// p has attended: its accumulated score, or (score_mode 1) that score over
// the number of queries that attended to it, p - pos + 1 (an entry, once
// cached, has seen every later query).
__device__ __forceinline__ float rank_key(float score, long long p, int pos, int score_mode) {
  return score_mode ? __fdiv_rn(score, (float)(p - pos + 1)) : score;
}

// Lexicographic (score, position) minimum carried with the slot index.
struct ArgMin {
  float s;
  int p;
  int slot;  // -2 = none, -1 = the new token, >= 0 = cache slot
};
__device__ __forceinline__ bool am_less(const ArgMin &a, const ArgMin &b) {
  if (a.slot == -2) return false;
  if (b.slot == -2) return true;
  return a.s < b.s || (a.s == b.s && a.p < b.p);
}
__device__ __forceinline__ ArgMin warp_argmin(ArgMin a) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    ArgMin b;
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    b.p = __shfl_xor_sync(0xffffffffu, a.p, o);
    b.slot = __shfl_xor_sync(0xffffffffu, a.slot, o);
    if (am_less(b, a)) a = b;
  }
  return a;
}

}  // namespace h2o
