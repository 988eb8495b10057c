// common.cuh — device helpers shared by the H2O kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "internal.h"

namespace h2o {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Elements of T in one 16-byte vector.
template <typename T> struct VecN;
template <> struct VecN<float> { static constexpr int N = 4; };
template <> struct VecN<__nv_bfloat16> { static constexpr int N = 8; };

// Storage element of an fp8 cache: one e4m3 byte (sign, 4 exponent bits with
// bias 7, 3 mantissa bits; largest finite 448).  Each cached row carries one
// fp32 scale and reads back as code * scale.
struct e4m3 {
  uint8_t bits;
};
template <typename S> constexpr bool is_fp8() { return std::is_same<S, e4m3>::value; }

// How a lane reads a stored row: 16 bytes per load, 8 for an fp8 row (so an
// fp8 row of d codes maps onto as many lanes, with as few registers, as a
// bf16 row).
template <typename S> struct Lane {
  static constexpr int VB = 16;
  using V = uint4;
};
template <> struct Lane<e4m3> {
  static constexpr int VB = 8;
  using V = uint2;
};

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

// Four e4m3 codes (byte i of w is element i) as floats, through the hardware
// e4m3x2 -> f16x2 conversion (exact: every e4m3 value is an f16 value).
// Measured on GB300 the fastest of the unpack forms tried (integer bit
// placement and mixed-precision FMAs were slower).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float *x) {
  const __half2_raw a = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
  const __half2_raw b = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  x[0] = __half2float(__ushort_as_half(a.x));
  x[1] = __half2float(__ushort_as_half(a.y));
  x[2] = __half2float(__ushort_as_half(b.x));
  x[3] = __half2float(__ushort_as_half(b.y));
}
template <> struct Unpack<e4m3> {
  // 8 codes (byte i is element i)
  __device__ __forceinline__ static void run(const uint2 &v, float *x) {
    e4m3x4_to_f32(v.x, x);
    e4m3x4_to_f32(v.y, x + 4);
  }
};
// One lane's share of a stored row (Lane<S>::VB bytes at p) as floats.
template <typename S> __device__ __forceinline__ void unpack_lane(const uint8_t *p, float *x) {
  Unpack<S>::run(*(const typename Lane<S>::V *)p, x);
}

// N consecutive elements of T as floats, 16 bytes per load (N a multiple of
// the elements in 16 bytes): plain loads (shared memory), and read-only
// global loads.
template <typename T, int N> __device__ __forceinline__ void load_f32(const T *p, float *x) {
  constexpr int V = VecN<T>::N;
  static_assert(N % V == 0, "whole 16-byte vectors");
#pragma unroll
  for (int i = 0; i < N / V; ++i) Unpack<T>::run(*(const uint4 *)(p + i * V), x + i * V);
}
template <typename T, int N> __device__ __forceinline__ void load_f32_nc(const T *p, float *x) {
  constexpr int V = VecN<T>::N;
  static_assert(N % V == 0, "whole 16-byte vectors");
#pragma unroll
  for (int i = 0; i < N / V; ++i) Unpack<T>::run(ld_nc16(p + i * V), x + i * V);
}

// a[i] = p * x[i] + a[i] for a pair (i = 0, 1): one packed fp32 FMA
// instruction, each lane rounded as a scalar fmaf would be.
__device__ __forceinline__ void fma_pair(float &a0, float &a1, float p, float x0, float x1) {
  unsigned long long acc, pp, xx;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(pp) : "f"(p));
  asm("mov.b64 %0, {%1, %2};" : "=l"(xx) : "f"(x0), "f"(x1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(pp), "l"(xx));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}

// Two products of packed 16-bit pairs accumulated in fp32 with the
// mixed-precision FMA (fp32 accumulator, f16 / bf16 multiplicands): element 0
// of each operand is its low half.  Products of two bf16 (or two f16) values
// are exact in fp32, so this is an fp32 dot product without unpacking.
__device__ __forceinline__ float fma2_bf16(uint32_t a, uint32_t b, float c) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}
__device__ __forceinline__ float fma2_f16(uint32_t a, uint32_t b, float c) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}
// Two e4m3 codes (low byte = element 0) as an f16x2 word (element 0 in the
// low half); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

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

// One lane's share of q for the K dot products of a stored row type S, kept
// packed: bf16 rows take the raw bf16 q (mixed bf16 FMA), fp8 rows take q in
// f16 (mixed f16 FMA after the e4m3 -> f16 conversion), fp32 rows keep
// prescaled fp32 q.  `scale` is the factor that turns the accumulated dot
// into the log2-domain logit (times the row's K scale for fp8).
template <typename S, int EPL> struct QLane {
  float v[EPL];
  float scale;
  template <typename T> __device__ __forceinline__ void load(const T *q, float qscale) {
    load_f32<T, EPL>(q, v);
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] *= qscale;
    scale = 1.f;
  }
  __device__ __forceinline__ float dot(const uint8_t *row) const {
    float x[EPL];
    unpack_lane<S>(row, x);
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) d = fmaf(v[e], x[e], d);
    return d;
  }
};
template <int EPL> struct QLane<__nv_bfloat16, EPL> {
  uint32_t w[EPL / 2];
  float scale;
  template <typename T> __device__ __forceinline__ void load(const T *q, float qscale) {
    static_assert(std::is_same<T, __nv_bfloat16>::value, "bf16 rows take bf16 queries");
#pragma unroll
    for (int i = 0; i < EPL / 8; ++i) {
      const uint4 u = *(const uint4 *)(q + 8 * i);
      w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
    }
    scale = qscale;
  }
  __device__ __forceinline__ float dot(const uint8_t *row) const {
    const uint4 k = *(const uint4 *)row;
    float d = 0.f;
    d = fma2_bf16(w[0], k.x, d);
    d = fma2_bf16(w[1], k.y, d);
    d = fma2_bf16(w[2], k.z, d);
    d = fma2_bf16(w[3], k.w, d);
    return d;
  }
};
template <int EPL> struct QLane<e4m3, EPL> {
  static_assert(EPL == 8, "an fp8 lane reads 8 codes");
  uint32_t w[4];
  float scale;
  // q in f16: scaled by a power of two when max|q| would leave f16's range
  // (undone in `scale`); warp-collective (every lane of the warp calls it).
  template <typename T> __device__ __forceinline__ void load(const T *q, float qscale) {
    float v[8];
    load_f32<T, 8>(q, v);
    float qmax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) qmax = fmaxf(qmax, fabsf(v[e]));
    qmax = warp_max(qmax);
    int ex = 0;
    frexpf(qmax, &ex);  // qmax < 2^ex
    const int sh = ex > 14 ? 14 - ex : 0;  // keep |q| below 2^14
    const float qs = ldexpf(1.f, sh);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(v[2 * i] * qs, v[2 * i + 1] * qs);
      w[i] = *(const uint32_t *)&h;
    }
    scale = qscale * ldexpf(1.f, -sh);
  }
  __device__ __forceinline__ float dot(const uint8_t *row) const {
    const uint2 k = *(const uint2 *)row;
    float d = 0.f;
    d = fma2_f16(w[0], e4m3x2_to_f16x2(k.x), d);
    d = fma2_f16(w[1], e4m3x2_to_f16x2(k.x >> 16), d);
    d = fma2_f16(w[2], e4m3x2_to_f16x2(k.y), d);
    d = fma2_f16(w[3], e4m3x2_to_f16x2(k.y >> 16), d);
    return d;
  }
};

// Transposed butterfly reduction: each of the LPR lanes of a group holds
// partial sums of the same ITER rows; afterwards lane `sub` of the group holds
// the full sum of row sub / (LPR / ITER).  At each of the first log2(ITER)
// levels a lane keeps half of its rows and sends the other half to its
// partner, so the group spends (ITER - 1) + log2(LPR / ITER) shuffles instead
// of ITER * log2(LPR).
template <int ITER, int LPR>
__device__ __forceinline__ float xreduce(float (&x)[ITER], int sub) {
  static_assert(ITER >= 1 && ITER <= LPR && (ITER & (ITER - 1)) == 0, "ITER a power of two <= LPR");
#pragma unroll
  for (int n = ITER, o = LPR / 2; n > 1; n >>= 1, o >>= 1) {
    const bool up = (sub & o) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float send = up ? x[j] : x[j + n / 2];
      const float keep = up ? x[j + n / 2] : x[j];
      x[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
#pragma unroll
  for (int o = LPR / (2 * ITER); o >= 1; o >>= 1) x[0] += __shfl_xor_sync(0xffffffffu, x[0], o);
  return x[0];
}

// Warp-collective quantisation of one row of 32 * PER values into an fp8
// cache row: lane L holds elements L*PER .. L*PER+PER-1 in x.  scale =
// amax / 448 (fp32 division; 0 for an all-zero row), code = e4m3 of x / scale
// rounded to nearest even and saturated at 448 (0 when scale is 0).  Returns
// the lane's PER codes packed little-end first; every lane gets the scale.
template <int PER>
__device__ __forceinline__ uint32_t quant_row_e4m3(const float *x, float &scale) {
  static_assert(PER == 2 || PER == 4, "a lane packs 2 or 4 codes");
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) amax = fmaxf(amax, fabsf(x[e]));
  amax = warp_max(amax);
  scale = __fdiv_rn(amax, 448.f);
  uint32_t packed = 0u;
  if (scale > 0.f) {
#pragma unroll
    for (int e = 0; e < PER; ++e)
      packed |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[e], scale), __NV_SATFINITE, __NV_E4M3) << (8 * e);
  }
  return packed;
}
// Store a lane's PER packed codes at byte offset lane * PER of a row.
template <int PER>
__device__ __forceinline__ void store_codes(uint8_t *row, int lane, uint32_t packed) {
  if (PER == 4)
    *(uint32_t *)(row + lane * 4) = packed;
  else
    *(uint16_t *)(row + lane * 2) = (uint16_t)packed;
}

// s += w by compensated (Kahan) summation: c carries, negated, the low-order
// part that earlier additions to s lost, so a score that is a sum of millions
// of small weights keeps its accuracy (W. Kahan, "Further remarks on reducing
// truncation errors", Comm. ACM 8(1), 1965).  Returns the new s.
__device__ __forceinline__ float kahan_add(float &s, float &c, float w) {
  const float y = w - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
  return t;
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
// Warp-wide am_less minimum, the same in every lane.  Candidate keys are
// non-negative floats (sums of softmax weights, or those over a positive
// count), whose bit patterns order like their values, and positions are
// non-negative: two unsigned min-reductions give the lexicographic (key,
// position) minimum ("none" entries carry all-ones bits and lose), a ballot
// finds the lane holding it.
__device__ __forceinline__ ArgMin warp_argmin(ArgMin a) {
  const unsigned kb = (a.slot == -2) ? 0xFFFFFFFFu : __float_as_uint(a.s);
  const unsigned kmin = __reduce_min_sync(0xffffffffu, kb);
  const unsigned pb = (kb == kmin) ? (unsigned)a.p : 0xFFFFFFFFu;
  const unsigned pmin = __reduce_min_sync(0xffffffffu, pb);
  const int src = __ffs(__ballot_sync(0xffffffffu, kb == kmin && pb == pmin)) - 1;
  ArgMin r;
  r.s = __shfl_sync(0xffffffffu, a.s, src);
  r.p = __shfl_sync(0xffffffffu, a.p, src);
  r.slot = __shfl_sync(0xffffffffu, a.slot, src);
  return r;
}

}  // namespace h2o
