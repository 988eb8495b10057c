// prefill_simt.cu — prefill passes on the FMA pipe (fp32 caches, and any
// shape the tensor-core path does not take).
//
// H2O summary page, "Algorithm / figure walkthrough" step 1: the prompt is
// attended causally and every prompt key's accumulated score is the sum of the
// softmax weights it receives, i.e. the causal column sum
//   colsum_j = sum_{i >= j} exp(s_ij - LSE_i),  s_ij = q_i . k_j / sqrt(d).
// Pass 1 (flash-style, online softmax over key tiles) writes O and the row
// log-sum-exp LSE_i; pass 2 recomputes the logits tile by tile with the key
// as the register operand, so each thread group owns one key column and sums
// down it: deterministic, no atomics.
#include "common.cuh"

namespace h2o {
namespace {

constexpr int kThreads = 128;
constexpr int kTile = 32;  // queries (pass 1) or keys (pass 2) per CTA, and rows per staged tile
constexpr int kTPR = 4;    // threads per row

template <typename T> __device__ __forceinline__ float4 load4(const T *p);
template <> __device__ __forceinline__ float4 load4<float>(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p) {
  const uint2 w = *reinterpret_cast<const uint2 *>(p);
  return make_float4(bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y));
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

// Pass 1: CTA = 32 queries x 4 threads; thread `part` owns float4 chunks
// part, part+4, ... of the row (interleaved: conflict-free shared reads).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) attn_simt(const T *__restrict__ Q, const T *__restrict__ K,
                                                      const T *__restrict__ V, T *__restrict__ O,
                                                      float *__restrict__ lse, int L, float qscale) {
  constexpr int NC = D / 4, CPT = NC / kTPR;
  __shared__ float4 sK[kTile][NC];
  __shared__ float4 sV[kTile][NC];
  const int h = blockIdx.y;
  const int tid = threadIdx.x, qi = tid / kTPR, part = tid % kTPR;
  const int i = blockIdx.x * kTile + qi;
  const size_t hb = (size_t)h * L * D;

  float4 q[CPT], o[CPT];
#pragma unroll
  for (int cc = 0; cc < CPT; ++cc) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < L) x = load4<T>(Q + hb + (size_t)i * D + 4 * (part + kTPR * cc));
    q[cc] = make_float4(x.x * qscale, x.y * qscale, x.z * qscale, x.w * qscale);
    o[cc] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, l = 0.f;
  const int kend = min(L, (int)(blockIdx.x + 1) * kTile);
  for (int k0 = 0; k0 < kend; k0 += kTile) {
    __syncthreads();
    for (int idx = tid; idx < kTile * NC; idx += kThreads) {
      const int r = idx / NC, cch = idx % NC, j = k0 + r;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (j < L) {
        kv = load4<T>(K + hb + (size_t)j * D + 4 * cch);
        vv = load4<T>(V + hb + (size_t)j * D + 4 * cch);
      }
      sK[r][cch] = kv;
      sV[r][cch] = vv;
    }
    __syncthreads();
    float s[kTile];
    float tmax = -INFINITY;
#pragma unroll
    for (int r = 0; r < kTile; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int cc = 0; cc < CPT; ++cc) acc = dot4(q[cc], sK[r][part + kTPR * cc], acc);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      const int j = k0 + r;
      s[r] = (j <= i && j < L) ? acc : -INFINITY;
      tmax = fmaxf(tmax, s[r]);
    }
    const float mnew = fmaxf(m, tmax);
    if (mnew == -INFINITY) continue;
    const float corr = exp2f(m - mnew);
    l *= corr;
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
      o[cc].x *= corr; o[cc].y *= corr; o[cc].z *= corr; o[cc].w *= corr;
    }
#pragma unroll
    for (int r = 0; r < kTile; ++r) {
      const float p = exp2f(s[r] - mnew);
      l += p;
#pragma unroll
      for (int cc = 0; cc < CPT; ++cc) {
        const float4 v = sV[r][part + kTPR * cc];
        o[cc].x = fmaf(p, v.x, o[cc].x); o[cc].y = fmaf(p, v.y, o[cc].y);
        o[cc].z = fmaf(p, v.z, o[cc].z); o[cc].w = fmaf(p, v.w, o[cc].w);
      }
    }
    m = mnew;
  }
  if (i < L) {
    const float inv = 1.f / l;
    if (O) {
      T *orow = O + hb + (size_t)i * D;
#pragma unroll
      for (int cc = 0; cc < CPT; ++cc) {
        const int c0 = 4 * (part + kTPR * cc);
        orow[c0 + 0] = from_f32<T>(o[cc].x * inv);
        orow[c0 + 1] = from_f32<T>(o[cc].y * inv);
        orow[c0 + 2] = from_f32<T>(o[cc].z * inv);
        orow[c0 + 3] = from_f32<T>(o[cc].w * inv);
      }
    }
    if (part == 0) lse[(size_t)h * L + i] = m * kLn2 + logf(l);
  }
}

// Pass 2: CTA = 32 keys x 4 threads; query tiles from the CTA's first key on.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) colsum_simt(const T *__restrict__ Q, const T *__restrict__ K,
                                                        const float *__restrict__ lse,
                                                        float *__restrict__ colsum, int L, float qscale) {
  constexpr int NC = D / 4, CPT = NC / kTPR;
  __shared__ float4 sQ[kTile][NC];
  __shared__ float sL[kTile];
  const int h = blockIdx.y;
  const int tid = threadIdx.x, kj = tid / kTPR, part = tid % kTPR;
  const int j = blockIdx.x * kTile + kj;
  const size_t hb = (size_t)h * L * D;
  float4 kr[CPT];
#pragma unroll
  for (int cc = 0; cc < CPT; ++cc) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < L) x = load4<T>(K + hb + (size_t)j * D + 4 * (part + kTPR * cc));
    kr[cc] = make_float4(x.x * qscale, x.y * qscale, x.z * qscale, x.w * qscale);
  }
  float cs = 0.f;
  for (int q0 = blockIdx.x * kTile; q0 < L; q0 += kTile) {
    __syncthreads();
    for (int idx = tid; idx < kTile * NC; idx += kThreads) {
      const int r = idx / NC, cch = idx % NC, i = q0 + r;
      sQ[r][cch] = (i < L) ? load4<T>(Q + hb + (size_t)i * D + 4 * cch) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < kTile) sL[tid] = (q0 + tid < L) ? lse[(size_t)h * L + q0 + tid] * kLog2e : 0.f;
    __syncthreads();
#pragma unroll 4
    for (int r = 0; r < kTile; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int cc = 0; cc < CPT; ++cc) acc = dot4(kr[cc], sQ[r][part + kTPR * cc], acc);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      const int i = q0 + r;
      if (i >= j && i < L) cs += exp2f(acc - sL[r]);
    }
  }
  if (part == 0 && j < L) colsum[(size_t)h * L + j] = cs;
}

template <typename T, int D>
cudaError_t attn_t(const CacheView &c, const void *Q, const void *K, const void *V, void *O, float *lse,
                   int L, cudaStream_t st) {
  dim3 grid((unsigned)((L + kTile - 1) / kTile), (unsigned)c.nh);
  attn_simt<T, D><<<grid, kThreads, 0, st>>>((const T *)Q, (const T *)K, (const T *)V, (T *)O, lse, L,
                                             kLog2e / sqrtf((float)D));
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t colsum_t(const CacheView &c, const void *Q, const void *K, const float *lse, float *colsum,
                     int L, cudaStream_t st) {
  dim3 grid((unsigned)((L + kTile - 1) / kTile), (unsigned)c.nh);
  colsum_simt<T, D><<<grid, kThreads, 0, st>>>((const T *)Q, (const T *)K, lse, colsum, L,
                                               kLog2e / sqrtf((float)D));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_attn_simt(const CacheView &c, const void *Q, const void *K, const void *V,
                                     void *O, float *lse, int L, cudaStream_t st) {
  if (c.nh > 65535) return cudaErrorInvalidValue;
  if (c.dtype == 1) {
    if (c.d == 128) return attn_t<__nv_bfloat16, 128>(c, Q, K, V, O, lse, L, st);
    if (c.d == 64) return attn_t<__nv_bfloat16, 64>(c, Q, K, V, O, lse, L, st);
  } else {
    if (c.d == 128) return attn_t<float, 128>(c, Q, K, V, O, lse, L, st);
    if (c.d == 64) return attn_t<float, 64>(c, Q, K, V, O, lse, L, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_colsum_simt(const CacheView &c, const void *Q, const void *K, const float *lse,
                                       float *colsum, int L, cudaStream_t st) {
  if (c.nh > 65535) return cudaErrorInvalidValue;
  if (c.dtype == 1) {
    if (c.d == 128) return colsum_t<__nv_bfloat16, 128>(c, Q, K, lse, colsum, L, st);
    if (c.d == 64) return colsum_t<__nv_bfloat16, 64>(c, Q, K, lse, colsum, L, st);
  } else {
    if (c.d == 128) return colsum_t<float, 128>(c, Q, K, lse, colsum, L, st);
    if (c.d == 64) return colsum_t<float, 64>(c, Q, K, lse, colsum, L, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace h2o
