// Merge of partial attention results computed over disjoint key sets (split-key
// attention).  Part p holds, for every query row, its output O_p (already
// divided by its own normaliser) and log-normaliser lse_p.  A part is the block
// state (m = lse_p, l = 1, O~ = O_p), and the generic merge rule of the
// Exercises page ("Exercises -- Flash attention and efficient attention", the
// two- and three-block merges) combines them:
//     m = max_p lse_p,  f_p = e^(lse_p - m),  l = sum_p f_p,
//     O = sum_p f_p O_p / l,  lse = m + ln l.
// A part with lse_p = -inf saw no key and carries zero weight; a row whose parts
// are all empty gets O = 0 and lse = -inf ("Flash attention and efficient
// attention: Worked examples", Cell D2).
//
// One warp per row; lane t owns columns t, t + 32, ...  The pass reads every part
// once and writes the result once, so it is bound by device-memory bandwidth.
#pragma once
#include <cuda_bf16.h>

namespace fa {

struct MergeParams {
  const void* o_parts;     // [P][R][d]
  const float* lse_parts;  // [P][R]
  void* o;                 // [R][d]
  float* lse;              // [R] or null
  long long R;             // rows: B * H * N
  int P, d;
};

constexpr int MERGE_ROWS = 8;  // rows (warps) per CTA

template <typename T>
__device__ __forceinline__ float load_elem(const T* p);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void store_elem(T* p, float v);
template <>
__device__ __forceinline__ void store_elem<float>(float* p, float v) {
  *p = v;
}
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

template <typename T, int CPL>  // CPL = columns per lane, d <= 32 * CPL
__global__ void __launch_bounds__(MERGE_ROWS * 32) merge_kernel(const MergeParams p) {
  const long long row = static_cast<long long>(blockIdx.x) * MERGE_ROWS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.R) return;
  const T* parts = static_cast<const T*>(p.o_parts);

  float m = -INFINITY;
  for (int q = lane; q < p.P; q += 32) m = fmaxf(m, p.lse_parts[static_cast<size_t>(q) * p.R + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const float m_ref = (m == -INFINITY) ? 0.f : m;

  float acc[CPL];
#pragma unroll
  for (int t = 0; t < CPL; ++t) acc[t] = 0.f;
  float l = 0.f;
  for (int q = 0; q < p.P; ++q) {
    const float f = expf(p.lse_parts[static_cast<size_t>(q) * p.R + row] - m_ref);  // same in every lane
    l += f;
    if (f == 0.f) continue;  // an empty part (or one negligible against the others)
    const T* src = parts + (static_cast<size_t>(q) * p.R + row) * p.d;
#pragma unroll
    for (int t = 0; t < CPL; ++t) {
      const int c = lane + 32 * t;
      if (c < p.d) acc[t] = fmaf(f, load_elem(src + c), acc[t]);
    }
  }
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  T* dst = static_cast<T*>(p.o) + static_cast<size_t>(row) * p.d;
#pragma unroll
  for (int t = 0; t < CPL; ++t) {
    const int c = lane + 32 * t;
    if (c < p.d) store_elem(dst + c, acc[t] * inv);
  }
  if (p.lse && lane == 0) p.lse[row] = (l > 0.f) ? m_ref + logf(l) : -INFINITY;
}

// Vectorised form for rows of d * sizeof(T) = 16 * LPR bytes (LPR a power of two
// <= 32, 16-byte aligned tensors): LPR lanes share a row, each lane moves 16
// bytes per part, and a warp covers 32 / LPR rows.  The part loop is unrolled so
// that several 16-byte loads per lane are in flight.
template <typename T>
__device__ __forceinline__ void acc16(float* a, float f, const uint4& v);
template <>
__device__ __forceinline__ void acc16<float>(float* a, float f, const uint4& v) {
  a[0] = fmaf(f, __uint_as_float(v.x), a[0]);
  a[1] = fmaf(f, __uint_as_float(v.y), a[1]);
  a[2] = fmaf(f, __uint_as_float(v.z), a[2]);
  a[3] = fmaf(f, __uint_as_float(v.w), a[3]);
}
template <>
__device__ __forceinline__ void acc16<__nv_bfloat16>(float* a, float f, const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = fmaf(f, __uint_as_float(w[i] << 16), a[2 * i]);           // low half: element 2i
    a[2 * i + 1] = fmaf(f, __uint_as_float(w[i] & 0xffff0000u), a[2 * i + 1]);
  }
}
template <typename T>
__device__ __forceinline__ uint4 pack16(const float* a);
template <>
__device__ __forceinline__ uint4 pack16<float>(const float* a) {
  return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]), __float_as_uint(a[3]));
}
template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float* a) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T, int LPR>
__global__ void __launch_bounds__(MERGE_ROWS * 32) merge_vec_kernel(const MergeParams p) {
  constexpr int VW = 16 / sizeof(T);  // elements per 16-byte vector
  constexpr int RPW = 32 / LPR;       // rows per warp
  const int lane = threadIdx.x & 31;
  const long long row =
      (static_cast<long long>(blockIdx.x) * MERGE_ROWS + (threadIdx.x >> 5)) * RPW + lane / LPR;
  if (row >= p.R) return;  // whole row groups leave together; no shuffles below
  const int sub = lane % LPR;

  float m = -INFINITY;
  for (int q = 0; q < p.P; ++q) m = fmaxf(m, p.lse_parts[static_cast<size_t>(q) * p.R + row]);
  const float m_ref = (m == -INFINITY) ? 0.f : m;

  float acc[VW];
#pragma unroll
  for (int i = 0; i < VW; ++i) acc[i] = 0.f;
  float l = 0.f;
  const uint4* src = reinterpret_cast<const uint4*>(p.o_parts) + static_cast<size_t>(row) * LPR + sub;
  const size_t part_stride = static_cast<size_t>(p.R) * LPR;  // in 16-byte vectors
  int q = 0;
  for (; q + 4 <= p.P; q += 4) {
    uint4 v[4];
    float f[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u] = __ldg(src + (q + u) * part_stride);
      f[u] = expf(p.lse_parts[static_cast<size_t>(q + u) * p.R + row] - m_ref);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      l += f[u];
      if (f[u] != 0.f) acc16<T>(acc, f[u], v[u]);  // an empty part's values are never used
    }
  }
  for (; q < p.P; ++q) {
    const float f = expf(p.lse_parts[static_cast<size_t>(q) * p.R + row] - m_ref);
    l += f;
    if (f != 0.f) acc16<T>(acc, f, __ldg(src + q * part_stride));
  }
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < VW; ++i) acc[i] *= inv;
  reinterpret_cast<uint4*>(p.o)[static_cast<size_t>(row) * LPR + sub] = pack16<T>(acc);
  if (p.lse && sub == 0) p.lse[row] = (l > 0.f) ? m_ref + logf(l) : -INFINITY;
}

}  // namespace fa
