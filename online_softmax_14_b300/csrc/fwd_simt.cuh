// Float32 attention forward on the CUDA cores (FFMA), one warp per query row.
//
// The online-softmax recurrence of "The Flash Attention" page (running max m,
// normaliser l, accumulator acc; c = exp(m_old - m_new) rescales l and acc when the
// max moves; divide once at the end), streamed over key blocks of 32 keys that a
// CTA of 8 warps (8 query rows) shares through shared memory.  Lane j scores key
// j of the block; the block max and sum are warp-shuffle reductions; lane t owns
// output columns t, t+32, ... of its row.  A fully masked row (l = 0) writes the
// zero vector and lse = -inf ("Flash attention and efficient attention: Worked
// examples", Cell D2).
//
// This path serves float32 inputs, whose 1e-5 accuracy the tensor cores' reduced
// precision formats cannot meet; the bfloat16 path uses tcgen05 (fwd_tc.cuh).
#pragma once
#include "ptx.cuh"

namespace fa {

struct SimtParams {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;         // may be null
  const int* kv_len;  // may be null
  int BH, H, N, d;    // N queries per head
  int Nk;             // keys per head
  float scale;        // score multiplier (> 0)
  float scale_log2;   // scale * log2(e)
  int causal;         // 0 none, else key k visible to row i iff k < i + qoff
  int qoff;           // (Nk - N) + 1 (causal 1) or (Nk - N) (causal 2, strict)
};

constexpr int SIMT_ROWS = 8;   // query rows (warps) per CTA
constexpr int SIMT_KEYS = 32;  // keys per block

template <int DP>  // DP = d rounded up to a multiple of 32 (32, 64, 96 or 128)
__global__ void __launch_bounds__(SIMT_ROWS * 32) fwd_f32_simt_kernel(const SimtParams p) {
  constexpr int CPL = DP / 32;  // output columns per lane
  __shared__ float sK[SIMT_KEYS][DP + 1];  // +1: lanes read different rows of one column
  __shared__ float sV[SIMT_KEYS][DP];
  __shared__ float sQ[SIMT_ROWS][DP];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int b = bh / p.H;
  const int row0 = blockIdx.x * SIMT_ROWS;
  const int row = row0 + warp;
  const int N = p.N, Nk = p.Nk, d = p.d;
  const size_t head = static_cast<size_t>(bh) * N * d;     // q, o
  const size_t head_k = static_cast<size_t>(bh) * Nk * d;  // k, v

  int kv_limit = Nk;
  if (p.kv_len) kv_limit = min(Nk, max(0, p.kv_len[b]));
  // keys this CTA needs: causal rows see keys < row + qoff; padding stops at kv_limit
  int n_keys = kv_limit;
  if (p.causal) n_keys = min(n_keys, max(0, row0 + SIMT_ROWS - 1 + p.qoff));

  for (int c = lane; c < DP; c += 32)
    sQ[warp][c] = (row < N && c < d) ? p.q[head + static_cast<size_t>(row) * d + c] : 0.f;

  float m = -INFINITY, l = 0.f;  // m in raw score units (scale > 0 keeps the max)
  float acc[CPL];
#pragma unroll
  for (int t = 0; t < CPL; ++t) acc[t] = 0.f;

  for (int k0 = 0; k0 < n_keys; k0 += SIMT_KEYS) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < SIMT_KEYS * DP; idx += blockDim.x) {
      const int kr = idx / DP, c = idx % DP;
      const bool in = (k0 + kr < Nk) && c < d;
      const size_t g = head_k + static_cast<size_t>(k0 + kr) * d + c;
      sK[kr][c] = in ? p.k[g] : 0.f;
      sV[kr][c] = in ? p.v[g] : 0.f;
    }
    __syncthreads();
    if (row >= N) continue;

    // score of key k0 + lane for this row: S = q . k (scale applied in the exponent)
    float s = 0.f;
#pragma unroll 8
    for (int c = 0; c < DP; ++c) s = fmaf(sQ[warp][c], sK[lane][c], s);
    const int key = k0 + lane;
    const bool vis = key < kv_limit && (!p.causal || key < row + p.qoff);
    if (!vis) s = -INFINITY;

    float mb = s;  // block max (warp reduction)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    const float m_new = fmaxf(m, mb);
    const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
    const float c = exp2f((m - m_ref) * p.scale_log2);  // rescale of what is accumulated so far
    const float pj = exp2f((s - m_ref) * p.scale_log2);  // exp(scale * (s - m)), 0 when masked
    float ps = pj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * c + ps;
#pragma unroll
    for (int t = 0; t < CPL; ++t) acc[t] *= c;
    for (int j = 0; j < SIMT_KEYS; ++j) {
      const float pb = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
      for (int t = 0; t < CPL; ++t) acc[t] = fmaf(pb, sV[j][lane + 32 * t], acc[t]);
    }
    m = m_new;
  }

  if (row < N) {
    const float inv = (l > 0.f) ? 1.f / l : 0.f;  // guard: l = 0 -> zero vector
#pragma unroll
    for (int t = 0; t < CPL; ++t) {
      const int c = lane + 32 * t;
      if (c < d) p.o[head + static_cast<size_t>(row) * d + c] = acc[t] * inv;
    }
    if (p.lse && lane == 0)
      p.lse[static_cast<size_t>(bh) * N + row] = (l > 0.f) ? fmaf(m, p.scale, logf(l)) : -INFINITY;
  }
}

}  // namespace fa
