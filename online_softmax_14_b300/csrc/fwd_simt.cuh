// Float32 attention forward on the CUDA cores (FFMA).
//
// The online-softmax recurrence of "The Flash Attention" page (running max m,
// normaliser l, accumulator acc; c = exp(m_old - m_new) rescales l and acc when the
// max moves; divide once at the end), for a CTA of 8 query rows.  The CTA's 8
// warps split the keys: warp w takes key blocks w, w + 8, ... (32 keys per block,
// key j of a block on lane j) for all 8 rows, so that a short key range is not
// walked block after block by every warp.  Each warp keeps its own (m, l, acc) per
// row; at the end the eight states of a row are merged with the block-merge rule
// of the Exercises page (two- and three-block merges: each state is weighted by
// exp(m_w - m), m the largest of the m_w) and divided once.  A fully masked row
// (l = 0) writes the zero vector and lse = -inf ("Flash attention and efficient
// attention: Worked examples", Cell D2).
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

constexpr int SIMT_ROWS = 8;   // query rows per CTA
constexpr int SIMT_WARPS = 8;  // warps per CTA, splitting the keys
constexpr int SIMT_KEYS = 32;  // keys per block (one per lane)

template <int DP>  // DP = d rounded up to a multiple of 32 (32, 64, 96 or 128)
__global__ void __launch_bounds__(SIMT_WARPS * 32) fwd_f32_simt_kernel(const SimtParams p) {
  constexpr int CPL = DP / 32;  // output columns per lane
  constexpr int R = SIMT_ROWS;
  __shared__ float sQ[R][DP];
  __shared__ float sM[SIMT_WARPS][R], sL[SIMT_WARPS][R];
  __shared__ float sAcc[SIMT_WARPS][R][DP];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int b = bh / p.H;
  const int row0 = blockIdx.x * R;
  const int N = p.N, Nk = p.Nk, d = p.d;
  const size_t head = static_cast<size_t>(bh) * N * d;     // q, o
  const size_t head_k = static_cast<size_t>(bh) * Nk * d;  // k, v

  int kv_limit = Nk;
  if (p.kv_len) kv_limit = min(Nk, max(0, p.kv_len[b]));
  // keys this CTA needs: causal rows see keys < row + qoff; padding stops at kv_limit
  int n_keys = kv_limit;
  if (p.causal) n_keys = min(n_keys, max(0, row0 + R - 1 + p.qoff));

  for (int i = threadIdx.x; i < R * DP; i += blockDim.x) {
    const int r = i / DP, c = i % DP;
    sQ[r][c] = (row0 + r < N && c < d) ? p.q[head + static_cast<size_t>(row0 + r) * d + c] : 0.f;
  }
  __syncthreads();

  // m in raw score units (scale > 0 keeps the max)
  float m[R], l[R], acc[R][CPL];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int t = 0; t < CPL; ++t) acc[r][t] = 0.f;
  }

  for (int k0 = warp * SIMT_KEYS; k0 < n_keys; k0 += SIMT_WARPS * SIMT_KEYS) {
    // scores of key k0 + lane against the CTA's rows: S = q . k (scale in the exponent)
    const int key = k0 + lane;
    const float* krow = p.k + head_k + static_cast<size_t>(min(key, Nk - 1)) * d;
    float s[R];
#pragma unroll
    for (int r = 0; r < R; ++r) s[r] = 0.f;
    // the key row in chunks of 16 loads, all issued before their FMAs
    for (int c0 = 0; c0 < DP; c0 += 16) {
      float kc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) kc[i] = (key < Nk && c0 + i < d) ? krow[c0 + i] : 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int r = 0; r < R; ++r) s[r] = fmaf(sQ[r][c0 + i], kc[i], s[r]);
    }
    float pj[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const bool vis = key < kv_limit && (!p.causal || key < row0 + r + p.qoff);
      const float sr = vis ? s[r] : -INFINITY;
      float mb = sr;  // block max (warp reduction)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      const float m_new = fmaxf(m[r], mb);
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float c = exp2f((m[r] - m_ref) * p.scale_log2);  // rescale of what is accumulated so far
      pj[r] = exp2f((sr - m_ref) * p.scale_log2);           // exp(scale * (s - m)), 0 when masked
      float ps = pj[r];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[r] = l[r] * c + ps;
#pragma unroll
      for (int t = 0; t < CPL; ++t) acc[r][t] *= c;
      m[r] = m_new;
    }
    // acc += p V over the block's keys, 8 keys at a time with their V rows loaded
    // first; lane t owns columns lane + 32 t (keys past Nk have p = 0 and read as 0)
    for (int j0 = 0; j0 < SIMT_KEYS; j0 += 8) {
      float vv[8][CPL];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int kj = k0 + j0 + jj;
        const float* vrow = p.v + head_k + static_cast<size_t>(min(kj, Nk - 1)) * d;
#pragma unroll
        for (int t = 0; t < CPL; ++t) vv[jj][t] = (kj < Nk && lane + 32 * t < d) ? vrow[lane + 32 * t] : 0.f;
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float pb = __shfl_sync(0xffffffffu, pj[r], j0 + jj);
#pragma unroll
          for (int t = 0; t < CPL; ++t) acc[r][t] = fmaf(pb, vv[jj][t], acc[r][t]);
        }
    }
  }

  // each warp's state per row, then warp r merges row r
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (lane == 0) {
      sM[warp][r] = m[r];
      sL[warp][r] = l[r];
    }
#pragma unroll
    for (int t = 0; t < CPL; ++t) sAcc[warp][r][lane + 32 * t] = acc[r][t];
  }
  __syncthreads();
  static_assert(SIMT_WARPS == R, "warp r merges row r");
  const int r = warp, row = row0 + warp;
  if (row < N) {
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < SIMT_WARPS; ++w) mm = fmaxf(mm, sM[w][r]);
    const float m_ref = (mm == -INFINITY) ? 0.f : mm;
    float ll = 0.f, o[CPL];
#pragma unroll
    for (int t = 0; t < CPL; ++t) o[t] = 0.f;
#pragma unroll
    for (int w = 0; w < SIMT_WARPS; ++w) {
      const float f = exp2f((sM[w][r] - m_ref) * p.scale_log2);  // 0 for a warp that saw no key
      ll = fmaf(f, sL[w][r], ll);
#pragma unroll
      for (int t = 0; t < CPL; ++t) o[t] = fmaf(f, sAcc[w][r][lane + 32 * t], o[t]);
    }
    const float inv = (ll > 0.f) ? 1.f / ll : 0.f;  // guard: l = 0 -> zero vector
#pragma unroll
    for (int t = 0; t < CPL; ++t) {
      const int c = lane + 32 * t;
      if (c < d) p.o[head + static_cast<size_t>(row) * d + c] = o[t] * inv;
    }
    if (p.lse && lane == 0)
      p.lse[static_cast<size_t>(bh) * N + row] = (ll > 0.f) ? fmaf(mm, p.scale, logf(ll)) : -INFINITY;
  }
}

}  // namespace fa
