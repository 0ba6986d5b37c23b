// Standard attention, the comparator of "Foundations -- Flash attention and
// efficient attention", section 10: the N x N score matrix S and the
// probabilities P are written to device memory in full, then read back.
//
//     S = scale * Q K^T        (float32, every entry, masked ones included)
//     P = softmax_rows(S)      (masked entries -> 0; bfloat16 for the product)
//     O = P V                  (bfloat16), lse = ln sum_j exp(S_ij) over visible keys
//
// This is not the hot path: it is kept to measure what the tiled kernels save
// (the Exercises page's memory-size and HBM-traffic exercises put the quadratic
// term at nearly all of the traffic).  The products still run on the tensor
// cores, so the comparison is of memory traffic, not of arithmetic units.
//
// Kernels:
//  * std_gemm_kernel -- C = A B^T (B K-major) or C = A B (B MN-major) per batch
//    slice, 128 x 128 output tiles, K in 64-element chunks through a TMA ring;
//    A, B bf16; C float32 times alpha (for S) or bf16 (for O).  One thread issues
//    the MMAs into tensor memory; the four warps then read one output row each
//    (tensor-memory lane = row) and store it.
//  * std_softmax_kernel -- one warp per row of S: max (pass 1), sum of
//    exponentials (pass 2), P and lse (pass 3), the plain two-pass stable softmax
//    with a third pass to write P.
#pragma once
#include "ptx.cuh"

namespace fa {

enum : unsigned {
  ST_STD_TIMEOUT = 1u << 24,
};

struct StdGemmParams {
  void* c;            // [batch][M][ldc] float32 (alpha applied) or bf16
  long long ldc;      // row stride of C, elements
  long long c_batch;  // batch stride of C, elements
  int M, N, K;        // C is M x N; K is the contraction length
  int tiles_n;        // ceil(N / 128)
  float alpha;
  unsigned* status;
  unsigned long long timeout_ns;
};

template <int STAGES>
struct StdGemmLayout {
  static constexpr int A_BYTES = 128 * 128;        // 128 rows x 64 elements (128 B)
  static constexpr int B_BYTES = 128 * 128;        // 128 N x 64 K, either major
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int OFF_BAR = STAGES * STAGE;   // full[S], empty[S], acc_full
  static constexpr int OFF_MISC = OFF_BAR + (2 * STAGES + 1) * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
};

// B_MN = false: B is [N][K] (K-major), C = A B^T.  B_MN = true: B is [K][N]
// (MN-major, loaded as two 64-column blocks per K chunk), C = A B.
template <int STAGES, bool B_MN, bool OUT_F32>
__global__ void __launch_bounds__(128)
    std_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const StdGemmParams p) {
  using L = StdGemmLayout<STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full = sbase + L::OFF_BAR, empty = full + 8 * STAGES, acc_full = empty + 8 * STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* issued = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tm = static_cast<int>(blockIdx.x) / p.tiles_n, tn = static_cast<int>(blockIdx.x) % p.tiles_n;
  const int z = static_cast<int>(blockIdx.y);
  const int m0 = tm * 128, n0 = tn * 128;
  const int n_k = (p.K + 63) / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    *issued = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
  constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer --
    for (int c = 0; c < n_k; ++c) {
      const int s = c % STAGES;
      if (c >= STAGES && !mbar_wait(empty + 8 * s, ((c / STAGES) - 1) & 1, wc, ST_STD_TIMEOUT)) break;
      mbar_arrive_expect_tx(full + 8 * s, L::STAGE);
      const uint32_t a_dst = sbase + s * L::STAGE, b_dst = a_dst + L::A_BYTES;
      tma_load_3d(a_dst, &tm_a, full + 8 * s, c * 64, m0, z);
      if (B_MN) {
        tma_load_3d(b_dst, &tm_b, full + 8 * s, n0, c * 64, z);              // N 0-63 of the tile
        tma_load_3d(b_dst + L::B_BYTES / 2, &tm_b, full + 8 * s, n0 + 64, c * 64, z);  // N 64-127
      } else {
        tma_load_3d(b_dst, &tm_b, full + 8 * s, c * 64, n0, z);
      }
      *issued = c + 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer --
    constexpr uint32_t IDESC = idesc_bf16_f32(128, 128, B_MN);
    for (int c = 0; c < n_k; ++c) {
      const int s = c % STAGES;
      if (!mbar_wait_w(full + 8 * s, (c / STAGES) & 1, wc, ST_STD_TIMEOUT)) break;
      tc_fence_after();
      const uint32_t a = sbase + s * L::STAGE, b = a + L::A_BYTES;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // A K-major: 16 elements = 32 bytes along the row; B MN-major: 16 K rows
        // of 128 bytes, the two 64-column blocks 8 KB apart
        const uint64_t da = sdesc_sw128(a + kk * 32, 16, 1024);
        const uint64_t db = B_MN ? sdesc_sw128(b + kk * 2048, L::B_BYTES / 2, 1024) : sdesc_sw128(b + kk * 32, 16, 1024);
        umma_ss_w(tmem, da, db, IDESC, (c > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit_w(empty + 8 * s);
    }
    // also after a failed wait: the epilogue then finds the abort flag set and
    // only drains what was issued
    umma_commit_w(acc_full);
  }

  // --------------------------------------------------------------- epilogue --
  // thread r holds output row m0 + r (tensor-memory lane r)
  bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, wc, ST_STD_TIMEOUT)) && !*abort_flag;
  if (ok) {
    tc_fence_after();
    const int row = m0 + warp * 32 + lane;
    const uint32_t col = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t v[32];
      FA_TMEM_LD32(col + cb * 32, v);
      tmem_wait_ld();
      FA_REG_FENCE32(v);
      const int c0 = n0 + cb * 32;
      if (row < p.M) {
        if (OUT_F32) {
          float* dst = static_cast<float*>(p.c) + z * p.c_batch + static_cast<long long>(row) * p.ldc + c0;
          if (c0 + 32 <= p.N && (p.ldc & 3) == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              reinterpret_cast<float4*>(dst)[i] =
                  make_float4(__uint_as_float(v[4 * i]) * p.alpha, __uint_as_float(v[4 * i + 1]) * p.alpha,
                              __uint_as_float(v[4 * i + 2]) * p.alpha, __uint_as_float(v[4 * i + 3]) * p.alpha);
          } else {
            for (int i = 0; i < 32 && c0 + i < p.N; ++i) dst[i] = __uint_as_float(v[i]) * p.alpha;
          }
        } else {
          __nv_bfloat16* dst =
              static_cast<__nv_bfloat16*>(p.c) + z * p.c_batch + static_cast<long long>(row) * p.ldc + c0;
          if (c0 + 32 <= p.N && (p.ldc & 7) == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<uint4*>(dst)[i] = make_uint4(
                  pack_bf16x2(__uint_as_float(v[8 * i]), __uint_as_float(v[8 * i + 1])),
                  pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                  pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                  pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
          } else {
            for (int i = 0; i < 32 && c0 + i < p.N; ++i) dst[i] = __float2bfloat16_rn(__uint_as_float(v[i]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // an aborted CTA may not exit while copies it issued are still landing
    bool drained = true;
    const int n_iss = *issued;
    for (int c = max(0, n_iss - STAGES); c < n_iss; ++c)
      drained &= mbar_wait_drain(full + 8 * (c % STAGES), (c / STAGES) & 1, DRAIN_NS);
    if (!drained) atomicOr(p.status, ST_DRAIN);
  }
  if (warp == 1) {
    // nothing may be in flight on the tensor cores when the CTA frees TMEM
    if (!mbar_wait_drain(acc_full, 0, DRAIN_NS) && lane == 0) atomicOr(p.status, ST_DRAIN);
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

struct StdSoftmaxParams {
  const float* s;           // [BH][Nq][ld] scores (scale already applied)
  __nv_bfloat16* p;         // [BH][Nq][ld] probabilities (columns < Nk written)
  float* lse;               // [BH][Nq] or null
  const int* kv_len;        // [B] or null
  long long ld;
  int BH, H, Nq, Nk;
  int causal, qoff;         // key j visible to query i iff j < i + qoff (causal)
};

// One warp per row, 8 rows per CTA.  Masked entries count as -inf: pass 1 takes
// the row max m, pass 2 the sum l of exp(s - m), pass 3 writes exp(s - m) / l.  A
// row with no visible key gets P = 0 and lse = -inf ("Flash attention and
// efficient attention: Worked examples", Cell D2).
__global__ void __launch_bounds__(256) std_softmax_kernel(const StdSoftmaxParams p) {
  const long long row_id = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row_id >= static_cast<long long>(p.BH) * p.Nq) return;
  const int bh = static_cast<int>(row_id / p.Nq), i = static_cast<int>(row_id % p.Nq);
  int lim = p.Nk;
  if (p.kv_len) lim = min(lim, max(0, p.kv_len[bh / p.H]));
  if (p.causal) lim = min(lim, max(0, i + p.qoff));
  const float* srow = p.s + (static_cast<long long>(bh) * p.Nq + i) * p.ld;
  __nv_bfloat16* prow = p.p + (static_cast<long long>(bh) * p.Nq + i) * p.ld;
  float m = -INFINITY;
  for (int j = lane; j < lim; j += 32) m = fmaxf(m, srow[j]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float l = 0.f;
  if (lim > 0)
    for (int j = lane; j < lim; j += 32) l += expf(srow[j] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  for (int j = lane; j < p.Nk; j += 32)
    prow[j] = __float2bfloat16_rn(j < lim ? expf(srow[j] - m) * inv : 0.f);
  if (p.lse && lane == 0) p.lse[row_id] = (l > 0.f) ? m + logf(l) : -INFINITY;
}

}  // namespace fa
