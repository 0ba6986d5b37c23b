// BFloat16 attention backward on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// The backward pass recomputes the scores and probabilities instead of reading a
// stored N x N matrix ("Question bank -- Flash attention and efficient
// attention", the recomputation items: S and P are rebuilt from Q, K and the
// saved per-row statistics).  With P = softmax(scale Q K^T) and O = P V, the
// chain rule gives, for L = sum(O * dO):
//     dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO_ic O_ic  (= sum_j P_ij dP_ij),
//     dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q.
// P is rebuilt from the forward's lse: P_ij = exp(scale S_ij - lse_i), which is
// already normalised, so no second softmax pass is needed.
//
// Two kernels:
//  * bwd_preprocess_kernel -- D_i and lse2_i = lse_i log2(e) into the workspace
//    (row stride Np = N rounded up to 64; padding rows get D = 0, lse2 = +inf so
//    that their probabilities are exactly 0), and zeroes dQ.
//  * bwd_bf16_tc_kernel -- one CTA per (batch, head, 128-key tile).  K and V stay
//    in shared memory; the CTA streams 64-query tiles (Q_t, dO_t, lse2_t, D_t)
//    through a TMA ring and, per tile t, runs five MMAs:
//       MMA1  S^T_t  = K Q_t^T            (128 x 64, TMEM)
//       MMA2  dP^T_t = V dO_t^T           (128 x 64, TMEM)
//       MMA3  dV    += P^T_t dO_t          (128 x d, TMEM; A = P^T from TMEM)
//       MMA4  dK    += dS^T_t Q_t          (128 x d, TMEM; A = dS^T from SMEM)
//       MMA5  dQ^T_t = K^T dS_t            (d x 64, TMEM; A = K read MN-major)
//    issued in the order MMA3_t, MMA1_{t+1}, MMA2_{t+1}, MMA4_t, MMA5_t so that
//    the next tile's products are queued while tile t's softmax runs.
//    dQ is produced transposed so that TMEM lane = head-dim column: a warp's 32
//    lanes then hold 32 consecutive floats of one query row, and the reduction
//    into global dQ (red.global.add.f32) is one coalesced 128-byte access per
//    warp instruction.  dS carries the factor `scale`, so dK and dQ need no
//    further scaling.
//
// Roles (384 threads):
//   warp 0     TMA producer: K, V once; then Q_t, dO_t (tensor maps) and the
//              lse2_t, D_t rows (bulk copies) into a STAGES-deep ring.
//   warp 1     MMA issuer (one thread) and tensor-memory owner.
//   warps 4-7  elementwise warpgroup 0: even tiles t;  warps 8-11: odd tiles.
//              Thread r owns key row r (TMEM lane r) of S^T and dP^T:
//                P^T = 2^(S^T scale log2e - lse2) with the causal / padding mask,
//                written back to TMEM as bf16 (aliasing S^T), then
//                dS^T = P^T (dP^T - D) scale -> bf16, 128B-swizzled into SMEM,
//              and, as TMEM lane r of dQ^T, adds head-dim column r of the tile's
//              64 dQ rows into global memory.  At the end warpgroup 0 writes dV
//              and warpgroup 1 writes dK.
//
// Tensor memory (512 columns, f32 unless noted):
//   [0,128)   two 64-column buffers, one per tile parity: S^T_t, then P^T_t
//             (bf16, first 32 columns), then dQ^T_t
//   [128,256) two dP^T buffers, one per tile parity
//   [256,384) dV   [384,512) dK
//
// Every wait is bounded, as in the forward kernel: a wait that runs out records
// a status bit, the CTA drains what it has in flight and exits.
#pragma once
#include "ptx.cuh"

namespace fa {

enum : unsigned {
  ST_BWD_TIMEOUT_KV = 1u << 8,
  ST_BWD_TIMEOUT_Q = 1u << 9,
  ST_BWD_TIMEOUT_S = 1u << 10,
  ST_BWD_TIMEOUT_P = 1u << 11,
  ST_BWD_TIMEOUT_DP = 1u << 12,
  ST_BWD_TIMEOUT_DS = 1u << 13,
  ST_BWD_TIMEOUT_DQ = 1u << 14,
  ST_BWD_TIMEOUT_DQE = 1u << 15,
  ST_BWD_TIMEOUT_EMPTY = 1u << 16,
  ST_BWD_TIMEOUT_DONE = 1u << 17,
};

struct BwdPreParams {
  const __nv_bfloat16* o;   // [BH, N, D]
  const __nv_bfloat16* dO;  // [BH, N, D]
  const float* lse;         // [BH, N]
  float* dq;                // [BH, N, D], zeroed here
  float* lse2;              // workspace [BH, Np]
  float* dd;                // workspace [BH, Np]
  int BH, N, Np;
};

// One warp per row: D = sum_c dO_c O_c (f32), lse2 = lse * log2(e) (+inf where
// lse = -inf or the row is padding), dq row = 0.  Grid: BH * Np / 64 blocks of
// 256 threads, 8 rows per warp.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdPreParams p) {
  constexpr int EPL = D / 32;  // elements per lane
  const int chunks = p.Np / 64;
  const int bh = static_cast<int>(blockIdx.x) / chunks;
  const int row0 = (static_cast<int>(blockIdx.x) % chunks) * 64 + (threadIdx.x >> 5) * 8;
  const int lane = threadIdx.x & 31;
  for (int rr = 0; rr < 8; ++rr) {
    const int row = row0 + rr;
    const size_t ws = static_cast<size_t>(bh) * p.Np + row;
    if (row >= p.N) {
      if (lane == 0) {
        p.lse2[ws] = INFINITY;
        p.dd[ws] = 0.f;
      }
      continue;
    }
    const size_t base = (static_cast<size_t>(bh) * p.N + row) * D + lane * EPL;
    float acc = 0.f;
    if constexpr (EPL == 4) {
      const uint2 a = *reinterpret_cast<const uint2*>(p.o + base);
      const uint2 g = *reinterpret_cast<const uint2*>(p.dO + base);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 af = __bfloat1622float2(a2[i]), gf = __bfloat1622float2(g2[i]);
        acc = fmaf(af.x, gf.x, acc);
        acc = fmaf(af.y, gf.y, acc);
      }
      *reinterpret_cast<float4*>(p.dq + base) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(p.o + base);
      const __nv_bfloat162 g = *reinterpret_cast<const __nv_bfloat162*>(p.dO + base);
      const float2 af = __bfloat1622float2(a), gf = __bfloat1622float2(g);
      acc = fmaf(af.x, gf.x, fmaf(af.y, gf.y, 0.f));
      *reinterpret_cast<float2*>(p.dq + base) = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const float l = p.lse[static_cast<size_t>(bh) * p.N + row];
      p.lse2[ws] = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
      p.dd[ws] = acc;
    }
  }
}

struct BwdParams {
  float* dq;                // [BH, N, D], accumulated with red.add
  float* dk;                // [BH, N, D]
  float* dv;                // [BH, N, D]
  const float* lse2;        // [BH, Np]
  const float* dd;          // [BH, Np]
  const int* kv_len;        // [B] or null
  int BH, H, N, Np;
  int n_kt;                 // key tiles per head
  float scale;              // score multiplier
  float scale_log2;         // scale * log2(e)
  int causal;               // 0 none, 1 key k visible iff k <= row, 2 iff k < row
  unsigned* status;
  unsigned long long timeout_ns;
};

template <int STAGES>
struct BwdLayout {
  static constexpr int D = 128;
  static constexpr int BN = 128;                   // keys per CTA
  static constexpr int BM = 64;                    // queries per tile
  static constexpr int KB = D / 64;                // 128-byte column blocks
  static constexpr int KV_COLBLK = BN * 128;       // 16 KB
  static constexpr int KV_TILE = BN * D * 2;       // 32 KB
  static constexpr int Q_COLBLK = BM * 128;        // 8 KB
  static constexpr int Q_TILE = BM * D * 2;        // 16 KB
  static constexpr int DS_TILE = BN * BM * 2;      // 16 KB: 128 key rows x 128 bytes
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_TILE;
  static constexpr int OFF_Q = 2 * KV_TILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_TILE;
  static constexpr int OFF_DS = OFF_DO + STAGES * Q_TILE;
  static constexpr int OFF_LSE = OFF_DS + 2 * DS_TILE;
  static constexpr int OFF_DD = OFF_LSE + STAGES * BM * 4;
  static constexpr int OFF_BAR = OFF_DD + STAGES * BM * 4;
  // barriers: kv_full, q_full[S], q_empty[S], s_full[2], p_full[2], dp_full[2],
  //           ds_full[2], dq_full[2], dq_empty, dkv_done, drain
  static constexpr int NBAR = 1 + 2 * STAGES + 2 * 5 + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 384, TM_COLS = 512;
  static constexpr uint32_t Q_TX = 2 * Q_TILE + 2 * BM * 4;
  static_assert(BYTES <= 232448, "shared memory budget");
};

template <int STAGES>
__global__ void __launch_bounds__(384, 1)
    bwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using L = BwdLayout<STAGES>;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = kv_full + 1;
  uint64_t* q_empty = q_full + STAGES;
  uint64_t* s_full = q_empty + STAGES;
  uint64_t* p_full = s_full + 2;
  uint64_t* dp_full = p_full + 2;
  uint64_t* ds_full = dp_full + 2;
  uint64_t* dq_full = ds_full + 2;
  uint64_t* dq_empty = dq_full + 2;
  uint64_t* dkv_done = dq_empty + 1;
  uint64_t* drain = dkv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // head-major; within a head the key tiles with the most query tiles first
  const int bh = static_cast<int>(blockIdx.x) / p.n_kt;
  const int kt = static_cast<int>(blockIdx.x) % p.n_kt;
  const int b = bh / p.H;
  const int k0 = kt * L::BN;
  int kv_limit = p.N;
  if (p.kv_len) kv_limit = min(p.N, max(0, p.kv_len[b]));
  const int n_qt = (p.N + L::BM - 1) / L::BM;
  const int i0 = p.causal ? k0 / L::BM : 0;  // first query tile that sees a key of this tile
  const int n_it = (k0 < kv_limit) ? n_qt - i0 : 0;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 128);
      mbar_init(&dp_full[s], 1);
      mbar_init(&ds_full[s], 128);
      mbar_init(&dq_full[s], 1);
    }
    mbar_init(dq_empty, 128);
    mbar_init(dkv_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
  constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;

  int issued = 0;  // query tiles whose loads the producer has issued
  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && n_it > 0) {
      mbar_arrive_expect_tx(kv_full, 2 * L::KV_TILE);
#pragma unroll
      for (int kb = 0; kb < L::KB; ++kb) {
        tma_load_3d(smem + L::OFF_K + kb * L::KV_COLBLK, &tm_k, kv_full, kb * 64, k0, bh);
        tma_load_3d(smem + L::OFF_V + kb * L::KV_COLBLK, &tm_v, kv_full, kb * 64, k0, bh);
      }
      for (int t = 0; t < n_it; ++t) {
        const int st = t % STAGES;
        if (t >= STAGES && !mbar_wait(&q_empty[st], ((t / STAGES) - 1) & 1, wc, ST_BWD_TIMEOUT_EMPTY)) break;
        const int q0 = (i0 + t) * L::BM;
        mbar_arrive_expect_tx(&q_full[st], L::Q_TX);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
          tma_load_3d(smem + L::OFF_Q + st * L::Q_TILE + kb * L::Q_COLBLK, &tm_q, &q_full[st], kb * 64, q0, bh);
          tma_load_3d(smem + L::OFF_DO + st * L::Q_TILE + kb * L::Q_COLBLK, &tm_do, &q_full[st], kb * 64, q0, bh);
        }
        const size_t ws = static_cast<size_t>(bh) * p.Np + q0;
        bulk_load(smem + L::OFF_LSE + st * L::BM * 4, p.lse2 + ws, L::BM * 4, &q_full[st]);
        bulk_load(smem + L::OFF_DD + st * L::BM * 4, p.dd + ws, L::BM * 4, &q_full[st]);
        issued = t + 1;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0 && n_it > 0) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(128, L::BM, false, false);  // K Q^T, V dO^T
      constexpr uint32_t IDESC_G = idesc_bf16_f32(128, D, true, false);       // P^T dO, dS^T Q
      constexpr uint32_t IDESC_Q = idesc_bf16_f32(D, L::BM, true, true);      // K^T dS
      const uint32_t sk = smem_u32(smem + L::OFF_K), sv = smem_u32(smem + L::OFF_V);
      const uint32_t sq = smem_u32(smem + L::OFF_Q), sdo = smem_u32(smem + L::OFF_DO);
      const uint32_t sds = smem_u32(smem + L::OFF_DS);

      // S^T_t (or dP^T_t): A = K (or V) K-major, B = Q_t (or dO_t) K-major
      auto mma_scores = [&](uint32_t d_tm, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t adesc = sdesc_sw128(a_base + (kk >> 2) * L::KV_COLBLK + (kk & 3) * 32, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(b_base + (kk >> 2) * L::Q_COLBLK + (kk & 3) * 32, 16, 1024);
          umma_ss(d_tm, adesc, bdesc, IDESC_S, kk > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(kv_full, 0, wc, ST_BWD_TIMEOUT_KV);
      if (ok) ok = mbar_wait(&q_full[0], 0, wc, ST_BWD_TIMEOUT_Q);
      if (ok) {
        tc_fence_after();
        mma_scores(tmem + L::TM_S, sk, sq);
        umma_commit(&s_full[0]);
        mma_scores(tmem + L::TM_DP, sv, sdo);
        umma_commit(&dp_full[0]);
      }
      // Issue order per tile t: MMA3_t, then S and dP of tile t+1, then MMA4_t and
      // MMA5_t.  The elementwise warps build P_t and dS_t while the tensor cores
      // work on the queued products, so the pipe never waits on one tile's
      // softmax before it can start the next tile's scores.
      for (int t = 0; ok && t < n_it; ++t) {
        const int st = t % STAGES, pb = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        const int t1 = t + 1, st1 = t1 % STAGES;
        // MMA3: dV += P^T_t dO_t   (A = P^T bf16 in TMEM, B = dO_t MN-major)
        if (!mbar_wait(&p_full[pb], ph, wc, ST_BWD_TIMEOUT_P)) break;
        tc_fence_after();
        {
          const uint32_t pt = tmem + L::TM_S + pb * 64;
#pragma unroll
          for (int kk = 0; kk < L::BM / 16; ++kk) {
            const uint64_t bdesc = sdesc_sw128(sdo + st * L::Q_TILE + kk * 2048, L::Q_COLBLK, 1024);
            umma_ts(tmem + L::TM_DV, pt + kk * 8, bdesc, IDESC_G, (t > 0 || kk > 0) ? 1u : 0u);
          }
        }
        // S^T_{t+1} and dP^T_{t+1}.  Buffer (t+1)&1 last held dQ^T_{t-1}, which
        // its warpgroup must have read out; dP buffer (t+1)&1 held dP^T_{t-1},
        // read before dS_{t-1} was published (waited for at tile t-1).
        if (t1 < n_it) {
          if (!mbar_wait(&q_full[st1], (t1 / STAGES) & 1, wc, ST_BWD_TIMEOUT_Q)) break;
          if (t >= 1 && !mbar_wait(dq_empty, (t - 1) & 1, wc, ST_BWD_TIMEOUT_DQE)) break;
          tc_fence_after();
          mma_scores(tmem + L::TM_S + (t1 & 1) * 64, sk, sq + st1 * L::Q_TILE);
          umma_commit(&s_full[t1 & 1]);
          mma_scores(tmem + L::TM_DP + (t1 & 1) * 64, sv, sdo + st1 * L::Q_TILE);
          umma_commit(&dp_full[t1 & 1]);
        }
        // MMA4: dK += dS^T_t Q_t   (A = dS^T K-major in SMEM, B = Q_t MN-major)
        if (!mbar_wait(&ds_full[pb], ph, wc, ST_BWD_TIMEOUT_DS)) break;
        tc_fence_after();
        const uint32_t ds_base = sds + pb * L::DS_TILE;
#pragma unroll
        for (int kk = 0; kk < L::BM / 16; ++kk) {
          const uint64_t adesc = sdesc_sw128(ds_base + kk * 32, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(sq + st * L::Q_TILE + kk * 2048, L::Q_COLBLK, 1024);
          umma_ss(tmem + L::TM_DK, adesc, bdesc, IDESC_G, (t > 0 || kk > 0) ? 1u : 0u);
        }
        // MMA5: dQ^T_t = K^T dS_t into S buffer pb (P_t there was consumed by
        // MMA3_t, which the tensor cores finish first: they run in issue order).
        // A = K MN-major, B = dS^T read as [query][key] MN-major.
#pragma unroll
        for (int kk = 0; kk < L::BN / 16; ++kk) {
          const uint64_t adesc = sdesc_sw128(sk + kk * 2048, L::KV_COLBLK, 1024);
          const uint64_t bdesc = sdesc_sw128(ds_base + kk * 2048, L::DS_TILE, 1024);
          umma_ss(tmem + L::TM_S + pb * 64, adesc, bdesc, IDESC_Q, kk > 0 ? 1u : 0u);
        }
        umma_commit(&dq_full[pb]);
        umma_commit(&q_empty[st]);
      }
      umma_commit(dkv_done);
      // nothing may be in flight on the tensor cores when the CTA frees TMEM
      umma_commit(drain);
      if (!mbar_wait_drain(drain, 0, DRAIN_NS)) atomicOr(p.status, ST_DRAIN);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------- elementwise WGs --
    const int wg = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;  // TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool key_ok = (k0 + r) < kv_limit;
    const float sl = p.scale_log2, scale = p.scale;
    const uint32_t ds_row = smem_u32(smem + L::OFF_DS) + r * 128;
    bool ok = true;
    for (int t = wg; t < n_it; t += 2) {
      const int st = t % STAGES, pb = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      const int q0 = (i0 + t) * L::BM;
      if (!__all_sync(0xffffffffu, mbar_wait(&q_full[st], (t / STAGES) & 1, wc, ST_BWD_TIMEOUT_Q) &&
                                       mbar_wait(&s_full[pb], ph, wc, ST_BWD_TIMEOUT_S))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      const uint32_t s_col = lane_base + L::TM_S + pb * 64;
      FA_TMEM_LD32(s_col + 0, sr + 0);
      FA_TMEM_LD32(s_col + 32, sr + 32);
      tmem_wait_ld();
      FA_REG_FENCE32(sr + 0);
      FA_REG_FENCE32(sr + 32);
      const float* lse2 = reinterpret_cast<const float*>(smem + L::OFF_LSE + st * L::BM * 4);
      const float* dd = reinterpret_cast<const float*>(smem + L::OFF_DD + st * L::BM * 4);
      // causal: key k0 + r is visible to query q0 + j iff j >= r - (q0 - k0), one
      // later in the strict mode (a query does not see its own key)
      const int jmin = p.causal ? r - (q0 - k0) + (p.causal == 2 ? 1 : 0) : -1;
      float pr[64];
#pragma unroll
      for (int j4 = 0; j4 < 64; j4 += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lse2 + j4);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j4 + u;
          const float e = ex2_approx(fmaf(__uint_as_float(sr[j]), sl, -lv[u]));
          pr[j] = (key_ok && j >= jmin) ? e : 0.f;
        }
      }
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(pr[2 * i], pr[2 * i + 1]);
      FA_TMEM_ST32(s_col, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[pb]);

      if (!__all_sync(0xffffffffu, mbar_wait(&dp_full[pb], ph, wc, ST_BWD_TIMEOUT_DP))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dpr[64];
      FA_TMEM_LD32(lane_base + L::TM_DP + pb * 64 + 0, dpr + 0);
      FA_TMEM_LD32(lane_base + L::TM_DP + pb * 64 + 32, dpr + 32);
      tmem_wait_ld();
      FA_REG_FENCE32(dpr + 0);
      FA_REG_FENCE32(dpr + 32);
      uint32_t dsk[32];
#pragma unroll
      for (int j4 = 0; j4 < 64; j4 += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(dd + j4);
        const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
        float g[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) g[u] = pr[j4 + u] * (__uint_as_float(dpr[j4 + u]) - dv4[u]) * scale;
        dsk[j4 / 2] = pack_bf16x2(g[0], g[1]);
        dsk[j4 / 2 + 1] = pack_bf16x2(g[2], g[3]);
      }
      // row r of the 128B-swizzled K-major tile: 16-byte chunk c lands at c ^ (r & 7)
      const uint32_t row_addr = ds_row + pb * L::DS_TILE;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(row_addr + ((c ^ (r & 7)) << 4), dsk[4 * c], dsk[4 * c + 1], dsk[4 * c + 2], dsk[4 * c + 3]);
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&ds_full[pb]);

      // dQ^T_t: lane r holds head-dim column r of query rows q0 .. q0+63
      if (!__all_sync(0xffffffffu, mbar_wait(&dq_full[pb], ph, wc, ST_BWD_TIMEOUT_DQ))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t qr[64];
      FA_TMEM_LD32(s_col + 0, qr + 0);
      FA_TMEM_LD32(s_col + 32, qr + 32);
      tmem_wait_ld();
      FA_REG_FENCE32(qr + 0);
      FA_REG_FENCE32(qr + 32);
      tc_fence_before();
      mbar_arrive(dq_empty);
      float* dst = p.dq + (static_cast<size_t>(bh) * p.N + q0) * D + r;
      const int jn = min(64, p.N - q0);
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j < jn) red_add_f32(dst + static_cast<size_t>(j) * D, __uint_as_float(qr[j]));
    }

    // ------------------------------------------------------------ epilogue --
    // warpgroup 0 writes dV, warpgroup 1 writes dK: TMEM lane r = key row k0 + r
    if (ok && n_it > 0 && !__all_sync(0xffffffffu, mbar_wait(dkv_done, 0, wc, ST_BWD_TIMEOUT_DONE))) ok = false;
    if (ok) {
      tc_fence_after();
      const int key = k0 + r;
      float* out = (wg == 0 ? p.dv : p.dk) + (static_cast<size_t>(bh) * p.N + key) * D;
      const uint32_t col = lane_base + (wg == 0 ? L::TM_DV : L::TM_DK);
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t v[32];
        if (n_it > 0) {
          FA_TMEM_LD32(col + cb * 32, v);
          tmem_wait_ld();
          FA_REG_FENCE32(v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (key < p.N) {
          float4* o4 = reinterpret_cast<float4*>(out + cb * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && n_it > 0 && *abort_flag) {
    // an aborted CTA may not exit while copies it issued are still landing
    bool ok = mbar_wait_drain(kv_full, 0, DRAIN_NS);
    for (int t = max(0, issued - STAGES); t < issued; ++t)
      ok &= mbar_wait_drain(&q_full[t % STAGES], (t / STAGES) & 1, DRAIN_NS);
    if (!ok) atomicOr(p.status, ST_DRAIN);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  }
}

}  // namespace fa
