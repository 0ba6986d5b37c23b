// BFloat16 attention forward on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA computes one 128-row query tile of one (batch, head).  It streams the
// head's keys and values in 128-key tiles and keeps, per query row, the running
// max m, normaliser l and accumulator acc of the online softmax ("The Flash
// Attention" page, online recurrence panel):
//     m_new = max(m, m'),  c = 2^(m - m_new),
//     l <- l c + sum_j 2^(s_j - m_new),   acc <- acc c + sum_j 2^(s_j - m_new) V_j,
//     O = acc / l once at the end, with O = 0 and lse = -inf when l = 0
//     ("Flash attention and efficient attention: Worked examples", Cell D2).
// Scores live in the base-2 domain, s = S * scale * log2(e), so every exponential
// is one ex2.  The N x N score matrix never leaves the SM: S and P exist only as
// one 128 x 128 tile in tensor memory.
//
// Roles (256 threads):
//   warp 0     TMA producer: Q once, then K_j and V_j into a STAGES-deep ring.
//   warp 1     MMA issuer (one thread) and tensor-memory owner:
//                S_j = Q K_j^T    (A, B from shared memory, K-major, 128B swizzle)
//                O  += P_j V_j    (A = P from tensor memory, B = V MN-major)
//   warps 4-7  softmax: thread r owns query row r, which is tensor-memory lane r.
//
// Tensor memory (512 columns, f32 unless noted):
//   [0,128) S buffer 0   [128,256) S buffer 1   [256,256+D) O accumulator
//   [256+D, +64) P buffer 0 (bf16 pairs)   [320+D, +64) P buffer 1
// S is double-buffered so S_{j+1} = Q K_{j+1}^T runs on the tensor cores while
// the softmax warps turn S_j into P_j.
//
// Rescaling is lazy: the running reference m is moved only when a block's max
// exceeds it by more than 8 (base-2 units).  l and acc always share the same
// reference, so O = acc / l is unchanged -- the merge identity of the Exercises
// page ("top and bottom both get multiplied by e^-m, which cancels") -- while the
// tensor-memory round trip that rescales acc is skipped for most blocks.  Terms
// stay below 2^8, far from overflow in f32 and bf16.
#pragma once
#include "ptx.cuh"

namespace fa {

// Bits of the global status word (a timeout names the barrier it gave up on).
enum : unsigned {
  ST_TIMEOUT_Q = 1u << 0,
  ST_TIMEOUT_K = 1u << 1,
  ST_TIMEOUT_V = 1u << 2,
  ST_TIMEOUT_P = 1u << 3,
  ST_TIMEOUT_S = 1u << 4,
  ST_TIMEOUT_O = 1u << 5,
  ST_TIMEOUT_EMPTY = 1u << 6,
  ST_DRAIN = 1u << 7,
};

struct TcParams {
  __nv_bfloat16* o;   // [B, H, N, D]
  float* lse;         // [B, H, N] or null
  const int* kv_len;  // [B] or null
  int BH, H, N;
  int n_qt;           // query tiles per head
  float scale_log2;   // scale * log2(e), > 0
  int causal;
  unsigned* status;
  unsigned long long timeout_ns;
  int inject;         // test hook: 1 = producer stops after the first K/V tile
};

template <int D, int STAGES>
struct TcLayout {
  static constexpr int BM = 128, BN = 128;
  static constexpr int KB = D / 64;                // 64-element (128-byte) column blocks
  static constexpr int COLBLK = 128 * 128;         // bytes of one 128-row column block
  static constexpr int TILE = BM * D * 2;          // bytes of a Q, K or V tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = TILE;
  static constexpr int OFF_V = OFF_K + STAGES * TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * TILE;
  // barriers: q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full[2], o_done, drain
  static constexpr int NBAR = 1 + 3 * STAGES + 2 + 2 + 1 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256;
  static constexpr uint32_t TM_P0 = 256 + D, TM_P1 = 256 + D + 64;
  static constexpr uint32_t TM_COLS = 512;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(TM_P1 + 64 <= TM_COLS, "tensor memory budget");
  static_assert(BYTES <= 232448, "shared memory budget");
};

template <int D, int STAGES>
__global__ void __launch_bounds__(256, 1)
    fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  using L = TcLayout<D, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + STAGES;
  uint64_t* kv_empty = v_full + STAGES;
  uint64_t* s_full = kv_empty + STAGES;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Head-major order: consecutive CTAs share one head's K/V, which then stays in
  // L2; within a head the heaviest causal tiles go first.
  const int bh = static_cast<int>(blockIdx.x) / p.n_qt;
  const int qt = p.n_qt - 1 - static_cast<int>(blockIdx.x) % p.n_qt;
  const int b = bh / p.H;
  const int q0 = qt * L::BM;
  int kv_limit = p.N;
  if (p.kv_len) kv_limit = min(p.N, max(0, p.kv_len[b]));
  int n_kv = (kv_limit + L::BN - 1) / L::BN;
  if (p.causal) n_kv = min(n_kv, qt + 1);  // rows q0..q0+127 see keys <= q0+127

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 128);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
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

  int issued = 0;  // K/V tiles whose loads the producer has issued (warp 0, lane 0)
  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && n_kv > 0) {
      mbar_arrive_expect_tx(q_full, L::TILE);
#pragma unroll
      for (int kb = 0; kb < L::KB; ++kb)
        tma_load_3d(smem + L::OFF_Q + kb * L::COLBLK, &tm_q, q_full, kb * 64, q0, bh);
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % STAGES;
        if (j >= STAGES && !mbar_wait(&kv_empty[st], ((j / STAGES) - 1) & 1, wc, ST_TIMEOUT_EMPTY)) break;
        if (p.inject == 1 && j == 1) break;  // test hook: starve the consumers
        mbar_arrive_expect_tx(&k_full[st], L::TILE);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb)
          tma_load_3d(smem + L::OFF_K + st * L::TILE + kb * L::COLBLK, &tm_k, &k_full[st], kb * 64, j * L::BN, bh);
        mbar_arrive_expect_tx(&v_full[st], L::TILE);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb)
          tma_load_3d(smem + L::OFF_V + st * L::TILE + kb * L::COLBLK, &tm_v, &v_full[st], kb * 64, j * L::BN, bh);
        issued = j + 1;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, true);
      const uint32_t sq = smem_u32(smem + L::OFF_Q);
      const uint32_t sk = smem_u32(smem + L::OFF_K);
      const uint32_t sv = smem_u32(smem + L::OFF_V);

      auto issue_pv = [&](int jj) -> bool {
        const int st = jj % STAGES, pb = jj & 1;
        if (!mbar_wait(&p_full[pb], (jj >> 1) & 1, wc, ST_TIMEOUT_P)) return false;
        if (!mbar_wait(&v_full[st], (jj / STAGES) & 1, wc, ST_TIMEOUT_V)) return false;
        tc_fence_after();
        const uint32_t pt = tmem + (pb ? L::TM_P1 : L::TM_P0);
#pragma unroll
        for (int kk = 0; kk < L::BN / 16; ++kk) {
          // V_j rows kk*16 .. kk*16+15 (2 KB apart per 16 rows); MN blocks 16 KB apart
          const uint64_t bdesc = sdesc_sw128(sv + st * L::TILE + kk * 2048, L::COLBLK, 1024);
          umma_ts(tmem + L::TM_O, pt + kk * 8, bdesc, IDESC_PV, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(o_done);
        umma_commit(&kv_empty[st]);
        return true;
      };

      bool ok = mbar_wait(q_full, 0, wc, ST_TIMEOUT_Q);
      if (ok) tc_fence_after();
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % STAGES;
        if (!mbar_wait(&k_full[st], (j / STAGES) & 1, wc, ST_TIMEOUT_K)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_tm = tmem + ((j & 1) ? L::TM_S1 : L::TM_S0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major operands: 16 elements (32 bytes) per step inside a 128-byte row
          const uint32_t off = (kk >> 2) * L::COLBLK + (kk & 3) * 32;
          const uint64_t adesc = sdesc_sw128(sq + off, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(sk + st * L::TILE + off, 16, 1024);
          umma_ss(s_tm, adesc, bdesc, IDESC_QK, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
        if (j > 0 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(n_kv - 1);
      // nothing may be in flight on the tensor cores when the CTA frees TMEM
      umma_commit(drain);
      if (!mbar_wait_drain(drain, 0, DRAIN_NS)) atomicOr(p.status, ST_DRAIN);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- softmax --
    const int r = threadIdx.x - 128;  // row in the tile == tensor-memory lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int qrow = q0 + r;
    const float sl = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      // tcgen05.ld/st are warp-collective: the whole warp goes on or stops together
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (j >> 1) & 1, wc, ST_TIMEOUT_S))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
      const uint32_t s_col = lane_base + (sb ? L::TM_S1 : L::TM_S0);
      FA_TMEM_LD32(s_col + 0, sr + 0);
      FA_TMEM_LD32(s_col + 32, sr + 32);
      FA_TMEM_LD32(s_col + 64, sr + 64);
      FA_TMEM_LD32(s_col + 96, sr + 96);
      tmem_wait_ld();
      FA_REG_FENCE32(sr + 0);
      FA_REG_FENCE32(sr + 32);
      FA_REG_FENCE32(sr + 64);
      FA_REG_FENCE32(sr + 96);

      const int k0 = j * L::BN;
      if (k0 + L::BN > kv_limit || (p.causal && k0 + L::BN - 1 > q0)) {
        int lim = kv_limit - k0;
        if (p.causal) lim = min(lim, qrow - k0 + 1);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) sr[i] = __float_as_uint(-INFINITY);
      }
      // row max as a tree: 8 independent chains, then combine
      float mx8[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mx8[t] = __uint_as_float(sr[t]);
#pragma unroll
      for (int i = 8; i < 128; i += 8)
#pragma unroll
        for (int t = 0; t < 8; ++t) mx8[t] = fmaxf(mx8[t], __uint_as_float(sr[i + t]));
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_blk = mx * sl;
      const float m_new = (m_blk > m + 8.f) ? m_blk : m;  // lazy reference move
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float c = ex2_approx(m - m_ref);               // 0 on the first block, 1 if unchanged
      float rs4[4] = {0.f, 0.f, 0.f, 0.f};  // row sum in 4 independent chains
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * i]), sl, -m_ref));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * i + 1]), sl, -m_ref));
        rs4[i & 3] += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l = l * c + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
      const uint32_t p_col = lane_base + (sb ? L::TM_P1 : L::TM_P0);
      FA_TMEM_ST32(p_col + 0, pk + 0);
      FA_TMEM_ST32(p_col + 32, pk + 32);
      if (j > 0) {
        // acc holds blocks < j once O += P_{j-1} V_{j-1} has finished
        if (!__all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, wc, ST_TIMEOUT_O))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, m_new != m)) {
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t orr[32];
            FA_TMEM_LD32(lane_base + L::TM_O + cb * 32, orr);
            tmem_wait_ld();
            FA_REG_FENCE32(orr);
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * c);
            FA_TMEM_ST32(lane_base + L::TM_O + cb * 32, orr);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
      m = m_new;
    }

    if (ok && n_kv > 0 && !__all_sync(0xffffffffu, mbar_wait(o_done, (n_kv - 1) & 1, wc, ST_TIMEOUT_O)))
      ok = false;
    if (ok) {
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;  // guard: l = 0 -> zero vector
      const size_t orow = (static_cast<size_t>(bh) * p.N + qrow) * D;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t orr[32];
        if (n_kv > 0) {
          FA_TMEM_LD32(lane_base + L::TM_O + cb * 32, orr);
          tmem_wait_ld();
          FA_REG_FENCE32(orr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = 0u;
        }
        uint32_t ob[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          ob[i] = pack_bf16x2(__uint_as_float(orr[2 * i]) * inv, __uint_as_float(orr[2 * i + 1]) * inv);
        if (qrow < p.N) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + orow + cb * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(ob[4 * i], ob[4 * i + 1], ob[4 * i + 2], ob[4 * i + 3]);
        }
      }
      if (p.lse && qrow < p.N)
        p.lse[static_cast<size_t>(bh) * p.N + qrow] = (l > 0.f) ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && n_kv > 0 && *abort_flag) {
    // an aborted CTA may not exit while copies it issued are still landing
    bool ok = mbar_wait_drain(q_full, 0, DRAIN_NS);
    for (int j = max(0, issued - STAGES); j < issued; ++j) {
      const int st = j % STAGES;
      ok &= mbar_wait_drain(&k_full[st], (j / STAGES) & 1, DRAIN_NS);
      ok &= mbar_wait_drain(&v_full[st], (j / STAGES) & 1, DRAIN_NS);
    }
    if (!ok) atomicOr(p.status, ST_DRAIN);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  }
}

}  // namespace fa
