// BFloat16 attention forward on the 5th-generation tensor cores (tcgen05, sm_103a),
// two query tiles per CTA.
//
// One CTA computes query tiles 2p and 2p+1 (256 rows) of one (batch, head).  Both
// tiles stream the same key/value tiles, so each K_j, V_j is loaded once for two
// tiles.  Each tile keeps, per query row, the running max m, normaliser l and
// accumulator acc of the online softmax ("The Flash Attention" page, online
// recurrence panel):
//     m_new = max(m, m'),  c = 2^(m - m_new),
//     l <- l c + sum_j 2^(s_j - m_new),   acc <- acc c + sum_j 2^(s_j - m_new) V_j,
//     O = acc / l once at the end, with O = 0 and lse = -inf when l = 0
//     ("Flash attention and efficient attention: Worked examples", Cell D2).
// Scores live in the base-2 domain, s = S * scale * log2(e), so every exponential
// is one ex2.  The N x N score matrix never leaves the SM.
//
// Why two tiles: with one tile the tensor cores idle while that tile's softmax
// runs, because the next product O += P V needs its result.  Here the MMA warp
// issues S0_j, S1_j, then alternates PV0_j, S0_{j+1}, PV1_j, S1_{j+1}, ...: while
// one warpgroup turns S into P, the tensor cores work on the other tile.
//
// Roles (384 threads; warps 10-11 only join the start and the end):
//   warps 0-3   softmax of tile 0: thread r owns row r = tensor-memory lane r
//   warps 4-7   softmax of tile 1
//   warp 8      TMA producer: Q0, Q1 once, then K_j, V_j through a ring of NS slots
//   warp 9      MMA issuer (lane 0 of the converged warp) and tensor-memory owner
//
// Tensor memory (512 columns, f32 unless noted):
//   [0,128) S0, then P0 (bf16 pairs in its first 64 columns)   [128,256) S1 / P1
//   [256,256+D) O0 accumulator   [256+D,256+2D) O1 accumulator
// P_j aliases S_j: the tensor cores run in issue order, so S_{j+1}, issued after
// PV_j, overwrites P_j only once PV_j has read it.
//
// Rescaling is lazy: a row's reference m moves only when a block's max exceeds it
// by more than 8 (base 2).  l and acc always share the reference, so acc / l is
// unchanged -- the cancellation argument of the Exercises page: numerator and
// denominator carry the same factor e^-m -- and the O round trip through tensor
// memory happens only for blocks that move the reference.  Terms stay below 2^8.
#pragma once
#include "exp2_poly.cuh"
#include "ptx.cuh"

// Every FA_FWD_EXP2_FMA_EVERY-th pair of scores takes its exponentials on the FMA
// pipe (exp2_fma2) instead of the special-function unit; 0 = none.
#ifndef FA_FWD_EXP2_FMA_EVERY
#define FA_FWD_EXP2_FMA_EVERY 0
#endif

namespace fa {

// Pair i of each 16-pair quarter of a row takes the FMA-pipe exponential.
__host__ __device__ constexpr bool exp2_on_fma(int i) {
  return FA_FWD_EXP2_FMA_EVERY > 0 && (i + 1) % (FA_FWD_EXP2_FMA_EVERY > 0 ? FA_FWD_EXP2_FMA_EVERY : 1) == 0;
}

// Register shares (launch: 384 threads x 168): warpgroup 2 (producer, MMA issuer,
// two idle warps) keeps FWD_REGS_LOW, the two softmax warpgroups get
// FWD_REGS_HIGH; 128 x 56 + 256 x 208 = 60416 <= 64512.
constexpr uint32_t FWD_REGS_LOW = 56, FWD_REGS_HIGH = 208;
static_assert(128 * FWD_REGS_LOW + 256 * FWD_REGS_HIGH <= 384 * 168, "register split exceeds the launch");

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
  int Nk;             // keys per head (N is the number of queries)
  int n_qt;           // query tiles per head
  float scale_log2;   // scale * log2(e), > 0
  int causal;         // 0 none, 1 key k visible iff k <= row, 2 iff k < row
  int qoff;           // causal: key k is visible to query row i iff k < i + qoff, where
                      // qoff = (Nk - N) + 1 (causal 1) or (Nk - N) (causal 2, strict)
  unsigned* status;
  unsigned long long timeout_ns;
  int inject;         // test hook: 1 = producer stops after the first K/V tile
};


// NS = number of K/V slots: K_j and V_j stream through one ring of tile-sized
// slots in the order K_0, V_0, K_1, V_1, ...; load number c (K_j: c = 2j, V_j:
// c = 2j + 1) uses slot c % NS.
template <int D, int NS>
struct TcLayout {
  static constexpr int BM = 128, BN = 128;
  static constexpr int KB = D / 64;           // 64-element (128-byte) column blocks
  static constexpr int COLBLK = 128 * 128;    // bytes of one 128-row column block
  static constexpr int TILE = BM * D * 2;     // bytes of a Q, K or V tile
  static constexpr int OFF_Q = 0;             // Q0, Q1
  static constexpr int OFF_KV = 2 * TILE;     // NS slots
  static constexpr int OFF_BAR = OFF_KV + NS * TILE;
  // barriers: q_full, kv_full[NS], kv_empty[NS], s_full[2], p_full[2], o_done[2], drain
  static constexpr int NBAR = 1 + 2 * NS + 6 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 256 + D, TM_COLS = 512;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BYTES <= 232448, "shared memory budget");
};

template <int D, int NS>
__global__ void __launch_bounds__(384, 1)
    fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  using L = TcLayout<D, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;         // [NS]
  uint64_t* kv_empty = kv_full + NS;    // [NS]
  uint64_t* s_full = kv_empty + NS;     // [2], one per query tile
  uint64_t* p_full = s_full + 2;        // [2]
  uint64_t* o_done = p_full + 2;        // [2]
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Head-major order: consecutive CTAs share one head's K/V in L2; within a head
  // the pairs with the most key tiles (causal) go first.
  const int n_pair = (p.n_qt + 1) >> 1;
  const int bh = static_cast<int>(blockIdx.x) / n_pair;
  const int pr = n_pair - 1 - static_cast<int>(blockIdx.x) % n_pair;
  const int b = bh / p.H;
  const int q0 = pr * 2 * L::BM;  // first row of tile 0; tile 1 starts at q0 + 128
  int kv_limit = p.Nk;
  if (p.kv_len) kv_limit = min(p.Nk, max(0, p.kv_len[b]));
  const int n_kv_all = (kv_limit + L::BN - 1) / L::BN;
  // key tiles query tile qt needs (0 for a tile entirely past N): under a causal
  // mask, up to the tile holding the last key its last row can see
  auto tiles = [&](int qt) -> int {
    if (qt >= p.n_qt) return 0;
    if (!p.causal) return n_kv_all;
    const int last_key = min(qt * L::BM + L::BM, p.N) - 1 + p.qoff - 1;
    return last_key < 0 ? 0 : min(n_kv_all, last_key / L::BN + 1);
  };
  const int n_t0 = tiles(2 * pr), n_t1 = tiles(2 * pr + 1);
  const int n_max = max(n_t0, n_t1);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8) = 0;
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, L::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
  constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;

  // K/V loads (c = 0, 1, ...) the producer has issued; kept in shared memory so
  // that it holds no register in the other roles
  volatile int* issued = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);
  if (warp == 8) {
    reg_lower<FWD_REGS_LOW>();
    // ------------------------------------------------------------ producer --
    if (lane == 0 && n_max > 0) {
      const int nq = (n_t1 > 0) ? 2 : 1;
      mbar_arrive_expect_tx(q_full, nq * L::TILE);
      for (int i = 0; i < nq; ++i)
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb)
          tma_load_3d(smem + L::OFF_Q + i * L::TILE + kb * L::COLBLK, &tm_q, q_full, kb * 64, q0 + i * L::BM, bh);
      for (int c = 0; c < 2 * n_max; ++c) {
        const int slot = c % NS;
        if (c >= NS && !mbar_wait(&kv_empty[slot], ((c / NS) - 1) & 1, wc, ST_TIMEOUT_EMPTY)) break;
        if (p.inject == 1 && c == 2) break;  // test hook: starve the consumers after K_0, V_0
        mbar_arrive_expect_tx(&kv_full[slot], L::TILE);
        const CUtensorMap* src = (c & 1) ? &tm_v : &tm_k;
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb)
          tma_load_3d(smem + L::OFF_KV + slot * L::TILE + kb * L::COLBLK, src, &kv_full[slot], kb * 64,
                      (c >> 1) * L::BN, bh);
        *issued = c + 1;
      }
    }
  } else if (warp == 9) {
    reg_lower<FWD_REGS_LOW>();
    // ---------------------------------------------------------- MMA issuer --
    // the whole warp runs the issue code; lane 0 issues (see umma_ss_w)
    if (n_max > 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, true);
      const uint32_t sq = smem_u32(smem + L::OFF_Q);
      const uint32_t skv = smem_u32(smem + L::OFF_KV);
      // Descriptors of the tile bases; an operand at byte offset `off` from a
      // base is that descriptor plus off >> 4 (the start-address field is the
      // low 14 bits and every shared address here is below 2^18, so no carry).
      const uint64_t dq_base = sdesc_sw128(sq, 16, 1024);
      const uint64_t dk_base = sdesc_sw128(skv, 16, 1024);
      const uint64_t dv_base = sdesc_sw128(skv, L::COLBLK, 1024);
      auto issue_s = [&](uint32_t tm_s, uint32_t q_off, uint64_t* bar, int j) {  // S_i = Q_i K_j^T
        const uint64_t ka = dk_base + ((((2 * j) % NS) * L::TILE) >> 4);
        const uint64_t qa = dq_base + (q_off >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::COLBLK + (kk & 3) * 32) >> 4;
          umma_ss_w(tm_s, qa + off, ka + off, IDESC_QK, kk > 0 ? 1u : 0u);
        }
        umma_commit_w(bar);
      };
      // O_i += P_i V_j.  Only the tile's last product signals o_done (for the
      // epilogue): an earlier PV_i(j-1) is known complete once S_i(j), issued
      // after it, has signalled s_full, because a commit tracks every earlier
      // tensor-core operation of this thread.
      auto issue_pv = [&](uint32_t tm_o, uint32_t tm_p, uint64_t* bar, int j, bool last) {
        const uint64_t va = dv_base + ((((2 * j + 1) % NS) * L::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < L::BN / 16; ++kk)
          umma_ts_w(tm_o, tm_p + kk * 8, va + (kk * 2048 >> 4), IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        if (last) umma_commit_w(bar);
      };
      const uint32_t tS0 = tmem + L::TM_S0, tS1 = tmem + L::TM_S1;
      const uint32_t tO0 = tmem + L::TM_O0, tO1 = tmem + L::TM_O1;

      bool ok = mbar_wait_w(q_full, 0, wc, ST_TIMEOUT_Q) && mbar_wait_w(&kv_full[0], 0, wc, ST_TIMEOUT_K);
      if (ok) {
        tc_fence_after();
        if (n_t0 > 0) issue_s(tS0, 0, &s_full[0], 0);
        if (n_t1 > 0) issue_s(tS1, L::TILE, &s_full[1], 0);
        umma_commit_w(&kv_empty[0]);
      }
      for (int j = 0; ok && j < n_max; ++j) {
        const int j1 = j + 1;
        const int cv = 2 * j + 1, ck = 2 * j1;  // load numbers of V_j and K_{j+1}
        // every tile that reads K_{j+1} or V_j waits for it once, before its first use
        bool k1_ready = false, v_ready = false;
        auto wait_v = [&]() -> bool {
          if (v_ready) return true;
          v_ready = mbar_wait_w(&kv_full[cv % NS], (cv / NS) & 1, wc, ST_TIMEOUT_V);
          return v_ready;
        };
        auto wait_k1 = [&]() -> bool {
          if (k1_ready) return true;
          k1_ready = mbar_wait_w(&kv_full[ck % NS], (ck / NS) & 1, wc, ST_TIMEOUT_K);
          if (k1_ready) tc_fence_after();
          return k1_ready;
        };
        // tile 0: PV0_j, then S0_{j+1}
        if (j < n_t0) {
          if (!wait_v() || !mbar_wait_w(&p_full[0], j & 1, wc, ST_TIMEOUT_P)) break;
          tc_fence_after();
          issue_pv(tO0, tS0, &o_done[0], j, j + 1 == n_t0);
        }
        if (j1 < n_t0) {
          if (!wait_k1()) break;
          issue_s(tS0, 0, &s_full[0], j1);
        }
        // tile 1: PV1_j, then S1_{j+1}
        if (j < n_t1) {
          if (!wait_v() || !mbar_wait_w(&p_full[1], j & 1, wc, ST_TIMEOUT_P)) break;
          tc_fence_after();
          issue_pv(tO1, tS1, &o_done[1], j, j + 1 == n_t1);
        }
        if (j1 < n_t1) {
          if (!wait_k1()) break;
          issue_s(tS1, L::TILE, &s_full[1], j1);
        }
        umma_commit_w(&kv_empty[cv % NS]);                 // V_j: read by every PV above
        if (j1 < n_max) umma_commit_w(&kv_empty[ck % NS]);  // K_{j+1}: read by every S above
      }
      // nothing may be in flight on the tensor cores when the CTA frees TMEM
      umma_commit_w(drain);
      if (!mbar_wait_drain(drain, 0, DRAIN_NS) && lane == 0) atomicOr(p.status, ST_DRAIN);
    }
  } else if (warp < 8) {
    reg_raise<FWD_REGS_HIGH>();
    // ------------------------------------------------------------- softmax --
    const int ti = warp >> 2;          // query tile 0 or 1 (warps 10-11 have no role)
    const int r = threadIdx.x & 127;   // row in the tile == tensor-memory lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + (ti ? L::TM_S1 : L::TM_S0);
    const uint32_t o_col = lane_base + (ti ? L::TM_O1 : L::TM_O0);
    // key k is visible to this row iff k < qlim (causal modes)
    const int qlim = q0 + ti * L::BM + r + p.qoff;
    const int n_kv = ti ? n_t1 : n_t0;
    const int qt0c = q0 + ti * L::BM + p.qoff;  // qlim of the tile's first row
    const float sl = p.scale_log2;
    // l: the row sum of the probabilities as computed (float32), for lse;
    // dl: how much the bf16 values the P V product uses differ from them, for
    // the largest probability of each block (see below)
    float m = -INFINITY, l = 0.f, dl = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      // tcgen05.ld/st are warp-collective: the whole warp goes on or stops together
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[ti], j & 1, wc, ST_TIMEOUT_S))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
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
      // causal: key k visible iff k < row + qoff
      if (k0 + L::BN > kv_limit || (p.causal && k0 + L::BN > qt0c)) {
        int lim = kv_limit - k0;
        if (p.causal) lim = min(lim, qlim - k0);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) sr[i] = __float_as_uint(-INFINITY);
      }
      // row max: 8 independent chains of three-input max
      float mx8[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mx8[t] = fmaxf(__uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1]));
#pragma unroll
      for (int i = 16; i < 128; i += 16)
#pragma unroll
        for (int t = 0; t < 8; ++t)
          mx8[t] = fmax3(mx8[t], __uint_as_float(sr[i + 2 * t]), __uint_as_float(sr[i + 2 * t + 1]));
      const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      const float m_blk = mx * sl;
      const float m_new = (m_blk > m + 8.f) ? m_blk : m;  // lazy reference move
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float c = ex2_approx(m - m_ref);               // 0 on the first block, 1 if unchanged
      // The product O += P V sees P rounded to bf16.  A row whose weight sits on
      // one key (large logits) then has O = v (p~ / p): off by up to 2^-9 |v|
      // when p is normalised by the float32 sum.  Adding p~ - p of each block's
      // largest probability (the same fma and ex2 as below, so the same bits)
      // to the normaliser of O makes that term exact; lse keeps the float32 sum.
      const float p_mx = ex2_approx(fmaf(mx, sl, -m_ref));
      dl = dl * c + (__bfloat162float(__float2bfloat16_rn(p_mx)) - p_mx);
      // x = s * scale*log2(e) - m_ref two scores at a time (f32x2), p = 2^x, row
      // sum in 4 independent chains; P in quarters of 32 scores (16 packed
      // columns) keeps register use low
      const uint64_t sl2 = f2_pack(sl, sl), nm2 = f2_pack(-m_ref, -m_ref);
      // row sum in two f32x2 chains: one packed add per pair of scores
      uint64_t rs2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t x2 =
              f2_fma(f2_pack(__uint_as_float(sr[32 * h + 2 * i]), __uint_as_float(sr[32 * h + 2 * i + 1])), sl2, nm2);
          uint64_t p2;
          if (exp2_on_fma(i)) {
            p2 = exp2_fma2(x2);  // this pair on the FMA pipe
          } else {
            float x0, x1;
            f2_unpack(x2, x0, x1);
            p2 = f2_pack(ex2_approx(x0), ex2_approx(x1));
          }
          rs2[i & 1] = f2_add(rs2[i & 1], p2);
          float p0, p1;
          f2_unpack(p2, p0, p1);
          pk[i] = pack_bf16x2(p0, p1);
        }
        FA_TMEM_ST16(s_col + 16 * h, pk);
      }
      float ra, rb, rc, rd;
      f2_unpack(rs2[0], ra, rb);
      f2_unpack(rs2[1], rc, rd);
      l = l * c + ((ra + rb) + (rc + rd));
      if (j > 0 && __any_sync(0xffffffffu, m_new != m)) {
        // The accumulator already holds blocks < j: PV_{j-1} was issued before
        // S_j, and s_full for S_j tracks every earlier tensor-core operation.
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t orr[32];
          FA_TMEM_LD32(o_col + cb * 32, orr);
          tmem_wait_ld();
          FA_REG_FENCE32(orr);
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * c);
          FA_TMEM_ST32(o_col + cb * 32, orr);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[ti]);
      m = m_new;
    }

    if (ok && n_kv > 0 && !__all_sync(0xffffffffu, mbar_wait(&o_done[ti], 0, wc, ST_TIMEOUT_O))) ok = false;
    const int qrow = qlim - p.qoff;
    if (ok && qt0c - p.qoff < p.N) {
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / (l + dl) : 0.f;  // guard: l = 0 -> zero vector
      const size_t orow = (static_cast<size_t>(bh) * p.N + qrow) * D;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t orr[32];
        if (n_kv > 0) {
          FA_TMEM_LD32(o_col + cb * 32, orr);
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
  } else {
    reg_lower<FWD_REGS_LOW>();  // warps 10-11: no role
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8 && lane == 0 && n_max > 0 && *abort_flag) {
    // an aborted CTA may not exit while copies it issued are still landing
    bool ok = mbar_wait_drain(q_full, 0, DRAIN_NS);
    const int n_iss = *issued;
    for (int c = max(0, n_iss - NS); c < n_iss; ++c)
      ok &= mbar_wait_drain(&kv_full[c % NS], (c / NS) & 1, DRAIN_NS);
    if (!ok) atomicOr(p.status, ST_DRAIN);
  }
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  }
}

}  // namespace fa
