// BFloat16 attention forward on the 5th-generation tensor cores (tcgen05, sm_103a),
// persistent, two query tiles per work item.
//
// The grid has one CTA per SM (each holds all of an SM's tensor memory).  A CTA
// runs a list of work items; an item is query tiles 2p and 2p+1 (256 rows) of
// one (batch, head).  Both tiles stream the same key/value tiles, so each K_j,
// V_j is loaded once for two tiles.  Each tile keeps, per query row, the running
// max m, normaliser l and accumulator acc of the online softmax ("The Flash
// Attention" page, online recurrence panel):
//     m_new = max(m, m'),  c = 2^(m - m_new),
//     l <- l c + sum_j 2^(s_j - m_new),   acc <- acc c + sum_j 2^(s_j - m_new) V_j,
//     O = acc / l once at the end, with O = 0 and lse = -inf when l = 0
//     ("Flash attention and efficient attention: Worked examples", Cell D2).
// Scores live in the base-2 domain, s = S * scale * log2(e), so every exponential
// is one ex2.  The N x N score matrix never leaves the SM.
//
// Scheduling (the Question bank's causal block-skipping item: under a causal
// mask the query tiles of a head have unequal work).  The host gives every CTA
// its item list (WorkList in worklist.cuh): longest first within groups of heads
// whose K and V fit in L2 together, each item to the CTA with the least work so
// far.  Items run back to back: the producer loads the next item's Q as soon as the MMA warp
// has issued the last products reading the current one, the K/V ring runs on,
// and the next item's first S products run while the softmax warpgroups write
// the current item's O.
//
// Why two tiles: with one tile the tensor cores idle while that tile's softmax
// runs, because the next product O += P V needs its result.  Here the MMA warp
// issues S0_j, S1_j, then alternates PV0_j, S0_{j+1}, PV1_j, S1_{j+1}, ...: while
// one warpgroup turns S into P, the tensor cores work on the other tile.
//
// Roles (384 threads; warps 10-11 only join the start and the end):
//   warps 0-3   softmax of tile 0: thread r owns row r = tensor-memory lane r
//   warps 4-7   softmax of tile 1
//   warp 8      TMA producer: per item Q0, Q1, then K_j, V_j through a ring of NS slots
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
#include "worklist.cuh"

// Every FA_FWD_EXP2_FMA_EVERY_D<d>-th pair of scores takes its exponentials on
// the FMA pipe (exp2_fma2) instead of the special-function unit; 0 = none.  At
// d = 64 a key tile costs the tensor cores half as much as at d = 128 while the
// exponentials stay the same, so there the special-function unit is the bound
// and part of the work moves to the FMA pipe.
#ifndef FA_FWD_EXP2_FMA_EVERY_D128
#define FA_FWD_EXP2_FMA_EVERY_D128 0
#endif
#ifndef FA_FWD_EXP2_FMA_EVERY_D64
#define FA_FWD_EXP2_FMA_EVERY_D64 0
#endif

namespace fa {

// Pair i of each 16-pair quarter of a row takes the FMA-pipe exponential.
template <int D>
__host__ __device__ constexpr bool exp2_on_fma(int i) {
  constexpr int E = D == 64 ? FA_FWD_EXP2_FMA_EVERY_D64 : FA_FWD_EXP2_FMA_EVERY_D128;
  return E > 0 && (i + 1) % (E > 0 ? E : 1) == 0;
}

// Register shares (launch: 384 threads x 168): warpgroup 2 (producer, MMA issuer,
// two idle warps) keeps FWD_REGS_LOW, the two softmax warpgroups get
// FWD_REGS_HIGH; 128 x 48 + 256 x 224 = 63488 <= 64512.
constexpr uint32_t FWD_REGS_LOW = 48, FWD_REGS_HIGH = 224;
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
// slots in the order K_0, V_0, K_1, V_1, ... (continuing from one item to the
// next); load number c (K_j of an item: c = c_item + 2j, V_j: + 1) uses slot
// c % NS.
template <int D, int NS>
struct TcLayout {
  static constexpr int BM = 128, BN = 128;
  static constexpr int KB = D / 64;           // 64-element (128-byte) column blocks
  static constexpr int COLBLK = 128 * 128;    // bytes of one 128-row column block
  static constexpr int TILE = BM * D * 2;     // bytes of a Q, K or V tile
  static constexpr int OFF_Q = 0;             // Q0, Q1
  static constexpr int OFF_KV = 2 * TILE;     // NS slots
  static constexpr int OFF_EPI = OFF_KV + NS * TILE;  // 2 KB per softmax warp (O epilogue)
  static constexpr int OFF_BAR = OFF_EPI + 8 * 2048;
  // barriers: q_full, q_empty, kv_full[NS], kv_empty[NS], s_full[2], p_full[2], o_done[2], drain,
  //           s_free[2], pv_done[2] (separate-P layout only)
  static constexpr int NBAR = 2 + 2 * NS + 6 + 1 + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 256 + D, TM_COLS = 512;
  // At d = 64, P_i gets columns of its own ([384, 448), [448, 512)) instead of
  // aliasing S_i: S_i(j+1) can then be formed while the softmax still turns
  // S_i(j) into P_i(j).  At d = 128 the accumulators leave no room.
  static constexpr bool SEP_P = D == 64;
  static constexpr uint32_t TM_P0 = SEP_P ? 384 : TM_S0, TM_P1 = SEP_P ? 448 : TM_S1;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BYTES <= 232448, "shared memory budget");
};

// Writes a warp's 32 rows x 32 bf16 -- lane i holds row i as 16 packed pairs --
// to rows row0 + i (i < rows) of `out` (row stride ld elements), columns [col,
// col + 32).  Stored straight from the registers, one instruction would touch 32
// rows 16 bytes each, at half the SM's store rate; through the warp's 2 KB slice
// of shared memory `buf` they come back so that 4 lanes store one row's 64
// contiguous bytes.  The 16-byte chunks of a row are rotated by (row / 2) mod 4,
// so that neither the row-wise writes nor the chunk-wise reads meet a bank twice
// within a 128-byte wavefront.
__device__ __forceinline__ void warp_store_rows_bf16x32(const uint32_t (&w)[16], uint32_t buf, __nv_bfloat16* out,
                                                        size_t row0, size_t ld, int col, int rows) {
  const int lane = threadIdx.x & 31;
  const uint32_t rot = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + lane * 64 + ((c ^ rot) << 4)), "r"(w[4 * c]),
                 "r"(w[4 * c + 1]), "r"(w[4 * c + 2]), "r"(w[4 * c + 3])
                 : "memory");
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 8 * i + (lane >> 2), ch = lane & 3;
    uint4 x;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                 : "r"(buf + row * 64 + ((ch ^ ((row >> 1) & 3)) << 4))
                 : "memory");
    if (row < rows) *reinterpret_cast<uint4*>(out + (row0 + row) * ld + col + 8 * ch) = x;
  }
  __syncwarp();
}

// Shared-memory addresses (32-bit) of the forward kernel's buffers and
// barriers, from the 1024-aligned base of its dynamic shared memory.  Each
// role builds its own copy (from smem_u32_fresh) after changing its register
// budget, so that no address is held across that change.
template <int D, int NS>
struct FwdSmem {
  using L = TcLayout<D, NS>;
  uint32_t base;
  __device__ __forceinline__ explicit FwdSmem(uint32_t raw) : base((raw + 1023u) & ~1023u) {}
  __device__ __forceinline__ uint32_t bar(int i) const { return base + L::OFF_BAR + 8 * i; }
  __device__ __forceinline__ uint32_t q_full() const { return bar(0); }
  // the MMA warp has issued every product reading Q0, Q1 of an item
  __device__ __forceinline__ uint32_t q_empty() const { return bar(1); }
  __device__ __forceinline__ uint32_t kv_full(int s) const { return bar(2 + s); }
  __device__ __forceinline__ uint32_t kv_empty(int s) const { return bar(2 + NS + s); }
  __device__ __forceinline__ uint32_t s_full(int t) const { return bar(2 + 2 * NS + t); }  // one per query tile
  __device__ __forceinline__ uint32_t p_full(int t) const { return bar(4 + 2 * NS + t); }
  __device__ __forceinline__ uint32_t o_done(int t) const { return bar(6 + 2 * NS + t); }
  __device__ __forceinline__ uint32_t drain() const { return bar(8 + 2 * NS); }
  // separate-P layout: the softmax has read S_t (one phase per block)
  __device__ __forceinline__ uint32_t s_free(int t) const { return bar(9 + 2 * NS + t); }
  // separate-P layout: P_t V has run, so P_t and O_t may be written (one phase per block)
  __device__ __forceinline__ uint32_t pv_done(int t) const { return bar(11 + 2 * NS + t); }
};

// One item's geometry, computed alike by every role.
struct FwdItem {
  int bh, q0;        // (batch*head), first query row of tile 0 (tile 1 starts at q0 + 128)
  int kv_limit;      // keys past kv_limit are padding
  int n_t0, n_t1;    // key tiles each query tile needs (0 for a tile entirely past N)
  int n_max;
};

template <int BM, int BN>
__device__ __forceinline__ FwdItem fwd_item(const TcParams& p, const WorkList& sc, int k) {
  int bh, pr;  // units of a head: its query-tile pairs, the last one heaviest under a causal mask
  wl_item(sc, k, (p.n_qt + 1) >> 1, true, bh, pr);
  FwdItem it;
  it.bh = bh;
  it.q0 = pr * 2 * BM;
  it.kv_limit = p.Nk;
  if (p.kv_len) it.kv_limit = min(p.Nk, max(0, p.kv_len[bh / p.H]));
  const int n_kv_all = (it.kv_limit + BN - 1) / BN;
  // key tiles query tile qt needs: under a causal mask, up to the tile holding
  // the last key its last row can see
  auto tiles = [&](int qt) -> int {
    if (qt >= p.n_qt) return 0;
    if (!p.causal) return n_kv_all;
    const int last_key = min(qt * BM + BM, p.N) - 1 + p.qoff - 1;
    return last_key < 0 ? 0 : min(n_kv_all, last_key / BN + 1);
  };
  it.n_t0 = tiles(2 * pr);
  it.n_t1 = tiles(2 * pr + 1);
  it.n_max = max(it.n_t0, it.n_t1);
  return it;
}

template <int D, int NS>
__global__ void __launch_bounds__(384, 1)
    fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const TcParams p,
                        const __grid_constant__ WorkList sc) {
  using L = TcLayout<D, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  // K/V loads and Q loads the producer has issued (for the sm.drain() of an aborted
  // CTA); kept in shared memory so that they hold no register in other roles
  volatile int* issued_kv = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);
  volatile int* issued_q = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    const FwdSmem<D, NS> sm(smem_u32_fresh(smem_raw));
    mbar_init(sm.q_full(), 1);
    mbar_init(sm.q_empty(), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(sm.kv_full(s), 1);
      mbar_init(sm.kv_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.s_full(i), 1);
      mbar_init(sm.p_full(i), 128);
      mbar_init(sm.o_done(i), 1);
      mbar_init(sm.s_free(i), 128);
      mbar_init(sm.pv_done(i), 1);
    }
    mbar_init(sm.drain(), 1);
    *abort_flag = 0;
    *issued_kv = 0;
    *issued_q = 0;
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
  constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;

  if (warp == 8) {
    reg_lower<FWD_REGS_LOW>();
    const FwdSmem<D, NS> sm(smem_u32_fresh(smem_raw));
    const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
    const int n_items = wl_count(sc);
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      int c = 0, nq = 0;  // K/V loads, Q loads issued
      bool go = true;
      for (int k = 0; go && k < n_items; ++k) {
        const FwdItem it = fwd_item<L::BM, L::BN>(p, sc, k);
        if (it.n_max == 0) continue;
        // Q0, Q1 of this item overwrite the previous item's once every product
        // reading them has run
        if (nq > 0 && !mbar_wait(sm.q_empty(), (nq - 1) & 1, wc, ST_TIMEOUT_EMPTY)) break;
        const int ntile = (it.n_t1 > 0) ? 2 : 1;
        mbar_arrive_expect_tx(sm.q_full(), ntile * L::TILE);
        for (int i = 0; i < ntile; ++i)
#pragma unroll
          for (int kb = 0; kb < L::KB; ++kb)
            tma_load_3d(sm.base + L::OFF_Q + i * L::TILE + kb * L::COLBLK, &tm_q, sm.q_full(), kb * 64, it.q0 + i * L::BM,
                        it.bh);
        *issued_q = ++nq;
        for (int cl = 0; cl < 2 * it.n_max; ++cl, ++c) {
          const int slot = c % NS;
          if (c >= NS && !mbar_wait(sm.kv_empty(slot), ((c / NS) - 1) & 1, wc, ST_TIMEOUT_EMPTY)) {
            go = false;
            break;
          }
          if (p.inject == 1 && c == 2) {  // test hook: starve the consumers after K_0, V_0
            go = false;
            break;
          }
          mbar_arrive_expect_tx(sm.kv_full(slot), L::TILE);
          const CUtensorMap* src = (cl & 1) ? &tm_v : &tm_k;
#pragma unroll
          for (int kb = 0; kb < L::KB; ++kb)
            tma_load_3d(sm.base + L::OFF_KV + slot * L::TILE + kb * L::COLBLK, src, sm.kv_full(slot), kb * 64,
                        (cl >> 1) * L::BN, it.bh);
          *issued_kv = c + 1;
        }
      }
    }
    tc_fence_before();
    cta_bar_sync<384>();
    if (lane == 0 && *abort_flag) {
      // an aborted CTA may not exit while copies it issued are still landing
      const int nq = *issued_q, n_iss = *issued_kv;
      bool drained = nq == 0 || mbar_wait_drain(sm.q_full(), (nq - 1) & 1, DRAIN_NS);
      for (int c = max(0, n_iss - NS); c < n_iss; ++c)
        drained &= mbar_wait_drain(sm.kv_full(c % NS), (c / NS) & 1, DRAIN_NS);
      if (!drained) atomicOr(p.status, ST_DRAIN);
    }
  } else if (warp == 9) {
    reg_lower<FWD_REGS_LOW>();
    const FwdSmem<D, NS> sm(smem_u32_fresh(smem_raw));
    const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
    const int n_items = wl_count(sc);
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    // ---------------------------------------------------------- MMA issuer --
    // the whole warp runs the issue code; lane 0 issues (see umma_ss_w)
    constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, true);
    const uint32_t sq = sm.base + L::OFF_Q;
    const uint32_t skv = sm.base + L::OFF_KV;
    // Descriptors of the tile bases; an operand at byte offset `off` from a
    // base is that descriptor plus off >> 4 (the start-address field is the
    // low 14 bits and every shared address here is below 2^18, so no carry).
    const uint64_t dq_base = sdesc_sw128(sq, 16, 1024);
    const uint64_t dk_base = sdesc_sw128(skv, 16, 1024);
    const uint64_t dv_base = sdesc_sw128(skv, L::COLBLK, 1024);
    // S_i = Q_i K^T, K in the slot of load number ck
    auto issue_s = [&](uint32_t tm_s, uint32_t q_off, uint32_t bar, int ck) {
      const uint64_t ka = dk_base + (((ck % NS) * L::TILE) >> 4);
      const uint64_t qa = dq_base + (q_off >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * L::COLBLK + (kk & 3) * 32) >> 4;
        umma_ss_w(tm_s, qa + off, ka + off, IDESC_QK, kk > 0 ? 1u : 0u);
      }
      umma_commit_w(bar);
    };
    // O_i += P_i V, V in the slot of load number cv.  Only a tile's last
    // product of an item signals o_done (for the epilogue): an earlier PV_i(j-1)
    // is known complete once S_i(j), issued after it, has signalled s_full,
    // because a commit tracks every earlier tensor-core operation of this thread.
    auto issue_pv = [&](uint32_t tm_o, uint32_t tm_p, uint32_t bar, int cv, bool first, bool last) {
      const uint64_t va = dv_base + (((cv % NS) * L::TILE) >> 4);
#pragma unroll
      for (int kk = 0; kk < L::BN / 16; ++kk)
        umma_ts_w(tm_o, tm_p + kk * 8, va + (kk * 2048 >> 4), IDESC_PV, (!first || kk > 0) ? 1u : 0u);
      if (last) umma_commit_w(bar);
    };
    const uint32_t tS0 = tmem + L::TM_S0, tS1 = tmem + L::TM_S1;
    const uint32_t tO0 = tmem + L::TM_O0, tO1 = tmem + L::TM_O1;
    const uint32_t tP0 = tmem + L::TM_P0, tP1 = tmem + L::TM_P1;

    int c = 0, nq = 0;    // K/V loads consumed, items started
    int jb0 = 0, jb1 = 0; // blocks of each query tile done in earlier items (s_full / p_full phases)
    bool ok = true;
    for (int k = 0; ok && k < n_items; ++k) {
      const FwdItem it = fwd_item<L::BM, L::BN>(p, sc, k);
      if (it.n_max == 0) continue;
      const int n_t0 = it.n_t0, n_t1 = it.n_t1, n_max = it.n_max;
      ok = mbar_wait_w(sm.q_full(), nq & 1, wc, ST_TIMEOUT_Q) && mbar_wait_w(sm.kv_full(c % NS), (c / NS) & 1, wc, ST_TIMEOUT_K);
      ++nq;
      if (!ok) break;
      tc_fence_after();
      if constexpr (L::SEP_P) {
        // S_i of the item's first block reuses columns the softmax read last
        ok = (n_t0 == 0 || jb0 == 0 || mbar_wait_w(sm.s_free(0), (jb0 - 1) & 1, wc, ST_TIMEOUT_S)) &&
             (n_t1 == 0 || jb1 == 0 || mbar_wait_w(sm.s_free(1), (jb1 - 1) & 1, wc, ST_TIMEOUT_S));
        if (!ok) break;
        tc_fence_after();
      }
      if (n_t0 > 0) issue_s(tS0, 0, sm.s_full(0), c);
      if (n_t1 > 0) issue_s(tS1, L::TILE, sm.s_full(1), c);
      umma_commit_w(sm.kv_empty(c % NS));
      if (n_max == 1) umma_commit_w(sm.q_empty());  // every product reading Q0, Q1 issued
      for (int j = 0; ok && j < n_max; ++j) {
        const int cv = c + 2 * j + 1, ck = c + 2 * j + 2;  // load numbers of V_j and K_{j+1}
        const int j1 = j + 1;
        // every tile that reads K_{j+1} or V_j waits for it once, before its first use
        bool k1_ready = false, v_ready = false;
        auto wait_v = [&]() -> bool {
          if (v_ready) return true;
          v_ready = mbar_wait_w(sm.kv_full(cv % NS), (cv / NS) & 1, wc, ST_TIMEOUT_V);
          return v_ready;
        };
        auto wait_k1 = [&]() -> bool {
          if (k1_ready) return true;
          k1_ready = mbar_wait_w(sm.kv_full(ck % NS), (ck / NS) & 1, wc, ST_TIMEOUT_K);
          if (k1_ready) tc_fence_after();
          return k1_ready;
        };
        if constexpr (L::SEP_P) {
          // S0_{j+1} and S1_{j+1} as soon as the softmax has read S0_j, S1_j; then
          // PV0_j and PV1_j (P in columns of its own), each committing pv_done
          if (j1 < n_t0) {
            if (!mbar_wait_w(sm.s_free(0), (jb0 + j) & 1, wc, ST_TIMEOUT_S) || !wait_k1()) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(tS0, 0, sm.s_full(0), ck);
          }
          if (j1 < n_t1) {
            if (!mbar_wait_w(sm.s_free(1), (jb1 + j) & 1, wc, ST_TIMEOUT_S) || !wait_k1()) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(tS1, L::TILE, sm.s_full(1), ck);
          }
          if (j < n_t0) {
            if (!wait_v() || !mbar_wait_w(sm.p_full(0), (jb0 + j) & 1, wc, ST_TIMEOUT_P)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(tO0, tP0, sm.o_done(0), cv, j == 0, j + 1 == n_t0);
            umma_commit_w(sm.pv_done(0));
          }
          if (j < n_t1) {
            if (!wait_v() || !mbar_wait_w(sm.p_full(1), (jb1 + j) & 1, wc, ST_TIMEOUT_P)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(tO1, tP1, sm.o_done(1), cv, j == 0, j + 1 == n_t1);
            umma_commit_w(sm.pv_done(1));
          }
          umma_commit_w(sm.kv_empty(cv % NS));
          if (j1 < n_max) umma_commit_w(sm.kv_empty(ck % NS));
          if (j1 == n_max - 1) umma_commit_w(sm.q_empty());
          continue;
        }
        // tile 0: PV0_j, then S0_{j+1}
        if (j < n_t0) {
          if (!wait_v() || !mbar_wait_w(sm.p_full(0), (jb0 + j) & 1, wc, ST_TIMEOUT_P)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(tO0, tS0, sm.o_done(0), cv, j == 0, j + 1 == n_t0);
        }
        if (j1 < n_t0) {
          if (!wait_k1()) {
            ok = false;
            break;
          }
          issue_s(tS0, 0, sm.s_full(0), ck);
        }
        // tile 1: PV1_j, then S1_{j+1}
        if (j < n_t1) {
          if (!wait_v() || !mbar_wait_w(sm.p_full(1), (jb1 + j) & 1, wc, ST_TIMEOUT_P)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(tO1, tS1, sm.o_done(1), cv, j == 0, j + 1 == n_t1);
        }
        if (j1 < n_t1) {
          if (!wait_k1()) {
            ok = false;
            break;
          }
          issue_s(tS1, L::TILE, sm.s_full(1), ck);
        }
        umma_commit_w(sm.kv_empty(cv % NS));                 // V_j: read by every PV above
        if (j1 < n_max) umma_commit_w(sm.kv_empty(ck % NS));  // K_{j+1}: read by every S above
        if (j1 == n_max - 1) umma_commit_w(sm.q_empty());        // the item's last S products are issued
      }
      c += 2 * n_max;
      jb0 += n_t0;
      jb1 += n_t1;
    }
    // nothing may be in flight on the tensor cores when the CTA frees TMEM
    umma_commit_w(sm.drain());
    if (!mbar_wait_drain(sm.drain(), 0, DRAIN_NS) && lane == 0) atomicOr(p.status, ST_DRAIN);
    tc_fence_before();
    cta_bar_sync<384>();
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  } else if (warp < 8) {
    reg_raise<FWD_REGS_HIGH>();
    const FwdSmem<D, NS> sm(smem_u32_fresh(smem_raw));
    const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
    const int n_items = wl_count(sc);
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    // ------------------------------------------------------------- softmax --
    const int ti = warp >> 2;          // query tile 0 or 1 (warps 10-11 have no role)
    const int r = threadIdx.x & 127;   // row in the tile == tensor-memory lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + (ti ? L::TM_S1 : L::TM_S0);
    const uint32_t p_col = lane_base + (ti ? L::TM_P1 : L::TM_P0);  // = s_col unless SEP_P
    const uint32_t o_col = lane_base + (ti ? L::TM_O1 : L::TM_O0);
    const float sl = p.scale_log2;
    int jb = 0, no = 0;  // blocks of this tile done in earlier items; items that signalled o_done
    bool ok = true;
    for (int k = 0; ok && k < n_items; ++k) {
      const FwdItem it = fwd_item<L::BM, L::BN>(p, sc, k);
      const int bh = it.bh, kv_limit = it.kv_limit;
      // key k is visible to this row iff k < qlim (causal modes)
      const int qlim = it.q0 + ti * L::BM + r + p.qoff;
      const int n_kv = ti ? it.n_t1 : it.n_t0;
      const int qt0c = it.q0 + ti * L::BM + p.qoff;  // qlim of the tile's first row
      // l: the row sum of the probabilities as computed (float32), for lse;
      // dl: how much the bf16 values the P V product uses differ from them, for
      // the largest probability of each block (see below)
      float m = -INFINITY, l = 0.f, dl = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        // tcgen05.ld/st are warp-collective: the whole warp goes on or stops together
        if (!__all_sync(0xffffffffu, mbar_wait(sm.s_full(ti), (jb + j) & 1, wc, ST_TIMEOUT_S))) {
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
        if constexpr (L::SEP_P) {
          tc_fence_before();
          mbar_arrive(sm.s_free(ti));  // S_(j+1) may overwrite the scores now
        }

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
        if constexpr (L::SEP_P) {
          // P_j and the accumulator's rescale wait for P V of the previous block
          // (with S_j formed ahead of it, s_full no longer implies it has run)
          if (jb + j > 0 && !__all_sync(0xffffffffu, mbar_wait(sm.pv_done(ti), (jb + j - 1) & 1, wc, ST_TIMEOUT_P))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
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
            if (exp2_on_fma<D>(i)) {
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
          FA_TMEM_ST16(p_col + 16 * h, pk);
        }
        float ra, rb, rc, rd;
        f2_unpack(rs2[0], ra, rb);
        f2_unpack(rs2[1], rc, rd);
        l = l * c + ((ra + rb) + (rc + rd));
        if (j > 0 && __any_sync(0xffffffffu, m_new != m)) {
          // The accumulator already holds blocks < j: PV_{j-1} was issued before
          // S_j, and s_full for S_j tracks every earlier tensor-core operation
          // (separate-P layout: the pv_done wait above).
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
        mbar_arrive(sm.p_full(ti));
        m = m_new;
      }
      jb += n_kv;
      if (ok && n_kv > 0 && !__all_sync(0xffffffffu, mbar_wait(sm.o_done(ti), no & 1, wc, ST_TIMEOUT_O))) ok = false;
      if (n_kv > 0) ++no;
      const int qrow = qlim - p.qoff;
      if (ok && qt0c - p.qoff < p.N) {
        tc_fence_after();
        const float inv = (l > 0.f) ? 1.f / (l + dl) : 0.f;  // guard: l = 0 -> zero vector
        const int qr0 = qt0c - p.qoff + (warp & 3) * 32;  // this warp's first row
        const int rows = min(32, p.N - qr0);
        const uint32_t buf = sm.base + L::OFF_EPI + warp * 2048;
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
          warp_store_rows_bf16x32(ob, buf, p.o, static_cast<size_t>(bh) * p.N + qr0, D, cb * 32, rows);
        }
        if (p.lse && qrow < p.N)
          p.lse[static_cast<size_t>(bh) * p.N + qrow] = (l > 0.f) ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
        // the next item's first P V overwrites this tile's accumulator only after
        // this warpgroup's p_full for it, i.e. after these loads
        tc_fence_before();
      }
    }
    tc_fence_before();
    cta_bar_sync<384>();
  } else {
    reg_lower<FWD_REGS_LOW>();  // warps 10-11: no role
    cta_bar_sync<384>();
  }
}

}  // namespace fa
