// BFloat16 attention backward on the 5th-generation tensor cores (tcgen05, sm_103a):
// the row preprocess and the per-key-tile kernel for dK and dV.  dQ comes from
// bwd_dq_kernel (bwd_dq.cuh).
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
// Why dQ has a kernel of its own.  dQ sums over key tiles, dK and dV over query
// tiles; one CTA can accumulate only one side in tensor memory.  Adding the other
// side's partial tiles into device memory (a tiled reduce-add per 128 x 128 tile)
// runs on the SM's path for reductions, which measured about 24 bytes per cycle
// per SM on B300 whatever issues them: 64 KB of dQ per tile needs at least 2700
// cycles, more than the tile's products.  So the per-key-tile kernel here makes
// no dQ, and bwd_dq_kernel, per query tile, recomputes S and dP and accumulates
// dQ in tensor memory: seven products per tile instead of five, no reductions,
// and a deterministic dQ.
//
// Kernels:
//  * bwd_preprocess_kernel -- nl_i = -lse_i log2(e) and nd_i = -D_i scale into
//    the workspace (row stride Np = N rounded up to 128; padding rows get nl =
//    -inf, so that their probabilities are exactly 0, and nd = 0).  With them
//    P = 2^(S scale log2e + nl) and dS = P (dP scale + nd) take one packed FMA
//    (and one packed multiply) per pair of entries.
//  * bwd_dkdv_kernel -- persistent; an item is (batch*head, 128-key tile).  K and
//    V stay in shared memory; the CTA streams 128-query tiles (Q_t with its nl_t
//    and nd_t rows, and dO_t) through a 2-stage TMA ring and, per tile t, runs
//    four MMAs (128 x 128 x 128 each):
//       MMA1  S^T_t  = K Q_t^T            (A = K, B = Q_t, both from SMEM)
//       MMA2  dP^T_t = V dO_t^T           (A = V, B = dO_t)
//       MMA3  dV    += P^T_t dO_t          (A = P^T from TMEM, B = dO_t MN-major)
//       MMA4  dK    += dS^T_t Q_t          (A = dS^T from SMEM, B = Q_t MN-major)
//    issued as MMA3_t, MMA1_{t+1}, MMA4_t, MMA2_{t+1}: each product overwrites a
//    tensor-memory region only after the product reading it was issued, and the
//    tensor cores run in issue order.  While the elementwise warps form dS^T_t,
//    the tensor cores run MMA3_t and MMA1_{t+1}; while they form P^T_{t+1},
//    MMA4_t and MMA2_{t+1}.  dS carries the factor `scale`, so dK needs no
//    further scaling.
//
// Roles (384 threads):
//   warp 0     TMA producer: per item K, V; then Q_t + nl_t + nd_t and dO_t into
//              the ring (separate full / empty barriers for Q and dO).
//   warp 1     MMA issuer (lane 0 of the converged warp) and tensor-memory owner.
//   warps 2-3  no role.
//   warps 4-7  elementwise warpgroup 0, query columns 0-63 of every tile;
//   warps 8-11 elementwise warpgroup 1, query columns 64-127.
//              Thread r owns key row r (TMEM lane r) of S^T and dP^T:
//                P^T = 2^(S^T scale log2e + nl) with the causal / padding mask,
//                written back to TMEM as bf16 (aliasing S^T); then
//                dS^T = P^T (dP^T scale + nd) -> bf16, into shared memory.
//              At the end of an item warpgroup 0 writes dV and warpgroup 1 dK.
//
// dS^T goes through shared memory rather than tensor memory: measured on B300,
// the elementwise warps' tcgen05.st of dS^T slowed the product running beside
// it (MMA3, whose A operand it reads from tensor memory) more than the shared-
// memory stores and the extra shared-memory operand of MMA4 cost (3.6 % of the
// backward).  The same move for P^T gained nothing, and for the dQ kernel's dS
// it lost 6 %: that kernel's products already read close to the shared
// memory's bandwidth.
//
// Tensor memory (512 columns, f32 unless noted):
//   [0,128)   S^T_t, then P^T_t (bf16: queries 0-63 in [0,32), 64-127 in [64,96))
//   [128,256) dP^T_t
//   [256,384) dV   [384,512) dK
//
// Every wait is bounded, as in the forward kernel: a wait that runs out records
// a status bit, the CTA drains what it has in flight and exits.
#pragma once
#include "exp2_poly.cuh"
#include "ptx.cuh"
#include "worklist.cuh"

// Every FA_BWD_EXP2_FMA_EVERY-th pair of probabilities takes its exponentials on
// the FMA pipe (exp2_fma2) instead of the special-function unit; 0 = none.
#ifndef FA_BWD_EXP2_FMA_EVERY
#define FA_BWD_EXP2_FMA_EVERY 0
#endif

namespace fa {

enum : unsigned {
  ST_BWD_TIMEOUT_KV = 1u << 8,
  ST_BWD_TIMEOUT_Q = 1u << 9,
  ST_BWD_TIMEOUT_S = 1u << 10,
  ST_BWD_TIMEOUT_P = 1u << 11,
  ST_BWD_TIMEOUT_DP = 1u << 12,
  ST_BWD_TIMEOUT_DS = 1u << 13,
  ST_BWD_TIMEOUT_DQ = 1u << 14,
  ST_BWD_TIMEOUT_EMPTY = 1u << 16,
  ST_BWD_TIMEOUT_DONE = 1u << 17,
  ST_BWD_SMEM_ALIGN = 1u << 19,   // dynamic shared memory base not aligned enough (kernel did nothing)
};

// Register shares (launch: 384 threads x 168): warps 0-3 (producer, MMA issuer,
// idle) keep BWD_REGS_LOW, the elementwise warpgroups get BWD_REGS_HIGH.
constexpr uint32_t BWD_REGS_LOW = 56, BWD_REGS_HIGH = 216;
static_assert(128 * BWD_REGS_LOW + 256 * BWD_REGS_HIGH <= 384 * 168, "register split exceeds the launch");

struct BwdPreParams {
  const __nv_bfloat16* o;   // [BH, N, D]
  const __nv_bfloat16* dO;  // [BH, N, D]
  const float* lse;         // [BH, N]
  float* nl;                // workspace [BH, Np]: -lse log2(e)
  float* nd;                // workspace [BH, Np]: -D scale
  int BH, N, Np;
  float scale;
};

// D = sum_c dO_c O_c (f32) per row; nl = -lse log2(e) (-inf where lse = -inf
// or the row is padding); nd = -D scale.  Half a warp per row (16 lanes x 8
// elements, 16-byte loads); a warp takes 8 rows and issues all of its loads
// before the first reduction.  Grid: BH * Np / 64 blocks of 256 threads.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdPreParams p) {
  static_assert(D == 128, "16 lanes x 8 elements per row");
  const int chunks = p.Np / 64;
  const int bh = static_cast<int>(blockIdx.x) / chunks;
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const int row0 = (static_cast<int>(blockIdx.x) % chunks) * 64 + (threadIdx.x >> 5) * 8 + half;
  uint4 a[4], g[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int row = row0 + 2 * s;
    if (row < p.N) {
      const size_t base = (static_cast<size_t>(bh) * p.N + row) * D + hl * 8;
      a[s] = *reinterpret_cast<const uint4*>(p.o + base);
      g[s] = *reinterpret_cast<const uint4*>(p.dO + base);
    } else {
      a[s] = make_uint4(0u, 0u, 0u, 0u);
      g[s] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[s]);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g[s]);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 af = __bfloat1622float2(a2[i]), gf = __bfloat1622float2(g2[i]);
      acc = fmaf(af.x, gf.x, acc);
      acc = fmaf(af.y, gf.y, acc);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);  // within the half
    const int row = row0 + 2 * s;
    if (hl == 0) {
      const size_t ws = static_cast<size_t>(bh) * p.Np + row;
      if (row < p.N) {
        const float l = p.lse[static_cast<size_t>(bh) * p.N + row];
        p.nl[ws] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
        p.nd[ws] = -acc * p.scale;
      } else {
        p.nl[ws] = -INFINITY;
        p.nd[ws] = 0.f;
      }
    }
  }
}

struct BwdParams {
  float* dq;                // [BH, N, D], written once per row by bwd_dq_kernel
  float* dk;                // [BH, Nk, D]
  float* dv;                // [BH, Nk, D]
  const float* nl;          // [BH, Np]: -lse log2(e)
  const float* nd;          // [BH, Np]: -D scale
  const __nv_bfloat16* q;   // [BH, N, D]: the dQ kernel copies its rows into tensor memory
  const int* kv_len;        // [B] or null
  int BH, H, N, Np;         // N queries per head
  int Nk;                   // keys per head
  int n_qt, n_kt;           // query tiles, key tiles per head
  float scale;              // score multiplier
  float scale_log2;         // scale * log2(e)
  int causal;               // 0 none, else key k visible to query row i iff k < i + qoff
  int qoff;                 // (Nk - N) + 1 (causal 1) or (Nk - N) (causal 2, strict)
  unsigned* status;
  unsigned long long timeout_ns;
  int inject;               // test hook: 2 = the dK/dV producer stops after the first Q / dO tile
};

template <int STAGES>
struct BwdLayout {
  static constexpr int D = 128;
  static constexpr int BN = 128;                   // keys per item
  static constexpr int BM = 128;                   // queries per tile
  static constexpr int KB = D / 64;                // 128-byte column blocks
  static constexpr int COLBLK = 128 * 128;         // 16 KB: 128 rows x 128 bytes
  static constexpr int TILE = 128 * D * 2;         // 32 KB: a K, V, Q or dO tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * TILE;
  static constexpr int OFF_DS = OFF_DO + STAGES * TILE;    // dS^T_t, K-major (MMA4's A); epilogue staging
  static constexpr int OFF_STAT = OFF_DS + TILE;            // per stage: nl[128], nd[128]
  static constexpr int OFF_BAR = OFF_STAT + STAGES * 1024;
  // barriers: kv_full, kv_free, q_full[S], do_full[S], q_empty[S], do_empty[S], s_full, p_full,
  //           dp_full, ds_full, dkv_done, drain
  static constexpr int NBAR = 2 + 4 * STAGES + 6;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // the dynamic shared memory starts 1024-byte aligned (checked at launch): no slack
  static constexpr int BYTES = OFF_MISC + 32;
  // S^T, then P^T (bf16, in each half's own columns) | dP^T | dV | dK
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 384, TM_COLS = 512;
  static_assert(BYTES <= 232448, "shared memory budget");
};

// Shared-memory addresses (32-bit) of the dK/dV kernel's buffers and barriers,
// from the 1024-aligned base of its dynamic shared memory.  Each role builds its
// own copy (from smem_u32_fresh) after changing its register budget, so that no
// address is held across that change.
template <int STAGES>
struct BwdSmem {
  using L = BwdLayout<STAGES>;
  uint32_t base;
  __device__ __forceinline__ explicit BwdSmem(uint32_t raw) : base((raw + 1023u) & ~1023u) {}
  __device__ __forceinline__ uint32_t bar(int i) const { return base + L::OFF_BAR + 8 * i; }
  __device__ __forceinline__ uint32_t kv_full() const { return bar(0); }
  // every product of an item that reads K or V has been issued (one phase per item)
  __device__ __forceinline__ uint32_t kv_free() const { return bar(1); }
  __device__ __forceinline__ uint32_t q_full(int s) const { return bar(2 + s); }  // Q_t, nl_t, nd_t landed
  __device__ __forceinline__ uint32_t do_full(int s) const { return bar(2 + STAGES + s); }
  __device__ __forceinline__ uint32_t q_empty(int s) const { return bar(2 + 2 * STAGES + s); }  // MMA4_t done
  __device__ __forceinline__ uint32_t do_empty(int s) const { return bar(2 + 3 * STAGES + s); }  // MMA3_t done
  __device__ __forceinline__ uint32_t s_full() const { return bar(2 + 4 * STAGES); }
  __device__ __forceinline__ uint32_t p_full() const { return bar(3 + 4 * STAGES); }
  __device__ __forceinline__ uint32_t dp_full() const { return bar(4 + 4 * STAGES); }
  __device__ __forceinline__ uint32_t ds_full() const { return bar(5 + 4 * STAGES); }
  __device__ __forceinline__ uint32_t dkv_done() const { return bar(6 + 4 * STAGES); }
  __device__ __forceinline__ uint32_t drain() const { return bar(7 + 4 * STAGES); }
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later reads of
// them by the tensor cores (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// A group of 8 MMAs (K = 128): A K-major in shared memory (two 16 KB column
// blocks, 32 bytes per step), B MN-major (16 rows = 2 KB per step).
__device__ __forceinline__ void umma_ss_kmn8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_UMMA_HEAD FA_UMMA_SS_FIRST FA_UMMA_SS(2, 128) FA_UMMA_SS(4, 256) FA_UMMA_SS(6, 384)
                   FA_UMMA_SS(1024, 512) FA_UMMA_SS(1026, 640) FA_UMMA_SS(1028, 768) FA_UMMA_SS(1030, 896) "}" ::"r"(d),
               "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
               : "memory");
}

// Writes a warp's 32 x 32 block of f32 -- lane i holds row i, v its 32 columns --
// to rows row0 + i (i < rows) of `out` (row stride ld floats), columns [col,
// col + 32).  Stored straight from the registers, one instruction would touch 32
// rows 16 bytes each; instead each half-row of 16 columns goes through the warp's
// 2 KB slice of shared memory `buf` and comes back so that 4 lanes store one row's
// 64 contiguous bytes (8 rows per instruction).  The 16-byte chunks of a row are
// rotated by (row / 2) mod 4, so that neither the row-wise writes nor the
// chunk-wise reads meet a bank twice within a 128-byte wavefront.
__device__ __forceinline__ void warp_store_rows_f32x32(const uint32_t (&v)[32], uint32_t buf, float* out,
                                                       size_t row0, size_t ld, int col, int rows) {
  const int lane = threadIdx.x & 31;
  const uint32_t wrow = buf + lane * 64;
  const uint32_t rot = (lane >> 1) & 3;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      st_shared_v4(wrow + ((c ^ rot) << 4), v[16 * hh + 4 * c], v[16 * hh + 4 * c + 1], v[16 * hh + 4 * c + 2],
                   v[16 * hh + 4 * c + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = 8 * i + (lane >> 2), ch = lane & 3;
      float x[4];
      ld_shared_v4f(buf + row * 64 + ((ch ^ ((row >> 1) & 3)) << 4), x);
      if (row < rows)
        *reinterpret_cast<float4*>(out + (row0 + row) * ld + col + 16 * hh + 4 * ch) = make_float4(x[0], x[1], x[2], x[3]);
    }
    __syncwarp();
  }
}

// One dK/dV work item: a 128-key tile of one (batch, head), and the range of
// query tiles that see it (under a causal mask, from the tile holding the key
// tile's first visible query on).  Each role computes it alike.
struct BwdItem {
  int bh, k0, kv_limit, i0, n_it;
};
template <int BN, int BM, typename Params>
__device__ __forceinline__ BwdItem bwd_item(const Params& p, const WorkList& w, int k) {
  int bh, kt;  // units of a head: its key tiles, the first one heaviest under a causal mask
  wl_item(w, k, p.n_kt, false, bh, kt);
  BwdItem g;
  g.bh = bh;
  g.k0 = kt * BN;
  g.kv_limit = p.Nk;
  if (p.kv_len) g.kv_limit = min(p.Nk, max(0, p.kv_len[bh / p.H]));
  // causal: key k0 is visible to query rows i >= k0 - qoff + 1
  g.i0 = p.causal ? max(0, g.k0 - p.qoff + 1) / BM : 0;
  g.n_it = (g.k0 < g.kv_limit && g.i0 < p.n_qt) ? p.n_qt - g.i0 : 0;
  return g;
}

template <int STAGES>
__global__ void __launch_bounds__(384, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p, const __grid_constant__ WorkList sc) {
  using L = BwdLayout<STAGES>;
  constexpr int D = L::D;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the layout fills the shared memory: it needs a 1024-byte aligned base
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, ST_BWD_SMEM_ALIGN);
    return;
  }
  uint8_t* smem = smem_raw;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* issued_q = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);
  volatile int* issued_do = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 12);
  volatile int* issued_kv = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 16);  // K/V loads issued
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the dQ kernel that follows reads nothing this kernel writes: its CTAs may
  // take each SM as soon as this kernel's CTA there has finished
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (threadIdx.x == 0) {
    const BwdSmem<STAGES> sm(smem_u32_fresh(smem_raw));
    mbar_init(sm.kv_full(), 1);
    mbar_init(sm.kv_free(), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(sm.q_full(s), 1);
      mbar_init(sm.do_full(s), 1);
      mbar_init(sm.q_empty(s), 1);
      mbar_init(sm.do_empty(s), 1);
    }
    mbar_init(sm.s_full(), 1);
    mbar_init(sm.p_full(), 256);
    mbar_init(sm.dp_full(), 1);
    mbar_init(sm.ds_full(), 256);
    mbar_init(sm.dkv_done(), 1);
    mbar_init(sm.drain(), 1);
    *abort_flag = 0;
    *issued_q = 0;
    *issued_do = 0;
    *issued_kv = 0;
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
  constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;

  if (warp == 0) {
    reg_lower<BWD_REGS_LOW>();
    const BwdSmem<STAGES> sm(smem_u32_fresh(smem_raw));
    const uint32_t sbase = sm.base;
    const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
    const int n_items = wl_count(sc);
    // ------------------------------------------------------------ producer --
    // Per item: K and V (once the previous item's last products reading them
    // have been issued and run), then Q_t + nl_t + nd_t and dO_t of every query
    // tile through the ring.  T counts query tiles over all of the CTA's items
    // (ring slot and barrier phases).
    if (lane == 0) {
      int T = 0, ni = 0;
      bool go = true;
      for (int k = 0; go && k < n_items; ++k) {
        const BwdItem g = bwd_item<L::BN, L::BM>(p, sc, k);
        if (g.n_it == 0) continue;
        if (ni > 0 && !mbar_wait(sm.kv_free(), (ni - 1) & 1, wc, ST_BWD_TIMEOUT_EMPTY)) break;
        mbar_arrive_expect_tx(sm.kv_full(), 2 * L::TILE);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
          tma_load_3d(sbase + L::OFF_K + kb * L::COLBLK, &tm_k, sm.kv_full(), kb * 64, g.k0, g.bh);
          tma_load_3d(sbase + L::OFF_V + kb * L::COLBLK, &tm_v, sm.kv_full(), kb * 64, g.k0, g.bh);
        }
        *issued_kv = ++ni;
        for (int t = 0; t < g.n_it; ++t, ++T) {
          const int st = T % STAGES;
          const uint32_t eph = ((T / STAGES) - 1) & 1;
          const int q0 = (g.i0 + t) * L::BM;
          if (p.inject == 2 && T == 1) {  // test hook: starve the consumers after the first tile
            go = false;
            break;
          }
          if (T >= STAGES && !mbar_wait(sm.q_empty(st), eph, wc, ST_BWD_TIMEOUT_EMPTY)) {
            go = false;
            break;
          }
          mbar_arrive_expect_tx(sm.q_full(st), L::TILE + 1024);
#pragma unroll
          for (int kb = 0; kb < L::KB; ++kb)
            tma_load_3d(sbase + L::OFF_Q + st * L::TILE + kb * L::COLBLK, &tm_q, sm.q_full(st), kb * 64, q0, g.bh);
          // nl and nd of the tile's 128 queries (rows padded to a multiple of 128)
          const size_t ws = static_cast<size_t>(g.bh) * p.Np + q0;
          bulk_load(sbase + L::OFF_STAT + st * 1024, p.nl + ws, 512, sm.q_full(st));
          bulk_load(sbase + L::OFF_STAT + st * 1024 + 512, p.nd + ws, 512, sm.q_full(st));
          *issued_q = T + 1;
          if (T >= STAGES && !mbar_wait(sm.do_empty(st), eph, wc, ST_BWD_TIMEOUT_EMPTY)) {
            go = false;
            break;
          }
          mbar_arrive_expect_tx(sm.do_full(st), L::TILE);
#pragma unroll
          for (int kb = 0; kb < L::KB; ++kb)
            tma_load_3d(sbase + L::OFF_DO + st * L::TILE + kb * L::COLBLK, &tm_do, sm.do_full(st), kb * 64, q0, g.bh);
          *issued_do = T + 1;
        }
      }
    }
    tc_fence_before();
    cta_bar_sync<384>();
    if (lane == 0 && *abort_flag) {
      // an aborted CTA may not exit while copies it issued are still landing
      const int nk = *issued_kv, nq = *issued_q, nd = *issued_do;
      bool drained = nk == 0 || mbar_wait_drain(sm.kv_full(), (nk - 1) & 1, DRAIN_NS);
      for (int t = max(0, nq - STAGES); t < nq; ++t)
        drained &= mbar_wait_drain(sm.q_full(t % STAGES), (t / STAGES) & 1, DRAIN_NS);
      for (int t = max(0, nd - STAGES); t < nd; ++t)
        drained &= mbar_wait_drain(sm.do_full(t % STAGES), (t / STAGES) & 1, DRAIN_NS);
      if (!drained) atomicOr(p.status, ST_DRAIN);
    }
  } else if (warp == 1) {
    reg_lower<BWD_REGS_LOW>();
    const BwdSmem<STAGES> sm(smem_u32_fresh(smem_raw));
    const uint32_t sbase = sm.base;
    const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
    const int n_items = wl_count(sc);
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    // ---------------------------------------------------------- MMA issuer --
    // the whole warp runs the issue code; lane 0 issues (see umma_ss_w)
    constexpr uint32_t IDESC_S = idesc_bf16_f32(128, L::BM, false, false);  // K Q^T, V dO^T
    constexpr uint32_t IDESC_G = idesc_bf16_f32(128, D, true, false);       // P^T dO, dS^T Q
    // Descriptors of the operand bases; an operand at byte offset `off` from a
    // base is that descriptor plus off >> 4 (the start-address field is the
    // low 14 bits and every shared address here is below 2^18, so no carry).
    const uint64_t d_k = sdesc_sw128(sbase + L::OFF_K, 16, 1024);  // K-major: K, V, Q, dO
    const uint64_t d_v = sdesc_sw128(sbase + L::OFF_V, 16, 1024);
    const uint64_t d_q = sdesc_sw128(sbase + L::OFF_Q, 16, 1024);
    const uint64_t d_do = sdesc_sw128(sbase + L::OFF_DO, 16, 1024);
    const uint64_t m_q = sdesc_sw128(sbase + L::OFF_Q, L::COLBLK, 1024);  // MN-major: Q, dO
    const uint64_t m_do = sdesc_sw128(sbase + L::OFF_DO, L::COLBLK, 1024);
    const uint64_t d_ds = sdesc_sw128(sbase + L::OFF_DS, 16, 1024);  // K-major: dS^T
    constexpr uint32_t TILE16 = L::TILE >> 4;

    // S^T = K Q_t^T or dP^T = V dO_t^T: both operands K-major, two column blocks each
    static_assert(D == 128 && L::COLBLK == 16384 && L::BM == 128, "group issue shapes");
    auto mma_scores = [&](uint32_t d_tm, uint64_t a, uint64_t b) { umma_ss_k8(d_tm, a, b, IDESC_S, 0u); };
    // dV += P^T dO_t (A = P^T) or dK += dS^T Q_t (A = dS^T): A from tensor memory,
    // bf16 pairs with queries 0-63 in columns [0, 32) and 64-127 in [64, 96) of
    // its region (each warpgroup's half in its own columns); B MN-major, 16
    // queries = 2 KB per step.  The accumulator starts over at an item's first tile.
    auto mma_grad = [&](uint32_t d_tm, uint32_t a_tm, uint64_t b, bool first) {
      umma_ts_h_mn8(d_tm, a_tm, b, IDESC_G, first ? 0u : 1u);
    };
    // Per item: MMA1_0, MMA2_0, then per tile t
    //   MMA3_t, MMA1_{t+1}, MMA4_t, MMA2_{t+1}.
    // T0 is the CTA-wide index of the item's first query tile.
    int T0 = 0, ni = 0;
    bool ok = true;
    for (int k = 0; ok && k < n_items; ++k) {
      const int n_it = bwd_item<L::BN, L::BM>(p, sc, k).n_it;
      if (n_it == 0) continue;
      const int s0 = T0 % STAGES;
      const uint32_t ph0 = (T0 / STAGES) & 1;
      // S columns: the previous item's last P^T was read by its MMA3, issued
      // before; dP columns: its last dS^T by its MMA4, issued before
      ok = mbar_wait_w(sm.kv_full(), ni & 1, wc, ST_BWD_TIMEOUT_KV) &&
           mbar_wait_w(sm.q_full(s0), ph0, wc, ST_BWD_TIMEOUT_Q);
      if (!ok) break;
      tc_fence_after();
      mma_scores(tmem + L::TM_S, d_k, d_q + s0 * TILE16);
      umma_commit_w(sm.s_full());
      if (!mbar_wait_w(sm.do_full(s0), ph0, wc, ST_BWD_TIMEOUT_Q)) {
        ok = false;
        break;
      }
      tc_fence_after();
      mma_scores(tmem + L::TM_DP, d_v, d_do + s0 * TILE16);
      umma_commit_w(sm.dp_full());
      if (n_it == 1) umma_commit_w(sm.kv_free());  // no later product reads K or V
      for (int t = 0; t < n_it; ++t) {
        const int T = T0 + t;
        const int st = T % STAGES, st1 = (T + 1) % STAGES;
        const uint32_t ph = T & 1, ph1 = ((T + 1) / STAGES) & 1;
        const bool next = t + 1 < n_it;
        // MMA3: dV += P^T_t dO_t (dV starts over at t = 0: the warpgroups arrive
        // on p_full for an item only after writing out the previous item's dV and
        // dK).  Its commit also covers MMA2_t, the other reader of dO_t.
        if (!mbar_wait_w(sm.p_full(), ph, wc, ST_BWD_TIMEOUT_P)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_grad(tmem + L::TM_DV, tmem + L::TM_S, m_do + st * TILE16, t == 0);
        umma_commit_w(sm.do_empty(st));
        // MMA1: S^T_{t+1} into the S columns (P^T_t was read by MMA3_t, issued
        // before: the tensor cores run in issue order)
        if (next) {
          if (!mbar_wait_w(sm.q_full(st1), ph1, wc, ST_BWD_TIMEOUT_Q)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_scores(tmem + L::TM_S, d_k, d_q + st1 * TILE16);
          umma_commit_w(sm.s_full());
        }
        // MMA4: dK += dS^T_t Q_t; its commit frees Q_t's stage (MMA1_t read it before)
        if (!mbar_wait_w(sm.ds_full(), ph, wc, ST_BWD_TIMEOUT_DS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        umma_ss_kmn8(tmem + L::TM_DK, d_ds, m_q + st * TILE16, IDESC_G, t == 0 ? 0u : 1u);
        umma_commit_w(sm.q_empty(st));
        // MMA2: dP^T_{t+1} into the dP columns (dS^T_t was read by MMA4_t)
        if (next) {
          if (!mbar_wait_w(sm.do_full(st1), ph1, wc, ST_BWD_TIMEOUT_Q)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_scores(tmem + L::TM_DP, d_v, d_do + st1 * TILE16);
          umma_commit_w(sm.dp_full());
          if (t + 2 == n_it) umma_commit_w(sm.kv_free());  // the item's last reader of K and V
        }
      }
      if (!ok) break;
      umma_commit_w(sm.dkv_done());  // dV, dK of the item are complete
      T0 += n_it;
      ++ni;
    }
    // nothing may be in flight on the tensor cores when the CTA frees TMEM
    umma_commit_w(sm.drain());
    if (!mbar_wait_drain(sm.drain(), 0, DRAIN_NS) && lane == 0) atomicOr(p.status, ST_DRAIN);
    tc_fence_before();
    cta_bar_sync<384>();
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  } else if (warp >= 4) {
    reg_raise<BWD_REGS_HIGH>();
    const BwdSmem<STAGES> sm(smem_u32_fresh(smem_raw));
    const uint32_t sbase = sm.base;
    const WaitCtl wc{abort_flag, p.status, p.timeout_ns};
    const int n_items = wl_count(sc);
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    // ---------------------------------------------------- elementwise WGs --
    // Both warpgroups take every tile: warpgroup h owns query columns
    // [64 h, 64 h + 64).  Thread r is key row r (TMEM lane r) of S^T and dP^T.
    const int h = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + L::TM_S + h * 64;   // this half's S^T, then its P^T
    const uint32_t dp_col = lane_base + L::TM_DP + h * 64;  // this half's dP^T
    const uint32_t ds_row = sbase + L::OFF_DS + h * L::COLBLK + r * 128;  // this key row's dS^T
    const float sl = p.scale_log2, scale = p.scale;
    const uint32_t stat = sbase + L::OFF_STAT + h * 256;  // + stage * 1024: nl; + 512: nd
    bool ok = true;
    int T0 = 0, ni = 0;
    for (int k = 0; ok && k < n_items; ++k) {
      const BwdItem g = bwd_item<L::BN, L::BM>(p, sc, k);
      const int bh = g.bh, k0 = g.k0, i0 = g.i0, n_it = g.n_it;
      const bool key_ok = (k0 + r) < g.kv_limit;
      const int jrow = k0 + r - p.qoff + 1;  // causal: first visible query row of key k0 + r
      for (int t = 0; t < n_it; ++t) {
        const int T = T0 + t;
        const int st = T % STAGES;
        const int q0 = (i0 + t) * L::BM + h * 64;  // first query of this half of tile t
        // q_full is already complete here (S^T_t exists); waiting on it makes the
        // stage's nl / nd rows visible to these threads
        if (!__all_sync(0xffffffffu, mbar_wait(sm.s_full(), T & 1, wc, ST_BWD_TIMEOUT_S) &&
                                         mbar_wait(sm.q_full(st), (T / STAGES) & 1, wc, ST_BWD_TIMEOUT_Q))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float pr[64];  // P^T_t of this thread's key row over the half's 64 queries
        {
          uint32_t sr[64];
          FA_TMEM_LD32(s_col, sr);
          FA_TMEM_LD32(s_col + 32, sr + 32);
          tmem_wait_ld();
          FA_REG_FENCE32(sr);
          FA_REG_FENCE32(sr + 32);
          // causal: key k0 + r is visible to query q0 + j iff k0 + r < q0 + j + qoff
          const int jmin = p.causal ? jrow - q0 : -1;
          // only tiles on the diagonal or past a key-padding edge mask anything
          if (__any_sync(0xffffffffu, !key_ok || jmin > 0)) {
#pragma unroll
            for (int w = 0; w < 64; ++w)
              if (!key_ok || w < jmin) sr[w] = __float_as_uint(-INFINITY);
          }
          const uint32_t nl_s = stat + st * 1024;
          const uint64_t sl2 = f2_pack(sl, sl);
#pragma unroll
          for (int j4 = 0; j4 < 64; j4 += 4) {
            float nl[4];
            ld_shared_v4f(nl_s + j4 * 4, nl);
#pragma unroll
            for (int w = 0; w < 4; w += 2) {
              const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[j4 + w]), __uint_as_float(sr[j4 + w + 1])), sl2,
                                         f2_pack(nl[w], nl[w + 1]));
              constexpr int E = FA_BWD_EXP2_FMA_EVERY > 0 ? FA_BWD_EXP2_FMA_EVERY : 1;
              if (FA_BWD_EXP2_FMA_EVERY > 0 && ((j4 + w) / 2 + 1) % E == 0) {
                f2_unpack(exp2_fma2(x2), pr[j4 + w], pr[j4 + w + 1]);  // FMA pipe
              } else {
                float x0, x1;
                f2_unpack(x2, x0, x1);
                pr[j4 + w] = ex2_approx(x0);
                pr[j4 + w + 1] = ex2_approx(x1);
              }
            }
          }
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(pr[2 * i], pr[2 * i + 1]);
          FA_TMEM_ST32(s_col, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(sm.p_full());

        if (!__all_sync(0xffffffffu, mbar_wait(sm.dp_full(), T & 1, wc, ST_BWD_TIMEOUT_DP))) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          uint32_t dpr[64];
          FA_TMEM_LD32(dp_col, dpr);
          FA_TMEM_LD32(dp_col + 32, dpr + 32);
          tmem_wait_ld();
          FA_REG_FENCE32(dpr);
          FA_REG_FENCE32(dpr + 32);
          const uint32_t nd_s = stat + st * 1024 + 512;
          const uint64_t sc2 = f2_pack(scale, scale);
          uint32_t dsk[32];
#pragma unroll
          for (int j4 = 0; j4 < 64; j4 += 4) {
            float nd[4];
            ld_shared_v4f(nd_s + j4 * 4, nd);
#pragma unroll
            for (int w = 0; w < 4; w += 2) {
              // dS = P (dP scale - D scale)
              const uint64_t gr =
                  f2_mul(f2_fma(f2_pack(__uint_as_float(dpr[j4 + w]), __uint_as_float(dpr[j4 + w + 1])), sc2,
                                f2_pack(nd[w], nd[w + 1])),
                         f2_pack(pr[j4 + w], pr[j4 + w + 1]));
              float g0, g1;
              f2_unpack(gr, g0, g1);
              dsk[(j4 + w) / 2] = pack_bf16x2(g0, g1);
            }
          }
          // dS^T as MMA4's A operand, K-major in shared memory: this half's 64
          // queries are column block h, key row r is 128 bytes with its 16-byte
          // chunks rotated by r mod 8 (the 128-byte swizzle).  MMA4_{t-1}, the last
          // reader of the buffer, ran before dP^T_t was formed.
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(ds_row + ((c ^ (r & 7)) << 4), dsk[4 * c], dsk[4 * c + 1], dsk[4 * c + 2], dsk[4 * c + 3]);
          fence_proxy_async_smem();
        }
        tc_fence_before();  // the dP^T loads complete before MMA2_{t+1} overwrites the columns
        mbar_arrive(sm.ds_full());
      }

      // ---------------------------------------------------------- epilogue --
      // warpgroup 0 writes dV, warpgroup 1 writes dK: TMEM lane r = key row k0 + r
      if (ok && n_it > 0 && !__all_sync(0xffffffffu, mbar_wait(sm.dkv_done(), ni & 1, wc, ST_BWD_TIMEOUT_DONE)))
        ok = false;
      if (ok) {
        tc_fence_after();
        const int key0 = k0 + (warp & 3) * 32;  // this warp's first key row
        const size_t row0 = static_cast<size_t>(bh) * p.Nk + key0;
        const int rows = min(32, p.Nk - key0);
        const uint32_t col = lane_base + (h == 0 ? L::TM_DV : L::TM_DK);
        // staging: the first 2 KB of this warp's own rows of the dS^T buffer (free:
        // the item's products have run, and its next dS^T rows come after this)
        const uint32_t buf = sbase + L::OFF_DS + h * L::COLBLK + (warp & 3) * 4096;
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
          warp_store_rows_f32x32(v, buf, h == 0 ? p.dv : p.dk, row0, D, cb * 32, rows);
        }
        // the next item's first MMA3 / MMA4 overwrite dV and dK only after these
        // warpgroups' p_full for it, i.e. after these loads
        tc_fence_before();
      }
      if (n_it > 0) {
        T0 += n_it;
        ++ni;
      }
    }
    tc_fence_before();
    cta_bar_sync<384>();
  } else {
    reg_lower<BWD_REGS_LOW>();  // warps 2-3: no role
    cta_bar_sync<384>();
  }
}

}  // namespace fa
