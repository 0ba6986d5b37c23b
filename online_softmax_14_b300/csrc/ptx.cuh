// Inline-PTX wrappers for sm_103a: mbarriers, TMA tensor loads, tcgen05 (UMMA,
// tensor memory) and a few ALU helpers.  Every wait on an mbarrier is bounded:
// after a time limit it records an error code in a global status word and tells
// the other roles of the CTA to stop, so a broken pipeline ends with a status the
// host can read instead of a hung GPU.
#pragma once
#include <cstdint>
#include <cuda.h>  // CUtensorMap (type only; no driver symbols are linked)

namespace fa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The same conversion in a volatile asm: every call is a separate value, so a
// role of a warp-specialised kernel can take its own copy after changing its
// register budget instead of keeping one from before the change live.
__device__ __forceinline__ uint32_t smem_u32_fresh(const void* p) {
  uint32_t a;
  asm volatile("{\n\t.reg .u64 t;\n\tcvta.to.shared.u64 t, %1;\n\tcvt.u32.u64 %0, t;\n\t}" : "=r"(a) : "l"(p));
  return a;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier ---
// Barriers are named by their 32-bit shared-memory address (smem_u32); the
// pointer forms below convert and forward.  Kernels with many barriers keep
// the addresses as 32-bit values so that warps with small register budgets do
// not hold 64-bit pointers.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) { mbar_init(smem_u32(bar), count); }
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) { mbar_arrive(smem_u32(bar)); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  mbar_arrive_expect_tx(smem_u32(bar), bytes);
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared state for bounded waits: a per-CTA abort flag (shared memory) and the
// library's global status word.
struct WaitCtl {
  volatile int* abort_flag;  // shared memory
  unsigned int* status;      // global memory
  uint64_t timeout_ns;
};

// Wait until the phase with the given parity has completed.  Returns false if the
// CTA was told to abort or the wait ran past the time limit (which then records
// `code` in the status word and raises the abort flag).
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, const WaitCtl& w, unsigned code) {
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        *w.abort_flag = 1;
        atomicOr(w.status, code);
        return false;
      }
    }
  }
}

// mbar_wait for a whole converged warp: every lane tests the barrier and the
// outcome is made warp-uniform (a phase, once complete, stays complete).
__device__ __forceinline__ bool mbar_wait_w(uint32_t a, uint32_t parity, const WaitCtl& w, unsigned code) {
  if (__any_sync(0xffffffffu, mbar_try_wait(a, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (__any_sync(0xffffffffu, mbar_try_wait(a, parity))) return true;
    if ((it & 63u) == 0u) {
      if (__any_sync(0xffffffffu, *w.abort_flag != 0)) return false;
      if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > w.timeout_ns)) {
        if ((threadIdx.x & 31) == 0) {
          *w.abort_flag = 1;
          atomicOr(w.status, code);
        }
        return false;
      }
    }
  }
}

// Wait with a limit, ignoring the abort flag: used only while draining work that
// is already in flight before a CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t a, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w, unsigned code) {
  return mbar_wait(smem_u32(bar), parity, w, code);
}
__device__ __forceinline__ bool mbar_wait_w(uint64_t* bar, uint32_t parity, const WaitCtl& w, unsigned code) {
  return mbar_wait_w(smem_u32(bar), parity, w, code);
}
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  return mbar_wait_drain(smem_u32(bar), parity, limit_ns);
}

// ---------------------------------------------- programmatic dependent launch ---
// Lets the next kernel on the stream, launched with programmatic stream
// serialization, start its CTAs once every CTA of this grid has executed this
// (or exited).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the grids this one was allowed to overlap have completed and their
// memory operations are visible (returns at once without such a dependency).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// -------------------------------------------------------------------- TMA ---
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled load global -> shared, completion counted in bytes on `bar`.
// x (innermost coordinate, elements) must make x * sizeof(elem) a multiple of 16.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
  tma_load_3d(smem_u32(dst), m, smem_u32(bar), x, y, z);
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void ld_shared_v4f(uint32_t addr, float* v) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
               : "r"(addr)
               : "memory");
}
// ---------------------------------------------------------------- tcgen05 ---
// Tensor-memory allocation (whole warp).  The allocated base address is written
// to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// tcgen05.mma, issued from a converged warp: D[tmem] (+)= A * B, bf16 in, f32
// accumulate; A from shared memory (umma_ss_w) or tensor memory (umma_ts_w), B
// from shared memory.  All 32 lanes of the issuing warp run the issue code (the
// operands are warp-uniform) and lane 0 alone executes the tensor-core
// instruction through a predicate.  Measured on B300: a barrier test between two
// groups of MMAs stalls the tensor pipe for ~190 cycles when one lane runs the
// issue code on its own, and for ~20 cycles when the warp stays converged.
__device__ __forceinline__ void umma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "mov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "mov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// A whole K = 16 NK group of MMAs in one asm block: lane 0 of the converged warp
// issues NK tcgen05.mma, the first accumulating iff `accumulate` != 0 and the
// rest always accumulating.  Operand addresses of step kk are the base plus a
// fixed offset: descriptor offsets in 16-byte units (the start-address field),
// tensor-memory A offsets in columns.  Measured on B300: a group of 8 goes out in
// about 15 cycles this way, against about 300 when each MMA is its own asm
// statement, and the issuing warp is free again that much sooner.
//   *_k8 / *_k4: K-major shared-memory operand, 128-byte swizzle, two 16 KB
//                column blocks of 64 elements (steps 0-3 in the first, 4-7 in the
//                second), 32 bytes per step;
//   *_mn8:       MN-major shared-memory B, 16 rows (2 KB) per step;
//   A in tensor memory (ts): 8 columns per step, contiguous (_c) or split in
//                two 32-column halves 64 columns apart (_h).
#define FA_UMMA_HEAD                                                                               \
  "{\n\t.reg .pred e, p;\n\t.reg .b32 l, t1;\n\t.reg .b64 a1, b1;\n\t"                             \
  "mov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\tsetp.ne.b32 p, %4, 0;\n\t"
#define FA_UMMA_SS_FIRST "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
#define FA_UMMA_TS_FIRST "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
#define FA_UMMA_SS(OA, OB)                                                                         \
  "add.s64 a1, %1, " #OA ";\n\tadd.s64 b1, %2, " #OB ";\n\t"                                       \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, 1;\n\t"
#define FA_UMMA_TS(OA, OB)                                                                         \
  "add.u32 t1, %1, " #OA ";\n\tadd.s64 b1, %2, " #OB ";\n\t"                                       \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t1], b1, %3, 1;\n\t"

__device__ __forceinline__ void umma_ss_k8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_UMMA_HEAD FA_UMMA_SS_FIRST FA_UMMA_SS(2, 2) FA_UMMA_SS(4, 4) FA_UMMA_SS(6, 6)
                   FA_UMMA_SS(1024, 1024) FA_UMMA_SS(1026, 1026) FA_UMMA_SS(1028, 1028) FA_UMMA_SS(1030, 1030) "}" ::"r"(d),
               "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
               : "memory");
}
__device__ __forceinline__ void umma_ss_k4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_UMMA_HEAD FA_UMMA_SS_FIRST FA_UMMA_SS(2, 2) FA_UMMA_SS(4, 4) FA_UMMA_SS(6, 6) "}" ::"r"(d), "l"(a),
               "l"(b), "r"(idesc), "r"(accumulate)
               : "memory");
}
// A from tensor memory (contiguous), B MN-major
__device__ __forceinline__ void umma_ts_c_mn8(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_UMMA_HEAD FA_UMMA_TS_FIRST FA_UMMA_TS(8, 128) FA_UMMA_TS(16, 256) FA_UMMA_TS(24, 384)
                   FA_UMMA_TS(32, 512) FA_UMMA_TS(40, 640) FA_UMMA_TS(48, 768) FA_UMMA_TS(56, 896) "}" ::"r"(d),
               "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
               : "memory");
}
// A from tensor memory (two halves 64 columns apart), B MN-major
__device__ __forceinline__ void umma_ts_h_mn8(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_UMMA_HEAD FA_UMMA_TS_FIRST FA_UMMA_TS(8, 128) FA_UMMA_TS(16, 256) FA_UMMA_TS(24, 384)
                   FA_UMMA_TS(64, 512) FA_UMMA_TS(72, 640) FA_UMMA_TS(80, 768) FA_UMMA_TS(88, 896) "}" ::"r"(d),
               "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
               : "memory");
}
// A from tensor memory (contiguous), B K-major
__device__ __forceinline__ void umma_ts_c_k8(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_UMMA_HEAD FA_UMMA_TS_FIRST FA_UMMA_TS(8, 2) FA_UMMA_TS(16, 4) FA_UMMA_TS(24, 6)
                   FA_UMMA_TS(32, 1024) FA_UMMA_TS(40, 1026) FA_UMMA_TS(48, 1028) FA_UMMA_TS(56, 1030) "}" ::"r"(d),
               "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
               : "memory");
}

// Lane 0 (the lane that issued the MMAs) arrives once on `bar` when every
// tcgen05.mma it has issued so far is done.
__device__ __forceinline__ void umma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\t"
      "mov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void umma_commit_w(uint64_t* bar) { umma_commit_w(smem_u32(bar)); }

// Instruction descriptor, kind::f16 with bf16 A and B, f32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   15 A major (1 = MN-major), 16 B major (1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn_major, bool a_mn_major = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   bits 0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 version (1), 61-63 layout (2 = 128B swizzle).
// K-major: rows of 128 bytes, 8-row atoms of 1024 bytes, SBO = atom stride.
// MN-major: 64-element rows along MN, LBO = stride between 64-wide MN blocks,
//           SBO = stride between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16) |
         (static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// 32 lanes x 32 bits, 32 consecutive columns per thread.
#define FA_TMEM_LD32(taddr, r)                                                                                 \
  asm volatile(                                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"       \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                              \
      : "=r"((r)[0]), "=r"((r)[1]), "=r"((r)[2]), "=r"((r)[3]), "=r"((r)[4]), "=r"((r)[5]), "=r"((r)[6]),      \
        "=r"((r)[7]), "=r"((r)[8]), "=r"((r)[9]), "=r"((r)[10]), "=r"((r)[11]), "=r"((r)[12]),                \
        "=r"((r)[13]), "=r"((r)[14]), "=r"((r)[15]), "=r"((r)[16]), "=r"((r)[17]), "=r"((r)[18]),             \
        "=r"((r)[19]), "=r"((r)[20]), "=r"((r)[21]), "=r"((r)[22]), "=r"((r)[23]), "=r"((r)[24]),             \
        "=r"((r)[25]), "=r"((r)[26]), "=r"((r)[27]), "=r"((r)[28]), "=r"((r)[29]), "=r"((r)[30]),             \
        "=r"((r)[31])                                                                                         \
      : "r"(taddr))

#define FA_TMEM_ST32(taddr, r)                                                                                 \
  asm volatile(                                                                                               \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16," \
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),                        \
      "r"((r)[0]), "r"((r)[1]), "r"((r)[2]), "r"((r)[3]), "r"((r)[4]), "r"((r)[5]), "r"((r)[6]), "r"((r)[7]), \
      "r"((r)[8]), "r"((r)[9]), "r"((r)[10]), "r"((r)[11]), "r"((r)[12]), "r"((r)[13]), "r"((r)[14]),         \
      "r"((r)[15]), "r"((r)[16]), "r"((r)[17]), "r"((r)[18]), "r"((r)[19]), "r"((r)[20]), "r"((r)[21]),       \
      "r"((r)[22]), "r"((r)[23]), "r"((r)[24]), "r"((r)[25]), "r"((r)[26]), "r"((r)[27]), "r"((r)[28]),       \
      "r"((r)[29]), "r"((r)[30]), "r"((r)[31])                                                                \
      : "memory")

// 32 lanes x 32 bits, 16 consecutive columns per thread.
#define FA_TMEM_ST16(taddr, r)                                                                                 \
  asm volatile(                                                                                               \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" \
      ::"r"(taddr), "r"((r)[0]), "r"((r)[1]), "r"((r)[2]), "r"((r)[3]), "r"((r)[4]), "r"((r)[5]), "r"((r)[6]),  \
      "r"((r)[7]), "r"((r)[8]), "r"((r)[9]), "r"((r)[10]), "r"((r)[11]), "r"((r)[12]), "r"((r)[13]),          \
      "r"((r)[14]), "r"((r)[15])                                                                              \
      : "memory")

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Registers written by tcgen05.ld are valid only after tcgen05.wait::ld.  The
// compiler sees them as defined at the load, so after each wait this empty asm
// "rewrites" them: every later use then depends on a point after the wait.
#define FA_REG_FENCE32(r)                                                                                     \
  asm volatile(""                                                                                             \
               : "+r"((r)[0]), "+r"((r)[1]), "+r"((r)[2]), "+r"((r)[3]), "+r"((r)[4]), "+r"((r)[5]),          \
                 "+r"((r)[6]), "+r"((r)[7]), "+r"((r)[8]), "+r"((r)[9]), "+r"((r)[10]), "+r"((r)[11]),        \
                 "+r"((r)[12]), "+r"((r)[13]), "+r"((r)[14]), "+r"((r)[15]), "+r"((r)[16]), "+r"((r)[17]),    \
                 "+r"((r)[18]), "+r"((r)[19]), "+r"((r)[20]), "+r"((r)[21]), "+r"((r)[22]), "+r"((r)[23]),    \
                 "+r"((r)[24]), "+r"((r)[25]), "+r"((r)[26]), "+r"((r)[27]), "+r"((r)[28]), "+r"((r)[29]),    \
                 "+r"((r)[30]), "+r"((r)[31]))
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Barrier 1 across all `nthreads` threads of the CTA, executed from inside a
// role's own branch.  Warp-specialised kernels end each role with it (instead of
// one __syncthreads after the branches join), so that no value has to stay live
// into a join shared by roles with different register budgets.
// The warp reconverges first: bar.sync is warp-aligned, and some roles reach it
// after work done by one lane.
template <int nthreads>
__device__ __forceinline__ void cta_bar_sync() {
  __syncwarp();
  asm volatile("bar.sync 1, %0;" ::"n"(nthreads) : "memory");
}

// Per-warp register budget of a warp-specialised kernel: a warp's role lowers
// or raises its share of the registers the CTA was launched with.  Every warp of
// a warpgroup takes the same value; the raised and lowered shares must add up
// to no more than the launch's registers (threads x registers per thread), or
// the raise would wait for registers that never come.
template <uint32_t N>
__device__ __forceinline__ void reg_raise() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}
template <uint32_t N>
__device__ __forceinline__ void reg_lower() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------- ALU ---
// Packed pair of floats in one 64-bit register: the sm_100 family's f32x2
// arithmetic (fma/add on both halves in one instruction).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x on the special-function unit (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Pack two floats to bf16x2, round to nearest even; `lo` lands in the low half
// (the lower address in memory order).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace fa
