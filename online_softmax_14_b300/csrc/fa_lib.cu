// libfa: the C ABI declared in include/fa.h.  Host-side argument checks, TMA
// tensor-map construction, kernel selection and launch, and the device status
// word that the kernels' bounded waits report into.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <map>
#include <memory>
#include <queue>
#include <tuple>
#include <vector>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "fa.h"
#include "ptx.cuh"
#include "fwd_simt.cuh"
#include "fwd_tc.cuh"
#include "bwd_tc.cuh"
#include "bwd_dq.cuh"
#include "merge.cuh"
#include "std_attn.cuh"

namespace fa {
// Status word of the current device: kernels OR their timeout codes into it;
// fa_check_device_error takes it (reads and clears it in one atomic exchange).
__device__ unsigned int g_status_word;
// Where the exchange leaves the word it took, for the host to copy back.
__device__ unsigned int g_status_taken;

__global__ void status_take_kernel(unsigned int* status, unsigned int* taken) { *taken = atomicExch(status, 0u); }
}  // namespace fa

namespace {

constexpr int kVersion = 200;  // 0.2.0
constexpr int kMaxDevices = 64;
constexpr int kSlotsD128 = 4;  // K/V ring slots of the forward (32 KB each at d = 128)
constexpr int kSlotsD64 = 8;   // (16 KB each at d = 64)
constexpr int kStagesBwd = 2;
constexpr int kStagesStdS = 2;   // standard attention, S = Q K^T: K = d fits in two 64-element chunks
constexpr int kStagesStdO = 3;   // standard attention, O = P V: K = Nk streams through three stages

thread_local char t_err[512] = "";
std::atomic<unsigned long long> g_timeout_ns{1000ull * 1000 * 1000};
std::atomic<int> g_inject{0};

fa_status fail(fa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return s;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceState {
  bool ready = false;
  unsigned long long ctx_id = 0;   // the CUDA context the fields below belong to
  int cc_major = 0, cc_minor = 0;
  int sm_count = 0;
  unsigned int* status = nullptr;  // device address of fa::g_status_word
  unsigned int* taken = nullptr;   // device address of fa::g_status_taken
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

using PFN_ctx_get_current = CUresult (*)(CUcontext*);
using PFN_ctx_get_id = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (creating the device's
// primary context if none is current yet).  Device addresses of the library's
// variables and the kernels' attributes belong to one context: after a
// cudaDeviceReset the caller gets a new context and they are set up again.
fa_status current_context_id(int dev, unsigned long long* id) {
  static PFN_ctx_get_current get_current = nullptr;
  static PFN_ctx_get_id get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_ctx_get_current>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_ctx_get_id>(p);
  });
  if (!get_current || !get_id) return fail(FA_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId unavailable from the driver");
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuCtxGetCurrent failed");
  if (!ctx) {
    cudaError_t e = cudaSetDevice(dev);  // makes the device's primary context current
    if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return fail(FA_ERR_CUDA, "no CUDA context after cudaSetDevice");
  }
  if (get_id(ctx, id) != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuCtxGetId failed");
  return FA_OK;
}

// Per-device set-up, done with that device current, once per CUDA context: read
// the compute capability, resolve the status words' device addresses, raise
// the kernels' dynamic shared-memory limit.
fa_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  unsigned long long ctx_id = 0;
  fa_status st = current_context_id(dev, &ctx_id);
  if (st != FA_OK) return st;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready || s.ctx_id != ctx_id) {
    s.ready = false;
    if ((e = cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (s.cc_major != 10 || s.cc_minor != 3)
      return fail(FA_ERR_UNSUPPORTED, "libfa is built for sm_103a; device %d is sm_%d%d", dev, s.cc_major,
                  s.cc_minor);
    void* addr = nullptr;
    if ((e = cudaGetSymbolAddress(&addr, fa::g_status_word)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    s.status = static_cast<unsigned int*>(addr);
    if ((e = cudaGetSymbolAddress(&addr, fa::g_status_taken)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(status copy)");
    s.taken = static_cast<unsigned int*>(addr);
    using L128 = fa::TcLayout<128, kSlotsD128>;
    using L64 = fa::TcLayout<64, kSlotsD64>;
    if ((e = cudaFuncSetAttribute(fa::fwd_bf16_tc_kernel<128, kSlotsD128>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, L128::BYTES)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(d=128)");
    if ((e = cudaFuncSetAttribute(fa::fwd_bf16_tc_kernel<64, kSlotsD64>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, L64::BYTES)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(d=64)");
    if ((e = cudaFuncSetAttribute(fa::bwd_dkdv_kernel<kStagesBwd>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  fa::BwdLayout<kStagesBwd>::BYTES)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(bwd dK dV)");
    if ((e = cudaFuncSetAttribute(fa::bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  fa::DqLayout::BYTES)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(bwd dQ)");
    if ((e = cudaFuncSetAttribute(fa::std_gemm_kernel<kStagesStdS, false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  fa::StdGemmLayout<kStagesStdS>::BYTES)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(standard S)");
    if ((e = cudaFuncSetAttribute(fa::std_gemm_kernel<kStagesStdO, true, false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  fa::StdGemmLayout<kStagesStdO>::BYTES)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(standard O)");
    s.ctx_id = ctx_id;
    s.ready = true;
  }
  *out = &s;
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [BH, N, d] bf16 viewed as a 3-D tensor (d innermost); 64 x rows x 1 boxes with
// 128-byte swizzle.  Rows past N read as zero.
fa_status make_map(CUtensorMap* m, const void* base, int d, int N, int BH, const char* name, int rows = 128) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return FA_OK;
}

// [BH, rows, cols] bf16 with row stride `ld` elements (ld * 2 a multiple of 16),
// 64 x 128 x 1 boxes with 128-byte swizzle; columns past `cols` read as zero.
fa_status make_map_strided(CUtensorMap* m, const void* base, int cols, int rows, int BH, long long ld,
                           const char* name) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(rows) * ld * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// causal: 0 none, 1 key j visible to query i iff j <= i, 2 iff j < i (strict)
fa_status check_causal(int causal) {
  if (causal < 0 || causal > 2) return fail(FA_ERR_INVALID, "causal must be 0, 1 or 2 (got %d)", causal);
  return FA_OK;
}

// Causal rule in the kernels' form, key j visible to query i iff j < i + qoff:
// the queries are the last Nq positions of the key sequence (query i at
// position i + Nk - Nq), and the strict mode excludes the query's own position.
int causal_qoff(int Nq, int Nk, int causal) { return (Nk - Nq) + (causal == 2 ? 0 : 1); }

fa_status check_common(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H,
                       int N, int d, float scale, uintptr_t align) {
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID, "q, k, v and o must be non-null device pointers");
  if (B < 1 || H < 1 || N < 1 || d < 1)
    return fail(FA_ERR_INVALID, "sizes must be >= 1 (B=%d H=%d N=%d d=%d)", B, H, N, d);
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(FA_ERR_INVALID, "scale must be finite and > 0");
  if (!aligned(q, align) || !aligned(k, align) || !aligned(v, align) || !aligned(o, align))
    return fail(FA_ERR_INVALID, "q, k, v, o must be %d-byte aligned", (int)align);
  if (lse && !aligned(lse, 4)) return fail(FA_ERR_INVALID, "lse must be 4-byte aligned");
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1ll << 30) || static_cast<long long>(N) * d > (1ll << 38))
    return fail(FA_ERR_UNSUPPORTED, "problem too large (B*H=%lld, N*d=%lld)", bh, (long long)N * d);
  return FA_OK;
}

// Work list of a persistent launch (fa::WorkList), built on the host once per
// problem shape and kind of kernel.  weights[u] is the work of unit u of a head
// (key tiles processed, plus two for an item's fixed costs); kv_len values live
// on the device and are not looked at (a padded problem just balances less
// well).  Heads are taken in groups whose operands (head_bytes each) fit in
// about 48 MB of L2; within a group the items go heaviest first, each to the
// CTA with the least work so far.
struct WorkKey {
  int kind, BH, N, Nk, causal, qoff, D, G;
  bool operator<(const WorkKey& o) const {
    return std::tie(kind, BH, N, Nk, causal, qoff, D, G) <
           std::tie(o.kind, o.BH, o.N, o.Nk, o.causal, o.qoff, o.D, o.G);
  }
};
std::map<WorkKey, std::unique_ptr<fa::WorkList>> g_work;
std::mutex g_work_mu;

const fa::WorkList* work_list(const WorkKey& key, const std::vector<int>& weights, double head_bytes) {
  std::lock_guard<std::mutex> lk(g_work_mu);
  auto found = g_work.find(key);
  if (found != g_work.end()) return found->second.get();
  auto wl = std::make_unique<fa::WorkList>();
  const int BH = key.BH, G = key.G, units = static_cast<int>(weights.size());
  const long long n_items = static_cast<long long>(BH) * units;
  wl->n_items = static_cast<int>(n_items);
  wl->table = 0;
  if (n_items <= fa::WL_MAX_ITEMS && G <= fa::WL_MAX_CTAS) {
    const int hpg = std::max(1, static_cast<int>(48.0 * 1024 * 1024 / head_bytes));
    std::vector<std::vector<uint32_t>> lists(G);
    using Load = std::pair<long long, int>;  // (work so far, CTA)
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int c = 0; c < G; ++c) heap.push({0, c});
    std::vector<std::pair<int, uint32_t>> group;  // (weight, item id)
    for (int g0 = 0; g0 < BH; g0 += hpg) {
      group.clear();
      for (int bh = g0; bh < std::min(BH, g0 + hpg); ++bh)
        for (int u = 0; u < units; ++u) group.push_back({weights[u], static_cast<uint32_t>(bh * units + u)});
      std::stable_sort(group.begin(), group.end(), [](const auto& a, const auto& b) { return a.first > b.first; });
      for (const auto& it : group) {
        Load ld = heap.top();
        heap.pop();
        lists[ld.second].push_back(it.second);
        heap.push({ld.first + it.first, ld.second});
      }
    }
    int pos = 0;
    for (int c = 0; c < G; ++c) {
      wl->start[c] = static_cast<uint16_t>(pos);
      for (uint32_t id : lists[c]) wl->list[pos++] = id;
    }
    wl->start[G] = static_cast<uint16_t>(pos);
    wl->table = 1;
  }
  const fa::WorkList* out = wl.get();
  g_work[key] = std::move(wl);
  return out;
}

// Key tiles query tile qt needs, as the kernels compute it (without kv_len).
int tiles_needed(int qt, int n_qt, int N, int Nk, int causal, int qoff) {
  const int n_kv_all = (Nk + 127) / 128;
  if (qt >= n_qt) return 0;
  if (!causal) return n_kv_all;
  const int last_key = std::min(qt * 128 + 128, N) - 1 + qoff - 1;
  return last_key < 0 ? 0 : std::min(n_kv_all, last_key / 128 + 1);
}

const fa::WorkList* fwd_work_list(int BH, int N, int Nk, int causal, int qoff, int D, int G) {
  const int n_qt = (N + 127) / 128, n_pair = (n_qt + 1) / 2;
  std::vector<int> w(n_pair);
  for (int pr = 0; pr < n_pair; ++pr)
    w[pr] = tiles_needed(2 * pr, n_qt, N, Nk, causal, qoff) + tiles_needed(2 * pr + 1, n_qt, N, Nk, causal, qoff) + 2;
  return work_list(WorkKey{0, BH, N, Nk, causal, qoff, D, G}, w, 2.0 * Nk * D * 2);  // K and V of a head
}

// dK/dV kernel: units are the key tiles of a head
const fa::WorkList* bwd_work_list(int BH, int N, int Nk, int causal, int qoff, int D, int G) {
  const int n_qt = (N + 127) / 128, n_kt = (Nk + 127) / 128;
  std::vector<int> w(n_kt);
  for (int kt = 0; kt < n_kt; ++kt) {
    const int k0 = kt * 128;
    const int i0 = causal ? std::max(0, k0 - qoff + 1) / 128 : 0;
    w[kt] = ((k0 < Nk && i0 < n_qt) ? n_qt - i0 : 0) + 2;
  }
  // Q, dO, K and V of a head
  return work_list(WorkKey{1, BH, N, Nk, causal, qoff, D, G}, w, 2.0 * (N + Nk) * D * 2);
}

// dQ kernel: units are the query tiles of a head
const fa::WorkList* dq_work_list(int BH, int N, int Nk, int causal, int qoff, int D, int G) {
  const int n_qt = (N + 127) / 128;
  std::vector<int> w(n_qt);
  for (int qt = 0; qt < n_qt; ++qt) w[qt] = tiles_needed(qt, n_qt, N, Nk, causal, qoff) + 2;
  return work_list(WorkKey{3, BH, N, Nk, causal, qoff, D, G}, w, 2.0 * (N + Nk) * D * 2);
}

template <int D, int STAGES>
fa_status launch_tc(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* kv_len, int B,
                    int H, int N, int Nk, float scale, int causal, cudaStream_t stream, const DeviceState& ds) {
  using L = fa::TcLayout<D, STAGES>;
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  fa_status s;
  if ((s = make_map(&mq, q, D, N, BH, "q")) != FA_OK) return s;
  if ((s = make_map(&mk, k, D, Nk, BH, "k")) != FA_OK) return s;
  if ((s = make_map(&mv, v, D, Nk, BH, "v")) != FA_OK) return s;
  fa::TcParams p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.kv_len = kv_len;
  p.BH = BH;
  p.H = H;
  p.N = N;
  p.Nk = Nk;
  p.n_qt = (N + 127) / 128;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.causal = causal;
  p.qoff = causal_qoff(N, Nk, causal);
  p.status = ds.status;
  p.timeout_ns = g_timeout_ns.load();
  p.inject = g_inject.load();
  // persistent grid: one CTA per SM (each holds all of an SM's tensor memory),
  // fewer when there are fewer items
  const long long n_items = static_cast<long long>((p.n_qt + 1) / 2) * BH;
  if (n_items > 0x7fffffffll) return fail(FA_ERR_UNSUPPORTED, "problem too large");
  const int G = static_cast<int>(std::min<long long>(std::max(1, ds.sm_count), n_items));
  const fa::WorkList* sc = fwd_work_list(BH, N, Nk, causal, p.qoff, D, G);
  fa::fwd_bf16_tc_kernel<D, STAGES><<<static_cast<unsigned>(G), 384, L::BYTES, stream>>>(mq, mk, mv, p, *sc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch fwd_bf16_tc_kernel");
  return FA_OK;
}

template <int DP>
fa_status launch_simt(const fa::SimtParams& p, cudaStream_t stream) {
  dim3 grid((p.N + fa::SIMT_ROWS - 1) / fa::SIMT_ROWS, p.BH);
  fa::fwd_f32_simt_kernel<DP><<<grid, fa::SIMT_WARPS * 32, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch fwd_f32_simt_kernel");
  return FA_OK;
}

// Row stride of the backward workspace arrays: N rounded up to the 128-query tile.
long long bwd_np(int N) { return (static_cast<long long>(N) + 127) / 128 * 128; }

size_t bwd_ws_bytes(int B, int H, int N) {
  return static_cast<size_t>(2) * static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(bwd_np(N)) *
         sizeof(float);
}

fa_status launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                     const int32_t* kv_len, float* dq, float* dk, float* dv, float* ws, int B, int H, int N, int Nk,
                     float scale, int causal, cudaStream_t stream, const DeviceState& ds) {
  constexpr int D = 128;
  using L = fa::BwdLayout<kStagesBwd>;
  const int BH = B * H;
  const long long Np = bwd_np(N);
  const long long pre_blocks = static_cast<long long>(BH) * (Np / 64);
  const long long n_kt = (Nk + L::BN - 1) / L::BN, n_qt = (N + fa::DqLayout::BM - 1) / fa::DqLayout::BM;
  const long long kv_items = n_kt * BH, q_items = n_qt * BH;
  if (pre_blocks > 0x7fffffffll || kv_items > 0x7fffffffll || q_items > 0x7fffffffll)
    return fail(FA_ERR_UNSUPPORTED, "grid too large");
  // persistent grids: one CTA per SM, fewer when there are fewer tiles
  const int G_kv = static_cast<int>(std::min<long long>(std::max(1, ds.sm_count), kv_items));
  const int G_q = static_cast<int>(std::min<long long>(std::max(1, ds.sm_count), q_items));

  // every tensor map is built before anything is enqueued, so that a failure
  // here leaves the stream untouched
  CUtensorMap mq, mk, mv, mdo;
  fa_status s;
  if ((s = make_map(&mq, q, D, N, BH, "q", 128)) != FA_OK) return s;
  if ((s = make_map(&mk, k, D, Nk, BH, "k", 128)) != FA_OK) return s;
  if ((s = make_map(&mv, v, D, Nk, BH, "v", 128)) != FA_OK) return s;
  if ((s = make_map(&mdo, dO, D, N, BH, "dO", 128)) != FA_OK) return s;

  fa::BwdPreParams pp{};
  pp.o = static_cast<const __nv_bfloat16*>(o);
  pp.dO = static_cast<const __nv_bfloat16*>(dO);
  pp.lse = lse;
  pp.nl = ws;
  pp.nd = ws + static_cast<size_t>(BH) * Np;
  pp.BH = BH;
  pp.N = N;
  pp.Np = static_cast<int>(Np);
  pp.scale = scale;
  fa::bwd_preprocess_kernel<D><<<static_cast<unsigned>(pre_blocks), 256, 0, stream>>>(pp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch bwd_preprocess_kernel");

  fa::BwdParams p{};
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.nl = pp.nl;
  p.nd = pp.nd;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv_len = kv_len;
  p.BH = BH;
  p.H = H;
  p.N = N;
  p.Np = static_cast<int>(Np);
  p.Nk = Nk;
  p.n_qt = static_cast<int>(n_qt);
  p.n_kt = static_cast<int>(n_kt);
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.causal = causal;
  p.qoff = causal_qoff(N, Nk, causal);
  p.status = ds.status;
  p.timeout_ns = g_timeout_ns.load();
  p.inject = g_inject.load();
  const fa::WorkList* wl_kv = bwd_work_list(BH, N, Nk, causal, p.qoff, D, G_kv);
  fa::bwd_dkdv_kernel<kStagesBwd><<<static_cast<unsigned>(G_kv), 384, L::BYTES, stream>>>(mq, mk, mv, mdo, p, *wl_kv);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch bwd_dkdv_kernel");
  const fa::WorkList* wl_q = dq_work_list(BH, N, Nk, causal, p.qoff, D, G_q);
  // programmatic stream serialization: the dQ kernel's CTAs start on the SMs the
  // dK/dV kernel's CTAs leave (it reads nothing that kernel writes, and waits for
  // it before completing)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(G_q));
  cfg.blockDim = dim3(384);
  cfg.dynamicSmemBytes = fa::DqLayout::BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, fa::bwd_dq_kernel, mk, mv, mdo, p, *wl_q)) != cudaSuccess)
    return cuda_fail(e, "launch bwd_dq_kernel");
  return FA_OK;
}


// Standard attention's workspace: S (float32) and P (bf16), each [BH][Nq][ld]
// with ld = Nk rounded up to 64 (rows of P 128-byte aligned for the tensor map).
long long std_ld(int Nk) { return (static_cast<long long>(Nk) + 63) / 64 * 64; }
size_t std_ws_bytes(int B, int H, int Nq, int Nk) {
  return static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(Nq) * static_cast<size_t>(std_ld(Nk)) * 6;
}

fa_status launch_std(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* kv_len,
                     void* ws, int B, int H, int N, int Nk, int d, float scale, int causal, cudaStream_t stream,
                     const DeviceState& ds) {
  const int BH = B * H;
  const long long ld = std_ld(Nk);
  float* s_buf = static_cast<float*>(ws);
  __nv_bfloat16* p_buf = reinterpret_cast<__nv_bfloat16*>(s_buf + static_cast<size_t>(BH) * N * ld);
  CUtensorMap mq, mk, mp, mv;
  fa_status s;
  if ((s = make_map(&mq, q, d, N, BH, "q")) != FA_OK) return s;
  if ((s = make_map(&mk, k, d, Nk, BH, "k")) != FA_OK) return s;
  if ((s = make_map_strided(&mp, p_buf, Nk, N, BH, ld, "p")) != FA_OK) return s;
  if ((s = make_map(&mv, v, d, Nk, BH, "v", 64)) != FA_OK) return s;
  const long long tiles_m = (N + 127) / 128, tiles_n = (Nk + 127) / 128;
  if (tiles_m * tiles_n > 0x7fffffffll || BH > 65535) return fail(FA_ERR_UNSUPPORTED, "grid too large");
  // S = scale Q K^T, every entry
  fa::StdGemmParams gs{};
  gs.c = s_buf;
  gs.ldc = ld;
  gs.c_batch = static_cast<long long>(N) * ld;
  gs.M = N;
  gs.N = Nk;
  gs.K = d;
  gs.tiles_n = static_cast<int>(tiles_n);
  gs.alpha = scale;
  gs.status = ds.status;
  gs.timeout_ns = g_timeout_ns.load();
  fa::std_gemm_kernel<kStagesStdS, false, true>
      <<<dim3(static_cast<unsigned>(tiles_m * tiles_n), BH), 128, fa::StdGemmLayout<kStagesStdS>::BYTES, stream>>>(
          mq, mk, gs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch std_gemm_kernel (S)");
  // P = softmax(S) with the mask, lse
  fa::StdSoftmaxParams sp{};
  sp.s = s_buf;
  sp.p = p_buf;
  sp.lse = lse;
  sp.kv_len = kv_len;
  sp.ld = ld;
  sp.BH = BH;
  sp.H = H;
  sp.Nq = N;
  sp.Nk = Nk;
  sp.causal = causal;
  sp.qoff = causal_qoff(N, Nk, causal);
  const long long rows = static_cast<long long>(BH) * N;
  fa::std_softmax_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(sp);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch std_softmax_kernel");
  // O = P V over every key
  fa::StdGemmParams go{};
  go.c = o;
  go.ldc = d;
  go.c_batch = static_cast<long long>(N) * d;
  go.M = N;
  go.N = d;
  go.K = Nk;
  go.tiles_n = 1;
  go.alpha = 1.f;
  go.status = ds.status;
  go.timeout_ns = g_timeout_ns.load();
  fa::std_gemm_kernel<kStagesStdO, true, false>
      <<<dim3(static_cast<unsigned>(tiles_m), BH), 128, fa::StdGemmLayout<kStagesStdO>::BYTES, stream>>>(mp, mv, go);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch std_gemm_kernel (O)");
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_fwd_qk(int dtype, const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* kv_len, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                    void* stream) {
  t_err[0] = '\0';
  fa_status s;
  if ((s = check_causal(causal)) != FA_OK) return s;
  if (Nk < 1) return fail(FA_ERR_INVALID, "Nk must be >= 1 (got %d)", Nk);
  if (static_cast<long long>(Nk) * d > (1ll << 38)) return fail(FA_ERR_UNSUPPORTED, "problem too large (Nk*d)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == FA_BF16) {
    if ((s = check_common(q, k, v, o, lse, B, H, Nq, d, scale, 16)) != FA_OK) return s;
    if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "bf16 path serves d = 64 or 128 (got %d)", d);
    DeviceState* ds = nullptr;
    if ((s = device_state(&ds)) != FA_OK) return s;
    if (d == 128) return launch_tc<128, kSlotsD128>(q, k, v, o, lse, kv_len, B, H, Nq, Nk, scale, causal, st, *ds);
    return launch_tc<64, kSlotsD64>(q, k, v, o, lse, kv_len, B, H, Nq, Nk, scale, causal, st, *ds);
  }
  if (dtype == FA_FP32) {
    if ((s = check_common(q, k, v, o, lse, B, H, Nq, d, scale, 4)) != FA_OK) return s;
    if (d > 128) return fail(FA_ERR_UNSUPPORTED, "fp32 path serves d <= 128 (got %d)", d);
    if (static_cast<long long>(B) * H > 65535) return fail(FA_ERR_UNSUPPORTED, "fp32 path serves B*H <= 65535");
    DeviceState* ds = nullptr;
    if ((s = device_state(&ds)) != FA_OK) return s;
    fa::SimtParams p{};
    p.q = static_cast<const float*>(q);
    p.k = static_cast<const float*>(k);
    p.v = static_cast<const float*>(v);
    p.o = static_cast<float*>(o);
    p.lse = lse;
    p.kv_len = kv_len;
    p.BH = B * H;
    p.H = H;
    p.N = Nq;
    p.Nk = Nk;
    p.d = d;
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.causal = causal;
    p.qoff = causal_qoff(Nq, Nk, causal);
    if (d <= 32) return launch_simt<32>(p, st);
    if (d <= 64) return launch_simt<64>(p, st);
    if (d <= 96) return launch_simt<96>(p, st);
    return launch_simt<128>(p, st);
  }
  return fail(FA_ERR_INVALID, "unknown dtype %d", dtype);
}

fa_status fa_fwd_ex(int dtype, const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* kv_len, int B, int H, int N, int d, float scale, int causal, void* stream) {
  return fa_fwd_qk(dtype, q, k, v, o, lse, kv_len, B, H, N, N, d, scale, causal, stream);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, void* stream) {
  return fa_fwd_ex(FA_BF16, q, k, v, o, lse, nullptr, B, H, N, d, scale, causal, stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  return bwd_ws_bytes(B, H, N);
}

fa_status fa_bwd_qk(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    const int32_t* kv_len, float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes,
                    int B, int H, int Nq, int Nk, int d, float scale, int causal, void* stream) {
  t_err[0] = '\0';
  fa_status s;
  if ((s = check_causal(causal)) != FA_OK) return s;
  if (Nk < 1) return fail(FA_ERR_INVALID, "Nk must be >= 1 (got %d)", Nk);
  if (static_cast<long long>(Nk) * d > (1ll << 38)) return fail(FA_ERR_UNSUPPORTED, "problem too large (Nk*d)");
  if ((s = check_common(q, k, v, o, lse, B, H, Nq, d, scale, 16)) != FA_OK) return s;
  if (!dO || !lse || !dq || !dk || !dv || !workspace)
    return fail(FA_ERR_INVALID, "dO, lse, dq, dk, dv and workspace must be non-null device pointers");
  if (!aligned(dO, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(workspace, 16))
    return fail(FA_ERR_INVALID, "dO, dq, dk, dv and workspace must be 16-byte aligned");
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "bf16 backward serves d = 128 (got %d)", d);
  const size_t need = bwd_ws_bytes(B, H, Nq);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu bytes required", workspace_bytes,
                need);
  DeviceState* ds = nullptr;
  if ((s = device_state(&ds)) != FA_OK) return s;
  return launch_bwd(q, k, v, o, dO, lse, kv_len, dq, dk, dv, static_cast<float*>(workspace), B, H, Nq, Nk, scale,
                    causal, static_cast<cudaStream_t>(stream), *ds);
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    const int32_t* kv_len, float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes,
                    int B, int H, int N, int d, float scale, int causal, void* stream) {
  return fa_bwd_qk(q, k, v, o, dO, lse, kv_len, dq, dk, dv, workspace, workspace_bytes, B, H, N, N, d, scale, causal,
                   stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 float scale, int causal, void* stream) {
  return fa_bwd_ex(q, k, v, o, dO, lse, nullptr, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale, causal,
                   stream);
}

fa_status fa_merge(int dtype, const void* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int B,
                   int H, int N, int d, void* stream) {
  t_err[0] = '\0';
  if (!o_parts || !lse_parts || !o) return fail(FA_ERR_INVALID, "o_parts, lse_parts and o must be non-null");
  if (B < 1 || H < 1 || N < 1 || d < 1 || n_parts < 1)
    return fail(FA_ERR_INVALID, "sizes must be >= 1 (B=%d H=%d N=%d d=%d n_parts=%d)", B, H, N, d, n_parts);
  if (d > 256) return fail(FA_ERR_UNSUPPORTED, "merge serves d <= 256 (got %d)", d);
  if (n_parts > 4096) return fail(FA_ERR_UNSUPPORTED, "merge serves at most 4096 parts (got %d)", n_parts);
  if (dtype != FA_BF16 && dtype != FA_FP32) return fail(FA_ERR_INVALID, "unknown dtype %d", dtype);
  const uintptr_t al = (dtype == FA_FP32) ? 4 : 2;
  if (!aligned(o_parts, al) || !aligned(o, al) || !aligned(lse_parts, 4) || (lse && !aligned(lse, 4)))
    return fail(FA_ERR_INVALID, "misaligned pointer (o_parts/o need %d bytes, lse 4)", (int)al);
  const long long R = static_cast<long long>(B) * H * N;
  const long long blocks = (R + fa::MERGE_ROWS - 1) / fa::MERGE_ROWS;
  if (R > (1ll << 40) || blocks > 0x7fffffffll) return fail(FA_ERR_UNSUPPORTED, "problem too large");
  fa_status s;
  DeviceState* ds = nullptr;
  if ((s = device_state(&ds)) != FA_OK) return s;
  fa::MergeParams p{o_parts, lse_parts, o, lse, R, n_parts, d};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 block(fa::MERGE_ROWS * 32);
  // 16-byte vectors when a row is 16, 32, ..., 512 bytes and both tensors are 16-byte aligned
  const int row_bytes = d * static_cast<int>(al);
  const int lpr = row_bytes / 16;
  if (row_bytes % 16 == 0 && lpr >= 1 && lpr <= 32 && (lpr & (lpr - 1)) == 0 && aligned(o_parts, 16) &&
      aligned(o, 16)) {
    const long long rows_per_cta = static_cast<long long>(fa::MERGE_ROWS) * (32 / lpr);
    const dim3 vgrid(static_cast<unsigned>((R + rows_per_cta - 1) / rows_per_cta));
#define FA_MERGE_VEC(T)                                                                            \
  switch (lpr) {                                                                                   \
    case 1: fa::merge_vec_kernel<T, 1><<<vgrid, block, 0, st>>>(p); break;                         \
    case 2: fa::merge_vec_kernel<T, 2><<<vgrid, block, 0, st>>>(p); break;                         \
    case 4: fa::merge_vec_kernel<T, 4><<<vgrid, block, 0, st>>>(p); break;                         \
    case 8: fa::merge_vec_kernel<T, 8><<<vgrid, block, 0, st>>>(p); break;                         \
    case 16: fa::merge_vec_kernel<T, 16><<<vgrid, block, 0, st>>>(p); break;                       \
    default: fa::merge_vec_kernel<T, 32><<<vgrid, block, 0, st>>>(p); break;                       \
  }
    if (dtype == FA_FP32) {
      FA_MERGE_VEC(float)
    } else {
      FA_MERGE_VEC(__nv_bfloat16)
    }
#undef FA_MERGE_VEC
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch merge_vec_kernel");
    return FA_OK;
  }
  const dim3 grid(static_cast<unsigned>(blocks));
  if (dtype == FA_FP32) {
    if (d <= 128) fa::merge_kernel<float, 4><<<grid, block, 0, st>>>(p);
    else fa::merge_kernel<float, 8><<<grid, block, 0, st>>>(p);
  } else {
    if (d <= 128) fa::merge_kernel<__nv_bfloat16, 4><<<grid, block, 0, st>>>(p);
    else fa::merge_kernel<__nv_bfloat16, 8><<<grid, block, 0, st>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch merge_kernel");
  return FA_OK;
}

size_t fa_std_workspace_size(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  return std_ws_bytes(B, H, N, N);
}

fa_status fa_std_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* kv_len,
                     void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                     void* stream) {
  t_err[0] = '\0';
  fa_status s;
  if ((s = check_causal(causal)) != FA_OK) return s;
  if ((s = check_common(q, k, v, o, lse, B, H, N, d, scale, 16)) != FA_OK) return s;
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "standard attention serves d = 64 or 128 (got %d)", d);
  if (!workspace || !aligned(workspace, 16)) return fail(FA_ERR_INVALID, "workspace must be a 16-byte aligned device pointer");
  const size_t need = std_ws_bytes(B, H, N, N);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu bytes required", workspace_bytes, need);
  DeviceState* ds = nullptr;
  if ((s = device_state(&ds)) != FA_OK) return s;
  return launch_std(q, k, v, o, lse, kv_len, workspace, B, H, N, N, d, scale, causal,
                    static_cast<cudaStream_t>(stream), *ds);
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID: return "FA_ERR_INVALID";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_UNKNOWN_STATUS";
  }
}

const char* fa_last_error_string(void) { return t_err; }

fa_status fa_check_device_error(void* stream) {
  t_err[0] = '\0';
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  DeviceState* ds = nullptr;
  fa_status s = device_state(&ds);
  if (s != FA_OK) return s;
  // Take the word (read and clear in one atomic exchange on the device, so a bit
  // a kernel on another stream sets meanwhile is never lost), then copy it back.
  unsigned int word = 0;
  {
    static std::mutex take_mu;  // one copy-back slot per device
    std::lock_guard<std::mutex> lk(take_mu);
    fa::status_take_kernel<<<1, 1, 0, st>>>(ds->status, ds->taken);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch status_take_kernel");
    if ((e = cudaMemcpyAsync(&word, ds->taken, sizeof(word), cudaMemcpyDeviceToHost, st)) != cudaSuccess)
      return cuda_fail(e, "read status word");
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  }
  if (word == 0) return FA_OK;
  if (word & fa::ST_BWD_SMEM_ALIGN)
    return fail(FA_ERR_CUDA, "backward kernel found its shared memory base misaligned and did nothing (status bits "
                "0x%x)", word);
  return fail(FA_ERR_TIMEOUT, "kernel pipeline wait timed out (status bits 0x%x)", word);
}

void fa_set_wait_timeout_ms(int ms) {
  if (ms < 1) ms = 1;
  g_timeout_ns.store(static_cast<unsigned long long>(ms) * 1000ull * 1000ull);
}

void fa_debug_inject(int code) { g_inject.store(code); }

int fa_version(void) { return kVersion; }

}  // extern "C"

// ------------------------------------------------------------------------------
// Backward without any allocation.
//
// Some callers cannot allocate device memory at the moment they need a
// gradient. Examples: code that runs inside a custom allocator's own callbacks,
// a runtime whose memory pool is fixed and fully handed out at start-up, and
// embedded hosts whose policy forbids cudaMalloc after initialisation. They
// cannot provide the backward's workspace, so for them the library keeps it in
// a fixed device array that is part of the loaded module. Every GPU that loads
// the library holds this array until the process exits.
//
// Limit: the workspace is two float32 arrays of B*H*Np rows (Np = N rounded up
// to 128), so B*H*Np may be at most FA_BWD_NOALLOC_MAX_ROWS (4 MiB in total).
// Calls share the array: two calls that run at the same time on the GPU (for
// instance on different streams) overwrite each other's workspace and give
// wrong gradients, so such calls must be ordered. Nothing in the array needs to
// start at zero. Every row a call reads has first been written by that same
// call's preprocess kernel, so stale contents from an earlier call do no harm.
namespace {

static __device__ __align__(256) float g_bwd_noalloc_scratch[2 * FA_BWD_NOALLOC_MAX_ROWS];

float* g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// The array's device address for the current device, looked up with that
// device current, again whenever the CUDA context has changed (the host-side
// name of the array is only a stand-in and must never be handed to a kernel).
fa_status noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  unsigned long long ctx_id = 0;
  fa_status st = current_context_id(dev, &ctx_id);
  if (st != FA_OK) return st;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx_id) {
    void* addr = nullptr;
    if ((e = cudaGetSymbolAddress(&addr, g_bwd_noalloc_scratch)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(backward scratch)");
    g_noalloc_ptr[dev] = static_cast<float*>(addr);
    g_noalloc_ctx[dev] = ctx_id;
  }
  *out = g_noalloc_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, float* dq, float* dk, float* dv, int B, int H, int N, int d,
                                    float scale, int causal, void* stream) {
  t_err[0] = '\0';
  fa_status s;
  if ((s = check_causal(causal)) != FA_OK) return s;
  if ((s = check_common(q, k, v, o, lse, B, H, N, d, scale, 16)) != FA_OK) return s;
  if (!dO || !lse || !dq || !dk || !dv)
    return fail(FA_ERR_INVALID, "dO, lse, dq, dk and dv must be non-null device pointers");
  if (!aligned(dO, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return fail(FA_ERR_INVALID, "dO, dq, dk and dv must be 16-byte aligned");
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "bf16 backward serves d = 128 (got %d)", d);
  const long long rows = static_cast<long long>(B) * H * bwd_np(N);
  if (rows > FA_BWD_NOALLOC_MAX_ROWS)
    return fail(FA_ERR_UNSUPPORTED,
                "fa_bwd_noalloc: B*H*Np = %lld rows (Np = N rounded up to 128) exceeds its fixed scratch of %d rows; "
                "use fa_bwd with a caller-supplied workspace",
                rows, (int)FA_BWD_NOALLOC_MAX_ROWS);
  DeviceState* ds = nullptr;
  if ((s = device_state(&ds)) != FA_OK) return s;
  float* ws = nullptr;
  if ((s = noalloc_scratch(&ws)) != FA_OK) return s;
  return launch_bwd(q, k, v, o, dO, lse, nullptr, dq, dk, dv, ws, B, H, N, N, scale, causal,
                    static_cast<cudaStream_t>(stream), *ds);
}
