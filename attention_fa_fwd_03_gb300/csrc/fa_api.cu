// C ABI of the attention library: argument validation, TMA map encoding and
// dispatch to the per-head-dim kernels. Nothing here allocates device memory.
//
// The checks follow the conventions of include/fa.h: errors are returned
// before anything is launched and never abort the process (page
// "R/ag_flash_attn.R" (ggmlR), the f32-only backward note: an abort inside the
// library took the whole session down, so every shape error is reported to
// the caller instead).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/fa.h"
#include "fa_launch.h"

namespace fa {

__device__ uint32_t g_device_status;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Default bound of every device wait, in SM clock cycles: FA_WAIT_TIMEOUT_MS
// (default 4000 ms) at 2.2 GHz, above the GB300's highest SM clock, so at any
// real clock the wait lasts at least that long.
uint64_t default_wait_cycles() {
  static const uint64_t cycles = [] {
    const char* env = std::getenv("FA_WAIT_TIMEOUT_MS");
    long ms = env ? std::strtol(env, nullptr, 10) : 0;
    if (ms <= 0) ms = 4000;
    return static_cast<uint64_t>(ms) * 2200000ull;
  }();
  return cycles;
}

// Process-wide override of the bound of the ordinary waits (0: the default),
// set by fa_set_wait_limit_cycles for tests of the give-up path.
std::atomic<uint64_t> g_wait_override{0};

uint64_t wait_timeout_cycles() {
  const uint64_t o = g_wait_override.load(std::memory_order_relaxed);
  return o != 0 ? o : default_wait_cycles();
}

// The waits at exit that let in-flight copies and MMAs finish keep the default
// bound whatever the override is.
void set_waits(WaitCfg* wc) {
  wc->timeout_cycles = wait_timeout_cycles();
  wc->drain_cycles = default_wait_cycles();
}

bool status_ptr(uint32_t** p) {
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return false;
  *p = static_cast<uint32_t*>(addr);
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [lo, hi) byte ranges of two buffers intersect.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

constexpr int kMaxSeq = 1 << 22;        // keeps every grid dimension within limits
constexpr int64_t kMaxHeads = 1 << 24;  // B * Hq

fa_status check_common(int B, int Hq, int Hkv, int Tq, int Tkv, int D, float scale, int causal,
                       int window, fa_dtype dt) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tkv < 1) return FA_ERR_INVALID_ARG;
  if (Tq > kMaxSeq || Tkv > kMaxSeq) return FA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * Hq > kMaxHeads) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  // every kernel runs a 1-D grid of (head or group) x (128-row block) CTAs
  if (static_cast<int64_t>(B) * Hq * ((Tq + 127) / 128) > INT32_MAX ||
      static_cast<int64_t>(B) * Hkv * ((Tkv + 127) / 128) > INT32_MAX)
    return FA_ERR_INVALID_ARG;
  if (!(D == 64 || D == 96 || D == 128 || D == 256)) return FA_ERR_UNSUPPORTED_HEAD_DIM;
  if (dt != FA_FP16 && dt != FA_BF16) return FA_ERR_UNSUPPORTED_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (window < 0) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Mask-free attention with grouped query heads: the Tq rows of the r query
// heads of one KV group are consecutive in memory ([B, Hq, Tq, D] is
// [B, Hkv, r * Tq, D], and the LSE and D-vector [B, Hq, Tq] likewise), and
// without a mask every row sees the same keys, so the call is the same
// problem with Hq' = Hkv and Tq' = r * Tq. Below one 128-row tile this packs
// the heads' rows into shared tiles instead of padding each head's few rows
// to a tile of its own (and the dK/dV kernel then walks one query tile per
// key tile instead of r). Rows with Tq <= min_tq are left alone.
void fold_group_rows(int causal, int window, int Hkv, int min_tq, int* Hq, int* Tq) {
  if (causal || window > 0 || *Hq == Hkv || *Tq >= kBM || *Tq <= min_tq) return;
  *Tq *= *Hq / Hkv;
  *Hq = Hkv;
}

AttnShape make_shape(int B, int Hq, int Hkv, int Tq, int Tkv, int causal, int window,
                     float scale) {
  AttnShape s;
  s.B = B; s.Hq = Hq; s.Hkv = Hkv; s.Tq = Tq; s.Tkv = Tkv;
  s.causal = causal; s.window = window;
  s.scale_log2 = scale * kLog2e;
  return s;
}

}  // namespace

bool encode_tile_map(CUtensorMap* map, const void* base, bool bf16, int D, int T, int BH,
                     int box_rows) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(D) * 2 * static_cast<cuuint64_t>(T)};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                              3, const_cast<void*>(base), dims, strides, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_sm_count() {
  static std::atomic<int> cached[64] = {};  // callers on several host threads share it
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace fa

using namespace fa;

namespace fa_selftest {

// Two warps, two mbarriers that never complete (count 2, one arrival). Warp 0
// waits with the given limit and gives up; warp 1 waits with four times that
// limit and leaves through the abort flag warp 0 raised.
__global__ void fa_selftest_wait_kernel(uint32_t* status, uint64_t cycles) {
  __shared__ __align__(8) uint64_t never[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::mbar_init(fa::smem_u32(&never[0]), 2);
    fa::mbar_init(fa::smem_u32(&never[1]), 2);
    fa::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) fa::mbar_arrive(fa::smem_u32(&never[warp]));
  __syncwarp();
  fa::mbar_wait(fa::smem_u32(&never[warp]), 0, warp == 0 ? cycles : 4 * cycles, &abort_flag, status);
  __syncthreads();
}

}  // namespace fa_selftest

extern "C" {

fa_status fa_selftest_wait_timeout(unsigned int timeout_ms, cudaStream_t stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return FA_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  if (!status_ptr(&status)) return FA_ERR_LAUNCH;
  const uint64_t cycles = static_cast<uint64_t>(timeout_ms) * 2200000ull;
  fa_selftest::fa_selftest_wait_kernel<<<1, 64, 0, stream>>>(status, cycles);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_set_wait_limit_cycles(unsigned long long cycles) {
  g_wait_override.store(static_cast<uint64_t>(cycles), std::memory_order_relaxed);
  return FA_OK;
}

int fa_abi_version(void) { return 101; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED_HEAD_DIM: return "unsupported head dim (64, 96, 128, 256)";
    case FA_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype (fp16, bf16)";
    case FA_ERR_MISALIGNED: return "buffer not 16-byte aligned";
    case FA_ERR_LAUNCH: return "CUDA launch or driver call failed";
    case FA_ERR_TIMEOUT: return "a bounded device wait gave up";
  }
  return "unknown status";
}

size_t fa_bwd_workspace_size(int B, int Hq, int Tq) {
  if (B < 1 || Hq < 1 || Tq < 1) return 0;
  const size_t bytes = static_cast<size_t>(B) * Hq * Tq * sizeof(float);
  return (bytes + 255) / 256 * 256;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int Tq, int Tkv, int D, float scale, int causal, int window,
                 fa_dtype dt, cudaStream_t stream) {
  fa_status st = check_common(B, Hq, Hkv, Tq, Tkv, D, scale, causal, window, dt);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  const size_t nq = static_cast<size_t>(B) * Hq * Tq * D * 2;
  const size_t nkv = static_cast<size_t>(B) * Hkv * Tkv * D * 2;
  const size_t nl = static_cast<size_t>(B) * Hq * Tq * 4;
  if (overlap(o, nq, q, nq) || overlap(o, nq, k, nkv) || overlap(o, nq, v, nkv) ||
      overlap(lse, nl, q, nq) || overlap(lse, nl, k, nkv) || overlap(lse, nl, v, nkv) ||
      overlap(lse, nl, o, nq))
    return FA_ERR_INVALID_ARG;
  FwdLaunch a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  int hq = Hq, tq = Tq;  // short query blocks keep the split-key kernel
  fold_group_rows(causal, window, Hkv, kDecodeMaxTq, &hq, &tq);
  a.s = make_shape(B, hq, Hkv, tq, Tkv, causal, window, scale);
  a.bf16 = dt == FA_BF16;
  if (!status_ptr(&a.wc.status)) return FA_ERR_LAUNCH;
  set_waits(&a.wc);
  a.stream = stream;
  cudaError_t e;
  switch (D) {
    case 64: e = launch_fwd_d64(a); break;
    case 96: e = launch_fwd_d96(a); break;
    case 128: e = launch_fwd_d128(a); break;
    default: e = launch_fwd_d256(a); break;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // extern "C"

namespace {

// Shared path of fa_bwd and its three phase calls. Pointers a phase does not
// read or write may be null; everything it does use is checked.
fa_status bwd_common(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                     int Tq, int Tkv, int D, float scale, int causal, int window, fa_dtype dt,
                     void* dvec, size_t dvec_bytes, cudaStream_t stream, int phases) {
  fa_status st = check_common(B, Hq, Hkv, Tq, Tkv, D, scale, causal, window, dt);
  if (st != FA_OK) return st;
  const bool pre = phases & kPhaseDvec, dkv = phases & kPhaseDkv, dqp = phases & kPhaseDq;
  const bool need_qkv = dkv || dqp;
  if (!dO || !dvec) return FA_ERR_INVALID_ARG;
  if (pre && !o) return FA_ERR_INVALID_ARG;
  if (need_qkv && (!q || !k || !v || !lse)) return FA_ERR_INVALID_ARG;
  if (dkv && (!dk || !dv)) return FA_ERR_INVALID_ARG;
  if (dqp && !dq) return FA_ERR_INVALID_ARG;
  if (dvec_bytes < fa_bwd_workspace_size(B, Hq, Tq)) return FA_ERR_INVALID_ARG;
  const void* all[10] = {q, k, v, o, dO, lse, dq, dk, dv, dvec};
  for (const void* p : all)
    if (p && !aligned16(p)) return FA_ERR_MISALIGNED;
  const size_t nq = static_cast<size_t>(B) * Hq * Tq * D * 2;
  const size_t nkv = static_cast<size_t>(B) * Hkv * Tkv * D * 2;
  const size_t nl = static_cast<size_t>(B) * Hq * Tq * 4;
  // outputs of the requested phases (the D-vector is an output of pass 1 and
  // an input of passes 2-3)
  const void* ins[6] = {q, k, v, o, dO, lse};
  const size_t in_n[6] = {nq, nkv, nkv, nq, nq, nl};
  const void* outs[4] = {dqp ? dq : nullptr, dkv ? dk : nullptr, dkv ? dv : nullptr, dvec};
  const size_t out_n[4] = {nq, nkv, nkv, dvec_bytes};
  for (int i = 0; i < 4; ++i) {
    if (!outs[i]) continue;
    for (int j = 0; j < 6; ++j)
      if (ins[j] && overlap(outs[i], out_n[i], ins[j], in_n[j])) return FA_ERR_INVALID_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (outs[j] && overlap(outs[i], out_n[i], outs[j], out_n[j])) return FA_ERR_INVALID_ARG;
  }
  BwdLaunch a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.dout = dO; a.lse = lse;
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.dvec = static_cast<float*>(dvec);
  a.scale = scale;
  int hq = Hq, tq = Tq;
  fold_group_rows(causal, window, Hkv, 0, &hq, &tq);
  a.s = make_shape(B, hq, Hkv, tq, Tkv, causal, window, scale);
  a.s_rows = make_shape(B, Hq, Hkv, Tq, Tkv, causal, window, scale);
  a.bf16 = dt == FA_BF16;
  if (!status_ptr(&a.wc.status)) return FA_ERR_LAUNCH;
  set_waits(&a.wc);
  a.stream = stream;
  cudaError_t e;
  switch (D) {
    case 64: e = launch_bwd_d64(a, phases); break;
    case 96: e = launch_bwd_d96(a, phases); break;
    case 128: e = launch_bwd_d128(a, phases); break;
    default: e = launch_bwd_d256(a, phases); break;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Tq,
                 int Tkv, int D, float scale, int causal, int window, fa_dtype dt,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !workspace) {
    // keep the shape errors first, as for every entry point
    fa_status st = check_common(B, Hq, Hkv, Tq, Tkv, D, scale, causal, window, dt);
    return st != FA_OK ? st : FA_ERR_INVALID_ARG;
  }
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Tq, Tkv, D, scale, causal,
                    window, dt, workspace, workspace_bytes, stream, kPhaseAll);
}

fa_status fa_bwd_preprocess(const void* o, const void* dO, float* dvec, int B, int Hq, int Tq,
                            int D, fa_dtype dt, cudaStream_t stream) {
  // the D-vector does not depend on the mask, scale or KV shape
  return bwd_common(nullptr, nullptr, nullptr, o, dO, nullptr, nullptr, nullptr, nullptr, B, Hq,
                    Hq, Tq, 1, D, 1.f, 0, 0, dt, dvec, fa_bwd_workspace_size(B, Hq, Tq), stream,
                    kPhaseDvec);
}

fa_status fa_bwd_dkv(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* dvec, void* dk, void* dv, int B, int Hq,
                     int Hkv, int Tq, int Tkv, int D, float scale, int causal, int window,
                     fa_dtype dt, cudaStream_t stream) {
  return bwd_common(q, k, v, nullptr, dO, lse, nullptr, dk, dv, B, Hq, Hkv, Tq, Tkv, D, scale,
                    causal, window, dt, const_cast<float*>(dvec),
                    fa_bwd_workspace_size(B, Hq, Tq), stream, kPhaseDkv);
}

fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO,
                    const float* lse, const float* dvec, void* dq, int B, int Hq, int Hkv,
                    int Tq, int Tkv, int D, float scale, int causal, int window, fa_dtype dt,
                    cudaStream_t stream) {
  return bwd_common(q, k, v, nullptr, dO, lse, dq, nullptr, nullptr, B, Hq, Hkv, Tq, Tkv, D,
                    scale, causal, window, dt, const_cast<float*>(dvec),
                    fa_bwd_workspace_size(B, Hq, Tq), stream, kPhaseDq);
}

fa_status fa_device_status(unsigned int* bits, int clear, cudaStream_t stream) {
  if (!bits) return FA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_LAUNCH;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v)) != cudaSuccess) return FA_ERR_LAUNCH;
  if (clear && v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  *bits = v;
  return v == 0 ? FA_OK : FA_ERR_TIMEOUT;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory at all, not even the small D-vector workspace fa_bwd asks for — for
// example a plug-in running inside a host program that owns every device
// allocation, or a loop that must not call the allocator (which may
// synchronise the device) once it is running. The D-vector lives instead in
// the fixed array below, which every device that loads this library keeps
// until the process exits.
namespace {

// Largest B * Hq * Tq the array holds: 2^20 fp32 values (4 MiB).
constexpr size_t kNoallocMaxRows = size_t(1) << 20;

// Device address of the array, looked up once per device with that device
// current, and kept together with the id of the CUDA context it belongs to.
// A device reset (cudaDeviceReset) destroys that context and with it the
// address; the next call then runs in a new context with another id and looks
// the address up again instead of launching against freed memory.
struct NoallocSlot {
  unsigned long long ctx_id;
  float* ptr;
};
std::mutex g_noalloc_mutex;
NoallocSlot g_noalloc_slot[64] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void load_ctx_calls() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
          cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

// Id of the context current on this thread (0 when none is current yet).
bool current_ctx_id(unsigned long long* id) {
  *id = 0;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
  if (ctx == nullptr) return true;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

static __device__ __align__(256) float g_noalloc_scratch[kNoallocMaxRows];

namespace {

fa_status noalloc_scratch(float** out) {
  std::call_once(g_ctx_once, load_ctx_calls);
  if (!g_ctx_current || !g_ctx_id) return FA_ERR_LAUNCH;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  unsigned long long id = 0;
  if (!current_ctx_id(&id)) return FA_ERR_LAUNCH;
  NoallocSlot& slot = g_noalloc_slot[dev];
  if (slot.ptr == nullptr || id == 0 || slot.ctx_id != id) {
    // set-up on this device (and context): the runtime creates the context
    // if none is current yet
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_LAUNCH;
    if (!current_ctx_id(&id) || id == 0) return FA_ERR_LAUNCH;
    slot.ptr = static_cast<float*>(p);
    slot.ctx_id = id;
  }
  *out = slot.ptr;
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_noalloc_max_rows(void) { return kNoallocMaxRows; }

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                         int Hq, int Hkv, int Tq, int Tkv, int D, float scale, int causal,
                         int window, fa_dtype dt, cudaStream_t stream) {
  fa_status st = check_common(B, Hq, Hkv, Tq, Tkv, D, scale, causal, window, dt);
  if (st != FA_OK) return st;
  if (static_cast<size_t>(B) * Hq * Tq > kNoallocMaxRows) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  float* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != FA_OK) return st;
  // The D-vector is fully rewritten by the first launch of every call, so
  // nothing in the array has to start at zero.
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Tq, Tkv, D, scale, causal,
                    window, dt, scratch, kNoallocMaxRows * sizeof(float), stream, kPhaseAll);
}

}  // extern "C"
