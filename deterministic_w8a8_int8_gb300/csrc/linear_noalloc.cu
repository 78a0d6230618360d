// linear_noalloc.cu -- prism_w8a8_linear_noalloc: the W8A8 linear for callers
// that cannot hand the library a workspace.
//
// prism_w8a8_linear needs caller-provided scratch memory whenever it splits
// K (an int32 accumulator tile plus arrival counters).  Some callers cannot
// obtain that memory: a plugin host that only passes its own input and output
// buffers, a latency-critical loop in which cudaMalloc (which may synchronise
// the whole device) is not acceptable, or a process whose device memory budget
// is fixed before it starts.  This entry point serves them: its scratch is a
// fixed array compiled into the library, so it allocates nothing.
//
// Costs and rules of that choice:
//   - The array (PRISM_NOALLOC_SCRATCH_BYTES) is reserved on every GPU that
//     loads the library, for the life of the process.
//   - Shapes whose split-K scratch would not fit are rejected with
//     PRISM_ERR_UNSUPPORTED; nothing is enqueued.
//   - All calls on a device share the one array.  Each call clears the part
//     it uses (cudaMemsetAsync on the call's stream) before its kernel runs,
//     so stale contents from an earlier call never leak into a result; but
//     two calls whose work overlaps on the GPU (different streams, or
//     different host threads without ordering) race on the array and may
//     produce wrong results.  Order such calls on one stream.
//   - The device address of the array is looked up by the first call made
//     in each CUDA context (cudaGetSymbolAddress, with that context's device
//     current) and cached under the context's unique id.  Make that first
//     call before any stream capture begins.  A context torn down and made
//     again (cudaDeviceReset, primary-context release) has a new id, so the
//     next call looks the address up again instead of using a stale one.
//   - The stream must belong to the current device; a stream of another
//     device is refused (the array is per device).
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace prism {
namespace {

// The fixed scratch region.  In host code the name is only a stand-in for
// the symbol; the kernel receives the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PRISM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
// per device ordinal: the context the cached address belongs to, and the address
unsigned long long g_scratch_ctx[kMaxDevices] = {};
void* g_scratch_ptr[kMaxDevices] = {};

// Unique id of the calling thread's current context (driver entry points
// fetched once through the runtime, as for the tensor-map encoder).
cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) {
    // no context yet on this thread: the runtime makes the current device's
    // primary context current (a caller's own current context is never replaced)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of g_noalloc_scratch in the current context (looked up once
// per context, with the context's device current).
cudaError_t scratch_for_current_device(void** out) {
  unsigned long long ctx = 0;
  cudaError_t e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

// The stream belongs to the current device (NULL: the legacy default stream
// of the current device).
cudaError_t stream_on_current_device(cudaStream_t stream, bool* ok) {
  int dev = 0, sdev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaStreamGetDevice(stream, &sdev);
  if (e != cudaSuccess) return e;
  *ok = sdev == dev;
  return cudaSuccess;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace prism

extern "C" int prism_w8a8_linear_noalloc(const int8_t* q, int64_t ldq, const float* a_scale, const int8_t* w,
                                         int64_t ldw, const float* w_scale, const void* residual_bf16,
                                         int64_t ldr, void* out_bf16, int64_t ldo, int32_t* acc_out,
                                         int64_t M, int64_t N, int64_t K, int split_k, void* cuda_stream) {
  using prism::aligned_to;
  if (M < 0 || N < 0 || K <= 0 || split_k < 0) return PRISM_ERR_INVALID_ARG;
  if (split_k > PRISM_MAX_SPLIT_K) return PRISM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return PRISM_OK;
  if (q == nullptr || a_scale == nullptr || w == nullptr || w_scale == nullptr || out_bf16 == nullptr)
    return PRISM_ERR_INVALID_ARG;
  if (ldq < K || ldw < K || ldo < N || (residual_bf16 != nullptr && ldr < N)) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
  if (ldq % 16 != 0 || ldw % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned_to(q, 16) || !aligned_to(w, 16) || !aligned_to(out_bf16, 2) || !aligned_to(a_scale, 4) ||
      !aligned_to(w_scale, 4))
    return PRISM_ERR_ALIGNMENT;
  if (residual_bf16 != nullptr && !aligned_to(residual_bf16, 2)) return PRISM_ERR_ALIGNMENT;
  if (acc_out != nullptr && !aligned_to(acc_out, 4)) return PRISM_ERR_ALIGNMENT;
  if (M > 65535LL * 128) return PRISM_ERR_UNSUPPORTED;

  // bytes of the scratch array that must be zero for this call (the automatic
  // schedule falls back to whole tiles when its partial sums do not fit)
  const size_t zero = prism::linear_workspace_zero_bytes(M, N, K, split_k, PRISM_NOALLOC_SCRATCH_BYTES);
  if (zero == SIZE_MAX) return PRISM_ERR_UNSUPPORTED;

  prism::LinearArgs a{};
  a.q = q;
  a.ldq = ldq;
  a.a_scale = a_scale;
  a.w = w;
  a.ldw = ldw;
  a.w_scale = w_scale;
  a.residual = static_cast<const uint16_t*>(residual_bf16);
  a.ldr = ldr;
  a.out = static_cast<uint16_t*>(out_bf16);
  a.ldo = ldo;
  a.acc_out = acc_out;
  a.M = M;
  a.N = N;
  a.K = K;
  a.split = split_k;
  a.no_pdl = 1;  // the scratch clear below must complete before the kernel starts
  a.pair_io = aligned_to(out_bf16, 4) && ldo % 2 == 0 &&
              (residual_bf16 == nullptr || (aligned_to(residual_bf16, 4) && ldr % 2 == 0));
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  bool same_device = false;
  const int st0 = prism::record_cuda(prism::stream_on_current_device(stream, &same_device));
  if (st0 != PRISM_OK) return st0;
  if (!same_device) return PRISM_ERR_INVALID_ARG;
  if (zero > 0) {
    void* scratch = nullptr;
    const int st = prism::record_cuda(prism::scratch_for_current_device(&scratch));
    if (st != PRISM_OK) return st;
    const int st2 = prism::record_cuda(cudaMemsetAsync(scratch, 0, zero, stream));
    if (st2 != PRISM_OK) return st2;
    a.ws = scratch;
    a.ws_bytes = PRISM_NOALLOC_SCRATCH_BYTES;
  }
  return prism::record_cuda(prism::launch_linear(a, stream));
}
