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
//   - The device address of the array is looked up once per device, by the
//     first call made while that device is current (cudaGetSymbolAddress).
//     Make that first call before any stream capture begins.
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace prism {
namespace {

// The fixed scratch region.  In host code the name is only a stand-in for
// the symbol; the kernel receives the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PRISM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
