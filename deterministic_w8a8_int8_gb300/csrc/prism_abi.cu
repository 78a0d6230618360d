// prism_abi.cu -- the extern "C" boundary of libprism.so: host-side argument
// checks (returned as prism_status before anything is enqueued) and dispatch
// to the kernel launchers.  See include/prism.h for the contract.
#include <mutex>

#include "common.cuh"

namespace prism {

thread_local int g_last_cuda_error = 0;

int record_cuda(cudaError_t e) {
  if (e != cudaSuccess) g_last_cuda_error = static_cast<int>(e);
  return e == cudaSuccess ? PRISM_OK : PRISM_ERR_CUDA;
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_attr_mutex;
struct AttrEntry {
  const void* kernel;
  int bytes;
};
AttrEntry g_attr[kMaxDevices][8];
int g_attr_n[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  for (int i = 0; i < g_attr_n[dev]; ++i)
    if (g_attr[dev][i].kernel == kernel && g_attr[dev][i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (g_attr_n[dev] < 8) g_attr[dev][g_attr_n[dev]++] = AttrEntry{kernel, bytes};
  return cudaSuccess;
}

}  // namespace prism

using prism::aligned;

extern "C" {

int prism_version(void) { return 100; }

int prism_last_cuda_error(char* buf, size_t buf_bytes) {
  const int e = prism::g_last_cuda_error;
  prism::g_last_cuda_error = 0;
  if (buf != nullptr && buf_bytes > 0) {
    const char* msg = e == 0 ? "no error" : cudaGetErrorString(static_cast<cudaError_t>(e));
    size_t i = 0;
    for (; i + 1 < buf_bytes && msg[i] != '\0'; ++i) buf[i] = msg[i];
    buf[i] = '\0';
  }
  return e;
}

const char* prism_status_string(int status) {
  switch (status) {
    case PRISM_OK: return "ok";
    case PRISM_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or bad stride)";
    case PRISM_ERR_ALIGNMENT: return "misaligned pointer or stride, or K not a multiple of 16";
    case PRISM_ERR_UNSUPPORTED: return "unsupported size (K, split_k or candidate count beyond the limits)";
    case PRISM_ERR_WORKSPACE: return "workspace missing or too small";
    case PRISM_ERR_CUDA: return "CUDA launch or runtime error";
    default: return "unknown status";
  }
}

int prism_quant_act(const void* x_bf16, int64_t ldx, const float* inv_smooth, int64_t M, int64_t K,
                    int8_t* q, int64_t ldq, float* a_scale, void* cuda_stream) {
  if (M < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (M == 0) return PRISM_OK;
  if (x_bf16 == nullptr || q == nullptr || a_scale == nullptr) return PRISM_ERR_INVALID_ARG;
  if (ldx < K || ldq < K) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
  if (ldx % 8 != 0 || ldq % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned(x_bf16, 16) || !aligned(q, 16) || !aligned(a_scale, 4)) return PRISM_ERR_ALIGNMENT;
  if (inv_smooth != nullptr && !aligned(inv_smooth, 16)) return PRISM_ERR_ALIGNMENT;
  if (M > (static_cast<int64_t>(1) << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  return prism::record_cuda(prism::launch_quant_act(x_bf16, ldx, inv_smooth, M, K, q, ldq, a_scale, nullptr, M,
                                                     nullptr, static_cast<cudaStream_t>(cuda_stream)));
}

int prism_smooth_requant(const int8_t* q, int64_t ldq, const uint16_t* d_f16, int64_t ldd, const float* smooth,
                         int64_t N, int64_t K, int8_t* w, int64_t ldw, float* w_scale, void* cuda_stream) {
  if (N < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (N == 0) return PRISM_OK;
  if (q == nullptr || d_f16 == nullptr || w == nullptr || w_scale == nullptr) return PRISM_ERR_INVALID_ARG;
  if (K % 32 != 0) return PRISM_ERR_ALIGNMENT;
  if (ldq < K || ldw < K || ldd < K / 32) return PRISM_ERR_INVALID_ARG;
  if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
  if (ldq % 16 != 0 || ldw % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(d_f16, 2) || !aligned(w_scale, 4)) return PRISM_ERR_ALIGNMENT;
  if (smooth != nullptr && !aligned(smooth, 16)) return PRISM_ERR_ALIGNMENT;
  if (N > (static_cast<int64_t>(1) << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  // w == q (in place) is allowed only with one stride for both.
  if (static_cast<const void*>(w) == static_cast<const void*>(q) && ldw != ldq) return PRISM_ERR_INVALID_ARG;
  return prism::record_cuda(prism::launch_smooth_requant(q, ldq, d_f16, ldd, smooth, N, K, w, ldw, w_scale,
                                                          static_cast<cudaStream_t>(cuda_stream)));
}

static int linear_impl(const int8_t* q, int64_t ldq, const float* a_scale, const int8_t* w, int64_t ldw,
                       const float* w_scale, const void* residual_bf16, int64_t ldr, void* out_bf16,
                       int64_t ldo, int32_t* acc_out, int64_t M, int64_t N, int64_t K, int split_k,
                       void* workspace, size_t workspace_bytes, const int32_t* res_rows, int64_t M_res,
                       uint32_t* err, int acc_only, void* cuda_stream);

static size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

size_t prism_w4a8_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k) {
  if (M <= 0 || N <= 0 || K <= 0 || split_k < 0 || split_k > PRISM_MAX_SPLIT_K) return 0;
  if (prism::linear_w4_packed(M)) return 0;   // few rows: packed weights streamed directly
  return align256(static_cast<size_t>(N) * static_cast<size_t>(K)) + prism::linear_workspace_bytes(M, N, K, split_k);
}

int prism_unpack_w4(const uint8_t* w4, int64_t ldw4, int64_t N, int64_t K, int8_t* w, int64_t ldw, void* cuda_stream) {
  if (N < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (N == 0) return PRISM_OK;
  if (w4 == nullptr || w == nullptr) return PRISM_ERR_INVALID_ARG;
  if (K % 32 != 0) return PRISM_ERR_ALIGNMENT;
  if (ldw4 < K / 2 || ldw < K) return PRISM_ERR_INVALID_ARG;
  if (ldw4 % 16 != 0 || ldw % 16 != 0 || !aligned(w4, 16) || !aligned(w, 16)) return PRISM_ERR_ALIGNMENT;
  return prism::record_cuda(prism::launch_unpack_w4(w4, ldw4, N, K, w, ldw, static_cast<cudaStream_t>(cuda_stream)));
}

int prism_w4a8_linear(const int8_t* q, int64_t ldq, const float* a_scale, const uint8_t* w4, int64_t ldw4,
                      const float* w_scale, const void* residual_bf16, int64_t ldr, void* out_bf16, int64_t ldo,
                      int32_t* acc_out, int64_t M, int64_t N, int64_t K, int split_k, void* workspace,
                      size_t workspace_bytes, void* cuda_stream) {
  if (M < 0 || N < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (split_k < 0) return PRISM_ERR_INVALID_ARG;
  if (split_k > PRISM_MAX_SPLIT_K) return PRISM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return PRISM_OK;
  if (w4 == nullptr) return PRISM_ERR_INVALID_ARG;
  if (K % 32 != 0) return PRISM_ERR_ALIGNMENT;
  if (ldw4 < K / 2) return PRISM_ERR_INVALID_ARG;
  if (ldw4 % 16 != 0 || !aligned(w4, 16)) return PRISM_ERR_ALIGNMENT;
  const cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if (prism::linear_w4_packed(M)) {
    // few rows: the dp4a kernel streams the packed codes (the W8A8 call's
    // argument rules, with the packed row as the weight)
    if (q == nullptr || a_scale == nullptr || w_scale == nullptr || out_bf16 == nullptr) return PRISM_ERR_INVALID_ARG;
    if (ldq < K || ldo < N || (residual_bf16 != nullptr && ldr < N)) return PRISM_ERR_INVALID_ARG;
    if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
    if (ldq % 16 != 0 || !aligned(q, 16) || !aligned(out_bf16, 2) || !aligned(a_scale, 4) || !aligned(w_scale, 4))
      return PRISM_ERR_ALIGNMENT;
    if ((residual_bf16 != nullptr && !aligned(residual_bf16, 2)) || (acc_out != nullptr && !aligned(acc_out, 4)))
      return PRISM_ERR_ALIGNMENT;
    prism::LinearArgs a{};
    a.q = q;
    a.ldq = ldq;
    a.a_scale = a_scale;
    a.w = reinterpret_cast<const int8_t*>(w4);
    a.ldw = ldw4;
    a.w_scale = w_scale;
    a.residual = static_cast<const uint16_t*>(residual_bf16);
    a.ldr = ldr;
    a.out = static_cast<uint16_t*>(out_bf16);
    a.ldo = ldo;
    a.acc_out = acc_out;
    a.M = M;
    a.N = N;
    a.K = K;
    return prism::record_cuda(prism::launch_linear_gemv_w4(a, stream));
  }
  // more rows: unpack into the head of the workspace, then the W8A8 kernel
  // with the rest of it
  const size_t head = align256(static_cast<size_t>(N) * static_cast<size_t>(K));
  if (workspace == nullptr || workspace_bytes < head) return PRISM_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PRISM_ERR_ALIGNMENT;
  int8_t* w8 = static_cast<int8_t*>(workspace);
  const int st = prism::record_cuda(prism::launch_unpack_w4(w4, ldw4, N, K, w8, K, stream));
  if (st != PRISM_OK) return st;
  void* rest = workspace_bytes > head ? static_cast<char*>(workspace) + head : nullptr;
  return linear_impl(q, ldq, a_scale, w8, K, w_scale, residual_bf16, ldr, out_bf16, ldo, acc_out, M, N, K, split_k,
                     rest, workspace_bytes - head, nullptr, 0, nullptr, 0, cuda_stream);
}

int prism_w8a8_gemm_s32(const int8_t* q, int64_t ldq, const int8_t* w, int64_t ldw, int32_t* acc, int64_t M,
                        int64_t N, int64_t K, int split_k, void* workspace, size_t workspace_bytes,
                        void* cuda_stream) {
  return linear_impl(q, ldq, nullptr, w, ldw, nullptr, nullptr, 0, nullptr, 0, acc, M, N, K, split_k, workspace,
                     workspace_bytes, nullptr, 0, nullptr, 1, cuda_stream);
}

int prism_w8a8_epilogue(const int32_t* acc, int64_t ldc, const float* a_scale, const float* w_scale,
                        const void* residual_bf16, int64_t ldr, void* out_bf16, int64_t ldo, int64_t M, int64_t N,
                        void* cuda_stream) {
  if (M < 0 || N < 0) return PRISM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return PRISM_OK;
  if (acc == nullptr || a_scale == nullptr || w_scale == nullptr || out_bf16 == nullptr) return PRISM_ERR_INVALID_ARG;
  if (ldc < N || ldo < N || (residual_bf16 != nullptr && ldr < N)) return PRISM_ERR_INVALID_ARG;
  if (!aligned(acc, 4) || !aligned(a_scale, 4) || !aligned(w_scale, 4) || !aligned(out_bf16, 2) ||
      (residual_bf16 != nullptr && !aligned(residual_bf16, 2)))
    return PRISM_ERR_ALIGNMENT;
  return prism::record_cuda(prism::launch_epilogue(acc, ldc, a_scale, w_scale,
                                                   static_cast<const uint16_t*>(residual_bf16), ldr,
                                                   static_cast<uint16_t*>(out_bf16), ldo, M, N,
                                                   static_cast<cudaStream_t>(cuda_stream)));
}

static int check_quant_args(const void* x_bf16, int64_t ldx, const float* inv_smooth, int64_t M, int64_t K) {
  if (M < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (M > 0 && x_bf16 == nullptr) return PRISM_ERR_INVALID_ARG;
  if (ldx < K) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
  if (ldx % 8 != 0 || !aligned(x_bf16, 16)) return PRISM_ERR_ALIGNMENT;
  if (inv_smooth != nullptr && !aligned(inv_smooth, 16)) return PRISM_ERR_ALIGNMENT;
  if (M > (static_cast<int64_t>(1) << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  return PRISM_OK;
}

int prism_act_amax(const void* x_bf16, int64_t ldx, const float* inv_smooth, int64_t M, int64_t K, float* amax,
                   void* cuda_stream) {
  const int st = check_quant_args(x_bf16, ldx, inv_smooth, M, K);
  if (st != PRISM_OK || M == 0) return st;
  if (amax == nullptr) return PRISM_ERR_INVALID_ARG;
  if (!aligned(amax, 4)) return PRISM_ERR_ALIGNMENT;
  prism::QuantCall c{};
  c.x = x_bf16;
  c.ldx = ldx;
  c.inv_s = inv_smooth;
  c.M = M;
  c.K = K;
  c.amax_out = amax;
  return prism::record_cuda(prism::launch_quant(c, static_cast<cudaStream_t>(cuda_stream)));
}

int prism_quant_act_amax(const void* x_bf16, int64_t ldx, const float* inv_smooth, const float* amax, int64_t M,
                         int64_t K, int8_t* q, int64_t ldq, float* a_scale, void* cuda_stream) {
  const int st = check_quant_args(x_bf16, ldx, inv_smooth, M, K);
  if (st != PRISM_OK || M == 0) return st;
  if (amax == nullptr || q == nullptr || a_scale == nullptr) return PRISM_ERR_INVALID_ARG;
  if (ldq < K) return PRISM_ERR_INVALID_ARG;
  if (ldq % 16 != 0 || !aligned(q, 16) || !aligned(a_scale, 4) || !aligned(amax, 4)) return PRISM_ERR_ALIGNMENT;
  prism::QuantCall c{};
  c.x = x_bf16;
  c.ldx = ldx;
  c.inv_s = inv_smooth;
  c.M = M;
  c.K = K;
  c.q = q;
  c.ldq = ldq;
  c.a_scale = a_scale;
  c.amax_in = amax;
  return prism::record_cuda(prism::launch_quant(c, static_cast<cudaStream_t>(cuda_stream)));
}

int prism_quant_act_rows(const void* x_bf16, int64_t ldx, int64_t M_x, const int32_t* rows, int64_t n_rows,
                         const float* inv_smooth, int64_t K, int8_t* q, int64_t ldq, float* a_scale,
                         int32_t* dev_error_word, void* cuda_stream) {
  if (n_rows < 0 || M_x < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (n_rows == 0) return PRISM_OK;
  if (x_bf16 == nullptr || rows == nullptr || q == nullptr || a_scale == nullptr || M_x == 0)
    return PRISM_ERR_INVALID_ARG;
  if (ldx < K || ldq < K) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
  if (ldx % 8 != 0 || ldq % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned(x_bf16, 16) || !aligned(q, 16) || !aligned(a_scale, 4) || !aligned(rows, 4)) return PRISM_ERR_ALIGNMENT;
  if (inv_smooth != nullptr && !aligned(inv_smooth, 16)) return PRISM_ERR_ALIGNMENT;
  if (dev_error_word != nullptr && !aligned(dev_error_word, 4)) return PRISM_ERR_ALIGNMENT;
  if (n_rows > (static_cast<int64_t>(1) << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  return prism::record_cuda(prism::launch_quant_act(x_bf16, ldx, inv_smooth, n_rows, K, q, ldq, a_scale, rows, M_x,
                                                     reinterpret_cast<uint32_t*>(dev_error_word),
                                                     static_cast<cudaStream_t>(cuda_stream)));
}

int prism_w8a8_kernel_kind(int64_t M, int64_t N, int64_t K) { return prism::linear_kernel_kind(M, N, K); }

int prism_device_status(uint32_t* flags) {
  if (flags == nullptr) return PRISM_ERR_INVALID_ARG;
  uint32_t a = 0, b = 0;
  int st = prism::record_cuda(prism::read_and_clear_kernel_error(&a));
  if (st == PRISM_OK) st = prism::record_cuda(prism::read_and_clear_f16_status(&b));
  *flags = a | b;
  return st;
}

int prism_debug_wait_expiry(uint64_t limit_ns) {
  const unsigned long long v = limit_ns == 0 ? 2000000000ull : static_cast<unsigned long long>(limit_ns);
  const int withhold = limit_ns != 0 ? 1 : 0;
  int st = prism::record_cuda(prism::set_tc_wait_expiry(v, withhold));
  if (st == PRISM_OK) st = prism::record_cuda(prism::set_f16_wait_expiry(v, withhold));
  return st;
}

int prism_w8a8_auto_split(int64_t M, int64_t N, int64_t K) { return prism::linear_auto_split(M, N, K); }

size_t prism_w8a8_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k) {
  if (M <= 0 || N <= 0 || K <= 0 || split_k < 0 || split_k > PRISM_MAX_SPLIT_K) return 0;
  return prism::linear_workspace_bytes(M, N, K, split_k);
}

// acc_only: only the dense int32 accumulators (acc_out) are produced; the
// scales, residual and output are then NULL and unused.
static int linear_impl(const int8_t* q, int64_t ldq, const float* a_scale, const int8_t* w, int64_t ldw,
                       const float* w_scale, const void* residual_bf16, int64_t ldr, void* out_bf16,
                       int64_t ldo, int32_t* acc_out, int64_t M, int64_t N, int64_t K, int split_k,
                       void* workspace, size_t workspace_bytes, const int32_t* res_rows, int64_t M_res,
                       uint32_t* err, int acc_only, void* cuda_stream) {
  if (M < 0 || N < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (split_k < 0) return PRISM_ERR_INVALID_ARG;
  if (split_k > PRISM_MAX_SPLIT_K) return PRISM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return PRISM_OK;
  if (q == nullptr || w == nullptr) return PRISM_ERR_INVALID_ARG;
  if (acc_only) {
    if (acc_out == nullptr) return PRISM_ERR_INVALID_ARG;
  } else {
    if (a_scale == nullptr || w_scale == nullptr || out_bf16 == nullptr) return PRISM_ERR_INVALID_ARG;
    if (ldo < N || (residual_bf16 != nullptr && ldr < N)) return PRISM_ERR_INVALID_ARG;
    if (!aligned(out_bf16, 2) || !aligned(a_scale, 4) || !aligned(w_scale, 4)) return PRISM_ERR_ALIGNMENT;
  }
  if (ldq < K || ldw < K) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
  if (ldq % 16 != 0 || ldw % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned(q, 16) || !aligned(w, 16)) return PRISM_ERR_ALIGNMENT;
  if (residual_bf16 != nullptr && !aligned(residual_bf16, 2)) return PRISM_ERR_ALIGNMENT;
  if (acc_out != nullptr && !aligned(acc_out, 4)) return PRISM_ERR_ALIGNMENT;
  if (M > 65535LL * 128 || N > (1LL << 31) * 64) return PRISM_ERR_UNSUPPORTED;

  const size_t need = prism::linear_workspace_bytes(M, N, K, split_k);
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
  a.res_rows = res_rows;
  a.M_res = M_res;
  a.err = err;
  a.acc_only = acc_only;
  a.pair_io = !acc_only && aligned(out_bf16, 4) && ldo % 2 == 0 &&
              (residual_bf16 == nullptr || (aligned(residual_bf16, 4) && ldr % 2 == 0));
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return PRISM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PRISM_ERR_ALIGNMENT;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
  }
  return prism::record_cuda(prism::launch_linear(a, static_cast<cudaStream_t>(cuda_stream)));
}

int prism_w8a8_linear(const int8_t* q, int64_t ldq, const float* a_scale, const int8_t* w, int64_t ldw,
                      const float* w_scale, const void* residual_bf16, int64_t ldr, void* out_bf16,
                      int64_t ldo, int32_t* acc_out, int64_t M, int64_t N, int64_t K, int split_k,
                      void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return linear_impl(q, ldq, a_scale, w, ldw, w_scale, residual_bf16, ldr, out_bf16, ldo, acc_out, M, N, K, split_k,
                     workspace, workspace_bytes, nullptr, 0, nullptr, 0, cuda_stream);
}

int prism_quant_act_f16(const void* x_bf16, int64_t ldx, const float* inv_smooth, int64_t M, int64_t K,
                        uint16_t* qh, int64_t ldqh, float* a_scale, void* cuda_stream) {
  if (M < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (M == 0) return PRISM_OK;
  if (x_bf16 == nullptr || qh == nullptr || a_scale == nullptr) return PRISM_ERR_INVALID_ARG;
  if (ldx < K || ldqh < K) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
  if (ldx % 8 != 0 || ldqh % 8 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned(x_bf16, 16) || !aligned(qh, 16) || !aligned(a_scale, 4)) return PRISM_ERR_ALIGNMENT;
  if (inv_smooth != nullptr && !aligned(inv_smooth, 16)) return PRISM_ERR_ALIGNMENT;
  if (M > (static_cast<int64_t>(1) << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  prism::QuantCall c{};
  c.x = x_bf16;
  c.ldx = ldx;
  c.inv_s = inv_smooth;
  c.M = M;
  c.K = K;
  c.a_scale = a_scale;
  c.M_x = M;
  c.qh = qh;
  c.ldqh = ldqh;
  return prism::record_cuda(prism::launch_quant(c, static_cast<cudaStream_t>(cuda_stream)));
}

int prism_codes_to_f16(const int8_t* w, int64_t ldw, int64_t rows, int64_t K, uint16_t* wh, int64_t ldwh,
                       void* cuda_stream) {
  if (rows < 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (rows == 0) return PRISM_OK;
  if (w == nullptr || wh == nullptr) return PRISM_ERR_INVALID_ARG;
  if (ldw < K || ldwh < K) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0 || ldw % 16 != 0 || ldwh % 8 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned(w, 16) || !aligned(wh, 16)) return PRISM_ERR_ALIGNMENT;
  if (K > PRISM_MAX_K || rows > (static_cast<int64_t>(1) << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  // the binary16 rows must not overlap the int8 rows they are made from
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(w), h0 = reinterpret_cast<uintptr_t>(wh);
  const uintptr_t w1 = w0 + static_cast<uintptr_t>((rows - 1) * ldw + K);
  const uintptr_t h1 = h0 + static_cast<uintptr_t>((rows - 1) * ldwh + K) * 2;
  if (w0 < h1 && h0 < w1) return PRISM_ERR_INVALID_ARG;
  return prism::record_cuda(prism::launch_codes_to_f16(w, ldw, rows, K, wh, ldwh,
                                                       static_cast<cudaStream_t>(cuda_stream)));
}

size_t prism_w8a8_f16_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k) {
  if (M <= 0 || N <= 0 || K <= 0 || split_k < 0 || split_k > PRISM_MAX_SPLIT_K) return 0;
  return prism::linear_f16_workspace_bytes(M, N, K, split_k);
}

int prism_w8a8_linear_f16(const uint16_t* qh, int64_t ldq, const float* a_scale, const uint16_t* wh, int64_t ldw,
                          const float* w_scale, const void* residual_bf16, int64_t ldr, void* out_bf16, int64_t ldo,
                          int32_t* acc_out, int64_t M, int64_t N, int64_t K, int split_k, void* workspace,
                          size_t workspace_bytes, void* cuda_stream) {
  if (M < 0 || N < 0 || K <= 0 || split_k < 0) return PRISM_ERR_INVALID_ARG;
  if (split_k > PRISM_MAX_SPLIT_K) return PRISM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return PRISM_OK;
  if (qh == nullptr || wh == nullptr || a_scale == nullptr || w_scale == nullptr || out_bf16 == nullptr)
    return PRISM_ERR_INVALID_ARG;
  if (ldq < K || ldw < K || ldo < N || (residual_bf16 != nullptr && ldr < N)) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (K > PRISM_MAX_K) return PRISM_ERR_UNSUPPORTED;
  if (ldq % 8 != 0 || ldw % 8 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned(qh, 16) || !aligned(wh, 16) || !aligned(out_bf16, 2) || !aligned(a_scale, 4) ||
      !aligned(w_scale, 4))
    return PRISM_ERR_ALIGNMENT;
  if (residual_bf16 != nullptr && !aligned(residual_bf16, 2)) return PRISM_ERR_ALIGNMENT;
  if (acc_out != nullptr && !aligned(acc_out, 4)) return PRISM_ERR_ALIGNMENT;
  // tile indices and grid dimensions stay within int32 and the launch limits
  if (((M + 127) / 128) * ((N + 127) / 128) > (1LL << 31) - 1 || (N + 255) / 256 > 65535)
    return PRISM_ERR_UNSUPPORTED;
  const size_t need = prism::linear_f16_workspace_bytes(M, N, K, split_k);
  prism::LinearF16Args a{};
  a.qh = qh;
  a.ldq = ldq;
  a.a_scale = a_scale;
  a.wh = wh;
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
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return PRISM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PRISM_ERR_ALIGNMENT;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
  }
  return prism::record_cuda(prism::launch_linear_f16(a, static_cast<cudaStream_t>(cuda_stream)));
}

int prism_w8a8_linear_rows(const int8_t* q, int64_t ldq, const float* a_scale, const int8_t* w, int64_t ldw,
                           const float* w_scale, const void* residual_bf16, int64_t ldr, int64_t M_res,
                           const int32_t* residual_rows, void* out_bf16, int64_t ldo, int32_t* acc_out,
                           int64_t M, int64_t N, int64_t K, int split_k, void* workspace,
                           size_t workspace_bytes, int32_t* dev_error_word, void* cuda_stream) {
  if (M < 0 || M_res < 0) return PRISM_ERR_INVALID_ARG;
  if (M > 0 && N > 0) {
    if (residual_bf16 == nullptr || residual_rows == nullptr || M_res == 0) return PRISM_ERR_INVALID_ARG;
    if (!aligned(residual_rows, 4) || (dev_error_word != nullptr && !aligned(dev_error_word, 4)))
      return PRISM_ERR_ALIGNMENT;
    // Output rows may be residual rows of other CTAs' tiles: no overlap.
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out_bf16), r0 = reinterpret_cast<uintptr_t>(residual_bf16);
    const uintptr_t o1 = o0 + static_cast<uintptr_t>((M - 1) * ldo + N) * 2;
    const uintptr_t r1 = r0 + static_cast<uintptr_t>((M_res - 1) * ldr + N) * 2;
    if (o0 < r1 && r0 < o1) return PRISM_ERR_INVALID_ARG;
  }
  return linear_impl(q, ldq, a_scale, w, ldw, w_scale, residual_bf16, ldr, out_bf16, ldo, acc_out, M, N, K, split_k,
                     workspace, workspace_bytes, residual_rows, M_res,
                     reinterpret_cast<uint32_t*>(dev_error_word), 0, cuda_stream);
}

int prism_candidate_readout(const void* hidden_bf16, int64_t ldh, const float* inv_smooth,
                            const int8_t* lm_head, int64_t ldw, const float* lm_scale, int64_t V,
                            int64_t K, const int32_t* cand_offsets, const int32_t* cand_ids, int64_t P,
                            int64_t T, float* logits, float* probs, int32_t* dev_error_word,
                            void* workspace, size_t workspace_bytes, void* cuda_stream) {
  (void)workspace;   // no scratch: prism_readout_workspace_bytes is 0 for every shape
  (void)workspace_bytes;
  if (P < 0 || T < 0 || V <= 0 || K <= 0) return PRISM_ERR_INVALID_ARG;
  if (P == 0) return T == 0 ? PRISM_OK : PRISM_ERR_INVALID_ARG;
  if (hidden_bf16 == nullptr || lm_head == nullptr || lm_scale == nullptr || cand_offsets == nullptr ||
      logits == nullptr || probs == nullptr)
    return PRISM_ERR_INVALID_ARG;
  if (T > 0 && cand_ids == nullptr) return PRISM_ERR_INVALID_ARG;
  if (ldh < K || ldw < K) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (P > (1LL << 31) - 1 || K > PRISM_MAX_READOUT_K || T > P * PRISM_MAX_CANDIDATES || V > (1LL << 31) - 1)
    return PRISM_ERR_UNSUPPORTED;
  if (ldh % 8 != 0 || ldw % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (!aligned(hidden_bf16, 16) || !aligned(lm_head, 16) || !aligned(lm_scale, 4) ||
      !aligned(cand_offsets, 4) || !aligned(cand_ids, 4) || !aligned(logits, 4) || !aligned(probs, 4))
    return PRISM_ERR_ALIGNMENT;
  if (inv_smooth != nullptr && !aligned(inv_smooth, 16)) return PRISM_ERR_ALIGNMENT;
  if (dev_error_word != nullptr && !aligned(dev_error_word, 4)) return PRISM_ERR_ALIGNMENT;
  if (P > (1LL << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  return prism::record_cuda(prism::launch_readout(hidden_bf16, ldh, inv_smooth, lm_head, ldw, lm_scale, V,
                                                   K, cand_offsets, cand_ids, P, T, logits, probs,
                                                   reinterpret_cast<uint32_t*>(dev_error_word),
                                                   static_cast<cudaStream_t>(cuda_stream)));
}

int prism_candidate_logits(const void* hidden_bf16, int64_t ldh, const float* inv_smooth,
                           const int8_t* lm_head_shard, int64_t ldw, const float* lm_scale_shard, int64_t v0,
                           int64_t V_shard, int64_t V, int64_t K, const int32_t* cand_offsets,
                           const int32_t* cand_ids, int64_t P, int64_t T, float* logits, int32_t* dev_error_word,
                           void* cuda_stream) {
  if (P < 0 || T < 0 || V <= 0 || K <= 0 || v0 < 0 || V_shard < 0 || v0 + V_shard > V)
    return PRISM_ERR_INVALID_ARG;
  if (P == 0) return T == 0 ? PRISM_OK : PRISM_ERR_INVALID_ARG;
  if (hidden_bf16 == nullptr || cand_offsets == nullptr || logits == nullptr) return PRISM_ERR_INVALID_ARG;
  if (V_shard > 0 && (lm_head_shard == nullptr || lm_scale_shard == nullptr)) return PRISM_ERR_INVALID_ARG;
  if (T > 0 && cand_ids == nullptr) return PRISM_ERR_INVALID_ARG;
  if (ldh < K || (V_shard > 0 && ldw < K)) return PRISM_ERR_INVALID_ARG;
  if (K % 16 != 0) return PRISM_ERR_ALIGNMENT;
  if (P > (1LL << 31) - 1 || K > PRISM_MAX_READOUT_K || T > P * PRISM_MAX_CANDIDATES || V > (1LL << 31) - 1)
    return PRISM_ERR_UNSUPPORTED;
  if (ldh % 8 != 0 || (V_shard > 0 && ldw % 16 != 0)) return PRISM_ERR_ALIGNMENT;
  if (!aligned(hidden_bf16, 16) || !aligned(lm_head_shard, 16) || !aligned(lm_scale_shard, 4) ||
      !aligned(cand_offsets, 4) || !aligned(cand_ids, 4) || !aligned(logits, 4))
    return PRISM_ERR_ALIGNMENT;
  if (inv_smooth != nullptr && !aligned(inv_smooth, 16)) return PRISM_ERR_ALIGNMENT;
  if (dev_error_word != nullptr && !aligned(dev_error_word, 4)) return PRISM_ERR_ALIGNMENT;
  if (P > (1LL << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  return prism::record_cuda(prism::launch_readout_logits(
      hidden_bf16, ldh, inv_smooth, lm_head_shard, ldw, lm_scale_shard, v0, V_shard, V, K, cand_offsets, cand_ids, P,
      T, logits, reinterpret_cast<uint32_t*>(dev_error_word), static_cast<cudaStream_t>(cuda_stream)));
}

int prism_candidate_softmax(const float* logits, const int32_t* cand_offsets, int64_t P, int64_t T, float* probs,
                            int32_t* dev_error_word, void* cuda_stream) {
  if (P < 0 || T < 0) return PRISM_ERR_INVALID_ARG;
  if (P == 0) return T == 0 ? PRISM_OK : PRISM_ERR_INVALID_ARG;
  if (cand_offsets == nullptr || probs == nullptr || (T > 0 && logits == nullptr)) return PRISM_ERR_INVALID_ARG;
  if (P > (1LL << 31) - 1 || T > P * PRISM_MAX_CANDIDATES) return PRISM_ERR_UNSUPPORTED;
  if (!aligned(logits, 4) || !aligned(cand_offsets, 4) || !aligned(probs, 4)) return PRISM_ERR_ALIGNMENT;
  if (dev_error_word != nullptr && !aligned(dev_error_word, 4)) return PRISM_ERR_ALIGNMENT;
  return prism::record_cuda(prism::launch_candidate_softmax(logits, cand_offsets, P, T, probs,
                                                            reinterpret_cast<uint32_t*>(dev_error_word),
                                                            static_cast<cudaStream_t>(cuda_stream)));
}

size_t prism_readout_workspace_bytes(int64_t P, int64_t T, int64_t K) {
  (void)P;
  (void)T;
  (void)K;
  return 0;
}

}  // extern "C"
