// common.cuh -- device helpers shared by the libprism kernels (sm_103a).
//
// Every floating-point step that decides a stored value is written with an
// explicit round-to-nearest-even intrinsic (__fmul_rn, __fadd_rn, __fdiv_rn,
// __int2float_rn, __float2int_rn) so that the compiler can neither contract
// it into a fused multiply-add nor reorder it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <algorithm>
#include <utility>

#include "prism.h"

namespace prism {

// ----------------------------------------------------------------- bf16 ---
__device__ __forceinline__ float bf16_lo(uint32_t pair) {
  return __uint_as_float(pair << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t pair) {
  return __uint_as_float(pair & 0xffff0000u);
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
// binary32 -> bf16, round to nearest even (finite values; NaN -> quiet NaN).
__device__ __forceinline__ uint32_t float_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

// The epilogue of the W8A8 linear: ((float(acc) * a) * w) [+ r], each step
// one binary32 RN operation, then bf16 round-to-nearest-even.
__device__ __forceinline__ uint32_t epilogue_bf16(int32_t acc, float a, float w) {
  float t = __int2float_rn(acc);
  t = __fmul_rn(t, a);
  t = __fmul_rn(t, w);
  return float_to_bf16_rne(t);
}
__device__ __forceinline__ uint32_t epilogue_bf16_res(int32_t acc, float a, float w, float r) {
  float t = __int2float_rn(acc);
  t = __fmul_rn(t, a);
  t = __fmul_rn(t, w);
  t = __fadd_rn(t, r);
  return float_to_bf16_rne(t);
}

// ------------------------------------------------------ cp.async / ldmatrix
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte asynchronous copy global -> shared; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x32 s8, row) * B(32x8 s8, col) + C, exact int32.
__device__ __forceinline__ void mma_s8_16832(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Streaming 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Raise a kernel's dynamic shared-memory limit once per device (the attribute
// is per device context).  Thread-safe; idempotent.
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

// Remember a failed CUDA call for prism_last_cuda_error; map to a status.
int record_cuda(cudaError_t e);

}  // namespace prism

// Programmatic dependent launch: every library kernel is launched so that it
// may start while the previous kernel of its stream is still finishing.  It
// lets its own dependents launch at once (pdl_trigger: the runtime starts a
// dependent grid only when every CTA of this one has started and signalled,
// or exited, so a multi-wave grid cannot be starved), and waits for its
// predecessor to complete, with its memory visible, before touching any data
// (pdl_wait).  Without a predecessor kernel the wait returns at once.
namespace prism {
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Kernel, typename... Args>
cudaError_t launch_kernel(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                          Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
}  // namespace prism

// Internal launchers (one per kernel family), defined in their .cu files.
namespace prism {
// One quantiser call.  rows: null, or output row m quantises x row rows[m]
// of M_x (err gets PRISM_DEV_ERR_ROW_RANGE for an index outside [0, M_x);
// may be null).  amax_out: write only the row maxima.  amax_in: quantise
// with these row maxima.  At most one of rows, amax_out, amax_in.
struct QuantCall {
  const void* x;
  int64_t ldx;
  const float* inv_s;
  int64_t M, K;
  int8_t* q;
  int64_t ldq;
  float* a_scale;
  const int32_t* rows;
  int64_t M_x;
  uint32_t* err;
  float* amax_out;
  const float* amax_in;
  uint16_t* qh;     // non-null: the codes as binary16 values, row stride ldqh (plain mode only; q unused)
  int64_t ldqh;
};
cudaError_t launch_quant(const QuantCall& c, cudaStream_t stream);
cudaError_t launch_quant_act(const void* x, int64_t ldx, const float* inv_s, int64_t M, int64_t K, int8_t* q,
                             int64_t ldq, float* a_scale, const int32_t* rows, int64_t M_x, uint32_t* err,
                             cudaStream_t stream);

struct LinearArgs {
  const int8_t* q;
  int64_t ldq;
  const float* a_scale;
  const int8_t* w;
  int64_t ldw;
  const float* w_scale;
  const uint16_t* residual;
  int64_t ldr;
  uint16_t* out;
  int64_t ldo;
  int32_t* acc_out;
  int64_t M, N, K;
  int split;            // 0: automatic schedule; >= 1: explicit split-K
  int pair_io;          // 1: out/residual rows allow 4-byte bf16 pairs
  int no_pdl;           // 1: launch without overlapping the stream's previous work
  void* ws;             // caller's workspace (256-byte aligned) or null
  size_t ws_bytes;      // its size
  int32_t* ws_acc;      // split-K > 1: [M, N] int32, zero between calls (set by the launcher)
  uint32_t* ws_count;   // split-K > 1: [tiles] arrival counters, zero between calls
  const int32_t* res_rows;  // null, or the residual row of output row m is res_rows[m] ...
  int64_t M_res;            // ... of the residual's M_res rows
  uint32_t* err;            // PRISM_DEV_ERR_* bits (row index out of range), or null
  int acc_only;             // 1: write only acc_out (dense [M, N] int32); no scales, out, residual
};

// The residual row of output row m: row m itself, or row res_rows[m] (the
// last layer restricted to answer positions).  Null for an index outside
// [0, M_res), after setting PRISM_DEV_ERR_ROW_RANGE: that row's outputs
// become NaN and nothing outside the residual is read.
__device__ __forceinline__ const uint16_t* residual_row(const LinearArgs& a, int64_t m) {
  if (a.res_rows == nullptr) return a.residual + m * a.ldr;
  const int64_t r = __ldg(a.res_rows + m);
  if (r < 0 || r >= a.M_res) {
    if (a.err != nullptr) atomicOr(a.err, PRISM_DEV_ERR_ROW_RANGE);
    return nullptr;
  }
  return a.residual + r * a.ldr;
}
constexpr uint32_t kBf16NaN = 0x7fc0u;
// Workspace bytes a call needs (split 0 = the automatic schedule).
size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int split);
// Leading bytes of the workspace that must be zero when a call starts, for a
// workspace of cap bytes (SIZE_MAX: the call cannot run within cap).
size_t linear_workspace_zero_bytes(int64_t M, int64_t N, int64_t K, int split, size_t cap);
// Dispatch between the contraction kernels (linear_tc.cu): by token rows the
// dp4a weight stream, the mma.sync weight stream or the tcgen05 kernel;
// PRISM_LINEAR_PATH forces one (diagnostics).  linear_w4_packed: whether a
// W4A8 call streams its packed weights through the dp4a kernel.
int linear_kernel_kind(int64_t M, int64_t N, int64_t K);
bool linear_w4_packed(int64_t M);
int linear_auto_split(int64_t M, int64_t N, int64_t K);
cudaError_t launch_linear(const LinearArgs& a, cudaStream_t stream);
int mma_auto_split(int64_t M, int64_t N, int64_t K);
cudaError_t launch_linear_gemv(const LinearArgs& a, cudaStream_t stream);
// W4A8 on few rows: a.w points at packed 4-bit codes [N, K/2] (row stride
// a.ldw bytes), K % 32 == 0.
cudaError_t launch_linear_gemv_w4(const LinearArgs& a, cudaStream_t stream);
// Packed 4-bit codes [N, K/2] -> int8 [N, K] (K % 32 == 0, 16-byte rows).
cudaError_t launch_unpack_w4(const uint8_t* w4, int64_t ldw4, int64_t N, int64_t K, int8_t* w8, int64_t ldw8,
                             cudaStream_t stream);
cudaError_t launch_linear_mma(const LinearArgs& a, cudaStream_t stream);
// The mma.sync weight-streaming kernel for calls of up to 16 token rows
// (linear_stream.cu) and its workspace bytes.
cudaError_t launch_linear_stream(const LinearArgs& a, cudaStream_t stream);
size_t stream_workspace_bytes(int64_t M, int64_t N, int64_t K, int split);
// Streaming multiprocessors of the current device (one persistent CTA each).
int sm_count();
// Sticky device error bits raised by kernels (bounded waits that expired).
cudaError_t read_and_clear_kernel_error(uint32_t* out);
// Test mode of the tensor-core kernels' bounded waits: the pipeline waits'
// limit, and whether each CTA withholds its first chunk-complete signal.
cudaError_t set_tc_wait_expiry(unsigned long long limit_ns, int withhold);

// The linear on binary16 codes (linear_f16.cu): the same contraction and
// epilogue as launch_linear, with q and w given as binary16 values.
struct LinearF16Args {
  const uint16_t* qh;   // [M, K] activation codes, row stride ldq elements
  int64_t ldq;
  const float* a_scale;
  const uint16_t* wh;   // [N, K] weight codes, row stride ldw elements
  int64_t ldw;
  const float* w_scale;
  const uint16_t* residual;
  int64_t ldr;
  uint16_t* out;
  int64_t ldo;
  int32_t* acc_out;
  int64_t M, N, K;
  int split;            // 0: balanced schedule; >= 1: explicit split-K
  void* ws;             // workspace (256-byte aligned, zero between calls)
  size_t ws_bytes;
};
size_t linear_f16_workspace_bytes(int64_t M, int64_t N, int64_t K, int split);
cudaError_t launch_linear_f16(const LinearF16Args& a, cudaStream_t stream);
// int8 codes [rows, K] -> binary16 codes (exact), K % 16 == 0.
cudaError_t launch_codes_to_f16(const int8_t* w, int64_t ldw, int64_t rows, int64_t K, uint16_t* wh, int64_t ldwh,
                                cudaStream_t stream);
cudaError_t read_and_clear_f16_status(uint32_t* out);
cudaError_t set_f16_wait_expiry(unsigned long long limit_ns, int withhold);

// SmoothQuant requantisation of Q8_0 weights (requant.cu).
cudaError_t launch_smooth_requant(const int8_t* q, int64_t ldq, const uint16_t* d, int64_t ldd, const float* s,
                                  int64_t N, int64_t K, int8_t* w, int64_t ldw, float* w_scale,
                                  cudaStream_t stream);

// The epilogue alone on given int32 accumulators (epilogue.cu).
cudaError_t launch_epilogue(const int32_t* acc, int64_t ldc, const float* a_scale, const float* w_scale,
                            const uint16_t* residual, int64_t ldr, uint16_t* out, int64_t ldo, int64_t M, int64_t N,
                            cudaStream_t stream);

cudaError_t launch_readout(const void* h, int64_t ldh, const float* inv_s, const int8_t* W,
                           int64_t ldw, const float* lm_scale, int64_t V, int64_t K,
                           const int32_t* off, const int32_t* ids, int64_t P, int64_t T,
                           float* logits, float* probs, uint32_t* err, cudaStream_t stream);
// A vocabulary shard's logits (rows [v0, v0 + Vs) of the V-row head; -0.0 for
// other shards' candidates) and the softmax on combined logits (readout.cu).
cudaError_t launch_readout_logits(const void* h, int64_t ldh, const float* inv_s, const int8_t* W_shard,
                                  int64_t ldw, const float* lm_scale_shard, int64_t v0, int64_t Vs, int64_t V,
                                  int64_t K, const int32_t* off, const int32_t* ids, int64_t P, int64_t T,
                                  float* logits, uint32_t* err, cudaStream_t stream);
cudaError_t launch_candidate_softmax(const float* logits, const int32_t* off, int64_t P, int64_t T, float* probs,
                                     uint32_t* err, cudaStream_t stream);
}  // namespace prism
