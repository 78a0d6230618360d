// epilogue.cu -- the fixed-order epilogue on given int32 accumulators
// (StartLux-Prism, "Bitwise consistency is not lossless quantization": with
// tensor parallelism the int32 partial sums are combined before scaling; this
// kernel is the scaling that follows the combine).
//
//   out[m, n] = bf16_rne(((float(acc[m, n]) * a_scale[m]) * w_scale[n]) [+ residual[m, n]])
//
// the same sequence of binary32 round-to-nearest operations as the linear
// kernels' epilogue (common.cuh), so a tensor-parallel layer gives the bits
// of the one-device layer.  HBM-bound: 4 bytes in, 2 out (plus 2 of
// residual) per element.  Each thread takes 8 consecutive channels of a row:
// two 16-byte accumulator loads, one 16-byte residual load and one 16-byte
// store when the layouts allow, element accesses otherwise.
#include "common.cuh"

namespace prism {
namespace {

constexpr int kThreads = 256;
constexpr int kCols = 8;

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    epilogue_kernel(const int32_t* __restrict__ acc, int64_t ldc, const float* __restrict__ a_scale,
                    const float* __restrict__ w_scale, const uint16_t* residual, int64_t ldr, uint16_t* out,
                    int64_t ldo, int64_t M, int64_t N) {
  pdl_trigger();
  pdl_wait();
  const int64_t chunks = (N + kCols - 1) / kCols;
  const int64_t total = M * chunks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t m = i / chunks, n0 = (i - m * chunks) * kCols;
    const float as = __ldg(a_scale + m);
    const int32_t* ar = acc + m * ldc + n0;
    if (kVec && n0 + kCols <= N) {
      const int4 c0 = __ldg(reinterpret_cast<const int4*>(ar));
      const int4 c1 = __ldg(reinterpret_cast<const int4*>(ar) + 1);
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w_scale + n0));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w_scale + n0) + 1);
      const int32_t v[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      uint32_t rw[4] = {0u, 0u, 0u, 0u};
      if (residual != nullptr) {
        const uint4 r = *reinterpret_cast<const uint4*>(residual + m * ldr + n0);
        rw[0] = r.x;
        rw[1] = r.y;
        rw[2] = r.z;
        rw[3] = r.w;
      }
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 2 * j;
        o[j] = residual != nullptr
                   ? epilogue_bf16_res(v[e], as, w[e], bf16_lo(rw[j])) |
                         (epilogue_bf16_res(v[e + 1], as, w[e + 1], bf16_hi(rw[j])) << 16)
                   : epilogue_bf16(v[e], as, w[e]) | (epilogue_bf16(v[e + 1], as, w[e + 1]) << 16);
      }
      *reinterpret_cast<uint4*>(out + m * ldo + n0) = make_uint4(o[0], o[1], o[2], o[3]);
      continue;
    }
    for (int j = 0; j < kCols && n0 + j < N; ++j) {
      const int64_t n = n0 + j;
      const float ws = __ldg(w_scale + n);
      out[m * ldo + n] = static_cast<uint16_t>(
          residual != nullptr ? epilogue_bf16_res(ar[j], as, ws, bf16_bits_to_float(residual[m * ldr + n]))
                              : epilogue_bf16(ar[j], as, ws));
    }
  }
}

}  // namespace

cudaError_t launch_epilogue(const int32_t* acc, int64_t ldc, const float* a_scale, const float* w_scale,
                            const uint16_t* residual, int64_t ldr, uint16_t* out, int64_t ldo, int64_t M, int64_t N,
                            cudaStream_t stream) {
  auto al = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
  const bool vec = al(acc, 16) && ldc % 4 == 0 && al(w_scale, 16) && al(out, 16) && ldo % 8 == 0 &&
                   (residual == nullptr || (al(residual, 16) && ldr % 8 == 0));
  const int64_t items = M * ((N + kCols - 1) / kCols);
  // enough CTAs for every SM several times over, at most one item per thread
  const int64_t ctas = std::min<int64_t>((items + kThreads - 1) / kThreads, 152 * 16);
  auto kernel = vec ? epilogue_kernel<true> : epilogue_kernel<false>;
  return launch_kernel(kernel, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), 0, stream, true, acc, ldc, a_scale,
                       w_scale, residual, ldr, out, ldo, M, N);
}

}  // namespace prism
