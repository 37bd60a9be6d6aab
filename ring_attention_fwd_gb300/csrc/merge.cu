// merge.cu -- LogSumExp merge of two partial attention states, in place.
//
// "Ring Attention如何让大模型突破百万Token上下文…" (answer.freetools.me),
// section "Online Softmax": partial denominators combine as
// l = l1 e^{m1-m} + l2 e^{m2-m}, or in log space with lse = m + ln l.  The
// normalised outputs are re-weighted by each part's share of the total mass.
//
// HBM-bound elementwise kernel: each block owns whole rows, so every thread
// reads lse_a of its row before any thread of the block overwrites it.  The
// state (O_a) and the partial (O_b) are both float32, both bf16, or a float32
// state folding a bf16 partial (a ring host keeping its running output in
// float32 across rounds while each round's partial arrives in bf16).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"

namespace ra {
namespace mrg {

template <typename T, int VEC>
struct Vec;
template <>
struct Vec<float, 4> {
  using type = float4;
};
template <>
struct Vec<__nv_bfloat16, 8> {
  using type = uint4;
};
template <>
struct Vec<__nv_bfloat16, 4> {
  using type = uint2;
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float v, float& x) { x = v; }
__device__ __forceinline__ void from_f(float v, __nv_bfloat16& x) { x = __float2bfloat16_rn(v); }

template <typename T, typename TB, int VEC>
__global__ void __launch_bounds__(1024) merge_kernel(T* __restrict__ Oa, float* la, const TB* __restrict__ Ob,
                                                     const float* lb, int64_t rows, int D, int cpr, int rpb,
                                                     CheckRec* chk) {
  const int tid = threadIdx.x;
  const int rsub = tid / cpr;
  const int ch = tid % cpr;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * rpb + rsub;
  const bool active = rsub < rpb && row < rows && RA_CHECK_RANGE(chk, SITE_MERGE_LSE, row, 1, rows) &&
                     RA_CHECK_RANGE(chk, SITE_MERGE_O, row * D + static_cast<int64_t>(ch) * VEC, VEC, rows * D);
  float A = -INFINITY, Bv = -INFINITY;
  if (active) {
    A = la[row];
    Bv = lb[row];
  }
  __syncthreads();  // all reads of la in this block precede its writes below
  if (!active) return;
  const float M = fmaxf(A, Bv);
  float wa = 0.f, wb = 0.f, lse = -INFINITY;
  if (M != -INFINITY) {
    const float ea = expf(A - M);
    const float eb = expf(Bv - M);
    const float tot = ea + eb;
    lse = M + logf(tot);
    wa = ea / tot;
    wb = eb / tot;
  }
  const int64_t base = row * D + static_cast<int64_t>(ch) * VEC;
  if constexpr (VEC == 1) {
    T out;
    from_f(wa * to_f(Oa[base]) + wb * to_f(Ob[base]), out);
    Oa[base] = out;
  } else {
    using V = typename Vec<T, VEC>::type;
    using VB = typename Vec<TB, VEC>::type;
    V va = *reinterpret_cast<const V*>(Oa + base);
    VB vb = *reinterpret_cast<const VB*>(Ob + base);
    T* ea = reinterpret_cast<T*>(&va);
    const TB* eb = reinterpret_cast<const TB*>(&vb);
#pragma unroll
    for (int k = 0; k < VEC; ++k) from_f(wa * to_f(ea[k]) + wb * to_f(eb[k]), ea[k]);
    *reinterpret_cast<V*>(Oa + base) = va;
  }
  if (ch == 0) la[row] = lse;
}

template <typename T, typename TB, int VEC>
cudaError_t run(void* O_a, float* lse_a, const void* O_b, const float* lse_b, int64_t rows, int64_t D,
                cudaStream_t stream, CheckRec* chk) {
  const int cpr = static_cast<int>(D / VEC);
  int rpb = 256 / cpr;
  if (rpb < 1) rpb = 1;
  const int threads = rpb * cpr;
  const int64_t blocks = (rows + rpb - 1) / rpb;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  merge_kernel<T, TB, VEC><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<T*>(O_a), lse_a, static_cast<const TB*>(O_b), lse_b, rows, static_cast<int>(D), cpr, rpb, chk);
  return cudaGetLastError();
}

__global__ void fill_kernel(float* x, int64_t n, float value) {
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x)
    x[k] = value;
}

}  // namespace mrg

cudaError_t launch_fill(float* x, int64_t n, float value, cudaStream_t stream, int num_sms) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
  mrg::fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, n, value);
  return cudaGetLastError();
}

cudaError_t launch_merge(void* O_a, float* lse_a, const void* O_b, const float* lse_b, int64_t rows,
                         int64_t D, int kind, cudaStream_t stream, int /*num_sms*/, CheckRec* chk) {
  if (rows == 0) return cudaSuccess;
  using bf = __nv_bfloat16;
  const uintptr_t a = reinterpret_cast<uintptr_t>(O_a), b = reinterpret_cast<uintptr_t>(O_b);
  if (kind == MERGE_BF16) {
    if (D % 8 == 0 && ((a | b) & 15) == 0) return mrg::run<bf, bf, 8>(O_a, lse_a, O_b, lse_b, rows, D, stream, chk);
    return mrg::run<bf, bf, 1>(O_a, lse_a, O_b, lse_b, rows, D, stream, chk);
  }
  if (kind == MERGE_F32_BF16) {
    if (D % 4 == 0 && (a & 15) == 0 && (b & 7) == 0)
      return mrg::run<float, bf, 4>(O_a, lse_a, O_b, lse_b, rows, D, stream, chk);
    return mrg::run<float, bf, 1>(O_a, lse_a, O_b, lse_b, rows, D, stream, chk);
  }
  if (D % 4 == 0 && ((a | b) & 15) == 0) return mrg::run<float, float, 4>(O_a, lse_a, O_b, lse_b, rows, D, stream, chk);
  return mrg::run<float, float, 1>(O_a, lse_a, O_b, lse_b, rows, D, stream, chk);
}

}  // namespace ra
