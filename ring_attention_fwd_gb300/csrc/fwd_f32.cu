// fwd_f32.cu -- ring-order blockwise attention forward in float32 (SIMT).
//
// Same method and schedule as the bf16 tensor-core kernel (query block i
// visits KV blocks j = i, i-1, ... mod N, online softmax per row; "Ring
// Attention" explainer, aiqz.cc, §分块注意力), in plain float32 FMA
// arithmetic: the float32 inputs are used at full precision, which the
// tensor cores' tf32 mode could not match.
//
// One CTA of 256 threads per work unit (64 query rows of one head in one
// query block); KV tiles of 64 rows.  Thread t owns query row t/4 and, for the
// scores, key columns (t%4) + 4k; for the output, head-dim columns (t%4) + 4k.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace ra {
namespace f32 {

constexpr int BM = 64;
constexpr int BN = 64;
constexpr int THREADS = 256;
constexpr int DMAX = 128;

struct Params {
  RingGeom g;
  int S, D;
  int64_t num_units;
  float scale_log2;
  const float* Q;
  const float* K;
  const float* V;
  float* O;
  float* LSE;
  int64_t n_rows;   // B*H*S: extent of Q, K, V, O (rows of D) and LSE
  CheckRec* chk;
};

__global__ void __launch_bounds__(THREADS) fwd_f32_kernel(const Params p) {
  extern __shared__ float sm[];
  const int D = p.D;
  const int ldk = D + 1;                       // padded K rows: conflict-free column reads
  float* sQ = sm;                              // [BM][D]
  float* sK = sQ + BM * D;                     // [BN][D+1]
  float* sV = sK + BN * ldk;                   // [BN][D]
  float* sP = sV + BN * D;                     // [BM][BN+1]
  const RingGeom& g = p.g;
  const int tid = threadIdx.x;
  const int r = tid >> 2;                      // query row in tile
  const int sub = tid & 3;
  const int ncol = D >> 2;                     // output columns per thread (D % 4 == 0)

  for (int64_t u = blockIdx.x; u < p.num_units; u += gridDim.x) {
    const Unit w = unit_at(g, u);
    const int64_t head0 = static_cast<int64_t>(w.bh) * p.S;
    const int rq = w.r0 + r;
    __syncthreads();
    for (int e = tid; e < BM * D; e += THREADS) {
      const int rr = e / D, d = e % D;
      const int lr = w.r0 + rr;
      const int64_t qi = (head0 + static_cast<int64_t>(w.i) * g.c + lr) * D + d;
      sQ[e] = (lr < g.c && RA_CHECK_RANGE(p.chk, SITE_F32_Q, qi, 1, p.n_rows * D)) ? p.Q[qi] : 0.f;
    }
    float m = -INFINITY, l = 0.f;
    float o[DMAX / 4];
#pragma unroll
    for (int k = 0; k < DMAX / 4; ++k) o[k] = 0.f;

    for (int s = 0; s < g.N; ++s) {
      const int j = ring_block(w.i, s, g.N);
      if (!block_visited(g, w.i, j)) continue;
      const int last = kt_last(g, w.i, j, w.r0);
      const int lim = key_limit(g, w.i, j, rq);
      for (int kt = 0; kt <= last; ++kt) {
        __syncthreads();
        for (int e = tid; e < BN * D; e += THREADS) {
          const int rr = e / D, d = e % D;
          const int lk = kt * BN + rr;
          const int64_t gi = (head0 + static_cast<int64_t>(j) * g.c + lk) * D + d;
          const bool in = lk < g.c && RA_CHECK_RANGE(p.chk, SITE_F32_KV, gi, 1, p.n_rows * D);
          sK[rr * ldk + d] = in ? p.K[gi] : 0.f;
          sV[rr * D + d] = in ? p.V[gi] : 0.f;
        }
        __syncthreads();
        const bool masked = tile_masked(g, w.i, j, kt, w.r0);
        float sc[BN / 4];
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < BN / 4; ++k) {
          const int kc = sub + 4 * k;
          const float* qr = sQ + r * D;
          const float* kr = sK + kc * ldk;
          float acc = 0.f;
          for (int d = 0; d < D; ++d) acc = fmaf(qr[d], kr[d], acc);
          if (masked && kt * BN + kc >= lim) acc = -INFINITY;
          sc[k] = acc;
          mx = fmaxf(mx, acc);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m, mx * p.scale_log2);
        const float alpha = (m == -INFINITY) ? 0.f : hw_exp2(m - m_new);
        const float mref = (m_new == -INFINITY) ? 0.f : m_new;
        float rs = 0.f;
#pragma unroll
        for (int k = 0; k < BN / 4; ++k) {
          const float pv = hw_exp2(fmaf(sc[k], p.scale_log2, -mref));
          rs += pv;
          sP[r * (BN + 1) + sub + 4 * k] = pv;
        }
        rs += __shfl_xor_sync(0xffffffffu, rs, 1);
        rs += __shfl_xor_sync(0xffffffffu, rs, 2);
        l = l * alpha + rs;
        m = m_new;
#pragma unroll
        for (int k = 0; k < DMAX / 4; ++k) o[k] *= alpha;
        __syncthreads();
        for (int k = 0; k < BN; ++k) {
          const float pk = sP[r * (BN + 1) + k];
          const float* vr = sV + k * D + sub;
#pragma unroll
          for (int cc = 0; cc < DMAX / 4; ++cc)
            if (cc < ncol) o[cc] = fmaf(pk, vr[4 * cc], o[cc]);
        }
      }
    }
    const int64_t orow = head0 + static_cast<int64_t>(w.i) * g.c + rq;
    if (rq < g.c && RA_CHECK_RANGE(p.chk, SITE_F32_O, orow * D, D, p.n_rows * D) &&
        RA_CHECK_RANGE(p.chk, SITE_F32_LSE, orow, 1, p.n_rows)) {
      const int64_t row = orow;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < DMAX / 4; ++cc)
        if (cc < ncol) p.O[row * D + sub + 4 * cc] = o[cc] * inv;
      if (sub == 0) p.LSE[row] = l > 0.f ? (m + hw_log2(l)) * 0.6931471805599453f : -INFINITY;
    }
  }
}

}  // namespace f32

cudaError_t launch_fwd_f32(const FwdArgs& a) {
  using namespace f32;
  Params p;
  p.g.N = static_cast<int>(a.N);
  p.g.c = static_cast<int>(a.S / a.N);
  p.g.causal = a.causal;
  p.g.striped = a.striped;
  p.g.strict = a.strict;
  p.g.kt_w = BN;
  p.g.n_kt = (p.g.c + BN - 1) / BN;
  p.g.mb_h = BM;
  p.g.n_mb = (p.g.c + BM - 1) / BM;
  p.S = static_cast<int>(a.S);
  p.D = static_cast<int>(a.D);
  p.num_units = a.B * a.H * a.N * p.g.n_mb;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
  p.n_rows = a.B * a.H * a.S;
  p.chk = a.chk;
  p.Q = static_cast<const float*>(a.Q);
  p.K = static_cast<const float*>(a.K);
  p.V = static_cast<const float*>(a.V);
  p.O = static_cast<float*>(a.O);
  p.LSE = a.LSE;
  const size_t smem = sizeof(float) * (BM * a.D + BN * (a.D + 1) + BN * a.D + BM * (BN + 1));
  {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(fwd_f32_kernel),
                                     static_cast<int>(sizeof(float) * (BM * DMAX + BN * (DMAX + 1) +
                                                                       BN * DMAX + BM * (BN + 1))));
    if (e != cudaSuccess) return e;
  }
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 8;
  const int grid = static_cast<int>(p.num_units < cap ? p.num_units : cap);
  if (a.ev) cudaEventRecord(a.ev[0], a.stream);
  fwd_f32_kernel<<<grid > 0 ? grid : 1, THREADS, smem, a.stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (a.ev) cudaEventRecord(a.ev[1], a.stream);
  return e;
}

}  // namespace ra
