// decode.cu -- ring decode: one new query token per (batch, head) against a
// KV cache spread over N ring blocks.
//
// "Ring Attention with Blockwise Transformers for Near Infinite Context"
// reading notes, §5.6: at inference the query has length 1 and the long KV
// cache is spread along the ring, so no host holds all of it.  "Ring
// Attention如何让大模型突破百万Token上下文…", "局限与未来": decode computes little
// per token, which split-KV ("Flash Decoding") variants address.  Block j of
// an S-row cache is rows [j*c, min((j+1)*c, S)), c = ceil(S/N); the result is
// the LogSumExp merge of the blocks' partial states ("Online Softmax").
//
// HBM-bound: every cached key and value row is read once and used for 4*D
// flops.  Two kernels:
//  1. split_kernel, persistent.  A work item is a chunk of rows inside one
//     ring block (items never straddle blocks, so each partial belongs to one
//     block).  One producer thread streams the chunk's K and V rows into a
//     3-stage shared-memory ring with linear bulk copies (a head's rows are
//     contiguous); 8 consumer warps score and accumulate.  Each half-warp owns
//     a quarter of every stage's rows and keeps its own online-softmax state,
//     so stages need no block-wide barrier; the 16 states are merged once per
//     item into a normalised partial (o[D] f32, lse f32).
//  2. combine_kernel: one CTA per (b, h) merges that head's partials.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace ra {
namespace dec {

constexpr int HD = 128;                               // head dimension
constexpr int R = 64;                                 // cache rows per stage
constexpr int NST = 3;                                // stages
constexpr uint32_t ROW_BYTES = HD * 2;                // one bf16 row
constexpr uint32_t HALF_STAGE = R * ROW_BYTES;        // K (or V) rows of a stage: 16 KB
constexpr uint32_t STAGE_BYTES = 2 * HALF_STAGE;
constexpr int CONSUMERS = 256;                        // 8 warps
constexpr int THREADS = CONSUMERS + 32;               // + the producer warp
constexpr int RG = CONSUMERS / 16;                    // row groups (half-warps)
constexpr int STATE_FLOATS = HD + 2;                  // o[HD], m, l
constexpr uint32_t OFF_STATE = NST * STAGE_BYTES;
constexpr uint32_t OFF_BAR = OFF_STATE + RG * STATE_FLOATS * 4;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 128;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;     // 2 s
constexpr float LN2 = 0.6931471805599453f;
constexpr float LOG2E = 1.4426950408889634f;

struct Bars {
  uint64_t full[NST], empty[NST];
  int abort;
};

struct Params {
  const __nv_bfloat16* q;   // [BH, HD]
  const __nv_bfloat16* K;   // [BH, S, HD]
  const __nv_bfloat16* V;
  float* part_o;            // [items, HD]
  float* part_lse;          // [items]
  int64_t S, c, chunk, cpb, items;
  int N;
  float scale_log2;         // log2(e) / sqrt(HD)
  unsigned int* status;
  int64_t BH;
  CheckRec* chk;
};

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// Head and cache rows [lo, hi) of work item w.
__device__ __forceinline__ void item_rows(const Params& p, int64_t w, int64_t& bh, int64_t& lo, int64_t& hi) {
  const int64_t per_head = p.N * p.cpb;
  bh = w / per_head;
  const int64_t rem = w % per_head;
  const int64_t j = rem / p.cpb, ch = rem % p.cpb;
  const int64_t blo = min64(j * p.c, p.S), bhi = min64((j + 1) * p.c, p.S);
  lo = min64(blo + ch * p.chunk, bhi);
  hi = min64(lo + p.chunk, bhi);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS) : "memory"); }

__global__ void __launch_bounds__(THREADS, 2) split_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  float* state = reinterpret_cast<float*>(smem + OFF_STATE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], CONSUMERS / 32);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&bars->abort, p.status, WAIT_LIMIT_NS};

  if (warp == CONSUMERS / 32) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t ns = 0;
      bool ok = true;
      for (int64_t w = blockIdx.x; w < p.items && ok; w += gridDim.x) {
        int64_t bh, lo, hi;
        item_rows(p, w, bh, lo, hi);
        for (int64_t r0 = lo; r0 < hi; r0 += R, ++ns) {
          const uint32_t bytes = static_cast<uint32_t>(min64(R, hi - r0)) * ROW_BYTES;
          const int st = ns % NST;
          if (!(ok = mbar_wait(&bars->empty[st], ((ns / NST) & 1) ^ 1, wc, ST_DEC_WAIT | 1))) break;
          const int64_t g = (bh * p.S + r0) * HD;
          if (!(ok = RA_CHECK_RANGE(p.chk, SITE_DEC_KV, g, bytes / 2, p.BH * p.S * HD))) break;
          mbar_arrive_expect_tx(&bars->full[st], 2 * bytes);
          bulk_load(smem + st * STAGE_BYTES, p.K + g, bytes, &bars->full[st]);
          bulk_load(smem + st * STAGE_BYTES + HALF_STAGE, p.V + g, bytes, &bars->full[st]);
        }
      }
      // Outlive every copy issued into this CTA's shared memory.
      for (uint32_t k = (ns > NST ? ns - NST : 0); k < ns; ++k)
        mbar_drain(&bars->full[k % NST], (k / NST) & 1, 200000000ull);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Thread = (row group rg, dims [8*dg, 8*dg+8)).  Every consumer runs the
  // same item loop and meets the same named barriers, also after a failed
  // wait (it then skips the arithmetic): no thread can strand the others.
  const int rg = tid >> 4, dg = tid & 15;
  uint32_t ns = 0;
  bool ok = true;
  for (int64_t w = blockIdx.x; w < p.items; w += gridDim.x) {
    int64_t bh, lo, hi;
    item_rows(p, w, bh, lo, hi);
    float qv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (RA_CHECK_RANGE(p.chk, SITE_DEC_Q, bh * HD + dg * 8, 8, p.BH * HD))
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(p.q + bh * HD + dg * 8), qv);
#pragma unroll
    for (int i = 0; i < 8; ++i) qv[i] *= p.scale_log2;
    float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;
    for (int64_t r0 = lo; r0 < hi; r0 += R, ++ns) {
      const int nr = static_cast<int>(min64(R, hi - r0));
      const int st = ns % NST;
      if (ok) ok = mbar_wait(&bars->full[st], (ns / NST) & 1, wc, ST_DEC_WAIT | 2);
      if (!ok) continue;
      const uint8_t* sk = smem + st * STAGE_BYTES + dg * 16;
      const uint8_t* sv = sk + HALF_STAGE;
      float s[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int row = rg + 16 * k;
        float d = 0.f;
        if (row < nr) {
          float kf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(sk + row * ROW_BYTES), kf);
#pragma unroll
          for (int i = 0; i < 8; ++i) d = fmaf(qv[i], kf[i], d);
        }
        d += __shfl_xor_sync(0xffffffffu, d, 8);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        s[k] = row < nr ? d : -INFINITY;
      }
      const float mn = fmaxf(m, fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3])));
      if (mn != -INFINITY) {
        const float alpha = hw_exp2(m - mn);
        l *= alpha;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] *= alpha;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int row = rg + 16 * k;
          if (row < nr) {
            const float pk = hw_exp2(s[k] - mn);
            l += pk;
            float vf[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(sv + row * ROW_BYTES), vf);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = fmaf(pk, vf[i], o[i]);
          }
        }
        m = mn;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[st]);
    }
    // ---- merge the 16 row-group states of this item
    float* my = state + rg * STATE_FLOATS;
#pragma unroll
    for (int i = 0; i < 8; ++i) my[dg * 8 + i] = o[i];
    if (dg == 0) {
      my[HD] = m;
      my[HD + 1] = l;
    }
    consumers_sync();
    if (tid < HD) {
      float M = -INFINITY;
      for (int r = 0; r < RG; ++r) M = fmaxf(M, state[r * STATE_FLOATS + HD]);
      float L = 0.f, acc = 0.f;
      if (M != -INFINITY) {
        for (int r = 0; r < RG; ++r) {
          const float mr = state[r * STATE_FLOATS + HD];
          if (mr == -INFINITY) continue;
          const float wr = hw_exp2(mr - M);
          L = fmaf(state[r * STATE_FLOATS + HD + 1], wr, L);
          acc = fmaf(state[r * STATE_FLOATS + tid], wr, acc);
        }
      }
      if (RA_CHECK_RANGE(p.chk, SITE_DEC_PART, w * HD + tid, 1, p.items * HD)) {
        p.part_o[w * HD + tid] = M == -INFINITY ? 0.f : acc / L;
        if (tid == 0) p.part_lse[w] = M == -INFINITY ? -INFINITY : (M + hw_log2(L)) * LN2;
      }
    }
    consumers_sync();
  }
}

// One CTA (HD threads) per (b, h): merge the head's n partials.
__global__ void __launch_bounds__(HD) combine_kernel(const float* __restrict__ part_o,
                                                     const float* __restrict__ part_lse, int64_t n,
                                                     __nv_bfloat16* __restrict__ O, float* __restrict__ LSE,
                                                     CheckRec* chk) {
  __shared__ float red[HD / 32];
  const int64_t bh = blockIdx.x;
  const int d = threadIdx.x;
  if (!RA_CHECK_RANGE(chk, SITE_DEC_PART, bh * n * HD, n * HD, static_cast<int64_t>(gridDim.x) * n * HD)) return;
  const float* lse = part_lse + bh * n;
  const float* po = part_o + bh * n * HD;
  float M = -INFINITY;
  for (int64_t i = d; i < n; i += HD) M = fmaxf(M, lse[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if ((d & 31) == 0) red[d >> 5] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int k = 1; k < HD / 32; ++k) M = fmaxf(M, red[k]);
  float L = 0.f, acc = 0.f;
  if (M != -INFINITY) {
    for (int64_t i = 0; i < n; ++i) {
      const float li = lse[i];
      if (li == -INFINITY) continue;
      const float wi = hw_exp2((li - M) * LOG2E);
      L += wi;
      acc = fmaf(wi, po[i * HD + d], acc);
    }
  }
  if (!RA_CHECK_RANGE(chk, SITE_DEC_OUT, bh * HD + d, 1, static_cast<int64_t>(gridDim.x) * HD)) return;
  O[bh * HD + d] = __float2bfloat16_rn(M == -INFINITY ? 0.f : acc / L);
  if (d == 0) LSE[bh] = M == -INFINITY ? -INFINITY : M + logf(L);
}

}  // namespace dec

cudaError_t launch_decode_bf16(const DecodeArgs& a) {
  static_assert(dec::SMEM_BYTES <= 232448 / 2, "two CTAs per SM");
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(dec::split_kernel), dec::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dec::Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.K = static_cast<const __nv_bfloat16*>(a.K);
  p.V = static_cast<const __nv_bfloat16*>(a.V);
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  p.S = a.S;
  p.c = a.plan.c;
  p.chunk = a.plan.chunk;
  p.cpb = a.plan.cpb;
  p.items = a.plan.items;
  p.N = static_cast<int>(a.N);
  p.scale_log2 = dec::LOG2E / sqrtf(static_cast<float>(dec::HD));
  p.status = a.status;
  p.BH = a.B * a.H;
  p.chk = a.chk;
  const int64_t slots = 2 * static_cast<int64_t>(a.num_sms);
  const int grid = static_cast<int>(p.items < slots ? p.items : slots);
  if (a.ev) cudaEventRecord(a.ev[0], a.stream);
  dec::split_kernel<<<grid, dec::THREADS, dec::SMEM_BYTES, a.stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.ev) cudaEventRecord(a.ev[1], a.stream);
  dec::combine_kernel<<<static_cast<unsigned>(a.B * a.H), dec::HD, 0, a.stream>>>(
      a.part_o, a.part_lse, a.plan.items / (a.B * a.H), static_cast<__nv_bfloat16*>(a.O), a.LSE, a.chk);
  e = cudaGetLastError();
  if (a.ev) cudaEventRecord(a.ev[2], a.stream);
  return e;
}

}  // namespace ra
