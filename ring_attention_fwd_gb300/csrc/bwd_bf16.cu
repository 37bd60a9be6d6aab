// bwd_bf16.cu -- ring-order backward of blockwise attention, bf16 in / f32
// accumulate, head dim 128, for sm_103a (tcgen05, TMEM, TMA).
//
// The method's backward re-sweeps the KV blocks along the ring from the saved
// softmax state ("Ring Attention with Blockwise Transformers for Near Infinite
// Context" notes, §5.2; recompute in the backward: "Ring Attention" explainer,
// aiqz.cc, §工程实现).  What it computes is the gradient of the forward's
// definition:  P = exp(S - LSE), dV = P^T dO, dP = dO V^T,
// D_vec = rowsum(dO * O), dS = P * (dP - D_vec), dQ = dS K / sqrt(d),
// dK = dS^T Q / sqrt(d).
//
// Three launches, no atomics (dQ, dK, dV are each written by one CTA):
//   1. prep_kernel  -D_vec and -LSE*log2(e) per query row, stored negated
//                   per 128-row query tile (rows past a block's end get 0 and
//                   -inf, so they drop out of P by themselves).
//   2. dkv_kernel   KV-stationary.  A work unit is one 128-row KV tile of one
//                   head, held in shared memory, with dK and dV accumulating
//                   in TMEM while the query tiles of blocks i = j, j+1, ...
//                   (mod N) that see KV block j -- the hosts block j travels
//                   to around the ring -- stream past.  Per query tile:
//                   S^T = K Q^T, dP^T = V dO^T; P^T (bf16) is packed over
//                   S^T and dS^T over dP^T in TMEM; dV += P^T dO and
//                   dK += dS^T Q read them from there.
//   3. dq_kernel    Query-stationary, visiting KV tiles in the forward's ring
//                   order; Q sits in TMEM as an A operand, dO in shared
//                   memory.  Per KV tile: S = Q K^T, dP = dO V^T; P is taken
//                   from S while dP is still being computed; dS (bf16) goes to
//                   its own TMEM region; dQ += dS K accumulates in TMEM.  S
//                   and dP are released as soon as they are in registers, so
//                   the next tile's S and dP MMAs overlap this tile's work.
// Every MMA is 128 wide.  Overlap: the elementwise warps release S as soon as
// it is in registers, so the next tile's S MMA runs while they compute; in the
// dK/dV kernel P^T goes over S^T and dS^T over dP^T, and the next write into
// each region follows the MMA that reads it.  The elementwise arithmetic runs
// on pairs of values with packed f32x2 FMAs, adds and multiplies.
// Both main kernels: warp 0 TMA producer (one thread), warp 1 MMA issuer and
// TMEM owner (the whole warp runs the issue loop so its operands stay
// warp-uniform; one elected lane issues each tcgen05 instruction -- a single
// issuing thread in a divergent branch reaches only ~2/3 of the tensor rate
// with 128-wide MMAs), warps 2-9 the elementwise work, one thread per TMEM
// lane (row): warp w reads lane quadrant w % 4 (the quadrant a warp may
// address), warps 2-5 own columns [0, 64) and warps 6-9 columns [64, 128), and
// each writes its packed bf16 results only over columns it has read.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace ra {
namespace bwd {

constexpr int BT = 128;        // rows per KV tile and per query tile
constexpr int HD = 128;
constexpr int THREADS = 320;
constexpr uint32_t TILE_BYTES = BT * HD * 2;  // 32 KB
constexpr uint32_t BOX_BYTES = TILE_BYTES / 2;
constexpr uint32_t VEC_BYTES = BT * 4;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;


// Descriptors of a 128B-swizzled tile (two 64-column boxes): the K-slice kk
// (16 elements) of a K-major operand, or of an MN-major operand, as offsets
// from the tile's kk = 0 descriptor.
__device__ __forceinline__ uint64_t kdesc0(uint32_t tile) { return sdesc(tile, 16, 1024, SWZ_128B); }
__device__ __forceinline__ uint64_t mndesc0(uint32_t tile) { return sdesc(tile, BOX_BYTES, 1024, SWZ_128B); }
__device__ __forceinline__ uint64_t kslice(uint64_t d0, int kk) {
  return sdesc_add(d0, (kk >> 2) * BOX_BYTES + (kk & 3) * 32);
}
__device__ __forceinline__ uint64_t mnslice(uint64_t d0, int kk) { return sdesc_add(d0, kk * 16 * 128); }
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int kk) { return kslice(kdesc0(tile), kk); }
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int kk) { return mnslice(mndesc0(tile), kk); }

// Store 128 f32 TMEM columns of this thread's lane as one bf16 row (scaled).
__device__ __forceinline__ void store_row_bf16(uint32_t tcol, __nv_bfloat16* out, float sc, bool ok, int ncols) {
  for (int ch = 0; ch < ncols / 32; ++ch) {
    uint32_t v[32];
    tmem_ld32(tcol + ch * 32, v);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
      pk[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * sc, __uint_as_float(v[2 * k + 1]) * sc);
    if (ok) {
      uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
    }
  }
}

// Add ncols f32 TMEM columns of this thread's lane, scaled, into an f32 row in
// global memory that this thread alone owns (ring-step accumulation).
__device__ __forceinline__ void add_row_f32(uint32_t tcol, float* out, float sc, bool ok, int ncols) {
  for (int ch = 0; ch < ncols / 32; ++ch) {
    uint32_t v[32];
    tmem_ld32(tcol + ch * 32, v);
    tmem_ld_wait();
    if (ok) {
      float4* dst = reinterpret_cast<float4*>(out + ch * 32);
#pragma unroll
      for (int v4 = 0; v4 < 8; ++v4) {
        float4 a = dst[v4];
        a.x = fmaf(__uint_as_float(v[4 * v4]), sc, a.x);
        a.y = fmaf(__uint_as_float(v[4 * v4 + 1]), sc, a.y);
        a.z = fmaf(__uint_as_float(v[4 * v4 + 2]), sc, a.z);
        a.w = fmaf(__uint_as_float(v[4 * v4 + 3]), sc, a.w);
        dst[v4] = a;
      }
    }
  }
}

struct Params {
  RingGeom g;        // kt_w = mb_h = 128
  int S;
  int64_t num_units;
  float scale_log2;  // log2(e) / sqrt(D)
  float inv_sqrt_d;
  const float* nlse2;  // [BH][N][n_mb][128]: -LSE * log2(e)
  const float* ndvec;  // [BH][N][n_mb][128]: -D_vec
  __nv_bfloat16* dQ;   // bf16 outputs (accumulate == 0)
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  float* dQf;          // f32 accumulators, added to (accumulate == 1)
  float* dKf;
  float* dVf;
  int accumulate;
  unsigned int* status;
  int64_t BH;          // heads (B*H)
  int64_t vec_rows;    // rows of nlse2 / ndvec: BH * N * n_mb * 128
  CheckRec* chk;
  unsigned long long* clk;   // clock record of this launch (kernel timing) or null
};

__device__ __forceinline__ int64_t vec_row(const RingGeom& g, int bh, int i, int qt) {
  return ((static_cast<int64_t>(bh) * g.N + i) * g.n_mb + qt) * BT;
}

// ============================================================== dK, dV
namespace kv {
// Q tiles (with their -LSE*log2(e) rows) and dO tiles (with their -D_vec rows) stream
// through separate rings.  Q is the first operand a tile needs (S^T) and the
// last one it releases (dK), so it gets the deeper ring; dO is released after
// dV, a tile earlier.
constexpr int QSTAGE = 3;
constexpr int DSTAGE = 2;
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + TILE_BYTES;
constexpr uint32_t OFF_Q = OFF_V + TILE_BYTES;               // QSTAGE tiles
constexpr uint32_t OFF_DO = OFF_Q + QSTAGE * TILE_BYTES;     // DSTAGE tiles
constexpr uint32_t OFF_LSE = OFF_DO + DSTAGE * TILE_BYTES;   // QSTAGE x nlse2[128]
constexpr uint32_t OFF_DVEC = OFF_LSE + QSTAGE * VEC_BYTES;  // DSTAGE x ndvec[128]
constexpr uint32_t OFF_BAR = OFF_DVEC + DSTAGE * VEC_BYTES;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Bars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[QSTAGE], q_empty[QSTAGE];
  uint64_t do_full[DSTAGE], do_empty[DSTAGE];
  uint64_t s_full, dp_full, p_full, ds_full, dkv_full, dkv_empty, drain;
  uint32_t tmem_base;
  int abort;
};

// Work units (bh, j, kt): heaviest first inside a head.
__device__ __forceinline__ void unit_at(const RingGeom& g, int64_t u, int& bh, int& j, int& kt) {
  const int64_t per_head = static_cast<int64_t>(g.N) * g.n_kt;
  bh = static_cast<int>(u / per_head);
  const int rem = static_cast<int>(u % per_head);
  if (g.causal && g.striped) {   // work falls with kt only
    kt = rem / g.N;
    j = rem % g.N;
  } else {                       // contiguous causal: falls with j, then kt
    j = rem / g.n_kt;
    kt = rem % g.n_kt;
  }
}
// KV block j meets query blocks i = j + s (mod N); the contiguous causal sweep
// never reaches blocks i < j.
__device__ __forceinline__ bool q_block_visited(const RingGeom& g, int i, int j) {
  return !(g.causal && !g.striped && i < j);
}
// First query tile of block i that sees KV tile kt of block j.
__device__ __forceinline__ int qt_first(const RingGeom& g, int i, int j, int kt) {
  return diag_type(g, i, j) ? kt : 0;
}
__device__ __forceinline__ int unit_steps(const RingGeom& g, int j, int kt) {
  int T = 0;
  for (int s = 0; s < g.N; ++s) {
    const int i = (j + s) % g.N;
    if (q_block_visited(g, i, j)) T += g.n_mb - qt_first(g, i, j, kt);
  }
  return T;
}
// Packed bf16 column of the 16-query K-slice kk of P^T (inside the S^T region)
// and of dS^T (inside the dP^T region): warpgroup g (queries [64g, 64g+64))
// packs its values at [64g, 64g+32) of the region it has just read.
__device__ __forceinline__ uint32_t pcol(int kk) { return 64 * (kk >> 2) + 8 * (kk & 3); }

__global__ void __launch_bounds__(THREADS, 1)
dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const RingGeom& g = p.g;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, ST_BWD_WAIT | 0xff);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int s = 0; s < QSTAGE; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    for (int s = 0; s < DSTAGE; ++s) {
      mbar_init(&bars->do_full[s], 1);
      mbar_init(&bars->do_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->dkv_empty, 256);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  clock_mark(p.clk, 0);
  // TMEM: dV [0,128) dK [128,256) S^T [256,384) dP^T [384,512); P^T is packed
  // (bf16) over S^T and dS^T over dP^T once each has been read.
  const uint32_t T_DV = tmem, T_DK = tmem + 128, T_S = tmem + 256, T_DP = tmem + 384;
  const WaitCtx wc{&bars->abort, p.status, WAIT_LIMIT_NS};
  const int grid = gridDim.x, cta = blockIdx.x;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      uint32_t nq = 0, ndo = 0, nkv = 0, kve_ph = 0;
      bool ok = true;
      for (int64_t r = 0; ok; ++r) {
        const int64_t u = snake_pos(r, cta, grid);
        if (u >= p.num_units) break;
        int bh, j, kt;
        unit_at(g, u, bh, j, kt);
        if (nkv > 0) {
          if (!(ok = mbar_wait(&bars->kv_empty, kve_ph, wc, ST_BWD_WAIT | 1))) break;
          kve_ph ^= 1;
        }
        mbar_arrive_expect_tx(&bars->kv_full, 2 * TILE_BYTES);
        const int krow = j * g.c + kt * BT;
        for (int h = 0; h < 2; ++h) {
          if (!RA_CHECK_BOX(p.chk, SITE_DKV_TMA_KV, h * 64, krow, bh, HD, p.S, p.BH, 8)) continue;
          tma_load_3d(smem + OFF_K + h * BOX_BYTES, &tmK, &bars->kv_full, h * 64, krow, bh);
          tma_load_3d(smem + OFF_V + h * BOX_BYTES, &tmV, &bars->kv_full, h * 64, krow, bh);
        }
        ++nkv;
        for (int s = 0; s < g.N && ok; ++s) {
          const int i = (j + s) % g.N;
          if (!q_block_visited(g, i, j)) continue;
          for (int qt = qt_first(g, i, j, kt); qt < g.n_mb; ++qt) {
            const int qrow = i * g.c + qt * BT;
            const int64_t vrow = vec_row(g, bh, i, qt);
            const int sq = nq % QSTAGE;
            if (!(ok = mbar_wait(&bars->q_empty[sq], ((nq / QSTAGE) & 1) ^ 1, wc, ST_BWD_WAIT | 2))) break;
            mbar_arrive_expect_tx(&bars->q_full[sq], TILE_BYTES + VEC_BYTES);
            for (int h = 0; h < 2; ++h)
              if (RA_CHECK_BOX(p.chk, SITE_DKV_TMA_Q, h * 64, qrow, bh, HD, p.S, p.BH, 8))
                tma_load_3d(smem + OFF_Q + sq * TILE_BYTES + h * BOX_BYTES, &tmQ, &bars->q_full[sq], h * 64, qrow,
                            bh);
            if (RA_CHECK_RANGE(p.chk, SITE_DKV_VEC, vrow, BT, p.vec_rows))
              bulk_load(smem + OFF_LSE + sq * VEC_BYTES, p.nlse2 + vrow, VEC_BYTES, &bars->q_full[sq]);
            ++nq;
            const int sd = ndo % DSTAGE;
            if (!(ok = mbar_wait(&bars->do_empty[sd], ((ndo / DSTAGE) & 1) ^ 1, wc, ST_BWD_WAIT | 0xb))) break;
            mbar_arrive_expect_tx(&bars->do_full[sd], TILE_BYTES + VEC_BYTES);
            for (int h = 0; h < 2; ++h)
              if (RA_CHECK_BOX(p.chk, SITE_DKV_TMA_DO, h * 64, qrow, bh, HD, p.S, p.BH, 8))
                tma_load_3d(smem + OFF_DO + sd * TILE_BYTES + h * BOX_BYTES, &tmDO, &bars->do_full[sd], h * 64,
                            qrow, bh);
            if (RA_CHECK_RANGE(p.chk, SITE_DKV_VEC, vrow, BT, p.vec_rows))
              bulk_load(smem + OFF_DVEC + sd * VEC_BYTES, p.ndvec + vrow, VEC_BYTES, &bars->do_full[sd]);
            ++ndo;
          }
        }
      }
      if (!ok) {
        for (uint32_t k = (nq > QSTAGE ? nq - QSTAGE : 0); k < nq; ++k)
          mbar_drain(&bars->q_full[k % QSTAGE], (k / QSTAGE) & 1, 200000000ull);
        for (uint32_t k = (ndo > DSTAGE ? ndo - DSTAGE : 0); k < ndo; ++k)
          mbar_drain(&bars->do_full[k % DSTAGE], (k / DSTAGE) & 1, 200000000ull);
        if (nkv > 0) mbar_drain(&bars->kv_full, (nkv - 1) & 1, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop (warp-uniform operands); one elected
    // lane issues each tcgen05 instruction.
    {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t ID_KK = idesc_bf16_f32(BT, BT, 0, 0);   // A, B K-major, N = 128
      constexpr uint32_t ID_TM = idesc_bf16_f32(BT, HD, 0, 1);   // A from TMEM, B MN-major
      const uint64_t dK0 = kdesc0(sbase + OFF_K), dV0 = kdesc0(sbase + OFF_V);
      uint32_t it = 0, kv_ph = 0, pf_ph = 0, dsf_ph = 0, dkve_ph = 0;
      bool ok = true, first_unit = true;
      auto issue_s = [=](int st) {   // S^T = K Q^T
        const uint64_t bq = kdesc0(sbase + OFF_Q + st * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) mma_ss_w(T_S, kslice(dK0, kk), kslice(bq, kk), ID_KK, kk > 0);
      };
      auto issue_dp = [=](int sd) {  // dP^T = V dO^T
        const uint64_t bdo = kdesc0(sbase + OFF_DO + sd * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) mma_ss_w(T_DP, kslice(dV0, kk), kslice(bdo, kk), ID_KK, kk > 0);
      };
      // Per tile the tensor pipe runs dV(t), S^T(t+1), dK(t), dP^T(t+1).  The
      // S region holds S^T(t), then P^T(t) (written by the elementwise warps),
      // read by dV(t); S^T(t+1) is issued after dV(t), so it overwrites P^T only
      // once it has been read.  Likewise the dP^T region: dP^T(t), dS^T(t),
      // read by dK(t), then dP^T(t+1).
      for (int64_t r = 0; ok; ++r) {
        const int64_t u = snake_pos(r, cta, grid);
        if (u >= p.num_units) break;
        int bh, j, kt;
        unit_at(g, u, bh, j, kt);
        const int T = unit_steps(g, j, kt);
        if (!(ok = mbar_wait_w(&bars->kv_full, kv_ph, wc, ST_BWD_WAIT | 3))) break;
        kv_ph ^= 1;
        if (!(ok = mbar_wait_w(&bars->q_full[it % QSTAGE], (it / QSTAGE) & 1, wc, ST_BWD_WAIT | 4))) break;
        tc_fence_after();
        issue_s(it % QSTAGE);    // S region: last read by the previous tile's dV MMAs
        mma_commit_w(&bars->s_full);
        if (!(ok = mbar_wait_w(&bars->do_full[it % DSTAGE], (it / DSTAGE) & 1, wc, ST_BWD_WAIT | 0xc))) break;
        tc_fence_after();
        issue_dp(it % DSTAGE);   // dP^T region: last read by the previous tile's dK MMAs
        mma_commit_w(&bars->dp_full);
        for (int t = 0; t < T && ok; ++t, ++it) {
          const int st = it % QSTAGE, sd = it % DSTAGE;
          const int nst = (it + 1) % QSTAGE, nsd = (it + 1) % DSTAGE;
          if (!(ok = mbar_wait_w(&bars->p_full, pf_ph, wc, ST_BWD_WAIT | 5))) break;
          pf_ph ^= 1;
          if (t == 0 && !first_unit) {
            if (!(ok = mbar_wait_w(&bars->dkv_empty, dkve_ph, wc, ST_BWD_WAIT | 6))) break;
            dkve_ph ^= 1;
          }
          tc_fence_after();
          const uint32_t acc = t > 0 ? 1u : 0u;
          const uint64_t mdo = mndesc0(sbase + OFF_DO + sd * TILE_BYTES), mq = mndesc0(sbase + OFF_Q + st * TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)   // dV += P^T dO  (P^T in the S region)
            mma_ts_w(T_DV, T_S + pcol(kk), mnslice(mdo, kk), ID_TM, (kk > 0) | acc);
          if (t + 1 < T) {   // next tile's S^T, behind the dV MMAs that read P^T
            if (!(ok = mbar_wait_w(&bars->q_full[nst], ((it + 1) / QSTAGE) & 1, wc, ST_BWD_WAIT | 0xa))) break;
            tc_fence_after();
            issue_s(nst);
            mma_commit_w(&bars->s_full);
          }
          if (!(ok = mbar_wait_w(&bars->ds_full, dsf_ph, wc, ST_BWD_WAIT | 0x10))) break;
          dsf_ph ^= 1;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)   // dK += dS^T Q  (dS^T in the dP^T region)
            mma_ts_w(T_DK, T_DP + pcol(kk), mnslice(mq, kk), ID_TM, (kk > 0) | acc);
          mma_commit_w(&bars->q_empty[st]);
          mma_commit_w(&bars->do_empty[sd]);   // the dO slot holds D_vec, read until dS^T was stored
          if (t + 1 < T) {
            if (!(ok = mbar_wait_w(&bars->do_full[nsd], ((it + 1) / DSTAGE) & 1, wc, ST_BWD_WAIT | 0xc))) break;
            tc_fence_after();
            issue_dp(nsd);
            mma_commit_w(&bars->dp_full);
          }
        }
        if (!ok) break;
        mma_commit_w(&bars->kv_empty);
        mma_commit_w(&bars->dkv_full);
        first_unit = false;
      }
      mma_commit_w(&bars->drain);
      mbar_drain(&bars->drain, 0, 200000000ull);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ P^T and dS^T, epilogue
    const int grp = (warp - 2) >> 2;                     // query columns [64*grp, +64)
    const int quad = warp & 3;
    const int t_row = quad * 32 + lane;                  // key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    uint32_t it = 0, s_ph = 0, dp_ph = 0, dkv_ph = 0;
    bool ok = true;
    for (int64_t r = 0; ok; ++r) {
      const int64_t u = snake_pos(r, cta, grid);
      if (u >= p.num_units) break;
      int bh, j, kt;
      unit_at(g, u, bh, j, kt);
      const int lk = kt * BT + t_row;                    // key row inside block j
      const bool key_ok = lk < g.c;
      for (int s = 0; s < g.N && ok; ++s) {
        const int i = (j + s) % g.N;
        if (!q_block_visited(g, i, j)) continue;
        const bool dpair = diag_type(g, i, j);
        const int incl = diag_incl(g, i, j);
        for (int qt = qt_first(g, i, j, kt); qt < g.n_mb && ok; ++qt, ++it) {
          const int st = it % QSTAGE, sd = it % DSTAGE;
          if (!(ok = mbar_wait(&bars->q_full[st], (it / QSTAGE) & 1, wc, ST_BWD_WAIT | 7))) break;
          if (!(ok = mbar_wait(&bars->do_full[sd], (it / DSTAGE) & 1, wc, ST_BWD_WAIT | 0xe))) break;
          if (!(ok = mbar_wait(&bars->s_full, s_ph, wc, ST_BWD_WAIT | 8))) break;
          s_ph ^= 1;
          tc_fence_after();
          const uint32_t tS = T_S + lane_off + 64 * grp;
          const uint32_t tDP = T_DP + lane_off + 64 * grp;
          uint32_t sv[64];
          tmem_ld32(tS, sv);
          tmem_ld32(tS + 32, sv + 32);
          tmem_ld_wait();
          // P^T while the previous tile's dK and this tile's dP^T run; it goes
          // over this group's own S^T columns, so dV can start at once.
          // Query column q of the tile is visible to this key row iff q >= vis_lo.
          int vis_lo = 0;
          if (!key_ok) vis_lo = BT;
          else if (dpair && qt == kt) vis_lo = t_row + 1 - incl;
          const float* nlse2 = reinterpret_cast<const float*>(smem + OFF_LSE + st * VEC_BYTES) + 64 * grp;
          const float* ndvec = reinterpret_cast<const float*>(smem + OFF_DVEC + sd * VEC_BYTES) + 64 * grp;
          const int q0 = 64 * grp;
          float pv[64];
          // Exponent arguments two at a time (packed f32x2 FMA, each lane
          // rounded as fmaf): s * log2(e)/sqrt(d) - LSE*log2(e).
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c);
            const float2 a01 = __ffma2_rn(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2v,
                                          make_float2(l4.x, l4.y));
            const float2 a23 = __ffma2_rn(make_float2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sl2v,
                                          make_float2(l4.z, l4.w));
            pv[c] = hw_exp2(a01.x);
            pv[c + 1] = hw_exp2(a01.y);
            pv[c + 2] = hw_exp2(a23.x);
            pv[c + 3] = hw_exp2(a23.y);
          }
          if (vis_lo > q0) {   // some column of this thread hidden (diagonal or ragged tile)
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (q0 + c < vis_lo) pv[c] = 0.f;
          }
          {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) pk[c >> 1] = pack_bf16x2(pv[c], pv[c + 1]);
            tmem_st16(tS, pk);
            tmem_st16(tS + 16, pk + 16);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->p_full);
          if (!(ok = mbar_wait(&bars->dp_full, dp_ph, wc, ST_BWD_WAIT | 0xf))) break;
          dp_ph ^= 1;
          tc_fence_after();
          uint32_t dpv[64];
          tmem_ld32(tDP, dpv);
          tmem_ld32(tDP + 32, dpv + 32);
          tmem_ld_wait();
          {
            uint32_t dk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {   // dS^T = P^T (dP^T - D_vec), two lanes at a time
              const float2 nd2 = *reinterpret_cast<const float2*>(ndvec + c);
              const float2 ds = __fmul2_rn(make_float2(pv[c], pv[c + 1]),
                                           __fadd2_rn(make_float2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])),
                                                      nd2));
              dk[c >> 1] = pack_bf16x2(ds.x, ds.y);
            }
            tmem_st16(tDP, dk);            // dS^T over this group's own dP^T columns
            tmem_st16(tDP + 16, dk + 16);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->ds_full);
        }
      }
      if (!ok) break;
      // ---- epilogue: group 0 writes dV, group 1 writes dK / sqrt(d)
      if (!(ok = mbar_wait(&bars->dkv_full, dkv_ph, wc, ST_BWD_WAIT | 9))) break;
      dkv_ph ^= 1;
      tc_fence_after();
      const int64_t krow = static_cast<int64_t>(bh) * p.S + static_cast<int64_t>(j) * g.c + lk;
      const bool st_ok = key_ok && RA_CHECK_RANGE(p.chk, SITE_DKV_OUT, krow * HD, HD, p.BH * p.S * HD);
      if (p.accumulate) {
        if (grp == 0)
          add_row_f32(T_DV + lane_off, p.dVf + krow * HD, 1.f, st_ok, HD);
        else
          add_row_f32(T_DK + lane_off, p.dKf + krow * HD, p.inv_sqrt_d, st_ok, HD);
      } else if (grp == 0) {
        store_row_bf16(T_DV + lane_off, p.dV + krow * HD, 1.f, st_ok, HD);
      } else {
        store_row_bf16(T_DK + lane_off, p.dK + krow * HD, p.inv_sqrt_d, st_ok, HD);
      }
      tc_fence_before();
      mbar_arrive(&bars->dkv_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  clock_mark(p.clk, 1);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
}  // namespace kv

// ============================================================== dQ
namespace q {
// K tiles stream through a 4-stage ring and V tiles through a 2-stage one: K
// is the first operand a tile needs (S) and the last it releases (dQ += dS K),
// V is released as soon as dP has been computed.
constexpr int KSTAGE = 4;
constexpr int VSTAGE = 2;
constexpr uint32_t OFF_DO = 0;                              // dO tile of the unit
constexpr uint32_t OFF_K = OFF_DO + TILE_BYTES;             // KSTAGE tiles
constexpr uint32_t OFF_V = OFF_K + KSTAGE * TILE_BYTES;     // VSTAGE tiles
constexpr uint32_t OFF_BAR = OFF_V + VSTAGE * TILE_BYTES;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Bars {
  uint64_t do_full, do_empty;
  uint64_t k_full[KSTAGE], k_empty[KSTAGE], v_full[VSTAGE], v_empty[VSTAGE];
  uint64_t qo_full, qo_empty, s_full, s_free, dp_full, dp_free, p_full, ds_free, dq_full, dq_empty, drain;
  uint32_t tmem_base;
  int abort;
};
// Packed bf16 column of the 16-key K-slice kk of dS inside the dS region:
// warpgroup g (keys [64g, 64g+64)) packs its dS at [32g, 32g+32).
__device__ __forceinline__ uint32_t pcol(int kk) { return 32 * (kk >> 2) + 8 * (kk & 3); }

__global__ void __launch_bounds__(THREADS, 1)
dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
          const __grid_constant__ CUtensorMap tmDO, const __nv_bfloat16* __restrict__ Q, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const RingGeom& g = p.g;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, ST_BWD_WAIT | 0xfe);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 1);
    for (int s = 0; s < KSTAGE; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < VSTAGE; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->qo_full, 256);
    mbar_init(&bars->qo_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 256);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, 256);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, 256);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  clock_mark(p.clk, 0);
  // TMEM: dQ [0,128) Q [128,192) (bf16 rows, A operand) dS [192,256) (bf16, A operand)
  //       S [256,384) dP [384,512).  S and dP are free again as soon as they are
  //       in registers, so the next KV tile's S and dP MMAs overlap this tile's
  //       elementwise work.
  const uint32_t T_DQ = tmem, T_Q = tmem + 128, T_DS = tmem + 192, T_S = tmem + 256, T_DP = tmem + 384;
  const WaitCtx wc{&bars->abort, p.status, WAIT_LIMIT_NS};
  const int grid = gridDim.x, cta = blockIdx.x;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      uint32_t nk = 0, nv = 0, nd = 0, de_ph = 0;
      bool ok = true;
      for (int64_t r = 0; ok; ++r) {
        const int64_t u = snake_pos(r, cta, grid);
        if (u >= p.num_units) break;
        const Unit w = unit_at(g, u);
        if (nd > 0) {
          if (!(ok = mbar_wait(&bars->do_empty, de_ph, wc, ST_BWD_WAIT | 0x11))) break;
          de_ph ^= 1;
        }
        mbar_arrive_expect_tx(&bars->do_full, TILE_BYTES);
        for (int h = 0; h < 2; ++h)
          if (RA_CHECK_BOX(p.chk, SITE_DQ_TMA_DO, h * 64, w.i * g.c + w.r0, w.bh, HD, p.S, p.BH, 8))
            tma_load_3d(smem + OFF_DO + h * BOX_BYTES, &tmDO, &bars->do_full, h * 64, w.i * g.c + w.r0, w.bh);
        ++nd;
        for (int s = 0; s < g.N && ok; ++s) {
          const int j = ring_block(w.i, s, g.N);
          if (!block_visited(g, w.i, j)) continue;
          const int last = kt_last(g, w.i, j, w.r0);
          for (int kt = 0; kt <= last; ++kt) {
            const int krow = j * g.c + kt * BT;
            const int sk = nk % KSTAGE;
            if (!(ok = mbar_wait(&bars->k_empty[sk], ((nk / KSTAGE) & 1) ^ 1, wc, ST_BWD_WAIT | 0x12))) break;
            mbar_arrive_expect_tx(&bars->k_full[sk], TILE_BYTES);
            for (int h = 0; h < 2; ++h)
              if (RA_CHECK_BOX(p.chk, SITE_DQ_TMA_K, h * 64, krow, w.bh, HD, p.S, p.BH, 8))
                tma_load_3d(smem + OFF_K + sk * TILE_BYTES + h * BOX_BYTES, &tmK, &bars->k_full[sk], h * 64, krow,
                            w.bh);
            ++nk;
            const int sv = nv % VSTAGE;
            if (!(ok = mbar_wait(&bars->v_empty[sv], ((nv / VSTAGE) & 1) ^ 1, wc, ST_BWD_WAIT | 0x1a))) break;
            mbar_arrive_expect_tx(&bars->v_full[sv], TILE_BYTES);
            for (int h = 0; h < 2; ++h)
              if (RA_CHECK_BOX(p.chk, SITE_DQ_TMA_V, h * 64, krow, w.bh, HD, p.S, p.BH, 8))
                tma_load_3d(smem + OFF_V + sv * TILE_BYTES + h * BOX_BYTES, &tmV, &bars->v_full[sv], h * 64, krow,
                            w.bh);
            ++nv;
          }
        }
      }
      if (!ok) {
        for (uint32_t k = (nk > KSTAGE ? nk - KSTAGE : 0); k < nk; ++k)
          mbar_drain(&bars->k_full[k % KSTAGE], (k / KSTAGE) & 1, 200000000ull);
        for (uint32_t k = (nv > VSTAGE ? nv - VSTAGE : 0); k < nv; ++k)
          mbar_drain(&bars->v_full[k % VSTAGE], (k / VSTAGE) & 1, 200000000ull);
        if (nd > 0) mbar_drain(&bars->do_full, (nd - 1) & 1, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop (warp-uniform operands); one elected
    // lane issues each tcgen05 instruction.
    {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t ID_KK = idesc_bf16_f32(BT, BT, 0, 0);   // B K-major, N = 128
      constexpr uint32_t ID_TM = idesc_bf16_f32(BT, HD, 0, 1);   // A (TMEM), B MN-major
      const uint64_t dDO0 = kdesc0(sbase + OFF_DO);
      uint32_t it = 0, de_ph = 0, qo_ph = 0, sf_ph = 0, df_ph = 0, pf_ph = 0, dqe_ph = 0;
      bool ok = true, first_unit = true, first_s = true, first_dp = true;
      auto issue_s = [=](int st) {   // S = Q K^T  (Q from TMEM)
        const uint64_t bk = kdesc0(sbase + OFF_K + st * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) mma_ts_w(T_S, T_Q + kk * 8, kslice(bk, kk), ID_KK, kk > 0);
      };
      auto issue_dp = [=](int sv) {  // dP = dO V^T  (dO from shared memory)
        const uint64_t bv = kdesc0(sbase + OFF_V + sv * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) mma_ss_w(T_DP, kslice(dDO0, kk), kslice(bv, kk), ID_KK, kk > 0);
      };
      // S for KV tile k_it once its K tile has landed and the previous S is in
      // registers, then dP once its V tile has landed and the previous dP is in
      // registers.
      auto issue_tile = [&](uint32_t k_it) -> bool {
        if (!mbar_wait_w(&bars->k_full[k_it % KSTAGE], (k_it / KSTAGE) & 1, wc, ST_BWD_WAIT | 0x14)) return false;
        if (!first_s) {
          if (!mbar_wait_w(&bars->s_free, sf_ph, wc, ST_BWD_WAIT | 0x1c)) return false;
          sf_ph ^= 1;
        }
        first_s = false;
        tc_fence_after();
        issue_s(k_it % KSTAGE);
        mma_commit_w(&bars->s_full);
        if (!mbar_wait_w(&bars->v_full[k_it % VSTAGE], (k_it / VSTAGE) & 1, wc, ST_BWD_WAIT | 0x15)) return false;
        if (!first_dp) {
          if (!mbar_wait_w(&bars->dp_free, df_ph, wc, ST_BWD_WAIT | 0x1d)) return false;
          df_ph ^= 1;
        }
        first_dp = false;
        tc_fence_after();
        issue_dp(k_it % VSTAGE);
        mma_commit_w(&bars->dp_full);
        mma_commit_w(&bars->v_empty[k_it % VSTAGE]);   // V is done with once dP is computed
        return true;
      };
      for (int64_t r = 0; ok; ++r) {
        const int64_t u = snake_pos(r, cta, grid);
        if (u >= p.num_units) break;
        const Unit w = unit_at(g, u);
        const int T = unit_tiles(g, w.i, w.r0);
        if (!(ok = mbar_wait_w(&bars->do_full, de_ph, wc, ST_BWD_WAIT | 0x13))) break;
        de_ph ^= 1;
        if (!(ok = mbar_wait_w(&bars->qo_full, qo_ph, wc, ST_BWD_WAIT | 0x1e))) break;
        qo_ph ^= 1;
        if (!(ok = issue_tile(it))) break;
        for (int t = 0; t < T && ok; ++t, ++it) {
          const int st = it % KSTAGE;
          if (t + 1 < T && !(ok = issue_tile(it + 1))) break;
          if (!(ok = mbar_wait_w(&bars->p_full, pf_ph, wc, ST_BWD_WAIT | 0x16))) break;
          pf_ph ^= 1;
          if (t == 0 && !first_unit) {
            if (!(ok = mbar_wait_w(&bars->dq_empty, dqe_ph, wc, ST_BWD_WAIT | 0x17))) break;
            dqe_ph ^= 1;
          }
          tc_fence_after();
          const uint64_t mk = mndesc0(sbase + OFF_K + st * TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)   // dQ += dS K  (dS from TMEM, K MN-major)
            mma_ts_w(T_DQ, T_DS + pcol(kk), mnslice(mk, kk), ID_TM, (kk > 0) | (t > 0 ? 1u : 0u));
          mma_commit_w(&bars->ds_free);
          mma_commit_w(&bars->k_empty[st]);
          if (t == T - 1) {
            mma_commit_w(&bars->do_empty);
            mma_commit_w(&bars->qo_empty);
            mma_commit_w(&bars->dq_full);
          }
        }
        first_unit = false;
      }
      mma_commit_w(&bars->drain);
      mbar_drain(&bars->drain, 0, 200000000ull);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------- Q rows, dS, epilogue
    const int grp = (warp - 2) >> 2;                     // key columns [64*grp, +64)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;                    // query row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    uint32_t s_ph = 0, dp_ph = 0, dsf_ph = 0, dq_ph = 0, qoe_ph = 0;
    bool ok = true, first_unit = true, first_ds = true;
    for (int64_t r = 0; ok; ++r) {
      const int64_t u = snake_pos(r, cta, grid);
      if (u >= p.num_units) break;
      const Unit w = unit_at(g, u);
      const int rq = w.r0 + row;
      const int64_t grow = static_cast<int64_t>(w.bh) * p.S + static_cast<int64_t>(w.i) * g.c + rq;
      // ---- this unit's Q row into TMEM: group g copies head-dim columns [64g, 64g+64)
      if (!first_unit) {
        if (!(ok = mbar_wait(&bars->qo_empty, qoe_ph, wc, ST_BWD_WAIT | 0x1b))) break;
        qoe_ph ^= 1;
        tc_fence_after();
      }
      first_unit = false;
      {
        uint32_t v[32];
        const uint4* s4 = reinterpret_cast<const uint4*>(Q + grow * HD + 64 * grp);
        const bool inb = w.i * g.c + rq < p.S &&
                         RA_CHECK_RANGE(p.chk, SITE_DQ_Q, grow * HD + 64 * grp, 64, p.BH * p.S * HD);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 x = inb ? __ldg(s4 + k) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * k] = x.x;
          v[4 * k + 1] = x.y;
          v[4 * k + 2] = x.z;
          v[4 * k + 3] = x.w;
        }
        tmem_st32(T_Q + lane_off + 32 * grp, v);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&bars->qo_full);
      const int64_t vr = vec_row(g, w.bh, w.i, w.r0 / BT) + row;
      const bool vr_ok = RA_CHECK_RANGE(p.chk, SITE_DQ_VEC, vr, 1, p.vec_rows);
      const float nl = vr_ok ? p.nlse2[vr] : -INFINITY;   // -inf past the block end: P = 0
      const float2 nl2 = make_float2(nl, nl);
      const float ndv = vr_ok ? p.ndvec[vr] : 0.f;
      const float2 nd2 = make_float2(ndv, ndv);
      for (int s = 0; s < g.N && ok; ++s) {
        const int j = ring_block(w.i, s, g.N);
        if (!block_visited(g, w.i, j)) continue;
        const int last = kt_last(g, w.i, j, w.r0);
        const int lim = key_limit(g, w.i, j, rq);
        for (int kt = 0; kt <= last && ok; ++kt) {
          // P from S as soon as S is ready (the dP MMA may still be running)
          if (!(ok = mbar_wait(&bars->s_full, s_ph, wc, ST_BWD_WAIT | 0x18))) break;
          s_ph ^= 1;
          tc_fence_after();
          uint32_t pv[64];
          tmem_ld32(T_S + lane_off + 64 * grp, pv);
          tmem_ld32(T_S + lane_off + 64 * grp + 32, pv + 32);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bars->s_free);
          const int rk0 = kt * BT + 64 * grp;                // first key row handled here
#pragma unroll
          for (int c = 0; c < 64; c += 2) {   // exponent arguments two at a time (packed f32x2 FMA)
            const float2 a = __ffma2_rn(make_float2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])), sl2v, nl2);
            pv[c] = __float_as_uint(hw_exp2(a.x));
            pv[c + 1] = __float_as_uint(hw_exp2(a.y));
          }
          if (tile_masked(g, w.i, j, kt, w.r0)) {            // diagonal or ragged tile only
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (rk0 + c >= lim) pv[c] = 0u;
          }
          if (!(ok = mbar_wait(&bars->dp_full, dp_ph, wc, ST_BWD_WAIT | 0x1f))) break;
          dp_ph ^= 1;
          tc_fence_after();
          uint32_t dpv[64];
          tmem_ld32(T_DP + lane_off + 64 * grp, dpv);
          tmem_ld32(T_DP + lane_off + 64 * grp + 32, dpv + 32);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bars->dp_free);
          uint32_t dk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {   // dS = P (dP - D_vec), two lanes at a time
            const float2 ds = __fmul2_rn(make_float2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])),
                                         __fadd2_rn(make_float2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])),
                                                    nd2));
            dk[c >> 1] = pack_bf16x2(ds.x, ds.y);
          }
          if (!first_ds) {   // the dS region: the previous tile's dQ MMAs must have read it
            if (!(ok = mbar_wait(&bars->ds_free, dsf_ph, wc, ST_BWD_WAIT | 0x20))) break;
            dsf_ph ^= 1;
            tc_fence_after();
          }
          first_ds = false;
          tmem_st32(T_DS + lane_off + 32 * grp, dk);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->p_full);
        }
      }
      if (!ok) break;
      // ---- epilogue: this group's 64 columns of the dQ row, / sqrt(d)
      if (!(ok = mbar_wait(&bars->dq_full, dq_ph, wc, ST_BWD_WAIT | 0x19))) break;
      dq_ph ^= 1;
      tc_fence_after();
      const bool st_ok =
          rq < g.c && RA_CHECK_RANGE(p.chk, SITE_DQ_OUT, grow * HD + grp * 64, 64, p.BH * p.S * HD);
      if (p.accumulate)
        add_row_f32(T_DQ + lane_off + grp * 64, p.dQf + grow * HD + grp * 64, p.inv_sqrt_d, st_ok, 64);
      else
        store_row_bf16(T_DQ + lane_off + grp * 64, p.dQ + grow * HD + grp * 64, p.inv_sqrt_d, st_ok, 64);
      tc_fence_before();
      mbar_arrive(&bars->dq_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  clock_mark(p.clk, 1);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
}  // namespace q

// One warp per padded query row: writes -D_vec = -sum_d dO*O and -LSE*log2(e)
// (0 and -inf for rows past the block end or with LSE = -inf), negated so the
// main kernels add them with packed f32x2 FMAs and adds.
__global__ void __launch_bounds__(256) prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                   const __nv_bfloat16* __restrict__ dO, const float* __restrict__ LSE,
                                                   float* nlse2, float* ndvec, RingGeom g, int S, int64_t rows,
                                                   int64_t n_rows, CheckRec* chk) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;
  const int r = static_cast<int>(w % BT);
  const int64_t t1 = w / BT;
  const int qt = static_cast<int>(t1 % g.n_mb);
  const int64_t t2 = t1 / g.n_mb;
  const int i = static_cast<int>(t2 % g.N);
  const int64_t bh = t2 / g.N;
  const int lr = qt * BT + r;
  float dv = 0.f, l2 = INFINITY;   // D_vec and LSE*log2(e)
  if (lr < g.c && RA_CHECK_RANGE(chk, SITE_PREP_IN, (bh * S + static_cast<int64_t>(i) * g.c + lr) * HD + lane * 4, 4,
                                 n_rows * HD) &&
      RA_CHECK_RANGE(chk, SITE_PREP_LSE, bh * S + static_cast<int64_t>(i) * g.c + lr, 1, n_rows)) {
    const int64_t row = bh * S + static_cast<int64_t>(i) * g.c + lr;
    const uint2 a = *reinterpret_cast<const uint2*>(O + row * HD + lane * 4);
    const uint2 b = *reinterpret_cast<const uint2*>(dO + row * HD + lane * 4);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 fa = __bfloat1622float2(a2[k]);
      const float2 fb = __bfloat1622float2(b2[k]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    dv = acc;
    const float l = LSE[row];
    l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
  }
  if (lane == 0 && RA_CHECK_RANGE(chk, SITE_PREP_OUT, w, 1, rows)) {
    nlse2[w] = -l2;
    ndvec[w] = -dv;
  }
}

}  // namespace bwd

cudaError_t launch_bwd_bf16(const BwdArgs& a, const void* tmap_q, const void* tmap_k, const void* tmap_v,
                            const void* tmap_do) {
  using namespace bwd;
  Params p;
  p.g.N = static_cast<int>(a.N);
  p.g.c = static_cast<int>(a.S / a.N);
  p.g.causal = a.causal;
  p.g.striped = a.striped;
  p.g.strict = a.strict;
  p.g.kt_w = BT;
  p.g.n_kt = (p.g.c + BT - 1) / BT;
  p.g.mb_h = BT;
  p.g.n_mb = p.g.n_kt;
  p.S = static_cast<int>(a.S);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
  p.inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a.D)));
  p.nlse2 = a.nlse2;
  p.ndvec = a.ndvec;
  p.accumulate = a.accumulate;
  p.dQ = a.accumulate ? nullptr : static_cast<__nv_bfloat16*>(a.dQ);
  p.dK = a.accumulate ? nullptr : static_cast<__nv_bfloat16*>(a.dK);
  p.dV = a.accumulate ? nullptr : static_cast<__nv_bfloat16*>(a.dV);
  p.dQf = a.accumulate ? static_cast<float*>(a.dQ) : nullptr;
  p.dKf = a.accumulate ? static_cast<float*>(a.dK) : nullptr;
  p.dVf = a.accumulate ? static_cast<float*>(a.dV) : nullptr;
  p.status = a.status;
  p.BH = a.B * a.H;
  p.chk = a.chk;
  const CUtensorMap& mq = *static_cast<const CUtensorMap*>(tmap_q);
  const CUtensorMap& mk = *static_cast<const CUtensorMap*>(tmap_k);
  const CUtensorMap& mv = *static_cast<const CUtensorMap*>(tmap_v);
  const CUtensorMap& mdo = *static_cast<const CUtensorMap*>(tmap_do);

  const int64_t prow = a.B * a.H * a.N * p.g.n_mb * BT;   // padded query rows
  p.vec_rows = prow;
  if (a.ev) cudaEventRecord(a.ev[0], a.stream);
  prep_kernel<<<static_cast<unsigned>((prow * 32 + 255) / 256), 256, 0, a.stream>>>(
      static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.LSE, a.nlse2, a.ndvec, p.g,
      p.S, prow, a.B * a.H * a.S, a.chk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  e = raise_smem_limit(reinterpret_cast<const void*>(kv::dkv_kernel), kv::SMEM_BYTES);
  if (e == cudaSuccess) e = raise_smem_limit(reinterpret_cast<const void*>(q::dq_kernel), q::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t units = a.B * a.H * a.N * p.g.n_kt;   // KV tiles = query tiles
  p.num_units = units;
  const int grid = static_cast<int>(units < a.num_sms ? units : a.num_sms);
  if (a.ev) cudaEventRecord(a.ev[1], a.stream);
  p.clk = a.clk_dkv;
  kv::dkv_kernel<<<grid, THREADS, kv::SMEM_BYTES, a.stream>>>(mq, mk, mv, mdo, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.ev) cudaEventRecord(a.ev[2], a.stream);
  p.clk = a.clk_dq;
  q::dq_kernel<<<grid, THREADS, q::SMEM_BYTES, a.stream>>>(mk, mv, mdo, static_cast<const __nv_bfloat16*>(a.Q), p);
  e = cudaGetLastError();
  if (a.ev) cudaEventRecord(a.ev[3], a.stream);
  return e;
}

}  // namespace ra
