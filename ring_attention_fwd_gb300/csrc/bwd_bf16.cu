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
// Three launches:
//   1. prep_kernel   D_vec and LSE*log2(e) per query row, stored per 128-row
//                    query tile (rows past a block's end get D_vec = 0 and
//                    +inf, so they drop out of P by themselves); zero the f32
//                    dQ accumulator.
//   2. bwd_kernel    one persistent CTA per SM; a work unit is one 128-row KV
//                    tile of one head, stationary in shared memory and with
//                    dK, dV accumulating in TMEM.  KV block j travels the ring
//                    to hosts j, j+1, ... so the unit visits the query tiles
//                    of blocks i = j, j+1, ... (mod N) that see it.  Per query
//                    tile:  S^T = K Q^T and dP^T = V dO^T (tensor cores),
//                    P^T and dS^T by 4 softmax warps (one thread per key row),
//                    dV += P^T dO, dK += dS^T Q, dQ^T = K^T dS^T (tensor
//                    cores), then dQ^T is added into the f32 accumulator with
//                    coalesced reductions.
//   3. dq_kernel     dQ = accumulator / sqrt(d) -> bf16.
// TMEM columns: dV [0,128) dK [128,256) S^T/P^T [256,384) dP^T/dQ^T [384,512).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace ra {
namespace bwd {

constexpr int BT = 128;        // rows per KV tile and per query tile
constexpr int HD = 128;
constexpr int THREADS = 256;   // warp 0 TMA, warp 1 MMA, warps 4-7 softmax / dQ / epilogue
constexpr int NSTAGE = 2;
constexpr uint32_t TILE_BYTES = BT * HD * 2;  // 32 KB
constexpr uint32_t BOX_BYTES = TILE_BYTES / 2;
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + TILE_BYTES;
constexpr uint32_t OFF_Q = OFF_V + TILE_BYTES;                  // NSTAGE tiles
constexpr uint32_t OFF_DO = OFF_Q + NSTAGE * TILE_BYTES;        // NSTAGE tiles
constexpr uint32_t OFF_DS = OFF_DO + NSTAGE * TILE_BYTES;       // dS^T tile
constexpr uint32_t OFF_VEC = OFF_DS + TILE_BYTES;               // NSTAGE x (lse2[128], dvec[128])
constexpr uint32_t VEC_BYTES = BT * 4;
constexpr uint32_t OFF_BAR = OFF_VEC + NSTAGE * 2 * VEC_BYTES;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

struct Bars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[NSTAGE], q_empty[NSTAGE];
  uint64_t s_full, p_full, dq_full, dq_empty, dkv_full, dkv_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Params {
  RingGeom g;        // kt_w = 128 (KV tile), mb_h = 128 (query tile)
  int S;
  int64_t num_units;
  float scale_log2;  // log2(e) / sqrt(D)
  float inv_sqrt_d;
  const float* lse2;   // [BH][N][n_qt][128]
  const float* dvec;   // [BH][N][n_qt][128]
  float* dq_acc;       // [BH][S][128]
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  unsigned int* status;
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

// Query blocks visited by KV block j: i = j + s (mod N), s = 0..N-1; the
// contiguous causal sweep never reaches blocks i < j.
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

__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int kk) {   // K-major operand, K-slice kk
  return sdesc(tile + (kk >> 2) * BOX_BYTES + (kk & 3) * 32, 16, 1024, SWZ_128B);
}
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int kk) {  // MN-major operand, K-slice kk
  return sdesc(tile + kk * 16 * 128, BOX_BYTES, 1024, SWZ_128B);
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const RingGeom& g = p.g;
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, ST_BWD_WAIT | 0xff);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, 128);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->dkv_empty, 128);
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
  const uint32_t T_DV = tmem, T_DK = tmem + 128, T_S = tmem + 256, T_DP = tmem + 384;
  const WaitCtx wc{&bars->abort, p.status, WAIT_LIMIT_NS};
  const int grid = gridDim.x, cta = blockIdx.x;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      uint32_t it = 0, nkv = 0, kve_ph = 0;
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
          tma_load_3d(smem + OFF_K + h * BOX_BYTES, &tmK, &bars->kv_full, h * 64, krow, bh);
          tma_load_3d(smem + OFF_V + h * BOX_BYTES, &tmV, &bars->kv_full, h * 64, krow, bh);
        }
        ++nkv;
        for (int s = 0; s < g.N && ok; ++s) {
          const int i = (j + s) % g.N;
          if (!q_block_visited(g, i, j)) continue;
          for (int qt = qt_first(g, i, j, kt); qt < g.n_mb; ++qt, ++it) {
            const int st = it % NSTAGE;
            const uint32_t ph = (it / NSTAGE) & 1;
            if (!(ok = mbar_wait(&bars->q_empty[st], ph ^ 1, wc, ST_BWD_WAIT | 2))) break;
            mbar_arrive_expect_tx(&bars->q_full[st], 2 * TILE_BYTES + 2 * VEC_BYTES);
            const int qrow = i * g.c + qt * BT;
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(smem + OFF_Q + st * TILE_BYTES + h * BOX_BYTES, &tmQ, &bars->q_full[st], h * 64, qrow, bh);
              tma_load_3d(smem + OFF_DO + st * TILE_BYTES + h * BOX_BYTES, &tmDO, &bars->q_full[st], h * 64, qrow,
                          bh);
            }
            const int64_t vrow = ((static_cast<int64_t>(bh) * g.N + i) * g.n_mb + qt) * BT;
            bulk_load(smem + OFF_VEC + st * 2 * VEC_BYTES, p.lse2 + vrow, VEC_BYTES, &bars->q_full[st]);
            bulk_load(smem + OFF_VEC + st * 2 * VEC_BYTES + VEC_BYTES, p.dvec + vrow, VEC_BYTES, &bars->q_full[st]);
          }
        }
      }
      if (!ok) {
        for (uint32_t k = (it > NSTAGE ? it - NSTAGE : 0); k < it; ++k)
          mbar_drain(&bars->q_full[k % NSTAGE], (k / NSTAGE) & 1, 200000000ull);
        if (nkv > 0) mbar_drain(&bars->kv_full, (nkv - 1) & 1, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_KK = idesc_bf16_f32(BT, BT, 0, 0);   // A K-major, B K-major
      constexpr uint32_t ID_KM = idesc_bf16_f32(BT, HD, 0, 1);   // A K-major (or TMEM), B MN-major
      constexpr uint32_t ID_MM = idesc_bf16_f32(HD, BT, 1, 1);   // A MN-major, B MN-major
      const uint32_t sK = sbase + OFF_K, sV = sbase + OFF_V, sDS = sbase + OFF_DS;
      uint32_t it = 0, kv_ph = 0, pf_ph = 0, dqe_ph = 0, dkve_ph = 0;
      bool ok = true, first_unit = true, first_step = true;
      for (int64_t r = 0; ok; ++r) {
        const int64_t u = snake_pos(r, cta, grid);
        if (u >= p.num_units) break;
        int bh, j, kt;
        unit_at(g, u, bh, j, kt);
        const int T = unit_steps(g, j, kt);
        if (!(ok = mbar_wait(&bars->kv_full, kv_ph, wc, ST_BWD_WAIT | 3))) break;
        kv_ph ^= 1;
        for (int t = 0; t < T && ok; ++t, ++it) {
          const int st = it % NSTAGE;
          const uint32_t ph = (it / NSTAGE) & 1;
          const uint32_t sQ = sbase + OFF_Q + st * TILE_BYTES, sDO = sbase + OFF_DO + st * TILE_BYTES;
          if (t == 0) {
            if (!(ok = mbar_wait(&bars->q_full[st], ph, wc, ST_BWD_WAIT | 4))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) mma_ss(T_S, kdesc(sK, kk), kdesc(sQ, kk), ID_KK, kk > 0);
          }
          if (!first_step) {   // dP^T region still holds the previous dQ^T until drained
            if (!(ok = mbar_wait(&bars->dq_empty, dqe_ph, wc, ST_BWD_WAIT | 5))) break;
            dqe_ph ^= 1;
            tc_fence_after();
          }
          first_step = false;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) mma_ss(T_DP, kdesc(sV, kk), kdesc(sDO, kk), ID_KK, kk > 0);
          mma_commit(&bars->s_full);
          if (!(ok = mbar_wait(&bars->p_full, pf_ph, wc, ST_BWD_WAIT | 6))) break;
          pf_ph ^= 1;
          if (t == 0 && !first_unit) {
            if (!(ok = mbar_wait(&bars->dkv_empty, dkve_ph, wc, ST_BWD_WAIT | 7))) break;
            dkve_ph ^= 1;
          }
          tc_fence_after();
          const uint32_t acc = t > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)   // dV += P^T dO  (P^T from TMEM)
            mma_ts(T_DV, T_S + kk * 8, mndesc(sDO, kk), ID_KM, (kk > 0) | acc);
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)   // dK += dS^T Q
            mma_ss(T_DK, kdesc(sDS, kk), mndesc(sQ, kk), ID_KM, (kk > 0) | acc);
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)   // dQ^T = K^T dS^T
            mma_ss(T_DP, mndesc(sK, kk), mndesc(sDS, kk), ID_MM, kk > 0);
          mma_commit(&bars->dq_full);
          mma_commit(&bars->q_empty[st]);
          if (t + 1 < T) {   // next query tile's S^T (S region: P^T already consumed in order)
            const int nst = (it + 1) % NSTAGE;
            const uint32_t nph = ((it + 1) / NSTAGE) & 1;
            if (!(ok = mbar_wait(&bars->q_full[nst], nph, wc, ST_BWD_WAIT | 8))) break;
            tc_fence_after();
            const uint32_t nQ = sbase + OFF_Q + nst * TILE_BYTES;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) mma_ss(T_S, kdesc(sK, kk), kdesc(nQ, kk), ID_KK, kk > 0);
          }
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty);
        mma_commit(&bars->dkv_full);
        first_unit = false;
      }
      mma_commit(&bars->drain);
      mbar_drain(&bars->drain, 0, 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------- softmax / dQ / epilogue
    const int quad = warp & 3;
    const int t_row = quad * 32 + lane;                  // TMEM lane = key row (dQ^T: head-dim row)
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t it = 0, s_ph = 0, dq_ph = 0, dkv_ph = 0;
    bool ok = true;
    for (int64_t r = 0; ok; ++r) {
      const int64_t u = snake_pos(r, cta, grid);
      if (u >= p.num_units) break;
      int bh, j, kt;
      unit_at(g, u, bh, j, kt);
      const bool key_ok = kt * BT + t_row < g.c;
      for (int s = 0; s < g.N && ok; ++s) {
        const int i = (j + s) % g.N;
        if (!q_block_visited(g, i, j)) continue;
        const bool dtype_pair = diag_type(g, i, j);
        const int incl = diag_incl(g, i, j);
        for (int qt = qt_first(g, i, j, kt); qt < g.n_mb && ok; ++qt, ++it) {
          const int st = it % NSTAGE;
          if (!(ok = mbar_wait(&bars->q_full[st], (it / NSTAGE) & 1, wc, ST_BWD_WAIT | 9))) break;
          if (!(ok = mbar_wait(&bars->s_full, s_ph, wc, ST_BWD_WAIT | 10))) break;
          s_ph ^= 1;
          tc_fence_after();
          // query column r is visible to this key row iff r >= vis_lo
          int vis_lo = 0;
          if (!key_ok) vis_lo = BT;
          else if (dtype_pair && qt == kt) vis_lo = t_row + 1 - incl;
          const float* lse2 = reinterpret_cast<const float*>(smem + OFF_VEC + st * 2 * VEC_BYTES);
          const float* dvec = lse2 + BT;
          const uint32_t ds_row = sbase + OFF_DS + t_row * 128;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t sv[32], dpv[32];
            tmem_ld32(T_S + lane_off + ch * 32, sv);
            tmem_ld32(T_DP + lane_off + ch * 32, dpv);
            tmem_ld_wait();
            uint32_t pk[16], dk[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const int c0 = ch * 32 + k;
              float p0 = hw_exp2(fmaf(__uint_as_float(sv[k]), sl2, -lse2[c0]));
              float p1 = hw_exp2(fmaf(__uint_as_float(sv[k + 1]), sl2, -lse2[c0 + 1]));
              if (c0 < vis_lo) p0 = 0.f;
              if (c0 + 1 < vis_lo) p1 = 0.f;
              const float d0 = p0 * (__uint_as_float(dpv[k]) - dvec[c0]);
              const float d1 = p1 * (__uint_as_float(dpv[k + 1]) - dvec[c0 + 1]);
              pk[k >> 1] = pack_bf16x2(p0, p1);
              dk[k >> 1] = pack_bf16x2(d0, d1);
            }
            tmem_st16(T_S + lane_off + ch * 16, pk);
            // dS^T row, 128B-swizzled: 16-byte chunk q of box b at b*16K + row*128 + ((q ^ row%8) * 16)
            const uint32_t box = ds_row + (ch >> 1) * BOX_BYTES;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint32_t chunk = ((ch & 1) * 4 + q4) ^ (t_row & 7);
              st_shared_v4(box + chunk * 16, dk[4 * q4], dk[4 * q4 + 1], dk[4 * q4 + 2], dk[4 * q4 + 3]);
            }
          }
          tmem_st_wait();
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&bars->p_full);
          // ---- drain dQ^T (lane = head-dim index) into the f32 accumulator
          if (!(ok = mbar_wait(&bars->dq_full, dq_ph, wc, ST_BWD_WAIT | 11))) break;
          dq_ph ^= 1;
          tc_fence_after();
          const int qvalid = g.c - qt * BT;    // query rows of this tile inside block i
          float* acc = p.dq_acc + (static_cast<int64_t>(bh) * p.S + static_cast<int64_t>(i) * g.c + qt * BT) * HD + t_row;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t v[32];
            tmem_ld32(T_DP + lane_off + ch * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int q = ch * 32 + k;
              if (q < qvalid) atomicAdd(acc + static_cast<int64_t>(q) * HD, __uint_as_float(v[k]));
            }
          }
          tc_fence_before();
          mbar_arrive(&bars->dq_empty);
        }
      }
      if (!ok) break;
      // ---- epilogue: dV, dK rows of this KV tile
      if (!(ok = mbar_wait(&bars->dkv_full, dkv_ph, wc, ST_BWD_WAIT | 12))) break;
      dkv_ph ^= 1;
      tc_fence_after();
      const int64_t krow = static_cast<int64_t>(bh) * p.S + static_cast<int64_t>(j) * g.c + kt * BT + t_row;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t tcol = (which == 0 ? T_DV : T_DK) + lane_off;
        const float sc = which == 0 ? 1.f : p.inv_sqrt_d;
        __nv_bfloat16* out = (which == 0 ? p.dV : p.dK) + krow * HD;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tmem_ld32(tcol + ch * 32, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * sc, __uint_as_float(v[2 * k + 1]) * sc);
          if (key_ok) {
            uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->dkv_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// One warp per padded query row: D_vec = sum_d dO*O, lse2 = LSE*log2(e) (or
// D_vec = 0, lse2 = +inf for rows past the block end or with LSE = -inf), and
// zero that row of the dQ accumulator.
__global__ void __launch_bounds__(256) prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                   const __nv_bfloat16* __restrict__ dO, const float* __restrict__ LSE,
                                                   float* lse2, float* dvec, float* dq_acc, RingGeom g, int S,
                                                   int64_t rows) {
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
  float dv = 0.f, l2 = INFINITY;
  if (lr < g.c) {
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
    reinterpret_cast<float4*>(dq_acc + row * HD)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (lane == 0) {
    lse2[w] = l2;
    dvec[w] = dv;
  }
}

__global__ void __launch_bounds__(256) dq_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dQ,
                                                 float scale, int64_t n4) {
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n4;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(acc)[k];
    uint2 o;
    o.x = pack_bf16x2(v.x * scale, v.y * scale);
    o.y = pack_bf16x2(v.z * scale, v.w * scale);
    reinterpret_cast<uint2*>(dQ)[k] = o;
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
  p.g.kt_w = BT;
  p.g.n_kt = (p.g.c + BT - 1) / BT;
  p.g.mb_h = BT;
  p.g.n_mb = p.g.n_kt;
  p.S = static_cast<int>(a.S);
  p.num_units = a.B * a.H * a.N * p.g.n_kt;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
  p.inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a.D)));
  p.lse2 = a.lse2;
  p.dvec = a.dvec;
  p.dq_acc = a.dq_acc;
  p.dK = static_cast<__nv_bfloat16*>(a.dK);
  p.dV = static_cast<__nv_bfloat16*>(a.dV);
  p.status = a.status;

  const int64_t prow = a.B * a.H * a.N * p.g.n_mb * BT;   // padded query rows
  const int64_t pblocks = (prow * 32 + 255) / 256;
  prep_kernel<<<static_cast<unsigned>(pblocks), 256, 0, a.stream>>>(
      static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.LSE, a.lse2, a.dvec,
      a.dq_acc, p.g, p.S, prow);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  static bool attr_done = false;
  if (!attr_done) {
    e = cudaFuncSetAttribute(bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int grid = static_cast<int>(p.num_units < a.num_sms ? p.num_units : a.num_sms);
  bwd_kernel<<<grid, THREADS, SMEM_BYTES, a.stream>>>(*static_cast<const CUtensorMap*>(tmap_q),
                                                      *static_cast<const CUtensorMap*>(tmap_k),
                                                      *static_cast<const CUtensorMap*>(tmap_v),
                                                      *static_cast<const CUtensorMap*>(tmap_do), p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int64_t n4 = a.B * a.H * a.S * a.D / 4;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > static_cast<int64_t>(a.num_sms) * 16) blocks = static_cast<int64_t>(a.num_sms) * 16;
  dq_kernel<<<static_cast<unsigned>(blocks > 0 ? blocks : 1), 256, 0, a.stream>>>(
      a.dq_acc, static_cast<__nv_bfloat16*>(a.dQ), p.inv_sqrt_d, n4);
  return cudaGetLastError();
}

}  // namespace ra
