// ffn.cu -- blockwise gated feedforward on the tensor cores.
//
// "Ring Attention with Blockwise Transformers for Near Infinite Context"
// reading notes: the feedforward acts on each host's own block only and runs
// blockwise, so its largest activation is bounded per block (§5.2, §5.3); the
// experiments use LLaMA-style models, whose feedforward is gated:
//     Y = (silu(X W1^T) * (X W3^T)) W2^T,   W1, W3: [f, h],  W2: [h, f].
// A call processes the T rows of X in blocks of `block_rows`; per block two
// launches of one GEMM kernel (C = A B^T, both operands K-major bf16):
//   up:   H = silu(X W1^T) * (X W3^T)   -- B tile = 128 rows of W1 followed by
//         the same 128 rows of W3, so one N=256 MMA computes both halves and
//         the epilogue pairs them column by column;
//   down: Y = H W2^T                    -- B tile = 256 rows of W2.
// H (block_rows x f, bf16) is the only intermediate: the caller's workspace.
//
// Consecutive launches of one call overlap (programmatic dependent launch):
// every launch after the first may start on SMs the previous one has left,
// e.g. during the down GEMM's last partial wave.  The up GEMM computes at once
// and waits for the previous grid only before its first store into H (which
// the previous down GEMM reads); the down GEMM waits before it loads H.
//
// Kernel: persistent, one CTA per SM, 192 threads.  Warp 0 (one thread) loads
// A and B K-chunks of 64 columns with TMA into a 4-stage ring (48 KB a stage,
// 128-byte swizzle); warp 1 (the whole warp, one elected lane issuing) issues
// tcgen05.mma M=128 N=256 K=16 into one of two TMEM accumulators (256 columns
// each) and commits; warps 2-5
// drain the other accumulator (one thread per row) while the next tile's
// MMAs run.  Tiles are handed out dynamically (an atomic counter per launch,
// taken by the TMA thread and passed to the MMA and epilogue warps through a
// small shared-memory ring), numbered M-fastest so the CTAs working at the
// same time share the B (weight) tiles in L2 and A stays resident; a CTA that
// starts early (while the previous launch drains) simply takes more tiles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace ra {
namespace ffn {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;                  // 16 KB: one 64-column box
constexpr uint32_t B_BYTES = BN * BK * 2;                  // 32 KB: two 128-row boxes
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr int THREADS = 192;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;          // 2 s
constexpr float LOG2E = 1.4426950408889634f;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, 0, 0);
constexpr int TSLOTS = 4;                                  // tile ids in flight per CTA

struct Bars {
  uint64_t full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain;
  uint64_t tid_full[TSLOTS], tid_empty[TSLOTS];
  int tile_id[TSLOTS];
  uint32_t tmem_base;
  int abort;
};

struct Params {
  int m_tiles, n_tiles, k_chunks;
  int M;                 // valid rows of A / the output
  int b_row_step;        // B-map rows per N tile: 128 (gated) or 256 (plain)
  int b1_row_off;        // row of the second B box inside the tile: 0 (gated, W3 map) or 128 (plain)
  int gated;
  __nv_bfloat16* out;    // row-major, leading dimension ldo
  int64_t ldo;
  int* tile_counter;     // zero before the launch
  unsigned int* status;
  int K, b_rows;         // A and B maps: K columns; B map rows (W1/W3: f, W2: h)
  CheckRec* chk;
};

__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) { return sdesc(saddr, 16, 1024, SWZ_128B); }

// Programmatic dependent launch: let the next grid of the stream be scheduled,
// and wait until the previous grid has completed and its writes are visible
// (both no-ops when the launch did not opt in).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_previous() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float silu_times(float a, float b) {
  return a * __frcp_rn(1.f + hw_exp2(-a * LOG2E)) * b;
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
            const __grid_constant__ CUtensorMap tmB1, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, ST_FFN_WAIT | 0xff);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], 128);
    }
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < TSLOTS; ++s) {
      mbar_init(&bars->tid_full[s], 1);
      mbar_init(&bars->tid_empty[s], 1 + 128);   // one lane of the MMA warp and the 128 epilogue threads
    }
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
  pdl_launch_dependents();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtx wc{&bars->abort, p.status, WAIT_LIMIT_NS};
  const int tiles = p.m_tiles * p.n_tiles;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB0);
      tma_prefetch_desc(&tmB1);
      if (!p.gated) pdl_wait_previous();       // A (= H) is the previous grid's output
      uint32_t it = 0;
      bool ok = true;
      for (uint32_t lt = 0; ok; ++lt) {
        int t = atomicAdd(p.tile_counter, 1);
        if (t >= tiles) t = -1;                  // no tile left: tell the other roles to stop
        const int slot = lt % TSLOTS;
        if (!(ok = mbar_wait(&bars->tid_empty[slot], ((lt / TSLOTS) & 1) ^ 1, wc, ST_FFN_WAIT | 5))) break;
        bars->tile_id[slot] = t;
        mbar_arrive(&bars->tid_full[slot]);
        if (t < 0) break;
        const int m = t % p.m_tiles, n = t / p.m_tiles;
        for (int kc = 0; kc < p.k_chunks; ++kc, ++it) {
          const int st = it % STAGES;
          if (!(ok = mbar_wait(&bars->empty[st], ((it / STAGES) & 1) ^ 1, wc, ST_FFN_WAIT | 1))) break;
          mbar_arrive_expect_tx(&bars->full[st], STAGE_BYTES);
          uint8_t* s = smem + st * STAGE_BYTES;
          if (RA_CHECK_BOX(p.chk, SITE_FFN_TMA, kc * BK, m * BM, 0, p.K, p.M, 1, 8))
            tma_load_3d(s, &tmA, &bars->full[st], kc * BK, m * BM, 0);
          if (RA_CHECK_BOX(p.chk, SITE_FFN_TMA, kc * BK, n * p.b_row_step, 0, p.K, p.b_rows, 1, 8))
            tma_load_3d(s + A_BYTES, &tmB0, &bars->full[st], kc * BK, n * p.b_row_step, 0);
          if (RA_CHECK_BOX(p.chk, SITE_FFN_TMA, kc * BK, n * p.b_row_step + p.b1_row_off, 0, p.K, p.b_rows, 1, 8))
            tma_load_3d(s + A_BYTES + B_BYTES / 2, &tmB1, &bars->full[st], kc * BK, n * p.b_row_step + p.b1_row_off,
                        0);
        }
      }
      for (uint32_t k = (it > STAGES ? it - STAGES : 0); k < it; ++k)
        mbar_drain(&bars->full[k % STAGES], (k / STAGES) & 1, 200000000ull);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // The whole warp runs the issue loop (warp-uniform operands); one elected
    // lane issues each tcgen05 instruction.
    {
      uint32_t it = 0;
      bool ok = true;
      for (uint32_t lt = 0; ok; ++lt) {
        const int slot = lt % TSLOTS;
        if (!(ok = mbar_wait_w(&bars->tid_full[slot], (lt / TSLOTS) & 1, wc, ST_FFN_WAIT | 6))) break;
        const int t = bars->tile_id[slot];
        if (lane == 0) mbar_arrive(&bars->tid_empty[slot]);   // one of the 129 arrivals
        if (t < 0) break;
        const uint32_t buf = lt & 1;
        if (!(ok = mbar_wait_w(&bars->acc_empty[buf], ((lt >> 1) & 1) ^ 1, wc, ST_FFN_WAIT | 2))) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int kc = 0; kc < p.k_chunks; ++kc, ++it) {
          const int st = it % STAGES;
          if (!(ok = mbar_wait_w(&bars->full[st], (it / STAGES) & 1, wc, ST_FFN_WAIT | 3))) break;
          tc_fence_after();
          const uint64_t a0 = kdesc(sbase + st * STAGE_BYTES);
          const uint64_t b0 = kdesc(sbase + st * STAGE_BYTES + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_ss_w(d, sdesc_add(a0, kk * 32), sdesc_add(b0, kk * 32), IDESC, (kc | kk) != 0);
          mma_commit_w(&bars->empty[st]);
        }
        if (!ok) break;
        mma_commit_w(&bars->acc_full[buf]);
      }
      mma_commit_w(&bars->drain);
      mbar_drain(&bars->drain, 0, 200000000ull);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int quad = warp & 3;                       // TMEM lane quadrant of this warp
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    if (p.gated) pdl_wait_previous();          // the previous grid may still read the out buffer (H)
    for (uint32_t lt = 0;; ++lt) {
      const int slot = lt % TSLOTS;
      if (!mbar_wait(&bars->tid_full[slot], (lt / TSLOTS) & 1, wc, ST_FFN_WAIT | 7)) break;
      const int t = bars->tile_id[slot];
      mbar_arrive(&bars->tid_empty[slot]);
      if (t < 0) break;
      const int m = t % p.m_tiles, n = t / p.m_tiles;
      const uint32_t buf = lt & 1;
      if (!mbar_wait(&bars->acc_full[buf], (lt >> 1) & 1, wc, ST_FFN_WAIT | 4)) break;
      tc_fence_after();
      const int row = m * BM + quad * 32 + lane;
      [[maybe_unused]] const int64_t out_cols = p.gated ? 128 : BN;
      const bool ok = row < p.M && RA_CHECK_RANGE(p.chk, SITE_FFN_OUT, static_cast<int64_t>(row) * p.ldo + n * out_cols,
                                                  out_cols, static_cast<int64_t>(p.M) * p.ldo);
      const uint32_t acc = tmem + buf * BN + lane_off;
      if (p.gated) {
        __nv_bfloat16* dst = p.out + static_cast<int64_t>(row) * p.ldo + static_cast<int64_t>(n) * 128;
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t g[32], u[32], pk[16];
          tmem_ld32(acc + ch * 32, g);
          tmem_ld32(acc + 128 + ch * 32, u);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack_bf16x2(silu_times(__uint_as_float(g[2 * k]), __uint_as_float(u[2 * k])),
                                silu_times(__uint_as_float(g[2 * k + 1]), __uint_as_float(u[2 * k + 1])));
          if (ok) {
            uint4* o4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) o4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else {
        __nv_bfloat16* dst = p.out + static_cast<int64_t>(row) * p.ldo + static_cast<int64_t>(n) * BN;
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t v32[32], pk[16];
          tmem_ld32(acc + ch * 32, v32);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k) pk[k] = pack_bf16x2(__uint_as_float(v32[2 * k]), __uint_as_float(v32[2 * k + 1]));
          if (ok) {
            uint4* o4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) o4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace ffn

cudaError_t launch_ffn_gemm(const FfnGemmArgs& a, const void* tmap_a, const void* tmap_b0, const void* tmap_b1) {
  {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(ffn::gemm_kernel), ffn::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  ffn::Params p;
  p.m_tiles = static_cast<int>((a.M + ffn::BM - 1) / ffn::BM);
  p.n_tiles = static_cast<int>(a.gated ? a.N / 128 : a.N / ffn::BN);
  p.k_chunks = static_cast<int>(a.K / ffn::BK);
  p.M = static_cast<int>(a.M);
  p.b_row_step = a.gated ? 128 : ffn::BN;
  p.b1_row_off = a.gated ? 0 : 128;
  p.gated = a.gated;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.ldo = a.ldo;
  p.tile_counter = a.tile_counter;
  p.status = a.status;
  p.K = static_cast<int>(a.K);
  p.b_rows = static_cast<int>(a.N);
  p.chk = a.chk;
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  const int grid = static_cast<int>(tiles < a.num_sms ? tiles : a.num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(ffn::THREADS);
  cfg.dynamicSmemBytes = ffn::SMEM_BYTES;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, ffn::gemm_kernel, *static_cast<const CUtensorMap*>(tmap_a),
                            *static_cast<const CUtensorMap*>(tmap_b0), *static_cast<const CUtensorMap*>(tmap_b1), p);
}

}  // namespace ra
