// probe.cu -- issue-rate probe of the 5th-generation tensor core (measurement
// aid behind ra_probe_mma; not part of the attention path).
//
// One CTA per SM: one thread issues `iters` tcgen05.mma kind::f16 (M = 128,
// K = 16, bf16 in, f32 accumulate) back to back into one TMEM accumulator,
// eight per loop trip over the K-slices of a 128-deep tile (as the attention
// kernels issue them), commits, waits, and records clock64.  A comes from
// shared memory (SS) or from TMEM (TS); B always from shared memory
// (K-major, 128-byte swizzle).
// Operands are small pseudo-random bf16 values.  With `switch_every` = k > 0
// the instructions alternate between two accumulators every k MMAs (as a
// kernel does when it interleaves two tiles' GEMMs).  The kernels of this
// library are shaped by what this measures: the clocks an MMA instruction of
// each width costs, and what switching accumulators adds.  `variant` adds,
// per group of eight MMAs, the steps a kernel's MMA thread takes between
// groups: bit 0 accumulate flag computed at run time; bit 1 a commit to an
// mbarrier; bit 2 a wait on an already completed mbarrier and a tcgen05
// fence; bit 3 (with bit 1) waiting for the group issued two groups earlier
// to complete; bit 4 (with bit 1) waiting for the previous group; bit 5
// issues from the whole warp with one elected lane instead of one thread.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ra {
namespace probe {

constexpr int THREADS = 128;
constexpr uint32_t BOX = 128 * 64 * 2;       // 128 rows x 64 K (bf16), 128B-swizzled
constexpr uint32_t A_BYTES = 2 * BOX;         // 128 rows x 128 K: two boxes
constexpr uint32_t B_BYTES = 4 * BOX;         // up to 256 rows x 128 K
constexpr uint32_t SMEM_BYTES = A_BYTES + B_BYTES + 1024;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int kMaxCtas = 1024;

__device__ unsigned long long g_clk[kMaxCtas];

// K-slice kk (16 wide) of a 128-deep K-major tile stored as 64-column boxes
// of `box` bytes each.
__device__ __forceinline__ uint64_t kslice(uint64_t d0, int kk, uint32_t box) {
  return sdesc_add(d0, (kk >> 2) * box + (kk & 3) * 32);
}

// Pseudo-random bf16 bit pairs in [-1, 1) (a 32-bit integer hash of the index).
__device__ __forceinline__ uint32_t noise_bf16x2(uint32_t i) {
  uint32_t h = i * 0x9E3779B1u;
  h ^= h >> 15;
  h *= 0x2C1B3C6Du;
  h ^= h >> 12;
  const uint32_t lo = 0x3F80u | ((h & 0x7Fu) << 0) | ((h & 0x80u) << 8);   // +-[1, 2) with a random mantissa
  const uint32_t hi = 0x3F00u | ((h >> 8) & 0x7Fu) | (((h >> 15) & 1u) << 15);   // +-[0.5, 1)
  return lo | (hi << 16);
}

// WARP: the whole warp 0 runs the issue loop (warp-uniform operands) and one
// elected lane issues each tcgen05 instruction; otherwise thread 0 alone.
template <bool TS, bool WARP>
__global__ void __launch_bounds__(THREADS, 1) mma_kernel(int n, int iters, int switch_every, int variant,
                                                         unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t bar, done_bar, grp_bar[4];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(status, 0u, ST_PROBE_WAIT | 0xff);
    return;
  }
  for (uint32_t i = threadIdx.x * 16; i < A_BYTES + B_BYTES; i += THREADS * 16)
    *reinterpret_cast<uint4*>(smem + i) = make_uint4(noise_bf16x2(i), noise_bf16x2(i + 4), noise_bf16x2(i + 8),
                                                     noise_bf16x2(i + 12));
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init(&done_bar, 1);
    for (int g = 0; g < 4; ++g) mbar_init(&grp_bar[g], 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_arrive(&done_bar);       // phase 0 complete: waits on it return at once
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // zeroed smem visible to the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t t_a = tmem + 256;              // TS: A operand, 8 K-slices x 8 columns
  if (TS) {                                     // fill the TMEM A operand: each warp its lane quadrant
    uint32_t z[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) z[k] = noise_bf16x2(threadIdx.x * 64 + k);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    tmem_st32(t_a + lane_off, z);
    tmem_st32(t_a + 32 + lane_off, z);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (WARP ? warp == 0 : threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(n), 0, 0);
    const uint64_t a0 = sdesc(sbase, 16, 1024, SWZ_128B);
    const uint64_t b0 = sdesc(sbase + A_BYTES, 16, 1024, SWZ_128B);
    const uint32_t b_box = static_cast<uint32_t>(n) * 128;   // one 64-column box of B (n rows)
    const WaitCtx wg{&abort_flag, status, WAIT_LIMIT_NS};
    const long long t0 = clock64();
    int since = 0;
    uint32_t d = tmem;
    bool ok_g = true;
    for (int i = 0, g = 0; i < iters && ok_g; i += 8, ++g) {
      const int dep = (variant & 8) ? 2 : ((variant & 16) ? 1 : 0);
      if ((variant & 2) && dep && g >= dep) {   // the group issued `dep` groups earlier has completed
        const int h = g - dep;
        ok_g = mbar_wait(&grp_bar[h & 3], (h >> 2) & 1, wg, ST_PROBE_WAIT | 2);
        tc_fence_after();
      }
      if (variant & 4) {
        ok_g = ok_g && mbar_wait(&done_bar, 0, wg, ST_PROBE_WAIT | 3);
        tc_fence_after();
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t acc = (variant & 1) ? static_cast<uint32_t>((kk > 0) | (i > 0)) : 1u;
        if (WARP) {
          if (TS)
            mma_ts_w(d, t_a + kk * 8, kslice(b0, kk, b_box), idesc, acc);
          else
            mma_ss_w(d, kslice(a0, kk, BOX), kslice(b0, kk, b_box), idesc, acc);
        } else if (TS) {
          mma_ts(d, t_a + kk * 8, kslice(b0, kk, b_box), idesc, acc);
        } else {
          mma_ss(d, kslice(a0, kk, BOX), kslice(b0, kk, b_box), idesc, acc);
        }
        if (switch_every && ++since == switch_every) {   // the other accumulator: columns [128, 256)
          since = 0;
          d ^= 128u;
        }
      }
      if (variant & 2) {
        if (WARP)
          mma_commit_w(&grp_bar[g & 3]);
        else
          mma_commit(&grp_bar[g & 3]);
      }
    }
    if (WARP)
      mma_commit_w(&bar);
    else
      mma_commit(&bar);
    const WaitCtx wc{&abort_flag, status, WAIT_LIMIT_NS};
    const bool ok = mbar_wait(&bar, 0, wc, ST_PROBE_WAIT | 1);
    if (!ok) mbar_drain(&bar, 0, 200000000ull);
    const long long t1 = clock64();
    if (blockIdx.x < kMaxCtas && (threadIdx.x & 31) == 0)
      g_clk[blockIdx.x] = ok ? static_cast<unsigned long long>(t1 - t0) : 0ull;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace probe

cudaError_t launch_probe_mma(int ts, int n, int iters, int switch_every, int variant, int num_sms,
                             unsigned int* status, double* clk_per_mma) {
  static bool attr_done = false;
  cudaError_t e;
  if (!attr_done) {
    e = cudaFuncSetAttribute(probe::mma_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             probe::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(probe::mma_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               probe::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(probe::mma_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               probe::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(probe::mma_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               probe::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  iters = (iters + 7) / 8 * 8;   // whole tiles of 8 K-slices
  const int grid = num_sms < probe::kMaxCtas ? num_sms : probe::kMaxCtas;
  const bool warp_wide = (variant & 32) != 0;
  variant &= 31;
  if (ts && warp_wide)
    probe::mma_kernel<true, true><<<grid, probe::THREADS, probe::SMEM_BYTES>>>(n, iters, switch_every, variant, status);
  else if (ts)
    probe::mma_kernel<true, false><<<grid, probe::THREADS, probe::SMEM_BYTES>>>(n, iters, switch_every, variant, status);
  else if (warp_wide)
    probe::mma_kernel<false, true><<<grid, probe::THREADS, probe::SMEM_BYTES>>>(n, iters, switch_every, variant, status);
  else
    probe::mma_kernel<false, false><<<grid, probe::THREADS, probe::SMEM_BYTES>>>(n, iters, switch_every, variant, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return e;
  unsigned long long clk[probe::kMaxCtas];
  if ((e = cudaMemcpyFromSymbol(clk, probe::g_clk, sizeof(unsigned long long) * grid)) != cudaSuccess) return e;
  double sum = 0.0;
  int good = 0;
  for (int i = 0; i < grid; ++i)
    if (clk[i]) {
      sum += static_cast<double>(clk[i]);
      ++good;
    }
  *clk_per_mma = good ? sum / good / iters : -1.0;
  return cudaSuccess;
}

}  // namespace ra
