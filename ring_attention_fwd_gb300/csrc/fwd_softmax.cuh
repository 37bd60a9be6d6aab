// fwd_softmax.cuh -- the softmax warps of the bf16 forward kernels: the
// online-softmax update of one 128-row query tile per warpgroup, and the
// epilogue.  Shared by the one-CTA-per-SM kernel (fwd_bf16.cu) and the SM-pair
// kernel (fwd_bf16_pair.cu), which therefore compute the same values in the
// same order.
//
// Method ("Ring Attention" explainer, aiqz.cc, §分块注意力): per row, the running
// max m, denominator l and unnormalised O; for each score tile S the row max
// grows to m', P = exp(S - m'), l = l * exp(m - m') + rowsum(P), and O is
// rescaled by exp(m - m') before O += P V; at the end O / l and
// LSE = m + ln l.  Here, per thread (one row): S is read from TMEM, masked on
// diagonal and ragged tiles, P (bf16) is written back over S for the P.V MMA,
// and O is rescaled in TMEM only when the max grew by more than 2^8 (O and l
// then share a stale reference max, which cancels in O / l).  The arithmetic
// runs on pairs of scores (packed f32x2 FMA and add, three-input max).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace ra {
namespace fwdsm {

constexpr int BM = 128;        // rows per Q tile
constexpr int BN = 128;        // keys per KV tile
constexpr int HD = 128;        // head dim
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units: p <= 2^8 between rescales

// The softmax role of warps 2-9: warps 2-5 own Q tile 0, warps 6-9 Q tile 1,
// one thread per row; warp w reads TMEM lane quadrant w % 4.  TMEM columns:
// S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512).
//   p          the kernel's parameters (g, S, num_units, scale_log2, O, LSE,
//              timing, BH, chk, O_acc, LSE_acc);
//   s_full, o_full   this CTA's S-ready and O-ready barriers, one per tile;
//   slot, nslots     this CTA's (or CTA pair's) place in the snake over the units;
//   row_base   first row of this CTA's two tiles inside a unit;
//   timer      whether this thread keeps the per-(host, step) timing;
//   arrive_p(q), arrive_o(q)   P of tile q written / O of tile q read.
template <class P, class ArriveP, class ArriveO>
__device__ __forceinline__ void softmax_role(const P& p, uint64_t* s_full, uint64_t* o_full, uint32_t tmem, int warp,
                                             int lane, int slot, int nslots, int row_base, bool timer,
                                             const WaitCtx& wc, ArriveP arrive_p, ArriveO arrive_o) {
  const RingGeom& g = p.g;
  const int q = (warp - 2) >> 2;         // Q tile 0 or 1
  const int quad = warp & 3;             // TMEM lane quadrant of this warp
  const int row = quad * 32 + lane;      // row inside the Q tile
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tS = tmem + lane_off + q * 128;
  const uint32_t tO = tmem + lane_off + 256 + q * 128;
  const float sl2 = p.scale_log2;
  const float2 sl2v = make_float2(sl2, sl2);
  uint32_t s_ph = 0, o_ph = 0;
  bool ok = true;
  for (int64_t r = 0; ok; ++r) {
    const int64_t u = snake_pos(r, slot, nslots);
    if (u >= p.num_units) break;
    const Unit w = unit_at(g, u);
    const int rq = w.r0 + row_base + q * BM + row;  // row inside query block i
    float fold_lse_a = -INFINITY;        // fold mode: the state row's LSE, read while the unit runs
    if (p.O_acc && rq < g.c) {           // and its O row brought into L2 for the unit's end
      const int64_t gi = static_cast<int64_t>(w.bh) * p.S + static_cast<int64_t>(w.i) * g.c + rq;
      const char* srow = reinterpret_cast<const char*>(p.O_acc + gi * HD);
#pragma unroll
      for (int k = 0; k < 4; ++k) asm volatile("prefetch.global.L2 [%0];" ::"l"(srow + 128 * k));
      if (RA_CHECK_RANGE(p.chk, SITE_FWD_FOLD, gi, 1, p.BH * p.S)) fold_lse_a = p.LSE_acc[gi];
    }
    float m_use = -INFINITY, l = 0.f;
    int t = 0, s_prev = -1;
    uint64_t t_step0 = 0;
    for (int s = 0; s < g.N && ok; ++s) {
      const int j = ring_block(w.i, s, g.N);
      if (!block_visited(g, w.i, j)) continue;
      const int last = kt_last(g, w.i, j, w.r0);
      const int lim = key_limit(g, w.i, j, rq);
      for (int kt = 0; kt <= last; ++kt, ++t) {
        if (!(ok = mbar_wait(&s_full[q], s_ph, wc, ST_FWD_WAIT | 9))) break;
        s_ph ^= 1;
        tc_fence_after();
        if (timer && kt == 0) {
          const uint64_t now = globaltimer_ns();
          if (s_prev >= 0) atomicAdd(&p.timing[w.i * g.N + s_prev], now - t_step0);
          s_prev = s;
          t_step0 = now;
        }
        float sv[BN];
        uint32_t* su = reinterpret_cast<uint32_t*>(sv);
        tmem_ld32(tS + 0, su);
        tmem_ld32(tS + 32, su + 32);
        tmem_ld32(tS + 64, su + 64);
        tmem_ld32(tS + 96, su + 96);
        tmem_ld_wait();
        if (tile_masked(g, w.i, j, kt, w.r0)) {
          const int rk0 = kt * BN;
#pragma unroll
          for (int k = 0; k < BN; ++k)
            if (rk0 + k >= lim) sv[k] = -INFINITY;
        }
        // Row max as 4 independent chains of three-input maxima (two new
        // values per instruction).
        float mx0 = fmaxf(sv[0], sv[4]), mx1 = fmaxf(sv[1], sv[5]), mx2 = fmaxf(sv[2], sv[6]),
              mx3 = fmaxf(sv[3], sv[7]);
#pragma unroll
        for (int k = 8; k < BN; k += 8) {
          mx0 = fmax3(mx0, sv[k], sv[k + 4]);
          mx1 = fmax3(mx1, sv[k + 1], sv[k + 5]);
          mx2 = fmax3(mx2, sv[k + 2], sv[k + 6]);
          mx3 = fmax3(mx3, sv[k + 3], sv[k + 7]);
        }
        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        // Rescale only when the max grew by more than the threshold: O and
        // l then share a stale reference max, which cancels in O / l.
        const float mt = mx * sl2;
        const bool grow = mt > m_use + RESCALE_THRESHOLD;
        float alpha = 1.f;
        if (grow) {
          alpha = hw_exp2(m_use - mt);   // 0 when nothing was seen before
          l *= alpha;
          m_use = mt;
        }
        const bool rescale_o = (t > 0) && __any_sync(0xffffffffu, grow);
#if RA_CHECKS
        if (rescale_o && grow) RA_COUNT(p.chk, EV_FWD_RESCALE_ROWS, 1);
        if (rescale_o && lane == 0) RA_COUNT(p.chk, EV_FWD_RESCALE_WARPS, 1);
#endif
        const float mref = (m_use == -INFINITY) ? 0.f : m_use;
        const float2 nm2 = make_float2(-mref, -mref);
        // Exponent arguments and the row sum two lanes at a time (packed
        // f32x2 FMA and add): the sum runs as an even and an odd chain.
        float2 rs2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 a = __ffma2_rn(make_float2(sv[ch * 32 + k], sv[ch * 32 + k + 1]), sl2v, nm2);
            const float2 pp = make_float2(hw_exp2(a.x), hw_exp2(a.y));
            rs2 = __fadd2_rn(rs2, pp);
            pk[k >> 1] = pack_bf16x2(pp.x, pp.y);
          }
          tmem_st16(tS + ch * 16, pk);
        }
        l += rs2.x + rs2.y;
        if (rescale_o) {   // O_q is idle: PV_q(t-1) completed before S_q(t) was signalled
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t ov[32];
            tmem_ld32(tO + ch * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(ov[k]), __uint_as_float(ov[k + 1])),
                                           make_float2(alpha, alpha));
              ov[k] = __float_as_uint(o2.x);
              ov[k + 1] = __float_as_uint(o2.y);
            }
            tmem_st32(tO + ch * 32, ov);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        arrive_p(q);
      }
    }
    if (!ok) break;
    // ---- epilogue: O / l -> bf16, LSE = (m + log2 l) * ln 2
    if (!(ok = mbar_wait(&o_full[q], o_ph, wc, ST_FWD_WAIT | 10))) break;
    o_ph ^= 1;
    tc_fence_after();
    if (timer && s_prev >= 0) atomicAdd(&p.timing[w.i * g.N + s_prev], globaltimer_ns() - t_step0);
    bool valid = rq < g.c;
    const int64_t grow_idx = static_cast<int64_t>(w.bh) * p.S + static_cast<int64_t>(w.i) * g.c + rq;
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    if (p.O_acc) {
      // Fold mode: LogSumExp-merge this call's partial (O = acc / l, lse_b) into the row of the
      // running float32 state, which this thread alone owns.  A state row with LSE -inf is
      // empty and is not read; a partial with no visible key leaves the row as it is.
      if (valid && !(RA_CHECK_RANGE(p.chk, SITE_FWD_FOLD, grow_idx * HD, HD, p.BH * p.S * HD) &&
                     RA_CHECK_RANGE(p.chk, SITE_FWD_FOLD, grow_idx, 1, p.BH * p.S)))
        valid = false;
      const float lse_b = l > 0.f ? (m_use + hw_log2(l)) * 0.6931471805599453f : -INFINITY;
      const float lse_a = valid ? fold_lse_a : -INFINITY;
      const bool fold = valid && lse_b != -INFINITY;
      float wa = 0.f, wb = 0.f, lse_n = lse_a;
      if (fold) {
        const float M = fmaxf(lse_a, lse_b);
        const float ea = expf(lse_a - M), eb = expf(lse_b - M);
        lse_n = M + logf(ea + eb);
        wa = ea / (ea + eb);
        wb = eb / (ea + eb) * inv_l;   // the partial's O is acc * inv_l
      }
      float4* srow4 = reinterpret_cast<float4*>(p.O_acc + grow_idx * HD);
      const bool read_a = fold && lse_a != -INFINITY;
      // The state row streams through two register buffers: chunk ch + 1's eight 16-byte loads
      // are in flight while chunk ch is combined and stored.
      float4 st[2][8];
#pragma unroll
      for (int v4 = 0; v4 < 8; ++v4) st[0][v4] = read_a ? srow4[v4] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if (ch + 1 < 4) {
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            st[(ch + 1) & 1][v4] = read_a ? srow4[(ch + 1) * 8 + v4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        uint32_t ov[32];
        tmem_ld32(tO + ch * 32, ov);
        tmem_ld_wait();
        if (fold) {
          float4* dst = srow4 + ch * 8;
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            float4 a = st[ch & 1][v4];
            a.x = fmaf(wb, __uint_as_float(ov[4 * v4]), wa * a.x);
            a.y = fmaf(wb, __uint_as_float(ov[4 * v4 + 1]), wa * a.y);
            a.z = fmaf(wb, __uint_as_float(ov[4 * v4 + 2]), wa * a.z);
            a.w = fmaf(wb, __uint_as_float(ov[4 * v4 + 3]), wa * a.w);
            dst[v4] = a;
          }
        }
      }
      if (fold) p.LSE_acc[grow_idx] = lse_n;
      tc_fence_before();
      arrive_o(q);
      continue;
    }
    __nv_bfloat16* orow = p.O + grow_idx * HD;
    if (valid && !RA_CHECK_RANGE(p.chk, SITE_FWD_O, grow_idx * HD, HD, p.BH * p.S * HD)) valid = false;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t ov[32];
      tmem_ld32(tO + ch * 32, ov);
      tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        pk[k] = pack_bf16x2(__uint_as_float(ov[2 * k]) * inv_l, __uint_as_float(ov[2 * k + 1]) * inv_l);
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
      }
    }
    if (valid && RA_CHECK_RANGE(p.chk, SITE_FWD_LSE, grow_idx, 1, p.BH * p.S))
      p.LSE[grow_idx] = l > 0.f ? (m_use + hw_log2(l)) * 0.6931471805599453f : -INFINITY;
    tc_fence_before();
    arrive_o(q);
  }
}

}  // namespace fwdsm
}  // namespace ra
