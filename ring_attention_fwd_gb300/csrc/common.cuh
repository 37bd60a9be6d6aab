// common.cuh -- shared by the kernels and the host library: the ring-order
// work schedule, the per-element visibility rule, and launcher declarations.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "checks.cuh"

namespace ra {

// Geometry of one call.  The sequence of S rows is cut into N blocks of
// c = S/N rows (one per virtual ring host).  Storage row p = i*c + r is row r
// of block i; for the striped layout it holds token r*N + i, for the
// contiguous layout token p.
struct RingGeom {
  int N;        // ring size (blocks)
  int c;        // rows per block
  int causal;   // 0/1
  int striped;  // 0 = contiguous, 1 = striped
  int kt_w;     // rows per KV tile
  int n_kt;     // KV tiles per block = ceil(c / kt_w)
  int mb_h;     // query rows per work unit
  int n_mb;     // work units per query block = ceil(c / mb_h)
  int strict;   // 1: diag-type pairs never see the key at the query's own row
                //    (one striped pair j > i evaluated as a 1-block problem)
};

// Ring order: at step s, query block i meets KV block (i - s) mod N (host i
// receives from host i-1 and forwards to i+1).
__host__ __device__ __forceinline__ int ring_block(int i, int s, int N) {
  int j = i - s;
  return j < 0 ? j + N : j;
}

// Contiguous causal: blocks j > i hold only future tokens and are skipped
// whole.  Every other block pair is visited.
__host__ __device__ __forceinline__ bool block_visited(const RingGeom& g, int i, int j) {
  return !(g.causal && !g.striped && j > i);
}

// Block pairs whose mask depends on the row/column inside the block: the
// diagonal block of a contiguous causal sweep, and every striped causal pair.
__host__ __device__ __forceinline__ bool diag_type(const RingGeom& g, int i, int j) {
  return g.causal && (g.striped || j == i);
}

// Inside a diag-type pair (i, j), query row rq sees key row rk iff
// rk < rq, or rk == rq and the key token is not later than the query token:
// contiguous j == i (same token), striped j <= i (token rk*N+j <= rq*N+i).
// So rk is visible iff rk < rq + incl, with incl = 1 if (contiguous or j <= i).
__host__ __device__ __forceinline__ int diag_incl(const RingGeom& g, int i, int j) {
  return (!g.strict && (!g.striped || j <= i)) ? 1 : 0;
}

// Last KV tile of block j that a unit of query rows [r0, r0 + mb_h) needs.
__host__ __device__ __forceinline__ int kt_last(const RingGeom& g, int i, int j, int r0) {
  int last = g.n_kt - 1;
  if (diag_type(g, i, j)) {
    int d = (r0 + g.mb_h - 1) / g.kt_w;
    if (d < last) last = d;
  }
  return last;
}

// Does KV tile kt of pair (i, j) need the per-element mask for rows
// [r0, r0 + mb_h)?  Ragged last tile, or a diag-type pair whose tile reaches
// the unit's first row.
__host__ __device__ __forceinline__ bool tile_masked(const RingGeom& g, int i, int j, int kt, int r0) {
  if ((kt + 1) * g.kt_w > g.c) return true;
  return diag_type(g, i, j) && (kt * g.kt_w + g.kt_w - 1 >= r0);
}

// Exclusive upper bound on visible key rows rk for query row rq in a masked
// tile of pair (i, j): rk visible iff rk < key_limit.
__host__ __device__ __forceinline__ int key_limit(const RingGeom& g, int i, int j, int rq) {
  int lim = g.c;
  if (diag_type(g, i, j)) {
    int d = rq + diag_incl(g, i, j);
    if (d < lim) lim = d;
  }
  return lim;
}

// Number of KV tiles in the sweep of the unit (i, r0).
__host__ __device__ __forceinline__ int unit_tiles(const RingGeom& g, int i, int r0) {
  int T = 0;
  for (int s = 0; s < g.N; ++s) {
    int j = ring_block(i, s, g.N);
    if (block_visited(g, i, j)) T += kt_last(g, i, j, r0) + 1;
  }
  return T;
}

// Work units are (bh, i, m): head bh, query block i, rows [m*mb_h, ...).
// Enumeration order, per head, heaviest first (longest-processing-time) so a
// static snake assignment balances CTAs; all units of one head are adjacent
// so concurrently running CTAs share that head's K/V in L2.
struct Unit {
  int bh, i, r0;
};
__host__ __device__ __forceinline__ Unit unit_at(const RingGeom& g, int64_t u) {
  const int64_t per_head = static_cast<int64_t>(g.N) * g.n_mb;
  Unit w;
  w.bh = static_cast<int>(u / per_head);
  const int rem = static_cast<int>(u % per_head);
  int i, m;
  if (g.causal && !g.striped) {        // work grows with i, then m
    i = g.N - 1 - rem / g.n_mb;
    m = g.n_mb - 1 - rem % g.n_mb;
  } else if (g.causal) {               // striped: work grows with m only
    m = g.n_mb - 1 - rem / g.N;
    i = rem % g.N;
  } else {
    i = rem / g.n_mb;
    m = rem % g.n_mb;
  }
  w.i = i;
  w.r0 = m * g.mb_h;
  return w;
}
// Snake assignment: in round r CTA `cta` of `grid` takes position
// r*grid + cta (r even) or r*grid + grid-1-cta (r odd).
__host__ __device__ __forceinline__ int64_t snake_pos(int64_t r, int cta, int grid) {
  return r * grid + ((r & 1) ? (grid - 1 - cta) : cta);
}

// Device status codes written on a bounded-wait time-out (first one wins).
enum : unsigned int {
  ST_OK = 0,
  ST_FWD_WAIT = 0x100,  // | role/barrier id
  ST_BWD_WAIT = 0x200,
  ST_DEC_WAIT = 0x300,
  ST_FFN_WAIT = 0x400,
};

// Raises `func`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device (the attribute is per device, so a process driving
// several GPUs sets it on each).  Thread-safe; defined in host.cu.
cudaError_t raise_smem_limit(const void* func, int bytes);

// ----------------------------------------------------------- launchers
// All return cudaError_t of the launch; arguments are validated by the caller.
struct FwdArgs {
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  float* LSE;
  int64_t B, H, S, D, N;
  int causal, striped;
  int strict;                  // see RingGeom::strict (0 for whole-sequence calls)
  int withhold_first_q;        // test aid, bf16 kernel: see ra_set_wait_test
  unsigned int* status;
  unsigned long long* timing;  // [N*N] or null
  cudaStream_t stream;
  int num_sms;
  cudaEvent_t* ev;             // null, or 2 events recorded before/after the kernel
  CheckRec* chk;               // per-device check record (used by the checked build only)
  float* O_acc = nullptr;      // bf16 kernel, fold mode: running float32 state [B,H,S,D] and its
  float* LSE_acc = nullptr;    //   LSE [B,H,S], merged with this call's partial instead of writing O, LSE
  unsigned long long* clk = nullptr;   // bf16 kernels: clock record (4 words) or null
};
cudaError_t launch_fwd_f32(const FwdArgs& a);
cudaError_t launch_fwd_bf16(const FwdArgs& a, const void* tmap_q, const void* tmap_k,
                            const void* tmap_v);
// The same forward on SM pairs (2-CTA clusters, cta_group::2 MMAs); `tmap_k64`
// views K with 64-row boxes.
cudaError_t launch_fwd_bf16_pair(const FwdArgs& a, const void* tmap_q, const void* tmap_k64,
                                 const void* tmap_v);
// How many 2-CTA clusters of the pair kernel the current device holds at once
// (0: none fits; -1: the query failed).  Cached per device.
int fwd_pair_clusters();
// Operand types of the merge: state O_a / partial O_b.
enum : int { MERGE_F32 = 0, MERGE_BF16 = 1, MERGE_F32_BF16 = 2 };
cudaError_t launch_merge(void* O_a, float* lse_a, const void* O_b, const float* lse_b, int64_t rows,
                         int64_t D, int kind, cudaStream_t stream, int num_sms, CheckRec* chk);
cudaError_t launch_fill(float* x, int64_t n, float value, cudaStream_t stream, int num_sms);

struct BwdArgs {
  const void* Q;
  const void* K;
  const void* V;
  const void* O;
  const float* LSE;
  const void* dO;
  void* dQ;        // bf16 outputs, or f32 accumulators when `accumulate`
  void* dK;
  void* dV;
  float* nlse2;    // [B,H,N,ceil(c/128),128] float32 workspace: -LSE * log2(e)
  float* ndvec;    // same layout: -rowsum(dO * O)
  int64_t B, H, S, D, N;
  int causal, striped;
  int strict;      // see RingGeom::strict (0 for whole-sequence calls)
  int accumulate;  // 1: add the gradients into f32 dQ/dK/dV instead of writing bf16
  unsigned int* status;
  cudaStream_t stream;
  int num_sms;
  cudaEvent_t* ev;   // null, or 4 events: before prep, dK/dV and dQ kernels, and after
  CheckRec* chk;
  unsigned long long* clk_dkv = nullptr;   // clock records (4 words) of the two main kernels, or null
  unsigned long long* clk_dq = nullptr;
};
cudaError_t launch_bwd_bf16(const BwdArgs& a, const void* tmap_q, const void* tmap_k,
                            const void* tmap_v, const void* tmap_do);

// Ring decode work split.  The S-row cache of a head is cut into N ring blocks
// of c = ceil(S/N) rows; each block into cpb chunks of `chunk` rows (a multiple
// of 64), so that the whole call has about kDecodeItems work items.  Depends on
// the sizes only, so the workspace size is known without a device.
struct DecodePlan {
  int64_t c, chunk, cpb, items;
};
constexpr int64_t kDecodeItems = 16 * 152;   // 16 per SM of a 152-SM GB300
constexpr int64_t kDecodeMinChunk = 256;
__host__ __forceinline__ bool decode_plan(int64_t BH, int64_t S, int64_t N, DecodePlan* pl) {
  if (BH < 1 || S < 1 || N < 1 || N > (int64_t{1} << 30)) return false;
  if (BH > (int64_t{1} << 40) / N) return false;
  const int64_t c = (S + N - 1) / N;
  int64_t want = (kDecodeItems + BH * N - 1) / (BH * N);
  if (want < 1) want = 1;
  auto up64 = [](int64_t x) { return (x + 63) / 64 * 64; };
  int64_t chunk = up64((c + want - 1) / want);
  const int64_t floor_chunk = up64(c) < kDecodeMinChunk ? up64(c) : kDecodeMinChunk;
  if (chunk < floor_chunk) chunk = floor_chunk;
  pl->c = c;
  pl->chunk = chunk;
  pl->cpb = (c + chunk - 1) / chunk;
  pl->items = BH * N * pl->cpb;
  return true;
}

struct DecodeArgs {
  const void* q;     // [B, H, D] bf16
  const void* K;     // [B, H, S, D] bf16
  const void* V;
  void* O;           // [B, H, D] bf16
  float* LSE;        // [B, H]
  float* part_o;     // [plan.items, D] f32 workspace
  float* part_lse;   // [plan.items] f32 workspace
  int64_t B, H, S, N;
  DecodePlan plan;
  unsigned int* status;
  cudaStream_t stream;
  int num_sms;
  cudaEvent_t* ev;   // null, or 3 events: before the split kernel, between, after the combine
  CheckRec* chk;
};
cudaError_t launch_decode_bf16(const DecodeArgs& a);

// One GEMM of the blockwise feedforward: out[M, *] from A [M, K] (tensor map
// tmap_a) and B [*, K] (maps tmap_b0, tmap_b1), all bf16 K-major.
//   gated: out[:, N] = silu(A W1^T) * (A W3^T), b0 = W1 [N, K], b1 = W3 [N, K]
//   plain: out[:, N] = A W^T, b0 = b1 = W [N, K]
struct FfnGemmArgs {
  int64_t M, N, K;
  int gated;
  void* out;
  int64_t ldo;
  unsigned int* status;
  cudaStream_t stream;
  int num_sms;
  int overlap_previous;   // 1: may start while the previous launch (of the same call) drains
  int* tile_counter;      // device int, zero before the launch (dynamic tile scheduler)
  CheckRec* chk;
};
cudaError_t launch_ffn_gemm(const FfnGemmArgs& a, const void* tmap_a, const void* tmap_b0, const void* tmap_b1);


}  // namespace ra
