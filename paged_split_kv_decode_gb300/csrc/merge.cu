// K3: log2-LSE merge of contiguous partial rows (mlxcel PR #1004, Merge contract
// section: v_in [N, H, D] normalised per row, lse_in [N, H] in log2 units,
// o_indptr [M + 1] grouping contiguous rows; a group of one is the identity).
//
// HBM-bound stream: each input row of one head is D floats read once, each output
// row D floats written once.  A row whose LSE is -inf is an empty partial: weight
// zero, and its v is not used.  One warp owns one (output row, head); lanes hold
// float4 slices of D.  The first 16 / NV input rows are loaded together with the
// first 32 LSE values (the rows do not depend on the maximum), and later rows in
// batches of the same size, so a group of up to 16 rows costs one round trip to
// memory after the group bounds.  The SKIP form, for partials with many empty rows,
// reads each batch's LSE values first and loads only the live rows' v.  When the
// partial kernel before it on the stream allows it, the merge launches early, reads
// o_indptr, then waits for that grid.  Large merges on their own stream whole input
// rows through shared memory instead (merge_stream_kernel below).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

constexpr int kMergeWarps = 8;

// NV: float4 slices per lane (D <= 128 * NV).  WIDE batches 16 / NV rows for grids of
// about one wave (latency-bound); the narrow form batches half as many rows with
// fewer registers, so more warps per SM keep loads in flight on large grids.
// INL: the group bounds come in the launch's parameters (`inl`), not from o_indptr.
template <int NV, bool WIDE, bool SKIP, bool INL>
__global__ void __launch_bounds__(kMergeWarps * 32, WIDE ? 1 : (NV >= (SKIP ? 4 : 8) ? 2 : 3))
    merge_states_kernel(const float *__restrict__ v_in, const float *__restrict__ lse_in,
                        const int32_t *__restrict__ o_indptr, int64_t num_out, int H, int D,
                        float *__restrict__ v_out, float *__restrict__ lse_out,
                        const __grid_constant__ IndptrParam<INL> inl) {
  constexpr int U = WIDE ? (NV >= 8 ? 2 : 16 / NV) : (NV >= 8 ? 1 : 8 / NV);  // rows per batch
  const int lane = threadIdx.x & 31;
  const int64_t gw = int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (gw >= num_out * H) return;
  const int64_t r = gw / H;
  const int h = int(gw - r * H);
  // o_indptr is in place before the partial kernel starts; the partials are not.
  int lo, hi;
  if constexpr (INL) {
    lo = inl.v[r];
    hi = inl.v[r + 1];
  } else {
    lo = __ldg(o_indptr + r);
    hi = __ldg(o_indptr + r + 1);
  }
  wait_for_prior_grid();
  const int n = hi - lo;
  const int D4 = D >> 2;
  float4 *out4 = reinterpret_cast<float4 *>(v_out + (r * H + h) * int64_t(D));

  float4 v[U][NV];
  // Rows first .. first + count - 1 (at most U) of the group; lw holds, in lane i,
  // the LSE of row w0 + i of the current 32-row window, and j0 = first - w0.
  auto load_rows = [&](int first, int count, float lw, int j0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      bool ok = u < count;
      if constexpr (SKIP) ok = __shfl_sync(0xffffffffu, lw, (j0 + u) & 31) != neg_inf() && ok;
      const float4 *src =
          reinterpret_cast<const float4 *>(v_in + (int64_t(lo + first + u) * H + h) * D);
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int d4 = lane + 32 * k;
        v[u][k] = (ok && d4 < D4) ? __ldcs(src + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };

  const float l_first = lane < n ? __ldg(lse_in + int64_t(lo + lane) * H + h) : neg_inf();
  // (SKIP loads only the live rows below; row 0 here serves the identity case)
  load_rows(0, SKIP ? min(n, 1) : n, l_first, 0);

  if (n == 1) {  // identity: w = 1, l = 1, out = v bit for bit
    const float l = __shfl_sync(0xffffffffu, l_first, 0);
    const bool live = l != neg_inf();
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int d4 = lane + 32 * k;
      if (d4 < D4) out4[d4] = live ? v[0][k] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (lse_out && lane == 0) lse_out[r * H + h] = l;
    return;
  }

  float M = l_first;
  for (int i = lane + 32; i < n; i += 32) M = fmaxf(M, __ldg(lse_in + int64_t(lo + i) * H + h));
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (n <= 0 || M == neg_inf()) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int d4 = lane + 32 * k;
      if (d4 < D4) out4[d4] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (lse_out && lane == 0) lse_out[r * H + h] = neg_inf();
    return;
  }

  float4 acc[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float sw = 0.f;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int cnt = min(32, n - i0);
    const float l = i0 == 0 ? l_first
                            : (lane < cnt ? __ldg(lse_in + int64_t(lo + i0 + lane) * H + h) : neg_inf());
    const float w_mine = lane < cnt ? ex2(l - M) : 0.f;
    sw += w_mine;
    if constexpr (SKIP) {
      // Only the window's live rows, U at a time in increasing order (the same sum,
      // in the same order, as visiting every row and skipping zero weights).
      unsigned live = __ballot_sync(0xffffffffu, lane < cnt && l != neg_inf());
      while (live) {
        int idx[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          idx[u] = live ? __ffs(live) - 1 : -1;
          live &= live - 1u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float4 *src =
              reinterpret_cast<const float4 *>(v_in + (int64_t(lo + i0 + max(idx[u], 0)) * H + h) * D);
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            const int d4 = lane + 32 * k;
            v[u][k] = (idx[u] >= 0 && d4 < D4) ? __ldcs(src + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (idx[u] < 0) break;  // warp-uniform
          const float w = __shfl_sync(0xffffffffu, w_mine, idx[u]);
          if (w == 0.f) continue;
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            acc[k].x = fmaf(w, v[u][k].x, acc[k].x);
            acc[k].y = fmaf(w, v[u][k].y, acc[k].y);
            acc[k].z = fmaf(w, v[u][k].z, acc[k].z);
            acc[k].w = fmaf(w, v[u][k].w, acc[k].w);
          }
        }
      }
      continue;
    }
    for (int j = 0; j < cnt; j += U) {
      if (i0 + j > 0) load_rows(i0 + j, cnt - j, l, j);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float w = j + u < cnt ? __shfl_sync(0xffffffffu, w_mine, (j + u) & 31) : 0.f;
        if (w == 0.f) continue;  // an empty row (LSE -inf): its v is not used, whatever it holds
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          acc[k].x = fmaf(w, v[u][k].x, acc[k].x);
          acc[k].y = fmaf(w, v[u][k].y, acc[k].y);
          acc[k].z = fmaf(w, v[u][k].z, acc[k].z);
          acc[k].w = fmaf(w, v[u][k].w, acc[k].w);
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, off);
  const float inv = 1.f / sw;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int d4 = lane + 32 * k;
    if (d4 < D4)
      __stcs(out4 + d4, make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv));
  }
  if (lse_out && lane == 0) lse_out[r * H + h] = M + log2f(sw);
}

// Large grids with an even head count: one warp merges heads h and h + 1 of one
// output row.  The group bounds are read once for both, their LSE pairs come in one
// 8-byte load per row, and both heads' rows are in flight together, which doubles
// the bytes a warp has outstanding at the cost of running two blocks per SM.
template <int NV, bool SKIP, bool INL>
__global__ void __launch_bounds__(kMergeWarps * 32, 2)
    merge_pair_kernel(const float *__restrict__ v_in, const float *__restrict__ lse_in,
                      const int32_t *__restrict__ o_indptr, int64_t num_out, int H, int D,
                      float *__restrict__ v_out, float *__restrict__ lse_out,
                      const __grid_constant__ IndptrParam<INL> inl) {
  constexpr int U = NV >= 8 ? 1 : 8 / NV;  // rows per batch and head
  const int lane = threadIdx.x & 31;
  const int Hp = H >> 1;
  const int64_t gw = int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (gw >= num_out * Hp) return;
  const int64_t r = gw / Hp;
  const int h0 = 2 * int(gw - r * Hp);
  int lo, hi;
  if constexpr (INL) {
    lo = inl.v[r];
    hi = inl.v[r + 1];
  } else {
    lo = __ldg(o_indptr + r);
    hi = __ldg(o_indptr + r + 1);
  }
  wait_for_prior_grid();
  const int n = hi - lo;
  const int D4 = D >> 2;

  float4 v[2][U][NV];
  // rows first .. first + count - 1 of both heads; lw[t] holds, in lane i, head t's
  // LSE of row w0 + i of the current 32-row window, and j0 = first - w0
  auto load_rows = [&](int first, int count, const float2 lw, int j0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      bool ok0 = u < count, ok1 = ok0;
      if constexpr (SKIP) {
        ok0 = __shfl_sync(0xffffffffu, lw.x, (j0 + u) & 31) != neg_inf() && ok0;
        ok1 = __shfl_sync(0xffffffffu, lw.y, (j0 + u) & 31) != neg_inf() && ok1;
      }
      const float4 *src = reinterpret_cast<const float4 *>(v_in + (int64_t(lo + first + u) * H + h0) * D);
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int d4 = lane + 32 * k;
        v[0][u][k] = (ok0 && d4 < D4) ? __ldcs(src + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[1][u][k] = (ok1 && d4 < D4) ? __ldcs(src + D4 + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };
  auto lse_pair = [&](int i) -> float2 {  // LSE of heads h0, h0 + 1 for group row i
    return __ldg(reinterpret_cast<const float2 *>(lse_in + int64_t(lo + i) * H + h0));
  };
  const float2 ninf2 = make_float2(neg_inf(), neg_inf());
  const float2 l_first = lane < n ? lse_pair(lane) : ninf2;
  load_rows(0, n, l_first, 0);
  float4 *out4 = reinterpret_cast<float4 *>(v_out + (r * H + h0) * int64_t(D));

  if (n == 1) {  // identity: out = v bit for bit
    const float l0 = __shfl_sync(0xffffffffu, l_first.x, 0), l1 = __shfl_sync(0xffffffffu, l_first.y, 0);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int d4 = lane + 32 * k;
      if (d4 < D4) {
        out4[d4] = l0 != neg_inf() ? v[0][0][k] : make_float4(0.f, 0.f, 0.f, 0.f);
        out4[D4 + d4] = l1 != neg_inf() ? v[1][0][k] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (lse_out && lane == 0) {
      lse_out[r * H + h0] = l0;
      lse_out[r * H + h0 + 1] = l1;
    }
    return;
  }

  float M0 = l_first.x, M1 = l_first.y;
  for (int i = lane + 32; i < n; i += 32) {
    const float2 l = lse_pair(i);
    M0 = fmaxf(M0, l.x);
    M1 = fmaxf(M1, l.y);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    M0 = fmaxf(M0, __shfl_xor_sync(0xffffffffu, M0, off));
    M1 = fmaxf(M1, __shfl_xor_sync(0xffffffffu, M1, off));
  }
  // an empty or all -inf group gives 0 and -inf (per head)
  const bool live0 = n > 0 && M0 != neg_inf(), live1 = n > 0 && M1 != neg_inf();
  const float Ms0 = live0 ? M0 : 0.f, Ms1 = live1 ? M1 : 0.f;

  float4 acc[2][NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) acc[0][k] = acc[1][k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float sw0 = 0.f, sw1 = 0.f;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int cnt = min(32, n - i0);
    const float2 l = i0 == 0 ? l_first : (lane < cnt ? lse_pair(i0 + lane) : ninf2);
    const float w0_mine = lane < cnt ? ex2(l.x - Ms0) : 0.f;
    const float w1_mine = lane < cnt ? ex2(l.y - Ms1) : 0.f;
    sw0 += w0_mine;
    sw1 += w1_mine;
    for (int j = 0; j < cnt; j += U) {
      if (i0 + j > 0) load_rows(i0 + j, cnt - j, l, j);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool in = j + u < cnt;
        const float w0 = in ? __shfl_sync(0xffffffffu, w0_mine, (j + u) & 31) : 0.f;
        const float w1 = in ? __shfl_sync(0xffffffffu, w1_mine, (j + u) & 31) : 0.f;
        if (w0 != 0.f) {  // an empty row (LSE -inf): its v is not used, whatever it holds
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            acc[0][k].x = fmaf(w0, v[0][u][k].x, acc[0][k].x);
            acc[0][k].y = fmaf(w0, v[0][u][k].y, acc[0][k].y);
            acc[0][k].z = fmaf(w0, v[0][u][k].z, acc[0][k].z);
            acc[0][k].w = fmaf(w0, v[0][u][k].w, acc[0][k].w);
          }
        }
        if (w1 != 0.f) {
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            acc[1][k].x = fmaf(w1, v[1][u][k].x, acc[1][k].x);
            acc[1][k].y = fmaf(w1, v[1][u][k].y, acc[1][k].y);
            acc[1][k].z = fmaf(w1, v[1][u][k].z, acc[1][k].z);
            acc[1][k].w = fmaf(w1, v[1][u][k].w, acc[1][k].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    sw0 += __shfl_xor_sync(0xffffffffu, sw0, off);
    sw1 += __shfl_xor_sync(0xffffffffu, sw1, off);
  }
  const float inv0 = live0 ? 1.f / sw0 : 0.f, inv1 = live1 ? 1.f / sw1 : 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int d4 = lane + 32 * k;
    if (d4 < D4) {
      __stcs(out4 + d4, make_float4(acc[0][k].x * inv0, acc[0][k].y * inv0, acc[0][k].z * inv0, acc[0][k].w * inv0));
      __stcs(out4 + D4 + d4,
             make_float4(acc[1][k].x * inv1, acc[1][k].y * inv1, acc[1][k].z * inv1, acc[1][k].w * inv1));
    }
  }
  if (lse_out && lane == 0) {
    lse_out[r * H + h0] = live0 ? M0 + log2f(sw0) : neg_inf();
    lse_out[r * H + h0 + 1] = live1 ? M1 + log2f(sw1) : neg_inf();
  }
}

// Large merges without a preceding partial kernel (merge_states on its own): three
// CTAs per SM, each streaming a contiguous range of whole input rows (every head's V,
// then the row's LSE values) through a ring of four stages in shared memory, each row
// by two bulk asynchronous copies that a producer warp issues.  The register-held
// loads of the forms above keep about 128 KB per SM in flight (the register file
// bounds them), and ncu put that form at 73% of peak DRAM throughput with its warps
// waiting on loads; the rings keep about 200 KB per SM in flight.  Measured at
// H = 32, D = 128: 6.82 TB/s at 1M output rows against 6.00, 6.39 against 6.02 at 16K
// (one CTA per SM with a 13-stage ring: 5.57; two per SM: 6.73).  Consumer thread t
// owns float4 chunks t + 256 j of a row and, for each chunk's head, a running
// maximum: a row whose LSE exceeds it rescales that head's sum and weighted V first
// (online, so the group's maximum is not needed up front).  A one-row group gives
// weight 1 and sum 1, so out = v and lse_out = lse exactly.  A wait that runs out
// fills the CTA's unfinished output rows with NaN (there is no fault word here).
constexpr int kStreamConsumers = 8;                              // warps
constexpr int kStreamThreads = 32 * (kStreamConsumers + 1);      // + the producer warp
constexpr int kStreamCtas = 3;                                   // per SM
constexpr uint32_t kStreamRing = 68 * 1024;                      // per CTA
constexpr int kStreamMaxStages = 32;

struct StreamParams {
  const float *v_in;
  const float *lse_in;
  const int32_t *o_indptr;
  int64_t num_out;
  int H, D, stages;
  uint32_t row_bytes, lse_bytes, stage_bytes;
  float *v_out;
  float *lse_out;
  long long wait_limit;  // cycles before a wait gives up
  int withhold_from;     // testing aid: no copies from this input row of a CTA's range on
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// A bounded wait with no fault word to report to: false after the limit.
__device__ __forceinline__ bool stream_wait(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

template <int C>  // float4 chunks per consumer thread: H * D / 4 = 256 * C
__global__ void __launch_bounds__(kStreamThreads, kStreamCtas) merge_stream_kernel(const StreamParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(p.stages) * p.stage_bytes);
  uint64_t *empty = full + p.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kStreamConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();
  wait_for_prior_grid();
  // This CTA's output rows [r0, r1): the group boundaries nearest to its equal share of
  // the input rows (o_indptr is non-decreasing; lower bound of the share's first row).
  const int32_t base = __ldg(p.o_indptr), total = __ldg(p.o_indptr + p.num_out) - base;
  auto first_row = [&](int64_t b) -> int64_t {
    if (b >= gridDim.x) return p.num_out;
    const int64_t t = base + int64_t(total) * b / gridDim.x;
    int64_t lo = 0, hi = p.num_out;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (__ldg(p.o_indptr + mid) < t) lo = mid + 1;
      else hi = mid;
    }
    return lo;
  };
  const int64_t r0 = first_row(blockIdx.x), r1 = first_row(int64_t(blockIdx.x) + 1);
  if (r1 <= r0) return;
  const int32_t g0 = __ldg(p.o_indptr + r0), g1 = __ldg(p.o_indptr + r1);
  const int S = p.stages;

  if (warp == kStreamConsumers) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      int32_t issued = 0;
      for (int32_t k = 0; k < g1 - g0; ++k) {
        if (k >= p.withhold_from) break;  // testing aid: the consumers' wait for row k runs out
        const int s = k % S;
        if (k >= S && !stream_wait(smem_u32(empty + s), uint32_t(k / S - 1) & 1u, p.wait_limit)) break;
        const int64_t row = int64_t(g0) + k;
        const uint32_t dst = smem_u32(smem + size_t(s) * p.stage_bytes);
        mbar_arrive_expect_tx(smem_u32(full + s), p.row_bytes + p.lse_bytes);
        bulk_load(dst, p.v_in + row * p.H * p.D, p.row_bytes, smem_u32(full + s));
        bulk_load(dst + p.row_bytes, p.lse_in + row * p.H, p.lse_bytes, smem_u32(full + s));
        issued = k + 1;
      }
      // No copy in flight at exit, also after a wait ran out: the last S issued rows'
      // barriers complete once they land (each stage's earlier row was consumed before
      // its next copy was issued, so every such wait is for the phase in progress).
      for (int32_t k = issued > S ? issued - S : 0; k < issued; ++k)
        stream_wait(smem_u32(full + k % S), uint32_t(k / S) & 1u, p.wait_limit);
    }
    return;
  }
  // ------------------------------------------------------------- consumer warps
  const int t = threadIdx.x;
  const int D4 = p.D >> 2;
  int head[C];
#pragma unroll
  for (int j = 0; j < C; ++j) head[j] = (t + 256 * j) / D4;
  bool ok = true;
  for (int64_t r = r0; r < r1 && ok; ++r) {
    const int32_t lo = __ldg(p.o_indptr + r), n = __ldg(p.o_indptr + r + 1) - lo;
    float M[C], sw[C];
    float4 acc[C];
#pragma unroll
    for (int j = 0; j < C; ++j) {
      M[j] = neg_inf();
      sw[j] = 0.f;
      acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int32_t i = 0; i < n; ++i) {
      const int32_t k = lo + i - g0;
      const int s = k % S;
      ok = __all_sync(0xffffffffu, stream_wait(smem_u32(full + s), uint32_t(k / S) & 1u, p.wait_limit));
      if (!ok) break;
      const uint8_t *stage = smem + size_t(s) * p.stage_bytes;
      const float *lse_row = reinterpret_cast<const float *>(stage + p.row_bytes);
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const float l = lse_row[head[j]];
        if (l == neg_inf()) continue;  // an empty partial: its v is not used
        const float4 v = reinterpret_cast<const float4 *>(stage)[t + 256 * j];
        if (l > M[j]) {
          const float a = ex2(M[j] - l);   // 0 while M is -inf
          acc[j].x *= a;
          acc[j].y *= a;
          acc[j].z *= a;
          acc[j].w *= a;
          sw[j] *= a;
          M[j] = l;
        }
        const float w = ex2(l - M[j]);
        acc[j].x = fmaf(w, v.x, acc[j].x);
        acc[j].y = fmaf(w, v.y, acc[j].y);
        acc[j].z = fmaf(w, v.z, acc[j].z);
        acc[j].w = fmaf(w, v.w, acc[j].w);
        sw[j] += w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(empty + s));
    }
    if (!ok) {  // a wait ran out: this row and the rest of the range read as NaN
      const float nan = __int_as_float(0x7fc00000);
      for (int64_t q = r; q < r1; ++q) {
        float4 *o4 = reinterpret_cast<float4 *>(p.v_out + q * p.H * p.D);
#pragma unroll
        for (int j = 0; j < C; ++j) {
          o4[t + 256 * j] = make_float4(nan, nan, nan, nan);
          if (p.lse_out && (t + 256 * j) % D4 == 0) p.lse_out[q * p.H + head[j]] = nan;
        }
      }
      break;
    }
    float4 *out4 = reinterpret_cast<float4 *>(p.v_out + r * p.H * p.D);
#pragma unroll
    for (int j = 0; j < C; ++j) {
      const bool live = M[j] != neg_inf();
      const float inv = live ? 1.f / sw[j] : 0.f;
      __stcs(out4 + t + 256 * j, make_float4(acc[j].x * inv, acc[j].y * inv, acc[j].z * inv, acc[j].w * inv));
      if (p.lse_out && (t + 256 * j) % D4 == 0) p.lse_out[r * p.H + head[j]] = live ? M[j] + log2f(sw[j]) : neg_inf();
    }
  }
}

template <int C>
cudaError_t launch_stream_c(const DeviceInfo &dev, cudaStream_t s, const StreamParams &p, size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(merge_stream_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  merge_stream_kernel<C><<<dim3(static_cast<unsigned>(kStreamCtas * dev.num_sms)), kStreamThreads, smem, s>>>(p);
  return cudaGetLastError();
}

// The streaming form when it applies: H * D / 4 a multiple of 256 with at most 4
// chunks per thread (more spill at three CTAs per SM), 16-byte LSE rows, at least 8
// output rows per CTA (below that the one-wave forms above are faster: 1K rows at
// H = 32 take 33 us there and 40 us here), and four stages in the ring.  Returns false
// to fall back.
bool launch_stream(const DeviceInfo &dev, cudaStream_t s, const float *v_in, const float *lse_in,
                   const int32_t *o_indptr, int64_t num_out, int H, int D, float *v_out, float *lse_out,
                   cudaError_t &e) {
  const int64_t chunks = int64_t(H) * D / 4;
  if (chunks % 256 != 0 || chunks / 256 > 4 || H % 4 != 0 || num_out < 8LL * kStreamCtas * dev.num_sms) return false;
  if (reinterpret_cast<uintptr_t>(lse_in) % 16 != 0) return false;
  StreamParams p;
  p.v_in = v_in;
  p.lse_in = lse_in;
  p.o_indptr = o_indptr;
  p.num_out = num_out;
  p.H = H;
  p.D = D;
  p.row_bytes = uint32_t(H) * uint32_t(D) * 4u;
  p.lse_bytes = uint32_t(H) * 4u;
  p.stage_bytes = p.row_bytes + p.lse_bytes;
  p.stages = std::min<int>(kStreamMaxStages, int(kStreamRing / p.stage_bytes));
  p.v_out = v_out;
  p.lse_out = lse_out;
  p.wait_limit = dev.test_wait_limit > 0 ? dev.test_wait_limit : kWaitLimitCycles;
  p.withhold_from = dev.test_withhold_from >= 0 ? dev.test_withhold_from : 0x7fffffff;
  const size_t smem = size_t(p.stages) * p.stage_bytes + 2 * sizeof(uint64_t) * size_t(p.stages);
  if (p.stages < 4 || smem > size_t(dev.smem_optin)) return false;
  switch (chunks / 256) {
    case 1: e = launch_stream_c<1>(dev, s, p, smem); break;
    case 2: e = launch_stream_c<2>(dev, s, p, smem); break;
    case 4: e = launch_stream_c<4>(dev, s, p, smem); break;
    default: return false;
  }
  return true;
}

template <int NV, bool SKIP, bool INL>
cudaError_t launch_form(dim3 grid, bool wide, bool early, cudaStream_t s, const float *v_in, const float *lse_in,
                        const int32_t *o_indptr, int64_t num_out, int H, int D, float *v_out,
                        float *lse_out, const IndptrParam<INL> &inl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;
  if (wide)
    return cudaLaunchKernelEx(&cfg, merge_states_kernel<NV, true, SKIP, INL>, v_in, lse_in, o_indptr,
                              num_out, H, D, v_out, lse_out, inl);
  return cudaLaunchKernelEx(&cfg, merge_states_kernel<NV, false, SKIP, INL>, v_in, lse_in, o_indptr, num_out,
                            H, D, v_out, lse_out, inl);
}

template <int NV, bool SKIP, bool INL>
cudaError_t launch_pair_impl(dim3 grid, bool early, cudaStream_t s, const float *v_in, const float *lse_in,
                        const int32_t *o_indptr, int64_t num_out, int H, int D, float *v_out, float *lse_out,
                        const IndptrParam<INL> &inl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, merge_pair_kernel<NV, SKIP, INL>, v_in, lse_in, o_indptr, num_out, H, D, v_out,
                            lse_out, inl);
}
template <int NV, bool SKIP, bool INL>
cudaError_t launch_pair(dim3 grid, bool early, cudaStream_t s, const float *v_in, const float *lse_in,
                        const int32_t *o_indptr, int64_t num_out, int H, int D, float *v_out, float *lse_out,
                        const IndptrParam<INL> &inl) {
  if constexpr (NV <= 2)
    return launch_pair_impl<NV, SKIP, INL>(grid, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out, inl);
  else
    return cudaErrorInvalidValue;  // (not selected: the launcher takes this form only for NV <= 2)
}

template <int NV>
cudaError_t launch_nv(dim3 grid, bool wide, bool early, bool skip, const InlineIndptr *inl, cudaStream_t s,
                      const float *v_in, const float *lse_in, const int32_t *o_indptr, int64_t num_out, int H,
                      int D, float *v_out, float *lse_out) {
  // Large grids, even H, D <= 256 (two heads' rows fit the registers) and 8-byte
  // aligned LSE rows: two heads per warp.
  if (NV <= 2 && !wide && H % 2 == 0 && reinterpret_cast<uintptr_t>(lse_in) % 8 == 0) {
    const int64_t blocks = (num_out * (H / 2) + kMergeWarps - 1) / kMergeWarps;
    const dim3 g2(static_cast<unsigned>(blocks));
    const NoInline none{};
    if (inl)
      return skip ? launch_pair<NV, true, true>(g2, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out, *inl)
                  : launch_pair<NV, false, true>(g2, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out, *inl);
    return skip ? launch_pair<NV, true, false>(g2, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out, none)
                : launch_pair<NV, false, false>(g2, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out, none);
  }
  if (inl)
    return skip ? launch_form<NV, true, true>(grid, wide, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out,
                                              lse_out, *inl)
                : launch_form<NV, false, true>(grid, wide, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out,
                                               lse_out, *inl);
  const NoInline none{};
  return skip ? launch_form<NV, true, false>(grid, wide, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out,
                                             lse_out, none)
              : launch_form<NV, false, false>(grid, wide, early, s, v_in, lse_in, o_indptr, num_out, H, D, v_out,
                                              lse_out, none);
}

}  // namespace

psd_status launch_merge(const float *v_in, const float *lse_in, const int32_t *o_indptr,
                        int64_t num_out, int32_t H, int32_t D, float *v_out, float *lse_out,
                        const DeviceInfo &dev, cudaStream_t s, bool after_partial, bool skip_empty,
                        const int32_t *o_indptr_host) {
  if (num_out == 0 || H == 0) return PSD_OK;
  InlineIndptr block;
  const InlineIndptr *inl = nullptr;
  if (o_indptr_host && num_out + 1 <= kInlineIndptr) {
    std::memcpy(block.v, o_indptr_host, sizeof(int32_t) * size_t(num_out + 1));
    inl = &block;
  }
  cudaError_t e;
  if (!after_partial && !inl && launch_stream(dev, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out, e)) {
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "merge_states launch: %s", cudaGetErrorString(e));
    return PSD_OK;
  }
  const int64_t warps = num_out * H;
  const int64_t blocks = (warps + kMergeWarps - 1) / kMergeWarps;
  if (blocks > 0x7fffffffLL) return fail(PSD_ERR_UNSUPPORTED, "merge_states: grid too large");
  const dim3 grid(static_cast<unsigned>(blocks));
  // up to two wide blocks per SM cover the grid in one wave
  const bool wide = blocks <= 2LL * dev.num_sms;
  if (D <= 128)
    e = launch_nv<1>(grid, wide, after_partial, skip_empty, inl, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out);
  else if (D <= 256)
    e = launch_nv<2>(grid, wide, after_partial, skip_empty, inl, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out);
  else if (D <= 512)
    e = launch_nv<4>(grid, wide, after_partial, skip_empty, inl, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out);
  else
    e = launch_nv<8>(grid, wide, after_partial, skip_empty, inl, s, v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "merge_states launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

}  // namespace psd
