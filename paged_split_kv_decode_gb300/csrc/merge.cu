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
// o_indptr, then waits for that grid.
#include <cuda_runtime.h>

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
  load_rows(0, n, l_first, 0);

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

template <int NV>
cudaError_t launch_nv(dim3 grid, bool wide, bool early, bool skip, const InlineIndptr *inl, cudaStream_t s,
                      const float *v_in, const float *lse_in, const int32_t *o_indptr, int64_t num_out, int H,
                      int D, float *v_out, float *lse_out) {
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
  const int64_t warps = num_out * H;
  const int64_t blocks = (warps + kMergeWarps - 1) / kMergeWarps;
  if (blocks > 0x7fffffffLL) return fail(PSD_ERR_UNSUPPORTED, "merge_states: grid too large");
  const dim3 grid(static_cast<unsigned>(blocks));
  // up to two wide blocks per SM cover the grid in one wave
  const bool wide = blocks <= 2LL * dev.num_sms;
  cudaError_t e;
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
