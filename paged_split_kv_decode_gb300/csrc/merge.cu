// K3: log2-LSE merge of contiguous partial rows (mlxcel PR #1004, Merge contract
// section: v_in [N, H, D] normalised per row, lse_in [N, H] in log2 units,
// o_indptr [M + 1] grouping contiguous rows; a group of one is the identity).
//
// HBM-bound stream: each input row of one head is D floats read once, each output
// row D floats written once.  One warp owns one (output row, head); lanes hold
// float4 slices of D; up to 8 input rows (4 when D > 128) are loaded before they
// are accumulated so every warp keeps several rows of loads in flight.
#include <cuda_runtime.h>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

constexpr int kMergeWarps = 8;

template <int NV>  // float4 slices per lane: D <= 128 * NV
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_states_kernel(const float *__restrict__ v_in, const float *__restrict__ lse_in,
                        const int32_t *__restrict__ o_indptr, int64_t num_out, int H, int D,
                        float *__restrict__ v_out, float *__restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (gw >= num_out * H) return;
  const int64_t r = gw / H;
  const int h = int(gw - r * H);
  const int lo = __ldg(o_indptr + r), hi = __ldg(o_indptr + r + 1);
  const int n = hi - lo;
  const int D4 = D >> 2;
  float4 *out4 = reinterpret_cast<float4 *>(v_out + (r * H + h) * int64_t(D));

  if (n == 1) {  // identity: w = 1, l = 1, out = v bit for bit
    const float l = __ldg(lse_in + int64_t(lo) * H + h);
    const bool live = l != neg_inf();
    const float4 *src = reinterpret_cast<const float4 *>(v_in + (int64_t(lo) * H + h) * D);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int d4 = lane + 32 * k;
      if (d4 < D4) out4[d4] = live ? __ldcs(src + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (lse_out && lane == 0) lse_out[r * H + h] = l;
    return;
  }

  float M = neg_inf();
  for (int i = lane; i < n; i += 32) M = fmaxf(M, __ldg(lse_in + int64_t(lo + i) * H + h));
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
    const float w_mine =
        lane < cnt ? ex2(__ldg(lse_in + int64_t(lo + i0 + lane) * H + h) - M) : 0.f;
    sw += w_mine;
    constexpr int U = NV == 1 ? 8 : 4;  // input rows in flight per warp
    for (int j = 0; j < cnt; j += U) {
      float4 v[U][NV];
      float w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        w[u] = __shfl_sync(0xffffffffu, w_mine, (j + u) & 31);
        const bool ok = j + u < cnt;
        const float4 *src =
            reinterpret_cast<const float4 *>(v_in + (int64_t(lo + i0 + j + u) * H + h) * D);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          const int d4 = lane + 32 * k;
          v[u][k] = (ok && d4 < D4) ? __ldcs(src + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!ok) w[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          acc[k].x = fmaf(w[u], v[u][k].x, acc[k].x);
          acc[k].y = fmaf(w[u], v[u][k].y, acc[k].y);
          acc[k].z = fmaf(w[u], v[u][k].z, acc[k].z);
          acc[k].w = fmaf(w[u], v[u][k].w, acc[k].w);
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

}  // namespace

psd_status launch_merge(const float *v_in, const float *lse_in, const int32_t *o_indptr,
                        int64_t num_out, int32_t H, int32_t D, float *v_out, float *lse_out,
                        const DeviceInfo &dev, cudaStream_t s) {
  (void)dev;
  if (num_out == 0 || H == 0) return PSD_OK;
  const int64_t warps = num_out * H;
  const int64_t blocks = (warps + kMergeWarps - 1) / kMergeWarps;
  if (blocks > 0x7fffffffLL) return fail(PSD_ERR_UNSUPPORTED, "merge_states: grid too large");
  const dim3 grid(static_cast<unsigned>(blocks));
  const dim3 block(kMergeWarps * 32);
  if (D <= 128)
    merge_states_kernel<1><<<grid, block, 0, s>>>(v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out);
  else if (D <= 256)
    merge_states_kernel<2><<<grid, block, 0, s>>>(v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out);
  else if (D <= 512)
    merge_states_kernel<4><<<grid, block, 0, s>>>(v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out);
  else
    merge_states_kernel<8><<<grid, block, 0, s>>>(v_in, lse_in, o_indptr, num_out, H, D, v_out, lse_out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "merge_states launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

}  // namespace psd
