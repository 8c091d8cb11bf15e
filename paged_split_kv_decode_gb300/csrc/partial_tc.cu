// K2: split-KV partial attention on tensor cores, for many query rows per KV head:
// the stacked level-0 request of the cascade (M*G rows) and the MLA latent shape
// (128 heads over one 576-wide latent, V = its first 512 columns, fp8-e4m3).
//
// mlxcel PR #1004, Decomposition section: level 0 is one request with M*G query
// heads per KV head, so QK^T and PV become dense [rows x D] x [D x tokens]
// contractions over each K/V tile read once.  ROCm ATOM PR #1701, section 3.2:
// fp8 latent rows decode to code * scale; here the scale is folded into the score
// scale (K) and the output (V), and codes widen exactly to bf16 in shared memory.
//
// Layout: grid = (work items, Hkv, row tiles of 64).  4 warps per dv slice of up
// to 256 columns; each warp owns 16 query rows for the whole tile, so no warp
// merge is needed.  K/V tiles of 16 tokens stream through a 4-stage cp.async ring
// (zero-fill past the tile's last token); QK^T and PV run as bf16 m16n8k16 MMAs
// with f32 accumulators, the probabilities are re-packed from the QK^T
// accumulators as the PV A operand.
#include <cuda_runtime.h>

#include <algorithm>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

constexpr int kRows = 64;    // query rows per CTA
constexpr int kTok = 16;     // tokens per tile
constexpr int kStagesTC = 4;

struct TCParams {
  const __nv_bfloat16 *q;
  const uint8_t *k_pool;
  const uint8_t *v_pool;
  const int32_t *page_indices;
  const psd_work_item *items;
  const int32_t *members;
  const int32_t *member_row_base;
  float *v_out;
  float *lse_out;
  FaultRef fault;
  int64_t num_pages;
  int Hq_req, Hkv, page_size, Gm, G_cta;
  float q_scale, v_scale;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// 8 e4m3 codes -> 8 bf16 (exact), as one 16-byte word.
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 c) {
  uint32_t w[2] = {c.x, c.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 a = e4m3x2_to_float2(w[i] & 0xffffu);
    const float2 b = e4m3x2_to_float2(w[i] >> 16);
    o[2 * i] = pack_bf16(a.x, a.y);
    o[2 * i + 1] = pack_bf16(b.x, b.y);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int DQK, int DV, bool FP8, bool LATENT>
struct TCShape {
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int DVT = DV > 256 ? 256 : DV;  // dv columns per warp group
  static constexpr int NDVT = DV / DVT;
  static constexpr int THREADS = 128 * NDVT;
  static constexpr int QS = DQK + 8;                // padded bf16 row strides
  static constexpr int VS = DV + 8;
  static constexpr int K_RAW = kTok * DQK * ESZ;    // one stage of K as stored
  static constexpr int V_RAW = LATENT ? 0 : kTok * DV * ESZ;
  // bf16 stages keep the padded layout directly; fp8 stages hold raw codes and
  // are widened into one padded bf16 tile before the MMAs.
  static constexpr int K_STAGE = FP8 ? K_RAW : kTok * QS * 2;
  static constexpr int V_STAGE = LATENT ? 0 : (FP8 ? V_RAW : kTok * VS * 2);
  static constexpr int STAGE = K_STAGE + V_STAGE;
  static constexpr int Q_BYTES = kRows * QS * 2;
  static constexpr int CVT_BYTES = FP8 ? kTok * QS * 2 + (LATENT ? 0 : kTok * VS * 2) : 0;
  static constexpr int SMEM = Q_BYTES + kStagesTC * STAGE + CVT_BYTES;
};

template <int DQK, int DV, bool FP8, bool LATENT>
__global__ void __launch_bounds__(TCShape<DQK, DV, FP8, LATENT>::THREADS)
    partial_tc_kernel(const TCParams p) {
  using S = TCShape<DQK, DV, FP8, LATENT>;
  extern __shared__ __align__(128) uint8_t smem[];
  dependents_may_launch();  // the merge that follows only waits for this grid
  uint8_t *sQ = smem;
  uint8_t *sStage = smem + S::Q_BYTES;
  uint8_t *sCvt = sStage + kStagesTC * S::STAGE;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wrow = (warp & 3) * 16;  // this warp's first query row in the tile
  const int dvt = warp >> 2;         // this warp's dv slice
  const psd_work_item it = p.items[blockIdx.x];
  const int kv = blockIdx.y;
  const int row0 = blockIdx.z * kRows;

  // ---- query tile [64][DQK] bf16, padded rows; rows past G_cta are zero
  for (int c = tid; c < kRows * (DQK / 8); c += S::THREADS) {
    const int j = c / (DQK / 8), cc = c - j * (DQK / 8);
    const int g = row0 + j;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (g < p.G_cta) {
      const int m = g / p.Gm;
      const int qb = it.q_index >= 0 ? it.q_index : __ldg(p.members + m);
      const int head = kv * p.Gm + (g - m * p.Gm);
      v = __ldg(reinterpret_cast<const uint4 *>(p.q + (int64_t(qb) * p.Hq_req + head) * DQK) + cc);
    }
    *reinterpret_cast<uint4 *>(sQ + (size_t(j) * S::QS + cc * 8) * 2) = v;
  }

  const int n_tiles = (it.n_tokens + kTok - 1) / kTok;
  const int P = p.page_size;
  const int64_t k_tok_stride = int64_t(p.Hkv) * DQK * S::ESZ;  // bytes between slots
  const int64_t v_tok_stride = int64_t(p.Hkv) * DV * S::ESZ;

  auto load_tile = [&](int ti) {
    uint8_t *st = sStage + (ti % kStagesTC) * S::STAGE;
    constexpr int KCH = DQK * S::ESZ / 16;  // 16-byte chunks per K row
    constexpr int VCH = LATENT ? 0 : DV * S::ESZ / 16;
    for (int c = tid; c < kTok * (KCH + VCH); c += S::THREADS) {
      const bool isv = c >= kTok * KCH;
      const int cc0 = isv ? c - kTok * KCH : c;
      const int ch = isv ? VCH : KCH;
      const int r = cc0 / ch, cc = cc0 - r * ch;
      const int t = ti * kTok + r;
      const uint8_t *src = p.k_pool;
      uint32_t bytes = 0;
      if (t < it.n_tokens) {
        const int id = __ldg(p.page_indices + it.page_off + t / P);
        if (id >= 0 && int64_t(id) < p.num_pages) {
          const int64_t slot = int64_t(id) * P + (t % P);
          src = isv ? p.v_pool + slot * v_tok_stride + int64_t(kv) * DV * S::ESZ + cc * 16
                    : p.k_pool + slot * k_tok_stride + int64_t(kv) * DQK * S::ESZ + cc * 16;
          bytes = 16;
        } else {
          raise_fault(p.fault, PSD_FAULT_PAGE_ID);
        }
      }
      uint32_t dst;
      if (FP8)
        dst = smem_u32(st + (isv ? S::K_STAGE : 0) + (isv ? r * DV : r * DQK) + cc * 16);
      else
        dst = smem_u32(st + (isv ? S::K_STAGE + r * S::VS * 2 : r * S::QS * 2) + cc * 16);
      cp_async16(dst, src, bytes);
    }
  };

#pragma unroll
  for (int s = 0; s < kStagesTC - 1; ++s) {
    if (s < n_tiles) load_tile(s);
    cp_async_commit();
  }

  constexpr int NT = S::DVT / 8;  // n8 tiles of the output slice
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {neg_inf(), neg_inf()};
  float l_run[2] = {0.f, 0.f};

  for (int ti = 0; ti < n_tiles; ++ti) {
    cp_async_wait<kStagesTC - 2>();
    __syncthreads();
    if (ti + kStagesTC - 1 < n_tiles) load_tile(ti + kStagesTC - 1);
    cp_async_commit();

    const uint8_t *st = sStage + (ti % kStagesTC) * S::STAGE;
    const uint8_t *kt;  // padded bf16 [16][QS]
    const uint8_t *vt;  // padded bf16 [16][VS or QS], already offset to column 0
    int vstride;
    if (FP8) {
      for (int c = tid; c < kTok * (DQK / 8); c += S::THREADS) {
        const int r = c / (DQK / 8), cc = c - r * (DQK / 8);
        const uint2 raw = *reinterpret_cast<const uint2 *>(st + r * DQK + cc * 8);
        *reinterpret_cast<uint4 *>(sCvt + (size_t(r) * S::QS + cc * 8) * 2) = e4m3x8_to_bf16x8(raw);
      }
      if (!LATENT) {
        uint8_t *cv = sCvt + kTok * S::QS * 2;
        for (int c = tid; c < kTok * (DV / 8); c += S::THREADS) {
          const int r = c / (DV / 8), cc = c - r * (DV / 8);
          const uint2 raw = *reinterpret_cast<const uint2 *>(st + S::K_STAGE + r * DV + cc * 8);
          *reinterpret_cast<uint4 *>(cv + (size_t(r) * S::VS + cc * 8) * 2) = e4m3x8_to_bf16x8(raw);
        }
      }
      __syncthreads();
      kt = sCvt;
      vt = LATENT ? sCvt : sCvt + kTok * S::QS * 2;
      vstride = LATENT ? S::QS : S::VS;
    } else {
      kt = st;
      vt = LATENT ? st : st + S::K_STAGE;
      vstride = LATENT ? S::QS : S::VS;
    }

    // ---- S = Q K^T for this warp's 16 rows and the tile's 16 tokens
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const uint32_t qa = smem_u32(sQ + (size_t(wrow + (lane & 15)) * S::QS + (lane >> 4) * 8) * 2);
      const int btok = (lane & 7) + ((lane >> 4) << 3);
      const int bk = ((lane >> 3) & 1) * 8;
      const uint32_t kb = smem_u32(kt + (size_t(btok) * S::QS + bk) * 2);
#pragma unroll 4
      for (int kk = 0; kk < DQK / 16; ++kk) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(qa + kk * 32, a0, a1, a2, a3);
        ldsm_x4(kb + kk * 32, b0, b1, b2, b3);
        mma_bf16(s[0], a0, a1, a2, a3, b0, b1);
        mma_bf16(s[1], a0, a1, a2, a3, b2, b3);
      }
    }
    // ---- scale, mask, online softmax (rows r0 = lane/4 and r1 = lane/4 + 8)
    const int tok_base = ti * kTok + (lane & 3) * 2;
    float tmax[2] = {neg_inf(), neg_inf()};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool ok = tok_base + n * 8 + (j & 1) < it.n_tokens;
        s[n][j] = ok ? s[n][j] * p.q_scale : neg_inf();
        tmax[j >> 1] = fmaxf(tmax[j >> 1], s[n][j]);
      }
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
      tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
      const float m_new = fmaxf(m_run[h], tmax[h]);
      alpha[h] = ex2(m_run[h] - m_new);
      m_run[h] = m_new;
    }
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        s[n][j] = ex2(s[n][j] - m_run[j >> 1]);
        psum[j >> 1] += s[n][j];
      }
    l_run[0] = l_run[0] * alpha[0] + psum[0];
    l_run[1] = l_run[1] * alpha[1] + psum[1];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    // ---- O += P V  (P from the QK^T accumulators, V via transposed ldmatrix)
    const uint32_t pa0 = pack_bf16(s[0][0], s[0][1]);
    const uint32_t pa1 = pack_bf16(s[0][2], s[0][3]);
    const uint32_t pa2 = pack_bf16(s[1][0], s[1][1]);
    const uint32_t pa3 = pack_bf16(s[1][2], s[1][3]);
    {
      const int vtok = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int vcol = dvt * S::DVT + (lane >> 4) * 8;
      const uint32_t vb = smem_u32(vt + (size_t(vtok) * vstride + vcol) * 2);
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + n * 16, b0, b1, b2, b3);
        mma_bf16(o[n], pa0, pa1, pa2, pa3, b0, b1);
        mma_bf16(o[n + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
    }
  }
  cp_async_wait<0>();

  // ---- epilogue: normalise and write this warp's rows
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int g = row0 + wrow + (lane >> 2) + h * 8;
    if (g >= p.G_cta) continue;
    const int m = g / p.Gm;
    const int row = it.q_index >= 0 ? it.out_row : __ldg(p.member_row_base + m) + it.out_row;
    const int head = kv * p.Gm + (g - m * p.Gm);
    const int64_t orow = int64_t(row) * p.Hq_req + head;
    const bool live = m_run[h] != neg_inf();
    const float inv = live ? p.v_scale / l_run[h] : 0.f;
    float *dst = p.v_out + orow * DV + dvt * S::DVT + (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      *reinterpret_cast<float2 *>(dst + n * 8) = make_float2(o[n][2 * h] * inv, o[n][2 * h + 1] * inv);
    if (dvt == 0 && (lane & 3) == 0) p.lse_out[orow] = live ? m_run[h] + log2f(l_run[h]) : neg_inf();
  }
}

template <int DQK, int DV, bool FP8, bool LATENT>
psd_status launch_tc(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  using S = TCShape<DQK, DV, FP8, LATENT>;
  TCParams p;
  p.q = reinterpret_cast<const __nv_bfloat16 *>(L.q);
  p.k_pool = reinterpret_cast<const uint8_t *>(L.k_pool);
  p.v_pool = reinterpret_cast<const uint8_t *>(L.v_pool);
  p.page_indices = L.page_indices;
  p.items = L.items;
  p.members = L.members;
  p.member_row_base = L.member_row_base;
  p.v_out = L.v_out;
  p.lse_out = L.lse_out;
  p.fault = L.fault;
  p.num_pages = L.num_pages;
  p.Hq_req = L.Hq_req;
  p.Hkv = L.Hkv;
  p.page_size = L.page_size;
  p.Gm = L.Gm;
  p.G_cta = L.G_cta;
  p.q_scale = L.q_scale;
  p.v_scale = L.v_scale;
  const size_t smem = S::SMEM;
  if (smem > size_t(dev.smem_optin))
    return fail(PSD_ERR_UNSUPPORTED, "tensor-core partial needs %zu bytes of shared memory", smem);
  auto kern = partial_tc_kernel<DQK, DV, FP8, LATENT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  }
  dim3 grid(unsigned(L.num_items), unsigned(L.Hkv), unsigned((L.G_cta + kRows - 1) / kRows));
  kern<<<grid, S::THREADS, smem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "partial (tensor cores) launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

}  // namespace

bool partial_tc_supports(const PartialLaunch &p) {
  const bool fp8 = p.kv_dtype == PSD_FP8_E4M3;
  if (p.latent_v) return p.Dqk == 576 && p.Dv == 512;
  (void)fp8;
  return p.Dqk == p.Dv && (p.Dqk == 64 || p.Dqk == 128 || p.Dqk == 256);
}

psd_status launch_partial_tc(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  if (L.num_items == 0) return PSD_OK;
  const bool fp8 = L.kv_dtype == PSD_FP8_E4M3;
  if (L.latent_v) {
    if (L.Dqk == 576 && L.Dv == 512)
      return fp8 ? launch_tc<576, 512, true, true>(L, dev, s) : launch_tc<576, 512, false, true>(L, dev, s);
  } else if (L.Dqk == L.Dv) {
    switch (L.Dqk) {
      case 64: return fp8 ? launch_tc<64, 64, true, false>(L, dev, s) : launch_tc<64, 64, false, false>(L, dev, s);
      case 128: return fp8 ? launch_tc<128, 128, true, false>(L, dev, s) : launch_tc<128, 128, false, false>(L, dev, s);
      case 256: return fp8 ? launch_tc<256, 256, true, false>(L, dev, s) : launch_tc<256, 256, false, false>(L, dev, s);
      default: break;
    }
  }
  return fail(PSD_ERR_UNSUPPORTED, "tensor-core partial: Dqk %d, Dv %d, fp8 %d, latent %d", L.Dqk,
              L.Dv, int(fp8), int(L.latent_v));
}

}  // namespace psd
