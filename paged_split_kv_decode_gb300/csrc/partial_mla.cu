// K2t: split-KV partial attention for the MLA latent shape on the 5th-generation
// tensor cores (tcgen05.mma with TMEM accumulators).
//
// Shape: 128 query heads over one 576-wide latent KV head stored as fp8-e4m3 with
// a per-tensor scale; V is the first 512 columns of the same latent rows (ROCm
// ATOM PR #1701, section 3.2: fp8 latent dequantised as value * scale; mlxcel PR
// #1004, Decomposition and Merge contract sections for the split-KV partial and
// its (V, LSE) outputs in log2 units).
//
// GB300 design.  One CTA per (work item, half of the 512 V columns): its O half
// [128 x 256] f32 lives in TMEM (256 columns) beside two S buffers [128 x 32]
// (64 columns), and Q [128 x 576] bf16 stays in shared memory for the whole item
// (147 KB, 128-byte swizzle, loaded once by TMA).  Per 32-token tile:
//   * the four row warps load the tile's fp8 latent rows with 128-bit loads,
//     widen them exactly to bf16 (e4m3 -> f16 -> f32 -> bf16) into a 128B-swizzled
//     K tile (double buffered), and arrive on an mbarrier;
//   * one control thread issues S = Q K^T (36 MMAs of M=128, N=32, K=16) into TMEM
//     and commits to an mbarrier, then O += P V (2 MMAs of M=128, N=256, K=16,
//     V read MN-major straight from the same K tile);
//   * each row thread (thread = head = TMEM lane) reads its 32 scores with
//     tcgen05.ld, keeps a lazily-updated running max (O is rescaled in TMEM only
//     when the max grows by more than 2^8), writes P as bf16 into a 64B-swizzled
//     tile and sums the same rounded P into l.
// The k_scale folds into the score scale and v_scale into the output.  Two CTAs
// per item (one per V half) both compute S; the tile is read from HBM once and
// from L2 by the second CTA.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

constexpr int kTokM = 32;                       // tokens per tile
constexpr int kDqkM = 576, kDvM = 512, kDvHalf = 256, kRowsM = 128;
constexpr int kQBoxes = kDqkM / 64;             // 9 boxes of 64 columns
constexpr uint32_t kQBytes = kRowsM * kDqkM * 2;        // 147456
constexpr uint32_t kKTileBytes = kTokM * kDqkM * 2;     // 36864
constexpr uint32_t kPBytes = kRowsM * kTokM * 2;        // 8192
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK0 = kOffQ + kQBytes;
constexpr uint32_t kOffK1 = kOffK0 + kKTileBytes;
constexpr uint32_t kOffP = kOffK1 + kKTileBytes;
constexpr uint32_t kOffBar = kOffP + kPBytes;          // 229376
constexpr uint32_t kSmemMLA = kOffBar + 256 + 1024;    // barriers + alignment slack
constexpr int kThreadsM = 160;                  // 4 row warps + 1 control warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;      // S buffer b at kColS + 32 b
constexpr float kLazyRescale = 8.f;             // log2 units

// mbarrier slots (uint64 each) at kOffBar
enum { BQ = 0, BK0 = 1, BK1 = 2, BS0 = 3, BS1 = 4, BP = 5, BPV0 = 6, BPV1 = 7, BSLOT = 8 };

struct MLAParams {
  const uint8_t *k_pool;
  const int32_t *page_indices;
  const psd_work_item *items;
  const int32_t *order;
  float *v_out;
  float *lse_out;
  int32_t *fault;
  int64_t num_pages;
  int Hq_req, page_size;
  float q_scale, v_scale;
};

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(swz & 7u) << 61);
}
// kind::f16 instruction descriptor: f32 accumulate, bf16 A and B.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
#define PSD_TMEM_LD32(taddr, r)                                                                        \
  asm volatile(                                                                                        \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15," \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                      \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),          \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),      \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),   \
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),   \
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])                                           \
      : "r"(taddr))
#define PSD_TMEM_ST32(taddr, r)                                                                        \
  asm volatile(                                                                                        \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15," \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),          \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),        \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),  \
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),            \
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),            \
      "r"(r[30]), "r"(r[31])                                                                         \
      : "memory")
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// 8 e4m3 codes -> 8 bf16, exact.
__device__ __forceinline__ uint4 cvt8(uint32_t w0, uint32_t w1) {
  const float2 a = e4m3x2_to_float2(w0 & 0xffffu), b = e4m3x2_to_float2(w0 >> 16);
  const float2 c = e4m3x2_to_float2(w1 & 0xffffu), d = e4m3x2_to_float2(w1 >> 16);
  return make_uint4(pack2_bf16(a.x, a.y), pack2_bf16(b.x, b.y), pack2_bf16(c.x, c.y), pack2_bf16(d.x, d.y));
}

__global__ void __launch_bounds__(kThreadsM, 1)
    partial_mla_kernel(const __grid_constant__ CUtensorMap tmQ, const MLAParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + BSLOT);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const psd_work_item it = p.items[p.order ? __ldg(p.order + blockIdx.x) : blockIdx.x];
  const int half = blockIdx.z;                    // which 256 V columns
  const int P = p.page_size;
  const int n_tiles = (it.n_tokens + kTokM - 1) / kTokM;

  if (tid == 0) {
    mbar_init(bar(BQ), 1);
    mbar_init(bar(BK0), 128);
    mbar_init(bar(BK1), 128);
    mbar_init(bar(BS0), 1);
    mbar_init(bar(BS1), 1);
    mbar_init(bar(BP), 128);
    mbar_init(bar(BPV0), 1);
    mbar_init(bar(BPV1), 1);
    fence_mbar_init();
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 4) {
    // ------------------------------------------------------------ control thread
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(BQ), kQBytes);
#pragma unroll 1
      for (int b = 0; b < kQBoxes; ++b)
        tma_load_3d(smem_u32(sm + kOffQ + b * (kRowsM * 128)), &tmQ, b * 64, 0, it.q_index, bar(BQ));
      bool ok = mbar_wait(bar(BQ), 0, p.fault);
      const uint32_t id_qk = idesc_bf16(128, kTokM, false, false);
      const uint32_t id_pv = idesc_bf16(128, kDvHalf, false, true);
      const uint32_t q_base = smem_u32(sm + kOffQ);
      const uint32_t p_base = smem_u32(sm + kOffP);
      for (int i = 0; ok && i <= n_tiles; ++i) {
        if (i < n_tiles) {  // S(i) = Q K(i)^T
          const int b = i & 1;
          ok = mbar_wait(bar(BK0 + b), uint32_t(i >> 1) & 1u, p.fault);
          if (!ok) break;
          tc_fence_after();
          const uint32_t k_base = smem_u32(sm + (b ? kOffK1 : kOffK0));
#pragma unroll 4
          for (int k16 = 0; k16 < kDqkM / 16; ++k16) {
            const uint32_t ko = (k16 & 3) * 32u;  // 16 columns within the 64-column box
            umma(tmem + kColS + 32 * b,
                 smem_desc(q_base + (k16 >> 2) * (kRowsM * 128) + ko, 16, 1024, 2),
                 smem_desc(k_base + (k16 >> 2) * (kTokM * 128) + ko, 16, 1024, 2), id_qk, k16 > 0);
          }
          umma_commit(bar(BS0 + b));
        }
        if (i > 0) {  // O += P(i-1) V(i-1)
          const int j = i - 1, b = j & 1;
          ok = mbar_wait(bar(BP), uint32_t(j) & 1u, p.fault);
          if (!ok) break;
          tc_fence_after();
          const uint32_t v_base = smem_u32(sm + (b ? kOffK1 : kOffK0)) + half * 4 * (kTokM * 128);
#pragma unroll
          for (int k = 0; k < kTokM / 16; ++k)
            umma(tmem + kColO, smem_desc(p_base + k * 32, 16, 512, 4),
                 smem_desc(v_base + k * 16 * 128, kTokM * 128, 1024, 2), id_pv, (j > 0 || k > 0));
          umma_commit(bar(BPV0 + b));
        }
      }
    }
  } else {
    // ---------------------------------------------------- row / converter threads
    const int row = tid;                          // head = TMEM lane
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    const int ct = tid >> 2, cq = tid & 3;        // converter: token ct, 144-column quarter cq
    uint4 raw[9];
    auto fetch = [&](int i) {                     // 144 fp8 of token ct of tile i
      const int tok = i * kTokM + ct;
      if (i < n_tiles && tok < it.n_tokens) {
        const int id = __ldg(p.page_indices + it.page_off + tok / P);
        if (id >= 0 && int64_t(id) < p.num_pages) {
          const uint4 *src = reinterpret_cast<const uint4 *>(
              p.k_pool + (int64_t(id) * P + tok % P) * kDqkM + cq * 144);
#pragma unroll
          for (int k = 0; k < 9; ++k) raw[k] = __ldg(src + k);
          return;
        }
        atomicOr(p.fault, PSD_FAULT_PAGE_ID);
      }
#pragma unroll
      for (int k = 0; k < 9; ++k) raw[k] = make_uint4(0u, 0u, 0u, 0u);
    };
    auto convert = [&](int i) {                   // raw -> bf16 K tile i (128B swizzle)
      uint8_t *kt = sm + ((i & 1) ? kOffK1 : kOffK0);
      const uint32_t w[36] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w,
                              raw[2].x, raw[2].y, raw[2].z, raw[2].w, raw[3].x, raw[3].y, raw[3].z, raw[3].w,
                              raw[4].x, raw[4].y, raw[4].z, raw[4].w, raw[5].x, raw[5].y, raw[5].z, raw[5].w,
                              raw[6].x, raw[6].y, raw[6].z, raw[6].w, raw[7].x, raw[7].y, raw[7].z, raw[7].w,
                              raw[8].x, raw[8].y, raw[8].z, raw[8].w};
#pragma unroll
      for (int j = 0; j < 18; ++j) {
        const int c = cq * 18 + j;                // 8-column chunk of the 576
        *reinterpret_cast<uint4 *>(kt + (c >> 3) * (kTokM * 128) + ct * 128 +
                                   (((c & 7) ^ (ct & 7)) << 4)) = cvt8(w[2 * j], w[2 * j + 1]);
      }
      fence_proxy_async();
      mbar_arrive(bar(BK0 + (i & 1)));
    };

    float m_ref = neg_inf(), l_sum = 0.f;
    bool ok = true;
    if (n_tiles > 0) {
      fetch(0);
      convert(0);
      fetch(1);
    }
    for (int i = 0; i < n_tiles && ok; ++i) {
      // convert tile i+1 once PV(i-1) has released its buffer
      if (i + 1 < n_tiles) {
        if (i >= 1) ok = mbar_wait(bar(BPV0 + ((i - 1) & 1)), uint32_t((i - 1) >> 1) & 1u, p.fault);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        convert(i + 1);
        fetch(i + 2);
      }
      // scores of tile i
      ok = mbar_wait(bar(BS0 + (i & 1)), uint32_t(i >> 1) & 1u, p.fault);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[32];
      PSD_TMEM_LD32(lane_base + kColS + 32 * (i & 1), r);
      tmem_ld_wait();
      const int valid = min(kTokM, it.n_tokens - i * kTokM);
      float s[32];
      float mt = neg_inf();
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s[c] = c < valid ? __uint_as_float(r[c]) * p.q_scale : neg_inf();
        mt = fmaxf(mt, s[c]);
      }
      // PV(i-1) must be done before P is rewritten or O rescaled
      if (i >= 1) {
        ok = mbar_wait(bar(BPV0 + ((i - 1) & 1)), uint32_t((i - 1) >> 1) & 1u, p.fault);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      const bool grow = mt > m_ref + kLazyRescale;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? mt : m_ref;
        if (i >= 1) {  // rescale this warp's O rows in TMEM
          const float alpha = ex2(m_ref - m_new);
#pragma unroll 1
          for (int cb = 0; cb < kDvHalf / 32; ++cb) {
            uint32_t o[32];
            PSD_TMEM_LD32(lane_base + kColO + cb * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            PSD_TMEM_ST32(lane_base + kColO + cb * 32, o);
          }
          tmem_st_wait();
          l_sum *= alpha;
        }
        m_ref = m_new;
      }
      // P = 2^(s - m_ref) as bf16 (64B-swizzled [128 x 32]); l sums the rounded P
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        pk[c] = pack2_bf16(ex2(s[2 * c] - m_ref), ex2(s[2 * c + 1] - m_ref));
        l_sum += bf16_lo(pk[c]) + bf16_hi(pk[c]);
      }
      uint8_t *prow = sm + kOffP;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const uint32_t lin = uint32_t(row) * 64u + ch * 16u;
        *reinterpret_cast<uint4 *>(prow + (lin ^ (((lin >> 7) & 3u) << 4))) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(bar(BP));
    }
    // epilogue: O / l for this row and V half
    if (ok && n_tiles > 0) {
      const int j = n_tiles - 1;
      ok = mbar_wait(bar(BPV0 + (j & 1)), uint32_t(j >> 1) & 1u, p.fault);
    }
    if (__all_sync(0xffffffffu, ok) && n_tiles > 0) {
      tc_fence_after();
      const int64_t orow = int64_t(it.out_row) * p.Hq_req + row;
      float *dst = p.v_out + orow * kDvM + half * kDvHalf;
      const float inv = p.v_scale / l_sum;
#pragma unroll 1
      for (int cb = 0; cb < kDvHalf / 32; ++cb) {
        uint32_t o[32];
        PSD_TMEM_LD32(lane_base + kColO + cb * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<float4 *>(dst + cb * 32 + c) =
              make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                          __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
      }
      if (half == 0) p.lse_out[orow] = m_ref + log2f(l_sum);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

bool encode_q_map(CUtensorMap *map, const DeviceInfo &dev, const void *q, int batch, int Hq) {
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(dev.encode_tiled);
  if (!encode) return false;
  cuuint64_t dims[3] = {cuuint64_t(kDqkM), cuuint64_t(Hq), cuuint64_t(batch)};
  cuuint64_t strides[2] = {cuuint64_t(kDqkM) * 2, cuuint64_t(Hq) * kDqkM * 2};
  cuuint32_t box[3] = {64, cuuint32_t(kRowsM), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool partial_mla_supports(const PartialLaunch &L) {
  return L.latent_v && L.kv_dtype == PSD_FP8_E4M3 && L.Dqk == kDqkM && L.Dv == kDvM &&
         L.G_cta == kRowsM && L.Hq_req == kRowsM && L.Hkv == 1 && L.page_size % kTokM == 0;
}

psd_status launch_partial_mla(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  if (L.num_items == 0) return PSD_OK;
  if (size_t(dev.smem_optin) < kSmemMLA)
    return fail(PSD_ERR_UNSUPPORTED, "MLA tcgen05 partial needs %u bytes of shared memory", kSmemMLA);
  CUtensorMap tmQ;
  if (!encode_q_map(&tmQ, dev, L.q, L.q_batch, L.Hq_req))
    return fail(PSD_ERR_CUDA, "cuTensorMapEncodeTiled failed for q");
  MLAParams p;
  p.k_pool = reinterpret_cast<const uint8_t *>(L.k_pool);
  p.page_indices = L.page_indices;
  p.items = L.items;
  p.order = L.order;
  p.v_out = L.v_out;
  p.lse_out = L.lse_out;
  p.fault = L.fault;
  p.num_pages = L.num_pages;
  p.Hq_req = L.Hq_req;
  p.page_size = L.page_size;
  p.q_scale = L.q_scale;
  p.v_scale = L.v_scale;
  cudaError_t e = cudaFuncSetAttribute(partial_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kSmemMLA));
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  const dim3 grid(static_cast<unsigned>(L.num_items), 1, 2);
  partial_mla_kernel<<<grid, kThreadsM, kSmemMLA, s>>>(tmQ, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "partial (MLA tcgen05) launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

}  // namespace psd
