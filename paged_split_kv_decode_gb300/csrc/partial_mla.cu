// K2t: split-KV partial attention for the MLA latent shape on the 5th-generation
// tensor cores (tcgen05.mma with TMEM accumulators).
//
// Shape: 128 query heads over one 576-wide latent KV head stored as fp8-e4m3 with
// a per-tensor scale; V is the first 512 columns of the same latent rows (ROCm
// ATOM PR #1701, section 3.2: fp8 latent dequantised as value * scale; mlxcel PR
// #1004, Decomposition and Merge contract sections for the split-KV partial and
// its (V, LSE) outputs in log2 units).
//
// GB300 design.  One CTA per (work item, half of the 512 V columns).  TMEM (512
// columns) holds the O half [128 x 256] f32, two S buffers [128 x 32] f32, and the
// first 384 of Q's 576 columns as the MMA's A operand (f16 pairs); the remaining
// 192 Q columns stay in shared memory (128-byte swizzle).  Keeping most of Q in
// TMEM is what makes 32-token tiles pay: with Q in shared memory every M=128,
// N=32 MMA re-read a 4 KB slice of it and the QK^T steps were bound by
// shared-memory bandwidth.  The MMAs run in f16: e4m3 codes widen exactly to f16
// with one hardware conversion per pair, Q is converted from bf16 once per item
// (exact for |q| in [2^-14, 65504]; overflow sets a fault bit), and P in f16
// keeps 3 more mantissa bits than bf16.  Warp roles, per 32-token tile:
//   * converter warps 4-7 load the tile's fp8 latent rows with 128-bit loads (two
//     tiles ahead) and widen them into a 128B-swizzled f16 K tile (2 buffers,
//     freed when S is done) and this CTA's V half (3 buffers, freed when PV is
//     done);
//   * the control thread (warp 8) issues S = Q K^T (24 MMAs with A in TMEM, 12
//     from shared memory; M=128, N=32, K=16) and O += P V (2 MMAs of M=128, N=256,
//     K=16, V MN-major), each group committed to an mbarrier;
//   * row warps 0-3 (thread = head = TMEM lane) first move their Q row into TMEM,
//     then per tile read 32 scores with tcgen05.ld, keep a lazily-updated running
//     max (O is rescaled in TMEM only when the max grows by more than 2^8), write
//     P as f16 into a 64B-swizzled tile and sum the same rounded P into l.
// The k_scale folds into the score scale and v_scale into the output.  The two CTAs
// of an item (one per V half) both compute S; the tile is read from HBM once and
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
constexpr int kQHeadBoxes = 6;                  // Q[:, 0:384] moves to TMEM
constexpr uint32_t kQBytes = kRowsM * kDqkM * 2;        // 147456 (TMA landing)
constexpr uint32_t kQBoxBytes = kRowsM * 128;           // 16384
constexpr uint32_t kKTileBytes = kTokM * kDqkM * 2;     // 36864
constexpr uint32_t kVTileBytes = kTokM * kDvHalf * 2;   // 16384
constexpr uint32_t kPBytes = kRowsM * kTokM * 2;        // 8192
// Shared memory: Q tail (3 boxes) | K0 | K1 | V0 | V1 | V2 | P | barriers.  Q lands
// by TMA with its 6 head boxes over K0..V1, which are free until the head has
// moved to TMEM.
constexpr uint32_t kOffQT = 0;
constexpr uint32_t kOffK0 = kOffQT + 3 * kQBoxBytes;    // 49152
constexpr uint32_t kOffK1 = kOffK0 + kKTileBytes;
constexpr uint32_t kOffV0 = kOffK1 + kKTileBytes;
constexpr uint32_t kOffP = kOffV0 + 3 * kVTileBytes;
constexpr uint32_t kOffQHead = kOffK0;                  // 6 landing boxes
constexpr uint32_t kOffBar = kOffP + kPBytes;
constexpr uint32_t kSmemMLA = kOffBar + 256 + 1024;     // barriers + alignment slack
static_assert(kOffQHead + kQHeadBoxes * kQBoxBytes <= kOffP, "Q head landing overlaps P");
constexpr int kThreadsM = 288;                  // 4 row + 4 converter + 1 control warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 320;  // S buffer b at kColS + 32 b
constexpr float kLazyRescale = 8.f;             // log2 units

// mbarrier slots (uint64 each) at kOffBar
enum { BQ = 0, BQREADY = 1, BK0 = 2, BK1 = 3, BS0 = 4, BS1 = 5, BP = 6, BPV0 = 7, BPV1 = 8, BPV2 = 9,
       BSLOT = 10 };

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
// kind::f16 instruction descriptor: f32 accumulate, f16 A and B.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// A operand in TMEM (f16 pairs per 32-bit column, row m in lane m), accumulating.
__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Accumulating form (enable-input-d always set).
__device__ __forceinline__ void umma_acc(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.eq.u32 p, 1, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc)
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

__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float f16_lo(uint32_t w) { return __low2float(*reinterpret_cast<__half2 *>(&w)); }
__device__ __forceinline__ float f16_hi(uint32_t w) { return __high2float(*reinterpret_cast<__half2 *>(&w)); }
// Two e4m3 codes (low 16 bits) -> f16x2, exact (hardware conversion).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  uint32_t h2;
  asm("{\n\t.reg .b16 lo;\n\tmov.b32 {lo, _}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(h2) : "r"(w));
  return h2;
}
// 8 e4m3 codes -> 8 f16, exact.
__device__ __forceinline__ uint4 cvt8(uint32_t w0, uint32_t w1) {
  return make_uint4(e4m3x2_to_f16x2(w0 & 0xffffu), e4m3x2_to_f16x2(w0 >> 16), e4m3x2_to_f16x2(w1 & 0xffffu),
                    e4m3x2_to_f16x2(w1 >> 16));
}
// 8 bf16 -> 8 f16 (exact inside the f16 range); *bad is set on overflow.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, bool *bad) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float a = bf16_lo(w[k]), b = bf16_hi(w[k]);
    o[k] = pack2_f16(a, b);
    *bad |= (fabsf(a) > 65504.f) | (fabsf(b) > 65504.f);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(kThreadsM, 1)
    partial_mla_kernel(const __grid_constant__ CUtensorMap tmQ, const MLAParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  dependents_may_launch();  // the merge that follows only waits for this grid
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
    mbar_init(bar(BQREADY), 256);
    mbar_init(bar(BK0), 128);
    mbar_init(bar(BK1), 128);
    mbar_init(bar(BS0), 1);
    mbar_init(bar(BS1), 1);
    mbar_init(bar(BP), 128);
    mbar_init(bar(BPV0), 1);
    mbar_init(bar(BPV1), 1);
    mbar_init(bar(BPV2), 1);
    fence_mbar_init();
  }
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 8) {
    // ------------------------------------------------------------ control thread
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(BQ), kQBytes);
#pragma unroll 1
      for (int b = 0; b < kQBoxes; ++b) {
        const uint32_t dst = b < kQHeadBoxes ? kOffQHead + b * kQBoxBytes : kOffQT + (b - kQHeadBoxes) * kQBoxBytes;
        tma_load_3d(smem_u32(sm + dst), &tmQ, b * 64, 0, it.q_index, bar(BQ));
      }
      bool ok = mbar_wait(bar(BQREADY), 0, p.fault);  // head in TMEM, tail in f16
      tc_fence_after();
      const uint32_t id_qk = idesc_f16(128, kTokM, false, false);
      const uint32_t id_pv = idesc_f16(128, kDvHalf, false, true);
      // Base descriptors, built once; operand steps add compile-time offsets (>> 4)
      // to the start-address field, which never carries out of it (< 256 KB).
      const uint64_t qtd = smem_desc(smem_u32(sm + kOffQT), 16, 1024, 2);
      const uint64_t kd0 = smem_desc(smem_u32(sm + kOffK0), 16, 1024, 2);
      const uint64_t kd1 = smem_desc(smem_u32(sm + kOffK1), 16, 1024, 2);
      const uint64_t pd = smem_desc(smem_u32(sm + kOffP), 16, 512, 4);
      const uint64_t vd0 = smem_desc(smem_u32(sm + kOffV0), kTokM * 128, 1024, 2);
      for (int i = 0; ok && i <= n_tiles; ++i) {
        if (i < n_tiles) {  // S(i) = Q K(i)^T: 24 steps with A in TMEM, 12 from shared memory
          const int b = i & 1;
          ok = mbar_wait(bar(BK0 + b), uint32_t(i >> 1) & 1u, p.fault);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kdb = b ? kd1 : kd0;
          const uint32_t d_s = tmem + kColS + 32 * b;
          umma_tmem_a(d_s, tmem + kColQ, kdb, id_qk, 0);
#pragma unroll
          for (int k16 = 1; k16 < 4 * kQHeadBoxes; ++k16)
            umma_tmem_a(d_s, tmem + kColQ + 8 * k16, kdb + (((k16 >> 2) * (kTokM * 128) + (k16 & 3) * 32) >> 4),
                        id_qk, 1);
#pragma unroll
          for (int k16 = 4 * kQHeadBoxes; k16 < kDqkM / 16; ++k16)
            umma_acc(d_s, qtd + ((((k16 >> 2) - kQHeadBoxes) * kQBoxBytes + (k16 & 3) * 32) >> 4),
                     kdb + (((k16 >> 2) * (kTokM * 128) + (k16 & 3) * 32) >> 4), id_qk);
          umma_commit(bar(BS0 + b));
        }
        if (i > 0) {  // O += P(i-1) V(i-1)
          const int j = i - 1, vb = j % 3;
          ok = mbar_wait(bar(BP), uint32_t(j) & 1u, p.fault);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vdb = vd0 + ((vb * kVTileBytes) >> 4);
          umma(tmem + kColO, pd, vdb, id_pv, j > 0);
#pragma unroll
          for (int k = 1; k < kTokM / 16; ++k)
            umma_acc(tmem + kColO, pd + ((k * 32) >> 4), vdb + ((k * 16 * 128) >> 4), id_pv);
          umma_commit(bar(BPV0 + vb));
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ converter warps
    const int ctid = tid - 128;
    const int ct = ctid >> 2, cq = ctid & 3;      // token ct of a tile, 144-column quarter cq
    // Q tail: bf16 -> f16 in place (same 2-byte swizzled layout)
    bool ok = mbar_wait(bar(BQ), 0, p.fault);
    bool bad = false;
    if (ok) {
      for (int c = ctid; c < 3 * int(kQBoxBytes) / 16; c += 128) {
        uint4 *q16 = reinterpret_cast<uint4 *>(sm + kOffQT) + c;
        *q16 = bf16x8_to_f16x8(*q16, &bad);
      }
    }
    if (bad) atomicOr(p.fault, PSD_FAULT_RANGE);
    fence_proxy_async();
    mbar_arrive(bar(BQREADY));
    // the K/V buffers hold the Q head until the row warps have moved it to TMEM
    ok = ok && mbar_wait(bar(BQREADY), 0, p.fault);
    auto fetch = [&](uint4 (&raw)[9], int i) {  // 144 fp8 of token ct of tile i
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
    // Tile i is widened from `raw` into K buffer i%2 (all 576 columns, for QK) and
    // V buffer i%3 (this CTA's 256 V columns, for PV); `raw` is then refilled with
    // tile i + 2, so two tiles' loads are always in flight.
    auto step = [&](uint4 (&raw)[9], int i) {
      if (i >= 2) {  // QK(i-2) released the K buffer
        ok = mbar_wait(bar(BS0 + (i & 1)), uint32_t((i - 2) >> 1) & 1u, p.fault);
        if (!__all_sync(0xffffffffu, ok)) return false;
      }
      if (i >= 3) {  // PV(i-3) released the V buffer
        ok = mbar_wait(bar(BPV0 + i % 3), uint32_t((i - 3) / 3) & 1u, p.fault);
        if (!__all_sync(0xffffffffu, ok)) return false;
      }
      uint8_t *kt = sm + ((i & 1) ? kOffK1 : kOffK0);
      uint8_t *vt = sm + kOffV0 + (i % 3) * kVTileBytes;
#pragma unroll
      for (int j = 0; j < 18; ++j) {
        const int c = cq * 18 + j;                // 8-column chunk of the 576
        const uint4 r = raw[j >> 1];
        const uint4 h = cvt8((j & 1) ? r.z : r.x, (j & 1) ? r.w : r.y);
        const uint32_t sw = (((c & 7) ^ (ct & 7)) << 4) + ct * 128;
        *reinterpret_cast<uint4 *>(kt + (c >> 3) * (kTokM * 128) + sw) = h;
        const int cv = c - 32 * half;             // V column chunk of this CTA's half
        if (cv >= 0 && cv < 32) *reinterpret_cast<uint4 *>(vt + (cv >> 3) * (kTokM * 128) + sw) = h;
      }
      fence_proxy_async();
      mbar_arrive(bar(BK0 + (i & 1)));
      fetch(raw, i + 2);
      return true;
    };
    uint4 rawA[9], rawB[9];
    fetch(rawA, 0);
    fetch(rawB, 1);
    for (int i = 0; i < n_tiles && ok; i += 2) {
      if (!step(rawA, i)) break;
      if (i + 1 < n_tiles && !step(rawB, i + 1)) break;
    }
  } else {
    // ------------------------------------------------------------------ row warps
    const int row = tid;                          // head = TMEM lane
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    // Q head (columns 0..383) of this row: bf16 from the landing boxes -> f16 pairs
    // -> TMEM columns kColQ + 32 b (box b), the layout the MMA reads A from.
    bool ok = mbar_wait(bar(BQ), 0, p.fault);
    if (__all_sync(0xffffffffu, ok)) {
      bool bad = false;
#pragma unroll 1
      for (int b = 0; b < kQHeadBoxes; ++b) {
        uint32_t qw[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4 *>(sm + kOffQHead + b * kQBoxBytes + row * 128 +
                                                           ((c ^ (row & 7)) << 4));
          const uint4 h = bf16x8_to_f16x8(v, &bad);
          qw[4 * c] = h.x;
          qw[4 * c + 1] = h.y;
          qw[4 * c + 2] = h.z;
          qw[4 * c + 3] = h.w;
        }
        PSD_TMEM_ST32(lane_base + kColQ + 32 * b, qw);
      }
      tmem_st_wait();
      if (bad) atomicOr(p.fault, PSD_FAULT_RANGE);
    }
    tc_fence_before();
    mbar_arrive(bar(BQREADY));
    float m_ref = neg_inf(), l_sum = 0.f;
    for (int i = 0; i < n_tiles && ok; ++i) {
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
        ok = mbar_wait(bar(BPV0 + (i - 1) % 3), uint32_t((i - 1) / 3) & 1u, p.fault);
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
      // P = 2^(s - m_ref) as f16 (64B-swizzled [128 x 32]); l sums the rounded P
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        pk[c] = pack2_f16(ex2(s[2 * c] - m_ref), ex2(s[2 * c + 1] - m_ref));
        l_sum += f16_lo(pk[c]) + f16_hi(pk[c]);
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
      ok = mbar_wait(bar(BPV0 + j % 3), uint32_t(j / 3) & 1u, p.fault);
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
  if (warp == 8) {
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
