// K2t: split-KV partial attention for the MLA latent shape on the 5th-generation
// tensor cores (tcgen05.mma with TMEM accumulators).
//
// Shape: 128 query heads over one 576-wide latent KV head stored as fp8-e4m3 with
// a per-tensor scale; V is the first 512 columns of the same latent rows (ROCm
// ATOM PR #1701, section 3.2: fp8 latent dequantised as value * scale; mlxcel PR
// #1004, Decomposition and Merge contract sections for the split-KV partial and
// its (V, LSE) outputs in log2 units).
//
// GB300 design.  One CTA per (work item, half of the 512 V columns), 64-token
// tiles.  TMEM (512 columns) holds the O half [128 x 256] f32, S [128 x 64] f32 and
// the first 384 of Q's 576 columns as the MMA's A operand (f16 pairs); the other
// 192 Q columns stay in shared memory (128-byte swizzle).  An M=128, K=16 MMA costs
// about the same issue time at N=32 and N=64, so 64-token tiles halve the QK^T
// instruction count per token; to fit them, the f16 K tile is never whole in
// shared memory: it streams through a ring of 64-column blocks [64 tokens x 64],
// each released by the commit of the four MMAs that read it.  The MMAs run in
// f16: e4m3 codes widen exactly to f16 with one hardware conversion per pair, Q is
// converted from bf16 once per item (exact for |q| in [2^-14, 65504]; overflow
// sets a fault bit), and P in f16 keeps 3 more mantissa bits than bf16.  Roles:
//   * eight converter warps, in two groups taking alternate tiles, hold a tile of
//     fp8 latent rows in registers (128-bit loads issued two tiles ahead) and
//     widen them block by block into the K ring and into this CTA's V half (3
//     tile buffers, freed when PV is done);
//   * the control warp issues S = Q K^T block by block (24 MMAs with
//     A in TMEM, 12 from shared memory; M=128, N=64, K=16) and O += P V (4 MMAs of
//     M=128, N=256, K=16, V MN-major), each group committed to an mbarrier;
//   * row warps 0-3 (thread = head = TMEM lane) first move their Q row into TMEM,
//     then per tile read 64 scores with tcgen05.ld, free S, keep a lazily-updated
//     running max (O is rescaled in TMEM only when the max grows by more than 2^8),
//     write P as f16 into a 128B-swizzled tile and sum P (in f32) into l.
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

constexpr int kTokM = 64;                       // tokens per tile
constexpr int kDqkM = 576, kDvM = 512, kDvHalf = 256, kRowsM = 128;
constexpr int kQBoxes = kDqkM / 64;             // 9 boxes of 64 columns
constexpr int kKBlocks = kDqkM / 64;            // 9 K blocks of 64 columns per tile
constexpr int kQHeadBoxes = 6;                  // Q[:, 0:384] moves to TMEM
constexpr int kGroupSlots = 4;                  // K ring slots of each converter group
constexpr int kRing = 2 * kGroupSlots;          // K ring slots
constexpr int kVBufs = 3;                       // V tile buffers
constexpr uint32_t kQBytes = kRowsM * kDqkM * 2;        // 147456 (TMA landing)
constexpr uint32_t kQBoxBytes = kRowsM * 128;           // 16384
constexpr uint32_t kKBlockBytes = kTokM * 128;          // 8192: 64 tokens x 64 f16
constexpr uint32_t kVTileBytes = kTokM * kDvHalf * 2;   // 32768
constexpr uint32_t kPBytes = kRowsM * kTokM * 2;        // 16384
// Shared memory: Q tail (3 boxes) | K ring | V0 | V1 | V2 | P | barriers.  Q lands by
// TMA with its 6 head boxes over the K ring and V, free until the head is in TMEM.
constexpr uint32_t kOffQT = 0;
constexpr uint32_t kOffK = kOffQT + 3 * kQBoxBytes;     // 49152
constexpr uint32_t kOffV0 = kOffK + kRing * kKBlockBytes;
constexpr uint32_t kOffP = kOffV0 + kVBufs * kVTileBytes;
constexpr uint32_t kOffQHead = kOffK;                   // 6 landing boxes
constexpr uint32_t kOffBar = kOffP + kPBytes;
constexpr uint32_t kSmemMLA = kOffBar + 512 + 1024;     // barriers + alignment slack
static_assert(kOffQHead + kQHeadBoxes * kQBoxBytes <= kOffP, "Q head landing overlaps P");
// Warp w runs on sub-partition w % 4.  Row warps 0-3 (one per TMEM lane quadrant);
// the control warp 4 shares sub-partition 0 only with row warp 0, since issue
// slots taken by busy warps there slow its MMA issue several-fold; the converter
// warps are 5-7, 9-11, 13, 14 (sub-partitions 1-3); warps 8 and 12 stay idle.
constexpr int kConvWarps = 8;
constexpr int kCtrlWarp = 4;
constexpr int kThreadsM = 32 * 15;
__host__ __device__ constexpr bool is_converter_warp(int w) { return w >= 5 && w <= 14 && (w & 3) != 0; }
__host__ __device__ constexpr int converter_index(int w) { return (w - 5) - (w - 4) / 4; }  // 0..7
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 320;
constexpr float kLazyRescale = 8.f;             // log2 units

// mbarrier slots (uint64 each) at kOffBar
enum { BQ = 0, BQREADY, BSFULL, BSFREE, BPFULL, BDRAIN, BPV0, BKFULL0 = BPV0 + kVBufs,
       BKEMPTY0 = BKFULL0 + kRing, BSLOT = BKEMPTY0 + kRing };
static_assert(BSLOT * 8 + 4 <= 512, "barrier area");

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
// One lane of the (converged) warp: the lowest active one.
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
  return e != 0;
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
#define PSD_TMEM_LD16(taddr, r)                                                                        \
  asm volatile(                                                                                        \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];" \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),          \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),      \
        "=r"(r[14]), "=r"(r[15])                                                                     \
      : "r"(taddr))
#define PSD_TMEM_ST16(taddr, r)                                                                        \
  asm volatile(                                                                                        \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" \
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),    \
      "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),  \
      "r"(r[15])                                                                                     \
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
    mbar_init(bar(BQREADY), 32 * kConvWarps + 128);
    mbar_init(bar(BSFULL), 1);
    mbar_init(bar(BSFREE), 4);   // one arrival per row warp
    mbar_init(bar(BPFULL), 4);
    mbar_init(bar(BDRAIN), 1);
    for (int b = 0; b < kVBufs; ++b) mbar_init(bar(BPV0 + b), 1);
    for (int r = 0; r < kRing; ++r) {
      mbar_init(bar(BKFULL0 + r), kConvWarps / 2);  // one arrival per warp of a group
      mbar_init(bar(BKEMPTY0 + r), 1);
    }
    fence_mbar_init();
  }
  if (warp == kCtrlWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == kCtrlWarp) {
    // ------------------------------------------------------------- control warp
    // The whole warp runs the loop and waits; one elected lane issues the MMAs.
    // A wait on the issuing thread alone stalls the MMAs it has queued much
    // longer, and each wait costs tensor-pipe time, so the loop waits for K
    // blocks three at a time (a group's warps arrive on blocks in order, so the
    // third block's barrier covers the first two) and never for V (the same
    // warps store V before they arrive for the tile's last K block).
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(BQ), kQBytes);
#pragma unroll 1
      for (int b = 0; b < kQBoxes; ++b) {
        const uint32_t dst = b < kQHeadBoxes ? kOffQHead + b * kQBoxBytes : kOffQT + (b - kQHeadBoxes) * kQBoxBytes;
        tma_load_3d(smem_u32(sm + dst), &tmQ, b * 64, 0, it.q_index, bar(BQ));
      }
    }
    __syncwarp();
    bool ok = __all_sync(0xffffffffu, mbar_wait(bar(BQREADY), 0, p.fault));  // head in TMEM, tail in f16
    tc_fence_after();
    const uint32_t id_qk = idesc_f16(128, kTokM, false, false);
    const uint32_t id_pv = idesc_f16(128, kDvHalf, false, true);
    // Base descriptors, built once; operand steps add offsets (>> 4) to the
    // start-address field, which never carries out of it (< 256 KB).
    const uint64_t qtd = smem_desc(smem_u32(sm + kOffQT), 16, 1024, 2);
    const uint64_t kd = smem_desc(smem_u32(sm + kOffK), 16, 1024, 2);
    const uint64_t pd = smem_desc(smem_u32(sm + kOffP), 16, 1024, 2);
    const uint64_t vd = smem_desc(smem_u32(sm + kOffV0), kTokM * 128, 1024, 2);
    const uint32_t d_s = tmem + kColS;
    for (int i = 0; ok && i <= n_tiles; ++i) {
      if (i < n_tiles) {  // S(i) = Q K(i)^T, block by block
        if (i > 0) {      // the row warps have read S(i-1)
          ok = __all_sync(0xffffffffu, mbar_wait(bar(BSFREE), uint32_t(i - 1) & 1u, p.fault));
          if (!ok) break;
        }
        // block b of tile i is block c of converter group i % 2, in that group's slots
        const int c0 = (i >> 1) * kKBlocks, sbase = (i & 1) * kGroupSlots;
#pragma unroll 1
        for (int b = 0; b < kKBlocks; ++b) {
          const int c = c0 + b, slot = sbase + c % kGroupSlots;
          if (b % 3 == 0) {  // blocks b .. b+2 are in place once block b+2 is
            const int cw = c + 2;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(BKFULL0 + sbase + cw % kGroupSlots),
                                                   uint32_t(cw / kGroupSlots) & 1u, p.fault));
            if (!ok) break;
            tc_fence_after();
          }
          if (elect_one()) {
            const uint64_t kb = kd + ((slot * kKBlockBytes) >> 4);
            if (b < kQHeadBoxes) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                umma_tmem_a(d_s, tmem + kColQ + 8 * (4 * b + j), kb + ((j * 32) >> 4), id_qk, (b | j) != 0);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                umma_acc(d_s, qtd + (((b - kQHeadBoxes) * kQBoxBytes + j * 32) >> 4), kb + ((j * 32) >> 4), id_qk);
            }
            umma_commit(bar(BKEMPTY0 + slot));
            if (b == kKBlocks - 1) umma_commit(bar(BSFULL));
          }
          __syncwarp();
        }
        if (!ok) break;
      }
      if (i > 0) {  // O += P(i-1) V(i-1)
        const int j = i - 1, vb = j % kVBufs;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(BPFULL), uint32_t(j) & 1u, p.fault));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t vdb = vd + ((vb * kVTileBytes) >> 4);
#pragma unroll
          for (int k = 0; k < kTokM / 16; ++k)
            umma(tmem + kColO, pd + ((k * 32) >> 4), vdb + ((k * 16 * 128) >> 4), id_pv, (j | k) != 0);
          umma_commit(bar(BPV0 + vb));
        }
        __syncwarp();
      }
    }
    // every MMA this warp issued has completed before TMEM is released
    if (elect_one()) umma_commit(bar(BDRAIN));
    __syncwarp();
    mbar_wait(bar(BDRAIN), 0, p.fault);
  } else if (is_converter_warp(warp)) {
    // ------------------------------------------------------------ converter warps
    const int cwi = converter_index(warp);
    const int ctid = cwi * 32 + lane;
    // Q tail: bf16 -> f16 in place (same 2-byte swizzled layout)
    bool ok = mbar_wait(bar(BQ), 0, p.fault);
    bool bad = false;
    if (ok) {
      for (int c = ctid; c < 3 * int(kQBoxBytes) / 16; c += 32 * kConvWarps) {
        uint4 *q16 = reinterpret_cast<uint4 *>(sm + kOffQT) + c;
        *q16 = bf16x8_to_f16x8(*q16, &bad);
      }
    }
    if (bad) atomicOr(p.fault, PSD_FAULT_RANGE);
    fence_proxy_async();
    mbar_arrive(bar(BQREADY));
    // Two groups of four warps take alternate tiles.  A thread of a group owns
    // token ct of its tiles and slices 2 cw, 2 cw + 1 (32 bytes) of each 64-column
    // block.  The proxy fence that publishes a block also waits for the thread's
    // global loads in flight, so a group loads its next tile (i + 2) only after
    // the last fence of tile i; the other group's tile gives those loads time to
    // land before this group's next fence.
    const int grp = cwi >> 2;
    const int gtid = ctid & 127;
    const int ct = gtid >> 1, cw = gtid & 1;
    auto source = [&](int i) -> const uint4 * {  // token ct of tile i, or nullptr
      const int tok = i * kTokM + ct;
      if (i < n_tiles && tok < it.n_tokens) {
        const int id = __ldg(p.page_indices + it.page_off + tok / P);
        if (id >= 0 && int64_t(id) < p.num_pages)
          return reinterpret_cast<const uint4 *>(p.k_pool + (int64_t(id) * P + tok % P) * kDqkM) + 2 * cw;
        atomicOr(p.fault, PSD_FAULT_PAGE_ID);
      }
      return nullptr;
    };
    uint4 raw[2 * kKBlocks];
    auto load = [&](int i) {
      const uint4 *src = source(i);
#pragma unroll
      for (int b = 0; b < kKBlocks; ++b) {
        raw[2 * b] = src ? __ldg(src + 4 * b) : make_uint4(0u, 0u, 0u, 0u);
        raw[2 * b + 1] = src ? __ldg(src + 4 * b + 1) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    const uint32_t row_off = uint32_t(ct) * 128;
    uint32_t cpos[4];  // swizzled 16-byte chunk offsets of this thread's 4 chunks
#pragma unroll
    for (int k = 0; k < 4; ++k) cpos[k] = uint32_t((4 * cw + k) ^ (ct & 7)) << 4;
    load(grp);
    // the K ring and V buffers hold the Q head until the row warps have moved it
    ok = ok && mbar_wait(bar(BQREADY), 0, p.fault);
    // Tile i is widened block by block into the K ring (all 576 columns, for QK)
    // and V buffer i%3 (this CTA's 256 V columns, for PV).
    for (int i = grp; i < n_tiles && ok; i += 2) {
      uint8_t *vt = sm + kOffV0 + (i % kVBufs) * kVTileBytes;
#pragma unroll
      for (int b = 0; b < kKBlocks; ++b) {
        // this group's block c goes to its own slot c % kGroupSlots, so a slot's uses
        // come from one group in order and no wait runs more than a phase ahead
        const int c = (i >> 1) * kKBlocks + b, slot = grp * kGroupSlots + c % kGroupSlots;
        if (c >= kGroupSlots) {  // the QK MMAs of the slot's previous block are done
          ok = mbar_wait(bar(BKEMPTY0 + slot), uint32_t(c / kGroupSlots - 1) & 1u, p.fault);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        const int vblk = b - 4 * half;  // V block of this CTA's half, or outside [0, 4)
        if (vblk == 0 && i >= kVBufs) {  // PV(i-3) released V buffer i%3
          ok = mbar_wait(bar(BPV0 + i % kVBufs), uint32_t(i / kVBufs - 1) & 1u, p.fault);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        const uint4 h[4] = {cvt8(raw[2 * b].x, raw[2 * b].y), cvt8(raw[2 * b].z, raw[2 * b].w),
                            cvt8(raw[2 * b + 1].x, raw[2 * b + 1].y), cvt8(raw[2 * b + 1].z, raw[2 * b + 1].w)};
        uint8_t *kt = sm + kOffK + slot * kKBlockBytes + row_off;
#pragma unroll
        for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4 *>(kt + cpos[k]) = h[k];
        if (vblk >= 0 && vblk < 4) {
          uint8_t *vrow = vt + vblk * kKBlockBytes + row_off;
#pragma unroll
          for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4 *>(vrow + cpos[k]) = h[k];
        }
        fence_proxy_async();  // each thread's stores, then one arrival per warp
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BKFULL0 + slot));
      }
      load(i + 2);
    }
  } else if (warp < 4) {
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
    const bool qpos = p.q_scale >= 0.f;
    for (int i = 0; i < n_tiles && ok; ++i) {
      ok = mbar_wait(bar(BSFULL), uint32_t(i) & 1u, p.fault);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t r0[32], r1[32];
      PSD_TMEM_LD32(lane_base + kColS, r0);
      PSD_TMEM_LD32(lane_base + kColS + 32, r1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BSFREE));    // QK(i+1) may overwrite S
      const int valid = min(kTokM, it.n_tokens - i * kTokM);
      const bool partial = valid < kTokM;
      float s[64];  // raw scores q.k (scaled below)
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s[c] = __uint_as_float(r0[c]);
        s[c + 32] = __uint_as_float(r1[c]);
      }
      // max of the scaled valid scores = q_scale times the raw max (min if q_scale < 0)
      float mr = qpos ? neg_inf() : -neg_inf();
      if (!partial) {
#pragma unroll
        for (int c = 0; c < 64; ++c) mr = qpos ? fmaxf(mr, s[c]) : fminf(mr, s[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < valid) mr = qpos ? fmaxf(mr, s[c]) : fminf(mr, s[c]);
      }
      const float mt = mr * p.q_scale;
      // PV(i-1) must be done before P is rewritten or O rescaled
      if (i >= 1) {
        ok = mbar_wait(bar(BPV0 + (i - 1) % kVBufs), uint32_t((i - 1) / kVBufs) & 1u, p.fault);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      const bool grow = mt > m_ref + kLazyRescale;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? mt : m_ref;
        if (i >= 1) {  // rescale this warp's O rows in TMEM
          const float alpha = ex2(m_ref - m_new);
#pragma unroll 1
          for (int cb = 0; cb < kDvHalf / 16; ++cb) {  // 16 columns at a time: 64 scores stay live
            uint32_t o[16];
            PSD_TMEM_LD16(lane_base + kColO + cb * 16, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            PSD_TMEM_ST16(lane_base + kColO + cb * 16, o);
          }
          tmem_st_wait();
          l_sum *= alpha;
        }
        m_ref = m_new;
      }
      // P = 2^(q_scale s - m_ref) as f16 ([128 x 64], 128B-swizzled rows).  l sums P in
      // f32 before the f16 rounding the PV MMA sees: at most 2^-11 relative per term.
      uint8_t *prow = sm + kOffP + row * 128;
      const float2 qs2 = make_float2(p.q_scale, p.q_scale), nm2 = make_float2(-m_ref, -m_ref);
      float2 lacc = make_float2(0.f, 0.f);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t pk[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int t = 8 * ch + 2 * c;
          const float2 x = __ffma2_rn(make_float2(s[t], s[t + 1]), qs2, nm2);
          float a = ex2(x.x), b = ex2(x.y);
          if (partial) {
            a = t < valid ? a : 0.f;
            b = t + 1 < valid ? b : 0.f;
          }
          lacc = __fadd2_rn(lacc, make_float2(a, b));
          pk[c] = pack2_f16(a, b);
        }
        *reinterpret_cast<uint4 *>(prow + ((ch ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l_sum += lacc.x + lacc.y;
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BPFULL));
    }
    // epilogue: O / l for this row and V half
    if (ok && n_tiles > 0) {
      const int j = n_tiles - 1;
      ok = mbar_wait(bar(BPV0 + j % kVBufs), uint32_t(j / kVBufs) & 1u, p.fault);
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
  if (warp == kCtrlWarp) {
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
