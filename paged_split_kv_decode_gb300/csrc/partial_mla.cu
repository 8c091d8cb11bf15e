// K2t: split-KV partial attention for the MLA latent shape on the 5th-generation
// tensor cores, computed straight on the fp8-e4m3 latent (tcgen05.mma
// kind::f8f6f4, TMEM accumulators).
//
// Shape: 128 query heads over one 576-wide latent KV head stored as fp8-e4m3 with
// a per-tensor scale; V is the first 512 columns of the same latent rows (ROCm
// ATOM PR #1701, section 3.2: fp8 latent dequantised as value * scale; mlxcel PR
// #1004, Decomposition and Merge contract sections for the split-KV partial and
// its (V, LSE) outputs in log2 units).
//
// GB300 design.  One CTA per (work item, half of the 512 V columns), 64-token
// tiles, one tile per 64-row page block.
//   * Operands.  The latent tile is loaded by TMA as nine [64 tokens x 64 B] boxes
//     with the 64-byte swizzle and used as it lands: K-major for S = Q K^T and,
//     for this CTA's four V boxes, MN-major for O += P V.  No widening, no copy.
//   * Precision.  Q and P enter the e4m3 MMAs as two terms each, hi = e4m3(x) and
//     lo = e4m3(x - hi), which keeps 8 significant bits: a bf16 query row scaled
//     by a power of two (its largest element to [128, 256)) splits exactly down
//     to about 2^-10 of that element, and P carries a 2^-8 relative error.  The
//     two-term S costs 36 MMAs of M=128, N=64, K=32 per tile, the same count and
//     issue time as the K=16 f16 form; PV is 4 MMAs of N=256.
//   * TMEM (512 columns): O's half [128 x 256] f32, two S buffers [128 x 64] f32,
//     Q_hi[:, 0:512] as the A operand (4 e4m3 per column).  The row warps write P
//     (hi and lo, 32 columns) over the S buffer it came from and the PV MMAs read
//     A from there.  Q_hi[:, 512:576] and Q_lo stay in shared memory.
//   * Roles: row warps 0-3 (thread = head = TMEM lane) convert Q once per item and
//     run a lazily rescaled online softmax (O is rescaled in TMEM only when the
//     running max grows by more than 2^4, so P <= 2^8 fits e4m3); control warp 4
//     issues the MMAs (converged warp, one elected lane); producer warp 5 issues
//     the TMA loads of four tile buffers and zeroes the rows past the end of a
//     ragged last tile.
//   * Per tile the control warp waits twice (tile landed, P written) and commits
//     twice (S ready, tile and P consumed).
//   * When the rows feed this library's merge, consecutive items of one request in
//     a CTA's run accumulate into one partial (O, max and sum carry over), written
//     at the last of them; the rows of the others are marked empty (LSE -inf).
// The k_scale and the query row's power of two fold into the score scale, v_scale
// into the output.  The two CTAs of an item both compute S; the tile is read from
// HBM once and from L2 by the second CTA.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <vector>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

constexpr int kTokM = 64;                       // tokens per tile
constexpr int kDqkM = 576, kDvM = 512, kDvHalf = 256, kRowsM = 128;
constexpr int kBoxes = kDqkM / 64;              // 9 column boxes of 64 e4m3
constexpr int kNB = 4;                          // tile buffers
constexpr uint32_t kBoxBytes = kTokM * 64;              // 4096: [64 tokens x 64 B]
constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;     // 36864
constexpr uint32_t kQBoxBytes = kRowsM * 64;            // 8192: [128 rows x 64 e4m3]
constexpr uint32_t kQLandBytes = kRowsM * 128;          // 16384: [128 rows x 64 bf16]
constexpr uint32_t kQBytes = kBoxes * kQLandBytes;      // 147456 bf16 query rows
// Shared memory: 4 tile buffers | Q in e4m3 (Q_hi box 8, Q_lo boxes 0..8) | barriers.
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffQS = kOffK + kNB * kTileBytes;           // 147456
constexpr uint32_t kOffQHiTail = kOffQS;
constexpr uint32_t kOffQLo = kOffQS + kQBoxBytes;
constexpr uint32_t kOffBar = kOffQS + (1 + kBoxes) * kQBoxBytes;  // 229376
constexpr uint32_t kSmemMLA = kOffBar + 256 + 1024;              // barriers + alignment slack
// A query lands in bf16 (before the e4m3 split) when the tiles issued so far are
// consumed: boxes 0-4 over the Q area, boxes 5-6 and 7-8 in the tile buffers of the
// third and fourth tiles to come (g = tiles issued so far).
__host__ __device__ constexpr uint32_t q_land_at(int b, int g) {
  return b < 5 ? kOffQS + uint32_t(b) * kQLandBytes
               : b < 7 ? kOffK + uint32_t((g + 3) % kNB) * kTileBytes + uint32_t(b - 5) * kQLandBytes
                       : kOffK + uint32_t((g + 2) % kNB) * kTileBytes + uint32_t(b - 7) * kQLandBytes;
}
static_assert(5 * kQLandBytes <= (1 + kBoxes) * kQBoxBytes, "Q landing overruns the Q area");
static_assert(2 * kQLandBytes <= kTileBytes, "two landing boxes per tile buffer");
static_assert(kOffQS % 1024 == 0 && kTileBytes % 1024 == 0, "128B-swizzled landing boxes need 1024-byte alignment");
static_assert(8 * (256 + 1) <= (1 + kBoxes) * kQBoxBytes, "range scan scratch");
constexpr int kRowWarps = 4, kCtrlWarp = 4, kProdWarp = 5;
constexpr int kThreadsM = 32 * 6;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;   // S buffer b at kColS + 64 b
constexpr float kLazyRescale = 4.f;             // log2 units
constexpr float kPBias = 4.f;                   // P = 2^(score - m + 4) <= 2^8
// Run partition costs in tokens of tile work.  A least-squares fit of per-CTA
// cycles (clock64 traces, 128-request batch) gives about 2240 cycles per 64-token
// tile and about 23K per request boundary (an O write-out and a query switch,
// about 11.5K each), i.e. 330 token-equivalents each.  An item's tokens are counted
// in whole tiles.
constexpr int kItemCostTok = 330, kSplitCostTok = 330;
constexpr int kMaxPairs = 128;  // pairs whose runs the launch parameters carry

// mbarrier slots (uint64 each) at kOffBar
enum { BQ = 0, BQSEEN, BQREADY, BORDY, BDRAIN, BSFULL0, BPFULL0 = BSFULL0 + 2, BKFULL0 = BPFULL0 + 2,
       BKEMPTY0 = BKFULL0 + kNB, BSLOT = BKEMPTY0 + kNB };
static_assert(BSLOT * 8 + 20 <= 256, "barrier area");

struct MLAParams {
  const int32_t *page_indices;
  const psd_work_item *items;
  int num_items;
  float *v_out;
  float *lse_out;
  FaultRef fault;
  int64_t num_pages;
  int Hq_req, page_size;
  int merge_runs;  // rows feed the merge: accumulate consecutive items of one request
  float q_scale, v_scale;
  // Runs of the CTA pairs, computed on the host: pair x starts at tile run_tile[x]
  // of item run_item[x] and ends where pair x + 1 starts.  A run may end inside an
  // item (when the rows feed the merge and the previous item of the same request is
  // in the run): its partial then goes to the previous item's row, which the run
  // left empty.  Without them (has_runs 0) each CTA computes a run of whole items.
  int has_runs;
  int32_t run_item[kMaxPairs + 1], run_tile[kMaxPairs + 1];
  long long wait_limit;  // cycles before a wait gives up
  int withhold_from;     // testing aid: no loads for an item's tiles from this index on
};

// Item b continues item a's partial: the next chunk of the same request, whose row
// follows a's in the request's merge group.
__device__ __forceinline__ bool continues(const psd_work_item &a, const psd_work_item &b) {
  return b.q_index == a.q_index && b.out_row == a.out_row + 1 && a.n_tokens > 0 && b.n_tokens > 0;
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // 64-byte swizzle (layout code 4), descriptor version 1
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(4) << 61);
}
// kind::f8f6f4 instruction descriptor: f32 accumulate, e4m3 A and B (format 0).
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool b_mn) {
  return (1u << 4) | (uint32_t(b_mn) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// A operand in TMEM (row m in lane m, 4 e4m3 per 32-bit column in K order).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
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

// Two floats -> two e4m3 codes (round to nearest even, saturating), `lo` in byte 0.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t v;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(hi), "f"(lo));
  return v;
}
// Four floats -> hi and lo e4m3 words (element k in byte k): hi = e4m3(x),
// lo = e4m3(x - hi); the subtraction is exact in f32.
__device__ __forceinline__ void split4(float x0, float x1, float x2, float x3, uint32_t &hi, uint32_t &lo) {
  const uint32_t h01 = e4m3x2(x0, x1), h23 = e4m3x2(x2, x3);
  const float2 d01 = e4m3x2_to_float2(h01), d23 = e4m3x2_to_float2(h23);
  hi = h01 | (h23 << 16);
  lo = e4m3x2(x0 - d01.x, x1 - d01.y) | (e4m3x2(x2 - d23.x, x3 - d23.y) << 16);
}
__device__ __forceinline__ void st_global_v8(float *dst, float a, float b, float c, float d, float e, float f,
                                             float g, float h) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d),
               "f"(e), "f"(f), "f"(g), "f"(h)
               : "memory");
}
// Byte offset of 16-byte chunk c of row r in a 64-byte-swizzled box of 64-byte rows.
__device__ __forceinline__ uint32_t sw64(int r, int c) { return uint32_t(r) * 64 + (uint32_t(c ^ ((r >> 1) & 3)) << 4); }

__global__ void __launch_bounds__(kThreadsM, 1)
    partial_mla_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const MLAParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  dependents_may_launch();  // the merge that follows only waits for this grid
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + BSLOT);
  // this pair's items [begin, end), the first item from tile srange[2], the last
  // item up to tile srange[3] (0: to its end)
  int *srange = reinterpret_cast<int *>(tslot + 1);
  long long *sscan = reinterpret_cast<long long *>(sm + kOffQS);   // scratch until a query lands
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.z;                    // which 256 V columns
  const int P = p.page_size;

  if (tid == 0) {
    mbar_init(bar(BQ), 1);
    mbar_init(bar(BQSEEN), kRowWarps);
    mbar_init(bar(BQREADY), kRowWarps);
    mbar_init(bar(BORDY), kRowWarps);
    mbar_init(bar(BDRAIN), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(BSFULL0 + b), 1);
      mbar_init(bar(BPFULL0 + b), kRowWarps);
    }
    for (int b = 0; b < kNB; ++b) {
      mbar_init(bar(BKFULL0 + b), 1);
      mbar_init(bar(BKEMPTY0 + b), 1);
    }
    fence_mbar_init();
    srange[0] = srange[1] = srange[2] = srange[3] = 0;
  }
  if (warp == kCtrlWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // This CTA pair's items: the contiguous run of the (request-major) item list whose
  // first cost units fall in its 1/gridDim.x share of the total cost.  An item costs
  // its tokens plus the O write-out of one item, plus a query split where the
  // request changes (in tokens of tile work).  Items stay whole, and consecutive
  // items mostly belong to one request and reuse its split query.
  if (p.has_runs) {
    if (tid == 0) {
      const int x = blockIdx.x;
      srange[0] = p.run_item[x];
      srange[1] = p.run_item[x + 1] + (p.run_tile[x + 1] > 0 ? 1 : 0);
      srange[2] = p.run_tile[x];
      srange[3] = p.run_tile[x + 1];
    }
  } else {
    const int n = p.num_items;
    const int per = (n + kThreadsM - 1) / kThreadsM;
    const int a0 = min(n, tid * per), a1 = min(n, a0 + per);
    auto cost = [&](int i) -> long long {
      const psd_work_item it = p.items[i];
      const bool first = i == 0 || __ldg(&p.items[i - 1].q_index) != it.q_index;
      const bool writes = !p.merge_runs || i + 1 == n || !continues(it, p.items[i + 1]);
      const int tiled = (it.n_tokens + kTokM - 1) / kTokM * kTokM;
      return it.n_tokens > 0 ? tiled + (writes ? kItemCostTok : 0) + (first ? kSplitCostTok : 0) : 0;
    };
    long long part = 0;
    for (int i = a0; i < a1; ++i) part += cost(i);
    sscan[tid] = part;
    __syncthreads();
    if (tid == 0) {  // exclusive scan of the per-thread sums; the total at the end
      long long acc = 0;
      for (int t = 0; t < kThreadsM; ++t) {
        const long long v = sscan[t];
        sscan[t] = acc;
        acc += v;
      }
      sscan[kThreadsM] = acc;
    }
    __syncthreads();
    const long long total = sscan[kThreadsM];
    const long long lo_t = total * blockIdx.x / gridDim.x, hi_t = total * (blockIdx.x + 1) / gridDim.x;
    long long start = sscan[tid];
    int c_lo = 0, c_hi = 0;  // items starting before lo_t / hi_t
    for (int i = a0; i < a1; ++i) {
      c_lo += start < lo_t;
      c_hi += start < hi_t;
      start += cost(i);
    }
    if (c_lo) atomicAdd(srange, c_lo);
    if (c_hi) atomicAdd(srange + 1, c_hi);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int begin = srange[0], end = srange[1], first_tile = srange[2], end_tile = srange[3];
  // tiles [j0, j1) of item m of the run
  auto tile_lo = [&](int m) { return m == begin ? first_tile : 0; };
  auto tile_hi = [&](int m, int nt) { return m == end - 1 && end_tile > 0 ? end_tile : nt; };

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer warp
    // Loads run ahead across item boundaries.  A query switch waits until every
    // tile issued so far is consumed (the query lands over the Q area and two tile
    // buffers), and the two tiles that follow go into those buffers only once the
    // row warps have split the query.
    bool ok = true;
    int g = 0, issued = 0, nq = 0, cur_q = -1, gate = -kNB;
    bool withheld = false;
    for (int m = begin; m < end && ok && !withheld; ++m) {
      const psd_work_item it = p.items[m];
      const int nt = (it.n_tokens + kTokM - 1) / kTokM;
      if (nt <= 0) continue;  // (the planner emits no empty items)
      const int j0 = tile_lo(m), j1 = tile_hi(m, nt);
      if (j1 <= j0) continue;  // (the run planner emits no empty tile range)
      if (it.q_index != cur_q) {
        if (g > 0)
          ok = __all_sync(0xffffffffu, mbar_wait(bar(BKEMPTY0 + (g - 1) % kNB), uint32_t((g - 1) / kNB) & 1u, p.fault, p.wait_limit));
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(BQ), kQBytes);
#pragma unroll 1
          for (int b = 0; b < kBoxes; ++b)
            tma_load_3d(smem_u32(sm + q_land_at(b, g)), &tmQ, b * 64, 0, it.q_index, bar(BQ));
        }
        __syncwarp();
        cur_q = it.q_index;
        gate = g + 2;
        ++nq;
      }
#pragma unroll 1
      for (int j = j0; j < j1; ++j) {
        if (j >= p.withhold_from) {
          // testing aid: this tile and every later one go unloaded, so the control
          // warp's wait for it runs out; every tile before it was loaded.
          withheld = true;
          break;
        }
        const int buf = g % kNB;
        if (g >= kNB)  // PV(g - 4) has read the buffer
          ok = mbar_wait(bar(BKEMPTY0 + buf), uint32_t(g / kNB - 1) & 1u, p.fault, p.wait_limit);
        if (ok && g >= gate && g < gate + 2)  // a query landing box sits in this buffer
          ok = mbar_wait(bar(BQREADY), uint32_t(nq - 1) & 1u, p.fault, p.wait_limit);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const int tok = j * kTokM;
        if (lane == 0) {
          int page = __ldg(p.page_indices + it.page_off + tok / P);
          if (page < 0 || int64_t(page) >= p.num_pages) {  // out of range: load the zero fill
            raise_fault(p.fault, PSD_FAULT_PAGE_ID);
            page = -1;
          }
          mbar_arrive_expect_tx(bar(BKFULL0 + buf), kTileBytes);
          const uint32_t dst = smem_u32(sm + kOffK + buf * kTileBytes);
#pragma unroll 1
          for (int b = 0; b < kBoxes; ++b)
            tma_load_3d(dst + b * kBoxBytes, &tmK, b * 64, tok % P, page, bar(BKFULL0 + buf));
        }
        __syncwarp();
        issued = ++g;
      }
    }
    // No copy of this CTA may still be in flight when it exits.
    if (nq > 0) mbar_wait(bar(BQ), uint32_t(nq - 1) & 1u, p.fault, p.wait_limit);
    for (int t = max(0, issued - kNB); t < issued; ++t)   // the last tile of each buffer
      mbar_wait(bar(BKFULL0 + t % kNB), uint32_t(t / kNB) & 1u, p.fault, p.wait_limit);
  } else if (warp == kCtrlWarp) {
    // ------------------------------------------------------------- control warp
    // The whole warp waits; one elected lane issues.  (A wait on the issuing thread
    // alone stalls the MMAs it has queued far longer.)  Order: S(g) = Q K(g)^T, then
    // O += P(g-1) V(g-1); across an item boundary S of the next item is issued
    // before the last PV of the previous one, except at a query switch.
    const uint32_t id_qk = idesc_e4m3(128, kTokM, false);
    const uint32_t id_pv = idesc_e4m3(128, kDvHalf, true);
    // Base descriptors, built once; operand steps add offsets (>> 4) to the
    // start-address field, which never carries out of it (< 256 KB).
    const uint64_t kd = smem_desc(smem_u32(sm + kOffK), 16, 512);
    const uint64_t qhd = smem_desc(smem_u32(sm + kOffQHiTail), 16, 512);
    const uint64_t qld = smem_desc(smem_u32(sm + kOffQLo), 16, 512);
    // V (MN-major): 64-column atoms one box apart, 8-token groups 512 bytes apart
    const uint64_t vd = smem_desc(smem_u32(sm + kOffK + 4 * half * kBoxBytes), kBoxBytes, 512);
    bool ok = true;
    int g = 0, nq = 0, cur_q = -1, npart = 0;
    int pend = -1, pend_po = 0;  // tile whose PV is still to issue, and its partial's ordinal
    bool pend_first = false;     // ... which is the first tile of that item
    bool pend_cont = false;      // ... which adds to the previous item's O
    auto issue_pv = [&]() -> bool {
      const int t = pend, buf = t % kNB;
      bool r = __all_sync(0xffffffffu, mbar_wait(bar(BPFULL0 + (t & 1)), uint32_t(t >> 1) & 1u, p.fault, p.wait_limit));
      // The previous partial's O has been read out.  BORDY completes once per read-out
      // and the row warps read out partial k only after PV of partial k is issued,
      // so they are never two phases ahead of this wait.
      if (r && pend_first && !pend_cont && pend_po > 0)
        r = __all_sync(0xffffffffu, mbar_wait(bar(BORDY), uint32_t(pend_po - 1) & 1u, p.fault, p.wait_limit));
      if (!r) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint32_t a_p = tmem + kColS + 64 * (t & 1);   // P (hi | lo) over S buffer t % 2
        const uint64_t vb = vd + ((buf * kTileBytes) >> 4);
#pragma unroll
        for (int k = 0; k < 2; ++k) {  // tokens 32 k .. 32 k + 31
          const uint64_t vbk = vb + ((k * 32 * 64) >> 4);
          mma_ts(tmem + kColO, a_p + 8 * k, vbk, id_pv, (pend_first && !pend_cont && k == 0) ? 0u : 1u);
          mma_ts(tmem + kColO, a_p + 16 + 8 * k, vbk, id_pv, 1u);
        }
        umma_commit(bar(BKEMPTY0 + buf));
      }
      __syncwarp();
      pend = -1;
      return true;
    };
    for (int m = begin; m < end && ok; ++m) {
      const psd_work_item it = p.items[m];
      const int nt = (it.n_tokens + kTokM - 1) / kTokM;
      if (nt <= 0) continue;  // (the planner emits no empty items)
      const int j0 = tile_lo(m), j1 = tile_hi(m, nt);
      if (j1 <= j0) continue;  // (the run planner emits no empty tile range)
      const bool cont = p.merge_runs && m > begin && continues(p.items[m - 1], it);
      if (!cont) ++npart;
      if (it.q_index != cur_q) {
        // the split of the next query waits for every PV issued so far
        if (pend >= 0) ok = issue_pv();
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(BQREADY), uint32_t(nq) & 1u, p.fault, p.wait_limit));
        if (!ok) break;
        tc_fence_after();
        cur_q = it.q_index;
        ++nq;
      }
#pragma unroll 1
      for (int j = j0; j < j1; ++j) {
        const int buf = g % kNB;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(BKFULL0 + buf), uint32_t(g / kNB) & 1u, p.fault, p.wait_limit));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t d_s = tmem + kColS + 64 * (g & 1);
          const uint64_t kb = kd + ((buf * kTileBytes) >> 4);
#pragma unroll
          for (int b = 0; b < kBoxes; ++b) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t kbh = kb + ((b * kBoxBytes + h * 32) >> 4);
              if (b < kBoxes - 1)
                mma_ts(d_s, tmem + kColQ + 16 * b + 8 * h, kbh, id_qk, (b | h) != 0);
              else
                mma_ss(d_s, qhd + ((h * 32) >> 4), kbh, id_qk, 1u);
              mma_ss(d_s, qld + ((b * kQBoxBytes + h * 32) >> 4), kbh, id_qk, 1u);
            }
          }
          umma_commit(bar(BSFULL0 + (g & 1)));
        }
        __syncwarp();
        if (pend >= 0 && !(ok = issue_pv())) break;
        pend = g++;
        pend_first = j == j0;
        pend_cont = cont;
        pend_po = npart - 1;
      }
    }
    if (ok && pend >= 0) issue_pv();
    // every MMA this warp issued has completed before TMEM is released
    if (elect_one()) umma_commit(bar(BDRAIN));
    __syncwarp();
    mbar_wait(bar(BDRAIN), 0, p.fault, p.wait_limit);
  } else if (warp < kRowWarps) {
    // ------------------------------------------------------------------ row warps
    const int row = tid;                          // head = TMEM lane
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    bool ok = true;
    int g = 0, nq = 0, cur_q = -1;
    float qs = 0.f;  // score scale of this row for the current query
    float m_ref = neg_inf(), l_sum = 0.f;  // running max (log2, biased P) and sum
    for (int m = begin; m < end && ok; ++m) {
      const psd_work_item it = p.items[m];
      const int nt = (it.n_tokens + kTokM - 1) / kTokM;
      if (nt <= 0) continue;  // (the planner emits no empty items)
      const int j0 = tile_lo(m), j1 = tile_hi(m, nt);
      if (j1 <= j0) continue;  // (the run planner emits no empty tile range)
      // A continued item adds to the previous item's O, m_ref and l_sum.
      const bool cont = p.merge_runs && m > begin && continues(p.items[m - 1], it);
      if (it.q_index != cur_q) {
        // Query split.  Pass 1 moves the bf16 row from the landing boxes to TMEM
        // columns 0..287 (free between items) and takes its largest magnitude;
        // pass 2 scales the row by 2^k (largest element to [128, 256)) and writes
        // hi = e4m3(x), lo = e4m3(x - hi): Q_hi[0:512] to TMEM, the rest to shared
        // memory over the landing boxes, once every row warp has read them.
        ok = __all_sync(0xffffffffu, mbar_wait(bar(BQ), uint32_t(nq) & 1u, p.fault, p.wait_limit));
        if (!ok) break;
        float amax = 0.f;
#pragma unroll 1
        for (int b = 0; b < kBoxes; ++b) {
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(sm + q_land_at(b, g) + row * 128 + ((c ^ (row & 7)) << 4));
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[c])), fabsf(bf16_hi(w[c]))));
          PSD_TMEM_ST32(lane_base + 32 * b, w);
        }
        tmem_st_wait();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BQSEEN));
        ok = __all_sync(0xffffffffu, mbar_wait(bar(BQSEEN), uint32_t(nq) & 1u, p.fault, p.wait_limit));
        if (!ok) break;
        // power of two: amax * 2^k in [128, 256); zero and subnormal rows keep k = 0
        const int ex = int((__float_as_uint(amax) >> 23) & 0xffu) - 127;
        const int kq = ex > -127 ? max(-120, min(120, 7 - ex)) : 0;
        const float qmul = __uint_as_float(uint32_t(127 + kq) << 23);
        qs = p.q_scale * __uint_as_float(uint32_t(127 - kq) << 23);
#pragma unroll 1
        for (int b = 0; b < kBoxes; ++b) {
          uint32_t w[32], hi[16], lo[16];
          PSD_TMEM_LD32(lane_base + 32 * b, w);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c)
            split4(bf16_lo(w[2 * c]) * qmul, bf16_hi(w[2 * c]) * qmul, bf16_lo(w[2 * c + 1]) * qmul,
                   bf16_hi(w[2 * c + 1]) * qmul, hi[c], lo[c]);
          if (b < kBoxes - 1) {
            PSD_TMEM_ST16(lane_base + kColQ + 16 * b, hi);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4 *>(sm + kOffQHiTail + sw64(row, c)) =
                  make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4 *>(sm + kOffQLo + b * kQBoxBytes + sw64(row, c)) =
                make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
        }
        tmem_st_wait();
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BQREADY));
        cur_q = it.q_index;
        ++nq;
      }

      if (!cont) {
        m_ref = neg_inf();
        l_sum = 0.f;
      }
      const bool qpos = qs >= 0.f;
      const int tail = it.n_tokens - (nt - 1) * kTokM;   // valid tokens of the last tile
#pragma unroll 1
      for (int j = j0; j < j1; ++j, ++g) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(BSFULL0 + (g & 1)), uint32_t(g >> 1) & 1u, p.fault, p.wait_limit));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_col = lane_base + kColS + 64 * (g & 1);
        uint32_t r0[32], r1[32];
        PSD_TMEM_LD32(s_col, r0);
        PSD_TMEM_LD32(s_col + 32, r1);
        tmem_ld_wait();
        const int valid = j == nt - 1 ? tail : kTokM;
        const bool partial = valid < kTokM;
        float s[64];  // raw scores (q 2^k) . k_codes
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(r0[c]);
          s[c + 32] = __uint_as_float(r1[c]);
        }
        // max of the scaled valid scores = qs times the raw max (min if qs < 0)
        float mr = qpos ? neg_inf() : -neg_inf();
        if (!partial) {
#pragma unroll
          for (int c = 0; c < 64; ++c) mr = qpos ? fmaxf(mr, s[c]) : fminf(mr, s[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < valid) mr = qpos ? fmaxf(mr, s[c]) : fminf(mr, s[c]);
        }
        const float mt = mr * qs;
        const bool grow = mt > m_ref + kLazyRescale;
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? mt : m_ref;
          if (j > j0 || cont) {  // PV(g-1) must be done; then rescale this warp's O rows in TMEM
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(BKEMPTY0 + (g - 1) % kNB), uint32_t((g - 1) / kNB) & 1u, p.fault, p.wait_limit));
            if (!ok) break;
            tc_fence_after();
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
            l_sum *= alpha;
          }
          m_ref = m_new;
        }
        // P = 2^(qs s - m_ref + 4) <= 2^8, split into e4m3 hi and lo words (4 tokens
        // each) and written over the first 32 columns of this S buffer.  l sums the
        // unsplit P in f32.
        const float2 qs2 = make_float2(qs, qs), nb2 = make_float2(kPBias - m_ref, kPBias - m_ref);
        float2 lacc = make_float2(0.f, 0.f);
        uint32_t pw[32];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int t = 4 * c;
          const float2 x01 = __ffma2_rn(make_float2(s[t], s[t + 1]), qs2, nb2);
          const float2 x23 = __ffma2_rn(make_float2(s[t + 2], s[t + 3]), qs2, nb2);
          float a0 = ex2(x01.x), a1 = ex2(x01.y), a2 = ex2(x23.x), a3 = ex2(x23.y);
          if (partial) {
            a0 = t < valid ? a0 : 0.f;
            a1 = t + 1 < valid ? a1 : 0.f;
            a2 = t + 2 < valid ? a2 : 0.f;
            a3 = t + 3 < valid ? a3 : 0.f;
          }
          lacc = __fadd2_rn(lacc, __fadd2_rn(make_float2(a0, a1), make_float2(a2, a3)));
          split4(a0, a1, a2, a3, pw[c], pw[16 + c]);
        }
        l_sum += lacc.x + lacc.y;
        PSD_TMEM_ST32(s_col, pw);
        if (partial) {
          // Rows past the item's last token (still inside its page) may hold anything:
          // zero them in this CTA's four V boxes, so that P = 0 never meets a NaN.
          // S of this tile is complete, so its MMAs no longer read the buffer.
          uint8_t *vt = sm + kOffK + (g % kNB) * kTileBytes + 4 * half * kBoxBytes;
          const int n16 = (kTokM - valid) * 4;   // 16-byte chunks per box
#pragma unroll 1
          for (int c = row; c < 4 * n16; c += 32 * kRowWarps)
            *reinterpret_cast<uint4 *>(vt + (c / n16) * kBoxBytes + valid * 64 + (c % n16) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async();
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BPFULL0 + (g & 1)));
      }
      if (!ok) break;
      if (p.merge_runs && m + 1 < end && continues(it, p.items[m + 1])) {
        // The next item continues this partial: this item's row is empty (LSE -inf,
        // v not written; the merge does not read it), and O is not read out.
        if (half == 0) p.lse_out[int64_t(it.out_row) * p.Hq_req + row] = neg_inf();
        continue;
      }
      // epilogue: O / l for this row and V half, once the item's last PV is done
      ok = __all_sync(0xffffffffu, mbar_wait(bar(BKEMPTY0 + (g - 1) % kNB), uint32_t((g - 1) / kNB) & 1u, p.fault, p.wait_limit));
      if (!ok) break;
      tc_fence_after();
      // a run that ends inside this item writes to the previous item's (empty) row
      const int out_row = m == end - 1 && end_tile > 0 ? it.out_row - 1 : it.out_row;
      const int64_t orow = int64_t(out_row) * p.Hq_req + row;
      float *dst = p.v_out + orow * kDvM + half * kDvHalf;
      const float inv = p.v_scale / l_sum;
#pragma unroll 1
      for (int cb = 0; cb < kDvHalf / 32; ++cb) {
        uint32_t o[32];
        PSD_TMEM_LD32(lane_base + kColO + cb * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; c += 8)
          st_global_v8(dst + cb * 32 + c, __uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                       __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv,
                       __uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv,
                       __uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
      }
      if (half == 0) p.lse_out[orow] = m_ref - kPBias + log2f(l_sum);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BORDY));   // PV of the next partial may overwrite O
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

// Latent pool [num_pages][page_size][576] e4m3 as a 3-D map; a box is 64 columns of
// 64 consecutive token rows of one page, landing with the 64-byte swizzle.
bool encode_latent_map(CUtensorMap *map, const DeviceInfo &dev, const void *pool, int64_t num_pages,
                       int page_size) {
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(dev.encode_tiled);
  if (!encode) return false;
  cuuint64_t dims[3] = {cuuint64_t(kDqkM), cuuint64_t(page_size), cuuint64_t(num_pages)};
  cuuint64_t strides[2] = {cuuint64_t(kDqkM), cuuint64_t(page_size) * kDqkM};
  cuuint32_t box[3] = {64, cuuint32_t(kTokM), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(pool), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The pairs' runs: contiguous stretches of the item list that minimise the largest
// run cost (binary search on the bound, greedy fill), in the cost units of the
// in-kernel partition, plus an O write-out for a run that ends inside a request and
// a query split for one that starts inside it.  When the rows feed the merge, a run
// may end inside item i at a tile boundary if item i - 1 belongs to the same request
// and to the run (the run's partial then goes to row i - 1); otherwise runs hold
// whole items.  The optimum lies in [max(mean, largest item), mean + largest item].
void plan_runs(const PartialLaunch &L, int pairs, MLAParams &p) {
  const int n = L.num_items;
  const psd_work_item *it = L.items_host;
  std::vector<int64_t> c(static_cast<size_t>(n));
  std::vector<int32_t> ntl(static_cast<size_t>(n));
  std::vector<char> first(static_cast<size_t>(n)), writes(static_cast<size_t>(n)), split_ok(static_cast<size_t>(n));
  int64_t total = 0, cmax = 0;
  for (int i = 0; i < n; ++i) {
    const size_t k = size_t(i);
    ntl[k] = it[i].n_tokens > 0 ? (it[i].n_tokens + kTokM - 1) / kTokM : 0;
    first[k] = i == 0 || it[i - 1].q_index != it[i].q_index;
    const bool cont_next = i + 1 < n && it[i + 1].q_index == it[i].q_index &&
                           it[i + 1].out_row == it[i].out_row + 1 && it[i].n_tokens > 0 && it[i + 1].n_tokens > 0;
    writes[k] = !L.merge_runs || !cont_next;
    split_ok[k] = L.merge_runs && i > 0 && ntl[k] >= 2 && it[i - 1].n_tokens > 0 &&
                  it[i - 1].q_index == it[i].q_index && it[i].out_row == it[i - 1].out_row + 1;
    c[k] = ntl[k] > 0 ? int64_t(ntl[k]) * kTokM + (writes[k] ? kItemCostTok : 0) + (first[k] ? kSplitCostTok : 0) : 0;
    total += c[k];
    cmax = std::max(cmax, c[k]);
  }
  // Greedy fill under bound B; returns the number of runs (pairs + 1 when B is too
  // small) and, when `rec`, the run starts.
  auto fill = [&](int64_t B, bool rec) {
    int runs = 1, start = 0;
    int64_t acc = 0;
    if (rec) {
      p.run_item[0] = 0;
      p.run_tile[0] = 0;
    }
    for (int i = 0; i < n; ++i) {
      const size_t k = size_t(i);
      if (acc + c[k] <= B || i == start) {
        acc += c[k];
        continue;
      }
      int tiles = 0;  // tiles of item i that stay in this run
      if (split_ok[k] && i - 1 >= start) {
        const int64_t room = B - acc - kItemCostTok - (first[k] ? kSplitCostTok : 0);
        tiles = room >= kTokM ? int(std::min<int64_t>(room / kTokM, ntl[k] - 1)) : 0;
      }
      if (runs == pairs) return pairs + 1;
      if (rec) {
        p.run_item[runs] = i;
        p.run_tile[runs] = tiles;
      }
      ++runs;
      start = i;
      acc = tiles > 0 ? int64_t(ntl[k] - tiles) * kTokM + (writes[k] ? kItemCostTok : 0) + kSplitCostTok
                      : c[k] + (first[k] ? 0 : kSplitCostTok);
    }
    if (rec)
      for (int x = runs; x <= pairs; ++x) {
        p.run_item[x] = n;
        p.run_tile[x] = 0;
      }
    return runs;
  };
  const int64_t mean = (total + pairs - 1) / pairs;
  int64_t lo = std::max(mean, cmax), hi = mean + cmax + kItemCostTok + kSplitCostTok;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (fill(mid, false) <= pairs) hi = mid;
    else lo = mid + 1;
  }
  fill(lo, true);
  p.has_runs = 1;
}

}  // namespace

bool partial_mla_supports(const PartialLaunch &L) {
  return L.latent_v && L.kv_dtype == PSD_FP8_E4M3 && L.Dqk == kDqkM && L.Dv == kDvM &&
         L.G_cta == kRowsM && L.Hq_req == kRowsM && L.Hkv == 1 && L.page_size % kTokM == 0 &&
         reinterpret_cast<uintptr_t>(L.k_pool) % 16 == 0 && reinterpret_cast<uintptr_t>(L.q) % 16 == 0;
}

psd_status launch_partial_mla(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  if (L.num_items == 0) return PSD_OK;
  if (size_t(dev.smem_optin) < kSmemMLA)
    return fail(PSD_ERR_UNSUPPORTED, "MLA tcgen05 partial needs %u bytes of shared memory", kSmemMLA);
  // The query rows arrive by TMA, which this kernel points at device memory only.
  cudaPointerAttributes qa;
  if (cudaPointerGetAttributes(&qa, L.q) != cudaSuccess || (qa.type != cudaMemoryTypeDevice &&
                                                           qa.type != cudaMemoryTypeManaged)) {
    (void)cudaGetLastError();
    return fail(PSD_ERR_UNSUPPORTED, "the MLA tcgen05 partial takes q in device memory only");
  }
  CUtensorMap tmQ, tmK;
  if (!encode_q_map(&tmQ, dev, L.q, L.q_batch, L.Hq_req))
    return fail(PSD_ERR_CUDA, "cuTensorMapEncodeTiled failed for q");
  if (!encode_latent_map(&tmK, dev, L.k_pool, L.num_pages, L.page_size))
    return fail(PSD_ERR_CUDA, "cuTensorMapEncodeTiled failed for the latent pool");
  MLAParams p;
  p.page_indices = L.page_indices;
  p.items = L.items;
  p.num_items = L.num_items;
  p.v_out = L.v_out;
  p.lse_out = L.lse_out;
  p.fault = L.fault;
  p.num_pages = L.num_pages;
  p.Hq_req = L.Hq_req;
  p.page_size = L.page_size;
  p.merge_runs = L.merge_runs ? 1 : 0;
  p.q_scale = L.q_scale;
  p.v_scale = L.v_scale;
  p.wait_limit = dev.test_wait_limit > 0 ? dev.test_wait_limit : kWaitLimitCycles;
  p.withhold_from = dev.test_withhold_from >= 0 ? dev.test_withhold_from : 0x7fffffff;
  cudaError_t e = cudaFuncSetAttribute(partial_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kSmemMLA));
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  // persistent: one CTA pair per two SMs, each pair a token-balanced run of items
  const int pairs = std::max(1, std::min(L.num_items, dev.num_sms / 2));
  p.has_runs = 0;
  if (L.items_host && pairs <= kMaxPairs) plan_runs(L, pairs, p);
  const dim3 grid(static_cast<unsigned>(pairs), 1, 2);
  partial_mla_kernel<<<grid, kThreadsM, kSmemMLA, s>>>(tmQ, tmK, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "partial (MLA tcgen05) launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

}  // namespace psd
