// K2t: the stacked level-0 rows of the cascade on the 5th-generation tensor cores
// (tcgen05.mma kind::f16: bf16 operands, f32 accumulators in TMEM).
//
// Work unit (mlxcel PR #1004, Decomposition section): a task is one (level-0 chunk,
// KV head, block of up to 128 stacked rows).  The stacked rows of a KV head are the
// M members' G query heads, h0 = kv*(M*G) + m*G + g, so every K/V element of the
// shared span crosses from HBM (and L2) into shared memory once for all of them:
// with 64 stacked rows the 16-row-group form moved each tile four times.  Outputs
// are the per-chunk partials of the Merge contract section: rows normalised by
// their own denominator, LSE = m + log2 l in log2 units.
//
// GB300 design.
//   * Persistent: one CTA per SM takes a contiguous range of tasks ordered (KV head,
//     row block, chunk); the loads run ahead across task boundaries, so a task pays no
//     pipeline ramp.  When the rows feed the merge, a CTA's consecutive chunks of one
//     KV head and row block form a run: O, max and sum carry over, one partial per run
//     is written and the run's other chunk rows are marked empty, so the merge reads a
//     few live rows per member instead of one per chunk (128 with a 65536-token
//     prefix, where the merge took 26 us).
//   * Tiles of 64 tokens, loaded by TMA in [16 tokens x 64 columns] boxes with the
//     128-byte swizzle (one box per page segment and 64 columns) into a ring of 5
//     stages of 32 KB (D = 128).  Two producer warps take alternate tiles, one copy
//     per lane.  Page positions past the item's last page load with the page
//     coordinate -1, which the TMA fills with zeros.
//   * S = Q K^T: M = 128 rows (rows past the stacked count are zero), N = 64 tokens,
//     D/16 MMAs with K = 16; Q from a shared-memory tile (two, one per task parity),
//     K straight from the ring (both K-major).  S has three TMEM buffers, so S of
//     tile g + 1 runs on the tensor cores while the row warps take the softmax of
//     tile g.
//   * O += P V: P as two bf16 terms, hi = bf16(P) and lo = bf16(P - hi), written by
//     the row warps over the S buffer they came from (TMEM A operand); V straight
//     from the ring, read MN-major.  8 MMAs of N = D per tile.  The two terms keep
//     about 16 bits of P; a single bf16 P would cost up to 2^-9 |v|.
//   * TMEM (512 columns at D = 128): two O buffers [128 x D] f32 (a run's O is read
//     out while the next run accumulates) and three S buffers [128 x 64].
//   * Roles: row warps 0-3 (thread = stacked row = TMEM lane) run a lazily rescaled
//     online softmax (O is rescaled in TMEM only when a row's running max grows by
//     more than 2^8, so P <= 2^8) and zero the V rows past the last token of a
//     ragged tile; control warp 4 issues the MMAs (converged warp, one elected
//     lane); producer warps 5-6 issue the TMA loads; epilogue warps 7-10 gather the
//     members' query rows two runs ahead and read out each finished run's O / l
//     and LSE.  Clock traces put the row warps on the critical path: a task boundary
//     cost them about 9000 cycles (read-out, query gather) before the epilogue warps
//     took that work.
//   * Per tile the control warp waits twice (tile landed, P written) and commits
//     twice (S ready; tile and P consumed), issuing S(g + 2) before PV(g).
// Every mbarrier wait is bounded; a CTA never exits with a copy in flight and
// always releases its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

constexpr int kTok0 = 64;                   // tokens per tile
constexpr int kSub0 = 16;                   // tokens per TMA box (one page segment)
constexpr int kRows0 = 128;                 // stacked rows per task (TMEM lanes)
// Warp roles: 0-3 row warps, 4 control, 5-6 producers, 7-10 epilogue.  Two producer
// warps take alternate tiles: one thread issuing an SM's tensor copies streamed the
// pool at 3.6-4.2 TB/s, two or more streams per SM at 4.5-4.9 TB/s (loads-only probe,
// 268 MB, one CTA per SM).
constexpr int kRowWarps0 = 4, kCtrlWarp0 = 4, kProdWarp0 = 5, kProducers0 = 2, kEpiWarp0 = 7, kEpiWarps0 = 4;
constexpr int kThreads0 = 32 * (kEpiWarp0 + kEpiWarps0);
constexpr uint32_t kRingBytes0 = 160 * 1024;  // one CTA per SM: the ring, then two Q tiles
constexpr int kMaxStages0 = 10;
constexpr float kLazy0 = 8.f;               // log2 units
// S buffers in TMEM: S(g + 1) may be issued before PV(g - 1), which still reads P(g - 1)
// from its buffer, so the tensor cores compute the next scores while the row warps
// take the softmax of this tile.  (With two buffers S(g + 1) waited for PV(g - 1),
// which put a PV and an S in series between two softmaxes: about 700 cycles a tile.)
constexpr int kSBufs0 = 3;

template <int D>
struct L0Layout {
  static constexpr int kBoxes = D / 64;                         // 64-column boxes per row
  static constexpr uint32_t kBoxBytes = kTok0 * 128;            // one box column of a tile: 8 KB
  static constexpr uint32_t kHalfBytes = kBoxes * kBoxBytes;    // K (or V) of a tile
  static constexpr uint32_t kStageBytes = 2 * kHalfBytes;
  static constexpr int kStages = int(kRingBytes0 / kStageBytes);  // 5 at D = 128, 10 at D = 64
  static constexpr uint32_t kQBoxBytes = kRows0 * 128;          // 16 KB: 64 columns of 128 rows
  static constexpr uint32_t kQBytes = kBoxes * kQBoxBytes;      // one task's query rows
  static constexpr uint32_t kOffQ = kStages * kStageBytes;      // two Q tiles (tasks k % 2)
  static constexpr uint32_t kOffBar = kOffQ + 2 * kQBytes;
  static constexpr uint32_t kSmem = kOffBar + 512 + 1024;       // barriers, TMEM slot, alignment slack
  // TMEM columns: two O buffers [128 x D] f32, three S buffers [128 x 64], and per task
  // parity a row's l and m (row warps to epilogue warps)
  static constexpr uint32_t kColO = 0, kColS = 2 * D, kColLM = kColS + kSBufs0 * kTok0;
  static constexpr uint32_t kTmemCols = kColLM + 4 <= 256 ? 256 : 512;
  static_assert(kStages <= kMaxStages0, "barrier slots");
  // The control warp issues S(g + 2) before PV(g), and only PV(g) frees the stage of
  // tile g: with fewer than three stages tile g + 2 has no stage to land in.
  static_assert(kStages >= 3, "S runs two tiles ahead of PV");
  static_assert(kSmem <= 227u * 1024u, "shared memory");
  static_assert(kStageBytes % 1024 == 0 && kOffQ % 1024 == 0 && kQBytes % 1024 == 0,
                "128B-swizzled tiles need 1024-byte alignment");
};

// mbarrier slots (uint64 each) at kOffBar; the TMEM slot after them.
enum {
  B0_KFULL = 0, B0_KEMPTY = kMaxStages0,  // per stage: tile landed / tile and P consumed (PV done)
  B0_SFULL = 2 * kMaxStages0,             // [3] S of tile g in S buffer g % 3 is complete
  B0_PFULL = B0_SFULL + kSBufs0,          // [3] P of tile g written (row warps)
  B0_QFULL = B0_PFULL + kSBufs0,          // [2] Q tile k % 2 written (epilogue warps)
  B0_QFREE = B0_QFULL + 2,                // [2] every S MMA of task k has read Q tile k % 2
  B0_OFULL = B0_QFREE + 2,                // [2] every PV of task k is complete (O buffer k % 2)
  B0_LREADY = B0_OFULL + 2,               // [2] l and m of task k's rows in TMEM (row warps)
  B0_OFREE = B0_LREADY + 2,               // [2] task k's O, l, m read out (epilogue warps)
  B0_DRAIN = B0_OFREE + 2,
  B0_SLOT
};
static_assert(B0_SLOT * 8 + 4 <= 512, "barrier area");

struct L0Params {
  const __nv_bfloat16 *q;
  const int32_t *page_indices;
  const psd_work_item *items;
  const int32_t *members;
  const int32_t *member_row_base;
  uint32_t inl_items, inl_members, inl_row_base;  // offsets in the inline lists
  float *v_out;
  float *lse_out;
  FaultRef fault;
  int64_t num_pages;
  int num_tasks;      // items x Hkv x row blocks
  int n_items, Hkv, n_rb;  // level-0 items, KV heads, row blocks per (item, KV head)
  int runs;           // the rows feed this library's merge: accumulate runs of chunks
  int Hq_req, page_size, Gm, G_rows;
  float q_scale, v_scale;  // q_scale > 0
  long long wait_limit;
  int withhold_from;  // testing aid: no loads for an item's tiles from this index on
};

// Shared-memory matrix descriptor, 128-byte swizzle (layout code 2), version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
// kind::f16 instruction descriptor: f32 accumulate, bf16 A and B, A K-major, B
// K-major or (b_mn) MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(b_mn) << 16) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// A operand in TMEM: row m in lane m, two bf16 per 32-bit column in K order.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void commit_to(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ bool elect_lane() {
  uint32_t e;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
  return e != 0;
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 32 consecutive columns of this warp's 32 lanes (one 32-bit value per lane each).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t (&r)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
}
__device__ __forceinline__ void tmem_st2(uint32_t taddr, const uint32_t (&r)[2]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(r[0]), "r"(r[1]) : "memory");
}
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void st_v8(float *dst, const float (&v)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "f"(v[0]), "f"(v[1]), "f"(v[2]),
               "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}


// CAP > 0: the items, members and row bases come in the launch's parameters.
template <int D, int CAP>
__global__ void __launch_bounds__(kThreads0, 1)
    partial_l0_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const L0Params p, const __grid_constant__ ListParam<CAP> lists) {
  using Lay = L0Layout<D>;
  constexpr int NS = Lay::kStages;
  constexpr bool INL = CAP != 0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  dependents_may_launch();  // whatever follows waits for this grid on its own
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *ring = sm;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::kOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + B0_SLOT);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const psd_work_item *items = p.items;
  const int32_t *members = p.members, *row_base = p.member_row_base;
  if constexpr (INL) {
    items = reinterpret_cast<const psd_work_item *>(lists.bytes + p.inl_items);
    members = reinterpret_cast<const int32_t *>(lists.bytes + p.inl_members);
    row_base = reinterpret_cast<const int32_t *>(lists.bytes + p.inl_row_base);
  }
  auto ld_list = [](const int32_t *a) -> int32_t {
    if constexpr (INL) return *a;
    else return __ldg(a);
  };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.page_size;
  // Tasks are numbered t = (kv * n_rb + rb) * n_items + item: the chunks of one KV
  // head and row block are consecutive.  This CTA takes the contiguous range
  // [tb, te), k = t - tb.  At one time the CTAs read the same chunk positions of the
  // different KV heads, so the pages' rows are read together.
  const int tb = int(int64_t(blockIdx.x) * p.num_tasks / gridDim.x);
  const int te = int(int64_t(blockIdx.x + 1) * p.num_tasks / gridDim.x);
  const int n_mine = te - tb;
  // Runs: maximal ranges of this CTA's tasks with the same KV head and row block (the
  // same query rows).  When the partial rows feed the merge, a run's chunks accumulate
  // into one partial (O, running max and sum carry over), written to the row of the
  // run's last chunk; the rows of its other chunks are empty (LSE -inf), which the
  // merge reads as no tokens.  Otherwise every task is a run of its own.
  const int kvrb0 = p.n_items > 0 ? tb / p.n_items : 0;
  auto new_run = [&](int k) { return k == 0 || !p.runs || (tb + k) % p.n_items == 0; };
  auto run_of = [&](int k) { return p.runs ? (tb + k) / p.n_items - kvrb0 : k; };
  auto last_of_run = [&](int k) { return k == n_mine - 1 || new_run(k + 1); };
  auto run_first = [&](int r) { return p.runs ? max(0, (kvrb0 + r) * p.n_items - tb) : r; };
  auto run_end = [&](int r) { return p.runs ? min(n_mine, (kvrb0 + r + 1) * p.n_items - tb) : r + 1; };
  const int n_runs = n_mine > 0 ? run_of(n_mine - 1) + 1 : 0;
  struct Task {
    psd_work_item it;
    int kv, row0, rows, n_tiles;
  };
  auto task = [&](int k) {
    const int t = tb + k;
    Task x;
    const int kvrb = t / p.n_items;
    x.it = items[t - kvrb * p.n_items];
    x.kv = kvrb / p.n_rb;
    x.row0 = (kvrb - x.kv * p.n_rb) * kRows0;
    x.rows = min(kRows0, p.G_rows - x.row0);
    x.n_tiles = (x.it.n_tokens + kTok0 - 1) / kTok0;
    return x;
  };
  // The stacked row g of a task (member g / G, head kv*G + g % G): its request and head.
  auto row_source = [&](const Task &x, int g_row, int &qb, int &head) {
    const int m = g_row / p.Gm;
    qb = x.it.q_index >= 0 ? x.it.q_index : ld_list(members + m);
    head = x.kv * p.Gm + (g_row - m * p.Gm);
    return m;
  };

  if (tid == 0) {
    for (int b = 0; b < NS; ++b) {
      mbar_init(bar(B0_KFULL + b), 1);
      mbar_init(bar(B0_KEMPTY + b), 1);
    }
    for (int b = 0; b < kSBufs0; ++b) {
      mbar_init(bar(B0_SFULL + b), 1);
      mbar_init(bar(B0_PFULL + b), kRowWarps0);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B0_QFULL + b), kEpiWarps0);
      mbar_init(bar(B0_QFREE + b), 1);
      mbar_init(bar(B0_OFULL + b), 1);
      mbar_init(bar(B0_LREADY + b), kRowWarps0);
      mbar_init(bar(B0_OFREE + b), kEpiWarps0);
    }
    mbar_init(bar(B0_DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == kCtrlWarp0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(Lay::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;

  if (warp >= kProdWarp0 && warp < kProdWarp0 + kProducers0) {
    // ----------------------------------------------------------- producer warps
    // Producer pw loads the tiles g with g % kProducers0 == pw, into the stages g % NS
    // (a stage may pass from one producer to the other; the wait for the PV that read
  // it orders the two).
    const int pw = warp - kProdWarp0;
    const uint64_t pol = l2_evict_first_policy();
    bool ok = true;
    int g = 0;  // tiles of this CTA so far (all tasks, both producers)
    bool withheld = false;
    for (int k = 0; k < n_mine && ok && !withheld; ++k) {
      const Task x = task(k);
      const int n_item_pages = (x.it.n_tokens + P - 1) / P;
      // The item's page ids, 32 positions per window, one per lane (a dependent load
      // per box would put an L2 round trip in front of every copy).
      int win = 0;
      int pid = lane < n_item_pages ? __ldg(p.page_indices + x.it.page_off + lane) : -1;
      for (int j = 0; j < x.n_tiles; ++j, ++g) {
        if (j >= p.withhold_from) {
          // testing aid: neither producer loads this tile or any later one (both walk
          // every tile, so both stop here), so the control warp's wait for it runs out;
          // every tile before it was loaded, after waits for PVs that were issued.
          withheld = true;
          break;
        }
        if (g % kProducers0 != pw) continue;
        const int buf = g % NS;
        if (g >= NS)  // PV(g - NS) has read the stage
          ok = __all_sync(0xffffffffu, mbar_wait(bar(B0_KEMPTY + buf), uint32_t(g / NS - 1) & 1u, p.fault,
                                                 p.wait_limit));
        if (!ok) break;
        int ids[kTok0 / kSub0];
#pragma unroll
        for (int i = 0; i < kTok0 / kSub0; ++i) {  // warp-uniform positions
          const int pos = (j * kTok0 + i * kSub0) / P;
          if (pos - win >= 32) {
            win = pos;
            pid = win + lane < n_item_pages ? __ldg(p.page_indices + x.it.page_off + win + lane) : -1;
          }
          ids[i] = pos < n_item_pages ? __shfl_sync(0xffffffffu, pid, pos - win) : -1;
        }
        // One copy per lane: a single thread issues a tensor copy about every 180
        // cycles (clock traces), far too slowly to keep the ring full.
        if (lane == 0) mbar_arrive_expect_tx(bar(B0_KFULL + buf), Lay::kStageBytes);
        __syncwarp();
        constexpr int kCopies = (kTok0 / kSub0) * Lay::kBoxes * 2;   // 16 at D = 128
        static_assert(kCopies <= 32, "one copy per lane");
        if (lane < kCopies) {
          const int i = lane / (2 * Lay::kBoxes), c = (lane >> 1) % Lay::kBoxes, v = lane & 1;
          const int tok = j * kTok0 + i * kSub0;
          const int pos = tok / P;
          int id = ids[0];
#pragma unroll
          for (int q = 1; q < kTok0 / kSub0; ++q) id = i == q ? ids[q] : id;
          if (pos < n_item_pages && (id < 0 || int64_t(id) >= p.num_pages)) {
            raise_fault(p.fault, PSD_FAULT_PAGE_ID);
            id = -1;  // past the item's pages, or out of range: the zero fill
          }
          const uint32_t off = (v ? Lay::kHalfBytes : 0u) + c * Lay::kBoxBytes + i * (kSub0 * 128);
          tma_load_4d(smem_u32(ring + buf * Lay::kStageBytes + off), v ? &tmV : &tmK, c * 64, x.kv, tok - pos * P,
                      id, bar(B0_KFULL + buf), pol);
        }
        __syncwarp();
      }
    }
    // No copy of this CTA may still be in flight when it exits (each producer waits
    // for its own).  After a failed wait g counts only the tiles this warp reached.
    for (int t = g > NS ? g - NS : 0; t < g; ++t)
      if (t % kProducers0 == pw) mbar_wait(bar(B0_KFULL + t % NS), uint32_t(t / NS) & 1u, p.fault, p.wait_limit);
  } else if (warp == kCtrlWarp0) {
    // ------------------------------------------------------------- control warp
    const uint32_t id_s = idesc_bf16(kRows0, kTok0, false);
    const uint32_t id_pv = idesc_bf16(kRows0, D, true);
    // Q and K: K-major, 8-row groups 1024 bytes apart.  V: MN-major, 64-column atoms
    // one box column (8 KB) apart, 8-token groups 1024 bytes apart.  Operand steps add
    // offsets (>> 4) to the start-address field, which never carries out of it.
    const uint64_t qd = desc_sw128(smem_u32(sm + Lay::kOffQ), 16, 1024);
    const uint64_t kd = desc_sw128(smem_u32(ring), 16, 1024);
    const uint64_t vd = desc_sw128(smem_u32(ring + Lay::kHalfBytes), Lay::kBoxBytes, 1024);
    bool ok = true;
    // PVs still to issue, oldest first: PV(g) is issued after S(g + 2)
    struct Pend {
      int t, k;             // tile, run
      bool first, last;     // the run's first / last tile
    };
    Pend q0{0, 0, false, false}, q1{0, 0, false, false};   // the queue's two slots
    int pn = 0;
    auto issue_pv = [&]() -> bool {
      const Pend e = q0;
      const int t = e.t, buf = t % NS;
      bool r = __all_sync(0xffffffffu, mbar_wait(bar(B0_PFULL + t % kSBufs0), uint32_t(t / kSBufs0) & 1u, p.fault,
                                                 p.wait_limit));
      // the first PV of run k overwrites O buffer k % 2: run k - 2 must have been read out
      if (r && e.first && e.k >= 2)
        r = __all_sync(0xffffffffu, mbar_wait(bar(B0_OFREE + (e.k & 1)), uint32_t((e.k - 2) >> 1) & 1u,
                                              p.fault, p.wait_limit));
      if (!r) return false;
      fence_after();
      if (elect_lane()) {
        const uint32_t a_p = tmem + Lay::kColS + kTok0 * (t % kSBufs0);   // P hi | P lo over S buffer t % 3
        const uint32_t d_o = tmem + Lay::kColO + D * (e.k & 1);
        const uint64_t vb = vd + ((buf * Lay::kStageBytes) >> 4);
#pragma unroll
        for (int k = 0; k < kTok0 / 16; ++k) {  // tokens 16 k .. 16 k + 15: two 8-token groups
          const uint64_t vbk = vb + ((k * 2 * 1024) >> 4);
          mma_f16_ts(d_o, a_p + 8 * k, vbk, id_pv, (e.first && k == 0) ? 0u : 1u);
          mma_f16_ts(d_o, a_p + 32 + 8 * k, vbk, id_pv, 1u);
        }
        commit_to(bar(B0_KEMPTY + buf));
        if (e.last) commit_to(bar(B0_OFULL + (e.k & 1)));
      }
      __syncwarp();
      q0 = q1;
      --pn;
      return true;
    };
    int g = 0;
    uint64_t qk = qd;
    for (int k = 0; k < n_mine && ok; ++k) {
      const Task x = task(k);
      const int run = run_of(k);
      const bool run_ends = last_of_run(k);
      if (new_run(k)) {
        // Run r's query rows arrive after run r - 2 is read out, which needs its last
        // PV: issue every pending PV of run r - 2 or earlier first.
        while (ok && pn > 0 && q0.k <= run - 2) ok = issue_pv();
        if (!ok) break;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B0_QFULL + (run & 1)), uint32_t(run >> 1) & 1u, p.fault,
                                               p.wait_limit));
        if (!ok) break;
        fence_after();
        qk = qd + (((run & 1) * Lay::kQBytes) >> 4);
      }
      for (int j = 0; j < x.n_tiles; ++j, ++g) {
        const int buf = g % NS;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B0_KFULL + buf), uint32_t(g / NS) & 1u, p.fault,
                                               p.wait_limit));
        if (!ok) break;
        fence_after();
        if (elect_lane()) {  // S(g) = Q K^T into S buffer g % 3 (PV(g - 3) has read its P)
          const uint64_t kb = kd + ((buf * Lay::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * Lay::kQBoxBytes + (kk & 3) * 32;
            const uint32_t boff = (kk >> 2) * Lay::kBoxBytes + (kk & 3) * 32;
            mma_f16_ss(tmem + Lay::kColS + kTok0 * (g % kSBufs0), qk + (aoff >> 4), kb + (boff >> 4), id_s,
                       kk > 0 ? 1u : 0u);
          }
          commit_to(bar(B0_SFULL + g % kSBufs0));
          if (run_ends && j == x.n_tiles - 1) commit_to(bar(B0_QFREE + (run & 1)));   // Q tile may be refilled
        }
        __syncwarp();
        if (pn == 2 && !(ok = issue_pv())) break;   // PV(g - 2)
        const Pend e{g, run, new_run(k) && j == 0, run_ends && j == x.n_tiles - 1};
        if (pn == 0) q0 = e;
        else q1 = e;
        ++pn;
      }
    }
    while (ok && pn > 0) ok = issue_pv();
    // every MMA this warp issued has completed before TMEM is released
    if (elect_lane()) commit_to(bar(B0_DRAIN));
    __syncwarp();
    mbar_wait(bar(B0_DRAIN), 0u, p.fault, p.wait_limit);
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue warps
    // Thread = stacked row r = TMEM lane (a warp reaches the lanes of its quadrant,
    // warp % 4).  Two jobs per run: gather a later run's query rows into its Q tile,
    // and read out a finished run's O / l with its LSE.
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_base = tmem + (uint32_t(32 * (warp & 3)) << 16);
    // Run u's query rows into Q tile u % 2, 128-byte swizzled like a TMA box; rows past
    // the stacked count are zero.
    auto load_q = [&](int u) -> bool {
      if (u >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar(B0_QFREE + (u & 1)), uint32_t((u - 2) >> 1) & 1u,
                                                        p.fault, p.wait_limit)))
        return false;
      const Task x = task(run_first(u));
      const bool live = r < x.rows;
      const uint4 *src = nullptr;
      if (live) {
        int qb, head;
        row_source(x, x.row0 + r, qb, head);
        src = reinterpret_cast<const uint4 *>(p.q + (int64_t(qb) * p.Hq_req + head) * D);
      }
      uint8_t *qt = sm + Lay::kOffQ + (u & 1) * Lay::kQBytes + r * 128;
      uint4 v[D / 8];
#pragma unroll
      for (int j = 0; j < D / 8; ++j) v[j] = live ? __ldg(src + j) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        *reinterpret_cast<uint4 *>(qt + (j >> 3) * Lay::kQBoxBytes + (((j & 7) ^ (r & 7)) << 4)) = v[j];
      fence_proxy_async();  // generic writes, read by the MMAs (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B0_QFULL + (u & 1)));
      return true;
    };
    bool ok = true;
    if (n_runs > 0) ok = load_q(0);
    if (ok && n_runs > 1) ok = load_q(1);
    for (int u = 0; u < n_runs && ok; ++u) {
      const int k_last = run_end(u) - 1;
      const Task x = task(k_last);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B0_OFULL + (u & 1)), uint32_t(u >> 1) & 1u, p.fault,
                                             p.wait_limit));
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B0_LREADY + (u & 1)), uint32_t(u >> 1) & 1u, p.fault,
                                               p.wait_limit));
      if (!ok) break;
      fence_after();
      if (32 * (warp & 3) < x.rows) {
        const bool live = r < x.rows;
        uint32_t lmw[2];
        tmem_ld2(lane_base + Lay::kColLM + 2 * (u & 1), lmw);
        ld_wait();
        const float l_sum = __uint_as_float(lmw[0]), m_run = __uint_as_float(lmw[1]);
        int qb, head = 0;
        const int m = live ? row_source(x, x.row0 + r, qb, head) : 0;
        const int rbase = x.it.q_index >= 0 ? 0 : (live ? ld_list(row_base + m) : 0);
        const int64_t orow = int64_t(rbase + x.it.out_row) * p.Hq_req + head;
        float *dst = p.v_out + orow * D;
        const float inv = p.v_scale / l_sum;
        const uint32_t o_col = lane_base + Lay::kColO + D * (u & 1);
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          tmem_ld32(o_col + 32 * cb, o);
          ld_wait();
          if (live) {
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              const float v[8] = {__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                  __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv,
                                  __uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv,
                                  __uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv};
              st_v8(dst + 32 * cb + c, v);
            }
          }
        }
        if (live) {
          p.lse_out[orow] = m_run + log2f(l_sum);
          // the run's other chunks: empty rows (their v is not read by the merge)
          for (int k = run_first(u); k < k_last; ++k) {
            const int base = x.it.q_index >= 0 ? 0 : rbase;
            p.lse_out[int64_t(base + task(k).it.out_row) * p.Hq_req + head] = neg_inf();
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B0_OFREE + (u & 1)));   // the first PV of run u + 2 may overwrite O
      if (u + 2 < n_runs) ok = load_q(u + 2);
    }
  } else {
    // ------------------------------------------------------------------ row warps
    const int r = tid;                                  // stacked row in a task = TMEM lane
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    bool ok = true;
    const float qs = p.q_scale;
    int g = 0;  // tiles consumed so far (all tasks)
    float m_run = neg_inf(), l_sum = 0.f;  // the run's, m_run in log2 units of the scaled score
    for (int k = 0; k < n_mine && ok; ++k) {
      const Task x = task(k);
      const int run = run_of(k);
      const bool first_task = new_run(k);
      const bool warp_live = warp * 32 < x.rows;
      const bool warp_full = warp * 32 + 32 <= x.rows;   // every row of this warp is live
      const int row_valid = r < x.rows ? kTok0 : 0;
      const uint32_t o_col = lane_base + Lay::kColO + D * (run & 1);
      if (first_task) {
        m_run = neg_inf();
        l_sum = 0.f;
      }
      for (int j = 0; j < x.n_tiles; ++j, ++g) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B0_SFULL + g % kSBufs0), uint32_t(g / kSBufs0) & 1u, p.fault,
                                               p.wait_limit));
        if (!ok) break;
        fence_after();
        const int valid_tile = min(kTok0, x.it.n_tokens - j * kTok0);
        const uint32_t s_col = lane_base + Lay::kColS + kTok0 * (g % kSBufs0);
        if (warp_live) {
          uint32_t w[64];
          tmem_ld32(s_col, *reinterpret_cast<uint32_t(*)[32]>(w));
          tmem_ld32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(w + 32));
          ld_wait();
          // Full tiles of fully live warps need no mask; otherwise masked scores are
          // -inf (a dead row's scores are garbage, NaN included).
          const bool masked = !(warp_full && valid_tile == kTok0);
          const int valid = min(valid_tile, row_valid);
          float smax = neg_inf();
          if (!masked) {
#pragma unroll
            for (int c = 0; c < 64; ++c) smax = fmaxf(smax, __uint_as_float(w[c]));
          } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const float s = c < valid ? __uint_as_float(w[c]) : neg_inf();
              w[c] = __float_as_uint(s);
              smax = fmaxf(smax, s);
            }
          }
          const float tmax = smax * qs;   // qs > 0
          const bool grow = tmax > m_run + kLazy0;
          if (__any_sync(0xffffffffu, grow)) {
            const float m_new = grow ? tmax : m_run;
            if (j > 0 || !first_task) {  // PV(g - 1) of this run must be done; rescale O in TMEM
              ok = __all_sync(0xffffffffu, mbar_wait(bar(B0_KEMPTY + (g - 1) % NS), uint32_t((g - 1) / NS) & 1u,
                                                     p.fault, p.wait_limit));
              if (!ok) break;
              fence_after();
              const float alpha = grow ? ex2(m_run - m_new) : 1.f;
#pragma unroll 1
              for (int cb = 0; cb < D / 32; ++cb) {
                uint32_t o[32];
                tmem_ld32(o_col + 32 * cb, o);
                ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                tmem_st32(o_col + 32 * cb, o);
              }
              l_sum *= alpha;
            }
            m_run = m_new;
          }
          // P = 2^(s qs - m_run) <= 2^8 (0 for masked tokens), as bf16 hi and lo words
          // of two tokens each; l sums the unsplit P in f32.  A row with no valid token
          // yet (m_run = -inf) gets P = 0 through the -inf scores.
          const float nm = m_run == neg_inf() ? 0.f : -m_run;
          uint32_t ph[32], pl[32];
          float2 lacc = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float a = ex2(fmaf(__uint_as_float(w[2 * c]), qs, nm));
            const float b = ex2(fmaf(__uint_as_float(w[2 * c + 1]), qs, nm));
            lacc = __fadd2_rn(lacc, make_float2(a, b));
            ph[c] = bf16x2_bits(a, b);
            pl[c] = bf16x2_bits(a - bf16_lo(ph[c]), b - bf16_hi(ph[c]));
          }
          l_sum += lacc.x + lacc.y;
          tmem_st32(s_col, ph);
          tmem_st32(s_col + 32, pl);
        }
        if (valid_tile < kTok0) {
          // Rows past the item's last token (inside its last page) may hold anything,
          // NaN included: zero them in this stage's V boxes, so that P = 0 never meets
          // a NaN.  The tile has landed (S of it is complete).
          uint8_t *vt = ring + (g % NS) * Lay::kStageBytes + Lay::kHalfBytes;
          const int n16 = (kTok0 - valid_tile) * 8;   // 16-byte chunks per box column
#pragma unroll 1
          for (int c = r; c < Lay::kBoxes * n16; c += 32 * kRowWarps0)
            *reinterpret_cast<uint4 *>(vt + (c / n16) * Lay::kBoxBytes + valid_tile * 128 + (c % n16) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async();
        }
        st_wait();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B0_PFULL + g % kSBufs0));
      }
      if (!ok) break;
      if (!last_of_run(k)) continue;
      // l and m of this run's rows for the epilogue warps; their slot was read out for
      // run - 2 (normally long done)
      if (run >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B0_OFREE + (run & 1)), uint32_t((run - 2) >> 1) & 1u, p.fault,
                                               p.wait_limit));
      if (!ok) break;
      {
        const uint32_t lmw[2] = {__float_as_uint(l_sum), __float_as_uint(m_run)};
        tmem_st2(lane_base + Lay::kColLM + 2 * (run & 1), lmw);
        st_wait();
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B0_LREADY + (run & 1)));
    }
  }
  fence_before();
  __syncthreads();
  if (warp == kCtrlWarp0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Lay::kTmemCols));
  }
}

bool encode_l0_map(CUtensorMap *map, const DeviceInfo &dev, const void *pool, int64_t num_pages, int page_size,
                   int Hkv, int D) {
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(dev.encode_tiled);
  if (!encode) return false;
  cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(page_size), cuuint64_t(num_pages)};
  cuuint64_t strides[3] = {cuuint64_t(D) * 2, cuuint64_t(Hkv) * D * 2, cuuint64_t(page_size) * Hkv * D * 2};
  cuuint32_t box[4] = {64, 1, cuuint32_t(kSub0), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int CAP>
psd_status run_l0(dim3 grid, cudaStream_t s, const CUtensorMap &tmK, const CUtensorMap &tmV, const L0Params &p,
                  const InlineLists *lists) {
  auto kern = partial_l0_kernel<D, CAP>;
  constexpr size_t smem = L0Layout<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  if constexpr (CAP == 0) {
    kern<<<grid, kThreads0, smem, s>>>(tmK, tmV, p, NoInline{});
  } else {
    ListParam<CAP> blk;
    std::memcpy(blk.bytes, lists->bytes, lists->used);
    kern<<<grid, kThreads0, smem, s>>>(tmK, tmV, p, blk);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "partial (level-0 tcgen05) launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

template <int D>
psd_status launch_l0(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  CUtensorMap tmK, tmV;
  if (!encode_l0_map(&tmK, dev, L.k_pool, L.num_pages, L.page_size, L.Hkv, D) ||
      !encode_l0_map(&tmV, dev, L.v_pool, L.num_pages, L.page_size, L.Hkv, D))
    return fail(PSD_ERR_CUDA, "cuTensorMapEncodeTiled (128B swizzle) failed for the KV pool");
  L0Params p;
  p.q = reinterpret_cast<const __nv_bfloat16 *>(L.q);
  p.page_indices = L.page_indices;
  p.items = L.items;
  p.members = L.members;
  p.member_row_base = L.member_row_base;
  p.inl_items = L.inl_items;
  p.inl_members = L.inl_members;
  p.inl_row_base = L.inl_row_base;
  p.v_out = L.v_out;
  p.lse_out = L.lse_out;
  p.fault = L.fault;
  p.num_pages = L.num_pages;
  p.Hq_req = L.Hq_req;
  p.page_size = L.page_size;
  p.Gm = L.Gm;
  p.G_rows = L.G_cta;
  p.Hkv = L.Hkv;
  p.n_items = L.num_items;
  p.runs = L.merge_runs ? 1 : 0;
  p.n_rb = (L.G_cta + kRows0 - 1) / kRows0;
  const int64_t tasks = int64_t(L.num_items) * L.Hkv * p.n_rb;
  if (tasks > 0x7fffffffLL) return fail(PSD_ERR_UNSUPPORTED, "level-0 tcgen05 partial: %lld tasks", (long long)tasks);
  p.num_tasks = int(tasks);
  p.q_scale = L.q_scale;
  p.v_scale = L.v_scale;
  p.wait_limit = dev.test_wait_limit > 0 ? dev.test_wait_limit : kWaitLimitCycles;
  p.withhold_from = dev.test_withhold_from >= 0 ? dev.test_withhold_from : 0x7fffffff;
  // persistent: one CTA per SM (its shared memory and 512 TMEM columns fill the SM)
  const int sms = dev.num_sms > 0 ? dev.num_sms : 1;
  const dim3 grid(unsigned(tasks < sms ? tasks : sms));
  if (!L.inline_lists) return run_l0<D, 0>(grid, s, tmK, tmV, p, nullptr);
  const size_t used = L.inline_lists->used;
  if (used <= 4096) return run_l0<D, 4096>(grid, s, tmK, tmV, p, L.inline_lists);
  if (used <= 8192) return run_l0<D, 8192>(grid, s, tmK, tmV, p, L.inline_lists);
  if (used <= 16384) return run_l0<D, 16384>(grid, s, tmK, tmV, p, L.inline_lists);
  return fail(PSD_ERR_INVALID_ARG, "inline lists of %zu bytes", used);
}

}  // namespace

bool partial_l0_supports(const PartialLaunch &p) {
  // q_scale > 0: the kernel takes the row max of the raw scores before scaling
  return p.kv_dtype == PSD_BF16 && !p.latent_v && p.Dqk == p.Dv && (p.Dqk == 64 || p.Dqk == 128) &&
         p.G_cta >= 1 && p.page_size % kSub0 == 0 && p.q_scale > 0.f;
}

psd_status launch_partial_l0(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  if (L.num_items == 0) return PSD_OK;
  switch (L.Dqk) {
    case 64: return launch_l0<64>(L, dev, s);
    case 128: return launch_l0<128>(L, dev, s);
    default: return fail(PSD_ERR_UNSUPPORTED, "level-0 tcgen05 partial: head dim %d", L.Dqk);
  }
}

}  // namespace psd
