// K1t: split-KV partial attention with QK^T and PV on the tensor cores, in 16-row
// groups: small query groups (G = Hq/Hkv <= 16) in one CTA per (item, KV head),
// and the stacked level-0 rows (M*G) split over grid.z groups of 16.
//
// Same work unit as the CUDA-core kernel (mlxcel PR #1004, Decomposition section:
// one CTA owns all query heads of one KV head for one (request, page tile), so
// each K/V element is read from HBM once) and the same outputs (Merge contract
// section: rows normalised by their own denominator, LSE = m + log2 l in log2
// units).  The difference is where the arithmetic runs: at G = 4 the CUDA-core
// kernel spends ~90 issue slots per (token, KV head) on unpacking, FMAs and
// shuffles and cannot keep up with HBM, while one m16n8k16 MMA covers 16 tokens x
// 16 dims for all G rows (padded to 16) in one issue slot.
//
// GB300 shape: grid = (work items, Hkv, blocks of up to 64 rows), 4 warps, 3 CTAs
// per SM.  Each tile is 16 slots of one page loaded by TMA in 64-column boxes with
// the 128-byte swizzle, so ldmatrix reads are bank-conflict free.  Per tile and
// warp: S = Q K^T (D/16 x 2 MMAs, Q fragments held in registers), online softmax on
// the accumulator fragments, P re-packed as the A operand, O += P V (D/8 MMAs, V
// via transposed ldmatrix).  Two ways to spread a CTA's work over its warps:
//   - up to 48 rows (small query groups): one CTA per 16-row group, in which warp
//     w streams tiles w, w+4, ... through a private 2-stage ring and the four warp
//     states merge through shared memory;
//   - more rows (stacked level-0 rows, large groups): one CTA per block of 64 rows,
//     in which warp w owns rows 16w..16w+15 and every warp consumes every tile of
//     one CTA-wide 8-stage ring, so a tile crosses from L2 to the SM once for 64
//     rows, not once per 16.  The last warp to release a stage refills it.  With
//     only 2 or 3 groups the per-group CTAs win: a block would leave warps idle.
//     A block's CTA runs four times as long as a group's, so the launch takes the
//     blocks only when they fill at least one wave of resident CTAs; fewer, longer
//     CTAs would set the launch's tail.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

constexpr int kWarpsS = 4;
constexpr int kStagesS = 2;
constexpr int kTileTok = 16;
constexpr float kLazyRescale = 8.f;  // log2 units

struct TCSParams {
  const __nv_bfloat16 *q;
  const int32_t *page_indices;
  const psd_work_item *items;
  const int32_t *order;
  const int32_t *members;
  const int32_t *member_row_base;
  uint32_t inl_items, inl_order, inl_members, inl_row_base;  // offsets in the inline lists
  int has_order;
  float *v_out;
  float *lse_out;
  FaultRef fault;
  int64_t num_pages;
  int Hq_req, Dqk, Dv, page_size, Gm, G_cta;
  int tpp_log2;  // log2(page_size / 16), or -1
  // Fused cascade launch: CTAs [0, n_l0_tasks) are level-0 tasks of nseg segments;
  // segment s owns tasks [seg_task_end[s-1], seg_task_end[s]) = its items from
  // seg_item0[s] times its ceil(seg_rows[s] / 16) row groups, with member entries
  // from seg_member0[s].  The rest take level-1 items l1_base + order[...].  A plain
  // launch has n_l0_tasks = 0 and l1_base = 0.
  int n_l0_tasks, l1_base, nseg;
  int allow_shared;  // rows > 48 take 64-row blocks (the shared-tile form)
  int seg_task_end[PartialLaunch::kMaxFusedSegments], seg_item0[PartialLaunch::kMaxFusedSegments];
  int seg_rows[PartialLaunch::kMaxFusedSegments], seg_member0[PartialLaunch::kMaxFusedSegments];
  float q_scale, v_scale;
  // Testing aid: tiles at this index and later get no loads (INT_MAX: all do), and a
  // wait gives up after wait_limit cycles.
  int withhold_from;
  long long wait_limit;
};

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
// The same two loads at a compile-time byte offset from `addr` (folded into the
// instruction's address).
template <int OFF>
__device__ __forceinline__ void ldsm_x4_at(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                           uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4 + %5];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr), "n"(OFF));
}
template <int OFF>
__device__ __forceinline__ void ldsm_x4_t_at(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                             uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4 + %5];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr), "n"(OFF));
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F &&f) {
  if constexpr (N > 0) {
    static_for<N - 1>(f);
    f(std::integral_constant<int, N - 1>{});
  }
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of (row, 8-column chunk `col8`) in a tile stored as 64-column boxes
// of 16 rows x 128 bytes with the 128-byte swizzle (16-byte chunk index XOR row%8).
__device__ __forceinline__ uint32_t sw128(int row, int col8) {
  return uint32_t((col8 >> 3) * (kTileTok * 128) + row * 128 + (((col8 & 7) ^ (row & 7)) << 4));
}

// CTAs per (item, KV head) for `rows` query rows: one per 16-row group (the
// private form), or, where the launch allows it and there are more than 3 groups,
// one per block of up to 4 groups (the shared-tile form).
__host__ __device__ __forceinline__ bool tcs_shared_tiles(int rows, bool allow) { return allow && rows > 48; }
__host__ __device__ __forceinline__ int tcs_blocks(int rows, bool allow) {
  const int groups = (rows + 15) >> 4;
  return tcs_shared_tiles(rows, allow) ? (groups + kWarpsS - 1) / kWarpsS : groups;
}

// CAP > 0: the work lists come in the launch's parameters (`lists`, CAP bytes), not
// from global memory.
template <int D, int CAP>
__global__ void __launch_bounds__(kWarpsS * 32, D >= 256 ? 1 : 3)
    partial_tcs_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const TCSParams p,
                       const __grid_constant__ ListParam<CAP> lists) {
  constexpr bool INL = CAP != 0;
  constexpr int KSTEPS = D / 16;
  constexpr int NT = D / 8;                       // n8 tiles of the output
  constexpr uint32_t TILE_BYTES = kTileTok * D * 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  dependents_may_launch();  // the merge that follows only waits for this grid

  // 128-byte-swizzled TMA boxes need 1024-byte aligned destinations.
  uint8_t *base = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const psd_work_item *items = p.items;
  const int32_t *order = p.order, *members = p.members, *row_base = p.member_row_base;
  if constexpr (INL) {
    items = reinterpret_cast<const psd_work_item *>(lists.bytes + p.inl_items);
    order = p.has_order ? reinterpret_cast<const int32_t *>(lists.bytes + p.inl_order) : nullptr;
    members = reinterpret_cast<const int32_t *>(lists.bytes + p.inl_members);
    row_base = reinterpret_cast<const int32_t *>(lists.bytes + p.inl_row_base);
  }
  // list entries: parameter-space loads when inline, read-only global loads otherwise
  auto ld_list = [](const int32_t *a) -> int32_t {
    if constexpr (INL) return *a;
    else return __ldg(a);
  };
  int item_index, block, G_rows, member0 = 0;
  if (int(blockIdx.x) < p.n_l0_tasks) {
    const int task = int(blockIdx.x);
    int sg = 0;
    while (sg + 1 < p.nseg && task >= p.seg_task_end[sg]) ++sg;
    const int local = task - (sg ? p.seg_task_end[sg - 1] : 0);
    const int cpi = tcs_blocks(p.seg_rows[sg], p.allow_shared);
    item_index = p.seg_item0[sg] + local / cpi;
    block = local - (local / cpi) * cpi;
    G_rows = p.seg_rows[sg];
    member0 = p.seg_member0[sg];
  } else {
    const int j = blockIdx.x - p.n_l0_tasks;
    item_index = p.l1_base + (order ? ld_list(order + j) : j);
    block = blockIdx.z;
    G_rows = p.G_cta;
  }
  const psd_work_item it = items[item_index];
  const int kv = blockIdx.y;
  // Shared-tile form: warp w owns rows row0 .. row0 + 15 of the block's 64; warps
  // past the last row group only take part in the barrier set-up.
  const bool shared_tiles = tcs_shared_tiles(G_rows, p.allow_shared);
  const int row0 = shared_tiles ? block * 16 * kWarpsS + 16 * warp : block * 16;
  const int rows = min(16, G_rows - row0);
  const int n_active = shared_tiles ? min(kWarpsS, ((G_rows + 15) >> 4) - block * kWarpsS) : kWarpsS;
  const int P = p.page_size;
  const int TPP = P / kTileTok;
  const size_t ring_total = size_t(kWarpsS) * kStagesS * 2 * TILE_BYTES;
  const size_t red_total = size_t(kWarpsS) * 16 * (D + 2) * sizeof(float);
  uint64_t *bars_all = reinterpret_cast<uint64_t *>(base + (ring_total > red_total ? ring_total : red_total));
  uint32_t *released = reinterpret_cast<uint32_t *>(bars_all + kWarpsS * kStagesS);  // shared form
  uint8_t *ring = shared_tiles ? base : base + size_t(warp) * kStagesS * 2 * TILE_BYTES;
  uint64_t *bars = shared_tiles ? bars_all : bars_all + warp * kStagesS;
  if (shared_tiles) {
    if (threadIdx.x == 0) {
      for (int s = 0; s < kWarpsS * kStagesS; ++s) {
        mbar_init(smem_u32(&bars_all[s]), 1);
        released[s] = 0u;
      }
      fence_mbar_init();
    }
    __syncthreads();
    if (warp >= n_active) return;
  }

  // ---- Q fragments (rows >= G_cta are zero), pre-scaling is applied to S
  uint32_t qa[KSTEPS][4];
  {
    const int r0 = lane >> 2, c0 = (lane & 3) * 2;
    const __nv_bfloat16 *qrow[2] = {nullptr, nullptr};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int g = row0 + r0 + 8 * h;
      if (g < G_rows) {
        const int m = g / p.Gm;
        const int qb = it.q_index >= 0 ? it.q_index : ld_list(members + member0 + m);
        const int head = kv * p.Gm + (g - m * p.Gm);
        qrow[h] = p.q + (int64_t(qb) * p.Hq_req + head) * p.Dqk;
      }
    }
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const int c = kk * 16 + c0;
      qa[kk][0] = qrow[0] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[0] + c)) : 0u;
      qa[kk][1] = qrow[1] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[1] + c)) : 0u;
      qa[kk][2] = qrow[0] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[0] + c + 8)) : 0u;
      qa[kk][3] = qrow[1] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[1] + c + 8)) : 0u;
    }
  }

  const int n_tiles = (it.n_tokens + kTileTok - 1) / kTileTok;
  const int my_tiles = shared_tiles ? n_tiles
                                    : (n_tiles > warp ? (n_tiles - warp + kWarpsS - 1) / kWarpsS : 0);
  const int n_item_pages = (it.n_tokens + P - 1) / P;
  const uint64_t pol = l2_evict_first_policy();
  auto tile_pos = [&](int t) { return p.tpp_log2 >= 0 ? t >> p.tpp_log2 : t / TPP; };
  auto load_window = [&](int first) {
    const int pos = first + lane;
    return pos < n_item_pages ? __ldg(p.page_indices + it.page_off + pos) : -1;
  };
  int win_i = 0, pid_i = load_window(0);
  int win_c = 0, pid_c = pid_i;
  auto page_id = [&](int pos, int &win, int &pid) {
    if (pos - win >= 32) {
      win = pos & ~31;
      pid = load_window(win);
    }
    return __shfl_sync(0xffffffffu, pid, pos - win);
  };

  if (!shared_tiles) {
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < kStagesS; ++s) mbar_init(smem_u32(&bars[s]), 1);
      fence_mbar_init();
    }
    __syncwarp();
  }
  // stages of the ring this warp reads, and the tile of the item its i-th use holds
  const int n_stages = shared_tiles ? kWarpsS * kStagesS : kStagesS;
  auto tile_of = [&](int i) { return shared_tiles ? i : warp + i * kWarpsS; };

  auto issue = [&](int i) {  // all lanes call; lane 0 issues
    const int s = i % n_stages;
    const int t = tile_of(i);
    const int pos = tile_pos(t);
    const int id = page_id(pos, win_i, pid_i);
    if (lane == 0) {
      const int slot0 = (t - pos * TPP) * kTileTok;
      const uint32_t bar = smem_u32(&bars[s]);
      if (t >= p.withhold_from) {
        // testing aid: no load and no arrival, so the wait for this tile runs out.
        // Every later tile is withheld as well, and the tiles before it were waited
        // for first, so no copy is in flight when that wait gives up.
      } else if (id < 0 || int64_t(id) >= p.num_pages) {
        raise_fault(p.fault, PSD_FAULT_PAGE_ID);
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, 2 * TILE_BYTES);
        uint8_t *kb = ring + size_t(s) * 2 * TILE_BYTES;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(smem_u32(kb + c * kTileTok * 128), &tmK, c * 64, kv, slot0, id, bar, pol);
          tma_load_4d(smem_u32(kb + TILE_BYTES + c * kTileTok * 128), &tmV, c * 64, kv, slot0, id,
                      bar, pol);
        }
      }
    }
  };
  if (!shared_tiles || warp == 0) {
    const int pre = my_tiles < n_stages ? my_tiles : n_stages;
    for (int i = 0; i < pre; ++i) issue(i);
  }

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {neg_inf(), neg_inf()};
  float l_run[2] = {0.f, 0.f};

  // ldmatrix lane roles: QK^T B operand (K rows = tokens), PV B operand (V^T)
  const int kb_tok = (lane & 7) + ((lane >> 4) << 3);
  const int kb_c8 = (lane >> 3) & 1;
  const int vb_tok = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int vb_c8 = lane >> 4;
  // 16-byte chunk 2j + c of a box row sits at chunk (2j + c) ^ (row % 8), i.e. at
  // the byte offset of chunk c XOR 32 j (the row starts 128-byte aligned): one
  // per-lane offset for j = 0; later boxes add 2 KB (immediates).
  const uint32_t ko0 = uint32_t(kb_tok * 128 + ((kb_c8 ^ (kb_tok & 7)) << 4));
  const uint32_t vo0 = uint32_t(vb_tok * 128 + ((vb_c8 ^ (vb_tok & 7)) << 4));

  // V fragment masks of a tail tile in the shared form (tokens tk, tk+1 and tk+8,
  // tk+9 of the transposed ldmatrix); the private form zeroes the rows in its stage.
  const int tk = (lane & 3) * 2;
  int failed_at = -1;  // the tile whose wait ran out
  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % n_stages;
    const int t = tile_of(i);
    const int id = page_id(tile_pos(t), win_c, pid_c);
    const bool page_ok = id >= 0 && int64_t(id) < p.num_pages;
    const int valid = page_ok ? min(kTileTok, it.n_tokens - t * kTileTok) : 0;
    const bool ok = mbar_wait(smem_u32(&bars[s]), uint32_t(i / n_stages) & 1u, p.fault, p.wait_limit);
    if (!__all_sync(0xffffffffu, ok)) {
      failed_at = i;
      break;
    }
    if (valid > 0) {
      uint8_t *stage = ring + size_t(s) * 2 * TILE_BYTES;
      const bool vmask = shared_tiles && valid < kTileTok;
      const uint32_t m_lo = (tk < valid ? 0x0000FFFFu : 0u) | (tk + 1 < valid ? 0xFFFF0000u : 0u);
      const uint32_t m_hi = (tk + 8 < valid ? 0x0000FFFFu : 0u) | (tk + 9 < valid ? 0xFFFF0000u : 0u);
      if (!shared_tiles && valid < kTileTok) {
        // Tail tile: V rows past the last token hold other slots (or NaN canaries);
        // P is 0 there, so make them 0 too before the MMA multiplies them.
        constexpr int CH = (D / 64) * 8;  // 16-byte chunks per row
        for (int idx = lane; idx < (kTileTok - valid) * CH; idx += 32) {
          const int r = valid + idx / CH, c = idx % CH;
          *reinterpret_cast<uint4 *>(stage + TILE_BYTES + (c >> 3) * (kTileTok * 128) + r * 128 +
                                     (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async();  // these generic writes precede the next TMA into the slot
        __syncwarp();
      }
      const uint32_t kbase = smem_u32(stage);
      const uint32_t vbase = kbase + TILE_BYTES;
      // S = Q K^T over the tile's 16 tokens: even and odd k-steps accumulate apart
      // (two shorter MMA chains), then add
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t kq = kbase + ko0;
      static_for<KSTEPS>([&](auto kc) {
        constexpr int kk = decltype(kc)::value;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_at<(kk >> 2) * kTileTok * 128>(kq ^ uint32_t(32 * (kk & 3)), b0, b1, b2, b3);
        float(&acc)[2][4] = (kk & 1) ? sd : sc;
        mma16816(acc[0], qa[kk], b0, b1);
        mma16816(acc[1], qa[kk], b2, b3);
      });
      // scale, mask (tail tiles only), online softmax (rows lane/4 and lane/4 + 8)
      float tmax[2] = {neg_inf(), neg_inf()};
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[n][j] = (sc[n][j] + sd[n][j]) * p.q_scale;
      if (valid < kTileTok) {
        const int tok0 = (lane & 3) * 2;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (n * 8 + tok0 + (j & 1) >= valid) sc[n][j] = neg_inf();
      }
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) tmax[j >> 1] = fmaxf(tmax[j >> 1], sc[n][j]);
      // Lazy rescale: the running max moves only when a row's tile max exceeds it by
      // more than 2^8 (P <= 2^8 otherwise, far inside f32 and bf16 range).
      bool grow[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
        tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
        grow[h] = tmax[h] > m_run[h] + kLazyRescale;
      }
      if (__any_sync(0xffffffffu, grow[0] || grow[1])) {
        const float a0 = grow[0] ? ex2(m_run[0] - tmax[0]) : 1.f;
        const float a1 = grow[1] ? ex2(m_run[1] - tmax[1]) : 1.f;
        l_run[0] *= a0;
        l_run[1] *= a1;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][0] *= a0;
          o[n][1] *= a0;
          o[n][2] *= a1;
          o[n][3] *= a1;
        }
        if (grow[0]) m_run[0] = tmax[0];
        if (grow[1]) m_run[1] = tmax[1];
      }
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          sc[n][j] = ex2(sc[n][j] - m_run[j >> 1]);
          l_run[j >> 1] += sc[n][j];
        }
      // P as two bf16 terms, P = hi + lo with |lo| <= 2^-9 |P|: both go through the
      // MMA so P V keeps ~16 mantissa bits (one bf16 P would cost up to 2^-10 |v|
      // on short chunks).
      uint32_t pa[4], pl[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x0 = sc[k >> 1][(k & 1) * 2], x1 = sc[k >> 1][(k & 1) * 2 + 1];
        pa[k] = pack_bf16x2(x0, x1);
        pl[k] = pack_bf16x2(x0 - bf16_lo(pa[k]), x1 - bf16_hi(pa[k]));
      }
      // O += P V (in the shared form, V of a tail tile's dead tokens is zeroed in
      // the fragments)
      const uint32_t vq = vbase + vo0;
      auto pv = [&](auto masked) {
        static_for<NT / 2>([&](auto nc) {
          constexpr int n = 2 * decltype(nc)::value;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t_at<(n >> 3) * kTileTok * 128>(vq ^ uint32_t(32 * ((n >> 1) & 3)), b0, b1, b2, b3);
          if constexpr (decltype(masked)::value) {
            b0 &= m_lo;
            b1 &= m_hi;
            b2 &= m_lo;
            b3 &= m_hi;
          }
          mma16816(o[n], pa, b0, b1);
          mma16816(o[n + 1], pa, b2, b3);
          mma16816(o[n], pl, b0, b1);
          mma16816(o[n + 1], pl, b2, b3);
        });
      };
      if (vmask) pv(std::true_type{});
      else pv(std::false_type{});
    }
    __syncwarp();
    if (!shared_tiles) {
      if (i + kStagesS < my_tiles) issue(i + kStagesS);
    } else {
      // Release the stage; the warp whose release completes this use refills it.
      // The counter only grows: use u of a stage is complete at (u + 1) * n_active.
      uint32_t last = 0;
      if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(&released[s], 1u) == uint32_t(i / n_stages + 1) * uint32_t(n_active) - 1u;
      }
      if (__shfl_sync(0xffffffffu, last, 0) && i + n_stages < my_tiles) {
        __threadfence_block();
        issue(i + n_stages);
      }
    }
  }

  if (failed_at >= 0) {
    // A wait ran out.  Copies issued for tiles failed_at .. failed_at + n_stages - 1
    // (by this warp, or in the shared form by whichever warp refilled the stage) land
    // before it goes on: it waits for each such tile that the testing aid did not
    // withhold.  Each stage's previous use is consumed, so every wait is for the phase
    // in progress; a tile nobody issued only runs out the limit once more.
    for (int j = failed_at; j < failed_at + n_stages && j < my_tiles; ++j)
      if (tile_of(j) < p.withhold_from)
        mbar_wait(smem_u32(&bars[j % n_stages]), uint32_t(j / n_stages) & 1u, p.fault, p.wait_limit);
  }

  if (shared_tiles) {  // this warp's rows are complete: write them
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = (lane >> 2) + 8 * h;
      if (r >= rows) continue;
      const int g = row0 + r;
      const bool live = m_run[h] != neg_inf();
      const float f = live ? p.v_scale / l_run[h] : 0.f;
      const int m = g / p.Gm;
      const int row = it.q_index >= 0 ? it.out_row : ld_list(row_base + member0 + m) + it.out_row;
      const int head = kv * p.Gm + (g - m * p.Gm);
      const int64_t orow = int64_t(row) * p.Hq_req + head;
      float *dst = p.v_out + orow * p.Dv + (lane & 3) * 2;
#pragma unroll
      for (int n = 0; n < NT; ++n)
        *reinterpret_cast<float2 *>(dst + n * 8) = make_float2(o[n][2 * h] * f, o[n][2 * h + 1] * f);
      if ((lane & 3) == 0) p.lse_out[orow] = live ? m_run[h] + log2f(l_run[h]) : neg_inf();
    }
    return;
  }

  // ---- merge the four warps through shared memory (rings no longer used).  Only
  // the live rows are staged; each row's 8-float blocks are XOR-rotated by row % 4
  // so the fragment stores of four rows fall in four bank groups.
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  __syncthreads();
  float *red_o = reinterpret_cast<float *>(base);               // [kWarpsS][16][D]
  float *red_m = red_o + size_t(kWarpsS) * 16 * D;               // [kWarpsS][16]
  float *red_l = red_m + kWarpsS * 16;                           // [kWarpsS][16]
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = (lane >> 2) + 8 * h;
    if (r < rows) {
      float *dst = red_o + (size_t(warp) * 16 + r) * D;
      const int rot = (r & 3) << 3;
#pragma unroll
      for (int n = 0; n < NT; ++n)
        *reinterpret_cast<float2 *>(dst + ((n * 8 + (lane & 3) * 2) ^ rot)) =
            make_float2(o[n][2 * h], o[n][2 * h + 1]);
      if ((lane & 3) == 0) {
        red_m[warp * 16 + r] = m_run[h];
        red_l[warp * 16 + r] = l_run[h];
      }
    }
  }
  __syncthreads();
  constexpr int D4 = D / 4;
  for (int idx = threadIdx.x; idx < rows * D4; idx += kWarpsS * 32) {
    const int r = idx / D4, d = (idx - r * D4) * 4;
    const int g = row0 + r;
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kWarpsS; ++w) M = fmaxf(M, red_m[w * 16 + r]);
    float L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarpsS; ++w) {
      const float sc = ex2(red_m[w * 16 + r] - M);
      L = fmaf(sc, red_l[w * 16 + r], L);
      const float4 v = *reinterpret_cast<const float4 *>(red_o + (size_t(w) * 16 + r) * D +
                                                         (d ^ ((r & 3) << 3)));
      O.x = fmaf(sc, v.x, O.x);
      O.y = fmaf(sc, v.y, O.y);
      O.z = fmaf(sc, v.z, O.z);
      O.w = fmaf(sc, v.w, O.w);
    }
    const bool live = M != neg_inf();
    const float f = live ? p.v_scale / L : 0.f;
    const int m = g / p.Gm;
    const int row = it.q_index >= 0 ? it.out_row : ld_list(row_base + member0 + m) + it.out_row;
    const int head = kv * p.Gm + (g - m * p.Gm);
    const int64_t orow = int64_t(row) * p.Hq_req + head;
    *reinterpret_cast<float4 *>(p.v_out + orow * p.Dv + d) = make_float4(O.x * f, O.y * f, O.z * f, O.w * f);
    if (d == 0) p.lse_out[orow] = live ? M + log2f(L) : neg_inf();
  }
}

bool encode_sw128_map(CUtensorMap *map, const DeviceInfo &dev, const void *pool, int64_t num_pages,
                      int page_size, int Hkv, int D) {
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(dev.encode_tiled);
  if (!encode) return false;
  cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(page_size), cuuint64_t(num_pages)};
  cuuint64_t strides[3] = {cuuint64_t(D) * 2, cuuint64_t(Hkv) * D * 2,
                           cuuint64_t(page_size) * Hkv * D * 2};
  cuuint32_t box[4] = {64, 1, cuuint32_t(kTileTok), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
size_t tcs_smem_bytes() {
  const size_t ring = size_t(kWarpsS) * kStagesS * 2 * kTileTok * D * 2;
  const size_t red = size_t(kWarpsS) * 16 * (D + 2) * sizeof(float);
  return std::max(ring, red) + 1024 /* base alignment */ +
         kWarpsS * kStagesS * (sizeof(uint64_t) + sizeof(uint32_t)) /* barriers, release counters */;
}

template <int D, int CAP>
psd_status run_tcs(dim3 grid, size_t smem, cudaStream_t s, const CUtensorMap &tmK, const CUtensorMap &tmV,
                   const TCSParams &p, const InlineLists *lists);

template <int D>
psd_status launch_tcs(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  CUtensorMap tmK, tmV;
  if (!encode_sw128_map(&tmK, dev, L.k_pool, L.num_pages, L.page_size, L.Hkv, D) ||
      !encode_sw128_map(&tmV, dev, L.v_pool, L.num_pages, L.page_size, L.Hkv, D))
    return fail(PSD_ERR_CUDA, "cuTensorMapEncodeTiled (128B swizzle) failed for the KV pool");
  TCSParams p;
  p.q = reinterpret_cast<const __nv_bfloat16 *>(L.q);
  p.page_indices = L.page_indices;
  p.items = L.items;
  p.order = L.order;
  p.members = L.members;
  p.member_row_base = L.member_row_base;
  p.inl_items = L.inl_items;
  p.inl_order = L.inl_order;
  p.inl_members = L.inl_members;
  p.inl_row_base = L.inl_row_base;
  p.has_order = L.order != nullptr;
  p.v_out = L.v_out;
  p.lse_out = L.lse_out;
  p.fault = L.fault;
  p.num_pages = L.num_pages;
  p.Hq_req = L.Hq_req;
  p.Dqk = L.Dqk;
  p.Dv = L.Dv;
  p.page_size = L.page_size;
  p.Gm = L.Gm;
  p.G_cta = L.G_cta;
  const int tpp = L.page_size / kTileTok;
  p.tpp_log2 = (tpp & (tpp - 1)) == 0 ? __builtin_ctz(unsigned(tpp)) : -1;
  p.q_scale = L.q_scale;
  p.v_scale = L.v_scale;
  p.withhold_from = dev.test_withhold_from >= 0 ? dev.test_withhold_from : 0x7fffffff;
  p.wait_limit = dev.test_wait_limit > 0 ? dev.test_wait_limit : kWaitLimitCycles;
  p.n_l0_tasks = 0;
  p.l1_base = 0;
  p.nseg = 0;
  // The shared-tile form only where its CTAs fill a wave (3 resident per SM).
  const int64_t wave = int64_t(dev.num_sms > 0 ? dev.num_sms : 1) * 3;
  if (L.fused_segments > 0) {
    int64_t blocks = 0;
    for (int sg = 0; sg < L.fused_segments && sg < PartialLaunch::kMaxFusedSegments; ++sg)
      if (tcs_shared_tiles(L.seg_rows[sg], true))
        blocks += int64_t(L.seg_items[sg]) * tcs_blocks(L.seg_rows[sg], true) * L.Hkv;
    p.allow_shared = blocks >= wave;
  } else {
    p.allow_shared = tcs_shared_tiles(L.G_cta, true) &&
                     int64_t(L.num_items) * tcs_blocks(L.G_cta, true) * L.Hkv >= wave;
  }
  unsigned grid_x = static_cast<unsigned>(L.num_items),
           grid_z = static_cast<unsigned>(tcs_blocks(L.G_cta, p.allow_shared));
  if (L.fused_segments > 0) {  // level-0 items of every segment precede L.items' level-1 items
    if (L.fused_segments > PartialLaunch::kMaxFusedSegments)
      return fail(PSD_ERR_UNSUPPORTED, "fused cascade launch: %d segments > %d", L.fused_segments,
                  PartialLaunch::kMaxFusedSegments);
    int64_t tasks = 0;
    int item0 = 0;
    for (int sg = 0; sg < L.fused_segments; ++sg) {
      tasks += int64_t(L.seg_items[sg]) * tcs_blocks(L.seg_rows[sg], p.allow_shared);
      if (tasks > 0x7fffffffLL) return fail(PSD_ERR_UNSUPPORTED, "fused cascade launch: too many tasks");
      p.seg_task_end[sg] = int(tasks);
      p.seg_item0[sg] = item0;
      p.seg_rows[sg] = L.seg_rows[sg];
      p.seg_member0[sg] = L.seg_member0[sg];
      item0 += L.seg_items[sg];
    }
    p.nseg = L.fused_segments;
    p.n_l0_tasks = int(tasks);
    p.l1_base = item0;
    grid_x = static_cast<unsigned>(p.n_l0_tasks + L.num_items);
    grid_z = 1;  // level-1 items have G_cta <= 16 rows (checked by the caller)
  }
  const size_t smem = tcs_smem_bytes<D>();
  const dim3 grid(grid_x, static_cast<unsigned>(L.Hkv), grid_z);
  if (!L.inline_lists) return run_tcs<D, 0>(grid, smem, s, tmK, tmV, p, nullptr);
  const size_t used = L.inline_lists->used;
  if (used <= 4096) return run_tcs<D, 4096>(grid, smem, s, tmK, tmV, p, L.inline_lists);
  if (used <= 8192) return run_tcs<D, 8192>(grid, smem, s, tmK, tmV, p, L.inline_lists);
  if (used <= 16384) return run_tcs<D, 16384>(grid, smem, s, tmK, tmV, p, L.inline_lists);
  return fail(PSD_ERR_INVALID_ARG, "inline lists of %zu bytes", used);
}

template <int D, int CAP>
psd_status run_tcs(dim3 grid, size_t smem, cudaStream_t s, const CUtensorMap &tmK, const CUtensorMap &tmV,
                   const TCSParams &p, const InlineLists *lists) {
  auto kern = partial_tcs_kernel<D, CAP>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  }
  if constexpr (CAP == 0) {
    kern<<<grid, kWarpsS * 32, smem, s>>>(tmK, tmV, p, NoInline{});
  } else {
    ListParam<CAP> blk;
    std::memcpy(blk.bytes, lists->bytes, lists->used);
    kern<<<grid, kWarpsS * 32, smem, s>>>(tmK, tmV, p, blk);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "partial (small-group tensor cores) launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

}  // namespace

bool partial_tcs_supports(const PartialLaunch &p) {
  return p.kv_dtype == PSD_BF16 && !p.latent_v && p.Dqk == p.Dv &&
         (p.Dqk == 64 || p.Dqk == 128 || p.Dqk == 256) && p.G_cta >= 1 && p.G_cta <= 256 &&
         p.page_size % kTileTok == 0;
}

psd_status launch_partial_tcs(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  if (L.num_items == 0 && L.fused_l0_items == 0) return PSD_OK;
  switch (L.Dqk) {
    case 64: return launch_tcs<64>(L, dev, s);
    case 128: return launch_tcs<128>(L, dev, s);
    case 256: return launch_tcs<256>(L, dev, s);
    default: return fail(PSD_ERR_UNSUPPORTED, "small-group tensor-core partial: head dim %d", L.Dqk);
  }
}

}  // namespace psd
