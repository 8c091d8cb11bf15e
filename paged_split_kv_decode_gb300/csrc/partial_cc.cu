// K1: split-KV partial attention on CUDA cores for G = Hq/Hkv <= 8.
//
// mlxcel PR #1004 ("compute shared prompt prefixes once per decode batch"),
// Decomposition section: one CTA owns all G query heads of one KV head for one
// (request, page tile), so every K/V element is read from HBM exactly once and
// reused by the G heads; Merge contract section: each row leaves normalised by
// its own denominator with LSE = m + log2(l) in log2 units.
//
// GB300 shape: grid = (work items, Hkv), 4 warps, 4 CTAs per SM (16 warps).  The
// item's tokens are cut into ring tiles of gcd(page_size, 8) consecutive slots of
// one page; warp w streams tiles w, w+4, ... through a private 3-stage ring: one
// TMA box per tile for K and one for V ({D, 1 head, tile slots}), completing on an
// mbarrier, L2 evict-first.  A token row is D/8 lanes x 16 bytes (128-bit shared
// loads).  The G partial dot products of a lane are summed over the row's lanes by
// a halving ("transpose") butterfly that leaves one full score per lane, so the
// exponentials are computed once per (head, token); products use packed f32x2
// FMAs.  The online softmax advances once per tile, and the four warp states are
// merged through shared memory.  Queries are pre-scaled by sm_scale*log2(e) so
// scores are already in log2 units.  CTAs visit items longest first.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

constexpr int kWarps = 4;
constexpr int kStages = 3;

struct CCParams {
  const __nv_bfloat16 *q;
  const int32_t *page_indices;
  const psd_work_item *items;
  const int32_t *members;
  const int32_t *member_row_base;
  float *v_out;
  float *lse_out;
  FaultRef fault;
  int64_t num_pages;
  const int32_t *order;  // CTA -> item (longest items first), or NULL
  int Hq_req, Dqk, Dv, page_size, sub, Gm, G_cta;  // sub = tokens per ring tile
  int tpp_log2;  // log2(page_size / sub), or -1 if not a power of two
  float q_scale, v_scale;
  // Testing aid: tiles at this index and later get no loads (INT_MAX: all do), and a
  // wait gives up after wait_limit cycles.
  int withhold_from;
  long long wait_limit;
};

// Sums G per-lane values over the LPT lanes of a token slot, halving the number
// of values per lane at each butterfly step: afterwards lane l holds the full sum
// of value (l % LPT) / (LPT / G).  log2(G) select/shuffle halvings plus
// log2(LPT / G) plain steps instead of G * log2(LPT) shuffles.
template <int G, int LPT>
__device__ __forceinline__ float transpose_reduce(float (&v)[G], int lane) {
  float cur[G];
#pragma unroll
  for (int g = 0; g < G; ++g) cur[g] = v[g];
  int off = LPT / 2;
#pragma unroll
  for (int n = G; n > 1; n >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;  // this lane keeps the upper half
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = upper ? cur[k] : cur[k + n / 2];
      const float keep = upper ? cur[k + n / 2] : cur[k];
      cur[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = cur[0];
#pragma unroll
  for (; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, G <= 4 ? 4 : 2)
    partial_cc_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const CCParams p) {
  constexpr int LPT = D / 8;         // lanes per token row (8 bf16 = 16 bytes per lane)
  constexpr int TPS = 32 / LPT;      // tokens per warp step
  constexpr int HL = LPT / G;        // lanes per head after the transpose reduce
  static_assert(G <= LPT, "one score per lane needs G <= D / 8");
  extern __shared__ __align__(1024) uint8_t smem[];
  dependents_may_launch();  // the merge that follows only waits for this grid

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const psd_work_item it = p.items[p.order ? __ldg(p.order + blockIdx.x) : blockIdx.x];
  const int kv = blockIdx.y;
  const int P = p.page_size;
  const int SUB = p.sub;          // ring tile = SUB consecutive slots of one page
  const int TPP = P / SUB;        // tiles per page
  const int steps = SUB / TPS > 0 ? SUB / TPS : 1;
  const uint32_t tile_bytes = uint32_t(SUB) * D * 2;
  uint8_t *ring = smem + size_t(warp) * kStages * 2 * tile_bytes;
  const size_t stage_total = size_t(kWarps) * kStages * 2 * tile_bytes;
  const size_t red_total = size_t(kWarps) * G * (D + 2) * sizeof(float);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (stage_total > red_total ? stage_total : red_total)) +
                   warp * kStages;

  const int tslot = lane / LPT;
  const int sl = lane % LPT;
  const int d0 = sl * 8;
  const int my_head = sl / HL;  // the head whose score this lane holds after a reduce

  // Query rows of this CTA, pre-scaled into log2 units, as float pairs.
  float2 q2[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (g < p.G_cta) {
      const int m = g / p.Gm;
      const int qb = it.q_index >= 0 ? it.q_index : __ldg(p.members + m);
      const int head = kv * p.Gm + (g - m * p.Gm);
      const uint4 r = __ldg(reinterpret_cast<const uint4 *>(
          p.q + (int64_t(qb) * p.Hq_req + head) * p.Dqk + d0));
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        q2[g][e] = make_float2(bf16_lo(w[e]) * p.q_scale, bf16_hi(w[e]) * p.q_scale);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) q2[g][e] = make_float2(0.f, 0.f);
    }
  }

  const int n_tiles = (it.n_tokens + SUB - 1) / SUB;
  const int my_tiles = n_tiles > warp ? (n_tiles - warp + kWarps - 1) / kWarps : 0;
  const int n_item_pages = (it.n_tokens + P - 1) / P;
  const uint64_t pol = l2_evict_first_policy();

  // Tile t of the item sits in page position t / TPP at slot (t % TPP) * SUB.
  auto tile_pos = [&](int t) { return p.tpp_log2 >= 0 ? t >> p.tpp_log2 : t / TPP; };
  // Page ids of the item, 32 positions per window, one per lane; a window is
  // reloaded (warp-uniformly) only when a position leaves it.
  auto load_window = [&](int base) {
    const int pos = base + lane;
    return pos < n_item_pages ? __ldg(p.page_indices + it.page_off + pos) : -1;
  };
  int win_i = 0, pid_i = load_window(0);  // window used to issue loads
  int win_c = 0, pid_c = pid_i;           // window used to consume tiles
  auto page_id = [&](int pos, int &win, int &pid) {  // all lanes, warp-uniform pos
    if (pos - win >= 32) {
      win = pos & ~31;
      pid = load_window(win);
    }
    return __shfl_sync(0xffffffffu, pid, pos - win);
  };

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int i) {  // all lanes call; lane 0 issues
    const int s = i % kStages;
    const int t = warp + i * kWarps;
    const int pos = tile_pos(t);
    const int id = page_id(pos, win_i, pid_i);
    if (lane == 0) {
      const int slot0 = (t - pos * TPP) * SUB;
      const uint32_t bar = smem_u32(&bars[s]);
      if (t >= p.withhold_from) {
        // testing aid: no load and no arrival, so the wait for this tile runs out.
        // Every later tile is withheld as well, and the tiles before it were waited
        // for first, so no copy is in flight when that wait gives up.
      } else if (id < 0 || int64_t(id) >= p.num_pages) {
        raise_fault(p.fault, PSD_FAULT_PAGE_ID);
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, 2 * tile_bytes);
        uint8_t *kb = ring + size_t(s) * 2 * tile_bytes;
        tma_load_4d(smem_u32(kb), &tmK, 0, kv, slot0, id, bar, pol);
        tma_load_4d(smem_u32(kb + tile_bytes), &tmV, 0, kv, slot0, id, bar, pol);
      }
    }
  };
  {
    const int pre = my_tiles < kStages ? my_tiles : kStages;
    for (int i = 0; i < pre; ++i) issue(i);
  }

  float m_run = neg_inf(), l_run = 0.f;  // for my_head, over this lane's token slot
  float2 acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[g][e] = make_float2(0.f, 0.f);

  // One ring tile: scores, online-softmax update, P V.  MASKED handles a tile with
  // fewer than SUB valid tokens (the item's last tile, or a skipped page).
  auto tile = [&](auto masked_tag, const uint8_t *kb, const uint8_t *vb, int valid) {
    constexpr bool MASKED = decltype(masked_tag)::value;
    float sc[8];
    float mt = neg_inf();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < steps) {
        const int tok = u * TPS + tslot;
        const bool ok = !MASKED || tok < valid;
        float part[G];
        if (ok) {
          const uint4 r = *reinterpret_cast<const uint4 *>(kb + (size_t(tok) * D + d0) * 2);
          const uint32_t w[4] = {r.x, r.y, r.z, r.w};
          float2 k2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) k2[e] = make_float2(bf16_lo(w[e]), bf16_hi(w[e]));
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float2 a = __fmul2_rn(q2[g][0], k2[0]);
#pragma unroll
            for (int e = 1; e < 4; ++e) a = __ffma2_rn(q2[g][e], k2[e], a);
            part[g] = a.x + a.y;
          }
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) part[g] = 0.f;
        }
        const float sv = transpose_reduce<G, LPT>(part, lane);
        sc[u] = ok ? sv : neg_inf();
        mt = fmaxf(mt, sc[u]);
      }
    }
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    // online softmax: rescale only when some head's running max moved
    const float m_new = fmaxf(m_run, mt);
    if (!__all_sync(0xffffffffu, m_new == m_run)) {
      const float alpha = ex2(m_run - m_new);  // 0 while m_run is -inf
      l_run *= alpha;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float ag = __shfl_sync(0xffffffffu, alpha, tslot * LPT + g * HL);
        const float2 a2 = make_float2(ag, ag);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][e] = __fmul2_rn(acc[g][e], a2);
      }
      m_run = m_new;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < steps) {
        const int tok = u * TPS + tslot;
        const float pm = ex2(sc[u] - m_run);  // 0 for masked tokens
        l_run += pm;
        float pg[G];
#pragma unroll
        for (int g = 0; g < G; ++g) pg[g] = __shfl_sync(0xffffffffu, pm, tslot * LPT + g * HL);
        if (!MASKED || tok < valid) {
          const uint4 r = *reinterpret_cast<const uint4 *>(vb + (size_t(tok) * D + d0) * 2);
          const uint32_t w[4] = {r.x, r.y, r.z, r.w};
          float2 v2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v2[e] = make_float2(bf16_lo(w[e]), bf16_hi(w[e]));
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float2 p2 = make_float2(pg[g], pg[g]);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[g][e] = __ffma2_rn(p2, v2[e], acc[g][e]);
          }
        }
      }
    }
  };

  const bool exact_steps = steps * TPS == SUB;
  int failed_at = -1;  // the tile whose wait ran out
  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % kStages;
    const int t = warp + i * kWarps;
    const int id = page_id(tile_pos(t), win_c, pid_c);
    const bool page_ok = id >= 0 && int64_t(id) < p.num_pages;
    const int valid = page_ok ? min(SUB, it.n_tokens - t * SUB) : 0;
    const bool ok = mbar_wait(smem_u32(&bars[s]), uint32_t(i / kStages) & 1u, p.fault, p.wait_limit);
    if (!__all_sync(0xffffffffu, ok)) {
      failed_at = i;
      break;
    }
    const uint8_t *kb = ring + size_t(s) * 2 * tile_bytes;
    const uint8_t *vb = kb + tile_bytes;
    if (valid == SUB && exact_steps)
      tile(std::integral_constant<bool, false>(), kb, vb, valid);
    else if (valid > 0)
      tile(std::integral_constant<bool, true>(), kb, vb, valid);
    __syncwarp();
    if (i + kStages < my_tiles) issue(i + kStages);
  }
  if (failed_at >= 0) {
    // A wait ran out.  The copies this warp issued for tiles failed_at ..
    // failed_at + kStages - 1 land before it goes on: it waits for each such tile that
    // the testing aid did not withhold.  Each stage's previous use is consumed, so every
    // wait is for the phase in progress; a tile it never loaded only runs out the limit
    // once more.
    for (int j = failed_at; j < failed_at + kStages && j < my_tiles; ++j)
      if (warp + j * kWarps < p.withhold_from)
        mbar_wait(smem_u32(&bars[j % kStages]), uint32_t(j / kStages) & 1u, p.fault, p.wait_limit);
  }

  // Combine the token slots of the warp (all slots share m_run per head).
#pragma unroll
  for (int off = LPT; off < 32; off <<= 1) {
    l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[g][e].x += __shfl_xor_sync(0xffffffffu, acc[g][e].x, off);
        acc[g][e].y += __shfl_xor_sync(0xffffffffu, acc[g][e].y, off);
      }
  }

  // Merge the four warps through shared memory (the rings are no longer used).
  __syncthreads();
  float *red_acc = reinterpret_cast<float *>(smem);          // [kWarps][G][D]
  float *red_m = red_acc + size_t(kWarps) * G * D;            // [kWarps][G]
  float *red_l = red_m + kWarps * G;                          // [kWarps][G]
  if (tslot == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float4 *dst = reinterpret_cast<float4 *>(red_acc + (size_t(warp) * G + g) * D + d0);
      dst[0] = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
      dst[1] = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
    }
    if (sl % HL == 0) {
      red_m[warp * G + my_head] = m_run;
      red_l[warp * G + my_head] = l_run;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < p.G_cta * D; idx += kWarps * 32) {
    const int g = idx / D, d = idx - g * D;
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * G + g]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float sc = ex2(red_m[w * G + g] - M);
      L = fmaf(sc, red_l[w * G + g], L);
      O = fmaf(sc, red_acc[(size_t(w) * G + g) * D + d], O);
    }
    const bool live = M != neg_inf();
    const int m = g / p.Gm;
    const int row = it.q_index >= 0 ? it.out_row : __ldg(p.member_row_base + m) + it.out_row;
    const int head = kv * p.Gm + (g - m * p.Gm);
    const int64_t o = int64_t(row) * p.Hq_req + head;
    p.v_out[o * p.Dv + d] = live ? O / L * p.v_scale : 0.f;
    if (d == 0) p.lse_out[o] = live ? M + log2f(L) : neg_inf();
  }
}

int ring_tile_tokens(int page_size) {  // gcd(page_size, 8)
  int a = page_size, b = 8;
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

template <int D, int G>
size_t cc_smem_bytes(int sub) {
  const size_t stage = size_t(kWarps) * kStages * 2 * size_t(sub) * D * 2;
  const size_t red = size_t(kWarps) * G * (D + 2) * sizeof(float);
  return std::max(stage, red) + size_t(kWarps) * kStages * sizeof(uint64_t);
}

bool encode_pool_map(CUtensorMap *map, const DeviceInfo &dev, const void *pool, int64_t num_pages,
                     int page_size, int sub, int Hkv, int D) {
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(dev.encode_tiled);
  if (!encode) return false;
  cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(page_size), cuuint64_t(num_pages)};
  cuuint64_t strides[3] = {cuuint64_t(D) * 2, cuuint64_t(Hkv) * D * 2,
                           cuuint64_t(page_size) * Hkv * D * 2};
  cuuint32_t box[4] = {cuuint32_t(D), 1, cuuint32_t(sub), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, int G>
psd_status launch_cc(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  const int sub = ring_tile_tokens(L.page_size);
  CUtensorMap tmK, tmV;
  if (!encode_pool_map(&tmK, dev, L.k_pool, L.num_pages, L.page_size, sub, L.Hkv, D) ||
      !encode_pool_map(&tmV, dev, L.v_pool, L.num_pages, L.page_size, sub, L.Hkv, D))
    return fail(PSD_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");
  CCParams p;
  p.q = reinterpret_cast<const __nv_bfloat16 *>(L.q);
  p.page_indices = L.page_indices;
  p.items = L.items;
  p.order = L.order;
  p.members = L.members;
  p.member_row_base = L.member_row_base;
  p.v_out = L.v_out;
  p.lse_out = L.lse_out;
  p.fault = L.fault;
  p.num_pages = L.num_pages;
  p.Hq_req = L.Hq_req;
  p.Dqk = L.Dqk;
  p.Dv = L.Dv;
  p.page_size = L.page_size;
  p.sub = sub;
  {
    const int tpp = L.page_size / sub;
    p.tpp_log2 = (tpp & (tpp - 1)) == 0 ? __builtin_ctz(unsigned(tpp)) : -1;
  }
  p.Gm = L.Gm;
  p.G_cta = L.G_cta;
  p.q_scale = L.q_scale;
  p.v_scale = L.v_scale;
  p.withhold_from = dev.test_withhold_from >= 0 ? dev.test_withhold_from : 0x7fffffff;
  p.wait_limit = dev.test_wait_limit > 0 ? dev.test_wait_limit : kWaitLimitCycles;
  const size_t smem = cc_smem_bytes<D, G>(sub);
  if (smem > size_t(dev.smem_optin))
    return fail(PSD_ERR_UNSUPPORTED, "page_size %d needs %zu bytes of shared memory", L.page_size, smem);
  auto kern = partial_cc_kernel<D, G>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  }
  dim3 grid(unsigned(L.num_items), unsigned(L.Hkv)), block(kWarps * 32);
  kern<<<grid, block, smem, s>>>(tmK, tmV, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "partial (CUDA cores) launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

template <int D>
psd_status launch_cc_d(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  if (L.G_cta <= 1) return launch_cc<D, 1>(L, dev, s);
  if (L.G_cta <= 2) return launch_cc<D, 2>(L, dev, s);
  if (L.G_cta <= 4) return launch_cc<D, 4>(L, dev, s);
  return launch_cc<D, 8>(L, dev, s);
}

}  // namespace

bool partial_cc_supports(const PartialLaunch &p) {
  return p.kv_dtype == PSD_BF16 && !p.latent_v && p.Dqk == p.Dv &&
         (p.Dqk == 64 || p.Dqk == 128 || p.Dqk == 256) && p.G_cta >= 1 && p.G_cta <= 8;
}

psd_status launch_partial_cc(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  if (L.num_items == 0) return PSD_OK;
  switch (L.Dqk) {
    case 64: return launch_cc_d<64>(L, dev, s);
    case 128: return launch_cc_d<128>(L, dev, s);
    case 256: return launch_cc_d<256>(L, dev, s);
    default: return fail(PSD_ERR_UNSUPPORTED, "CUDA-core partial: head dim %d", L.Dqk);
  }
}

}  // namespace psd
