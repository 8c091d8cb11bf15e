// RoPE + KV append: the step before paged decode, for the new token of each request
// (ROCm ATOM PR #1701, section 1 and 3.3: one fused kernel ropes every query and the
// new token's rope part of K, concatenates the non-rope latent with it, and writes
// the KV row only for the slots this rank owns; 3.2: fp8 KV stored as codes that
// dequantise as code * scale.  mlxcel PR #1004, Left out / unsure: fused RoPE +
// KV-append decode kernels precede this path).
//
// Arithmetic, fixed so results are reproducible bit for bit: the rotation runs in
// f32 with every product and sum rounded on its own (no contraction into FMAs),
// x' = x c - y s, y' = y c + x s; q and bf16 pools take the round-to-nearest-even
// bf16 of x'; fp8 pools take the saturating round-to-nearest-even E4M3 code of
// x' / scale (the quotient rounded to f32 first).
//
// GB300 shape: one CTA per new token; threads stride over the query rope pairs
// (every head), then over the K row (latent part copied or quantised, rope part
// rotated) and the V row.  The vectorised form moves 8 pairs or 8 columns per thread
// with 16-byte accesses, so a decode token's work is one round of loads; the scalar
// form serves odd widths and unaligned pointers.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device.cuh"
#include "kernels.h"

namespace psd {

namespace {

struct RopeParams {
  __nv_bfloat16 *q;
  const __nv_bfloat16 *k_nope, *k_rope, *v;
  const float *cos_sin;
  const int32_t *positions, *slot_mapping;
  void *k_pool, *v_pool;
  int32_t *fault;
  int64_t num_slots;
  int T, Hq, Dq, q_rope_col, Hkv, Dn, Dr, Dv, rot, neox, max_position, fp8;
  float k_scale, v_scale;
};

__device__ __forceinline__ void rotate(float x, float y, float c, float s, float &xo, float &yo) {
  xo = __fsub_rn(__fmul_rn(x, c), __fmul_rn(y, s));
  yo = __fadd_rn(__fmul_rn(y, c), __fmul_rn(x, s));
}

// Saturating round-to-nearest-even E4M3 code of v (hardware conversion of a pair).
__device__ __forceinline__ uint8_t e4m3_code(float v) {
  uint16_t two;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(0.f), "f"(v));
  return uint8_t(two & 0xFF);
}

__device__ __forceinline__ void store_kv(void *pool, int64_t idx, float v, bool fp8, float scale) {
  if (fp8)
    static_cast<uint8_t *>(pool)[idx] = e4m3_code(__fdiv_rn(v, scale));
  else
    static_cast<__nv_bfloat16 *>(pool)[idx] = __float2bfloat16_rn(v);
}

// First and second element of rope pair i (frequency i) in a rope block of `rot`.
__device__ __forceinline__ void pair_index(int i, int rot, bool neox, int &a, int &b) {
  if (neox) {
    a = i;
    b = i + rot / 2;
  } else {
    a = 2 * i;
    b = 2 * i + 1;
  }
}

__global__ void __launch_bounds__(256) rope_append_kernel(const RopeParams p) {
  const int t = blockIdx.x;
  const int pos = __ldg(p.positions + t);
  if (pos < 0 || pos >= p.max_position) {  // no table row: leave the token untouched
    if (threadIdx.x == 0) atomicOr(p.fault, PSD_FAULT_RANGE);
    return;
  }
  const int half = p.rot / 2;
  const bool neox = p.neox != 0;
  const float *cs = p.cos_sin + int64_t(pos) * p.rot;

  // ---- queries: every head, every token
  const int q_pairs = p.Hq * half;
  for (int j = threadIdx.x; j < q_pairs; j += blockDim.x) {
    const int h = j / half, i = j - h * half;
    int a, b;
    pair_index(i, p.rot, neox, a, b);
    __nv_bfloat16 *row = p.q + (int64_t(t) * p.Hq + h) * p.Dq + p.q_rope_col;
    float xo, yo;
    rotate(__bfloat162float(row[a]), __bfloat162float(row[b]), __ldg(cs + i), __ldg(cs + half + i), xo, yo);
    row[a] = __float2bfloat16_rn(xo);
    row[b] = __float2bfloat16_rn(yo);
  }

  // ---- KV row of the slot this rank owns
  const int slot = __ldg(p.slot_mapping + t);
  if (slot < 0) return;
  if (int64_t(slot) >= p.num_slots) {
    if (threadIdx.x == 0) atomicOr(p.fault, PSD_FAULT_PAGE_ID);
    return;
  }
  const bool fp8 = p.fp8 != 0;
  const int Dk = p.Dn + p.Dr;
  const int64_t k_base = int64_t(slot) * p.Hkv * Dk;
  // latent / non-rope part, then the rope part (rotated pairs; columns past rot copied)
  for (int j = threadIdx.x; j < p.Hkv * p.Dn; j += blockDim.x) {
    const int h = j / p.Dn, d = j - h * p.Dn;
    store_kv(p.k_pool, k_base + int64_t(h) * Dk + d,
             __bfloat162float(p.k_nope[(int64_t(t) * p.Hkv + h) * p.Dn + d]), fp8, p.k_scale);
  }
  const int k_pairs = p.Hkv * half;
  for (int j = threadIdx.x; j < k_pairs; j += blockDim.x) {
    const int h = j / half, i = j - h * half;
    int a, b;
    pair_index(i, p.rot, neox, a, b);
    const __nv_bfloat16 *src = p.k_rope + (int64_t(t) * p.Hkv + h) * p.Dr;
    float xo, yo;
    rotate(__bfloat162float(src[a]), __bfloat162float(src[b]), __ldg(cs + i), __ldg(cs + half + i), xo, yo);
    const int64_t dst = k_base + int64_t(h) * Dk + p.Dn;
    store_kv(p.k_pool, dst + a, xo, fp8, p.k_scale);
    store_kv(p.k_pool, dst + b, yo, fp8, p.k_scale);
  }
  const int tail = p.Dr - p.rot;
  for (int j = threadIdx.x; j < p.Hkv * tail; j += blockDim.x) {
    const int h = j / tail, d = p.rot + (j - h * tail);
    store_kv(p.k_pool, k_base + int64_t(h) * Dk + p.Dn + d,
             __bfloat162float(p.k_rope[(int64_t(t) * p.Hkv + h) * p.Dr + d]), fp8, p.k_scale);
  }
  if (p.v_pool) {
    const int64_t v_base = int64_t(slot) * p.Hkv * p.Dv;
    for (int j = threadIdx.x; j < p.Hkv * p.Dv; j += blockDim.x)
      store_kv(p.v_pool, v_base + j, __bfloat162float(p.v[int64_t(t) * p.Hkv * p.Dv + j]), fp8, p.v_scale);
  }
}

// ------------------------------------------------------------ vectorised form
// Same arithmetic and rounding, 8 pairs or 8 columns per thread with 16-byte loads
// and stores; used when rot_dim % 16 == 0 and every row width and column offset is a
// multiple of 8 elements (the host checks alignment of the base pointers too).
struct F8 {
  float v[8];
};
__device__ __forceinline__ F8 load_bf16x8(const __nv_bfloat16 *p) {
  const uint4 w = *reinterpret_cast<const uint4 *>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
  F8 f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f.v[2 * k] = __uint_as_float(u[k] << 16);
    f.v[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
  }
  return f;
}
__device__ __forceinline__ uint4 pack_bf16x8(const F8 &f) {
  uint32_t u[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(f.v[2 * k]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(f.v[2 * k + 1]));
    u[k] = lo | (hi << 16);
  }
  return make_uint4(u[0], u[1], u[2], u[3]);
}
__device__ __forceinline__ F8 load_f32x8(const float *p) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  F8 f = {{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
  return f;
}
// Stores 8 values at element offset `idx` of a pool: 16 bytes of bf16 or 8 E4M3 codes.
__device__ __forceinline__ void store8(void *pool, int64_t idx, const F8 &f, bool fp8, float scale) {
  if (fp8) {
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k >> 2] |= uint32_t(e4m3_code(__fdiv_rn(f.v[k], scale))) << (8 * (k & 3));
    *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(pool) + idx) = make_uint2(w[0], w[1]);
  } else {
    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(pool) + idx) = pack_bf16x8(f);
  }
}
// Rotates 8 pairs starting at frequency i0 of the rope block at `src`: neox pairs
// (i, i + half) are two runs of 8; interleaved pairs (2i, 2i + 1) are one run of 16.
__device__ __forceinline__ void rotate8(const __nv_bfloat16 *src, int i0, int half, bool neox, const float *cs,
                                        F8 &xo, F8 &yo) {
  const F8 c = load_f32x8(cs + i0), s = load_f32x8(cs + half + i0);
  F8 x, y;
  if (neox) {
    x = load_bf16x8(src + i0);
    y = load_bf16x8(src + half + i0);
  } else {
    const F8 a = load_bf16x8(src + 2 * i0), b = load_bf16x8(src + 2 * i0 + 8);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x.v[k] = a.v[2 * k];
      y.v[k] = a.v[2 * k + 1];
      x.v[4 + k] = b.v[2 * k];
      y.v[4 + k] = b.v[2 * k + 1];
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) rotate(x.v[k], y.v[k], c.v[k], s.v[k], xo.v[k], yo.v[k]);
}
// Writes rotated pairs back in the source layout: two runs of 8 (neox) or one run
// of 16 interleaved values.
template <typename Store>
__device__ __forceinline__ void put_pairs(const F8 &xo, const F8 &yo, int i0, int half, bool neox, Store st) {
  if (neox) {
    st(i0, xo);
    st(half + i0, yo);
  } else {
    F8 a, b;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      a.v[2 * k] = xo.v[k];
      a.v[2 * k + 1] = yo.v[k];
      b.v[2 * k] = xo.v[4 + k];
      b.v[2 * k + 1] = yo.v[4 + k];
    }
    st(2 * i0, a);
    st(2 * i0 + 8, b);
  }
}

__global__ void __launch_bounds__(256) rope_append_vec_kernel(const RopeParams p) {
  const int t = blockIdx.x;
  const int pos = __ldg(p.positions + t);
  const int slot = __ldg(p.slot_mapping + t);
  if (pos < 0 || pos >= p.max_position) {
    if (threadIdx.x == 0) atomicOr(p.fault, PSD_FAULT_RANGE);
    return;
  }
  const int half = p.rot / 2, G = half / 8;  // groups of 8 pairs per head
  const bool neox = p.neox != 0, fp8 = p.fp8 != 0;
  const float *cs = p.cos_sin + int64_t(pos) * p.rot;
  for (int j = threadIdx.x; j < p.Hq * G; j += blockDim.x) {
    const int h = j / G, i0 = 8 * (j - h * G);
    __nv_bfloat16 *row = p.q + (int64_t(t) * p.Hq + h) * p.Dq + p.q_rope_col;
    F8 xo, yo;
    rotate8(row, i0, half, neox, cs, xo, yo);
    put_pairs(xo, yo, i0, half, neox, [&](int col, const F8 &f) {
      *reinterpret_cast<uint4 *>(row + col) = pack_bf16x8(f);
    });
  }
  if (slot < 0) return;
  if (int64_t(slot) >= p.num_slots) {
    if (threadIdx.x == 0) atomicOr(p.fault, PSD_FAULT_PAGE_ID);
    return;
  }
  const int Dk = p.Dn + p.Dr;
  const int64_t k_base = int64_t(slot) * p.Hkv * Dk;
  const int n8 = p.Dn / 8, t8 = (p.Dr - p.rot) / 8;
  for (int j = threadIdx.x; j < p.Hkv * n8; j += blockDim.x) {
    const int h = j / n8, d = 8 * (j - h * n8);
    store8(p.k_pool, k_base + int64_t(h) * Dk + d, load_bf16x8(p.k_nope + (int64_t(t) * p.Hkv + h) * p.Dn + d), fp8,
           p.k_scale);
  }
  for (int j = threadIdx.x; j < p.Hkv * G; j += blockDim.x) {
    const int h = j / G, i0 = 8 * (j - h * G);
    const __nv_bfloat16 *src = p.k_rope + (int64_t(t) * p.Hkv + h) * p.Dr;
    F8 xo, yo;
    rotate8(src, i0, half, neox, cs, xo, yo);
    const int64_t dst = k_base + int64_t(h) * Dk + p.Dn;
    put_pairs(xo, yo, i0, half, neox,
              [&](int col, const F8 &f) { store8(p.k_pool, dst + col, f, fp8, p.k_scale); });
  }
  for (int j = threadIdx.x; j < p.Hkv * t8; j += blockDim.x) {
    const int h = j / t8, d = p.rot + 8 * (j - h * t8);
    store8(p.k_pool, k_base + int64_t(h) * Dk + p.Dn + d,
           load_bf16x8(p.k_rope + (int64_t(t) * p.Hkv + h) * p.Dr + d), fp8, p.k_scale);
  }
  if (p.v_pool) {
    const int64_t v_base = int64_t(slot) * p.Hkv * p.Dv;
    for (int j = threadIdx.x; j < p.Hkv * p.Dv / 8; j += blockDim.x)
      store8(p.v_pool, v_base + 8 * int64_t(j), load_bf16x8(p.v + int64_t(t) * p.Hkv * p.Dv + 8 * j), fp8,
             p.v_scale);
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

psd_status launch_rope_append(const psd_rope_append_args *a, cudaStream_t s) {
  if (a->num_tokens == 0) return PSD_OK;
  RopeParams p;
  p.q = static_cast<__nv_bfloat16 *>(a->q);
  p.k_nope = static_cast<const __nv_bfloat16 *>(a->k_nope);
  p.k_rope = static_cast<const __nv_bfloat16 *>(a->k_rope);
  p.v = static_cast<const __nv_bfloat16 *>(a->v);
  p.cos_sin = a->cos_sin;
  p.positions = a->positions;
  p.slot_mapping = a->slot_mapping;
  p.k_pool = a->k_pool;
  p.v_pool = a->v_pool;
  p.fault = a->fault_dev;
  p.num_slots = a->num_pages * int64_t(a->page_size);
  p.T = a->num_tokens;
  p.Hq = a->Hq;
  p.Dq = a->Dq;
  p.q_rope_col = a->q_rope_col;
  p.Hkv = a->Hkv;
  p.Dn = a->Dk_nope;
  p.Dr = a->Dk_rope;
  p.Dv = a->Dv;
  p.rot = a->rot_dim;
  p.neox = a->neox;
  p.max_position = a->max_position;
  p.fp8 = a->kv_dtype == PSD_FP8_E4M3;
  p.k_scale = a->k_scale;
  p.v_scale = a->v_scale;
  const bool vec = a->rot_dim % 16 == 0 && a->q_rope_col % 8 == 0 && a->Dq % 8 == 0 && a->Dk_nope % 8 == 0 &&
                   a->Dk_rope % 8 == 0 && a->Dv % 8 == 0 && aligned16(a->q) && aligned16(a->k_nope) &&
                   aligned16(a->k_rope) && aligned16(a->v) && aligned16(a->cos_sin) && aligned16(a->k_pool) &&
                   aligned16(a->v_pool);
  if (vec)
    rope_append_vec_kernel<<<a->num_tokens, 256, 0, s>>>(p);
  else
    rope_append_kernel<<<a->num_tokens, 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "rope_append launch: %s", cudaGetErrorString(e));
  return PSD_OK;
}

}  // namespace psd
