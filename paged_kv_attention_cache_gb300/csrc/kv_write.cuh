// KV_CACHE_WRITE, the per-token part shared by the write kernels and the
// decode call that writes its new rows itself ("How serving works in
// Tlaloc", sections 1-2: slot -1 is padding and is never written; the pools
// are updated in place).  One warp moves one token: its K row and V row are
// each H_kv*d elements, contiguous in the source and in the pool.
#pragma once

#include "common.cuh"

namespace tl {

// A token's K and V rows as 16-byte vectors (16-bit or f32 pools: a copy).
__device__ __forceinline__ void write_token_rows(const int4* __restrict__ ks,
                                                 const int4* __restrict__ vs,
                                                 int4* __restrict__ kd, int4* __restrict__ vd,
                                                 int row_vecs, int lane) {
  for (int i = lane; i < row_vecs; i += 32) {
    const int4 a = __ldg(ks + i);
    const int4 b = __ldg(vs + i);
    kd[i] = a;
    vd[i] = b;
  }
}

// The K and V rows of TPW consecutive tokens t0 .. t0 + TPW - 1 (those below
// n_tokens) by one warp, rows of exactly 32 * VPL 16-byte vectors: the slots
// first, then every load of the live tokens' rows (2 * TPW * VPL vectors per
// lane in flight), then the stores.  Slot -1 is padding; a slot outside
// [0, n_slots) is reported and its token skipped.
template <int VPL, int TPW>
__device__ __forceinline__ void write_tokens_vec(const int4* __restrict__ k_new,
                                                 const int4* __restrict__ v_new,
                                                 int4* __restrict__ k_cache,
                                                 int4* __restrict__ v_cache,
                                                 const int64_t* __restrict__ slot_mapping,
                                                 int64_t t0, int64_t n_tokens, int64_t n_slots,
                                                 int lane, uint32_t* error_word) {
  constexpr int RV = 32 * VPL;  // vectors per row
  int64_t slot[TPW];
#pragma unroll
  for (int j = 0; j < TPW; ++j) slot[j] = t0 + j < n_tokens ? __ldg(slot_mapping + t0 + j) : -1;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < TPW; ++j) {
    if (slot[j] != -1 && (slot[j] < 0 || slot[j] >= n_slots)) {
      bad = true;
      slot[j] = -1;
    }
  }
  if (bad && lane == 0) report(error_word, TL_DEVERR_SLOT_RANGE);
  int4 kx[TPW][VPL], vx[TPW][VPL];
#pragma unroll
  for (int j = 0; j < TPW; ++j)
    if (slot[j] >= 0) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        kx[j][v] = __ldg(k_new + (t0 + j) * RV + lane + 32 * v);
        vx[j][v] = __ldg(v_new + (t0 + j) * RV + lane + 32 * v);
      }
    }
#pragma unroll
  for (int j = 0; j < TPW; ++j)
    if (slot[j] >= 0) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        k_cache[slot[j] * RV + lane + 32 * v] = kx[j][v];
        v_cache[slot[j] * RV + lane + 32 * v] = vx[j][v];
      }
    }
}

// The fp8 write: each lane converts 8 elements at a time (one 16-byte bf16
// vector or two f32 vectors) to e4m3fn codes, nearest with ties to even and
// clamped to +-448 by the satfinite conversion; NaN gives the NaN code 0x7F.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(hi) : "f"(d), "f"(c));
  uint32_t r = (uint32_t)lo | ((uint32_t)hi << 16);
  // one NaN code whatever the input's sign and payload
  if (a != a) r = (r & 0xffffff00u) | 0x7Fu;
  if (b != b) r = (r & 0xffff00ffu) | 0x7F00u;
  if (c != c) r = (r & 0xff00ffffu) | 0x7F0000u;
  if (d != d) r = (r & 0x00ffffffu) | 0x7F000000u;
  return r;
}

template <bool SRC_F32>
__device__ __forceinline__ uint2 load_as_e4m3x8(const void* src, int64_t i8) {
  float f[8];
  if (SRC_F32) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(src) + 2 * i8);
    const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 2 * i8 + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(src) + i8);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  return make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
}

// Eight elements (one 16-byte bf16 vector, or two f32 vectors in x[0], x[1])
// as e4m3 codes.
template <bool SRC_F32>
__device__ __forceinline__ uint2 e4m3x8_of(const uint4* x) {
  float f[8];
  if (SRC_F32) {
    const uint32_t w[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
#pragma unroll
    for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(w[k]);
  } else {
    const uint32_t w[4] = {x[0].x, x[0].y, x[0].z, x[0].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  return make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
}

// The fp8 write of TPW consecutive tokens by one warp, rows of exactly
// 32 * UPL units of 8 elements: the slots, then every load of the live
// tokens' rows, then the conversions and the stores (as write_tokens_vec).
template <bool SRC_F32, int UPL, int TPW>
__device__ __forceinline__ void write_tokens_e4m3_vec(const void* k_new, const void* v_new,
                                                      uint2* __restrict__ k_cache,
                                                      uint2* __restrict__ v_cache,
                                                      const int64_t* __restrict__ slot_mapping,
                                                      int64_t t0, int64_t n_tokens,
                                                      int64_t n_slots, int lane,
                                                      uint32_t* error_word) {
  constexpr int RU = 32 * UPL;        // units per row
  constexpr int W = SRC_F32 ? 2 : 1;  // 16-byte loads per unit
  const uint4* ks = static_cast<const uint4*>(k_new);
  const uint4* vs = static_cast<const uint4*>(v_new);
  int64_t slot[TPW];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < TPW; ++j) {
    slot[j] = t0 + j < n_tokens ? __ldg(slot_mapping + t0 + j) : -1;
    if (slot[j] != -1 && (slot[j] < 0 || slot[j] >= n_slots)) {
      bad = true;
      slot[j] = -1;
    }
  }
  if (bad && lane == 0) report(error_word, TL_DEVERR_SLOT_RANGE);
  uint4 kx[TPW][UPL][W], vx[TPW][UPL][W];
#pragma unroll
  for (int j = 0; j < TPW; ++j)
    if (slot[j] >= 0) {
#pragma unroll
      for (int u = 0; u < UPL; ++u)
#pragma unroll
        for (int w = 0; w < W; ++w) {
          kx[j][u][w] = __ldg(ks + ((t0 + j) * RU + lane + 32 * u) * W + w);
          vx[j][u][w] = __ldg(vs + ((t0 + j) * RU + lane + 32 * u) * W + w);
        }
    }
#pragma unroll
  for (int j = 0; j < TPW; ++j)
    if (slot[j] >= 0) {
#pragma unroll
      for (int u = 0; u < UPL; ++u) {
        k_cache[slot[j] * RU + lane + 32 * u] = e4m3x8_of<SRC_F32>(kx[j][u]);
        v_cache[slot[j] * RU + lane + 32 * u] = e4m3x8_of<SRC_F32>(vx[j][u]);
      }
    }
}

// A token's K and V rows converted to e4m3 codes, 8 elements per lane step.
template <bool SRC_F32>
__device__ __forceinline__ void write_token_rows_e4m3(const void* k_new, const void* v_new,
                                                      uint2* __restrict__ k_cache,
                                                      uint2* __restrict__ v_cache, int64_t t,
                                                      int64_t slot, int row_8s, int lane) {
  for (int i = lane; i < row_8s; i += 32) {
    k_cache[slot * row_8s + i] = load_as_e4m3x8<SRC_F32>(k_new, t * row_8s + i);
    v_cache[slot * row_8s + i] = load_as_e4m3x8<SRC_F32>(v_new, t * row_8s + i);
  }
}

// int8 pools: one (token, KV head) row of d new values as int8 codes and its
// f32 scale, by one warp.  The format is read from the int8 weight
// quantisation of "How serving works in Tlaloc" ("Int8 weights (opt-in)":
// one scale per channel, max |x| / 127, codes rounded half to even), with
// the row as the channel: s = m / 127 over the row's finite values, code =
// rint(x / s) clamped to +-127, both IEEE binary32 divisions.  A row whose s
// is 0 gets codes 0; a non-finite value gets code 0 and is reported.
template <bool SRC_F32>
__device__ __forceinline__ float new_value(const void* src, int64_t i) {
  if (SRC_F32) return __ldg(static_cast<const float*>(src) + i);
  return __uint_as_float((uint32_t)__ldg(static_cast<const unsigned short*>(src) + i) << 16);
}

template <bool SRC_F32>
__device__ void quantize_row_int8(const void* src, int64_t base, int d, int8_t* codes,
                                  float* scale, int lane, uint32_t* error_word) {
  float m = 0.f;
  bool bad = false;
  for (int e = lane; e < d; e += 32) {
    const float x = new_value<SRC_F32>(src, base + e);
    if (isfinite(x))
      m = fmaxf(m, fabsf(x));
    else
      bad = true;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float sc = __fdiv_rn(m, 127.f);
  for (int e = lane; e < d; e += 32) {
    const float x = new_value<SRC_F32>(src, base + e);
    float r = 0.f;
    if (isfinite(x) && sc > 0.f) r = fminf(fmaxf(rintf(__fdiv_rn(x, sc)), -127.f), 127.f);
    codes[e] = (int8_t)__float2int_rn(r);
  }
  if (lane == 0) *scale = sc;
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(error_word, TL_DEVERR_VALUE_RANGE);
}

// d = 128: the K and V rows of token t, KV head g into int8 pools by one
// warp, lane l owning elements 4l .. 4l + 3 (one 8- or 16-byte load per row,
// both rows loaded before either is quantised; the values stay in registers
// for both passes).  The same arithmetic as quantize_row_int8.
template <bool SRC_F32>
__device__ __forceinline__ void load4(const void* src, int64_t i4, float* x) {
  if (SRC_F32) {
    const float4 a = __ldg(static_cast<const float4*>(src) + i4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  } else {
    const uint2 a = __ldg(static_cast<const uint2*>(src) + i4);
    x[0] = __uint_as_float(a.x << 16);
    x[1] = __uint_as_float(a.x & 0xffff0000u);
    x[2] = __uint_as_float(a.y << 16);
    x[3] = __uint_as_float(a.y & 0xffff0000u);
  }
}
__device__ __forceinline__ void quantize4_int8(const float* x, int8_t* codes, float* scale,
                                               int lane, uint32_t* error_word) {
  float m = 0.f;
  bool bad = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (isfinite(x[k]))
      m = fmaxf(m, fabsf(x[k]));
    else
      bad = true;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float sc = __fdiv_rn(m, 127.f);
  uint32_t packed = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float r = 0.f;
    if (isfinite(x[k]) && sc > 0.f) r = fminf(fmaxf(rintf(__fdiv_rn(x[k], sc)), -127.f), 127.f);
    packed |= (uint32_t)(uint8_t)(int8_t)__float2int_rn(r) << (8 * k);
  }
  reinterpret_cast<uint32_t*>(codes)[lane] = packed;
  if (lane == 0) *scale = sc;
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(error_word, TL_DEVERR_VALUE_RANGE);
}
template <bool SRC_F32>
__device__ __forceinline__ void write_head_rows_int8_d128(const void* k_new, const void* v_new,
                                                          int8_t* k_codes, int8_t* v_codes,
                                                          float* k_scales, float* v_scales,
                                                          int64_t t, int g, int64_t slot,
                                                          int page_size, int h_kv, int lane,
                                                          uint32_t* error_word) {
  const int64_t page = slot / page_size, off = slot % page_size;
  const int64_t src4 = (t * h_kv + g) * 32 + lane;  // 4-element group of this lane
  const int64_t dst = (slot * h_kv + g) * 128, si = (page * h_kv + g) * page_size + off;
  float kx[4], vx[4];
  load4<SRC_F32>(k_new, src4, kx);
  load4<SRC_F32>(v_new, src4, vx);
  quantize4_int8(kx, k_codes + dst, k_scales + si, lane, error_word);
  quantize4_int8(vx, v_codes + dst, v_scales + si, lane, error_word);
}

// The K and V rows of token t, KV head g into int8 pools, by one warp: codes
// at the pool layout, scales at [num_pages][H_kv][page_size].
template <bool SRC_F32>
__device__ __forceinline__ void write_head_rows_int8(const void* k_new, const void* v_new,
                                                     int8_t* k_codes, int8_t* v_codes,
                                                     float* k_scales, float* v_scales, int64_t t,
                                                     int g, int64_t slot, int page_size, int h_kv,
                                                     int d, int lane, uint32_t* error_word) {
  const int64_t page = slot / page_size, off = slot % page_size;
  const int64_t src = (t * h_kv + g) * d, dst = (slot * h_kv + g) * d;
  const int64_t si = (page * h_kv + g) * page_size + off;
  quantize_row_int8<SRC_F32>(k_new, src, d, k_codes + dst, k_scales + si, lane, error_word);
  quantize_row_int8<SRC_F32>(v_new, src, d, v_codes + dst, v_scales + si, lane, error_word);
}

}  // namespace tl
