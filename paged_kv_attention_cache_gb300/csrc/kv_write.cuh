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
