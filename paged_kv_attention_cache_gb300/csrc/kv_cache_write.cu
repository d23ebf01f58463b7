// KV_CACHE_WRITE: scatter new K/V rows into the paged pool by slot
// ("How serving works in Tlaloc", sections 1-2: slot -1 is padding and is
// never written; the pools are updated in place).
//
// One warp moves one token: the K row and the V row are each H_kv*d elements,
// contiguous in both the source and the pool, so the copy is 16-byte vector
// loads and stores, fully coalesced.  A grid-stride loop over tokens keeps the
// grid a multiple of the SM count.
#include "common.cuh"

namespace tl {

__global__ void __launch_bounds__(256) kv_cache_write_kernel(
    const int4* __restrict__ k_new, const int4* __restrict__ v_new, int4* __restrict__ k_cache,
    int4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int32_t n_tokens,
    int64_t n_slots, int32_t row_vecs, uint32_t* error_word) {
  const int lane = threadIdx.x & 31;
  const int warps_per_cta = blockDim.x >> 5;
  const int64_t first = (int64_t)blockIdx.x * warps_per_cta + (threadIdx.x >> 5);
  const int64_t stride = (int64_t)gridDim.x * warps_per_cta;
  for (int64_t t = first; t < n_tokens; t += stride) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;  // padding
    if (slot < 0 || slot >= n_slots) {
      if (lane == 0) report(error_word, TL_DEVERR_SLOT_RANGE);
      continue;
    }
    const int4* ks = k_new + t * row_vecs;
    const int4* vs = v_new + t * row_vecs;
    int4* kd = k_cache + slot * row_vecs;
    int4* vd = v_cache + slot * row_vecs;
    for (int i = lane; i < row_vecs; i += 32) {
      const int4 a = __ldg(ks + i);
      const int4 b = __ldg(vs + i);
      kd[i] = a;
      vd[i] = b;
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

template <bool SRC_F32>
__global__ void __launch_bounds__(256) kv_cache_write_fp8_kernel(
    const void* __restrict__ k_new, const void* __restrict__ v_new, uint2* __restrict__ k_cache,
    uint2* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int32_t n_tokens,
    int64_t n_slots, int32_t row_8s, uint32_t* error_word) {
  const int lane = threadIdx.x & 31;
  const int warps_per_cta = blockDim.x >> 5;
  const int64_t first = (int64_t)blockIdx.x * warps_per_cta + (threadIdx.x >> 5);
  const int64_t stride = (int64_t)gridDim.x * warps_per_cta;
  for (int64_t t = first; t < n_tokens; t += stride) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;  // padding
    if (slot < 0 || slot >= n_slots) {
      if (lane == 0) report(error_word, TL_DEVERR_SLOT_RANGE);
      continue;
    }
    for (int i = lane; i < row_8s; i += 32) {
      k_cache[slot * row_8s + i] = load_as_e4m3x8<SRC_F32>(k_new, t * row_8s + i);
      v_cache[slot * row_8s + i] = load_as_e4m3x8<SRC_F32>(v_new, t * row_8s + i);
    }
  }
}

}  // namespace tl

extern "C" tl_status tl_kv_cache_write_fp8(const void* k_new, const void* v_new,
                                           tl_dtype src_dtype, void* k_cache, void* v_cache,
                                           const int64_t* slot_mapping, int32_t n_tokens,
                                           int32_t num_pages, int32_t page_size, int32_t h_kv,
                                           int32_t d, uint32_t* error_word, void* stream) {
  using namespace tl;
  if (n_tokens < 0 || num_pages <= 0 || page_size <= 0 || h_kv <= 0 || d <= 0)
    return TL_ERR_INVALID_ARG;
  if (src_dtype != TL_F32 && src_dtype != TL_BF16) return TL_ERR_UNSUPPORTED;
  if (n_tokens == 0) return TL_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return TL_ERR_INVALID_ARG;
  const int64_t row = (int64_t)h_kv * d;  // elements of one token
  if (row % 16 != 0) return TL_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(k_cache) & 7u) ||
      (reinterpret_cast<uintptr_t>(v_cache) & 7u) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return TL_ERR_INVALID_ARG;
  const int threads = 256;
  const int warps = threads / 32;
  int64_t blocks = ((int64_t)n_tokens + warps - 1) / warps;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  const int64_t n_slots = (int64_t)num_pages * page_size;
  if (src_dtype == TL_F32)
    kv_cache_write_fp8_kernel<true><<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        k_new, v_new, (uint2*)k_cache, (uint2*)v_cache, slot_mapping, n_tokens, n_slots,
        (int32_t)(row / 8), error_word);
  else
    kv_cache_write_fp8_kernel<false><<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        k_new, v_new, (uint2*)k_cache, (uint2*)v_cache, slot_mapping, n_tokens, n_slots,
        (int32_t)(row / 8), error_word);
  return launch_status();
}

extern "C" tl_status tl_kv_cache_write(const void* k_new, const void* v_new, void* k_cache,
                                       void* v_cache, const int64_t* slot_mapping,
                                       int32_t n_tokens, int32_t num_pages, int32_t page_size,
                                       int32_t h_kv, int32_t d, tl_dtype dtype,
                                       uint32_t* error_word, void* stream) {
  using namespace tl;
  if (n_tokens < 0 || num_pages <= 0 || page_size <= 0 || h_kv <= 0 || d <= 0)
    return TL_ERR_INVALID_ARG;
  if (dtype != TL_F32 && dtype != TL_BF16) return TL_ERR_UNSUPPORTED;
  if (n_tokens == 0) return TL_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return TL_ERR_INVALID_ARG;
  const int64_t row_bytes = (int64_t)h_kv * d * (dtype == TL_F32 ? 4 : 2);
  if (row_bytes % 16 != 0) return TL_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return TL_ERR_INVALID_ARG;
  const int threads = 256;
  const int warps = threads / 32;
  int64_t blocks = ((int64_t)n_tokens + warps - 1) / warps;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  kv_cache_write_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      (const int4*)k_new, (const int4*)v_new, (int4*)k_cache, (int4*)v_cache, slot_mapping,
      n_tokens, (int64_t)num_pages * page_size, (int32_t)(row_bytes / 16), error_word);
  return launch_status();
}
