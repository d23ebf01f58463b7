// KV_CACHE_WRITE: scatter new K/V rows into the paged pool by slot
// ("How serving works in Tlaloc", sections 1-2: slot -1 is padding and is
// never written; the pools are updated in place).
//
// The K row and the V row of a token are each H_kv*d elements, contiguous in
// both the source and the pool, so the copy is 16-byte vector loads and
// stores, fully coalesced.  For rows of 32 * 1, 2, 4 or 8 vectors a warp takes
// kWriteTpw tokens and issues every load of their rows before any store (the
// copy is bound by how many bytes are in flight, not by instructions); other
// row sizes take a generic loop, one token per warp.  Measured on the 16K-row
// prefill chunk (80 MB): 14.7 us per write back to back; 1, 2 or 4 tokens per
// warp, and persistent forms (each warp walking a range with the next slots
// prefetched, or each row moved by bulk copies through shared memory, one
// token per lane in flight) were no faster or slower (15.0-21.3 us).
#include <algorithm>

#include "kv_write.cuh"

namespace tl {

constexpr int kWriteTpw = 2;  // tokens per warp of the vectorised write


template <int VPL>
__global__ void __launch_bounds__(256) kv_cache_write_vec_kernel(
    const int4* __restrict__ k_new, const int4* __restrict__ v_new, int4* __restrict__ k_cache,
    int4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int32_t n_tokens,
    int64_t n_slots, uint32_t* error_word) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5) * kWriteTpw;
  for (int64_t t0 = warp * kWriteTpw; t0 < n_tokens; t0 += stride)
    write_tokens_vec<VPL, kWriteTpw>(k_new, v_new, k_cache, v_cache, slot_mapping, t0, n_tokens,
                                     n_slots, lane, error_word);
}

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
    write_token_rows(k_new + t * row_vecs, v_new + t * row_vecs, k_cache + slot * row_vecs,
                     v_cache + slot * row_vecs, row_vecs, lane);
  }
}

template <bool SRC_F32, int UPL>
__global__ void __launch_bounds__(256) kv_cache_write_fp8_vec_kernel(
    const void* __restrict__ k_new, const void* __restrict__ v_new, uint2* __restrict__ k_cache,
    uint2* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int32_t n_tokens,
    int64_t n_slots, uint32_t* error_word) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5) * kWriteTpw;
  for (int64_t t0 = warp * kWriteTpw; t0 < n_tokens; t0 += stride)
    write_tokens_e4m3_vec<SRC_F32, UPL, kWriteTpw>(k_new, v_new, k_cache, v_cache, slot_mapping,
                                                   t0, n_tokens, n_slots, lane, error_word);
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
    write_token_rows_e4m3<SRC_F32>(k_new, v_new, k_cache, v_cache, t, slot, row_8s, lane);
  }
}

// One warp per (token, KV head): its K row and its V row.  Codes at the pool
// layout [num_pages][page_size][H_kv][d], scales at [num_pages][H_kv][page_size].
template <bool SRC_F32>
__global__ void __launch_bounds__(256) kv_cache_write_int8_kernel(
    const void* __restrict__ k_new, const void* __restrict__ v_new, int8_t* __restrict__ k_codes,
    int8_t* __restrict__ v_codes, float* __restrict__ k_scales, float* __restrict__ v_scales,
    const int64_t* __restrict__ slot_mapping, int32_t n_tokens, int32_t page_size, int32_t h_kv,
    int32_t d, int64_t n_slots, uint32_t* error_word) {
  const int lane = threadIdx.x & 31;
  const int warps_per_cta = blockDim.x >> 5;
  const int64_t first = (int64_t)blockIdx.x * warps_per_cta + (threadIdx.x >> 5);
  const int64_t stride = (int64_t)gridDim.x * warps_per_cta;
  const int64_t rows = (int64_t)n_tokens * h_kv;
  for (int64_t r = first; r < rows; r += stride) {
    const int64_t t = r / h_kv;
    const int g = (int)(r % h_kv);
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;  // padding
    if (slot < 0 || slot >= n_slots) {
      if (lane == 0 && g == 0) report(error_word, TL_DEVERR_SLOT_RANGE);
      continue;
    }
    if (d == 128)
      write_head_rows_int8_d128<SRC_F32>(k_new, v_new, k_codes, v_codes, k_scales, v_scales, t, g,
                                         slot, page_size, h_kv, lane, error_word);
    else
      write_head_rows_int8<SRC_F32>(k_new, v_new, k_codes, v_codes, k_scales, v_scales, t, g,
                                    slot, page_size, h_kv, d, lane, error_word);
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
  const int64_t n_slots = (int64_t)num_pages * page_size;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t units = row / 8;  // 8-element units per row
  if (units % 32 == 0 && (units / 32 == 1 || units / 32 == 2 || units / 32 == 4)) {
    const int64_t vb = std::min<int64_t>(
        ((int64_t)n_tokens + warps * kWriteTpw - 1) / (warps * kWriteTpw), (int64_t)num_sms() * 16);
    const dim3 grid((unsigned)vb);
    uint2* kc = (uint2*)k_cache;
    uint2* vc = (uint2*)v_cache;
#define TL_FP8_VEC(F32, U)                                                                     \
  kv_cache_write_fp8_vec_kernel<F32, U><<<grid, threads, 0, st>>>(k_new, v_new, kc, vc,         \
                                                                  slot_mapping, n_tokens,       \
                                                                  n_slots, error_word)
    if (src_dtype == TL_F32) {
      if (units == 32) TL_FP8_VEC(true, 1);
      else if (units == 64) TL_FP8_VEC(true, 2);
      else TL_FP8_VEC(true, 4);
    } else {
      if (units == 32) TL_FP8_VEC(false, 1);
      else if (units == 64) TL_FP8_VEC(false, 2);
      else TL_FP8_VEC(false, 4);
    }
#undef TL_FP8_VEC
    return launch_status();
  }
  int64_t blocks = ((int64_t)n_tokens + warps - 1) / warps;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
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
  const int64_t n_slots = (int64_t)num_pages * page_size;
  const int64_t row_vecs = row_bytes / 16;
  if (row_vecs % 32 == 0 && row_vecs <= 32 * 8) {
    // one wave of warps covers the call (grid-stride beyond 16 CTAs per SM)
    int64_t blocks = ((int64_t)n_tokens + warps * kWriteTpw - 1) / (warps * kWriteTpw);
    blocks = std::min<int64_t>(blocks, (int64_t)num_sms() * 16);
    const dim3 grid((unsigned)blocks);
    cudaStream_t st = (cudaStream_t)stream;
    auto a = (const int4*)k_new;
    auto b = (const int4*)v_new;
    auto c = (int4*)k_cache;
    auto d4 = (int4*)v_cache;
    switch (row_vecs / 32) {
      case 1: kv_cache_write_vec_kernel<1><<<grid, threads, 0, st>>>(a, b, c, d4, slot_mapping, n_tokens, n_slots, error_word); break;
      case 2: kv_cache_write_vec_kernel<2><<<grid, threads, 0, st>>>(a, b, c, d4, slot_mapping, n_tokens, n_slots, error_word); break;
      case 4: kv_cache_write_vec_kernel<4><<<grid, threads, 0, st>>>(a, b, c, d4, slot_mapping, n_tokens, n_slots, error_word); break;
      case 8: kv_cache_write_vec_kernel<8><<<grid, threads, 0, st>>>(a, b, c, d4, slot_mapping, n_tokens, n_slots, error_word); break;
      default: goto generic;
    }
    return launch_status();
  }
generic:
  {
    int64_t blocks = ((int64_t)n_tokens + warps - 1) / warps;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    kv_cache_write_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        (const int4*)k_new, (const int4*)v_new, (int4*)k_cache, (int4*)v_cache, slot_mapping,
        n_tokens, n_slots, (int32_t)row_vecs, error_word);
  }
  return launch_status();
}

extern "C" tl_status tl_kv_cache_write_int8(const void* k_new, const void* v_new,
                                            tl_dtype src_dtype, int8_t* k_codes, int8_t* v_codes,
                                            float* k_scales, float* v_scales,
                                            const int64_t* slot_mapping, int32_t n_tokens,
                                            int32_t num_pages, int32_t page_size, int32_t h_kv,
                                            int32_t d, uint32_t* error_word, void* stream) {
  using namespace tl;
  if (n_tokens < 0 || num_pages <= 0 || page_size <= 0 || h_kv <= 0 || d <= 0)
    return TL_ERR_INVALID_ARG;
  if (src_dtype != TL_F32 && src_dtype != TL_BF16) return TL_ERR_UNSUPPORTED;
  if (d > 1024) return TL_ERR_UNSUPPORTED;
  if (n_tokens == 0) return TL_OK;
  if (!k_new || !v_new || !k_codes || !v_codes || !k_scales || !v_scales || !slot_mapping)
    return TL_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(k_scales) & 3u) ||
      (reinterpret_cast<uintptr_t>(v_scales) & 3u) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return TL_ERR_INVALID_ARG;
  const int threads = 256;
  const int warps = threads / 32;
  int64_t blocks = ((int64_t)n_tokens * h_kv + warps - 1) / warps;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  const int64_t n_slots = (int64_t)num_pages * page_size;
  if (src_dtype == TL_F32)
    kv_cache_write_int8_kernel<true><<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        k_new, v_new, k_codes, v_codes, k_scales, v_scales, slot_mapping, n_tokens, page_size,
        h_kv, d, n_slots, error_word);
  else
    kv_cache_write_int8_kernel<false><<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        k_new, v_new, k_codes, v_codes, k_scales, v_scales, slot_mapping, n_tokens, page_size,
        h_kv, d, n_slots, error_word);
  return launch_status();
}
