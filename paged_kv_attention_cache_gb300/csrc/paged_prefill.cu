// PAGED_ATTENTION, batched right-aligned prefill, folded over key tiles with
// an online softmax ("How serving works in Tlaloc", section 1: right-aligned
// rows, padding at slot -1, causal length = position + 1; section 2: a row's
// pages are gathered once for all its tokens, and "Blockwise attention": the
// keys are folded block by block into a running max, sum and P.V, so no score
// tensor wider than one tile exists).
//
// Grid: (query tile of 64 tokens, query head, row).  Each CTA reads only the
// key range its live tokens can see ([min lo, max p]), in tiles of 64 keys
// gathered from the row's pages with 16-byte cp.async into a 2-stage shared
// memory ring; Q.K^T and P.V run on mma.sync m16n8k16 (bf16 in, f32
// accumulate), the online softmax in registers.  A CTA never touches another
// row, and its arithmetic does not depend on B, so a row gives the same bits
// batched or alone.
#include "common.cuh"

namespace tl {

constexpr int kPfRows = 64;     // query tokens per CTA
constexpr int kPfKeys = 64;     // keys per tile
constexpr int kPfWarps = 4;
constexpr int kPfThreads = kPfWarps * 32;

struct PrefillParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int32_t* block_table;
  const int32_t* positions;
  float* out;
  int32_t max_pages_per_seq;
  int32_t B, T, h_q, h_kv, group;
  int32_t num_pages, page_size, window;
  float scale_log2;
  uint32_t* error_word;
};

template <int D>
struct PfSmem {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kQBytes = kPfRows * kRowBytes;
  static constexpr int kTileBytes = kPfKeys * kRowBytes;  // K or V
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kTotal = kQBytes + 2 * kStageBytes;
};

__device__ __forceinline__ uint32_t swz(int row, int unit, int row_bytes) {
  return (uint32_t)(row * row_bytes + ((unit ^ (row & 7)) << 4));
}

// Gather one tile of keys [j0, j0+64) of row b, KV head g: rows past
// j_last (or on a bad page) are zero-filled.
template <int D>
__device__ __forceinline__ void load_kv_tile(const PrefillParams& P, int b, int g, int j0,
                                             int j_last, uint32_t kdst, uint32_t vdst) {
  constexpr int U = D / 8;  // 16-byte units per row
  const int tid = threadIdx.x;
  for (int r = tid >> 1; r < kPfKeys; r += kPfThreads / 2) {
    const int j = j0 + r;
    bool live = j <= j_last;
    int64_t page = 0;
    if (live) {
      page = __ldg(P.block_table + (size_t)b * P.max_pages_per_seq + j / P.page_size);
      if (page < 0 || page >= P.num_pages) {
        report(P.error_word, TL_DEVERR_PAGE_RANGE);
        live = false;
        page = 0;
      }
    }
    const size_t row =
        (((size_t)page * P.page_size + (live ? j % P.page_size : 0)) * P.h_kv + g) * D;
    const __nv_bfloat16* ks = P.k_cache + row;
    const __nv_bfloat16* vs = P.v_cache + row;
    const uint32_t n = live ? 16u : 0u;
#pragma unroll
    for (int i = 0; i < U / 2; ++i) {
      const int u = (tid & 1) + 2 * i;
      cp_async_16(kdst + swz(r, u, D * 2), ks + u * 8, n);
      cp_async_16(vdst + swz(r, u, D * 2), vs + u * 8, n);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 2) prefill_mma_kernel(PrefillParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_range[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_qt = (P.T + kPfRows - 1) / kPfRows;
  const int qt = n_qt - 1 - (int)blockIdx.x;  // heaviest (latest) tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / P.group;
  const int t0 = qt * kPfRows;
  const int32_t* pos_row = P.positions + (size_t)b * P.T;
  const int64_t cap = (int64_t)P.max_pages_per_seq * P.page_size;

  // key range of the tile's live tokens
  if (tid == 0) {
    s_range[0] = INT32_MAX;
    s_range[1] = -1;
  }
  __syncthreads();
  if (tid < kPfRows && t0 + tid < P.T) {
    int p = pos_row[t0 + tid];
    if (p >= cap) {
      report(P.error_word, TL_DEVERR_CONTEXT_RANGE);
      p = -1;
    }
    if (p >= 0) {
      const int lo = (P.window > 0 && p - P.window + 1 > 0) ? p - P.window + 1 : 0;
      atomicMin(&s_range[0], lo);
      atomicMax(&s_range[1], p);
    }
  }
  __syncthreads();
  const int kmin = s_range[0], kmax = s_range[1];

  const int qr = lane >> 2, qc = (lane & 3) * 2;
  // this thread's two rows (tokens) and their causal ranges
  const int tA = t0 + warp * 16 + qr, tB = tA + 8;
  int pA = tA < P.T ? pos_row[tA] : -1, pB = tB < P.T ? pos_row[tB] : -1;
  if (pA >= cap) pA = -1;
  if (pB >= cap) pB = -1;
  const int loA = (P.window > 0 && pA - P.window + 1 > 0) ? pA - P.window + 1 : 0;
  const int loB = (P.window > 0 && pB - P.window + 1 > 0) ? pB - P.window + 1 : 0;

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

  if (kmax >= 0) {
    const uint32_t sbase = smem_u32(smem);
    const uint32_t qaddr = sbase;
    const uint32_t stage0 = sbase + PfSmem<D>::kQBytes;
    // Q tile (rows past T, or padding, load whatever is there: their output is 0)
    {
      constexpr int U = D / 8;
      for (int r = tid >> 1; r < kPfRows; r += kPfThreads / 2) {
        const int t = min(t0 + r, P.T - 1);
        const __nv_bfloat16* src = P.q + (((size_t)b * P.T + t) * P.h_q + h) * D;
#pragma unroll
        for (int i = 0; i < U / 2; ++i) {
          const int u = (tid & 1) + 2 * i;
          cp_async_16(qaddr + swz(r, u, D * 2), src + u * 8, 16u);
        }
      }
    }
    const int tile_first = kmin / kPfKeys, tile_last = kmax / kPfKeys;
    load_kv_tile<D>(P, b, g, tile_first * kPfKeys, kmax, stage0,
                    stage0 + PfSmem<D>::kTileBytes);
    cp_async_commit();

    uint32_t qa[D / 16][4];
    for (int kt = tile_first; kt <= tile_last; ++kt) {
      const int st = (kt - tile_first) & 1;
      if (kt < tile_last) {
        const uint32_t nst = stage0 + (st ^ 1) * PfSmem<D>::kStageBytes;
        load_kv_tile<D>(P, b, g, (kt + 1) * kPfKeys, kmax, nst, nst + PfSmem<D>::kTileBytes);
      }
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      if (kt == tile_first) {
        const int mi = lane >> 3, ri = lane & 7;
        const int row = warp * 16 + (mi & 1) * 8 + ri;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ldmatrix_x4(qaddr + swz(row, 2 * ks + (mi >> 1), D * 2), qa[ks][0], qa[ks][1],
                      qa[ks][2], qa[ks][3]);
      }
      const uint32_t kaddr = stage0 + st * PfSmem<D>::kStageBytes;
      const uint32_t vaddr = kaddr + PfSmem<D>::kTileBytes;
      const int j0 = kt * kPfKeys;
      // S = Q K^T (16 x 64 per warp)
      float s[kPfKeys / 8][4];
#pragma unroll
      for (int n = 0; n < kPfKeys / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      {
        const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
        for (int n2 = 0; n2 < kPfKeys / 16; ++n2) {
          const int key = n2 * 16 + (mi >> 1) * 8 + ri;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(kaddr + swz(key, 2 * ks + (mi & 1), D * 2), b0, b1, b2, b3);
            mma_bf16_16816(s[2 * n2], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
            mma_bf16_16816(s[2 * n2 + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
          }
        }
      }
      // mask, scale, online softmax
      float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
      for (int n = 0; n < kPfKeys / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + n * 8 + qc + e;
          s[n][e] = (j >= loA && j <= pA) ? s[n][e] * P.scale_log2 : -INFINITY;
          s[n][2 + e] = (j >= loB && j <= pB) ? s[n][2 + e] * P.scale_log2 : -INFINITY;
          mxA = fmaxf(mxA, s[n][e]);
          mxB = fmaxf(mxB, s[n][2 + e]);
        }
      }
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
      const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
      const float baseA = nA == -INFINITY ? 0.f : nA;  // a row with no live key yet
      const float baseB = nB == -INFINITY ? 0.f : nB;
      const float cA = fast_exp2(mA - baseA), cB = fast_exp2(mB - baseB);
      mA = nA;
      mB = nB;
      float sumA = 0.f, sumB = 0.f;
#pragma unroll
      for (int n = 0; n < kPfKeys / 8; ++n) {
        s[n][0] = fast_exp2(s[n][0] - baseA);
        s[n][1] = fast_exp2(s[n][1] - baseA);
        s[n][2] = fast_exp2(s[n][2] - baseB);
        s[n][3] = fast_exp2(s[n][3] - baseB);
        sumA += s[n][0] + s[n][1];
        sumB += s[n][2] + s[n][3];
      }
      lA = lA * cA + sumA;
      lB = lB * cB + sumB;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= cA;
        o[n][1] *= cA;
        o[n][2] *= cB;
        o[n][3] *= cB;
      }
      // O += P V
      {
        const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
        for (int kk = 0; kk < kPfKeys / 16; ++kk) {
          // P = hi + lo (bf16 pair): two MMAs keep f32-level accuracy
          uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
          split_bf16x2(s[2 * kk][0], s[2 * kk][1], h0, l0);
          split_bf16x2(s[2 * kk][2], s[2 * kk][3], h1, l1);
          split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], h2, l2);
          split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], h3, l3);
          const int key = kk * 16 + (mi & 1) * 8 + ri;
#pragma unroll
          for (int nd2 = 0; nd2 < D / 16; ++nd2) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(vaddr + swz(key, 2 * nd2 + (mi >> 1), D * 2), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * nd2], h0, h1, h2, h3, b0, b1);
            mma_bf16_16816(o[2 * nd2], l0, l1, l2, l3, b0, b1);
            mma_bf16_16816(o[2 * nd2 + 1], h0, h1, h2, h3, b2, b3);
            mma_bf16_16816(o[2 * nd2 + 1], l0, l1, l2, l3, b2, b3);
          }
        }
      }
      __syncthreads();  // the stage is rewritten by the next iteration's loads
    }
    cp_async_wait<0>();
  }
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  const float invA = (pA >= 0 && lA > 0.f) ? 1.f / lA : 0.f;
  const float invB = (pB >= 0 && lB > 0.f) ? 1.f / lB : 0.f;
  if (tA < P.T) {
    float* dst = P.out + (((size_t)b * P.T + tA) * P.h_q + h) * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<float2*>(dst + n * 8 + qc) = make_float2(o[n][0] * invA, o[n][1] * invA);
  }
  if (tB < P.T) {
    float* dst = P.out + (((size_t)b * P.T + tB) * P.h_q + h) * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<float2*>(dst + n * 8 + qc) = make_float2(o[n][2] * invB, o[n][3] * invB);
  }
}

}  // namespace tl

extern "C" size_t tl_paged_attn_prefill_workspace_size(int32_t B, int32_t T, int32_t h_q,
                                                       int32_t h_kv, int32_t d) {
  if (B <= 0 || T <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || h_q % h_kv) return 0;
  return 256;
}

extern "C" tl_status tl_paged_attn_prefill(const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_table,
                                           int32_t max_pages_per_seq, const int32_t* positions,
                                           float* out, int32_t B, int32_t T, int32_t h_q,
                                           int32_t h_kv, int32_t d, int32_t num_pages,
                                           int32_t page_size, int32_t window, float scale,
                                           tl_dtype dtype, void* workspace,
                                           size_t workspace_bytes, uint32_t* error_word,
                                           void* stream) {
  using namespace tl;
  if (B <= 0 || T <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || num_pages <= 0 ||
      page_size <= 0 || max_pages_per_seq <= 0 || window < 0)
    return TL_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_table || !positions || !out)
    return TL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return TL_ERR_INVALID_ARG;
  if (h_q % h_kv) return TL_ERR_INVALID_ARG;
  if (dtype != TL_BF16 || d != 128 || (page_size & (page_size - 1)) || page_size < 8 ||
      page_size > 128)
    return TL_ERR_UNSUPPORTED;
  (void)workspace;
  (void)workspace_bytes;
  PrefillParams P;
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  P.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  P.block_table = block_table;
  P.positions = positions;
  P.out = out;
  P.max_pages_per_seq = max_pages_per_seq;
  P.B = B;
  P.T = T;
  P.h_q = h_q;
  P.h_kv = h_kv;
  P.group = h_q / h_kv;
  P.num_pages = num_pages;
  P.page_size = page_size;
  P.window = window;
  P.scale_log2 = scale * kLog2e;
  P.error_word = error_word;
  const int n_qt = (T + kPfRows - 1) / kPfRows;
  if (B > 65535 || h_q > 65535) return TL_ERR_UNSUPPORTED;
  auto kern = prefill_mma_kernel<128>;
  const int sm = PfSmem<128>::kTotal;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sm) != cudaSuccess)
    return TL_ERR_CUDA;
  kern<<<dim3(n_qt, h_q, B), kPfThreads, sm, (cudaStream_t)stream>>>(P);
  return launch_status();
}
