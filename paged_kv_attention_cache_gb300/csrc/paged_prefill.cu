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
#include "tcgen05.cuh"

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


// ------------------------------------------------------- tcgen05 prefill --
//
// One CTA per (pair of query tiles, KV head, row).  A query tile packs
// tokens_per_tile = 128/group consecutive tokens of one row with all `group`
// query heads that share the KV head, as the 128 M rows (row r = token
// r/group, head r%group); the CTA holds two consecutive tiles (Q0, Q1), so
// every K/V tile it streams feeds 256 rows.  Keys are folded in tiles of 128
// over the range the CTA's live tokens can see ([min lo, max p]); every MMA
// has N = 128 (keys for S, head dimension for P.V), the width at which the
// 5th-generation tensor core runs near its peak.
//   warp 0      TMA producer: Q0 and Q1 once (a 3-D map (d, H_q, token), box
//               64 x group x tokens), then K and V tiles into rings of kKS /
//               kVS stages, boxes of 8 or 16 rows of the pool map (one page
//               run each); boxes past the sequence or on bad pages load
//               zeros; the last V tile's rows past the CTA's last position
//               are zeroed.
//   warp 1      TMEM owner (512 columns: S0/P0 [0,128), S1/P1 [128,256),
//               O0 [256,384), O1 [384,512)) and MMA issuer (one lane), in the
//               order PV0_j, S0_{j+1}, PV1_j, S1_{j+1}: S_a = Q_a K^T (8 MMAs,
//               K = 128 from shared-memory descriptors), O_a += P_a V (16
//               MMAs: hi and lo bf16 parts of P, A read from TMEM).
//   warps 2-5   softmax for Q0, warps 6-9 for Q1, one thread per M row: load
//               the row of S_a (four 32-column loads, one wait), mask by the
//               row's causal / window range (skipped when the whole warp sees
//               only live keys), running max in log2 units with a lazy
//               rescale (O and the sum change only when the max grows by
//               more than 2^8), write P = hi + lo bf16 over each 32-column
//               chunk's own columns; finally the epilogue O / l.
// While one warpgroup computes softmax on its tile, the tensor core works on
// the other tile, so the two overlap.  P_a aliases S_a: S_a(j+1) is issued
// after PV_a(j) and the tensor core runs a thread's MMAs in order, and when
// S_a(j+1) is complete so is PV_a(j) (its O is stable for a rescale).  All
// waits are bounded.
constexpr int kBN = 128;             // keys per tile
constexpr int kTcKS = 3;             // K stages
constexpr int kTcVS = 2;             // V stages
constexpr int kTcThreads = 10 * 32;
constexpr int kTcQBytes = 32768;     // one query tile: 128 rows x 128 d x bf16
constexpr int kTcKVBytes = kBN * 256;  // 128 keys x 128 d x bf16 (two 16 KiB halves)
constexpr int kTcSmem = 2 * kTcQBytes + (kTcKS + kTcVS) * kTcKVBytes + 1024;
constexpr uint32_t kTcCols = 512;
constexpr float kRescaleLog2 = 8.f;

struct TcShared {
  unsigned long long q_full, k_full[kTcKS], k_empty[kTcKS], v_full[kTcVS], v_empty[kTcVS], v_fix;
  unsigned long long s_full[2], p_full[2], o_done[2], mma_drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct TcRange {
  int kmin, kmax;  // key range of the CTA's live tokens (kmax < 0: none)
};

// Every warp computes the CTA's key range itself (no shared state needed).
__device__ __forceinline__ TcRange tc_tile_range(const PrefillParams& P, int b, int t0, int ntok,
                                                 int64_t cap) {
  int kmin = INT32_MAX, kmax = -1;
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < ntok; i += 32) {
    const int t = t0 + i;
    if (t >= P.T) break;
    int p = P.positions[(size_t)b * P.T + t];
    if (p >= cap) p = -1;
    if (p >= 0) {
      const int lo = (P.window > 0 && p - P.window + 1 > 0) ? p - P.window + 1 : 0;
      kmin = min(kmin, lo);
      kmax = max(kmax, p);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  return {kmin, kmax};
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(PrefillParams P, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, int box_rows) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ TcShared sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase, sK = sbase + 2 * kTcQBytes, sV = sK + kTcKS * kTcKVBytes;
  volatile int* abort_flag = &sh.abort_flag;

  const int tpt = 128 / P.group;                 // tokens per query tile
  const int rows_used = tpt * P.group;
  const int n_pairs = (P.T + 2 * tpt - 1) / (2 * tpt);
  // grid (row x KV head, pair): the latest (heaviest) pairs of every row and
  // head launch first, so the long CTAs do not end up in the tail
  const int qp = n_pairs - 1 - (int)blockIdx.y;
  const int g = (int)blockIdx.x % P.h_kv, b = (int)blockIdx.x / P.h_kv;
  const int t0 = qp * 2 * tpt;
  const int64_t cap = (int64_t)P.max_pages_per_seq * P.page_size;
  const TcRange rg = tc_tile_range(P, b, t0, 2 * tpt, cap);

  if (rg.kmax < 0) {  // no live token: the outputs are 0
    for (int idx = threadIdx.x; idx < 2 * rows_used * 32; idx += kTcThreads) {
      const int r = idx >> 5, c = (idx & 31) * 4;
      const int a = r / rows_used, rr = r % rows_used;
      const int t = t0 + a * tpt + rr / P.group;
      if (t < P.T)
        *reinterpret_cast<float4*>(
            P.out + (((size_t)b * P.T + t) * P.h_q + (size_t)g * P.group + rr % P.group) * 128 + c) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  const int tile0 = rg.kmin / kBN, n_tiles = rg.kmax / kBN - tile0 + 1;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sh.q_full), 1);
    for (int i = 0; i < kTcKS; ++i) {
      mbar_init(smem_u32(&sh.k_full[i]), 1);
      mbar_init(smem_u32(&sh.k_empty[i]), 1);
    }
    for (int i = 0; i < kTcVS; ++i) {
      mbar_init(smem_u32(&sh.v_full[i]), 1);
      mbar_init(smem_u32(&sh.v_empty[i]), 1);
    }
    mbar_init(smem_u32(&sh.v_fix), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh.s_full[i]), 1);
      mbar_init(smem_u32(&sh.p_full[i]), 4);
      mbar_init(smem_u32(&sh.o_done[i]), 1);
    }
    mbar_init(smem_u32(&sh.mma_drain), 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::alloc(smem_u32(&sh.tmem_base), kTcCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // -------------------------------------------------------------- TMA
    const int nbox = kBN / box_rows;  // boxes per row half of a tile (8 or 16)
    const int n_slots = P.num_pages * P.page_size;
    const int32_t* bt_row = P.block_table + (size_t)b * P.max_pages_per_seq;
    const int last_blk = rg.kmax / P.page_size;
    int win_blk0 = -1, win = -1;
    uint32_t k_issued = 0, v_issued = 0;
    if (lane == 0) {
      const uint32_t qbytes = (uint32_t)(64 * rows_used * 2);  // one half of one tile
      mbar_arrive_expect_tx(smem_u32(&sh.q_full), 4 * qbytes);
      for (int a = 0; a < 2; ++a)
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sQ + a * kTcQBytes + h * (kTcQBytes / 2), &qmap, h * 64, g * P.group,
                      b * P.T + t0 + a * tpt, smem_u32(&sh.q_full));
    }
    for (int j = 0; j < n_tiles; ++j) {
      const int key0 = (tile0 + j) * kBN;
      const int bmin = key0 / P.page_size;
      const int bmax = min((key0 + kBN - 1) / P.page_size, last_blk);
      if (win_blk0 < 0 || bmin < win_blk0 || bmax >= win_blk0 + 32) {
        win_blk0 = bmin;
        const int blk = win_blk0 + lane;
        win = blk <= last_blk ? __ldg(bt_row + blk) : -1;
      }
      // this lane's boxes: lanes < 2*nbox (two row halves); box bi of half
      const int half = lane / nbox, bi = lane % nbox;
      const int kb = key0 + bi * box_rows;
      const int blk = kb / P.page_size;
      const int pg = __shfl_sync(0xffffffffu, win, (blk - win_blk0) & 31);
      const bool box_ok = blk <= last_blk && pg >= 0 && pg < P.num_pages;
      if (blk <= last_blk && !box_ok && lane < 2 * nbox) report(P.error_word, TL_DEVERR_PAGE_RANGE);
      const int slot0 = box_ok ? pg * P.page_size + kb % P.page_size : n_slots;
      const uint32_t boff = half * (kTcKVBytes / 2) + bi * box_rows * 128;
      {
        const int st = j % kTcKS;
        if (!mbar_wait(smem_u32(&sh.k_empty[st]), ((j / kTcKS) & 1) ^ 1, abort_flag)) break;
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&sh.k_full[st]), kTcKVBytes);
        __syncwarp();
        if (lane < 2 * nbox)
          tma_load_3d(sK + st * kTcKVBytes + boff, &kmap, half * 64, g, slot0,
                      smem_u32(&sh.k_full[st]));
        ++k_issued;
      }
      {
        const int st = j % kTcVS;
        if (!mbar_wait(smem_u32(&sh.v_empty[st]), ((j / kTcVS) & 1) ^ 1, abort_flag)) break;
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&sh.v_full[st]), kTcKVBytes);
        __syncwarp();
        if (lane < 2 * nbox)
          tma_load_3d(sV + st * kTcKVBytes + boff, &vmap, half * 64, g, slot0,
                      smem_u32(&sh.v_full[st]));
        ++v_issued;
        if (j == n_tiles - 1) {
          // rows past the CTA's last position may hold anything: zero them
          if (!mbar_wait(smem_u32(&sh.v_full[st]), (j / kTcVS) & 1, abort_flag)) break;
          const int first_dead = rg.kmax + 1 - key0;  // 1..kBN
          const uint32_t vt = sV + st * kTcKVBytes;
          for (int idx = lane; idx < (kBN - first_dead) * 16; idx += 32) {
            const int row = first_dead + (idx >> 4), hu = idx & 15;
            const uint32_t a = vt + (hu >> 3) * (kTcKVBytes / 2) + row * 128 + ((hu & 7) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u) : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sh.v_fix));
        }
      }
    }
    // drain: the copies this warp issued have landed before the CTA exits
    bool drained = true;
    for (uint32_t i = k_issued > (uint32_t)kTcKS ? k_issued - kTcKS : 0; i < k_issued; ++i)
      drained &= mbar_drain(smem_u32(&sh.k_full[i % kTcKS]), (i / kTcKS) & 1);
    for (uint32_t i = v_issued > (uint32_t)kTcVS ? v_issued - kTcVS : 0; i < v_issued; ++i)
      drained &= mbar_drain(smem_u32(&sh.v_full[i % kTcVS]), (i / kTcVS) & 1);
    drained &= mbar_drain(smem_u32(&sh.q_full), 0);
    if (!drained) *abort_flag = 1;
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idS = tc::idesc_bf16(128, kBN, 0, 0);
      const uint32_t idPV = tc::idesc_bf16(128, 128, 0, 1);
      auto issue_s = [&](int a, int j) {  // S_a(j) into TMEM columns [128a, 128a+128)
        const uint32_t kt = sK + (j % kTcKS) * kTcKVBytes;
        const uint32_t qt = sQ + a * kTcQBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t qo = (k >> 2) * (kTcQBytes / 2) + (k & 3) * 32;
          const uint32_t ko = (k >> 2) * (kTcKVBytes / 2) + (k & 3) * 32;
          tc::mma_ss(tmem + a * 128, tc::sdesc(qt + qo, 16, 1024), tc::sdesc(kt + ko, 16, 1024),
                     idS, k > 0);
        }
        tc::commit(smem_u32(&sh.s_full[a]));
      };
      auto issue_pv = [&](int a, int j) {  // O_a += P_a(j) V(j)
        const uint32_t vt = sV + (j % kTcVS) * kTcKVBytes;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k)  // P chunk c = k/2 holds hi at +0, lo at +16
            tc::mma_ts(tmem + 256 + a * 128,
                       tmem + a * 128 + 32 * (k >> 1) + 8 * (k & 1) + 16 * part,
                       tc::sdesc(vt + k * 2048, kTcKVBytes / 2, 1024), idPV,
                       (j > 0 || part > 0 || k > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(smem_u32(&sh.q_full), 0, abort_flag) &&
                mbar_wait(smem_u32(&sh.k_full[0]), 0, abort_flag);
      if (ok) {
        tc::fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        tc::commit(smem_u32(&sh.k_empty[0]));
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        const bool last = j == n_tiles - 1;
        if (!mbar_wait(last ? smem_u32(&sh.v_fix) : smem_u32(&sh.v_full[j % kTcVS]),
                       last ? 0 : (j / kTcVS) & 1, abort_flag))
          break;
        if (!mbar_wait(smem_u32(&sh.p_full[0]), j & 1, abort_flag)) break;
        tc::fence_after();
        issue_pv(0, j);
        if (last) {
          tc::commit(smem_u32(&sh.o_done[0]));
        } else {
          if (!mbar_wait(smem_u32(&sh.k_full[(j + 1) % kTcKS]), ((j + 1) / kTcKS) & 1,
                         abort_flag))
            break;
          tc::fence_after();
          issue_s(0, j + 1);
        }
        if (!mbar_wait(smem_u32(&sh.p_full[1]), j & 1, abort_flag)) break;
        tc::fence_after();
        issue_pv(1, j);
        tc::commit(smem_u32(&sh.v_empty[j % kTcVS]));
        if (last) {
          tc::commit(smem_u32(&sh.o_done[1]));
        } else {
          issue_s(1, j + 1);
          tc::commit(smem_u32(&sh.k_empty[(j + 1) % kTcKS]));
        }
      }
      // every MMA this thread issued is done before TMEM is released
      tc::commit(smem_u32(&sh.mma_drain));
      if (!mbar_drain(smem_u32(&sh.mma_drain), 0)) *abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- softmax
    const int a = (warp - 2) >> 2;  // query tile of this warpgroup
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t colS = a * 128, colO = 256 + a * 128;
    const int t = t0 + a * tpt + row / P.group, h = g * P.group + row % P.group;
    int p = -1;
    if (row < rows_used && t < P.T) {
      p = P.positions[(size_t)b * P.T + t];
      if (p >= cap) {
        report(P.error_word, TL_DEVERR_CONTEXT_RANGE);
        p = -1;
      }
    }
    const int lo = (P.window > 0 && p - P.window + 1 > 0) ? p - P.window + 1 : 0;
    const float sc = P.scale_log2;
    float m_used = -INFINITY, l = 0.f;  // running max of the scores in log2 units
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!mbar_wait(smem_u32(&sh.s_full[a]), j & 1, abort_flag)) { ok = false; break; }
      tc::fence_after();
      const int key0 = (tile0 + j) * kBN;
      const int cmin = lo - key0, cmax = p - key0;  // live columns [cmin, cmax]
      const bool all_live = __all_sync(0xffffffffu, cmin <= 0 && cmax >= kBN - 1);
      // the tile's 128 scores of this row: four loads, one wait
      float s[kBN];
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q) tc::ld32(tmem + lane_base + colS + q * 32, s + q * 32);
      tc::wait_ld();
      if (!all_live) {
#pragma unroll
        for (int c = 0; c < kBN; ++c) s[c] = (c >= cmin && c <= cmax) ? s[c] : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
      for (int c = 8; c < kBN; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sc;
      const bool need = l > 0.f && mt > m_used + kRescaleLog2;
      float corr = 1.f;
      if (need) {
        corr = fast_exp2(m_used - mt);
        m_used = mt;
      }
      if (m_used == -INFINITY) m_used = mt;  // first live key of this row
      const float base = m_used == -INFINITY ? 0.f : m_used;
      // P = exp2(s*sc - base) as hi + lo bf16 over each 32-column chunk's own columns
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q) {
        uint32_t pk[32];  // [0,16) hi, [16,32) lo
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = fast_exp2(fmaf(s[q * 32 + 2 * i], sc, -base));
          const float x1 = fast_exp2(fmaf(s[q * 32 + 2 * i + 1], sc, -base));
          ls[i & 3] += x0 + x1;
          split_bf16x2(x0, x1, pk[i], pk[16 + i]);
        }
        tc::st16(tmem + lane_base + colS + q * 32, pk);
        tc::st16(tmem + lane_base + colS + q * 32 + 16, pk + 16);
      }
      l = l * corr + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      if (__any_sync(0xffffffffu, need)) {
        // PV_a(j-1) is complete (S_a(j) was issued after it) and PV_a(j)
        // waits for this tile's P: rescale O_a now
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float o[32];
          tc::ld32(tmem + lane_base + colO + q * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tc::st32(tmem + lane_base + colO + q * 32, o);
        }
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.p_full[a]));
    }
    // epilogue: O / l
    if (ok && mbar_wait(smem_u32(&sh.o_done[a]), 0, abort_flag)) {
      tc::fence_after();
      const float inv = (p >= 0 && l > 0.f) ? 1.f / l : 0.f;
      float* dst = P.out + (((size_t)b * P.T + t) * P.h_q + h) * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float o[32];
        tc::ld32(tmem + lane_base + colO + q * 32, o);
        tc::wait_ld();
        if (row < rows_used && t < P.T) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + q * 32 + i) =
                make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();  // every wait above is bounded, so every thread gets here
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tmem, kTcCols);
  }
  if (threadIdx.x == 0 && sh.abort_flag) report(P.error_word, TL_DEVERR_TIMEOUT);
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
  if (!(scale > 0.f) || scale > 3.0e38f) return TL_ERR_INVALID_ARG;
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
  if (h_q / h_kv > 128 || B > 65535 || h_kv > 65535) return TL_ERR_UNSUPPORTED;
  if ((int64_t)num_pages * page_size >= ((int64_t)1 << 31) || (int64_t)B * T >= ((int64_t)1 << 31))
    return TL_ERR_UNSUPPORTED;
  const int group = h_q / h_kv;
  const int tpt = 128 / group;
  const int box_rows = page_size % 16 == 0 ? 16 : 8;
  CUtensorMap qmap, kmap, vmap;
  {
    const uint64_t qd[3] = {128, (uint64_t)h_q, (uint64_t)B * T};
    const uint64_t qs[2] = {128 * 2, (uint64_t)h_q * 128 * 2};
    const uint32_t qb[3] = {64, (uint32_t)group, (uint32_t)tpt};
    const uint64_t kd[3] = {128, (uint64_t)h_kv, (uint64_t)num_pages * page_size};
    const uint64_t ks[2] = {128 * 2, (uint64_t)h_kv * 128 * 2};
    const uint32_t kb[3] = {64, 1, (uint32_t)box_rows};
    if (!encode_bf16_tensor_map(&qmap, q, 3, qd, qs, qb, true) ||
        !encode_bf16_tensor_map(&kmap, k_cache, 3, kd, ks, kb, true) ||
        !encode_bf16_tensor_map(&vmap, v_cache, 3, kd, ks, kb, true))
      return TL_ERR_CUDA;
  }
  if (cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTcSmem) != cudaSuccess)
    return TL_ERR_CUDA;
  const int n_pairs = (T + 2 * tpt - 1) / (2 * tpt);
  if ((int64_t)B * h_kv > 0x7fffffff || n_pairs > 65535) return TL_ERR_UNSUPPORTED;
  prefill_tc_kernel<<<dim3(B * h_kv, n_pairs), kTcThreads, kTcSmem, (cudaStream_t)stream>>>(
      P, qmap, kmap, vmap, box_rows);
  return launch_status();
}
