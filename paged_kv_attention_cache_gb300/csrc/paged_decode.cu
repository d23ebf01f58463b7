// PAGED_ATTENTION, decode: one query token per sequence, split-K over the
// sequence's keys ("flash-decoding"), then a log-sum-exp combine.
//
// What it computes is defined in "How serving works in Tlaloc", section 2
// (gather through the block table, dot, masked softmax, dot; causal length =
// position + 1) and section 3 (sliding window p-W+1 .. p).  The split-K merge
// is the same fold as the page's "Blockwise attention" bullet (running max,
// running sum, running P.V), applied across CTAs instead of loop iterations.
//
// Three launches on the caller's stream:
//   1. decode_plan_kernel (1 CTA): per sequence, the 16-key chunks it reads
//      ([lo/16, p/16]); a split size (in chunks) that gives about
//      kTargetItems work items for the whole batch; an exclusive scan of the
//      splits per sequence.  Zeroes the work counter.
//   2. decode_bf16_kernel / decode_f32_kernel (persistent, 2 CTAs per SM):
//      CTAs take work items (split s, KV head g) from an atomic counter.  The 4
//      warps of a CTA take the item's chunks round-robin; each warp streams its
//      chunks' K and V rows from the pool into its own shared-memory ring with
//      16-byte cp.async (3 stages), and keeps a running (max, sum, P.V) per
//      query head of the group.  bf16: Q.K^T and P.V run on mma.sync
//      m16n8k16 with the query-head group as the M rows, so the ALUs stay far
//      from the limit even at 8 query heads per KV head.  The warps' states
//      are merged in shared memory and written as one partial per (split,
//      query head).
//   3. decode_combine_kernel: one warp per (sequence, query head) merges the
//      sequence's partials in split order.
// Every reduction has a fixed order, so results repeat bit for bit and do not
// depend on the pool's page placement.
#include "common.cuh"

namespace tl {

constexpr int kChunk = 16;           // keys per step (one mma N=16 / K=16 tile)
constexpr int kTargetItems = 8192;   // work items (split x KV head) per call
constexpr int kMinSplitChunks = 8;   // 128 keys
constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = kDecodeWarps * 32;
constexpr int kStages = 3;

inline int64_t decode_max_splits(int B, int h_kv) {
  return (int64_t)(kTargetItems + h_kv - 1) / h_kv + B;
}

struct DecodeWorkspace {
  int32_t* ctrl;       // [0] split size in chunks, [1] total splits, [2] work counter
  int32_t* split_off;  // [B+1] first split of each sequence
  float* ml;           // [max_splits][h_q][2]   (running max in log2 units, sum)
  float* acc;          // [max_splits][h_q][d]   (unnormalised P.V)
};

inline size_t decode_ws_layout(int B, int h_q, int h_kv, int d, DecodeWorkspace* w,
                               char* base) {
  const int64_t ms = decode_max_splits(B, h_kv);
  size_t off = 0;
  const size_t ctrl = off;
  off += 256;
  const size_t so = off;
  off = align_up(off + sizeof(int32_t) * (size_t)(B + 1), 256);
  const size_t ml = off;
  off = align_up(off + sizeof(float) * 2 * (size_t)ms * h_q, 256);
  const size_t acc = off;
  off = align_up(off + sizeof(float) * (size_t)ms * h_q * d, 256);
  if (w) {
    w->ctrl = reinterpret_cast<int32_t*>(base + ctrl);
    w->split_off = reinterpret_cast<int32_t*>(base + so);
    w->ml = reinterpret_cast<float*>(base + ml);
    w->acc = reinterpret_cast<float*>(base + acc);
  }
  return off;
}

struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* context_lens;
  float* out;
  int32_t max_pages_per_seq;
  int32_t B, h_q, h_kv, group;
  int32_t num_pages, page_size, window;
  float scale_log2;  // scale * log2(e): scores are kept in log2 units
  DecodeWorkspace ws;
  uint32_t* error_word;
};

// Causal range of sequence b: keys lo..p (empty when L <= 0 or L too long).
__device__ __forceinline__ void seq_range(const DecodeParams& P, int b, int& lo, int& p) {
  const int L = P.context_lens[b];
  const int64_t cap = (int64_t)P.max_pages_per_seq * P.page_size;
  p = L - 1;
  if (L > cap) {
    report(P.error_word, TL_DEVERR_CONTEXT_RANGE);
    p = -1;
  }
  lo = (P.window > 0 && p - P.window + 1 > 0) ? p - P.window + 1 : 0;
}

__device__ __forceinline__ int seq_chunks(const DecodeParams& P, int b) {
  int lo, p;
  seq_range(P, b, lo, p);
  return p < 0 ? 0 : p / kChunk - lo / kChunk + 1;
}

// ------------------------------------------------------------------ plan --

__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeParams P, int target_splits) {
  __shared__ long long red[32];
  __shared__ int warp_incl[32];
  __shared__ int carry_s;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, wid = tid >> 5;
  const int nwarps = nt >> 5;
  long long total = 0;
  for (int b = tid; b < P.B; b += nt) total += seq_chunks(P, b);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  if (lane == 0) red[wid] = total;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  long long total_chunks = 0;
  for (int w = 0; w < nwarps; ++w) total_chunks += red[w];
  const long long s = (total_chunks + target_splits - 1) / target_splits;
  const int split = (int)(s < kMinSplitChunks ? kMinSplitChunks : s);
  // exclusive scan of the splits per sequence, nt sequences at a time
  for (int base = 0; base < P.B; base += nt) {
    const int b = base + tid;
    const int n = b < P.B ? (seq_chunks(P, b) + split - 1) / split : 0;
    int x = n;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_incl[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int v = lane < nwarps ? warp_incl[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      warp_incl[lane] = v;
    }
    __syncthreads();
    const int carry = carry_s;
    const int before = carry + (wid > 0 ? warp_incl[wid - 1] : 0) + x - n;
    if (b < P.B) P.ws.split_off[b] = before;
    const int chunk_total = warp_incl[nwarps - 1];
    __syncthreads();
    if (tid == 0) carry_s = carry + chunk_total;
    __syncthreads();
  }
  if (tid == 0) {
    P.ws.split_off[P.B] = carry_s;
    P.ws.ctrl[0] = split;
    P.ws.ctrl[1] = carry_s;
    P.ws.ctrl[2] = 0;
  }
}

// Work item -> (sequence, split within the sequence): the last b with
// split_off[b] <= s.
__device__ __forceinline__ int find_seq(const int32_t* split_off, int B, int s) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(split_off + mid) <= s) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct ItemInfo {
  int b, g, lo, p, c_begin, c_end;  // chunks [c_begin, c_end)
};

__device__ __forceinline__ bool next_item(const DecodeParams& P, int* s_item, ItemInfo& it) {
  if (threadIdx.x == 0) *s_item = atomicAdd(P.ws.ctrl + 2, 1);
  __syncthreads();
  const int item = *s_item;
  const int total = P.ws.ctrl[1] * P.h_kv;
  __syncthreads();  // everyone has read *s_item before it is rewritten
  if (item >= total) return false;
  const int s = item / P.h_kv;
  it.g = item - s * P.h_kv;
  it.b = find_seq(P.ws.split_off, P.B, s);
  const int split = P.ws.ctrl[0];
  const int k = s - P.ws.split_off[it.b];
  seq_range(P, it.b, it.lo, it.p);
  const int c0 = it.lo / kChunk, c1 = it.p / kChunk + 1;
  it.c_begin = c0 + k * split;
  it.c_end = min(c1, it.c_begin + split);
  return true;
}

// Merge the per-warp states in shared memory and write the item's partial.
// Warp w's rows start at merge + w*warp_stride: row r holds P.V in [0, D),
// the running max (log2 units) at D and the running sum at D+1.
template <int D>
__device__ __forceinline__ void merge_and_store(const DecodeParams& P, const ItemInfo& it,
                                                int s_global, const float* merge,
                                                int warp_stride) {
  constexpr int RS = D + 2;
  for (int idx = threadIdx.x; idx < P.group * (D + 1); idx += kDecodeThreads) {
    const int r = idx / (D + 1), e = idx - r * (D + 1);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, merge[w * warp_stride + r * RS + D]);
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float* mr = merge + w * warp_stride + r * RS;
      const float f = mr[D] == -INFINITY ? 0.f : fast_exp2(mr[D] - M);
      a += f * (e < D ? mr[e] : mr[D + 1]);
    }
    const size_t row = (size_t)s_global * P.h_q + (size_t)it.g * P.group + r;
    if (e < D) {
      P.ws.acc[row * D + e] = a;
    } else {
      P.ws.ml[row * 2 + 0] = M;
      P.ws.ml[row * 2 + 1] = a;
    }
  }
}

__device__ __forceinline__ int item_split_index(const DecodeParams& P, const ItemInfo& it) {
  return __ldg(P.ws.split_off + it.b) + (it.c_begin - it.lo / kChunk) / P.ws.ctrl[0];
}

// ------------------------------------------------------------ bf16 kernel --
//
// Per warp and stage: K chunk then V chunk, 16 rows of D bf16 each.  Row r's
// 16-byte unit u is stored at unit u ^ (r & 7) so that ldmatrix reads of 8
// rows hit 8 different bank groups.

template <int D>
struct Bf16Smem {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kChunkBytes = kChunk * kRowBytes;      // one of K or V
  static constexpr int kStageBytes = 2 * kChunkBytes;         // K + V
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kMergeBytes = 16 * (D + 2) * 4;        // per warp
  static_assert(kMergeBytes <= kWarpBytes, "merge area overlays the warp's ring");
  static constexpr int kTotal = kDecodeWarps * kWarpBytes + 64;
};

// Issue the cp.async copies of one chunk's K and V rows into a stage; returns
// the mask of rows that hold a live key (bit r for row r).
template <int D>
__device__ __forceinline__ uint32_t issue_chunk(const DecodeParams& P, const ItemInfo& it,
                                                int chunk, uint32_t stage_addr, int lane,
                                                int elem_bytes) {
  constexpr int U = D * 2 / 16;  // bf16: 16-byte units per row
  const int r = lane >> 1;
  const int j = chunk * kChunk + r;
  bool live = j >= it.lo && j <= it.p;
  int64_t page = 0;
  if (live) {
    page = __ldg(P.block_table + (size_t)it.b * P.max_pages_per_seq + j / P.page_size);
    if (page < 0 || page >= P.num_pages) {
      live = false;
      report(P.error_word, TL_DEVERR_PAGE_RANGE);
      page = 0;
    }
  }
  const size_t row_elem =
      (((size_t)page * P.page_size + (live ? j % P.page_size : 0)) * P.h_kv + it.g) * D;
  const char* ks = static_cast<const char*>(P.k_cache) + row_elem * elem_bytes;
  const char* vs = static_cast<const char*>(P.v_cache) + row_elem * elem_bytes;
  const uint32_t kd = stage_addr + r * (D * 2);
  const uint32_t vd = kd + Bf16Smem<D>::kChunkBytes;
  const uint32_t nbytes = live ? 16u : 0u;
#pragma unroll
  for (int i = 0; i < U / 2; ++i) {
    const int u = (lane & 1) + 2 * i;
    const uint32_t phys = (uint32_t)((u ^ (r & 7)) << 4);
    cp_async_16(kd + phys, ks + u * 16, nbytes);
    cp_async_16(vd + phys, vs + u * 16, nbytes);
  }
  const uint32_t ballot = __ballot_sync(0xffffffffu, live);
  uint32_t mask = 0;
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) mask |= ((ballot >> (2 * rr)) & 1u) << rr;
  return mask;
}

template <int D, bool TWO_ROWS>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_bf16_kernel(DecodeParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_item;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* wbase = smem + warp * Bf16Smem<D>::kWarpBytes;
  const uint32_t wbase_u32 = smem_u32(wbase);
  const int qr = lane >> 2, qc = (lane & 3) * 2;  // fragment row / column pair
  ItemInfo it;
  while (next_item(P, &s_item, it)) {
    const int s_global = item_split_index(P, it);
    // Q fragments (rows = query heads of the group, zero past the group)
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(P.q) +
                              ((size_t)it.b * P.h_q + (size_t)it.g * P.group) * D;
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int e0 = ks * 16 + qc;
      qa[ks][0] = qr < P.group ? *reinterpret_cast<const uint32_t*>(qb + qr * D + e0) : 0u;
      qa[ks][2] = qr < P.group ? *reinterpret_cast<const uint32_t*>(qb + qr * D + e0 + 8) : 0u;
      if (TWO_ROWS) {
        qa[ks][1] =
            qr + 8 < P.group ? *reinterpret_cast<const uint32_t*>(qb + (qr + 8) * D + e0) : 0u;
        qa[ks][3] = qr + 8 < P.group
                        ? *reinterpret_cast<const uint32_t*>(qb + (qr + 8) * D + e0 + 8)
                        : 0u;
      } else {
        qa[ks][1] = 0u;
        qa[ks][3] = 0u;
      }
    }
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // this warp's chunks: c_begin + warp + 4*i
    const int first = it.c_begin + warp;
    const int n_my = first < it.c_end ? (it.c_end - first + kDecodeWarps - 1) / kDecodeWarps : 0;
    // live-row masks of the chunks in flight, oldest first (registers)
    uint32_t mq[kStages - 1];
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
      mq[st] = 0u;
      if (st < n_my)
        mq[st] = issue_chunk<D>(P, it, first + st * kDecodeWarps,
                                wbase_u32 + st * Bf16Smem<D>::kStageBytes, lane, 2);
      cp_async_commit();
    }
    for (int i = 0; i < n_my; ++i) {
      uint32_t newest = 0u;
      {
        const int ni = i + kStages - 1;
        if (ni < n_my)
          newest = issue_chunk<D>(P, it, first + ni * kDecodeWarps,
                                  wbase_u32 + (ni % kStages) * Bf16Smem<D>::kStageBytes, lane, 2);
        cp_async_commit();
      }
      cp_async_wait<kStages - 1>();
      __syncwarp();
      const int st = i % kStages;
      const uint32_t mask = mq[0];
#pragma unroll
      for (int k = 0; k < kStages - 2; ++k) mq[k] = mq[k + 1];
      mq[kStages - 2] = newest;
      const uint32_t kaddr = wbase_u32 + st * Bf16Smem<D>::kStageBytes;
      const uint32_t vaddr = kaddr + Bf16Smem<D>::kChunkBytes;
      // S = Q K^T over the chunk's 16 keys (two n-tiles of 8 keys)
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int mi = lane >> 3, ri = lane & 7;
        const int tok = (mi >> 1) * 8 + ri;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int u = 2 * ks + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kaddr + tok * (D * 2) + ((u ^ (tok & 7)) << 4), b0, b1, b2, b3);
          mma_bf16_16816(s[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(s[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
      // mask and scale (log2 units)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = n * 8 + qc + e;
          const bool ok = (mask >> key) & 1u;
          s[n][e] = ok ? s[n][e] * P.scale_log2 : -INFINITY;
          s[n][2 + e] = ok ? s[n][2 + e] * P.scale_log2 : -INFINITY;
          mx0 = fmaxf(mx0, s[n][e]);
          mx1 = fmaxf(mx1, s[n][2 + e]);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      const float mn0 = fmaxf(m0, mx0);
      const float base0 = mn0 == -INFINITY ? 0.f : mn0;  // no live key seen yet
      const float c0 = fast_exp2(m0 - base0);
      m0 = mn0;
      float p[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        p[n][0] = fast_exp2(s[n][0] - base0);
        p[n][1] = fast_exp2(s[n][1] - base0);
      }
      l0 = l0 * c0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
      float c1 = c0;
      if (TWO_ROWS) {
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn1 = fmaxf(m1, mx1);
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        c1 = fast_exp2(m1 - base1);
        m1 = mn1;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          p[n][2] = fast_exp2(s[n][2] - base1);
          p[n][3] = fast_exp2(s[n][3] - base1);
        }
        l1 = l1 * c1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
      }
      // rows 8-15 carry either the second half of the group (TWO_ROWS) or the
      // low bf16 part of rows 0-7's probabilities; both rescale with their row
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= c0;
        o[n][1] *= c0;
        o[n][2] *= c1;
        o[n][3] *= c1;
      }
      // O += P V with P = hi + lo (bf16 pair, ~16 significant bits)
      uint32_t h0, l0w, h2, l2w;
      split_bf16x2(p[0][0], p[0][1], h0, l0w);
      split_bf16x2(p[1][0], p[1][1], h2, l2w);
      {
        const int mi = lane >> 3, ri = lane & 7;
        const int tok = (mi & 1) * 8 + ri;
        if (!TWO_ROWS) {
          // A rows 0-7 = hi part, rows 8-15 = lo part of the same query heads
#pragma unroll
          for (int nd2 = 0; nd2 < D / 16; ++nd2) {
            const int u = 2 * nd2 + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(vaddr + tok * (D * 2) + ((u ^ (tok & 7)) << 4), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * nd2], h0, l0w, h2, l2w, b0, b1);
            mma_bf16_16816(o[2 * nd2 + 1], h0, l0w, h2, l2w, b2, b3);
          }
        } else {
          uint32_t h1, l1w, h3, l3w;
          split_bf16x2(p[0][2], p[0][3], h1, l1w);
          split_bf16x2(p[1][2], p[1][3], h3, l3w);
#pragma unroll
          for (int nd2 = 0; nd2 < D / 16; ++nd2) {
            const int u = 2 * nd2 + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(vaddr + tok * (D * 2) + ((u ^ (tok & 7)) << 4), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * nd2], h0, h1, h2, h3, b0, b1);
            mma_bf16_16816(o[2 * nd2], l0w, l1w, l2w, l3w, b0, b1);
            mma_bf16_16816(o[2 * nd2 + 1], h0, h1, h2, h3, b2, b3);
            mma_bf16_16816(o[2 * nd2 + 1], l0w, l1w, l2w, l3w, b2, b3);
          }
        }
      }
      __syncwarp();
    }
    cp_async_wait<0>();
    __syncwarp();
    // quad sums, then the warp's state into its merge rows
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    if (TWO_ROWS) {
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
    // the warp's state goes into the start of its own ring (its copies are done)
    constexpr int RS = D + 2;
    float* mrow = reinterpret_cast<float*>(wbase);
    if (qr < P.group) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        mrow[qr * RS + n * 8 + qc] = TWO_ROWS ? o[n][0] : o[n][0] + o[n][2];
        mrow[qr * RS + n * 8 + qc + 1] = TWO_ROWS ? o[n][1] : o[n][1] + o[n][3];
      }
      if ((lane & 3) == 0) {
        mrow[qr * RS + D] = m0;
        mrow[qr * RS + D + 1] = l0;
      }
    }
    if (TWO_ROWS && qr + 8 < P.group) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        mrow[(qr + 8) * RS + n * 8 + qc] = o[n][2];
        mrow[(qr + 8) * RS + n * 8 + qc + 1] = o[n][3];
      }
      if ((lane & 3) == 0) {
        mrow[(qr + 8) * RS + D] = m1;
        mrow[(qr + 8) * RS + D + 1] = l1;
      }
    }
    __syncthreads();
    merge_and_store<D>(P, it, s_global, reinterpret_cast<const float*>(smem),
                       Bf16Smem<D>::kWarpBytes / 4);
    __syncthreads();
  }
}

// ------------------------------------------------------------- f32 kernel --
//
// IEEE f32 pools ("How serving works in Tlaloc": f32 keys and values, dots in
// f32).  Computed on the CUDA cores in f32: no tensor-core rounding of the
// operands.  Each warp walks its chunks one key at a time: lanes hold D/32
// elements of each query head, a warp sum gives each score, and a scalar
// online softmax folds it in.

constexpr int kF32MaxGroup = 16;

template <int D>
__global__ void __launch_bounds__(kDecodeThreads) decode_f32_kernel(DecodeParams P) {
  constexpr int E = D / 32;
  constexpr int RS = D + 2;
  __shared__ float merge[kDecodeWarps][kF32MaxGroup][RS];
  __shared__ int s_item;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ItemInfo it;
  while (next_item(P, &s_item, it)) {
    const int s_global = item_split_index(P, it);
    const float* qb =
        static_cast<const float*>(P.q) + ((size_t)it.b * P.h_q + (size_t)it.g * P.group) * D;
    float qv[kF32MaxGroup][E], o[kF32MaxGroup][E], m[kF32MaxGroup], l[kF32MaxGroup];
#pragma unroll
    for (int r = 0; r < kF32MaxGroup; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        qv[r][e] = r < P.group ? qb[r * D + lane + 32 * e] * P.scale_log2 : 0.f;
        o[r][e] = 0.f;
      }
    }
    for (int c = it.c_begin + warp; c < it.c_end; c += kDecodeWarps) {
      for (int jj = 0; jj < kChunk; ++jj) {
        const int j = c * kChunk + jj;
        if (j < it.lo || j > it.p) continue;
        const int64_t page =
            __ldg(P.block_table + (size_t)it.b * P.max_pages_per_seq + j / P.page_size);
        if (page < 0 || page >= P.num_pages) {
          if (lane == 0) report(P.error_word, TL_DEVERR_PAGE_RANGE);
          continue;
        }
        const size_t row = (((size_t)page * P.page_size + j % P.page_size) * P.h_kv + it.g) * D;
        float kv[E], vv[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          kv[e] = __ldg(static_cast<const float*>(P.k_cache) + row + lane + 32 * e);
          vv[e] = __ldg(static_cast<const float*>(P.v_cache) + row + lane + 32 * e);
        }
#pragma unroll
        for (int r = 0; r < kF32MaxGroup; ++r) {
          if (r >= P.group) break;
          float part = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) part = fmaf(qv[r][e], kv[e], part);
          const float s = warp_sum(part);
          const float mn = fmaxf(m[r], s);
          const float corr = fast_exp2(m[r] - mn);
          const float pj = fast_exp2(s - mn);
          m[r] = mn;
          l[r] = l[r] * corr + pj;
#pragma unroll
          for (int e = 0; e < E; ++e) o[r][e] = fmaf(pj, vv[e], o[r][e] * corr);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kF32MaxGroup; ++r) {
      if (r >= P.group) break;
#pragma unroll
      for (int e = 0; e < E; ++e) merge[warp][r][lane + 32 * e] = o[r][e];
      if (lane == 0) {
        merge[warp][r][D] = m[r];
        merge[warp][r][D + 1] = l[r];
      }
    }
    __syncthreads();
    merge_and_store<D>(P, it, s_global, &merge[0][0][0], kF32MaxGroup * RS);
    __syncthreads();
  }
}

// --------------------------------------------------------------- combine --

template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(DecodeParams P) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t wi = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (wi >= (int64_t)P.B * P.h_q) return;
  const int b = (int)(wi / P.h_q), h = (int)(wi - (int64_t)b * P.h_q);
  const int s0 = P.ws.split_off[b], s1 = P.ws.split_off[b + 1];
  float* out = P.out + (size_t)wi * D;
  float M = -INFINITY;
  for (int s = s0; s < s1; ++s) M = fmaxf(M, P.ws.ml[((size_t)s * P.h_q + h) * 2]);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int s = s0; s < s1; ++s) {
    const size_t row = (size_t)s * P.h_q + h;
    const float mi = P.ws.ml[row * 2];
    const float f = mi == -INFINITY ? 0.f : fast_exp2(mi - M);
    L += f * P.ws.ml[row * 2 + 1];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] += f * P.ws.acc[row * D + lane * E + e];
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) out[lane * E + e] = acc[e] * inv;
}

}  // namespace tl

// ------------------------------------------------------------------- host --

extern "C" size_t tl_paged_attn_decode_workspace_size(int32_t B, int32_t h_q, int32_t h_kv,
                                                      int32_t d) {
  if (B <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || h_q % h_kv) return 0;
  return tl::decode_ws_layout(B, h_q, h_kv, d, nullptr, nullptr);
}

extern "C" tl_status tl_paged_attn_decode(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_table,
                                          int32_t max_pages_per_seq,
                                          const int32_t* context_lens, float* out, int32_t B,
                                          int32_t h_q, int32_t h_kv, int32_t d,
                                          int32_t num_pages, int32_t page_size, int32_t window,
                                          float scale, tl_dtype dtype, void* workspace,
                                          size_t workspace_bytes, uint32_t* error_word,
                                          void* stream) {
  using namespace tl;
  if (B <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || num_pages <= 0 || page_size <= 0 ||
      max_pages_per_seq <= 0 || window < 0)
    return TL_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out)
    return TL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return TL_ERR_INVALID_ARG;
  if (h_q % h_kv) return TL_ERR_INVALID_ARG;
  const int group = h_q / h_kv;
  if (dtype != TL_BF16 && dtype != TL_F32) return TL_ERR_UNSUPPORTED;
  if ((d != 64 && d != 128) || group > 16 || page_size > 256) return TL_ERR_UNSUPPORTED;
  const size_t need = decode_ws_layout(B, h_q, h_kv, d, nullptr, nullptr);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return TL_ERR_WORKSPACE;

  DecodeParams P;
  P.q = q;
  P.k_cache = k_cache;
  P.v_cache = v_cache;
  P.block_table = block_table;
  P.context_lens = context_lens;
  P.out = out;
  P.max_pages_per_seq = max_pages_per_seq;
  P.B = B;
  P.h_q = h_q;
  P.h_kv = h_kv;
  P.group = group;
  P.num_pages = num_pages;
  P.page_size = page_size;
  P.window = window;
  P.scale_log2 = scale * kLog2e;
  decode_ws_layout(B, h_q, h_kv, d, &P.ws, static_cast<char*>(workspace));
  P.error_word = error_word;
  cudaStream_t st = (cudaStream_t)stream;

  const int target_splits = (kTargetItems + h_kv - 1) / h_kv;
  decode_plan_kernel<<<1, 1024, 0, st>>>(P, target_splits);
  if (launch_status() != TL_OK) return TL_ERR_CUDA;

  const int grid = num_sms() * 2;
  if (dtype == TL_BF16) {
#define TL_LAUNCH_BF16(DD, TWO)                                                           \
  do {                                                                                    \
    auto kern = decode_bf16_kernel<DD, TWO>;                                              \
    const int sm = Bf16Smem<DD>::kTotal;                                                  \
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sm) !=    \
        cudaSuccess)                                                                      \
      return TL_ERR_CUDA;                                                                 \
    kern<<<grid, kDecodeThreads, sm, st>>>(P);                                            \
  } while (0)
    if (d == 128) {
      if (group > 8) TL_LAUNCH_BF16(128, true); else TL_LAUNCH_BF16(128, false);
    } else {
      if (group > 8) TL_LAUNCH_BF16(64, true); else TL_LAUNCH_BF16(64, false);
    }
#undef TL_LAUNCH_BF16
  } else {
    if (d == 128) decode_f32_kernel<128><<<grid, kDecodeThreads, 0, st>>>(P);
    else decode_f32_kernel<64><<<grid, kDecodeThreads, 0, st>>>(P);
  }
  if (launch_status() != TL_OK) return TL_ERR_CUDA;

  const int64_t warps = (int64_t)B * h_q;
  const unsigned cblocks = (unsigned)((warps + 3) / 4);
  if (d == 128) decode_combine_kernel<128><<<cblocks, 128, 0, st>>>(P);
  else decode_combine_kernel<64><<<cblocks, 128, 0, st>>>(P);
  return launch_status();
}
