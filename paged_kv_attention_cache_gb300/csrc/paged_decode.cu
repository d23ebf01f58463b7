// PAGED_ATTENTION, decode: one query token per sequence (or q_len tokens at
// its end: the multi-token / speculative-verify shape), split-K over the
// sequence's keys ("flash-decoding") with a log-sum-exp merge of the splits.
// The table may be a ring (the windowed pool of section 3): logical block k
// is then read from entry k % ring_pages, keys still in position order.
//
// What it computes is defined in "How serving works in Tlaloc", section 2
// (gather through the block table, dot, masked softmax, dot; causal length =
// position + 1) and section 3 (sliding window p-W+1 .. p).  The split merge
// is the fold of the page's "Blockwise attention" bullet (running max, running
// sum, running P.V), applied across work items instead of loop iterations.
//
// Launches on the caller's stream:
//   1. decode_plan_kernel (1 CTA): per sequence the 16-key chunks it reads
//      ([lo/16, p/16]), cut into pieces (splits): bulk pieces sized for about
//      kTargetItems work items, then a last round of small pieces from every
//      long sequence's end; one descriptor per piece in item order, partial
//      indices contiguous per sequence.  Zeroes the work counter and writes
//      the zero output of sequences with nothing to read.
//   2. bf16 / e4m3 / int8: decode_bf16_kernel, a programmatic dependent
//      launch of the plan (it becomes resident while the plan runs and waits
//      for its results), persistent, one CTA per SM, every warp independent:
//      a warp takes work items (piece x KV head) from an atomic counter and
//      streams their chunks (16 keys of K and V, 8 KiB at d=128 in 16 bits)
//      through its own ring of shared-memory stages filled by TMA; Q.K^T and
//      P.V run on mma.sync m16n8k16, with the query-head group (times the
//      q_len tokens, token-major) as the M rows, or, for one-byte pools with
//      at most 8 rows, with the keys as the M rows and the group as the N
//      columns; each row masked to its own causal range, online softmax in
//      registers (details below).  At the end of an item the warp writes
//      from its registers: a sequence with one piece writes its output
//      directly, otherwise the item writes a partial.
//      f32: decode_f32_kernel (CUDA-core dots in f32) writes partials.
//   3. decode_combine_kernel merges the partials of sequences with several
//      pieces, one thread per 4 outputs and G groups of such threads per
//      output row (G grows as the batch shrinks and the pieces of a sequence
//      multiply); after the bf16 / one-byte kernel it is a programmatic
//      dependent launch too.  (Merging inside
//      the attention kernel, by the last piece of each (sequence, KV head)
//      to finish, measured slower: every sequence's last piece is in the
//      small round, so all merges fall in the kernel's last microseconds,
//      each a chain of dependent partial reads against a saturated memory
//      system.)
// Every reduction has a fixed order, so results repeat bit for bit and do not
// depend on the pool's page placement.
#include <algorithm>

#include "common.cuh"
#include "kv_write.cuh"

namespace tl {

// Decode timeline, a build option (-DTL_DECODE_TRACE=1; the default library
// has none of it): %globaltimer stamps (ns) of the phases of a call, in a
// device array read by tl_decode_trace_read.  Slots as in the header's
// TL_TRACE_*: a stamp taken once is one thread's, the attention kernel's end
// is the latest of its CTAs', the combine's start the earliest and its end
// the latest.
#ifndef TL_DECODE_TRACE
#define TL_DECODE_TRACE 0
#endif
#if TL_DECODE_TRACE
__device__ unsigned long long g_trace[TL_TRACE_SLOTS];
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define TL_TRACE_SET(slot) (g_trace[slot] = trace_now())
#define TL_TRACE_MAX(slot) atomicMax(&g_trace[slot], trace_now())
#define TL_TRACE_MIN(slot) atomicMin(&g_trace[slot], trace_now())
#else
#define TL_TRACE_SET(slot) ((void)0)
#define TL_TRACE_MAX(slot) ((void)0)
#define TL_TRACE_MIN(slot) ((void)0)
#endif

constexpr int kChunk = 16;            // keys per step (one mma N=16 / K=16 tile)
constexpr float kLazyLog2 = 8.f;      // the running max moves by more than 2^8 only
// Work items (split x KV head) per call.  Fewer, longer items mean fewer
// partials for the merge and less per-item overhead; the last round of small
// pieces keeps the warps' finishing times close either way.  Measured on
// GB300 (one box, builds side by side): 12288 -> 6144 took the 64-sequence
// Llama-3-8B step from 0.2013 to 0.1955 ms, the long-context batch from
// 0.601 to 0.587 ms, the e4m3 step from 0.120 to 0.113 ms and the 4-token
// verify batch from 0.237 to 0.215 ms; 4096 and 8192 were slower overall.
#ifndef TL_DECODE_ITEMS
#define TL_DECODE_ITEMS 6144
#endif
constexpr int kTargetItems = TL_DECODE_ITEMS;
constexpr int kMinSplitChunks = 8;    // 128 keys
constexpr int kDecodeWarps = 4;       // f32 kernel
constexpr int kDecodeThreads = kDecodeWarps * 32;

// Pieces per call: the plan keeps them within ceil(kTargetItems / h_kv) + 2B
// (each of its two rounds rounds up once per sequence).
__host__ __device__ inline int64_t decode_max_splits(int B, int h_kv) {
  return (int64_t)(kTargetItems + h_kv - 1) / h_kv + 2 * (int64_t)B;
}

struct DecodeWorkspace {
  int32_t* ctrl;       // [0] split size in chunks, [1] total splits, [2] work counter
  int32_t* split_off;  // [B+1] first split of each sequence
  int4* desc;          // [max_splits][2] per-split descriptor (see SplitDesc)
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
  const size_t ds = off;
  off = align_up(off + 2 * sizeof(int4) * (size_t)ms, 256);
  const size_t ml = off;
  off = align_up(off + sizeof(float) * 2 * (size_t)ms * h_q, 256);
  const size_t acc = off;
  off = align_up(off + sizeof(float) * (size_t)ms * h_q * d, 256);
  if (w) {
    w->ctrl = reinterpret_cast<int32_t*>(base + ctrl);
    w->split_off = reinterpret_cast<int32_t*>(base + so);
    w->desc = reinterpret_cast<int4*>(base + ds);
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
  int32_t B, h_q, h_kv, group, d;
  int32_t num_pages, page_size, window;
  int32_t ring_pages;  // > 0: the table's first ring_pages entries are a ring
  int32_t ps_shift;    // log2(page_size) when it is a power of two, else -1
  int32_t q_len;       // query tokens per sequence (positions L - q_len .. L - 1)
  int32_t rows;        // q_len * group: M rows of one work item (token-major)
  int32_t hq_all;      // q_len * h_q: outputs per sequence
  float scale_log2;    // scale * log2(e): scores are kept in log2 units
  DecodeWorkspace ws;
  uint32_t* error_word;
  // new rows written by the call itself (tl_paged_attn_decode_write; n_new 0
  // otherwise): the plan launch's extra CTAs scatter them into the pools
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  void* k_dst;
  void* v_dst;
  int32_t n_new;
  int32_t new_kind;   // 0 copy (same dtype), 1 e4m3 codes of bf16 rows, 2 of f32 rows,
                      // 3 int8 codes and scales of bf16 rows, 4 of f32 rows
  int32_t row_units;  // 16-byte vectors (copy) or 8-element steps (e4m3) of one row
  // int8 pools: the per-(slot, KV head) scales, [num_pages][H_kv][page_size]
  const float* k_scales;
  const float* v_scales;
};

// Logical block of key j and its offset in the page (a shift and a mask for
// power-of-two page sizes: a division by a runtime value costs dozens of
// dependent instructions, and the producer computes several per chunk).
__device__ __forceinline__ int page_of(const DecodeParams& P, int j) {
  return P.ps_shift >= 0 ? j >> P.ps_shift : j / P.page_size;
}
__device__ __forceinline__ int in_page(const DecodeParams& P, int j) {
  return P.ps_shift >= 0 ? j & (P.page_size - 1) : j % P.page_size;
}

// Block-table entry of logical block blk of sequence b.  With a ring
// ("How serving works in Tlaloc", section 3, windowed KV pool) logical block
// blk lives on ring page blk % ring_pages, so keys keep their position order
// and a ring gives the same bits as a full-history table.
__device__ __forceinline__ int32_t table_entry(const DecodeParams& P, int b, int blk) {
  const int e = P.ring_pages > 0 ? blk % P.ring_pages : blk;
  return __ldg(P.block_table + (size_t)b * P.max_pages_per_seq + e);
}

// Key range of sequence b: lo..p, the union over its q_len queries (the last
// at position p = L - 1, the first at L - q_len); empty when L <= 0 or L is
// past the table.
__device__ __forceinline__ void seq_range(const DecodeParams& P, int b, int& lo, int& p,
                                          bool report_errors) {
  const int L = P.context_lens[b];
  const int64_t cap = (int64_t)P.max_pages_per_seq * P.page_size;
  p = L - 1;
  if (P.ring_pages == 0 && L > cap) {  // a ring's positions are not bounded by its width
    if (report_errors) report(P.error_word, TL_DEVERR_CONTEXT_RANGE);
    p = -1;
  }
  const int first = p - (P.q_len - 1);
  lo = (P.window > 0 && first - P.window + 1 > 0) ? first - P.window + 1 : 0;
}

__device__ __forceinline__ int seq_chunks(const DecodeParams& P, int b, bool report_errors) {
  int lo, p;
  seq_range(P, b, lo, p, report_errors);
  return p < 0 ? 0 : p / kChunk - lo / kChunk + 1;
}

// ------------------------------------------------------------------ plan --
//
// Work items are pieces of a sequence's chunk range (times the KV heads),
// taken by the warps in item order from an atomic counter.  The order ends
// with a round of small pieces: the last ~15% of every sequence longer than
// 2 * kMinSplitChunks chunks is cut into pieces of kSmallChunks (or more, to
// stay in the split budget), and those pieces come after every bulk piece.
// The warps that finish their last bulk piece early then take the small
// ones, so they all run out of work within about one small piece of each
// other.  A piece's partial index keeps a sequence's pieces contiguous for
// the merge whatever their place in the order.

// Build knobs, measured side by side on GB300 with the 6,144-item target:
// small pieces of 2, 4 or 8 chunks time within 0.3% on every decode line;
// a 15% tail beats 8% (the step 0.2007 ms against 0.1955, e4m3 0.125
// against 0.113) and 25% (0.1969).
#ifndef TL_DECODE_SMALL_CHUNKS
#define TL_DECODE_SMALL_CHUNKS 4
#endif
#ifndef TL_DECODE_TAIL_PCT
#define TL_DECODE_TAIL_PCT 15
#endif
constexpr int kSmallChunks = TL_DECODE_SMALL_CHUNKS;  // chunks per small piece (4: 64 keys)
constexpr int kTailPct = TL_DECODE_TAIL_PCT;          // share of a sequence in small pieces

__device__ __forceinline__ int tail_chunks(int n) {
  return n < 2 * kMinSplitChunks ? 0 : min(n, (kTailPct * n + 99) / 100);
}

// Sums of two values over the block (every thread gets them); red holds one
// slot per warp for each.
__device__ __forceinline__ void block_sum2(long long& x, long long& y, long long (*red)[32]) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
  }
  if (lane == 0) {
    red[0][wid] = x;
    red[1][wid] = y;
  }
  __syncthreads();
  x = lane < nw ? red[0][lane] : 0;
  y = lane < nw ? red[1][lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
  }
  __syncthreads();  // red is reused by the next call
}

// Exclusive scan of x over the block in thread order; total gets the sum.
__device__ __forceinline__ long long block_excl_scan(long long x, long long* tmp,
                                                     long long& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) tmp[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    long long v = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    tmp[lane] = v;
  }
  __syncthreads();
  const long long before = (wid > 0 ? tmp[wid - 1] : 0) + inc - x;
  total = tmp[nw - 1];
  __syncthreads();
  return before;
}

// Sum of x over the warp (every lane gets it).
__device__ __forceinline__ long long warp_sum64(long long x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Descriptors of one round of nseq sequences (base .. base + nseq - 1):
// rec[j] = {first bulk piece, first small piece, bulk pieces, small pieces}
// of sequence base + j, rng[j] = its {lo, p}.  Thread i writes the round's
// pieces i, i + nthreads, ...: bulk pieces bulk0 .. bulk0 + nb - 1 (at
// [bulk0, ...)), then small pieces small0 .. small0 + ns - 1 (at NB + ...);
// a piece's sequence is the last one whose first piece of that kind is at or
// before it (a binary search of rec).  Each piece also asks L2 for the
// block-table entries its first chunk reads, so the attention kernel's
// first table load of the item hits.
__device__ __forceinline__ void write_piece_descs(const DecodeParams& P, const int4* rec,
                                                  const int2* rng, int base, int nseq, int bulk0,
                                                  int nb, int small0, int ns, int NB, int split,
                                                  int small, int i, int nthreads) {
  for (; i < nb + ns; i += nthreads) {
    const bool bulk = i < nb;
    const int pidx = bulk ? bulk0 + i : small0 + (i - nb);
    int lo_s = 0, hi_s = nseq;
    while (lo_s < hi_s) {
      const int mid = (lo_s + hi_s) >> 1;
      const int st = bulk ? rec[mid].x : rec[mid].y;
      if (st <= pidx) lo_s = mid + 1;
      else hi_s = mid;
    }
    const int j = lo_s - 1;
    const int4 r = rec[j];
    const int lo_j = rng[j].x, p_j = rng[j].y, bj = base + j;
    const int n_j = p_j < 0 ? 0 : p_j / kChunk - lo_j / kChunk + 1;
    const int c0 = lo_j / kChunk, c1 = c0 + n_j, cm = c1 - tail_chunks(n_j);
    const int first = r.x + r.y, pieces = r.z + r.w;
    int cb, ce, slot, part;
    if (bulk) {
      const int k = pidx - r.x;
      cb = c0 + k * split;
      ce = min(cm, cb + split);
      slot = pidx;
      part = first + k;
    } else {
      const int k = pidx - r.y;
      cb = cm + k * small;
      ce = min(c1, cb + small);
      slot = NB + pidx;
      part = first + r.z + k;
    }
    P.ws.desc[2 * slot] = make_int4(bj, cb, ce, pieces);
    P.ws.desc[2 * slot + 1] = make_int4(lo_j, p_j, part, 0);
    const int blk = page_of(P, cb * kChunk);
    const int e = P.ring_pages > 0 ? blk % P.ring_pages : blk;
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(P.block_table + (size_t)bj * P.max_pages_per_seq + e));
  }
}

// Batches of at most kWarpPlanMax sequences: every thread reads one
// sequence's range into shared memory, then warp 0 plans alone: lane l takes
// sequences l*K .. l*K + K - 1 (K = ceil(B / 32)), the sums are warp
// shuffles and the placement one warp scan of the lanes' (bulk << 32 | small)
// piece counts, with no block barrier between the steps.  Same arithmetic,
// same pieces as the block-wide path.  The loops stay rolled: the plan runs
// once per call from a cold instruction cache, where straight-line code costs
// more than the loop overhead.
constexpr int kWarpPlanMax = 128;
constexpr int kWriteWarps = 8;  // writing warps per CTA of a warp-planned launch

// One CTA.  Up to kWarpPlanMax sequences: warp 0 plans alone (above).
// Larger batches: thread t keeps sequence t's range in registers (sequences
// past the block size are re-read in each pass); three block reductions fix
// the piece sizes, and one scan of (bulk pieces << 32 | small pieces) places
// every piece.  Either way every thread then writes descriptors, one piece
// at a time.  first_dynamic: items below it are taken without the counter
// (the attention kernel's warp w starts with item w).
__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeParams P, int target_splits,
                                                           int first_dynamic) {
  __shared__ long long red[2][32];
  __shared__ long long tmp[32];
  __shared__ int4 rec[1024];  // per sequence of a round: first bulk / small position, counts
  __shared__ int2 rng[1024];  // its lo, p
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
  if (blockIdx.x == 0 && tid == 0) TL_TRACE_SET(TL_TRACE_PLAN_START);
  // the attention kernel may launch now: it waits for this grid's results
  // (griddepcontrol.wait) after its own set-up
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  if (blockIdx.x > 0) {
    // CTAs past the first write the call's new rows: one warp per token (per
    // token and KV head for int8 pools), slot -1 skipped, a slot outside the
    // pools reported and skipped
    // a block enlarged for the warp plan writes with kWriteWarps of its
    // warps, so the rows still spread over as many SMs
    const int wpc = P.B <= kWarpPlanMax ? min(nw, kWriteWarps) : nw;
    if (wid >= wpc) return;
    const int64_t first = (int64_t)(blockIdx.x - 1) * wpc + wid;
    const int64_t stride = (int64_t)(gridDim.x - 1) * wpc;
    const int64_t n_slots = (int64_t)P.num_pages * P.page_size;
    if (P.new_kind >= 3) {
      // int8 pools: one warp per (token, KV head) row; the scales written
      // here are read by the attention kernel after this grid
      for (int64_t r = first; r < (int64_t)P.n_new * P.h_kv; r += stride) {
        const int64_t t = r / P.h_kv;
        const int g = (int)(r % P.h_kv);
        const int64_t slot = P.slot_mapping[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= n_slots) {
          if (lane == 0 && g == 0) report(P.error_word, TL_DEVERR_SLOT_RANGE);
          continue;
        }
        int8_t* kd = static_cast<int8_t*>(P.k_dst);
        int8_t* vd = static_cast<int8_t*>(P.v_dst);
        float* ksc = const_cast<float*>(P.k_scales);
        float* vsc = const_cast<float*>(P.v_scales);
        if (P.d == 128) {
          if (P.new_kind == 3)
            write_head_rows_int8_d128<false>(P.k_new, P.v_new, kd, vd, ksc, vsc, t, g, slot,
                                             P.page_size, P.h_kv, lane, P.error_word);
          else
            write_head_rows_int8_d128<true>(P.k_new, P.v_new, kd, vd, ksc, vsc, t, g, slot,
                                            P.page_size, P.h_kv, lane, P.error_word);
        } else if (P.new_kind == 3) {
          write_head_rows_int8<false>(P.k_new, P.v_new, kd, vd, ksc, vsc, t, g, slot,
                                      P.page_size, P.h_kv, P.d, lane, P.error_word);
        } else {
          write_head_rows_int8<true>(P.k_new, P.v_new, kd, vd, ksc, vsc, t, g, slot,
                                     P.page_size, P.h_kv, P.d, lane, P.error_word);
        }
      }
      return;
    }
    // rows of 32 x 1, 2, 4 (or 8) units: every load before any store
    const int u = P.row_units;
    const int upl = u % 32 == 0 ? u / 32 : 0;
    if (P.new_kind == 0 && (upl == 1 || upl == 2 || upl == 4 || upl == 8)) {
      const int4* kn = static_cast<const int4*>(P.k_new);
      const int4* vn = static_cast<const int4*>(P.v_new);
      int4* kd = static_cast<int4*>(P.k_dst);
      int4* vd = static_cast<int4*>(P.v_dst);
      for (int64_t t = first; t < P.n_new; t += stride) {
        if (upl == 1) write_tokens_vec<1, 1>(kn, vn, kd, vd, P.slot_mapping, t, P.n_new, n_slots, lane, P.error_word);
        else if (upl == 2) write_tokens_vec<2, 1>(kn, vn, kd, vd, P.slot_mapping, t, P.n_new, n_slots, lane, P.error_word);
        else if (upl == 4) write_tokens_vec<4, 1>(kn, vn, kd, vd, P.slot_mapping, t, P.n_new, n_slots, lane, P.error_word);
        else write_tokens_vec<8, 1>(kn, vn, kd, vd, P.slot_mapping, t, P.n_new, n_slots, lane, P.error_word);
      }
      return;
    }
    if ((P.new_kind == 1 || P.new_kind == 2) && (upl == 1 || upl == 2 || upl == 4)) {
      uint2* kd = static_cast<uint2*>(P.k_dst);
      uint2* vd = static_cast<uint2*>(P.v_dst);
      for (int64_t t = first; t < P.n_new; t += stride) {
#define TL_E4M3_VEC(F32, U) \
  write_tokens_e4m3_vec<F32, U, 1>(P.k_new, P.v_new, kd, vd, P.slot_mapping, t, P.n_new, n_slots, lane, P.error_word)
        if (P.new_kind == 1) {
          if (upl == 1) TL_E4M3_VEC(false, 1);
          else if (upl == 2) TL_E4M3_VEC(false, 2);
          else TL_E4M3_VEC(false, 4);
        } else {
          if (upl == 1) TL_E4M3_VEC(true, 1);
          else if (upl == 2) TL_E4M3_VEC(true, 2);
          else TL_E4M3_VEC(true, 4);
        }
#undef TL_E4M3_VEC
      }
      return;
    }
    for (int64_t t = first; t < P.n_new; t += stride) {
      const int64_t slot = P.slot_mapping[t];
      if (slot == -1) continue;
      if (slot < 0 || slot >= n_slots) {
        if (lane == 0) report(P.error_word, TL_DEVERR_SLOT_RANGE);
        continue;
      }
      if (P.new_kind == 0)
        write_token_rows(static_cast<const int4*>(P.k_new) + t * u,
                         static_cast<const int4*>(P.v_new) + t * u,
                         static_cast<int4*>(P.k_dst) + slot * u,
                         static_cast<int4*>(P.v_dst) + slot * u, u, lane);
      else if (P.new_kind == 1)
        write_token_rows_e4m3<false>(P.k_new, P.v_new, static_cast<uint2*>(P.k_dst),
                                     static_cast<uint2*>(P.v_dst), t, slot, u, lane);
      else
        write_token_rows_e4m3<true>(P.k_new, P.v_new, static_cast<uint2*>(P.k_dst),
                                    static_cast<uint2*>(P.v_dst), t, slot, u, lane);
    }
    return;
  }
  if (P.B <= kWarpPlanMax) {
    __shared__ int s_plan[4];  // split, small, bulk pieces (-1: refused), small pieces
    if (tid < P.B) {  // the block holds at least B threads
      int lo, p;
      seq_range(P, tid, lo, p, true);
      rng[tid] = make_int2(lo, p);
    }
    __syncthreads();
    if (wid == 0) {
      const int K = (P.B + 31) >> 5, b0 = min(lane * K, P.B), b1 = min(b0 + K, P.B);
      long long C = 0, T = 0;
#pragma unroll 1
      for (int b = b0; b < b1; ++b) {
        const int n = rng[b].y < 0 ? 0 : rng[b].y / kChunk - rng[b].x / kChunk + 1;
        C += n;
        T += tail_chunks(n);
      }
      C = warp_sum64(C);
      T = warp_sum64(T);
      const long long half = max(target_splits / 2, 1);
      const int small = (int)max((long long)kSmallChunks, (T + P.B + half - 1) / half);
      long long TP = 0;
#pragma unroll 1
      for (int b = b0; b < b1; ++b) {
        const int n = rng[b].y < 0 ? 0 : rng[b].y / kChunk - rng[b].x / kChunk + 1;
        TP += (tail_chunks(n) + small - 1) / small;
      }
      TP = warp_sum64(TP);
      const long long budget = (long long)target_splits + P.B - TP;
      const long long sb = (C - T + budget - 1) / budget;
      const int split = (int)(sb < kMinSplitChunks ? kMinSplitChunks : sb);
      long long x = 0;  // this lane's (bulk << 32 | small) pieces
#pragma unroll 1
      for (int b = b0; b < b1; ++b) {
        const int n = rng[b].y < 0 ? 0 : rng[b].y / kChunk - rng[b].x / kChunk + 1;
        const int t = tail_chunks(n);
        x += ((long long)((n - t + split - 1) / split) << 32) | ((t + small - 1) / small);
      }
      long long inc = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      const long long tot = __shfl_sync(0xffffffffu, inc, 31);
      const int NB = (int)(tot >> 32), NS = (int)(tot & 0xffffffffll);
      if (NB + NS > decode_max_splits(P.B, P.h_kv)) {
        // past the workspace's bound (see the block-wide path): refused
        for (int b = lane; b <= P.B; b += 32) P.ws.split_off[b] = 0;
        if (lane == 0) {
          report(P.error_word, TL_DEVERR_PLAN_CAPACITY);
          P.ws.ctrl[0] = split;
          P.ws.ctrl[1] = 0;
          P.ws.ctrl[2] = first_dynamic;
          s_plan[2] = -1;
        }
      } else {
        long long pos = inc - x;
#pragma unroll 1
        for (int b = b0; b < b1; ++b) {
          const int n = rng[b].y < 0 ? 0 : rng[b].y / kChunk - rng[b].x / kChunk + 1;
          const int t = tail_chunks(n);
          const int nb = (n - t + split - 1) / split, ntl = (t + small - 1) / small;
          const int pos_b = (int)(pos >> 32), pos_t = (int)(pos & 0xffffffffll);
          P.ws.split_off[b] = pos_b + pos_t;
          rec[b] = make_int4(pos_b, pos_t, nb, ntl);
          pos += ((long long)nb << 32) | ntl;
        }
        if (lane == 0) {
          P.ws.split_off[P.B] = NB + NS;
          P.ws.ctrl[0] = split;
          P.ws.ctrl[1] = NB + NS;
          P.ws.ctrl[2] = first_dynamic;
          s_plan[0] = split;
          s_plan[1] = small;
          s_plan[2] = NB;
          s_plan[3] = NS;
        }
      }
    }
    __syncthreads();
    if (s_plan[2] < 0) return;
    if (tid == 0) TL_TRACE_SET(TL_TRACE_PLAN_PLACED);
    write_piece_descs(P, rec, rng, 0, P.B, 0, s_plan[2], 0, s_plan[3], s_plan[2], s_plan[0],
                      s_plan[1], tid, nt);
#if TL_DECODE_TRACE
    __syncthreads();
    if (tid == 0) TL_TRACE_SET(TL_TRACE_PLAN_END);
#endif
    return;
  }
  int lo0 = 0, p0 = -1, n0 = 0;  // sequence tid
  if (tid < P.B) {
    seq_range(P, tid, lo0, p0, true);
    n0 = p0 < 0 ? 0 : p0 / kChunk - lo0 / kChunk + 1;
  }
  // chunks of the batch and of the small-piece round
  long long C = tid < P.B ? n0 : 0, T = tail_chunks(n0);
  for (int b = tid + nt; b < P.B; b += nt) {
    const int n = seq_chunks(P, b, true);
    C += n;
    T += tail_chunks(n);
  }
  block_sum2(C, T, red);
  // small pieces: at most target/2 + B of them
  const long long half = max(target_splits / 2, 1);
  const int small = (int)max((long long)kSmallChunks, (T + P.B + half - 1) / half);
  long long TP = (tail_chunks(n0) + small - 1) / small, unused = 0;
  for (int b = tid + nt; b < P.B; b += nt) TP += (tail_chunks(seq_chunks(P, b, false)) + small - 1) / small;
  block_sum2(TP, unused, red);
  // bulk pieces: at most (target + B - TP) + B of them, so every piece fits
  // the target + 2B descriptors and partials the workspace holds
  const long long budget = (long long)target_splits + P.B - TP;
  const long long sb = (C - T + budget - 1) / budget;
  const int split = (int)(sb < kMinSplitChunks ? kMinSplitChunks : sb);
  long long NB = (n0 - tail_chunks(n0) + split - 1) / split;
  for (int b = tid + nt; b < P.B; b += nt) {
    const int n = seq_chunks(P, b, false);
    NB += (n - tail_chunks(n) + split - 1) / split;
  }
  block_sum2(NB, unused, red);
  // the workspace holds decode_max_splits(B, h_kv) descriptors and partials;
  // the two rounds above stay within it by construction, and a total past it
  // is refused here (nothing is attended, every output comes out 0)
  if (NB + TP > decode_max_splits(P.B, P.h_kv)) {
    for (int b = tid; b <= P.B; b += nt) P.ws.split_off[b] = 0;
    if (tid == 0) {
      report(P.error_word, TL_DEVERR_PLAN_CAPACITY);
      P.ws.ctrl[0] = split;
      P.ws.ctrl[1] = 0;
      P.ws.ctrl[2] = first_dynamic;
    }
    return;
  }
  // descriptors: bulk pieces at [0, NB) and small pieces at [NB, NB + TP) in
  // sequence order; partial indices split_off[b] + k, bulk pieces first
  long long carry = 0;  // (bulk << 32) | small pieces before this round of sequences
  for (int base = 0; base < P.B; base += nt) {
    const int b = base + tid;
    int lo = lo0, p = p0, n = n0;
    if (base > 0) {
      lo = 0; p = -1; n = 0;
      if (b < P.B) {
        seq_range(P, b, lo, p, false);
        n = p < 0 ? 0 : p / kChunk - lo / kChunk + 1;
      }
    } else if (b >= P.B) {
      n = 0;
    }
    const int t = tail_chunks(n);
    const int nb = (n - t + split - 1) / split, ntl = (t + small - 1) / small;
    long long tot;
    const long long pos = carry + block_excl_scan(((long long)nb << 32) | ntl, tmp, tot);
    if (b < P.B) {
      const int pos_b = (int)(pos >> 32), pos_t = (int)(pos & 0xffffffffll);
      P.ws.split_off[b] = pos_b + pos_t;  // partial index of the sequence's first piece
      rec[tid] = make_int4(pos_b, pos_t, nb, ntl);
      rng[tid] = make_int2(lo, p);
    }
    __syncthreads();
    write_piece_descs(P, rec, rng, base, min(nt, P.B - base), (int)(carry >> 32),
                      (int)(tot >> 32), (int)(carry & 0xffffffffll), (int)(tot & 0xffffffffll),
                      (int)NB, split, small, tid, nt);
    __syncthreads();  // rec and rng are rewritten by the next round
    carry += tot;
  }
  if (tid == 0) {
    const int total = (int)(carry >> 32) + (int)(carry & 0xffffffffll);
    P.ws.split_off[P.B] = total;
    P.ws.ctrl[0] = split;
    P.ws.ctrl[1] = total;
    P.ws.ctrl[2] = first_dynamic;
    TL_TRACE_SET(TL_TRACE_PLAN_END);  // after the last round's barrier
  }
}

struct ItemInfo {
  int b, g, lo, p, c_begin, c_end;  // chunks [c_begin, c_end)
  int s_global, nsplits;            // split index in the partial arrays; splits of b
};

// Piece descriptor written by the plan kernel, in item order: {b, c_begin,
// c_end, pieces of b}, {lo, p, partial index, 0}.
__device__ __forceinline__ void describe_item(const DecodeParams& P, int item, ItemInfo& it) {
  const int s = item / P.h_kv;
  const int4 d0 = __ldcg(P.ws.desc + 2 * s), d1 = __ldcg(P.ws.desc + 2 * s + 1);
  it.g = item - s * P.h_kv;
  it.b = d0.x;
  it.c_begin = d0.y;
  it.c_end = d0.z;
  it.nsplits = d0.w;
  it.lo = d1.x;
  it.p = d1.y;
  it.s_global = d1.z;
}

// ------------------------------------------------------ bf16 decode kernel --
//
// Persistent, one CTA per SM, every warp independent (no CTA barrier after
// set-up).  A warp owns whole work items (piece x KV head), taken from an
// atomic counter, and streams their 16-key chunks through a private ring of
// shared-memory stages (one chunk per stage, two for one-byte pools): one
// lane per box issues the stage's tiled TMA boxes (a 3-D tensor map of the
// pool (d, H_kv, slot), boxes of 8 or 16 rows = one page run, 4 boxes per
// 8 KiB stage at page size 16) completing on the stage's mbarrier by
// transaction bytes, all but one stage ahead of the one the warp computes.  The
// stream runs across item boundaries: the next item's descriptor and
// block-table window are fetched during the current item's last kGrabLead
// stages, and each item's Q rows arrive by a bulk copy into one of the ring's
// Q slots.  Stage layout: the stage's K chunks then its V chunks, each as
// [row half (64 elements = 128 B)][16 rows][128 B] in the
// TMA 128-byte swizzle (16-byte unit u of row r at unit u ^ (r & 7), so
// ldmatrix reads of 8 rows hit 8 different bank groups).  A box of a block
// past the sequence's last page, or of a bad page, gets an out-of-range slot
// and arrives as zeros; V rows past the last position in the last page are
// zeroed before use (they may hold anything).  At the end of an item the
// warp writes the output (one split) or a partial straight from its
// registers.

constexpr int kGrabLead = 4;  // stages left to issue when a warp starts fetching its next item

// Warps per CTA and stages per warp of a kernel variant.  The one-byte
// kernels with at most 8 rows (keys as the MMA's rows) fit 168 registers:
// 12 warps (three per SMSP) with 2-stage rings, one 8 KiB stage in flight
// per warp (measured on the 64-sequence Llama-3-8B layer over e4m3 pools:
// 0.1335 ms per step with 8 warps x 3 stages, 0.1196 ms with 12 x 2).  The
// others take up to 235 registers: 8 warps (two per SMSP).  With more than
// 8 rows a Q slot is 4 KiB and three stages would leave room for 6 warps:
// two stages keep 8 (the 4-token verify batch: 0.2605 ms per call with
// 6 x 3, 0.2369 ms with 8 x 2); with at most 8 rows three stages fit 7-8
// warps and time within 1% of two.
template <bool TWO_ROWS, bool KV8>
struct DecodeShape {
  static constexpr bool kKeysAsRows = KV8 && !TWO_ROWS;
  static constexpr int kWarps = kKeysAsRows ? 12 : 8;
  static constexpr int kRing = (kKeysAsRows || TWO_ROWS) ? 2 : 3;
};

// Per-warp shared memory: RING stages of kCps chunks of K and V as the TMA
// lands them (16-bit or one-byte elements, rows split in 128-byte parts; a
// one-byte stage holds two chunks, the same 8 KiB as one 16-bit chunk, so
// each stage's issue and wait serve 32 keys) and RING Q slots.
template <int D, bool KV8, bool I8, int RING>
struct WarpSmem {
  static constexpr int kRing = RING;                      // stages (and Q slots) per warp
  static constexpr int kCps = KV8 ? 2 : 1;                 // chunks per stage
  static constexpr int kRowBytes = D * (KV8 ? 1 : 2);
  static constexpr int kHalves = kRowBytes / 128;          // 128-byte parts of a row
  static constexpr int kHalfBytes = kChunk * 128;          // 16 rows of one part
  static constexpr int kChunkBytes = kHalves * kHalfBytes;  // one of K or V
  static constexpr int kStageBytes = 2 * kCps * kChunkBytes;  // K chunks, then V chunks
  // int8 pools: a stage's key scales, [K, V][chunk][16] f32, in static
  // shared memory (kept out of the 1 KiB-aligned per-warp area)
  static constexpr int kScaleBytes = I8 ? 2 * kCps * kChunk * 4 : 0;
  __host__ __device__ static int qslot_bytes(int rows) {
    return (rows * D * 2 + 1023) / 1024 * 1024;
  }
  __host__ __device__ static int warp_bytes(int rows) {
    return kRing * (kStageBytes + qslot_bytes(rows));
  }
};

// m16n8k16 with f32 accumulation on bf16 or fp16 operands.
template <bool F16>
__device__ __forceinline__ void mma_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if (F16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    mma_bf16_16816(c, a0, a1, a2, a3, b0, b1);
}

// (a, b) ~ hi + lo as fp16 pairs (about 22 significant bits together).
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(hi) : "f"(b), "f"(a));
  float ah, bh;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
      : "=f"(ah), "=f"(bh)
      : "r"(hi));
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(lo) : "f"(b - bh), "f"(a - ah));
}

template <bool F16>
__device__ __forceinline__ void split16(float a, float b, uint32_t& hi, uint32_t& lo) {
  if (F16)
    split_f16x2(a, b, hi, lo);
  else
    split_bf16x2(a, b, hi, lo);
}

// An 8 x 8 matrix of 16-bit elements held as m8n8 fragments (lane 4g + t:
// row g, columns 2t and 2t + 1 in the low and high halves) transposed
// across the warp: lane 4g + t gets row g of the transpose.
__device__ __forceinline__ uint32_t transpose_m8n8_b16(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(r) : "r"(x));
  return r;
}

// One bf16 pair as an fp16 pair (queries against an e4m3 pool; finite
// values beyond +-65504 become infinite).
__device__ __forceinline__ uint32_t bf16x2_as_f16x2(uint32_t x) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n"
      : "=r"(r)
      : "f"(__uint_as_float(x & 0xffff0000u)), "f"(__uint_as_float(x << 16)));
  return r;
}

// True when a finite bf16 element of the pair x became infinite in the fp16
// pair h (|x| > 65504).
__device__ __forceinline__ bool f16_overflowed(uint32_t x, uint32_t h) {
  const bool lo = ((x >> 7) & 0xffu) != 0xffu && (h & 0x7fffu) == 0x7c00u;
  const bool hi = ((x >> 23) & 0xffu) != 0xffu && ((h >> 16) & 0x7fffu) == 0x7c00u;
  return lo || hi;
}

// Four e4m3 codes (one 32-bit register, low byte first) as two fp16 pairs:
// codes 0,1 in lo and 2,3 in hi; exact.  The register's halves feed the two
// conversions directly.
__device__ __forceinline__ void e4m3x4_as_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n"
      " cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}


// a compile-time int for generic lambdas
template <int N>
struct IntC {
  static constexpr int value = N;
};

// Four int8 codes (one 32-bit register, low byte first) as two fp16 pairs:
// codes 0,1 in lo and 2,3 in hi; exact.  A code c + 128 as the low byte
// under the high byte 0x64 is the fp16 1024 + c + 128, so one packed
// subtraction of 1152 leaves c.
__device__ __forceinline__ void i8x4_as_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140u);
  hi = __byte_perm(u, 0x64646464u, 0x4342u);
  asm("sub.rn.f16x2 %0, %0, %1;\n" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;\n" : "+r"(hi) : "r"(0x64806480u));
}
// The two halves of an fp16 pair as floats (exact).
__device__ __forceinline__ void f16x2_to_floats(uint32_t x, float& lo, float& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
      : "=f"(lo), "=f"(hi)
      : "r"(x));
}
// The same without the subtraction: each value is 1152 + c, exact.  The
// int8 keys-as-rows path widens K this way and takes 1152 x (the query row's
// sum) out of each dot product before the K scale, one add per score instead
// of two packed subtractions per four codes.
__device__ __forceinline__ void i8x4_as_f16x2x2_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140u);
  hi = __byte_perm(u, 0x64646464u, 0x4342u);
}
// The same for a transposed pair of code pairs (bytes: key k codes c, c+1;
// key k+1 codes c, c+1): lo = (key k, key k+1) at code c, hi at code c+1.
__device__ __forceinline__ void i8x4_keys_as_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4240u);
  hi = __byte_perm(u, 0x64646464u, 0x4341u);
  asm("sub.rn.f16x2 %0, %0, %1;\n" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;\n" : "+r"(hi) : "r"(0x64806480u));
}

struct ItemSlot {
  int b, g, lo, p, c_begin, c_end, s_global, nsplits;
};

template <int NW, int R>
struct WarpShared {
  unsigned long long full[NW][R], qfull[NW][R];
  uint32_t stage_mask[NW][R];
  ItemSlot slot[NW][R];
  int abort_flag;
};

template <int D, bool TWO_ROWS, bool KV8, bool I8 = false>
__global__ void __launch_bounds__(DecodeShape<TWO_ROWS, KV8>::kWarps * 32, 1)
    decode_bf16_kernel(DecodeParams P, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, int box_rows) {
  static_assert(!I8 || KV8, "int8 pools take the one-byte path");
  using S = DecodeShape<TWO_ROWS, KV8>;
  using L = WarpSmem<D, KV8, I8, S::kRing>;
  constexpr int R = L::kRing;  // stages per warp
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ WarpShared<S::kWarps, R> sh;
  __shared__ __align__(128) unsigned char scale_sm[I8 ? S::kWarps * R * L::kScaleBytes : 16];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t sbase0 = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* smem0 = smem_raw + (sbase0 - smem_u32(smem_raw));
  volatile int* abort_flag = &sh.abort_flag;
  if (threadIdx.x == 0) sh.abort_flag = 0;
  if (threadIdx.x == 32) {  // the pools' tensor maps into the descriptor cache
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
  }
  if (lane == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(smem_u32(&sh.full[w][i]), 1);
      mbar_init(smem_u32(&sh.qfull[w][i]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // launched as a programmatic dependent of the plan kernel: its results
  // (work counter, descriptors, offsets) are read only after this wait
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (blockIdx.x == 0 && threadIdx.x == 0) TL_TRACE_SET(TL_TRACE_ATTN_RELEASED);
  // the combine kernel may launch now (it too waits for this grid's results)
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int qslot = L::qslot_bytes(P.rows);
  const uint64_t kv_policy = l2_evict_first();
  const uint32_t ring = sbase0 + w * L::warp_bytes(P.rows);
  // int8 pools: the stages' scales
  const uint32_t scale_ring = smem_u32(scale_sm) + w * R * L::kScaleBytes;
  const uint32_t qbase = ring + R * L::kStageBytes;
  const unsigned char* qbase_ptr = smem0 + (qbase - sbase0);
  const int total_items = __ldcg(P.ws.ctrl + 1) * P.h_kv;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(P.q);
  const int n_slots = P.num_pages * P.page_size;
  constexpr int CPS = L::kCps;
  // chunks of a stage that share one softmax step: both of an e4m3 stage
  // when the group fits rows 0-7 (registers allow it there), else one
  constexpr int NJ = (KV8 && !TWO_ROWS) ? CPS : 1;
  static_assert(NJ == 1 || NJ == 2, "a stage holds one or two chunks");
  const int nbox = kChunk / box_rows;             // boxes per row half of a chunk
  const int per_kind = CPS * L::kHalves * nbox;   // boxes of K (or V) per stage
  const int nreq = 2 * per_kind;                  // TMA requests per stage
  const int rq_kind = lane / per_kind;            // lane's box: K or V,
  const int rq_rem = lane % per_kind;
  const int rq_sub = rq_rem / (L::kHalves * nbox);  // chunk of the stage,
  const int rq_rem2 = rq_rem % (L::kHalves * nbox);
  const int rq_half = rq_rem2 / nbox, rq_box = rq_rem2 % nbox;  // row part and rows
  const CUtensorMap* rq_map = rq_kind == 0 ? &kmap : &vmap;
  const bool one_page = P.page_size % kChunk == 0;

  // ---------------------------------------------------------- issue side
  // items: icur (being issued) and inext, fetched in three steps, one per
  // issued chunk, once icur has kGrabLead chunks left to issue: the atomic,
  // the descriptor, the block-table window.  Taking the next item this late
  // (instead of items ahead) keeps the warps' finishing times close.
  ItemInfo icur, inext;
  bool icur_live = false;
  int icur_last_blk = 0;
  int icur_c = 0, iwin_blk0 = 0, iwin = -1, nwin_blk0 = 0, nwin = -1;
  // the first item is the warp's index in the grid (the counter starts past
  // them); later ones come from the counter
  int grab = blockIdx.x * (blockDim.x >> 5) + w;
  int nstate = 1;  // 0 idle, 1 item id known, 2 descriptor loading, 3 ready, 4 no items left
  uint32_t gs_issue = 0;
  int items_issued = 0;
  auto fetch_step = [&]() {
    if (nstate == 0) {
      if (lane == 0) grab = atomicAdd(P.ws.ctrl + 2, 1);
      nstate = 1;
    } else if (nstate == 1) {
      const int id = __shfl_sync(0xffffffffu, grab, 0);
      if (id >= total_items) {
        nstate = 4;
      } else {
        describe_item(P, id, inext);
        nstate = 2;
      }
    } else if (nstate == 2) {
      nwin_blk0 = page_of(P, inext.c_begin * kChunk);
      const int blk = nwin_blk0 + lane;
      nwin = blk <= page_of(P, inext.p) ? table_entry(P, inext.b, blk) : -1;
      nstate = 3;
    }
  };
  // the first item's descriptor loads alongside the item count (its piece
  // index is inside the workspace's descriptors whatever the count: the
  // grid's warps are fewer than the pieces target)
  if (grab / P.h_kv < decode_max_splits(P.B, P.h_kv)) {
    describe_item(P, grab, inext);
    nstate = grab >= total_items ? 4 : 2;
  }
  while (nstate < 3) fetch_step();

  // Start issuing the next item: publish its descriptor, copy its Q rows.
  // False when there is no item left.
  auto start_item = [&]() -> bool {
    while (nstate < 3) fetch_step();  // a fetch that started late completes here
    if (nstate == 4) return false;
    icur = inext;
    nstate = 0;
    icur_last_blk = page_of(P, icur.p);
    iwin_blk0 = nwin_blk0;
    iwin = nwin;
    icur_c = icur.c_begin;
    icur_live = true;
    const int q = items_issued % R;
    if (lane == 0) {
      ItemSlot& d = sh.slot[w][q];
      d.b = icur.b; d.g = icur.g; d.lo = icur.lo; d.p = icur.p;
      d.c_begin = icur.c_begin; d.c_end = icur.c_end;
      d.s_global = icur.s_global; d.nsplits = icur.nsplits;
      // the item's rows: the group's heads of each of the q_len tokens
      const uint32_t qbytes = (uint32_t)(P.group * D * 2);
      mbar_arrive_expect_tx(smem_u32(&sh.qfull[w][q]), qbytes * P.q_len);
      for (int t = 0; t < P.q_len; ++t)
        bulk_g2s(qbase + q * qslot + t * qbytes,
                 qg + (((size_t)icur.b * P.q_len + t) * P.h_q + (size_t)icur.g * P.group) * D,
                 qbytes, smem_u32(&sh.qfull[w][q]));
    }
    ++items_issued;
    return true;
  };

  // Issue the next stage of the stream: CPS chunks of the current item
  // (starting a new item when needed; a stage past the item's last chunk
  // reads zeros there and the compute side skips it).
  auto issue_next = [&]() {
    if (!icur_live && !start_item()) return;
    if (nstate < 3 && icur.c_end - icur_c <= kGrabLead * CPS) fetch_step();
    const int stage = (int)(gs_issue % R);
    const int j0 = icur_c * kChunk;
    const int last_blk = icur_last_blk;
    const int bmin = page_of(P, j0);
    const int bmax = min(page_of(P, j0 + CPS * kChunk - 1), last_blk);
    if (bmin < iwin_blk0 || bmax >= iwin_blk0 + 32) {  // the next 32 blocks
      iwin_blk0 = bmin;
      const int blk = iwin_blk0 + lane;
      iwin = blk <= last_blk
                 ? table_entry(P, icur.b, blk)
                 : -1;
    }
    uint32_t mask = 0u;  // live keys of the stage (16 bits per chunk)
    int slot0 = n_slots;  // first pool slot of this lane's box (n_slots: read as zeros)
    int64_t scale0 = 0;   // int8 pools: the lane's chunk's first scale (0: a stand-in)
    if (one_page) {
      // pages of a multiple of 16 keys: each chunk is one run of one page.
      // The stage's live keys are the range [lo, p] clipped to it; each
      // lane looks up the page of its own box's chunk, and chunks on a bad
      // page (any lane of that chunk sees it) are reported and read as zeros
      const int jm = j0 + rq_sub * kChunk;
      const int pr = __shfl_sync(0xffffffffu, iwin, (page_of(P, jm) - iwin_blk0) & 31);
      const int first = min(max(icur.lo - j0, 0), CPS * kChunk);
      const int last = min(icur.p - j0, CPS * kChunk - 1);
      mask = first <= last ? (0xffffffffu >> (31 - last)) & (0xffffffffu << first) : 0u;
      const bool page_ok = jm <= icur.p && pr >= 0 && pr < P.num_pages;
      const uint32_t sub_bits = 0xffffu << (16 * rq_sub);
      const uint32_t bad = __reduce_or_sync(0xffffffffu, (!page_ok && (mask & sub_bits)) ? sub_bits : 0u);
      if (bad != 0u) {
        if (lane == 0) report(P.error_word, TL_DEVERR_PAGE_RANGE);
        mask &= ~bad;
      }
      if (page_ok) {
        slot0 = pr * P.page_size + in_page(P, jm);
        if (I8) scale0 = ((int64_t)pr * P.h_kv + icur.g) * P.page_size + in_page(P, jm);
      }
    } else {
      const int jr = j0 + (CPS == 2 ? lane : (lane & 15));
      const int pr = __shfl_sync(0xffffffffu, iwin, (page_of(P, jr) - iwin_blk0) & 31);
      bool live = jr >= icur.lo && jr <= icur.p;
      if (live && (pr < 0 || pr >= P.num_pages)) {
        if (CPS == 2 || lane < 16) report(P.error_word, TL_DEVERR_PAGE_RANGE);
        live = false;
      }
      mask = __ballot_sync(0xffffffffu, live) & (CPS == 2 ? 0xffffffffu : 0xffffu);
      const int jb = j0 + rq_sub * kChunk + rq_box * box_rows;
      const int blk = page_of(P, jb);
      const int pb = __shfl_sync(0xffffffffu, iwin, (blk - iwin_blk0) & 31);
      const bool box_ok = jb <= icur.p && blk <= last_blk && pb >= 0 && pb < P.num_pages;
      if (box_ok) slot0 = pb * P.page_size + in_page(P, jb);
    }
    const uint32_t bar = smem_u32(&sh.full[w][stage]);
    if (lane == 0) {
      sh.stage_mask[w][stage] = mask;
      uint32_t tx = L::kStageBytes + L::kScaleBytes;
#ifdef TL_TEST_STALL_FIRST_STAGE
      // failure-path test build only: the first stage of warp 0 of CTA 0
      // expects 16 bytes that no copy delivers, so the wait for it runs out
      // (the copies it does issue all land before the CTA exits)
      if (blockIdx.x == 0 && w == 0 && gs_issue == 0) tx += 16;
#endif
      mbar_arrive_expect_tx(bar, tx);
    }
    // no warp barrier here: a box may land before lane 0's expectation (the
    // transaction count then runs negative), and the phase cannot complete
    // before lane 0 has arrived
    if (lane < nreq)  // the pools are read once per call: first out of L2
      tma_load_3d_hint(ring + stage * L::kStageBytes + (rq_kind * CPS + rq_sub) * L::kChunkBytes +
                           rq_half * L::kHalfBytes + rq_box * box_rows * 128,
                       rq_map, rq_half * (KV8 ? 128 : 64), icur.g, slot0, bar, kv_policy);
    if constexpr (I8) {
      // the stage's key scales: lanes nreq .. nreq + 2 CPS - 1 copy the 16
      // scales (64 bytes, contiguous within a page and head) of K, then V,
      // of chunk rq_sub; a chunk the item does not read copies a stand-in
      // (the pool's first 16 scales) so that the byte count always holds
      const int li = lane - nreq;
      if (li >= 0 && li < 2 * CPS)
        bulk_g2s(scale_ring + stage * L::kScaleBytes + (li / CPS * CPS + rq_sub) * kChunk * 4,
                 (li < CPS ? P.k_scales : P.v_scales) + scale0, kChunk * 4, bar);
    }
    ++gs_issue;
    icur_c += CPS;
    if (icur_c >= icur.c_end) icur_live = false;
  };

  for (int t = 0; t < R - 1; ++t) issue_next();

  // -------------------------------------------------------- compute side
  const int qr = lane >> 2, qc = (lane & 3) * 2;
  // One-byte pools with at most 8 rows take the keys as the MMA's rows:
  // S^T = K Q^T (16 keys x 8 columns) and O^T += V^T P^T (16 d x 8 columns),
  // half the MMAs and half the accumulators of rows-as-rows.  Column c holds
  // row c; with at most 4 rows, columns 4-7 repeat rows 0-3 and carry the
  // low parts of P (dup).
  constexpr bool KT = S::kKeysAsRows;
  const bool dup = KT && P.rows <= 4;
  const int qrow = dup ? (qr & 3) : qr;  // the query row of this lane's B-operand column
  uint32_t gs_c = 0;
  int items_c = 0;
  bool stop = false;
  while (!stop && items_c < items_issued) {
    const int q = items_c % R;
    if (!mbar_wait(smem_u32(&sh.qfull[w][q]), (items_c / R) & 1, abort_flag)) break;
    const ItemSlot it = sh.slot[w][q];
    const unsigned char* qs = qbase_ptr + q * qslot;
    uint32_t qa[D / 16][4];
    bool q_over = false;  // a finite query element beyond fp16's range (e4m3 pools)
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      // K step ks covers d = 16ks .. 16ks+15.  16-bit pools: the A fragment's
      // columns (2t, 2t+1) and (2t+8, 2t+9) are those d.  e4m3 pools: they are
      // d = 16ks+4t+(0,1) and 16ks+4t+(2,3), the order in which a lane's one
      // 4-byte read of a K row lands (the same permutation of the summed d
      // on both operands leaves Q.K^T unchanged)
      const int e0 = ks * 16 + (KV8 ? 4 * (lane & 3) : qc);
      const int e2 = KV8 ? e0 + 2 : e0 + 8;
      qa[ks][0] =
          qrow < P.rows ? *reinterpret_cast<const uint32_t*>(qs + (qrow * D + e0) * 2) : 0u;
      qa[ks][2] =
          qrow < P.rows ? *reinterpret_cast<const uint32_t*>(qs + (qrow * D + e2) * 2) : 0u;
      if (TWO_ROWS) {
        qa[ks][1] = qr + 8 < P.rows
                        ? *reinterpret_cast<const uint32_t*>(qs + ((qr + 8) * D + e0) * 2)
                        : 0u;
        qa[ks][3] = qr + 8 < P.rows
                        ? *reinterpret_cast<const uint32_t*>(qs + ((qr + 8) * D + e2) * 2)
                        : 0u;
      } else {
        qa[ks][1] = 0u;
        qa[ks][3] = 0u;
      }
      if (KV8) {  // the tensor core takes fp16 for both operands here
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t h = bf16x2_as_f16x2(qa[ks][k]);
          q_over |= f16_overflowed(qa[ks][k], h);
          qa[ks][k] = h;
        }
      }
    }
    if (KV8 && __any_sync(0xffffffffu, q_over) && lane == 0)
      report(P.error_word, TL_DEVERR_VALUE_RANGE);
    __syncwarp();
    // int8 keys as rows: -1152 x the sum of the fp16 query values of the
    // lane's score columns 2t and 2t + 1 (the B fragments hold column g's
    // values at four d a K step; the sum over t completes a column)
    float kb0 = 0.f, kb1 = 0.f;
    if constexpr (I8 && KT) {
      float part = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
        for (int k = 0; k < 4; k += 2) {
          float x0, x1;
          f16x2_to_floats(qa[ks][k], x0, x1);
          part += x0 + x1;
        }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      kb0 = -1152.f * __shfl_sync(0xffffffffu, part, 8 * (lane & 3));
      kb1 = -1152.f * __shfl_sync(0xffffffffu, part, 8 * (lane & 3) + 4);
    }

    // rows-as-rows: o[n] is n-tile n of O (16 rows x 8 d); keys-as-rows:
    // o[j] is O^T for d = 16j .. 16j + 15 (16 d x 8 columns)
    constexpr int NO = KT ? D / 16 : D / 8;
    float o[NO][4];
#pragma unroll
    for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    // with several query tokens, each row has its own key range: row r is
    // token r / group, at position p - (q_len - 1 - r / group)
    // (keys-as-rows: the rows of columns 2t and 2t + 1)
    const int ra = KT ? (dup ? (qc & 3) : qc) : qr;
    const int rb = KT ? ra + 1 : qr + 8;
    const int pr0 = it.p - (P.q_len - 1 - ra / P.group);
    const int pr1 = it.p - (P.q_len - 1 - rb / P.group);
    const int lr0 = (P.window > 0 && pr0 - P.window + 1 > 0) ? pr0 - P.window + 1 : 0;
    const int lr1 = (P.window > 0 && pr1 - P.window + 1 > 0) ? pr1 - P.window + 1 : 0;
    for (int c0 = it.c_begin; c0 < it.c_end; c0 += CPS, ++gs_c) {
      issue_next();  // keeps R-1 stages in flight ahead of this one
      const int stage = (int)(gs_c % R);
      if (!mbar_wait(smem_u32(&sh.full[w][stage]), (gs_c / R) & 1, abort_flag)) {
        stop = true;
        break;
      }
      if (TL_DECODE_TRACE && gs_c == 0 && blockIdx.x == 0 && threadIdx.x == 0)
        TL_TRACE_SET(TL_TRACE_ATTN_FIRST_STAGE);
      const uint32_t smask = sh.stage_mask[w][stage];
      const int nlive = min(CPS, it.c_end - c0);  // the stage's chunks inside the item
#pragma unroll 1
    for (int sub0 = 0; sub0 < nlive; sub0 += NJ) {
      // chunks sub0 .. sub0+nj-1 of the stage share one softmax step; nj is a
      // compile-time count, so a full stage runs as straight-line code
      auto step = [&](auto nj_c) {
      constexpr int nj = decltype(nj_c)::value;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        if (j >= nj) break;
        // V rows past the sequence's end (its last chunk only) may hold anything
        const int c = c0 + sub0 + j;
        const uint32_t vaddr = ring + stage * L::kStageBytes + (CPS + sub0 + j) * L::kChunkBytes;
        const int first_dead = it.p + 1 - c * kChunk;
        if (first_dead < kChunk) {
          const int n_dead = kChunk - max(first_dead, 0);
          for (int idx = lane; idx < n_dead * L::kHalves * 8; idx += 32) {
            const int row = kChunk - n_dead + idx / (L::kHalves * 8);
            const int hu = idx % (L::kHalves * 8);
            const uint32_t a = vaddr + (hu >> 3) * L::kHalfBytes + row * 128 + ((hu & 7) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();  // these stores precede the stage's next TMA fill
          __syncwarp();
        }
      }
      if constexpr (KT) {
      // S^T = K Q^T per chunk: lane (g, t) gets the scores of keys g and
      // g + 8 in columns 2t and 2t + 1 (s[j] = {(2t, g), (2t+1, g), (2t, g+8),
      // (2t+1, g+8)}).  K's A fragments are the same widened codes as the B
      // fragments of rows-as-rows: key rows g and g + 8, d permuted as there.
      float s[NJ][4];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        if (j >= nj) continue;
        const uint32_t kaddr = ring + stage * L::kStageBytes + (sub0 + j) * L::kChunkBytes;
        float s2[4] = {0.f, 0.f, 0.f, 0.f};
        const int mi = lane >> 3, row = (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < D / 16; ks += 2) {
          const int u = ks + (mi >> 1);
          uint32_t w[4];
          ldmatrix_x4(kaddr + row * 128 + ((u ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t a0, a1, a2, a3;
            if constexpr (I8) {
              i8x4_as_f16x2x2_biased(w[2 * h], a0, a2);
              i8x4_as_f16x2x2_biased(w[2 * h + 1], a1, a3);
            } else {
              e4m3x4_as_f16x2x2(w[2 * h], a0, a2);
              e4m3x4_as_f16x2x2(w[2 * h + 1], a1, a3);
            }
            mma_16816<true>(h ? s2 : s[j], a0, a1, a2, a3, qa[ks + h][0], qa[ks + h][2]);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) s[j][e] += s2[e];
      }
      if constexpr (I8) {  // each key's dot products, less the bias, times its K scale
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          if (j >= nj) break;
          float k0, k1;
          const uint32_t sa = scale_ring + stage * L::kScaleBytes + ((sub0 + j) * kChunk + qr) * 4;
          asm volatile("ld.shared.f32 %0, [%1];\n" : "=f"(k0) : "r"(sa));
          asm volatile("ld.shared.f32 %0, [%1];\n" : "=f"(k1) : "r"(sa + 32));
          s[j][0] = (s[j][0] + kb0) * k0;
          s[j][1] = (s[j][1] + kb1) * k0;
          s[j][2] = (s[j][2] + kb0) * k1;
          s[j][3] = (s[j][3] + kb1) * k1;
        }
      }
      constexpr uint32_t all_keys = nj == 1 ? 0xffffu : 0xffffffffu;
      if (P.q_len == 1 && ((smask >> (16 * sub0)) & all_keys) == all_keys) {
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[j][e] = j < nj ? s[j][e] * P.scale_log2 : -INFINITY;
      } else {
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
          for (int hk = 0; hk < 2; ++hk) {
            const int key = qr + 8 * hk;
            const bool ok = j < nj && ((smask >> (16 * (sub0 + j) + key)) & 1u);
            bool ok0 = ok, ok1 = ok;
            if (P.q_len > 1) {
              const int kp = (c0 + sub0 + j) * kChunk + key;
              ok0 = ok && kp >= lr0 && kp <= pr0;
              ok1 = ok && kp >= lr1 && kp <= pr1;
            }
            s[j][2 * hk] = ok0 ? s[j][2 * hk] * P.scale_log2 : -INFINITY;
            s[j][2 * hk + 1] = ok1 ? s[j][2 * hk + 1] * P.scale_log2 : -INFINITY;
          }
      }
      // the lazy running max of rows-as-rows, per column (m0: 2t, m1: 2t + 1);
      // a column's keys span the 8 lanes of one t
      bool over = m0 == -INFINITY || m1 == -INFINITY;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
          over |= s[j][2 * hk] > m0 + kLazyLog2;
          over |= s[j][2 * hk + 1] > m1 + kLazyLog2;
        }
      float p[NJ][4];
      if (!__any_sync(0xffffffffu, over)) {
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          p[j][0] = fast_exp2(s[j][0] - m0);
          p[j][1] = fast_exp2(s[j][1] - m1);
          p[j][2] = fast_exp2(s[j][2] - m0);
          p[j][3] = fast_exp2(s[j][3] - m1);
          sum0 += p[j][0] + p[j][2];
          sum1 += p[j][1] + p[j][3];
        }
        l0 += sum0;
        l1 += sum1;
      } else {
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][2]));
          mx1 = fmaxf(mx1, fmaxf(s[j][1], s[j][3]));
        }
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
        }
        const float mn0 = (m0 == -INFINITY || mx0 > m0 + kLazyLog2) ? fmaxf(m0, mx0) : m0;
        const float mn1 = (m1 == -INFINITY || mx1 > m1 + kLazyLog2) ? fmaxf(m1, mx1) : m1;
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;  // no live key seen yet
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float f0 = fast_exp2(m0 - base0), f1 = fast_exp2(m1 - base1);
        m0 = mn0;
        m1 = mn1;
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          p[j][0] = fast_exp2(s[j][0] - base0);
          p[j][1] = fast_exp2(s[j][1] - base1);
          p[j][2] = fast_exp2(s[j][2] - base0);
          p[j][3] = fast_exp2(s[j][3] - base1);
          sum0 += p[j][0] + p[j][2];
          sum1 += p[j][1] + p[j][3];
        }
        l0 = l0 * f0 + sum0;
        l1 = l1 * f1 + sum1;
        if (__any_sync(0xffffffffu, f0 != 1.f || f1 != 1.f)) {
#pragma unroll
          for (int n = 0; n < NO; ++n) {
            o[n][0] *= f0;
            o[n][1] *= f1;
            o[n][2] *= f0;
            o[n][3] *= f1;
          }
        }
      }
#pragma unroll
      for (int jc = 0; jc < NJ; ++jc) {
        if (jc >= nj) break;
        const uint32_t vaddr =
            ring + stage * L::kStageBytes + (CPS + sub0 + jc) * L::kChunkBytes;
        if constexpr (I8) {  // each probability times its key's V scale
          float v0, v1;
          const uint32_t sa =
              scale_ring + stage * L::kScaleBytes + ((CPS + sub0 + jc) * kChunk + qr) * 4;
          asm volatile("ld.shared.f32 %0, [%1];\n" : "=f"(v0) : "r"(sa));
          asm volatile("ld.shared.f32 %0, [%1];\n" : "=f"(v1) : "r"(sa + 32));
          // a scale of a slot outside the live keys may be anything: bounded
          // to [0, 3e38] (NaN to 0), it leaves their p = 0 at 0
          v0 = fminf(fmaxf(v0, 0.f), 3.0e38f);
          v1 = fminf(fmaxf(v1, 0.f), 3.0e38f);
          p[jc][0] *= v0;
          p[jc][1] *= v0;
          p[jc][2] *= v1;
          p[jc][3] *= v1;
        }
        // P^T as the B operand: the fp16 pairs (columns 2t, 2t + 1) of keys g
        // and g + 8 form the 8 x 8 blocks P^T[keys 0-7] and P^T[keys 8-15];
        // their transposes give lane (g, t) keys 2t, 2t + 1 (and 2t + 8,
        // 2t + 9) of column g.  P = hi + lo (fp16 pair, ~22 significant bits):
        // with dup, columns 4-7 take the low parts; otherwise the low parts
        // go through a second MMA into the same accumulators.
        uint32_t xh0, xl0, xh1, xl1;
        split_f16x2(p[jc][0], p[jc][1], xh0, xl0);
        split_f16x2(p[jc][2], p[jc][3], xh1, xl1);
        const bool lo_cols = qc >= 4;  // lanes t = 2, 3: columns 4-7
        const uint32_t bh0 = transpose_m8n8_b16(dup && lo_cols ? xl0 : xh0);
        const uint32_t bh1 = transpose_m8n8_b16(dup && lo_cols ? xl1 : xh1);
        // V^T's A fragments from the e4m3 (int8) codes as in rows-as-rows:
        // the transposing ldmatrix of unit j gives, after the byte permute
        // and widening, keys (2t, 2t+1) and (2t+8, 2t+9) at d = 16j + 2g
        // (A rows g) and 16j + 2g + 1 (A rows g + 8).  o[j] then holds
        // O[column 2t, 2t + 1][d = 16j + 2g] (elements 0, 1) and
        // [d = 16j + 2g + 1] (elements 2, 3).
        const int mi = lane >> 3, row = (mi & 1) * 8 + (lane & 7);
        auto pv = [&](auto two_c) {
          constexpr bool two = decltype(two_c)::value != 0;
          uint32_t bl0 = 0u, bl1 = 0u;
          if (two) {
            bl0 = transpose_m8n8_b16(xl0);
            bl1 = transpose_m8n8_b16(xl1);
          }
#pragma unroll
          for (int j0 = 0; j0 < D / 16; j0 += 2) {
            const int u = j0 + (mi >> 1);
            uint32_t w[4];
            ldmatrix_x4_trans(vaddr + row * 128 + ((u ^ (row & 7)) << 4), w[0], w[1], w[2],
                              w[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t a0, b0, a1, b1;
              if constexpr (I8) {
                i8x4_keys_as_f16x2x2(w[2 * h], a0, b0);
                i8x4_keys_as_f16x2x2(w[2 * h + 1], a1, b1);
              } else {
                e4m3x4_as_f16x2x2(__byte_perm(w[2 * h], 0u, 0x3120u), a0, b0);
                e4m3x4_as_f16x2x2(__byte_perm(w[2 * h + 1], 0u, 0x3120u), a1, b1);
              }
              mma_16816<true>(o[j0 + h], a0, b0, a1, b1, bh0, bh1);
              if (two) mma_16816<true>(o[j0 + h], a0, b0, a1, b1, bl0, bl1);
            }
          }
        };
        if (dup)
          pv(IntC<0>());
        else
          pv(IntC<1>());
      }
      } else {
        // S = Q K^T over each chunk's 16 keys (two n-tiles of 8 keys); even and
        // odd K steps accumulate separately (two independent MMA chains)
        float s[NJ][2][4];
  #pragma unroll
        for (int j = 0; j < NJ; ++j) {
  #pragma unroll
          for (int n = 0; n < 2; ++n) s[j][n][0] = s[j][n][1] = s[j][n][2] = s[j][n][3] = 0.f;
          if (j >= nj) continue;
          const uint32_t kaddr = ring + stage * L::kStageBytes + (sub0 + j) * L::kChunkBytes;
          float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          if constexpr (KV8) {
            // the B fragment of key row n0 + g straight from the e4m3 codes:
            // lane (g, t) takes codes 16ks+4t .. +3 of the row (an 8 x 8 b16
            // ldmatrix fragment of the 16-byte unit), widened exactly to two
            // fp16 pairs; one ldmatrix.x4 covers both key halves of two K steps
            const int mi = lane >> 3, row = (mi & 1) * 8 + (lane & 7);
  #pragma unroll
            for (int ks = 0; ks < D / 16; ks += 2) {
              const int u = ks + (mi >> 1);
              uint32_t w[4];
              ldmatrix_x4(kaddr + row * 128 + ((u ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
  #pragma unroll
              for (int h = 0; h < 2; ++h)
  #pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                  uint32_t b0, b1;
                  if constexpr (I8)
                    i8x4_as_f16x2x2(w[2 * h + nt], b0, b1);
                  else
                    e4m3x4_as_f16x2x2(w[2 * h + nt], b0, b1);
                  mma_16816<true>((h ? s2 : s[j])[nt], qa[ks + h][0], qa[ks + h][1],
                                  qa[ks + h][2], qa[ks + h][3], b0, b1);
                }
            }
          } else {
            const int mi = lane >> 3, ri = lane & 7;
            const int tok = (mi >> 1) * 8 + ri;
  #pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const int u = 2 * ks + (mi & 1);
              uint32_t b0, b1, b2, b3;
              ldmatrix_x4(
                  kaddr + (u >> 3) * L::kHalfBytes + tok * 128 + (((u & 7) ^ (tok & 7)) << 4), b0,
                  b1, b2, b3);
              float(*acc)[4] = (ks & 1) ? s2 : s[j];
              mma_16816<KV8>(acc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
              mma_16816<KV8>(acc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
            }
          }
  #pragma unroll
          for (int n = 0; n < 2; ++n)
  #pragma unroll
            for (int e = 0; e < 4; ++e) s[j][n][e] += s2[n][e];
        }
        if constexpr (I8) {
          // int8 pools: each key's dot product times its K scale (this lane's
          // keys 8n + qc and 8n + qc + 1 of each chunk)
  #pragma unroll
          for (int j = 0; j < NJ; ++j) {
            if (j >= nj) break;
  #pragma unroll
            for (int n = 0; n < 2; ++n) {
              float k0, k1;
              asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];\n"
                           : "=f"(k0), "=f"(k1)
                           : "r"(scale_ring + stage * L::kScaleBytes +
                                 ((sub0 + j) * kChunk + n * 8 + qc) * 4));
              s[j][n][0] *= k0;
              s[j][n][1] *= k1;
              s[j][n][2] *= k0;
              s[j][n][3] *= k1;
            }
          }
        }
        // scores in log2 units; keys outside the stage's live set (or, with
        // several query tokens, outside a row's own range) score -inf.  A stage
        // whose keys are all live skips the per-key tests.
        constexpr uint32_t all_keys = nj == 1 ? 0xffffu : 0xffffffffu;
        if (P.q_len == 1 && ((smask >> (16 * sub0)) & all_keys) == all_keys) {
  #pragma unroll
          for (int j = 0; j < NJ; ++j)
  #pragma unroll
            for (int n = 0; n < 2; ++n)
  #pragma unroll
              for (int e = 0; e < 2; ++e) {
                s[j][n][e] = j < nj ? s[j][n][e] * P.scale_log2 : -INFINITY;
                s[j][n][2 + e] = j < nj ? s[j][n][2 + e] * P.scale_log2 : -INFINITY;
              }
        } else {
  #pragma unroll
        for (int j = 0; j < NJ; ++j)
  #pragma unroll
        for (int n = 0; n < 2; ++n) {
  #pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = n * 8 + qc + e;
            const bool ok = j < nj && ((smask >> (16 * (sub0 + j) + key)) & 1u);
            bool ok0 = ok, ok1 = ok;
            if (P.q_len > 1) {
              const int kp = (c0 + sub0 + j) * kChunk + key;
              ok0 = ok && kp >= lr0 && kp <= pr0;
              ok1 = ok && kp >= lr1 && kp <= pr1;
            }
            s[j][n][e] = ok0 ? s[j][n][e] * P.scale_log2 : -INFINITY;
            s[j][n][2 + e] = ok1 ? s[j][n][2 + e] * P.scale_log2 : -INFINITY;
          }
        }
        }
        // Lazy running max: the base moves only when a score passes it by more
        // than 2^8 (P stays below 256), so O is rescaled rarely.  When no score
        // of the warp passes its row's base (one vote), P is taken against the
        // base as it stands; otherwise the rows' maxima are reduced, the bases
        // moved and O rescaled.  Both give the same bits where the base stays.
        bool over = m0 == -INFINITY || (TWO_ROWS && m1 == -INFINITY);
  #pragma unroll
        for (int j = 0; j < NJ; ++j)
  #pragma unroll
          for (int n = 0; n < 2; ++n)
  #pragma unroll
            for (int e = 0; e < 2; ++e) {
              over |= s[j][n][e] > m0 + kLazyLog2;
              if (TWO_ROWS) over |= s[j][n][2 + e] > m1 + kLazyLog2;
            }
        float p[NJ][2][4];
        if (!__any_sync(0xffffffffu, over)) {
          float sum0 = 0.f;
  #pragma unroll
          for (int j = 0; j < NJ; ++j) {
  #pragma unroll
            for (int n = 0; n < 2; ++n) {
              p[j][n][0] = fast_exp2(s[j][n][0] - m0);
              p[j][n][1] = fast_exp2(s[j][n][1] - m0);
            }
            sum0 += p[j][0][0] + p[j][0][1] + p[j][1][0] + p[j][1][1];
          }
          l0 = l0 + sum0;
          if (TWO_ROWS) {
            float sum1 = 0.f;
  #pragma unroll
            for (int j = 0; j < NJ; ++j) {
  #pragma unroll
              for (int n = 0; n < 2; ++n) {
                p[j][n][2] = fast_exp2(s[j][n][2] - m1);
                p[j][n][3] = fast_exp2(s[j][n][3] - m1);
              }
              sum1 += p[j][0][2] + p[j][0][3] + p[j][1][2] + p[j][1][3];
            }
            l1 = l1 + sum1;
          }
        } else {
          float mx0 = -INFINITY, mx1 = -INFINITY;
  #pragma unroll
          for (int j = 0; j < NJ; ++j)
  #pragma unroll
            for (int n = 0; n < 2; ++n)
  #pragma unroll
              for (int e = 0; e < 2; ++e) {
                mx0 = fmaxf(mx0, s[j][n][e]);
                mx1 = fmaxf(mx1, s[j][n][2 + e]);
              }
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
          const float mn0 = (m0 == -INFINITY || mx0 > m0 + kLazyLog2) ? fmaxf(m0, mx0) : m0;
          const float base0 = mn0 == -INFINITY ? 0.f : mn0;  // no live key seen yet
          const float c0 = fast_exp2(m0 - base0);
          m0 = mn0;
          float sum0 = 0.f;
  #pragma unroll
          for (int j = 0; j < NJ; ++j) {
  #pragma unroll
            for (int n = 0; n < 2; ++n) {
              p[j][n][0] = fast_exp2(s[j][n][0] - base0);
              p[j][n][1] = fast_exp2(s[j][n][1] - base0);
            }
            sum0 += p[j][0][0] + p[j][0][1] + p[j][1][0] + p[j][1][1];
          }
          l0 = l0 * c0 + sum0;
          float c1 = c0;
          if (TWO_ROWS) {
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn1 = (m1 == -INFINITY || mx1 > m1 + kLazyLog2) ? fmaxf(m1, mx1) : m1;
            const float base1 = mn1 == -INFINITY ? 0.f : mn1;
            c1 = fast_exp2(m1 - base1);
            m1 = mn1;
            float sum1 = 0.f;
  #pragma unroll
            for (int j = 0; j < NJ; ++j) {
  #pragma unroll
              for (int n = 0; n < 2; ++n) {
                p[j][n][2] = fast_exp2(s[j][n][2] - base1);
                p[j][n][3] = fast_exp2(s[j][n][3] - base1);
              }
              sum1 += p[j][0][2] + p[j][0][3] + p[j][1][2] + p[j][1][3];
            }
            l1 = l1 * c1 + sum1;
          }
          // rows 8-15 hold either the second half of the group (TWO_ROWS) or
          // the low part of rows 0-7's probabilities; both rescale with their row
          if (__any_sync(0xffffffffu, c0 != 1.f || c1 != 1.f)) {
  #pragma unroll
            for (int n = 0; n < D / 8; ++n) {
              o[n][0] *= c0;
              o[n][1] *= c0;
              o[n][2] *= c1;
              o[n][3] *= c1;
            }
          }
        }
  #pragma unroll
        for (int jc = 0; jc < NJ; ++jc) {
          if (jc >= nj) break;
          const uint32_t vaddr =
              ring + stage * L::kStageBytes + (CPS + sub0 + jc) * L::kChunkBytes;
          if constexpr (I8) {
            // int8 pools: each probability times its key's V scale (a key
            // outside the live set has p = 0 and keeps it, whatever its scale)
  #pragma unroll
            for (int n = 0; n < 2; ++n) {
              float v0, v1;
              asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];\n"
                           : "=f"(v0), "=f"(v1)
                           : "r"(scale_ring + stage * L::kScaleBytes +
                                 ((CPS + sub0 + jc) * kChunk + n * 8 + qc) * 4));
              p[jc][n][0] = p[jc][n][0] > 0.f ? p[jc][n][0] * v0 : 0.f;
              p[jc][n][1] = p[jc][n][1] > 0.f ? p[jc][n][1] * v1 : 0.f;
              if (TWO_ROWS) {
                p[jc][n][2] = p[jc][n][2] > 0.f ? p[jc][n][2] * v0 : 0.f;
                p[jc][n][3] = p[jc][n][3] > 0.f ? p[jc][n][3] * v1 : 0.f;
              }
            }
          }
          // O += P V with P = hi + lo (bf16 pair, ~16 significant bits)
          uint32_t h0, l0w, h2, l2w;
          split16<KV8>(p[jc][0][0], p[jc][0][1], h0, l0w);
          split16<KV8>(p[jc][1][0], p[jc][1][1], h2, l2w);
          if constexpr (KV8) {
            // V's B fragments from the e4m3 codes: a transposing ldmatrix of
            // 16-byte unit j (its 16-bit elements being code pairs) hands lane
            // (g, t) the codes 2g and 2g+1 of keys 2t and 2t+1 (and of 2t+8,
            // 2t+9 from the second key half).  One byte permute pairs the keys
            // per code, and the two conversions give the B fragments of d
            // 16j+2g (n-tile 2j) and 16j+2g+1 (n-tile 2j+1).  The accumulators
            // of n-tiles 2j and 2j+1 then hold output columns 16j+4t+(0,2) and
            // 16j+4t+(1,3).
            const int mi = lane >> 3, row = (mi & 1) * 8 + (lane & 7);
            uint32_t h1 = 0u, l1w = 0u, h3 = 0u, l3w = 0u;
            if (TWO_ROWS) {
              split16<true>(p[jc][0][2], p[jc][0][3], h1, l1w);
              split16<true>(p[jc][1][2], p[jc][1][3], h3, l3w);
            }
  #pragma unroll
            for (int j0 = 0; j0 < D / 16; j0 += 2) {
              // units j0 and j0 + 1 of key rows 0-7 and 8-15
              const int u = j0 + (mi >> 1);
              uint32_t w[4];
              ldmatrix_x4_trans(vaddr + row * 128 + ((u ^ (row & 7)) << 4), w[0], w[1], w[2],
                                w[3]);
  #pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int j = j0 + h;
                // bytes (k 2t: 2g, 2g+1; k 2t+1: 2g, 2g+1) -> (2g: k, k+1; 2g+1: k, k+1)
                uint32_t a0, b0, a1, b1;
                if constexpr (I8) {
                  i8x4_keys_as_f16x2x2(w[2 * h], a0, b0);
                  i8x4_keys_as_f16x2x2(w[2 * h + 1], a1, b1);
                } else {
                  e4m3x4_as_f16x2x2(__byte_perm(w[2 * h], 0u, 0x3120u), a0, b0);
                  e4m3x4_as_f16x2x2(__byte_perm(w[2 * h + 1], 0u, 0x3120u), a1, b1);
                }
                if (!TWO_ROWS) {
                  mma_16816<true>(o[2 * j], h0, l0w, h2, l2w, a0, a1);
                  mma_16816<true>(o[2 * j + 1], h0, l0w, h2, l2w, b0, b1);
                } else {
                  mma_16816<true>(o[2 * j], h0, h1, h2, h3, a0, a1);
                  mma_16816<true>(o[2 * j], l0w, l1w, l2w, l3w, a0, a1);
                  mma_16816<true>(o[2 * j + 1], h0, h1, h2, h3, b0, b1);
                  mma_16816<true>(o[2 * j + 1], l0w, l1w, l2w, l3w, b0, b1);
                }
              }
            }
          } else {
            const int mi = lane >> 3, ri = lane & 7;
            const int tok = (mi & 1) * 8 + ri;
            if (!TWO_ROWS) {
  #pragma unroll
              for (int nd2 = 0; nd2 < D / 16; ++nd2) {
                const int u = 2 * nd2 + (mi >> 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(
                    vaddr + (u >> 3) * L::kHalfBytes + tok * 128 + (((u & 7) ^ (tok & 7)) << 4), b0,
                    b1, b2, b3);
                mma_16816<KV8>(o[2 * nd2], h0, l0w, h2, l2w, b0, b1);
                mma_16816<KV8>(o[2 * nd2 + 1], h0, l0w, h2, l2w, b2, b3);
              }
            } else {
              uint32_t h1, l1w, h3, l3w;
              split16<KV8>(p[jc][0][2], p[jc][0][3], h1, l1w);
              split16<KV8>(p[jc][1][2], p[jc][1][3], h3, l3w);
  #pragma unroll
              for (int nd2 = 0; nd2 < D / 16; ++nd2) {
                const int u = 2 * nd2 + (mi >> 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(
                    vaddr + (u >> 3) * L::kHalfBytes + tok * 128 + (((u & 7) ^ (tok & 7)) << 4), b0,
                    b1, b2, b3);
                mma_16816<KV8>(o[2 * nd2], h0, h1, h2, h3, b0, b1);
                mma_16816<KV8>(o[2 * nd2], l0w, l1w, l2w, l3w, b0, b1);
                mma_16816<KV8>(o[2 * nd2 + 1], h0, h1, h2, h3, b2, b3);
                mma_16816<KV8>(o[2 * nd2 + 1], l0w, l1w, l2w, l3w, b2, b3);
              }
            }
          }
        }
      }
      __syncwarp();
      };
      if constexpr (NJ == 1)
        step(IntC<1>());
      else if (nlive - sub0 >= NJ)
        step(IntC<NJ>());
      else
        step(IntC<1>());
    }
    }
    if (stop) break;
    // ------------------------------------------------------ finish the item
    if constexpr (KT) {
      // a column's sum spans the 8 lanes of one t; with dup, the low parts
      // (columns 4-7, lanes t = 2, 3) join their rows (lanes t - 2)
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, x);
        l1 += __shfl_xor_sync(0xffffffffu, l1, x);
      }
      if (dup) {
#pragma unroll
        for (int n = 0; n < NO; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[n][e] += __shfl_xor_sync(0xffffffffu, o[n][e], 2);
      }
      const bool writer = !dup || qc < 4;
      const bool live0 = writer && ra < P.rows, live1 = writer && rb < P.rows;
      const int h0r = (ra / P.group) * P.h_q + it.g * P.group + ra % P.group;
      const int h1r = (rb / P.group) * P.h_q + it.g * P.group + rb % P.group;
      // column e (0: 2t, 1: 2t + 1) of this lane: d = 16j + 2g and 16j + 2g + 1
      auto write_col = [&](float* dst, int e, float f, bool keep_in_l2, uint64_t pol) {
#pragma unroll
        for (int j = 0; j < NO; ++j) {
          float* d2 = dst + 16 * j + 2 * qr;
          const float v0 = (e ? o[j][1] : o[j][0]) * f, v1 = (e ? o[j][3] : o[j][2]) * f;
          if (keep_in_l2)
            st_f32x2_hint(d2, v0, v1, pol);
          else
            *reinterpret_cast<float2*>(d2) = make_float2(v0, v1);
        }
      };
      if (it.nsplits == 1) {
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
        if (live0) write_col(P.out + ((size_t)it.b * P.hq_all + h0r) * D, 0, i0, false, 0);
        if (live1) write_col(P.out + ((size_t)it.b * P.hq_all + h1r) * D, 1, i1, false, 0);
      } else {
        const uint64_t keep = l2_evict_last();
        if (live0) {
          const size_t rowi = (size_t)it.s_global * P.hq_all + h0r;
          write_col(P.ws.acc + rowi * D, 0, 1.f, true, keep);
          if (qr == 0) st_f32x2_hint(P.ws.ml + rowi * 2, m0, l0, keep);
        }
        if (live1) {
          const size_t rowi = (size_t)it.s_global * P.hq_all + h1r;
          write_col(P.ws.acc + rowi * D, 1, 1.f, true, keep);
          if (qr == 0) st_f32x2_hint(P.ws.ml + rowi * 2, m1, l1, keep);
        }
      }
    } else {
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      if (TWO_ROWS) {
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      }
      const bool single = it.nsplits == 1;
      // output index of rows qr and qr + 8 among the sequence's q_len * h_q
      const int h0r = (qr / P.group) * P.h_q + it.g * P.group + qr % P.group;
      const int h1r = ((qr + 8) / P.group) * P.h_q + it.g * P.group + (qr + 8) % P.group;
      // One output row of this lane, times f: 16-bit pools hold float pairs at
      // columns 8n + 2t (n-tile n), e4m3 pools float quads at 16j + 4t (n-tile
      // 2j: columns +0 and +2; n-tile 2j+1: +1 and +3).  Row qr adds the low
      // part of P carried in rows 8-15 unless TWO_ROWS; with TWO_ROWS, rows
      // 8-15 are row qr + 8.
      auto write_row = [&](float* dst, bool second, float f, bool keep_in_l2, uint64_t pol) {
        if constexpr (KV8) {
  #pragma unroll
          for (int j = 0; j < D / 16; ++j) {
            const float* x = o[2 * j];
            const float* y = o[2 * j + 1];
            const float v0 = second ? x[2] : (TWO_ROWS ? x[0] : x[0] + x[2]);
            const float v1 = second ? y[2] : (TWO_ROWS ? y[0] : y[0] + y[2]);
            const float v2 = second ? x[3] : (TWO_ROWS ? x[1] : x[1] + x[3]);
            const float v3 = second ? y[3] : (TWO_ROWS ? y[1] : y[1] + y[3]);
            float* d4 = dst + 16 * j + 4 * (lane & 3);
            if (keep_in_l2)
              st_f32x4_hint(d4, v0 * f, v1 * f, v2 * f, v3 * f, pol);
            else
              *reinterpret_cast<float4*>(d4) = make_float4(v0 * f, v1 * f, v2 * f, v3 * f);
          }
        } else {
  #pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            const float v0 = second ? o[n][2] : (TWO_ROWS ? o[n][0] : o[n][0] + o[n][2]);
            const float v1 = second ? o[n][3] : (TWO_ROWS ? o[n][1] : o[n][1] + o[n][3]);
            float* d2 = dst + n * 8 + qc;
            if (keep_in_l2)
              st_f32x2_hint(d2, v0 * f, v1 * f, pol);
            else
              *reinterpret_cast<float2*>(d2) = make_float2(v0 * f, v1 * f);
          }
        }
      };
      if (single) {
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
        if (qr < P.rows) write_row(P.out + ((size_t)it.b * P.hq_all + h0r) * D, false, i0, false, 0);
        if (TWO_ROWS && qr + 8 < P.rows)
          write_row(P.out + ((size_t)it.b * P.hq_all + h1r) * D, true, i1, false, 0);
      } else {
        // partials stay in L2 for the combine kernel that follows
        const uint64_t keep = l2_evict_last();
        if (qr < P.rows) {
          const size_t rowi = (size_t)it.s_global * P.hq_all + h0r;
          write_row(P.ws.acc + rowi * D, false, 1.f, true, keep);
          if ((lane & 3) == 0) st_f32x2_hint(P.ws.ml + rowi * 2, m0, l0, keep);
        }
        if (TWO_ROWS && qr + 8 < P.rows) {
          const size_t rowi = (size_t)it.s_global * P.hq_all + h1r;
          write_row(P.ws.acc + rowi * D, true, 1.f, true, keep);
          if ((lane & 3) == 0) st_f32x2_hint(P.ws.ml + rowi * 2, m1, l1, keep);
        }
      }
    }
    ++items_c;
  }
  // drain: every copy this warp issued has landed before it exits (each is
  // the latest phase of its barrier)
  bool drained = true;
  for (uint32_t i = gs_c; i < gs_issue; ++i)
    drained &= mbar_drain(smem_u32(&sh.full[w][i % R]), (i / R) & 1);
  for (int i = items_c; i < items_issued; ++i)
    drained &= mbar_drain(smem_u32(&sh.qfull[w][i % R]), (i / R) & 1);
  if (!drained) *abort_flag = 1;
  __syncthreads();  // every wait above is bounded, so every thread gets here
  if (threadIdx.x == 0 && sh.abort_flag) report(P.error_word, TL_DEVERR_TIMEOUT);
  if (threadIdx.x == 0) TL_TRACE_MAX(TL_TRACE_ATTN_END);
}

// ------------------------------------------------------------- f32 kernel --
//
// IEEE f32 pools ("How serving works in Tlaloc": f32 keys and values, dots in
// f32).  Computed on the CUDA cores in f32: no tensor-core rounding of the
// operands.  CTAs take work items from the counter; each warp walks its
// chunks one key at a time (lanes hold D/32 elements of each query head, a
// warp sum gives each score, a scalar online softmax folds it in); the warps
// merge in shared memory and write a partial that decode_combine_kernel
// merges.

constexpr int kF32MaxGroup = 16;

template <int D>
__global__ void __launch_bounds__(kDecodeThreads) decode_f32_kernel(DecodeParams P) {
  constexpr int E = D / 32;
  constexpr int RS = D + 2;
  __shared__ float merge[kDecodeWarps][kF32MaxGroup][RS];
  __shared__ int s_item;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int total_items = __ldcg(P.ws.ctrl + 1) * P.h_kv;
  for (;;) {
    if (threadIdx.x == 0) s_item = atomicAdd(P.ws.ctrl + 2, 1);
    __syncthreads();
    const int item = s_item;
    __syncthreads();
    if (item >= total_items) break;
    ItemInfo it;
    describe_item(P, item, it);
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
            table_entry(P, it.b, j / P.page_size);
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
    for (int idx = threadIdx.x; idx < P.group * (D + 1); idx += kDecodeThreads) {
      const int r = idx / (D + 1), e = idx - r * (D + 1);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, merge[w][r][D]);
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        const float f = merge[w][r][D] == -INFINITY ? 0.f : fast_exp2(merge[w][r][D] - M);
        a += f * (e < D ? merge[w][r][e] : merge[w][r][D + 1]);
      }
      const size_t rowi = (size_t)it.s_global * P.h_q + (size_t)it.g * P.group + r;
      if (e < D) {
        P.ws.acc[rowi * D + e] = a;
      } else {
        P.ws.ml[rowi * 2 + 0] = M;
        P.ws.ml[rowi * 2 + 1] = a;
      }
    }
    __syncthreads();
  }
}

// --------------------------------------------------------------- combine --
//
// Merges each sequence's piece partials.  Sequences with one piece were
// written by the main kernel when skip_single is set; sequences with none
// output 0.
//
// A (sequence, output row) takes kTpr x G threads: G groups of D/4 threads,
// each thread 4 outputs.  Group r folds the pieces r, r + G, r + 2G, ... in
// that order, 8 at a time: their (m, l) and partial rows are loaded together
// (one round of loads per 8 pieces), then
//   M' = max(M, m_s),  a = a 2^(M - M') + sum_s 2^(m_s - M') acc_s,
//   l = l 2^(M - M') + sum_s 2^(m_s - M') l_s.
// With G > 1 the groups' (M, l, a) meet in shared memory and group 0 folds
// groups 1 .. G-1 into its own in that order, by the same rule; out = a / l.
// More groups shorten the chain of dependent load rounds of a sequence with
// many pieces (few long sequences), at the price of more threads; the host
// picks G from the pieces a sequence can have.  The partials come from the
// previous kernel: reads go to L2 (ld.global.cg).
template <int D, bool GROUPED>
__global__ void __launch_bounds__(512) decode_combine_kernel(DecodeParams P, int skip_single,
                                                              int groups) {
  constexpr int kTpr = D / 4;   // threads per output row and group
  constexpr int kBatch = 8;     // pieces per round of loads
  const int G = GROUPED ? groups : 1;  // one group: the loop's strides are constants
  extern __shared__ float4 cmb_sm[];  // G > 1: per thread (a) then (M, l)
  // a no-op unless launched as a programmatic dependent of the attention kernel
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (threadIdx.x == 0) TL_TRACE_MIN(TL_TRACE_COMBINE_START);
  const int t = threadIdx.x;
  const int c = t % kTpr;
  const int r = (t / kTpr) % G;
  const int rows_per_block = blockDim.x / (kTpr * G);
  const int64_t row = (int64_t)blockIdx.x * rows_per_block + t / (kTpr * G);  // b * hq_all + h
  const bool live = row < (int64_t)P.B * P.hq_all;
  int s0 = 0, ns = 0, h = 0;
  if (live) {
    const int b = (int)(row / P.hq_all);
    h = (int)(row - (int64_t)b * P.hq_all);
    s0 = __ldcg(P.ws.split_off + b);
    ns = __ldcg(P.ws.split_off + b + 1) - s0;
  }
  const bool fold = live && (ns > 1 || (ns == 1 && !skip_single));
  float M = -INFINITY, l = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  if (fold) {
    const float2* ml = reinterpret_cast<const float2*>(P.ws.ml) + (size_t)s0 * P.hq_all + h;
    const float4* acc =
        reinterpret_cast<const float4*>(P.ws.acc + ((size_t)s0 * P.hq_all + h) * D + 4 * c);
    const size_t acc_stride = (size_t)P.hq_all * D / 4;  // float4 units
    for (int s = r; s < ns; s += G * kBatch) {
      float2 mlv[kBatch];
      float4 av[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int su = s + u * G;
        if (su < ns) {
          mlv[u] = __ldcg(ml + (size_t)su * P.hq_all);
          av[u] = __ldcg(acc + (size_t)su * acc_stride);
        } else {
          mlv[u] = make_float2(-INFINITY, 0.f);
          av[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float Mn = M;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) Mn = fmaxf(Mn, mlv[u].x);
      if (Mn == -INFINITY) continue;  // no key seen yet by any piece
      const float cm = M == -INFINITY ? 0.f : fast_exp2(M - Mn);
      l *= cm;
      a.x *= cm; a.y *= cm; a.z *= cm; a.w *= cm;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float f = mlv[u].x == -INFINITY ? 0.f : fast_exp2(mlv[u].x - Mn);
        l += f * mlv[u].y;
        a.x += f * av[u].x; a.y += f * av[u].y; a.z += f * av[u].z; a.w += f * av[u].w;
      }
      M = Mn;
    }
  }
  if (GROUPED) {
    cmb_sm[t] = a;
    cmb_sm[blockDim.x + t] = make_float4(M, l, 0.f, 0.f);
    __syncthreads();
  }
  if (live && r == 0 && (ns == 0 || fold)) {
    for (int g = 1; g < G; ++g) {
      const float4 a2 = cmb_sm[t + g * kTpr];
      const float4 ml2 = cmb_sm[blockDim.x + t + g * kTpr];
      const float Mn = fmaxf(M, ml2.x);
      if (Mn == -INFINITY) continue;
      const float f0 = M == -INFINITY ? 0.f : fast_exp2(M - Mn);
      const float f1 = ml2.x == -INFINITY ? 0.f : fast_exp2(ml2.x - Mn);
      l = l * f0 + ml2.y * f1;
      a.x = a.x * f0 + a2.x * f1; a.y = a.y * f0 + a2.y * f1;
      a.z = a.z * f0 + a2.z * f1; a.w = a.w * f0 + a2.w * f1;
      M = Mn;
    }
    // a sequence with nothing to read (ns == 0) folds nothing: l = 0, out 0
    const float inv = l > 0.f ? 1.f / l : 0.f;
    *reinterpret_cast<float4*>(P.out + row * D + 4 * c) =
        make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
  }
#if TL_DECODE_TRACE
  __syncthreads();
  if (t == 0) TL_TRACE_MAX(TL_TRACE_COMBINE_END);
#endif
}

// Groups per row of the combine: a sequence has at most about
// ceil(pieces target / B) + 2 pieces; one group per 24 of them, a power of
// two up to a 512-thread row (16 groups at d = 128, 32 at d = 64).  Measured on GB300 (Llama-3-8B heads, whole calls): B = 16
// with ~50 pieces a sequence 56.5 -> 53.9 us with 4 groups; B = 4 at 32K keys
// 107.4 -> 92.9 us with 8; at B >= 32 (<= 26 pieces) more groups only add
// CTAs (B = 64: 195.7 us with 1, 199.0 with 4).
static int combine_groups(int B, int h_kv, int d) {
  const int64_t est = ((int64_t)kTargetItems / h_kv + B - 1) / B + 2;
  int g = 1;
  while (g * 2 * (d / 4) <= 512 && est >= 24 * g) g *= 2;
  return g;
}

// Launches the combine over B * rows_per_seq output rows.
static cudaError_t launch_combine(const DecodeParams& P, int B, int rows_per_seq, int d,
                                  int skip_single, bool dependent, cudaStream_t st) {
  const int G = combine_groups(B, P.h_kv, d);
  const int tpr = d / 4 * G;                      // threads per output row
  const int threads = std::max(256, tpr);
  const int64_t rows = (int64_t)B * rows_per_seq;
  const int64_t per_block = threads / tpr;
  cudaLaunchAttribute cattr[1];
  cattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  cattr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3((unsigned)((rows + per_block - 1) / per_block));
  ccfg.blockDim = dim3(threads);
  ccfg.dynamicSmemBytes = G > 1 ? (size_t)threads * 2 * sizeof(float4) : 0;
  ccfg.stream = st;
  ccfg.attrs = cattr;
  ccfg.numAttrs = dependent ? 1 : 0;
  if (G > 1)
    return d == 128 ? cudaLaunchKernelEx(&ccfg, decode_combine_kernel<128, true>, P, skip_single, G)
                    : cudaLaunchKernelEx(&ccfg, decode_combine_kernel<64, true>, P, skip_single, G);
  return d == 128 ? cudaLaunchKernelEx(&ccfg, decode_combine_kernel<128, false>, P, skip_single, 1)
                  : cudaLaunchKernelEx(&ccfg, decode_combine_kernel<64, false>, P, skip_single, 1);
}

}  // namespace tl

// ------------------------------------------------------------------- host --

extern "C" tl_status tl_decode_trace_reset(void) {
#if TL_DECODE_TRACE
  unsigned long long init[TL_TRACE_SLOTS] = {};
  init[TL_TRACE_COMBINE_START] = ~0ull;
  if (cudaDeviceSynchronize() != cudaSuccess) return TL_ERR_CUDA;
  if (cudaMemcpyToSymbol(tl::g_trace, init, sizeof(init)) != cudaSuccess) return TL_ERR_CUDA;
  return TL_OK;
#else
  return TL_ERR_UNSUPPORTED;
#endif
}

extern "C" tl_status tl_decode_trace_read(uint64_t* stamps, int32_t n) {
#if TL_DECODE_TRACE
  if (!stamps || n < 1 || n > TL_TRACE_SLOTS) return TL_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return TL_ERR_CUDA;
  if (cudaMemcpyFromSymbol(stamps, tl::g_trace, sizeof(uint64_t) * n) != cudaSuccess)
    return TL_ERR_CUDA;
  return TL_OK;
#else
  (void)stamps;
  (void)n;
  return TL_ERR_UNSUPPORTED;
#endif
}

extern "C" size_t tl_paged_attn_decode_workspace_size(int32_t B, int32_t h_q, int32_t h_kv,
                                                      int32_t d) {
  if (B <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || h_q % h_kv) return 0;
  return tl::decode_ws_layout(B, h_q, h_kv, d, nullptr, nullptr);
}

namespace tl {
// The new rows a decode call writes itself (tl_paged_attn_decode_write):
// n rows of k_new / v_new in new_dtype, scattered by slot into the pools.
struct NewRows {
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  const int64_t* slot_mapping = nullptr;
  int32_t n = 0;
  tl_dtype new_dtype = TL_BF16;
  void* k_dst = nullptr;
  void* v_dst = nullptr;
};

// Warps per CTA of a bf16 / one-byte kernel variant: its shape's count, or
// as many as the dynamic shared memory holds (227 KiB less 2 KiB for the
// static state, the int8 scale rings and the 1 KiB alignment pad).
template <int D, bool TWO, bool K8, bool I8>
static int decode_warps(int rows) {
  using S = DecodeShape<TWO, K8>;
  using L = WarpSmem<D, K8, I8, S::kRing>;
  static_assert(sizeof(WarpShared<S::kWarps, S::kRing>) <= 2048, "static state over 2 KiB");
  const int scales = I8 ? S::kWarps * S::kRing * L::kScaleBytes : 0;
  return std::min(S::kWarps, (227 * 1024 - 3072 - scales) / L::warp_bytes(rows));
}

static tl_status decode_impl(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, int32_t max_pages_per_seq,
                             const int32_t* context_lens, float* out, int32_t B, int32_t q_len,
                             int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                             int32_t page_size, int32_t window, int32_t ring_pages, float scale,
                             tl_dtype dtype, void* workspace, size_t workspace_bytes,
                             uint32_t* error_word, void* stream, const NewRows& nr = NewRows(),
                             const float* k_scales = nullptr, const float* v_scales = nullptr) {
  if (B <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || num_pages <= 0 || page_size <= 0 ||
      max_pages_per_seq <= 0 || window < 0)
    return TL_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out)
    return TL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return TL_ERR_INVALID_ARG;
  if (h_q % h_kv || q_len <= 0) return TL_ERR_INVALID_ARG;
  const int group = h_q / h_kv;
  // the M rows of a work item: the group's heads of each query token
  if ((int64_t)q_len * group > 16 || (q_len > 1 && dtype == TL_F32)) return TL_ERR_UNSUPPORTED;
  const int rows = q_len * group;
  if (dtype != TL_BF16 && dtype != TL_F32 && dtype != TL_FP8_E4M3) return TL_ERR_UNSUPPORTED;
  if ((d != 64 && d != 128) || group > 16 || page_size > 256) return TL_ERR_UNSUPPORTED;
  // the bf16 and e4m3 paths move pages with TMA boxes of 8 or 16 rows; e4m3
  // rows are one 128-byte box wide
  if (dtype != TL_F32 && page_size % 8 != 0) return TL_ERR_UNSUPPORTED;
  if (dtype == TL_FP8_E4M3 && d != 128) return TL_ERR_UNSUPPORTED;
  if ((int64_t)num_pages * page_size >= ((int64_t)1 << 31)) return TL_ERR_UNSUPPORTED;
  // int8 pools (the one-byte path with per-key scales): a chunk's 16 scales
  // of one head are one aligned 64-byte copy
  const bool i8 = k_scales != nullptr || v_scales != nullptr;
  if (i8) {
    if (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales))
      return TL_ERR_INVALID_ARG;
    if (dtype != TL_FP8_E4M3 || page_size % 16 != 0) return TL_ERR_UNSUPPORTED;
  }
  const size_t need = decode_ws_layout(B, q_len * h_q, h_kv, d, nullptr, nullptr);
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
  P.d = d;
  P.num_pages = num_pages;
  P.page_size = page_size;
  P.window = window;
  P.ring_pages = ring_pages;
  P.ps_shift = -1;
  if ((page_size & (page_size - 1)) == 0)
    for (int s = 0; s < 31; ++s)
      if ((1 << s) == page_size) P.ps_shift = s;
  P.q_len = q_len;
  P.rows = rows;
  P.hq_all = q_len * h_q;
  P.scale_log2 = scale * kLog2e;
  decode_ws_layout(B, q_len * h_q, h_kv, d, &P.ws, static_cast<char*>(workspace));
  P.error_word = error_word;
  // the call's own new rows: validated like tl_kv_cache_write / _fp8
  P.k_new = nr.k_new;
  P.v_new = nr.v_new;
  P.slot_mapping = nr.slot_mapping;
  P.k_dst = nr.k_dst;
  P.v_dst = nr.v_dst;
  P.n_new = 0;
  P.new_kind = 0;
  P.row_units = 0;
  P.k_scales = k_scales;
  P.v_scales = v_scales;
  if (nr.n < 0) return TL_ERR_INVALID_ARG;
  if (nr.n > 0) {
    if (!nr.k_new || !nr.v_new || !nr.slot_mapping || !nr.k_dst || !nr.v_dst)
      return TL_ERR_INVALID_ARG;
    if (!aligned16(nr.k_new) || !aligned16(nr.v_new) ||
        (reinterpret_cast<uintptr_t>(nr.slot_mapping) & 7u))
      return TL_ERR_INVALID_ARG;
    const int64_t row = (int64_t)h_kv * d;
    if (i8) {
      if (nr.new_dtype != TL_BF16 && nr.new_dtype != TL_F32) return TL_ERR_UNSUPPORTED;
      P.new_kind = nr.new_dtype == TL_BF16 ? 3 : 4;
      P.row_units = 0;
    } else if (dtype == TL_FP8_E4M3) {
      if (nr.new_dtype != TL_BF16 && nr.new_dtype != TL_F32) return TL_ERR_UNSUPPORTED;
      if (row % 16 != 0) return TL_ERR_INVALID_ARG;
      P.new_kind = nr.new_dtype == TL_BF16 ? 1 : 2;
      P.row_units = (int32_t)(row / 8);
    } else {
      if (nr.new_dtype != dtype) return TL_ERR_UNSUPPORTED;
      const int64_t row_bytes = row * (dtype == TL_F32 ? 4 : 2);
      if (row_bytes % 16 != 0) return TL_ERR_INVALID_ARG;
      P.new_kind = 0;
      P.row_units = (int32_t)(row_bytes / 16);
    }
    P.n_new = nr.n;
  }
  cudaStream_t st = (cudaStream_t)stream;

  // warps per CTA of the bf16 / one-byte kernel (up to its shape's count,
  // as many as the stages fit)
  const bool kv8 = dtype == TL_FP8_E4M3;
  const bool two = rows > 8;
  int warps = 0;
  if (dtype != TL_F32) {
    warps = i8    ? (two ? decode_warps<128, true, true, true>(rows)
                         : decode_warps<128, false, true, true>(rows))
            : kv8 ? (two ? decode_warps<128, true, true, false>(rows)
                         : decode_warps<128, false, true, false>(rows))
            : d == 128 ? (two ? decode_warps<128, true, false, false>(rows)
                              : decode_warps<128, false, false, false>(rows))
                       : (two ? decode_warps<64, true, false, false>(rows)
                              : decode_warps<64, false, false, false>(rows));
  }
  const int target_splits = (kTargetItems + h_kv - 1) / h_kv;
  // plan block: up to kWarpPlanMax sequences one warp plans and 1024
  // threads write the descriptors; larger batches spread their sequences over
  // the threads (and loop past 1024), where a smaller block makes the block
  // reductions and the scan cheaper
  const int plan_threads =
      B <= kWarpPlanMax ? 1024
                        : (int)std::min<int64_t>(1024, std::max<int64_t>(256, align_up((size_t)B, 32)));
  // the plan CTA, then (for a call that writes its new rows) CTAs with one
  // warp per new row, up to one per SM
  // (int8 pools: one warp per token and KV head)
  const int64_t write_warps = P.new_kind >= 3 ? (int64_t)P.n_new * h_kv : P.n_new;
  const int wpc = B <= kWarpPlanMax ? kWriteWarps : plan_threads / 32;
  const int64_t write_ctas =
      P.n_new > 0 ? std::min<int64_t>(num_sms(), (write_warps + wpc - 1) / wpc) : 0;
  decode_plan_kernel<<<(unsigned)(1 + write_ctas), plan_threads, 0, st>>>(P, target_splits,
                                                                          num_sms() * warps);
  if (launch_status() != TL_OK) return TL_ERR_CUDA;

  if (dtype == TL_BF16 || dtype == TL_FP8_E4M3) {
    // 3-D tensor maps of the pools: (d, H_kv, slot), boxes of one 128-byte
    // row part x 1 x box_rows (64 bf16 or 128 e4m3 elements)
    const int esz = kv8 ? 1 : 2;
    const int box_rows = page_size % 16 == 0 ? 16 : 8;
    CUtensorMap kmap, vmap;
    const uint64_t dims[3] = {(uint64_t)d, (uint64_t)h_kv, (uint64_t)num_pages * page_size};
    const uint64_t strides[2] = {(uint64_t)d * esz, (uint64_t)h_kv * d * esz};
    const uint32_t box[3] = {(uint32_t)(128 / esz), 1, (uint32_t)box_rows};
    const bool enc = kv8 ? (encode_u8_tensor_map(&kmap, k_cache, 3, dims, strides, box, true) &&
                            encode_u8_tensor_map(&vmap, v_cache, 3, dims, strides, box, true))
                         : (encode_bf16_tensor_map(&kmap, k_cache, 3, dims, strides, box, true) &&
                            encode_bf16_tensor_map(&vmap, v_cache, 3, dims, strides, box, true));
    if (!enc) return TL_ERR_CUDA;
#define TL_LAUNCH_W(DD, TWO, K8, I8V)                                                     \
  do {                                                                                    \
    auto kern = decode_bf16_kernel<DD, TWO, K8, I8V>;                                     \
    const int sm =                                                                        \
        warps * WarpSmem<DD, K8, I8V, DecodeShape<TWO, K8>::kRing>::warp_bytes(rows) + 1024; \
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sm) !=    \
        cudaSuccess)                                                                      \
      return TL_ERR_CUDA;                                                                 \
    cudaLaunchAttribute attr[1];                                                          \
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;                      \
    attr[0].val.programmaticStreamSerializationAllowed = 1;                               \
    cudaLaunchConfig_t cfg = {};                                                          \
    cfg.gridDim = dim3(num_sms());                                                        \
    cfg.blockDim = dim3(warps * 32);                                                      \
    cfg.dynamicSmemBytes = sm;                                                            \
    cfg.stream = st;                                                                      \
    cfg.attrs = attr;                                                                     \
    cfg.numAttrs = 1;                                                                     \
    if (cudaLaunchKernelEx(&cfg, kern, P, kmap, vmap, box_rows) != cudaSuccess)           \
      return TL_ERR_CUDA;                                                                 \
  } while (0)
    // template arguments: d, two row groups (rows > 8), one-byte codes, int8
    if (i8) {
      if (rows > 8) TL_LAUNCH_W(128, true, true, true);
      else TL_LAUNCH_W(128, false, true, true);
    } else if (kv8) {
      if (rows > 8) TL_LAUNCH_W(128, true, true, false);
      else TL_LAUNCH_W(128, false, true, false);
    } else if (d == 128) {
      if (rows > 8) TL_LAUNCH_W(128, true, false, false);
      else TL_LAUNCH_W(128, false, false, false);
    } else {
      if (rows > 8) TL_LAUNCH_W(64, true, false, false);
      else TL_LAUNCH_W(64, false, false, false);
    }
#undef TL_LAUNCH_W
    if (launch_status() != TL_OK) return TL_ERR_CUDA;
    // the merge, a programmatic dependent of the attention kernel: its CTAs
    // take the SMs as the attention CTAs leave
    if (launch_combine(P, B, P.hq_all, d, 1, true, st) != cudaSuccess) return TL_ERR_CUDA;
    return launch_status();
  }
  const int grid = num_sms() * 2;
  if (d == 128) decode_f32_kernel<128><<<grid, kDecodeThreads, 0, st>>>(P);
  else decode_f32_kernel<64><<<grid, kDecodeThreads, 0, st>>>(P);
  if (launch_status() != TL_OK) return TL_ERR_CUDA;
  if (launch_combine(P, B, h_q, d, 0, false, st) != cudaSuccess) return TL_ERR_CUDA;
  return launch_status();
}
}  // namespace tl

extern "C" tl_status tl_paged_attn_decode(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_table,
                                          int32_t max_pages_per_seq,
                                          const int32_t* context_lens, float* out, int32_t B,
                                          int32_t h_q, int32_t h_kv, int32_t d,
                                          int32_t num_pages, int32_t page_size, int32_t window,
                                          float scale, tl_dtype dtype, void* workspace,
                                          size_t workspace_bytes, uint32_t* error_word,
                                          void* stream) {
  return tl::decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, context_lens, out,
                         B, 1, h_q, h_kv, d, num_pages, page_size, window, 0, scale, dtype,
                         workspace, workspace_bytes, error_word, stream);
}

extern "C" tl_status tl_paged_attn_decode_int8(
    const void* q, const int8_t* k_codes, const int8_t* v_codes, const float* k_scales,
    const float* v_scales, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* context_lens, float* out, int32_t B, int32_t h_q, int32_t h_kv, int32_t d,
    int32_t num_pages, int32_t page_size, int32_t window, float scale, void* workspace,
    size_t workspace_bytes, uint32_t* error_word, void* stream) {
  if (!k_scales || !v_scales) return TL_ERR_INVALID_ARG;
  return tl::decode_impl(q, k_codes, v_codes, block_table, max_pages_per_seq, context_lens, out,
                         B, 1, h_q, h_kv, d, num_pages, page_size, window, 0, scale,
                         TL_FP8_E4M3, workspace, workspace_bytes, error_word, stream,
                         tl::NewRows(), k_scales, v_scales);
}

extern "C" tl_status tl_paged_attn_decode_write_int8(
    const void* q, const void* k_new, const void* v_new, tl_dtype new_dtype,
    const int64_t* slot_mapping, int32_t n_new, int8_t* k_codes, int8_t* v_codes,
    float* k_scales, float* v_scales, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* context_lens, float* out, int32_t B, int32_t h_q, int32_t h_kv, int32_t d,
    int32_t num_pages, int32_t page_size, int32_t window, float scale, void* workspace,
    size_t workspace_bytes, uint32_t* error_word, void* stream) {
  if (!k_scales || !v_scales) return TL_ERR_INVALID_ARG;
  tl::NewRows nr;
  nr.k_new = k_new;
  nr.v_new = v_new;
  nr.slot_mapping = slot_mapping;
  nr.n = n_new;
  nr.new_dtype = new_dtype;
  nr.k_dst = k_codes;
  nr.v_dst = v_codes;
  return tl::decode_impl(q, k_codes, v_codes, block_table, max_pages_per_seq, context_lens, out,
                         B, 1, h_q, h_kv, d, num_pages, page_size, window, 0, scale,
                         TL_FP8_E4M3, workspace, workspace_bytes, error_word, stream, nr,
                         k_scales, v_scales);
}

extern "C" tl_status tl_paged_attn_decode_write(
    const void* q, const void* k_new, const void* v_new, tl_dtype new_dtype,
    const int64_t* slot_mapping, int32_t n_new, void* k_cache, void* v_cache,
    const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* context_lens,
    float* out, int32_t B, int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
    int32_t page_size, int32_t window, float scale, tl_dtype dtype, void* workspace,
    size_t workspace_bytes, uint32_t* error_word, void* stream) {
  tl::NewRows nr;
  nr.k_new = k_new;
  nr.v_new = v_new;
  nr.slot_mapping = slot_mapping;
  nr.n = n_new;
  nr.new_dtype = new_dtype;
  nr.k_dst = k_cache;
  nr.v_dst = v_cache;
  return tl::decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, context_lens, out,
                         B, 1, h_q, h_kv, d, num_pages, page_size, window, 0, scale, dtype,
                         workspace, workspace_bytes, error_word, stream, nr);
}

extern "C" tl_status tl_paged_attn_decode_write_ring(
    const void* q, const void* k_new, const void* v_new, tl_dtype new_dtype,
    const int64_t* slot_mapping, int32_t n_new, void* k_cache, void* v_cache,
    const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* context_lens,
    float* out, int32_t B, int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
    int32_t page_size, int32_t window, int32_t ring_pages, float scale, tl_dtype dtype,
    void* workspace, size_t workspace_bytes, uint32_t* error_word, void* stream) {
  if (ring_pages <= 0 || ring_pages > max_pages_per_seq || window <= 0 || page_size <= 0 ||
      (int64_t)ring_pages * page_size < window)
    return TL_ERR_INVALID_ARG;
  tl::NewRows nr;
  nr.k_new = k_new;
  nr.v_new = v_new;
  nr.slot_mapping = slot_mapping;
  nr.n = n_new;
  nr.new_dtype = new_dtype;
  nr.k_dst = k_cache;
  nr.v_dst = v_cache;
  return tl::decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, context_lens, out,
                         B, 1, h_q, h_kv, d, num_pages, page_size, window, ring_pages, scale,
                         dtype, workspace, workspace_bytes, error_word, stream, nr);
}

extern "C" tl_status tl_paged_attn_decode_ring(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* context_lens, float* out, int32_t B, int32_t h_q,
    int32_t h_kv, int32_t d, int32_t num_pages, int32_t page_size, int32_t window,
    int32_t ring_pages, float scale, tl_dtype dtype, void* workspace, size_t workspace_bytes,
    uint32_t* error_word, void* stream) {
  // the ring must be part of the table and must hold one window
  if (ring_pages <= 0 || ring_pages > max_pages_per_seq || window <= 0 || page_size <= 0 ||
      (int64_t)ring_pages * page_size < window)
    return TL_ERR_INVALID_ARG;
  return tl::decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, context_lens, out,
                         B, 1, h_q, h_kv, d, num_pages, page_size, window, ring_pages, scale,
                         dtype, workspace, workspace_bytes, error_word, stream);
}

extern "C" tl_status tl_paged_attn_decode_ring_int8(
    const void* q, const int8_t* k_codes, const int8_t* v_codes, const float* k_scales,
    const float* v_scales, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* context_lens, float* out, int32_t B, int32_t h_q, int32_t h_kv, int32_t d,
    int32_t num_pages, int32_t page_size, int32_t window, int32_t ring_pages, float scale,
    void* workspace, size_t workspace_bytes, uint32_t* error_word, void* stream) {
  if (!k_scales || !v_scales) return TL_ERR_INVALID_ARG;
  // the ring must be part of the table and must hold one window
  if (ring_pages <= 0 || ring_pages > max_pages_per_seq || window <= 0 || page_size <= 0 ||
      (int64_t)ring_pages * page_size < window)
    return TL_ERR_INVALID_ARG;
  return tl::decode_impl(q, k_codes, v_codes, block_table, max_pages_per_seq, context_lens, out,
                         B, 1, h_q, h_kv, d, num_pages, page_size, window, ring_pages, scale,
                         TL_FP8_E4M3, workspace, workspace_bytes, error_word, stream,
                         tl::NewRows(), k_scales, v_scales);
}

extern "C" size_t tl_paged_attn_decode_multi_workspace_size(int32_t B, int32_t q_len,
                                                            int32_t h_q, int32_t h_kv, int32_t d) {
  if (B <= 0 || q_len <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || h_q % h_kv) return 0;
  return tl::decode_ws_layout(B, q_len * h_q, h_kv, d, nullptr, nullptr);
}

extern "C" tl_status tl_paged_attn_decode_multi_int8(
    const void* q, const int8_t* k_codes, const int8_t* v_codes, const float* k_scales,
    const float* v_scales, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* context_lens, float* out, int32_t B, int32_t q_len, int32_t h_q, int32_t h_kv,
    int32_t d, int32_t num_pages, int32_t page_size, int32_t window, float scale,
    void* workspace, size_t workspace_bytes, uint32_t* error_word, void* stream) {
  if (!k_scales || !v_scales) return TL_ERR_INVALID_ARG;
  return tl::decode_impl(q, k_codes, v_codes, block_table, max_pages_per_seq, context_lens, out,
                         B, q_len, h_q, h_kv, d, num_pages, page_size, window, 0, scale,
                         TL_FP8_E4M3, workspace, workspace_bytes, error_word, stream,
                         tl::NewRows(), k_scales, v_scales);
}

extern "C" tl_status tl_paged_attn_decode_multi(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* context_lens, float* out, int32_t B, int32_t q_len,
    int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages, int32_t page_size, int32_t window,
    float scale, tl_dtype dtype, void* workspace, size_t workspace_bytes, uint32_t* error_word,
    void* stream) {
  return tl::decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, context_lens, out,
                         B, q_len, h_q, h_kv, d, num_pages, page_size, window, 0, scale, dtype,
                         workspace, workspace_bytes, error_word, stream);
}
