// PAGED_ATTENTION, batched right-aligned prefill, folded over key tiles with
// an online softmax ("How serving works in Tlaloc", section 1: right-aligned
// rows, padding at slot -1, causal length = position + 1; section 2: a row's
// pages are gathered once for all its tokens, and "Blockwise attention": the
// keys are folded block by block into a running max, sum and P.V, so no score
// tensor wider than one tile exists).
//
// Four launches, the last three programmatic dependents of their predecessor
// (resident while it finishes, waiting for its results).  A pre-pass converts
// the V rows each row's tokens can see from the bf16 pages to fp16, once,
// into the workspace, laid out as [row][KV head][key][d] (exact for |v| in
// [2^-14, 65504]; larger finite values are reported; keys past the row's
// last position are zeros), notes whether any of them exceeds 8 in
// magnitude, and counts each query-tile pair's key tiles; a one-CTA plan
// orders the pairs heaviest first and sets each row's flag.  Then the
// persistent attention kernel (one CTA per SM) takes work items (pair of
// query tiles, KV head, row) and runs them on the 5th-generation tensor
// core: once for the rows without a flag (P as one fp16 value), then once
// for the flagged rows (P as the sum of two fp16 parts), each launch
// skipping the other's rows.  A query tile packs tokens_per_tile =
// 128/group consecutive tokens of one row with all `group` query heads that
// share the KV head, as the 128 M rows (row r = token r/group, head
// r%group); the CTA holds two consecutive tiles (Q0, Q1), so every K/V tile
// it streams feeds 256 rows.  Keys are folded in tiles of 128 over the range
// the CTA's live tokens can see ([min lo, max p]); every MMA is M=128 x
// N=128 x K=16 (N = keys for S, the head dimension for P.V).
//   warp 0      TMA producer: Q0 and Q1 once (a 3-D map (d, H_q, token), box
//               64 x group x tokens), then K and V tiles into rings of kTcKS /
//               kTcVS stages: K in boxes of 8 or 16 rows of the pool map (one
//               page run each; boxes past the sequence or on bad pages load
//               zeros), V as two 64 x 128 boxes of the fp16 workspace.
//   warp 1      TMEM owner (512 columns: S0/P0 [0,128), S1/P1 [128,256),
//               O0 [256,384), O1 [384,512)) and MMA issuer (one lane), in the
//               order PV0_j, S0_{j+1}, PV1_j, S1_{j+1}: S_a = Q_a K^T (8 MMAs,
//               bf16 operands from shared-memory descriptors), O_a += P_a V
//               (8 MMAs, fp16, A read from TMEM).
//   warps 2-5   softmax for Q0, warps 6-9 for Q1, one thread per M row: load
//               the row of S_a (four 32-column loads, one wait), mask by the
//               row's causal / window range (skipped when the whole warp sees
//               only live keys), running max in log2 units with a lazy
//               rescale (O and the sum change only when the max grows by
//               more than 2^8), write P rounded to fp16 into the first 64
//               columns of S_a, and add the rounded values to the row sum;
//               finally the epilogue: O / l staged in shared memory the
//               finished tile no longer needs, written by TMA stores.
// P is rounded to fp16 rather than bf16: bf16's 8-bit significand makes the
// weights of a peaked softmax off by up to 2^-9, which moves an output by
// several 1e-3 when |V| is a few units; fp16's 11 bits and a sum over the same
// rounded weights keep the output a convex combination of V rows with
// weights within 2^-11 relative.  V is converted once per call rather than
// per CTA: every V tile feeds all the CTAs of its row and head, and a
// conversion inside the attention kernel would add two shared-memory passes
// per tile per CTA next to the tensor core's own operand reads, which
// already use most of that bandwidth.
// While one warpgroup computes softmax on its tile, the tensor core works on
// the other tile, so the two overlap.  P_a aliases S_a: S_a(j+1) is issued
// after PV_a(j) and the tensor core runs a thread's MMAs in order, and when
// S_a(j+1) is complete so is PV_a(j) (its O is stable for a rescale).  A CTA
// never touches another row and its arithmetic does not depend on B, so a row
// gives the same bits batched or alone.  All waits are bounded.
#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace tl {

// Prefill step trace, a build option (-DTL_PREFILL_TRACE=1; the default
// library has none of it): the MMA-issuing thread of each attention CTA adds
// its clock64 cycles from its first item to its last, its 128-key steps (one
// step: both query tiles' S and P.V over one key tile), its items, and the
// cycles it spent waiting for the softmax warps' P and for the producer's K
// and V tiles; the first warp of each softmax warpgroup adds the cycles it
// waited for S and the cycles from S's arrival to its P's release; all to
// its CTA's row of a device array read by tl_prefill_trace_read (both
// launches of a call add to the same rows).
#ifndef TL_PREFILL_TRACE
#define TL_PREFILL_TRACE 0
#endif
#if TL_PREFILL_TRACE
constexpr int kPtraceCtas = 1024;
__device__ unsigned long long g_ptrace[kPtraceCtas][TL_PTRACE_FIELDS];
__device__ __forceinline__ long long ptrace_clk() { return clock64(); }
#else
__device__ __forceinline__ long long ptrace_clk() { return 0; }
#endif

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
  int32_t n_pairs;       // query-tile pairs per row
  int32_t* pair_tiles;   // [B][n_pairs] key tiles each pair reads (0: no live token)
  int32_t* order;        // [B * n_pairs] pairs, most key tiles first
  int32_t* row_start;    // [B] first key of each row's fp16 V copy (a multiple of kBN)
  int32_t v_keys;        // keys per row (and KV head) of the fp16 V copy
  int32_t ring_pages;    // > 0: the table's first ring_pages entries are a ring
  int32_t kv8;           // e4m3 or int8 pools: K is read from a bf16 copy like V
  uint16_t* ws_k;        // the bf16 copy of K, laid out like the V copy
  const float* k_scales; // int8 pools: the pools' scales, [num_pages][h_kv][page_size]
  const float* v_scales;
  float* ws_ks;          // int8 pools: each copied key's scales, [B][h_kv][v_keys]
  float* ws_vs;
  float* ws_ivs;         // and 1 / its V scale (0 for a zero scale)
  int32_t* ctrl;         // [0], [1] work counters of the two attention kernels,
                         // [2] first work item of the flagged rows
  int32_t cvt_gx;        // pre-pass CTAs per row (64-key tiles of the V copy)
  int32_t* cta_big;      // [B][cvt_gx] 1: the pre-pass CTA saw a V value with |v| > 8
  int32_t* row_big;      // [B] 1: the row reads a V value with |v| > 8 (P split in two)
  uint16_t* ws_kt;       // 16-bit pools read by the all-TS kernel: an fp16 K^T copy,
                         // [B][h_kv][key tile][d][128 keys] (else null)
};

// Position bound of the call: the table width, or none for a ring (whose
// positions are not bounded by its width).
__host__ __device__ __forceinline__ int64_t position_cap(const PrefillParams& P) {
  return P.ring_pages > 0 ? (int64_t)INT32_MAX + 1 : (int64_t)P.max_pages_per_seq * P.page_size;
}
// Block-table entry index of logical block blk ("How serving works in
// Tlaloc", section 3, windowed KV pool: block blk lives on ring page
// blk % ring_pages).
__device__ __forceinline__ int table_index(const PrefillParams& P, int blk) {
  return P.ring_pages > 0 ? blk % P.ring_pages : blk;
}

constexpr int kBN = 128;             // keys per tile
#ifndef TL_PREFILL_QB
#define TL_PREFILL_QB 3
#endif
#ifndef TL_PREFILL_KS
#define TL_PREFILL_KS 2
#endif
#ifndef TL_PREFILL_VS
#define TL_PREFILL_VS 2
#endif
constexpr int kTcQB = TL_PREFILL_QB;  // query-tile buffers (two in use, one filling)
constexpr int kTcQBI8 = 2;           // int8 pools: two (the key-scale ring takes the third's room)
constexpr int kScR = 4;              // int8 pools: key-scale tiles in flight
constexpr int kScBytes = 3 * 128 * 4;  // one key tile's K scales, V scales and 1 / V scales
constexpr int kTcKS = TL_PREFILL_KS;  // K stages
constexpr int kTcVS = TL_PREFILL_VS;  // V stages
constexpr int kTcWarps = 10;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kItemSlots = 4;        // work items fetched ahead of their use
constexpr int kItemReaders = kTcWarps - 1;  // the MMA warp and the eight softmax warps
constexpr int kCvtThreads = 256;
constexpr int kTcQBytes = 32768;     // one query tile: 128 rows x 128 d x bf16
constexpr int kTcKVBytes = kBN * 256;  // 128 keys x 128 d x 16-bit (two 16 KiB halves)
constexpr int kTcSmem = kTcQB * kTcQBytes + (kTcKS + kTcVS) * kTcKVBytes + 1024;
constexpr int kTcSmemI8 = kTcQBI8 * kTcQBytes + (kTcKS + kTcVS) * kTcKVBytes + kScR * kScBytes + 1024;
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 8192;   // two halves (rows without and with the split-P flag);
                                     // key-tile counts at or above 4095 share a half's last bucket

// Workspace layout: [counter | pair_tiles | order | row_start | fp16 V
// (| bf16 K for e4m3 pools)], each part 256-byte aligned; the copies are
// [B][h_kv][v_keys][128].
struct WsLayout {
  size_t tiles, order, rows, cta_big, row_big, v, k, ks, vs, ivs, kt, total;
};
constexpr int kCvtKeys = 64;  // keys per pre-pass CTA (divides kBN)
// kv8: e4m3 or int8 pools (a bf16 copy of K); i8: int8 pools (and the keys'
// scales, [B][h_kv][v_keys] f32 each: K, V and 1 / V).
// kt: 16-bit pools read by the all-TS attention kernel (an fp16 K^T copy
// the size of the V copy).
inline WsLayout ws_layout(int64_t B, int64_t n_pairs, int64_t h_kv, int64_t v_keys, bool kv8,
                          bool i8 = false, bool kt = false) {
  const size_t pairs = (size_t)(B * n_pairs) * 4;
  const size_t copy = (size_t)B * h_kv * (size_t)v_keys * 128 * 2;
  const size_t gx = (size_t)((v_keys + kCvtKeys - 1) / kCvtKeys);
  WsLayout L;
  L.tiles = 256;
  L.order = L.tiles + align_up(pairs, 256);
  L.rows = L.order + align_up(pairs, 256);
  L.cta_big = L.rows + align_up((size_t)B * 4, 256);
  L.row_big = L.cta_big + align_up((size_t)B * gx * 4, 256);
  L.v = L.row_big + align_up((size_t)B * 4, 256);
  L.k = L.v + copy;
  const size_t scales = align_up((size_t)B * h_kv * (size_t)v_keys * 4, 256);
  L.ks = L.k + (kv8 ? copy : 0);
  L.vs = L.ks + (i8 ? scales : 0);
  L.ivs = L.vs + (i8 ? scales : 0);
  L.kt = L.ivs + (i8 ? scales : 0);
  L.total = L.kt + (kt ? copy : 0);
  return L;
}
// The all-TS attention kernel (prefill_ts.cuh), a build option
// (-DTL_PREFILL_ALL_TS=1; the default library keeps the paired SS/TS
// kernel, which measured faster: the single-tile chain exposes the MMAs'
// completion latency).  With it, the calls that take it: 16-bit pools with
// 1, 2, 4, 8 or 16 KV heads (a power-of-two unit count for the pre-pass's
// K^T copy); d is 128 for every prefill call.
#ifndef TL_PREFILL_ALL_TS
#define TL_PREFILL_ALL_TS 0
#endif
inline bool ts_path(tl_dtype dtype, int64_t h_kv) {
  return TL_PREFILL_ALL_TS && dtype == TL_BF16 && h_kv >= 1 && h_kv <= 16 &&
         (h_kv & (h_kv - 1)) == 0;
}
// Keys per row of the V copy: the table's positions, or for a ring the
// ring's positions plus the rounding of the copy's start and end to tiles.
// Always whole 128-key tiles, so a key tile of a row lies wholly inside or
// wholly outside its copy.
inline int64_t v_copy_keys(int64_t max_pages_per_seq, int64_t page_size, int64_t ring_pages) {
  if (ring_pages > 0) return align_up((size_t)(ring_pages * page_size), kBN) + 2 * kBN;
  return align_up((size_t)(max_pages_per_seq * page_size), kBN);
}
// Keys per row of a copy that holds any row whose tokens read at most
// max_row_keys keys (from the first key its first token sees to its last
// position): the span plus the rounding of its start and end to tiles.
inline int64_t v_copy_keys_for_span(int64_t max_row_keys) {
  return align_up((size_t)max_row_keys, kBN) + 2 * kBN;
}
#ifndef TL_PREFILL_REREAD_CH
#define TL_PREFILL_REREAD_CH 1
#endif
constexpr int kRereadCh = TL_PREFILL_REREAD_CH;  // 32-column chunks of S reread per TMEM round trip
constexpr int64_t kMinCopyKeys = 3 * kBN;  // the smallest copy a call accepts (one key + rounding)
constexpr uint32_t kTcCols = 512;
constexpr float kRescaleLog2 = 8.f;
// bf16 bit patterns (sign cleared) of the finite values fp16 cannot hold:
// [65536, max finite]; 65280 (0x477F) is the largest bf16 below fp16's
// overflow threshold.
constexpr uint32_t kBf16TooBig = 0x4780u, kBf16Inf = 0x7F80u;
// A row whose V holds a value of magnitude above 8 (bf16 bits 0x4100, e4m3
// code 0x50, sign cleared; NaN and infinities included) takes P.V with P
// split into two fp16 parts.  P rounded once to fp16 moves an output by up
// to 2^-11 * max |v_j - o|: far below 1e-3 for V of N(0,1) scale (|v| < 8),
// but up to several 1e-3 for values beyond 8; hi + lo carries about 22
// significant bits.
constexpr uint32_t kBf16Big = 0x4100u, kE4m3Big = 0x50u;
// ... or whose V has a root mean square above 1.25 over a 64-key tile of the
// pre-pass (N(0, 1) values have 1.0): the rounding error of one fp16 P grows
// with the spread of V as well as with its largest value.
constexpr float kRmsBig2 = 1.5625f;  // 1.25^2

// Sum of squares of eight fp16 values.
__device__ __forceinline__ float sumsq_f16x8(uint4 h) {
  float a = 0.f;
  const uint32_t w[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float lo, hi;
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
        : "=f"(lo), "=f"(hi)
        : "r"(w[k]));
    a = fmaf(lo, lo, a);
    a = fmaf(hi, hi, a);
  }
  return a;
}

struct TcShared {
  unsigned long long q_full[kTcQB], q_free[kTcQB];
  unsigned long long k_full[kTcKS], k_empty[kTcKS], v_full[kTcVS], v_empty[kTcVS];
  unsigned long long s_full[2], p_full[2], o_done[2], o_free[2], stg_full[2], stg_free[2];
  unsigned long long item_full[kItemSlots], item_empty[kItemSlots], mma_drain;
  unsigned long long sc_full[kScR], sc_empty[kScR];  // int8 pools: the key-scale ring
  int item[kItemSlots];
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

// Two f32 -> one f16x2 register (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// The two halves of an f16x2 register as f32 (exact).
__device__ __forceinline__ void unpack_f16x2(uint32_t x, float& lo, float& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
      : "=f"(lo), "=f"(hi)
      : "r"(x));
}
// (d0, d1) = (a0, a1) * b + c, two f32 FMAs in one packed instruction
// (b and c hold the same value twice).
__device__ __forceinline__ void fma_f32x2(float a0, float a1, uint64_t b, uint64_t c, float& d0,
                                          float& d1) {
  uint64_t a, d;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(a) : "f"(a0), "f"(a1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(d0), "=f"(d1) : "l"(d));
}
__device__ __forceinline__ uint64_t f32_twice(float x) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};\n" : "=l"(r) : "f"(x));
  return r;
}
// acc + lo + hi of an f16x2 register, each half widened exactly to f32 by
// the add itself.
__device__ __forceinline__ float add_f16x2_halves(float acc, uint32_t x) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n add.rn.f32.f16 %0, l, %0;\n"
      " add.rn.f32.f16 %0, h, %0;\n}\n"
      : "+f"(acc)
      : "r"(x));
  return acc;
}
// Two bf16 (one register) -> two fp16 (one register).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  return pack_f16x2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}
// (s0, s1) += (a0, a1)^2 in one packed f32 FMA.
__device__ __forceinline__ void sq_acc_f32x2(float a0, float a1, float& s0, float& s1) {
  uint64_t a, acc;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(acc) : "f"(s0), "f"(s1));
  asm("fma.rn.f32x2 %0, %1, %1, %0;\n" : "+l"(acc) : "l"(a));
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(s0), "=f"(s1) : "l"(acc));
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// ------------------------------------------------------- V pre-pass --
// Grid (64-key tile, row).  Each CTA first finds its row's live
// positions [pmin, pmax]; the attention kernel reads V keys in
// [start, end): start = the first key any live token can see, rounded down
// to its 128-key tile, end = pmax + 1 rounded up to a 128-key tile (clamped
// to the workspace).
// The tile's page numbers go to shared memory; then every thread moves
// 16-byte units (key-major: one key's h_kv x 128 values are contiguous in
// the pool), kCvtUnroll independent loads in flight.
constexpr int kCvtUnroll = 8;
constexpr int kCvtBlocksPerSm = 4;  // register bound: the scan and page-lookup phases of
                                    // one CTA overlap the copies of the others

// Two e4m3 codes (low byte first) as an fp16 pair, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  const uint16_t c = (uint16_t)two;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(c));
  return r;
}
// Two e4m3 codes as a bf16 pair, exact (every e4m3 value is a bf16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  float lo, hi;
  unpack_f16x2(e4m3x2_to_f16x2(two), lo, hi);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight int8 codes (low byte first) as fp16 and as bf16 values, exact (every
// integer of magnitude at most 128 is both).
__device__ __forceinline__ void i8x8_to_f16_bf16(uint2 c, uint4& f16, uint4& bf16) {
  uint32_t h[4], b[4];
  const uint32_t w[2] = {c.x, c.y};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t word = w[k >> 1] >> (16 * (k & 1));
    const float lo = (float)(int8_t)(word & 0xffu), hi = (float)(int8_t)((word >> 8) & 0xffu);
    h[k] = pack_f16x2(lo, hi);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(b[k]) : "f"(hi), "f"(lo));
  }
  f16 = make_uint4(h[0], h[1], h[2], h[3]);
  bf16 = make_uint4(b[0], b[1], b[2], b[3]);
}
// Eight int8 codes times one scale, each product rounded to fp16.
__device__ __forceinline__ uint4 i8x8_scaled_f16(uint2 c, float sc) {
  uint32_t h[4];
  const uint32_t w[2] = {c.x, c.y};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t word = w[k >> 1] >> (16 * (k & 1));
    h[k] = pack_f16x2((float)(int8_t)(word & 0xffu) * sc, (float)(int8_t)((word >> 8) & 0xffu) * sc);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}
// Largest |code| of eight int8 codes.
__device__ __forceinline__ uint32_t i8x8_max_abs(uint2 c) {
  const uint32_t m = __vmaxu4(__vabsss4(c.x), __vabsss4(c.y));
  return max(max(m & 0xffu, (m >> 8) & 0xffu), max((m >> 16) & 0xffu, m >> 24));
}

// KIND 0: bf16 pools (V to fp16); 1: e4m3 pools (V to fp16, K to bf16);
// 2: int8 pools (K codes to bf16; V to fp16 as codes in a tile with the
// split-P flag, else as code x V scale; and each key's scales).
template <int KIND>
__global__ void __launch_bounds__(kCvtThreads, kCvtBlocksPerSm)
    prefill_v_f16_kernel(PrefillParams P, uint16_t* __restrict__ ws, int* counter) {
  constexpr bool KV8 = KIND != 0;  // one byte per element
  __shared__ int s_min[kCvtThreads / 32], s_max[kCvtThreads / 32];
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    counter[0] = 0;  // work items of the single-fp16 attention kernel
    counter[1] = 0;  // and of the split-P one
  }
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __shared__ int s_page[kCvtKeys];  // page of each key of the tile; -1: write zeros
  __shared__ int s_slot[kCvtKeys];  // its slot in the pool (-1 with the page)
  const int b = (int)blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t cap = position_cap(P);
  if (blockIdx.x == 0) {
    // the key tiles every query-tile pair of row b reads (the attention
    // kernel's own range rule), for the heaviest-first order
    const int span = 2 * (128 / P.group);
    for (int qp = warp; qp < P.n_pairs; qp += kCvtThreads / 32) {
      int kmin = INT32_MAX, kmax = -1;
      for (int i = lane; i < span; i += 32) {
        const int t = qp * span + i;
        if (t >= P.T) break;
        const int p = P.positions[(size_t)b * P.T + t];
        if (p >= 0 && p < cap) {
          kmin = min(kmin, (P.window > 0 && p - P.window + 1 > 0) ? p - P.window + 1 : 0);
          kmax = max(kmax, p);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
        kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
      }
      if (lane == 0)
        P.pair_tiles[(size_t)b * P.n_pairs + qp] = kmax >= 0 ? kmax / kBN - kmin / kBN + 1 : 0;
    }
  }
  int pmin = INT32_MAX, pmax = -1;
#pragma unroll 8
  for (int t = threadIdx.x; t < P.T; t += kCvtThreads) {  // eight loads in flight
    const int p = __ldg(P.positions + (size_t)b * P.T + t);
    if (p >= 0 && p < cap) {
      pmin = min(pmin, p);
      pmax = max(pmax, p);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
    pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
  }
  if (lane == 0) {
    s_min[warp] = pmin;
    s_max[warp] = pmax;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kCvtThreads / 32; ++w) {
    pmin = min(pmin, s_min[w]);
    pmax = max(pmax, s_max[w]);
  }
  int32_t* big_flag = P.cta_big + (size_t)b * P.cvt_gx + blockIdx.x;
  if (pmax < 0) {  // no live token: the attention kernel reads nothing
    if (blockIdx.x == 0 && threadIdx.x == 0) P.row_start[b] = 0;
    if (threadIdx.x == 0) *big_flag = 0;
    return;
  }
  const int lo = (P.window > 0 && pmin - P.window + 1 > 0) ? pmin - P.window + 1 : 0;
  const int start = lo / kBN * kBN;
  const int end = (int)min((int64_t)(pmax / kBN + 1) * kBN, (int64_t)start + P.v_keys);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    P.row_start[b] = start;
    // the copy holds v_keys keys per row (the workspace's size): a row that
    // reads more, within the table's positions, is reported (its outputs
    // are undefined; nothing is read or written outside the workspace)
    if (pmax - start + 1 > P.v_keys) report(P.error_word, TL_DEVERR_CONTEXT_RANGE);
    // a ring holds the call only if every key a token needs is still in it:
    // the call spans lo..pmax, at most ring_pages * page_size positions
    if (P.ring_pages > 0 && (int64_t)pmax - lo + 1 > (int64_t)P.ring_pages * P.page_size)
      report(P.error_word, TL_DEVERR_CONTEXT_RANGE);
  }
  const int k0 = start + (int)blockIdx.x * kCvtKeys;  // this CTA's keys of the copy
  if (k0 >= end) {
    if (threadIdx.x == 0) *big_flag = 0;
    return;
  }
  for (int r = threadIdx.x; r < kCvtKeys; r += kCvtThreads) {
    const int k = k0 + r;
    int page = -1;  // keys past pmax: zeros
    if (k <= pmax) {
      page = __ldg(P.block_table + (size_t)b * P.max_pages_per_seq + table_index(P, k / P.page_size));
      if (page < 0 || page >= P.num_pages) {
        report(P.error_word, TL_DEVERR_PAGE_RANGE);
        page = -1;  // bad page: zeros
      }
    }
    s_page[r] = page;
    s_slot[r] = page < 0 ? -1 : page * P.page_size + k % P.page_size;
  }
  __syncthreads();
  const int r0 = 0, r1 = min(end - k0, kCvtKeys);  // keys of the tile to write
  float sumsq = 0.f;    // sum of squares of this thread's live V values
  int n_vals = 0;       // and their count
  if constexpr (KIND == 2) {
    // int8 pools, two passes over the tile's V codes.  First the tile's
    // split-P flag (some |code x v_scale| above 8, NaN included, or an RMS
    // above 1.25); then the copies.  A flagged tile keeps V as its codes
    // (exact in fp16; the attention kernel applies the V scales to the
    // probabilities), any other tile is copied as fp16(code x v_scale) with
    // unit V scales beside it, so that a row with no flagged tile takes P.V
    // exactly as 16-bit pools do.  K is copied as its codes (bf16, exact).
    const int units = P.h_kv * 16;  // 8-code units per key
    const int total = (r1 - r0) * units;
    const uint8_t* v8 = reinterpret_cast<const uint8_t*>(P.v_cache);
    const uint8_t* k8 = reinterpret_cast<const uint8_t*>(P.k_cache);
    // unit idx of the tile: key r, unit u (a shift and a mask when the unit
    // count is a power of two, as for 1, 2, 4, 8 or 16 KV heads)
    const int ushift = (units & (units - 1)) == 0 ? __ffs(units) - 1 : -1;
    auto split_idx = [&](int idx, int& r, int& u) {
      if (ushift >= 0) {
        r = r0 + (idx >> ushift);
        u = idx & (units - 1);
      } else {
        r = r0 + idx / units;
        u = idx - (r - r0) * units;
      }
    };
    // a key's scale of KV head g: [page][g][position in the page]
    auto scale_index = [&](int r, int g) {
      const int in_page = s_slot[r] - s_page[r] * P.page_size;
      return ((size_t)s_page[r] * P.h_kv + g) * P.page_size + in_page;
    };
    bool big_i8 = false;
    for (int base = 0; base < total; base += kCvtThreads * kCvtUnroll) {
      uint2 c[kCvtUnroll];
      float vs[kCvtUnroll];
#pragma unroll
      for (int i = 0; i < kCvtUnroll; ++i) {
        const int idx = base + i * kCvtThreads + (int)threadIdx.x;
        c[i] = make_uint2(0u, 0u);
        vs[i] = 0.f;
        if (idx < total) {
          int r, u;
          split_idx(idx, r, u);
          if (s_page[r] >= 0) {
            const size_t row = (size_t)s_slot[r] * P.h_kv * 128;
            c[i] = __ldg(reinterpret_cast<const uint2*>(v8 + row) + u);
            vs[i] = __ldg(P.v_scales + scale_index(r, u >> 4));
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kCvtUnroll; ++i) {
        const int idx = base + i * kCvtThreads + (int)threadIdx.x;
        int r = 0, u = 0;
        if (idx < total) split_idx(idx, r, u);
        if (idx < total && s_page[r] >= 0) {
          uint4 f16, bf16;
          i8x8_to_f16_bf16(c[i], f16, bf16);
          big_i8 |= !((float)i8x8_max_abs(c[i]) * vs[i] <= 8.f);
          sumsq = fmaf(sumsq_f16x8(f16), vs[i] * vs[i], sumsq);
          n_vals += 8;
        }
      }
    }
    // the tile's flag: a fixed-order reduction (it must repeat bit for bit)
    __shared__ float s_sq2[kCvtThreads / 32];
    __shared__ int s_n2[kCvtThreads / 32];
    __shared__ int s_big;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sumsq += __shfl_xor_sync(0xffffffffu, sumsq, o);
      n_vals += __shfl_xor_sync(0xffffffffu, n_vals, o);
    }
    if (lane == 0) {
      s_sq2[warp] = sumsq;
      s_n2[warp] = n_vals;
    }
    const int any_big = __syncthreads_or(big_i8);
    if (threadIdx.x == 0) {
      float tot = 0.f;
      int cnt = 0;
      for (int w = 0; w < kCvtThreads / 32; ++w) {
        tot += s_sq2[w];
        cnt += s_n2[w];
      }
      const bool wide = !(tot <= kRmsBig2 * (float)cnt);  // NaN counts as wide
      s_big = (any_big || wide) ? 1 : 0;
      *big_flag = s_big;
    }
    __syncthreads();
    const bool tile_big = s_big != 0;
    // each key's K scale and (a flagged tile) V scale per KV head, or unit V
    // scales (0 for keys past pmax and bad pages, whose copies are 0)
    for (int idx = threadIdx.x; idx < (r1 - r0) * P.h_kv; idx += kCvtThreads) {
      const int r = r0 + idx / P.h_kv, g = idx % P.h_kv;
      float ksc = 0.f, vsc = 0.f;
      if (s_page[r] >= 0) {
        ksc = __ldg(P.k_scales + scale_index(r, g));
        vsc = tile_big ? __ldg(P.v_scales + scale_index(r, g)) : 1.f;
      }
      const size_t di = ((size_t)b * P.h_kv + g) * P.v_keys + (k0 - start + r);
      P.ws_ks[di] = ksc;
      P.ws_vs[di] = vsc;
      P.ws_ivs[di] = vsc > 0.f ? 1.f / vsc : 0.f;
    }
    for (int base = 0; base < total; base += kCvtThreads * kCvtUnroll) {
      uint2 a[kCvtUnroll], c[kCvtUnroll];
      float vs[kCvtUnroll];
#pragma unroll
      for (int i = 0; i < kCvtUnroll; ++i) {
        const int idx = base + i * kCvtThreads + (int)threadIdx.x;
        a[i] = c[i] = make_uint2(0u, 0u);
        vs[i] = 0.f;
        if (idx < total) {
          int r, u;
          split_idx(idx, r, u);
          if (s_page[r] >= 0) {
            const size_t row = (size_t)s_slot[r] * P.h_kv * 128;
            a[i] = __ldg(reinterpret_cast<const uint2*>(v8 + row) + u);
            c[i] = __ldg(reinterpret_cast<const uint2*>(k8 + row) + u);
            if (!tile_big) vs[i] = __ldg(P.v_scales + scale_index(r, u >> 4));
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kCvtUnroll; ++i) {
        const int idx = base + i * kCvtThreads + (int)threadIdx.x;
        if (idx < total) {
          int r, u;
          split_idx(idx, r, u);
          const size_t dst =
              (((size_t)b * P.h_kv + (u >> 4)) * P.v_keys + (k0 - start + r)) * 128 + (u & 15) * 8;
          uint4 f16, bf16;
          i8x8_to_f16_bf16(a[i], f16, bf16);
          *reinterpret_cast<uint4*>(ws + dst) = tile_big ? f16 : i8x8_scaled_f16(a[i], vs[i]);
          i8x8_to_f16_bf16(c[i], f16, bf16);
          *reinterpret_cast<uint4*>(P.ws_k + dst) = bf16;
        }
      }
    }
    return;
  }
  const int units = P.h_kv * 16;                                // 16-byte units per key
  const int total = (r1 - r0) * units;
  uint32_t vmax = 0;  // max |bf16 bits| seen, per half-word
  uint32_t cmax = 0;  // e4m3 pools: max |code| seen, per byte
  if ((units & (units - 1)) == 0 && units <= kCvtThreads) {
    // a power-of-two unit count: each thread keeps one unit u of every
    // kpp-th key, so its source and destination offsets are fixed but for
    // the key (no division per unit); 8 keys' loads in flight
    const int kpp = kCvtThreads / units;
    const int u = (int)threadIdx.x & (units - 1), kof = (int)threadIdx.x / units;
    const size_t dst0 =
        (((size_t)b * P.h_kv + (u >> 4)) * P.v_keys + (k0 - start)) * 128 + (u & 15) * 8;
    const int nkeys = r1 - r0;
    float sq0 = 0.f, sq1 = 0.f;  // bf16 pools: two sums of squares (packed FMAs)
    for (int rb = kof; rb < nkeys; rb += kpp * kCvtUnroll) {
      uint4 x[kCvtUnroll];  // bf16 V, or (e4m3) V in .x.y and K in .z.w
#pragma unroll
      for (int i = 0; i < kCvtUnroll; ++i) {
        const int r = rb + i * kpp;
        x[i] = make_uint4(0u, 0u, 0u, 0u);
        const int slot = r < nkeys ? s_slot[r] : -1;
        if (slot >= 0) {
          const size_t row = (size_t)slot * P.h_kv * 128;
          if (KV8) {
            const uint2 a = __ldg(reinterpret_cast<const uint2*>(
                                      reinterpret_cast<const uint8_t*>(P.v_cache) + row) + u);
            const uint2 c = __ldg(reinterpret_cast<const uint2*>(
                                      reinterpret_cast<const uint8_t*>(P.k_cache) + row) + u);
            x[i] = make_uint4(a.x, a.y, c.x, c.y);
          } else {
            x[i] = __ldg(reinterpret_cast<const uint4*>(P.v_cache + row) + u);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kCvtUnroll; ++i) {
        const int r = rb + i * kpp;
        if (r >= nkeys) break;
        const size_t dst = dst0 + (size_t)r * 128;
        const uint4 y = x[i];
        const bool live = s_slot[r] >= 0;
        if (KV8) {  // e4m3 values are exact in both fp16 and bf16
          cmax = __vmaxu4(cmax, __vmaxu4(y.x & 0x7f7f7f7fu, y.y & 0x7f7f7f7fu));
          const uint4 f16 = make_uint4(e4m3x2_to_f16x2(y.x), e4m3x2_to_f16x2(y.x >> 16),
                                       e4m3x2_to_f16x2(y.y), e4m3x2_to_f16x2(y.y >> 16));
          *reinterpret_cast<uint4*>(ws + dst) = f16;
          sumsq += sumsq_f16x8(f16);  // zeros for a dead key
          *reinterpret_cast<uint4*>(P.ws_k + dst) =
              make_uint4(e4m3x2_to_bf16x2(y.z), e4m3x2_to_bf16x2(y.z >> 16),
                         e4m3x2_to_bf16x2(y.w), e4m3x2_to_bf16x2(y.w >> 16));
        } else {
          vmax = max_u16x2(vmax, max_u16x2(max_u16x2(y.x & 0x7fff7fffu, y.y & 0x7fff7fffu),
                                           max_u16x2(y.z & 0x7fff7fffu, y.w & 0x7fff7fffu)));
          const uint32_t w[4] = {y.x, y.y, y.z, y.w};
          uint32_t h[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // the bf16 pair as f32 (exact): fp16 for the copy, squares for the RMS
            const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
            h[k] = pack_f16x2(lo, hi);
            sq_acc_f32x2(lo, hi, sq0, sq1);
          }
          *reinterpret_cast<uint4*>(ws + dst) = make_uint4(h[0], h[1], h[2], h[3]);
        }
        n_vals += live ? 8 : 0;
      }
    }
    sumsq += sq0 + sq1;
    if (KIND == 0 && P.ws_kt != nullptr) {
      // the fp16 K^T copy of the all-TS attention kernel: per KV head, key
      // tile and d, the tile's 128 keys; this CTA's 64 keys are one half of
      // a tile.  A thread takes a block of 8 keys x 8 d (eight 16-byte row
      // reads), transposes it in registers (byte permutes of fp16 halves)
      // and writes 8 d rows of 8 keys, 16 bytes each; keys past the CTA's
      // range and of bad pages are zeros
      const int kr0 = k0 - start, kofs = kr0 % kBN;
      const size_t tile_row = (size_t)(kr0 / kBN) * kBN;
      bool k_over = false;
      for (int blk = threadIdx.x; blk < (kCvtKeys / 8) * units; blk += kCvtThreads) {
        const int uu = blk & (units - 1), kg = blk / units;
        const int g = uu >> 4, d8 = (uu & 15) * 8;
        uint32_t h[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = kg * 8 + i;
          const int slot = r < nkeys ? s_slot[r] : -1;
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (slot >= 0) x = __ldg(reinterpret_cast<const uint4*>(P.k_cache + (size_t)slot * P.h_kv * 128) + uu);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t lo = w[k] & 0x7fffu, hi = (w[k] >> 16) & 0x7fffu;
            k_over |= (lo >= kBf16TooBig && lo < kBf16Inf) || (hi >= kBf16TooBig && hi < kBf16Inf);
            h[i][k] = bf16x2_to_f16x2(w[k]);
          }
        }
        uint16_t* dst0 = P.ws_kt + ((size_t)(b * P.h_kv + g) * P.v_keys + tile_row + d8) * 128 +
                         kofs + kg * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {  // d row d8 + e: keys (2w, 2w + 1) in word w
          const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
          const uint4 out = make_uint4(__byte_perm(h[0][e >> 1], h[1][e >> 1], sel),
                                       __byte_perm(h[2][e >> 1], h[3][e >> 1], sel),
                                       __byte_perm(h[4][e >> 1], h[5][e >> 1], sel),
                                       __byte_perm(h[6][e >> 1], h[7][e >> 1], sel));
          *reinterpret_cast<uint4*>(dst0 + (size_t)e * 128) = out;
        }
      }
      if (k_over) report(P.error_word, TL_DEVERR_VALUE_RANGE);
    }
  } else
  // units of 8 elements: 16 bytes of a bf16 row, 8 bytes of an e4m3 row
  for (int base = 0; base < total; base += kCvtThreads * kCvtUnroll) {
    uint4 x[kCvtUnroll];  // bf16 V, or (e4m3) V in .x.y and K in .z.w
#pragma unroll
    for (int i = 0; i < kCvtUnroll; ++i) {
      const int idx = base + i * kCvtThreads + (int)threadIdx.x;
      x[i] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < total) {
        const int r = r0 + idx / units, u = idx % units;
        const int page = s_page[r];
        if (page >= 0) {
          const size_t row = ((size_t)page * P.page_size + (k0 + r) % P.page_size) * P.h_kv * 128;
          if (KV8) {
            const uint8_t* v8 = reinterpret_cast<const uint8_t*>(P.v_cache);
            const uint8_t* k8 = reinterpret_cast<const uint8_t*>(P.k_cache);
            const uint2 a = __ldg(reinterpret_cast<const uint2*>(v8 + row) + u);
            const uint2 c = __ldg(reinterpret_cast<const uint2*>(k8 + row) + u);
            x[i] = make_uint4(a.x, a.y, c.x, c.y);
          } else {
            x[i] = __ldg(reinterpret_cast<const uint4*>(P.v_cache + row) + u);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kCvtUnroll; ++i) {
      const int idx = base + i * kCvtThreads + (int)threadIdx.x;
      if (idx < total) {
        const int r = r0 + idx / units, u = idx % units;
        const size_t dst =
            (((size_t)b * P.h_kv + (u >> 4)) * P.v_keys + (k0 - start + r)) * 128 + (u & 15) * 8;
        uint4 y = x[i];
        const bool live = s_page[r] >= 0;
        if (KV8) {  // e4m3 values are exact in both fp16 and bf16
          cmax = __vmaxu4(cmax, __vmaxu4(y.x & 0x7f7f7f7fu, y.y & 0x7f7f7f7fu));
          const uint4 f16 = make_uint4(e4m3x2_to_f16x2(y.x), e4m3x2_to_f16x2(y.x >> 16),
                                       e4m3x2_to_f16x2(y.y), e4m3x2_to_f16x2(y.y >> 16));
          *reinterpret_cast<uint4*>(ws + dst) = f16;
          if (live) sumsq += sumsq_f16x8(f16);
          *reinterpret_cast<uint4*>(P.ws_k + dst) =
              make_uint4(e4m3x2_to_bf16x2(y.z), e4m3x2_to_bf16x2(y.z >> 16),
                         e4m3x2_to_bf16x2(y.w), e4m3x2_to_bf16x2(y.w >> 16));
        } else {
          vmax = max_u16x2(vmax, max_u16x2(max_u16x2(y.x & 0x7fff7fffu, y.y & 0x7fff7fffu),
                                           max_u16x2(y.z & 0x7fff7fffu, y.w & 0x7fff7fffu)));
          y = make_uint4(bf16x2_to_f16x2(y.x), bf16x2_to_f16x2(y.y), bf16x2_to_f16x2(y.z),
                         bf16x2_to_f16x2(y.w));
          *reinterpret_cast<uint4*>(ws + dst) = y;
          if (live) sumsq += sumsq_f16x8(y);
        }
        n_vals += live ? 8 : 0;
      }
    }
  }
  const uint32_t m0 = vmax & 0xffffu, m1 = vmax >> 16;
  if ((m0 >= kBf16TooBig && m0 < kBf16Inf) || (m1 >= kBf16TooBig && m1 < kBf16Inf))
    report(P.error_word, TL_DEVERR_VALUE_RANGE);
  cmax = __vmaxu4(cmax, cmax >> 16);
  cmax = __vmaxu4(cmax, cmax >> 8);
  // the tile's V root mean square: a fixed-order reduction (the flag, and so
  // the row's arithmetic, must repeat bit for bit)
  __shared__ float s_sq[kCvtThreads / 32];
  __shared__ int s_n[kCvtThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sumsq += __shfl_xor_sync(0xffffffffu, sumsq, o);
    n_vals += __shfl_xor_sync(0xffffffffu, n_vals, o);
  }
  if (lane == 0) {
    s_sq[warp] = sumsq;
    s_n[warp] = n_vals;
  }
  const bool big = m0 > kBf16Big || m1 > kBf16Big || (cmax & 0xffu) > kE4m3Big;
  const int any_big = __syncthreads_or(big);
  if (threadIdx.x == 0) {
    float tot = 0.f;
    int cnt = 0;
    for (int w = 0; w < kCvtThreads / 32; ++w) {
      tot += s_sq[w];
      cnt += s_n[w];
    }
    const bool wide = !(tot <= kRmsBig2 * (float)cnt);  // NaN counts as wide
    *big_flag = (any_big || wide) ? 1 : 0;
  }
}

// ------------------------------------------------------------ plan --
// One CTA.  Each row's split-P flag (any of its pre-pass CTAs saw |v| > 8);
// then a counting sort of the pairs into P.order: the pairs of rows without
// the flag first, then those of flagged rows, each group by key tiles, most
// first (pairs with no live token last).  ctrl[2] = the first work item of
// the flagged rows: the single-fp16 attention kernel takes the items before
// it, the split-P kernel the rest.  Ties keep no particular order; every
// pair computes the same bits whichever CTA takes it and when.
__device__ __forceinline__ int plan_bucket(const PrefillParams& P, int e) {
  constexpr int kHalf = kPlanBuckets / 2;
  const int t = min(P.pair_tiles[e], kHalf - 1);
  return __ldcg(P.row_big + e / P.n_pairs) ? t : kHalf + t;  // a higher bucket goes first
}

__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(PrefillParams P) {
  __shared__ int cur[kPlanBuckets];  // counts, then each bucket's next slot
  __shared__ int wsum[kPlanThreads / 32];
  __shared__ int n_flagged;
  constexpr int kPer = kPlanBuckets / kPlanThreads;  // buckets per thread
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, n_e = P.B * P.n_pairs;
  for (int k = tid; k < kPlanBuckets; k += kPlanThreads) cur[k] = 0;
  if (tid == 0) n_flagged = 0;
  // the pre-pass (this grid's predecessor) writes the pair counts; the
  // attention kernel may launch now and waits for this grid in turn
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __syncthreads();
  // each row's flag, a warp per row
  for (int b = wid; b < P.B; b += kPlanThreads / 32) {
    int any = 0;
    for (int x = lane; x < P.cvt_gx; x += 32) any |= __ldcg(P.cta_big + (size_t)b * P.cvt_gx + x);
    any = __reduce_or_sync(0xffffffffu, any);
    if (lane == 0) {
      P.row_big[b] = any ? 1 : 0;
      if (any) atomicAdd(&n_flagged, 1);
    }
  }
  __syncthreads();
  if (tid == 0) P.ctrl[2] = (P.B - n_flagged) * P.n_pairs * P.h_kv;
  for (int e = tid; e < n_e; e += kPlanThreads) atomicAdd(&cur[plan_bucket(P, e)], 1);
  __syncthreads();
  // slots go to the buckets from the top down: thread t owns buckets
  // [kPer t, kPer t + kPer); above = the pairs in the buckets of higher
  // threads = total - (inclusive prefix sum over threads up to t)
  int local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) local += cur[kPer * tid + i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = lane < kPlanThreads / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane < kPlanThreads / 32) wsum[lane] = v;
  }
  __syncthreads();
  int above = wsum[kPlanThreads / 32 - 1] - (incl + (wid > 0 ? wsum[wid - 1] : 0));
#pragma unroll
  for (int i = kPer - 1; i >= 0; --i) {
    const int k = kPer * tid + i, c = cur[k];
    cur[k] = above;
    above += c;
  }
  __syncthreads();
  for (int e = tid; e < n_e; e += kPlanThreads) P.order[atomicAdd(&cur[plan_bucket(P, e)], 1)] = e;
}

// S_a = Q_a K^T into TMEM columns [128a, 128a+128): eight K=16 steps over
// the 128-byte-swizzled K-major Q and K tiles; then a commit to s_full_a.
__device__ __forceinline__ void tc_issue_s(uint32_t tmem, int a, uint32_t kbase, uint32_t qbase,
                                           uint32_t s_full_a) {
  const uint32_t idS = tc::idesc_bf16(128, kBN, 0, 0);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t off = (k >> 2) * (kTcQBytes / 2) + (k & 3) * 32;
    tc::mma_ss(tmem + a * 128, tc::sdesc(qbase + off, 16, 1024), tc::sdesc(kbase + off, 16, 1024),
               idS, k > 0);
  }
  tc::commit(s_full_a);
}
// O_a (+)= P_a V in fp16: P_a from TMEM (keys [16k, 16k+16) in columns
// [8k, 8k+8) of S_a), V MN-major from shared memory.  With `split`, P is
// hi + lo: keys [16k, 16k+16) have hi in columns 32 (k/2) + 8 (k%2) + [0, 8)
// and lo 16 columns further, and both products are accumulated.
__device__ __forceinline__ void tc_issue_pv(uint32_t tmem, int a, uint32_t vbase, bool acc,
                                            bool split) {
  const uint32_t idPV = tc::idesc_f16(128, 128, 0, 1);
  if (!split) {
#pragma unroll
    for (int k = 0; k < kBN / 16; ++k)
      tc::mma_ts(tmem + 256 + a * 128, tmem + a * 128 + 8 * k,
                 tc::sdesc(vbase + k * 2048, kTcKVBytes / 2, 1024), idPV,
                 (acc || k > 0) ? 1u : 0u);
  } else {
#pragma unroll
    for (int k = 0; k < kBN / 16; ++k) {
      const uint32_t col = tmem + a * 128 + 32 * (k >> 1) + 8 * (k & 1);
      const uint64_t vd = tc::sdesc(vbase + k * 2048, kTcKVBytes / 2, 1024);
      tc::mma_ts(tmem + 256 + a * 128, col, vd, idPV, (acc || k > 0) ? 1u : 0u);
      tc::mma_ts(tmem + 256 + a * 128, col + 16, vd, idPV, 1u);
    }
  }
}

// The P of one row of a score tile when the row's V holds a value of
// magnitude above 8: P = hi + lo, both fp16.  Keys [32q, 32q + 32) put hi in
// columns [32q, 32q + 16) of the tile's S columns (taddr: this thread's lane
// at the first of them) and the remainder lo in [32q + 16, 32q + 32), the
// columns of their own scores, so each chunk of scores is reread just before
// its P replaces it.  Returns the row's sum of the unrounded f32 values.
//
// int8 pools: P' = p x v_scale goes into P.V (hi + lo as above) and the sum
// takes p.  A tile whose V copy already carries its scales has unit scales.
template <bool I8, int CH = 1>
__device__ __forceinline__ float tc_softmax_split(uint32_t taddr, int cmin, int cmax,
                                                  bool all_live, float sc, float base,
                                                  const float* scl) {
  float ls[4] = {0.f, 0.f, 0.f, 0.f};
  const uint64_t sc2 = f32_twice(sc), nb2 = f32_twice(-base);
#pragma unroll 1
  for (int q0 = 0; q0 < kBN / 32; q0 += CH) {
  float xx[CH][32];
#pragma unroll
  for (int c = 0; c < CH; ++c) tc::ld32(taddr + 32 * (q0 + c), xx[c]);
  tc::wait_ld();
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int q = q0 + c;
    float* x = xx[c];
    if (I8) {  // int8 pools: the K scales (scl[0, 128))
#pragma unroll
      for (int c = 0; c < 32; ++c) x[c] *= scl[32 * q + c];
    }
    if (!all_live) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        x[c] = (32 * q + c >= cmin && 32 * q + c <= cmax) ? x[c] : -INFINITY;
    }
    uint32_t pk[16], pl[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float y0, y1, h0, h1;
      fma_f32x2(x[2 * i], x[2 * i + 1], sc2, nb2, y0, y1);
      const float e0 = fast_exp2(y0), e1 = fast_exp2(y1);
      // int8 pools: P' = p x v_scale (scl[128, 256)) into P.V
      const float v0 = I8 ? scl[kBN + 32 * q + 2 * i] : 1.f;
      const float v1 = I8 ? scl[kBN + 32 * q + 2 * i + 1] : 1.f;
      const float w0 = I8 ? (e0 > 0.f ? e0 * v0 : 0.f) : e0;
      const float w1 = I8 ? (e1 > 0.f ? e1 * v1 : 0.f) : e1;
      pk[i] = pack_f16x2(w0, w1);
      unpack_f16x2(pk[i], h0, h1);
      pl[i] = pack_f16x2(w0 - h0, w1 - h1);
      ls[i & 3] += e0 + e1;
    }
    tc::st16(taddr + 32 * q, pk);
    tc::st16(taddr + 32 * q + 16, pl);
  }
  }
  return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// One work item: a pair of query tiles of one row and KV head.  Item idx is
// KV head idx % h_kv of pair order[idx / h_kv] (pairs most key tiles first);
// every warp decodes the same item itself (tc_tile_range is warp-wide).
struct TcItem {
  int b, g, t0, tile0, n_tiles;
  TcRange rg;
};

__device__ __forceinline__ TcItem tc_item(const PrefillParams& P, int idx, int tpt, int n_pairs,
                                          int64_t cap) {
  TcItem it;
  const int e = P.order[idx / P.h_kv];
  const int qp = e % n_pairs;
  it.b = e / n_pairs;
  it.g = idx % P.h_kv;
  it.t0 = qp * 2 * tpt;
  it.rg = tc_tile_range(P, it.b, it.t0, 2 * tpt, cap);
  it.tile0 = it.rg.kmax >= 0 ? it.rg.kmin / kBN : 0;
  it.n_tiles = it.rg.kmax >= 0 ? it.rg.kmax / kBN - it.tile0 + 1 : 0;
  return it;
}

// The seq-th work item of this CTA, -1 when the queue is exhausted or the
// CTA aborts.  Warp 0 takes items from the global counter into a ring of
// kItemSlots slots; the MMA and softmax warps read them (lane 0 frees the
// slot).
__device__ __forceinline__ int tc_fetch(TcShared& sh, uint32_t seq, int* counter, int i_begin,
                                        int i_end, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const uint32_t slot = seq % kItemSlots, ph = (seq / kItemSlots) & 1;
  int idx = -1;
  if (threadIdx.x < 32) {
    if (!mbar_wait(smem_u32(&sh.item_empty[slot]), ph ^ 1, abort_flag)) return -1;
    if (lane == 0) {
      const int v = i_begin + atomicAdd(counter, 1);
      sh.item[slot] = v < i_end ? v : -1;
      mbar_arrive(smem_u32(&sh.item_full[slot]));
    }
    if (!mbar_wait(smem_u32(&sh.item_full[slot]), ph, abort_flag)) return -1;
    idx = *reinterpret_cast<volatile int*>(&sh.item[slot]);
  } else {
    if (!mbar_wait(smem_u32(&sh.item_full[slot]), ph, abort_flag)) return -1;
    idx = *reinterpret_cast<volatile int*>(&sh.item[slot]);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.item_empty[slot]));
  }
  return idx;
}

// Persistent attention kernel: one CTA per SM, work items from the counter
// at the head of the workspace (zeroed by the V pre-pass).  Across items the
// K / V rings keep streaming; the query tiles rotate over kTcQB buffers (the
// s-th tile of this CTA, s = 2 x item + a, lives in buffer s % kTcQB), and a
// finished tile's buffer stages its output for the TMA stores before the
// tile three steps later is loaded into it.
template <bool SPLIT, bool I8>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(PrefillParams P, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap omap, int box_rows, int* counter) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ TcShared sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  constexpr int QB = I8 ? kTcQBI8 : kTcQB;  // query-tile buffers
  const uint32_t sQ = sbase, sK = sbase + QB * kTcQBytes, sV = sK + kTcKS * kTcKVBytes;
  // int8 pools: a ring of kScR key tiles' scales, [K 128 | V 128] f32 each
  const uint32_t sSc = sV + kTcVS * kTcKVBytes;
  const float* sc_ring = reinterpret_cast<const float*>(smem_raw + (sSc - smem_u32(smem_raw)));
  volatile int* abort_flag = &sh.abort_flag;

  const int tpt = 128 / P.group;  // tokens per query tile
  const int rows_used = tpt * P.group;
  const int n_pairs = (P.T + 2 * tpt - 1) / (2 * tpt);
  const int n_items = n_pairs * P.B * P.h_kv;
  const int64_t cap = position_cap(P);
  if (SPLIT) {
    // the split-P kernel has work only when some row is flagged: read the
    // plan's first flagged item before any set-up
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (__ldcg(P.ctrl + 2) >= n_items) return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < QB; ++i) {
      mbar_init(smem_u32(&sh.q_full[i]), 1);
      mbar_init(smem_u32(&sh.q_free[i]), 1);
    }
    for (int i = 0; i < kTcKS; ++i) {
      mbar_init(smem_u32(&sh.k_full[i]), 1);
      mbar_init(smem_u32(&sh.k_empty[i]), 1);
    }
    for (int i = 0; i < kTcVS; ++i) {
      mbar_init(smem_u32(&sh.v_full[i]), 1);
      mbar_init(smem_u32(&sh.v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh.s_full[i]), 1);
      mbar_init(smem_u32(&sh.p_full[i]), 4);
      mbar_init(smem_u32(&sh.o_done[i]), 1);
      mbar_init(smem_u32(&sh.o_free[i]), 4);
      mbar_init(smem_u32(&sh.stg_full[i]), 128);
      mbar_init(smem_u32(&sh.stg_free[i]), 1);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(smem_u32(&sh.item_full[i]), 1);
      mbar_init(smem_u32(&sh.item_empty[i]), kItemReaders);
    }
    mbar_init(smem_u32(&sh.mma_drain), 1);
    for (int i = 0; i < kScR; ++i) {
      mbar_init(smem_u32(&sh.sc_full[i]), 1);
      mbar_init(smem_u32(&sh.sc_empty[i]), 8);  // the eight softmax warps
    }
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::alloc(smem_u32(&sh.tmem_base), kTcCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sh.tmem_base;
  // launched as a programmatic dependent of the plan kernel (the split-P
  // kernel: of the single-fp16 one): the workspace (work counter, schedule,
  // V copy, row flags) is read only after this wait
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  // the split-P kernel may launch now: its CTAs take the SMs this kernel's
  // CTAs leave, and it waits for this grid in turn
  if (!SPLIT) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // this kernel's work items: those of rows without the split-P flag, or
  // those of flagged rows (the plan puts them last)
  const int first_split = __ldcg(P.ctrl + 2);
  const int i_begin = SPLIT ? first_split : 0, i_end = SPLIT ? n_items : first_split;

  if (warp == 0) {
    // ------------------------------------------------------ K / V producer
    const int nbox = kBN / box_rows;  // boxes per row half of a tile (8 or 16)
    const int n_slots = P.num_pages * P.page_size;
    uint32_t k_issued = 0, v_issued = 0, q_issued = 0;  // query tile s goes to buffer s % QB
    uint32_t sc_issued = 0;                              // int8 pools: scale tiles
    bool ok = true;
    // query tile a of the item (lane 0): wait until its buffer's previous
    // tile has been written out, then load it
#define load_q(a)                                                                               \
  {                                                                                             \
    if (lane == 0) {                                                                            \
      const uint32_t buf = q_issued % QB, use = q_issued / QB;                            \
      if (mbar_wait(smem_u32(&sh.q_free[buf]), (use & 1) ^ 1, abort_flag)) {                    \
        mbar_arrive_expect_tx(smem_u32(&sh.q_full[buf]), (uint32_t)(2 * 64 * rows_used * 2));   \
        for (int h = 0; h < 2; ++h)                                                             \
          tma_load_3d(sQ + buf * kTcQBytes + h * (kTcQBytes / 2), &qmap, h * 64,                \
                      it.g * P.group, it.b * P.T + it.t0 + (a) * tpt, smem_u32(&sh.q_full[buf])); \
        ++q_issued;                                                                             \
      } else {                                                                                  \
        ok = false;                                                                             \
      }                                                                                         \
    }                                                                                           \
    ok = __shfl_sync(0xffffffffu, ok, 0);                                                       \
    q_issued = __shfl_sync(0xffffffffu, q_issued, 0);                                           \
  }
    for (uint32_t seq = 0; ok; ++seq) {
      const int idx = tc_fetch(sh, seq, counter, i_begin, i_end, abort_flag);
      if (idx < 0) break;
      const TcItem it = tc_item(P, idx, tpt, n_pairs, cap);
      if (it.rg.kmax < 0) continue;
      const int32_t* bt_row = P.block_table + (size_t)it.b * P.max_pages_per_seq;
      const int last_blk = it.rg.kmax / P.page_size;
      const int vstart = __ldg(P.row_start + it.b);  // the row's first key in the V copy
      int win_blk0 = -1, win = -1;
      load_q(0)
      for (int j = 0; j < it.n_tiles && ok; ++j) {
        const int key0 = (it.tile0 + j) * kBN;
        const int bmin = key0 / P.page_size;
        const int bmax = min((key0 + kBN - 1) / P.page_size, last_blk);
        if (win_blk0 < 0 || bmin < win_blk0 || bmax >= win_blk0 + 32) {
          win_blk0 = bmin;
          const int blk = win_blk0 + lane;
          win = blk <= last_blk ? __ldg(bt_row + table_index(P, blk)) : -1;
        }
        // this lane's boxes: lanes < 2*nbox (two row halves); box bi of half
        const int half = lane / nbox, bi = lane % nbox;
        const int kb = key0 + bi * box_rows;
        const int blk = kb / P.page_size;
        const int pg = __shfl_sync(0xffffffffu, win, (blk - win_blk0) & 31);
        const bool box_ok = blk <= last_blk && pg >= 0 && pg < P.num_pages;
        if (blk <= last_blk && !box_ok && lane < 2 * nbox)
          report(P.error_word, TL_DEVERR_PAGE_RANGE);
        const int slot0 = box_ok ? pg * P.page_size + kb % P.page_size : n_slots;
        const uint32_t boff = half * (kTcKVBytes / 2) + bi * box_rows * 128;
        {
          const uint32_t st = k_issued % kTcKS;
          if (!mbar_wait(smem_u32(&sh.k_empty[st]), ((k_issued / kTcKS) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(smem_u32(&sh.k_full[st]), kTcKVBytes);
          __syncwarp();
          if (P.kv8) {  // e4m3 pools: the bf16 copy, laid out like the V copy
            if (lane < 2)
              tma_load_3d(sK + st * kTcKVBytes + lane * (kTcKVBytes / 2), &kmap, lane * 64,
                          key0 - vstart, it.b * P.h_kv + it.g, smem_u32(&sh.k_full[st]));
          } else if (lane < 2 * nbox) {
            tma_load_3d(sK + st * kTcKVBytes + boff, &kmap, half * 64, it.g, slot0,
                        smem_u32(&sh.k_full[st]));
          }
          ++k_issued;
        }
        {
          const uint32_t st = v_issued % kTcVS;
          if (!mbar_wait(smem_u32(&sh.v_empty[st]), ((v_issued / kTcVS) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(smem_u32(&sh.v_full[st]), kTcKVBytes);
            for (int hh = 0; hh < 2; ++hh)
              tma_load_3d(sV + st * kTcKVBytes + hh * (kTcKVBytes / 2), &vmap, hh * 64,
                          key0 - vstart, it.b * P.h_kv + it.g, smem_u32(&sh.v_full[st]));
          }
          __syncwarp();
          ++v_issued;
        }
        if (I8) {
          // the tile's K and V scales (512 bytes each) into the scale ring
          const uint32_t st = sc_issued % kScR;
          if (!mbar_wait(smem_u32(&sh.sc_empty[st]), ((sc_issued / kScR) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            // (a row that reads past the copy was reported by the pre-pass:
            // its scale tiles are taken from the copy's start, in bounds)
            const int kc = key0 - vstart + kBN <= P.v_keys ? key0 - vstart : 0;
            const size_t si = ((size_t)it.b * P.h_kv + it.g) * P.v_keys + kc;
            const uint32_t bar = smem_u32(&sh.sc_full[st]), part = kScBytes / 3;
            mbar_arrive_expect_tx(bar, kScBytes);
            bulk_g2s(sSc + st * kScBytes, P.ws_ks + si, part, bar);
            bulk_g2s(sSc + st * kScBytes + part, P.ws_vs + si, part, bar);
            bulk_g2s(sSc + st * kScBytes + 2 * part, P.ws_ivs + si, part, bar);
          }
          __syncwarp();
          ++sc_issued;
        }
        if (j == 0) load_q(1)  // the second tile's buffer frees up later
      }
    }
#undef load_q
    // drain: the copies this warp issued have landed before the CTA exits
    bool drained = true;
    for (uint32_t i = k_issued > (uint32_t)kTcKS ? k_issued - kTcKS : 0; i < k_issued; ++i)
      drained &= mbar_drain(smem_u32(&sh.k_full[i % kTcKS]), (i / kTcKS) & 1);
    for (uint32_t i = v_issued > (uint32_t)kTcVS ? v_issued - kTcVS : 0; i < v_issued; ++i)
      drained &= mbar_drain(smem_u32(&sh.v_full[i % kTcVS]), (i / kTcVS) & 1);
    for (uint32_t i = q_issued > (uint32_t)QB ? q_issued - QB : 0; i < q_issued; ++i)
      drained &= mbar_drain(smem_u32(&sh.q_full[i % QB]), (i / QB) & 1);
    for (uint32_t i = sc_issued > (uint32_t)kScR ? sc_issued - kScR : 0; i < sc_issued; ++i)
      drained &= mbar_drain(smem_u32(&sh.sc_full[i % kScR]), (i / kScR) & 1);
    if (!drained) *abort_flag = 1;
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
#define issue_s(a, kt, qbuf) \
  tc_issue_s(tmem, (a), sK + ((kt) % kTcKS) * kTcKVBytes, sQ + (qbuf) * kTcQBytes, \
             smem_u32(&sh.s_full[(a)]))
#define issue_pv(a, vt, acc) \
  tc_issue_pv(tmem, (a), sV + ((vt) % kTcVS) * kTcKVBytes, (acc), SPLIT)
    uint32_t kt = 0, vt = 0, tiles = 0, n = 0;  // K / V tiles, S tiles, live items
    bool ok = true;
    long long t_first = 0, wait_p = 0, wait_kv = 0;  // the step trace (zero without it)
    // a wait for the softmax's P, or for the producer's K / V, with its cycles
    auto wait_for_p = [&](uint32_t bar, uint32_t ph) {
      const long long t0 = ptrace_clk();
      const bool r = mbar_wait(bar, ph, abort_flag);
      wait_p += ptrace_clk() - t0;
      return r;
    };
    auto wait_for_kv = [&](uint32_t bar, uint32_t ph) {
      const long long t0 = ptrace_clk();
      const bool r = mbar_wait(bar, ph, abort_flag);
      wait_kv += ptrace_clk() - t0;
      return r;
    };
    for (uint32_t seq = 0; ok; ++seq) {
      const int idx = tc_fetch(sh, seq, counter, i_begin, i_end, abort_flag);
      if (idx < 0) break;
      const TcItem it = tc_item(P, idx, tpt, n_pairs, cap);
      if (it.rg.kmax < 0) continue;
      if (lane == 0) {
        if (n == 0) t_first = ptrace_clk();
        const uint32_t qb0 = (2 * n) % QB, qb1 = (2 * n + 1) % QB;
        ok = mbar_wait(smem_u32(&sh.q_full[qb0]), ((2 * n) / QB) & 1, abort_flag) &&
             wait_for_kv(smem_u32(&sh.k_full[kt % kTcKS]), (kt / kTcKS) & 1);
        if (ok) {
          tc::fence_after();
          issue_s(0, kt, qb0);
        }
        ok = ok && mbar_wait(smem_u32(&sh.q_full[qb1]), ((2 * n + 1) / QB) & 1, abort_flag);
        if (ok) {
          tc::fence_after();
          issue_s(1, kt, qb1);
          tc::commit(smem_u32(&sh.k_empty[kt % kTcKS]));
        }
        for (int j = 0; j < it.n_tiles && ok; ++j, ++tiles) {
          const bool last = j == it.n_tiles - 1;
          if (!wait_for_kv(smem_u32(&sh.v_full[vt % kTcVS]), (vt / kTcVS) & 1) ||
              !wait_for_p(smem_u32(&sh.p_full[0]), tiles & 1) ||
              (j == 0 && n > 0 &&
               !mbar_wait(smem_u32(&sh.o_free[0]), (n - 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc::fence_after();
          issue_pv(0, vt, j > 0);
          if (last) {
            tc::commit(smem_u32(&sh.o_done[0]));
          } else {
            if (!wait_for_kv(smem_u32(&sh.k_full[(kt + 1) % kTcKS]), ((kt + 1) / kTcKS) & 1)) {
              ok = false;
              break;
            }
            tc::fence_after();
            issue_s(0, kt + 1, qb0);
          }
          if (!wait_for_p(smem_u32(&sh.p_full[1]), tiles & 1) ||
              (j == 0 && n > 0 &&
               !mbar_wait(smem_u32(&sh.o_free[1]), (n - 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc::fence_after();
          issue_pv(1, vt, j > 0);
          tc::commit(smem_u32(&sh.v_empty[vt % kTcVS]));
          ++vt;
          if (last) {
            tc::commit(smem_u32(&sh.o_done[1]));
          } else {
            issue_s(1, kt + 1, qb1);
            tc::commit(smem_u32(&sh.k_empty[(kt + 1) % kTcKS]));
            ++kt;
          }
        }
        ++kt;
        ++n;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
#undef issue_s
#undef issue_pv
    if (lane == 0) {
      // every MMA this thread issued is done before TMEM is released
      tc::commit(smem_u32(&sh.mma_drain));
      if (!mbar_drain(smem_u32(&sh.mma_drain), 0)) *abort_flag = 1;
#if TL_PREFILL_TRACE
      if (n > 0 && blockIdx.x < kPtraceCtas) {
        unsigned long long* row = g_ptrace[blockIdx.x];
        atomicAdd(row + TL_PTRACE_CYCLES, (unsigned long long)(ptrace_clk() - t_first));
        atomicAdd(row + TL_PTRACE_STEPS, (unsigned long long)tiles);
        atomicAdd(row + TL_PTRACE_ITEMS, (unsigned long long)n);
        atomicAdd(row + TL_PTRACE_WAIT_P, (unsigned long long)wait_p);
        atomicAdd(row + TL_PTRACE_WAIT_KV, (unsigned long long)wait_kv);
      }
#endif
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax, epilogue
    const int a = (warp - 2) >> 2;  // query tile of this warpgroup (warps 2-5, 6-9)
    const int row = 32 * (warp & 3) + lane;
    const int wtid = row;           // thread index inside the warpgroup
    const bool leader = (warp & 3) == 2 && lane == 0;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t colS = a * 128, colO = 256 + a * 128;
    const float sc = P.scale_log2;
    uint32_t tiles = 0, n = 0;
    bool ok = true;
    long long sm_wait_s = 0, sm_busy = 0;  // the step trace (zero without it)
    for (uint32_t seq = 0; ok; ++seq) {
      const int idx = tc_fetch(sh, seq, counter, i_begin, i_end, abort_flag);
      if (idx < 0) break;
      const TcItem it = tc_item(P, idx, tpt, n_pairs, cap);
      const int ta0 = it.t0 + a * tpt;  // first token of this tile
      if (it.rg.kmax < 0) {
        // no live token in the pair: the outputs are 0 (coalesced, one row per warp step)
        for (int e = wtid; e < rows_used * 32; e += 128) {
          const int r = e >> 5, c = (e & 31) * 4, t = ta0 + r / P.group;
          if (t < P.T)
            *reinterpret_cast<float4*>(P.out + (((size_t)it.b * P.T + t) * P.h_q +
                                                (size_t)it.g * P.group + r % P.group) *
                                                   128 +
                                       c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        continue;
      }
      const int t = ta0 + row / P.group;
      int p = -1;
      if (row < rows_used && t < P.T) {
        p = P.positions[(size_t)it.b * P.T + t];
        if (p >= cap) {
          report(P.error_word, TL_DEVERR_CONTEXT_RANGE);
          p = -1;
        }
      }
      const int lo = (P.window > 0 && p - P.window + 1 > 0) ? p - P.window + 1 : 0;
      float m_used = -INFINITY, l = 0.f;  // running max of the scores in log2 units
      for (int j = 0; j < it.n_tiles; ++j, ++tiles) {
        const long long tw = ptrace_clk();
        if (!mbar_wait(smem_u32(&sh.s_full[a]), tiles & 1, abort_flag)) {
          ok = false;
          break;
        }
        const long long ts = ptrace_clk();
        sm_wait_s += ts - tw;
        tc::fence_after();
        const int key0 = (it.tile0 + j) * kBN;
        const int cmin = lo - key0, cmax = p - key0;  // live columns [cmin, cmax]
        const bool all_live = __all_sync(0xffffffffu, cmin <= 0 && cmax >= kBN - 1);
        // int8 pools: the tile's key scales (K at [0, 128), V at [128, 256),
        // 1 / V at [256, 384))
        const float* scl = sc_ring + (tiles % kScR) * (kScBytes / 4);
        if (I8 && !mbar_wait(smem_u32(&sh.sc_full[tiles % kScR]), (tiles / kScR) & 1, abort_flag)) {
          ok = false;
          break;
        }
        // the tile's 128 scores of this row: four loads, one wait
        float s[kBN];
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) tc::ld32(tmem + lane_base + colS + q * 32, s + q * 32);
        tc::wait_ld();
        if (I8) {  // s_j = (q . codes_j) x k_scale_j
#pragma unroll
          for (int c = 0; c < kBN; c += 2) {  // packed: two keys per multiply
            uint64_t sv, kv;
            asm("mov.b64 %0, {%1, %2};\n" : "=l"(sv) : "f"(s[c]), "f"(s[c + 1]));
            asm("ld.shared.b64 %0, [%1];\n" : "=l"(kv) : "r"(smem_u32(scl + c)));
            asm("mul.rn.f32x2 %0, %0, %1;\n" : "+l"(sv) : "l"(kv));
            asm("mov.b64 {%0, %1}, %2;\n" : "=f"(s[c]), "=f"(s[c + 1]) : "l"(sv));
          }
        }
        if (!all_live) {
#pragma unroll
          for (int c = 0; c < kBN; ++c) s[c] = (c >= cmin && c <= cmax) ? s[c] : -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[i], s[8 + i]);
#pragma unroll
        for (int c = 16; c < kBN; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = max3(mx[i], s[c + i], s[c + 8 + i]);
        const float mt =
            max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sc;
        const bool need = l > 0.f && mt > m_used + kRescaleLog2;
        float corr = 1.f;
        if (need) {
          corr = fast_exp2(m_used - mt);
          m_used = mt;
        }
        if (m_used == -INFINITY) m_used = mt;  // first live key of this row
        const float base = m_used == -INFINITY ? 0.f : m_used;
        // P = fp16(exp2(s*sc - base)), keys 2c and 2c+1 in column c; the sum
        // takes the same rounded values.  Packed f32x2 FMAs scale two scores
        // at once; the sum widens each fp16 half inside its add.
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
        const uint64_t sc2 = f32_twice(sc), nb2 = f32_twice(-base);
        if constexpr (!SPLIT) {
          // (int8 pools: the scores above carry their K scales, and a row
          // without the split-P flag has every V tile copied with its V
          // scales applied, so P.V takes P as for 16-bit pools)
#pragma unroll
          for (int q = 0; q < kBN / 32; ++q) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float y0, y1;
              fma_f32x2(s[q * 32 + 2 * i], s[q * 32 + 2 * i + 1], sc2, nb2, y0, y1);
              pk[i] = pack_f16x2(fast_exp2(y0), fast_exp2(y1));
              ls[i & 3] = add_f16x2_halves(ls[i & 3], pk[i]);
            }
            tc::st16(tmem + lane_base + colS + q * 16, pk);
          }
        } else {
          ls[0] = tc_softmax_split<I8, kRereadCh>(tmem + lane_base + colS, cmin, cmax, all_live, sc,
                                                 base, scl);
        }
        l = l * corr + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
        if (__any_sync(0xffffffffu, need)) {
          // PV_a(j-1) is complete (S_a(j) was issued after it) and PV_a(j)
          // waits for this tile's P: rescale O_a now (never at j = 0, where
          // l is still 0)
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
        if (I8 && lane == 0) mbar_arrive(smem_u32(&sh.sc_empty[tiles % kScR]));
        sm_busy += ptrace_clk() - ts;
      }
      if (!ok) break;
      // epilogue: O / l.  The tile's own query buffer, free since its last S
      // MMA, stages the output for TMA stores in two rounds of two
      // 128-byte-swizzled d quarters (32 KiB each); then O_a is released to
      // the next item's P.V and, after the second store has read it, the
      // buffer to the query tile three steps later.
      const uint32_t buf = (2 * n + a) % QB, stage = sQ + buf * kTcQBytes;
      const float inv = (p >= 0 && l > 0.f) ? 1.f / l : 0.f;
      ok = mbar_wait(smem_u32(&sh.o_done[a]), n & 1, abort_flag);
      if (ok) tc::fence_after();
      // round r: wait for the previous round's store to have read the
      // staging area, move d quarters 2r, 2r+1 from TMEM to it one quarter at
      // a time (after r = 1, release O_a), and let the leader store them
#define TL_PREFILL_STAGE_ROUND(r)                                                              \
  {                                                                                            \
    const uint32_t R = 2 * n + (r); /* staging rounds of this warpgroup */                     \
    if (R > 0 && !mbar_wait(smem_u32(&sh.stg_free[a]), (R - 1) & 1, abort_flag)) ok = false;   \
    _Pragma("unroll") for (int qq = 0; qq < 2; ++qq) {                                         \
      float o[32];                                                                             \
      if (ok) {                                                                                \
        tc::ld32(tmem + lane_base + colO + (2 * (r) + qq) * 32, o);                            \
        tc::wait_ld();                                                                         \
        _Pragma("unroll") for (int i = 0; i < 8; ++i) {                                        \
          const uint32_t adr = stage + qq * 16384 + row * 128 + ((i ^ (row & 7)) << 4);        \
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(adr),                \
                       "f"(o[4 * i] * inv), "f"(o[4 * i + 1] * inv), "f"(o[4 * i + 2] * inv),  \
                       "f"(o[4 * i + 3] * inv)                                                 \
                       : "memory");                                                            \
        }                                                                                      \
      }                                                                                        \
    }                                                                                          \
    if ((r) == 1) { /* O_a is out of TMEM: the next item's P.V may overwrite it */             \
      tc::fence_before();                                                                      \
      __syncwarp();                                                                            \
      if (lane == 0) mbar_arrive(smem_u32(&sh.o_free[a]));                                     \
    }                                                                                          \
    fence_proxy_async_smem();                                                                  \
    mbar_arrive(smem_u32(&sh.stg_full[a]));                                                    \
    if (leader) {                                                                              \
      if (mbar_wait(smem_u32(&sh.stg_full[a]), R & 1, abort_flag) && !*abort_flag) {           \
        for (int qq = 0; qq < 2; ++qq)                                                         \
          tma_store_4d(&omap, (2 * (r) + qq) * 32, it.g * P.group, ta0, it.b,                  \
                       stage + qq * 16384);                                                    \
        bulk_commit_group();                                                                   \
        bulk_wait_read_all();                                                                  \
      }                                                                                        \
      mbar_arrive(smem_u32(&sh.stg_free[a]));                                                  \
    }                                                                                          \
  }
      TL_PREFILL_STAGE_ROUND(0)
      TL_PREFILL_STAGE_ROUND(1)
#undef TL_PREFILL_STAGE_ROUND
      if (leader) mbar_arrive(smem_u32(&sh.q_free[buf]));
      ++n;
      ok = ok && !*abort_flag;
    }
#if TL_PREFILL_TRACE
    if (leader && blockIdx.x < kPtraceCtas) {
      atomicAdd(&g_ptrace[blockIdx.x][TL_PTRACE_SM_WAIT_S], (unsigned long long)sm_wait_s);
      atomicAdd(&g_ptrace[blockIdx.x][TL_PTRACE_SM_BUSY], (unsigned long long)sm_busy);
    }
#endif
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

#if TL_PREFILL_ALL_TS
#include "prefill_ts.cuh"
#endif

namespace tl {

static size_t prefill_ws_size(int32_t B, int32_t T, int32_t h_q, int32_t h_kv, int32_t d,
                              int32_t max_pages_per_seq, int32_t page_size, int32_t ring_pages,
                              tl_dtype dtype) {
  if (B <= 0 || T <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || h_q % h_kv ||
      max_pages_per_seq <= 0 || page_size <= 0 || ring_pages < 0 ||
      (dtype != TL_BF16 && dtype != TL_FP8_E4M3 && dtype != TL_INT8))
    return 0;
  const int tpt = std::max(1, 128 / (h_q / h_kv));
  const int64_t n_pairs = (T + 2 * tpt - 1) / (2 * tpt);
  return ws_layout(B, n_pairs, h_kv, v_copy_keys(max_pages_per_seq, page_size, ring_pages),
                   dtype != TL_BF16, dtype == TL_INT8, ts_path(dtype, h_kv))
      .total;
}

static tl_status prefill_impl(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, int32_t max_pages_per_seq,
                              const int32_t* positions, float* out, int32_t B, int32_t T,
                              int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                              int32_t page_size, int32_t window, int32_t ring_pages, float scale,
                              tl_dtype dtype, void* workspace, size_t workspace_bytes,
                              uint32_t* error_word, void* stream,
                              const float* k_scales = nullptr, const float* v_scales = nullptr) {
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
  // (e4m3 and int8 pools: q and out as for bf16; the pools hold one byte per element)
  if ((dtype != TL_BF16 && dtype != TL_FP8_E4M3 && dtype != TL_INT8) || d != 128 ||
      (page_size & (page_size - 1)) || page_size < 8 || page_size > 128)
    return TL_ERR_UNSUPPORTED;
  if ((int64_t)max_pages_per_seq * page_size >= ((int64_t)1 << 31)) return TL_ERR_UNSUPPORTED;
  const bool i8 = dtype == TL_INT8;
  const bool kv8 = dtype == TL_FP8_E4M3 || i8;  // one byte per element, K read from a copy
  if (kv8 && (!aligned16(k_cache) || !aligned16(v_cache))) return TL_ERR_INVALID_ARG;
  if (i8 && (!k_scales || !v_scales || (reinterpret_cast<uintptr_t>(k_scales) & 3u) ||
             (reinterpret_cast<uintptr_t>(v_scales) & 3u)))
    return TL_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return TL_ERR_WORKSPACE;
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
  P.ring_pages = ring_pages;
  P.scale_log2 = scale * kLog2e;
  P.error_word = error_word;
  if (h_q / h_kv > 128 || B > 65535 || h_kv > 65535) return TL_ERR_UNSUPPORTED;
  if ((int64_t)num_pages * page_size >= ((int64_t)1 << 31) || (int64_t)B * T >= ((int64_t)1 << 31))
    return TL_ERR_UNSUPPORTED;
  const int group = h_q / h_kv;
  const int tpt = 128 / group;
  const int box_rows = page_size % 16 == 0 ? 16 : 8;
  // keys per row of the copies: the table's (or the ring's) positions when
  // the workspace holds them; otherwise as many 128-key tiles as it holds
  // (a workspace sized by tl_paged_attn_prefill_workspace_size_keys), at
  // least kMinCopyKeys
  const int n_pairs = (T + 2 * tpt - 1) / (2 * tpt);
  int64_t v_keys = v_copy_keys(max_pages_per_seq, page_size, ring_pages);
  if (v_keys >= ((int64_t)1 << 31)) return TL_ERR_UNSUPPORTED;
  const bool ts = ts_path(dtype, h_kv);
  if (workspace_bytes < ws_layout(B, n_pairs, h_kv, v_keys, kv8, i8, ts).total) {
    const WsLayout full = ws_layout(B, n_pairs, h_kv, v_keys, kv8, i8, ts);
    const size_t copies = full.total - full.v;  // copies and scales of every row at v_keys keys
    const size_t room = workspace_bytes > full.v ? workspace_bytes - full.v : 0;
    // their bytes per key of a row (over all rows and KV heads; the rounding
    // of each array to 256 bytes aside: the loop below checks the layout)
    const size_t per_key = copies / (size_t)v_keys + 1;
    int64_t fit = (int64_t)(room / per_key);
    fit = fit / kBN * kBN;
    while (fit >= kMinCopyKeys &&
           ws_layout(B, n_pairs, h_kv, fit, kv8, i8, ts).total > workspace_bytes)
      fit -= kBN;
    if (fit < kMinCopyKeys) return TL_ERR_WORKSPACE;
    v_keys = fit;
  }
  const WsLayout L = ws_layout(B, n_pairs, h_kv, v_keys, kv8, i8, ts);
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  int* counter = reinterpret_cast<int*>(wsb);
  uint16_t* ws_v = reinterpret_cast<uint16_t*>(wsb + L.v);
  P.n_pairs = n_pairs;
  P.pair_tiles = reinterpret_cast<int32_t*>(wsb + L.tiles);
  P.order = reinterpret_cast<int32_t*>(wsb + L.order);
  P.row_start = reinterpret_cast<int32_t*>(wsb + L.rows);
  P.v_keys = (int32_t)v_keys;
  P.kv8 = kv8 ? 1 : 0;
  P.ws_k = kv8 ? reinterpret_cast<uint16_t*>(wsb + L.k) : nullptr;
  P.k_scales = k_scales;
  P.v_scales = v_scales;
  P.ws_ks = i8 ? reinterpret_cast<float*>(wsb + L.ks) : nullptr;
  P.ws_vs = i8 ? reinterpret_cast<float*>(wsb + L.vs) : nullptr;
  P.ws_ivs = i8 ? reinterpret_cast<float*>(wsb + L.ivs) : nullptr;
  P.ctrl = counter;
  P.cvt_gx = (int32_t)((v_keys + kCvtKeys - 1) / kCvtKeys);
  P.cta_big = reinterpret_cast<int32_t*>(wsb + L.cta_big);
  P.row_big = reinterpret_cast<int32_t*>(wsb + L.row_big);
  P.ws_kt = ts ? reinterpret_cast<uint16_t*>(wsb + L.kt) : nullptr;
  CUtensorMap qmap, kmap, vmap, omap, ktmap;
  {
    const uint64_t qd[3] = {128, (uint64_t)h_q, (uint64_t)B * T};
    const uint64_t qs[2] = {128 * 2, (uint64_t)h_q * 128 * 2};
    const uint32_t qb[3] = {64, (uint32_t)group, (uint32_t)tpt};
    const uint64_t kd[3] = {128, (uint64_t)h_kv, (uint64_t)num_pages * page_size};
    const uint64_t ks[2] = {128 * 2, (uint64_t)h_kv * 128 * 2};
    const uint32_t kb[3] = {64, 1, (uint32_t)box_rows};
    // the workspace's fp16 V: (d, key - row start, row x KV head), 16-bit
    // elements like bf16
    const uint64_t vd[3] = {128, (uint64_t)v_keys, (uint64_t)B * h_kv};
    const uint64_t vs[2] = {128 * 2, (uint64_t)v_keys * 128 * 2};
    const uint32_t vb[3] = {64, (uint32_t)kBN, 1};
    // the output, f32 (d, h_q, T, B): a TMA store box is one d quarter of a
    // query tile, clipped at T
    const uint64_t od[4] = {128, (uint64_t)h_q, (uint64_t)T, (uint64_t)B};
    const uint64_t os[3] = {128 * 4, (uint64_t)h_q * 128 * 4, (uint64_t)T * h_q * 128 * 4};
    const uint32_t ob[4] = {32, (uint32_t)group, (uint32_t)tpt, 1};
    if (!encode_f32_tensor_map(&omap, out, 4, od, os, ob, true)) return TL_ERR_CUDA;
    // e4m3 pools: K is read from its bf16 copy, with the V copy's map shape
    if (!encode_bf16_tensor_map(&qmap, q, 3, qd, qs, qb, true) ||
        !(kv8 ? encode_bf16_tensor_map(&kmap, P.ws_k, 3, vd, vs, vb, true)
              : encode_bf16_tensor_map(&kmap, k_cache, 3, kd, ks, kb, true)) ||
        !encode_bf16_tensor_map(&vmap, ws_v, 3, vd, vs, vb, true))
      return TL_ERR_CUDA;
    // the all-TS kernel's K^T copy: (key in the tile, key tile x 128 + d,
    // row x KV head), the V copy's shape; boxes of 64 keys x 128 d
    if (ts && !encode_bf16_tensor_map(&ktmap, P.ws_kt, 3, vd, vs, vb, true)) return TL_ERR_CUDA;
  }
  auto tc_fast = i8 ? prefill_tc_kernel<false, true> : prefill_tc_kernel<false, false>;
  auto tc_split = i8 ? prefill_tc_kernel<true, true> : prefill_tc_kernel<true, false>;
  const int tc_smem = i8 ? kTcSmemI8 : kTcSmem;
  if (cudaFuncSetAttribute(tc_fast, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(tc_split, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_smem) !=
          cudaSuccess)
    return TL_ERR_CUDA;
  const int64_t n_items = (int64_t)n_pairs * B * h_kv;
  if (n_items > 0x7fffffff - 65536) return TL_ERR_UNSUPPORTED;
  const int grid = (int)std::min<int64_t>(num_sms(), n_items);
  const dim3 cvt_grid((unsigned)P.cvt_gx, B);
  if (i8)
    prefill_v_f16_kernel<2><<<cvt_grid, kCvtThreads, 0, (cudaStream_t)stream>>>(P, ws_v, counter);
  else if (kv8)
    prefill_v_f16_kernel<1><<<cvt_grid, kCvtThreads, 0, (cudaStream_t)stream>>>(P, ws_v, counter);
  else
    prefill_v_f16_kernel<0><<<cvt_grid, kCvtThreads, 0, (cudaStream_t)stream>>>(P, ws_v, counter);
  if (launch_status() != TL_OK) return TL_ERR_CUDA;
  // the plan and the attention kernel are programmatic dependent launches:
  // each becomes resident while its predecessor finishes and waits for its
  // results (griddepcontrol.wait)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = (cudaStream_t)stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  if (cudaLaunchKernelEx(&cfg, prefill_plan_kernel, P) != cudaSuccess) return TL_ERR_CUDA;
  cfg.gridDim = dim3(grid);
  // rows whose V holds no value above 8 in magnitude (single fp16 P), then
  // the others (P split in two); each kernel skips the other's rows
  if (ts) {
#if TL_PREFILL_ALL_TS
    if (cudaFuncSetAttribute(prefill_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTsSmem) != cudaSuccess)
      return TL_ERR_CUDA;
    cfg.blockDim = dim3(kTsThreads);
    cfg.dynamicSmemBytes = kTsSmem;
    if (cudaLaunchKernelEx(&cfg, prefill_ts_kernel, P, qmap, ktmap, vmap, omap, counter) !=
        cudaSuccess)
      return TL_ERR_CUDA;
#endif
  } else {
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = tc_smem;
    if (cudaLaunchKernelEx(&cfg, tc_fast, P, qmap, kmap, vmap, omap, box_rows, counter) !=
        cudaSuccess)
      return TL_ERR_CUDA;
  }
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = tc_smem;
  if (cudaLaunchKernelEx(&cfg, tc_split, P, qmap, kmap, vmap, omap, box_rows, counter + 1) !=
      cudaSuccess)
    return TL_ERR_CUDA;
  return launch_status();
}

// The ring must be part of the table and hold one window.
static bool ring_args_ok(int32_t max_pages_per_seq, int32_t page_size, int32_t window,
                         int32_t ring_pages) {
  return ring_pages > 0 && ring_pages <= max_pages_per_seq && window > 0 && page_size > 0 &&
         (int64_t)ring_pages * page_size >= window;
}

}  // namespace tl

extern "C" tl_status tl_prefill_trace_reset(void) {
#if TL_PREFILL_TRACE
  if (cudaDeviceSynchronize() != cudaSuccess) return TL_ERR_CUDA;
  static unsigned long long zeros[tl::kPtraceCtas][TL_PTRACE_FIELDS];
  if (cudaMemcpyToSymbol(tl::g_ptrace, zeros, sizeof(zeros)) != cudaSuccess) return TL_ERR_CUDA;
  return TL_OK;
#else
  return TL_ERR_UNSUPPORTED;
#endif
}

extern "C" tl_status tl_prefill_trace_read(uint64_t* rows, int32_t n_ctas) {
#if TL_PREFILL_TRACE
  if (!rows || n_ctas < 1 || n_ctas > tl::kPtraceCtas) return TL_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return TL_ERR_CUDA;
  if (cudaMemcpyFromSymbol(rows, tl::g_ptrace,
                           sizeof(uint64_t) * TL_PTRACE_FIELDS * (size_t)n_ctas) != cudaSuccess)
    return TL_ERR_CUDA;
  return TL_OK;
#else
  (void)rows;
  (void)n_ctas;
  return TL_ERR_UNSUPPORTED;
#endif
}

extern "C" size_t tl_paged_attn_prefill_workspace_size(int32_t B, int32_t T, int32_t h_q,
                                                       int32_t h_kv, int32_t d,
                                                       int32_t max_pages_per_seq,
                                                       int32_t page_size) {
  return tl::prefill_ws_size(B, T, h_q, h_kv, d, max_pages_per_seq, page_size, 0, TL_BF16);
}

extern "C" size_t tl_paged_attn_prefill_workspace_size_ex(int32_t B, int32_t T, int32_t h_q,
                                                          int32_t h_kv, int32_t d,
                                                          int32_t max_pages_per_seq,
                                                          int32_t page_size, int32_t ring_pages,
                                                          tl_dtype dtype) {
  return tl::prefill_ws_size(B, T, h_q, h_kv, d, max_pages_per_seq, page_size, ring_pages, dtype);
}

extern "C" size_t tl_paged_attn_prefill_ring_workspace_size(int32_t B, int32_t T, int32_t h_q,
                                                            int32_t h_kv, int32_t d,
                                                            int32_t max_pages_per_seq,
                                                            int32_t page_size,
                                                            int32_t ring_pages) {
  if (ring_pages <= 0) return 0;
  return tl::prefill_ws_size(B, T, h_q, h_kv, d, max_pages_per_seq, page_size, ring_pages,
                             TL_BF16);
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
  return tl::prefill_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, positions, out, B,
                          T, h_q, h_kv, d, num_pages, page_size, window, 0, scale, dtype,
                          workspace, workspace_bytes, error_word, stream);
}

extern "C" tl_status tl_paged_attn_prefill_ring(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* positions, float* out, int32_t B, int32_t T,
    int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages, int32_t page_size, int32_t window,
    int32_t ring_pages, float scale, tl_dtype dtype, void* workspace, size_t workspace_bytes,
    uint32_t* error_word, void* stream) {
  if (!tl::ring_args_ok(max_pages_per_seq, page_size, window, ring_pages))
    return TL_ERR_INVALID_ARG;
  return tl::prefill_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, positions, out, B,
                          T, h_q, h_kv, d, num_pages, page_size, window, ring_pages, scale, dtype,
                          workspace, workspace_bytes, error_word, stream);
}

extern "C" tl_status tl_paged_attn_prefill_int8(
    const void* q, const int8_t* k_codes, const int8_t* v_codes, const float* k_scales,
    const float* v_scales, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* positions, float* out, int32_t B, int32_t T, int32_t h_q, int32_t h_kv,
    int32_t d, int32_t num_pages, int32_t page_size, int32_t window, float scale,
    void* workspace, size_t workspace_bytes, uint32_t* error_word, void* stream) {
  if (!k_scales || !v_scales) return TL_ERR_INVALID_ARG;
  return tl::prefill_impl(q, k_codes, v_codes, block_table, max_pages_per_seq, positions, out, B,
                          T, h_q, h_kv, d, num_pages, page_size, window, 0, scale, TL_INT8,
                          workspace, workspace_bytes, error_word, stream, k_scales, v_scales);
}

extern "C" tl_status tl_paged_attn_prefill_ring_int8(
    const void* q, const int8_t* k_codes, const int8_t* v_codes, const float* k_scales,
    const float* v_scales, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* positions, float* out, int32_t B, int32_t T, int32_t h_q, int32_t h_kv,
    int32_t d, int32_t num_pages, int32_t page_size, int32_t window, int32_t ring_pages,
    float scale, void* workspace, size_t workspace_bytes, uint32_t* error_word, void* stream) {
  if (!k_scales || !v_scales) return TL_ERR_INVALID_ARG;
  if (!tl::ring_args_ok(max_pages_per_seq, page_size, window, ring_pages))
    return TL_ERR_INVALID_ARG;
  return tl::prefill_impl(q, k_codes, v_codes, block_table, max_pages_per_seq, positions, out, B,
                          T, h_q, h_kv, d, num_pages, page_size, window, ring_pages, scale,
                          TL_INT8, workspace, workspace_bytes, error_word, stream, k_scales,
                          v_scales);
}

extern "C" size_t tl_paged_attn_prefill_workspace_size_keys(int32_t B, int32_t T, int32_t h_q,
                                                            int32_t h_kv, int32_t d,
                                                            int32_t max_row_keys,
                                                            tl_dtype dtype) {
  if (B <= 0 || T <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || h_q % h_kv || max_row_keys <= 0 ||
      (dtype != TL_BF16 && dtype != TL_FP8_E4M3 && dtype != TL_INT8))
    return 0;
  const int tpt = std::max(1, 128 / (h_q / h_kv));
  const int64_t n_pairs = (T + 2 * tpt - 1) / (2 * tpt);
  return tl::ws_layout(B, n_pairs, h_kv, tl::v_copy_keys_for_span(max_row_keys),
                       dtype != TL_BF16, dtype == TL_INT8, tl::ts_path(dtype, h_kv))
      .total;
}
