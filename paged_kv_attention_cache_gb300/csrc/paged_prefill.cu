// PAGED_ATTENTION, batched right-aligned prefill, folded over key tiles with
// an online softmax ("How serving works in Tlaloc", section 1: right-aligned
// rows, padding at slot -1, causal length = position + 1; section 2: a row's
// pages are gathered once for all its tokens, and "Blockwise attention": the
// keys are folded block by block into a running max, sum and P.V, so no score
// tensor wider than one tile exists).
//
// Two launches.  A pre-pass converts the V rows each row's tokens can see
// from the bf16 pages to fp16, once, into the workspace, laid out as
// [row][KV head][key][d] (exact for |v| in [2^-14, 65504]; larger finite
// values are reported; keys past the row's last position are zeros).  Then
// the attention kernel runs one CTA per (pair of query tiles, KV head, row)
// on the 5th-generation tensor core.  A query tile packs tokens_per_tile =
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
#include "common.cuh"
#include "tcgen05.cuh"

namespace tl {

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

constexpr int kBN = 128;             // keys per tile
constexpr int kTcKS = 3;             // K stages
constexpr int kTcVS = 2;             // V stages
constexpr int kTcThreads = 10 * 32;
constexpr int kCvtThreads = 256;
constexpr int kTcQBytes = 32768;     // one query tile: 128 rows x 128 d x bf16
constexpr int kTcKVBytes = kBN * 256;  // 128 keys x 128 d x 16-bit (two 16 KiB halves)
constexpr int kTcSmem = 2 * kTcQBytes + (kTcKS + kTcVS) * kTcKVBytes + 1024;
constexpr uint32_t kTcCols = 512;
constexpr float kRescaleLog2 = 8.f;
// bf16 bit patterns (sign cleared) of the finite values fp16 cannot hold:
// [65536, max finite]; 65280 (0x477F) is the largest bf16 below fp16's
// overflow threshold.
constexpr uint32_t kBf16TooBig = 0x4780u, kBf16Inf = 0x7F80u;

struct TcShared {
  unsigned long long q_full, k_full[kTcKS], k_empty[kTcKS], v_full[kTcVS], v_empty[kTcVS];
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
// Two bf16 (one register) -> two fp16 (one register).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  return pack_f16x2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
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
// Grid (key tile of 128, row).  Each CTA first finds its row's live
// positions [pmin, pmax]; the attention kernel reads V keys in
// [start, end): start = the first key any live token can see, rounded down
// to a tile, end = pmax + 1 rounded up to a tile (clamped to the workspace).
// The tile's page numbers go to shared memory; then every thread moves
// 16-byte units (key-major: one key's h_kv x 128 values are contiguous in
// the pool), kCvtUnroll independent loads in flight.
constexpr int kCvtUnroll = 8;

__global__ void __launch_bounds__(kCvtThreads)
    prefill_v_f16_kernel(PrefillParams P, uint16_t* __restrict__ ws, int max_ctx) {
  __shared__ int s_min[kCvtThreads / 32], s_max[kCvtThreads / 32];
  __shared__ int s_page[kBN];  // page of each key of the tile; -1: write zeros
  const int b = (int)blockIdx.y, k0 = (int)blockIdx.x * kBN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t cap = (int64_t)P.max_pages_per_seq * P.page_size;
  int pmin = INT32_MAX, pmax = -1;
  for (int t = threadIdx.x; t < P.T; t += kCvtThreads) {
    const int p = P.positions[(size_t)b * P.T + t];
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
  if (pmax < 0) return;  // no live token: the attention kernel reads nothing
  const int lo = (P.window > 0 && pmin - P.window + 1 > 0) ? pmin - P.window + 1 : 0;
  const int start = lo / kBN * kBN, end = min((pmax / kBN + 1) * kBN, max_ctx);
  if (k0 + kBN <= start || k0 >= end) return;
  for (int r = threadIdx.x; r < kBN; r += kCvtThreads) {
    const int k = k0 + r;
    int page = -1;  // keys past pmax: zeros
    if (k <= pmax) {
      page = __ldg(P.block_table + (size_t)b * P.max_pages_per_seq + k / P.page_size);
      if (page < 0 || page >= P.num_pages) {
        report(P.error_word, TL_DEVERR_PAGE_RANGE);
        page = -1;  // bad page: zeros
      }
    }
    s_page[r] = page;
  }
  __syncthreads();
  const int r0 = max(start - k0, 0), r1 = min(end - k0, kBN);  // keys of the tile to write
  const int units = P.h_kv * 16;                                // 16-byte units per key
  const int total = (r1 - r0) * units;
  uint32_t vmax = 0;  // max |bf16 bits| seen, per half-word
  for (int base = 0; base < total; base += kCvtThreads * kCvtUnroll) {
    uint4 x[kCvtUnroll];
#pragma unroll
    for (int i = 0; i < kCvtUnroll; ++i) {
      const int idx = base + i * kCvtThreads + (int)threadIdx.x;
      x[i] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < total) {
        const int r = r0 + idx / units, u = idx % units;
        const int page = s_page[r];
        if (page >= 0)
          x[i] = __ldg(reinterpret_cast<const uint4*>(
                           P.v_cache +
                           ((size_t)page * P.page_size + (k0 + r) % P.page_size) * P.h_kv * 128) +
                       u);
      }
    }
#pragma unroll
    for (int i = 0; i < kCvtUnroll; ++i) {
      const int idx = base + i * kCvtThreads + (int)threadIdx.x;
      if (idx < total) {
        const int r = r0 + idx / units, u = idx % units;
        uint4 y = x[i];
        vmax = max_u16x2(vmax, max_u16x2(max_u16x2(y.x & 0x7fff7fffu, y.y & 0x7fff7fffu),
                                         max_u16x2(y.z & 0x7fff7fffu, y.w & 0x7fff7fffu)));
        y = make_uint4(bf16x2_to_f16x2(y.x), bf16x2_to_f16x2(y.y), bf16x2_to_f16x2(y.z),
                       bf16x2_to_f16x2(y.w));
        *reinterpret_cast<uint4*>(ws + (((size_t)b * P.h_kv + (u >> 4)) * max_ctx + k0 + r) * 128 +
                                  (u & 15) * 8) = y;
      }
    }
  }
  const uint32_t m0 = vmax & 0xffffu, m1 = vmax >> 16;
  if ((m0 >= kBf16TooBig && m0 < kBf16Inf) || (m1 >= kBf16TooBig && m1 < kBf16Inf))
    report(P.error_word, TL_DEVERR_VALUE_RANGE);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(PrefillParams P, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap omap, int box_rows) {
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
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_u32(&sh.v_full[st]), kTcKVBytes);
          for (int hh = 0; hh < 2; ++hh)
            tma_load_3d(sV + st * kTcKVBytes + hh * (kTcKVBytes / 2), &vmap, hh * 64, key0,
                        b * P.h_kv + g, smem_u32(&sh.v_full[st]));
        }
        __syncwarp();
        ++v_issued;
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
      const uint32_t idPV = tc::idesc_f16(128, 128, 0, 1);
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
      auto issue_pv = [&](int a, int j) {  // O_a += P_a(j) V(j), fp16
        const uint32_t vt = sV + (j % kTcVS) * kTcKVBytes;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)  // keys [16k, 16k+16): P columns [8k, 8k+8)
          tc::mma_ts(tmem + 256 + a * 128, tmem + a * 128 + 8 * k,
                     tc::sdesc(vt + k * 2048, kTcKVBytes / 2, 1024), idPV,
                     (j > 0 || k > 0) ? 1u : 0u);
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
        if (!mbar_wait(smem_u32(&sh.v_full[j % kTcVS]), (j / kTcVS) & 1, abort_flag)) break;
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
    const int t = t0 + a * tpt + row / P.group;
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
      // takes the same rounded values
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = fast_exp2(fmaf(s[q * 32 + 2 * i], sc, -base));
          const float x1 = fast_exp2(fmaf(s[q * 32 + 2 * i + 1], sc, -base));
          pk[i] = pack_f16x2(x0, x1);
          float r0, r1;
          unpack_f16x2(pk[i], r0, r1);
          ls[i & 3] += r0 + r1;
        }
        tc::st16(tmem + lane_base + colS + q * 16, pk);
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
    // epilogue: O / l, staged in shared memory that the finished tile no
    // longer needs (tile 0: the K ring, free once O_0 is done because every S
    // MMA was issued before PV_0 of the last tile; tile 1: the Q tiles) as
    // four 128-byte-swizzled quarters of d, then written by TMA stores whose
    // box is the tile's (d quarter, heads of the group, tokens), clipped at T
    const bool have = ok && mbar_wait(smem_u32(&sh.o_done[a]), 0, abort_flag);
    const uint32_t stage = a == 0 ? sK : sQ;
    if (have) {
      tc::fence_after();
      const float inv = (p >= 0 && l > 0.f) ? 1.f / l : 0.f;
      float o[128];
#pragma unroll
      for (int q = 0; q < 4; ++q) tc::ld32(tmem + lane_base + colO + q * 32, o + q * 32);
      tc::wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t adr = stage + q * 16384 + row * 128 + ((i ^ (row & 7)) << 4);
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(adr),
                       "f"(o[q * 32 + 4 * i] * inv), "f"(o[q * 32 + 4 * i + 1] * inv),
                       "f"(o[q * 32 + 4 * i + 2] * inv), "f"(o[q * 32 + 4 * i + 3] * inv)
                       : "memory");
        }
    }
    fence_proxy_async_smem();
    named_barrier(1 + a, 128);  // every thread of the warpgroup gets here
    if ((warp & 3) == 2 && lane == 0 && !*abort_flag) {
      for (int q = 0; q < 4; ++q)
        tma_store_4d(&omap, q * 32, g * P.group, t0 + a * tpt, b, stage + q * 16384);
      bulk_commit_group();
      bulk_wait_read_all();
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
                                                       int32_t h_kv, int32_t d,
                                                       int32_t max_pages_per_seq,
                                                       int32_t page_size) {
  if (B <= 0 || T <= 0 || h_q <= 0 || h_kv <= 0 || d <= 0 || h_q % h_kv ||
      max_pages_per_seq <= 0 || page_size <= 0)
    return 0;
  // the fp16 copy of V: [B][h_kv][max_pages_per_seq * page_size][d]
  return (size_t)B * h_kv * ((size_t)max_pages_per_seq * page_size) * d * 2;
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
  if ((int64_t)max_pages_per_seq * page_size >= ((int64_t)1 << 31)) return TL_ERR_UNSUPPORTED;
  const size_t ws_need = tl_paged_attn_prefill_workspace_size(B, T, h_q, h_kv, d,
                                                              max_pages_per_seq, page_size);
  if (!workspace || !aligned16(workspace) || workspace_bytes < ws_need) return TL_ERR_WORKSPACE;
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
  const int max_ctx = max_pages_per_seq * page_size;
  CUtensorMap qmap, kmap, vmap, omap;
  {
    const uint64_t qd[3] = {128, (uint64_t)h_q, (uint64_t)B * T};
    const uint64_t qs[2] = {128 * 2, (uint64_t)h_q * 128 * 2};
    const uint32_t qb[3] = {64, (uint32_t)group, (uint32_t)tpt};
    const uint64_t kd[3] = {128, (uint64_t)h_kv, (uint64_t)num_pages * page_size};
    const uint64_t ks[2] = {128 * 2, (uint64_t)h_kv * 128 * 2};
    const uint32_t kb[3] = {64, 1, (uint32_t)box_rows};
    // the workspace's fp16 V: (d, key, row x KV head), 16-bit elements like bf16
    const uint64_t vd[3] = {128, (uint64_t)max_ctx, (uint64_t)B * h_kv};
    const uint64_t vs[2] = {128 * 2, (uint64_t)max_ctx * 128 * 2};
    const uint32_t vb[3] = {64, (uint32_t)kBN, 1};
    // the output, f32 (d, h_q, T, B): a TMA store box is one d quarter of a
    // query tile, clipped at T
    const uint64_t od[4] = {128, (uint64_t)h_q, (uint64_t)T, (uint64_t)B};
    const uint64_t os[3] = {128 * 4, (uint64_t)h_q * 128 * 4, (uint64_t)T * h_q * 128 * 4};
    const uint32_t ob[4] = {32, (uint32_t)group, (uint32_t)tpt, 1};
    if (!encode_f32_tensor_map(&omap, out, 4, od, os, ob, true)) return TL_ERR_CUDA;
    if (!encode_bf16_tensor_map(&qmap, q, 3, qd, qs, qb, true) ||
        !encode_bf16_tensor_map(&kmap, k_cache, 3, kd, ks, kb, true) ||
        !encode_bf16_tensor_map(&vmap, workspace, 3, vd, vs, vb, true))
      return TL_ERR_CUDA;
  }
  if (cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTcSmem) != cudaSuccess)
    return TL_ERR_CUDA;
  const int n_pairs = (T + 2 * tpt - 1) / (2 * tpt);
  if ((int64_t)B * h_kv > 0x7fffffff || n_pairs > 65535) return TL_ERR_UNSUPPORTED;
  prefill_v_f16_kernel<<<dim3((max_ctx + kBN - 1) / kBN, B), kCvtThreads, 0,
                         (cudaStream_t)stream>>>(P, static_cast<uint16_t*>(workspace), max_ctx);
  prefill_tc_kernel<<<dim3(B * h_kv, n_pairs), kTcThreads, kTcSmem, (cudaStream_t)stream>>>(
      P, qmap, kmap, vmap, omap, box_rows);
  return launch_status();
}
