// Prefill attention with every MMA in TMEM-operand form (included by
// paged_prefill.cu after its other kernels; it shares their helpers).
//
// The S = Q K^T and O += P V of one 128-row query tile, both as tcgen05 TS
// MMAs of one shape and type: M128 N128 K16 fp16, A from TMEM (Q, then P),
// B from shared memory MN-major (the workspace's K^T copy, then its V copy).
// A stream of such MMAs keeps the tensor pipe at its full rate (64 cycles a
// K16 step on GB300), where S from shared memory (SS) interleaved with TS
// P.V costs half as much again per MMA, whatever their order (the MMA probe,
// probe_mma.cu).  One query tile at a time: TMEM holds two S tiles of
// consecutive key tiles (S(j+1) is computed while the softmax works on
// S(j)), O, P and Q:
//   S0 [0, 128), S1 [128, 256), O [256, 384), P [384, 448), Q [448, 512).
// A work item is still a (query-tile pair, KV head) of the plan; its two
// tiles run one after the other, each over its own key range.
//
// Warps: 0 TMA producer (Q tiles, K^T and V tiles); 1 TMEM owner and MMA
// issuer (one lane); 2-5 softmax, one thread per row; 6-9 converter and
// epilogue: the tile's Q from shared memory to fp16 in TMEM, and the
// previous tile's O / l out through shared memory and TMA stores.
// Used for 16-bit pools, d = 128, rows without the split-P flag.
namespace tl {

constexpr int kTsThreads = 320;
constexpr int kTsQB = 2, kTsKS = 2, kTsVS = 2;
constexpr uint32_t kTsColO = 256, kTsColP = 384, kTsColQ = 448;
constexpr int kTsSmem = (kTsQB * kTcQBytes + (kTsKS + kTsVS) * kTcKVBytes) + 1024;

struct TsShared {
  unsigned long long q_full[kTsQB], q_free[kTsQB];
  unsigned long long k_full[kTsKS], k_empty[kTsKS], v_full[kTsVS], v_empty[kTsVS];
  unsigned long long s_full[2], p_full, p_free, qt_full, qt_free, o_done, o_free;
  unsigned long long l_full, l_free, stg_full, stg_free;
  unsigned long long item_full[kItemSlots], item_empty[kItemSlots], mma_drain;
  int item[kItemSlots];
  float inv_l[128];
  uint32_t tmem_base;
  int abort_flag;
};

// One query tile of an item: tile a of the pair, its tokens and key tiles.
struct TsTile {
  int t0, tile0, n;  // first token; first key tile and key tiles (n = 0: no live token)
  int kmin, kmax;
};
__device__ __forceinline__ TsTile ts_tile(const PrefillParams& P, const TcItem& it, int a, int tpt,
                                          int64_t cap) {
  TsTile t;
  t.t0 = it.t0 + a * tpt;
  const TcRange rg = tc_tile_range(P, it.b, t.t0, tpt, cap);
  t.kmin = rg.kmin;
  t.kmax = rg.kmax;
  t.tile0 = rg.kmax >= 0 ? rg.kmin / kBN : 0;
  t.n = rg.kmax >= 0 ? rg.kmax / kBN - t.tile0 + 1 : 0;
  return t;
}

// The item ring of tc_fetch, for this kernel's shared state.
__device__ __forceinline__ int ts_fetch(TsShared& sh, uint32_t seq, int* counter, int i_end,
                                        volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const uint32_t slot = seq % kItemSlots, ph = (seq / kItemSlots) & 1;
  int idx = -1;
  if (threadIdx.x < 32) {
    if (!mbar_wait(smem_u32(&sh.item_empty[slot]), ph ^ 1, abort_flag)) return -1;
    if (lane == 0) {
      const int v = atomicAdd(counter, 1);
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

// Eight bf16 (one 16-byte unit) as four fp16 pairs; `over` collects the
// finite values fp16 cannot hold.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x, bool& over) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t h[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo = w[k] & 0x7fffu, hi = (w[k] >> 16) & 0x7fffu;
    over |= (lo >= kBf16TooBig && lo < kBf16Inf) || (hi >= kBf16TooBig && hi < kBf16Inf);
    h[k] = bf16x2_to_f16x2(w[k]);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

__global__ void __launch_bounds__(kTsThreads, 1)
    prefill_ts_kernel(PrefillParams P, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap ktmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap omap, int* counter) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ TsShared sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase, sK = sQ + kTsQB * kTcQBytes, sV = sK + kTsKS * kTcKVBytes;
  volatile int* abort_flag = &sh.abort_flag;

  const int tpt = 128 / P.group;  // tokens per query tile
  const int rows_used = tpt * P.group;
  const int n_pairs = (P.T + 2 * tpt - 1) / (2 * tpt);
  const int64_t cap = position_cap(P);
  const uint32_t id16 = tc::idesc_f16(128, 128, 0, 1);  // every MMA of the kernel

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTsQB; ++i) {
      mbar_init(smem_u32(&sh.q_full[i]), 1);
      mbar_init(smem_u32(&sh.q_free[i]), 1);
    }
    for (int i = 0; i < kTsKS; ++i) {
      mbar_init(smem_u32(&sh.k_full[i]), 1);
      mbar_init(smem_u32(&sh.k_empty[i]), 1);
    }
    for (int i = 0; i < kTsVS; ++i) {
      mbar_init(smem_u32(&sh.v_full[i]), 1);
      mbar_init(smem_u32(&sh.v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&sh.s_full[i]), 1);
    mbar_init(smem_u32(&sh.p_full), 4);   // the four softmax warps
    mbar_init(smem_u32(&sh.p_free), 1);   // commit after each P.V
    mbar_init(smem_u32(&sh.qt_full), 4);  // the four converter warps
    mbar_init(smem_u32(&sh.qt_free), 1);  // commit after a tile's last S
    mbar_init(smem_u32(&sh.o_done), 1);   // commit after a tile's last P.V
    mbar_init(smem_u32(&sh.o_free), 4);   // the four epilogue warps
    mbar_init(smem_u32(&sh.l_full), 4);
    mbar_init(smem_u32(&sh.l_free), 4);
    mbar_init(smem_u32(&sh.stg_full), 128);
    mbar_init(smem_u32(&sh.stg_free), 1);
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(smem_u32(&sh.item_full[i]), 1);
      mbar_init(smem_u32(&sh.item_empty[i]), kTsThreads / 32 - 1);
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
  // a programmatic dependent of the plan kernel: the workspace (counter,
  // schedule, copies) is read only after this wait; the split-P kernel may
  // launch now and waits for this grid in turn
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int i_end = __ldcg(P.ctrl + 2);  // this kernel's items: those before the flagged rows'

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t kt = 0, vt = 0, ts = 0;
    bool ok = true;
    for (uint32_t seq = 0; ok; ++seq) {
      const int idx = ts_fetch(sh, seq, counter, i_end, abort_flag);
      if (idx < 0) break;
      const TcItem it = tc_item(P, idx, tpt, n_pairs, cap);
      const int vstart = __ldg(P.row_start + it.b);
      for (int a = 0; a < 2 && ok; ++a) {
        const TsTile tt = ts_tile(P, it, a, tpt, cap);
        if (tt.n == 0) continue;
        if (lane == 0) {  // the tile's Q, once its buffer's last output store has read it
          const uint32_t buf = ts % kTsQB;
          if (mbar_wait(smem_u32(&sh.q_free[buf]), ((ts / kTsQB) & 1) ^ 1, abort_flag)) {
            mbar_arrive_expect_tx(smem_u32(&sh.q_full[buf]), (uint32_t)(2 * 64 * rows_used * 2));
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sQ + buf * kTcQBytes + h * (kTcQBytes / 2), &qmap, h * 64,
                          it.g * P.group, it.b * P.T + tt.t0, smem_u32(&sh.q_full[buf]));
          } else {
            ok = false;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++ts;
        for (int j = 0; j < tt.n && ok; ++j) {
          const int key0 = (tt.tile0 + j) * kBN;
          if (lane == 0) {
            const uint32_t sk = kt % kTsKS, sv = vt % kTsVS;
            ok = mbar_wait(smem_u32(&sh.k_empty[sk]), ((kt / kTsKS) & 1) ^ 1, abort_flag);
            if (ok) {
              // K^T tile: two boxes of 64 keys x 128 d (the copy's key halves)
              mbar_arrive_expect_tx(smem_u32(&sh.k_full[sk]), kTcKVBytes);
              for (int h = 0; h < 2; ++h)
                tma_load_3d(sK + sk * kTcKVBytes + h * (kTcKVBytes / 2), &ktmap, h * 64,
                            key0 - vstart, it.b * P.h_kv + it.g, smem_u32(&sh.k_full[sk]));
            }
            ok = ok && mbar_wait(smem_u32(&sh.v_empty[sv]), ((vt / kTsVS) & 1) ^ 1, abort_flag);
            if (ok) {
              mbar_arrive_expect_tx(smem_u32(&sh.v_full[sv]), kTcKVBytes);
              for (int h = 0; h < 2; ++h)
                tma_load_3d(sV + sv * kTcKVBytes + h * (kTcKVBytes / 2), &vmap, h * 64,
                            key0 - vstart, it.b * P.h_kv + it.g, smem_u32(&sh.v_full[sv]));
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          ++kt;
          ++vt;
        }
      }
    }
    // drain: the copies this warp issued have landed before the CTA exits
    bool drained = true;
    if (lane == 0) {
      for (uint32_t i = kt > (uint32_t)kTsKS ? kt - kTsKS : 0; i < kt; ++i)
        drained &= mbar_drain(smem_u32(&sh.k_full[i % kTsKS]), (i / kTsKS) & 1);
      for (uint32_t i = vt > (uint32_t)kTsVS ? vt - kTsVS : 0; i < vt; ++i)
        drained &= mbar_drain(smem_u32(&sh.v_full[i % kTsVS]), (i / kTsVS) & 1);
      for (uint32_t i = ts > (uint32_t)kTsQB ? ts - kTsQB : 0; i < ts; ++i)
        drained &= mbar_drain(smem_u32(&sh.q_full[i % kTsQB]), (i / kTsQB) & 1);
      if (!drained) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    uint32_t kt = 0, vt = 0, sg = 0, pg = 0, ts = 0;
    bool ok = true;
    long long t_first = 0, wait_p = 0, wait_kv = 0;  // the step trace (zero without it)
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
      const int idx = ts_fetch(sh, seq, counter, i_end, abort_flag);
      if (idx < 0) break;
      const TcItem it = tc_item(P, idx, tpt, n_pairs, cap);
      for (int a = 0; a < 2 && ok; ++a) {
        const TsTile tt = ts_tile(P, it, a, tpt, cap);
        if (tt.n == 0) continue;
        if (lane == 0) {
          if (ts == 0) t_first = ptrace_clk();
          // S(j) into S buffer sg % 2: Q (TMEM) x the K^T tile; the tile's
          // last S frees the Q columns for the next tile's Q
          int s_next = 0;  // the tile's next S to issue
          auto issue_s = [&]() -> bool {
            const uint32_t sk = kt % kTsKS;
            if (!wait_for_kv(smem_u32(&sh.k_full[sk]), (kt / kTsKS) & 1)) return false;
            tc::fence_after();
            const uint32_t kb = sK + sk * kTcKVBytes;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc::mma_ts(tmem + 128 * (sg & 1), tmem + kTsColQ + 8 * k,
                         tc::sdesc(kb + k * 2048, kTcKVBytes / 2, 1024), id16, k > 0 ? 1u : 0u);
            tc::commit(smem_u32(&sh.s_full[sg & 1]));
            tc::commit(smem_u32(&sh.k_empty[sk]));
            ++kt;
            ++sg;
            if (++s_next == tt.n) tc::commit(smem_u32(&sh.qt_free));
            return true;
          };
          ok = mbar_wait(smem_u32(&sh.qt_full), ts & 1, abort_flag);
          if (ok) tc::fence_after();
          ok = ok && issue_s();
          if (ok && tt.n > 1) ok = issue_s();
          for (int j = 0; j < tt.n && ok; ++j) {
            const uint32_t sv = vt % kTsVS;
            if (!wait_for_p(smem_u32(&sh.p_full), pg & 1) ||
                !wait_for_kv(smem_u32(&sh.v_full[sv]), (vt / kTsVS) & 1) ||
                (j == 0 && ts > 0 && !mbar_wait(smem_u32(&sh.o_free), (ts - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            tc::fence_after();
            const uint32_t vb = sV + sv * kTcKVBytes;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc::mma_ts(tmem + kTsColO, tmem + kTsColP + 8 * k,
                         tc::sdesc(vb + k * 2048, kTcKVBytes / 2, 1024), id16,
                         (j > 0 || k > 0) ? 1u : 0u);
            tc::commit(smem_u32(&sh.p_free));
            tc::commit(smem_u32(&sh.v_empty[sv]));
            ++vt;
            ++pg;
            if (j == tt.n - 1) tc::commit(smem_u32(&sh.o_done));
            if (j + 2 < tt.n) ok = issue_s();
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++ts;
      }
    }
    if (lane == 0) {
      // every MMA this thread issued is done before TMEM is released
      tc::commit(smem_u32(&sh.mma_drain));
      if (!mbar_drain(smem_u32(&sh.mma_drain), 0)) *abort_flag = 1;
#if TL_PREFILL_TRACE
      if (ts > 0 && blockIdx.x < kPtraceCtas) {
        unsigned long long* row = g_ptrace[blockIdx.x];
        atomicAdd(row + TL_PTRACE_CYCLES, (unsigned long long)(ptrace_clk() - t_first));
        atomicAdd(row + TL_PTRACE_STEPS, (unsigned long long)pg);
        atomicAdd(row + TL_PTRACE_ITEMS, (unsigned long long)ts);
        atomicAdd(row + TL_PTRACE_WAIT_P, (unsigned long long)wait_p);
        atomicAdd(row + TL_PTRACE_WAIT_KV, (unsigned long long)wait_kv);
      }
#endif
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ softmax
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float sc = P.scale_log2;
    uint32_t sg = 0, pg = 0, ts = 0;
    bool ok = true;
    long long sm_wait_s = 0, sm_busy = 0;  // the step trace (zero without it)
    for (uint32_t seq = 0; ok; ++seq) {
      const int idx = ts_fetch(sh, seq, counter, i_end, abort_flag);
      if (idx < 0) break;
      const TcItem it = tc_item(P, idx, tpt, n_pairs, cap);
      for (int a = 0; a < 2 && ok; ++a) {
        const TsTile tt = ts_tile(P, it, a, tpt, cap);
        if (tt.n == 0) continue;
        const int t = tt.t0 + row / P.group;
        int p = -1;
        if (row < rows_used && t < P.T) {
          p = P.positions[(size_t)it.b * P.T + t];
          if (p >= cap) {
            report(P.error_word, TL_DEVERR_CONTEXT_RANGE);
            p = -1;
          }
        }
        const int lo = (P.window > 0 && p - P.window + 1 > 0) ? p - P.window + 1 : 0;
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; j < tt.n; ++j) {
          const long long tw = ptrace_clk();
          if (!mbar_wait(smem_u32(&sh.s_full[sg & 1]), (sg >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const long long tsb = ptrace_clk();
          sm_wait_s += tsb - tw;
          tc::fence_after();
          const int key0 = (tt.tile0 + j) * kBN;
          const int cmin = lo - key0, cmax = p - key0;  // live columns [cmin, cmax]
          const bool all_live = __all_sync(0xffffffffu, cmin <= 0 && cmax >= kBN - 1);
          float s[kBN];
#pragma unroll
          for (int q = 0; q < kBN / 32; ++q)
            tc::ld32(tmem + lane_base + 128 * (sg & 1) + q * 32, s + q * 32);
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
          // P = fp16(exp2(s*sc - base)); the sum takes the same rounded values
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
          const uint64_t sc2 = f32_twice(sc), nb2 = f32_twice(-base);
          uint32_t pk[kBN / 2];
#pragma unroll
          for (int i = 0; i < kBN / 2; ++i) {
            float y0, y1;
            fma_f32x2(s[2 * i], s[2 * i + 1], sc2, nb2, y0, y1);
            pk[i] = pack_f16x2(fast_exp2(y0), fast_exp2(y1));
            ls[i & 3] = add_f16x2_halves(ls[i & 3], pk[i]);
          }
          l = l * corr + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
          // the P columns and O are free once the previous P.V is done
          if (pg > 0 && !mbar_wait(smem_u32(&sh.p_free), (pg - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after();
          if (__any_sync(0xffffffffu, need)) {  // never at j = 0, where l is still 0
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float o[32];
              tc::ld32(tmem + lane_base + kTsColO + q * 32, o);
              tc::wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= corr;
              tc::st32(tmem + lane_base + kTsColO + q * 32, o);
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::st16(tmem + lane_base + kTsColP + q * 16, pk + 16 * q);
          tc::wait_st();
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sh.p_full));
          sm_busy += ptrace_clk() - tsb;
          ++sg;
          ++pg;
        }
        if (!ok) break;
        // the row's 1 / l for the epilogue, once it has taken the previous tile's
        if (ts > 0 && !mbar_wait(smem_u32(&sh.l_free), (ts - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        sh.inv_l[row] = (p >= 0 && l > 0.f) ? 1.f / l : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.l_full));
        ++ts;
        ok = ok && !*abort_flag;
      }
    }
#if TL_PREFILL_TRACE
    // the step trace's softmax fields, from this one warpgroup: counted twice
    // so that per-step figures divide by two steps as for the paired kernel
    if (warp == 2 && lane == 0 && blockIdx.x < kPtraceCtas) {
      atomicAdd(&g_ptrace[blockIdx.x][TL_PTRACE_SM_WAIT_S], (unsigned long long)(2 * sm_wait_s));
      atomicAdd(&g_ptrace[blockIdx.x][TL_PTRACE_SM_BUSY], (unsigned long long)(2 * sm_busy));
    }
#endif
  } else {
    // ------------------------------------------------ converter, epilogue
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const bool leader = warp == 6 && lane == 0;
    uint32_t ts = 0, rounds = 0;
    bool ok = true;
    bool q_over = false;
    // the previous tile's output: O / l through its own Q buffer (free
    // since its Q went to TMEM) in two rounds of two 128-byte-swizzled d
    // quarters, TMA stores clipped at T; then the buffer goes back to the
    // producer
    struct Pending {
      int b, g, t0, ts;
      bool live;
    } prev = {0, 0, 0, 0, false};
    auto epilogue = [&](const Pending& e) -> bool {
      const uint32_t buf = e.ts % kTsQB, stage = sQ + buf * kTcQBytes;
      if (!mbar_wait(smem_u32(&sh.l_full), e.ts & 1, abort_flag)) return false;
      const float inv = sh.inv_l[row];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.l_free));
      if (!mbar_wait(smem_u32(&sh.o_done), e.ts & 1, abort_flag)) return false;
      tc::fence_after();
      for (int r = 0; r < 2; ++r, ++rounds) {
        if (rounds > 0 && !mbar_wait(smem_u32(&sh.stg_free), (rounds - 1) & 1, abort_flag))
          return false;
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          float o[32];
          tc::ld32(tmem + lane_base + kTsColO + (2 * r + qq) * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t adr = stage + qq * 16384 + row * 128 + ((i ^ (row & 7)) << 4);
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(adr),
                         "f"(o[4 * i] * inv), "f"(o[4 * i + 1] * inv), "f"(o[4 * i + 2] * inv),
                         "f"(o[4 * i + 3] * inv)
                         : "memory");
          }
        }
        if (r == 1) {  // O is out of TMEM: the next tile's P.V may overwrite it
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sh.o_free));
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&sh.stg_full));
        if (leader) {
          if (mbar_wait(smem_u32(&sh.stg_full), rounds & 1, abort_flag) && !*abort_flag) {
            for (int qq = 0; qq < 2; ++qq)
              tma_store_4d(&omap, (2 * r + qq) * 32, e.g * P.group, e.t0, e.b, stage + qq * 16384);
            bulk_commit_group();
            bulk_wait_read_all();
          }
          mbar_arrive(smem_u32(&sh.stg_free));
        }
      }
      if (leader) mbar_arrive(smem_u32(&sh.q_free[buf]));
      return true;
    };
    for (uint32_t seq = 0; ok; ++seq) {
      const int idx = ts_fetch(sh, seq, counter, i_end, abort_flag);
      if (idx < 0) break;
      const TcItem it = tc_item(P, idx, tpt, n_pairs, cap);
      for (int a = 0; a < 2 && ok; ++a) {
        const TsTile tt = ts_tile(P, it, a, tpt, cap);
        if (tt.n == 0) {
          // no live token in the tile: its outputs are 0 (coalesced, one row a warp step)
          for (int e = row; e < rows_used * 32; e += 128) {
            const int r = e >> 5, c = (e & 31) * 4, tk = tt.t0 + r / P.group;
            if (tk < P.T)
              *reinterpret_cast<float4*>(P.out + (((size_t)it.b * P.T + tk) * P.h_q +
                                                  (size_t)it.g * P.group + r % P.group) *
                                                     128 +
                                         c) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          continue;
        }
        // this tile's Q: bf16 from its buffer to fp16 in TMEM, once the
        // previous tile's last S has read the Q columns
        const uint32_t buf = ts % kTsQB;
        ok = mbar_wait(smem_u32(&sh.q_full[buf]), (ts / kTsQB) & 1, abort_flag) &&
             (ts == 0 || mbar_wait(smem_u32(&sh.qt_free), (ts - 1) & 1, abort_flag));
        if (!ok) break;
        tc::fence_after();
        {
          const uint32_t qb = sQ + buf * kTcQBytes;
          uint32_t qh[64];
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint4 x;
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                           : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                           : "r"(qb + hf * (kTcQBytes / 2) + row * 128 + ((c ^ (row & 7)) << 4)));
              if (row >= rows_used) x = make_uint4(0u, 0u, 0u, 0u);  // rows past the box
              const uint4 h = bf16x8_to_f16x8(x, q_over);
              qh[32 * hf + 4 * c] = h.x;
              qh[32 * hf + 4 * c + 1] = h.y;
              qh[32 * hf + 4 * c + 2] = h.z;
              qh[32 * hf + 4 * c + 3] = h.w;
            }
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::st16(tmem + lane_base + kTsColQ + q * 16, qh + 16 * q);
          tc::wait_st();
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.qt_full));
        // the previous tile's output, while this tile's S and softmax run
        if (prev.live && !epilogue(prev)) {
          ok = false;
          break;
        }
        prev = {it.b, it.g, tt.t0, (int)ts, true};
        ++ts;
        ok = ok && !*abort_flag;
      }
    }
    if (ok && prev.live) ok = epilogue(prev);
    if (__any_sync(0xffffffffu, q_over) && lane == 0) report(P.error_word, TL_DEVERR_VALUE_RANGE);
    if (leader) bulk_wait_read_all();
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
