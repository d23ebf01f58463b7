// tcgen05.mma cost by shape: the cycles one CTA's tensor core spends per K16
// MMA when n MMAs are issued back to back by one thread (8 at a time, the
// loop unrolled and the descriptors formed from constants, so the thread
// issues faster than the pipe retires) and committed once.
// A measurement tool, built as its own library (not part of libtlpa.so):
// python -m paged_kv_attention_cache_gb300.probe_mma.  Operands are zeros in
// shared memory (the timing does not depend on values); the commit's wait is
// bounded and a wait that gives up reports -1.
//
// Forms (all M = 128 unless named, K = 16, f32 accumulator in TMEM):
//   0 SS N=128 bf16     1 TS N=128 fp16 (A from TMEM)   2 SS N=256 bf16
//   3 TS N=256 fp16     4 SS N=128, accumulator switched every 8 MMAs
//   5 SS N=64           6 SS N=192                      7 SS M=64 N=128
//   8 SS N=32
//   9 the attention kernel's order, groups of 8: TS N=128 into columns 256
//     (A from columns 0..63), SS N=128 into 0, TS into 384 (A from 128..191),
//     SS into 128 (P.V and S of two query tiles in turn)
//  10 form 9 while warps 1-3 load 32-column TMEM blocks of their lanes
//     (columns 128..255) in a loop, as softmax warps do (timing only: the
//     loaded values are not used)
//  11 the same groups in the order PV0, PV1, S0, S1: no S group right after
//     the P.V group that read the columns it overwrites
//  12 form 9's kinds and order with no column shared between the groups: the
//     TS groups read A from columns 448..511, which no MMA writes, and
//     accumulate into 256..383
//  13 groups of 8 alternating SS bf16 and SS fp16 (same operands, another
//     instruction descriptor)
//  14 groups alternating TS bf16 (A from TMEM) and SS bf16
//  15 groups alternating TS fp16 and TS bf16
//  16 groups TS bf16, SS bf16, SS bf16 in turn (one TS group to two SS)
//  17 groups TS bf16, TS bf16, SS bf16 in turn (two TS groups to one SS)
//  18 one query tile with Q in TMEM: groups alternating S = Q K^T (TS bf16,
//     A = Q in columns 448..511, D = columns 0..127 or 128..255 in turn) and
//     O += P V (TS fp16, A = the P in the other S buffer, D = 256..383)
//  19 SS groups whose A alternates between two shared-memory tiles and whose
//     D alternates between columns 0 and 128 (S0, S1 alone)
//  20 TS groups whose A alternates between columns 0 and 128 and whose D
//     alternates between 256 and 384 (PV0, PV1 alone)
//  21 TS groups, A always from columns 0..63, D alternating 256 / 384
//  22 TS groups, A alternating 0 / 128, D always 256
//  23 TS groups, A fixed (448), D alternating 0 / 256, each group starting
//     a fresh accumulator (the first MMA of a group does not accumulate)
//  24 form 22 with every group starting a fresh accumulator
//  25 one query tile, all TS, no MMA reading what an MMA wrote: S = Q K^T
//     (A = Q in columns 448..511) into 0..127 or 128..255 in turn, fresh
//     each group, alternating with O += P V (A = P in columns 384..447,
//     D = 256..383)
//  26 form 25 with both groups fp16 and S's B operand K-major (as K tiles
//     are), P.V's MN-major (as V tiles are)
//  27 form 26 with S in bf16
//  28 form 26 with P.V too starting a fresh accumulator each group
//  29 form 26 with S too accumulating (no fresh accumulator anywhere)
//  30 TS fp16, A fixed (448), D in turn 0, 256, 128, 256 (three accumulators)
//  31 TS fp16, A fixed (448), D in turn 0, 128, 256, 384 (four accumulators)
//  32 TS fp16, D fixed (256), A alternating 384 / 448
//  33 TS fp16, D fixed (0), A alternating 256 / 384
//  34 TS fp16, D fixed (256), A alternating 0 / 64
//  35 TS fp16, (A, D) alternating (448, 0) / (384, 256): one S buffer
//  36 TS fp16, (A, D) in turn (448, 0), (384, 256), (448, 128), (384, 256)
//  37 form 36 with both B operands K-major (one instruction descriptor)
//  38 form 37 with P read from the other S buffer (as when P replaces S)
//  39 TS fp16 N=64, A fixed (448), D = 0, MN-major B
//  40 two query tiles with Q in TMEM and 64-key S tiles, all TS fp16
//     MN-major: per tile, 8 S MMAs N=64 (A = Q_a at 384 + 64a, D = 64a) then
//     4 P.V MMAs N=128 (A = P_a in S_a's columns, D = O_a at 256 + 128a)
//  41 the attention order PV0, S0, PV1, S1 with P.V too from shared memory:
//     S = SS bf16 (B K-major) into 0 / 128, P.V = SS fp16 (A K-major at the
//     Q tile's place + 32 KiB, B MN-major) into 256 / 384
// The marginal cost per MMA is (t(n1) - t(n0)) / (n1 - n0), which takes out
// the issue-to-first-MMA and commit latencies.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tcgen05.cuh"

namespace tl {
namespace probe {

constexpr int kForms = 42;
constexpr int kSmemBytes = 100 * 1024;

__device__ __forceinline__ long long clk() {
  long long c;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
  return c;
}
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One K tile (8 MMAs) of form F, unrolled with its descriptors formed from
// constants, so that the issuing thread runs ahead of the tensor pipe.
template <int F>
__device__ __forceinline__ void issue8(uint32_t tm, uint32_t sb, uint32_t id_ss, uint32_t id_ts,
                                       int i8) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t a_ss = tc::sdesc(sb + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
    const uint64_t b_ss = tc::sdesc(sb + 32768 + (kk >> 2) * 32768 + (kk & 3) * 32, 16, 1024);
    const uint64_t b_ts = tc::sdesc(sb + 32768 + kk * 2048, 16384, 1024);
    if (F == 1 || F == 3) {
      // A: fp16 in TMEM columns [0, 64) (8 columns a K step); D at column 256
      tc::mma_ts(tm + 256, tm + 8 * kk, b_ts, id_ts, i8 > 0 || kk > 0);
    } else if (F == 13) {
      const uint32_t id = (i8 & 1) ? tc::idesc_f16(128, 128, 0, 0) : id_ss;
      tc::mma_ss(tm + 128 * (i8 & 1), a_ss, b_ss, id, kk > 0);
    } else if (F == 14) {
      if (i8 & 1)
        tc::mma_ss(tm, a_ss, b_ss, id_ss, kk > 0);
      else
        tc::mma_ts(tm + 256, tm + 448 + 8 * kk, b_ts, tc::idesc_bf16(128, 128, 0, 1), 1u);
    } else if (F == 19) {
      const uint64_t a2 = tc::sdesc(sb + (i8 & 1) * 65536 + (kk >> 2) * 16384 + (kk & 3) * 32, 16,
                                    1024);
      tc::mma_ss(tm + 128 * (i8 & 1), a2, b_ss, id_ss, kk > 0);
    } else if (F == 41) {
      const int g = i8 & 3, tile = g >> 1;
      if ((g & 1) == 0)
        tc::mma_ss(tm + 256 + 128 * tile,
                   tc::sdesc(sb + 65536 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), b_ts,
                   id_ts, 1u);
      else
        tc::mma_ss(tm + 128 * tile, a_ss, b_ss, id_ss, kk > 0);
    } else if (F == 39) {
      tc::mma_ts(tm, tm + 448 + 8 * kk, b_ts, tc::idesc_f16(128, 64, 0, 1), 1u);
    } else if (F == 40) {
      // groups of 8: S0 (8 x N=64), PV0 (4) + PV0 (4, next K half), S1, PV1
      const int g = i8 & 3, tile = g >> 1;
      if ((g & 1) == 0)
        tc::mma_ts(tm + 64 * tile, tm + 384 + 64 * tile + 8 * kk, b_ts, tc::idesc_f16(128, 64, 0, 1),
                   kk > 0);
      else
        tc::mma_ts(tm + 256 + 128 * tile, tm + 64 * tile + 8 * (kk & 3), b_ts, id_ts, 1u);
    } else if (F == 37 || F == 38) {
      const int g = i8 & 3;
      const uint32_t id = tc::idesc_f16(128, 128, 0, 0);
      if ((g & 1) == 0)
        tc::mma_ts(tm + 128 * (g >> 1), tm + 448 + 8 * kk, b_ss, id, 1u);
      else
        tc::mma_ts(tm + 256, tm + (F == 37 ? 384u : 128u * ((g >> 1) ^ 1)) + 8 * kk, b_ss, id, 1u);
    } else if (F >= 35) {
      const int g = i8 & 3;
      const uint32_t a = (g & 1) ? 384u : 448u;
      const uint32_t d = (g & 1) ? 256u : (F == 35 ? 0u : 128u * (g >> 1));
      tc::mma_ts(tm + d, tm + a + 8 * kk, b_ts, id_ts, 1u);
    } else if (F >= 32) {
      const uint32_t a0 = F == 32 ? 384u : F == 33 ? 256u : 0u;
      const uint32_t a1 = F == 32 ? 448u : F == 33 ? 384u : 64u;
      const uint32_t d = F == 33 ? 0u : 256u;
      tc::mma_ts(tm + d, tm + ((i8 & 1) ? a1 : a0) + 8 * kk, b_ts, id_ts, 1u);
    } else if (F == 30 || F == 31) {
      const int g = i8 & 3;
      const uint32_t d = F == 30 ? (g & 1 ? 256u : 128u * (g >> 1)) : 128u * g;
      tc::mma_ts(tm + d, tm + 448 + 8 * kk, b_ts, id_ts, 1u);
    } else if (F == 28 || F == 29) {
      if ((i8 & 1) == 0)
        tc::mma_ts(tm + 128 * ((i8 >> 1) & 1), tm + 448 + 8 * kk, b_ss,
                   tc::idesc_f16(128, 128, 0, 0), F == 29 ? 1u : (uint32_t)(kk > 0));
      else
        tc::mma_ts(tm + 256, tm + 384 + 8 * kk, b_ts, id_ts, F == 29 ? 1u : (uint32_t)(kk > 0));
    } else if (F == 26 || F == 27) {
      if ((i8 & 1) == 0)
        tc::mma_ts(tm + 128 * ((i8 >> 1) & 1), tm + 448 + 8 * kk, b_ss,
                   F == 26 ? tc::idesc_f16(128, 128, 0, 0) : tc::idesc_bf16(128, 128, 0, 0),
                   kk > 0);
      else
        tc::mma_ts(tm + 256, tm + 384 + 8 * kk, b_ts, id_ts, 1u);
    } else if (F == 25) {
      if ((i8 & 1) == 0)
        tc::mma_ts(tm + 128 * ((i8 >> 1) & 1), tm + 448 + 8 * kk, b_ts,
                   tc::idesc_bf16(128, 128, 0, 1), kk > 0);
      else
        tc::mma_ts(tm + 256, tm + 384 + 8 * kk, b_ts, id_ts, 1u);
    } else if (F == 23) {
      tc::mma_ts(tm + 256 * (i8 & 1), tm + 448 + 8 * kk, b_ts, id_ts, kk > 0);
    } else if (F == 24) {
      tc::mma_ts(tm + 256, tm + 128 * (i8 & 1) + 8 * kk, b_ts, id_ts, kk > 0);
    } else if (F >= 20) {
      const uint32_t a_col = F == 21 ? 0u : 128u * (i8 & 1);
      const uint32_t d_col = F == 22 ? 256u : 256u + 128u * (i8 & 1);
      tc::mma_ts(tm + d_col, tm + a_col + 8 * kk, b_ts, id_ts, 1u);
    } else if (F == 18) {
      const int buf = (i8 >> 1) & 1;  // the S buffer this pair of groups writes
      if ((i8 & 1) == 0)
        tc::mma_ts(tm + 128 * buf, tm + 448 + 8 * kk, b_ts, tc::idesc_bf16(128, 128, 0, 1),
                   kk > 0);
      else
        tc::mma_ts(tm + 256, tm + 128 * (buf ^ 1) + 8 * kk, b_ts, id_ts, 1u);
    } else if (F == 16 || F == 17) {
      const int ph = i8 % 3;
      const bool ts_grp = F == 16 ? ph == 0 : ph < 2;
      if (ts_grp)
        tc::mma_ts(tm + 256, tm + 448 + 8 * kk, b_ts, tc::idesc_bf16(128, 128, 0, 1), 1u);
      else
        tc::mma_ss(tm, a_ss, b_ss, id_ss, kk > 0);
    } else if (F == 15) {
      const uint32_t id = (i8 & 1) ? tc::idesc_bf16(128, 128, 0, 1) : id_ts;
      tc::mma_ts(tm + 256, tm + 448 + 8 * kk, b_ts, id, 1u);
    } else if (F == 12) {
      const int grp = i8 & 3;  // PV0, S0, PV1, S1 without shared columns
      if ((grp & 1) == 0)
        tc::mma_ts(tm + 256, tm + 448 + 8 * kk, b_ts, id_ts, 1u);
      else
        tc::mma_ss(tm + 128 * (grp >> 1), a_ss, b_ss, id_ss, kk > 0);
    } else if (F == 11) {
      const int grp = i8 & 3;  // PV0, PV1, S0, S1
      const int tile = grp & 1;
      if (grp < 2)
        tc::mma_ts(tm + 256 + 128 * tile, tm + 128 * tile + 8 * kk, b_ts, id_ts, kk > 0);
      else
        tc::mma_ss(tm + 128 * tile, a_ss, b_ss, id_ss, kk > 0);
    } else if (F >= 9) {
      const int grp = i8 & 3;  // PV0, S0, PV1, S1
      const int tile = grp >> 1;
      if ((grp & 1) == 0)
        tc::mma_ts(tm + 256 + 128 * tile, tm + 128 * tile + 8 * kk, b_ts, id_ts, kk > 0);
      else
        tc::mma_ss(tm + 128 * tile, a_ss, b_ss, id_ss, kk > 0);
    } else {
      // A: K-major bf16 at sb (two 64-element K blocks of 16 KiB); B: K-major
      // at sb + 32 KiB (two blocks of 32 KiB, room for N = 256)
      const uint32_t d = F == 4 && (i8 & 1) ? tm + 256 : tm;
      tc::mma_ss(d, a_ss, b_ss, id_ss, i8 > 0 || kk > 0);
    }
  }
}

template <int F>
__global__ void __launch_bounds__(128) mma_issue_kernel(int n8, long long* out) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint32_t tbase;
  __shared__ __align__(8) unsigned long long bar;
  __shared__ uint32_t stop;  // form 10: set when the timing thread is done
  const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t sb = (s0 + 1023u) & ~1023u;  // 96 KiB of zeros from here
  for (int i = threadIdx.x; i < 96 * 1024 / 16; i += blockDim.x)
    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(sb + i * 16), "r"(0u));
  const uint32_t bar_a = (uint32_t)__cvta_generic_to_shared(&bar);
  if (threadIdx.x == 0) {
    stop = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_a));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (threadIdx.x < 32) tc::alloc((uint32_t)__cvta_generic_to_shared(&tbase), 512);
  asm volatile("fence.proxy.async.shared::cta;");
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm = tbase;
  if (threadIdx.x == 0) {
    constexpr int N = F == 2 || F == 3 ? 256 : F == 5 ? 64 : F == 6 ? 192 : F == 8 ? 32 : 128;
    constexpr int M = F == 7 ? 64 : 128;
    const uint32_t id_ss = tc::idesc_bf16(M, N, 0, 0);
    const uint32_t id_ts = tc::idesc_f16(128, N, 0, 1);
    const long long t0 = clk();
    const unsigned long long g0 = gtimer();
#pragma unroll 1
    for (int i8 = 0; i8 < n8; ++i8) issue8<F>(tm, sb, id_ss, id_ts, i8);
    tc::commit(bar_a);
    bool done = false;
    for (long long n = 0; n < (1ll << 26) && !done; ++n) {
      uint32_t ok;
      asm volatile(
          "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0; "
          "selp.u32 %0, 1, 0, p; }"
          : "=r"(ok)
          : "r"(bar_a)
          : "memory");
      done = ok != 0;
    }
    out[0] = done ? clk() - t0 : -1;
    out[1] = done ? (long long)(gtimer() - g0) : -1;
    asm volatile("st.volatile.shared.u32 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(&stop)));
  } else if (F == 10 && threadIdx.x >= 32) {
    // warps 1-3: TMEM loads of their lane quarter until the timing thread is
    // done (bounded)
    const uint32_t lanes = (uint32_t)(32 * (threadIdx.x >> 5)) << 16;
    float v[32], acc = 0.f;
    for (int r = 0; r < (1 << 20); ++r) {
      uint32_t st;
      asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(st)
                   : "r"((uint32_t)__cvta_generic_to_shared(&stop)));
      // one decision per warp: the TMEM loads below are warp-collective
      if (__shfl_sync(0xffffffffu, st, 0)) break;
      for (int q = 0; q < 4; ++q) tc::ld32(tm + lanes + 128 + 32 * q, v);
      tc::wait_ld();
      acc += v[0];
    }
    if (acc == 12345.f) out[2] = 1;  // keeps the loads
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (threadIdx.x < 32) tc::dealloc(tm, 512);
}

template <int F>
cudaError_t launch_probe(int n8, long long* d) {
  cudaFuncSetAttribute(mma_issue_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kSmemBytes);
  mma_issue_kernel<F><<<1, 128, kSmemBytes>>>(n8, d);
  return cudaGetLastError();
}

}  // namespace probe
}  // namespace tl

// Cycles (clock64) and nanoseconds (%globaltimer) from the first MMA's issue
// to the commit's arrival for n_mma (a multiple of 8) back-to-back MMAs of
// `form` on one CTA of the current device, in cycles_ns[0] and [1] (-1 when
// the bounded wait gave up).  Returns 0, 1 for a bad form or count, 3 for a
// CUDA error.
extern "C" int tl_probe_mma_cycles(int form, int n_mma, long long* cycles_ns) {
  using namespace tl::probe;
  if (form < 0 || form >= kForms || n_mma < 8 || n_mma > 4096 || n_mma % 8 || !cycles_ns)
    return 1;
  long long* d = nullptr;
  if (cudaMalloc(&d, 3 * sizeof(long long)) != cudaSuccess) return 3;
  const int n8 = n_mma / 8;
  cudaError_t e;
  switch (form) {
    case 0: e = launch_probe<0>(n8, d); break;
    case 1: e = launch_probe<1>(n8, d); break;
    case 2: e = launch_probe<2>(n8, d); break;
    case 3: e = launch_probe<3>(n8, d); break;
    case 4: e = launch_probe<4>(n8, d); break;
    case 5: e = launch_probe<5>(n8, d); break;
    case 6: e = launch_probe<6>(n8, d); break;
    case 7: e = launch_probe<7>(n8, d); break;
    case 8: e = launch_probe<8>(n8, d); break;
    case 9: e = launch_probe<9>(n8, d); break;
    case 10: e = launch_probe<10>(n8, d); break;
    case 11: e = launch_probe<11>(n8, d); break;
    case 12: e = launch_probe<12>(n8, d); break;
    case 13: e = launch_probe<13>(n8, d); break;
    case 14: e = launch_probe<14>(n8, d); break;
    case 15: e = launch_probe<15>(n8, d); break;
    case 16: e = launch_probe<16>(n8, d); break;
    case 17: e = launch_probe<17>(n8, d); break;
    case 18: e = launch_probe<18>(n8, d); break;
    case 19: e = launch_probe<19>(n8, d); break;
    case 20: e = launch_probe<20>(n8, d); break;
    case 21: e = launch_probe<21>(n8, d); break;
    case 22: e = launch_probe<22>(n8, d); break;
    case 23: e = launch_probe<23>(n8, d); break;
    case 24: e = launch_probe<24>(n8, d); break;
    case 25: e = launch_probe<25>(n8, d); break;
    case 26: e = launch_probe<26>(n8, d); break;
    case 27: e = launch_probe<27>(n8, d); break;
    case 28: e = launch_probe<28>(n8, d); break;
    case 29: e = launch_probe<29>(n8, d); break;
    case 30: e = launch_probe<30>(n8, d); break;
    case 31: e = launch_probe<31>(n8, d); break;
    case 32: e = launch_probe<32>(n8, d); break;
    case 33: e = launch_probe<33>(n8, d); break;
    case 34: e = launch_probe<34>(n8, d); break;
    case 35: e = launch_probe<35>(n8, d); break;
    case 36: e = launch_probe<36>(n8, d); break;
    case 37: e = launch_probe<37>(n8, d); break;
    case 38: e = launch_probe<38>(n8, d); break;
    case 39: e = launch_probe<39>(n8, d); break;
    case 40: e = launch_probe<40>(n8, d); break;
    default: e = launch_probe<41>(n8, d); break;
  }
  if (e == cudaSuccess) e = cudaMemcpy(cycles_ns, d, 2 * sizeof(long long), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return e == cudaSuccess ? 0 : 3;
}
