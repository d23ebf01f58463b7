// Device helpers shared by the paged-attention kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tl_paged_attn.h"

#define TL_DEVINLINE __device__ __forceinline__

namespace tl {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- cp.async --

TL_DEVINLINE uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes < 16 zero-fills the rest
// (src_bytes = 0 reads nothing and writes 16 zero bytes).
TL_DEVINLINE void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
TL_DEVINLINE void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
TL_DEVINLINE void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ------------------------------------------------------ ldmatrix / mma.sync --

TL_DEVINLINE void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
TL_DEVINLINE void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                    uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
TL_DEVINLINE void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                 uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two f32 -> one bf16x2 register (round to nearest even); lo in the low half.
TL_DEVINLINE uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// (a, b) ~ hi + lo with hi = bf16(a, b) and lo = bf16 of the remainders: the
// pair carries about 16 significant bits, so a bf16 x bf16 product of the
// pair with an exact bf16 operand keeps f32-level accuracy in two MMAs.
TL_DEVINLINE void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  const float ah = __uint_as_float(hi << 16);
  const float bh = __uint_as_float(hi & 0xffff0000u);
  lo = pack_bf16x2(a - ah, b - bh);
}

TL_DEVINLINE float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

TL_DEVINLINE float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
TL_DEVINLINE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- mbarrier --
// Every wait in this library is bounded: after kWaitCycles of polling it sets
// the CTA's abort flag and gives up, and every other wait of the CTA gives up
// as soon as it sees the flag, so no kernel can spin forever.

#ifndef TL_WAIT_CYCLES
#define TL_WAIT_CYCLES (1ll << 31)  // about one second at 2 GHz
#endif
constexpr long long kWaitCycles = TL_WAIT_CYCLES;

TL_DEVINLINE void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
TL_DEVINLINE void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
TL_DEVINLINE void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
TL_DEVINLINE void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Arrive on `bar` once all of this thread's earlier cp.async copies have landed
// (the arrival counts against the barrier's expected count).
TL_DEVINLINE void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completing `bytes` of transaction count on `bar`.
TL_DEVINLINE void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Tiled TMA load of a 3-D box, completing its bytes on `bar`.  The
// innermost coordinate times the element size must be a multiple of 16 bytes.
TL_DEVINLINE void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// The same load with an L2 eviction-priority policy (see l2_evict_first).
TL_DEVINLINE void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                   uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;\n"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar),
      "l"(policy)
      : "memory");
}
// L2 policies: data read once (the KV pools in decode) goes first when L2
// needs room; data written to be read back soon (split partials) stays.
TL_DEVINLINE uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
TL_DEVINLINE uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
TL_DEVINLINE void st_f32x4_hint(float* ptr, float a, float b, float c, float d, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;\n" ::"l"(ptr), "f"(a),
               "f"(b), "f"(c), "f"(d), "l"(policy)
               : "memory");
}
TL_DEVINLINE void st_f32x2_hint(float* ptr, float a, float b, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;\n" ::"l"(ptr), "f"(a), "f"(b),
               "l"(policy)
               : "memory");
}
// Tiled TMA store of a 4-D box from shared memory (bulk-group completion);
// elements past the tensor's extent are not written.
TL_DEVINLINE void tma_store_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3,
                               uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];\n"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
      : "memory");
}
TL_DEVINLINE void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Wait until every committed bulk store of this thread has read its source.
TL_DEVINLINE void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
TL_DEVINLINE void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}
TL_DEVINLINE void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
TL_DEVINLINE bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of `bar` with the given parity; false on timeout or abort.
TL_DEVINLINE bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// Bounded wait that ignores the abort flag: used to drain a CTA's own copies
// in flight before it exits.
TL_DEVINLINE bool mbar_drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
}

TL_DEVINLINE void report(uint32_t* error_word, uint32_t bit) {
  if (error_word) atomicOr(error_word, bit);
}

}  // namespace tl

// ------------------------------------------------------------ host helpers --

namespace tl {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int num_sms();  // SM count of the current device (cached per device)

// Encode a tiled bf16 tensor map of `rank` dims (dims[0] innermost, strides
// in bytes for dims 1..rank-1) with the given box and 128-byte swizzle when
// `swizzle128`; out-of-range boxes fill with zeros.  False on failure.
bool encode_bf16_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides, const uint32_t* box, bool swizzle128);
// The same for f32 elements.
bool encode_f32_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides, const uint32_t* box, bool swizzle128);
// The same for 8-bit elements (e4m3 codes).
bool encode_u8_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box, bool swizzle128);

inline tl_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

}  // namespace tl
