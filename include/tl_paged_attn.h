/*
 * tl_paged_attn.h -- paged attention over a block-table KV cache, for GB300
 * (sm_103a).  C ABI: plain pointers and sizes, no framework types.
 *
 * The operations and their arguments follow "How serving works in Tlaloc":
 *   - section 1 "From a model to DXIR": per layer, KV_CACHE_WRITE (K and V)
 *     then PAGED_ATTENTION; a prefill call holds one right-aligned row per
 *     sequence, padding tokens first with slot -1 (never written), each live
 *     token with its own position, causal length = position + 1;
 *   - section 2 "From DXIR to StableHLO": attention gathers the pages a
 *     sequence's block table names, takes a dot, a masked softmax and a dot;
 *     a prefill row's pages are shared by all its tokens; "Blockwise
 *     attention": a context spanning several 2,048-key blocks is folded one
 *     block at a time with a running max, sum and P.V, so no context-wide
 *     score tensor exists;
 *   - section 3 "The serving artifact": the pool is numBlocks pages of
 *     blockSize tokens for K and for V; the argument roles are POSITIONS,
 *     BLOCK_TABLES, SEQ_LENS, SLOT_MAPPING, KV_POOL_IN/OUT, and the pools are
 *     updated in place; "Sliding-window layers": a window W reads positions
 *     p-W+1 .. p only.
 * Grouped-query sharing and the paging data structure follow "Serving Models",
 * "Change the cache at the architectural level" and "Logical histories and
 * physical pages".
 *
 * Conventions shared by every entry point
 *   Layout.   k_cache, v_cache: [num_pages][page_size][H_kv][d], row-major,
 *             so slot s = page * page_size + offset is one contiguous row of
 *             H_kv * d elements.  block_table: [B][max_pages_per_seq] int32;
 *             entry i of row b is the physical page of the sequence's logical
 *             block i (positions i*page_size .. (i+1)*page_size-1); entries
 *             past the sequence's last page are never read.  Query head h
 *             reads KV head h / (H_q / H_kv).
 *   Memory.   Every pointer is a DEVICE pointer owned by the caller, except
 *             where stated.  The library allocates nothing.  Base pointers
 *             must be 16-byte aligned.  All work is enqueued on `stream`
 *             (a cudaStream_t; NULL = the legacy default stream); nothing
 *             synchronises.
 *   Errors.   Arguments are validated on the host before any launch; on a
 *             non-TL_OK return nothing was enqueued and nothing was written.
 *             Launch failures return TL_ERR_CUDA.  Values the host cannot see
 *             (slots, block-table entries, lengths, positions) are checked on
 *             the device: an access they would take out of range is skipped
 *             (the key counts as masked, the row as not written) and the
 *             matching TL_DEVERR_* bit is OR-ed into *error_word when
 *             error_word is not NULL.  Pipeline waits inside a kernel are
 *             bounded (about a second); one that gives up sets
 *             TL_DEVERR_TIMEOUT and the kernel returns.
 *   Unused slots.  Slots of a listed page past a sequence's last position
 *             may hold anything, NaN included: they are never weighted.
 */
#ifndef TL_PAGED_ATTN_H
#define TL_PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TL_OK = 0,
  TL_ERR_INVALID_ARG = 1,   /* a null pointer, a bad size, misalignment */
  TL_ERR_UNSUPPORTED = 2,   /* valid, but not a shape or dtype the library runs */
  TL_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  TL_ERR_DEVICE_BOUNDS = 4, /* tl_get_device_error only: a device-side check found a value
                               out of range (any TL_DEVERR_* bit but TL_DEVERR_TIMEOUT) */
  TL_ERR_WORKSPACE = 5,     /* workspace missing or smaller than required */
  TL_ERR_DEVICE_TIMEOUT = 6 /* tl_get_device_error only: an in-kernel wait gave up
                               (TL_DEVERR_TIMEOUT; outputs invalid) */
} tl_status;

typedef enum {
  TL_F32 = 0,       /* IEEE binary32 */
  TL_BF16 = 1,      /* bfloat16 */
  TL_FP8_E4M3 = 2,  /* e4m3fn codes (fp8 KV pools only; see tl_kv_cache_write_fp8) */
  TL_INT8 = 3       /* int8 codes with per-row f32 scales (the workspace query of
                       tl_paged_attn_prefill_int8; the int8 calls take no dtype) */
} tl_dtype;

/* Bits OR-ed into *error_word by the device-side checks. */
#define TL_DEVERR_SLOT_RANGE 1u    /* a slot outside [0, num_pages*page_size), not -1 */
#define TL_DEVERR_PAGE_RANGE 2u    /* a needed block-table entry outside [0, num_pages) */
#define TL_DEVERR_CONTEXT_RANGE 4u /* a length / position past max_pages_per_seq*page_size */
#define TL_DEVERR_TIMEOUT 8u       /* an internal pipeline wait gave up (outputs invalid) */
#define TL_DEVERR_VALUE_RANGE 16u  /* a finite value beyond fp16's +-65504 where the path rounds to
                                      fp16: V in prefill, q in decode over e4m3 or int8 pools
                                      (outputs invalid); or a non-finite value written into an
                                      int8 pool (written as code 0) */
#define TL_DEVERR_PLAN_CAPACITY 32u /* the decode plan cut the batch into more pieces than its
                                       workspace holds: nothing was attended and every output
                                       is 0 (a library fault; the plan's arithmetic keeps the
                                       pieces within the bound) */

/*
 * The device-side error word ("How serving works in Tlaloc", the Triton
 * backend bullets: a request the pool cannot serve is refused by name).
 * Every entry point that launches work takes an optional `error_word`
 * (a device uint32, owned by the caller, zeroed by the caller before the
 * calls it should cover); kernels OR TL_DEVERR_* bits into it and never
 * clear it.  tl_get_device_error reads it once the work enqueued on `stream`
 * before this call has finished (it synchronises `stream`), stores the bits
 * in *bits (when bits is not NULL) and, with clear != 0, zeroes the word
 * afterwards on the same stream.  Returns TL_OK when no bit is set,
 * TL_ERR_DEVICE_TIMEOUT when TL_DEVERR_TIMEOUT is set, TL_ERR_DEVICE_BOUNDS
 * when any other bit is set, TL_ERR_INVALID_ARG for a NULL or misaligned
 * error_word and TL_ERR_CUDA when the copy or the synchronisation fails.
 */
tl_status tl_get_device_error(uint32_t* error_word, uint32_t* bits, int32_t clear, void* stream);

/* ---- Decode timeline (tracing; a build option) ---------------------------
 * A library built with -DTL_DECODE_TRACE=1 (the default build has none of
 * it; `python -m paged_kv_attention_cache_gb300.trace` builds one beside the
 * default library and runs it) records, in every bf16 and one-byte decode
 * call, %globaltimer stamps (ns, one clock for the whole GPU) of the call's
 * phases into a device array: slot TL_TRACE_* below.  A stamp taken once is
 * one thread's; TL_TRACE_ATTN_END and TL_TRACE_COMBINE_END keep the latest CTA,
 * TL_TRACE_COMBINE_START the earliest, across calls since the last reset.
 * tl_decode_trace_reset zeroes the stamps (the combine's start to all ones)
 * after synchronising the device; tl_decode_trace_read synchronises the
 * device and copies the first n (1..TL_TRACE_SLOTS) stamps to host memory at
 * `stamps`.  Trace one call at a time: reset, call, read.  Both return
 * TL_ERR_UNSUPPORTED from a library built without the option (nothing else
 * is done), TL_ERR_INVALID_ARG for a NULL `stamps` or n out of range, and
 * TL_ERR_CUDA when the synchronisation or the copy fails.
 */
#define TL_TRACE_PLAN_START 0       /* the plan kernel's first instruction (block 0) */
#define TL_TRACE_PLAN_PLACED 1      /* every piece placed (batches of up to 128 sequences) */
#define TL_TRACE_PLAN_END 2         /* every descriptor written */
#define TL_TRACE_ATTN_RELEASED 3    /* attention CTA 0 past its wait for the plan */
#define TL_TRACE_ATTN_FIRST_STAGE 4 /* its warp 0's first stage of keys arrived */
#define TL_TRACE_ATTN_END 5         /* the last attention CTA done */
#define TL_TRACE_COMBINE_START 6    /* the first combine CTA past its wait */
#define TL_TRACE_COMBINE_END 7      /* the last combine CTA done */
#define TL_TRACE_SLOTS 8
tl_status tl_decode_trace_reset(void);
tl_status tl_decode_trace_read(uint64_t* stamps, int32_t n);

/* ---- Prefill step trace (a build option) ---------------------------------
 * A library built with -DTL_PREFILL_TRACE=1 (absent from the default build;
 * `python -m paged_kv_attention_cache_gb300.trace --prefill` builds and runs
 * one) adds, in every prefill call, to one row of TL_PTRACE_FIELDS counters
 * per attention CTA (row = the CTA's index, up to 1024): the MMA-issuing
 * thread's clock64 cycles from its first item to its last, the 128-key steps
 * it issued (both query tiles' S and P.V over one key tile), its items, and
 * the cycles it waited for the softmax warps' P and for the producer's K and
 * V tiles; then, summed over the two softmax warpgroups (their first warps),
 * the cycles they waited for S and the cycles from S's arrival to their P's
 * release.  tl_prefill_trace_reset zeroes the rows after synchronising the
 * device; tl_prefill_trace_read synchronises the device and copies the first
 * n_ctas rows (1..1024) to host memory at `rows` (n_ctas x TL_PTRACE_FIELDS
 * uint64).  Both return TL_ERR_UNSUPPORTED from a library built without the
 * option (nothing else is done), TL_ERR_INVALID_ARG for a NULL `rows` or
 * n_ctas out of range, TL_ERR_CUDA when the synchronisation or copy fails.
 */
#define TL_PTRACE_CYCLES 0
#define TL_PTRACE_STEPS 1
#define TL_PTRACE_ITEMS 2
#define TL_PTRACE_WAIT_P 3
#define TL_PTRACE_WAIT_KV 4
#define TL_PTRACE_SM_WAIT_S 5
#define TL_PTRACE_SM_BUSY 6
#define TL_PTRACE_FIELDS 7
tl_status tl_prefill_trace_reset(void);
tl_status tl_prefill_trace_read(uint64_t* rows, int32_t n_ctas);

/* Name of a status, for messages (never NULL). */
const char* tl_status_string(tl_status status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t tl_version(void);

/*
 * KV_CACHE_WRITE ("How serving works in Tlaloc", sections 1-2): for every
 * token t in [0, n_tokens) with slot_mapping[t] != -1,
 *     k_cache row slot_mapping[t] = k_new[t],  v_cache row slot_mapping[t] = v_new[t]
 * byte for byte.  Slot -1 is padding and writes nothing.  The pools are
 * updated in place; no other byte of them changes.
 *   k_new, v_new   [n_tokens][H_kv][d] in `dtype`
 *   k_cache, v_cache  [num_pages][page_size][H_kv][d] in `dtype`, in place
 *   slot_mapping   [n_tokens] int64
 *   Two live tokens with the same slot: which one lands is unspecified.
 * Returns TL_ERR_INVALID_ARG for null pointers (n_tokens > 0), non-positive
 * sizes, H_kv*d*elem not a multiple of 16 bytes, or misaligned pointers.
 */
tl_status tl_kv_cache_write(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                            const int64_t* slot_mapping, int32_t n_tokens, int32_t num_pages,
                            int32_t page_size, int32_t h_kv, int32_t d, tl_dtype dtype,
                            uint32_t* error_word, void* stream);

/*
 * KV_CACHE_WRITE into fp8 pools ("How serving works in Tlaloc", the FP8 KV
 * cache paragraph of its quantisation section): the pools hold e4m3fn codes
 * (1 byte per element, no scale), the layout and the slot rule as above.
 * Each element of the new rows (k_new / v_new: [n_tokens][h_kv][d] of
 * src_dtype TL_F32 or TL_BF16) is clamped to +-448 and rounded to the
 * nearest code, ties to an even mantissa; NaN gives the code 0x7F.
 *   k_cache, v_cache  [num_pages][page_size][h_kv][d] uint8 codes, 8-byte
 *                     aligned; other arguments and errors as above
 *                     (h_kv * d a multiple of 16).
 */
tl_status tl_kv_cache_write_fp8(const void* k_new, const void* v_new, tl_dtype src_dtype,
                                void* k_cache, void* v_cache, const int64_t* slot_mapping,
                                int32_t n_tokens, int32_t num_pages, int32_t page_size,
                                int32_t h_kv, int32_t d, uint32_t* error_word, void* stream);

/*
 * KV_CACHE_WRITE into int8 pools.  "How serving works in Tlaloc" names int8
 * KV pools as a next step ("What would make it faster") without a format;
 * the format is read from the same page's "Int8 weights (opt-in)" paragraph
 * (one f32 scale per output channel, max |W| / 127, codes rounded half to
 * even), with a (token, KV head) row of d values as the channel.  For every
 * token t with slot_mapping[t] != -1 and every KV head g, the row x =
 * new[t][g][0..d) (src_dtype TL_F32 or TL_BF16, widened exactly) gets
 *     s = m / 127   (m the largest magnitude of the row's finite values)
 *     code_e = round-half-even(x_e / s), clamped to +-127
 * with both divisions in binary32.  A row whose s is 0 writes codes 0 and
 * scale 0; a non-finite value writes code 0 and sets TL_DEVERR_VALUE_RANGE.
 * Slot -1 writes nothing; no other byte of the pools changes.
 *   k_new, v_new       [n_tokens][h_kv][d] in src_dtype, 16-byte aligned
 *   k_codes, v_codes   [num_pages][page_size][h_kv][d] int8, in place
 *   k_scales, v_scales [num_pages][h_kv][page_size] float32, in place (the
 *                      scales of one page and head are contiguous)
 *   slot_mapping       [n_tokens] int64
 * Returns TL_ERR_INVALID_ARG for null pointers (n_tokens > 0), non-positive
 * sizes or misaligned pointers; TL_ERR_UNSUPPORTED for d > 1024 or another
 * src_dtype.
 */
tl_status tl_kv_cache_write_int8(const void* k_new, const void* v_new, tl_dtype src_dtype,
                                 int8_t* k_codes, int8_t* v_codes, float* k_scales,
                                 float* v_scales, const int64_t* slot_mapping, int32_t n_tokens,
                                 int32_t num_pages, int32_t page_size, int32_t h_kv, int32_t d,
                                 uint32_t* error_word, void* stream);

/*
 * Bytes of workspace tl_paged_attn_decode needs for these sizes (an upper
 * bound that holds for every content of context_lens).  Returns 0 when the
 * sizes are invalid.
 */
size_t tl_paged_attn_decode_workspace_size(int32_t B, int32_t h_q, int32_t h_kv, int32_t d);

/*
 * PAGED_ATTENTION, decode ("How serving works in Tlaloc", sections 1-3): one
 * query token per sequence.  Sequence b has causal length L = context_lens[b]
 * (its query sits at position L-1, its own K/V already written); with
 * p = L-1 and lo = (window > 0 ? max(0, p-window+1) : 0), for every query
 * head h (KV head g = h / (h_q/h_kv)):
 *     s_j = scale * <q[b][h], K_g(j)>,  j = lo..p,  K_g(j) found through
 *           page block_table[b][j / page_size], offset j % page_size
 *     out[b][h] = sum_j softmax(s)_j * V_g(j)
 * L <= 0 gives out[b][h] = 0.  Each sequence's keys are cut into pieces
 * attended independently (split-K) and merged with a log-sum-exp combine in a
 * fixed order; the result does not depend on where the pages are in the pool,
 * and repeats bit for bit.  The call enqueues three kernels on `stream` (a
 * plan, the attention kernel, the merge); the last two are programmatic
 * dependent launches of their predecessor within the call, and the call as a
 * whole keeps ordinary stream order with the work around it.
 *   q            [B][h_q][d] in `dtype`
 *   k_cache, v_cache  as above, in `dtype` (read only)
 *   block_table  [B][max_pages_per_seq] int32
 *   context_lens [B] int32
 *   out          [B][h_q][d] float32
 *   scale        multiplies the dot products (e.g. 1/sqrt(d))
 *   workspace    device scratch of at least
 *                tl_paged_attn_decode_workspace_size(B, h_q, h_kv, d) bytes,
 *                256-byte aligned; its contents need no initialisation and
 *                are garbage afterwards.  Calls that overlap in time must not
 *                share a workspace.
 * Supported: dtype TL_BF16 or TL_F32, or TL_FP8_E4M3 for e4m3 pools (q bf16,
 * d = 128; the codes widen exactly to fp16 for the tensor core, and q is
 * rounded to fp16: a finite |q| beyond 65504 sets TL_DEVERR_VALUE_RANGE),
 * d in {64, 128},
 * h_q % h_kv == 0 with
 * h_q/h_kv <= 16, page_size in [1, 256] (a multiple of 8 for TL_BF16, whose
 * pages move as TMA boxes of 8 or 16 rows), num_pages*page_size < 2^31.
 * Otherwise TL_ERR_UNSUPPORTED.
 */
tl_status tl_paged_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t max_pages_per_seq,
                               const int32_t* context_lens, float* out, int32_t B, int32_t h_q,
                               int32_t h_kv, int32_t d, int32_t num_pages, int32_t page_size,
                               int32_t window, float scale, tl_dtype dtype, void* workspace,
                               size_t workspace_bytes, uint32_t* error_word, void* stream);

/*
 * PAGED_ATTENTION decode over int8 pools (written by tl_kv_cache_write_int8):
 * tl_paged_attn_decode with every K/V element read as code x its row's
 * scale.  The scores are s_j = scale * k_scale(j) * <q, codes of K_g(j)>
 * (the codes widen exactly to fp16, q is rounded to fp16: a finite |q|
 * beyond 65504 sets TL_DEVERR_VALUE_RANGE), and each probability is
 * multiplied by its key's v_scale before the P.V product.
 *   q                  [B][h_q][d] bf16
 *   k_codes, v_codes, k_scales, v_scales  as tl_kv_cache_write_int8 writes
 *                      them (read only; the scales 16-byte aligned)
 *   the other arguments, the workspace (tl_paged_attn_decode_workspace_size)
 *   and the errors as tl_paged_attn_decode.
 * Supported: d = 128, h_q % h_kv == 0 with h_q/h_kv <= 16, page_size a
 * multiple of 16 in [16, 256] (a chunk of 16 keys' scales of one head is one
 * 64-byte copy), num_pages*page_size < 2^31.  Otherwise TL_ERR_UNSUPPORTED.
 */
tl_status tl_paged_attn_decode_int8(const void* q, const int8_t* k_codes, const int8_t* v_codes,
                                    const float* k_scales, const float* v_scales,
                                    const int32_t* block_table, int32_t max_pages_per_seq,
                                    const int32_t* context_lens, float* out, int32_t B,
                                    int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                                    int32_t page_size, int32_t window, float scale,
                                    void* workspace, size_t workspace_bytes,
                                    uint32_t* error_word, void* stream);

/*
 * tl_kv_cache_write_int8 of the n_new rows k_new / v_new ([n_new][h_kv][d],
 * new_dtype TL_BF16 or TL_F32) at slot_mapping [n_new] (int64, -1 = padding)
 * followed by tl_paged_attn_decode_int8, in one call (the write runs in the
 * decode's first launch, as in tl_paged_attn_decode_write): the result, the
 * pools (codes and scales) afterwards and the error bits are those of the two
 * calls.  Arguments and support as the two calls.
 */
tl_status tl_paged_attn_decode_write_int8(const void* q, const void* k_new, const void* v_new,
                                          tl_dtype new_dtype, const int64_t* slot_mapping,
                                          int32_t n_new, int8_t* k_codes, int8_t* v_codes,
                                          float* k_scales, float* v_scales,
                                          const int32_t* block_table, int32_t max_pages_per_seq,
                                          const int32_t* context_lens, float* out, int32_t B,
                                          int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                                          int32_t page_size, int32_t window, float scale,
                                          void* workspace, size_t workspace_bytes,
                                          uint32_t* error_word, void* stream);

/*
 * KV_CACHE_WRITE then PAGED_ATTENTION decode in one call ("How serving works
 * in Tlaloc", section 1: each step writes its tokens' K/V, then attends):
 * the result, the pools afterwards and the error bits are those of
 * tl_kv_cache_write (tl_kv_cache_write_fp8 for e4m3 pools) of the n_new rows
 * k_new / v_new [n_new][h_kv][d] at slot_mapping [n_new] (int64, -1 =
 * padding, never written) followed by tl_paged_attn_decode on the same
 * stream.  The rows are written by extra CTAs of the decode's first launch,
 * so the call enqueues three kernels instead of four.
 *   new_dtype    dtype of k_new / v_new: the pool's dtype for TL_BF16 and
 *                TL_F32 pools (a copy); TL_BF16 or TL_F32 for TL_FP8_E4M3
 *                pools (converted to e4m3 codes, nearest with ties to even,
 *                clamped to +-448, NaN to the NaN code)
 *   k_cache, v_cache  the pools, written in place, then read
 *   other arguments, workspace size and support as tl_paged_attn_decode.
 * Errors: as the two calls; a slot outside the pools sets
 * TL_DEVERR_SLOT_RANGE and that row is skipped.  Duplicate live slots are a
 * caller error (which row lands is unspecified).
 */
tl_status tl_paged_attn_decode_write(const void* q, const void* k_new, const void* v_new,
                                     tl_dtype new_dtype, const int64_t* slot_mapping,
                                     int32_t n_new, void* k_cache, void* v_cache,
                                     const int32_t* block_table, int32_t max_pages_per_seq,
                                     const int32_t* context_lens, float* out, int32_t B,
                                     int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                                     int32_t page_size, int32_t window, float scale,
                                     tl_dtype dtype, void* workspace, size_t workspace_bytes,
                                     uint32_t* error_word, void* stream);

/*
 * Decode without any device allocation, for callers that cannot allocate on
 * this path: a host framework that owns all device memory through its own
 * pool, or a latency-bound loop that cannot afford an allocator call.  There
 * is no counterpart in the paper; it is a deployment convenience.
 *
 * Same arguments, result and errors as tl_paged_attn_decode, without the
 * workspace: the scratch comes from a fixed array of
 * TL_DECODE_NOALLOC_SCRATCH_BYTES inside the library's device memory, which
 * every GPU that loads the library holds until the process exits.  The first
 * call on a device (with that device current) looks up the array's address;
 * make that first call before any stream capture.  Returns TL_ERR_WORKSPACE
 * when tl_paged_attn_decode_workspace_size(B, h_q, h_kv, d) exceeds the
 * array (for example B=64, h_q=32, h_kv=8, d=128 needs about 27 MB and fits).
 * All calls on a device share the array, which keeps the last call's
 * contents (nothing in it needs to start at zero); calls whose GPU work
 * overlaps (other streams or host threads) race on it and must be serialised.
 * The address is kept per device for the process's primary context: calls
 * from another context (cuCtxCreate) or after cudaDeviceReset would use a
 * stale address, so this entry point is for callers on the primary context
 * that do not reset the device while the library is loaded.
 */
#define TL_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)
tl_status tl_paged_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, int32_t max_pages_per_seq,
                                       const int32_t* context_lens, float* out, int32_t B,
                                       int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                                       int32_t page_size, int32_t window, float scale,
                                       tl_dtype dtype, uint32_t* error_word, void* stream);

/*
 * Bytes of workspace tl_paged_attn_prefill needs (0 for invalid sizes): the
 * kernel's work counter (256 bytes), the key-tile count and the schedule of
 * every query-tile pair (two int32 arrays of B * n_pairs entries, each
 * rounded up to 256 bytes; n_pairs = ceil(T / (2 * floor(128 / (h_q/h_kv))))),
 * each row's first key (B int32, rounded up to 256 bytes), a flag per 64 keys
 * of each row (B * ceil(max_pages_per_seq * page_size / 64) int32, rounded up
 * to 256 bytes), a flag per row (B int32, rounded up to 256 bytes), and an
 * fp16 copy of the V rows the call reads, [B][h_kv][n_keys][d] with n_keys =
 * max_pages_per_seq * page_size rounded up to a multiple of 128
 * (B * h_kv * n_keys * d * 2 bytes).  It grows with the table's width; a
 * workspace sized by tl_paged_attn_prefill_workspace_size_keys for the
 * call's rows instead does not.
 */
size_t tl_paged_attn_prefill_workspace_size(int32_t B, int32_t T, int32_t h_q, int32_t h_kv,
                                            int32_t d, int32_t max_pages_per_seq,
                                            int32_t page_size);

/*
 * Workspace bytes of a prefill call (tl_paged_attn_prefill, _prefill_int8,
 * _prefill_ring; dtype TL_BF16, TL_FP8_E4M3 or TL_INT8) whose rows each read
 * at most max_row_keys keys: from the first key the row's first live token
 * sees (window-clipped) to the row's last position.  The size does not
 * depend on the table's width.  A call takes the copies' size from the
 * workspace it is given (the table's positions when the workspace holds
 * them, otherwise as many whole 128-key tiles as fit, at least 384); a row
 * that reads more keys than that sets TL_DEVERR_CONTEXT_RANGE and its
 * outputs are undefined.  0 for invalid sizes.
 */
size_t tl_paged_attn_prefill_workspace_size_keys(int32_t B, int32_t T, int32_t h_q, int32_t h_kv,
                                                 int32_t d, int32_t max_row_keys,
                                                 tl_dtype dtype);

/* Workspace bytes of any prefill call (0 for invalid sizes): ring_pages 0 for
 * a full-history table (tl_paged_attn_prefill, tl_paged_attn_prefill_int8) or
 * > 0 for a ring (tl_paged_attn_prefill_ring); dtype TL_BF16, TL_FP8_E4M3 for
 * e4m3 pools, which add a bf16 copy of K as large as the V copy, or TL_INT8
 * for int8 pools, which add that copy and the copied keys' K scales, V
 * scales and reciprocal V scales (three f32 arrays of B * h_kv *
 * max_pages_per_seq * page_size, each rounded up to 256 bytes). */
size_t tl_paged_attn_prefill_workspace_size_ex(int32_t B, int32_t T, int32_t h_q, int32_t h_kv,
                                               int32_t d, int32_t max_pages_per_seq,
                                               int32_t page_size, int32_t ring_pages,
                                               tl_dtype dtype);

/*
 * PAGED_ATTENTION, batched prefill ("How serving works in Tlaloc", sections
 * 1-2, "Blockwise attention"): B rows of T tokens.  Token (b,t) with position
 * p = positions[b][t] >= 0 attends exactly like a decode query of causal
 * length p+1 (and the same window rule) over its own row's pages; p < 0 marks
 * padding, whose output is 0.  The keys are folded tile by tile (128 keys,
 * a finer fold than the pages' 2,048-key blocks; the result is the same up to
 * rounding) with an online softmax; no score tensor wider than one tile
 * exists.  A row's result does not depend on the other rows (batched equals
 * solo, bit for bit).
 *   q            [B][T][h_q][d] bf16
 *   positions    [B][T] int32, -1 = padding
 *   out          [B][T][h_q][d] float32
 *   workspace    device scratch of tl_paged_attn_prefill_workspace_size(B, T,
 *                h_q, h_kv, d, max_pages_per_seq, page_size) bytes (copies as
 *                wide as the table), or of tl_paged_attn_prefill_workspace_size_keys
 *                (copies as wide as the call's rows need), 256-byte aligned;
 *                TL_ERR_WORKSPACE when it is missing, misaligned or holds less
 *                than 384 keys per row.  It receives the call's fp16 copy of V
 *                and work counters, so calls that may overlap on the GPU must
 *                not share one.
 *   other arguments as for decode.
 * Supported: dtype TL_BF16, or TL_FP8_E4M3 for e4m3 pools (q stays bf16; the
 * codes widen exactly: K to a bf16 copy, V to an fp16 copy in the workspace,
 * sized by tl_paged_attn_prefill_workspace_size_ex), d = 128,
 * h_q % h_kv == 0 with h_q/h_kv <= 128, page_size a power of two in
 * [8, 128].  Otherwise TL_ERR_UNSUPPORTED.
 * scale must be positive and finite (TL_ERR_INVALID_ARG otherwise).
 * Arithmetic: Q.K^T with bf16 operands and f32 accumulation; P.V with V
 * converted bf16 -> fp16 (exact for |v| in [2^-14, 65504]; smaller
 * magnitudes land on fp16's subnormal grid, a change below 2^-25) and f32
 * accumulation.  For a row whose V (in the keys the call reads) holds no
 * value of magnitude above 8, P is rounded to fp16 and the softmax sum is
 * taken over the same rounded P, so each output is a convex combination of
 * V rows with weights within 2^-11 relative of the exact ones; any other row
 * takes P as the sum of two fp16 parts (a second P.V product, about 22
 * significant bits), so a large |v| does not magnify the rounding.  A finite
 * V entry beyond +-65504 in a key range the call reads sets
 * TL_DEVERR_VALUE_RANGE and leaves the outputs undefined.
 */
tl_status tl_paged_attn_prefill(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int32_t max_pages_per_seq,
                                const int32_t* positions, float* out, int32_t B, int32_t T,
                                int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                                int32_t page_size, int32_t window, float scale, tl_dtype dtype,
                                void* workspace, size_t workspace_bytes, uint32_t* error_word,
                                void* stream);

/*
 * PAGED_ATTENTION, batched prefill over int8 pools (written by
 * tl_kv_cache_write_int8): tl_paged_attn_prefill with every K/V element read
 * as code x its row's scale.  The scores are s_j = scale * k_scale(j) *
 * <q, codes of K_g(j)> (Q.K^T on the tensor core with bf16 q and the codes
 * widened exactly to bf16, f32 accumulation, then the K scale in f32).  V is
 * read in 64-key tiles: a tile whose values code x v_scale all lie within
 * +-8 with a root mean square up to 1.25 is used as fp16(code x v_scale)
 * (one rounding, 2^-12 relative), and a row made only of such tiles takes
 * P.V as tl_paged_attn_prefill does (P rounded once to fp16, the softmax
 * sum over the same rounded values); any other tile keeps its codes (exact
 * in fp16) and its row takes each p_j x v_scale split into two fp16 parts,
 * with the sum over the unscaled p_j.
 *   q                  [B][T][h_q][d] bf16;  positions [B][T] int32 (-1 = pad)
 *   k_codes, v_codes, k_scales, v_scales  as tl_kv_cache_write_int8 writes
 *                      them (read only; codes 16-byte aligned)
 *   out                [B][T][h_q][d] float32
 *   workspace          at least tl_paged_attn_prefill_workspace_size_ex(B, T,
 *                      h_q, h_kv, d, max_pages_per_seq, page_size, 0, TL_INT8)
 *                      bytes, 256-byte aligned
 *   the other arguments, support and errors as tl_paged_attn_prefill.
 */
tl_status tl_paged_attn_prefill_int8(const void* q, const int8_t* k_codes, const int8_t* v_codes,
                                     const float* k_scales, const float* v_scales,
                                     const int32_t* block_table, int32_t max_pages_per_seq,
                                     const int32_t* positions, float* out, int32_t B, int32_t T,
                                     int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                                     int32_t page_size, int32_t window, float scale,
                                     void* workspace, size_t workspace_bytes,
                                     uint32_t* error_word, void* stream);

/*
 * Sliding-window attention over a ring ("How serving works in Tlaloc",
 * section 2, the bullet on sliding layers whose table is a ring; section 3,
 * the windowed KV pool).  Each sequence holds a ring of ring_pages pages:
 * logical block k lives on the page block_table[b][k % ring_pages], so
 * position p overwrites position p - ring_pages * page_size, which has left
 * the window; the caller's slot_mapping for tl_kv_cache_write follows the
 * same rule.  Only the first ring_pages entries of each table row are read,
 * and positions / context lengths are not bounded by the table's width.
 * Keys are visited in position order, so the result is bit-identical to the
 * same call over a full-history table.
 * The ring must hold the window: 0 < ring_pages <= max_pages_per_seq,
 * window > 0 and ring_pages * page_size >= window; otherwise
 * TL_ERR_INVALID_ARG.  For prefill, a call of n tokens starting at position
 * p0 needs min(p0, window - 1) + n positions of ring; a row whose call spans
 * more sets TL_DEVERR_CONTEXT_RANGE (its outputs are undefined).
 * All other arguments, layouts and errors as for tl_paged_attn_decode /
 * tl_paged_attn_prefill.
 */
tl_status tl_paged_attn_decode_ring(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_table, int32_t max_pages_per_seq,
                                    const int32_t* context_lens, float* out, int32_t B,
                                    int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                                    int32_t page_size, int32_t window, int32_t ring_pages,
                                    float scale, tl_dtype dtype, void* workspace,
                                    size_t workspace_bytes, uint32_t* error_word, void* stream);

/*
 * Multi-token decode: q_len query tokens at the end of each sequence, at
 * positions L - q_len .. L - 1 with L = context_lens[b] (their K/V written
 * first), each attending with its own causal length (and window) over the
 * sequence's pages.  This is the verify step of speculative decoding (the
 * DGX Spark optimization-ladder page, rung D6: draft blocks of 6 to 8 tokens
 * checked by a multi-token attention kernel) and a short chunk of chunked
 * prefill ("How serving works in Tlaloc", section 4); it gives the same
 * results as tl_paged_attn_prefill on the same tokens, within the tolerance,
 * and for q_len = 1 is tl_paged_attn_decode.  K and V of each sequence are
 * read once for all its tokens, as in decode.
 *   q    [B][q_len][h_q][d] bf16;  out [B][q_len][h_q][d] float32.
 * Supported: bf16 pools with d in {64, 128}, or TL_FP8_E4M3 pools with
 * d = 128 (bf16 q, as for tl_paged_attn_decode), q_len * (h_q / h_kv) <= 16
 * (the tokens' heads of one KV head form the MMA rows); otherwise
 * TL_ERR_UNSUPPORTED.  tl_paged_attn_decode_multi_int8 is the same over int8
 * pools (arguments as tl_paged_attn_decode_int8, plus q_len).
 * Workspace: tl_paged_attn_decode_multi_workspace_size(B, q_len, h_q, h_kv, d).
 * Other arguments and errors as for tl_paged_attn_decode.
 */
size_t tl_paged_attn_decode_multi_workspace_size(int32_t B, int32_t q_len, int32_t h_q,
                                                 int32_t h_kv, int32_t d);
tl_status tl_paged_attn_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, int32_t max_pages_per_seq,
                                     const int32_t* context_lens, float* out, int32_t B,
                                     int32_t q_len, int32_t h_q, int32_t h_kv, int32_t d,
                                     int32_t num_pages, int32_t page_size, int32_t window,
                                     float scale, tl_dtype dtype, void* workspace,
                                     size_t workspace_bytes, uint32_t* error_word, void* stream);

/* Workspace bytes of tl_paged_attn_prefill_ring (0 for invalid sizes or
 * ring_pages <= 0): as for tl_paged_attn_prefill, but the fp16 V copy holds
 * align_up(ring_pages * page_size, 128) + 256 keys per row and KV head. */
size_t tl_paged_attn_prefill_ring_workspace_size(int32_t B, int32_t T, int32_t h_q,
                                                 int32_t h_kv, int32_t d,
                                                 int32_t max_pages_per_seq, int32_t page_size,
                                                 int32_t ring_pages);

tl_status tl_paged_attn_prefill_ring(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, int32_t max_pages_per_seq,
                                     const int32_t* positions, float* out, int32_t B, int32_t T,
                                     int32_t h_q, int32_t h_kv, int32_t d, int32_t num_pages,
                                     int32_t page_size, int32_t window, int32_t ring_pages,
                                     float scale, tl_dtype dtype, void* workspace,
                                     size_t workspace_bytes, uint32_t* error_word, void* stream);

/*
 * Sliding-window decode and prefill over rings of int8 pools: the ring rule
 * of tl_paged_attn_decode_ring / tl_paged_attn_prefill_ring ("How serving
 * works in Tlaloc", section 3, the windowed KV pool) over the int8 pools and
 * arithmetic of tl_paged_attn_decode_int8 / tl_paged_attn_prefill_int8 (the
 * pools as tl_kv_cache_write_int8 writes them, its scales per slot and KV
 * head following their slots through the ring).  Arguments, refusals and
 * errors as there; the prefill's workspace is
 * tl_paged_attn_prefill_workspace_size_ex(B, T, h_q, h_kv, d,
 * max_pages_per_seq, page_size, ring_pages, TL_INT8) bytes, the decode's
 * tl_paged_attn_decode_workspace_size(B, h_q, h_kv, d).
 */
tl_status tl_paged_attn_decode_ring_int8(const void* q, const int8_t* k_codes,
                                         const int8_t* v_codes, const float* k_scales,
                                         const float* v_scales, const int32_t* block_table,
                                         int32_t max_pages_per_seq, const int32_t* context_lens,
                                         float* out, int32_t B, int32_t h_q, int32_t h_kv,
                                         int32_t d, int32_t num_pages, int32_t page_size,
                                         int32_t window, int32_t ring_pages, float scale,
                                         void* workspace, size_t workspace_bytes,
                                         uint32_t* error_word, void* stream);
tl_status tl_paged_attn_prefill_ring_int8(const void* q, const int8_t* k_codes,
                                          const int8_t* v_codes, const float* k_scales,
                                          const float* v_scales, const int32_t* block_table,
                                          int32_t max_pages_per_seq, const int32_t* positions,
                                          float* out, int32_t B, int32_t T, int32_t h_q,
                                          int32_t h_kv, int32_t d, int32_t num_pages,
                                          int32_t page_size, int32_t window, int32_t ring_pages,
                                          float scale, void* workspace, size_t workspace_bytes,
                                          uint32_t* error_word, void* stream);

/*
 * tl_paged_attn_decode_write over rings: the step's rows written at their
 * ring slots (the caller's slot_mapping follows the ring rule: position p of
 * sequence b at page block_table[b][(p / page_size) % ring_pages], offset
 * p % page_size), then tl_paged_attn_decode_ring, in one call.  Arguments,
 * refusals and errors as those two calls.
 */
tl_status tl_paged_attn_decode_write_ring(const void* q, const void* k_new, const void* v_new,
                                          tl_dtype new_dtype, const int64_t* slot_mapping,
                                          int32_t n_new, void* k_cache, void* v_cache,
                                          const int32_t* block_table, int32_t max_pages_per_seq,
                                          const int32_t* context_lens, float* out, int32_t B,
                                          int32_t h_q, int32_t h_kv, int32_t d,
                                          int32_t num_pages, int32_t page_size, int32_t window,
                                          int32_t ring_pages, float scale, tl_dtype dtype,
                                          void* workspace, size_t workspace_bytes,
                                          uint32_t* error_word, void* stream);

tl_status tl_paged_attn_decode_multi_int8(const void* q, const int8_t* k_codes,
                                          const int8_t* v_codes, const float* k_scales,
                                          const float* v_scales, const int32_t* block_table,
                                          int32_t max_pages_per_seq, const int32_t* context_lens,
                                          float* out, int32_t B, int32_t q_len, int32_t h_q,
                                          int32_t h_kv, int32_t d, int32_t num_pages,
                                          int32_t page_size, int32_t window, float scale,
                                          void* workspace, size_t workspace_bytes,
                                          uint32_t* error_word, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TL_PAGED_ATTN_H */
