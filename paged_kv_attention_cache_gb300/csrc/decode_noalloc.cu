// tl_paged_attn_decode_noalloc: paged decode for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc on the path that runs attention: a host
// framework that owns all device memory through its own pool (a stray
// allocation breaks its accounting or fragments its arena), or a latency-bound
// serving loop that cannot pay for an allocator call and the synchronisation
// it may bring.  For them this entry point takes the decode's scratch from a
// fixed array in the library's own device memory instead of a caller buffer.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its TL_DECODE_NOALLOC_SCRATCH_BYTES until the process exits.
// Its device address is looked up once per device, on the first call made
// while that device is current; later calls reuse it.  The address belongs to
// the device's primary context: a caller that resets the device, or calls
// from a context of its own, must not use this entry point.
//
// All calls on a device share the one array and leave the last call's
// contents in it.  Nothing in it needs to start at zero: the decode's plan
// kernel writes every field (split offsets, descriptors, the work counter)
// that the later kernels read.  Two calls whose work overlaps on the GPU
// (other streams, or other host threads) race on the array; serialise them.
#include <mutex>

#include "common.cuh"

namespace tl {

static __device__ __align__(256) unsigned char g_decode_scratch[TL_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
}  // namespace

// The scratch array's device address on the current device (set up on the
// first call for that device).  Null on failure.
static void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();  // leave no sticky error behind for the caller
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace tl

extern "C" tl_status tl_paged_attn_decode_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* context_lens, float* out, int32_t B, int32_t h_q,
    int32_t h_kv, int32_t d, int32_t num_pages, int32_t page_size, int32_t window, float scale,
    tl_dtype dtype, uint32_t* error_word, void* stream) {
  const size_t need = tl_paged_attn_decode_workspace_size(B, h_q, h_kv, d);
  if (need == 0) return TL_ERR_INVALID_ARG;
  if (need > (size_t)TL_DECODE_NOALLOC_SCRATCH_BYTES) return TL_ERR_WORKSPACE;
  void* scratch = tl::scratch_on_current_device();
  if (!scratch) return TL_ERR_CUDA;
  return tl_paged_attn_decode(q, k_cache, v_cache, block_table, max_pages_per_seq, context_lens,
                              out, B, h_q, h_kv, d, num_pages, page_size, window, scale, dtype,
                              scratch, (size_t)TL_DECODE_NOALLOC_SCRATCH_BYTES, error_word,
                              stream);
}
