// Library-wide entry points of the C ABI: status names, version, device info.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace tl {

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType type, const void* base,
                              int rank, const uint64_t* dims, const uint64_t* strides,
                              const uint32_t* box, bool swizzle128) {
  auto enc = tensor_map_encoder();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides[i];
  }
  const CUresult r =
      enc(map, type, (cuuint32_t)rank, const_cast<void*>(base), gdim,
          gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_bf16_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides, const uint32_t* box, bool swizzle128) {
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box,
                           swizzle128);
}

bool encode_u8_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box, bool swizzle128) {
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rank, dims, strides, box,
                           swizzle128);
}

bool encode_f32_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides, const uint32_t* box, bool swizzle128) {
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, rank, dims, strides, box,
                           swizzle128);
}

int num_sms() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace tl

extern "C" const char* tl_status_string(tl_status status) {
  switch (status) {
    case TL_OK: return "TL_OK";
    case TL_ERR_INVALID_ARG: return "TL_ERR_INVALID_ARG: a null pointer, bad size or misaligned pointer";
    case TL_ERR_UNSUPPORTED: return "TL_ERR_UNSUPPORTED: valid arguments, but not a shape or dtype the library runs";
    case TL_ERR_CUDA: return "TL_ERR_CUDA: a CUDA call or kernel launch failed";
    case TL_ERR_DEVICE_BOUNDS: return "TL_ERR_DEVICE_BOUNDS: a device-side check found a value out of range";
    case TL_ERR_WORKSPACE: return "TL_ERR_WORKSPACE: workspace missing or too small";
    case TL_ERR_DEVICE_TIMEOUT: return "TL_ERR_DEVICE_TIMEOUT: an in-kernel wait gave up (outputs invalid)";
  }
  return "unknown tl_status";
}

extern "C" int32_t tl_version(void) { return 1 * 10000 + 1 * 100 + 0; }

// The error word is read after the stream's earlier work (a copy ordered on
// the stream, then a synchronisation of the stream), and cleared after the
// read on the same stream when asked.
extern "C" tl_status tl_get_device_error(uint32_t* error_word, uint32_t* bits, int32_t clear,
                                         void* stream) {
  if (!error_word || (reinterpret_cast<uintptr_t>(error_word) & 3u)) return TL_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, error_word, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return TL_ERR_CUDA;
  if (clear && cudaMemsetAsync(error_word, 0, sizeof(uint32_t), st) != cudaSuccess)
    return TL_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TL_ERR_CUDA;
  if (bits) *bits = word;
  if (word & TL_DEVERR_TIMEOUT) return TL_ERR_DEVICE_TIMEOUT;
  return word ? TL_ERR_DEVICE_BOUNDS : TL_OK;
}
