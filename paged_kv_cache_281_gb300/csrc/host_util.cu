// Host helpers: tensor-map encoding through the driver entry point, cached
// device properties, CUDA error mapping and the device status block.
#include <cudaTypedefs.h>

#include <mutex>

#include "host_util.h"

namespace pkv {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_info_once[kMaxDevices];
}  // namespace

// cuTensorMapEncodeTiled, looked up once through the runtime (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

int cuda_fail(cudaError_t err, const char* what) {
  return fail(PKV_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

int current_device_info(const DeviceInfo** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_EINVAL, "device ordinal %d unsupported", dev);
  std::call_once(g_info_once[dev], [dev]() {
    DeviceInfo& d = g_info[dev];
    d.ok = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) ==
               cudaSuccess &&
           cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) ==
               cudaSuccess &&
           cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) ==
               cudaSuccess &&
           cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                  dev) == cudaSuccess;
  });
  if (!g_info[dev].ok) return fail(PKV_ECUDA, "could not query device %d", dev);
  if (g_info[dev].cc_major != 10 || g_info[dev].cc_minor != 3)
    return fail(PKV_ECUDA, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                g_info[dev].cc_major, g_info[dev].cc_minor);
  *out = &g_info[dev];
  return PKV_OK;
}

int encode_tile_map_2d(CUtensorMap* map, const void* base, uint64_t inner_elems,
                       uint64_t outer_rows, uint64_t row_stride_bytes, uint32_t box_inner,
                       uint32_t box_outer) {
  if (!encode_fn()) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[2] = {inner_elems, outer_rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PKV_ECUDA, "cuTensorMapEncodeTiled failed (%d) for %llu x %llu rows, box %u x %u",
                (int)r, (unsigned long long)inner_elems, (unsigned long long)outer_rows,
                box_inner, box_outer);
  return PKV_OK;
}

int encode_tile_map_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                       const uint64_t strides_bytes[2], const uint32_t box[3]) {
  if (!encode_fn()) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t s[2] = {strides_bytes[0], strides_bytes[1]};
  cuuint32_t b[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), d, s,
                        b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled (3d) failed (%d)", (int)r);
  return PKV_OK;
}

int encode_row_group_map(CUtensorMap* map, const void* base, uint64_t D, uint64_t rows,
                         uint32_t box_rows) {
  if (!encode_fn()) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled is not available");
  // dimensions, innermost first: 64 elements of a half row, 8 rows of a
  // group, the D / 64 halves of a row, the groups
  cuuint64_t d[4] = {64, 8, D / 64, rows / 8};
  cuuint64_t s[3] = {D * 2, 128, 8 * D * 2};
  cuuint32_t b[4] = {64, 8, (cuuint32_t)(D / 64), box_rows / 8};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), d, s,
                        b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PKV_ECUDA, "cuTensorMapEncodeTiled (row groups) failed (%d)", (int)r);
  return PKV_OK;
}

int encode_byte_rows_map(CUtensorMap* map, const void* base, uint64_t row_bytes,
                         uint64_t rows, uint32_t box_rows, bool swizzle128) {
  if (!encode_fn()) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)row_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PKV_ECUDA, "cuTensorMapEncodeTiled (bytes) failed (%d) for %llu rows of %llu",
                (int)r, (unsigned long long)rows, (unsigned long long)row_bytes);
  return PKV_OK;
}

int check_launch(const char* what) {
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, what);
  return PKV_OK;
}

}  // namespace pkv

using pkv::fail;

extern "C" int pkv_status_reset(int32_t* dev_status, void* stream) {
  PKV_REQUIRE(dev_status, "pkv_status_reset: dev_status is NULL");
  cudaError_t err =
      cudaMemsetAsync(dev_status, 0, 4 * sizeof(int32_t), static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return pkv::cuda_fail(err, "pkv_status_reset");
  return pkv::ok();
}

extern "C" int pkv_check_status(const int32_t* dev_status, void* stream) {
  PKV_REQUIRE(dev_status, "pkv_check_status: dev_status is NULL");
  int32_t h[4] = {0, 0, 0, 0};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(h, dev_status, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (err == cudaSuccess) err = cudaStreamSynchronize(st);
  if (err != cudaSuccess) return pkv::cuda_fail(err, "pkv_check_status");
  if (h[0] == 0) return pkv::ok();
  static const char* names[] = {"?", "kv_append", "block_copy", "decode_plan", "decode",
                                "decode_combine", "prefill"};
  const char* kname = (h[2] >= 1 && h[2] <= 6) ? names[h[2]] : "?";
  if (h[0] == PKV_ETIMEOUT)
    return fail(PKV_ETIMEOUT, "%s: a pipeline wait expired (site %d, %d events)", kname, h[1],
                h[3]);
  return fail(h[0] == PKV_EDEVICE ? PKV_EDEVICE : h[0],
              "%s: device range check fired (value %d, %d events)", kname, h[1], h[3]);
}
