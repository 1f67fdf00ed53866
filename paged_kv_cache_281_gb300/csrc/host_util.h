// Host-side CUDA helpers used by the launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace pkv {

struct DeviceInfo {
  bool ok = false;
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  int max_smem_optin = 0;
};

// Properties of the current device, queried once per device. Fails unless the
// device is sm_103 (the only architecture the kernels are compiled for).
int current_device_info(const DeviceInfo** out);

int cuda_fail(cudaError_t err, const char* what);
int check_launch(const char* what);

// Row-major bf16 matrix of `outer_rows` rows, `inner_elems` elements each, rows
// `row_stride_bytes` apart; tiles of box_outer rows x box_inner elements,
// 128-byte swizzled in shared memory.
int encode_tile_map_2d(CUtensorMap* map, const void* base, uint64_t inner_elems,
                       uint64_t outer_rows, uint64_t row_stride_bytes, uint32_t box_inner,
                       uint32_t box_outer);

int encode_tile_map_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                       const uint64_t strides_bytes[2], const uint32_t box[3]);

// A bf16 pool of `rows` rows of D elements (D = 64 or 128, rows a multiple
// of 8) seen as 8-row groups: one box of `box_rows` rows (a multiple of 8)
// lands in shared memory as [8-row group][64-column half][8 rows x 128 B],
// 128-byte swizzled. The box is addressed by (0, 0, 0, first row / 8).
int encode_row_group_map(CUtensorMap* map, const void* base, uint64_t D, uint64_t rows,
                         uint32_t box_rows);

// `rows` rows of `row_bytes` bytes (a multiple of 16, at most 128 when
// swizzled), tiles of box_rows whole rows, 128-byte swizzled or plain.
int encode_byte_rows_map(CUtensorMap* map, const void* base, uint64_t row_bytes,
                         uint64_t rows, uint32_t box_rows, bool swizzle128);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pkv
