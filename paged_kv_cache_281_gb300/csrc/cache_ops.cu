// kv_append and block_copy: the two bit-exact cache writers.
//
// kv_append ("Batching, Scheduling, and Paging", section PagedAttention): each
// new token's key and value rows go to the slot its block table assigned.
// block_copy (same page, section Block sharing): copy-on-write duplicates a
// whole physical block before a divergent write lands in it.
//
// Both are pure data movement, bound by HBM bandwidth (or by launch latency
// at decode sizes). Every thread moves 16-byte vectors; one (token, head) row
// of D bf16 is D/8 consecutive vectors, so a warp touches whole 128-byte lines
// on both the read and the write side.
#include "device.cuh"
#include "host_util.h"

namespace pkv {

namespace {

struct AppendArgs {
  const uint4* k_new;
  const uint4* v_new;
  const int32_t* slot_mapping;
  uint4* k_cache;
  uint4* v_cache;
  int64_t num_slots;      // num_blocks * block_size
  int32_t T;
  int32_t Hkv;
  int32_t vec_per_row;    // D / 8
  int32_t block_size;
  int32_t* status;
};

// One thread per 16-byte vector of the new rows; grid-stride over T*Hkv*D/8.
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
  // a plan launched after this kernel may start launching; it waits for this
  // kernel's writes before it reads anything
  grid_dep_launch();
  const int64_t vec_per_tok = (int64_t)a.Hkv * a.vec_per_row;
  const int64_t total = (int64_t)a.T * vec_per_tok;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t t = (int32_t)(i / vec_per_tok);
    const int64_t rem = i - (int64_t)t * vec_per_tok;
    const int32_t h = (int32_t)(rem / a.vec_per_row);
    const int32_t c = (int32_t)(rem - (int64_t)h * a.vec_per_row);
    const int32_t slot = __ldg(a.slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= a.num_slots) {
      if (h == 0 && c == 0) record_status(a.status, PKV_EDEVICE, slot, kKernelAppend);
      continue;
    }
    const int32_t blk = slot / a.block_size;
    const int32_t off = slot - blk * a.block_size;
    const int64_t dst = (((int64_t)blk * a.Hkv + h) * a.block_size + off) * a.vec_per_row + c;
    a.k_cache[dst] = __ldg(a.k_new + i);
    a.v_cache[dst] = __ldg(a.v_new + i);
  }
}

struct CopyArgs {
  uint4* k_cache;
  uint4* v_cache;
  const int32_t* pairs;
  int32_t n;
  int32_t num_blocks;
  int64_t vec_per_block;  // Hkv * B * D / 8
  int32_t* status;
};

// One CTA per (pair, pool): blockIdx.x picks the pair, blockIdx.y the pool
// (0 keys, 1 values). Each thread moves up to eight 16-byte vectors per pass,
// all loads issued before the stores, so a CTA keeps a whole 32 KB block
// (8 heads, B = 16, D = 128) in flight.
__global__ void __launch_bounds__(256) block_copy_kernel(const CopyArgs a) {
  const int32_t p = blockIdx.x;
  const int32_t src = __ldg(a.pairs + 2 * p);
  const int32_t dst = __ldg(a.pairs + 2 * p + 1);
  if (src < 0 || src >= a.num_blocks || dst < 0 || dst >= a.num_blocks) {
    if (blockIdx.y == 0 && threadIdx.x == 0)
      record_status(a.status, PKV_EDEVICE, (src < 0 || src >= a.num_blocks) ? src : dst,
                    kKernelBlockCopy);
    return;
  }
  uint4* pool = blockIdx.y == 0 ? a.k_cache : a.v_cache;
  const uint4* s = pool + (int64_t)src * a.vec_per_block;
  uint4* d = pool + (int64_t)dst * a.vec_per_block;
  constexpr int kUnroll = 8;
  for (int64_t i0 = 0; i0 < a.vec_per_block; i0 += kUnroll * 256) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * 256 + threadIdx.x;
      if (i < a.vec_per_block) v[u] = __ldg(s + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * 256 + threadIdx.x;
      if (i < a.vec_per_block) d[i] = v[u];
    }
  }
}

struct SwapArgs {
  uint4* k_cache;
  uint4* v_cache;
  const int32_t* blocks;
  uint4* k_buf;
  uint4* v_buf;
  int32_t n;
  int32_t num_blocks;
  int64_t vec_per_block;
  int32_t to_buffer;  // 1: pool -> buffer (swap-out), 0: buffer -> pool (swap-in)
  int32_t* status;
};

// blockIdx.y picks the listed block, blockIdx.z the pool (0 keys, 1 values);
// blockIdx.x strides over the block's vectors. The buffer may be pinned host
// memory reached over the CPU-GPU link.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const SwapArgs a) {
  const int32_t i = blockIdx.y;
  const int32_t blk = __ldg(a.blocks + i);
  if (blk < 0 || blk >= a.num_blocks) {
    if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0)
      record_status(a.status, PKV_EDEVICE, blk, kKernelBlockCopy);
    return;
  }
  uint4* pool = (blockIdx.z == 0 ? a.k_cache : a.v_cache) + (int64_t)blk * a.vec_per_block;
  uint4* buf = (blockIdx.z == 0 ? a.k_buf : a.v_buf) + (int64_t)i * a.vec_per_block;
  const uint4* src = a.to_buffer ? pool : buf;
  uint4* dst = a.to_buffer ? buf : pool;
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < a.vec_per_block;
       j += (int64_t)gridDim.x * blockDim.x)
    dst[j] = src[j];
}

// ---------------------------------------------------------------------------
// kv_append into FP8 (e4m3) pages. Per (token, head, tensor) row:
// the row's largest magnitude amax sets scale = amax / 448 and the codes
// e4m3(x * (448 / amax)) (fp32 quotients and product, round to nearest even,
// saturating); a row of zeros gets scale 0 and zero codes. Codes land in
// [N][Hkv][B][D] bytes, the scale in [N][Hkv][B] floats.
struct AppendFp8Args {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int32_t* slot_mapping;
  uint8_t* k8;
  uint8_t* v8;
  float* ks;
  float* vs;
  int64_t num_slots;
  int32_t T;
  int32_t Hkv;
  int32_t D;
  int32_t block_size;
  int32_t* status;
};

__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b16 c;\n\tcvt.rn.satfinite.e4m3x2.f32 c, %1, %2;\n\tcvt.u32.u16 %0, c;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Four lanes per row: each lane holds D / 4 consecutive elements (two or
// four 16-byte loads in flight), the row's amax is a reduction over its four
// lanes, and each lane stores its D / 4 codes in 16-byte pieces. A warp
// covers eight rows per pass.
template <int D>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(const AppendFp8Args a) {
  grid_dep_launch();  // as in kv_append_kernel
  constexpr int E = D / 4;    // elements per lane: 32 (D=128) or 16 (D=64)
  constexpr int V = E / 8;    // 16-byte input vectors per lane
  const int sub = threadIdx.x & 3;
  const int64_t rows = (int64_t)a.T * a.Hkv * 2;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 2; w < rows;
       w += ((int64_t)gridDim.x * blockDim.x) >> 2) {
    const int which = (int)(w & 1);           // 0 keys, 1 values
    const int64_t th = w >> 1;
    const int32_t t = (int32_t)(th / a.Hkv);
    const int32_t h = (int32_t)(th - (int64_t)t * a.Hkv);
    const int32_t slot = __ldg(a.slot_mapping + t);
    // the four lanes of a row share t, h and slot: every branch below is
    // uniform across the row's lanes, so the row's shuffles stay converged
    const bool skip = slot < 0 || slot >= a.num_slots;
    if (slot >= a.num_slots && h == 0 && which == 0 && sub == 0)
      record_status(a.status, PKV_EDEVICE, slot, kKernelAppend);
    const unsigned group = 0xfu << (threadIdx.x & 28);
    if (skip) continue;
    const uint4* src = reinterpret_cast<const uint4*>(
        (which ? a.v_new : a.k_new) + ((int64_t)t * a.Hkv + h) * D + sub * E);
    uint4 u[V];
#pragma unroll
    for (int k = 0; k < V; ++k) u[k] = __ldg(src + k);
    float x[E];
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const uint32_t wv[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[8 * k + 2 * e] = bf16_lo_to_f32(wv[e]);
        x[8 * k + 2 * e + 1] = bf16_hi_to_f32(wv[e]);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int off = 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(group, amax, off));
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
    const int32_t blk = slot / a.block_size;
    const int32_t off = slot - blk * a.block_size;
    const int64_t row = ((int64_t)blk * a.Hkv + h) * a.block_size + off;
    uint32_t c[E / 4];
#pragma unroll
    for (int k = 0; k < E / 4; ++k) {
      const uint32_t c01 =
          e4m3x2_from_f32(__fmul_rn(x[4 * k], inv), __fmul_rn(x[4 * k + 1], inv));
      const uint32_t c23 =
          e4m3x2_from_f32(__fmul_rn(x[4 * k + 2], inv), __fmul_rn(x[4 * k + 3], inv));
      c[k] = c01 | (c23 << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>((which ? a.v8 : a.k8) + row * D + sub * E);
#pragma unroll
    for (int k = 0; k < E / 16; ++k) dst[k] = make_uint4(c[4 * k], c[4 * k + 1], c[4 * k + 2], c[4 * k + 3]);
    if (sub == 0) (which ? a.vs : a.ks)[row] = __fdiv_rn(amax, 448.f);
  }
}

// Device-usable address of a buffer, or an error for memory the GPU cannot
// reach (pageable host memory).
int device_address(void* p, void** out, const char* who) {
  cudaPointerAttributes attr;
  cudaError_t err = cudaPointerGetAttributes(&attr, p);
  if (err != cudaSuccess) return cuda_fail(err, who);
  if (attr.type == cudaMemoryTypeUnregistered || attr.devicePointer == nullptr)
    return fail(PKV_EINVAL,
                "%s: buffer %p is pageable host memory; use device or pinned host memory", who, p);
  *out = attr.devicePointer;
  return PKV_OK;
}

int check_shape(int32_t Hkv, int32_t D, int32_t block_size, const char* who) {
  PKV_REQUIRE(Hkv > 0, "%s: Hkv must be > 0 (got %d)", who, Hkv);
  PKV_REQUIRE(D == 64 || D == 128, "%s: D must be 64 or 128 (got %d)", who, D);
  PKV_REQUIRE(block_size == 8 || block_size == 16 || block_size == 32,
              "%s: block_size must be 8, 16 or 32 (got %d)", who, block_size);
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_kv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                             int32_t T, void* k_cache, void* v_cache, int32_t num_blocks,
                             int32_t Hkv, int32_t D, int32_t block_size, int32_t* dev_status,
                             void* stream) {
  if (int rc = check_shape(Hkv, D, block_size, "pkv_kv_append")) return rc;
  PKV_REQUIRE(T >= 0, "pkv_kv_append: T must be >= 0 (got %d)", T);
  PKV_REQUIRE(num_blocks > 0 && (int64_t)num_blocks * block_size < (int64_t(1) << 31),
              "pkv_kv_append: num_blocks * block_size must be in [1, 2^31)");
  if (T == 0) return ok();
  PKV_REQUIRE(k_new && v_new && slot_mapping && k_cache && v_cache, "pkv_kv_append: NULL pointer");
  PKV_REQUIRE(aligned16(k_new) && aligned16(v_new) && aligned16(k_cache) && aligned16(v_cache),
              "pkv_kv_append: bf16 arrays must be 16-byte aligned");
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;
  AppendArgs a;
  a.k_new = static_cast<const uint4*>(k_new);
  a.v_new = static_cast<const uint4*>(v_new);
  a.slot_mapping = slot_mapping;
  a.k_cache = static_cast<uint4*>(k_cache);
  a.v_cache = static_cast<uint4*>(v_cache);
  a.num_slots = (int64_t)num_blocks * block_size;
  a.T = T;
  a.Hkv = Hkv;
  a.vec_per_row = D / 8;
  a.block_size = block_size;
  a.status = dev_status;
  const int64_t total = (int64_t)T * Hkv * (D / 8);
  const int64_t want = (total + 255) / 256;
  const int64_t cap = (int64_t)dev->sm_count * 8;  // 8 resident CTAs of 256 per SM
  const int grid = (int)(want < cap ? want : cap);
  kv_append_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  if (int rc = check_launch("pkv_kv_append")) return rc;
  return ok();
}

extern "C" int pkv_kv_append_fp8(const void* k_new, const void* v_new,
                                 const int32_t* slot_mapping, int32_t T, void* k_codes,
                                 void* v_codes, float* k_scales, float* v_scales,
                                 int32_t num_blocks, int32_t Hkv, int32_t D, int32_t block_size,
                                 int32_t* dev_status, void* stream) {
  if (int rc = check_shape(Hkv, D, block_size, "pkv_kv_append_fp8")) return rc;
  PKV_REQUIRE(T >= 0, "pkv_kv_append_fp8: T must be >= 0 (got %d)", T);
  PKV_REQUIRE(num_blocks > 0 && (int64_t)num_blocks * block_size < (int64_t(1) << 31),
              "pkv_kv_append_fp8: num_blocks * block_size must be in [1, 2^31)");
  if (T == 0) return ok();
  PKV_REQUIRE(k_new && v_new && slot_mapping && k_codes && v_codes && k_scales && v_scales,
              "pkv_kv_append_fp8: NULL pointer");
  PKV_REQUIRE(aligned16(k_new) && aligned16(v_new) && aligned16(k_codes) && aligned16(v_codes) &&
                  aligned16(k_scales) && aligned16(v_scales),
              "pkv_kv_append_fp8: arrays must be 16-byte aligned");
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;
  AppendFp8Args a;
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.slot_mapping = slot_mapping;
  a.k8 = static_cast<uint8_t*>(k_codes);
  a.v8 = static_cast<uint8_t*>(v_codes);
  a.ks = k_scales;
  a.vs = v_scales;
  a.num_slots = (int64_t)num_blocks * block_size;
  a.T = T;
  a.Hkv = Hkv;
  a.D = D;
  a.block_size = block_size;
  a.status = dev_status;
  const int64_t rows = (int64_t)T * Hkv * 2;
  const int64_t want = (rows + 63) / 64;  // 64 rows per CTA of 256 threads
  const int64_t cap = (int64_t)dev->sm_count * 8;
  const int grid = (int)(want < cap ? want : cap);
  if (D == 128)
    kv_append_fp8_kernel<128><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  else
    kv_append_fp8_kernel<64><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  if (int rc = check_launch("pkv_kv_append_fp8")) return rc;
  return ok();
}

extern "C" int pkv_block_copy(void* k_cache, void* v_cache, const int32_t* pairs, int32_t n,
                              int32_t num_blocks, int32_t Hkv, int32_t D, int32_t block_size,
                              int32_t* dev_status, void* stream) {
  if (int rc = check_shape(Hkv, D, block_size, "pkv_block_copy")) return rc;
  PKV_REQUIRE(n >= 0, "pkv_block_copy: n must be >= 0 (got %d)", n);
  PKV_REQUIRE(num_blocks > 0, "pkv_block_copy: num_blocks must be > 0");
  if (n == 0) return ok();
  PKV_REQUIRE(k_cache && v_cache && pairs, "pkv_block_copy: NULL pointer");
  PKV_REQUIRE(aligned16(k_cache) && aligned16(v_cache),
              "pkv_block_copy: pools must be 16-byte aligned");
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;
  CopyArgs a;
  a.k_cache = static_cast<uint4*>(k_cache);
  a.v_cache = static_cast<uint4*>(v_cache);
  a.pairs = pairs;
  a.n = n;
  a.num_blocks = num_blocks;
  a.vec_per_block = (int64_t)Hkv * block_size * D / 8;
  a.status = dev_status;
  dim3 grid((unsigned)n, 2);
  block_copy_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  if (int rc = check_launch("pkv_block_copy")) return rc;
  return ok();
}

extern "C" int pkv_swap_blocks(void* k_cache, void* v_cache, const int32_t* blocks, int32_t n,
                               int32_t num_blocks, int32_t Hkv, int32_t D, int32_t block_size,
                               void* k_buf, void* v_buf, int32_t to_buffer, int32_t* dev_status,
                               void* stream) {
  if (int rc = check_shape(Hkv, D, block_size, "pkv_swap_blocks")) return rc;
  PKV_REQUIRE(n >= 0 && n <= 65535, "pkv_swap_blocks: n must be in [0, 65535] (got %d)", n);
  PKV_REQUIRE(num_blocks > 0, "pkv_swap_blocks: num_blocks must be > 0");
  PKV_REQUIRE(to_buffer == 0 || to_buffer == 1, "pkv_swap_blocks: to_buffer must be 0 or 1");
  if (n == 0) return ok();
  PKV_REQUIRE(k_cache && v_cache && blocks && k_buf && v_buf, "pkv_swap_blocks: NULL pointer");
  PKV_REQUIRE(aligned16(k_cache) && aligned16(v_cache) && aligned16(k_buf) && aligned16(v_buf),
              "pkv_swap_blocks: arrays must be 16-byte aligned");
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;
  void* kd = nullptr;
  void* vd = nullptr;
  if (int rc = device_address(k_buf, &kd, "pkv_swap_blocks")) return rc;
  if (int rc = device_address(v_buf, &vd, "pkv_swap_blocks")) return rc;
  SwapArgs a;
  a.k_cache = static_cast<uint4*>(k_cache);
  a.v_cache = static_cast<uint4*>(v_cache);
  a.blocks = blocks;
  a.k_buf = static_cast<uint4*>(kd);
  a.v_buf = static_cast<uint4*>(vd);
  a.n = n;
  a.num_blocks = num_blocks;
  a.vec_per_block = (int64_t)Hkv * block_size * D / 8;
  a.to_buffer = to_buffer;
  a.status = dev_status;
  int64_t per_block = (a.vec_per_block + 255) / 256;
  if (per_block > 16) per_block = 16;
  dim3 grid((unsigned)per_block, (unsigned)n, 2);
  swap_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  if (int rc = check_launch("pkv_swap_blocks")) return rc;
  return ok();
}
