// Record writer: bf16 latent [n][512] + bf16 rope [n][64] -> fp8_ds_mla
// records [n][656].  The rule is the one the gfx950 sparse-MLA page states for
// vLLM's concat_and_cache_ds_mla writer (module docstring, "Preconditions"):
// per 128-wide block, scale = pow2ceil(max(amax, 1e-4) / 448), latent stored
// as E4M3(x / scale), scales as f32, rope bf16 bit for bit.
//
// One warp per record: lane l owns latent dims [16 l, 16 l + 16), i.e. block
// l / 8; the block amax is reduced over the 8 lanes of the block.  Loads and
// stores are 16-byte vectors; a warp writes its record's 656 bytes at once.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Smallest power of two >= y for a positive normal float.
__device__ __forceinline__ float pow2ceil_pos(float y) {
  uint32_t b = __float_as_uint(y);
  uint32_t e = b >> 23;              // biased exponent (sign is 0)
  if (b & 0x7FFFFFu) e += 1;          // not a power of two: next binade
  return __uint_as_float(e << 23);
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  __nv_fp8x2_storage_t s = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
  return uint32_t(s);
}

__global__ void __launch_bounds__(32 * kWarpsPerBlock)
pack_records_kernel(const uint16_t* __restrict__ latent, int64_t latent_stride,
                    const uint16_t* __restrict__ rope, int64_t rope_stride, int64_t n,
                    uint8_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t rec = int64_t(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (rec >= n) return;
  const uint16_t* src = latent + rec * latent_stride + lane * 16;
  uint4 a = *reinterpret_cast<const uint4*>(src);
  uint4 b = *reinterpret_cast<const uint4*>(src + 8);
  uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_lo(w[i]);
    x[2 * i + 1] = bf16_hi(w[i]);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = pow2ceil_pos(fmaxf(amax, 1e-4f) / 448.0f);
  // 1 / scale is a power of two as well: exact.
  const float inv = __uint_as_float((254u - (__float_as_uint(scale) >> 23)) << 23);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo = e4m3x2(x[4 * i] * inv, x[4 * i + 1] * inv);
    uint32_t hi = e4m3x2(x[4 * i + 2] * inv, x[4 * i + 3] * inv);
    c[i] = lo | (hi << 16);
  }
  uint8_t* dst = out + rec * kRecordBytes;
  *reinterpret_cast<uint4*>(dst + lane * 16) = make_uint4(c[0], c[1], c[2], c[3]);
  if ((lane & 7) == 0) *reinterpret_cast<float*>(dst + kScaleOffset + 4 * (lane >> 3)) = scale;
  if (lane < 8) {
    uint4 r = *reinterpret_cast<const uint4*>(rope + rec * rope_stride + lane * 8);
    *reinterpret_cast<uint4*>(dst + kRopeOffset + lane * 16) = r;
  }
}

}  // namespace

cudaError_t launch_pack(const void* latent, int64_t latent_stride, const void* rope,
                        int64_t rope_stride, int64_t n, void* kv_out, cudaStream_t stream) {
  int64_t blocks = (n + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  pack_records_kernel<<<unsigned(blocks), 32 * kWarpsPerBlock, 0, stream>>>(
      static_cast<const uint16_t*>(latent), latent_stride, static_cast<const uint16_t*>(rope),
      rope_stride, n, static_cast<uint8_t*>(kv_out));
  return cudaGetLastError();
}

}  // namespace smla
