// Device helpers shared by the MTP kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mtp.h"

namespace mtp {

constexpr int kWarp = 32;

// Status word bits (1 << mtp_status).
__device__ __forceinline__ void flag_status(int32_t* status, int code) {
  if (status) atomicOr(status, 1 << code);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN stays NaN-ish).
__device__ __forceinline__ uint16_t f_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// 16-byte streaming load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Ordered (value desc, index asc) argmax combine.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Element k of an fp32 or bf16 array.
__device__ __forceinline__ float load_elem(const void* p, int dt, size_t k) {
  return dt == MTP_DTYPE_BF16 ? bf16_to_f(((const uint16_t*)p)[k]) : ((const float*)p)[k];
}

__device__ __forceinline__ void store_elem(void* p, int dt, size_t k, float v) {
  if (dt == MTP_DTYPE_BF16) ((uint16_t*)p)[k] = f_to_bf16(v);
  else ((float*)p)[k] = v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024); all threads get it.
__device__ __forceinline__ float block_sum(float v, float* sh /*[32]*/) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  float t = 0.f;
  if (w == 0) {
    t = lane < nw ? sh[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) sh[0] = t;
  }
  __syncthreads();
  return sh[0];
}

}  // namespace mtp
