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

// fp32 -> bf16 bits, round to nearest even; infinities stay infinite, NaN stays NaN.
__device__ __forceinline__ uint16_t f_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  // a NaN stays a (quiet) NaN with its sign: the rounding add below would
  // carry the all-ones NaN into the sign bit and leave -0
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
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

// Store with release semantics at system scope: writes ordered before it (by
// this thread, or by threads synchronised with it) are visible to the host
// before the stored value is.
__device__ __forceinline__ void st_release_sys(int32_t* p, int32_t v) {
  asm volatile("st.release.sys.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// Programmatic dependent launch: wait for the previous kernel in the stream
// (a no-op when this grid was launched without the attribute), and let the
// next kernel's blocks be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Sum of squares of n elements (n % 8 == 0, 16-byte aligned) of an fp32 or
// bf16 row, block-wide, vector loads with independent iterations.
__device__ __forceinline__ float row_sumsq(const void* src, int dt, size_t base, int n, float* red) {
  float ss = 0.f;
  if (dt == MTP_DTYPE_BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(src) + base);
#pragma unroll 4
    for (int i = threadIdx.x; i < n / 8; i += blockDim.x) {
      const uint4 w = __ldg(p + i);
      const float f[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                          bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + base);
#pragma unroll 4
    for (int i = threadIdx.x; i < n / 4; i += blockDim.x) {
      const float4 v = p[i];
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
  }
  return block_sum(ss, red);
}

// dst[k] = src[base + k] * scale * w[k] for k < n (n % 8 == 0), to fp32 shared memory.
__device__ __forceinline__ void row_stage(float* dst, const void* src, int dt, size_t base, int n, float scale,
                                          const float* w) {
  if (dt == MTP_DTYPE_BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(src) + base);
#pragma unroll 2
    for (int i = threadIdx.x; i < n / 8; i += blockDim.x) {
      const uint4 v = __ldg(p + i);
      const float f[8] = {bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y),
                          bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w)};
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[8 * i + j] = f[j] * scale * (w ? w[8 * i + j] : 1.f);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + base);
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll 4
    for (int i = threadIdx.x; i < n / 4; i += blockDim.x) {
      float4 v = p[i];
      if (w) {
        const float4 ww = reinterpret_cast<const float4*>(w)[i];
        v = make_float4(v.x * scale * ww.x, v.y * scale * ww.y, v.z * scale * ww.z, v.w * scale * ww.w);
      } else {
        v = make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
      }
      d4[i] = v;
    }
  }
}

// ------------------------------------------------------ mbarrier / bulk copy
constexpr unsigned kWaitLimit = 1u << 24;  // try_wait polls before a wait gives up

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; false when the poll budget runs out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned limit = kWaitLimit) {
  for (unsigned i = 0; i < limit; ++i)
    if (mbar_try(bar, parity)) return true;
  return false;
}

// Bulk asynchronous copy global -> shared (16-byte aligned, size % 16 == 0),
// completing on an mbarrier transaction count.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<A&&>(args)...);
}

}  // namespace mtp
