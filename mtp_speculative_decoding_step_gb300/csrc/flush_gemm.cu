// Flush path on the 5th-generation tensor cores (sm_103a).
//
// A flush writes up to 256 completed pairs (token at S+1, target hidden at S,
// "Ollama qwen3_5 MTP loader and SelfDraft path", Facts: pairing, 256-token
// cap) into the draft KV. For a one-layer head the K/V of a slot depend only on
// its pair, so a flush of M pairs is two dense contractions:
//   h0[M, H]      = x[M, 2H] . W_fc^T          x = [norm_e(E[tok]) ; norm_h(hid)]
//   kv[M, 2 kw]   = b[M, H] . [W_k ; W_v]^T    b = norm_in(h0)
// followed by the per-head k_norm + RoPE + cache store.
//
// k_tc_gemm: D[M, N] (fp32) = A[M, K] . B[N, K]^T with A, B bf16 and K-major.
// One CTA owns a 128 x BN tile of D for a K range:
//   warp 0, one thread : TMA producer (128B-swizzled 64-wide K tiles of A, B)
//   warp 1, one thread : tcgen05.mma issuer (M128 x N BN x K16 per instruction)
//   warps 0-3          : epilogue, TMEM -> registers -> global (fp32)
// The accumulator lives in tensor memory (BN columns). Split-K CTAs write
// partial tiles [split][M][N] that the consumer kernel sums in split order.
// Every mbarrier wait is bounded: on expiry the CTA raises the status word,
// waits (bounded) for its own copies, frees its TMEM and returns.
#include <mutex>

#include "kernels.h"
#include "tc_common.cuh"

namespace mtp {

using namespace tc;

struct TcGemmArgs {
  int M, N, K;
  int n_split_b;     // columns [0, n_split_b) come from map b0, the rest from map b1
  int ksplit;        // number of K splits (gridDim.z)
  float* D;          // [ksplit][M][ldd]
  long long ldd;
  int32_t* status;
  const uint8_t* pf[2];  // ranges the next kernel streams, prefetched into L2 (or null)
  long long pf_bytes[2];
};

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <int BN, int STAGES, int MH>
__global__ void __launch_bounds__(128, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb0,
              const __grid_constant__ CUtensorMap tb1, const TcGemmArgs a) {
  // MH row halves of 128 per CTA share every B tile; accumulator h lives in
  // TMEM columns [h*BN, (h+1)*BN).
  constexpr uint32_t kABytes = MH * kTileM * kTileK * 2;
  constexpr uint32_t kBBytes = BN * kTileK * 2;
  constexpr uint32_t kStage = kABytes + kBBytes;
  constexpr uint32_t kCols = MH * BN;
  constexpr uint32_t kTmemCols = kCols <= 32 ? 32 : (kCols <= 64 ? 64 : (kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512)));
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + STAGES * kStage);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kTileM * MH, n0 = blockIdx.y * BN;
  const int nk_total = a.K / kTileK;
  const int per = (nk_total + a.ksplit - 1) / a.ksplit;
  const int kb = blockIdx.z * per;
  const int nk = min(per, nk_total - kb);
  const CUtensorMap* tb = n0 < a.n_split_b ? &tb0 : &tb1;
  const int nb = n0 < a.n_split_b ? n0 : n0 - a.n_split_b;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(accf), 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // TMA producer. The weight tiles (B) do not depend on the previous kernel:
    // the first ring of them is requested before waiting for it, the
    // activations (A) after. Weight tiles further ahead are prefetched into L2
    // kPrefetch steps before their shared-memory load, so the loads the
    // pipeline waits on hit L2.
    constexpr int kPrefetch = STAGES;
    const int pre = min(nk, STAGES);
    for (int i = 0; i < pre; ++i) {
      mbar_expect_tx(smem_u32(&full[i]), kStage);
      tma_load_2d(smem_u32(base + i * kStage + kABytes), tb, (kb + i) * kTileK, nb, smem_u32(&full[i]));
    }
    for (int i = STAGES; i < min(nk, STAGES + kPrefetch); ++i) tma_prefetch_2d(tb, (kb + i) * kTileK, nb);
    pdl_wait();
    for (int i = 0; i < pre; ++i)
      tma_load_2d(smem_u32(base + i * kStage), &ta, (kb + i) * kTileK, m0, smem_u32(&full[i]));
    for (int i = pre; i < nk; ++i) {
      const int s = i % STAGES, r = i / STAGES;
      if (!mbar_wait(smem_u32(&empty[s]), (r - 1) & 1)) { *s_fail = 1; break; }
      if (i + kPrefetch < nk) tma_prefetch_2d(tb, (kb + i + kPrefetch) * kTileK, nb);
      uint8_t* as = base + s * kStage;
      mbar_expect_tx(smem_u32(&full[s]), kStage);
      tma_load_2d(smem_u32(as), &ta, (kb + i) * kTileK, m0, smem_u32(&full[s]));
      tma_load_2d(smem_u32(as + kABytes), tb, (kb + i) * kTileK, nb, smem_u32(&full[s]));
    }
    // the next kernel's weights: this CTA's share of each range, into L2
    const long long nb_cta = (long long)gridDim.x * gridDim.y * gridDim.z;
    const long long cta = ((long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    for (int q = 0; q < 2; ++q) {
      if (!a.pf[q]) continue;
      const long long share = ((a.pf_bytes[q] + nb_cta - 1) / nb_cta + 15) & ~15LL;
      const long long lo = cta * share, hi = min(a.pf_bytes[q], lo + share) & ~15LL;
      for (long long o = lo; o < hi; o += 65536) prefetch_l2(a.pf[q] + o, (uint32_t)min(65536LL, hi - o));
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = idesc_bf16(kTileM, BN);
    bool ok = true;
    for (int i = 0; i < nk && ok; ++i) {
      const int s = i % STAGES, r = i / STAGES;
      if (!mbar_wait(smem_u32(&full[s]), r & 1)) { ok = false; break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t as = smem_u32(base + s * kStage), bs = as + kABytes;
#pragma unroll
      for (int kk = 0; kk < kTileK / 16; ++kk)
#pragma unroll
        for (int h = 0; h < MH; ++h)
          mma_bf16(tmem + (uint32_t)(h * BN), sdesc(as + h * kTileM * kTileK * 2 + kk * 32), sdesc(bs + kk * 32),
                   idesc, (i > 0 || kk > 0) ? 1u : 0u);
      mma_commit(smem_u32(&empty[s]));
    }
    if (!ok) *s_fail = 1;
    mma_commit(smem_u32(accf));
  }
  __syncwarp();

  // epilogue: TMEM lanes 32w..32w+31 hold rows m0 + 32w + lane; the partials
  // are written only once the previous kernel (a reader of D) has finished
  pdl_wait();
  pdl_trigger();
  const bool got = mbar_wait(smem_u32(accf), 0);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (got) {
#pragma unroll 1
    for (int h = 0; h < MH; ++h) {
      const int row = m0 + h * kTileM + warp * 32 + lane;
      float* drow = a.D + ((size_t)blockIdx.z * a.M + row) * a.ldd + n0;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(h * BN + c), v);
        if (row < a.M) {
          float4* d4 = reinterpret_cast<float4*>(drow + c);
#pragma unroll
          for (int j = 0; j < 4; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && (!got || *s_fail)) {
    flag_status(a.status, MTP_ERR_TIMEOUT);
    // let any copy still in flight land before the shared memory is released
    for (int s = 0; s < STAGES; ++s) mbar_wait(smem_u32(&full[s]), 0);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------ host side

// D[split][M][N] = A[M][K] . [B0; B1]^T  (B0 rows [0, n0rows), B1 the rest).
template <int BN, int STAGES, int MH>
static bool tc_gemm_t(const void* A, int M, int K, const void* B0, int n0rows, const void* B1, int N, int ksplit,
                      float* D, int32_t* status, cudaStream_t s, const void* const* pf, const long long* pf_bytes) {
  if (M < 1 || K % kTileK != 0 || N % BN != 0 || n0rows % BN != 0 || ksplit < 1) return false;
  CUtensorMap ta, tb0, tb1;
  if (!make_map(&ta, A, M, K, kTileM * MH)) return false;
  if (!make_map(&tb0, B0, n0rows, K, BN)) return false;
  if (!make_map(&tb1, B1 ? B1 : B0, B1 ? N - n0rows : n0rows, K, BN)) return false;
  TcGemmArgs a;
  a.M = M; a.N = N; a.K = K; a.n_split_b = n0rows; a.ksplit = ksplit; a.D = D; a.ldd = N; a.status = status;
  for (int q = 0; q < 2; ++q) {
    a.pf[q] = pf ? static_cast<const uint8_t*>(pf[q]) : nullptr;
    a.pf_bytes[q] = pf && pf[q] ? pf_bytes[q] : 0;
  }
  const int smem = STAGES * (kTileM * MH + BN) * kTileK * 2 + 1024 + 256;
  auto k = k_tc_gemm<BN, STAGES, MH>;
  {
    // the dynamic shared memory limit, raised once per device
    static std::mutex mu;
    static bool set[kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev]) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      set[dev] = true;
    }
  }
  dim3 grid((M + kTileM * MH - 1) / (kTileM * MH), N / BN, ksplit);
  const cudaError_t e = launch_pdl(k, grid, dim3(128), (size_t)smem, s, ta, tb0, tb1, a);
  count_launch();
  return e == cudaSuccess;
}

// mh: 128-row halves per CTA (1 or 2); bn: 128, 160, 256 (mh 1) or 128, 256 (mh 2).
bool launch_tc_gemm(const void* A, int M, int K, const void* B0, int n0rows, const void* B1, int N, int bn,
                    int ksplit, float* D, int32_t* status, cudaStream_t s, int mh, const void* const* pf,
                    const long long* pf_bytes) {
  if (mh == 2 && bn == 256) return tc_gemm_t<256, 3, 2>(A, M, K, B0, n0rows, B1, N, ksplit, D, status, s, pf, pf_bytes);
  if (mh == 2) return tc_gemm_t<128, 4, 2>(A, M, K, B0, n0rows, B1, N, ksplit, D, status, s, pf, pf_bytes);
  if (bn == 256) return tc_gemm_t<256, 4, 1>(A, M, K, B0, n0rows, B1, N, ksplit, D, status, s, pf, pf_bytes);
  if (bn == 160) return tc_gemm_t<160, 5, 1>(A, M, K, B0, n0rows, B1, N, ksplit, D, status, s, pf, pf_bytes);
  return tc_gemm_t<128, 6, 1>(A, M, K, B0, n0rows, B1, N, ksplit, D, status, s, pf, pf_bytes);
}

}  // namespace mtp
