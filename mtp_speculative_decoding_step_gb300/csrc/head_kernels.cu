// MTP drafter head kernels for sm_103a: the batch-1..8 GEMV family (fc, QKV,
// o_proj, gate/up, down, lm_head) with fused RMSNorm prologues and residual /
// SwiGLU / logits+argmax epilogues, the per-head q/k norm + RoPE + KV append,
// and split-slot decode attention.
//
// The head's forward is the one given on the "support the qwen3_5_mtp
// drafter" issue page, section "Upstream contract to port":
//   h = fc(concat(pre_fc_norm_embedding(embed(tok)), pre_fc_norm_hidden(hidden)))
// followed by one full-attention decoder layer and the final norm, with the
// target's tied lm_head borrowed for the logits.
//
// All of it is HBM-bound at these batch widths: every kernel streams its
// weight matrix exactly once with 16-byte L1-bypassing loads, keeps the
// activations (fp32) in shared memory and accumulates in fp32.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <algorithm>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

static unsigned long long g_launches = 0;
void count_launch(int n) { __atomic_fetch_add(&g_launches, (unsigned long long)n, __ATOMIC_RELAXED); }
unsigned long long launches_so_far() { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

// ---------------------------------------------------------------- GEMV

template <typename WT>
struct Vec;
template <>
struct Vec<uint16_t> {  // 8 bf16 per 16-byte vector
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& w, float* f) {
    f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
    f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
    f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
  }
};
template <>
struct Vec<float> {  // 4 fp32 per 16-byte vector
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& w, float* f) {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
  }
};

// fp8 e4m3 weights (the quantised draft head): 16 per 16-byte vector, widened
// exactly through f16 pairs.
struct fp8e4m3 {
  uint8_t v;
};
template <>
struct Vec<fp8e4m3> {
  static constexpr int N = 16;
  __device__ __forceinline__ static void unpack(const uint4& w, float* f) {
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h0, h1;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h0) : "h"((unsigned short)(wd[i] & 0xFFFFu)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h1) : "h"((unsigned short)(wd[i] >> 16)));
      f[4 * i + 0] = __half2float(__ushort_as_half((unsigned short)(h0 & 0xFFFFu)));
      f[4 * i + 1] = __half2float(__ushort_as_half((unsigned short)(h0 >> 16)));
      f[4 * i + 2] = __half2float(__ushort_as_half((unsigned short)(h1 & 0xFFFFu)));
      f[4 * i + 3] = __half2float(__ushort_as_half((unsigned short)(h1 >> 16)));
    }
  }
};

template <typename WT, int MT, int RPW>
__device__ __forceinline__ void gemv_fma(float (&acc)[RPW][MT], const uint4 (&w)[RPW], const float* xs,
                                         int KS, int kb) {
  constexpr int VN = Vec<WT>::N;
  if constexpr (MT <= 4) {
    // x of every item held in registers, reused across the RPW rows
    float xv[MT][VN];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float4* p = reinterpret_cast<const float4*>(xs + m * KS + kb);
#pragma unroll
      for (int j = 0; j < VN / 4; ++j) {
        float4 t = p[j];
        xv[m][4 * j] = t.x; xv[m][4 * j + 1] = t.y; xv[m][4 * j + 2] = t.z; xv[m][4 * j + 3] = t.w;
      }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      float wf[VN];
      Vec<WT>::unpack(w[i], wf);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float a = acc[i][m];
#pragma unroll
        for (int j = 0; j < VN; ++j) a = fmaf(wf[j], xv[m][j], a);
        acc[i][m] = a;
      }
    }
  } else {
    // wide batches: rows unpacked once, x of one item at a time
    float wf[RPW][VN];
#pragma unroll
    for (int i = 0; i < RPW; ++i) Vec<WT>::unpack(w[i], wf[i]);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float xv[VN];
      const float4* p = reinterpret_cast<const float4*>(xs + m * KS + kb);
#pragma unroll
      for (int j = 0; j < VN / 4; ++j) {
        float4 t = p[j];
        xv[4 * j] = t.x; xv[4 * j + 1] = t.y; xv[4 * j + 2] = t.z; xv[4 * j + 3] = t.w;
      }
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        float a = acc[i][m];
#pragma unroll
        for (int j = 0; j < VN; ++j) a = fmaf(wf[i][j], xv[j], a);
        acc[i][m] = a;
      }
    }
  }
}

// Block-reduce MT partial sums at once (one barrier round);
// every thread gets all MT totals, each summed in a fixed order.
template <int MT>
__device__ __forceinline__ void block_sum_n(float (&v)[MT], float* red /* >= 32 * MT */) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int m = 0; m < MT; ++m) v[m] = warp_sum(v[m]);
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int m = 0; m < MT; ++m) red[m * 32 + w] = v[m];
  __syncthreads();
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float t = 0.f;
    for (int k = 0; k < nw; ++k) t += red[m * 32 + k];
    v[m] = t;
  }
  __syncthreads();
}

// Stage x[m][k0 .. k0+KS) (fp32) into shared memory, applying the prologue.
// All items are handled together: one pass for their sums of squares, one
// barrier round, one staging pass.
template <int MT>
__device__ void gemv_prologue(const GemvArgs& a, float* xs, int k0, int KS, float* red) {
  const int tid = threadIdx.x;
  if (a.pro == PRO_DUAL) {
    // x = [norm_e(E[tok]) ; norm_h(hidden)]; this block's slice may take a
    // part of each half, and each part needs its half's norm.
    const int H = a.K / 2;
    const int ke1 = min(k0 + KS, H), kh0 = max(k0, H);
    const bool use_e = k0 < ke1, use_h = kh0 < k0 + KS;
    size_t be[MT], bh[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      be[m] = 0;
      bh[m] = 0;
      if (m < a.M) {
        int t = a.tok[a.tok_idx[m]];
        if (t < 0 || t >= a.vocab) {  // a bad token id reads row 0 and raises the status word
          if (tid == 0 && use_e) flag_status(a.status, MTP_ERR_BAD_ARG);
          t = 0;
        }
        be[m] = (size_t)t * (size_t)H;
        bh[m] = (size_t)a.hid_off[m];
      }
    }
    float ss[2 * MT];  // [0, MT): embedding rows, [MT, 2 MT): hidden rows
#pragma unroll
    for (int m = 0; m < 2 * MT; ++m) ss[m] = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      if (half == 0 ? !use_e : !use_h) continue;
      const void* src = half == 0 ? a.E : a.hid;
      const int dt = half == 0 ? a.wdt : a.hid_dt;
      if (dt == MTP_DTYPE_BF16) {
        for (int i = tid; i < H / 8; i += blockDim.x) {
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m < a.M) {
              const size_t b = half == 0 ? be[m] : bh[m];
              const uint4 w = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(src) + b) + i);
              const float f[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                                  bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
              float& acc = ss[half * MT + m];
#pragma unroll
              for (int j = 0; j < 8; ++j) acc = fmaf(f[j], f[j], acc);
            }
          }
        }
      } else {
        for (int i = tid; i < H / 4; i += blockDim.x) {
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m < a.M) {
              const size_t b = half == 0 ? be[m] : bh[m];
              const float4 v = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + b) + i);
              float& acc = ss[half * MT + m];
              acc = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, acc))));
            }
          }
        }
      }
    }
    block_sum_n<2 * MT>(ss, red);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m >= a.M) continue;
      if (use_e)
        row_stage(xs + m * KS, a.E, a.wdt, be[m] + k0, ke1 - k0, rsqrtf(ss[m] / (float)H + a.eps), a.nw + k0);
      if (use_h)
        row_stage(xs + m * KS + (kh0 - k0), a.hid, a.hid_dt, bh[m] + (kh0 - H), k0 + KS - kh0,
                  rsqrtf(ss[MT + m] / (float)H + a.eps), a.nw2 + (kh0 - H));
    }
  } else if (a.pro == PRO_NORM) {
    float ss[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) ss[m] = 0.f;
    for (int i = tid; i < a.K / 4; i += blockDim.x) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < a.M) {
          const float4 v = reinterpret_cast<const float4*>(a.x + (size_t)m * a.ldx)[i];
          ss[m] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss[m]))));
        }
      }
    }
    block_sum_n<MT>(ss, red);
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (m < a.M)
        row_stage(xs + m * KS, a.x + (size_t)m * a.ldx, MTP_DTYPE_F32, k0, KS, rsqrtf(ss[m] / (float)a.K + a.eps),
                  a.nw + k0);
  } else {
    for (int m = 0; m < a.M; ++m)
      row_stage(xs + m * KS, a.x + (size_t)m * a.ldx, MTP_DTYPE_F32, k0, KS, 1.f, nullptr);
  }
  for (int m = a.M; m < MT; ++m)
    for (int k = tid; k < KS; k += blockDim.x) xs[m * KS + k] = 0.f;
}

// PRO_NORM with the norm's scale left for the epilogue: RMSNorm(x) * nw =
// r (x * nw) with r = rsqrt(mean(x^2) + eps) one scalar per item, so
// W RMSNorm(x) nw = r W (x * nw). Stage x * nw over the slice in one pass and
// keep each thread's sum of squares of x over the slice; the block's sums meet
// at the epilogue (across the K splits in the split combine), which applies r.
// No pass over the whole row and no barrier round stand before the weights.
template <int MT>
__device__ void gemv_stage_deferred(const GemvArgs& a, float* xs, int k0, int KS, float (&ss)[MT]) {
  const float4* w4 = reinterpret_cast<const float4*>(a.nw + k0);
#pragma unroll
  for (int m = 0; m < MT; ++m) ss[m] = 0.f;
  for (int i = threadIdx.x; i < KS / 4; i += blockDim.x) {
    const float4 ww = w4[i];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < a.M) {
        v = reinterpret_cast<const float4*>(a.x + (size_t)m * a.ldx + k0)[i];
        ss[m] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss[m]))));
        v = make_float4(v.x * ww.x, v.y * ww.y, v.z * ww.z, v.w * ww.w);
      }
      reinterpret_cast<float4*>(xs + m * KS)[i] = v;
    }
  }
}

// Split-K combine and epilogue of one block group, shared by the GEMV
// kernels. s_out[m][l] holds this block's partial of row group*ROWS + l for
// item m; every thread of the block calls it.
template <int MT, int ROWS>
__device__ void gemv_finish(const GemvArgs& a, float (*s_out)[ROWS], int group, int split, int* s_last_p,
                            bool defer = false, const float* rv_pre = nullptr) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int& s_last = *s_last_p;
  // Deterministic split-K: every split stores its partial; the last block of
  // the group sums them in split order.
  if (a.S > 1) {
    for (int t = tid; t < a.M * ROWS; t += blockDim.x) {
      const int m = t / ROWS, l = t - m * ROWS;
      a.part[((size_t)split * MT + m) * a.N + (size_t)group * ROWS + l] = s_out[m][l];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&a.counters[group], 1) == a.S - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int t = tid; t < a.M * ROWS; t += blockDim.x) {
      const int m = t / ROWS, l = t - m * ROWS;
      // the splits' partials (and sums of squares) eight at a time in flight,
      // summed in split order: the group's last block is on the kernel's tail
      float sum = 0.f, q = 0.f;
      for (int s0 = 0; s0 < a.S; s0 += 8) {
        float ps[8], qs[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int sp = s0 + u;
          ps[u] = sp < a.S ? __ldcg(&a.part[((size_t)sp * MT + m) * a.N + (size_t)group * ROWS + l]) : 0.f;
          qs[u] = (defer && sp < a.S) ? __ldcg(&a.ssq[sp * MT + m]) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          sum += ps[u];
          q += qs[u];
        }
      }
      // the deferred norm scale from the splits' sums of squares
      if (defer) sum *= rsqrtf(q / (float)a.K + a.eps);
      s_out[m][l] = sum;
    }
    if (tid == 0) a.counters[group] = 0;
    __syncthreads();
  }

  if (a.epi == EPI_SWIGLU) {
    constexpr int HALF = ROWS / 2;
    for (int t = tid; t < a.M * HALF; t += blockDim.x) {
      const int m = t / HALF, l = t - m * HALF;
      const float g = s_out[m][l], u = s_out[m][l + HALF];
      a.y[(size_t)m * a.ldy + (size_t)group * HALF + l] = g / (1.f + expf(-g)) * u;
    }
    if (a.walk) {
      // walking blocks: the last group to finish clears the group counter
      // (every group has been taken by then) and this count
      __syncthreads();
      if (tid == 0 && atomicAdd(a.done, 1) == a.ngroups - 1) {
        *a.walk = 0;
        *a.done = 0;
      }
    }
    return;
  }
  if (a.wscale) {  // per-row scales of quantised weights
    __syncthreads();
    for (int t = tid; t < a.M * ROWS; t += blockDim.x) {
      const int m = t / ROWS, l = t - m * ROWS;
      s_out[m][l] *= a.wscale[(size_t)group * ROWS + l];
    }
    __syncthreads();
  }
  for (int t = tid; t < a.M * ROWS; t += blockDim.x) {
    const int m = t / ROWS, l = t - m * ROWS;
    const size_t n = (size_t)group * ROWS + l;
    float v = s_out[m][l];
    if (a.epi == EPI_RESID) v += (rv_pre && t == tid) ? *rv_pre : a.resid[(size_t)m * a.ldr + n];
    a.y[(size_t)m * a.ldy + n] = v;
    if (a.epi == EPI_LOGITS && !isfinite(v)) flag_status(a.status, MTP_ERR_NONFINITE);
    if (a.qzero) a.qzero[(size_t)m * a.ldqz + n] = 0.f;
  }
  if (a.epi != EPI_LOGITS) return;

  // Group argmax (value desc, id asc) per item, then the last group block
  // reduces all groups into the token.
  if (warp < a.M) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int l = lane; l < ROWS; l += 32) {
      const float v = s_out[warp][l];
      const int i = group * ROWS + l;
      if (better(v, i, bv, bi)) { bv = v; bi = i; }
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      a.gmax[(size_t)warp * a.ngroups + group] = bv;
      a.gidx[(size_t)warp * a.ngroups + group] = bi;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.done, 1) == a.ngroups - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // The groups' maxima of each item, reduced by the whole block (this runs
  // once per launch, at its very end, so it is on the path to the next
  // kernel): thread t takes groups t, t + blockDim, ... with four loads in
  // flight, then warp and block reductions. s_out is free again: the block's
  // own outputs are stored.
  float* sv = &s_out[0][0];
  const int nw = (int)(blockDim.x >> 5);
  for (int m = 0; m < a.M; ++m) {
    const float* gm = a.gmax + (size_t)m * a.ngroups;
    const int* gx = a.gidx + (size_t)m * a.ngroups;
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int g0 = tid; g0 < a.ngroups; g0 += 4 * (int)blockDim.x) {
      float v[4];
      int ix[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int g = g0 + u * (int)blockDim.x;
        v[u] = g < a.ngroups ? __ldcg(gm + g) : -INFINITY;
        ix[u] = g < a.ngroups ? __ldcg(gx + g) : 0x7FFFFFFF;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (better(v[u], ix[u], bv, bi)) { bv = v[u]; bi = ix[u]; }
    }
    warp_argmax(bv, bi);
    __syncthreads();  // the previous item's block reduction has read sv
    if (lane == 0) {
      sv[2 * warp] = bv;
      sv[2 * warp + 1] = __int_as_float(bi);
    }
    __syncthreads();
    if (warp == 0) {
      bv = lane < nw ? sv[2 * lane] : -INFINITY;
      bi = lane < nw ? __float_as_int(sv[2 * lane + 1]) : 0x7FFFFFFF;
      warp_argmax(bv, bi);
      // an item whose logits are all NaN (flagged) still gets a token in range
      if (lane == 0 && a.amax_out) a.amax_out[a.amax_idx[m]] = bi == 0x7FFFFFFF ? 0 : bi;
    }
  }
  if (tid == 0) {
    *a.done = 0;
    if (a.walk) *a.walk = 0;  // every group has been taken and finished
  }
}

template <typename WT, int MT>
__global__ void __launch_bounds__(256, 2) k_gemv(const __grid_constant__ GemvArgs a) {
  constexpr int VN = Vec<WT>::N;
  constexpr int RPW = MT <= 4 ? 8 : 4;
  constexpr int ROWS = 8 * RPW;
  extern __shared__ __align__(16) float xs[];
  __shared__ float s_out[MT][ROWS];
  __shared__ float s_red[64 * MT];
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = blockIdx.x / a.S, split = blockIdx.x - group * a.S;
  const int k0 = gemv_slice_start(a.K, a.S, split), KS = gemv_slice_start(a.K, a.S, split + 1) - k0;

  // This warp's RPW consecutive physical rows.
  const int l0 = warp * RPW;
  const WT* W;
  if (a.epi == EPI_SWIGLU) {
    constexpr int HALF = ROWS / 2;
    const int prow = group * HALF + (l0 % HALF);
    W = reinterpret_cast<const WT*>(a.w[l0 < HALF ? 0 : 1]) + (size_t)prow * a.K;
  } else {
    const int v = group * ROWS + l0;
    int s = 0, start = 0;
    while (v >= a.seg_end[s]) { start = a.seg_end[s]; ++s; }
    W = reinterpret_cast<const WT*>(a.w[s]) + (size_t)(v - start) * a.K;
  }
  W += k0;

  // The weights do not depend on the previous kernel: issue this warp's first
  // loads before waiting for it. Each lane keeps one 16-byte vector of each
  // of its RPW rows in flight; with one item the next vector set is issued
  // before the current one is consumed (two sets in flight).
  // the residual (written several kernels back) of the output this thread
  // stores in the epilogue, read before the wait
  float rv = 0.f;
  if (a.epi == EPI_RESID && tid < a.M * ROWS) {
    const int m = tid / ROWS, l = tid - m * ROWS;
    rv = a.resid[(size_t)m * a.ldr + (size_t)group * ROWS + l];
  }
  const int nvec = KS / VN;
  int v0 = lane;
  bool has0 = v0 < nvec;
  uint4 w0[RPW];
  if (has0) {
#pragma unroll
    for (int i = 0; i < RPW; ++i) w0[i] = ldg_stream(W + (size_t)i * a.K + (size_t)v0 * VN);
  }
  pdl_wait();
  pdl_trigger();

  const bool defer = a.pro == PRO_NORM;
  float ssq[MT];
  if (defer)
    gemv_stage_deferred<MT>(a, xs, k0, KS, ssq);
  else
    gemv_prologue<MT>(a, xs, k0, KS, s_red);
  __syncthreads();

  float acc[RPW][MT];
#pragma unroll
  for (int i = 0; i < RPW; ++i)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[i][m] = 0.f;

  if constexpr (MT == 1) {
    uint4 w1[RPW];
    while (has0) {
      const bool has1 = v0 + 32 < nvec;
      if (has1) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) w1[i] = ldg_stream(W + (size_t)i * a.K + (size_t)(v0 + 32) * VN);
      }
      gemv_fma<WT, MT, RPW>(acc, w0, xs, KS, v0 * VN);
      if (!has1) break;
      v0 += 32;
      has0 = v0 + 32 < nvec;
      if (has0) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) w0[i] = ldg_stream(W + (size_t)i * a.K + (size_t)(v0 + 32) * VN);
      }
      gemv_fma<WT, MT, RPW>(acc, w1, xs, KS, v0 * VN);
      v0 += 32;
    }
  } else {
    while (has0) {
      gemv_fma<WT, MT, RPW>(acc, w0, xs, KS, v0 * VN);
      v0 += 32;
      has0 = v0 < nvec;
      if (has0) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) w0[i] = ldg_stream(W + (size_t)i * a.K + (size_t)v0 * VN);
      }
    }
  }

#pragma unroll
  for (int i = 0; i < RPW; ++i)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[i][m] = warp_sum(acc[i][m]);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m) s_out[m][l0 + i] = acc[i][m];
  }
  if (defer) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float v = warp_sum(ssq[m]);
      if (lane == 0) s_red[m * 32 + warp] = v;
    }
  }
  __syncthreads();
  if (defer) {
    // the block's sums of squares over its slice, in warp order
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float q = 0.f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) q += s_red[m * 32 + w];
      ssq[m] = q;
    }
    if (a.S == 1) {
      for (int t = tid; t < MT * ROWS; t += blockDim.x) {
        const int m = t / ROWS, l = t - m * ROWS;
        s_out[m][l] *= rsqrtf(ssq[m] / (float)a.K + a.eps);
      }
      __syncthreads();
    } else if (tid == 0) {
      // every block of this split has the same sums (same slice, same order)
#pragma unroll
      for (int m = 0; m < MT; ++m) a.ssq[split * MT + m] = ssq[m];
    }
  }

  gemv_finish<MT, ROWS>(a, s_out, group, split, &s_last, defer, &rv);
}

// ------------------------------------------ fp8 head GEMV on the tensor cores
//
// The e4m3 head streamed through mma.sync m16n8k16 (f16 inputs, fp32
// accumulators) instead of widened element by element: one cvt.e4m3x2 per two
// codes and one MMA per 256 codes, where the CUDA-core loop spends about two
// and a half instructions per code. Every e4m3 value is exact in f16. Each
// activation x is split into three f16 parts after scaling by a power of two
// 2^e (per item and block, chosen so that max|x| 2^e lies in [2^14, 2^15)):
// hi = f16(x'), mid = f16(x' - hi), lo = f16(x' - hi - mid), together 33
// significant bits. The products of a code and a part are exact in fp32, the
// sums accumulate in fp32, and the result is scaled back by 2^-e.
//
// A warp owns 16 rows: lane (g, t) loads 16-byte chunks of rows g and g + 8,
// the A operand. The k order inside one MMA is a permutation of the chunk's
// columns, the same for A and for the parts (the B operand, one column per
// part), so it cancels in the sum. 128 rows per block of 8 warps.
constexpr int kFp8MmaRows = 128;

__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^e such that v 2^e lies in [2^14, 2^15) (v = f 2^E, f in [0.5, 1)); 0 for
// a zero or non-finite v
__device__ __forceinline__ int fp8_part_exp(float v) {
  int E = 0;
  frexpf(v, &E);
  return (v > 0.f && isfinite(v)) ? min(max(15 - E, -126), 126) : 0;
}

// hi, mid and lo f16 parts of four scaled activations, stored at columns
// k..k+3 of three consecutive part rows PS halves apart
__device__ __forceinline__ void fp8_parts4(uint16_t* dst, int PS, float4 v) {
  const float x[4] = {v.x, v.y, v.z, v.w};
  uint16_t p[3][4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const __half hi = __float2half_rn(x[c]);
    const float r1 = x[c] - __half2float(hi);
    const __half mid = __float2half_rn(r1);
    const __half lo = __float2half_rn(r1 - __half2float(mid));
    p[0][c] = __half_as_ushort(hi);
    p[1][c] = __half_as_ushort(mid);
    p[2][c] = __half_as_ushort(lo);
  }
#pragma unroll
  for (int q = 0; q < 3; ++q)
    *reinterpret_cast<uint2*>(dst + q * PS) =
        make_uint2((uint32_t)p[q][0] | ((uint32_t)p[q][1] << 16), (uint32_t)p[q][2] | ((uint32_t)p[q][3] << 16));
}

template <int MT>
__global__ void __launch_bounds__(256, 2) k_gemv_fp8_mma(const __grid_constant__ GemvArgs a) {
  constexpr int NP = 3 * MT;        // parts: hi, mid, lo of each item
  constexpr int NT = (NP + 7) / 8;  // n-tiles of 8 parts
  extern __shared__ __align__(16) float xs[];
  __shared__ float s_out[MT][kFp8MmaRows];
  __shared__ float s_red[64 * MT];
  __shared__ int s_e[MT];
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  // Without a K split the grid may be narrower than the group count: a block
  // then walks groups blockIdx.x, + gridDim.x, ..., with one prologue, and the
  // next group's first codes in flight during this group's epilogue.
  const bool walk = a.S == 1;
  int group = walk ? blockIdx.x : blockIdx.x / a.S;
  const int split = walk ? 0 : blockIdx.x - group * a.S;
  const int k0 = gemv_slice_start(a.K, a.S, split), KS = gemv_slice_start(a.K, a.S, split + 1) - k0;
  const int PS = KS + 4;  // halves between parts (8 bytes of padding against bank conflicts)
  uint16_t* xp = reinterpret_cast<uint16_t*>(xs + MT * KS);

  // rows l0 + g and l0 + g + 8 of the group, in the virtual row space
  const int l0 = warp * 16;
  const uint8_t* WA;
  const uint8_t* WB;
  auto set_rows = [&](int grp) {
    const int v = grp * kFp8MmaRows + l0 + g;
    int sg = 0, start = 0;
    while (v >= a.seg_end[sg]) { start = a.seg_end[sg]; ++sg; }
    WA = reinterpret_cast<const uint8_t*>(a.w[sg]) + (size_t)(v - start) * a.K + k0;
    const int v8 = v + 8;
    sg = 0; start = 0;
    while (v8 >= a.seg_end[sg]) { start = a.seg_end[sg]; ++sg; }
    WB = reinterpret_cast<const uint8_t*>(a.w[sg]) + (size_t)(v8 - start) * a.K + k0;
  };
  set_rows(group);

  // A set is 256 columns: four steps of 64, lane t taking the 16-column chunk
  // 4 u + t of step u, of both its rows.
  const int nchunk = KS / 16, nset = (nchunk + 15) / 16;
  auto load_set = [&](uint4 (&w)[8], int j) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = 16 * j + 4 * u + t;
      if (q < nchunk) {
        w[2 * u] = ldg_stream(WA + 16 * q);
        w[2 * u + 1] = ldg_stream(WB + 16 * q);
      } else {
        w[2 * u] = w[2 * u + 1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  // the codes do not depend on the previous kernel: the first set (both sets
  // for one item, where the registers allow) in flight before waiting for it
  uint4 w0[8], w1[8];
  load_set(w0, 0);
  if (MT == 1 && nset > 1) load_set(w1, 1);
  pdl_wait();
  pdl_trigger();

  if (a.pro == PRO_NORM) {
    // x = RMSNorm(row) * nw: one pass for the sums of squares and the largest
    // |row * nw| of this slice (which, times the norm's scale, bounds max |x|),
    // then the parts straight from the normalised row
    float ss[MT], mx[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) ss[m] = mx[m] = 0.f;
    for (int i = tid; i < a.K / 4; i += blockDim.x) {
      const int k = 4 * i;
      const bool mine = k >= k0 && k < k0 + KS;
      const float4 ww = mine ? reinterpret_cast<const float4*>(a.nw)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < a.M) {
          const float4 v = reinterpret_cast<const float4*>(a.x + (size_t)m * a.ldx)[i];
          ss[m] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss[m]))));
          mx[m] = fmaxf(mx[m], fmaxf(fmaxf(fabsf(v.x * ww.x), fabsf(v.y * ww.y)),
                                     fmaxf(fabsf(v.z * ww.z), fabsf(v.w * ww.w))));
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      ss[m] = warp_sum(ss[m]);
      mx[m] = warp_max(mx[m]);
    }
    if (lane == 0)
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        s_red[m * 32 + warp] = ss[m];
        s_red[(MT + m) * 32 + warp] = mx[m];
      }
    __syncthreads();
    float inv[MT], up[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float t2 = 0.f, mm = 0.f;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
        t2 += s_red[m * 32 + i];
        mm = fmaxf(mm, s_red[(MT + m) * 32 + i]);
      }
      inv[m] = rsqrtf(t2 / (float)a.K + a.eps);
      const int e = fp8_part_exp(inv[m] * mm);
      up[m] = __int_as_float((127 + e) << 23);
      if (tid == 0) s_e[m] = e;
    }
    for (int i = tid; i < MT * (KS / 4); i += blockDim.x) {
      const int m = i / (KS / 4), k = 4 * (i - m * (KS / 4));
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < a.M) {
        const float4 x4 = *reinterpret_cast<const float4*>(a.x + (size_t)m * a.ldx + k0 + k);
        const float4 ww = *reinterpret_cast<const float4*>(a.nw + k0 + k);
        // the normalised element as the CUDA-core path forms it, then 2^e
        v = make_float4(x4.x * inv[m] * ww.x * up[m], x4.y * inv[m] * ww.y * up[m], x4.z * inv[m] * ww.z * up[m],
                        x4.w * inv[m] * ww.w * up[m]);
      }
      fp8_parts4(xp + 3 * m * PS + k, PS, v);
    }
  } else {
    gemv_prologue<MT>(a, xs, k0, KS, s_red);
    __syncthreads();
    // the power of two of each item: max |x| over this block's slice
    float mx[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      mx[m] = 0.f;
      for (int k = tid; k < KS; k += blockDim.x) mx[m] = fmaxf(mx[m], fabsf(xs[m * KS + k]));
      mx[m] = warp_max(mx[m]);
    }
    if (lane == 0)
#pragma unroll
      for (int m = 0; m < MT; ++m) s_red[m * 32 + warp] = mx[m];
    __syncthreads();
    if (tid < MT) {
      float v = 0.f;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) v = fmaxf(v, s_red[tid * 32 + i]);
      s_e[tid] = fp8_part_exp(v);
    }
    __syncthreads();
    for (int i = tid; i < MT * (KS / 4); i += blockDim.x) {
      const int m = i / (KS / 4), k = 4 * (i - m * (KS / 4));
      const float up = __int_as_float((127 + s_e[m]) << 23);
      const float4 x4 = *reinterpret_cast<const float4*>(xs + m * KS + k);
      fp8_parts4(xp + 3 * m * PS + k, PS, make_float4(x4.x * up, x4.y * up, x4.z * up, x4.w * up));
    }
  }
  __syncthreads();
  if (MT > 1 && nset > 1) load_set(w1, 1);

  // lane (g, t) reads part 8 n + g: the B operand's column g
  const uint16_t* xb = xp + g * PS + 16 * t;
  for (;;) {
    float d[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) d[n][0] = d[n][1] = d[n][2] = d[n][3] = 0.f;
    auto compute_set = [&](const uint4 (&w)[8], int j) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = 16 * j + 4 * u + t;
        const bool ok = q < nchunk;
        const uint32_t wa[4] = {w[2 * u].x, w[2 * u].y, w[2 * u].z, w[2 * u].w};
        const uint32_t wb[4] = {w[2 * u + 1].x, w[2 * u + 1].y, w[2 * u + 1].z, w[2 * u + 1].w};
#pragma unroll
        for (int sw = 0; sw < 4; ++sw) {
          // columns 16 q + 4 sw + {0, 1} are k = 2t, 2t+1; + {2, 3} are k = 2t+8, 2t+9
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2(wa[sw], a0, a2);
          e4m3x4_to_f16x2(wb[sw], a1, a3);
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            uint2 b = make_uint2(0u, 0u);
            if (ok && 8 * n + g < 3 * a.M)
              b = *reinterpret_cast<const uint2*>(xb + 8 * n * PS + 256 * j + 64 * u + 4 * sw);
            mma_f16(d[n], a0, a1, a2, a3, b.x, b.y);
          }
        }
      }
    };
    for (int j = 0; j < nset; j += 2) {
      compute_set(w0, j);
      if (j + 2 < nset) load_set(w0, j + 2);
      if (j + 1 >= nset) break;
      compute_set(w1, j + 1);
      if (j + 3 < nset) load_set(w1, j + 3);
    }

    // d[n] = D[row g | g + 8][part 8 n + 2 t | + 1]: item m sums parts 3m..3m+2
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float r0 = 0.f, r8 = 0.f;
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int p = 8 * n + 2 * t + c;
          if (p >= 3 * m && p < 3 * m + 3) {
            r0 += d[n][c];
            r8 += d[n][2 + c];
          }
        }
      r0 += __shfl_xor_sync(0xFFFFFFFFu, r0, 1);
      r0 += __shfl_xor_sync(0xFFFFFFFFu, r0, 2);
      r8 += __shfl_xor_sync(0xFFFFFFFFu, r8, 1);
      r8 += __shfl_xor_sync(0xFFFFFFFFu, r8, 2);
      if (t == 0) {
        const float back = __int_as_float((127 - s_e[m]) << 23);
        s_out[m][l0 + g] = r0 * back;
        s_out[m][l0 + g + 8] = r8 * back;
      }
    }
    __syncthreads();
    const int next = walk ? group + (int)gridDim.x : a.ngroups;
    if (next < a.ngroups) {
      set_rows(next);
      load_set(w0, 0);
      if (nset > 1) load_set(w1, 1);
    }
    gemv_finish<MT, kFp8MmaRows>(a, s_out, group, split, &s_last);
    if (next >= a.ngroups) break;
    group = next;
    __syncthreads();  // s_out and s_last are reused
  }
}

template <int MT>
static void launch_gemv_fp8_mma_t(const GemvArgs& a, int smem, cudaStream_t s) {
  auto k = k_gemv_fp8_mma<MT>;
  if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  // without a K split, at most the two blocks per SM that stay resident
  const int grid = a.S == 1 ? std::min(a.ngroups, 2 * device_sm_count()) : a.ngroups * a.S;
  launch_pdl(k, dim3(grid), dim3(256), smem, s, a);
  count_launch();
}

// ------------------------------------------------ walking GEMV, one item
//
// The one-item logits or SwiGLU GEMV over more than a wave of whole row groups
// (no K split: the tied lm_head, gate/up) with resident blocks that walk groups: x is staged
// once per block, the next group is taken from a counter one group ahead and
// its first weight vectors are in flight during the current group's
// epilogue. Groups are taken in order as blocks free up, so the balance is
// that of launching one block per group, without a block's launch, staging
// and cold first loads per group.
template <typename WT>
__global__ void __launch_bounds__(256, 2) k_gemv_walk(const __grid_constant__ GemvArgs a) {
  constexpr int MT = 1, RPW = 8, ROWS = 8 * RPW, VN = Vec<WT>::N;
  extern __shared__ __align__(16) float xs[];  // x over the whole row
  __shared__ float s_out[MT][ROWS];
  __shared__ float s_red[64];
  __shared__ int s_last, s_next;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvec = a.K / VN, l0 = warp * RPW;
  auto rows_of = [&](int g) -> const WT* {
    if (a.epi == EPI_SWIGLU) {
      constexpr int HALF = ROWS / 2;
      const int prow = g * HALF + (l0 % HALF);
      return reinterpret_cast<const WT*>(a.w[l0 < HALF ? 0 : 1]) + (size_t)prow * a.K;
    }
    const int v = g * ROWS + l0;
    int sg = 0, start = 0;
    while (v >= a.seg_end[sg]) { start = a.seg_end[sg]; ++sg; }
    return reinterpret_cast<const WT*>(a.w[sg]) + (size_t)(v - start) * a.K;
  };
  int group = blockIdx.x;
  const WT* W = rows_of(group);
  uint4 w0[RPW], w1[RPW];
  if (lane < nvec) {
#pragma unroll
    for (int i = 0; i < RPW; ++i) w0[i] = ldg_stream(W + (size_t)i * a.K + (size_t)lane * VN);
  }
  pdl_wait();
  pdl_trigger();
  // the block's second group (the counter starts at zero for every launch)
  if (tid == 0) s_next = (int)gridDim.x + atomicAdd(a.walk, 1);
  const bool defer = a.pro == PRO_NORM;
  float ssq[MT];
  if (defer)
    gemv_stage_deferred<MT>(a, xs, 0, a.K, ssq);
  else
    gemv_prologue<MT>(a, xs, 0, a.K, s_red);
  float r = 1.f;
  if (defer) {  // the RMSNorm scale of the whole row, once for all groups
    const float v = warp_sum(ssq[0]);
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    float q = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) q += s_red[w];
    r = rsqrtf(q / (float)a.K + a.eps);
  }
  __syncthreads();

  for (;;) {
    float acc[RPW][MT];
#pragma unroll
    for (int i = 0; i < RPW; ++i) acc[i][0] = 0.f;
    int v0 = lane;
    bool has0 = v0 < nvec;
    while (has0) {
      const bool has1 = v0 + 32 < nvec;
      if (has1) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) w1[i] = ldg_stream(W + (size_t)i * a.K + (size_t)(v0 + 32) * VN);
      }
      gemv_fma<WT, MT, RPW>(acc, w0, xs, a.K, v0 * VN);
      if (!has1) break;
      v0 += 32;
      has0 = v0 + 32 < nvec;
      if (has0) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) w0[i] = ldg_stream(W + (size_t)i * a.K + (size_t)(v0 + 32) * VN);
      }
      gemv_fma<WT, MT, RPW>(acc, w1, xs, a.K, v0 * VN);
      v0 += 32;
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) acc[i][0] = warp_sum(acc[i][0]);
    if (lane == 0)
#pragma unroll
      for (int i = 0; i < RPW; ++i) s_out[0][l0 + i] = acc[i][0] * r;
    __syncthreads();
    // the next group's first vectors in flight during this group's epilogue,
    // and the group after it taken now
    const int next = s_next;
    if (next < a.ngroups) {
      W = rows_of(next);
      if (lane < nvec) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) w0[i] = ldg_stream(W + (size_t)i * a.K + (size_t)lane * VN);
      }
    }
    __syncthreads();  // every thread has read s_next
    if (tid == 0 && next < a.ngroups) s_next = (int)gridDim.x + atomicAdd(a.walk, 1);
    gemv_finish<MT, ROWS>(a, s_out, group, 0, &s_last);
    if (next >= a.ngroups) break;
    group = next;
    __syncthreads();  // s_out, s_last and s_next are reused
  }
}

template <typename WT>
static void launch_gemv_walk_t(const GemvArgs& a, int smem, cudaStream_t s) {
  auto k = k_gemv_walk<WT>;
  if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const int grid = std::min(a.ngroups, 2 * device_sm_count());
  launch_pdl(k, dim3(grid), dim3(256), smem, s, a);
  count_launch();
}

// The walking GEMV takes one-item logits and SwiGLU jobs (the lm_head and
// gate/up: their last group to finish clears the group counter) without a K
// split and with more groups than one wave of resident blocks.
bool gemv_walks(int mt, const GemvArgs& a) {
  return mt == 1 && a.S == 1 && a.walk && (a.epi == EPI_LOGITS || a.epi == EPI_SWIGLU) &&
         a.wdt != kDtypeFp8 && a.ngroups > 2 * device_sm_count();
}

template <typename WT, int MT>
static void launch_gemv_t(const GemvArgs& a, int smem, cudaStream_t s) {
  auto k = k_gemv<WT, MT>;
  if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  launch_pdl(k, dim3(a.ngroups * a.S), dim3(256), smem, s, a);
  count_launch();
}

void launch_gemv(int mt, const GemvArgs& a, int smem, cudaStream_t s) {
  if (gemv_walks(mt, a)) {
    if (a.wdt == MTP_DTYPE_BF16)
      launch_gemv_walk_t<uint16_t>(a, smem, s);
    else
      launch_gemv_walk_t<float>(a, smem, s);
    return;
  }
  if (a.wdt == kDtypeFp8 && gemv_fp8_mma(a.N)) {
    switch (mt) {
      case 1: launch_gemv_fp8_mma_t<1>(a, smem, s); break;
      case 2: launch_gemv_fp8_mma_t<2>(a, smem, s); break;
      case 4: launch_gemv_fp8_mma_t<4>(a, smem, s); break;
      default: launch_gemv_fp8_mma_t<8>(a, smem, s); break;
    }
    return;
  }
  if (a.wdt == kDtypeFp8) {
    switch (mt) {
      case 1: launch_gemv_t<fp8e4m3, 1>(a, smem, s); break;
      case 2: launch_gemv_t<fp8e4m3, 2>(a, smem, s); break;
      case 4: launch_gemv_t<fp8e4m3, 4>(a, smem, s); break;
      default: launch_gemv_t<fp8e4m3, 8>(a, smem, s); break;
    }
    return;
  }
  const bool bf = a.wdt == MTP_DTYPE_BF16;
  switch (mt) {
    case 1: bf ? launch_gemv_t<uint16_t, 1>(a, smem, s) : launch_gemv_t<float, 1>(a, smem, s); break;
    case 2: bf ? launch_gemv_t<uint16_t, 2>(a, smem, s) : launch_gemv_t<float, 2>(a, smem, s); break;
    case 4: bf ? launch_gemv_t<uint16_t, 4>(a, smem, s) : launch_gemv_t<float, 4>(a, smem, s); break;
    default: bf ? launch_gemv_t<uint16_t, 8>(a, smem, s) : launch_gemv_t<float, 8>(a, smem, s); break;
  }
}

// One block per row of a bf16 matrix: scale = max|w| / 448 (1 for an all-zero
// row), codes = e4m3(w / scale), round to nearest even, saturating.
__global__ void k_quant_e4m3(const uint16_t* w, int cols, uint8_t* q, float* scale) {
  __shared__ float red[32];
  const uint16_t* row = w + (size_t)blockIdx.x * cols;
  float amax = 0.f;
  for (int k = threadIdx.x; k < cols; k += blockDim.x) amax = fmaxf(amax, fabsf(bf16_to_f(row[k])));
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
  const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
  if (threadIdx.x == 0) scale[blockIdx.x] = sc;
  uint16_t* qr = reinterpret_cast<uint16_t*>(q + (size_t)blockIdx.x * cols);
  for (int k = threadIdx.x; k < cols / 2; k += blockDim.x) {
    const float x0 = bf16_to_f(row[2 * k]) / sc, x1 = bf16_to_f(row[2 * k + 1]) / sc;
    unsigned short c;
    // the second operand lands in the low byte: element 2k first in memory
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(x1), "f"(x0));
    qr[k] = c;
  }
}

void launch_quant_e4m3(const uint16_t* w, int rows, int cols, uint8_t* q, float* scale, cudaStream_t s) {
  k_quant_e4m3<<<rows, 256, 0, s>>>(w, cols, q, scale);
  count_launch();
}

// ------------------------------------------------- q/k norm, RoPE, KV append

// Rotate the pair (x0 at i, x1 at i + dh/2) to position `pos`: angle =
// pos * theta^(-2i/dh). `freq` is that frequency in double (computed on the
// host at load); the angle is formed and reduced modulo 2*pi in double and
// its sine/cosine taken in fp32 (error ~2^-24 rad after reduction).
__device__ __forceinline__ void rope_pair(float& x0, float& x1, int pos, double freq) {
  // the angle and its reduction to [0, 2 pi) in double (a multiply by 1 / (2 pi)
  // instead of a divide: this part's double-precision rate is low)
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  double ang = (double)pos * freq;
  ang -= two_pi * floor(ang * inv_two_pi);
  float s, c;
  sincosf((float)ang, &s, &c);
  const float y0 = x0 * c - x1 * s;
  const float y1 = x1 * c + x0 * s;
  x0 = y0;
  x1 = y1;
}

// grid (M, nq + nkv), block dh/2 threads: thread i owns the pair (i, i + dh/2).
__device__ __forceinline__ float qkv_at(const QkvPostArgs& a, int m, int col) {
  const float* p = a.qkv + (size_t)m * a.ld + col;
  if (a.nsplit == 1) return p[0];
  float t[8];  // split-K partials (at most 8): all loads in flight, summed in split order
#pragma unroll
  for (int s = 0; s < 8; ++s) t[s] = s < a.nsplit ? p[(size_t)s * a.split_stride] : 0.f;
  float v = t[0];
#pragma unroll
  for (int s = 1; s < 8; ++s) v += t[s];
  return v;
}

__global__ void k_qkv_post(const __grid_constant__ QkvPostArgs a) {
  __shared__ float red[32];
  const int m = blockIdx.x, h = blockIdx.y + (a.q_off < 0 ? a.nq : 0), i = threadIdx.x, half = a.dh / 2;
  // the norm weights and the RoPE frequency are constants of the model: read
  // them before waiting for the GEMM that produced qkv
  const float* nw = h < a.nq ? a.wq : a.wk;
  const float w0 = nw[i], w1 = nw[i + half];
  const double freq = a.inv_freq[i];
  pdl_wait();
  pdl_trigger();
  const int slot = a.slot[m], row = a.row[m];
  if (h < a.nq) {
    const int qd = a.qdst[m];
    if (qd < 0 || a.q_off < 0) return;  // uniform across the block
    float x0 = qkv_at(a, m, a.q_off + h * a.dh + i), x1 = qkv_at(a, m, a.q_off + h * a.dh + i + half);
    const float ss = block_sum(x0 * x0 + x1 * x1, red);
    const float inv = rsqrtf(ss / (float)a.dh + a.eps);
    x0 = x0 * inv * w0;
    x1 = x1 * inv * w1;
    rope_pair(x0, x1, slot, freq);
    float* dst = a.q_out + (size_t)qd * a.nq * a.dh + h * a.dh;
    dst[i] = x0;
    dst[i + half] = x1;
  } else {
    const int g = h - a.nq;
    float x0 = qkv_at(a, m, a.k_off + g * a.dh + i), x1 = qkv_at(a, m, a.k_off + g * a.dh + i + half);
    const float ss = block_sum(x0 * x0 + x1 * x1, red);
    const float inv = rsqrtf(ss / (float)a.dh + a.eps);
    x0 = x0 * inv * w0;
    x1 = x1 * inv * w1;
    rope_pair(x0, x1, slot, freq);
    const size_t off = (((size_t)row * a.nkv + g) * a.cap + slot) * a.dh;
    store_elem(a.kc, a.wdt, off + i, x0);
    store_elem(a.kc, a.wdt, off + i + half, x1);
    store_elem(a.vc, a.wdt, off + i, qkv_at(a, m, a.v_off + g * a.dh + i));
    store_elem(a.vc, a.wdt, off + i + half, qkv_at(a, m, a.v_off + g * a.dh + i + half));
  }
}

// One block per (pair, half): half 0 = RMSNorm_e(E[tok]), half 1 =
// RMSNorm_h(hidden), written as bf16 into the pair's row of x. Each thread
// keeps its (at most two) 8-element vectors in registers between the sum of
// squares and the store, so the source row is read once.
__global__ void k_flush_x(const __grid_constant__ FlushXArgs a) {
  __shared__ float red[32];
  const int m = blockIdx.x, half = blockIdx.y, H = a.H, nv = H / 8;
  const float* w = half == 0 ? a.nw_e : a.nw_h;
  float4 wv[2][2];  // this thread's norm weights, read before the wait (constants of the model)
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    wv[u][0] = wv[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < nv) {
      wv[u][0] = reinterpret_cast<const float4*>(w)[2 * i];
      wv[u][1] = reinterpret_cast<const float4*>(w)[2 * i + 1];
    }
  }
  pdl_wait();
  pdl_trigger();
  size_t base;
  if (half == 0) {
    int t = a.tok[a.tok_idx[m]];
    if (t < 0 || t >= a.vocab) {
      if (threadIdx.x == 0) flag_status(a.status, MTP_ERR_BAD_ARG);
      t = 0;
    }
    base = (size_t)t * H;
  } else {
    base = (size_t)a.hid_item[m] * H;
  }
  const void* src = half == 0 ? a.E : a.hid;
  const int dt = half == 0 ? a.wdt : a.hid_dt;
  float f[2][8];
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    if (i < nv) {
      if (dt == MTP_DTYPE_BF16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(src) + base) + i);
        f[u][0] = bf16lo(v.x); f[u][1] = bf16hi(v.x); f[u][2] = bf16lo(v.y); f[u][3] = bf16hi(v.y);
        f[u][4] = bf16lo(v.z); f[u][5] = bf16hi(v.z); f[u][6] = bf16lo(v.w); f[u][7] = bf16hi(v.w);
      } else {
        const float4* p4 = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + base) + 2 * i;
        const float4 u0 = __ldg(p4), u1 = __ldg(p4 + 1);
        f[u][0] = u0.x; f[u][1] = u0.y; f[u][2] = u0.z; f[u][3] = u0.w;
        f[u][4] = u1.x; f[u][5] = u1.y; f[u][6] = u1.z; f[u][7] = u1.w;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(f[u][j], f[u][j], ss);
    }
  }
  const float inv = rsqrtf(block_sum(ss, red) / (float)H + a.eps);
  uint16_t* x = a.x + (size_t)m * 2 * H + (size_t)half * H;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    if (i < nv) {
      const float4 w0 = wv[u][0], w1 = wv[u][1];
      const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = (uint32_t)f_to_bf16(f[u][2 * j] * inv * ww[2 * j]) |
               ((uint32_t)f_to_bf16(f[u][2 * j + 1] * inv * ww[2 * j + 1]) << 16);
      reinterpret_cast<uint4*>(x)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Threads for a row of n vectors with at most `per` vectors per thread.
static int row_threads(int n, int per) {
  int t = (n + per - 1) / per;
  t = (t + 31) / 32 * 32;
  return t < 32 ? 32 : (t > 1024 ? 1024 : t);
}

void launch_flush_x(const FlushXArgs& a, int M, cudaStream_t s) {
  launch_pdl(k_flush_x, dim3(M, 2), dim3(row_threads(a.H / 8, 2)), 0, s, a);
  count_launch();
}

// b[m] = bf16(RMSNorm(sum of the split-K partials of row m) * w): one block per
// row, each thread holding at most four float4 of the summed row in registers.
__global__ void k_flush_norm(const float* part, int nsplit, long long split_stride, int H, const float* w,
                             float eps, uint16_t* b) {
  __shared__ float red[32];
  const int m = blockIdx.x, n4 = H / 4;
  float4 wv[4];  // this thread's norm weights, read before the wait (constants of the model)
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    wv[u] = i < n4 ? reinterpret_cast<const float4*>(w)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();
  pdl_trigger();
  const float* p = part + (size_t)m * H;
  float4 v[4];
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < n4) {
      for (int sidx = 0; sidx < nsplit; ++sidx) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(p + (size_t)sidx * split_stride) + i);
        acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
      }
    }
    v[u] = acc;
    ss += acc.x * acc.x + acc.y * acc.y + acc.z * acc.z + acc.w * acc.w;
  }
  const float inv = rsqrtf(block_sum(ss, red) / (float)H + eps);
  uint2* out = reinterpret_cast<uint2*>(b + (size_t)m * H);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    if (i < n4) {
      const float4 ww = wv[u];
      out[i] = make_uint2((uint32_t)f_to_bf16(v[u].x * inv * ww.x) | ((uint32_t)f_to_bf16(v[u].y * inv * ww.y) << 16),
                          (uint32_t)f_to_bf16(v[u].z * inv * ww.z) | ((uint32_t)f_to_bf16(v[u].w * inv * ww.w) << 16));
    }
  }
}

void launch_flush_norm(const float* part, int nsplit, long long split_stride, int M, int H, const float* w,
                       float eps, uint16_t* b, cudaStream_t s) {
  launch_pdl(k_flush_norm, dim3(M), dim3(row_threads(H / 4, 4)), 0, s, part, nsplit, split_stride, H, w, eps, b);
  count_launch();
}

void launch_qkv_post(const QkvPostArgs& a, cudaStream_t s) {
  // without q (flush) only the kv heads have work
  launch_pdl(k_qkv_post, dim3(a.M, (a.q_off < 0 ? 0 : a.nq) + a.nkv), dim3(a.dh / 2), 0, s, a);
  count_launch();
}

// ------------------------------------------------------- decode attention

// One block per (chunk of a.chunk slots, kv head, head item). Thread 0 streams
// the chunk's K and V rows (contiguous in the cache) through a ring of NS
// shared-memory stages of 64 slots with bulk asynchronous copies, so the next
// tiles load while the block computes the scores of the G query heads of the
// group against the current one, keeps an online softmax, and accumulates P.V
// with one thread per head dimension. Partials (o, running max, running sum)
// are merged by k_attn_merge.
template <int DH, typename KT>
struct AttnRing {
  static constexpr int TS = 64;
  static constexpr int kTileBytes = 2 * TS * DH * (int)sizeof(KT);
  static constexpr int NS = (200 * 1024) / kTileBytes >= 3 ? 3 : ((200 * 1024) / kTileBytes >= 2 ? 2 : 1);
};

template <int DH, int G, typename KT>
__global__ void __launch_bounds__(256) k_attn_chunk(const __grid_constant__ AttnArgs a) {
  constexpr int TS = AttnRing<DH, KT>::TS;
  constexpr int NS = AttnRing<DH, KT>::NS;
  constexpr int EPL = DH / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  KT* ks = reinterpret_cast<KT*>(smem);
  KT* vs = ks + NS * TS * DH;
  float* qs = reinterpret_cast<float*>(vs + NS * TS * DH);
  float* ps = qs + G * DH;          // [G][TS]
  float* st = ps + G * TS;          // [G][4]: running max, alpha, running sum
  uint64_t* bar = reinterpret_cast<uint64_t*>(st + 4 * 8);

  const int c = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
  const int L = a.slot[m] + 1;
  const int t0 = c * a.chunk;
  if (t0 >= L) return;
  const int n = min(a.chunk, L - t0);
  const int nt = (n + TS - 1) / TS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(smem_u32(&bar[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < G) { st[4 * tid] = -INFINITY; st[4 * tid + 1] = 0.f; st[4 * tid + 2] = 0.f; }
  __syncthreads();
  pdl_wait();  // the cache rows of this call's new slots come from k_qkv_post
  const size_t base = (((size_t)a.row[m] * a.nkv + g) * a.cap + t0) * DH;
  auto issue = [&](int i) {  // tile i into ring slot i % NS
    const int slot = i % NS;
    const int rows = min(TS, n - i * TS);
    const uint32_t bytes = (uint32_t)(rows * DH * sizeof(KT));
    mbar_expect_tx(smem_u32(&bar[slot]), 2 * bytes);
    bulk_g2s(smem_u32(ks + slot * TS * DH), reinterpret_cast<const KT*>(a.kc) + base + (size_t)i * TS * DH, bytes,
             smem_u32(&bar[slot]));
    bulk_g2s(smem_u32(vs + slot * TS * DH), reinterpret_cast<const KT*>(a.vc) + base + (size_t)i * TS * DH, bytes,
             smem_u32(&bar[slot]));
  };
  if (tid == 0)
    for (int i = 0; i < min(nt, NS); ++i) issue(i);
  pdl_trigger();
  const float* qg = a.q + (size_t)m * a.nq * DH + (size_t)g * G * DH;
  float qr[G][EPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < EPL; ++e) qr[h][e] = qg[h * DH + lane * EPL + e];

  float o[G];
#pragma unroll
  for (int h = 0; h < G; ++h) o[h] = 0.f;
  bool ok = true;
  int issued = min(nt, NS);
  for (int i = 0; i < nt; ++i) {
    const int rows = min(TS, n - i * TS);
    const int slot = i % NS;
    const bool got = mbar_wait(smem_u32(&bar[slot]), (i / NS) & 1);
    if (__syncthreads_or(!got)) { ok = false; break; }
    const KT* kt = ks + slot * TS * DH;
    const KT* vt = vs + slot * TS * DH;
    // scores: warp w takes keys KPW*w .. KPW*w + KPW-1 of the tile; lane owns
    // EPL dims of every key; the KPW keys x 8 head slots of partial dots are
    // reduced across the warp by a halving butterfly, leaving lane l with the
    // NF sums t = l*NF + u (u < NF) of key t/8, head slot t%8.
    {
      constexpr int KPW = TS / 8, NV = KPW * 8, NF = NV / 32;
      float v[NV];
      const int kb = warp * KPW;
#pragma unroll
      for (int kk = 0; kk < KPW; ++kk) {
        float kv[EPL];
        const int j = kb + kk < rows ? kb + kk : rows - 1;
        const KT* kr = kt + (size_t)j * DH + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e)
          kv[e] = sizeof(KT) == 2 ? bf16_to_f(((const uint16_t*)kr)[e]) : ((const float*)kr)[e];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          float d = 0.f;
          if (h < G) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) d = fmaf(qr[h][e], kv[e], d);
          }
          v[kk * 8 + h] = d;
        }
      }
#pragma unroll
      for (int o = 16, n = NV; o >= 1; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int t = 0; t < n / 2; ++t) {
          const float send = up ? v[t] : v[t + n / 2];
          const float keep = up ? v[t + n / 2] : v[t];
          v[t] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
      }
#pragma unroll
      for (int u = 0; u < NF; ++u) {
        const int t = lane * NF + u, key = kb + t / 8, h = t % 8;
        if (key < rows && h < G) ps[h * TS + key] = v[u] * a.scale;
      }
    }
    __syncthreads();
    // online softmax update: warp h owns query head h
    if (warp < G) {
      const int h = warp;
      float mx = -INFINITY;
      for (int j = lane; j < rows; j += 32) mx = fmaxf(mx, ps[h * TS + j]);
      mx = warp_max(mx);
      const float m_old = st[4 * h];
      const float m_new = fmaxf(m_old, mx);
      const float alpha = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
      float sum = 0.f;
      for (int j = lane; j < rows; j += 32) {
        const float e = expf(ps[h * TS + j] - m_new);
        ps[h * TS + j] = e;
        sum += e;
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        st[4 * h] = m_new;
        st[4 * h + 1] = alpha;
        st[4 * h + 2] = st[4 * h + 2] * alpha + sum;
      }
    }
    __syncthreads();
    for (int d = tid; d < DH; d += blockDim.x) {
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = o[h] * st[4 * h + 1];
      const KT* vr = vt + d;
      int j = 0;
      for (; j + 4 <= rows; j += 4) {
        float vv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          vv[u] = sizeof(KT) == 2 ? bf16_to_f(((const uint16_t*)vr)[(size_t)(j + u) * DH])
                                  : ((const float*)vr)[(size_t)(j + u) * DH];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 pp = *reinterpret_cast<const float4*>(ps + h * TS + j);
          acc[h] = fmaf(pp.x, vv[0], fmaf(pp.y, vv[1], fmaf(pp.z, vv[2], fmaf(pp.w, vv[3], acc[h]))));
        }
      }
      for (; j < rows; ++j) {
        const float v = sizeof(KT) == 2 ? bf16_to_f(((const uint16_t*)vr)[(size_t)j * DH]) : ((const float*)vr)[(size_t)j * DH];
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = fmaf(ps[h * TS + j], v, acc[h]);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) o[h] = acc[h];
    }
    __syncthreads();  // every thread is done with this slot: refill it
    if (tid == 0 && issued < nt) issue(issued);
    issued = min(nt, issued + 1);
  }
  if (!ok) {
    if (tid == 0) {
      flag_status(a.status, MTP_ERR_TIMEOUT);
      // let the copies in flight land before exit: the last tile issued into each slot
      for (int j = max(0, issued - NS); j < issued; ++j) mbar_wait(smem_u32(&bar[j % NS]), (j / NS) & 1);
    }
    return;
  }
  for (int d = tid; d < DH; d += blockDim.x) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const size_t hq = (size_t)m * a.nq + g * G + h;
      a.po[(hq * a.max_chunks + c) * DH + d] = o[h];
    }
  }
  if (tid < G) {
    const size_t hq = (size_t)m * a.nq + g * G + tid;
    a.pml[(hq * a.max_chunks + c) * 2 + 0] = st[4 * tid];
    a.pml[(hq * a.max_chunks + c) * 2 + 1] = st[4 * tid + 2];
  }
}

// grid (nq, Mh), block DH threads: merge the chunk partials of one query head.
template <int DH>
__global__ void k_attn_merge(const __grid_constant__ AttnArgs a) {
  extern __shared__ float wch[];  // per-chunk weight exp(m_c - M)
  __shared__ float red[32];
  const int h = blockIdx.x, m = blockIdx.y, d = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const int L = a.slot[m] + 1;
  const int nch = (L + a.chunk - 1) / a.chunk;
  const size_t hq = (size_t)m * a.nq + h;
  const float* ml = a.pml + hq * a.max_chunks * 2;
  float mx = -INFINITY;
  for (int c = d; c < nch; c += DH) mx = fmaxf(mx, ml[2 * c]);
  // block max through the sum helper's scratch: negate-free max reduction
  mx = warp_max(mx);
  if ((d & 31) == 0) red[d >> 5] = mx;
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < DH / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  float den = 0.f;
  for (int c = d; c < nch; c += DH) {
    const float w = expf(ml[2 * c] - M);
    wch[c] = w;
    den = fmaf(ml[2 * c + 1], w, den);
  }
  den = block_sum(den, red);
  const float* po = a.po + hq * a.max_chunks * DH + d;
  float num = 0.f;
  int c = 0;
  for (; c + 16 <= nch; c += 16) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) v[u] = po[(size_t)(c + u) * DH];
#pragma unroll
    for (int u = 0; u < 16; ++u) num = fmaf(v[u], wch[c + u], num);
  }
  for (; c < nch; ++c) num = fmaf(po[(size_t)c * DH], wch[c], num);
  a.o[(size_t)m * a.nq * DH + (size_t)h * DH + d] = num / den;
}

template <int DH, int G, typename KT>
static void attn_t(const AttnArgs& a0, int sms, cudaStream_t s) {
  constexpr int TS = AttnRing<DH, KT>::TS, NS = AttnRing<DH, KT>::NS;
  const size_t smem = 2 * (size_t)NS * TS * DH * sizeof(KT) + (size_t)(G * DH + G * TS + 32) * sizeof(float) + 64;
  auto k = k_attn_chunk<DH, G, KT>;
  // blocks of this instance resident on one SM, looked up once per device
  static std::mutex mu;
  static int resident[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  int per_sm;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (resident[dev] <= 0) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      int nb = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, 256, smem) != cudaSuccess || nb < 1) nb = 1;
      cudaGetLastError();
      resident[dev] = nb;
    }
    per_sm = resident[dev];
  }
  AttnArgs a = a0;
  a.chunk = attn_chunk_slots(a, (long long)per_sm * sms);
  int maxL = 0;
  for (int m = 0; m < a.Mh; ++m) maxL = max(maxL, a.slot[m] + 1);
  const int nch = (maxL + a.chunk - 1) / a.chunk;
  launch_pdl(k, dim3(nch, a.nkv, a.Mh), dim3(256), smem, s, a);
  count_launch();
  launch_attn_merge(a, s);
}

// Slots per block: the smallest whole number of 64-slot units (never below
// kAttnChunk, the partial buffers' unit) whose blocks all fit one wave of the
// resident blocks; a wave more would cost a whole block's time for a few.
int attn_chunk_slots(const AttnArgs& a, long long slots) {
  long long total = 0;
  int maxL = 0;
  for (int m = 0; m < a.Mh; ++m) {
    total += a.slot[m] + 1;
    maxL = max(maxL, a.slot[m] + 1);
  }
  auto blocks = [&](int chunk) {
    long long b = 0;
    for (int m = 0; m < a.Mh; ++m) b += (a.slot[m] + chunk) / chunk;
    return b * a.nkv;
  };
  int chunk = (int)(((total * a.nkv + slots - 1) / slots + 63) / 64 * 64);
  if (chunk < kAttnChunk) chunk = kAttnChunk;
  while (chunk < maxL && blocks(chunk) > slots) chunk += 64;
  return chunk;
}

void launch_attn_merge(const AttnArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)a.max_chunks * sizeof(float);
  if (a.dh == 256) launch_pdl(k_attn_merge<256>, dim3(a.nq, a.Mh), dim3(256), smem, s, a);
  else if (a.dh == 128) launch_pdl(k_attn_merge<128>, dim3(a.nq, a.Mh), dim3(128), smem, s, a);
  else launch_pdl(k_attn_merge<64>, dim3(a.nq, a.Mh), dim3(64), smem, s, a);
  count_launch();
}

void launch_attention(const AttnArgs& a, int sms, cudaStream_t s) {
  if (launch_attention_mma(a, sms, s)) return;
  const int G = a.nq / a.nkv;
  const bool bf = a.wdt == MTP_DTYPE_BF16;
#define MTP_ATTN_CASE(DHV, GV)                                                \
  if (a.dh == DHV && G == GV) {                                               \
    if (bf) attn_t<DHV, GV, uint16_t>(a, sms, s); else attn_t<DHV, GV, float>(a, sms, s); \
    return;                                                                   \
  }
  MTP_ATTN_CASE(256, 6)
  MTP_ATTN_CASE(256, 1)
  MTP_ATTN_CASE(256, 2)
  MTP_ATTN_CASE(256, 4)
  MTP_ATTN_CASE(256, 8)
  MTP_ATTN_CASE(128, 1)
  MTP_ATTN_CASE(128, 2)
  MTP_ATTN_CASE(128, 4)
  MTP_ATTN_CASE(128, 6)
  MTP_ATTN_CASE(128, 8)
  MTP_ATTN_CASE(64, 1)
  MTP_ATTN_CASE(64, 2)
  MTP_ATTN_CASE(64, 4)
  MTP_ATTN_CASE(64, 8)
#undef MTP_ATTN_CASE
}

// ------------------------------------------------------------ small kernels

__global__ void k_norm_copy(const void* src, int dt, int n, float shift, float* dst) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = load_elem(src, dt, i) + shift;
}

void launch_norm_copy(const void* src, int dt, int n, float shift, float* dst, cudaStream_t s) {
  k_norm_copy<<<(n + 255) / 256, 256, 0, s>>>(src, dt, n, shift, dst);
  count_launch();
}

// grid (rows, nkv): set lengths, trim target lengths, zero dropped slots.
__global__ void k_rollback(const __grid_constant__ RollbackArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, g = blockIdx.y;
  if (a.keep[r] < 0) return;
  if (g == 0 && threadIdx.x == 0) {
    a.len[r] = a.keep[r];
    if (a.target_len && a.n_acc) a.target_len[r] -= a.block - (a.n_acc[r] + 1);
  }
  if (!a.zero_tail || a.old_len[r] <= a.keep[r]) return;
  const size_t off = (((size_t)r * a.nkv + g) * a.cap + a.keep[r]) * a.dh * a.esize;
  const size_t bytes = (size_t)(a.old_len[r] - a.keep[r]) * a.dh * a.esize;
  unsigned char* kp = reinterpret_cast<unsigned char*>(a.kc) + off;
  unsigned char* vp = reinterpret_cast<unsigned char*>(a.vc) + off;
  for (size_t b = threadIdx.x; b < bytes; b += blockDim.x) { kp[b] = 0; vp[b] = 0; }
}

void launch_rollback(const RollbackArgs& a, cudaStream_t s) {
  launch_pdl(k_rollback, dim3(a.rows, a.nkv), dim3(256), 0, s, a);
  count_launch();
}

struct LenArgs {
  int32_t* len;
  int rows;
  int v[kMaxRows];
};
__global__ void k_set_len(const __grid_constant__ LenArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = threadIdx.x;
  if (r < a.rows) a.len[r] = a.v[r];
}

void launch_set_len(int32_t* len, int rows, const int* h_len, cudaStream_t s) {
  LenArgs a;
  a.len = len;
  a.rows = rows;
  for (int r = 0; r < rows; ++r) a.v[r] = h_len[r];
  launch_pdl(k_set_len, dim3(1), dim3(kMaxRows), 0, s, a);
  count_launch();
}

}  // namespace mtp
