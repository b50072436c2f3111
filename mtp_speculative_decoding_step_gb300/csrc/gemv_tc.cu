// Batched GEMV on the 5th-generation tensor cores, for head calls that carry
// several items (rows of a batch, or pending pairs): y[m][n] = sum_k W[n][k]
// x[m][k] over the head's weight matrices ("Upstream contract to port": the
// fc, q/k/v, o, gate/up, down and tied lm_head projections of one MTP step).
//
// With more than a few items the CUDA-core GEMV runs out of FMA issue slots
// before it runs out of HBM bandwidth (eight fp32 FMAs per bf16 weight). Here
// the weights are the MMA's A operand: every CTA streams 128 weight rows by
// 64-column K tiles through TMA into shared memory and one thread issues
// tcgen05.mma of M 128 x N NI x K 16, so the tensor cores do the FMAs and the
// kernel is bound by the weight stream alone.
//
// Activations keep (close to) fp32 precision: each item's fp32 row x is
// carried as two bf16 rows, x_hi = bf16(x) and x_lo = bf16(x - x_hi), so the
// B operand holds NI = 2 * MI rows (MI items padded to a multiple of 8). Both
// products are exact in the fp32 accumulator and the epilogue adds the two
// columns; x_hi + x_lo carries 16 significant bits. The hi/lo pair costs
// nothing extra: M 128 needs N >= 16 anyway.
//
//   k_tcx_prep  : prologue (plain / RMSNorm / embedding+hidden dual norm) and
//                 the hi/lo split into X2[NI][K] (bf16, K-major)
//   k_tc_gemv   : warp 0 lane 0 = TMA producer, warp 1 lane 0 = MMA issuer,
//                 4 warps = epilogue (TMEM -> registers -> fp32 partials);
//                 split-K CTAs write partials [split][item][row]; with one
//                 split a store or logits job is written in place, and the
//                 logits epilogue (q cleared, each tile's argmax) runs here
//   k_tcv_finish / k_tcv_logits: sum the splits in split order and apply
//                 the epilogue (store, residual, SwiGLU, logits + two-level
//                 argmax)
//   k_tcv_argmax: after the in-place logits epilogue, the per-item argmax
//                 over the tiles' pairs
// Every mbarrier wait is bounded; on expiry the CTA raises the status word,
// waits (bounded) for its own copies, frees its TMEM and returns.
#include "kernels.h"
#include "tc_common.cuh"

namespace mtp {

using namespace tc;

// ------------------------------------------------------------ prologue

__device__ __forceinline__ void split_store8(const float* v, uint16_t* hi, uint16_t* lo, int i) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint16_t h0 = f_to_bf16(v[2 * j]), h1 = f_to_bf16(v[2 * j + 1]);
    const uint16_t l0 = f_to_bf16(v[2 * j] - bf16_to_f(h0)), l1 = f_to_bf16(v[2 * j + 1] - bf16_to_f(h1));
    h[j] = (uint32_t)h0 | ((uint32_t)h1 << 16);
    l[j] = (uint32_t)l0 | ((uint32_t)l1 << 16);
  }
  reinterpret_cast<uint4*>(hi)[i] = make_uint4(h[0], h[1], h[2], h[3]);
  reinterpret_cast<uint4*>(lo)[i] = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void load8(const void* src, int dt, size_t base, int i, float* f) {
  if (dt == MTP_DTYPE_BF16) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(src) + base) + i);
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
  } else {
    const float4* p4 = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + base) + 2 * i;
    const float4 u0 = __ldg(p4), u1 = __ldg(p4 + 1);
    f[0] = u0.x; f[1] = u0.y; f[2] = u0.z; f[3] = u0.w; f[4] = u1.x; f[5] = u1.y; f[6] = u1.z; f[7] = u1.w;
  }
}

// grid (MI, parts), parts = 2 for the dual prologue (embedding half, hidden
// half) else 1. Items m >= M write zero rows.
__global__ void k_tcx_prep(const __grid_constant__ TcxPrepArgs a) {
  __shared__ float red[32];
  const int m = blockIdx.x, part = blockIdx.y;
  // the norm weights are constants of the head: this thread's two vectors of
  // them are loaded before waiting for the previous kernel
  const float* wpre = a.pro == PRO_DUAL ? (part == 0 ? a.nw : a.nw2) : (a.pro == PRO_NORM ? a.nw : nullptr);
  float4 wv[2][2];
  if (wpre && m < a.M) {
    const int nv0 = (a.pro == PRO_DUAL ? a.K / 2 : a.K) / 8;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = threadIdx.x + u * blockDim.x;
      if (i < nv0) {
        wv[u][0] = __ldg(reinterpret_cast<const float4*>(wpre) + 2 * i);
        wv[u][1] = __ldg(reinterpret_cast<const float4*>(wpre) + 2 * i + 1);
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  const int L = a.pro == PRO_DUAL ? a.K / 2 : a.K;
  const int k0 = part * L, nv = L / 8;
  uint16_t* hi = a.X2 + (size_t)m * a.K + k0;
  uint16_t* lo = a.X2 + (size_t)(a.MI + m) * a.K + k0;
  if (m >= a.M) {
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
      reinterpret_cast<uint4*>(hi)[i] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(lo)[i] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const void* src;
  int dt;
  size_t base;
  const float* w;
  if (a.pro == PRO_DUAL) {
    if (part == 0) {
      int t = a.tok[a.tok_idx[m]];
      if (t < 0 || t >= a.vocab) {  // a bad token id reads row 0 and raises the status word
        if (threadIdx.x == 0) flag_status(a.status, MTP_ERR_BAD_ARG);
        t = 0;
      }
      src = a.E; dt = a.wdt; base = (size_t)t * L; w = a.nw;
    } else {
      src = a.hid; dt = a.hid_dt; base = (size_t)a.hid_off[m]; w = a.nw2;
    }
  } else {
    src = a.x + (size_t)m * a.ldx; dt = MTP_DTYPE_F32; base = 0;
    w = a.pro == PRO_NORM ? a.nw : nullptr;
  }
  if (!w) {
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
      float f[8];
      load8(src, dt, base, i, f);
      split_store8(f, hi, lo, i);
    }
    return;
  }
  // normalised rows: at most two vectors per thread, held across the sum
  float f[2][8];
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    if (i < nv) {
      load8(src, dt, base, i, f[u]);
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(f[u][j], f[u][j], ss);
    }
  }
  const float inv = rsqrtf(block_sum(ss, red) / (float)L + a.eps);
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    if (i < nv) {
      const float4 w0 = wv[u][0], w1 = wv[u][1];
      const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = f[u][j] * inv * ww[j];
      split_store8(v, hi, lo, i);
    }
  }
}

static int prep_threads(int nv, bool hold) {
  int t = hold ? (nv + 1) / 2 : nv;
  t = (t + 31) / 32 * 32;
  return t < 32 ? 32 : (t > 1024 ? 1024 : t);
}

void launch_tcx_prep(const TcxPrepArgs& a, cudaStream_t s) {
  const bool dual = a.pro == PRO_DUAL;
  const int L = dual ? a.K / 2 : a.K;
  launch_pdl(k_tcx_prep, dim3(a.MI, dual ? 2 : 1), dim3(prep_threads(L / 8, a.pro != PRO_PLAIN)), 0, s, a);
  count_launch();
}

// ------------------------------------------------------------ contraction

struct TcGemvArgs {
  int N, K, ksplit, M, swiglu;
  int seg_end[3];
  float* out;  // out[split * ld_split + item * ld_item + row]
  long long ld_item, ld_split;
  int32_t* status;
  // fused logits epilogue (one split, out = the logits): item m's draft
  // distribution row cleared (or null) and the tile's (max, index) of each
  // item at gmax / gidx[m * tiles + tile]
  int fuse_logits;
  float* qzero;
  long long ldqz;
  float* gmax;
  int* gidx;
};

template <int NI, int STAGES>
__global__ void __launch_bounds__(128) k_tc_gemv(const __grid_constant__ CUtensorMap w0,
                                                 const __grid_constant__ CUtensorMap w1,
                                                 const __grid_constant__ CUtensorMap w2,
                                                 const __grid_constant__ CUtensorMap xm, const TcGemvArgs a) {
  constexpr int MI = NI / 2;
  constexpr uint32_t kABytes = kTileM * kTileK * 2;
  constexpr uint32_t kBBytes = NI * kTileK * 2;
  constexpr uint32_t kStage = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = NI <= 32 ? 32 : (NI <= 64 ? 64 : (NI <= 128 ? 128 : 256));
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + STAGES * kStage);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int v0 = tile * kTileM;
  const int nk_total = a.K / kTileK;
  const int per = (nk_total + a.ksplit - 1) / a.ksplit;
  const int kb = split * per;
  const int nk = min(per, nk_total - kb);

  // weight rows of this tile: one map (a segment of the virtual row space), or
  // 64 gate rows then the matching 64 up rows
  const CUtensorMap* wa = &w0;
  int ra = v0;
  if (!a.swiglu) {
    int sg = 0, start = 0;
    while (sg < 2 && v0 >= a.seg_end[sg]) { start = a.seg_end[sg]; ++sg; }
    wa = sg == 0 ? &w0 : (sg == 1 ? &w1 : &w2);
    ra = v0 - start;
  }

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
    auto load_a = [&](int s, int i) {
      uint8_t* as = base + s * kStage;
      const int x = (kb + i) * kTileK;
      if (a.swiglu) {
        tma_load_2d(smem_u32(as), &w0, x, tile * (kTileM / 2), smem_u32(&full[s]));
        tma_load_2d(smem_u32(as + kABytes / 2), &w1, x, tile * (kTileM / 2), smem_u32(&full[s]));
      } else {
        tma_load_2d(smem_u32(as), wa, x, ra, smem_u32(&full[s]));
      }
    };
    auto load_b = [&](int s, int i) {
      tma_load_2d(smem_u32(base + s * kStage + kABytes), &xm, (kb + i) * kTileK, 0, smem_u32(&full[s]));
    };
    // the weights do not depend on the previous kernel: start their stream
    // before waiting for the activations
    const int pre = min(nk, STAGES);
    for (int i = 0; i < pre; ++i) {
      mbar_expect_tx(smem_u32(&full[i]), kStage);
      load_a(i, i);
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i) load_b(i, i);
    for (int i = pre; i < nk; ++i) {
      const int s = i % STAGES, r = i / STAGES;
      if (!mbar_wait(smem_u32(&empty[s]), (r - 1) & 1)) { *s_fail = 1; break; }
      mbar_expect_tx(smem_u32(&full[s]), kStage);
      load_a(s, i);
      load_b(s, i);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16(kTileM, NI);
    bool ok = true;
    for (int i = 0; i < nk && ok; ++i) {
      const int s = i % STAGES, r = i / STAGES;
      if (!mbar_wait(smem_u32(&full[s]), r & 1)) { ok = false; break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t as = smem_u32(base + s * kStage), bs = as + kABytes;
#pragma unroll
      for (int kk = 0; kk < kTileK / 16; ++kk)
        mma_bf16(tmem, sdesc(as + kk * 32), sdesc(bs + kk * 32), idesc, (i > 0 || kk > 0) ? 1u : 0u);
      mma_commit(smem_u32(&empty[s]));
    }
    if (!ok) *s_fail = 1;
    mma_commit(smem_u32(accf));
  }
  __syncwarp();

  // epilogue: TMEM lane 32w + l holds virtual row v0 + 32w + l; column c < MI
  // is item c's x_hi product, column MI + c its x_lo product
  __shared__ float s_bv[4][MI];
  __shared__ int s_bi[4][MI];
  pdl_wait();
  // warp-uniform: the TMEM loads and the argmax shuffles are warp-wide
  const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(accf), 0));
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  pdl_trigger();
  bool bad = false;
  if (got) {
    const int row = v0 + warp * 32 + lane;
    float* o = a.out + (size_t)split * a.ld_split + row;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c = 0; c < MI; c += 8) {
      float hv[8], lv[8];
      tmem_ld8(tl + (uint32_t)c, hv);
      tmem_ld8(tl + (uint32_t)(MI + c), lv);
      if (a.fuse_logits) {
        // the logit (+0: a lone split's sum, as the split combine forms it),
        // the cleared q entry, and the warp's (max, lowest index) per item
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int m = c + j;
          if (m < a.M) {
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF;
            if (row < a.N) {
              const float x = hv[j] + lv[j] + 0.f;
              o[(size_t)m * a.ld_item] = x;
              if (a.qzero) a.qzero[(size_t)m * a.ldqz + row] = 0.f;
              bad |= !isfinite(x);
              bv = x;
              bi = row;
            }
            warp_argmax(bv, bi);
            if (lane == 0) { s_bv[warp][m] = bv; s_bi[warp][m] = bi; }
          }
        }
      } else if (row < a.N) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c + j < a.M) o[(size_t)(c + j) * a.ld_item] = hv[j] + lv[j];
      }
    }
  }
  if (bad) flag_status(a.status, MTP_ERR_NONFINITE);
  const bool all_got = __syncthreads_and(got);
  if (a.fuse_logits && threadIdx.x < a.M) {
    // the tile's pair per item; an index in range even when nothing compares
    const int m = threadIdx.x;
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    if (all_got)
      for (int w = 0; w < 4; ++w)
        if (better(s_bv[w][m], s_bi[w][m], bv, bi)) { bv = s_bv[w][m]; bi = s_bi[w][m]; }
    if (bi == 0x7FFFFFFF) bi = min(v0, a.N - 1);
    a.gmax[(size_t)m * gridDim.x + tile] = bv;
    a.gidx[(size_t)m * gridDim.x + tile] = bi;
  }
  if (threadIdx.x == 0 && (!all_got || *s_fail)) {
    flag_status(a.status, MTP_ERR_TIMEOUT);
    for (int s = 0; s < STAGES; ++s) mbar_wait(smem_u32(&full[s]), 0);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int NI, int STAGES>
constexpr int tc_gemv_smem() { return STAGES * (kTileM + NI) * kTileK * 2 + 1024 + 256; }

// the stage counts of launch_tc_gemv's instances
constexpr int kTcvSmem16 = tc_gemv_smem<16, 6>(), kTcvSmem32 = tc_gemv_smem<32, 6>(),
              kTcvSmem64 = tc_gemv_smem<64, 5>(), kTcvSmem128 = tc_gemv_smem<128, 4>();

// From the shared memory alone (228 KB per SM, 1 KB of it reserved per
// resident CTA; 128 threads and 32 TMEM columns per CTA are never the limit):
// two CTAs at 8 items, one above. (Splits chosen from the occupancy query's
// count instead ran the 8-row draft step at 532 us against 513 us.)
int tc_gemv_blocks_per_sm(int NI) {
  const int smem = NI <= 16 ? kTcvSmem16 : (NI <= 32 ? kTcvSmem32 : (NI <= 64 ? kTcvSmem64 : kTcvSmem128));
  const int n = (228 * 1024) / (smem + 1024);
  return n > 1 ? n : 1;
}

template <int NI, int STAGES>
static bool tc_gemv_t(const TcGemvLaunch& L, const TcGemvArgs& a, cudaStream_t s) {
  CUtensorMap wm[3], xm;
  const int box_rows = L.swiglu ? kTileM / 2 : kTileM;
  for (int i = 0; i < 3; ++i) {
    const int i2 = i < L.nmaps ? i : L.nmaps - 1;
    if (!make_map(&wm[i], L.w[i2], L.rows[i2], L.K, box_rows)) return false;
  }
  if (!make_map(&xm, L.X2, NI, L.K, NI)) return false;
  const int smem = tc_gemv_smem<NI, STAGES>();
  auto k = k_tc_gemv<NI, STAGES>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((L.N + kTileM - 1) / kTileM, L.ksplit);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, wm[0], wm[1], wm[2], xm, a);
  count_launch();
  return e == cudaSuccess;
}

bool launch_tc_gemv(const TcGemvLaunch& L, cudaStream_t s) {
  if (L.K % kTileK != 0 || L.M < 1 || L.M > L.NI / 2 || L.ksplit < 1 || L.nmaps < 1 || L.nmaps > 3) return false;
  if (L.swiglu && (L.N % kTileM != 0 || L.nmaps != 2)) return false;
  TcGemvArgs a;
  a.N = L.N; a.K = L.K; a.ksplit = L.ksplit; a.M = L.M; a.swiglu = L.swiglu;
  for (int i = 0; i < 3; ++i) a.seg_end[i] = L.seg_end[i];
  a.out = L.out; a.ld_item = L.ld_item; a.ld_split = L.ld_split; a.status = L.status;
  a.fuse_logits = L.fuse_logits && L.ksplit == 1 && !L.swiglu ? 1 : 0;
  a.qzero = L.qzero; a.ldqz = L.ldqz; a.gmax = L.gmax; a.gidx = L.gidx;
  if (a.fuse_logits && (!a.gmax || !a.gidx)) return false;
  switch (L.NI) {
    case 16: return tc_gemv_t<16, 6>(L, a, s);
    case 32: return tc_gemv_t<32, 6>(L, a, s);
    case 64: return tc_gemv_t<64, 5>(L, a, s);
    case 128: return tc_gemv_t<128, 4>(L, a, s);
    default: return false;
  }
}

// ------------------------------------------------------------ epilogue

// grid (ceil(nout / 256), M), block 256: thread t of block (x, m) owns output
// o = 256 x + t of item m (store, residual and SwiGLU epilogues).
__global__ void __launch_bounds__(256) k_tcv_finish(const __grid_constant__ TcFinishArgs a) {
  const int tid = threadIdx.x;
  const int m = blockIdx.y, o = blockIdx.x * 256 + tid;
  // the residual stream was written several kernels back: read it before the wait
  const float rv = (a.epi == EPI_RESID && o < a.nout) ? a.resid[(size_t)m * a.ldr + o] : 0.f;
  pdl_wait();
  pdl_trigger();
  const float* p = a.part + (size_t)m * a.ld_item;
  if (o >= a.nout) return;
  float v;
  if (a.epi == EPI_SWIGLU) {
    const size_t r = (size_t)(o >> 6) * 128 + (o & 63);
    // every split's partial in flight at once (tcv_splits makes at most 8), summed in split order
    float gs[8], us[8];
#pragma unroll
    for (int sp = 0; sp < 8; ++sp) {
      gs[sp] = sp < a.ksplit ? __ldcg(p + (size_t)sp * a.ld_split + r) : 0.f;
      us[sp] = sp < a.ksplit ? __ldcg(p + (size_t)sp * a.ld_split + r + 64) : 0.f;
    }
    float g = 0.f, up = 0.f;
#pragma unroll
    for (int sp = 0; sp < 8; ++sp) {
      g += gs[sp];
      up += us[sp];
    }
    v = g / (1.f + expf(-g)) * up;
  } else {
    float ps[8];
#pragma unroll
    for (int sp = 0; sp < 8; ++sp) ps[sp] = sp < a.ksplit ? __ldcg(p + (size_t)sp * a.ld_split + o) : 0.f;
    v = 0.f;
#pragma unroll
    for (int sp = 0; sp < 8; ++sp) v += ps[sp];
    v += rv;
  }
  if (a.write_y) a.y[(size_t)m * a.ldy + o] = v;
}

// Logits epilogue: grid ceil(nout / 256), block 256. Block x takes outputs
// o = 256 x + t of every item (split partials summed in split order, or the
// logits the contraction wrote directly), its argmax per item, and the last
// block to finish reduces each item's blocks into its token. One counter
// update per block, not per (block, item): the single counter is the one
// address every block of the launch updates.
__global__ void __launch_bounds__(256) k_tcv_logits(const __grid_constant__ TcFinishArgs a) {
  __shared__ float sv[8];
  __shared__ int si[8];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int o = blockIdx.x * 256 + tid, ng = (int)gridDim.x;
  pdl_wait();
  pdl_trigger();
  for (int m = 0; m < a.M; ++m) {
    const float* p = a.part + (size_t)m * a.ld_item;
    float v = -INFINITY;
    if (o < a.nout) {
      float ps[8];
#pragma unroll
      for (int sp = 0; sp < 8; ++sp) ps[sp] = sp < a.ksplit ? __ldcg(p + (size_t)sp * a.ld_split + o) : 0.f;
      v = 0.f;
#pragma unroll
      for (int sp = 0; sp < 8; ++sp) v += ps[sp];
      if (a.write_y) a.y[(size_t)m * a.ldy + o] = v;
      if (!isfinite(v)) flag_status(a.status, MTP_ERR_NONFINITE);
      if (a.qzero) a.qzero[(size_t)m * a.ldqz + o] = 0.f;
    }
    float bv = o < a.nout ? v : -INFINITY;
    int bi = o < a.nout ? o : 0x7FFFFFFF;
    warp_argmax(bv, bi);
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
    __syncthreads();
    if (warp == 0) {
      bv = lane < 8 ? sv[lane] : -INFINITY;
      bi = lane < 8 ? si[lane] : 0x7FFFFFFF;
      warp_argmax(bv, bi);
      if (lane == 0) {
        a.gmax[(size_t)m * ng + blockIdx.x] = bv;
        a.gidx[(size_t)m * ng + blockIdx.x] = bi;
      }
    }
    __syncthreads();  // sv and si are reused by the next item
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.done, 1) == ng - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // one warp per item, eight loads in flight per lane: this runs once per
  // launch, at its end, on the path to the next kernel
  for (int mm = warp; mm < a.M; mm += 8) {
    float cv = -INFINITY;
    int ci = 0x7FFFFFFF;
    for (int g0 = lane; g0 < ng; g0 += 8 * 32) {
      float x[8];
      int ix[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int g = g0 + 32 * u;
        x[u] = g < ng ? __ldcg(&a.gmax[(size_t)mm * ng + g]) : -INFINITY;
        ix[u] = g < ng ? __ldcg(&a.gidx[(size_t)mm * ng + g]) : 0x7FFFFFFF;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (better(x[u], ix[u], cv, ci)) { cv = x[u]; ci = ix[u]; }
    }
    warp_argmax(cv, ci);
    // an item whose logits are all NaN (flagged above) still gets a token in range
    if (lane == 0 && a.amax_out) a.amax_out[a.amax_idx[mm]] = ci == 0x7FFFFFFF ? 0 : ci;
  }
  if (tid == 0) *a.done = 0;
}

// The launch-wide argmax after the fused logits epilogue: one warp per item
// over its per-tile (max, index) pairs (a.nout of them), eight loads in
// flight per lane; a launch of one block.
__global__ void __launch_bounds__(256) k_tcv_argmax(const __grid_constant__ TcFinishArgs a) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, ng = a.nout;
  for (int mm = warp; mm < a.M; mm += 8) {
    float cv = -INFINITY;
    int ci = 0x7FFFFFFF;
    for (int g0 = lane; g0 < ng; g0 += 8 * 32) {
      float x[8];
      int ix[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int g = g0 + 32 * u;
        x[u] = g < ng ? __ldcg(&a.gmax[(size_t)mm * ng + g]) : -INFINITY;
        ix[u] = g < ng ? __ldcg(&a.gidx[(size_t)mm * ng + g]) : 0x7FFFFFFF;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (better(x[u], ix[u], cv, ci)) { cv = x[u]; ci = ix[u]; }
    }
    warp_argmax(cv, ci);
    if (lane == 0 && a.amax_out) a.amax_out[a.amax_idx[mm]] = ci == 0x7FFFFFFF ? 0 : ci;
  }
}

void launch_tcv_argmax(const TcFinishArgs& a, cudaStream_t s) {
  launch_pdl(k_tcv_argmax, dim3(1), dim3(256), 0, s, a);
  count_launch();
}

void launch_tcv_finish(const TcFinishArgs& a, cudaStream_t s) {
  if (a.epi == EPI_LOGITS)
    launch_pdl(k_tcv_logits, dim3((a.nout + 255) / 256), dim3(256), 0, s, a);
  else
    launch_pdl(k_tcv_finish, dim3((a.nout + 255) / 256, a.M), dim3(256), 0, s, a);
  count_launch();
}

}  // namespace mtp
