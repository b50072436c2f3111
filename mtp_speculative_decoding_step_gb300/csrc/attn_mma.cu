// Decode attention on the tensor cores (bf16 K/V cache, head dim 128 or 256,
// up to 8 query heads per KV head).
//
// One block (8 warps) per (chunk of slots, KV head, head item), as in the
// CUDA-core kernel, with the same partial outputs (o, running max, running
// sum per query head) for k_attn_merge. Per tile of 64 slots:
//   S = Q K^T   rows 0-7 of the A operand hold the G query heads rounded to
//               bf16, rows 8-15 the bf16 rounding of what that left over, so
//               one m16n8k16 MMA gives both halves of every score (their sum
//               carries q to about 16 significant bits; K is bf16 already and
//               every product is exact). Each warp takes DH/8 of the head
//               dimensions for all 64 slots; the 8 partial score tiles are
//               summed through shared memory.
//   softmax     warp h < G: the online update of head h (running max and sum
//               in fp32), P written back as bf16 rows h (P rounded) and h + 8
//               (what the rounding left over).
//   O += P V    each warp owns DH/8 output dimensions; rows 0-7 and 8-15 of
//               its accumulators add up to the head's P V.
// K and V tiles stream from the cache into a ring of three stages with 16-byte
// asynchronous copies (cp.async), each 16-byte chunk of a slot's row placed at
// chunk ^ (slot & 7), so that the 8-row matrix loads (ldmatrix) that feed the
// MMAs hit 8 different bank groups.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

namespace {

constexpr int kMmaTS = 64;       // slots per tile
constexpr int kMmaNS = 3;        // ring stages
constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kSStride = kMmaTS + 8;  // floats per row of the partial-score tiles

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi); two values per call,
// packed low element first.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const uint16_t h0 = f_to_bf16(x0), h1 = f_to_bf16(x1);
  const uint16_t l0 = f_to_bf16(x0 - bf16_to_f(h0)), l1 = f_to_bf16(x1 - bf16_to_f(h1));
  hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
  lo = (uint32_t)l0 | ((uint32_t)l1 << 16);
}

template <int DH>
struct MmaLayout {
  static constexpr int RB = DH * 2;                 // bytes per slot row (bf16)
  static constexpr int TILE = kMmaTS * RB;          // one K (or V) tile
  static constexpr size_t K = 0;                    // ring: K tiles then V tiles
  static constexpr size_t V = (size_t)kMmaNS * TILE;
  static constexpr size_t S = 2 * (size_t)kMmaNS * TILE;            // [warps][8][kSStride] fp32
  static constexpr size_t P = S + (size_t)kMmaWarps * 8 * kSStride * 4;  // [16][64] bf16, swizzled
  static constexpr size_t ST = P + 16 * kMmaTS * 2;                 // [8][4] fp32 stats
  static constexpr size_t TOTAL = ST + 8 * 4 * 4;
};

// Byte offset of 16-byte chunk c of row r in a tile of rows of rb bytes.
__device__ __forceinline__ uint32_t swz(int r, int c, int rb) { return (uint32_t)(r * rb + ((c ^ (r & 7)) << 4)); }

template <int DH>
__global__ void __launch_bounds__(kMmaThreads, 1) k_attn_mma(const __grid_constant__ AttnArgs a) {
  using Lay = MmaLayout<DH>;
  constexpr int RB = Lay::RB, CH = RB / 16;  // chunks per row
  constexpr int DW = DH / kMmaWarps;         // head dimensions per warp
  constexpr int KSW = DW / 16;               // score k-steps per warp
  constexpr int NB2 = DW / 8;                // output n-blocks per warp
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  float* sS = reinterpret_cast<float*>(smem + Lay::S);
  uint16_t* sP = reinterpret_cast<uint16_t*>(smem + Lay::P);
  float* st = reinterpret_cast<float*>(smem + Lay::ST);  // per head: running max, alpha, running sum

  const int c = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
  const int L = a.slot[m] + 1;
  const int t0 = c * a.chunk;
  if (t0 >= L) return;
  const int n = min(a.chunk, L - t0);
  const int nt = (n + kMmaTS - 1) / kMmaTS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.nq / a.nkv;
  const int gr = lane >> 2, gc = lane & 3;  // fragment row group and column pair

  for (int i = tid; i < 16 * kMmaTS / 2; i += kMmaThreads) reinterpret_cast<uint32_t*>(sP)[i] = 0u;
  if (tid < 8) {
    st[4 * tid] = -INFINITY;
    st[4 * tid + 1] = 0.f;
    st[4 * tid + 2] = 0.f;
  }
  const size_t base = ((size_t)a.row[m] * a.nkv + g) * a.cap + t0;  // first slot row of the chunk
  const uint16_t* kc = reinterpret_cast<const uint16_t*>(a.kc);
  const uint16_t* vc = reinterpret_cast<const uint16_t*>(a.vc);
  // tile i into ring stage i % NS: each thread copies chunks tid, tid + 256, ...
  // of the K and V tiles; slots past the chunk's end are zero-filled
  auto issue = [&](int i) {
    if (i < nt) {
      const int stage = i % kMmaNS;
      const int rows = min(kMmaTS, n - i * kMmaTS);
#pragma unroll
      for (int j = 0; j < kMmaTS * CH / kMmaThreads; ++j) {
        const int q = tid + j * kMmaThreads, r = q / CH, ch = q - r * CH;
        const bool in = r < rows;
        const size_t src = (base + (size_t)i * kMmaTS + (in ? r : 0)) * DH + (size_t)ch * 8;
        const uint32_t off = swz(r, ch, RB);
        cp_async16(sbase + (uint32_t)Lay::K + stage * Lay::TILE + off, kc + src, in ? 16u : 0u);
        cp_async16(sbase + (uint32_t)Lay::V + stage * Lay::TILE + off, vc + src, in ? 16u : 0u);
      }
    }
    cp_async_commit();  // one group per tile index, empty past the end
  };
  // Tiles whose slots all lie below this call's first new slot hold cache rows
  // written by earlier calls: they are requested before waiting for k_qkv_post,
  // which writes the new ones; the rest after it.
  int pre = 0;
  while (pre < kMmaNS && (pre >= nt || t0 + (pre + 1) * kMmaTS <= a.first_new[m])) issue(pre++);
  pdl_wait();
  pdl_trigger();
  for (int i = pre; i < kMmaNS; ++i) issue(i);

  // this warp's A fragments of Q: rows 0-7 the heads rounded to bf16, rows
  // 8-15 what that left over (heads >= G are zero)
  uint32_t qa[KSW][4];
  {
    const float* qg = a.q + (size_t)m * a.nq * DH + (size_t)g * G * DH;
#pragma unroll
    for (int ks = 0; ks < KSW; ++ks) {
      const int d0 = warp * DW + ks * 16 + 2 * gc;
      float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
      if (gr < G) {
        const float* qr = qg + (size_t)gr * DH;
        x0 = qr[d0];
        x1 = qr[d0 + 1];
        x2 = qr[d0 + 8];
        x3 = qr[d0 + 9];
      }
      split2(x0, x1, qa[ks][0], qa[ks][1]);
      split2(x2, x3, qa[ks][2], qa[ks][3]);
    }
  }
  float oacc[NB2][4];
#pragma unroll
  for (int j = 0; j < NB2; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

  for (int i = 0; i < nt; ++i) {
    const int stage = i % kMmaNS;
    const int rows = min(kMmaTS, n - i * kMmaTS);
    cp_async_wait<kMmaNS - 1>();
    __syncthreads();
    const uint32_t kt = sbase + (uint32_t)Lay::K + stage * Lay::TILE;
    const uint32_t vt = sbase + (uint32_t)Lay::V + stage * Lay::TILE;
    // partial scores of this warp's dimensions, 8 blocks of 8 slots
    {
      float* sw = sS + (size_t)warp * 8 * kSStride;
#pragma unroll
      for (int nb = 0; nb < kMmaTS / 8; ++nb) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int key = nb * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < KSW; ++ks) {
          const int ch = (warp * DW + ks * 16) / 8 + ((lane >> 3) & 1);
          uint32_t b0, b1;
          ldsm_x2(kt + swz(key, ch, RB), b0, b1);
          mma_bf16(acc, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        }
        // rows gr (rounded q) and gr + 8 (remainder) of the same head
        *reinterpret_cast<float2*>(sw + gr * kSStride + nb * 8 + 2 * gc) = make_float2(acc[0] + acc[2], acc[1] + acc[3]);
      }
    }
    __syncthreads();
    // online softmax: warp h owns head h
    if (warp < G) {
      const int h = warp;
      float s[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int k = lane + 32 * u;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kMmaWarps; ++w) v += sS[((size_t)w * 8 + h) * kSStride + k];
        s[u] = k < rows ? v * a.scale : -INFINITY;
      }
      const float mx = warp_max(fmaxf(s[0], s[1]));
      const float m_old = st[4 * h];
      const float m_new = fmaxf(m_old, mx);
      const float alpha = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int k = lane + 32 * u;
        const float p = k < rows ? expf(s[u] - m_new) : 0.f;
        sum += p;
        const uint16_t ph = f_to_bf16(p), pl = f_to_bf16(p - bf16_to_f(ph));
        const int kc8 = k >> 3, ke = k & 7;
        sP[(swz(h, kc8, 2 * kMmaTS) >> 1) + ke] = ph;
        sP[(swz(h + 8, kc8, 2 * kMmaTS) >> 1) + ke] = pl;
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        st[4 * h] = m_new;
        st[4 * h + 1] = alpha;
        st[4 * h + 2] = st[4 * h + 2] * alpha + sum;
      }
    }
    __syncthreads();
    // O = O alpha + P V over this warp's NB2 blocks of 8 dimensions
    {
      const float al = gr < G ? st[4 * gr + 1] : 1.f;
#pragma unroll
      for (int j = 0; j < NB2; ++j) {
        oacc[j][0] *= al;
        oacc[j][1] *= al;
        oacc[j][2] *= al;
        oacc[j][3] *= al;
      }
      const uint32_t pt = sbase + (uint32_t)Lay::P;
#pragma unroll
      for (int ks = 0; ks < kMmaTS / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        {
          const int r = (lane & 7) + 8 * ((lane >> 3) & 1), ch = 2 * ks + (lane >> 4);
          ldsm_x4(pt + swz(r, ch, 2 * kMmaTS), a0, a1, a2, a3);
        }
        const int key = ks * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int j = 0; j < NB2; j += 2) {
          const int ch = (warp * DW + j * 8) / 8 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vt + swz(key, ch, RB), b0, b1, b2, b3);
          mma_bf16(oacc[j], a0, a1, a2, a3, b0, b1);
          mma_bf16(oacc[j + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();  // every warp is done with this stage: refill it
    issue(i + kMmaNS);
  }
  cp_async_wait<0>();
  // partial output of this chunk: rows gr and gr + 8 of head gr
  if (gr < G) {
    const size_t hq = (size_t)m * a.nq + (size_t)g * G + gr;
    float* po = a.po + (hq * a.max_chunks + c) * DH;
#pragma unroll
    for (int j = 0; j < NB2; ++j) {
      const int d = warp * DW + j * 8 + 2 * gc;
      *reinterpret_cast<float2*>(po + d) = make_float2(oacc[j][0] + oacc[j][2], oacc[j][1] + oacc[j][3]);
    }
  }
  if (tid < G) {
    const size_t hq = (size_t)m * a.nq + (size_t)g * G + tid;
    a.pml[(hq * a.max_chunks + c) * 2 + 0] = st[4 * tid];
    a.pml[(hq * a.max_chunks + c) * 2 + 1] = st[4 * tid + 2];
  }
}

template <int DH>
bool attn_mma_t(const AttnArgs& a0, int sms, cudaStream_t s) {
  using Lay = MmaLayout<DH>;
  auto k = k_attn_mma<DH>;
  static std::mutex mu;
  static int resident[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  int per_sm;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (resident[dev] == 0) {
      int nb = 0;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay::TOTAL) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, kMmaThreads, Lay::TOTAL) != cudaSuccess || nb < 1)
        nb = -1;
      cudaGetLastError();
      resident[dev] = nb;
    }
    per_sm = resident[dev];
  }
  if (per_sm < 1) return false;
  AttnArgs a = a0;
  a.chunk = attn_chunk_slots(a, (long long)per_sm * sms);
  int maxL = 0;
  for (int m = 0; m < a.Mh; ++m) maxL = max(maxL, a.slot[m] + 1);
  const int nch = (maxL + a.chunk - 1) / a.chunk;
  launch_pdl(k, dim3(nch, a.nkv, a.Mh), dim3(kMmaThreads), Lay::TOTAL, s, a);
  count_launch();
  launch_attn_merge(a, s);
  return true;
}

}  // namespace

bool launch_attention_mma(const AttnArgs& a, int sms, cudaStream_t s) {
  const int G = a.nkv > 0 ? a.nq / a.nkv : 0;
  if (a.wdt != MTP_DTYPE_BF16 || G < 1 || G > 8 || a.nq != G * a.nkv) return false;
  if ((reinterpret_cast<uintptr_t>(a.kc) & 15) != 0 || (reinterpret_cast<uintptr_t>(a.vc) & 15) != 0) return false;
  if (a.dh == 256) return attn_mma_t<256>(a, sms, s);
  if (a.dh == 128) return attn_mma_t<128>(a, sms, s);
  return false;
}

}  // namespace mtp
