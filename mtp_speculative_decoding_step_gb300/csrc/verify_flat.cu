// Greedy verify for many rows as one balanced stream.
//
// With every row greedy and no repetition penalty, the verify is an argmax
// per (row, position) followed by the accept chain ("greedy is a special case
// of sampled decoding": acceptance reduces to argmax-match, Ollama MLX-runner
// commit log). When many rows are verified at once the target logits
// [rows][depth+1][V] are one long array; here it is cut into equal
// contiguous ranges, one per CTA, sized so that the whole grid is resident at
// once and every SM streams the same number of bytes, whatever the row count.
// A range may span several (row, position) segments: each thread keeps its
// running (value, id) maximum and hands it to the segment's shared-memory slot
// (a 64-bit key whose order is value desc, id asc) when it crosses a segment
// boundary. Each CTA stores one key per segment it touched, at index
// cta + segment (unique, since consecutive ranges share at most one segment).
// A second kernel, one warp per row, combines the few keys of each position
// and walks the accept chain.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

constexpr int kFlatThreads = 256;
constexpr int kFlatBlocksPerSM = 4;
constexpr int kFlatVec = 8;       // 16-byte loads in flight per thread
constexpr int kFlatMaxSeg = 64;   // segments one range may touch
constexpr long long kFlatMinRange = 4096;  // floats per CTA at least

// Order key of (value, id): larger value first, then lower id; -0 counts as
// +0 (they compare equal). NaN never reaches here (it never beats a maximum).
__device__ __forceinline__ unsigned long long argmax_key(float v, int id) {
  uint32_t u = __float_as_uint(v + 0.0f);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}

__global__ void __launch_bounds__(kFlatThreads, kFlatBlocksPerSM)
    k_verify_greedy_flat(const __grid_constant__ VerifyArgs a, long long N, long long L,
                         unsigned long long* part) {
  __shared__ unsigned long long s_key[kFlatMaxSeg];
  const long long V = a.V;
  const long long lo = (long long)blockIdx.x * L;
  const long long hi = min(lo + L, N);
  const long long t0 = lo / V;
  const int nseg = (int)((hi - 1) / V - t0 + 1);
  for (int i = threadIdx.x; i < nseg; i += kFlatThreads) s_key[i] = 0ull;  // 0: nothing seen
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(a.logits + lo);
  const long long n4 = (hi - lo) / 4;  // V, L and N are multiples of 4
  long long t = t0;
  long long B = (t0 + 1) * V;  // first element of the next segment
  float bv = -INFINITY;
  int bi = -1;
  float nf = 0.f;  // x * 0: NaN once a NaN or an infinity has been read
  auto hand_over = [&]() {
    if (bi >= 0) atomicMax(&s_key[t - t0], argmax_key(bv, bi));
    bv = -INFINITY;
    bi = -1;
  };
  // batches of kFlatVec 16-byte loads per thread, all in flight before the
  // batch is reduced (measured faster here than two half batches pipelined
  // with an L2 prefetch ahead)
  for (long long base = 0; base < n4; base += (long long)kFlatVec * kFlatThreads) {
    uint4 buf[kFlatVec];
#pragma unroll
    for (int e = 0; e < kFlatVec; ++e) {
      const long long j = base + e * kFlatThreads + threadIdx.x;
      if (j < n4) buf[e] = ldg_stream(src + j);
    }
#pragma unroll
    for (int e = 0; e < kFlatVec; ++e) {
      const long long j = base + e * kFlatThreads + threadIdx.x;
      if (j < n4) {
        const long long p = lo + 4 * j;
        while (p >= B) {  // this thread's next element lies in a later segment
          hand_over();
          ++t;
          B += V;
        }
        const int i0 = (int)(p - (B - V));
        const float x[4] = {__uint_as_float(buf[e].x), __uint_as_float(buf[e].y), __uint_as_float(buf[e].z),
                            __uint_as_float(buf[e].w)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          nf = fmaf(x[q], 0.f, nf);
          // a thread sees its ids in ascending order: strict > keeps the lowest on ties
          if (x[q] > bv) { bv = x[q]; bi = i0 + q; }
        }
      }
    }
  }
  hand_over();
  __syncthreads();
  for (int i = threadIdx.x; i < nseg; i += kFlatThreads) part[blockIdx.x + t0 + i] = s_key[i];
  if (__syncthreads_or(isnan(nf)) && threadIdx.x == 0) flag_status(a.status, MTP_ERR_NONFINITE);
}

// One warp per row: lane i combines the keys of position i, then the accept
// chain: drafts x_1.. equal to the argmax of the row before them are accepted;
// the first mismatch (or the bonus row) gives its argmax as the last token.
__global__ void __launch_bounds__(32) k_verify_greedy_flat_finish(const __grid_constant__ VerifyArgs a, long long L,
                                                                  const unsigned long long* part) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, d = a.depth, lane = threadIdx.x;
  const long long V = a.V;
  int am = 0;
  if (lane <= d) {
    const long long t = (long long)r * (d + 1) + lane;
    const long long c_lo = t * V / L, c_hi = ((t + 1) * V - 1) / L;
    unsigned long long best = 0ull;
    for (long long c = c_lo; c <= c_hi; ++c) best = max(best, part[c + t]);
    // nothing comparable (every logit NaN or -inf): id 0, the lowest
    am = best ? (int)(0xFFFFFFFFu - (uint32_t)best) : 0;
  }
  const int32_t* dr = a.drafts + (size_t)r * d;
  const int x = lane < d ? dr[lane] : -1;
  const bool match = lane < d && x >= 0 && x < a.V && x == am;
  const unsigned miss = __ballot_sync(0xFFFFFFFFu, lane < d && !match);
  const int nacc = miss ? __ffs(miss) - 1 : d;
  const int y = __shfl_sync(0xFFFFFFFFu, am, nacc);
  const int ov = lane < nacc ? x : (lane == nacc ? y : -1);
  if (lane <= d) {
    a.out_tok[(size_t)r * (d + 1) + lane] = ov;
    if (a.h_rec) a.h_rec[(size_t)r * (d + 2) + 1 + lane] = ov;
  }
  __syncwarp();
  if (lane == 0) {
    a.n_acc[r] = nacc;
    // the record's tokens are visible to the host before its count
    if (a.h_rec) st_release_sys(a.h_rec + (size_t)r * (d + 2), nacc);
    if (a.stats) {
      int32_t* st = a.stats + (size_t)r * (d + 2);
      st[0] += 1;
      if (nacc < d) st[1] += 1;
      for (int i = 1; i <= nacc; ++i) st[1 + i] += 1;
    }
  }
}

bool launch_verify_greedy_flat(const VerifyArgs& a, void* d_part, size_t part_bytes, cudaStream_t s) {
  const long long V = a.V;
  if (V % 4 != 0 || (reinterpret_cast<uintptr_t>(a.logits) & 15) != 0 || a.depth + 1 > 32) return false;
  const long long tasks = (long long)a.rows * (a.depth + 1);
  const long long N = tasks * V;
  const long long slots = (long long)device_sm_count() * kFlatBlocksPerSM;
  long long L = (N + slots - 1) / slots;
  L = std::max(L, kFlatMinRange);
  L = std::min(L, (long long)(kFlatMaxSeg - 2) * V);  // a range touches at most kFlatMaxSeg segments
  L = (L + 3) / 4 * 4;
  const long long G = (N + L - 1) / L;
  if (G > kFlatMaxCTAs || (size_t)(G + tasks) * sizeof(unsigned long long) > part_bytes) return false;
  unsigned long long* part = static_cast<unsigned long long*>(d_part);
  launch_pdl(k_verify_greedy_flat, dim3((unsigned)G), dim3(kFlatThreads), 0, s, a, N, L, part);
  count_launch();
  launch_pdl(k_verify_greedy_flat_finish, dim3(a.rows), dim3(32), 0, s, a, L,
             static_cast<const unsigned long long*>(part));
  count_launch();
  return true;
}

}  // namespace mtp
