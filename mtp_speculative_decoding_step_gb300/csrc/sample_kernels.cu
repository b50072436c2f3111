// Sampling transforms and rejection-sampling verify for sm_103a.
//
// The sampler chain (temperature, repetition penalty over a ring history,
// top-k, top-p, min-p) and the unified greedy/sampled verify follow the
// Ollama MLX-runner commit log ("greedy is a special case of sampled decoding
// -- at temperature 0 the sampler yields a point mass, so rejection-sampling
// acceptance reduces to argmax-match"; sampler transforms commit). Readings
// where the pages are silent:
//   * penalty applies once per distinct window token: z/r if z > 0 else z*r;
//   * tokens are ordered by (transformed logit desc, id asc); top-k keeps the
//     first k, top-p the shortest prefix whose cumulative exp(z - zmax)
//     reaches top_p of the top-k total, min-p keeps exp(z - zmax) >= min_p;
//     the kept set is their intersection, renormalised;
//   * draws are inverse-CDF in ascending id order with a pre-drawn uniform.
//
// One thread-block cluster of 8 CTAs works on one (row, position): each CTA
// holds a contiguous slice of the vocabulary in shared memory, and the CTAs
// combine histograms, sums and arg-maxima through distributed shared memory.
// Sums that decide a threshold are exact integers (values scaled by 2^40), so
// every result is independent of thread scheduling.
#include <cooperative_groups.h>

#include <algorithm>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace mtp {

constexpr int kST = 512;  // threads per sampling CTA
constexpr double kFix = 1099511627776.0;  // 2^40

__device__ __forceinline__ uint32_t desc_key(float z) {
  uint32_t u = __float_as_uint(z);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending in z
  return ~u;                                        // ascending in -z
}

__device__ __forceinline__ uint64_t to_fix(float w) {
  return w > 0.f ? (uint64_t)__float2ull_rn(w * 1099511627776.0f) : 0ull;
}

__device__ __forceinline__ float penalize(float z, float r) { return z > 0.f ? z / r : z * r; }

struct Mail {
  unsigned long long u[4];
  float f[4];
  int i[4];
};

struct SampleSmem {
  Mail mail[2];
  unsigned long long hist[2][256];
  unsigned long long tot[256];
  unsigned long long wsum[kST / 32];
  int wtok[160];
  int nwin;
  int sel_bin;
  unsigned long long sel_rem;
  int found;
  int ccount;
  int fin_kf;
  int fin_valid;
  unsigned long long fin_sf;
  int fin_draw;
};

// Cluster context for one task.
struct Clu {
  cg::cluster_group cl;
  SampleSmem* sm;
  int ph;
  int rank;
  __device__ Clu(SampleSmem* s) : cl(cg::this_cluster()), sm(s), ph(0), rank((int)cg::this_cluster().block_rank()) {}

  // Publish (f, i, u) scalars from thread 0 and return every CTA's values.
  __device__ Mail* publish() {
    cl.sync();
    Mail* m = &sm->mail[ph];
    ph ^= 1;
    return m;
  }
  __device__ Mail* remote(Mail* local, int r) { return cl.map_shared_rank(local, r); }
};

// Argmax (value desc, id asc) over the block, result to all threads.
__device__ void block_argmax(float& v, int& i, float* sv, int* si) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  warp_argmax(v, i);
  __syncthreads();
  if (lane == 0) { sv[w] = v; si[w] = i; }
  __syncthreads();
  if (w == 0) {
    v = lane < kST / 32 ? sv[lane] : -INFINITY;
    i = lane < kST / 32 ? si[lane] : 0x7FFFFFFF;
    warp_argmax(v, i);
    if (lane == 0) { sv[0] = v; si[0] = i; }
  }
  __syncthreads();
  v = sv[0];
  i = si[0];
}

__device__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int k = 0; k < kST / 32; ++k) t += sh[k];  // fixed order
  __syncthreads();
  return t;
}

// Sum a per-CTA u64 over the cluster (rank order).
__device__ unsigned long long cluster_sum_u64(Clu& c, unsigned long long local) {
  if (threadIdx.x == 0) c.sm->mail[c.ph].u[0] = local;
  Mail* m = c.publish();
  unsigned long long t = 0;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) t += c.remote(m, r)->u[0];
  return t;
}

// Radix selection over the cluster: among active elements ordered by
// (key asc, id asc) with integer weights, find the key K* of the element at
// which the running weight first reaches `target`, and how much of the
// target remains within the elements whose key is K*. The digits start at the
// highest bit where the active keys differ (from their cluster-wide min and
// max), so the bins spread over the keys actually present.
template <class Act, class Wt>
__device__ void radix_select(Clu& c, const float* zs, int n_local, Act active, Wt weight,
                             unsigned long long target, uint32_t& key_out, unsigned long long& rem_out) {
  SampleSmem* sm = c.sm;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int j = threadIdx.x; j < n_local; j += kST)
    if (active(j)) {
      const uint32_t k = desc_key(zs[j]);
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xFFFFFFFFu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xFFFFFFFFu, kmax, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sm->wsum[threadIdx.x >> 5] = ((unsigned long long)kmin << 32) | kmax;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = 0xFFFFFFFFu, b = 0u;
    for (int w = 0; w < kST / 32; ++w) {
      a = min(a, (uint32_t)(sm->wsum[w] >> 32));
      b = max(b, (uint32_t)sm->wsum[w]);
    }
    sm->mail[c.ph].u[0] = a;
    sm->mail[c.ph].u[1] = b;
  }
  Mail* mm = c.publish();
  kmin = 0xFFFFFFFFu;
  kmax = 0u;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) {
    kmin = min(kmin, (uint32_t)c.remote(mm, r)->u[0]);
    kmax = max(kmax, (uint32_t)c.remote(mm, r)->u[1]);
  }
  const uint32_t diff = kmin ^ kmax;
  int hi = diff ? 31 - __clz(diff) : -1;
  uint32_t mask = hi >= 0 ? ~((hi == 31) ? 0xFFFFFFFFu : ((2u << hi) - 1u)) : 0xFFFFFFFFu;
  uint32_t prefix = kmin & mask;
  while (hi >= 0) {
    const int lo = hi >= 7 ? hi - 7 : 0;
    const uint32_t dmask = (1u << (hi - lo + 1)) - 1u;
    unsigned long long* h = sm->hist[c.ph];
    for (int b = threadIdx.x; b < 256; b += kST) h[b] = 0;
    __syncthreads();
    // warp-aggregated: lanes with the same bin add their weights (split in
    // 24-bit halves so the 32-bit warp sums stay exact), one atomic per bin
    for (int base = 0; base < n_local; base += kST) {
      const int j = base + threadIdx.x;
      bool act = j < n_local && active(j);
      const uint32_t k = act ? desc_key(zs[j]) : 0u;
      act = act && (k & mask) == prefix;
      const uint32_t bin = act ? ((k >> lo) & dmask) : 0xFFFFFFFFu;
      const unsigned long long w = act ? weight(j) : 0ull;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, bin);
      const unsigned sl = __reduce_add_sync(peers, (unsigned)(w & 0xFFFFFFull));
      const unsigned sh = __reduce_add_sync(peers, (unsigned)(w >> 24));
      if (act && (int)(threadIdx.x & 31) == __ffs(peers) - 1)
        atomicAdd(&h[bin], ((unsigned long long)sh << 24) + (unsigned long long)sl);
    }
    c.cl.sync();
    for (int b = threadIdx.x; b < 256; b += kST) {
      unsigned long long t = 0;
#pragma unroll
      for (int r = 0; r < kClusterCTAs; ++r) t += c.cl.map_shared_rank(h, r)[b];
      sm->tot[b] = t;
    }
    c.ph ^= 1;
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      unsigned long long s8 = 0;
      for (int b = 0; b < 8; ++b) s8 += sm->tot[lane * 8 + b];
      unsigned long long incl = s8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
      }
      unsigned long long cum = incl - s8;
      const bool mine = cum < target && target <= incl;
      if (mine) {
        for (int b = 0; b < 8; ++b) {
          const unsigned long long t = sm->tot[lane * 8 + b];
          if (cum < target && target <= cum + t) {
            sm->sel_bin = lane * 8 + b;
            sm->sel_rem = target - cum;
            break;
          }
          cum += t;
        }
      }
      const unsigned any = __ballot_sync(0xFFFFFFFFu, mine);
      if (!any && lane == 0) {  // target above the total: keep everything
        sm->sel_bin = (int)dmask;
        sm->sel_rem = target;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sm->sel_bin << lo;
    mask |= dmask << lo;
    target = sm->sel_rem;
    __syncthreads();
    hi = lo - 1;
  }
  key_out = prefix;
  rem_out = target;
}

// Among active elements with key == K* (ids ascending over the cluster),
// return the id of the n-th (1-based), or INT_MAX if n covers all of them.
template <class Act>
__device__ int tie_cut(Clu& c, const float* zs, int n_local, int v0, Act active, uint32_t K,
                       unsigned long long n) {
  SampleSmem* sm = c.sm;
  unsigned long long cnt = 0;
  for (int j = threadIdx.x; j < n_local; j += kST)
    if (active(j) && desc_key(zs[j]) == K) ++cnt;
  cnt = block_sum_u64(cnt, sm->wsum);
  if (threadIdx.x == 0) sm->mail[c.ph].u[0] = cnt;
  Mail* m = c.publish();
  unsigned long long before = 0, total = 0;
  int owner = -1;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) {
    const unsigned long long t = c.remote(m, r)->u[0];
    if (owner < 0 && before + t >= n) owner = r;
    if (owner < 0) before += t;
    total += t;
  }
  if (n >= total) return 0x7FFFFFFF;
  int cut = -1;
  if (c.rank == owner) {
    // scan this slice in id order, 512 elements at a time
    unsigned long long need = n - before;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (threadIdx.x == 0) sm->found = -1;
    __syncthreads();
    for (int base = 0; base < n_local; base += kST) {
      const int j = base + threadIdx.x;
      const unsigned flag = (j < n_local && active(j) && desc_key(zs[j]) == K) ? 1u : 0u;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, flag);
      __syncthreads();
      if (lane == 0) sm->wsum[w] = __popc(bal);
      __syncthreads();
      unsigned long long wbefore = 0, chunk = 0;
      for (int k = 0; k < kST / 32; ++k) {
        if (k < w) wbefore += sm->wsum[k];
        chunk += sm->wsum[k];
      }
      const unsigned long long incl = wbefore + __popc(bal & ((2u << lane) - 1u));
      if (flag && incl == need) sm->found = v0 + j;
      __syncthreads();
      if (chunk >= need) break;
      need -= chunk;
    }
    cut = sm->found;
  }
  if (threadIdx.x == 0) sm->mail[c.ph].i[0] = cut;
  m = c.publish();
  return c.remote(m, owner)->i[0];
}

// Inverse-CDF draw over the cluster with per-element integer weights:
// smallest id whose cumulative weight exceeds u * total. Returns -1 if the
// total is zero.
template <class Wt>
__device__ int cluster_draw(Clu& c, int n_local, int v0, Wt weight, float u) {
  SampleSmem* sm = c.sm;
  unsigned long long loc = 0;
  for (int j = threadIdx.x; j < n_local; j += kST) loc += weight(j);
  loc = block_sum_u64(loc, sm->wsum);
  if (threadIdx.x == 0) sm->mail[c.ph].u[0] = loc;
  Mail* m = c.publish();
  unsigned long long tot = 0;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) tot += c.remote(m, r)->u[0];
  if (tot == 0) return -1;
  const unsigned long long target = (unsigned long long)floor((double)u * (double)tot) + 1ull;
  unsigned long long tv[kClusterCTAs];
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) tv[r] = c.remote(m, r)->u[0];
  unsigned long long before = 0;
  int owner = kClusterCTAs - 1;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) {
    if (before + tv[r] >= target) { owner = r; break; }
    before += tv[r];
  }
  int pick = -1;
  if (c.rank == owner) {
    const unsigned long long need = target - before;
    const int per_t = (n_local + kST - 1) / kST;
    const int a0 = min(threadIdx.x * per_t, n_local), a1 = min(a0 + per_t, n_local);
    unsigned long long loc2 = 0;
    for (int j = a0; j < a1; ++j) loc2 += weight(j);
    // exclusive block scan of the per-thread sums
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    unsigned long long incl = loc2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (threadIdx.x == 0) sm->found = -1;
    __syncthreads();
    if (lane == 31) sm->wsum[w] = incl;
    __syncthreads();
    unsigned long long wbefore = 0;
    for (int k = 0; k < w; ++k) wbefore += sm->wsum[k];
    unsigned long long cum = wbefore + incl - loc2;
    if (cum < need && need <= cum + loc2) {
      for (int j = a0; j < a1; ++j) {
        const unsigned long long x = weight(j);
        cum += x;
        if (x > 0 && cum >= need) { sm->found = v0 + j; break; }
      }
    }
    __syncthreads();
    pick = sm->found;
  }
  if (threadIdx.x == 0) sm->mail[c.ph].i[0] = pick;
  m = c.publish();
  return c.remote(m, owner)->i[0];
}

// Load the penalty window of position i into shared memory.
__device__ void load_window(SampleSmem* sm, const int32_t* hist, int W, const int32_t* drafts, int i) {
  const int drop = i < W ? i : W;
  const int nh = W - drop;
  const int first = i > W ? i - W : 0;
  const int nd = i - first;
  for (int t = threadIdx.x; t < nh + nd; t += kST)
    sm->wtok[t] = t < nh ? hist[drop + t] : drafts[first + t - nh];
  if (threadIdx.x == 0) sm->nwin = nh + nd;
  __syncthreads();
}

// Mark window tokens that fall in [v0, v0+n) in the bitmap (each once).
__device__ void build_bitmap(SampleSmem* sm, uint32_t* bits, int v0, int n) {
  for (int w = threadIdx.x; w < (n + 31) / 32; w += kST) bits[w] = 0u;
  __syncthreads();
  for (int t = threadIdx.x; t < sm->nwin; t += kST) {
    const int v = sm->wtok[t] - v0;
    if (v >= 0 && v < n) atomicOr(&bits[v >> 5], 1u << (v & 31));
  }
  __syncthreads();
}

__device__ __forceinline__ bool bit(const uint32_t* bits, int j) { return (bits[j >> 5] >> (j & 31)) & 1u; }

__device__ __forceinline__ bool in_prefix(uint32_t key, int v, uint32_t K, int cut) {
  return key < K || (key == K && v <= cut);
}

// ------------------------------------------------------------ candidate path
// Most rows keep a small support (top-k set, or a peaky top-p/min-p prefix).
// Each CTA selects its local top-C keys with block-local passes, the cluster
// exchanges them once, and every CTA sorts the union by (key, id) -- the
// oracle's (transformed logit desc, id asc) order -- and cuts top-k, top-p and
// min-p on that list. The first C entries of the sorted union are the global
// top-C, so the cut is exact whenever it falls inside them (always with top-k
// <= C); otherwise the full cluster radix path below is used.

constexpr int kCandTopP = 128;  // local candidates per CTA when no top-k is set

struct CandBufs {
  uint32_t* ckey;  // [C] local candidates
  int* cid;
  uint32_t* mkey;  // [P] merged, sorted
  int* mid;
  unsigned long long* sw;  // [C] draw weights in id order
  int* sid;
  int C, P;
};

__device__ __forceinline__ float key_to_z(uint32_t K) {
  uint32_t u = ~K;
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

// Exactly min(C, n) local elements satisfy in_prefix(key, v0 + j, K, cut).
// kmin / kmax: the range of the block's keys (from the staging pass).
__device__ void local_select(SampleSmem* sm, const float* zs, int n, int v0, int C, uint32_t kmin, uint32_t kmax,
                             uint32_t& Kout, int& cut) {
  if (n <= C) { Kout = 0xFFFFFFFFu; cut = 0x7FFFFFFF; return; }
  const uint32_t diff = kmin ^ kmax;
  int hi = diff ? 31 - __clz(diff) : -1;
  uint32_t mask = hi >= 0 ? ~((hi == 31) ? 0xFFFFFFFFu : ((2u << hi) - 1u)) : 0xFFFFFFFFu;
  uint32_t prefix = kmin & mask;
  unsigned long long target = (unsigned long long)C;
  unsigned long long ties = (unsigned long long)n;  // all keys equal when hi < 0
  unsigned long long* h = sm->hist[0];
  while (hi >= 0) {
    const int lo = hi >= 7 ? hi - 7 : 0;
    const uint32_t dmask = (1u << (hi - lo + 1)) - 1u;
    __syncthreads();
    for (int b = threadIdx.x; b < 256; b += kST) h[b] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kST) {
      const int j = base + threadIdx.x;
      const uint32_t k = j < n ? desc_key(zs[j]) : 0u;
      const bool act = j < n && (k & mask) == prefix;
      if (!__any_sync(0xFFFFFFFFu, act)) continue;
      const uint32_t bin = act ? ((k >> lo) & dmask) : 0xFFFFFFFFu;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, bin);
      if (act && (int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[bin], (unsigned long long)__popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      unsigned long long s8 = 0;
      for (int b = 0; b < 8; ++b) s8 += h[lane * 8 + b];
      unsigned long long incl = s8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      unsigned long long cum = incl - s8;
      if (cum < target && target <= incl) {
        for (int b = 0; b < 8; ++b) {
          const unsigned long long t = h[lane * 8 + b];
          if (cum < target && target <= cum + t) {
            sm->sel_bin = lane * 8 + b;
            sm->sel_rem = target - cum;
            sm->fin_sf = t;  // elements in the chosen bin
            break;
          }
          cum += t;
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sm->sel_bin << lo;
    mask |= dmask << lo;
    target = sm->sel_rem;
    if (lo == 0) ties = sm->fin_sf;  // the last digit resolves the key: its bin holds the ties
    hi = lo - 1;
  }
  Kout = prefix;
  // ties at K: keep the first `target` of them in index order
  if (target >= ties) { cut = 0x7FFFFFFF; __syncthreads(); return; }
  unsigned long long need = target;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) sm->found = 0x7FFFFFFF;
  __syncthreads();
  for (int base = 0; base < n; base += kST) {
    const int j = base + threadIdx.x;
    const unsigned flag = (j < n && desc_key(zs[j]) == prefix) ? 1u : 0u;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, flag);
    __syncthreads();
    if (lane == 0) sm->wsum[w] = __popc(bal);
    __syncthreads();
    unsigned long long wbefore = 0, chunk = 0;
    for (int k = 0; k < kST / 32; ++k) {
      if (k < w) wbefore += sm->wsum[k];
      chunk += sm->wsum[k];
    }
    const unsigned long long incl = wbefore + __popc(bal & ((2u << lane) - 1u));
    if (flag && incl == need) sm->found = v0 + j;
    __syncthreads();
    if (chunk >= need) break;
    need -= chunk;
  }
  cut = sm->found;
  __syncthreads();
}

// Local candidates in one histogram pass: bins are 256 equal slices of the
// block's value range [zmin, zmax] (bin 0 holds the largest); bin index is
// weakly monotone in z, so every bin is a contiguous range of the (key, id)
// order. All elements of the bins up to and including the one holding the
// C-th largest are written out -- a superset of the local top-C. Returns the
// count, or -1 if it would exceed cap (the caller then selects exactly).
__device__ int local_candidates(SampleSmem* sm, const float* zs, int n, int v0, int C, int cap, uint32_t kmin,
                                uint32_t kmax, uint32_t* ckey, int* cid) {
  const float zmax = key_to_z(kmin), zmin = key_to_z(kmax);
  const float span = zmax - zmin;
  const float scale = span > 0.f ? 255.99f / span : 0.f;
  unsigned int* h = reinterpret_cast<unsigned int*>(sm->hist[0]);
  for (int b = threadIdx.x; b < 256; b += kST) h[b] = 0u;
  if (threadIdx.x == 0) sm->ccount = 0;
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += kST) {
    const int b = min(255, (int)((zmax - zs[j]) * scale));
    atomicAdd(&h[b], 1u);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned int s8 = 0;
    for (int b = 0; b < 8; ++b) s8 += h[lane * 8 + b];
    unsigned int incl = s8;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    unsigned int cum = incl - s8;
    if (cum < (unsigned)C && (unsigned)C <= incl) {
      for (int b = 0; b < 8; ++b) {
        cum += h[lane * 8 + b];
        if (cum >= (unsigned)C) {
          sm->sel_bin = lane * 8 + b;
          sm->fin_draw = (int)cum;  // elements in bins <= sel_bin
          break;
        }
      }
    }
  }
  __syncthreads();
  const int B = sm->sel_bin, total = sm->fin_draw;
  __syncthreads();
  if (total > cap) return -1;
  for (int j = threadIdx.x; j < n; j += kST) {
    const int b = min(255, (int)((zmax - zs[j]) * scale));
    if (b <= B) {
      const int pos = atomicAdd(&sm->ccount, 1);
      ckey[pos] = desc_key(zs[j]);
      cid[pos] = v0 + j;
    }
  }
  __syncthreads();
  return sm->ccount;
}

__device__ __forceinline__ bool pair_gt(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia > ib);
}

// Ascending (key, id) sort of kST pairs, one per thread, with distinct ids:
// a bitonic network, its compare-exchanges over shuffles below a warp's span
// and through shared memory (sk, si: kST entries each) above it. On return
// thread t holds the t-th smallest pair. For one pair per thread this takes
// fewer block barriers than a digit-by-digit radix selection.
__device__ void block_sort(uint32_t& key, int& id, uint32_t* sk, int* si) {
  const int t = threadIdx.x;
#pragma unroll
  for (int size = 2; size <= kST; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint32_t ok;
      int oi;
      if (stride >= 32) {
        __syncthreads();
        sk[t] = key;
        si[t] = id;
        __syncthreads();
        ok = sk[t ^ stride];
        oi = si[t ^ stride];
      } else {
        ok = __shfl_xor_sync(0xFFFFFFFFu, key, stride);
        oi = __shfl_xor_sync(0xFFFFFFFFu, id, stride);
      }
      const bool asc = (t & size) == 0;
      const bool low = (t & stride) == 0;
      const bool other_less = ok < key || (ok == key && oi < id);
      if (low == asc ? other_less : !other_less) {
        key = ok;
        id = oi;
      }
    }
  }
  __syncthreads();
}
// The k-th smallest (1 <= k <= kST) of kST pairs, one per thread with
// distinct ids, to every thread (sorts them with block_sort).
__device__ void block_kth_pair(uint32_t key, int id, int k, uint32_t* sk, int* si, SampleSmem* sm, uint32_t& K,
                               int& I) {
  block_sort(key, id, sk, si);
  if ((int)threadIdx.x == k - 1) {
    sm->sel_rem = key;
    sm->found = id;
  }
  __syncthreads();
  K = (uint32_t)sm->sel_rem;
  I = sm->found;
  __syncthreads();
}
// Sentinel id of thread t for block_sort (above every vocabulary id).
__device__ __forceinline__ int sort_sentinel() { return 0x7FFFFFFF - (kST - 1) + (int)threadIdx.x; }

// Ascending (key, id) bitonic sort of P (power of two) entries in shared memory.
__device__ void bitonic_sort(uint32_t* key, int* id, int P) {
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += kST) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool asc = (i & k) == 0;
          const uint32_t ka = key[i], kb = key[ixj];
          const int ia = id[i], ib = id[ixj];
          if (pair_gt(ka, ia, kb, ib) == asc) {
            key[i] = kb; key[ixj] = ka;
            id[i] = ib; id[ixj] = ia;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Ascending (key, id) sort of L <= 2 * kST entries with distinct ids: every
// entry's position is its count of smaller (key, id) pairs, so positions are a
// permutation of 0..L-1.
__device__ void rank_sort(uint32_t* key, int* id, int L) {
  uint32_t rk[2];
  int ri[2], pos[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t = threadIdx.x + u * kST;
    pos[u] = -1;
    if (t < L) {
      rk[u] = key[t];
      ri[u] = id[t];
      int cnt = 0;
      for (int q = 0; q < L; ++q) cnt += pair_gt(rk[u], ri[u], key[q], id[q]);
      pos[u] = cnt;
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 2; ++u)
    if (pos[u] >= 0) { key[pos[u]] = rk[u]; id[pos[u]] = ri[u]; }
  __syncthreads();
}

// Merge kClusterCTAs sorted runs held back to back in key/id (run r at
// [off[r], off[r+1]), L <= kMergePer * kST in total) into one ascending (key,
// id) list: an entry's final position is its index in its own run plus, for
// every other run, the count of entries below it there (a binary search).
constexpr int kMergePer = 8;

__device__ void merge_runs(uint32_t* key, int* id, const int* off, int L) {
  uint32_t rk[kMergePer];
  int ri[kMergePer], pos[kMergePer];
#pragma unroll
  for (int u = 0; u < kMergePer; ++u) {
    const int t = threadIdx.x + u * kST;
    pos[u] = -1;
    if (t < L) {
      rk[u] = key[t];
      ri[u] = id[t];
      int own = 0;
      while (t >= off[own + 1]) ++own;
      int p = t - off[own];
      for (int q = 0; q < kClusterCTAs; ++q) {
        if (q == own) continue;
        int lo = off[q], hi = off[q + 1];
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (pair_gt(rk[u], ri[u], key[mid], id[mid])) lo = mid + 1;
          else hi = mid;
        }
        p += lo - off[q];
      }
      pos[u] = p;
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kMergePer; ++u)
    if (pos[u] >= 0) { key[pos[u]] = rk[u]; id[pos[u]] = ri[u]; }
  __syncthreads();
}

// Warp 0: first index j < L at which the running sum of w(j) reaches target
// (L if never). w must be cheap and deterministic.
template <class W>
__device__ int warp_find_cross(int L, unsigned long long target, W w, unsigned long long* total_out) {
  const int lane = threadIdx.x & 31;
  const int chunk = (L + 31) / 32;
  const int a = min(lane * chunk, L), b = min(a + chunk, L);
  unsigned long long loc = 0;
  for (int j = a; j < b; ++j) loc += w(j);
  unsigned long long incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned long long total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  if (total_out) *total_out = total;
  int found = L;
  unsigned long long cum = incl - loc;
  if (cum < target && target <= incl) {
    for (int j = a; j < b; ++j) {
      cum += w(j);
      if (cum >= target) { found = j; break; }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) found = min(found, __shfl_xor_sync(0xFFFFFFFFu, found, o));
  return found;
}

// Weighted selection in a shared-memory list, by one CTA: among the n entries
// (key[i], id[i]) taken in (key asc, id asc) order, find the entry at which the
// running weight first reaches target (1 <= target <= the total). The weight
// is a function of the key (equal keys weigh the same), so digit passes over
// the key settle K*, and the n-th tie at K* (n = ceil(remaining / weight)) is
// the one with n-1 smaller ids (the ties are gathered into tie_buf, which holds
// tie_cap ids). Returns false (nothing decided) when more than tie_cap entries
// tie at K*.
template <class Wk>
__device__ bool list_select(SampleSmem* sm, const uint32_t* key, const int* id, int n, unsigned long long target,
                            Wk wk, int* tie_buf, int tie_cap, uint32_t& Kout, int& idout) {
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int i = threadIdx.x; i < n; i += kST) {
    kmin = min(kmin, key[i]);
    kmax = max(kmax, key[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xFFFFFFFFu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xFFFFFFFFu, kmax, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm->wsum[threadIdx.x >> 5] = ((unsigned long long)kmin << 32) | kmax;
  __syncthreads();
  kmin = 0xFFFFFFFFu;
  kmax = 0u;
  for (int w = 0; w < kST / 32; ++w) {
    kmin = min(kmin, (uint32_t)(sm->wsum[w] >> 32));
    kmax = max(kmax, (uint32_t)sm->wsum[w]);
  }
  const uint32_t diff = kmin ^ kmax;
  int hi = diff ? 31 - __clz(diff) : -1;
  uint32_t mask = hi >= 0 ? ~((hi == 31) ? 0xFFFFFFFFu : ((2u << hi) - 1u)) : 0xFFFFFFFFu;
  uint32_t prefix = kmin & mask;
  unsigned long long* h = sm->hist[0];
  while (hi >= 0) {
    const int lo = hi >= 7 ? hi - 7 : 0;
    const uint32_t dmask = (1u << (hi - lo + 1)) - 1u;
    __syncthreads();
    for (int b = threadIdx.x; b < 256; b += kST) h[b] = 0ull;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kST) {
      const uint32_t k = key[i];
      if ((k & mask) == prefix) atomicAdd(&h[(k >> lo) & dmask], wk(k));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      unsigned long long s8 = 0;
      for (int b = 0; b < 8; ++b) s8 += h[lane * 8 + b];
      unsigned long long incl = s8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      unsigned long long cum = incl - s8;
      const bool mine = cum < target && target <= incl;
      if (mine) {
        for (int b = 0; b < 8; ++b) {
          const unsigned long long t = h[lane * 8 + b];
          if (cum < target && target <= cum + t) {
            sm->sel_bin = lane * 8 + b;
            sm->sel_rem = target - cum;
            break;
          }
          cum += t;
        }
      }
      if (!__ballot_sync(0xFFFFFFFFu, mine) && lane == 0) {  // target above the total: the last bin
        sm->sel_bin = (int)dmask;
        sm->sel_rem = target;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sm->sel_bin << lo;
    mask |= dmask << lo;
    target = sm->sel_rem;
    hi = lo - 1;
  }
  const uint32_t K = prefix;
  const unsigned long long ew = wk(K);
  const unsigned long long need = ew > 0 ? (target + ew - 1) / ew : 1ull;
  // ties at K, gathered, and the need-th of them in id order (each tie's rank
  // is its count of smaller tie ids)
  if (threadIdx.x == 0) { sm->found = -1; sm->ccount = 0; }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kST)
    if (key[i] == K) {
      const int pos = atomicAdd(&sm->ccount, 1);
      if (pos < tie_cap) tie_buf[pos] = id[i];
    }
  __syncthreads();
  const int ties = sm->ccount;
  if (ties > tie_cap) return false;
  const unsigned long long want = need < (unsigned long long)ties ? need : (unsigned long long)ties;
  for (int t = threadIdx.x; t < ties; t += kST) {
    const int me = tie_buf[t];
    int rank = 0;
    for (int q = 0; q < ties; ++q) rank += tie_buf[q] < me;
    if ((unsigned long long)rank == want - 1) sm->found = me;
  }
  __syncthreads();
  Kout = K;
  idout = sm->found;
  __syncthreads();
  return idout >= 0;
}

// Candidate path for a sampled row whose zs holds transformed logits and
// whose global max is mx. Returns false (nothing decided) when the cut is not
// guaranteed to lie inside the exact part of the union.
__device__ bool candidate_transform(Clu& c, const float* zs, int v0, int n, int V, const RowParams& p, float mx,
                                    uint32_t kmin, uint32_t kmax, CandBufs& cb, TDesc& d) {
  SampleSmem* sm = c.sm;
  const int k = (p.top_k > 0 && p.top_k < V) ? p.top_k : 0;
  if (k == 0 && !(p.top_p > 0.f && p.top_p < 1.f) && !(p.min_p > 0.f)) return false;  // nothing to cut
  const int C = k > 0 ? k : kCandTopP;
  int got = n <= cb.C ? -1 : local_candidates(sm, zs, n, v0, C, cb.C, kmin, kmax, cb.ckey, cb.cid);
  if (got < 0) {  // few elements, or a flat slice: select exactly min(C, n)
    uint32_t K;
    int cut;
    local_select(sm, zs, n, v0, min(C, cb.C), kmin, kmax, K, cut);
    if (threadIdx.x == 0) sm->ccount = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += kST) {
      const uint32_t key = desc_key(zs[j]);
      if (in_prefix(key, v0 + j, K, cut)) {
        const int pos = atomicAdd(&sm->ccount, 1);
        cb.ckey[pos] = key;
        cb.cid[pos] = v0 + j;
      }
    }
    __syncthreads();
  }
  // without top-k the union is merged from sorted runs: sort this CTA's run
  if (k == 0 && sm->ccount <= 2 * kST) rank_sort(cb.ckey, cb.cid, sm->ccount);
  unsigned long long sall = 0;
  if (k == 0)
    for (int j = threadIdx.x; j < n; j += kST) sall += to_fix(expf(zs[j] - mx));
  sall = block_sum_u64(sall, sm->wsum);
  if (threadIdx.x == 0) {
    sm->mail[c.ph].u[0] = (unsigned long long)sm->ccount;
    sm->mail[c.ph].u[1] = sall;
    sm->mail[c.ph].i[0] = sm->ccount < n ? 1 : 0;
  }
  Mail* m = c.publish();
  int off[kClusterCTAs + 1];
  off[0] = 0;
  unsigned long long S_all = 0;
  bool truncated = false, runs_sorted = true;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) {
    Mail* x = c.remote(m, r);
    off[r + 1] = off[r] + (int)x->u[0];
    S_all += x->u[1];
    truncated |= x->i[0] != 0;
    runs_sorted &= (int)x->u[0] <= 2 * kST;
  }
  const int L = off[kClusterCTAs];
  int Pd = 1;
  while (Pd < L) Pd <<= 1;
  for (int t = threadIdx.x; t < Pd; t += kST) {
    if (t < L) {
      int r = 0;
      while (t >= off[r + 1]) ++r;
      cb.mkey[t] = c.cl.map_shared_rank(cb.ckey, r)[t - off[r]];
      cb.mid[t] = c.cl.map_shared_rank(cb.cid, r)[t - off[r]];
    } else {
      cb.mkey[t] = 0xFFFFFFFFu;
      cb.mid[t] = 0x7FFFFFFF;
    }
  }
  __syncthreads();
  int Ls = L;  // length of the sorted prefix of mkey / mid
  bool sorted = false;
  if (k > 0 && k <= 2 * kST) {
    // only the top-k of the union matters: select them, then sort just those
    uint32_t Kk = 0xFFFFFFFFu;
    int ck = 0x7FFFFFFF;
    bool sel = L <= k || list_select(sm, cb.mkey, cb.mid, L, (unsigned long long)k,
                                     [](uint32_t) { return 1ull; }, cb.sid, min(cb.C, 2 * kST), Kk, ck);
    if (sel) {
      uint32_t* skey = reinterpret_cast<uint32_t*>(cb.sw);
      if (threadIdx.x == 0) sm->ccount = 0;
      __syncthreads();
      for (int t = threadIdx.x; t < L; t += kST)
        if (in_prefix(cb.mkey[t], cb.mid[t], Kk, ck)) {
          const int pos = atomicAdd(&sm->ccount, 1);
          skey[pos] = cb.mkey[t];
          cb.sid[pos] = cb.mid[t];
        }
      __syncthreads();
      Ls = sm->ccount;
      rank_sort(skey, cb.sid, Ls);
      for (int t = threadIdx.x; t < Ls; t += kST) { cb.mkey[t] = skey[t]; cb.mid[t] = cb.sid[t]; }
      __syncthreads();
      sorted = true;
    }
  }
  if (!sorted) {
    if (k == 0 && runs_sorted && L <= kMergePer * kST) merge_runs(cb.mkey, cb.mid, off, L);
    else bitonic_sort(cb.mkey, cb.mid, Pd);
  }
  if (threadIdx.x < 32) {
    auto fx = [&](int j) { return to_fix(expf(key_to_z(cb.mkey[j]) - mx)); };
    const int Kk = k > 0 ? min(k, Ls) : Ls;
    unsigned long long SE = 0;
    if (k > 0) {
      warp_find_cross(Kk, ~0ull, fx, &SE);
    } else {
      SE = S_all;
    }
    int Kf = Kk;
    bool reached = true;
    if (p.top_p > 0.f && p.top_p < 1.f) {
      const unsigned long long target = (unsigned long long)ceil((double)p.top_p * (double)SE);
      const int j = warp_find_cross(Kk, target, fx, nullptr);
      if (j < Kk) Kf = min(Kf, j + 1);
      else reached = false;
    }
    if (p.min_p > 0.f) {
      const int lane = threadIdx.x;
      int first = Kk;
      for (int j = lane; j < Kk; j += 32)
        if (!(expf(key_to_z(cb.mkey[j]) - mx) >= p.min_p)) { first = j; break; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xFFFFFFFFu, first, o));
      if (first < Kf) { Kf = first; reached = true; }
    }
    if (Kf < 1) Kf = 1;
    bool valid;
    if (k > 0) valid = true;
    else if (!truncated) valid = true;  // the union holds every element
    else valid = reached && Kf < C;
    unsigned long long Sf = 0;
    warp_find_cross(Kf, ~0ull, fx, &Sf);
    if (threadIdx.x == 0) {
      sm->fin_kf = Kf;
      sm->fin_valid = valid ? 1 : 0;
      sm->fin_sf = Sf;
    }
  }
  __syncthreads();
  if (!sm->fin_valid) return false;
  const int Kf = sm->fin_kf;
  d.k_key = 0xFFFFFFFFu;
  d.k_cut = 0x7FFFFFFF;
  if (Kf >= Ls && !truncated) {  // nothing cut
    d.p_key = 0xFFFFFFFFu;
    d.p_cut = 0x7FFFFFFF;
  } else {
    d.p_key = cb.mkey[Kf - 1];
    d.p_cut = cb.mid[Kf - 1];
  }
  d.m = mx;
  d.S = (float)((double)sm->fin_sf / kFix);
  d.kept = Kf;
  __syncthreads();
  return true;
}

// Inverse-CDF draw over the first Kf sorted candidates, in ascending id order,
// with weights to_fix(exp(z - m) / S) -- the q values the draft writes.
__device__ int candidate_draw(const TDesc& d, CandBufs& cb, float u, SampleSmem* sm) {
  const int Kf = d.kept;
  for (int j = threadIdx.x; j < Kf; j += kST) {
    const int id = cb.mid[j];
    int rank = 0;
    for (int i = 0; i < Kf; ++i) rank += cb.mid[i] < id;
    cb.sid[rank] = id;
    cb.sw[rank] = to_fix(expf(key_to_z(cb.mkey[j]) - d.m) / d.S);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long tot = 0;
    warp_find_cross(Kf, ~0ull, [&](int j) { return cb.sw[j]; }, &tot);
    int pick = -1;
    if (tot > 0) {
      const unsigned long long target = (unsigned long long)floor((double)u * (double)tot) + 1ull;
      const int j = warp_find_cross(Kf, target, [&](int j) { return cb.sw[j]; }, nullptr);
      pick = j < Kf ? cb.sid[j] : cb.sid[Kf - 1];
    }
    if (threadIdx.x == 0) sm->fin_draw = pick;
  }
  __syncthreads();
  return sm->fin_draw;
}

// Top-p cut without top-k, for a support too wide for the candidate union.
// Transformed logits z <= mx fall into kFlatBins equal slices of
// [mx - span, mx] (bin 0 holds the largest); the bin index is weakly monotone
// in z, so every bin is a contiguous range of the (key, id) order. One pass
// adds each element's fixed-point weight to its bin; each CTA then sums 256 of
// the cluster's bins, the cluster finds the bin in which the running mass
// reaches ceil(top_p * SE), and that bin's elements are gathered and sorted to
// find the exact crossing element. Elements beyond the span weigh 0 and follow
// every binned element, so they never hold the crossing. Sets the top-p fields
// of d and returns true, or returns false (nothing decided) when the crossing
// bin holds more than kMergePer * kST elements (or 2 * kST in one CTA). Without
// min-p the kept set's fixed-point mass is returned in *S_exact (else 0).
constexpr int kFlatBins = 256 * kClusterCTAs;
constexpr float kFlatSpan = 30.f;  // exp(-30) * 2^40 rounds to 0

__device__ bool flat_top_p(Clu& c, const float* zs, int v0, int n, const RowParams& p, float mx, float zmin,
                           CandBufs& cb, TDesc& d, unsigned long long* S_exact) {
  SampleSmem* sm = c.sm;
  float span = mx - zmin;
  if (!(span > 0.f)) return false;  // one distinct value, or non-finite input
  if (span > kFlatSpan) span = kFlatSpan;
  const float scale = ((float)kFlatBins - 0.01f) / span;
  auto bin_of = [&](float z) {  // kFlatBins for elements beyond the span (and NaN)
    const float t = (mx - z) * scale;
    return t < (float)kFlatBins ? (int)t : kFlatBins;
  };
  unsigned long long* hw = reinterpret_cast<unsigned long long*>(cb.mkey);  // aliases the merge buffers
  for (int b = threadIdx.x; b < kFlatBins; b += kST) hw[b] = 0ull;
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += kST) {
    const float z = zs[j];
    const int b = bin_of(z);
    if (b < kFlatBins) {
      const unsigned long long w = to_fix(expf(z - mx));
      if (w) atomicAdd(&hw[b], w);
    }
  }
  c.cl.sync();
  unsigned long long own = 0;
  if (threadIdx.x < 256) {
    const int b = c.rank * 256 + threadIdx.x;
#pragma unroll
    for (int r = 0; r < kClusterCTAs; ++r) own += c.cl.map_shared_rank(hw, r)[b];
    sm->tot[threadIdx.x] = own;
  }
  own = block_sum_u64(own, sm->wsum);
  if (threadIdx.x == 0) sm->mail[c.ph].u[0] = own;
  Mail* m = c.publish();  // also ends every remote read of hw
  unsigned long long SE = 0;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) SE += c.remote(m, r)->u[0];
  if (SE == 0) return false;
  const unsigned long long target = (unsigned long long)ceil((double)p.top_p * (double)SE);
  unsigned long long tv[kClusterCTAs];
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) tv[r] = c.remote(m, r)->u[0];
  unsigned long long before = 0;
  int owner = kClusterCTAs - 1;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) {
    if (before + tv[r] >= target) { owner = r; break; }
    before += tv[r];
  }
  if (c.rank == owner && threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const unsigned long long need = target - before;
    unsigned long long s8 = 0;
    for (int b = 0; b < 8; ++b) s8 += sm->tot[lane * 8 + b];
    unsigned long long incl = s8;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    unsigned long long cum = incl - s8;
    int fb = -1;
    unsigned long long fr = 0;
    if (cum < need && need <= incl) {
      for (int b = 0; b < 8; ++b) {
        const unsigned long long t = sm->tot[lane * 8 + b];
        if (cum < need && need <= cum + t) {
          fb = owner * 256 + lane * 8 + b;
          fr = need - cum;
          break;
        }
        cum += t;
      }
    }
    const unsigned who = __ballot_sync(0xFFFFFFFFu, fb >= 0);
    const int src = who ? __ffs(who) - 1 : 0;
    fb = __shfl_sync(0xFFFFFFFFu, fb, src);
    fr = __shfl_sync(0xFFFFFFFFu, fr, src);
    if (lane == 0) {
      sm->mail[c.ph].i[0] = fb;  // -1 only if the bins do not add up: nothing is gathered
      sm->mail[c.ph].u[0] = fr;
    }
  }
  m = c.publish();
  const int bstar = c.remote(m, owner)->i[0];
  const unsigned long long rem = c.remote(m, owner)->u[0];
  // gather the crossing bin
  if (threadIdx.x == 0) sm->ccount = 0;
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += kST) {
    const float z = zs[j];
    if (bin_of(z) == bstar) {
      const int pos = atomicAdd(&sm->ccount, 1);
      if (pos < cb.C) {
        cb.ckey[pos] = desc_key(z);
        cb.cid[pos] = v0 + j;
      }
    }
  }
  __syncthreads();
  const int mine = sm->ccount;
  if (threadIdx.x == 0) sm->mail[c.ph].u[0] = (unsigned long long)mine;
  m = c.publish();
  int off[kClusterCTAs + 1];
  off[0] = 0;
  bool over = false;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) {
    const int cnt = (int)c.remote(m, r)->u[0];
    over |= cnt > cb.C || cnt > 2 * kST;
    off[r + 1] = off[r] + cnt;
  }
  const int L = off[kClusterCTAs];
  if (over || L == 0 || L > kMergePer * kST || L > cb.P) return false;
  for (int t = threadIdx.x; t < L; t += kST) {
    int r = 0;
    while (t >= off[r + 1]) ++r;
    cb.mkey[t] = c.cl.map_shared_rank(cb.ckey, r)[t - off[r]];
    cb.mid[t] = c.cl.map_shared_rank(cb.cid, r)[t - off[r]];
  }
  __syncthreads();
  auto wk = [&](uint32_t k) { return to_fix(expf(key_to_z(k) - mx)); };
  uint32_t K;
  int cut;
  if (!list_select(sm, cb.mkey, cb.mid, L, rem, wk, cb.sid, min(cb.C, 2 * kST), K, cut)) return false;
  d.p_key = K;
  d.p_cut = cut;
  d.kept = -1;
  *S_exact = 0ull;
  if (!(p.min_p > 0.f)) {
    // the kept mass, exactly: every bin before the crossing bin (target - rem)
    // plus that bin's entries up to the crossing
    unsigned long long loc = 0;
    for (int t = threadIdx.x; t < L; t += kST)
      if (in_prefix(cb.mkey[t], cb.mid[t], K, cut)) loc += wk(cb.mkey[t]);
    *S_exact = (target - rem) + block_sum_u64(loc, sm->wsum);
  }
  return true;
}

// Transform one row of logits in the cluster. On return zs holds the
// transformed logits (penalised, then / T) and `d` the descriptor; greedy rows
// only get d.argmax.
__device__ bool transform_row(Clu& c, float* zs, uint32_t* bits, int v0, int n, int V, const float* lg,
                              const RowParams& p, TDesc& d, int32_t* status, CandBufs& cb) {
  SampleSmem* sm = c.sm;
  build_bitmap(sm, bits, v0, n);
  // one pass: stage, repetition penalty, argmax of the penalised logits,
  // temperature, and the range of the transformed keys
  const bool pen = p.rep_penalty != 1.f;
  const bool smp = !p.greedy;
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  bool bad = false;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  auto one = [&](int j, float z) {
    if (pen && bit(bits, j)) z = penalize(z, p.rep_penalty);
    if (!isfinite(z)) bad = true;
    if (better(z, v0 + j, bv, bi)) { bv = z; bi = v0 + j; }
    if (smp) {
      z = z / p.temperature + 0.0f;
      const uint32_t k = desc_key(z);
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
    zs[j] = z;
  };
  if ((v0 & 3) == 0 && (n & 3) == 0) {
    const float4* l4 = reinterpret_cast<const float4*>(lg + v0);
    const int n4 = n / 4;
    for (int b0 = 0; b0 < n4; b0 += 8 * kST) {  // all of a batch's loads in flight first
      float4 xb[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j4 = b0 + u * kST + threadIdx.x;
        if (j4 < n4) xb[u] = __ldg(l4 + j4);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j4 = b0 + u * kST + threadIdx.x;
        if (j4 < n4) {
          one(4 * j4, xb[u].x);
          one(4 * j4 + 1, xb[u].y);
          one(4 * j4 + 2, xb[u].z);
          one(4 * j4 + 3, xb[u].w);
        }
      }
    }
  } else {
    for (int j = threadIdx.x; j < n; j += kST) one(j, lg[v0 + j]);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, MTP_ERR_NONFINITE);
  __shared__ float sv[kST / 32];
  __shared__ int si[kST / 32];
  block_argmax(bv, bi, sv, si);
  if (smp) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xFFFFFFFFu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xFFFFFFFFu, kmax, o));
    }
    if ((threadIdx.x & 31) == 0) sm->wsum[threadIdx.x >> 5] = ((unsigned long long)kmin << 32) | kmax;
    __syncthreads();
    kmin = 0xFFFFFFFFu;
    kmax = 0u;
    for (int w = 0; w < kST / 32; ++w) {
      kmin = min(kmin, (uint32_t)(sm->wsum[w] >> 32));
      kmax = max(kmax, (uint32_t)sm->wsum[w]);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    sm->mail[c.ph].f[0] = bv;
    sm->mail[c.ph].i[0] = bi;
    sm->mail[c.ph].f[1] = smp ? key_to_z(kmax) : 0.f;  // smallest transformed logit of the slice
  }
  Mail* m = c.publish();
  float gv = -INFINITY, zmin = INFINITY;
  int gi = 0x7FFFFFFF;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) {
    Mail* x = c.remote(m, r);
    if (better(x->f[0], x->i[0], gv, gi)) { gv = x->f[0]; gi = x->i[0]; }
    zmin = fminf(zmin, x->f[1]);
  }
  d.argmax = gi < V ? gi : 0;  // nothing comparable (every logit NaN): id 0
  d.k_key = 0xFFFFFFFFu;
  d.k_cut = 0x7FFFFFFF;
  d.p_key = 0xFFFFFFFFu;
  d.p_cut = 0x7FFFFFFF;
  d.m = 0.f;
  d.S = 1.f;
  d.kept = 1;
  if (p.greedy) return false;

  d.m = gv / p.temperature + 0.0f;
  const float mx = d.m;
  // rows without top-k try the binned top-p cut first; top-k rows (and rows
  // the binned cut cannot settle) take the candidate union, then the radix path
  const bool flat_ok = !(p.top_k > 0 && p.top_k < V) && p.top_p > 0.f && p.top_p < 1.f;
  unsigned long long S_exact = 0;
  const bool flat_done = flat_ok && flat_top_p(c, zs, v0, n, p, mx, zmin, cb, d, &S_exact);
  if (flat_done && S_exact > 0) {
    d.S = (float)((double)S_exact / kFix);
    return false;
  }
  if (!flat_done && candidate_transform(c, zs, v0, n, V, p, mx, kmin, kmax, cb, d)) return true;

  if (p.top_k > 0 && p.top_k < V) {
    uint32_t K;
    unsigned long long rem;
    radix_select(c, zs, n, [](int) { return true; }, [](int) { return 1ull; },
                 (unsigned long long)p.top_k, K, rem);
    d.k_key = K;
    d.k_cut = tie_cut(c, zs, n, v0, [](int) { return true; }, K, rem);
  }
  const uint32_t kK = d.k_key;
  const int kC = d.k_cut;
  auto in_k = [&](int j) { return in_prefix(desc_key(zs[j]), v0 + j, kK, kC); };
  auto e_of = [&](int j) { return expf(zs[j] - mx); };

  if (p.top_p > 0.f && p.top_p < 1.f && !flat_done) {
    unsigned long long loc = 0;
    for (int j = threadIdx.x; j < n; j += kST)
      if (in_k(j)) loc += to_fix(e_of(j));
    loc = block_sum_u64(loc, sm->wsum);
    const unsigned long long SE = cluster_sum_u64(c, loc);
    const unsigned long long target = (unsigned long long)ceil((double)p.top_p * (double)SE);
    uint32_t K;
    unsigned long long rem;
    radix_select(c, zs, n, in_k, [&](int j) { return to_fix(e_of(j)); }, target, K, rem);
    // every element tied at K carries the same weight
    float zt = 0.f;
    // find the weight of a tied element: any element with key K (zs value is determined by K)
    {
      uint32_t u = ~K;
      u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
      zt = __uint_as_float(u);
    }
    const unsigned long long ew = to_fix(expf(zt - mx));
    const unsigned long long need = ew > 0 ? (rem + ew - 1) / ew : 1ull;
    d.p_key = K;
    d.p_cut = tie_cut(c, zs, n, v0, in_k, K, need);
  }
  const uint32_t pK = d.p_key;
  const int pC = d.p_cut;
  auto kept = [&](int j) {
    const uint32_t key = desc_key(zs[j]);
    if (!in_prefix(key, v0 + j, kK, kC) || !in_prefix(key, v0 + j, pK, pC)) return false;
    return !(p.min_p > 0.f) || expf(zs[j] - mx) >= p.min_p;
  };
  unsigned long long loc = 0, cnt = 0;
  for (int j = threadIdx.x; j < n; j += kST)
    if (kept(j)) { loc += to_fix(e_of(j)); ++cnt; }
  loc = block_sum_u64(loc, sm->wsum);
  cnt = block_sum_u64(cnt, sm->wsum);
  if (threadIdx.x == 0) { sm->mail[c.ph].u[0] = loc; sm->mail[c.ph].u[1] = cnt; }
  m = c.publish();
  unsigned long long S = 0, K = 0;
#pragma unroll
  for (int r = 0; r < kClusterCTAs; ++r) { S += c.remote(m, r)->u[0]; K += c.remote(m, r)->u[1]; }
  d.S = (float)((double)S / kFix);
  d.kept = (int)K;
  return false;
}

// Evaluate the transformed distribution at v from the raw logit.
__device__ __forceinline__ float eval_p(const TDesc& d, const RowParams& p, float raw, bool pen, int v) {
  float z = raw;
  if (pen && p.rep_penalty != 1.f) z = penalize(z, p.rep_penalty);
  if (p.greedy) return v == d.argmax ? 1.f : 0.f;
  z = z / p.temperature + 0.0f;
  const uint32_t key = desc_key(z);
  if (!in_prefix(key, v, d.k_key, d.k_cut) || !in_prefix(key, v, d.p_key, d.p_cut)) return 0.f;
  const float e = expf(z - d.m);
  if (p.min_p > 0.f && !(e >= p.min_p)) return 0.f;
  return e / d.S;
}

__device__ __forceinline__ void slice_of(int V, int rank, int& v0, int& n) {
  const int per = (V + kClusterCTAs - 1) / kClusterCTAs;
  v0 = rank * per;
  n = V - v0;
  if (n > per) n = per;
  if (n < 0) n = 0;
}

// Draft-side sampling (mode 0) or verify descriptors (mode 1).
__global__ void __launch_bounds__(kST, 1) k_sample(const __grid_constant__ SampleArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  Clu c(sm);
  pdl_wait();
  pdl_trigger();
  const int task = blockIdx.x / kClusterCTAs;
  int v0, n;
  slice_of(a.V, c.rank, v0, n);
  const int per = (a.V + kClusterCTAs - 1) / kClusterCTAs;
  float* zs = reinterpret_cast<float*>(dyn + sizeof(SampleSmem));
  uint32_t* bits = reinterpret_cast<uint32_t*>(zs + per);
  CandBufs cb;
  cb.C = a.cand;
  cb.P = a.merge;
  cb.ckey = reinterpret_cast<uint32_t*>((reinterpret_cast<uintptr_t>(bits + (per + 31) / 32) + 15) & ~uintptr_t(15));
  cb.cid = reinterpret_cast<int*>(cb.ckey + cb.C);
  cb.mkey = reinterpret_cast<uint32_t*>(cb.cid + cb.C);
  cb.mid = reinterpret_cast<int*>(cb.mkey + cb.P);
  cb.sid = cb.mid + cb.P;
  cb.sw = reinterpret_cast<unsigned long long*>(cb.sid + cb.C + (cb.C & 1));

  int r, i;
  const float* lg;
  if (a.mode == 0) {
    r = task;
    i = a.pos;
    lg = a.logits + (size_t)r * a.ld;
  } else {
    r = task / (a.depth + 1);
    i = task - r * (a.depth + 1);
    lg = a.logits + ((size_t)r * (a.depth + 1) + i) * a.V;
  }
  const RowParams p = a.p[r];
  load_window(sm, a.hist + (size_t)r * a.W, a.W, a.drafts + (size_t)r * a.depth, i);
  TDesc d;
  const bool fast = transform_row(c, zs, bits, v0, n, a.V, lg, p, d, a.status, cb);

  if (a.mode == 1) {
    if (c.rank == 0 && threadIdx.x == 0) a.desc[task] = d;
  } else if (p.greedy) {
    if (c.rank == 0 && threadIdx.x == 0) a.draft_out[(size_t)r * a.depth + i] = d.argmax;
  } else {
    float* q = a.q + ((size_t)r * a.depth + i) * a.V;
    const float mx = d.m, S = d.S;
    for (int j = threadIdx.x; j < n; j += kST) {
      const uint32_t key = desc_key(zs[j]);
      float pv = 0.f;
      if (in_prefix(key, v0 + j, d.k_key, d.k_cut) && in_prefix(key, v0 + j, d.p_key, d.p_cut)) {
        const float e = expf(zs[j] - mx);
        if (!(p.min_p > 0.f) || e >= p.min_p) pv = e / S;
      }
      zs[j] = pv;  // zs now holds q for this slice
      q[v0 + j] = pv;
    }
    __syncthreads();
    const float u = a.u[(size_t)r * a.depth + i];
    const int x = fast ? candidate_draw(d, cb, u, sm) : cluster_draw(c, n, v0, [&](int j) { return to_fix(zs[j]); }, u);
    if (c.rank == 0 && threadIdx.x == 0) a.draft_out[(size_t)r * a.depth + i] = x >= 0 ? x : d.argmax;
  }
  c.cl.sync();  // keep shared memory alive until every remote read is done
}

// Per-row accept chain and the one draw.
__global__ void __launch_bounds__(kST, 1) k_verify(const __grid_constant__ VerifyArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  Clu c(sm);
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x / kClusterCTAs;
  const int d = a.depth;
  int v0, n;
  slice_of(a.V, c.rank, v0, n);
  const int per = (a.V + kClusterCTAs - 1) / kClusterCTAs;
  uint32_t* bits = reinterpret_cast<uint32_t*>(dyn + sizeof(SampleSmem) + sizeof(float) * per);
  const RowParams p = a.p[r];
  const TDesc* desc = a.desc + (size_t)r * (d + 1);
  const int32_t* dr = a.drafts + (size_t)r * d;
  const float* lg = a.logits + (size_t)r * (d + 1) * a.V;
  const float* uu = a.u + (size_t)r * (d + 1);

  // accept chain, every position at once (every CTA evaluates it identically):
  // lane j of warp 0 tests draft x_{j+1} against target row j. The penalty
  // window of row j is the W tokens starting at j of (history ++ drafts).
  {
    const int32_t* hist = a.hist + (size_t)r * a.W;
    for (int t = threadIdx.x; t < a.W + d; t += kST) sm->wtok[t] = t < a.W ? hist[t] : dr[t - a.W];
    __syncthreads();
    if (threadIdx.x < 32) {
      const int j = threadIdx.x;
      bool acc = false;
      if (j < d) {
        const int x = dr[j];
        if (x >= 0 && x < a.V) {  // an out-of-range draft is rejected, never dereferenced
          if (p.greedy) {
            acc = x == desc[j].argmax;
          } else {
            bool pen = false;
            for (int t = j; t < j + a.W; ++t) pen |= sm->wtok[t] == x;
            const float pv = eval_p(desc[j], p, __ldg(lg + (size_t)j * a.V + x), pen, x);
            // an argmax draft is a point mass: q(x) = 1
            const float qv = p.argmax_draft ? 1.f : __ldg(a.q + ((size_t)r * d + j) * a.V + x);
            acc = qv > 0.f && uu[j] < pv / qv;
          }
        }
      }
      const unsigned rej = ~__ballot_sync(0xFFFFFFFFu, acc) & (d >= 32 ? 0xFFFFFFFFu : ((1u << d) - 1u));
      if (j == 0) sm->fin_kf = rej ? __ffs(rej) - 1 : d;
    }
    __syncthreads();
  }
  const int nacc = sm->fin_kf;
  int y;
  if (p.greedy) {
    y = desc[nacc].argmax;
  } else {
    load_window(sm, a.hist + (size_t)r * a.W, a.W, dr, nacc);
    build_bitmap(sm, bits, v0, n);
    const TDesc dn = desc[nacc];
    const float* ln = lg + (size_t)nacc * a.V;
    const float* qn = nacc < d && !p.argmax_draft ? a.q + ((size_t)r * d + nacc) * a.V : nullptr;
    // the rejected draft of an argmax-drafted row: its q is 1 there, 0 elsewhere
    const int xr = nacc < d && p.argmax_draft ? dr[nacc] : -1;
    float* ws = reinterpret_cast<float*>(dyn + sizeof(SampleSmem));
    // draw weights of this slice, computed once: the residual max(p - q, 0)
    // after a rejection, else p (the bonus row)
    auto stage = [&](bool residual) {
      const bool dense_q = residual && qn != nullptr;
      const bool vec = (n & 3) == 0 && (reinterpret_cast<uintptr_t>(ln + v0) & 15) == 0 &&
                       (!dense_q || (reinterpret_cast<uintptr_t>(qn + v0) & 15) == 0);
      if (vec) {
        const float4* l4 = reinterpret_cast<const float4*>(ln + v0);
        const float4* q4 = dense_q ? reinterpret_cast<const float4*>(qn + v0) : nullptr;
        const int n4 = n / 4;
        for (int b0 = 0; b0 < n4; b0 += 4 * kST) {
          float4 lv[4], qv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j4 = b0 + u * kST + threadIdx.x;
            if (j4 < n4) {
              lv[u] = __ldg(l4 + j4);
              qv[u] = dense_q ? __ldg(q4 + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j4 = b0 + u * kST + threadIdx.x;
            if (j4 < n4) {
              const float lx[4] = {lv[u].x, lv[u].y, lv[u].z, lv[u].w};
              const float qx[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = 4 * j4 + e;
                const float pv = eval_p(dn, p, lx[e], bit(bits, j), v0 + j);
                const float rv = residual ? pv - (v0 + j == xr ? 1.f : qx[e]) : pv;
                ws[j] = rv > 0.f ? rv : 0.f;
              }
            }
          }
        }
        __syncthreads();
        return;
      }
      for (int b0 = 0; b0 < n; b0 += 8 * kST) {
        float lv[8], qv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = b0 + u * kST + threadIdx.x;
          if (j < n) {
            lv[u] = __ldg(ln + v0 + j);
            qv[u] = dense_q ? __ldg(qn + v0 + j) : 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = b0 + u * kST + threadIdx.x;
          if (j < n) {
            const float pv = eval_p(dn, p, lv[u], bit(bits, j), v0 + j);
            const float rv = residual ? pv - (v0 + j == xr ? 1.f : qv[u]) : pv;
            ws[j] = rv > 0.f ? rv : 0.f;
          }
        }
      }
      __syncthreads();
    };
    y = -1;
    if (nacc < d) {
      stage(true);
      y = cluster_draw(c, n, v0, [&](int j) { return to_fix(ws[j]); }, uu[d]);
    }
    if (y < 0) {
      stage(false);
      y = cluster_draw(c, n, v0, [&](int j) { return to_fix(ws[j]); }, uu[d]);
    }
    if (y < 0) y = dn.argmax;
  }
  if (c.rank == 0 && threadIdx.x == 0) {
    a.n_acc[r] = nacc;
    int32_t* o = a.out_tok + (size_t)r * (d + 1);
    for (int i = 0; i <= d; ++i) o[i] = i < nacc ? dr[i] : (i == nacc ? y : -1);
    if (a.h_rec) {
      // the record's tokens are visible to the host before its count
      int32_t* hr = a.h_rec + (size_t)r * (d + 2);
      for (int i = 0; i <= d; ++i) hr[1 + i] = o[i];
      st_release_sys(hr, nacc);
    }
    if (a.stats) {
      int32_t* s = a.stats + (size_t)r * (d + 2);
      s[0] += 1;
      if (nacc < d) s[1] += 1;
      for (int i = 1; i <= nacc; ++i) s[1 + i] += 1;
    }
  }
  c.cl.sync();
}

// Verify of greedy rows without a repetition penalty, in one launch. With
// point-mass p and q the Leviathan/Chen rule accepts x_i exactly when x_i is
// the argmax of target row i-1, and the correction or bonus token is the
// argmax of the first unmatched row. One cluster per row (16 CTAs where the
// device schedules them, else 8, halved while rows x CTAs exceeds the SM
// count): each CTA takes the argmax (value desc, id
// asc) of its vocabulary slice for every position, with the loads of several
// positions in flight together, the cluster combines the slices through DSMEM,
// and rank 0 walks the accept chain and writes the outputs.
constexpr int kGreedyMaxPos = 17;
constexpr int kGreedyBuf = 16;  // float4 loads in flight per thread
constexpr int kGreedyGroup = 4;  // positions reduced together

template <bool WIDE>
__global__ void __launch_bounds__(kST, WIDE ? 2 : 1) k_verify_greedy(const __grid_constant__ VerifyArgs a) {
  __shared__ float s_v[kGreedyMaxPos];
  __shared__ int s_i[kGreedyMaxPos];
  __shared__ int s_am[kGreedyMaxPos];
  __shared__ float wv[kGreedyGroup][kST / 32];
  __shared__ int wi[kGreedyGroup][kST / 32];
  cg::cluster_group cl = cg::this_cluster();
  const int nc = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int r = blockIdx.x / nc;
  const int d = a.depth;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = ((a.V + nc - 1) / nc + 3) & ~3;
  const int v0 = min(rank * per, a.V);
  const int n = min(per, a.V - v0);
  pdl_wait();
  pdl_trigger();
  const float* lg = a.logits + (size_t)r * (d + 1) * a.V;
  bool bad = false;
  const bool vec = a.vec_ok != 0;
  const int n4 = vec ? n / 4 : 0;
  const int U = max(1, (n4 + kST - 1) / kST);
  const int G = vec ? max(1, min(kGreedyGroup, kGreedyBuf / U)) : 1;
  if constexpr (WIDE) {
    // Wide slices (many rows per launch, or a large vocabulary; 16-byte
    // loads): every position's slice streamed back to back in chunks of B
    // loads per thread, the next chunk in flight while the current one is
    // reduced, across position boundaries too. Four independent (value, id)
    // chains per thread, one per vector lane; the block argmax of a position
    // is taken when its last chunk has been reduced.
    // (The launcher takes this instance only where the 16-byte loads apply.
    // Two CTAs share an SM: B = 4 keeps a thread within 64 registers.)
    constexpr int B = 4;
    constexpr int step = B * kST;
    if (threadIdx.x <= d) { s_v[threadIdx.x] = -INFINITY; s_i[threadIdx.x] = 0x7FFFFFFF; }  // an empty slice
    __syncthreads();
    const int nch = (n4 + step - 1) / step;
    const int total = (d + 1) * nch;
    float v[4];
    int id[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) { v[q] = -INFINITY; id[q] = 0x7FFFFFFF; }
    float4 b0[B], b1[B];
    auto load = [&](float4 (&b)[B], int c) {
      if (c >= total) return;
      const int pi = c / nch, base = (c - pi * nch) * step;
      const float4* src = reinterpret_cast<const float4*>(lg + (size_t)pi * a.V + v0);
#pragma unroll
      for (int e = 0; e < B; ++e) {
        const int j4 = base + e * kST + threadIdx.x;
        if (j4 < n4) { const uint4 t = ldg_stream(src + j4); b[e] = make_float4(__uint_as_float(t.x), __uint_as_float(t.y), __uint_as_float(t.z), __uint_as_float(t.w)); }
      }
    };
    auto reduce = [&](const float4 (&b)[B], int c) {
      if (c >= total) return;  // uniform over the block, like the test below
      const int pi = c / nch, base = (c - pi * nch) * step;
#pragma unroll
      for (int e = 0; e < B; ++e) {
        const int j4 = base + e * kST + threadIdx.x;
        if (j4 < n4) {
          const float x[4] = {b[e].x, b[e].y, b[e].z, b[e].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (!isfinite(x[q])) bad = true;
            if (better(x[q], v0 + 4 * j4 + q, v[q], id[q])) { v[q] = x[q]; id[q] = v0 + 4 * j4 + q; }
          }
        }
      }
      if (c - pi * nch == nch - 1) {  // the position's last chunk: its block argmax
        float bvv = -INFINITY;
        int bii = 0x7FFFFFFF;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (better(v[q], id[q], bvv, bii)) { bvv = v[q]; bii = id[q]; }
          v[q] = -INFINITY;
          id[q] = 0x7FFFFFFF;
        }
        warp_argmax(bvv, bii);
        if (lane == 0) { wv[0][warp] = bvv; wi[0][warp] = bii; }
        __syncthreads();
        if (warp == 0) {
          float x = lane < kST / 32 ? wv[0][lane] : -INFINITY;
          int i = lane < kST / 32 ? wi[0][lane] : 0x7FFFFFFF;
          warp_argmax(x, i);
          if (lane == 0) { s_v[pi] = x; s_i[pi] = i; }
        }
        __syncthreads();
      }
    };
    load(b0, 0);
    for (int c = 0; c < total; c += 2) {
      load(b1, c + 1);
      reduce(b0, c);
      load(b0, c + 2);
      reduce(b1, c + 1);
    }
  } else  // grouped positions, all loads of a group in flight together
  for (int i0 = 0; i0 <= d; i0 += G) {
    const int gi = min(G, d + 1 - i0);
    float bv[kGreedyGroup];
    int bi[kGreedyGroup];
#pragma unroll
    for (int e = 0; e < kGreedyGroup; ++e) { bv[e] = -INFINITY; bi[e] = 0x7FFFFFFF; }
    if (vec) {
      float4 buf[kGreedyBuf];
#pragma unroll
      for (int e = 0; e < kGreedyBuf; ++e) {
        const int pi = e / U, j4 = (e - pi * U) * kST + threadIdx.x;
        if (pi < gi && j4 < n4)
          buf[e] = __ldg(reinterpret_cast<const float4*>(lg + (size_t)(i0 + pi) * a.V + v0) + j4);
      }
#pragma unroll
      for (int e = 0; e < kGreedyBuf; ++e) {
        const int pi = e / U, j4 = (e - pi * U) * kST + threadIdx.x;
        if (pi < gi && j4 < n4) {
          const float x[4] = {buf[e].x, buf[e].y, buf[e].z, buf[e].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (!isfinite(x[q])) bad = true;
            // slot pi of bv/bi holds position i0 + pi (e is ascending in pi)
#pragma unroll
            for (int t = 0; t < kGreedyGroup; ++t)
              if (t == pi && better(x[q], v0 + 4 * j4 + q, bv[t], bi[t])) { bv[t] = x[q]; bi[t] = v0 + 4 * j4 + q; }
          }
        }
      }
      // the tail that does not fill a float4
      for (int j = 4 * n4 + threadIdx.x; j < n; j += kST)
        for (int pi = 0; pi < gi; ++pi) {
          const float x = __ldg(lg + (size_t)(i0 + pi) * a.V + v0 + j);
          if (!isfinite(x)) bad = true;
#pragma unroll
          for (int t = 0; t < kGreedyGroup; ++t)
            if (t == pi && better(x, v0 + j, bv[t], bi[t])) { bv[t] = x; bi[t] = v0 + j; }
        }
    } else {
      for (int j = threadIdx.x; j < n; j += kST) {
        const float x = __ldg(lg + (size_t)i0 * a.V + v0 + j);
        if (!isfinite(x)) bad = true;
        if (better(x, v0 + j, bv[0], bi[0])) { bv[0] = x; bi[0] = v0 + j; }
      }
    }
    // block argmax of every position of the group: warps, then one warp each
#pragma unroll
    for (int t = 0; t < kGreedyGroup; ++t) {
      if (t < gi) {
        float v = bv[t];
        int i = bi[t];
        warp_argmax(v, i);
        if (lane == 0) { wv[t][warp] = v; wi[t][warp] = i; }
      }
    }
    __syncthreads();
    if (warp < gi) {
      float v = lane < kST / 32 ? wv[warp][lane] : -INFINITY;
      int i = lane < kST / 32 ? wi[warp][lane] : 0x7FFFFFFF;
      warp_argmax(v, i);
      if (lane == 0) { s_v[i0 + warp] = v; s_i[i0 + warp] = i; }
    }
    __syncthreads();
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(a.status, MTP_ERR_NONFINITE);
  cl.sync();
  if (rank == 0 && warp <= d) {
    // warp i combines position i: lane q reads CTA q's slice argmax
    float v = -INFINITY;
    int id = 0x7FFFFFFF;
    if (lane < nc) {
      v = *cl.map_shared_rank(&s_v[warp], lane);
      id = *cl.map_shared_rank(&s_i[warp], lane);
    }
    warp_argmax(v, id);
    if (lane == 0) s_am[warp] = id < a.V ? id : 0;  // nothing comparable (every logit NaN): id 0
  }
  __syncthreads();
  if (rank == 0 && warp == 0) {
    const int am = lane <= d ? s_am[lane] : 0x7FFFFFFF;
    const int32_t* dr = a.drafts + (size_t)r * d;
    // accepted prefix: drafts x_i (i = 1..d) equal to the argmax of row i-1
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
  cl.sync();  // keep shared memory alive until rank 0 has read it
}

// ------------------------------------------------------------ streaming verify
// Throughput form of the sampled verify for many tasks (rows x positions) whose
// sampled rows all cut to a top-k of at most kStreamTopK. With top-k set, the
// kept set and every probability the verify needs come from the k largest
// transformed logits, so one CTA per task reads its target row once: it
// penalises, tracks the argmax, and keeps the (key, id)-smallest candidates in
// shared memory under a threshold that tightens to the exact k-th each time the
// buffer fills. The descriptor it writes is the one the cluster path
// computes (same keys, same fixed-point sums, same cut rules); the task also
// evaluates the accept test of the draft its row judges and stores its kept
// list. k_verify_finish then walks each row's accept chain and draws the
// correction or bonus token over the stopping position's kept list, in id
// order, with the cluster path's inverse-CDF rule.
constexpr int kStreamCap = 1536;  // candidate entries (>= 2 kStreamTopK), small enough for two CTAs per SM
constexpr int kStreamChunk = 32 * kST;  // elements per round of the 4-byte-load path (32 per thread)

constexpr int kRingChunk = 8192;            // floats per ring stage (32 KB)
constexpr size_t kStreamSmemMax = 226 * 1024;  // dynamic shared memory the streaming kernel may take

// Dynamic shared memory of the streaming kernel: sampler scratch, candidate
// buffers, the penalty bitmap, then (16-byte rows) a ring of ns stages of
// kRingChunk floats and their mbarriers. The ring takes 2 stages where they
// fit (*ring_ns = 0 otherwise); at V = 152064 the whole is about 108 KB, so
// two CTAs share an SM.
struct StreamLayout {
  size_t ckey, bits, ring, bar, total;
  int ns;
  __host__ __device__ StreamLayout(int V, int ns_want) {
    ckey = (sizeof(SampleSmem) + 15) & ~size_t(15);
    bits = ckey + 3 * sizeof(uint32_t) * kStreamCap;
    ring = (bits + sizeof(uint32_t) * ((V + 31) / 32 + 1) + 127) & ~size_t(127);
    ns = ns_want;
    bar = ring + (size_t)ns * kRingChunk * sizeof(float);
    total = bar + 16 * (size_t)(ns > 0 ? ns : 1) + 16;  // full and empty mbarriers
  }
};

size_t verify_stream_smem(int V, int* ring_ns) {
  const StreamLayout base(V, 0);
  int ns = (int)((kStreamSmemMax - base.ring - 64) / (kRingChunk * sizeof(float)));
  ns = ns > 2 ? 2 : ns;  // two stages: at the full vocabulary two CTAs fit on an SM
  if (ns < 2) ns = 0;
  if (ring_ns) *ring_ns = ns;
  return StreamLayout(V, ns).total;
}

// Keep exactly the k (key, id)-smallest of the buffered candidates; the
// threshold becomes the k-th. Out of line: it runs rarely, and the streaming
// loop keeps its registers.
// Smallest penalised logit z whose transformed value z / T + 0 reaches the
// transformed value of key K (division rounds monotonically, so every z below
// it transforms below): the streaming loop skips the division for them. -inf
// (no skipping) when K admits everything or the search does not settle.
__device__ float stream_z_cut(uint32_t K, float T) {
  if (K == 0xFFFFFFFFu) return -INFINITY;
  const float tt = key_to_z(K);
  if (!isfinite(tt)) return -INFINITY;
  auto reaches = [&](float z) { return z / T + 0.0f >= tt; };
  float z = tt * T;
  if (!isfinite(z)) return -INFINITY;
  for (int it = 0; it < 64; ++it) {
    if (reaches(z)) {
      const float lo = nextafterf(z, -INFINITY);
      if (!reaches(lo)) return z;
      z = lo;
    } else {
      z = nextafterf(z, INFINITY);
    }
  }
  return -INFINITY;
}

// The k-th entry (1 <= k <= n) of n shared-memory (key, id) pairs with
// distinct ids, in (key asc, id asc) order: digit passes of up to 8 bits from
// the highest bit where the keys differ, counting into 32-bit bins with one
// atomic per group of lanes that share a digit; then the ties at the settled
// key are gathered (tie holds n ids) and the wanted one is the tie with the
// right count of smaller ids.
__device__ void stream_select(SampleSmem* sm, const uint32_t* key, const int* id, int n, int k, int* tie,
                              uint32_t& Kout, int& idout) {
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int i = threadIdx.x; i < n; i += kST) {
    kmin = min(kmin, key[i]);
    kmax = max(kmax, key[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xFFFFFFFFu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xFFFFFFFFu, kmax, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm->wsum[threadIdx.x >> 5] = ((unsigned long long)kmin << 32) | kmax;
  __syncthreads();
  kmin = 0xFFFFFFFFu;
  kmax = 0u;
  for (int w = 0; w < kST / 32; ++w) {
    kmin = min(kmin, (uint32_t)(sm->wsum[w] >> 32));
    kmax = max(kmax, (uint32_t)sm->wsum[w]);
  }
  const uint32_t diff = kmin ^ kmax;
  int hi = diff ? 31 - __clz(diff) : -1;
  uint32_t mask = hi >= 0 ? ~((hi == 31) ? 0xFFFFFFFFu : ((2u << hi) - 1u)) : 0xFFFFFFFFu;
  uint32_t prefix = kmin & mask;
  uint32_t target = (uint32_t)k;
  uint32_t* h = reinterpret_cast<uint32_t*>(sm->hist[0]);
  while (hi >= 0) {
    const int lo = hi >= 7 ? hi - 7 : 0;
    const uint32_t dmask = (1u << (hi - lo + 1)) - 1u;
    __syncthreads();
    for (int b = threadIdx.x; b < 256; b += kST) h[b] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kST) {
      const uint32_t kk = key[i];
      if ((kk & mask) == prefix) {
        const uint32_t dg = (kk >> lo) & dmask;
        const unsigned peers = __match_any_sync(__activemask(), dg);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[dg], (uint32_t)__popc(peers));
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      uint32_t s8 = 0;
      for (int b = 0; b < 8; ++b) s8 += h[lane * 8 + b];
      uint32_t incl = s8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      uint32_t cum = incl - s8;
      if (cum < target && target <= incl) {
        for (int b = 0; b < 8; ++b) {
          const uint32_t t = h[lane * 8 + b];
          if (cum < target && target <= cum + t) {
            sm->sel_bin = lane * 8 + b;
            sm->sel_rem = target - cum;
            break;
          }
          cum += t;
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sm->sel_bin << lo;
    mask |= dmask << lo;
    target = (uint32_t)sm->sel_rem;
    hi = lo - 1;
  }
  const uint32_t K = prefix;
  if (threadIdx.x == 0) { sm->found = -1; sm->ccount = 0; }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kST)
    if (key[i] == K) tie[atomicAdd(&sm->ccount, 1)] = id[i];
  __syncthreads();
  const int ties = sm->ccount;
  for (int t = threadIdx.x; t < ties; t += kST) {
    const int me = tie[t];
    int rank = 0;
    for (int q = 0; q < ties; ++q) rank += tie[q] < me;
    if ((uint32_t)rank == target - 1) sm->found = me;
  }
  __syncthreads();
  Kout = K;
  idout = sm->found;
  __syncthreads();
}

__device__ __noinline__ void stream_compact(SampleSmem* sm, uint32_t* ckey, int* cid, int* tie, int k, int* cnt,
                                            int* kept_n, uint32_t* thrK, int* thrI, float* zcut, float T) {
  const int n = min(*cnt, kStreamCap);
  uint32_t K;
  int cut;
  stream_select(sm, ckey, cid, n, k, tie, K, cut);
  if (threadIdx.x == 0) *kept_n = 0;
  __syncthreads();
  for (int t = threadIdx.x; t < n; t += kST)
    if (in_prefix(ckey[t], cid[t], K, cut)) {
      const int pos = atomicAdd(kept_n, 1);
      tie[pos] = (int)ckey[t];
      tie[kStreamTopK + pos] = cid[t];
    }
  __syncthreads();
  const int kept = *kept_n;
  for (int t = threadIdx.x; t < kept; t += kST) { ckey[t] = (uint32_t)tie[t]; cid[t] = tie[kStreamTopK + t]; }
  if (threadIdx.x == 0) { *cnt = kept; *thrK = K; *thrI = cut; *zcut = stream_z_cut(K, T); }
  __syncthreads();
}

template <bool VEC>
__global__ void __launch_bounds__(kST, 2) k_verify_stream(const __grid_constant__ VerifyArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  const StreamLayout lay(a.V, VEC ? a.ring_ns : 0);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(dyn + lay.ckey);
  int* cid = reinterpret_cast<int*>(ckey + kStreamCap);
  int* tie = cid + kStreamCap;
  uint32_t* bits = reinterpret_cast<uint32_t*>(dyn + lay.bits);
  float* ring = reinterpret_cast<float*>(dyn + lay.ring);
  uint64_t* bar = reinterpret_cast<uint64_t*>(dyn + lay.bar);
  __shared__ int s_cnt, s_kept;
  __shared__ uint32_t s_thrK;
  __shared__ int s_thrI;
  __shared__ float s_zc;
  __shared__ float s_bv[kST / 32];
  __shared__ int s_bi[kST / 32];
  pdl_wait();
  pdl_trigger();
  const int d = a.depth, V = a.V;
  const int task = blockIdx.x, r = task / (d + 1), i = task - r * (d + 1);
  const RowParams p = a.p[r];
  const float* lg = a.logits + ((size_t)r * (d + 1) + i) * V;
  const int32_t* dr = a.drafts + (size_t)r * d;
  // 16-byte rows stream through the ring: its first stages are requested
  // before the rest of the setup
  const int NS = lay.ns;
  const int nch = (V + kRingChunk - 1) / kRingChunk;
  const unsigned lim = a.wait_limit ? a.wait_limit : kWaitLimit;
  auto issue = [&](int c) {
    if (c == a.stall_stage) return;  // test hook: this stage never lands, its waits run out
    const int slot = c % NS;
    const uint32_t bytes = (uint32_t)min(kRingChunk, V - c * kRingChunk) * 4u;
    mbar_expect_tx(smem_u32(&bar[slot]), bytes);
    bulk_g2s(smem_u32(ring + (size_t)slot * kRingChunk), lg + (size_t)c * kRingChunk, bytes, smem_u32(&bar[slot]));
  };
  uint64_t* empty = bar + NS;  // a stage is free again once every warp has arrived on it
  if constexpr (VEC) {
    if (threadIdx.x == 0) {
      for (int s = 0; s < NS; ++s) {
        mbar_init(smem_u32(&bar[s]), 1);
        mbar_init(smem_u32(&empty[s]), kST / 32);
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0)
      for (int c = 0; c < min(nch, NS); ++c) issue(c);
  }
  load_window(sm, a.hist + (size_t)r * a.W, a.W, dr, i);
  const bool pen = p.rep_penalty != 1.f;
  if (pen) build_bitmap(sm, bits, 0, V);
  const bool smp = !p.greedy;
  // Every row keeps candidates: a sampled row its top-k of the transformed
  // logits z / T, a greedy row its top-1 of z (T = 1).
  const int kk = smp ? p.top_k : 1;  // 1 <= top_k <= kStreamTopK < V (checked by the host)
  const float TT = smp ? p.temperature : 1.f;
  if (threadIdx.x == 0) { s_cnt = 0; s_thrK = 0xFFFFFFFFu; s_thrI = 0x7FFFFFFF; s_zc = -INFINITY; }
  __syncthreads();

  auto pen_z = [&](float raw, int j) { return pen && bit(bits, j) ? penalize(raw, p.rep_penalty) : raw; };
  auto key_of = [&](float raw, int j) { return desc_key(pen_z(raw, j) / TT + 0.0f); };
  auto append = [&](uint32_t key, int j) {
    const int pos = atomicAdd(&s_cnt, 1);
    if (pos < kStreamCap) { ckey[pos] = key; cid[pos] = j; return true; }
    return false;
  };
  auto compact = [&]() { stream_compact(sm, ckey, cid, tie, kk, &s_cnt, &s_kept, &s_thrK, &s_thrI, &s_zc, TT); };
  // A first threshold before anything is kept, from the first span of the
  // row: the kk-th smallest of the threads' smallest keys there. At least kk
  // elements lie at or below it, so the top kk all do (kept inclusively).
  auto first_threshold = [&](uint32_t mk) {
    uint32_t K0;
    int i0;
    block_kth_pair(mk, threadIdx.x, kk, reinterpret_cast<uint32_t*>(tie), tie + kST, sm, K0, i0);
    if (threadIdx.x == 0) { s_thrK = K0; s_thrI = 0x7FFFFFFF; s_zc = stream_z_cut(K0, TT); }
    __syncthreads();
  };
  // One element of the stream (window tokens arrive as NaN and fail every
  // test: they are offered after the stream with their penalised logits).
  // An append that finds the buffer full raises `overflow`; the rescan below
  // then recovers it.
  // The argmax of the penalised logits is tracked on the elements that reach
  // zc: the largest z has the smallest key, so it always does.
  bool overflow = false;
  float gv = -INFINITY;
  int gi = 0x7FFFFFFF;
  // x * 0 is 0 for every finite x and NaN for NaN or an infinity: one
  // dependent FMA per element finds a non-finite logit anywhere in the row
  float nf = 0.f;
  auto offer = [&](float z, int j, uint32_t thrK, int thrI, float zc) {
    if (z >= zc) {  // below zc an element cannot pass: no division
      if (better(z, j, gv, gi)) { gv = z; gi = j; }
      const uint32_t key = desc_key(z / TT + 0.0f);
      if (in_prefix(key, j, thrK, thrI) && !append(key, j)) overflow = true;
    }
  };
  const float kNaN = __int_as_float(0x7FC00000);
  auto comp = [](const float4& v, int q) { return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w)); };
  if constexpr (VEC) {
    // thread t takes float4 u kST + t (u < 4) of each 8192-float stage;
    // no barriers between elements, one per stage
    uint32_t thrK = 0xFFFFFFFFu;
    int thrI = 0x7FFFFFFF;
    float zc = -INFINITY;
    bool ok = true;
    int issued = min(nch, NS);
    // No block barrier per stage: each warp waits for a stage to land, and
    // releases it on the stage's empty barrier when done; thread 0 refills a
    // stage once all warps have released it. A wait that runs out ends the
    // loop for its whole warp (at the first stage, before the block-wide
    // threshold, for the whole block), so no barrier is left half-reached.
    for (int c = 0; c < nch; ++c) {
      const int slot = c % NS;
      const bool got = mbar_wait(smem_u32(&bar[slot]), (c / NS) & 1, lim);
      if (c == 0 ? !__syncthreads_and(got) : !__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }
      const float4* src = reinterpret_cast<const float4*>(ring + (size_t)slot * kRingChunk);
      const int n4 = min(kRingChunk, V - c * kRingChunk) / 4;
      if (c == 0) {
        uint32_t mk = 0xFFFFFFFFu;
        for (int u = 0; u < kRingChunk / 4 / kST; ++u) {
          const int j4 = u * kST + threadIdx.x;
          if (j4 < n4) {
            const float4 v = src[j4];
#pragma unroll
            for (int q = 0; q < 4; ++q) mk = min(mk, key_of(comp(v, q), 4 * j4 + q));
          }
        }
        first_threshold(mk);
        thrK = s_thrK;
        thrI = s_thrI;
        zc = s_zc;
      }
      // one compare per element into a mask (bit 4u + q); the few elements
      // at or above zc are then taken one by one from the stage
      uint32_t hit = 0;
#pragma unroll
      for (int u = 0; u < kRingChunk / 4 / kST; ++u) {
        const int j4 = u * kST + threadIdx.x;
        if (j4 < n4) {
          const float4 v = src[j4];
          const int j0 = c * kRingChunk + 4 * j4;
          const uint32_t skip = pen ? bits[j0 >> 5] >> (j0 & 31) : 0u;  // window tokens: offered after
          const uint32_t h = (v.x >= zc ? 1u : 0u) | (v.y >= zc ? 2u : 0u) | (v.z >= zc ? 4u : 0u) |
                             (v.w >= zc ? 8u : 0u);
          hit |= (h & ~skip & 0xFu) << (4 * u);
          nf = fmaf(v.w, 0.f, fmaf(v.z, 0.f, fmaf(v.y, 0.f, fmaf(v.x, 0.f, nf))));
        }
      }
      while (hit) {
        const int bq = __ffs(hit) - 1;
        hit &= hit - 1;
        const int j4 = (bq >> 2) * kST + threadIdx.x;
        offer(reinterpret_cast<const float*>(src)[4 * j4 + (bq & 3)], c * kRingChunk + 4 * j4 + (bq & 3), thrK, thrI,
              zc);
      }
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&empty[slot]));
      bool refilled = true;
      if (threadIdx.x == 0 && issued < nch) {
        // every warp has released this stage: refill it
        refilled = mbar_wait(smem_u32(&empty[slot]), (c / NS) & 1, lim);
        if (refilled) issue(issued);
      }
      if (threadIdx.x < 32 && !__all_sync(0xFFFFFFFFu, refilled)) { ok = false; break; }
      issued = min(nch, issued + 1);
    }
    if (__syncthreads_or(!ok)) {
      // a stage never arrived: raise the status word, let the copies in
      // flight land before the shared memory is released, and leave a task
      // result that stays in range (no accept, the kept list {0}); the row's
      // outputs are not meaningful and the status word says so
      if (threadIdx.x == 0) {
        flag_status(a.status, MTP_ERR_TIMEOUT);
        for (int j = max(0, issued - NS); j < issued; ++j) mbar_wait(smem_u32(&bar[j % NS]), (j / NS) & 1, lim);
        TDesc dd;
        dd.argmax = 0;
        dd.k_key = 0xFFFFFFFFu;
        dd.k_cut = 0x7FFFFFFF;
        dd.p_key = desc_key(0.f);
        dd.p_cut = 0;
        dd.m = 0.f;
        dd.S = 1.f;
        dd.kept = 1;
        a.wdesc[task] = dd;
        a.acc[task] = 0;
        a.kid[(size_t)task * kStreamTopK] = 0;
        a.kkey[(size_t)task * kStreamTopK] = dd.p_key;
      }
      return;  // block-uniform: every thread saw the same vote
    }
  } else {
    // 4-byte loads: thread t takes element e kST + t (e < 32) of each span of
    // kStreamChunk, the next span's loads in flight while one is processed
    const int nround = (V + kStreamChunk - 1) / kStreamChunk;
    auto load = [&](float (&b)[32], int c) {
      if (c >= nround) return;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int j = c * kStreamChunk + e * kST + threadIdx.x;
        b[e] = j < V ? __ldg(lg + j) : kNaN;
      }
    };
    float nb[32];
    load(nb, 0);
    {
      uint32_t mk = 0xFFFFFFFFu;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int j = e * kST + threadIdx.x;
        if (j < V) mk = min(mk, key_of(nb[e], j));
      }
      first_threshold(mk);
    }
    const uint32_t thrK = s_thrK;
    const int thrI = s_thrI;
    const float zc = s_zc;
    for (int c = 0; c < nround; ++c) {
      float b[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) b[e] = nb[e];
      load(nb, c + 1);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int j = c * kStreamChunk + e * kST + threadIdx.x;
        if (j < V) nf = fmaf(b[e], 0.f, nf);
        offer(j < V && !(pen && bit(bits, j)) ? b[e] : kNaN, j, thrK, thrI, zc);
      }
    }
  }
  if (__syncthreads_or(isnan(nf)) && threadIdx.x == 0) flag_status(a.status, MTP_ERR_NONFINITE);
  if (pen) {
    // the window tokens the stream skipped, each once, with their penalised
    // logits, under the final threshold
    __syncthreads();
    const uint32_t thrK = s_thrK;
    const int thrI = s_thrI;
    for (int t = threadIdx.x; t < sm->nwin; t += kST) {
      const int v = sm->wtok[t];
      bool first = v >= 0 && v < V;
      for (int u = 0; u < t && first; ++u) first = sm->wtok[u] != v;
      if (!first) continue;
      const float z = pen_z(__ldg(lg + v), v);
      if (better(z, v, gv, gi)) { gv = z; gi = v; }
      const uint32_t key = desc_key(z / TT + 0.0f);
      if (in_prefix(key, v, thrK, thrI) && !append(key, v)) overflow = true;
    }
    __syncthreads();
  }
  // Overflow (rare: the first threshold admitted more than the buffer holds):
  // the held entries' exact top kk bound the row's kk-th, so keep that bound,
  // empty the buffer and offer the whole row again under it; repeat until
  // everything that passes fits. Each pass tightens the bound.
  while (__syncthreads_or(overflow)) {
    if (threadIdx.x == 0 && s_cnt > kStreamCap) s_cnt = kStreamCap;
    __syncthreads();
    compact();
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    const uint32_t thrK = s_thrK;
    const int thrI = s_thrI;
    const float zc = s_zc;
    overflow = false;
    for (int j = threadIdx.x; j < V; j += kST) offer(pen_z(__ldg(lg + j), j), j, thrK, thrI, zc);
  }
  __syncthreads();
  const int nheld = s_cnt;
  if (nheld <= kST) {
    // the held entries sorted at once: their first kk are the row's top kk, in order
    uint32_t x = threadIdx.x < nheld ? ckey[threadIdx.x] : 0xFFFFFFFFu;
    int xi = threadIdx.x < nheld ? cid[threadIdx.x] : sort_sentinel();
    block_sort(x, xi, reinterpret_cast<uint32_t*>(tie), tie + kST);
    if ((int)threadIdx.x < kk) {
      ckey[threadIdx.x] = x;
      cid[threadIdx.x] = xi;
    }
    if (threadIdx.x == 0) s_cnt = min(nheld, kk);
    __syncthreads();
  } else {
    compact();
    rank_sort(ckey, cid, s_cnt);
  }
  const int L = s_cnt;  // == kk: V > kk elements were all offered
  block_argmax(gv, gi, s_bv, s_bi);
  if (gi == 0x7FFFFFFF) gi = 0;  // nothing comparable (non-finite input): id 0

  TDesc dd;
  dd.argmax = gi;
  dd.k_key = 0xFFFFFFFFu;
  dd.k_cut = 0x7FFFFFFF;
  dd.p_key = 0xFFFFFFFFu;
  dd.p_cut = 0x7FFFFFFF;
  dd.m = 0.f;
  dd.S = 1.f;
  dd.kept = 1;
  if (smp) {
    // the largest transformed logit: z / T rounds monotonically in z
    const float mx = key_to_z(ckey[0]);
    // the cut rules of the cluster path's candidate list (top-k list sorted by
    // (key, id)): top-p on its fixed-point mass, then min-p, at least one kept
    if (threadIdx.x < 32) {
      auto fx = [&](int j) { return to_fix(expf(key_to_z(ckey[j]) - mx)); };
      unsigned long long SE = 0;
      warp_find_cross(L, ~0ull, fx, &SE);
      int Kf = L;
      if (p.top_p > 0.f && p.top_p < 1.f) {
        const unsigned long long target = (unsigned long long)ceil((double)p.top_p * (double)SE);
        const int j = warp_find_cross(L, target, fx, nullptr);
        if (j < L) Kf = min(Kf, j + 1);
      }
      if (p.min_p > 0.f) {
        int first = L;
        for (int j = threadIdx.x; j < L; j += 32)
          if (!(expf(key_to_z(ckey[j]) - mx) >= p.min_p)) { first = j; break; }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xFFFFFFFFu, first, o));
        if (first < Kf) Kf = first;
      }
      if (Kf < 1) Kf = 1;
      unsigned long long Sf = 0;
      warp_find_cross(Kf, ~0ull, fx, &Sf);
      if (threadIdx.x == 0) { sm->fin_kf = Kf; sm->fin_sf = Sf; }
    }
    __syncthreads();
    const int Kf = sm->fin_kf;
    dd.p_key = ckey[Kf - 1];
    dd.p_cut = cid[Kf - 1];
    dd.m = mx;
    dd.S = (float)((double)sm->fin_sf / kFix);
    dd.kept = Kf;
    int32_t* kid = a.kid + (size_t)task * kStreamTopK;
    uint32_t* kkey = a.kkey + (size_t)task * kStreamTopK;
    for (int t = threadIdx.x; t < Kf; t += kST) { kid[t] = cid[t]; kkey[t] = ckey[t]; }
  }
  if (threadIdx.x == 0) {
    a.wdesc[task] = dd;
    // the accept test of draft x_{i+1} against this target row
    int acc = 0;
    if (i < d) {
      const int x = dr[i];
      if (x >= 0 && x < V) {  // an out-of-range draft is rejected, never dereferenced
        if (p.greedy) {
          acc = x == dd.argmax;
        } else {
          const float pv = eval_p(dd, p, __ldg(lg + x), pen && bit(bits, x), x);
          // an argmax draft is a point mass: q(x) = 1
          const float qv = p.argmax_draft ? 1.f : __ldg(a.q + ((size_t)r * d + i) * V + x);
          acc = qv > 0.f && a.u[(size_t)r * (d + 1) + i] < pv / qv;
        }
      }
    }
    a.acc[task] = acc;
  }
}

// Per row: the accept chain from the tasks' flags, then the correction (after
// a rejection: norm(max(p - q, 0)) at the stopping position) or the bonus
// token (p_d), drawn over that position's kept list in id order.
__global__ void __launch_bounds__(kStreamTopK) k_verify_finish(const __grid_constant__ VerifyArgs a) {
  __shared__ int s_id[kStreamTopK];
  __shared__ unsigned long long s_w[kStreamTopK];
  __shared__ int s_nacc, s_pick;
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, d = a.depth;
  const RowParams p = a.p[r];
  const int32_t* dr = a.drafts + (size_t)r * d;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const bool ok = lane < d && a.acc[(size_t)r * (d + 1) + lane] != 0;
    const unsigned rej = ~__ballot_sync(0xFFFFFFFFu, ok) & (d >= 32 ? 0xFFFFFFFFu : ((1u << d) - 1u));
    if (lane == 0) s_nacc = rej ? __ffs(rej) - 1 : d;
  }
  __syncthreads();
  const int nacc = s_nacc;
  const int tn = r * (d + 1) + nacc;
  const TDesc dn = a.wdesc[tn];
  int y = dn.argmax;
  if (!p.greedy) {
    const int Kf = dn.kept;
    const int32_t* kid = a.kid + (size_t)tn * kStreamTopK;
    const uint32_t* kkey = a.kkey + (size_t)tn * kStreamTopK;
    const float* qn = nacc < d && !p.argmax_draft ? a.q + ((size_t)r * d + nacc) * a.V : nullptr;
    const int xr = nacc < d && p.argmax_draft ? dr[nacc] : -1;
    const float uu = a.u[(size_t)r * (d + 1) + d];
    // place entry t at its rank in id order with its weight
    auto draw = [&](bool residual) {
      for (int t = threadIdx.x; t < Kf; t += blockDim.x) {
        const int id = kid[t];
        int rank = 0;
        for (int q = 0; q < Kf; ++q) rank += kid[q] < id;
        const float pv = expf(key_to_z(kkey[t]) - dn.m) / dn.S;
        float w = pv;
        if (residual) w = pv - (id == xr ? 1.f : (qn ? __ldg(qn + id) : 0.f));
        s_id[rank] = id;
        s_w[rank] = to_fix(w > 0.f ? w : 0.f);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        unsigned long long tot = 0;
        warp_find_cross(Kf, ~0ull, [&](int j) { return s_w[j]; }, &tot);
        int pick = -1;
        if (tot > 0) {
          const unsigned long long target = (unsigned long long)floor((double)uu * (double)tot) + 1ull;
          const int j = warp_find_cross(Kf, target, [&](int j) { return s_w[j]; }, nullptr);
          pick = j < Kf ? s_id[j] : s_id[Kf - 1];
        }
        if (threadIdx.x == 0) s_pick = pick;
      }
      __syncthreads();
      return s_pick;
    };
    int yy = -1;
    if (nacc < d) yy = draw(true);
    if (yy < 0) yy = draw(false);
    if (yy >= 0) y = yy;
  }
  if (threadIdx.x == 0) {
    a.n_acc[r] = nacc;
    int32_t* o = a.out_tok + (size_t)r * (d + 1);
    for (int i = 0; i <= d; ++i) o[i] = i < nacc ? dr[i] : (i == nacc ? y : -1);
    if (a.h_rec) {
      // the record's tokens are visible to the host before its count
      int32_t* hr = a.h_rec + (size_t)r * (d + 2);
      for (int i = 0; i <= d; ++i) hr[1 + i] = o[i];
      st_release_sys(hr, nacc);
    }
    if (a.stats) {
      int32_t* st = a.stats + (size_t)r * (d + 2);
      st[0] += 1;
      if (nacc < d) st[1] += 1;
      for (int i = 1; i <= nacc; ++i) st[1 + i] += 1;
    }
  }
}

// ------------------------------------------------------------ top-k transform
// Low-latency exact transform of one (row, position) whose row cuts to a
// top-k of at most kStreamTopK (or is greedy), one 8-CTA cluster per task:
//  1. each CTA stages its vocabulary slice (repetition penalty, the argmax of
//     the penalised logits, z / T and its key), and every thread keeps the
//     smallest (key, id) it saw;
//  2. every CTA copies the cluster's 4096 thread minima and selects their
//     k-th smallest: k distinct elements lie at or below it, so the row's
//     top-k does too;
//  3. each CTA gathers its elements at or below that bound (typically a little
//     over k in all), the cluster exchanges them once, and every CTA selects
//     and sorts the exact top-k of the union;
//  4. the candidate path's cut rules on that sorted list (top-p on the
//     fixed-point mass of the top-k, min-p, at least one token) give the
//     descriptor, so every decision equals the cluster path's.
// If the bound admits more elements than the buffers hold (heavy ties), the
// exact k-th comes from the cluster radix selection and the gather is redone.
// Draft steps (mode 0) write q and draw; verify tasks (mode 1) write the
// descriptor, the accept test of the draft their row judges and the kept list
// that k_verify_finish draws from.
constexpr int kTkLocCap = 512;     // candidates one CTA may gather
constexpr int kTkMergeCap = 1024;  // candidates of the whole cluster
constexpr int kTkLocalK = 64;      // top-k up to this bound from each CTA's own thread minima

__host__ __device__ inline int tk_per(int V) { return (((V + kClusterCTAs - 1) / kClusterCTAs) + 3) & ~3; }

struct TkLayout {
  size_t zs, bits, tmk, tmi, allk, alli, tie, lk, li, mk, mi, sk, si, sw, sid, total;
  __host__ __device__ explicit TkLayout(int V) {
    const int per = tk_per(V);
    size_t o = (sizeof(SampleSmem) + 15) & ~size_t(15);
    zs = o;
    o += 4 * (size_t)per;
    bits = o;
    o += 4 * (size_t)((per + 31) / 32 + 1);
    o = (o + 15) & ~size_t(15);
    tmk = o; o += 4 * kST;
    tmi = o; o += 4 * kST;
    allk = o; o += 4 * kST * kClusterCTAs;
    alli = o; o += 4 * kST * kClusterCTAs;
    tie = o; o += 4 * kST * kClusterCTAs;
    lk = o; o += 4 * kTkLocCap;
    li = o; o += 4 * kTkLocCap;
    mk = o; o += 4 * kTkMergeCap;
    mi = o; o += 4 * kTkMergeCap;
    sk = o; o += 4 * kStreamTopK;
    si = o; o += 4 * kStreamTopK;
    o = (o + 7) & ~size_t(7);
    sw = o; o += 8 * kStreamTopK;
    sid = o; o += 4 * kStreamTopK;
    total = o;
  }
};

__global__ void __launch_bounds__(kST, 1) k_topk(const __grid_constant__ TopkArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  const TkLayout lay(a.V);
  float* zs = reinterpret_cast<float*>(dyn + lay.zs);
  uint32_t* bits = reinterpret_cast<uint32_t*>(dyn + lay.bits);
  uint32_t* tmk = reinterpret_cast<uint32_t*>(dyn + lay.tmk);
  int* tmi = reinterpret_cast<int*>(dyn + lay.tmi);
  uint32_t* allk = reinterpret_cast<uint32_t*>(dyn + lay.allk);
  int* alli = reinterpret_cast<int*>(dyn + lay.alli);
  int* tie = reinterpret_cast<int*>(dyn + lay.tie);
  uint32_t* lk = reinterpret_cast<uint32_t*>(dyn + lay.lk);
  int* li = reinterpret_cast<int*>(dyn + lay.li);
  uint32_t* mk = reinterpret_cast<uint32_t*>(dyn + lay.mk);
  int* mi = reinterpret_cast<int*>(dyn + lay.mi);
  uint32_t* sk = reinterpret_cast<uint32_t*>(dyn + lay.sk);
  int* si = reinterpret_cast<int*>(dyn + lay.si);
  unsigned long long* sw = reinterpret_cast<unsigned long long*>(dyn + lay.sw);
  int* sid = reinterpret_cast<int*>(dyn + lay.sid);
  __shared__ float s_bv[kST / 32];
  __shared__ int s_bi[kST / 32];
  Clu c(sm);
  const int task = blockIdx.x / kClusterCTAs;
  int r, i;
  const float* lg;
  if (a.mode == 0) {
    r = task;
    i = a.pos;
    lg = a.logits + (size_t)r * a.ld;
  } else {
    r = task / (a.depth + 1);
    i = task - r * (a.depth + 1);
    lg = a.logits + ((size_t)r * (a.depth + 1) + i) * a.V;
  }
  const RowParams p = a.p[r];
  const int per = tk_per(a.V);
  const int v0 = min(c.rank * per, a.V);
  const int n = min(per, a.V - v0);
  const int32_t* dr = a.drafts + (size_t)r * a.depth;
  // The penalty window (history, then this call's earlier drafts) and its
  // bitmap before the wait: the drafts of earlier positions come from kernels
  // that had finished before the previous one could start.
  load_window(sm, a.hist + (size_t)r * a.W, a.W, dr, i);
  const bool pen = p.rep_penalty != 1.f;
  if (pen) build_bitmap(sm, bits, v0, n);
  pdl_wait();
  pdl_trigger();
  const bool smp = !p.greedy;
  const float T = smp ? p.temperature : 1.f;

  // 1. stage the slice: penalty, argmax of the penalised logits, z / T, keys,
  //    and each thread's smallest (key, id). A thread keeps four independent
  //    chains, one per vector lane, merged at the end; ids ascend within a
  //    chain, so strict comparisons keep the lowest id on ties.
  float bz[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  int bzi[4] = {0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF};
  uint32_t tk[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
  int ti[4] = {0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF};
  float nf = 0.f;  // x * 0: NaN once a NaN or an infinity has been read
  {
    const float4* l4 = reinterpret_cast<const float4*>(lg + v0);
    const int n4 = n / 4;
    for (int b0 = 0; b0 < n4; b0 += 4 * kST) {
      float4 xb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j4 = b0 + u * kST + threadIdx.x;
        if (j4 < n4) xb[u] = __ldg(l4 + j4);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j4 = b0 + u * kST + threadIdx.x;
        if (j4 < n4) {
          const float xs[4] = {xb[u].x, xb[u].y, xb[u].z, xb[u].w};
          const uint32_t wb = pen ? bits[j4 >> 3] >> ((4 * j4) & 31) : 0u;
          float zt4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            nf = fmaf(xs[e], 0.f, nf);
            const float z = ((wb >> e) & 1u) ? penalize(xs[e], p.rep_penalty) : xs[e];
            if (z > bz[e]) { bz[e] = z; bzi[e] = v0 + j; }
            zt4[e] = z / T + 0.0f;
            const uint32_t key = desc_key(zt4[e]);
            if (key < tk[e]) { tk[e] = key; ti[e] = v0 + j; }
          }
          reinterpret_cast<float4*>(zs)[j4] = make_float4(zt4[0], zt4[1], zt4[2], zt4[3]);
        }
      }
    }
  }
  float bzv = bz[0];
  int bzid = bzi[0];
  uint32_t tkk = tk[0];
  int tid_ = ti[0];
#pragma unroll
  for (int e = 1; e < 4; ++e) {
    if (better(bz[e], bzi[e], bzv, bzid)) { bzv = bz[e]; bzid = bzi[e]; }
    if (tk[e] < tkk || (tk[e] == tkk && ti[e] < tid_)) { tkk = tk[e]; tid_ = ti[e]; }
  }
  if (tkk == 0xFFFFFFFFu && tid_ == 0x7FFFFFFF) tid_ = 0x7FFFFFFF - (c.rank * kST + (int)threadIdx.x);  // distinct placeholder
  if (__syncthreads_or(isnan(nf)) && threadIdx.x == 0) flag_status(a.status, MTP_ERR_NONFINITE);
  tmk[threadIdx.x] = tkk;
  tmi[threadIdx.x] = tid_;
  block_argmax(bzv, bzid, s_bv, s_bi);
  // small k: this CTA's k-th smallest thread minimum (k distinct elements of
  // the slice lie at or below it); the cluster's smallest such bound is
  // published with the argmax
  const int k = p.top_k;  // 2 <= k <= kStreamTopK < V for sampled rows (checked by the host)
  const bool local_bound = !p.greedy && k <= kTkLocalK;
  uint32_t Kc = 0xFFFFFFFFu;
  int Ic = 0x7FFFFFFF;
  if (local_bound) block_kth_pair(tkk, tid_, k, reinterpret_cast<uint32_t*>(tie), tie + kST, sm, Kc, Ic);
  if (threadIdx.x == 0) {
    sm->mail[c.ph].f[0] = bzv;
    sm->mail[c.ph].i[0] = bzid;
    sm->mail[c.ph].u[0] = ((unsigned long long)Kc << 32) | (uint32_t)Ic;
  }
  Mail* m = c.publish();
  float gv = -INFINITY;
  int gi = 0x7FFFFFFF;
#pragma unroll
  for (int q = 0; q < kClusterCTAs; ++q) {
    Mail* x = c.remote(m, q);
    if (better(x->f[0], x->i[0], gv, gi)) { gv = x->f[0]; gi = x->i[0]; }
  }
  const int argmax = gi < a.V ? gi : 0;  // nothing comparable (every logit NaN): id 0
  unsigned long long kb = ~0ull;
#pragma unroll
  for (int q = 0; q < kClusterCTAs; ++q) kb = min(kb, c.remote(m, q)->u[0]);

  if (!smp) {  // greedy: the point mass at the argmax
    if (c.rank == 0 && threadIdx.x == 0) {
      if (a.mode == 0) {
        a.draft_out[(size_t)r * a.depth + i] = argmax;
      } else {
        TDesc dd;
        dd.argmax = argmax;
        dd.k_key = 0xFFFFFFFFu;
        dd.k_cut = 0x7FFFFFFF;
        dd.p_key = 0xFFFFFFFFu;
        dd.p_cut = 0x7FFFFFFF;
        dd.m = 0.f;
        dd.S = 1.f;
        dd.kept = 1;
        a.wdesc[task] = dd;
        a.acc[task] = (i < a.depth && dr[i] == argmax) ? 1 : 0;
      }
    }
    c.cl.sync();  // every CTA has read this one's mail
    return;
  }

  // 2. the bound: for small k the smallest of the CTAs' own k-th thread
  //    minima; else the k-th smallest of the cluster's thread minima (either
  //    way k distinct elements lie at or below it, so the top-k does too)
  uint32_t K0 = (uint32_t)(kb >> 32);
  int I0 = (int)(uint32_t)kb;
  if (!local_bound) {
    for (int t = threadIdx.x; t < kST * kClusterCTAs; t += kST) {
      const int rr = t / kST, q = t - rr * kST;
      allk[t] = c.cl.map_shared_rank(tmk, rr)[q];
      alli[t] = c.cl.map_shared_rank(tmi, rr)[q];
    }
    __syncthreads();
    stream_select(sm, allk, alli, kST * kClusterCTAs, k, tie, K0, I0);
  }

  // 3. gather the elements at or below the bound, exchange them once
  auto gather = [&](uint32_t K, int cut) {
    if (threadIdx.x == 0) sm->ccount = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += kST) {
      const uint32_t key = desc_key(zs[j]);
      if (in_prefix(key, v0 + j, K, cut)) {
        const int pos = atomicAdd(&sm->ccount, 1);
        if (pos < kTkLocCap) {
          lk[pos] = key;
          li[pos] = v0 + j;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) sm->mail[c.ph].i[0] = sm->ccount;
    return c.publish();
  };
  int off[kClusterCTAs + 1];
  auto offsets = [&](Mail* mm) {
    bool over = false;
    off[0] = 0;
#pragma unroll
    for (int q = 0; q < kClusterCTAs; ++q) {
      const int cq = c.remote(mm, q)->i[0];
      over |= cq > kTkLocCap;
      off[q + 1] = off[q] + min(cq, kTkLocCap);
    }
    return over || off[kClusterCTAs] > kTkMergeCap;
  };
  if (offsets(gather(K0, I0))) {
    // too many at the bound: the exact k-th by cluster radix selection
    uint32_t Kx;
    unsigned long long rem;
    radix_select(c, zs, n, [](int) { return true; }, [](int) { return 1ull; }, (unsigned long long)k, Kx, rem);
    const int cut = tie_cut(c, zs, n, v0, [](int) { return true; }, Kx, rem);
    offsets(gather(Kx, cut));
  }
  const int M = min(off[kClusterCTAs], kTkMergeCap);
  for (int t = threadIdx.x; t < M; t += kST) {
    int q = 0;
    while (t >= off[q + 1]) ++q;
    mk[t] = c.cl.map_shared_rank(lk, q)[t - off[q]];
    mi[t] = c.cl.map_shared_rank(li, q)[t - off[q]];
  }
  __syncthreads();
  // the exact top-k of the union (it holds at least k), sorted by (key, id)
  int L;
  if (M <= kST) {
    // one entry per thread, sorted at once: the first k are the top-k in order
    uint32_t x = threadIdx.x < M ? mk[threadIdx.x] : 0xFFFFFFFFu;
    int xi = threadIdx.x < M ? mi[threadIdx.x] : sort_sentinel();
    block_sort(x, xi, reinterpret_cast<uint32_t*>(tie), tie + kST);
    if ((int)threadIdx.x < k) {
      sk[threadIdx.x] = x;
      si[threadIdx.x] = xi;
    }
    __syncthreads();
    L = min(M, k);
  } else {
    uint32_t Kk = 0xFFFFFFFFu;
    int Ik = 0x7FFFFFFF;
    stream_select(sm, mk, mi, M, k, tie, Kk, Ik);
    if (threadIdx.x == 0) sm->ccount = 0;
    __syncthreads();
    for (int t = threadIdx.x; t < M; t += kST)
      if (in_prefix(mk[t], mi[t], Kk, Ik)) {
        const int pos = atomicAdd(&sm->ccount, 1);
        if (pos < kStreamTopK) {
          sk[pos] = mk[t];
          si[pos] = mi[t];
        }
      }
    __syncthreads();
    L = min(sm->ccount, kStreamTopK);  // == k
    rank_sort(sk, si, L);
  }

  // 4. cut rules on the sorted top-k: top-p on its fixed-point mass, then
  //    min-p, at least one token kept
  const float mx = key_to_z(sk[0]);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    auto fx = [&](int j) { return to_fix(expf(key_to_z(sk[j]) - mx)); };
    unsigned long long SE = 0;
    warp_find_cross(L, ~0ull, fx, &SE);
    int Kf = L;
    if (p.top_p > 0.f && p.top_p < 1.f) {
      const unsigned long long target = (unsigned long long)ceil((double)p.top_p * (double)SE);
      const int j = warp_find_cross(L, target, fx, nullptr);
      if (j < L) Kf = min(Kf, j + 1);
    }
    if (p.min_p > 0.f) {
      int first = L;
      for (int j = lane; j < L; j += 32)
        if (!(expf(key_to_z(sk[j]) - mx) >= p.min_p)) { first = j; break; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xFFFFFFFFu, first, o));
      if (first < Kf) Kf = first;
    }
    if (Kf < 1) Kf = 1;
    unsigned long long Sf = 0;
    warp_find_cross(Kf, ~0ull, fx, &Sf);
    if (lane == 0) {
      sm->fin_kf = Kf;
      sm->fin_sf = Sf;
    }
  }
  __syncthreads();
  TDesc dd;
  dd.argmax = argmax;
  dd.k_key = 0xFFFFFFFFu;
  dd.k_cut = 0x7FFFFFFF;
  dd.kept = sm->fin_kf;
  dd.p_key = sk[dd.kept - 1];
  dd.p_cut = si[dd.kept - 1];
  dd.m = mx;
  dd.S = (float)((double)sm->fin_sf / kFix);
  const int Kf = dd.kept;

  if (a.mode == 1) {
    if (c.rank == 0) {
      int32_t* kid = a.kid + (size_t)task * kStreamTopK;
      uint32_t* kkey = a.kkey + (size_t)task * kStreamTopK;
      for (int t = threadIdx.x; t < Kf; t += kST) { kid[t] = si[t]; kkey[t] = sk[t]; }
      if (threadIdx.x == 0) {
        a.wdesc[task] = dd;
        // the accept test of draft x_{i+1} against this target row
        int acc = 0;
        if (i < a.depth) {
          const int x = dr[i];
          if (x >= 0 && x < a.V) {  // an out-of-range draft is rejected, never dereferenced
            bool px = false;
            for (int t = 0; t < sm->nwin; ++t) px |= sm->wtok[t] == x;
            const float pv = eval_p(dd, p, __ldg(lg + x), pen && px, x);
            // an argmax draft is a point mass: q(x) = 1
            const float qv = p.argmax_draft ? 1.f : __ldg(a.q + ((size_t)r * a.depth + i) * a.V + x);
            acc = qv > 0.f && a.u[(size_t)r * (a.depth + 1) + i] < pv / qv;
          }
        }
        a.acc[task] = acc;
      }
    }
  } else {
    // q is optional when no row is sampled (greedy rows with a penalty come here)
    float* qr = a.q ? a.q + ((size_t)r * a.depth + i) * a.V : nullptr;
    if (!qr) {
    } else if (a.q_zeroed) {
      // q is zero but for the kept prefix of the (key, id) order, renormalised:
      // the kept entries that fall in this CTA's slice, with the values the
      // full write below gives them
      for (int t = threadIdx.x; t < Kf; t += kST) {
        const int id = si[t];
        if (id >= v0 && id < v0 + n) {
          const float ev = expf(key_to_z(sk[t]) - mx);
          qr[id] = (!(p.min_p > 0.f) || ev >= p.min_p) ? ev / dd.S : 0.f;
        }
      }
    } else {
      // q over the slice: the kept prefix of the (key, id) order, renormalised
      float4* q4 = reinterpret_cast<float4*>(qr + v0);
      for (int j4 = threadIdx.x; j4 < n / 4; j4 += kST) {
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * j4 + e;
          o[e] = 0.f;
          if (in_prefix(desc_key(zs[j]), v0 + j, dd.p_key, dd.p_cut)) {
            const float ev = expf(zs[j] - mx);
            if (!(p.min_p > 0.f) || ev >= p.min_p) o[e] = ev / dd.S;
          }
        }
        q4[j4] = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
    if (c.rank == 0) {
      // the draw: the kept entries in id order, weights to_fix(q)
      for (int t = threadIdx.x; t < Kf; t += kST) {
        const int id = si[t];
        int rank = 0;
        for (int q = 0; q < Kf; ++q) rank += si[q] < id;
        sid[rank] = id;
        sw[rank] = to_fix(expf(key_to_z(sk[t]) - dd.m) / dd.S);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        unsigned long long tot = 0;
        warp_find_cross(Kf, ~0ull, [&](int j) { return sw[j]; }, &tot);
        int pick = -1;
        if (tot > 0) {
          const float u = a.u[(size_t)r * a.depth + i];
          const unsigned long long target = (unsigned long long)floor((double)u * (double)tot) + 1ull;
          const int j = warp_find_cross(Kf, target, [&](int j) { return sw[j]; }, nullptr);
          pick = j < Kf ? sid[j] : sid[Kf - 1];
        }
        if (threadIdx.x == 0) a.draft_out[(size_t)r * a.depth + i] = pick >= 0 ? pick : argmax;
      }
    }
  }
  c.cl.sync();  // keep shared memory alive until every remote read is done
}

bool topk_fits(const RowParams* p, int rows, int V, const float* logits, long long ld) {
  if (V % 4 != 0 || (reinterpret_cast<uintptr_t>(logits) & 15) != 0 || ld % 4 != 0 ||
      TkLayout(V).total > 226 * 1024)
    return false;
  for (int r = 0; r < rows; ++r)
    if (!p[r].greedy && !(p[r].top_k >= 1 && p[r].top_k <= kStreamTopK && p[r].top_k < V)) return false;
  return true;
}

void launch_topk(const TopkArgs& a, cudaStream_t s) {
  const int smem = (int)TkLayout(a.V).total;
  cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaLaunchConfig_t cfg = {};
  const int tasks = a.mode == 0 ? a.rows : a.rows * (a.depth + 1);
  cfg.gridDim = dim3(tasks * kClusterCTAs);
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCTAs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, k_topk, a);
  count_launch();
}

// ------------------------------------------------------------ flat transform
// Rows with a wide support (no top-k below V) spread every (row, position)
// over parts of its vocabulary, one CTA per part, through a chain of four
// short kernels (each waits for the previous one at griddepcontrol.wait):
//   k_fl_stats    every task, P parts: argmax of the penalised logits and
//                 their minimum; zeroes the task's histogram and counters
//   k_fl_hist     sampled tasks, Ps parts: fixed-point weights exp(z' - m)
//                 (z' = z / T + 0) added into kFlatBins equal value slices of
//                 [m - span, m] (the cluster path's binning), and the min-p
//                 mass
//   k_fl_gather   sampled tasks, Ps parts: the bin in which the running mass
//                 reaches ceil(top_p * SE), and its elements, into a per-task
//                 list; the task's last CTA then takes the exact crossing
//                 element of that list in (key, id) order (a weighted
//                 selection), the kept mass S and the descriptor (if the bin
//                 holds more than the list: an exact block-level radix
//                 selection over the row)
//   k_fl_sums     every row, P2 parts of 16 warp slices each: the accept
//                 chain (verify), each slice's sums of the draw weights (and,
//                 for a draft step, q); the row's last CTA finds the slice and
//                 then the element where the running weight reaches the
//                 draw's target, and writes the outputs. Greedy rows take the
//                 argmax chain from the first kernel's part maxima.
// The keys, weights, cut rules and draws are those of the cluster path.
__device__ __forceinline__ unsigned long long fl_amax_key(float v, int id) {
  uint32_t u = __float_as_uint(v + 0.0f);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ float fl_key_value(unsigned long long k) {
  uint32_t u = (uint32_t)(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

struct FlTask {
  int r, i;
  const float* lg;
};
__device__ __forceinline__ FlTask fl_task(const FlatArgs& a, int t) {
  FlTask x;
  if (a.mode == 0) {
    x.r = t;
    x.i = a.pos;
    x.lg = a.logits + (size_t)t * a.ld;
  } else {
    x.r = t / (a.depth + 1);
    x.i = t - x.r * (a.depth + 1);
    x.lg = a.logits + (size_t)t * a.V;
  }
  return x;
}
__host__ __device__ __forceinline__ int fl_per(int V, int P) { return ((V + P - 1) / P + 3) & ~3; }

// The j-th sampled task (grid row of the histogram and gather kernels).
__device__ __forceinline__ int fl_sampled_task(const FlatArgs& a, int j) {
  if (a.mode == 0) return a.srow[j];
  const int tpr = a.depth + 1, s = j / tpr;
  return a.srow[s] * tpr + (j - s * tpr);
}

// The task's transform scale: maximum transformed logit m, the argmax of the
// penalised logits, and the bin scale of [m - span, m].
struct FlScale {
  float mx, scale;
  int amax;
};
// Every warp: the task's P (<= 64) part slots, two per lane (loads only).
struct FlSlots {
  unsigned long long best;
  float zm;
};
__device__ __forceinline__ FlSlots fl_slots(const FlatArgs& a, int t) {
  const int lane = threadIdx.x & 31;
  const unsigned long long* am = a.amax + (size_t)t * a.P;
  const float* zn = a.zmin + (size_t)t * a.P;
  FlSlots s;
  s.best = lane < a.P ? __ldcg(am + lane) : 0ull;
  s.zm = lane < a.P ? __ldcg(zn + lane) : INFINITY;
  if (lane + 32 < a.P) {
    s.best = max(s.best, __ldcg(am + lane + 32));
    s.zm = fminf(s.zm, __ldcg(zn + lane + 32));
  }
  return s;
}
__device__ FlScale fl_scale_of(FlSlots sl, const RowParams& rp) {
  unsigned long long best = sl.best;
  float zm = sl.zm;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
    zm = fminf(zm, __shfl_xor_sync(0xFFFFFFFFu, zm, o));
  }
  FlScale s;
  s.amax = best ? (int)(0xFFFFFFFFu - (uint32_t)best) : 0;
  const float zmax = best ? fl_key_value(best) : -INFINITY;
  const float T = rp.greedy ? 1.f : rp.temperature;
  s.mx = zmax / T + 0.0f;
  const float zlo = zm / T + 0.0f;
  float span = s.mx - zlo;
  if (!(span > 0.f)) span = 0.f;
  if (span > kFlatSpan) span = kFlatSpan;
  s.scale = span > 0.f ? ((float)kFlatBins - 0.01f) / span : 0.f;
  return s;
}
__device__ __forceinline__ FlScale fl_scale(const FlatArgs& a, int t, const RowParams& rp) {
  return fl_scale_of(fl_slots(a, t), rp);
}
__device__ __forceinline__ int fl_bin(const FlScale& s, float z) {
  const float t = (s.mx - z) * s.scale;
  return t < (float)kFlatBins ? (int)t : kFlatBins;  // beyond the span (and NaN): no bin
}

// Sub-bins of bin b: its order keys (from a little above its top value to a
// little below its bottom one) cut into kFlatBins equal ranges of 2^sh keys.
// sub_of is monotone in the key (clamped at both ends), so the sub-bins keep
// the (key asc) order whatever the rounding of the bin edges.
struct FlSub {
  uint32_t k0;
  int sh;
};
__device__ __forceinline__ FlSub fl_sub(const FlScale& s, int b) {
  const float zt = s.mx - (float)b / s.scale, zb = s.mx - (float)(b + 1) / s.scale;
  const float top = zt + fabsf(zt) * 1e-6f + 1e-30f, bot = zb - fabsf(zb) * 1e-6f - 1e-30f;
  FlSub u;
  u.k0 = desc_key(top);
  const uint32_t k1 = desc_key(bot);
  const uint32_t span = k1 > u.k0 ? k1 - u.k0 : 1u;
  const int nb = 32 - __clz(span);
  u.sh = nb > 11 ? nb - 11 : 0;
  return u;
}
__device__ __forceinline__ int fl_sub_of(const FlSub& u, uint32_t key) {
  if (key <= u.k0) return 0;
  const uint32_t q = (key - u.k0) >> u.sh;
  return q < (uint32_t)kFlatBins ? (int)q : kFlatBins - 1;
}

// The crossing of a task's histogram: total mass SE, the bin b in which the
// running mass reaches target = ceil(top_p SE) (b = -1 when SE is 0) and the
// mass still needed there.
struct FlCross {
  unsigned long long SE, need, target;
  int b;
};
constexpr int kFlPer = kFlatBins / kST;  // histogram bins per thread
__device__ __forceinline__ void fl_bins_load(const unsigned long long* h, unsigned long long (&v)[kFlPer]) {
#pragma unroll
  for (int b = 0; b < kFlPer; ++b) v[b] = __ldcg(&h[threadIdx.x * kFlPer + b]);
}
// Every thread of the block, from its kFlPer bins: the crossing, into *out
// (shared memory). One block scan.
__device__ void fl_cross(SampleSmem* sm, const unsigned long long (&v)[kFlPer], float top_p, FlCross* out) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long s = 0;
#pragma unroll
  for (int b = 0; b < kFlPer; ++b) s += v[b];
  unsigned long long incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) sm->wsum[w] = incl;
  if (threadIdx.x == 0) out->b = -1;
  __syncthreads();
  unsigned long long before = 0, SE = 0;
  for (int q = 0; q < kST / 32; ++q) {
    if (q < w) before += sm->wsum[q];
    SE += sm->wsum[q];
  }
  const unsigned long long target = (unsigned long long)ceil((double)top_p * (double)SE);
  unsigned long long cum = before + incl - s;
  if (SE > 0 && cum < target && target <= cum + s) {
#pragma unroll
    for (int b = 0; b < kFlPer; ++b) {
      if (cum < target && target <= cum + v[b]) {
        out->b = threadIdx.x * kFlPer + b;
        out->need = target - cum;
        break;
      }
      cum += v[b];
    }
  }
  if (threadIdx.x == 0) {
    out->SE = SE;
    out->target = target;
  }
  __syncthreads();
}

// A rolled pass over one thread's 16-byte items j4 = t0 + u * stride, u < nu
// (nu the same for every thread that takes part, so the body may hold warp
// collectives), with the next two items' loads in flight. The body is one
// copy of the per-item code, which stays in the instruction cache across
// iterations; the kernels here run it a few times per launch, where an
// unrolled copy per item would be fetched cold each time. first: item u = 0.
template <class F>
__device__ __forceinline__ void fl_rolled(const float4* p, int t0, int stride, int n4, int nu, float4 first,
                                          F&& body) {
  float4 a = first, b = make_float4(0.f, 0.f, 0.f, 0.f);
  if (t0 + stride < n4) b = __ldg(p + t0 + stride);
#pragma unroll 1
  for (int u = 0; u < nu; ++u) {
    const int j4 = t0 + u * stride;
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j4 + 2 * stride < n4) c = __ldg(p + j4 + 2 * stride);
    body(a, j4, j4 < n4);
    a = b;
    b = c;
  }
}
__device__ __forceinline__ float4 fl_first(const float4* p, int j4, int n4) {
  return j4 < n4 ? __ldg(p + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ size_t fl_bits_off() { return (sizeof(SampleSmem) + 15) & ~size_t(15); }

__global__ void __launch_bounds__(kST) k_fl_stats(const __grid_constant__ FlatArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  uint32_t* bits = reinterpret_cast<uint32_t*>(dyn + fl_bits_off());
  __shared__ float s_bv[kST / 32];
  __shared__ int s_bi[kST / 32];
  __shared__ float s_mn[kST / 32];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y, p = blockIdx.x;
  const FlTask k = fl_task(a, t);
  const RowParams rp = a.p[k.r];
  // this task's share of the scratch the next kernels accumulate into
  for (int b = p * kST + threadIdx.x; b < kFlatBins; b += a.P * kST) {
    a.hist_w[(size_t)t * kFlatBins + b] = 0ull;
    a.sub_w[(size_t)t * kFlatBins + b] = 0ull;
  }
  if (p == 0 && threadIdx.x == 0) {
    a.sminp[t] = 0ull;
    a.ccnt[t] = 0;
    a.gcnt[t] = 0;
    if (k.i == 0 || a.mode == 0) a.scnt[k.r] = 0;
  }
  const int per = fl_per(a.V, a.P);
  const int v0 = min(p * per, a.V), n = min(per, a.V - v0);
  load_window(sm, a.hist + (size_t)k.r * a.W, a.W, a.drafts + (size_t)k.r * a.depth, k.i);
  const bool pen = rp.rep_penalty != 1.f;
  if (pen) build_bitmap(sm, bits, v0, n);
  // four independent chains per thread (one per vector lane): ids ascend
  // within a chain, so strict > keeps the lowest id on ties
  float bz[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  int bzi[4] = {0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF};
  float mn = INFINITY, nf = 0.f;
  const float4* l4 = reinterpret_cast<const float4*>(k.lg + v0);
  const int n4 = n / 4;
  fl_rolled(l4, threadIdx.x, kST, n4, (n4 - (int)threadIdx.x + kST - 1) / kST, fl_first(l4, threadIdx.x, n4),
            [&](const float4& x, int j4, bool valid) {
              const float xs[4] = {x.x, x.y, x.z, x.w};
              const uint32_t wb = pen ? bits[j4 >> 3] >> ((4 * j4) & 31) : 0u;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                nf = fmaf(xs[e], 0.f, nf);
                const float z = ((wb >> e) & 1u) ? penalize(xs[e], rp.rep_penalty) : xs[e];
                if (z > bz[e]) { bz[e] = z; bzi[e] = v0 + 4 * j4 + e; }
                mn = fminf(mn, z);
              }
            });
  float bv = bz[0];
  int bi = bzi[0];
#pragma unroll
  for (int e = 1; e < 4; ++e)
    if (better(bz[e], bzi[e], bv, bi)) { bv = bz[e]; bi = bzi[e]; }
  if (__syncthreads_or(isnan(nf)) && threadIdx.x == 0) flag_status(a.status, MTP_ERR_NONFINITE);
  block_argmax(bv, bi, s_bv, s_bi);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
  if ((threadIdx.x & 31) == 0) s_mn[threadIdx.x >> 5] = mn;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m2 = INFINITY;
    for (int w = 0; w < kST / 32; ++w) m2 = fminf(m2, s_mn[w]);
    a.amax[(size_t)t * a.P + p] = (bi >= 0 && bi < a.V) ? fl_amax_key(bv, bi) : 0ull;
    a.zmin[(size_t)t * a.P + p] = m2;
  }
}

// Adds w to a 64-bit bin held as two 32-bit words, with native 32-bit shared
// atomics: the low word wraps modulo 2^32 and the thread whose add wrapped it
// carries one into the high word, so hi * 2^32 + lo stays the exact sum.
__device__ __forceinline__ void fl_bin_add(uint32_t* lo, uint32_t* hi, int b, unsigned long long w) {
  const uint32_t wl = (uint32_t)w, wh = (uint32_t)(w >> 32);
  const uint32_t old = atomicAdd(&lo[b], wl);
  const uint32_t c = old + wl < old ? 1u : 0u;
  if (wh + c) atomicAdd(&hi[b], wh + c);
}
// The gather's sub-bin histogram: after the resolve's layout (SampleSmem, the
// candidate list, its tie buffer and a bitmap of the whole row) and after the
// part's bitmap.
__host__ __device__ __forceinline__ size_t fl_sub_off(int V, int per) {
  const size_t base = (sizeof(SampleSmem) + 15) & ~size_t(15);
  const size_t res = base + 12 * (size_t)kFlatCandCap + 4 * (size_t)((V + 31) / 32 + 1);
  const size_t part = base + 4 * (size_t)((per + 31) / 32 + 1);
  return ((res > part ? res : part) + 15) & ~size_t(15);
}
__host__ __device__ __forceinline__ size_t fl_hist_off(int per) {
  return (((sizeof(SampleSmem) + 15) & ~size_t(15)) + 4 * (size_t)((per + 31) / 32 + 1) + 15) & ~size_t(15);
}

// The target logits are inputs of the whole chain (the kernel before the
// first one of the chain has finished once any later one starts), so the
// histogram, gather and sums kernels load their first batch of them before
// waiting for the kernel before them.
__global__ void __launch_bounds__(kST) k_fl_hist(const __grid_constant__ FlatArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  const int per = fl_per(a.V, a.Ps);
  uint32_t* bits = reinterpret_cast<uint32_t*>(dyn + fl_bits_off());
  uint32_t* lo = reinterpret_cast<uint32_t*>(dyn + fl_hist_off(per));
  uint32_t* hi = lo + kFlatBins;
  const int t = fl_sampled_task(a, blockIdx.y), p = blockIdx.x;
  const FlTask k = fl_task(a, t);
  const RowParams rp = a.p[k.r];
  const int v0 = min(p * per, a.V), n = min(per, a.V - v0);
  const float4* l4 = reinterpret_cast<const float4*>(k.lg + v0);
  const int n4 = n / 4;
  const float4 x0 = fl_first(l4, threadIdx.x, n4);
  for (int b = threadIdx.x; b < 2 * kFlatBins; b += kST) lo[b] = 0u;
  load_window(sm, a.hist + (size_t)k.r * a.W, a.W, a.drafts + (size_t)k.r * a.depth, k.i);
  const bool pen = rp.rep_penalty != 1.f;
  if (pen) build_bitmap(sm, bits, v0, n);
  pdl_wait();
  pdl_trigger();
  const FlScale sc = fl_scale(a, t, rp);
  const bool minp = rp.min_p > 0.f;
  unsigned long long smp = 0ull;
  fl_rolled(l4, threadIdx.x, kST, n4, (n4 - (int)threadIdx.x + kST - 1) / kST, x0,
            [&](const float4& x, int j4, bool valid) {
              const float xs[4] = {x.x, x.y, x.z, x.w};
              const uint32_t wb = pen ? bits[j4 >> 3] >> ((4 * j4) & 31) : 0u;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float z = (((wb >> e) & 1u) ? penalize(xs[e], rp.rep_penalty) : xs[e]) / rp.temperature + 0.0f;
                const int b = fl_bin(sc, z);
                if (b < kFlatBins) {
                  const float ev = expf(z - sc.mx);
                  const unsigned long long w = to_fix(ev);
                  if (w) {
                    fl_bin_add(lo, hi, b, w);
                    if (minp && ev >= rp.min_p) smp += w;
                  }
                }
              }
            });
  __syncthreads();
  for (int b = threadIdx.x; b < kFlatBins; b += kST) {
    const unsigned long long v = ((unsigned long long)hi[b] << 32) + lo[b];
    if (v) atomicAdd(&a.hist_w[(size_t)t * kFlatBins + b], v);
  }
  if (minp) {
    const unsigned long long tot = block_sum_u64(smp, sm->wsum);
    if (threadIdx.x == 0 && tot) atomicAdd(&a.sminp[t], tot);
  }
}

__device__ void fl_resolve_task(const FlatArgs& a, int t, unsigned char* dyn, const FlScale* sc_in,
                                const FlCross* cr_in);

__global__ void __launch_bounds__(kST) k_fl_gather(const __grid_constant__ FlatArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  uint32_t* bits = reinterpret_cast<uint32_t*>(dyn + fl_bits_off());
  __shared__ FlCross s_cr;
  __shared__ int s_last;
  const int t = fl_sampled_task(a, blockIdx.y), p = blockIdx.x;
  const FlTask k = fl_task(a, t);
  const RowParams rp = a.p[k.r];
  if (!(rp.top_p > 0.f && rp.top_p < 1.f)) {
    // nothing to gather: one CTA writes the descriptor
    pdl_wait();
    pdl_trigger();
    if (p == 0) fl_resolve_task(a, t, dyn, nullptr, nullptr);
    return;
  }
  const int per = fl_per(a.V, a.Ps);
  const int v0 = min(p * per, a.V), n = min(per, a.V - v0);
  const float4* l4 = reinterpret_cast<const float4*>(k.lg + v0);
  const int n4 = n / 4;
  const float4 x0 = fl_first(l4, threadIdx.x, n4);
  load_window(sm, a.hist + (size_t)k.r * a.W, a.W, a.drafts + (size_t)k.r * a.depth, k.i);
  const bool pen = rp.rep_penalty != 1.f;
  if (pen) build_bitmap(sm, bits, v0, n);
  pdl_wait();
  pdl_trigger();
  // one round trip: the histogram bins and the part slots
  unsigned long long hv[kFlPer];
  fl_bins_load(a.hist_w + (size_t)t * kFlatBins, hv);
  const FlScale sc = fl_scale(a, t, rp);
  fl_cross(sm, hv, rp.top_p, &s_cr);
  const int bstar = s_cr.b;
  if (bstar >= 0) {
    const int lane = threadIdx.x & 31;
    uint32_t* ckey = a.ckey + (size_t)t * kFlatCandCap;
    int32_t* cid = a.cid + (size_t)t * kFlatCandCap;
    // the crossing bin's mass per sub-bin (its elements are few: a sparse
    // shared histogram, flushed where non-zero)
    const FlSub su = fl_sub(sc, bstar);
    uint32_t* slo = reinterpret_cast<uint32_t*>(dyn + fl_sub_off(a.V, per));
    uint32_t* shi = slo + kFlatBins;
    for (int b = threadIdx.x; b < 2 * kFlatBins; b += kST) slo[b] = 0u;
    __syncthreads();
    // every thread runs the block's largest item count (warp-uniform appends)
    fl_rolled(l4, threadIdx.x, kST, n4, (n4 + kST - 1) / kST, x0, [&](const float4& x, int j4, bool valid) {
      float zz[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t mm = 0u;  // elements of this vector in the crossing bin
      if (valid) {
        const float xs[4] = {x.x, x.y, x.z, x.w};
        const uint32_t wb = pen ? bits[j4 >> 3] >> ((4 * j4) & 31) : 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          zz[e] = (((wb >> e) & 1u) ? penalize(xs[e], rp.rep_penalty) : xs[e]) / rp.temperature + 0.0f;
          if (fl_bin(sc, zz[e]) == bstar) mm |= 1u << e;
        }
      }
      if (__any_sync(0xFFFFFFFFu, mm != 0u)) {
        // one list append per warp: exclusive scan of the lanes' counts
        const int c = __popc(mm);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += t2;
        }
        int base = 0;
        if (lane == 31) base = atomicAdd(&a.ccnt[t], incl);
        int pos = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - c;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((mm >> e) & 1u) {
            const uint32_t key = desc_key(zz[e]);
            if (pos < kFlatCandCap) {
              ckey[pos] = key;
              cid[pos] = v0 + 4 * j4 + e;
            }
            ++pos;
            const unsigned long long w = to_fix(expf(zz[e] - sc.mx));
            if (w) fl_bin_add(slo, shi, fl_sub_of(su, key), w);
          }
      }
    });
    __syncthreads();
    for (int b = threadIdx.x; b < kFlatBins; b += kST) {
      const unsigned long long v = ((unsigned long long)shi[b] << 32) + slo[b];
      if (v) atomicAdd(&a.sub_w[(size_t)t * kFlatBins + b], v);
    }
  }
  // the last of the task's CTAs to finish resolves its descriptor
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&a.gcnt[t], 1) == a.Ps - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  fl_resolve_task(a, t, dyn, &sc, &s_cr);
}

// Exact crossing inside bin bstar of one row by one CTA, when the gathered
// list overflowed (heavily tied logits): radix selection over the keys of the
// bin's elements with their fixed-point weights (digit passes over the row),
// then the right tie in id order. Returns the (key, id) bound, and in *in_bin
// the weight of the bin's elements up to and including it.
template <class Z>
__device__ void fl_exact_cut(SampleSmem* sm, int V, Z zof, const FlScale& sc, int bstar, unsigned long long need,
                             uint32_t& Kout, int& cutout, unsigned long long* in_bin) {
  auto wk = [&](uint32_t key) { return to_fix(expf(key_to_z(key) - sc.mx)); };
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int j = threadIdx.x; j < V; j += kST) {
    const float z = zof(j);
    if (fl_bin(sc, z) == bstar) {
      const uint32_t key = desc_key(z);
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xFFFFFFFFu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xFFFFFFFFu, kmax, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm->wsum[threadIdx.x >> 5] = ((unsigned long long)kmin << 32) | kmax;
  __syncthreads();
  kmin = 0xFFFFFFFFu;
  kmax = 0u;
  for (int w = 0; w < kST / 32; ++w) {
    kmin = min(kmin, (uint32_t)(sm->wsum[w] >> 32));
    kmax = max(kmax, (uint32_t)sm->wsum[w]);
  }
  const uint32_t diff = kmin ^ kmax;
  int hi = diff ? 31 - __clz(diff) : -1;
  uint32_t mask = hi >= 0 ? ~((hi == 31) ? 0xFFFFFFFFu : ((2u << hi) - 1u)) : 0xFFFFFFFFu;
  uint32_t prefix = kmin & mask;
  unsigned long long target = need;
  unsigned long long* h = sm->hist[0];
  while (hi >= 0) {
    const int lo = hi >= 7 ? hi - 7 : 0;
    const uint32_t dmask = (1u << (hi - lo + 1)) - 1u;
    __syncthreads();
    for (int b = threadIdx.x; b < 256; b += kST) h[b] = 0ull;
    __syncthreads();
    for (int j = threadIdx.x; j < V; j += kST) {
      const float z = zof(j);
      if (fl_bin(sc, z) != bstar) continue;
      const uint32_t key = desc_key(z);
      if ((key & mask) == prefix) atomicAdd(&h[(key >> lo) & dmask], wk(key));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      unsigned long long s8 = 0;
      for (int b = 0; b < 8; ++b) s8 += h[lane * 8 + b];
      unsigned long long incl = s8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      unsigned long long cum = incl - s8;
      const bool mine = cum < target && target <= incl;
      if (mine) {
        for (int b = 0; b < 8; ++b) {
          const unsigned long long t = h[lane * 8 + b];
          if (cum < target && target <= cum + t) {
            sm->sel_bin = lane * 8 + b;
            sm->sel_rem = target - cum;
            break;
          }
          cum += t;
        }
      }
      if (!__ballot_sync(0xFFFFFFFFu, mine) && lane == 0) {  // target above the total: the last digit
        sm->sel_bin = (int)dmask;
        sm->sel_rem = target;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sm->sel_bin << lo;
    mask |= dmask << lo;
    target = sm->sel_rem;
    hi = lo - 1;
  }
  const uint32_t K = prefix;
  const unsigned long long ew = wk(K);
  const unsigned long long want = ew > 0 ? (target + ew - 1) / ew : 1ull;  // the want-th tie in id order
  // ties at K in id order: per-thread contiguous ranges, block exclusive scan of their counts
  const int chunk = (V + kST - 1) / kST;
  const int a0 = min((int)threadIdx.x * chunk, V), a1 = min(a0 + chunk, V);
  unsigned long long c = 0;
  for (int j = a0; j < a1; ++j) {
    const float z = zof(j);
    if (fl_bin(sc, z) == bstar && desc_key(z) == K) ++c;
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (threadIdx.x == 0) sm->found = 0x7FFFFFFF;
  __syncthreads();
  if (lane == 31) sm->wsum[w] = incl;
  __syncthreads();
  unsigned long long before = 0;
  for (int q = 0; q < w; ++q) before += sm->wsum[q];
  unsigned long long cum = before + incl - c;
  if (cum < want && want <= cum + c) {
    for (int j = a0; j < a1; ++j) {
      const float z = zof(j);
      if (fl_bin(sc, z) == bstar && desc_key(z) == K && ++cum == want) {
        sm->found = j;
        break;
      }
    }
  }
  __syncthreads();
  const int cut = sm->found;  // 0x7FFFFFFF: every tie (the target lies past them)
  // the bin's weight up to and including the bound
  unsigned long long loc = 0;
  for (int j = threadIdx.x; j < V; j += kST) {
    const float z = zof(j);
    if (fl_bin(sc, z) == bstar) {
      const uint32_t key = desc_key(z);
      if (in_prefix(key, j, K, cut)) loc += wk(key);
    }
  }
  *in_bin = block_sum_u64(loc, sm->wsum);
  Kout = K;
  cutout = cut;
}

// Every thread of the block (warp 0 holds the entries): of n <= 32 entries
// with distinct ids, one per lane of warp 0 (have), the one where the running
// weight in (key asc, id asc) order first reaches need. Returns false when no
// entry is found; else *K, *cut and *in_w (the weight of the entries up to
// and including it).
template <class Wk>
__device__ bool fl_warp_cross(bool have, uint32_t kk, int ii, int n, unsigned long long need, Wk wk, uint32_t* K,
                              int* cut, unsigned long long* in_w, int* s_ok, uint32_t* s_K, int* s_cut,
                              unsigned long long* s_in) {
  if (threadIdx.x == 0) *s_ok = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    if (!have) {
      kk = 0xFFFFFFFFu;
      ii = 0x7FFFFFFF;
    }
    const unsigned long long ww = have ? wk(kk) : 0ull;
    unsigned long long before = 0;
    for (int j = 0; j < n; ++j) {
      const uint32_t kj = __shfl_sync(0xFFFFFFFFu, kk, j);
      const int ij = __shfl_sync(0xFFFFFFFFu, ii, j);
      const unsigned long long wj = __shfl_sync(0xFFFFFFFFu, ww, j);
      if (kj < kk || (kj == kk && ij < ii)) before += wj;
    }
    if (have && ww > 0 && before < need && need <= before + ww) {  // exactly one entry
      *s_K = kk;
      *s_cut = ii;
      *s_in = before + ww;
      *s_ok = 1;
    }
  }
  __syncthreads();
  const bool ok = *s_ok != 0;
  if (ok) {
    *K = *s_K;
    *cut = *s_cut;
    *in_w = *s_in;
  }
  __syncthreads();
  return ok;
}

// Every thread of the block, from its kFlPer bins of a histogram: the bin b
// where the running mass reaches need (out->b = -1 when it does not) and the
// mass still needed there, into *out (shared memory). One block scan.
__device__ __forceinline__ void fl_reach(SampleSmem* sm, const unsigned long long (&v)[kFlPer],
                                         unsigned long long need, FlCross* out) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long s = 0;
#pragma unroll
  for (int b = 0; b < kFlPer; ++b) s += v[b];
  unsigned long long incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) sm->wsum[w] = incl;
  if (threadIdx.x == 0) out->b = -1;
  __syncthreads();
  unsigned long long cum = incl - s;
  for (int q = 0; q < w; ++q) cum += sm->wsum[q];
  if (cum < need && need <= cum + s) {
#pragma unroll
    for (int b = 0; b < kFlPer; ++b) {
      if (cum < need && need <= cum + v[b]) {
        out->b = threadIdx.x * kFlPer + b;
        out->need = need - cum;
        break;
      }
      cum += v[b];
    }
  }
  __syncthreads();
}

// One CTA: of up to 2 kST (key, id) entries with distinct ids (cnt of them
// in key[], id[] of global memory), the entry where the running weight in
// (key asc, id asc) order first reaches need, weight(key) being each entry's
// fixed-point weight. A bitonic sort over the block (two entries per thread;
// shuffles below a warp's span, shared memory above), then a block scan of
// the weights. Returns false when no entry is found; else *K, *cut (the
// entry) and *in_w (the weight of the entries up to and including it).
template <class Wk>
__device__ bool fl_sorted_cross(const uint32_t* gkey, const int32_t* gid, int cnt, unsigned long long need, Wk wk,
                                uint32_t* sk, int* si, unsigned long long* wsum, uint32_t* K, int* cut,
                                unsigned long long* in_w, int* s_ok, uint32_t* s_K, int* s_cut,
                                unsigned long long* s_in) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  uint32_t k[2];
  int id[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int i = 2 * t + e;
    const bool real = i < cnt;
    k[e] = real ? __ldcg(gkey + i) : 0xFFFFFFFFu;
    id[e] = real ? __ldcg(gid + i) : 0x7FFFFFFF - (2 * kST - 1) + i;  // distinct, above every vocabulary id
  }
#pragma unroll
  for (int size = 2; size <= 2 * kST; size <<= 1) {
    const bool asc = ((2 * t) & size) == 0;
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride == 1) {
        if (pair_gt(k[0], id[0], k[1], id[1]) == asc) {
          const uint32_t tk = k[0]; k[0] = k[1]; k[1] = tk;
          const int ti = id[0]; id[0] = id[1]; id[1] = ti;
        }
        continue;
      }
      uint32_t ok[2];
      int oi[2];
      if (stride < 64) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          ok[e] = __shfl_xor_sync(0xFFFFFFFFu, k[e], stride >> 1);
          oi[e] = __shfl_xor_sync(0xFFFFFFFFu, id[e], stride >> 1);
        }
      } else {
        __syncthreads();
        sk[2 * t] = k[0]; sk[2 * t + 1] = k[1];
        si[2 * t] = id[0]; si[2 * t + 1] = id[1];
        __syncthreads();
        const int pt = t ^ (stride >> 1);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          ok[e] = sk[2 * pt + e];
          oi[e] = si[2 * pt + e];
        }
      }
      const bool low = ((2 * t) & stride) == 0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool other_less = pair_gt(k[e], id[e], ok[e], oi[e]);
        if (low == asc ? other_less : !other_less) {
          k[e] = ok[e];
          id[e] = oi[e];
        }
      }
    }
  }
  // entries 2t, 2t+1 in order: their weights and the block's running weight
  unsigned long long wt[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) wt[e] = 2 * t + e < cnt ? wk(k[e]) : 0ull;
  const unsigned long long mine = wt[0] + wt[1];
  unsigned long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  __syncthreads();
  if (lane == 31) wsum[w] = incl;
  if (t == 0) *s_ok = 0;
  __syncthreads();
  unsigned long long before = incl - mine;
  for (int q = 0; q < w; ++q) before += wsum[q];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    if (wt[e] > 0 && before < need && need <= before + wt[e]) {  // exactly one entry
      *s_K = k[e];
      *s_cut = id[e];
      *s_in = before + wt[e];
      *s_ok = 1;
    }
    before += wt[e];
  }
  __syncthreads();
  const bool ok = *s_ok != 0;
  if (ok) {
    *K = *s_K;
    *cut = *s_cut;
    *in_w = *s_in;
  }
  __syncthreads();
  return ok;
}

// One CTA: the descriptor of a sampled task t (shared memory laid out as
// SampleSmem, then the candidate list, its tie buffer and a bitmap of the
// whole row). sc_in and cr_in: the scale and crossing the calling CTA already
// holds (null: computed here).
__device__ void fl_resolve_task(const FlatArgs& a, int t, unsigned char* dyn, const FlScale* sc_in,
                                const FlCross* cr_in) {
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  uint32_t* mk = reinterpret_cast<uint32_t*>(dyn + fl_bits_off());
  int* mi = reinterpret_cast<int*>(mk + kFlatCandCap);
  int* tie = mi + kFlatCandCap;
  uint32_t* bits = reinterpret_cast<uint32_t*>(tie + kFlatCandCap);
  __shared__ FlCross s_cr;
  __shared__ uint32_t s_K;
  __shared__ int s_cut, s_ok;
  __shared__ unsigned long long s_in;
  const FlTask k = fl_task(a, t);
  const RowParams rp = a.p[k.r];
  const bool topp = rp.top_p > 0.f && rp.top_p < 1.f;
  FlScale sc;
  const FlCross* cr = cr_in;
  if (sc_in) {
    sc = *sc_in;
  } else {
    unsigned long long hv[kFlPer];
    fl_bins_load(a.hist_w + (size_t)t * kFlatBins, hv);
    sc = fl_scale(a, t, rp);
    fl_cross(sm, hv, topp ? rp.top_p : 1.f, &s_cr);
    cr = &s_cr;
  }
  TDesc d;
  d.argmax = sc.amax;
  d.k_key = 0xFFFFFFFFu;
  d.k_cut = 0x7FFFFFFF;
  d.p_key = 0xFFFFFFFFu;
  d.p_cut = 0x7FFFFFFF;
  d.kept = -1;
  unsigned long long S = cr->SE;
  const int bstar = cr->b;
  if (topp && bstar >= 0) {
    auto wk = [&](uint32_t key) { return to_fix(expf(key_to_z(key) - sc.mx)); };
    const unsigned long long need = cr->need;
    uint32_t K = 0xFFFFFFFFu;
    int cut = 0x7FFFFFFF;
    unsigned long long in_bin = 0;
    // one round trip: the list's length and its first 32 entries
    const int lane = threadIdx.x & 31;
    const int cnt = __ldcg(&a.ccnt[t]);
    uint32_t k0 = 0xFFFFFFFFu;
    int i0 = 0x7FFFFFFF;
    if (threadIdx.x < 32) {
      k0 = __ldcg(&a.ckey[(size_t)t * kFlatCandCap + lane]);
      i0 = __ldcg(&a.cid[(size_t)t * kFlatCandCap + lane]);
    }
    bool ok = false;
    if (cnt >= 1 && cnt <= 32) {
      // a short list: warp 0, one entry per lane
      ok = fl_warp_cross(threadIdx.x < 32 && lane < cnt, k0, i0, cnt, need, wk, &K, &cut, &in_bin, &s_ok, &s_K,
                         &s_cut, &s_in);
    } else if (cnt > 32 && cnt <= kFlatCandCap) {
      // the crossing sub-bin of the gather's sub-histogram, then that
      // sub-bin's entries of the list (typically a few) on warp 0
      static_assert(kFlatCandCap <= 2 * kST, "two list entries per thread");
      unsigned long long sv[kFlPer];
      fl_bins_load(a.sub_w + (size_t)t * kFlatBins, sv);
      uint32_t ek[2];
      int ei[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int q = 2 * threadIdx.x + e;
        ek[e] = q < cnt ? __ldcg(&a.ckey[(size_t)t * kFlatCandCap + q]) : 0xFFFFFFFFu;
        ei[e] = q < cnt ? __ldcg(&a.cid[(size_t)t * kFlatCandCap + q]) : -1;
      }
      FlCross& sc2 = s_cr;  // reused: the calling CTA's crossing was read above
      __syncthreads();
      fl_reach(sm, sv, need, &sc2);
      const int sstar = sc2.b;
      if (sstar >= 0) {
        const unsigned long long need2 = sc2.need;
        const FlSub su = fl_sub(sc, bstar);
        if (threadIdx.x == 0) sm->ccount = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if (ei[e] >= 0 && fl_sub_of(su, ek[e]) == sstar) {
            const int pos = atomicAdd(&sm->ccount, 1);
            if (pos < 32) {
              mk[pos] = ek[e];
              mi[pos] = ei[e];
            }
          }
        __syncthreads();
        const int c2 = sm->ccount;
        if (c2 >= 1 && c2 <= 32) {
          const bool have = threadIdx.x < 32 && lane < c2;
          const uint32_t kk = have ? mk[lane] : 0xFFFFFFFFu;
          const int ii = have ? mi[lane] : 0x7FFFFFFF;
          unsigned long long in2 = 0;
          ok = fl_warp_cross(have, kk, ii, c2, need2, wk, &K, &cut, &in2, &s_ok, &s_K, &s_cut, &s_in);
          if (ok) in_bin = (need - need2) + in2;
        }
      }
      if (!ok)
        ok = fl_sorted_cross(a.ckey + (size_t)t * kFlatCandCap, a.cid + (size_t)t * kFlatCandCap, cnt, need, wk, mk,
                             mi, sm->wsum, &K, &cut, &in_bin, &s_ok, &s_K, &s_cut, &s_in);
    }
    if (!ok) {
      load_window(sm, a.hist + (size_t)k.r * a.W, a.W, a.drafts + (size_t)k.r * a.depth, k.i);
      const bool pen = rp.rep_penalty != 1.f;
      if (pen) build_bitmap(sm, bits, 0, a.V);
      auto zof = [&](int j) {
        float z = __ldg(k.lg + j);
        if (pen && bit(bits, j)) z = penalize(z, rp.rep_penalty);
        return z / rp.temperature + 0.0f;
      };
      fl_exact_cut(sm, a.V, zof, sc, bstar, need, K, cut, &in_bin);
    }
    d.p_key = K;
    d.p_cut = cut;
    // the kept mass: every bin before the crossing one, then that bin's
    // elements up to the bound; with min-p the shorter of the two prefixes
    S = (cr->target - need) + in_bin;
    if (rp.min_p > 0.f && !(expf(key_to_z(K) - sc.mx) >= rp.min_p)) S = __ldcg(&a.sminp[t]);
  } else if (rp.min_p > 0.f) {
    S = __ldcg(&a.sminp[t]);
  }
  d.m = sc.mx;
  d.S = (float)((double)S / kFix);
  if (threadIdx.x == 0) a.desc[t] = d;
}

// Warp 0 (every lane): the row's accept chain over its d drafts, from the
// descriptors, the raw target logits at the drafts and q. Lane i evaluates
// draft x_{i+1} against target row i under row i's penalty window; hw holds
// the row's history (W) then its drafts (d), staged by the block.
__device__ int fl_chain(const FlatArgs& a, int r, const RowParams& rp, const int* hw) {
  const int lane = threadIdx.x & 31, d = a.depth;
  bool acc = false;
  if (lane < d) {
    const int x = hw[a.W + lane];
    if (x >= 0 && x < a.V) {  // an out-of-range draft is rejected, never dereferenced
      const int t = r * (d + 1) + lane;
      const TDesc dd = a.desc[t];
      const float raw = __ldg(a.logits + (size_t)t * a.V + x);
      const float qv = rp.argmax_draft ? 1.f : __ldg(a.q + ((size_t)r * d + lane) * a.V + x);
      bool px = false;
      const int drop = lane < a.W ? lane : a.W;
      for (int q = drop; q < a.W; ++q) px |= hw[q] == x;
      for (int q = lane > a.W ? lane - a.W : 0; q < lane; ++q) px |= hw[a.W + q] == x;
      const float pv = eval_p(dd, rp, raw, px, x);
      acc = qv > 0.f && a.u[(size_t)r * (d + 1) + lane] < pv / qv;
    }
  }
  const unsigned rej = ~__ballot_sync(0xFFFFFFFFu, acc) & (d >= 32 ? 0xFFFFFFFFu : ((1u << d) - 1u));
  return rej ? __ffs(rej) - 1 : d;
}

// The draw's row: its task, descriptor, weights of element v.
struct FlDraw {
  int n, tn;
  bool residual;
  const float* lg;
  const float* qn;
  int xr;
  TDesc dn;
};
__device__ FlDraw fl_draw_row(const FlatArgs& a, int r, int n, const RowParams& rp) {
  FlDraw w;
  w.n = n;
  w.tn = a.mode == 0 ? r : r * (a.depth + 1) + n;
  w.lg = a.mode == 0 ? a.logits + (size_t)r * a.ld : a.logits + (size_t)w.tn * a.V;
  w.residual = a.mode == 1 && n < a.depth;
  w.qn = (w.residual && !rp.argmax_draft) ? a.q + ((size_t)r * a.depth + n) * a.V : nullptr;
  w.xr = (w.residual && rp.argmax_draft) ? a.drafts[(size_t)r * a.depth + n] : -1;
  w.dn = a.desc[w.tn];
  return w;
}

// Warp slice wi of part p (of P2) of a row: [*s0, *s0 + *sn) within the
// part, which starts at *v0. Every bound is a multiple of 4.
__device__ __forceinline__ void fl_slice(const FlatArgs& a, int p, int wi, int* v0, int* s0, int* sn) {
  const int per = fl_per(a.V, a.P2);
  *v0 = min(p * per, a.V);
  const int n = min(per, a.V - *v0);
  const int wsz = fl_per(n, kST / 32);
  *s0 = min(wi * wsz, n);
  *sn = min(wsz, n - *s0);
}

// The penalty window of position i from hw = history (W) then drafts: the W
// tokens hw[i, i + W).
__device__ void window_from(SampleSmem* sm, const int* hw, int W, int i) {
  for (int q = threadIdx.x; q < W; q += kST) sm->wtok[q] = hw[i + q];
  if (threadIdx.x == 0) sm->nwin = W;
  __syncthreads();
}

__device__ void fl_pick_greedy(const FlatArgs& a, int r);
__device__ void fl_pick_row(const FlatArgs& a, int r, unsigned char* dyn, const FlDraw& w, const RowParams& rp);

__global__ void __launch_bounds__(kST, 2) k_fl_sums(const __grid_constant__ FlatArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  uint32_t* bits = reinterpret_cast<uint32_t*>(dyn + fl_bits_off());
  __shared__ int s_n, s_last;
  __shared__ int s_hw[128 + 32];
  const int r = blockIdx.y, p = blockIdx.x;
  const RowParams rp = a.p[r];
  if (rp.greedy) {
    pdl_wait();
    pdl_trigger();
    if (p == 0) fl_pick_greedy(a, r);
    return;
  }
  const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int v0, s0, sn;
  fl_slice(a, p, wi, &v0, &s0, &sn);
  const int n = min(fl_per(a.V, a.P2), a.V - v0);
  // history then drafts: inputs of the chain, staged before the wait
  for (int q = threadIdx.x; q < a.W + a.depth; q += kST)
    s_hw[q] = q < a.W ? a.hist[(size_t)r * a.W + q] : a.drafts[(size_t)r * a.depth + q - a.W];
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < 32) {
    const int nn = a.mode == 0 ? a.pos : fl_chain(a, r, rp, s_hw);
    if (threadIdx.x == 0) s_n = nn;
  }
  __syncthreads();
  // one round trip: the drawn row's descriptor and this warp's slice of it
  const FlDraw w = fl_draw_row(a, r, s_n, rp);
  const float4* l4 = reinterpret_cast<const float4*>(w.lg + v0 + s0);
  const float4* q4 = w.qn ? reinterpret_cast<const float4*>(w.qn + v0 + s0) : nullptr;
  const int n4 = sn / 4;
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 xa = zero4, qa = zero4;
  if (lane < n4) {
    xa = __ldg(l4 + lane);
    if (q4) qa = __ldg(q4 + lane);
  }
  window_from(sm, s_hw, a.W, w.n);
  const bool pen = rp.rep_penalty != 1.f;
  if (pen) build_bitmap(sm, bits, v0, n);
  // each warp sums its own slice (lanes read consecutive 16-byte vectors); a
  // rolled loop with the next vector in flight, one copy of the element code
  float4* o4 = a.mode == 0 ? reinterpret_cast<float4*>(a.q + ((size_t)r * a.depth + a.pos) * a.V + v0 + s0) : nullptr;
  unsigned long long wp = 0, wr = 0;
  const int nu = (n4 - lane + 31) / 32;
#pragma unroll 1
  for (int u = 0; u < nu; ++u) {
    const int j4 = lane + 32 * u;
    float4 xn = zero4, qn = zero4;
    if (j4 + 32 < n4) {
      xn = __ldg(l4 + j4 + 32);
      if (q4) qn = __ldg(q4 + j4 + 32);
    }
    const int jj = s0 + 4 * j4;  // index within the part
    float4 pv4 = zero4;
#pragma unroll 1
    for (int e = 0; e < 4; ++e) {
      const float x = e == 0 ? xa.x : (e == 1 ? xa.y : (e == 2 ? xa.z : xa.w));
      const float qx = e == 0 ? qa.x : (e == 1 ? qa.y : (e == 2 ? qa.z : qa.w));
      const int v = v0 + jj + e;
      const float pv = eval_p(w.dn, rp, x, pen && bit(bits, jj + e), v);
      wp += to_fix(pv);
      if (w.residual) {
        const float qv = w.xr >= 0 ? (v == w.xr ? 1.f : 0.f) : qx;
        const float rv = pv - qv;
        wr += to_fix(rv > 0.f ? rv : 0.f);
      }
      if (e == 0) pv4.x = pv;
      else if (e == 1) pv4.y = pv;
      else if (e == 2) pv4.z = pv;
      else pv4.w = pv;
    }
    if (o4) o4[j4] = pv4;
    xa = xn;
    qa = qn;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    wp += __shfl_xor_sync(0xFFFFFFFFu, wp, o);
    wr += __shfl_xor_sync(0xFFFFFFFFu, wr, o);
  }
  if (lane == 0) {
    unsigned long long* ws = a.wsum + ((((size_t)r * a.P2 + p) * (kST / 32)) + wi) * 2;
    ws[0] = wr;
    ws[1] = wp;
  }
  // the last of the row's CTAs to finish draws
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&a.scnt[r], 1) == a.P2 - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  fl_pick_row(a, r, dyn, w, rp);
}

// The row's outputs: accepted count nacc (verify) and the drawn token y.
__device__ void fl_write_row(const FlatArgs& a, int r, int nacc, int y) {
  const int d = a.depth;
  const int32_t* dr = a.drafts + (size_t)r * d;
  if (a.mode == 0) {
    a.draft_out[(size_t)r * d + a.pos] = y;
    return;
  }
  a.n_acc[r] = nacc;
  int32_t* o = a.out_tok + (size_t)r * (d + 1);
  for (int i = 0; i <= d; ++i) o[i] = i < nacc ? dr[i] : (i == nacc ? y : -1);
  if (a.h_rec) {
    // the record's tokens are visible to the host before its count
    int32_t* hr = a.h_rec + (size_t)r * (d + 2);
    for (int i = 0; i <= d; ++i) hr[1 + i] = o[i];
    st_release_sys(hr, nacc);
  }
  if (a.stats) {
    int32_t* st = a.stats + (size_t)r * (d + 2);
    st[0] += 1;
    if (nacc < d) st[1] += 1;
    for (int i = 1; i <= nacc; ++i) st[1 + i] += 1;
  }
}

// Warp 0 of one CTA, greedy row: point masses at the argmax of each position
// (the first kernel's part maxima); accept while the draft is the argmax of
// the row before it.
__device__ void fl_pick_greedy(const FlatArgs& a, int r) {
  if (threadIdx.x >= 32) return;
  const int d = a.depth, lane = threadIdx.x;
  const int np = a.mode == 0 ? 1 : d + 1;
  int am = 0;
  for (int i = 0; i < np; ++i) {
    const int t = a.mode == 0 ? r : r * (d + 1) + i;
    const unsigned long long* slot = a.amax + (size_t)t * a.P;
    unsigned long long best = lane < a.P ? __ldcg(slot + lane) : 0ull;
    if (lane + 32 < a.P) best = max(best, __ldcg(slot + lane + 32));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
    if (lane == i) am = best ? (int)(0xFFFFFFFFu - (uint32_t)best) : 0;
  }
  int nacc = 0, y;
  if (a.mode == 0) {
    y = __shfl_sync(0xFFFFFFFFu, am, 0);
  } else {
    const int x = lane < d ? a.drafts[(size_t)r * d + lane] : -1;
    const unsigned miss = __ballot_sync(0xFFFFFFFFu, lane < d && !(x >= 0 && x < a.V && x == am));
    nacc = miss ? __ffs(miss) - 1 : d;
    y = __shfl_sync(0xFFFFFFFFu, am, nacc);
  }
  if (lane == 0) fl_write_row(a, r, nacc, y);
}

// One CTA (the row's last to finish its sums), sampled row: the draw from
// the slices' sums, then the element inside the chosen slice.
__device__ void fl_pick_row(const FlatArgs& a, int r, unsigned char* dyn, const FlDraw& w, const RowParams& rp) {
  SampleSmem* sm = reinterpret_cast<SampleSmem*>(dyn);
  uint32_t* bits = reinterpret_cast<uint32_t*>(dyn + fl_bits_off());
  __shared__ int s_slice, s_y;
  __shared__ unsigned long long s_need;
  __shared__ unsigned long long s_wr[kST / 32], s_wp[kST / 32];
  const int d = a.depth, lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int NS = a.P2 * (kST / 32);
  // the row's slices in order, two per thread: one round trip
  const unsigned long long* ws = a.wsum + (size_t)r * NS * 2;
  unsigned long long pr0 = 0, pr1 = 0, pp0 = 0, pp1 = 0;
  if (2 * (int)threadIdx.x < NS) {
    pr0 = __ldcg(ws + 4 * threadIdx.x + 0);
    pp0 = __ldcg(ws + 4 * threadIdx.x + 1);
  }
  if (2 * (int)threadIdx.x + 1 < NS) {
    pr1 = __ldcg(ws + 4 * threadIdx.x + 2);
    pp1 = __ldcg(ws + 4 * threadIdx.x + 3);
  }
  // block scans of both sums at once
  const unsigned long long mr = pr0 + pr1, mp = pp0 + pp1;
  unsigned long long ir = mr, ip = mp;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long xr = __shfl_up_sync(0xFFFFFFFFu, ir, o);
    const unsigned long long xp = __shfl_up_sync(0xFFFFFFFFu, ip, o);
    if (lane >= o) {
      ir += xr;
      ip += xp;
    }
  }
  __syncthreads();
  if (lane == 31) {
    s_wr[wi] = ir;
    s_wp[wi] = ip;
  }
  if (threadIdx.x == 0) {
    // rounding left the target past the total: the last slice
    s_slice = NS - 1;
    s_need = 1ull;
    s_y = -1;
  }
  __syncthreads();
  unsigned long long tr = 0, tp = 0, br = 0, bp = 0;
  for (int q = 0; q < kST / 32; ++q) {
    if (q < wi) {
      br += s_wr[q];
      bp += s_wp[q];
    }
    tr += s_wr[q];
    tp += s_wp[q];
  }
  const bool use_r = w.residual && tr > 0;
  const unsigned long long tot = use_r ? tr : tp;
  int y = -1;
  if (tot > 0) {
    const float uu = a.mode == 0 ? a.u[(size_t)r * d + a.pos] : a.u[(size_t)r * (d + 1) + d];
    const unsigned long long target = (unsigned long long)floor((double)uu * (double)tot) + 1ull;
    const unsigned long long w0 = use_r ? pr0 : pp0, mine = use_r ? mr : mp;
    const unsigned long long excl = use_r ? br + ir - mr : bp + ip - mp;
    if (excl < target && target <= excl + mine) {
      const bool first = target <= excl + w0;
      s_slice = first ? 2 * threadIdx.x : 2 * threadIdx.x + 1;
      s_need = first ? target - excl : target - excl - w0;
    }
    __syncthreads();
    int v0, s0, sn;
    fl_slice(a, s_slice / (kST / 32), s_slice % (kST / 32), &v0, &s0, &sn);
    // the window of the drawn row is in shared memory already
    const bool pen = rp.rep_penalty != 1.f;
    if (pen) build_bitmap(sm, bits, v0 + s0, sn);
    if (threadIdx.x < 32) {
      // warp 0 walks the slice in chunks of 128 elements (a rolled loop, the
      // next chunk's loads in flight): smallest id whose running weight
      // reaches need
      unsigned long long need = s_need;
      const float4* l4 = reinterpret_cast<const float4*>(w.lg + v0 + s0);
      const float4* q4 = w.qn ? reinterpret_cast<const float4*>(w.qn + v0 + s0) : nullptr;
      const int n4 = sn / 4;
      const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 xa = zero4, qa = zero4;
      if (lane < n4) {
        xa = __ldg(l4 + lane);
        if (q4) qa = __ldg(q4 + lane);
      }
#pragma unroll 1
      for (int b0 = 0; b0 < n4; b0 += 32) {
        const int j4 = b0 + lane;
        float4 xn = zero4, qn = zero4;
        if (j4 + 32 < n4) {
          xn = __ldg(l4 + j4 + 32);
          if (q4) qn = __ldg(q4 + j4 + 32);
        }
        unsigned long long wt[4] = {0ull, 0ull, 0ull, 0ull};
        if (j4 < n4) {
#pragma unroll 1
          for (int e = 0; e < 4; ++e) {
            const float x = e == 0 ? xa.x : (e == 1 ? xa.y : (e == 2 ? xa.z : xa.w));
            const float qx = e == 0 ? qa.x : (e == 1 ? qa.y : (e == 2 ? qa.z : qa.w));
            const int v = v0 + s0 + 4 * j4 + e;
            const float pv = eval_p(w.dn, rp, x, pen && bit(bits, 4 * j4 + e), v);
            unsigned long long wgt;
            if (!use_r) {
              wgt = to_fix(pv);
            } else {
              const float qv = w.xr >= 0 ? (v == w.xr ? 1.f : 0.f) : qx;
              const float rv = pv - qv;
              wgt = to_fix(rv > 0.f ? rv : 0.f);
            }
            if (e == 0) wt[0] = wgt;
            else if (e == 1) wt[1] = wgt;
            else if (e == 2) wt[2] = wgt;
            else wt[3] = wgt;
          }
        }
        const unsigned long long ls = wt[0] + wt[1] + wt[2] + wt[3];
        unsigned long long li = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long x = __shfl_up_sync(0xFFFFFFFFu, li, o);
          if (lane >= o) li += x;
        }
        const unsigned long long ct = __shfl_sync(0xFFFFFFFFu, li, 31);
        if (need <= ct) {
          const unsigned long long ex = li - ls;
          if (ex < need && need <= li) {
            unsigned long long cum = ex;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              cum += wt[e];
              if (wt[e] > 0 && cum >= need) {
                s_y = v0 + s0 + 4 * j4 + e;
                break;
              }
            }
          }
          break;  // warp-uniform: every lane saw the same chunk total
        }
        need -= ct;
        xa = xn;
        qa = qn;
      }
    }
    __syncthreads();
    y = s_y;
  }
  if (y < 0) y = w.dn.argmax;
  if (threadIdx.x == 0) fl_write_row(a, r, a.mode == 0 ? 0 : w.n, y);
}

static size_t fl_align(size_t b) { return (b + 255) & ~size_t(255); }

size_t flat_workspace_bytes(int rows, int tasks) {
  const size_t T = (size_t)tasks, R = (size_t)rows, P = kFlatMaxParts;
  return fl_align(sizeof(TDesc) * T) + fl_align(8 * T * P) + fl_align(4 * T * P) + 2 * fl_align(8 * T * kFlatHistBins) +
         fl_align(8 * T) + fl_align(4 * T) + 2 * fl_align(4 * T * kFlatCandCap) + fl_align(16 * R * P * (kST / 32)) +
         fl_align(4 * R) + fl_align(4 * T) + fl_align(4 * R);
}

bool flat_fits(const RowParams* p, int rows, int V, const float* logits, long long ld) {
  if (V % 4 != 0 || V < 2048 || (reinterpret_cast<uintptr_t>(logits) & 15) != 0 || ld % 4 != 0) return false;
  for (int r = 0; r < rows; ++r)
    if (!p[r].greedy && p[r].top_k > 0 && p[r].top_k < V) return false;
  return true;
}

bool launch_flat(FlatArgs a, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!ws || ws_bytes < flat_workspace_bytes(a.rows, a.tasks) || a.depth + 1 > 32) return false;
  if ((reinterpret_cast<uintptr_t>(a.q) & 15) != 0) return false;
  const int sms = device_sm_count();
  a.nsr = 0;
  for (int r = 0; r < a.rows; ++r)
    if (!a.p[r].greedy) a.srow[a.nsr++] = r;
  const int nst = a.nsr * (a.mode == 0 ? 1 : a.depth + 1);
  // parts per unit: about two CTAs per SM over the units that do the work
  auto parts = [&](int units) { return std::max(1, std::min({2 * sms / std::max(units, 1), kFlatMaxParts, a.V / 2048})); };
  a.P = parts(a.tasks);
  a.Ps = parts(nst);
  a.P2 = a.nsr ? parts(a.nsr) : 1;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t T = (size_t)a.tasks, R = (size_t)a.rows, PM = kFlatMaxParts;
  auto take = [&](size_t bytes) {
    uint8_t* q = w;
    w += fl_align(bytes);
    return q;
  };
  a.desc = reinterpret_cast<TDesc*>(take(sizeof(TDesc) * T));
  a.amax = reinterpret_cast<unsigned long long*>(take(8 * T * PM));
  a.zmin = reinterpret_cast<float*>(take(4 * T * PM));
  a.hist_w = reinterpret_cast<unsigned long long*>(take(8 * T * kFlatHistBins));
  a.sub_w = reinterpret_cast<unsigned long long*>(take(8 * T * kFlatHistBins));
  a.sminp = reinterpret_cast<unsigned long long*>(take(8 * T));
  a.ccnt = reinterpret_cast<int32_t*>(take(4 * T));
  a.ckey = reinterpret_cast<uint32_t*>(take(4 * T * kFlatCandCap));
  a.cid = reinterpret_cast<int32_t*>(take(4 * T * kFlatCandCap));
  a.wsum = reinterpret_cast<unsigned long long*>(take(16 * R * PM * (kST / 32)));
  a.nstop = reinterpret_cast<int32_t*>(take(4 * R));
  a.gcnt = reinterpret_cast<int32_t*>(take(4 * T));
  a.scnt = reinterpret_cast<int32_t*>(take(4 * R));
  const size_t base = (sizeof(SampleSmem) + 15) & ~size_t(15);
  auto sm_part = [&](int P) { return base + 4 * (size_t)((fl_per(a.V, P) + 31) / 32 + 1); };
  const size_t sm_hist = fl_hist_off(fl_per(a.V, a.Ps)) + 8 * (size_t)kFlatBins;
  if (fl_sub_off(a.V, fl_per(a.V, a.Ps)) + 8 * (size_t)kFlatBins > 226 * 1024 || sm_hist > 226 * 1024) return false;
  {
    // the kernels' dynamic shared memory limit, raised once per device
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      for (auto k : {k_fl_stats, k_fl_hist, k_fl_gather, k_fl_sums})
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 226 * 1024);
      done[dev] = true;
    }
  }
  launch_pdl(k_fl_stats, dim3(a.P, a.tasks), dim3(kST), sm_part(a.P), s, a);
  int n = 1;
  if (nst > 0) {
    launch_pdl(k_fl_hist, dim3(a.Ps, nst), dim3(kST), sm_hist, s, a);
    launch_pdl(k_fl_gather, dim3(a.Ps, nst), dim3(kST), fl_sub_off(a.V, fl_per(a.V, a.Ps)) + 8 * (size_t)kFlatBins,
               s, a);
    n += 2;
  }
  launch_pdl(k_fl_sums, dim3(a.P2, a.rows), dim3(kST), sm_part(a.P2), s, a);
  count_launch(n + 1);
  return true;
}

static int sample_smem(int V, int C = 0, int P = 0) {
  const int per = (V + kClusterCTAs - 1) / kClusterCTAs;
  const size_t cand = 16 + (size_t)C * 8 + (size_t)P * 8 + (size_t)C * 4 + 4 + (size_t)C * 8;
  return (int)(sizeof(SampleSmem) + sizeof(float) * per + sizeof(uint32_t) * ((per + 31) / 32) + cand + 32);
}

template <class Args>
static void launch_cluster(void (*k)(Args), const Args& a, int tasks, int V, cudaStream_t s, int C = 0, int P = 0) {
  const int smem = sample_smem(V, C, P);
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tasks * kClusterCTAs);
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCTAs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, k, a);
  count_launch();
}

void launch_sample(const SampleArgs& a0, cudaStream_t s) {
  if (a0.mode == 0 && topk_fits(a0.p, a0.rows, a0.V, a0.logits, a0.ld)) {
    TopkArgs t;
    memset(&t, 0, sizeof(t));
    t.mode = 0; t.rows = a0.rows; t.V = a0.V; t.W = a0.W; t.depth = a0.depth; t.pos = a0.pos;
    t.logits = a0.logits; t.ld = a0.ld; t.hist = a0.hist; t.drafts = a0.drafts; t.u = a0.u; t.q = a0.q;
    t.draft_out = a0.draft_out; t.status = a0.status; t.q_zeroed = a0.q_zeroed;
    for (int r = 0; r < a0.rows; ++r) t.p[r] = a0.p[r];
    launch_topk(t, s);
    return;
  }
  if (a0.mode == 0 && a0.flat_ws && flat_fits(a0.p, a0.rows, a0.V, a0.logits, a0.ld)) {
    FlatArgs f;
    memset(&f, 0, sizeof(f));
    f.mode = 0; f.rows = a0.rows; f.V = a0.V; f.W = a0.W; f.depth = a0.depth; f.pos = a0.pos; f.tasks = a0.rows;
    f.logits = a0.logits; f.ld = a0.ld; f.hist = a0.hist; f.drafts = a0.drafts; f.u = a0.u; f.q = a0.q;
    f.draft_out = a0.draft_out; f.status = a0.status;
    for (int r = 0; r < a0.rows; ++r) f.p[r] = a0.p[r];
    if (launch_flat(f, a0.flat_ws, a0.flat_ws_bytes, s)) return;
  }
  SampleArgs a = a0;
  int C = 1;
  for (int r = 0; r < a.rows; ++r) {
    if (a.p[r].greedy) continue;
    const int c = (a.p[r].top_k > 0 && a.p[r].top_k < a.V) ? a.p[r].top_k : kCandTopP;
    C = c > C ? c : C;
  }
  C = C * 4 < (C > 1024 ? C : 1024) ? C * 4 : (C > 1024 ? C : 1024);  // room for the value-binned superset
  int P = 1;
  while (P < kClusterCTAs * C) P <<= 1;
  a.cand = C;
  a.merge = P;
  const int tasks = a.mode == 0 ? a.rows : a.rows * (a.depth + 1);
  launch_cluster(k_sample, a, tasks, a.V, s, C, P);
}

void launch_verify(const VerifyArgs& a, cudaStream_t s) { launch_cluster(k_verify, a, a.rows, a.V, s); }

void launch_verify_stream(const VerifyArgs& a0, cudaStream_t s) {
  VerifyArgs a = a0;
  int ns = 0;
  size_t smem = verify_stream_smem(a.V, &ns);
  // rows starting on 16-byte boundaries stream through the shared-memory ring
  // (bulk copies); others take 4-byte loads into registers
  const bool vec = (a.V & 3) == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15) == 0 && ns >= 2;
  a.ring_ns = vec ? ns : 0;
  if (!vec) smem = StreamLayout(a.V, 0).total;
  auto k = vec ? k_verify_stream<true> : k_verify_stream<false>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_pdl(k, dim3(a.rows * (a.depth + 1)), dim3(kST), smem, s, a);
  count_launch();
  launch_verify_finish(a, s);
}

void launch_verify_finish(const VerifyArgs& a, cudaStream_t s) {
  launch_pdl(k_verify_finish, dim3(a.rows), dim3(kStreamTopK), 0, s, a);
  count_launch();
}

// Per device: whether each greedy-verify instance can be launched in 16-CTA
// clusters (checked once per device, under a lock).
struct GreedyDevInfo {
  bool ready = false;
  int wide16[2] = {0, 0};
};

void launch_verify_greedy(const VerifyArgs& a0, cudaStream_t s) {
  VerifyArgs a = a0;
  a.vec_ok = (a.V % 4 == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15) == 0) ? 1 : 0;
  static std::mutex mu;
  static GreedyDevInfo info[kMaxDevices];
  const int sms = device_sm_count();
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kST);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void (*kern[2])(VerifyArgs) = {k_verify_greedy<false>, k_verify_greedy<true>};
  int wide16[2];
  {
    std::lock_guard<std::mutex> lock(mu);
    GreedyDevInfo& in = info[dev];
    if (!in.ready) {
      for (int w = 0; w < 2; ++w) {
        in.wide16[w] = 0;
        if (cudaFuncSetAttribute(kern[w], cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
          int nclusters = 0;
          cfg.gridDim = dim3(16);
          attr[0].val.clusterDim.x = 16;
          if (cudaOccupancyMaxActiveClusters(&nclusters, kern[w], &cfg) == cudaSuccess && nclusters > 0)
            in.wide16[w] = 1;
        }
      }
      cudaGetLastError();
      in.ready = true;
    }
    wide16[0] = in.wide16[0];
    wide16[1] = in.wide16[1];
  }
  // one row per cluster; many rows take narrower clusters so that rows x CTAs
  // fits one wave (each CTA then streams a wider slice). Slices wider than one
  // round of the grouped loads take the double-buffered instance.
  const int nc0 = (wide16[0] && wide16[1]) ? 16 : kClusterCTAs;
  int nc = nc0;
  while (nc > 1 && a.rows * nc > sms) nc /= 2;
  int per = ((a.V + nc - 1) / nc + 3) & ~3;
  const int w = (a.vec_ok && (per / 4 + kST - 1) / kST > kGreedyBuf) ? 1 : 0;
  if (w) {  // the wide instance fits two CTAs per SM: twice the CTAs per row
    nc = nc0;
    while (nc > 1 && a.rows * nc > 2 * sms) nc /= 2;
  }
  cfg.gridDim = dim3(a.rows * nc);
  attr[0].val.clusterDim.x = nc;
  cudaLaunchKernelEx(&cfg, kern[w], a);
  count_launch();
}

}  // namespace mtp
