// C ABI of the MTP speculative-decoding step: validation, the head handle,
// and the launch sequence of one head call. See include/mtp.h for the
// contract of every entry point.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mtp.h"
#include "kernels.h"

using namespace mtp;

constexpr int kTcFlushMinItems = 16;  // below this the flush stays on the GEMV path

namespace mtp {
unsigned long long launches_so_far();

int device_sm_count() {
  static std::mutex mu;
  static int sms[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  std::lock_guard<std::mutex> lock(mu);
  if (sms[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 1;
    }
    sms[dev] = n;
  }
  return sms[dev];
}
}  // namespace mtp

namespace {
// One-shot test hook of the streaming verify's bounded waits
// (mtp_test_verify_stall): the ring stage to leave unfilled and the polls
// before a wait gives up.
std::atomic<int> g_stall_stage{-1};
std::atomic<unsigned> g_stall_polls{0};
}  // namespace

namespace {

// The fifteen tensors of the published head ("support the qwen3_5_mtp
// drafter" issue, "Where the MTP weights actually live").
enum TensorId {
  T_FC, T_NORM, T_PRE_E, T_PRE_H, T_IN, T_POST, T_GATE, T_UP, T_DOWN, T_Q, T_K, T_V, T_O, T_QN, T_KN, T_COUNT
};
const char* kNames[T_COUNT] = {
    "fc.weight",
    "norm.weight",
    "pre_fc_norm_embedding.weight",
    "pre_fc_norm_hidden.weight",
    "layers.0.input_layernorm.weight",
    "layers.0.post_attention_layernorm.weight",
    "layers.0.mlp.gate_proj.weight",
    "layers.0.mlp.up_proj.weight",
    "layers.0.mlp.down_proj.weight",
    "layers.0.self_attn.q_proj.weight",
    "layers.0.self_attn.k_proj.weight",
    "layers.0.self_attn.v_proj.weight",
    "layers.0.self_attn.o_proj.weight",
    "layers.0.self_attn.q_norm.weight",
    "layers.0.self_attn.k_norm.weight",
};

// Norm weights that take +1.0 in the raw-HF layout ("Upstream contract to
// port", sanitize paragraph: seven suffixes).
const char* kShiftSuffixes[7] = {
    ".input_layernorm.weight", ".post_attention_layernorm.weight", ".q_norm.weight", ".k_norm.weight",
    "norm.weight",             "pre_fc_norm_embedding.weight",    "pre_fc_norm_hidden.weight",
};

bool ends_with(const std::string& s, const char* suf) {
  const size_t n = std::strlen(suf);
  return s.size() >= n && s.compare(s.size() - n, n, suf) == 0;
}

enum ProfKind {
  PK_FC, PK_QKV, PK_QKV_POST, PK_ATTN, PK_O, PK_GATEUP, PK_DOWN, PK_LMHEAD, PK_SAMPLE, PK_FLUSH_FC, PK_FLUSH_KV,
  PK_ROLLBACK, PK_COUNT
};
const char* kProfNames[PK_COUNT] = {"fc",      "qkv",    "qkv_post", "attention", "o_proj",   "gate_up",
                                    "down",    "lm_head", "sample",  "flush_fc",  "flush_kv", "rollback"};

struct GemvPlan {
  int mt, S, ngroups, smem;
};

}  // namespace

struct mtp_handle {
  mtp_config cfg;
  std::string arch;
  int sms = 0;
  const void* w[T_COUNT] = {};
  const void* embed = nullptr;
  const void* lm = nullptr;
  mtp_kv kv{};
  float* norms = nullptr;
  float* nrm[T_COUNT] = {};
  // scratch
  float *h0 = nullptr, *qkv = nullptr, *qrot = nullptr, *o = nullptr, *h1 = nullptr, *mlp = nullptr,
        *h2 = nullptr, *logits = nullptr, *po = nullptr, *pml = nullptr, *part = nullptr, *gmax = nullptr;
  int *gidx = nullptr, *counters = nullptr, *done = nullptr, *walk = nullptr;
  float* ssq = nullptr;                   // per-split sums of squares of a GEMV's x, [S][8]
  uint16_t *xb = nullptr, *bb = nullptr;  // bf16 activations of the tensor-core flush
  double* inv_freq = nullptr;             // RoPE frequencies theta^(-2i/dh), [dh/2]
  float* tcpart = nullptr;                // split-K partial tiles of the tensor-core flush
  uint16_t* x2 = nullptr;                 // hi/lo bf16 activations of the tensor-core GEMV
  float* tvpart = nullptr;                // its split-K partials
  uint8_t* flat_ws = nullptr;             // scratch of the draft-side flat transform
  size_t flat_ws_bytes = 0;
  bool tc_gemv = false;                   // batched GEMVs on tcgen05 (bf16 weights)
  uint8_t* lmq = nullptr;                 // fp8 e4m3 copy of the draft head (mtp_set_draft_head)
  float* lmq_scale = nullptr;             // its per-row scales
  bool lm_fp8 = false;
  int32_t* status = nullptr;
  size_t part_floats = 0;
  int max_chunks = 0, lm_groups_max = 0, counters_n = 0;
  std::vector<void*> allocs;
  // host mirror of the row lengths
  std::vector<int> len, keep, drafted_len;
  // profiling
  uint32_t prof = 0;  // bit mask of profiled kinds
  std::vector<cudaEvent_t> ev_pool;
  struct Rec { int kind; cudaEvent_t a, b; };
  std::vector<Rec> recs;
  size_t ev_next = 0;
};

namespace {

mtp_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? MTP_OK : MTP_ERR_CUDA; }

template <typename T>
mtp_status alloc(mtp_handle* h, T** p, size_t n) {
  void* q = nullptr;
  if (n == 0) n = 1;
  if (cudaMalloc(&q, n * sizeof(T)) != cudaSuccess) return MTP_ERR_CUDA;
  h->allocs.push_back(q);
  *p = static_cast<T*>(q);
  return MTP_OK;
}

void free_all(mtp_handle* h) {
  for (void* p : h->allocs) cudaFree(p);
  h->allocs.clear();
  for (auto e : h->ev_pool) cudaEventDestroy(e);
  h->ev_pool.clear();
}

int esize(int dt) { return dt == MTP_DTYPE_BF16 ? 2 : 4; }

GemvPlan plan_gemv(int N, int K, int M, int sms, bool fp8 = false) {
  GemvPlan p;
  p.mt = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
  const bool mma = fp8 && gemv_fp8_mma(N);
  const int rows = gemv_rows_per_group(p.mt, mma);
  p.ngroups = N / rows;
  // A block streams one K-slice of its group's rows with a fixed number of
  // loads in flight per lane, so its time follows the slice length. K is cut
  // so that the grid comes as close as it can to the two blocks per SM that
  // stay resident together (slices of at least 64 columns); grids wider than
  // that run in waves and keep whole rows.
  const int units = K / 16;
  p.S = std::max(1, std::min({16, 2 * sms / std::max(p.ngroups, 1), std::max(1, units / 4)}));
  // the staged activations (fp32), and on the tensor-core fp8 path their
  // three f16 parts besides
  auto smem = [&](int S) {
    const long long ks = gemv_slice_max(K, S);
    return p.mt * ks * 4 + (mma ? 3LL * p.mt * (ks + 4) * 2 : 0LL);
  };
  while (p.S < units && smem(p.S) > 96 * 1024) ++p.S;
  p.smem = (int)smem(p.S);
  return p;
}

// Profiling brackets around a launch group.
struct ProfScope {
  mtp_handle* h;
  cudaStream_t s;
  int kind;
  cudaEvent_t b = nullptr;
  ProfScope(mtp_handle* hh, cudaStream_t ss, int k) : h(hh), s(ss), kind(k) {
    if (!(h->prof >> kind & 1u)) return;
    cudaEvent_t a = next();
    b = next();
    cudaEventRecord(a, s);
    h->recs.push_back({kind, a, b});
  }
  ~ProfScope() {
    if (b) cudaEventRecord(b, s);
  }
  cudaEvent_t next() {
    if (h->ev_next >= h->ev_pool.size()) {
      cudaEvent_t e;
      cudaEventCreate(&e);
      h->ev_pool.push_back(e);
    }
    return h->ev_pool[h->ev_next++];
  }
};

// One GEMV over a list of items, in passes of at most 8.
struct GemvJob {
  const void* w[3];
  int seg_end[3];
  int N, K, pro, epi;
  // item-indexed operands (row stride in elements)
  const float* x;
  long long ldx;
  const float* nw;
  const float* nw2;
  float* y;
  long long ldy;
  const float* resid;
  long long ldr;
  // dual prologue sources
  const int32_t* tok;
  const int* tok_idx;        // per item
  const void* hid;
  const long long* hid_off;  // per item, elements
  int hid_dt;
  int32_t* amax_out;
  const int* amax_idx;
  bool fp8;               // w[0] holds e4m3 codes with per-row scales wscale
  const float* wscale;
  float* qzero;           // logits jobs: item m's draft distribution row (stride ldqz) zeroed
  long long ldqz;
};

// Batches of at least this many items run their GEMVs on the tensor cores:
// below it the CUDA-core GEMV keeps up with HBM.
constexpr int kTcGemvMinItems = 5;

// K splits of a tensor-core GEMV: the count (at most 8, at least 8 K tiles
// each) whose CTAs best fill whole waves of the `slots` resident CTAs, i.e.
// the largest C / (slots * ceil(C / slots)) for C = tiles * ks; ties keep the
// fewer splits. (Doubling the splits while the grid stays under the slots
// gives 320 CTAs for 304 slots at 40 row tiles: a second wave of 16.)
int tcv_splits(int tiles, int ktiles, int slots) {
  int best = 1;
  double best_e = 0.0;
  for (int ks = 1; ks <= 8; ++ks) {
    if (ks > 1 && ktiles / ks < 8) break;
    const long long C = (long long)tiles * ks;
    const long long waves = (C + slots - 1) / slots;
    const double e = (double)C / (double)(waves * slots);
    if (e > best_e + 1e-9) { best_e = e; best = ks; }
  }
  return best;
}

// Weight maps of a GEMV job on the tensor-core path; false if the job's row
// layout does not tile (segment boundaries off the 128-row grid).
bool tc_layout(const GemvJob& j, TcGemvLaunch& L) {
  std::memset(&L, 0, sizeof(L));
  L.N = j.N; L.K = j.K;
  if (j.K % 64 != 0) return false;
  if (j.epi == EPI_SWIGLU) {
    const int I = j.N / 2;
    if (I % 64 != 0) return false;
    L.swiglu = 1; L.nmaps = 2;
    L.w[0] = j.w[0]; L.w[1] = j.w[1]; L.w[2] = j.w[1];
    L.rows[0] = L.rows[1] = L.rows[2] = I;
    L.seg_end[0] = L.seg_end[1] = L.seg_end[2] = j.N;
    return true;
  }
  int start = 0;
  for (int sg = 0; sg < 3; ++sg) {
    L.seg_end[sg] = j.seg_end[sg];
    if (j.seg_end[sg] <= start) continue;
    if (j.seg_end[sg] < j.N && j.seg_end[sg] % 128 != 0) return false;
    L.w[L.nmaps] = j.w[sg];
    L.rows[L.nmaps] = j.seg_end[sg] - start;
    ++L.nmaps;
    start = j.seg_end[sg];
  }
  for (int i = L.nmaps; i < 3; ++i) { L.w[i] = L.w[L.nmaps - 1]; L.rows[i] = L.rows[L.nmaps - 1]; }
  return L.nmaps > 0 && start == j.N;
}

// prologue + hi/lo split, tcgen05 contraction, split sum + epilogue; passes of
// at most kTcGemvMaxItems items.
bool run_gemv_tc(mtp_handle* h, const GemvJob& j, int M, cudaStream_t s) {
  TcGemvLaunch L = {};
  if (!tc_layout(j, L)) return false;
  const int tiles = (j.N + 127) / 128;
  for (int m0 = 0; m0 < M; m0 += kTcGemvMaxItems) {
    const int mp = std::min(kTcGemvMaxItems, M - m0);
    const int NI = mp <= 8 ? 16 : (mp <= 16 ? 32 : (mp <= 32 ? 64 : 128));
    const int ks = tcv_splits(tiles, j.K / 64, h->sms * tc_gemv_blocks_per_sm(NI));
    TcxPrepArgs p;
    std::memset(&p, 0, sizeof(p));
    p.pro = j.pro; p.K = j.K; p.M = mp; p.MI = NI / 2;
    p.x = j.x ? j.x + (size_t)m0 * j.ldx : nullptr;
    p.ldx = j.ldx; p.nw = j.nw; p.nw2 = j.nw2; p.eps = h->cfg.eps;
    p.E = h->embed; p.wdt = h->cfg.dtype; p.vocab = h->cfg.vocab;
    p.tok = j.tok; p.hid = j.hid; p.hid_dt = j.hid_dt; p.X2 = h->x2; p.status = h->status;
    for (int m = 0; m < mp; ++m) {
      if (j.tok_idx) p.tok_idx[m] = j.tok_idx[m0 + m];
      if (j.hid_off) p.hid_off[m] = j.hid_off[m0 + m];
    }
    launch_tcx_prep(p, s);
    const bool direct = ks == 1 && (j.epi == EPI_STORE || j.epi == EPI_LOGITS);
    // one split of the logits: the contraction's own epilogue writes them,
    // clears q and takes each tile's argmax (no pass that reads them back)
    const bool fuse = direct && j.epi == EPI_LOGITS;
    float* y = j.y + (size_t)m0 * j.ldy;
    float* qz = j.qzero ? j.qzero + (size_t)m0 * j.ldqz : nullptr;
    L.M = mp; L.NI = NI; L.ksplit = ks; L.X2 = h->x2; L.status = h->status;
    L.out = direct ? y : h->tvpart;
    L.ld_item = direct ? j.ldy : j.N;
    L.ld_split = (long long)mp * j.N;
    L.fuse_logits = fuse ? 1 : 0;
    L.qzero = fuse ? qz : nullptr;
    L.ldqz = j.ldqz;
    L.gmax = h->gmax;
    L.gidx = h->gidx;
    if (!launch_tc_gemv(L, s)) return false;
    if (direct && j.epi == EPI_STORE) continue;
    TcFinishArgs f;
    std::memset(&f, 0, sizeof(f));
    f.part = L.out; f.ld_item = L.ld_item; f.ld_split = L.ld_split; f.ksplit = ks; f.M = mp; f.epi = j.epi;
    f.nout = j.epi == EPI_SWIGLU ? j.N / 2 : j.N;
    f.write_y = direct ? 0 : 1;
    f.y = y; f.ldy = j.ldy;
    f.resid = j.resid ? j.resid + (size_t)m0 * j.ldr : nullptr;
    f.ldr = j.ldr;
    f.gmax = h->gmax; f.gidx = h->gidx; f.done = h->done; f.amax_out = j.amax_out; f.status = h->status;
    for (int m = 0; m < mp; ++m) f.amax_idx[m] = j.amax_idx ? j.amax_idx[m0 + m] : 0;
    f.qzero = qz;
    f.ldqz = j.ldqz;
    if (fuse) {
      f.nout = tiles;  // the per-tile pairs
      launch_tcv_argmax(f, s);
    } else {
      launch_tcv_finish(f, s);
    }
  }
  return true;
}

void run_gemv(mtp_handle* h, const GemvJob& j, int M, cudaStream_t s) {
  if (!j.fp8 && h->tc_gemv && M >= kTcGemvMinItems && run_gemv_tc(h, j, M, s)) return;
  for (int m0 = 0; m0 < M; m0 += 8) {
    const int mp = std::min(8, M - m0);
    const GemvPlan pl = plan_gemv(j.N, j.K, mp, h->sms, j.fp8);
    GemvArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int i = 0; i < 3; ++i) { a.w[i] = j.w[i]; a.seg_end[i] = j.seg_end[i]; }
    a.N = j.N; a.K = j.K; a.S = pl.S; a.ngroups = pl.ngroups;
    a.pro = j.pro; a.epi = j.epi; a.M = mp; a.wdt = j.fp8 ? kDtypeFp8 : h->cfg.dtype;
    a.wscale = j.fp8 ? j.wscale : nullptr;
    a.x = j.x ? j.x + (size_t)m0 * j.ldx : nullptr;
    a.ldx = j.ldx;
    a.nw = j.nw; a.nw2 = j.nw2; a.eps = h->cfg.eps;
    a.E = h->embed;
    a.vocab = h->cfg.vocab;
    a.tok = j.tok;
    a.hid = j.hid;
    a.hid_dt = j.hid_dt;
    for (int m = 0; m < mp; ++m) {
      if (j.tok_idx) a.tok_idx[m] = j.tok_idx[m0 + m];
      if (j.hid_off) a.hid_off[m] = j.hid_off[m0 + m];
      if (j.amax_idx) a.amax_idx[m] = j.amax_idx[m0 + m];
    }
    a.y = j.y + (size_t)m0 * j.ldy;
    a.ldy = j.ldy;
    a.resid = j.resid ? j.resid + (size_t)m0 * j.ldr : nullptr;
    a.ldr = j.ldr;
    a.part = h->part;
    a.ssq = h->ssq;
    a.counters = h->counters;
    a.gmax = h->gmax;
    a.gidx = h->gidx;
    a.done = h->done;
    a.walk = h->walk;
    a.amax_out = j.amax_out;
    a.status = h->status;
    a.qzero = j.qzero ? j.qzero + (size_t)m0 * j.ldqz : nullptr;
    a.ldqz = j.ldqz;
    launch_gemv(pl.mt, a, pl.smem, s);
  }
}

bool fast_greedy(const mtp_sampling& p) { return (p.temperature <= 0.f || p.top_k == 1) && p.rep_penalty == 1.f; }

mtp_status check_params(const mtp_sampling* hp, int rows) {
  if (!hp) return MTP_ERR_BAD_ARG;
  for (int r = 0; r < rows; ++r) {
    const mtp_sampling& p = hp[r];
    if (!(p.temperature >= 0.f) || !(p.rep_penalty > 0.f) || !(p.top_p > 0.f && p.top_p <= 1.f) ||
        !(p.min_p >= 0.f && p.min_p < 1.f) || p.top_k < 0 || p.top_k > 1024 || (p.flags & ~MTP_SAMPLE_ARGMAX_DRAFT) != 0)
      return MTP_ERR_BAD_ARG;
  }
  return MTP_OK;
}

RowParams row_params(const mtp_sampling& p) {
  RowParams r;
  r.temperature = p.temperature;
  r.rep_penalty = p.rep_penalty;
  r.top_p = p.top_p;
  r.min_p = p.min_p;
  r.top_k = p.top_k;
  r.greedy = (p.temperature <= 0.f || p.top_k == 1) ? 1 : 0;
  r.argmax_draft = (p.flags & MTP_SAMPLE_ARGMAX_DRAFT) && !r.greedy ? 1 : 0;
  return r;
}

// The parameters the draft step samples with: an argmax-drafted row drafts
// greedily (after its repetition penalty); the verify keeps the row's own.
mtp_sampling draft_params(const mtp_sampling& p) {
  mtp_sampling d = p;
  if (p.flags & MTP_SAMPLE_ARGMAX_DRAFT) d.temperature = 0.f;
  d.flags = 0;
  return d;
}

// Items of one head call. Head items (one per row, the row's newest pair)
// come first so that per-row activations stay contiguous.
struct Items {
  int n = 0, n_head = 0;
  std::vector<int> row, slot, tok_idx, head_of_row;
  std::vector<long long> hid_off;
};

// fc -> input norm -> q/k/v -> q/k norm + RoPE + KV append for every item;
// q is kept for head items.
mtp_status run_front(mtp_handle* h, const Items& it, const int32_t* tok, const void* hid, int hid_dt,
                     bool need_q, cudaStream_t s, int pk_fc, int pk_kv) {
  const mtp_config& c = h->cfg;
  const int H = c.hidden, qw = c.n_q * c.head_dim, kw = c.n_kv * c.head_dim;
  const long long ldq = qw + 2 * kw;
  {
    ProfScope ps(h, s, pk_fc);
    GemvJob j;
    std::memset(&j, 0, sizeof(j));
    j.w[0] = h->w[T_FC];
    j.seg_end[0] = H; j.seg_end[1] = H; j.seg_end[2] = H;
    j.N = H; j.K = 2 * H; j.pro = PRO_DUAL; j.epi = EPI_STORE;
    j.nw = h->nrm[T_PRE_E]; j.nw2 = h->nrm[T_PRE_H];
    j.y = h->h0; j.ldy = H;
    j.tok = tok; j.tok_idx = it.tok_idx.data();
    j.hid = hid; j.hid_off = it.hid_off.data(); j.hid_dt = hid_dt;
    run_gemv(h, j, it.n, s);
  }
  {
    ProfScope ps(h, s, pk_kv);
    GemvJob j;
    std::memset(&j, 0, sizeof(j));
    if (need_q) {
      j.w[0] = h->w[T_Q]; j.w[1] = h->w[T_K]; j.w[2] = h->w[T_V];
        j.seg_end[0] = qw; j.seg_end[1] = qw + kw; j.seg_end[2] = qw + 2 * kw;
      j.N = qw + 2 * kw;
      j.y = h->qkv;
    } else {
      j.w[0] = h->w[T_K]; j.w[1] = h->w[T_V]; j.w[2] = h->w[T_V];
        j.seg_end[0] = kw; j.seg_end[1] = 2 * kw; j.seg_end[2] = 2 * kw;
      j.N = 2 * kw;
      j.y = h->qkv + qw;
    }
    j.ldy = ldq;
    j.K = H; j.pro = PRO_NORM; j.epi = EPI_STORE;
    j.x = h->h0; j.ldx = H; j.nw = h->nrm[T_IN];
    run_gemv(h, j, it.n, s);
  }
  {
    ProfScope ps(h, s, PK_QKV_POST);
    for (int m0 = 0; m0 < it.n; m0 += kMaxItems) {
      const int mp = std::min(kMaxItems, it.n - m0);
      QkvPostArgs a;
      std::memset(&a, 0, sizeof(a));
      a.qkv = h->qkv + (size_t)m0 * ldq;
      a.ld = ldq; a.q_off = need_q ? 0 : -1; a.k_off = qw; a.v_off = qw + kw; a.nsplit = 1; a.split_stride = 0;
      a.M = mp; a.nq = c.n_q; a.nkv = c.n_kv; a.dh = c.head_dim; a.wdt = c.dtype;
      a.eps = c.eps; a.theta = c.rope_theta;
      a.wq = h->nrm[T_QN]; a.wk = h->nrm[T_KN]; a.inv_freq = h->inv_freq;
      a.q_out = h->qrot;
      a.kc = h->kv.k; a.vc = h->kv.v; a.cap = c.kv_capacity;
      for (int m = 0; m < mp; ++m) {
        a.row[m] = it.row[m0 + m];
        a.slot[m] = it.slot[m0 + m];
        a.qdst[m] = (short)((need_q && m0 + m < it.n_head) ? m0 + m : -1);
      }
      launch_qkv_post(a, s);
    }
  }
  return cuda_ok(cudaGetLastError());
}

// attention -> o_proj + residual -> post norm -> gate/up SwiGLU -> down +
// residual -> final norm -> lm_head (+ argmax) for the head items.
mtp_status run_back(mtp_handle* h, const Items& it, float* logits, long long ld_logits, int32_t* amax_out,
                    const std::vector<int>& amax_idx, cudaStream_t s, float* qzero = nullptr, long long ldqz = 0) {
  const mtp_config& c = h->cfg;
  const int H = c.hidden, qw = c.n_q * c.head_dim, I = c.inter;
  const int R = it.n_head;
  {
    ProfScope ps(h, s, PK_ATTN);
    for (int m0 = 0; m0 < R; m0 += kMaxRows) {
      AttnArgs a;
      std::memset(&a, 0, sizeof(a));
      const int mp = std::min(kMaxRows, R - m0);
      a.q = h->qrot + (size_t)m0 * qw;
      a.kc = h->kv.k; a.vc = h->kv.v; a.cap = c.kv_capacity;
      a.Mh = mp; a.nq = c.n_q; a.nkv = c.n_kv; a.dh = c.head_dim; a.wdt = c.dtype;
      a.max_chunks = h->max_chunks;
      a.scale = 1.0f / std::sqrt((float)c.head_dim);
      a.po = h->po; a.pml = h->pml; a.o = h->o + (size_t)m0 * qw; a.status = h->status;
      for (int m = 0; m < mp; ++m) {
        a.row[m] = it.row[m0 + m];
        a.slot[m] = it.slot[m0 + m];
        // every item of this call on the same row gets its K/V slot written now
        int fn = a.slot[m];
        for (int q = 0; q < it.n; ++q)
          if (it.row[q] == a.row[m]) fn = std::min(fn, it.slot[q]);
        a.first_new[m] = fn;
      }
      launch_attention(a, h->sms, s);
    }
  }
  GemvJob j;
  {
    ProfScope ps(h, s, PK_O);
    std::memset(&j, 0, sizeof(j));
    j.w[0] = h->w[T_O]; j.seg_end[0] = H; j.seg_end[1] = H; j.seg_end[2] = H;
    j.N = H; j.K = qw; j.pro = PRO_PLAIN; j.epi = EPI_RESID;
    j.x = h->o; j.ldx = qw; j.y = h->h1; j.ldy = H; j.resid = h->h0; j.ldr = H;
    run_gemv(h, j, R, s);
  }
  {
    ProfScope ps(h, s, PK_GATEUP);
    std::memset(&j, 0, sizeof(j));
    j.w[0] = h->w[T_GATE]; j.w[1] = h->w[T_UP];
    j.N = 2 * I; j.K = H; j.pro = PRO_NORM; j.epi = EPI_SWIGLU;
    j.x = h->h1; j.ldx = H; j.nw = h->nrm[T_POST]; j.y = h->mlp; j.ldy = I;
    run_gemv(h, j, R, s);
  }
  {
    ProfScope ps(h, s, PK_DOWN);
    std::memset(&j, 0, sizeof(j));
    j.w[0] = h->w[T_DOWN]; j.seg_end[0] = H; j.seg_end[1] = H; j.seg_end[2] = H;
    j.N = H; j.K = I; j.pro = PRO_PLAIN; j.epi = EPI_RESID;
    j.x = h->mlp; j.ldx = I; j.y = h->h2; j.ldy = H; j.resid = h->h1; j.ldr = H;
    run_gemv(h, j, R, s);
  }
  {
    ProfScope ps(h, s, PK_LMHEAD);
    std::memset(&j, 0, sizeof(j));
    j.w[0] = h->lm_fp8 ? static_cast<const void*>(h->lmq) : h->lm;
    j.fp8 = h->lm_fp8;
    j.wscale = h->lmq_scale;
    j.seg_end[0] = c.vocab; j.seg_end[1] = c.vocab; j.seg_end[2] = c.vocab;
    j.N = c.vocab; j.K = H; j.pro = PRO_NORM; j.epi = EPI_LOGITS;
    j.x = h->h2; j.ldx = H; j.nw = h->nrm[T_NORM]; j.y = logits; j.ldy = ld_logits;
    j.amax_out = amax_out; j.amax_idx = amax_out ? amax_idx.data() : nullptr;
    j.qzero = qzero; j.ldqz = ldqz;
    run_gemv(h, j, R, s);
  }
  return cuda_ok(cudaGetLastError());
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// The streaming verify takes calls with more (row, position) tasks than one
// wave of 8-CTA clusters holds (two CTAs per SM), where every sampled row cuts
// to a top-k of at most kStreamTopK below the vocabulary.
bool stream_verify_fits(int rows, int depth, int vocab, const mtp_sampling* hp) {
  const int sms = device_sm_count();
  // the streaming kernel's shared memory (with the penalty bitmap) must fit
  if (vocab > (1 << 20) || verify_stream_smem(vocab) > 226 * 1024 ||
      (long long)rows * (depth + 1) * kClusterCTAs <= 2LL * sms)
    return false;
  for (int r = 0; r < rows; ++r) {
    const RowParams rp = row_params(hp[r]);
    if (!rp.greedy && !(rp.top_k >= 1 && rp.top_k <= kStreamTopK && rp.top_k < vocab)) return false;
  }
  return true;
}

// Rows without a top-k below V (and greedy rows beside them): the flat
// transform chain over many CTAs per task. False, launching nothing, where it
// does not apply.
bool flat_rows(int rows, int depth, int vocab, int hist_w, const float* d_logits, const int32_t* d_draft,
               const float* d_q, const mtp_sampling* hp, const int32_t* d_hist, const float* d_u, int32_t* d_n_acc,
               int32_t* d_out_tok, int32_t* d_stats, int32_t* h_rec, int32_t* d_status, void* ws, size_t ws_bytes,
               cudaStream_t s) {
  FlatArgs f;
  std::memset(&f, 0, sizeof(f));
  for (int r = 0; r < rows; ++r) f.p[r] = row_params(hp[r]);
  if (!flat_fits(f.p, rows, vocab, d_logits, vocab)) return false;
  f.mode = 1; f.rows = rows; f.V = vocab; f.W = hist_w; f.depth = depth; f.tasks = rows * (depth + 1);
  f.logits = d_logits; f.ld = vocab; f.hist = d_hist; f.drafts = d_draft; f.u = d_u; f.q = const_cast<float*>(d_q);
  f.n_acc = d_n_acc; f.out_tok = d_out_tok; f.stats = d_stats; f.h_rec = h_rec; f.status = d_status;
  return launch_flat(f, ws, ws_bytes, s);
}

// Every sampled row cuts to a top-k of at most kStreamTopK and the rows fit
// the one-cluster-per-task top-k transform.
bool topk_rows(int rows, int vocab, const float* logits, const mtp_sampling* hp) {
  RowParams rp[kMaxRows];
  for (int r = 0; r < rows; ++r) rp[r] = row_params(hp[r]);
  return topk_fits(rp, rows, vocab, logits, vocab);
}

// K splits so that (M tiles) x (N tiles) x splits fills at most one wave.
int tc_splits(int mtiles, int ntiles, int ktiles, int sms, int max_splits) {
  int best = 1;
  for (int k = 1; k <= max_splits; ++k)
    if (mtiles * ntiles * k <= sms && ktiles / k >= 4) best = k;
  return best;
}

// Flush of mp pairs on tcgen05: x -> fc -> input norm -> k/v -> k_norm + RoPE + store.
mtp_status flush_tensor_cores(mtp_handle* h, const Items& all, int m0, int mp, const int32_t* d_tok,
                              const void* d_hid, int hid_dtype, cudaStream_t s) {
  const mtp_config& c = h->cfg;
  const int H = c.hidden, kw = c.n_kv * c.head_dim;
  {
    ProfScope ps(h, s, PK_FLUSH_FC);
    FlushXArgs x;
    std::memset(&x, 0, sizeof(x));
    x.E = h->embed; x.wdt = c.dtype; x.H = H; x.vocab = c.vocab;
    x.tok = d_tok; x.hid = d_hid; x.hid_dt = hid_dtype;
    x.nw_e = h->nrm[T_PRE_E]; x.nw_h = h->nrm[T_PRE_H]; x.eps = c.eps;
    x.x = h->xb; x.status = h->status;
    for (int m = 0; m < mp; ++m) {
      x.tok_idx[m] = all.tok_idx[m0 + m];
      x.hid_item[m] = (int)(all.hid_off[m0 + m] / H);
    }
    launch_flush_x(x, mp, s);
    // 128 x 160 tiles measured fastest on the 256-pair flush (the 256-row
    // variants hold fewer pipeline stages and expose more TMA latency)
    const int mh = 1;
    const int bn = H % 160 == 0 ? 160 : 128;
    const int ks = tc_splits((mp + 128 * mh - 1) / (128 * mh), H / bn, 2 * H / 64, h->sms, 8);
    // the k/v weights of the next contraction go to L2 while fc streams its own
    const void* pf[2] = {h->w[T_K], h->w[T_V]};
    const long long pfb[2] = {2LL * kw * H, 2LL * kw * H};
    if (!launch_tc_gemm(h->xb, mp, 2 * H, h->w[T_FC], H, nullptr, H, bn, ks, h->tcpart, h->status, s, mh, pf, pfb))
      return MTP_ERR_CUDA;
    launch_flush_norm(h->tcpart, ks, (long long)mp * H, mp, H, h->nrm[T_IN], c.eps, h->bb, s);
  }
  {
    ProfScope ps(h, s, PK_FLUSH_KV);
    const int mh = 1;
    const int ks = tc_splits((mp + 128 * mh - 1) / (128 * mh), 2 * kw / 128, H / 64, h->sms, 8);
    if (!launch_tc_gemm(h->bb, mp, H, h->w[T_K], kw, h->w[T_V], 2 * kw, 128, ks, h->tcpart, h->status, s, mh))
      return MTP_ERR_CUDA;
    QkvPostArgs a;
    std::memset(&a, 0, sizeof(a));
    a.qkv = h->tcpart; a.ld = 2 * kw; a.q_off = -1; a.k_off = 0; a.v_off = kw;
    a.nsplit = ks; a.split_stride = (long long)mp * 2 * kw;
    a.M = mp; a.nq = c.n_q; a.nkv = c.n_kv; a.dh = c.head_dim; a.wdt = c.dtype;
    a.eps = c.eps; a.theta = c.rope_theta;
    a.wq = h->nrm[T_QN]; a.wk = h->nrm[T_KN]; a.q_out = h->qrot; a.inv_freq = h->inv_freq;
    a.kc = h->kv.k; a.vc = h->kv.v; a.cap = c.kv_capacity;
    for (int m = 0; m < mp; ++m) {
      a.row[m] = all.row[m0 + m];
      a.slot[m] = all.slot[m0 + m];
      a.qdst[m] = -1;
    }
    launch_qkv_post(a, s);
  }
  return cuda_ok(cudaGetLastError());
}

}  // namespace

extern "C" {

int32_t mtp_default_block_size(const mtp_config* cfg) { return cfg ? cfg->mtp_layers + 2 : -1; }

mtp_status mtp_set_draft_head(mtp_t h, mtp_stream stream, int32_t format) {
  if (!h || (format != MTP_HEAD_BF16 && format != MTP_HEAD_FP8)) return MTP_ERR_BAD_ARG;
  const mtp_config& c = h->cfg;
  if (format == MTP_HEAD_FP8) {
    if (c.dtype != MTP_DTYPE_BF16 || c.hidden % 16 != 0) return MTP_ERR_CONFIG_BOUNDS;
    mtp_status st = MTP_OK;
    if (!h->lmq) st = alloc(h, &h->lmq, (size_t)c.vocab * c.hidden);
    if (st == MTP_OK && !h->lmq_scale) st = alloc(h, &h->lmq_scale, (size_t)c.vocab);
    if (st != MTP_OK) return st;
    launch_quant_e4m3(static_cast<const uint16_t*>(h->lm), c.vocab, c.hidden, h->lmq, h->lmq_scale,
                      reinterpret_cast<cudaStream_t>(stream));
  }
  h->lm_fp8 = format == MTP_HEAD_FP8;
  return cuda_ok(cudaGetLastError());
}

const char* mtp_status_str(mtp_status s) {
  switch (s) {
    case MTP_OK: return "ok";
    case MTP_ERR_UNSUPPORTED_ARCH: return "unsupported draft architecture";
    case MTP_ERR_MISSING_TENSOR: return "missing head tensor";
    case MTP_ERR_DUP_TENSOR: return "duplicate head tensor";
    case MTP_ERR_UNKNOWN_TENSOR: return "unknown head tensor";
    case MTP_ERR_SHAPE: return "tensor shape or dtype mismatch";
    case MTP_ERR_CONFIG_BOUNDS: return "config scalar out of bounds";
    case MTP_ERR_NOT_BOUND: return "drafter not bound to a target embedding";
    case MTP_ERR_KV_CAPACITY: return "draft KV capacity exceeded";
    case MTP_ERR_BAD_ARG: return "bad argument";
    case MTP_ERR_NONFINITE: return "non-finite logits";
    case MTP_ERR_TIMEOUT: return "timeout";
    case MTP_ERR_CUDA: return "CUDA error";
    case MTP_ERR_LAYOUT: return "mixed raw-HF and split tensor layouts";
  }
  return "unknown status";
}

mtp_status mtp_load(const mtp_config* cfg, const mtp_tensor* tensors, int32_t n_tensors, const void* d_embed,
                    const void* d_lm_head, mtp_kv kv, const int32_t* h_len, mtp_stream stream, mtp_t* out) {
  if (!out) return MTP_ERR_BAD_ARG;
  *out = nullptr;
  if (!cfg || !tensors || n_tensors < 0) return MTP_ERR_BAD_ARG;
  const mtp_config& c = *cfg;
  if (!c.architecture || std::strcmp(c.architecture, "qwen3_5_mtp") != 0) return MTP_ERR_UNSUPPORTED_ARCH;
  // config scalar bounds
  const bool dims_ok = c.hidden >= 256 && c.hidden <= 16384 && c.hidden % 256 == 0 && c.n_q >= 1 &&
                       c.n_kv >= 1 && c.n_q % c.n_kv == 0 && c.n_q / c.n_kv <= 8 && c.n_q <= 128 &&
                       (c.head_dim == 64 || c.head_dim == 128 || c.head_dim == 256) && c.inter >= 256 &&
                       c.inter % 256 == 0 && c.inter <= 65536 && c.vocab >= 64 && c.vocab % 64 == 0 &&
                       c.vocab <= (1 << 20) && c.mtp_layers == 1 && c.max_rows >= 1 && c.max_rows <= kMaxRows &&
                       c.kv_capacity >= 64 && c.kv_capacity % 64 == 0 && c.kv_capacity <= (1 << 20) &&
                       c.max_depth >= 1 && c.max_depth <= 16 && c.eps > 0.f && c.eps < 1.f &&
                       c.rope_theta > 1.f && (c.dtype == MTP_DTYPE_F32 || c.dtype == MTP_DTYPE_BF16) &&
                       ((c.n_q * c.head_dim) % 256 == 0);
  if (!dims_ok) return MTP_ERR_CONFIG_BOUNDS;
  if (!d_embed) return MTP_ERR_NOT_BOUND;
  if (!kv.k || !kv.v || !kv.len) return MTP_ERR_BAD_ARG;

  // tensor table: layout, inventory, duplicates, shapes
  int raw = -1;
  const void* ptr[T_COUNT] = {};
  bool seen[T_COUNT] = {};
  for (int i = 0; i < n_tensors; ++i) {
    if (!tensors[i].name) return MTP_ERR_BAD_ARG;
    std::string nm = tensors[i].name;
    const int is_raw = nm.rfind("mtp.", 0) == 0 ? 1 : 0;
    if (raw < 0) raw = is_raw;
    if (raw != is_raw) return MTP_ERR_LAYOUT;
    const std::string base = is_raw ? nm.substr(4) : nm;
    int id = -1;
    for (int t = 0; t < T_COUNT; ++t)
      if (base == kNames[t]) id = t;
    if (id < 0) return MTP_ERR_UNKNOWN_TENSOR;
    if (seen[id]) return MTP_ERR_DUP_TENSOR;
    seen[id] = true;
  }
  for (int t = 0; t < T_COUNT; ++t)
    if (!seen[t]) return MTP_ERR_MISSING_TENSOR;
  const int H = c.hidden, qw = c.n_q * c.head_dim, kw = c.n_kv * c.head_dim, I = c.inter, dh = c.head_dim;
  const long long want[T_COUNT][2] = {{H, 2 * H}, {H, 0},  {H, 0},  {H, 0},  {H, 0},  {H, 0},  {I, H}, {I, H},
                                      {H, I},     {qw, H}, {kw, H}, {kw, H}, {H, qw}, {dh, 0}, {dh, 0}};
  bool shifted[T_COUNT] = {};
  for (int i = 0; i < n_tensors; ++i) {
    const mtp_tensor& t = tensors[i];
    std::string nm = t.name;
    const std::string base = raw ? nm.substr(4) : nm;
    int id = 0;
    for (int k = 0; k < T_COUNT; ++k)
      if (base == kNames[k]) id = k;
    const bool vec = want[id][1] == 0;
    if (!t.data || t.dtype != c.dtype || t.ndim != (vec ? 1 : 2) || t.shape[0] != want[id][0] ||
        (!vec && t.shape[1] != want[id][1]))
      return MTP_ERR_SHAPE;
    ptr[id] = t.data;
    if (raw)
      for (auto suf : kShiftSuffixes)
        if (ends_with(nm, suf)) shifted[id] = true;
  }

  mtp_handle* h = new mtp_handle();
  h->cfg = c;
  h->arch = c.architecture;
  h->cfg.architecture = h->arch.c_str();
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev);
  if (h->sms <= 0) h->sms = 152;
  for (int t = 0; t < T_COUNT; ++t) h->w[t] = ptr[t];
  h->embed = d_embed;
  h->lm = d_lm_head ? d_lm_head : d_embed;
  h->kv = kv;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  mtp_status st = MTP_OK;
  const int R = c.max_rows;
  // norm copies (fp32, shifted once for the raw-HF layout)
  const int norm_ids[7] = {T_NORM, T_PRE_E, T_PRE_H, T_IN, T_POST, T_QN, T_KN};
  size_t norm_total = 0;
  for (int id : norm_ids) norm_total += want[id][0];
  st = alloc(h, &h->norms, norm_total);
  size_t off = 0;
  for (int id : norm_ids) {
    if (st != MTP_OK) break;
    h->nrm[id] = h->norms + off;
    launch_norm_copy(ptr[id], c.dtype, (int)want[id][0], shifted[id] ? 1.0f : 0.0f, h->nrm[id], s);
    off += want[id][0];
  }
  // scratch
  h->max_chunks = (c.kv_capacity + kAttnChunk - 1) / kAttnChunk;
  if (st == MTP_OK) st = alloc(h, &h->h0, (size_t)kMaxItems * H);
  if (st == MTP_OK) st = alloc(h, &h->qkv, (size_t)kMaxItems * (qw + 2 * kw));
  if (st == MTP_OK) st = alloc(h, &h->qrot, (size_t)R * qw);
  if (st == MTP_OK) st = alloc(h, &h->o, (size_t)R * qw);
  if (st == MTP_OK) st = alloc(h, &h->h1, (size_t)R * H);
  if (st == MTP_OK) st = alloc(h, &h->mlp, (size_t)R * I);
  if (st == MTP_OK) st = alloc(h, &h->h2, (size_t)R * H);
  if (st == MTP_OK) st = alloc(h, &h->logits, (size_t)R * c.vocab);
  if (st == MTP_OK) st = alloc(h, &h->po, (size_t)std::min(R, kMaxRows) * c.n_q * h->max_chunks * dh);
  if (st == MTP_OK) st = alloc(h, &h->pml, (size_t)std::min(R, kMaxRows) * c.n_q * h->max_chunks * 2);
  // split-K partials and counters: worst case over every GEMV shape and width
  size_t part = 0;
  int groups = 0, smax = 1;
  const int shapes[7][2] = {{H, 2 * H}, {qw + 2 * kw, H}, {2 * kw, H}, {H, qw}, {2 * I, H}, {H, I}, {c.vocab, H}};
  for (int mt : {1, 2, 4, 8}) {
    for (auto& sh : shapes) {
      GemvPlan pl = plan_gemv(sh[0], sh[1], mt, h->sms);
      if (pl.S > 1) part = std::max(part, (size_t)pl.S * pl.mt * sh[0]);
      groups = std::max(groups, pl.ngroups);
      smax = std::max(smax, pl.S);
    }
    // the fp8 draft head (mtp_set_draft_head)
    GemvPlan pl = plan_gemv(c.vocab, H, mt, h->sms, true);
    if (pl.S > 1) part = std::max(part, (size_t)pl.S * pl.mt * c.vocab);
    groups = std::max(groups, pl.ngroups);
    smax = std::max(smax, pl.S);
  }
  h->part_floats = part;
  h->lm_groups_max = c.vocab / gemv_rows_per_group(8);
  h->lm_groups_max = std::max(h->lm_groups_max, c.vocab / gemv_rows_per_group(1));
  h->counters_n = groups;
  if (st == MTP_OK) st = alloc(h, &h->part, part);
  if (st == MTP_OK) st = alloc(h, &h->ssq, (size_t)smax * 8);
  if (c.dtype == MTP_DTYPE_BF16) {
    if (st == MTP_OK) st = alloc(h, &h->xb, (size_t)kMaxItems * 2 * H);
    if (st == MTP_OK) st = alloc(h, &h->bb, (size_t)kMaxItems * H);
    if (st == MTP_OK) st = alloc(h, &h->tcpart, (size_t)kMaxItems * std::max(8 * H, 8 * 2 * kw));
    // tensor-core GEMV: hi/lo activations [2 * kTcGemvMaxItems][K] and the
    // split partials of the widest shape
    const int kmax = std::max(std::max(2 * H, I), qw);
    size_t tvp = 0;
    for (auto& sh : shapes)
      for (int NI : {16, 32, 64, 128}) {
        const int ks = tcv_splits((sh[0] + 127) / 128, sh[1] / 64, h->sms * tc_gemv_blocks_per_sm(NI));
        tvp = std::max(tvp, (size_t)ks * kTcGemvMaxItems * sh[0]);
      }
    if (st == MTP_OK) st = alloc(h, &h->x2, (size_t)2 * kTcGemvMaxItems * kmax);
    if (st == MTP_OK) st = alloc(h, &h->tvpart, tvp);
    h->tc_gemv = st == MTP_OK;
  }
  // per-group argmax pairs: 8 items of the CUDA-core head, or up to
  // kTcGemvMaxItems items of the tensor-core head per 128-row tile
  const size_t gslots = std::max((size_t)8 * h->lm_groups_max, (size_t)kTcGemvMaxItems * ((c.vocab + 127) / 128));
  if (st == MTP_OK) st = alloc(h, &h->gmax, gslots);
  if (st == MTP_OK) st = alloc(h, &h->gidx, gslots);
  if (st == MTP_OK) st = alloc(h, &h->counters, (size_t)groups);
  if (st == MTP_OK) st = alloc(h, &h->done, 1);
  if (st == MTP_OK) st = alloc(h, &h->walk, 1);
  if (st == MTP_OK) st = alloc(h, &h->status, 1);
  h->flat_ws_bytes = flat_workspace_bytes(R, R);
  if (st == MTP_OK) st = alloc(h, &h->flat_ws, h->flat_ws_bytes);
  if (st == MTP_OK) st = alloc(h, &h->inv_freq, (size_t)dh / 2);
  if (st == MTP_OK) {
    std::vector<double> f(dh / 2);
    for (int i = 0; i < dh / 2; ++i) f[i] = std::pow((double)c.rope_theta, -2.0 * i / (double)dh);
    st = cuda_ok(cudaMemcpy(h->inv_freq, f.data(), sizeof(double) * f.size(), cudaMemcpyHostToDevice));
  }
  if (st == MTP_OK) st = cuda_ok(cudaMemsetAsync(h->counters, 0, sizeof(int) * groups, s));
  if (st == MTP_OK) st = cuda_ok(cudaMemsetAsync(h->done, 0, sizeof(int), s));
  if (st == MTP_OK) st = cuda_ok(cudaMemsetAsync(h->walk, 0, sizeof(int), s));
  if (st == MTP_OK) st = cuda_ok(cudaMemsetAsync(h->status, 0, sizeof(int32_t), s));
  h->len.assign(R, 0);
  h->keep.assign(R, -1);
  h->drafted_len.assign(R, 0);
  if (h_len)
    for (int r = 0; r < R; ++r) {
      if (h_len[r] < 0 || h_len[r] > c.kv_capacity) st = MTP_ERR_BAD_ARG;
      h->len[r] = h_len[r];
    }
  if (st == MTP_OK) launch_set_len(h->kv.len, R, h->len.data(), s);
  if (st == MTP_OK) st = cuda_ok(cudaGetLastError());
  if (st == MTP_OK) st = cuda_ok(cudaStreamSynchronize(s));
  if (st != MTP_OK) {
    free_all(h);
    delete h;
    return st;
  }
  *out = h;
  return MTP_OK;
}

mtp_status mtp_free(mtp_t h) {
  if (!h) return MTP_ERR_BAD_ARG;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
  return MTP_OK;
}

mtp_status mtp_get_lengths(mtp_t h, int32_t* h_len) {
  if (!h || !h_len) return MTP_ERR_BAD_ARG;
  for (int r = 0; r < h->cfg.max_rows; ++r) h_len[r] = h->len[r];
  return MTP_OK;
}

mtp_status mtp_set_lengths(mtp_t h, mtp_stream stream, const int32_t* h_len) {
  if (!h || !h_len) return MTP_ERR_BAD_ARG;
  for (int r = 0; r < h->cfg.max_rows; ++r)
    if (h_len[r] < 0 || h_len[r] > h->cfg.kv_capacity) return MTP_ERR_BAD_ARG;
  for (int r = 0; r < h->cfg.max_rows; ++r) { h->len[r] = h_len[r]; h->keep[r] = -1; }
  launch_set_len(h->kv.len, h->cfg.max_rows, h->len.data(), reinterpret_cast<cudaStream_t>(stream));
  return cuda_ok(cudaGetLastError());
}

int32_t* mtp_device_status(mtp_t h) { return h ? h->status : nullptr; }

mtp_status mtp_flush(mtp_t h, mtp_stream stream, int32_t rows, const int32_t* h_pairs, int32_t pmax,
                     const int32_t* d_tok, const void* d_hid, int32_t hid_dtype) {
  if (!h || !h_pairs || rows < 1 || rows > h->cfg.max_rows || pmax < 1 || !d_tok || !d_hid ||
      (hid_dtype != MTP_DTYPE_F32 && hid_dtype != MTP_DTYPE_BF16))
    return MTP_ERR_BAD_ARG;
  const mtp_config& c = h->cfg;
  for (int r = 0; r < rows; ++r) {
    if (h_pairs[r] < 0 || h_pairs[r] > pmax) return MTP_ERR_BAD_ARG;
    if ((long long)h->len[r] + h_pairs[r] > c.kv_capacity) return MTP_ERR_KV_CAPACITY;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Items all;
  for (int r = 0; r < rows; ++r)
    for (int j = 0; j < h_pairs[r]; ++j) {
      all.row.push_back(r);
      all.slot.push_back(h->len[r] + j);
      all.tok_idx.push_back(r * pmax + j);
      all.hid_off.push_back(((long long)r * pmax + j) * c.hidden);
    }
  all.n = (int)all.row.size();
  if (c.dtype == MTP_DTYPE_BF16 && all.n >= kTcFlushMinItems) {
    for (int m0 = 0; m0 < all.n; m0 += kMaxItems) {
      const int mp = std::min(kMaxItems, all.n - m0);
      mtp_status st = flush_tensor_cores(h, all, m0, mp, d_tok, d_hid, hid_dtype, s);
      if (st != MTP_OK) return st;
    }
  } else
  for (int m0 = 0; m0 < all.n; m0 += kMaxItems) {
    Items it;
    const int mp = std::min(kMaxItems, all.n - m0);
    it.n = mp;
    it.n_head = 0;
    it.row.assign(all.row.begin() + m0, all.row.begin() + m0 + mp);
    it.slot.assign(all.slot.begin() + m0, all.slot.begin() + m0 + mp);
    it.tok_idx.assign(all.tok_idx.begin() + m0, all.tok_idx.begin() + m0 + mp);
    it.hid_off.assign(all.hid_off.begin() + m0, all.hid_off.begin() + m0 + mp);
    mtp_status st = run_front(h, it, d_tok, d_hid, hid_dtype, false, s, PK_FLUSH_FC, PK_FLUSH_KV);
    if (st != MTP_OK) return st;
  }
  for (int r = 0; r < rows; ++r) { h->len[r] += h_pairs[r]; h->keep[r] = -1; }
  launch_set_len(h->kv.len, c.max_rows, h->len.data(), s);
  return cuda_ok(cudaGetLastError());
}

mtp_status mtp_draft(mtp_t h, mtp_stream stream, int32_t rows, int32_t depth, const int32_t* h_pairs,
                     int32_t pmax, const int32_t* d_tok, const void* d_hid, int32_t hid_dtype,
                     const mtp_sampling* h_params, const int32_t* d_hist, int32_t hist_w, const float* d_u,
                     int32_t* d_draft, float* d_q, float* d_logits, float* d_hidden) {
  if (!h || rows < 1 || rows > h->cfg.max_rows || depth < 1 || depth > h->cfg.max_depth || !h_pairs ||
      pmax < 1 || !d_tok || !d_hid || !d_draft || hist_w < 0 || hist_w > 128 || (hist_w > 0 && !d_hist) ||
      (hid_dtype != MTP_DTYPE_F32 && hid_dtype != MTP_DTYPE_BF16))
    return MTP_ERR_BAD_ARG;
  mtp_status st = check_params(h_params, rows);
  if (st != MTP_OK) return st;
  const mtp_config& c = h->cfg;
  bool all_fast = true, any_sampled = false;
  for (int r = 0; r < rows; ++r) {
    const mtp_sampling dp = draft_params(h_params[r]);
    all_fast &= fast_greedy(dp);
    any_sampled |= !row_params(dp).greedy;
  }
  if (any_sampled && (!d_q || !d_u)) return MTP_ERR_BAD_ARG;
  int total = 0;
  for (int r = 0; r < rows; ++r) {
    if (h_pairs[r] < 1 || h_pairs[r] > pmax) return MTP_ERR_BAD_ARG;
    if ((long long)h->len[r] + h_pairs[r] + depth - 1 > c.kv_capacity) return MTP_ERR_KV_CAPACITY;
    total += h_pairs[r];
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int H = c.hidden, V = c.vocab;

  // step-1 items: head items first, then the pending pairs
  Items it1;
  it1.n_head = rows;
  for (int r = 0; r < rows; ++r) {
    const int j = h_pairs[r] - 1;
    it1.row.push_back(r);
    it1.slot.push_back(h->len[r] + j);
    it1.tok_idx.push_back(r * pmax + j);
    it1.hid_off.push_back(((long long)r * pmax + j) * H);
  }
  for (int r = 0; r < rows; ++r)
    for (int j = 0; j + 1 < h_pairs[r]; ++j) {
      it1.row.push_back(r);
      it1.slot.push_back(h->len[r] + j);
      it1.tok_idx.push_back(r * pmax + j);
      it1.hid_off.push_back(((long long)r * pmax + j) * H);
    }
  it1.n = (int)it1.row.size();
  if (it1.n > kMaxItems) return MTP_ERR_BAD_ARG;

  std::vector<int> amax_idx(rows);
  SampleArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  sa.mode = 0; sa.rows = rows; sa.V = V; sa.W = hist_w; sa.depth = depth;
  sa.hist = d_hist; sa.drafts = d_draft; sa.u = d_u; sa.q = d_q; sa.draft_out = d_draft;
  sa.status = h->status;
  sa.flat_ws = h->flat_ws; sa.flat_ws_bytes = h->flat_ws_bytes;
  for (int r = 0; r < rows; ++r) sa.p[r] = row_params(draft_params(h_params[r]));
  // with the top-k sampler, each step's logits epilogue clears that step's q
  // rows and the sampler writes their kept entries only
  if (!all_fast && d_q && topk_fits(sa.p, rows, V, d_logits ? d_logits : h->logits, d_logits ? (long long)depth * V : V))
    sa.q_zeroed = 1;

  for (int k = 1; k <= depth; ++k) {
    Items itk;
    const Items* it = &it1;
    const int32_t* tok = d_tok;
    const void* hid = d_hid;
    int hdt = hid_dtype;
    if (k > 1) {
      itk.n = rows;
      itk.n_head = rows;
      for (int r = 0; r < rows; ++r) {
        itk.row.push_back(r);
        itk.slot.push_back(h->len[r] + h_pairs[r] + k - 2);
        itk.tok_idx.push_back(r * depth + (k - 2));
        itk.hid_off.push_back((long long)r * H);
      }
      it = &itk;
      tok = d_draft;
      hid = h->h2;
      hdt = MTP_DTYPE_F32;
    }
    st = run_front(h, *it, tok, hid, hdt, true, s, PK_FC, PK_QKV);
    if (st != MTP_OK) return st;
    float* lg = d_logits ? d_logits + (size_t)(k - 1) * V : h->logits;
    const long long ldl = d_logits ? (long long)depth * V : V;
    for (int r = 0; r < rows; ++r) amax_idx[r] = r * depth + (k - 1);
    st = run_back(h, *it, lg, ldl, all_fast ? d_draft : nullptr, amax_idx, s,
                  sa.q_zeroed ? d_q + (size_t)(k - 1) * V : nullptr, (long long)depth * V);
    if (st != MTP_OK) return st;
    if (!all_fast) {
      ProfScope ps(h, s, PK_SAMPLE);
      sa.pos = k - 1;
      sa.logits = lg;
      sa.ld = ldl;
      launch_sample(sa, s);
    }
    if (d_hidden) {
      st = cuda_ok(cudaMemcpy2DAsync(d_hidden + (size_t)(k - 1) * H, sizeof(float) * depth * H, h->h2,
                                     sizeof(float) * H, sizeof(float) * H, rows, cudaMemcpyDeviceToDevice, s));
      if (st != MTP_OK) return st;
    }
  }
  for (int r = 0; r < rows; ++r) {
    h->keep[r] = h->len[r] + h_pairs[r];
    h->len[r] += h_pairs[r] + depth - 1;
  }
  for (int r = rows; r < c.max_rows; ++r) h->keep[r] = -1;
  launch_set_len(h->kv.len, c.max_rows, h->len.data(), s);
  return cuda_ok(cudaGetLastError());
}

size_t spec_verify_workspace_bytes(int32_t rows, int32_t depth, int32_t vocab) {
  (void)vocab;
  if (rows < 1 || depth < 1) return 0;
  const size_t tasks = (size_t)rows * (depth + 1);
  // descriptors, then (streaming path) accept flags and kept lists; or (the
  // greedy stream over many rows) one 64-bit key per range and segment
  const size_t lists = align256(sizeof(TDesc) * tasks) + align256(sizeof(int32_t) * tasks) +
                       2 * align256(sizeof(int32_t) * tasks * kStreamTopK);
  return std::max({lists, align256(sizeof(unsigned long long) * (tasks + kFlatMaxCTAs)),
                   flat_workspace_bytes(rows, (int)tasks)});
}

}  // extern "C"

namespace mtp {

mtp_status spec_verify_impl(mtp_stream stream, int32_t rows, int32_t depth, int32_t vocab, const float* d_logits,
                            const int32_t* d_draft, const float* d_q, const mtp_sampling* h_params,
                            const int32_t* d_hist, int32_t hist_w, const float* d_u, int32_t* d_n_acc,
                            int32_t* d_out_tok, int32_t* d_stats, int32_t* h_out, int32_t* d_status,
                            void* d_workspace, size_t workspace_bytes, bool allow_stream) {
  if (rows < 1 || rows > kMaxRows || depth < 1 || depth > 16 || vocab < 1 || !d_logits || !d_draft ||
      hist_w < 0 || hist_w > 128 || (hist_w > 0 && !d_hist) || !d_u || !d_n_acc || !d_out_tok || !d_workspace)
    return MTP_ERR_BAD_ARG;
  mtp_status st = check_params(h_params, rows);
  if (st != MTP_OK) return st;
  bool dense_q = false;  // some row's draft distribution is a dense q (sampled, not argmax-drafted)
  for (int r = 0; r < rows; ++r) {
    const RowParams rp = row_params(h_params[r]);
    dense_q |= !rp.greedy && !rp.argmax_draft;
  }
  if (dense_q && !d_q) return MTP_ERR_BAD_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the host record: written by the verify kernel itself when the device can
  // address the caller's page-locked buffer, else copied after it
  int32_t* h_rec = nullptr;
  if (h_out) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, h_out) == cudaSuccess && at.type == cudaMemoryTypeHost && at.devicePointer)
      h_rec = static_cast<int32_t*>(at.devicePointer);
    cudaGetLastError();
  }
  bool all_fast_greedy = true;
  for (int r = 0; r < rows; ++r) all_fast_greedy &= fast_greedy(h_params[r]);
  if (all_fast_greedy) {
    VerifyArgs va;
    std::memset(&va, 0, sizeof(va));
    va.rows = rows; va.V = vocab; va.depth = depth;
    va.logits = d_logits; va.drafts = d_draft; va.n_acc = d_n_acc; va.out_tok = d_out_tok; va.stats = d_stats;
    va.h_rec = h_rec; va.status = d_status;
    // one balanced stream over all target rows (measured faster than one
    // cluster per row from a single row on: 10.3 against 16.4 us per round at
    // batch 1, V = 152064); the single cluster launch takes what it cannot
    // (rows not 16-byte aligned, V % 4 != 0)
    if (!launch_verify_greedy_flat(va, d_workspace, workspace_bytes, s)) launch_verify_greedy(va, s);
  } else if (allow_stream && (stream_verify_fits(rows, depth, vocab, h_params) || topk_rows(rows, vocab, d_logits, h_params))) {
    // rows that cut to a small top-k: many tasks stream (one CTA per task),
    // fewer take one cluster per task; both write the descriptors, accept
    // flags and kept lists that the per-row finish draws from
    const bool streaming = stream_verify_fits(rows, depth, vocab, h_params);
    const size_t tasks = (size_t)rows * (depth + 1);
    uint8_t* w = static_cast<uint8_t*>(d_workspace);
    VerifyArgs va;
    std::memset(&va, 0, sizeof(va));
    va.rows = rows; va.V = vocab; va.W = hist_w; va.depth = depth;
    va.logits = d_logits; va.drafts = d_draft; va.q = d_q; va.hist = d_hist; va.u = d_u;
    va.wdesc = reinterpret_cast<TDesc*>(w);
    va.desc = va.wdesc;
    w += align256(sizeof(TDesc) * tasks);
    va.acc = reinterpret_cast<int32_t*>(w);
    w += align256(sizeof(int32_t) * tasks);
    va.kid = reinterpret_cast<int32_t*>(w);
    w += align256(sizeof(int32_t) * tasks * kStreamTopK);
    va.kkey = reinterpret_cast<uint32_t*>(w);
    va.n_acc = d_n_acc; va.out_tok = d_out_tok; va.stats = d_stats; va.h_rec = h_rec; va.status = d_status;
    for (int r = 0; r < rows; ++r) va.p[r] = row_params(h_params[r]);
    if (streaming) {
      va.stall_stage = g_stall_stage.exchange(-1);
      va.wait_limit = va.stall_stage >= 0 ? g_stall_polls.load() : 0u;
      launch_verify_stream(va, s);
    } else {
      TopkArgs t;
      std::memset(&t, 0, sizeof(t));
      t.mode = 1; t.rows = rows; t.V = vocab; t.W = hist_w; t.depth = depth;
      t.logits = d_logits; t.ld = vocab; t.hist = d_hist; t.drafts = d_draft; t.u = d_u;
      t.q = const_cast<float*>(d_q);
      t.wdesc = va.wdesc; t.acc = va.acc; t.kid = va.kid; t.kkey = va.kkey; t.status = d_status;
      for (int r = 0; r < rows; ++r) t.p[r] = va.p[r];
      launch_topk(t, s);
      launch_verify_finish(va, s);
    }
  } else if (!(allow_stream && flat_rows(rows, depth, vocab, hist_w, d_logits, d_draft, d_q, h_params, d_hist, d_u,
                                         d_n_acc, d_out_tok, d_stats, h_rec, d_status, d_workspace, workspace_bytes,
                                         s))) {
    // every other mix: one 8-CTA cluster per task for the descriptors, then
    // one per row for the accept chain and the draw
    TDesc* desc = static_cast<TDesc*>(d_workspace);
    SampleArgs sa;
    std::memset(&sa, 0, sizeof(sa));
    sa.mode = 1; sa.rows = rows; sa.V = vocab; sa.W = hist_w; sa.depth = depth;
    sa.logits = d_logits; sa.hist = d_hist; sa.drafts = d_draft; sa.desc = desc; sa.status = d_status;
    for (int r = 0; r < rows; ++r) sa.p[r] = row_params(h_params[r]);
    launch_sample(sa, s);
    VerifyArgs va;
    std::memset(&va, 0, sizeof(va));
    va.rows = rows; va.V = vocab; va.W = hist_w; va.depth = depth;
    va.logits = d_logits; va.drafts = d_draft; va.q = d_q; va.hist = d_hist; va.u = d_u; va.desc = desc;
    va.n_acc = d_n_acc; va.out_tok = d_out_tok; va.stats = d_stats; va.h_rec = h_rec; va.status = d_status;
    for (int r = 0; r < rows; ++r) va.p[r] = sa.p[r];
    launch_verify(va, s);
  }
  st = cuda_ok(cudaGetLastError());
  if (st != MTP_OK) return st;
  if (h_out && !h_rec) {
    const size_t pitch = sizeof(int32_t) * (depth + 2);
    st = cuda_ok(cudaMemcpy2DAsync(h_out, pitch, d_n_acc, sizeof(int32_t), sizeof(int32_t), rows,
                                   cudaMemcpyDeviceToHost, s));
    if (st == MTP_OK)
      st = cuda_ok(cudaMemcpy2DAsync(h_out + 1, pitch, d_out_tok, sizeof(int32_t) * (depth + 1),
                                     sizeof(int32_t) * (depth + 1), rows, cudaMemcpyDeviceToHost, s));
  }
  return st;
}

}  // namespace mtp

extern "C" {

mtp_status spec_verify(mtp_stream stream, int32_t rows, int32_t depth, int32_t vocab, const float* d_logits,
                       const int32_t* d_draft, const float* d_q, const mtp_sampling* h_params,
                       const int32_t* d_hist, int32_t hist_w, const float* d_u, int32_t* d_n_acc,
                       int32_t* d_out_tok, int32_t* d_stats, int32_t* h_out, int32_t* d_status,
                       void* d_workspace) {
  return mtp::spec_verify_impl(stream, rows, depth, vocab, d_logits, d_draft, d_q, h_params, d_hist, hist_w, d_u,
                               d_n_acc, d_out_tok, d_stats, h_out, d_status, d_workspace,
                               spec_verify_workspace_bytes(rows, depth, vocab), true);
}

mtp_status mtp_test_verify_stall(int32_t stage, int32_t wait_polls) {
  if (stage < 0 || wait_polls < 1) return MTP_ERR_BAD_ARG;
  g_stall_polls.store((unsigned)wait_polls);
  g_stall_stage.store(stage);
  return MTP_OK;
}

mtp_status kv_rollback(mtp_t h, mtp_stream stream, int32_t rows, const int32_t* d_n_acc, int32_t* d_target_len,
                       int32_t depth, int32_t zero_tail) {
  if (!h || rows < 1 || rows > h->cfg.max_rows || depth < 1 || (d_target_len && !d_n_acc)) return MTP_ERR_BAD_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ProfScope ps(h, s, PK_ROLLBACK);
  RollbackArgs a;
  std::memset(&a, 0, sizeof(a));
  a.len = h->kv.len; a.rows = rows; a.zero_tail = zero_tail ? 1 : 0;
  a.kc = h->kv.k; a.vc = h->kv.v; a.cap = h->cfg.kv_capacity;
  a.nkv = h->cfg.n_kv; a.dh = h->cfg.head_dim; a.esize = esize(h->cfg.dtype);
  a.n_acc = d_n_acc; a.target_len = d_target_len; a.block = depth + 1;
  for (int r = 0; r < rows; ++r) {
    a.keep[r] = h->keep[r];
    a.old_len[r] = h->len[r];
  }
  launch_rollback(a, s);
  for (int r = 0; r < rows; ++r)
    if (h->keep[r] >= 0) { h->len[r] = h->keep[r]; h->keep[r] = -1; }
  return cuda_ok(cudaGetLastError());
}

int64_t mtp_kernel_launches(void) { return (int64_t)launches_so_far(); }

mtp_status mtp_profile_enable(mtp_t h, int32_t mask) {
  if (!h) return MTP_ERR_BAD_ARG;
  h->prof = (uint32_t)mask;
  return MTP_OK;
}

int32_t mtp_profile_kinds(void) { return PK_COUNT; }

const char* mtp_profile_kind_name(int32_t kind) { return kind >= 0 && kind < PK_COUNT ? kProfNames[kind] : ""; }

mtp_status mtp_profile_read(mtp_t h, float* h_ms, int32_t* h_launches) {
  if (!h || !h_ms || !h_launches) return MTP_ERR_BAD_ARG;
  for (int k = 0; k < PK_COUNT; ++k) { h_ms[k] = 0.f; h_launches[k] = 0; }
  for (auto& r : h->recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return MTP_ERR_CUDA;
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    h_ms[r.kind] += ms;
    h_launches[r.kind] += 1;
  }
  h->recs.clear();
  h->ev_next = 0;
  return MTP_OK;
}

}  // extern "C"
