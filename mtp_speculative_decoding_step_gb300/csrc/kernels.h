// Internal launch interface between the C ABI (mtp_api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mtp.h"

namespace mtp {

// Count of kernels launched by this library (for the benchmark's launch tally).
void count_launch(int n = 1);

constexpr int kMaxItems = 256;   // pairs per head call (the pages' flush cap)
constexpr int kMaxRows = 64;
constexpr int kAttnChunk = 128;  // smallest KV slot range of a decode-attention block
constexpr int kClusterCTAs = 8;  // CTAs per sampling cluster

enum { PRO_PLAIN = 0, PRO_NORM = 1, PRO_DUAL = 2 };
enum { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3 };

// y[m][n] = sum_k W[n][k] x[m][k] over a virtual row space (several weight
// segments, or gate/up halves), batch of M <= MT items, fp32 accumulate.
struct GemvArgs {
  const void* w[3];
  int seg_end[3];
  int N, K, S, ngroups;
  int pro, epi, M, wdt;
  const float* x;
  long long ldx;
  const float* nw;
  const float* nw2;
  float eps;
  const void* E;
  int vocab;
  const int32_t* tok;
  int tok_idx[8];
  const void* hid;
  long long hid_off[8];
  int hid_dt;
  float* y;
  long long ldy;
  const float* resid;
  long long ldr;
  float* part;
  int* counters;
  float* gmax;
  int* gidx;
  int* done;
  int32_t* amax_out;
  int amax_idx[8];
  int32_t* status;
  const float* wscale;  // per-row scales of quantised weights (fp8), or null
  float* ssq;           // [S][MT] sums of squares of x per K split (deferred RMSNorm scale)
  float* qzero;         // logits epilogue: item m's draft distribution row (stride ldqz), zeroed
  long long ldqz;       // where the logits go (the sampler then writes its kept entries only)
  int* walk;            // group counter of the walking GEMV (zero between launches), or null
};
// weight dtype code of the quantised (fp8 e4m3) draft head, beside MTP_DTYPE_*
constexpr int kDtypeFp8 = 8;
// Per-row e4m3 quantisation of a bf16 [rows][cols] matrix (cols even).
void launch_quant_e4m3(const uint16_t* w, int rows, int cols, uint8_t* q, float* scale, cudaStream_t s);

// The fp8 head runs on the tensor cores (128 rows per block group) when its
// row count allows; otherwise on the CUDA cores.
inline bool gemv_fp8_mma(int N) { return N % 128 == 0; }
// rows per block group for a batch width MT
inline int gemv_rows_per_group(int mt, bool fp8_mma = false) { return fp8_mma ? 128 : 8 * (mt <= 4 ? 8 : 4); }
// K-slices of a GEMV: split `sp` of S covers [start(sp), start(sp + 1)), cut
// on 16-element boundaries (K a multiple of 16); lengths differ by at most 16.
__host__ __device__ inline int gemv_slice_start(int K, int S, int sp) {
  return (int)((long long)sp * (K / 16) / S) * 16;
}
inline int gemv_slice_max(int K, int S) { return ((K / 16 + S - 1) / S) * 16; }
void launch_gemv(int mt, const GemvArgs& a, int smem_bytes, cudaStream_t s);

// Per-item per-head q_norm / k_norm + RoPE + KV append.
struct QkvPostArgs {
  const float* qkv;      // item m's projections at qkv + m*ld (+ s*split_stride, summed over splits)
  long long ld;
  int q_off, k_off, v_off;  // column offsets; q_off < 0: no q
  int nsplit;
  long long split_stride;
  int M, nq, nkv, dh, wdt;
  float eps, theta;
  const double* inv_freq;  // [dh/2] RoPE frequencies theta^(-2i/dh)
  const float* wq;
  const float* wk;
  float* q_out;          // [n_head][qw] for items with qdst >= 0
  void* kc;
  void* vc;
  long long cap;
  int row[kMaxItems];
  int slot[kMaxItems];
  short qdst[kMaxItems];
};
void launch_qkv_post(const QkvPostArgs& a, cudaStream_t s);

// Flush on tensor cores: bf16 activations for the two contractions.
struct FlushXArgs {
  const void* E;
  int wdt, H, vocab;
  const int32_t* tok;
  const void* hid;
  int hid_dt;
  const float* nw_e;
  const float* nw_h;
  float eps;
  uint16_t* x;           // [M][2H] bf16
  int32_t* status;
  int tok_idx[kMaxItems];
  int hid_item[kMaxItems];  // hidden of item m at hid + hid_item[m] * H
};
void launch_flush_x(const FlushXArgs& a, int M, cudaStream_t s);
// b[m] = bf16(rmsnorm(sum_s part[s][m], w))
void launch_flush_norm(const float* part, int nsplit, long long split_stride, int M, int H, const float* w,
                       float eps, uint16_t* b, cudaStream_t s);
// D[split][M][N] = A[M][K] . [B0; B1]^T on tcgen05 (bf16 in, fp32 out).
// pf[2] / pf_bytes[2]: two ranges the next kernel streams (prefetched into L2
// once this kernel's own loads are issued), or null.
bool launch_tc_gemm(const void* A, int M, int K, const void* B0, int n0rows, const void* B1, int N, int bn,
                    int ksplit, float* D, int32_t* status, cudaStream_t s, int mh = 1,
                    const void* const* pf = nullptr, const long long* pf_bytes = nullptr);

// Batched GEMV on tcgen05 (bf16 weights, kTcGemvMaxItems items per pass).
constexpr int kTcGemvMaxItems = 64;

// X2[NI][K] bf16: rows m < MI hold bf16(x_m), rows MI + m hold the rounding
// residue bf16(x_m - bf16(x_m)); x_m after the prologue; items M..MI-1 zero.
struct TcxPrepArgs {
  int pro, K, M, MI;
  const float* x;
  long long ldx;
  const float* nw;
  const float* nw2;
  float eps;
  const void* E;
  int wdt, vocab;
  const int32_t* tok;
  const void* hid;
  int hid_dt;
  uint16_t* X2;
  int32_t* status;
  int tok_idx[kTcGemvMaxItems];
  long long hid_off[kTcGemvMaxItems];
};
void launch_tcx_prep(const TcxPrepArgs& a, cudaStream_t s);

// out[split][item][row] (strides ld_split, ld_item) = W[row] . x[item] over the
// virtual row space: segments w[0..nmaps) ending at seg_end, or (swiglu) 128-row
// tiles of 64 gate rows (w[0]) then the matching 64 up rows (w[1]).
struct TcGemvLaunch {
  const void* w[3];
  int rows[3];
  int nmaps;
  int seg_end[3];
  int swiglu;
  int N, K, M, NI, ksplit;
  const uint16_t* X2;
  float* out;
  long long ld_item, ld_split;
  int32_t* status;
  // one split, out = the logits: the epilogue also clears item m's row of
  // qzero (stride ldqz; or null) and leaves each tile's (max, index) per item
  // in gmax / gidx[m * tiles + tile] for launch_tcv_argmax
  int fuse_logits;
  float* qzero;
  long long ldqz;
  float* gmax;
  int* gidx;
};
bool launch_tc_gemv(const TcGemvLaunch& L, cudaStream_t s);
// CTAs of the tensor-core GEMV with NI activation columns resident per SM
// (by its shared memory)
int tc_gemv_blocks_per_sm(int NI);

// Sum the split partials (split order) and apply the epilogue; outputs
// o < nout (nout = N, or N/2 for SwiGLU).
struct TcFinishArgs {
  const float* part;
  long long ld_item, ld_split;
  int ksplit, M, epi, nout, write_y;
  float* y;
  long long ldy;
  const float* resid;
  long long ldr;
  float* gmax;
  int* gidx;
  int* done;
  int32_t* amax_out;
  int32_t* status;
  int amax_idx[kTcGemvMaxItems];
  float* qzero;         // logits: item m's draft distribution row (stride ldqz) zeroed beside them
  long long ldqz;
};
void launch_tcv_finish(const TcFinishArgs& a, cudaStream_t s);
// After a fused logits epilogue: amax_out[amax_idx[m]] = the argmax of item m
// over its a.nout tile pairs in gmax / gidx (lowest index on ties).
void launch_tcv_argmax(const TcFinishArgs& a, cudaStream_t s);

// Decode attention of the head items over slots 0..slot (split over chunks).
struct AttnArgs {
  const float* q;        // [Mh][nq*dh]
  const void* kc;
  const void* vc;
  long long cap;
  int Mh, nq, nkv, dh, wdt, max_chunks;
  int chunk;             // slots per block (a multiple of 64, >= kAttnChunk; set by the launcher)
  float scale;
  float* po;             // [Mh][nq][max_chunks][dh]
  float* pml;            // [Mh][nq][max_chunks][2]
  float* o;              // [Mh][nq*dh]
  int32_t* status;
  int row[kMaxRows];
  int slot[kMaxRows];
  // the first cache slot of item m's row that this call's k_qkv_post writes
  // (slots below it are final before the attention starts; 0: none known)
  int first_new[kMaxRows];
};
void launch_attention(const AttnArgs& a, int sms, cudaStream_t s);
// The tensor-core instance (bf16 cache, head dim 128 or 256, at most 8 query
// heads per KV head); false, with nothing launched, for any other shape.
bool launch_attention_mma(const AttnArgs& a, int sms, cudaStream_t s);
// Slots per attention block for `slots` resident blocks, and the merge of the
// blocks' partial outputs.
int attn_chunk_slots(const AttnArgs& a, long long slots);
void launch_attn_merge(const AttnArgs& a, cudaStream_t s);

// Copy a norm vector to fp32 adding `shift`.
void launch_norm_copy(const void* src, int dt, int n, float shift, float* dst, cudaStream_t s);

// Set device lengths, trim target lengths, zero dropped draft slots.
struct RollbackArgs {
  int32_t* len;
  int rows;
  int keep[kMaxRows];
  int old_len[kMaxRows];
  int zero_tail;
  void* kc;
  void* vc;
  long long cap;
  int nkv, dh, esize;
  const int32_t* n_acc;
  int32_t* target_len;
  int block;
};
void launch_rollback(const RollbackArgs& a, cudaStream_t s);
void launch_set_len(int32_t* len, int rows, const int* h_len, cudaStream_t s);

// ---------------------------------------------------------------- sampling
struct RowParams {
  float temperature, rep_penalty, top_p, min_p;
  int top_k, greedy;
  int argmax_draft;  // the draft was the argmax: q is the point mass at it
};

// Transform descriptor of one (row, position): enough to evaluate p(v) at any v.
struct TDesc {
  float m;          // max transformed logit
  float S;          // normaliser of the kept set
  uint32_t k_key;   // top-k prefix bound on the descending key
  int k_cut;        // id bound among keys equal to k_key
  uint32_t p_key;   // top-p prefix bound
  int p_cut;
  int argmax;       // argmax of the penalised logits
  int kept;         // support size
};

struct SampleArgs {
  int mode;                  // 0 = draft step, 1 = verify descriptors
  int rows, V, W, depth, pos;  // pos: draft step index k-1 (draft mode)
  const float* logits;       // draft: [rows][ld] ; verify: [rows][depth+1][V]
  long long ld;
  const int32_t* hist;       // [rows][W]
  const int32_t* drafts;     // [rows][depth]
  const float* u;            // draft: [rows][depth]
  float* q;                  // draft: [rows][depth][V]
  int32_t* draft_out;        // draft: [rows][depth]
  TDesc* desc;               // verify: [rows][depth+1]
  int32_t* status;
  int cand;                  // local candidates per CTA (set by launch_sample)
  int merge;                 // merged candidate buffer (power of two)
  void* flat_ws;             // draft: scratch of the flat transform (flat_workspace_bytes), or null
  size_t flat_ws_bytes;
  int q_zeroed;              // draft: the logits epilogue cleared this step's q rows (the top-k path writes its kept entries only)
  RowParams p[kMaxRows];
};
void launch_sample(const SampleArgs& a, cudaStream_t s);

// Flat transform of rows with a wide support (no top-k below V: top-p, min-p
// or plain temperature over the whole vocabulary) as a chain of short kernels
// that spread every (row, position) over many CTAs: statistics (penalised
// argmax and minimum), a weighted value histogram, the gather of the top-p
// crossing bin (its last CTA resolves the descriptor), then the draw's sums
// (their last CTA draws: q and the draft token of a draft step; the accept
// chain and the correction or bonus token of a verify).
struct FlatArgs {
  int mode;                  // 0 draft step, 1 verify
  int rows, V, W, depth, pos, tasks;
  int P;                     // parts per task of the argmax/minimum pass (every task)
  int Ps;                    // parts per task of the histogram and gather passes (sampled tasks)
  int P2;                    // parts per row of the sums pass
  int nsr;                   // sampled rows, listed in srow
  const float* logits;       // mode 0: row r at logits + r * ld; mode 1: [rows][depth+1][V]
  long long ld;
  const int32_t* hist;       // [rows][W]
  const int32_t* drafts;     // [rows][depth]
  const float* u;            // mode 0: [rows][depth]; mode 1: [rows][depth+1]
  float* q;                  // mode 0: out [rows][depth][V]; mode 1: the drafts' q (null if unused)
  int32_t* draft_out;        // mode 0
  int32_t* n_acc;            // mode 1 outputs
  int32_t* out_tok;
  int32_t* stats;
  int32_t* h_rec;
  int32_t* status;
  // scratch (flat_workspace_bytes), descriptors first
  TDesc* desc;               // [tasks]
  unsigned long long* amax;  // [tasks][P]
  float* zmin;               // [tasks][P]
  unsigned long long* hist_w;  // [tasks][kFlatHistBins]
  unsigned long long* sub_w;   // [tasks][kFlatHistBins] mass per sub-bin of the crossing bin
  unsigned long long* sminp;   // [tasks]
  int32_t* ccnt;             // [tasks]
  uint32_t* ckey;            // [tasks][kFlatCandCap]
  int32_t* cid;
  unsigned long long* wsum;  // [rows][P2][16 warp slices][2]
  int32_t* nstop;            // [rows]
  int32_t* gcnt;             // [tasks] gathering CTAs done (the last resolves)
  int32_t* scnt;             // [rows] summing CTAs done (the last draws)
  RowParams p[kMaxRows];
  int srow[kMaxRows];        // the rows that are not greedy, in order
};
constexpr int kFlatHistBins = 2048;
constexpr int kFlatCandCap = 1024;
constexpr int kFlatMaxParts = 64;
size_t flat_workspace_bytes(int rows, int tasks);
bool flat_fits(const RowParams* p, int rows, int V, const float* logits, long long ld);
// Lays the scratch out in ws (desc at offset 0), picks the parts per task and
// launches the chain; false (nothing launched) if ws_bytes is too small or q
// does not start on a 16-byte boundary.
bool launch_flat(FlatArgs a, void* ws, size_t ws_bytes, cudaStream_t s);

struct VerifyArgs {
  int rows, V, W, depth;
  const float* logits;
  const int32_t* drafts;
  const float* q;
  const int32_t* hist;
  const float* u;
  const TDesc* desc;
  int32_t* n_acc;
  int32_t* out_tok;
  int32_t* stats;
  int32_t* status;
  int vec_ok;  // logits rows 16-byte aligned (set by the greedy launcher)
  int32_t* h_rec;  // device-visible [rows][depth+2] host record (n_acc, out_tok), or null
  // streaming path only: per (row, position) descriptors (written here, the
  // same array as desc), accept flags and kept lists
  TDesc* wdesc;      // [rows][depth+1]
  int32_t* acc;      // [rows][depth+1]
  int32_t* kid;      // [rows][depth+1][kStreamTopK] kept ids, in (key, id) order
  uint32_t* kkey;    // [rows][depth+1][kStreamTopK] their keys
  int ring_ns;       // stages of the shared-memory ring the target rows stream through
  // bounded waits of the streaming path: polls before a wait gives up (0 =
  // the default), and a ring stage left unfilled (-1 = none) so that a test
  // can make its waits run out (mtp_test_verify_stall)
  unsigned wait_limit;
  int stall_stage;
  RowParams p[kMaxRows];
};
void launch_verify(const VerifyArgs& a, cudaStream_t s);
// Streaming verify for many (row, position) tasks whose sampled rows all have
// 1 <= top_k <= kStreamTopK < V: one CTA per task reads its target row once
// and keeps the exact top-k in shared memory; a second launch walks each
// row's accept chain and draws over the stopping position's kept list.
constexpr int kStreamTopK = 256;
void launch_verify_stream(const VerifyArgs& a, cudaStream_t s);
// The per-row accept chain and draw over the kept lists (wdesc, acc, kid, kkey).
void launch_verify_finish(const VerifyArgs& a, cudaStream_t s);

// Exact top-k transform of rows that cut to a top-k of at most kStreamTopK
// (or are greedy), one 8-CTA cluster per task: draft steps (mode 0: q and the
// draw) or verify tasks (mode 1: descriptor, accept test and kept list for
// launch_verify_finish).
struct TopkArgs {
  int mode;
  int rows, V, W, depth, pos;
  const float* logits;   // mode 0: [rows][ld]; mode 1: [rows][depth+1][V]
  long long ld;
  const int32_t* hist;   // [rows][W]
  const int32_t* drafts; // [rows][depth]
  const float* u;        // mode 0: [rows][depth]; mode 1: [rows][depth+1]
  float* q;              // mode 0: out [rows][depth][V]; mode 1: the drafts' q (in)
  int32_t* draft_out;    // mode 0
  TDesc* wdesc;          // mode 1: [rows][depth+1]
  int32_t* acc;
  int32_t* kid;
  uint32_t* kkey;
  int32_t* status;
  int q_zeroed;          // mode 0: q already holds zeros; write the kept entries only
  RowParams p[kMaxRows];
};
bool topk_fits(const RowParams* p, int rows, int V, const float* logits, long long ld);
void launch_topk(const TopkArgs& a, cudaStream_t s);
size_t verify_stream_smem(int V, int* ring_ns = nullptr);
// All rows greedy without a repetition penalty: argmax matches in one launch
// (depth <= 16; desc, q, hist and u unused).
void launch_verify_greedy(const VerifyArgs& a, cudaStream_t s);
// The same for many rows as one balanced stream over [rows][depth+1][V]
// (equal ranges per CTA, one key per touched segment in d_part, then a
// per-row finish). False, launching nothing, where it does not apply (V % 4,
// alignment, or more than kFlatMaxCTAs ranges or part_bytes of keys needed).
constexpr int kFlatMaxCTAs = 2048;
bool launch_verify_greedy_flat(const VerifyArgs& a, void* d_part, size_t part_bytes, cudaStream_t s);

// Multiprocessor count of the current device (looked up once per device).
constexpr int kMaxDevices = 64;
int device_sm_count();

// spec_verify with the streaming path allowed or not (the workspace of
// spec_verify_workspace_bytes holds its lists; a descriptors-only scratch does not).
mtp_status spec_verify_impl(mtp_stream stream, int32_t rows, int32_t depth, int32_t vocab, const float* d_logits,
                            const int32_t* d_draft, const float* d_q, const mtp_sampling* h_params,
                            const int32_t* d_hist, int32_t hist_w, const float* d_u, int32_t* d_n_acc,
                            int32_t* d_out_tok, int32_t* d_stats, int32_t* h_out, int32_t* d_status,
                            void* d_workspace, size_t workspace_bytes, bool allow_stream);

}  // namespace mtp
