/*
 * mtp.h — C ABI of the GB300 multi-token-prediction (MTP) speculative
 * decoding step: the MTP drafter head, the batched flush of completed pairs
 * into the draft KV cache, the sampling transforms, the rejection-sampling
 * verify and the KV rollback.
 *
 * Conventions for every entry point
 *  - Pointers named d_* are CUDA device pointers; h_* are host pointers.
 *    No torch or CUDA C++ types appear; `mtp_stream` is a cudaStream_t.
 *  - Every call is asynchronous on the given stream, allocates nothing, never
 *    reads device memory on the host and never synchronises, so a caller can
 *    capture a whole round into a CUDA graph. Only mtp_load / mtp_free
 *    allocate and free (the handle's scratch and norm copies) and may block.
 *  - Arguments are validated on the host before any launch; a bad argument
 *    returns a status and launches nothing. Faults seen on the device (a
 *    non-finite logit, a bounded wait that ran out) are OR-ed, as
 *    1 << MTP_ERR_*, into a device status word that the caller reads at its
 *    one per-round synchronisation: the handle's word (mtp_device_status) for
 *    the head calls, the caller's d_status for spec_verify, which takes no
 *    handle. The outputs of a call whose status word gained a bit carry no
 *    meaning; spec_verify's still stay in range (token ids in [0, V), counts
 *    in [0, depth]).
 *  - The caller owns every buffer it passes. Large weights, the borrowed
 *    embedding / lm_head and the KV buffers are borrowed by mtp_load and must
 *    outlive the handle.
 *
 * Notation: H hidden, nq / nkv query / key-value heads, dh head_dim, I SwiGLU
 * intermediate, V vocabulary, R rows (independent sequences), d draft depth.
 */
#ifndef MTP_H
#define MTP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mtp_stream; /* cudaStream_t */
typedef struct mtp_handle* mtp_t;

typedef enum {
  MTP_OK = 0,
  MTP_ERR_UNSUPPORTED_ARCH = 1, /* architecture is not "qwen3_5_mtp" */
  MTP_ERR_MISSING_TENSOR = 2,   /* one of the 15 head tensors is absent */
  MTP_ERR_DUP_TENSOR = 3,       /* a tensor name appears twice */
  MTP_ERR_UNKNOWN_TENSOR = 4,   /* a name outside the 15-tensor inventory */
  MTP_ERR_SHAPE = 5,            /* a tensor's shape or dtype disagrees with the config */
  MTP_ERR_CONFIG_BOUNDS = 6,    /* a config scalar is out of range */
  MTP_ERR_NOT_BOUND = 7,        /* no borrowed embedding was given (bind skipped) */
  MTP_ERR_KV_CAPACITY = 8,      /* a write would pass the KV capacity */
  MTP_ERR_BAD_ARG = 9,          /* null pointer, bad count, bad sampling parameter */
  MTP_ERR_NONFINITE = 10,       /* device status bit: a non-finite logit was seen */
  MTP_ERR_TIMEOUT = 11,         /* device status bit: a bounded wait on an asynchronous copy ran out */
  MTP_ERR_CUDA = 12,            /* a CUDA runtime call failed */
  MTP_ERR_LAYOUT = 13           /* tensor names mix the raw-HF "mtp." and split layouts */
} mtp_status;

enum { MTP_DTYPE_F32 = 0, MTP_DTYPE_BF16 = 1 };

/* Head configuration. Mirrors the text_config scalars of a qwen3_5_mtp
 * drafter ("support the qwen3_5_mtp drafter" issue, "Where the MTP weights
 * actually live": hidden_size, head_dim, mtp_num_hidden_layers). Bounds are
 * checked at load ("bound the qwen3_5_mtp drafter config scalars at load"). */
typedef struct {
  const char* architecture; /* must equal "qwen3_5_mtp" */
  int32_t hidden;           /* H, multiple of 256, <= 16384 */
  int32_t n_q, n_kv;        /* query / kv heads; n_q % n_kv == 0 */
  int32_t head_dim;         /* dh in {64, 128, 256} */
  int32_t inter;            /* I, multiple of 256 */
  int32_t vocab;            /* V, <= 1 << 20 */
  int32_t mtp_layers;       /* must be 1 (the published head has one layer) */
  int32_t max_rows;         /* R, 1..64 */
  int32_t kv_capacity;      /* slots per row, multiple of 64 */
  int32_t max_depth;        /* drafts per round, 1..16 */
  float eps;                /* RMSNorm epsilon */
  float rope_theta;         /* RoPE base */
  int32_t dtype;            /* MTP_DTYPE_F32 or MTP_DTYPE_BF16: weights, embedding, KV */
} mtp_config;

/* One named head tensor (device memory, row-major). Names follow either the
 * raw-HF layout ("mtp.fc.weight", ...) or the split drafter layout
 * ("fc.weight", ...). In the raw-HF layout the loader adds 1.0 to the seven
 * RMSNorm weights (suffixes .input_layernorm.weight,
 * .post_attention_layernorm.weight, .q_norm.weight, .k_norm.weight,
 * norm.weight, pre_fc_norm_embedding.weight, pre_fc_norm_hidden.weight) exactly
 * once ("Upstream contract to port", sanitize paragraph). */
typedef struct {
  const char* name;
  const void* data;
  int32_t dtype;
  int32_t ndim;     /* 1 or 2 */
  int64_t shape[2];
} mtp_tensor;

/* Per-row sampling parameters. temperature 0 (or top_k 1) is greedy: the
 * point mass at the argmax ("greedy is a special case of sampled decoding",
 * Ollama MLX-runner commit log). rep_penalty 1, top_k 0, top_p 1, min_p 0
 * disable their transforms.
 *
 * flags: 0, or MTP_SAMPLE_ARGMAX_DRAFT on a sampled row: the drafter proposes
 * the argmax of its (penalised) logits instead of a sample, and spec_verify
 * treats that draft as a point mass q (q(x) = 1): x is accepted with
 * probability p(x) and a rejection draws from p with x removed, so the
 * committed tokens still follow p. This is the drafter flag
 * supports_greedy_draft_argmax ("feat(inference): support the qwen3_5_mtp
 * drafter" issue, Upstream contract to port); mtp_draft then needs neither
 * d_q nor d_u for the row, and spec_verify reads no q for it. */
#define MTP_SAMPLE_ARGMAX_DRAFT 1
typedef struct {
  float temperature;  /* >= 0 */
  float rep_penalty;  /* > 0 */
  float top_p;        /* (0, 1] */
  float min_p;        /* [0, 1) */
  int32_t top_k;      /* 0 = off, else 1..1024 */
  int32_t flags;      /* 0 or MTP_SAMPLE_ARGMAX_DRAFT; other bits are rejected
                         (frequency penalty is not implemented) */
} mtp_sampling;

/* Draft KV cache buffers, caller-owned device memory, borrowed by mtp_load.
 * k, v: [max_rows][n_kv][kv_capacity][head_dim] in the config dtype.
 * len:  [max_rows] int32, the number of valid slots per row; the library
 *       keeps it equal to its host-side lengths after every call. */
typedef struct {
  void* k;
  void* v;
  int32_t* len;
} mtp_kv;

/* Default round budget including the bonus token: mtp_layers + 2 (the
 * drafter's block_size, "Upstream contract to port"). Drafts per round are
 * block_size - 1. */
int32_t mtp_default_block_size(const mtp_config* cfg);

const char* mtp_status_str(mtp_status s);

/* Validate the config and the tensor table, copy the seven norm vectors into
 * library memory as fp32 (with the raw-HF +1.0 applied once), borrow every
 * matrix, the embedding and the lm_head (NULL = tied to embed, the drafter's
 * bind fallback), borrow the KV buffers, set every row length to h_len[r]
 * (or 0 if h_len is NULL) and allocate the scratch. Blocks until the copies
 * finish. Errors: UNSUPPORTED_ARCH, MISSING/DUP/UNKNOWN_TENSOR, LAYOUT, SHAPE,
 * CONFIG_BOUNDS, NOT_BOUND (embed NULL), BAD_ARG, CUDA. On error *out is NULL
 * and nothing stays allocated. */
mtp_status mtp_load(const mtp_config* cfg, const mtp_tensor* tensors, int32_t n_tensors,
                    const void* d_embed, const void* d_lm_head, mtp_kv kv,
                    const int32_t* h_len, mtp_stream stream, mtp_t* out);

mtp_status mtp_free(mtp_t h);

/* Host view of the per-row draft KV lengths (the library's source of truth;
 * mirrored into kv.len on the device). h_len: [max_rows]. */
mtp_status mtp_get_lengths(mtp_t h, int32_t* h_len);

/* Set row lengths (e.g. after the caller pre-filled or restored the cache). */
mtp_status mtp_set_lengths(mtp_t h, mtp_stream stream, const int32_t* h_len);

/* Device pointer of the handle's status word (int32, OR of 1 << status). */
int32_t* mtp_device_status(mtp_t h);

/*
 * mtp_flush — write completed pairs into the draft KV.
 * Slot S pairs the token at S+1 with the target hidden at S ("Ollama qwen3_5
 * MTP loader and SelfDraft path", Facts: pairing and the 256-token flush cap).
 * Row r's pairs j = 0..h_pairs[r]-1 go to slots len[r] + j, and len[r]
 * advances by h_pairs[r]. For a one-layer head a slot's K and V depend only on
 * its own pair (fc, input norm, k/v projections, k_norm, RoPE), so the flush
 * computes exactly those; no attention is needed.
 *   d_tok [rows][pmax] int32, d_hid [rows][pmax][H] in hid_dtype.
 * Errors: BAD_ARG (rows > max_rows, a count < 0 or > pmax), KV_CAPACITY.
 */
mtp_status mtp_flush(mtp_t h, mtp_stream stream, int32_t rows, const int32_t* h_pairs,
                     int32_t pmax, const int32_t* d_tok, const void* d_hid, int32_t hid_dtype);

/*
 * mtp_draft — propose `depth` tokens per row with one head call per token.
 * The first call consumes h_pairs[r] >= 1 pairs of row r at slots len[r]..:
 * the first h_pairs[r]-1 are pending completed pairs (flushed in the same
 * pass), the last is the newest pair (token c_T, target hidden at T-1) and
 * yields the step-1 logits. Step k >= 2 consumes the step-(k-1) draft token
 * and the head's own pre-norm hidden h2 at the next slot.
 * Token selection per row: greedy rows take the argmax of the (penalised)
 * logits; sampled rows apply the transform chain (repetition penalty over the
 * window "last hist_w of d_hist[r] ++ drafts so far", temperature, top-k,
 * top-p, min-p) and draw by inverse CDF with d_u[r][k-1].
 *   d_tok [rows][pmax] int32, d_hid [rows][pmax][H] (hid_dtype)
 *   h_params [rows] (host), d_hist [rows][hist_w] int32 (oldest first, -1 empty)
 *   d_u [rows][depth] float in [0,1) (may be NULL if every row is greedy)
 *   d_draft [rows][depth] int32 out
 *   d_q [rows][depth][V] float out: the distribution each sampled draft was
 *       drawn from (rows that are greedy are left untouched); may be NULL if
 *       every row is greedy
 *   d_logits [rows][depth][V] float out (optional, NULL to skip)
 *   d_hidden [rows][depth][H] float out: h2 per step (optional)
 * After the call len[r] has advanced by h_pairs[r] + depth - 1; kv_rollback
 * keeps only the slots of the first call (len before + h_pairs[r]).
 * Errors: BAD_ARG, KV_CAPACITY.
 */
mtp_status mtp_draft(mtp_t h, mtp_stream stream, int32_t rows, int32_t depth,
                     const int32_t* h_pairs, int32_t pmax, const int32_t* d_tok,
                     const void* d_hid, int32_t hid_dtype, const mtp_sampling* h_params,
                     const int32_t* d_hist, int32_t hist_w, const float* d_u,
                     int32_t* d_draft, float* d_q, float* d_logits, float* d_hidden);

/*
 * spec_verify — rejection-sampling verify of a block of target logits
 * (Leviathan et al., Chen et al.; "greedy is a special case of sampled
 * decoding", Ollama MLX-runner commit log).
 * For each row r, with p_i the transformed target distribution of row i
 * (window "last hist_w of d_hist[r] ++ x_1..x_i"):
 *   for i = 1..d: accept x_i iff q_i(x_i) > 0 and u[i-1] < p_{i-1}(x_i)/q_i(x_i)
 *   first reject at i: y ~ norm(max(p_{i-1} - q_i, 0)) with u[d]
 *   all accepted:      y ~ p_d with u[d]          (the bonus token)
 * Greedy rows: accept iff x_i == argmax p_{i-1}; y = argmax of the stopping row.
 *   d_logits [rows][depth+1][vocab] float, d_draft [rows][depth] int32
 *   d_q [rows][depth][vocab] float (ignored for greedy rows; NULL if all greedy)
 *   h_params [rows] (host), d_hist [rows][hist_w], d_u [rows][depth+1]
 *   d_n_acc [rows] out, d_out_tok [rows][depth+1] out (accepted drafts, then y,
 *   then -1), d_stats [rows][depth+2] int32 accumulated (NULL to skip):
 *   [0] rounds, [1] rounds with a rejection (rollbacks), [1+i] accepts at i.
 *   h_out (optional, pinned host, [rows][depth+2]): n_acc then out_tok per row,
 *   the round's one device->host read. Page-locked memory the device can
 *   address (cudaHostAlloc / cudaMallocHost) is written by the verify kernel
 *   itself; other host memory gets a copy enqueued after the kernel. Either
 *   way it is complete once the stream has reached the end of this call. In
 *   device-addressable memory each row's n_acc is stored after its out_tok
 *   with release semantics at system scope: a host that set n_acc negative
 *   beforehand may poll it instead of waiting for the stream.
 *   d_status (optional, device int32): OR-ed with 1 << MTP_ERR_NONFINITE when
 *   a target logit the verify reads is NaN or infinite, and with
 *   1 << MTP_ERR_TIMEOUT when a bounded wait of the streaming path ran out
 *   (fail-closed errors, "Ollama qwen3_5 MTP loader and SelfDraft path",
 *   Facts). The caller clears it; NULL drops these reports.
 *   d_workspace: spec_verify_workspace_bytes(rows, depth, vocab) bytes (the
 *   transform descriptors, then the streaming path's accept flags and kept lists).
 * Calls with more (row, position) tasks than one wave of 8-CTA clusters holds,
 * whose sampled rows all cut to a top-k of at most 256 below the vocabulary,
 * take a streaming path: one CTA per task reads its target row once. Its
 * results are identical.
 * Errors: BAD_ARG.
 */
size_t spec_verify_workspace_bytes(int32_t rows, int32_t depth, int32_t vocab);

mtp_status spec_verify(mtp_stream stream, int32_t rows, int32_t depth, int32_t vocab,
                       const float* d_logits, const int32_t* d_draft, const float* d_q,
                       const mtp_sampling* h_params, const int32_t* d_hist, int32_t hist_w,
                       const float* d_u, int32_t* d_n_acc, int32_t* d_out_tok,
                       int32_t* d_stats, int32_t* h_out, int32_t* d_status, void* d_workspace);

/*
 * mtp_set_draft_head — which copy of the tied output head the drafter reads.
 * MTP_HEAD_BF16 (the default): the borrowed head itself. MTP_HEAD_FP8: an fp8
 * e4m3 copy with one fp32 scale per row (scale = max|row| / 448, codes =
 * e4m3(w / scale), round to nearest even, saturating), made from the borrowed
 * head by this call and owned by the handle (vocab * hidden bytes + vocab
 * floats, allocated on the first request). The draft logits become
 * scale[v] * sum_k e4m3(code[v,k]) * x[k]: half the head's bytes per draft
 * step, a draft-only change ("Ollama qwen3_5 MTP loader and SelfDraft path",
 * Facts: quantizing the draft's tied output head; the format is not stated
 * there). spec_verify is untouched: it reads the target's logits. Call again
 * after the borrowed head's contents change. bf16 heads only; asynchronous on
 * the stream. Errors: BAD_ARG, CONFIG_BOUNDS (fp32 head or hidden % 16),
 * CUDA.
 */
#define MTP_HEAD_BF16 0
#define MTP_HEAD_FP8 1
mtp_status mtp_set_draft_head(mtp_t h, mtp_stream stream, int32_t format);

/*
 * Draft-depth controller (host-side; "Ollama qwen3_5 MTP loader and SelfDraft
 * path", Facts: depth control; Ollama MLX-runner commit "choose the
 * speculative draft length to maximize throughput"). It picks the depth N in
 * [0, max_depth] that maximises committed(N) / cost(N): committed(N) =
 * 1 + sum_{i<=N} prod_{j<=i} a_j from per-position acceptance a_j (Laplace-
 * smoothed counts of rounds that reached position j), cost(N) = the mean
 * measured seconds of a round at depth N (an unmeasured depth extends its
 * measured neighbours linearly). N never exceeds one past the deepest position
 * with data. Every 4th round it returns one past its choice (a probe); while
 * the choice is plain decode each probe doubles that interval, up to 512
 * rounds. Before any other choice it runs one round of plain decode (depth 0)
 * to measure the base cost.
 * State persists for the object's lifetime. No GPU work; not thread-safe.
 *   mtp_depth_ctl_next: depth to draft this round (0 = plain decode).
 *   mtp_depth_ctl_observe: feed back the round actually run (depth, accepted
 *     drafts n_acc <= depth, wall-clock seconds > 0); BAD_ARG otherwise.
 *   mtp_depth_ctl_state: optional host outputs a[max_depth] (acceptance
 *     estimates), cost[max_depth+1] (seconds per round), the probe interval.
 */
typedef struct mtp_depth_ctl* mtp_depth_ctl_t;
mtp_status mtp_depth_ctl_create(int32_t max_depth, mtp_depth_ctl_t* out);
void mtp_depth_ctl_free(mtp_depth_ctl_t c);
int32_t mtp_depth_ctl_next(mtp_depth_ctl_t c);
mtp_status mtp_depth_ctl_observe(mtp_depth_ctl_t c, int32_t depth, int32_t n_acc, double round_seconds);
mtp_status mtp_depth_ctl_state(mtp_depth_ctl_t c, double* h_accept, double* h_cost, int32_t* h_interval);

/*
 * spec_verify_noalloc — spec_verify without a caller-provided workspace, for
 * callers that cannot allocate device memory (a host whose own pool owns all
 * device memory, or code running where a cudaMalloc would stall the device or
 * is forbidden). The pages have no counterpart; it exists for such hosts.
 * Same arguments and results as spec_verify minus d_workspace (d_status
 * included). The scratch
 * (one 32-byte descriptor per verified row and position) is a fixed array
 * inside the library, 1088 descriptors (34,816 bytes) per device, held for
 * the life of the process: rows * (depth + 1) above 1088 returns
 * MTP_ERR_BAD_ARG. The first call on a device, with that device current, looks
 * up the array's address; make it before capturing a stream into a graph.
 * Every call shares the array, so calls that can run at the same time on the
 * GPU (unordered streams) race on it. Allocates nothing.
 */
mtp_status spec_verify_noalloc(mtp_stream stream, int32_t rows, int32_t depth, int32_t vocab,
                               const float* d_logits, const int32_t* d_draft, const float* d_q,
                               const mtp_sampling* h_params, const int32_t* d_hist, int32_t hist_w,
                               const float* d_u, int32_t* d_n_acc, int32_t* d_out_tok,
                               int32_t* d_stats, int32_t* h_out, int32_t* d_status);

/*
 * kv_rollback — drop speculative cache slots after a verify.
 * Draft KV: row r keeps only the slots of the last mtp_draft's first head call
 * (its length becomes the length before that call + h_pairs[r]); with
 * zero_tail the dropped slots are zeroed. Target KV (optional): each
 * d_target_len[r] is trimmed by block - (d_n_acc[r] + 1), block = depth + 1
 * verified positions: the positions past the accepted drafts and the one
 * committed correction or bonus token are dropped ("support the qwen3_5_mtp
 * drafter" issue, comment on qualifying the qwen3_5 path). Rows never drafted
 * are left as they are.
 * Errors: BAD_ARG.
 */
mtp_status kv_rollback(mtp_t h, mtp_stream stream, int32_t rows, const int32_t* d_n_acc,
                       int32_t* d_target_len, int32_t depth, int32_t zero_tail);

/* Test hook of the streaming verify's bounded waits: the next spec_verify
 * call that takes the streaming path leaves ring stage `stage` of every task
 * unfilled (a copy that never lands) and gives each wait `wait_polls` polls,
 * so its waits run out; it then reports MTP_ERR_TIMEOUT in d_status, writes
 * in-range outputs and leaves the context usable. One-shot, process-wide, not
 * for production use. Errors: BAD_ARG (stage < 0 or wait_polls < 1). */
mtp_status mtp_test_verify_stall(int32_t stage, int32_t wait_polls);

/* Number of kernels this library has launched in the process so far. */
int64_t mtp_kernel_launches(void);

/* Timing hook for the benchmark: kernels of the kinds selected by `mask`
 * (bit i = kind i, -1 = all, 0 = off) are bracketed by CUDA events on the
 * launching stream; mtp_profile_read synchronises those events and returns,
 * per kernel kind, the summed milliseconds and the launch count since the
 * last read. Kinds are listed by mtp_profile_kind_name(i) for
 * i < mtp_profile_kinds(). */
mtp_status mtp_profile_enable(mtp_t h, int32_t mask);
int32_t mtp_profile_kinds(void);
const char* mtp_profile_kind_name(int32_t kind);
mtp_status mtp_profile_read(mtp_t h, float* h_ms, int32_t* h_launches);

#ifdef __cplusplus
}
#endif
#endif /* MTP_H */
