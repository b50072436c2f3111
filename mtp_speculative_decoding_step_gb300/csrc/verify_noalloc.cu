// spec_verify_noalloc: spec_verify for callers that cannot allocate device
// memory. Some hosts of this library own every byte of device memory through
// their own pool, or run inside a region where a device allocation would
// stall the whole device (cudaMalloc synchronises) or is not allowed at all;
// such callers cannot provide spec_verify's workspace. This entry point keeps
// that scratch (one transform descriptor per verified row and position) in a
// fixed array compiled into the library instead.
//
// The array lives in every device that loads the library, for the life of the
// process. Its device address is looked up once per device, on the first call
// made with that device current; make that first call before capturing a
// stream into a graph. All calls share the one array: calls whose kernels can
// overlap on the GPU (different streams, no ordering between them) race on it.
// Each call writes every descriptor it reads, so nothing needs clearing.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mtp.h"
#include "kernels.h"

namespace {

// rows * (depth + 1) descriptors at most: 64 rows at the deepest block (16 + 1).
constexpr int kNoAllocDescs = mtp::kMaxRows * 17;

__device__ __align__(256) mtp::TDesc g_verify_scratch[kNoAllocDescs];

constexpr int kMaxDevices = 64;
void* g_addr[kMaxDevices] = {};
std::mutex g_mu;

// Device address of the scratch array for the current device (set up once).
mtp_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MTP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return MTP_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MTP_OK;
}

}  // namespace

extern "C" mtp_status spec_verify_noalloc(mtp_stream stream, int32_t rows, int32_t depth, int32_t vocab,
                                          const float* d_logits, const int32_t* d_draft, const float* d_q,
                                          const mtp_sampling* h_params, const int32_t* d_hist, int32_t hist_w,
                                          const float* d_u, int32_t* d_n_acc, int32_t* d_out_tok,
                                          int32_t* d_stats, int32_t* h_out, int32_t* d_status) {
  if (rows < 1 || depth < 1 || (long long)rows * (depth + 1) > kNoAllocDescs) return MTP_ERR_BAD_ARG;
  void* scratch = nullptr;
  const mtp_status st = scratch_address(&scratch);
  if (st != MTP_OK) return st;
  // the scratch holds descriptors only: the streaming path (which also needs
  // per-task kept lists) stays off
  return mtp::spec_verify_impl(stream, rows, depth, vocab, d_logits, d_draft, d_q, h_params, d_hist, hist_w, d_u,
                               d_n_acc, d_out_tok, d_stats, h_out, d_status, scratch, sizeof(g_verify_scratch),
                               false);
}
