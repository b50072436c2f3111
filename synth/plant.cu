// Device-side synthetic target rows for the benchmark loop: the same rule as
// plant_logits() in synth/__init__.py, applied in place to the verify block
// the drafts just produced. Row i (i < depth) gets logit[x_{i+1}] = max + 1
// when coin i is set; otherwise, if x_{i+1} was the row's argmax, its logit
// becomes second - 1. The row maxima come in precomputed (top1, top2, arg1).
// This is input generation for the benchmark, not part of the library.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void synth_plant_kernel(float* lg, long long vocab, const int32_t* draft, int depth,
                                   const uint8_t* coins, const float* top1, const float* top2,
                                   const int64_t* arg1) {
  const int i = threadIdx.x;
  if (i >= depth) return;
  const int x = draft[i];
  if (x < 0 || x >= vocab) return;
  float* p = lg + (long long)i * vocab + x;
  if (coins[i]) *p = top1[i] + 1.0f;
  else if (arg1[i] == x) *p = top2[i] - 1.0f;
}

extern "C" int synth_plant(void* stream, float* lg, long long vocab, const int32_t* draft, int depth,
                           const uint8_t* coins, const float* top1, const float* top2, const int64_t* arg1) {
  if (depth < 1 || depth > 32) return (int)cudaErrorInvalidValue;
  synth_plant_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(lg, vocab, draft, depth, coins, top1, top2, arg1);
  return (int)cudaGetLastError();
}
