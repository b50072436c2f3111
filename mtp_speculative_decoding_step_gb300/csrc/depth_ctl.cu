// Draft-depth controller (host code, part of libmtp).
//
// "Ollama qwen3_5 MTP loader and SelfDraft path", Facts: depth control, and the
// commit "choose the speculative draft length to maximize throughput" of the
// Ollama MLX-runner log: the controller drafts the depth N that maximises
// committed tokens per wall-clock second, committed(N) / cost(N), from live
// per-position acceptance and a per-width round cost, with N = 0 (plain
// decode) as the floor and at most one past the acceptance frontier. It
// probes one deeper than its choice every 4 rounds; while the choice is plain
// decode the probe interval doubles, up to 512 rounds. Its state lives as long
// as the object, across requests.
//
// Model:
//   a_i         = P(draft i accepted | drafts 1..i-1 accepted), estimated from
//                 the rounds that reached position i (Laplace-smoothed)
//   committed(N)= 1 + sum_{i=1..N} prod_{j<=i} a_j     (accepted drafts + the
//                 correction or bonus token)
//   cost(N)     = mean measured seconds of a round at depth N; an unmeasured
//                 depth extends the nearest measured ones linearly
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <new>
#include <vector>

#include "../../include/mtp.h"

struct mtp_depth_ctl {
  int max_depth = 0;
  std::vector<double> tried, accepted;  // per position i (1-based index i-1)
  std::vector<double> cost_sum, cost_n;  // per depth 0..max_depth
  int chosen = 0;
  long long round = 0;
  int interval = 4;            // rounds between probes
  long long next_probe = 4;
  int last_probe_choice = -1;  // the choice when the last probe was scheduled
};

namespace {

constexpr int kProbeBase = 4;
constexpr int kProbeMax = 512;

double accept_rate(const mtp_depth_ctl* c, int i) {  // i: 1-based position
  return (c->accepted[i - 1] + 0.5) / (c->tried[i - 1] + 1.0);
}

// Largest position with acceptance data (0: none yet).
int frontier(const mtp_depth_ctl* c) {
  int f = 0;
  for (int i = 1; i <= c->max_depth; ++i)
    if (c->tried[i - 1] > 0) f = i;
  return f;
}

double cost_of(const mtp_depth_ctl* c, int n) {
  auto known = [&](int k) { return c->cost_n[k] > 0; };
  auto mean = [&](int k) { return c->cost_sum[k] / c->cost_n[k]; };
  if (known(n)) return mean(n);
  // nearest measured depths below and above
  int lo = -1, hi = -1;
  for (int k = n - 1; k >= 0; --k)
    if (known(k)) { lo = k; break; }
  for (int k = n + 1; k <= c->max_depth; ++k)
    if (known(k)) { hi = k; break; }
  if (lo >= 0 && hi >= 0) return mean(lo) + (mean(hi) - mean(lo)) * (n - lo) / (double)(hi - lo);
  if (lo >= 0) {  // extend the slope of the two measured depths below, else a flat cost
    int lo2 = -1;
    for (int k = lo - 1; k >= 0; --k)
      if (known(k)) { lo2 = k; break; }
    const double slope = lo2 >= 0 ? (mean(lo) - mean(lo2)) / (double)(lo - lo2) : 0.0;
    return mean(lo) + std::max(slope, 0.0) * (n - lo);
  }
  if (hi >= 0) {  // below every measured depth: extend the slope of the two lowest
    int hi2 = -1;
    for (int k = hi + 1; k <= c->max_depth; ++k)
      if (known(k)) { hi2 = k; break; }
    const double slope = hi2 >= 0 ? (mean(hi2) - mean(hi)) / (double)(hi2 - hi) : 0.0;
    return std::max(mean(hi) - std::max(slope, 0.0) * (hi - n), 1e-9);
  }
  return 1.0;  // nothing measured: every depth costs the same
}

int best_depth(const mtp_depth_ctl* c) {
  const int top = std::min(c->max_depth, frontier(c) + 1);
  int best = 0;
  double best_v = -1.0, committed = 1.0, run = 1.0;
  for (int n = 0; n <= top; ++n) {
    if (n > 0) {
      run *= accept_rate(c, n);
      committed += run;
    }
    const double v = committed / std::max(cost_of(c, n), 1e-12);
    if (v > best_v * (1.0 + 1e-12)) { best_v = v; best = n; }
  }
  return best;
}

}  // namespace

extern "C" {

mtp_status mtp_depth_ctl_create(int32_t max_depth, mtp_depth_ctl_t* out) {
  if (!out || max_depth < 0 || max_depth > 64) return MTP_ERR_BAD_ARG;
  mtp_depth_ctl* c = new (std::nothrow) mtp_depth_ctl();
  if (!c) return MTP_ERR_CUDA;
  c->max_depth = max_depth;
  c->tried.assign(max_depth, 0.0);
  c->accepted.assign(max_depth, 0.0);
  c->cost_sum.assign(max_depth + 1, 0.0);
  c->cost_n.assign(max_depth + 1, 0.0);
  c->chosen = 0;
  *out = c;
  return MTP_OK;
}

void mtp_depth_ctl_free(mtp_depth_ctl_t c) { delete c; }

int32_t mtp_depth_ctl_next(mtp_depth_ctl_t c) {
  if (!c) return 0;
  // the floor first: a round of plain decode measures the base cost that every
  // deeper round is weighed against
  if (c->cost_n[0] == 0) return 0;
  c->chosen = best_depth(c);
  ++c->round;
  if (c->round < c->next_probe) return c->chosen;
  // a probe round: one past the choice. While the choice is plain decode
  // (speculation does not pay), each probe doubles the interval, up to 512
  // rounds; any deeper choice keeps probing every 4.
  if (c->chosen == 0 && c->last_probe_choice == 0) c->interval = std::min(c->interval * 2, kProbeMax);
  else if (c->chosen != 0) c->interval = kProbeBase;
  c->last_probe_choice = c->chosen;
  c->next_probe = c->round + c->interval;
  return c->chosen < c->max_depth ? c->chosen + 1 : c->chosen;
}

mtp_status mtp_depth_ctl_observe(mtp_depth_ctl_t c, int32_t depth, int32_t n_acc, double round_seconds) {
  if (!c || depth < 0 || depth > c->max_depth || n_acc < 0 || n_acc > depth || !(round_seconds > 0.0))
    return MTP_ERR_BAD_ARG;
  // positions 1..n_acc were accepted; position n_acc+1 (if drafted) was rejected
  for (int i = 1; i <= std::min(depth, n_acc + 1); ++i) {
    c->tried[i - 1] += 1.0;
    if (i <= n_acc) c->accepted[i - 1] += 1.0;
  }
  c->cost_sum[depth] += round_seconds;
  c->cost_n[depth] += 1.0;
  return MTP_OK;
}

mtp_status mtp_depth_ctl_state(mtp_depth_ctl_t c, double* h_accept, double* h_cost, int32_t* h_interval) {
  if (!c) return MTP_ERR_BAD_ARG;
  for (int i = 1; i <= c->max_depth; ++i)
    if (h_accept) h_accept[i - 1] = accept_rate(c, i);
  for (int n = 0; n <= c->max_depth; ++n)
    if (h_cost) h_cost[n] = cost_of(c, n);
  if (h_interval) *h_interval = c->interval;
  return MTP_OK;
}

}  // extern "C"
