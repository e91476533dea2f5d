// Host-side internals shared by the library's translation units: the handle,
// small helpers, and the per-logits-type operations.  The kernels of each
// (target type, draft type) pair are instantiated in a translation unit of
// their own (pair_*.cu), so that the four compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

#include "spec_verify.h"
#include "verify_kernel.cuh"
#include "diag_kernel.cuh"
#include "filter_kernel.cuh"
#include "hist_kernel.cuh"

struct spec_verify_s {
  int device = 0;
  int max_B = 0, k = 0, V = 0, nchunk = 0;
  int num_sms = 0;
  int blocks_per_sm[2][2] = {{0, 0}, {0, 0}};  // [target is bf16][draft is bf16]
  int fin_spread_smem = 0;                     // see finish_spread_smem
  void* ws = nullptr;                          // one device allocation for the workspace
  size_t ws_bytes = 0;
  float2* part = nullptr;
  float* xD = nullptr;
  sv::Cand* cand = nullptr;
  unsigned* cand_over = nullptr;
  sv::DiagNorm* dnorm = nullptr;  // [max_B, k] (diagnostics)
  // one-shot timing marks around the next stream pass
  cudaEvent_t mark_before = nullptr, mark_after = nullptr;
  // staging for spec_verify_run_host (allocated on first use)
  void* stage = nullptr;
  size_t stage_bytes = 0;
  // gate policy (spec_verify_set_gate_policy): schedule entries, cumulative floor
  int n_sched = 0;
  float sched[SV_MAX_K] = {};
  float min_cum = 0.f;
  // sampler filters (spec_verify_set_filters) and their buffer, allocated on
  // first use: each row's kept set
  sv::Filter filt[2] = {{0, 1.f, 0.f}, {0, 1.f, 0.f}};
  void* fbuf = nullptr;
  size_t fbuf_bytes = 0;
};

namespace sv {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Dynamic shared memory for a finishing CTA that is to have its SM to itself:
// just over half of an SM's shared memory, or 0 where the device cannot give
// that much to one CTA.  Two finishing CTAs on one SM slow each other's
// dependent chains (measured: about 1 us per call on the 128K-vocabulary
// batch), so a grid that fits one CTA per SM asks for this much.
inline int finish_spread_smem(int device) {
  int per_sm = 0, optin = 0;
  if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
    return 0;
  const int want = per_sm / 2 + 1024;
  return want <= optin && want > static_cast<int>(sizeof(FinishShared)) ? want : 0;
}

inline bool filter_on(const Filter& f) { return f.top_k != 0 || f.top_p < 1.f || f.min_p > 0.f; }

// The operations of one (target type, draft type) pair of logits.
struct PairOps {
  // opt every kernel of the pair into its shared memory; how many stream CTAs fit on an SM
  cudaError_t (*configure)(int* blocks_per_sm, int fin_spread_smem);
  // one verifying call of variant `mode` (kModeSample, kModePolicy, kModeGreedy), with the
  // sampler filters' prefix when `filtered`
  sv_status (*verify)(spec_verify_t h, Params& P, int mode, int blocks_per_sm, bool dense_likely,
                      bool filtered, cudaStream_t st);
  // the acceptance diagnostics, with the sampler filters' prefix when `filtered`
  sv_status (*diagnostics)(spec_verify_t h, Params& P, int blocks_per_sm, bool filtered, float* min_sum,
                           float* pq_sum, float* argmax_q, cudaStream_t st);
};

extern const PairOps ops_f32_f32, ops_f32_bf16, ops_bf16_f32, ops_bf16_bf16;

inline const PairOps& pair_ops(bool target_bf16, bool draft_bf16) {
  if (target_bf16) return draft_bf16 ? ops_bf16_bf16 : ops_bf16_f32;
  return draft_bf16 ? ops_f32_bf16 : ops_f32_f32;
}

}  // namespace sv
