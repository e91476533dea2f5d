// Host side of the C ABI declared in include/spec_verify.h: handle and
// workspace management and argument validation.  The launches of each call
// (the stream pass, then the finishing pass as a programmatic dependent
// launch) are in launch.cuh, instantiated per pair of logits types in the
// pair_*.cu translation units.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "handle.h"


namespace {

using sv::align_up;
using sv::filter_on;

size_t elem_size(sv_dtype d) { return d == SV_BF16 ? 2 : 4; }

bool valid_dtype(int d) { return d == SV_F32 || d == SV_BF16; }

// every pair of logits types: kernel attributes, stream CTAs per SM
cudaError_t configure_all(int (*blocks_per_sm)[2], int fin_spread_smem) {
  cudaError_t e = sv::ops_f32_f32.configure(&blocks_per_sm[0][0], fin_spread_smem);
  if (e == cudaSuccess) e = sv::ops_f32_bf16.configure(&blocks_per_sm[0][1], fin_spread_smem);
  if (e == cudaSuccess) e = sv::ops_bf16_f32.configure(&blocks_per_sm[1][0], fin_spread_smem);
  if (e == cudaSuccess) e = sv::ops_bf16_bf16.configure(&blocks_per_sm[1][1], fin_spread_smem);
  return e;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" {

const char* spec_verify_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_EINVAL: return "invalid argument";
    case SV_ENOMEM: return "out of memory";
    case SV_ECUDA: return "CUDA error";
    case SV_EUNSUPPORTED: return "unsupported size";
  }
  return "unknown status";
}

int spec_verify_launches_per_run(void) { return 2; }

int spec_verify_launches_per_filtered_run(void) { return 7; }

sv_status spec_verify_mark_next(spec_verify_t h, void* ev_before, void* ev_after) {
  if (!h || (ev_before == nullptr) != (ev_after == nullptr)) return SV_EINVAL;
  h->mark_before = static_cast<cudaEvent_t>(ev_before);
  h->mark_after = static_cast<cudaEvent_t>(ev_after);
  return SV_OK;
}

sv_status spec_verify_init(spec_verify_t* out, int max_B, int k, int V, int device) {
  if (!out) return SV_EINVAL;
  *out = nullptr;
  if (max_B < 1 || k < 1 || V < 1) return SV_EINVAL;
  if (k > SV_MAX_K || V > SV_MAX_V) return SV_EUNSUPPORTED;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return SV_ECUDA;
  DeviceGuard g(device);
  if (!g.ok) return SV_ECUDA;

  spec_verify_s* h = new (std::nothrow) spec_verify_s();
  if (!h) return SV_ENOMEM;
  h->device = device;
  h->max_B = max_B;
  h->k = k;
  h->V = V;
  h->nchunk = (V + sv::kChunk - 1) / sv::kChunk;
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    delete h;
    return SV_ECUDA;
  }
  h->fin_spread_smem = sv::finish_spread_smem(device);
  const cudaError_t e = configure_all(h->blocks_per_sm, h->fin_spread_smem);
  if (e != cudaSuccess) {
    delete h;
    return SV_ECUDA;
  }

  const size_t rows = 2 * static_cast<size_t>(k) + 1;
  const size_t n_part = static_cast<size_t>(max_B) * rows * h->nchunk;
  const size_t n_rowc = static_cast<size_t>(max_B) * k;
  size_t off = 0;
  const size_t o_part = off; off = align_up(off + n_part * sizeof(float2), 256);
  const size_t o_xd = off;   off = align_up(off + static_cast<size_t>(max_B) * rows * sizeof(float), 256);
  const size_t n_cand = n_rowc * h->nchunk * sv::kTopM;
  const size_t o_cd = off;   off = align_up(off + n_cand * sizeof(sv::Cand), 256);
  const size_t o_co = off;   off = align_up(off + n_rowc * sizeof(unsigned), 256);
  const size_t o_dn = off;   off = align_up(off + n_rowc * sizeof(sv::DiagNorm), 256);
  if (cudaMalloc(&h->ws, off) != cudaSuccess) {
    delete h;
    return SV_ENOMEM;
  }
  h->ws_bytes = off;
  char* base = static_cast<char*>(h->ws);
  h->part = reinterpret_cast<float2*>(base + o_part);
  h->xD = reinterpret_cast<float*>(base + o_xd);
  h->cand = reinterpret_cast<sv::Cand*>(base + o_cd);
  h->cand_over = reinterpret_cast<unsigned*>(base + o_co);
  h->dnorm = reinterpret_cast<sv::DiagNorm*>(base + o_dn);
  // everything starts at zero except the candidate slots, which start empty
  // (all bits set: token id -1); the finishing pass restores both after use
  if (cudaMemset(h->ws, 0, off) != cudaSuccess ||
      cudaMemset(h->cand, 0xFF, n_cand * sizeof(sv::Cand)) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return SV_ECUDA;
  }
  *out = h;
  return SV_OK;
}

}  // extern "C"

namespace {

// Whether a call may need the dense residual pass.  It does not when the call
// is greedy, or when every row is gated on the candidate fast path: uniform
// settings, or the handle's schedule, with every floor (the step's threshold
// or the cumulative floor, whichever is higher) above the fast path's bound.
// Per-sequence settings are device data: their presence counts as likely.
bool dense_residuals_likely(spec_verify_t h, float temperature, sv_gate gate_mode, float threshold,
                            const uint8_t* gate_mode_per_seq, const float* threshold_per_seq) {
  if (temperature == 0.f) return false;
  auto fast_floor = [&](float t) {
    return std::max(t, h->min_cum) * (1.0f - 1.0f / 1024.0f) * (sv::kTopM + 1) > 1.0f;
  };
  const bool has_sched = h->n_sched > 0;
  bool all_fast = gate_mode == SV_GATED_MU && !gate_mode_per_seq &&
                  (has_sched || (!threshold_per_seq && fast_floor(threshold)));
  for (int j = 0; has_sched && j < h->k; ++j)
    all_fast = all_fast && fast_floor(h->sched[j < h->n_sched ? j : h->n_sched - 1]);
  return !all_fast;
}

// The device address of page-locked host memory the device can read, or null
// (device memory, pageable or unknown memory)
const void* host_device_view(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Validate what every verifying call shares and fill the launch arguments
// (outputs and draws left empty).  SV_OK with *empty = true: nothing to do.
sv_status prepare_params(spec_verify_t h, const void* target_logits, sv_dtype tdt,
                         const void* draft_logits, sv_dtype ddt, const int32_t* draft_tokens, int B,
                         float temperature, sv_gate gate_mode, float threshold,
                         const uint8_t* gate_mode_per_seq, const float* threshold_per_seq,
                         sv::Params& P, bool* empty) {
  *empty = false;
  if (!h) return SV_EINVAL;
  if (B < 0 || B > h->max_B) return SV_EINVAL;
  if (!valid_dtype(tdt) || !valid_dtype(ddt)) return SV_EINVAL;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SV_EINVAL;
  if (gate_mode != SV_PLAIN && gate_mode != SV_GATED_MU) return SV_EINVAL;
  // a schedule replaces the sequences' thresholds, which then go unchecked
  const bool default_tau_used =
      (gate_mode == SV_GATED_MU || gate_mode_per_seq) && !threshold_per_seq && h->n_sched == 0;
  if (default_tau_used && !(threshold > 0.f && threshold <= 1.f)) return SV_EINVAL;
  if (B == 0) {
    *empty = true;
    return SV_OK;
  }
  if (!target_logits || !draft_logits || !draft_tokens) return SV_EINVAL;
  const int k = h->k, V = h->V;
  P = sv::Params{};
  P.Lt = target_logits;
  P.Ld = draft_logits;
  P.D = draft_tokens;
  P.B = B;
  P.k = k;
  P.V = V;
  P.nchunk = h->nchunk;
  P.rows = 2 * k + 1;
  const long long total = static_cast<long long>(B) * P.rows * h->nchunk;
  if (total >= (1ll << 31)) return SV_EUNSUPPORTED;
  P.total_chunks = static_cast<unsigned>(total);
  P.div_nchunk = sv::make_fastdiv(static_cast<unsigned>(h->nchunk));
  P.div_rows = sv::make_fastdiv(static_cast<unsigned>(P.rows));
  P.greedy = temperature == 0.f ? 1 : 0;
  P.c = P.greedy ? 0.f : static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  P.T = temperature;
  P.gate_default = gate_mode == SV_GATED_MU ? 1 : 0;
  P.tau_default = threshold;
  P.gate_per_seq = gate_mode_per_seq;
  P.tau_per_seq = threshold_per_seq;
  P.has_sched = h->n_sched > 0 ? 1 : 0;
  P.min_cum = h->min_cum;
  for (int j = 0; j < k; ++j)
    P.tau_step[j] = h->n_sched > 0 ? h->sched[j < h->n_sched ? j : h->n_sched - 1] : 0.f;
  P.part = h->part;
  P.xD = h->xD;
  P.cand = h->cand;
  P.cand_over = h->cand_over;
  const size_t row_t = static_cast<size_t>(V) * elem_size(tdt);
  const size_t row_d = static_cast<size_t>(V) * elem_size(ddt);
  P.vec_t = (row_t % 16 == 0) && (reinterpret_cast<uintptr_t>(target_logits) % 16 == 0);
  P.vec_d = (row_d % 16 == 0) && (reinterpret_cast<uintptr_t>(draft_logits) % 16 == 0);
  return SV_OK;
}

}  // namespace

extern "C" {

sv_status spec_verify_run_ex(spec_verify_t h, const void* target_logits, sv_dtype tdt,
                             const void* draft_logits, sv_dtype ddt, const int32_t* draft_tokens,
                             int B, float temperature, sv_gate gate_mode, float threshold,
                             const uint8_t* gate_mode_per_seq, const float* threshold_per_seq,
                             uint64_t seed, uint64_t seq_offset, const float* u_accept,
                             const float* u_residual, int32_t* accepted_len, int32_t* tokens,
                             float* accept_prob, int8_t* flags, uint64_t* counters,
                             float* row_stats, void* cuda_stream) {
  sv::Params P;
  bool empty = false;
  const sv_status ps = prepare_params(h, target_logits, tdt, draft_logits, ddt, draft_tokens, B,
                                      temperature, gate_mode, threshold, gate_mode_per_seq,
                                      threshold_per_seq, P, &empty);
  if (ps != SV_OK || empty) return ps;
  if (!accepted_len || !tokens || !accept_prob) return SV_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return SV_ECUDA;
  P.seed = seed;
  P.seq_offset = seq_offset;
  P.u0 = u_accept;
  P.u1 = u_residual;
  P.accepted_len = accepted_len;
  P.tokens = tokens;
  P.alpha = accept_prob;
  P.flags = flags;
  P.counters = reinterpret_cast<unsigned long long*>(counters);
  P.row_stats = row_stats;

  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int tb = tdt == SV_BF16, db = ddt == SV_BF16;
  const int bps = h->blocks_per_sm[tb][db] > 0 ? h->blocks_per_sm[tb][db] : 1;
  const bool dense_likely =
      dense_residuals_likely(h, temperature, gate_mode, threshold, gate_mode_per_seq, threshold_per_seq);
  // sampler filters (temperature > 0: a greedy call is one-hot already)
  const bool filtered = !P.greedy && (filter_on(h->filt[0]) || filter_on(h->filt[1]));
  const int mode = P.greedy ? sv::kModeGreedy
                            : (P.has_sched || P.min_cum > 0.f ? sv::kModePolicy : sv::kModeSample);
  return sv::pair_ops(tb, db).verify(h, P, mode, bps, dense_likely, filtered, st);
}

sv_status spec_verify_diagnostics(spec_verify_t h, const void* target_logits, sv_dtype tdt,
                                  const void* draft_logits, sv_dtype ddt,
                                  const int32_t* draft_tokens, int B, float temperature,
                                  sv_gate gate_mode, float threshold,
                                  const uint8_t* gate_mode_per_seq, const float* threshold_per_seq,
                                  float* min_sum, float* pq_sum, float* argmax_q, void* cuda_stream) {
  sv::Params P;
  bool empty = false;
  const sv_status ps = prepare_params(h, target_logits, tdt, draft_logits, ddt, draft_tokens, B,
                                      temperature, gate_mode, threshold, gate_mode_per_seq,
                                      threshold_per_seq, P, &empty);
  if (ps != SV_OK || empty) return ps;
  if (!min_sum && !pq_sum && !argmax_q) return SV_OK;
  if (!h->dnorm) return SV_EUNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return SV_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int tb = tdt == SV_BF16, db = ddt == SV_BF16;
  const int bps = h->blocks_per_sm[tb][db] > 0 ? h->blocks_per_sm[tb][db] : 1;
  const bool filtered = !P.greedy && (filter_on(h->filt[0]) || filter_on(h->filt[1]));
  return sv::pair_ops(tb, db).diagnostics(h, P, bps, filtered, min_sum, pq_sum, argmax_q, st);
}

sv_status spec_verify_run(spec_verify_t h, const void* target_logits, sv_dtype tdt,
                          const void* draft_logits, sv_dtype ddt, const int32_t* draft_tokens,
                          int B, float temperature, sv_gate gate_mode, float threshold,
                          const uint8_t* gate_mode_per_seq, const float* threshold_per_seq,
                          uint64_t seed, int32_t* accepted_len, int32_t* tokens,
                          float* accept_prob, int8_t* flags, uint64_t* counters,
                          void* cuda_stream) {
  return spec_verify_run_ex(h, target_logits, tdt, draft_logits, ddt, draft_tokens, B, temperature,
                            gate_mode, threshold, gate_mode_per_seq, threshold_per_seq, seed, 0,
                            nullptr, nullptr, accepted_len, tokens, accept_prob, flags, counters,
                            nullptr, cuda_stream);
}

sv_status spec_verify_run_host(spec_verify_t h, const void* target_logits, sv_dtype tdt,
                               const void* draft_logits, sv_dtype ddt, const int32_t* draft_tokens,
                               int B, float temperature, sv_gate gate_mode, float threshold,
                               const uint8_t* gate_mode_per_seq, const float* threshold_per_seq,
                               uint64_t seed, int32_t* accepted_len, int32_t* tokens,
                               float* accept_prob, int8_t* flags, uint64_t* counters,
                               void* cuda_stream) {
  if (!h) return SV_EINVAL;
  if (B < 0 || B > h->max_B || !valid_dtype(tdt) || !valid_dtype(ddt)) return SV_EINVAL;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !accepted_len || !tokens || !accept_prob)
    return SV_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return SV_ECUDA;
  const size_t k = h->k, V = h->V, mB = h->max_B;
  // staging layout sized for max_B and fp32 logits (the larger element type)
  size_t off = 0;
  const size_t o_t = off; off = align_up(off + mB * (k + 1) * V * 4, 256);
  const size_t o_d = off; off = align_up(off + mB * k * V * 4, 256);
  const size_t o_D = off; off = align_up(off + mB * k * 4, 256);
  const size_t o_g = off; off = align_up(off + mB, 256);
  const size_t o_tau = off; off = align_up(off + mB * 4, 256);
  const size_t o_al = off; off = align_up(off + mB * 4, 256);
  const size_t o_tok = off; off = align_up(off + mB * (k + 1) * 4, 256);
  const size_t o_ap = off; off = align_up(off + mB * k * 4, 256);
  const size_t o_fl = off; off = align_up(off + mB * k, 256);
  const size_t o_cnt = off; off = align_up(off + SV_NUM_COUNTERS * 8, 256);
  if (!h->stage) {
    if (cudaMalloc(&h->stage, off) != cudaSuccess) {
      h->stage = nullptr;
      return SV_ENOMEM;
    }
    h->stage_bytes = off;
  }
  char* s = static_cast<char*>(h->stage);
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const size_t bt = static_cast<size_t>(B) * (k + 1) * V * elem_size(tdt);
  const size_t bd = static_cast<size_t>(B) * k * V * elem_size(ddt);
  // Logits in page-locked host memory that the device can address are read
  // in place over the host link -- the kernels' own reads are the transfer --
  // when the call reads them about once (no dense residual pass, no sampler
  // filters); otherwise they are copied into the staging buffer first.  The
  // link's bandwidth is the same either way; in place, the copy no longer
  // precedes the verification as a separate step.
  const bool in_place = !filter_on(h->filt[0]) && !filter_on(h->filt[1]) &&
                        !dense_residuals_likely(h, temperature, gate_mode, threshold, gate_mode_per_seq,
                                                threshold_per_seq);
  const void* lt = in_place ? host_device_view(target_logits) : nullptr;
  const void* ld = in_place ? host_device_view(draft_logits) : nullptr;
  bool ok = true;
  if (!lt) {
    ok = ok && cudaMemcpyAsync(s + o_t, target_logits, bt, cudaMemcpyHostToDevice, st) == cudaSuccess;
    lt = s + o_t;
  }
  if (!ld) {
    ok = ok && cudaMemcpyAsync(s + o_d, draft_logits, bd, cudaMemcpyHostToDevice, st) == cudaSuccess;
    ld = s + o_d;
  }
  ok = ok && cudaMemcpyAsync(s + o_D, draft_tokens, static_cast<size_t>(B) * k * 4, cudaMemcpyHostToDevice, st) == cudaSuccess;
  if (gate_mode_per_seq)
    ok = ok && cudaMemcpyAsync(s + o_g, gate_mode_per_seq, static_cast<size_t>(B), cudaMemcpyHostToDevice, st) == cudaSuccess;
  if (threshold_per_seq)
    ok = ok && cudaMemcpyAsync(s + o_tau, threshold_per_seq, static_cast<size_t>(B) * 4, cudaMemcpyHostToDevice, st) == cudaSuccess;
  if (counters) ok = ok && cudaMemsetAsync(s + o_cnt, 0, SV_NUM_COUNTERS * 8, st) == cudaSuccess;
  if (!ok) return SV_ECUDA;
  sv_status rc = spec_verify_run_ex(
      h, lt, tdt, ld, ddt, reinterpret_cast<const int32_t*>(s + o_D), B, temperature,
      gate_mode, threshold, gate_mode_per_seq ? reinterpret_cast<const uint8_t*>(s + o_g) : nullptr,
      threshold_per_seq ? reinterpret_cast<const float*>(s + o_tau) : nullptr, seed, 0, nullptr,
      nullptr, reinterpret_cast<int32_t*>(s + o_al), reinterpret_cast<int32_t*>(s + o_tok),
      reinterpret_cast<float*>(s + o_ap), flags ? reinterpret_cast<int8_t*>(s + o_fl) : nullptr,
      counters ? reinterpret_cast<uint64_t*>(s + o_cnt) : nullptr, nullptr, cuda_stream);
  if (rc != SV_OK) return rc;
  ok = ok && cudaMemcpyAsync(accepted_len, s + o_al, static_cast<size_t>(B) * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(tokens, s + o_tok, static_cast<size_t>(B) * (k + 1) * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(accept_prob, s + o_ap, static_cast<size_t>(B) * k * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  if (flags) ok = ok && cudaMemcpyAsync(flags, s + o_fl, static_cast<size_t>(B) * k, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  if (counters) ok = ok && cudaMemcpyAsync(counters, s + o_cnt, SV_NUM_COUNTERS * 8, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
  return ok ? SV_OK : SV_ECUDA;
}

sv_status spec_verify_set_gate_policy(spec_verify_t h, const float* schedule, int n_schedule,
                                      float min_cum) {
  if (!h) return SV_EINVAL;
  if (schedule ? (n_schedule < 1 || n_schedule > SV_MAX_K) : n_schedule != 0) return SV_EINVAL;
  for (int j = 0; j < n_schedule; ++j)
    if (!(schedule[j] >= 0.f && schedule[j] <= 1.f)) return SV_EINVAL;
  if (!(min_cum >= 0.f && min_cum <= 1.f)) return SV_EINVAL;
  h->n_sched = n_schedule;
  for (int j = 0; j < SV_MAX_K; ++j) h->sched[j] = j < n_schedule ? schedule[j] : 0.f;
  h->min_cum = min_cum;
  return SV_OK;
}

sv_status spec_verify_set_filters(spec_verify_t h, int top_k_t, float top_p_t, float min_p_t, int top_k_d,
                                  float top_p_d, float min_p_d) {
  if (!h) return SV_EINVAL;
  const int kk[2] = {top_k_t, top_k_d};
  const float pp[2] = {top_p_t, top_p_d}, mm[2] = {min_p_t, min_p_d};
  for (int i = 0; i < 2; ++i)
    if (kk[i] < 0 || !(pp[i] > 0.f && pp[i] <= 1.f) || !(mm[i] >= 0.f && mm[i] <= 1.f)) return SV_EINVAL;
  for (int i = 0; i < 2; ++i) h->filt[i] = sv::Filter{kk[i], pp[i], mm[i]};
  return SV_OK;
}

sv_status spec_verify_free(spec_verify_t h) {
  if (!h) return SV_OK;
  sv_status rc = SV_OK;
  {
    DeviceGuard g(h->device);
    if (!g.ok || cudaDeviceSynchronize() != cudaSuccess) rc = SV_ECUDA;
    if (h->ws && cudaFree(h->ws) != cudaSuccess) rc = SV_ECUDA;
    if (h->stage && cudaFree(h->stage) != cudaSuccess) rc = SV_ECUDA;
    if (h->fbuf && cudaFree(h->fbuf) != cudaSuccess) rc = SV_ECUDA;
  }
  delete h;
  return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point (spec_verify_run_noalloc).
//
// For callers that may not allocate device memory at the point where they
// verify (device memory reserved up front by their own allocator, or no
// cudaMalloc / cudaFree between decode steps because those synchronise the
// device): the workspace lives in one static device buffer instead of a
// handle's allocation, and the call goes through the same validation and the
// same two launches as spec_verify_run_ex, on a handle built on the stack.
//
// Buffer layout (fixed, so that the candidate slots keep their empty marker
// from one call to the next whatever the shapes):
//   [0, 4 MiB)                  candidate slots, all bits set when empty
//   [4 MiB, 4 MiB + 64 KiB)     row-overflow flags, zero when clear
//   [4 MiB + 64 KiB, 8 MiB)     chunk statistics, then drafted-token logits
// The finishing pass empties every slot and clears every flag it reads, so a
// completed call leaves the buffer as set-up left it.  Calls on one device
// share the buffer and must not overlap.

namespace {

constexpr size_t kNaCandBytes = static_cast<size_t>(SV_NOALLOC_MAX_CAND_SLOTS) * sizeof(sv::Cand);
constexpr size_t kNaOverBytes = static_cast<size_t>(SV_NOALLOC_MAX_ROWS) * sizeof(unsigned);
static_assert(kNaCandBytes == (4u << 20), "candidate region is 4 MiB");
static_assert(kNaCandBytes + kNaOverBytes + SV_NOALLOC_STATS_BYTES == SV_NOALLOC_SCRATCH_BYTES,
              "scratch layout");

static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

struct NoallocDevice {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  int blocks_per_sm[2][2] = {{0, 0}, {0, 0}};
  int fin_spread_smem = 0;
};
constexpr int kNaMaxDevices = 64;
NoallocDevice g_na[kNaMaxDevices];
std::mutex g_na_mutex;

// once per device, with that device current: the buffer's address, the
// kernels' attributes, and the empty marker in every candidate slot
sv_status noalloc_setup(int dev, NoallocDevice** out) {
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoallocDevice& d = g_na[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SV_ECUDA;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SV_ECUDA;
    d.fin_spread_smem = sv::finish_spread_smem(dev);
    if (configure_all(d.blocks_per_sm, d.fin_spread_smem) != cudaSuccess) return SV_ECUDA;
    unsigned char* base = static_cast<unsigned char*>(p);
    // a set-up redone after a failed call: that call's kernels (if any ran)
    // are finished before the slots and flags are reset
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemset(base, 0xFF, kNaCandBytes) != cudaSuccess ||
        cudaMemset(base + kNaCandBytes, 0, kNaOverBytes) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return SV_ECUDA;
    d.base = base;
    d.ready = true;
  }
  *out = &d;
  return SV_OK;
}

}  // namespace

extern "C" sv_status spec_verify_run_noalloc(const void* target_logits, sv_dtype tdt,
                                             const void* draft_logits, sv_dtype ddt,
                                             const int32_t* draft_tokens, int B, int k, int V,
                                             float temperature, sv_gate gate_mode, float threshold,
                                             const uint8_t* gate_mode_per_seq,
                                             const float* threshold_per_seq, uint64_t seed,
                                             int32_t* accepted_len, int32_t* tokens,
                                             float* accept_prob, int8_t* flags, uint64_t* counters,
                                             void* cuda_stream) {
  if (B < 0 || k < 1 || V < 1) return SV_EINVAL;
  if (k > SV_MAX_K || V > SV_MAX_V) return SV_EUNSUPPORTED;
  // sizes against the fixed buffer, before anything touches the device
  const size_t nchunk = (static_cast<size_t>(V) + sv::kChunk - 1) / sv::kChunk;
  const size_t rows = 2 * static_cast<size_t>(k) + 1;
  const size_t slots = static_cast<size_t>(B) * k * nchunk * sv::kTopM;
  const size_t part_bytes = align_up(static_cast<size_t>(B) * rows * nchunk * sizeof(float2), 256);
  const size_t xd_bytes = align_up(static_cast<size_t>(B) * rows * sizeof(float), 256);
  if (slots > SV_NOALLOC_MAX_CAND_SLOTS || static_cast<size_t>(B) * k > SV_NOALLOC_MAX_ROWS ||
      part_bytes + xd_bytes > SV_NOALLOC_STATS_BYTES)
    return SV_EUNSUPPORTED;
  if (B == 0) return SV_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ECUDA;
  if (dev < 0 || dev >= kNaMaxDevices) return SV_EUNSUPPORTED;
  NoallocDevice* d = nullptr;
  const sv_status st = noalloc_setup(dev, &d);
  if (st != SV_OK) return st;

  // a handle on the stack whose workspace points into the buffer
  spec_verify_s h;
  h.device = dev;
  h.max_B = B;
  h.k = k;
  h.V = V;
  h.nchunk = static_cast<int>(nchunk);
  h.num_sms = d->num_sms;
  h.fin_spread_smem = d->fin_spread_smem;
  for (int a = 0; a < 2; ++a)
    for (int b = 0; b < 2; ++b) h.blocks_per_sm[a][b] = d->blocks_per_sm[a][b];
  h.cand = reinterpret_cast<sv::Cand*>(d->base);
  h.cand_over = reinterpret_cast<unsigned*>(d->base + kNaCandBytes);
  h.part = reinterpret_cast<float2*>(d->base + kNaCandBytes + kNaOverBytes);
  h.xD = reinterpret_cast<float*>(d->base + kNaCandBytes + kNaOverBytes + part_bytes);
  const sv_status rc = spec_verify_run_ex(&h, target_logits, tdt, draft_logits, ddt, draft_tokens, B,
                                          temperature, gate_mode, threshold, gate_mode_per_seq,
                                          threshold_per_seq, seed, 0, nullptr, nullptr, accepted_len,
                                          tokens, accept_prob, flags, counters, nullptr, cuda_stream);
  if (rc == SV_ECUDA) {
    // a launch failed, possibly after the stream pass had written candidate
    // slots that no finishing pass will empty: the next call sets up again
    std::lock_guard<std::mutex> lock(g_na_mutex);
    d->ready = false;
  }
  return rc;
}
