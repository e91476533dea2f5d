// Host side of the C ABI declared in include/spec_verify.h: handle and
// workspace management, argument validation, and the two launches of a call
// (the stream pass, then the finishing pass as a programmatic dependent launch).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "spec_verify.h"
#include "verify_kernel.cuh"
#include "diag_kernel.cuh"
#include "filter_kernel.cuh"

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
  // sampler filters (spec_verify_set_filters) and their buffers, allocated on
  // the first filtered call: masked copies of the logits, per-row thresholds
  sv::Filter filt[2] = {{0, 1.f, 0.f}, {0, 1.f, 0.f}};
  void* fbuf = nullptr;
  size_t fbuf_bytes = 0;
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t elem_size(sv_dtype d) { return d == SV_BF16 ? 2 : 4; }

constexpr int kFinCluster = 4;  // CTAs sharing a sequence's dense residual
constexpr int kFinWarm = 2;     // warming CTAs of a single-CTA finishing grid

bool valid_dtype(int d) { return d == SV_F32 || d == SV_BF16; }

// every warp of a stream CTA owns a ring of kDepth chunk stages
template <typename TT, typename TD>
constexpr int dyn_smem() {
  return sv::Stages<TT, TD>::kWarpsPerCta * sv::Stages<TT, TD>::kDepth * sv::Stages<TT, TD>::kBytes;
}

// opt the kernel into its dynamic shared memory and ask how many CTAs fit on an SM
template <typename TT, typename TD>
constexpr int pair_smem() {
  return sv::PairStages<TT, TD>::kWarpsPerCta * sv::PairStages<TT, TD>::kDepth *
         sv::PairStages<TT, TD>::kBytes;
}

// Dynamic shared memory for a finishing CTA that is to have its SM to itself:
// just over half of an SM's shared memory, or 0 where the device cannot give
// that much to one CTA.  Two finishing CTAs on one SM slow each other's
// dependent chains (measured: about 1 us per call on the 128K-vocabulary
// batch), so a grid that fits one CTA per SM asks for this much.
int finish_spread_smem(int device) {
  int per_sm = 0, optin = 0;
  if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
    return 0;
  const int want = per_sm / 2 + 1024;
  return want <= optin && want > static_cast<int>(sizeof(sv::FinishShared)) ? want : 0;
}

template <typename TT, typename TD, int G>
cudaError_t configure_one(int fin_spread_smem) {
  cudaError_t e = cudaFuncSetAttribute(sv::stream_kernel<TT, TD, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<TT, TD>());
  if (e != cudaSuccess) return e;
  const int fin = static_cast<int>(sizeof(sv::FinishShared));
  const int fin_max = fin_spread_smem > fin ? fin_spread_smem : fin;
  e = cudaFuncSetAttribute(sv::finish_kernel<TT, TD, G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           fin_max);
  if (e != cudaSuccess || G == sv::kModeGreedy) return e;
  return cudaFuncSetAttribute(sv::finish_kernel<TT, TD, G, G != sv::kModeGreedy>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, fin_max);
}

// every variant (sampling, sampling with a gate policy, greedy) of a dtype
// pair: opt the kernels into their dynamic shared memory and ask how many
// stream CTAs fit on an SM
template <typename TT, typename TD>
cudaError_t configure(int* blocks_per_sm, int fin_spread_smem) {
  cudaError_t e = configure_one<TT, TD, sv::kModeSample>(fin_spread_smem);
  if (e == cudaSuccess) e = configure_one<TT, TD, sv::kModePolicy>(fin_spread_smem);
  if (e == cudaSuccess) e = configure_one<TT, TD, sv::kModeGreedy>(fin_spread_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sv::stream_kernel<TT, TD, sv::kModeStats>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<TT, TD>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sv::pair_kernel<TT, TD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair_smem<TT, TD>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sv::select_kernel<TT, TD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(sv::SelShared)));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm,
                                                       sv::stream_kernel<TT, TD, sv::kModeSample>,
                                                       sv::Stages<TT, TD>::kThreadsPerCta,
                                                       dyn_smem<TT, TD>());
}

// a programmatic dependent launch: the kernel may become resident while the
// previous kernel in the stream drains (it calls griddepcontrol.wait before it
// reads what that kernel writes)
template <typename K, typename... A>
cudaError_t launch_dependent(K kernel, unsigned grid, unsigned threads, size_t smem, cudaStream_t st,
                             A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// the stream pass (variant G), with the handle's one-shot timing marks around it
template <typename TT, typename TD, int G>
sv_status launch_stream(spec_verify_t h, const sv::Params& P, int blocks_per_sm, cudaStream_t st) {
  long long grid = static_cast<long long>(h->num_sms) * blocks_per_sm;
  // a warp takes whole chunks, so more than total_chunks / warps-per-CTA CTAs idle
  const long long need = (static_cast<long long>(P.total_chunks) + sv::Stages<TT, TD>::kWarpsPerCta - 1) /
                         sv::Stages<TT, TD>::kWarpsPerCta;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  const bool marked = h->mark_before != nullptr;
  if (marked && cudaEventRecord(h->mark_before, st) != cudaSuccess) return SV_ECUDA;
  // a programmatic dependent launch: resident early, it waits for the previous
  // kernel in the stream before touching memory
  if (launch_dependent(sv::stream_kernel<TT, TD, G>, static_cast<unsigned>(grid),
                       sv::Stages<TT, TD>::kThreadsPerCta, dyn_smem<TT, TD>(), st, P) != cudaSuccess)
    return SV_ECUDA;
  if (cudaGetLastError() != cudaSuccess) return SV_ECUDA;
  if (marked) {
    const cudaError_t e = cudaEventRecord(h->mark_after, st);
    h->mark_before = h->mark_after = nullptr;
    if (e != cudaSuccess) return SV_ECUDA;
  }
  return SV_OK;
}

template <typename TT, typename TD, int G>
sv_status launch(spec_verify_t h, const sv::Params& P, int blocks_per_sm, bool dense_likely,
                 cudaStream_t st) {
  const sv_status rs = launch_stream<TT, TD, G>(h, P, blocks_per_sm, st);
  if (rs != SV_OK) return rs;
  // the finishing pass: one CTA per sequence, allowed to launch while the
  // stream pass drains; it waits (griddepcontrol.wait) before reading its output
  cudaLaunchConfig_t cfg = {};
  // a cluster of CTAs per sequence at a time (two CTAs per SM at most; larger
  // batches loop).  When dense residuals are likely (plain rows, or gated rows
  // off the candidate fast path) and the whole batch fits at once, clusters of
  // up to kFinCluster CTAs share the re-read of the stop row pair; otherwise
  // one CTA per sequence (more sequences in flight beats wider sequences)
  int csize = 1;
  if (dense_likely)
    for (int c = kFinCluster; c > 1; c /= 2)
      if (static_cast<long long>(P.B) * c <= 2ll * h->num_sms) {
        csize = c;
        break;
      }
  const int max_clusters = 2 * h->num_sms / csize;
  const int clusters = P.B < max_clusters ? P.B : max_clusters;
  // warming CTAs in front of single-CTA clusters, while every CTA still has
  // an SM slot at once (two per SM)
  sv::Params Pf = P;
  Pf.fin_warm = csize == 1 && clusters + kFinWarm <= 2 * h->num_sms ? kFinWarm : 0;
  const int grid = clusters * csize + Pf.fin_warm;
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(sv::kFinThreads);
  // a grid that fits one CTA per SM gets it (finish_spread_smem)
  cfg.dynamicSmemBytes = h->fin_spread_smem > 0 && grid <= h->num_sms
                             ? static_cast<size_t>(h->fin_spread_smem)
                             : sizeof(sv::FinishShared);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(csize);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = csize > 1 ? 2 : 1;
  // the finishing kernel with the dense pass (clusters) when dense residuals
  // are likely; otherwise the one without it (greedy calls never need it)
  cudaError_t e;
  if (G != sv::kModeGreedy && dense_likely)
    e = cudaLaunchKernelEx(&cfg, sv::finish_kernel<TT, TD, G, G != sv::kModeGreedy>, Pf);
  else
    e = cudaLaunchKernelEx(&cfg, sv::finish_kernel<TT, TD, G, false>, Pf);
  if (e != cudaSuccess) return SV_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

// the kernel variant G for the call's logits types (tb / db: bf16)
template <int G>
sv_status launch_mode(spec_verify_t h, const sv::Params& P, int bps, bool dense_likely, bool tb, bool db,
                      cudaStream_t st) {
  if (tb && db) return launch<uint16_t, uint16_t, G>(h, P, bps, dense_likely, st);
  if (tb && !db) return launch<uint16_t, float, G>(h, P, bps, dense_likely, st);
  if (!tb && db) return launch<float, uint16_t, G>(h, P, bps, dense_likely, st);
  return launch<float, float, G>(h, P, bps, dense_likely, st);
}


// the acceptance diagnostics: the stream pass, the per-position merge, and
// (temperature > 0) the pair sweep and its reduction, each launch a
// programmatic dependent of the one before
template <typename TT, typename TD, bool kGreedy>
sv_status launch_diag(spec_verify_t h, const sv::Params& P, int blocks_per_sm, float* min_sum,
                      float* pq_sum, float* argmax_q, cudaStream_t st) {
  const sv_status rs = launch_stream<TT, TD, kGreedy ? sv::kModeGreedy : sv::kModeStats>(h, P, blocks_per_sm, st);
  if (rs != SV_OK) return rs;
  const unsigned npos = static_cast<unsigned>(P.B * P.k);
  const unsigned small_grid = (npos + sv::kDiagWarps - 1) / sv::kDiagWarps;
  if (launch_dependent(sv::diag_norm_kernel<kGreedy>, small_grid, sv::kDiagThreads, 0, st, P, h->dnorm,
                       min_sum, pq_sum, argmax_q) != cudaSuccess)
    return SV_ECUDA;
  if (!kGreedy) {
    const unsigned total = npos * static_cast<unsigned>(P.nchunk);
    constexpr int kW = sv::PairStages<TT, TD>::kWarpsPerCta;
    long long grid = h->num_sms;
    const long long need = (static_cast<long long>(total) + kW - 1) / kW;
    if (grid > need) grid = need;
    if (launch_dependent(sv::pair_kernel<TT, TD>, static_cast<unsigned>(grid),
                         sv::PairStages<TT, TD>::kThreadsPerCta, pair_smem<TT, TD>(), st, P,
                         static_cast<const sv::DiagNorm*>(h->dnorm), total) != cudaSuccess)
      return SV_ECUDA;
    if (launch_dependent(sv::diag_reduce_kernel<TD>, small_grid, sv::kDiagThreads, 0, st, P,
                         static_cast<const sv::DiagNorm*>(h->dnorm), min_sum, pq_sum, argmax_q) != cudaSuccess)
      return SV_ECUDA;
  }
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

bool filter_on(const sv::Filter& f) { return f.top_k != 0 || f.top_p < 1.f || f.min_p > 0.f; }

// the filter prefix of a call: statistics pass, per-row thresholds, masked
// copies; on return P reads the masked copies
template <typename TT, typename TD>
sv_status launch_filters(spec_verify_t h, sv::Params& P, int blocks_per_sm, cudaStream_t st) {
  const size_t rows_all = static_cast<size_t>(h->max_B) * (2 * h->k + 1);
  const size_t bt = static_cast<size_t>(h->max_B) * (h->k + 1) * h->V * sizeof(float);
  const size_t bd = static_cast<size_t>(h->max_B) * h->k * h->V * sizeof(float);
  const size_t o_t = 0, o_d = align_up(bt, 256), o_key = align_up(o_d + bd, 256);
  const size_t o_first = align_up(o_key + rows_all * sizeof(unsigned), 256);
  const size_t need = align_up(o_first + rows_all * sizeof(int), 256);
  if (!h->fbuf) {
    if (cudaMalloc(&h->fbuf, need) != cudaSuccess) {
      h->fbuf = nullptr;
      return SV_ENOMEM;
    }
    h->fbuf_bytes = need;
  }
  char* base = static_cast<char*>(h->fbuf);
  sv::FilterParams F;
  F.f[0] = h->filt[0];
  F.f[1] = h->filt[1];
  F.key = reinterpret_cast<unsigned*>(base + o_key);
  F.first = reinterpret_cast<int*>(base + o_first);
  F.Lt_m = base + o_t;
  F.Ld_m = base + o_d;
  sv_status rs = launch_stream<TT, TD, sv::kModeStats>(h, P, blocks_per_sm, st);
  if (rs != SV_OK) return rs;
  const unsigned nrows = static_cast<unsigned>(P.B * P.rows);
  if (launch_dependent(sv::select_kernel<TT, TD>, nrows, sv::kSelThreads, sizeof(sv::SelShared), st, P, F) !=
      cudaSuccess)
    return SV_ECUDA;
  // one CTA per row at a time, at most eight per SM
  long long grid = static_cast<long long>(P.B) * P.rows;
  if (grid > 8ll * h->num_sms) grid = 8ll * h->num_sms;
  if (grid < 1) grid = 1;
  if (launch_dependent(sv::mask_kernel<TT, TD>, static_cast<unsigned>(grid), static_cast<unsigned>(sv::kMaskThreads),
                       0, st, P, F) != cudaSuccess)
    return SV_ECUDA;
  P.Lt = F.Lt_m;
  P.Ld = F.Ld_m;
  P.vec_t = (static_cast<size_t>(P.V) * sizeof(TT)) % 16 == 0;
  P.vec_d = (static_cast<size_t>(P.V) * sizeof(TD)) % 16 == 0;
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

template <int G>
sv_status launch_mode_filtered(spec_verify_t h, sv::Params& P, int bps, bool dense_likely, bool tb, bool db,
                               cudaStream_t st) {
  sv_status rs;
  if (tb && db) rs = launch_filters<uint16_t, uint16_t>(h, P, bps, st);
  else if (tb && !db) rs = launch_filters<uint16_t, float>(h, P, bps, st);
  else if (!tb && db) rs = launch_filters<float, uint16_t>(h, P, bps, st);
  else rs = launch_filters<float, float>(h, P, bps, st);
  if (rs != SV_OK) return rs;
  return launch_mode<G>(h, P, bps, dense_likely, tb, db, st);
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

int spec_verify_launches_per_filtered_run(void) { return 5; }

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
  h->fin_spread_smem = finish_spread_smem(device);
  cudaError_t e = configure<float, float>(&h->blocks_per_sm[0][0], h->fin_spread_smem);
  if (e == cudaSuccess) e = configure<float, uint16_t>(&h->blocks_per_sm[0][1], h->fin_spread_smem);
  if (e == cudaSuccess) e = configure<uint16_t, float>(&h->blocks_per_sm[1][0], h->fin_spread_smem);
  if (e == cudaSuccess) e = configure<uint16_t, uint16_t>(&h->blocks_per_sm[1][1], h->fin_spread_smem);
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
  if (!P.greedy && (filter_on(h->filt[0]) || filter_on(h->filt[1]))) {
    if (P.has_sched || P.min_cum > 0.f)
      return launch_mode_filtered<sv::kModePolicy>(h, P, bps, dense_likely, tb, db, st);
    return launch_mode_filtered<sv::kModeSample>(h, P, bps, dense_likely, tb, db, st);
  }
  if (P.greedy) return launch_mode<sv::kModeGreedy>(h, P, bps, false, tb, db, st);
  if (P.has_sched || P.min_cum > 0.f) return launch_mode<sv::kModePolicy>(h, P, bps, dense_likely, tb, db, st);
  return launch_mode<sv::kModeSample>(h, P, bps, dense_likely, tb, db, st);
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
  if (!P.greedy && (filter_on(h->filt[0]) || filter_on(h->filt[1]))) {
    sv_status rs;
    if (tb && db) rs = launch_filters<uint16_t, uint16_t>(h, P, bps, st);
    else if (tb && !db) rs = launch_filters<uint16_t, float>(h, P, bps, st);
    else if (!tb && db) rs = launch_filters<float, uint16_t>(h, P, bps, st);
    else rs = launch_filters<float, float>(h, P, bps, st);
    if (rs != SV_OK) return rs;
  }
  if (P.greedy) {
    if (tb && db) return launch_diag<uint16_t, uint16_t, true>(h, P, bps, min_sum, pq_sum, argmax_q, st);
    if (tb && !db) return launch_diag<uint16_t, float, true>(h, P, bps, min_sum, pq_sum, argmax_q, st);
    if (!tb && db) return launch_diag<float, uint16_t, true>(h, P, bps, min_sum, pq_sum, argmax_q, st);
    return launch_diag<float, float, true>(h, P, bps, min_sum, pq_sum, argmax_q, st);
  }
  if (tb && db) return launch_diag<uint16_t, uint16_t, false>(h, P, bps, min_sum, pq_sum, argmax_q, st);
  if (tb && !db) return launch_diag<uint16_t, float, false>(h, P, bps, min_sum, pq_sum, argmax_q, st);
  if (!tb && db) return launch_diag<float, uint16_t, false>(h, P, bps, min_sum, pq_sum, argmax_q, st);
  return launch_diag<float, float, false>(h, P, bps, min_sum, pq_sum, argmax_q, st);
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
    d.fin_spread_smem = finish_spread_smem(dev);
    cudaError_t e = configure<float, float>(&d.blocks_per_sm[0][0], d.fin_spread_smem);
    if (e == cudaSuccess) e = configure<float, uint16_t>(&d.blocks_per_sm[0][1], d.fin_spread_smem);
    if (e == cudaSuccess) e = configure<uint16_t, float>(&d.blocks_per_sm[1][0], d.fin_spread_smem);
    if (e == cudaSuccess) e = configure<uint16_t, uint16_t>(&d.blocks_per_sm[1][1], d.fin_spread_smem);
    if (e != cudaSuccess) return SV_ECUDA;
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
