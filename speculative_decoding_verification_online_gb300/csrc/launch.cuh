// Launch sequences of the library's calls, as templates over the (target,
// draft) logits types.  Included only by the pair_*.cu translation units, each
// of which instantiates them for one pair (see handle.h).
#pragma once

#include "handle.h"

namespace sv {
namespace {

constexpr int kFinCluster = 4;  // CTAs sharing a sequence's dense residual
constexpr int kFinWarm = 2;     // warming CTAs of a single-CTA finishing grid

// every warp of a stream CTA owns a ring of kDepth chunk stages
template <typename TT, typename TD>
constexpr int dyn_smem() {
  return Stages<TT, TD>::kWarpsPerCta * Stages<TT, TD>::kDepth * Stages<TT, TD>::kBytes;
}

// opt the kernel into its dynamic shared memory and ask how many CTAs fit on an SM
template <typename TT, typename TD>
constexpr int pair_smem() {
  return PairStages<TT, TD>::kWarpsPerCta * PairStages<TT, TD>::kDepth *
         PairStages<TT, TD>::kBytes;
}

template <typename TT, typename TD, int G, bool kFilt>
cudaError_t configure_one(int fin_spread_smem) {
  cudaError_t e = cudaFuncSetAttribute(stream_kernel<TT, TD, G, kFilt>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<TT, TD>());
  if (e != cudaSuccess) return e;
  const int fin = static_cast<int>(sizeof(FinishShared));
  const int fin_max = fin_spread_smem > fin ? fin_spread_smem : fin;
  e = cudaFuncSetAttribute(finish_kernel<TT, TD, G, false, kFilt>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           fin_max);
  if (e != cudaSuccess || G == kModeGreedy) return e;
  return cudaFuncSetAttribute(finish_kernel<TT, TD, G, G != kModeGreedy, kFilt>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, fin_max);
}

// every variant (sampling, sampling with a gate policy, greedy) of a dtype
// pair: opt the kernels into their dynamic shared memory and ask how many
// stream CTAs fit on an SM
template <typename TT, typename TD>
cudaError_t configure(int* blocks_per_sm, int fin_spread_smem) {
  cudaError_t e = configure_one<TT, TD, kModeSample, false>(fin_spread_smem);
  if (e == cudaSuccess) e = configure_one<TT, TD, kModePolicy, false>(fin_spread_smem);
  if (e == cudaSuccess) e = configure_one<TT, TD, kModeGreedy, false>(fin_spread_smem);
  if (e == cudaSuccess) e = configure_one<TT, TD, kModeSample, true>(fin_spread_smem);
  if (e == cudaSuccess) e = configure_one<TT, TD, kModePolicy, true>(fin_spread_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_kernel<TT, TD, kModeStats, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<TT, TD>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_kernel<TT, TD, kModeGather, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<TT, TD>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_kernel<TT, TD, kModeStats, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<TT, TD>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pair_kernel<TT, TD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair_smem<TT, TD>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pair_kernel<TT, TD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair_smem<TT, TD>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(select_kernel<TT, TD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(SelShared)));
  // several histogram CTAs per SM need the largest shared-memory split
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(hist_kernel<TT, TD>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm,
                                                       stream_kernel<TT, TD, kModeSample, false>,
                                                       Stages<TT, TD>::kThreadsPerCta,
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

// the stream pass (variant G; kFilt: the sampler filters applied as chunks
// load), with the handle's one-shot timing marks around it
template <typename TT, typename TD, int G, bool kFilt>
sv_status launch_stream(spec_verify_t h, const Params& P, int blocks_per_sm, cudaStream_t st) {
  long long grid = static_cast<long long>(h->num_sms) * blocks_per_sm;
  // a warp takes whole chunks, so more than total_chunks / warps-per-CTA CTAs idle
  const long long need = (static_cast<long long>(P.total_chunks) + Stages<TT, TD>::kWarpsPerCta - 1) /
                         Stages<TT, TD>::kWarpsPerCta;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  const bool marked = h->mark_before != nullptr;
  if (marked && cudaEventRecord(h->mark_before, st) != cudaSuccess) return SV_ECUDA;
  // a programmatic dependent launch: resident early, it waits for the previous
  // kernel in the stream before touching memory
  if (launch_dependent(stream_kernel<TT, TD, G, kFilt>, static_cast<unsigned>(grid),
                       Stages<TT, TD>::kThreadsPerCta, dyn_smem<TT, TD>(), st, P) != cudaSuccess)
    return SV_ECUDA;
  if (cudaGetLastError() != cudaSuccess) return SV_ECUDA;
  if (marked) {
    const cudaError_t e = cudaEventRecord(h->mark_after, st);
    h->mark_before = h->mark_after = nullptr;
    if (e != cudaSuccess) return SV_ECUDA;
  }
  return SV_OK;
}

template <typename TT, typename TD, int G, bool kFilt>
sv_status launch(spec_verify_t h, const Params& P, int blocks_per_sm, bool dense_likely,
                 cudaStream_t st) {
  const sv_status rs = launch_stream<TT, TD, G, kFilt>(h, P, blocks_per_sm, st);
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
  Params Pf = P;
  Pf.fin_warm = csize == 1 && clusters + kFinWarm <= 2 * h->num_sms ? kFinWarm : 0;
  const int grid = clusters * csize + Pf.fin_warm;
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kFinThreads);
  // a grid that fits one CTA per SM gets it (finish_spread_smem)
  cfg.dynamicSmemBytes = h->fin_spread_smem > 0 && grid <= h->num_sms
                             ? static_cast<size_t>(h->fin_spread_smem)
                             : sizeof(FinishShared);
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
  if (G != kModeGreedy && dense_likely)
    e = cudaLaunchKernelEx(&cfg, finish_kernel<TT, TD, G, G != kModeGreedy, kFilt>, Pf);
  else
    e = cudaLaunchKernelEx(&cfg, finish_kernel<TT, TD, G, false, kFilt>, Pf);
  if (e != cudaSuccess) return SV_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

// the acceptance diagnostics: the stream pass, the per-position merge, and
// (temperature > 0) the pair sweep and its reduction, each launch a
// programmatic dependent of the one before (kFilt: the rows as the sampler
// filters leave them, applied as logits load)
template <typename TT, typename TD, bool kGreedy, bool kFilt>
sv_status launch_diag(spec_verify_t h, const Params& P, int blocks_per_sm, float* min_sum,
                      float* pq_sum, float* argmax_q, cudaStream_t st) {
  static_assert(!(kGreedy && kFilt), "a greedy call is one-hot already");
  const sv_status rs = launch_stream<TT, TD, kGreedy ? kModeGreedy : kModeStats, kFilt>(h, P, blocks_per_sm, st);
  if (rs != SV_OK) return rs;
  const unsigned npos = static_cast<unsigned>(P.B * P.k);
  const unsigned small_grid = (npos + kDiagWarps - 1) / kDiagWarps;
  if (launch_dependent(diag_norm_kernel<kGreedy>, small_grid, kDiagThreads, 0, st, P, h->dnorm,
                       min_sum, pq_sum, argmax_q) != cudaSuccess)
    return SV_ECUDA;
  if (!kGreedy) {
    const unsigned total = npos * static_cast<unsigned>(P.nchunk);
    constexpr int kW = PairStages<TT, TD>::kWarpsPerCta;
    long long grid = h->num_sms;
    const long long need = (static_cast<long long>(total) + kW - 1) / kW;
    if (grid > need) grid = need;
    if (launch_dependent(pair_kernel<TT, TD, kFilt>, static_cast<unsigned>(grid),
                         PairStages<TT, TD>::kThreadsPerCta, pair_smem<TT, TD>(), st, P,
                         static_cast<const DiagNorm*>(h->dnorm), total) != cudaSuccess)
      return SV_ECUDA;
    if (launch_dependent(diag_reduce_kernel<TT, TD>, small_grid, kDiagThreads, 0, st, P,
                         static_cast<const DiagNorm*>(h->dnorm), min_sum, pq_sum, argmax_q) != cudaSuccess)
      return SV_ECUDA;
  }
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

// The selection after the statistics pass: top-k rows' bounds, the gathering
// pass and the short lists' selection when a side gathers, then select_kernel
// (every row not selected before).  gc, gl, done: the gathering buffers.
template <typename TT, typename TD>
sv_status launch_selection(spec_verify_t h, const Params& P, FilterParams& F, int blocks_per_sm, char* gc,
                           char* gl, char* done, cudaStream_t st) {
  const unsigned nrows = static_cast<unsigned>(P.B * P.rows);
  if (gathers_row(F.f[0], P.nchunk) || gathers_row(F.f[1], P.nchunk)) {
    // top-k rows: each row's lower bound from its chunk maxima, then the
    // gathering pass keeps every logit at or above it, chunk by chunk
    if (launch_dependent(bound_kernel<TT, TD>, (nrows + kBoundWarps - 1) / kBoundWarps, 32 * kBoundWarps, 0, st,
                         P, F) != cudaSuccess)
      return SV_ECUDA;
    Params Pg = P;
    Pg.fthr = F.gbound;  // the gathering pass takes each row's bound in the threshold slot
    Pg.ffirst = F.first;
    Pg.gcount = reinterpret_cast<unsigned*>(gc);
    Pg.glist = reinterpret_cast<float*>(gl);
    const sv_status rs = launch_stream<TT, TD, kModeGather, true>(h, Pg, blocks_per_sm, st);
    if (rs != SV_OK) return rs;
    F.gcount = Pg.gcount;
    F.glist = Pg.glist;
    // gathered rows whose lists are short: selected by a small CTA each
    F.done = reinterpret_cast<int*>(done);
    if (launch_dependent(list_select_kernel<TT, TD>, nrows, kLSelThreads, 0, st, P, F) != cudaSuccess)
      return SV_ECUDA;
  }
  if (launch_dependent(select_kernel<TT, TD>, nrows, kSelThreads, sizeof(SelShared), st, P, F) !=
      cudaSuccess)
    return SV_ECUDA;
  return SV_OK;
}

// The filter prefix of a call: each row's kept set (a threshold and, for
// top_k = 1, the kept index).  When every filtered side holds bf16 logits and
// none is top_k = 1, hist_kernel finds it from one read of each row;
// otherwise the statistics pass of the raw rows, then (top-k rows) the
// gathering passes, then select_kernel.  The call's kernels then apply them on
// the fly (P.fthr, P.ffirst: every logit outside a row's kept set reads as
// -inf).
template <typename TT, typename TD>
sv_status launch_filters(spec_verify_t h, Params& P, int blocks_per_sm, cudaStream_t st) {
  const size_t rows_all = static_cast<size_t>(h->max_B) * (2 * h->k + 1);
  const size_t chunks_all = rows_all * h->nchunk;
  const size_t o_key = 0, o_first = align_up(rows_all * sizeof(unsigned), 256);
  const size_t o_thr = align_up(o_first + rows_all * sizeof(int), 256);
  const size_t o_gb = align_up(o_thr + rows_all * sizeof(float), 256);
  const size_t o_gc = align_up(o_gb + rows_all * sizeof(float), 256);
  const size_t o_gl = align_up(o_gc + chunks_all * sizeof(unsigned), 256);
  const size_t o_done = align_up(o_gl + chunks_all * kGatherCap * sizeof(float), 256);
  const size_t need = align_up(o_done + rows_all * sizeof(int), 256);
  if (!h->fbuf) {
    if (cudaMalloc(&h->fbuf, need) != cudaSuccess) {
      h->fbuf = nullptr;
      return SV_ENOMEM;
    }
    h->fbuf_bytes = need;
  }
  char* base = static_cast<char*>(h->fbuf);
  FilterParams F;
  F.f[0] = h->filt[0];
  F.f[1] = h->filt[1];
  F.key = reinterpret_cast<unsigned*>(base + o_key);
  F.first = reinterpret_cast<int*>(base + o_first);
  F.thr = reinterpret_cast<float*>(base + o_thr);
  F.gbound = reinterpret_cast<float*>(base + o_gb);
  F.gcount = nullptr;
  F.glist = nullptr;
  F.done = nullptr;
  const unsigned nrows = static_cast<unsigned>(P.B * P.rows);
  if (hist_selects(F.f[0], sizeof(TT) == 2) && hist_selects(F.f[1], sizeof(TD) == 2)) {
    if (launch_dependent(hist_kernel<TT, TD>, nrows, kHThreads, 0, st, P, F) != cudaSuccess) return SV_ECUDA;
  } else {
    sv_status rs = launch_stream<TT, TD, kModeStats, false>(h, P, blocks_per_sm, st);
    if (rs != SV_OK) return rs;
    rs = launch_selection<TT, TD>(h, P, F, blocks_per_sm, base + o_gc, base + o_gl, base + o_done, st);
    if (rs != SV_OK) return rs;
  }
  P.fthr = F.thr;
  P.ffirst = F.first;
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}


// one verifying call: the sampler filters' prefix when asked for, then the
// stream pass and the finishing pass of the variant
template <typename TT, typename TD>
sv_status verify_pair(spec_verify_t h, Params& P, int mode, int bps, bool dense_likely, bool filtered,
                      cudaStream_t st) {
  if (mode == kModeGreedy) return launch<TT, TD, kModeGreedy, false>(h, P, bps, false, st);
  if (filtered) {
    const sv_status rs = launch_filters<TT, TD>(h, P, bps, st);
    if (rs != SV_OK) return rs;
    if (mode == kModePolicy) return launch<TT, TD, kModePolicy, true>(h, P, bps, dense_likely, st);
    return launch<TT, TD, kModeSample, true>(h, P, bps, dense_likely, st);
  }
  if (mode == kModePolicy) return launch<TT, TD, kModePolicy, false>(h, P, bps, dense_likely, st);
  return launch<TT, TD, kModeSample, false>(h, P, bps, dense_likely, st);
}

// the acceptance diagnostics, after the sampler filters' prefix when asked for
template <typename TT, typename TD>
sv_status diag_pair(spec_verify_t h, Params& P, int bps, bool filtered, float* min_sum, float* pq_sum,
                    float* argmax_q, cudaStream_t st) {
  if (P.greedy) return launch_diag<TT, TD, true, false>(h, P, bps, min_sum, pq_sum, argmax_q, st);
  if (filtered) {
    const sv_status rs = launch_filters<TT, TD>(h, P, bps, st);
    if (rs != SV_OK) return rs;
    return launch_diag<TT, TD, false, true>(h, P, bps, min_sum, pq_sum, argmax_q, st);
  }
  return launch_diag<TT, TD, false, false>(h, P, bps, min_sum, pq_sum, argmax_q, st);
}

}  // namespace

template <typename TT, typename TD>
constexpr PairOps make_ops() {
  return PairOps{&configure<TT, TD>, &verify_pair<TT, TD>, &diag_pair<TT, TD>};
}

}  // namespace sv
