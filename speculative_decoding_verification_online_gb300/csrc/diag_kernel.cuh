// diag_kernel.cuh -- closed-form acceptance diagnostics of every draft
// position (mlxcel PR #992, "The acceptance ceiling"): for a draft drawn from
// q_j, modified rejection sampling accepts with probability
// sum_x min(p_j(x), mu_j(x)) (plain mode: the maximal-coupling bound
// 1 - TV(p_j, q_j)), sampler-match with sum_x p_j(x) q_j(x), and the argmax
// rule with q_j(argmax p_j).  mu_j is the gate's retained measure (Strata PR
// #3416, "Approach") with the handle's policy (regolith audit, "schedule
// behavior"); the cumulative floor uses the drafted prefix D_0..D_{j-1}.
//
// min(p, mu) needs both rows' normalisers before any term can be formed, so
// the diagnostics read the rows twice.  With sampler filters every row's kept
// set comes first (as for a verifying call) and launches 1, 3 and 4 read every
// logit outside it as -inf.  Launches, each a programmatic dependent of the
// one before:
//   1. stream_kernel<kModeStats> (or <kModeGreedy> at temperature 0): chunk
//      statistics and drafted-token logits of every row;
//   2. diag_norm_kernel: one warp per (sequence, position) merges the two rows'
//      chunk statistics (and, under a cumulative floor, the earlier draft rows'
//      for the prefix product) into a DiagNorm record; at temperature 0 it
//      writes the final one-hot values and the call ends here;
//   3. pair_kernel: the bandwidth-bound sweep over every (p_j, q_j) chunk
//      pair, shaped like the stream pass (one CTA per SM, per-warp cp.async
//      rings, work from a shared-memory counter), one partial record per chunk
//      pair -- written over the chunk statistics, which are no longer needed;
//   4. diag_reduce_kernel: one warp per (sequence, position) adds the partials
//      in chunk order (deterministic) and looks up q at the argmax.
#pragma once

#include "verify_kernel.cuh"

namespace sv {

constexpr int kDiagThreads = 256;
constexpr int kDiagWarps = kDiagThreads / 32;

// what the sweep needs of a (sequence, position): both rows' normalisers and
// the gate's predicate q >= tau_e && cprev * q >= mc_e (floors that do not
// apply are -1, which every q passes)
struct __align__(16) DiagNorm {
  float Mt, invSt, Md, invSd;
  float tau_e, cprev, mc_e;
  int bad;
};

// the merged statistics of workspace row r of sequence b, by one warp (the
// finishing pass's merge): scaled max and 1 / sum, or (greedy) the first
// index of the row's largest logit; bad for an invalid row
struct RowMerge {
  float M, invS;
  int targ;
  bool bad;
};

template <bool kGreedy>
__device__ __forceinline__ RowMerge merge_row(const Params& P, int b, int r, int lane) {
  const int nch = P.nchunk;
  const float2* part = P.part + (static_cast<int64_t>(b) * P.rows + r) * nch;
  RowMerge out{0.f, 0.f, -1, true};
  // every lane runs the same trip count (a lane without a chunk adds
  // nothing), so the warp reaches its shuffles converged
  const int niter = (nch + 31) >> 5;
  if constexpr (kGreedy) {
    // (max, first index of the max) per chunk; a negative index marks a bad chunk
    float M = -INFINITY;
    int bc = nch;
    bool bad = false;
#pragma unroll 1
    for (int i = 0; i < niter; ++i) {
      const int ch = lane + 32 * i;
      const float2 ms = ch < nch ? ldcg_f2(part + ch) : make_float2(-INFINITY, 0.f);
      if (__float_as_int(ms.y) < 0) bad = true;
      if (ms.x > M) {
        M = ms.x;
        bc = ch;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float oM = __shfl_xor_sync(0xffffffffu, M, o);
      const int obc = __shfl_xor_sync(0xffffffffu, bc, o);
      if (oM > M || (oM == M && obc < bc)) {
        M = oM;
        bc = obc;
      }
    }
    out.bad = __any_sync(0xffffffffu, bad) || M == -INFINITY || bc >= nch;
    if (!out.bad) out.targ = __float_as_int(ldcg_f2(part + bc).y);
  } else {
    float M = -INFINITY;
#pragma unroll 1
    for (int i = 0; i < niter; ++i) {
      const int ch = lane + 32 * i;
      M = fmaxf(M, ch < nch ? ldcg_f2(part + ch).x : -INFINITY);
    }
    M = warp_max(M);
    dfloat S = df(0.f);
#pragma unroll 1
    for (int i = 0; i < niter; ++i) {
      const int ch = lane + 32 * i;
      const float2 ms = ch < nch ? ldcg_f2(part + ch) : make_float2(-INFINITY, 0.f);
      S = df_add(S, df(ms.x == -INFINITY ? ms.y * 0.f : ms.y * exp2f(ms.x - M)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S = df_add(S, shfl_xor_df(S, o));
    out.M = M;
    out.invS = (1.f / S.hi) * (1.f - S.lo / S.hi);
    out.bad = M == -INFINITY || !isfinite(S.hi) || !(S.hi > 0.f);
  }
  return out;
}

__device__ __forceinline__ void write_diag(int64_t o, float mn, float pq, float aq, float* min_sum,
                                           float* pq_sum, float* argmax_q) {
  if (min_sum) min_sum[o] = mn;
  if (pq_sum) pq_sum[o] = pq;
  if (argmax_q) argmax_q[o] = aq;
}

// launch 2: one warp per (sequence b, position j)
template <bool kGreedy>
__global__ void __launch_bounds__(kDiagThreads)
    diag_norm_kernel(const __grid_constant__ Params P, DiagNorm* __restrict__ norm, float* min_sum,
                     float* pq_sum, float* argmax_q) {
  const int lane = threadIdx.x & 31;
  const int g = static_cast<int>(blockIdx.x) * kDiagWarps + (threadIdx.x >> 5);
  const int k = P.k, V = P.V;
  const bool live = g < P.B * k;
  const int b = live ? g / k : 0, j = live ? g % k : 0;
  // inputs alone, before the wait on the stream pass
  const bool gated = seq_gated(P, b);
  const float tau = step_tau(P, b, j);
  const bool bad_tau = gated && !P.has_sched && !(tau > 0.f && tau <= 1.f);
  const bool cum = gated && P.min_cum > 0.f;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!live) return;

  const RowMerge t = merge_row<kGreedy>(P, b, j, lane);
  const RowMerge d = merge_row<kGreedy>(P, b, k + 1 + j, lane);
  bool bad = t.bad || d.bad || bad_tau;
  // the drafted prefix's product of draft probabilities (one-hot q at T = 0)
  float cprev = 1.f;
  if (cum) {
#pragma unroll 1
    for (int i = 0; i < j && !bad; ++i) {
      const int di = __ldg(P.D + static_cast<int64_t>(b) * k + i);
      const RowMerge ri = merge_row<kGreedy>(P, b, k + 1 + i, lane);
      if (ri.bad || di < 0 || di >= V) {
        bad = true;
      } else if constexpr (kGreedy) {
        cprev *= di == ri.targ ? 1.f : 0.f;
      } else {
        cprev *= prob_of(__ldcg(P.xD + static_cast<int64_t>(b) * P.rows + k + 1 + i), ri.M, P.c, ri.invS);
      }
    }
  }
  const float tau_e = gated ? tau : -1.f;
  const float mc_e = cum ? P.min_cum : -1.f;
  if (lane != 0) return;
  const int64_t o = static_cast<int64_t>(b) * k + j;
  if constexpr (kGreedy) {
    // one-hot p and q at t* and d*: they coincide or they do not
    if (bad) {
      write_diag(o, NAN, NAN, NAN, min_sum, pq_sum, argmax_q);
    } else {
      const bool same = t.targ == d.targ;
      const bool adm = 1.f >= tau_e && cprev >= mc_e;  // q(d*) = 1
      write_diag(o, (same && adm) ? 1.f : 0.f, same ? 1.f : 0.f, same ? 1.f : 0.f, min_sum, pq_sum,
                 argmax_q);
    }
  } else {
    norm[o] = DiagNorm{t.M, t.invS, d.M, d.invS, tau_e, cprev, mc_e, bad ? 1 : 0};
  }
}

// launch 3: the pair sweep.  Shape of the stream pass; a stage holds a chunk of
// the target row and the same chunk of the draft row.
template <typename TT, typename TD>
struct PairStages {
  static constexpr int kBytesT = kChunk * static_cast<int>(sizeof(TT));
  static constexpr int kBytes = kBytesT + kChunk * static_cast<int>(sizeof(TD));
  static constexpr int kDepth = 2;
  // 192 KB of rings per CTA: 12 warps for bf16 pairs, 8 mixed, 6 for fp32
  static constexpr int kWarpsPerCta = (192 * 1024) / (kBytes * kDepth);
  static constexpr int kThreadsPerCta = 32 * kWarpsPerCta;
};

struct PairQueue {
  int4 item[kItemRing];      // (b, j, ch, 1); w = 0: no more work
  DiagNorm nrm[kItemRing];   // the item's DiagNorm, copied asynchronously
  float fthr[kItemRing][2];  // (filtered calls) the target and draft rows'
  int ffirst[kItemRing][2];  // thresholds and kept indices, likewise
};

// partial record of chunk pair (b, j, ch): (sum min(p, mu), sum p q, largest
// target logit, unused), over the chunk statistics' storage
__device__ __forceinline__ float4* pair_partials(const Params& P) { return reinterpret_cast<float4*>(P.part); }

template <typename T>
__device__ __forceinline__ void stage8(const unsigned char* stage, int o, float (&x)[8]) {
  if constexpr (sizeof(T) == 2) {
    const uint4 u = *reinterpret_cast<const uint4*>(stage + o * 2);
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
  } else {
    const float4 a = *reinterpret_cast<const float4*>(stage + o * 4);
    const float4 c = *reinterpret_cast<const float4*>(stage + o * 4 + 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
  }
}

// kFilt: the call's sampler filters applied to both rows as they are read
template <typename TT, typename TD, bool kFilt>
__global__ void __launch_bounds__(PairStages<TT, TD>::kThreadsPerCta, 1)
    pair_kernel(const __grid_constant__ Params P, const DiagNorm* __restrict__ norm, unsigned total) {
  constexpr int S = PairStages<TT, TD>::kDepth;
  constexpr int kStage = PairStages<TT, TD>::kBytes;
  constexpr int kBT = PairStages<TT, TD>::kBytesT;
  extern __shared__ __align__(128) unsigned char rings[];
  __shared__ PairQueue queues[PairStages<TT, TD>::kWarpsPerCta];
  __shared__ unsigned cta_next;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* ring = rings + warp * S * kStage;
  PairQueue& Q = queues[warp];
  const int k = P.k, V = P.V, nch = P.nchunk;
  const float c = P.c;
  float4* out = pair_partials(P);

  if (threadIdx.x == 0) cta_next = 0u;
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the DiagNorm records (and the free chunk-statistics storage) come from the
  // preceding launches
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // lane 0: the warp's next pair index x = (b k + j) nch + ch, or kNoWork
  auto next = [&]() -> unsigned {
    const unsigned i = atomicAdd(&cta_next, 1u);
    const unsigned long long x = blockIdx.x + static_cast<unsigned long long>(i) * gridDim.x;
    return x < total ? static_cast<unsigned>(x) : kNoWork;
  };
  auto put = [&](int slot, unsigned x) {
    if (x == kNoWork) {
      Q.item[slot] = make_int4(0, 0, 0, 0);
      return;
    }
    const unsigned rg = fastdiv(x, P.div_nchunk);  // b k + j
    const int ch = static_cast<int>(x - rg * static_cast<unsigned>(nch));
    const int b = static_cast<int>(rg / static_cast<unsigned>(k)), j = static_cast<int>(rg % k);
    Q.item[slot] = make_int4(b, j, ch, 1);
    cp_async16(&Q.nrm[slot], norm + rg);
    cp_async16(reinterpret_cast<unsigned char*>(&Q.nrm[slot]) + 16,
               reinterpret_cast<const unsigned char*>(norm + rg) + 16);
    if constexpr (kFilt) {
      const int64_t gt = static_cast<int64_t>(b) * P.rows + j, gd = gt + k + 1;
      cp_async4(&Q.fthr[slot][0], P.fthr + gt);
      cp_async4(&Q.fthr[slot][1], P.fthr + gd);
      cp_async4(&Q.ffirst[slot][0], P.ffirst + gt);
      cp_async4(&Q.ffirst[slot][1], P.ffirst + gd);
    }
  };
  if (lane == 0) put(0, next());
  __syncwarp();
  int issued = 0;
  auto issue_next = [&]() {
    const int4 it = Q.item[issued % kItemRing];
    if (it.w > 0) {
      unsigned char* st = ring + (issued % S) * kStage;
      const int c0 = it.z * kChunk;
      Lane<TT>::issue(static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(it.x) * (k + 1) + it.y) * V, st, c0,
                      V, P.vec_t != 0, lane);
      Lane<TD>::issue(static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(it.x) * k + it.y) * V, st + kBT, c0,
                      V, P.vec_d != 0, lane);
    }
    if (lane == 0) put((issued + 1) % kItemRing, it.w > 0 ? next() : kNoWork);
    ++issued;
    cp_async_commit();
    __syncwarp();
  };
#pragma unroll
  for (int s = 0; s < S - 1; ++s) issue_next();
  for (int n = 0;; ++n) {
    const int4 it = Q.item[n % kItemRing];
    if (it.w <= 0) break;
    issue_next();
    cp_async_wait<S - 1>();
    __syncwarp();
    const DiagNorm nm = Q.nrm[n % kItemRing];  // landed with the item's commit group
    float thr_t = 0.f, thr_d = 0.f;            // likewise
    int first_t = -1, first_d = -1;
    if constexpr (kFilt) {
      thr_t = Q.fthr[n % kItemRing][0];
      thr_d = Q.fthr[n % kItemRing][1];
      first_t = Q.ffirst[n % kItemRing][0];
      first_d = Q.ffirst[n % kItemRing][1];
    }
    const unsigned char* st = ring + (n % S) * kStage;
    if (!nm.bad) {
      float amin = 0.f, apq = 0.f, best = -INFINITY;
      const int c0 = it.z * kChunk;
      // lane l takes entries (32 g + l) 8 .. + 7, g = 0..7; the terms use the
      // fast exp2 (the sums' tolerance is far above its error), and without a
      // cumulative floor the gate is one compare
      auto sweep = [&](auto cum) {
#pragma unroll 2
        for (int g = 0; g < kChunk / 256; ++g) {
          const int o = (32 * g + lane) * 8;
          float xt[8], xd[8], mn[8], pq[8];
          stage8<TT>(st, o, xt);
          stage8<TD>(st + kBT, o, xd);
          if constexpr (kFilt) {
            filt8(xt, c0 + o, thr_t, first_t);
            filt8(xd, c0 + o, thr_d, first_d);
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float p = ex2_approx(fmaf(xt[e], c, -nm.Mt)) * nm.invSt;
            const float q = ex2_approx(fmaf(xd[e], c, -nm.Md)) * nm.invSd;
            bool adm = q >= nm.tau_e;
            if constexpr (decltype(cum)::value) adm = adm && nm.cprev * q >= nm.mc_e;
            mn[e] = fminf(p, adm ? q : 0.f);
            pq[e] = p * q;
            best = fmaxf(best, xt[e]);
          }
          amin += ((mn[0] + mn[1]) + (mn[2] + mn[3])) + ((mn[4] + mn[5]) + (mn[6] + mn[7]));
          apq += ((pq[0] + pq[1]) + (pq[2] + pq[3])) + ((pq[4] + pq[5]) + (pq[6] + pq[7]));
        }
      };
      if (nm.mc_e >= 0.f) sweep(std::true_type{});
      else sweep(std::false_type{});
      amin = warp_sum(amin);
      apq = warp_sum(apq);
      best = warp_max(best);
      // the chunk's largest target logit; the reduction finds the first index
      // of the row's largest in the first chunk that holds it
      if (lane == 0)
        out[(static_cast<int64_t>(it.x) * k + it.y) * nch + it.z] = make_float4(amin, apq, best, 0.f);
    }
    __syncwarp();
  }
  cp_async_wait<0>();
}

// launch 4: one warp per (sequence b, position j): the partials added in
// chunk order, the argmax's q looked up
template <typename TT, typename TD>
__global__ void __launch_bounds__(kDiagThreads)
    diag_reduce_kernel(const __grid_constant__ Params P, const DiagNorm* __restrict__ norm, float* min_sum,
                       float* pq_sum, float* argmax_q) {
  const int lane = threadIdx.x & 31;
  const int g = static_cast<int>(blockIdx.x) * kDiagWarps + (threadIdx.x >> 5);
  const int k = P.k, V = P.V, nch = P.nchunk;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (g >= P.B * k) return;
  const DiagNorm nm = norm[g];
  if (nm.bad) {
    if (lane == 0) write_diag(g, NAN, NAN, NAN, min_sum, pq_sum, argmax_q);
    return;
  }
  const float4* part = pair_partials(P) + static_cast<int64_t>(g) * nch;
  float amin = 0.f, apq = 0.f, best = -INFINITY;
  int bch = 0x7fffffff;  // the first chunk holding the row's largest target logit
  // the same trip count on every lane: the shuffles below run converged
  const int niter = (nch + 31) >> 5;
#pragma unroll 1
  for (int i = 0; i < niter; ++i) {
    const int ch = lane + 32 * i;
    if (ch >= nch) continue;
    const float4 r = __ldcg(part + ch);
    amin += r.x;
    apq += r.y;
    if (r.z > best) {  // chunks in increasing order per lane: the first one kept
      best = r.z;
      bch = ch;
    }
  }
  amin = warp_sum(amin);
  apq = warp_sum(apq);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, s);
    const int oc = __shfl_xor_sync(0xffffffffu, bch, s);
    if (ob > best || (ob == best && oc < bch)) {
      best = ob;
      bch = oc;
    }
  }
  // the first index of that logit in that chunk of the target row (the
  // largest logit is kept by every sampler filter, so the raw row serves)
  const int b = g / k, j = g % k;
  int bidx = 0x7fffffff;
  if (bch < nch) {
    // lane l holds entries [64 l, 64 l + 64) of the chunk, loaded at once
    // (entries past V read as -inf)
    const TT* trow = static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (k + 1) + j) * V;
    const int v0 = bch * kChunk + 64 * lane;
    float x[8][8];
#pragma unroll
    for (int h = 0; h < 8; ++h) load8<TT>(trow, v0 + 8 * h, V, P.vec_t != 0, x[h]);
#pragma unroll
    for (int h = 7; h >= 0; --h)
#pragma unroll
      for (int e = 7; e >= 0; --e)
        if (x[h][e] == best) bidx = v0 + 8 * h + e;  // the last assignment is the first index
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) bidx = min(bidx, __shfl_xor_sync(0xffffffffu, bidx, s));
  }
  if (lane == 0) {
    const TD* drow = static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * k + j) * V;
    float aq = NAN;
    if (bidx < V) {
      float xq = logit_at<TD>(drow, bidx);
      if (P.fthr) {  // the draft row as its sampler filter leaves it
        const int64_t gd = static_cast<int64_t>(b) * P.rows + k + 1 + j;
        xq = filt1(xq, bidx, P.fthr[gd], P.ffirst[gd]);
      }
      aq = prob_of(xq, nm.Md, P.c, nm.invSd);
    }
    write_diag(g, amin, apq, aq, min_sum, pq_sum, argmax_q);
  }
}

}  // namespace sv
