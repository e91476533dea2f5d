// Fused batched speculative-decoding verification kernel for sm_103a.
//
// One launch verifies a whole batch.  Work is a list of items (sequence b,
// row r, chunk c) in sequence-major order, where rows 0..k are the target
// rows and rows k+1..2k the draft rows of b, and a chunk is kChunk = 8192
// consecutive vocabulary entries.  Persistent CTAs pull items from a global
// counter (so a CTA that is busy finishing a sequence simply takes fewer
// items) and run a cp.async pipeline of S chunk stages in shared memory:
//
//   1. stream the chunk once (16-byte cp.async per thread, each warp copying
//      512 contiguous bytes per instruction; every thread later reads back
//      exactly the pieces it copied, so the pipeline needs no extra barrier),
//      take the chunk max m and s = sum exp((L - m) / T) -- the one-read row
//      statistics of the temperature softmax (mlxcel PR #992, "What changed":
//      p and q are full-vocabulary temperature softmaxes in fp32); record the
//      logit at the drafted token when it lies in the chunk; for draft rows
//      of gated sequences keep the tokens whose in-chunk probability reaches
//      the gate (at most floor(1/threshold) of them, a superset of the tokens
//      the gate admits) in a per-row candidate list;
//   2. publish (m, s) and bump the sequence's completion counter with an
//      acq_rel atomic; the CTA that completes the last item of sequence b
//      finishes b (no CTA ever waits for another, so nothing can hang):
//   3. combine the chunk partials into row max / sum, evaluate every draft
//      position -- gate, retained measure mu, alpha = min(1, p(D)/mu(D)),
//      Philox u0, the accept test p > 0 && u0 * mu <= p (Strata PR #3416,
//      "Approach"; mlxcel PR #992, "What changed") -- and stop at the first
//      position not accepted;
//   4. sample the stop row: the normalised positive part of p - mu after a
//      rejection or NULL, p itself for the bonus row.  Chunk sums of the
//      residual come from the partials (minus the admitted tokens' min(p, q)
//      in gated mode), a prefix over chunks finds the chunk holding u1 * Z,
//      and one re-read of that chunk with a block-wide scan finds the token.
//      Plain-mode rejections need q everywhere, so they re-read the stop row
//      pair once to form the chunk sums.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "philox.cuh"
#include "spec_verify.h"

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kEPT = 32;                    // elements per thread per chunk
constexpr int kChunk = kThreads * kEPT;     // vocabulary entries per work item
constexpr int kTopM = 4;                    // gate candidates per chunk / admitted tokens per row
constexpr int kRowCap = 64;                 // gate candidates kept per draft row
constexpr int kMaxChunks = (SV_MAX_V + kChunk - 1) / kChunk;
constexpr int kMaxRows = 2 * SV_MAX_K + 1;
constexpr int kRing = 8;                    // fetched item indices kept per CTA
constexpr float kBoundary = 1e-6f;
// Candidates are kept against a threshold lowered by this factor so that
// rounding cannot drop an admitted token; the gated fast path needs
// slack * threshold * (kTopM + 1) > 1, i.e. threshold > ~0.2002.
constexpr float kGateSlack = 1.0f - 1.0f / 1024.0f;

struct Params {
  const void* Lt;  // [B, k+1, V]
  const void* Ld;  // [B, k, V]
  const int32_t* D;
  int B, k, V, nchunk, rows, items_per_seq;
  unsigned total_items;
  float c;     // log2(e) / T, rounded once
  float T;
  int gate_default;
  float tau_default;
  const uint8_t* gate_per_seq;
  const float* tau_per_seq;
  uint64_t seed, seq_offset;
  const float* u0;
  const float* u1;
  int32_t* accepted_len;
  int32_t* tokens;
  float* alpha;
  int8_t* flags;
  unsigned long long* counters;
  float* row_stats;
  // workspace
  float2* part;        // [B, rows, nchunk] (chunk max of raw logits, sum of exp2((L - m) c))
  float* xD;           // [B, rows] raw logit at the drafted token (rows j < k and draft rows)
  float* cand_v;       // [B, k, kRowCap] raw logits of gate candidates
  int* cand_i;         // [B, k, kRowCap] their token ids
  unsigned* cand_n;    // [B, k] candidates appended (> kRowCap: overflow); reset by the finisher
  unsigned* seq_done;  // [B] completion counters, reset by the finisher
  unsigned* work;      // [1] next item to hand out, reset by the last CTA to exit
  unsigned* exit_count;  // [1]
  int vec_t, vec_d;    // rows allow 16-byte vector loads
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ float2 ldcg_f2(const float2* p) { return __ldcg(p); }

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(f32x2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}
__device__ __forceinline__ double warp_incl_scan_d(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// one logit as float
template <typename T> __device__ __forceinline__ float logit_at(const T* row, int64_t v);
template <> __device__ __forceinline__ float logit_at<uint16_t>(const uint16_t* row, int64_t v) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(row + v)) << 16);
}
template <> __device__ __forceinline__ float logit_at<float>(const float* row, int64_t v) {
  return __ldg(row + v);
}

// eight consecutive logits [v0, v0 + 8) as floats; -inf past V
template <typename T>
__device__ __forceinline__ void load8(const T* row, int v0, int V, bool vec, float (&x)[8]);
template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* row, int v0, int V, bool vec,
                                                float (&x)[8]) {
  if (vec && v0 + 8 <= V) {
    const uint4 u = __ldcg(reinterpret_cast<const uint4*>(row + v0));
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (v0 + e < V) ? logit_at<uint16_t>(row, v0 + e) : -INFINITY;
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* row, int v0, int V, bool vec,
                                             float (&x)[8]) {
  if (vec && v0 + 8 <= V) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(row + v0));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(row + v0) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (v0 + e < V) ? logit_at<float>(row, v0 + e) : -INFINITY;
  }
}

// probability of a token with raw logit x in a row with raw max M and
// 1/sum invS: exp2((x - M) * c) * invS.  Every decision uses this one formula.
__device__ __forceinline__ float prob_of(float x, float M, float c, float invS) {
  return exp2f((x - M) * c) * invS;
}

__device__ __forceinline__ bool gate_fast_path(float tau) {
  return tau * kGateSlack * static_cast<float>(kTopM + 1) > 1.0f;
}

// ------------------------------------------------------- chunk registers
//
// Thread t = 32 w + l owns NV 16-byte slots of the chunk: slot i is vector
// index w * 32 NV + 32 i + l (each copy instruction of a warp moves 512
// contiguous bytes).  bf16: 4 slots of 8 entries kept packed; f32: 8 slots of
// 4.  A slot that lies wholly inside the row of an aligned tensor travels by
// cp.async into the stage; other slots (ragged tail, unaligned rows) are read
// directly, entries past V reading as -inf.

template <typename T> struct Chunk;

template <> struct Chunk<uint16_t> {
  static constexpr int kNV = 4, kVE = 8;
  uint32_t w[16];
  __device__ __forceinline__ static void issue(const uint16_t* row, unsigned char* stage, int c0, int V,
                                               int warp, int lane) {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int sv = warp * 32 * kNV + 32 * i + lane;
      const int v0 = c0 + sv * kVE;
      if (v0 + kVE <= V) cp_async16(stage + sv * 16, row + v0);
    }
  }
  __device__ __forceinline__ void load(const uint16_t* row, const unsigned char* stage, int c0, int V,
                                       bool vec, int warp, int lane) {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int sv = warp * 32 * kNV + 32 * i + lane;
      const int v0 = c0 + sv * kVE;
      if (vec && v0 + kVE <= V) {
        const uint4 u = *reinterpret_cast<const uint4*>(stage + sv * 16);
        w[4 * i + 0] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int a = v0 + 2 * q;
          const uint32_t lo = a < V ? static_cast<uint32_t>(__ldg(row + a)) : 0xFF80u;
          const uint32_t hi = a + 1 < V ? static_cast<uint32_t>(__ldg(row + a + 1)) : 0xFF80u;
          w[4 * i + q] = lo | (hi << 16);
        }
      }
    }
  }
  __device__ __forceinline__ float max() const {
    uint32_t m = w[0];
#pragma unroll
    for (int q = 1; q < 16; ++q) m = bmax2(m, w[q]);
    return fmaxf(bf16_lo(m), bf16_hi(m));
  }
  __device__ __forceinline__ float expsum(float m, float c) const {
    const f32x2 mm = pk(m, m), cc = pk(c, c);
    f32x2 acc = pk(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      float a, b;
      upk(mul2(sub2(pk(bf16_lo(w[q]), bf16_hi(w[q])), mm), cc), a, b);
      acc = add2(acc, pk(ex2_approx(a), ex2_approx(b)));
    }
    float s0, s1;
    upk(acc, s0, s1);
    return s0 + s1;
  }
  template <typename F>
  __device__ __forceinline__ void for_each(int c0, int warp, int lane, F&& f) const {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int v0 = c0 + (warp * 32 * kNV + 32 * i + lane) * kVE;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f(v0 + 2 * q, bf16_lo(w[4 * i + q]));
        f(v0 + 2 * q + 1, bf16_hi(w[4 * i + q]));
      }
    }
  }
};

template <> struct Chunk<float> {
  static constexpr int kNV = 8, kVE = 4;
  float x[32];
  __device__ __forceinline__ static void issue(const float* row, unsigned char* stage, int c0, int V,
                                               int warp, int lane) {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int sv = warp * 32 * kNV + 32 * i + lane;
      const int v0 = c0 + sv * kVE;
      if (v0 + kVE <= V) cp_async16(stage + sv * 16, row + v0);
    }
  }
  __device__ __forceinline__ void load(const float* row, const unsigned char* stage, int c0, int V,
                                       bool vec, int warp, int lane) {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int sv = warp * 32 * kNV + 32 * i + lane;
      const int v0 = c0 + sv * kVE;
      if (vec && v0 + kVE <= V) {
        const float4 u = *reinterpret_cast<const float4*>(stage + sv * 16);
        x[4 * i + 0] = u.x; x[4 * i + 1] = u.y; x[4 * i + 2] = u.z; x[4 * i + 3] = u.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[4 * i + e] = v0 + e < V ? __ldg(row + v0 + e) : -INFINITY;
      }
    }
  }
  __device__ __forceinline__ float max() const {
    float m = x[0];
#pragma unroll
    for (int e = 1; e < 32; ++e) m = fmaxf(m, x[e]);
    return m;
  }
  __device__ __forceinline__ float expsum(float m, float c) const {
    const f32x2 mm = pk(m, m), cc = pk(c, c);
    f32x2 acc = pk(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float a, b;
      upk(mul2(sub2(pk(x[e], x[e + 1]), mm), cc), a, b);
      acc = add2(acc, pk(ex2_approx(a), ex2_approx(b)));
    }
    float s0, s1;
    upk(acc, s0, s1);
    return s0 + s1;
  }
  template <typename F>
  __device__ __forceinline__ void for_each(int c0, int warp, int lane, F&& f) const {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int v0 = c0 + (warp * 32 * kNV + 32 * i + lane) * kVE;
#pragma unroll
      for (int e = 0; e < 4; ++e) f(v0 + e, x[4 * i + e]);
    }
  }
};

// ---------------------------------------------------------- shared state

struct Shared {
  // streaming phase
  float red_max[kWarps];
  float red_sum[kWarps];
  int ncand;
  float cand_v[kTopM];
  int cand_i[kTopM];
  unsigned ring[kRing];
  int fin_b;
  // finishing phase
  float rowM[kMaxRows];
  float rowInvS[kMaxRows];
  double rowS[kMaxRows];
  float xD[kMaxRows];
  int Dv[SV_MAX_K];
  unsigned candn[SV_MAX_K];
  double tile[kMaxChunks];
  double wbase[kWarps];
  float wtot[kWarps];
  int bad;
  int jstar;
  int stop_flag;
  int boundary;
  unsigned overflow_rows;
  int tstar;
  double before;
  int pick;
  int last_pos;
  int nadm[SV_MAX_K];
  int adm_i[SV_MAX_K][kTopM];
  float adm_q[SV_MAX_K][kTopM];
  float adm_p[SV_MAX_K][kTopM];
};

__device__ __forceinline__ bool seq_gated(const Params& P, int b) {
  return P.gate_per_seq ? (P.gate_per_seq[b] != 0) : (P.gate_default != 0);
}
__device__ __forceinline__ float seq_tau(const Params& P, int b) {
  return P.tau_per_seq ? P.tau_per_seq[b] : P.tau_default;
}

// ------------------------------------------------------------ finishing

// residual weight of token v with target logit xt (and draft logit xd in the
// dense mode).  mode 0: p (bonus row, or degenerate residual); mode 1: p, or
// max(0, p - q) on the admitted list; mode 2: max(0, p - mu) with mu from the
// draft logit (mu = q, or q on q >= tau in gated mode).
struct ResidualEval {
  int mode;
  float Mt, invSt, Md, invSd, c, tau;
  bool gated;
  int nadm;
  const int* adm_i;
  const float* adm_q;
  __device__ __forceinline__ float operator()(int v, float xt, float xd) const {
    const float p = prob_of(xt, Mt, c, invSt);
    if (mode == 0) return p;
    if (mode == 1) {
      for (int a = 0; a < nadm; ++a)
        if (adm_i[a] == v) return fmaxf(p - adm_q[a], 0.f);
      return p;
    }
    const float q = prob_of(xd, Md, c, invSd);
    const float mu = (!gated || q >= tau) ? q : 0.f;
    return fmaxf(p - mu, 0.f);
  }
};

template <typename TT, typename TD>
__device__ void finish_sequence(const Params& P, int b, Shared& sh) {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k, R = P.rows, nch = P.nchunk, V = P.V;
  const bool gated = seq_gated(P, b);
  const float tau = seq_tau(P, b);
  const bool fastgate = gated && gate_fast_path(tau);
  const float c = P.c;
  const uint64_t s_idx = P.seq_offset + static_cast<uint64_t>(b);
  const TT* Lt = static_cast<const TT*>(P.Lt);
  const TD* Ld = static_cast<const TD*>(P.Ld);

  // phase A: everything the decisions need, in one round of loads
  if (tid == 0) {
    sh.bad = (gated && !(tau > 0.f && tau <= 1.f)) ? 1 : 0;
    sh.boundary = 0;
    sh.pick = -1;
    sh.last_pos = -1;
    sh.overflow_rows = 0u;
  }
  if (tid < R) sh.xD[tid] = __ldcg(P.xD + static_cast<int64_t>(b) * R + tid);
  if (tid < k) {
    sh.Dv[tid] = __ldg(P.D + static_cast<int64_t>(b) * k + tid);
    sh.candn[tid] = fastgate ? __ldcg(P.cand_n + static_cast<int64_t>(b) * k + tid) : 0u;
    sh.nadm[tid] = 0;
  }
  // candidate entries of every draft row, read before the counts are known
  // (slots past kCandPerThread * kThreads, i.e. k > 8, are read in phase B)
  constexpr int kCandPerThread = 2;
  float cv[kCandPerThread];
  int ci[kCandPerThread];
  if (fastgate) {
#pragma unroll
    for (int u = 0; u < kCandPerThread; ++u) {
      const int e = tid + u * kThreads;
      if (e < k * kRowCap) {
        cv[u] = __ldcg(P.cand_v + static_cast<int64_t>(b) * k * kRowCap + e);
        ci[u] = __ldcg(P.cand_i + static_cast<int64_t>(b) * k * kRowCap + e);
      }
    }
  }
  // F1: row max / sum from the chunk partials (fp64 accumulation)
  for (int r = warp; r < R; r += kWarps) {
    const float2* pr = P.part + (static_cast<int64_t>(b) * R + r) * nch;
    float M = -INFINITY;
    for (int ch = lane; ch < nch; ch += 32) M = fmaxf(M, ldcg_f2(pr + ch).x);
    M = warp_max(M);
    double S = 0.0;
    for (int ch = lane; ch < nch; ch += 32) {
      const float2 ms = ldcg_f2(pr + ch);
      S += (ms.x == -INFINITY) ? static_cast<double>(ms.y * 0.f)
                               : static_cast<double>(ms.y) * static_cast<double>(exp2f((ms.x - M) * c));
    }
    S = warp_sum_d(S);
    if (lane == 0) {
      sh.rowM[r] = M;
      sh.rowS[r] = S;
      sh.rowInvS[r] = static_cast<float>(1.0 / S);
      if (M == -INFINITY || !isfinite(S) || !(S > 0.0)) sh.bad = 1;
      if (P.row_stats) {
        const float mo = M / P.T;
        P.row_stats[(static_cast<int64_t>(b) * R + r) * 2 + 0] = mo;
        P.row_stats[(static_cast<int64_t>(b) * R + r) * 2 + 1] =
            static_cast<float>(static_cast<double>(mo) + log(S));
      }
    }
  }
  __syncthreads();

  // phase B: admitted tokens of every draft row and their target probability
  // (one more round of loads, overlapping the decisions below)
  if (fastgate && !sh.bad) {
    auto admit = [&](int e, float x, int v) {
      const int j = e / kRowCap, s = e - j * kRowCap;
      const unsigned n = sh.candn[j];
      if (n > static_cast<unsigned>(kRowCap)) {
        if (s == 0) atomicOr(&sh.overflow_rows, 1u << j);
        return;
      }
      if (s >= static_cast<int>(n)) return;
      const int rd = k + 1 + j;
      const float q = prob_of(x, sh.rowM[rd], c, sh.rowInvS[rd]);
      if (q >= tau) {
        const int a = atomicAdd(&sh.nadm[j], 1);
        if (a < kTopM) {
          const float xt = logit_at<TT>(Lt + (static_cast<int64_t>(b) * (k + 1) + j) * V, v);
          sh.adm_i[j][a] = v;
          sh.adm_q[j][a] = q;
          sh.adm_p[j][a] = prob_of(xt, sh.rowM[j], c, sh.rowInvS[j]);
        } else {
          atomicOr(&sh.overflow_rows, 1u << j);
        }
      }
    };
#pragma unroll
    for (int u = 0; u < kCandPerThread; ++u)
      if (tid + u * kThreads < k * kRowCap) admit(tid + u * kThreads, cv[u], ci[u]);
    for (int e = tid + kCandPerThread * kThreads; e < k * kRowCap; e += kThreads)
      admit(e, __ldcg(P.cand_v + static_cast<int64_t>(b) * k * kRowCap + e),
            __ldcg(P.cand_i + static_cast<int64_t>(b) * k * kRowCap + e));
  }

  // F2: every draft position (one lane each): gate, mu, alpha, accept test
  if (warp == 0) {
    bool ok = true, acc = false, is_null = false, near = false;
    float alpha = 0.f;
    if (lane < k) {
      const int d = sh.Dv[lane];
      ok = d >= 0 && d < V;
      if (ok && !sh.bad) {
        const int rt = lane, rd = k + 1 + lane;
        const float p = prob_of(sh.xD[rt], sh.rowM[rt], c, sh.rowInvS[rt]);
        const float q = prob_of(sh.xD[rd], sh.rowM[rd], c, sh.rowInvS[rd]);
        const bool admitted = !gated || q >= tau;
        const float mu = admitted ? q : 0.f;
        is_null = !admitted;
        alpha = is_null ? 0.f : (mu > 0.f ? fminf(1.f, p / mu) : (p > 0.f ? 1.f : 0.f));
        const float u0 = P.u0 ? P.u0[static_cast<int64_t>(b) * k + lane]
                              : philox_uniform(P.seed, s_idx, static_cast<uint32_t>(lane), 0u);
        acc = !is_null && p > 0.f && u0 * mu <= p;
        near = (gated && fabsf(q - tau) < kBoundary) ||
               (!is_null && mu > 0.f && p < mu && fabsf(u0 - p / mu) < kBoundary);
      }
    }
    const bool any_bad = __any_sync(0xffffffffu, !ok) || sh.bad;
    const unsigned accm = __ballot_sync(0xffffffffu, lane < k && acc);
    int jstar = __ffs(~accm) - 1;
    if (jstar > k || jstar < 0) jstar = k;
    const unsigned nearm = __ballot_sync(0xffffffffu, near && lane <= jstar);
    const unsigned nullm = __ballot_sync(0xffffffffu, is_null);
    if (lane < k) {
      const int64_t o = static_cast<int64_t>(b) * k + lane;
      P.alpha[o] = any_bad ? 0.f : alpha;
      if (P.flags) {
        int8_t f;
        if (any_bad) f = SV_FLAG_INVALID;
        else if (lane < jstar) f = SV_FLAG_ACCEPT;
        else if (lane == jstar) f = is_null ? SV_FLAG_NULL : SV_FLAG_REJECT;
        else f = SV_FLAG_UNREACHED;
        P.flags[o] = f;
      }
    }
    if (lane == 0) {
      sh.bad = any_bad ? 1 : 0;
      sh.jstar = jstar;
      sh.stop_flag = jstar < k ? (((nullm >> jstar) & 1u) ? SV_FLAG_NULL : SV_FLAG_REJECT)
                               : SV_FLAG_ACCEPT;
      sh.boundary = __popc(nearm);
    }
  }
  __syncthreads();

  const int jstar = sh.jstar;
  int32_t* tok = P.tokens + static_cast<int64_t>(b) * (k + 1);
  if (fastgate && tid < k) P.cand_n[static_cast<int64_t>(b) * k + tid] = 0u;  // ready for the next call
  if (sh.bad) {
    if (tid <= k) tok[tid] = -1;
    if (tid == 0) {
      P.accepted_len[b] = -1;
      if (P.counters) atomicAdd(P.counters + SV_CNT_INVALID, 1ull);
    }
    return;
  }

  // F3: the stop row's residual (or bonus) weights, chunk by chunk
  const int rt = jstar, rd = k + 1 + jstar;
  const TT* trow = Lt + (static_cast<int64_t>(b) * (k + 1) + jstar) * V;
  const TD* drow = jstar < k ? Ld + (static_cast<int64_t>(b) * k + jstar) * V : nullptr;
  int mode = 0;
  if (jstar < k) mode = (fastgate && !((sh.overflow_rows >> jstar) & 1u)) ? 1 : 2;
  const int nadm = mode == 1 ? min(sh.nadm[jstar], kTopM) : 0;

  const ResidualEval ev{mode, sh.rowM[rt], sh.rowInvS[rt],
                        jstar < k ? sh.rowM[rd] : 0.f, jstar < k ? sh.rowInvS[rd] : 0.f,
                        c, tau, gated, nadm, jstar < k ? sh.adm_i[jstar] : sh.adm_i[0],
                        jstar < k ? sh.adm_q[jstar] : sh.adm_q[0]};

  auto chunk_sums_from_partials = [&](int use_mode) {
    const float2* pr = P.part + (static_cast<int64_t>(b) * R + rt) * nch;
    for (int ch = tid; ch < nch; ch += kThreads) {
      const float2 ms = ldcg_f2(pr + ch);
      double t = (ms.x == -INFINITY)
                     ? 0.0
                     : static_cast<double>(ms.y) * static_cast<double>(exp2f((ms.x - ev.Mt) * c)) *
                           (1.0 / sh.rowS[rt]);
      if (use_mode == 1) {
        for (int a = 0; a < nadm; ++a)
          if (sh.adm_i[jstar][a] / kChunk == ch)
            t -= static_cast<double>(fminf(sh.adm_p[jstar][a], sh.adm_q[jstar][a]));
        if (t < 0.0) t = 0.0;
      }
      sh.tile[ch] = t;
    }
  };

  if (mode == 2) {
    // dense: one re-read of the stop row pair, a warp per chunk
    for (int ch = warp; ch < nch; ch += kWarps) {
      float acc = 0.f;
      const int c0 = ch * kChunk;
#pragma unroll 4
      for (int u = 0; u < kChunk / 8 / 32; ++u) {
        const int v0 = c0 + (u * 32 + lane) * 8;
        if (v0 < V) {
          float xt[8], xd[8];
          load8<TT>(trow, v0, V, P.vec_t != 0, xt);
          load8<TD>(drow, v0, V, P.vec_d != 0, xd);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (v0 + e < V) acc += ev(v0 + e, xt[e], xd[e]);
        }
      }
      const double t = warp_sum_d(static_cast<double>(acc));
      if (lane == 0) sh.tile[ch] = t;
    }
  } else {
    chunk_sums_from_partials(mode);
  }
  __syncthreads();

  // total mass; a residual without mass falls back to p
  double Z;
  {
    double z = 0.0;
    for (int ch = lane; ch < nch; ch += 32) z += sh.tile[ch];
    Z = warp_sum_d(z);
  }
  int degenerate = 0;
  ResidualEval ev2 = ev;
  if (!(Z > 0.0)) {
    __syncthreads();
    chunk_sums_from_partials(0);
    __syncthreads();
    double z = 0.0;
    for (int ch = lane; ch < nch; ch += 32) z += sh.tile[ch];
    Z = warp_sum_d(z);
    ev2.mode = 0;
    degenerate = 1;
  }

  const float u1 = P.u1 ? P.u1[b] : philox_uniform(P.seed, s_idx, static_cast<uint32_t>(jstar), 1u);
  const double y = static_cast<double>(u1) * Z;

  // the chunk holding y: first chunk whose inclusive prefix exceeds y
  if (warp == 0) {
    double carry = 0.0;
    int found = -1;
    double before = 0.0;
    for (int g0 = 0; g0 < nch && found < 0; g0 += 32) {
      const int ch = g0 + lane;
      const double t = ch < nch ? sh.tile[ch] : 0.0;
      const double incl = warp_incl_scan_d(t, lane) + carry;
      const unsigned m = __ballot_sync(0xffffffffu, ch < nch && incl > y);
      if (m) {
        const int src = __ffs(m) - 1;
        found = g0 + src;
        before = __shfl_sync(0xffffffffu, incl - t, src);
      }
      carry = __shfl_sync(0xffffffffu, incl, 31);
    }
    if (found < 0) {
      // rounding left y at or past the total: take the last chunk with mass
      int last = -1;
      for (int ch = lane; ch < nch; ch += 32)
        if (sh.tile[ch] > 0.0) last = ch;
      for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      found = last < 0 ? 0 : last;
      before = INFINITY;  // forces the last-positive fallback inside the chunk
    }
    if (lane == 0) {
      sh.tstar = found;
      sh.before = before;
    }
  }
  __syncthreads();

  // one re-read of the chosen chunk: thread i owns entries [c0 + 32 i, c0 + 32 i + 32)
  {
    const int c0 = sh.tstar * kChunk;
    const int e0 = c0 + tid * kEPT;
    const double yl = y - sh.before;
    float r[kEPT];
#pragma unroll
    for (int g = 0; g < kEPT / 8; ++g) {
      float xt[8], xd[8];
      load8<TT>(trow, e0 + 8 * g, V, P.vec_t != 0, xt);
      if (ev2.mode == 2) load8<TD>(drow, e0 + 8 * g, V, P.vec_d != 0, xd);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int v = e0 + 8 * g + e;
        r[8 * g + e] = v < V ? ev2(v, xt[e], ev2.mode == 2 ? xd[e] : 0.f) : 0.f;
      }
    }
    // per-thread total (pairwise), warp scan in fp32, block offsets in fp64.
    // Thread i's range is [lo_i, hi_i) with lo_{i+1} == hi_i bit for bit, so
    // exactly one thread claims any y below the chunk total.
    float pw[kEPT / 2];
#pragma unroll
    for (int e = 0; e < kEPT / 2; ++e) pw[e] = r[2 * e] + r[2 * e + 1];
#pragma unroll
    for (int w = kEPT / 4; w >= 1; w >>= 1)
#pragma unroll
      for (int e = 0; e < w; ++e) pw[e] = pw[2 * e] + pw[2 * e + 1];
    const float tot = pw[0];
    const float wincl = warp_incl_scan(tot, lane);
    float wexcl = __shfl_up_sync(0xffffffffu, wincl, 1);
    if (lane == 0) wexcl = 0.f;
    if (lane == 31) sh.wtot[warp] = wincl;
    __syncthreads();
    if (lane == 0) {
      double base = 0.0;
      for (int w = 0; w < warp; ++w) base += static_cast<double>(sh.wtot[w]);
      sh.wbase[warp] = base;
    }
    __syncwarp();
    const double wbase = sh.wbase[warp];
    const double lo = wbase + static_cast<double>(wexcl), hi = wbase + static_cast<double>(wincl);
    int lastpos = -1;
#pragma unroll
    for (int e = 0; e < kEPT; ++e)
      if (r[e] > 0.f) lastpos = e0 + e;
    if (lo <= yl && yl < hi) {
      const float target = static_cast<float>(yl - lo);
      float run = 0.f, prev = 0.f;
      int pick = lastpos;  // rounding inside the thread: its last positive entry
      bool hit = false;
      for (int e = 0; e < kEPT; ++e) {
        prev = run;
        run += r[e];
        if (run > target) {
          pick = e0 + e;
          hit = true;
          break;
        }
      }
      if (!hit) prev = run = static_cast<float>(hi - lo);
      sh.pick = pick;
      const double cl = (sh.before + lo + static_cast<double>(prev)) / Z;
      const double chh = (sh.before + lo + static_cast<double>(run)) / Z;
      if (fabs(u1 - cl) < kBoundary || fabs(u1 - chh) < kBoundary) sh.boundary += 1;
    }
    atomicMax(&sh.last_pos, lastpos);
  }
  __syncthreads();

  if (tid == 0) {
    int pick = sh.pick;
    if (pick < 0) {
      pick = sh.last_pos;
      sh.boundary += 1;
    }
    P.accepted_len[b] = jstar;
    tok[jstar] = pick;
    if (P.counters) {
      atomicAdd(P.counters + SV_CNT_TESTED, static_cast<unsigned long long>(jstar < k ? jstar + 1 : k));
      atomicAdd(P.counters + SV_CNT_ACCEPTED, static_cast<unsigned long long>(jstar));
      if (jstar < k) {
        atomicAdd(P.counters + (sh.stop_flag == SV_FLAG_NULL ? SV_CNT_NULL : SV_CNT_REJECTED), 1ull);
      } else {
        atomicAdd(P.counters + SV_CNT_BONUS, 1ull);
      }
      if (sh.boundary) atomicAdd(P.counters + SV_CNT_BOUNDARY, static_cast<unsigned long long>(sh.boundary));
      if (degenerate) atomicAdd(P.counters + SV_CNT_DEGENERATE, 1ull);
    }
  }
  if (tid < jstar) tok[tid] = sh.Dv[tid];
  if (tid > jstar && tid <= k) tok[tid] = -1;
}

// ----------------------------------------------------------- the kernel

template <typename TT, typename TD>
struct Stages {
  static constexpr int kBytes = kChunk * static_cast<int>(sizeof(TT) > sizeof(TD) ? sizeof(TT) : sizeof(TD));
  static constexpr int kDepth = kBytes <= 16384 ? 4 : 3;
  static constexpr int kMinBlocks = kBytes <= 16384 ? 3 : 2;
};

template <typename TT, typename TD>
__device__ __forceinline__ void issue_item(const Params& P, unsigned item, unsigned char* stage,
                                           int warp, int lane) {
  const int b = static_cast<int>(item / static_cast<unsigned>(P.items_per_seq));
  const int rem = static_cast<int>(item - static_cast<unsigned>(b) * P.items_per_seq);
  const int r = rem / P.nchunk;
  const int c0 = (rem - r * P.nchunk) * kChunk;
  if (r <= P.k) {
    if (P.vec_t)
      Chunk<TT>::issue(static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (P.k + 1) + r) * P.V,
                       stage, c0, P.V, warp, lane);
  } else {
    if (P.vec_d)
      Chunk<TD>::issue(static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * P.k + (r - P.k - 1)) * P.V,
                       stage, c0, P.V, warp, lane);
  }
}

// one work item: chunk statistics, drafted-token logit, gate candidates, and
// the publication of all of it.  On entry *ticket / ticket_b (thread 0) hold
// the completion count the previous item observed and its sequence; *fin_out
// returns, to every thread, the sequence that previous item completed (or -1),
// and *ticket the count this item observes.
template <typename T>
__device__ __forceinline__ void process_item(const Params& P, Shared& sh, const T* row,
                                             const unsigned char* stage, int b, int r, int ch,
                                             bool is_draft, int tid, int warp, int lane,
                                             unsigned* ticket, int ticket_b, int* fin_out) {
  const int k = P.k;
  const int c0 = ch * kChunk;
  const bool vec = is_draft ? P.vec_d != 0 : P.vec_t != 0;
  const int j = is_draft ? r - k - 1 : r;
  int d = -1;
  if (tid == 0 && j < k) d = __ldg(P.D + static_cast<int64_t>(b) * k + j);

  Chunk<T> regs;
  regs.load(row, stage, c0, P.V, vec, warp, lane);
  const float mine = regs.max();
  const float mw = warp_max(mine);
  if (lane == 0) sh.red_max[warp] = mw;
  __syncthreads();
  float m_c = sh.red_max[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) m_c = fmaxf(m_c, sh.red_max[w]);
  const float s_t = warp_sum(regs.expsum(m_c == -INFINITY ? 0.f : m_c, P.c));
  if (lane == 0) sh.red_sum[warp] = s_t;
  if (tid == 0)  // the previous item's completion count has had a whole item to return
    sh.fin_b = (ticket_b >= 0 && *ticket == static_cast<unsigned>(P.items_per_seq - 1)) ? ticket_b : -1;
  __syncthreads();
  float s_c = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) s_c += sh.red_sum[w];
  *fin_out = sh.fin_b;

  bool want_cand = false;
  if (is_draft) {
    const float tau = seq_tau(P, b);
    want_cand = seq_gated(P, b) && gate_fast_path(tau);
    if (want_cand) {
      // tokens with in-chunk probability >= slack * tau: a superset of the
      // admitted set (q <= in-chunk probability), at most 1/(slack tau) of them
      float thr = INFINITY;
      if (s_c > 0.f && isfinite(s_c)) thr = m_c + log2f(tau * kGateSlack * s_c) / P.c;
      if (mine >= thr) {
        regs.for_each(c0, warp, lane, [&](int v, float x) {
          if (x >= thr && v < P.V) {
            const int slot = atomicAdd(&sh.ncand, 1);
            if (slot < kTopM) {
              sh.cand_v[slot] = x;
              sh.cand_i[slot] = v;
            }
          }
        });
      }
      __syncthreads();
    }
  }

  if (tid == 0) {
    const int R = P.rows;
    P.part[(static_cast<int64_t>(b) * R + r) * P.nchunk + ch] = make_float2(m_c, s_c);
    if (d >= c0 && d < c0 + kChunk && d < P.V) {
      constexpr int kVE = Chunk<T>::kVE;
      const int v0 = d - (d - c0) % kVE;
      const float x = (vec && v0 + kVE <= P.V) ? (sizeof(T) == 2
                          ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(stage)[d - c0]) << 16)
                          : reinterpret_cast<const float*>(stage)[d - c0])
                                              : logit_at<T>(row, d);
      P.xD[static_cast<int64_t>(b) * R + r] = x;
    }
    if (want_cand) {
      const int n = sh.ncand;
      if (n > 0) {
        const int64_t rowc = static_cast<int64_t>(b) * k + j;
        const unsigned add = n > kTopM ? static_cast<unsigned>(kRowCap + 1) : static_cast<unsigned>(n);
        const unsigned base = atomicAdd(P.cand_n + rowc, add);
        if (n <= kTopM)
          for (int s = 0; s < n; ++s)
            if (base + s < static_cast<unsigned>(kRowCap)) {
              P.cand_v[rowc * kRowCap + base + s] = sh.cand_v[s];
              P.cand_i[rowc * kRowCap + base + s] = sh.cand_i[s];
            }
      }
      sh.ncand = 0;
    }
    *ticket = atom_add_acq_rel(P.seq_done + b, 1u);
  }
}

template <typename TT, typename TD>
__global__ void __launch_bounds__(kThreads, Stages<TT, TD>::kMinBlocks) verify_kernel(const Params P) {
  constexpr int S = Stages<TT, TD>::kDepth;
  constexpr int kStage = Stages<TT, TD>::kBytes;
  extern __shared__ __align__(128) unsigned char stages[];
  __shared__ Shared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned total = P.total_items;
  const int k = P.k, nch = P.nchunk;

  if (tid == 0) {
    sh.ncand = 0;
    sh.fin_b = -1;
    for (int s = 0; s <= S; ++s) sh.ring[s] = atomicAdd(P.work, 1u);
  }
  __syncthreads();
#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    const unsigned it_idx = sh.ring[s];
    if (it_idx < total) issue_item<TT, TD>(P, it_idx, stages + s * kStage, warp, lane);
    cp_async_commit();
  }

  unsigned pending = 0;   // thread 0: item index fetched one iteration ago
  unsigned ticket = 0;    // thread 0: completion count seen by the last item
  int ticket_b = -1;      // thread 0: sequence of the last item
  int fin = -1;           // sequence to finish (broadcast during the next item)
  for (int it = 0;; ++it) {
    const unsigned cur = sh.ring[it % kRing];
    if (cur >= total) break;
    {
      const unsigned nx = sh.ring[(it + S - 1) % kRing];
      if (nx < total) issue_item<TT, TD>(P, nx, stages + ((it + S - 1) % S) * kStage, warp, lane);
      cp_async_commit();
    }
    if (tid == 0) {
      if (it > 0) sh.ring[(it + S) % kRing] = pending;
      pending = atomicAdd(P.work, 1u);
    }
    cp_async_wait<S - 1>();

    const int b = static_cast<int>(cur / static_cast<unsigned>(P.items_per_seq));
    const int rem = static_cast<int>(cur - static_cast<unsigned>(b) * P.items_per_seq);
    const int r = rem / nch;
    const int ch = rem - r * nch;
    const unsigned char* stage = stages + (it % S) * kStage;
    if (r <= k) {
      const TT* row = static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (k + 1) + r) * P.V;
      process_item<TT>(P, sh, row, stage, b, r, ch, false, tid, warp, lane, &ticket, ticket_b, &fin);
    } else {
      const TD* row = static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * k + (r - k - 1)) * P.V;
      process_item<TD>(P, sh, row, stage, b, r, ch, true, tid, warp, lane, &ticket, ticket_b, &fin);
    }
    if (tid == 0) ticket_b = b;
    if (fin >= 0) {  // uniform: every thread read sh.fin_b after the same barrier
      finish_sequence<TT, TD>(P, fin, sh);
      if (tid == 0) P.seq_done[fin] = 0u;  // ready for the next call
      __syncthreads();
    }
  }
  // the last item's completion
  if (tid == 0) {
    sh.fin_b = (ticket_b >= 0 && ticket == static_cast<unsigned>(P.items_per_seq - 1)) ? ticket_b : -1;
    sh.ring[0] = pending;  // consume the outstanding fetch
  }
  __syncthreads();
  fin = sh.fin_b;
  if (fin >= 0) {
    finish_sequence<TT, TD>(P, fin, sh);
    if (tid == 0) P.seq_done[fin] = 0u;
  }
  cp_async_wait<0>();
  if (tid == 0) {
    __threadfence();
    const unsigned e = atomicAdd(P.exit_count, 1u);
    if (e == gridDim.x - 1) {  // every CTA has stopped fetching: reset for the next call
      atomicExch(P.work, 0u);
      atomicExch(P.exit_count, 0u);
    }
  }
}

}  // namespace sv
