// Batched speculative-decoding verification kernels for sm_103a.
//
// A call is two launches on one stream:
//
// stream_kernel -- the bandwidth-bound pass.  Rows are cut into chunks of
//   kChunk = 2048 vocabulary entries; rows 0..k of a sequence are its target
//   rows, rows k+1..2k its draft rows.  One CTA per SM; every warp works on
//   its own: it takes its CTA's chunks one at a time from a shared-memory
//   counter, streams them through a private cp.async ring of S chunk stages
//   in shared memory (each lane copies and later reads back its own 16-byte
//   slots, so no barrier is involved after the start), and per
//   chunk publishes the chunk statistics of the temperature softmax (mlxcel PR
//   #992, "What changed": p and q are full-vocabulary temperature softmaxes in
//   fp32), the logit at the drafted token when that token lies in the chunk,
//   and -- for draft rows of gated sequences -- the tokens whose in-chunk
//   probability reaches the gate (at most floor(1/threshold) of them, a
//   superset of the tokens the gate admits).
//
// finish_kernel -- one CTA per sequence, launched as a programmatic dependent
//   launch so that its start-up overlaps the end of the stream pass.  It
//   combines the chunk statistics into row statistics, evaluates every draft
//   position -- gate, retained measure mu, alpha = min(1, p(D)/mu(D)), Philox
//   u0, the accept test p > 0 && u0 * mu <= p (Strata PR #3416, "Approach";
//   mlxcel PR #992, "What changed") -- stops at the first position not
//   accepted, and samples the stop row: the normalised positive part of p - mu
//   after a rejection or NULL, p itself for the bonus row.  Chunk sums of the
//   residual come from the chunk statistics (minus the admitted tokens'
//   min(p, q) in gated mode), a prefix over chunks finds the chunk holding
//   u1 * Z, and one re-read of that chunk with a block-wide scan finds the
//   token.  Plain-mode rejections need q everywhere, so they re-read the stop
//   row pair once to form the chunk sums.
//
// Row statistics live in a scaled log2 domain: with c = log2(e) / T, a chunk
// with raw maximum m stores mc = fl(m * c) and s = sum_v exp2(fma(x_v, c, -mc)),
// and a token's probability is exp2(fma(x, c, -Mc)) / S for the row's (Mc, S).
// One FFMA per entry, and the stored reference mc is exactly the one removed.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include <cooperative_groups.h>

#include "philox.cuh"
#include "spec_verify.h"

namespace sv {

namespace cg = cooperative_groups;

constexpr int kChunk = 2048;                // vocabulary entries per chunk statistic
constexpr int kTopM = 4;                    // gate candidate slots per chunk / admitted tokens per row
constexpr int kMaxChunks = (SV_MAX_V + kChunk - 1) / kChunk;
constexpr int kMaxRows = 2 * SV_MAX_K + 1;
constexpr float kBoundary = 1e-6f;
// Candidates are kept against a threshold lowered by this factor so that
// rounding cannot drop an admitted token; the gated fast path needs
// slack * threshold * (kTopM + 1) > 1, i.e. threshold > ~0.2002.
constexpr float kGateSlack = 1.0f - 1.0f / 1024.0f;

// Kernel variants, chosen per call on the host: the sampling rule, the same
// with a gate policy (per-step thresholds and/or a cumulative floor), and
// greedy decoding (temperature 0, which honours the policy too).  Each is its
// own instantiation, so the plain sampling path carries no policy code.
// kModeStats is the stream pass alone (chunk statistics and drafted-token
// logits, no gate candidates), for the acceptance diagnostics and the sampler
// filters.  kModeGather is the sampler filters' gathering pass: every chunk
// keeps the logits at or above its row's lower bound (see process_chunk_gather).
enum : int { kModeSample = 0, kModePolicy = 1, kModeGreedy = 2, kModeStats = 3, kModeGather = 4 };

// gathered logits kept per chunk by the gathering pass (more: the row's
// selection reads the whole row itself)
constexpr int kGatherCap = 32;

struct Cand {  // a gate candidate: raw logit and token id (id -1: empty slot)
  float x;
  int v;
};

// floor(n / d) for a divisor fixed per call, as a multiply-high and a shift
// (Granlund & Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, the round-up variant): with s = ceil(log2 d)
// and m = floor(2^32 (2^s - d) / d) + 1, floor(n / d) = (mulhi(n, m) + n) >> s
// for every 32-bit n.
struct FastDiv {
  unsigned d, m, s;
};
__host__ __device__ inline FastDiv make_fastdiv(unsigned d) {
  unsigned s = 0;
  while ((1ull << s) < d) ++s;
  const unsigned long long m = ((1ull << 32) * ((1ull << s) - d)) / d + 1;
  return FastDiv{d, static_cast<unsigned>(m), s};
}
__device__ __forceinline__ unsigned fastdiv(unsigned n, const FastDiv& f) {
  return static_cast<unsigned>((static_cast<unsigned long long>(__umulhi(n, f.m)) + n) >> f.s);
}

struct Params {
  const void* Lt;  // [B, k+1, V]
  const void* Ld;  // [B, k, V]
  const int32_t* D;
  int B, k, V, nchunk, rows;
  unsigned total_chunks;  // B * rows * nchunk
  FastDiv div_nchunk, div_rows;
  float c;     // log2(e) / T, rounded once (0 when greedy)
  float T;
  int greedy;  // T = 0: one-hot p and q at each row's first largest logit
  int gate_default;
  float tau_default;
  const uint8_t* gate_per_seq;
  const float* tau_per_seq;
  // gate policy of the gated sequences: per-step thresholds that replace the
  // sequence's own (has_sched), and the cumulative floor on the drafted
  // prefix's product of draft probabilities (0: off)
  int has_sched;
  float min_cum;
  float tau_step[SV_MAX_K];
  uint64_t seed, seq_offset;
  const float* u0;
  const float* u1;
  int32_t* accepted_len;
  int32_t* tokens;
  float* alpha;
  int8_t* flags;
  unsigned long long* counters;
  float* row_stats;
  // the sampler filters' gathering pass (kModeGather): per chunk up to
  // kGatherCap logits x with fl(x c) >= the row's bound (passed in fthr), and
  // how many there were
  float* glist;        // [B * rows * nchunk, kGatherCap]
  unsigned* gcount;    // [B * rows * nchunk]
  // workspace
  float2* part;        // [B, rows, nchunk] (mc, s) per chunk
  float* xD;           // [B, rows] raw logit at the drafted token (rows j < k and draft rows)
  Cand* cand;          // [B, k, nchunk, kTopM] gate candidates of draft rows; emptied by the finisher
  unsigned* cand_over; // [B, k] a chunk had more than kTopM candidates; cleared by the finisher
  int vec_t, vec_d;    // rows allow 16-byte vector loads
  // finishing grid: CTAs [0, fin_warm) run the finishing code once, writing
  // nothing, while the stream pass drains (see finish_kernel)
  int fin_warm;
  // sampler filters, per row g = b * rows + r (null: the call has none): the
  // row keeps its logits x >= fthr[g] (-inf keeps every one), or -- when
  // ffirst[g] >= 0, a top_k = 1 row -- only the entry at index ffirst[g]; the
  // others read as -inf
  const float* fthr;
  const int* ffirst;
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float2 ldcg_f2(const float2* p) { return __ldcg(p); }

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two fp32 values in one 64-bit register pair, for the packed fp32x2 FMA of
// sm_100 and later: one instruction computes both lanes, each rounded exactly
// as the scalar fma would round it.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_pack(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(f32x2 r) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
  return make_float2(a, b);
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
__device__ __forceinline__ int warp_excl_scan_int(int v, int lane, int& total) {
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - v;
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

// probability of a token with raw logit x in a row with scaled max Mc and
// 1/sum invS: exp2(fma(x, c, -Mc)) * invS.  Every decision uses this formula.
// The product is rounded on its own (__fmul_rn is never fused into a later
// add): p - q of two equal rows is then exactly 0, where a fused
// fma(e, invS, -q) would leave q's rounding error as residual mass.
__device__ __forceinline__ float prob_of(float x, float Mc, float c, float invS) {
  return __fmul_rn(exp2f(fmaf(x, c, -Mc)), invS);
}

// A gated stop row's residual per chunk is the chunk's mass (from its
// statistics, relative rounding error below 5e-6: a 64-term sum per lane,
// five merge levels, three more roundings) minus its admitted tokens'
// min(p, q).  A remainder within kResidualTol of the chunk's mass is that
// rounding, not mass: the chunk counts as empty.
constexpr float kResidualTol = 1e-5f;

__device__ __forceinline__ bool gate_fast_path(float tau) {
  return tau * kGateSlack * static_cast<float>(kTopM + 1) > 1.0f;
}

__device__ __forceinline__ bool seq_gated(const Params& P, int b) {
  return P.gate_per_seq ? (P.gate_per_seq[b] != 0) : (P.gate_default != 0);
}
__device__ __forceinline__ float seq_tau(const Params& P, int b) {
  return P.tau_per_seq ? P.tau_per_seq[b] : P.tau_default;
}
// the gate threshold of step j of sequence b: the schedule's entry when the
// policy has one, else the sequence's threshold
__device__ __forceinline__ float step_tau(const Params& P, int b, int j) {
  return P.has_sched ? P.tau_step[j] : seq_tau(P, b);
}
// a floor under everything the gate can require of q at step j: q >= tau_j,
// and q >= cprev * q >= min_cum because the prefix product cprev is at most 1;
// the stream pass keeps candidates against it
__device__ __forceinline__ float step_floor(const Params& P, int b, int j) {
  return fmaxf(step_tau(P, b, j), P.min_cum);
}
// gate admission of a token with draft probability q at a step with
// threshold tau behind a prefix product cprev: both floors, equality passes
// (cum: the policy has a cumulative floor)
__device__ __forceinline__ bool gate_admits(float q, float tau, float cprev, bool cum, float min_cum) {
  return q >= tau && (!cum || cprev * q >= min_cum);
}

// ---- sampler filters applied on the fly (see Params::fthr)

// one logit x at index v of a row with filter (thr, first)
__device__ __forceinline__ float filt1(float x, int v, float thr, int first) {
  if (first >= 0) return v == first ? x : -INFINITY;
  return x < thr ? -INFINITY : x;  // ordered: a NaN stays (the row is then invalid)
}
// eight consecutive logits [v0, v0 + 8)
__device__ __forceinline__ void filt8(float (&x)[8], int v0, float thr, int first) {
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = filt1(x[e], v0 + e, thr, first);
}
// the smallest bf16 value >= thr, as bf16 bits in both halves of a word: for
// bf16 logits x, x >= thr iff x >= that value
__device__ __forceinline__ uint32_t bf16_ceil_pair(float thr) {
  const uint32_t u = __float_as_uint(thr);
  uint32_t h = u >> 16;
  // dropped low bits: truncation lowered a positive value (round its
  // magnitude up) and raised a negative one (already above thr)
  if ((u & 0xffffu) != 0u && !(u & 0x80000000u)) h += 1u;
  return h | (h << 16);
}

// ------------------------------------------------------- chunk registers
//
// A warp holds one chunk: lane l owns NV 16-byte slots, slot i being vector
// index 32 i + l of the chunk (each copy instruction of the warp moves 512
// contiguous bytes).  bf16 entries stay packed in pairs.  The stage always ends
// up holding the whole chunk: 16-byte slots inside the row arrive by cp.async,
// slots past V are filled with -inf, and a partial last slot -- or every slot
// of a row that is not 16-byte aligned -- is read directly.

template <typename T> struct Lane;

template <> struct Lane<uint16_t> {
  static constexpr int kVE = 8;
  static constexpr int kNV = kChunk / 32 / kVE;  // 8 slots, 64 entries
  uint32_t w[4 * kNV];
  __device__ __forceinline__ static void issue(const uint16_t* row, unsigned char* stage, int c0, int V,
                                               bool vec, int lane) {
    if (vec && c0 + kChunk <= V) {
#pragma unroll
      for (int i = 0; i < kNV; ++i) cp_async16(stage + (32 * i + lane) * 16, row + c0 + (32 * i + lane) * kVE);
      return;
    }
#pragma unroll 1
    for (int i = 0; i < kNV; ++i) {
      const int sv = 32 * i + lane;
      const int v0 = c0 + sv * kVE;
      if (vec && v0 + kVE <= V) {
        cp_async16(stage + sv * 16, row + v0);
      } else {
        uint32_t t[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int a = v0 + 2 * q;
          const uint32_t lo = a < V ? static_cast<uint32_t>(__ldg(row + a)) : 0xFF80u;
          const uint32_t hi = a + 1 < V ? static_cast<uint32_t>(__ldg(row + a + 1)) : 0xFF80u;
          t[q] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(stage + sv * 16) = make_uint4(t[0], t[1], t[2], t[3]);
      }
    }
  }
  __device__ __forceinline__ void load(const unsigned char* stage, int lane) {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const uint4 u = *reinterpret_cast<const uint4*>(stage + (32 * i + lane) * 16);
      w[4 * i + 0] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
    }
  }
  __device__ __forceinline__ float max() const {
    uint32_t m0 = w[0], m1 = w[1];
#pragma unroll
    for (int q = 2; q < 4 * kNV; q += 2) {
      m0 = bmax2(m0, w[q]);
      m1 = bmax2(m1, w[q + 1]);
    }
    const uint32_t m = bmax2(m0, m1);
    return fmaxf(bf16_lo(m), bf16_hi(m));
  }
  // f(slot, entry, value) for every entry, in increasing index order
  template <class F>
  __device__ __forceinline__ void visit(F&& f) const {
#pragma unroll
    for (int i = 0; i < kNV; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f(i, 2 * q, bf16_lo(w[4 * i + q]));
        f(i, 2 * q + 1, bf16_hi(w[4 * i + q]));
      }
  }
  // sum_v exp2(fma(x_v, c, nmc)), four independent accumulators; the fma
  // goes two lanes per instruction (packed fp32x2, each lane rounded as the
  // scalar fma).  Packed adds for the accumulators measured slower on long
  // streams (1024 x 262144 bf16), so the adds stay scalar.
  __device__ __forceinline__ float expsum(float c, float nmc) const {
    const f32x2 cc = f2_pack(c, c), nn = f2_pack(nmc, nmc);
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int q = 0; q < 4 * kNV; q += 2) {
      const float2 t01 = f2_unpack(f2_fma(f2_pack(bf16_lo(w[q]), bf16_hi(w[q])), cc, nn));
      const float2 t23 = f2_unpack(f2_fma(f2_pack(bf16_lo(w[q + 1]), bf16_hi(w[q + 1])), cc, nn));
      a0 += ex2_approx(t01.x);
      a1 += ex2_approx(t01.y);
      a2 += ex2_approx(t23.x);
      a3 += ex2_approx(t23.y);
    }
    return (a0 + a1) + (a2 + a3);
  }
  // sampler filter: entries below the threshold (both halves of thr2 hold its
  // bf16 ceiling) become -inf; the ordered compare keeps a NaN
  __device__ __forceinline__ void mask(uint32_t thr2) {
#pragma unroll
    for (int q = 0; q < 4 * kNV; ++q) {
      uint32_t m;
      asm("set.lt.u32.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(w[q]), "r"(thr2));
      w[q] = (w[q] & ~m) | (0xFF80FF80u & m);
    }
  }
  // a top_k = 1 row: every entry but chunk offset o_keep becomes -inf
  __device__ __forceinline__ void keep_only(int o_keep, int lane) {
#pragma unroll
    for (int i = 0; i < kNV; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int o = (32 * i + lane) * kVE + 2 * q;
        const uint32_t lo = o == o_keep ? 0x0000ffffu : 0u, hi = o + 1 == o_keep ? 0xffff0000u : 0u;
        w[4 * i + q] = (w[4 * i + q] & (lo | hi)) | (0xFF80FF80u & ~(lo | hi));
      }
  }
  // entries x of slot i with fma(x, c, nmc) >= lts, as a bit mask
  __device__ __forceinline__ unsigned slot_hits(int i, float c, float nmc, float lts) const {
    unsigned m = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      m |= (fmaf(bf16_lo(w[4 * i + q]), c, nmc) >= lts ? 1u : 0u) << (2 * q);
      m |= (fmaf(bf16_hi(w[4 * i + q]), c, nmc) >= lts ? 1u : 0u) << (2 * q + 1);
    }
    return m;
  }
};

template <> struct Lane<float> {
  static constexpr int kVE = 4;
  static constexpr int kNV = kChunk / 32 / kVE;  // 16 slots, 64 entries
  float x[4 * kNV];
  __device__ __forceinline__ static void issue(const float* row, unsigned char* stage, int c0, int V,
                                               bool vec, int lane) {
    if (vec && c0 + kChunk <= V) {
#pragma unroll
      for (int i = 0; i < kNV; ++i) cp_async16(stage + (32 * i + lane) * 16, row + c0 + (32 * i + lane) * kVE);
      return;
    }
#pragma unroll 1
    for (int i = 0; i < kNV; ++i) {
      const int sv = 32 * i + lane;
      const int v0 = c0 + sv * kVE;
      if (vec && v0 + kVE <= V) {
        cp_async16(stage + sv * 16, row + v0);
      } else {
        float t[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) t[e] = v0 + e < V ? __ldg(row + v0 + e) : -INFINITY;
        *reinterpret_cast<float4*>(stage + sv * 16) = make_float4(t[0], t[1], t[2], t[3]);
      }
    }
  }
  __device__ __forceinline__ void load(const unsigned char* stage, int lane) {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const float4 u = *reinterpret_cast<const float4*>(stage + (32 * i + lane) * 16);
      x[4 * i + 0] = u.x; x[4 * i + 1] = u.y; x[4 * i + 2] = u.z; x[4 * i + 3] = u.w;
    }
  }
  __device__ __forceinline__ float max() const {
    float m0 = fmaxf(x[0], x[1]), m1 = fmaxf(x[2], x[3]);
#pragma unroll
    for (int e = 4; e < 4 * kNV; e += 4) {
      m0 = fmaxf(m0, fmaxf(x[e], x[e + 1]));
      m1 = fmaxf(m1, fmaxf(x[e + 2], x[e + 3]));
    }
    return fmaxf(m0, m1);
  }
  template <class F>
  __device__ __forceinline__ void visit(F&& f) const {
#pragma unroll
    for (int i = 0; i < kNV; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) f(i, e, x[4 * i + e]);
  }
  __device__ __forceinline__ float expsum(float c, float nmc) const {
    const f32x2 cc = f2_pack(c, c), nn = f2_pack(nmc, nmc);
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int e = 0; e < 4 * kNV; e += 4) {
      const float2 t01 = f2_unpack(f2_fma(f2_pack(x[e], x[e + 1]), cc, nn));
      const float2 t23 = f2_unpack(f2_fma(f2_pack(x[e + 2], x[e + 3]), cc, nn));
      a0 += ex2_approx(t01.x);
      a1 += ex2_approx(t01.y);
      a2 += ex2_approx(t23.x);
      a3 += ex2_approx(t23.y);
    }
    return (a0 + a1) + (a2 + a3);
  }
  __device__ __forceinline__ unsigned slot_hits(int i, float c, float nmc, float lts) const {
    unsigned m = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) m |= (fmaf(x[4 * i + e], c, nmc) >= lts ? 1u : 0u) << e;
    return m;
  }
  // sampler filter: entries below the threshold become -inf (a NaN stays)
  __device__ __forceinline__ void mask(float thr) {
#pragma unroll
    for (int e = 0; e < 4 * kNV; ++e) x[e] = x[e] < thr ? -INFINITY : x[e];
  }
  __device__ __forceinline__ void keep_only(int o_keep, int lane) {
#pragma unroll
    for (int i = 0; i < kNV; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((32 * i + lane) * kVE + e != o_keep) x[4 * i + e] = -INFINITY;
  }
};

// ------------------------------------------------------- stream kernel

// launch shape of the stream pass: independent warps per CTA, each with a
// ring of kDepth chunk stages
template <typename TT, typename TD>
struct Stages {
  static constexpr int kBytes = kChunk * static_cast<int>(sizeof(TT) > sizeof(TD) ? sizeof(TT) : sizeof(TD));
  // one CTA per SM: 16 warps with two 4 KB stages each (bf16 rows, 128 KB of
  // rings), 8 warps with three 8 KB stages otherwise (192 KB).  For bf16 rows
  // two stages measured faster than three on the 128K-vocabulary batch
  // (40.8 against 41.4 us per step): each warp holds less unfinished work when
  // its CTA's chunks run out, and 16 warps still keep ~19 MB in flight.
  static constexpr int kDepth = kBytes <= 4096 ? 2 : 3;
  static constexpr int kWarpsPerCta = kBytes <= 4096 ? 16 : 8;
  static constexpr int kThreadsPerCta = 32 * kWarpsPerCta;
  static constexpr int kMinBlocks = 1;
};

// ---- work distribution
//
// The stream pass's work is the list of all chunks, sequence-major: chunk
// index x = (b * rows + r) * nchunk + ch.  The grid holds one CTA per SM, and
// CTA c owns chunks c, c + NC, c + 2 NC, ... (NC CTAs), so the grid sweeps
// memory front to back and every SM gets the same share.  Inside a CTA the
// warps take the CTA's chunks one at a time from a shared-memory counter.
// Measured on this part: warps on one SM drift apart by several
// microseconds, so balancing inside the SM pays; SMs given equal shares end
// up to a few microseconds apart, at random from call to call, but handing
// out work across SMs takes global atomics, whose replies under the logits
// stream come back too late (a stream of them as the work queue, or only for
// the last part of the work, made the pass slower), so none are used.

constexpr int kItemRing = 8;       // decoded chunks known to a warp (in flight or next)
constexpr unsigned kNoWork = 0xffffffffu;

struct WarpQueue {
  int4 item[kItemRing];  // (b, r, ch, 1) of a chunk to stream; w = 0: no more work
  int d[kItemRing];      // the drafted token of the chunk's row (rows j < k), copied asynchronously
};
// a filtered call's queue also holds each chunk's row filter (threshold, kept index)
struct WarpQueueFilt : WarpQueue {
  float fthr[kItemRing];
  int ffirst[kItemRing];
};

// lane 0: the warp's next chunk index, or kNoWork
__device__ __forceinline__ unsigned next_chunk(const Params& P, unsigned* cta_next) {
  const unsigned i = atomicAdd(cta_next, 1u);
  const unsigned long long x = blockIdx.x + static_cast<unsigned long long>(i) * gridDim.x;
  return x < P.total_chunks ? static_cast<unsigned>(x) : kNoWork;
}

// lane 0: decode chunk index x into item slot `slot` and start the copy of
// its drafted token (and, kFilt, of its row's filter)
template <bool kFilt, typename Queue>
__device__ __forceinline__ void put_item(const Params& P, Queue& Q, int slot, unsigned x) {
  if (x == kNoWork) {
    Q.item[slot] = make_int4(0, 0, 0, 0);
    return;
  }
  const unsigned rg = fastdiv(x, P.div_nchunk);
  const int ch = static_cast<int>(x - rg * static_cast<unsigned>(P.nchunk));
  const unsigned b = fastdiv(rg, P.div_rows);
  const int r = static_cast<int>(rg - b * static_cast<unsigned>(P.rows));
  Q.item[slot] = make_int4(static_cast<int>(b), r, ch, 1);
  const int j = r <= P.k ? r : r - P.k - 1;
  if (j < P.k) cp_async4(&Q.d[slot], P.D + static_cast<int64_t>(b) * P.k + j);
  if constexpr (kFilt) {
    cp_async4(&Q.fthr[slot], P.fthr + rg);
    cp_async4(&Q.ffirst[slot], P.ffirst + rg);
  }
}

// a hint: the line holding p is brought into L2 (no data returned, no effect
// on what any later load reads)
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// How many of a CTA's first chunks the stream pass prefetches into L2 before
// its programmatic wait, per warp.  While the previous call's finishing pass
// runs and this grid's wait is released, DRAM is nearly idle; each warp's
// first copy then finds its lines in L2.  Measured on the 128K-vocabulary
// batch (64 sequences, k = 5, bf16): 39.3 us per step without, 38.8 us with
// one chunk per warp, 39.0 us with two (a full ring), 40.3 us with four --
// deeper prefetches slow the step.
constexpr int kPrefetchPerWarp = 1;

// Warp `warp` of the CTA prefetches chunks i = warp, warp + W, ... < n of the
// CTA's share (chunk index blockIdx.x + i gridDim.x), one 128-byte line per
// lane and step, every address inside the chunk's row.  The addresses come
// from the launch arguments alone: nothing is read.
template <typename TT, typename TD>
__device__ __forceinline__ void prefetch_first_chunks(const Params& P, int n, int warp, int lane) {
  constexpr int W = Stages<TT, TD>::kWarpsPerCta;
  for (int i = warp; i < n; i += W) {
    const unsigned long long x = blockIdx.x + static_cast<unsigned long long>(i) * gridDim.x;
    if (x >= P.total_chunks) break;
    const unsigned rg = fastdiv(static_cast<unsigned>(x), P.div_nchunk);
    const int ch = static_cast<int>(static_cast<unsigned>(x) - rg * static_cast<unsigned>(P.nchunk));
    const unsigned b = fastdiv(rg, P.div_rows);
    const int r = static_cast<int>(rg - b * static_cast<unsigned>(P.rows));
    const int c0 = ch * kChunk;
    const int len = min(kChunk, P.V - c0);
    const char* base;
    int bytes;
    if (r <= P.k) {
      base = static_cast<const char*>(P.Lt) +
             ((static_cast<int64_t>(b) * (P.k + 1) + r) * P.V + c0) * static_cast<int64_t>(sizeof(TT));
      bytes = len * static_cast<int>(sizeof(TT));
    } else {
      base = static_cast<const char*>(P.Ld) +
             ((static_cast<int64_t>(b) * P.k + (r - P.k - 1)) * P.V + c0) * static_cast<int64_t>(sizeof(TD));
      bytes = len * static_cast<int>(sizeof(TD));
    }
    for (int o = lane * 128; o < bytes; o += 32 * 128) prefetch_l2(base + o);
  }
}

template <typename TT, typename TD>
__device__ __forceinline__ void issue_chunk(const Params& P, int b, int r, int ch, unsigned char* stage,
                                            int lane) {
  const int c0 = ch * kChunk;
  if (r <= P.k)
    Lane<TT>::issue(static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (P.k + 1) + r) * P.V,
                    stage, c0, P.V, P.vec_t != 0, lane);
  else
    Lane<TD>::issue(static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * P.k + (r - P.k - 1)) * P.V,
                    stage, c0, P.V, P.vec_d != 0, lane);
}

// entry o of a staged chunk as float
template <typename T>
__device__ __forceinline__ float stage_logit(const unsigned char* stage, int o) {
  if constexpr (sizeof(T) == 2)
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(stage)[o]) << 16);
  else
    return reinterpret_cast<const float*>(stage)[o];
}

// one chunk of a greedy call (temperature 0), by one warp: the chunk's largest
// logit and the first index holding it, or index -1 when the chunk holds a
// NaN or +inf logit (!(x <= FLT_MAX) holds exactly for those; -inf is allowed)
template <typename T>
__device__ __forceinline__ void process_chunk_greedy(const Params& P, const unsigned char* stage, int b,
                                                     int r, int ch, int lane) {
  Lane<T> regs;
  regs.load(stage, lane);
  const float m = warp_max(regs.max());
  int first = kChunk;
  bool nonfinite = false;
  regs.visit([&](int i, int e, float x) {
    const int o = (32 * i + lane) * Lane<T>::kVE + e;
    if (x == m && o < first) first = o;
    nonfinite |= !(x <= 3.402823466e38f);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
  const bool bad = __any_sync(0xffffffffu, nonfinite);
  if (lane == 0)
    P.part[(static_cast<int64_t>(b) * P.rows + r) * P.nchunk + ch] =
        make_float2(m, __int_as_float(bad ? -1 : ch * kChunk + first));
}

// one chunk of the sampler filters' gathering pass, by one warp: the logits x
// with fl(x c) >= th (the row's lower bound of its top-k set; +inf: a row
// that gathers nothing), up to kGatherCap of them in index order of the
// lanes' slots, and their count
template <typename T>
__device__ __forceinline__ void process_chunk_gather(const Params& P, const unsigned char* stage, int b, int r,
                                                     int ch, int lane, float th) {
  const int64_t x = (static_cast<int64_t>(b) * P.rows + r) * P.nchunk + ch;
  if (th == INFINITY) {
    if (lane == 0) P.gcount[x] = 0u;
    return;
  }
  Lane<T> regs;
  regs.load(stage, lane);
  unsigned hits[Lane<T>::kNV];
  int mine = 0;
#pragma unroll
  for (int i = 0; i < Lane<T>::kNV; ++i) {
    hits[i] = regs.slot_hits(i, P.c, 0.f, th);  // fma(x, c, 0) is fl(x c)
    mine += __popc(hits[i]);
  }
  int total;
  int slot = warp_excl_scan_int(mine, lane, total);
  float* out = P.glist + x * kGatherCap;
  if (mine > 0) {
#pragma unroll
    for (int i = 0; i < Lane<T>::kNV; ++i) {
      unsigned m = hits[i];
      while (m) {
        const int e = __ffs(m) - 1;
        m &= m - 1;
        if (slot < kGatherCap) out[slot] = stage_logit<T>(stage, (32 * i + lane) * Lane<T>::kVE + e);
        ++slot;
      }
    }
  }
  if (lane == 0) P.gcount[x] = static_cast<unsigned>(total);
}

// one chunk, by one warp: statistics, drafted-token logit, gate candidates
// (kFilt: of the row as its sampler filter leaves it, threshold fthr or kept
// index ffirst)
template <typename T, bool kPol, bool kCand, bool kFilt>
__device__ __forceinline__ void process_chunk(const Params& P, const unsigned char* stage, int b, int r,
                                              int ch, int d, int lane, float fthr, int ffirst) {
  const int k = P.k;
  const int c0 = ch * kChunk;
  const bool is_draft = r > k;
  const int j = is_draft ? r - k - 1 : r;

  Lane<T> regs;
  regs.load(stage, lane);
  if constexpr (kFilt) {
    if (ffirst >= 0) regs.keep_only(ffirst - c0, lane);
    else if constexpr (sizeof(T) == 2) regs.mask(bf16_ceil_pair(fthr));
    else regs.mask(fthr);
  }
  // each lane sums against its own reference fl(m_l c); the warp then merges
  const float mine = regs.max();
  const float mct = mine == -INFINITY ? -INFINITY : mine * P.c;
  float s_l = regs.expsum(P.c, mine == -INFINITY ? 0.f : -mct);
  const float mc = warp_max(mct);
  s_l = mct == -INFINITY ? s_l * 0.f : s_l * ex2_approx(mct - mc);
  const float s = warp_sum(s_l);
  if (lane == 0) P.part[(static_cast<int64_t>(b) * P.rows + r) * P.nchunk + ch] = make_float2(mc, s);

  // the logit at the drafted token, written by the lane whose slot holds it
  if (j < k && d >= c0 && d < c0 + kChunk && d < P.V) {
    const int sv = (d - c0) / Lane<T>::kVE;
    if ((sv & 31) == lane) {
      float x = stage_logit<T>(stage, d - c0);
      if constexpr (kFilt) x = filt1(x, d, fthr, ffirst);
      P.xD[static_cast<int64_t>(b) * P.rows + r] = x;
    }
  }

  // gated draft rows keep candidates only on the fast path (slack tau (kTopM + 1)
  // > 1), and a chunk can hold one only if s <= 1 / (slack tau) (the chunk's
  // largest term contributes 1 to s): s < kTopM + 1 rules out almost every
  // chunk before the row's gate settings are even read
  if (kCand && is_draft && s < static_cast<float>(kTopM + 1)) {
    const float tau = kPol ? step_floor(P, b, j) : seq_tau(P, b);
    if (seq_gated(P, b) && gate_fast_path(tau) && s > 0.f && isfinite(s)) {
      // a token's in-chunk probability exp2(fma(x, c, -mc)) / s reaches
      // slack * tau iff fma(x, c, -mc) >= lts = log2(slack tau s); that set is a
      // superset of the admitted tokens (q <= in-chunk probability) and holds
      // at most 1/(slack tau) tokens.  lts <= 0 is needed for any token at all,
      // which rules out almost every chunk at once (s is warp-uniform).
      const float lts = log2f(tau * kGateSlack * s);
      if (lts <= 0.f) {
        // lanes whose own maximum could reach it (a small margin absorbs the
        // rounding of mct - mc against the fused form)
        const bool maybe = mct - mc >= lts - 1.0f / 256.0f;
        int mine_n = 0;
        unsigned hits[Lane<T>::kNV];
#pragma unroll
        for (int i = 0; i < Lane<T>::kNV; ++i) {
          hits[i] = maybe ? regs.slot_hits(i, P.c, -mc, lts) : 0u;
          mine_n += __popc(hits[i]);
        }
        int total;
        int slot = warp_excl_scan_int(mine_n, lane, total);
        const int64_t base = ((static_cast<int64_t>(b) * k + j) * P.nchunk + ch) * kTopM;
        if (mine_n > 0) {
#pragma unroll
          for (int i = 0; i < Lane<T>::kNV; ++i) {
            unsigned m = hits[i];
            while (m) {
              const int e = __ffs(m) - 1;
              m &= m - 1;
              // the value comes from the stage (a register array indexed by a
              // run-time entry would go through local memory)
              const int o = (32 * i + lane) * Lane<T>::kVE + e;
              if (slot < kTopM) P.cand[base + slot] = Cand{stage_logit<T>(stage, o), c0 + o};
              ++slot;
            }
          }
        }
        if (lane == 0 && total > kTopM) P.cand_over[static_cast<int64_t>(b) * k + j] = 1u;
      }
    }
  }
}

// kFilt: the call's sampler filters are applied to every chunk as it is loaded
template <typename TT, typename TD, int kMode, bool kFilt>
__global__ void __launch_bounds__(Stages<TT, TD>::kThreadsPerCta, Stages<TT, TD>::kMinBlocks)
    stream_kernel(const __grid_constant__ Params P) {
  constexpr bool kPol = kMode == kModePolicy;
  constexpr bool kCand = kMode != kModeStats && kMode != kModeGather;
  constexpr int S = Stages<TT, TD>::kDepth;
  constexpr int kStage = Stages<TT, TD>::kBytes;
  extern __shared__ __align__(128) unsigned char stages[];
  using Queue = typename std::conditional<kFilt, WarpQueueFilt, WarpQueue>::type;
  __shared__ Queue queues[Stages<TT, TD>::kWarpsPerCta];
  __shared__ unsigned cta_next;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* ring = stages + warp * S * kStage;
  Queue& Q = queues[warp];
  const int k = P.k;

  // item n (the warp's n-th chunk) is decoded at step n - 1, issued into ring
  // slot n % S at step n (S - 1 steps ahead of its use) and consumed at loop
  // iteration n; the copy of its drafted token rides in the commit group of
  // step n - 1, so it has landed when the chunk has.
  if (threadIdx.x == 0) cta_next = 0u;
  __syncthreads();
  // This grid is itself a programmatic dependent launch: its CTAs may be
  // resident while the previous kernel in the stream (the producer of the
  // logits, or the previous call's finishing pass, which reads the workspace)
  // drains, and read no global memory before that kernel has completed.  Only
  // L2 prefetches of the first chunks go out before: a prefetch returns no
  // data, and a load after the wait reads what the producer wrote whether or
  // not the line was prefetched (L2 is where device writes become visible).
  prefetch_first_chunks<TT, TD>(P, kPrefetchPerWarp * Stages<TT, TD>::kWarpsPerCta, warp, lane);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Then the finishing grid may launch: its CTAs take SMs as this grid's CTAs
  // retire, run their input-only prologue (the inputs are complete: see the
  // wait above), and wait for this grid to complete and its memory to be
  // visible.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lane == 0) put_item<kFilt>(P, Q, 0, next_chunk(P, &cta_next));
  __syncwarp();
  int issued = 0;
  auto issue_next = [&]() {
    const int4 it = Q.item[issued % kItemRing];
    if (it.w > 0) issue_chunk<TT, TD>(P, it.x, it.y, it.z, ring + (issued % S) * kStage, lane);
    if (lane == 0) put_item<kFilt>(P, Q, (issued + 1) % kItemRing, it.w > 0 ? next_chunk(P, &cta_next) : kNoWork);
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
    const int d = Q.d[n % kItemRing];  // landed with the commit group of step n - 1
    float fthr = 0.f;  // likewise
    int ffirst = -1;
    if constexpr (kFilt) {
      fthr = Q.fthr[n % kItemRing];
      ffirst = Q.ffirst[n % kItemRing];
    }
    const unsigned char* stage = ring + (n % S) * kStage;
    if constexpr (kMode == kModeGreedy) {
      if (it.y <= k) process_chunk_greedy<TT>(P, stage, it.x, it.y, it.z, lane);
      else process_chunk_greedy<TD>(P, stage, it.x, it.y, it.z, lane);
    } else if constexpr (kMode == kModeGather) {
      // (the row's bound rides in the filter-threshold slot of the queue)
      if (it.y <= k) process_chunk_gather<TT>(P, stage, it.x, it.y, it.z, lane, fthr);
      else process_chunk_gather<TD>(P, stage, it.x, it.y, it.z, lane, fthr);
    } else if (it.y <= k) {
      process_chunk<TT, kPol, kCand, kFilt>(P, stage, it.x, it.y, it.z, d, lane, fthr, ffirst);
    } else {
      process_chunk<TD, kPol, kCand, kFilt>(P, stage, it.x, it.y, it.z, d, lane, fthr, ffirst);
    }
    __syncwarp();
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------ finishing
//
// The finishing pass runs once per sequence over a long, mostly straight code
// path, so it is written compactly (rolled loops, partials and residual
// weights staged in shared memory).  Its sums are float-float (an fp32 pair
// with ~2^-44 relative error, built from error-free two-sums): fp64 would be
// as precise, but fp64 is a narrow, long-latency pipe on this part and this
// path is all dependent steps.

constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kFinPartCap = 4096;  // chunk statistics of a sequence staged in shared memory
constexpr int kCandCap = 256;      // gate candidates of a sequence gathered in shared memory

struct dfloat {
  float hi, lo;
};
__device__ __forceinline__ dfloat df(float a) { return {a, 0.f}; }
// error-free sum (Knuth's two-sum), renormalised
__device__ __forceinline__ dfloat df_add(dfloat a, dfloat b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb) + (a.lo + b.lo);
  const float hi = s + e;
  return {hi, e - (hi - s)};
}
__device__ __forceinline__ dfloat df_sub(dfloat a, dfloat b) { return df_add(a, {-b.hi, -b.lo}); }
__device__ __forceinline__ dfloat df_mul(dfloat a, float b) {
  const float p = a.hi * b;
  const float e = fmaf(a.lo, b, fmaf(a.hi, b, -p));
  const float hi = p + e;
  return {hi, e - (hi - p)};
}
__device__ __forceinline__ bool df_lt(dfloat a, dfloat b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ bool df_le(dfloat a, dfloat b) { return a.hi < b.hi || (a.hi == b.hi && a.lo <= b.lo); }
__device__ __forceinline__ float df_f(dfloat a) { return a.hi + a.lo; }
__device__ __forceinline__ dfloat shfl_xor_df(dfloat v, int o) {
  return {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ dfloat shfl_up_df(dfloat v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ dfloat shfl_df(dfloat v, int src) {
  return {__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}
__device__ __forceinline__ dfloat warp_sum_df(dfloat v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
  return v;
}
// every lane computes the sum and selects it (no divergent branch between
// the shuffles)
__device__ __forceinline__ dfloat warp_incl_scan_df(dfloat v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const dfloat n = shfl_up_df(v, o);
    const dfloat t = df_add(v, n);
    v.hi = lane >= o ? t.hi : v.hi;
    v.lo = lane >= o ? t.lo : v.lo;
  }
  return v;
}

struct FinishShared {
  float2 part[kFinPartCap];  // the sequence's chunk statistics (when they fit)
  float tile[kMaxChunks];    // residual mass of every chunk of the stop row
  dfloat prefix[kMaxChunks]; // inclusive prefix sums of tile
  float rowM[kMaxRows];      // scaled row max Mc
  float rowInvS[kMaxRows];
  dfloat rowS[kMaxRows];
  float xD[kMaxRows];
  // inputs read before the stream pass has finished
  int Dv[SV_MAX_K];
  float u0[SV_MAX_K];
  float u1[SV_MAX_K + 1];    // the residual draw for every possible stop position
  int gated;
  float tau;                 // the sequence's threshold (no policy)
  float tau_j[SV_MAX_K];     // each step's gate threshold (policy, greedy)
  float cprev[SV_MAX_K];     // product of q_i(D_i) over i < j (cumulative floor only)
  unsigned fast_rows;        // draft rows whose admitted set comes from candidates
  // gate candidates gathered from the per-chunk slots
  int ncand;
  int cand_j[kCandCap];
  int cand_v[kCandCap];
  float cand_x[kCandCap];
  int nadm[SV_MAX_K];
  int adm_i[SV_MAX_K][kTopM];
  float adm_q[SV_MAX_K][kTopM];
  float adm_p[SV_MAX_K][kTopM];
  unsigned overflow_rows;    // draft rows whose admitted set is not fully known
  dfloat wtot[kFinWarps];
  int wlast[kFinWarps];
  int bad;
  int jstar;
  int stop_flag;
  int boundary;
  int tstar;
  int degenerate;
  int mode;
  int pick;
  dfloat before;
  dfloat Z;
  dfloat y;
  int fmode;  // the stop row's sampling mode (-1: the sequence is done)
  int dry;    // a warming run: global memory is read, never written
  int targ[kMaxRows];  // greedy calls: each row's first largest logit
  float fthr[kMaxRows];  // filtered calls: each row's sampler-filter threshold and kept index
  int ffirst[kMaxRows];
};

// residual weights of eight consecutive entries [v0, v0 + 8): max(0, p - mu)
// with mu = 0 (mode 0: the bonus row, or a residual without mass), mu = q on
// the admitted tokens listed (mode 1), or mu from the draft logits (mode 2:
// q where q >= tau and, with a policy, cprev q >= min_cum -- the gate's
// predicate; a plain row, or a policy without a cumulative floor, sets the
// unused floors to -1, which every q passes).  Entries past V weigh 0.
struct ResidualEval {
  int mode;
  float Mt, invSt, Md, invSd, c, tau, cprev, min_cum;
  int nadm;
  const int* adm_i;
  const float* adm_q;
};

template <bool kPol>
__device__ __forceinline__ void residual8(const ResidualEval& e, const float (&xt)[8], const float (&xd)[8],
                                          int v0, int V, float (&r)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float p = prob_of(xt[i], e.Mt, e.c, e.invSt);
    float mu = 0.f;
    if (e.mode == 2) {
      const float q = prob_of(xd[i], e.Md, e.c, e.invSd);
      if constexpr (kPol) mu = (q >= e.tau && e.cprev * q >= e.min_cum) ? q : 0.f;
      else mu = q >= e.tau ? q : 0.f;
    }
    r[i] = v0 + i < V ? fmaxf(p - mu, 0.f) : 0.f;
  }
  if (e.mode == 1) {
#pragma unroll 1
    for (int a = 0; a < e.nadm; ++a) {
      const int o = e.adm_i[a] - v0;
      if (o >= 0 && o < 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i == o) r[i] = fmaxf(r[i] - e.adm_q[a], 0.f);
      }
    }
  }
}

// what the finishing pass of sequence b needs from the inputs alone: drafted
// tokens, the Philox draws (or the explicit uniforms), the gate.  Runs before
// the wait on the stream pass.
template <int kMode>
__device__ __forceinline__ void finish_prologue(const Params& P, int b, FinishShared& sh, bool dry) {
  const int tid = threadIdx.x, k = P.k;
  const uint64_t s_idx = P.seq_offset + static_cast<uint64_t>(b);
  if (!dry) {
    // the sequence's chunk statistics, drafted-token logits and (gated)
    // candidate slots, pulled into L2 while the stream pass drains: 180 MB
    // of streamed logits have evicted the early ones, and L2 is the point of
    // coherence, so the stream pass's last writes to these lines land there
    // and the loads after the wait hit
    const int R = P.rows, nch = P.nchunk;
    const char* pb = reinterpret_cast<const char*>(P.part + static_cast<int64_t>(b) * R * nch);
    const int np = (R * nch * static_cast<int>(sizeof(float2)) + 127) / 128;
#pragma unroll 1
    for (int i = tid; i < np; i += kFinThreads) prefetch_l2(pb + i * 128);
    if (tid == kFinThreads - 1) prefetch_l2(P.xD + static_cast<int64_t>(b) * R);
    if (kMode != kModeGreedy && seq_gated(P, b)) {
      const char* cb = reinterpret_cast<const char*>(P.cand + static_cast<int64_t>(b) * k * nch * kTopM);
      const int nc = (k * nch * kTopM * static_cast<int>(sizeof(Cand)) + 127) / 128;
#pragma unroll 1
      for (int i = tid; i < nc; i += kFinThreads) prefetch_l2(cb + i * 128);
    }
  }
  if (tid <= k) {
    // draw 0 at position tid (the accept test), draw 1 at position tid (the
    // residual or bonus sample, should the sequence stop there)
#pragma unroll 1
    for (int draw = 0; draw < 2; ++draw) {
      float u;
      if (draw == 0 && P.u0) u = tid < k ? P.u0[static_cast<int64_t>(b) * k + tid] : 0.f;
      else if (draw == 1 && P.u1) u = P.u1[b];
      else u = philox_uniform(P.seed, s_idx, static_cast<uint32_t>(tid), static_cast<uint32_t>(draw));
      if (draw == 0 && tid < k) sh.u0[tid] = u;
      if (draw == 1) sh.u1[tid] = u;
    }
  }
  if (P.fthr && tid < P.rows) {
    // the rows' sampler filters, chosen before the stream pass started (so
    // complete when this grid launched)
    sh.fthr[tid] = P.fthr[static_cast<int64_t>(b) * P.rows + tid];
    sh.ffirst[tid] = P.ffirst[static_cast<int64_t>(b) * P.rows + tid];
  }
  if (tid < k) {
    sh.Dv[tid] = __ldg(P.D + static_cast<int64_t>(b) * k + tid);
    sh.nadm[tid] = 0;
    if constexpr (kMode != kModeSample) {
      sh.tau_j[tid] = step_tau(P, b, tid);
      sh.cprev[tid] = 1.f;
    }
  }
  if constexpr (kMode == kModePolicy) {
    if (tid < 32) {
      // rows whose admitted set the stream pass collected (same predicate there)
      const bool fast = tid < k && seq_gated(P, b) && gate_fast_path(step_floor(P, b, tid));
      const unsigned m = __ballot_sync(0xffffffffu, fast);
      if (tid == 0) sh.fast_rows = m;
    }
  }
  if (tid == 0) {
    const bool gated = seq_gated(P, b);
    const float tau = seq_tau(P, b);
    sh.gated = gated ? 1 : 0;
    sh.tau = tau;
    if constexpr (kMode == kModeSample)
      sh.fast_rows = (gated && gate_fast_path(tau)) ? (k >= 32 ? 0xffffffffu : (1u << k) - 1u) : 0u;
    // the sequence's own threshold is checked where it is used (no schedule)
    sh.bad = (gated && !P.has_sched && !(tau > 0.f && tau <= 1.f)) ? 1 : 0;
    sh.ncand = 0;
    sh.overflow_rows = 0u;
    sh.boundary = 0;
    sh.pick = -1;
    sh.dry = dry ? 1 : 0;
  }
}

template <typename TT, typename TD, bool kPol, bool kFilt>
__device__ void finish_front(const Params& P, int b, FinishShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k, R = P.rows, nch = P.nchunk, V = P.V;
  const bool gated = sh.gated != 0;
  const unsigned fast_rows = sh.fast_rows;
  const bool cum = kPol && P.min_cum > 0.f;
  const float c = P.c;
  const TT* Lt = static_cast<const TT*>(P.Lt);
  const float2* seq_part = P.part + static_cast<int64_t>(b) * R * nch;
  const bool staged = R * nch <= kFinPartCap;
  const bool dry = sh.dry != 0;

  // step 1: what the stream pass left -- drafted-token logits, chunk
  // statistics, and (gated) the candidate slots, gathered into a list and
  // emptied for the next call -- in one round of independent loads: every
  // load of a round is issued before any value is used or any global store
  // (which might alias a later load) is made
  const float xdv = tid < R ? __ldcg(P.xD + static_cast<int64_t>(b) * R + tid) : 0.f;
  const unsigned over =
      tid < k && ((fast_rows >> tid) & 1u) ? __ldcg(P.cand_over + static_cast<int64_t>(b) * k + tid) : 0u;
  bool pending = true;
  auto consume_first = [&]() {
    if (tid < R) sh.xD[tid] = xdv;
    if (over) {
      atomicOr(&sh.overflow_rows, 1u << tid);
      if (!dry) P.cand_over[static_cast<int64_t>(b) * k + tid] = 0u;
    }
    pending = false;
  };
  {
    // up to kBatch chunk statistics and kBatch candidate slots per thread per
    // round
    constexpr int kBatch = 8;
    const int np = staged ? R * nch : 0;
    const int ns = fast_rows ? k * nch * kTopM : 0;
    Cand* sc = P.cand + static_cast<int64_t>(b) * k * nch * kTopM;
    const int nmax = np > ns ? np : ns;
#pragma unroll 1
    for (int base = 0; base < nmax; base += kBatch * kFinThreads) {
      float2 pv[kBatch], cd[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int e = base + i * kFinThreads + tid;
        if (e < np) pv[i] = ldcg_f2(seq_part + e);
        cd[i] = e < ns ? ldcg_f2(reinterpret_cast<const float2*>(sc + e)) : make_float2(0.f, __int_as_float(-1));
      }
      if (pending) consume_first();
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int e = base + i * kFinThreads + tid;
        if (e < np) sh.part[e] = pv[i];
        const int v = __float_as_int(cd[i].y);
        if (v >= 0) {  // a candidate: gather it and empty the slot for the next call
          if (!dry) sc[e].v = -1;
          const int j = e / (nch * kTopM);
          const int n = atomicAdd(&sh.ncand, 1);
          if (n < kCandCap && v < V) {
            sh.cand_j[n] = j;
            sh.cand_v[n] = v;
            sh.cand_x[n] = cd[i].x;
          } else {
            atomicOr(&sh.overflow_rows, 1u << j);
          }
        }
      }
    }
    if (pending) consume_first();
  }
  __syncthreads();
  auto part_at = [&](int r, int ch) -> float2 {
    return staged ? sh.part[r * nch + ch] : ldcg_f2(seq_part + static_cast<int64_t>(r) * nch + ch);
  };

  // step 2: the target logits of the candidates go out (a candidate thread
  // uses them in step 3) while half-warps merge the chunk statistics of
  // rows r0 + 0 and r0 + 1 (both halves of a warp loop together)
  const int nc = min(sh.ncand, kCandCap);
  int cj = 0, cv = 0;
  float cx = 0.f, cxt = 0.f;
  if (tid < nc) {
    cj = sh.cand_j[tid];
    cv = sh.cand_v[tid];
    cx = sh.cand_x[tid];
    cxt = logit_at<TT>(Lt + (static_cast<int64_t>(b) * (k + 1) + cj) * V, cv);
    if constexpr (kFilt) cxt = filt1(cxt, cv, sh.fthr[cj], sh.ffirst[cj]);
  }
  {
    // the loops run the same trip count on every lane (a lane without an
    // entry adds nothing), so the warp reaches its shuffles converged
    const int half = lane >> 4, l16 = lane & 15;
    const int niter = (nch + 15) >> 4;
#pragma unroll 1
    for (int r0 = 2 * warp; r0 < R; r0 += 2 * kFinWarps) {
      const int r = r0 + half;
      const bool live = r < R;
      float M = -INFINITY;
#pragma unroll 1
      for (int i = 0; i < niter; ++i) {
        const int ch = l16 + 16 * i;
        const float m = live && ch < nch ? part_at(r, ch).x : -INFINITY;
        M = fmaxf(M, m);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      dfloat S = df(0.f);
#pragma unroll 1
      for (int i = 0; i < niter; ++i) {
        const int ch = l16 + 16 * i;
        const float2 ms = live && ch < nch ? part_at(r, ch) : make_float2(-INFINITY, 0.f);
        S = df_add(S, df(ms.x == -INFINITY ? ms.y * 0.f : ms.y * exp2f(ms.x - M)));
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) S = df_add(S, shfl_xor_df(S, o));
      if (live && l16 == 0) {
        sh.rowM[r] = M;
        sh.rowS[r] = S;
        sh.rowInvS[r] = (1.f / S.hi) * (1.f - S.lo / S.hi);  // 1 / (hi + lo) to float precision
        if (M == -INFINITY || !isfinite(S.hi) || !(S.hi > 0.f)) sh.bad = 1;
        if (P.row_stats && !dry) {
          // (max, log-sum-exp) of L / T: Mc ln 2 and Mc ln 2 + ln S
          const float mo = M * 0.69314718f;
          P.row_stats[(static_cast<int64_t>(b) * R + r) * 2 + 0] = mo;
          P.row_stats[(static_cast<int64_t>(b) * R + r) * 2 + 1] = mo + (logf(S.hi) + S.lo / S.hi);
        }
      }
    }
  }
  __syncthreads();

  // step 3: the admitted tokens among the candidates, with their target
  // probability; and, in warp 0, every draft position: gate, mu, alpha, accept
  // test.  With a cumulative floor a candidate's admission needs the prefix
  // product of its step, which warp 0 computes first.
  auto admit_candidates = [&]() {
    if (tid < nc && !sh.bad) {
      const int rd = k + 1 + cj;
      const float q = prob_of(cx, sh.rowM[rd], c, sh.rowInvS[rd]);
      if (kPol ? gate_admits(q, sh.tau_j[cj], sh.cprev[cj], cum, P.min_cum) : q >= sh.tau) {
        const int a = atomicAdd(&sh.nadm[cj], 1);
        if (a < kTopM) {
          sh.adm_i[cj][a] = cv;
          sh.adm_q[cj][a] = q;
          sh.adm_p[cj][a] = prob_of(cxt, sh.rowM[cj], c, sh.rowInvS[cj]);
        } else {
          atomicOr(&sh.overflow_rows, 1u << cj);
        }
      }
    }
  };
  if (!cum) admit_candidates();
  if (warp == 0) {
    bool ok = true, acc = false, is_null = false, near = false;
    float alpha = 0.f, p = 0.f, q = 1.f;
    if (lane < k) {
      const int d = sh.Dv[lane];
      ok = d >= 0 && d < V;
      if (ok && !sh.bad) {
        const int rt = lane, rd = k + 1 + lane;
        p = prob_of(sh.xD[rt], sh.rowM[rt], c, sh.rowInvS[rt]);
        q = prob_of(sh.xD[rd], sh.rowM[rd], c, sh.rowInvS[rd]);
      }
    }
    float cprev = 1.f;
    if (cum) {
      // exclusive prefix product of q_i(D_i) over the positions (lanes past k
      // hold 1)
      float incl = q;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl *= y;
      }
      cprev = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) cprev = 1.f;
      if (lane < k) sh.cprev[lane] = cprev;
    }
    if (lane < k && ok && !sh.bad) {
      const float tau = kPol ? sh.tau_j[lane] : sh.tau;
      const bool admitted = !gated || gate_admits(q, tau, cprev, cum, P.min_cum);
      const float mu = admitted ? q : 0.f;
      is_null = !admitted;
      alpha = is_null ? 0.f : (mu > 0.f ? fminf(1.f, p / mu) : (p > 0.f ? 1.f : 0.f));
      const float u0 = sh.u0[lane];
      acc = !is_null && p > 0.f && u0 * mu <= p;
      bool gate_near = fabsf(q - tau) < kBoundary;
      if constexpr (kPol)
        gate_near = (tau > 0.f && gate_near) || (cum && fabsf(cprev * q - P.min_cum) < kBoundary);
      near = (gated && gate_near) || (!is_null && mu > 0.f && p < mu && fabsf(u0 - p / mu) < kBoundary);
    }
    const bool any_bad = __any_sync(0xffffffffu, !ok) || sh.bad;
    const unsigned accm = __ballot_sync(0xffffffffu, lane < k && acc);
    int jstar = __ffs(~accm) - 1;
    if (jstar > k || jstar < 0) jstar = k;
    const unsigned nearm = __ballot_sync(0xffffffffu, near && lane <= jstar);
    const unsigned nullm = __ballot_sync(0xffffffffu, is_null);
    if (lane < k && !dry) {
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
  if (cum) {
    __syncthreads();  // the prefix products
    admit_candidates();
  }
  __syncthreads();

  const int jstar = sh.jstar;
  int32_t* tok = P.tokens + static_cast<int64_t>(b) * (k + 1);
  if (sh.bad) {
    if (tid <= k && !dry) tok[tid] = -1;
    if (tid == 0) {
      if (!dry) {
        P.accepted_len[b] = -1;
        if (P.counters) atomicAdd(P.counters + SV_CNT_INVALID, 1ull);
      }
      sh.fmode = -1;  // done: nothing left to sample
    }
    return;
  }

  // the stop row's sampling mode: 0 the bonus row (p), 1 a gated row whose
  // admitted set is known (p minus the admitted tokens' q), 2 the dense
  // residual (q everywhere: the stop row pair is re-read)
  if (tid == 0) {
    int mode = 0;
    if (jstar < k) mode = (((fast_rows & ~sh.overflow_rows) >> jstar) & 1u) || dry ? 1 : 2;
    sh.fmode = mode;  // a warming run never re-reads a dense stop row pair
  }
}

// A greedy call (temperature 0): p and q are one-hot at each row's first
// largest logit t*_j (target) and d*_j (draft), so the rule reduces to: a
// gated position is NULL where D differs from d*_j, a position is accepted
// where D equals t*_j (alpha is 1 there, 0 elsewhere), and the stop row emits
// t*_{j*} -- the residual (p - mu)+ is one-hot at t*_{j*}, or empty when
// t*_{j*} = d*_{j*}, which falls back to p: the same token.  No uniform is used.
template <typename TT, typename TD>
__device__ void finish_greedy(const Params& P, int b, FinishShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k, R = P.rows, nch = P.nchunk, V = P.V;
  const bool gated = sh.gated != 0;
  const float2* seq_part = P.part + static_cast<int64_t>(b) * R * nch;
  const bool staged = R * nch <= kFinPartCap;
  const bool dry = sh.dry != 0;
  if (staged) {
#pragma unroll 4
    for (int e = tid; e < R * nch; e += kFinThreads) sh.part[e] = ldcg_f2(seq_part + e);
  }
  __syncthreads();
  auto part_at = [&](int r, int ch) -> float2 {
    return staged ? sh.part[r * nch + ch] : ldcg_f2(seq_part + static_cast<int64_t>(r) * nch + ch);
  };
  // each row's largest logit and the first chunk holding it (half-warps)
  {
    const int half = lane >> 4, l16 = lane & 15;
    const int niter = (nch + 15) >> 4;
#pragma unroll 1
    for (int r0 = 2 * warp; r0 < R; r0 += 2 * kFinWarps) {
      const int r = r0 + half;
      const bool live = r < R;
      float M = -INFINITY;
      int bc = nch;
      bool bad = false;
      // the same trip count on every lane: the shuffles below run converged
#pragma unroll 1
      for (int i = 0; i < niter; ++i) {
        const int ch = l16 + 16 * i;
        const bool in = live && ch < nch;
        const float2 ms = in ? part_at(r, ch) : make_float2(-INFINITY, 0.f);
        if (__float_as_int(ms.y) < 0) bad = true;
        if (ms.x > M) {
          M = ms.x;
          bc = ch;
        }
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const float oM = __shfl_xor_sync(0xffffffffu, M, o);
        const int obc = __shfl_xor_sync(0xffffffffu, bc, o);
        if (oM > M || (oM == M && obc < bc)) {
          M = oM;
          bc = obc;
        }
      }
      const unsigned badm = __ballot_sync(0xffffffffu, live && bad);
      const bool anybad = ((badm >> (16 * half)) & 0xffffu) != 0u;
      if (live && l16 == 0) {
        if (anybad || M == -INFINITY || bc >= nch) {
          sh.bad = 1;
          sh.targ[r] = -1;
        } else {
          sh.targ[r] = __float_as_int(part_at(r, bc).y);
        }
        if (P.row_stats && !dry) {
          P.row_stats[(static_cast<int64_t>(b) * R + r) * 2 + 0] = M;
          P.row_stats[(static_cast<int64_t>(b) * R + r) * 2 + 1] = M;
        }
      }
    }
  }
  __syncthreads();
  int32_t* tok = P.tokens + static_cast<int64_t>(b) * (k + 1);
  if (warp == 0) {
    bool ok = true, acc = false, is_null = false;
    // one-hot q: q_j(D_j) is 1 where D_j is the draft argmax, else 0, and the
    // prefix product in front of step j is 1 iff every earlier draft is
    const bool hit = lane < k && sh.Dv[lane] == sh.targ[k + 1 + lane];
    const unsigned hitm = __ballot_sync(0xffffffffu, hit);
    if (lane < k) {
      const int d = sh.Dv[lane];
      ok = d >= 0 && d < V;
      const float q = hit ? 1.f : 0.f;
      const float cprev = ((~hitm) & ((1u << lane) - 1u)) == 0u ? 1.f : 0.f;
      is_null = gated && !gate_admits(q, sh.tau_j[lane], cprev, P.min_cum > 0.f, P.min_cum);
      acc = ok && !is_null && d == sh.targ[lane];
    }
    const bool any_bad = __any_sync(0xffffffffu, !ok) || sh.bad;
    const unsigned accm = __ballot_sync(0xffffffffu, lane < k && acc);
    int jstar = __ffs(~accm) - 1;
    if (jstar > k || jstar < 0) jstar = k;
    const unsigned nullm = __ballot_sync(0xffffffffu, lane < k && is_null);
    if (dry) {
      // a warming run: nothing is written
    } else if (lane < k) {
      const int64_t o = static_cast<int64_t>(b) * k + lane;
      P.alpha[o] = (!any_bad && acc) ? 1.f : 0.f;
      if (P.flags) {
        int8_t f;
        if (any_bad) f = SV_FLAG_INVALID;
        else if (lane < jstar) f = SV_FLAG_ACCEPT;
        else if (lane == jstar) f = is_null ? SV_FLAG_NULL : SV_FLAG_REJECT;
        else f = SV_FLAG_UNREACHED;
        P.flags[o] = f;
      }
    }
    if (dry) {
      // a warming run: nothing is written
    } else if (any_bad) {
      if (lane <= k) tok[lane] = -1;
      if (lane == 0) {
        P.accepted_len[b] = -1;
        if (P.counters) atomicAdd(P.counters + SV_CNT_INVALID, 1ull);
      }
    } else {
      if (lane < jstar) tok[lane] = sh.Dv[lane];
      if (lane == jstar) tok[lane] = sh.targ[jstar];
      if (lane > jstar && lane <= k) tok[lane] = -1;
      if (lane == 0) {
        P.accepted_len[b] = jstar;
        if (P.counters) {
          atomicAdd(P.counters + SV_CNT_TESTED, static_cast<unsigned long long>(jstar < k ? jstar + 1 : k));
          atomicAdd(P.counters + SV_CNT_ACCEPTED, static_cast<unsigned long long>(jstar));
          if (jstar < k) {
            atomicAdd(P.counters + (((nullm >> jstar) & 1u) ? SV_CNT_NULL : SV_CNT_REJECTED), 1ull);
            if (sh.targ[jstar] == sh.targ[k + 1 + jstar]) atomicAdd(P.counters + SV_CNT_DEGENERATE, 1ull);
          } else {
            atomicAdd(P.counters + SV_CNT_BONUS, 1ull);
          }
        }
      }
    }
  }
  if (tid == 0) sh.fmode = -1;  // nothing left to sample
}

// The dense residual's chunk masses sum max(0, p - mu) over the stop row pair
// of sequence b (mu = q, or q on q >= tau when gated), one warp per chunk: the
// CTAs of a cluster share the chunks (CTA r of n takes chunks r * 8 + w, then
// every 8 n) and write the masses into the leading CTA's shared memory.  Lanes
// take 8-entry groups lane, lane + 32, ... (16-byte coalesced loads), four
// groups of both rows issued before use.
template <typename TT, typename TD, bool kPol, bool kFilt>
__device__ void dense_chunk_sums(const Params& P, int b, const FinishShared& lead, float* lead_tile,
                                 int rank, int csize) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int k = P.k, V = P.V, nch = P.nchunk;
  const int jstar = lead.jstar;
  const int rt = jstar, rd = k + 1 + jstar;
  const TT* trow = static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (k + 1) + jstar) * V;
  const TD* drow = static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * k + jstar) * V;
  const bool gated = lead.gated != 0;
  const ResidualEval ev{2, lead.rowM[rt], lead.rowInvS[rt], lead.rowM[rd], lead.rowInvS[rd], P.c,
                        gated ? (kPol ? lead.tau_j[jstar] : lead.tau) : -1.f,
                        kPol ? lead.cprev[jstar] : 1.f,
                        kPol && gated && P.min_cum > 0.f ? P.min_cum : -1.f, 0, nullptr, nullptr};
  const bool vt = P.vec_t != 0, vd = P.vec_d != 0;
  constexpr int kLaneGroups = kChunk / 8 / 32;
  // bf16 row pairs: a lane's whole share of the chunk (eight 16-byte loads
  // per row) in flight at once, kept raw until each group is evaluated; the
  // ragged or unaligned chunk, and wider types, four groups at a time
  constexpr bool kNarrow = sizeof(TT) == 2 && sizeof(TD) == 2;
#pragma unroll 1
  for (int ch = rank * kFinWarps + warp; ch < nch; ch += csize * kFinWarps) {
    const int c0 = ch * kChunk;
    float acc = 0.f;
    if (kNarrow && vt && vd && c0 + kChunk <= V) {
      uint4 rt[kLaneGroups], rd[kLaneGroups];
#pragma unroll
      for (int g = 0; g < kLaneGroups; ++g) {
        rt[g] = __ldcg(reinterpret_cast<const uint4*>(trow + c0 + (g * 32 + lane) * 8));
        rd[g] = __ldcg(reinterpret_cast<const uint4*>(drow + c0 + (g * 32 + lane) * 8));
      }
#pragma unroll
      for (int g = 0; g < kLaneGroups; ++g) {
        float xt[8] = {bf16_lo(rt[g].x), bf16_hi(rt[g].x), bf16_lo(rt[g].y), bf16_hi(rt[g].y),
                       bf16_lo(rt[g].z), bf16_hi(rt[g].z), bf16_lo(rt[g].w), bf16_hi(rt[g].w)};
        float xd[8] = {bf16_lo(rd[g].x), bf16_hi(rd[g].x), bf16_lo(rd[g].y), bf16_hi(rd[g].y),
                       bf16_lo(rd[g].z), bf16_hi(rd[g].z), bf16_lo(rd[g].w), bf16_hi(rd[g].w)};
        if constexpr (kFilt) {  // (rt, rd here are the raw vectors: the rows are jstar, k + 1 + jstar)
          filt8(xt, c0 + (g * 32 + lane) * 8, lead.fthr[jstar], lead.ffirst[jstar]);
          filt8(xd, c0 + (g * 32 + lane) * 8, lead.fthr[k + 1 + jstar], lead.ffirst[k + 1 + jstar]);
        }
        float rr[8];
        residual8<kPol>(ev, xt, xd, c0 + (g * 32 + lane) * 8, V, rr);
        acc += ((rr[0] + rr[1]) + (rr[2] + rr[3])) + ((rr[4] + rr[5]) + (rr[6] + rr[7]));
      }
    } else {
#pragma unroll 1
      for (int h = 0; h < kLaneGroups; h += 4) {
        float xt[4][8], xd[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          load8<TT>(trow, c0 + ((h + u) * 32 + lane) * 8, V, vt, xt[u]);
          load8<TD>(drow, c0 + ((h + u) * 32 + lane) * 8, V, vd, xd[u]);
        }
        if constexpr (kFilt) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            filt8(xt[u], c0 + ((h + u) * 32 + lane) * 8, lead.fthr[rt], lead.ffirst[rt]);
            filt8(xd[u], c0 + ((h + u) * 32 + lane) * 8, lead.fthr[rd], lead.ffirst[rd]);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float rr[8];
          residual8<kPol>(ev, xt[u], xd[u], c0 + ((h + u) * 32 + lane) * 8, V, rr);
          acc += ((rr[0] + rr[1]) + (rr[2] + rr[3])) + ((rr[4] + rr[5]) + (rr[6] + rr[7]));
        }
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) lead_tile[ch] = acc;
  }
}

template <typename TT, typename TD, bool kPol, bool kDense, bool kFilt>
__device__ void finish_back(const Params& P, int b, FinishShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k, R = P.rows, nch = P.nchunk, V = P.V;
  const bool gated = sh.gated != 0;
  const float c = P.c;
  const TT* Lt = static_cast<const TT*>(P.Lt);
  const TD* Ld = static_cast<const TD*>(P.Ld);
  const float2* seq_part = P.part + static_cast<int64_t>(b) * R * nch;
  const bool staged = R * nch <= kFinPartCap;
  auto part_at = [&](int r, int ch) -> float2 {
    return staged ? sh.part[r * nch + ch] : ldcg_f2(seq_part + static_cast<int64_t>(r) * nch + ch);
  };
  const int jstar = sh.jstar;
  int32_t* tok = P.tokens + static_cast<int64_t>(b) * (k + 1);
  const int rt = jstar, rd = k + 1 + jstar;
  const TT* trow = Lt + (static_cast<int64_t>(b) * (k + 1) + jstar) * V;
  const TD* drow = jstar < k ? Ld + (static_cast<int64_t>(b) * k + jstar) * V : nullptr;
  const int mode = sh.fmode;
  const int nadm = mode == 1 ? min(sh.nadm[jstar], kTopM) : 0;
  const float u1 = sh.u1[jstar];
  ResidualEval ev{mode, sh.rowM[rt], sh.rowInvS[rt],
                  jstar < k ? sh.rowM[rd] : 0.f, jstar < k ? sh.rowInvS[rd] : 0.f,
                  c, gated && jstar < k ? (kPol ? sh.tau_j[jstar] : sh.tau) : -1.f,
                  kPol && jstar < k ? sh.cprev[jstar] : 1.f,
                  kPol && gated && P.min_cum > 0.f ? P.min_cum : -1.f, nadm,
                  jstar < k ? sh.adm_i[jstar] : sh.adm_i[0],
                  jstar < k ? sh.adm_q[jstar] : sh.adm_q[0]};
  const bool vt = P.vec_t != 0, vd = P.vec_d != 0;

  // Without the dense pass (kDense false: a call whose stop rows are all
  // expected on the candidate fast path), a dense stop row pair -- possible
  // only when candidates overflow -- gets every chunk's residual mass from
  // the chunk pass of step 5, one chunk per iteration (it < nch), before the
  // search and the pick (it == nch).  Keeping the dense pass out of that
  // kernel measured about 1 us faster per call on the 128K-vocabulary batch.
#pragma unroll 1
  for (int it = !kDense && mode == 2 ? 0 : nch;; ++it) {
    const bool masses = it < nch;
    if (!masses) {
      // warp 0: chunk masses (from the chunk statistics in modes 0 / 1), the total
      // Z (a residual without mass falls back to p), and the chunk holding
      // y = u1 Z: the first chunk whose inclusive prefix exceeds y
      if (warp == 0) {
        const float invS = sh.rowInvS[rt];
        auto chunk_sums = [&](int use_mode) {
#pragma unroll 1
          for (int ch = lane; ch < nch; ch += 32) {
            const float2 ms = part_at(rt, ch);
            const float m = ms.x == -INFINITY ? 0.f : __fmul_rn(ms.y * exp2f(ms.x - ev.Mt), invS);
            float t = m;
            if (use_mode == 1) {
#pragma unroll 1
              for (int a = 0; a < nadm; ++a)
                if (sh.adm_i[jstar][a] / kChunk == ch) t -= fminf(sh.adm_p[jstar][a], sh.adm_q[jstar][a]);
              t = t > kResidualTol * m ? t : 0.f;
            }
            sh.tile[ch] = t;
          }
          __syncwarp();
        };
        // one pass gives every chunk's inclusive prefix (float-float) and the total
        auto scan_all = [&]() {
          dfloat carry = df(0.f);
#pragma unroll 1
          for (int g0 = 0; g0 < nch; g0 += 32) {
            const int ch = g0 + lane;
            const float t = ch < nch ? sh.tile[ch] : 0.f;
            const dfloat incl = df_add(warp_incl_scan_df(df(t), lane), carry);
            if (ch < nch) sh.prefix[ch] = incl;
            carry = shfl_df(incl, 31);
          }
          __syncwarp();
          return carry;
        };
        if (mode != 2) chunk_sums(mode);  // mode 2: the masses are in sh.tile
        dfloat Z = scan_all();
        int degenerate = 0;
        if (!(Z.hi > 0.f)) {
          chunk_sums(0);
          Z = scan_all();
          degenerate = 1;
        }
        // the first chunk whose inclusive prefix exceeds y = u1 Z, and the last
        // chunk with mass
        const dfloat y = df_mul(Z, u1);
        dfloat before = df(0.f);
        int found = -1, last = -1;
#pragma unroll 1
        for (int g0 = 0; g0 < nch; g0 += 32) {
          const int ch = g0 + lane;
          const bool in = ch < nch;
          if (in && sh.tile[ch] > 0.f) last = ch;
          const unsigned m = __ballot_sync(0xffffffffu, in && df_lt(y, sh.prefix[ch]));
          if (found < 0 && m) {
            found = g0 + __ffs(m) - 1;
            before = df_sub(sh.prefix[found], df(sh.tile[found]));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
        if (found < 0) {  // rounding left y at or past the total: the last chunk with mass
          found = last < 0 ? 0 : last;
          before = df(INFINITY);  // forces the last-positive fallback inside the chunk
        }
        if (lane == 0) {
          sh.tstar = found;
          sh.before = before;
          sh.Z = Z;
          sh.y = y;
          sh.degenerate = degenerate;
          sh.mode = degenerate ? 0 : mode;
        }
      }
      __syncthreads();
      ev.mode = sh.mode;
    }

    // step 5: one re-read of the chosen chunk (or, in the mass pass, of chunk
    // it); thread i evaluates entries [8 i, 8 i + 8), then a block-wide scan.  Thread i's range is [lo_i, hi_i)
    // with lo_{i+1} == hi_i bit for bit (the same float-float sums), so exactly
    // one thread claims any y below the chunk total.
    const int c0 = (masses ? it : sh.tstar) * kChunk;
    const int e0 = tid * 8;
    float r8[8];
    {
      float xt[8], xd[8];
      load8<TT>(trow, c0 + e0, V, vt, xt);
      if (ev.mode == 2) load8<TD>(drow, c0 + e0, V, vd, xd);
      if constexpr (kFilt) {
        filt8(xt, c0 + e0, sh.fthr[rt], sh.ffirst[rt]);
        if (ev.mode == 2) filt8(xd, c0 + e0, sh.fthr[rd], sh.ffirst[rd]);
      }
      residual8<kPol>(ev, xt, xd, c0 + e0, V, r8);
    }
    {
      int lastpos = -1;
      float t0 = 0.f, t1 = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e & 1) t1 += r8[e]; else t0 += r8[e];
        if (r8[e] > 0.f) lastpos = c0 + e0 + e;
      }
      const dfloat tot = df_add(df(t0), df(t1));
      const dfloat wincl = warp_incl_scan_df(tot, lane);
      dfloat wexcl = shfl_up_df(wincl, 1);
      if (lane == 0) wexcl = df(0.f);
      int wl = lastpos;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wl = max(wl, __shfl_xor_sync(0xffffffffu, wl, o));
      if (lane == 31) sh.wtot[warp] = wincl;
      if (lane == 0) sh.wlast[warp] = wl;
      __syncthreads();
      // every thread forms its warp's base from the (at most 8) warp totals
      dfloat wbase = df(0.f);
#pragma unroll 1
      for (int w = 0; w < warp; ++w) wbase = df_add(wbase, sh.wtot[w]);
      const dfloat lo = df_add(wbase, wexcl), hi = df_add(wbase, wincl);
      if (masses && tid == 0) {  // the chunk's residual mass: the warp totals in order
        dfloat tot = df(0.f);
        for (int w = 0; w < kFinWarps; ++w) tot = df_add(tot, sh.wtot[w]);
        sh.tile[it] = df_f(tot);
      }
      const dfloat yl = df_sub(sh.y, sh.before);
      if (!masses && df_le(lo, yl) && df_lt(yl, hi)) {
        const float target = df_f(df_sub(yl, lo));
        float run = 0.f, prev = 0.f;
        int pick = lastpos;  // rounding inside the thread: its last positive entry
        bool hit = false;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (!hit) {
            prev = run;
            run += r8[e];
            if (run > target) {
              pick = c0 + e0 + e;
              hit = true;
            }
          }
        }
        if (!hit) prev = run = df_f(df_sub(hi, lo));
        sh.pick = pick;
        const float Zf = df_f(sh.Z);
        const float cl = df_f(df_add(df_add(sh.before, lo), df(prev))) / Zf;
        const float chh = df_f(df_add(df_add(sh.before, lo), df(run))) / Zf;
        if (fabsf(u1 - cl) < kBoundary || fabsf(u1 - chh) < kBoundary) atomicAdd(&sh.boundary, 1);
      }
    }
    __syncthreads();
    if (!masses) break;
  }

  // step 6: outputs
  if (sh.dry) return;
  if (tid == 0) {
    int pick = sh.pick;
    if (pick < 0) {
      for (int w = 0; w < kFinWarps; ++w) pick = max(pick, sh.wlast[w]);
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
      if (sh.degenerate) atomicAdd(P.counters + SV_CNT_DEGENERATE, 1ull);
    }
  }
  if (tid < jstar) tok[tid] = sh.Dv[tid];
  if (tid > jstar && tid <= k) tok[tid] = -1;
}

// The finishing grid runs in clusters of one or more CTAs (a cluster per
// sequence at a time).  The leading CTA does all the work of a sequence except
// the dense residual's chunk masses, which every CTA of the cluster shares.
template <typename TT, typename TD, int kMode, bool kDense, bool kFilt>
__global__ void __launch_bounds__(kFinThreads, 2) finish_kernel(const __grid_constant__ Params P) {
  constexpr bool kPol = kMode == kModePolicy;
  extern __shared__ __align__(16) unsigned char fin_smem[];
  FinishShared& sh = *reinterpret_cast<FinishShared*>(fin_smem);
  cg::cluster_group cluster = cg::this_cluster();
  // clusters only with the dense pass
  const int csize = kDense ? static_cast<int>(cluster.num_blocks()) : 1;
  const int rank = kDense ? static_cast<int>(cluster.block_rank()) : 0;
  const int cid = (static_cast<int>(blockIdx.x) - P.fin_warm) / csize;
  const int ncl = (static_cast<int>(gridDim.x) - P.fin_warm) / csize;
  FinishShared* lead = csize > 1 ? cluster.map_shared_rank(&sh, 0) : &sh;
  // the next call's stream pass may launch (it waits for this grid to
  // complete before it touches memory)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // A warming CTA (single-CTA clusters only; the grid's first CTAs, so the
  // first to take SMs as stream CTAs retire) runs the finishing code of one
  // sequence without waiting for the stream pass, on whatever the workspace
  // holds (the previous call's statistics, or lines being rewritten), and
  // writes no global memory: what it computes is discarded.  Code that runs
  // once per SM per call is otherwise fetched from DRAM at every step of the
  // chain -- the streamed logits have evicted it from L2 -- and the real
  // CTAs, which start after the wait, now find it in L2.  Both kinds go
  // through the same loop, so they execute the same instructions.
  const bool warm = static_cast<int>(blockIdx.x) < P.fin_warm;
  const int first = warm ? P.B - 1 - static_cast<int>(blockIdx.x) % P.B : cid;
  const int stop = warm ? first + 1 : P.B;
  const int stride = warm ? 1 : ncl;
  // the first sequence's input-only work overlaps the end of the stream pass;
  // then wait for the stream pass (programmatic dependent launch) before
  // reading its output
  if (rank == 0 && first < P.B) finish_prologue<kMode>(P, first, sh, warm);
  if (!warm) asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll 1
  for (int b = first; b < stop; b += stride) {
    if (rank == 0) {
      if (b != first) {
        __syncthreads();
        finish_prologue<kMode>(P, b, sh, false);
      }
      __syncthreads();
      if constexpr (kMode == kModeGreedy) finish_greedy<TT, TD>(P, b, sh);
      else finish_front<TT, TD, kPol, kFilt>(P, b, sh);
      __syncthreads();
    }
    if (csize > 1) cluster.sync();  // the leading CTA's decision, visible to the cluster
    const int fmode = lead->fmode;
    if constexpr (kDense) {
      if (fmode == 2) dense_chunk_sums<TT, TD, kPol, kFilt>(P, b, *lead, lead->tile, rank, csize);
      if (csize > 1) cluster.sync();  // every chunk mass is in the leading CTA
      else __syncthreads();
    }
    if (rank == 0 && fmode >= 0) finish_back<TT, TD, kPol, kDense, kFilt>(P, b, sh);
  }
}

}  // namespace sv
