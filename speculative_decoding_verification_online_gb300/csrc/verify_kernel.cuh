// Batched speculative-decoding verification kernels for sm_103a.
//
// A call is two launches on one stream:
//
// stream_kernel -- the bandwidth-bound pass.  Work is a list of items (sequence
//   b, row r, chunk c), where rows 0..k are the target rows and rows k+1..2k the
//   draft rows of b and a chunk is kChunk = 8192 consecutive vocabulary entries.
//   Persistent CTAs take items round-robin through a cp.async pipeline of S
//   chunk stages in shared memory (16-byte copies, each warp moving 512
//   contiguous bytes per instruction; every thread later reads back exactly the
//   pieces it copied, so the pipeline needs no barrier of its own).  Per item
//   it reads the chunk once and publishes the chunk statistics of the
//   temperature softmax (mlxcel PR #992, "What changed": p and q are
//   full-vocabulary temperature softmaxes in fp32), the logit at the drafted
//   token when that token lies in the chunk, and -- for draft rows of gated
//   sequences -- the tokens whose in-chunk probability reaches the gate (at
//   most floor(1/threshold) per chunk, a superset of the tokens the gate
//   admits) appended to a per-row candidate list.
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

#include "philox.cuh"
#include "spec_verify.h"

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kEPT = 32;                    // entries per thread per chunk
constexpr int kChunk = kThreads * kEPT;     // vocabulary entries per work item
constexpr int kTopM = 4;                    // gate candidates per chunk / admitted tokens per row
constexpr int kRowCap = 64;                 // gate candidates kept per draft row
constexpr int kMaxChunks = (SV_MAX_V + kChunk - 1) / kChunk;
constexpr int kMaxRows = 2 * SV_MAX_K + 1;
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
  float2* part;        // [B, rows, nchunk] (mc, s) per chunk
  float* xD;           // [B, rows] raw logit at the drafted token (rows j < k and draft rows)
  float* cand_v;       // [B, k, kRowCap] raw logits of gate candidates
  int* cand_i;         // [B, k, kRowCap] their token ids
  unsigned* cand_n;    // [B, k] candidates appended (> kRowCap: overflow); reset by the finisher
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

// probability of a token with raw logit x in a row with scaled max Mc and
// 1/sum invS: exp2(fma(x, c, -Mc)) * invS.  Every decision uses this formula.
__device__ __forceinline__ float prob_of(float x, float Mc, float c, float invS) {
  return exp2f(fmaf(x, c, -Mc)) * invS;
}

__device__ __forceinline__ bool gate_fast_path(float tau) {
  return tau * kGateSlack * static_cast<float>(kTopM + 1) > 1.0f;
}

// ------------------------------------------------------- chunk registers
//
// Thread t = 32 w + l owns NV 16-byte slots of the chunk: slot i is vector
// index w * 32 NV + 32 i + l.  bf16: 4 slots of 8 entries kept packed; f32: 8
// slots of 4.  A slot that lies wholly inside the row of an aligned tensor
// travels by cp.async into the stage; other slots (ragged tail, unaligned
// rows) are read directly, entries past V reading as -inf.

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
  // sum_v exp2(fma(x_v, c, nmc)), four independent accumulators
  __device__ __forceinline__ float expsum(float c, float nmc) const {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int q = 0; q < 16; q += 2) {
      a0 += ex2_approx(fmaf(bf16_lo(w[q]), c, nmc));
      a1 += ex2_approx(fmaf(bf16_hi(w[q]), c, nmc));
      a2 += ex2_approx(fmaf(bf16_lo(w[q + 1]), c, nmc));
      a3 += ex2_approx(fmaf(bf16_hi(w[q + 1]), c, nmc));
    }
    return (a0 + a1) + (a2 + a3);
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
    float m0 = fmaxf(x[0], x[1]), m1 = fmaxf(x[2], x[3]);
#pragma unroll
    for (int e = 4; e < 32; e += 4) {
      m0 = fmaxf(m0, fmaxf(x[e], x[e + 1]));
      m1 = fmaxf(m1, fmaxf(x[e + 2], x[e + 3]));
    }
    return fmaxf(m0, m1);
  }
  __device__ __forceinline__ float expsum(float c, float nmc) const {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      a0 += ex2_approx(fmaf(x[e], c, nmc));
      a1 += ex2_approx(fmaf(x[e + 1], c, nmc));
      a2 += ex2_approx(fmaf(x[e + 2], c, nmc));
      a3 += ex2_approx(fmaf(x[e + 3], c, nmc));
    }
    return (a0 + a1) + (a2 + a3);
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

__device__ __forceinline__ bool seq_gated(const Params& P, int b) {
  return P.gate_per_seq ? (P.gate_per_seq[b] != 0) : (P.gate_default != 0);
}
__device__ __forceinline__ float seq_tau(const Params& P, int b) {
  return P.tau_per_seq ? P.tau_per_seq[b] : P.tau_default;
}

// ------------------------------------------------------- stream kernel

template <typename TT, typename TD>
struct Stages {
  static constexpr int kBytes = kChunk * static_cast<int>(sizeof(TT) > sizeof(TD) ? sizeof(TT) : sizeof(TD));
  static constexpr int kDepth = kBytes <= 16384 ? 4 : 3;
  static constexpr int kMinBlocks = kBytes <= 16384 ? 3 : 2;
};

struct StreamShared {
  __align__(16) float red_max[kWarps];
  __align__(16) float red_sum[kWarps];
  int ncand;
  float cand_v[kTopM];
  int cand_i[kTopM];
};

__device__ __forceinline__ void decode_item(const Params& P, unsigned item, int& b, int& r, int& ch) {
  b = static_cast<int>(item / static_cast<unsigned>(P.items_per_seq));
  const int rem = static_cast<int>(item - static_cast<unsigned>(b) * P.items_per_seq);
  r = rem / P.nchunk;
  ch = rem - r * P.nchunk;
}

template <typename TT, typename TD>
__device__ __forceinline__ void issue_item(const Params& P, unsigned item, unsigned char* stage,
                                           int warp, int lane) {
  int b, r, ch;
  decode_item(P, item, b, r, ch);
  const int c0 = ch * kChunk;
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

// one work item: chunk statistics, drafted-token logit, gate candidates
template <typename T>
__device__ __forceinline__ void process_item(const Params& P, StreamShared& sh, const T* row,
                                             const unsigned char* stage, int b, int r, int ch,
                                             bool is_draft, int tid, int warp, int lane) {
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
  const float4 ma = *reinterpret_cast<const float4*>(&sh.red_max[0]);
  const float4 mb = *reinterpret_cast<const float4*>(&sh.red_max[4]);
  const float m_c = fmaxf(fmaxf(fmaxf(ma.x, ma.y), fmaxf(ma.z, ma.w)), fmaxf(fmaxf(mb.x, mb.y), fmaxf(mb.z, mb.w)));
  // scaled reference: mc = fl(m c); an all -inf chunk uses 0 so that -inf entries give 0
  const float mc = m_c == -INFINITY ? -INFINITY : m_c * P.c;
  const float nmc = m_c == -INFINITY ? 0.f : -mc;
  const float s_t = warp_sum(regs.expsum(P.c, nmc));
  if (lane == 0) sh.red_sum[warp] = s_t;
  __syncthreads();
  const float4 sa = *reinterpret_cast<const float4*>(&sh.red_sum[0]);
  const float4 sb = *reinterpret_cast<const float4*>(&sh.red_sum[4]);
  const float s_c = ((sa.x + sa.y) + (sa.z + sa.w)) + ((sb.x + sb.y) + (sb.z + sb.w));

  bool want_cand = false;
  if (is_draft) {
    const float tau = seq_tau(P, b);
    want_cand = seq_gated(P, b) && gate_fast_path(tau);
    if (want_cand) {
      // in-chunk probability exp2(x c - mc) / s >= slack * tau: a superset of
      // the admitted set (q <= in-chunk probability), at most 1/(slack tau) tokens
      float thr = INFINITY;
      if (s_c > 0.f && isfinite(s_c)) thr = (mc + log2f(tau * kGateSlack * s_c)) / P.c;
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
    P.part[(static_cast<int64_t>(b) * R + r) * P.nchunk + ch] = make_float2(mc, s_c);
    if (d >= c0 && d < c0 + kChunk && d < P.V) {
      constexpr int kVE = Chunk<T>::kVE;
      const int v0 = d - (d - c0) % kVE;
      float x;
      if (vec && v0 + kVE <= P.V) {
        if (sizeof(T) == 2)
          x = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(stage)[d - c0]) << 16);
        else
          x = reinterpret_cast<const float*>(stage)[d - c0];
      } else {
        x = logit_at<T>(row, d);
      }
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
  }
}

template <typename TT, typename TD>
__global__ void __launch_bounds__(kThreads, Stages<TT, TD>::kMinBlocks) stream_kernel(const Params P) {
  constexpr int S = Stages<TT, TD>::kDepth;
  constexpr int kStage = Stages<TT, TD>::kBytes;
  extern __shared__ __align__(128) unsigned char stages[];
  __shared__ StreamShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned total = P.total_items;
  const unsigned G = gridDim.x;
  const int k = P.k;
  if (tid == 0) sh.ncand = 0;

  // prologue: the first S - 1 items of this CTA in flight
#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    const unsigned item = blockIdx.x + static_cast<unsigned>(s) * G;
    if (item < total) issue_item<TT, TD>(P, item, stages + s * kStage, warp, lane);
    cp_async_commit();
  }
  int it = 0;
  for (unsigned item = blockIdx.x; item < total; item += G, ++it) {
    {
      const unsigned nx = item + static_cast<unsigned>(S - 1) * G;
      if (nx < total) issue_item<TT, TD>(P, nx, stages + ((it + S - 1) % S) * kStage, warp, lane);
      cp_async_commit();
    }
    cp_async_wait<S - 1>();
    int b, r, ch;
    decode_item(P, item, b, r, ch);
    const unsigned char* stage = stages + (it % S) * kStage;
    if (r <= k) {
      const TT* row = static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (k + 1) + r) * P.V;
      process_item<TT>(P, sh, row, stage, b, r, ch, false, tid, warp, lane);
    } else {
      const TD* row = static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * k + (r - k - 1)) * P.V;
      process_item<TD>(P, sh, row, stage, b, r, ch, true, tid, warp, lane);
    }
  }
  cp_async_wait<0>();
  // let the finishing grid start its prologue; its griddepcontrol.wait still
  // waits for this grid to complete and its memory to be visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ finishing

struct FinishShared {
  float rowM[kMaxRows];      // scaled row max Mc
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
__device__ void finish_sequence(const Params& P, int b, FinishShared& sh) {
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
  // row statistics from the chunk statistics (fp64 accumulation)
  for (int r = warp; r < R; r += kWarps) {
    const float2* pr = P.part + (static_cast<int64_t>(b) * R + r) * nch;
    float M = -INFINITY;
    for (int ch = lane; ch < nch; ch += 32) M = fmaxf(M, ldcg_f2(pr + ch).x);
    M = warp_max(M);
    double S = 0.0;
    for (int ch = lane; ch < nch; ch += 32) {
      const float2 ms = ldcg_f2(pr + ch);
      S += (ms.x == -INFINITY) ? static_cast<double>(ms.y * 0.f)
                               : static_cast<double>(ms.y) * static_cast<double>(exp2f(ms.x - M));
    }
    S = warp_sum_d(S);
    if (lane == 0) {
      sh.rowM[r] = M;
      sh.rowS[r] = S;
      sh.rowInvS[r] = static_cast<float>(1.0 / S);
      if (M == -INFINITY || !isfinite(S) || !(S > 0.0)) sh.bad = 1;
      if (P.row_stats) {
        // (max, log-sum-exp) of L / T: Mc ln 2 and Mc ln 2 + ln S
        const double mo = static_cast<double>(M) * 0.6931471805599453;
        P.row_stats[(static_cast<int64_t>(b) * R + r) * 2 + 0] = static_cast<float>(mo);
        P.row_stats[(static_cast<int64_t>(b) * R + r) * 2 + 1] = static_cast<float>(mo + log(S));
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

  // every draft position (one lane each): gate, mu, alpha, accept test
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

  // the stop row's residual (or bonus) weights, chunk by chunk
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
                     : static_cast<double>(ms.y) * static_cast<double>(exp2f(ms.x - ev.Mt)) *
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

template <typename TT, typename TD>
__global__ void __launch_bounds__(kThreads, 2) finish_kernel(const Params P) {
  __shared__ FinishShared sh;
  // wait for the stream pass (programmatic dependent launch) before reading its output
  asm volatile("griddepcontrol.wait;" ::: "memory");
  finish_sequence<TT, TD>(P, blockIdx.x, sh);
}

}  // namespace sv
