// filter_kernel.cuh -- the sampler's filter chain before the softmax (mlxcel
// PR #992, "What changed": temperature, top-k, top-p, min-p, then the softmax
// of the survivors; top_k == 1 is greedy), applied to every row of a call as
// a masked copy of the logits (-inf outside the kept set).  The verification
// kernels then run unchanged on the copies: the temperature softmax of a
// masked row is exactly the filtered distribution.
//
// Each filter keeps the tokens at or above a logit threshold (ties kept), so a
// row's kept set is {x : key(x) >= K} for one key K in an order-preserving
// integer encoding of the logits; top_k == 1 keeps the first largest logit
// only.  select_kernel (one CTA per row) finds K by radix descent over the
// keys, 8 bits a level, with per-warp histograms of counts (top-k) and of
// fixed-point masses 2^40 exp2(x c - Mc) (top-p: integer sums, so the
// decisions do not depend on the order of the additions); min-p is a
// threshold on x itself, found by bisection over the keys.  mask_kernel then
// writes the masked copy.
#pragma once

#include <type_traits>

#include "verify_kernel.cuh"

namespace sv {

struct Filter {
  int top_k;     // 0: off; 1: greedy (first largest logit only)
  float top_p;   // 1: off
  float min_p;   // 0: off
};

struct FilterParams {
  Filter f[2];          // [0] target rows, [1] draft rows
  unsigned* key;        // [B * rows] threshold key of each row (kept: key >= K)
  int* first;           // [B * rows] top_k == 1: the index kept, else -1
  void* Lt_m;           // masked copies, same layouts and types as the inputs
  void* Ld_m;
};

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr float kMassScalef = 1099511627776.0f;  // 2^40: masses as integers

// order-preserving keys: a larger logit has a larger key (NaN never occurs:
// such rows are invalid and not filtered)
__device__ __forceinline__ unsigned key_of(float x) {
  const unsigned u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_of_key(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <typename T> __device__ __forceinline__ float row_at(const T* row, int v);
template <> __device__ __forceinline__ float row_at<uint16_t>(const uint16_t* row, int v) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(row + v)) << 16);
}
template <> __device__ __forceinline__ float row_at<float>(const float* row, int v) { return __ldg(row + v); }

struct SelShared {
  unsigned cnt[kSelWarps][256];
  unsigned long long mass[kSelWarps][256];
  unsigned long long hcnt[256];    // level histograms, summed over warps
  unsigned long long hmass[256];
  int digit;
  unsigned long long above;        // count or mass of keys above the chosen digit
  unsigned long long wsum[kSelWarps];
  int wfirst[kSelWarps];
  unsigned long long Sk;           // mass of the top-k survivors
  unsigned kmax;                   // the row's largest key
  float Mc;
  int bad;
};

// one pass over the row: per-digit counts and fixed-point masses of the keys
// that share `prefix` on the bits above `shift + 8`
template <typename T>
__device__ void sel_histogram(const T* row, int V, float c, float Mc, unsigned prefix, int shift,
                              bool masses, SelShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kSelWarps * 256; i += kSelThreads) {
    (&sh.cnt[0][0])[i] = 0u;
    (&sh.mass[0][0])[i] = 0ull;
  }
  __syncthreads();
  const unsigned hi_mask = shift + 8 >= 32 ? 0u : (0xffffffffu << (shift + 8));
#pragma unroll 4
  for (int v = tid; v < V; v += kSelThreads) {
    const float x = row_at<T>(row, v);
    const unsigned kx = key_of(x);
    if ((kx & hi_mask) != (prefix & hi_mask)) continue;
    const int d = static_cast<int>((kx >> shift) & 255u);
    atomicAdd(&sh.cnt[warp][d], 1u);
    if (masses) {
      const float w = exp2f(fmaf(x, c, -Mc));
      atomicAdd(&sh.mass[warp][d], __float2ull_rn(w * kMassScalef));  // exact power-of-two scaling
    }
  }
  __syncthreads();
  for (int d = tid; d < 256; d += kSelThreads) {
    unsigned long long a = 0, m = 0;
    for (int w = 0; w < kSelWarps; ++w) {
      a += sh.cnt[w][d];
      m += sh.mass[w][d];
    }
    sh.hcnt[d] = a;
    sh.hmass[d] = m;
  }
  (void)lane;
  __syncthreads();
}

// thread 0: the largest digit d with (sum of the level histogram over digits
// >= d) + carry >= target; records it and the sum strictly above it
__device__ __forceinline__ void sel_descend(const unsigned long long* h, unsigned long long carry,
                                            double target, SelShared& sh) {
  if (threadIdx.x == 0) {
    unsigned long long acc = carry;
    int d = 255;
    for (; d > 0; --d) {
      if (static_cast<double>(acc + h[d]) >= target) break;
      acc += h[d];
    }
    sh.digit = d;
    sh.above = acc;
  }
  __syncthreads();
}

// the key K of each row (and the first index for top_k == 1)
template <typename TT, typename TD>
__global__ void __launch_bounds__(kSelThreads)
    select_kernel(const __grid_constant__ Params P, const __grid_constant__ FilterParams F) {
  extern __shared__ __align__(16) unsigned char sel_smem[];
  SelShared& sh = *reinterpret_cast<SelShared*>(sel_smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = static_cast<int>(blockIdx.x);  // b * rows + r
  const int b = g / P.rows, r = g % P.rows;
  const bool draft = r > P.k;
  const Filter f = F.f[draft ? 1 : 0];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int V = P.V;
  const bool use_k = f.top_k >= 2 && f.top_k < V;
  const bool use_p = f.top_p < 1.f;
  const bool use_m = f.min_p > 0.f;
  if (f.top_k != 1 && !use_k && !use_p && !use_m) {
    if (tid == 0) {
      F.key[g] = 0u;
      F.first[g] = -1;
    }
    return;
  }
  // the row's scaled maximum from the chunk statistics (one warp)
  if (warp == 0) {
    const float2* part = P.part + static_cast<int64_t>(g) * P.nchunk;
    float M = -INFINITY;
    for (int ch = lane; ch < P.nchunk; ch += 32) M = fmaxf(M, ldcg_f2(part + ch).x);
    M = warp_max(M);
    if (lane == 0) {
      sh.Mc = M;
      sh.bad = !(M > -INFINITY) || !isfinite(M);
    }
  }
  __syncthreads();
  const float Mc = sh.Mc, c = P.c;
  if (sh.bad) {  // an invalid row: the verification flags it; nothing to filter
    if (tid == 0) {
      F.key[g] = 0u;
      F.first[g] = -1;
    }
    return;
  }
  auto run = [&](const auto* row) {
    using T = typename std::remove_const<typename std::remove_pointer<decltype(row)>::type>::type;
    if (f.top_k == 1) {
      // greedy: the first index holding the largest logit
      float best = -INFINITY;
      int bi = 0x7fffffff;
      for (int v = tid; v < V; v += kSelThreads) {
        const float x = row_at<T>(row, v);
        if (x > best) {
          best = x;
          bi = v;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ob > best || (ob == best && oi < bi)) {
          best = ob;
          bi = oi;
        }
      }
      if (lane == 0) {
        sh.wsum[warp] = __float_as_uint(best);
        sh.wfirst[warp] = bi;
      }
      __syncthreads();
      if (tid == 0) {
        float tb = -INFINITY;
        int ti = 0x7fffffff;
        for (int w = 0; w < kSelWarps; ++w) {
          const float wb = __uint_as_float(static_cast<unsigned>(sh.wsum[w]));
          if (wb > tb || (wb == tb && sh.wfirst[w] < ti)) {
            tb = wb;
            ti = sh.wfirst[w];
          }
        }
        F.key[g] = key_of(tb);
        F.first[g] = ti;
      }
      return;
    }
    const int levels = sizeof(T) == 2 ? 2 : 4;  // bf16 keys have 16 significant bits
    // top-k: the k-th largest key, and (for top-p) the mass at or above it
    unsigned K = 0u;
    if (use_k) {
      unsigned prefix = 0u;
      unsigned long long carry_c = 0ull, carry_m = 0ull;
      for (int l = 0; l < levels; ++l) {
        const int shift = 24 - 8 * l;
        sel_histogram<T>(row, V, c, Mc, prefix, shift, use_p, sh);
        sel_descend(sh.hcnt, carry_c, static_cast<double>(f.top_k), sh);
        const int d = sh.digit;
        if (tid == 0) {
          unsigned long long mabove = 0ull;
          for (int e = 255; e > d; --e) mabove += sh.hmass[e];
          carry_m += mabove;
          if (l == levels - 1) sh.Sk = carry_m + sh.hmass[d];
        }
        carry_c = sh.above;
        prefix |= static_cast<unsigned>(d) << shift;
        __syncthreads();
      }
      K = prefix;
    }
    // top-p on the top-k survivors: the largest key K' (>= K) whose mass at
    // or above reaches top_p * S_k
    if (use_p) {
      unsigned prefix = 0u;
      unsigned long long carry = 0ull;
      for (int l = 0; l < levels; ++l) {
        const int shift = 24 - 8 * l;
        sel_histogram<T>(row, V, c, Mc, prefix, shift, true, sh);
        if (l == 0 && !use_k && tid == 0) {  // no top-k: every token survives
          unsigned long long all = 0ull;
          for (int e = 0; e < 256; ++e) all += sh.hmass[e];
          sh.Sk = all;
        }
        __syncthreads();
        const double target = static_cast<double>(f.top_p) * static_cast<double>(sh.Sk);
        sel_descend(sh.hmass, carry, target, sh);
        carry = sh.above;
        prefix |= static_cast<unsigned>(sh.digit) << shift;
        __syncthreads();
      }
      if (prefix > K) K = prefix;
    }
    // min-p: keep fma(x, c, -Mc) >= log2(min_p), i.e. the keys from the
    // smallest one whose logit passes (bisection: the test is monotone in
    // the logit), but never above the row's largest key
    if (use_m) {
      unsigned km = 0u;
      for (int v = tid; v < V; v += kSelThreads) km = max(km, key_of(row_at<T>(row, v)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) km = max(km, __shfl_xor_sync(0xffffffffu, km, o));
      if (lane == 0) sh.wfirst[warp] = static_cast<int>(km);
      __syncthreads();
      if (tid == 0) {
        unsigned kmax = 0u;
        for (int w = 0; w < kSelWarps; ++w) kmax = max(kmax, static_cast<unsigned>(sh.wfirst[w]));
        const float lmp = log2f(f.min_p);
        // the answer lies in (lo, hi]: +inf passes; the patterns below -inf
        // (NaN) count as failing
        unsigned lo = 0u, hi = key_of(INFINITY);
        while (hi - lo > 1u) {
          const unsigned mid = lo + (hi - lo) / 2u;
          const float xm = float_of_key(mid);
          if (!isnan(xm) && fmaf(xm, c, -Mc) >= lmp) hi = mid;
          else lo = mid;
        }
        sh.kmax = min(hi, kmax);
      }
      __syncthreads();
      if (sh.kmax > K) K = sh.kmax;
    }
    if (tid == 0) {
      F.key[g] = K;
      F.first[g] = -1;
    }
  };
  if (!draft) run(static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (P.k + 1) + r) * V);
  else run(static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * P.k + (r - P.k - 1)) * V);
}

// the masked copies: x where key(x) >= K of its row (or only at the kept index
// for top_k == 1), -inf elsewhere; one thread per 8 entries
template <typename T>
__device__ __forceinline__ void mask8(const T* src, T* dst, int64_t o, int v0, int V, unsigned K, int first) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int v = v0 + e;
    if (v >= V) break;
    const float x = row_at<T>(src + o, v);
    // a NaN stays, whatever its sign, so that the row is still rejected as invalid
    const bool keep = isnan(x) || (first >= 0 ? v == first : key_of(x) >= K);
    if constexpr (sizeof(T) == 2) {
      dst[o + v] = keep ? src[o + v] : static_cast<uint16_t>(0xFF80u);
    } else {
      dst[o + v] = keep ? x : -INFINITY;
    }
  }
}

template <typename TT, typename TD>
__global__ void __launch_bounds__(256) mask_kernel(const __grid_constant__ Params P, FilterParams F,
                                                   long long groups_per_row) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long total = static_cast<long long>(P.B) * P.rows * groups_per_row;
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < total; i += static_cast<long long>(gridDim.x) * 256ll) {
    const int g = static_cast<int>(i / groups_per_row);
    const int v0 = static_cast<int>(i - static_cast<long long>(g) * groups_per_row) * 8;
    const int b = g / P.rows, r = g % P.rows;
    const unsigned K = F.key[g];
    const int first = F.first[g];
    if (r <= P.k) {
      const int64_t o = (static_cast<int64_t>(b) * (P.k + 1) + r) * P.V;
      mask8<TT>(static_cast<const TT*>(P.Lt), static_cast<TT*>(F.Lt_m), o, v0, P.V, K, first);
    } else {
      const int64_t o = (static_cast<int64_t>(b) * P.k + (r - P.k - 1)) * P.V;
      mask8<TD>(static_cast<const TD*>(P.Ld), static_cast<TD*>(F.Ld_m), o, v0, P.V, K, first);
    }
  }
}

}  // namespace sv
