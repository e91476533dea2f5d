// filter_kernel.cuh -- the sampler's filter chain before the softmax (mlxcel
// PR #992, "What changed": temperature, top-k, top-p, min-p, then the softmax
// of the survivors; top_k == 1 is greedy).  Each row's kept set is found here
// (and, for bf16 rows, in hist_kernel.cuh); the verifying and diagnostics
// kernels then read every logit outside it as -inf, applying the row's
// threshold as they load (the temperature softmax of a row masked that way is
// exactly the filtered distribution).
//
// Each filter keeps the tokens at or above a logit threshold (ties kept), so a
// row's kept set is {x : key(x) >= K} for one key K in an order-preserving
// integer encoding of the logits; top_k == 1 keeps the first largest logit
// only.  select_kernel (one CTA per row) finds K by radix descent over the
// keys, 8 bits a level, with per-warp histograms of counts (top-k) and of
// fixed-point masses 2^40 exp2(x c - Mc) (top-p: integer sums, so the
// decisions do not depend on the order of the additions); min-p is a
// threshold on x itself, found by bisection over the keys.
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
  float* thr;           // [B * rows] the same threshold as a logit: kept x >= thr (-inf: all)
  // top-k rows: the gathering pass before the selection (null: none) --
  // gbound [B * rows] each row's lower bound of fl(x c) over its top-k set
  // (+inf: not gathered), glist / gcount what the pass kept per chunk
  float* gbound;
  const float* glist;
  const unsigned* gcount;
  int* done;            // [B * rows] the row was selected by list_select_kernel (null: none was)
};

// rows whose top-k set the gathering pass collects: top_k >= 2 within the
// number of chunks (see select_kernel), and a bound found among at most
// kBoundCap chunk maxima
constexpr int kBoundCap = 512;
__host__ __device__ inline bool gathers_row(const Filter& f, int nchunk) {
  return f.top_k >= 2 && f.top_k <= nchunk && nchunk <= kBoundCap;
}

constexpr int kSelThreads = 512;
// A selecting CTA sweeps its row with one 16-byte load per thread per step,
// used at once (its registers are at the two-CTAs-per-SM cap), so each step
// would wait a full DRAM round trip; every thread therefore also pulls its
// entries kSelAhead steps ahead into L2 (no registers), and the loads hit L2.
constexpr int kSelAhead = 4;
constexpr int kListCap = 4096;  // logits gathered for an in-shared-memory selection
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
// a row's threshold key as a logit threshold: key(x) >= K iff x >= float_of_key(K)
// for every non-NaN x but -0 against +0 (which compare equal as logits, as in
// the filters' own tie rule); K = 0 keeps every logit
__device__ __forceinline__ float thr_of_key(unsigned K) { return K == 0u ? -INFINITY : float_of_key(K); }

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
  unsigned long long h0mass[256];  // the level-0 mass histogram (all keys), kept for top-p
  unsigned lkey[kListCap];         // gathered logits' keys
  unsigned long long lmass[kListCap];
  int ln;
  unsigned kmax;                   // the row's largest key
  float Mc;
  int bad;
};

// one pass over the row: per-digit counts and fixed-point masses of the keys
// that share `prefix` on the bits above `shift + 8`.  A thread reads eight
// consecutive entries at a time and keeps a running (digit, count, mass) that
// it adds to its warp's histogram only when the digit changes: neighbouring
// logits mostly share their leading digits, so the shared-memory atomics stay
// few.
template <typename T>
__device__ void sel_histogram(const T* row, int V, bool vec, float c, float Mc, unsigned prefix, int shift,
                              bool masses, SelShared& sh) {
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < kSelWarps * 256; i += kSelThreads) {
    (&sh.cnt[0][0])[i] = 0u;
    (&sh.mass[0][0])[i] = 0ull;
  }
  __syncthreads();
  const unsigned hi_mask = shift + 8 >= 32 ? 0u : (0xffffffffu << (shift + 8));
  const unsigned want = prefix & hi_mask;
  int cd = -1;
  unsigned cc = 0u;
  unsigned long long cm = 0ull;
#pragma unroll
  for (int a = 0; a < kSelAhead; ++a)
    if (tid * 8 + a * kSelThreads * 8 < V) prefetch_l2(row + tid * 8 + a * kSelThreads * 8);
#pragma unroll 1
  for (int v0 = tid * 8; v0 < V; v0 += kSelThreads * 8) {
    if (v0 + kSelAhead * kSelThreads * 8 < V) prefetch_l2(row + v0 + kSelAhead * kSelThreads * 8);
    float x[8];
    load8<T>(row, v0, V, vec, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const unsigned kx = key_of(x[e]);
      if (v0 + e >= V || (kx & hi_mask) != want) continue;
      const int d = static_cast<int>((kx >> shift) & 255u);
      const unsigned long long wq = masses ? __float2ull_rn(ex2_approx(fmaf(x[e], c, -Mc)) * kMassScalef) : 0ull;
      if (d != cd) {
        if (cd >= 0) {
          atomicAdd(&sh.cnt[warp][cd], cc);
          if (masses) atomicAdd(&sh.mass[warp][cd], cm);
        }
        cd = d;
        cc = 0u;
        cm = 0ull;
      }
      ++cc;
      cm += wq;
    }
  }
  if (cd >= 0) {
    atomicAdd(&sh.cnt[warp][cd], cc);
    if (masses) atomicAdd(&sh.mass[warp][cd], cm);
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
  __syncthreads();
}

// warp 0: the largest digit d with (sum of the level histogram over digits
// >= d) + carry >= target; records it and the sum strictly above it.  The
// sums are integers, so comparing them with ceil(target) is exact; lane l
// holds digits 255 - 8l - i, i = 0..7, and a scan over the lanes gives each
// digit's sum from the top.
__device__ __forceinline__ void sel_descend(const unsigned long long* h, unsigned long long carry,
                                            double target, SelShared& sh) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const double tc = ceil(target);
    const unsigned long long tu = tc <= 0.0 ? 0ull : (tc >= 1.8e19 ? ~0ull : static_cast<unsigned long long>(tc));
    unsigned long long v[8], lsum = 0ull;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = h[255 - 8 * lane - i];
      lsum += v[i];
    }
    unsigned long long incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    unsigned long long acc = carry + (incl - lsum);  // sum of the digits above this lane's
    int hit = -1;
    unsigned long long above = 0ull;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (hit < 0 && acc + v[i] >= tu) {
        hit = 255 - 8 * lane - i;
        above = acc;
      }
      acc += v[i];
    }
    // the digit 0 takes whatever is left (the target is always reached by then)
    if (lane == 31 && hit < 0) {
      hit = 0;
      above = acc - v[7];
    }
    const unsigned m = __ballot_sync(0xffffffffu, hit >= 0);
    const int src = __ffs(m) - 1;
    const int d = __shfl_sync(0xffffffffu, hit, src);
    const unsigned long long ab = __shfl_sync(0xffffffffu, above, src);
    if (lane == 0) {
      sh.digit = d;
      sh.above = ab;
    }
  }
  __syncthreads();
}

// over a list in shared memory: the largest key K such that the weights
// (counts when w is null) of the entries with key >= K, among those with key
// >= floor, reach target -- the radix descent of sel_histogram, 8 bits a level
static __device__ unsigned list_descend(const unsigned* keys, const unsigned long long* w, int n, unsigned floor,
                                 double target, SelShared& sh) {
  const int tid = threadIdx.x;
  unsigned prefix = 0u;
  unsigned long long carry = 0ull;
  for (int l = 0; l < 4; ++l) {
    const int shift = 24 - 8 * l;
    const unsigned hi_mask = shift + 8 >= 32 ? 0u : (0xffffffffu << (shift + 8));
    for (int d = tid; d < 256; d += kSelThreads) sh.hcnt[d] = 0ull;
    __syncthreads();
    for (int i = tid; i < n; i += kSelThreads) {
      const unsigned kx = keys[i];
      if (kx < floor || (kx & hi_mask) != (prefix & hi_mask)) continue;
      atomicAdd(&sh.hcnt[(kx >> shift) & 255u], w ? w[i] : 1ull);
    }
    __syncthreads();
    sel_descend(sh.hcnt, carry, target, sh);
    carry = sh.above;
    prefix |= static_cast<unsigned>(sh.digit) << shift;
    __syncthreads();
  }
  return prefix;
}

constexpr int kRankCap = 512;  // lists this short are selected by ranks (one entry per thread)

// the same selection as list_descend for a short list (n <= kRankCap): each
// thread takes one entry and sums the weights of the entries at or above it
// (a sweep of the list, read by every thread at once), and the answer is the
// largest key whose sum reaches the target -- one pass instead of four radix
// levels with their barriers.  When no key reaches it (the radix descent then
// ends at its lowest prefix), the smallest key at or above floor.
static __device__ unsigned rank_select(const unsigned* keys, const unsigned long long* w, int n,
                                       unsigned floor, double target, SelShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const double tc = ceil(target);
  const unsigned long long tu = tc <= 0.0 ? 0ull : (tc >= 1.8e19 ? ~0ull : static_cast<unsigned long long>(tc));
  unsigned best = 0u, lowest = 0xffffffffu;
  bool hit = false;
  if (tid < n) {
    const unsigned ki = keys[tid];
    if (ki >= floor) {
      unsigned long long acc = 0ull;
#pragma unroll 4
      for (int j = 0; j < n; ++j) {
        const unsigned kj = keys[j];
        if (kj >= ki) acc += w ? w[j] : 1ull;
      }
      hit = acc >= tu;
      best = hit ? ki : 0u;
      lowest = ki;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
    lowest = min(lowest, __shfl_xor_sync(0xffffffffu, lowest, o));
  }
  const unsigned any = __ballot_sync(0xffffffffu, hit);
  if (lane == 0) {
    sh.wfirst[warp] = static_cast<int>(best);
    sh.wsum[warp] = (static_cast<unsigned long long>(any != 0u) << 32) | lowest;
  }
  __syncthreads();
  unsigned K = 0u, low = 0xffffffffu;
  bool found = false;
  for (int q = 0; q < kSelWarps; ++q) {
    K = max(K, static_cast<unsigned>(sh.wfirst[q]));
    low = min(low, static_cast<unsigned>(sh.wsum[q] & 0xffffffffull));
    found |= (sh.wsum[q] >> 32) != 0ull;
  }
  __syncthreads();
  return found ? K : (low == 0xffffffffu ? floor : low);
}

static __device__ unsigned list_select(const unsigned* keys, const unsigned long long* w, int n, unsigned floor,
                                       double target, SelShared& sh) {
  if (n <= kRankCap) return rank_select(keys, w, n, floor, target, sh);
  return list_descend(keys, w, n, floor, target, sh);
}

// Each row's lower bound of its top-k set for the gathering pass: the k-th
// largest scaled chunk maximum (k distinct logits reach it, so the k-th
// largest logit does too, and rounding is monotone), +inf for a row that is
// not gathered.  One warp per row; the row's chunk maxima are staged in the
// warp's shared memory and every lane ranks its own against all of them.
constexpr int kBoundWarps = 8;
template <typename TT, typename TD>
__global__ void __launch_bounds__(32 * kBoundWarps)
    bound_kernel(const __grid_constant__ Params P, const __grid_constant__ FilterParams F) {
  __shared__ unsigned keys[kBoundWarps][kBoundCap];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = static_cast<int>(blockIdx.x) * kBoundWarps + warp;  // b * rows + r
  if (g >= P.B * P.rows) return;
  const Filter f = F.f[g % P.rows > P.k ? 1 : 0];
  const int n = P.nchunk;
  if (!gathers_row(f, n)) {
    if (lane == 0) F.gbound[g] = INFINITY;
    return;
  }
  const float2* part = P.part + static_cast<int64_t>(g) * n;
  for (int ch = lane; ch < n; ch += 32) keys[warp][ch] = key_of(ldcg_f2(part + ch).x);
  __syncwarp();
  // the k-th largest key (counted with its repeats): the key with fewer than k
  // keys above it and at least k at or above
  unsigned K = 0u;
  for (int i = lane; i < n; i += 32) {
    const unsigned ki = keys[warp][i];
    int gt = 0, ge = 0;
    for (int j = 0; j < n; ++j) {
      const unsigned kj = keys[warp][j];
      gt += kj > ki;
      ge += kj >= ki;
    }
    if (gt < f.top_k && f.top_k <= ge) K = ki;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) K = max(K, __shfl_xor_sync(0xffffffffu, K, o));
  // a NaN chunk maximum (an invalid row) ranks as a key like any other; such
  // a row is rejected by the verification whatever is gathered
  if (lane == 0) F.gbound[g] = float_of_key(K);
}

// Rows whose top-k set the gathering pass collected in full (no chunk over
// its cap, at most kRankCap logits in all): the whole selection by a small CTA
// per row on the row's list in shared memory -- a bitonic sort by decreasing
// key, then top-k by position (the k-th largest key with its repeats), top-p
// by a prefix sum over the top-k survivors' masses, min-p by bisection: the
// decisions of select_kernel's list path.  Writes each such row's key,
// threshold and kept index and done[g] = 1; every other row gets done[g] = 0
// and is selected by select_kernel.
constexpr int kLSelThreads = 256;
constexpr int kLSelWarps = kLSelThreads / 32;
template <typename TT, typename TD>
__global__ void __launch_bounds__(kLSelThreads)
    list_select_kernel(const __grid_constant__ Params P, const __grid_constant__ FilterParams F) {
  __shared__ unsigned key[kRankCap];
  __shared__ unsigned long long mass[kRankCap];
  __shared__ unsigned long long wred[kLSelWarps];
  __shared__ float wmax[kLSelWarps];
  __shared__ int wint[kLSelWarps];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = static_cast<int>(blockIdx.x);  // b * rows + r
  const Filter f = F.f[g % P.rows > P.k ? 1 : 0];
  const int nch = P.nchunk;
  const bool use_p = f.top_p < 1.f, use_m = f.min_p > 0.f;
  if (!(f.top_k < P.V && gathers_row(f, nch))) {
    if (tid == 0) F.done[g] = 0;
    return;
  }
  // the row's scaled maximum; the counts of chunks tid and tid + kLSelThreads
  // (nch <= kBoundCap = 2 kLSelThreads) and their list offsets (block scans
  // in chunk order)
  const float2* part = P.part + static_cast<int64_t>(g) * nch;
  const unsigned* cnt = F.gcount + static_cast<int64_t>(g) * nch;
  float M = -INFINITY;
  unsigned m0 = 0u, m1 = 0u;
  if (tid < nch) {
    M = ldcg_f2(part + tid).x;
    m0 = __ldcg(cnt + tid);
  }
  if (tid + kLSelThreads < nch) {
    M = fmaxf(M, ldcg_f2(part + tid + kLSelThreads).x);
    m1 = __ldcg(cnt + tid + kLSelThreads);
  }
  const int over = (m0 > static_cast<unsigned>(kGatherCap)) || (m1 > static_cast<unsigned>(kGatherCap));
  if (over) m0 = m1 = 0u;
  M = warp_max(M);
  if (lane == 0) wmax[warp] = M;
  int tot0, tot1;
  const int w0 = warp_excl_scan_int(static_cast<int>(m0), lane, tot0);
  const int w1 = warp_excl_scan_int(static_cast<int>(m1), lane, tot1);
  if (lane == 0) {
    wint[warp] = tot0;
    wred[warp] = static_cast<unsigned long long>(tot1);
  }
  const int anyover = __syncthreads_or(over);
  int base0 = 0, all0 = 0, base1 = 0, all1 = 0;
  M = -INFINITY;
  for (int w = 0; w < kLSelWarps; ++w) {
    if (w < warp) {
      base0 += wint[w];
      base1 += static_cast<int>(wred[w]);
    }
    all0 += wint[w];
    all1 += static_cast<int>(wred[w]);
    M = fmaxf(M, wmax[w]);
  }
  const int n = all0 + all1;
  base1 += all0;
  __syncthreads();
  if (!(M > -INFINITY) || !isfinite(M)) {  // an invalid row: nothing to filter
    if (tid == 0) {
      F.key[g] = 0u;
      F.first[g] = -1;
      F.thr[g] = -INFINITY;
      F.done[g] = 1;
    }
    return;
  }
  if (anyover || n > kRankCap) {
    if (tid == 0) F.done[g] = 0;
    return;
  }
  const float c = P.c, Mc = M;
  // the list: every thread copies its chunks' entries to their offsets
  const float* lst = F.glist + static_cast<int64_t>(g) * nch * kGatherCap;
  auto copy_chunk = [&](int ch, unsigned m, int o) {
#pragma unroll 4
    for (unsigned i = 0; i < m; ++i) {
      const float x = __ldcg(lst + ch * kGatherCap + i);
      key[o + i] = key_of(x);
      mass[o + i] = use_p ? __float2ull_rn(ex2_approx(fmaf(x, c, -Mc)) * kMassScalef) : 0ull;
    }
  };
  copy_chunk(tid, m0, base0 + w0);
  copy_chunk(tid + kLSelThreads, m1, base1 + w1);
  int N = 32;
  while (N < n) N <<= 1;
  for (int i = n + tid; i < N; i += kLSelThreads) {  // padding below every logit's key
    key[i] = 0u;
    mass[i] = 0ull;
  }
  __syncthreads();
  // bitonic sort by decreasing key (blocks with (i & k) == 0 run descending;
  // the last merge, k = N, is descending throughout)
  for (int k = 2; k <= N; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < N; i += kLSelThreads) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned a = key[i], b = key[l];
          if ((i & k) == 0 ? a < b : a > b) {
            key[i] = b;
            key[l] = a;
            const unsigned long long t = mass[i];
            mass[i] = mass[l];
            mass[l] = t;
          }
        }
      }
      __syncthreads();
    }
  // n >= top_k: each of the top_k chunks at or above the bound gave its maximum
  unsigned K = key[f.top_k - 1];
  if (use_p) {
    // inclusive prefix sums of the masses in sorted order (thread t: entries
    // 2t and 2t + 1; N <= 2 kLSelThreads)
    const int i0 = 2 * tid;
    const unsigned long long a0 = i0 < N ? mass[i0] : 0ull, a1 = i0 + 1 < N ? mass[i0 + 1] : 0ull;
    const unsigned long long run = a0 + a1;
    unsigned long long incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) wred[warp] = incl;
    __syncthreads();
    unsigned long long before = incl - run;
    for (int w = 0; w < warp; ++w) before += wred[w];
    if (i0 < N) mass[i0] = before + a0;
    if (i0 + 1 < N) mass[i0 + 1] = before + a0 + a1;
    __syncthreads();
    // S_k: the prefix up to the last entry at or above K; then the largest key
    // (the first tie group) whose prefix reaches ceil(top_p S_k)
    int last = 0;
    for (int i = tid; i < N; i += kLSelThreads)
      if (key[i] >= K && (i + 1 == N || key[i + 1] < K)) last = i;
    last = __reduce_max_sync(0xffffffffu, last);
    if (lane == 0) wint[warp] = last;
    __syncthreads();
    for (int w = 0; w < kLSelWarps; ++w) last = max(last, wint[w]);
    const double tc = ceil(static_cast<double>(f.top_p) * static_cast<double>(mass[last]));
    const unsigned long long tu = tc <= 0.0 ? 0ull : static_cast<unsigned long long>(tc);
    int hit = N;
    for (int i = tid; i <= last; i += kLSelThreads)
      if ((i + 1 == N || key[i + 1] != key[i]) && mass[i] >= tu) hit = min(hit, i);
    hit = __reduce_min_sync(0xffffffffu, hit);
    __syncthreads();
    if (lane == 0) wint[warp] = hit;
    __syncthreads();
    for (int w = 0; w < kLSelWarps; ++w) hit = min(hit, wint[w]);
    if (hit < N && key[hit] > K) K = key[hit];
  }
  if (tid == 0) {
    if (use_m) {
      // min-p: the smallest key whose logit passes, never above the row's largest
      const unsigned kmax = key[0];
      const float lmp = log2f(f.min_p);
      unsigned lo = 0u, hi = key_of(INFINITY);
      while (hi - lo > 1u) {
        const unsigned mid = lo + (hi - lo) / 2u;
        const float xm = float_of_key(mid);
        if (!isnan(xm) && fmaf(xm, c, -Mc) >= lmp) hi = mid;
        else lo = mid;
      }
      K = max(K, min(hi, kmax));
    }
    F.key[g] = K;
    F.first[g] = -1;
    F.thr[g] = thr_of_key(K);
    F.done[g] = 1;
  }
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
  if (F.done && __ldcg(F.done + g)) return;  // selected by list_select_kernel
  const int V = P.V;
  const bool use_k = f.top_k >= 2 && f.top_k < V;
  const bool use_p = f.top_p < 1.f;
  const bool use_m = f.min_p > 0.f;
  if (f.top_k != 1 && !use_k && !use_p && !use_m) {
    if (tid == 0) {
      F.key[g] = 0u;
      F.first[g] = -1;
      F.thr[g] = -INFINITY;
    }
    return;
  }
  // the row's scaled maximum from the chunk statistics, and the first chunk
  // holding it (one warp)
  if (warp == 0) {
    const float2* part = P.part + static_cast<int64_t>(g) * P.nchunk;
    float M = -INFINITY;
    int mch = P.nchunk;
    for (int ch = lane; ch < P.nchunk; ch += 32) {
      const float m = ldcg_f2(part + ch).x;
      if (m > M) {
        M = m;
        mch = ch;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float oM = __shfl_xor_sync(0xffffffffu, M, o);
      const int och = __shfl_xor_sync(0xffffffffu, mch, o);
      if (oM > M || (oM == M && och < mch)) {
        M = oM;
        mch = och;
      }
    }
    if (lane == 0) {
      sh.Mc = M;
      sh.digit = mch;
      sh.bad = !(M > -INFINITY) || !isfinite(M);
    }
  }
  __syncthreads();
  const float Mc = sh.Mc, c = P.c;
  const int mch = sh.digit;
  __syncthreads();
  if (sh.bad) {  // an invalid row: the verification flags it; nothing to filter
    if (tid == 0) {
      F.key[g] = 0u;
      F.first[g] = -1;
      F.thr[g] = -INFINITY;
    }
    return;
  }
  auto run = [&](const auto* row) {
    using T = typename std::remove_const<typename std::remove_pointer<decltype(row)>::type>::type;
    const bool vec = (draft ? P.vec_d : P.vec_t) != 0;
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
        F.thr[g] = tb;
      }
      return;
    }
    const int levels = sizeof(T) == 2 ? 2 : 4;  // bf16 keys have 16 significant bits
    unsigned K = 0u;
    // With top-k (k at most the number of chunks): the k-th largest chunk
    // maximum is a lower bound of the k-th largest logit (the k chunk maxima
    // are k distinct logits), and rounding is monotone, so every logit of the
    // top-k set has fl(x c) at or above the k-th largest scaled chunk maximum.
    // One pass gathers those logits; the selections then run on the list.
    bool listed = false;
    // the gathering pass's lists, when it ran and no chunk of the row overflowed
    bool gathered = false;
    if (use_k && F.gcount && gathers_row(f, P.nchunk)) {
      if (tid == 0) {
        sh.ln = 0;
        sh.bad = 0;
      }
      __syncthreads();
      const unsigned* cnt = F.gcount + static_cast<int64_t>(g) * P.nchunk;
      const float* lst = F.glist + static_cast<int64_t>(g) * P.nchunk * kGatherCap;
      for (int ch = tid; ch < P.nchunk; ch += kSelThreads) {
        const unsigned m = __ldcg(cnt + ch);
        if (m > static_cast<unsigned>(kGatherCap)) {
          sh.bad = 1;  // (shared flag reused: the row reads itself below)
          continue;
        }
        const int base = m ? atomicAdd(&sh.ln, static_cast<int>(m)) : 0;
        for (unsigned i = 0; i < m; ++i) {
          const float x = __ldcg(lst + ch * kGatherCap + i);
          if (base + static_cast<int>(i) < kListCap) {
            sh.lkey[base + i] = key_of(x);
            sh.lmass[base + i] = use_p ? __float2ull_rn(ex2_approx(fmaf(x, c, -Mc)) * kMassScalef) : 0ull;
          }
        }
      }
      __syncthreads();
      gathered = !sh.bad;
      __syncthreads();
      if (tid == 0) sh.bad = 0;
      __syncthreads();
    }
    if (use_k && f.top_k <= P.nchunk && !gathered) {
      const float2* part = P.part + static_cast<int64_t>(g) * P.nchunk;
      for (int ch = tid; ch < P.nchunk; ch += kSelThreads) sh.lkey[ch] = key_of(ldcg_f2(part + ch).x);
      if (tid == 0) sh.ln = 0;
      __syncthreads();
      const float th = float_of_key(list_select(sh.lkey, nullptr, P.nchunk, 0u,
                                                 static_cast<double>(f.top_k), sh));
      // warp-uniform trip count: the ballots below need every lane
#pragma unroll
      for (int a = 0; a < kSelAhead; ++a) {
        const int vp = warp * 256 + lane * 8 + a * kSelWarps * 256;
        if (vp < V) prefetch_l2(row + vp);
      }
      // two 256-entry blocks per warp and iteration, both loads issued before
      // either is used
#pragma unroll 1
      for (int wb = warp * 256; wb < V; wb += 2 * kSelWarps * 256) {
        float x[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int v0 = wb + u * kSelWarps * 256 + lane * 8;
          if (v0 + kSelAhead * kSelWarps * 256 < V) prefetch_l2(row + v0 + kSelAhead * kSelWarps * 256);
          load8<T>(row, v0, V, vec, x[u]);  // entries past V read as -inf
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int v0 = wb + u * kSelWarps * 256 + lane * 8;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const bool take = v0 + e < V && x[u][e] * c >= th;
            const unsigned m = __ballot_sync(0xffffffffu, take);
            if (m == 0u) continue;
            int base = 0;
            if (lane == __ffs(m) - 1) base = atomicAdd(&sh.ln, __popc(m));
            base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
            const int pos = base + __popc(m & ((1u << lane) - 1u));
            if (take && pos < kListCap) {
              sh.lkey[pos] = key_of(x[u][e]);
              sh.lmass[pos] = use_p ? __float2ull_rn(ex2_approx(fmaf(x[u][e], c, -Mc)) * kMassScalef) : 0ull;
            }
          }
        }
      }
      __syncthreads();
    }
    if (use_k && f.top_k <= P.nchunk) {
      const int n = sh.ln;
      if (n <= kListCap) {
        listed = true;
        K = list_select(sh.lkey, nullptr, n, 0u, static_cast<double>(f.top_k), sh);
        if (use_p) {
          // S_k: the mass of the top-k survivors; then top-p among them
          unsigned long long part_sum = 0ull;
          for (int i = tid; i < n; i += kSelThreads)
            if (sh.lkey[i] >= K) part_sum += sh.lmass[i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) part_sum += __shfl_xor_sync(0xffffffffu, part_sum, o);
          if (lane == 0) sh.wsum[warp] = part_sum;
          __syncthreads();
          if (tid == 0) {
            unsigned long long t = 0ull;
            for (int w = 0; w < kSelWarps; ++w) t += sh.wsum[w];
            sh.Sk = t;
          }
          __syncthreads();
          const unsigned Kp = list_select(sh.lkey, sh.lmass, n, K,
                                          static_cast<double>(f.top_p) * static_cast<double>(sh.Sk), sh);
          if (Kp > K) K = Kp;
        }
      }
      __syncthreads();
    }
    // top-k by radix descent over the whole row: the k-th largest key, and
    // (for top-p) the mass at or above it
    if (use_k && !listed) {
      unsigned prefix = 0u;
      unsigned long long carry_c = 0ull, carry_m = 0ull;
      for (int l = 0; l < levels; ++l) {
        const int shift = 24 - 8 * l;
        sel_histogram<T>(row, V, vec, c, Mc, prefix, shift, use_p, sh);
        if (l == 0 && use_p)
          for (int d = tid; d < 256; d += kSelThreads) sh.h0mass[d] = sh.hmass[d];
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
    if (use_p && !listed) {
      unsigned prefix = 0u;
      unsigned long long carry = 0ull;
      for (int l = 0; l < levels; ++l) {
        const int shift = 24 - 8 * l;
        if (l == 0 && use_k) {
          // the level-0 masses are the top-k pass's
          for (int d = tid; d < 256; d += kSelThreads) sh.hmass[d] = sh.h0mass[d];
          __syncthreads();
        } else {
          sel_histogram<T>(row, V, vec, c, Mc, prefix, shift, true, sh);
        }
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
      // the row's largest key lies in the chunk holding the largest scaled max
      unsigned km = 0u;
      const int c0 = mch * kChunk;
      for (int v = c0 + tid; v < min(V, c0 + kChunk); v += kSelThreads) km = max(km, key_of(row_at<T>(row, v)));
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
      F.thr[g] = thr_of_key(K);
    }
  };
  if (!draft) run(static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (P.k + 1) + r) * V);
  else run(static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * P.k + (r - P.k - 1)) * V);
}

}  // namespace sv
