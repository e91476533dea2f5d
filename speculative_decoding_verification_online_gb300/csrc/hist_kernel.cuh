// hist_kernel.cuh -- the sampler filters of bf16 rows from one read of each
// row (mlxcel PR #992, "What changed": temperature, top-k, top-p, min-p, then
// the softmax of the survivors).
//
// A bf16 logit takes one of 65536 values, so a row's histogram over the
// values decides every filter exactly: top-k is the value at which the count
// from the top first reaches k; and since equal logits carry equal masses,
// the mass of a value is its count times the fixed-point mass
// 2^40 exp2(x c - Mc) of one of its tokens -- the same integers the list and
// radix selections of filter_kernel.cuh sum token by token -- so top-p is the
// value at which the mass from the top first reaches ceil(top_p S_k).  The
// counters cover the magnitudes [2^-15, 2^9) of both signs, 3072 values each
// (24 KB of shared memory, a CTA per row, five CTAs per SM); side counters
// take the rest: zeros (+0 and -0, equal as logits), the tiny values
// 0 < |x| < 2^-15 (kept in a short list, each with its own mass), and
// |x| >= 2^9 (counted, with the largest of the negative ones).  The row's
// maximum comes from the same read (packed bf16 maxima); min-p alone needs
// nothing else, and its rows count nothing.  A top-k row counts its first
// logits in full and then only the logits at or above their k-th largest
// (hist_sweep_cut): the decisions never look below the row's k-th largest.  A row whose answer lies outside
// the exact counters -- a logit >= 2^9, a threshold among the tiny values or
// below -2^9, a tiny list over its cap, or logits below -2^9 whose masses are
// not all zero under top-p -- is selected by a radix descent over its 16-bit
// keys in up to four more reads: the same decisions, slower.
#pragma once

#include "filter_kernel.cuh"

namespace sv {

constexpr int kHThreads = 256;
constexpr int kHWarps = kHThreads / 32;
constexpr unsigned kMagLo = 0x3800u;  // bf16 magnitude bits of 2^-15
constexpr unsigned kMagHi = 0x4400u;  // and of 2^9
constexpr int kHSide = static_cast<int>(kMagHi - kMagLo);  // exact counters per sign
// The counters: [0, kHSide) negative values and [kHSide, 2 kHSide) positive
// ones, each at (magnitude bits - kMagLo), then zero and the two tiny classes.
constexpr int kHZero = 2 * kHSide, kHNegTiny = kHZero + 1, kHPosTiny = kHZero + 2;
constexpr int kHBins = 2 * kHSide + 3;
// The scans take them by rank, in decreasing order of value: positive values,
// the tiny positive ones, zero, the tiny negative ones, negative values.
constexpr int kRPosTiny = kHSide, kRZero = kHSide + 1, kRNegTiny = kHSide + 2, kRNeg0 = kHSide + 3;
// The scans sum blocks of 128 counters, contiguous in memory and in rank:
// rank blocks [0, kHPB) are the positive counters from the top (each block
// in decreasing order of its counters), block kHPB the three side counters,
// blocks (kHPB, kHNBlk) the negative counters (increasing order).
constexpr int kHBlk = 128;
constexpr int kHPB = kHSide / kHBlk;       // 24 blocks per sign
constexpr int kHNBlk = 2 * kHPB + 1;       // 49 rank blocks
static_assert(kHSide % kHBlk == 0 && kHNBlk <= 64, "two blocks per lane in a crossing");
constexpr int kTinyCap = 64;              // tiny values listed per sign
constexpr unsigned kKeyNegInf = 0x007fu;  // 16-bit key of -inf
constexpr unsigned kKeyPosInf = 0xff80u;  // and of +inf

// the rows of a side that hist_kernel selects: bf16 logits with any filter
// but top_k = 1 (whose kept index select_kernel finds), or no filter at all
__host__ __device__ inline bool hist_selects(const Filter& f, bool bf16) {
  const bool on = f.top_k != 0 || f.top_p < 1.f || f.min_p > 0.f;
  return !on || (bf16 && f.top_k != 1);
}

struct alignas(16) HistShared {  // (16-byte loads of the counters)
  union {
    unsigned cnt[kHBins];
    struct {  // the radix fallback's level histograms, one per warp
      unsigned c[kHWarps][256];
      unsigned long long m[kHWarps][256];
    } fb;
  };
  float tiny[2][kTinyCap];  // [0] negative, [1] positive
  unsigned ntiny[2];
  unsigned nbelow, kbelow;  // logits <= -2^9 (-inf too) and their largest 16-bit key
  unsigned nabove;          // finite logits >= 2^9
  int bad;                  // a NaN or +inf: an invalid row
  uint4 queue[kHWarps][2 * 32];  // per warp: vectors at or above a top-k row's cut, to count
  unsigned bcnt[kHNBlk];    // per block of 32 ranks: counts and masses
  unsigned long long bmass[kHNBlk];
  unsigned long long wsum[kHWarps];  // per warp: its blocks' mass
  unsigned wmax[kHWarps];
  int hit;
  unsigned long long hit_incl;
  int dig;
  unsigned long long dig_above, dig_total;
};
static_assert(sizeof(unsigned[kHBins]) >= sizeof(unsigned[kHWarps][256]) + sizeof(unsigned long long[kHWarps][256]),
              "the fallback's histograms fit the counters' memory");

// 16-bit order-preserving key of a bf16 pattern, and the 32-bit key (key_of)
// of the same value as fp32
__device__ __forceinline__ unsigned key16_of(unsigned h) {
  return (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
}
__device__ __forceinline__ unsigned key32_of16(unsigned k16) {
  return (k16 << 16) | (k16 < 0x8000u ? 0xffffu : 0u);
}
__device__ __forceinline__ float value_of16(unsigned k16) { return float_of_key(key32_of16(k16)); }

__device__ __forceinline__ unsigned long long mass_of(float x, float c, float Mc) {
  return __float2ull_rn(ex2_approx(fmaf(x, c, -Mc)) * kMassScalef);
}

__device__ __forceinline__ bool rank_tiny(int r) { return r == kRPosTiny || r == kRNegTiny; }
// bf16 pattern of an exact rank or of zero (as -0, which the thresholds treat like +0)
__device__ __forceinline__ unsigned rank_bits(int r) {
  if (r < kHSide) return static_cast<unsigned>(kHSide - 1 - r) + kMagLo;
  if (r == kRZero) return 0x8000u;
  return 0x8000u | (static_cast<unsigned>(r - kRNeg0) + kMagLo);
}

// ---- the read

// everything outside the exact counters
__device__ __forceinline__ void hist_rare(unsigned h, HistShared& sh) {
  const unsigned a = h & 0x7fffu;
  const bool neg = (h & 0x8000u) != 0u;
  if (a == 0u) {
    atomicAdd(&sh.cnt[kHZero], 1u);
  } else if (a < kMagLo) {
    const int s = neg ? 0 : 1;
    const unsigned slot = atomicAdd(&sh.ntiny[s], 1u);
    if (slot < static_cast<unsigned>(kTinyCap)) sh.tiny[s][slot] = __uint_as_float(h << 16);
  } else if (a > 0x7f80u || (!neg && a == 0x7f80u)) {
    sh.bad = 1;  // NaN or +inf
  } else if (neg) {
    atomicAdd(&sh.nbelow, 1u);
    atomicMax(&sh.kbelow, key16_of(h));
  } else {
    atomicAdd(&sh.nabove, 1u);
  }
}

// one logit (bf16 pattern h) into its counter
__device__ __forceinline__ void hist_one(unsigned h, HistShared& sh) {
  const unsigned d = (h & 0x7fffu) - kMagLo;
  if (d < static_cast<unsigned>(kHSide)) atomicAdd(&sh.cnt[d + ((h & 0x8000u) ? 0u : kHSide)], 1u);
  else hist_rare(h, sh);
}

// the entries (bit 2e + s: half s of word e) of eight logits, out of line:
// most vectors have none
static __device__ __noinline__ void hist_some8(uint4 u, unsigned bits, HistShared& sh) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  while (bits) {
    const int i = __ffs(bits) - 1;
    bits &= bits - 1u;
    hist_one((i & 1) ? w[i >> 1] >> 16 : w[i >> 1] & 0xffffu, sh);
  }
}

// packed bf16 maximum that keeps a NaN (either operand NaN: NaN)
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// both bf16 halves of v below the same halves of t (ordered: a NaN is not below)
__device__ __forceinline__ bool both_below(uint32_t v, uint32_t t) {
  uint32_t r;
  asm("{\n\t.reg .pred p, q;\n\tsetp.lt.bf16x2 p|q, %1, %2;\n\tand.pred p, p, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(v), "r"(t));
  return r != 0u;
}

// What a sweep does with each 16-byte vector (eight logits): kMaxOnly the
// packed maximum alone; kCountAll the maximum and every logit into its counter.
enum : int { kMaxOnly = 0, kCountAll = 1 };

template <int kHow>
__device__ __forceinline__ void hist_visit(const uint4& u, unsigned& mx, HistShared& sh) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) mx = bmax2(mx, w[e]);
  if constexpr (kHow != kMaxOnly) {
    unsigned rare = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // both magnitudes minus kMagLo at once: when both are at least kMagLo
      // nothing borrows, and d < kHSide exactly when neither d nor
      // d + 0x7400 has bit 15 set; any other word goes out of line whole
      const uint32_t d2 = (w[e] & 0x7fff7fffu) - (kMagLo | (kMagLo << 16));
      if (((d2 | (d2 + 0x74007400u)) & 0x80008000u) == 0u) {
        // both counters at once: kHSide added to each positive half (the sum
        // stays below 2 kHSide, so nothing carries between the halves)
        const uint32_t i2 = d2 + ((~w[e] >> 15) & 0x00010001u) * static_cast<uint32_t>(kHSide);
        atomicAdd(&sh.cnt[i2 & 0xffffu], 1u);
        atomicAdd(&sh.cnt[i2 >> 16], 1u);
      } else {
        rare |= 3u << (2 * e);
      }
    }
    if (rare) hist_some8(u, rare, sh);
  }
}

// a streamed 16-byte load that leaves L1 to the kernel's own data
__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// the row's vectors [first, nv) (first: this thread's first vector): two sets
// of four 16-byte vectors per thread, one in flight while the other is visited
template <int kHow>
__device__ __forceinline__ void hist_sweep(const uint4* r4, int nv, unsigned& mx, HistShared& sh, int first) {
  // past nv: -inf, which does not raise the maximum (a count skips them)
  const uint4 none = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  uint4 a[4], b[4];
  auto load4 = [&](int base, uint4(&u)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = base + q * kHThreads;
      u[q] = i < nv ? ldg_stream(r4 + i) : none;
    }
  };
  auto visit4 = [&](int base, const uint4(&u)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (kHow == kMaxOnly || base + q * kHThreads < nv) hist_visit<kHow>(u[q], mx, sh);
  };
  int base = first;
  load4(base, a);
  load4(base + 4 * kHThreads, b);
#pragma unroll 1
  for (; base < nv; base += 8 * kHThreads) {
    visit4(base, a);
    load4(base + 8 * kHThreads, a);
    visit4(base + 4 * kHThreads, b);
    load4(base + 12 * kHThreads, b);
  }
}

// ---- the crossings over the ranks (the largest values first)

// rank r's count, and the fixed-point mass of all its logits (a tiny class:
// summed over its list, 0 when the list overflowed -- the caller then falls
// back)
__device__ __forceinline__ unsigned rank_count(int r, const HistShared& sh) {
  if (r < kHSide) return sh.cnt[2 * kHSide - 1 - r];
  if (r >= kRNeg0) return sh.cnt[r - kRNeg0];
  if (r == kRZero) return sh.cnt[kHZero];
  return sh.ntiny[r == kRPosTiny ? 1 : 0];
}
__device__ __forceinline__ unsigned long long rank_mass(int r, unsigned n, float c, float Mc,
                                                        const HistShared& sh) {
  if (n == 0u) return 0ull;
  if (rank_tiny(r)) {
    if (n > static_cast<unsigned>(kTinyCap)) return 0ull;
    const int s = r == kRPosTiny;
    unsigned long long m = 0ull;
    for (unsigned e = 0; e < n; ++e) m += mass_of(sh.tiny[s][e], c, Mc);
    return m;
  }
  return static_cast<unsigned long long>(n) * mass_of(__uint_as_float(rank_bits(r) << 16), c, Mc);
}

// the exact sum over the warp of 64-bit values whose total is below 2^64: four
// 16-bit slices, each summed by one warp reduction (at most 2^21 each)
__device__ __forceinline__ unsigned long long warp_sum_exact(unsigned long long v) {
  const unsigned lo = static_cast<unsigned>(v), hi = static_cast<unsigned>(v >> 32);
  const unsigned s0 = __reduce_add_sync(0xffffffffu, lo & 0xffffu);
  const unsigned s1 = __reduce_add_sync(0xffffffffu, lo >> 16);
  const unsigned s2 = __reduce_add_sync(0xffffffffu, hi & 0xffffu);
  const unsigned s3 = __reduce_add_sync(0xffffffffu, hi >> 16);
  return static_cast<unsigned long long>(s0) + (static_cast<unsigned long long>(s1) << 16) +
         (static_cast<unsigned long long>(s2) << 32) + (static_cast<unsigned long long>(s3) << 48);
}
__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// lane l's four ranks of rank block q, in rank order: their first rank, and
// their counts (side block: lanes 0..2 one rank each)
__device__ __forceinline__ int lane_ranks(int q, int lane, const HistShared& sh, unsigned (&n)[4]) {
  if (q < kHPB) {  // positive counters, decreasing
    const int top = 2 * kHSide - 1 - q * kHBlk - 4 * lane;  // counter of the lane's first rank
    const uint4 u = *reinterpret_cast<const uint4*>(&sh.cnt[top - 3]);
    n[0] = u.w;
    n[1] = u.z;
    n[2] = u.y;
    n[3] = u.x;
    return q * kHBlk + 4 * lane;
  }
  if (q > kHPB) {  // negative counters, increasing
    const int lo = (q - kHPB - 1) * kHBlk + 4 * lane;
    const uint4 u = *reinterpret_cast<const uint4*>(&sh.cnt[lo]);
    n[0] = u.x;
    n[1] = u.y;
    n[2] = u.z;
    n[3] = u.w;
    return kRNeg0 + lo;
  }
  n[0] = lane < 3 ? rank_count(kHSide + lane, sh) : 0u;  // the side counters
  n[1] = n[2] = n[3] = 0u;
  return kHSide + min(lane, 2);
}

// the four ranks' masses from their counts (0 where the count is)
__device__ __forceinline__ void lane_masses(int q, int r0, const unsigned (&n)[4], float c, float Mc,
                                            const HistShared& sh, unsigned long long (&m)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = 0ull;
  if (q == kHPB) {
    m[0] = rank_mass(r0, n[0], c, Mc, sh);
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (n[i]) m[i] = static_cast<unsigned long long>(n[i]) * mass_of(__uint_as_float(rank_bits(r0 + i) << 16), c, Mc);
}

// the rank blocks' sums of counts and (masses) of masses; returns the total mass
static __device__ unsigned long long hist_block_sums(bool masses, float c, float Mc, HistShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long wtot = 0ull;
#pragma unroll 1
  for (int q = warp; q < kHNBlk; q += kHWarps) {
    unsigned n[4];
    const int r0 = lane_ranks(q, lane, sh, n);
    const unsigned cs = __reduce_add_sync(0xffffffffu, (n[0] + n[1]) + (n[2] + n[3]));
    unsigned long long ms = 0ull;
    if (masses && cs) {
      unsigned long long m[4];
      lane_masses(q, r0, n, c, Mc, sh, m);
      ms = warp_sum_exact((m[0] + m[1]) + (m[2] + m[3]));
    }
    if (lane == 0) {
      sh.bcnt[q] = cs;
      sh.bmass[q] = ms;
    }
    wtot += ms;
  }
  if (lane == 0) sh.wsum[warp] = wtot;
  __syncthreads();
  unsigned long long t = 0ull;
#pragma unroll
  for (int w = 0; w < kHWarps; ++w) t += sh.wsum[w];
  return t;
}

// the first rank at which the running counts (by_mass false) or masses reach
// target, and the running mass through it (masses: the block sums hold them);
// rank -1 when the target is not reached.  Warp 0: the rank blocks two per
// lane, then the block's lanes, then the lane's four ranks.
static __device__ void hist_cross(bool by_mass, bool masses, unsigned long long target, float c, float Mc,
                                  HistShared& sh, int* rank, unsigned long long* mass_incl) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int q0 = 2 * lane, q1 = q0 + 1;
    const unsigned long long c0 = q0 < kHNBlk ? sh.bcnt[q0] : 0ull, c1 = q1 < kHNBlk ? sh.bcnt[q1] : 0ull;
    const unsigned long long m0 = masses && q0 < kHNBlk ? sh.bmass[q0] : 0ull;
    const unsigned long long m1 = masses && q1 < kHNBlk ? sh.bmass[q1] : 0ull;
    const unsigned long long ic = warp_incl_scan_u64(c0 + c1, lane);
    const unsigned long long im = masses ? warp_incl_scan_u64(m0 + m1, lane) : 0ull;
    const unsigned hit = __ballot_sync(0xffffffffu, (by_mass ? im : ic) >= target);
    int res = -1;
    unsigned long long resm = 0ull;
    if (hit) {
      const int f = __ffs(hit) - 1;
      // the sums before lane f's blocks, and which of its two blocks
      unsigned long long bc = __shfl_sync(0xffffffffu, ic - (c0 + c1), f);
      unsigned long long bm = __shfl_sync(0xffffffffu, im - (m0 + m1), f);
      const unsigned long long fc0 = __shfl_sync(0xffffffffu, c0, f), fm0 = __shfl_sync(0xffffffffu, m0, f);
      int q = 2 * f;
      if ((by_mass ? bm + fm0 : bc + fc0) < target) {
        bc += fc0;
        bm += fm0;
        ++q;
      }
      // the block's lanes
      unsigned n[4];
      const int r0 = lane_ranks(q, lane, sh, n);
      unsigned long long m[4] = {0ull, 0ull, 0ull, 0ull};
      if (masses) lane_masses(q, r0, n, c, Mc, sh, m);
      const unsigned long long lc = (n[0] + n[1]) + (n[2] + n[3]);
      const unsigned long long lm = (m[0] + m[1]) + (m[2] + m[3]);
      const unsigned long long jc = warp_incl_scan_u64(lc, lane) + bc;
      const unsigned long long jm = masses ? warp_incl_scan_u64(lm, lane) + bm : 0ull;
      const unsigned hit2 = __ballot_sync(0xffffffffu, (by_mass ? jm : jc) >= target);
      if (hit2) {
        const int f2 = __ffs(hit2) - 1;
        // the lane's ranks in order
        int rr = -1;
        unsigned long long ac = jc - lc, am = jm - lm, at = 0ull;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ac += n[i];
          am += m[i];
          if (rr < 0 && (by_mass ? am : ac) >= target) {
            rr = r0 + i;
            at = am;
          }
        }
        res = __shfl_sync(0xffffffffu, rr, f2);
        resm = __shfl_sync(0xffffffffu, at, f2);
      }
    }
    if (lane == 0) {
      sh.hit = res;
      sh.hit_incl = resm;
    }
  }
  __syncthreads();
  *rank = sh.hit;
  *mass_incl = sh.hit_incl;
  __syncthreads();
}

// A top-k row's read in two parts.  The first set of vectors (four per
// thread: the row's first 8192 logits) is counted in full; the k-th largest of
// those logits is at most the row's k-th largest, so every rank the top-k and
// top-p decisions look at -- those at or above the row's k-th largest, whose
// values are then all at or above the cut -- is counted whole when the rest of
// the read counts only the vectors holding a logit at or above the cut.
// Counters below the cut stay partial, and nothing reads them: the counts'
// crossing lies at or above the row's k-th largest, and the top-p target is a
// fraction of the mass through it.  A crossing among the first logits outside
// the exact ranks (none, or a tiny class) sets no cut.
//
// Few vectors reach the cut (about one in twenty on Zipf-like rows), spread at
// random, so a lane that meets one does not count it alone -- the warp would
// issue the whole count for it -- but appends it to its warp's queue (a ballot
// and its prefix count place it); each time 32 are queued the warp counts
// them, one vector per lane.  A vector holding a NaN is never below the cut,
// so an invalid row is still seen.
static __device__ void hist_sweep_cut(const uint4* r4, int nv, int top_k, unsigned& mx, HistShared& sh) {
  const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const uint4 none = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  {
    uint4 a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = tid + q * kHThreads;
      a[q] = i < nv ? ldg_stream(r4 + i) : none;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (tid + q * kHThreads < nv) hist_visit<kCountAll>(a[q], mx, sh);
  }
  __syncthreads();  // the first logits' counts are in
  hist_block_sums(false, 0.f, 0.f, sh);
  int bk;
  unsigned long long unused;
  hist_cross(false, false, static_cast<unsigned long long>(top_k), 0.f, 0.f, sh, &bk, &unused);
  uint32_t cut2 = 0xff80ff80u;  // -inf: no vector is below it
  if (bk >= 0 && !rank_tiny(bk)) {
    const uint32_t t = rank_bits(bk);
    cut2 = t | (t << 16);
  }
  uint4* queue = sh.queue[warp];
  int qn = 0;  // vectors queued (the same on every lane)
  const unsigned lt = (1u << lane) - 1u;
  auto take = [&](const uint4& u, bool in) {
    const uint32_t v = bmax2_nan(bmax2_nan(u.x, u.y), bmax2_nan(u.z, u.w));
    mx = bmax2(mx, v);  // (a NaN half leaves mx's half; the row is invalid anyway)
    const bool hit = in && !both_below(v, cut2);
    const unsigned ball = __ballot_sync(0xffffffffu, hit);
    if (ball) {
      if (hit) queue[qn + __popc(ball & lt)] = u;
      qn += __popc(ball);
      if (qn >= 32) {
        __syncwarp();
        qn -= 32;
        hist_visit<kCountAll>(queue[qn + lane], mx, sh);
        __syncwarp();
      }
    }
  };
  // the rest, from the thread's fifth vector, two sets of four in flight; the
  // loop runs on the warp's first lane's position, so every lane takes every
  // ballot (lanes past the row take nothing)
  uint4 a[4], b[4];
  auto load4 = [&](int base, uint4(&u)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = base + q * kHThreads;
      u[q] = i < nv ? ldg_stream(r4 + i) : none;
    }
  };
  auto take4 = [&](int base, const uint4(&u)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) take(u[q], base + q * kHThreads < nv);
  };
  int base = tid + 4 * kHThreads;
  load4(base, a);
  load4(base + 4 * kHThreads, b);
#pragma unroll 1
  for (; base - lane < nv; base += 8 * kHThreads) {
    take4(base, a);
    load4(base + 8 * kHThreads, a);
    take4(base + 4 * kHThreads, b);
    load4(base + 12 * kHThreads, b);
  }
  __syncwarp();
  if (lane < qn) hist_visit<kCountAll>(queue[lane], mx, sh);
}

__device__ __forceinline__ unsigned long long ceil_target(double t) {
  const double tc = ceil(t);
  return tc <= 0.0 ? 0ull : (tc >= 1.8e19 ? ~0ull : static_cast<unsigned long long>(tc));
}

// ---- the radix fallback: two 8-bit levels over the 16-bit keys

// one read of the row: per digit, counts and masses of the keys >= floor16
// (level 0: by high byte; level 1: by low byte among the keys whose high byte
// is hi), summed per warp and then merged into warp 0's histogram
__device__ __forceinline__ void fb_put(unsigned h, unsigned floor16, int hi, float c, float Mc, HistShared& sh,
                                       int warp) {
  const unsigned k16 = key16_of(h);
  if (k16 < floor16 || (hi >= 0 && static_cast<int>(k16 >> 8) != hi)) return;
  const int d = static_cast<int>(hi < 0 ? k16 >> 8 : k16 & 255u);
  atomicAdd(&sh.fb.c[warp][d], 1u);
  atomicAdd(&sh.fb.m[warp][d], mass_of(__uint_as_float(h << 16), c, Mc));
}
static __device__ void fb_level(const uint16_t* row, int V, bool vec, unsigned floor16, int hi, float c, float Mc,
                                HistShared& sh) {
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kHWarps * 256; i += kHThreads) {
    (&sh.fb.c[0][0])[i] = 0u;
    (&sh.fb.m[0][0])[i] = 0ull;
  }
  __syncthreads();
  if (vec) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
#pragma unroll 1
    for (int i = threadIdx.x; i < (V >> 3); i += kHThreads) {
      const uint4 u = ldg_stream(r4 + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        fb_put(w[e] & 0xffffu, floor16, hi, c, Mc, sh, warp);
        fb_put(w[e] >> 16, floor16, hi, c, Mc, sh, warp);
      }
    }
  } else {
#pragma unroll 1
    for (int v = threadIdx.x; v < V; v += kHThreads) fb_put(__ldg(row + v), floor16, hi, c, Mc, sh, warp);
  }
  __syncthreads();
  for (int d = threadIdx.x; d < 256; d += kHThreads) {
    unsigned cs = 0u;
    unsigned long long ms = 0ull;
#pragma unroll
    for (int w = 0; w < kHWarps; ++w) {
      cs += sh.fb.c[w][d];
      ms += sh.fb.m[w][d];
    }
    sh.fb.c[0][d] = cs;
    sh.fb.m[0][d] = ms;
  }
  __syncthreads();
}

// the highest digit d whose weight from the top, plus carry, reaches target;
// the weight strictly above it and the level's total (one thread: the
// fallback is rare)
static __device__ void fb_descend(bool masses, unsigned long long carry, unsigned long long target,
                                  HistShared& sh) {
  if (threadIdx.x == 0) {
    unsigned long long acc = carry, tot = 0ull;
    int d = -1;
    unsigned long long above = 0ull;
    for (int e = 255; e >= 0; --e) {
      const unsigned long long w = masses ? sh.fb.m[0][e] : sh.fb.c[0][e];
      tot += w;
      if (d < 0 && acc + w >= target) {
        d = e;
        above = acc;
      }
      acc += w;
    }
    if (d < 0) {  // not reached (rounding of an empty tail): the lowest digit
      d = 0;
      above = acc - (masses ? sh.fb.m[0][0] : sh.fb.c[0][0]);
    }
    sh.dig = d;
    sh.dig_above = above;
    sh.dig_total = tot;
  }
  __syncthreads();
}

// the whole row by radix descent: top-k by counts, S_k, top-p among the
// survivors by masses (the decisions of select_kernel's radix path)
static __device__ unsigned fb_select(const uint16_t* row, int V, bool vec, const Filter& f, bool use_k, bool use_p,
                                     float c, float Mc, HistShared& sh) {
  unsigned K16 = 0u;
  unsigned long long Sk = 0ull;
  if (use_k) {
    fb_level(row, V, vec, 0u, -1, c, Mc, sh);
    fb_descend(false, 0ull, static_cast<unsigned long long>(f.top_k), sh);
    const int d0 = sh.dig;
    const unsigned long long cabove = sh.dig_above;
    unsigned long long mabove = 0ull;
    if (threadIdx.x == 0)
      for (int e = 255; e > d0; --e) mabove += sh.fb.m[0][e];
    __syncthreads();
    fb_level(row, V, vec, 0u, d0, c, Mc, sh);
    fb_descend(false, cabove, static_cast<unsigned long long>(f.top_k), sh);
    const int d1 = sh.dig;
    K16 = (static_cast<unsigned>(d0) << 8) | static_cast<unsigned>(d1);
    if (threadIdx.x == 0) {
      unsigned long long m = mabove;
      for (int e = 255; e >= d1; --e) m += sh.fb.m[0][e];
      sh.dig_total = m;  // S_k
    }
    __syncthreads();
    Sk = sh.dig_total;
    __syncthreads();
  }
  if (use_p) {
    fb_level(row, V, vec, K16, -1, c, Mc, sh);
    if (!use_k) {
      if (threadIdx.x == 0) {
        unsigned long long t = 0ull;
        for (int e = 0; e < 256; ++e) t += sh.fb.m[0][e];
        sh.dig_total = t;
      }
      __syncthreads();
      Sk = sh.dig_total;
      __syncthreads();  // (fb_descend rewrites it)
    }
    const unsigned long long tu = ceil_target(static_cast<double>(f.top_p) * static_cast<double>(Sk));
    fb_descend(true, 0ull, tu, sh);
    const int d0 = sh.dig;
    const unsigned long long above = sh.dig_above;
    fb_level(row, V, vec, K16, d0, c, Mc, sh);
    fb_descend(true, above, tu, sh);
    const unsigned Kp = (static_cast<unsigned>(d0) << 8) | static_cast<unsigned>(sh.dig);
    if (Kp > K16) K16 = Kp;
  }
  return use_k || use_p ? key32_of16(K16) : 0u;
}

// One CTA per row g = b * rows + r of a call whose rows are all bf16 or
// unfiltered (any top_k but 1): writes each row's key, logit threshold and
// kept index (-1).
template <typename TT, typename TD>
__global__ void __launch_bounds__(kHThreads, 5)
    hist_kernel(const __grid_constant__ Params P, const __grid_constant__ FilterParams F) {
  __shared__ HistShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = static_cast<int>(blockIdx.x);
  const int b = g / P.rows, r = g % P.rows;
  const bool draft = r > P.k;
  const Filter f = F.f[draft ? 1 : 0];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int V = P.V;
  const bool use_k = f.top_k >= 2 && f.top_k < V;
  const bool use_p = f.top_p < 1.f;
  const bool use_m = f.min_p > 0.f;
  auto finish = [&](unsigned K) {
    if (tid == 0) {
      F.key[g] = K;
      F.first[g] = -1;
      F.thr[g] = thr_of_key(K);
    }
  };
  if (!use_k && !use_p && !use_m) {
    finish(0u);
    return;
  }
  auto run = [&](const auto* rowp) {
    using T = typename std::remove_const<typename std::remove_pointer<decltype(rowp)>::type>::type;
    if constexpr (sizeof(T) != 2) {
      finish(0u);  // not reached: the host sends rows of other types to the other selections
    } else {
      const uint16_t* row = rowp;
      const bool vec = (draft ? P.vec_d : P.vec_t) != 0;
      const bool count = use_k || use_p;  // min-p alone needs the maximum only
      for (int i = tid; i < kHBins; i += kHThreads) sh.cnt[i] = 0u;
      if (tid == 0) {
        sh.ntiny[0] = sh.ntiny[1] = 0u;
        sh.nbelow = sh.nabove = 0u;
        sh.kbelow = 0u;
        sh.bad = 0;
      }
      __syncthreads();
      unsigned mx = 0xff80ff80u;  // packed running maximum (max.bf16x2 passes NaN over)
      if (vec) {
        const uint4* r4 = reinterpret_cast<const uint4*>(row);
        if (use_k) hist_sweep_cut(r4, V >> 3, f.top_k, mx, sh);
        else if (count) hist_sweep<kCountAll>(r4, V >> 3, mx, sh, tid);
        else hist_sweep<kMaxOnly>(r4, V >> 3, mx, sh, tid);
      } else {
#pragma unroll 4
        for (int v = tid; v < V; v += kHThreads) {
          const unsigned h = __ldg(row + v);
          mx = bmax2(mx, h | 0xff800000u);
          if (count) hist_one(h, sh);
        }
      }
      // the row's largest key
      unsigned km = max(key16_of(mx & 0xffffu), key16_of(mx >> 16));
      km = __reduce_max_sync(0xffffffffu, km);
      if (lane == 0) sh.wmax[warp] = km;
      __syncthreads();
      km = 0u;
#pragma unroll
      for (int w = 0; w < kHWarps; ++w) km = max(km, sh.wmax[w]);
      // a NaN or +inf, or nothing above -inf: an invalid row
      if (sh.bad || km <= kKeyNegInf || km >= kKeyPosInf) {
        finish(0u);
        return;
      }
      const float c = P.c;
      const float Mc = value_of16(km) * c;  // fl(x_max c), as the statistics pass writes it
      const unsigned nt0 = sh.ntiny[0], nt1 = sh.ntiny[1];
      unsigned K = 0u;
      bool fallback = sh.nabove > 0u;
      if (!fallback && count) {
        // top-k: the rank where the counts reach k, S_k the masses through
        // it; top-p: the rank where the masses reach ceil(top_p S_k) (at or
        // before it)
        unsigned long long Sk = hist_block_sums(use_p, c, Mc, sh);
        int bk = kHBins - 1;  // the last rank of the top-k survivors
        if (use_k) {
          hist_cross(false, use_p, static_cast<unsigned long long>(f.top_k), c, Mc, sh, &bk, &Sk);
          if (bk < 0 || rank_tiny(bk)) fallback = true;
          else K = key32_of16(key16_of(rank_bits(bk)));
        }
        if (!fallback && use_p) {
          // masses outside the counters: the tiny lists among the survivors
          // must be whole, and (no top-k) the logits below -2^9 must weigh
          // nothing (the largest of them decides)
          fallback = (kRPosTiny <= bk && nt1 > static_cast<unsigned>(kTinyCap)) ||
                     (kRNegTiny <= bk && nt0 > static_cast<unsigned>(kTinyCap)) ||
                     (!use_k && sh.nbelow > 0u && mass_of(value_of16(sh.kbelow), c, Mc) != 0ull);
          if (!fallback) {
            const unsigned long long tu = ceil_target(static_cast<double>(f.top_p) * static_cast<double>(Sk));
            int bp;
            unsigned long long unused;
            hist_cross(true, true, tu, c, Mc, sh, &bp, &unused);
            if (bp < 0 || rank_tiny(bp)) fallback = true;
            else K = max(K, key32_of16(key16_of(rank_bits(bp))));
          }
        }
        __syncthreads();  // (the fallback reuses the counters' memory)
      }
      if (fallback && count) K = fb_select(row, V, vec, f, use_k, use_p, c, Mc, sh);
      if (use_m && warp == 0) {
        // min-p: the smallest bf16 value whose logit passes (the test is
        // monotone in the logit), never above the row's largest -- the kept
        // set of the 32-bit bisection of the other selections.  A 32-way
        // search over the 16-bit keys: the answer lies in (lo, hi], +inf
        // passes, the patterns below -inf (NaN) count as failing.
        const float lmp = log2f(f.min_p);
        unsigned lo = kKeyNegInf - 1u, hi = kKeyPosInf;
        while (hi - lo > 1u) {
          const unsigned step = (hi - lo + 31u) / 32u;
          const unsigned probe = min(hi, lo + 1u + static_cast<unsigned>(lane) * step);
          const bool pass = probe >= kKeyNegInf && fmaf(value_of16(probe), c, -Mc) >= lmp;
          const unsigned ballot = __ballot_sync(0xffffffffu, pass);
          // the first passing probe bounds the answer from above, the probe
          // before it from below; none passing: the last probe from below
          const int first = ballot ? __ffs(ballot) - 1 : 32;
          if (first < 32) {
            const unsigned nlo = first == 0 ? lo : lo + 1u + static_cast<unsigned>(first - 1) * step;
            hi = min(hi, lo + 1u + static_cast<unsigned>(first) * step);
            lo = nlo;
          } else {
            lo = lo + 1u + 31u * step;
          }
        }
        K = max(K, key32_of16(min(hi, km)));
      }
      finish(K);
    }
  };
  if (!draft) run(static_cast<const TT*>(P.Lt) + (static_cast<int64_t>(b) * (P.k + 1) + r) * V);
  else run(static_cast<const TD*>(P.Ld) + (static_cast<int64_t>(b) * P.k + (r - P.k - 1)) * V);
}

}  // namespace sv
