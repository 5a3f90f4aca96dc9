// kps_row.cuh — the one-CTA-per-row kernel (included by kps.cu inside namespace kps).
//
// For batches that fill the GPU every CTA takes whole rows on its own: the row is
// read straight from global memory with 16-byte loads (several in flight per
// thread), there are no cluster barriers and no staging ring, and two CTAs share
// an SM, so a batch of a few hundred rows has every row in flight at once.
//
//   top-k and one-element rows (at most 1024 kept):
//     a sample of 2048 transformed elements (64 runs of 32 spread over the row)
//     gives a threshold tau that about 2.5k + 512 elements of the row reach.  One
//     pass writes the -inf background of the filtered row and appends every
//     element whose raw value can reach tau to its warp's segment of a
//     shared-memory buffer (ballots only: no atomics, no division).  The buffer is
//     then divided by T exactly and cut to tau; when it holds at least k entries
//     and no segment overflowed, its exact k-th entry (value desc, index asc) is
//     the row's.  Otherwise an exact digit select over the row (re-read from L2)
//     replaces the sample.  Top-p (a mass histogram over the survivors), the race
//     and the scatter of the kept values work on the k survivors only.
//   top-p-only rows: pass A divides by T, takes the row maximum M and fills an
//     approximate mass histogram (4096 bins of width 1/64 below H = the sample
//     maximum + 16); the bins whose prefix mass lies within 1e-4 of p * S form a
//     band that must hold the boundary.  Pass B sums the exact fixed-point softmax
//     mass S, races and writes every element above the band and collects the band,
//     which is sorted and cut exactly.  Pass A keeps the row in L2 for pass B.
//   keep-all rows (no top-k, p >= 1): a maximum pass, then the race and write.
//
// The method is the one of the Ascend "torch_npu.npu_top_k_top_p_sample" page
// (topK valid range, topP rule, Sample formulas), MiniMind "Chapter 10: inference
// generation" (§10.4-§10.7) and the C++ post-processing blog (penalty over the set
// of seen ids).  The kernel never waits on another CTA or on memory it does not
// load itself, so it has no timeouts.

static_assert(kThreads == 512, "the block helpers of kps.cu assume 512 threads");

constexpr int kRT = kThreads;           // threads per CTA
constexpr int kRW = kRT / 32;
constexpr int kRU = 4;                  // 16-byte loads each thread keeps in flight
constexpr int kRCap = 6144;             // candidate / band buffer entries (u64 order words)
constexpr int kRSeg = kRCap / kRW;      // the part of the buffer each warp appends to
constexpr int kRKeepAllV = 4096;        // rows this short are taken whole (no sample)
constexpr int kRMaxV = 262144;          // the row's penalty bitmap lives in shared memory
constexpr int kRRuns = 64;              // sampled runs of 32 consecutive elements
constexpr int kRSamp = kRRuns * 32;
constexpr int kRLin = 2048;             // linear count bins of the buffer selection
constexpr float kRHeadroom = 16.0f;     // top-p-only rows: H = sample maximum + headroom
constexpr int kRSurvBins = 1024;        // linear mass bins of top-p over the survivors
constexpr int kRHistWords = 6144;
constexpr int kRRank = 256;             // boundary-bin entries ranked pairwise
constexpr int kRSortMax = 4096;         // largest band the bitonic network sorts
static_assert(kRSeg * kRW == kRCap, "buffer segments");

constexpr int kRMaxItems = 256;        // work units one CTA may own in one launch
constexpr int kRMaxTeam = 4;           // CTAs that may share one row (the cluster size)

struct RLayout {
  size_t bitmap, cw, hist, wbuf, red, misc, items, ords, total;
};

__host__ __device__ inline RLayout make_rlayout(int64_t V) {
  RLayout L;
  size_t off = 0;
  L.bitmap = off; off += align16(size_t((V + 31) / 32) * 4);
  L.cw = off;     off += size_t(kRCap) * 8;     // candidates / band (order words)
  L.hist = off;   off += size_t(kRHistWords) * 4;
  L.wbuf = off;   off += size_t(kTopKMax) * 8;  // sample keys, gathered bins, survivors
  L.red = off;    off += 64 * 8;
  L.misc = off;   off += 64 * 8;
  L.items = off;  off += size_t(kRMaxItems) * 4;
  L.ords = off;   off += size_t(kRMaxItems) * 4;  // pre-pass record of each item (-1: none)
  L.total = off;
  return L;
}

// misc slots (u64) used by the row kernel
enum RMisc {
  kMSel0 = 0, kMSel1 = 1, kMSel2 = 2,  // digit-select results
  kMFound = 4,                         // int32: index found by the tie scan
  kMBin = 8, kMAbove = 9, kMHit = 10,  // bin searches
  kMCut = 11, kMBlo = 12, kMBhi = 13,  // list cut, band bounds
  kMCnt = 16,                          // uint32 counter
  kMSeg = 20,                          // uint32[kRW]: per-warp segment counts (8 slots)
  kMPush = 32,                         // [8][kRMaxTeam]: values pushed by the CTAs sharing a row
};

// ---- loads -------------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long l2_policy_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ unsigned long long l2_policy_last() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ unsigned long long l2_policy_normal() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte read-only load with an L2 eviction policy (not kept in L1).
__device__ __forceinline__ uint4 ld_row16(const uint4* p, unsigned long long pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

template <bool kBF16>
__device__ __forceinline__ void unpack16(const uint4 w, float* v) {
  if (kBF16) {
    v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xFFFF0000u);
    v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xFFFF0000u);
    v[4] = __uint_as_float(w.z << 16); v[5] = __uint_as_float(w.z & 0xFFFF0000u);
    v[6] = __uint_as_float(w.w << 16); v[7] = __uint_as_float(w.w & 0xFFFF0000u);
  } else {
    v[0] = __uint_as_float(w.x); v[1] = __uint_as_float(w.y);
    v[2] = __uint_as_float(w.z); v[3] = __uint_as_float(w.w);
  }
}

// Shared-memory add without a return value (the pointer must address shared memory).
__device__ __forceinline__ void sh_red_add(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// Out-of-line IEEE division: the rare paths call it, so the common path never pays for
// (or speculates) the full division sequence.
__device__ __noinline__ float rdiv_ieee(float x, float d) { return __fdiv_rn(x, d); }

// Penalty of a seen element (applied after NaN -> -inf).
__device__ __forceinline__ float rpenal(float x, float pen) {
  return (x > 0.0f) ? rdiv_ieee(x, pen) : __fmul_rn(x, pen);
}
// x / T rounded to nearest: the multiply-and-correct quotient inside its safe range, the
// IEEE division outside it.
__device__ __forceinline__ float rdiv(float x, const FixedDivisor& dv) {
  const float q = div_fast(x, dv);
  if (dv.fast && div_ok(x, q)) return q;
  return rdiv_ieee(x, dv.T);
}
// Transformed value: NaN -> -inf, the penalty if the element was seen, x / T
// (unless the row is greedy), -0 -> +0.
__device__ __forceinline__ float rtransform(float x, bool seen, float pen, const FixedDivisor& dv, bool identity) {
  if (isnan(x)) x = -INFINITY;
  if (seen) x = rpenal(x, pen);
  if (!identity) x = rdiv(x, dv);
  return __fadd_rn(x, 0.0f);
}
// Floor of 0 <= f < 2^22, by an add rounded down at the scale where the spacing is 1.
__device__ __forceinline__ int rfloor_small(float f) {
  return __float_as_int(__fadd_rd(f, 8388608.0f)) - 0x4B000000;
}

// A raw value below which x / T cannot be kept by a threshold value tv:
// fl(x / T) >= tv implies x >= T * (tv - spacing(tv)).  -inf when tv is not a
// normal number with room (then every element is tested exactly).
__device__ __forceinline__ float raw_floor(float tv, float T, bool identity) {
  if (identity) return tv;
  const float a = fabsf(tv);
  if (!(a >= 1e-30f) || !(a <= 1e30f)) return -INFINITY;
  const float up = __uint_as_float(__float_as_uint(a) + 1u) - a;
  return __double2float_rd(static_cast<double>(T) * (static_cast<double>(tv) - 2.0 * static_cast<double>(up)));
}

struct RowCtx {
  const uint4* x;          // the row of logits as 16-byte vectors
  const float* q;          // the row of q (nullptr: generated draws, or sampling off)
  float* out;              // the row of the filtered logits, or nullptr
  int V;
  int nv;                  // vectors in the row
  int g0, g1;              // the vectors [g0, g1) this CTA covers (a part of a shared row)
  const uint32_t* bitmap;  // seen ids of the row
  bool pen_on;
  float pen;
  float T;
  FixedDivisor div;        // T with its reciprocal
  bool identity;
  bool race;               // a race is run: q given or generated (else sampling off)
  bool gen;                // generated draws
  unsigned long long seed, step;
  int64_t row;             // the row (the generator's counter)
};

// The race's q of token idx, and of the four tokens 4h .. 4h + 3 (loaded, or generated).
// (The generator is called out of line here, so the loaded-q code stays small.)
__device__ __noinline__ float gen_q1_call(unsigned long long seed, unsigned long long step, int64_t row, int idx) {
  return gen_q1(seed, step, row, idx);
}
__device__ __noinline__ float4 gen_q4_call(unsigned long long seed, unsigned long long step, int64_t row, int h) {
  return gen_q4(seed, step, row, h);
}
__device__ __forceinline__ float rq1(const RowCtx& rc, int idx) {
  return rc.gen ? gen_q1_call(rc.seed, rc.step, rc.row, idx) : __ldg(rc.q + idx);
}
__device__ __forceinline__ float4 rq4(const RowCtx& rc, int h) {
  return rc.gen ? gen_q4_call(rc.seed, rc.step, rc.row, h) : __ldcs(reinterpret_cast<const float4*>(rc.q) + h);
}

// Seen-bits of the G elements of vector g (G divides 32, so they share one word).
template <int G>
__device__ __forceinline__ uint32_t rseen_bits(const uint32_t* bitmap, bool pen_on, int g) {
  if (!pen_on) return 0u;
  const int v0 = g * G;
  return (bitmap[v0 >> 5] >> (v0 & 31)) & ((1u << G) - 1u);
}

// One pass over the row: f(valid, y, key, index) per element with the warp converged.
template <bool kBF16, class F>
__device__ __forceinline__ void rrow_pass(const RowCtx& rc, unsigned long long pol, F&& f) {
  constexpr int G = kBF16 ? 8 : 4;
  const uint4* xr = rc.x;
  const int g0 = rc.g0, g1 = rc.g1;
  const uint32_t* bitmap = rc.bitmap;
  const bool pen_on = rc.pen_on, identity = rc.identity;
  const float pen = rc.pen;
  const FixedDivisor dv = rc.div;
  for (int base = g0; base < g1; base += kRT * kRU) {
    uint4 w[kRU];
#pragma unroll
    for (int u = 0; u < kRU; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      w[u] = g < g1 ? ld_row16(xr + g, pol) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kRU; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      const bool in = g < g1;
      float v[G];
      unpack16<kBF16>(w[u], v);
      const uint32_t bits = in ? rseen_bits<G>(bitmap, pen_on, g) : 0u;
#pragma unroll
      for (int e = 0; e < G; ++e) {
        const float y = in ? rtransform(v[e], (bits >> e) & 1u, pen, dv, identity) : 0.0f;
        f(in, y, in ? fkey(y) : 0u, g * G + e);
      }
    }
  }
}

// ---- block helpers (kRT threads) ---------------------------------------------------------
__device__ __forceinline__ void rblock_max2(unsigned long long& a, unsigned long long& b, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_max_u64(a);
  b = warp_max_u64(b);
  if (lane == 0) {
    red[warp] = a;
    red[kRW + warp] = b;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long x = lane < kRW ? red[lane] : 0ull;
    unsigned long long y = lane < kRW ? red[kRW + lane] : 0ull;
    x = warp_max_u64(x);
    y = warp_max_u64(y);
    if (lane == 0) {
      red[48] = x;
      red[49] = y;
    }
  }
  __syncthreads();
  a = red[48];
  b = red[49];
  __syncthreads();
}
// Sum of s and maxima of a and b over the block, in one exchange.
__device__ __forceinline__ void rblock_sum_max2(unsigned long long& s, unsigned long long& a, unsigned long long& b,
                                                unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
  a = warp_max_u64(a);
  b = warp_max_u64(b);
  if (lane == 0) {
    red[warp] = s;
    red[kRW + warp] = a;
    red[2 * kRW + warp] = b;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long x = lane < kRW ? red[lane] : 0ull;
    unsigned long long y = lane < kRW ? red[kRW + lane] : 0ull;
    unsigned long long z = lane < kRW ? red[2 * kRW + lane] : 0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    y = warp_max_u64(y);
    z = warp_max_u64(z);
    if (lane == 0) {
      red[48] = x;
      red[49] = y;
      red[50] = z;
    }
  }
  __syncthreads();
  s = red[48];
  a = red[49];
  b = red[50];
  __syncthreads();
}
__device__ __forceinline__ unsigned long long rblock_sum_u64(unsigned long long v, unsigned long long* red) {
  unsigned long long a = 0, b = 0;
  rblock_sum_max2(v, a, b, red);
  return v;
}
// Exclusive scan in thread order; *total gets the sum.
__device__ __forceinline__ unsigned long long rblock_excl_scan_u64(unsigned long long v, unsigned long long* total,
                                                                   unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long x = warp_incl_scan_u64(v, lane);
  if (lane == 31) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long s = lane < kRW ? red[lane] : 0ull;
    const unsigned long long t = warp_incl_scan_u64(s, lane);
    if (lane < kRW) red[lane] = t - s;
    if (lane == kRW - 1) red[48] = t;
  }
  __syncthreads();
  const unsigned long long res = red[warp] + x - v;
  *total = red[48];
  __syncthreads();
  return res;
}

// Warp-aggregated append of `take` entries through a shared counter; returns the
// position of the first (positions >= capacity are dropped by the caller).
__device__ __forceinline__ uint32_t rwarp_reserve(uint32_t take, uint32_t& cnt) {
  const int lane = threadIdx.x & 31;
  const uint32_t incl = warp_incl_scan_u32(take, lane);
  const uint32_t tot = __shfl_sync(kFull, incl, 31);
  uint32_t b = 0;
  if (tot && lane == 31) b = atomicAdd(&cnt, tot);
  b = __shfl_sync(kFull, b, 31);
  return b + incl - take;
}

// Bitonic sort of a[0..N) (N a power of two) into descending order.
__device__ void rbitonic_desc(unsigned long long* a, int N) {
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = threadIdx.x; t < (N >> 1); t += kRT) {
        const int i = 2 * t - (t & (j - 1));
        const int l = i + j;
        const unsigned long long x = a[i], y = a[l];
        const bool desc = (i & k) == 0;
        if (desc ? (x < y) : (x > y)) {
          a[i] = y;
          a[l] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Moves the nonzero entries of a[0..kRCap) to the front, in order, and zero-fills the
// rest; returns their count.  Each thread reads a run of entries that other threads
// wrote, so it starts with a barrier of its own.
__device__ __noinline__ int rcompact_nonzero(unsigned long long* a, unsigned long long* red) {
  // warp w reads its kRSeg entries striped over its lanes (entry w * kRSeg + 32 e + lane):
  // conflict-free shared loads, and (e, lane) order is the entries' order
  constexpr int per = kRSeg / 32;
  static_assert(per * 32 == kRSeg && kRSeg * kRW == kRCap, "striped segments");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  unsigned long long v[per];
  unsigned m[per];
  uint32_t wtot = 0;
  __syncthreads();
#pragma unroll
  for (int e = 0; e < per; ++e) {
    v[e] = a[warp * kRSeg + e * 32 + lane];
    m[e] = __ballot_sync(kFull, v[e] != 0ull);
    wtot += __popc(m[e]);
  }
  uint32_t tot;
  uint32_t pos = __shfl_sync(kFull, block_excl_scan_u32(lane == 0 ? wtot : 0u, &tot, red), 0);
#pragma unroll
  for (int e = 0; e < per; ++e) {
    if (v[e] != 0ull) a[pos + __popc(m[e] & lt)] = v[e];
    pos += __popc(m[e]);
  }
  __syncthreads();
  for (int i = static_cast<int>(tot) + static_cast<int>(threadIdx.x); i < kRCap; i += kRT) a[i] = 0ull;
  __syncthreads();
  return static_cast<int>(tot);
}

// A mass histogram of nb bins whose u64 weights (< 2^42) are split into three
// 14-bit limbs, one u32 array each: a bin takes up to 2^18 additions (any row of
// at most 262144 elements) without a limb overflowing.
struct RBins3 {
  uint32_t* base;
  int nb;
  __device__ __forceinline__ void clear() const {
    for (int i = threadIdx.x; i < 3 * nb; i += kRT) base[i] = 0u;
  }
  __device__ __forceinline__ void add(int b, unsigned long long w) const {
    sh_red_add(base + b, static_cast<uint32_t>(w & 0x3FFFu));
    sh_red_add(base + nb + b, static_cast<uint32_t>((w >> 14) & 0x3FFFu));
    sh_red_add(base + 2 * nb + b, static_cast<uint32_t>(w >> 28));
  }
  __device__ __forceinline__ unsigned long long get(int b) const {
    return static_cast<unsigned long long>(base[b]) + (static_cast<unsigned long long>(base[nb + b]) << 14) +
           (static_cast<unsigned long long>(base[2 * nb + b]) << 28);
  }
};
struct RBins1 {
  uint32_t* base;
  int nb;
  __device__ __forceinline__ void clear() const {
    for (int i = threadIdx.x; i < nb; i += kRT) base[i] = 0u;
  }
  __device__ __forceinline__ void add(int b, unsigned long long w) const {
    sh_red_add(base + b, static_cast<uint32_t>(w));
  }
  __device__ __forceinline__ unsigned long long get(int b) const { return base[b]; }
};

// ---- exact selection over the whole row (fallback) ---------------------------------------

// The element of the order (value desc, index asc) at which the cumulative weight
// first reaches need (1 <= need <= total): weight 1 (kMass false) or the fixed-point
// softmax mass against the row maximum M.  Four 8-bit digit passes over the keys,
// then, among equal keys, one scan in index order.  The row is re-read each pass.
template <bool kBF16, bool kMass>
__device__ __noinline__ Thresh rrow_select(const RowCtx& rc, unsigned long long need, float M, uint32_t* hist,
                                           unsigned long long* red, unsigned long long* misc) {
  constexpr int G = kBF16 ? 8 : 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long pol = l2_policy_normal();
  using H = typename std::conditional<kMass, RBins3, RBins1>::type;
  const H hb{hist, 256};
  uint32_t prefix = 0, pmask = 0;
  unsigned long long binw = 0;
  for (int d = 0; d < 4; ++d) {
    const int shift = 24 - 8 * d;
    hb.clear();
    __syncthreads();
    rrow_pass<kBF16>(rc, pol, [&](bool valid, float y, uint32_t key, int) {
      if (!valid || (key & pmask) != prefix) return;
      const unsigned long long w = kMass ? fixed_mass(softmax_weight(y, M)) : 1ull;
      if (w) hb.add(static_cast<int>((key >> shift) & 0xFFu), w);
    });
    __syncthreads();
    if (warp == 0) {
      unsigned long long b[8];
      unsigned long long sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        b[e] = hb.get(255 - 8 * lane - e);
        sum += b[e];
      }
      const unsigned long long inc = warp_incl_scan_u64(sum, lane);
      const unsigned m = __ballot_sync(kFull, inc >= need);
      if (m) {
        if (lane == __ffs(m) - 1) {
          unsigned long long acc = inc - sum;
          for (int e = 0; e < 8; ++e) {
            if (acc + b[e] >= need) {
              misc[kMSel0] = static_cast<unsigned long long>(255 - 8 * lane - e);
              misc[kMSel1] = need - acc;
              misc[kMSel2] = b[e];
              break;
            }
            acc += b[e];
          }
        }
      } else if (lane == 0) {  // need above the total: cannot happen for a valid need
        misc[kMSel0] = 0ull;
        misc[kMSel1] = 1ull;
        misc[kMSel2] = 1ull;
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(misc[kMSel0]) << shift;
    pmask |= 0xFFu << shift;
    need = misc[kMSel1];
    binw = misc[kMSel2];
    __syncthreads();
  }
  // equal keys: keep the nt smallest indices, nt = ceil(need / weight of one)
  const unsigned long long w1 = kMass ? fixed_mass(softmax_weight(kfloat(prefix), M)) : 1ull;
  const unsigned long long nt = w1 ? (need + w1 - 1) / w1 : 1ull;
  const unsigned long long ties = w1 ? binw / w1 : 1ull;
  if (nt >= ties) return Thresh{prefix, INT_MAX};
  int32_t* found = reinterpret_cast<int32_t*>(misc + kMFound);
  if (threadIdx.x == 0) *found = INT_MAX;
  __syncthreads();
  unsigned long long seen = 0;
  for (int base = rc.g0; base < rc.g1; base += kRT) {
    const int g = base + static_cast<int>(threadIdx.x);
    uint32_t cnt = 0, flags = 0;
    if (g < rc.g1) {
      float v[G];
      unpack16<kBF16>(ld_row16(rc.x + g, pol), v);
      const uint32_t bits = rseen_bits<G>(rc.bitmap, rc.pen_on, g);
#pragma unroll
      for (int e = 0; e < G; ++e)
        if (fkey(rtransform(v[e], (bits >> e) & 1u, rc.pen, rc.div, rc.identity)) == prefix) {
          flags |= 1u << e;
          ++cnt;
        }
    }
    uint32_t total;
    const uint32_t ex = block_excl_scan_u32(cnt, &total, red);
    if (cnt && seen + ex < nt && nt <= seen + ex + cnt) {
      unsigned long long s = seen + ex;
      for (int e = 0; e < G; ++e)
        if ((flags >> e) & 1u) {
          if (++s == nt) *found = g * G + e;
        }
    }
    seen += total;
    __syncthreads();
    if (*found != INT_MAX || seen >= nt) break;
  }
  const Thresh th{prefix, *found};
  __syncthreads();
  return th;
}

// ---- selection inside the buffer (order words; zero entries are empty slots) -------------

// Exact k-th largest of the nonzero order words of cw[0..n) (at least k of them):
// eight 8-bit digit rounds with warp-aggregated counts.  Order words are distinct,
// so the result is one entry.
__device__ __noinline__ Thresh rbuf_radix(const unsigned long long* cw, int n, uint32_t k, uint32_t* h,
                                          unsigned long long* misc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long prefix = 0, pmask = 0;
  for (int d = 0; d < 8; ++d) {
    const int shift = 56 - 8 * d;
    for (int i = threadIdx.x; i < 256; i += kRT) h[i] = 0u;
    __syncthreads();
    for (int base = 0; base < n; base += kRT) {
      const int i = base + static_cast<int>(threadIdx.x);
      const unsigned long long w = i < n ? cw[i] : 0ull;
      const bool take = w != 0ull && (w & pmask) == prefix;
      const int bin = take ? static_cast<int>((w >> shift) & 0xFFull) : -1;
      const unsigned peers = __match_any_sync(kFull, bin);
      if (take && lane == __ffs(peers) - 1) sh_red_add(&h[bin], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t b[8];
      uint32_t sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        b[e] = h[255 - 8 * lane - e];
        sum += b[e];
      }
      const uint32_t inc = warp_incl_scan_u32(sum, lane);
      const unsigned m = __ballot_sync(kFull, inc >= k);
      if (m) {
        if (lane == __ffs(m) - 1) {
          uint32_t acc = inc - sum;
          for (int e = 0; e < 8; ++e) {
            if (acc + b[e] >= k) {
              misc[kMSel0] = static_cast<unsigned long long>(255 - 8 * lane - e);
              misc[kMSel1] = k - acc;
              break;
            }
            acc += b[e];
          }
        }
      } else if (lane == 0) {
        misc[kMSel0] = 0ull;
        misc[kMSel1] = 1ull;
      }
    }
    __syncthreads();
    prefix |= misc[kMSel0] << shift;
    pmask |= 0xFFull << shift;
    k = static_cast<uint32_t>(misc[kMSel1]);
    __syncthreads();
  }
  return Thresh{static_cast<uint32_t>(prefix >> 32), static_cast<int32_t>(~static_cast<uint32_t>(prefix))};
}

// Linear bin of a key below the buffer maximum mx (bin 0 holds the largest keys).
__device__ __forceinline__ int rlin_bin(uint32_t key, uint32_t mx, float s) {
  const int b = static_cast<int>(__fmul_rn(static_cast<float>(mx - key), s));
  return b < kRLin ? b : kRLin - 1;
}

// Exact k-th entry (value desc, index asc) of the nonzero order words of cw[0..n)
// (at least k of them), whose keys lie in [mn, mx]: a count histogram over linear
// key bins finds the bin holding it and that bin's entries are ranked pairwise; a
// bin too large for that goes to the radix.
__device__ __noinline__ Thresh rbuf_kth(const unsigned long long* cw, int n, uint32_t k, uint32_t mx, uint32_t mn,
                                        uint32_t* hist, unsigned long long* wb, unsigned long long* red,
                                        unsigned long long* misc) {
  uint32_t& s_cnt = *reinterpret_cast<uint32_t*>(misc + kMCnt);
  if (mx != mn) {
    const float s = static_cast<float>(kRLin) / (static_cast<float>(mx - mn) + 1.0f);
    for (int i = threadIdx.x; i < kRLin; i += kRT) hist[i] = 0u;
    if (threadIdx.x == 0) {
      misc[kMBin] = ~0ull;
      misc[kMHit] = 0ull;
      s_cnt = 0u;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kRT) {
      const unsigned long long w = cw[i];
      if (w) sh_red_add(&hist[rlin_bin(static_cast<uint32_t>(w >> 32), mx, s)], 1u);
    }
    __syncthreads();
    constexpr int per = kRLin / kRT;
    uint32_t c[per];
    uint32_t sum = 0;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      c[e] = hist[per * threadIdx.x + e];
      sum += c[e];
    }
    uint32_t tot;
    const uint32_t ex = block_excl_scan_u32(sum, &tot, red);
    if (ex < k && ex + sum >= k) {
      uint32_t acc = ex;
#pragma unroll
      for (int e = 0; e < per; ++e) {
        if (acc < k && acc + c[e] >= k) {
          misc[kMBin] = static_cast<unsigned long long>(per * threadIdx.x + e);
          misc[kMAbove] = acc;
        }
        acc += c[e];
      }
    }
    __syncthreads();
    const unsigned long long beta = misc[kMBin];
    const uint32_t above = static_cast<uint32_t>(misc[kMAbove]);
    if (beta != ~0ull && hist[beta] <= static_cast<uint32_t>(kRRank)) {
      for (int i = threadIdx.x; i < n; i += kRT) {
        const unsigned long long w = cw[i];
        if (w && rlin_bin(static_cast<uint32_t>(w >> 32), mx, s) == static_cast<int>(beta))
          wb[atomicAdd(&s_cnt, 1u)] = w;
      }
      __syncthreads();
      const int m = static_cast<int>(s_cnt);
      const uint32_t want = k - above - 1;  // entries of the bin that come before the k-th
      for (int i = threadIdx.x; i < m; i += kRT) {
        const unsigned long long wi = wb[i];
        uint32_t r = 0;
        for (int j = 0; j < m; ++j) r += wb[j] > wi ? 1u : 0u;
        if (r == want) misc[kMHit] = wi;
      }
      __syncthreads();
      const unsigned long long w = misc[kMHit];
      __syncthreads();
      if (w != 0ull)
        return Thresh{static_cast<uint32_t>(w >> 32), static_cast<int32_t>(~static_cast<uint32_t>(w))};
    }
    __syncthreads();
  }
  return rbuf_radix(cw, n, k, hist, misc);
}

// Copies the nonzero entries of cw[0..n) kept by th to out[0..cap), in buffer order;
// returns their count, at most cap.  Positions come from one block-wide scan (a shared
// counter would serialise one atomic per warp and round).
__device__ __forceinline__ int rbuf_gather(const unsigned long long* cw, int n, Thresh th, unsigned long long* out,
                                           int cap, unsigned long long* red) {
  // warp w reads entries w * kRSeg + 32 e + lane (conflict-free; (e, lane) order is the
  // buffer order)
  constexpr int per = kRSeg / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  unsigned long long w[per];
  unsigned m[per];
  uint32_t wtot = 0;
#pragma unroll
  for (int e = 0; e < per; ++e) {
    const int i = warp * kRSeg + e * 32 + lane;
    w[e] = i < n ? cw[i] : 0ull;
    const bool keep = w[e] != 0ull && kept_by(static_cast<uint32_t>(w[e] >> 32),
                                              static_cast<int32_t>(~static_cast<uint32_t>(w[e])), th.key, th.idx);
    w[e] = keep ? w[e] : 0ull;
    m[e] = __ballot_sync(kFull, keep);
    wtot += __popc(m[e]);
  }
  uint32_t tot;
  uint32_t pos = __shfl_sync(kFull, block_excl_scan_u32(lane == 0 ? wtot : 0u, &tot, red), 0);
#pragma unroll
  for (int e = 0; e < per; ++e) {
    if (w[e] != 0ull) {
      const uint32_t q = pos + __popc(m[e] & lt);
      if (q < static_cast<uint32_t>(cap)) out[q] = w[e];
    }
    pos += __popc(m[e]);
  }
  __syncthreads();
  return static_cast<int>(tot) < cap ? static_cast<int>(tot) : cap;
}

// ---- the sample ----------------------------------------------------------------------------

// Keys of kRSamp transformed elements: 64 runs of 32 consecutive elements spread
// evenly over the row (V > kRKeepAllV), one load per run and lane issued together.
struct SampleLoads {
  float x[kRRuns / kRW];
  int idx[kRRuns / kRW];
};
template <bool kBF16>
__device__ __forceinline__ void rsample_fetch(const RowCtx& rc, SampleLoads* sl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int u = 0; u < kRRuns / kRW; ++u) {
    const int j = warp + u * kRW;
    sl->idx[u] = static_cast<int>(static_cast<int64_t>(j) * (rc.V - 32) / (kRRuns - 1)) + lane;
    if (kBF16) {
      const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(rc.x) + sl->idx[u]);
      sl->x[u] = __uint_as_float(static_cast<uint32_t>(b) << 16);
    } else {
      sl->x[u] = __ldg(reinterpret_cast<const float*>(rc.x) + sl->idx[u]);
    }
  }
}
// The sample's keys (the row's seen bits set), then a barrier.
__device__ __forceinline__ void rsample_finish(const RowCtx& rc, const SampleLoads& sl, uint32_t* samp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int u = 0; u < kRRuns / kRW; ++u) {
    const int j = warp + u * kRW;
    const bool seen = rc.pen_on && ((rc.bitmap[sl.idx[u] >> 5] >> (sl.idx[u] & 31)) & 1u);
    samp[j * 32 + lane] = fkey(rtransform(sl.x[u], seen, rc.pen, rc.div, rc.identity));
  }
  __syncthreads();
}
template <bool kBF16>
__device__ __forceinline__ void rsample_load(const RowCtx& rc, uint32_t* samp) {
  SampleLoads sl;
  rsample_fetch<kBF16>(rc, &sl);
  rsample_finish(rc, sl, samp);
}

// The r-th largest sample key, rounded down: at least r samples are >= it.  The digit
// rounds start below the bits every sample key shares (found from the smallest and largest
// key), so that the keys spread over the 2048 bins of the first round instead of meeting
// in a few (shared-memory adds to one word serialise); two 11-bit rounds of the offsets
// from the smallest key.
__device__ __noinline__ uint32_t rsample_rank(const uint32_t* samp, uint32_t r, uint32_t* h, unsigned long long* red,
                                              unsigned long long* misc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t mx = 0u, mn = 0xFFFFFFFFu;
  for (int i = threadIdx.x; i < kRSamp; i += kRT) {
    mx = samp[i] > mx ? samp[i] : mx;
    mn = samp[i] < mn ? samp[i] : mn;
  }
  mx = __reduce_max_sync(kFull, mx);
  mn = __reduce_min_sync(kFull, mn);
  if (lane == 0) red[warp] = (static_cast<unsigned long long>(mx) << 32) | mn;
  __syncthreads();
  {
    const unsigned long long v = red[lane & (kRW - 1)];
    mx = __reduce_max_sync(kFull, static_cast<uint32_t>(v >> 32));
    mn = __reduce_min_sync(kFull, static_cast<uint32_t>(v));
  }
  __syncthreads();  // red is reused by the scans below
  const uint32_t span = mx - mn;
  if (span == 0u) return mn;
  int top = 32 - __clz(span);  // offsets have this many bits
  uint32_t prefix = 0, pmask = 0, need = r;
  constexpr int per = 2048 / kRT;
  for (int d = 0; d < 2 && top > 0; ++d) {
    const int width = top < 11 ? top : 11;
    const int shift = top - width;
    const uint32_t dmask = (1u << width) - 1u;
    for (int i = threadIdx.x; i < 2048; i += kRT) h[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < kRSamp; i += kRT) {
      const uint32_t o = samp[i] - mn;
      if ((o & pmask) == prefix) sh_red_add(&h[(o >> shift) & dmask], 1u);
    }
    __syncthreads();
    uint32_t c[per];
    uint32_t sum = 0;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      c[e] = h[2047 - per * threadIdx.x - e];
      sum += c[e];
    }
    uint32_t tot;
    const uint32_t ex = block_excl_scan_u32(sum, &tot, red);
    if (ex < need && ex + sum >= need) {
      uint32_t acc = ex;
#pragma unroll
      for (int e = 0; e < per; ++e) {
        if (acc < need && acc + c[e] >= need) {
          misc[kMSel0] = static_cast<unsigned long long>(2047 - per * threadIdx.x - e);
          misc[kMSel1] = need - acc;
        }
        acc += c[e];
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(misc[kMSel0]) << shift;
    pmask |= dmask << shift;
    need = static_cast<uint32_t>(misc[kMSel1]);
    top = shift;
    __syncthreads();
  }
  return mn + prefix;
}

// ---- top-k rows ----------------------------------------------------------------------------

// The streaming pass: the -inf background of the filtered row, and every element whose
// penalised raw value is >= tau_raw (NaN: nothing passes) appended, as (raw key, index),
// to this warp's segment seg[0..kRSeg).  keep_all: NaN counts as -inf and everything
// passes.  Returns the warp's count (above kRSeg: the segment overflowed).
template <bool kBF16>
__device__ __forceinline__ uint32_t rk_stream(const RowCtx& rc, float tau_raw, bool keep_all, unsigned long long* seg,
                                              unsigned long long pol) {
  constexpr int G = kBF16 ? 8 : 4;
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const uint4* xr = rc.x;
  float* out = rc.out;
  const int g1 = rc.g1;  // this CTA's part of the row: [rc.g0, g1)
  const uint32_t* bitmap = rc.bitmap;
  const bool pen_on = rc.pen_on;
  const float pen = rc.pen;
  const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  uint32_t wcnt = 0;
  for (int base = rc.g0; base < g1; base += kRT * kRU) {
    uint4 w[kRU];
#pragma unroll
    for (int u = 0; u < kRU; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      w[u] = g < g1 ? ld_row16(xr + g, pol) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kRU; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      const bool in = g < g1;
      if (out != nullptr && in) {
        float4* o = reinterpret_cast<float4*>(out) + g * (G / 4);
#pragma unroll
        for (int h = 0; h < G / 4; ++h) __stcs(o + h, ninf);
      }
      float v[G];
      unpack16<kBF16>(w[u], v);
      if (keep_all) {
#pragma unroll
        for (int e = 0; e < G; ++e) v[e] = isnan(v[e]) ? -INFINITY : v[e];
      }
      const uint32_t bits = in ? rseen_bits<G>(bitmap, pen_on, g) : 0u;
      if (__any_sync(kFull, bits != 0u)) {
#pragma unroll
        for (int e = 0; e < G; ++e)
          if ((bits >> e) & 1u) v[e] = rpenal(v[e], pen);
      }
      bool pass[G];
      bool any = false;
#pragma unroll
      for (int e = 0; e < G; ++e) {
        pass[e] = in && v[e] >= tau_raw;
        any |= pass[e];
      }
      if (__any_sync(kFull, any)) {
#pragma unroll
        for (int e = 0; e < G; ++e) {
          const unsigned m = __ballot_sync(kFull, pass[e]);
          if (pass[e]) {
            const uint32_t pos = wcnt + __popc(m & lt);
            if (pos < static_cast<uint32_t>(kRSeg)) seg[pos] = order_word(fkey(v[e]), g * G + e);
          }
          wcnt += __popc(m);
        }
      }
    }
  }
  return wcnt;
}

// Turns the warp segments of raw candidates into a zero-padded array of exact keys
// (x / T) that are >= tau_key.  Returns their count; *top = the largest order word,
// *mn = the smallest key.
__device__ __noinline__ uint32_t rk_normalize(unsigned long long* cw, const uint32_t* segcnt, uint32_t tau_key,
                                              FixedDivisor dv, bool identity, unsigned long long* red,
                                              unsigned long long* top, uint32_t* mn) {
  unsigned long long cnt = 0, best = 0, nmn = 0;
  for (int i = threadIdx.x; i < kRCap; i += kRT) {
    const int w = i / kRSeg;
    unsigned long long wd = 0;
    if (i - w * kRSeg < static_cast<int>(segcnt[w])) {
      const unsigned long long r = cw[i];
      const float x = kfloat(static_cast<uint32_t>(r >> 32));
      const uint32_t key = fkey(__fadd_rn(identity ? x : rdiv(x, dv), 0.0f));
      if (key >= tau_key) {
        wd = (static_cast<unsigned long long>(key) << 32) | (r & 0xFFFFFFFFull);
        ++cnt;
        best = wd > best ? wd : best;
        const unsigned long long nk = static_cast<uint32_t>(~key);
        nmn = nk > nmn ? nk : nmn;
      }
    }
    cw[i] = wd;
  }
  rblock_sum_max2(cnt, best, nmn, red);
  *top = best;
  *mn = ~static_cast<uint32_t>(nmn);
  return static_cast<uint32_t>(cnt);
}

// Top-p target: ceil(p * S) clamped to [1, S].
__device__ __forceinline__ unsigned long long rtopp_target(float p, unsigned long long S) {
  return ceil_mul_p(p, S);
}

// Cut of a list sorted in descending order (kl[0..n), n <= kRSortMax): the number of
// leading entries kept by top-p, given the mass `above` of everything before the list
// and the target tq.  0 when the boundary is not in the list.
__device__ __noinline__ int rlist_topp_cut(const unsigned long long* kl, int n, float M, unsigned long long above,
                                           unsigned long long tq, unsigned long long* red, unsigned long long* misc) {
  constexpr int per = kRSortMax / kRT;
  unsigned long long w[per];
  unsigned long long sum = 0;
#pragma unroll
  for (int e = 0; e < per; ++e) {
    const int i = per * static_cast<int>(threadIdx.x) + e;
    w[e] = i < n ? fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(kl[i] >> 32)), M)) : 0ull;
    sum += w[e];
  }
  if (threadIdx.x == 0) misc[kMCut] = 0ull;
  unsigned long long total;
  const unsigned long long ex = rblock_excl_scan_u64(sum, &total, red);
  if (above < tq) {
    unsigned long long acc = above + ex;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      if (acc < tq && acc + w[e] >= tq) misc[kMCut] = static_cast<unsigned long long>(per * threadIdx.x + e + 1);
      acc += w[e];
    }
  }
  __syncthreads();
  const int L = static_cast<int>(misc[kMCut]);
  __syncthreads();
  return L;
}

// Top-p over the survivors kl[0..n) (1 < n <= 1024, maximum M): a fixed-point mass
// histogram over linear bins of [smallest value, M] finds the bin holding the boundary
// and that bin's entries are ranked pairwise; a large bin is sorted instead.  Returns
// the last kept entry.  scratch: 2 * kRRank + 1024 u64.
__device__ __noinline__ Thresh rk_topp(unsigned long long* kl, int n, float M, float p, uint32_t* hist,
                                       unsigned long long* scratch, unsigned long long* red,
                                       unsigned long long* misc) {
  uint32_t& s_cnt = *reinterpret_cast<uint32_t*>(misc + kMCnt);
  unsigned long long* mass = scratch + 2 * kRRank;
  unsigned long long part = 0, nmn = 0, dummy = 0;
  for (int i = threadIdx.x; i < n; i += kRT) {
    const uint32_t key = static_cast<uint32_t>(kl[i] >> 32);
    const unsigned long long m = fixed_mass(softmax_weight(kfloat(key), M));
    mass[i] = m;
    part += m;
    const unsigned long long nk = static_cast<uint32_t>(~key);
    nmn = nk > nmn ? nk : nmn;
  }
  const RBins3 hb{hist, kRSurvBins};
  hb.clear();
  if (threadIdx.x == 0) {
    misc[kMBin] = ~0ull;
    misc[kMHit] = 0ull;
    s_cnt = 0u;
  }
  rblock_sum_max2(part, nmn, dummy, red);
  const unsigned long long S = part;
  const unsigned long long tq = rtopp_target(p, S);
  const float lo = kfloat(~static_cast<uint32_t>(nmn));
  const float span = __fsub_rn(M, lo);
  const float s = (span > 0.0f && span < INFINITY) ? __fdiv_rn(static_cast<float>(kRSurvBins), span) : 0.0f;
  auto bin_of = [&](float y) -> int {
    if (!(s > 0.0f) || y == M) return 0;
    const float f = __fmul_rn(__fsub_rn(M, y), s);
    return f < static_cast<float>(kRSurvBins) ? static_cast<int>(f) : kRSurvBins - 1;
  };
  for (int i = threadIdx.x; i < n; i += kRT)
    if (mass[i]) hb.add(bin_of(kfloat(static_cast<uint32_t>(kl[i] >> 32))), mass[i]);
  __syncthreads();
  constexpr int per = kRSurvBins / kRT;
  unsigned long long c[per];
  unsigned long long sum = 0;
#pragma unroll
  for (int e = 0; e < per; ++e) {
    c[e] = hb.get(per * threadIdx.x + e);
    sum += c[e];
  }
  unsigned long long tot;
  const unsigned long long ex = rblock_excl_scan_u64(sum, &tot, red);
  if (ex < tq && ex + sum >= tq) {
    unsigned long long acc = ex;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      if (acc < tq && acc + c[e] >= tq) {
        misc[kMBin] = static_cast<unsigned long long>(per * threadIdx.x + e);
        misc[kMAbove] = acc;
      }
      acc += c[e];
    }
  }
  __syncthreads();
  const int beta = static_cast<int>(misc[kMBin]);
  const unsigned long long above = misc[kMAbove];
  if (misc[kMBin] != ~0ull) {
    unsigned long long* gw = scratch;           // the bin's order words
    unsigned long long* gm = scratch + kRRank;  // and masses
    for (int i = threadIdx.x; i < n; i += kRT) {
      if (mass[i] && bin_of(kfloat(static_cast<uint32_t>(kl[i] >> 32))) == beta) {
        const uint32_t pos = atomicAdd(&s_cnt, 1u);
        if (pos < static_cast<uint32_t>(kRRank)) {
          gw[pos] = kl[i];
          gm[pos] = mass[i];
        }
      }
    }
    __syncthreads();
    const int m = static_cast<int>(s_cnt);
    if (m <= kRRank) {
      for (int i = threadIdx.x; i < m; i += kRT) {
        const unsigned long long wi = gw[i];
        unsigned long long exm = above;
        for (int j = 0; j < m; ++j) exm += gw[j] > wi ? gm[j] : 0ull;
        if (exm < tq && tq <= exm + gm[i]) misc[kMHit] = wi;
      }
    }
    __syncthreads();
  }
  const unsigned long long hit = misc[kMHit];
  __syncthreads();
  if (hit != 0ull) return Thresh{static_cast<uint32_t>(hit >> 32), static_cast<int32_t>(~static_cast<uint32_t>(hit))};
  // large boundary bin: sort the survivors and cut the prefix
  int N = 1;
  while (N < n) N <<= 1;
  for (int i = n + static_cast<int>(threadIdx.x); i < N; i += kRT) kl[i] = 0ull;
  __syncthreads();
  rbitonic_desc(kl, N);
  const int L = rlist_topp_cut(kl, n, M, 0ull, tq, red, misc);
  const unsigned long long w = kl[(L > 0 ? L : n) - 1];
  return Thresh{static_cast<uint32_t>(w >> 32), static_cast<int32_t>(~static_cast<uint32_t>(w))};
}

// Race over the entries of kl[0..n) kept by th (best race word and the first of the
// order), writing their values to the filtered row.
__device__ __forceinline__ void rlist_race(const unsigned long long* kl, int n, Thresh th, float M, const RowCtx& rc,
                                           float eps, unsigned long long& rb, unsigned long long& first) {
  for (int i = threadIdx.x; i < n; i += kRT) {
    const unsigned long long w = kl[i];
    const uint32_t key = static_cast<uint32_t>(w >> 32);
    const int32_t idx = static_cast<int32_t>(~static_cast<uint32_t>(w));
    if (w == 0ull || !kept_by(key, idx, th.key, th.idx)) continue;
    first = w > first ? w : first;
    const float y = kfloat(key);
    if (rc.race) {
      const float r = __fdiv_rn(softmax_weight(y, M), __fadd_rn(rq1(rc, idx), eps));
      if (!isnan(r)) {
        const unsigned long long c = order_word(fkey(r), idx);
        rb = c > rb ? c : rb;
      }
    }
    if (rc.out) rc.out[idx] = y;
  }
}

struct RowSmem {
  uint32_t* bitmap;
  unsigned long long* cw;
  uint32_t* hist;
  unsigned long long* wbuf;
  unsigned long long* red;
  unsigned long long* misc;
};

constexpr Thresh kKeepAll{1u, -1};  // kept_by(any real key) holds; empty slots (key 0) fail

// Top-k and one-element rows; returns the chosen index.
// The CTAs that work on one row.  C == 1: this CTA alone (barriers are __syncthreads);
// C > 1: the C CTAs of the thread-block cluster, each on its own part of the row,
// exchanging partial results through distributed shared memory.
struct Team {
  int C;
  int rank;
  __device__ __forceinline__ void sync() const {
    if (C > 1) {
      cg::this_cluster().sync();
    } else {
      __syncthreads();
    }
  }
  // Pushes v (thread 0's copy) into slot q of every member; a sync() must follow
  // before the slots are read.
  __device__ __forceinline__ void push(unsigned long long* misc, int q, unsigned long long v) const {
    if (threadIdx.x != 0) return;
    unsigned long long* slot = misc + kMPush + kRMaxTeam * q + rank;
    if (C > 1) {
      cg::cluster_group cl = cg::this_cluster();
      for (int r = 0; r < C; ++r) *cl.map_shared_rank(slot, r) = v;
    } else {
      *slot = v;
    }
  }
  __device__ __forceinline__ unsigned long long get(const unsigned long long* misc, int q, int r) const {
    return misc[kMPush + kRMaxTeam * q + r];
  }
  __device__ __forceinline__ unsigned long long max_of(const unsigned long long* misc, int q) const {
    unsigned long long m = 0;
    for (int r = 0; r < C; ++r) m = get(misc, q, r) > m ? get(misc, q, r) : m;
    return m;
  }
  __device__ __forceinline__ unsigned long long sum_of(const unsigned long long* misc, int q) const {
    unsigned long long s = 0;
    for (int r = 0; r < C; ++r) s += get(misc, q, r);
    return s;
  }
  template <class T>
  __device__ __forceinline__ T* remote(T* p, int r) const {
    return C > 1 ? cg::this_cluster().map_shared_rank(p, r) : p;
  }
};

template <bool kBF16>
__device__ __noinline__ int32_t rk_row(const RowCtx& rc, const RowSmem& sm, const Team& tm, uint32_t keff, bool single,
                                       bool topp_on, float p, float eps, bool exact, bool sampled) {
  uint32_t& s_cnt = *reinterpret_cast<uint32_t*>(sm.misc + kMCnt);
  uint32_t* segcnt = reinterpret_cast<uint32_t*>(sm.misc + kMSeg);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool keep_all = rc.V <= kRKeepAllV && !exact;
  RowCtx whole = rc;  // the whole row (rc is this CTA's part when a team shares the row)
  whole.g0 = 0;
  whole.g1 = rc.nv;
  uint32_t tau_key = 0u;
  float tau_raw = -INFINITY;
  if (exact) {
    tau_raw = __int_as_float(0x7fffffff);  // nothing passes: the exact select below takes over
  } else if (!keep_all) {
    uint32_t* samp = reinterpret_cast<uint32_t*>(sm.wbuf);
    if (!sampled) rsample_load<kBF16>(rc, samp);
    // the streaming pass's first two rounds of loads, asked of L2 during the selection
    for (int o = static_cast<int>(threadIdx.x) * 128; o < 2 * kRT * kRU * 16 && o < (rc.g1 - rc.g0) * 16; o += kRT * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(rc.x + rc.g0) + o));
    const int64_t want = (5 * static_cast<int64_t>(keff)) / 2 + 512;
    int64_t r = (want * kRSamp + rc.V - 1) / rc.V + 1;
    if (r > kRSamp) r = kRSamp;
    tau_key = rsample_rank(samp, static_cast<uint32_t>(r), sm.hist, sm.red, sm.misc);
    const float tv = kfloat(tau_key);
    // a threshold at or below -inf would take the whole row: go to the exact select
    tau_raw = (tau_key > kKeyNegInf && !isnan(tv)) ? raw_floor(tv, rc.T, rc.identity) : __int_as_float(0x7fffffff);
  }
  const uint32_t wc = rk_stream<kBF16>(rc, tau_raw, keep_all, sm.cw + warp * kRSeg, l2_policy_first());
  if (lane == 0) segcnt[warp] = wc;
  __syncthreads();
  if (tm.C > 1) {
    // a team streamed the parts of one row against the same threshold (every member
    // samples the same elements): rank 0 appends the others' warp segments behind its own
    // (a segment that would overflow marks the buffer overflowed), then goes on alone
    tm.sync();
    if (tm.rank == 0) {
      uint32_t own = segcnt[warp];
      for (int r = 1; r < tm.C; ++r) {
        const uint32_t other = *tm.remote(segcnt + warp, r);
        const unsigned long long* src = tm.remote(sm.cw + warp * kRSeg, r);
        const bool fits = own <= static_cast<uint32_t>(kRSeg) && other <= static_cast<uint32_t>(kRSeg) &&
                          own + other <= static_cast<uint32_t>(kRSeg);
        if (fits)
          for (uint32_t i = lane; i < other; i += 32) sm.cw[warp * kRSeg + own + i] = src[i];
        own = fits ? own + other : static_cast<uint32_t>(kRSeg) + 1u;
      }
      __syncwarp();
      if (lane == 0) segcnt[warp] = own;
    }
    tm.sync();  // the other members' segments are read; they leave the row
    if (tm.rank != 0) return -1;
  }
  bool over = false;
#pragma unroll
  for (int w = 0; w < kRW; ++w) over |= segcnt[w] > static_cast<uint32_t>(kRSeg);
  unsigned long long top;
  uint32_t mn;
  uint32_t n = rk_normalize(sm.cw, segcnt, tau_key, rc.div, rc.identity, sm.red, &top, &mn);
  if (over || n < keff) {
    // the sample missed: exact k-th element over the row, then collect the k kept
    const Thresh th = rrow_select<kBF16, false>(whole, keff, 0.0f, sm.hist, sm.red, sm.misc);
    for (int i = threadIdx.x; i < kRCap; i += kRT) sm.cw[i] = 0ull;
    if (threadIdx.x == 0) s_cnt = 0u;
    __syncthreads();
    unsigned long long b0 = 0, b1 = 0;
    rrow_pass<kBF16>(whole, l2_policy_normal(), [&](bool valid, float, uint32_t key, int idx) {
      const bool keep = valid && kept_by(key, idx, th.key, th.idx);
      const uint32_t pos = rwarp_reserve(keep ? 1u : 0u, s_cnt);
      if (keep && pos < static_cast<uint32_t>(kRCap)) {
        const unsigned long long w = order_word(key, idx);
        sm.cw[pos] = w;
        b0 = w > b0 ? w : b0;
        const unsigned long long nk = static_cast<uint32_t>(~key);
        b1 = nk > b1 ? nk : b1;
      }
    });
    rblock_max2(b0, b1, sm.red);
    top = b0;
    mn = ~static_cast<uint32_t>(b1);
    n = keff;  // exactly keff elements are kept by th
  }
  const uint32_t mx = static_cast<uint32_t>(top >> 32);
  const float M = kfloat(mx);
  if (single) {
    const int32_t idx = static_cast<int32_t>(~static_cast<uint32_t>(top));
    if (threadIdx.x == 0 && rc.out) rc.out[idx] = M;
    return idx;
  }
  const Thresh tk = n > keff ? rbuf_kth(sm.cw, kRCap, keff, mx, mn, sm.hist, sm.wbuf, sm.red, sm.misc) : kKeepAll;
  const int ns = rbuf_gather(sm.cw, kRCap, tk, sm.wbuf, kTopKMax, sm.red);  // the k survivors
  Thresh th = kKeepAll;
  if (topp_on && ns > 1) th = rk_topp(sm.wbuf, ns, M, p, sm.hist, sm.cw, sm.red, sm.misc);
  unsigned long long rb = 0, first = 0;
  rlist_race(sm.wbuf, ns, th, M, rc, eps, rb, first);
  rblock_max2(rb, first, sm.red);
  const unsigned long long c = rb ? rb : first;
  return static_cast<int32_t>(~static_cast<uint32_t>(c));
}

// ---- rows shared by the CTAs of a cluster: top-p-only and keep-all rows -------------------


// The largest penalised raw value of this CTA's part of the row, as a key.
template <bool kBF16>
__device__ __noinline__ unsigned long long rrow_max_key(const RowCtx& rc, unsigned long long pol,
                                                        unsigned long long* red) {
  constexpr int G = kBF16 ? 8 : 4;
  constexpr uint32_t kNegInf = kBF16 ? 0xFF80FF80u : 0xFF800000u;  // -inf in every lane
  const uint4* xr = rc.x;
  const int g0 = rc.g0, g1 = rc.g1;
  const uint32_t* bitmap = rc.bitmap;
  const bool pen_on = rc.pen_on;
  const float pen = rc.pen;
  float xm = -INFINITY;
  for (int base = g0; base < g1; base += kRT * kRU) {
    uint4 w[kRU];
#pragma unroll
    for (int u = 0; u < kRU; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      w[u] = g < g1 ? ld_row16(xr + g, pol) : make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
    }
#pragma unroll
    for (int u = 0; u < kRU; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      float v[G];
      unpack16<kBF16>(w[u], v);
      const uint32_t bits = g < g1 ? rseen_bits<G>(bitmap, pen_on, g) : 0u;
      if (bits) {
#pragma unroll
        for (int e = 0; e < G; ++e)
          if ((bits >> e) & 1u) v[e] = rpenal(v[e], pen);
      }
#pragma unroll
      for (int e = 0; e < G; ++e) xm = fmaxf(xm, v[e]);  // NaN is ignored (it counts as -inf)
    }
  }
  unsigned long long k = fkey(xm), dummy = 0;
  rblock_max2(k, dummy, red);
  return k;
}
// The transformed maximum from the largest raw key (division by T > 0 is monotone).
__device__ __forceinline__ float rmax_transformed(unsigned long long kraw, const RowCtx& rc) {
  const float m = kfloat(static_cast<uint32_t>(kraw));
  return __fadd_rn(rc.identity ? m : rdiv(m, rc.div), 0.0f);
}

// This CTA's part of the row with a known kept threshold: race over the kept elements
// and write every element of the part (kept: its value, else -inf).  *rb, *first: the
// block's best race word and first kept order word.
template <bool kBF16>
__device__ __noinline__ void rrow_race_write(const RowCtx& rc, Thresh th, float M, float eps, unsigned long long pol,
                                             unsigned long long* red, unsigned long long* rb_out,
                                             unsigned long long* first_out) {
  constexpr int G = kBF16 ? 8 : 4;
  unsigned long long rb = 0, first = 0;
  for (int g = rc.g0 + static_cast<int>(threadIdx.x); g < rc.g1; g += kRT) {
    float v[G];
    unpack16<kBF16>(ld_row16(rc.x + g, pol), v);
    const uint32_t bits = rseen_bits<G>(rc.bitmap, rc.pen_on, g);
    float qv[G];
    if (rc.race) {
#pragma unroll
      for (int h = 0; h < G / 4; ++h) {
        const float4 t = rq4(rc, g * (G / 4) + h);
        qv[4 * h] = t.x; qv[4 * h + 1] = t.y; qv[4 * h + 2] = t.z; qv[4 * h + 3] = t.w;
      }
    }
    float o[G];
#pragma unroll
    for (int e = 0; e < G; ++e) {
      const float y = rtransform(v[e], (bits >> e) & 1u, rc.pen, rc.div, rc.identity);
      const uint32_t key = fkey(y);
      const int idx = g * G + e;
      const bool kept = kept_by(key, idx, th.key, th.idx);
      o[e] = kept ? y : -INFINITY;
      if (kept) {
        const unsigned long long ow = order_word(key, idx);
        first = ow > first ? ow : first;
        if (rc.race) {
          const float r = __fdiv_rn(softmax_weight(y, M), __fadd_rn(qv[e], eps));
          if (!isnan(r)) {
            const unsigned long long c = order_word(fkey(r), idx);
            rb = c > rb ? c : rb;
          }
        }
      }
    }
    if (rc.out) {
      float4* op = reinterpret_cast<float4*>(rc.out) + g * (G / 4);
#pragma unroll
      for (int h = 0; h < G / 4; ++h) __stcs(op + h, make_float4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]));
    }
  }
  rblock_max2(rb, first, red);
  *rb_out = rb;
  *first_out = first;
}

// Index of the first element (lowest index) whose transformed value equals M: the first
// of the order, which every kept set holds.  Re-reads the whole row (rc covers it).
template <bool kBF16>
__device__ __noinline__ int32_t rrow_first_max(const RowCtx& rc, float M, unsigned long long* red) {
  const uint32_t km = fkey(M);
  unsigned long long best = 0, dummy = 0;
  rrow_pass<kBF16>(rc, l2_policy_normal(), [&](bool valid, float, uint32_t key, int idx) {
    if (valid && key == km) {
      const unsigned long long w = static_cast<uint32_t>(~static_cast<uint32_t>(idx));
      best = w > best ? w : best;
    }
  });
  rblock_max2(best, dummy, red);
  return static_cast<int32_t>(~static_cast<uint32_t>(best));
}

// ---- top-p-only rows: pass A (histogram), pass B (race, write, band) -------------------

constexpr int kRPBins = 2048;           // mass bins of top-p-only rows: width 1/32 below H
constexpr float kRPScale = 32.0f;
static_assert(kRPBins == kExpBins, "one bin factor per mass bin");

// The reference H of a top-p-only row lies on the 1/32 grid (rounded up) with |H| < 2^18,
// so every bin top H - b/32 (b < 2048) is a float exactly.  Rows whose H cannot (an
// infinite or huge maximum) take the exact whole-row selection.
__device__ __forceinline__ float pgrid_up(float h) {
  return __fmul_rn(ceilf(__fmul_rn(h, kRPScale)), 1.0f / kRPScale);
}
__device__ __forceinline__ bool pgrid_ok(float h) { return fabsf(h) < 262144.0f; }  // false for NaN, inf

// The weight of y against the reference H (on the grid, H >= y): its bin
// b = floor(32 (H - y)) of the exact difference, i.e. H - (b + 1)/32 < y <= H - b/32
// (kRPBins when b is not in [0, 2048): no mass), and the weight relative to the bin top
// c = H - b/32 (exact), exp(-(c - y)) as an integer w24 in units of 2^-24 (w24_weight;
// c - y is exact to 2^-30, so the error is the exponential's).  The mass of an element is
// w24 * 2^-24 * exp(-b/32) against exp(H), with exp(-b/32) from the table kExpBin; every
// total, prefix and race below is taken in this one arithmetic, so they agree with each
// other exactly.  The bin is first taken from the rounded difference fl(H - y), which may
// lie across a bin edge from the exact one; comparing y with the exact bin edges then
// moves it to the bin of the exact difference, so bins order the elements exactly and pass
// B can classify them by comparing y with the same edges.
struct PW {
  int b;
  uint32_t w24;
  float wf;    // w24 as a float (exact)
  float frac;  // c - y, in [0, 1/32) up to the rounding of H - y: the position inside the bin
};
__device__ __forceinline__ PW pweight(float y, float H) {
  const float d = __fsub_rn(H, y);
  const float t = __fmaf_rd(d, kRPScale, 8388608.0f);  // floor(32 d) + 2^23 (exact product)
  uint32_t bu = __float_as_uint(t) - 0x4B000000u;
  float c = __fmaf_rn(__fsub_rn(t, 8388608.0f), -1.0f / kRPScale, H);  // H - b/32, exact
  // to the bin of the exact difference (c and c -+ 1/32 are exact; one step suffices, as
  // fl(H - y) is within 2^-19 of H - y below the last bin edge)
  if (y > c) {
    c = __fadd_rn(c, 1.0f / kRPScale);
    --bu;
  } else if (y <= __fsub_rn(c, 1.0f / kRPScale)) {
    c = __fsub_rn(c, 1.0f / kRPScale);
    ++bu;
  }
  const float frac = __fsub_rn(c, y);
  const float v = w24_weight(frac);  // an integer in [2^23, 2^24)
  PW r;
  r.b = bu < static_cast<uint32_t>(kRPBins) ? static_cast<int>(bu) : kRPBins;
  r.w24 = __float_as_uint(v) - 0x4A800000u;
  r.wf = v;
  r.frac = frac;
  return r;
}

constexpr int kRPSub = 1024;  // sub-bins of the boundary bin (by position inside it)

// Sub-bin of an element of the boundary bin: non-decreasing in H - y.
__device__ __forceinline__ int psub(const PW& w) {
  return rfloor_small(fminf(fmaxf(__fmul_rn(w.frac, kRPScale * kRPSub), 0.0f), static_cast<float>(kRPSub - 1)));
}

// Race quotient of an element of a top-p-only row before its bin factor: its weight
// w24 / (q + eps) (by the approximate reciprocal), as a key that is 0 for NaN or a negative
// quotient and otherwise orders like the quotient.  The full quotient is this times
// 2^-24 exp(-b/32), rounded once more, so the best of a bin is the bin's best key.
__device__ __forceinline__ uint32_t prace_key(float wf, float q, float eps) {
  const float u = __fmul_rn(wf, rrcp_approx(__fadd_rn(q, eps)));
  return u >= 0.0f ? (__float_as_uint(u) & 0x7FFFFFFFu) + 1u : 0u;
}
__device__ __forceinline__ float prace_value(uint32_t key, float f24) {
  return __fmul_rn(__uint_as_float(key - 1u), f24);
}

// The largest of a shared 64-bit word and w, kept in the word (a shared-window address);
// the key in its high half is read first, so the common case, an element that does not
// beat its bin's best, is one load and one compare.
__device__ __forceinline__ void sh_max_word(uint32_t a, uint32_t key, unsigned long long w) {
  uint32_t hi;
  asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(hi) : "r"(a + 4u));
  if (key >= hi) asm volatile("red.shared.max.u64 [%0], %1;" ::"r"(a), "l"(w) : "memory");
}

// Pass A of top-p-only rows over this CTA's part: the exact transformed values, binned
// against H with their 24-bit weights summed per bin in two 12/13-bit limbs
// (h[b], h[kRPBins + b]: a bin takes any row of at most 2^18 elements without overflow),
// and per bin the best race word (race key, index; the lower index on equal keys) in
// ub[b].  Returns the part's largest value as a key.
// kDraw: 0 q loaded, 1 q generated, 2 sampling off (the per-bin word is then the bin's
// first element of the order: its value key and index).
template <bool kBF16, int kDraw>
__device__ __noinline__ unsigned long long rp_pass_a_t(const RowCtx& rc, float H, float eps, uint32_t* h,
                                                       unsigned long long* ub, unsigned long long* red) {
  constexpr int G = kBF16 ? 8 : 4;
  constexpr int kUA = kBF16 ? 1 : 2;  // vectors in flight per thread (q rides along)
  const unsigned long long pol = l2_policy_last();
  const uint4* xr = rc.x;
  constexpr bool kGen = kDraw == 1;
  const bool race = kDraw != 2;
  const float4* qr = reinterpret_cast<const float4*>(rc.q);
  const unsigned long long seed = rc.seed, step = rc.step;
  const int64_t row = rc.row;
  const int g0 = rc.g0, g1 = rc.g1;
  const uint32_t* bitmap = rc.bitmap;
  const bool pen_on = rc.pen_on, identity = rc.identity;
  const float pen = rc.pen;
  const FixedDivisor dv = rc.div;
  for (int i = threadIdx.x; i < 2 * kRPBins; i += kRT) h[i] = 0u;
  for (int i = threadIdx.x; i < kRPBins; i += kRT) ub[i] = 0ull;
  __syncthreads();
  float ymax = -INFINITY;
  for (int base = g0; base < g1; base += kRT * kUA) {
    uint4 w[kUA];
    float4 qv[kUA][G / 4];
#pragma unroll
    for (int u = 0; u < kUA; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      w[u] = g < g1 ? ld_row16(xr + g, pol) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int hh = 0; hh < G / 4; ++hh)
        qv[u][hh] = (race && g < g1)
                        ? (kGen ? gen_q4(seed, step, row, g * (G / 4) + hh) : __ldcs(qr + g * (G / 4) + hh))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kUA; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      if (g >= g1) continue;
      float v[G];
      unpack16<kBF16>(w[u], v);
      const uint32_t bits = rseen_bits<G>(bitmap, pen_on, g);
      if (bits) {
#pragma unroll
        for (int e = 0; e < G; ++e)
          if ((bits >> e) & 1u) v[e] = rpenal(v[e], pen);
      }
#pragma unroll
      for (int e = 0; e < G; ++e) {
        // a NaN logit stays NaN here: it has no bin, no race and no part in the maximum,
        // exactly as the -inf it stands for
        const float y = __fadd_rn(identity ? v[e] : rdiv(v[e], dv), 0.0f);
        ymax = fmaxf(ymax, y);
        const PW pw = pweight(y, H);
        if (pw.b < kRPBins) {
          sh_red_add(&h[pw.b], pw.w24 & 0xFFFu);
          sh_red_add(&h[kRPBins + pw.b], pw.w24 >> 12);
          const float4 q4 = qv[u][e / 4];
          const float qe = (e & 3) == 0 ? q4.x : (e & 3) == 1 ? q4.y : (e & 3) == 2 ? q4.z : q4.w;
          const uint32_t key = kDraw == 2 ? fkey(y) : prace_key(pw.wf, qe, eps);
          sh_max_word(smem_u32(ub + pw.b), key, order_word(key, g * G + e));
        }
      }
    }
  }
  unsigned long long kmax = fkey(__fadd_rn(ymax, 0.0f)), dummy = 0;
  rblock_max2(kmax, dummy, red);
  return kmax;
}

// Pass A with q loaded or generated (one instantiation each, so neither pays for the other).
template <bool kBF16>
__device__ __forceinline__ unsigned long long rp_pass_a(const RowCtx& rc, float H, float eps, uint32_t* h,
                                                        unsigned long long* ub, unsigned long long* red) {
  return rc.gen ? rp_pass_a_t<kBF16, 1>(rc, H, eps, h, ub, red)
                : rc.race ? rp_pass_a_t<kBF16, 0>(rc, H, eps, h, ub, red) : rp_pass_a_t<kBF16, 2>(rc, H, eps, h, ub, red);
}

// Pass B of top-p-only rows over this CTA's part, once the boundary bin bstar is known:
// an element in a bin above it (H - y < bstar / 32) is kept and written; one of bin
// bstar goes to its warp's segment of cw (its key and index); the rest is written as
// -inf.  The race over the kept bins is already decided by pass A's per-bin words.
// Returns the warp's segment count.
template <bool kBF16>
__device__ __noinline__ uint32_t rp_pass_b(const RowCtx& rc, float H, int bstar, unsigned long long* cw) {
  constexpr int G = kBF16 ? 8 : 4;
  constexpr int kUB = kBF16 ? 2 : 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  unsigned long long* seg = cw + warp * kRSeg;
  const unsigned long long pol = l2_policy_first();
  const uint4* xr = rc.x;
  float* out = rc.out;
  const int g0 = rc.g0, g1 = rc.g1;
  const uint32_t* bitmap = rc.bitmap;
  const bool pen_on = rc.pen_on, identity = rc.identity;
  const float pen = rc.pen;
  const FixedDivisor dv = rc.div;
  // bin b holds H - (b + 1)/32 < y <= H - b/32 (pweight), so y is kept (b < bstar) exactly
  // when y > H - bstar/32 and in the band (b = bstar) when not kept and y > H - (bstar + 1)/32
  // (both edges exact floats)
  const float ykeep = __fmaf_rn(static_cast<float>(bstar), -1.0f / kRPScale, H);
  const float yband = bstar < kRPBins ? __fmaf_rn(static_cast<float>(bstar + 1), -1.0f / kRPScale, H) : ykeep;
  uint32_t wcnt = 0;
  for (int base = g0; base < g1; base += kRT * kUB) {
    uint4 w[kUB];
#pragma unroll
    for (int u = 0; u < kUB; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      w[u] = g < g1 ? ld_row16(xr + g, pol) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUB; ++u) {
      const int g = base + u * kRT + static_cast<int>(threadIdx.x);
      const bool in = g < g1;
      float v[G];
      unpack16<kBF16>(w[u], v);
      const uint32_t bits = in ? rseen_bits<G>(bitmap, pen_on, g) : 0u;
      if (__any_sync(kFull, bits != 0u)) {
#pragma unroll
        for (int e = 0; e < G; ++e)
          if ((bits >> e) & 1u) v[e] = rpenal(v[e], pen);
      }
      uint32_t kmask = 0, bmask = 0;
#pragma unroll
      for (int e = 0; e < G; ++e) {
        v[e] = __fadd_rn(identity ? v[e] : rdiv(v[e], dv), 0.0f);  // NaN: neither kept nor in the band
        kmask |= (in && v[e] > ykeep ? 1u : 0u) << e;
        bmask |= (in && v[e] <= ykeep && v[e] > yband ? 1u : 0u) << e;
      }
      if (__any_sync(kFull, bmask != 0u)) {
#pragma unroll
        for (int e = 0; e < G; ++e) {
          const bool take = (bmask >> e) & 1u;
          const unsigned m = __ballot_sync(kFull, take);
          if (take) {
            const uint32_t pos = wcnt + __popc(m & lt);
            if (pos < static_cast<uint32_t>(kRSeg)) seg[pos] = order_word(fkey(v[e]), g * G + e);
          }
          wcnt += __popc(m);
        }
      }
      if (in && out) {
        float4* op = reinterpret_cast<float4*>(out) + g * (G / 4);
#pragma unroll
        for (int hh = 0; hh < G / 4; ++hh) {
          float o[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) o[t] = ((kmask >> (4 * hh + t)) & 1u) ? v[4 * hh + t] : -INFINITY;
          __stcs(op + hh, make_float4(o[0], o[1], o[2], o[3]));
        }
      }
    }
  }
  return wcnt;
}

// ---- the pre-pass record of a top-p-only row --------------------------------------------
//
// With a workspace large enough, pass A of the top-p-only rows runs before the row kernel
// in a kernel of its own (kps_prepass_kernel) that spreads every such row over many CTAs.
// They merge their bin sums and per-bin race words into the row's record with global
// atomics; the row kernel reads the record instead of running pass A, and zeroes it for
// the next launch.
constexpr size_t kPRecBytes = 32896;  // sums u64[2048], race words u64[2048], M, H, padding
constexpr int kPreMaxChunks = 8;      // CTAs of the pre-pass per row, at most (measured: 8 beat 13-16 at B=256)

struct PRec {
  unsigned long long* sums;  // per bin: the sum of w24 over the row
  unsigned long long* ub;    // per bin: the best race word
  unsigned long long* M;     // the row's largest value as a key
  uint32_t* H;               // the reference H (float bits)
};
__device__ __forceinline__ PRec prec_at(const Params& P, int j) {
  unsigned char* b = P.pre + static_cast<size_t>(j) * kPRecBytes;
  return PRec{reinterpret_cast<unsigned long long*>(b), reinterpret_cast<unsigned long long*>(b + 16384),
              reinterpret_cast<unsigned long long*>(b + 32768), reinterpret_cast<uint32_t*>(b + 32776)};
}

// Rows whose pass A the pre-pass takes: top-p-only rows of a row past the keep-all size,
// outside exact mode.  Every kernel agrees on it.
__device__ __forceinline__ bool row_prepass(const Params& P, int64_t r) {
  if (P.exact || P.V <= kRKeepAllV || row_is_kmode(P, r)) return false;
  const float p = P.top_p[r];
  return !isnan(p) && p < 1.0f;
}

// Rows r' < r with row_prepass (the ordinal of row r among them); block-wide.
__device__ int prepass_ordinal(const Params& P, int64_t r, unsigned long long* red) {
  unsigned long long c = 0;
  for (int64_t i = threadIdx.x; i < r; i += kRT) c += row_prepass(P, i) ? 1ull : 0ull;
  return static_cast<int>(rblock_sum_u64(c, red));
}

// The zeroed state every record is left in: this member's share of it (members split the
// bins; rank 0 takes M and H).
__device__ __forceinline__ void prec_clear(const PRec& rec, const Team& tm) {
  const int b0 = kRPBins * tm.rank / tm.C, b1 = kRPBins * (tm.rank + 1) / tm.C;
  for (int b = b0 + static_cast<int>(threadIdx.x); b < b1; b += kRT) {
    rec.sums[b] = 0ull;
    rec.ub[b] = 0ull;
  }
  if (tm.rank == 0 && threadIdx.x == 0) {
    *rec.M = 0ull;
    *rec.H = 0u;
  }
}

// Top-p-only (topp true) and keep-all rows, shared by the CTAs of team tm; rc covers this
// CTA's part.  Returns the chosen index on the team's rank 0 (-1 elsewhere).
template <bool kBF16>
__device__ __noinline__ int32_t rwide_row(const RowCtx& rc, const RowSmem& sm, const Team& tm, bool topp, float p,
                                          float eps, bool exact, const PRec* rec) {
  uint32_t* segcnt = reinterpret_cast<uint32_t*>(sm.misc + kMSeg);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  RowCtx whole = rc;
  whole.g0 = 0;
  whole.g1 = rc.nv;
  // the exact whole-row selection, by rank 0 alone (the other members leave the row)
  auto exact_row = [&]() -> int32_t {
    const float M = rmax_transformed(rrow_max_key<kBF16>(whole, l2_policy_last(), sm.red), whole);
    Thresh th{0u, INT_MAX};
    if (topp) {
      unsigned long long part = 0;
      rrow_pass<kBF16>(whole, l2_policy_normal(), [&](bool valid, float y, uint32_t, int) {
        if (valid) part += fixed_mass(softmax_weight(y, M));
      });
      const unsigned long long tq = rtopp_target(p, rblock_sum_u64(part, sm.red));
      th = rrow_select<kBF16, true>(whole, tq, M, sm.hist, sm.red, sm.misc);
    }
    unsigned long long rb, first;
    rrow_race_write<kBF16>(whole, th, M, eps, l2_policy_normal(), sm.red, &rb, &first);
    return static_cast<int32_t>(~static_cast<uint32_t>(rb ? rb : first));
  };
  if (exact) return tm.rank == 0 ? exact_row() : -1;
  if (!topp) {
    // keep-all: the maximum, then the race and the write of every part
    tm.push(sm.misc, 0, rrow_max_key<kBF16>(rc, l2_policy_last(), sm.red));
    tm.sync();
    const float M = rmax_transformed(tm.max_of(sm.misc, 0), rc);
    unsigned long long rb, first;
    rrow_race_write<kBF16>(rc, Thresh{0u, INT_MAX}, M, eps, l2_policy_first(), sm.red, &rb, &first);
    tm.push(sm.misc, 1, rb);
    tm.push(sm.misc, 2, first);
    tm.sync();
    const unsigned long long c = tm.max_of(sm.misc, 1) ? tm.max_of(sm.misc, 1) : tm.max_of(sm.misc, 2);
    tm.sync();  // nobody reuses the slots before every member has read them
    return tm.rank == 0 ? static_cast<int32_t>(~static_cast<uint32_t>(c)) : -1;
  }

  // reference H: the sample maximum + headroom (every member samples the same elements),
  // or the pre-pass's, with its pass A
  float H, Mr = 0.0f;
  bool from_rec = false;  // bins and race words come from the pre-pass record
  if (rec) {
    // the pre-pass runs as the prerequisite grid of this launch: wait for its records
    asm volatile("griddepcontrol.wait;" ::: "memory");
    H = __uint_as_float(__ldcg(rec->H));
    Mr = kfloat(static_cast<uint32_t>(__ldcg(rec->M)));
    tm.sync();  // every member has read H and M before the record is cleared
    if (!pgrid_ok(H) || Mr > H) {
      // no pass A in the record, or the sample missed the top of the row: clear it and
      // go on as without one
      prec_clear(*rec, tm);
      if (!pgrid_ok(H)) return tm.rank == 0 ? exact_row() : -1;
      H = pgrid_up(Mr);
      if (!pgrid_ok(H)) return tm.rank == 0 ? exact_row() : -1;
      rec = nullptr;
    } else {
      from_rec = true;
    }
  } else {
    if (rc.V > kRKeepAllV) {
      uint32_t* samp = reinterpret_cast<uint32_t*>(sm.wbuf);
      rsample_load<kBF16>(whole, samp);
      unsigned long long a = 0, b = 0;
      for (int i = threadIdx.x; i < kRSamp; i += kRT) a = samp[i] > a ? samp[i] : a;
      rblock_max2(a, b, sm.red);
      H = __fadd_rn(kfloat(static_cast<uint32_t>(a)), kRHeadroom);
    } else {
      tm.push(sm.misc, 0, rrow_max_key<kBF16>(rc, l2_policy_last(), sm.red));
      tm.sync();
      H = rmax_transformed(tm.max_of(sm.misc, 0), rc);
    }
    H = pgrid_up(H);
    if (!pgrid_ok(H)) return tm.rank == 0 ? exact_row() : -1;  // the same decision in every member
  }
  float M;
  if (from_rec) {
    M = Mr;
  } else {
    // pass A; again with H = M when the sample missed the top of the row by more than the headroom
    tm.push(sm.misc, 1, rp_pass_a<kBF16>(rc, H, eps, sm.hist, sm.cw, sm.red));
    tm.sync();
    M = kfloat(static_cast<uint32_t>(tm.max_of(sm.misc, 1)));
    if (M > H) {
      H = pgrid_up(M);
      tm.sync();  // every member has read slot 1 and is done with the sample
      if (!pgrid_ok(H)) return tm.rank == 0 ? exact_row() : -1;
      tm.push(sm.misc, 1, rp_pass_a<kBF16>(rc, H, eps, sm.hist, sm.cw, sm.red));
      tm.sync();
    }
  }
  // bin factors exp(-b/32), the bin masses summed over the members, their total S, and
  // the bin bstar holding the boundary (its prefix reaches p * S)
  float* ftab = reinterpret_cast<float*>(sm.wbuf);
  for (int b = threadIdx.x; b < kRPBins; b += kRT) ftab[b] = kExpBin.v[b];
  double above = 0.0, tq = 0.0;
  int bstar;
  unsigned long long ubest[kRPBins / kRT];  // the best race word of each of this thread's bins
  {
    constexpr int per = kRPBins / kRT;
    double m[per];
    double sum = 0.0;
    // this thread's bins, every load of a source issued before any is used
    const int b0 = per * static_cast<int>(threadIdx.x);
    unsigned long long cb[per];
    float fb[per];
#pragma unroll
    for (int e = 0; e < per; ++e) fb[e] = kExpBin.v[b0 + e];
    if (from_rec) {
#pragma unroll
      for (int e = 0; e < per; ++e) {
        cb[e] = __ldcg(rec->sums + b0 + e);
        ubest[e] = __ldcg(rec->ub + b0 + e);
      }
    } else {
#pragma unroll
      for (int e = 0; e < per; ++e) {
        cb[e] = 0ull;
        ubest[e] = 0ull;
      }
      for (int r = 0; r < tm.C; ++r) {
        const uint32_t* hr = tm.remote(sm.hist, r);
        const unsigned long long* ur = tm.remote(sm.cw, r);
        uint32_t lo[per], hi[per];
        unsigned long long x[per];
#pragma unroll
        for (int e = 0; e < per; ++e) {
          lo[e] = hr[b0 + e];
          hi[e] = hr[kRPBins + b0 + e];
          x[e] = ur[b0 + e];
        }
#pragma unroll
        for (int e = 0; e < per; ++e) {
          cb[e] += static_cast<unsigned long long>(lo[e]) + (static_cast<unsigned long long>(hi[e]) << 12);
          ubest[e] = x[e] > ubest[e] ? x[e] : ubest[e];
        }
      }
    }
#pragma unroll
    for (int e = 0; e < per; ++e) {
      m[e] = static_cast<double>(cb[e]) * 5.9604644775390625e-8 * static_cast<double>(fb[e]);
      sum += m[e];
    }
    if (threadIdx.x == 0) sm.misc[kMBin] = static_cast<unsigned long long>(kRPBins);
    const int lane2 = threadIdx.x & 31, warp2 = threadIdx.x >> 5;
    double x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(kFull, x, o);
      if (lane2 >= o) x += y;
    }
    double* redd = reinterpret_cast<double*>(sm.red);
    if (lane2 == 31) redd[warp2] = x;
    __syncthreads();
    if (warp2 == 0) {
      const double sv = lane2 < kRW ? redd[lane2] : 0.0;
      double t = sv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(kFull, t, o);
        if (lane2 >= o) t += y;
      }
      if (lane2 < kRW) redd[kRW + lane2] = t - sv;
      if (lane2 == kRW - 1) redd[48] = t;
    }
    __syncthreads();
    const double S = redd[48];
    tq = static_cast<double>(p) * S;
    double acc = redd[kRW + warp2] + x - sum;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      const int b = per * static_cast<int>(threadIdx.x) + e;
      const double after = acc + m[e];
      if (acc < tq && after >= tq) {
        sm.misc[kMBin] = static_cast<unsigned long long>(b);
        reinterpret_cast<double*>(sm.misc)[kMAbove] = acc;
      }
      acc = after;
    }
    __syncthreads();
    bstar = static_cast<int>(sm.misc[kMBin]);
    above = reinterpret_cast<const double*>(sm.misc)[kMAbove];
  }
  // the race over the bins above the boundary bin (rank 0): each bin's best key scaled by
  // the bin's factor, with the index of its element
  unsigned long long rb = 0;
  if (tm.rank == 0) {
#pragma unroll
    for (int e = 0; e < kRPBins / kRT; ++e) {
      const int b = (kRPBins / kRT) * static_cast<int>(threadIdx.x) + e;
      if (b < bstar && ubest[e]) {
        unsigned long long c = ubest[e];  // sampling off: already the bin's first element of the order
        if (rc.race) {
          const float rv = prace_value(static_cast<uint32_t>(ubest[e] >> 32), __fmul_rn(ftab[b], 5.9604644775390625e-8f));
          c = order_word(fkey(rv), static_cast<int32_t>(~static_cast<uint32_t>(ubest[e])));
        }
        rb = c > rb ? c : rb;
      }
    }
    unsigned long long dummy = 0;
    rblock_max2(rb, dummy, sm.red);
  }
  tm.sync();  // every member is done reading the histograms, the per-bin words and the slots
  if (from_rec) prec_clear(*rec, tm);

  // pass B over this CTA's part
  const uint32_t wcnt = rp_pass_b<kBF16>(rc, H, bstar, sm.cw);
  if (lane == 0) segcnt[warp] = wcnt;
  __syncthreads();
  bool over = false;
#pragma unroll
  for (int w = 0; w < kRW; ++w) over |= segcnt[w] > static_cast<uint32_t>(kRSeg);
  for (int i = threadIdx.x; i < kRCap; i += kRT) {  // empty slots of every segment become zero
    const int w = i / kRSeg;
    if (i - w * kRSeg >= static_cast<int>(segcnt[w])) sm.cw[i] = 0ull;
  }
  const int nb = over ? kRCap + 1 : rcompact_nonzero(sm.cw, sm.red);
  tm.push(sm.misc, 6, static_cast<unsigned long long>(nb));
  tm.sync();
  int total = 0;
  bool fits = bstar < kRPBins;
  for (int r = 0; r < tm.C; ++r) {
    const int n = static_cast<int>(tm.get(sm.misc, 6, r));
    fits = fits && n <= kRCap;
    total += n;
  }
  fits = fits && total <= kRSortMax;
  if (tm.rank == 0 && fits && tm.C > 1) {
    // gather the other members' band entries behind this CTA's own
    int off = static_cast<int>(tm.get(sm.misc, 6, 0));
    for (int r = 1; r < tm.C; ++r) {
      const int n = static_cast<int>(tm.get(sm.misc, 6, r));
      const unsigned long long* src = tm.remote(sm.cw, r);
      for (int i = threadIdx.x; i < n; i += kRT) sm.cw[off + i] = src[i];
      off += n;
    }
  }
  tm.sync();  // the band is gathered; the other members may reuse their buffers
  if (tm.rank != 0) return -1;
  // the boundary inside bin bstar: a histogram of the band's exact weights over 1024
  // sub-bins (by position in the bin) finds the sub-bin holding it, whose few entries are
  // ranked pairwise; a crowded sub-bin sorts the whole band instead
  const float fbf = ftab[bstar];
  const double fb = static_cast<double>(fbf) * 5.9604644775390625e-8;
  int L = 0;           // > 0: the sorted band's kept prefix (sort path)
  bool have_th = false;
  Thresh bth{0u, -1};  // the boundary entry (sub-bin path)
  if (fits) {
    uint32_t* sh = sm.hist;  // kRPSub words of low limbs, then kRPSub of high limbs
    for (int i = threadIdx.x; i < 2 * kRPSub; i += kRT) sh[i] = 0u;
    uint32_t& s_cnt = *reinterpret_cast<uint32_t*>(sm.misc + kMCnt);
    if (threadIdx.x == 0) {
      sm.misc[kMBin] = ~0ull;
      sm.misc[kMHit] = 0ull;
      s_cnt = 0u;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < total; i += kRT) {
      const PW w = pweight(kfloat(static_cast<uint32_t>(sm.cw[i] >> 32)), H);
      const int sb = psub(w);
      sh_red_add(&sh[sb], w.w24 & 0xFFFu);
      sh_red_add(&sh[kRPSub + sb], w.w24 >> 12);
    }
    __syncthreads();
    constexpr int per = kRPSub / kRT;
    double m[per];
    double sum = 0.0;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      const int b = per * static_cast<int>(threadIdx.x) + e;
      m[e] = static_cast<double>(static_cast<unsigned long long>(sh[b]) +
                                 (static_cast<unsigned long long>(sh[kRPSub + b]) << 12)) * fb;
      sum += m[e];
    }
    const int lane2 = threadIdx.x & 31, warp2 = threadIdx.x >> 5;
    double x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(kFull, x, o);
      if (lane2 >= o) x += y;
    }
    double* redd = reinterpret_cast<double*>(sm.red);
    if (lane2 == 31) redd[warp2] = x;
    __syncthreads();
    if (warp2 == 0) {
      const double sv = lane2 < kRW ? redd[lane2] : 0.0;
      double t = sv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(kFull, t, o);
        if (lane2 >= o) t += y;
      }
      if (lane2 < kRW) redd[kRW + lane2] = t - sv;
    }
    __syncthreads();
    double acc = above + redd[kRW + warp2] + x - sum;
    if (above < tq) {
#pragma unroll
      for (int e = 0; e < per; ++e) {
        const int b = per * static_cast<int>(threadIdx.x) + e;
        if (acc < tq && acc + m[e] >= tq) {
          sm.misc[kMBin] = static_cast<unsigned long long>(b);
          reinterpret_cast<double*>(sm.misc)[kMAbove] = acc;
        }
        acc += m[e];
      }
    }
    __syncthreads();
    const unsigned long long beta = sm.misc[kMBin];
    const double before = reinterpret_cast<const double*>(sm.misc)[kMAbove];
    if (beta != ~0ull) {
      // the entries of sub-bin beta, with their weights
      unsigned long long* gw = sm.wbuf;  // order words
      double* gm = reinterpret_cast<double*>(sm.wbuf + kRRank);
      for (int i = threadIdx.x; i < total; i += kRT) {
        const unsigned long long wd = sm.cw[i];
        const PW w = pweight(kfloat(static_cast<uint32_t>(wd >> 32)), H);
        if (psub(w) == static_cast<int>(beta)) {
          const uint32_t pos = atomicAdd(&s_cnt, 1u);
          if (pos < static_cast<uint32_t>(kRRank)) {
            gw[pos] = wd;
            gm[pos] = static_cast<double>(w.w24) * fb;
          }
        }
      }
      __syncthreads();
      const int mcount = static_cast<int>(s_cnt);
      if (mcount <= kRRank) {
        for (int i = threadIdx.x; i < mcount; i += kRT) {
          const unsigned long long wi = gw[i];
          double ex = before;
          for (int j = 0; j < mcount; ++j) ex += gw[j] > wi ? gm[j] : 0.0;
          if (ex < tq && tq <= ex + gm[i]) sm.misc[kMHit] = wi;
        }
      }
      __syncthreads();
      const unsigned long long hit = sm.misc[kMHit];
      if (hit) {
        have_th = true;
        bth = Thresh{static_cast<uint32_t>(hit >> 32), static_cast<int32_t>(~static_cast<uint32_t>(hit))};
      }
      __syncthreads();
    }
    if (!have_th) {
      // crowded sub-bin: sort the band and cut the first entry whose prefix reaches tq
      int N = 1;
      while (N < total) N <<= 1;
      rbitonic_desc(sm.cw, N);
      constexpr int per2 = kRSortMax / kRT;
      double wv[per2];
      double sum2 = 0.0;
#pragma unroll
      for (int e = 0; e < per2; ++e) {
        const int i = per2 * static_cast<int>(threadIdx.x) + e;
        wv[e] = i < total ? static_cast<double>(pweight(kfloat(static_cast<uint32_t>(sm.cw[i] >> 32)), H).w24) * fb : 0.0;
        sum2 += wv[e];
      }
      if (threadIdx.x == 0) sm.misc[kMCut] = 0ull;
      double x2 = sum2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(kFull, x2, o);
        if (lane2 >= o) x2 += y;
      }
      if (lane2 == 31) redd[warp2] = x2;
      __syncthreads();
      if (warp2 == 0) {
        const double sv = lane2 < kRW ? redd[lane2] : 0.0;
        double t = sv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(kFull, t, o);
          if (lane2 >= o) t += y;
        }
        if (lane2 < kRW) redd[kRW + lane2] = t - sv;
      }
      __syncthreads();
      double acc2 = above + redd[kRW + warp2] + x2 - sum2;
      if (above < tq) {
#pragma unroll
        for (int e = 0; e < per2; ++e) {
          const int i = per2 * static_cast<int>(threadIdx.x) + e;
          if (i < total && acc2 < tq && acc2 + wv[e] >= tq) sm.misc[kMCut] = static_cast<unsigned long long>(i + 1);
          acc2 += wv[e];
        }
      }
      __syncthreads();
      L = static_cast<int>(sm.misc[kMCut]);
      __syncthreads();
      if (L > 0) {
        have_th = true;
        const unsigned long long wl = sm.cw[L - 1];
        bth = Thresh{static_cast<uint32_t>(wl >> 32), static_cast<int32_t>(~static_cast<uint32_t>(wl))};
      }
    }
  }
  if (!have_th) {
    // the band overflowed or missed the boundary: the exact selection over the whole row
    // (fixed-point masses against the true maximum), then race and write all of it again
    unsigned long long part = 0;
    rrow_pass<kBF16>(whole, l2_policy_normal(), [&](bool valid, float y, uint32_t, int) {
      if (valid) part += fixed_mass(softmax_weight(y, M));
    });
    const unsigned long long tqx = rtopp_target(p, rblock_sum_u64(part, sm.red));
    const Thresh th = rrow_select<kBF16, true>(whole, tqx, M, sm.hist, sm.red, sm.misc);
    unsigned long long rb2, first2;
    rrow_race_write<kBF16>(whole, th, M, eps, l2_policy_normal(), sm.red, &rb2, &first2);
    return static_cast<int32_t>(~static_cast<uint32_t>(rb2 ? rb2 : first2));
  }
  // race over the kept part of the boundary bin, in pass A's arithmetic
  {
    const float f24b = __fmul_rn(fbf, 5.9604644775390625e-8f);
    float rbest = -1.0f;
    int ridx = INT_MAX;
    unsigned long long gfirst = 0;  // sampling off: the first kept entry of the order
    for (int i = threadIdx.x; i < total; i += kRT) {
      const unsigned long long wd = sm.cw[i];
      const uint32_t key = static_cast<uint32_t>(wd >> 32);
      const int32_t idx = static_cast<int32_t>(~static_cast<uint32_t>(wd));
      if (!kept_by(key, idx, bth.key, bth.idx)) continue;
      gfirst = wd > gfirst ? wd : gfirst;
      const float y = kfloat(key);
      const uint32_t rk = rc.race ? prace_key(pweight(y, H).wf, rq1(rc, idx), eps) : 0u;
      const float r = rk ? prace_value(rk, f24b) : -1.0f;
      if (rk && (r > rbest || (r == rbest && idx < ridx))) {
        rbest = r;
        ridx = idx;
      }
      if (rc.out) rc.out[idx] = y;
    }
    unsigned long long c = !rc.race ? gfirst : rbest >= 0.0f ? order_word(fkey(rbest), ridx) : 0ull;
    c = c > rb ? c : rb;
    unsigned long long dummy = 0;
    rblock_max2(c, dummy, sm.red);
    rb = c;
  }
  if (rb) return static_cast<int32_t>(~static_cast<uint32_t>(rb));
  return rrow_first_max<kBF16>(whole, M, sm.red);  // every race quotient was NaN
}

// ---- work units and the kernel -----------------------------------------------------------

__device__ __forceinline__ bool row_is_wide(const Params& P, int64_t row) { return !row_is_kmode(P, row); }

// The work units of the launch: every wide row (top-p-only or keep-all) is one unit for
// all C CTAs of a cluster; top-k and one-element rows come C to a unit, one per CTA, unless
// every row fits a cluster of its own (then rank 0 takes it and the rows spread over more
// SMs).  Units go round-robin over the clusters: the wide units first, or, when a pre-pass
// runs alongside (its rows wait for it), last.  Writes this CTA's items in unit order
// (>= 0: a row of its own, -1: nothing in that unit, <= -2: wide row -(item + 2)) and
// returns their count, or -1 when they do not fit kRMaxItems.
__device__ int rbuild_items(const Params& P, int C, int rank, int cluster, int nclusters, int32_t* items,
                            int32_t* ords, unsigned long long* red) {
  if (P.B <= kRT) {
    // one row per thread: its class read once, one scan of the packed counts
    // (wide << 40 | pre-pass << 20 | top-k; B < 2^20)
    const int64_t r = threadIdx.x;
    const bool valid = r < P.B;
    const bool wide = valid && row_is_wide(P, r);
    const bool pre = P.pre != nullptr && valid && row_prepass(P, r);
    const unsigned long long v =
        valid ? (wide ? (1ull << 40) : 1ull) + (pre ? (1ull << 20) : 0ull) : 0ull;
    unsigned long long tot;
    const unsigned long long ex = rblock_excl_scan_u64(v, &tot, red);
    const int64_t nwide = static_cast<int64_t>(tot >> 40), nk = static_cast<int64_t>(tot & 0xFFFFFull);
    const int per = P.B <= nclusters ? 1 : C;  // top-k rows per unit
    const int64_t kunits = (nk + per - 1) / per;
    const int64_t units = nwide + kunits;
    const bool wide_last = P.pre != nullptr;
    const int64_t mine = units > cluster ? (units - 1 - cluster) / nclusters + 1 : 0;
    if ((units + nclusters - 1) / nclusters > kRMaxItems) return -1;  // the same answer in every CTA
    for (int i = threadIdx.x; i < mine; i += kRT) {
      items[i] = -1;
      ords[i] = -1;
    }
    __syncthreads();
    if (valid) {
      int64_t unit, slot;
      if (wide) {
        unit = static_cast<int64_t>(ex >> 40) + (wide_last ? kunits : 0);
        slot = rank;
      } else {
        const int64_t ko = static_cast<int64_t>(ex & 0xFFFFFull);
        unit = (wide_last ? 0 : nwide) + ko / per;
        slot = (per == 1 && P.V > kRKeepAllV) ? rank : ko % per;  // one row per unit: the CTAs share it
      }
      if (unit % nclusters == cluster && slot == rank) {
        items[unit / nclusters] = wide ? static_cast<int32_t>(-(r + 2)) : static_cast<int32_t>(r);
        const unsigned long long po = (ex >> 20) & 0xFFFFFull;
        if (pre && po < static_cast<unsigned long long>(P.pre_rows)) ords[unit / nclusters] = static_cast<int32_t>(po);
      }
    }
    __syncthreads();
    return static_cast<int>(mine);
  }
  unsigned long long nwide = 0, dummy0 = 0, dummy1 = 0;
  for (int64_t r = threadIdx.x; r < P.B; r += kRT) nwide += row_is_wide(P, r) ? 1ull : 0ull;
  rblock_sum_max2(nwide, dummy0, dummy1, red);
  const int64_t nk = P.B - static_cast<int64_t>(nwide);
  const int per = P.B <= nclusters ? 1 : C;  // top-k rows per unit
  const int64_t kunits = (nk + per - 1) / per;
  const int64_t units = static_cast<int64_t>(nwide) + kunits;
  const bool wide_last = P.pre != nullptr;
  const int64_t mine = units > cluster ? (units - 1 - cluster) / nclusters + 1 : 0;
  if ((units + nclusters - 1) / nclusters > kRMaxItems) return -1;  // the same answer in every CTA
  for (int i = threadIdx.x; i < mine; i += kRT) {
    items[i] = -1;
    ords[i] = -1;
  }
  __syncthreads();
  unsigned long long wbase = 0, kbase = 0, pbase = 0;
  for (int64_t base = 0; base < P.B; base += kRT) {
    const int64_t r = base + threadIdx.x;
    const bool valid = r < P.B;
    const bool wide = valid && row_is_wide(P, r);
    // one scan of (wide count << 32 | top-k count)
    const unsigned long long v = valid ? (wide ? (1ull << 32) : 1ull) : 0ull;
    unsigned long long tot;
    const unsigned long long ex = rblock_excl_scan_u64(v, &tot, red);
    // ordinals among the pre-pass rows (only with records)
    const bool pre = P.pre != nullptr && valid && row_prepass(P, r);
    unsigned long long ptot = 0, pex = 0;
    if (P.pre != nullptr) pex = rblock_excl_scan_u64(pre ? 1ull : 0ull, &ptot, red);
    if (valid) {
      int64_t unit, slot;
      if (wide) {
        unit = static_cast<int64_t>(wbase + (ex >> 32)) + (wide_last ? kunits : 0);
        slot = rank;
      } else {
        const int64_t ko = static_cast<int64_t>(kbase + (ex & 0xFFFFFFFFull));
        unit = (wide_last ? 0 : static_cast<int64_t>(nwide)) + ko / per;
        slot = (per == 1 && P.V > kRKeepAllV) ? rank : ko % per;  // one row per unit: the CTAs share it
      }
      if (unit % nclusters == cluster && slot == rank) {
        items[unit / nclusters] = wide ? static_cast<int32_t>(-(r + 2)) : static_cast<int32_t>(r);
        const unsigned long long po = pbase + pex;
        if (pre && po < static_cast<unsigned long long>(P.pre_rows)) ords[unit / nclusters] = static_cast<int32_t>(po);
      }
    }
    wbase += tot >> 32;
    kbase += tot & 0xFFFFFFFFull;
    pbase += ptot;
  }
  __syncthreads();
  return static_cast<int>(mine);
}

// Copies a row's seen bits (V <= kRMaxV tokens; bits of tokens >= V cleared) into the
// bitmap: 16-byte loads, all in flight at once, when the row's words allow them.
__device__ __forceinline__ void rseen_copy(const uint32_t* src, int V, uint32_t* bitmap) {
  const int W = (V + 31) / 32;
  if ((W & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
    constexpr int kPer = (kRMaxV / 128 + kRT - 1) / kRT;  // 16-byte vectors per thread
    const int W4 = W / 4;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = static_cast<int>(threadIdx.x) + u * kRT;
      v[u] = i < W4 ? __ldcg(s4 + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = static_cast<int>(threadIdx.x) + u * kRT;
      if (i < W4) {
        if (i == W4 - 1 && (V & 31)) v[u].w &= (1u << (V & 31)) - 1u;
        reinterpret_cast<uint4*>(bitmap)[i] = v[u];
      }
    }
  } else {
    for (int w0 = static_cast<int>(threadIdx.x); w0 < W; w0 += 4 * kRT) {
      uint32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = seen_word_at(src, V, w0 + u * kRT);  // 0 past the row
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (w0 + u * kRT < W) bitmap[w0 + u * kRT] = v[u];
    }
  }
}

// The parameters of a row and its context for part `part` of `nparts` (a team member's
// share of the vectors); sets the seen bits of the row in the bitmap (which is clear), or
// copies the caller's seen bits of the row into it.
struct RowFlags {
  int32_t k;
  float p;
  bool pen_on, single, topp_on;
  int32_t b0, b1;  // the row's seen ids
};
template <bool kBF16>
__device__ __forceinline__ RowFlags row_setup(const Params& P, int64_t row, const RowSmem& sm, int part, int nparts,
                                              RowCtx* rcp, bool sample = false) {
  constexpr int G = kBF16 ? 8 : 4;
  const size_t esize = kBF16 ? 2 : 4;
  const int V = static_cast<int>(P.V);
  RowFlags f;
  f.k = P.top_k[row];
  f.p = P.top_p[row];
  const float T = P.temperature[row];
  const bool greedyT = !(T > 0.0f) || isinf(T);
  f.pen_on = ((P.seen_indptr && P.seen_ids) || P.seen_bits) && P.penalty && (P.penalty[row] > 0.0f);
  const bool topk_on = f.k >= 1 && static_cast<int64_t>(f.k) <= (P.V < kTopKMax ? P.V : kTopKMax);
  const bool p_nan = isnan(f.p);
  f.single = greedyT || (!p_nan && f.p <= 0.0f) || (topk_on && f.k == 1);
  f.topp_on = !f.single && !p_nan && f.p > 0.0f && f.p < 1.0f;
  RowCtx& rc = *rcp;
  rc.x = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(P.logits) + row * P.V * esize);
  rc.q = P.q ? P.q + row * P.V : nullptr;  // none: sampling off or generated draws
  rc.gen = P.gen != 0;
  rc.race = rc.q != nullptr || rc.gen;
  rc.seed = P.seed;
  rc.step = P.step;
  rc.row = row;
  rc.out = P.need_logits ? P.out_filtered + row * P.V : nullptr;
  rc.V = V;
  rc.nv = V / G;
  rc.g0 = static_cast<int>(static_cast<int64_t>(rc.nv) * part / nparts);
  rc.g1 = static_cast<int>(static_cast<int64_t>(rc.nv) * (part + 1) / nparts);
  rc.bitmap = sm.bitmap;
  rc.pen_on = f.pen_on;
  rc.pen = f.pen_on ? P.penalty[row] : 1.0f;
  rc.T = T;
  rc.div = make_divisor(greedyT ? 1.0f : T);
  rc.identity = greedyT;
  // the sample of a top-k row (its threshold comes first): loads issued before the
  // seen ids', transformed once the bitmap is built
  SampleLoads sl;
  if (sample) rsample_fetch<kBF16>(rc, &sl);
  // the caller's seen bits of the row: their loads ride along with the sample's (no thread
  // reads the bitmap again before the barrier below)
  if (f.pen_on && P.seen_bits) rseen_copy(P.seen_bits + row * seen_words(P.V), V, sm.bitmap);
  __syncthreads();  // the bitmap of the previous row is clear
  f.b0 = 0;
  f.b1 = 0;
  if (f.pen_on && !P.seen_bits) {
    f.b0 = P.seen_indptr[row];
    f.b1 = P.seen_indptr[row + 1];
    for (int32_t t = f.b0 + static_cast<int32_t>(threadIdx.x); t < f.b1; t += kRT) {
      const int32_t id = P.seen_ids[t];
      if (id >= 0 && id < V) atomicOr(&sm.bitmap[id >> 5], 1u << (id & 31));
    }
  }
  __syncthreads();
  if (sample) rsample_finish(rc, sl, reinterpret_cast<uint32_t*>(sm.wbuf));
  return f;
}
// Clears the row's seen bits again (seen bits given: the next row overwrites every word).
__device__ __forceinline__ void row_teardown(const Params& P, int64_t row, const RowFlags& f, const RowSmem& sm) {
  if (!f.pen_on || P.seen_bits) return;
  const int V = static_cast<int>(P.V);
  for (int32_t t = f.b0 + static_cast<int32_t>(threadIdx.x); t < f.b1; t += kRT) {
    const int32_t id = P.seen_ids[t];
    if (id >= 0 && id < V) sm.bitmap[id >> 5] = 0u;
  }
}

// The pre-pass: pass A of every top-p-only row with a record, each row cut into chunks
// spread over the grid (as many as the grid holds, up to kPreMaxChunks).  Every CTA of a
// row samples the same elements for H; each runs pass A over its chunk in shared memory
// and merges the bin sums and race words into the row's record with global atomics.
template <bool kBF16>
__global__ void __launch_bounds__(kRT, 2) kps_prepass_kernel(const Params P) {
  extern __shared__ __align__(16) unsigned char r_smem[];
  debug_fill_smem(r_smem, false);
  const RLayout lay = make_rlayout(P.V);
  RowSmem sm;
  sm.bitmap = reinterpret_cast<uint32_t*>(r_smem + lay.bitmap);
  sm.cw = reinterpret_cast<unsigned long long*>(r_smem + lay.cw);
  sm.hist = reinterpret_cast<uint32_t*>(r_smem + lay.hist);
  sm.wbuf = reinterpret_cast<unsigned long long*>(r_smem + lay.wbuf);
  sm.red = reinterpret_cast<unsigned long long*>(r_smem + lay.red);
  sm.misc = reinterpret_cast<unsigned long long*>(r_smem + lay.misc);
  // the row kernel may start now: its rows that need a record wait for this grid to end
  asm volatile("griddepcontrol.launch_dependents;");
  const int V = static_cast<int>(P.V);
  for (int w = threadIdx.x; w < (V + 31) / 32; w += kRT) sm.bitmap[w] = 0u;
  unsigned long long cnt = 0;
  for (int64_t r = threadIdx.x; r < P.B; r += kRT) cnt += row_prepass(P, r) ? 1ull : 0ull;
  cnt = rblock_sum_u64(cnt, sm.red);
  const int np = static_cast<int>(cnt < static_cast<unsigned long long>(P.pre_rows) ? cnt : P.pre_rows);
  if (np == 0) return;
  // the whole grid (CTAs past the units leave at once, making room for the row kernel)
  int nch = static_cast<int>(gridDim.x) / np;
  nch = nch < 1 ? 1 : (nch > kPreMaxChunks ? kPreMaxChunks : nch);
  const int units = np * nch;
  int64_t& s_row = *reinterpret_cast<int64_t*>(sm.misc + kMFound);
  for (int u = static_cast<int>(blockIdx.x); u < units; u += static_cast<int>(gridDim.x)) {
    const int j = u / nch, c = u - (u / nch) * nch;
    // the j-th row with row_prepass
    if (threadIdx.x == 0) s_row = -1;
    unsigned long long run = 0;
    for (int64_t b0 = 0; b0 < P.B; b0 += kRT) {
      const int64_t r = b0 + threadIdx.x;
      const unsigned long long v = (r < P.B && row_prepass(P, r)) ? 1ull : 0ull;
      unsigned long long tot;
      const unsigned long long ex = rblock_excl_scan_u64(v, &tot, sm.red);
      if (v && run + ex == static_cast<unsigned long long>(j)) s_row = r;
      run += tot;
      if (run > static_cast<unsigned long long>(j)) break;  // the same for every thread
    }
    __syncthreads();
    const int64_t row = s_row;
    RowCtx rc;
    // the sample (the same elements in every chunk's CTA) is loaded alongside the seen ids
    const RowFlags f = row_setup<kBF16>(P, row, sm, c, nch, &rc, true);
    const uint32_t* samp = reinterpret_cast<const uint32_t*>(sm.wbuf);
    unsigned long long a = 0, b = 0;
    for (int i = threadIdx.x; i < kRSamp; i += kRT) a = samp[i] > a ? samp[i] : a;
    rblock_max2(a, b, sm.red);
    const float H = pgrid_up(__fadd_rn(kfloat(static_cast<uint32_t>(a)), kRHeadroom));
    const PRec rec = prec_at(P, j);
    if (c == 0 && threadIdx.x == 0) *rec.H = __float_as_uint(H);
    if (pgrid_ok(H)) {
      const unsigned long long kmax = rp_pass_a<kBF16>(rc, H, P.eps, sm.hist, sm.cw, sm.red);
      for (int bb = threadIdx.x; bb < kRPBins; bb += kRT) {
        const unsigned long long sb =
            static_cast<unsigned long long>(sm.hist[bb]) + (static_cast<unsigned long long>(sm.hist[kRPBins + bb]) << 12);
        if (sb) atomicAdd(rec.sums + bb, sb);
        const unsigned long long wb = sm.cw[bb];
        if (wb) atomicMax(rec.ub + bb, wb);
      }
      if (threadIdx.x == 0) atomicMax(rec.M, kmax);
    }
    __syncthreads();
    row_teardown(P, row, f, sm);
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kRT, 2) kps_row_kernel(const Params P) {
  extern __shared__ __align__(16) unsigned char r_smem[];
  debug_fill_smem(r_smem, true);
  const RLayout lay = make_rlayout(P.V);
  RowSmem sm;
  sm.bitmap = reinterpret_cast<uint32_t*>(r_smem + lay.bitmap);
  sm.cw = reinterpret_cast<unsigned long long*>(r_smem + lay.cw);
  sm.hist = reinterpret_cast<uint32_t*>(r_smem + lay.hist);
  sm.wbuf = reinterpret_cast<unsigned long long*>(r_smem + lay.wbuf);
  sm.red = reinterpret_cast<unsigned long long*>(r_smem + lay.red);
  sm.misc = reinterpret_cast<unsigned long long*>(r_smem + lay.misc);
  int32_t* items = reinterpret_cast<int32_t*>(r_smem + lay.items);
  int32_t* ords = reinterpret_cast<int32_t*>(r_smem + lay.ords);
  const int V = static_cast<int>(P.V);
  for (int w = threadIdx.x; w < (V + 31) / 32; w += kRT) sm.bitmap[w] = 0u;

  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int cluster = static_cast<int>(blockIdx.x) / C;
  const int nclusters = static_cast<int>(gridDim.x) / C;
  int nitems = rbuild_items(P, C, rank, cluster, nclusters, items, ords, sm.red);
  const bool shared_rows = nitems >= 0;
  if (!shared_rows) {
    // too many units for the item list: every CTA takes rows on its own, round-robin
    nitems = P.B > blockIdx.x ? static_cast<int>((P.B - 1 - blockIdx.x) / gridDim.x + 1) : 0;
  }
  const Team alone{1, 0};
  const Team team = shared_rows ? Team{C, rank} : alone;

  for (int it = 0; it < nitems; ++it) {
    int64_t row;
    bool wide;
    int32_t ord = -1;  // the row's pre-pass record
    if (shared_rows) {
      const int32_t item = items[it];
      if (item == -1) continue;
      wide = item <= -2;
      row = wide ? static_cast<int64_t>(-(item + 2)) : static_cast<int64_t>(item);
      ord = ords[it];
    } else {
      row = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(it) * gridDim.x;
      wide = row_is_wide(P, row);
    }
    // with every row in a cluster of its own, a top-k row (longer than the rows taken whole)
    // is shared by the cluster's CTAs, each streaming its part against the same threshold
    const bool kteam = !wide && shared_rows && P.B <= nclusters && P.V > kRKeepAllV;
    const Team& tm = (wide || kteam) ? team : alone;
    RowCtx rc;
    const bool sample = !wide && !P.exact && P.V > kRKeepAllV;
    const RowFlags f = row_setup<kBF16>(P, row, sm, tm.rank, tm.C, &rc, sample);
    int32_t chosen;
    if (!wide) {
      chosen = rk_row<kBF16>(rc, sm, tm, f.single ? 1u : static_cast<uint32_t>(f.k), f.single, f.topp_on, f.p, P.eps,
                             P.exact != 0, sample);
    } else {
      PRec rec;
      if (!shared_rows && P.pre && row_prepass(P, row)) {
        const int j = prepass_ordinal(P, row, sm.red);
        ord = j < P.pre_rows ? j : -1;
      }
      if (ord >= 0) rec = prec_at(P, ord);
      chosen = rwide_row<kBF16>(rc, sm, tm, f.topp_on, f.p, P.eps, P.exact != 0, ord >= 0 ? &rec : nullptr);
    }
    if (threadIdx.x == 0 && chosen >= 0) {
      const long long tok = eos_epilogue(P, row, chosen);
      P.out_idx[row] = tok;
      seen_append(P, row, tok);
    }
    __syncthreads();
    row_teardown(P, row, f, sm);
  }
  // members of a cluster leave together: no CTA exits while another may still read its
  // shared memory
  if (C > 1) cl.sync();
}
