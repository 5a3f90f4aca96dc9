// kps_stream.cuh — the streaming sampler: one CTA walks whole rows through a
// TMA ring.  Included by kps.cu inside namespace kps (uses its helpers).
//
// For batches large enough to give every SM its own rows, the row never needs
// to live on chip: a persistent grid of 1024-thread CTAs streams each row once
// from HBM through a ring of shared-memory stages filled by cp.async.bulk, and
// keeps only what the selection needs.
//
//   top-k rows (and one-element rows, as k = 1): a raw-space prefilter
//     against a running threshold lets only elements that can still rank
//     reach the exact division by T; those are kept in a candidate buffer.
//     When the buffer passes kSHigh entries it is cut to its exact top-k
//     (value desc, index asc) and the threshold rises to the k-th entry, so
//     later elements must beat it strictly (later equal values have larger
//     indices).  The -inf filtered output streams out as the data passes.
//     At the row's end: exact top-k, then a sort of the <= 1024 survivors for
//     the top-p cut (exact fixed-point prefix), the race on q gathered at the
//     kept indices, and the kept values scattered over the -inf output.
//   top-p-only rows: the ring pass finds the row maximum; three more passes
//     over the row (served from L2) build a mass histogram over linear bins
//     of (max - x), refine inside the boundary bin while collecting its
//     elements, rank the few elements of the final bin exactly, then run the
//     race and write the filtered logits.
//   rows with every element kept: one more pass for the race and the output.
//
// Everything is block-local: no clusters, no distributed shared memory.

constexpr int kST = 512;             // consumer threads (the block helpers below run over them)
constexpr int kSW = kST / 32;
constexpr int kSThreads = kST + 32;  // plus one producer warp that only issues TMA copies
constexpr int kStageElems = 4096;    // elements per ring stage (two float4 per consumer thread)
constexpr int kSPer = kStageElems / (4 * kST);

// Barrier among the consumer warps only (named barrier 1); the producer warp never joins it.
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kST) : "memory"); }
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
constexpr int kSCap = 6144;          // candidate buffer entries
constexpr int kSHigh = 2048;         // cut the buffer when it holds more than this
constexpr int kSMaxStages = 8;
constexpr int kSMinStages = 3;
constexpr int kSMaxV = 262144;       // the row's penalty bitmap lives in shared memory
constexpr int kSRank = 256;          // boundary-bin elements ranked pairwise

struct SLayout {
  size_t ring, ckey, cidx, bitmap, hist, kbuf, red, misc, bars, rows, total;
  int stages;
  size_t stage_bytes;
};

__host__ __device__ inline SLayout make_slayout(int64_t V, bool bf16, int stages) {
  SLayout L;
  L.stages = stages;
  L.stage_bytes = align16(size_t(kStageElems) * (bf16 ? 2 : 4));
  size_t off = 0;
  L.ring = off;   off += size_t(stages) * L.stage_bytes;
  L.ckey = off;   off += size_t(kSCap) * 4;
  L.cidx = off;   off += size_t(kSCap) * 4;
  L.bitmap = off; off += align16(size_t((V + 31) / 32) * 4);
  L.hist = off;   off += size_t(kLinBins) * 8;
  L.kbuf = off;   off += size_t(kTopKMax) * 8;  // survivors (order words) / fine histogram
  L.red = off;    off += 64 * 8;
  L.misc = off;   off += 32 * 8;
  L.bars = off;   off += align16(size_t(2 * stages) * 8);  // full[stages], empty[stages]
  L.rows = off;   off += size_t(kMaxRowList) * 4;
  L.total = off;
  return L;
}

// ---- block helpers for kST threads --------------------------------------------------------
__device__ unsigned long long sblock_max_u64(unsigned long long v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_u64(v);
  if (lane == 0) red[warp] = v;
  csync();
  if (warp == 0) {
    v = lane < kSW ? red[lane] : 0ull;
    v = warp_max_u64(v);
    if (lane == 0) red[32] = v;
  }
  csync();
  v = red[32];
  csync();
  return v;
}
__device__ unsigned long long sblock_sum_u64(unsigned long long v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane == 0) red[warp] = v;
  csync();
  if (warp == 0) {
    v = lane < kSW ? red[lane] : 0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (lane == 0) red[32] = v;
  }
  csync();
  v = red[32];
  csync();
  return v;
}
// Exclusive scan over the block (thread order); *total gets the sum.
__device__ unsigned long long sblock_excl_scan_u64(unsigned long long v, unsigned long long* total,
                                                   unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long x = warp_incl_scan_u64(v, lane);
  if (lane == 31) red[warp] = x;
  csync();
  if (warp == 0) {
    const unsigned long long s = lane < kSW ? red[lane] : 0ull;
    const unsigned long long t = warp_incl_scan_u64(s, lane);
    if (lane < kSW) red[lane] = t - s;
    if (lane == kSW - 1) red[32] = t;
  }
  csync();
  const unsigned long long res = red[warp] + x - v;
  *total = red[32];
  csync();
  return res;
}

// k-th largest (1-based) of the values key(i) over entries i < n with pred(i), exact,
// block-local; 4 passes of 8-bit digits with warp-aggregated counts into h[256].
// Returns the key; *above gets how many selected entries are strictly larger.
template <class KeyF, class PredF>
__device__ uint32_t sblock_kth_largest(int n, uint32_t k, KeyF keyf, PredF pred, uint32_t* h,
                                       unsigned long long* misc, uint32_t* above) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t prefix = 0, pmask = 0, acc_above = 0;
  for (int d = 0; d < 4; ++d) {
    const int shift = 24 - 8 * d;
    for (int i = threadIdx.x; i < kBins; i += kST) h[i] = 0u;
    csync();
    for (int base = 0; base < n; base += kST) {
      const int i = base + threadIdx.x;
      bool take = false;
      uint32_t key = 0;
      if (i < n && pred(i)) {
        key = keyf(i);
        take = (key & pmask) == prefix;
      }
      const int bin = static_cast<int>((key >> shift) & 0xFFu);
      const unsigned peers = __match_any_sync(kFull, take ? bin : -1);
      if (take && lane == __ffs(peers) - 1) atomicAdd(&h[bin], static_cast<uint32_t>(__popc(peers)));
    }
    csync();
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
        const int L = __ffs(m) - 1;
        if (lane == L) {
          uint32_t acc = inc - sum;
          int beta = 255 - 8 * lane;
          for (int e = 0; e < 8; ++e) {
            if (acc + b[e] >= k) {
              beta = 255 - 8 * lane - e;
              break;
            }
            acc += b[e];
          }
          misc[0] = static_cast<unsigned long long>(beta);
          misc[1] = k - acc;
          misc[2] = acc;
        }
      } else if (lane == 0) {
        misc[0] = 0ull;  // k exceeds the selection: keep everything (cannot happen for valid k)
        misc[1] = 1ull;
        misc[2] = 0ull;
      }
    }
    csync();
    prefix |= static_cast<uint32_t>(misc[0]) << shift;
    pmask |= 0xFFu << shift;
    k = static_cast<uint32_t>(misc[1]);
    acc_above += static_cast<uint32_t>(misc[2]);
    csync();
  }
  *above = acc_above;
  return prefix;
}

// Exact top-k (value desc, index asc) of the candidate buffer: returns the
// threshold (key, index) of the k-th entry.  n >= k >= 1.
__device__ Thresh sblock_topk_threshold(const uint32_t* ckey, const int32_t* cidx, int n, uint32_t k,
                                        uint32_t* h, unsigned long long* misc, unsigned long long* red) {
  uint32_t above = 0;
  const uint32_t kk = sblock_kth_largest(
      n, k, [&](int i) { return ckey[i]; }, [&](int) { return true; }, h, misc, &above);
  // ties at kk: keep the (k - above) smallest indices
  unsigned long long ties = 0, imax = 0;
  for (int i = threadIdx.x; i < n; i += kST)
    if (ckey[i] == kk) {
      ++ties;
      const unsigned long long w = static_cast<uint32_t>(cidx[i]);
      imax = w > imax ? w : imax;
    }
  ties = sblock_sum_u64(ties, red);
  imax = sblock_max_u64(imax, red);
  const uint32_t j = k - above;
  if (static_cast<unsigned long long>(j) >= ties) return Thresh{kk, static_cast<int32_t>(imax)};
  uint32_t above2 = 0;
  const uint32_t nidx = sblock_kth_largest(
      n, j, [&](int i) { return ~static_cast<uint32_t>(cidx[i]); }, [&](int i) { return ckey[i] == kk; }, h, misc,
      &above2);
  return Thresh{kk, static_cast<int32_t>(~nidx)};
}

// Keeps the buffer entries kept by th (all reads before any write); returns the new size.
__device__ int sblock_compact(uint32_t* ckey, int32_t* cidx, int n, Thresh th, unsigned long long* red) {
  constexpr int kPer = (kSCap + kST - 1) / kST;
  uint32_t kk[kPer];
  int32_t ii[kPer];
  uint32_t cnt = 0;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = threadIdx.x * kPer + u;
    kk[u] = 0u;
    ii[u] = 0;
    if (i < n && kept_by(ckey[i], cidx[i], th.key, th.idx)) {
      kk[u] = ckey[i];
      ii[u] = cidx[i];
      ++cnt;
    }
  }
  unsigned long long total;
  unsigned long long pos = sblock_excl_scan_u64(cnt, &total, red);
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    if (kk[u] != 0u) {
      ckey[pos] = kk[u];
      cidx[pos] = ii[u];
      ++pos;
    }
  }
  csync();
  return static_cast<int>(total);
}

// A raw value below which x / T cannot be kept by a threshold value tv:
// fl(x / T) >= tv implies x >= T * (tv - spacing(tv)).  -inf when tv is not a
// normal number with room.
__device__ __forceinline__ float raw_floor(float tv, float T, bool identity) {
  if (identity) return tv;
  const float a = fabsf(tv);
  if (!(a >= 1e-30f) || !(a <= 1e30f)) return -INFINITY;
  const float up = __uint_as_float(__float_as_uint(a) + 1u) - a;
  return __double2float_rd(static_cast<double>(T) * (static_cast<double>(tv) - 2.0 * static_cast<double>(up)));
}

// Transformed value of element x at row position v: NaN -> -inf, penalty if
// the bitmap bit is set, then x / T (unless identity), then -0 -> +0.
__device__ __forceinline__ float stransform(float x, bool pen_bit, float pen, float T, bool identity) {
  if (isnan(x)) x = -INFINITY;
  if (pen_bit) x = (x > 0.0f) ? __fdiv_rn(x, pen) : __fmul_rn(x, pen);
  if (!identity) x = __fdiv_rn(x, T);
  return __fadd_rn(x, 0.0f);
}

// One pass over a row straight from global memory (L2): f(valid, y, key, v) per
// element, whole warp converged; v is the row position.  Each thread keeps
// kSU 16-byte loads in flight before it uses them.
constexpr int kSU = 4;
template <bool kBF16, class F>
__device__ __forceinline__ void srow_pass(const Params& P, int64_t row, const uint32_t* bitmap, bool pen_on,
                                          float pen, float T, bool identity, F&& f) {
  const int64_t V = P.V;
  const int n4 = static_cast<int>((V + 3) >> 2);
  for (int base = 0; base < n4; base += kST * kSU) {
    float vv[kSU][4];
#pragma unroll
    for (int u = 0; u < kSU; ++u) {
      const int g = base + u * kST + threadIdx.x;
      if (g < n4) {
        if (kBF16) {
          const uint2 w = __ldcg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(P.logits) + row * V) + g);
          vv[u][0] = __uint_as_float(w.x << 16);
          vv[u][1] = __uint_as_float(w.x & 0xFFFF0000u);
          vv[u][2] = __uint_as_float(w.y << 16);
          vv[u][3] = __uint_as_float(w.y & 0xFFFF0000u);
        } else {
          const float4 w = __ldcg(reinterpret_cast<const float4*>(static_cast<const float*>(P.logits) + row * V) + g);
          vv[u][0] = w.x; vv[u][1] = w.y; vv[u][2] = w.z; vv[u][3] = w.w;
        }
      } else {
        vv[u][0] = vv[u][1] = vv[u][2] = vv[u][3] = 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < kSU; ++u) {
      const int g = base + u * kST + threadIdx.x;
      const bool in = g < n4;
      const int v0 = 4 * g;
      const uint32_t bits = (in && pen_on) ? (bitmap[v0 >> 5] >> (v0 & 31)) & 0xFu : 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool valid = in && (v0 + e) < V;
        const float y = valid ? stransform(vv[u][e], (bits >> e) & 1u, pen, T, identity) : 0.0f;
        f(valid, y, valid ? fkey(y) : 0u, v0 + e);
      }
    }
  }
}

// Block-local exact selection over a row read from global memory, for the
// top-p-only path when its small structures overflow: the shortest prefix of
// the order whose fixed-point mass reaches ceil(p * S).
template <bool kBF16>
__device__ Thresh srow_mass_select(const Params& P, int64_t row, const uint32_t* bitmap, bool pen_on, float pen,
                                   float T, bool identity, float M, float p, uint32_t* h32,
                                   unsigned long long* h, unsigned long long* misc, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t prefix = 0, pmask = 0;
  unsigned long long tau = 0;
  (void)h32;
  for (int d = 0; d < 4; ++d) {
    const int shift = 24 - 8 * d;
    for (int i = threadIdx.x; i < kBins; i += kST) h[i] = 0ull;
    csync();
    srow_pass<kBF16>(P, row, bitmap, pen_on, pen, T, identity, [&](bool valid, float y, uint32_t key, int) {
      if (!valid || (key & pmask) != prefix) return;
      const unsigned long long w = fixed_mass(softmax_weight(y, M));
      if (w) atomicAdd(&h[(key >> shift) & 0xFFu], w);
    });
    csync();
    if (warp == 0) {
      unsigned long long b[8];
      unsigned long long sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        b[e] = h[255 - 8 * lane - e];
        sum += b[e];
      }
      const unsigned long long inc = warp_incl_scan_u64(sum, lane);
      if (d == 0) {
        const unsigned long long total = __shfl_sync(kFull, inc, 31);
        const double t = ceil(static_cast<double>(p) * static_cast<double>(total));
        unsigned long long tt = static_cast<unsigned long long>(t);
        if (tt < 1ull) tt = 1ull;
        if (tt > total) tt = total;
        tau = tt;
      }
      const unsigned m = __ballot_sync(kFull, inc >= tau);
      if (m) {
        const int L = __ffs(m) - 1;
        if (lane == L) {
          unsigned long long acc = inc - sum;
          int beta = 255 - 8 * lane;
          for (int e = 0; e < 8; ++e) {
            if (acc + b[e] >= tau) {
              beta = 255 - 8 * lane - e;
              misc[2] = b[e];
              break;
            }
            acc += b[e];
          }
          misc[0] = static_cast<unsigned long long>(beta);
          misc[1] = tau - acc;
        }
      } else if (lane == 0) {
        misc[0] = 0ull;
        misc[1] = 1ull;
        misc[2] = 1ull;
      }
    }
    csync();
    prefix |= static_cast<uint32_t>(misc[0]) << shift;
    pmask |= 0xFFu << shift;
    tau = misc[1];
    csync();
  }
  // ties at `prefix`: keep the ceil(tau / w) smallest indices (scan in index order)
  const unsigned long long w1 = fixed_mass(softmax_weight(kfloat(prefix), M));
  const unsigned long long need = w1 ? (tau + w1 - 1) / w1 : 1ull;
  // count-and-locate in index order: tiles of kST*4 positions
  int32_t* found = reinterpret_cast<int32_t*>(misc + 4);
  if (threadIdx.x == 0) *found = INT_MAX;
  csync();
  unsigned long long seen = 0;
  const int64_t V = P.V;
  const int n4 = static_cast<int>((V + 3) >> 2);
  for (int base = 0; base < n4; base += kST) {
    uint32_t cnt = 0;
    uint32_t flags = 0;
    const int g = base + threadIdx.x;
    if (g < n4) {
      float vv[4];
      if (kBF16) {
        const uint2 u = __ldcg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(P.logits) + row * V) + g);
        vv[0] = __uint_as_float(u.x << 16); vv[1] = __uint_as_float(u.x & 0xFFFF0000u);
        vv[2] = __uint_as_float(u.y << 16); vv[3] = __uint_as_float(u.y & 0xFFFF0000u);
      } else {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(static_cast<const float*>(P.logits) + row * V) + g);
        vv[0] = v.x; vv[1] = v.y; vv[2] = v.z; vv[3] = v.w;
      }
      const int v0 = 4 * g;
      const uint32_t bits = pen_on ? (bitmap[v0 >> 5] >> (v0 & 31)) & 0xFu : 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (v0 + e < V && fkey(stransform(vv[e], (bits >> e) & 1u, pen, T, identity)) == prefix) {
          flags |= 1u << e;
          ++cnt;
        }
      }
    }
    unsigned long long total;
    const unsigned long long ex = sblock_excl_scan_u64(cnt, &total, red);
    if (cnt && seen + ex < need && need <= seen + ex + cnt) {
      unsigned long long s = seen + ex;
      for (int e = 0; e < 4; ++e)
        if ((flags >> e) & 1u) {
          ++s;
          if (s == need) *found = 4 * g + e;
        }
    }
    seen += total;
    csync();
    if (*found != INT_MAX || seen >= need) break;
  }
  csync();
  return Thresh{prefix, *found};
}

// A plain u64 histogram with the Bins interface sfind_bin uses (whole-row top-p path).
struct U64Bins {
  unsigned long long* base;
  int nb;
  __device__ __forceinline__ unsigned long long get(int b) const { return base[b]; }
};
// ---- selection inside the candidate buffer by linear bins -------------------------------

// Linear bin of y below hi (bin 0 holds the largest values); monotone non-increasing in y.
__device__ __forceinline__ int sbin(float y, float hi, float s) {
  if (!(y < hi)) return 0;
  const float f = __fmul_rn(__fsub_rn(hi, y), s);
  if (!(f < static_cast<float>(kLinBins))) return kLinBins - 1;
  return static_cast<int>(f);
}
__device__ __forceinline__ float sbin_scale(float hi, float lo) {
  const float span = __fsub_rn(hi, lo);
  return (span > 0.0f && span < INFINITY) ? __fdiv_rn(static_cast<float>(kLinBins), span) : 0.0f;
}

// Largest and smallest key of the buffer.
__device__ void sbuf_range(const uint32_t* ckey, int n, unsigned long long* red, uint32_t* mx, uint32_t* mn) {
  unsigned long long a = 0, b = 0;
  for (int i = threadIdx.x; i < n; i += kST) {
    const unsigned long long k = ckey[i];
    a = k > a ? k : a;
    const unsigned long long nk = ~static_cast<uint32_t>(ckey[i]);
    b = nk > b ? nk : b;
  }
  a = sblock_max_u64(a, red);
  b = sblock_max_u64(b, red);
  *mx = static_cast<uint32_t>(a);
  *mn = ~static_cast<uint32_t>(b);
}

// First bin whose cumulative weight (from bin 0) reaches tau (nb a multiple of kST);
// thread t owns nb/kST consecutive bins.  Returns -1 if none.  *above: weight before it.
template <class H>
__device__ int sfind_bin(const H& h, unsigned long long tau, unsigned long long* red,
                         unsigned long long* misc, unsigned long long* above) {
  const int per = h.nb / kST;
  unsigned long long part = 0;
  for (int e = 0; e < per; ++e) part += h.get(per * threadIdx.x + e);
  unsigned long long S;
  const unsigned long long ex = sblock_excl_scan_u64(part, &S, red);
  if (threadIdx.x == 0) misc[8] = ~0ull;
  csync();
  if (ex < tau && ex + part >= tau) {
    unsigned long long acc = ex;
    for (int e = 0; e < per; ++e) {
      const unsigned long long w = h.get(per * threadIdx.x + e);
      if (acc + w >= tau) {
        misc[8] = static_cast<unsigned long long>(per * threadIdx.x + e);
        misc[9] = acc;
        break;
      }
      acc += w;
    }
  }
  csync();
  const unsigned long long b = misc[8];
  *above = misc[9];
  csync();
  return b == ~0ull ? -1 : static_cast<int>(b);
}

// A value threshold that keeps at least k buffer entries, tight to one linear bin of the
// buffer's range: returns (key, INT_MAX), i.e. "key >= threshold key".
__device__ Thresh scut_value(const uint32_t* ckey, int n, uint32_t k, unsigned long long* hist,
                             unsigned long long* red, unsigned long long* misc) {
  uint32_t mx, mn;
  sbuf_range(ckey, n, red, &mx, &mn);
  if (mx == mn) return Thresh{mn, INT_MAX};
  const float hi = kfloat(mx);
  const float s = sbin_scale(hi, kfloat(mn));
  if (!(s > 0.0f)) return Thresh{mn, INT_MAX};
  const Bins<1> hb{reinterpret_cast<uint32_t*>(hist), kLinBins};
  hb.clear(kST);
  csync();
  for (int i = threadIdx.x; i < n; i += kST) hb.add(sbin(kfloat(ckey[i]), hi, s), 1ull);
  csync();
  unsigned long long above;
  const int beta = sfind_bin(hb, k, red, misc, &above);
  if (beta < 0) return Thresh{mn, INT_MAX};
  unsigned long long b = 0;  // max of ~key over the kept bins = the smallest kept key
  for (int i = threadIdx.x; i < n; i += kST)
    if (sbin(kfloat(ckey[i]), hi, s) <= beta) {
      const unsigned long long nk = ~ckey[i];
      b = nk > b ? nk : b;
    }
  b = sblock_max_u64(b, red);
  return Thresh{~static_cast<uint32_t>(b), INT_MAX};
}

// Exact k-th entry (value desc, index asc) of the buffer: the bin holding it from a
// linear-bin count histogram, then pairwise ranking of that bin's entries; the radix
// select when the bin is large.
__device__ Thresh sexact_kth(const uint32_t* ckey, const int32_t* cidx, int n, uint32_t k,
                             unsigned long long* hist, unsigned long long* kbuf, unsigned long long* red,
                             unsigned long long* misc, uint32_t& s_cnt, Thresh& s_th) {
  uint32_t mx, mn;
  sbuf_range(ckey, n, red, &mx, &mn);
  const float hi = kfloat(mx);
  const float s = mx == mn ? 0.0f : sbin_scale(hi, kfloat(mn));
  if (s > 0.0f) {
    const Bins<1> hb{reinterpret_cast<uint32_t*>(hist), kLinBins};
    hb.clear(kST);
    csync();
    for (int i = threadIdx.x; i < n; i += kST) hb.add(sbin(kfloat(ckey[i]), hi, s), 1ull);
    csync();
    unsigned long long above;
    const int beta = sfind_bin(hb, k, red, misc, &above);
    if (beta >= 0 && hb.get(beta) <= static_cast<unsigned long long>(kSRank)) {
      if (threadIdx.x == 0) { s_cnt = 0u; misc[10] = 0ull; }
      csync();
      for (int i = threadIdx.x; i < n; i += kST)
        if (sbin(kfloat(ckey[i]), hi, s) == beta) kbuf[atomicAdd(&s_cnt, 1u)] = order_word(ckey[i], cidx[i]);
      csync();
      const int m = static_cast<int>(s_cnt);
      const unsigned long long want = k - above - 1;  // entries of the bin that come before it
      for (int i = threadIdx.x; i < m; i += kST) {
        const unsigned long long wi = kbuf[i];
        unsigned long long r = 0;
        for (int j = 0; j < m; ++j) r += kbuf[j] > wi ? 1ull : 0ull;
        if (r == want) {
          s_th = Thresh{static_cast<uint32_t>(wi >> 32), static_cast<int32_t>(~static_cast<uint32_t>(wi))};
          misc[10] = 1ull;
        }
      }
      csync();
      const bool ok = misc[10] != 0ull;
      const Thresh t = s_th;
      csync();
      if (ok) return t;
    }
  }
  return sblock_topk_threshold(ckey, cidx, n, k, reinterpret_cast<uint32_t*>(hist), misc, red);
}

// Top-p inside the k survivors held in the buffer (maximum M, k-th value xk): mass
// histogram over linear bins of [xk, M], then an exact prefix over the boundary bin's
// entries.  Returns false when that bin is large (the caller sorts instead).
__device__ bool stopp_small(const uint32_t* ckey, const int32_t* cidx, int n, float M, float xk, float p,
                            unsigned long long* hist, unsigned long long* kbuf, unsigned long long* red,
                            unsigned long long* misc, uint32_t& s_cnt, Thresh& s_th, Thresh* out) {
  const float s = sbin_scale(M, xk);
  const Bins<3> hm{reinterpret_cast<uint32_t*>(hist), 1024};  // sbin / 2: 1024 bins
  hm.clear(kST);
  csync();
  for (int i = threadIdx.x; i < n; i += kST) {
    const float y = kfloat(ckey[i]);
    const unsigned long long w = fixed_mass(softmax_weight(y, M));
    if (w) hm.add(s > 0.0f ? (sbin(y, M, s) >> 1) : 0, w);
  }
  csync();
  unsigned long long S = 0;
  {
    unsigned long long part = 0;
    for (int e = 0; e < 1024 / kST; ++e) part += hm.get((1024 / kST) * threadIdx.x + e);
    S = sblock_sum_u64(part, red);
  }
  const double td = ceil(static_cast<double>(p) * static_cast<double>(S));
  unsigned long long tq = static_cast<unsigned long long>(td);
  if (tq < 1ull) tq = 1ull;
  if (tq > S) tq = S;
  unsigned long long above;
  const int beta = sfind_bin(hm, tq, red, misc, &above);
  if (beta < 0) return false;
  if (threadIdx.x == 0) { s_cnt = 0u; misc[10] = 0ull; }
  csync();
  for (int i = threadIdx.x; i < n; i += kST)
    if ((s > 0.0f ? (sbin(kfloat(ckey[i]), M, s) >> 1) : 0) == beta) {
      const uint32_t pos = atomicAdd(&s_cnt, 1u);
      if (pos < static_cast<uint32_t>(kSRank)) kbuf[pos] = order_word(ckey[i], cidx[i]);
    }
  csync();
  const int m = static_cast<int>(s_cnt);
  if (m > kSRank) {
    csync();
    return false;
  }
  const unsigned long long need = tq - above;
  for (int i = threadIdx.x; i < m; i += kST) {
    const unsigned long long wi = kbuf[i];
    const unsigned long long self = fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(wi >> 32)), M));
    unsigned long long ex = 0;
    for (int j = 0; j < m; ++j)
      if (kbuf[j] > wi) ex += fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(kbuf[j] >> 32)), M));
    if (ex < need && need <= ex + self) {
      s_th = Thresh{static_cast<uint32_t>(wi >> 32), static_cast<int32_t>(~static_cast<uint32_t>(wi))};
      misc[10] = 1ull;
    }
  }
  csync();
  const bool ok = misc[10] != 0ull;
  *out = s_th;
  csync();
  return ok;
}

template <bool kBF16>
__global__ void __launch_bounds__(kSThreads, 1) kps_stream_kernel(const Params P, const int stages) {
  extern __shared__ __align__(16) unsigned char s_smem[];
  unsigned char* smem = s_smem;
  const SLayout L = make_slayout(P.V, kBF16, stages);
  unsigned char* ring = smem + L.ring;
  uint32_t* ckey = reinterpret_cast<uint32_t*>(smem + L.ckey);
  int32_t* cidx = reinterpret_cast<int32_t*>(smem + L.cidx);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L.bitmap);
  unsigned long long* hist = reinterpret_cast<unsigned long long*>(smem + L.hist);
  unsigned long long* kbuf = reinterpret_cast<unsigned long long*>(smem + L.kbuf);
  unsigned long long* red = reinterpret_cast<unsigned long long*>(smem + L.red);
  unsigned long long* misc = reinterpret_cast<unsigned long long*>(smem + L.misc);
  unsigned long long* full = reinterpret_cast<unsigned long long*>(smem + L.bars);
  unsigned long long* empty = full + stages;
  uint32_t& s_cnt = *reinterpret_cast<uint32_t*>(misc + 16);
  Thresh& s_th = *reinterpret_cast<Thresh*>(misc + 17);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const int64_t V = P.V;
  const size_t esize = kBF16 ? 2 : 4;
  const int nch = static_cast<int>((V + kStageElems - 1) / kStageElems);  // chunks per row

  // the rows this CTA owns (built by all threads, producer included)
  int32_t* rowlist = reinterpret_cast<int32_t*>(smem + L.rows);
  int my_rows = 0;
  if (P.filter == 0) {
    my_rows = P.B > blockIdx.x ? static_cast<int>((P.B - 1 - blockIdx.x) / gridDim.x + 1) : 0;
  } else {
    my_rows = build_row_list<kSThreads>(P, blockIdx.x, gridDim.x, rowlist, red);
  }
  auto row_at = [&](int i) -> int64_t {
    return P.filter == 0 ? static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(i) * gridDim.x
                         : static_cast<int64_t>(rowlist[i]);
  };
  if (threadIdx.x == 0)
    for (int q = 0; q < stages; ++q) {
      mbar_init(full + q, 1);
      mbar_init(empty + q, kSW);
    }
  for (int w = threadIdx.x; w < (V + 31) / 32; w += kSThreads) bitmap[w] = 0u;
  __syncthreads();

  if (warp == kSW) {
    // ---- producer warp: one lane streams every chunk of every owned row -----------------
    if (lane == 0) {
      int st = 0;
      uint32_t rnd = 0;  // how many times the ring has wrapped
      for (int ri = 0; ri < my_rows; ++ri) {
        const unsigned char* src = static_cast<const unsigned char*>(P.logits) + row_at(ri) * V * esize;
        for (int c = 0; c < nch; ++c) {
          if (rnd > 0 && !mbar_wait_bounded(empty + st, (rnd - 1) & 1u)) atomicMax(P.status, kStatusTimeout);
          const int64_t off = static_cast<int64_t>(c) * kStageElems;
          const int64_t cnt = V - off < kStageElems ? V - off : kStageElems;
          const uint32_t bytes = static_cast<uint32_t>(cnt * esize);
          mbar_expect_tx(full + st, bytes);
          bulk_g2s(ring + st * L.stage_bytes, src + off * esize, bytes, full + st);
          if (++st == stages) {
            st = 0;
            ++rnd;
          }
        }
      }
    }
    return;
  }

  // ---- consumer warps ---------------------------------------------------------------------
  bool timed_out = false;
  int cs = 0;           // stage of the next chunk
  uint32_t cpar = 0;    // and the phase parity it completes with
  for (int ri = 0; ri < my_rows; ++ri) {
    const int64_t row = row_at(ri);
    const int32_t k = P.top_k[row];
    const float p = P.top_p[row];
    const float T = P.temperature[row];
    const bool greedyT = !(T > 0.0f) || isinf(T);
    const bool pen_on = P.seen_indptr && P.seen_ids && P.penalty && (P.penalty[row] > 0.0f);
    const float pen = pen_on ? P.penalty[row] : 1.0f;
    const bool topk_on = k >= 1 && static_cast<int64_t>(k) <= (V < kTopKMax ? V : kTopKMax);
    const bool p_nan = isnan(p);
    const bool single = greedyT || (!p_nan && p <= 0.0f) || (topk_on && k == 1);
    const bool topp_on = !single && !p_nan && p > 0.0f && p < 1.0f;
    const bool kmode = single || topk_on;
    const uint32_t keff = single ? 1u : static_cast<uint32_t>(k);
    const bool identity = greedyT;  // no division on greedy rows
    float* orow = P.need_logits ? P.out_filtered + row * V : nullptr;
    const float* qrow = P.q + row * V;

    // penalty bitmap for this row
    int32_t b0 = 0, b1 = 0;
    if (pen_on) {
      b0 = P.seen_indptr[row];
      b1 = P.seen_indptr[row + 1];
      for (int32_t t = b0 + threadIdx.x; t < b1; t += kST) {
        const int32_t id = P.seen_ids[t];
        if (id >= 0 && static_cast<int64_t>(id) < V) atomicOr(&bitmap[id >> 5], 1u << (id & 31));
      }
    }
    if (threadIdx.x == 0) s_cnt = 0u;
    csync();

    // running threshold of k mode (keeps every real element until the first cut)
    Thresh tau{0u, -1};
    float tau_raw = -INFINITY;
    uint32_t rawmax = 0;  // top-p-only / keep-all rows: max key of the penalised row

    // ---- the ring pass ---------------------------------------------------------------
    for (int c = 0; c < nch; ++c) {
      const int s = cs;
      const uint32_t parity = cpar;
      if (++cs == stages) {
        cs = 0;
        cpar ^= 1u;
      }
      if (!mbar_wait_bounded(full + s, parity)) {
        timed_out = true;
        if (threadIdx.x == 0) atomicMax(P.status, kStatusTimeout);
      }
      const int off = c * kStageElems;
      const int cnt = static_cast<int>(V - off < kStageElems ? V - off : kStageElems);
      float vv[kSPer][4];
#pragma unroll
      for (int u = 0; u < kSPer; ++u) {
        const int q4 = u * kST + threadIdx.x;  // float4 index within the stage
        if (4 * q4 < cnt) {
          if (kBF16) {
            const uint2 w = reinterpret_cast<const uint2*>(ring + s * L.stage_bytes)[q4];
            vv[u][0] = __uint_as_float(w.x << 16);
            vv[u][1] = __uint_as_float(w.x & 0xFFFF0000u);
            vv[u][2] = __uint_as_float(w.y << 16);
            vv[u][3] = __uint_as_float(w.y & 0xFFFF0000u);
          } else {
            const float4 w = reinterpret_cast<const float4*>(ring + s * L.stage_bytes)[q4];
            vv[u][0] = w.x; vv[u][1] = w.y; vv[u][2] = w.z; vv[u][3] = w.w;
          }
        } else {
          vv[u][0] = vv[u][1] = vv[u][2] = vv[u][3] = 0.0f;
        }
      }
      // the stage is in registers: hand it back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
#pragma unroll
      for (int u = 0; u < kSPer; ++u) {
        const int e0 = 4 * (u * kST + threadIdx.x);
        const uint32_t bits = (pen_on && e0 < cnt) ? (bitmap[(off + e0) >> 5] >> (e0 & 31)) & 0xFu : 0u;
        if (__any_sync(kFull, bits != 0u)) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if ((bits >> e) & 1u) vv[u][e] = (vv[u][e] > 0.0f) ? __fdiv_rn(vv[u][e], pen) : __fmul_rn(vv[u][e], pen);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) vv[u][e] = isnan(vv[u][e]) ? -INFINITY : vv[u][e];
        if (kmode) {
          if (orow && e0 < cnt) {
            if (e0 + 4 <= cnt) {
              __stcs(reinterpret_cast<float4*>(orow + off + e0), make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY));
            } else {
              for (int e = 0; e < 4; ++e)
                if (e0 + e < cnt) orow[off + e0 + e] = -INFINITY;
            }
          }
          bool pass[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pass[e] = (e0 + e < cnt) && vv[u][e] >= tau_raw;
          if (__any_sync(kFull, pass[0] || pass[1] || pass[2] || pass[3])) {
            uint32_t ck[4] = {0u, 0u, 0u, 0u};
            uint32_t ncand = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (!pass[e]) continue;
              const float y = __fadd_rn(identity ? vv[u][e] : __fdiv_rn(vv[u][e], T), 0.0f);
              const uint32_t ky = fkey(y);
              if (kept_by(ky, off + e0 + e, tau.key, tau.idx)) {
                ck[e] = ky;
                ++ncand;
              }
            }
            const uint32_t incl = warp_incl_scan_u32(ncand, lane);
            const uint32_t wtot = __shfl_sync(kFull, incl, 31);
            if (wtot) {
              uint32_t wb = 0;
              if (lane == 31) wb = atomicAdd(&s_cnt, wtot);
              wb = __shfl_sync(kFull, wb, 31);
              uint32_t pos = wb + incl - ncand;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (ck[e]) {
                  if (pos < static_cast<uint32_t>(kSCap)) {
                    ckey[pos] = ck[e];
                    cidx[pos] = off + e0 + e;
                  }
                  ++pos;
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (e0 + e >= cnt) continue;
            const uint32_t kx = fkey(__fadd_rn(vv[u][e], 0.0f));
            rawmax = kx > rawmax ? kx : rawmax;
          }
        }
      }
      csync();  // every warp has appended: the buffer count is final
      if (kmode && s_cnt > static_cast<uint32_t>(kSHigh)) {
        // cut the buffer to a value threshold that keeps >= k entries (one linear bin of
        // slack); if equal values keep it too full, cut exactly to the top k
        const int n = static_cast<int>(s_cnt < static_cast<uint32_t>(kSCap) ? s_cnt : kSCap);
        Thresh t = scut_value(ckey, n, keff, hist, red, misc);
        int nn = sblock_compact(ckey, cidx, n, t, red);
        if (nn > kSHigh) {
          t = sblock_topk_threshold(ckey, cidx, nn, keff, reinterpret_cast<uint32_t*>(hist), misc, red);
          nn = sblock_compact(ckey, cidx, nn, t, red);
        }
        // a later element is kept only if it is kept by t (later indices lose ties)
        tau = t;
        if (threadIdx.x == 0) s_cnt = static_cast<uint32_t>(nn);
        tau_raw = raw_floor(kfloat(tau.key), T, identity);
        csync();
      }
    }

    int32_t chosen = -1;
    if (kmode) {
      // ---- exact top-k of the buffer, top-p inside it, race ---------------------
      int n = static_cast<int>(s_cnt < static_cast<uint32_t>(kSCap) ? s_cnt : kSCap);
      const Thresh tk = sexact_kth(ckey, cidx, n, keff, hist, kbuf, red, misc, s_cnt, s_th);
      n = sblock_compact(ckey, cidx, n, tk, red);  // exactly keff entries
      uint32_t mx, mn;
      sbuf_range(ckey, n, red, &mx, &mn);
      const float M = kfloat(mx);
      Thresh th = tk;
      if (topp_on && n > 1) {
        Thresh tp;
        if (stopp_small(ckey, cidx, n, M, kfloat(tk.key), p, hist, kbuf, red, misc, s_cnt, s_th, &tp)) {
          th = tp;
        } else {
          // large boundary bin: sort the survivors and cut the exact prefix
          int N = 2;
          while (N < n) N <<= 1;
          for (int t = threadIdx.x; t < N; t += kST) kbuf[t] = t < n ? order_word(ckey[t], cidx[t]) : 0ull;
          csync();
          for (int kk = 2; kk <= N; kk <<= 1) {
            for (int jj = kk >> 1; jj > 0; jj >>= 1) {
              for (int t = threadIdx.x; t < (N >> 1); t += kST) {
                const int a = 2 * t - (t & (jj - 1));
                const int b = a + jj;
                const unsigned long long x = kbuf[a], y = kbuf[b];
                const bool desc = (a & kk) == 0;
                if (desc ? (x < y) : (x > y)) {
                  kbuf[a] = y;
                  kbuf[b] = x;
                }
              }
              csync();
            }
          }
          const int t0 = 2 * threadIdx.x, t1 = t0 + 1;  // n <= 1024 = 2 * kST
          const unsigned long long e0 =
              t0 < n ? fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(kbuf[t0] >> 32)), M)) : 0ull;
          const unsigned long long e1 =
              t1 < n ? fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(kbuf[t1] >> 32)), M)) : 0ull;
          unsigned long long S;
          const unsigned long long ex = sblock_excl_scan_u64(e0 + e1, &S, red);
          const double td = ceil(static_cast<double>(p) * static_cast<double>(S));
          unsigned long long tq = static_cast<unsigned long long>(td);
          if (tq < 1ull) tq = 1ull;
          if (tq > S) tq = S;
          if (threadIdx.x == 0) misc[11] = static_cast<unsigned long long>(n - 1);
          csync();
          if (t0 < n && ex < tq && ex + e0 >= tq) misc[11] = static_cast<unsigned long long>(t0);
          if (t1 < n && ex + e0 < tq && ex + e0 + e1 >= tq) misc[11] = static_cast<unsigned long long>(t1);
          csync();
          const unsigned long long w = kbuf[misc[11]];
          th = Thresh{static_cast<uint32_t>(w >> 32), static_cast<int32_t>(~static_cast<uint32_t>(w))};
          csync();
        }
      }
      // race over the kept survivors (q gathered at their indices)
      unsigned long long rb = 0, first = 0;
      for (int t = threadIdx.x; t < n; t += kST) {
        const uint32_t key = ckey[t];
        const int32_t idx = cidx[t];
        if (!kept_by(key, idx, th.key, th.idx)) continue;
        const unsigned long long ow = order_word(key, idx);
        first = ow > first ? ow : first;
        const float w = softmax_weight(kfloat(key), M);
        const float r = __fdiv_rn(w, __fadd_rn(__ldg(qrow + idx), P.eps));
        if (isnan(r)) continue;
        const unsigned long long cand = order_word(fkey(r), idx);
        rb = cand > rb ? cand : rb;
      }
      rb = sblock_max_u64(rb, red);
      first = sblock_max_u64(first, red);
      chosen = rb ? static_cast<int32_t>(~static_cast<uint32_t>(rb)) : static_cast<int32_t>(~static_cast<uint32_t>(first));
      // kept values over the -inf output streamed during the pass
      if (orow)
        for (int t = threadIdx.x; t < n; t += kST)
          if (kept_by(ckey[t], cidx[t], th.key, th.idx)) orow[cidx[t]] = kfloat(ckey[t]);
    } else {
      // ---- rows without top-k: the ring pass gave the maximum -------------------
      const unsigned long long mx = sblock_max_u64(rawmax, red);
      const float Mraw = kfloat(static_cast<uint32_t>(mx));
      const float M = __fadd_rn(identity ? Mraw : __fdiv_rn(Mraw, T), 0.0f);
      Thresh th{0u, -1};  // keep everything
      if (topp_on) {
        // mass histogram over linear bins of (M - y)
        for (int t = threadIdx.x; t < kLinBins; t += kST) hist[t] = 0ull;
        csync();
        srow_pass<kBF16>(P, row, bitmap, pen_on, pen, T, identity, [&](bool valid, float y, uint32_t, int) {
          if (!valid) return;
          const int b = lin_bin_mass(y, M);
          if (b < kLinBins) {
            const unsigned long long w = fixed_mass(softmax_weight(y, M));
            if (w) atomicAdd(&hist[b], w);
          }
        });
        csync();
        // boundary bin over the 2048 linear bins
        unsigned long long S = 0;
        {
          unsigned long long part = 0;
          for (int e = 0; e < kLinBins / kST; ++e) part += hist[(kLinBins / kST) * threadIdx.x + e];
          S = sblock_sum_u64(part, red);
        }
        const double td = ceil(static_cast<double>(p) * static_cast<double>(S));
        unsigned long long tq = static_cast<unsigned long long>(td);
        if (tq < 1ull) tq = 1ull;
        if (tq > S) tq = S;
        unsigned long long above1 = 0;
        const int b1i = sfind_bin(U64Bins{hist, kLinBins}, tq, red, misc, &above1);
        const unsigned long long beta1 = b1i < 0 ? ~0ull : static_cast<unsigned long long>(b1i);
        bool ok = beta1 != ~0ull;
        if (ok) {
          // finer bins inside beta1, collecting its elements
          const int bb = static_cast<int>(beta1);
          for (int t = threadIdx.x; t < kFineBins; t += kST) kbuf[t] = 0ull;
          if (threadIdx.x == 0) s_cnt = 0u;
          csync();
          srow_pass<kBF16>(P, row, bitmap, pen_on, pen, T, identity, [&](bool valid, float y, uint32_t key, int v) {
            const bool take = valid && lin_bin_mass(y, M) == bb;
            if (take) {
              const unsigned long long w = fixed_mass(softmax_weight(y, M));
              if (w) atomicAdd(&kbuf[fine_bin_mass(y, M, bb)], w);
            }
            const unsigned m = __ballot_sync(kFull, take);
            if (!m) return;
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(&s_cnt, static_cast<uint32_t>(__popc(m)));
            base = __shfl_sync(kFull, base, 0);
            if (take) {
              const uint32_t pos = base + __popc(m & ((1u << lane) - 1u));
              if (pos < static_cast<uint32_t>(kSCap)) {
                ckey[pos] = key;
                cidx[pos] = v;
              }
            }
          });
          csync();
          const int nb1 = static_cast<int>(s_cnt);
          ok = nb1 <= kSCap;
          if (ok) {
            const unsigned long long tq2 = tq - above1;
            unsigned long long above2 = 0;
            const int b2i = sfind_bin(U64Bins{kbuf, kFineBins}, tq2, red, misc, &above2);
            const unsigned long long beta2 = b2i < 0 ? ~0ull : static_cast<unsigned long long>(b2i);
            const unsigned long long tq3 = tq2 - above2;
            ok = beta2 != ~0ull;
            if (ok) {
              // rank the elements of the final bin: the one whose exclusive prefix mass
              // (in the order) is < tq3 <= prefix + own mass ends the kept prefix
              uint32_t nsm = 0;
              for (int t = threadIdx.x; t < nb1; t += kST)
                if (fine_bin_mass(kfloat(ckey[t]), M, bb) == static_cast<int>(beta2)) ++nsm;
              nsm = static_cast<uint32_t>(sblock_sum_u64(nsm, red));
              ok = nsm <= static_cast<uint32_t>(kSRank);
              if (ok) {
                // gather the final bin into kbuf (the fine histogram is no longer needed)
                if (threadIdx.x == 0) s_cnt = 0u;
                csync();
                for (int t = threadIdx.x; t < nb1; t += kST)
                  if (fine_bin_mass(kfloat(ckey[t]), M, bb) == static_cast<int>(beta2)) {
                    const uint32_t pos = atomicAdd(&s_cnt, 1u);
                    kbuf[pos] = order_word(ckey[t], cidx[t]);
                  }
                csync();
                const int nr = static_cast<int>(s_cnt);
                if (threadIdx.x == 0) { misc[10] = 0ull; s_th = Thresh{0u, -1}; }
                csync();
                for (int t = threadIdx.x; t < nr; t += kST) {
                  const unsigned long long wi = kbuf[t];
                  const unsigned long long self =
                      fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(wi >> 32)), M));
                  unsigned long long exm = 0;
                  for (int u = 0; u < nr; ++u)
                    if (kbuf[u] > wi) exm += fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(kbuf[u] >> 32)), M));
                  if (exm < tq3 && tq3 <= exm + self) {
                    s_th = Thresh{static_cast<uint32_t>(wi >> 32), static_cast<int32_t>(~static_cast<uint32_t>(wi))};
                    misc[10] = 1ull;
                  }
                }
                csync();
                ok = misc[10] != 0ull;
                th = s_th;
                csync();
              }
            }
          }
        }
        if (!ok)
          th = srow_mass_select<kBF16>(P, row, bitmap, pen_on, pen, T, identity, M, p,
                                       reinterpret_cast<uint32_t*>(hist), hist, misc, red);
      }
      // race over the kept set and the filtered output, one more pass
      unsigned long long rb = 0;
      srow_pass<kBF16>(P, row, bitmap, pen_on, pen, T, identity, [&](bool valid, float y, uint32_t key, int v) {
        const bool kp = valid && kept_by(key, v, th.key, th.idx);
        if (valid && orow) orow[v] = kp ? y : -INFINITY;
        if (!kp) return;
        const float w = softmax_weight(y, M);
        const float r = __fdiv_rn(w, __fadd_rn(__ldcs(qrow + v), P.eps));
        if (isnan(r)) return;
        const unsigned long long cand = order_word(fkey(r), v);
        rb = cand > rb ? cand : rb;
      });
      rb = sblock_max_u64(rb, red);
      if (rb) {
        chosen = static_cast<int32_t>(~static_cast<uint32_t>(rb));
      } else {
        // every score was NaN: the first element of the order
        unsigned long long fb = 0;
        srow_pass<kBF16>(P, row, bitmap, pen_on, pen, T, identity, [&](bool valid, float, uint32_t key, int v) {
          if (valid && kept_by(key, v, th.key, th.idx)) {
            const unsigned long long w = order_word(key, v);
            fb = w > fb ? w : fb;
          }
        });
        fb = sblock_max_u64(fb, red);
        chosen = static_cast<int32_t>(~static_cast<uint32_t>(fb));
      }
    }
    if (threadIdx.x == 0) P.out_idx[row] = chosen;
    // clear this row's penalty bits
    csync();
    if (pen_on)
      for (int32_t t = b0 + threadIdx.x; t < b1; t += kST) {
        const int32_t id = P.seen_ids[t];
        if (id >= 0 && static_cast<int64_t>(id) < V) bitmap[id >> 5] = 0u;
      }
    csync();
  }
  // every chunk the producer issued has been consumed (waited on) above; nothing is in flight
  (void)timed_out;
}
