// kps.cu — GB300 (sm_103a) kernels and C ABI for the decode-step sampler.
//
// One thread-block cluster owns one row of the [B, V] logits matrix.  The row
// is split into CS contiguous chunks, one per CTA; each chunk is staged into
// shared memory with a TMA bulk copy (cp.async.bulk + mbarrier) and stays
// there for the whole row, so logits are read from HBM exactly once.  All
// selection steps then run on shared memory, and the CTAs combine their
// partial results through distributed shared memory (DSMEM) and cluster
// barriers:
//
//   load  -> penalty (scatter over the seen ids, once per distinct id)
//         -> temperature (x / T, IEEE) and the row maximum
//         -> top-k: exact radix select of the k-th element in the order
//            (value desc, index asc) — 4 passes of 8-bit digits over
//            order-preserving uint32 keys, count histograms
//         -> top-p: the same radix select weighted by softmax mass, held
//            in 2^-40 fixed point so the sums are exact and order-free
//         -> exponential race: argmax of e / (q + eps) over the kept set
//         -> filtered logits written back in vocabulary order.
//
// The method follows the Ascend "torch_npu.npu_top_k_top_p_sample" page
// (topK valid range, topP full-sort rule, Sample formulas), MiniMind
// "Chapter 10: inference generation" (§10.4 temperature, §10.5 top-k, §10.6
// top-p, §10.7 repetition penalty) and the C++ post-processing blog
// (penalty over the set of seen ids, softmax).  Selection is by radix
// histograms rather than the sorts and quickselects on those pages.
//
// Nothing here waits without a bound: the TMA wait gives up after ~2 s of
// clock cycles, records KPS_ERR_TIMEOUT in the status word and carries on
// with the same control flow, so the cluster barriers always complete.

#include "kps.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cooperative_groups.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

namespace cg = cooperative_groups;

namespace kps {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;          // 8-bit radix digits
constexpr int kSuper = 16;          // super-bins of 16 bins each
constexpr int kTopKMax = 1024;      // top-k is active for 1 <= k <= min(V, 1024)
constexpr float kFixScale = 1099511627776.0f;  // 2^40: fixed-point unit of softmax mass
constexpr long long kSpinCycles = 4000000000LL;  // bounded wait (~2 s)
constexpr int kSmemCap2PerSM = 110 * 1024;  // per-CTA budget for two CTAs per SM
constexpr unsigned kFull = 0xffffffffu;
constexpr int kStatusTimeout = KPS_ERR_TIMEOUT;

// Cluster exchange slots (u64 each) in shared memory.
enum Slot { kSlotMax = 0, kSlotRace = 1, kSlotTie = 2, kNumSlots = 4 };

struct Params {
  const void* logits;
  int64_t B, V;
  const int32_t* top_k;
  const float* top_p;
  const float* temperature;
  const int32_t* seen_indptr;
  const int32_t* seen_ids;
  const float* penalty;
  const float* q;
  float eps;
  int need_logits;
  int64_t* out_idx;
  float* out_filtered;
  int* status;
  int nc;       // elements per CTA (multiple of 8)
  int use_tma;  // every row starts on a 16-byte boundary
};

// ------------------------------------------------------------------------------------------
// Shared-memory layout (identical on host and device).
// ------------------------------------------------------------------------------------------
struct Layout {
  size_t xs, raw, bitmap, hist, sup, red, slots, mbar, misc, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline Layout make_layout(int nc, bool bf16) {
  Layout L;
  size_t off = 0;
  L.xs = off;     off += align16(size_t(nc) * 4);
  L.raw = off;    off += bf16 ? align16(size_t(nc) * 2) : 0;
  L.bitmap = off; off += align16(size_t((nc + 31) / 32) * 4);
  L.hist = off;   off += 2 * kBins * 8;
  L.sup = off;    off += 2 * kSuper * 8;
  L.red = off;    off += 40 * 8;
  L.slots = off;  off += kNumSlots * 8;
  L.mbar = off;   off += 16;
  L.misc = off;   off += 16 * 8;
  L.total = off;
  return L;
}

// ------------------------------------------------------------------------------------------
// Small device helpers
// ------------------------------------------------------------------------------------------

// Order-preserving map float -> uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t u = __float_as_uint(x);
  return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
}
__device__ __forceinline__ float kfloat(uint32_t k) {
  uint32_t u = k ^ ((k & 0x80000000u) ? 0x80000000u : 0xFFFFFFFFu);
  return __uint_as_float(u);
}

// Kept test for a threshold (tk, ti) in the order (value desc, index asc).
__device__ __forceinline__ bool kept_by(uint32_t key, int32_t idx, uint32_t tk, int32_t ti) {
  return key > tk || (key == tk && idx <= ti);
}

// Softmax weight exp(x - M) in fp32.  The difference x - M is carried exactly
// as hi + lo (Knuth's TwoSum) and the exponential is corrected to first order,
// e * (1 + lo), so the weight does not inherit the rounding of the subtraction.
// x == M gives exactly 1 (which keeps +-inf maxima finite).
__device__ __forceinline__ float softmax_weight(float x, float M) {
  if (x == M) return 1.0f;
  float s = __fsub_rn(x, M);
  if (!(s > -INFINITY)) return 0.0f;
  float bb = __fsub_rn(s, x);
  float lo = __fadd_rn(__fsub_rn(x, __fsub_rn(s, bb)), __fsub_rn(-M, bb));
  float e = expf(s);
  return __fmaf_rn(e, lo, e);
}
__device__ __forceinline__ unsigned long long fixed_mass(float w) {
  return __float2ull_rn(w * kFixScale);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: returns false if the phase did not complete within kSpinCycles.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kSpinCycles) return false;
  }
  return true;
}
// Bulk global -> shared copy completing on an mbarrier (addresses 16-byte aligned,
// size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(kFull, v, o);
    v = w > v ? w : v;
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
// Inclusive prefix sum across the warp.
__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned long long w = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += w;
  }
  return v;
}

// Block-wide max of a u64; every thread gets the result.
__device__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_u64(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kWarps ? red[lane] : 0ull;
    v = warp_max_u64(v);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  v = red[32];
  __syncthreads();
  return v;
}

// Cluster-wide max of a u64 through one exchange slot; every thread gets it.
__device__ unsigned long long cluster_max_u64(cg::cluster_group& cl, unsigned long long local,
                                              unsigned long long* slot, unsigned long long* bcast) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int CS = static_cast<int>(cl.num_blocks());
  if (threadIdx.x == 0) *slot = local;
  cl.sync();
  if (warp == 0) {
    unsigned long long v = 0;
    for (int r = lane; r < CS; r += 32) {
      unsigned long long w = *cl.map_shared_rank(slot, r);
      v = w > v ? w : v;
    }
    v = warp_max_u64(v);
    if (lane == 0) *bcast = v;
  }
  __syncthreads();
  return *bcast;
}

// ------------------------------------------------------------------------------------------
// Per-CTA context for one row
// ------------------------------------------------------------------------------------------
struct Ctx {
  float* xs;            // transformed values of this CTA's chunk
  int32_t c0;           // row index of xs[0]
  int n;                // elements in this chunk
  int n4;               // float4 groups covering the chunk (tail padded with key 0)
  float M;              // row maximum (transformed)
  unsigned long long* hist;  // [2][kBins]
  unsigned long long* sup;   // [2][kSuper]
  unsigned long long* red;
  unsigned long long* slots;
  unsigned long long* misc;
};

// Result of a radix select: the last kept element's key and index.
struct Thresh {
  uint32_t key;
  int32_t idx;
};

// Block-wide exclusive scan of small counts; returns the exclusive prefix, *total gets the sum.
__device__ uint32_t block_excl_scan_u32(uint32_t v, uint32_t* total, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t w = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += w;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < kWarps ? static_cast<uint32_t>(red[lane]) : 0u;
    uint32_t t = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t w = __shfl_up_sync(kFull, t, o);
      if (lane >= o) t += w;
    }
    if (lane < kWarps) red[lane] = t - s;  // exclusive prefix of warp totals
    if (lane == kWarps - 1) red[32] = t;
  }
  __syncthreads();
  uint32_t res = static_cast<uint32_t>(red[warp]) + x - v;
  *total = static_cast<uint32_t>(red[32]);
  __syncthreads();
  return res;
}

// Finds, in index order, the j-th (1-based) element of this CTA's chunk with
// key == tkey that is kept by (rk, ri).  Returns its row index, or -1.
__device__ int32_t local_nth_tie(const Ctx& c, uint32_t tkey, uint32_t rk, int32_t ri, uint32_t j) {
  int32_t* found = reinterpret_cast<int32_t*>(c.misc + 8);
  if (threadIdx.x == 0) *found = -1;
  __syncthreads();
  for (int base = 0; base < c.n4; base += kThreads) {
    const int g = base + threadIdx.x;
    uint32_t cnt = 0;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (g < c.n4) {
      v = reinterpret_cast<const float4*>(c.xs)[g];
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t key = fkey(vv[e]);
        const int32_t gi = c.c0 + 4 * g + e;
        cnt += (key == tkey && key != 0 && kept_by(key, gi, rk, ri)) ? 1u : 0u;
      }
    }
    uint32_t total;
    const uint32_t excl = block_excl_scan_u32(cnt, &total, c.red);
    if (cnt && excl < j && j <= excl + cnt) {
      const float vv[4] = {v.x, v.y, v.z, v.w};
      uint32_t seen = excl;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t key = fkey(vv[e]);
        const int32_t gi = c.c0 + 4 * g + e;
        if (key == tkey && key != 0 && kept_by(key, gi, rk, ri)) {
          ++seen;
          if (seen == j) *found = gi;
        }
      }
    }
    __syncthreads();
    const int32_t f = *found;
    if (f >= 0) return f;
    if (total >= j) return -1;  // inconsistent (cannot happen for valid data)
    j -= total;
  }
  return -1;
}

// Exact radix select over the cluster's row, restricted to the elements kept by
// (rk, ri).  kMass = false: find the k-th element of the order (target = k).
// kMass = true: find the shortest prefix of the order whose softmax mass
// reaches p * (mass of the restricted set).  Returns the threshold of the
// selected prefix.  Every CTA of the cluster computes the same answer.
template <bool kMass>
__device__ Thresh radix_select(cg::cluster_group& cl, Ctx& c, unsigned long long target_k, float p,
                               uint32_t rk, int32_t ri) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int CS = static_cast<int>(cl.num_blocks());
  const float4* x4 = reinterpret_cast<const float4*>(c.xs);
  uint32_t prefix = 0, pmask = 0;
  unsigned long long tau = target_k;
  unsigned long long tie_weight = 0;
  bool ok = true;
  int cur = 0;
  for (int d = 0; d < 4; ++d) {
    const int shift = 24 - 8 * d;
    unsigned long long* h = c.hist + cur * kBins;
    unsigned long long* s = c.sup + cur * kSuper;
    for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0ull;
    __syncthreads();
    for (int g = threadIdx.x; g < c.n4; g += kThreads) {
      const float4 v = x4[g];
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t key = fkey(vv[e]);
        const int32_t gi = c.c0 + 4 * g + e;
        if (key != 0 && (key & pmask) == prefix && kept_by(key, gi, rk, ri)) {
          unsigned long long w = 1ull;
          if (kMass) w = fixed_mass(softmax_weight(vv[e], c.M));
          if (w) atomicAdd(&h[(key >> shift) & 0xFF], w);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x < kBins) {
      unsigned long long v = h[threadIdx.x];
#pragma unroll
      for (int o = 8; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
      if ((threadIdx.x & 15) == 0) s[threadIdx.x >> 4] = v;
    }
    cl.sync();
    if (warp == 0) {
      // super-bins, largest keys first: lane l covers super-bin 15 - l
      unsigned long long sv = 0;
      if (lane < kSuper)
        for (int r = 0; r < CS; ++r) sv += *cl.map_shared_rank(s + (kSuper - 1 - lane), r);
      if (kMass && d == 0) {
        const unsigned long long total = warp_sum_u64(sv);
        double t = ceil(static_cast<double>(p) * static_cast<double>(total));
        unsigned long long tt = static_cast<unsigned long long>(t);
        if (tt < 1ull) tt = 1ull;
        if (tt > total) tt = total;
        tau = tt;
      }
      const unsigned long long inc = warp_incl_scan_u64(sv, lane);
      unsigned m = __ballot_sync(kFull, lane < kSuper && inc >= tau);
      unsigned long long bin_w = 0, new_tau = tau;
      int beta = 0;
      bool good = (m != 0u) && tau > 0;
      if (good) {
        const int L = __ffs(m) - 1;
        const unsigned long long above = L > 0 ? __shfl_sync(kFull, inc, L - 1) : 0ull;
        const int sigma = kSuper - 1 - L;
        unsigned long long bv = 0;
        if (lane < 16)
          for (int r = 0; r < CS; ++r) bv += *cl.map_shared_rank(h + sigma * 16 + (15 - lane), r);
        const unsigned long long inc2 = warp_incl_scan_u64(bv, lane);
        const unsigned m2 = __ballot_sync(kFull, lane < 16 && above + inc2 >= tau);
        if (m2 == 0u) {
          good = false;
        } else {
          const int L2 = __ffs(m2) - 1;
          const unsigned long long above2 = above + (L2 > 0 ? __shfl_sync(kFull, inc2, L2 - 1) : 0ull);
          bin_w = __shfl_sync(kFull, bv, L2);
          beta = sigma * 16 + (15 - L2);
          new_tau = tau - above2;
        }
      }
      if (lane == 0) {
        c.misc[0] = static_cast<unsigned long long>(beta);
        c.misc[1] = new_tau;
        c.misc[2] = bin_w;
        c.misc[3] = good ? 1ull : 0ull;
        c.misc[4] = tau;
      }
    }
    __syncthreads();
    const int beta = static_cast<int>(c.misc[0]);
    tau = c.misc[1];
    tie_weight = c.misc[2];
    ok = ok && (c.misc[3] != 0ull);
    __syncthreads();
    if (!ok) break;  // uniform across the cluster (identical inputs to the decision)
    prefix |= static_cast<uint32_t>(beta) << shift;
    pmask |= 0xFFu << shift;
    cur ^= 1;
  }
  if (!ok) return Thresh{rk, ri};  // degenerate input: keep the whole restricted set

  const uint32_t key = prefix;
  // weight of one element equal to the threshold key
  const unsigned long long w1 = kMass ? fixed_mass(softmax_weight(kfloat(key), c.M)) : 1ull;
  if (w1 == 0ull) return Thresh{key, key == rk ? ri : INT_MAX};
  const unsigned long long ties = tie_weight / w1;
  const unsigned long long need = (tau + w1 - 1) / w1;  // ties to keep, >= 1
  if (need >= ties) return Thresh{key, key == rk ? ri : INT_MAX};

  // Split inside the ties: the need-th tie in index order.  CTAs own contiguous
  // index ranges in rank order, so find the owner from the per-CTA tie counts
  // (the last pass's local histograms, still intact), then search it.
  const int last = cur ^ 1;
  const int beta_last = static_cast<int>(key & 0xFFu);
  int owner = -1;
  unsigned long long jloc = 0;
  if (warp == 0) {
    unsigned long long t = 0;
    if (lane < CS) t = *cl.map_shared_rank(c.hist + last * kBins + beta_last, lane) / w1;
    const unsigned long long inc = warp_incl_scan_u64(t, lane);
    const unsigned m = __ballot_sync(kFull, lane < CS && inc >= need);
    if (m) {
      const int L = __ffs(m) - 1;
      const unsigned long long before = L > 0 ? __shfl_sync(kFull, inc, L - 1) : 0ull;
      owner = L;
      jloc = need - before;
    }
    if (lane == 0) {
      c.misc[5] = static_cast<unsigned long long>(static_cast<long long>(owner));
      c.misc[6] = jloc;
    }
  }
  __syncthreads();
  owner = static_cast<int>(static_cast<long long>(c.misc[5]));
  jloc = c.misc[6];
  __syncthreads();
  const int rank = static_cast<int>(cl.block_rank());
  if (rank == owner) {
    const int32_t f = local_nth_tie(c, key, rk, ri, static_cast<uint32_t>(jloc));
    if (threadIdx.x == 0) {
      for (int r = 0; r < CS; ++r)
        *cl.map_shared_rank(c.slots + kSlotTie, r) = static_cast<unsigned long long>(static_cast<uint32_t>(f));
    }
  }
  cl.sync();
  int32_t ti = static_cast<int32_t>(static_cast<uint32_t>(c.slots[kSlotTie]));
  if (owner < 0 || ti < 0) ti = (key == rk) ? ri : INT_MAX;  // degenerate: keep all ties
  return Thresh{key, ti};
}

// ------------------------------------------------------------------------------------------
// The kernel: one cluster per row.
// ------------------------------------------------------------------------------------------
template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 2) kps_sample_kernel(const Params P) {
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char smem[];
  const Layout L = make_layout(P.nc, kBF16);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L.bitmap);
  unsigned long long* mbar = reinterpret_cast<unsigned long long*>(smem + L.mbar);

  const int CS = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int64_t row = blockIdx.x / CS;
  const int64_t V = P.V;
  const int32_t c0 = rank * P.nc;
  int n = static_cast<int>(V - c0);
  n = n < 0 ? 0 : (n > P.nc ? P.nc : n);
  const int n4 = (n + 3) >> 2;

  Ctx c;
  c.xs = xs;
  c.c0 = c0;
  c.n = n;
  c.n4 = n4;
  c.hist = reinterpret_cast<unsigned long long*>(smem + L.hist);
  c.sup = reinterpret_cast<unsigned long long*>(smem + L.sup);
  c.red = reinterpret_cast<unsigned long long*>(smem + L.red);
  c.slots = reinterpret_cast<unsigned long long*>(smem + L.slots);
  c.misc = reinterpret_cast<unsigned long long*>(smem + L.misc);

  // ---- stage this CTA's chunk into shared memory --------------------------------------
  const size_t esize = kBF16 ? 2 : 4;
  void* stage = kBF16 ? static_cast<void*>(smem + L.raw) : static_cast<void*>(xs);
  const unsigned char* gsrc = static_cast<const unsigned char*>(P.logits) + (row * V + c0) * esize;
  const uint32_t bytes = static_cast<uint32_t>(n * esize);
  const bool tma = P.use_tma && bytes > 0;
  if (threadIdx.x == 0) mbar_init(mbar, 1);
  __syncthreads();
  if (tma && threadIdx.x == 0) {
    mbar_expect_tx(mbar, bytes);
    constexpr uint32_t kPiece = 16384;
    for (uint32_t off = 0; off < bytes; off += kPiece) {
      const uint32_t len = bytes - off < kPiece ? bytes - off : kPiece;
      bulk_g2s(static_cast<unsigned char*>(stage) + off, gsrc + off, len, mbar);
    }
  }

  // row parameters (uniform across the cluster)
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

  if (pen_on)
    for (int w = threadIdx.x; w < (n + 31) / 32; w += kThreads) bitmap[w] = 0u;

  if (!tma) {
    for (int i = threadIdx.x; i < n; i += kThreads) {
      if (kBF16) {
        const __nv_bfloat16 h = reinterpret_cast<const __nv_bfloat16*>(gsrc)[i];
        xs[i] = __bfloat162float(h);
      } else {
        xs[i] = reinterpret_cast<const float*>(gsrc)[i];
      }
    }
  }
  bool timed_out = false;
  if (tma) {
    if (!mbar_wait_bounded(mbar, 0)) {
      timed_out = true;
      if (threadIdx.x == 0) atomicMax(P.status, kStatusTimeout);
    }
  }
  if (kBF16 && tma) {
    const __nv_bfloat16* raw = reinterpret_cast<const __nv_bfloat16*>(smem + L.raw);
    for (int i = threadIdx.x; i < n; i += kThreads) xs[i] = __bfloat162float(raw[i]);
  }
  __syncthreads();

  // ---- repetition penalty: scatter over the seen ids, once per distinct id --------------
  if (pen_on) {
    const int32_t b0 = P.seen_indptr[row], b1 = P.seen_indptr[row + 1];
    for (int32_t j = b0 + threadIdx.x; j < b1; j += kThreads) {
      const int32_t id = P.seen_ids[j];
      const int32_t li = id - c0;
      if (id >= 0 && static_cast<int64_t>(id) < V && li >= 0 && li < n) {
        const uint32_t bit = 1u << (li & 31);
        const uint32_t old = atomicOr(&bitmap[li >> 5], bit);
        if (!(old & bit)) {
          const float s = xs[li];
          xs[li] = (s > 0.0f) ? __fdiv_rn(s, pen) : __fmul_rn(s, pen);
        }
      }
    }
    __syncthreads();
  }

  // ---- temperature, NaN -> -inf, padding, row maximum -----------------------------------
  unsigned long long best = 0;  // (key << 32) | ~index: max gives max key, then lowest index
  {
    float4* x4 = reinterpret_cast<float4*>(xs);
    for (int g = threadIdx.x; g < n4; g += kThreads) {
      float4 v = x4[g];
      float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 4 * g + e;
        float x = vv[e];
        if (i >= n) {
          x = __uint_as_float(0xFFFFFFFFu);  // padding: key 0
        } else {
          if (isnan(x)) x = -INFINITY;
          if (!greedyT) x = __fdiv_rn(x, T);
          x = __fadd_rn(x, 0.0f);  // -0 -> +0: equal values share one key
          const unsigned long long cand =
              (static_cast<unsigned long long>(fkey(x)) << 32) | static_cast<uint32_t>(~(c0 + i));
          best = cand > best ? cand : best;
        }
        vv[e] = x;
      }
      x4[g] = make_float4(vv[0], vv[1], vv[2], vv[3]);
    }
  }
  best = block_max_u64(best, c.red);
  const unsigned long long rowbest = cluster_max_u64(cl, best, c.slots + kSlotMax, c.misc + 10);
  const uint32_t mkey = static_cast<uint32_t>(rowbest >> 32);
  const int32_t v0 = static_cast<int32_t>(~static_cast<uint32_t>(rowbest));
  c.M = kfloat(mkey);

  // ---- selection: top-k then top-p, as one threshold in the order -----------------------
  Thresh th{0u, -1};  // keeps every real element (padding has key 0)
  if (single) {
    th = Thresh{mkey, v0};
  } else {
    if (topk_on) th = radix_select<false>(cl, c, static_cast<unsigned long long>(k), 0.0f, th.key, th.idx);
    if (topp_on) th = radix_select<true>(cl, c, 0ull, p, th.key, th.idx);
  }

  // ---- exponential race over the kept set ----------------------------------------------
  int32_t chosen = v0;
  if (!single) {
    const float* qrow = P.q + row * V;
    const bool q_vec = P.use_tma != 0;  // same 16-byte alignment condition as the logits rows
    unsigned long long rb = 0;
    const float4* x4 = reinterpret_cast<const float4*>(xs);
    for (int g = threadIdx.x; g < n4; g += kThreads) {
      const float4 v = x4[g];
      const float vv[4] = {v.x, v.y, v.z, v.w};
      bool kp[4];
      int nk = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kp[e] = kept_by(fkey(vv[e]), c0 + 4 * g + e, th.key, th.idx);
        nk += kp[e];
      }
      if (!nk) continue;
      float qq[4];
      if (nk == 4 && q_vec) {
        const float4 q4 = __ldcs(reinterpret_cast<const float4*>(qrow + c0) + g);
        qq[0] = q4.x; qq[1] = q4.y; qq[2] = q4.z; qq[3] = q4.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) qq[e] = kp[e] ? __ldcs(qrow + c0 + 4 * g + e) : 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!kp[e]) continue;
        const float w = softmax_weight(vv[e], c.M);
        const float r = __fdiv_rn(w, __fadd_rn(qq[e], P.eps));
        if (isnan(r)) continue;
        const unsigned long long cand = (static_cast<unsigned long long>(fkey(r)) << 32) |
                                        static_cast<uint32_t>(~(c0 + 4 * g + e));
        rb = cand > rb ? cand : rb;
      }
    }
    rb = block_max_u64(rb, c.red);
    rb = cluster_max_u64(cl, rb, c.slots + kSlotRace, c.misc + 11);
    if (rb != 0ull) chosen = static_cast<int32_t>(~static_cast<uint32_t>(rb));
  }

  // ---- filtered logits in vocabulary order -------------------------------------------
  if (P.need_logits && n > 0) {
    float* orow = P.out_filtered + row * V + c0;
    const float4* x4 = reinterpret_cast<const float4*>(xs);
    if (P.use_tma && (n & 3) == 0) {
      for (int g = threadIdx.x; g < n4; g += kThreads) {
        const float4 v = x4[g];
        float4 o;
        o.x = kept_by(fkey(v.x), c0 + 4 * g + 0, th.key, th.idx) ? v.x : -INFINITY;
        o.y = kept_by(fkey(v.y), c0 + 4 * g + 1, th.key, th.idx) ? v.y : -INFINITY;
        o.z = kept_by(fkey(v.z), c0 + 4 * g + 2, th.key, th.idx) ? v.z : -INFINITY;
        o.w = kept_by(fkey(v.w), c0 + 4 * g + 3, th.key, th.idx) ? v.w : -INFINITY;
        __stcs(reinterpret_cast<float4*>(orow) + g, o);
      }
    } else {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const float x = xs[i];
        orow[i] = kept_by(fkey(x), c0 + i, th.key, th.idx) ? x : -INFINITY;
      }
    }
  }
  if (rank == 0 && threadIdx.x == 0) P.out_idx[row] = chosen;

  // a CTA that gave up on its copy waits (bounded) for it before leaving
  if (timed_out) (void)mbar_wait_bounded(mbar, 0);
  // no CTA leaves while another may still read its shared memory
  cl.sync();
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
struct LaunchCfg {
  int cs;
  int nc;
  size_t smem;
};

static int device_smem_optin() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  return v;
}

static int device_sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return v;
}

static int round_up8(int64_t x) { return static_cast<int>((x + 7) / 8 * 8); }

// Kernel attributes are per device: set them once for each device that launches.
template <bool kBF16>
static cudaError_t prepare_kernel() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  const int optin = device_smem_optin();
  err = cudaFuncSetAttribute(kps_sample_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(kps_sample_kernel<kBF16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (err == cudaSuccess) done[dev] = true;
  return err;
}

template <bool kBF16>
static bool cluster_fits(int cs, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = cs;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kps_sample_kernel<kBF16>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return n > 0;
}

// Chooses the cluster size: the smallest power of two whose per-CTA chunk fits
// two CTAs per SM, else the smallest that fits at all; then, for small
// batches, wider clusters so more SMs work on each row.
template <bool kBF16>
static kps_status choose_launch(int64_t B, int64_t V, LaunchCfg* out) {
  const int optin = device_smem_optin();
  const int sms = device_sm_count();
  if (optin <= 0 || sms <= 0) return KPS_ERR_CUDA;
  if (prepare_kernel<kBF16>() != cudaSuccess) return KPS_ERR_CUDA;
  const int sizes[] = {1, 2, 4, 8, 16};
  int pick = -1;
  for (int cs : sizes) {
    if (cs > 8) break;
    const int nc = round_up8((V + cs - 1) / cs);
    if (make_layout(nc, kBF16).total <= static_cast<size_t>(kSmemCap2PerSM)) { pick = cs; break; }
  }
  if (pick < 0) {
    for (int cs : sizes) {
      const int nc = round_up8((V + cs - 1) / cs);
      if (make_layout(nc, kBF16).total <= static_cast<size_t>(optin) &&
          cluster_fits<kBF16>(cs, make_layout(nc, kBF16).total)) { pick = cs; break; }
    }
  }
  if (pick < 0) return KPS_ERR_UNSUPPORTED;
  // small batches: spread each row over more SMs (chunks of at least 4096 elements)
  while (pick < 16 && B * pick * 2 <= sms && (V + pick * 2 - 1) / (pick * 2) >= 4096) {
    const int nc2 = round_up8((V + pick * 2 - 1) / (pick * 2));
    if (!cluster_fits<kBF16>(pick * 2, make_layout(nc2, kBF16).total)) break;
    pick *= 2;
  }
  out->cs = pick;
  out->nc = round_up8((V + pick - 1) / pick);
  out->smem = make_layout(out->nc, kBF16).total;
  if (!cluster_fits<kBF16>(out->cs, out->smem)) return KPS_ERR_UNSUPPORTED;
  return KPS_OK;
}

}  // namespace kps

// ------------------------------------------------------------------------------------------
// C ABI
// ------------------------------------------------------------------------------------------
extern "C" {

size_t kps_workspace_size(int64_t B, int64_t V, kps_dtype dt) {
  if (B < 0 || V < 1 || (dt != KPS_F32 && dt != KPS_BF16)) return 0;
  return 256;
}

int64_t kps_max_vocab(kps_dtype dt) {
  const int optin = kps::device_smem_optin();
  if (optin <= 0) return 0;
  const bool bf = dt == KPS_BF16;
  // largest chunk that fits one CTA, times the widest cluster
  int lo = 8, hi = 1 << 20;
  while (lo < hi) {
    const int mid = ((lo + hi + 1) / 2) / 8 * 8;
    if (mid <= lo) break;
    if (kps::make_layout(mid, bf).total <= static_cast<size_t>(optin)) lo = mid; else hi = mid - 8;
  }
  return static_cast<int64_t>(lo) * 16;
}

const char* kps_status_string(kps_status s) {
  switch (s) {
    case KPS_OK: return "ok";
    case KPS_ERR_INVALID_ARG: return "invalid argument";
    case KPS_ERR_UNSUPPORTED: return "unsupported size";
    case KPS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case KPS_ERR_CUDA: return "CUDA error";
    case KPS_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

kps_status kps_query_launch(int64_t B, int64_t V, kps_dtype dt, int* cluster_size, int64_t* chunk_elems,
                            size_t* smem_bytes) {
  if (V < 1 || V > INT32_MAX || B < 0 || (dt != KPS_F32 && dt != KPS_BF16)) return KPS_ERR_INVALID_ARG;
  kps::LaunchCfg cfg;
  const kps_status st = dt == KPS_BF16 ? kps::choose_launch<true>(B, V, &cfg) : kps::choose_launch<false>(B, V, &cfg);
  if (st != KPS_OK) return st;
  if (cluster_size) *cluster_size = cfg.cs;
  if (chunk_elems) *chunk_elems = cfg.nc;
  if (smem_bytes) *smem_bytes = cfg.smem;
  return KPS_OK;
}

kps_status kps_sample(const void* logits, kps_dtype dt, int64_t B, int64_t V, const int32_t* top_k,
                      const float* top_p, const float* temperature, const int32_t* seen_indptr,
                      const int32_t* seen_ids, const float* penalty, const float* q, float eps, int need_logits,
                      int64_t* out_idx, float* out_filtered, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  if (dt != KPS_F32 && dt != KPS_BF16) return KPS_ERR_INVALID_ARG;
  if (V < 1 || V > INT32_MAX || B < 0) return KPS_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || std::isinf(eps)) return KPS_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < kps_workspace_size(B, V, dt))
    return KPS_ERR_WORKSPACE;
  if (B == 0) return KPS_OK;
  if (B > INT32_MAX / 16) return KPS_ERR_INVALID_ARG;
  if (!logits || !top_k || !top_p || !temperature || !q || !out_idx) return KPS_ERR_INVALID_ARG;
  if (need_logits && !out_filtered) return KPS_ERR_INVALID_ARG;
  const bool pen = seen_indptr && seen_ids && penalty;

  kps::LaunchCfg cfg;
  const kps_status st =
      dt == KPS_BF16 ? kps::choose_launch<true>(B, V, &cfg) : kps::choose_launch<false>(B, V, &cfg);
  if (st != KPS_OK) return st;

  kps::Params P;
  P.logits = logits;
  P.B = B;
  P.V = V;
  P.top_k = top_k;
  P.top_p = top_p;
  P.temperature = temperature;
  P.seen_indptr = pen ? seen_indptr : nullptr;
  P.seen_ids = pen ? seen_ids : nullptr;
  P.penalty = pen ? penalty : nullptr;
  P.q = q;
  P.eps = eps;
  P.need_logits = need_logits ? 1 : 0;
  P.out_idx = out_idx;
  P.out_filtered = need_logits ? out_filtered : nullptr;
  P.status = static_cast<int*>(workspace);
  P.nc = cfg.nc;
  const size_t esize = dt == KPS_BF16 ? 2 : 4;
  const bool aligned = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && ((V * esize) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(q) % 16 == 0) && (V % 4 == 0) &&
                       (!need_logits || reinterpret_cast<uintptr_t>(out_filtered) % 16 == 0);
  P.use_tma = aligned ? 1 : 0;

  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(B * cfg.cs));
  lc.blockDim = dim3(kps::kThreads);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cfg.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaError_t e = dt == KPS_BF16 ? cudaLaunchKernelEx(&lc, kps::kps_sample_kernel<true>, P)
                                 : cudaLaunchKernelEx(&lc, kps::kps_sample_kernel<false>, P);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return KPS_ERR_CUDA;
  }
  return KPS_OK;
}

kps_status kps_last_device_status(void* workspace, cudaStream_t stream, int* out) {
  if (!workspace || !out) return KPS_ERR_INVALID_ARG;
  int h = 0;
  if (cudaMemcpyAsync(&h, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return KPS_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KPS_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), stream) != cudaSuccess) return KPS_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KPS_ERR_CUDA;
  *out = h;
  return KPS_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// No-allocation entry point: the scratch lives in a fixed device array.
// ------------------------------------------------------------------------------------------
namespace kps {
constexpr size_t kNoallocScratchBytes = 4096;
constexpr int kMaxDevices = 64;
// File-scope scratch for kps_sample_noalloc.  In host code this name is only a
// stand-in for the symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device with that device current.  Returns nullptr on failure.
static void* noalloc_scratch_address() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}
}  // namespace kps

extern "C" kps_status kps_sample_noalloc(const void* logits, kps_dtype dt, int64_t B, int64_t V,
                                         const int32_t* top_k, const float* top_p, const float* temperature,
                                         const int32_t* seen_indptr, const int32_t* seen_ids,
                                         const float* penalty, const float* q, float eps, int need_logits,
                                         int64_t* out_idx, float* out_filtered, cudaStream_t stream) {
  const size_t need = kps_workspace_size(B, V, dt);
  if (need == 0) return KPS_ERR_INVALID_ARG;
  if (need > kps::kNoallocScratchBytes) return KPS_ERR_UNSUPPORTED;
  if (B == 0) return KPS_OK;
  void* scratch = kps::noalloc_scratch_address();
  if (!scratch) return KPS_ERR_CUDA;
  // the shared array keeps the previous call's status word: clear it on this stream first
  if (cudaMemsetAsync(scratch, 0, need, stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return KPS_ERR_CUDA;
  }
  return kps_sample(logits, dt, B, V, top_k, top_p, temperature, seen_indptr, seen_ids, penalty, q, eps,
                    need_logits, out_idx, out_filtered, scratch, kps::kNoallocScratchBytes, stream);
}
