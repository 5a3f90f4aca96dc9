// kps.cu — GB300 (sm_103a) kernels and C ABI for the decode-step sampler.
//
// A persistent grid of thread-block clusters walks the rows of the [B, V]
// logits matrix; a cluster of CS CTAs owns one row at a time, CTA r holding
// the contiguous chunk [r*nc, (r+1)*nc) in shared memory.  Each chunk is
// staged with a TMA bulk copy (cp.async.bulk + mbarrier), so logits are read
// from HBM once; CTAs combine partial results through distributed shared
// memory (DSMEM) and cluster barriers.  Per row:
//
//   load -> penalty (scatter over the seen ids, once per distinct id)
//        -> raw pass: NaN -> -inf, -0 -> +0, row maximum and the maximum of
//           every 128-element group.  Division by a positive temperature is
//           monotone, so maxima (and any order bound) can be taken before it.
//   top-k rows (1 < k <= min(V, 1024)):
//        -> t0 = (a lower bound of) the k-th largest group maximum divided by
//           T: k groups have a maximum >= it, so the row's k-th value is >= t0.
//        -> candidate pass: only elements that can reach t0 are divided by T;
//           those >= t0 are kept in a per-CTA list and counted in 2048 linear
//           bins of (M - y).  The chunk is then free: the TMA load of the
//           CTA's next row starts here and overlaps the rest of this row.
//        -> the bin holding the k-th element is found from the cluster-wide
//           histogram; its few elements are gathered to every CTA and ranked
//           exactly, giving the k-th element (value desc, index asc).
//        -> top-p inside the k survivors: the same bin search weighted by
//           softmax mass in 2^-40 fixed point, then an exact prefix over the
//           boundary bin's elements.
//        -> race over the kept candidates (q gathered at their indices).
//   top-p-only rows: the chunk is divided by T in place; a mass histogram over
//        linear bins of (M - x), then a finer one inside the boundary bin,
//        locates the boundary, resolved exactly as above; the race and the
//        filtered-logit write are one fused pass.
//   Any overflow of the small candidate structures falls back to an exact
//   radix select over the whole resident row.
//
// Softmax mass is held in 2^-40 fixed point (uint64), so every sum is exact
// and independent of summation order; weights are expf of the difference
// x - max carried exactly (TwoSum).
//
// The method follows the Ascend "torch_npu.npu_top_k_top_p_sample" page
// (topK valid range, topP full-sort rule, Sample formulas), MiniMind
// "Chapter 10: inference generation" (§10.4 temperature, §10.5 top-k, §10.6
// top-p, §10.7 repetition penalty) and the C++ post-processing blog
// (penalty over the set of seen ids, softmax).  Selection is by bounds,
// histograms and small exact rankings instead of the sorts and quickselects
// on those pages.
//
// Nothing here waits without a bound: a TMA wait that gives up after ~2 s of
// clock cycles records KPS_ERR_TIMEOUT in the status word and gives the copy
// one more bound before its buffer is read or reused; a copy still out after
// that stops all further copies of the CTA, which carries on with the same
// control flow (so the cluster barriers always complete) and waits for it once
// more before it exits.

#include "kps.h"
#include "kps_fixed.h"
#include "kps_div.h"
#include "kps_weights.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cooperative_groups.h>
#include <nvtx3/nvToolsExt.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

namespace cg = cooperative_groups;

namespace kps {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCS = 16;          // widest cluster
constexpr int kBins = 256;          // 8-bit radix digits (fallback radix select)
constexpr int kSuper = 16;          // super-bins of 16 bins each (fallback radix select)
constexpr int kTopKMax = 1024;      // top-k is active for 1 <= k <= min(V, 1024)
constexpr int kCapLoc = 1024;       // candidates one CTA may hold
constexpr int kGallCap = 2048;      // group maxima one row may have for the top-k bound
constexpr int kGroupSplit = 8;      // groups of 128 elements split up to 8 ways (16 elements)
constexpr int kGatherTopP = 256;    // top-k rows with at most this many survivors cut top-p on rank 0
constexpr int kLinBins = 2048;      // linear count bins of the top-k candidate pass
static_assert(kLinBins == 1 << 11, "the k-th bound keeps 11 bits of the key span");
constexpr int kLinBinsP = 1024;     // linear mass bins (width 1/16 of d = max - x) of top-p-only rows
constexpr int kFineBins = 1024;     // linear bins of the refinement histogram (top-p-only rows)
constexpr int kSmall = 64;          // boundary-bin elements resolved by exact ranking
constexpr int kMaxChunk = 65536;    // largest per-CTA chunk the layout supports
constexpr long long kSpinCycles = 4000000000LL;  // bounded wait (~2 s)
constexpr int kSmemCap2PerSM = 112 * 1024;  // per-CTA budget for two CTAs per SM
constexpr unsigned kFull = 0xffffffffu;
constexpr int kStatusTimeout = KPS_ERR_TIMEOUT;
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // key of -inf; key 0 marks padding

// Shared-memory exchange slots (u64).  Arrays of kMaxCS are filled by every CTA
// of the cluster (push), so each CTA reduces them locally after the barrier.
enum Slot {
  kSlotMax = 0,                       // [kMaxCS] row maximum pushes
  kSlotRace = kSlotMax + kMaxCS,      // [kMaxCS] race winner pushes
  kSlotFlag = kSlotRace + kMaxCS,     // [kMaxCS] per-CTA flags
  kSlotV0 = kSlotFlag + kMaxCS,       // [kMaxCS] first-of-order pushes
  kSlotTie = kSlotV0 + kMaxCS,        // split tie (fallback radix select)
  kSlotSmallCnt,                      // size of this CTA's boundary list
  kNumSlots
};

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
  int use_tma;  // every row of logits, q and out starts on a 16-byte boundary
  int filter;   // rows this launch takes: 0 all, 1 top-k/one-element rows, 2 the others
  int exact;    // row kernel: skip the sample and the band, always select over the whole row
  unsigned char* pre;  // row kernel: per-row records of the pre-pass (nullptr: no pre-pass)
  int pre_rows;        // records available (the first pre_rows top-p-only rows use them)
  int gen;             // race with generated Exp(1) draws (q is then nullptr)
  unsigned long long seed, step;  // their generator's key and the decode step
  unsigned char* finished;        // [B] end-of-sequence flags (nullptr: no epilogue)
  long long eos;                  // the end-of-sequence token
  int* unfinished;                // rows still unfinished after the step (nullptr: not counted)
  uint32_t* seen_bits;            // [B, (V + 31) / 32] seen-token bits in place of the seen ids
  int update_seen;                // set the bit of each row's emitted token after the step
};

// Words of one row of the seen-token bits.
__host__ __device__ __forceinline__ int64_t seen_words(int64_t V) { return (V + 31) / 32; }

// Seen word w of a row's bits with the bits of tokens >= V cleared (0 past the row).
__device__ __forceinline__ uint32_t seen_word_at(const uint32_t* row_bits, int64_t V, int64_t w) {
  const int64_t hi = V - 32 * w;  // tokens of this word below V
  if (hi <= 0) return 0u;
  const uint32_t x = __ldcg(row_bits + w);
  return hi >= 32 ? x : (x & ((1u << hi) - 1u));
}

constexpr int kMaxRowList = 256;  // rows one worker (CTA or cluster) may own in a filtered launch

// True for rows of the one-pass top-k path: top-k active, or a single element kept
// (greedy temperature, top_p <= 0, or k == 1).  Every kernel and worker agrees on it.
__device__ __forceinline__ bool row_is_kmode(const Params& P, int64_t row) {
  const int32_t k = P.top_k[row];
  const float p = P.top_p[row];
  const float T = P.temperature[row];
  const bool greedyT = !(T > 0.0f) || isinf(T);
  const bool topk_on = k >= 1 && static_cast<int64_t>(k) <= (P.V < 1024 ? P.V : 1024);
  return topk_on || greedyT || (!isnan(p) && p <= 0.0f);
}

// Rows worker w of nw owns in a filtered launch: the matching rows whose rank among
// matching rows is w mod nw, in row order, written to list; returns how many.
template <int NT>
__device__ int build_row_list(const Params& P, int64_t w, int64_t nw, int32_t* list, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = NT / 32;
  int64_t running = 0;
  int count = 0;
  for (int64_t base = 0; base < P.B; base += NT) {
    const int64_t row = base + threadIdx.x;
    const bool m = row < P.B && (row_is_kmode(P, row) == (P.filter == 1));
    const unsigned bal = __ballot_sync(0xffffffffu, m);
    if (lane == 0) red[warp] = __popc(bal);
    __syncthreads();
    uint32_t before = 0, total = 0;
    for (int q = 0; q < NW; ++q) {
      const uint32_t c = static_cast<uint32_t>(red[q]);
      if (q < warp) before += c;
      total += c;
    }
    const int64_t rank = running + before + __popc(bal & ((1u << lane) - 1u));
    if (m && rank % nw == w) {
      const int64_t slot = rank / nw;
      if (slot < kMaxRowList) list[slot] = static_cast<int32_t>(row);
    }
    running += total;
    __syncthreads();
  }
  if (running > w) count = static_cast<int>((running - 1 - w) / nw + 1);
  return count < kMaxRowList ? count : kMaxRowList;
}

// ------------------------------------------------------------------------------------------
// Shared-memory layout (identical on host and device).
// ------------------------------------------------------------------------------------------
struct Layout {
  size_t xs, raw, cand_key, cand_idx, hist, fine, sup, small, gmax, red, slots, mbar, misc, rows, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline Layout make_layout(int nc, bool bf16) {
  Layout L;
  size_t off = 0;
  L.xs = off;       off += align16(size_t(nc) * 4);
  L.raw = off;      off += bf16 ? align16(size_t(nc) * 2) : 0;
  L.cand_key = off; off += size_t(kCapLoc) * 4;  // also the penalty bitmap (nc/8 bytes)
  L.cand_idx = off; off += size_t(kCapLoc) * 4;
  L.hist = off;     off += size_t(3 * 1024) * 4;  // histograms (u32 counts or 16-bit mass limbs),
                                                   // also the gathered group maxima
  L.fine = off;     off += size_t(3 * kFineBins) * 4;
  L.sup = off;      off += size_t(kLinBinsP / 32 + kFineBins / 32) * 8;
  L.small = off;    off += size_t(2 * kSmall) * 8;  // own boundary list, then the gathered one
  L.gmax = off;     off += align16(size_t((nc + 127) / 128) * 4 * kGroupSplit);
  L.red = off;      off += 40 * 8;
  L.slots = off;    off += size_t(kNumSlots) * 8;
  L.mbar = off;     off += 16;
  L.misc = off;     off += 16 * 8;
  L.rows = off;     off += size_t(kMaxRowList) * 4;
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
// u64 form of an (key, index) pair whose unsigned order is the order (value desc, index asc)
__device__ __forceinline__ unsigned long long order_word(uint32_t key, int32_t idx) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~idx);
}

// Softmax weight exp(x - M) in fp32.  The difference x - M is carried exactly
// as hi + lo (Knuth's TwoSum) and the exponential is corrected to first order,
// e * (1 + lo), so the weight does not inherit the rounding of the subtraction.
// x == M gives exactly 1 (which keeps +-inf maxima finite).
// ---- generated Exp(1) draws ------------------------------------------------------------
//
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2,
// 3", SC'11, section 4 and its Philox-4x32 round constants): ten rounds of two
// 32x32 -> 64-bit products whose halves are mixed into the other counter words, the key
// bumped by its Weyl increments between rounds.  The draw of row b, token v at step s
// under seed k: counter (v / 4, b, s low, s high), key (k low, k high), word v mod 4,
// u = (2 (w >> 9) + 1) 2^-24, q = -log(u).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}
__device__ __forceinline__ float exp_of_word(uint32_t w) {
  return -logf(__fmul_rn(static_cast<float>(2u * (w >> 9) + 1u), 5.9604644775390625e-8f));
}
// The four draws of tokens 4g .. 4g + 3 of a row.
__device__ __forceinline__ float4 gen_q4(unsigned long long seed, unsigned long long step, int64_t row, int64_t g) {
  const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(g), static_cast<uint32_t>(row),
                                           static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32)),
                                static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  return make_float4(exp_of_word(w.x), exp_of_word(w.y), exp_of_word(w.z), exp_of_word(w.w));
}
// The draw of token v of a row.
__device__ __forceinline__ float gen_q1(unsigned long long seed, unsigned long long step, int64_t row, int64_t v) {
  const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(row),
                                           static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32)),
                                static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const int e = static_cast<int>(v & 3);
  return exp_of_word(e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w);
}

// The end-of-sequence epilogue of a row's chosen token (MiniMind, "Chapter 10: inference
// generation", the generate loop): a finished row emits the end-of-sequence token, a row
// that emits it becomes finished, and the rows left unfinished are counted.
__device__ __forceinline__ long long eos_epilogue(const Params& P, int64_t row, int32_t chosen) {
  if (!P.finished) return chosen;
  const bool was = P.finished[row] != 0;
  const long long out = was ? P.eos : static_cast<long long>(chosen);
  const bool now = was || out == P.eos;
  if (now && !was) P.finished[row] = 1;
  if (!now && P.unfinished) atomicAdd(P.unfinished, 1);
  return out;
}

// The emitted token of a row joins its seen set (every reader of the row's bits in
// this launch has read them by now: the token depends on what each of them computed).
__device__ __forceinline__ void seen_append(const Params& P, int64_t row, long long tok) {
  if (!P.update_seen || tok < 0 || tok >= P.V) return;
  atomicOr(P.seen_bits + row * seen_words(P.V) + (tok >> 5), 1u << (tok & 31));
}

__device__ __forceinline__ unsigned long long fixed_mass(float w) {
  return fixed_mass_of(w);
}

// Linear bin of y in [lo, M]: min(nb - 1, floor((M - y) * s)); monotone
// non-increasing in y (bin 0 holds the largest values).
__device__ __forceinline__ int lin_bin_scaled(float y, float M, float s, int nb) {
  if (y == M) return 0;
  const float d = __fsub_rn(M, y);
  const float f = __fmul_rn(d, s);
  if (!(f < static_cast<float>(nb))) return nb - 1;
  return static_cast<int>(f);
}
// First histogram of top-p-only rows: bins of width 1/16 in d = M - x over
// [0, 64); returns kLinBinsP for d >= 64 (zero fixed-point mass).
__device__ __forceinline__ int lin_bin_mass(float x, float M) {
  if (x == M) return 0;
  const float d = __fsub_rn(M, x);
  if (!(d < 64.0f)) return kLinBinsP;
  return static_cast<int>(d * 16.0f);
}
// Refinement inside first-level bin b: kFineBins bins over d in [b/16, (b+1)/16).
__device__ __forceinline__ int fine_bin_mass(float x, float M, int b) {
  const float d = (x == M) ? 0.0f : __fsub_rn(M, x);
  const float f = __fmul_rn(__fsub_rn(d, static_cast<float>(b) * 0.0625f), 16.0f * kFineBins);
  if (!(f > 0.0f)) return 0;
  if (!(f < static_cast<float>(kFineBins))) return kFineBins - 1;
  return static_cast<int>(f);
}

// A raw value below which x / T cannot reach t0 = fl(g / T) (T finite > 0):
// any x < g - 4 * T * ulp(t0) has x / T at least 3.5 ulp below t0.  Returns
// -inf when t0 is not a normal number with room (then every element is tested).
__device__ __forceinline__ float raw_lower_bound(float g, float t0, float T) {
  const float a = fabsf(t0);
  if (!(a >= 1e-30f) || !(a <= 1e30f) || isinf(g)) return -INFINITY;
  const float up = __uint_as_float(__float_as_uint(a) + 1u) - a;  // spacing above |t0|
  const double gap = 4.0 * static_cast<double>(T) * static_cast<double>(up);
  return __double2float_rd(static_cast<double>(g) - gap);
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
// Bounded wait: returns false if the phase did not complete within `cycles`.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity,
                                                  long long cycles = kSpinCycles) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > cycles) return false;
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
__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned long long w = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += w;
  }
  return v;
}
__device__ __forceinline__ uint32_t warp_incl_scan_u32(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t w = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += w;
  }
  return v;
}

// Block-wide sum of a u64; every thread gets the result.
__device__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kWarps ? red[lane] : 0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  v = red[32];
  __syncthreads();
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

// Block-wide exclusive scan of u32 values; *total gets the sum.
__device__ uint32_t block_excl_scan_u32(uint32_t v, uint32_t* total, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t x = warp_incl_scan_u32(v, lane);
  if (lane == 31) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint32_t s = lane < kWarps ? static_cast<uint32_t>(red[lane]) : 0u;
    const uint32_t t = warp_incl_scan_u32(s, lane);
    if (lane < kWarps) red[lane] = t - s;
    if (lane == kWarps - 1) red[32] = t;
  }
  __syncthreads();
  const uint32_t res = static_cast<uint32_t>(red[warp]) + x - v;
  *total = static_cast<uint32_t>(red[32]);
  __syncthreads();
  return res;
}

// Sum over the cluster of the value at the same shared-memory address in
// every CTA (loads issued together).
template <typename T>
__device__ __forceinline__ unsigned long long remote_sum(cg::cluster_group& cl, T* p, int CS) {
  unsigned long long s = 0;
  for (int r = 0; r < CS; r += 4) {
    T v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = r + u < CS ? *cl.map_shared_rank(p, r + u) : T(0);
#pragma unroll
    for (int u = 0; u < 4; ++u) s += static_cast<unsigned long long>(v[u]);
  }
  return s;
}

// A histogram of nb bins in shared memory.  L = 1: u32 counts.  L = 3: a fixed-point
// mass split into three 16-bit limbs, one u32 array each (shared-memory 64-bit atomics
// are slow; 32-bit ones are not).  A bin may take up to 65536 additions without a limb
// overflowing, so the exact u64 sum is limb0 + (limb1 << 16) + (limb2 << 32).
template <int L>
struct Bins {
  uint32_t* base;
  int nb;
  __device__ __forceinline__ void clear(int nthreads) const {
    for (int i = threadIdx.x; i < L * nb; i += nthreads) base[i] = 0u;
  }
  __device__ __forceinline__ void add(int b, unsigned long long w) const {
    if (L == 1) {
      atomicAdd(base + b, static_cast<uint32_t>(w));
    } else {
      atomicAdd(base + b, static_cast<uint32_t>(w & 0xFFFFu));
      atomicAdd(base + nb + b, static_cast<uint32_t>((w >> 16) & 0xFFFFu));
      atomicAdd(base + 2 * nb + b, static_cast<uint32_t>(w >> 32));
    }
  }
  __device__ __forceinline__ unsigned long long get(int b) const {
    if (L == 1) return base[b];
    return static_cast<unsigned long long>(base[b]) + (static_cast<unsigned long long>(base[nb + b]) << 16) +
           (static_cast<unsigned long long>(base[2 * nb + b]) << 32);
  }
  // the same bin of CTA r of the cluster
  __device__ __forceinline__ unsigned long long get_rank(cg::cluster_group& cl, int b, int r) const {
    const uint32_t* rb = cl.map_shared_rank(base, r);
    if (L == 1) return rb[b];
    return static_cast<unsigned long long>(rb[b]) + (static_cast<unsigned long long>(rb[nb + b]) << 16) +
           (static_cast<unsigned long long>(rb[2 * nb + b]) << 32);
  }
  // the bin summed over the cluster (loads issued together)
  __device__ __forceinline__ unsigned long long get_cluster(cg::cluster_group& cl, int b, int CS) const {
    unsigned long long s = 0;
    for (int l = 0; l < L; ++l) s += remote_sum(cl, base + l * nb + b, CS) << (16 * l);
    return s;
  }
};

// Pushes a u64 into slot array `arr` (index = own rank) of every CTA of the cluster.
__device__ __forceinline__ void push_all(cg::cluster_group& cl, unsigned long long* arr, int rank, int CS,
                                         unsigned long long v) {
  for (int r = 0; r < CS; ++r) *cl.map_shared_rank(arr + rank, r) = v;
}
__device__ __forceinline__ unsigned long long max_of(const unsigned long long* arr, int CS) {
  unsigned long long m = 0;
  for (int r = 0; r < CS; ++r) m = arr[r] > m ? arr[r] : m;
  return m;
}

// ------------------------------------------------------------------------------------------
// Per-CTA context for one row
// ------------------------------------------------------------------------------------------
struct Ctx {
  float* xs;            // this CTA's chunk (raw, then transformed where a path needs it)
  int32_t c0;           // row index of xs[0]
  int n;                // elements in this chunk
  int n4;               // float4 groups covering the chunk (tail padded with key 0)
  float M;              // row maximum (transformed)
  uint32_t* cand_key;   // candidate list of this CTA (transformed keys)
  int32_t* cand_idx;
  uint32_t* hist;            // 3072 words: 2048 counts, 1024-bin limb histogram, or radix bins
  uint32_t* fine;            // 3 x kFineBins words: 1024-bin limb histogram
  unsigned long long* sup;   // kLinBins/32 + kFineBins/32 u64 (fallback radix uses two 16-entry halves)
  unsigned long long* small; // [kSmall] own boundary list, [kSmall] gathered list
  uint32_t* gmax;            // this CTA's group maxima (raw keys)
  unsigned long long* red;
  unsigned long long* slots;
  unsigned long long* misc;
};

// Result of a selection: the last kept element's key and index.
struct Thresh {
  uint32_t key;
  int32_t idx;
};

// Element sources for the fallback radix select.  for_each calls
// f(valid, key, index, value) with the whole warp converged.
struct SrcData {  // the CTA's resident chunk (transformed values)
  const float* xs;
  int n4;
  int32_t c0;
  template <class F>
  __device__ __forceinline__ void for_each(F&& f) const {
    for (int base = 0; base < n4; base += kThreads) {
      const int g = base + threadIdx.x;
      const bool in = g < n4;
      const float4 v = in ? reinterpret_cast<const float4*>(xs)[g] : make_float4(0.f, 0.f, 0.f, 0.f);
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t key = fkey(vv[e]);
        f(in && key != 0u, key, c0 + 4 * g + e, vv[e]);
      }
    }
  }
};
struct SrcCand {  // this CTA's candidate list (unordered)
  const uint32_t* key;
  const int32_t* idx;
  int n;
  template <class F>
  __device__ __forceinline__ void for_each(F&& f) const {
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + threadIdx.x;
      const bool in = i < n;
      const uint32_t k = in ? key[i] : 0u;
      f(in && k != 0u, k, in ? idx[i] : 0, kfloat(k));
    }
  }
};

// j-th (1-based) smallest index among this CTA's elements with key == tkey kept by (rk, ri).
__device__ int32_t nth_tie(const SrcData& s, const Ctx& c, uint32_t tkey, uint32_t rk, int32_t ri, uint32_t j) {
  int32_t* found = reinterpret_cast<int32_t*>(c.misc + 8);
  if (threadIdx.x == 0) *found = -1;
  __syncthreads();
  for (int base = 0; base < s.n4; base += kThreads) {
    const int g = base + threadIdx.x;
    uint32_t cnt = 0;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (g < s.n4) {
      v = reinterpret_cast<const float4*>(s.xs)[g];
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t key = fkey(vv[e]);
        cnt += (key == tkey && key != 0 && kept_by(key, s.c0 + 4 * g + e, rk, ri)) ? 1u : 0u;
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
        if (key == tkey && key != 0 && kept_by(key, s.c0 + 4 * g + e, rk, ri)) {
          ++seen;
          if (seen == j) *found = s.c0 + 4 * g + e;
        }
      }
    }
    __syncthreads();
    const int32_t f = *found;
    if (f >= 0) return f;
    if (total >= j) return -1;
    j -= total;
  }
  return -1;
}
// Same over the (unordered) candidate list: the tie whose index has exactly j-1
// smaller tie indices.
__device__ int32_t nth_tie(const SrcCand& s, const Ctx& c, uint32_t tkey, uint32_t rk, int32_t ri, uint32_t j) {
  int32_t* found = reinterpret_cast<int32_t*>(c.misc + 8);
  if (threadIdx.x == 0) *found = -1;
  __syncthreads();
  for (int i = threadIdx.x; i < s.n; i += kThreads) {
    if (s.key[i] != tkey || !kept_by(s.key[i], s.idx[i], rk, ri)) continue;
    uint32_t smaller = 0;
    for (int m = 0; m < s.n; ++m)
      smaller += (s.key[m] == tkey && s.idx[m] < s.idx[i] && kept_by(s.key[m], s.idx[m], rk, ri)) ? 1u : 0u;
    if (smaller + 1 == j) *found = s.idx[i];
  }
  __syncthreads();
  return *found;
}

// Exact distributed radix select over the cluster's elements from `src`,
// restricted to those kept by (rk, ri).  kMass = false: the target is a count
// (find the target-th element of the order).  kMass = true: the target is a
// fixed-point mass (find the shortest prefix whose mass reaches it); with
// p_mode the target is ceil(p * total mass of the restricted set).  Returns
// the threshold of the selected prefix.  Every CTA computes the same answer.
// Used when the fast paths' small structures overflow.
template <class Src, bool kMass>
__device__ __noinline__ Thresh radix_select(cg::cluster_group& cl, Ctx& c, const Src& src, unsigned long long target,
                               bool p_mode, float p, uint32_t rk, int32_t ri) {
  constexpr int L = kMass ? 3 : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int CS = static_cast<int>(cl.num_blocks());
  uint32_t prefix = 0, pmask = 0;
  unsigned long long tau = target;
  unsigned long long tie_weight = 0;
  bool ok = true;
  int cur = 0;
  for (int d = 0; d < 4; ++d) {
    const int shift = 24 - 8 * d;
    const Bins<L> h{c.hist + cur * 3 * kBins, kBins};
    unsigned long long* s = c.sup + cur * kSuper;
    h.clear(kThreads);
    __syncthreads();
    src.for_each([&](bool valid, uint32_t key, int32_t idx, float x) {
      const bool take = valid && (key & pmask) == prefix && kept_by(key, idx, rk, ri);
      const int bin = static_cast<int>((key >> shift) & 0xFFu);
      if (kMass) {
        if (take) {
          const unsigned long long w = fixed_mass(softmax_weight(x, c.M));
          if (w) h.add(bin, w);
        }
      } else {
        if (take) h.add(bin, 1ull);
      }
    });
    __syncthreads();
    if (threadIdx.x < kBins) {
      unsigned long long v = h.get(threadIdx.x);
#pragma unroll
      for (int o = 8; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
      if ((threadIdx.x & 15) == 0) s[threadIdx.x >> 4] = v;
    }
    cl.sync();
    if (warp == 0) {
      // super-bins, largest keys first: lane l covers super-bin 15 - l
      const unsigned long long sv = lane < kSuper ? remote_sum(cl, s + (kSuper - 1 - (lane & 15)), CS) : 0ull;
      if (p_mode && d == 0) {
        unsigned long long total = sv;
#pragma unroll
        for (int o = 16; o; o >>= 1) total += __shfl_xor_sync(kFull, total, o);
        tau = ceil_mul_p(p, total);
      }
      const unsigned long long inc = warp_incl_scan_u64(sv, lane);
      const unsigned m = __ballot_sync(kFull, lane < kSuper && inc >= tau);
      unsigned long long bin_w = 0, new_tau = tau;
      int beta = 0;
      bool good = (m != 0u) && tau > 0;
      if (good) {
        const int L0 = __ffs(m) - 1;
        const unsigned long long above = L0 > 0 ? __shfl_sync(kFull, inc, L0 - 1) : 0ull;
        const int sigma = kSuper - 1 - L0;
        const unsigned long long bv = lane < 16 ? h.get_cluster(cl, sigma * 16 + (15 - (lane & 15)), CS) : 0ull;
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
  const unsigned long long w1 = kMass ? fixed_mass(softmax_weight(kfloat(key), c.M)) : 1ull;
  if (w1 == 0ull) return Thresh{key, key == rk ? ri : INT_MAX};
  const unsigned long long ties = tie_weight / w1;
  const unsigned long long need = (tau + w1 - 1) / w1;  // ties to keep, >= 1
  if (need >= ties) return Thresh{key, key == rk ? ri : INT_MAX};

  // Split inside the ties: the need-th tie in index order.  CTAs own contiguous
  // index ranges in rank order; the owner comes from the per-CTA tie counts
  // (the last pass's local histograms, still intact).
  const int last = cur ^ 1;
  const int beta_last = static_cast<int>(key & 0xFFu);
  const Bins<L> hl{c.hist + last * 3 * kBins, kBins};
  if (warp == 0) {
    unsigned long long t = 0;
    if (lane < CS) t = hl.get_rank(cl, beta_last, lane) / w1;
    const unsigned long long inc = warp_incl_scan_u64(t, lane);
    const unsigned m = __ballot_sync(kFull, lane < CS && inc >= need);
    int owner = -1;
    unsigned long long jloc = 0;
    if (m) {
      const int L0 = __ffs(m) - 1;
      const unsigned long long before = L0 > 0 ? __shfl_sync(kFull, inc, L0 - 1) : 0ull;
      owner = L0;
      jloc = need - before;
    }
    if (lane == 0) {
      c.misc[5] = static_cast<unsigned long long>(static_cast<long long>(owner));
      c.misc[6] = jloc;
    }
  }
  __syncthreads();
  const int owner = static_cast<int>(static_cast<long long>(c.misc[5]));
  const unsigned long long jloc = c.misc[6];
  __syncthreads();
  if (static_cast<int>(cl.block_rank()) == owner) {
    const int32_t f = nth_tie(src, c, key, rk, ri, static_cast<uint32_t>(jloc));
    if (threadIdx.x == 0)
      for (int r = 0; r < CS; ++r)
        *cl.map_shared_rank(c.slots + kSlotTie, r) = static_cast<unsigned long long>(static_cast<uint32_t>(f));
  }
  cl.sync();
  int32_t ti = static_cast<int32_t>(static_cast<uint32_t>(c.slots[kSlotTie]));
  if (owner < 0 || ti < 0) ti = (key == rk) ? ri : INT_MAX;  // degenerate: keep all ties
  return Thresh{key, ti};
}

// A lower bound on the k-th largest (1 <= k <= n) of n keys in shared memory: the lower
// edge of the bin that holds the k-th largest, the bins being the keys' offsets from the
// smallest key shifted right until at most kLinBins remain (one counting pass; the bound
// is at most one bin below the exact value).  Block-local; `h` is kLinBins words of
// scratch.
__device__ __noinline__ uint32_t local_kth_lower(Ctx& c, const uint32_t* keys, int n, uint32_t k, uint32_t* h) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t mx = 0u, mn = 0xFFFFFFFFu;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint32_t key = keys[i];
    mx = key > mx ? key : mx;
    mn = key < mn ? key : mn;
  }
  mx = __reduce_max_sync(kFull, mx);
  mn = __reduce_min_sync(kFull, mn);
  if (lane == 0) c.red[warp] = (static_cast<unsigned long long>(mx) << 32) | mn;
  for (int i = threadIdx.x; i < kLinBins; i += kThreads) h[i] = 0u;
  __syncthreads();
  {
    const unsigned long long v = c.red[lane & (kWarps - 1)];
    mx = __reduce_max_sync(kFull, static_cast<uint32_t>(v >> 32));
    mn = __reduce_min_sync(kFull, static_cast<uint32_t>(v));
  }
  __syncthreads();  // c.red is reused by the scan below
  const uint32_t span = mx - mn;
  if (span == 0u) return mn;
  // kLinBins = 2^11: keep the top 11 bits of the span
  const int used = 32 - __clz(span);
  const int shift = used > 11 ? used - 11 : 0;
  for (int i = threadIdx.x; i < n; i += kThreads) atomicAdd(&h[(keys[i] - mn) >> shift], 1u);
  __syncthreads();
  // thread t owns bins kLinBins-1-4t ... kLinBins-4-4t (largest first)
  constexpr int per = kLinBins / kThreads;
  uint32_t cnt[per];
  uint32_t sum = 0;
#pragma unroll
  for (int e = 0; e < per; ++e) {
    cnt[e] = h[kLinBins - 1 - (per * static_cast<int>(threadIdx.x) + e)];
    sum += cnt[e];
  }
  uint32_t tot;
  const uint32_t ex = block_excl_scan_u32(sum, &tot, c.red);
  if (ex < k && ex + sum >= k) {
    uint32_t acc = ex;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      if (acc < k && acc + cnt[e] >= k)
        c.misc[0] = static_cast<unsigned long long>(kLinBins - 1 - (per * static_cast<int>(threadIdx.x) + e));
      acc += cnt[e];
    }
  }
  __syncthreads();
  const uint32_t beta = static_cast<uint32_t>(c.misc[0]);
  __syncthreads();
  return mn + (beta << shift);  // the smallest key of bin beta
}

// After cl.sync: scans the cluster-wide histogram (nb bins in `h`, super sums
// of 32 bins in `sup`, both per CTA) in increasing bin order for the first bin
// where the cumulative weight reaches tau (p_mode: tau = ceil(p * total)).
struct Boundary {
  int beta;                 // -1 when no bin reaches tau
  unsigned long long above; // weight of the bins before beta
  unsigned long long binw;  // weight of bin beta
  unsigned long long tau;   // target used
};
template <int L>
__device__ __noinline__ Boundary find_boundary(cg::cluster_group& cl, Ctx& c, const Bins<L>& h, unsigned long long* sup,
                                  unsigned long long tau, bool p_mode, float p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int CS = static_cast<int>(cl.num_blocks());
  const int nsup = h.nb / 32;
  if (warp == 0) {
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    const unsigned long long s0 = i0 < nsup ? remote_sum(cl, sup + (i0 < nsup ? i0 : 0), CS) : 0ull;
    const unsigned long long s1 = i1 < nsup ? remote_sum(cl, sup + (i1 < nsup ? i1 : 0), CS) : 0ull;
    const unsigned long long inc = warp_incl_scan_u64(s0 + s1, lane);
    if (p_mode) {
      const unsigned long long total = __shfl_sync(kFull, inc, 31);
      tau = ceil_mul_p(p, total);
    }
    const unsigned m = __ballot_sync(kFull, inc >= tau && tau > 0);
    int beta = -1;
    unsigned long long above = 0, binw = 0;
    if (m) {
      const int Ls = __ffs(m) - 1;
      const unsigned long long before = Ls > 0 ? __shfl_sync(kFull, inc, Ls - 1) : 0ull;
      const unsigned long long s0L = __shfl_sync(kFull, s0, Ls);
      const int sigma = (before + s0L >= tau) ? 2 * Ls : 2 * Ls + 1;
      const unsigned long long abv = (sigma == 2 * Ls) ? before : before + s0L;
      const unsigned long long bv = h.get_cluster(cl, sigma * 32 + lane, CS);
      const unsigned long long inc2 = warp_incl_scan_u64(bv, lane);
      const unsigned m2 = __ballot_sync(kFull, abv + inc2 >= tau);
      if (m2) {
        const int L2 = __ffs(m2) - 1;
        above = abv + (L2 > 0 ? __shfl_sync(kFull, inc2, L2 - 1) : 0ull);
        binw = __shfl_sync(kFull, bv, L2);
        beta = sigma * 32 + L2;
      }
    }
    if (lane == 0) {
      c.misc[0] = static_cast<unsigned long long>(static_cast<long long>(beta));
      c.misc[1] = above;
      c.misc[2] = binw;
      c.misc[3] = tau;
    }
  }
  __syncthreads();
  Boundary b;
  b.beta = static_cast<int>(static_cast<long long>(c.misc[0]));
  b.above = c.misc[1];
  b.binw = c.misc[2];
  b.tau = c.misc[3];
  __syncthreads();
  return b;
}

// Super sums of 32 bins into sup; block-wide, before cl.sync.
template <int L>
__device__ __forceinline__ void super_sums(const Bins<L>& h, unsigned long long* sup) {
  for (int t = threadIdx.x; t < h.nb / 4; t += kThreads) {
    unsigned long long v = h.get(4 * t) + h.get(4 * t + 1) + h.get(4 * t + 2) + h.get(4 * t + 3);
    v += __shfl_xor_sync(kFull, v, 1);
    v += __shfl_xor_sync(kFull, v, 2);
    v += __shfl_xor_sync(kFull, v, 4);
    if ((t & 7) == 0) sup[t >> 3] = v;
  }
}

// After cl.sync: gathers every CTA's boundary list (order words, count in
// kSlotSmallCnt) into the second half of c.small and finds, among them, the
// element whose exclusive prefix weight in the order satisfies
// excl < need <= excl + w (count mode: w = 1; mass mode: w = fixed mass).
// Returns false (uniformly) if the lists do not fit.
template <bool kMass>
__device__ __noinline__ bool resolve_small(cg::cluster_group& cl, Ctx& c, unsigned long long need, Thresh* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int CS = static_cast<int>(cl.num_blocks());
  unsigned long long* all = c.small + kSmall;
  uint32_t* meta = reinterpret_cast<uint32_t*>(c.misc + 12);  // [0] total, [1] found
  uint32_t* offs = reinterpret_cast<uint32_t*>(c.red);       // [kMaxCS] list offsets
  if (warp == 0) {
    const uint32_t cnt = lane < CS ? static_cast<uint32_t>(*cl.map_shared_rank(c.slots + kSlotSmallCnt, lane)) : 0u;
    const uint32_t inc = warp_incl_scan_u32(cnt, lane);
    const uint32_t tot = __shfl_sync(kFull, inc, 31);
    const bool fits = __all_sync(kFull, cnt <= static_cast<uint32_t>(kSmall)) && tot <= static_cast<uint32_t>(kSmall);
    if (lane < CS) offs[lane] = inc - cnt;
    if (lane == 0) {
      meta[0] = fits ? tot : 0xFFFFFFFFu;
      meta[1] = 0u;
    }
  }
  __syncthreads();
  const uint32_t total = meta[0];
  if (total == 0xFFFFFFFFu) {
    __syncthreads();
    return false;
  }
  for (uint32_t t = threadIdx.x; t < total; t += kThreads) {
    int r = 0;
    while (r + 1 < CS && offs[r + 1] <= t) ++r;
    all[t] = *cl.map_shared_rank(c.small + (t - offs[r]), r);
  }
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < total; i += kThreads) {
    const unsigned long long wi = all[i];
    unsigned long long excl = 0, self = 1;
    if (kMass) self = fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(wi >> 32)), c.M));
    for (uint32_t j = 0; j < total; ++j) {
      const unsigned long long wj = all[j];
      if (wj > wi)
        excl += kMass ? fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(wj >> 32)), c.M)) : 1ull;
    }
    if (excl < need && need <= excl + self) {
      out->key = static_cast<uint32_t>(wi >> 32);
      out->idx = static_cast<int32_t>(~static_cast<uint32_t>(wi));
      meta[1] = 1u;
    }
  }
  __syncthreads();
  const bool ok = meta[1] != 0u;
  __syncthreads();
  return ok;
}

// Debug build (-DKPS_DEBUG_SENTINEL): every word of the block's dynamic shared memory
// starts as a NaN pattern, so a word read before any thread of the launch wrote it shows
// up as a wrong result instead of a previous launch's leftovers.  A barrier follows (a
// cluster barrier when the launch has clusters, so that no member pushes into a CTA that
// is still filling).  In other builds this is nothing.
__device__ __forceinline__ void debug_fill_smem(unsigned char* base, bool cluster) {
#ifdef KPS_DEBUG_SENTINEL
  uint32_t nbytes;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(nbytes));
  uint32_t* w = reinterpret_cast<uint32_t*>(base);
  for (uint32_t i = threadIdx.x; i < nbytes / 4; i += blockDim.x) w[i] = 0x7FBADBADu;
  if (cluster) {
    cg::this_cluster().sync();
  } else {
    __syncthreads();
  }
#else
  (void)base;
  (void)cluster;
#endif
}

// ------------------------------------------------------------------------------------------
// The kernel: a persistent grid of clusters, one row per cluster at a time.
// ------------------------------------------------------------------------------------------
template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 2) kps_sample_kernel(const Params P) {
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char smem[];
  debug_fill_smem(smem, true);
  const Layout L = make_layout(P.nc, kBF16);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L.cand_key);
  unsigned long long* mbar = reinterpret_cast<unsigned long long*>(smem + L.mbar);
  // block-shared scalars live in the dynamic layout (misc[14], misc[15])
  uint32_t& sh_cnt = *reinterpret_cast<uint32_t*>(smem + L.misc + 14 * 8);
  Thresh& sh_thresh = *reinterpret_cast<Thresh*>(smem + L.misc + 15 * 8);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const int CS = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int64_t V = P.V;
  const int32_t c0 = rank * P.nc;
  int n = static_cast<int>(V - c0);
  n = n < 0 ? 0 : (n > P.nc ? P.nc : n);
  const int n4 = (n + 3) >> 2;
  const size_t esize = kBF16 ? 2 : 4;
  const uint32_t bytes = static_cast<uint32_t>(n * esize);
  const bool tma = P.use_tma && bytes > 0;
  const int64_t cid = blockIdx.x / CS;
  const int64_t ncl = gridDim.x / CS;

  Ctx c;
  c.xs = xs;
  c.c0 = c0;
  c.n = n;
  c.n4 = n4;
  c.cand_key = reinterpret_cast<uint32_t*>(smem + L.cand_key);
  c.cand_idx = reinterpret_cast<int32_t*>(smem + L.cand_idx);
  c.hist = reinterpret_cast<uint32_t*>(smem + L.hist);
  c.fine = reinterpret_cast<uint32_t*>(smem + L.fine);
  c.sup = reinterpret_cast<unsigned long long*>(smem + L.sup);
  c.small = reinterpret_cast<unsigned long long*>(smem + L.small);
  c.gmax = reinterpret_cast<uint32_t*>(smem + L.gmax);
  c.red = reinterpret_cast<unsigned long long*>(smem + L.red);
  c.slots = reinterpret_cast<unsigned long long*>(smem + L.slots);
  c.misc = reinterpret_cast<unsigned long long*>(smem + L.misc);

  void* stage = kBF16 ? static_cast<void*>(smem + L.raw) : static_cast<void*>(xs);
  auto gsrc_of = [&](int64_t row) {
    return static_cast<const unsigned char*>(P.logits) + (row * V + c0) * esize;
  };
  // dead: a copy of this CTA did not land within two bounds; no further copies are issued
  // (block-uniform, decided by a barrier vote)
  bool dead = false;
  uint32_t dead_parity = 0;
  auto issue_load = [&](int64_t row) {
    if (tma && !dead && threadIdx.x == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_expect_tx(mbar, bytes);
      // one bulk copy per chunk: a copy's cost is mostly fixed, not proportional to its size
      constexpr uint32_t kPiece = 1u << 20;
      const unsigned char* src = gsrc_of(row);
      for (uint32_t off = 0; off < bytes; off += kPiece) {
        const uint32_t len = bytes - off < kPiece ? bytes - off : kPiece;
        bulk_g2s(static_cast<unsigned char*>(stage) + off, src + off, len, mbar);
      }
    }
  };

  // the rows this cluster owns (every CTA of the cluster computes the same list)
  int32_t* rowlist = reinterpret_cast<int32_t*>(smem + L.rows);
  int my_rows = 0;
  if (P.filter == 0) {
    my_rows = P.B > cid ? static_cast<int>((P.B - 1 - cid) / ncl + 1) : 0;
  } else {
    my_rows = build_row_list<kThreads>(P, cid, ncl, rowlist, c.red);
  }
  auto row_at = [&](int i) -> int64_t {
    return P.filter == 0 ? cid + static_cast<int64_t>(i) * ncl : static_cast<int64_t>(rowlist[i]);
  };

  if (threadIdx.x == 0) mbar_init(mbar, 1);
#ifdef KPS_TEST_SPIN_CYCLES
  // test build: the first wait goes to a second barrier that no copy completes, with a
  // bound of KPS_TEST_SPIN_CYCLES, so that the timeout path below runs deterministically
  if (threadIdx.x == 0) mbar_init(mbar + 1, 1);
#endif
  __syncthreads();
  if (my_rows > 0) issue_load(row_at(0));
  uint32_t parity = 0;

  // groups of 128 elements over the row (the last CTA's partial group included)
  int G128 = 0;
  for (int r = 0; r < CS; ++r) {
    int nr = static_cast<int>(V - static_cast<int64_t>(r) * P.nc);
    nr = nr < 0 ? 0 : (nr > P.nc ? P.nc : nr);
    G128 += (((nr + 3) >> 2) + 31) >> 5;
  }

  for (int ri = 0; ri < my_rows; ++ri, parity ^= 1u) {
    const int64_t row = row_at(ri);
    const int64_t next = ri + 1 < my_rows ? row_at(ri + 1) : -1;
    bool next_issued = false;

    // ---- row parameters (uniform across the cluster) ---------------------------------
    const int32_t k = P.top_k[row];
    const float p = P.top_p[row];
    const float T = P.temperature[row];
    const bool greedyT = !(T > 0.0f) || isinf(T);
    const bool pen_on = ((P.seen_indptr && P.seen_ids) || P.seen_bits) && P.penalty && (P.penalty[row] > 0.0f);
    const float pen = pen_on ? P.penalty[row] : 1.0f;
    const bool pen_bits = pen_on && P.seen_bits;
    const bool topk_on = k >= 1 && static_cast<int64_t>(k) <= (V < kTopKMax ? V : kTopKMax);
    const bool p_nan = isnan(p);
    const bool single = greedyT || (!p_nan && p <= 0.0f) || (topk_on && k == 1);
    const bool topp_on = !single && !p_nan && p > 0.0f && p < 1.0f;
    // top-k bound: split the 128-element groups until there are at least k of them
    // (while the gathered maxima still fit kGallCap)
    int gsh = 0;
    if (topk_on && !single)
      while ((1 << gsh) < kGroupSplit && (G128 << gsh) < k && (G128 << (gsh + 1)) <= kGallCap) ++gsh;

    // prefetch up to four seen ids per thread while the chunk is in flight
    int32_t pid[4];
    int32_t b0 = 0, b1 = 0;
    if (pen_bits) {
      // the chunk's seen bits: bit li of word w is token c0 + 32 w + li (a chunk starts on
      // a multiple of 8, so a word of it may straddle two words of the row)
      const uint32_t* rb = P.seen_bits + row * seen_words(V);
      const int sh = c0 & 31;
      const int64_t w0 = c0 >> 5;
      for (int w = threadIdx.x; w < (n + 31) / 32; w += kThreads) {
        const uint32_t lo = seen_word_at(rb, V, w0 + w);
        const uint32_t hi = sh ? seen_word_at(rb, V, w0 + w + 1) : 0u;
        uint32_t x = __funnelshift_r(lo, hi, sh);
        const int left = n - 32 * w;  // chunk elements in this word
        if (left < 32) x &= (1u << left) - 1u;
        bitmap[w] = x;
      }
    } else if (pen_on) {
      b0 = P.seen_indptr[row];
      b1 = P.seen_indptr[row + 1];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int32_t j = b0 + threadIdx.x + u * kThreads;
        pid[u] = j < b1 ? P.seen_ids[j] : -1;
      }
      for (int w = threadIdx.x; w < (n + 31) / 32; w += kThreads) bitmap[w] = 0u;
    }

    // ---- wait for the chunk --------------------------------------------------------
    if (!tma) {
      const unsigned char* src = gsrc_of(row);
      for (int i = threadIdx.x; i < n; i += kThreads) {
        if (kBF16) xs[i] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(src)[i]);
        else xs[i] = reinterpret_cast<const float*>(src)[i];
      }
    } else if (!dead) {
#ifdef KPS_TEST_SPIN_CYCLES
      const bool ok = ri == 0 ? mbar_wait_bounded(mbar + 1, 0u, KPS_TEST_SPIN_CYCLES) : mbar_wait_bounded(mbar, parity);
#else
      const bool ok = mbar_wait_bounded(mbar, parity);
#endif
      if (__syncthreads_or(!ok)) {
        // the copy did not land in time: report it, and give it one more bound before its
        // buffer is read (or reused by the next row's copy)
        if (threadIdx.x == 0) atomicMax(P.status, kStatusTimeout);
        const bool late = mbar_wait_bounded(mbar, parity);
        if (__syncthreads_or(!late)) {
          dead = true;
          dead_parity = parity;
        }
      }
      if (kBF16) {
        const __nv_bfloat16* raw = reinterpret_cast<const __nv_bfloat16*>(smem + L.raw);
        for (int i = threadIdx.x; i < n; i += kThreads) xs[i] = __bfloat162float(raw[i]);
      }
    }
    __syncthreads();

    // ---- repetition penalty: scatter over the seen ids, once per distinct id -----------
    if (pen_bits) {
      for (int w = threadIdx.x; w < (n + 31) / 32; w += kThreads) {
        for (uint32_t x = bitmap[w]; x; x &= x - 1u) {
          const int li = 32 * w + __ffs(x) - 1;
          const float s = xs[li];
          xs[li] = (s > 0.0f) ? __fdiv_rn(s, pen) : __fmul_rn(s, pen);
        }
      }
      __syncthreads();
    } else if (pen_on) {
      auto apply = [&](int32_t id) {
        const int32_t li = id - c0;
        if (id >= 0 && static_cast<int64_t>(id) < V && li >= 0 && li < n) {
          const uint32_t bit = 1u << (li & 31);
          const uint32_t old = atomicOr(&bitmap[li >> 5], bit);
          if (!(old & bit)) {
            const float s = xs[li];
            xs[li] = (s > 0.0f) ? __fdiv_rn(s, pen) : __fmul_rn(s, pen);
          }
        }
      };
#pragma unroll
      for (int u = 0; u < 4; ++u) apply(pid[u]);
      for (int32_t j = b0 + threadIdx.x + 4 * kThreads; j < b1; j += kThreads) apply(P.seen_ids[j]);
      __syncthreads();
    }

    // ---- raw pass: NaN -> -inf, -0 -> +0, padding, group maxima, chunk maximum --------
    uint32_t tmax = 0;
    {
      float4* x4 = reinterpret_cast<float4*>(xs);
      for (int base = 0; base < n4; base += kThreads) {
        const int g = base + threadIdx.x;
        uint32_t gk = 0;
        if (g < n4) {
          const float4 v = x4[g];
          float vv[4] = {v.x, v.y, v.z, v.w};
          bool changed = false;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = vv[e];
            float y;
            if (4 * g + e >= n) y = __uint_as_float(0xFFFFFFFFu);  // padding: key 0
            else y = isnan(x) ? -INFINITY : __fadd_rn(x, 0.0f);
            changed |= __float_as_uint(y) != __float_as_uint(x);
            const uint32_t key = fkey(y);
            gk = key > gk ? key : gk;
            vv[e] = y;
          }
          if (changed) x4[g] = make_float4(vv[0], vv[1], vv[2], vv[3]);
        }
        // the warp's 32 float4s are 1 << gsh groups of 128 >> gsh consecutive elements
        tmax = gk > tmax ? gk : tmax;
        if (gsh == 0) {
          gk = __reduce_max_sync(kFull, gk);
        } else {
          for (int o = 16 >> gsh; o; o >>= 1) {
            const uint32_t y = __shfl_xor_sync(kFull, gk, o);
            gk = y > gk ? y : gk;
          }
        }
        if ((lane & ((32 >> gsh) - 1)) == 0 && base + 32 * warp < n4)
          c.gmax[(((base >> 5) + warp) << gsh) + (lane >> (5 - gsh))] = gk;
      }
    }
    {
      const unsigned long long m = block_max_u64(tmax, c.red);
      if (threadIdx.x == 0) push_all(cl, c.slots + kSlotMax, rank, CS, m);
      cl.sync();
    }
    const uint32_t mraw_key = static_cast<uint32_t>(max_of(c.slots + kSlotMax, CS));
    const float Mraw = kfloat(mraw_key);
    const float M = greedyT ? Mraw : __fdiv_rn(Mraw, T);  // max of x / T is (max x) / T
    c.M = M;
    const uint32_t mkey = fkey(M);

    float* orow = P.need_logits ? P.out_filtered + row * V + c0 : nullptr;
    bool neg_inf_written = false;
    auto write_neg_inf = [&]() {
      if (P.use_tma && (n & 3) == 0) {
        const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        for (int g = threadIdx.x; g < n4; g += kThreads) __stcs(reinterpret_cast<float4*>(orow) + g, ninf);
      } else {
        for (int i = threadIdx.x; i < n; i += kThreads) orow[i] = -INFINITY;
      }
      neg_inf_written = true;
    };

    Thresh th{0u, -1};  // keeps every real element (padding has key 0)
    int32_t chosen = -1;
    bool cand_mode = false;  // kept set and values live in the candidate lists
    int ncand = 0;
    bool transformed = greedyT;  // xs holds transformed values

    auto transform_in_place = [&]() {
      if (transformed) return;
      float4* x4 = reinterpret_cast<float4*>(xs);
      for (int g = threadIdx.x; g < n4; g += kThreads) {
        float4 v = x4[g];
        if (4 * g + 0 < n) v.x = __fdiv_rn(v.x, T);
        if (4 * g + 1 < n) v.y = __fdiv_rn(v.y, T);
        if (4 * g + 2 < n) v.z = __fdiv_rn(v.z, T);
        if (4 * g + 3 < n) v.w = __fdiv_rn(v.w, T);
        x4[g] = v;
      }
      __syncthreads();
      transformed = true;
    };
    // First element of the order among this CTA's elements whose transformed value
    // equals M, pushed and reduced over the cluster.
    auto first_of_order = [&]() -> int32_t {
      const float lo = transformed ? M : raw_lower_bound(Mraw, M, T);
      unsigned long long b = 0;
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const float x = xs[i];
        if (!(x >= lo)) continue;
        const float y = transformed ? x : __fdiv_rn(x, T);
        if (fkey(y) == mkey) {
          const unsigned long long w = order_word(mkey, c0 + i);
          b = w > b ? w : b;
        }
      }
      b = block_max_u64(b, c.red);
      if (threadIdx.x == 0) push_all(cl, c.slots + kSlotV0, rank, CS, b);
      cl.sync();
      return static_cast<int32_t>(~static_cast<uint32_t>(max_of(c.slots + kSlotV0, CS)));
    };

    if (single) {
      // ---- one element kept: the first of the order -----------------------------
      chosen = first_of_order();
      th = Thresh{mkey, chosen};
    } else if (topk_on) {
      // ---- top-k: lower bound from the group maxima ------------------------------
      const int ng_full = ((P.nc + 127) / 128) << gsh;
      const int G = G128 << gsh;
      bool fast = G >= k && G <= kGallCap;
      if (fast) {
        uint32_t* gall = reinterpret_cast<uint32_t*>(c.hist) + kBins;  // after the 256 count words
        for (int i = threadIdx.x; i < G; i += kThreads) {
          const int r = i / ng_full, j = i - r * ng_full;
          gall[i] = *cl.map_shared_rank(c.gmax + j, r);
        }
        __syncthreads();
        uint32_t gkey = local_kth_lower(c, gall, G, static_cast<uint32_t>(k), c.fine);
        if (gkey < kKeyNegInf) gkey = kKeyNegInf;
        const float g = kfloat(gkey);  // <= the k-th largest raw group maximum
        const float t0 = __fdiv_rn(g, T);
        const uint32_t t0key = fkey(t0);
        const float lo = raw_lower_bound(g, t0, T);
        const float span = __fsub_rn(M, t0);
        const float s = (span > 0.0f && span < INFINITY) ? __fdiv_rn(static_cast<float>(kLinBins), span) : 0.0f;
        // candidate pass: count histogram over linear bins of (M - y)
        __syncthreads();  // gall (inside hist) is dead from here
        const Bins<1> hk{c.hist, kLinBins};
        hk.clear(kThreads);
        if (threadIdx.x == 0) sh_cnt = 0u;
        __syncthreads();
        const float4* x4 = reinterpret_cast<const float4*>(xs);
        for (int base = 0; base < n4; base += kThreads) {
          const int gi = base + threadIdx.x;
          uint32_t ck[4] = {0u, 0u, 0u, 0u};
          int cnt = 0;
          if (gi < n4) {
            const float4 v = x4[gi];
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (vv[e] >= lo && fkey(vv[e]) != 0u) {
                const float y = __fdiv_rn(vv[e], T);
                const uint32_t ky = fkey(y);
                if (ky >= t0key) {
                  ck[e] = ky;
                  ++cnt;
                  const int b = s > 0.0f ? lin_bin_scaled(y, M, s, kLinBins) : 0;
                  hk.add(b, 1ull);
                }
              }
            }
          }
          const uint32_t incl = warp_incl_scan_u32(static_cast<uint32_t>(cnt), lane);
          const uint32_t wtot = __shfl_sync(kFull, incl, 31);
          if (wtot) {
            uint32_t wb = 0;
            if (lane == 31) wb = atomicAdd(&sh_cnt, wtot);
            wb = __shfl_sync(kFull, wb, 31);
            uint32_t pos = wb + incl - cnt;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (ck[e]) {
                if (pos < static_cast<uint32_t>(kCapLoc)) {
                  c.cand_key[pos] = ck[e];
                  c.cand_idx[pos] = c0 + 4 * gi + e;
                }
                ++pos;
              }
            }
          }
        }
        // the filtered output is -inf outside the kept set: stream it now, the kept
        // values are scattered over it at the end of the row
        if (orow) write_neg_inf();
        __syncthreads();
        ncand = static_cast<int>(sh_cnt);
        super_sums(hk, c.sup);
        if (threadIdx.x == 0) push_all(cl, c.slots + kSlotFlag, rank, CS, static_cast<unsigned long long>(ncand));
        cl.sync();
        bool lists_ok = true;
        uint32_t coff = 0, ctot = 0;  // this CTA's offset among the cluster's candidates, their count
        for (int r = 0; r < CS; ++r) {
          const uint32_t nr = static_cast<uint32_t>(c.slots[kSlotFlag + r]);
          lists_ok = lists_ok && nr <= static_cast<uint32_t>(kCapLoc);
          coff += r < rank ? nr : 0u;
          ctot += nr;
        }
        if (lists_ok && ctot >= static_cast<uint32_t>(k) && ctot <= static_cast<uint32_t>(kGatherTopP)) {
          // few candidates: rank 0 gathers all of them and takes the k-th (and the top-p cut
          // over the k survivors) by pairwise ranks; no cluster histogram, no boundary search
          unsigned long long* gw = reinterpret_cast<unsigned long long*>(c.fine);  // rank 0: words
          unsigned long long* gm = gw + kGatherTopP;                                // masses
          uint32_t* gr = reinterpret_cast<uint32_t*>(gw + 2 * kGatherTopP);         // ranks
          for (int i = threadIdx.x; i < ncand; i += kThreads)
            *cl.map_shared_rank(gw + coff + i, 0) = order_word(c.cand_key[i], c.cand_idx[i]);
          cl.sync();  // rank 0 holds the candidates
          if (rank == 0) {
            if (threadIdx.x == 0) c.misc[13] = ~0ull;
            for (uint32_t i = threadIdx.x; i < ctot; i += kThreads) {
              const unsigned long long wi = gw[i];
              uint32_t r = 0;
              for (uint32_t j = 0; j < ctot; ++j) r += gw[j] > wi ? 1u : 0u;
              gr[i] = r;
              if (r == static_cast<uint32_t>(k) - 1u) c.misc[13] = wi;  // the k-th: the top-k cut
            }
            __syncthreads();
            if (threadIdx.x == 0) c.misc[12] = c.misc[13];
            __syncthreads();
            if (topp_on) {
              unsigned long long part = 0;
              for (uint32_t i = threadIdx.x; i < ctot; i += kThreads) {
                gm[i] = gr[i] < static_cast<uint32_t>(k)
                            ? fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(gw[i] >> 32)), M))
                            : 0ull;
                part += gm[i];
              }
              const unsigned long long S = block_sum_u64(part, c.red);
              const unsigned long long tq = ceil_mul_p(p, S);
              if (S > 0ull) {
                for (uint32_t i = threadIdx.x; i < ctot; i += kThreads) {
                  if (gr[i] >= static_cast<uint32_t>(k)) continue;
                  const unsigned long long wi = gw[i];
                  unsigned long long excl = 0;
                  for (uint32_t j = 0; j < ctot; ++j) excl += gw[j] > wi ? gm[j] : 0ull;
                  if (excl < tq && tq <= excl + gm[i]) c.misc[12] = wi;  // the top-p cut
                }
              }
              __syncthreads();
              if (threadIdx.x == 0 && S > 0ull) c.misc[13] = c.misc[12];
              __syncthreads();
            }
            if (threadIdx.x == 0) {
              for (int r = 0; r < CS; ++r) *cl.map_shared_rank(c.slots + kSlotTie, r) = c.misc[13];
            }
          }
          cl.sync();  // every CTA holds the cut
          const unsigned long long cut = c.slots[kSlotTie];
          th = Thresh{static_cast<uint32_t>(cut >> 32), static_cast<int32_t>(~static_cast<uint32_t>(cut))};
          cand_mode = true;
          if (next >= 0) {
            issue_load(next);
            next_issued = true;
          }
          fast = false;  // the general search below is not needed
        } else {
        const Boundary bk = find_boundary(cl, c, hk, c.sup, static_cast<unsigned long long>(k), false, 0.0f);
        fast = lists_ok && bk.beta >= 0 && bk.binw <= static_cast<unsigned long long>(kSmall);
        if (fast) {
          // the k-th element lies in bin beta: rank that bin's elements exactly
          if (threadIdx.x == 0) sh_cnt = 0u;
          __syncthreads();
          for (int i = threadIdx.x; i < ncand; i += kThreads) {
            const uint32_t key = c.cand_key[i];
            const int b = s > 0.0f ? lin_bin_scaled(kfloat(key), M, s, kLinBins) : 0;
            if (b == bk.beta) {
              const uint32_t pos = atomicAdd(&sh_cnt, 1u);
              if (pos < static_cast<uint32_t>(kSmall)) c.small[pos] = order_word(key, c.cand_idx[i]);
            }
          }
          __syncthreads();
          if (threadIdx.x == 0) c.slots[kSlotSmallCnt] = sh_cnt;
          cl.sync();
          Thresh tk{0u, -1};
          if (threadIdx.x == 0) sh_thresh = Thresh{0u, -1};
          __syncthreads();
          fast = resolve_small<false>(cl, c, static_cast<unsigned long long>(k) - bk.above, &sh_thresh);
          tk = sh_thresh;
          __syncthreads();
          if (fast) {
            // the chunk is no longer needed: start the next row's load now
            __syncthreads();
            if (next >= 0) {
              issue_load(next);
              next_issued = true;
            }
            cand_mode = true;
            th = tk;
            bool topp_done = false;
            if (topp_on && k <= kGatherTopP) {
              // few survivors: rank 0 gathers the k of them from every CTA and cuts top-p
              // over them alone by pairwise ranks (no cluster histogram, no boundary search)
              if (threadIdx.x == 0) sh_cnt = 0u;
              __syncthreads();
              uint32_t mine = 0;
              for (int i = threadIdx.x; i < ncand; i += kThreads)
                mine += kept_by(c.cand_key[i], c.cand_idx[i], tk.key, tk.idx) ? 1u : 0u;
              mine = __reduce_add_sync(kFull, mine);
              if (lane == 0 && mine) atomicAdd(&sh_cnt, mine);
              __syncthreads();
              if (threadIdx.x == 0) push_all(cl, c.slots + kSlotFlag, rank, CS, sh_cnt);
              cl.sync();
              uint32_t off = 0, total = 0;
              for (int r = 0; r < CS; ++r) {
                const uint32_t nr = static_cast<uint32_t>(c.slots[kSlotFlag + r]);
                off += r < rank ? nr : 0u;
                total += nr;
              }
              unsigned long long* gw = reinterpret_cast<unsigned long long*>(c.fine);  // rank 0: words
              unsigned long long* gm = gw + kGatherTopP;                                // and masses
              if (total <= static_cast<uint32_t>(kGatherTopP)) {
                if (threadIdx.x == 0) sh_cnt = 0u;
                __syncthreads();
                for (int i = threadIdx.x; i < ncand; i += kThreads) {
                  if (!kept_by(c.cand_key[i], c.cand_idx[i], tk.key, tk.idx)) continue;
                  const uint32_t pos = off + atomicAdd(&sh_cnt, 1u);
                  *cl.map_shared_rank(gw + pos, 0) = order_word(c.cand_key[i], c.cand_idx[i]);
                }
              }
              cl.sync();  // rank 0 holds the survivors
              if (rank == 0) {
                unsigned long long part = 0;
                if (total <= static_cast<uint32_t>(kGatherTopP)) {
                  for (uint32_t i = threadIdx.x; i < total; i += kThreads) {
                    gm[i] = fixed_mass(softmax_weight(kfloat(static_cast<uint32_t>(gw[i] >> 32)), M));
                    part += gm[i];
                  }
                }
                const unsigned long long S = block_sum_u64(part, c.red);
                const unsigned long long tq = ceil_mul_p(p, S);
                if (threadIdx.x == 0) c.misc[13] = ~0ull;  // not found
                __syncthreads();
                if (total <= static_cast<uint32_t>(kGatherTopP) && S > 0ull) {
                  for (uint32_t i = threadIdx.x; i < total; i += kThreads) {
                    const unsigned long long wi = gw[i];
                    unsigned long long excl = 0;
                    for (uint32_t j = 0; j < total; ++j) excl += gw[j] > wi ? gm[j] : 0ull;
                    if (excl < tq && tq <= excl + gm[i]) c.misc[13] = wi;
                  }
                }
                __syncthreads();
                if (threadIdx.x == 0) {
                  for (int r = 0; r < CS; ++r) *cl.map_shared_rank(c.slots + kSlotTie, r) = c.misc[13];
                }
              }
              cl.sync();  // every CTA holds the cut (or ~0: take the general path)
              const unsigned long long cut = c.slots[kSlotTie];
              if (cut != ~0ull) {
                th = Thresh{static_cast<uint32_t>(cut >> 32), static_cast<int32_t>(~static_cast<uint32_t>(cut))};
                topp_done = true;
              }
            }
            if (topp_on && !topp_done) {
              // mass histogram of the k survivors over linear bins of (M - y)
              const float xk = kfloat(tk.key);
              const float span2 = __fsub_rn(M, xk);
              const float s2 =
                  (span2 > 0.0f && span2 < INFINITY) ? __fdiv_rn(static_cast<float>(kLinBins), span2) : 0.0f;
              // hist is still read by other CTAs until the next barrier: use `fine` as a
              // 1024-bin histogram (half resolution)
              const Bins<3> hm{c.fine, kFineBins};
              hm.clear(kThreads);
              __syncthreads();
              for (int i = threadIdx.x; i < ncand; i += kThreads) {
                const uint32_t key = c.cand_key[i];
                if (!kept_by(key, c.cand_idx[i], tk.key, tk.idx)) continue;
                const float y = kfloat(key);
                const int b = s2 > 0.0f ? (lin_bin_scaled(y, M, s2, kLinBins) >> 1) : 0;
                const unsigned long long w = fixed_mass(softmax_weight(y, M));
                if (w) hm.add(b, w);
              }
              __syncthreads();
              super_sums(hm, c.sup);
              cl.sync();
              const Boundary bp = find_boundary(cl, c, hm, c.sup, 0ull, true, p);
              bool ok2 = bp.beta >= 0;
              if (ok2) {
                if (threadIdx.x == 0) sh_cnt = 0u;
                __syncthreads();
                for (int i = threadIdx.x; i < ncand; i += kThreads) {
                  const uint32_t key = c.cand_key[i];
                  if (!kept_by(key, c.cand_idx[i], tk.key, tk.idx)) continue;
                  const int b = s2 > 0.0f ? (lin_bin_scaled(kfloat(key), M, s2, kLinBins) >> 1) : 0;
                  if (b == bp.beta) {
                    const uint32_t pos = atomicAdd(&sh_cnt, 1u);
                    if (pos < static_cast<uint32_t>(kSmall)) c.small[pos] = order_word(key, c.cand_idx[i]);
                  }
                }
                __syncthreads();
                if (threadIdx.x == 0) c.slots[kSlotSmallCnt] = sh_cnt;
              }
              cl.sync();
              if (ok2) {
                if (threadIdx.x == 0) sh_thresh = tk;
                __syncthreads();
                ok2 = resolve_small<true>(cl, c, bp.tau - bp.above, &sh_thresh);
                th = sh_thresh;
                __syncthreads();
              }
              if (!ok2) {
                const SrcCand scand{c.cand_key, c.cand_idx, ncand};
                th = radix_select<SrcCand, true>(cl, c, scand, 0ull, true, p, tk.key, tk.idx);
              }
            }
          }
        }
        }
      }
      if (!cand_mode) {
        // exact fallback over the whole resident row; the barrier first lets every CTA
        // finish reading the histograms the fast attempt left in shared memory
        cl.sync();
        transform_in_place();
        const SrcData sdata{xs, n4, c0};
        const Thresh tk = radix_select<SrcData, false>(cl, c, sdata, static_cast<unsigned long long>(k), false,
                                                       0.0f, 0u, -1);
        th = tk;
        if (topp_on) th = radix_select<SrcData, true>(cl, c, sdata, 0ull, true, p, tk.key, tk.idx);
      }
    } else if (topp_on) {
      // ---- top-p over the whole row ----------------------------------------------
      transform_in_place();
      const Bins<3> h{c.hist, kLinBinsP};
      h.clear(kThreads);
      __syncthreads();
      const float4* x4 = reinterpret_cast<const float4*>(xs);
      for (int g = threadIdx.x; g < n4; g += kThreads) {
        const float4 v = x4[g];
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (fkey(vv[e]) == 0u) continue;
          const int b = lin_bin_mass(vv[e], M);
          if (b < kLinBinsP) {
            const unsigned long long w = fixed_mass(softmax_weight(vv[e], M));
            if (w) h.add(b, w);
          }
        }
      }
      __syncthreads();
      super_sums(h, c.sup);
      cl.sync();
      const Boundary b1 = find_boundary(cl, c, h, c.sup, 0ull, true, p);
      bool ok = b1.beta >= 0;
      Boundary b2{-1, 0, 0, 0};
      if (ok) {
        // finer histogram inside bin beta (into `fine`; hist is still being read)
        const Bins<3> hf{c.fine, kFineBins};
        hf.clear(kThreads);
        __syncthreads();
        for (int g = threadIdx.x; g < n4; g += kThreads) {
          const float4 v = x4[g];
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (fkey(vv[e]) == 0u || lin_bin_mass(vv[e], M) != b1.beta) continue;
            const unsigned long long w = fixed_mass(softmax_weight(vv[e], M));
            if (w) hf.add(fine_bin_mass(vv[e], M, b1.beta), w);
          }
        }
        __syncthreads();
        // super sums go to the second half of sup (the first half is still being read)
        super_sums(hf, c.sup + kLinBinsP / 32);
      }
      cl.sync();
      if (ok) {
        b2 = find_boundary(cl, c, Bins<3>{c.fine, kFineBins}, c.sup + kLinBinsP / 32, b1.tau - b1.above, false, 0.0f);
        ok = b2.beta >= 0;
      }
      if (ok) {
        if (threadIdx.x == 0) sh_cnt = 0u;
        __syncthreads();
        for (int g = threadIdx.x; g < n4; g += kThreads) {
          const float4 v = x4[g];
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t key = fkey(vv[e]);
            if (key == 0u || lin_bin_mass(vv[e], M) != b1.beta || fine_bin_mass(vv[e], M, b1.beta) != b2.beta) continue;
            const uint32_t pos = atomicAdd(&sh_cnt, 1u);
            if (pos < static_cast<uint32_t>(kSmall)) c.small[pos] = order_word(key, c0 + 4 * g + e);
          }
        }
        __syncthreads();
        if (threadIdx.x == 0) c.slots[kSlotSmallCnt] = sh_cnt;
      }
      cl.sync();
      if (ok) {
        if (threadIdx.x == 0) sh_thresh = Thresh{0u, -1};
        __syncthreads();
        ok = resolve_small<true>(cl, c, b2.tau - b2.above, &sh_thresh);
        th = sh_thresh;
        __syncthreads();
      }
      if (!ok) {
        const SrcData sdata{xs, n4, c0};
        th = radix_select<SrcData, true>(cl, c, sdata, 0ull, true, p, 0u, -1);
      }
    } else {
      transform_in_place();  // top-k and top-p both skipped: every element is kept
    }

    // ---- exponential race over the kept set, and the filtered-logit write --------------
    const float* qrow = P.q ? P.q + row * V : nullptr;  // none: sampling off or generated draws
    const bool race = qrow != nullptr || P.gen != 0;
    unsigned long long rb = 0;
    if (single || (cand_mode && !race)) {
      // nothing to race (sampling off takes the first element of the order below)
    } else if (cand_mode) {
      for (int i = threadIdx.x; i < ncand; i += kThreads) {
        const uint32_t key = c.cand_key[i];
        const int32_t idx = c.cand_idx[i];
        if (!kept_by(key, idx, th.key, th.idx)) continue;
        const float w = softmax_weight(kfloat(key), M);
        const float qv = P.gen ? gen_q1(P.seed, P.step, row, idx) : __ldg(qrow + idx);
        const float r = __fdiv_rn(w, __fadd_rn(qv, P.eps));
        if (isnan(r)) continue;
        const unsigned long long cand = order_word(fkey(r), idx);
        rb = cand > rb ? cand : rb;
      }
    } else {
      const bool vec = P.use_tma != 0 && (n & 3) == 0;
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
        if (orow) {
          if (vec) {
            __stcs(reinterpret_cast<float4*>(orow) + g,
                   make_float4(kp[0] ? vv[0] : -INFINITY, kp[1] ? vv[1] : -INFINITY, kp[2] ? vv[2] : -INFINITY,
                               kp[3] ? vv[3] : -INFINITY));
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (4 * g + e < n) orow[4 * g + e] = kp[e] ? vv[e] : -INFINITY;
          }
        }
        if (!nk || !race) continue;
        float qq[4];
        if (P.gen) {
          // c0 is a multiple of 4: the group's four draws in one generator block
          const float4 q4 = gen_q4(P.seed, P.step, row, (c0 >> 2) + g);
          qq[0] = q4.x; qq[1] = q4.y; qq[2] = q4.z; qq[3] = q4.w;
        } else if (nk == 4 && vec) {
          const float4 q4 = __ldcs(reinterpret_cast<const float4*>(qrow + c0) + g);
          qq[0] = q4.x; qq[1] = q4.y; qq[2] = q4.z; qq[3] = q4.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) qq[e] = kp[e] ? __ldcs(qrow + c0 + 4 * g + e) : 0.0f;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (!kp[e]) continue;
          const float w = softmax_weight(vv[e], M);
          const float r = __fdiv_rn(w, __fadd_rn(qq[e], P.eps));
          if (isnan(r)) continue;
          const unsigned long long cand = order_word(fkey(r), c0 + 4 * g + e);
          rb = cand > rb ? cand : rb;
        }
      }
    }
    if (!single) {
      rb = block_max_u64(rb, c.red);
      if (threadIdx.x == 0) push_all(cl, c.slots + kSlotRace, rank, CS, rb);
      cl.sync();
      rb = max_of(c.slots + kSlotRace, CS);
      if (rb != 0ull) {
        chosen = static_cast<int32_t>(~static_cast<uint32_t>(rb));
      } else if (cand_mode) {
        // every score was NaN: the first element of the order (the best candidate)
        unsigned long long b = 0;
        for (int i = threadIdx.x; i < ncand; i += kThreads) {
          const unsigned long long w = order_word(c.cand_key[i], c.cand_idx[i]);
          b = w > b ? w : b;
        }
        b = block_max_u64(b, c.red);
        if (threadIdx.x == 0) push_all(cl, c.slots + kSlotV0, rank, CS, b);
        cl.sync();
        chosen = static_cast<int32_t>(~static_cast<uint32_t>(max_of(c.slots + kSlotV0, CS)));
      } else {
        chosen = first_of_order();
      }
    }

    // filtered logits for the paths that did not write them above
    if (orow && (single || cand_mode)) {
      if (!neg_inf_written) write_neg_inf();
      __syncthreads();
      if (single) {
        if (threadIdx.x == 0 && th.idx >= c0 && th.idx < c0 + n) orow[th.idx - c0] = M;
      } else {
        for (int i = threadIdx.x; i < ncand; i += kThreads)
          if (kept_by(c.cand_key[i], c.cand_idx[i], th.key, th.idx)) orow[c.cand_idx[i] - c0] = kfloat(c.cand_key[i]);
      }
    }
    if (rank == 0 && threadIdx.x == 0) {
      const long long tok = eos_epilogue(P, row, chosen);
      P.out_idx[row] = tok;
      seen_append(P, row, tok);
    }

    // the chunk buffer is free: start the next row's load if it has not started yet
    __syncthreads();
    if (!next_issued && next >= 0) issue_load(next);
  }

  // a CTA that gave up on a copy waits (bounded) for it once more before leaving
  if (dead) (void)mbar_wait_bounded(mbar, dead_parity);
  // no CTA leaves while another may still read its shared memory
  cl.sync();
}


#include "kps_row.cuh"

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
struct LaunchCfg {
  int cs;
  int nc;
  size_t smem;
  int clusters;  // clusters that can be resident at once (the persistent grid size)
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
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, kps_sample_kernel<kBF16>);
  if (err != cudaSuccess) return err;
  const int optin = device_smem_optin() - static_cast<int>(fa.sharedSizeBytes);
  err = cudaFuncSetAttribute(kps_sample_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(kps_sample_kernel<kBF16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (err == cudaSuccess) done[dev] = true;
  return err;
}

template <bool kBF16>
static int active_clusters(int cs, size_t smem) {
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
    return 0;
  }
  return n;
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

// The cluster kernel's shapes for one (device, dtype, V), independent of the batch: for each
// power-of-two cluster size whether it runs, its chunk, shared memory and resident clusters,
// and the base size (the smallest whose per-CTA chunk fits two CTAs per SM, else the smallest
// that fits at all).  Occupancy queries are slow, so this is computed once per shape.
struct ClusterShapes {
  kps_status status;  // KPS_OK when some size runs
  int base;           // index into sizes of the base cluster size
  int sms;
  int fits[5];
  int nc[5];
  size_t smem[5];
  int clusters[5];
};
constexpr int kClusterSizes[5] = {1, 2, 4, 8, 16};

template <bool kBF16>
static ClusterShapes cluster_shapes(int64_t V) {
  ClusterShapes cs{};
  cs.status = KPS_ERR_UNSUPPORTED;
  cs.base = -1;
  const int optin = device_smem_optin();
  cs.sms = device_sm_count();
  if (optin <= 0 || cs.sms <= 0 || prepare_kernel<kBF16>() != cudaSuccess) {
    cs.status = KPS_ERR_CUDA;
    return cs;
  }
  for (int i = 0; i < 5; ++i) {
    const int c = kClusterSizes[i];
    cs.nc[i] = round_up8((V + c - 1) / c);
    cs.smem[i] = make_layout(cs.nc[i], kBF16).total;
    cs.fits[i] = cs.nc[i] <= kMaxChunk && cs.smem[i] <= static_cast<size_t>(optin) && cluster_fits<kBF16>(c, cs.smem[i]);
    cs.clusters[i] = cs.fits[i] ? active_clusters<kBF16>(c, cs.smem[i]) : 0;
    if (cs.clusters[i] <= 0) cs.fits[i] = 0;
  }
  for (int i = 0; i < 4 && cs.base < 0; ++i)  // sizes up to 8 whose chunk fits two CTAs per SM
    if (cs.fits[i] && cs.smem[i] <= static_cast<size_t>(kSmemCap2PerSM)) cs.base = i;
  for (int i = 0; i < 5 && cs.base < 0; ++i)
    if (cs.fits[i]) cs.base = i;
  if (cs.base >= 0) cs.status = KPS_OK;
  return cs;
}

// The cluster size for a batch of B rows: the base size, widened for small batches so more
// SMs work on each row (chunks of at least 4096 elements).  Depends on B only through the
// widening, which every caller computes from the same table.
static kps_status launch_from_shapes(const ClusterShapes& cs, int64_t B, int64_t V, LaunchCfg* out) {
  if (cs.status != KPS_OK) return cs.status;
  int i = cs.base;
  while (i < 4 && B * kClusterSizes[i] * 2 <= cs.sms && (V + kClusterSizes[i] * 2 - 1) / (kClusterSizes[i] * 2) >= 4096 &&
         cs.fits[i + 1])
    ++i;
  out->cs = kClusterSizes[i];
  out->nc = cs.nc[i];
  out->smem = cs.smem[i];
  out->clusters = cs.clusters[i];
  return KPS_OK;
}

template <bool kBF16>
static kps_status choose_launch(int64_t B, int64_t V, LaunchCfg* out) {
  const ClusterShapes cs = cluster_shapes<kBF16>(V);
  return launch_from_shapes(cs, B, V, out);
}

// The kernel the calling thread's last successful kps_sample launched (1 cluster, 2 row).
static thread_local int t_last_kernel = 0;
static thread_local int t_last_launches = 0;
static thread_local int t_last_cluster = 0;  // CTAs per cluster of that launch

// Kernel choice, per call (kps_step_opts.kernel_policy): 0 = automatic, 1 = cluster kernel
// only, 2 = row kernel where supported, 3 = row kernel with the exact whole-row selection
// forced (a test hook).
constexpr int64_t kRowMinRows = 64;  // automatic: the row kernel from this batch size up
constexpr size_t kWorkspaceMin = 256;  // the status word (and its alignment)
constexpr int64_t kMaxPreRows = 1024;  // top-p-only rows with a pre-pass record, at most

// Pre-pass records a workspace of `bytes` holds for a batch of B rows.
inline int64_t pre_rows_for(int64_t B, int64_t V, size_t bytes) {
  if (V <= kRKeepAllV || bytes <= kWorkspaceMin) return 0;
  int64_t n = static_cast<int64_t>((bytes - kWorkspaceMin) / kPRecBytes);
  n = n < B ? n : B;
  return n < kMaxPreRows ? n : kMaxPreRows;
}

constexpr int kRowTeams[] = {2, 1};  // cluster sizes tried, widest first: CTAs sharing a top-p-only row

struct RowCfg {
  size_t smem;
  int cs;        // cluster size
  int clusters;  // clusters resident at once (the persistent grid, in clusters)
};

template <bool kBF16>
static cudaError_t prepare_row_kernel() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, kps_row_kernel<kBF16>);
  if (err != cudaSuccess) return err;
  const int optin = device_smem_optin() - static_cast<int>(fa.sharedSizeBytes);
  err = cudaFuncSetAttribute(kps_row_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (err != cudaSuccess) return err;
  err = cudaFuncGetAttributes(&fa, kps_prepass_kernel<kBF16>);
  if (err != cudaSuccess) return err;
  const int optin2 = device_smem_optin() - static_cast<int>(fa.sharedSizeBytes);
  err = cudaFuncSetAttribute(kps_prepass_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin2);
  if (err == cudaSuccess) done[dev] = true;
  return err;
}

// Shared memory and resident grid of the row kernel; false if it cannot run this V.
template <bool kBF16>
static bool choose_row(int64_t V, RowCfg* out) {
  if (V > kRMaxV) return false;
  if (prepare_row_kernel<kBF16>() != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  const size_t smem = make_rlayout(V).total;
  for (int cs : kRowTeams) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(kRT);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = cs;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kps_row_kernel<kBF16>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    if (n > 0) {
      out->smem = smem;
      out->cs = cs;
      out->clusters = n;
      return true;
    }
  }
  return false;
}

// Launch decisions depend on (device, dtype, V), plus the batch size only through the
// cluster kernel's widening (launch_from_shapes, cheap), so the batch-independent part is
// computed once per shape and cached: kps_sample then costs one lookup and one launch.
struct CachedShape {
  int dev;
  int dt;
  int64_t V;
  bool row_ok;
  RowCfg row;
  ClusterShapes cluster;
};

static kps_status lookup_shape(kps_dtype dt, int64_t V, CachedShape* out) {
  static std::mutex mu;
  static CachedShape cache[32];
  static int used = 0, next = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return KPS_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    const CachedShape& c = cache[i];
    if (c.dev == dev && c.dt == static_cast<int>(dt) && c.V == V) {
      *out = c;
      return KPS_OK;
    }
  }
  CachedShape c{};
  c.dev = dev;
  c.dt = static_cast<int>(dt);
  c.V = V;
  RowCfg rcfg{};
  c.row_ok = dt == KPS_BF16 ? choose_row<true>(V, &rcfg) : choose_row<false>(V, &rcfg);
  c.row = rcfg;
  c.cluster = dt == KPS_BF16 ? cluster_shapes<true>(V) : cluster_shapes<false>(V);
  if (used < 32) {
    cache[used++] = c;
  } else {
    cache[next] = c;
    next = (next + 1) % 32;
  }
  *out = c;
  return KPS_OK;
}

}  // namespace kps

namespace kps {
// An NVTX range around each public sampling call: it names the call in a profiler's timeline
// (Nsight Systems, ncu's NVTX filters) and costs a pointer check when no tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace kps

// ------------------------------------------------------------------------------------------
// C ABI
// ------------------------------------------------------------------------------------------
extern "C" {

size_t kps_workspace_size(int64_t B, int64_t V, kps_dtype dt) {
  if (B < 0 || V < 1 || (dt != KPS_F32 && dt != KPS_BF16)) return 0;
  if (V <= kps::kRKeepAllV) return kps::kWorkspaceMin;
  const int64_t rows = B < kps::kMaxPreRows ? B : kps::kMaxPreRows;
  return kps::kWorkspaceMin + static_cast<size_t>(rows) * kps::kPRecBytes;
}

int64_t kps_max_vocab(kps_dtype dt) {
  if (dt != KPS_F32 && dt != KPS_BF16) return 0;
  const int optin = kps::device_smem_optin();
  if (optin <= 0) return 0;
  const bool bf = dt == KPS_BF16;
  if ((bf ? kps::prepare_kernel<true>() : kps::prepare_kernel<false>()) != cudaSuccess) return 0;
  // the largest chunk (a multiple of 8) whose layout fits one CTA: binary search over its
  // eighths, keeping a chunk that fits in lo
  int lo = 0, hi = kps::kMaxChunk / 8;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (kps::make_layout(mid * 8, bf).total <= static_cast<size_t>(optin)) lo = mid; else hi = mid - 1;
  }
  if (lo == 0) return 0;
  const int nc = lo * 8;
  const size_t smem = kps::make_layout(nc, bf).total;
  // times the widest cluster the device runs with that much shared memory per CTA
  for (int cs = 16; cs >= 1; cs /= 2) {
    const bool fits = bf ? kps::cluster_fits<true>(cs, smem) : kps::cluster_fits<false>(cs, smem);
    if (fits) return static_cast<int64_t>(nc) * cs;
  }
  return 0;
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

// The host-side checks of the arguments every entry point shares (the workspace aside);
// KPS_OK when the call may go ahead.
static kps_status check_args(kps_dtype dt, int64_t B, int64_t V, float eps, const void* logits, const int32_t* top_k,
                             const float* top_p, const float* temperature, const int64_t* out_idx, int need_logits,
                             const float* out_filtered) {
  if (dt != KPS_F32 && dt != KPS_BF16) return KPS_ERR_INVALID_ARG;
  if (V < 1 || V > INT32_MAX || B < 0) return KPS_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || std::isinf(eps)) return KPS_ERR_INVALID_ARG;
  if (B == 0) return KPS_OK;
  if (B > INT32_MAX / 16) return KPS_ERR_INVALID_ARG;
  if (!logits || !top_k || !top_p || !temperature || !out_idx) return KPS_ERR_INVALID_ARG;  // q: may be NULL
  if (need_logits && !out_filtered) return KPS_ERR_INVALID_ARG;
  return KPS_OK;
}

// The sampling step; q given (or NULL) or, with gen, generated from (seed, step).
static kps_status sample_impl(const void* logits, kps_dtype dt, int64_t B, int64_t V, const int32_t* top_k,
                              const float* top_p, const float* temperature, const int32_t* seen_indptr,
                              const int32_t* seen_ids, const float* penalty, const float* q, float eps,
                              int need_logits, int64_t* out_idx, float* out_filtered, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream, int gen, unsigned long long seed,
                              unsigned long long step, unsigned char* finished = nullptr, long long eos = 0,
                              int* unfinished = nullptr, uint32_t* seen_bits = nullptr, int update_seen = 0,
                              int policy = 0) {
  if (dt != KPS_F32 && dt != KPS_BF16) return KPS_ERR_INVALID_ARG;
  if (V < 1 || V > INT32_MAX || B < 0) return KPS_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || std::isinf(eps)) return KPS_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < kps::kWorkspaceMin)
    return KPS_ERR_WORKSPACE;
  {
    const kps_status st = check_args(dt, B, V, eps, logits, top_k, top_p, temperature, out_idx, need_logits, out_filtered);
    if (st != KPS_OK || B == 0) return st;
  }
  if (seen_bits && (seen_indptr || seen_ids)) return KPS_ERR_INVALID_ARG;  // one form of the seen set
  if (seen_bits && (reinterpret_cast<uintptr_t>(seen_bits) & 3u) != 0) return KPS_ERR_INVALID_ARG;
  if (update_seen && !seen_bits) return KPS_ERR_INVALID_ARG;
  const bool pen = (seen_indptr && seen_ids && penalty) || (seen_bits && penalty);

  const size_t esize = dt == KPS_BF16 ? 2 : 4;
  const bool aligned = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && ((V * esize) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(q) % 16 == 0) && (V % 4 == 0) &&  // a NULL q is aligned
                       (!need_logits || reinterpret_cast<uintptr_t>(out_filtered) % 16 == 0);
  const bool want_row =
      aligned && (policy >= 2 || (policy == 0 && B >= kps::kRowMinRows));
  kps::RowCfg rcfg;
  kps::LaunchCfg cfg{};
  bool use_row = false;
  {
    kps::CachedShape cs;
    const kps_status st = kps::lookup_shape(dt, V, &cs);
    if (st != KPS_OK) return st;
    use_row = want_row && cs.row_ok;
    rcfg = cs.row;
    const kps_status cst = kps::launch_from_shapes(cs.cluster, B, V, &cfg);
    if (!use_row && cst != KPS_OK) return cst;
  }

  kps::Params P;
  P.logits = logits;
  P.B = B;
  P.V = V;
  P.top_k = top_k;
  P.top_p = top_p;
  P.temperature = temperature;
  P.seen_indptr = pen && !seen_bits ? seen_indptr : nullptr;
  P.seen_ids = pen && !seen_bits ? seen_ids : nullptr;
  P.penalty = pen ? penalty : nullptr;
  P.seen_bits = seen_bits;
  P.update_seen = update_seen ? 1 : 0;
  P.q = gen ? nullptr : q;
  P.gen = gen ? 1 : 0;
  P.seed = seed;
  P.step = step;
  P.finished = finished;
  P.eos = eos;
  P.unfinished = finished ? unfinished : nullptr;
  if (P.unfinished && cudaMemsetAsync(P.unfinished, 0, sizeof(int), stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return KPS_ERR_CUDA;
  }
  P.eps = eps;
  P.need_logits = need_logits ? 1 : 0;
  P.out_idx = out_idx;
  P.out_filtered = need_logits ? out_filtered : nullptr;
  P.status = static_cast<int*>(workspace);
  P.nc = cfg.nc;
  P.use_tma = aligned ? 1 : 0;
  P.filter = 0;
  P.exact = policy == 3 ? 1 : 0;
  P.pre = nullptr;
  P.pre_rows = 0;

  if (use_row) {
    // the pre-pass pays when rows outnumber the clusters (then the top-k rows come C to a
    // cluster and a top-p-only row would keep its pair of CTAs busy the longest); with
    // fewer rows every row has a cluster of its own from the start
    const int64_t pre_rows = (P.exact || B <= rcfg.clusters) ? 0 : kps::pre_rows_for(B, V, workspace_bytes);
    if (pre_rows > 0) {
      // pass A of the top-p-only rows first, over the whole resident grid
      P.pre = static_cast<unsigned char*>(workspace) + kps::kWorkspaceMin;
      P.pre_rows = static_cast<int>(pre_rows);
      cudaLaunchConfig_t pl = {};
      pl.gridDim = dim3(static_cast<unsigned>(rcfg.clusters * rcfg.cs));
      pl.blockDim = dim3(kps::kRT);
      pl.dynamicSmemBytes = rcfg.smem;
      pl.stream = stream;
      cudaError_t e = dt == KPS_BF16 ? cudaLaunchKernelEx(&pl, kps::kps_prepass_kernel<true>, P)
                                     : cudaLaunchKernelEx(&pl, kps::kps_prepass_kernel<false>, P);
      if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return KPS_ERR_CUDA;
      }
    }
    // a persistent grid of resident clusters; a cluster's CTAs share the top-p-only and
    // keep-all rows and take the other rows one each
    const int64_t ncl = B < rcfg.clusters ? B : rcfg.clusters;
    cudaLaunchConfig_t rl = {};
    rl.gridDim = dim3(static_cast<unsigned>(ncl * rcfg.cs));
    rl.blockDim = dim3(kps::kRT);
    rl.dynamicSmemBytes = rcfg.smem;
    rl.stream = stream;
    cudaLaunchAttribute rattr[2];
    rattr[0].id = cudaLaunchAttributeClusterDimension;
    rattr[0].val.clusterDim.x = rcfg.cs;
    rattr[0].val.clusterDim.y = 1;
    rattr[0].val.clusterDim.z = 1;
    // after a pre-pass: start at once (programmatic dependent launch); only the rows that
    // read its records wait for it
    rattr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    rattr[1].val.programmaticStreamSerializationAllowed = 1;
    rl.attrs = rattr;
    rl.numAttrs = P.pre ? 2 : 1;
    cudaError_t e = dt == KPS_BF16 ? cudaLaunchKernelEx(&rl, kps::kps_row_kernel<true>, P)
                                   : cudaLaunchKernelEx(&rl, kps::kps_row_kernel<false>, P);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return KPS_ERR_CUDA;
    }
    kps::t_last_kernel = 2;
    kps::t_last_launches = P.pre ? 2 : 1;
    kps::t_last_cluster = rcfg.cs;
    return KPS_OK;
  }

  cudaLaunchConfig_t lc = {};
  const int64_t clusters = B < cfg.clusters ? B : cfg.clusters;  // persistent: clusters walk the rows
  lc.gridDim = dim3(static_cast<unsigned>(clusters * cfg.cs));
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
  kps::t_last_kernel = 1;
  kps::t_last_launches = 1;
  kps::t_last_cluster = cfg.cs;
  return KPS_OK;
}

kps_status kps_sample(const void* logits, kps_dtype dt, int64_t B, int64_t V, const int32_t* top_k,
                      const float* top_p, const float* temperature, const int32_t* seen_indptr,
                      const int32_t* seen_ids, const float* penalty, const float* q, float eps, int need_logits,
                      int64_t* out_idx, float* out_filtered, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  const kps::NvtxRange range("kps_sample");
  return sample_impl(logits, dt, B, V, top_k, top_p, temperature, seen_indptr, seen_ids, penalty, q, eps,
                     need_logits, out_idx, out_filtered, workspace, workspace_bytes, stream, 0, 0ull, 0ull);
}

kps_status kps_sample_seeded(const void* logits, kps_dtype dt, int64_t B, int64_t V, const int32_t* top_k,
                             const float* top_p, const float* temperature, const int32_t* seen_indptr,
                             const int32_t* seen_ids, const float* penalty, unsigned long long seed,
                             unsigned long long step, float eps, int need_logits, int64_t* out_idx,
                             float* out_filtered, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const kps::NvtxRange range("kps_sample_seeded");
  return sample_impl(logits, dt, B, V, top_k, top_p, temperature, seen_indptr, seen_ids, penalty, nullptr, eps,
                     need_logits, out_idx, out_filtered, workspace, workspace_bytes, stream, 1, seed, step);
}

kps_status kps_sample_step(const void* logits, kps_dtype dt, int64_t B, int64_t V, const int32_t* top_k,
                           const float* top_p, const float* temperature, const int32_t* seen_indptr,
                           const int32_t* seen_ids, const float* penalty, const kps_step_opts* opts, float eps,
                           int need_logits, int64_t* out_idx, float* out_filtered, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  const kps::NvtxRange range("kps_sample_step");
  if (!opts) return KPS_ERR_INVALID_ARG;
  if (opts->unfinished && !opts->finished) return KPS_ERR_INVALID_ARG;
  if (opts->kernel_policy < 0 || opts->kernel_policy > 3) return KPS_ERR_INVALID_ARG;
  return sample_impl(logits, dt, B, V, top_k, top_p, temperature, seen_indptr, seen_ids, penalty,
                     opts->generate ? nullptr : opts->q, eps, need_logits, out_idx, out_filtered, workspace,
                     workspace_bytes, stream, opts->generate ? 1 : 0, opts->seed, opts->step, opts->finished,
                     static_cast<long long>(opts->eos_id), opts->unfinished, opts->seen_bits, opts->update_seen,
                     opts->kernel_policy);
}

int kps_last_kernel(void) { return kps::t_last_kernel; }

int kps_last_launch_count(void) { return kps::t_last_launches; }

int kps_last_cluster_size(void) { return kps::t_last_cluster; }

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
  const kps::NvtxRange range("kps_sample_noalloc");
  // every argument is checked before the shared array is touched: a rejected call queues nothing
  {
    const kps_status st = check_args(dt, B, V, eps, logits, top_k, top_p, temperature, out_idx, need_logits, out_filtered);
    if (st != KPS_OK || B == 0) return st;
  }
  const size_t need = kps::kWorkspaceMin;  // the status word; no room for pre-pass records
  void* scratch = kps::noalloc_scratch_address();
  if (!scratch) return KPS_ERR_CUDA;
  // the shared array keeps the previous call's status word: clear it on this stream first
  if (cudaMemsetAsync(scratch, 0, need, stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return KPS_ERR_CUDA;
  }
  return kps_sample(logits, dt, B, V, top_k, top_p, temperature, seen_indptr, seen_ids, penalty, q, eps,
                    need_logits, out_idx, out_filtered, scratch, need, stream);
}
