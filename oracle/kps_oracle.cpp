// kps_oracle.cpp — plain, slow, single-threaded CPU oracle for the per-step
// token-sampling post-process (repetition penalty -> temperature -> top-k ->
// top-p -> exponential race).
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
// this file: only the tests, the smoke check and the benchmark's CPU-baseline
// leg use it.  It shares no code, header or constant with the CUDA library.
//
// Sources (the three pages this method is described on):
//   [NPU]  Ascend API reference "torch_npu.npu_top_k_top_p_sample":
//          topK item 2 (valid range 1 <= k <= min(V,1024), otherwise skip),
//          the topP full-sort fallback (sort desc, cumsum, drop where the
//          exclusive cumsum exceeds top_p), and the Sample formula
//          (probs = softmax(filtered); idx = argmax(probs / (q + eps))).
//   [MM10] MiniMind "Chapter 10: inference generation": §10.4 temperature
//          (logits / T), §10.5 top-k threshold mask, §10.6 top-p via sorted
//          softmax cumsum with the mask shifted right by one, §10.7 repetition
//          penalty (score > 0 ? score / p : score * p over the unique seen ids).
//   [CPP]  "LLM sampling post-processing summary: the C++ implementation":
//          repetition_penalty over a set of ids (duplicates applied once),
//          softmax (max, exp, sum) and the top_p rule "smallest set whose
//          mass reaches top_p".
//
// Readings fixed where the pages are silent or disagree (each one is listed
// with its reason in the design notes):
//   * penalty first, then temperature; both are IEEE fp32 operations
//     (x / p, x * p, x / T), exactly as the GPU performs them;
//   * NaN logits become -inf before anything else;
//   * a row whose temperature is not a finite positive number is greedy:
//     no division, the kept set is the single best element;
//   * penalty <= 0 or NaN skips the penalty for that row; seen ids outside
//     [0, V) are ignored;
//   * total order "pi": value descending, then index ascending;
//   * top-k keeps exactly the first k elements under pi when
//     1 <= k <= min(V, 1024) and is the identity otherwise [NPU topK item 2];
//   * softmax over the top-k set in double with e_v = exp(x_v - M); an element
//     equal to the maximum M gets weight exactly 1 (so +-inf maxima are finite);
//   * top-p keeps the shortest pi-prefix whose mass reaches p * S: an element
//     is kept while the exclusive prefix mass is < p * S [MM10 §10.6 worked
//     example keeps the token that first reaches the threshold]; p <= 0 keeps
//     one element, p >= 1 or NaN skips the stage;
//   * race: r_v = (e_v / S_P) / (q_v + eps) in double over the kept set P,
//     argmax with the lower index winning an exact tie, NaN scores ignored,
//     the pi-first element if every score is NaN;
//   * filtered output: the transformed value at kept positions, -inf elsewhere.
//   * sampling off (q absent): the first element of the order in the kept set,
//     i.e. the argmax of the filtered row with the lowest index among equals.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

float bf16_bits_to_float(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// One row of the method, written out step by step.
struct RowResult {
  int64_t idx;
  int64_t kept;
  double race_gap;  // (best - second best) / best race score, +inf if < 2 scores
  double topp_gap;  // distance of the deciding cumsums from p*S, relative to p*S
};

// The row's terms up to the top-k set: the transformed row x (NaN -> -inf, penalty,
// temperature), the order pi restricted to its first nK elements, their softmax weights
// e and the sum S.
struct RowTerms {
  bool greedy;
  int64_t nK;
  std::vector<int64_t> order;  // order[0 .. nK) sorted under pi
  std::vector<double> e;       // e[i] = exp(x[order[i]] - M), i < nK
  double S;
};

RowTerms row_terms(std::vector<float>& x, int64_t V, int32_t k, float T,
                   const int32_t* ids, int64_t nids, bool pen_on, float pen) {
  const float NEG_INF = -std::numeric_limits<float>::infinity();
  RowTerms t;

  // NaN logits are treated as -inf.
  for (int64_t v = 0; v < V; ++v)
    if (std::isnan(x[v])) x[v] = NEG_INF;

  // Repetition penalty over the SET of seen ids [MM10 §10.7, CPP repetition_penalty].
  if (pen_on) {
    std::vector<char> seen(static_cast<size_t>(V), 0);
    for (int64_t j = 0; j < nids; ++j) {
      int64_t id = ids[j];
      if (id < 0 || id >= V || seen[id]) continue;
      seen[id] = 1;
      float s = x[id];
      x[id] = (s > 0.0f) ? (s / pen) : (s * pen);
    }
  }

  // Temperature [MM10 §10.4]: x / T, or greedy when T is not finite and positive.
  t.greedy = !(T > 0.0f) || std::isinf(T);
  if (!t.greedy)
    for (int64_t v = 0; v < V; ++v) x[v] = x[v] / T;

  // Total order pi: value descending, index ascending.
  auto before = [&x](int64_t a, int64_t b) {
    return x[a] > x[b] || (x[a] == x[b] && a < b);
  };
  std::vector<int64_t>& order = t.order;
  order.resize(static_cast<size_t>(V));
  for (int64_t v = 0; v < V; ++v) order[v] = v;

  // Top-k [NPU topK item 2; MM10 §10.5]: exactly the first k under pi.
  const bool topk_on = (k >= 1) && (static_cast<int64_t>(k) <= std::min<int64_t>(V, 1024));
  int64_t nK = V;
  if (topk_on) {
    nK = k;
    std::nth_element(order.begin(), order.begin() + (nK - 1), order.end(), before);
    std::sort(order.begin(), order.begin() + nK, before);
  } else {
    std::sort(order.begin(), order.end(), before);
  }
  t.nK = nK;

  // Softmax over K in double [CPP softmax; NPU topK softmax step].
  const double M = static_cast<double>(x[order[0]]);
  std::vector<double>& e = t.e;
  e.resize(static_cast<size_t>(nK));
  double S = 0.0;
  for (int64_t i = 0; i < nK; ++i) {
    double xv = static_cast<double>(x[order[i]]);
    e[i] = (xv == M) ? 1.0 : std::exp(xv - M);
    S += e[i];
  }
  t.S = S;
  return t;
}

RowResult sample_row(std::vector<float>& x, int64_t V, int32_t k, float p, float T,
                     const int32_t* ids, int64_t nids, bool pen_on, float pen,
                     const float* qrow, float eps, float* out_row) {
  const float NEG_INF = -std::numeric_limits<float>::infinity();
  const RowTerms t = row_terms(x, V, k, T, ids, nids, pen_on, pen);
  const bool greedy = t.greedy;
  const int64_t nK = t.nK;
  const std::vector<int64_t>& order = t.order;
  const std::vector<double>& e = t.e;
  const double S = t.S;

  // Top-p [NPU topP fallback; MM10 §10.6; CPP top_p].
  int64_t nP = nK;
  double topp_gap = std::numeric_limits<double>::infinity();
  if (greedy || p <= 0.0f) {
    nP = 1;
  } else if (p < 1.0f) {
    const double target = static_cast<double>(p) * S;
    double c = 0.0, c_before_last = 0.0;
    nP = 0;
    while (nP < nK && c < target) {
      c_before_last = c;
      c += e[nP];
      ++nP;
    }
    double lo = target - c_before_last;  // > 0: the last kept element was needed
    double hi = c - target;              // >= 0: the prefix reaches the target
    topp_gap = std::min(std::fabs(lo), std::fabs(hi)) / target;
  }

  // Sampling off (no q) [NPU scenario table: Sample disabled; MM10 generation loop and
  // "greedy mode": without sampling the next token is the argmax of the filtered logits,
  // the first one among equal maxima]: the first element of the order, which every
  // kept set holds.
  if (!qrow) {
    if (out_row) {
      for (int64_t v = 0; v < V; ++v) out_row[v] = NEG_INF;
      for (int64_t i = 0; i < nP; ++i) out_row[order[i]] = x[order[i]];
    }
    return RowResult{order[0], nP, std::numeric_limits<double>::infinity(), topp_gap};
  }

  // Exponential race [NPU Sample]: argmax of (e / S_P) / (q + eps).
  double SP = 0.0;
  for (int64_t i = 0; i < nP; ++i) SP += e[i];
  int64_t best = -1;
  double rbest = 0.0, rsecond = -std::numeric_limits<double>::infinity();
  for (int64_t i = 0; i < nP; ++i) {
    int64_t v = order[i];
    double r = (e[i] / SP) / (static_cast<double>(qrow[v]) + static_cast<double>(eps));
    if (std::isnan(r)) continue;
    if (best < 0 || r > rbest || (r == rbest && v < best)) {
      if (best >= 0) rsecond = std::max(rsecond, rbest);
      best = v;
      rbest = r;
    } else {
      rsecond = std::max(rsecond, r);
    }
  }
  if (best < 0) best = order[0];
  double race_gap = std::numeric_limits<double>::infinity();
  if (nP >= 2 && std::isfinite(rsecond) && rbest != 0.0)
    race_gap = (rbest - rsecond) / std::fabs(rbest);

  // Filtered logits [NPU Sample, logits_top_kp_select]: kept values, -inf elsewhere.
  if (out_row) {
    for (int64_t v = 0; v < V; ++v) out_row[v] = NEG_INF;
    for (int64_t i = 0; i < nP; ++i) out_row[order[i]] = x[order[i]];
  }
  return RowResult{best, nP, race_gap, topp_gap};
}

}  // namespace

extern "C" {

// Returns 0 on success, 1 on an invalid argument.  dtype: 0 = fp32, 1 = bf16.
// seen_indptr / seen_ids / penalty may all be NULL (no penalty).
// q may be NULL: sampling off (the first element of the kept set's order).
// out_filtered may be NULL when need_logits == 0.  The three diagnostic
// outputs (kept count, race gap, top-p gap per row) may be NULL.
int kpso_sample(const void* logits, int dtype, int64_t B, int64_t V,
                const int32_t* top_k, const float* top_p, const float* temperature,
                const int32_t* seen_indptr, const int32_t* seen_ids, const float* penalty,
                const float* q, float eps, int need_logits,
                int64_t* out_idx, float* out_filtered,
                int64_t* out_kept, double* out_race_gap, double* out_topp_gap) {
  if (B < 0 || V < 1 || !logits || !top_k || !top_p || !temperature || !out_idx)
    return 1;
  if (dtype != 0 && dtype != 1) return 1;
  if (need_logits && !out_filtered) return 1;
  std::vector<float> x(static_cast<size_t>(V));
  for (int64_t b = 0; b < B; ++b) {
    if (dtype == 0) {
      const float* row = static_cast<const float*>(logits) + b * V;
      for (int64_t v = 0; v < V; ++v) x[v] = row[v];
    } else {
      const uint16_t* row = static_cast<const uint16_t*>(logits) + b * V;
      for (int64_t v = 0; v < V; ++v) x[v] = bf16_bits_to_float(row[v]);
    }
    bool pen_on = seen_indptr && seen_ids && penalty && (penalty[b] > 0.0f);
    const int32_t* ids = nullptr;
    int64_t nids = 0;
    if (pen_on) {
      ids = seen_ids + seen_indptr[b];
      nids = static_cast<int64_t>(seen_indptr[b + 1]) - seen_indptr[b];
      if (nids < 0) nids = 0;
    }
    RowResult r = sample_row(x, V, top_k[b], top_p[b], temperature[b], ids, nids, pen_on,
                             pen_on ? penalty[b] : 1.0f, q ? q + b * V : nullptr, eps,
                             need_logits ? out_filtered + b * V : nullptr);
    out_idx[b] = r.idx;
    if (out_kept) out_kept[b] = r.kept;
    if (out_race_gap) out_race_gap[b] = r.race_gap;
    if (out_topp_gap) out_topp_gap[b] = r.topp_gap;
  }
  return 0;
}

// The terms of row b (for checking a result at a near-tie against the definition rather
// than against this oracle's own choice): the transformed row x_out[V], the first nK
// elements of the order pi in order_out, their weights e_out and S.  order_out and e_out
// hold V entries.  Returns nK (>= 1), or -1 on an invalid argument; *greedy_out is 1 for
// a greedy row.
int64_t kpso_row_terms(const void* logits, int dtype, int64_t B, int64_t V, int64_t b,
                       const int32_t* top_k, const float* temperature,
                       const int32_t* seen_indptr, const int32_t* seen_ids, const float* penalty,
                       float* x_out, int64_t* order_out, double* e_out, double* S_out,
                       int* greedy_out) {
  if (b < 0 || b >= B || V < 1 || !logits || !top_k || !temperature || !x_out || !order_out ||
      !e_out || !S_out || !greedy_out)
    return -1;
  if (dtype != 0 && dtype != 1) return -1;
  std::vector<float> x(static_cast<size_t>(V));
  if (dtype == 0) {
    const float* row = static_cast<const float*>(logits) + b * V;
    for (int64_t v = 0; v < V; ++v) x[v] = row[v];
  } else {
    const uint16_t* row = static_cast<const uint16_t*>(logits) + b * V;
    for (int64_t v = 0; v < V; ++v) x[v] = bf16_bits_to_float(row[v]);
  }
  bool pen_on = seen_indptr && seen_ids && penalty && (penalty[b] > 0.0f);
  const int32_t* ids = nullptr;
  int64_t nids = 0;
  if (pen_on) {
    ids = seen_ids + seen_indptr[b];
    nids = static_cast<int64_t>(seen_indptr[b + 1]) - seen_indptr[b];
    if (nids < 0) nids = 0;
  }
  const RowTerms t = row_terms(x, V, top_k[b], temperature[b], ids, nids, pen_on, pen_on ? penalty[b] : 1.0f);
  for (int64_t v = 0; v < V; ++v) x_out[v] = x[v];
  for (int64_t i = 0; i < t.nK; ++i) {
    order_out[i] = t.order[i];
    e_out[i] = t.e[i];
  }
  *S_out = t.S;
  *greedy_out = t.greedy ? 1 : 0;
  return t.nK;
}

// ---- Exp(1) draws from a counter-based generator (sampling without a supplied q) ---------
//
// Philox4x32-10 [Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11, section 4 (the Philox S-box: a 32x32 -> 64-bit multiply whose halves are mixed
// into the other words, 10 rounds, the key bumped by the Weyl increments between rounds)
// and its table of round constants for Philox-4x32].
static void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c[0];
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c[2];
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n1 = lo1, n2 = hi0 ^ c[3] ^ k1, n3 = lo0;
    c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
    k0 += 0x9E3779B9u;  // the Weyl increments of the key
    k1 += 0xBB67AE85u;
  }
}

// The draw of row b, token v at decode step `step` under `seed`: Philox4x32-10 with key
// (seed low, seed high) on the counter (v / 4, b, step low, step high), word v mod 4;
// u = (2 * (word >> 9) + 1) * 2^-24 in (0, 1) (exact in fp32); q = -log(u) rounded to fp32.
static float exp_draw(uint64_t seed, uint64_t step, int64_t b, int64_t v) {
  uint32_t c[4] = {static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(b), static_cast<uint32_t>(step),
                   static_cast<uint32_t>(step >> 32)};
  philox4x32_10(c, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const uint32_t w = c[v & 3];
  const double u = static_cast<double>(2u * (w >> 9) + 1u) * (1.0 / 16777216.0);
  return static_cast<float>(-std::log(u));
}

// The raw generator, for its known-answer tests: c (4 words) is replaced by its output.
void kpso_philox4x32_10(uint32_t* c, uint32_t k0, uint32_t k1) { philox4x32_10(c, k0, k1); }

// q[B, V] of the generated Exp(1) draws (the q a seeded kps call races with).
int kpso_exp_draws(int64_t B, int64_t V, uint64_t seed, uint64_t step, float* q) {
  if (B < 0 || V < 1 || !q) return 1;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t v = 0; v < V; ++v) q[b * V + v] = exp_draw(seed, step, b, v);
  return 0;
}

// The end-of-sequence epilogue of a decode step [MM10 generate loop: a finished sequence
// emits eos_token_id (torch.where on the finished flags), then finished |= the token
// equals eos_token_id, and the loop stops once every sequence is finished].  Updates idx
// and finished in place; returns the number of rows left unfinished.
int64_t kpso_eos_epilogue(int64_t* idx, uint8_t* finished, int64_t eos, int64_t B) {
  int64_t left = 0;
  for (int64_t b = 0; b < B; ++b) {
    if (finished[b]) idx[b] = eos;
    if (idx[b] == eos) finished[b] = 1;
    if (!finished[b]) ++left;
  }
  return left;
}

// The seen set of each row as the sorted list of distinct ids [MM10 §10.7: the penalty
// runs over the unique ids of the sequence so far], read from its bit form: bit v % 32
// of word b * W + v / 32 (W = ceil(V / 32)) marks token v of row b; bits of tokens >= V
// are not ids.  indptr [B + 1] always; ids (room for indptr[B]) when non-NULL.  Returns
// the number of ids.
int64_t kpso_seen_ids_from_bits(const uint32_t* bits, int64_t B, int64_t V, int32_t* indptr, int32_t* ids) {
  const int64_t W = (V + 31) / 32;
  int64_t n = 0;
  indptr[0] = 0;
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t v = 0; v < V; ++v) {
      if ((bits[b * W + v / 32] >> (v % 32)) & 1u) {
        if (ids) ids[n] = static_cast<int32_t>(v);
        ++n;
      }
    }
    indptr[b + 1] = static_cast<int32_t>(n);
  }
  return n;
}

// One decode step's growth of the seen sets [MM10 generate loop: the step's token is
// appended to each sequence, so the next step's unique ids are the old ones plus that
// token]: the bit of idx[b] is set in row b when 0 <= idx[b] < V.
void kpso_seen_append(uint32_t* bits, const int64_t* idx, int64_t B, int64_t V) {
  const int64_t W = (V + 31) / 32;
  for (int64_t b = 0; b < B; ++b)
    if (idx[b] >= 0 && idx[b] < V) bits[b * W + idx[b] / 32] |= 1u << (idx[b] % 32);
}

}  // extern "C"
