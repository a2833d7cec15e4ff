// oasis_oracle.cpp -- sequential CPU restatement of the OasisKV look-ahead
// sparse decode step.  TEST INFRASTRUCTURE ONLY (see oasis_oracle.h).
//
// Written from the method's description, not from any printed code: every
// loop below follows the definition it names, in double precision, with no
// blocking, fusion or reordering beyond what that definition states.
#include "oasis_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <numeric>
#include <set>
#include <vector>

namespace {

// bf16 bit pattern -> exact double (bf16 is the top half of an IEEE float).
double widen(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

int blocks_of(int ctx, int B) { return ctx <= 0 ? 0 : (ctx + B - 1) / B; }

// Number of valid tokens of logical block b in a context of ctx tokens.
int valid_tokens(int ctx, int b, int B) {
  int v = ctx - b * B;
  return v < 0 ? 0 : (v > B ? B : v);
}

size_t kv_index(int r, int h, int b, int kv, int t, int i, int Hkv, int NBmax,
                int B, int d) {
  return ((((static_cast<size_t>(r) * Hkv + h) * NBmax + b) * 2 + kv) * B + t) *
             static_cast<size_t>(d) + i;
}

size_t summ_index(int r, int h, int b, int which, int i, int Hkv, int NBmax,
                  int d) {
  return (((static_cast<size_t>(r) * Hkv + h) * NBmax + b) * 2 + which) *
             static_cast<size_t>(d) + i;
}

bool dims_ok(int R, int Hq, int Hkv, int NBmax, int B, int d) {
  return R > 0 && Hq > 0 && Hkv > 0 && Hq % Hkv == 0 && NBmax > 0 && B > 0 &&
         d > 0;
}

// softmax(x . k * scale) . v over the gathered tokens, in double.
void attend(const std::vector<const uint16_t*>& keys,
            const std::vector<const uint16_t*>& vals, const uint16_t* x, int d,
            double scale, float* out) {
  const size_t n = keys.size();
  if (n == 0) {  // nothing resident: the output is defined as zero
    for (int i = 0; i < d; ++i) out[i] = 0.0f;
    return;
  }
  std::vector<double> logit(n);
  for (size_t t = 0; t < n; ++t) {
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += widen(x[i]) * widen(keys[t][i]);
    logit[t] = dot * scale;
  }
  const double m = *std::max_element(logit.begin(), logit.end());
  double z = 0.0;
  std::vector<double> w(n);
  for (size_t t = 0; t < n; ++t) {
    w[t] = std::exp(logit[t] - m);
    z += w[t];
  }
  for (int i = 0; i < d; ++i) {
    double acc = 0.0;
    for (size_t t = 0; t < n; ++t) acc += w[t] * widen(vals[t][i]);
    out[i] = static_cast<float>(acc / z);
  }
}

}  // namespace

extern "C" int orc_summary_build(const uint16_t* host_kv, const int32_t* ctx_len,
                                 int R, int Hkv, int NBmax, int B, int d,
                                 uint16_t* summ) {
  if (!host_kv || !ctx_len || !summ || !dims_ok(R, Hkv, Hkv, NBmax, B, d))
    return -1;
  for (int r = 0; r < R; ++r) {
    const int nb = std::min(blocks_of(ctx_len[r], B), NBmax);
    for (int h = 0; h < Hkv; ++h)
      for (int b = 0; b < nb; ++b) {
        const int valid = valid_tokens(ctx_len[r], b, B);
        for (int i = 0; i < d; ++i) {
          uint16_t lo = host_kv[kv_index(r, h, b, 0, 0, i, Hkv, NBmax, B, d)];
          uint16_t hi = lo;
          for (int t = 1; t < valid; ++t) {
            uint16_t k = host_kv[kv_index(r, h, b, 0, t, i, Hkv, NBmax, B, d)];
            if (widen(k) < widen(lo)) lo = k;
            if (widen(k) > widen(hi)) hi = k;
          }
          summ[summ_index(r, h, b, 0, i, Hkv, NBmax, d)] = lo;
          summ[summ_index(r, h, b, 1, i, Hkv, NBmax, d)] = hi;
        }
      }
  }
  return 0;
}

extern "C" int orc_attention_rh(const uint16_t* host_kv, const int32_t* ctx_len,
                                const int32_t* res, const uint16_t* q,
                                const uint16_t* qd, int D, int R, int Hq, int Hkv,
                                int NBmax, int B, int d, int K, double scale,
                                int r, int h, float* out) {
  if (!host_kv || !ctx_len || !res || !q || !qd || !out ||
      !dims_ok(R, Hq, Hkv, NBmax, B, d) || D < 1 || K <= 0 || r < 0 || r >= R ||
      h < 0 || h >= Hkv)
    return -1;
  const int G = Hq / Hkv;
  const int ctx = ctx_len[r];
  // Gather the tokens of every occupied slot of this (r, h).
  std::vector<const uint16_t*> keys, vals;
  const int32_t* row = res + (static_cast<size_t>(r) * Hkv + h) * K;
  for (int s = 0; s < K; ++s) {
    const int id = row[s];
    if (id < 0 || id >= NBmax) continue;
    const int valid = valid_tokens(ctx, id, B);
    for (int t = 0; t < valid; ++t) {
      keys.push_back(host_kv + kv_index(r, h, id, 0, t, 0, Hkv, NBmax, B, d));
      vals.push_back(host_kv + kv_index(r, h, id, 1, t, 0, Hkv, NBmax, B, d));
    }
  }
  // Query vector `which`: 0 = the normal query, 1 + e = draft e.
  const size_t plane = static_cast<size_t>(R) * Hq * d;
  for (int which = 0; which <= D; ++which) {
    const uint16_t* src = which == 0 ? q : qd + (which - 1) * plane;
    for (int g = 0; g < G; ++g) {
      const int j = h * G + g;
      const uint16_t* x = src + (static_cast<size_t>(r) * Hq + j) * d;
      attend(keys, vals, x, d, scale, out + (static_cast<size_t>(which) * G + g) * d);
    }
  }
  return 0;
}

extern "C" int orc_score_rh(const uint16_t* summ, const int32_t* ctx_len,
                            const uint16_t* qd, int D, int R, int Hq, int Hkv,
                            int NBmax, int d, int B, int r, int h,
                            float* scores) {
  if (!summ || !ctx_len || !qd || !scores || !dims_ok(R, Hq, Hkv, NBmax, B, d) ||
      D < 1 || r < 0 || r >= R || h < 0 || h >= Hkv)
    return -1;
  const int G = Hq / Hkv;
  const int nb = std::min(blocks_of(ctx_len[r], B), NBmax);
  for (int b = 0; b < NBmax; ++b) {
    if (b >= nb) {
      scores[b] = -std::numeric_limits<float>::infinity();
      continue;
    }
    double acc = 0.0;
    for (int e = 0; e < D; ++e)
      for (int g = 0; g < G; ++g) {
        const uint16_t* x =
            qd + ((static_cast<size_t>(e) * R + r) * Hq + h * G + g) * d;
        for (int i = 0; i < d; ++i) {
          const double xi = widen(x[i]);
          const double lo = widen(summ[summ_index(r, h, b, 0, i, Hkv, NBmax, d)]);
          const double hi = widen(summ[summ_index(r, h, b, 1, i, Hkv, NBmax, d)]);
          acc += std::max(xi * lo, xi * hi);
        }
      }
    scores[b] = static_cast<float>(acc);
  }
  return 0;
}

extern "C" int orc_topk_rh(const float* scores, int NB, int K, int32_t* topk) {
  if (!scores || !topk || NB < 0 || K <= 0) return -1;
  std::vector<int> ids(NB);
  std::iota(ids.begin(), ids.end(), 0);
  std::sort(ids.begin(), ids.end(), [scores](int a, int b) {
    if (scores[a] != scores[b]) return scores[a] > scores[b];
    return a < b;
  });
  const int take = std::min(K, NB);
  for (int i = 0; i < K; ++i) topk[i] = i < take ? ids[i] : -1;
  return 0;
}

extern "C" int orc_admit_evict_rh(int32_t* res, int32_t* stamp,
                                  const int32_t* topk, int K, int C, int step,
                                  int32_t* admit_ids, int32_t* admit_slots,
                                  int32_t* evict_ids, int32_t* n_admit) {
  if (!res || !stamp || !topk || !admit_ids || !admit_slots || !evict_ids ||
      !n_admit || K <= 0 || C < 0 || C > K)
    return -1;
  std::set<int> selected;  // T, the step's top-K set
  for (int i = 0; i < K; ++i)
    if (topk[i] >= 0) selected.insert(topk[i]);
  std::set<int> resident;
  for (int s = 0; s < K; ++s)
    if (res[s] >= 0) resident.insert(res[s]);

  // (i) every resident block that was selected again is stamped with t.
  for (int s = 0; s < K; ++s)
    if (res[s] >= 0 && selected.count(res[s])) stamp[s] = step;

  // (ii) missing blocks, best-ranked first.
  std::vector<int> missing;
  for (int i = 0; i < K; ++i)
    if (topk[i] >= 0 && !resident.count(topk[i])) missing.push_back(topk[i]);

  // (iii) eviction candidates: slots whose block was not selected, empty
  // slots first, then least recently selected, then lower block id, then
  // lower slot index.
  std::vector<int> cand;
  for (int s = 0; s < K; ++s)
    if (res[s] < 0 || !selected.count(res[s])) cand.push_back(s);
  std::sort(cand.begin(), cand.end(), [res, stamp](int a, int b) {
    const int ea = res[a] >= 0, eb = res[b] >= 0;
    if (ea != eb) return ea < eb;
    if (stamp[a] != stamp[b]) return stamp[a] < stamp[b];
    if (res[a] != res[b]) return res[a] < res[b];
    return a < b;
  });

  // (iv) the cap.
  const int n = std::min(static_cast<int>(missing.size()), C);

  // (v) pair the i-th best missing block with the i-th eviction candidate.
  for (int i = 0; i < C; ++i) {
    admit_ids[i] = admit_slots[i] = evict_ids[i] = -1;
  }
  for (int i = 0; i < n; ++i) {
    const int s = cand[i];
    evict_ids[i] = res[s];
    res[s] = missing[i];
    stamp[s] = step;
    admit_ids[i] = missing[i];
    admit_slots[i] = s;
  }
  *n_admit = n;
  return 0;
}

extern "C" int orc_step_rh(const uint16_t* host_kv, const uint16_t* summ,
                           const int32_t* ctx_len, int32_t* res, int32_t* stamp,
                           const uint16_t* q, const uint16_t* qd, int D, int R,
                           int Hq, int Hkv, int NBmax, int B, int d, int K, int C,
                           int step, double scale, int r, int h,
                           float* attn_out, float* scores_scratch,
                           int32_t* topk, int32_t* admit_ids,
                           int32_t* admit_slots, int32_t* evict_ids,
                           int32_t* n_admit) {
  if (orc_attention_rh(host_kv, ctx_len, res, q, qd, D, R, Hq, Hkv, NBmax, B, d,
                       K, scale, r, h, attn_out))
    return -1;
  if (orc_score_rh(summ, ctx_len, qd, D, R, Hq, Hkv, NBmax, d, B, r, h,
                   scores_scratch))
    return -1;
  const int nb = std::min(blocks_of(ctx_len[r], B), NBmax);
  if (orc_topk_rh(scores_scratch, nb, K, topk)) return -1;
  const size_t off = (static_cast<size_t>(r) * Hkv + h) * K;
  return orc_admit_evict_rh(res + off, stamp + off, topk, K, C, step, admit_ids,
                            admit_slots, evict_ids, n_admit);
}

extern "C" int orc_demand_rh(const uint16_t* summ, const int32_t* ctx_len,
                             int32_t* res, int32_t* stamp, const uint16_t* q,
                             int R, int Hq, int Hkv, int NBmax, int B, int d,
                             int K, int step, int r, int h, float* scores,
                             int32_t* topk, int32_t* admit_ids,
                             int32_t* admit_slots, int32_t* evict_ids,
                             int32_t* n_admit) {
  if (!res || !stamp || r < 0 || r >= R || h < 0 || h >= Hkv) return -1;
  // The normal query ranks the blocks as one plane of query vectors.
  if (orc_score_rh(summ, ctx_len, q, 1, R, Hq, Hkv, NBmax, d, B, r, h, scores))
    return -1;
  const int nb = std::min(blocks_of(ctx_len[r], B), NBmax);
  if (orc_topk_rh(scores, nb, K, topk)) return -1;
  // Every missing block of that top-K is admitted: the cap is K.
  const size_t off = (static_cast<size_t>(r) * Hkv + h) * K;
  return orc_admit_evict_rh(res + off, stamp + off, topk, K, K, step, admit_ids,
                            admit_slots, evict_ids, n_admit);
}

extern "C" int orc_stall_step_rh(
    const uint16_t* host_kv, const uint16_t* summ, const int32_t* ctx_len,
    int32_t* res, int32_t* stamp, const uint16_t* q, const uint16_t* qd, int D,
    int R, int Hq, int Hkv, int NBmax, int B, int d, int K, int C, int step,
    double scale, int r, int h, float* dm_scores, int32_t* dm_topk,
    int32_t* dm_admit_ids, int32_t* dm_admit_slots, int32_t* dm_evict_ids,
    int32_t* dm_n_admit, float* attn_out, float* scores_scratch, int32_t* topk,
    int32_t* admit_ids, int32_t* admit_slots, int32_t* evict_ids,
    int32_t* n_admit) {
  if (orc_demand_rh(summ, ctx_len, res, stamp, q, R, Hq, Hkv, NBmax, B, d, K,
                    step, r, h, dm_scores, dm_topk, dm_admit_ids, dm_admit_slots,
                    dm_evict_ids, dm_n_admit))
    return -1;
  return orc_step_rh(host_kv, summ, ctx_len, res, stamp, q, qd, D, R, Hq, Hkv,
                     NBmax, B, d, K, C, step, scale, r, h, attn_out,
                     scores_scratch, topk, admit_ids, admit_slots, evict_ids,
                     n_admit);
}

extern "C" int orc_remote_fetch_rh(const int32_t* ids, int n, int32_t* local_map,
                                   int32_t* count, int capacity, int NBmax,
                                   int32_t* miss_ids, int32_t* miss_slots,
                                   int32_t* n_miss) {
  if (!ids || !local_map || !count || !miss_ids || !miss_slots || !n_miss ||
      n < 0 || capacity < 0 || NBmax <= 0 || *count < 0)
    return -1;
  int full = 0;
  *n_miss = 0;
  for (int i = 0; i < n; ++i) {
    const int id = ids[i];
    if (id < 0) continue;
    if (id >= NBmax) return -1;
    if (local_map[id] >= 0) continue;  // already held by the decode side
    if (*count >= capacity) {          // no slot left: stays remote
      full = 1;
      continue;
    }
    local_map[id] = *count;
    miss_ids[*n_miss] = id;
    miss_slots[*n_miss] = *count;
    ++*n_miss;
    ++*count;
  }
  return full;
}

extern "C" int orc_append_token(uint16_t* host_kv, uint16_t* summ,
                                const int32_t* ctx_len, const uint16_t* k_new,
                                const uint16_t* v_new, int R, int Hkv,
                                int NBmax, int B, int d, int r) {
  if (!host_kv || !summ || !ctx_len || !k_new || !v_new ||
      !dims_ok(R, Hkv, Hkv, NBmax, B, d) || r < 0 || r >= R)
    return -1;
  const int pos = ctx_len[r];
  if (pos < 0 || pos >= NBmax * B) return -1;
  const int b = pos / B, t = pos % B;
  for (int h = 0; h < Hkv; ++h)
    for (int i = 0; i < d; ++i) {
      const uint16_t k = k_new[static_cast<size_t>(h) * d + i];
      host_kv[kv_index(r, h, b, 0, t, i, Hkv, NBmax, B, d)] = k;
      host_kv[kv_index(r, h, b, 1, t, i, Hkv, NBmax, B, d)] =
          v_new[static_cast<size_t>(h) * d + i];
      uint16_t& lo = summ[summ_index(r, h, b, 0, i, Hkv, NBmax, d)];
      uint16_t& hi = summ[summ_index(r, h, b, 1, i, Hkv, NBmax, d)];
      if (t == 0) {
        lo = hi = k;
      } else {
        if (widen(k) < widen(lo)) lo = k;
        if (widen(k) > widen(hi)) hi = k;
      }
    }
  return 0;
}
