// strata_merge.cuh -- the merge of vocabulary-slice records (strata_merge_shards).
//
// Each slice of a row reported its k best penalised entries, its top_n raw entries and the
// log-sum-exp of its raw logits (strata_shard_rows).  The row's top_k list is among the union of
// the slices' lists, and so is its top_n raw list ("#19 serve: per-request temperature/top_p/
// top_k/min_p/penalties sampling", "min_p and the penalties": penalties, then top_k over the
// whole vocabulary; "#3200 [Engine] OpenAI logprobs / top_logprobs / allowed_token_ids ...",
// "Approach": log-probabilities of the raw logits).  One block per row ranks the union exactly
// (an entry's rank is its index in its own list plus the entries of the other lists above it,
// found by binary search: keys are distinct, since the id is part of the key), combines the
// log-sum-exps, and runs the same tail as a whole-row call: min_p, top_p, temperature, the
// Philox draw at the slot's counter, the counter advance and the outputs.
#pragma once

#include "strata_kernel.cuh"

namespace strata {

constexpr int MT = 256;  // threads of a merge block (one row)

struct MParams {
  const unsigned char* rec;  // [G][B][STRATA_SHARD_RECORD_BYTES]
  int G, B, top_n;
  const int32_t* row_slot;
  const long long* row_pos;
  int32_t* out_ids;
  float* chosen_lp;
  int32_t* top_ids;
  float* top_lps;
  int32_t* topk_ids;
  float* topk_vals;
  int32_t* kept;
  const SlotDev* slots;
  unsigned long long* ctr;
  int max_slots;
  uint32_t* err;
};

// Entries of a descending list of n keys (32-bit words `words` apart, key first) above `key`.
__device__ __forceinline__ int above_in(const uint32_t* list, int words, int n, uint64_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const uint2 o = *reinterpret_cast<const uint2*>(list + mid * words);
    if (((static_cast<uint64_t>(o.y) << 32) | o.x) > key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(MT) merge_kernel(MParams P) {
  __shared__ uint4 pen[STRATA_MAX_SHARDS * KMAX];                    // every slice's penalised list
  __shared__ uint64_t raw[STRATA_MAX_SHARDS * STRATA_MAX_TOP_N];     // every slice's raw list
  __shared__ uint4 sorted_pen[KMAX];
  __shared__ uint64_t sorted_raw[STRATA_MAX_TOP_N];
  __shared__ int cnt_p[STRATA_MAX_SHARDS], cnt_r[STRATA_MAX_SHARDS];
  __shared__ float lse_s;
  __shared__ int tot_s[2];

  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int G = P.G;
  const int slot = P.row_slot[row];
  const bool valid = slot >= 0 && slot < P.max_slots;
  SlotDev sp = {};
  if (valid) sp = P.slots[slot];
  const bool sampled = valid && (sp.flags & SLOT_SAMPLED) != 0u;
  const int k_row = valid ? min(max(sp.k, 1), KMAX) : 0;
  const int n_row = P.top_ids != nullptr ? P.top_n : 0;
  auto record = [&](int g) { return P.rec + (static_cast<size_t>(g) * P.B + row) * STRATA_SHARD_RECORD_BYTES; };

  // headers: counts (clamped to what this row uses) and the slices' log-sum-exps, combined by warp 0
  if (wid == 0) {
    float l = -INFINITY;
    int np = 0, nr = 0;
    if (lane < G) {
      const uint4 h = *reinterpret_cast<const uint4*>(record(lane));
      np = min(static_cast<int>(min(h.x, static_cast<uint32_t>(KMAX))), k_row);
      nr = min(static_cast<int>(min(h.y, static_cast<uint32_t>(STRATA_MAX_TOP_N))), n_row);
      l = __uint_as_float(h.z);
      cnt_p[lane] = np;
      cnt_r[lane] = nr;
    }
    float M = l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, off));
    float s = (lane < G && l != -INFINITY) ? expf(l - M) : 0.0f;
    int tp = np, tr = nr;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      s += __shfl_xor_sync(FULL_MASK, s, off);
      tp += __shfl_xor_sync(FULL_MASK, tp, off);
      tr += __shfl_xor_sync(FULL_MASK, tr, off);
    }
    if (lane == 0) {
      lse_s = (M == -INFINITY || !(s > 0.0f)) ? -INFINITY : M + logf(s);
      tot_s[0] = tp;
      tot_s[1] = tr;
    }
  }
  __syncthreads();
  // the lists, slice g at pen[g * KMAX] and raw[g * STRATA_MAX_TOP_N]
  for (int i = tid; i < G * KMAX; i += MT) {
    const int g = i / KMAX, j = i - g * KMAX;
    if (j < cnt_p[g]) pen[i] = *reinterpret_cast<const uint4*>(record(g) + REC_PEN + 16 * j);
  }
  for (int i = tid; i < G * STRATA_MAX_TOP_N; i += MT) {
    const int g = i / STRATA_MAX_TOP_N, j = i - g * STRATA_MAX_TOP_N;
    if (j < cnt_r[g]) {
      const uint2 o = *reinterpret_cast<const uint2*>(record(g) + REC_RAW + 8 * j);
      raw[i] = (static_cast<uint64_t>(o.y) << 32) | o.x;
    }
  }
  __syncthreads();
  // exact ranks over the union
  for (int i = tid; i < G * KMAX; i += MT) {
    const int g = i / KMAX, j = i - g * KMAX;
    if (j >= cnt_p[g]) continue;
    const uint4 e = pen[i];
    const uint64_t key = (static_cast<uint64_t>(e.y) << 32) | e.x;
    int rank = j;
    for (int h = 0; h < G && rank < k_row; ++h)
      if (h != g) rank += above_in(reinterpret_cast<const uint32_t*>(pen + h * KMAX), 4, cnt_p[h], key);
    if (rank < k_row) sorted_pen[rank] = e;
  }
  for (int i = tid; i < G * STRATA_MAX_TOP_N; i += MT) {
    const int g = i / STRATA_MAX_TOP_N, j = i - g * STRATA_MAX_TOP_N;
    if (j >= cnt_r[g]) continue;
    const uint64_t key = raw[i];
    int rank = j;
    for (int h = 0; h < G && rank < n_row; ++h)
      if (h != g) rank += above_in(reinterpret_cast<const uint32_t*>(raw + h * STRATA_MAX_TOP_N), 2, cnt_r[h], key);
    if (rank < n_row) sorted_raw[rank] = key;
  }
  __syncthreads();
  const int k_eff = min(k_row, tot_s[0]), n_eff = min(n_row, tot_s[1]);
  const float lse = lse_s;

  if (wid == 1 && n_row > 0) {  // top-N raw alternatives and their log-probabilities
    for (int i = lane; i < n_row; i += 32) {
      const long long o = static_cast<long long>(row) * P.top_n + i;
      if (i < n_eff) {
        const uint64_t key = sorted_raw[i];
        P.top_ids[o] = static_cast<int32_t>(key_id(key));
        P.top_lps[o] = key_value(static_cast<uint32_t>(key >> 32)) - lse;
      } else {
        P.top_ids[o] = -1;
        P.top_lps[o] = -INFINITY;
      }
    }
  }
  if (wid != 0) return;

  // the tail (warp 0): cuts, the counter, the draw and the outputs, as in a whole-row call
  Tail tl = {};
  if (valid && k_eff > 0) tail_cuts(sorted_pen, k_eff, sampled, sp, lane, tl);
  unsigned long long ctr_old = 0ull;
  int r_slot = 0;
  if (sampled) {
    const int rs0 = lane < P.B ? P.row_slot[lane] : -1, rs1 = lane + 32 < P.B ? P.row_slot[lane + 32] : -1;
    r_slot = slot_rows(rs0, rs1, P.row_slot, P.B, slot, lane);
    if (lane == 0) ctr_old = atomicAdd(&P.ctr[slot], r_slot == 1 ? (1ull << 16) : 1ull);
  }
  int out = -1;
  float chosen_raw = __int_as_float(0x7FC00000);
  if (!valid) {
    if (lane == 0) atomicOr(P.err, STRATA_DEVERR_SLOT);
  } else if (k_eff == 0) {
    if (lane == 0) atomicOr(P.err, STRATA_DEVERR_NOCAND);
    if (sampled) slot_arrival_done(r_slot, slot, P.ctr, ctr_old, lane);
  } else {
    int j = 0;
    if (sampled) {
      uint32_t x0 = 0u;
      if (lane == 0) x0 = philox_word0(sp.seed, static_cast<uint64_t>(P.row_pos[row]), ctr_old >> 16);
      slot_arrival_done(r_slot, slot, P.ctr, ctr_old, lane);
      j = tail_draw(tl, __shfl_sync(FULL_MASK, x0, 0), lane);
    }
    out = static_cast<int>(tail_id(tl, j));
    chosen_raw = tail_raw(tl, j);
  }
  if (lane == 0) {
    P.out_ids[row] = out;
    if (P.kept != nullptr) {
      P.kept[2 * row] = tl.m1;
      P.kept[2 * row + 1] = tl.m2;
    }
    if (P.chosen_lp != nullptr) P.chosen_lp[row] = (out >= 0) ? chosen_raw - lse : __int_as_float(0x7FC00000);
  }
  if (P.topk_ids != nullptr) {
    const long long o = static_cast<long long>(row) * KMAX;
    const bool ia = valid && lane < k_eff, ib = valid && lane + 32 < k_eff;
    P.topk_ids[o + lane] = ia ? static_cast<int32_t>(key_id((static_cast<uint64_t>(tl.ea.y) << 32) | tl.ea.x)) : -1;
    P.topk_ids[o + lane + 32] = ib ? static_cast<int32_t>(key_id((static_cast<uint64_t>(tl.eb.y) << 32) | tl.eb.x)) : -1;
    if (P.topk_vals != nullptr) {
      P.topk_vals[o + lane] = ia ? tl.va : __int_as_float(0x7FC00000);
      P.topk_vals[o + lane + 32] = ib ? tl.vb : __int_as_float(0x7FC00000);
    }
  }
}

}  // namespace strata
