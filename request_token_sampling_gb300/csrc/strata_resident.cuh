// strata_resident.cuh -- the row kernel for chunks that fit in shared memory whole.
//
// A row is split over a thread-block cluster of `cs` CTAs, each holding its chunk of the row
// (at most RES_MAX_CHUNK_BYTES) resident in shared memory for its whole life.  A CTA
//   1. issues every bulk copy of its chunk at entry (one mbarrier per 16 KiB piece), then builds
//      the history table of its id range while the bytes land, and runs the first pass piece by
//      piece: per thread the maximum and the sum of exp against a lazily moved reference;
//   2. takes its own threshold T = the K-th largest of its threads' maxima (threads that own no
//      history id; K = max(top_k, top_n)), rescans from shared memory only the threads whose
//      maximum reaches T, adds the penalised ids of the history table, and ranks the candidates
//      into its exact local top_k (penalised) and top_n (raw) lists;
//   3. sends both lists and its two (max, sum) pairs to the row's leader with asynchronous DSMEM
//      stores completed on one mbarrier (the other CTAs are done then);
//   4. the leader merges the sorted slices: the K-th largest of their heads bounds the row's K-th
//      largest from below, so only the entries at or above it are ranked, by counting; one warp
//      then runs min_p, top_p, temperature and the draw, with the Philox word computed at entry
//      whenever the draw counter can be taken there.
// Nothing is read twice from global memory except the leader's allowed-id and chosen-id logits
// (from L2, fetched ahead of use).  Every wait is a bounded mbarrier poll.
//
// The chain it computes is defined on the pages "#19 serve: per-request temperature/top_p/top_k/
// min_p/penalties sampling" (section "What changed") and "#3200 [Engine] OpenAI logprobs /
// top_logprobs / allowed_token_ids for the CUDA/HIP engine" (sections "Problem and result",
// "Approach").
#pragma once

#include "strata_kernel.cuh"

namespace strata {

constexpr int RES_MAX_CHUNK_BYTES = 64 * 1024;               // a chunk held whole in shared memory
constexpr int RES_PIECES = RES_MAX_CHUNK_BYTES / PIECE_BYTES; // bulk copies per chunk, at most
constexpr int RES_CAP = 256;                                  // candidate entries per list per CTA
constexpr int RES_SORT_MAX = RES_CAP;                         // candidates ranked by counting, at most
constexpr int RES_MERGE_BYTES = 2 * RES_SORT_MAX * 8 + RES_SORT_MAX * 16 + RES_SORT_MAX * 8;  // leader's merge scratch
constexpr int RES_QW_MAX = 16;                                // thread maxima each warp publishes, at most
constexpr int RBAR_REC = RES_PIECES;                          // leader: every CTA's candidates have landed
constexpr int RBAR_STALL = RES_PIECES + 1;                    // nothing arrives (STRATA_FLAG_TEST_STALL)
constexpr int RBAR_X0 = RES_PIECES + 2;                       // every CTA's published record has landed
constexpr int RNBAR = RES_PIECES + 3;

// Control words of the resident kernel (the candidate counters and the timeout flag sit where the
// streaming kernel keeps them, so its candidate and wait helpers serve both).
enum : int {
  RCTL_NP = CTL_CAND_PEN,  // candidates in the penalised / raw lists
  RCTL_NR = CTL_CAND_RAW,
  RCTL_FB_P = 2,           // leader: the penalised / raw merge needs exact rounds
  RCTL_TIMEOUT = CTL_TIMEOUT,
  RCTL_LSE = 4,            // leader: log-sum-exp of the row / of the allowed subset (float bits)
  RCTL_LSE_A = 5,
  RCTL_FB_R = 6,
  RCTL_ADV = 7,            // the value the counter's advancing atomic returned (its completion)
  RCTL_X0 = 8,             // Philox word 0 for the draw, when the counter was taken at entry
  RCTL_PAIR = 9,           // this CTA's (max, sum) of the row and of the allowed subset (4 words)
  RCTL_TOT_P = 13,         // leader: entries received in the penalised / raw lists
  RCTL_TOT_R = 14,
  RCTL_T = 15,             // the threshold key (atomicMin target)
  RCTL_TLO = 16,           // leader: the merge bounds of the penalised / raw lists (64-bit, atomicMin)
  RCTL_TLO_R = 18,
  RCTL_MP = 20,            // leader: merge survivors of the penalised / raw lists
  RCTL_MR = 21,
  RCTL_WORDS = 24
};
static_assert(RCTL_NP == 0 && RCTL_NR == 1 && RCTL_TIMEOUT == 3, "control words shared with the streaming kernel");
static_assert(RCTL_TLO % 2 == 0 && RCTL_TLO_R % 2 == 0, "64-bit control words");

struct RLayout {
  uint32_t data, mbar, hash, hflag, wkey, red, ctl, cand_pen, cand_raw, abits, mbits, xrec, recv_cnt, recv_pkey,
      recv_praw, recv_raw, sorted_pen, sorted_raw, total;
};

// Shared-memory layout of one CTA of the resident kernel; identical in every CTA of a launch.
// `data` holds the chunk (bytes rounded up to 16: the ragged last vector is completed with -inf).
// The allowed-id bitmap lives in the candidate region when it fits there: it is read only between
// the first pass and the first candidate append, with a block barrier in between.
__host__ __device__ inline RLayout make_res_layout(int chunk, int esz, int hash_cap, int cs, int kmax, int nmax,
                                                   int qw, bool allowed, bool mask) {
  RLayout L;
  uint32_t o = 0;
  L.data = o;  // the chunk; the leader's merge scratch once its own candidates are sent
  o += align_up(max(static_cast<uint32_t>(chunk) * static_cast<uint32_t>(esz), static_cast<uint32_t>(RES_MERGE_BYTES)), 16);
  L.mbar = o;
  o = align_up(o + RNBAR * 8, 16);
  L.hash = o;
  o += align_up(static_cast<uint32_t>(hash_cap) * 4, 16);
  L.hflag = o;
  o += NT / 8;
  L.wkey = o;
  o += NW * RES_QW_MAX * 4;
  L.red = o;
  o += NW * 16;
  L.ctl = o;
  o = align_up(o + RCTL_WORDS * 4, 16);
  L.cand_pen = o;  // RES_CAP entries of (key lo, key hi, raw logit, 0)
  o += RES_CAP * 16;
  L.cand_raw = o;  // RES_CAP raw keys
  o += RES_CAP * 8;
  const uint32_t bw = align_up((static_cast<uint32_t>(chunk) + 31) / 32 * 4, 16);
  const bool abits_in_cand = bw <= static_cast<uint32_t>(RES_CAP) * 24u;
  L.abits = abits_in_cand ? L.cand_pen : o;
  o += (allowed && !abits_in_cand) ? bw : 0u;
  L.mbits = o;
  o += mask ? bw : 0u;
  L.xrec = o;  // every CTA's published record: its NW * qw keys, then its two (max, sum) pairs
  o += static_cast<uint32_t>(cs * (NW * qw + 4)) * 4;
  L.recv_cnt = o;  // leader: entries each CTA sent (penalised, raw)
  o += align_up(static_cast<uint32_t>(cs) * 8, 16);
  L.recv_pkey = o;  // leader: each CTA's penalised keys, kmax per CTA, in rank order
  o = align_up(o + static_cast<uint32_t>(cs * kmax) * 8, 16);
  L.recv_praw = o;  // their raw logits
  o = align_up(o + static_cast<uint32_t>(cs * kmax) * 4, 16);
  L.recv_raw = o;   // leader: each CTA's raw keys, nmax per CTA, in rank order
  o = align_up(o + static_cast<uint32_t>(cs * nmax) * 8, 16);
  L.sorted_pen = o;
  o += static_cast<uint32_t>(kmax) * 16;
  L.sorted_raw = o;
  o += static_cast<uint32_t>(nmax) * 8;
  L.total = align_up(o, 128);
  return L;
}

__host__ __device__ inline bool res_layout_aligned(const RLayout& L) {
  const uint32_t r[] = {L.data, L.mbar, L.hash, L.hflag, L.wkey, L.red, L.ctl, L.cand_pen, L.cand_raw, L.abits,
                        L.mbits, L.xrec, L.recv_cnt, L.recv_pkey, L.recv_praw, L.recv_raw, L.sorted_pen,
                        L.sorted_raw};
  for (uint32_t x : r)
    if (x % 16u != 0u) return false;
  return true;
}

// First pass over this thread's vectors of piece p (all in shared memory), 16 elements at a time:
// the running max and the sum of exp(x - ref) in two partial sums, the reference moving only when a
// batch's max passes it by LAZY_SHIFT.
template <int DT>
__device__ __forceinline__ void res_pass_piece(const unsigned char* data, int p, int n_vec, float& ref, float& mx,
                                               float& s0, float& s1) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  constexpr int RB = BATCH_VECS<DT>;
#pragma unroll
  for (int r0 = 0; r0 < VR; r0 += RB) {
    float x[RB][EPV];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int v = p * PIECE_VECS + static_cast<int>(threadIdx.x) + (r0 + r) * NT;
      if (v < n_vec) {
        load_vec<DT>(data, v, x[r]);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) x[r][e] = -INFINITY;
      }
    }
    float pm = x[0][0];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int e = 0; e < EPV; ++e) pm = fmaxf(pm, x[r][e]);
    mx = fmaxf(mx, pm);
    if (pm > ref + LAZY_SHIFT) {
      const float f = (ref == -INFINITY) ? 0.0f : ex2_approx((ref - pm) * LOG2E);
      s0 *= f;
      s1 *= f;
      ref = pm;
    }
    if (ref != -INFINITY) {
      const float mb = ref * LOG2E;
#pragma unroll
      for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int e = 0; e < EPV; e += 2) {
          s0 += ex2_approx(fmaf(x[r][e], LOG2E, -mb));
          s1 += ex2_approx(fmaf(x[r][e + 1], LOG2E, -mb));
        }
    }
  }
}

// A threshold key for a thread that owns history ids: the largest order key of min(raw,
// penalised) over its elements (vectors tid, tid + NT, ... of the resident chunk).  Both the raw
// and the penalised value of that id reach it.  The history table is looked up only for elements
// that could raise the key.
template <int DT>
__device__ __noinline__ uint32_t res_safe_key(const unsigned char* data, int n_vec, int n_el, const uint32_t* htab,
                                              int hash_bits, float rep, float freq, float pres) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  uint32_t best = 0u;
  for (int v = threadIdx.x; v < n_vec; v += NT) {
    float x[EPV];
    load_vec<DT>(data, v, x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const uint32_t loc = static_cast<uint32_t>(v * EPV + e);
      if (loc >= static_cast<uint32_t>(n_el) || order_key(x[e]) <= best) continue;
      const uint32_t c = hash_count(htab, hash_bits, loc);
      best = max(best, order_key(c != 0u ? fminf(x[e], penalize(x[e], c, rep, freq, pres)) : x[e]));
    }
  }
  return best;
}

// Exact argmax rounds over the resident chunk: the `need` largest keys in order (list 0: penalised
// values, with their raw logits, into cand_pen; list 1: raw values into cand_raw).  Only taken when
// more candidates reach the threshold than the candidate buffer holds (very long runs of ties); out
// of line.  A penalised value needs the history table only for the elements of threads that own a
// history id (`hflag`; thread t owns vectors t, t + NT, ...).  Every thread of the block calls it.
template <int DT>
__device__ __noinline__ int res_exact_rounds(const unsigned char* data, int n_vec, int n_el, int lo, int list,
                                             int need, bool penal, const uint32_t* htab, int hash_bits,
                                             const uint32_t* hflag, float rep, float freq, float pres,
                                             uint64_t* red64, uint4* cand_pen, uint64_t* cand_raw) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool owner = list == 0 && penal && ((hflag[tid >> 5] >> (tid & 31)) & 1u);
  uint64_t prev = ~0ull;
  int got = 0;
  for (int r = 0; r < need; ++r) {
    uint64_t best = 0ull;
    float best_raw = 0.0f;
    for (int v = tid; v < n_vec; v += NT) {
      float x[EPV];
      load_vec<DT>(data, v, x);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const uint32_t loc = static_cast<uint32_t>(v * EPV + e);
        if (loc >= static_cast<uint32_t>(n_el)) continue;
        float pv = x[e];
        if (owner) {
          const uint32_t c = hash_count(htab, hash_bits, loc);
          if (c != 0u) pv = penalize(pv, c, rep, freq, pres);
        }
        const uint32_t o = order_key(pv);
        if (o == 0u) continue;
        const uint64_t key = sel_key(o, static_cast<uint32_t>(lo) + loc);
        if (key < prev && key > best) {
          best = key;
          best_raw = x[e];
        }
      }
    }
    const uint64_t m = block_max_u64(best, red64, lane, wid);
    if (m == 0ull) break;
    if (best == m) {  // keys are distinct: one thread holds it
      if (list == 0) cand_pen[r] = make_uint4(static_cast<uint32_t>(m), static_cast<uint32_t>(m >> 32), __float_as_uint(best_raw), 0u);
      else cand_raw[r] = m;
    }
    prev = m;
    got = r + 1;
  }
  __syncthreads();
  return got;
}

// Add `n` occurrences of chunk-local id `loc` to the open-addressing count table: returns the
// entry's index when this call created it, -1 when the id was already there, -2 when the table is
// full.
__device__ __forceinline__ int hash_add_n(uint32_t* tab, int bits, uint32_t loc, uint32_t n) {
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t h = hash_slot(loc, bits);
  for (uint32_t i = 0; i <= mask; ++i) {
    uint32_t cur = *reinterpret_cast<volatile uint32_t*>(&tab[h]);
    if (cur == HASH_EMPTY) {
      const uint32_t prev = atomicCAS(&tab[h], HASH_EMPTY, (loc << HASH_CNT_BITS) | n);
      if (prev == HASH_EMPTY) return static_cast<int>(h);
      cur = prev;
    }
    if ((cur >> HASH_CNT_BITS) == loc) {
      atomicAdd(&tab[h], n);
      return -1;
    }
    h = (h + 1u) & mask;
  }
  return -2;
}

// Rank of `key` in a dense list of 64-bit keys padded with zero keys to a multiple of 8 entries
// (at least n): the number of larger keys, eight independent broadcast loads per iteration summed in
// four partial counts.  A short loop rather than a fully unrolled one: the kernel's code stays small.
// `stride_words` is the entry size in 32-bit words (key first).
__device__ __forceinline__ int rank_pad(const uint32_t* list, int stride_words, int n, uint64_t key) {
  int a[4] = {0, 0, 0, 0};
  const int n8 = (n + 7) & ~7;
#pragma unroll 1
  for (int j = 0; j < n8; j += 8) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint2 o = *reinterpret_cast<const uint2*>(list + (j + t) * stride_words);
      a[t & 3] += ((static_cast<uint64_t>(o.y) << 32) | o.x) > key;
    }
  }
  return (a[0] + a[1]) + (a[2] + a[3]);
}

// Exact argmax rounds over the received slices of one list (the leader's rare fallback, when its
// bound leaves more than RES_SORT_MAX survivors): the k largest keys in order to sorted[] (entry
// size `out_words`, key first, then the payload for the penalised list).  Every thread calls it.
__device__ __noinline__ int leader_rounds(int cs, int stride, int k, const uint2* recv_cnt, bool pen,
                                          const uint64_t* keys, const uint32_t* pays, uint32_t* sorted,
                                          int out_words, uint64_t* red64) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  uint64_t prev = ~0ull;
  int got = 0;
  for (int r = 0; r < k; ++r) {
    uint64_t best = 0ull;
    uint32_t best_pay = 0u;
    for (int j = tid; j < cs * stride; j += NT) {
      const int c = j / stride, i = j - c * stride;
      const int cnt = min(static_cast<int>(pen ? recv_cnt[c].x : recv_cnt[c].y), stride);
      if (i >= cnt) continue;
      const uint64_t key = keys[j];
      if (key < prev && key > best) {
        best = key;
        best_pay = pays != nullptr ? pays[j] : 0u;
      }
    }
    const uint64_t m = block_max_u64(best, red64, lane, wid);
    if (m == 0ull) break;
    if (best == m) {  // keys are distinct: one thread holds it
      sorted[r * out_words] = static_cast<uint32_t>(m);
      sorted[r * out_words + 1] = static_cast<uint32_t>(m >> 32);
      if (out_words > 2) sorted[r * out_words + 2] = best_pay;
    }
    prev = m;
    got = r + 1;
  }
  __syncthreads();
  return got;
}

// ------------------------------------------------------------------------------ the kernel
template <int DT, bool MASK, bool OWN = false>
__global__ void __launch_bounds__(NT, 3) res_kernel(const KParams P) {
  extern __shared__ __align__(128) unsigned char sm[];
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int EPV = 16 / ESZ;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool early = (P.flags & STRATA_FLAG_EARLY_LOAD) != 0u;
  const bool own_out = OWN && early;
  if (!early) grid_dep_wait();  // inputs may be the previous kernel's outputs
  if (!own_out) grid_dep_launch();

  const uint32_t crank = cluster_ctarank();
  const int cs = P.cs;
  const int row = blockIdx.x / cs;
  const bool mask_launch = MASK && P.mode == MODE_SAMPLE && P.allowed_off != nullptr;
  const RLayout L = make_res_layout(P.chunk, ESZ, P.hash_cap, cs, P.kmax, P.nmax, P.qw, P.allowed_off != nullptr,
                                    mask_launch);
  const int lo = static_cast<int>(crank) * P.chunk;
  const int hi = min(P.V, lo + P.chunk);
  const int n_el = max(0, hi - lo);
  const int bytes = n_el * ESZ;
  const int bytes_al = bytes & ~15;
  const int n_vec = (bytes + 15) >> 4;
  const int n_full = bytes_al >> 4;
  const int n_pieces = (bytes_al + PIECE_BYTES - 1) / PIECE_BYTES;
  constexpr int cap = RES_CAP;

  unsigned char* data = sm + L.data;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + L.mbar);
  const char* grow = static_cast<const char*>(P.logits) + (static_cast<long long>(row) * P.ld + lo) * ESZ;

  int slot = -1;
  unsigned long long pos = 0ull;
  int chosen_id = -1;
  int a_beg = 0, a_end = 0;
  auto load_meta1 = [&]() {
    if (P.mode == MODE_SAMPLE) {
      slot = P.row_slot[row];
      pos = static_cast<unsigned long long>(P.row_pos[row]);
    } else if (P.chosen != nullptr) {
      chosen_id = P.chosen[row];
    }
    if (P.allowed_off != nullptr) {
      a_beg = P.allowed_off[row];
      a_end = P.allowed_off[row + 1];
    }
  };
  if (tid != 0) load_meta1();

  // ---- 1. every bulk copy of the chunk at entry ------------------------------------------------
  if (tid == 0) {
    for (int p = 0; p < n_pieces; ++p) mbar_init(&mbar[p], 1);
    fence_proxy_async_smem();
    for (int p = 0; p < n_pieces; ++p) {
      const uint32_t nb = static_cast<uint32_t>(min(PIECE_BYTES, bytes_al - p * PIECE_BYTES));
      mbar_arrive_expect_tx(&mbar[p], nb);
      bulk_g2s(data + p * PIECE_BYTES, grow + p * PIECE_BYTES, nb, &mbar[p]);
    }
    mbar_init(&mbar[RBAR_REC], cs > 1 ? cs - 1 : 1);  // one arrival per other CTA (leader only)
    mbar_init(&mbar[RBAR_STALL], 1);
    mbar_init(&mbar[RBAR_X0], 2);                     // the announced bytes + this CTA's own record
    fence_mbar_init();
    mbar_arrive_expect_tx(&mbar[RBAR_X0], static_cast<uint32_t>((cs - 1) * (NW * P.qw + 4) * 4));
    load_meta1();
  }
  // the ragged last vector (a chunk whose bytes are not a multiple of 16): read directly and
  // completed with -inf, so that the whole chunk is whole vectors in shared memory
  if (tid == 32 && n_vec > n_full) {
    uint32_t wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) wv[i] = DT == 0 ? 0xFF800000u : 0xFF80FF80u;
    for (int e = 0; e < n_el - n_full * EPV; ++e) {
      if constexpr (DT == 0) {
        wv[e] = __float_as_uint(reinterpret_cast<const float*>(grow)[n_full * EPV + e]);
      } else {
        const uint32_t b = reinterpret_cast<const uint16_t*>(grow)[n_full * EPV + e];
        const int sh = 16 * (e & 1);
        wv[e >> 1] = (wv[e >> 1] & ~(0xFFFFu << sh)) | (b << sh);
      }
    }
    *reinterpret_cast<uint4*>(data + n_full * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }

  uint32_t* htab = reinterpret_cast<uint32_t*>(sm + L.hash);
  uint32_t* hflag = reinterpret_cast<uint32_t*>(sm + L.hflag);
  uint32_t* wkey = reinterpret_cast<uint32_t*>(sm + L.wkey);
  uint64_t* red64 = reinterpret_cast<uint64_t*>(sm + L.red);
  float4* red4 = reinterpret_cast<float4*>(sm + L.red);
  uint32_t* ctl = reinterpret_cast<uint32_t*>(sm + L.ctl);
  uint4* cand_pen = reinterpret_cast<uint4*>(sm + L.cand_pen);
  uint64_t* cand_raw = reinterpret_cast<uint64_t*>(sm + L.cand_raw);
  uint32_t* abits = reinterpret_cast<uint32_t*>(sm + L.abits);
  uint32_t* mbits = reinterpret_cast<uint32_t*>(sm + L.mbits);
  uint2* recv_cnt = reinterpret_cast<uint2*>(sm + L.recv_cnt);
  uint32_t* xrec = reinterpret_cast<uint32_t*>(sm + L.xrec);
  uint64_t* recv_pkey = reinterpret_cast<uint64_t*>(sm + L.recv_pkey);
  uint32_t* recv_praw = reinterpret_cast<uint32_t*>(sm + L.recv_praw);
  uint64_t* recv_raw = reinterpret_cast<uint64_t*>(sm + L.recv_raw);
  uint4* sorted_pen = reinterpret_cast<uint4*>(sm + L.sorted_pen);
  uint64_t* sorted_raw = reinterpret_cast<uint64_t*>(sm + L.sorted_raw);

  const int bw_words = (P.chunk + 31) >> 5;
  if (P.allowed_off != nullptr)
    for (int i = tid; i < bw_words; i += NT) {
      abits[i] = 0u;
      if (mask_launch) mbits[i] = 0u;
    }
  for (int i = tid; i < P.hash_cap; i += NT) htab[i] = HASH_EMPTY;
  if (tid < NT / 32) hflag[tid] = 0u;
  if (tid < RCTL_WORDS) ctl[tid] = (tid == RCTL_T || (tid >= RCTL_TLO && tid < RCTL_TLO_R + 2)) ? 0xFFFFFFFFu : 0u;
  for (int i = tid; i < NW * RES_QW_MAX; i += NT) wkey[i] = 0u;
  __syncthreads();           // tables zeroed, barriers initialised, the ragged vector in place
  cluster_arrive_relaxed();  // this CTA is running (remote stores wait for every CTA, below)

  // ---- row metadata, second level ---------------------------------------------------------------
  bool valid = true;
  SlotDev sp{};
  if (P.mode == MODE_SAMPLE) {
    valid = static_cast<unsigned>(slot) < static_cast<unsigned>(P.max_slots);
    if (valid) sp = P.slots[slot];
  }
  const bool sampled = valid && (sp.flags & SLOT_SAMPLED);
  const int k_row = (P.mode == MODE_SAMPLE && valid) ? min(max(sp.k, 1), P.kmax) : 0;
  const int n_row = P.nmax;
  const int kp = max(k_row, n_row);
  const bool kept_hist = P.ring != nullptr;
  const bool penal = (P.mode == MODE_SAMPLE) && valid && (sp.flags & SLOT_PENAL) && P.hash_cap > 0 &&
                     (kept_hist || (P.hist_off != nullptr && slot < P.n_hist_slots));
  int h_len = 0;
  uint32_t h_start = 0u, h_mask = 0xFFFFFFFFu;
  const int32_t* hb = P.hist;
  if (penal) {
    if (kept_hist) {
      hb = P.ring + static_cast<size_t>(slot) * STRATA_HISTORY_CAP;
      h_mask = STRATA_HISTORY_CAP - 1;
    } else {
      const int hs = P.hist_off[slot], he = P.hist_off[slot + 1];
      h_len = min(sp.last_n, max(0, he - hs));
      h_start = static_cast<uint32_t>(he - h_len);
    }
  }
  int aid[APRE];  // the first allowed ids of this thread
#pragma unroll
  for (int t = 0; t < APRE; ++t) {
    const int j = a_beg + tid + t * NT;
    aid[t] = j < a_end ? P.allowed[j] : -1;
  }

  // The draw counter (leader's warp 0 of a sampled row).  A call that owns its outputs takes it
  // now, before the next call may launch, and computes its Philox word while the bytes land; a
  // call that waited for its predecessor at entry issues the atomic after the first pass (its value
  // is first needed by the draw); a call with early loads and shared outputs takes it after
  // waiting for its predecessor, before the draw.
  const bool ctr_warp = k_row > 0 && wid == 0 && crank == 0 && sampled;
  const bool ctr_thread = ctr_warp && lane == 0;
  const bool ctr_at_entry = own_out;
  unsigned long long ctr_old = 0ull;
  int rs_pre[2] = {-1, -1};
  if (crank == 0 && wid == 0 && P.mode == MODE_SAMPLE) {
    rs_pre[0] = lane < P.B ? P.row_slot[lane] : -1;
    rs_pre[1] = lane + 32 < P.B ? P.row_slot[lane + 32] : -1;
  }
  int r_slot = 0;
  if (ctr_at_entry && ctr_warp) {
    const int rs = slot_rows(rs_pre[0], rs_pre[1], P.row_slot, P.B, slot, lane);
    if (lane == 0) {
      const unsigned long long v = atomicAdd(&P.ctr[slot], rs == 1 ? (1ull << 16) : 1ull);
      uint32_t adv = 0u;
      if (rs > 1 && (v & 0xFFFFull) + 1ull == static_cast<unsigned long long>(rs))
        adv = static_cast<uint32_t>(atomicAdd(&P.ctr[slot], (1ull << 16) - static_cast<unsigned long long>(rs)));
      ctl[RCTL_ADV] = adv;  // stores both returned values: both atomics have been performed
      ctr_old = v;
      ctl[RCTL_X0] = philox_word0(sp.seed, pos, v >> 16);
    }
  }
  if (own_out) {
    // the counters are taken before any CTA lets the next call launch: that call's atomics on
    // these words come after these have returned
    __syncthreads();
    grid_dep_launch();
  }

  // ---- the history window: this thread's first ids are fetched ahead of the first pass and the
  // table of this chunk's id range is built after it (a kept history read with early loads waits
  // for the previous call first) ------------------------------------------------------------------
  // repeats of an id among the lanes of a warp are counted by one lane (windows repeat popular ids,
  // and atomics on one table word serialise)
  auto add_hist = [&](int id) {
    const bool in = id >= lo && id < hi;
    const uint32_t loc = static_cast<uint32_t>(id - lo);
    const uint32_t grp = __match_any_sync(__activemask(), in ? loc : 0x80000000u | static_cast<uint32_t>(lane));
    if (in && (grp & ((1u << lane) - 1u)) == 0u) {
      const uint32_t owner = (loc / EPV) % NT;
      atomicOr(&hflag[owner >> 5], 1u << (owner & 31));
      if (hash_add_n(htab, P.hash_bits, loc, static_cast<uint32_t>(__popc(grp))) == -2)
        atomicOr(P.err, STRATA_DEVERR_HISTORY);
    }
  };
  const bool hist_late = penal && kept_hist && early;
  if (penal && kept_hist && !early) {
    const unsigned long long n = P.hlen[slot];
    h_len = static_cast<int>(min(static_cast<unsigned long long>(sp.last_n), n));
    h_start = static_cast<uint32_t>(n - static_cast<unsigned long long>(h_len)) & h_mask;
  }
  int hid[HPRE];
#pragma unroll
  for (int j = 0; j < HPRE; ++j) {
    const int i = tid + j * NT;
    hid[j] = (penal && !hist_late && i < h_len) ? hb[(h_start + static_cast<uint32_t>(i)) & h_mask] : -1;
  }

  // ---- first pass as the pieces land --------------------------------------------------------------
  float ref = -INFINITY, mx = -INFINITY, s0 = 0.0f, s1 = 0.0f;
  {
    const int n_iter = (n_vec + PIECE_VECS - 1) / PIECE_VECS;
#pragma unroll 1
    for (int p = 0; p < n_iter; ++p) {
      if (p < n_pieces) wait_bar(&mbar[p], ctl, P.err, false, 0u);
      res_pass_piece<DT>(data, p, n_vec, ref, mx, s0, s1);
    }
  }
  if (!early && ctr_warp) {  // the previous kernel ended before this one started
    r_slot = slot_rows(rs_pre[0], rs_pre[1], P.row_slot, P.B, slot, lane);
    if (lane == 0) ctr_old = atomicAdd(&P.ctr[slot], r_slot == 1 ? (1ull << 16) : 1ull);
  }
  if (hist_late) {
    grid_dep_wait();
    const unsigned long long n = P.hlen[slot];
    h_len = static_cast<int>(min(static_cast<unsigned long long>(sp.last_n), n));
    h_start = static_cast<uint32_t>(n - static_cast<unsigned long long>(h_len)) & h_mask;
#pragma unroll
    for (int j = 0; j < HPRE; ++j) {
      const int i = tid + j * NT;
      hid[j] = i < h_len ? hb[(h_start + static_cast<uint32_t>(i)) & h_mask] : -1;
    }
  }
  if (penal) {
#pragma unroll
    for (int j = 0; j < HPRE; ++j) add_hist(hid[j]);
    for (int i = tid + HPRE * NT; i < h_len; i += NT) add_hist(hb[(h_start + static_cast<uint32_t>(i)) & h_mask]);
  }

  // allowed subset: this chunk's ids, each counted once, into (max, sum of exp)
  MaxSum al{-INFINITY, 0.0f};
  {
    auto add_allowed = [&](int id) {
      if (id >= lo && id < hi) {
        const uint32_t loc = static_cast<uint32_t>(id - lo);
        const uint32_t bit = 1u << (loc & 31);
        if (!(atomicOr(&abits[loc >> 5], bit) & bit)) online_add(al, elem_at<DT>(data, loc));
      }
    };
#pragma unroll
    for (int t = 0; t < APRE; ++t) add_allowed(aid[t]);
    for (int j = a_beg + tid + APRE * NT; j < a_end; j += NT) add_allowed(P.allowed[j]);
  }

  // ---- 2. the CTA's threshold and (max, sum) pairs ------------------------------------------------
  const uint32_t kall = tid < n_vec ? order_key(mx) : 0u;
  __syncthreads();  // the history table and its owner flags are complete
  const bool own_hist = penal && ((hflag[tid >> 5] >> (tid & 31)) & 1u);
  // a threshold key must be a value that both the raw and the penalised value of one id reach: a
  // thread that owns a history id publishes nothing, unless its warp has fewer than qw threads
  // without one; then it publishes the best min(raw, penalised) over its elements
  uint32_t kthr = own_hist ? 0u : kall;
  if (penal) {
    const uint32_t plain = __ballot_sync(FULL_MASK, !own_hist);
    if (own_hist && kall != 0u && __popc(plain) < P.qw)
      kthr = res_safe_key<DT>(data, n_vec, n_el, htab, P.hash_bits, sp.rep, sp.freq, sp.pres);
  }
  {
    uint32_t kk = kthr;
#pragma unroll 1
    for (int r = 0; r < P.qw; ++r) {  // the warp's r-th largest thread maximum, then drop it
      const uint32_t m = __reduce_max_sync(FULL_MASK, kk);
      if (lane == 0) wkey[r * NW + wid] = m;  // dense: key r * NW + w is warp w's r-th largest
      const uint32_t b = __ballot_sync(FULL_MASK, kk == m);
      if (lane == __ffs(b) - 1) kk = 0u;
    }
    const MaxSum wrow = warp_ms_fast(MaxSum{ref, s0 + s1});
    const MaxSum wal = warp_ms_fast(al);
    if (lane == 0) red4[wid] = make_float4(wrow.m, wrow.s, wal.m, wal.s);
  }
  __syncthreads();  // the published keys and per-warp pairs; the allowed bitmap is no longer read
  const int Q = NW * P.qw;  // keys this CTA publishes
  const int XW = Q + 4;      // record stride in words (a multiple of 4)
  if (wid == 0) {
    // the CTA's (max, sum) pairs: lanes 0..NW-1 combine the row's, lanes 16..16+NW-1 the allowed
    // subset's; then this CTA's record (keys, pairs) in its own slot of every CTA's records
    const int g = lane >> 4, w8 = lane & 15;
    float m = -INFINITY, sum = 0.0f;
    if (w8 < NW) {
      const float4 t = red4[w8];
      m = g ? t.z : t.x;
      sum = g ? t.w : t.y;
    }
    float M = m;
#pragma unroll
    for (int off = NW / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, off));
    float sc = (m == -INFINITY || !(sum > 0.0f)) ? 0.0f : sum * ex2_approx((m - M) * LOG2E);
#pragma unroll
    for (int off = NW / 2; off > 0; off >>= 1) sc += __shfl_xor_sync(FULL_MASK, sc, off);
    const float Ma = __shfl_sync(FULL_MASK, M, 16), Sa = __shfl_sync(FULL_MASK, sc, 16);
    uint32_t* own = xrec + crank * XW;
    for (int i = lane; i < Q; i += 32) own[i] = wkey[i];
    if (lane == 0)
      *reinterpret_cast<uint4*>(own + Q) =
          make_uint4(__float_as_uint(M), __float_as_uint(sc), __float_as_uint(Ma), __float_as_uint(Sa));
    __syncwarp();
    if (lane == 0) mbar_arrive(&mbar[RBAR_X0]);  // own record in place (release by this lane)
    __syncwarp();
  }
  // the candidate lists' first RES_SORT_MAX entries are zero (the padding the ranks count over);
  // the allowed-id bitmap that shared the region is no longer read
  for (int i = tid; i < RES_SORT_MAX; i += NT) {
    cand_pen[i] = make_uint4(0u, 0u, 0u, 0u);
    cand_raw[i] = 0ull;
  }
  cluster_wait();  // every CTA of the cluster is running: remote stores are safe from here on
  if (wid == 0 && lane < cs && static_cast<uint32_t>(lane) != crank) {
    const uint4* own = reinterpret_cast<const uint4*>(xrec + crank * XW);
    const uint32_t dst = dsmem_addr(smem_u32(xrec + crank * XW), static_cast<uint32_t>(lane));
    const uint32_t bar = dsmem_addr(smem_u32(&mbar[RBAR_X0]), static_cast<uint32_t>(lane));
#pragma unroll 1
    for (int i = 0; i < XW / 4; ++i) {
      const uint4 v = own[i];
      st_async_v4(dst + 16u * i, v.x, v.y, v.z, v.w, bar);
    }
  }
  wait_bar(&mbar[RBAR_X0], ctl, P.err, true);  // every CTA's record is here
  // T = the kp-th largest of the row's cs * Q published keys (zeros included, so T = 0 when fewer
  // than kp real keys exist): the smallest published key with fewer than kp keys above it.  They are
  // values of distinct ids without a penalty, so at least kp ids of the row reach T, raw and
  // penalised alike.  One thread per key counts, lpk consecutive lanes per key over records
  // sub, sub + lpk, ...
  if (kp > 0) {
    const int nk = cs * Q;
    const int qlog = 31 - __clz(Q);  // Q is a power of two
    int lpk = 1;
    while (lpk < 16 && nk * lpk * 2 <= NT) lpk *= 2;
    const int llog = 31 - __clz(lpk), sub = tid & (lpk - 1);
#pragma unroll 1
    for (int base = 0; base < nk * lpk; base += NT) {
      const int i = (base + tid) >> llog;
      uint32_t u = 0xFFFFFFFFu;
      int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
      if (i < nk) {
        u = xrec[(i >> qlog) * XW + (i & (Q - 1))];
#pragma unroll 1
        for (int c = sub; c < cs; c += lpk) {
          const uint4* rk = reinterpret_cast<const uint4*>(xrec + c * XW);
#pragma unroll 4
          for (int j = 0; j < (Q >> 2); ++j) {
            const uint4 v = rk[j];
            a0 += v.x > u;
            a1 += v.y > u;
            a2 += v.z > u;
            a3 += v.w > u;
          }
        }
      }
      int above = (a0 + a1) + (a2 + a3);
      for (int off = 1; off < lpk; off <<= 1) above += __shfl_xor_sync(FULL_MASK, above, off);
      const uint32_t cand = (i < nk && sub == 0 && above < kp) ? u : 0xFFFFFFFFu;
      const uint32_t wmin = __reduce_min_sync(FULL_MASK, cand);
      if (lane == 0 && wmin != 0xFFFFFFFFu) atomicMin(&ctl[RCTL_T], wmin);
    }
  }
  __syncthreads();  // T, the zeroed candidate lists
  const uint32_t T = (kp > 0 && cs * Q >= kp) ? ctl[RCTL_T] : 0u;

  // ---- 3. candidates from shared memory: every element at or above T --------------------------
  const bool masked = mask_launch && a_end > a_beg && k_row > 0;
  const bool pen_from_t = k_row > 0 && !masked;
  if (kp > 0) {
    const float Tf = T == 0u ? -INFINITY : key_value(T);
    const bool want = kall != 0u && kall >= T && (n_row > 0 || pen_from_t);
    const bool to_raw = n_row > 0;
    if (want) {
      // this thread's vectors (at most 16 in a resident chunk): count the hits, take their places
      // with one atomic per list, then write them (a hit costs no atomic of its own)
      constexpr int VPT = RES_MAX_CHUNK_BYTES / 16 / NT;
      auto hits_of = [&](int j, float (&x)[EPV]) -> uint32_t {
        const int v = tid + j * NT;
        uint32_t good = 0u;
        if (v < n_vec) {
          load_vec<DT>(data, v, x);
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const uint32_t loc = static_cast<uint32_t>(v * EPV + e);
            // NaN compares false; order key 0 is NaN; history ids are the table's
            if (x[e] >= Tf && loc < static_cast<uint32_t>(n_el) && order_key(x[e]) != 0u &&
                !(own_hist && hash_count(htab, P.hash_bits, loc) != 0u))
              good |= 1u << e;
          }
        }
        return good;
      };
      int cnt = 0;
#pragma unroll 4
      for (int j = 0; j < VPT; ++j) {
        float x[EPV];
        cnt += __popc(hits_of(j, x));
      }
      int bp = 0, br = 0;
      if (pen_from_t) bp = static_cast<int>(atomicAdd(&ctl[RCTL_NP], static_cast<uint32_t>(cnt)));
      if (to_raw) br = static_cast<int>(atomicAdd(&ctl[RCTL_NR], static_cast<uint32_t>(cnt)));
#pragma unroll 1
      for (int j = 0; j < VPT && cnt > 0; ++j) {
        float x[EPV];
        uint32_t good = hits_of(j, x);
        const int v = tid + j * NT;
#pragma unroll 1
        for (; good != 0u; good &= good - 1u, ++bp, ++br, --cnt) {
          const int e = __ffs(good) - 1;
          const float xv = pick(x, e);
          const uint64_t key = sel_key(order_key(xv), static_cast<uint32_t>(lo + v * EPV + e));
          if (pen_from_t && bp < cap)
            cand_pen[bp] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32), __float_as_uint(xv), 0u);
          if (to_raw && br < cap) cand_raw[br] = key;
        }
      }
    }
    if (penal) {  // penalised ids: raw value for the raw list, penalised value for the other
      int cr = 0, cp = 0;
      for (int i = tid; i < P.hash_cap; i += NT) {
        const uint32_t ent = htab[i];
        if (ent == HASH_EMPTY) continue;
        const uint32_t loc = ent >> HASH_CNT_BITS;
        const float raw = elem_at<DT>(data, loc);
        const uint32_t o = order_key(raw);
        cr += (o != 0u && o >= T && to_raw) ? 1 : 0;
        const uint32_t op = order_key(penalize(raw, ent & ((1u << HASH_CNT_BITS) - 1u), sp.rep, sp.freq, sp.pres));
        cp += (op != 0u && op >= T && pen_from_t) ? 1 : 0;
      }
      int br = cr > 0 ? static_cast<int>(atomicAdd(&ctl[RCTL_NR], static_cast<uint32_t>(cr))) : 0;
      int bp = cp > 0 ? static_cast<int>(atomicAdd(&ctl[RCTL_NP], static_cast<uint32_t>(cp))) : 0;
      for (int i = tid; i < P.hash_cap && (cr > 0 || cp > 0); i += NT) {
        const uint32_t ent = htab[i];
        if (ent == HASH_EMPTY) continue;
        const uint32_t loc = ent >> HASH_CNT_BITS;
        const float raw = elem_at<DT>(data, loc);
        const uint32_t id = static_cast<uint32_t>(lo) + loc;
        const uint32_t o = order_key(raw);
        if (o != 0u && o >= T && to_raw) {
          if (br < cap) cand_raw[br] = sel_key(o, id);
          ++br;
          --cr;
        }
        const uint32_t op = order_key(penalize(raw, ent & ((1u << HASH_CNT_BITS) - 1u), sp.rep, sp.freq, sp.pres));
        if (op != 0u && op >= T && pen_from_t) {
          const uint64_t key = sel_key(op, id);
          if (bp < cap)
            cand_pen[bp] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32), __float_as_uint(raw), 0u);
          ++bp;
          --cp;
        }
      }
    }
    if (masked)  // every named id of this chunk once, with its penalised value
      masked_candidates<DT>(data, lo, hi, aid[0], aid[1], aid[2], aid[3], P.allowed, a_beg + tid + APRE * NT, a_end,
                            mbits, penal, htab, P.hash_bits, sp.rep, sp.freq, sp.pres, ctl, cand_pen, cap);
  }
  __syncthreads();  // candidate lists complete

  int np = static_cast<int>(ctl[RCTL_NP]);
  int nr = static_cast<int>(ctl[RCTL_NR]);
  // More candidates than one warp sorts (long runs of ties): argmax rounds over the candidate
  // buffer, which holds every candidate unless it overflowed; then rounds over the whole chunk.
  // The sorted lists' regions serve as the rounds' scratch (the leader fills them only later).
  const bool ordered_r = n_row > 0 && nr > RES_SORT_MAX;
  const bool ordered_p = k_row > 0 && np > RES_SORT_MAX;
  if (n_row > 0 && nr > RES_SORT_MAX) {
    if (nr <= cap)
      nr = buffer_rounds(reinterpret_cast<uint32_t*>(cand_raw), 2, nr, n_row, reinterpret_cast<uint32_t*>(sorted_raw),
                         red64);
    else
      nr = res_exact_rounds<DT>(data, n_vec, n_el, lo, 1, n_row, penal, htab, P.hash_bits, hflag, sp.rep, sp.freq,
                                sp.pres, red64, cand_pen, cand_raw);
  }
  if (k_row > 0 && np > RES_SORT_MAX) {
    if (np <= cap)
      np = buffer_rounds(reinterpret_cast<uint32_t*>(cand_pen), 4, np, k_row, reinterpret_cast<uint32_t*>(sorted_pen),
                         red64);
    else if (MASK && masked)
      np = masked_rounds<DT>(data, lo, hi, aid[0], aid[1], aid[2], aid[3], P.allowed, a_beg + tid + APRE * NT, a_end,
                             k_row, penal, htab, P.hash_bits, sp.rep, sp.freq, sp.pres, red64, cand_pen);
    else
      np = res_exact_rounds<DT>(data, n_vec, n_el, lo, 0, k_row, penal, htab, P.hash_bits, hflag, sp.rep, sp.freq,
                                sp.pres, red64, cand_pen, cand_raw);
  }
  if (k_row == 0) np = 0;
  if (n_row == 0) nr = 0;

  // ---- send this CTA's best k_row / n_row, each with its rank, and its pairs to the leader ------
  // (threads 0..127: the penalised list, 128..255: the raw list; a rank is the number of larger keys
  // in the zero-padded list; after exact rounds the lists are already in order)
  const int sent_p = min(np, k_row), sent_r = min(nr, n_row);
  const uint32_t leader_bar = dsmem_addr(smem_u32(&mbar[RBAR_REC]), 0);
  {
    const int half = tid & (NT / 2 - 1);
    if (tid < NT / 2) {
      for (int i = half; i < np; i += NT / 2) {
        const uint4 ent = cand_pen[i];
        const uint64_t ki = (static_cast<uint64_t>(ent.y) << 32) | ent.x;
        const int rank = ordered_p ? i : rank_pad(reinterpret_cast<const uint32_t*>(cand_pen), 4, np, ki);
        if (rank < k_row) {
          uint64_t* key_p = recv_pkey + crank * P.kmax + rank;
          uint32_t* raw_p = recv_praw + crank * P.kmax + rank;
          if (crank == 0) {
            *key_p = ki;
            *raw_p = ent.z;
          } else {
            st_async_v2(dsmem_addr(smem_u32(key_p), 0), ent.x, ent.y, leader_bar);
            st_async_b32(dsmem_addr(smem_u32(raw_p), 0), ent.z, leader_bar);
          }
        }
      }
    } else {
      for (int i = half; i < nr; i += NT / 2) {
        const uint64_t ki = cand_raw[i];
        const int rank = ordered_r ? i : rank_pad(reinterpret_cast<const uint32_t*>(cand_raw), 2, nr, ki);
        if (rank < n_row) {
          uint64_t* slot_r = recv_raw + crank * P.nmax + rank;
          if (crank == 0) *slot_r = ki;
          else st_async_v2(dsmem_addr(smem_u32(slot_r), 0), static_cast<uint32_t>(ki), static_cast<uint32_t>(ki >> 32), leader_bar);
        }
      }
    }
  }
  if (tid == 0) {
    if (crank == 0) {
      recv_cnt[0] = make_uint2(static_cast<uint32_t>(sent_p), static_cast<uint32_t>(sent_r));
    } else {
      st_async_v2(dsmem_addr(smem_u32(recv_cnt + crank), 0), static_cast<uint32_t>(sent_p),
                  static_cast<uint32_t>(sent_r), leader_bar);
      mbar_arrive_expect_tx_remote(leader_bar, static_cast<uint32_t>(8 + 12 * sent_p + 8 * sent_r));
    }
  }

  if (crank == 0) {
    // ---- 4. the leader: every slice in, then the exact merge -----------------------------------
    // allowed-subset and chosen-id logits, fetched from global memory ahead of use
    float alog[APRE] = {};
    float chosen_x = 0.0f;
    {
      const char* rbase = static_cast<const char*>(P.logits) + static_cast<long long>(row) * P.ld * ESZ;
      auto glogit = [&](int id) -> float {
        if constexpr (DT == 0) {
          return reinterpret_cast<const float*>(rbase)[id];
        } else {
          return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(rbase)[id]) << 16);
        }
      };
#pragma unroll
      for (int t = 0; t < APRE; ++t) alog[t] = (aid[t] >= 0 && aid[t] < P.V) ? glogit(aid[t]) : 0.0f;
      if (tid == 0 && chosen_id >= 0 && chosen_id < P.V) chosen_x = glogit(chosen_id);
    }
    if (P.flags & STRATA_FLAG_TEST_STALL) test_stall(&mbar[RBAR_STALL], ctl, P.err);
    if (cs > 1) wait_bar(&mbar[RBAR_REC], ctl, P.err, true);
    __syncthreads();  // every slice and pair (the leader's own included) is in place
    // the log-normalisers: lanes 0..15 of the last warp combine the row's pairs, 16..31 the
    // allowed subset's
    if (wid == NW - 1) {
      const int c = lane & 15;
      float m = -INFINITY, s_ = 0.0f;
      if (c < cs) {
        const float2 t = reinterpret_cast<const float2*>(xrec + c * XW + Q)[lane >> 4];
        m = t.x;
        s_ = t.y;
      }
      float M = m;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, off));
      float sc = (m == -INFINITY || !(s_ > 0.0f)) ? 0.0f : s_ * ex2_approx((m - M) * LOG2E);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sc += __shfl_xor_sync(FULL_MASK, sc, off);
      if (c == 0)
        ctl[RCTL_LSE + (lane >> 4)] = __float_as_uint((M == -INFINITY || !(sc > 0.0f)) ? -INFINITY : M + logf(sc));
    }
    // merge (threads 0..127: the penalised list, 128..255: the raw list).  Slice c holds cnt_c keys
    // in descending order.  The k-th largest key of the grid of slice heads (the first ceil(k / cs)
    // entries of every slice) bounds the row's k-th largest from below, so only the entries at or
    // above it survive; their ranks by counting give the order.  The leader's candidate region
    // (free now) holds the grids (keys) and the survivors (key, payload).
    {
      const bool pl = tid < NT / 2;
      const int h = tid & (NT / 2 - 1);
      const int stride = pl ? P.kmax : P.nmax;
      const int kk = pl ? k_row : n_row;
      const uint64_t* keys = pl ? recv_pkey : recv_raw;
      // scratch in the leader's chunk region: the two grids (keys), then the penalised survivors
      // (key, payload) and the raw survivors (keys)
      uint64_t* grid = reinterpret_cast<uint64_t*>(data) + (pl ? 0 : RES_SORT_MAX);
      uint4* surv_p = reinterpret_cast<uint4*>(data + 2 * RES_SORT_MAX * 8);
      uint64_t* surv_r = reinterpret_cast<uint64_t*>(data + 2 * RES_SORT_MAX * 8 + RES_SORT_MAX * 16);
      int tot = 0, g = 0;
      const int h0 = kk > 0 ? (kk + cs - 1) / cs : 1;
      for (int c = 0; c < cs; ++c) {
        const int cnt = min(static_cast<int>(pl ? recv_cnt[c].x : recv_cnt[c].y), stride);
        tot += cnt;
        g += min(cnt, h0);
      }
      if (h == 0) ctl[pl ? RCTL_TOT_P : RCTL_TOT_R] = static_cast<uint32_t>(tot);
      const int gn = cs * h0;  // grid entries (<= k + cs - 1 < RES_SORT_MAX)
      {
        uint64_t key = 0ull;
        if (kk > 0 && h < gn) {
          const int c = h / h0, i = h - c * h0;
          if (i < min(static_cast<int>(pl ? recv_cnt[c].x : recv_cnt[c].y), stride)) key = keys[c * stride + i];
        }
        grid[h] = key;
        for (int i = h; i < RES_SORT_MAX; i += NT / 2) {
          if (pl) surv_p[i] = make_uint4(0u, 0u, 0u, 0u);
          else surv_r[i] = 0ull;
        }
      }
      __syncthreads();
      const bool bound = kk > 0 && tot > kk && g >= kk;  // else every entry survives
      if (bound && h < gn) {
        const uint64_t u = grid[h];
        const int above = rank_pad(reinterpret_cast<const uint32_t*>(grid), 2, gn, u);
        if (u != 0ull && above < kk)
          atomicMin(reinterpret_cast<unsigned long long*>(ctl + (pl ? RCTL_TLO : RCTL_TLO_R)), static_cast<unsigned long long>(u));
      }
      __syncthreads();
      const uint64_t tlo = bound ? *reinterpret_cast<const unsigned long long*>(ctl + (pl ? RCTL_TLO : RCTL_TLO_R)) : 0ull;
      if (kk > 0 && h < stride) {  // entry h of every slice: count the survivors, one atomic, write
        int cnt = 0;
        for (int c = 0; c < cs; ++c)
          cnt += (h < min(static_cast<int>(pl ? recv_cnt[c].x : recv_cnt[c].y), stride) && keys[c * stride + h] >= tlo) ? 1 : 0;
        int at = cnt > 0 ? static_cast<int>(atomicAdd(&ctl[pl ? RCTL_MP : RCTL_MR], static_cast<uint32_t>(cnt))) : 0;
        for (int c = 0; c < cs && cnt > 0; ++c) {
          if (h >= min(static_cast<int>(pl ? recv_cnt[c].x : recv_cnt[c].y), stride)) continue;
          const uint64_t key = keys[c * stride + h];
          if (key < tlo) continue;
          if (at < RES_SORT_MAX) {
            if (pl) surv_p[at] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32), recv_praw[c * stride + h], 0u);
            else surv_r[at] = key;
          }
          ++at;
          --cnt;
        }
      }
      __syncthreads();
      const int ns = static_cast<int>(ctl[pl ? RCTL_MP : RCTL_MR]);
      if (kk > 0 && ns <= RES_SORT_MAX) {
        for (int i = h; i < ns; i += NT / 2) {
          if (pl) {
            const uint4 ent = surv_p[i];
            const uint64_t ki = (static_cast<uint64_t>(ent.y) << 32) | ent.x;
            const int rank = rank_pad(reinterpret_cast<const uint32_t*>(surv_p), 4, ns, ki);
            if (rank < kk) sorted_pen[rank] = ent;
          } else {
            const uint64_t ki = surv_r[i];
            const int rank = rank_pad(reinterpret_cast<const uint32_t*>(surv_r), 2, ns, ki);
            if (rank < kk) sorted_raw[rank] = ki;
          }
        }
      }
    }
    __syncthreads();
    const int tot_p = static_cast<int>(ctl[RCTL_TOT_P]), tot_r = static_cast<int>(ctl[RCTL_TOT_R]);
    // more survivors than the ranks cover (long runs of ties in a few slices): exact rounds
    if (k_row > 0 && static_cast<int>(ctl[RCTL_MP]) > RES_SORT_MAX)
      leader_rounds(cs, P.kmax, k_row, recv_cnt, true, recv_pkey, recv_praw, reinterpret_cast<uint32_t*>(sorted_pen), 4,
                    red64);
    if (n_row > 0 && static_cast<int>(ctl[RCTL_MR]) > RES_SORT_MAX)
      leader_rounds(cs, P.nmax, n_row, recv_cnt, false, recv_raw, nullptr, reinterpret_cast<uint32_t*>(sorted_raw), 2,
                    red64);
    const int k_eff = min(k_row, tot_p);
    const int n_eff = min(n_row, tot_r);
    const float lse = __uint_as_float(ctl[RCTL_LSE]), lse_a = __uint_as_float(ctl[RCTL_LSE_A]);

    // ---- the tail's first half on <= 64 survivors (one warp): min_p and top_p cuts and the
    // tempered cumulative weights; nothing here depends on the draw counter
    int m1 = 0, m2 = 0;
    float Ca = 0.0f, Cb = 0.0f, wa = 0.0f, wb = 0.0f;
    uint4 ea = make_uint4(0, 0, 0, 0), eb = make_uint4(0, 0, 0, 0);
    float va = 0.0f, vb = 0.0f;
    if (P.mode == MODE_SAMPLE && wid == 0 && valid && k_eff > 0) {
      ea = (lane < k_eff) ? sorted_pen[lane] : make_uint4(0, 0, 0, 0);
      eb = (lane + 32 < k_eff) ? sorted_pen[lane + 32] : make_uint4(0, 0, 0, 0);
      va = key_value(ea.y);
      vb = key_value(eb.y);
      m1 = m2 = 1;
      if (sampled) {
        const float v0 = __shfl_sync(FULL_MASK, va, 0);
        m1 = k_eff;
        if (sp.min_p > 0.0f) {  // min_p in logit space, float32
          const float thr = __fadd_rn(v0, sp.logminp);
          const uint32_t ba = __ballot_sync(FULL_MASK, lane < k_eff && va >= thr);
          const uint32_t bb = __ballot_sync(FULL_MASK, lane + 32 < k_eff && vb >= thr);
          m1 = max(1, __popc(ba) + __popc(bb));
        }
        // temperature-1 mass (top_p) and tempered weights (draw) over the min_p survivors; fp32
        // prefix sums decide unless a decision lies within 1e-5 of its boundary, then double-word
        // sums decide
        const bool ina = lane < m1, inb = lane + 32 < m1;
        // lanes outside the survivors divide a plain zero (a NaN or an infinity would take the
        // division's slow path)
        const float da = ina ? __fsub_rn(va, v0) : 0.0f, db = inb ? __fsub_rn(vb, v0) : 0.0f;
        const float Tm = sp.temperature;
        const float qa = ina ? expf(da) : 0.0f, qb = inb ? expf(db) : 0.0f;
        wa = ina ? expf(__fdiv_rn(da, Tm)) : 0.0f;
        wb = inb ? expf(__fdiv_rn(db, Tm)) : 0.0f;
        const float ca = warp_scan_f(qa, lane);
        Ca = warp_scan_f(wa, lane);
        const float cb = warp_scan_f(qb, lane) + __shfl_sync(FULL_MASK, ca, 31);
        Cb = warp_scan_f(wb, lane) + __shfl_sync(FULL_MASK, Ca, 31);
        m2 = m1;
        if (!(sp.top_p >= 1.0f)) {
          if (!(sp.top_p > 0.0f)) {
            m2 = 1;
          } else {
            const float tot_q = __shfl_sync(FULL_MASK, cb, 31);
            const float target = sp.top_p * tot_q, margin = 1e-5f * tot_q;
            const bool near = __any_sync(FULL_MASK, (ina && fabsf(ca - target) <= margin) ||
                                                        (inb && fabsf(cb - target) <= margin));
            if (!near) {
              const uint32_t la = __ballot_sync(FULL_MASK, ina && ca < target);
              const uint32_t lb = __ballot_sync(FULL_MASK, inb && cb < target);
              m2 = min(m1, __popc(la) + __popc(lb) + 1);
            } else {
              m2 = top_p_dw(qa, qb, ina, inb, sp.top_p, m1, lane);
            }
          }
        }
      }
    }

    // ---- outputs: with early loads and shared outputs the previous call owns outputs and counters
    // until it ends, so the leader waits for it here and only then takes the counter
    if (early && !own_out) {
      grid_dep_wait();
      if (ctr_warp) r_slot = slot_rows(rs_pre[0], rs_pre[1], P.row_slot, P.B, slot, lane);
      if (ctr_thread) ctr_old = atomicAdd(&P.ctr[slot], r_slot == 1 ? (1ull << 16) : 1ull);
    }

    if (P.allowed_off != nullptr && P.allowed_lps != nullptr) {
      const char* rbase = static_cast<const char*>(P.logits) + static_cast<long long>(row) * P.ld * ESZ;
      auto out_allowed = [&](int j, int id, float x) {
        if (id >= 0 && id < P.V) {
          P.allowed_lps[j] = x - lse_a;
        } else {
          P.allowed_lps[j] = __int_as_float(0x7FC00000);
          atomicOr(P.err, STRATA_DEVERR_ALLOWED);
        }
      };
#pragma unroll
      for (int t = 0; t < APRE; ++t)
        if (a_beg + tid + t * NT < a_end) out_allowed(a_beg + tid + t * NT, aid[t], alog[t]);
      for (int j = a_beg + tid + APRE * NT; j < a_end; j += NT) {
        const int id = P.allowed[j];
        float x = 0.0f;
        if (id >= 0 && id < P.V) {
          if constexpr (DT == 0) x = reinterpret_cast<const float*>(rbase)[id];
          else x = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(rbase)[id]) << 16);
        }
        out_allowed(j, id, x);
      }
    }
    if (P.mode == MODE_LOGPROBS && P.chosen_lp != nullptr && P.chosen != nullptr && tid == 0) {
      if (chosen_id >= 0 && chosen_id < P.V) {
        P.chosen_lp[row] = chosen_x - lse;
      } else {
        P.chosen_lp[row] = __int_as_float(0x7FC00000);
        atomicOr(P.err, STRATA_DEVERR_CHOSEN);
      }
    }
    if (n_row > 0 && P.top_ids != nullptr && wid == 1) {
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
    // the tail's second half: Philox(seed, position) at the slot's counter, the pick, the outputs
    if (P.mode == MODE_SAMPLE && wid == 0) {
      int out = -1;
      float chosen_raw = __int_as_float(0x7FC00000);
      if (!valid) {
        if (lane == 0) atomicOr(P.err, STRATA_DEVERR_SLOT);
      } else if (k_eff == 0) {
        if (lane == 0) atomicOr(P.err, STRATA_DEVERR_NOCAND);
        // a sampled row without a candidate still counted itself among its slot's arrivals
        if (sampled && !ctr_at_entry) slot_arrival_done(r_slot, slot, P.ctr, ctr_old, lane);
      } else {
        int j = 0;
        if (sampled) {
          uint32_t x0 = 0u;
          if (ctr_thread) x0 = ctr_at_entry ? ctl[RCTL_X0] : philox_word0(sp.seed, pos, ctr_old >> 16);
          if (!ctr_at_entry) slot_arrival_done(r_slot, slot, P.ctr, ctr_old, lane);
          x0 = __shfl_sync(FULL_MASK, x0, 0);
          const float u = static_cast<float>(x0 >> 8) * 0x1p-24f;
          const int last = m2 - 1;  // the draw reads prefixes below m2 only; W = C[m2 - 1]
          const float W = (last < 32) ? __shfl_sync(FULL_MASK, Ca, last) : __shfl_sync(FULL_MASK, Cb, last - 32);
          const float tgt = u * W, margin = 1e-5f * W;
          const bool ia = lane < m2, ib = lane + 32 < m2;
          const bool near = __any_sync(FULL_MASK, (ia && fabsf(Ca - tgt) <= margin) || (ib && fabsf(Cb - tgt) <= margin));
          if (!near) {
            const uint32_t ja = __ballot_sync(FULL_MASK, ia && Ca <= tgt);
            const uint32_t jb = __ballot_sync(FULL_MASK, ib && Cb <= tgt);
            j = min(__popc(ja) + __popc(jb), m2 - 1);
          } else {
            j = draw_dw(wa, wb, m2, u, lane);
          }
        }
        const uint32_t id_a = key_id((static_cast<uint64_t>(ea.y) << 32) | ea.x);
        const uint32_t id_b = key_id((static_cast<uint64_t>(eb.y) << 32) | eb.x);
        out = static_cast<int>(__shfl_sync(FULL_MASK, j < 32 ? id_a : id_b, j & 31));
        chosen_raw = __uint_as_float(__shfl_sync(FULL_MASK, j < 32 ? ea.z : eb.z, j & 31));  // raw logit of the pick
      }
      if (lane == 0) {
        P.out_ids[row] = out;
        if (P.kept != nullptr) {
          P.kept[2 * row] = m1;
          P.kept[2 * row + 1] = m2;
        }
        if (P.chosen_lp != nullptr) P.chosen_lp[row] = (out >= 0) ? chosen_raw - lse : __int_as_float(0x7FC00000);
      }
      if ((P.row_draft != nullptr || P.ring != nullptr) && valid)
        slot_window_done(P.row_slot, P.out_ids, P.row_draft, P.done, P.slot_keep, P.ring, P.hlen, P.B, slot, lane);
      if (P.topk_ids != nullptr) {
        const long long o = static_cast<long long>(row) * KMAX;
        const bool ia = valid && lane < k_eff, ib = valid && lane + 32 < k_eff;
        P.topk_ids[o + lane] = ia ? static_cast<int32_t>(key_id((static_cast<uint64_t>(ea.y) << 32) | ea.x)) : -1;
        P.topk_ids[o + lane + 32] = ib ? static_cast<int32_t>(key_id((static_cast<uint64_t>(eb.y) << 32) | eb.x)) : -1;
        if (P.topk_vals != nullptr) {
          P.topk_vals[o + lane] = ia ? va : __int_as_float(0x7FC00000);
          P.topk_vals[o + lane + 32] = ib ? vb : __int_as_float(0x7FC00000);
        }
      }
    }
    if (P.mode == MODE_SAMPLE && valid && sp.k > P.kmax && tid == 0) atomicOr(P.err, STRATA_DEVERR_SHAPE);
  }

  if (ctl[RCTL_TIMEOUT] != 0u) {
    // a wait ran out: a copy, or another CTA's stores into this one, may still be on the way, so
    // wait for each once more (bounded) before the CTA leaves
    for (int p = 0; p < n_pieces; ++p) wait_bar(&mbar[p], ctl, P.err, false, 0u);
    if (cs > 1) {
      wait_bar(&mbar[RBAR_X0], ctl, P.err, true);
      if (crank == 0) wait_bar(&mbar[RBAR_REC], ctl, P.err, true);
    }
  }
}

}  // namespace strata
