// strata_kernel.cuh -- the fused row kernel: one HBM pass per logit row.
//
// Each logit row is split over a thread-block cluster of `cs` CTAs (one chunk per CTA; few large
// chunks for pipelined calls, more smaller ones when a single call's latency matters).  A CTA
//   1. streams its chunk through a ring of shared-memory slots (16 KiB bulk copies, one mbarrier
//      per slot; the last warp done with a slot refills it) and, as each piece lands, runs the
//      first pass: per thread the running maximum and the sum of exp against a lazily moved
//      reference (log-sum-exp of the raw logits); meanwhile the row's metadata loads are in
//      flight, and the logits of its allowed and history ids are fetched behind the first piece;
//      the history table of the chunk's id range (bitmap + open-addressing counts + raw logits)
//      and the allowed-subset partial sums follow the last piece;
//   2. publishes to every CTA of the cluster, with asynchronous DSMEM stores completed on one
//      mbarrier per CTA, the qw largest thread maxima of each warp (logits that carry no
//      penalty) and its two (max, sum) pairs (row and allowed subset).  Every CTA then takes
//      T = the K-th largest of the published values (K = max(top_k, top_n)): they are values of
//      distinct ids, so the row's K-th largest value (raw, and penalised, since those ids carry no
//      penalty) is at least T;
//   3. rescans (from L2: the chunk passed through it moments ago) only the threads whose maximum
//      reaches T, adds the penalised ids of the history table, keeps its best <= K candidates (the
//      candidate lists live in the ring, free by then) and stores them into its own slice of the
//      cluster leader's receive lists (asynchronous DSMEM stores, one transaction-counted arrival
//      per CTA);
//   4. the leader ranks the received keys by counting (one thread per key), then one warp runs the
//      tail of the chain on <= 64 survivors: min_p, top_p, temperature, the Philox draw.
// Only the leader writes outputs (the allowed-subset and chosen-id log-probabilities from logits
// it reads back from global memory), so with early loads no other CTA waits for the previous call.
// Every wait on another CTA or on a copy is an mbarrier poll with an iteration limit.
//
// The chain it computes is defined on the pages "#19 serve: per-request temperature/top_p/top_k/
// min_p/penalties sampling" (section "What changed") and "#3200 [Engine] OpenAI logprobs /
// top_logprobs / allowed_token_ids for the CUDA/HIP engine" (sections "Problem and result",
// "Approach").  The pages' own kernel ran k full-vocabulary argmax rounds per token; this one
// reads each row from HBM once and selects in a single pass plus a small exact merge.
#pragma once

#include <math.h>
#include <stdint.h>

#include "../../include/strata_sample.h"
#include "strata_device.cuh"

namespace strata {

constexpr int NT = 256;                      // threads per CTA (three CTAs fit an SM)
constexpr int NW = NT / 32;                  // warps per CTA
constexpr int VR = 4;                        // 16-byte vectors per thread per piece
constexpr int PIECE_VECS = NT * VR;
constexpr int PIECE_BYTES = PIECE_VECS * 16; // 16 KiB per bulk copy
constexpr int MAX_SLOTS = 8;                 // ring slots: pieces in flight per CTA
constexpr int MAX_CS = 16;                   // CTAs per row (non-portable cluster size)
constexpr int KMAX = STRATA_MAX_TOP_K;
constexpr int NMAX = STRATA_MAX_TOP_N;
constexpr int QW_MAX = 16;                   // thread maxima a warp publishes, at most
constexpr int RANK_LIMIT = 256;              // candidates ranked by counting; beyond: argmax rounds
constexpr int HASH_CNT_BITS = 13;            // history table entry = (local id << 13) | count
constexpr uint32_t HASH_EMPTY = 0xFFFFFFFFu;
constexpr int REC_PEN = 16;                  // a slice record: penalised entries after the header
constexpr int REC_RAW = REC_PEN + 16 * 64;   // and the raw keys after the penalised entries
constexpr int MODE_SAMPLE = 0;
constexpr int MODE_LOGPROBS = 1;
constexpr uint32_t SLOT_SAMPLED = 1u;
constexpr uint32_t SLOT_PENAL = 2u;
constexpr long long WAIT_CYCLES = 4000000000LL;  // bounded waits: ~2 s at GB300 clocks
constexpr float LAZY_SHIFT = 16.0f;          // the exp reference moves only when the max passes it by this
// A CTA's record: its NW * qw keys, then 2 (max, sum) pairs; records sit NW * qw + 4 words apart
// (a multiple of 16 bytes, since NW * qw is a multiple of 8).
__host__ __device__ inline int xrec_words(int qw) { return NW * qw + 4; }
constexpr int HPRE = 2;                      // history ids per thread fetched ahead of the table build
constexpr int APRE = 4;                      // allowed ids per thread fetched ahead
constexpr int BAR_X0 = MAX_SLOTS;            // mbarrier: every CTA's published record has landed
constexpr int BAR_X1 = MAX_SLOTS + 1;        // mbarrier (leader): every CTA's candidates have landed
constexpr int BAR_STALL = MAX_SLOTS + 2;     // mbarrier nothing arrives at (STRATA_FLAG_TEST_STALL)
constexpr int NBAR = MAX_SLOTS + 3;

// Control words in shared memory.
enum : int {
  CTL_CAND_PEN = 0,  // candidates appended to this CTA's penalised / raw lists
  CTL_CAND_RAW = 1,
  CTL_T = 2,         // the row threshold (atomicMin target, starts at all ones)
  CTL_TIMEOUT = 3,
  CTL_LSE = 4,       // log-sum-exp of the row / of the allowed subset (float bits)
  CTL_LSE_A = 5,
  CTL_TOT_P = 6,     // leader: received entries per list
  CTL_TOT_R = 7,
  CTL_SLOT0 = 8,     // per ring slot: warps done with the piece it holds (the last one refills it)
  CTL_LAST0 = CTL_SLOT0 + MAX_SLOTS,  // per ring slot: the last piece issued into it
  CTL_CTR = CTL_LAST0 + MAX_SLOTS,    // leader, own outputs: the counter word (2) and a use of the
  CTL_WORDS = CTL_CTR + 3             // advancing atomic's value (1)
};

// A slot's keys as the kernel reads them (prepared and validated by the host).
struct __align__(16) SlotDev {
  float temperature;  // > 0 for sampled slots
  float top_p;
  float min_p;
  float logminp;      // host logf(min_p) when min_p > 0
  float rep, freq, pres;
  int32_t k;          // survivors: top_k (0 -> 20) for sampled slots, 1 for greedy slots
  int32_t last_n;     // history window
  uint32_t flags;     // SLOT_SAMPLED | SLOT_PENAL
  uint64_t seed;
};
static_assert(sizeof(SlotDev) == 48, "SlotDev layout");

struct KParams {
  const void* logits;
  long long ld;
  int B, V, cs, chunk, mode;
  const int32_t* row_slot;
  const long long* row_pos;
  const int32_t* hist;
  const int32_t* hist_off;
  int n_hist_slots;
  int32_t* out_ids;
  int top_n;          // row stride of top_ids / top_lps
  int nmax;           // alternatives to compute (top_n if requested, else 0)
  int kmax;           // receive entries per CTA for the penalised list (>= every row's k)
  float* chosen_lp;
  int32_t* top_ids;
  float* top_lps;
  const int32_t* chosen;
  const int32_t* allowed;
  const int32_t* allowed_off;
  float* allowed_lps;
  int32_t* topk_ids;
  float* topk_vals;
  int32_t* kept;
  const SlotDev* slots;
  unsigned long long* ctr;  // per slot: (draw counter << 16) | arrivals of the current call
  int max_slots;
  uint32_t* err;
  int hash_cap, hash_bits;
  int nslot;          // ring slots (pieces in flight) per CTA, 2..MAX_SLOTS
  int qw;             // thread maxima each warp publishes: 1, 2, 4 or 8
  uint32_t flags;
  const int32_t* row_draft;  // verify windows: the draft after each row (-1: none), or NULL
  int32_t* slot_keep;        // verify windows: rows kept per slot
  uint32_t* done;            // verify windows / kept histories: per-slot rows done in the current call
  int32_t* ring;             // kept histories: STRATA_HISTORY_CAP ids per slot, or NULL
  unsigned long long* hlen;  // kept histories: per-slot total length
  int id_off;                // vocabulary slices: the whole-row id of column 0 (0 otherwise)
  unsigned char* rec;        // vocabulary slices: [B][STRATA_SHARD_RECORD_BYTES] records, or NULL
};

// A history id relative to the row's first column (a slice's id offset; ids below the slice wrap
// to values no chunk holds).
__device__ __forceinline__ int slice_id(int id, int off) {
  return static_cast<int>(static_cast<uint32_t>(id) - static_cast<uint32_t>(off));
}

struct Layout {
  uint32_t data, mbar, abits, mbits, hash, hraw, hflag, wkey, red, ctl, sps, xrec;
  uint32_t cand_pen, cand_raw, recv_cnt, recv_pkey, recv_praw, recv_raw, sorted_pen, sorted_raw, total;
  int cand_cap;  // entries of each candidate list (they live in the ring once the first pass is done)
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Shared-memory layout of one CTA; identical in every CTA of a launch.  `data` is the ring of
// `nslot` pieces; once the first pass is done it holds the candidate lists.
__host__ __device__ inline Layout make_layout(int chunk, int hash_cap, int cs, int kmax, int nmax, int nslot, int qw,
                                              bool allowed, bool mask) {
  Layout L;
  uint32_t o = 0;
  L.data = o;
  const uint32_t ring = static_cast<uint32_t>(nslot) * PIECE_BYTES;
  o += ring;
  L.cand_cap = static_cast<int>(ring / 24u) & ~7;
  L.cand_pen = L.data;
  L.cand_raw = L.data + static_cast<uint32_t>(L.cand_cap) * 16u;
  L.mbar = o;
  o = align_up(o + NBAR * 8, 16);
  const uint32_t bw = align_up((static_cast<uint32_t>(chunk) + 31) / 32 * 4, 16);
  // allowed ids met in this chunk (calls with allowed lists only): in the ring, which is free from
  // the end of the first pass until the candidate lists move in, whenever the ring can hold it
  L.abits = bw <= ring ? L.data : o;
  o += (allowed && bw > ring) ? bw : 0u;
  L.mbits = o;  // allowed ids already in a masked row's top_k list (mask launches only)
  o += mask ? bw : 0u;
  L.hash = o;
  o += align_up(static_cast<uint32_t>(hash_cap) * 4, 16);
  L.hraw = o;   // raw logit of each history table entry
  o += align_up(static_cast<uint32_t>(hash_cap) * 4, 16);
  L.hflag = o;
  o += NT / 8;
  L.wkey = o;
  o += NW * QW_MAX * 4;
  L.red = o;
  o += NW * 16;
  L.ctl = o;
  o += CTL_WORDS * 4;
  o = align_up(o, 16);
  L.sps = o;  // the row's slot keys: one copy for the block instead of registers in every thread
  o += static_cast<uint32_t>(sizeof(SlotDev));
  L.xrec = o;
  o += static_cast<uint32_t>(cs * xrec_words(qw)) * 4;
  L.recv_cnt = o;
  o += MAX_CS * 8;
  L.recv_pkey = o;  // received penalised list: keys (8 B) and raw logits (4 B), kmax per CTA
  o = align_up(o + static_cast<uint32_t>(cs * kmax) * 8, 16);
  L.recv_praw = o;
  o = align_up(o + static_cast<uint32_t>(cs * kmax) * 4, 16);
  L.recv_raw = o;
  o += static_cast<uint32_t>(cs * nmax) * 8;
  o = align_up(o, 16);
  L.sorted_pen = o;
  o += static_cast<uint32_t>(kmax) * 16;
  L.sorted_raw = o;
  o += static_cast<uint32_t>(nmax) * 8;
  L.total = align_up(o, 128);
  return L;
}

// Every region starts on a 16-byte boundary (vector and bulk accesses rely on it).
__host__ __device__ inline bool layout_aligned(const Layout& L) {
  const uint32_t r[] = {L.data, L.mbar, L.abits, L.mbits, L.hash, L.hraw, L.hflag, L.wkey, L.red, L.ctl, L.sps, L.xrec,
                        L.cand_pen, L.cand_raw, L.recv_cnt, L.recv_pkey, L.recv_praw, L.recv_raw, L.sorted_pen,
                        L.sorted_raw};
  for (uint32_t x : r)
    if (x % 16u != 0u) return false;
  return true;
}

// ------------------------------------------------------------------------------ helpers
template <int DT>
__device__ __forceinline__ void load_vec(const unsigned char* data, int v, float (&x)[16 / (DT == 0 ? 4 : 2)]) {
  if constexpr (DT == 0) {
    const float4 f = reinterpret_cast<const float4*>(data)[v];
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
  } else {
    const uint4 u = reinterpret_cast<const uint4*>(data)[v];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

template <int DT>
__device__ __forceinline__ float elem_at(const unsigned char* data, uint32_t loc) {
  if constexpr (DT == 0) {
    return reinterpret_cast<const float*>(data)[loc];
  } else {
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(data)[loc]) << 16);
  }
}

// Vector v of a chunk in global memory (the row is in L2 by the time anything reads it again);
// elements at or beyond n_el read as -inf, so the ragged last vector never reads past the row.
template <int DT>
__device__ __forceinline__ void load_vec_g(const unsigned char* g, int v, int n_el, float (&x)[16 / (DT == 0 ? 4 : 2)]) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  if ((v + 1) * EPV <= n_el) {
    if constexpr (DT == 0) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(g) + v);
      x[0] = f.x;
      x[1] = f.y;
      x[2] = f.z;
      x[3] = f.w;
    } else {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(g) + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const int idx = v * EPV + e;
      if (idx < n_el) {
        if constexpr (DT == 0) x[e] = __ldg(reinterpret_cast<const float*>(g) + idx);
        else x[e] = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(g) + idx)) << 16);
      } else {
        x[e] = -INFINITY;
      }
    }
  }
}

// Element e (< N) of a small register array, by a chain of selects (no local-memory indexing).
template <int N>
__device__ __forceinline__ float pick(const float (&x)[N], int e) {
  float r = x[0];
#pragma unroll
  for (int k = 1; k < N; ++k) r = (e == k) ? x[k] : r;
  return r;
}

__device__ __forceinline__ bool bit_at(const uint32_t* bits, uint32_t loc) {
  return (bits[loc >> 5] >> (loc & 31)) & 1u;
}

__device__ __forceinline__ uint32_t hash_slot(uint32_t loc, int bits) {
  return (loc * 0x9E3779B1u) >> (32 - bits);
}

// Count one occurrence of chunk-local id `loc`: returns the entry's index when this call created it,
// -1 when the id was already there, -2 when the table is full.
__device__ int hash_add(uint32_t* tab, int bits, uint32_t loc) {
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t h = hash_slot(loc, bits);
  for (uint32_t n = 0; n <= mask; ++n) {
    uint32_t cur = *reinterpret_cast<volatile uint32_t*>(&tab[h]);
    if (cur == HASH_EMPTY) {
      const uint32_t prev = atomicCAS(&tab[h], HASH_EMPTY, (loc << HASH_CNT_BITS) | 1u);
      if (prev == HASH_EMPTY) return static_cast<int>(h);
      cur = prev;
    }
    if ((cur >> HASH_CNT_BITS) == loc) {
      atomicAdd(&tab[h], 1u);
      return -1;
    }
    h = (h + 1u) & mask;
  }
  return -2;
}

__device__ uint32_t hash_count(const uint32_t* tab, int bits, uint32_t loc) {
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t h = hash_slot(loc, bits);
  for (uint32_t n = 0; n <= mask; ++n) {
    const uint32_t cur = tab[h];
    if (cur == HASH_EMPTY) return 0u;
    if ((cur >> HASH_CNT_BITS) == loc) return cur & ((1u << HASH_CNT_BITS) - 1u);
    h = (h + 1u) & mask;
  }
  return 0u;
}

// Bounded poll of an mbarrier phase (the one with the given parity).  On timeout the error word and a shared flag are
// set and the caller carries on with whatever has landed.
__device__ __forceinline__ void wait_bar(uint64_t* bar, uint32_t* ctl, uint32_t* err, bool cluster_scope,
                                         uint32_t parity = 0u) {
  if (cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return;
  const long long t0 = clock64();
  while (!(cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))) {
    if (clock64() - t0 > WAIT_CYCLES) {
      atomicOr(err, STRATA_DEVERR_TIMEOUT);
      ctl[CTL_TIMEOUT] = 1u;
      return;
    }
  }
}

// STRATA_FLAG_TEST_STALL: a bounded wait on an mbarrier nothing arrives at (it runs out).  Out of
// line, so that the common path carries none of it.
__device__ __noinline__ void test_stall(uint64_t* bar, uint32_t* ctl, uint32_t* err) { wait_bar(bar, ctl, err, false); }

__device__ __forceinline__ void online_add(MaxSum& a, float v) {
  if (v == -INFINITY || v != v) return;
  if (v > a.m) {
    a.s = (a.m == -INFINITY) ? 1.0f : a.s * ex2_approx((a.m - v) * LOG2E) + 1.0f;
    a.m = v;
  } else {
    a.s += ex2_approx((v - a.m) * LOG2E);
  }
}

template <int DT>
constexpr int BATCH_VECS = DT == 0 ? 4 : 2;  // 16 elements

// First pass over this thread's vectors of one piece, a batch of 16 elements at a time: the
// running max `mx`, the batch `bmx` that holds it, the second batch maximum `mx2` and its batch
// `bmx2`, the largest max `mx3` of the thread's other
// batches, and the sum of exp(x - ref) in two partial sums.  The reference `ref` moves to the piece's max only when that
// exceeds it by LAZY_SHIFT (or on the first finite piece), so the common piece costs one compare.
// `slot` holds piece p (vectors p * PIECE_VECS ...) for the vectors below n_full; the ragged last
// vector (n_full, when the chunk's bytes are not a multiple of 16) comes from global memory.
template <int DT>
__device__ __forceinline__ void pass1_piece(const unsigned char* slot, const unsigned char* gchunk, int p, int n_full,
                                            int n_vec, int n_el, float& ref, float& mx, float& mx2, float& mx3, int& bmx,
                                            int& bmx2, float& s0,
                                            float& s1) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  constexpr int RB = BATCH_VECS<DT>;  // vectors held at once: one batch of 16 elements
#pragma unroll
  for (int r0 = 0; r0 < VR; r0 += RB) {
    float x[RB][EPV];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int vl = static_cast<int>(threadIdx.x) + (r0 + r) * NT;
      const int v = p * PIECE_VECS + vl;
      if (v < n_full) {
        load_vec<DT>(slot, vl, x[r]);
      } else if (v < n_vec) {
        load_vec_g<DT>(gchunk, v, n_el, x[r]);
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
    if (pm > mx) {  // the two batches holding the thread's largest maxima, and the best of the rest
      mx3 = mx2;
      mx2 = mx;
      bmx2 = bmx;
      mx = pm;
      bmx = p * (VR / RB) + r0 / RB;
    } else if (pm > mx2) {
      mx3 = mx2;
      mx2 = pm;
      bmx2 = p * (VR / RB) + r0 / RB;
    } else {
      mx3 = fmaxf(mx3, pm);
    }
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

// Append one candidate that carries no penalty to both lists (two independent shared atomics).
__device__ __forceinline__ void append_both(uint32_t* ctl, uint4* cand_pen, uint64_t* cand_raw, int cap, uint64_t key,
                                            float raw, bool to_raw, bool to_pen) {
  const uint32_t ip = to_pen ? atomicAdd(&ctl[CTL_CAND_PEN], 1u) : 0u;
  const uint32_t ir = to_raw ? atomicAdd(&ctl[CTL_CAND_RAW], 1u) : 0u;
  if (to_pen && ip < static_cast<uint32_t>(cap))
    cand_pen[ip] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32), __float_as_uint(raw), 0u);
  if (to_raw && ir < static_cast<uint32_t>(cap)) cand_raw[ir] = key;
}

// Every element at or above T that carries no penalty, among the vectors of each thread named in
// `need` (one bit per lane of this warp; thread t owns vectors t, t + NT, ...): appended to both
// lists with its raw logit.  The warp scans one such thread's vectors at a time, each lane loading
// up to U of them at once, so a scan of a long chunk costs a round trip or two rather than one per
// vector.  `hist` marks the threads that own a history id (only their hits need the table lookup).
// Called by whole warps; a thread is named only when its maximum and its best other batch both reach T.
template <int DT>
__device__ __forceinline__ void warp_rescan(const unsigned char* g, uint32_t need, uint32_t hist, int wid, int lane,
                                         int n_vec, int n_el, int lo, float Tf, const uint32_t* htab, int hash_bits,
                                         uint32_t* ctl, uint4* cand_pen, uint64_t* cand_raw, int cap, bool to_raw,
                                         bool to_pen) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  constexpr int U = 32 / EPV;  // vectors in flight per lane (32 registers of elements)
#pragma unroll 1
  for (; need != 0u; need &= need - 1u) {
    const int src = __ffs(need) - 1;
    const int t = wid * 32 + src;
    const bool penal = (hist >> src) & 1u;
    const int nt = n_vec > t ? (n_vec - t + NT - 1) / NT : 0;  // vectors of thread t
#pragma unroll 1
    for (int j0 = 0; j0 < nt; j0 += 32 * U) {
      float x[U][EPV];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + lane + 32 * u;
        if (j < nt) {
          load_vec_g<DT>(g, t + j * NT, n_el, x[u]);
        } else {
#pragma unroll
          for (int e = 0; e < EPV; ++e) x[u][e] = -INFINITY;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        uint32_t hit = 0u;  // elements of this vector at or above T (NaN compares false)
#pragma unroll
        for (int e = 0; e < EPV; ++e) hit |= static_cast<uint32_t>(x[u][e] >= Tf) << e;
#pragma unroll 1
        for (; hit != 0u; hit &= hit - 1u) {
          const int e = __ffs(hit) - 1;
          const uint32_t loc = static_cast<uint32_t>((t + (j0 + lane + 32 * u) * NT) * EPV + e);
          if (loc >= static_cast<uint32_t>(n_el)) continue;
          const float xv = pick(x[u], e);
          const uint32_t o = order_key(xv);
          if (o == 0u || (penal && hash_count(htab, hash_bits, loc) != 0u)) continue;
          append_both(ctl, cand_pen, cand_raw, cap, sel_key(o, static_cast<uint32_t>(lo) + loc), xv, to_raw, to_pen);
        }
      }
    }
  }
}

// A masked row's top_k candidates: each of this thread's named ids inside the chunk, the first
// time any thread meets it (`mbits`), with its penalised value.  Out of line (mask launches only).
template <int DT>
__device__ __noinline__ void masked_candidates(const unsigned char* data, int lo, int hi, int a0, int a1, int a2,
                                               int a3, const int32_t* allowed, int j_first, int a_end,
                                               uint32_t* mbits, bool penal, const uint32_t* htab, int hash_bits,
                                               float rep, float freq, float pres, uint32_t* ctl, uint4* cand_pen,
                                               int cap) {
  auto add = [&](int id) {
    if (id < lo || id >= hi) return;
    const uint32_t loc = static_cast<uint32_t>(id - lo);
    const uint32_t bit = 1u << (loc & 31);
    if (atomicOr(&mbits[loc >> 5], bit) & bit) return;
    const float raw = elem_at<DT>(data, loc);
    const uint32_t c = penal ? hash_count(htab, hash_bits, loc) : 0u;
    const uint32_t op = order_key(c != 0u ? penalize(raw, c, rep, freq, pres) : raw);
    if (op == 0u) return;
    const uint32_t s = atomicAdd(&ctl[CTL_CAND_PEN], 1u);
    const uint64_t key = sel_key(op, static_cast<uint32_t>(id));
    if (s < static_cast<uint32_t>(cap))
      cand_pen[s] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32), __float_as_uint(raw), 0u);
  };
  add(a0);
  add(a1);
  add(a2);
  add(a3);
  for (int j = j_first; j < a_end; j += NT) add(allowed[j]);
}

// Block-wide max of a 64-bit key (all threads call; result in every thread).
__device__ __forceinline__ uint64_t block_max_u64(uint64_t x, uint64_t* red, int lane, int wid);

// A masked row's top_k list when its named ids overflow the candidate buffer: `need` argmax
// rounds over the named ids only (each thread's own ids, as in masked_candidates), in order, into
// the candidate buffer.  Every thread of the CTA calls it; returns the number found.
template <int DT>
__device__ __noinline__ int masked_rounds(const unsigned char* data, int lo, int hi, int a0, int a1, int a2, int a3,
                                          const int32_t* allowed, int j_first, int a_end, int need, bool penal,
                                          const uint32_t* htab, int hash_bits, float rep, float freq, float pres,
                                          uint64_t* red64, uint4* cand_pen) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  auto key_of = [&](int id) -> uint64_t {
    if (id < lo || id >= hi) return 0ull;
    const uint32_t loc = static_cast<uint32_t>(id - lo);
    const float raw = elem_at<DT>(data, loc);
    const uint32_t c = penal ? hash_count(htab, hash_bits, loc) : 0u;
    const uint32_t op = order_key(c != 0u ? penalize(raw, c, rep, freq, pres) : raw);
    return op == 0u ? 0ull : sel_key(op, static_cast<uint32_t>(id));
  };
  uint64_t prev = ~0ull;
  int got = 0;
  for (int r = 0; r < need; ++r) {
    uint64_t best = 0ull;
    auto consider = [&](int id) {
      const uint64_t k = key_of(id);
      if (k < prev && k > best) best = k;  // repeats of an id give the same key: taken once
    };
    consider(a0);
    consider(a1);
    consider(a2);
    consider(a3);
    for (int j = j_first; j < a_end; j += NT) consider(allowed[j]);
    best = block_max_u64(best, red64, lane, wid);
    if (best == 0ull) break;
    if (threadIdx.x == 0) {
      const float raw = elem_at<DT>(data, key_id(best) - static_cast<uint32_t>(lo));
      cand_pen[r] = make_uint4(static_cast<uint32_t>(best), static_cast<uint32_t>(best >> 32), __float_as_uint(raw), 0u);
    }
    prev = best;
    got = r + 1;
  }
  __syncthreads();
  return got;
}

// Block-wide max of a 64-bit key (all threads call; result in every thread).
__device__ __forceinline__ uint64_t block_max_u64(uint64_t x, uint64_t* red, int lane, int wid) {
  x = warp_max_u64(x);
  __syncthreads();
  if (lane == 0) red[wid] = x;
  __syncthreads();
  uint64_t r = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r = red[w] > r ? red[w] : r;
  return r;
}

// A threshold key for a thread that owns history ids: the largest order key of min(raw,
// penalised) over the batch of 16 elements that starts at vector `vb` (vectors vb, vb + NT, ...).
// Both the raw and the penalised value of that id reach it, so it bounds both candidate lists.
template <int DT>
__device__ __noinline__ uint32_t batch_safe_key(const unsigned char* gchunk, int vb, int n_vec, int n_el,
                                                const uint32_t* htab, int hash_bits, float rep, float freq,
                                                float pres) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  constexpr int RB = BATCH_VECS<DT>;
  uint32_t best = 0u;
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    const int v = vb + r * NT;
    if (v >= n_vec) continue;
    float x[EPV];
    load_vec_g<DT>(gchunk, v, n_el, x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const uint32_t loc = static_cast<uint32_t>(v * EPV + e);
      if (loc >= static_cast<uint32_t>(n_el)) continue;
      const uint32_t c = hash_count(htab, hash_bits, loc);
      const float y = c != 0u ? fminf(x[e], penalize(x[e], c, rep, freq, pres)) : x[e];
      best = max(best, order_key(y));
    }
  }
  return best;
}

// Published keys above `u` in records c = sub, sub + lpk, ... < cs of the record exchange (Q4 uint4
// of keys each, record stride 4 * Q4 + 4 words), counted in four independent sums.  The record
// length is a template constant, so the inner loop is fully unrolled: a runtime trip count there
// cost several times the loads it makes.
template <int Q4>
__device__ __forceinline__ int count_above_recs(const uint32_t* xrec, int sub, int lpk, int cs, uint32_t u) {
  int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll 1
  for (int c = sub; c < cs; c += lpk) {
    const uint4* rk = reinterpret_cast<const uint4*>(xrec + c * (4 * Q4 + 4));
#pragma unroll
    for (int j = 0; j < Q4; ++j) {
      const uint4 v = rk[j];
      a0 += v.x > u;
      a1 += v.y > u;
      a2 += v.z > u;
      a3 += v.w > u;
    }
  }
  return (a0 + a1) + (a2 + a3);
}

// Exact argmax rounds over this CTA's chunk: the `need` largest keys in order (penalised values
// for list 0, raw values for list 1), written to the candidate buffer.  Only taken when more
// candidates reach the row threshold than the buffer holds (heavy ties); kept out of line so the
// common path stays small.  A penalised value needs the history table only for the elements of
// threads that own a history id (`hflag`; thread t owns vectors t, t + NT, ...).  Every thread of
// the CTA calls it.  Returns the number found.
template <int DT>
__device__ __noinline__ int exact_rounds(const unsigned char* data, int n_vec, int n_el, int lo, int list, int need,
                                         bool penal, const uint32_t* htab, int hash_bits, const uint32_t* hflag,
                                         float rep, float freq, float pres, uint64_t* red64, uint4* cand_pen,
                                         uint64_t* cand_raw) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool owner = list == 0 && penal && ((hflag[tid >> 5] >> (tid & 31)) & 1u);
  uint64_t prev = ~0ull;
  int got = 0;
  for (int r = 0; r < need; ++r) {
    uint64_t best = 0ull;
    for (int v = tid; v < n_vec; v += NT) {
      float x[EPV];
      load_vec_g<DT>(data, v, n_el, x);
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
        if (key < prev && key > best) best = key;
      }
    }
    best = block_max_u64(best, red64, lane, wid);
    if (best == 0ull) break;
    if (tid == 0) {
      if (list == 0) {
        const float raw = elem_at<DT>(data, key_id(best) - static_cast<uint32_t>(lo));
        cand_pen[r] = make_uint4(static_cast<uint32_t>(best), static_cast<uint32_t>(best >> 32), __float_as_uint(raw), 0u);
      } else {
        cand_raw[r] = best;
      }
    }
    prev = best;
    got = r + 1;
  }
  __syncthreads();
  return got;
}

// The best `need` entries of a candidate list longer than RANK_LIMIT (heavy ties), in order, by
// argmax rounds over the list itself; they end up at the head of the list.  Entries are `words`
// 32-bit words with the 64-bit key first; keys are distinct.  `tmp` holds need * words words.
// Every thread of the CTA calls it; returns the number kept.
__device__ __noinline__ int buffer_rounds(uint32_t* list, int words, int n, int need, uint32_t* tmp, uint64_t* red64) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  uint64_t prev = ~0ull;
  int got = 0;
  for (int r = 0; r < need; ++r) {
    uint64_t best = 0ull;
    for (int i = tid; i < n; i += NT) {
      const uint2 o = *reinterpret_cast<const uint2*>(list + i * words);
      const uint64_t k = (static_cast<uint64_t>(o.y) << 32) | o.x;
      if (k < prev && k > best) best = k;
    }
    best = block_max_u64(best, red64, lane, wid);
    if (best == 0ull) break;
    for (int i = tid; i < n; i += NT) {
      const uint2 o = *reinterpret_cast<const uint2*>(list + i * words);
      if (((static_cast<uint64_t>(o.y) << 32) | o.x) == best)
        for (int w = 0; w < words; ++w) tmp[r * words + w] = list[i * words + w];
    }
    prev = best;
    got = r + 1;
  }
  __syncthreads();
  for (int i = tid; i < got * words; i += NT) list[i] = tmp[i];
  __syncthreads();
  return got;
}

// top_p survivors with double-word prefix sums (rare: the fp32 decision was within 1e-5 of its
// boundary).  Warp-wide: every lane of the warp calls it.
__device__ __noinline__ int top_p_dw(float qa, float qb, bool ina, bool inb, float top_p, int m1, int lane) {
  const DW a = warp_scan_dw(DW{qa, 0.0f}, lane);
  const DW b = dw_add(shfl_dw(a, 31), warp_scan_dw(DW{qb, 0.0f}, lane));
  const DW tg = dw_mul_f(shfl_dw(b, 31), top_p);
  const uint32_t la = __ballot_sync(FULL_MASK, ina && dw_less(a, tg));
  const uint32_t lb = __ballot_sync(FULL_MASK, inb && dw_less(b, tg));
  return min(m1, __popc(la) + __popc(lb) + 1);
}

// The draw's pick with double-word prefix sums (rare, as above).  Warp-wide.
__device__ __noinline__ int draw_dw(float wa, float wb, int m2, float u, int lane) {
  const DW a = warp_scan_dw(DW{wa, 0.0f}, lane);
  const DW b = dw_add(shfl_dw(a, 31), warp_scan_dw(DW{wb, 0.0f}, lane));
  const int last = m2 - 1;
  const DW Wd = (last < 32) ? shfl_dw(a, last) : shfl_dw(b, last - 32);
  const DW td = dw_mul_f(Wd, u);
  const uint32_t ja = __ballot_sync(FULL_MASK, lane < m2 && !dw_less(td, a));
  const uint32_t jb = __ballot_sync(FULL_MASK, lane + 32 < m2 && !dw_less(td, b));
  return min(__popc(ja) + __popc(jb), m2 - 1);
}

// The tail of a row on its ordered top_k list (one warp; lane i holds entries i and i + 32).
struct Tail {
  uint4 ea, eb;      // the entries: key low word, key high word, raw logit, 0
  float va, vb;      // their penalised logits
  float wa, wb;      // tempered weights over the top_p survivors
  float Ca, Cb;      // and their fp32 prefix sums
  int m1, m2;        // survivors of min_p, of top_p
};

// The tail's first half on k_eff > 0 ordered entries: min_p and top_p cuts and the tempered
// cumulative weights (nothing here depends on the draw counter).  A greedy row keeps its head.
__device__ __forceinline__ void tail_cuts(const uint4* sorted_pen, int k_eff, bool sampled, const SlotDev& sp,
                                          int lane, Tail& t) {
  t.ea = (lane < k_eff) ? sorted_pen[lane] : make_uint4(0, 0, 0, 0);
  t.eb = (lane + 32 < k_eff) ? sorted_pen[lane + 32] : make_uint4(0, 0, 0, 0);
  t.va = key_value(t.ea.y);
  t.vb = key_value(t.eb.y);
  t.m1 = t.m2 = 1;
  if (!sampled) return;
  const float v0 = __shfl_sync(FULL_MASK, t.va, 0);
  t.m1 = k_eff;
  if (sp.min_p > 0.0f) {  // min_p in logit space, float32
    const float thr = __fadd_rn(v0, sp.logminp);
    const uint32_t ba = __ballot_sync(FULL_MASK, lane < k_eff && t.va >= thr);
    const uint32_t bb = __ballot_sync(FULL_MASK, lane + 32 < k_eff && t.vb >= thr);
    t.m1 = max(1, __popc(ba) + __popc(bb));
  }
  // temperature-1 mass (top_p) and tempered weights (draw) over the min_p survivors.  Prefix sums
  // in fp32 decide unless a decision lies within 1e-5 of its boundary (the fp32 scan is good to
  // ~4e-7 relative); then double-word sums (TwoSum) decide.
  const bool ina = lane < t.m1, inb = lane + 32 < t.m1;
  // lanes outside the survivors divide a plain zero (a NaN or an infinity would take the
  // division's slow path)
  const float da = ina ? __fsub_rn(t.va, v0) : 0.0f, db = inb ? __fsub_rn(t.vb, v0) : 0.0f;
  const float Tm = sp.temperature;
  const float qa = ina ? expf(da) : 0.0f, qb = inb ? expf(db) : 0.0f;
  t.wa = ina ? expf(__fdiv_rn(da, Tm)) : 0.0f;
  t.wb = inb ? expf(__fdiv_rn(db, Tm)) : 0.0f;
  const float ca = warp_scan_f(qa, lane);
  t.Ca = warp_scan_f(t.wa, lane);
  const float cb = warp_scan_f(qb, lane) + __shfl_sync(FULL_MASK, ca, 31);
  t.Cb = warp_scan_f(t.wb, lane) + __shfl_sync(FULL_MASK, t.Ca, 31);
  t.m2 = t.m1;
  if (!(sp.top_p >= 1.0f)) {
    if (!(sp.top_p > 0.0f)) {
      t.m2 = 1;
    } else {
      const float tot_q = __shfl_sync(FULL_MASK, cb, 31);
      const float target = sp.top_p * tot_q, margin = 1e-5f * tot_q;
      const bool near = __any_sync(FULL_MASK, (ina && fabsf(ca - target) <= margin) ||
                                                  (inb && fabsf(cb - target) <= margin));
      if (!near) {
        const uint32_t la = __ballot_sync(FULL_MASK, ina && ca < target);
        const uint32_t lb = __ballot_sync(FULL_MASK, inb && cb < target);
        t.m2 = min(t.m1, __popc(la) + __popc(lb) + 1);
      } else {
        t.m2 = top_p_dw(qa, qb, ina, inb, sp.top_p, t.m1, lane);
      }
    }
  }
}

// The draw: the index of the first survivor whose cumulative tempered weight exceeds u * W (W the
// sum over the m2 top_p survivors), from the fp32 sums unless a prefix lies within 1e-5 of u * W.
__device__ __forceinline__ int tail_draw(const Tail& t, uint32_t x0, int lane) {
  const float u = static_cast<float>(x0 >> 8) * 0x1p-24f;
  const int last = t.m2 - 1;  // the draw reads prefixes below m2 only; W = C[m2 - 1]
  const float W = (last < 32) ? __shfl_sync(FULL_MASK, t.Ca, last) : __shfl_sync(FULL_MASK, t.Cb, last - 32);
  const float tgt = u * W, margin = 1e-5f * W;
  const bool ia = lane < t.m2, ib = lane + 32 < t.m2;
  const bool near = __any_sync(FULL_MASK, (ia && fabsf(t.Ca - tgt) <= margin) || (ib && fabsf(t.Cb - tgt) <= margin));
  if (!near) {
    const uint32_t ja = __ballot_sync(FULL_MASK, ia && t.Ca <= tgt);
    const uint32_t jb = __ballot_sync(FULL_MASK, ib && t.Cb <= tgt);
    return min(__popc(ja) + __popc(jb), t.m2 - 1);
  }
  return draw_dw(t.wa, t.wb, t.m2, u, lane);
}

// Entry j of the tail's list (warp-wide): id and raw logit.
__device__ __forceinline__ uint32_t tail_id(const Tail& t, int j) {
  const uint32_t id_a = key_id((static_cast<uint64_t>(t.ea.y) << 32) | t.ea.x);
  const uint32_t id_b = key_id((static_cast<uint64_t>(t.eb.y) << 32) | t.eb.x);
  return __shfl_sync(FULL_MASK, j < 32 ? id_a : id_b, j & 31);
}
__device__ __forceinline__ float tail_raw(const Tail& t, int j) {
  return __uint_as_float(__shfl_sync(FULL_MASK, j < 32 ? t.ea.z : t.eb.z, j & 31));
}

// A vocabulary slice's record of one row (the layout strata_shard_rows documents): the counts and
// the log-sum-exp, then the ordered penalised entries (key, raw logit) and raw keys, their ids
// moved from the slice's columns to whole-row ids (a key's low word is the complement of the id,
// so the id offset is subtracted from it).  Threads 0..63 and 64..83 of the leader write it.
__device__ __forceinline__ void write_record(unsigned char* rec, const uint4* sorted_pen, int n_pen,
                                             const uint64_t* sorted_raw, int n_raw, float lse, int id_off, int tid) {
  static_assert(STRATA_SHARD_RECORD_BYTES >= REC_RAW + STRATA_MAX_TOP_N * 8, "record layout");
  const uint32_t off = static_cast<uint32_t>(id_off);
  if (tid == 0)
    *reinterpret_cast<uint4*>(rec) = make_uint4(static_cast<uint32_t>(n_pen), static_cast<uint32_t>(n_raw),
                                                __float_as_uint(lse), 0u);
  if (tid < n_pen) {
    const uint4 e = sorted_pen[tid];
    *reinterpret_cast<uint4*>(rec + REC_PEN + 16 * tid) = make_uint4(e.x - off, e.y, e.z, 0u);
  } else if (tid >= KMAX && tid - KMAX < n_raw) {
    const uint64_t k = sorted_raw[tid - KMAX];
    *reinterpret_cast<uint2*>(rec + REC_RAW + 8 * (tid - KMAX)) =
        make_uint2(static_cast<uint32_t>(k) - off, static_cast<uint32_t>(k >> 32));
  }
}

// Entries CTA c stored in list `w` (0: penalised, 1: raw) of the leader, clamped to its slice.
__device__ __forceinline__ int recv_count(const uint2* recv_cnt, int c, int w, int stride) {
  const uint2 n = recv_cnt[c];
  return min(static_cast<int>(w == 0 ? n.x : n.y), stride);
}

// Rank of `key` among the received entries of one list (slices of `stride` entries per CTA;
// entry size `esz_words` 32-bit words, key in words 0-1): the number of larger keys.  Keys are
// distinct (the id is part of the key).
__device__ __forceinline__ int count_greater(const uint32_t* recv, int esz_words, int stride, const uint2* recv_cnt,
                                             int w, int cs, uint64_t key) {
  int rank = 0;
  for (int c = 0; c < cs; ++c) {
    const uint32_t* e = recv + static_cast<size_t>(c) * stride * esz_words;
    const int n = recv_count(recv_cnt, c, w, stride);
#pragma unroll 4
    for (int j = 0; j < n; ++j) {
      const uint2 o = *reinterpret_cast<const uint2*>(e + j * esz_words);
      rank += ((static_cast<uint64_t>(o.y) << 32) | o.x) > key;
    }
  }
  return rank;
}

// Rank of `key` in a dense list (entry size `esz_words` 32-bit words, key in words 0-1) padded
// with zero keys to `n8` entries, a multiple of 8: the number of larger keys, counted in four
// independent partial sums (every thread of a warp reads the same entry, a broadcast).
__device__ __forceinline__ int rank_desc(const uint32_t* list, int esz_words, int n8, uint64_t key) {
  int r[4] = {0, 0, 0, 0};
#pragma unroll 1
  for (int j = 0; j < n8; j += 8) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint2 o = *reinterpret_cast<const uint2*>(list + (j + t) * esz_words);
      r[t & 3] += ((static_cast<uint64_t>(o.y) << 32) | o.x) > key;
    }
  }
  return (r[0] + r[1]) + (r[2] + r[3]);
}

// Sort 8 keys in descending order in registers (Batcher's odd-even merge network, 19 exchanges).
__device__ __forceinline__ void sort8_desc(uint32_t (&v)[8]) {
  auto cx = [&](int i, int j) {
    const uint32_t a = v[i], b = v[j];
    v[i] = max(a, b);
    v[j] = min(a, b);
  };
  cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
  cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
  cx(1, 2); cx(5, 6);
  cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
  cx(2, 4); cx(3, 5);
  cx(1, 2); cx(3, 4); cx(5, 6);
}

// Rows of the call whose slot is `slot` (warp-wide; the first 64 row slots were fetched ahead into
// rs0/rs1).
__device__ __forceinline__ int slot_rows(int rs0, int rs1, const int32_t* row_slot, int B, int slot, int lane) {
  int r_s = __popc(__ballot_sync(FULL_MASK, rs0 == slot)) + __popc(__ballot_sync(FULL_MASK, rs1 == slot));
  for (int b0 = 64; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    r_s += __popc(__ballot_sync(FULL_MASK, b < B && row_slot[b] == slot));
  }
  return r_s;
}

// The end of a sampled row's arrival on its slot's packed counter word (lane 0 holds the value its
// atomic returned).  A slot with one row in the call advanced its counter in that same atomic; with
// r_s > 1 rows, each added one arrival, and the row that completes them advances the counter by one
// and clears them.
__device__ __forceinline__ void slot_arrival_done(int r_s, int slot, unsigned long long* ctr,
                                                  unsigned long long ctr_old, int lane) {
  if (r_s > 1 && lane == 0 && (ctr_old & 0xFFFFull) + 1ull == static_cast<unsigned long long>(r_s))
    atomicAdd(&ctr[slot], (1ull << 16) - static_cast<unsigned long long>(r_s));
}

// A call with own outputs takes its slot's counter at its start (warp-wide, the leader's warp 0 of a
// sampled row), the same way the draw takes it otherwise: one atomic for a slot with one row in
// the call; with several, one arrival each and the row completing them advances the counter.  The
// value waits in shared memory until the draw (no register held through the first pass); the
// stores need both atomics' returned values, so both have been performed when they are done.
// Out of line: plain calls never take it.
__device__ __noinline__ void take_counter_early(int rs0, int rs1, const int32_t* row_slot, int B, int slot,
                                                unsigned long long* ctr, uint32_t* ctl, int lane) {
  const int rs = slot_rows(rs0, rs1, row_slot, B, slot, lane);
  if (lane == 0) {
    const unsigned long long v = atomicAdd(&ctr[slot], rs == 1 ? (1ull << 16) : 1ull);
    uint32_t adv = 0u;
    if (rs > 1 && (v & 0xFFFFull) + 1ull == static_cast<unsigned long long>(rs))
      adv = static_cast<uint32_t>(atomicAdd(&ctr[slot], (1ull << 16) - static_cast<unsigned long long>(rs)));
    ctl[CTL_CTR] = static_cast<uint32_t>(v);
    ctl[CTL_CTR + 1] = static_cast<uint32_t>(v >> 32);
    ctl[CTL_CTR + 2] = adv;
  }
}

// The end of a slot's rows in a verify call or a call that keeps histories, run by the leader warp
// of every row of the slot once lane 0 has stored the row's pick.  The row publishes its pick and
// counts itself done in the slot's arrival word; the last row of the slot to finish reads every
// pick of the call (rows of the slot in row order), keeps 1 + the leading rows whose pick equals
// their draft (verify; a plain call keeps every row), appends the kept picks other than -1 to the
// slot's history ring and length (when kept), and clears the word for the next call.  Every row
// of the slot read its window before its candidates reached its leader, so no reader is left when
// the ring is written.  Warp-wide; out of line (plain calls without histories never take it).
__device__ __noinline__ void slot_window_done(const int32_t* row_slot, const int32_t* out_ids, const int32_t* row_draft,
                                              uint32_t* done, int32_t* slot_keep, int32_t* ring,
                                              unsigned long long* hlen, int B, int slot, int lane) {
  int r_s = 0;  // rows of this slot in the call
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    r_s += __popc(__ballot_sync(FULL_MASK, b < B && row_slot[b] == slot));
  }
  uint32_t last = 0u;
  if (lane == 0) {
    __threadfence();  // this row's pick is visible before it counts as done
    last = (atomicAdd(&done[slot], 1u) + 1u == static_cast<uint32_t>(r_s)) ? 1u : 0u;
  }
  if (__shfl_sync(FULL_MASK, last, 0) == 0u) return;
  __threadfence();  // every other row of the slot was done (and its pick visible) before this one
  int keep = r_s;
  if (row_draft != nullptr) {
    keep = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      const bool in = b < B && row_slot[b] == slot;
      const int t = in ? __ldcg(out_ids + b) : -1;
      const int d = in ? row_draft[b] : -1;
      const uint32_t m_in = __ballot_sync(FULL_MASK, in);
      const uint32_t m_stop = __ballot_sync(FULL_MASK, in && (d < 0 || t < 0 || t != d));
      if (m_stop != 0u) {  // the window ends at the first row whose pick differs from its draft
        keep += __popc(m_in & ((2u << (__ffs(m_stop) - 1)) - 1u));
        break;
      }
      keep += __popc(m_in);
    }
  }
  if (ring != nullptr) {
    const unsigned long long len = hlen[slot];
    int32_t* rs = ring + static_cast<size_t>(slot) * STRATA_HISTORY_CAP;
    const uint32_t lt = (1u << lane) - 1u;
    int seen = 0, app = 0;  // rows of the slot so far, picks appended so far
    for (int b0 = 0; b0 < B && seen < keep; b0 += 32) {
      const int b = b0 + lane;
      const bool in = b < B && row_slot[b] == slot;
      const int t = in ? __ldcg(out_ids + b) : -1;
      const uint32_t m_in = __ballot_sync(FULL_MASK, in);
      const bool kept = in && seen + __popc(m_in & lt) < keep;
      const uint32_t m_app = __ballot_sync(FULL_MASK, kept && t >= 0);
      if (kept && t >= 0) {
        const unsigned long long at = len + static_cast<unsigned long long>(app + __popc(m_app & lt));
        rs[at & static_cast<unsigned long long>(STRATA_HISTORY_CAP - 1)] = t;
      }
      seen += __popc(m_in);
      app += __popc(m_app);
    }
    if (lane == 0) hlen[slot] = len + static_cast<unsigned long long>(app);
  }
  if (lane == 0) {
    if (slot_keep != nullptr) slot_keep[slot] = keep;
    done[slot] = 0u;
  }
}

// ------------------------------------------------------------------------------ the kernel
// DT: 0 fp32 rows, 1 bf16 rows.  MASK: allowed ids restrict the sampling (STRATA_FLAG_ALLOWED_MASK);
// OWN: a call with own outputs and early loads (STRATA_FLAG_OWN_OUTPUTS).  Separate instantiations
// so that plain launches carry none of their state or code.  MINB: blocks per SM the registers
// are budgeted for: 3 (80 registers, some spilled to local memory) where calls of independent
// groups stream at once, 2 (no spills) for one stream of calls, whose blocks each walk the whole
// serial chain.
template <int DT, bool MASK, bool OWN = false, int MINB = 3>
__global__ void __launch_bounds__(NT, MINB) rows_kernel(const KParams P) {
  extern __shared__ __align__(128) unsigned char sm[];
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int EPV = 16 / ESZ;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool early = (P.flags & STRATA_FLAG_EARLY_LOAD) != 0u;
  // own outputs (early loads only): nothing of this call waits for the previous call; the draw
  // counters are taken before the next call may launch, which keeps them in call order
  const bool own_out = OWN && early;
  if (!early) grid_dep_wait();  // inputs may be the previous kernel's outputs
  // the next call may start its own loads now: launching it is what bounds a stream of calls
  // whose CTAs each take microseconds to reach their first copy (its outputs still wait for ours)
  if (!own_out) grid_dep_launch();

  const uint32_t crank = cluster_ctarank();
  const int cs = P.cs;
  const int row = blockIdx.x / cs;
  const bool mask_launch = MASK && P.mode == MODE_SAMPLE && P.allowed_off != nullptr;
  const Layout L = make_layout(P.chunk, P.hash_cap, cs, P.kmax, P.nmax, P.nslot, P.qw, P.allowed_off != nullptr,
                               mask_launch);
  const int lo = static_cast<int>(crank) * P.chunk;
  const int hi = min(P.V, lo + P.chunk);
  const int n_el = max(0, hi - lo);
  const int bytes = n_el * ESZ;
  const int bytes_al = bytes & ~15;
  const int n_vec = (bytes + 15) >> 4;
  const int n_full = bytes_al >> 4;  // vectors the bulk copies bring; a ragged last one is read directly
  const int n_pieces = (bytes_al + PIECE_BYTES - 1) / PIECE_BYTES;
  const int nslot = P.nslot;
  const int cap = L.cand_cap;
  const int Q = NW * P.qw;                                  // keys this CTA publishes
  const int XW = Q + 4;                                     // record stride in words
  const uint32_t rec_bytes = static_cast<uint32_t>(Q + 4) * 4u;

  unsigned char* data = sm + L.data;  // the ring of pieces in flight
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + L.mbar);
  const char* grow = static_cast<const char*>(P.logits) + (static_cast<long long>(row) * P.ld + lo) * ESZ;
  const unsigned char* gchunk = reinterpret_cast<const unsigned char*>(grow);

  // row metadata, first level: independent loads.  Thread 0 issues its own after the copies and
  // the barrier fence (a release fence behind outstanding loads would wait for them); every other
  // thread issues them first, so the three-level metadata chain starts at once.
  int slot = -1;
  unsigned long long pos = 0ull;
  int chosen_id = -1;
  int a_beg = 0, a_end = 0;
  auto load_meta1 = [&]() {
    if (P.mode == MODE_SAMPLE) {
      slot = P.row_slot[row];
      if (P.row_pos != nullptr) pos = static_cast<unsigned long long>(P.row_pos[row]);  // none for a slice
    } else if (P.chosen != nullptr) {
      chosen_id = P.chosen[row];
    }
    if (P.allowed_off != nullptr) {
      a_beg = P.allowed_off[row];
      a_end = P.allowed_off[row + 1];
    }
  };
  if (tid != 0) load_meta1();

  // ---- 1. barriers and the bulk copies of this chunk ----------------------------------------
  if (tid == 0) {  // the first pieces go out first; the exchange barriers are set up behind them
    const int n0 = min(nslot, n_pieces);
    for (int p = 0; p < n0; ++p) mbar_init(&mbar[p], 1);
    fence_proxy_async_smem();
    for (int p = 0; p < n0; ++p) {
      const uint32_t nb = static_cast<uint32_t>(min(PIECE_BYTES, bytes_al - p * PIECE_BYTES));
      mbar_arrive_expect_tx(&mbar[p], nb);
      bulk_g2s(data + p * PIECE_BYTES, grow + p * PIECE_BYTES, nb, &mbar[p]);
    }
    mbar_init(&mbar[BAR_X0], 2);                   // the announced bytes + this CTA's own record
    mbar_init(&mbar[BAR_X1], cs > 1 ? cs - 1 : 1); // one arrival per other CTA (leader only)
    mbar_init(&mbar[BAR_STALL], 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&mbar[BAR_X0], static_cast<uint32_t>(cs - 1) * rec_bytes);
  }
  if (tid == 0) load_meta1();



  uint32_t* abits = reinterpret_cast<uint32_t*>(sm + L.abits);
  uint32_t* mbits = reinterpret_cast<uint32_t*>(sm + L.mbits);
  uint32_t* htab = reinterpret_cast<uint32_t*>(sm + L.hash);
  uint32_t* hraw = reinterpret_cast<uint32_t*>(sm + L.hraw);
  uint32_t* hflag = reinterpret_cast<uint32_t*>(sm + L.hflag);
  uint32_t* wkey = reinterpret_cast<uint32_t*>(sm + L.wkey);
  uint64_t* red64 = reinterpret_cast<uint64_t*>(sm + L.red);
  float4* red4 = reinterpret_cast<float4*>(sm + L.red);
  uint32_t* ctl = reinterpret_cast<uint32_t*>(sm + L.ctl);
  uint32_t* xrec = reinterpret_cast<uint32_t*>(sm + L.xrec);
  uint4* cand_pen = reinterpret_cast<uint4*>(sm + L.cand_pen);
  uint64_t* cand_raw = reinterpret_cast<uint64_t*>(sm + L.cand_raw);
  uint2* recv_cnt = reinterpret_cast<uint2*>(sm + L.recv_cnt);
  uint64_t* recv_pkey = reinterpret_cast<uint64_t*>(sm + L.recv_pkey);
  uint32_t* recv_praw = reinterpret_cast<uint32_t*>(sm + L.recv_praw);
  uint64_t* recv_raw = reinterpret_cast<uint64_t*>(sm + L.recv_raw);
  uint4* sorted_pen = reinterpret_cast<uint4*>(sm + L.sorted_pen);
  uint64_t* sorted_raw = reinterpret_cast<uint64_t*>(sm + L.sorted_raw);

  const int bw_words = (P.chunk + 31) >> 5;
  const bool abits_in_ring = L.abits == L.data;  // then zeroed once the first pass is done
  if (P.allowed_off != nullptr && (mask_launch || !abits_in_ring))
    for (int i = tid; i < bw_words; i += NT) {
      if (!abits_in_ring) abits[i] = 0u;
      if (mask_launch) mbits[i] = 0u;
    }
  for (int i = tid; i < P.hash_cap; i += NT) htab[i] = HASH_EMPTY;
  if (tid < NT / 32) hflag[tid] = 0u;
  if (tid < CTL_WORDS)
    ctl[tid] = (tid == CTL_T) ? 0xFFFFFFFFu
                              : (tid >= CTL_LAST0 && tid < CTL_CTR ? static_cast<uint32_t>(tid - CTL_LAST0) : 0u);
  __syncthreads();           // tables zeroed, barriers initialised
  cluster_arrive_relaxed();  // this CTA is running (remote stores wait for every CTA, below)

  // ---- row metadata, second level ------------------------------------------------------------
  // the slot's keys: the three the set-up needs in registers, the rest read from the block's one
  // copy in shared memory (written by thread 0, read after the next barrier)
  bool valid = true;
  uint32_t sp_flags = 0u;
  int sp_k = 0, sp_last_n = 0;
  SlotDev* const sps = reinterpret_cast<SlotDev*>(sm + L.sps);
  if (P.mode == MODE_SAMPLE) {
    valid = static_cast<unsigned>(slot) < static_cast<unsigned>(P.max_slots);
    if (valid) {
      const SlotDev* g = P.slots + slot;
      sp_flags = g->flags;
      sp_k = g->k;
      sp_last_n = g->last_n;
      if (tid == 0) *sps = *g;
    } else if (tid == 0) {
      *sps = SlotDev{};
    }
  }
  const SlotDev& sp = *sps;
  const bool sampled = valid && (sp_flags & SLOT_SAMPLED);
  const int k_row = (P.mode == MODE_SAMPLE && valid) ? min(max(sp_k, 1), P.kmax) : 0;
  const int n_row = P.nmax;
  const int kp = max(k_row, n_row);
  const bool kept_hist = P.ring != nullptr;
  const bool penal = (P.mode == MODE_SAMPLE) && valid && (sp_flags & SLOT_PENAL) && P.hash_cap > 0 &&
                     (kept_hist || (P.hist_off != nullptr && slot < P.n_hist_slots));
  // the window: ids hb[(h_start + i) & h_mask] for i < h_len (a caller's CSR row, or the slot's ring)
  int h_len = 0;
  uint32_t h_start = 0u, h_mask = 0xFFFFFFFFu;
  const int32_t* hb = P.hist;
  if (penal) {
    if (kept_hist) {
      // the previous call appends to the ring, so its window is read after the first pass (below)
      hb = P.ring + static_cast<size_t>(slot) * STRATA_HISTORY_CAP;
      h_mask = STRATA_HISTORY_CAP - 1;
    } else {
      const int hs = P.hist_off[slot], he = P.hist_off[slot + 1];
      h_len = min(sp_last_n, max(0, he - hs));
      h_start = static_cast<uint32_t>(he - h_len);
    }
  }
  int aid[APRE];  // the first allowed ids of this thread, fetched ahead
#pragma unroll
  for (int t = 0; t < APRE; ++t) {
    const int j = a_beg + tid + t * NT;
    aid[t] = j < a_end ? P.allowed[j] : -1;
  }

  // The draw counter: a sampled row whose slot has no other row in the call reads and advances
  // its slot's packed word (counter << 16 | arrivals) in one atomic; otherwise each row adds one
  // arrival and reads the counter from the returned value, and the row that completes the slot's
  // arrivals also advances the counter and clears them.  Every row of the call sees the value
  // from before the call.  The leader's warp 0 issues it once the candidates are in.
  const bool ctr_warp = k_row > 0 && wid == 0 && crank == 0 && sampled && P.rec == nullptr;
  const bool ctr_thread = ctr_warp && lane == 0;
  unsigned long long ctr_old = 0ull;
  int rs_pre[2] = {-1, -1};  // row slots of the call, fetched ahead for the count of the slot's rows
  if (crank == 0 && wid == 0 && P.mode == MODE_SAMPLE) {
    rs_pre[0] = lane < P.B ? P.row_slot[lane] : -1;
    rs_pre[1] = lane + 32 < P.B ? P.row_slot[lane + 32] : -1;
  }
  int r_slot = 0;  // rows of this row's slot in the call (leader's warp 0)
  if (own_out) {
    // The counters now, before any CTA lets the next call launch: that call's atomics on these
    // words are issued after its launch, so after these have returned.
    if (ctr_warp) take_counter_early(rs_pre[0], rs_pre[1], P.row_slot, P.B, slot, P.ctr, ctl, lane);
    __syncthreads();
    grid_dep_launch();
  }

  int hid[HPRE];  // third metadata level: this thread's first history ids, for the table after the pass
#pragma unroll
  for (int j = 0; j < HPRE; ++j) {
    const int i = tid + j * NT;
    hid[j] = (penal && i < h_len) ? slice_id(hb[(h_start + static_cast<uint32_t>(i)) & h_mask], P.id_off) : -1;
  }

  // ---- 1b. first pass as pieces land ----------------------------------------------------------
  float ref = -INFINITY, mx = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY, s0 = 0.0f, s1 = 0.0f;
  int bmx = 0, bmx2 = 0;
  // logits of this thread's first allowed and history ids, fetched once their ids have landed
  // (after the first piece) and used after the pass
  float aval[APRE], hval[HPRE];
#pragma unroll
  for (int t = 0; t < APRE; ++t) aval[t] = 0.0f;
#pragma unroll
  for (int j = 0; j < HPRE; ++j) hval[j] = 0.0f;
  auto prefetch = [&]() {
#pragma unroll
    for (int t = 0; t < APRE; ++t)
      if (aid[t] >= lo && aid[t] < hi) aval[t] = elem_at<DT>(gchunk, static_cast<uint32_t>(aid[t] - lo));
#pragma unroll
    for (int j = 0; j < HPRE; ++j)
      if (hid[j] >= lo && hid[j] < hi) hval[j] = elem_at<DT>(gchunk, static_cast<uint32_t>(hid[j] - lo));
  };
  {
    // pieces stream through the ring: the last warp done with a slot refills it with the piece
    // nslot further on
    const int n_iter = (n_vec + PIECE_VECS - 1) / PIECE_VECS;
    if (n_iter == 0) prefetch();
    int si = 0;
    uint32_t ph = 0u;
#pragma unroll 1
    for (int p = 0; p < n_iter; ++p) {
      if (p < n_pieces) wait_bar(&mbar[si], ctl, P.err, false, ph);
      pass1_piece<DT>(data + si * PIECE_BYTES, gchunk, p, n_full, n_vec, n_el, ref, mx, mx2, mx3, bmx, bmx2, s0,
                      s1);
      if (p + nslot < n_pieces) {
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();  // this warp's reads of the slot are done before it counts
          if (atomicAdd(&ctl[CTL_SLOT0 + si], 1u) == NW - 1 && ctl[CTL_TIMEOUT] == 0u) {
            ctl[CTL_SLOT0 + si] = 0u;
            const int pn = p + nslot;
            ctl[CTL_LAST0 + si] = static_cast<uint32_t>(pn);
            fence_proxy_async_smem();
            const uint32_t nb = static_cast<uint32_t>(min(PIECE_BYTES, bytes_al - pn * PIECE_BYTES));
            mbar_arrive_expect_tx(&mbar[si], nb);
            bulk_g2s(data + si * PIECE_BYTES, grow + pn * PIECE_BYTES, nb, &mbar[si]);
          }
        }
      }
      if (p == 0) prefetch();
      if (++si == nslot) {
        si = 0;
        ph ^= 1u;
      }
    }
  }

  // allowed subset: this chunk's ids, each counted once, into (max, sum of exp)
  MaxSum al{-INFINITY, 0.0f};
  if (abits_in_ring && a_end > a_beg) {  // the ring's last piece is read by every warp, then cleared
    __syncthreads();
    for (int i = tid; i < bw_words; i += NT) abits[i] = 0u;
    __syncthreads();
  }
  {
    auto add_allowed = [&](int id, float x) {
      if (id >= lo && id < hi) {
        const uint32_t loc = static_cast<uint32_t>(id - lo);
        const uint32_t bit = 1u << (loc & 31);
        if (!(atomicOr(&abits[loc >> 5], bit) & bit)) online_add(al, x);
      }
    };
#pragma unroll
    for (int t = 0; t < APRE; ++t) add_allowed(aid[t], aval[t]);
    for (int j = a_beg + tid + APRE * NT; j < a_end; j += NT) {
      const int id = P.allowed[j];
      if (id >= lo && id < hi) add_allowed(id, elem_at<DT>(gchunk, static_cast<uint32_t>(id - lo)));
    }
  }

  // ---- history table of this chunk's id range, and the owners of its ids (a caller's window was
  // fetched before the first pass and has landed by now; a kept history is read now, after the
  // previous call: with early loads the first pass ran while that call finished) ---------------
  if (penal && kept_hist) {
    if (early) grid_dep_wait();
    const unsigned long long n = P.hlen[slot];
    h_len = static_cast<int>(min(static_cast<unsigned long long>(sp_last_n), n));
    h_start = static_cast<uint32_t>(n - static_cast<unsigned long long>(h_len)) & h_mask;
  }
  if (penal) {
    auto add_hist = [&](int id, bool have, float x) {
      if (id >= lo && id < hi) {
        const uint32_t loc = static_cast<uint32_t>(id - lo);
        const uint32_t owner = (loc / EPV) % NT;
        atomicOr(&hflag[owner >> 5], 1u << (owner & 31));
        const int h = hash_add(htab, P.hash_bits, loc);
        if (h == -2) atomicOr(P.err, STRATA_DEVERR_HISTORY);
        if (h >= 0) hraw[h] = __float_as_uint(have ? x : elem_at<DT>(gchunk, loc));  // the entry's creator
      }
    };
#pragma unroll
    for (int j = 0; j < HPRE; ++j) add_hist(hid[j], true, hval[j]);
    for (int i = tid + (kept_hist ? 0 : HPRE * NT); i < h_len; i += NT)
      add_hist(slice_id(hb[(h_start + static_cast<uint32_t>(i)) & h_mask], P.id_off), false, 0.0f);
  }
  __syncthreads();  // history table and owner flags complete

  // ---- 2. this CTA's record: the qw largest thread maxima of each warp and the (max, sum) pairs.
  // The candidate test key covers every id of the thread.  A threshold key must be a value that
  // both the raw and the penalised value of one id reach: a thread that owns no history id
  // publishes its maximum; one that owns some publishes nothing (a slightly weaker bound), unless
  // its warp has fewer than qw threads without history ids (long windows spread over the row),
  // in which case it publishes the best min(raw, penalised) over the batch that holds its maximum.
  const uint32_t kall = tid < n_vec ? order_key(mx) : 0u;
  uint32_t kthr = kall;
  if (penal) {
    const bool flagged = (hflag[tid >> 5] >> (tid & 31)) & 1u;
    const uint32_t plain = __ballot_sync(FULL_MASK, !flagged);
    if (flagged) kthr = 0u;
    if (flagged && kall != 0u && __popc(plain) < P.qw) {
      constexpr int RB = BATCH_VECS<DT>;
      const int vb = (bmx / (VR / RB)) * PIECE_VECS + (bmx % (VR / RB)) * RB * NT + tid;
      kthr = batch_safe_key<DT>(gchunk, vb, n_vec, n_el, htab, P.hash_bits, sp.rep, sp.freq, sp.pres);
    }
  }
  {
    uint32_t kk = kthr;
#pragma unroll 1
    for (int r = 0; r < P.qw; ++r) {  // the warp's r-th largest thread maximum, then drop it
      const uint32_t m = __reduce_max_sync(FULL_MASK, kk);
      if (lane == 0) wkey[wid * QW_MAX + r] = m;
      const uint32_t b = __ballot_sync(FULL_MASK, kk == m);
      if (lane == __ffs(b) - 1) kk = 0u;
    }
    // a thread whose maximum was published is the likeliest to reach T: bring the batch that holds
    // its maximum back into L1 now, so that the candidate scan after the exchange finds it there
    if (kk == 0u && kthr != 0u) {
      constexpr int RB = BATCH_VECS<DT>;
      const int vb = (bmx / (VR / RB)) * PIECE_VECS + (bmx % (VR / RB)) * RB * NT + tid;
#pragma unroll
      for (int r = 0; r < RB; ++r)
        if (vb + r * NT < n_full) prefetch_l1(gchunk + static_cast<size_t>(vb + r * NT) * 16);
    }
    const MaxSum wrow = warp_ms_fast(MaxSum{ref, s0 + s1});
    const MaxSum wal = warp_ms_fast(al);
    if (lane == 0) red4[wid] = make_float4(wrow.m, wrow.s, wal.m, wal.s);
  }
  __syncthreads();
  if (wid == 0) {
    // the CTA's (max, sum) pairs: lanes 0..NW-1 combine the row's, lanes 16..16+NW-1 the allowed
    // subset's (three shuffle steps each, side by side)
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
    // this CTA's record: key i = the (i / NW)-th largest of warp i % NW, then the two pairs
    static_assert(NW == 8, "record key i belongs to warp i % 8");
    uint32_t* own = xrec + crank * XW;
    for (int i = lane; i < Q; i += 32) own[i] = wkey[(i & (NW - 1)) * QW_MAX + (i >> 3)];
    if (lane == 0)
      *reinterpret_cast<uint4*>(own + Q) =
          make_uint4(__float_as_uint(M), __float_as_uint(sc), __float_as_uint(Ma), __float_as_uint(Sa));
    __syncwarp();
    if (lane == 0) mbar_arrive(&mbar[BAR_X0]);  // own record in place (release by this lane)
    __syncwarp();
  }
  cluster_wait();  // every CTA of the cluster is running: remote stores are safe from here on
  if (wid == 0 && lane < cs && static_cast<uint32_t>(lane) != crank) {
    const uint4* own = reinterpret_cast<const uint4*>(xrec + crank * XW);
    const uint32_t dst = dsmem_addr(smem_u32(xrec + crank * XW), static_cast<uint32_t>(lane));
    const uint32_t bar = dsmem_addr(smem_u32(&mbar[BAR_X0]), static_cast<uint32_t>(lane));
    const int n4 = (Q + 4) >> 2;
#pragma unroll 1
    for (int i = 0; i < n4; ++i) {
      const uint4 v = own[i];
      st_async_v4(dst + 16u * i, v.x, v.y, v.z, v.w, bar);
    }
  }
  wait_bar(&mbar[BAR_X0], ctl, P.err, true);  // every CTA's record is here

  // ---- the row threshold T and the log-normalisers -------------------------------------------
  // T = the kp-th largest of the cs*Q published keys (zeros included, so T = 0 when fewer than
  // kp real keys exist): the smallest published key with fewer than kp keys above it.  The keys
  // are values of distinct ids, so at least kp ids reach T.  One thread per key counts; the last
  // warp reduces the (max, sum) pairs meanwhile.
  if (kp > 0) {
    const int nk = cs * Q;
    const int qlog = 31 - __clz(Q);  // Q is a power of two
    // lpk consecutive lanes count for one key, lane `sub` over records sub, sub + lpk, ...
    int lpk = 1;
    while (lpk < 16 && nk * lpk * 2 <= NT) lpk *= 2;
    const int llog = 31 - __clz(lpk), sub = tid & (lpk - 1);
#pragma unroll 1
    for (int base = 0; base < nk * lpk; base += NT) {
      const int i = (base + tid) >> llog;
      uint32_t u = 0xFFFFFFFFu;
      int above = 0;
      if (i < nk) {
        u = xrec[(i >> qlog) * XW + (i & (Q - 1))];
        switch (P.qw) {  // the record length as a constant: the inner loop fully unrolled
          case 1: above = count_above_recs<2>(xrec, sub, lpk, cs, u); break;
          case 2: above = count_above_recs<4>(xrec, sub, lpk, cs, u); break;
          case 4: above = count_above_recs<8>(xrec, sub, lpk, cs, u); break;
          case 8: above = count_above_recs<16>(xrec, sub, lpk, cs, u); break;
          default: above = count_above_recs<32>(xrec, sub, lpk, cs, u); break;
        }
      }
      for (int off = 1; off < lpk; off <<= 1) above += __shfl_xor_sync(FULL_MASK, above, off);
      const uint32_t cand = (i < nk && sub == 0 && above < kp) ? u : 0xFFFFFFFFu;
      const uint32_t wmin = __reduce_min_sync(FULL_MASK, cand);
      if (lane == 0 && wmin != 0xFFFFFFFFu) atomicMin(&ctl[CTL_T], wmin);
    }
  }
  __syncthreads();
  const uint32_t T = cs * Q >= kp ? ctl[CTL_T] : 0u;  // fewer than kp published keys: no bound
  // the log-normalisers, by the last warp while the others look for candidates: lanes 0..15
  // combine the row's (max, sum) pairs, lanes 16..31 the allowed subset's
  if (wid == NW - 1) {
    const int c = lane & 15;
    float m = -INFINITY, sm_ = 0.0f;
    if (c < cs) {
      const float2 t = reinterpret_cast<const float2*>(xrec + c * XW + Q)[lane >> 4];
      m = t.x;
      sm_ = t.y;
    }
    float M = m;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, off));
    float sc = (m == -INFINITY || !(sm_ > 0.0f)) ? 0.0f : sm_ * ex2_approx((m - M) * LOG2E);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) sc += __shfl_xor_sync(FULL_MASK, sc, off);
    if (c == 0) ctl[CTL_LSE + (lane >> 4)] = __float_as_uint((M == -INFINITY || !(sc > 0.0f)) ? -INFINITY : M + logf(sc));
  }

  // ---- 3. candidates of this chunk: every element at or above T --------------------------------
  if (kp > 0) {
    // T as a float threshold (x >= Tf exactly when order_key(x) >= T, NaN never); T = 0 is no bound
    const float Tf = T == 0u ? -INFINITY : key_value(T);
    const bool own_hist = penal && ((hflag[tid >> 5] >> (tid & 31)) & 1u);  // only then can a hit be a history id
    // a masked row's top_k list holds exactly its named ids (below); T still serves the raw list
    const bool masked = mask_launch && a_end > a_beg && k_row > 0;
    const bool pen_from_t = k_row > 0 && !masked;
    const bool want = kall != 0u && kall >= T && (n_row > 0 || pen_from_t);
    const bool whole = want && order_key(mx3) >= T;  // a third batch also reaches T: a full rescan
    const int n_bat = (want && !whole) ? (order_key(mx2) >= T ? 2 : 1) : 0;
#pragma unroll 1
    for (int q = 0; q < n_bat; ++q) {
      constexpr int RB = BATCH_VECS<DT>;
      // every element at or above T sits in the batch that holds the max (and the second batch,
      // when its maximum reaches T): scan its 16 elements straight-line (independent loads), then
      // append the hits
      const int bq = q == 0 ? bmx : bmx2;
      const int vb = (bq / (VR / RB)) * PIECE_VECS + (bq % (VR / RB)) * RB * NT + tid;
      uint32_t hit = 0u;
      float xf[RB * EPV];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        float x[EPV];
        if (vb + r * NT < n_vec) {
          load_vec_g<DT>(gchunk, vb + r * NT, n_el, x);
        } else {
#pragma unroll
          for (int e = 0; e < EPV; ++e) x[e] = -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          xf[r * EPV + e] = x[e];
          hit |= static_cast<uint32_t>(x[e] >= Tf) << (r * EPV + e);
        }
      }
#pragma unroll 1
      for (; hit != 0u; hit &= hit - 1u) {
        const int b = __ffs(hit) - 1;
        const uint32_t loc = static_cast<uint32_t>((vb + (b / EPV) * NT) * EPV + (b % EPV));
        if (loc >= static_cast<uint32_t>(n_el)) continue;
        const float xv = pick(xf, b);
        const uint32_t o = order_key(xv);
        if (o == 0u || (own_hist && hash_count(htab, P.hash_bits, loc) != 0u)) continue;
        append_both(ctl, cand_pen, cand_raw, cap, sel_key(o, static_cast<uint32_t>(lo) + loc), xv, n_row > 0,
                    pen_from_t);
      }
    }
    const uint32_t need = __ballot_sync(FULL_MASK, whole);
    if (STRATA_UNLIKELY(need != 0u))
      warp_rescan<DT>(gchunk, need, __ballot_sync(FULL_MASK, own_hist), wid, lane, n_vec, n_el, lo, Tf, htab,
                      P.hash_bits, ctl, cand_pen, cand_raw, cap, n_row > 0, pen_from_t);
    if (penal) {  // penalised ids: raw value for the raw list, penalised value for the other
      for (int i = tid; i < P.hash_cap; i += NT) {
        const uint32_t ent = htab[i];
        if (ent == HASH_EMPTY) continue;
        const uint32_t loc = ent >> HASH_CNT_BITS;
        const uint32_t c = ent & ((1u << HASH_CNT_BITS) - 1u);
        const float raw = __uint_as_float(hraw[i]);
        const uint32_t id = static_cast<uint32_t>(lo) + loc;
        const uint32_t o = order_key(raw);
        if (o != 0u && o >= T && n_row > 0) {
          const uint32_t s = atomicAdd(&ctl[CTL_CAND_RAW], 1u);
          if (s < static_cast<uint32_t>(cap)) cand_raw[s] = sel_key(o, id);
        }
        const float pv = penalize(raw, c, sp.rep, sp.freq, sp.pres);
        const uint32_t op = order_key(pv);
        if (op != 0u && op >= T && pen_from_t) {
          const uint32_t s = atomicAdd(&ctl[CTL_CAND_PEN], 1u);
          const uint64_t key = sel_key(op, id);
          if (s < static_cast<uint32_t>(cap))
            cand_pen[s] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32), __float_as_uint(raw), 0u);
        }
      }
    }
    if (masked)  // every named id of this chunk once, with its penalised value
      masked_candidates<DT>(gchunk, lo, hi, aid[0], aid[1], aid[2], aid[3], P.allowed, a_beg + threadIdx.x + APRE * NT,
                            a_end, mbits, penal, htab, P.hash_bits, sp.rep, sp.freq, sp.pres, ctl, cand_pen, cap);
    __syncthreads();

    int np = static_cast<int>(ctl[CTL_CAND_PEN]);
    int nr = static_cast<int>(ctl[CTL_CAND_RAW]);
    // more candidates than the buffer holds (extreme ties): exact argmax rounds over the chunk
    // write its best k_row / n_row in order into the candidate buffers; more than RANK_LIMIT in
    // the buffer: argmax rounds over the buffer keep the best ones at its head
    if (STRATA_UNLIKELY(k_row > 0 && np > cap)) {
      if (MASK && masked)
        np = masked_rounds<DT>(gchunk, lo, hi, aid[0], aid[1], aid[2], aid[3], P.allowed, a_beg + tid + APRE * NT,
                               a_end, k_row, penal, htab, P.hash_bits, sp.rep, sp.freq, sp.pres, red64, cand_pen);
      else
        np = exact_rounds<DT>(gchunk, n_vec, n_el, lo, 0, k_row, penal, htab, P.hash_bits, hflag, sp.rep, sp.freq,
                              sp.pres, red64, cand_pen, cand_raw);
    } else if (STRATA_UNLIKELY(k_row > 0 && np > RANK_LIMIT)) {
      np = buffer_rounds(reinterpret_cast<uint32_t*>(cand_pen), 4, np, k_row, reinterpret_cast<uint32_t*>(sorted_pen),
                         red64);
    }
    if (STRATA_UNLIKELY(n_row > 0 && nr > cap))
      nr = exact_rounds<DT>(gchunk, n_vec, n_el, lo, 1, n_row, penal, htab, P.hash_bits, hflag, sp.rep, sp.freq,
                            sp.pres, red64, cand_pen, cand_raw);
    else if (STRATA_UNLIKELY(n_row > 0 && nr > RANK_LIMIT))
      nr = buffer_rounds(reinterpret_cast<uint32_t*>(cand_raw), 2, nr, n_row, reinterpret_cast<uint32_t*>(sorted_raw),
                         red64);
    if (k_row == 0) np = 0;
    if (n_row == 0) nr = 0;

    // keep this chunk's best k_row / n_row and store them into this CTA's slice of the leader's
    // lists (threads 0..255: penalised list, 256..511: raw list)
    const int sent_p = min(np, k_row), sent_r = min(nr, n_row);
    const uint32_t leader_bar = dsmem_addr(smem_u32(&mbar[BAR_X1]), 0);
    const int half = tid & (NT / 2 - 1);
    if (tid < NT / 2) {
      for (int i = half; i < np; i += NT / 2) {
        const uint4 ent = cand_pen[i];
        int out = i;
        if (np > k_row) {
          const uint64_t ki = (static_cast<uint64_t>(ent.y) << 32) | ent.x;
          const uint2* keys = reinterpret_cast<const uint2*>(cand_pen);
          int rank = 0;
#pragma unroll 4
          for (int j = 0; j < np; ++j) {
            const uint2 o = keys[2 * j];
            rank += ((static_cast<uint64_t>(o.y) << 32) | o.x) > ki;
          }
          out = rank < k_row ? rank : -1;
        }
        if (out >= 0) {
          uint64_t* key_p = recv_pkey + crank * P.kmax + out;
          uint32_t* raw_p = recv_praw + crank * P.kmax + out;
          if (crank == 0) {
            *key_p = (static_cast<uint64_t>(ent.y) << 32) | ent.x;
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
        int out = i;
        if (nr > n_row) {
          int rank = 0;
#pragma unroll 4
          for (int j = 0; j < nr; ++j) rank += cand_raw[j] > ki;
          out = rank < n_row ? rank : -1;
        }
        if (out >= 0) {
          uint64_t* slot_r = recv_raw + crank * P.nmax + out;
          if (crank == 0) *slot_r = ki;
          else st_async_v2(dsmem_addr(smem_u32(slot_r), 0), static_cast<uint32_t>(ki), static_cast<uint32_t>(ki >> 32), leader_bar);
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
  }

  if (kp == 0) __syncthreads();  // the log-normalisers are visible (the candidate phase has its own)
  const float lse = __uint_as_float(ctl[CTL_LSE]), lse_a = __uint_as_float(ctl[CTL_LSE_A]);

  // The leader alone writes the allowed-subset and chosen-id outputs (so no other CTA waits for the
  // previous call); it fetches those logits from global memory here, ahead of use.
  float alog[APRE] = {};
  float chosen_x = 0.0f;
  if (crank == 0) {
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

  // state of the tail (leader, warp 0)
  int k_eff = 0, n_eff = 0;
  Tail tl = {};

  // ---- 4. the leader ranks the received keys exactly -------------------------------------------
  if (crank == 0 && (P.flags & STRATA_FLAG_TEST_STALL)) test_stall(&mbar[BAR_STALL], ctl, P.err);
  if (kp > 0 && crank == 0) {
    if (cs > 1) wait_bar(&mbar[BAR_X1], ctl, P.err, true);
    if (ctr_warp && !own_out) r_slot = slot_rows(rs_pre[0], rs_pre[1], P.row_slot, P.B, slot, lane);
    __syncthreads();  // every slice (the leader's own included) is in place
    // slice offsets (every copying warp scans the counts itself), then warp c copies slice c into
    // the dense lists (the candidate buffers, free by now)
    {
      // every warp scans the slice counts itself; warp w copies slices w, w + NW, ... into the dense
      // lists (the candidate buffers, free by now) when a list fits them
      const uint2 n = lane < cs ? recv_cnt[lane] : make_uint2(0u, 0u);
      const int pc = min(static_cast<int>(n.x), P.kmax), rc = min(static_cast<int>(n.y), P.nmax);
      int ip = pc, ir = rc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int yp = __shfl_up_sync(FULL_MASK, ip, off), yr = __shfl_up_sync(FULL_MASK, ir, off);
        if (lane >= off) {
          ip += yp;
          ir += yr;
        }
      }
      const int tp = __shfl_sync(FULL_MASK, ip, 31), tr = __shfl_sync(FULL_MASK, ir, 31);
      if (wid == 0 && lane == 0) {
        ctl[CTL_TOT_P] = static_cast<uint32_t>(tp);
        ctl[CTL_TOT_R] = static_cast<uint32_t>(tr);
      }
      for (int c = wid; c < cs; c += NW) {
        const int my_p = __shfl_sync(FULL_MASK, pc, c), my_r = __shfl_sync(FULL_MASK, rc, c);
        const int off_p = __shfl_sync(FULL_MASK, ip, c) - my_p, off_r = __shfl_sync(FULL_MASK, ir, c) - my_r;
        if (tp <= cap - 8)
          for (int j = lane; j < my_p; j += 32) {
            const uint64_t k = recv_pkey[c * P.kmax + j];
            cand_pen[off_p + j] = make_uint4(static_cast<uint32_t>(k), static_cast<uint32_t>(k >> 32),
                                             recv_praw[c * P.kmax + j], 0u);
          }
        if (tr <= cap - 8)
          for (int j = lane; j < my_r; j += 32) cand_raw[off_r + j] = recv_raw[c * P.nmax + j];
      }
      if (wid == 0 && lane < 8) {  // zero keys pad both lists to a multiple of 8
        if (tp + lane < cap) cand_pen[tp + lane] = make_uint4(0u, 0u, 0u, 0u);
        if (tr + lane < cap) cand_raw[tr + lane] = 0ull;
      }
    }
    __syncthreads();
    const int tot_p = static_cast<int>(ctl[CTL_TOT_P]), tot_r = static_cast<int>(ctl[CTL_TOT_R]);
    // exact ranks by counting larger keys (first half of the threads: penalised list, second half:
    // raw list); a list longer than the dense buffer (heavy ties) is ranked over its slices
    const int half = tid & (NT / 2 - 1);
    if (tid < NT / 2) {
      for (int f = half; f < tot_p; f += NT / 2) {
        uint4 ent;
        int rank;
        if (STRATA_LIKELY(tot_p <= cap - 8)) {
          ent = cand_pen[f];
          rank = rank_desc(reinterpret_cast<const uint32_t*>(cand_pen), 4, (tot_p + 7) & ~7,
                           (static_cast<uint64_t>(ent.y) << 32) | ent.x);
        } else {
          int c = 0, j = f;
          for (int n = recv_count(recv_cnt, 0, 0, P.kmax); j >= n && c + 1 < cs; n = recv_count(recv_cnt, c, 0, P.kmax)) {
            j -= n;
            ++c;
          }
          const uint64_t k = recv_pkey[c * P.kmax + j];
          ent = make_uint4(static_cast<uint32_t>(k), static_cast<uint32_t>(k >> 32), recv_praw[c * P.kmax + j], 0u);
          rank = count_greater(reinterpret_cast<const uint32_t*>(recv_pkey), 2, P.kmax, recv_cnt, 0, cs, k);
        }
        if (rank < k_row) sorted_pen[rank] = ent;
      }
    } else {
      for (int f = half; f < tot_r; f += NT / 2) {
        uint64_t key;
        int rank;
        if (STRATA_LIKELY(tot_r <= cap - 8)) {
          key = cand_raw[f];
          rank = rank_desc(reinterpret_cast<const uint32_t*>(cand_raw), 2, (tot_r + 7) & ~7, key);
        } else {
          int c = 0, j = f;
          for (int n = recv_count(recv_cnt, 0, 1, P.nmax); j >= n && c + 1 < cs; n = recv_count(recv_cnt, c, 1, P.nmax)) {
            j -= n;
            ++c;
          }
          key = recv_raw[c * P.nmax + j];
          rank = count_greater(reinterpret_cast<const uint32_t*>(recv_raw), 2, P.nmax, recv_cnt, 1, cs, key);
        }
        if (rank < n_row) sorted_raw[rank] = key;
      }
    }
    __syncthreads();
    k_eff = min(k_row, tot_p);
    n_eff = min(n_row, tot_r);
    // the draw counter: issued after the block's last barrier (a barrier waits for a global atomic
    // before it to be performed), consumed by the draw, so the tail's first half hides its latency
    if (!early && ctr_thread) ctr_old = atomicAdd(&P.ctr[slot], r_slot == 1 ? (1ull << 16) : 1ull);

    // the tail's first half on <= 64 survivors (one warp); a vocabulary slice reports its lists
    // instead
    if (P.mode == MODE_SAMPLE && wid == 0 && valid && k_eff > 0 && P.rec == nullptr)
      tail_cuts(sorted_pen, k_eff, sampled, sp, lane, tl);
  }

  // a vocabulary slice: the row's record (its lists with whole-row ids, and its log-sum-exp)
  if (P.rec != nullptr && crank == 0)
    write_record(P.rec + static_cast<size_t>(row) * STRATA_SHARD_RECORD_BYTES, sorted_pen, k_eff, sorted_raw, n_eff,
                 lse, P.id_off, tid);

  // ---- outputs (leader only): with early loads the previous kernel owns outputs and counters
  // until it ends, unless this call has its own outputs (its counter was taken at the start) -----
  if (early && !own_out && crank == 0) {
    grid_dep_wait();
    if (ctr_thread) ctr_old = atomicAdd(&P.ctr[slot], r_slot == 1 ? (1ull << 16) : 1ull);
  }
  if (own_out && ctr_thread)  // taken at the start
    ctr_old = (static_cast<unsigned long long>(ctl[CTL_CTR + 1]) << 32) | ctl[CTL_CTR];

  // allowed-subset log-probabilities and the given chosen id
  if (crank == 0 && P.allowed_off != nullptr && P.allowed_lps != nullptr) {
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
  if (crank == 0 && P.mode == MODE_LOGPROBS && P.chosen_lp != nullptr && P.chosen != nullptr && tid == 0) {
    if (chosen_id >= 0 && chosen_id < P.V) {
      P.chosen_lp[row] = chosen_x - lse;
    } else {
      P.chosen_lp[row] = __int_as_float(0x7FC00000);
      atomicOr(P.err, STRATA_DEVERR_CHOSEN);
    }
  }

  if (kp > 0 && crank == 0) {
    // top-N raw alternatives and their log-probabilities
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
    if (P.mode == MODE_SAMPLE && wid == 0 && P.rec == nullptr) {
      int out = -1;
      float chosen_raw = __int_as_float(0x7FC00000);
      if (!valid) {
        if (lane == 0) atomicOr(P.err, STRATA_DEVERR_SLOT);
      } else if (k_eff == 0) {
        if (lane == 0) atomicOr(P.err, STRATA_DEVERR_NOCAND);
        // a sampled row without a candidate still counted itself among its slot's arrivals
        if (sampled && !own_out) slot_arrival_done(r_slot, slot, P.ctr, ctr_old, lane);
      } else {
        int j = 0;
        if (sampled) {
          uint32_t x0 = 0u;
          if (ctr_thread) x0 = philox_word0(sp.seed, pos, ctr_old >> 16);
          if (!own_out) slot_arrival_done(r_slot, slot, P.ctr, ctr_old, lane);
          j = tail_draw(tl, __shfl_sync(FULL_MASK, x0, 0), lane);
        }
        out = static_cast<int>(tail_id(tl, j));
        chosen_raw = tail_raw(tl, j);  // raw logit of the pick
      }
      if (lane == 0) {
        P.out_ids[row] = out;
        if (P.kept != nullptr) {
          P.kept[2 * row] = tl.m1;
          P.kept[2 * row + 1] = tl.m2;
        }
        if (P.chosen_lp != nullptr) P.chosen_lp[row] = (out >= 0) ? chosen_raw - lse : __int_as_float(0x7FC00000);
      }
      if ((P.row_draft != nullptr || P.ring != nullptr) && valid)
        slot_window_done(P.row_slot, P.out_ids, P.row_draft, P.done, P.slot_keep, P.ring, P.hlen, P.B, slot, lane);
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
  } else if (kp == 0 && P.mode == MODE_SAMPLE && crank == 0 && tid == 0 && P.rec == nullptr) {
    // no selection in this row: only an out-of-range slot gets here
    P.out_ids[row] = -1;
    if (P.kept != nullptr) {
      P.kept[2 * row] = 0;
      P.kept[2 * row + 1] = 0;
    }
    if (P.chosen_lp != nullptr) P.chosen_lp[row] = __int_as_float(0x7FC00000);
    atomicOr(P.err, STRATA_DEVERR_SLOT);
  }
  if (P.mode == MODE_SAMPLE && crank == 0 && P.topk_ids != nullptr && kp == 0 && tid < KMAX) {
    P.topk_ids[static_cast<long long>(row) * KMAX + tid] = -1;
    if (P.topk_vals != nullptr) P.topk_vals[static_cast<long long>(row) * KMAX + tid] = __int_as_float(0x7FC00000);
  }
  if (P.mode == MODE_SAMPLE && valid && sp_k > P.kmax && crank == 0 && tid == 0) atomicOr(P.err, STRATA_DEVERR_SHAPE);
  if (STRATA_UNLIKELY(ctl[CTL_TIMEOUT] != 0u)) {
    // a wait ran out: a copy, or another CTA's stores into this one, may still be on the way, so
    // wait for each once more (bounded) before the CTA leaves
    for (int si = 0; si < min(nslot, n_pieces); ++si) {
      const int pl = static_cast<int>(ctl[CTL_LAST0 + si]);
      wait_bar(&mbar[si], ctl, P.err, false, static_cast<uint32_t>(pl / nslot) & 1u);
    }
    if (cs > 1) {
      wait_bar(&mbar[BAR_X0], ctl, P.err, true);
      if (crank == 0) wait_bar(&mbar[BAR_X1], ctl, P.err, true);
    }
  }
}

}  // namespace strata
