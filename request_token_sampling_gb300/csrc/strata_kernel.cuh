// strata_kernel.cuh -- the fused row kernel: one HBM pass per logit row.
//
// Each logit row is split over a thread-block cluster of `cs` CTAs (one chunk per CTA).  A CTA
//   1. bulk-copies its chunk into shared memory (16 KiB pieces, one mbarrier each), and while the
//      bytes land builds the row's history table for its id range (bitmap + open-addressing
//      counts) and, as each piece completes, runs the first pass: the per-thread running max and
//      sum of exp (log-sum-exp of the raw logits);
//   2. derives a selection threshold t_c: the q-th largest per-thread maximum of the logits that
//      carry no penalty (q = ceil(K/cs), K = max(top_k, top_n)).  q distinct elements of the
//      chunk reach t_c, so min over the cluster of t_c bounds the row's K-th largest value from
//      below; the CTAs exchange t_c and their (max, sum) pairs through DSMEM (cluster barrier B0);
//   3. rescans only the threads whose maximum reaches the row threshold, adds the penalised ids
//      from the history table, keeps its best <= K candidates and sends them to the cluster's
//      leader CTA through DSMEM (cluster barrier B1);
//   4. the leader ranks the <= cs*K received keys exactly, then one warp runs the tail of the
//      chain on <= 64 survivors: min_p, top_p, temperature, the Philox draw.
// Every CTA writes the allowed-subset and chosen-id log-probabilities of its own id range.
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

constexpr int NT = 512;                      // threads per CTA
constexpr int NW = NT / 32;                  // warps per CTA
constexpr int VR = 4;                        // 16-byte vectors per thread per piece
constexpr int PIECE_VECS = NT * VR;
constexpr int PIECE_BYTES = PIECE_VECS * 16; // 32 KiB per bulk copy
constexpr int MAX_PIECES = 6;                // chunk <= 192 KiB
constexpr int MAX_CS = 16;                   // CTAs per row (non-portable cluster size)
constexpr int KMAX = STRATA_MAX_TOP_K;
constexpr int NMAX = STRATA_MAX_TOP_N;
constexpr int QMAX = 8;                      // per-CTA threshold rank handled by the warp stage
constexpr int LOCAL_CAP = 512;               // per-CTA candidate buffer (beyond: exact rounds)
constexpr int HASH_CNT_BITS = 13;            // history table entry = (local id << 13) | count
constexpr uint32_t HASH_EMPTY = 0xFFFFFFFFu;
constexpr int MODE_SAMPLE = 0;
constexpr int MODE_LOGPROBS = 1;
constexpr uint32_t SLOT_SAMPLED = 1u;
constexpr uint32_t SLOT_PENAL = 2u;
constexpr long long WAIT_CYCLES = 4000000000LL;  // bounded waits: ~2 s at GB300 clocks

// Control words in shared memory.
enum : int {
  CTL_CAND_PEN = 0,
  CTL_CAND_RAW = 1,
  CTL_TC = 2,
  CTL_CTR_LO = 3,
  CTL_CTR_HI = 4,
  CTL_TIMEOUT = 5,
  CTL_X0 = 6,        // first Philox word of the leader's row
  CTL_RECV_NP = 7,   // leader: entries received in the flat penalised / raw lists
  CTL_RECV_NR = 8,
  CTL_BASE_P = 9,    // this CTA's slice of the leader's lists
  CTL_BASE_R = 10,
  CTL_MAXP = 11,     // leader: largest high key word received per list, refined thresholds
  CTL_MAXR = 12,
  CTL_TP = 13,
  CTL_TR = 14,
  CTL_WORDS = 16
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
  uint32_t flags;
};

struct Layout {
  uint32_t data, mbar, hbits, abits, hash, dirty, tc, ms, wtop, red, ctl;
  uint32_t cand_pen, cand_raw, recv_pen, recv_raw, recv_cnt, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Shared-memory layout of one CTA; identical in every CTA of a launch.
__host__ __device__ inline Layout make_layout(int chunk, int esz, int hash_cap, int cs, int kmax,
                                              int nmax) {
  Layout L;
  uint32_t o = 0;
  L.data = o;
  o += align_up(static_cast<uint32_t>(chunk) * esz, 128);
  L.mbar = o;
  o += MAX_PIECES * 8;
  const uint32_t bw = align_up((static_cast<uint32_t>(chunk) + 31) / 32 * 4, 16);
  L.hbits = o;
  o += bw;
  L.abits = o;
  o += bw;
  L.hash = o;
  o += static_cast<uint32_t>(hash_cap) * 4;
  L.dirty = o;
  o += NT / 8;
  L.tc = o;
  o += MAX_CS * 4;
  o = align_up(o, 16);
  L.ms = o;
  o += MAX_CS * 16;
  L.wtop = o;
  o += NW * QMAX * 4;
  L.red = o;
  o += NW * 16 + 64;
  L.ctl = o;
  o += CTL_WORDS * 4;
  o = align_up(o, 16);
  L.cand_pen = o;
  o += LOCAL_CAP * 16;
  L.cand_raw = o;
  o += LOCAL_CAP * 8;
  L.recv_pen = o;
  o += static_cast<uint32_t>(cs * kmax) * 16;
  L.recv_raw = o;
  o += static_cast<uint32_t>(cs * nmax) * 8;
  L.recv_cnt = o;
  o += MAX_CS * 8;
  L.total = align_up(o, 128);
  return L;
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

__device__ __forceinline__ bool bit_at(const uint32_t* bits, uint32_t loc) {
  return (bits[loc >> 5] >> (loc & 31)) & 1u;
}

__device__ __forceinline__ uint32_t hash_slot(uint32_t loc, int bits) {
  return (loc * 0x9E3779B1u) >> (32 - bits);
}

// Count one occurrence of chunk-local id `loc`; false if the table is full.
__device__ bool hash_add(uint32_t* tab, int bits, uint32_t loc) {
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t h = hash_slot(loc, bits);
  for (uint32_t n = 0; n <= mask; ++n) {
    uint32_t cur = *reinterpret_cast<volatile uint32_t*>(&tab[h]);
    if (cur == HASH_EMPTY) {
      const uint32_t prev = atomicCAS(&tab[h], HASH_EMPTY, (loc << HASH_CNT_BITS) | 1u);
      if (prev == HASH_EMPTY) return true;
      cur = prev;
    }
    if ((cur >> HASH_CNT_BITS) == loc) {
      atomicAdd(&tab[h], 1u);
      return true;
    }
    h = (h + 1u) & mask;
  }
  return false;
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

// Bounded wait on piece `p` (phase 0).  On timeout the error word and a shared flag are set and
// the caller carries on, so every thread still reaches every cluster barrier.
__device__ __forceinline__ void wait_piece(uint64_t* mbar, int p, uint32_t* ctl, uint32_t* err) {
  if (mbar_try_wait(&mbar[p], 0)) return;
  const long long t0 = clock64();
  while (!mbar_try_wait(&mbar[p], 0)) {
    if (clock64() - t0 > WAIT_CYCLES) {
      atomicOr(err, STRATA_DEVERR_TIMEOUT);
      ctl[CTL_TIMEOUT] = 1u;
      return;
    }
  }
}

__device__ __forceinline__ void online_add(MaxSum& a, float v) {
  if (v == -INFINITY || v != v) return;
  if (v > a.m) {
    a.s = (a.m == -INFINITY) ? 1.0f : a.s * ex2_approx((a.m - v) * LOG2E) + 1.0f;
    a.m = v;
  } else {
    a.s += ex2_approx((v - a.m) * LOG2E);
  }
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

// Exact argmax rounds over this CTA's chunk: the `need` largest keys in order (penalised values
// for list 0, raw values for list 1), written to the candidate buffer.  Only taken when more
// candidates reach the row threshold than the buffer holds (heavy ties); kept out of line so the
// common path stays small.  Every thread of the CTA calls it.  Returns the number found.
template <int DT>
__device__ __noinline__ int exact_rounds(const unsigned char* data, int n_vec, int n_el, int lo, int list, int need,
                                         bool penal, const uint32_t* hbits, const uint32_t* htab, int hash_bits,
                                         float rep, float freq, float pres, uint64_t* red64, uint4* cand_pen,
                                         uint64_t* cand_raw) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  uint64_t prev = ~0ull;
  int got = 0;
  for (int r = 0; r < need; ++r) {
    uint64_t best = 0ull;
    for (int v = tid; v < n_vec; v += NT) {
      float x[EPV];
      load_vec<DT>(data, v, x);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const uint32_t loc = static_cast<uint32_t>(v * EPV + e);
        if (loc >= static_cast<uint32_t>(n_el)) continue;
        float pv = x[e];
        if (list == 0 && penal && bit_at(hbits, loc)) pv = penalize(pv, hash_count(htab, hash_bits, loc), rep, freq, pres);
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

// This thread's top two over the ids that carry no penalty (rare: taken only when the plain top
// two hold a penalised id).  Out of line to keep the common path's code small.
template <int DT>
__device__ __noinline__ void masked_top2(const unsigned char* data, int n_vec, int n_el, const uint32_t* hbits,
                                         float* v1o, int* i1o, float* v2o, int* i2o) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
  float v1 = -INFINITY, v2 = -INFINITY;
  int i1 = -1, i2 = -1;
#pragma unroll 1
  for (int v = threadIdx.x; v < n_vec; v += NT) {
    float x[EPV];
    load_vec<DT>(data, v, x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const int loc = v * EPV + e;
      if (loc < n_el && x[e] > v2 && !bit_at(hbits, static_cast<uint32_t>(loc))) {
        if (x[e] > v1) {
          v2 = v1;
          i2 = i1;
          v1 = x[e];
          i1 = loc;
        } else {
          v2 = x[e];
          i2 = loc;
        }
      }
    }
  }
  *v1o = v1;
  *i1o = i1;
  *v2o = v2;
  *i2o = i2;
}

// Every element of this thread at or above T (a thread whose second best reaches T): appended to
// both candidate lists one by one.  Out of line (rare).
template <int DT>
__device__ __noinline__ void rescan_thread(const unsigned char* data, int n_vec, int n_el, int lo, uint32_t T,
                                           bool penal, const uint32_t* hbits, uint32_t* ctl, uint4* cand_pen,
                                           uint64_t* cand_raw, bool to_raw, bool to_pen) {
  constexpr int EPV = 16 / (DT == 0 ? 4 : 2);
#pragma unroll 1
  for (int v = threadIdx.x; v < n_vec; v += NT) {
    float x[EPV];
    load_vec<DT>(data, v, x);
#pragma unroll 1
    for (int e = 0; e < EPV; ++e) {
      const uint32_t loc = static_cast<uint32_t>(v * EPV + e);
      const uint32_t o = order_key(x[e]);
      if (loc >= static_cast<uint32_t>(n_el) || o == 0u || o < T) continue;
      if (penal && bit_at(hbits, loc)) continue;
      const uint64_t key = sel_key(o, static_cast<uint32_t>(lo) + loc);
      if (to_raw) {
        const uint32_t i = atomicAdd(&ctl[CTL_CAND_RAW], 1u);
        if (i < LOCAL_CAP) cand_raw[i] = key;
      }
      if (to_pen) {
        const uint32_t i = atomicAdd(&ctl[CTL_CAND_PEN], 1u);
        if (i < LOCAL_CAP)
          cand_pen[i] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32), __float_as_uint(x[e]), 0u);
      }
    }
  }
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

// ------------------------------------------------------------------------------ the kernel
template <int DT>
__global__ void __launch_bounds__(NT, 2) rows_kernel(const KParams P) {
  extern __shared__ __align__(128) unsigned char sm[];
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int EPV = 16 / ESZ;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool early = (P.flags & STRATA_FLAG_EARLY_LOAD) != 0u;
  if (!early) grid_dep_wait();  // inputs may be the previous kernel's outputs

  const uint32_t crank = cluster_ctarank();
  const int cs = P.cs;
  const int row = blockIdx.x / cs;
  const Layout L = make_layout(P.chunk, ESZ, P.hash_cap, cs, P.kmax, P.nmax);
  const int lo = static_cast<int>(crank) * P.chunk;
  const int hi = min(P.V, lo + P.chunk);
  const int n_el = max(0, hi - lo);
  const int bytes = n_el * ESZ;
  const int bytes_al = bytes & ~15;
  const int n_vec = (bytes + 15) >> 4;
  const int n_pieces = (bytes_al + PIECE_BYTES - 1) / PIECE_BYTES;

  unsigned char* data = sm + L.data;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + L.mbar);
  const char* grow = static_cast<const char*>(P.logits) + (static_cast<long long>(row) * P.ld + lo) * ESZ;

  // ---- 1. the bulk copies of this chunk go out first ---------------------------------------
  if (wid == 0) {  // lane 0 initialises the piece barriers, lane p issues piece p
    if (lane == 0) {
      for (int p = 0; p < n_pieces; ++p) mbar_init(&mbar[p], 1);
      fence_mbar_init();
    }
    __syncwarp();
    for (int p = lane; p < n_pieces; p += 32) {
      const uint32_t nb = static_cast<uint32_t>(min(PIECE_BYTES, bytes_al - p * PIECE_BYTES));
      mbar_arrive_expect_tx(&mbar[p], nb);
      bulk_g2s(data + p * PIECE_BYTES, grow + p * PIECE_BYTES, nb, &mbar[p]);
    }
  }
  grid_dep_launch();

  uint32_t* hbits = reinterpret_cast<uint32_t*>(sm + L.hbits);
  uint32_t* abits = reinterpret_cast<uint32_t*>(sm + L.abits);
  uint32_t* htab = reinterpret_cast<uint32_t*>(sm + L.hash);
  uint32_t* tc_arr = reinterpret_cast<uint32_t*>(sm + L.tc);
  float4* ms_arr = reinterpret_cast<float4*>(sm + L.ms);
  uint32_t* wtop = reinterpret_cast<uint32_t*>(sm + L.wtop);
  uint64_t* red64 = reinterpret_cast<uint64_t*>(sm + L.red);
  float4* red4 = reinterpret_cast<float4*>(sm + L.red);
  uint32_t* ctl = reinterpret_cast<uint32_t*>(sm + L.ctl);
  uint4* cand_pen = reinterpret_cast<uint4*>(sm + L.cand_pen);
  uint64_t* cand_raw = reinterpret_cast<uint64_t*>(sm + L.cand_raw);
  const uint4* recv_pen = reinterpret_cast<const uint4*>(sm + L.recv_pen);
  const uint64_t* recv_raw = reinterpret_cast<const uint64_t*>(sm + L.recv_raw);

  // The ragged last vector (chunk bytes not a multiple of 16) is read with plain loads by its
  // owner thread, padded with -inf.
  if (bytes > bytes_al && tid == (n_vec - 1) % NT) {
    const int tv = n_vec - 1;
    if constexpr (DT == 0) {
      const float* g = reinterpret_cast<const float*>(grow);
      float* d = reinterpret_cast<float*>(data);
      for (int e = 0; e < EPV; ++e) {
        const int idx = tv * EPV + e;
        d[idx] = idx < n_el ? g[idx] : -INFINITY;
      }
    } else {
      const uint16_t* g = reinterpret_cast<const uint16_t*>(grow);
      uint16_t* d = reinterpret_cast<uint16_t*>(data);
      for (int e = 0; e < EPV; ++e) {
        const int idx = tv * EPV + e;
        d[idx] = idx < n_el ? g[idx] : static_cast<uint16_t>(0xFF80u);
      }
    }
  }

  const int bw_words = (P.chunk + 31) >> 5;
  for (int i = tid; i < bw_words; i += NT) {
    hbits[i] = 0u;
    abits[i] = 0u;
  }
  for (int i = tid; i < P.hash_cap; i += NT) htab[i] = HASH_EMPTY;
  if (tid < CTL_WORDS) ctl[tid] = 0u;
  __syncthreads();           // tables zeroed, piece barriers initialised
  cluster_arrive_relaxed();  // this CTA is running (DSMEM access waits for every CTA, below)

  // ---- row metadata (inputs only: slot keys are never written by a kernel) -------------------
  int slot = -1;
  bool valid = true;
  SlotDev sp{};
  if (P.mode == MODE_SAMPLE) {
    slot = P.row_slot[row];
    valid = static_cast<unsigned>(slot) < static_cast<unsigned>(P.max_slots);
    if (valid) sp = P.slots[slot];
  }
  const bool sampled = valid && (sp.flags & SLOT_SAMPLED);
  const int k_row = (P.mode == MODE_SAMPLE && valid) ? min(max(sp.k, 1), P.kmax) : 0;
  const int n_row = P.nmax;
  const int kp = max(k_row, n_row);
  const int q = (kp + cs - 1) / cs;
  const bool penal = (P.mode == MODE_SAMPLE) && valid && (sp.flags & SLOT_PENAL) && P.hist_off != nullptr &&
                     slot < P.n_hist_slots && P.hash_cap > 0;
  const unsigned long long pos = (P.mode == MODE_SAMPLE) ? static_cast<unsigned long long>(P.row_pos[row]) : 0ull;
  const int chosen_id = (P.mode == MODE_LOGPROBS && P.chosen != nullptr) ? P.chosen[row] : -1;
  int a_beg = 0, a_end = 0;
  if (P.allowed_off != nullptr) {
    a_beg = P.allowed_off[row];
    a_end = P.allowed_off[row + 1];
  }
  // the first two allowed ids of this thread: mark the chunk's dedup bits now (before the data)
  int aid[2];
  bool acount[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int j = a_beg + tid + t * NT;
    aid[t] = j < a_end ? P.allowed[j] : -1;
    acount[t] = false;
    if (aid[t] >= lo && aid[t] < hi) {
      const uint32_t loc = static_cast<uint32_t>(aid[t] - lo);
      const uint32_t bit = 1u << (loc & 31);
      acount[t] = !(atomicOr(&abits[loc >> 5], bit) & bit);
    }
  }

  // The draw counter: each sampled row adds one arrival to its slot's packed word (counter << 16 |
  // arrivals) and reads the counter from the returned value; the row that completes the slot's
  // arrivals also advances the counter and clears them, so every row of the call sees the value
  // from before the call.  Issued early, consumed just before the leader's merge.
  const bool ctr_warp = k_row > 0 && wid == 0 && crank == 0 && sampled;
  const bool ctr_thread = ctr_warp && lane == 0;
  int r_s = 0;
  unsigned long long ctr_old = 0ull;
  if (!early && ctr_thread) ctr_old = atomicAdd(&P.ctr[slot], 1ull);
  if (ctr_warp) {
    for (int b0 = 0; b0 < P.B; b0 += 32) {
      const int b = b0 + lane;
      r_s += __popc(__ballot_sync(FULL_MASK, b < P.B && P.row_slot[b] == slot));
    }
  }

  // ---- history table of this chunk's id range ------------------------------------------------
  if (penal) {
    const int hb = P.hist_off[slot], he = P.hist_off[slot + 1];
    const int h_len = min(sp.last_n, max(0, he - hb));
    const int h_start = he - h_len;
    for (int i = tid; i < h_len; i += NT) {
      const int id = P.hist[h_start + i];
      if (id >= lo && id < hi) {
        const uint32_t loc = static_cast<uint32_t>(id - lo);
        atomicOr(&hbits[loc >> 5], 1u << (loc & 31));
        if (!hash_add(htab, P.hash_bits, loc)) atomicOr(P.err, STRATA_DEVERR_HISTORY);
      }
    }
  }

  // ---- 1b. first pass as pieces land: running (max, sum of exp) and this thread's top two ------
  MaxSum acc{-INFINITY, 0.0f};
  float v1 = -INFINITY, v2 = -INFINITY;
  int i1 = -1, i2 = -1;
  {
    int waited = -1;
    int i = 0;
#pragma unroll 1
    for (int v = tid; v < n_vec; v += NT, ++i) {
      const int p = i / VR;
      if (p < n_pieces && p != waited) {
        wait_piece(mbar, p, ctl, P.err);
        waited = p;
      }
      float x[EPV];
      load_vec<DT>(data, v, x);
      float vm = x[0];
#pragma unroll
      for (int e = 1; e < EPV; ++e) vm = fmaxf(vm, x[e]);
      if (vm > acc.m) {
        acc.s = (acc.m == -INFINITY) ? 0.0f : acc.s * ex2_approx((acc.m - vm) * LOG2E);
        acc.m = vm;
      }
      if (acc.m != -INFINITY) {
        const float mb = acc.m * LOG2E;
        float t = 0.0f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) t += ex2_approx(fmaf(x[e], LOG2E, -mb));
        acc.s += t;
      }
      if (vm > v2) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const int loc = v * EPV + e;
          if (x[e] > v2 && loc < n_el) {
            if (x[e] > v1) {
              v2 = v1;
              i2 = i1;
              v1 = x[e];
              i1 = loc;
            } else {
              v2 = x[e];
              i2 = loc;
            }
          }
        }
      }
    }
  }
  for (int p = 0; p < n_pieces; ++p) wait_piece(mbar, p, ctl, P.err);  // all pieces visible here
  __syncthreads();  // history table and allowed dedup bits complete

  // this thread's top two over the ids that carry no penalty (the threshold's elements)
  if (penal && ((i1 >= 0 && bit_at(hbits, static_cast<uint32_t>(i1))) ||
                (i2 >= 0 && bit_at(hbits, static_cast<uint32_t>(i2)))))
    masked_top2<DT>(data, n_vec, n_el, hbits, &v1, &i1, &v2, &i2);
  const uint32_t o1 = (i1 >= 0) ? order_key(v1) : 0u;
  const uint32_t o2 = (i2 >= 0) ? order_key(v2) : 0u;

  // ---- 2. threshold t_c and the CTA's (max, sum) of the row and of the allowed subset ---------
  if (kp > 0 && q <= QMAX) {
    uint32_t key = o1;
    for (int r = 0; r < q; ++r) {
      const uint32_t mx = __reduce_max_sync(FULL_MASK, key);
      if (lane == 0) wtop[wid * q + r] = mx;
      const uint32_t bal = __ballot_sync(FULL_MASK, key == mx);
      if (lane == __ffs(bal) - 1) key = 0u;
    }
  }
  MaxSum al{-INFINITY, 0.0f};
#pragma unroll
  for (int t = 0; t < 2; ++t)
    if (acount[t]) online_add(al, elem_at<DT>(data, static_cast<uint32_t>(aid[t] - lo)));
  for (int j = a_beg + tid + 2 * NT; j < a_end; j += NT) {
    const int id = P.allowed[j];
    if (id >= lo && id < hi) {
      const uint32_t loc = static_cast<uint32_t>(id - lo);
      const uint32_t bit = 1u << (loc & 31);
      if (!(atomicOr(&abits[loc >> 5], bit) & bit)) online_add(al, elem_at<DT>(data, loc));
    }
  }
  {
    const MaxSum wrow = warp_ms_fast(acc);
    const MaxSum wal = warp_ms_fast(al);
    if (lane == 0) red4[wid] = make_float4(wrow.m, wrow.s, wal.m, wal.s);
  }
  __syncthreads();
  float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);
  uint32_t tq = 0u;
  if (wid == 0) {
    MaxSum r1{-INFINITY, 0.0f}, r2{-INFINITY, 0.0f};
    if (lane < NW) {
      const float4 t = red4[lane];
      r1 = {t.x, t.y};
      r2 = {t.z, t.w};
    }
    r1 = warp_ms_fast(r1);
    r2 = warp_ms_fast(r2);
    mine = make_float4(r1.m, r1.s, r2.m, r2.s);
    if (kp > 0 && q <= QMAX) {
      uint32_t vals[4];
      const int nv = NW * q;
#pragma unroll
      for (int j = 0; j < 4; ++j) vals[j] = (lane + 32 * j < nv) ? wtop[lane + 32 * j] : 0u;
      for (int r = 0; r < q; ++r) {
        const uint32_t lm = max(max(vals[0], vals[1]), max(vals[2], vals[3]));
        const uint32_t mx = __reduce_max_sync(FULL_MASK, lm);
        const uint32_t bal = __ballot_sync(FULL_MASK, lm == mx);
        if (lane == __ffs(bal) - 1) {
          if (vals[0] == mx) vals[0] = 0u;
          else if (vals[1] == mx) vals[1] = 0u;
          else if (vals[2] == mx) vals[2] = 0u;
          else vals[3] = 0u;
        }
        tq = mx;
      }
    }
  }

  // ---- exchange through DSMEM (cluster barrier B0) ---------------------------------------------
  cluster_wait();
  if (wid == 0 && lane < cs) {
    const uint32_t r = static_cast<uint32_t>(lane);
    dsmem_st_u32(dsmem_addr(smem_u32(tc_arr + crank), r), tq);
    dsmem_st_v4(dsmem_addr(smem_u32(ms_arr + crank), r), __float_as_uint(mine.x), __float_as_uint(mine.y),
                __float_as_uint(mine.z), __float_as_uint(mine.w));
  }
  cluster_arrive();
  cluster_wait();

  // every warp reduces the cluster's contributions itself (lane c holds CTA c's)
  uint32_t T;
  float lse, lse_a;
  {
    const bool in = lane < cs;
    const float4 t = in ? ms_arr[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    T = __reduce_min_sync(FULL_MASK, in ? tc_arr[lane] : 0xFFFFFFFFu);
    const MaxSum g = warp_ms_fast(MaxSum{t.x, t.y});
    const MaxSum ga = warp_ms_fast(MaxSum{t.z, t.w});
    lse = (g.m == -INFINITY || !(g.s > 0.0f)) ? -INFINITY : g.m + logf(g.s);
    lse_a = (ga.m == -INFINITY || !(ga.s > 0.0f)) ? -INFINITY : ga.m + logf(ga.s);
  }
  // state of the tail, carried across the wait for the previous kernel (leader, warp 0)
  int k_eff = 0, n_eff = 0, m1 = 0, m2 = 0, n_recv_p = 0;
  float Ca = 0.0f, Cb = 0.0f, wa = 0.0f, wb = 0.0f;  // tempered weights and their fp32 prefix sums
  uint4 ea = make_uint4(0, 0, 0, 0), eb = make_uint4(0, 0, 0, 0);
  float va = 0.0f, vb = 0.0f;

  // ---- 3. candidates of this chunk: every element at or above the row threshold T ------------
  if (kp > 0) {
    if (q > QMAX) T = 0u;  // no usable bound: every element is a candidate
    auto put = [&](uint64_t key, float raw, bool to_raw, bool to_pen) {
      if (to_raw && n_row > 0) {
        const uint32_t i = atomicAdd(&ctl[CTL_CAND_RAW], 1u);
        if (i < LOCAL_CAP) cand_raw[i] = key;
      }
      if (to_pen && k_row > 0) {
        const uint32_t i = atomicAdd(&ctl[CTL_CAND_PEN], 1u);
        if (i < LOCAL_CAP)
          cand_pen[i] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32),
                                   __float_as_uint(raw), 0u);
      }
    };
    // a thread whose second best reaches T may hold more: it rescans its own elements
    const bool full = (T == 0u && tid < n_vec) || (o2 != 0u && o2 >= T);
    if (full) rescan_thread<DT>(data, n_vec, n_el, lo, T, penal, hbits, ctl, cand_pen, cand_raw, n_row > 0, k_row > 0);
    {  // the common case: at most this thread's best reaches T (one warp-wide append per list)
      const bool one = !full && o1 != 0u && o1 >= T;
      const uint32_t bal = __ballot_sync(FULL_MASK, one);
      if (bal != 0u) {
        const int leader = __ffs(bal) - 1;
        const uint32_t before = __popc(bal & ((1u << lane) - 1u));
        uint32_t base_r = 0, base_p = 0;
        if (lane == leader) {
          if (n_row > 0) base_r = atomicAdd(&ctl[CTL_CAND_RAW], static_cast<uint32_t>(__popc(bal)));
          if (k_row > 0) base_p = atomicAdd(&ctl[CTL_CAND_PEN], static_cast<uint32_t>(__popc(bal)));
        }
        base_r = __shfl_sync(FULL_MASK, base_r, leader) + before;
        base_p = __shfl_sync(FULL_MASK, base_p, leader) + before;
        if (one) {
          const uint64_t key = sel_key(o1, static_cast<uint32_t>(lo + i1));
          if (n_row > 0 && base_r < LOCAL_CAP) cand_raw[base_r] = key;
          if (k_row > 0 && base_p < LOCAL_CAP)
            cand_pen[base_p] = make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32),
                                          __float_as_uint(v1), 0u);
        }
      }
    }
    if (penal) {  // penalised ids: raw value for the raw list, penalised value for the other
      for (int i = tid; i < P.hash_cap; i += NT) {
        const uint32_t ent = htab[i];
        if (ent == HASH_EMPTY) continue;
        const uint32_t loc = ent >> HASH_CNT_BITS;
        const uint32_t c = ent & ((1u << HASH_CNT_BITS) - 1u);
        const float raw = elem_at<DT>(data, loc);
        const uint32_t id = static_cast<uint32_t>(lo) + loc;
        const uint32_t o = order_key(raw);
        if (o != 0u && o >= T) put(sel_key(o, id), raw, true, false);
        const float pv = penalize(raw, c, sp.rep, sp.freq, sp.pres);
        const uint32_t op = order_key(pv);
        if (op != 0u && op >= T) put(sel_key(op, id), raw, false, true);
      }
    }
    __syncthreads();

    int np = static_cast<int>(ctl[CTL_CAND_PEN]);
    int nr = static_cast<int>(ctl[CTL_CAND_RAW]);
    // more candidates than the buffer holds (heavy ties): exact argmax rounds write the chunk's
    // best k_row / n_row in order into the candidate buffers
    if (k_row > 0 && np > LOCAL_CAP)
      np = exact_rounds<DT>(data, n_vec, n_el, lo, 0, k_row, penal, hbits, htab, P.hash_bits, sp.rep, sp.freq, sp.pres,
                            red64, cand_pen, cand_raw);
    if (n_row > 0 && nr > LOCAL_CAP)
      nr = exact_rounds<DT>(data, n_vec, n_el, lo, 1, n_row, penal, hbits, htab, P.hash_bits, sp.rep, sp.freq, sp.pres,
                            red64, cand_pen, cand_raw);

    // keep this chunk's best k_row / n_row and reserve their slice of the leader's lists
    const int sent_pen = min(np, k_row), sent_raw = min(nr, n_row);
    if (tid == 0) {
      const uint32_t ctl_leader = dsmem_addr(smem_u32(ctl), 0);
      ctl[CTL_BASE_P] = sent_pen > 0 ? dsmem_atomic_add(ctl_leader + 4u * CTL_RECV_NP, sent_pen) : 0u;
      ctl[CTL_BASE_R] = sent_raw > 0 ? dsmem_atomic_add(ctl_leader + 4u * CTL_RECV_NR, sent_raw) : 0u;
    }
    int out_p = -1, out_r = -1;
    uint4 ent_p = make_uint4(0, 0, 0, 0);
    uint64_t ent_r = 0ull;
    if (tid < np && k_row > 0) {
      ent_p = cand_pen[tid];
      out_p = tid;
      if (np > k_row) {
        const uint64_t ki = (static_cast<uint64_t>(ent_p.y) << 32) | ent_p.x;
        const uint2* keys = reinterpret_cast<const uint2*>(cand_pen);
        int rank = 0;
#pragma unroll 4
        for (int j = 0; j < np; ++j) {
          const uint2 o = keys[2 * j];
          rank += ((static_cast<uint64_t>(o.y) << 32) | o.x) > ki;
        }
        out_p = rank < k_row ? rank : -1;
      }
    }
    if (tid < nr && n_row > 0) {
      ent_r = cand_raw[tid];
      out_r = tid;
      if (nr > n_row) {
        int rank = 0;
#pragma unroll 4
        for (int j = 0; j < nr; ++j) rank += cand_raw[j] > ent_r;
        out_r = rank < n_row ? rank : -1;
      }
    }
    __syncthreads();
    if (out_p >= 0)
      dsmem_st_v4(dsmem_addr(smem_u32(sm + L.recv_pen) + (ctl[CTL_BASE_P] + out_p) * 16u, 0), ent_p.x, ent_p.y,
                  ent_p.z, 0u);
    if (out_r >= 0)
      dsmem_st_v2(dsmem_addr(smem_u32(sm + L.recv_raw) + (ctl[CTL_BASE_R] + out_r) * 8u, 0),
                  static_cast<uint32_t>(ent_r), static_cast<uint32_t>(ent_r >> 32));
    cluster_arrive();
    cluster_wait();  // B1: the leader holds every CTA's best candidates in two dense lists

    // ---- 4. the leader ranks the received keys exactly -----------------------------------------
    if (crank == 0) {
      const int tot_p = static_cast<int>(ctl[CTL_RECV_NP]);
      const int tot_r = static_cast<int>(ctl[CTL_RECV_NR]);
      uint4* sorted_pen = cand_pen;   // the leader's own candidates were sent before B1
      uint64_t* sorted_raw = reinterpret_cast<uint64_t*>(cand_pen + KMAX);
      const uint2* pkeys = reinterpret_cast<const uint2*>(recv_pen);
      if (tot_p <= 256 && tot_r <= 256) {
        // common case: warp 0 sorts the penalised list, warp 1 the raw list, each in registers;
        // no block barrier, each warp then reads its own sorted list back
        if (wid < 2) {
          const int n = wid == 0 ? tot_p : tot_r;
          const int need = wid == 0 ? k_row : n_row;
          if (n <= 128) {
            uint64_t kk[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int i = lane * 4 + r;
              kk[r] = i < n ? (wid == 0 ? ((static_cast<uint64_t>(pkeys[2 * i].y) << 32) | pkeys[2 * i].x) : recv_raw[i]) : 0ull;
            }
            warp_sort_desc<4>(kk, lane);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int i = lane * 4 + r;
              if (i < need && i < n) {
                if (wid == 0) sorted_pen[i] = make_uint4(static_cast<uint32_t>(kk[r]), static_cast<uint32_t>(kk[r] >> 32), 0u, 0u);
                else sorted_raw[i] = kk[r];
              }
            }
          } else {
            uint64_t kk[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const int i = lane * 8 + r;
              kk[r] = i < n ? (wid == 0 ? ((static_cast<uint64_t>(pkeys[2 * i].y) << 32) | pkeys[2 * i].x) : recv_raw[i]) : 0ull;
            }
            warp_sort_desc<8>(kk, lane);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const int i = lane * 8 + r;
              if (i < need && i < n) {
                if (wid == 0) sorted_pen[i] = make_uint4(static_cast<uint32_t>(kk[r]), static_cast<uint32_t>(kk[r] >> 32), 0u, 0u);
                else sorted_raw[i] = kk[r];
              }
            }
          }
          __syncwarp();
        }
      } else {
      uint32_t* hist = reinterpret_cast<uint32_t*>(cand_raw);            // 2 x 256 bins
      uint16_t* surv = reinterpret_cast<uint16_t*>(hist + 512);          // survivors of both lists
      // A long list is first cut by a threshold on the high key word: a 256-bin histogram of
      // (hi - T) over the list's range, scanned from the top, keeps the bin holding the
      // need-th largest value and everything above it (all of the top `need`, plus that bin).
      const bool cut_p = tot_p > max(2 * k_row, 32), cut_r = tot_r > max(2 * n_row, 32);
      const uint32_t Thi = T;
      if (cut_p || cut_r) {
        if (tid < 512 / 2) reinterpret_cast<uint2*>(hist)[tid] = make_uint2(0u, 0u);
        uint32_t mp = 0u, mr = 0u;
        for (int f = tid; f < tot_p; f += NT) mp = max(mp, pkeys[2 * f].y);
        for (int f = tid; f < tot_r; f += NT) mr = max(mr, static_cast<uint32_t>(recv_raw[f] >> 32));
        mp = __reduce_max_sync(FULL_MASK, mp);
        mr = __reduce_max_sync(FULL_MASK, mr);
        if (lane == 0) {
          atomicMax(&ctl[CTL_MAXP], mp);
          atomicMax(&ctl[CTL_MAXR], mr);
        }
        __syncthreads();
        const uint32_t span_p = ctl[CTL_MAXP] - Thi, span_r = ctl[CTL_MAXR] - Thi;
        const int sh_p = max(0, 32 - __clz(static_cast<int>(span_p | 1u)) - 8);
        const int sh_r = max(0, 32 - __clz(static_cast<int>(span_r | 1u)) - 8);
        if (cut_p)
          for (int f = tid; f < tot_p; f += NT) atomicAdd(&hist[(pkeys[2 * f].y - Thi) >> sh_p], 1u);
        if (cut_r)
          for (int f = tid; f < tot_r; f += NT) atomicAdd(&hist[256 + ((static_cast<uint32_t>(recv_raw[f] >> 32) - Thi) >> sh_r)], 1u);
        __syncthreads();
        if (wid < 2 && (wid == 0 ? cut_p : cut_r)) {  // warp 0: penalised list, warp 1: raw list
          const uint32_t* hh = hist + 256 * wid;
          const int need = wid == 0 ? k_row : n_row;
          uint32_t c[8], tsum = 0u;
#pragma unroll
          for (int j = 0; j < 8; ++j) {  // lane l holds bins 255-8l .. 248-8l (from the top)
            c[j] = hh[255 - (8 * lane + j)];
            tsum += c[j];
          }
          uint32_t incl = tsum;  // inclusive prefix over lanes = count in bins above this lane's
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const uint32_t y = __shfl_up_sync(FULL_MASK, incl, off);
            if (lane >= off) incl += y;
          }
          uint32_t run = incl - tsum;
          int bstar = -1;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            run += c[j];
            if (bstar < 0 && run >= static_cast<uint32_t>(need)) bstar = 255 - (8 * lane + j);
          }
          const uint32_t has = __ballot_sync(FULL_MASK, bstar >= 0);
          const int first = __ffs(has) - 1;  // lowest lane = highest bins
          const int b = __shfl_sync(FULL_MASK, bstar, first < 0 ? 0 : first);
          if (lane == 0) ctl[wid == 0 ? CTL_TP : CTL_TR] = first < 0 ? Thi : Thi + (static_cast<uint32_t>(b) << (wid == 0 ? sh_p : sh_r));
        }
        __syncthreads();
      }
      // survivors (indices into the received lists), then exact ranks among them; a cut that keeps
      // more than the survivor buffer holds (ties) is dropped and the whole list is ranked
      constexpr uint32_t SURV = 512;
      const uint32_t tp = cut_p ? ctl[CTL_TP] : 0u, tr = cut_r ? ctl[CTL_TR] : 0u;
      int n_sp = tot_p, n_sr = tot_r;
      bool use_sp = false, use_sr = false;
      if (cut_p || cut_r) {
        if (tid == 0) {
          ctl[CTL_BASE_P] = 0u;
          ctl[CTL_BASE_R] = 0u;
        }
        __syncthreads();
        for (int f0 = 0; f0 < max(tot_p, tot_r); f0 += NT) {
          const int f = f0 + tid;
          const bool kp_ = cut_p && f < tot_p && pkeys[2 * f].y >= tp;
          const bool kr_ = cut_r && f < tot_r && static_cast<uint32_t>(recv_raw[f] >> 32) >= tr;
          const uint32_t bp = __ballot_sync(FULL_MASK, kp_), br = __ballot_sync(FULL_MASK, kr_);
          uint32_t basep = 0, baser = 0;
          if (lane == 0) {
            if (bp) basep = atomicAdd(&ctl[CTL_BASE_P], static_cast<uint32_t>(__popc(bp)));
            if (br) baser = atomicAdd(&ctl[CTL_BASE_R], static_cast<uint32_t>(__popc(br)));
          }
          basep = __shfl_sync(FULL_MASK, basep, 0) + __popc(bp & ((1u << lane) - 1u));
          baser = __shfl_sync(FULL_MASK, baser, 0) + __popc(br & ((1u << lane) - 1u));
          if (kp_ && basep < SURV) surv[basep] = static_cast<uint16_t>(f);
          if (kr_ && baser < SURV) surv[SURV + baser] = static_cast<uint16_t>(f);
        }
        __syncthreads();
        use_sp = cut_p && ctl[CTL_BASE_P] <= SURV;
        use_sr = cut_r && ctl[CTL_BASE_R] <= SURV;
        if (use_sp) n_sp = static_cast<int>(ctl[CTL_BASE_P]);
        if (use_sr) n_sr = static_cast<int>(ctl[CTL_BASE_R]);
      }
      const int tot = n_sp + n_sr;
      int G = 1;  // threads per ranked key (a power of two)
      while (G < 32 && 2 * G * tot <= NT) G *= 2;
      for (int base = 0; base < tot; base += NT / G) {
        const int g = base + tid / G, sub = tid & (G - 1);
        int rank = 0;
        uint64_t ki = 0ull;
        int src = -1;
        if (g < n_sp) {
          src = use_sp ? surv[g] : g;
          const uint2 k2 = pkeys[2 * src];
          ki = (static_cast<uint64_t>(k2.y) << 32) | k2.x;
          for (int j = sub; j < n_sp; j += G) {
            const uint2 o = pkeys[2 * (use_sp ? surv[j] : j)];
            rank += ((static_cast<uint64_t>(o.y) << 32) | o.x) > ki;
          }
        } else if (g < tot) {
          src = use_sr ? surv[SURV + (g - n_sp)] : g - n_sp;
          ki = recv_raw[src];
          for (int j = sub; j < n_sr; j += G) rank += recv_raw[use_sr ? surv[SURV + j] : j] > ki;
        }
        for (int off = G >> 1; off > 0; off >>= 1) rank += __shfl_xor_sync(FULL_MASK, rank, off);
        if (sub == 0) {
          if (g < n_sp) {
            if (rank < k_row) sorted_pen[rank] = recv_pen[src];
          } else if (g < tot && rank < n_row) {
            sorted_raw[rank] = ki;
          }
        }
      }
      __syncthreads();
      }
      n_recv_p = tot_p;
      k_eff = min(k_row, tot_p);
      n_eff = min(n_row, tot_r);

      // the tail's first half on <= 64 survivors (one warp): min_p and top_p cuts and the
      // tempered cumulative weights; nothing here depends on the draw counter
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
          // temperature-1 mass (top_p) and tempered weights (draw) over the min_p survivors.
          // Prefix sums in fp32 decide unless a decision lies within 1e-5 of its boundary (the fp32
          // scan is good to ~4e-7 relative); then double-word sums (TwoSum) decide.
          const bool ina = lane < m1, inb = lane + 32 < m1;
          const float da = __fsub_rn(va, v0), db = __fsub_rn(vb, v0);
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
              const float tot = __shfl_sync(FULL_MASK, cb, 31);
              const float target = sp.top_p * tot, margin = 1e-5f * tot;
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
    }
  }

  // ---- outputs: with early loads the previous kernel owns outputs and counters until it ends --
  if (early) {
    grid_dep_wait();
    if (ctr_thread) ctr_old = atomicAdd(&P.ctr[slot], 1ull);
  }

  // allowed-subset log-probabilities and the given chosen id, for this chunk's ids
  if (P.allowed_off != nullptr && P.allowed_lps != nullptr) {
    auto out_allowed = [&](int j, int id) {
      if (id >= lo && id < hi) {
        P.allowed_lps[j] = elem_at<DT>(data, static_cast<uint32_t>(id - lo)) - lse_a;
      } else if ((id < 0 || id >= P.V) && crank == 0) {
        P.allowed_lps[j] = __int_as_float(0x7FC00000);
        atomicOr(P.err, STRATA_DEVERR_ALLOWED);
      }
    };
    if (a_beg + tid < a_end) out_allowed(a_beg + tid, aid[0]);
    if (a_beg + tid + NT < a_end) out_allowed(a_beg + tid + NT, aid[1]);
    for (int j = a_beg + tid + 2 * NT; j < a_end; j += NT) out_allowed(j, P.allowed[j]);
  }
  if (P.mode == MODE_LOGPROBS && P.chosen_lp != nullptr && P.chosen != nullptr && tid == 0) {
    if (chosen_id >= lo && chosen_id < hi) {
      P.chosen_lp[row] = elem_at<DT>(data, static_cast<uint32_t>(chosen_id - lo)) - lse;
    } else if ((chosen_id < 0 || chosen_id >= P.V) && crank == 0) {
      P.chosen_lp[row] = __int_as_float(0x7FC00000);
      atomicOr(P.err, STRATA_DEVERR_CHOSEN);
    }
  }

  if (kp > 0 && crank == 0) {
    const uint64_t* sorted_raw = reinterpret_cast<const uint64_t*>(cand_pen + KMAX);
    // top-N raw alternatives and their log-probabilities
    if (n_row > 0 && P.top_ids != nullptr && wid == 1) {  // warp 1 wrote the sorted raw list
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
      } else {
        int j = 0;
        if (sampled) {
          uint32_t x0 = 0u;
          if (ctr_thread) {
            if ((ctr_old & 0xFFFFull) + 1ull == static_cast<unsigned long long>(r_s))
              atomicAdd(&P.ctr[slot], (1ull << 16) - static_cast<unsigned long long>(r_s));
            x0 = philox_word0(sp.seed, pos, ctr_old >> 16);
          }
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
        if (P.chosen_lp != nullptr) {  // the raw logit travelled with the received entry
          const uint32_t kx = __shfl_sync(FULL_MASK, j < 32 ? ea.x : eb.x, j & 31);
          const uint32_t ky = __shfl_sync(FULL_MASK, j < 32 ? ea.y : eb.y, j & 31);
          for (int f0 = 0; f0 < n_recv_p; f0 += 32) {
            const int f = f0 + lane;
            const uint4 ent = f < n_recv_p ? recv_pen[f] : make_uint4(0, 0, 0, 0);
            const uint32_t bal = __ballot_sync(FULL_MASK, f < n_recv_p && ent.x == kx && ent.y == ky);
            if (bal != 0u) {
              chosen_raw = __shfl_sync(FULL_MASK, __uint_as_float(ent.z), __ffs(bal) - 1);
              break;
            }
          }
        }
      }
      if (lane == 0) {
        P.out_ids[row] = out;
        if (P.kept != nullptr) {
          P.kept[2 * row] = m1;
          P.kept[2 * row + 1] = m2;
        }
        if (P.chosen_lp != nullptr) P.chosen_lp[row] = (out >= 0) ? chosen_raw - lse : __int_as_float(0x7FC00000);
      }
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
  } else if (kp == 0 && P.mode == MODE_SAMPLE && crank == 0 && tid == 0) {
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
  if (P.mode == MODE_SAMPLE && valid && sp.k > P.kmax && crank == 0 && tid == 0) atomicOr(P.err, STRATA_DEVERR_SHAPE);
  if (ctl[CTL_TIMEOUT] != 0u) {  // a copy may still be in flight into this CTA: bounded wait again
    for (int p = 0; p < n_pieces; ++p) wait_piece(mbar, p, ctl, P.err);
  }
}

}  // namespace strata
