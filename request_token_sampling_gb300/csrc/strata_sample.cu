// strata_sample.cu -- host side of the C ABI declared in include/strata_sample.h.
//
// The context owns the device slot table (each request slot's prepared keys), one packed 64-bit
// word per slot holding its 48-bit draw counter and the 16-bit arrival count the kernel uses to
// advance it, and a device error word.  Keys are validated and prepared here (top_k 0 -> 20, logf(min_p) once on the host,
// penalty activity), mirrored on the host, and copied to the device on the caller's stream.
// On request (strata_history_enable) it also keeps each slot's run history on the device: a ring
// of the newest STRATA_HISTORY_CAP ids and a 64-bit length per slot, read and extended by the
// kernel itself.  Every sampling or logprobs call is one launch of the fused row kernel.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/strata_sample.h"
#include "strata_kernel.cuh"
#include "strata_merge.cuh"
#include "strata_resident.cuh"

using strata::KParams;
using strata::Layout;
using strata::SlotDev;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

// The kernel instance for a launch: streaming or resident chunk x logit type x allowed-id mask x
// own outputs; the streaming kernel's latency shape (`two`: few blocks, no call alongside) takes
// the instance whose registers are budgeted for two blocks per SM.
using KernelFn = void (*)(strata::KParams);
KernelFn kernel_for(int dtype, bool mask, bool own, bool resident = false, bool two = false) {
  static const KernelFn table[2][2][2][2] = {
      {{{strata::rows_kernel<0, false, false>, strata::rows_kernel<0, false, true>},
        {strata::rows_kernel<0, true, false>, strata::rows_kernel<0, true, true>}},
       {{strata::rows_kernel<1, false, false>, strata::rows_kernel<1, false, true>},
        {strata::rows_kernel<1, true, false>, strata::rows_kernel<1, true, true>}}},
      {{{strata::res_kernel<0, false, false>, strata::res_kernel<0, false, true>},
        {strata::res_kernel<0, true, false>, strata::res_kernel<0, true, true>}},
       {{strata::res_kernel<1, false, false>, strata::res_kernel<1, false, true>},
        {strata::res_kernel<1, true, false>, strata::res_kernel<1, true, true>}}}};
  static const KernelFn two_table[2][2] = {
      {strata::rows_kernel<0, false, false, 2>, strata::rows_kernel<0, true, false, 2>},
      {strata::rows_kernel<1, false, false, 2>, strata::rows_kernel<1, true, false, 2>}};
  if (two && !resident && !own) return two_table[dtype == STRATA_DTYPE_F32 ? 0 : 1][mask ? 1 : 0];
  return table[resident ? 1 : 0][dtype == STRATA_DTYPE_F32 ? 0 : 1][mask ? 1 : 0][own ? 1 : 0];
}

// Both kernels' instances may use up to `max_smem` of dynamic shared memory and non-portable
// cluster sizes (up to 16 blocks per row).
cudaError_t set_kernel_attributes(int max_smem) {
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 20 && e == cudaSuccess; ++i) {
    const void* k = reinterpret_cast<const void*>(
        i < 16 ? kernel_for(i & 1 ? STRATA_DTYPE_BF16 : STRATA_DTYPE_F32, (i >> 1) & 1, (i >> 2) & 1, (i >> 3) & 1)
               : kernel_for(i & 1 ? STRATA_DTYPE_BF16 : STRATA_DTYPE_F32, (i >> 1) & 1, false, false, true));
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem)) == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }
  return e;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(STRATA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Blocks per row.  Pipelined calls (early loads: the next call's loads overlap this one) are
// throughput-bound, so a row goes to few blocks that each stream up to PIPELINED_BYTES of logits
// (one stream of config-4 calls: 3.55 us per call over 20 calls and 2.37 over 200 with 4 blocks per
// row, against 4.06 and 3.26 with 8); otherwise a call is latency-bound, so rows split into blocks
// of about LATENCY_BYTES, enough of them to fill the GPU (but no block below MIN_CHUNK_ELEMS ids).
// With STRATA_FLAG_CONCURRENT a block streams up to STRATA_CONCURRENT_ROW_BYTES, or RING_BYTES for
// a call that keeps histories (it waits for the previous call before its penalties).
constexpr int PIPELINED_BYTES = 256 * 1024;
constexpr int RING_BYTES = 128 * 1024;
constexpr int LATENCY_BYTES = 64 * 1024;
constexpr int MIN_CHUNK_ELEMS = 2048;
constexpr int RING_SLOTS = 4;                 // pieces in flight per CTA when shared memory allows
// A pipelined call's blocks rescan their candidates through L1, and a fourth slot at three blocks
// per SM takes the shared-memory carveout to its maximum, which leaves L1 a fraction of its size:
// measured slower than three slots.  The same holds under the concurrency hint, where many calls
// stream at once: 20 calls over 8 groups ran 8-10 % faster with three slots than with four (the
// bytes in flight already saturate HBM; more only lengthen every other memory access's queue).
constexpr int RING_SLOTS_PIPELINED = 3;
constexpr int KEY_BINS = STRATA_MAX_TOP_K + 1;
constexpr int LASTN_BINS = STRATA_MAX_PENALTY_LAST_N + 1;

}  // namespace

struct strata_ctx {
  int device = 0;
  int num_sms = 0;
  int max_slots = 0, max_vocab = 0, max_rows = 0;
  int max_cluster = 8;
  int max_smem = 0;
  int smem_three = 0;  // the most dynamic shared memory per CTA that still fits three CTAs per SM
  SlotDev* d_slots = nullptr;
  unsigned long long* d_ctr = nullptr;
  uint32_t* d_done = nullptr;  // per slot: rows of the current verify call done (reset by the last)
  uint32_t* d_err = nullptr;
  int32_t* d_ring = nullptr;              // kept histories: STRATA_HISTORY_CAP ids per slot
  unsigned long long* d_hlen = nullptr;   // kept histories: per-slot total length
  std::vector<strata_sampling_params> h_params;
  std::vector<SlotDev> h_slots;
  // a sampling call that takes its draw counters after waiting for its predecessor was launched
  // with programmatic dependent launch, and may still be running: until a launch without PDL,
  // calls with own outputs take their counters that way too (so counters keep call order)
  bool late_counters_pending = false;
  // histograms over slots, for the launch shape: top_k of sampled slots, window of penal slots
  std::vector<int> k_bins, lastn_bins;
};

namespace {

SlotDev prepare(const strata_sampling_params& p) {
  SlotDev s{};
  const bool sampled = p.temperature > 0.0f;
  s.temperature = p.temperature;
  s.top_p = p.top_p;
  s.min_p = p.min_p;
  // "#19 ...", "min_p and the penalties": sel_logit >= sel_logit[0] + logf(min_p).  The host C
  // library's logf is evaluated once here so the device never computes it.
  s.logminp = p.min_p > 0.0f ? logf(p.min_p) : -INFINITY;
  s.rep = p.penalty_repeat;
  s.freq = p.penalty_freq;
  s.pres = p.penalty_present;
  s.k = sampled ? (p.top_k == 0 ? STRATA_DEFAULT_TOP_K : p.top_k) : 1;
  const bool neutral = p.penalty_repeat == 1.0f && p.penalty_freq == 0.0f && p.penalty_present == 0.0f;
  s.last_n = p.penalty_last_n;
  s.flags = (sampled ? strata::SLOT_SAMPLED : 0u) | ((!neutral && p.penalty_last_n > 0) ? strata::SLOT_PENAL : 0u);
  s.seed = p.seed;
  return s;
}

void bins_update(strata_ctx* c, const SlotDev& s, int delta) {
  if (s.flags & strata::SLOT_SAMPLED) c->k_bins[s.k] += delta;
  if (s.flags & strata::SLOT_PENAL) c->lastn_bins[s.last_n] += delta;
}

int max_k_sampled(const strata_ctx* c) {
  for (int k = STRATA_MAX_TOP_K; k >= 1; --k)
    if (c->k_bins[k] > 0) return k;
  return 0;
}

int max_lastn_penal(const strata_ctx* c) {
  for (int n = STRATA_MAX_PENALTY_LAST_N; n >= 1; --n)
    if (c->lastn_bins[n] > 0) return n;
  return 0;
}

int check_device(const strata_ctx* c) {
  int cur = -1;
  const cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != c->device) return fail(STRATA_EINVAL, "current device %d is not the context's device %d", cur, c->device);
  return STRATA_OK;
}

// Dynamic shared memory per CTA for three CTAs per SM, kept ~12 KB per SM below the largest
// shared-memory carveout: measured on GB300, a fourth 16 KiB ring slot that takes the carveout to
// its limit (and the L1 data cache down with it) costs more than the slot brings.
constexpr int SMEM_L1_MARGIN = 4 * 1024;
int smem_for_three(const cudaDeviceProp& prop) {
  const int per_sm = static_cast<int>(prop.sharedMemPerMultiprocessor);
  const int reserved = static_cast<int>(prop.reservedSharedMemPerBlock);
  return std::min(static_cast<int>(prop.sharedMemPerBlockOptin), per_sm / 3 - reserved - SMEM_L1_MARGIN) & ~127;
}

// Counter order under STRATA_FLAG_OWN_OUTPUTS.  A call that takes its counters after waiting for
// its predecessor relies on the chain of waits before it: the predecessor ended, and it had waited
// for its own predecessor, and so on.  A launch with own outputs waits for nothing and breaks that
// chain, so while a launch that takes its counters late may still be running (`pending`), every
// launch of the context (sampling or logprobs) drops the own-outputs bit and waits as usual.
uint32_t launch_flags(uint32_t flags, bool pending) { return pending ? flags & ~STRATA_FLAG_OWN_OUTPUTS : flags; }
// The pending state after a launch with `flags` (as launched; `sampling`: it takes counters).  A
// sampling launch that takes its counters late leaves them pending, PDL or not: the kernel lets
// the next launch start at its entry.  Otherwise a launch without PDL started after all earlier
// work had ended, and one with PDL leaves the state as it was.
bool pending_after(bool pending, uint32_t flags, bool sampling) {
  const bool early_counters = (flags & STRATA_FLAG_OWN_OUTPUTS) != 0u && (flags & STRATA_FLAG_EARLY_LOAD) != 0u;
  if (sampling && !early_counters) return true;
  return (flags & STRATA_FLAG_PDL) != 0u && pending;
}

struct Shape {
  int cs, chunk, smem, kmax, nmax, hash_cap, hash_bits, nslot, qw;
  bool resident;  // the chunk is held whole in shared memory (res_kernel); else it streams
  bool two;       // the latency shape: the instance with registers for two blocks per SM
};

// Keys each warp of a resident block publishes for the row's threshold: enough that the row's
// blocks together publish about 2 * kp of them (a power of two, at most RES_QW_MAX per warp).
int res_qw(int kp, int cs) {
  int qw = 1;
  while (qw < strata::RES_QW_MAX && cs * strata::NW * qw < 2 * kp) qw *= 2;
  return qw;
}

// The launch shape of a call: blocks per row (one cluster), the chunk each streams, ring slots,
// keys each warp publishes for the row threshold, history table size and shared memory.  Shared
// by the context calls and the allocation-free call.
int shape_for(int max_cluster, int max_smem, int smem_three, int num_sms, int mode, int esz, int B, int V, int kmax,
              int nmax, int lastn_max, bool with_hist, bool with_allowed, bool mask, bool pipelined,
              int concurrent_bytes, int forced, Shape* s, bool streaming = true) {
  const bool concurrent = concurrent_bytes > 0;
  const long long row_bytes = static_cast<long long>(V) * esz;
  s->nmax = nmax;
  s->kmax = kmax;
  const int kp_max = std::max(kmax, nmax);
  int cs;
  if (forced > 0) {
    if (forced > max_cluster) return fail(STRATA_ERANGE, "forced split %d above the cluster limit %d", forced, max_cluster);
    cs = forced;
  } else if (concurrent) {
    cs = static_cast<int>((row_bytes + concurrent_bytes - 1) / concurrent_bytes);
    cs = std::min(std::max(cs, 1), max_cluster);
  } else if (pipelined) {
    cs = static_cast<int>((row_bytes + PIPELINED_BYTES - 1) / PIPELINED_BYTES);
    cs = std::min(std::max(cs, 1), max_cluster);
  } else {
    const int cs_bytes = static_cast<int>((row_bytes + LATENCY_BYTES - 1) / LATENCY_BYTES);
    const int cs_fill = (num_sms + B - 1) / std::max(1, B);
    const int cs_small = std::max(1, (V + MIN_CHUNK_ELEMS - 1) / MIN_CHUNK_ELEMS);
    cs = std::max({cs_bytes, std::min(cs_fill, cs_small), 1});
    cs = std::min(cs, max_cluster);
  }
  s->hash_cap = 0;
  s->hash_bits = 0;
  s->resident = false;
  // the register budget: two blocks per SM (no spills) unless calls of other groups stream alongside
  s->two = !concurrent;
  if (mode == strata::MODE_SAMPLE && with_hist && lastn_max > 0) {
    int bits = 6;
    while ((1 << bits) < 2 * lastn_max) ++bits;
    s->hash_bits = bits;
    s->hash_cap = 1 << bits;
  }
  // The resident shape: every block holds its chunk whole (at most RES_MAX_CHUNK_BYTES).  Latency-
  // bound calls spread a row over enough blocks to fill the GPU; with the concurrency hint a row
  // takes the fewest blocks that hold it.  A forced split is resident when its chunks fit.
  if (!streaming) {
    const int cs_min = static_cast<int>((row_bytes + strata::RES_MAX_CHUNK_BYTES - 1) / strata::RES_MAX_CHUNK_BYTES);
    int rcs = 0;
    if (forced > 0) {
      if (forced >= cs_min && forced <= max_cluster) rcs = forced;
    } else if (cs_min <= max_cluster) {
      if (concurrent) {
        rcs = std::max(cs_min, 1);
      } else {
        const int cs_fill = (num_sms + B - 1) / std::max(1, B);
        const int cs_small = std::max(1, (V + MIN_CHUNK_ELEMS - 1) / MIN_CHUNK_ELEMS);
        rcs = std::min(std::max({cs_min, std::min(cs_fill, cs_small), 1}), max_cluster);
      }
    }
    if (rcs > 0) {
      int chunk = (V + rcs - 1) / rcs;
      chunk = (chunk + 15) / 16 * 16;
      const int rqw = res_qw(kp_max, rcs);
      const strata::RLayout RL = strata::make_res_layout(chunk, esz, s->hash_cap, rcs, kmax, nmax, rqw, with_allowed, mask);
      if (static_cast<long long>(chunk) * esz <= strata::RES_MAX_CHUNK_BYTES && static_cast<int>(RL.total) <= max_smem) {
        if (!strata::res_layout_aligned(RL)) return fail(STRATA_EINVAL, "internal: shared-memory layout not 16-byte aligned");
        s->resident = true;
        s->cs = rcs;
        s->chunk = chunk;
        s->qw = rqw;
        s->nslot = (chunk * esz + strata::PIECE_BYTES - 1) / strata::PIECE_BYTES;
        s->smem = static_cast<int>(RL.total);
        return STRATA_OK;
      }
    }
  }
  Layout L{};
  for (;;) {
    int chunk = (V + cs - 1) / cs;
    chunk = (chunk + 15) / 16 * 16;
    s->cs = cs;
    s->chunk = chunk;
    // keys per warp: enough that the row publishes about 2 * kp of them (a tight threshold)
    const int per_warp = (2 * kp_max + cs * strata::NW - 1) / (cs * strata::NW);
    int qw = 1;
    while (qw < per_warp && qw < strata::QW_MAX) qw *= 2;
    s->qw = qw;
    // the most ring slots that still leave room for three CTAs on the SM (at least 2)
    for (int ns = (pipelined || concurrent) ? RING_SLOTS_PIPELINED : RING_SLOTS; ns >= 2; --ns) {
      L = strata::make_layout(chunk, s->hash_cap, cs, kmax, nmax, ns, s->qw, with_allowed, mask);
      s->nslot = ns;
      if (static_cast<int>(L.total) <= smem_three) break;
    }
    // a chunk whose id bitmaps do not fit the block's shared memory: split the row further
    if (static_cast<int>(L.total) <= max_smem || forced > 0 || cs >= max_cluster) break;
    ++cs;
  }
  if (!strata::layout_aligned(L)) return fail(STRATA_EINVAL, "internal: shared-memory layout not 16-byte aligned");
  if (L.cand_cap < cs * std::max(kmax, nmax) + 8) return fail(STRATA_EINVAL, "internal: candidate lists too small");
  s->smem = static_cast<int>(L.total);
  if (s->smem > max_smem) return fail(STRATA_ERANGE, "shared memory %d above the device limit %d", s->smem, max_smem);
  return STRATA_OK;
}

int compute_shape(const strata_ctx* c, int mode, int dtype, int B, int V, int top_n_eff, bool with_hist,
                  bool with_allowed, uint32_t flags, Shape* s, bool verify = false) {
  const int esz = dtype == STRATA_DTYPE_F32 ? 4 : 2;
  const int kmax = mode == strata::MODE_SAMPLE ? std::max(1, max_k_sampled(c)) : 0;
  const bool mask = mode == strata::MODE_SAMPLE && with_allowed && (flags & STRATA_FLAG_ALLOWED_MASK) != 0u;
  // verify windows and calls that read kept histories are steps of one request's decode (the
  // latter wait for the previous call before their penalties): they take the latency split
  const bool pipelined = (flags & STRATA_FLAG_PDL) != 0u && (flags & STRATA_FLAG_EARLY_LOAD) != 0u &&
                         (flags & STRATA_FLAG_HISTORY_RING) == 0u && !verify;
  // the concurrency hint: a block streams up to STRATA_CONCURRENT_ROW_BYTES; a call that keeps
  // histories waits for the previous call before its penalties and takes RING_BYTES (measured
  // with 8 groups in flight: these were the fastest of the splits tried)
  int concurrent_bytes = 0;
  if ((flags & STRATA_FLAG_CONCURRENT) != 0u)
    concurrent_bytes = (flags & STRATA_FLAG_HISTORY_RING) != 0u ? RING_BYTES
                                                                : static_cast<int>(STRATA_CONCURRENT_ROW_BYTES);
  return shape_for(c->max_cluster, c->max_smem, c->smem_three, c->num_sms, mode, esz, B, V, kmax, top_n_eff,
                   max_lastn_penal(c),
                   with_hist, with_allowed, mask, pipelined, concurrent_bytes,
                   static_cast<int>((flags >> 8) & 0x1Fu), s, (flags & STRATA_FLAG_RESIDENT) == 0u);
}

// STRATA_SAMPLE_DEBUG=1 in the environment: one line per call on stderr (entry point, rows,
// vocabulary, flags and the launch shape chosen).  Read once per process.
bool trace_on() {
  static const bool on = [] {
    const char* v = std::getenv("STRATA_SAMPLE_DEBUG");
    return v != nullptr && v[0] != '\0' && v[0] != '0';
  }();
  return on;
}

int launch(strata_ctx* c, const KParams& P, int dtype, const Shape& sh, uint32_t flags, cudaStream_t stream,
           const char* entry) {
  if (trace_on())
    std::fprintf(stderr,
                 "strata: %s B=%d V=%d dtype=%s flags=0x%x kernel=%s split=%d chunk=%d ring_slots=%d qw=%d hash=%d "
                 "smem=%d grid=%d\n",
                 entry, P.B, P.V, dtype == STRATA_DTYPE_F32 ? "f32" : "bf16", flags,
                 sh.resident ? "resident" : sh.two ? "streaming-2" : "streaming", sh.cs, sh.chunk, sh.nslot, sh.qw, sh.hash_cap, sh.smem,
                 P.B * sh.cs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(P.B * sh.cs), 1, 1);
  cfg.blockDim = dim3(strata::NT, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(sh.smem);
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = static_cast<unsigned>(sh.cs);
  attrs[na].val.clusterDim.y = 1;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  if (flags & STRATA_FLAG_PDL) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  cudaError_t e;
  const bool mask = P.mode == strata::MODE_SAMPLE && (flags & STRATA_FLAG_ALLOWED_MASK) != 0u && P.allowed_off != nullptr;
  const bool own = (flags & STRATA_FLAG_OWN_OUTPUTS) != 0u && (flags & STRATA_FLAG_EARLY_LOAD) != 0u;
  e = cudaLaunchKernelEx(&cfg, kernel_for(dtype, mask, own, sh.resident, sh.two), P);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  (void)c;
  return STRATA_OK;
}

int check_rows_common(const strata_ctx* c, const void* logits, int dtype, int B, int V, int64_t ld, int top_n,
                      const float* chosen_lp, const int32_t* top_ids, const float* top_lps,
                      const int32_t* allowed, const int32_t* allowed_off, const float* allowed_lps) {
  if (c == nullptr) return fail(STRATA_EINVAL, "null context");
  if (dtype != STRATA_DTYPE_F32 && dtype != STRATA_DTYPE_BF16) return fail(STRATA_EINVAL, "dtype %d", dtype);
  if (B < 0) return fail(STRATA_EINVAL, "B=%d", B);
  if (B > c->max_rows) return fail(STRATA_ERANGE, "B=%d above max_rows %d", B, c->max_rows);
  if (V < 1) return fail(STRATA_EINVAL, "V=%d", V);
  if (V > c->max_vocab) return fail(STRATA_ERANGE, "V=%d above max_vocab %d", V, c->max_vocab);
  if (ld < V) return fail(STRATA_EINVAL, "ld=%lld below V=%d", static_cast<long long>(ld), V);
  if (top_n < 0 || top_n > STRATA_MAX_TOP_N) return fail(STRATA_EINVAL, "top_n=%d outside 0..%d", top_n, STRATA_MAX_TOP_N);
  if (B > 0 && logits == nullptr) return fail(STRATA_EINVAL, "null logits");
  const int esz = dtype == STRATA_DTYPE_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) != 0) return fail(STRATA_EALIGN, "logits not 16-byte aligned");
  if ((static_cast<long long>(ld) * esz) % 16 != 0) return fail(STRATA_EALIGN, "row stride of %lld bytes not a multiple of 16", static_cast<long long>(ld) * esz);
  if (top_n > 0 && ((top_ids == nullptr) != (top_lps == nullptr)))
    return fail(STRATA_EINVAL, "top_ids and top_lps must be given together");
  if (allowed_off != nullptr && (allowed == nullptr || allowed_lps == nullptr))
    return fail(STRATA_EINVAL, "allowed_off needs allowed and allowed_lps");
  (void)chosen_lp;
  return STRATA_OK;
}

}  // namespace

extern "C" {

int strata_version(void) { return 10000; }

const char* strata_last_error(void) { return g_err; }

void strata_default_params(strata_sampling_params* p) {
  if (p == nullptr) return;
  std::memset(p, 0, sizeof(*p));
  p->struct_size = sizeof(strata_sampling_params);
  p->temperature = 0.0f;
  p->top_k = 0;
  p->top_p = 1.0f;
  p->min_p = 0.0f;
  p->penalty_repeat = 1.0f;
  p->penalty_freq = 0.0f;
  p->penalty_present = 0.0f;
  p->penalty_last_n = STRATA_DEFAULT_LAST_N;
  p->seed = 0;
}

int strata_validate_params(const strata_sampling_params* p) {
  if (p == nullptr) return fail(STRATA_EINVAL, "null params");
  if (p->struct_size < sizeof(strata_sampling_params))
    return fail(STRATA_EINVAL, "struct_size %u below %zu", p->struct_size, sizeof(strata_sampling_params));
  const float fs[6] = {p->temperature, p->top_p, p->min_p, p->penalty_repeat, p->penalty_freq, p->penalty_present};
  const char* names[6] = {"temperature", "top_p", "min_p", "penalty_repeat", "penalty_freq", "penalty_present"};
  for (int i = 0; i < 6; ++i)
    if (!std::isfinite(fs[i])) return fail(STRATA_EINVAL, "%s is not finite", names[i]);
  if (p->top_k < 0 || p->top_k > STRATA_MAX_TOP_K)
    return fail(STRATA_EINVAL, "top_k=%d outside 0..%d (0 means %d)", p->top_k, STRATA_MAX_TOP_K, STRATA_DEFAULT_TOP_K);
  if (!(p->penalty_repeat > 0.0f)) return fail(STRATA_EINVAL, "penalty_repeat must be > 0");
  if (p->min_p < 0.0f) return fail(STRATA_EINVAL, "min_p must be >= 0");
  if (p->penalty_last_n < 0 || p->penalty_last_n > STRATA_MAX_PENALTY_LAST_N)
    return fail(STRATA_EINVAL, "penalty_last_n=%d outside 0..%d", p->penalty_last_n, STRATA_MAX_PENALTY_LAST_N);
  if (p->reserved != 0u) return fail(STRATA_EINVAL, "reserved field must be 0");
  return STRATA_OK;
}

int strata_create(strata_ctx** out, int device, int max_slots, int max_vocab, int max_rows) {
  if (out == nullptr) return fail(STRATA_EINVAL, "null output pointer");
  *out = nullptr;
  if (max_slots < 1 || max_slots > 65536) return fail(STRATA_EINVAL, "max_slots=%d outside 1..65536", max_slots);
  if (max_vocab < 1 || max_vocab > STRATA_MAX_VOCAB) return fail(STRATA_EINVAL, "max_vocab=%d outside 1..%d", max_vocab, STRATA_MAX_VOCAB);
  if (max_rows < 1 || max_rows > 65535) return fail(STRATA_EINVAL, "max_rows=%d outside 1..65535", max_rows);
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device < 0 || device >= ndev) return fail(STRATA_EINVAL, "device %d of %d", device, ndev);
  int cur = -1;
  if ((e = cudaGetDevice(&cur)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != device) return fail(STRATA_EINVAL, "device %d is not the calling thread's current device %d", device, cur);
  cudaDeviceProp prop;
  if ((e = cudaGetDeviceProperties(&prop, device)) != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (prop.major < 10) return fail(STRATA_ECUDA, "device %s (sm_%d%d) is not a Blackwell GPU", prop.name, prop.major, prop.minor);

  strata_ctx* c = new (std::nothrow) strata_ctx();
  if (c == nullptr) return fail(STRATA_ENOMEM, "host allocation");
  c->device = device;
  c->num_sms = prop.multiProcessorCount;
  c->max_slots = max_slots;
  c->max_vocab = max_vocab;
  c->max_rows = max_rows;
  c->max_smem = static_cast<int>(prop.sharedMemPerBlockOptin);
  c->smem_three = smem_for_three(prop);
  c->k_bins.assign(KEY_BINS, 0);
  c->lastn_bins.assign(LASTN_BINS, 0);

  auto cleanup = [&](int code) {
    strata_destroy(c);
    return code;
  };
  if ((e = set_kernel_attributes(c->max_smem)) != cudaSuccess) return cleanup(cuda_fail(e, "cudaFuncSetAttribute"));
  // The largest cluster the device can place with a typical shared-memory footprint.
  c->max_cluster = 8;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(strata::MAX_CS, 1, 1);
    cfg.blockDim = dim3(strata::NT, 1, 1);
    cfg.dynamicSmemBytes = 128 * 1024;
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = strata::MAX_CS;
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, strata::rows_kernel<0, false>, &cfg) == cudaSuccess && nclusters > 0)
      c->max_cluster = strata::MAX_CS;
    cudaGetLastError();
  }

  c->h_params.resize(max_slots);
  c->h_slots.resize(max_slots);
  strata_sampling_params d;
  strata_default_params(&d);
  const SlotDev sd = prepare(d);
  for (int i = 0; i < max_slots; ++i) {
    c->h_params[i] = d;
    c->h_slots[i] = sd;
  }
  if ((e = cudaMalloc(&c->d_slots, sizeof(SlotDev) * max_slots)) != cudaSuccess) return cleanup(fail(STRATA_ENOMEM, "cudaMalloc slots: %s", cudaGetErrorString(e)));
  if ((e = cudaMalloc(&c->d_ctr, sizeof(unsigned long long) * max_slots)) != cudaSuccess) return cleanup(fail(STRATA_ENOMEM, "cudaMalloc counters: %s", cudaGetErrorString(e)));
  if ((e = cudaMalloc(&c->d_err, sizeof(uint32_t))) != cudaSuccess) return cleanup(fail(STRATA_ENOMEM, "cudaMalloc error word: %s", cudaGetErrorString(e)));
  if ((e = cudaMalloc(&c->d_done, sizeof(uint32_t) * max_slots)) != cudaSuccess) return cleanup(fail(STRATA_ENOMEM, "cudaMalloc window words: %s", cudaGetErrorString(e)));
  if ((e = cudaMemset(c->d_done, 0, sizeof(uint32_t) * max_slots)) != cudaSuccess) return cleanup(cuda_fail(e, "window word reset"));
  if ((e = cudaMemcpy(c->d_slots, c->h_slots.data(), sizeof(SlotDev) * max_slots, cudaMemcpyHostToDevice)) != cudaSuccess) return cleanup(cuda_fail(e, "slot table upload"));
  if ((e = cudaMemset(c->d_ctr, 0, sizeof(unsigned long long) * max_slots)) != cudaSuccess) return cleanup(cuda_fail(e, "counter reset"));
  if ((e = cudaMemset(c->d_err, 0, sizeof(uint32_t))) != cudaSuccess) return cleanup(cuda_fail(e, "error word reset"));
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cleanup(cuda_fail(e, "create sync"));
  *out = c;
  return STRATA_OK;
}

void strata_destroy(strata_ctx* c) {
  if (c == nullptr) return;
  cudaDeviceSynchronize();
  cudaFree(c->d_slots);
  cudaFree(c->d_ctr);
  cudaFree(c->d_done);
  cudaFree(c->d_err);
  cudaFree(c->d_ring);
  cudaFree(c->d_hlen);
  delete c;
}

// ---- kept per-slot histories: slot s's id number i (0-based over its run) lives at
// d_ring[s * STRATA_HISTORY_CAP + i % STRATA_HISTORY_CAP] while it is among the newest CAP ids.
int strata_history_enable(strata_ctx* c) {
  if (c == nullptr) return fail(STRATA_EINVAL, "null context");
  int rc = check_device(c);
  if (rc != STRATA_OK) return rc;
  if (c->d_ring != nullptr) return STRATA_OK;
  const size_t ring_bytes = sizeof(int32_t) * STRATA_HISTORY_CAP * static_cast<size_t>(c->max_slots);
  cudaError_t e;
  if ((e = cudaMalloc(&c->d_ring, ring_bytes)) != cudaSuccess) {
    c->d_ring = nullptr;
    return fail(STRATA_ENOMEM, "cudaMalloc histories (%zu bytes): %s", ring_bytes, cudaGetErrorString(e));
  }
  if ((e = cudaMalloc(&c->d_hlen, sizeof(unsigned long long) * c->max_slots)) != cudaSuccess) {
    cudaFree(c->d_ring);
    c->d_ring = nullptr;
    c->d_hlen = nullptr;
    return fail(STRATA_ENOMEM, "cudaMalloc history lengths: %s", cudaGetErrorString(e));
  }
  if ((e = cudaMemset(c->d_hlen, 0, sizeof(unsigned long long) * c->max_slots)) != cudaSuccess ||
      (e = cudaDeviceSynchronize()) != cudaSuccess) {
    cudaFree(c->d_ring);
    cudaFree(c->d_hlen);
    c->d_ring = nullptr;
    c->d_hlen = nullptr;
    return cuda_fail(e, "history reset");
  }
  return STRATA_OK;
}

static int history_check(strata_ctx* c, int slot) {
  if (c == nullptr) return fail(STRATA_EINVAL, "null context");
  if (slot < 0 || slot >= c->max_slots) return fail(STRATA_ERANGE, "slot %d outside 0..%d", slot, c->max_slots - 1);
  if (c->d_ring == nullptr) return fail(STRATA_EINVAL, "histories not enabled (strata_history_enable)");
  return check_device(c);
}

int strata_history_set(strata_ctx* c, int slot, const int32_t* ids, int64_t n, void* stream) {
  int rc = history_check(c, slot);
  if (rc != STRATA_OK) return rc;
  if (n < 0) return fail(STRATA_EINVAL, "n=%lld", static_cast<long long>(n));
  if (n > 0 && ids == nullptr) return fail(STRATA_EINVAL, "null ids");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t cap = STRATA_HISTORY_CAP;
  const int64_t m = std::min(n, cap);
  int32_t* ring = c->d_ring + static_cast<size_t>(slot) * STRATA_HISTORY_CAP;
  // ids n-m .. n-1 go to ring positions (n-m) % cap onward, wrapping once at most
  const int64_t first = (n - m) % cap;
  const int64_t run1 = std::min(m, cap - first);
  // staged in pageable memory, so that the caller's array is free again when the call returns
  // (a page-locked source would be read later, by the copy engine)
  std::vector<int32_t> stage(ids + (n - m), ids + n);
  cudaError_t e;
  if (run1 > 0 && (e = cudaMemcpyAsync(ring + first, stage.data(), sizeof(int32_t) * run1, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "history upload");
  if (m > run1 && (e = cudaMemcpyAsync(ring, stage.data() + run1, sizeof(int32_t) * (m - run1), cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "history upload");
  const unsigned long long len = static_cast<unsigned long long>(n);
  if ((e = cudaMemcpyAsync(c->d_hlen + slot, &len, sizeof(len), cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "history length upload");
  return STRATA_OK;
}

int strata_history_get(strata_ctx* c, int slot, int32_t* ids, int max_n, int* n_out, int64_t* length, void* stream) {
  int rc = history_check(c, slot);
  if (rc != STRATA_OK) return rc;
  if (max_n < 0) return fail(STRATA_EINVAL, "max_n=%d", max_n);
  if (max_n > 0 && ids == nullptr) return fail(STRATA_EINVAL, "null ids");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long len = 0;
  cudaError_t e = cudaMemcpyAsync(&len, c->d_hlen + slot, sizeof(len), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "history length read");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "history length sync");
  const int64_t cap = STRATA_HISTORY_CAP;
  const int64_t n = static_cast<int64_t>(len);
  const int64_t m = std::min({n, cap, static_cast<int64_t>(max_n)});
  const int32_t* ring = c->d_ring + static_cast<size_t>(slot) * STRATA_HISTORY_CAP;
  const int64_t first = (n - m) % cap;
  const int64_t run1 = std::min(m, cap - first);
  if (run1 > 0 && (e = cudaMemcpyAsync(ids, ring + first, sizeof(int32_t) * run1, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "history read");
  if (m > run1 && (e = cudaMemcpyAsync(ids + run1, ring, sizeof(int32_t) * (m - run1), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "history read");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "history read sync");
  if (n_out != nullptr) *n_out = static_cast<int>(m);
  if (length != nullptr) *length = n;
  return STRATA_OK;
}

static int set_slot(strata_ctx* c, int slot, const strata_sampling_params* p, bool set_ctr, uint64_t ctr,
                    void* stream) {
  if (c == nullptr) return fail(STRATA_EINVAL, "null context");
  if (slot < 0 || slot >= c->max_slots) return fail(STRATA_ERANGE, "slot %d outside 0..%d", slot, c->max_slots - 1);
  if (set_ctr && ctr >= (1ull << 48)) return fail(STRATA_ERANGE, "counter %llu needs more than 48 bits", static_cast<unsigned long long>(ctr));
  int rc = strata_validate_params(p);
  if (rc != STRATA_OK) return rc;
  if ((rc = check_device(c)) != STRATA_OK) return rc;
  strata_sampling_params q = *p;
  q.struct_size = sizeof(strata_sampling_params);
  const SlotDev sd = prepare(q);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(c->d_slots + slot, &sd, sizeof(SlotDev), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "slot upload");
  if (set_ctr) {
    const unsigned long long v = static_cast<unsigned long long>(ctr) << 16;  // arrivals cleared
    if ((e = cudaMemcpyAsync(c->d_ctr + slot, &v, sizeof(v), cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return cuda_fail(e, "counter upload");
  }
  bins_update(c, c->h_slots[slot], -1);
  c->h_slots[slot] = sd;
  c->h_params[slot] = q;
  bins_update(c, sd, +1);
  return STRATA_OK;
}

int strata_set_slot_params(strata_ctx* c, int slot, const strata_sampling_params* p, int reset_counter,
                           void* stream) {
  return set_slot(c, slot, p, reset_counter != 0, 0ull, stream);
}

int strata_set_slot_state(strata_ctx* c, int slot, const strata_sampling_params* p, uint64_t counter,
                          void* stream) {
  return set_slot(c, slot, p, true, counter, stream);
}

int strata_get_slot_state(strata_ctx* c, int slot, strata_sampling_params* p, uint64_t* counter, void* stream) {
  if (c == nullptr) return fail(STRATA_EINVAL, "null context");
  if (slot < 0 || slot >= c->max_slots) return fail(STRATA_ERANGE, "slot %d outside 0..%d", slot, c->max_slots - 1);
  int rc = check_device(c);
  if (rc != STRATA_OK) return rc;
  if (p != nullptr) *p = c->h_params[slot];
  if (counter != nullptr) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned long long v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, c->d_ctr + slot, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "counter read");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "counter read sync");
    *counter = v >> 16;
  }
  return STRATA_OK;
}

int strata_read_errors(strata_ctx* c, uint32_t* bits, void* stream) {
  if (c == nullptr || bits == nullptr) return fail(STRATA_EINVAL, "null argument");
  int rc = check_device(c);
  if (rc != STRATA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, c->d_err, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "error word read");
  if ((e = cudaMemsetAsync(c->d_err, 0, sizeof(uint32_t), s)) != cudaSuccess) return cuda_fail(e, "error word clear");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "error word sync");
  *bits = v;
  c->late_counters_pending = false;  // the stream has drained
  return STRATA_OK;
}

int strata_launch_shape(strata_ctx* c, int mode, int dtype, int B, int V, int top_n, uint32_t flags, int* split,
                        int* chunk_elems, int* smem_bytes, int* grid) {
  if (c == nullptr) return fail(STRATA_EINVAL, "null context");
  const bool verify = mode == 2;  // strata_sample_verify
  if (mode != strata::MODE_SAMPLE && mode != strata::MODE_LOGPROBS && !verify) return fail(STRATA_EINVAL, "mode %d", mode);
  if (dtype != STRATA_DTYPE_F32 && dtype != STRATA_DTYPE_BF16) return fail(STRATA_EINVAL, "dtype %d", dtype);
  if (B < 1 || V < 1 || V > c->max_vocab || top_n < 0 || top_n > STRATA_MAX_TOP_N) return fail(STRATA_EINVAL, "shape");
  Shape sh;
  const int rc = compute_shape(c, verify ? strata::MODE_SAMPLE : mode, dtype, B, V, top_n, true, false, flags, &sh,
                               verify);
  if (rc != STRATA_OK) return rc;
  if (split) *split = sh.cs;
  if (chunk_elems) *chunk_elems = sh.chunk;
  if (smem_bytes) *smem_bytes = sh.smem;
  if (grid) *grid = B * sh.cs;
  return STRATA_OK;
}

static int sample_rows_impl(strata_ctx* c, const void* logits, int dtype, int B, int V, int64_t ld,
                            const int32_t* row_slot, const int64_t* row_pos, const int32_t* row_draft,
                            const int32_t* hist, const int32_t* hist_off, int n_hist_slots, int32_t* out_ids,
                            int32_t* slot_keep, int top_n, float* chosen_lp, int32_t* top_ids, float* top_lps,
                            const int32_t* allowed, const int32_t* allowed_off, float* allowed_lps, int32_t* topk_ids,
                            float* topk_vals, int32_t* kept, uint32_t flags, void* stream) {
  int rc = check_rows_common(c, logits, dtype, B, V, ld, top_n, chosen_lp, top_ids, top_lps, allowed, allowed_off,
                             allowed_lps);
  if (rc != STRATA_OK) return rc;
  if (B > 0 && (row_slot == nullptr || row_pos == nullptr || out_ids == nullptr))
    return fail(STRATA_EINVAL, "row_slot, row_pos and out_ids are required");
  const bool kept_hist = (flags & STRATA_FLAG_HISTORY_RING) != 0u;
  if (kept_hist) {
    if (hist != nullptr || hist_off != nullptr)
      return fail(STRATA_EINVAL, "STRATA_FLAG_HISTORY_RING takes the windows from the kept histories: hist and hist_off must be NULL");
    if (c->d_ring == nullptr) return fail(STRATA_EINVAL, "STRATA_FLAG_HISTORY_RING before strata_history_enable");
  }
  if (hist_off != nullptr && (hist == nullptr || n_hist_slots < 1))
    return fail(STRATA_EINVAL, "hist_off needs hist and n_hist_slots >= 1");
  if ((flags & STRATA_FLAG_OWN_OUTPUTS) != 0u && (kept_hist || row_draft != nullptr))
    return fail(STRATA_EINVAL, "STRATA_FLAG_OWN_OUTPUTS is for plain sampling calls (no verify windows, no kept histories)");
  if (hist_off == nullptr) n_hist_slots = 0;
  if ((rc = check_device(c)) != STRATA_OK) return rc;
  if (B == 0) return STRATA_OK;
  const int top_n_eff = (top_n > 0 && top_ids != nullptr) ? top_n : 0;
  Shape sh;
  if ((rc = compute_shape(c, strata::MODE_SAMPLE, dtype, B, V, top_n_eff, hist_off != nullptr || kept_hist,
                          allowed_off != nullptr, flags, &sh, row_draft != nullptr)) != STRATA_OK)
    return rc;
  KParams P{};
  P.logits = logits;
  P.ld = ld;
  P.B = B;
  P.V = V;
  P.cs = sh.cs;
  P.chunk = sh.chunk;
  P.mode = strata::MODE_SAMPLE;
  P.row_slot = row_slot;
  P.row_pos = reinterpret_cast<const long long*>(row_pos);
  P.hist = hist;
  P.hist_off = hist_off;
  P.n_hist_slots = n_hist_slots;
  P.out_ids = out_ids;
  P.top_n = top_n;
  P.nmax = sh.nmax;
  P.kmax = sh.kmax;
  P.chosen_lp = chosen_lp;
  P.top_ids = top_n_eff > 0 ? top_ids : nullptr;
  P.top_lps = top_n_eff > 0 ? top_lps : nullptr;
  P.chosen = nullptr;
  P.allowed = allowed;
  P.allowed_off = allowed_off;
  P.allowed_lps = allowed_lps;
  P.topk_ids = topk_ids;
  P.topk_vals = topk_vals;
  P.kept = kept;
  P.slots = c->d_slots;
  P.ctr = c->d_ctr;
  P.max_slots = c->max_slots;
  P.err = c->d_err;
  P.hash_cap = sh.hash_cap;
  P.hash_bits = sh.hash_bits;
  P.nslot = sh.nslot;
  P.qw = sh.qw;
  flags = launch_flags(flags, c->late_counters_pending);
  P.flags = flags;
  P.row_draft = row_draft;
  P.slot_keep = slot_keep;
  P.done = c->d_done;
  P.ring = kept_hist ? c->d_ring : nullptr;
  P.hlen = kept_hist ? c->d_hlen : nullptr;
  rc = launch(c, P, dtype, sh, flags, static_cast<cudaStream_t>(stream),
              row_draft != nullptr ? "sample_verify" : "sample_rows");
  if (rc == STRATA_OK) c->late_counters_pending = pending_after(c->late_counters_pending, flags, true);
  return rc;
}

int strata_sample_rows(strata_ctx* c, const void* logits, int dtype, int B, int V, int64_t ld,
                       const int32_t* row_slot, const int64_t* row_pos, const int32_t* hist,
                       const int32_t* hist_off, int n_hist_slots, int32_t* out_ids, int top_n, float* chosen_lp,
                       int32_t* top_ids, float* top_lps, const int32_t* allowed, const int32_t* allowed_off,
                       float* allowed_lps, int32_t* topk_ids, float* topk_vals, int32_t* kept, uint32_t flags,
                       void* stream) {
  return sample_rows_impl(c, logits, dtype, B, V, ld, row_slot, row_pos, nullptr, hist, hist_off, n_hist_slots, out_ids,
                          nullptr, top_n, chosen_lp, top_ids, top_lps, allowed, allowed_off, allowed_lps, topk_ids,
                          topk_vals, kept, flags, stream);
}

int strata_sample_verify(strata_ctx* c, const void* logits, int dtype, int B, int V, int64_t ld,
                         const int32_t* row_slot, const int64_t* row_pos, const int32_t* row_draft,
                         const int32_t* hist, const int32_t* hist_off, int n_hist_slots, int32_t* out_ids,
                         int32_t* slot_keep, int top_n, float* chosen_lp, int32_t* top_ids, float* top_lps,
                         uint32_t flags, void* stream) {
  if (B > 0 && (row_draft == nullptr || slot_keep == nullptr))
    return fail(STRATA_EINVAL, "row_draft and slot_keep are required");
  return sample_rows_impl(c, logits, dtype, B, V, ld, row_slot, row_pos, row_draft, hist, hist_off, n_hist_slots,
                          out_ids, slot_keep, top_n, chosen_lp, top_ids, top_lps, nullptr, nullptr, nullptr, nullptr,
                          nullptr, nullptr, flags, stream);
}

int strata_logprobs_rows(strata_ctx* c, const void* logits, int dtype, int B, int V, int64_t ld,
                         const int32_t* chosen, float* chosen_lp, int top_n, int32_t* top_ids, float* top_lps,
                         const int32_t* allowed, const int32_t* allowed_off, float* allowed_lps, uint32_t flags,
                         void* stream) {
  int rc = check_rows_common(c, logits, dtype, B, V, ld, top_n, chosen_lp, top_ids, top_lps, allowed, allowed_off,
                             allowed_lps);
  if (rc != STRATA_OK) return rc;
  if ((chosen == nullptr) != (chosen_lp == nullptr)) return fail(STRATA_EINVAL, "chosen and chosen_lp must be given together");
  if ((rc = check_device(c)) != STRATA_OK) return rc;
  if (B == 0) return STRATA_OK;
  const int top_n_eff = (top_n > 0 && top_ids != nullptr) ? top_n : 0;
  Shape sh;
  if ((rc = compute_shape(c, strata::MODE_LOGPROBS, dtype, B, V, top_n_eff, false, allowed_off != nullptr, flags, &sh)) !=
      STRATA_OK)
    return rc;
  KParams P{};
  P.logits = logits;
  P.ld = ld;
  P.B = B;
  P.V = V;
  P.cs = sh.cs;
  P.chunk = sh.chunk;
  P.mode = strata::MODE_LOGPROBS;
  P.top_n = top_n;
  P.nmax = sh.nmax;
  P.kmax = 0;
  P.chosen_lp = chosen_lp;
  P.top_ids = top_n_eff > 0 ? top_ids : nullptr;
  P.top_lps = top_n_eff > 0 ? top_lps : nullptr;
  P.chosen = chosen;
  P.allowed = allowed;
  P.allowed_off = allowed_off;
  P.allowed_lps = allowed_lps;
  P.slots = c->d_slots;
  P.ctr = c->d_ctr;
  P.max_slots = c->max_slots;
  P.err = c->d_err;
  P.nslot = sh.nslot;
  P.qw = sh.qw;
  flags = launch_flags(flags, c->late_counters_pending);
  P.flags = flags;
  rc = launch(c, P, dtype, sh, flags, static_cast<cudaStream_t>(stream), "logprobs_rows");
  if (rc == STRATA_OK) c->late_counters_pending = pending_after(c->late_counters_pending, flags, false);
  return rc;
}

int strata_shard_rows(strata_ctx* c, const void* logits, int dtype, int B, int V_shard, int64_t ld, int id_offset,
                      const int32_t* row_slot, const int32_t* hist, const int32_t* hist_off, int n_hist_slots,
                      int top_n, void* records, uint32_t flags, void* stream) {
  int rc = check_rows_common(c, logits, dtype, B, V_shard, ld, top_n, nullptr, nullptr, nullptr, nullptr, nullptr,
                             nullptr);
  if (rc != STRATA_OK) return rc;
  if (id_offset < 0 || static_cast<long long>(id_offset) + V_shard > 0x7FFFFFFFLL)
    return fail(STRATA_EINVAL, "id_offset=%d with V_shard=%d outside the int32 id range", id_offset, V_shard);
  if (B > 0 && (row_slot == nullptr || records == nullptr)) return fail(STRATA_EINVAL, "row_slot and records are required");
  if ((reinterpret_cast<uintptr_t>(records) & 15u) != 0) return fail(STRATA_EALIGN, "records not 16-byte aligned");
  if ((flags & ~(STRATA_FLAG_CONCURRENT | STRATA_FLAG_SPLIT(31))) != 0u)
    return fail(STRATA_EINVAL, "flags 0x%x: a slice call takes only STRATA_FLAG_CONCURRENT and STRATA_FLAG_SPLIT", flags);
  if (hist_off != nullptr && (hist == nullptr || n_hist_slots < 1))
    return fail(STRATA_EINVAL, "hist_off needs hist and n_hist_slots >= 1");
  if (hist_off == nullptr) n_hist_slots = 0;
  if ((rc = check_device(c)) != STRATA_OK) return rc;
  if (B == 0) return STRATA_OK;
  Shape sh;
  if ((rc = compute_shape(c, strata::MODE_SAMPLE, dtype, B, V_shard, top_n, hist_off != nullptr, false, flags, &sh)) !=
      STRATA_OK)
    return rc;
  KParams P{};
  P.logits = logits;
  P.ld = ld;
  P.B = B;
  P.V = V_shard;
  P.cs = sh.cs;
  P.chunk = sh.chunk;
  P.mode = strata::MODE_SAMPLE;
  P.row_slot = row_slot;
  P.hist = hist;
  P.hist_off = hist_off;
  P.n_hist_slots = n_hist_slots;
  P.top_n = top_n;
  P.nmax = sh.nmax;
  P.kmax = sh.kmax;
  P.slots = c->d_slots;
  P.ctr = c->d_ctr;
  P.max_slots = c->max_slots;
  P.err = c->d_err;
  P.hash_cap = sh.hash_cap;
  P.hash_bits = sh.hash_bits;
  P.nslot = sh.nslot;
  P.qw = sh.qw;
  P.flags = flags;
  P.id_off = id_offset;
  P.rec = static_cast<unsigned char*>(records);
  rc = launch(c, P, dtype, sh, flags, static_cast<cudaStream_t>(stream), "shard_rows");
  if (rc == STRATA_OK) c->late_counters_pending = pending_after(c->late_counters_pending, flags, false);
  return rc;
}

int strata_merge_shards(strata_ctx* c, const void* records, int n_shards, int B, const int32_t* row_slot,
                        const int64_t* row_pos, int32_t* out_ids, int top_n, float* chosen_lp, int32_t* top_ids,
                        float* top_lps, int32_t* topk_ids, float* topk_vals, int32_t* kept, uint32_t flags,
                        void* stream) {
  if (c == nullptr) return fail(STRATA_EINVAL, "null context");
  if (n_shards < 1 || n_shards > STRATA_MAX_SHARDS)
    return fail(STRATA_EINVAL, "n_shards=%d outside 1..%d", n_shards, STRATA_MAX_SHARDS);
  if (B < 0) return fail(STRATA_EINVAL, "B=%d", B);
  if (B > c->max_rows) return fail(STRATA_ERANGE, "B=%d above max_rows %d", B, c->max_rows);
  if (top_n < 0 || top_n > STRATA_MAX_TOP_N) return fail(STRATA_EINVAL, "top_n=%d outside 0..%d", top_n, STRATA_MAX_TOP_N);
  if (top_n > 0 && ((top_ids == nullptr) != (top_lps == nullptr)))
    return fail(STRATA_EINVAL, "top_ids and top_lps must be given together");
  if (B > 0 && (records == nullptr || row_slot == nullptr || row_pos == nullptr || out_ids == nullptr))
    return fail(STRATA_EINVAL, "records, row_slot, row_pos and out_ids are required");
  if ((reinterpret_cast<uintptr_t>(records) & 15u) != 0) return fail(STRATA_EALIGN, "records not 16-byte aligned");
  if (flags != 0u) return fail(STRATA_EINVAL, "flags 0x%x: the merge takes none", flags);
  int rc;
  if ((rc = check_device(c)) != STRATA_OK) return rc;
  if (B == 0) return STRATA_OK;
  strata::MParams M{};
  M.rec = static_cast<const unsigned char*>(records);
  M.G = n_shards;
  M.B = B;
  M.top_n = top_n;
  M.row_slot = row_slot;
  M.row_pos = reinterpret_cast<const long long*>(row_pos);
  M.out_ids = out_ids;
  M.chosen_lp = chosen_lp;
  M.top_ids = top_n > 0 ? top_ids : nullptr;
  M.top_lps = top_n > 0 ? top_lps : nullptr;
  M.topk_ids = topk_ids;
  M.topk_vals = topk_vals;
  M.kept = kept;
  M.slots = c->d_slots;
  M.ctr = c->d_ctr;
  M.max_slots = c->max_slots;
  M.err = c->d_err;
  if (trace_on())
    std::fprintf(stderr, "strata: merge_shards B=%d shards=%d top_n=%d grid=%d block=%d\n", B, n_shards, top_n, B,
                 strata::MT);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
  cfg.blockDim = dim3(strata::MT, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, strata::merge_kernel, M);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  c->late_counters_pending = pending_after(c->late_counters_pending, 0u, true);
  return STRATA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// strata_sample_rows_noalloc: the sampling call for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a framework whose allocator owns
// every byte of device memory, or a process that must not grow its device footprint once serving
// has started.  This entry point needs no context.  The only global memory it uses beyond the
// caller's inputs and outputs (one prepared key record and one packed counter word per row, the
// identity row-to-slot table and the device error word) lives in the file-scope array below,
// which every GPU that loads this library holds until the process exits.  Every call shares the
// array and it keeps the last call's contents; each call rewrites the parts it reads, so calls
// that overlap on the GPU (two streams at once) race and must not be issued.
// ---------------------------------------------------------------------------------------------
namespace {

constexpr int NA_MAX_ROWS = STRATA_NOALLOC_MAX_ROWS;
constexpr size_t NA_CTR = 256;                                          // error word at offset 0
constexpr size_t NA_SLOTS = NA_CTR + sizeof(unsigned long long) * NA_MAX_ROWS;
constexpr size_t NA_ROWSLOT = NA_SLOTS + sizeof(SlotDev) * NA_MAX_ROWS;
constexpr size_t NA_BYTES = NA_ROWSLOT + sizeof(int32_t) * NA_MAX_ROWS;

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_BYTES];

namespace {

struct NoallocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0, max_cluster = 8, max_smem = 0, smem_three = 0;
};
constexpr int NA_MAX_DEVICES = 64;
NoallocDevice g_na[NA_MAX_DEVICES];
std::mutex g_na_mu;

// Once per device, with that device current: the array's device address, kernel attributes and
// the identity row-to-slot table.  Runs inside the first call on the device (synchronously).
int noalloc_setup(int dev, NoallocDevice** out) {  // called with g_na_mu held
  NoallocDevice& d = g_na[dev];
  if (!d.ready) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.scratch), g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major < 10) return fail(STRATA_ECUDA, "device %s is not a Blackwell GPU", prop.name);
    d.num_sms = prop.multiProcessorCount;
    d.max_smem = static_cast<int>(prop.sharedMemPerBlockOptin);
    d.smem_three = smem_for_three(prop);
    if ((e = set_kernel_attributes(d.max_smem)) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    d.max_cluster = 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(strata::MAX_CS, 1, 1);
    cfg.blockDim = dim3(strata::NT, 1, 1);
    cfg.dynamicSmemBytes = 128 * 1024;
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = strata::MAX_CS;
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, strata::rows_kernel<0, false>, &cfg) == cudaSuccess && nclusters > 0)
      d.max_cluster = strata::MAX_CS;
    cudaGetLastError();
    static int32_t identity[NA_MAX_ROWS];
    for (int i = 0; i < NA_MAX_ROWS; ++i) identity[i] = i;
    if ((e = cudaMemcpy(d.scratch + NA_ROWSLOT, identity, sizeof(identity), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "row table upload");
    d.ready = true;
  }
  *out = &d;
  return STRATA_OK;
}

// Host staging of one call's key records and counter words: one static buffer, used under
// g_na_mu from the first write to the return of the copies that read it (a copy from pageable
// memory returns once the runtime holds the bytes), so host threads take turns.
struct NoallocStage {
  unsigned char head[NA_CTR + sizeof(unsigned long long) * NA_MAX_ROWS];
  SlotDev slots[NA_MAX_ROWS];
};
NoallocStage g_na_stage;

}  // namespace

extern "C" int strata_sample_rows_noalloc(const void* logits, int dtype, int B, int V, int64_t ld,
                                          const strata_sampling_params* row_params, const uint64_t* row_counters,
                                          const int64_t* row_pos, const int32_t* hist, const int32_t* hist_off,
                                          int32_t* out_ids, int top_n, float* chosen_lp, int32_t* top_ids,
                                          float* top_lps, void* stream) {
  if (dtype != STRATA_DTYPE_F32 && dtype != STRATA_DTYPE_BF16) return fail(STRATA_EINVAL, "dtype %d", dtype);
  if (B < 0) return fail(STRATA_EINVAL, "B=%d", B);
  if (B > NA_MAX_ROWS) return fail(STRATA_ERANGE, "B=%d above the %d rows this call's static scratch holds", B, NA_MAX_ROWS);
  if (V < 1 || V > STRATA_MAX_VOCAB) return fail(STRATA_ERANGE, "V=%d outside 1..%d", V, STRATA_MAX_VOCAB);
  if (ld < V) return fail(STRATA_EINVAL, "ld=%lld below V=%d", static_cast<long long>(ld), V);
  if (top_n < 0 || top_n > STRATA_MAX_TOP_N) return fail(STRATA_EINVAL, "top_n=%d outside 0..%d", top_n, STRATA_MAX_TOP_N);
  if (top_n > 0 && ((top_ids == nullptr) != (top_lps == nullptr)))
    return fail(STRATA_EINVAL, "top_ids and top_lps must be given together");
  if (B == 0) return STRATA_OK;
  if (logits == nullptr || row_params == nullptr || row_counters == nullptr || row_pos == nullptr || out_ids == nullptr)
    return fail(STRATA_EINVAL, "logits, row_params, row_counters, row_pos and out_ids are required");
  if (hist_off != nullptr && hist == nullptr) return fail(STRATA_EINVAL, "hist_off needs hist");
  const int esz = dtype == STRATA_DTYPE_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) != 0) return fail(STRATA_EALIGN, "logits not 16-byte aligned");
  if ((static_cast<long long>(ld) * esz) % 16 != 0) return fail(STRATA_EALIGN, "row stride not a multiple of 16 bytes");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= NA_MAX_DEVICES) return fail(STRATA_ERANGE, "device %d", dev);

  // keys and counters of this call, one slot per row
  std::lock_guard<std::mutex> lock(g_na_mu);
  NoallocStage& st = g_na_stage;
  std::memset(st.head, 0, NA_CTR);  // the device error word starts at zero
  unsigned long long* ctr = reinterpret_cast<unsigned long long*>(st.head + NA_CTR);
  int kmax_sampled = 0, max_lastn = 0;
  for (int b = 0; b < B; ++b) {
    int rc = strata_validate_params(&row_params[b]);
    if (rc != STRATA_OK) return rc;
    if (row_counters[b] >= (1ull << 48)) return fail(STRATA_ERANGE, "row %d counter needs more than 48 bits", b);
    strata_sampling_params q = row_params[b];
    q.struct_size = sizeof(strata_sampling_params);
    st.slots[b] = prepare(q);
    ctr[b] = static_cast<unsigned long long>(row_counters[b]) << 16;
    if (st.slots[b].flags & strata::SLOT_SAMPLED) kmax_sampled = std::max(kmax_sampled, st.slots[b].k);
    if (st.slots[b].flags & strata::SLOT_PENAL) max_lastn = std::max(max_lastn, st.slots[b].last_n);
  }
  NoallocDevice* nd = nullptr;
  int rc = noalloc_setup(dev, &nd);
  if (rc != STRATA_OK) return rc;

  // launch shape (same rules as a context's)
  const int top_n_eff = (top_n > 0 && top_ids != nullptr) ? top_n : 0;
  Shape sh;
  if ((rc = shape_for(nd->max_cluster, nd->max_smem, nd->smem_three, nd->num_sms, strata::MODE_SAMPLE, esz, B, V,
                      std::max(1, kmax_sampled),
                      top_n_eff, max_lastn, hist_off != nullptr, false, false, false, 0, 0, &sh)) != STRATA_OK)
    return rc;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((e = cudaMemcpyAsync(nd->scratch, st.head, NA_CTR + sizeof(unsigned long long) * B, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "counter upload");
  if ((e = cudaMemcpyAsync(nd->scratch + NA_SLOTS, st.slots, sizeof(SlotDev) * B, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "key upload");

  KParams P{};
  P.logits = logits;
  P.ld = ld;
  P.B = B;
  P.V = V;
  P.cs = sh.cs;
  P.chunk = sh.chunk;
  P.mode = strata::MODE_SAMPLE;
  P.row_slot = reinterpret_cast<const int32_t*>(nd->scratch + NA_ROWSLOT);
  P.row_pos = reinterpret_cast<const long long*>(row_pos);
  P.hist = hist;
  P.hist_off = hist_off;
  P.n_hist_slots = hist_off != nullptr ? B : 0;
  P.out_ids = out_ids;
  P.top_n = top_n;
  P.nmax = sh.nmax;
  P.kmax = sh.kmax;
  P.chosen_lp = chosen_lp;
  P.top_ids = top_n_eff > 0 ? top_ids : nullptr;
  P.top_lps = top_n_eff > 0 ? top_lps : nullptr;
  P.slots = reinterpret_cast<const SlotDev*>(nd->scratch + NA_SLOTS);
  P.ctr = reinterpret_cast<unsigned long long*>(nd->scratch + NA_CTR);
  P.max_slots = B;
  P.err = reinterpret_cast<uint32_t*>(nd->scratch);
  P.hash_cap = sh.hash_cap;
  P.hash_bits = sh.hash_bits;
  P.nslot = sh.nslot;
  P.qw = sh.qw;
  P.flags = 0;
  return launch(nullptr, P, dtype, sh, 0u, s, "sample_rows_noalloc");
}
