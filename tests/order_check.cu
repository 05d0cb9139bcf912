// Host-side check of the rule that keeps draw counters in call order when one context's calls
// with own outputs (counters taken at the start, before the next launch; no wait) and calls that
// take their counters after waiting for their predecessor share a stream.  Random streams of
// launches go through the library's own flag rule (launch_flags / pending_after) and an event model
// of programmatic dependent launch; every sampling call must take its counters after the one before
// it.  The library's host code is compiled in; nothing runs on a GPU.  Exit status 1 on a violation.
#include "../request_token_sampling_gb300/csrc/strata_sample.cu"
#include <random>

int main() {
  // Event model of one stream (integer times).  Launch i starts after launch i-1 triggered (PDL)
  // or after every earlier launch ended (no PDL).  With early loads a launch triggers at entry;
  // without them it first waits for launch i-1 to end, then triggers.  A launch with own outputs
  // takes its counters at start + 1 and triggers after that; it waits for nothing.  Any other
  // launch with early loads waits for launch i-1 to end before its counters (at its end); without
  // early loads it takes them during its work.  Only the immediate predecessor's end is waited for.
  std::mt19937 rng(7);
  long long runs = 0, bad = 0, own_taken = 0;
  const uint32_t kinds[] = {0u, STRATA_FLAG_PDL, STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD,
                            STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD | STRATA_FLAG_OWN_OUTPUTS,
                            STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD | STRATA_FLAG_OWN_OUTPUTS};
  for (int run = 0; run < 200000; ++run) {
    bool pending = false;
    long long prev_trigger = 0, prev_end = 0, all_end = 0, last_ctr = -1;
    const int n = 2 + static_cast<int>(rng() % 14);
    for (int i = 0; i < n; ++i) {
      const bool sampling = rng() % 4 != 0;
      const uint32_t fl = launch_flags(kinds[rng() % 5], pending);
      const bool pdl = (fl & STRATA_FLAG_PDL) != 0u, early = (fl & STRATA_FLAG_EARLY_LOAD) != 0u;
      const bool own = early && (fl & STRATA_FLAG_OWN_OUTPUTS) != 0u;
      const long long work = 2 + static_cast<long long>(rng() % 60);
      long long start = pdl ? prev_trigger + 1 : all_end + 1;
      long long trigger, ctr, end;
      if (own) {
        ctr = start + 1;
        trigger = ctr + 1;
        end = start + work + 2;
        ++own_taken;
      } else if (pdl && early) {
        trigger = start;
        const long long waited = std::max(start + work, prev_end + 1);
        ctr = waited + 1;
        end = ctr + 1;
      } else {
        if (pdl) start = std::max(start, prev_end + 1);  // waits for its predecessor at entry
        trigger = start;
        ctr = start + work / 2;
        end = start + work;
      }
      if (sampling) {
        if (ctr <= last_ctr) ++bad;
        last_ctr = ctr;
      }
      pending = pending_after(pending, fl, sampling);
      prev_trigger = trigger;
      prev_end = end;
      all_end = std::max(all_end, end);
    }
    ++runs;
  }
  std::printf("%lld runs, %lld bad, %lld launches took counters early\n", runs, bad, own_taken);
  return bad != 0 || own_taken == 0;
}
