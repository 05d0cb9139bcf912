// Host-side check of the kernel's shared-memory layout over every shape the launcher can ask for:
// each region starts on a 16-byte boundary, the candidate lists fit in the copy ring, and the
// allowed-id bitmap either fits in the ring (where it lives after the first pass) or sits in its
// own region without overlapping the next one.  Exit status 1 when any shape fails.
#include <cstdio>
#include "../request_token_sampling_gb300/csrc/strata_kernel.cuh"

int main() {
  long long n = 0, bad = 0;
  const int chunks[] = {16, 32, 48, 1008, 2000, 4096, 8000, 15520, 31040, 62080, 124160, 248320, 262144, 524288};
  const int hashes[] = {0, 64, 128, 256, 512, 1024, 2048, 4096, 8192};
  for (int chunk : chunks)
    for (int hc : hashes)
      for (int cs = 1; cs <= strata::MAX_CS; ++cs)
        for (int km = 0; km <= 64; ++km)
          for (int nm = 0; nm <= 20; ++nm)
            for (int ns = 2; ns <= strata::MAX_SLOTS; ++ns)
              for (int al = 0; al < 2; ++al)
                for (int mk = 0; mk < 2; ++mk) {
                  const int qw = 1 << (ns % 4);  // 1, 2, 4, 8
                  const strata::Layout L = strata::make_layout(chunk, hc, cs, km, nm, ns, qw, al, mk && al);
                  ++n;
                  const unsigned ring = static_cast<unsigned>(ns) * strata::PIECE_BYTES;
                  const unsigned bw = strata::align_up((static_cast<unsigned>(chunk) + 31) / 32 * 4, 16);
                  bool ok = strata::layout_aligned(L);
                  ok = ok && static_cast<unsigned>(L.cand_cap) * 24u <= ring;
                  ok = ok && (L.abits != L.data || bw <= ring);
                  ok = ok && (L.abits == L.data || !al || L.abits + bw <= L.mbits);
                  ok = ok && L.total >= L.sorted_raw;
                  if (!ok && ++bad <= 5)
                    std::printf("bad layout: chunk %d hash %d cs %d kmax %d nmax %d slots %d\n", chunk, hc, cs, km, nm, ns);
                }
  std::printf("%lld layouts, %lld bad\n", n, bad);
  return bad != 0;
}
