// Host-side check of both kernels' shared-memory layouts over every shape the launcher can ask
// for.  Streaming kernel: each region starts on a 16-byte boundary, the candidate lists fit in the
// copy ring, and the allowed-id bitmap either fits in the ring (where it lives after the first
// pass) or sits in its own region without overlapping the next one.  Resident kernel: each region
// is aligned, the chunk region holds every whole vector of the chunk, the allowed-id bitmap fits
// where it is placed (inside the candidate region or before the mask bitmap), and the regions
// follow one another without overlap.  Exit status 1 when any shape fails.
#include <cstdio>
#include "../request_token_sampling_gb300/csrc/strata_resident.cuh"

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
                  const int qw = 1 << ((ns + km) % 5);  // 1, 2, 4, 8, 16
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
  const int rchunks[] = {16, 32, 48, 1008, 2000, 4096, 8000, 15520, 16384, 31040, 32768};
  for (int esz : {4, 2})
    for (int chunk : rchunks) {
      if (chunk * esz > strata::RES_MAX_CHUNK_BYTES) continue;
      for (int hc : hashes)
        for (int cs = 1; cs <= strata::MAX_CS; ++cs)
          for (int km = 0; km <= 64; ++km)
            for (int nm = 0; nm <= 20; ++nm)
              for (int al = 0; al < 2; ++al)
                for (int mk = 0; mk < 2; ++mk) {
                  const int qw = 1 << ((km + nm + cs) % 5);  // 1..16
                  const strata::RLayout L = strata::make_res_layout(chunk, esz, hc, cs, km, nm, qw, al, mk && al);
                  ++n;
                  const unsigned bw = strata::align_up((static_cast<unsigned>(chunk) + 31) / 32 * 4, 16);
                  const unsigned nvec_bytes = (static_cast<unsigned>(chunk) * esz + 15) / 16 * 16;
                  bool ok = strata::res_layout_aligned(L);
                  ok = ok && L.mbar >= L.data + nvec_bytes;
                  ok = ok && L.hash >= L.mbar + strata::RNBAR * 8 && L.hflag >= L.hash + 4u * hc;
                  ok = ok && L.cand_raw == L.cand_pen + 16u * strata::RES_CAP;
                  ok = ok && (L.abits == L.cand_pen ? bw <= 24u * strata::RES_CAP : L.abits >= L.cand_raw + 8u * strata::RES_CAP);
                  ok = ok && (!al || L.abits == L.cand_pen || L.abits + bw <= L.mbits);
                  ok = ok && (!(mk && al) || L.mbits + bw <= L.xrec);
                  ok = ok && L.recv_cnt >= L.xrec + 4u * cs * (strata::NW * qw + 4) && L.recv_pkey >= L.recv_cnt + 8u * cs;
                  ok = ok && L.recv_praw >= L.recv_pkey + 8u * cs * km && L.recv_raw >= L.recv_praw + 4u * cs * km;
                  ok = ok && L.sorted_pen >= L.recv_raw + 8u * cs * nm && L.sorted_raw >= L.sorted_pen + 16u * km;
                  ok = ok && L.total >= L.sorted_raw + 8u * nm;
                  if (!ok && ++bad <= 10)
                    std::printf("bad resident layout: chunk %d esz %d hash %d cs %d kmax %d nmax %d\n", chunk, esz, hc, cs,
                                km, nm);
                }
    }
  std::printf("%lld layouts, %lld bad\n", n, bad);
  return bad != 0;
}
