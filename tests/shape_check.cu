// Host-side check of the launcher's shape rule over the shapes a GB300 context can be asked for:
// every call gets a shape whose blocks cover the row, whose shared memory fits the device, whose
// candidate lists hold what the merge needs, and whose ring keeps at least two slots (a forced
// split whose blocks cannot fit is refused with STRATA_ERANGE).  The library's host code is compiled into this program; nothing runs on a GPU.
// Exit status 1 when any shape fails.
#include "../request_token_sampling_gb300/csrc/strata_sample.cu"

int main() {
  // a GB300: 152 SMs, 16-CTA clusters, 227 KiB opt-in shared memory per block, 228 KiB per SM
  const int max_cluster = 16, max_smem = 232448, num_sms = 152;
  const int smem_three = std::min(max_smem, 233472 / 3 - 1024 - SMEM_L1_MARGIN) & ~127;
  long long n = 0, bad = 0, over_three = 0, refused = 0, resident = 0;
  const int Vs[] = {1, 17, 2048, 4099, 32000, 100003, 248320, 262144, 524288};
  const int Bs[] = {1, 5, 8, 64, 1024};
  const int concurrent_bytes[] = {0, 128 * 1024, 512 * 1024, 1024 * 1024};
  for (int mode : {strata::MODE_SAMPLE, strata::MODE_LOGPROBS})
    for (int esz : {4, 2})
      for (int V : Vs)
        for (int B : Bs)
          for (int kmax : {1, 20, 64})
            for (int nmax : {0, 5, 20})
              for (int lastn : {0, 64, 2048, 4096})
                for (int opts = 0; opts < 16; ++opts)
                  for (int cb : concurrent_bytes)
                    for (int forced : {0, 1, 2, 16})
                    for (int streaming = 0; streaming < 2; ++streaming) {
                      const bool with_hist = opts & 1, with_allowed = opts & 2, pipelined = opts & 8;
                      const bool mask = (opts & 4) && with_allowed && mode == strata::MODE_SAMPLE;
                      const int k = mode == strata::MODE_SAMPLE ? kmax : 0;
                      Shape s{};
                      const int rc = shape_for(max_cluster, max_smem, smem_three, num_sms, mode, esz, B, V, k, nmax,
                                               lastn, with_hist, with_allowed, mask, pipelined, cb, forced, &s,
                                               streaming != 0);
                      ++n;
                      if (forced > 0 && rc == STRATA_ERANGE && s.smem > max_smem) {  // a forced split refused cleanly
                        ++refused;
                        continue;
                      }
                      bool ok = rc == STRATA_OK;
                      ok = ok && s.cs >= 1 && s.cs <= max_cluster && (forced == 0 || s.cs == forced);
                      ok = ok && static_cast<long long>(s.cs) * s.chunk >= V && s.chunk % 16 == 0;
                      ok = ok && s.smem > 0 && s.smem <= max_smem;
                      if (s.resident) {  // the chunk held whole: at most 64 KiB, one bulk copy per 16 KiB piece
                        ok = ok && !streaming && static_cast<long long>(s.chunk) * esz <= strata::RES_MAX_CHUNK_BYTES;
                        ok = ok && s.nslot >= 1 && s.nslot <= strata::RES_PIECES &&
                             s.nslot * strata::PIECE_BYTES >= s.chunk * esz;
                        ok = ok && s.smem >= static_cast<int>(strata::make_res_layout(s.chunk, esz, s.hash_cap, s.cs,
                                                                                      s.kmax, s.nmax, s.qw, with_allowed,
                                                                                      mask).total);
                        ok = ok && s.cs * strata::NW * s.qw >= std::min(2 * std::max(k, nmax), s.cs * strata::NW * strata::RES_QW_MAX);
                        ++resident;
                      } else {
                        ok = ok && s.nslot >= 2 && s.nslot <= strata::MAX_SLOTS;
                      }
                      ok = ok && s.qw >= 1 && s.qw <= (s.resident ? strata::RES_QW_MAX : strata::QW_MAX) && (s.qw & (s.qw - 1)) == 0;
                      ok = ok && (s.hash_cap == 0 || s.hash_cap >= 2 * lastn);
                      if (ok && s.smem > smem_three) ++over_three;
                      if (!ok && ++bad <= 5)
                        std::printf("bad shape: rc %d mode %d esz %d V %d B %d k %d n %d lastn %d opts %d cb %d forced %d: "
                                    "cs %d chunk %d smem %d slots %d (%s)\n", rc, mode, esz, V, B, k, nmax, lastn, opts, cb,
                                    forced, s.cs, s.chunk, s.smem, s.nslot, g_err);
                    }
  std::printf("%lld shapes, %lld bad, %lld above three blocks per SM, %lld forced splits refused, %lld resident\n", n,
              bad, over_three, refused, resident);
  return bad != 0;
}
