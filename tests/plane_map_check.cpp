// Brute-force check of the stream-K plane map shared by the projection kernels and
// the kernels that add their partial planes (internal.h: gemv_cta_of_stage,
// gemv_plane_count).  For each launch shape, every stage is assigned to its CTA by
// the partition's definition (CTA c takes stages [floor(cT/C), floor((c+1)T/C))),
// and for every weight block of a segment the CTAs that touch it must be contiguous,
// their number must equal gemv_plane_count, and the closed-form CTA of each stage
// must match.  Prints "ok <cases>" or the first mismatch.
#include <cstdio>
#include <vector>

#include "internal.h"

using df2::GemvPlanes;

int main() {
  long long cases = 0;
  const int ksts[] = {1, 2, 3, 5, 16, 40, 136};
  const int nblks[] = {1, 2, 3, 7, 20, 80, 97};
  const int Cs[] = {1, 2, 3, 7, 64, 152, 304, 1000};
  const int T0s[] = {0, 1, 13, 800};
  for (int bshift : {6, 7})
    for (int kst : ksts)
      for (int nblk : nblks)
        for (int T0 : T0s)
          for (int C : Cs) {
            const long long T = T0 + static_cast<long long>(nblk) * kst;  // a segment after T0 stages of others
            if (C > T) continue;                                          // the plans never launch more CTAs than stages
            std::vector<int> cta(T);
            for (int c = 0; c < C; ++c)
              for (long long t = (c * T) / C; t < ((c + 1) * T) / C; ++t) cta[t] = c;
            for (long long t = 0; t < T; ++t)
              if (df2::gemv_cta_of_stage(t, C, T) != cta[t]) {
                std::printf("cta mismatch: T=%lld C=%d t=%lld got %d want %d\n", T, C, t,
                            df2::gemv_cta_of_stage(t, C, T), cta[t]);
                return 1;
              }
            GemvPlanes p;
            p.T = T;
            p.base = T0;
            p.C = C;
            p.kst = kst;
            p.bshift = bshift;
            for (int b = 0; b < nblk; ++b) {
              const long long s0 = T0 + static_cast<long long>(b) * kst;
              int lo = cta[s0], hi = cta[s0];
              for (long long t = s0; t < s0 + kst; ++t) {
                if (cta[t] < hi) {
                  std::printf("not monotone\n");
                  return 1;
                }
                hi = cta[t];
              }
              const int want = hi - lo + 1;
              for (int m : {b << bshift, (b << bshift) + (1 << bshift) - 1}) {
                const int got = df2::gemv_plane_count(p, m);
                if (got != want) {
                  std::printf("count mismatch: bshift=%d kst=%d nblk=%d T0=%d C=%d block=%d m=%d got %d want %d\n",
                              bshift, kst, nblk, T0, C, b, m, got, want);
                  return 1;
                }
              }
              ++cases;
            }
          }
  std::printf("ok %lld\n", cases);
  return 0;
}
