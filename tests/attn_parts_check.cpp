// Host check of the attention's part length (internal.h: attn_chunks_per_part) on the
// drafter's geometry (8 KV heads, a 2048-key window: 32 context chunks of 64 keys,
// 152 SMs): the lengths measured best at 1, 4 and 16 requests, and the rule's
// invariants for every request count, window and SM count in range (a power of two
// up to 16; at most 8 context parts unless 16 chunks a part do not get there; the
// grid at most 1.3 waves of two CTAs per SM unless 16 chunks a part).  Prints
// "ok <cases>" or the first failure.
#include <cstdio>

#include "internal.h"

int main() {
  const int want[][2] = {{1, 4}, {2, 4}, {4, 4}, {8, 8}, {12, 16}, {16, 16}};
  for (const auto& w : want) {
    const int c = df2::attn_chunks_per_part(w[0], 8, 32, 152);
    if (c != w[1]) {
      std::printf("2048-key window, %d requests: %d chunks a part, want %d\n", w[0], c, w[1]);
      return 1;
    }
  }
  long long cases = 0;
  for (int sms : {16, 132, 148, 152, 160})
    for (int nkv : {1, 2, 8})
      for (int nc = 1; nc <= 128; ++nc)
        for (int R = 1; R <= 256; ++R) {
          const int c = df2::attn_chunks_per_part(R, nkv, nc, sms);
          const int parts = (nc + c - 1) / c;
          const long long ctas = static_cast<long long>(R) * nkv * (parts + 1);
          const bool pow2 = c >= 1 && c <= 16 && (c & (c - 1)) == 0;
          const bool few = parts <= 8 || c == 16;
          const bool fits = 10 * ctas <= 26LL * sms || c == 16 || (c > 1 && (nc + c / 2 - 1) / (c / 2) > 8);
          if (!pow2 || !few || !fits) {
            std::printf("R=%d nkv=%d chunks=%d sms=%d: %d chunks a part\n", R, nkv, nc, sms, c);
            return 1;
          }
          // the smallest such length: half of it breaks one of the two limits
          if (c > 1) {
            const int h = c / 2, ph = (nc + h - 1) / h;
            const long long ch = static_cast<long long>(R) * nkv * (ph + 1);
            if (ph <= 8 && 10 * ch <= 26LL * sms) {
              std::printf("R=%d nkv=%d chunks=%d sms=%d: %d chunks a part, %d would do\n", R, nkv, nc, sms, c, h);
              return 1;
            }
          }
          ++cases;
        }
  std::printf("ok %lld\n", cases);
  return 0;
}
