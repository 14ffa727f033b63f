// Host-side check of the scan's shared-memory stage layout (compiled by nvcc
// as host code; no GPU): every staged 16-byte part lands inside its row and
// the stage buffer, no two parts collide, the two halves of every 32-byte
// sector land in one aligned 32-byte slot (host-cache layout), and the
// 8-byte block-column reads of rows r .. r + 7 fall in eight different
// 16-byte bank groups (both layouts).  Exit status 0 when all hold.
#include <cstdio>
#include <set>

#include "scan_core.cuh"

using namespace bpkv;

static int fails = 0;
#define CHECK(c, ...)                 \
  do {                                \
    if (!(c)) {                       \
      ++fails;                        \
      if (fails < 20) {               \
        std::printf(__VA_ARGS__);     \
        std::printf("\n");            \
      }                               \
    }                                 \
  } while (0)

static void check_layout(int sub, bool host, int rows) {
  const int pitch = row_pitch(sub, host);
  const int parts = 4 * sub;  // 16-byte parts per staged row
  const int sc_words = host ? kHostStageWords : kStageWords;
  std::set<int> used;
  for (int r = 0; r < rows; ++r) {
    for (int q = 0; q < parts; ++q) {
      const int w = staged_word(r, q, sub, host);
      CHECK(w % 4 == 0, "sub %d host %d row %d part %d: word %d not 16-byte aligned", sub, host, r, q, w);
      CHECK(w >= r * pitch && w + 4 <= (r + 1) * pitch, "sub %d host %d row %d part %d outside its row", sub, host, r,
            q);
      CHECK(w + 4 <= sc_words, "sub %d host %d row %d part %d runs into the scales", sub, host, r, q);
      CHECK(used.insert(w).second, "sub %d host %d row %d part %d collides", sub, host, r, q);
      if (host && (q & 1) == 0) {
        const int w2 = staged_word(r, q + 1, sub, host);
        CHECK(w / 8 == w2 / 8, "sub %d row %d sector %d split over slots %d and %d", sub, r, q / 2, w / 8, w2 / 8);
      }
    }
  }
  // block-column reads: block lb of chunk c is word 2 (lb % 2) of part 4 c + lb / 2
  for (int c = 0; c < sub; ++c) {
    for (int lb = 0; lb < kScanBlocks; ++lb) {
      for (int r0 = 0; r0 + 8 <= rows; r0 += 8) {
        std::set<int> groups;
        for (int r = r0; r < r0 + 8; ++r) groups.insert(((staged_word(r, 4 * c + lb / 2, sub, host) + 2 * (lb & 1)) / 4) % 8);
        CHECK(groups.size() == 8, "sub %d host %d chunk %d block %d rows %d..: %zu bank groups", sub, host, c, lb, r0,
              groups.size());
      }
    }
  }
  // the scales of the most slots a step can hold fit behind the rows
  const int sc_u16 = kPassSlots * kScanBlocks * sub;
  CHECK(sc_words * 2 + sc_u16 <= kStageU32 * 2, "sub %d host %d: scales overflow the stage", sub, host);
  CHECK((sc_words * 4) % 16 == 0, "scale region not 16-byte aligned");
}

int main() {
  check_layout(1, false, kStageRows);           // device caches: one chunk, up to 10 groups
  check_layout(1, true, kStageRows);            // host caches, multi-pass plans
  check_layout(kWideSub, true, kWideGroups * 32);  // host caches, wide steps
  if (fails) {
    std::printf("%d layout checks failed\n", fails);
    return 1;
  }
  std::printf("stage layout ok\n");
  return 0;
}
