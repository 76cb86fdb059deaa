// The window map of the attention kernel's window mode (WindowGeom::source_row, multiply-shift
// division by the launch's sizes) agrees with its division-by-division
// definition (source_token and the windowed layout [entries, H, pack *
// win_tokens]) for every row of a set of geometries: square and rectangular
// windows, packs of 1..64 windows per entry, cyclic shifts including wrap-around.
// Prints "ok" or the first mismatch.
#include <cstdio>
#include <cstdint>

#include "fa_window_geom.h"

using fa::WindowGeom;

static int check(int B, int H, int img_h, int img_w, int win_h, int win_w, int sh, int sw,
                 int D, int pack) {
  WindowGeom g{B, H, img_h, img_w, win_h, win_w, sh, sw, D, pack};
  g.finish();
  const long long nwin = g.windows(), Nw = g.win_tokens(), Ne = g.entry_tokens();
  const long long rows = (long long)B * H * g.tokens();
  for (long long row = 0; row < rows; ++row) {
    // The windowed layout, one division at a time.
    const long long te = row % Ne, eh = row / Ne;
    const long long h = eh % H, e = eh / H;
    const long long bw = e * pack + te / Nw, t = te % Nw;
    const long long w = bw % nwin, b = bw / nwin;
    const long long want = (b * H + h) * g.tokens() + g.source_token((int)w, (int)t);
    const long long got = g.source_row((uint32_t)row);
    if (got != want) {
      std::printf("mismatch B%d H%d %dx%d win %dx%d shift %d,%d pack %d row %lld: %lld != %lld\n",
                  B, H, img_h, img_w, win_h, win_w, sh, sw, pack, row, got, want);
      return 1;
    }
  }
  return 0;
}

int main() {
  const int geo[][4] = {{64, 64, 8, 8}, {64, 64, 16, 16}, {32, 48, 8, 4}, {12, 20, 4, 5},
                        {8, 8, 8, 8}, {7, 9, 7, 3}, {30, 30, 3, 3}};
  const int Bs[] = {1, 2, 3}, Hs[] = {1, 3, 8}, Ds[] = {32, 64, 128};
  for (const auto& q : geo) {
    const int img_h = q[0], img_w = q[1], win_h = q[2], win_w = q[3];
    const int shifts[][2] = {{0, 0}, {win_h / 2, win_w / 2}, {1, 2}, {img_h - 1, img_w - 1}};
    for (int B : Bs)
      for (int H : Hs)
        for (const auto& s : shifts)
          for (int D : Ds) {
            const int nw = (img_h / win_h) * (img_w / win_w);
            // every pack that divides the window count of the batch (the host
            // picks one of these)
            for (int pack = 1; pack <= 64; ++pack) {
              if ((B * nw) % pack) continue;
              if (check(B, H, img_h, img_w, win_h, win_w, s[0], s[1], D, pack)) return 1;
            }
          }
  }
  std::printf("ok\n");
  return 0;
}
