// fa_window_geom.h — the window / shifted-window geometry shared by the
// attention kernel's window mode (its producer gathers Q/K/V rows and its
// epilogue writes O/LSE rows through source_row) and the host set-up (plain
// C++ on the host, so the index map is checked there against its
// division-by-division definition).
#pragma once

#include <cstdint>

#include "fa_fastdiv.h"

namespace fa {

struct WindowGeom {
  int B, H, img_h, img_w, win_h, win_w, shift_h, shift_w, D;
  int pack;  // windows per batch entry; B * windows() is a multiple of it
  // Launch constants (finish()): log2 of the 16-byte chunks per row, and
  // dividers by the entry's rows, H, the window's tokens, the window count,
  // the windows per grid row and the window width.
  int chunk_shift;
  FastDiv div_entry, div_h, div_win, div_nwin, div_wpr, div_ww;
  void finish() {
    chunk_shift = D == 32 ? 2 : (D == 64 ? 3 : 4);
    div_entry = FastDiv::make((uint32_t)entry_tokens());
    div_h = FastDiv::make((uint32_t)H);
    div_win = FastDiv::make((uint32_t)win_tokens());
    div_nwin = FastDiv::make((uint32_t)windows());
    div_wpr = FastDiv::make((uint32_t)windows_w());
    div_ww = FastDiv::make((uint32_t)win_w);
  }
  FA_HD int windows_w() const { return img_w / win_w; }
  FA_HD int windows() const { return (img_h / win_h) * (img_w / win_w); }
  FA_HD int win_tokens() const { return win_h * win_w; }
  FA_HD int tokens() const { return img_h * img_w; }
  FA_HD int entry_tokens() const { return pack * win_tokens(); }
  // Original token index of local token `t` of window `w`.
  FA_HD int source_token(int w, int t) const {
    const int rs = (w / windows_w()) * win_h + t / win_w;
    const int cs = (w % windows_w()) * win_w + t % win_w;
    const int r = (rs + shift_h) % img_h;
    const int c = (cs + shift_w) % img_w;
    return r * img_w + c;
  }
  // Row of the [B, H, N] tensors that windowed row `row` (< 2^31) of the
  // [entries, H, entry_tokens] layout comes from (the same map as
  // source_token, by multiply-shift division; 0 <= shift < image size).
  FA_HD long long source_row(uint32_t row) const {
    const uint32_t eh = div_entry.div(row), te = div_entry.mod(row, eh);
    const uint32_t e = div_h.div(eh), h = div_h.mod(eh, e);
    const uint32_t wi = div_win.div(te), t = div_win.mod(te, wi);
    const uint32_t bw = e * (uint32_t)pack + wi;
    const uint32_t b = div_nwin.div(bw), w = div_nwin.mod(bw, b);
    const uint32_t wr = div_wpr.div(w), wc = div_wpr.mod(w, wr);
    const uint32_t tr = div_ww.div(t), tc = div_ww.mod(t, tr);
    int r = (int)(wr * (uint32_t)win_h + tr) + shift_h;
    int c = (int)(wc * (uint32_t)win_w + tc) + shift_w;
    if (r >= img_h) r -= img_h;
    if (c >= img_w) c -= img_w;
    return ((long long)b * H + h) * tokens() + (long long)r * img_w + c;
  }
};

}  // namespace fa
