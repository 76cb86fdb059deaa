// fa_window.cuh — window / shifted-window attention as batched attention:
// gather each window's tokens into its own batch entry, run the attention
// kernel on [B * windows, H, win_h * win_w, D], scatter O and LSE back
// ("Step 3.7 Flash" §3.2: collect the positions of a window into a batch and
// run scaled-dot-product attention on that larger batch).
//
// Small windows are packed: `pack` consecutive windows (of one image or the
// next) share one batch entry of pack * win_tokens rows, and the attention
// kernel keeps each row to the keys of its own window (segments of
// win_tokens), so a 128-row tile holds 128 / win_tokens windows instead of one.
//
// Token t of an img_h x img_w grid (row-major) sits at (r, c).  A cyclic
// shift by (shift_h, shift_w) moves it to ((r - shift_h) mod img_h,
// (c - shift_w) mod img_w); windows are win_h x win_w tiles of the shifted
// grid.  Both kernels copy 16-byte chunks (8 bf16) and are bound by HBM
// bandwidth: 2 * bytes(tensor) per tensor moved.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace fa {

struct WindowGeom {
  int B, H, img_h, img_w, win_h, win_w, shift_h, shift_w, D;
  int pack;  // windows per batch entry; B * windows() is a multiple of it
  __host__ __device__ int windows_w() const { return img_w / win_w; }
  __host__ __device__ int windows() const { return (img_h / win_h) * (img_w / win_w); }
  __host__ __device__ int win_tokens() const { return win_h * win_w; }
  __host__ __device__ int tokens() const { return img_h * img_w; }
  __host__ __device__ int entry_tokens() const { return pack * win_tokens(); }
  // Original token index of local token `t` of window `w`.
  __host__ __device__ int source_token(int w, int t) const {
    const int rs = (w / windows_w()) * win_h + t / win_w;
    const int cs = (w % windows_w()) * win_w + t % win_w;
    const int r = (rs + shift_h) % img_h;
    const int c = (cs + shift_w) % img_w;
    return r * img_w + c;
  }
};

// Window-major copy of three [B, H, N, D] tensors into
// [B * windows / pack, H, pack * win_tokens, D].  One thread per 16-byte chunk.
__global__ void __launch_bounds__(256) fa_window_gather_kernel(
    const uint4* __restrict__ s0, const uint4* __restrict__ s1, const uint4* __restrict__ s2,
    uint4* __restrict__ d0, uint4* __restrict__ d1, uint4* __restrict__ d2, WindowGeom g,
    long long chunks) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= chunks) return;
  const int per_row = g.D / 8;
  const long long row = i / per_row;                 // row of the windowed tensor
  const int part = (int)(i % per_row);
  const int te = (int)(row % g.entry_tokens());      // row within the batch entry
  const long long eh = row / g.entry_tokens();       // entry * H + h
  const int h = (int)(eh % g.H);
  const long long bw = (eh / g.H) * g.pack + te / g.win_tokens();  // b * windows + w
  const int t = te % g.win_tokens();
  const int w = (int)(bw % g.windows());
  const long long b = bw / g.windows();
  const long long src = (((b * g.H + h) * g.tokens() + g.source_token(w, t)) * per_row) + part;
  d0[i] = __ldg(s0 + src);
  d1[i] = __ldg(s1 + src);
  d2[i] = __ldg(s2 + src);
}

// Inverse of the gather for O (bf16 [entries, H, pack * win_tokens, D] ->
// [B, H, N, D]) and LSE (fp32 [entries, H, pack * win_tokens] -> [B, H, N]).
__global__ void __launch_bounds__(256) fa_window_scatter_kernel(
    const uint4* __restrict__ o_w, const float* __restrict__ lse_w, uint4* __restrict__ out,
    float* __restrict__ lse, WindowGeom g, long long chunks) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= chunks) return;
  const int per_row = g.D / 8;
  const long long row = i / per_row;
  const int part = (int)(i % per_row);
  const int te = (int)(row % g.entry_tokens());
  const long long eh = row / g.entry_tokens();
  const int h = (int)(eh % g.H);
  const long long bw = (eh / g.H) * g.pack + te / g.win_tokens();
  const int t = te % g.win_tokens();
  const int w = (int)(bw % g.windows());
  const long long b = bw / g.windows();
  const long long dst_row = (b * g.H + h) * g.tokens() + g.source_token(w, t);
  out[dst_row * per_row + part] = __ldg(o_w + i);
  if (part == 0) lse[dst_row] = __ldg(lse_w + row);
}

}  // namespace fa
