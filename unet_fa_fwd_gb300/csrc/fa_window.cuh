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
// grid.  Both kernels copy 16-byte chunks (8 bf16), 2 * bytes(tensor) per
// tensor moved; a chunk's source row is found with 32-bit multiply-shift
// divisions by the launch's sizes (set on the host by finish()), so the
// copies are not bound by index arithmetic.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fa_window_geom.h"

namespace fa {

// Window-major copy of three [B, H, N, D] tensors into
// [B * windows / pack, H, pack * win_tokens, D].  One thread per 16-byte chunk.
__global__ void __launch_bounds__(256) fa_window_gather_kernel(
    const uint4* __restrict__ s0, const uint4* __restrict__ s1, const uint4* __restrict__ s2,
    uint4* __restrict__ d0, uint4* __restrict__ d1, uint4* __restrict__ d2, WindowGeom g,
    long long chunks) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= chunks) return;
  const uint32_t row = (uint32_t)(i >> g.chunk_shift);  // row of the windowed tensor
  const int part = (int)(i & ((1 << g.chunk_shift) - 1));
  const long long src = (g.source_row(row) << g.chunk_shift) + part;
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
  const uint32_t row = (uint32_t)(i >> g.chunk_shift);
  const int part = (int)(i & ((1 << g.chunk_shift) - 1));
  const long long dst_row = g.source_row(row);
  out[(dst_row << g.chunk_shift) + part] = __ldg(o_w + i);
  if (part == 0) lse[dst_row] = __ldg(lse_w + row);
}

}  // namespace fa
