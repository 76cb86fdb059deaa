// fa_quant.cuh — the pre-pass of the FP8 forward (SageAttention-style, as in
// "算子加速：注意力、编译与融合", section "SageAttention": K is smoothed by
// subtracting its mean, then Q and K are quantised for a low-precision Q K^T;
// P and V stay 16-bit here).
//
//   mean_k[c]  = (1/Nk) sum_j k[j][c]                 per (b, h) and channel c
//   K~         = K - mean_k                            (scores shift by q_i . mean_k
//                                                       per row: softmax unchanged)
//   k_scale[b] = max |K~| over 128-key block b / 448, K8 = e4m3(K~ / k_scale)
//   q_scale[b] = max |Q|  over 128-row block b / 448, Q8 = e4m3(Q / q_scale)
//   lse_corr_i = scale * (q_i . mean_k)                added back to LSE_i
//
// 448 is the largest finite e4m3 value.  All kernels are bound by HBM
// bandwidth (each reads its bf16 input once and writes one byte per element).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace fa {

constexpr float kE4M3Max = 448.f;

// Partial per-channel sums of K: block (bh, split) sums tokens
// [split*per, (split+1)*per) into partial[bh][split][D].  256 threads =
// 256/D token lanes x D channels; coalesced along the channel.
template <int D>
__global__ void __launch_bounds__(256) fa_k_colsum_kernel(const __nv_bfloat16* __restrict__ k,
                                                          float* __restrict__ partial, int Nk,
                                                          int nsplit) {
  constexpr int LANES = 256 / D;
  const int bh = blockIdx.x, sp = blockIdx.y;
  const int per = (Nk + nsplit - 1) / nsplit;
  const int t0 = sp * per, t1 = min(Nk, t0 + per);
  const int c = threadIdx.x % D, r = threadIdx.x / D;
  float acc = 0.f;
  for (int t = t0 + r; t < t1; t += LANES) acc += __bfloat162float(k[((size_t)bh * Nk + t) * D + c]);
  __shared__ float red[256];
  red[threadIdx.x] = acc;
  __syncthreads();
  if (r == 0) {
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < LANES; ++i) sum += red[i * D + c];
    partial[((size_t)bh * nsplit + sp) * D + c] = sum;
  }
}

__global__ void fa_k_mean_kernel(const float* __restrict__ partial, float* __restrict__ mean,
                                 int BH, int D, int nsplit, int Nk) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BH * D) return;
  const int bh = i / D, c = i % D;
  float sum = 0.f;
  for (int sp = 0; sp < nsplit; ++sp) sum += partial[((size_t)bh * nsplit + sp) * D + c];
  mean[i] = sum / (float)Nk;
}

// One CTA of 128 threads per (bh, 128-row block); thread r owns row blk*128+r.
// IS_K: subtract the channel mean first.  Q: also write scale * (q_i . mean_k).
template <int D, bool IS_K>
__global__ void __launch_bounds__(128) fa_quant_rows_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ mean_k, uint8_t* __restrict__ x8,
    float* __restrict__ block_scale, float* __restrict__ lse_corr, int N, int nblk, float scale) {
  const int bh = blockIdx.x / nblk, blk = blockIdx.x % nblk;
  const int r = threadIdx.x;
  const int n = blk * 128 + r;
  __shared__ float smean[D];
  __shared__ float wmax[4];
  for (int c = r; c < D; c += 128) smean[c] = mean_k[(size_t)bh * D + c];
  __syncthreads();

  float val[D];
  float amax = 0.f, dot = 0.f;
  if (n < N) {
    const uint4* src = reinterpret_cast<const uint4*>(x + ((size_t)bh * N + n) * D);
#pragma unroll
    for (int v = 0; v < D / 8; ++v) {
      const uint4 u = __ldg(src + v);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h2[e]);
        const int c = v * 8 + e * 2;
        val[c] = IS_K ? f.x - smean[c] : f.x;
        val[c + 1] = IS_K ? f.y - smean[c + 1] : f.y;
      }
    }
#pragma unroll
    for (int c = 0; c < D; ++c) {
      amax = fmaxf(amax, fabsf(val[c]));
      if (!IS_K) dot = fmaf(val[c], smean[c], dot);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((r & 31) == 0) wmax[r >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
  const float s = amax > 0.f ? amax / kE4M3Max : 1.f;
  const float inv = 1.f / s;
  if (r == 0) block_scale[(size_t)bh * nblk + blk] = s;
  if (n < N) {
    uint4* dst = reinterpret_cast<uint4*>(x8 + ((size_t)bh * N + n) * D);
#pragma unroll
    for (int v = 0; v < D / 16; ++v) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // element c + b goes to byte b (little-endian order of the row)
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const __nv_fp8_storage_t q8 =
              __nv_cvt_float_to_fp8(val[v * 16 + e * 4 + b] * inv, __NV_SATFINITE, __NV_E4M3);
          word |= (uint32_t)q8 << (8 * b);
        }
        w[e] = word;
      }
      dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (!IS_K) lse_corr[(size_t)bh * N + n] = scale * dot;
  }
}

}  // namespace fa
