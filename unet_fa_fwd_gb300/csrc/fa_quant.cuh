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
// 448 is the largest finite e4m3 value.  Three launches: the column sums of K,
// their means, then the quantisation of K and Q (HBM bound: each input read
// once, one byte written per element).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace fa {

constexpr float kE4M3Max = 448.f;

// Partial per-channel sums of K: block (bh, split) sums tokens
// [split*per, (split+1)*per) into partial[bh][split][D].  256 threads: thread
// (r, part) reads the 16-byte chunk `part` (8 channels) of rows r, r + RL, ...,
// so a warp's loads cover whole rows contiguously.
template <int D>
__global__ void __launch_bounds__(256) fa_k_colsum_kernel(const __nv_bfloat16* __restrict__ k,
                                                          float* __restrict__ partial, int Nk,
                                                          int nsplit) {
  constexpr int PARTS = D / 8;          // 16-byte chunks per row
  constexpr int RL = 256 / PARTS;       // rows read per step
  const int bh = blockIdx.x, sp = blockIdx.y;
  const int per = (Nk + nsplit - 1) / nsplit;
  const int t0 = sp * per, t1 = min(Nk, t0 + per);
  const int part = threadIdx.x % PARTS, r = threadIdx.x / PARTS;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  const uint4* base = reinterpret_cast<const uint4*>(k + (size_t)bh * Nk * D) + part;
#pragma unroll 4
  for (int t = t0 + r; t < t1; t += RL) {
    const uint4 u = __ldg(base + (size_t)t * PARTS);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      acc[2 * e] += f.x;
      acc[2 * e + 1] += f.y;
    }
  }
  __shared__ float red[RL][D + 1];
#pragma unroll
  for (int e = 0; e < 8; ++e) red[r][part * 8 + e] = acc[e];
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += 256) {
    float sum = 0.f;
#pragma unroll 4
    for (int i = 0; i < RL; ++i) sum += red[i][c];
    partial[((size_t)bh * nsplit + sp) * D + c] = sum;
  }
}

// Channel means of K: mean[bh][c] = (sum of the nsplit partial sums) / Nk.
__global__ void fa_k_mean_kernel(const float* __restrict__ partial, float* __restrict__ mean,
                                 int BH, int D, int nsplit, int Nk) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BH * D) return;
  const int bh = i / D, c = i % D;
  float sum = 0.f;
  for (int sp = 0; sp < nsplit; ++sp) sum += partial[((size_t)bh * nsplit + sp) * D + c];
  mean[i] = sum / (float)Nk;
}

// Quantisation of K and Q in one launch: CTAs [0, BH*kt) take 128-key blocks
// of K, the rest 128-row blocks of Q.  Each CTA reads its block as 16-byte
// chunks (8 elements), chunk i by thread i mod 256, so a warp's
// loads and its 8-byte e4m3 stores cover whole rows contiguously.  A thread
// always holds the same 8 channels (256 is a multiple of the chunks per row),
// so it keeps their means in registers.  The block stays in registers as bf16
// (converted to fp32 twice: for the block max, then to quantise), so four
// CTAs fit an SM (three at D = 128) and more of the stream is in flight.  K: smoothed by the
// mean first.  Q: also writes lse_corr = scale * (q_i . mean_k), reduced
// across the D/8 lanes holding a row.
template <int D>
__global__ void __launch_bounds__(256, D == 128 ? 3 : 4) fa_quant_kernel(
    const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ q,
    const float* __restrict__ mean_k, uint8_t* __restrict__ k8,
    uint8_t* __restrict__ q8, float* __restrict__ k_scale, float* __restrict__ q_scale,
    float* __restrict__ lse_corr, int BH, int Nk, int Nq, int kt, int qt, float scale) {
  constexpr int PARTS = D / 8;                 // chunks per row (4, 8 or 16)
  constexpr int PER = 128 * PARTS / 256;       // chunks per thread (2, 4 or 8)
  const bool is_k = (int)blockIdx.x < BH * kt;
  const int cta = is_k ? (int)blockIdx.x : (int)blockIdx.x - BH * kt;
  const int nblk = is_k ? kt : qt;
  const int N = is_k ? Nk : Nq;
  const int bh = cta / nblk, blk = cta % nblk;
  const int tid = threadIdx.x;
  const int part = tid % PARTS;                // this thread's 8 channels: part*8 .. +7

  __shared__ float wmax[8];
  // the 8 channel means of this thread's chunk column
  float mean[8];
  {
    const float4* m4 = reinterpret_cast<const float4*>(mean_k + (size_t)bh * D + part * 8);
    const float4 a = __ldg(m4), b = __ldg(m4 + 1);
    mean[0] = a.x; mean[1] = a.y; mean[2] = a.z; mean[3] = a.w;
    mean[4] = b.x; mean[5] = b.y; mean[6] = b.z; mean[7] = b.w;
  }

  const size_t row0 = (size_t)bh * N + (size_t)blk * 128;
  const uint4* src = reinterpret_cast<const uint4*>((is_k ? k : q) + row0 * D);
  uint4 raw[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int r = (i * 256 + tid) / PARTS;
    raw[i] = blk * 128 + r < N ? __ldg(src + i * 256 + tid) : make_uint4(0u, 0u, 0u, 0u);
  }
  // fp32 values of chunk i (smoothed for K; rows past N are zero)
  auto values = [&](int i, float (&val)[8]) {
    const int r = (i * 256 + tid) / PARTS;
    const bool smooth = is_k && blk * 128 + r < N;
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      val[2 * e] = smooth ? f.x - mean[2 * e] : f.x;
      val[2 * e + 1] = smooth ? f.y - mean[2 * e + 1] : f.y;
    }
  };
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    float val[8];
    values(i, val);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(val[e]));
    if (!is_k) {
      const int r = (i * 256 + tid) / PARTS;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) dot = fmaf(val[e], mean[e], dot);
#pragma unroll
      for (int o = PARTS / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (part == 0 && blk * 128 + r < N) lse_corr[row0 + r] = scale * dot;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) wmax[tid >> 5] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, wmax[w]);
  const float s = amax > 0.f ? amax / kE4M3Max : 1.f;
  const float inv = 1.f / s;
  // Convert again from bf16 below rather than keep the first pass's fp32
  // values live across the barrier (that would double the registers).
#pragma unroll
  for (int i = 0; i < PER; ++i)
    asm volatile("" : "+r"(raw[i].x), "+r"(raw[i].y), "+r"(raw[i].z), "+r"(raw[i].w));
  if (tid == 0) (is_k ? k_scale : q_scale)[(size_t)bh * nblk + blk] = s;
  uint2* dst = reinterpret_cast<uint2*>((is_k ? k8 : q8) + row0 * D);
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int chunk = i * 256 + tid;
    if (blk * 128 + chunk / PARTS >= N) continue;
    float val[8];
    values(i, val);
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // element 4h + b of the chunk goes to byte b of word h (row order)
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const __nv_fp8_storage_t v8 =
            __nv_cvt_float_to_fp8(val[4 * h + b] * inv, __NV_SATFINITE, __NV_E4M3);
        word |= (uint32_t)v8 << (8 * b);
      }
      w[h] = word;
    }
    dst[chunk] = make_uint2(w[0], w[1]);
  }
}

}  // namespace fa
