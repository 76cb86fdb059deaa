// fa_diag.cuh — throughput probe of the exponential unit.
//
// The forward takes one exp2 per score (B·H·Nq·Nk per launch), issued as
// ex2.approx.ftz.f32 on the SM's special-function (MUFU) pipe.  This kernel
// measures how many of those one SM completes per clock: every thread runs 16
// independent chains y <- 2^y - 1 (y stays in (-1, 0]), so the pipe, not the
// dependency latency, sets the pace.  Four 256-thread CTAs per SM; each CTA
// times its loop with clock64 and the slowest CTA bounds the SM's rate.
#pragma once

#include <cstdint>

#include "sm100_ptx.cuh"

namespace fa {

constexpr int kDiagThreads = 256;
constexpr int kDiagCtasPerSm = 4;
constexpr int kDiagChains = 16;
constexpr int kDiagMaxCtas = 4096;

__device__ long long g_diag_clk[kDiagMaxCtas];
__device__ float g_diag_sink[kDiagMaxCtas];

__global__ void __launch_bounds__(kDiagThreads) fa_ex2_rate_kernel(int iters) {
  float y[kDiagChains];
#pragma unroll
  for (int k = 0; k < kDiagChains; ++k) y[k] = -0.001f * (float)((threadIdx.x % 7) + k);
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < kDiagChains; ++k) y[k] = ptx::ex2(y[k]) - 1.0f;
  }
  const long long t1 = clock64();
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kDiagChains; ++k) s += y[k];
  if (s == 1234.5f) g_diag_sink[blockIdx.x] = s;  // keeps the chains live
  if (threadIdx.x == 0) g_diag_clk[blockIdx.x] = t1 - t0;
}

}  // namespace fa
