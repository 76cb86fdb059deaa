// fa_attn_impl.cuh — body of the per-D attention launchers declared in
// fa_attn_launch.h (included only by fa_attn_d{32,64,128}.cu).
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_attn_launch.h"
#include "fa_log.h"

namespace fa {

constexpr int kLaunchMaxDevices = 64;

template <int D, bool F8, int MK, bool WIN = false>
int launch_one(const Params& prm, int device, int sm_count, cudaStream_t stream) {
  using C = Cfg<D, F8, MK>;
  static std::mutex mu;
  static bool ready[kLaunchMaxDevices] = {};
  if (device < 0 || device >= kLaunchMaxDevices) return FA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[device]) {
      if (cudaFuncSetAttribute(fa_fwd_kernel<D, F8, MK, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES) != cudaSuccess)
        return FA_ERR_CUDA;
      // The warpgroup register split (setmaxnreg) must fit in the registers
      // the launch reserves, or the increase would wait forever: refuse to
      // launch a build where it does not.
      cudaFuncAttributes fattr;
      if (cudaFuncGetAttributes(&fattr, fa_fwd_kernel<D, F8, MK, WIN>) != cudaSuccess) return FA_ERR_CUDA;
      if (2 * 128 * C::REGS_SOFTMAX + 128 * C::REGS_OTHER > fattr.numRegs * C::THREADS)
        return FA_ERR_UNSUPPORTED;
      ready[device] = true;
    }
  }
  const int grid = prm.num_units < sm_count ? prm.num_units : sm_count;
  static const char* kMaskNames[] = {"none", "key fp32x4", "fp32", "u8x16", "u8",
                                      "fp32 staged"};
  log_launch("fa_fwd_kernel<D=%d,%s,mask %s%s> tile %dx%d grid %d x %d threads smem %d B tmem %d cols "
             "stages %d units %d (single-tile from %d) key ranges %d BH %d Nq %d Nk %d "
             "mask %s causal %d seg %d",
             D, F8 ? "e4m3 QK" : "bf16", kMaskNames[MK], WIN ? ",window rows" : "", C::BM, C::BN, grid, C::THREADS,
             C::SMEM_BYTES, C::TMEM_COLS, C::STAGES, prm.num_units, prm.tail_start, prm.num_splits,
             prm.BH, prm.Nq, prm.Nk,
             prm.full_mask ? (prm.full_mask_bool ? "bool[B,h,Nq,Nk]" : "additive[B,h,Nq,Nk]")
                           : (prm.mask ? "key[B,Nk]" : "none"),
             prm.causal, prm.seg);
  fa_fwd_kernel<D, F8, MK, WIN><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D>
int launch_attention(const Params& prm, bool f8, int device, int sm_count, cudaStream_t stream) {
  if (f8) {
    // The e4m3 path takes a key-padding mask at most.
    switch (prm.mask_kind) {
      case kMaskNone: return launch_one<D, true, kMaskNone>(prm, device, sm_count, stream);
      case kMaskF32Vec: return launch_one<D, true, kMaskF32Vec>(prm, device, sm_count, stream);
      case kMaskF32Scalar: return launch_one<D, true, kMaskF32Scalar>(prm, device, sm_count, stream);
      default: return FA_ERR_UNSUPPORTED;
    }
  }
  if (prm.win) {
    if (prm.mask_kind != kMaskNone) return FA_ERR_UNSUPPORTED;
    return launch_one<D, false, kMaskNone, true>(prm, device, sm_count, stream);
  }
  switch (prm.mask_kind) {
    case kMaskNone: return launch_one<D, false, kMaskNone>(prm, device, sm_count, stream);
    case kMaskF32Vec: return launch_one<D, false, kMaskF32Vec>(prm, device, sm_count, stream);
    case kMaskF32Scalar: return launch_one<D, false, kMaskF32Scalar>(prm, device, sm_count, stream);
    case kMaskU8Vec: return launch_one<D, false, kMaskU8Vec>(prm, device, sm_count, stream);
    case kMaskU8Scalar: return launch_one<D, false, kMaskU8Scalar>(prm, device, sm_count, stream);
    case kMaskF32Staged: return launch_one<D, false, kMaskF32Staged>(prm, device, sm_count, stream);
    default: return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
