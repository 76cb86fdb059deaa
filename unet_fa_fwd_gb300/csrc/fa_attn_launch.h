// fa_attn_launch.h — host launchers of the attention kernel, one per head
// dimension.  Each is compiled in its own translation unit
// (fa_attn_d32.cu / fa_attn_d64.cu / fa_attn_d128.cu, built in parallel),
// holding that D's kernel instantiations: bf16 or e4m3 Q/K times the mask
// kinds of the general softmax path.
#pragma once

#include <cuda_runtime.h>

#include "fa_fwd_kernel.cuh"

namespace fa {

// Launch fa_fwd_kernel for this D on `stream` with a persistent grid of
// min(prm.num_units, sm_count) CTAs: e4m3 Q K^T when f8, the instantiation
// for prm.mask_kind.  Sets the kernel's shared-memory attribute on first use
// per device (thread-safe).  Returns FA_OK, FA_ERR_UNSUPPORTED (a mask kind
// the e4m3 path lacks; a build whose register split does not fit) or
// FA_ERR_CUDA.
int launch_attention_d32(const Params& prm, bool f8, int device, int sm_count, cudaStream_t stream);
int launch_attention_d64(const Params& prm, bool f8, int device, int sm_count, cudaStream_t stream);
int launch_attention_d128(const Params& prm, bool f8, int device, int sm_count, cudaStream_t stream);

}  // namespace fa
