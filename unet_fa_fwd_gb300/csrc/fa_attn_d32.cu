// fa_attn_d32.cu — the attention kernel's instantiations for head dimension 32
// (bf16 or e4m3 Q K^T, every mask kind) and their launcher.
#include "fa_attn_impl.cuh"

namespace fa {

int launch_attention_d32(const Params& prm, bool f8, int device, int sm_count, cudaStream_t stream) {
  return launch_attention<32>(prm, f8, device, sm_count, stream);
}

}  // namespace fa
