// Instances of the persistent attention kernel at head_dim 128 (one
// translation unit per head dim, compiled in parallel).
#include "attn_impl.cuh"

namespace pkv {

cudaError_t launch_attention_d128(const AttnParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                 const CUtensorMap& tm_q, int num_ctas, bool fp8, bool has_prefill, bool has_decode,
                                 bool overlap_prev, cudaStream_t stream) {
  return launch_dim<128>(p, tm_k, tm_v, tm_q, num_ctas, fp8, has_prefill, has_decode, overlap_prev, stream);
}

}  // namespace pkv
