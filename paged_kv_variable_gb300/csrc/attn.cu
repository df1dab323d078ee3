// Launch of the persistent attention kernel: the instance for the head dim
// (attn_d64.cu, attn_d128.cu, attn_d256.cu; the kernel itself is in
// attn_impl.cuh).
#include "kernels.h"

namespace pkv {

cudaError_t launch_attention_d64(const AttnParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, int,
                                 bool, bool, bool, bool, cudaStream_t);
cudaError_t launch_attention_d128(const AttnParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, int,
                                  bool, bool, bool, bool, cudaStream_t);
cudaError_t launch_attention_d256(const AttnParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, int,
                                  bool, bool, bool, bool, cudaStream_t);

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_q, int num_ctas, int head_dim, bool fp8, bool has_prefill,
                             bool has_decode, bool overlap_prev, cudaStream_t stream) {
  if (num_ctas == 0) return cudaSuccess;
  if (head_dim == 256)
    return launch_attention_d256(p, tm_k, tm_v, tm_q, num_ctas, fp8, has_prefill, has_decode, overlap_prev, stream);
  if (head_dim == 128)
    return launch_attention_d128(p, tm_k, tm_v, tm_q, num_ctas, fp8, has_prefill, has_decode, overlap_prev, stream);
  return launch_attention_d64(p, tm_k, tm_v, tm_q, num_ctas, fp8, has_prefill, has_decode, overlap_prev, stream);
}

}  // namespace pkv
