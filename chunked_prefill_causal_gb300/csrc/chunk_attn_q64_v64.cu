// Instantiations (bf16 cache, fp8 cache) of the chunk-attention kernel for head_dim_qk = 64, head_dim_v = 64.
#include "chunk_attn_impl.cuh"

namespace vpp {
template cudaError_t launch_chunk_attn_t<64, 64, false>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const AttnParams&, int,
                                                       cudaStream_t);
template cudaError_t launch_chunk_attn_t<64, 64, true>(const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, const AttnParams&, int,
                                                      cudaStream_t);
}  // namespace vpp
