// Instantiations (bf16 cache, fp8 cache) of the chunk-attention kernel for head_dim_qk = 128, head_dim_v = 128.
#include "chunk_attn_impl.cuh"

namespace vpp {
template cudaError_t launch_chunk_attn_t<128, 128, false>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const AttnParams&, int,
                                                       cudaStream_t);
template cudaError_t launch_chunk_attn_t<128, 128, true>(const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, const AttnParams&, int,
                                                      cudaStream_t);
}  // namespace vpp

#ifdef VPP_TIMELINE
// Timeline build only: copies out / clears the stamps of this instantiation.
extern "C" int vpp_timeline_read(long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, vpp::g_timeline, sizeof(vpp::g_timeline)));
}
extern "C" int vpp_timeline_clear() {
  static long long zero[2 * 4 * 64 * 4];
  return static_cast<int>(cudaMemcpyToSymbol(vpp::g_timeline, zero, sizeof(zero)));
}
#endif
