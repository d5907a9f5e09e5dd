// merge.cu -- a7: combine partial attention results over disjoint key ranges.
//
// "02 · 并行策略与 PP 切分" (deployment note), §7: context-parallel attention
// needs each partial result's log-sum-exp so that partials can be merged.
// With lse_s the natural-log denominator of range s and out_s its normalised
// output (Eq. (1) of the VPP technical review, §2.2, restricted to the range):
//     L = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - L) * out_s.
// One warp per (token, head) row; lane s < S holds lse_s, lanes then split the
// head dimension (float4 per lane).  Reads S x dv x 4 bytes per row, writes
// dv x 2 bytes: HBM-light and short next to the attention kernel.
#include "chunk_attn.cuh"
#include "ptx.cuh"

namespace vpp {

template <int DQ, int DV, bool F8>
cudaError_t launch_chunk_attn_t(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                const AttnParams&, int, cudaStream_t);

template <bool F8>
cudaError_t launch_chunk_attn_f(int dq, int dv, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, const AttnParams& p, int grid,
                                cudaStream_t stream) {
  if (dq == 64 && dv == 64) return launch_chunk_attn_t<64, 64, F8>(tm_q, tm_k, tm_v, p, grid, stream);
  if (dq == 64 && dv == 128) return launch_chunk_attn_t<64, 128, F8>(tm_q, tm_k, tm_v, p, grid, stream);
  if (dq == 128 && dv == 64) return launch_chunk_attn_t<128, 64, F8>(tm_q, tm_k, tm_v, p, grid, stream);
  if (dq == 128 && dv == 128) return launch_chunk_attn_t<128, 128, F8>(tm_q, tm_k, tm_v, p, grid, stream);
  if (dq == 192 && dv == 64) return launch_chunk_attn_t<192, 64, F8>(tm_q, tm_k, tm_v, p, grid, stream);
  if (dq == 192 && dv == 128) return launch_chunk_attn_t<192, 128, F8>(tm_q, tm_k, tm_v, p, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_chunk_attn(int dq, int dv, bool f8, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, const AttnParams& p, int grid,
                              cudaStream_t stream) {
  return f8 ? launch_chunk_attn_f<true>(dq, dv, tm_q, tm_k, tm_v, p, grid, stream)
            : launch_chunk_attn_f<false>(dq, dv, tm_q, tm_k, tm_v, p, grid, stream);
}

namespace {

template <int DV>
__global__ void __launch_bounds__(256) lse_merge_kernel(const float* __restrict__ ws_o,
                                                        const float* __restrict__ ws_lse,
                                                        int64_t ws_row0, int n_splits, int q_len,
                                                        int q_start, int heads,
                                                        uint16_t* __restrict__ out,
                                                        float* __restrict__ lse,
                                                        int64_t lse_stride) {
  constexpr int PER_LANE = DV / 32;  // 2 or 4 floats
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(q_len) * heads;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += wstride) {
    const int tok = static_cast<int>(r / heads);
    const int h = static_cast<int>(r - static_cast<int64_t>(tok) * heads);
    float my = -INFINITY;
    if (lane < n_splits)
      my = __ldg(&ws_lse[(ws_row0 + static_cast<int64_t>(lane) * q_len + tok) * heads + h]);
    float mx = my;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float w = (lane < n_splits) ? __expf(my - mx) : 0.f;
    float tot = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    float acc[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;
    for (int s = 0; s < n_splits; ++s) {
      const float ws = __shfl_sync(0xffffffffu, w, s);
      const float* src =
          ws_o + ((ws_row0 + static_cast<int64_t>(s) * q_len + tok) * heads + h) * DV + lane * PER_LANE;
      if (PER_LANE == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src));
        acc[0] += ws * v.x;
        acc[1] += ws * v.y;
        acc[2 % PER_LANE] += ws * v.z;
        acc[3 % PER_LANE] += ws * v.w;
      } else {
        const float2 v = __ldg(reinterpret_cast<const float2*>(src));
        acc[0] += ws * v.x;
        acc[1] += ws * v.y;
      }
    }
    const float inv = 1.f / tot;
    uint16_t* dst = out + (static_cast<int64_t>(q_start + tok) * heads + h) * DV + lane * PER_LANE;
    if (PER_LANE == 4) {
      uint2 pk;
      pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      pk.y = pack_bf16x2(acc[2 % PER_LANE] * inv, acc[3 % PER_LANE] * inv);
      *reinterpret_cast<uint2*>(dst) = pk;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lse && lane == 0) lse[static_cast<int64_t>(h) * lse_stride + q_start + tok] = mx + logf(tot);
  }
}

}  // namespace

cudaError_t launch_lse_merge(const float* ws_o, const float* ws_lse, int64_t ws_row0,
                             int n_splits, int q_len, int q_start, int heads, int dv,
                             uint16_t* out, float* lse, int64_t lse_stride, int num_sms,
                             cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(q_len) * heads;
  int64_t grid = (rows + 7) / 8;
  if (grid > static_cast<int64_t>(num_sms) * 16) grid = static_cast<int64_t>(num_sms) * 16;
  if (grid < 1) grid = 1;
  if (dv == 128)
    lse_merge_kernel<128><<<static_cast<int>(grid), 256, 0, stream>>>(
        ws_o, ws_lse, ws_row0, n_splits, q_len, q_start, heads, out, lse, lse_stride);
  else if (dv == 64)
    lse_merge_kernel<64><<<static_cast<int>(grid), 256, 0, stream>>>(
        ws_o, ws_lse, ws_row0, n_splits, q_len, q_start, heads, out, lse, lse_stride);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace vpp
