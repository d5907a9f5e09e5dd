// kv_append.cu -- a1: copy a chunk's new K/V rows into their paged cache slots.
//
// "VPP: Virtual Pipeline Parallelism for Efficient Chunked Prefill in
// Long-Context LLM Inference" (technical review), §2.1: prefill fills the KV
// cache that later chunks and decode read.  "02 · 并行策略与 PP 切分", §1:
// the cache is a pool of 64-token blocks.
//
// Cache layout [num_blocks][64][kv_heads][d]: one token's kv_heads x d values
// are contiguous in both the source chunk and the destination slot, so the
// append is a gather of whole rows.  Every thread moves 16-byte vectors;
// consecutive threads cover consecutive vectors of a row (coalesced loads and
// stores).  The kernel is HBM-bound: it moves 2 x C x kv_heads x (dq + dv) x 2
// bytes (read + write) for a bf16 chunk.
#include "common.cuh"
#include "ptx.cuh"

namespace vpp {
namespace {

struct SingleSeqPos {
  int64_t prefix;
  const int32_t* table;  // nullptr: contiguous cache
  __device__ __forceinline__ bool slot(int64_t t, int32_t num_blocks, int64_t* row) const {
    const int64_t pos = prefix + t;
    if (!table) {
      *row = pos;
      return pos < num_blocks;  // contiguous: num_blocks is the capacity in tokens
    }
    const int32_t blk = table[pos / kBlockTokens];
    if (blk < 0 || blk >= num_blocks) return false;
    *row = static_cast<int64_t>(blk) * kBlockTokens + pos % kBlockTokens;
    return true;
  }
};

struct VarlenPos {
  const VarlenPlan* plan;  // kernel parameter space
  const int32_t* table;
  __device__ __forceinline__ bool slot(int64_t t, int32_t num_blocks, int64_t* row) const {
    // Binary search of the sequence owning packed row t.
    int lo = 0, hi = plan->batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (plan->cu_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int64_t qlen = plan->cu_q[b + 1] - plan->cu_q[b];
    const int64_t pos = plan->ctx[b] - qlen + (t - plan->cu_q[b]);
    const int32_t blk =
        table[static_cast<int64_t>(b) * plan->max_blocks_per_seq + pos / kBlockTokens];
    if (blk < 0 || blk >= num_blocks) return false;
    *row = static_cast<int64_t>(blk) * kBlockTokens + pos % kBlockTokens;
    return true;
  }
};

// One grid-stride loop over (token, 16-byte vector) of K then V.
template <typename Pos>
__device__ __forceinline__ void append_rows_bf16(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                 int64_t tokens, int vec_per_row, Pos pos,
                                                 int32_t num_blocks, int* status) {
  const int64_t total = tokens * vec_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / vec_per_row;
    const int v = static_cast<int>(i - t * vec_per_row);
    int64_t row;
    if (!pos.slot(t, num_blocks, &row)) {
      if (v == 0) record_status(status, kStatusInvalid);
      continue;
    }
    dst[row * vec_per_row + v] = __ldg(&src[i]);
  }
}

template <typename Pos>
__global__ void __launch_bounds__(256) kv_append_bf16_kernel(const uint4* __restrict__ k_new,
                                                             const uint4* __restrict__ v_new,
                                                             uint4* k_cache, uint4* v_cache,
                                                             int64_t tokens, int k_vec, int v_vec,
                                                             int32_t num_blocks, Pos pos,
                                                             int* status) {
  append_rows_bf16(k_new, k_cache, tokens, k_vec, pos, num_blocks, status);
  append_rows_bf16(v_new, v_cache, tokens, v_vec, pos, num_blocks, status);
}

// float32 input: 8 floats (32 bytes) in, 8 bf16 (16 bytes) out per step.
__device__ __forceinline__ uint4 f32x8_to_bf16x8(const float4 a, const float4 b) {
  uint4 r;
  r.x = pack_bf16x2(a.x, a.y);
  r.y = pack_bf16x2(a.z, a.w);
  r.z = pack_bf16x2(b.x, b.y);
  r.w = pack_bf16x2(b.z, b.w);
  return r;
}

__device__ __forceinline__ void append_rows_f32(const float4* __restrict__ src, uint4* __restrict__ dst,
                                                int64_t tokens, int vec_per_row, SingleSeqPos pos,
                                                int32_t num_blocks, int* status) {
  const int64_t total = tokens * vec_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / vec_per_row;
    const int v = static_cast<int>(i - t * vec_per_row);
    int64_t row;
    if (!pos.slot(t, num_blocks, &row)) {
      if (v == 0) record_status(status, kStatusInvalid);
      continue;
    }
    dst[row * vec_per_row + v] = f32x8_to_bf16x8(__ldg(&src[2 * i]), __ldg(&src[2 * i + 1]));
  }
}

__global__ void __launch_bounds__(256) kv_append_f32_kernel(const float4* __restrict__ k_new,
                                                            const float4* __restrict__ v_new,
                                                            uint4* k_cache, uint4* v_cache,
                                                            int64_t tokens, int k_vec, int v_vec,
                                                            int32_t num_blocks, SingleSeqPos pos,
                                                            int* status) {
  append_rows_f32(k_new, k_cache, tokens, k_vec, pos, num_blocks, status);
  append_rows_f32(v_new, v_cache, tokens, v_vec, pos, num_blocks, status);
}

__global__ void __launch_bounds__(256) convert_f32_bf16_kernel(const float4* __restrict__ in,
                                                               uint4* __restrict__ out,
                                                               int64_t n8) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += stride)
    out[i] = f32x8_to_bf16x8(__ldg(&in[2 * i]), __ldg(&in[2 * i + 1]));
}

// Waits on a barrier that nothing completes; the bounded wait must give up.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_for(smem_u32(&bar), 0, limit_ns)) record_status(status, kStatusTimeout);
  }
  __syncthreads();
}

int grid_for(int64_t work_items, int num_sms) {
  const int64_t per_block = 256 * 4;  // four vectors per thread before striding
  int64_t g = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_kv_append(const void* k_new, const void* v_new, bool in_fp32, void* k_cache,
                             void* v_cache, const int32_t* block_table, int32_t num_blocks,
                             int64_t prefix_len, int64_t chunk_len, int kv_heads, int dq, int dv,
                             int* status, int num_sms, cudaStream_t stream) {
  const int k_vec = kv_heads * dq * 2 / 16;
  const int v_vec = kv_heads * dv * 2 / 16;
  SingleSeqPos pos{prefix_len, block_table};
  const int grid = grid_for(chunk_len * (k_vec + v_vec), num_sms);
  if (in_fp32) {
    kv_append_f32_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const float4*>(k_new), static_cast<const float4*>(v_new),
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), chunk_len, k_vec, v_vec,
        num_blocks, pos, status);
  } else {
    kv_append_bf16_kernel<SingleSeqPos><<<grid, 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), chunk_len, k_vec, v_vec,
        num_blocks, pos, status);
  }
  return cudaGetLastError();
}

namespace {
__global__ void __launch_bounds__(256) kv_append_varlen_kernel(const uint4* __restrict__ k_new,
                                                               const uint4* __restrict__ v_new,
                                                               uint4* k_cache, uint4* v_cache,
                                                               int k_vec, int v_vec,
                                                               int32_t num_blocks,
                                                               const int32_t* table,
                                                               const __grid_constant__ VarlenPlan plan,
                                                               int* status) {
  VarlenPos pos{&plan, table};
  const int64_t tokens = plan.cu_q[plan.batch];
  append_rows_bf16(k_new, k_cache, tokens, k_vec, pos, num_blocks, status);
  append_rows_bf16(v_new, v_cache, tokens, v_vec, pos, num_blocks, status);
}
}  // namespace

cudaError_t launch_kv_append_varlen(const void* k_new, const void* v_new, void* k_cache,
                                    void* v_cache, const int32_t* block_table,
                                    const VarlenPlan& plan, int32_t num_blocks, int kv_heads,
                                    int dq, int dv, int* status, int num_sms,
                                    cudaStream_t stream) {
  const int k_vec = kv_heads * dq * 2 / 16;
  const int v_vec = kv_heads * dv * 2 / 16;
  const int64_t tokens = plan.cu_q[plan.batch];
  const int grid = grid_for(tokens * (k_vec + v_vec), num_sms);
  kv_append_varlen_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), k_vec, v_vec, num_blocks,
      block_table, plan, status);
  return cudaGetLastError();
}

cudaError_t launch_convert_f32_bf16(const float* in, uint16_t* out, int64_t n, int num_sms,
                                    cudaStream_t stream) {
  const int64_t n8 = n / 8;  // callers pass n a multiple of 8 (head dims are multiples of 64)
  convert_f32_bf16_kernel<<<grid_for(n8, num_sms), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(in), reinterpret_cast<uint4*>(out), n8);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(int timeout_us, int* status, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(timeout_us) * 1000ull,
                                                     status);
  return cudaGetLastError();
}

}  // namespace vpp
