// chunk_attn.cuh -- parameters of the chunk-attention kernel (shared with api.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace vpp {

constexpr int kTileM = 128;        // query rows per tile (tokens x GQA heads)
constexpr int kTileN = 128;        // keys per KV tile
constexpr int kMaxAttnSegs = 64;   // prefill segments per launch

// One prefill segment: a chunk of one sequence (a7 splits its key range).
struct AttnSeg {
  int32_t q_start;     // first packed query row (token) of the segment in q/out
  int32_t q_len;       // C
  int32_t kv_len;      // P + C keys in the cache
  int32_t table_off;   // offset (entries) of the sequence's block-table row
  int32_t n_pairs;     // CTAs per (kv head, split): pairs of query tiles
  int32_t n_splits;    // key ranges (1 = write the final output directly)
  int32_t split_keys;  // keys per non-final range, multiple of kTileN
  int32_t cta_begin;   // first CTA index of this segment
  int32_t kv_base;     // contiguous cache: row of the segment's key 0
  int32_t pad0;
  int64_t ws_row0;     // first workspace row of this segment's partials
};

struct AttnParams {
  int32_t n_segs;
  int32_t heads;
  int32_t kv_heads;
  int32_t group;          // heads / kv_heads
  int32_t num_blocks;     // paged: blocks in the pool (an out-of-range block reads zeros)
  int32_t paged;          // 1: 4-D paged K/V maps, 0: 3-D contiguous maps
  float scale_log2;       // softmax scale * log2(e)
  int32_t pad0;
  const int32_t* block_table;
  uint16_t* out;          // bf16 [total_q][heads][dv]
  float* lse;             // [heads][lse_stride] float32, may be null
  int64_t lse_stride;
  float* ws_o;            // split partials, float32 [rows][heads][dv]
  float* ws_lse;          // [rows][heads]
  const float* k_scale;   // [kv_heads] factor on every key (fp8 cache), may be null
  const float* v_scale;   // [kv_heads] factor on every value (fp8 cache), may be null
  int* status;
  AttnSeg segs[kMaxAttnSegs];
};

// Smem and thread shape of one instantiation.
constexpr int kAttnThreads = 384;  // warp 0 TMA, warps 1/3 MMA, warp 2 TMEM, WG1/WG2 softmax
constexpr int kSmemLimit = 232448; // 227 KB per CTA on sm_103a
constexpr int kSubTileBytes = kTileN * 64 * 2;  // 128 keys x 64 bf16 (one 128B-swizzled block)

// fp8 (E4M3) cache: the codes of one half sub-tile (64 keys = one cache
// block x 64 dims, one byte each) land in a staging slot first and are
// widened into a ring slot; two staging slots per converter warp.
constexpr int kStageBytes = kBlockTokens * 64;
constexpr int kNumStages = 8;
// Threads of a CTA: over an fp8 cache a fourth warpgroup widens the codes.
__host__ __device__ constexpr int attn_threads(bool f8) { return f8 ? 512 : kAttnThreads; }

__host__ __device__ constexpr int attn_q_bytes(int dq) { return 2 * (dq / 64) * kSubTileBytes; }
__host__ __device__ constexpr int attn_stage_bytes(bool f8) { return f8 ? kNumStages * kStageBytes : 0; }
// The K/V ring is made of 16 KB sub-tile slots (128 keys x 64 dims); a K tile
// takes dq/64 consecutive slots and a V tile dv/64 (modulo the ring size).
__host__ __device__ constexpr int attn_num_slots(int dq, bool f8 = false) {
  return (kSmemLimit - attn_q_bytes(dq) - attn_stage_bytes(f8) - 2048) / kSubTileBytes > 12
             ? 12
             : (kSmemLimit - attn_q_bytes(dq) - attn_stage_bytes(f8) - 2048) / kSubTileBytes;
}
__host__ __device__ constexpr int attn_smem_bytes(int dq, int dv, bool f8 = false) {
  return 1024 + attn_q_bytes(dq) + attn_num_slots(dq, f8) * kSubTileBytes + attn_stage_bytes(f8) + 1024 +
         0 * dv;
}

// f8: K/V maps address E4M3 codes (uint8, no swizzle, box 64 dims x 64 keys)
// and the kernel computes in f16; otherwise bf16 maps and bf16 arithmetic.
cudaError_t launch_chunk_attn(int dq, int dv, bool f8, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, const AttnParams& p, int grid,
                              cudaStream_t stream);

// Merge of split partials for one segment (a7).
cudaError_t launch_lse_merge(const float* ws_o, const float* ws_lse, int64_t ws_row0,
                             int n_splits, int q_len, int q_start, int heads, int dv,
                             uint16_t* out, float* lse, int64_t lse_stride, int num_sms,
                             cudaStream_t stream);

}  // namespace vpp
