// decode.cu -- a8: split-KV attention of single-token decode rows over a paged
// KV cache (the decode half of a mixed micro-batch).
//
// "VPP: Virtual Pipeline Parallelism for Efficient Chunked Prefill in
// Long-Context LLM Inference" (technical review), §2.1: decode produces one
// token per step and must read the whole accumulated KV cache, so it is
// bound by memory bandwidth.  "Revisiting Pipeline Parallelism for LLM
// Serving", section "预备知识": a decode request contributes one token to a
// mixed micro-batch.  The arithmetic is Eq. (1) of the VPP review (§2.2) for
// a query at position ctx-1 that sees keys 0..ctx-1.
//
// Work item = (row, key range of split_tokens keys).  One CTA per item:
//   warp Hkv (last)   producer: for every 16-token step, one 1-D bulk copy of
//                     the step's K rows and one of its V rows (16 tokens x all
//                     kv heads are contiguous inside a 64-token block), into a
//                     ring of shared-memory stages with full/empty mbarriers.
//   warps 0..Hkv-1    warp h serves kv head h and its G query heads.  Scores:
//                     8 lanes per token (D/8 dims each, 4 tokens per pass),
//                     summed with three xor-shuffles.  Online softmax per head
//                     (running max and denominator, rescale only when the max
//                     grows by more than 2^8).  P V: each lane owns D/32
//                     output dims of every head; p is passed through shared
//                     memory.
// A range's result is final when the row has one range; otherwise the float32
// partial output and its LSE go to the workspace and decode_merge combines
// them ("02 · 并行策略与 PP 切分" note, §7).  HBM-bound: the algorithmic bytes
// are ctx x Hkv x (dq + dv) x 2 per row plus q, out and the partials.
//
// fp8 cache (F8): the stages hold E4M3 codes, and both products run on the
// tensor cores (warp-level mma.sync, f16 operands: every
// E4M3 value is an f16 value; f32 accumulation), which takes the per-element
// widening and the G multiply-adds per key off the CUDA cores.  kv head h's
// k_scale joins its score scale and its v_scale multiplies the output, so
// the cache bytes per row halve.
//
// Top-k mode (SP): the rows are the query tokens of one prefill chunk and each
// attends only the key positions its index row lists (DSA-style sparse
// attention: VPP technical review §7; "02 · 并行策略与 PP 切分" §5.1).  A work
// item is (token, range of 1024 list entries).  The producer warp gathers a
// step's 16 listed keys with one bulk copy per key for K and one for V (all kv
// heads of a key are contiguous); entries outside 0 .. position, or in a block
// outside the pool, are zero-filled, masked out of the softmax and reported as
// VPP_ERR_INVALID.
#include <algorithm>

#include "common.cuh"
#include "decode.cuh"
#include "ptx.cuh"

namespace vpp {
namespace {

constexpr int kStepTokens = 16;
// Stage ring: six fp8 stages (32 rows of 1 KB + 128 bytes of group padding)
// or three bf16 stages of 64 KB, for 8 kv heads of d 128.
constexpr int kDecodeRing = 6 * (32 * 1024 + 128);
constexpr int kDecodeSmem = kDecodeRing + 4096 + 256;  // ring + p exchange + barriers
constexpr float kLn2d = 0.69314718055994530942f;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 16-byte asynchronous copy global -> shared through the load/store path;
// the bytes past src_bytes (16 or 0) are written as zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most n of this thread's copy groups are pending (n < 8).
__device__ __forceinline__ void cp_async_wait(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
  }
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

// Four E4M3 codes (byte i of w = code i) -> two f16x2 words: lo holds codes 0
// and 1, hi codes 2 and 3, the lower code in the lower half (exact: every
// E4M3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two floats -> f16x2 (round to nearest even), `lo` in bits 0-15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// D (16 x 8, f32) += A (16 x 16, f16, row-major fragment) * B (16 x 8, f16,
// column fragment): the warp-level tensor-core product.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Offset of V row t in a stage: 16 K rows, then the V rows in four groups of
// 4 tokens, vgroup bytes apart.
template <bool F8>
__device__ __forceinline__ int v_row(int t, int row_bytes, int vgroup) {
  return F8 ? kStepTokens * row_bytes + (t >> 2) * vgroup + (t & 3) * row_bytes : (kStepTokens + t) * row_bytes;
}

template <int D, int G, bool F8, bool SP>
__global__ void __launch_bounds__(288, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int DPL = D / 8;     // score dims per lane (8 lanes per token)
  constexpr int OPL = D / 32;    // output dims per lane
  constexpr int ESZ = F8 ? 1 : 2;  // cache bytes per element
  extern __shared__ __align__(128) uint8_t smem[];
  const int hkv = p.kv_heads;
  const int row_bytes = hkv * D * ESZ;               // one token, all kv heads
  // A stage holds a step's 16 K rows as they lie in the cache (one bulk
  // copy), then its V rows in four groups of 4 tokens, vgroup bytes apart.
  // bf16: the groups are contiguous (one copy).  fp8: each group is its own
  // copy and the groups are 32 bytes apart, so that the four lanes of a
  // P V fragment group, which read the same dims of four tokens, read from
  // four groups and so from four different banks.  (Padding every row
  // instead needs 32 copies per step, which measured 1.6x slower.)
  const int vgroup = F8 ? 4 * row_bytes + 32 : 4 * row_bytes;
  const int stage_bytes = F8 ? kStepTokens * row_bytes + 4 * vgroup : 2 * kStepTokens * row_bytes;
  const int nstage = min(8, kDecodeRing / stage_bytes);
  float* pbuf = reinterpret_cast<float*>(smem + kDecodeRing);  // [hkv][16][G]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecodeRing + 8 * kStepTokens * 8 * 4);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(bars + 16);
  uint32_t* step_valid = reinterpret_cast<uint32_t*>(bars + 17);  // SP: valid-entry mask per stage
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------------------------------------------------- work item
  const int item = blockIdx.x;
  DecodeRow row;
  int split, n_splits, t_begin, t_end;
  const int32_t* list = nullptr;  // SP: this token's index row
  int64_t pos = 0;                // SP: this token's absolute position
  if (SP) {
    const int64_t i = item / p.topk_splits;
    split = item - static_cast<int>(i * p.topk_splits);
    int n = __ldg(p.topk_len + i);
    if (n < 1 || n > p.topk) {
      if (threadIdx.x == 0 && split == 0) record_status(p.status, kStatusInvalid);
      n = 0;
    }
    row.b = 0;
    row.q_row = static_cast<int32_t>(i);
    row.ctx = n;
    row.item0 = static_cast<int32_t>(i * p.topk_splits);
    list = p.topk_idx + i * p.topk;
    pos = p.topk_prefix + i;
    n_splits = n > 0 ? (n + p.split_tokens - 1) / p.split_tokens : 1;
    if (split >= n_splits) return;  // the token's list is shorter: no work, nothing written
  } else {
    int lo = 0, hi = p.n_rows - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.rows[mid].item0 <= item) lo = mid; else hi = mid - 1;
    }
    row = p.rows[lo];
    split = item - row.item0;
    n_splits = (row.ctx + p.split_tokens - 1) / p.split_tokens;
  }
  t_begin = split * p.split_tokens;
  t_end = min(row.ctx, t_begin + p.split_tokens);
  const int n_steps = (t_end - t_begin + kStepTokens - 1) / kStepTokens;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < nstage; ++i) {
      mbar_init(smem_u32(&bars[i]), 1);
      mbar_init(smem_u32(&bars[8 + i]), hkv);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Top-k mode over an fp8 cache: kv-head warp h gathers its own slices (d
  // bytes per key, 16-byte copies through the load/store path) of step sp's
  // listed keys into stage slot sl, at the same places as a whole-row copy
  // would put them, and returns the step's validity mask.  Invalid entries
  // (outside 0 .. position, or in a block outside the pool) and rows past the
  // range are zero-filled.  For 1 KB rows this measured ~1.25x faster than
  // the producer warp's per-key bulk copies; for bf16's 2 KB rows it measured
  // 1.2x slower, so bf16 keeps the producer (warp_gather below).
  auto sp_issue = [&](int h, int sp, int sl) -> uint32_t {
    const int t0 = t_begin + sp * kStepTokens;
    const int nt = min(kStepTokens, t_end - t0);
    int64_t src_row = 0;
    bool valid = false;
    if (lane < nt) {
      const int64_t key = __ldg(list + t0 + lane);
      if (key >= 0 && key <= pos) {
        if (p.block_table) {
          const int32_t blk = __ldg(p.block_table + key / kBlockTokens);
          valid = blk >= 0 && blk < p.num_blocks;
          src_row = static_cast<int64_t>(blk) * kBlockTokens + key % kBlockTokens;
        } else {
          valid = key < p.num_blocks;  // contiguous cache: num_blocks is the capacity in tokens
          src_row = key;
        }
      }
      if (!valid && h == 0) record_status(p.status, kStatusInvalid);
    }
    const uint32_t vm = __ballot_sync(0xffffffffu, valid && lane < kStepTokens) & 0xFFFFu;
    constexpr int kChunks = D * ESZ / 16;  // 16-byte pieces of one key's slice
    constexpr int kKeys = 32 / kChunks;    // keys per warp instruction
    const int c = lane % kChunks;
    const int kk = lane / kChunks;
    uint8_t* stage = smem + sl * stage_bytes;
    const uint8_t* kb = static_cast<const uint8_t*>(p.k_cache) + h * D * ESZ + c * 16;
    const uint8_t* vb = static_cast<const uint8_t*>(p.v_cache) + h * D * ESZ + c * 16;
#pragma unroll
    for (int i = 0; i < kStepTokens / kKeys; ++i) {
      const int t = i * kKeys + kk;
      const int64_t r = __shfl_sync(0xffffffffu, src_row, t);
      const bool v = (vm >> t) & 1u;
      const int64_t off = (v ? r : 0) * row_bytes;
      cp_async16(smem_u32(stage + t * row_bytes + h * D * ESZ + c * 16), kb + off, v ? 16u : 0u);
      cp_async16(smem_u32(stage + v_row<F8>(t, row_bytes, vgroup) + h * D * ESZ + c * 16), vb + off,
                 v ? 16u : 0u);
    }
    cp_async_commit();
    return vm;
  };
  const int sp_ahead = nstage - 1;  // steps gathered ahead of the one computed
  constexpr bool warp_gather = SP && F8;


  if (SP && warp == hkv) {
    // ------------------------------------------------------ producer (gather)
    if (warp_gather) return;  // the kv-head warps gather their own slices (sp_issue)
    // Lane t < 16 fetches the K row of list entry t0 + t, lane 16 + t its V row.
    int slot = 0;
    uint32_t phase = 0u;
    uint32_t filled = 0u, fill_phase = 0u;
    bool ok = true;
    const int t = lane & 15;
    const bool is_v = lane >= 16;
    for (int s = 0; s < n_steps; ++s) {
      const int t0 = t_begin + s * kStepTokens;
      const int nt = min(kStepTokens, t_end - t0);
      bool valid = false;
      int64_t src_row = 0;
      if (t < nt) {
        const int64_t key = __ldg(list + t0 + t);
        if (key >= 0 && key <= pos) {
          if (p.block_table) {
            const int32_t blk = __ldg(p.block_table + key / kBlockTokens);
            valid = blk >= 0 && blk < p.num_blocks;
            src_row = static_cast<int64_t>(blk) * kBlockTokens + key % kBlockTokens;
          } else {
            valid = key < p.num_blocks;  // contiguous cache: num_blocks is the capacity in tokens
            src_row = key;
          }
        }
        if (!valid && !is_v) record_status(p.status, kStatusInvalid);
      }
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid) & 0xFFFFu;  // K lanes decide
      bool w_ok = true;
      if (lane == 0) w_ok = mbar_wait(smem_u32(&bars[8 + slot]), phase ^ 1u, p.status, abort_flag);
      if (!__shfl_sync(0xffffffffu, w_ok ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      uint8_t* dstp = smem + slot * stage_bytes + (is_v ? v_row<F8>(t, row_bytes, vgroup) : t * row_bytes);
      if (t < nt && !valid) {  // zero-filled, so that P = 0 times it stays 0
        for (int b = 0; b < row_bytes; b += 16) *reinterpret_cast<uint4*>(dstp + b) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();  // before later bulk copies into these bytes
      }
      __syncwarp();
      const uint32_t full = smem_u32(&bars[slot]);
      if (lane == 0) {
        step_valid[slot] = vmask;
        mbar_arrive_expect_tx(full, 2u * static_cast<uint32_t>(__popc(vmask)) * row_bytes);
      }
      __syncwarp();
      if (t < nt && valid) {
        const uint8_t* base = static_cast<const uint8_t*>(is_v ? p.v_cache : p.k_cache);
        bulk_g2s(smem_u32(dstp), base + src_row * row_bytes, static_cast<uint32_t>(row_bytes), full);
      }
      filled |= 1u << slot;
      fill_phase = (fill_phase & ~(1u << slot)) | (phase << slot);
      if (++slot == nstage) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      for (int i = 0; i < nstage; ++i)
        if (filled & (1u << i)) mbar_wait_for(smem_u32(&bars[i]), (fill_phase >> i) & 1u, 100000000ull);
    }
  } else if (warp == hkv) {
    // ------------------------------------------------------ producer
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0u;
      uint32_t filled = 0u, fill_phase = 0u;
      bool ok = true;
      for (int s = 0; s < n_steps; ++s) {
        const int t0 = t_begin + s * kStepTokens;
        const int nt = min(kStepTokens, t_end - t0);
        int blk = p.block_table[static_cast<int64_t>(row.b) * p.max_blocks_per_seq + t0 / kBlockTokens];
        if (blk < 0 || blk >= p.num_blocks) {
          record_status(p.status, kStatusInvalid);
          blk = -1;
        }
        if (!mbar_wait(smem_u32(&bars[8 + slot]), phase ^ 1u, p.status, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t full = smem_u32(&bars[slot]);
        const uint32_t dst = smem_u32(smem + slot * stage_bytes);
        if (blk >= 0) {
          const int64_t off = (static_cast<int64_t>(blk) * kBlockTokens + t0 % kBlockTokens) * row_bytes;
          const uint32_t bytes = static_cast<uint32_t>(nt * row_bytes);
          mbar_arrive_expect_tx(full, 2 * bytes);
          bulk_g2s(dst, static_cast<const uint8_t*>(p.k_cache) + off, bytes, full);
          const uint8_t* vsrc = static_cast<const uint8_t*>(p.v_cache) + off;
          if (!F8) {
            bulk_g2s(dst + kStepTokens * row_bytes, vsrc, bytes, full);
          } else {
            for (int g4 = 0; 4 * g4 < nt; ++g4)
              bulk_g2s(dst + v_row<F8>(4 * g4, row_bytes, vgroup), vsrc + 4 * g4 * row_bytes,
                       static_cast<uint32_t>(min(4, nt - 4 * g4) * row_bytes), full);
          }
        } else {
          mbar_arrive(full);  // invalid block: the step's rows are skipped
        }
        filled |= 1u << slot;
        fill_phase = (fill_phase & ~(1u << slot)) | (phase << slot);
        if (++slot == nstage) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        for (int i = 0; i < nstage; ++i)
          if (filled & (1u << i)) mbar_wait_for(smem_u32(&bars[i]), (fill_phase >> i) & 1u, 100000000ull);
      }
    }
  } else if (warp < hkv && F8) {
    // ------------------------------------------ kv head `warp`, fp8 codes
    // Both products run on the tensor cores (mma.sync m16n8k16, f16 operands,
    // f32 accumulation).  Lane = 4 g + u: g is the fragment's group (a token
    // row of S^T, a dim row of O^T, a head column of the B operands), u the
    // thread in the group.
    //   S^T[16 tokens x 8 heads] = K[16 x D] Q^T[D x 8]: k-step s, logical
    //     k = 2u + b + 8c maps to dim u D/4 + 4s + 2c + b, so a thread's
    //     codes of one token are D/4 consecutive bytes.
    //   O^T[D x 8 heads] += V^T[D x 16 tokens] P^T[16 x 8]: tile i, row g
    //     is dim g D/8 + 2i, row g + 8 is dim g D/8 + 2i + 1; logical
    //     k = 2u + b + 8c maps to token 4u + b + 2c, so a thread reads D/8
    //     consecutive codes of each token of V group u.
    // Heads >= G are zero columns.  E4M3 codes widen exactly to f16; q is
    // scaled by a power of two per head into f16's range (undone on the
    // scores), P is in [0, 256].
    const int h = warp;
    const int gq = lane >> 2;
    const int u = lane & 3;
    constexpr int KS = D / 16;  // k-steps of S, tiles of O
    uint32_t qb[KS][2];
    float qscale;  // 2^-e of head gq
    {
      float qv[D / 4];
      if (gq < G) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (static_cast<int64_t>(row.q_row) * p.heads + h * G + gq) * D + u * (D / 4));
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint4 w = __ldg(src + c);
          bf16x2_to_f32(w.x, qv[8 * c + 0], qv[8 * c + 1]);
          bf16x2_to_f32(w.y, qv[8 * c + 2], qv[8 * c + 3]);
          bf16x2_to_f32(w.z, qv[8 * c + 4], qv[8 * c + 5]);
          bf16x2_to_f32(w.w, qv[8 * c + 6], qv[8 * c + 7]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < D / 4; ++i) qv[i] = 0.f;
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < D / 4; ++i) amax = fmaxf(amax, fabsf(qv[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // 2^e puts the head's largest |q| in [2^14, 2^15): below f16's largest
      // value, and every bf16 value of the head that is not negligible keeps
      // its 8 significant bits.
      const int e = amax > 0.f ? max(-60, min(60, 14 - ilogbf(amax))) : 0;
      const float up = ldexpf(1.f, e);
      qscale = ldexpf(1.f, -e);
#pragma unroll
      for (int s2 = 0; s2 < KS; ++s2) {
        qb[s2][0] = pack_f16x2(qv[4 * s2] * up, qv[4 * s2 + 1] * up);
        qb[s2][1] = pack_f16x2(qv[4 * s2 + 2] * up, qv[4 * s2 + 3] * up);
      }
    }
    // This thread's S^T columns are heads 2u and 2u + 1.
    const float sl = p.scale_log2 * __ldg(p.k_scale + h);
    const float slh[2] = {sl * __shfl_sync(0xffffffffu, qscale, 8 * u),
                          sl * __shfl_sync(0xffffffffu, qscale, 8 * u + 4)};
    const float vsc = __ldg(p.v_scale + h);
    float m[2] = {-INFINITY, -INFINITY};
    float lpart[2] = {0.f, 0.f};
    float o[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float* pw = pbuf + h * kStepTokens * 8;  // P of the step: [16 tokens][8 heads]
    int slot = 0;
    uint32_t phase = 0u;
    bool ok = true;
    uint32_t my_vm = 0u;  // warp_gather: lane i < nstage holds the validity mask of stage slot i
    if (warp_gather) {
      for (int sp = 0; sp < sp_ahead; ++sp) {
        if (sp < n_steps) {
          const uint32_t vm = sp_issue(h, sp, sp);
          if (lane == sp) my_vm = vm;
        } else {
          cp_async_commit();
        }
      }
    }
    for (int s = 0; s < n_steps; ++s) {
      const int t0 = t_begin + s * kStepTokens;
      const int nt = min(kStepTokens, t_end - t0);
      if (warp_gather) {
        // gather the step sp_ahead ahead into the slot computed last, then
        // wait for this step's copies
        const int spf = s + sp_ahead;
        const int slf = spf % nstage;
        if (spf < n_steps) {
          const uint32_t vm = sp_issue(h, spf, slf);
          if (lane == slf) my_vm = vm;
        } else {
          cp_async_commit();
        }
        cp_async_wait(sp_ahead);
        __syncwarp();
      } else {
        ok = mbar_wait(smem_u32(&bars[slot]), phase, p.status, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      const uint8_t* kst = smem + slot * stage_bytes;
      const uint32_t vmask = warp_gather ? __shfl_sync(0xffffffffu, my_vm, slot) : (SP ? step_valid[slot] : 0xFFFFu);
      // ---- S^T = K Q^T (two accumulator chains)
      // With D = 128 a thread reads 32 bytes of a row; odd groups read the
      // upper 16 first, so that the two groups of a quarter warp, whose rows
      // lie a multiple of 128 bytes apart, hit different banks.
      uint32_t kw[2][D / 16];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const uint4* src = reinterpret_cast<const uint4*>(kst + (gq + 8 * rr) * row_bytes + h * D + u * (D / 4));
        if (D == 128) {
          const int sw = gq & 1;
          const uint4 wa = src[sw];
          const uint4 wb = src[sw ^ 1];
          const uint4 w0 = sw ? wb : wa;
          const uint4 w1 = sw ? wa : wb;
          kw[rr][0] = w0.x;
          kw[rr][1] = w0.y;
          kw[rr][2] = w0.z;
          kw[rr][3] = w0.w;
          kw[rr][4 % (D / 16)] = w1.x;
          kw[rr][5 % (D / 16)] = w1.y;
          kw[rr][6 % (D / 16)] = w1.z;
          kw[rr][7 % (D / 16)] = w1.w;
        } else {
          const uint4 w = src[0];
          kw[rr][0] = w.x;
          kw[rr][1] = w.y;
          kw[rr][2] = w.z;
          kw[rr][3] = w.w;
        }
      }
      float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int s2 = 0; s2 < KS; ++s2) {
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(kw[0][s2], a0, a2);
        e4m3x4_to_f16x2x2(kw[1][s2], a1, a3);
        mma_16816(sa[s2 & 1], a0, a1, a2, a3, qb[s2][0], qb[s2][1]);
      }
      // sc[rr][hh]: token gq + 8 rr, head 2u + hh
      float sc[2][2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int t = gq + 8 * rr;
        const bool tv = t < nt && ((vmask >> t) & 1u);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          sc[rr][hh] = (tv && 2 * u + hh < G) ? (sa[0][2 * rr + hh] + sa[1][2 * rr + hh]) * slh[hh] : -INFINITY;
      }
      // ---- online softmax per head (the 8 lanes of one u hold its 16 tokens)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float mx = fmaxf(sc[0][hh], sc[1][hh]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (mx > m[hh] + 8.0f || (m[hh] == -INFINITY && mx != -INFINITY)) {  // uniform over the 8 lanes
          const float f = (m[hh] == -INFINITY) ? 0.f : ex2_approx(m[hh] - mx);
          lpart[hh] *= f;
#pragma unroll
          for (int i = 0; i < KS; ++i) {
            o[i][hh] *= f;
            o[i][2 + hh] *= f;
          }
          m[hh] = mx;
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const float pv = (m[hh] == -INFINITY) ? 0.f : ex2_approx(sc[rr][hh] - m[hh]);
          lpart[hh] += pv;
          pw[(gq + 8 * rr) * 8 + 2 * u + hh] = pv;
        }
      }
      __syncwarp();
      // ---- O^T += V^T P^T
      const uint32_t pb0 = pack_f16x2(pw[(4 * u) * 8 + gq], pw[(4 * u + 1) * 8 + gq]);
      const uint32_t pb1 = pack_f16x2(pw[(4 * u + 2) * 8 + gq], pw[(4 * u + 3) * 8 + gq]);
      uint32_t vw[4][D / 32];  // tokens 4u .. 4u + 3 (V group u): this thread's D/8 codes each
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int t = 4 * u + q4;
        const uint8_t* src = kst + v_row<F8>(t, row_bytes, vgroup) + h * D + gq * (D / 8);
        if (D == 128) {
          const uint4 w = *reinterpret_cast<const uint4*>(src);
          vw[q4][0] = w.x;
          vw[q4][1 % (D / 32)] = w.y;
          vw[q4][2 % (D / 32)] = w.z;
          vw[q4][3 % (D / 32)] = w.w;
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(src);
          vw[q4][0] = w.x;
          vw[q4][1 % (D / 32)] = w.y;
        }
        // rows past the range hold stale bytes: zero codes (P is 0 there)
#pragma unroll
        for (int c = 0; c < D / 32; ++c) vw[q4][c] = t < nt ? vw[q4][c] : 0u;
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < KS; ++i) {
        const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
        const uint32_t x = __byte_perm(vw[0][i >> 1], vw[1][i >> 1], sel);
        const uint32_t y = __byte_perm(vw[2][i >> 1], vw[3][i >> 1], sel);
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(x, a0, a1);
        e4m3x4_to_f16x2x2(y, a2, a3);
        mma_16816(o[i], a0, a1, a2, a3, pb0, pb1);
      }
      __syncwarp();
      if (!warp_gather && lane == 0) mbar_arrive(smem_u32(&bars[8 + slot]));
      if (++slot == nstage) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (ok) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float l = lpart[hh];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int j = 2 * u + hh;
        if (j >= G) continue;
        const bool empty = !(l > 0.f);  // top-k rows whose entries were all invalid
        const float inv = empty ? 0.f : vsc / l;
        const float lse_v = empty ? -INFINITY : m[hh] * kLn2d + logf(l);
        const int hq = h * G + j;
        // dims gq D/8 + 2i (o[i][hh]) and + 2i + 1 (o[i][2 + hh])
        if (n_splits == 1) {
          uint32_t pk[KS];
#pragma unroll
          for (int i = 0; i < KS; ++i) pk[i] = pack_bf16x2(o[i][hh] * inv, o[i][2 + hh] * inv);
          uint16_t* dst = p.out + (static_cast<int64_t>(row.q_row) * p.heads + hq) * D + gq * (D / 8);
#pragma unroll
          for (int c = 0; c < KS / 4; ++c)
            reinterpret_cast<uint4*>(dst)[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          if (p.lse && gq == 0) p.lse[static_cast<int64_t>(hq) * p.lse_stride + row.q_row] = lse_v;
        } else {
          float* dst = p.ws_o + (static_cast<int64_t>(item) * p.heads + hq) * D + gq * (D / 8);
#pragma unroll
          for (int c = 0; c < KS / 2; ++c)
            reinterpret_cast<float4*>(dst)[c] = make_float4(o[2 * c][hh] * inv, o[2 * c][2 + hh] * inv,
                                                            o[2 * c + 1][hh] * inv, o[2 * c + 1][2 + hh] * inv);
          if (gq == 0) p.ws_lse[static_cast<int64_t>(item) * p.heads + hq] = lse_v;
        }
      }
    }
  } else if (warp < hkv) {
    // ------------------------------------------------------ kv head `warp`
    const int h = warp;
    const int tt = lane >> 3;  // token within a pass of 4
    const int r = lane & 7;    // dim group
    const uint16_t* qrow = p.q + static_cast<int64_t>(row.q_row) * p.heads * D;
    float qf[G][DPL];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const uint4* src = reinterpret_cast<const uint4*>(qrow + (h * G + j) * D + r * DPL);
#pragma unroll
      for (int c = 0; c < DPL / 8; ++c) {
        const uint4 w = __ldg(src + c);
        bf16x2_to_f32(w.x, qf[j][8 * c + 0], qf[j][8 * c + 1]);
        bf16x2_to_f32(w.y, qf[j][8 * c + 2], qf[j][8 * c + 3]);
        bf16x2_to_f32(w.z, qf[j][8 * c + 4], qf[j][8 * c + 5]);
        bf16x2_to_f32(w.w, qf[j][8 * c + 6], qf[j][8 * c + 7]);
      }
    }
    const float sl = p.scale_log2;
    float m[G], lpart[G], o[G][OPL];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      m[j] = -INFINITY;
      lpart[j] = 0.f;
#pragma unroll
      for (int i = 0; i < OPL; ++i) o[j][i] = 0.f;
    }
    float* pw = pbuf + h * kStepTokens * G;
    int slot = 0;
    uint32_t phase = 0u;
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      const int t0 = t_begin + s * kStepTokens;
      const int nt = min(kStepTokens, t_end - t0);
      ok = mbar_wait(smem_u32(&bars[slot]), phase, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint8_t* kst = smem + slot * stage_bytes;
      const uint8_t* vst = kst + kStepTokens * row_bytes;
      const uint32_t vmask = SP ? step_valid[slot] : 0xFFFFu;
      // Scores of this step's 16 tokens (4 passes of 4 tokens).
      float sc[4][G];
#pragma unroll
      for (int ps = 0; ps < 4; ++ps) {
        const int t = 4 * ps + tt;
        float2 acc[G];  // even and odd dims, two lanes of work per packed FMA
#pragma unroll
        for (int j = 0; j < G; ++j) acc[j] = make_float2(0.f, 0.f);
        if (t < nt) {
          const uint8_t* kb = kst + t * row_bytes + (h * D + r * DPL) * 2;
#pragma unroll
          for (int c = 0; c < DPL / 8; ++c) {
            float kf[8];
            const uint4 w = reinterpret_cast<const uint4*>(kb)[c];
            bf16x2_to_f32(w.x, kf[0], kf[1]);
            bf16x2_to_f32(w.y, kf[2], kf[3]);
            bf16x2_to_f32(w.z, kf[4], kf[5]);
            bf16x2_to_f32(w.w, kf[6], kf[7]);
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
              for (int e = 0; e < 8; e += 2)
                acc[j] = ffma2(make_float2(qf[j][8 * c + e], qf[j][8 * c + e + 1]),
                               make_float2(kf[e], kf[e + 1]), acc[j]);
          }
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float v = acc[j].x + acc[j].y;
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          sc[ps][j] = (t < nt && ((vmask >> t) & 1u)) ? v * sl : -INFINITY;
        }
      }
      // Online softmax, per query head.
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float mx = fmax3(fmaxf(sc[0][j], sc[1][j]), sc[2][j], sc[3][j]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (mx > m[j] + 8.0f || (m[j] == -INFINITY && mx != -INFINITY)) {  // warp-uniform
          const float f = (m[j] == -INFINITY) ? 0.f : ex2_approx(m[j] - mx);
          lpart[j] *= f;
#pragma unroll
          for (int i = 0; i < OPL; ++i) o[j][i] *= f;
          m[j] = mx;
        }
        float ps_sum = 0.f;
#pragma unroll
        for (int ps = 0; ps < 4; ++ps) {
          // (a top-k step may hold no valid entry before any valid one: m = -inf)
          const float pv = (SP && m[j] == -INFINITY) ? 0.f : ex2_approx(sc[ps][j] - m[j]);
          ps_sum += pv;
          if (r == 0) pw[(4 * ps + tt) * G + j] = pv;
        }
        if (r == 0) lpart[j] += ps_sum;
      }
      __syncwarp();
      // O += P V over the step's tokens.
      for (int t = 0; t < nt; ++t) {
        float pv[G];
#pragma unroll
        for (int j = 0; j < G; ++j) pv[j] = pw[t * G + j];
        const uint16_t* vr = reinterpret_cast<const uint16_t*>(vst + t * row_bytes + (h * D + lane * OPL) * 2);
        float vf[OPL];
        if (OPL == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(vr);
          bf16x2_to_f32(w.x, vf[0], vf[1 % OPL]);
          bf16x2_to_f32(w.y, vf[2 % OPL], vf[3 % OPL]);
        } else {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vr);
          bf16x2_to_f32(w, vf[0], vf[1 % OPL]);
        }
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
          for (int i = 0; i < OPL; i += 2) {
            const float2 r = ffma2(make_float2(pv[j], pv[j]), make_float2(vf[i], vf[i + 1]),
                                   make_float2(o[j][i], o[j][i + 1]));
            o[j][i] = r.x;
            o[j][i + 1] = r.y;
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[8 + slot]));
      if (++slot == nstage) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (ok) {
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float l = lpart[j];
#pragma unroll
        for (int x = 1; x < 32; x <<= 1) l += __shfl_xor_sync(0xffffffffu, l, x);
        const bool empty = !(l > 0.f);  // top-k rows whose entries were all invalid
        const float inv = empty ? 0.f : 1.f / l;
        const float lse_v = empty ? -INFINITY : m[j] * kLn2d + logf(l);
        const int hq = h * G + j;
        if (n_splits == 1) {
          uint16_t* dst = p.out + (static_cast<int64_t>(row.q_row) * p.heads + hq) * D + lane * OPL;
          if (OPL == 4) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o[j][0] * inv, o[j][1 % OPL] * inv),
                                                        pack_bf16x2(o[j][2 % OPL] * inv, o[j][3 % OPL] * inv));
          } else {
            *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[j][0] * inv, o[j][1 % OPL] * inv);
          }
          if (p.lse && lane == 0) p.lse[static_cast<int64_t>(hq) * p.lse_stride + row.q_row] = lse_v;
        } else {
          float* dst = p.ws_o + (static_cast<int64_t>(item) * p.heads + hq) * D + lane * OPL;
#pragma unroll
          for (int i = 0; i < OPL; ++i) dst[i] = o[j][i] * inv;
          if (lane == 0) p.ws_lse[static_cast<int64_t>(item) * p.heads + hq] = lse_v;
        }
      }
    }
  }
}

// Combines the ranges of every multi-range row: one warp per (row, head).
template <int D, bool SP>
__global__ void __launch_bounds__(256) decode_merge_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int OPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t n = (SP ? p.topk_tokens : static_cast<int64_t>(p.n_rows)) * p.heads;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < n;
       w += wstride) {
    DecodeRow row;
    if (SP) {
      const int64_t i = w / p.heads;
      int len = __ldg(p.topk_len + i);
      if (len < 1 || len > p.topk) len = 0;
      row.q_row = static_cast<int32_t>(i);
      row.ctx = len;
      row.item0 = static_cast<int32_t>(i * p.topk_splits);
    } else {
      row = p.rows[w / p.heads];
    }
    const int hq = static_cast<int>(w % p.heads);
    const int ns = (row.ctx + p.split_tokens - 1) / p.split_tokens;
    if (ns <= 1) continue;
    float mx = -INFINITY;
    for (int s = lane; s < ns; s += 32)
      mx = fmaxf(mx, p.ws_lse[(static_cast<int64_t>(row.item0) + s) * p.heads + hq]);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x));
    if (mx == -INFINITY) mx = 0.f;  // every range empty: weights 0, output 0, lse -inf
    float acc[OPL];
#pragma unroll
    for (int i = 0; i < OPL; ++i) acc[i] = 0.f;
    float tot = 0.f;
    for (int s = 0; s < ns; ++s) {
      const int64_t it = static_cast<int64_t>(row.item0) + s;
      const float wgt = __expf(p.ws_lse[it * p.heads + hq] - mx);
      tot += wgt;
      const float* src = p.ws_o + (it * p.heads + hq) * D + lane * OPL;
#pragma unroll
      for (int i = 0; i < OPL; ++i) acc[i] += wgt * src[i];
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    uint16_t* dst = p.out + (static_cast<int64_t>(row.q_row) * p.heads + hq) * D + lane * OPL;
    if (OPL == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1 % OPL] * inv),
                                                  pack_bf16x2(acc[2 % OPL] * inv, acc[3 % OPL] * inv));
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1 % OPL] * inv);
    }
    if (p.lse && lane == 0)
      p.lse[static_cast<int64_t>(hq) * p.lse_stride + row.q_row] = tot > 0.f ? mx + logf(tot) : -INFINITY;
  }
}

template <int D, int G, bool F8, bool SP>
cudaError_t launch_t(const DecodeParams& p, int items, int num_sms, cudaStream_t st) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<D, G, F8, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kDecodeSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  decode_kernel<D, G, F8, SP><<<items, 32 * (p.kv_heads + 1), kDecodeSmem, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = SP ? p.topk_tokens : static_cast<int64_t>(p.n_rows);
  int grid = static_cast<int>(std::min<int64_t>((rows * p.heads + 7) / 8, static_cast<int64_t>(num_sms) * 16));
  if (grid < 1) grid = 1;
  decode_merge_kernel<D, SP><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(int head_dim_qk, int head_dim_v, int heads, int kv_heads) {
  if (head_dim_qk != head_dim_v || (head_dim_qk != 64 && head_dim_qk != 128)) return false;
  if (kv_heads < 1 || kv_heads > 8 || heads % kv_heads) return false;
  const int g = heads / kv_heads;
  // (128, 8) would hold 128 query values per lane and spill: the chunk kernel serves it.
  return g == 1 || g == 2 || g == 4 || (g == 8 && head_dim_qk == 64);
}

template <bool F8, bool SP>
cudaError_t launch_f(const DecodeParams& p, int items, int head_dim, int num_sms, cudaStream_t stream) {
  const int g = p.heads / p.kv_heads;
  if (head_dim == 128) {
    if (g == 1) return launch_t<128, 1, F8, SP>(p, items, num_sms, stream);
    if (g == 2) return launch_t<128, 2, F8, SP>(p, items, num_sms, stream);
    if (g == 4) return launch_t<128, 4, F8, SP>(p, items, num_sms, stream);
  } else if (head_dim == 64) {
    if (g == 1) return launch_t<64, 1, F8, SP>(p, items, num_sms, stream);
    if (g == 2) return launch_t<64, 2, F8, SP>(p, items, num_sms, stream);
    if (g == 4) return launch_t<64, 4, F8, SP>(p, items, num_sms, stream);
    if (g == 8) return launch_t<64, 8, F8, SP>(p, items, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeParams& p, int items, int head_dim, bool fp8, bool topk, int num_sms,
                          cudaStream_t stream) {
  if (topk)
    return fp8 ? launch_f<true, true>(p, items, head_dim, num_sms, stream)
               : launch_f<false, true>(p, items, head_dim, num_sms, stream);
  return fp8 ? launch_f<true, false>(p, items, head_dim, num_sms, stream)
             : launch_f<false, false>(p, items, head_dim, num_sms, stream);
}

}  // namespace vpp
