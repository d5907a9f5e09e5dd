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
// Work item = (row, key range of split_tokens keys).  A CTA takes one item,
// or, when the launch caps the CTA count, every ctas-th item in turn:
//   warp Hkv (last)   producer: for every 16-token step, one 1-D bulk copy of
//                     the step's K rows and four of its V rows (16 tokens x
//                     all kv heads are contiguous inside a 64-token block),
//                     into a ring of shared-memory stages with full/empty
//                     mbarriers.  The V rows go in four groups of 4 tokens
//                     shifted by a few 16-byte units (v_row), so that the
//                     fragment loads below spread over the banks.
//   warps 0..Hkv-1    warp h serves kv head h and its G <= 8 query heads, on
//                     the tensor cores (warp-level mma.sync m16n8k16, f32
//                     accumulation): S^T = K Q^T, an online softmax per head
//                     (running max and denominator, rescale only when the max
//                     grows by more than 2^8), O^T += V^T P^T.  The CUDA cores
//                     keep the softmax and the fragment shuffles; the G
//                     multiply-adds per cached element leave them.
// A range's result is final when the row has one range; otherwise the float32
// partial output and its LSE go to the workspace and decode_merge combines
// them ("02 · 并行策略与 PP 切分" note, §7).  HBM-bound: the algorithmic bytes
// are ctx x Hkv x (dq + dv) x element bytes per row plus q, out and the
// partials.
//
// bf16 cache: bf16 operands, read from the stages as they are.  fp8 cache
// (F8): the stages hold E4M3 codes, widened exactly to f16 operands (every
// E4M3 value is an f16 value); q is scaled per head by a power of two into
// f16's range.  kv head h's k_scale joins its score scale and its v_scale
// multiplies the output, so the cache bytes per row halve.
//
// Top-k mode (SP): the rows are the query tokens of one prefill chunk and each
// attends only the key positions its index row lists (DSA-style sparse
// attention: VPP technical review §7; "02 · 并行策略与 PP 切分" §5.1).  A work
// item is (token, range of 1024 list entries).  Gather warps (four for bf16,
// two for fp8) issue a step's 16 listed keys as one bulk copy per key for K
// and one for V, with the list and block-table loads resolved a group of
// steps ahead.  Entries outside 0 .. position, or in a block outside the
// pool, are zero-filled, masked out of the softmax and reported as
// VPP_ERR_INVALID.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "decode.cuh"
#include "ptx.cuh"

namespace vpp {
namespace {

constexpr int kStepTokens = 16;
// Top-k: warps issuing a step's per-key copies.  One warp issues a bulk copy
// about every 85 cycles, so bf16's 64 KB steps need four; fp8 (two CTAs per
// SM) runs best with two.
template <bool F8> constexpr int gather_warps() { return F8 ? 2 : 4; }
// Stage ring: six fp8 stages (32 rows of 1 KB + group and row padding) or
// three bf16 stages of 64 KB, for 8 kv heads of d 128.
constexpr int kDecodeRing = 6 * (32 * 1024 + 640);
// fp8: half the ring, three stages, so that two CTAs share an SM: decode rows
// measured 6% faster, and top-k gathers 1.2-1.5x faster, than with one CTA and
// six stages.  (bf16 stages are 64 KB: one CTA per SM.)
template <bool F8> constexpr int ring_bytes() { return F8 ? kDecodeRing / 2 : kDecodeRing; }
template <bool F8> constexpr int smem_bytes() { return ring_bytes<F8>() + 4096 + 256; }  // + p exchange, barriers
constexpr float kLn2d = 0.69314718055994530942f;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

// Two floats -> f16x2 (round to nearest even), `lo` in bits 0-15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// D (16 x 8, f32) += A (16 x 16, row-major fragment) * B (16 x 8, column
// fragment), f16 or bf16 operands: the warp-level tensor-core product.
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Offset of V row t in a stage: the K rows (kbytes), then the V rows in four
// groups of 4 tokens, each group contiguous and shifted by a few 16-byte
// units.  The four lanes of a P V fragment group read the same dims of four
// tokens, one from each group; with the shifts (fp8: 0, 32, 64, 96 bytes;
// bf16: 0, 16, 64, 80 bytes, whose lanes read 32 bytes in two 16-byte loads)
// the eight lanes of each quarter warp hit eight different bank groups.
// Top-k (SP): a lane of the group reads tokens 2u, 2u + 1, 2u + 8, 2u + 9
// instead, so the shift follows the token pair (t / 2) mod 4, and the second
// eight rows move 128 bytes further so that no row overlaps the next.
template <bool F8, bool SP>
__host__ __device__ constexpr int v_row(int t, int kbytes, int row_bytes) {
  const int g = SP ? (t >> 1) & 3 : t >> 2;
  return kbytes + t * row_bytes + (F8 ? 32 * g : 16 * (g & 1) + 64 * (g >> 1)) + (SP ? 128 * (t >> 3) : 0);
}
// The V area of a stage: 16 rows plus at most 256 bytes of shifts.
constexpr int kVShiftBytes = 256;

// Every V row of a stage is 16-byte aligned, ends before the next begins and
// inside the V area, for every row size the kernels use (a multiple of 64).
template <bool F8, bool SP>
constexpr bool v_rows_ok() {
  for (int rb = 64; rb <= 8 * 128 * (F8 ? 1 : 2); rb += 64) {
    for (int t = 0; t < kStepTokens; ++t) {
      const int a = v_row<F8, SP>(t, 0, rb);
      const int next = t + 1 < kStepTokens ? v_row<F8, SP>(t + 1, 0, rb) : kStepTokens * rb + kVShiftBytes;
      if (a % 16 != 0 || a + rb > next) return false;
    }
  }
  return true;
}
static_assert(v_rows_ok<false, false>() && v_rows_ok<false, true>() && v_rows_ok<true, false>() &&
                  v_rows_ok<true, true>(),
              "V rows of a stage overlap or leave the stage");

// Transposes an 8x8 matrix of 16-bit values held one row pair per lane
// (lane 4 r + c: row r, columns 2c and 2c + 1).
__device__ __forceinline__ uint32_t transpose8x8_b16(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// One work item: keys [t_begin, t_end) of a decode row (top-k: list entries
// [t_begin, t_end) of a query token), range `split` of the row's n_splits.
struct DecodeItem {
  DecodeRow row;
  int split, n_splits, t_begin, t_end, n_steps;
  const int32_t* list;  // SP: the token's index row
  int64_t pos;          // SP: the token's absolute position
  bool skip;            // SP: the token's list is shorter than this range (no work, nothing written)
};

// `report`: the one thread that records a top-k list length out of range.
template <bool SP>
__device__ __forceinline__ DecodeItem decode_item(const DecodeParams& p, int item, bool report) {
  DecodeItem it;
  it.list = nullptr;
  it.pos = 0;
  it.skip = false;
  if (SP) {
    const int64_t i = item / p.topk_splits;
    it.split = item - static_cast<int>(i * p.topk_splits);
    int n = __ldg(p.topk_len + i);
    if (n < 1 || n > p.topk) {
      if (report && it.split == 0) record_status(p.status, kStatusInvalid);
      n = 0;
    }
    it.row.b = 0;
    it.row.q_row = static_cast<int32_t>(i);
    it.row.ctx = n;
    it.row.item0 = static_cast<int32_t>(i * p.topk_splits);
    it.list = p.topk_idx + i * p.topk;
    it.pos = p.topk_prefix + i;
    it.n_splits = n > 0 ? (n + p.split_tokens - 1) / p.split_tokens : 1;
    it.skip = it.split >= it.n_splits;
  } else {
    int lo = 0, hi = p.n_rows - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.rows[mid].item0 <= item) lo = mid; else hi = mid - 1;
    }
    it.row = p.rows[lo];
    it.split = item - it.row.item0;
    it.n_splits = (it.row.ctx + p.split_tokens - 1) / p.split_tokens;
  }
  it.t_begin = it.split * p.split_tokens;
  it.t_end = min(it.row.ctx, it.t_begin + p.split_tokens);
  it.n_steps = it.skip ? 0 : (it.t_end - it.t_begin + kStepTokens - 1) / kStepTokens;
  return it;
}

// Persistent: CTA b takes items b, b + gridDim.x, ... in turn; each role
// keeps its place in the stage ring from one item to the next, so that the
// producer fills the ring with the next item's rows while the kv-head warps
// finish the current one.
template <int D, int G, bool F8, bool SP>
__global__ void __launch_bounds__(SP ? 32 * (8 + gather_warps<F8>()) : 288, F8 ? 2 : 1)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int ESZ = F8 ? 1 : 2;  // cache bytes per element
  extern __shared__ __align__(128) uint8_t smem[];
  const int hkv = p.kv_heads;
  const int row_bytes = hkv * D * ESZ;               // one token, all kv heads
  // A stage holds a step's 16 K rows as they lie in the cache (one bulk
  // copy), then its V rows in four groups of 4 tokens (one copy each; see
  // v_row).  (Padding every V row of a decode step instead needs 32 copies
  // per step, which measured 1.6x slower.)
  // Top-k K rows are copied one by one: padding after each puts the rows of
  // a fragment load in different banks (see the K reads).
  const int kstride = SP ? row_bytes + (F8 ? 16 : 64) : row_bytes;
  const int kbytes = kStepTokens * kstride;
  const int stage_bytes = kbytes + kStepTokens * row_bytes + kVShiftBytes;
  constexpr int kRing = ring_bytes<F8>();
  const int nstage = min(8, kRing / stage_bytes);
  float* pbuf = reinterpret_cast<float*>(smem + kRing);  // [hkv][16][G]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRing + 8 * kStepTokens * 8 * 4);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(bars + 16);
  uint32_t* step_valid = reinterpret_cast<uint32_t*>(bars + 17);  // SP: valid-entry mask per stage
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The ring starts zeroed.  A short step copies only its valid rows, so the
  // rows past them hold rows of an earlier step (finite cache values) or
  // zeros, and their P = 0 adds exactly nothing: the V fragments need no
  // mask.  (The fence orders these writes before the ring's bulk copies.)
  for (int i = threadIdx.x; i < kRing / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < nstage; ++i) {
      mbar_init(smem_u32(&bars[i]), SP ? gather_warps<F8>() : 1);
      mbar_init(smem_u32(&bars[8 + i]), hkv);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (SP && warp >= hkv) {
    // ------------------------------------------------------ gather warps
    // The NG gather warps share a step's 32 copies, the K row (c < 16) and
    // the V row (c >= 16) of each of its 16 listed keys: copy c is issued by
    // lane c / NG of gather warp c % NG.  The rows of the list entries are
    // resolved ahead, a group of 8 steps (128 entries) at a time (lane l
    // holds entries l + 32 j of a group): while group g is copied, the
    // block-table entries of group g + 1 and the list entries of group g + 2
    // are in flight, so that these dependent loads stay off the copy path.
    // Every gather warp resolves the rows itself and arrives on the stage's
    // full barrier with its own bytes.
    const int gw = warp - hkv;
    constexpr int NG = gather_warps<F8>();
    const int c = gw + NG * lane;  // this lane's copy (c < 32)
    const int t = c & 15;
    const bool is_v = c >= 16;
    int32_t key_a[4], blk_a[4], key_b[4];  // group g + 1: keys, table entries; group g + 2: keys
    int64_t row_c[4];                      // group g: source rows, -1 if invalid or past the range
    int t_begin = 0, t_end = 0;     // the current item's range of list entries
    const int32_t* list = nullptr;  // its token's index row
    int64_t pos = 0;                // its token's absolute position
    auto load_keys = [&](int grp, int32_t (&k)[4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = t_begin + grp * 128 + 32 * j + lane;
        k[j] = e < t_end ? __ldg(list + e) : -1;
      }
    };
    auto load_blocks = [&](const int32_t (&k)[4], int32_t (&bk)[4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        bk[j] = (p.block_table && k[j] >= 0 && k[j] <= pos) ? __ldg(p.block_table + k[j] / kBlockTokens) : 0;
    };
    auto resolve = [&](int grp) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = t_begin + grp * 128 + 32 * j + lane;
        const int64_t key = key_a[j];
        bool valid = false;
        int64_t r = -1;
        if (key >= 0 && key <= pos) {
          if (p.block_table) {
            valid = blk_a[j] >= 0 && blk_a[j] < p.num_blocks;
            r = static_cast<int64_t>(blk_a[j]) * kBlockTokens + key % kBlockTokens;
          } else {
            valid = key < p.num_blocks;  // contiguous cache: num_blocks is the capacity in tokens
            r = key;
          }
        }
        if (e < t_end && !valid && gw == 0) record_status(p.status, kStatusInvalid);
        row_c[j] = (e < t_end && valid) ? r : -1;
      }
    };
    int slot = 0;
    uint32_t phase = 0u;
    uint32_t filled = 0u, fill_phase = 0u;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
      const DecodeItem it = decode_item<SP>(p, item, false);
      if (it.skip) continue;
      t_begin = it.t_begin;
      t_end = it.t_end;
      list = it.list;
      pos = it.pos;
      const int n_steps = it.n_steps;
      load_keys(0, key_a);
      load_blocks(key_a, blk_a);
      load_keys(1, key_b);
      for (int s = 0; s < n_steps; ++s) {
        if ((s & 7) == 0) {
          resolve(s >> 3);
#pragma unroll
          for (int j = 0; j < 4; ++j) key_a[j] = key_b[j];
          load_blocks(key_a, blk_a);
          load_keys((s >> 3) + 2, key_b);
        }
        const int t0 = t_begin + s * kStepTokens;
        const int nt = min(kStepTokens, t_end - t0);
        const int kq = (s & 7) >> 1;
        const int64_t mine = kq == 0 ? row_c[0] : kq == 1 ? row_c[1] : kq == 2 ? row_c[2] : row_c[3];
        // the step's validity word (lane l < 16: entry l), then this lane's row
        const int64_t rl = __shfl_sync(0xffffffffu, mine, (s & 1) * 16 + (lane & 15));
        const uint32_t vmask = __ballot_sync(0xffffffffu, lane < 16 && rl >= 0) & 0xFFFFu;
        const int64_t src_row = __shfl_sync(0xffffffffu, mine, (s & 1) * 16 + t);
        const bool mine_in = c < 32 && t < nt;
        const bool valid = mine_in && ((vmask >> t) & 1u);
        const uint32_t cmask = __ballot_sync(0xffffffffu, valid);
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(smem_u32(&bars[8 + slot]), phase ^ 1u, p.status, abort_flag);
        if (!__shfl_sync(0xffffffffu, w_ok ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        uint8_t* dstp = smem + slot * stage_bytes + (is_v ? v_row<F8, true>(t, kbytes, row_bytes) : t * kstride);
        if (mine_in && !valid) {  // zero-filled, so that P = 0 times it stays 0
          for (int b = 0; b < row_bytes; b += 16) *reinterpret_cast<uint4*>(dstp + b) = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();  // before later bulk copies into these bytes
        }
        __syncwarp();
        const uint32_t full = smem_u32(&bars[slot]);
        if (lane == 0) {
          if (gw == 0) step_valid[slot] = vmask;
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(cmask)) * row_bytes);
        }
        __syncwarp();
        if (valid) {
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
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
        const DecodeItem it = decode_item<SP>(p, item, false);
        if (it.skip) continue;
        const DecodeRow row = it.row;
        const int t_begin = it.t_begin, t_end = it.t_end, n_steps = it.n_steps;
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
            for (int g4 = 0; 4 * g4 < nt; ++g4)
              bulk_g2s(dst + v_row<F8, false>(4 * g4, kbytes, row_bytes), vsrc + 4 * g4 * row_bytes,
                       static_cast<uint32_t>(min(4, nt - 4 * g4) * row_bytes), full);
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
      }
      if (!ok) {
        for (int i = 0; i < nstage; ++i)
          if (filled & (1u << i)) mbar_wait_for(smem_u32(&bars[i]), (fill_phase >> i) & 1u, 100000000ull);
      }
    }
  } else if (warp < hkv) {
    // ------------------------------------------------------ kv head `warp`
    // Both products run on the tensor cores (mma.sync m16n8k16, f16 operands,
    // f32 accumulation).  Lane = 4 g + u: g is the fragment's group (a token
    // row of S^T, a dim row of O^T, a head column of the B operands), u the
    // thread in the group.
    //   S^T[16 tokens x 8 heads] = K[16 x D] Q^T[D x 8]: k-step s, logical
    //     k = 2u + b + 8c maps to dim u D/4 + 4s + 2c + b, so a thread's
    //     codes of one token are D/4 consecutive ones.  (bf16 top-k: the
    //     same D/4 positions are taken from the 8-dim pieces 4c' + u, for
    //     q and K alike.)
    //   O^T[D x 8 heads] += V^T[D x 16 tokens] P^T[16 x 8]: tile i, row g
    //     is dim g D/8 + 2i, row g + 8 is dim g D/8 + 2i + 1; logical
    //     k = 2u + b + 8c maps to token 4u + b + 2c, so a thread reads D/8
    //     consecutive codes of each token of V group u, and P goes through
    //     shared memory.  (Top-k: k maps to token k itself, so P^T's
    //     fragment is P's accumulator fragment transposed in registers, and
    //     a thread reads tokens 2u, 2u + 1, 2u + 8, 2u + 9.)
    // Heads >= G are zero columns.  E4M3 codes widen exactly to f16; q is
    // scaled by a power of two per head into f16's range (undone on the
    // scores), P is in [0, 256].
    const int h = warp;
    const int gq = lane >> 2;
    const int u = lane & 3;
    constexpr int KS = D / 16;  // k-steps of S, tiles of O
    float* pw = pbuf + h * kStepTokens * 8;  // P of the step: [16 tokens][8 heads]
    int slot = 0;
    uint32_t phase = 0u;
    bool ok = true;
    // bf16 top-k: lane u's 16-byte pieces of a row are pieces 4c + u (see the
    // K reads); otherwise its D/4 elements are contiguous.
    constexpr bool kInterleaved = SP && !F8;
    // This lane's bf16 q words of an item (query head h G + gq; zeros for
    // gq >= G).  With a capped CTA count the next item's words are loaded
    // while the current item runs, so that an item starts without waiting
    // for them (fp8, two CTAs per SM, has no registers to spare for it).
    constexpr bool kPrefetchQ = !F8;
    auto load_q = [&](const DecodeItem& x, uint4 (&w)[D / 32]) {
      const uint4* qrow = reinterpret_cast<const uint4*>(
          p.q + (static_cast<int64_t>(x.row.q_row) * p.heads + h * G + min(gq, G - 1)) * D);
      const uint4* qsrc = kInterleaved ? qrow + u : qrow + u * (D / 32);
#pragma unroll
      for (int c = 0; c < D / 32; ++c)
        w[c] = (gq < G && !x.skip) ? __ldg(qsrc + (kInterleaved ? 4 * c : c)) : make_uint4(0u, 0u, 0u, 0u);
    };
    int item = blockIdx.x;
    DecodeItem it_next;
    uint4 q_next[D / 32];
    if (kPrefetchQ && item < p.n_items) {
      it_next = decode_item<SP>(p, item, threadIdx.x == 0);
      load_q(it_next, q_next);
    }
    for (; ok && item < p.n_items; item += gridDim.x) {
      DecodeItem it;
      uint4 q_cur[D / 32];
      if (kPrefetchQ) {
        it = it_next;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) q_cur[c] = q_next[c];
        if (item + static_cast<int>(gridDim.x) < p.n_items) {
          it_next = decode_item<SP>(p, item + gridDim.x, threadIdx.x == 0);
          load_q(it_next, q_next);
        }
      } else {
        it = decode_item<SP>(p, item, threadIdx.x == 0);
        load_q(it, q_cur);
      }
      if (it.skip) continue;  // the token's list is shorter: no work, nothing written
      const DecodeRow row = it.row;
      const int t_begin = it.t_begin, t_end = it.t_end, n_steps = it.n_steps, n_splits = it.n_splits;
      uint32_t qb[KS][2];
      float qscale = 1.f;  // fp8: 2^-e of head gq
      if (!F8) {
        // bf16 operands: q's pairs are the B fragment as they are.
        uint32_t qw[D / 8];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint4 w = q_cur[c];
          qw[4 * c] = w.x;
          qw[4 * c + 1] = w.y;
          qw[4 * c + 2] = w.z;
          qw[4 * c + 3] = w.w;
        }
#pragma unroll
        for (int s2 = 0; s2 < KS; ++s2) {
          qb[s2][0] = qw[2 * s2];
          qb[s2][1] = qw[2 * s2 + 1];
        }
      } else {
        // f16 operands: q scaled per head by a power of two into f16's range.
        float qv[D / 4];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint4 w = q_cur[c];
          bf16x2_to_f32(w.x, qv[8 * c + 0], qv[8 * c + 1]);
          bf16x2_to_f32(w.y, qv[8 * c + 2], qv[8 * c + 3]);
          bf16x2_to_f32(w.z, qv[8 * c + 4], qv[8 * c + 5]);
          bf16x2_to_f32(w.w, qv[8 * c + 6], qv[8 * c + 7]);
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
      const float sl = F8 ? p.scale_log2 * __ldg(p.k_scale + h) : p.scale_log2;
      const float slh[2] = {sl * __shfl_sync(0xffffffffu, qscale, 8 * u),
                            sl * __shfl_sync(0xffffffffu, qscale, 8 * u + 4)};
      const float vsc = F8 ? __ldg(p.v_scale + h) : 1.f;
      float m[2] = {-INFINITY, -INFINITY};
      float lpart[2] = {0.f, 0.f};
      float o[KS][4];
#pragma unroll
      for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      for (int s = 0; s < n_steps; ++s) {
        const int t0 = t_begin + s * kStepTokens;
        const int nt = min(kStepTokens, t_end - t0);
        ok = mbar_wait(smem_u32(&bars[slot]), phase, p.status, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint8_t* kst = smem + slot * stage_bytes;
        const uint32_t vmask = SP ? step_valid[slot] : 0xFFFFu;
        // ---- S^T = K Q^T (two accumulator chains)
        // A thread reads KW words (D/4 elements) of each of its two token rows.
        // Decode rows lie a multiple of 128 bytes apart, so a quarter warp's
        // two groups would hit the same banks: the 16-byte pieces are read in
        // an order that depends on the lane (and put back in place by
        // selects).  Top-k rows are copied one by one and padded instead (16
        // bytes past such a multiple for fp8, 64 for bf16, whose lanes take
        // interleaved pieces), and read in order: 7-12% faster top-k than the
        // lane-dependent order.
        constexpr int KW = D * ESZ / 16;  // 32-bit words of a thread's part of one K row
        uint32_t kw[2][KW];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          uint4 w[KW / 4];
          const uint4* src = reinterpret_cast<const uint4*>(kst + (gq + 8 * rr) * kstride +
                                                            (h * D + (kInterleaved ? 0 : u * (D / 4))) * ESZ);
          if (kInterleaved) {
            // pieces 4c + u: the four lanes of a group read four consecutive
            // 16-byte units, and rows 64 bytes past a multiple of 128 put the
            // next group's row in the other half of the banks
#pragma unroll
            for (int c = 0; c < KW / 4; ++c) w[c] = src[4 * c + u];
          } else if (KW / 4 == 4) {
            const int r = SP ? 0 : (u >> 1) | ((gq & 1) << 1);
#pragma unroll
            for (int c = 0; c < 4; ++c) w[c] = src[c ^ r];
            // w[c] holds piece c ^ r: two conditional swaps put piece j in w[j]
            if (r & 1) {
              const uint4 t0 = w[0], t2 = w[2];
              w[0] = w[1]; w[1] = t0; w[2] = w[3]; w[3] = t2;
            }
            if (r & 2) {
              const uint4 t0 = w[0], t1 = w[1];
              w[0] = w[2]; w[1] = w[3]; w[2] = t0; w[3] = t1;
            }
          } else if (KW / 4 == 2) {
            const int sw = SP ? 0 : gq & 1;
            const uint4 wa = src[sw], wb = src[sw ^ 1];
            w[0] = sw ? wb : wa;
            w[1 % (KW / 4)] = sw ? wa : wb;
          } else {
            w[0] = src[0];
          }
#pragma unroll
          for (int c = 0; c < KW / 4; ++c) {
            kw[rr][4 * c] = w[c].x;
            kw[rr][4 * c + 1] = w[c].y;
            kw[rr][4 * c + 2] = w[c].z;
            kw[rr][4 * c + 3] = w[c].w;
          }
        }
        // NCH independent accumulator chains (bf16: four, 4% faster than two;
        // fp8, two CTAs per SM, keeps two for registers), summed after.
        constexpr int NCH = (F8 || KS < 4) ? 2 : 4;
        float sa[NCH][4];
#pragma unroll
        for (int j = 0; j < NCH; ++j) sa[j][0] = sa[j][1] = sa[j][2] = sa[j][3] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < KS; ++s2) {
          if (F8) {
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_f16x2x2(kw[0][s2 % KW], a0, a2);
            e4m3x4_to_f16x2x2(kw[1][s2 % KW], a1, a3);
            mma_16816(sa[s2 % NCH], a0, a1, a2, a3, qb[s2][0], qb[s2][1]);
          } else {
            mma_16816_bf16(sa[s2 % NCH], kw[0][(2 * s2) % KW], kw[1][(2 * s2) % KW], kw[0][(2 * s2 + 1) % KW],
                           kw[1][(2 * s2 + 1) % KW], qb[s2][0], qb[s2][1]);
          }
        }
        if (NCH == 4) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sa[0][e] += sa[2 % NCH][e];
            sa[1][e] += sa[3 % NCH][e];
          }
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
        float pvr[2][2];  // top-k: P of tokens gq, gq + 8 for heads 2u, 2u + 1
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
            if (SP) {
              pvr[rr][hh] = pv;
            } else {
              pw[(gq + 8 * rr) * 8 + 2 * u + hh] = pv;
            }
          }
        }
        // ---- O^T += V^T P^T
        uint32_t pb0, pb1;
        if (SP) {
          // P^T's B fragment is the transpose of P in the accumulator layout:
          // tokens 2u, 2u + 1 (and + 8) of head gq after one 8x8 transpose each
          pb0 = transpose8x8_b16(F8 ? pack_f16x2(pvr[0][0], pvr[0][1]) : pack_bf16x2(pvr[0][0], pvr[0][1]));
          pb1 = transpose8x8_b16(F8 ? pack_f16x2(pvr[1][0], pvr[1][1]) : pack_bf16x2(pvr[1][0], pvr[1][1]));
        } else {
          __syncwarp();
          pb0 = F8 ? pack_f16x2(pw[(4 * u) * 8 + gq], pw[(4 * u + 1) * 8 + gq])
                   : pack_bf16x2(pw[(4 * u) * 8 + gq], pw[(4 * u + 1) * 8 + gq]);
          pb1 = F8 ? pack_f16x2(pw[(4 * u + 2) * 8 + gq], pw[(4 * u + 3) * 8 + gq])
                   : pack_bf16x2(pw[(4 * u + 2) * 8 + gq], pw[(4 * u + 3) * 8 + gq]);
        }
        // tokens 4u .. 4u + 3 (top-k: 2u, 2u + 1, 2u + 8, 2u + 9): this
        // thread's D/8 elements of each
        constexpr int VW = D * ESZ / 32;  // 32-bit words of them
        uint32_t vw[4][VW];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int t = SP ? 2 * u + (q4 & 1) + 8 * (q4 >> 1) : 4 * u + q4;
          const uint8_t* src = kst + v_row<F8, SP>(t, kbytes, row_bytes) + (h * D + gq * (D / 8)) * ESZ;
          uint32_t w[VW];
          if (VW == 8) {
            const uint4 w0 = reinterpret_cast<const uint4*>(src)[0];
            const uint4 w1 = reinterpret_cast<const uint4*>(src)[1];
            w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
            w[4 % VW] = w1.x; w[5 % VW] = w1.y; w[6 % VW] = w1.z; w[7 % VW] = w1.w;
          } else if (VW == 4) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(src);
            w[0] = w0.x; w[1 % VW] = w0.y; w[2 % VW] = w0.z; w[3 % VW] = w0.w;
          } else {
            const uint2 w0 = *reinterpret_cast<const uint2*>(src);
            w[0] = w0.x; w[1 % VW] = w0.y;
          }
#pragma unroll
          for (int c = 0; c < VW; ++c) vw[q4][c] = w[c];
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < KS; ++i) {
          uint32_t a0, a1, a2, a3;
          if (F8) {
            const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
            const uint32_t x = __byte_perm(vw[0][(i >> 1) % VW], vw[1][(i >> 1) % VW], sel);
            const uint32_t y = __byte_perm(vw[2][(i >> 1) % VW], vw[3][(i >> 1) % VW], sel);
            e4m3x4_to_f16x2x2(x, a0, a1);
            e4m3x4_to_f16x2x2(y, a2, a3);
            mma_16816(o[i], a0, a1, a2, a3, pb0, pb1);
          } else {
            // word i of a token holds dims 2i, 2i + 1 of the thread's part
            a0 = __byte_perm(vw[0][i % VW], vw[1][i % VW], 0x5410u);
            a1 = __byte_perm(vw[0][i % VW], vw[1][i % VW], 0x7632u);
            a2 = __byte_perm(vw[2][i % VW], vw[3][i % VW], 0x5410u);
            a3 = __byte_perm(vw[2][i % VW], vw[3][i % VW], 0x7632u);
            mma_16816_bf16(o[i], a0, a1, a2, a3, pb0, pb1);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[8 + slot]));
        if (++slot == nstage) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
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
cudaError_t launch_t(const DecodeParams& p, int items, int ctas, int num_sms, cudaStream_t st) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<D, G, F8, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<F8>());
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int warps = p.kv_heads + (SP ? gather_warps<F8>() : 1);
  // item + gridDim.x stays below 2^31 in the kernels' item loops
  if (items < 0 || items > INT32_MAX / 2) return cudaErrorInvalidValue;
  DecodeParams pk = p;
  pk.n_items = items;
  const int ctas_used = ctas > 0 ? std::min(items, ctas) : items;
  decode_kernel<D, G, F8, SP><<<ctas_used, 32 * warps, smem_bytes<F8>(), st>>>(pk);
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
  return g == 1 || g == 2 || g == 4 || g == 8;
}

template <bool F8, bool SP>
cudaError_t launch_f(const DecodeParams& p, int items, int head_dim, int num_sms, int ctas, cudaStream_t stream) {
  const int g = p.heads / p.kv_heads;
  if (head_dim == 128) {
    if (g == 1) return launch_t<128, 1, F8, SP>(p, items, ctas, num_sms, stream);
    if (g == 2) return launch_t<128, 2, F8, SP>(p, items, ctas, num_sms, stream);
    if (g == 4) return launch_t<128, 4, F8, SP>(p, items, ctas, num_sms, stream);
    if (g == 8) return launch_t<128, 8, F8, SP>(p, items, ctas, num_sms, stream);
  } else if (head_dim == 64) {
    if (g == 1) return launch_t<64, 1, F8, SP>(p, items, ctas, num_sms, stream);
    if (g == 2) return launch_t<64, 2, F8, SP>(p, items, ctas, num_sms, stream);
    if (g == 4) return launch_t<64, 4, F8, SP>(p, items, ctas, num_sms, stream);
    if (g == 8) return launch_t<64, 8, F8, SP>(p, items, ctas, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeParams& p, int items, int head_dim, bool fp8, bool topk, int num_sms,
                          int ctas, cudaStream_t stream) {
  if (topk)
    return fp8 ? launch_f<true, true>(p, items, head_dim, num_sms, ctas, stream)
               : launch_f<false, true>(p, items, head_dim, num_sms, ctas, stream);
  return fp8 ? launch_f<true, false>(p, items, head_dim, num_sms, ctas, stream)
             : launch_f<false, false>(p, items, head_dim, num_sms, ctas, stream);
}

}  // namespace vpp
