// chunk_attn_impl.cuh -- a2..a6: causal attention of one prefill chunk (or of
// several prefill segments of a mixed batch) over its cached prefix plus
// itself, on tcgen05 tensor cores.
//
// Method: Eq. (1) of "VPP: Virtual Pipeline Parallelism for Efficient Chunked
// Prefill in Long-Context LLM Inference" (technical review, §2.2),
// softmax(Q K^T / sqrt(d)) V, with token i attending to tokens <= i, for a
// chunk whose first token sits at absolute position P = kv_len - q_len (§2.3:
// a later chunk attends to the whole cached prefix plus itself).  The softmax
// is evaluated online over 128-key tiles (running max m and denominator l per
// row, exact after the final division); the result and ln(denominator) are
// written, or, when the key range is split, float32 partials and their LSE for
// the merge kernel ("02 · 并行策略与 PP 切分" note, §7: partial results over
// disjoint key ranges are combined through their LSE).
//
// CTA shape (384 threads over a bf16 cache, one CTA per SM):
//   warp 0      TMA producer: the CTA's two 128-row query tiles once, then K
//               and V tiles through a ring of 16 KB shared-memory slots (128
//               keys x 64 dims each).  A K tile takes dq/64 consecutive slots
//               and a V tile dv/64 (wrapping at the ring's end); each tile has
//               one full and one empty mbarrier, and slots are reused in order
//               as tiles are released.
//   warp 1, 3   MMA issuers, one elected lane each: warp 1 for query tile A,
//               warp 3 for tile B.  S = Q K^T into TMEM (kind::f16, bf16 in,
//               f32 accumulate), then O += P V with P read from TMEM (for
//               d_qk <= 128 as two chains: keys [0, 64) as soon as the
//               softmax has stored their P, keys [64, 128) once the rest is
//               stored).  Each
//               issuer emits blocks [PV(x, j-1), QK(x, j)] and the two take
//               turns (a shared counter, handed over four MMAs before the end
//               of a block), so the tensor core runs A's block j, B's block j,
//               A's block j+1, ...: the softmax of one tile runs
//               while the tensor core works on the other tile's block, and the
//               waits, commits and fences of one issuer (each leaves the tensor
//               core idle if it sits between the MMAs of a single issuing
//               thread) overlap the other issuer's MMAs.  With d_qk = 192 the
//               V tile is released right after its P V MMAs (see EARLY_V).
//   warp 2      allocates and frees the 512 TMEM columns.
//   warps 4-7   softmax + epilogue of query tile A; warps 8-11 of tile B.
//               Each thread owns one query row = one TMEM lane, so row max and
//               row sum need no shuffles.  The TMA/MMA warpgroup runs on 64
//               registers per thread so that the softmax threads get 216 and
//               hold a whole 128-score row without spilling.
//   Over an fp8 cache the CTA has 512 threads: warps 12-15 (one per SM
//               sub-partition) copy the K/V codes into staging slots and widen
//               them into the ring, and warpgroup 0 widens Q in place.
// TMEM columns: S_A [0,128) S_B [128,256) O_A [256,256+DV) O_B [256+DV,256+2DV).
// P (bf16 pairs) overwrites the first 64 columns of its S tile.
//
// Query rows: a 128-row tile holds 128/G consecutive tokens x the G query
// heads of one kv head (GQA packing), so every K/V tile loaded serves all
// 2 x 128 rows of the CTA.  The causal mask is applied only on tiles that
// reach past a row's position; prefix tiles are never masked.
//
// Every mbarrier wait is bounded; a timeout records VPP_ERR_TIMEOUT in the
// status word and every role leaves its loop.
#pragma once

#include <type_traits>

#include "chunk_attn.cuh"
#include "ptx.cuh"

namespace vpp {

// Tracing build only (compiled with -DVPP_TIMELINE=<cta>): clock64 stamps
// of the two MMA issuers and of the first softmax thread of each query tile,
// for CTA 0 and CTA <cta>, tiles 0..63.  The product build compiles them out.
#ifdef VPP_TIMELINE
static __device__ long long g_timeline[2][4][64][4];
__device__ __forceinline__ void timeline_stamp(int role, int j, int ev) {
  const int slot = blockIdx.x == 0 ? 0 : (blockIdx.x == VPP_TIMELINE ? 1 : -1);
  if (slot >= 0 && j < 64) g_timeline[slot][role][j][ev] = clock64();
}
#define VPP_STAMP(role, j, ev) timeline_stamp(role, j, ev)
#else
#define VPP_STAMP(role, j, ev) ((void)0)
#endif

namespace attn_detail {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay <= 256
constexpr int kRegsLow = 64;
constexpr int kRegsHigh = 216;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= 384 * 168, "register split exceeds the launch");
// Over an fp8 cache (512 threads, 128 registers each at launch) the
// converter warpgroup takes 40 and the softmax warpgroups 200.
constexpr int kRegsConvF8 = 40;
constexpr int kRegsHighF8 = 200;
static_assert(128 * kRegsLow + 128 * kRegsConvF8 + 256 * kRegsHighF8 <= 512 * 128,
              "fp8 register split exceeds the launch");
constexpr uint64_t kCleanupNs = 100000000ull;  // 0.1 s for clean-up waits after an abort

struct Ring {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ void advance(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

template <int DQ, int DV, bool F8>
struct Shape {
  static constexpr int NQC = DQ / 64;  // 64-dim sub-tiles of a K tile (and of Q)
  static constexpr int NVC = DV / 64;  // 64-dim sub-tiles of a V tile
  static constexpr int NSLOT = attn_num_slots(DQ, F8);
  static constexpr int NB = NSLOT;     // tile barriers (>= tiles that fit the ring)
  static constexpr int NSTG = F8 ? kNumStages : 0;  // staging slots of E4M3 codes
  static constexpr int NCONV = 4;                     // fp8: converter warps 12..15
  static_assert(!F8 || (NSTG % NCONV == 0 && NB % 2 == 0),
                "fp8: whole staging slots per converter; K tiles on even FULL barriers");
  static constexpr int REGS_HIGH = F8 ? kRegsHighF8 : kRegsHigh;
  static constexpr int QBYTES = attn_q_bytes(DQ);
  // Operands are bf16, or f16 over an fp8 cache (E4M3 widens exactly to f16).
  static constexpr uint32_t IDESC_QK =
      F8 ? idesc_f16_f32(kTileM, kTileN, false, false) : idesc_bf16_f32(kTileM, kTileN, false, false);
  static constexpr uint32_t IDESC_PV =
      F8 ? idesc_f16_f32(kTileM, DV, false, true) : idesc_bf16_f32(kTileM, DV, false, true);
  static constexpr uint32_t IDESC_PV64 =
      F8 ? idesc_f16_f32(kTileM, 64, false, true) : idesc_bf16_f32(kTileM, 64, false, true);
  // P V of a tile runs as two MMA chains over 16-key steps: the first covers
  // keys [0, 16 * PV0) and starts once the softmax has stored their P, while
  // the softmax still computes the exponentials of the remaining keys.  With
  // d_qk = 192 the split measured slower (the ring, not the softmax, limits
  // that shape), so it keeps one chain.
  static constexpr int PV0 = DQ > 128 ? 8 : 4;
  static constexpr int KP0 = 16 * PV0;  // keys of the first part
  static constexpr bool SPLIT_P = PV0 < kTileN / 16;  // PV0 = 8: one chain
  static_assert(PV0 >= 1 && PV0 <= kTileN / 16, "P V chain split out of range");
  // barrier indices: Q, S[2], P0[2], O[2], FINAL[2], TMP, P1[2], END, FULL[NB], EMPTY[NB],
  // STAGE[NSTG]
  static constexpr int B_Q = 0, B_S = 1, B_P = 3, B_O = 5, B_FINAL = 7, B_TMP = 9, B_P1 = 10,
                       B_END = 12, B_FULL = 13, B_EMPTY = 13 + NB, B_STG = 13 + 2 * NB,
                       NBARS = 13 + 2 * NB + NSTG;
  static_assert(NSLOT >= NQC + NVC, "ring must hold one K and one V tile");
  // With d_qk = 192 the ring holds under two K/V tile pairs, and the next K
  // tile can only start once V_{j-1} is free: V_{j-1} is released by its own
  // commit right after the P V MMAs rather than after the whole block (one
  // more commit per block, which costs the d_qk = 128 shapes more than it
  // gains them).
  static constexpr bool EARLY_V = DQ > 128;
  static_assert(DV <= 128, "O accumulators must fit TMEM next to two S tiles");
  // Tile t of the load order (K_0, V_0, K_1, V_1, ...) starts at ring position
  // tile_pos(t) (counted in slots from the first tile, not wrapped).
  __device__ __forceinline__ static int tile_pos(int t) {
    return (t >> 1) * (NQC + NVC) + ((t & 1) ? NQC : 0);
  }
  __device__ __forceinline__ static int tile_slots(int t) { return (t & 1) ? NVC : NQC; }
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* status,
                                          volatile uint32_t* abort) {
  const bool ok = mbar_wait(bar, parity, status, abort);
  return __all_sync(0xffffffffu, ok);
}

// p = 2^(s * scale * log2(e) - mref) for the scores of keys [K0, K1) of a
// row, two lanes of work per packed instruction, stored to TMEM as bf16 pairs
// (column c of the tile holds keys 2c, 2c + 1) every 16 keys, so that packed
// values do not pile up in registers; the fp32 values are added to rs4.
template <int K0, int K1, bool F16>
__device__ __forceinline__ void exps_to_tmem(const float (&sv)[128], float2 sl2, float2 nmb2,
                                             float2 (&rs4)[4], uint32_t tS) {
  static_assert(K0 % 16 == 0 && K1 % 16 == 0, "parts are whole 16-key MMA steps");
#pragma unroll
  for (int k = K0 / 16; k < K1 / 16; ++k) {
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = 8 * k + i;  // pair index
      const float2 xx = ffma2(make_float2(sv[2 * c], sv[2 * c + 1]), sl2, nmb2);
      const float a = ex2_approx(xx.x);
      const float b = ex2_approx(xx.y);
      rs4[c & 3] = fadd2(rs4[c & 3], make_float2(a, b));
      pk[i] = F16 ? pack_half2(a, b) : pack_bf16x2(a, b);
    }
    tmem_st8(tS + 8 * k, pk);
  }
}

}  // namespace attn_detail

template <int DQ, int DV, bool F8>
__global__ void __launch_bounds__(attn_threads(F8), 1)
    chunk_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ AttnParams p) {
  using namespace attn_detail;
  using S = Shape<DQ, DV, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + S::QBYTES;
  uint8_t* sStage = sRing + S::NSLOT * kSubTileBytes;  // fp8 cache only
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + S::NSTG * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::NBARS);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(tmem_slot + 1);
  volatile int* turn = reinterpret_cast<volatile int*>(tmem_slot + 2);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------------------------------------------------- work item
  int si = 0;
  while (si + 1 < p.n_segs && p.segs[si + 1].cta_begin <= static_cast<int>(blockIdx.x)) ++si;
  const AttnSeg& seg = p.segs[si];
  const int local = static_cast<int>(blockIdx.x) - seg.cta_begin;
  // CTA order: key range fastest, then query-tile pairs (heaviest first), then
  // kv head, so the CTAs resident at one time read the same kv head's K/V
  // tiles and share them through L2.
  const int split = local % seg.n_splits;
  const int rest = local / seg.n_splits;
  const int pair = seg.n_pairs - 1 - rest % seg.n_pairs;
  const int g = rest / seg.n_pairs;
  const int G = p.group;
  const int T = kTileM / G;       // tokens per query tile
  const int tok0 = pair * 2 * T;  // first token of tile A (segment-relative)
  const int P = seg.kv_len - seg.q_len;
  const int k_lo = split * seg.split_keys;
  const int k_hi = (split == seg.n_splits - 1) ? P + min(tok0 + 2 * T, seg.q_len)
                                               : (split + 1) * seg.split_keys;
  const int n_kv = (k_hi - k_lo + kTileN - 1) / kTileN;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *turn = 0;
    mbar_init(bar(S::B_Q), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(S::B_S + x), 1);
      mbar_init(bar(S::B_P + x), 128);
      mbar_init(bar(S::B_P1 + x), 128);
      mbar_init(bar(S::B_O + x), 1);
      mbar_init(bar(S::B_FINAL + x), 1);
    }
    mbar_init(bar(S::B_TMP), 1);
    mbar_init(bar(S::B_END), 10);  // the 8 softmax warps and the 2 MMA issuers
    for (int i = 0; i < S::NB; ++i) {
      // over an fp8 cache a tile is full once both halves of each of its
      // sub-tiles are widened
      // (K tiles, even t, use even barriers)
      mbar_init(bar(S::B_FULL + i), F8 ? 2 * ((i & 1) ? S::NVC : S::NQC) : 1);
      mbar_init(bar(S::B_EMPTY + i), 2);  // released by both MMA issuers
    }
    for (int i = 0; i < S::NSTG; ++i) mbar_init(bar(S::B_STG + i), 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  // Registers: the TMA/MMA/TMEM warpgroup needs few, the softmax warpgroups
  // hold a 128-float score row each: 384 threads x 168 at launch >=
  // 128 x kRegsLow + 256 x kRegsHigh.  Each branch starts with its own
  // setmaxnreg so that the code it dominates is compiled for that budget.
  if (warp < 4) {
    regs_dec<kRegsLow>();
    if constexpr (F8) {
      // ------------------------------------- Q over an fp8 cache
      // Q is loaded as bf16 and turned into f16 in place by the 128 threads
      // of this warpgroup before any MMA (the converter warpgroup's first
      // staging copies are in flight meanwhile).
      if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(bar(S::B_Q), 2 * S::NQC * kSubTileBytes);
        for (int x = 0; x < 2; ++x)
          for (int c = 0; c < S::NQC; ++c)
            tma_load_4d(smem_u32(sQ + (x * S::NQC + c) * kSubTileBytes), &tm_q, bar(S::B_Q),
                        c * 64, 0, g, seg.q_start + tok0 + x * T);
      }
      const bool qok = warp_wait(bar(S::B_Q), 0, p.status, abort_flag);
      if (qok) {
        // bf16 -> f16, 16 bytes per step; an element outside f16's range
        // (|q| > 65504) becomes infinite and is reported as invalid input.
        uint32_t amax = 0u;
        for (int ch = threadIdx.x; ch < 2 * S::NQC * (kSubTileBytes / 16); ch += 128) {
          uint4* qp = reinterpret_cast<uint4*>(sQ + ch * 16);
          uint4 w = *qp;
          uint32_t* wv = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            wv[i] = pack_half2(__uint_as_float(wv[i] << 16), __uint_as_float(wv[i] & 0xFFFF0000u));
            amax = __vmaxu2(amax, wv[i] & 0x7FFF7FFFu);
          }
          *qp = w;
        }
        if ((amax & 0xFFFFu) >= 0x7C00u || (amax >> 16) >= 0x7C00u) record_status(p.status, kStatusInvalid);
      }
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the four warps of this warpgroup
      if (!qok && warp == 0 && lane == 0) mbar_wait_for(bar(S::B_Q), 0, kCleanupNs);
    }
    if (!F8 && warp == 0 && lane == 0) {
      // ---------------------------------------------------- TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(S::B_Q), 2 * S::NQC * kSubTileBytes);
      for (int x = 0; x < 2; ++x)
        for (int c = 0; c < S::NQC; ++c)
          tma_load_4d(smem_u32(sQ + (x * S::NQC + c) * kSubTileBytes), &tm_q, bar(S::B_Q),
                      c * 64, 0, g, seg.q_start + tok0 + x * T);
      bool ok = true;
      int issued = 0;  // tiles whose loads were started
      int rq = 0;      // next tile whose release has not been observed
      auto block_coord = [&](int b) -> int {
        if (b * kBlockTokens >= seg.kv_len) return p.num_blocks;  // reads zeros
        const int e = p.block_table[seg.table_off + b];
        if (e < 0 || e >= p.num_blocks) {
          record_status(p.status, kStatusInvalid);
          return p.num_blocks;
        }
        return e;
      };
      // Loads the nsub sub-tiles (two 64-key blocks each) of tile t.
      auto load_tile = [&](const CUtensorMap* m, int nsub, int pos, uint32_t fb, int c0, int c1) {
        for (int c = 0; c < nsub; ++c) {
          const uint32_t d = smem_u32(sRing + ((pos + c) % S::NSLOT) * kSubTileBytes);
          if (p.paged) {
            tma_load_4d(d, m, fb, c * 64, g, 0, c0);
            tma_load_4d(d + kSubTileBytes / 2, m, fb, c * 64, g, 0, c1);
          } else {
            tma_load_3d(d, m, fb, c * 64, g, c0);
            tma_load_3d(d + kSubTileBytes / 2, m, fb, c * 64, g, c1);
          }
        }
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int key0 = k_lo + j * kTileN;
        int c0, c1;
        if (p.paged) {
          c0 = block_coord(key0 / kBlockTokens);
          c1 = block_coord(key0 / kBlockTokens + 1);
        } else {
          c0 = seg.kv_base + key0;
          c1 = c0 + kBlockTokens;
        }
        for (int part = 0; part < 2; ++part) {  // K, then V
          const int t = 2 * j + part;
          const int pos = S::tile_pos(t);
          const int nsub = S::tile_slots(t);
          // Tiles are released in load order: wait until every tile that used
          // these slots, and the tile that last used this barrier, is released.
          while (rq < t && (rq <= t - S::NB || S::tile_pos(rq) < pos + nsub - S::NSLOT)) {
            if (!mbar_wait(bar(S::B_EMPTY + rq % S::NB), (rq / S::NB) & 1u, p.status, abort_flag)) {
              ok = false;
              break;
            }
            ++rq;
          }
          if (!ok) break;
          const uint32_t fb = bar(S::B_FULL + t % S::NB);
          const CUtensorMap* m = part == 0 ? &tm_k : &tm_v;
          // Rows of the last loaded block at positions >= kv_len hold whatever
          // the pool holds there; their V rows are zeroed before the tile is
          // released so that P = 0 times them stays 0 (K rows there are masked
          // to -inf before the softmax).  This happens at most once per CTA.
          const int r0 = seg.kv_len - key0;
          const bool fix = part == 1 && p.paged && r0 > 0 && r0 < kTileN && (r0 % kBlockTokens) != 0;
          if (!fix) {
            mbar_arrive_expect_tx(fb, nsub * kSubTileBytes);
            load_tile(m, nsub, pos, fb, c0, c1);
          } else {
            mbar_arrive_expect_tx(bar(S::B_TMP), nsub * kSubTileBytes);
            load_tile(m, nsub, pos, bar(S::B_TMP), c0, c1);
            if (!mbar_wait(bar(S::B_TMP), 0, p.status, abort_flag)) {
              mbar_wait_for(bar(S::B_TMP), 0, kCleanupNs);
              ok = false;
              break;
            }
            const int r1 = (r0 + kBlockTokens - 1) / kBlockTokens * kBlockTokens;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int c = 0; c < nsub; ++c)
              for (int row = r0; row < r1; ++row) {
                uint4* rp = reinterpret_cast<uint4*>(sRing + ((pos + c) % S::NSLOT) * kSubTileBytes +
                                                     row * 128);
#pragma unroll
                for (int u = 0; u < 8; ++u) rp[u] = z;
              }
            fence_proxy_async_smem();
            mbar_arrive(fb);
          }
          ++issued;
        }
      }
      if (!ok) {
        // Let every copy this thread started land before the CTA exits.
        for (int t = issued > S::NB ? issued - S::NB : 0; t < issued; ++t)
          mbar_wait_for(bar(S::B_FULL + t % S::NB), (t / S::NB) & 1u, kCleanupNs);
        mbar_wait_for(bar(S::B_Q), 0, kCleanupNs);
      }
    } else if ((warp == 1 || warp == 3) && lane == 0) {
      // ---------------------------------------------------- MMA issuer
      const int x = warp == 1 ? 0 : 1;
      // Descriptors are built once; sub-tile and k-step offsets are added to
      // the start-address field (16-byte units; shared addresses stay below
      // 2^18, so the 14-bit field never carries).
      const uint64_t dq0 = sdesc_sw128(smem_u32(sQ + x * S::NQC * kSubTileBytes), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(sRing), 16, 1024);             // K-major
      const uint64_t dv0 = sdesc_sw128(smem_u32(sRing), kSubTileBytes, 1024);  // MN-major
      constexpr uint32_t kSub16 = kSubTileBytes >> 4;
      const uint32_t tS = tbase + x * kTileN;
      const uint32_t tO = tbase + 2 * kTileN + x * DV;
      // (over an fp8 cache Q was widened by this warpgroup before this point)
      bool ok = F8 ? *abort_flag == 0u : mbar_wait(bar(S::B_Q), 0, p.status, abort_flag);
      // Ring slots of K_j and V_{j-1}, advanced by one tile pair per block.
      int kslot = 0;
      int vslot = S::NQC - (S::NQC + S::NVC);  // becomes V_0's slot at j = 1
      if (vslot < 0) vslot += S::NSLOT;
      // Block j = [PV(x, j-1) if j > 0][QK(x, j) if j < n_kv]; blocks run in
      // the global order A0 B0 A1 B1 ...: block j of issuer x is number 2j+x.
      for (int j = 0; ok && j <= n_kv; ++j) {
        const int tk = 2 * j;      // tile index of K_j
        const int tv = 2 * j - 1;  // tile index of V_{j-1}
        if (j > 0) {
          kslot += S::NQC + S::NVC;
          if (kslot >= S::NSLOT) kslot -= S::NSLOT;
          vslot += S::NQC + S::NVC;
          if (vslot >= S::NSLOT) vslot -= S::NSLOT;
        }
        if (j > 0) {
          if (!(ok = mbar_wait(bar(S::B_FULL + tv % S::NB), (tv / S::NB) & 1u, p.status, abort_flag))) break;
          if (!(ok = mbar_wait(bar(S::B_P + x), (j - 1) & 1, p.status, abort_flag))) break;
          tc_fence_after();
          VPP_STAMP(x, j, 0);  // first part of P of tile j-1 seen
        }
        if (j < n_kv &&
            !(ok = mbar_wait(bar(S::B_FULL + tk % S::NB), (tk / S::NB) & 1u, p.status, abort_flag)))
          break;
        // Take the turn: a tight spin on the shared counter (the abort flag
        // and the time limit are checked every 256 polls), so that the first
        // MMA of this block follows the partner's hand-over within a few
        // cycles.
        if (*turn != 2 * j + x) {
          const uint64_t t0 = globaltimer_ns();
          for (uint32_t n = 1; *turn != 2 * j + x; ++n) {
            if ((n & 255u) != 0) continue;
            if (*abort_flag) { ok = false; break; }
            if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
              record_status(p.status, kStatusTimeout);
              *abort_flag = 1u;
              ok = false;
              break;
            }
          }
          if (!ok) break;
        }
        VPP_STAMP(x, j, 1);  // turn taken
        if (j > 0) {
          // O += P V for tile j-1 (P read from TMEM, V from the ring), as two
          // chains of 16-key steps: [0, PV0) now, [PV0, 8) once the softmax
          // has stored the rest of P.
          const bool adjacent = S::NVC == 1 || vslot + S::NVC <= S::NSLOT;
          auto pv_steps = [&](int k0, int k1) {
            if (adjacent) {
              // Adjacent V sub-tiles: one N = DV chain (LBO = one sub-tile).
              const uint64_t vb = dv0 + vslot * kSub16;
#pragma unroll
              for (int k = k0; k < k1; ++k)
                umma_ts(tO, tS + 8 * k, vb + k * (2048 >> 4), S::IDESC_PV, (j > 1 || k > 0) ? 1u : 0u);
            } else {
              // The V tile wraps around the ring: one N = 64 chain per sub-tile.
#pragma unroll
              for (int k = k0; k < k1; ++k)
#pragma unroll
                for (int h = 0; h < S::NVC; ++h) {
                  const int vs = vslot + h < S::NSLOT ? vslot + h : vslot + h - S::NSLOT;
                  umma_ts(tO + 64 * h, tS + 8 * k, dv0 + vs * kSub16 + k * (2048 >> 4), S::IDESC_PV64,
                          (j > 1 || k > 0) ? 1u : 0u);
                }
            }
          };
          pv_steps(0, S::PV0);
          if (S::SPLIT_P) {
            if (!(ok = mbar_wait(bar(S::B_P1 + x), (j - 1) & 1, p.status, abort_flag))) break;
            tc_fence_after();
            VPP_STAMP(x, j, 3);  // second part of P of tile j-1 seen
            pv_steps(S::PV0, kTileN / 16);
          }
          if (S::EARLY_V) umma_commit(bar(S::B_EMPTY + tv % S::NB));
        }
        if (j < n_kv) {
          // S = Q K^T for tile j; follows PV(x, j-1), which read P from the
          // same TMEM columns, in issue order.  The turn goes to the partner
          // before the last four MMAs: its first MMAs then queue behind them
          // and the tensor core does not drain between the two blocks.
#pragma unroll
          for (int c = 0; c < S::NQC; ++c) {
            const int ks = kslot + c < S::NSLOT ? kslot + c : kslot + c - S::NSLOT;
            const uint64_t kb = dk0 + ks * kSub16;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (c == S::NQC - 1 && k == 0) *turn = 2 * j + x + 1;
              umma_ss(tS, dq0 + c * kSub16 + 2 * k, kb + 2 * k, S::IDESC_QK, (c | k) ? 1u : 0u);
            }
          }
        }
        if (j == n_kv) *turn = 2 * j + x + 1;
        if (j < n_kv) {
          umma_commit(bar(S::B_S + x));
          umma_commit(bar(S::B_EMPTY + tk % S::NB));
        }
        if (j > 0 && !S::EARLY_V) umma_commit(bar(S::B_EMPTY + tv % S::NB));
        if (j == n_kv) umma_commit(bar(S::B_O + x));
        VPP_STAMP(x, j, 2);  // block issued
      }
      if (!ok) {
        *abort_flag = 1u;  // the partner issuer may be waiting for this turn
        // Every MMA issued so far must finish before TMEM is freed.
        umma_commit(bar(S::B_FINAL + x));
        mbar_wait_for(bar(S::B_FINAL + x), 0, kCleanupNs);
      }
    }
  } else if (F8 && warp >= 12) {
    if constexpr (F8) {
      regs_dec<kRegsConvF8>();
      // ---------------------------------- converters over an fp8 cache
      // Warps 12..15, one per SM sub-partition.  The K/V codes of a half
      // sub-tile (64 keys = one cache block x 64 dims) are copied by TMA into
      // one of the warp's two staging slots; the warp widens them exactly to
      // f16 into the 128B-swizzled ring slot layout the MMAs read
      // (the layout TMA writes for a bf16 cache), zeroing rows past the
      // sequence (the pool holds whatever codes there), and arrives on the
      // tile's FULL barrier.  Unit u (order: K_0's half sub-tiles, V_0's, K_1's,
      // ...) is widened by converter u % NCONV.
      auto block_coord = [&](int b) -> int {
        if (b * kBlockTokens >= seg.kv_len) return p.num_blocks;  // reads zeros
        const int e = p.block_table[seg.table_off + b];
        if (e < 0 || e >= p.num_blocks) {
          record_status(p.status, kStatusInvalid);
          return p.num_blocks;
        }
        return e;
      };
      constexpr int kUnits = 2 * (S::NQC + S::NVC);  // half sub-tiles per K/V tile pair
      constexpr int kSlotsPerWarp = S::NSTG / S::NCONV;
      const int total = n_kv * kUnits;
      const int cw = warp - 12;
      auto stage_slot = [&](int u) { return cw * kSlotsPerWarp + (u / S::NCONV) % kSlotsPerWarp; };
      auto stage_parity = [&](int u) { return static_cast<uint32_t>((u / S::NCONV) / kSlotsPerWarp) & 1u; };
      // tile pair j, K (part 0) or V (part 1), 64-dim sub-tile c, 64-key half hh
      auto unit = [&](int u, int& j, int& part, int& c, int& hh) {
        j = u / kUnits;
        const int r = u - j * kUnits;
        hh = r & 1;
        const int sub = r >> 1;
        part = sub >= S::NQC ? 1 : 0;
        c = part ? sub - S::NQC : sub;
      };
      // Starts the copy of unit u's codes into its staging slot (one lane).
      auto issue_stage = [&](int u) {
        int j, part, c, hh;
        unit(u, j, part, c, hh);
        const int key0 = k_lo + j * kTileN + hh * kBlockTokens;
        const int slot = stage_slot(u);
        const uint32_t sb = bar(S::B_STG + slot);
        const uint32_t d = smem_u32(sStage + slot * kStageBytes);
        const CUtensorMap* m = part ? &tm_v : &tm_k;
        mbar_arrive_expect_tx(sb, kStageBytes);
        if (p.paged)
          tma_load_4d(d, m, sb, c * 64, g, 0, block_coord(key0 / kBlockTokens));
        else
          tma_load_3d(d, m, sb, c * 64, g, seg.kv_base + key0);
      };
      int issued = cw;  // next unit whose staging copy this warp starts (lane 0)
      if (lane == 0)
        for (int n = 0; n < kSlotsPerWarp && issued < total; ++n, issued += S::NCONV) issue_stage(issued);
      bool ok = true;
      int rq = 0;     // next tile whose release has not been observed
      int done = cw;  // next unit of this warp whose staging slot is not consumed
      for (int u = cw; ok && u < total; u += S::NCONV) {
        int j, part, c, hh;
        unit(u, j, part, c, hh);
        const int t = 2 * j + part;
        const int pos = S::tile_pos(t);
        const int nsub = S::tile_slots(t);
        // Tiles are released in load order: wait until every tile that used
        // these slots, and the tile that last used this barrier, is released.
        while (rq < t && (rq <= t - S::NB || S::tile_pos(rq) < pos + nsub - S::NSLOT)) {
          if (!(ok = warp_wait(bar(S::B_EMPTY + rq % S::NB), (rq / S::NB) & 1u, p.status, abort_flag)))
            break;
          ++rq;
        }
        if (!ok) break;
        const int slot = stage_slot(u);
        if (!(ok = warp_wait(bar(S::B_STG + slot), stage_parity(u), p.status, abort_flag))) break;
        const uint8_t* src = sStage + slot * kStageBytes;
        uint8_t* dst = sRing + ((pos + c) % S::NSLOT) * kSubTileBytes + hh * kBlockTokens * 128;
        const int valid_rows = seg.kv_len - (k_lo + j * kTileN + hh * kBlockTokens);
#pragma unroll 4
        for (int it = 0; it < kBlockTokens * 4 / 32; ++it) {
          const int idx = it * 32 + lane;
          const int row = idx >> 2;  // key within the half (the swizzle phase is row & 7 either way)
          const int q4 = idx & 3;    // 16 codes: dims 16 q4 .. 16 q4 + 15
          uint4 w = *reinterpret_cast<const uint4*>(src + row * 64 + q4 * 16);
          if (row >= valid_rows) w = make_uint4(0u, 0u, 0u, 0u);
          uint32_t h[8];
          e4m3x4_to_f16x2x2(w.x, h[0], h[1]);
          e4m3x4_to_f16x2x2(w.y, h[2], h[3]);
          e4m3x4_to_f16x2x2(w.z, h[4], h[5]);
          e4m3x4_to_f16x2x2(w.w, h[6], h[7]);
          uint8_t* rp = dst + row * 128;
          *reinterpret_cast<uint4*>(rp + (((2 * q4) ^ (row & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(rp + (((2 * q4 + 1) ^ (row & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        done = u + S::NCONV;
        if (lane == 0) {
          mbar_arrive(bar(S::B_FULL + t % S::NB));  // one of the tile's 2 nsub arrivals
          if (issued < total) {
            issue_stage(issued);
            issued += S::NCONV;
          }
        }
      }
      if (!ok && lane == 0) {
        // Let every copy this warp started land before the CTA exits.
        for (int v = done; v < issued; v += S::NCONV)
          mbar_wait_for(bar(S::B_STG + stage_slot(v)), stage_parity(v), kCleanupNs);
      }
    }
  } else {
    regs_inc<S::REGS_HIGH>();
    // ------------------------------------------------------ softmax + epilogue
    const int x = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int tok = tok0 + x * T + row / G;
    const int hq = g * G + row % G;
    const int lim = min(P + tok, seg.kv_len - 1);  // last visible key (inclusive)
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = lane_base + x * kTileN;
    const uint32_t tO = lane_base + 2 * kTileN + x * DV;
    // Per-kv-head factors of an fp8 cache (key codes x k_scale, values x
    // v_scale): k_scale joins the score scale, v_scale the final division.
    const float sl = p.k_scale ? p.scale_log2 * __ldg(p.k_scale + g) : p.scale_log2;
    const float vsc = p.v_scale ? __ldg(p.v_scale + g) : 1.f;
    float m = -INFINITY;  // running max of score * scale * log2(e)
    float l = 0.f;        // running denominator, relative to 2^m
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = warp_wait(bar(S::B_S + x), j & 1, p.status, abort_flag))) break;
      tc_fence_after();
      if (row == 0) VPP_STAMP(2 + x, j, 0);  // S ready
      uint32_t u[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + 32 * q, u[q]);
      tmem_ld_wait();
      if (row == 0) VPP_STAMP(2 + x, j, 1);  // S in registers
      float sv[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(u[c >> 5][c & 31]);
      const int key0 = k_lo + j * kTileN;
      if (key0 + kTileN - 1 > lim) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (key0 + c > lim) sv[c] = -INFINITY;
      }
      // Row max: eight independent chains of 3-input max, then a tree.  Chain
      // i takes sv[i] and pairs sv[c + 2i], sv[c + 2i + 1] for c = 8 .. 104;
      // in the last step (sv[120..127], four pairs) chains i and i + 4 take the
      // same pair, which leaves the maximum unchanged.
      auto row_max = [&]() {
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = sv[i];
#pragma unroll
        for (int c = 8; c + 16 <= 128; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], sv[c + 2 * i], sv[c + 2 * i + 1]);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], sv[120 + 2 * (i & 3)], sv[121 + 2 * (i & 3)]);
        return fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                     fmaxf(mx8[6], mx8[7]));
      };
      // Exponentials of the tile's two key parts: the first part's P is stored
      // and signalled before the second part is computed, so that the first
      // P V chain runs meanwhile.
      const float2 sl2 = make_float2(sl, sl);
      float2 rs4[4];
      auto part = [&](auto k0, auto k1, float mref) {
        const float mb = (mref == -INFINITY) ? 0.f : mref;
        const float2 nmb2 = make_float2(-mb, -mb);
        exps_to_tmem<decltype(k0)::value, decltype(k1)::value, F8>(sv, sl2, nmb2, rs4, tS);
      };
      using K_0 = std::integral_constant<int, 0>;
      using K_P0 = std::integral_constant<int, S::KP0>;
      using K_N = std::integral_constant<int, kTileN>;
#pragma unroll
      for (int i = 0; i < 4; ++i) rs4[i] = make_float2(0.f, 0.f);
      if (j == 0) {
        m = row_max() * sl;
        part(K_0{}, K_P0{}, m);
      } else {
        // The first part's exponentials use the running max right away and
        // the row max of the whole tile is computed alongside.  Only when it
        // has grown by more than 2^8 are O and the denominator rescaled and
        // the first part redone, before the first part is released (rare
        // after the first tile; the result is exact either way since
        // numerator and denominator share the reference m).
        part(K_0{}, K_P0{}, m);
        const float m_new = fmaxf(m, row_max() * sl);
        const bool need = m_new > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O of this tile is idle here: PV(x, j-1) completed before S(x, j)
          // was committed, and PV(x, j) waits for this group's P.
          const float f = need ? ex2_approx(m - m_new) : 1.f;
          if (need) {
            l *= f;
            m = m_new;
          }
          tmem_st_wait();
#pragma unroll
          for (int q = 0; q < DV / 32; ++q) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * q, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tmem_st32(tO + 32 * q, o);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) rs4[i] = make_float2(0.f, 0.f);
          part(K_0{}, K_P0{}, m);  // rows whose m did not move recompute the same values
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(S::B_P + x));
      if (row == 0) VPP_STAMP(2 + x, j, 2);  // first part of P stored and signalled
      if (S::SPLIT_P) {
        part(K_P0{}, K_N{}, m);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(S::B_P1 + x));
        if (row == 0) VPP_STAMP(2 + x, j, 3);  // second part of P stored and signalled
      }
      const float2 rs2 = fadd2(fadd2(rs4[0], rs4[1]), fadd2(rs4[2], rs4[3]));
      const float rs = rs2.x + rs2.y;
      l += rs;
    }
    if (ok) ok = warp_wait(bar(S::B_O + x), 0, p.status, abort_flag);
    if (ok) {
      tc_fence_after();
      const bool valid = tok < seg.q_len;
      const float inv = vsc / l;
      const float lse_v = m * kLn2 + logf(l);
      if (seg.n_splits == 1) {
        uint16_t* orow = p.out + (static_cast<int64_t>(seg.q_start + tok) * p.heads + hq) * DV;
#pragma unroll
        for (int q = 0; q < DV / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * q, o);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * q);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        if (valid && p.lse) p.lse[static_cast<int64_t>(hq) * p.lse_stride + seg.q_start + tok] = lse_v;
      } else {
        const int64_t wrow = seg.ws_row0 + static_cast<int64_t>(split) * seg.q_len + tok;
        float* orow = p.ws_o + (wrow * p.heads + hq) * DV;
#pragma unroll
        for (int q = 0; q < DV / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * q, o);
          tmem_ld_wait();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(orow + 32 * q);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                   __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
          }
        }
        if (valid) p.ws_lse[wrow * p.heads + hq] = lse_v;
      }
    }
  }

  // TMEM is freed once the warps that use it are done: the softmax warps
  // (tcgen05.ld/st; they have waited for their tile's last MMA) and the two
  // MMA issuers (in the abort path after their MMAs have completed).  An
  // mbarrier rather than a CTA barrier: the warps of the TMA/MMA warpgroup
  // reach this point with lane 0 from a long role loop and the other lanes
  // from none, and bar.sync there was measured to release them before the
  // softmax warps had arrived; their other lanes, and the TMA producer (whose
  // copies have all landed), just leave.  Warp 2 waits, bounded beyond every
  // other wait, and frees TMEM.
  if (warp >= 4) {
    __syncwarp();
    tc_fence_before();
    if (lane == 0) mbar_arrive(bar(S::B_END));
  } else if ((warp == 1 || warp == 3) && lane == 0) {
    tc_fence_before();
    mbar_arrive(bar(S::B_END));
  }
  if (warp == 2) {
    mbar_wait_for(bar(S::B_END), 0, 2 * kWaitTimeoutNs + 2 * kCleanupNs);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int DQ, int DV, bool F8>
cudaError_t launch_chunk_attn_t(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, const AttnParams& p, int grid,
                                cudaStream_t stream) {
  constexpr int smem = attn_smem_bytes(DQ, DV, F8);
  static_assert(smem <= kSmemLimit, "shared memory budget");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64] = {};
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(chunk_attn_kernel<DQ, DV, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  chunk_attn_kernel<DQ, DV, F8><<<grid, attn_threads(F8), smem, stream>>>(tm_q, tm_k, tm_v, p);
  return cudaGetLastError();
}

}  // namespace vpp
