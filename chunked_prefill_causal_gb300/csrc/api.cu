// api.cu -- the C ABI of include/vpp.h: argument validation, TMA tensor maps,
// work planning and kernel launches.  Allocates no device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <vector>

#include "chunk_attn.cuh"
#include "common.cuh"
#include "decode.cuh"
#include "fp8.cuh"
#include "vpp.h"

namespace vpp {
__device__ int g_status_word;  // first device-side error since the last read
}

using namespace vpp;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int* status = nullptr;
  // Side stream for the decode rows of a mixed batch, so that they run beside
  // the prefill segments, and its fork / join events.
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr;
  cudaEvent_t ev_join = nullptr;
  std::mutex side_mutex;  // one fork ... join sequence at a time
};

std::mutex g_mutex;
DeviceState g_devices[64];
EncodeTiledFn g_encode = nullptr;

// One-time, per-device set-up: SM count, status-word address, driver entry
// point of cuTensorMapEncodeTiled.  Thread-safe.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VPP_ERR_CUDA;
  if (dev < 0 || dev >= 64) return VPP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_devices[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return VPP_ERR_CUDA;
    if (major != 10 || minor != 3) return VPP_ERR_UNSUPPORTED;  // built for sm_103a only
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&s.status), g_status_word) != cudaSuccess)
      return VPP_ERR_CUDA;
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          fn == nullptr)
        return VPP_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    // Highest priority: when the decode kernel runs on a share of the SMs,
    // its CTAs are placed before the prefill CTAs launched after it.
    int prio_lo = 0, prio_hi = 0;
    if (cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi) != cudaSuccess ||
        cudaStreamCreateWithPriority(&s.side, cudaStreamNonBlocking, prio_hi) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.ev_join, cudaEventDisableTiming) != cudaSuccess)
      return VPP_ERR_CUDA;
    s.ready = true;
  }
  *out = &s;
  return VPP_OK;
}

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

bool supported_dims(int dq, int dv) {
  return (dq == 64 || dq == 128 || dq == 192) && (dv == 64 || dv == 128);
}

int check_heads(int heads, int kv_heads) {
  if (heads <= 0 || kv_heads <= 0 || heads % kv_heads != 0) return VPP_ERR_INVALID;
  const int g = heads / kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return VPP_ERR_UNSUPPORTED;
  return VPP_OK;
}

// bf16 tensor map with 128-byte swizzle; an out-of-range box reads zeros.
int encode_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
               const cuuint64_t* strides, const cuuint32_t* box) {
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base),
                              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VPP_OK : VPP_ERR_INVALID;
}

// Q (and any [T][heads][d] tensor) viewed as [T][kv_heads][G][d]; a box is
// 64 dims x G heads x 1 kv head x 128/G tokens = 128 rows of 128 bytes.
int make_q_map(CUtensorMap* m, const void* q, int64_t total_q, int heads, int kv_heads, int dq) {
  const int G = heads / kv_heads;
  const cuuint64_t dims[4] = {(cuuint64_t)dq, (cuuint64_t)G, (cuuint64_t)kv_heads,
                              (cuuint64_t)total_q};
  const cuuint64_t strides[3] = {(cuuint64_t)dq * 2, (cuuint64_t)G * dq * 2,
                                 (cuuint64_t)heads * dq * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)(kTileM / G)};
  return encode_map(m, q, 4, dims, strides, box);
}

// Paged cache [num_blocks][64][kv_heads][d]: box = 64 dims x 1 head x 64 rows x 1 block.
int make_paged_map(CUtensorMap* m, const void* cache, int32_t num_blocks, int kv_heads, int d) {
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)kv_heads, (cuuint64_t)kBlockTokens,
                              (cuuint64_t)num_blocks};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)kv_heads * d * 2,
                                 (cuuint64_t)kBlockTokens * kv_heads * d * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kBlockTokens, 1};
  return encode_map(m, cache, 4, dims, strides, box);
}

// Contiguous cache [n_tokens][kv_heads][d]; rows past n_tokens read zeros.
int make_contig_map(CUtensorMap* m, const void* cache, int64_t n_tokens, int kv_heads, int d) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)kv_heads, (cuuint64_t)n_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)kv_heads * d * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBlockTokens};
  return encode_map(m, cache, 3, dims, strides, box);
}

// The same two cache layouts holding one-byte E4M3 codes: plain (unswizzled)
// boxes of 64 codes x 64 tokens, which the kernel widens itself.
int encode_map_u8(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box) {
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims,
                              strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VPP_OK : VPP_ERR_INVALID;
}

int make_paged_map_u8(CUtensorMap* m, const void* cache, int32_t num_blocks, int kv_heads, int d) {
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)kv_heads, (cuuint64_t)kBlockTokens,
                              (cuuint64_t)num_blocks};
  const cuuint64_t strides[3] = {(cuuint64_t)d, (cuuint64_t)kv_heads * d,
                                 (cuuint64_t)kBlockTokens * kv_heads * d};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kBlockTokens, 1};
  return encode_map_u8(m, cache, 4, dims, strides, box);
}

int make_contig_map_u8(CUtensorMap* m, const void* cache, int64_t n_tokens, int kv_heads, int d) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)kv_heads, (cuuint64_t)n_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)kv_heads * d};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBlockTokens};
  return encode_map_u8(m, cache, 3, dims, strides, box);
}

int pairs_for(int64_t q_len, int group) { return (int)ceil_div(q_len, 2 * (kTileM / group)); }

// Work plan of one chunk (a7).  Query tokens [t0, C) form the heavy group,
// launched first, whose key range [0, P + t0 + i] is cut into n_splits
// ranges of split_keys keys (the last range takes the rest); tokens [0, t0)
// form the light group, unsplit.  t0 = 0: a single group.
struct ChunkPlan {
  int t0;
  int n_splits;
  int split_keys;
};

// Key ranges of a group whose tokens sit after P_seg cached keys: S requested
// ranges of whole 128-key tiles, fewer when the prefix is short.
ChunkPlan uniform_plan(int64_t P_seg, int S, int t0) {
  if (S <= 1 || P_seg < kTileN) return ChunkPlan{t0, 1, 0};
  S = std::min(S, 16);
  const int64_t keys = round_up((size_t)ceil_div(P_seg, S), (size_t)kTileN);
  const int64_t S_eff = std::min<int64_t>(S, P_seg / keys + 1);
  if (S_eff <= 1) return ChunkPlan{t0, 1, 0};
  return ChunkPlan{t0, (int)S_eff, (int)keys};
}

// Cost model of a launch, fitted on GB300 to 55 timed gqa32k chunks (1 to 8
// key ranges for every token, or 2 for the heaviest eighth; 1.7% rms error,
// 5% at most): CTAs start in launch order on the first free SM (list
// scheduling); a CTA costs 12.5 ns per key of its range (whole 128-key tiles;
// d_qk + d_v = 256) plus 8 us of prologue and epilogue, 2 us more when it
// writes float32 partials; the merge kernel that follows a split costs 8 us
// plus its partials read at 6 TB/s.
constexpr double kKeyNs = 12.5;
constexpr double kCtaNs = 8000.0;
constexpr double kSplitCtaNs = 2000.0;
constexpr double kMergeNs = 8000.0;
constexpr double kMergeBytesPerNs = 6000.0;

double predict_ns(const ChunkPlan& pl, int64_t P, int64_t C, int G, int kv_heads, int dq, int dv,
                  int num_sms, std::vector<double>& heap, double give_up = 1e300) {
  const double key_ns = kKeyNs * (dq + dv) / 256.0;
  const int T2 = 2 * (kTileM / G);
  heap.assign(num_sms, 0.0);  // min-heap of SM free times
  double* h = heap.data();
  const int n = num_sms;
  double span = 0.0;  // latest SM free time so far: a lower bound of the result
  // The next CTA goes to the SM that frees first: add its cost to the root
  // and sift the root down.
  auto take = [&](double c) {
    const double v = h[0] + c;
    int i = 0;
    while (true) {
      int k = 2 * i + 1;
      if (k >= n) break;
      if (k + 1 < n && h[k + 1] < h[k]) ++k;
      if (h[k] >= v) break;
      h[i] = h[k];
      i = k;
    }
    h[i] = v;
    span = std::max(span, v);
  };
  for (int grp = 0; grp < 2; ++grp) {
    const int64_t a = grp == 0 ? pl.t0 : 0, b = grp == 0 ? C : pl.t0;
    if (b <= a) continue;
    const int S = grp == 0 ? pl.n_splits : 1;
    const int64_t P_seg = P + a, q = b - a;
    const int np = pairs_for(q, G);
    // CTA costs of one kv head in launch order (the same for every kv head).
    thread_local std::vector<double> cost;
    cost.clear();
    for (int r = 0; r < np; ++r) {
      const int pair = np - 1 - r;
      const int64_t hi = P_seg + std::min<int64_t>((int64_t)(pair + 1) * T2, q);
      for (int sp = 0; sp < S; ++sp) {
        const int64_t lo = (int64_t)sp * pl.split_keys;
        const int64_t end = sp == S - 1 ? hi : lo + pl.split_keys;
        cost.push_back((double)ceil_div(end - lo, kTileN) * kTileN * key_ns + kCtaNs + (S > 1 ? kSplitCtaNs : 0.0));
      }
    }
    for (int g = 0; g < kv_heads; ++g) {
      for (double c : cost) take(c);
      if (span > give_up) return span;  // already worse than the plan to beat
    }
  }
  if (pl.n_splits <= 1) return span;
  const double merge_bytes = (double)pl.n_splits * (C - pl.t0) * G * kv_heads * (dv + 1) * 4.0;
  return span + kMergeNs + merge_bytes / kMergeBytesPerNs;
}

struct PlanKey {
  int64_t P, C;
  int heads, kv_heads, dq, dv, requested, num_sms;
  bool operator==(const PlanKey& o) const {
    return P == o.P && C == o.C && heads == o.heads && kv_heads == o.kv_heads && dq == o.dq && dv == o.dv &&
           requested == o.requested && num_sms == o.num_sms;
  }
};
std::mutex g_plan_mutex;
PlanKey g_plan_keys[64];
ChunkPlan g_plans[64];
int g_plan_count = 0;

// Chooses the plan.  An explicit request of S ranges splits every query token
// the same way.  Otherwise, when the chunk is a few waves of CTAs, the model
// above picks between uniform plans (1 to 8 ranges) and plans whose heaviest
// query-tile pairs alone take 2 to 4 ranges, filling the last wave without
// paying the splitting costs on every CTA; a split plan must beat the unsplit
// one by 2%.  Plans are remembered per shape (the choice costs up to ~1 ms of
// host time for a new shape).
ChunkPlan plan_chunk(int64_t P, int64_t C, int heads, int kv_heads, int dq, int dv, int requested,
                     int num_sms) {
  if (requested >= 1 || C <= 0) return uniform_plan(P, requested, 0);
  const int G = heads / kv_heads;
  const int np = pairs_for(C, G);
  const int64_t base = (int64_t)np * kv_heads;
  if (base >= 6LL * num_sms || num_sms < 1) return ChunkPlan{0, 1, 0};
  const PlanKey key{P, C, heads, kv_heads, dq, dv, requested, num_sms};
  {
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    for (int i = 0; i < std::min(g_plan_count, 64); ++i)
      if (g_plan_keys[i] == key) return g_plans[i];
  }
  std::vector<double> heap;
  const int T2 = 2 * (kTileM / G);
  ChunkPlan best{0, 1, 0};
  const double t1 = predict_ns(best, P, C, G, kv_heads, dq, dv, num_sms, heap);
  double best_t = t1;
  auto consider = [&](const ChunkPlan& pl) {
    if (pl.n_splits <= 1) return;
    const double t = predict_ns(pl, P, C, G, kv_heads, dq, dv, num_sms, heap, std::min(best_t, 0.98 * t1));
    if (t < best_t && t < 0.98 * t1) {
      best_t = t;
      best = pl;
    }
  };
  for (int S = 2; S <= 8; ++S)
    if (base * S <= 8LL * num_sms && P / S >= 512) consider(uniform_plan(P, S, 0));
  // The h heaviest pairs of every kv head split into S ranges: h on a grid
  // of np/8, and the counts that bring the CTAs just under whole waves.
  for (int S = 2; S <= 3; ++S) {
    std::vector<int> hs;
    for (int h = std::max(1, np / 8); h < np; h += std::max(1, np / 8)) hs.push_back(h);
    for (int64_t w = (base + num_sms - 1) / num_sms; w <= (base + num_sms - 1) / num_sms + 2; ++w) {
      const int64_t h0 = (w * num_sms - base) / ((int64_t)kv_heads * (S - 1));
      for (int64_t h = h0 - 1; h <= h0 + 1; ++h)
        if (h >= 1 && h < np) hs.push_back((int)h);
    }
    for (int h : hs) {
      const int t0 = (np - h) * T2;
      consider(uniform_plan(P + t0, S, t0));
    }
  }
  std::lock_guard<std::mutex> lock(g_plan_mutex);
  g_plan_keys[g_plan_count % 64] = key;
  g_plans[g_plan_count % 64] = best;
  ++g_plan_count;
  return best;
}

size_t ws_q_bytes(int q_dtype, int64_t C, int heads, int dq) {
  return q_dtype == VPP_FP32 ? round_up((size_t)C * heads * dq * 2, 256) : 0;
}

// Workspace of a plan's split group: float32 partial outputs, then their
// LSEs, of its n_splits x (C - t0) token rows.
struct SplitWs {
  size_t o_bytes, lse_bytes;
  size_t total() const { return o_bytes + lse_bytes; }
};

SplitWs ws_split(const ChunkPlan& pl, int64_t C, int heads, int dv) {
  SplitWs w{0, 0};
  if (pl.n_splits <= 1) return w;
  const size_t rows = (size_t)pl.n_splits * (C - pl.t0);
  w.o_bytes = round_up(rows * heads * dv * 4, 256);
  w.lse_bytes = round_up(rows * heads * 4, 256);
  return w;
}

int chunk_attn_impl(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                    const int32_t* block_table, int32_t num_blocks, int64_t P, int64_t C,
                    int heads, int kv_heads, int dq, int dv, float scale, int num_splits,
                    void* out, float* lse, void* workspace, size_t ws_bytes, cudaStream_t st,
                    const float* k_scale = nullptr, const float* v_scale = nullptr, bool f8 = false) {
  if (P < 0 || C < 0 || num_blocks <= 0 || num_splits < 0) return VPP_ERR_INVALID;
  if (C == 0) return VPP_OK;  // pointers may be NULL for an empty chunk
  if (!q || !k_cache || !v_cache || !out) return VPP_ERR_INVALID;
  if (q_dtype != VPP_BF16 && q_dtype != VPP_FP32) return VPP_ERR_INVALID;
  if (int r = check_heads(heads, kv_heads)) return r;
  if (!supported_dims(dq, dv)) return VPP_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return VPP_ERR_INVALID;
  if (P + C > (int64_t)INT32_MAX / 2 || C > (int64_t)INT32_MAX / 2) return VPP_ERR_INVALID;
  if (block_table) {
    if ((int64_t)num_blocks * kBlockTokens < P + C) return VPP_ERR_INVALID;
  } else if ((int64_t)num_blocks < P + C) {
    return VPP_ERR_INVALID;
  }
  if (C == 0) return VPP_OK;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;

  const ChunkPlan pl = plan_chunk(P, C, heads, kv_heads, dq, dv, num_splits, ds->num_sms);
  const size_t need_q = ws_q_bytes(q_dtype, C, heads, dq);
  const SplitWs sw = ws_split(pl, C, heads, dv);
  const size_t need_s = sw.total();
  if (need_q + need_s > 0 && (!workspace || ws_bytes < need_q + need_s || !aligned16(workspace)))
    return VPP_ERR_WORKSPACE;

  const void* q_bf16 = q;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (q_dtype == VPP_FP32) {
    if (launch_convert_f32_bf16(static_cast<const float*>(q), reinterpret_cast<uint16_t*>(ws),
                                C * heads * dq, ds->num_sms, st) != cudaSuccess)
      return VPP_ERR_CUDA;
    q_bf16 = ws;
  }

  CUtensorMap tm_q, tm_k, tm_v;
  if (make_q_map(&tm_q, q_bf16, C, heads, kv_heads, dq)) return VPP_ERR_INVALID;
  if (block_table) {
    if (f8 ? make_paged_map_u8(&tm_k, k_cache, num_blocks, kv_heads, dq) ||
                 make_paged_map_u8(&tm_v, v_cache, num_blocks, kv_heads, dv)
           : make_paged_map(&tm_k, k_cache, num_blocks, kv_heads, dq) ||
                 make_paged_map(&tm_v, v_cache, num_blocks, kv_heads, dv))
      return VPP_ERR_INVALID;
  } else {
    if (f8 ? make_contig_map_u8(&tm_k, k_cache, P + C, kv_heads, dq) ||
                 make_contig_map_u8(&tm_v, v_cache, P + C, kv_heads, dv)
           : make_contig_map(&tm_k, k_cache, P + C, kv_heads, dq) ||
                 make_contig_map(&tm_v, v_cache, P + C, kv_heads, dv))
      return VPP_ERR_INVALID;
  }

  static AttnParams zero_params;  // value-initialised template
  AttnParams p = zero_params;
  p.n_segs = 0;
  p.heads = heads;
  p.kv_heads = kv_heads;
  p.group = heads / kv_heads;
  p.num_blocks = block_table ? num_blocks : 0;
  p.paged = block_table ? 1 : 0;
  p.scale_log2 = (scale > 0.f ? scale : 1.0f / std::sqrt((float)dq)) * 1.4426950408889634f;
  p.block_table = block_table;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.lse_stride = C;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.status = ds->status;
  // Segment 0: the heavy group (query tokens [t0, C), n_splits key ranges,
  // launched first); segment 1: the light group (tokens [0, t0), unsplit).
  int grid = 0;
  for (int grp = 0; grp < 2; ++grp) {
    const int64_t a = grp == 0 ? pl.t0 : 0, b = grp == 0 ? C : pl.t0;
    if (b <= a) continue;
    AttnSeg& s = p.segs[p.n_segs++];
    s.q_start = (int32_t)a;
    s.q_len = (int32_t)(b - a);
    s.kv_len = (int32_t)(P + b);
    s.table_off = 0;
    s.kv_base = 0;
    s.n_pairs = pairs_for(b - a, p.group);
    s.n_splits = grp == 0 ? pl.n_splits : 1;
    s.split_keys = s.n_splits > 1 ? pl.split_keys : 0;
    s.cta_begin = grid;
    s.ws_row0 = 0;
    const int64_t ctas = (int64_t)s.n_pairs * kv_heads * s.n_splits;
    if (grid + ctas > INT32_MAX) return VPP_ERR_INVALID;
    grid += (int)ctas;
  }
  if (pl.n_splits > 1) {
    p.ws_o = reinterpret_cast<float*>(ws + need_q);
    p.ws_lse = reinterpret_cast<float*>(ws + need_q + sw.o_bytes);
  }
  if (launch_chunk_attn(dq, dv, f8, tm_q, tm_k, tm_v, p, grid, st) != cudaSuccess) return VPP_ERR_CUDA;
  if (pl.n_splits > 1) {
    // the heavy group's rows: tokens [t0, C)
    if (launch_lse_merge(p.ws_o, p.ws_lse, 0, pl.n_splits, (int)(C - pl.t0), pl.t0, heads, dv,
                         static_cast<uint16_t*>(out), lse, C, ds->num_sms, st) != cudaSuccess)
      return VPP_ERR_CUDA;
  }
  return VPP_OK;
}

// Rows of a mixed batch served by the decode kernel, and the workspace their
// multi-range partials need.
bool is_decode_row(const int32_t* cu, int b, int heads, int kv_heads, int dq, int dv) {
  return cu[b + 1] - cu[b] == 1 && decode_supported(dq, dv, heads, kv_heads);
}

size_t decode_ws_bytes(const int32_t* cu, const int32_t* ctx, int32_t batch, int heads,
                       int kv_heads, int dq, int dv) {
  int64_t items = 0;
  bool any_multi = false;
  for (int b = 0; b < batch; ++b) {
    if (!is_decode_row(cu, b, heads, kv_heads, dq, dv)) continue;
    const int64_t n = ceil_div(std::max<int32_t>(ctx[b], 1), kDecodeSplitTokens);
    items += n;
    any_multi |= n > 1;
  }
  if (!any_multi) return 0;
  return round_up((size_t)items * heads * dv * 4, 256) + round_up((size_t)items * heads * 4, 256);
}

int build_varlen_plan(const int32_t* cu, const int32_t* ctx, int32_t batch, VarlenPlan* plan) {
  if (!cu || !ctx || batch <= 0 || batch > kMaxBatch) return VPP_ERR_INVALID;
  if (cu[0] != 0) return VPP_ERR_INVALID;
  plan->batch = batch;
  for (int b = 0; b < batch; ++b) {
    const int32_t ql = cu[b + 1] - cu[b];
    if (ql < 0 || ctx[b] < ql || ctx[b] < 0) return VPP_ERR_INVALID;
    plan->cu_q[b] = cu[b];
    plan->ctx[b] = ctx[b];
  }
  plan->cu_q[batch] = cu[batch];
  return VPP_OK;
}

bool scales_ok(const float* k_scale, const float* v_scale) {
  return k_scale && v_scale && !(reinterpret_cast<uintptr_t>(k_scale) & 3u) &&
         !(reinterpret_cast<uintptr_t>(v_scale) & 3u);
}

// Sequences of a mixed batch served by the chunk-attention kernel.
bool is_prefill_seg(const int32_t* cu, int b, int heads, int kv_heads, int dq, int dv) {
  return cu[b + 1] > cu[b] && !is_decode_row(cu, b, heads, kv_heads, dq, dv);
}

// Bytes of the bf16 widening of the fp8 cache rows the chunk-attention
// segments of a mixed batch read (their whole contexts).
size_t widen_ws_bytes(const int32_t* cu, const int32_t* ctx, int32_t batch, int heads, int kv_heads,
                      int dq, int dv) {
  int64_t rows = 0;
  for (int b = 0; b < batch; ++b)
    if (is_prefill_seg(cu, b, heads, kv_heads, dq, dv)) rows += ctx[b];
  if (rows == 0) return 0;
  return round_up((size_t)rows * kv_heads * dq * 2, 256) + round_up((size_t)rows * kv_heads * dv * 2, 256);
}

// Measured rates that split the SMs of a mixed batch: one decode CTA reads
// about 80 GB/s of a bf16 cache; a prefill CTA does about 9.9 TFLOP/s on one
// SM.
constexpr double kDecodeSmGBs = 80.0;
constexpr double kPrefillSmTFlops = 9.9;

// CTAs of the decode kernel in a mixed batch (0: one per work item).  The
// decode rows are HBM-bound and the prefill segments tensor-bound, but a
// kernel that starts first takes every SM.  So the decode kernel runs on a
// fixed share of the SMs, the one where both would finish together, and the
// prefill CTAs fill the rest (and the decode's SMs once it is done).  The
// share is rounded up by 10%: a decode that ends last leaves SMs idle (on
// the mixed workload, factors 0.9 / 1.0 / 1.1 / 1.2 / 1.3 / 1.5 measured
// 6.79 / 6.31 / 6.03 / 6.27 / 6.50 / 6.38 ms).  A batch without prefill
// segments, or whose decode needs nearly every SM anyway, runs one CTA per
// work item.  So does a decode over an E4M3 pool: with every SM it reads the
// codes at the copy bandwidth (9.25 GB in 1.4 ms for the mixed workload), and
// running it first and the prefill after measured as fast as the best share
// or faster (6.25 against 8.6 ms with the prefill contexts widened once; 8.81
// against 8.75-20.5 ms over factors 0.5-1.6 widening in the kernel).
int mixed_decode_ctas(int num_sms, bool fp8, double prefill_flops, double decode_bytes) {
  if (fp8 || prefill_flops <= 0.0 || decode_bytes <= 0.0 || num_sms < 2) return 0;
  const double r = (decode_bytes * kPrefillSmTFlops * 1e12) / (prefill_flops * kDecodeSmGBs * 1e9);
  const double sms = 1.1 * num_sms * r / (1.0 + r);
  if (sms >= 0.9 * num_sms) return 0;
  return std::max(1, (int)std::ceil(sms));
}

// CTAs of the top-k gather (0: one per work item).  Over a bf16 cache one
// persistent CTA per SM keeps each CTA's gather pipeline running from one
// item to the next: 2.5-6% faster on dsa128k's chunks.  Over an fp8 cache
// (two CTAs per SM) a capped grid measured no faster.
int topk_ctas(int num_sms, bool fp8) { return fp8 ? 0 : num_sms; }

// Mixed micro-batch over a paged cache, bf16 or (fp8) E4M3 codes with
// per-kv-head scales.  Decode rows read the codes directly.  Chunk-attention
// segments of an fp8 cache read the codes directly as well (the fp8 kernel
// widens them in shared memory), unless the workspace also holds the bf16
// widening of their contexts: then they are widened once into it and read by
// the bf16 kernel, which is faster.
int mixed_impl(bool fp8, const void* q, const void* k_cache, const void* v_cache,
               const float* k_scale, const float* v_scale, const int32_t* block_table,
               int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t* cu_seqlens_q,
               const int32_t* ctx_lens, int32_t batch, int heads, int kv_heads, int head_dim_qk,
               int head_dim_v, float softmax_scale, void* out, float* lse, void* workspace,
               size_t workspace_bytes, cudaStream_t st) {
  if (!q || !k_cache || !v_cache || !block_table || !out) return VPP_ERR_INVALID;
  if (num_blocks <= 0 || max_blocks_per_seq <= 0) return VPP_ERR_INVALID;
  if (int r = check_heads(heads, kv_heads)) return r;
  if (!supported_dims(head_dim_qk, head_dim_v)) return VPP_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return VPP_ERR_INVALID;
  static VarlenPlan zero_plan;
  VarlenPlan plan = zero_plan;
  if (int r = build_varlen_plan(cu_seqlens_q, ctx_lens, batch, &plan)) return r;
  for (int b = 0; b < batch; ++b)
    if (ceil_div(ctx_lens[b], kBlockTokens) > max_blocks_per_seq) return VPP_ERR_INVALID;
  const int64_t total_q = cu_seqlens_q[batch];
  if (total_q == 0) return VPP_OK;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;

  // Decode rows go to the split-KV decode kernel when it supports the shape;
  // every other sequence with queries becomes one chunk-attention segment.
  const size_t dws = decode_ws_bytes(cu_seqlens_q, ctx_lens, batch, heads, kv_heads, head_dim_qk,
                                     head_dim_v);
  if (dws > 0 && (!workspace || workspace_bytes < dws || !aligned16(workspace))) return VPP_ERR_WORKSPACE;
  const size_t wws =
      fp8 ? widen_ws_bytes(cu_seqlens_q, ctx_lens, batch, heads, kv_heads, head_dim_qk, head_dim_v) : 0;
  const bool widen = wws > 0 && workspace && aligned16(workspace) && workspace_bytes >= dws + wws;

  // Segments are ordered by per-CTA work (keys per CTA) so the heaviest CTAs
  // start first.
  int order[kMaxBatch];
  int n = 0;
  for (int b = 0; b < batch; ++b)
    if (is_prefill_seg(cu_seqlens_q, b, heads, kv_heads, head_dim_qk, head_dim_v)) order[n++] = b;
  std::stable_sort(order, order + n, [&](int a, int b) { return ctx_lens[a] > ctx_lens[b]; });

  CUtensorMap tm_q, tm_k, tm_v;
  if (make_q_map(&tm_q, q, total_q, heads, kv_heads, head_dim_qk)) return VPP_ERR_INVALID;
  int64_t kv_base[kMaxBatch];
  if (widen) {
    static WidenPlan zero_wplan;
    WidenPlan wp = zero_wplan;
    wp.n = n;
    wp.max_blocks_per_seq = max_blocks_per_seq;
    int64_t rows = 0;
    for (int i = 0; i < n; ++i) {
      wp.table_row[i] = order[i];
      wp.base[i] = rows;
      kv_base[i] = rows;
      rows += ctx_lens[order[i]];
    }
    wp.base[n] = rows;
    if (rows > INT32_MAX / 2) return VPP_ERR_INVALID;
    uint8_t* ws = static_cast<uint8_t*>(workspace) + dws;
    uint16_t* k16 = reinterpret_cast<uint16_t*>(ws);
    uint16_t* v16 = reinterpret_cast<uint16_t*>(ws + round_up((size_t)rows * kv_heads * head_dim_qk * 2, 256));
    if (make_contig_map(&tm_k, k16, rows, kv_heads, head_dim_qk) ||
        make_contig_map(&tm_v, v16, rows, kv_heads, head_dim_v))
      return VPP_ERR_INVALID;
    if (launch_kv_widen_fp8(k_cache, v_cache, k16, v16, kv_heads, head_dim_qk, head_dim_v, block_table,
                            num_blocks, wp, ds->status, ds->num_sms, st) != cudaSuccess)
      return VPP_ERR_CUDA;
  } else if (fp8 ? make_paged_map_u8(&tm_k, k_cache, num_blocks, kv_heads, head_dim_qk) ||
                       make_paged_map_u8(&tm_v, v_cache, num_blocks, kv_heads, head_dim_v)
                 : make_paged_map(&tm_k, k_cache, num_blocks, kv_heads, head_dim_qk) ||
                       make_paged_map(&tm_v, v_cache, num_blocks, kv_heads, head_dim_v)) {
    return VPP_ERR_INVALID;
  }

  const float scale_log2 =
      (softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)head_dim_qk)) * 1.4426950408889634f;

  // Decode rows, longest context first.
  static DecodeParams zero_dp;
  DecodeParams dp = zero_dp;
  int drows[kMaxBatch];
  int nd = 0;
  int64_t dp_items = 0;
  for (int b = 0; b < batch; ++b)
    if (is_decode_row(cu_seqlens_q, b, heads, kv_heads, head_dim_qk, head_dim_v) && ctx_lens[b] > 0)
      drows[nd++] = b;
  if (nd > 0) {
    std::stable_sort(drows, drows + nd, [&](int a, int b) { return ctx_lens[a] > ctx_lens[b]; });
    int64_t items = 0;
    for (int i = 0; i < nd; ++i) {
      const int b = drows[i];
      dp.rows[i].b = b;
      dp.rows[i].q_row = cu_seqlens_q[b];
      dp.rows[i].ctx = ctx_lens[b];
      dp.rows[i].item0 = (int32_t)items;
      items += ceil_div(ctx_lens[b], kDecodeSplitTokens);
    }
    if (items > INT32_MAX) return VPP_ERR_INVALID;
    dp_items = items;
    dp.n_rows = nd;
    dp.heads = heads;
    dp.kv_heads = kv_heads;
    dp.split_tokens = kDecodeSplitTokens;
    dp.num_blocks = num_blocks;
    dp.max_blocks_per_seq = max_blocks_per_seq;
    dp.scale_log2 = scale_log2;
    dp.q = static_cast<const uint16_t*>(q);
    dp.k_cache = k_cache;
    dp.v_cache = v_cache;
    dp.k_scale = fp8 ? k_scale : nullptr;
    dp.v_scale = fp8 ? v_scale : nullptr;
    dp.block_table = block_table;
    dp.out = static_cast<uint16_t*>(out);
    dp.lse = lse;
    dp.lse_stride = total_q;
    if (dws > 0) {
      dp.ws_o = static_cast<float*>(workspace);
      dp.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                           round_up((size_t)items * heads * head_dim_v * 4, 256));
    }
    dp.status = ds->status;
  }

  // The decode rows (HBM-bound) are launched first, on the side stream, and
  // the prefill segments (tensor-bound) on the caller's stream, so that the
  // two kernels' CTAs share the SMs instead of running one after the other:
  // the decode kernel on the share mixed_decode_ctas gives it, the prefill
  // CTAs on the rest.  They write disjoint rows of out / lse and disjoint
  // workspace.
  std::unique_lock<std::mutex> side_lock(ds->side_mutex, std::defer_lock);
  cudaStream_t dst = st;
  const bool fork = nd > 0 && n > 0;
  if (fork) {
    side_lock.lock();
    if (cudaEventRecord(ds->ev_fork, st) != cudaSuccess ||
        cudaStreamWaitEvent(ds->side, ds->ev_fork, 0) != cudaSuccess)
      return VPP_ERR_CUDA;
    dst = ds->side;
  }
  int err = VPP_OK;
  double prefill_flops = 0.0, decode_bytes = 0.0;
  for (int i = 0; i < n; ++i) {
    const double c = cu_seqlens_q[order[i] + 1] - cu_seqlens_q[order[i]];
    const double pre = ctx_lens[order[i]] - c;
    prefill_flops += 2.0 * (head_dim_qk + head_dim_v) * heads * (c * pre + c * (c + 1) / 2);
  }
  for (int i = 0; i < nd; ++i)
    decode_bytes += (double)ctx_lens[drows[i]] * kv_heads * (head_dim_qk + head_dim_v) * (fp8 ? 1 : 2);
  const int dctas = mixed_decode_ctas(ds->num_sms, fp8, prefill_flops, decode_bytes);
  if (nd > 0 && launch_decode(dp, (int)dp_items, head_dim_qk, fp8, false, ds->num_sms, dctas, dst) != cudaSuccess)
    err = VPP_ERR_CUDA;
  if (fork && cudaEventRecord(ds->ev_join, ds->side) != cudaSuccess) err = VPP_ERR_CUDA;
  if (err == VPP_OK) {
    static AttnParams zero_params;
    AttnParams p = zero_params;
    p.heads = heads;
    p.kv_heads = kv_heads;
    p.group = heads / kv_heads;
    p.num_blocks = num_blocks;
    p.paged = widen ? 0 : 1;
    p.scale_log2 = scale_log2;
    p.block_table = block_table;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.lse_stride = total_q;
    p.k_scale = fp8 ? k_scale : nullptr;
    p.v_scale = fp8 ? v_scale : nullptr;
    p.status = ds->status;
    for (int i0 = 0; i0 < n; i0 += kMaxAttnSegs) {
      const int cnt = std::min(kMaxAttnSegs, n - i0);
      int64_t cta = 0;
      p.n_segs = cnt;
      for (int i = 0; i < cnt; ++i) {
        const int b = order[i0 + i];
        AttnSeg& s = p.segs[i];
        s.q_start = cu_seqlens_q[b];
        s.q_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        s.kv_len = ctx_lens[b];
        s.table_off = b * max_blocks_per_seq;
        s.n_pairs = pairs_for(s.q_len, p.group);
        s.n_splits = 1;
        s.split_keys = 0;
        s.cta_begin = (int32_t)cta;
        s.kv_base = widen ? (int32_t)kv_base[i0 + i] : 0;
        s.ws_row0 = 0;
        cta += (int64_t)s.n_pairs * kv_heads;
      }
      if (cta > INT32_MAX) {
        err = VPP_ERR_INVALID;
        break;
      }
      if (launch_chunk_attn(head_dim_qk, head_dim_v, fp8 && !widen, tm_q, tm_k, tm_v, p, (int)cta, st) !=
          cudaSuccess) {
        err = VPP_ERR_CUDA;
        break;
      }
    }
  }
  // Join even after an error, so that the caller's stream covers every
  // launch that was made.
  if (fork && cudaStreamWaitEvent(st, ds->ev_join, 0) != cudaSuccess && err == VPP_OK) err = VPP_ERR_CUDA;
  return err;
}

// Top-k sparse prefix attention (DSA-style) of one chunk through the decode
// kernel's gather mode: one work item per (token, range of 1024 list entries).
size_t topk_ws_bytes(int64_t C, int32_t topk, int heads, int d) {
  const int64_t S = ceil_div(topk, kDecodeSplitTokens);
  if (S <= 1 || C <= 0) return 0;
  return round_up((size_t)C * S * heads * d * 4, 256) + round_up((size_t)C * S * heads * 4, 256);
}

int topk_impl(bool fp8, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
              const float* v_scale, const int32_t* block_table, int32_t num_blocks, int64_t P, int64_t C,
              const int32_t* topk_idx, const int32_t* topk_len, int32_t topk, int heads, int kv_heads, int d,
              float softmax_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
              cudaStream_t st) {
  if (P < 0 || C < 0 || num_blocks <= 0 || topk < 1) return VPP_ERR_INVALID;
  if (C == 0) return VPP_OK;  // pointers may be NULL for an empty chunk
  if (!q || !k_cache || !v_cache || !out || !topk_idx || !topk_len) return VPP_ERR_INVALID;
  if (fp8 && !scales_ok(k_scale, v_scale)) return VPP_ERR_INVALID;
  if (int r = check_heads(heads, kv_heads)) return r;
  if (!decode_supported(d, d, heads, kv_heads)) return VPP_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(topk_len) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return VPP_ERR_INVALID;
  if (block_table ? (int64_t)num_blocks * kBlockTokens < P + C : (int64_t)num_blocks < P + C)
    return VPP_ERR_INVALID;
  const int64_t S = ceil_div(topk, kDecodeSplitTokens);
  const int64_t items = C * S;
  if (items > INT32_MAX || C > INT32_MAX) return VPP_ERR_INVALID;
  const size_t need = topk_ws_bytes(C, topk, heads, d);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return VPP_ERR_WORKSPACE;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;
  static DecodeParams zero_dp;
  DecodeParams dp = zero_dp;
  dp.heads = heads;
  dp.kv_heads = kv_heads;
  dp.split_tokens = kDecodeSplitTokens;
  dp.num_blocks = num_blocks;
  dp.scale_log2 = (softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)d)) * 1.4426950408889634f;
  dp.q = static_cast<const uint16_t*>(q);
  dp.k_cache = k_cache;
  dp.v_cache = v_cache;
  dp.k_scale = fp8 ? k_scale : nullptr;
  dp.v_scale = fp8 ? v_scale : nullptr;
  dp.block_table = block_table;
  dp.out = static_cast<uint16_t*>(out);
  dp.lse = lse;
  dp.lse_stride = C;
  if (need > 0) {
    dp.ws_o = static_cast<float*>(workspace);
    dp.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         round_up((size_t)items * heads * d * 4, 256));
  }
  dp.status = ds->status;
  dp.topk_idx = topk_idx;
  dp.topk_len = topk_len;
  dp.topk = topk;
  dp.topk_splits = (int32_t)S;
  dp.topk_prefix = P;
  dp.topk_tokens = C;
  if (launch_decode(dp, (int)items, d, fp8, true, ds->num_sms, topk_ctas(ds->num_sms, fp8), st) != cudaSuccess)
    return VPP_ERR_CUDA;
  return VPP_OK;
}

}  // namespace

namespace vpp {
// Entry into the chunk-attention planner and launcher for other translation
// units of this library (same contract as vpp_chunk_attn_ex).
int run_chunk_attn(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                   const int32_t* block_table, int32_t num_blocks, int64_t prefix_len,
                   int64_t chunk_len, int heads, int kv_heads, int head_dim_qk, int head_dim_v,
                   float softmax_scale, int num_splits, void* out, float* lse, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  return chunk_attn_impl(q, q_dtype, k_cache, v_cache, block_table, num_blocks, prefix_len,
                         chunk_len, heads, kv_heads, head_dim_qk, head_dim_v, softmax_scale,
                         num_splits, out, lse, workspace, workspace_bytes, stream);
}
}  // namespace vpp

extern "C" {

const char* vpp_status_string(int status) {
  switch (status) {
    case VPP_OK: return "VPP_OK";
    case VPP_ERR_INVALID: return "VPP_ERR_INVALID: invalid argument";
    case VPP_ERR_UNSUPPORTED: return "VPP_ERR_UNSUPPORTED: unsupported shape or device";
    case VPP_ERR_CUDA: return "VPP_ERR_CUDA: a CUDA call failed";
    case VPP_ERR_TIMEOUT: return "VPP_ERR_TIMEOUT: a device-side wait timed out";
    case VPP_ERR_WORKSPACE: return "VPP_ERR_WORKSPACE: workspace missing or too small";
    default: return "unknown vpp status";
  }
}

int vpp_version(void) { return 100; }

int vpp_kv_append(const void* k_new, const void* v_new, int in_dtype, void* k_cache,
                  void* v_cache, const int32_t* block_table, int32_t num_blocks,
                  int64_t prefix_len, int64_t chunk_len, int kv_heads, int head_dim_qk,
                  int head_dim_v, void* stream) {
  if (prefix_len < 0 || chunk_len < 0 || num_blocks <= 0 || kv_heads <= 0) return VPP_ERR_INVALID;
  if (chunk_len == 0) return VPP_OK;  // pointers may be NULL for an empty chunk
  if (!k_new || !v_new || !k_cache || !v_cache) return VPP_ERR_INVALID;
  if (in_dtype != VPP_BF16 && in_dtype != VPP_FP32) return VPP_ERR_INVALID;
  if (head_dim_qk <= 0 || head_dim_v <= 0 || head_dim_qk % 64 || head_dim_v % 64)
    return VPP_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return VPP_ERR_INVALID;
  const int64_t end = prefix_len + chunk_len;
  if (block_table ? (int64_t)num_blocks * kBlockTokens < end : (int64_t)num_blocks < end)
    return VPP_ERR_INVALID;
  if (chunk_len == 0) return VPP_OK;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;
  if (launch_kv_append(k_new, v_new, in_dtype == VPP_FP32, k_cache, v_cache, block_table,
                       num_blocks, prefix_len, chunk_len, kv_heads, head_dim_qk, head_dim_v,
                       ds->status, ds->num_sms, as_stream(stream)) != cudaSuccess)
    return VPP_ERR_CUDA;
  return VPP_OK;
}

int vpp_kv_append_varlen(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int32_t* block_table, int32_t max_blocks_per_seq,
                         int32_t num_blocks, const int32_t* cu_seqlens_q,
                         const int32_t* ctx_lens, int32_t batch, int kv_heads, int head_dim_qk,
                         int head_dim_v, void* stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table) return VPP_ERR_INVALID;
  if (num_blocks <= 0 || kv_heads <= 0 || max_blocks_per_seq <= 0) return VPP_ERR_INVALID;
  if (head_dim_qk <= 0 || head_dim_v <= 0 || head_dim_qk % 64 || head_dim_v % 64)
    return VPP_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return VPP_ERR_INVALID;
  static VarlenPlan zero_plan;
  VarlenPlan plan = zero_plan;
  plan.max_blocks_per_seq = max_blocks_per_seq;
  if (int r = build_varlen_plan(cu_seqlens_q, ctx_lens, batch, &plan)) return r;
  for (int b = 0; b < batch; ++b)
    if (ceil_div(ctx_lens[b], kBlockTokens) > max_blocks_per_seq) return VPP_ERR_INVALID;
  if (plan.cu_q[batch] == 0) return VPP_OK;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;
  if (launch_kv_append_varlen(k_new, v_new, k_cache, v_cache, block_table, plan, num_blocks,
                              kv_heads, head_dim_qk, head_dim_v, ds->status, ds->num_sms,
                              as_stream(stream)) != cudaSuccess)
    return VPP_ERR_CUDA;
  return VPP_OK;
}

int vpp_chunk_attn(const void* q, const void* k_cache, const void* v_cache, int64_t prefix_len,
                   int64_t chunk_len, int heads, int kv_heads, int head_dim, void* out,
                   float* lse, void* stream) {
  if (prefix_len < 0 || chunk_len < 0) return VPP_ERR_INVALID;
  const int64_t cap = prefix_len + chunk_len;
  if (cap > INT32_MAX) return VPP_ERR_INVALID;
  return chunk_attn_impl(q, VPP_BF16, k_cache, v_cache, nullptr, (int32_t)std::max<int64_t>(cap, 1),
                         prefix_len, chunk_len, heads, kv_heads, head_dim, head_dim, 0.f, 1, out,
                         lse, nullptr, 0, as_stream(stream));
}

int vpp_chunk_attn_ex(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, int32_t num_blocks, int64_t prefix_len,
                      int64_t chunk_len, int heads, int kv_heads, int head_dim_qk,
                      int head_dim_v, float softmax_scale, int num_splits, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return chunk_attn_impl(q, q_dtype, k_cache, v_cache, block_table, num_blocks, prefix_len,
                         chunk_len, heads, kv_heads, head_dim_qk, head_dim_v, softmax_scale,
                         num_splits, out, lse, workspace, workspace_bytes, as_stream(stream));
}

int vpp_chunk_attn_plan(int64_t prefix_len, int64_t chunk_len, int heads, int kv_heads, int head_dim_qk,
                        int head_dim_v, int num_splits, int64_t* split_token) {
  if (prefix_len < 0 || chunk_len < 0 || num_splits < 0) return VPP_ERR_INVALID;
  if (int r = check_heads(heads, kv_heads)) return r;
  if (!supported_dims(head_dim_qk, head_dim_v)) return VPP_ERR_UNSUPPORTED;
  DeviceState* ds = nullptr;
  int num_sms = 152;
  if (device_state(&ds) == VPP_OK) num_sms = ds->num_sms;
  const ChunkPlan pl = plan_chunk(prefix_len, chunk_len, heads, kv_heads, head_dim_qk, head_dim_v, num_splits,
                                  num_sms);
  if (split_token) *split_token = pl.n_splits > 1 ? pl.t0 : 0;
  return pl.n_splits;
}

int vpp_chunk_attn_num_splits(int64_t prefix_len, int64_t chunk_len, int heads, int kv_heads,
                              int head_dim_qk, int head_dim_v, int num_splits) {
  return vpp_chunk_attn_plan(prefix_len, chunk_len, heads, kv_heads, head_dim_qk, head_dim_v, num_splits,
                             nullptr);
}

size_t vpp_chunk_attn_workspace_size(int q_dtype, int64_t prefix_len, int64_t chunk_len,
                                     int heads, int kv_heads, int head_dim_qk, int head_dim_v,
                                     int num_splits) {
  int64_t t0 = 0;
  const int S = vpp_chunk_attn_plan(prefix_len, chunk_len, heads, kv_heads, head_dim_qk, head_dim_v,
                                    num_splits, &t0);
  if (S < 1) return 0;
  return ws_q_bytes(q_dtype, chunk_len, heads, head_dim_qk) +
         ws_split(ChunkPlan{(int)t0, S, 0}, chunk_len, heads, head_dim_v).total();
}

int vpp_mixed_attn(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                   const int32_t* cu_seqlens_q, const int32_t* ctx_lens, int32_t batch,
                   int heads, int kv_heads, int head_dim_qk, int head_dim_v,
                   float softmax_scale, void* out, float* lse, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return mixed_impl(false, q, k_cache, v_cache, nullptr, nullptr, block_table, max_blocks_per_seq,
                    num_blocks, cu_seqlens_q, ctx_lens, batch, heads, kv_heads, head_dim_qk,
                    head_dim_v, softmax_scale, out, lse, workspace, workspace_bytes, as_stream(stream));
}

size_t vpp_mixed_attn_workspace_size(const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                     int32_t batch, int heads, int kv_heads, int head_dim_qk,
                                     int head_dim_v) {
  if (!cu_seqlens_q || !ctx_lens || batch <= 0 || batch > kMaxBatch) return 0;
  if (check_heads(heads, kv_heads) != VPP_OK) return 0;
  return decode_ws_bytes(cu_seqlens_q, ctx_lens, batch, heads, kv_heads, head_dim_qk, head_dim_v);
}

// ------------------------------------------------------------- fp8 (E4M3) KV cache
int vpp_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const float* k_scale, const float* v_scale, const int32_t* block_table,
                      int32_t num_blocks, int64_t prefix_len, int64_t chunk_len, int kv_heads,
                      int head_dim_qk, int head_dim_v, void* stream) {
  if (prefix_len < 0 || chunk_len < 0 || num_blocks <= 0 || kv_heads <= 0) return VPP_ERR_INVALID;
  if (chunk_len == 0) return VPP_OK;  // pointers may be NULL for an empty chunk
  if (!k_new || !v_new || !k_cache || !v_cache || !scales_ok(k_scale, v_scale)) return VPP_ERR_INVALID;
  if (head_dim_qk <= 0 || head_dim_v <= 0 || head_dim_qk % 64 || head_dim_v % 64)
    return VPP_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return VPP_ERR_INVALID;
  const int64_t end = prefix_len + chunk_len;
  if (block_table ? (int64_t)num_blocks * kBlockTokens < end : (int64_t)num_blocks < end)
    return VPP_ERR_INVALID;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;
  if (launch_kv_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, num_blocks,
                           prefix_len, chunk_len, kv_heads, head_dim_qk, head_dim_v, ds->status,
                           ds->num_sms, as_stream(stream)) != cudaSuccess)
    return VPP_ERR_CUDA;
  return VPP_OK;
}

int vpp_kv_append_varlen_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const float* k_scale, const float* v_scale, const int32_t* block_table,
                             int32_t max_blocks_per_seq, int32_t num_blocks,
                             const int32_t* cu_seqlens_q, const int32_t* ctx_lens, int32_t batch,
                             int kv_heads, int head_dim_qk, int head_dim_v, void* stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !scales_ok(k_scale, v_scale))
    return VPP_ERR_INVALID;
  if (num_blocks <= 0 || kv_heads <= 0 || max_blocks_per_seq <= 0) return VPP_ERR_INVALID;
  if (head_dim_qk <= 0 || head_dim_v <= 0 || head_dim_qk % 64 || head_dim_v % 64)
    return VPP_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return VPP_ERR_INVALID;
  static VarlenPlan zero_plan;
  VarlenPlan plan = zero_plan;
  plan.max_blocks_per_seq = max_blocks_per_seq;
  if (int r = build_varlen_plan(cu_seqlens_q, ctx_lens, batch, &plan)) return r;
  for (int b = 0; b < batch; ++b)
    if (ceil_div(ctx_lens[b], kBlockTokens) > max_blocks_per_seq) return VPP_ERR_INVALID;
  if (plan.cu_q[batch] == 0) return VPP_OK;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;
  if (launch_kv_append_fp8_varlen(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, plan,
                                  num_blocks, kv_heads, head_dim_qk, head_dim_v, ds->status, ds->num_sms,
                                  as_stream(stream)) != cudaSuccess)
    return VPP_ERR_CUDA;
  return VPP_OK;
}

// Bytes of the bf16 copy of keys 0 .. prefix_len + chunk_len - 1.
size_t fp8_widen_bytes(int64_t n, int kv_heads, int dq, int dv) {
  return round_up((size_t)n * kv_heads * dq * 2, 256) + round_up((size_t)n * kv_heads * dv * 2, 256);
}

int vpp_chunk_attn_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                       const float* v_scale, const int32_t* block_table, int32_t num_blocks,
                       int64_t prefix_len, int64_t chunk_len, int heads, int kv_heads, int head_dim_qk,
                       int head_dim_v, float softmax_scale, int num_splits, void* out, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream) {
  const int64_t P = prefix_len, C = chunk_len;
  if (C > 0 && !scales_ok(k_scale, v_scale)) return VPP_ERR_INVALID;
  cudaStream_t st = as_stream(stream);
  if (P >= 0 && C > 0 && P + C <= (int64_t)INT32_MAX / 2 && kv_heads > 0 && head_dim_qk > 0 && head_dim_v > 0 &&
      num_splits >= 0 && workspace && aligned16(workspace) && k_cache && v_cache && num_blocks > 0 &&
      (block_table ? (int64_t)num_blocks * kBlockTokens >= P + C : (int64_t)num_blocks >= P + C) &&
      check_heads(heads, kv_heads) == VPP_OK && supported_dims(head_dim_qk, head_dim_v)) {
    const int64_t n = P + C;
    const size_t wb = fp8_widen_bytes(n, kv_heads, head_dim_qk, head_dim_v);
    const size_t rest = vpp_chunk_attn_workspace_size(VPP_BF16, P, C, heads, kv_heads, head_dim_qk,
                                                      head_dim_v, num_splits);
    if (workspace_bytes >= wb + rest) {
      // The caller gave room for a bf16 copy of the visible keys: widen them
      // once and run the bf16 kernel on it.
      DeviceState* ds = nullptr;
      if (int r = device_state(&ds)) return r;
      static WidenPlan zero_plan;
      WidenPlan wp = zero_plan;
      wp.n = 1;
      wp.base[1] = n;
      uint8_t* ws = static_cast<uint8_t*>(workspace);
      uint16_t* k16 = reinterpret_cast<uint16_t*>(ws);
      uint16_t* v16 = reinterpret_cast<uint16_t*>(ws + round_up((size_t)n * kv_heads * head_dim_qk * 2, 256));
      if (!aligned16(q) || !q || !out) return VPP_ERR_INVALID;
      if (launch_kv_widen_fp8(k_cache, v_cache, k16, v16, kv_heads, head_dim_qk, head_dim_v, block_table,
                              num_blocks, wp, ds->status, ds->num_sms, st) != cudaSuccess)
        return VPP_ERR_CUDA;
      return chunk_attn_impl(q, VPP_BF16, k16, v16, nullptr, (int32_t)n, P, C, heads, kv_heads, head_dim_qk,
                             head_dim_v, softmax_scale, num_splits, out, lse, ws + wb, workspace_bytes - wb, st,
                             k_scale, v_scale);
    }
  }
  // The fp8 kernel reads the codes and widens them in shared memory.
  return chunk_attn_impl(q, VPP_BF16, k_cache, v_cache, block_table, num_blocks, prefix_len, chunk_len, heads,
                         kv_heads, head_dim_qk, head_dim_v, softmax_scale, num_splits, out, lse, workspace,
                         workspace_bytes, st, k_scale, v_scale, true);
}

size_t vpp_chunk_attn_fp8_workspace_size(int64_t prefix_len, int64_t chunk_len, int heads, int kv_heads,
                                         int head_dim_qk, int head_dim_v, int num_splits) {
  return vpp_chunk_attn_workspace_size(VPP_BF16, prefix_len, chunk_len, heads, kv_heads, head_dim_qk,
                                       head_dim_v, num_splits);
}

size_t vpp_chunk_attn_fp8_widen_workspace_size(int64_t prefix_len, int64_t chunk_len, int heads, int kv_heads,
                                               int head_dim_qk, int head_dim_v, int num_splits) {
  if (prefix_len < 0 || chunk_len <= 0 || kv_heads <= 0 || head_dim_qk <= 0 || head_dim_v <= 0) return 0;
  return fp8_widen_bytes(prefix_len + chunk_len, kv_heads, head_dim_qk, head_dim_v) +
         vpp_chunk_attn_workspace_size(VPP_BF16, prefix_len, chunk_len, heads, kv_heads, head_dim_qk,
                                       head_dim_v, num_splits);
}

int vpp_mixed_attn_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                       const float* v_scale, const int32_t* block_table, int32_t max_blocks_per_seq,
                       int32_t num_blocks, const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                       int32_t batch, int heads, int kv_heads, int head_dim_qk, int head_dim_v,
                       float softmax_scale, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!scales_ok(k_scale, v_scale)) return VPP_ERR_INVALID;
  return mixed_impl(true, q, k_cache, v_cache, k_scale, v_scale, block_table, max_blocks_per_seq,
                    num_blocks, cu_seqlens_q, ctx_lens, batch, heads, kv_heads, head_dim_qk,
                    head_dim_v, softmax_scale, out, lse, workspace, workspace_bytes, as_stream(stream));
}

size_t vpp_mixed_attn_fp8_workspace_size(const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                         int32_t batch, int heads, int kv_heads, int head_dim_qk,
                                         int head_dim_v) {
  if (!cu_seqlens_q || !ctx_lens || batch <= 0 || batch > kMaxBatch) return 0;
  if (check_heads(heads, kv_heads) != VPP_OK) return 0;
  return decode_ws_bytes(cu_seqlens_q, ctx_lens, batch, heads, kv_heads, head_dim_qk, head_dim_v);
}

size_t vpp_mixed_attn_fp8_widen_workspace_size(const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                               int32_t batch, int heads, int kv_heads, int head_dim_qk,
                                               int head_dim_v) {
  if (!cu_seqlens_q || !ctx_lens || batch <= 0 || batch > kMaxBatch) return 0;
  if (check_heads(heads, kv_heads) != VPP_OK) return 0;
  return decode_ws_bytes(cu_seqlens_q, ctx_lens, batch, heads, kv_heads, head_dim_qk, head_dim_v) +
         widen_ws_bytes(cu_seqlens_q, ctx_lens, batch, heads, kv_heads, head_dim_qk, head_dim_v);
}

// ------------------------------------------------------------- top-k sparse prefix
int vpp_topk_chunk_attn(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        int32_t num_blocks, int64_t prefix_len, int64_t chunk_len, const int32_t* topk_idx,
                        const int32_t* topk_len, int32_t topk, int heads, int kv_heads, int head_dim,
                        float softmax_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream) {
  return topk_impl(false, q, k_cache, v_cache, nullptr, nullptr, block_table, num_blocks, prefix_len, chunk_len,
                   topk_idx, topk_len, topk, heads, kv_heads, head_dim, softmax_scale, out, lse, workspace,
                   workspace_bytes, as_stream(stream));
}

int vpp_topk_chunk_attn_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                            const float* v_scale, const int32_t* block_table, int32_t num_blocks,
                            int64_t prefix_len, int64_t chunk_len, const int32_t* topk_idx,
                            const int32_t* topk_len, int32_t topk, int heads, int kv_heads, int head_dim,
                            float softmax_scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!scales_ok(k_scale, v_scale)) return VPP_ERR_INVALID;
  return topk_impl(true, q, k_cache, v_cache, k_scale, v_scale, block_table, num_blocks, prefix_len, chunk_len,
                   topk_idx, topk_len, topk, heads, kv_heads, head_dim, softmax_scale, out, lse, workspace,
                   workspace_bytes, as_stream(stream));
}

size_t vpp_topk_chunk_attn_workspace_size(int64_t chunk_len, int32_t topk, int heads, int head_dim) {
  if (chunk_len <= 0 || topk < 1 || heads <= 0 || head_dim <= 0) return 0;
  return topk_ws_bytes(chunk_len, topk, heads, head_dim);
}

int vpp_last_device_status(void* stream, int* code) {
  if (!code) return VPP_ERR_INVALID;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;
  cudaStream_t st = as_stream(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, ds->status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(ds->status, 0, sizeof(int), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return VPP_ERR_CUDA;
  *code = host;
  return VPP_OK;
}

int vpp_selftest_wait_timeout(int timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 5000000) return VPP_ERR_INVALID;
  DeviceState* ds = nullptr;
  if (int r = device_state(&ds)) return r;
  if (launch_wait_timeout_selftest(timeout_us, ds->status, as_stream(stream)) != cudaSuccess)
    return VPP_ERR_CUDA;
  return VPP_OK;
}

}  // extern "C"
