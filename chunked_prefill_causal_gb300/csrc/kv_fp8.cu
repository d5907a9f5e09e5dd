// kv_fp8.cu -- fp8 (E4M3) KV cache: quantising append, and the exact widening
// of cached codes to bf16 for callers that trade workspace for prefill speed.
//
// "02 · 并行策略与 PP 切分" (deployment note), §1 and §3.2: the KV cache is
// kept in fp8, about half the bytes per token of bf16, which nearly doubles
// the tokens one GPU holds.  Element format: E4M3 of the OCP 8-bit floating
// point specification (bias 7, 3 mantissa bits, largest finite 448).  One
// float32 scale per kv head for K and one for V; an element's value is
// E4M3(code) x scale.
//
// Append: code = E4M3 round-to-nearest-even of the float32 quotient x / scale
// (correctly rounded), magnitudes above 448 clamped to 448.  A thread turns 16
// bf16 values (32 bytes) into 16 codes (one 16-byte store); HBM-bound:
// 3 bytes per element (2 read, 1 written).
//
// Widening (optional prefill path): every E4M3 value is exactly a bf16
// value, so a caller that provides a workspace for the bf16 copy of the
// visible keys gets them widened once, without their scales (3 bytes per
// element again), and the bf16 attention kernel applies the scales (k_scale
// in the score scale, v_scale on the output), leaving the arithmetic exact.
// Without that workspace the fp8 attention kernel widens the codes itself.
#include "common.cuh"
#include "fp8.cuh"
#include "ptx.cuh"

namespace vpp {
namespace {

// x / s rounded to nearest even in float32, from y = RN(1/s): q = RN(x y) is
// within one ulp of x / s, the residual x - q s is exact with an FMA, and
// RN(q + (x - q s) y) is the correctly rounded quotient (Markstein's theorem
// on Newton-Raphson division: P. Markstein, "IA-64 and Elementary Functions",
// 2000; also Cornea, Harrison and Tang, 2002).  Quotients here stay far from
// overflow and underflow (|x| <= bf16 range, scales are ordinary factors);
// a zero x keeps its sign.
__device__ __forceinline__ float div_rn(float x, float s, float y) {
  const float q = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q, s, x);
  const float q1 = __fmaf_rn(r, y, q);
  return x == 0.f ? x : q1;
}

// 16 bf16 values -> 16 E4M3 codes, each divided by s first (y = RN(1/s)).
__device__ __forceinline__ uint4 quantise16(const uint4 a, const uint4 b, float s, float y) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w0 = w[2 * i], w1 = w[2 * i + 1];
    const float x0 = __uint_as_float(w0 << 16), x1 = __uint_as_float(w0 & 0xFFFF0000u);
    const float x2 = __uint_as_float(w1 << 16), x3 = __uint_as_float(w1 & 0xFFFF0000u);
    const uint32_t lo = pack_e4m3x2(div_rn(x0, s, y), div_rn(x1, s, y));
    const uint32_t hi = pack_e4m3x2(div_rn(x2, s, y), div_rn(x3, s, y));
    out[i] = lo | (hi << 16);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Two E4M3 codes to two floats (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  float2 f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
      : "=f"(f.x), "=f"(f.y)
      : "r"(h2));
  return f;
}

// 16 E4M3 codes -> 16 bf16 values (exact).
__device__ __forceinline__ void widen16(const uint4 c, uint4* dst) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f0 = e4m3x2_to_f32x2(static_cast<uint16_t>(w[i] & 0xFFFFu));
    const float2 f1 = e4m3x2_to_f32x2(static_cast<uint16_t>(w[i] >> 16));
    o[2 * i] = pack_bf16x2(f0.x, f0.y);
    o[2 * i + 1] = pack_bf16x2(f1.x, f1.y);
  }
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Cache row of packed new row t: single sequence (paged or contiguous).
struct SeqPos {
  int64_t prefix;
  const int32_t* table;  // nullptr: contiguous cache, num_blocks = capacity in tokens
  __device__ __forceinline__ bool slot(int64_t t, int32_t num_blocks, int64_t* row) const {
    const int64_t pos = prefix + t;
    if (!table) {
      *row = pos;
      return pos < num_blocks;
    }
    const int32_t blk = table[pos / kBlockTokens];
    if (blk < 0 || blk >= num_blocks) return false;
    *row = static_cast<int64_t>(blk) * kBlockTokens + pos % kBlockTokens;
    return true;
  }
};

// Cache row of packed new row t of a varlen batch.
struct BatchPos {
  const VarlenPlan* plan;
  const int32_t* table;
  __device__ __forceinline__ bool slot(int64_t t, int32_t num_blocks, int64_t* row) const {
    int lo = 0, hi = plan->batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (plan->cu_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int64_t qlen = plan->cu_q[lo + 1] - plan->cu_q[lo];
    const int64_t pos = plan->ctx[lo] - qlen + (t - plan->cu_q[lo]);
    const int32_t blk = table[static_cast<int64_t>(lo) * plan->max_blocks_per_seq + pos / kBlockTokens];
    if (blk < 0 || blk >= num_blocks) return false;
    *row = static_cast<int64_t>(blk) * kBlockTokens + pos % kBlockTokens;
    return true;
  }
};

// One grid-stride loop over (new row, 16-element vector) of one tensor, two
// vectors per thread and iteration (both loads issued before either store),
// with the (row, vector) index advanced by the stride instead of divided.
template <typename Pos>
__device__ __forceinline__ void quantise_rows(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                              const float* __restrict__ scale, int64_t tokens, int d,
                                              int vec_per_row, Pos pos, int32_t num_blocks, int* status) {
  const int64_t total = tokens * vec_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int vec_per_head = d / 16;
  const int64_t dt = stride / vec_per_row;
  const int dv = static_cast<int>(stride - dt * vec_per_row);
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t t = i / vec_per_row;
  int v = static_cast<int>(i - t * vec_per_row);
  auto advance = [&](int64_t& tt, int& vv) {
    tt += dt;
    vv += dv;
    if (vv >= vec_per_row) {
      vv -= vec_per_row;
      ++tt;
    }
  };
  for (; i < total; i += 2 * stride) {
    int64_t t2 = t;
    int v2 = v;
    advance(t2, v2);
    const bool has2 = i + stride < total;
    int64_t row = 0, row2 = 0;
    const bool ok1 = pos.slot(t, num_blocks, &row);
    const bool ok2 = has2 && pos.slot(t2, num_blocks, &row2);
    uint4 a1 = make_uint4(0u, 0u, 0u, 0u), b1 = a1, a2 = a1, b2 = a1;
    if (ok1) {
      a1 = __ldg(&src[2 * i]);
      b1 = __ldg(&src[2 * i + 1]);
    }
    if (ok2) {
      a2 = __ldg(&src[2 * (i + stride)]);
      b2 = __ldg(&src[2 * (i + stride) + 1]);
    }
    if (ok1) {
      const float sc = __ldg(scale + v / vec_per_head);
      dst[row * vec_per_row + v] = quantise16(a1, b1, sc, __frcp_rn(sc));
    } else if (v == 0) {
      record_status(status, kStatusInvalid);
    }
    if (ok2) {
      const float sc = __ldg(scale + v2 / vec_per_head);
      dst[row2 * vec_per_row + v2] = quantise16(a2, b2, sc, __frcp_rn(sc));
    } else if (has2 && v2 == 0) {
      record_status(status, kStatusInvalid);
    }
    t = t2;
    v = v2;
    advance(t, v);
  }
}

template <typename Pos>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* k_cache, uint4* v_cache,
    const float* __restrict__ k_scale, const float* __restrict__ v_scale, int64_t tokens, int kv_heads,
    int dq, int dv, int32_t num_blocks, Pos pos, int* status) {
  quantise_rows(k_new, k_cache, k_scale, tokens, dq, kv_heads * dq / 16, pos, num_blocks, status);
  quantise_rows(v_new, v_cache, v_scale, tokens, dv, kv_heads * dv / 16, pos, num_blocks, status);
}

__global__ void __launch_bounds__(256) kv_append_fp8_varlen_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* k_cache, uint4* v_cache,
    const float* __restrict__ k_scale, const float* __restrict__ v_scale, int kv_heads, int dq, int dv,
    int32_t num_blocks, const int32_t* table, const __grid_constant__ VarlenPlan plan, int* status) {
  BatchPos pos{&plan, table};
  const int64_t tokens = plan.cu_q[plan.batch];
  quantise_rows(k_new, k_cache, k_scale, tokens, dq, kv_heads * dq / 16, pos, num_blocks, status);
  quantise_rows(v_new, v_cache, v_scale, tokens, dv, kv_heads * dv / 16, pos, num_blocks, status);
}

// Widens the keys 0 .. ctx-1 of every listed sequence into consecutive rows
// of a contiguous bf16 buffer (row base[i] + t for token t of entry i).
__device__ __forceinline__ void widen_rows(const uint4* __restrict__ cache, uint4* __restrict__ dst,
                                           int vec_per_row, const WidenPlan& plan,
                                           const int32_t* __restrict__ table, int32_t num_blocks,
                                           int* status) {
  const int64_t total = plan.base[plan.n] * vec_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t r = i / vec_per_row;
    const int v = static_cast<int>(i - r * vec_per_row);
    int lo = 0, hi = plan.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (plan.base[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int64_t t = r - plan.base[lo];
    int64_t src;
    if (table) {
      const int32_t blk = table[static_cast<int64_t>(plan.table_row[lo]) * plan.max_blocks_per_seq +
                                t / kBlockTokens];
      if (blk < 0 || blk >= num_blocks) {
        if (v == 0) record_status(status, kStatusInvalid);
        dst[2 * i] = make_uint4(0u, 0u, 0u, 0u);
        dst[2 * i + 1] = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      src = static_cast<int64_t>(blk) * kBlockTokens + t % kBlockTokens;
    } else {
      src = t;  // contiguous cache (one sequence)
    }
    widen16(__ldg(&cache[src * vec_per_row + v]), dst + 2 * i);
  }
}

__global__ void __launch_bounds__(256) kv_widen_fp8_kernel(
    const uint4* __restrict__ k_cache, const uint4* __restrict__ v_cache, uint4* k_out, uint4* v_out,
    int kv_heads, int dq, int dv, const int32_t* __restrict__ table, int32_t num_blocks,
    const __grid_constant__ WidenPlan plan, int* status) {
  widen_rows(k_cache, k_out, kv_heads * dq / 16, plan, table, num_blocks, status);
  widen_rows(v_cache, v_out, kv_heads * dv / 16, plan, table, num_blocks, status);
}

int grid_for(int64_t work_items, int num_sms) {
  const int64_t per_block = 256 * 4;
  int64_t g = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                 const float* k_scale, const float* v_scale, const int32_t* block_table,
                                 int32_t num_blocks, int64_t prefix_len, int64_t chunk_len, int kv_heads,
                                 int dq, int dv, int* status, int num_sms, cudaStream_t stream) {
  SeqPos pos{prefix_len, block_table};
  const int grid = grid_for(chunk_len * kv_heads * (dq + dv) / 16, num_sms);
  kv_append_fp8_kernel<SeqPos><<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), k_scale, v_scale, chunk_len, kv_heads, dq, dv, num_blocks, pos, status);
  return cudaGetLastError();
}

cudaError_t launch_kv_append_fp8_varlen(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                        const float* k_scale, const float* v_scale,
                                        const int32_t* block_table, const VarlenPlan& plan,
                                        int32_t num_blocks, int kv_heads, int dq, int dv, int* status,
                                        int num_sms, cudaStream_t stream) {
  const int64_t tokens = plan.cu_q[plan.batch];
  const int grid = grid_for(tokens * kv_heads * (dq + dv) / 16, num_sms);
  kv_append_fp8_varlen_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), k_scale, v_scale, kv_heads, dq, dv, num_blocks, block_table, plan,
      status);
  return cudaGetLastError();
}

cudaError_t launch_kv_widen_fp8(const void* k_cache, const void* v_cache, uint16_t* k_out, uint16_t* v_out,
                                int kv_heads, int dq, int dv, const int32_t* block_table,
                                int32_t num_blocks, const WidenPlan& plan, int* status, int num_sms,
                                cudaStream_t stream) {
  const int grid = grid_for(plan.base[plan.n] * kv_heads * (dq + dv) / 16, num_sms);
  kv_widen_fp8_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache), reinterpret_cast<uint4*>(k_out),
      reinterpret_cast<uint4*>(v_out), kv_heads, dq, dv, block_table, num_blocks, plan, status);
  return cudaGetLastError();
}

}  // namespace vpp
