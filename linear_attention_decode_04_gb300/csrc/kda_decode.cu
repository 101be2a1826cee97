// kda_decode.cu -- fused single-token KDA decode step for GB300 (sm_103a).
//
// "P1" is the page "[ROCm][Perf] Kimi-K3 Fused kernel for KDA decode" (vLLM
// PR #50654 report).  P1 (功能与动机, 实现拆解 item 1) describes one launch
// that, per (sequence, value head), advances the width-4 causal conv state,
// runs the gated delta rule on a [128,128] fp32 state and applies the gated
// RMSNorm; the equations are the standard KDA definition spelled out in
// include/kda_decode.h.
//
// The step is bound by HBM: 64 KiB of state read and 64 KiB written per
// (sequence, head) (P1 实现拆解 item 1), about 95% of all bytes.  The
// arithmetic is two matvecs and a rank-1 update per state tile, so no tensor
// cores: the kernel streams the tile once, keeps it on chip between the
// reduction and the write, and overlaps everything else with that stream.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "kda_decode.h"

namespace {

constexpr int kDim = 128;              // key = value head dim
constexpr int kWidth = 4;              // conv taps
constexpr int kThreads = 256;          // 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kDim / kWarps;   // 16 key rows per warp
constexpr int kCsU4 = kDim * (kWidth - 1) * 2 / 16;  // 48 uint4 per block slice of conv state
constexpr int kXU4 = kDim * 2 / 16;                  // 16 uint4 per block slice of qkv

struct Params {
  const uint16_t* qkv;
  int64_t qkv_stride;
  const float* conv_w;
  const float* conv_b;
  uint16_t* conv_state;
  float* state;
  const float* g;
  const uint16_t* beta;
  const uint16_t* gate;
  int64_t gate_stride;
  const float* norm_w;
  const int32_t* slot_idx;
  uint16_t* out;
  int64_t out_stride;
  int N, H, num_slots;
  float eps, q_scale;
  int32_t* err;
};

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One CTA per (row n, head h).  Thread (warp w, lane l) owns value columns
// 4l..4l+3 of key rows 16w..16w+15: 64 fp32 of the tile, loaded with
// streaming 128-bit loads before anything else (the whole-state prefetch of
// P1 实现拆解 item 1) and kept in registers until the write.
template <bool kOutNorm, bool kUpdateConv>
__global__ void __launch_bounds__(kThreads, 2) kda_decode_tile_kernel(const Params p) {
  __shared__ __align__(16) uint16_t s_cs[3][kDim * (kWidth - 1)];  // old conv state, q|k|v
  __shared__ __align__(16) uint16_t s_x[3][kDim];                   // this token's q|k|v
  __shared__ __align__(16) float s_q[kDim], s_k[kDim], s_v[kDim], s_alpha[kDim];
  __shared__ __align__(16) float s_red[2][kWarps][kDim];
  __shared__ __align__(16) float s_delta[kDim];
  __shared__ float s_sum[4][4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x / p.H;
  const int h = blockIdx.x - n * p.H;
  const int64_t D = static_cast<int64_t>(p.H) * kDim;
  uint16_t* out_row = p.out + n * p.out_stride + static_cast<int64_t>(h) * kDim;

  // Padding rows (slot <= 0) write zeros and touch no state (P1 实现拆解
  // item 1; kernel excerpt in 关键源码片段).  The slot is uniform over the
  // CTA, so the early return keeps every later barrier paired.
  const int slot = __ldg(p.slot_idx + n);
  if (slot <= 0 || slot >= p.num_slots) {
    if (slot >= p.num_slots && tid == 0 && p.err) atomicOr(p.err, KDA_DEVERR_SLOT_RANGE);
    if (tid < kDim * 2 / 16) reinterpret_cast<uint4*>(out_row)[tid] = make_uint4(0, 0, 0, 0);
    return;
  }

  // 1. Stream the state tile in (evict-first: it is read exactly once).
  float* tile = p.state + (static_cast<int64_t>(slot) * p.H + h) * (kDim * kDim);
  const float4* tile4 = reinterpret_cast<const float4*>(tile);
  float4 a[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) a[r] = __ldcs(tile4 + (warp * kRowsPerWarp + r) * 32 + lane);

  // 2. Conv inputs: the three 768-byte conv-state slices and 256-byte qkv slices.
  if (tid < 3 * kCsU4) {
    const int c = tid / kCsU4, e = tid - c * kCsU4;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.conv_state + (static_cast<int64_t>(slot) * 3 * D + c * D + static_cast<int64_t>(h) * kDim) * (kWidth - 1));
    reinterpret_cast<uint4*>(s_cs[c])[e] = __ldg(src + e);
  } else if (tid < 3 * kCsU4 + 3 * kXU4) {
    const int t = tid - 3 * kCsU4, c = t / kXU4, e = t - c * kXU4;
    const uint4* src = reinterpret_cast<const uint4*>(p.qkv + n * p.qkv_stride + c * D +
                                                      static_cast<int64_t>(h) * kDim);
    reinterpret_cast<uint4*>(s_x[c])[e] = __ldg(src + e);
  }
  __syncthreads();

  // Conv-state advance: each channel's window drops its oldest tap and takes
  // the new input -- a pure move of bf16 bit patterns.
  if (kUpdateConv && tid < 3 * kCsU4) {
    const int c = tid / kCsU4, e = tid - c * kCsU4;
    uint16_t v[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int pos = e * 8 + t, j = pos / 3, k = pos - 3 * j;
      v[t] = (k < kWidth - 2) ? s_cs[c][3 * j + k + 1] : s_x[c][j];
    }
    uint4 w;
    w.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
    w.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
    w.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
    w.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
    uint4* dst = reinterpret_cast<uint4*>(
        p.conv_state + (static_cast<int64_t>(slot) * 3 * D + c * D + static_cast<int64_t>(h) * kDim) * (kWidth - 1));
    dst[e] = w;
  }

  // Conv (4 taps, width-major fp32 weights) + SiLU for the 384 channels, and
  // the per-key-channel decay alpha = exp(g).
  for (int idx = tid; idx < 4 * kDim; idx += kThreads) {
    if (idx < 3 * kDim) {
      const int c = idx >> 7, j = idx & (kDim - 1);
      const int64_t ch = c * D + static_cast<int64_t>(h) * kDim + j;
      const float* w = p.conv_w + c * kWidth * D + static_cast<int64_t>(h) * kDim + j;
      float y = p.conv_b ? __ldg(p.conv_b + ch) : 0.0f;
      y = fmaf(__ldg(w + 0 * D), bf16_to_f32(s_cs[c][3 * j + 0]), y);
      y = fmaf(__ldg(w + 1 * D), bf16_to_f32(s_cs[c][3 * j + 1]), y);
      y = fmaf(__ldg(w + 2 * D), bf16_to_f32(s_cs[c][3 * j + 2]), y);
      y = fmaf(__ldg(w + 3 * D), bf16_to_f32(s_x[c][j]), y);
      const float act = y / (1.0f + expf(-y));
      (c == 0 ? s_q : c == 1 ? s_k : s_v)[j] = act;
    } else {
      const int i = idx - 3 * kDim;
      s_alpha[i] = expf(__ldg(p.g + (static_cast<int64_t>(n) * p.H + h) * kDim + i));
    }
  }
  __syncthreads();

  // |q|^2, |k|^2 and q.k in one pass (three block sums).
  if (tid < kDim) {
    const float q = s_q[tid], k = s_k[tid];
    const float sq = warp_sum(q * q), sk = warp_sum(k * k), sqk = warp_sum(q * k);
    if (lane == 0) {
      s_sum[warp][0] = sq;
      s_sum[warp][1] = sk;
      s_sum[warp][2] = sqk;
    }
  }
  __syncthreads();
  const float ssq = (s_sum[0][0] + s_sum[1][0]) + (s_sum[2][0] + s_sum[3][0]);
  const float ssk = (s_sum[0][1] + s_sum[1][1]) + (s_sum[2][1] + s_sum[3][1]);
  const float sqk = (s_sum[0][2] + s_sum[1][2]) + (s_sum[2][2] + s_sum[3][2]);
  const float scale = (p.q_scale != 0.0f) ? p.q_scale : 0.088388347648318440550f;  // 1/sqrt(128)
  const float rq = scale / sqrtf(ssq + 1e-6f);
  const float rk = 1.0f / sqrtf(ssk + 1e-6f);
  const float qk = sqk * rq * rk;  // q^ . k^

  // 3. Decay the tile in registers and form the partial column sums
  //    u = (Diag(alpha) S)^T k^ and w = (Diag(alpha) S)^T q^ over this warp's rows.
  float4 u = make_float4(0.f, 0.f, 0.f, 0.f), w = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = warp * kRowsPerWarp + r;
    const float al = s_alpha[i], kh = s_k[i] * rk, qh = s_q[i] * rq;
    a[r].x *= al; a[r].y *= al; a[r].z *= al; a[r].w *= al;
    u.x = fmaf(kh, a[r].x, u.x); u.y = fmaf(kh, a[r].y, u.y);
    u.z = fmaf(kh, a[r].z, u.z); u.w = fmaf(kh, a[r].w, u.w);
    w.x = fmaf(qh, a[r].x, w.x); w.y = fmaf(qh, a[r].y, w.y);
    w.z = fmaf(qh, a[r].z, w.z); w.w = fmaf(qh, a[r].w, w.w);
  }
  reinterpret_cast<float4*>(s_red[0][warp])[lane] = u;
  reinterpret_cast<float4*>(s_red[1][warp])[lane] = w;
  __syncthreads();

  // 4. delta_j = beta (v_j - u_j); the readout of the updated state
  //    o = S'^T q^ = w + (q^ . k^) delta needs no second pass over S'.
  float o = 0.0f;
  if (tid < kDim) {
    float uj = 0.0f, wj = 0.0f;
#pragma unroll
    for (int r = 0; r < kWarps; ++r) {
      uj += s_red[0][r][tid];
      wj += s_red[1][r][tid];
    }
    const float beta = bf16_to_f32(__ldg(p.beta + static_cast<int64_t>(n) * p.H + h));
    const float dj = beta * (s_v[tid] - uj);
    s_delta[tid] = dj;
    o = fmaf(qk, dj, wj);
    if (kOutNorm) {
      const float ss = warp_sum(o * o);
      if (lane == 0) s_sum[warp][3] = ss;
    }
  }
  __syncthreads();

  // 5. S' = Diag(alpha) S + k^ delta^T, streamed out (evict-first).
  const float4 d = reinterpret_cast<const float4*>(s_delta)[lane];
  float4* tile4w = reinterpret_cast<float4*>(tile);
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = warp * kRowsPerWarp + r;
    const float kh = s_k[i] * rk;
    a[r].x = fmaf(kh, d.x, a[r].x); a[r].y = fmaf(kh, d.y, a[r].y);
    a[r].z = fmaf(kh, d.z, a[r].z); a[r].w = fmaf(kh, d.w, a[r].w);
    __stcs(tile4w + i * 32 + lane, a[r]);
  }

  // 6. Gated RMSNorm epilogue (or the raw readout) to bf16.
  if (tid < kDim) {
    float y = o;
    if (kOutNorm) {
      const float ss = (s_sum[0][3] + s_sum[1][3]) + (s_sum[2][3] + s_sum[3][3]);
      const float rr = 1.0f / sqrtf(ss * (1.0f / kDim) + p.eps);
      const float gt = bf16_to_f32(__ldg(p.gate + n * p.gate_stride + static_cast<int64_t>(h) * kDim + tid));
      y = o * rr * __ldg(p.norm_w + tid) * (1.0f / (1.0f + expf(-gt)));
    }
    out_row[tid] = f32_to_bf16(y);
  }
}

thread_local char g_last_error[512];

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <bool kOutNorm, bool kUpdateConv>
cudaError_t launch(const Params& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(p.N) * static_cast<unsigned>(p.H);
  kda_decode_tile_kernel<kOutNorm, kUpdateConv><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

extern "C" int kda_abi_version(void) { return KDA_DECODE_ABI_VERSION; }

extern "C" const char* kda_last_error(void) { return g_last_error; }

extern "C" const char* kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULLPTR: return "a required pointer is NULL";
    case KDA_ERR_SHAPE: return "unsupported or inconsistent shape";
    case KDA_ERR_ALIGN: return "pointer or row stride breaks the 16-byte alignment rule";
    case KDA_ERR_FLAGS: return "unknown flag bits";
    case KDA_ERR_LAUNCH: return "CUDA launch failed";
    case KDA_ERR_ABI: return "KdaDecodeArgs.struct_size does not match the library";
    default: return "unknown status";
  }
}

extern "C" int kda_decode(const KdaDecodeArgs* a, void* stream) {
  g_last_error[0] = '\0';
  // Validation touches no CUDA API and no device memory.
  if (!a) return fail(KDA_ERR_NULLPTR, "args is NULL");
  if (a->struct_size != sizeof(KdaDecodeArgs))
    return fail(KDA_ERR_ABI, "struct_size %u, library expects %zu", a->struct_size, sizeof(KdaDecodeArgs));
  if (a->head_dim != KDA_HEAD_DIM || a->conv_width != KDA_CONV_WIDTH)
    return fail(KDA_ERR_SHAPE, "head_dim %d / conv_width %d (need 128 / 4)", a->head_dim, a->conv_width);
  if (a->N < 0 || a->H < 1 || a->num_slots < 1)
    return fail(KDA_ERR_SHAPE, "N=%d H=%d num_slots=%d", a->N, a->H, a->num_slots);
  if (a->flags & ~(KDA_OUT_NORM | KDA_UPDATE_CONV_STATE)) return fail(KDA_ERR_FLAGS, "flags 0x%x", a->flags);
  if (a->N == 0) return KDA_OK;
  const bool norm = (a->flags & KDA_OUT_NORM) != 0;
  if (!a->qkv || !a->conv_weight || !a->conv_state || !a->state || !a->g || !a->beta || !a->slot_idx ||
      !a->out)
    return fail(KDA_ERR_NULLPTR, "a required tensor pointer is NULL");
  if (norm && (!a->gate || !a->norm_weight))
    return fail(KDA_ERR_NULLPTR, "KDA_OUT_NORM needs gate and norm_weight");
  const int64_t D = static_cast<int64_t>(a->H) * KDA_HEAD_DIM;
  if (static_cast<int64_t>(a->N) * a->H > 0x7fffffffLL)
    return fail(KDA_ERR_SHAPE, "N*H = %lld exceeds the grid limit", static_cast<long long>(a->N) * a->H);
  if (a->qkv_row_stride < 3 * D || a->out_row_stride < D || (norm && a->gate_row_stride < D))
    return fail(KDA_ERR_SHAPE, "row stride below the row width");
  if ((a->qkv_row_stride & 7) || (a->out_row_stride & 7) || (norm && (a->gate_row_stride & 7)))
    return fail(KDA_ERR_ALIGN, "row strides must be multiples of 8 elements");
  if (!aligned16(a->qkv) || !aligned16(a->conv_weight) || !aligned16(a->conv_state) ||
      !aligned16(a->state) || !aligned16(a->g) || !aligned16(a->out) ||
      (a->conv_bias && !aligned16(a->conv_bias)) ||
      (norm && (!aligned16(a->gate) || !aligned16(a->norm_weight))))
    return fail(KDA_ERR_ALIGN, "tensor pointers must be 16-byte aligned");

  Params p;
  p.qkv = a->qkv;
  p.qkv_stride = a->qkv_row_stride;
  p.conv_w = a->conv_weight;
  p.conv_b = a->conv_bias;
  p.conv_state = a->conv_state;
  p.state = a->state;
  p.g = a->g;
  p.beta = a->beta;
  p.gate = norm ? a->gate : nullptr;
  p.gate_stride = norm ? a->gate_row_stride : 0;
  p.norm_w = norm ? a->norm_weight : nullptr;
  p.slot_idx = a->slot_idx;
  p.out = a->out;
  p.out_stride = a->out_row_stride;
  p.N = a->N;
  p.H = a->H;
  p.num_slots = a->num_slots;
  p.eps = a->eps;
  p.q_scale = a->q_scale;
  p.err = a->err_flag;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool conv = (a->flags & KDA_UPDATE_CONV_STATE) != 0;
  cudaError_t e = norm ? (conv ? launch<true, true>(p, s) : launch<true, false>(p, s))
                       : (conv ? launch<false, true>(p, s) : launch<false, false>(p, s));
  if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "%s", cudaGetErrorString(e));
  return KDA_OK;
}
