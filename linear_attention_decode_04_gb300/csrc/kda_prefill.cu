// kda_prefill.cu -- chunked KDA prefill over a varlen batch for GB300
// (sm_103a): device code and C ABI.
//
// "P2" is the page "[ROCm][Perf] Kimi-K3 Remove prefill pipeline stall in
// chunk KDA" (vLLM PR #51862 report): prefill runs the KDA layer over whole
// sequences of a varlen batch with a chunked kernel (实现拆解 items 2-3).  P2
// prints none of that kernel's arithmetic; what it computes is the decode
// recurrence of include/kda_decode.h applied token by token, and the chunked
// evaluation below is exact up to rounding (derivation in the comments).
//
// Chunk form.  Within a chunk of L tokens t = 0..L-1 of one (sequence, head),
// with S0 the state before the chunk, G_t = g_0 + ... + g_t (per key channel,
// cumulative log decay), k^, q^ the normalised keys and queries, v~ the
// values and beta_t the write strengths, the recurrence
//     S_t = Diag(exp g_t) S_{t-1} + k^_t delta_t^T,
//     delta_t = beta_t (v~_t - (Diag(exp g_t) S_{t-1})^T k^_t),   o_t = S_t^T q^_t
// unrolls to S_t = Diag(exp G_t) S0 + sum_{s<=t} Diag(exp(G_t - G_s)) k^_s delta_s^T, so
//     (I + Diag(beta) P) Delta = Diag(beta) (V~ - K_G S0),   P_ts = sum_i k^_ti k^_si exp(G_ti - G_si)  (s < t)
//     O = Q_G S0 + R Delta,                                 R_ts = sum_i q^_ti k^_si exp(G_ti - G_si)  (s <= t)
//     S_L = Diag(exp G_{L-1}) S0 + K_E^T Delta
// with K_G = exp(G) . K^, Q_G = exp(G) . Q^ and K_E = exp(G_{L-1} - G) . K^
// (row-wise).  The output is evaluated in the decode step's cancellation-safe
// form instead: o_t = A_t^T q'_t + c_t v~_t, A_t the state before token t's
// update, q'_t = r_q ((q~_t - k~_t) + m_t k~_t) = q^_t - beta_t (q^_t.k^_t) k^_t
// and c_t = beta_t (q^_t.k^_t); that is, q^ replaced by q' in Q_G and R, R
// strictly lower (s < t), and E = Diag(c) V~ added to O.  When q~ = k~ the
// plain O cancels two terms of the size of the state down to |v~|; q' is then
// r_q m k~ (tiny) and no such cancellation occurs.  The triangular system is solved once for both right-hand
// sides, X = [U | W] with (I + Diag(beta) P) X = Diag(beta) [V~ | K_G], so
// Delta = U - W S0.  P and R are contractions over the key channels once the
// decay factor is split around a reference token m of the chunk:
// exp(G_t - G_s) = exp(G_t - G_m) exp(G_m - G_s); when a factor could leave
// the fp32 range the chunk takes them element by element instead.
//
// Tensor cores.  The contractions with the state (W S0, Q_G S0, K_E^T Delta)
// and R Delta run in the scan kernel as tcgen05.mma (kind::tf32, M = 128),
// with the state held in tensor memory for the whole sequence; P and R
// (between the tokens of a chunk) run in the chunk kernel as warp-level
// m16n8k8 tf32 MMAs.  Every operand is split into a tf32 high part and a
// tf32 remainder and three products are accumulated in fp32, which keeps
// close to fp32 accuracy.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "kda_chunk_metadata.h"
#include "kda_internal.h"
#include "kda_prefill.h"

namespace {

constexpr int kD = 128;           // head dim (key = value)
constexpr int kWidth = 4;         // conv taps
constexpr int kHist = kWidth - 1; // older taps carried between chunks
constexpr int kL = KDA_PREFILL_CHUNK;  // 32 tokens per chunk
constexpr int kWarps = 8;                        // scan kernel
constexpr int kThreads = kWarps * 32;
constexpr int kChunkWarps = 12;                  // chunk kernel: one thread per q|k|v channel
constexpr int kChunkThreads = kChunkWarps * 32;
constexpr int kCh = 3 * kD;       // q | k | v channels of one head
constexpr int kSA = 136;          // row stride (floats) of [token][128] operands
constexpr int kSP = 36;           // row stride (floats) of P (rows read as float4)
constexpr int kRef = 15;          // reference token of the split decay factors
constexpr float kMaxExponent = 80.0f;  // |G_t - G_m| above this: element-wise path

struct PrefillParams {
  const int32_t* cu;
  const int32_t* chunk_idx;   // [num_chunks][2] (sequence, chunk)
  const int64_t* chunk_off;   // [B + 1]
  int64_t num_chunks;
  float* ws;                  // per (chunk row, head) one record of kRec floats
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
  int64_t T;
  int B, H, num_slots;
  float eps, q_scale;
  int32_t* err;
  int conv_sd;                // conv state stored tap-first [slots][3][C]
  int fused_gate;             // g and beta hold raw logits (activated on load)
  const float* A_log;
  const float* dt_bias;
  float lower_bound;
  const int32_t* seq_order;   // [B] or NULL: the scan's sequence order
};

// Workspace image of one (chunk, head), written by the chunk kernel and
// copied verbatim (one bulk copy) into the scan kernel's shared memory.  The
// operands of the scan's tensor-core products are stored in the canonical
// K-major layout without swizzle, in the variant whose 8-row groups are
// adjacent: an N x K fp32 operand is tiled into core matrices of 8 rows x 16
// bytes (4 values of k), element (n, k) at (k / 4) * N * 4 + n * 4 + k % 4
// floats; the 8-row groups are 128 bytes apart (SBO) and the core matrices
// adjacent in K are N * 16 bytes apart (LBO).  Each product's B operand is
// one such block: [Q_G; W] (N = 64, K = 128 keys) and [K_E^T; R]
// (N = 160, K = 32 tokens).
__host__ __device__ constexpr int kpos(int n, int k, int N) { return (k >> 2) * (N * 4) + n * 4 + (k & 3); }
constexpr int kNB1 = 2 * kL;                  // [Q_G; W]: Q_G rows 0..31, W rows 32..63
constexpr int kNB2 = kD + kL;                 // [K_E^T; R]: K_E^T rows 0..127, R rows 128..159
constexpr int kOffB1 = 0;                     // [Q_G; W]   64 x 128
constexpr int kOffB2 = kOffB1 + kNB1 * kD;    // [K_E^T; R] 160 x 32 (R zero above its diagonal)
constexpr int kOffU = kOffB2 + kNB2 * kL;     // U     [32 tokens][128 values], row-major
constexpr int kOffC = kOffU + kL * kD;        // gamma = exp(G_{L-1}) [128]
constexpr int kImg = kOffC + kD;              // 17,536 floats = 70,144 bytes (copied in one piece)
constexpr int kOffE = kImg;                   // E = Diag(c) V~ [32 tokens][128 values], row-major
constexpr int kRec = kOffE + kL * kD;         // one workspace record: 21,632 floats = 86,528 bytes
constexpr int kSplit = kOffU;                 // the operands the scan splits into tf32 words
static_assert((kImg * 4) % 16 == 0 && (kRec * 4) % 16 == 0, "records must be whole 16-byte pieces");

// Chunk kernel shared memory (about 108 KB: two CTAs per SM).
struct __align__(16) ChunkSmem {
  union {
    uint16_t raw[kHist + kL][kCh];  // conv window: 3 older rows, then the chunk's inputs
    struct {
      float ek[kL][kSA];            // exp(G - G_m) k^
      float fk[kL][kSA];            // exp(G_m - G) k^
    } f;
  };
  float q[kL][kSA];                 // q^
  float k[kL][kSA];                 // k^
  float v[kL][kSA];                 // v~
  float G[kL][kSA];                 // cumulative log decay
  float P[kL][kSP];                 // P (strictly lower)
  float beta[kL];
  float c[kL];                      // beta_t (q^_t . k^_t), the weight of v~_t in o_t
  float egm[kD];                    // exp(G_m) per key channel (0 when G_m < -kMaxExponent)
  float cl[kD];                     // exp(G_{L-1} - G_m) per key channel
  int slow;                         // this chunk takes the element-wise P / R path
};

// Scan kernel shared memory (about 205 KB): two images (double buffer), the
// tf32 remainders of the image's tensor-core operands, the chunk's output
// rows (E by bulk copy, then D_O added), the MMA-completion and
// copy-completion barriers and the tensor-memory base address.
struct __align__(128) ScanSmem {
  float img[2][kImg];
  float lo[kSplit];
  float o[kL][kD];             // the chunk's output rows: E = Diag(c) V~ (bulk copy), then + D_O
  unsigned long long bar[2];   // the two MMA batches of a chunk
  unsigned long long full[2];  // image buffer 0 / 1 landed
  unsigned long long efull;    // E landed in o
  uint32_t tmem;
};

static_assert(sizeof(ScanSmem) <= 227 * 1024, "scan kernel shared memory above the 227 KB a CTA may use");
static_assert(2 * (sizeof(ChunkSmem) + 1024) <= 228 * 1024, "two chunk-kernel CTAs must fit one SM");

// Tensor-memory columns of the scan kernel (512 allocated; lane = value row):
// the fp32 state S^T, the chunk's output and S^T W^T accumulators, the
// state's tf32 high and low words (the A operand of the products with the
// state) and Delta^T's high and low words (the A operand of the products
// with Delta).  [S^T | O] and [O | S^T W^T] are each contiguous, so each of
// the two product batches is one MMA per step.
constexpr uint32_t kTS = 0, kTO = 128, kTD = 160, kTSH = 192, kTSL = 320, kTDH = 448, kTDL = 480;
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// tf32 keeps the top 19 bits of an fp32 word (sign, exponent, 10 mantissa
// bits).  An fp32 value x is split as hi = x with its low 13 bits cleared and
// lo = x - hi (exact in fp32), lo again cut to 19 bits: hi + lo carries 21
// significant bits, and the split costs integer and add instructions only.
__device__ __forceinline__ uint32_t tf32_hi(float x) { return __float_as_uint(x) & 0xFFFFE000u; }
__device__ __forceinline__ uint32_t tf32_lo(float x, uint32_t hi) {
  return __float_as_uint(x - __uint_as_float(hi)) & 0xFFFFE000u;
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// An A operand (16 x 8 tile) in registers, split into tf32 high and low parts.
struct FragA {
  uint32_t hi[4], lo[4];
};

__device__ __forceinline__ FragA make_a(float a0, float a1, float a2, float a3) {
  FragA f;
  const float a[4] = {a0, a1, a2, a3};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f.hi[e] = tf32_hi(a[e]);
    f.lo[e] = tf32_lo(a[e], f.hi[e]);
  }
  return f;
}

// c += A * B with B's two elements split as well: lo*hi + hi*lo + hi*hi.
__device__ __forceinline__ void mma3(float (&c)[4], const FragA& a, float b0, float b1) {
  const uint32_t h0 = tf32_hi(b0), h1 = tf32_hi(b1);
  const uint32_t l0 = tf32_lo(b0, h0), l1 = tf32_lo(b1, h1);
  mma_tf32(c, a.lo, h0, h1);
  mma_tf32(c, a.hi, l0, l1);
  mma_tf32(c, a.hi, h0, h1);
}

__device__ __forceinline__ void flag(const PrefillParams& p, int bits) {
  if (p.err) atomicOr(p.err, bits);
}

// One bulk copy (TMA engine) global -> shared, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// One asynchronous 16-byte copy global -> shared (cache-global form); with
// bytes = 0 nothing is read and the 16 bytes are zero-filled.  Completed by
// cp.async.wait_all.
__device__ __forceinline__ void cp16(void* dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(bytes)
               : "memory");
}

// ===================================================================== chunk
// One CTA per (chunk row c, head h), chunk row = (sequence b, chunk j) from
// the chunk metadata.  Everything that does not depend on the state entering
// the chunk: conv, norms, cumulative decays, P and R, the triangular solve
// for U and W, and the decayed Q_G and K_E.  Results go to the workspace
// image of (c, h).
__global__ void __launch_bounds__(kChunkThreads, 2) kda_prefill_chunk_kernel(const PrefillParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChunkSmem& S = *reinterpret_cast<ChunkSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, tq = lane & 3;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y;
  const int64_t D = static_cast<int64_t>(p.H) * kD;

  const int b = p.chunk_idx[2 * c], j = p.chunk_idx[2 * c + 1];
  if (b < 0 || b >= p.B || j < 0) {
    if (tid == 0 && h == 0) flag(p, KDA_DEVERR_SEQLENS);
    return;
  }
  const int64_t r0 = p.cu[b], r1 = p.cu[b + 1];
  const int64_t t0 = r0 + static_cast<int64_t>(kL) * j;
  if (r0 < 0 || r1 < r0 || r1 > p.T || t0 >= r1) {
    if (tid == 0 && h == 0) flag(p, KDA_DEVERR_SEQLENS);
    return;
  }
  const int slot = p.slot_idx[b];
  if (slot <= 0 || slot >= p.num_slots) return;  // the scan kernel zeroes and flags
  const int L = static_cast<int>(r1 - t0 < kL ? r1 - t0 : kL);
  float* ws = p.ws + (c * p.H + h) * static_cast<int64_t>(kRec);
  auto ch_global = [&](int ch) { return static_cast<int64_t>(ch >> 7) * D + static_cast<int64_t>(h) * kD + (ch & 127); };

  // ---- 1. inputs: the three older taps (conv state for the first chunk,
  // else the sequence's preceding tokens), the chunk's rows (zero past L),
  // g, beta.  Rows and g arrive by asynchronous 16-byte copies, all of a
  // thread's copies in flight at once.
  if (j == 0) {
    // tap r of channel c at c * 3 + r (dim-first) or r * C + c (tap-first)
    const uint16_t* cs = p.conv_state + static_cast<int64_t>(slot) * 3 * D * kHist;
    const int64_t sc = p.conv_sd ? 1 : kHist, sr = p.conv_sd ? 3 * D : 1;
    for (int ch = tid; ch < kCh; ch += kChunkThreads)
#pragma unroll
      for (int r = 0; r < kHist; ++r) S.raw[r][ch] = cs[ch_global(ch) * sc + r * sr];
  } else {
    for (int e = tid; e < kHist * 48; e += kChunkThreads) {
      const int r = e / 48, q = e - r * 48, seg = q >> 4, u = q & 15;
      cp16(&S.raw[r][seg * kD + 8 * u],
           p.qkv + (t0 - kHist + r) * p.qkv_stride + seg * D + static_cast<int64_t>(h) * kD + 8 * u, 16);
    }
  }
  for (int e = tid; e < kL * 48; e += kChunkThreads) {
    const int t = e / 48, q = e - t * 48, seg = q >> 4, u = q & 15;
    const int tr = t < L ? t : L - 1;  // rows past L: zero-filled (the source row is only an address)
    cp16(&S.raw[kHist + t][seg * kD + 8 * u],
         p.qkv + (t0 + tr) * p.qkv_stride + seg * D + static_cast<int64_t>(h) * kD + 8 * u, t < L ? 16 : 0);
  }
  if (!p.fused_gate) {
    for (int e = tid; e < kL * 32; e += kChunkThreads) {
      const int t = e >> 5, u = e & 31, tr = t < L ? t : L - 1;
      cp16(&S.G[t][4 * u], p.g + ((t0 + tr) * p.H + h) * kD + 4 * u, t < L ? 16 : 0);
    }
  } else {
    // the gate activation on the raw logits (the page's safe-gate variant;
    // standard KDA form): z = raw + dt_bias, g = lb * sigmoid(e^A_log z) for
    // a lower bound lb < 0, else g = -e^A_log softplus(z)
    const float a = expf(__ldg(p.A_log + h));
    for (int e = tid; e < kL * 32; e += kChunkThreads) {
      const int t = e >> 5, u = e & 31;
      float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < L) {
        val = __ldg(reinterpret_cast<const float4*>(p.g + ((t0 + t) * p.H + h) * kD) + u);
        float* vv = &val.x;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float z = vv[c] + (p.dt_bias ? __ldg(p.dt_bias + static_cast<int64_t>(h) * kD + 4 * u + c) : 0.0f);
          if (p.lower_bound < 0.0f) {
            vv[c] = p.lower_bound / (1.0f + expf(-a * z));
          } else {
            const float sp = (z > 0.0f) ? z + log1pf(expf(-z)) : log1pf(expf(z));
            vv[c] = -a * sp;
          }
        }
      }
      reinterpret_cast<float4*>(S.G[t])[u] = val;
    }
  }
  if (tid < kL) {
    float bt = 0.0f;
    if (tid < L) {
      bt = bf16f(p.beta[(t0 + tid) * p.H + h]);
      if (p.fused_gate) bt = 1.0f / (1.0f + expf(-bt));
    }
    S.beta[tid] = bt;
  }
  if (tid == 0) S.slow = 0;
  // this thread's conv taps and bias, loaded while the copies land
  float wa[kWidth], ba = 0.0f;
  {
    const int c = tid >> 7, j = tid & (kD - 1);
#pragma unroll
    for (int t = 0; t < kWidth; ++t)
      wa[t] = __ldg(p.conv_w + (c * kWidth + t) * D + static_cast<int64_t>(h) * kD + j);
    if (p.conv_b) ba = __ldg(p.conv_b + ch_global(tid));
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // ---- 2. conv + SiLU over the window (outputs past L are zero); thread
  // tid convolves channel tid of the head's q | k | v channels over all
  // tokens
  {
    const int c = tid >> 7, j = tid & (kD - 1);
    float x0 = bf16f(S.raw[0][tid]), x1 = bf16f(S.raw[1][tid]), x2 = bf16f(S.raw[2][tid]);
    float* dst = c == 0 ? &S.q[0][j] : c == 1 ? &S.k[0][j] : &S.v[0][j];
#pragma unroll
    for (int t = 0; t < kL; ++t) {
      const float x3 = bf16f(S.raw[kHist + t][tid]);
      float y = ba;
      y = fmaf(wa[0], x0, y);
      y = fmaf(wa[1], x1, y);
      y = fmaf(wa[2], x2, y);
      y = fmaf(wa[3], x3, y);
      dst[t * kSA] = t < L ? __fdividef(y, 1.0f + __expf(-y)) : 0.0f;
      x0 = x1; x1 = x2; x2 = x3;
    }
  }
  __syncthreads();

  // ---- 3. L2 norms (warp w: tokens w, w + 12, w + 24); cumulative decay
  const float qs = (p.q_scale != 0.0f) ? p.q_scale : 0.088388347648318440550f;  // 1/sqrt(128)
  // In place of q^_t the chunk carries q'_t = r_q ((q~_t - k~_t) + m_t k~_t),
  // m_t = (|k~_t|^2 + 1e-6 - beta_t q~_t.k~_t) r_k^2, and c_t = beta_t
  // (q^_t . k^_t): o_t = A_t^T q'_t + c_t v~_t with A_t the state before token
  // t's update (the decode step's cancellation-safe readout).  The three
  // sums run in one order, so q~.k~ equals |k~|^2 bit for bit when q~ equals
  // k~, and then q' = r_q m k~ is tiny: nothing of the size of the state
  // cancels in the output.
  for (int t = warp; t < kL; t += kChunkWarps) {
    const float4 qv = reinterpret_cast<float4*>(S.q[t])[lane];
    const float4 kv = reinterpret_cast<float4*>(S.k[t])[lane];
    const float sq = warp_sum(fmaf(qv.x, qv.x, fmaf(qv.y, qv.y, fmaf(qv.z, qv.z, qv.w * qv.w))));
    const float sk = warp_sum(fmaf(kv.x, kv.x, fmaf(kv.y, kv.y, fmaf(kv.z, kv.z, kv.w * kv.w))));
    const float sqk = warp_sum(fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, fmaf(qv.z, kv.z, qv.w * kv.w))));
    const float rq = qs * rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
    const float bt = S.beta[t];
    const float m = (fmaf(-bt, sqk, sk) + 1e-6f) * (rk * rk);
    const float4 qp = make_float4(rq * fmaf(m, kv.x, qv.x - kv.x), rq * fmaf(m, kv.y, qv.y - kv.y),
                                  rq * fmaf(m, kv.z, qv.z - kv.z), rq * fmaf(m, kv.w, qv.w - kv.w));
    reinterpret_cast<float4*>(S.q[t])[lane] = qp;
    reinterpret_cast<float4*>(S.k[t])[lane] = make_float4(kv.x * rk, kv.y * rk, kv.z * rk, kv.w * rk);
    if (lane == 0) S.c[t] = bt * sqk * rq * rk;
  }
  if (tid < kD) {
    float acc = 0.0f;
#pragma unroll 8
    for (int t = 0; t < kL; ++t) {
      acc += S.G[t][tid];
      S.G[t][tid] = acc;
    }
    // Whether the split factors exp(+-(G_t - G_m)) stay in range for this
    // channel (else the whole chunk takes the element-wise path), and the
    // per-channel constants that turn them into exp(G_t) and
    // exp(G_{L-1} - G_t).
    const float gm = S.G[kRef][tid];
    float dmax = 0.0f;
#pragma unroll 8
    for (int t = 0; t < kL; ++t) dmax = fmaxf(dmax, fabsf(S.G[t][tid] - gm));
    if (dmax > kMaxExponent) S.slow = 1;
    S.egm[tid] = gm > -kMaxExponent ? expf(gm) : 0.0f;
    S.cl[tid] = expf(S.G[kL - 1][tid] - gm);
  }
  __syncthreads();

  // ---- 4. split decay factors around the reference token (shared memory):
  // ek = exp(G - G_m) k^, fk = exp(G_m - G) k^ and, in place of q^, R's A
  // operand exp(G - G_m) q^; Q_G = exp(G) q^ = exp(G_m) exp(G - G_m) q^ and
  // gamma to the image; R's image cleared (its lower triangle is written
  // next); P cleared.  A chunk on the element-wise path keeps q^ and needs
  // only Q_G here.  Piece (t, keys 4 kg .. 4 kg + 3); consecutive threads
  // take consecutive t, so the image stores of Q_G are coalesced 16-byte
  // pieces.
  const bool slow = S.slow != 0;
  // E = Diag(c) V~ to the record (its own region, row-major)
  for (int e = tid; e < kL * kD / 4; e += kChunkThreads) {
    const int t = e >> 5, j4 = e & 31;
    const float ct = S.c[t];
    const float4 v4 = reinterpret_cast<const float4*>(S.v[t])[j4];
    reinterpret_cast<float4*>(ws + kOffE + t * kD)[j4] = make_float4(ct * v4.x, ct * v4.y, ct * v4.z, ct * v4.w);
  }
  for (int e = tid; e < kL * kD / 4; e += kChunkThreads) {
    const int t = e & (kL - 1), i0 = 4 * (e >> 5);
    const float4 G4 = *reinterpret_cast<const float4*>(&S.G[t][i0]);
    const float4 q4 = *reinterpret_cast<const float4*>(&S.q[t][i0]);
    const float gt[4] = {G4.x, G4.y, G4.z, G4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
    float qg[4];
    if (!slow) {
      const float4 Gm = *reinterpret_cast<const float4*>(&S.G[kRef][i0]);
      const float4 k4 = *reinterpret_cast<const float4*>(&S.k[t][i0]);
      const float4 eg4 = *reinterpret_cast<const float4*>(&S.egm[i0]);
      const float d[4] = {G4.x - Gm.x, G4.y - Gm.y, G4.z - Gm.z, G4.w - Gm.w};
      const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, egm[4] = {eg4.x, eg4.y, eg4.z, eg4.w};
      float ek[4], fk[4], eq[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float ed = expf(d[c]), rd = expf(-d[c]);
        ek[c] = ed * kv[c];
        fk[c] = rd * kv[c];
        eq[c] = ed * qv[c];
        qg[c] = egm[c] > 0.0f ? egm[c] * eq[c] : expf(gt[c]) * qv[c];
      }
      *reinterpret_cast<float4*>(&S.f.ek[t][i0]) = make_float4(ek[0], ek[1], ek[2], ek[3]);
      *reinterpret_cast<float4*>(&S.f.fk[t][i0]) = make_float4(fk[0], fk[1], fk[2], fk[3]);
      *reinterpret_cast<float4*>(&S.q[t][i0]) = make_float4(eq[0], eq[1], eq[2], eq[3]);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) qg[c] = expf(gt[c]) * qv[c];
    }
    *reinterpret_cast<float4*>(ws + kOffB1 + kpos(t, i0, kNB1)) = make_float4(qg[0], qg[1], qg[2], qg[3]);
  }
  if (tid < kD) ws[kOffC + tid] = expf(S.G[kL - 1][tid]);
  for (int e = tid; e < kL * kL; e += kChunkThreads) ws[kOffB2 + kpos(kD + (e >> 5), e & (kL - 1), kNB2)] = 0.0f;
  for (int e = tid; e < kL * kSP; e += kChunkThreads) (&S.P[0][0])[e] = 0.0f;
  __syncthreads();

  // ---- 5. P (strictly lower, shared memory) and R (lower, image) over the
  // key channels
  if (!slow) {
    // one 16 x 8 output tile y of P (mat 0) or R (mat 1) over all keys: the
    // tiles of the lower triangle, (rows 0-15, columns 0-15) and (rows 16-31,
    // columns 0-31); warps 0-5 take the six R tiles, warps 6-11 the six P
    // tiles
    auto tile = [&](const int mat, const int y) {
      const int mm = y < 2 ? 0 : 1, nn = y < 2 ? y : y - 2;
      const int ta = 16 * mm + g8;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int kk = 0; kk < kD / 8; ++kk) {
        const int i0 = 8 * kk + 2 * tq;
        float2 a02, a13;
        // A operand: exp(G - G_m) k^ (P) or exp(G - G_m) q^ (R), both formed above
        const float* arows = mat == 0 ? &S.f.ek[0][0] : &S.q[0][0];
        a02 = *reinterpret_cast<const float2*>(arows + ta * kSA + i0);
        a13 = *reinterpret_cast<const float2*>(arows + (ta + 8) * kSA + i0);
        const float2 bb = *reinterpret_cast<const float2*>(&S.f.fk[8 * nn + g8][i0]);
        mma3(acc, make_a(a02.x, a13.x, a02.y, a13.y), bb.x, bb.y);
      }
      const int s = 8 * nn + 2 * tq;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int te = ta + (e >> 1) * 8, se = s + (e & 1);
        if (mat == 0) {
          if (te > se) S.P[te][se] = acc[e];
        } else {
          if (te > se) ws[kOffB2 + kpos(kD + te, se, kNB2)] = acc[e];
        }
      }
    };
    if (warp < 6)
      tile(1, warp);
    else
      tile(0, warp - 6);
  } else {
    // element-wise: pairs (t, s), s <= t
    for (int e = tid; e < kL * (kL + 1) / 2; e += kChunkThreads) {
      int t = static_cast<int>((sqrtf(8.0f * e + 1.0f) - 1.0f) * 0.5f);
      while ((t + 1) * (t + 2) / 2 <= e) ++t;
      while (t * (t + 1) / 2 > e) --t;
      const int s = e - t * (t + 1) / 2;
      float pk = 0.0f, pq = 0.0f;
      for (int i = 0; i < kD; ++i) {
        const float fct = expf(S.G[t][i] - S.G[s][i]) * S.k[s][i];
        pk = fmaf(S.k[t][i], fct, pk);
        pq = fmaf(S.q[t][i], fct, pq);
      }
      if (t > s) {
        S.P[t][s] = pk;
        ws[kOffB2 + kpos(kD + t, s, kNB2)] = pq;
      }
    }
  }
  __syncthreads();

  // ---- 6. triangular solve (threads 0-255: one column of [U | W] each),
  // left-looking: x_t = beta_t (y_t - sum_{s<t} P_ts x_s), y = v~ (U) or
  // exp(G) k^ (W), W staged in the (now free) factor buffer; meanwhile
  // threads 256-383 write row i of K_E^T = exp(G_{L-1} - G) k^.  Off the
  // element-wise path both exponential factors come from the split ones:
  // exp(G_{L-1} - G) k^ = exp(G_{L-1} - G_m) fk, exp(G) k^ = exp(G_m) ek.
  if (tid >= 2 * kD) {
    const int i = tid - 2 * kD;
    const float GL = S.G[kL - 1][i], cl = S.cl[i];
#pragma unroll 4
    for (int t = 0; t < kL; t += 4) {
      float4 ke;
      if (!slow) {
        ke.x = cl * S.f.fk[t][i];
        ke.y = cl * S.f.fk[t + 1][i];
        ke.z = cl * S.f.fk[t + 2][i];
        ke.w = cl * S.f.fk[t + 3][i];
      } else {
        ke.x = expf(GL - S.G[t][i]) * S.k[t][i];
        ke.y = expf(GL - S.G[t + 1][i]) * S.k[t + 1][i];
        ke.z = expf(GL - S.G[t + 2][i]) * S.k[t + 2][i];
        ke.w = expf(GL - S.G[t + 3][i]) * S.k[t + 3][i];
      }
      *reinterpret_cast<float4*>(ws + kOffB2 + kpos(i, t, kNB2)) = ke;
    }
  } else {
    const bool vcol = tid < kD;
    const int i = tid - kD;
    const float egm = vcol ? 0.0f : S.egm[i];
    const bool split_y = !slow && egm > 0.0f;
    float x[kL];
#pragma unroll
    for (int t = 0; t < kL; ++t) {
      float a0 = vcol ? S.v[t][tid] : split_y ? egm * S.f.ek[t][i] : expf(S.G[t][i]) * S.k[t][i];
      float a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
      for (int s4 = 0; s4 < t / 4 + 1; ++s4) {
        if (4 * s4 >= t) break;
        const float4 pr = reinterpret_cast<const float4*>(S.P[t])[s4];
        if (4 * s4 + 0 < t) a0 = fmaf(-pr.x, x[4 * s4 + 0], a0);
        if (4 * s4 + 1 < t) a1 = fmaf(-pr.y, x[4 * s4 + 1], a1);
        if (4 * s4 + 2 < t) a2 = fmaf(-pr.z, x[4 * s4 + 2], a2);
        if (4 * s4 + 3 < t) a3 = fmaf(-pr.w, x[4 * s4 + 3], a3);
      }
      x[t] = S.beta[t] * ((a0 + a1) + (a2 + a3));
      if (vcol) ws[kOffU + t * kD + tid] = x[t];
      else S.f.ek[t][i] = x[t];  // W, staged
    }
  }
  __syncthreads();
  // W to the image as coalesced 16-byte pieces (t, keys 4 kg .. 4 kg + 3)
  for (int e = tid; e < kL * kD / 4; e += kChunkThreads) {
    const int t = e & (kL - 1), i0 = 4 * (e >> 5);
    *reinterpret_cast<float4*>(ws + kOffB1 + kpos(kL + t, i0, kNB1)) =
        *reinterpret_cast<const float4*>(&S.f.ek[t][i0]);
  }
}

// ====================================================================== scan
// tcgen05 helpers.  Shared-memory matrix descriptor of a canonical K-major
// operand without swizzle: start address, LBO (core matrices adjacent in K),
// SBO (8-row groups), descriptor version 1; all in 16-byte units.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFF) << 32) | (static_cast<uint64_t>(1) << 46);
}
// Instruction descriptor, kind::tf32: f32 accumulator, tf32 A and B, both
// K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
// D (tensor memory) (+)= A (tensor memory) x B (shared memory descriptor)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// three tf32 products of split operands: D += Alo*Bhi + Ahi*Blo + Ahi*Bhi
__device__ __forceinline__ void mma_ts3(uint32_t d, uint32_t ahi, uint32_t alo, uint64_t bhi, uint64_t blo,
                                        uint32_t idesc, uint32_t accumulate) {
  mma_ts(d, alo, bhi, idesc, accumulate);
  mma_ts(d, ahi, blo, idesc, 1);
  mma_ts(d, ahi, bhi, idesc, 1);
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// 16 consecutive columns of this warp's 32 lanes
__device__ __forceinline__ void tm_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tm_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 consecutive columns of this warp's 32 lanes; no wait (tm_wait_ld before use)
__device__ __forceinline__ void tm_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tm_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}

// Bounded wait on an mbarrier phase (2 s); false if it gave up.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    uint64_t now;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
    if (it == 0) t0 = now;
    else if (now - t0 > 2000000000ull) return false;
  }
}

// One CTA per (sequence, head): walks the sequence's chunks in order.  The
// state lives in tensor memory for the whole sequence (lane = value row,
// column = key) and every product with it runs on the 5th-generation tensor
// cores (tcgen05.mma, kind::tf32, issued by one thread, accumulators in
// tensor memory); chunk j's image (row chunk_offsets[b] + j of the
// workspace) arrives with one bulk copy while chunk j - 1 computes.
// Per chunk, two batches of products (M = 128 value rows):
//   [O^T | S^T W^T] = S^T [Q_G; W]^T              N = 64,  K = 128 keys
//   Delta^T = U^T - S^T W^T;  S^T <- S^T Diag(gamma)
//   [S^T | O^T] += Delta^T [K_E^T; R]^T           N = 160, K = 32 tokens
// Every operand is split into a tf32 high word and a tf32 remainder and three
// products are accumulated (lo*hi + hi*lo + hi*hi) in fp32.
template <bool kOutNorm>
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_scan_kernel(const PrefillParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ScanSmem& S = *reinterpret_cast<ScanSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = blockIdx.x / p.H, h = blockIdx.x - rank * p.H;
  const int b = p.seq_order ? p.seq_order[rank] : rank;
  if (b < 0 || b >= p.B) {
    if (tid == 0 && h == 0) flag(p, KDA_DEVERR_ORDER);
    return;
  }
  const int64_t D = static_cast<int64_t>(p.H) * kD;

  const int64_t r0 = p.cu[b], r1 = p.cu[b + 1];
  if (r0 < 0 || r1 < r0 || r1 > p.T) {
    if (tid == 0 && h == 0) flag(p, KDA_DEVERR_SEQLENS);
    return;
  }
  if (r1 == r0) return;  // empty sequence
  const int slot = p.slot_idx[b];
  if (slot <= 0 || slot >= p.num_slots) {
    // padding sequence: zero output rows of this head, touch nothing else
    for (int64_t e = tid; e < (r1 - r0) * (kD / 4); e += kThreads) {
      const int64_t row = r0 + e / (kD / 4);
      reinterpret_cast<uint2*>(p.out + row * p.out_stride + static_cast<int64_t>(h) * kD)[e % (kD / 4)] =
          make_uint2(0, 0);
    }
    if (slot >= p.num_slots && tid == 0 && h == 0) flag(p, KDA_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t n_chunks = (r1 - r0 + kL - 1) / kL;
  const int64_t c0 = p.chunk_off[b];
  if (c0 < 0 || p.chunk_off[b + 1] - c0 != n_chunks || c0 + n_chunks > p.num_chunks) {
    if (tid == 0 && h == 0) flag(p, KDA_DEVERR_SEQLENS);  // metadata does not match cu_seqlens
    return;
  }

  // warps w and w + 4 share tensor-memory lanes 32 (w % 4) .. + 31 and split
  // the columns: value row j = this thread's lane
  const int quad = warp & 3, half = warp >> 2;
  const int j = 32 * quad + lane;
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&S.bar[0])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&S.bar[1])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&S.full[0])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&S.full[1])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&S.efull)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&S.tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.tmem;
  const uint32_t tm = tbase + (static_cast<uint32_t>(32 * quad) << 16);  // this warp's lanes

  // state S^T row j, keys [64 half, 64 half + 64): fp32, high and low words
  float* Sg = p.state + (static_cast<int64_t>(slot) * p.H + h) * (kD * kD);
  float sx[64];  // all of this thread's loads in flight at once
#pragma unroll
  for (int e = 0; e < 64; ++e) sx[e] = Sg[static_cast<int64_t>(64 * half + e) * kD + j];
#pragma unroll
  for (int cc = 0; cc < 64; cc += 16) {
    uint32_t v[16], hi[16], lo[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float x = sx[cc + e];
      v[e] = __float_as_uint(x);
      hi[e] = tf32_hi(x);
      lo[e] = tf32_lo(x, hi[e]);
    }
    tm_st16(tm + kTS + 64 * half + cc, v);
    tm_st16(tm + kTSH + 64 * half + cc, hi);
    tm_st16(tm + kTSL + 64 * half + cc, lo);
  }
  tm_wait_st();

  // chunk jj's image: one bulk copy into buffer `buf`, issued by thread 0
  auto fetch = [&](int64_t jj, int buf) {
    if (tid == 0) {
      fence_proxy_async();  // earlier generic accesses to the buffer before the async-proxy write
      bulk_load(smem_u32(S.img[buf]), p.ws + ((c0 + jj) * p.H + h) * static_cast<int64_t>(kRec), kImg * 4,
                smem_u32(&S.full[buf]));
    }
  };
  // chunk jj's E: one bulk copy into the output rows (free once the previous
  // chunk's epilogue is done), issued by thread 0
  auto fetch_e = [&](int64_t jj) {
    if (tid == 0) {
      fence_proxy_async();  // the previous epilogue's reads before the async-proxy write
      bulk_load(smem_u32(&S.o[0][0]), p.ws + ((c0 + jj) * p.H + h) * static_cast<int64_t>(kRec) + kOffE,
                kL * kD * 4, smem_u32(&S.efull));
    }
  };
  fetch(0, 0);
  int pending = 0;           // buffer whose copy is in flight (-1: none)
  uint32_t pending_par = 0;  // and the phase its barrier completes
  int64_t e_pending = -1;    // chunk whose E copy is in flight (-1: none)
  constexpr uint32_t kId64 = idesc_tf32(kNB1), kId160 = idesc_tf32(kNB2);
  static_assert(kTD == kTO + kL, "the accumulators of [Q_G; W] must be adjacent");
  static_assert(kTO == kTS + kD, "the accumulators of [K_E^T; R] must be adjacent");
  const uint32_t lo_addr = smem_u32(S.lo);
  bool ok = true;
  // An image's tensor-core operands over float4 pieces [e0, e1): high words
  // in place, remainders to the same place in `lo`, fenced for the tensor
  // cores' view.
  auto split_operands = [&](float* imgp, int e0, int e1) {
    float4* im = reinterpret_cast<float4*>(imgp);
    float4* lo4 = reinterpret_cast<float4*>(S.lo);
    for (int e = e0 + tid; e < e1; e += kThreads) {
      float4 x = im[e], l;
      uint32_t hb;
      hb = tf32_hi(x.x); l.x = __uint_as_float(tf32_lo(x.x, hb)); x.x = __uint_as_float(hb);
      hb = tf32_hi(x.y); l.y = __uint_as_float(tf32_lo(x.y, hb)); x.y = __uint_as_float(hb);
      hb = tf32_hi(x.z); l.z = __uint_as_float(tf32_lo(x.z, hb)); x.z = __uint_as_float(hb);
      hb = tf32_hi(x.w); l.w = __uint_as_float(tf32_lo(x.w, hb)); x.w = __uint_as_float(hb);
      im[e] = x;
      lo4[e] = l;
    }
    fence_proxy_async();
  };
  const float4 nw4 = kOutNorm ? __ldg(reinterpret_cast<const float4*>(p.norm_w) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);

  for (int64_t jj = 0; jj < n_chunks; ++jj) {
    const int64_t t0 = r0 + kL * jj;
    const int L = static_cast<int>(r1 - t0 < kL ? r1 - t0 : kL);
    const int buf = static_cast<int>(jj & 1);
    const uint32_t par = static_cast<uint32_t>(jj & 1);
    ok = bar_wait(smem_u32(&S.full[buf]), static_cast<uint32_t>((jj >> 1) & 1));
    if (__syncthreads_or(!ok)) break;      // image jj landed; the other buffer and lo are free
    pending = -1;
    if (jj + 1 < n_chunks) {
      fetch(jj + 1, buf ^ 1);
      pending = buf ^ 1;
      pending_par = static_cast<uint32_t>(((jj + 1) >> 1) & 1);
    }
    fetch_e(jj);
    e_pending = jj;
    float* img = S.img[buf];
    const uint32_t img_addr = smem_u32(img);

    // [Q_G; W] of every chunk after the first was split while the previous
    // chunk's second product batch ran; the first chunk's is split here
    if (jj == 0) {
      split_operands(img, kOffB1 / 4, kOffB2 / 4);
      tc_fence_before();
      __syncthreads();
    }
    tc_fence_after();

    // ---- [D_O | D_Delta] = S^T [Q_G; W]^T  (N = 64, one B block; the two
    // accumulators are adjacent; K = 128 keys, 16 steps of 8)
    if (tid == 0) {
      // LBO = 64 rows x 16 B; one K step of 8 = two core-matrix columns = 2 LBO = 128 address units
      const uint64_t bh = sdesc(img_addr + 4 * kOffB1, kNB1 * 16, 128), bl = sdesc(lo_addr + 4 * kOffB1, kNB1 * 16, 128);
#pragma unroll 1
      for (int ks = 0; ks < kD / 8; ++ks)
        mma_ts3(tbase + kTO, tbase + kTSH + 8 * ks, tbase + kTSL + 8 * ks, bh + 128 * ks, bl + 128 * ks, kId64,
                ks > 0);
      mma_commit(smem_u32(&S.bar[0]));
    }
    // While those run (they read the split words, not the fp32 state):
    // S^T <- S^T Diag(gamma) over this thread's 64 keys, and the gate rows of
    // the tokens this warp writes out
    {
      const float* gC = img + kOffC + 64 * half;
      uint32_t r0[32], r1[32];
      tm_ld32_nowait(tm + kTS + 64 * half, r0);
      tm_ld32_nowait(tm + kTS + 64 * half + 32, r1);
      tm_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        r0[e] = __float_as_uint(__uint_as_float(r0[e]) * gC[e]);
        r1[e] = __float_as_uint(__uint_as_float(r1[e]) * gC[32 + e]);
      }
      tm_st32(tm + kTS + 64 * half, r0);
      tm_st32(tm + kTS + 64 * half + 32, r1);
    }
    uint2 gate_pf[4];
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const int t = warp * 4 + tt;
      gate_pf[tt] = make_uint2(0, 0);
      if (kOutNorm && t < L)
        gate_pf[tt] = __ldg(reinterpret_cast<const uint2*>(p.gate + (t0 + t) * p.gate_stride +
                                                           static_cast<int64_t>(h) * kD) + lane);
    }
    // [K_E^T; R] of this image (the first batch reads only [Q_G; W])
    split_operands(img, kOffB2 / 4, kSplit / 4);
    ok = bar_wait(smem_u32(&S.bar[0]), par);
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();

    // Delta^T = U^T - D_Delta for row j, tokens [16 half, 16 half + 16): split
    {
      uint32_t r[16], dh[16], dl[16];
      tm_ld16(tm + kTD + 16 * half, r);
      const float* ucol = img + kOffU + (16 * half) * kD + j;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float dv = ucol[e * kD] - __uint_as_float(r[e]);
        dh[e] = tf32_hi(dv);
        dl[e] = tf32_lo(dv, dh[e]);
      }
      tm_st16(tm + kTDH + 16 * half, dh);
      tm_st16(tm + kTDL + 16 * half, dl);
    }
    tm_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- [S^T | D_O] += Delta^T [K_E^T; R]^T  (N = 160, one B block; S^T and
    // the output accumulator are adjacent; K = 32 tokens, 4 steps of 8)
    if (tid == 0) {
      // LBO = 160 rows x 16 B; one K step = 2 LBO = 320 address units
      const uint64_t bh = sdesc(img_addr + 4 * kOffB2, kNB2 * 16, 128),
                     bl = sdesc(lo_addr + 4 * kOffB2, kNB2 * 16, 128);
#pragma unroll 1
      for (int ks = 0; ks < kL / 8; ++ks)
        mma_ts3(tbase + kTS, tbase + kTDH + 8 * ks, tbase + kTDL + 8 * ks, bh + 320 * ks, bl + 320 * ks, kId160, 1);
      mma_commit(smem_u32(&S.bar[1]));
    }
    // While it runs (it reads only [K_E^T; R]'s remainders): the next image's
    // [Q_G; W] split, once it has landed
    bool ok_next = true;
    if (jj + 1 < n_chunks) {
      ok_next = bar_wait(smem_u32(&S.full[buf ^ 1]), pending_par);
      if (ok_next) split_operands(S.img[buf ^ 1], kOffB1 / 4, kOffB2 / 4);
    }
    ok = bar_wait(smem_u32(&S.bar[1]), par) && ok_next && bar_wait(smem_u32(&S.efull), par);
    if (ok) e_pending = -1;
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();

    // the chunk's output rows (D_O added to E in shared memory); the new state's split words
    {
      uint32_t r[16];
      tm_ld16(tm + kTO + 16 * half, r);
#pragma unroll
      for (int e = 0; e < 16; ++e) S.o[16 * half + e][j] += __uint_as_float(r[e]);  // E + D_O
#pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        uint32_t v[32], hi[32];
        tm_ld32_nowait(tm + kTS + 64 * half + cc, v);
        tm_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float x = __uint_as_float(v[e]);
          hi[e] = tf32_hi(x);
          v[e] = tf32_lo(x, hi[e]);
        }
        tm_st32(tm + kTSH + 64 * half + cc, hi);
        tm_st32(tm + kTSL + 64 * half + cc, v);
      }
    }
    tm_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- gated RMSNorm (or raw o) to bf16; warp w writes tokens 4w..4w+3,
    // the four reductions interleaved
    {
      float4 y[4];
      float ss[4];
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        y[tt] = reinterpret_cast<const float4*>(S.o[warp * 4 + tt])[lane];
        ss[tt] = (y[tt].x * y[tt].x + y[tt].y * y[tt].y) + (y[tt].z * y[tt].z + y[tt].w * y[tt].w);
      }
      if (kOutNorm) {
#pragma unroll
        for (int m = 16; m > 0; m >>= 1)
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) ss[tt] += __shfl_xor_sync(0xffffffffu, ss[tt], m);
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          const float rr = rsqrtf(ss[tt] * (1.0f / kD) + p.eps);
          const uint2 gb = gate_pf[tt];
          y[tt].x = __fdividef(y[tt].x * rr * nw4.x, 1.0f + __expf(-__uint_as_float(gb.x << 16)));
          y[tt].y = __fdividef(y[tt].y * rr * nw4.y, 1.0f + __expf(-__uint_as_float(gb.x & 0xFFFF0000u)));
          y[tt].z = __fdividef(y[tt].z * rr * nw4.z, 1.0f + __expf(-__uint_as_float(gb.y << 16)));
          y[tt].w = __fdividef(y[tt].w * rr * nw4.w, 1.0f + __expf(-__uint_as_float(gb.y & 0xFFFF0000u)));
        }
      }
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int t = warp * 4 + tt;
        if (t < L)
          reinterpret_cast<uint2*>(p.out + (t0 + t) * p.out_stride + static_cast<int64_t>(h) * kD)[lane] =
              make_uint2(pack_bf16x2(y[tt].x, y[tt].y), pack_bf16x2(y[tt].z, y[tt].w));
      }
    }
  }
  if (!ok && pending >= 0) {
    // leaving early: let the copy in flight land before the shared memory goes away
    bar_wait(smem_u32(&S.full[pending]), pending_par);
  }
  if (!ok && e_pending >= 0) bar_wait(smem_u32(&S.efull), static_cast<uint32_t>(e_pending & 1));
  if (ok) {
    // ---- sequence end: state and conv window back to the slot.  The window
    // [old taps | tokens] ends with its last three inputs; for sequences of
    // fewer than three tokens some of them are old taps.
#pragma unroll
    for (int cc = 0; cc < 64; cc += 16) {
      uint32_t r[16];
      tm_ld16(tm + kTS + 64 * half + cc, r);
#pragma unroll
      for (int e = 0; e < 16; ++e) Sg[static_cast<int64_t>(64 * half + cc + e) * kD + j] = __uint_as_float(r[e]);
    }
    uint16_t* cs = p.conv_state + static_cast<int64_t>(slot) * 3 * D * kHist;
    const int64_t sc = p.conv_sd ? 1 : kHist, sr = p.conv_sd ? 3 * D : 1;  // dim-first or tap-first
    const int64_t len = r1 - r0;
    for (int ch = tid; ch < kCh; ch += kThreads) {
      const int64_t cg = static_cast<int64_t>(ch >> 7) * D + static_cast<int64_t>(h) * kD + (ch & 127);
      uint16_t w3[kHist];
#pragma unroll
      for (int r = 0; r < kHist; ++r) {
        const int64_t pos = len + r;  // position in the window [old taps (3) | tokens (len)]
        w3[r] = pos < kHist ? cs[cg * sc + pos * sr] : p.qkv[(r0 + pos - kHist) * p.qkv_stride + cg];
      }
#pragma unroll
      for (int r = 0; r < kHist; ++r) cs[cg * sc + r * sr] = w3[r];
    }
  } else if (tid == 0) {
    flag(p, KDA_DEVERR_TIMEOUT);  // a tensor-core step never completed; the slot is left as it was
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tbase));
}

std::mutex g_mutex;
bool g_attrs_set[64];

cudaError_t setup() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_attrs_set[dev]) {
    if ((e = cudaFuncSetAttribute(kda_prefill_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(sizeof(ChunkSmem)))) != cudaSuccess)
      return e;
    const int scan = static_cast<int>(sizeof(ScanSmem));
    if ((e = cudaFuncSetAttribute(kda_prefill_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  scan)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(kda_prefill_scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  scan)) != cudaSuccess)
      return e;
    g_attrs_set[dev] = true;
  }
  return cudaSuccess;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace

extern "C" int64_t kda_prefill_workspace_bytes(int64_t num_chunks, int32_t H) {
  if (num_chunks < 0 || H < 1) return -1;
  return num_chunks * H * static_cast<int64_t>(kRec) * 4;
}

extern "C" int kda_prefill_longest_first(const int32_t* cu_seqlens, int32_t B, int32_t* order) {
  kda_internal_clear_error();
  if (B < 0) return kda_internal_fail(KDA_ERR_SHAPE, "B=%d", B);
  if (B > 0 && (!cu_seqlens || !order)) return kda_internal_fail(KDA_ERR_NULLPTR, "cu_seqlens or order is NULL");
  // Lengths are taken in the comparison and the sort is std::sort, which
  // works in place: nothing here allocates and no exception can cross the C
  // boundary.  Ties are broken by index, so the order is unique and equals
  // the stable one (equal lengths in index order).
  const auto len = [cu_seqlens](int32_t i) {
    const int64_t n = static_cast<int64_t>(cu_seqlens[i + 1]) - cu_seqlens[i];
    return n < 0 ? int64_t{0} : n;
  };
  for (int32_t i = 0; i < B; ++i) order[i] = i;
  std::sort(order, order + B, [&](int32_t x, int32_t y) {
    const int64_t lx = len(x), ly = len(y);
    return lx > ly || (lx == ly && x < y);
  });
  return KDA_OK;
}

extern "C" int kda_prefill(const KdaPrefillArgs* a, void* stream) {
  kda_internal_clear_error();
  if (!a) return kda_internal_fail(KDA_ERR_NULLPTR, "args is NULL");
  if (a->struct_size != sizeof(KdaPrefillArgs))
    return kda_internal_fail(KDA_ERR_ABI, "struct_size %zu, library expects %zu", a->struct_size,
                             sizeof(KdaPrefillArgs));
  if (a->head_dim != KDA_HEAD_DIM || a->conv_width != KDA_CONV_WIDTH)
    return kda_internal_fail(KDA_ERR_SHAPE, "head_dim %d / conv_width %d (need 128 / 4)", a->head_dim,
                             a->conv_width);
  if (a->B < 0 || a->H < 1 || a->H > 65535 || a->num_slots < 1 || a->T < 0 || a->num_chunks < 0)
    return kda_internal_fail(KDA_ERR_SHAPE, "B=%d H=%d num_slots=%d T=%lld num_chunks=%lld", a->B, a->H,
                             a->num_slots, static_cast<long long>(a->T), static_cast<long long>(a->num_chunks));
  if (a->flags & ~(KDA_OUT_NORM | KDA_FUSED_GATE | KDA_CONV_STATE_SD))
    return kda_internal_fail(KDA_ERR_FLAGS, "flags 0x%x (KDA_OUT_NORM, KDA_FUSED_GATE, KDA_CONV_STATE_SD only)",
                             a->flags);
  if (static_cast<int64_t>(a->B) * a->H > 0x7fffffffLL || a->num_chunks > 0x7fffffffLL)
    return kda_internal_fail(KDA_ERR_SHAPE, "B*H or num_chunks too large");
  if (a->B == 0 || a->T == 0) return KDA_OK;
  const bool norm = (a->flags & KDA_OUT_NORM) != 0;
  const int64_t D = static_cast<int64_t>(a->H) * KDA_HEAD_DIM;
  if (!a->cu_seqlens || !a->chunk_offsets || !a->qkv || !a->conv_weight || !a->conv_state || !a->state || !a->g ||
      !a->beta || !a->slot_idx || !a->out || (a->num_chunks > 0 && (!a->chunk_indices || !a->workspace)))
    return kda_internal_fail(KDA_ERR_NULLPTR, "a required pointer is NULL");
  if (norm && (!a->gate || !a->norm_weight))
    return kda_internal_fail(KDA_ERR_NULLPTR, "KDA_OUT_NORM needs gate and norm_weight");
  const bool fused = (a->flags & KDA_FUSED_GATE) != 0;
  if (fused && !a->A_log) return kda_internal_fail(KDA_ERR_NULLPTR, "KDA_FUSED_GATE needs A_log");
  if (fused && (!aligned(a->A_log, 4) || (a->dt_bias && !aligned(a->dt_bias, 4))))
    return kda_internal_fail(KDA_ERR_ALIGN, "A_log / dt_bias must be 4-byte aligned");
  if (a->qkv_row_stride < 3 * D || a->out_row_stride < D || (norm && a->gate_row_stride < D))
    return kda_internal_fail(KDA_ERR_SHAPE, "a row stride is smaller than the row");
  if (a->workspace_bytes < kda_prefill_workspace_bytes(a->num_chunks, a->H))
    return kda_internal_fail(KDA_ERR_SHAPE, "workspace of %lld bytes, %lld needed",
                             static_cast<long long>(a->workspace_bytes),
                             static_cast<long long>(kda_prefill_workspace_bytes(a->num_chunks, a->H)));
  if (!aligned(a->qkv, 16) || (a->qkv_row_stride & 7) || !aligned(a->state, 16) || !aligned(a->g, 16) ||
      !aligned(a->out, 8) || (a->out_row_stride & 3) || !aligned(a->cu_seqlens, 4) || !aligned(a->slot_idx, 4) ||
      !aligned(a->chunk_indices, 8) || !aligned(a->chunk_offsets, 8) || !aligned(a->workspace, 16) ||
      !aligned(a->conv_weight, 4) || !aligned(a->conv_state, 2) || !aligned(a->beta, 2) ||
      !aligned(a->err_flag, 4) || !aligned(a->seq_order, 4) || (a->conv_bias && !aligned(a->conv_bias, 4)) ||
      (norm && (!aligned(a->gate, 8) || (a->gate_row_stride & 3) || !aligned(a->norm_weight, 16))))
    return kda_internal_fail(KDA_ERR_ALIGN, "a pointer or row stride is not aligned as required");
  cudaError_t e = setup();
  if (e != cudaSuccess) return kda_internal_fail(KDA_ERR_LAUNCH, "setup: %s", cudaGetErrorString(e));

  PrefillParams p;
  p.cu = a->cu_seqlens;
  p.chunk_idx = a->chunk_indices;
  p.chunk_off = a->chunk_offsets;
  p.num_chunks = a->num_chunks;
  p.ws = static_cast<float*>(a->workspace);
  p.qkv = a->qkv;
  p.qkv_stride = a->qkv_row_stride;
  p.conv_w = a->conv_weight;
  p.conv_b = a->conv_bias;
  p.conv_state = a->conv_state;
  p.state = a->state;
  p.g = a->g;
  p.beta = a->beta;
  p.gate = a->gate;
  p.gate_stride = a->gate_row_stride;
  p.norm_w = a->norm_weight;
  p.slot_idx = a->slot_idx;
  p.out = a->out;
  p.out_stride = a->out_row_stride;
  p.T = a->T;
  p.B = a->B;
  p.H = a->H;
  p.num_slots = a->num_slots;
  p.eps = a->eps;
  p.q_scale = a->q_scale;
  p.err = a->err_flag;
  p.conv_sd = (a->flags & KDA_CONV_STATE_SD) ? 1 : 0;
  p.fused_gate = fused ? 1 : 0;
  p.A_log = fused ? a->A_log : nullptr;
  p.dt_bias = fused ? a->dt_bias : nullptr;
  p.lower_bound = a->lower_bound;
  p.seq_order = a->seq_order;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->num_chunks > 0)
    kda_prefill_chunk_kernel<<<dim3(static_cast<unsigned>(a->num_chunks), static_cast<unsigned>(a->H)), kChunkThreads,
                               sizeof(ChunkSmem), s>>>(p);
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(a->B) * a->H));
  if (norm)
    kda_prefill_scan_kernel<true><<<grid, kThreads, sizeof(ScanSmem), s>>>(p);
  else
    kda_prefill_scan_kernel<false><<<grid, kThreads, sizeof(ScanSmem), s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return kda_internal_fail(KDA_ERR_LAUNCH, "launch: %s", cudaGetErrorString(e));
  return KDA_OK;
}
