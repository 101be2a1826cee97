// kda_decode_kernel.cuh -- device code of the fused KDA decode step
// (sm_103a): constants, parameter block, PTX wrappers and the persistent
// kernel.  Included once, by kda_decode.cu, which holds the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_decode.h"

namespace {

constexpr int kDim = 128;                      // key = value head dim
constexpr int kWidth = 4;                      // conv taps
constexpr int kStages = 3;                     // state tiles in flight per CTA
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;  // 256 math threads
constexpr int kThreads = kConsumers + 32;        // + one producer warp
constexpr int kRowsPerWarp = kDim / kConsumerWarps;  // 16 key rows per consumer warp
constexpr int kEarlyStages = 2;  // ring stages whose state may stream in before the previous kernel ends
constexpr uint32_t kTileBytes = kDim * kDim * 4;           // 64 KiB fp32 state tile
constexpr uint32_t kCsSliceBytes = kDim * (kWidth - 1) * 2;  // 768 B conv state per block
constexpr uint32_t kXSliceBytes = kDim * 2;                  // 256 B qkv per block
constexpr int kCsU4 = kCsSliceBytes / 16;                    // 48
constexpr uint64_t kWaitLimitNs = 2000000000ull;             // bounded waits: 2 s by default

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
  int total_units;  // N * H
  int early_prefetch;  // KDA_EARLY_PREFETCH
  int fused_gate;      // KDA_FUSED_GATE: g / beta are raw logits
  int conv_sd;         // KDA_CONV_STATE_SD: conv state [slots][3][C]
  const float* A_log;
  const float* dt_bias;
  float lower_bound;
  int* queue;          // work queue int32[2] (next dynamic unit, finished CTAs) or null
  int static_units;    // with a queue: units each CTA takes statically before drawing from it
  int withhold_unit;   // wait-path test: this unit's load is never signalled (-1: none)
  uint64_t wait_limit_ns;
  float eps, q_scale;
  int32_t* err;
  int T;                     // tokens per sequence (multi-token kernel; 1 otherwise)
  const int32_t* src_slot;   // multi-token kernel: source slot per sequence, or null
};

// Dynamic shared memory of one CTA (about 214 KB): the staged tiles and the
// per-unit inputs for kStages units, plus the consumers' scratch.
struct __align__(128) Smem {
  float tile[kStages][kDim * kDim];
  uint16_t cs[kStages][3][kDim * (kWidth - 1)];  // per block: [128][3] (DS) or [3][128] (SD)
  uint16_t x[kStages][3][kDim];
  float g[kStages][kDim];
  uint16_t gate[kStages][kDim];
  float q[kDim], k[kDim], v[kDim], alpha[kDim];
  float red[2][kConsumerWarps][kDim];
  float delta[kDim];
  float4 part[kConsumerWarps];    // per-warp |q~|^2, |k~|^2, q~.k~ over the warp's 16 key rows
  float osum[4];                  // per-warp sum of o_j^2 (warps 0-3)
  int info[kStages][4];           // slot, n (-1: no more units), h, withheld
  unsigned long long ready[kStages];  // info of the stage is written
  unsigned long long full[kStages];
  unsigned long long done[kStages];
  volatile int abort;
};

#ifdef KDA_DECODE_TIMELINE
// Timeline build only: one record per CTA (block, SM, start, first unit
// ready, end, units, consumer compute ns, consumer wait ns), appended by
// consumer thread 0 when the CTA finishes.
constexpr int kTimelineMax = 1 << 16;
__device__ unsigned long long g_timeline[kTimelineMax][8];
__device__ unsigned int g_timeline_n;
#endif

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

// ---- PTX wrappers: mbarrier, bulk async copies (TMA engine), barriers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Shared -> global bulk copy tracked by the issuing thread's bulk group.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
               "r"(src), "r"(bytes), "l"(policy)
               : "memory");
}

// L2 prefetch hint of a 16-byte aligned range (a multiple of 16 bytes): it
// only warms L2, so it may be issued before the data's producer has finished
// (its writes land in L2 as well and later reads see them).
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier 1 among the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Consumer-wide OR of a predicate (also a barrier).
__device__ __forceinline__ int consumer_any(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 2, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(kConsumers)
      : "memory");
  return r;
}

// Programmatic dependent launch: let the next kernel in the stream be
// scheduled now, and wait for the previous one to complete (with its memory
// visible) before touching anything it may have written.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void flag_error(const Params& p, int bits) {
  if (p.err) atomicOr(p.err, bits);
}

// Slot-independent inputs one consumer thread needs for a unit: its conv
// taps (thread tid: q channel tid or k channel tid-128, plus v channel tid
// for tid < 128), conv biases, beta, and the gate parameters of key channel
// tid-128 when the gate is fused.
struct UnitInputs {
  float wq[kWidth], wv[kWidth];
  float bq, bv, beta, gate_a, gate_bias;
};

__device__ __forceinline__ UnitInputs load_unit_inputs(const Params& p, int n, int h, int tid, int64_t D) {
  UnitInputs u;
  u.bq = u.bv = u.beta = u.gate_a = u.gate_bias = 0.0f;
  const int c = tid >> 7, j = tid & (kDim - 1);
  const float* w = p.conv_w + c * kWidth * D + static_cast<int64_t>(h) * kDim + j;
#pragma unroll
  for (int t = 0; t < kWidth; ++t) u.wq[t] = __ldg(w + t * D);
  if (p.conv_b) u.bq = __ldg(p.conv_b + c * D + static_cast<int64_t>(h) * kDim + j);
  if (tid < kDim) {
    const float* w2 = p.conv_w + 2 * kWidth * D + static_cast<int64_t>(h) * kDim + j;
#pragma unroll
    for (int t = 0; t < kWidth; ++t) u.wv[t] = __ldg(w2 + t * D);
    if (p.conv_b) u.bv = __ldg(p.conv_b + 2 * D + static_cast<int64_t>(h) * kDim + j);
    const float b = bf16_to_f32(__ldg(p.beta + static_cast<int64_t>(n) * p.H + h));
    u.beta = p.fused_gate ? 1.0f / (1.0f + expf(-b)) : b;
  } else {
#pragma unroll
    for (int t = 0; t < kWidth; ++t) u.wv[t] = 0.0f;
    if (p.fused_gate) {
      u.gate_a = expf(__ldg(p.A_log + h));
      if (p.dt_bias) u.gate_bias = __ldg(p.dt_bias + static_cast<int64_t>(h) * kDim + j);
    }
  }
  return u;
}

// Persistent kernel, one CTA per SM.  A unit is one (row n, head h) =
// unit index n*H + h.  Each CTA takes units statically (blockIdx.x +
// k*gridDim.x; the first ones can be prefetched before the previous kernel
// finishes).  With a work queue only the first p.static_units are static
// and the rest come from the queue (an atomic counter: CTAs that run ahead
// take more units, so every CTA finishes at nearly the same time); without
// one the static stride covers everything.
// Warp 8 is the producer: for each unit it publishes (slot, n, h) on the
// stage's `ready` barrier, streams the 64 KiB state tile and the unit's small
// inputs into the stage with bulk copies (`full` barrier), and once the
// consumers release the stage (`done`) streams the updated tile back out.
// Warps 0-7 compute.  Two tiles stream in while the consumers work on a third.
template <bool kOutNorm, bool kUpdateConv>
__global__ void __launch_bounds__(kThreads, 1) kda_decode_persistent_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int64_t D = static_cast<int64_t>(p.H) * kDim;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&S.ready[s]), 1);
      mbar_init(smem_addr(&S.full[s]), 1);
      mbar_init(smem_addr(&S.done[s]), kConsumerWarps);
    }
    S.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t in_bytes = kTileBytes + 3 * kCsSliceBytes + 3 * kXSliceBytes + kDim * 4 +
                              (kOutNorm ? kXSliceBytes : 0);
    // Slot-indexed inputs of a unit: its state tile and conv-state slices.
    auto load_slot_parts = [&](int stage, int h, int slot) {
      const uint32_t full = smem_addr(&S.full[stage]);
      bulk_load(smem_addr(S.tile[stage]), p.state + (static_cast<int64_t>(slot) * p.H + h) * (kDim * kDim),
                kTileBytes, full, policy);
      for (int c = 0; c < 3; ++c) {
        if (!p.conv_sd) {  // dim-first: one contiguous 768-byte slice per block
          bulk_load(smem_addr(S.cs[stage][c]),
                    p.conv_state +
                        (static_cast<int64_t>(slot) * 3 * D + c * D + static_cast<int64_t>(h) * kDim) * (kWidth - 1),
                    kCsSliceBytes, full, policy);
        } else {  // tap-first: one 256-byte channel run per tap
          for (int t = 0; t < kWidth - 1; ++t)
            bulk_load(smem_addr(S.cs[stage][c] + t * kDim),
                      p.conv_state + (static_cast<int64_t>(slot) * (kWidth - 1) + t) * 3 * D + c * D +
                          static_cast<int64_t>(h) * kDim,
                      kXSliceBytes, full, policy);
        }
      }
    };
    // Per-token inputs of a unit: qkv slices, g row, gate row.
    auto load_token_parts = [&](int stage, int n, int h) {
      const uint32_t full = smem_addr(&S.full[stage]);
      for (int c = 0; c < 3; ++c)
        bulk_load(smem_addr(S.x[stage][c]), p.qkv + n * p.qkv_stride + c * D + static_cast<int64_t>(h) * kDim,
                  kXSliceBytes, full, policy);
      bulk_load(smem_addr(S.g[stage]), p.g + (static_cast<int64_t>(n) * p.H + h) * kDim, kDim * 4, full, policy);
      if (kOutNorm)
        bulk_load(smem_addr(S.gate[stage]), p.gate + n * p.gate_stride + static_cast<int64_t>(h) * kDim,
                  kXSliceBytes, full, policy);
    };
    auto active = [&](int slot) { return slot > 0 && slot < p.num_slots; };
    // Write the stage's tile back if it held an active unit.
    auto store_stage = [&](int stage) {
      const int* prev = S.info[stage];
      if (active(prev[0])) {
        float* dst = p.state + (static_cast<int64_t>(prev[0]) * p.H + prev[2]) * (kDim * kDim);
        bulk_store(dst, smem_addr(S.tile[stage]), kTileBytes, policy);
        bulk_commit();
      }
    };
    int k_static = 0;  // static units taken so far
    auto next_unit = [&]() -> int {
      int u;
      if (k_static < p.static_units || p.queue == nullptr)
        u = blockIdx.x + (k_static++) * G;
      else
        u = p.static_units * G + atomicAdd(p.queue, 1);
      return u < p.total_units ? u : -1;
    };

    // L2 hints for a unit's per-token slices and its head's conv taps.
    auto warm_l2 = [&](int n, int h) {
      for (int c = 0; c < 3; ++c) l2_prefetch(p.qkv + n * p.qkv_stride + c * D + static_cast<int64_t>(h) * kDim, kXSliceBytes);
      l2_prefetch(p.g + (static_cast<int64_t>(n) * p.H + h) * kDim, kDim * 4);
      if (kOutNorm) l2_prefetch(p.gate + n * p.gate_stride + static_cast<int64_t>(h) * kDim, kXSliceBytes);
      for (int c = 0; c < 3; ++c)
        for (int t = 0; t < kWidth; ++t) l2_prefetch(p.conv_w + (c * kWidth + t) * D + static_cast<int64_t>(h) * kDim, kDim * 4);
      // beta: the 16-byte piece holding it, when that piece lies inside the
      // tensor (beta needs only 2-byte alignment); the norm weight
      const uintptr_t b0 = reinterpret_cast<uintptr_t>(p.beta);
      const uintptr_t b1 = reinterpret_cast<uintptr_t>(p.beta + static_cast<int64_t>(p.N) * p.H);
      const uintptr_t bp = reinterpret_cast<uintptr_t>(p.beta + static_cast<int64_t>(n) * p.H + h) & ~uintptr_t{15};
      if (bp >= b0 && bp + 16 <= b1) l2_prefetch(reinterpret_cast<const void*>(bp), 16);
      if (kOutNorm) l2_prefetch(p.norm_w, kDim * 4);
    };
    // First ring: static units.  With KDA_EARLY_PREFETCH the first two
    // units' state streams in before the previous kernel in the stream has
    // finished (the caller guarantees that kernel does not write the slot
    // indices, the state or the conv state), and their per-token slices and
    // conv taps are pulled into L2; everything per-token is read only after
    // it.  Without it the ring fills one stage at a time (each
    // stage once the one before it has landed), so that the first tile of
    // every CTA arrives early instead of all CTAs' three tiles arriving
    // together; with it the third stage follows the same rule.
    int it = 0;
    for (; it < kStages; ++it) {
      const int u = next_unit();
      if (u < 0) break;
      const int n = u / p.H, h = u - n * p.H;
      S.info[it][1] = n;
      S.info[it][2] = h;
      S.info[it][3] = (u == p.withhold_unit);
      if (p.early_prefetch && it < kEarlyStages) {
        const int slot = __ldg(p.slot_idx + n);
        S.info[it][0] = slot;
        if (active(slot) && !S.info[it][3]) {
          mbar_arrive_expect_tx(smem_addr(&S.full[it]), in_bytes);
          load_slot_parts(it, h, slot);
          warm_l2(n, h);
        }
      }
    }
    griddep_wait();
    for (int j = 0; j < it; ++j) {
      const int n = S.info[j][1], h = S.info[j][2];
      const bool early_j = p.early_prefetch && j < kEarlyStages;
      if (j > 0 && !early_j && !S.info[j - 1][3]) mbar_wait_bounded(smem_addr(&S.full[j - 1]), 0, p.wait_limit_ns);
      if (!early_j) {
        const int slot = __ldg(p.slot_idx + n);
        S.info[j][0] = slot;
        if (active(slot) && !S.info[j][3]) {
          mbar_arrive_expect_tx(smem_addr(&S.full[j]), in_bytes);
          load_slot_parts(j, h, slot);
        }
      }
      mbar_arrive(smem_addr(&S.ready[j]));
      if (S.info[j][3]) continue;  // withheld (wait-path test): never signalled
      if (active(S.info[j][0]))
        load_token_parts(j, n, h);
      else
        mbar_arrive(smem_addr(&S.full[j]));  // padding row: nothing to stream
    }

    // Steady state: the next unit and its slot are fetched one step ahead.
    int next = (it == kStages) ? next_unit() : -1;
    int next_slot = next >= 0 ? __ldg(p.slot_idx + next / p.H) : 0;
    bool ok = true;
    for (; next >= 0; ++it) {
      const int unit = next, slot = next_slot;
      next = next_unit();
      next_slot = next >= 0 ? __ldg(p.slot_idx + next / p.H) : 0;
      const int stage = it % kStages;
      const int n = unit / p.H, h = unit - n * p.H;
      // Stage reuse: the consumers must have released the previous unit in
      // this stage; write its tile back and let the copy engine finish
      // reading it before the stage is refilled.
      if (!mbar_wait_bounded(smem_addr(&S.done[stage]), ((it / kStages) - 1) & 1, p.wait_limit_ns)) {
        ok = false;
        break;
      }
      store_stage(stage);
      bulk_wait_read_all();
      S.info[stage][0] = slot;
      S.info[stage][1] = n;
      S.info[stage][2] = h;
      S.info[stage][3] = (unit == p.withhold_unit);
      mbar_arrive(smem_addr(&S.ready[stage]));
      if (S.info[stage][3]) continue;  // withheld (wait-path test): never signalled
      if (active(slot)) {
        mbar_arrive_expect_tx(smem_addr(&S.full[stage]), in_bytes);
        load_slot_parts(stage, h, slot);
        load_token_parts(stage, n, h);
      } else {
        mbar_arrive(smem_addr(&S.full[stage]));  // padding or out-of-range row
      }
    }
    // This CTA draws no more units: the last CTA to get here returns the
    // work queue to zero for the next call.  Done now rather than at exit,
    // so the atomic's round trip overlaps the units still in the ring.
    if (p.queue != nullptr) {
      __threadfence();
      if (atomicAdd(p.queue + 1, 1) == G - 1) {
        atomicExch(p.queue, 0);
        atomicExch(p.queue + 1, 0);
      }
    }
    // End of work: the consumers find n = -1 in the next stage they read.
    if (ok) {
      const int stage = it % kStages;
      if (it >= kStages) {
        ok = mbar_wait_bounded(smem_addr(&S.done[stage]), ((it / kStages) - 1) & 1, p.wait_limit_ns);
        if (ok) store_stage(stage);
      }
      if (ok) {
        bulk_wait_read_all();
        S.info[stage][1] = -1;
        mbar_arrive(smem_addr(&S.ready[stage]));
      }
    }
    // Drain: write back the units still held in the ring.
    for (int j = it > kStages - 1 ? it - kStages + 1 : 0; ok && j < it; ++j) {
      const int stage = j % kStages;
      ok = mbar_wait_bounded(smem_addr(&S.done[stage]), (j / kStages) & 1, p.wait_limit_ns);
      if (ok) store_stage(stage);
    }
    if (!ok) {
      flag_error(p, KDA_DEVERR_TIMEOUT);
      S.abort = 1;
    }
    // Before the CTA's shared memory goes away: every load this thread armed
    // has landed (normally long since) and every store has completed.
    for (int j = it > kStages ? it - kStages : 0; j < it; ++j) {
      const int stage = j % kStages;
      if (!mbar_wait_bounded(smem_addr(&S.full[stage]), (j / kStages) & 1, p.wait_limit_ns))
        flag_error(p, KDA_DEVERR_TIMEOUT);
    }
    bulk_wait_all();
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();
  const float scale = (p.q_scale != 0.0f) ? p.q_scale : 0.088388347648318440550f;  // 1/sqrt(128)
  const float nw = (kOutNorm && tid < kDim) ? __ldg(p.norm_w + tid) : 0.0f;
  UnitInputs cur, nxt;
  bool have_next = false;  // nxt holds the inputs of the coming unit
#ifdef KDA_DECODE_TIMELINE
  // thread 0's accumulators, in shared memory so that they take no registers:
  // start, first unit ready, wait, compute, units, loop top, vote passed
  __shared__ unsigned long long tl_acc[7];
  volatile unsigned long long* tl = tl_acc;
  if (tid == 0) {
    tl[0] = global_ns();
    for (int i = 1; i < 7; ++i) tl[i] = 0;
  }
#endif
  for (int it = 0;; ++it) {
#ifdef KDA_DECODE_TIMELINE
    if (tid == 0) {
      const unsigned long long now = global_ns();
      tl[5] = now;
      if (it > 0) tl[3] += now - tl[6];
    }
#endif
    const int stage = it % kStages;
    const uint32_t parity = (it / kStages) & 1;
    // Which unit is next, then its staged data.  The per-unit inputs that do
    // not depend on the slot (conv weights, beta, gate parameters) are
    // usually prefetched while the previous unit computed.
    const bool have_info = mbar_wait_bounded(smem_addr(&S.ready[stage]), parity, p.wait_limit_ns);
    int n = -1, h = 0;
    bool ok = have_info;
    if (have_info) {
      n = S.info[stage][1];
      h = S.info[stage][2];
      if (n >= 0) {
        if (have_next) {
          cur = nxt;
        } else {
          cur = load_unit_inputs(p, n, h, tid, D);
        }
        have_next = false;
        ok = mbar_wait_bounded(smem_addr(&S.full[stage]), parity, p.wait_limit_ns);
      }
    }
    // All consumers agree on going on (one vote for both waits; also the
    // barrier that guards the scratch).  Without a timeout every consumer
    // has read the same info, so the end-of-work test below is uniform.
    if (consumer_any(!ok || S.abort)) {
      if (tid == 0) {
        flag_error(p, KDA_DEVERR_TIMEOUT);
        S.abort = 1;
      }
      break;
    }
#ifdef KDA_DECODE_TIMELINE
    if (tid == 0) {
      const unsigned long long now = global_ns();
      tl[6] = now;
      tl[2] += now - tl[5];
      if (it == 0) tl[1] = now;
      if (n >= 0) tl[4] += 1;
    }
#endif
    if (n < 0) break;  // no more units
    // If the next unit is already published, start loading its inputs now;
    // they arrive while this unit computes.
    {
      const int s2 = (it + 1) % kStages;
      if (mbar_try_wait(smem_addr(&S.ready[s2]), ((it + 1) / kStages) & 1)) {
        const int n2 = S.info[s2][1], h2 = S.info[s2][2];
        if (n2 >= 0) {
          nxt = load_unit_inputs(p, n2, h2, tid, D);
          have_next = true;
        }
      }
    }
    const float* wq = cur.wq;
    const float* wv = cur.wv;
    const float bq = cur.bq, bv = cur.bv, beta = cur.beta, gate_a = cur.gate_a, gate_bias = cur.gate_bias;
    const int slot = S.info[stage][0];
    uint16_t* out_row = p.out + n * p.out_stride + static_cast<int64_t>(h) * kDim;

    // Padding rows (slot <= 0) write zeros and touch no state (P1 实现拆解
    // item 1; kernel excerpt in 关键源码片段).
    if (slot <= 0 || slot >= p.num_slots) {
      if (tid < kDim * 2 / 16) reinterpret_cast<uint4*>(out_row)[tid] = make_uint4(0, 0, 0, 0);
      if (slot >= p.num_slots && tid == 0) flag_error(p, KDA_DEVERR_SLOT_RANGE);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.done[stage]));
      continue;
    }

    // This warp's 16 rows of the staged tile into registers now: the reads
    // do not depend on the conv below and overlap it.
    float4 a[kRowsPerWarp];
    {
      const float4* tile4 = reinterpret_cast<const float4*>(S.tile[stage]);
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) a[r] = tile4[(warp * kRowsPerWarp + r) * 32 + lane];
    }

    // Conv-state advance: drop the oldest tap, append the new input (a pure
    // move of bf16 bit patterns).
    if (kUpdateConv && tid < 3 * kCsU4 && p.conv_sd) {
      // tap-first: taps 0, 1 take the old taps 1, 2; tap 2 takes the input
      const int c = tid / kCsU4, e = tid - c * kCsU4, t = e >> 4, q = e & 15;
      const uint4 v = (t < kWidth - 2) ? reinterpret_cast<const uint4*>(S.cs[stage][c] + (t + 1) * kDim)[q]
                                       : reinterpret_cast<const uint4*>(S.x[stage][c])[q];
      reinterpret_cast<uint4*>(p.conv_state + (static_cast<int64_t>(slot) * (kWidth - 1) + t) * 3 * D + c * D +
                               static_cast<int64_t>(h) * kDim)[q] = v;
    } else if (kUpdateConv && tid < 3 * kCsU4) {
      const int c = tid / kCsU4, e = tid - c * kCsU4;
      uint16_t v8[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int pos = e * 8 + t, j = pos / 3, k = pos - 3 * j;
        v8[t] = (k < kWidth - 2) ? S.cs[stage][c][3 * j + k + 1] : S.x[stage][c][j];
      }
      uint4 w4;
      w4.x = v8[0] | (static_cast<uint32_t>(v8[1]) << 16);
      w4.y = v8[2] | (static_cast<uint32_t>(v8[3]) << 16);
      w4.z = v8[4] | (static_cast<uint32_t>(v8[5]) << 16);
      w4.w = v8[6] | (static_cast<uint32_t>(v8[7]) << 16);
      uint4* dst = reinterpret_cast<uint4*>(
          p.conv_state + (static_cast<int64_t>(slot) * 3 * D + c * D + static_cast<int64_t>(h) * kDim) * (kWidth - 1));
      dst[e] = w4;
    }

    // Conv (4 taps) + SiLU on the 384 q|k|v channels; decay alpha = exp(g).
    {
      const int c = tid >> 7, j = tid & (kDim - 1);
      // tap t of channel j: [j][t] (dim-first) or [t][j] (tap-first)
      const int cs_j = p.conv_sd ? 1 : kWidth - 1, cs_t = p.conv_sd ? kDim : 1;
      const uint16_t* cs = S.cs[stage][c] + cs_j * j;
      float y = bq;
      y = fmaf(wq[0], bf16_to_f32(cs[0 * cs_t]), y);
      y = fmaf(wq[1], bf16_to_f32(cs[1 * cs_t]), y);
      y = fmaf(wq[2], bf16_to_f32(cs[2 * cs_t]), y);
      y = fmaf(wq[3], bf16_to_f32(S.x[stage][c][j]), y);
      const float act = __fdividef(y, 1.0f + __expf(-y));
      (c == 0 ? S.q : S.k)[j] = act;
      if (tid < kDim) {
        const uint16_t* csv = S.cs[stage][2] + cs_j * j;
        float yv = bv;
        yv = fmaf(wv[0], bf16_to_f32(csv[0 * cs_t]), yv);
        yv = fmaf(wv[1], bf16_to_f32(csv[1 * cs_t]), yv);
        yv = fmaf(wv[2], bf16_to_f32(csv[2 * cs_t]), yv);
        yv = fmaf(wv[3], bf16_to_f32(S.x[stage][2][j]), yv);
        S.v[j] = __fdividef(yv, 1.0f + __expf(-yv));
      } else {
        float g = S.g[stage][j];
        if (p.fused_gate) {
          // Gate activation (the page's safe-gate variant; standard KDA form).
          const float z = g + gate_bias;
          if (p.lower_bound < 0.0f) {
            g = p.lower_bound / (1.0f + expf(-gate_a * z));
          } else {
            const float sp = (z > 0.0f) ? z + log1pf(expf(-z)) : log1pf(expf(z));
            g = -gate_a * sp;
          }
        }
        S.alpha[j] = expf(g);
      }
    }
    const float gate_j = (kOutNorm && tid < kDim) ? bf16_to_f32(S.gate[stage][tid]) : 0.0f;
    consumer_sync();

    // Decay the staged tile and form partial column sums over this warp's 16
    // key rows with the unnormalised q~, k~ (the L2 norms are applied to the
    // sums afterwards): u~ = A^T k~, w~ = A^T q~, A = Diag(alpha) S kept in
    // registers.
    float al_r[kRowsPerWarp], kt_r[kRowsPerWarp], qt_r[kRowsPerWarp];
#pragma unroll
    for (int r4 = 0; r4 < kRowsPerWarp / 4; ++r4) {
      const float4 al4 = reinterpret_cast<const float4*>(S.alpha + warp * kRowsPerWarp)[r4];
      const float4 kt4 = reinterpret_cast<const float4*>(S.k + warp * kRowsPerWarp)[r4];
      const float4 qt4 = reinterpret_cast<const float4*>(S.q + warp * kRowsPerWarp)[r4];
      al_r[4 * r4] = al4.x; al_r[4 * r4 + 1] = al4.y; al_r[4 * r4 + 2] = al4.z; al_r[4 * r4 + 3] = al4.w;
      kt_r[4 * r4] = kt4.x; kt_r[4 * r4 + 1] = kt4.y; kt_r[4 * r4 + 2] = kt4.z; kt_r[4 * r4 + 3] = kt4.w;
      qt_r[4 * r4] = qt4.x; qt_r[4 * r4 + 1] = qt4.y; qt_r[4 * r4 + 2] = qt4.z; qt_r[4 * r4 + 3] = qt4.w;
    }
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f), w = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const float al = al_r[r], kt = kt_r[r], qt = qt_r[r];
      a[r].x *= al; a[r].y *= al; a[r].z *= al; a[r].w *= al;
      u.x = fmaf(kt, a[r].x, u.x); u.y = fmaf(kt, a[r].y, u.y);
      u.z = fmaf(kt, a[r].z, u.z); u.w = fmaf(kt, a[r].w, u.w);
      w.x = fmaf(qt, a[r].x, w.x); w.y = fmaf(qt, a[r].y, w.y);
      w.z = fmaf(qt, a[r].z, w.z); w.w = fmaf(qt, a[r].w, w.w);
    }
    reinterpret_cast<float4*>(S.red[0][warp])[lane] = u;
    reinterpret_cast<float4*>(S.red[1][warp])[lane] = w;
    // The warp's share of |q~|^2, |k~|^2 and q~.k~ over its 16 key rows, from
    // the rows every lane already holds.  The three sums run in the same
    // order, so q~.k~ equals |k~|^2 bit for bit whenever q~ equals k~.
    {
      float pqq = 0.0f, pkk = 0.0f, pqk = 0.0f;
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        pqq = fmaf(qt_r[r], qt_r[r], pqq);
        pkk = fmaf(kt_r[r], kt_r[r], pkk);
        pqk = fmaf(qt_r[r], kt_r[r], pqk);
      }
      if (lane == 0) S.part[warp] = make_float4(pqq, pkk, pqk, 0.0f);
    }
    consumer_sync();

    // L2 norms: q^ = rq q~, k^ = rk k~, and with u~ = A^T k~, w~ = A^T q~:
    // delta = beta (v - rk u~).  The readout of the updated state,
    // o = S'^T q^ = rq w~ + (q^.k^) delta, is evaluated without a second pass
    // over S' and rearranged so that its one cancellation happens inside a
    // single fused multiply-add:
    //   o = rq ((w~ - u~) + m u~) + beta (q^.k^) v,
    //   m = 1 - beta (q~.k~) rk^2 = (|k~|^2 + 1e-6 - beta q~.k~) rk^2.
    // When q~ is parallel to k~ and beta = 1, |o| can be far below |w|; the
    // plain sum w + (q^.k^) delta would then carry an fp32 rounding error of
    // the size of |w|.
    float o = 0.0f;
    if (tid < kDim) {
      // the eight warps' partials, summed by an 8-lane butterfly
      const float4 pr = S.part[lane & (kConsumerWarps - 1)];
      float ssq = pr.x, ssk = pr.y, sqk = pr.z;
#pragma unroll
      for (int off = kConsumerWarps / 2; off > 0; off >>= 1) {
        ssq += __shfl_xor_sync(0xffffffffu, ssq, off);
        ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
        sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
      }
      const float rq = scale * rsqrtf(ssq + 1e-6f);
      const float rk = rsqrtf(ssk + 1e-6f);
      float ut = 0.0f, wt = 0.0f;
#pragma unroll
      for (int r = 0; r < kConsumerWarps; ++r) {
        ut += S.red[0][r][tid];
        wt += S.red[1][r][tid];
      }
      const float vj = S.v[tid];
      const float dj = beta * (vj - rk * ut);
      S.delta[tid] = rk * dj;  // pass 2 adds k~ (rk delta)^T = k^ delta^T
      const float m = (fmaf(-beta, sqk, ssk) + 1e-6f) * (rk * rk);
      const float bqk = beta * sqk * rq * rk;  // beta (q^ . k^)
      o = fmaf(bqk, vj, rq * fmaf(m, ut, wt - ut));
      if (kOutNorm) {
        const float so = warp_sum(o * o);
        if (lane == 0) S.osum[warp] = so;
      }
    }
    consumer_sync();

    // S' = A + k^ delta^T written back into the stage, then handed to the
    // producer for the bulk store.
    const float4 d = reinterpret_cast<const float4*>(S.delta)[lane];
    float4* tile4w = reinterpret_cast<float4*>(S.tile[stage]);
#pragma unroll
    for (int r4 = 0; r4 < kRowsPerWarp / 4; ++r4) {
      const float4 kt4 = reinterpret_cast<const float4*>(S.k + warp * kRowsPerWarp)[r4];
      const float kt_4[4] = {kt4.x, kt4.y, kt4.z, kt4.w};
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const int r = 4 * r4 + i4, i = warp * kRowsPerWarp + r;
        const float kt = kt_4[i4];
        a[r].x = fmaf(kt, d.x, a[r].x); a[r].y = fmaf(kt, d.y, a[r].y);
        a[r].z = fmaf(kt, d.z, a[r].z); a[r].w = fmaf(kt, d.w, a[r].w);
        tile4w[i * 32 + lane] = a[r];
      }
    }
    fence_proxy_async_smem();  // generic-proxy writes before the async-proxy store
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&S.done[stage]));

    // Gated RMSNorm epilogue (or the raw readout) to bf16; the sum of o_j^2
    // is taken from o itself.
    if (tid < kDim) {
      float y = o;
      if (kOutNorm) {
        const float ss = (S.osum[0] + S.osum[1]) + (S.osum[2] + S.osum[3]);
        const float rr = rsqrtf(ss * (1.0f / kDim) + p.eps);
        y = o * rr * nw * __fdividef(1.0f, 1.0f + __expf(-gate_j));
      }
      out_row[tid] = f32_to_bf16(y);
    }
  }
#ifdef KDA_DECODE_TIMELINE
  if (tid == 0) {
    const unsigned long long te = global_ns();
    unsigned int smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const unsigned int i = atomicAdd(&g_timeline_n, 1u);
    if (i < kTimelineMax) {
      g_timeline[i][0] = blockIdx.x; g_timeline[i][1] = smid; g_timeline[i][2] = tl[0]; g_timeline[i][3] = tl[1];
      g_timeline[i][4] = te; g_timeline[i][5] = tl[4]; g_timeline[i][6] = tl[3]; g_timeline[i][7] = tl[2];
    }
  }
#endif
}

}  // namespace
