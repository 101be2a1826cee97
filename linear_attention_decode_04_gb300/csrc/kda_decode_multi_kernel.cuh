// kda_decode_multi_kernel.cuh -- device code of the multi-token
// (speculative) decode step (sm_103a).  Included once, by kda_decode.cu,
// after kda_decode_kernel.cuh, whose constants, parameter block and PTX
// wrappers it uses.
//
// A unit is one (sequence n, head h) with T = 1 + num_spec tokens.  Its
// source state tile (64 KiB) and conv window are streamed in once; the state
// then stays in the consumers' registers from token to token (after a
// token's rank-1 update the registers hold exactly the state the next token
// decays), and after every present token the updated tile is written into
// the stage and bulk-stored to that token's destination slot, the window
// likewise.  Per unit: 64 KiB read, 64 KiB written per present token.
#pragma once

#include "kda_decode_kernel.cuh"

namespace {

// Global -> shared bulk copy without a cache hint (data every CTA reuses).
__device__ __forceinline__ void bulk_load_plain(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

constexpr int kMaxT = KDA_MAX_TOKENS_PER_SEQ;
constexpr int kMStages = 2;           // units in flight per CTA (one computing, one loading)
constexpr int kMInfo = 4 + kMaxT;     // src, n (-1: no more units), h, withheld, dst[kMaxT]

// Dynamic shared memory of one CTA (about 188 KB).
struct __align__(128) MSmem {
  float tile[kMStages][kDim * kDim];
  uint16_t cs[kMStages][2][3][kDim * (kWidth - 1)];  // the sliding window (two buffers), in the pool's layout
  float w[kMStages][3][kWidth][kDim];  // the head's conv taps
  float b[kMStages][3][kDim];          // and conv bias (zero without one)
  uint16_t x[kMStages][kMaxT][3][kDim];
  float g[kMStages][kMaxT][kDim];
  uint16_t gate[kMStages][kMaxT][kDim];
  float q[kDim], v[kDim], alpha[kDim];
  float k[2][kDim];  // by token parity: the rank-1 update of a token reads its k~ while the next token's is written
  float red[2][kConsumerWarps][kDim];
  float delta[kDim];
  float4 part[kConsumerWarps];
  float osum[4];
  int info[kMStages][kMInfo];
  unsigned long long ready[kMStages];    // info of the stage is written (producer)
  unsigned long long full[kMStages];     // the unit's inputs have landed (producer + tx bytes)
  unsigned long long done[kMStages];     // the consumers are finished with the unit (8 warps)
  unsigned long long written[kMStages];  // a token's updated tile is in the stage (8 warps)
  unsigned long long freed[kMStages];    // the store of that tile has read it out (producer)
  volatile int abort;
};

template <bool kOutNorm, bool kUpdateConv>
__global__ void __launch_bounds__(kThreads, 1) kda_decode_multi_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  MSmem& S = *reinterpret_cast<MSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int T = p.T;
  const int64_t D = static_cast<int64_t>(p.H) * kDim;

  if (tid == 0) {
    for (int s = 0; s < kMStages; ++s) {
      mbar_init(smem_addr(&S.ready[s]), 1);
      mbar_init(smem_addr(&S.full[s]), 1);
      mbar_init(smem_addr(&S.done[s]), kConsumerWarps);
      mbar_init(smem_addr(&S.written[s]), kConsumerWarps);
      mbar_init(smem_addr(&S.freed[s]), 1);
    }
    S.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  __syncthreads();
  griddep_launch_dependents();

  auto valid = [&](int slot) { return slot > 0 && slot < p.num_slots; };

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const uint64_t policy = l2_evict_first_policy();
    int k_static = 0;
    bool queue_done = false;
    // This CTA draws no more units: the last CTA to do so returns the work
    // queue to zero for the next call.
    auto finish_queue = [&]() {
      if (queue_done) return;
      queue_done = true;
      if (p.queue != nullptr) {
        __threadfence();
        if (atomicAdd(p.queue + 1, 1) == G - 1) {
          atomicExch(p.queue, 0);
          atomicExch(p.queue + 1, 0);
        }
      }
    };
    auto next_unit = [&]() -> int {
      int u;
      if (k_static < kMStages || p.queue == nullptr)
        u = blockIdx.x + (k_static++) * G;
      else
        u = kMStages * G + atomicAdd(p.queue, 1);
      if (u >= p.total_units) {
        finish_queue();
        return -1;
      }
      return u;
    };
    // The unit's slots: source, then the destination of every token.
    auto set_info = [&](int st, int u) {
      const int n = u / p.H, h = u - n * p.H;
      S.info[st][1] = n;
      S.info[st][2] = h;
      S.info[st][3] = (u == p.withhold_unit);
      const int32_t* row = p.slot_idx + static_cast<int64_t>(n) * T;
      S.info[st][0] = p.src_slot ? __ldg(p.src_slot + n) : __ldg(row);
      for (int t = 0; t < T; ++t) S.info[st][4 + t] = __ldg(row + t);
    };
    auto n_present = [&](int st) {
      int c = 0;
      for (int t = 0; t < T; ++t) c += valid(S.info[st][4 + t]);
      return c;
    };
    auto active = [&](int st) { return valid(S.info[st][0]) && n_present(st) > 0; };
    const uint32_t tok_bytes = 3 * kXSliceBytes + kDim * 4 + (kOutNorm ? kXSliceBytes : 0);
    const uint32_t head_bytes = 3 * kWidth * kDim * 4 + (p.conv_b ? 3 * kDim * 4 : 0);
    auto unit_bytes = [&](int st) {
      return kTileBytes + 3 * kCsSliceBytes + head_bytes + tok_bytes * n_present(st);
    };
    // The source tile and window.
    auto load_src = [&](int st) {
      const int h = S.info[st][2], src = S.info[st][0];
      const uint32_t full = smem_addr(&S.full[st]);
      bulk_load(smem_addr(S.tile[st]), p.state + (static_cast<int64_t>(src) * p.H + h) * (kDim * kDim), kTileBytes,
                full, policy);
      // the head's conv taps and bias (L2-resident, shared by all sequences)
      for (int c = 0; c < 3; ++c) {
        for (int k = 0; k < kWidth; ++k)
          bulk_load_plain(smem_addr(S.w[st][c][k]), p.conv_w + (c * kWidth + k) * D + static_cast<int64_t>(h) * kDim,
                          kDim * 4, full);
        if (p.conv_b)
          bulk_load_plain(smem_addr(S.b[st][c]), p.conv_b + c * D + static_cast<int64_t>(h) * kDim, kDim * 4, full);
      }
      for (int c = 0; c < 3; ++c) {
        if (!p.conv_sd) {
          bulk_load(smem_addr(S.cs[st][0][c]),
                    p.conv_state +
                        (static_cast<int64_t>(src) * 3 * D + c * D + static_cast<int64_t>(h) * kDim) * (kWidth - 1),
                    kCsSliceBytes, full, policy);
        } else {
          for (int k = 0; k < kWidth - 1; ++k)
            bulk_load(smem_addr(S.cs[st][0][c] + k * kDim),
                      p.conv_state + (static_cast<int64_t>(src) * (kWidth - 1) + k) * 3 * D + c * D +
                          static_cast<int64_t>(h) * kDim,
                      kXSliceBytes, full, policy);
        }
      }
    };
    // The per-token inputs of the present tokens.
    auto load_tokens = [&](int st) {
      const int n = S.info[st][1], h = S.info[st][2];
      const uint32_t full = smem_addr(&S.full[st]);
      for (int t = 0; t < T; ++t) {
        if (!valid(S.info[st][4 + t])) continue;
        const int64_t row = static_cast<int64_t>(n) * T + t;
        for (int c = 0; c < 3; ++c)
          bulk_load(smem_addr(S.x[st][t][c]), p.qkv + row * p.qkv_stride + c * D + static_cast<int64_t>(h) * kDim,
                    kXSliceBytes, full, policy);
        bulk_load(smem_addr(S.g[st][t]), p.g + (row * p.H + h) * kDim, kDim * 4, full, policy);
        if (kOutNorm)
          bulk_load(smem_addr(S.gate[st][t]), p.gate + row * p.gate_stride + static_cast<int64_t>(h) * kDim,
                    kXSliceBytes, full, policy);
      }
    };
    // Publish a unit into a stage (info, then ready) and stream its inputs.
    bool sentinel = false;
    int pubs[kMStages] = {0, 0};  // phases of each stage's `full` barrier started so far
    auto publish = [&](int st, int u, bool info_set, bool src_armed) {
      if (!info_set) set_info(st, u);
      const bool act = active(st), held = S.info[st][3] != 0;
      if (!held) ++pubs[st];
      if (act && !held && !src_armed) {
        mbar_arrive_expect_tx(smem_addr(&S.full[st]), unit_bytes(st));
        load_src(st);
      }
      mbar_arrive(smem_addr(&S.ready[st]));
      if (held) return;  // wait-path test: never signalled
      if (act)
        load_tokens(st);
      else
        mbar_arrive(smem_addr(&S.full[st]));  // padding sequence or no present token
    };
    auto publish_end = [&](int st) {
      S.info[st][1] = -1;
      mbar_arrive(smem_addr(&S.ready[st]));
      sentinel = true;
    };

    // Ring fill.  With KDA_EARLY_PREFETCH the first unit's slots are read and
    // its source streams in before the previous kernel in the stream has
    // completed (the caller guarantees that kernel writes none of slot_idx,
    // src_slot, state and conv_state); per-token inputs wait for it.
    int units[kMStages];
    for (int st = 0; st < kMStages; ++st) units[st] = next_unit();
    bool early = false;
    if (p.early_prefetch && units[0] >= 0) {
      set_info(0, units[0]);
      if (active(0) && !S.info[0][3]) {
        mbar_arrive_expect_tx(smem_addr(&S.full[0]), unit_bytes(0));
        load_src(0);
      }
      early = true;
    }
    griddep_wait();
    for (int st = 0; st < kMStages; ++st) {
      if (units[st] >= 0)
        publish(st, units[st], st == 0 && early, st == 0 && early);
      else if (!sentinel)
        publish_end(st);
    }

    // Steady state: store each token's tile as the consumers hand it over,
    // then refill the stage with the unit after next.
    uint32_t wpar[kMStages] = {0u, 0u};
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int st = it % kMStages;
      if (units[st] < 0) break;  // the end-of-work sentinel (or nothing) is here
      if (active(st) && !S.info[st][3]) {
        const int h = S.info[st][2];
        for (int t = 0; t < T; ++t) {
          const int dst = S.info[st][4 + t];
          if (!valid(dst)) continue;
          ok = mbar_wait_bounded(smem_addr(&S.written[st]), wpar[st] & 1u, p.wait_limit_ns);
          if (!ok) break;
          ++wpar[st];
          bulk_store(p.state + (static_cast<int64_t>(dst) * p.H + h) * (kDim * kDim), smem_addr(S.tile[st]),
                     kTileBytes, policy);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(smem_addr(&S.freed[st]));
        }
      }
      if (!ok) break;
      ok = mbar_wait_bounded(smem_addr(&S.done[st]), (it / kMStages) & 1, p.wait_limit_ns);
      if (!ok) break;
      const int u = sentinel ? -1 : next_unit();
      units[st] = u;
      if (u >= 0)
        publish(st, u, false, false);
      else if (!sentinel)
        publish_end(st);
    }
    finish_queue();
    if (!ok) {
      flag_error(p, KDA_DEVERR_TIMEOUT);
      S.abort = 1;
      // Before the CTA's shared memory goes away: every load this thread
      // armed has landed (normally long since).
      for (int st = 0; st < kMStages; ++st) {
        if (pubs[st] > 0 &&
            !mbar_wait_bounded(smem_addr(&S.full[st]), (pubs[st] - 1) & 1, p.wait_limit_ns))
          flag_error(p, KDA_DEVERR_TIMEOUT);
      }
    }
    bulk_wait_all();
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();
  const float scale = (p.q_scale != 0.0f) ? p.q_scale : 0.088388347648318440550f;  // 1/sqrt(128)
  const float nw = (kOutNorm && tid < kDim) ? __ldg(p.norm_w + tid) : 0.0f;
  uint32_t wcnt0 = 0u, wcnt1 = 0u;  // updated tiles written into stage 0 / 1 so far
  for (int it = 0;; ++it) {
    const int st = it % kMStages;
    const uint32_t parity = (it / kMStages) & 1;
    const bool have_info = mbar_wait_bounded(smem_addr(&S.ready[st]), parity, p.wait_limit_ns);
    int n = -1, h = 0;
    bool ok = have_info;
    float gate_a = 0.0f, gate_bias = 0.0f;  // fused-gate parameters of key channel tid - 128
    if (have_info) {
      n = S.info[st][1];
      h = S.info[st][2];
      if (n >= 0) {
        if (p.fused_gate && tid >= kDim) {
          gate_a = expf(__ldg(p.A_log + h));
          if (p.dt_bias) gate_bias = __ldg(p.dt_bias + static_cast<int64_t>(h) * kDim + (tid - kDim));
        }
        ok = mbar_wait_bounded(smem_addr(&S.full[st]), parity, p.wait_limit_ns);
      }
    }
    if (consumer_any(!ok || S.abort)) {
      if (tid == 0) {
        flag_error(p, KDA_DEVERR_TIMEOUT);
        S.abort = 1;
      }
      break;
    }
    if (n < 0) break;  // no more units
    const int src = S.info[st][0];
    const bool src_ok = valid(src);
    if (src >= p.num_slots && tid == 0) flag_error(p, KDA_DEVERR_SLOT_RANGE);
    bool aborted = false;
    int wb = 0;  // window buffer holding the current window
    for (int t = 0; t < T; ++t) {
      const int dst = S.info[st][4 + t];
      const int64_t row = static_cast<int64_t>(n) * T + t;
      uint16_t* out_row = p.out + row * p.out_stride + static_cast<int64_t>(h) * kDim;
      // Padding sequence or absent token: zero output, no state.
      if (!src_ok || !valid(dst)) {
        if (tid < kDim * 2 / 16) reinterpret_cast<uint4*>(out_row)[tid] = make_uint4(0, 0, 0, 0);
        if (src_ok && dst >= p.num_slots && tid == 0) flag_error(p, KDA_DEVERR_SLOT_RANGE);
        continue;
      }
      const int kb = wb;  // k~ buffer of this token
      float beta = 0.0f;
      if (tid < kDim) {
        const float b = bf16_to_f32(__ldg(p.beta + row * p.H + h));
        beta = p.fused_gate ? 1.0f / (1.0f + expf(-b)) : b;
      }
      // The window after this token (oldest tap dropped, the input appended;
      // bit patterns) goes into the other window buffer and, with the flag,
      // to this token's destination slot.
      if (tid < 3 * kCsU4) {
        const int c = tid / kCsU4, e = tid - c * kCsU4;
        const uint16_t* cw = S.cs[st][wb][c];
        uint4 wnew;
        if (p.conv_sd) {
          const int k = e >> 4, q = e & 15;
          wnew = (k < kWidth - 2) ? reinterpret_cast<const uint4*>(cw + (k + 1) * kDim)[q]
                                  : reinterpret_cast<const uint4*>(S.x[st][t][c])[q];
        } else {
          uint16_t v8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int pos = e * 8 + i, j = pos / 3, k = pos - 3 * j;
            v8[i] = (k < kWidth - 2) ? cw[3 * j + k + 1] : S.x[st][t][c][j];
          }
          wnew.x = v8[0] | (static_cast<uint32_t>(v8[1]) << 16);
          wnew.y = v8[2] | (static_cast<uint32_t>(v8[3]) << 16);
          wnew.z = v8[4] | (static_cast<uint32_t>(v8[5]) << 16);
          wnew.w = v8[6] | (static_cast<uint32_t>(v8[7]) << 16);
        }
        reinterpret_cast<uint4*>(S.cs[st][wb ^ 1][c])[e] = wnew;
        if (kUpdateConv) {
          uint4* dstp;
          if (p.conv_sd) {
            const int k = e >> 4, q = e & 15;
            dstp = reinterpret_cast<uint4*>(p.conv_state + (static_cast<int64_t>(dst) * (kWidth - 1) + k) * 3 * D +
                                            c * D + static_cast<int64_t>(h) * kDim) + q;
          } else {
            dstp = reinterpret_cast<uint4*>(
                       p.conv_state +
                       (static_cast<int64_t>(dst) * 3 * D + c * D + static_cast<int64_t>(h) * kDim) * (kWidth - 1)) + e;
          }
          *dstp = wnew;
        }
      }
      // Conv (4 taps) + SiLU on the 384 q|k|v channels; decay alpha = exp(g).
      {
        const int c = tid >> 7, j = tid & (kDim - 1);
        const int cs_j = p.conv_sd ? 1 : kWidth - 1, cs_t = p.conv_sd ? kDim : 1;
        const uint16_t* cs = S.cs[st][wb][c] + cs_j * j;
        float y = p.conv_b ? S.b[st][c][j] : 0.0f;
        y = fmaf(S.w[st][c][0][j], bf16_to_f32(cs[0 * cs_t]), y);
        y = fmaf(S.w[st][c][1][j], bf16_to_f32(cs[1 * cs_t]), y);
        y = fmaf(S.w[st][c][2][j], bf16_to_f32(cs[2 * cs_t]), y);
        y = fmaf(S.w[st][c][3][j], bf16_to_f32(S.x[st][t][c][j]), y);
        (c == 0 ? S.q : S.k[kb])[j] = y / (1.0f + expf(-y));
        if (tid < kDim) {
          const uint16_t* csv = S.cs[st][wb][2] + cs_j * j;
          float yv = p.conv_b ? S.b[st][2][j] : 0.0f;
          yv = fmaf(S.w[st][2][0][j], bf16_to_f32(csv[0 * cs_t]), yv);
          yv = fmaf(S.w[st][2][1][j], bf16_to_f32(csv[1 * cs_t]), yv);
          yv = fmaf(S.w[st][2][2][j], bf16_to_f32(csv[2 * cs_t]), yv);
          yv = fmaf(S.w[st][2][3][j], bf16_to_f32(S.x[st][t][2][j]), yv);
          S.v[j] = yv / (1.0f + expf(-yv));
        } else {
          float g = S.g[st][t][j];
          if (p.fused_gate) {
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
      const float gate_j = (kOutNorm && tid < kDim) ? bf16_to_f32(S.gate[st][t][tid]) : 0.0f;
      consumer_sync();
      wb ^= 1;

      // Decay and partial column sums over this warp's 16 key rows of the
      // stage tile: the source state for the first present token, afterwards
      // the state the previous token wrote there (each warp reads back only
      // rows it wrote itself; the store engine only reads them).
      float4 a[kRowsPerWarp];
      {
        const float4* tile4 = reinterpret_cast<const float4*>(S.tile[st]);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) a[r] = tile4[(warp * kRowsPerWarp + r) * 32 + lane];
      }
      // alpha, k~, q~ of the warp's rows as float4 broadcasts, four rows at a time
      float4 u = make_float4(0.f, 0.f, 0.f, 0.f), w = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r4 = 0; r4 < kRowsPerWarp / 4; ++r4) {
        const float4 al4 = reinterpret_cast<const float4*>(S.alpha + warp * kRowsPerWarp)[r4];
        const float4 kt4 = reinterpret_cast<const float4*>(S.k[kb] + warp * kRowsPerWarp)[r4];
        const float4 qt4 = reinterpret_cast<const float4*>(S.q + warp * kRowsPerWarp)[r4];
        const float al_4[4] = {al4.x, al4.y, al4.z, al4.w};
        const float kt_4[4] = {kt4.x, kt4.y, kt4.z, kt4.w};
        const float qt_4[4] = {qt4.x, qt4.y, qt4.z, qt4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * r4 + i;
          const float al = al_4[i], kt = kt_4[i], qt = qt_4[i];
          a[r].x *= al; a[r].y *= al; a[r].z *= al; a[r].w *= al;
          u.x = fmaf(kt, a[r].x, u.x); u.y = fmaf(kt, a[r].y, u.y);
          u.z = fmaf(kt, a[r].z, u.z); u.w = fmaf(kt, a[r].w, u.w);
          w.x = fmaf(qt, a[r].x, w.x); w.y = fmaf(qt, a[r].y, w.y);
          w.z = fmaf(qt, a[r].z, w.z); w.w = fmaf(qt, a[r].w, w.w);
        }
      }
      reinterpret_cast<float4*>(S.red[0][warp])[lane] = u;
      reinterpret_cast<float4*>(S.red[1][warp])[lane] = w;
      {
        const int i = warp * kRowsPerWarp + (lane & (kRowsPerWarp - 1));
        const float qi = S.q[i], ki = S.k[kb][i];
        float pqq = qi * qi, pkk = ki * ki, pqk = qi * ki;
#pragma unroll
        for (int off = kRowsPerWarp / 2; off > 0; off >>= 1) {
          pqq += __shfl_xor_sync(0xffffffffu, pqq, off);
          pkk += __shfl_xor_sync(0xffffffffu, pkk, off);
          pqk += __shfl_xor_sync(0xffffffffu, pqk, off);
        }
        if (lane == 0) S.part[warp] = make_float4(pqq, pkk, pqk, 0.0f);
      }
      consumer_sync();

      // delta and the readout, in the decode step's cancellation-safe form.
      float o = 0.0f;
      if (tid < kDim) {
        const float4 pr = S.part[lane & (kConsumerWarps - 1)];
        float ssq = pr.x, ssk = pr.y, sqk = pr.z;
#pragma unroll
        for (int off = kConsumerWarps / 2; off > 0; off >>= 1) {
          ssq += __shfl_xor_sync(0xffffffffu, ssq, off);
          ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
          sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
        }
        const float rq = scale / sqrtf(ssq + 1e-6f);
        const float rk = 1.0f / sqrtf(ssk + 1e-6f);
        float ut = 0.0f, wt = 0.0f;
#pragma unroll
        for (int r = 0; r < kConsumerWarps; ++r) {
          ut += S.red[0][r][tid];
          wt += S.red[1][r][tid];
        }
        const float vj = S.v[tid];
        const float dj = beta * (vj - rk * ut);
        S.delta[tid] = rk * dj;
        const float m = (fmaf(-beta, sqk, ssk) + 1e-6f) * (rk * rk);
        const float bqk = beta * sqk * rq * rk;
        o = fmaf(bqk, vj, rq * fmaf(m, ut, wt - ut));
        if (kOutNorm) {
          const float so = warp_sum(o * o);
          if (lane == 0) S.osum[warp] = so;
        }
      }
      // The stage tile may be rewritten once the store of the tile written
      // before it has read it out; every consumer agrees before going on
      // (this vote is also the barrier that publishes delta).
      const uint32_t wc = st ? wcnt1 : wcnt0;
      bool fok = true;
      if (wc > 0) fok = mbar_wait_bounded(smem_addr(&S.freed[st]), (wc - 1) & 1u, p.wait_limit_ns);
      if (consumer_any(!fok || S.abort)) {
        if (tid == 0) {
          flag_error(p, KDA_DEVERR_TIMEOUT);
          S.abort = 1;
        }
        aborted = true;
        break;
      }

      // S' = A + k^ delta^T, written into the stage for the bulk store to this
      // token's slot (and for the next token).
      const float4 d = reinterpret_cast<const float4*>(S.delta)[lane];
      float4* tile4w = reinterpret_cast<float4*>(S.tile[st]);
#pragma unroll
      for (int r4 = 0; r4 < kRowsPerWarp / 4; ++r4) {
        const float4 kt4 = reinterpret_cast<const float4*>(S.k[kb] + warp * kRowsPerWarp)[r4];
        const float kt_4[4] = {kt4.x, kt4.y, kt4.z, kt4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * r4 + i;
          const float kt = kt_4[i];
          a[r].x = fmaf(kt, d.x, a[r].x); a[r].y = fmaf(kt, d.y, a[r].y);
          a[r].z = fmaf(kt, d.z, a[r].z); a[r].w = fmaf(kt, d.w, a[r].w);
          tile4w[(warp * kRowsPerWarp + r) * 32 + lane] = a[r];
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.written[st]));
      if (st) ++wcnt1; else ++wcnt0;

      if (tid < kDim) {
        float y = o;
        if (kOutNorm) {
          const float ss = (S.osum[0] + S.osum[1]) + (S.osum[2] + S.osum[3]);
          const float rr = 1.0f / sqrtf(ss * (1.0f / kDim) + p.eps);
          y = o * rr * nw * (1.0f / (1.0f + expf(-gate_j)));
        }
        out_row[tid] = f32_to_bf16(y);
      }
    }
    if (aborted) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&S.done[st]));
  }
}

}  // namespace
