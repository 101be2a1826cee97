// kda_decode_multi_kernel.cuh -- device code of the multi-token
// (speculative) decode step (sm_103a).  Included once, by kda_decode.cu,
// after kda_decode_kernel.cuh, whose constants, parameter block and PTX
// wrappers it uses.
//
// A unit is one (sequence n, head h) with T = 1 + num_spec tokens.  Its
// source state tile (64 KiB) and conv window are streamed in once.  The
// consumers first do everything that does not depend on the state for all
// present tokens at once (conv + SiLU, decays, L2 norms, the window after
// every token, stored straight to that token's slot), then run the
// recurrence token by token with the state in registers: one pass over the
// registers applies token m-1's rank-1 update, writes that state into the
// stage for the bulk store to token m-1's slot, and applies token m's decay
// and matvecs.  Per unit: 64 KiB read, 64 KiB written per present token.
#pragma once

#include "kda_decode_kernel.cuh"

namespace {

constexpr int kMaxT = KDA_MAX_TOKENS_PER_SEQ;
constexpr int kMStages = 2;           // units in flight per CTA (one computing, one loading)
// per-stage info: src, n (-1: no more units), h, withheld, dst[kMaxT],
// number of present tokens, present token indices[kMaxT]
constexpr int kMInfo = 5 + 2 * kMaxT;
constexpr int kMiDst = 4, kMiNp = 4 + kMaxT, kMiPt = 5 + kMaxT;

// Dynamic shared memory of one CTA for up to kTMax tokens per sequence.
// With kTMax <= 4 a spare tile gives every unit two output buffers: present
// token m's state goes to the stage tile (m even) or the spare (m odd), so
// the store of one token's tile runs while the next token's is written
// (about 225 KB).  With more tokens per sequence only the stage tile is
// used (about 186 KB).
template <int kTMax>
struct __align__(128) MSmemT {
  static constexpr int kOutBufs = kTMax <= 4 ? 2 : 1;
  static constexpr int kTiles = kMStages + kOutBufs - 1;  // stage tiles [0, 1], spare [2]
  float tile[kTiles][kDim * kDim];
  uint16_t cs[kMStages][3][kDim * (kWidth - 1)];  // the source window, in the pool's layout
  uint16_t x[kMStages][kTMax][3][kDim];
  float g[kMStages][kTMax][kDim];
  uint16_t gate[kMStages][kTMax][kDim];
  // per present token m of the unit being computed
  float q[kTMax][kDim], k[kTMax][kDim], v[kTMax][kDim], alpha[kTMax][kDim];
  float4 coef[kTMax];  // rq, rk, m = (|k~|^2 + 1e-6 - beta q~.k~) rk^2, beta (q^.k^)
  float beta[kTMax];
  float red[2][kConsumerWarps][kDim];
  float delta[kDim];
  float osum[4];
  int info[kMStages][kMInfo];
  unsigned long long ready[kMStages];   // info of the stage is written (producer)
  unsigned long long full[kMStages];    // the unit's inputs have landed (producer + tx bytes)
  unsigned long long done[kMStages];    // the consumers are finished with the unit (8 warps)
  unsigned long long written[kTiles];   // a token's updated state is in the tile (8 warps)
  unsigned long long freed[kTiles];     // the store of that tile has read it out (producer)
  volatile int abort;
};

// Wait until at most N of this thread's most recent bulk store groups are
// still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read_pending() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <bool kOutNorm, bool kUpdateConv, int kTMax>
__global__ void __launch_bounds__(kThreads, 1) kda_decode_multi_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  using MSmem = MSmemT<kTMax>;
  constexpr int kOutBufs = MSmem::kOutBufs, kTiles = MSmem::kTiles;
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
    }
    for (int b = 0; b < kTiles; ++b) {
      mbar_init(smem_addr(&S.written[b]), kConsumerWarps);
      mbar_init(smem_addr(&S.freed[b]), 1);
    }
    S.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  __syncthreads();
  griddep_launch_dependents();

  auto valid = [&](int slot) { return slot > 0 && slot < p.num_slots; };
  // output buffer of present token m of a unit in stage st
  auto out_buf = [&](int st, int m) { return (kOutBufs == 2 && (m & 1)) ? kMStages : st; };

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
      if (k_static < p.static_units || p.queue == nullptr)
        u = blockIdx.x + (k_static++) * G;
      else
        u = p.static_units * G + atomicAdd(p.queue, 1);
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
      int np = 0;
      for (int t = 0; t < T; ++t) {
        const int dst = __ldg(row + t);
        S.info[st][kMiDst + t] = dst;
        if (valid(dst)) S.info[st][kMiPt + np++] = t;
      }
      S.info[st][kMiNp] = np;
    };
    auto n_present = [&](int st) { return S.info[st][kMiNp]; };
    auto active = [&](int st) { return valid(S.info[st][0]) && n_present(st) > 0; };
    const uint32_t tok_bytes = 3 * kXSliceBytes + kDim * 4 + (kOutNorm ? kXSliceBytes : 0);
    auto unit_bytes = [&](int st) { return kTileBytes + 3 * kCsSliceBytes + tok_bytes * n_present(st); };
    // The source tile and window.
    auto load_src = [&](int st) {
      const int h = S.info[st][2], src = S.info[st][0];
      const uint32_t full = smem_addr(&S.full[st]);
      bulk_load(smem_addr(S.tile[st]), p.state + (static_cast<int64_t>(src) * p.H + h) * (kDim * kDim), kTileBytes,
                full, policy);
      for (int c = 0; c < 3; ++c) {
        if (!p.conv_sd) {
          bulk_load(smem_addr(S.cs[st][c]),
                    p.conv_state +
                        (static_cast<int64_t>(src) * 3 * D + c * D + static_cast<int64_t>(h) * kDim) * (kWidth - 1),
                    kCsSliceBytes, full, policy);
        } else {
          for (int k = 0; k < kWidth - 1; ++k)
            bulk_load(smem_addr(S.cs[st][c] + k * kDim),
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
      for (int m = 0; m < n_present(st); ++m) {
        const int t = S.info[st][kMiPt + m];
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
    uint32_t wpar0 = 0u, wpar1 = 0u, wpar2 = 0u;  // writes seen per output buffer
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int st = it % kMStages;
      if (units[st] < 0) break;  // the end-of-work sentinel (or nothing) is here
      if (active(st) && !S.info[st][3]) {
        const int h = S.info[st][2];
        int pending = -1;  // buffer of the issued store not yet known to have read its tile
        for (int m = 0; m < n_present(st); ++m) {
          const int dst = S.info[st][kMiDst + S.info[st][kMiPt + m]];
          const int b = out_buf(st, m);
          uint32_t& wp = (b == 0) ? wpar0 : (b == 1) ? wpar1 : wpar2;
          ok = mbar_wait_bounded(smem_addr(&S.written[b]), wp & 1u, p.wait_limit_ns);
          if (!ok) break;
          ++wp;
          bulk_store(p.state + (static_cast<int64_t>(dst) * p.H + h) * (kDim * kDim), smem_addr(S.tile[b]),
                     kTileBytes, policy);
          bulk_commit();
          // with two output buffers the previous store may finish reading
          // while this one starts; with one, each must finish first
          if (kOutBufs == 2) {
            if (pending >= 0) {
              bulk_wait_read_pending<1>();
              mbar_arrive(smem_addr(&S.freed[pending]));
            }
            pending = b;
          } else {
            bulk_wait_read_all();
            mbar_arrive(smem_addr(&S.freed[b]));
          }
        }
        if (pending >= 0) {
          bulk_wait_read_all();
          mbar_arrive(smem_addr(&S.freed[pending]));
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
  uint32_t wcnt0 = 0u, wcnt1 = 0u, wcnt2 = 0u;  // states written into each output buffer so far
  // Conv taps of this thread's channels (q or k channel tid, v channel tid
  // for tid < 128) and the gate parameters of key channel tid - 128, for the
  // head in w_head.  When the next unit is already published they are
  // loaded at the end of the current one, so their latency is off the next
  // unit's path.
  const int cq = tid >> 7, jq = tid & (kDim - 1);
  float wq[kWidth], wv[kWidth], bq = 0.0f, bv = 0.0f, gate_a = 0.0f, gate_bias = 0.0f;
  int w_head = -1;
  auto load_head = [&](int hh) {
    const int64_t wbase = static_cast<int64_t>(hh) * kDim + jq;
#pragma unroll
    for (int k = 0; k < kWidth; ++k) wq[k] = __ldg(p.conv_w + (cq * kWidth + k) * D + wbase);
    bq = p.conv_b ? __ldg(p.conv_b + cq * D + wbase) : 0.0f;
    if (tid < kDim) {
#pragma unroll
      for (int k = 0; k < kWidth; ++k) wv[k] = __ldg(p.conv_w + (2 * kWidth + k) * D + wbase);
      bv = p.conv_b ? __ldg(p.conv_b + 2 * D + wbase) : 0.0f;
    } else if (p.fused_gate) {
      gate_a = expf(__ldg(p.A_log + hh));
      gate_bias = p.dt_bias ? __ldg(p.dt_bias + wbase) : 0.0f;
    }
    w_head = hh;
  };
#ifdef KDA_DECODE_TIMELINE
  // timeline build: per CTA the time waiting for a unit's data, in the
  // state-independent phase, in the token loop, waiting for an output
  // buffer; thread 0's accumulators in shared memory so that they take no
  // registers: start, in, up, loop, freed, units, last timestamp
  __shared__ unsigned long long tl_acc[7];
  volatile unsigned long long* tl = tl_acc;
  if (tid == 0) {
    tl[0] = global_ns();
    for (int i = 1; i < 7; ++i) tl[i] = 0;
  }
#endif
  for (int it = 0;; ++it) {
#ifdef KDA_DECODE_TIMELINE
    if (tid == 0) tl[6] = global_ns();
#endif
    const int st = it % kMStages;
    const uint32_t parity = (it / kMStages) & 1;
    const bool have_info = mbar_wait_bounded(smem_addr(&S.ready[st]), parity, p.wait_limit_ns);
    int n = -1, h = 0;
    bool ok = have_info;
    if (have_info) {
      n = S.info[st][1];
      h = S.info[st][2];
      if (n >= 0) ok = mbar_wait_bounded(smem_addr(&S.full[st]), parity, p.wait_limit_ns);
    }
    // Agreement to go on; also the barrier that ends every use of the
    // previous unit's per-token scratch.
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
      tl[1] += now - tl[6];
      tl[6] = now;
      if (n >= 0) tl[5] += 1;
    }
#endif
    if (n < 0) break;  // no more units
    const int src = S.info[st][0];
    const bool src_ok = valid(src);
    if (src >= p.num_slots && tid == 0) flag_error(p, KDA_DEVERR_SLOT_RANGE);
    // Padding sequence or absent tokens: zero output rows, no state.
    for (int t = 0; t < T; ++t) {
      const int dst = S.info[st][kMiDst + t];
      if (src_ok && valid(dst)) continue;
      uint16_t* out_row = p.out + (static_cast<int64_t>(n) * T + t) * p.out_stride + static_cast<int64_t>(h) * kDim;
      if (tid < kDim * 2 / 16) reinterpret_cast<uint4*>(out_row)[tid] = make_uint4(0, 0, 0, 0);
      if (src_ok && dst >= p.num_slots && tid == 0) flag_error(p, KDA_DEVERR_SLOT_RANGE);
    }
    const int np = src_ok ? S.info[st][kMiNp] : 0;
    if (np == 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.done[st]));
      continue;
    }
    const int* pt = &S.info[st][kMiPt];  // present token indices

    // This warp's 16 rows of the source state into registers now: the reads
    // overlap the state-independent work below.
    float4 a[kRowsPerWarp];
    {
      const float4* tile4 = reinterpret_cast<const float4*>(S.tile[st]);
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) a[r] = tile4[(warp * kRowsPerWarp + r) * 32 + lane];
    }
    // ---- state-independent work of every present token.
    // Each thread holds its channels' sequences in registers: taps 0-2 the
    // source window, tap 3 + m the input of present token m (bf16 bits).
    if (w_head != h) load_head(h);
    {
      // beta of present token tid: loaded here, used after the conv below
      const uint16_t beta_bits =
          tid < np ? __ldg(p.beta + (static_cast<int64_t>(n) * T + pt[tid]) * p.H + h) : uint16_t{0};
      const int cs_j = p.conv_sd ? 1 : kWidth - 1, cs_t = p.conv_sd ? kDim : 1;
      uint16_t sq[kWidth - 1 + kTMax], sv[kWidth - 1 + kTMax];
#pragma unroll
      for (int i = 0; i < kWidth - 1; ++i) {
        sq[i] = S.cs[st][cq][cs_j * jq + cs_t * i];
        sv[i] = tid < kDim ? S.cs[st][2][cs_j * jq + cs_t * i] : uint16_t{0};
      }
#pragma unroll
      for (int m = 0; m < kTMax; ++m) {
        sq[kWidth - 1 + m] = m < np ? S.x[st][pt[m]][cq][jq] : uint16_t{0};
        sv[kWidth - 1 + m] = (m < np && tid < kDim) ? S.x[st][pt[m]][2][jq] : uint16_t{0};
      }
#pragma unroll
      for (int m = 0; m < kTMax; ++m) {
        if (m >= np) break;
        float y = bq;
#pragma unroll
        for (int k = 0; k < kWidth; ++k) y = fmaf(wq[k], bf16_to_f32(sq[m + k]), y);
        (cq == 0 ? S.q[m] : S.k[m])[jq] = __fdividef(y, 1.0f + __expf(-y));
        if (tid < kDim) {
          float yv = bv;
#pragma unroll
          for (int k = 0; k < kWidth; ++k) yv = fmaf(wv[k], bf16_to_f32(sv[m + k]), yv);
          S.v[m][jq] = __fdividef(yv, 1.0f + __expf(-yv));
        } else {
          float g = S.g[st][pt[m]][jq];
          if (p.fused_gate) {
            const float z = g + gate_bias;
            if (p.lower_bound < 0.0f) {
              g = p.lower_bound / (1.0f + expf(-gate_a * z));
            } else {
              const float sp = (z > 0.0f) ? z + log1pf(expf(-z)) : log1pf(expf(z));
              g = -gate_a * sp;
            }
          }
          S.alpha[m][jq] = expf(g);
        }
        // the window after token m (taps m+1 .. m+3, bit patterns) to its slot
        if (kUpdateConv) {
          const int64_t dst = S.info[st][kMiDst + pt[m]];
          const int64_t chq = cq * D + static_cast<int64_t>(h) * kDim + jq, chv = 2 * D + static_cast<int64_t>(h) * kDim + jq;
#pragma unroll
          for (int k = 0; k < kWidth - 1; ++k) {
            if (p.conv_sd) {
              p.conv_state[(dst * (kWidth - 1) + k) * 3 * D + chq] = sq[m + 1 + k];
              if (tid < kDim) p.conv_state[(dst * (kWidth - 1) + k) * 3 * D + chv] = sv[m + 1 + k];
            } else {
              p.conv_state[(dst * 3 * D + chq) * (kWidth - 1) + k] = sq[m + 1 + k];
              if (tid < kDim) p.conv_state[(dst * 3 * D + chv) * (kWidth - 1) + k] = sv[m + 1 + k];
            }
          }
        }
      }
      if (tid < np) {
        const float bt = bf16_to_f32(beta_bits);
        S.beta[tid] = p.fused_gate ? 1.0f / (1.0f + expf(-bt)) : bt;
      }
    }
    consumer_sync();
    // Per present token (warp m): |q~|^2, |k~|^2, q~.k~ in one fixed order
    // (so q~.k~ equals |k~|^2 bit for bit when q~ equals k~), then the
    // readout coefficients of the decode step's cancellation-safe form.
    if (warp < np) {
      const int m = warp;
      const float4 q4 = reinterpret_cast<const float4*>(S.q[m])[lane];
      const float4 k4 = reinterpret_cast<const float4*>(S.k[m])[lane];
      float ssq = fmaf(q4.x, q4.x, fmaf(q4.y, q4.y, fmaf(q4.z, q4.z, q4.w * q4.w)));
      float ssk = fmaf(k4.x, k4.x, fmaf(k4.y, k4.y, fmaf(k4.z, k4.z, k4.w * k4.w)));
      float sqk = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, q4.w * k4.w)));
      ssq = warp_sum(ssq);
      ssk = warp_sum(ssk);
      sqk = warp_sum(sqk);
      if (lane == 0) {
        const float beta = S.beta[m];
        const float rq = scale * rsqrtf(ssq + 1e-6f);
        const float rk = rsqrtf(ssk + 1e-6f);
        S.coef[m] = make_float4(rq, rk, (fmaf(-beta, sqk, ssk) + 1e-6f) * (rk * rk), beta * sqk * rq * rk);
      }
    }
    consumer_sync();

#ifdef KDA_DECODE_TIMELINE
    if (tid == 0) {
      const unsigned long long now = global_ns();
      tl[2] += now - tl[6];
      tl[6] = now;
    }
#endif
    // ---- the recurrence, token by token, state in registers.
    // Token mp's rank-1 update S' = A + k^ delta^T, and its state into its
    // output buffer for the bulk store to its slot.
    auto update_and_write = [&](int mp) {
      const int b = out_buf(st, mp);
      float4* tile4w = reinterpret_cast<float4*>(S.tile[b]);
      const float4 d = reinterpret_cast<const float4*>(S.delta)[lane];
#pragma unroll
      for (int r4 = 0; r4 < kRowsPerWarp / 4; ++r4) {
        const float4 kt4 = reinterpret_cast<const float4*>(S.k[mp] + warp * kRowsPerWarp)[r4];
        const float kt_4[4] = {kt4.x, kt4.y, kt4.z, kt4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * r4 + i;
          a[r].x = fmaf(kt_4[i], d.x, a[r].x); a[r].y = fmaf(kt_4[i], d.y, a[r].y);
          a[r].z = fmaf(kt_4[i], d.z, a[r].z); a[r].w = fmaf(kt_4[i], d.w, a[r].w);
          tile4w[(warp * kRowsPerWarp + r) * 32 + lane] = a[r];
        }
      }
      fence_proxy_async_smem();  // generic-proxy writes before the async-proxy store
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.written[b]));
      if (b == 0) ++wcnt0; else if (b == 1) ++wcnt1; else ++wcnt2;
    };
    bool aborted = false;
    for (int m = 0; m < np; ++m) {
      if (m > 0) update_and_write(m - 1);
      // decay and partial column sums of token m over this warp's 16 rows
      float4 u = make_float4(0.f, 0.f, 0.f, 0.f), w = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r4 = 0; r4 < kRowsPerWarp / 4; ++r4) {
        const float4 al4 = reinterpret_cast<const float4*>(S.alpha[m] + warp * kRowsPerWarp)[r4];
        const float4 kt4 = reinterpret_cast<const float4*>(S.k[m] + warp * kRowsPerWarp)[r4];
        const float4 qt4 = reinterpret_cast<const float4*>(S.q[m] + warp * kRowsPerWarp)[r4];
        const float al_4[4] = {al4.x, al4.y, al4.z, al4.w};
        const float kt_4[4] = {kt4.x, kt4.y, kt4.z, kt4.w};
        const float qt_4[4] = {qt4.x, qt4.y, qt4.z, qt4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * r4 + i;
          a[r].x *= al_4[i]; a[r].y *= al_4[i]; a[r].z *= al_4[i]; a[r].w *= al_4[i];
          u.x = fmaf(kt_4[i], a[r].x, u.x); u.y = fmaf(kt_4[i], a[r].y, u.y);
          u.z = fmaf(kt_4[i], a[r].z, u.z); u.w = fmaf(kt_4[i], a[r].w, u.w);
          w.x = fmaf(qt_4[i], a[r].x, w.x); w.y = fmaf(qt_4[i], a[r].y, w.y);
          w.z = fmaf(qt_4[i], a[r].z, w.z); w.w = fmaf(qt_4[i], a[r].w, w.w);
        }
      }
      reinterpret_cast<float4*>(S.red[0][warp])[lane] = u;
      reinterpret_cast<float4*>(S.red[1][warp])[lane] = w;
      consumer_sync();

      // delta and the readout o = rq ((w~ - u~) + m u~) + beta (q^.k^) v
      float o = 0.0f;
      if (tid < kDim) {
        const float4 cf = S.coef[m];  // rq, rk, m, beta (q^.k^)
        float ut = 0.0f, wt = 0.0f;
#pragma unroll
        for (int r = 0; r < kConsumerWarps; ++r) {
          ut += S.red[0][r][tid];
          wt += S.red[1][r][tid];
        }
        const float vj = S.v[m][tid];
        const float dj = S.beta[m] * (vj - cf.y * ut);
        S.delta[tid] = cf.y * dj;  // the update adds k~ (rk delta)^T = k^ delta^T
        o = fmaf(cf.w, vj, cf.x * fmaf(cf.z, ut, wt - ut));
        if (kOutNorm) {
          const float so = warp_sum(o * o);
          if (lane == 0) S.osum[warp] = so;
        }
      }
      // Token m's state goes into its output buffer next: the store of what
      // was written there before has to have read it out.  Every consumer
      // agrees before going on; this vote is also the barrier that publishes
      // delta.
      const int bn = out_buf(st, m);
      const uint32_t wc = (bn == 0) ? wcnt0 : (bn == 1) ? wcnt1 : wcnt2;
      bool fok = true;
#ifdef KDA_DECODE_TIMELINE
      const unsigned long long tl_f0 = tid == 0 ? global_ns() : 0ull;
#endif
      if (wc > 0) fok = mbar_wait_bounded(smem_addr(&S.freed[bn]), (wc - 1) & 1u, p.wait_limit_ns);
#ifdef KDA_DECODE_TIMELINE
      if (tid == 0) tl[4] += global_ns() - tl_f0;
#endif
      if (consumer_any(!fok || S.abort)) {
        if (tid == 0) {
          flag_error(p, KDA_DEVERR_TIMEOUT);
          S.abort = 1;
        }
        aborted = true;
        break;
      }
      // gated RMSNorm epilogue (or the raw readout) of token m
      if (tid < kDim) {
        const int t = pt[m];
        float y = o;
        if (kOutNorm) {
          const float ss = (S.osum[0] + S.osum[1]) + (S.osum[2] + S.osum[3]);
          const float rr = rsqrtf(ss * (1.0f / kDim) + p.eps);
          y = o * rr * nw * __fdividef(1.0f, 1.0f + __expf(-bf16_to_f32(S.gate[st][t][tid])));
        }
        p.out[(static_cast<int64_t>(n) * T + t) * p.out_stride + static_cast<int64_t>(h) * kDim + tid] = f32_to_bf16(y);
      }
    }
    if (aborted) break;
    update_and_write(np - 1);
    if (lane == 0) mbar_arrive(smem_addr(&S.done[st]));
    {  // the next unit's conv taps, if it is published already
      const int s2 = (it + 1) % kMStages;
      if (mbar_try_wait(smem_addr(&S.ready[s2]), ((it + 1) / kMStages) & 1)) {
        const int n2 = S.info[s2][1], h2 = S.info[s2][2];
        if (n2 >= 0 && h2 != w_head) load_head(h2);
      }
    }
#ifdef KDA_DECODE_TIMELINE
    if (tid == 0) tl[3] += global_ns() - tl[6];
#endif
  }
#ifdef KDA_DECODE_TIMELINE
  if (tid == 0) {
    const unsigned int i = atomicAdd(&g_timeline_n, 1u);
    if (i < kTimelineMax) {
      g_timeline[i][0] = blockIdx.x; g_timeline[i][1] = tl[4]; g_timeline[i][2] = tl[0]; g_timeline[i][3] = tl[2];
      g_timeline[i][4] = global_ns(); g_timeline[i][5] = tl[5]; g_timeline[i][6] = tl[3]; g_timeline[i][7] = tl[1];
    }
  }
#endif
}

}  // namespace
