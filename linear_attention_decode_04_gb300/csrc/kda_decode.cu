// kda_decode.cu -- C ABI of the fused single-token KDA decode step for
// GB300 (sm_103a); the device code is in kda_decode_kernel.cuh.
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

#include <mutex>

#include "kda_decode.h"
#include "kda_decode_kernel.cuh"
#include "kda_decode_multi_kernel.cuh"
#include "kda_internal.h"

namespace {

thread_local char g_last_error[512];

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

struct DeviceInfo {
  int sms = 0;
  bool attrs_set = false;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

// Dynamic shared memory opt-in limit of one CTA on sm_103a.
constexpr size_t kMaxDynSmem = 227 * 1024;
static_assert(sizeof(Smem) <= kMaxDynSmem, "decode kernel shared memory");
static_assert(sizeof(MSmemT<4>) <= kMaxDynSmem, "multi-token kernel shared memory (4 tokens)");
static_assert(sizeof(MSmemT<kMaxT>) <= kMaxDynSmem, "multi-token kernel shared memory");

template <bool kOutNorm, bool kUpdateConv>
cudaError_t set_attrs() {
  cudaError_t e = cudaFuncSetAttribute(kda_decode_persistent_kernel<kOutNorm, kUpdateConv>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sizeof(Smem)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kda_decode_multi_kernel<kOutNorm, kUpdateConv, 4>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sizeof(MSmemT<4>)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kda_decode_multi_kernel<kOutNorm, kUpdateConv, kMaxT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sizeof(MSmemT<kMaxT>)));
}

// Once per device: SM count and the large dynamic shared-memory opt-in for
// every kernel variant.  Not a stream operation, but it should run before
// any stream capture (the first call on a device does it).
cudaError_t device_setup(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.attrs_set) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = set_attrs<true, true>()) != cudaSuccess) return e;
    if ((e = set_attrs<true, false>()) != cudaSuccess) return e;
    if ((e = set_attrs<false, true>()) != cudaSuccess) return e;
    if ((e = set_attrs<false, false>()) != cudaSuccess) return e;
    d.attrs_set = true;
  }
  *sms = d.sms;
  return cudaSuccess;
}

// With a work queue, each CTA first takes a static prefix of its units (no
// atomics) and then draws from the queue.  The prefix keeps at least
// kQueueTailMin of a CTA's units dynamic, so the queue can even out the CTAs'
// end times, and is at most kQueueStaticCap long, so that on long launches
// (where per-SM bandwidth differences add up) most units stay dynamic.  On
// short launches (tens of units per CTA) only the last few are dynamic and
// pay the atomic's latency.  The first ring of every CTA is always static.
constexpr int kQueueTailMin = 2;
constexpr int kQueueStaticCap = 16;

template <bool kOutNorm, bool kUpdateConv>
cudaError_t launch(const Params& p_in, int sms, cudaStream_t stream) {
  Params p = p_in;
  {
    const int G = p.total_units < sms ? p.total_units : sms;
    const int ring = (p.T > 1 || p.src_slot != nullptr) ? kMStages : kStages;
    int prefix = p.total_units / G - kQueueTailMin;
    prefix = prefix < kQueueStaticCap ? prefix : kQueueStaticCap;
    p.static_units = prefix > ring ? prefix : ring;
  }
  // Every launch is a programmatic dependent launch: the CTAs may become
  // resident while the previous kernel in the stream drains, and wait for
  // it (griddepcontrol.wait) before touching its results.
  const bool multi = p.T > 1 || p.src_slot != nullptr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.total_units < sms ? p.total_units : sms));
  cfg.blockDim = dim3(kThreads);
  const bool small_t = p.T <= 4;  // up to 4 tokens: two output buffers per unit
  cfg.dynamicSmemBytes = !multi ? sizeof(Smem) : small_t ? sizeof(MSmemT<4>) : sizeof(MSmemT<kMaxT>);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = !multi   ? cudaLaunchKernelEx(&cfg, kda_decode_persistent_kernel<kOutNorm, kUpdateConv>, p)
                  : small_t ? cudaLaunchKernelEx(&cfg, kda_decode_multi_kernel<kOutNorm, kUpdateConv, 4>, p)
                            : cudaLaunchKernelEx(&cfg, kda_decode_multi_kernel<kOutNorm, kUpdateConv, kMaxT>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int kda_internal_fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

void kda_internal_clear_error() { g_last_error[0] = '\0'; }

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

namespace {
int validate(const KdaDecodeArgs* a, uint64_t wait_limit_ns, int32_t withhold_unit, Params* p);
int launch_validated(const Params& p, uint32_t flags, void* stream);

int decode_impl(const KdaDecodeArgs* a, void* stream, uint64_t wait_limit_ns, int32_t withhold_unit) {
  Params p;
  const int rc = validate(a, wait_limit_ns, withhold_unit, &p);
  if (rc != KDA_OK || a->N == 0) return rc;
  return launch_validated(p, a->flags, stream);
}
}  // namespace

extern "C" int kda_decode(const KdaDecodeArgs* a, void* stream) {
  return decode_impl(a, stream, kWaitLimitNs, -1);
}

extern "C" int kda_decode_wait_test(const KdaDecodeArgs* a, void* stream, uint64_t wait_limit_ns,
                                    int32_t withhold_unit) {
  if (wait_limit_ns == 0) return fail(KDA_ERR_SHAPE, "wait_limit_ns must be > 0");
  return decode_impl(a, stream, wait_limit_ns, withhold_unit);
}

namespace {
// Checks every argument and fills the kernel's parameter block; touches no
// CUDA API and no device memory.  N == 0 passes (the caller launches nothing).
int validate(const KdaDecodeArgs* a, uint64_t wait_limit_ns, int32_t withhold_unit, Params* out) {
  g_last_error[0] = '\0';
  if (!a) return fail(KDA_ERR_NULLPTR, "args is NULL");
  if (a->struct_size != sizeof(KdaDecodeArgs))
    return fail(KDA_ERR_ABI, "struct_size %u, library expects %zu", a->struct_size, sizeof(KdaDecodeArgs));
  if (a->head_dim != KDA_HEAD_DIM || a->conv_width != KDA_CONV_WIDTH)
    return fail(KDA_ERR_SHAPE, "head_dim %d / conv_width %d (need 128 / 4)", a->head_dim, a->conv_width);
  if (a->N < 0 || a->H < 1 || a->num_slots < 1)
    return fail(KDA_ERR_SHAPE, "N=%d H=%d num_slots=%d", a->N, a->H, a->num_slots);
  if (a->flags &
      ~(KDA_OUT_NORM | KDA_UPDATE_CONV_STATE | KDA_EARLY_PREFETCH | KDA_FUSED_GATE | KDA_CONV_STATE_SD))
    return fail(KDA_ERR_FLAGS, "flags 0x%x", a->flags);
  if (a->N == 0) return KDA_OK;
  const bool norm = (a->flags & KDA_OUT_NORM) != 0;
  if (!a->qkv || !a->conv_weight || !a->conv_state || !a->state || !a->g || !a->beta || !a->slot_idx ||
      !a->out)
    return fail(KDA_ERR_NULLPTR, "a required tensor pointer is NULL");
  if (norm && (!a->gate || !a->norm_weight))
    return fail(KDA_ERR_NULLPTR, "KDA_OUT_NORM needs gate and norm_weight");
  const bool fused_gate = (a->flags & KDA_FUSED_GATE) != 0;
  if (fused_gate && !a->A_log) return fail(KDA_ERR_NULLPTR, "KDA_FUSED_GATE needs A_log");
  if (fused_gate && ((reinterpret_cast<uintptr_t>(a->A_log) & 3u) ||
                     (reinterpret_cast<uintptr_t>(a->dt_bias) & 3u)))
    return fail(KDA_ERR_ALIGN, "A_log and dt_bias must be 4-byte aligned");
  if (reinterpret_cast<uintptr_t>(a->work_queue) & 3u) return fail(KDA_ERR_ALIGN, "work_queue must be 4-byte aligned");
  if (a->tokens_per_seq < 0 || a->tokens_per_seq > KDA_MAX_TOKENS_PER_SEQ)
    return fail(KDA_ERR_SHAPE, "tokens_per_seq %d (need 0 .. %d)", a->tokens_per_seq, KDA_MAX_TOKENS_PER_SEQ);
  if (reinterpret_cast<uintptr_t>(a->src_slot) & 3u) return fail(KDA_ERR_ALIGN, "src_slot must be 4-byte aligned");
  const int T = a->tokens_per_seq > 1 ? a->tokens_per_seq : 1;
  if (static_cast<int64_t>(a->N) * T > (1LL << 30))
    return fail(KDA_ERR_SHAPE, "N*tokens_per_seq = %lld rows is too many", static_cast<long long>(a->N) * T);
  const int64_t D = static_cast<int64_t>(a->H) * KDA_HEAD_DIM;
  if (static_cast<int64_t>(a->N) * a->H > (1LL << 30))
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

  Params& p = *out;
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
  p.total_units = a->N * a->H;
  p.early_prefetch = (a->flags & KDA_EARLY_PREFETCH) != 0;
  p.fused_gate = fused_gate;
  p.conv_sd = (a->flags & KDA_CONV_STATE_SD) != 0;
  p.A_log = fused_gate ? a->A_log : nullptr;
  p.dt_bias = fused_gate ? a->dt_bias : nullptr;
  p.lower_bound = a->lower_bound;
  p.queue = a->work_queue;
  p.withhold_unit = withhold_unit;
  p.wait_limit_ns = wait_limit_ns;
  p.T = T;
  p.src_slot = a->src_slot;
  return KDA_OK;
}

// Once-per-device set-up, then the launch of a validated parameter block.
int launch_validated(const Params& p, uint32_t flags, void* stream) {
  int sms = 0;
  cudaError_t es = device_setup(&sms);
  if (es != cudaSuccess) return fail(KDA_ERR_LAUNCH, "device set-up: %s", cudaGetErrorString(es));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool norm = (flags & KDA_OUT_NORM) != 0;
  const bool conv = (flags & KDA_UPDATE_CONV_STATE) != 0;
  cudaError_t e = norm ? (conv ? launch<true, true>(p, sms, s) : launch<true, false>(p, sms, s))
                       : (conv ? launch<false, true>(p, sms, s) : launch<false, false>(p, sms, s));
  if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "%s", cudaGetErrorString(e));
  return KDA_OK;
}
}  // namespace

#ifdef KDA_DECODE_TIMELINE
// Timeline build only (lib/libkda_decode_timeline.so): read and reset the
// per-CTA records of the decode kernel.  Not part of the product library.
extern "C" int kda_timeline_read(unsigned long long* host, int max_records, unsigned int* total) {
  cudaError_t e = cudaMemcpyFromSymbol(total, g_timeline_n, sizeof(unsigned int));
  if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "%s", cudaGetErrorString(e));
  const unsigned int avail = *total < static_cast<unsigned int>(kTimelineMax) ? *total : kTimelineMax;
  const int n = static_cast<int>(avail) < max_records ? static_cast<int>(avail) : max_records;
  if (n > 0) e = cudaMemcpyFromSymbol(host, g_timeline, static_cast<size_t>(n) * 8 * sizeof(unsigned long long));
  return e == cudaSuccess ? n : fail(KDA_ERR_LAUNCH, "%s", cudaGetErrorString(e));
}

extern "C" int kda_timeline_reset(void) {
  const unsigned int zero = 0;
  const cudaError_t e = cudaMemcpyToSymbol(g_timeline_n, &zero, sizeof zero);
  return e == cudaSuccess ? KDA_OK : fail(KDA_ERR_LAUNCH, "%s", cudaGetErrorString(e));
}
#endif

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot allocate device memory for the work queue: plugin
// interfaces whose enqueue step must not allocate, serving loops that fix
// their memory budget at start-up, and callers that reach the library only
// through this C ABI and hold no device allocator of their own.
// kda_decode_noalloc serves them with the dynamic schedule, keeping the queue
// in this file-scope device array instead of a caller-provided buffer.  Every
// GPU that loads the library holds the array until the process exits.
namespace {
constexpr size_t kNoAllocScratchBytes = 256;                    // stated maximum
constexpr size_t kNoAllocQueueBytes = 2 * sizeof(int32_t);      // what one call uses, whatever N and H
static_assert(kNoAllocQueueBytes <= kNoAllocScratchBytes, "the work queue must fit the static scratch array");
}  // namespace

static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

namespace {
// Device address of g_noalloc_scratch per device ordinal, looked up once with
// that device current (guarded by g_dev_mutex).  It stays valid as long as
// the device's primary context lives, which the library assumes for the life
// of the process.
int32_t* g_noalloc_ptr[64];
}  // namespace

extern "C" int kda_decode_noalloc(const KdaDecodeArgs* a, void* stream) {
  // Every argument is checked before anything is enqueued
  // (args->work_queue is ignored, so it is cleared in the checked copy).
  g_last_error[0] = '\0';
  if (!a) return fail(KDA_ERR_NULLPTR, "args is NULL");
  if (a->struct_size != sizeof(KdaDecodeArgs))
    return fail(KDA_ERR_ABI, "struct_size %u, library expects %zu", a->struct_size, sizeof(KdaDecodeArgs));
  KdaDecodeArgs b = *a;
  b.work_queue = nullptr;
  Params p;
  const int rc = validate(&b, kWaitLimitNs, -1, &p);
  if (rc != KDA_OK || b.N == 0) return rc;
  // Once per device, with that device current: the array's device address
  // (in host code the array's name is only a stand-in, never a pointer the
  // kernel can use).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(KDA_ERR_LAUNCH, "device ordinal %d out of range", dev);
  int32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_noalloc_ptr[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      g_noalloc_ptr[dev] = static_cast<int32_t*>(ptr);
    }
    scratch = g_noalloc_ptr[dev];
  }
  // The queue must start at zero; the array keeps whatever the last call left.
  e = cudaMemsetAsync(scratch, 0, kNoAllocQueueBytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "clearing the scratch: %s", cudaGetErrorString(e));
  p.queue = scratch;
  return launch_validated(p, b.flags, stream);
}
