// C ABI, argument validation, workspace plan and the head-group x sequence-trunk scheduler.
//
// Schedule (per call):
//   for each head group g of head_chunk q-heads (UPipe: one set of heads at a time, all groups
//   reusing one workspace - "Road to 5 million sequence length" talk, UPipe passage;
//   "Road to 5 Million Tokens" summary, section 2 item 6):
//     gather the group's Q (and K/V when they are on the device) into head-major workspace
//     (the single-GPU stand-in for the Ulysses all-to-all);
//     forward: for each query trunk m, fold key/value trunks n = 0..m (all n if not causal)
//       into running softmax state, finalising O and LSE on the last one (FPDT Technical Deep
//       Dive: Q_m attends K_1..K_m, statistics updated per trunk);
//     backward: pre-pass (dO gather, D = rowsum(dO*O), LSE prescale, zero dQ accumulator),
//       then one launch per key/value trunk n over all query rows that see it, then the dQ
//       conversion.
//   When K/V are pinned host memory every trunk is copied into one of two device slots on an
//   internal copy stream, one trunk ahead of the compute stream, with events ordering slot
//   reuse (FPDT Key Findings items 2-3 and Technical Deep Dive: host offload + double buffer,
//   separate streams for compute and host<->device copies).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "upipe.h"
#include "internal.h"

namespace upipe {
namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(UPIPE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define UPIPE_CUDA(call)                                  \
  do {                                                    \
    cudaError_t e_ = (call);                              \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);   \
  } while (0)

// ---- per-device state -----------------------------------------------------------------------
struct DevState {
  bool ready = false;
  cudaStream_t copy = nullptr;      // key/value trunks in, dK/dV trunks out
  cudaStream_t act_copy = nullptr;  // head-group activations in and out (bulk, with slack)
  cudaEvent_t slot_ready[2] = {nullptr, nullptr};
  cudaEvent_t slot_free[2] = {nullptr, nullptr};
  cudaEvent_t dkdv_done[2] = {nullptr, nullptr};  // a dK/dV slot is written (compute stream)
  cudaEvent_t dkdv_free[2] = {nullptr, nullptr};  // its copy to the host is done (copy stream)
  cudaEvent_t act_ready[2] = {nullptr, nullptr};  // a group's host activations staged in
  cudaEvent_t act_free[2] = {nullptr, nullptr};   // the group's kernels are done with them
  cudaEvent_t out_done[2] = {nullptr, nullptr};   // a group's outputs are in their staging
  cudaEvent_t out_free[2] = {nullptr, nullptr};   // ... and have been copied to the host
  cudaEvent_t entry = nullptr;
  cudaEvent_t copy_done = nullptr;
  cudaEvent_t act_done = nullptr;
  uint32_t* err = nullptr;  // 256-byte status word allocation
};
constexpr int kMaxDev = 64;
std::mutex g_mu;
DevState g_dev[kMaxDev];

int dev_state(int dev, DevState** out) {
  if (dev < 0 || dev >= kMaxDev) return fail(UPIPE_ERR_UNSUPPORTED, "device %d", dev);
  DevState& d = g_dev[dev];
  if (!d.ready) {
    UPIPE_CUDA(cudaStreamCreateWithFlags(&d.copy, cudaStreamNonBlocking));
    UPIPE_CUDA(cudaStreamCreateWithFlags(&d.act_copy, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
      UPIPE_CUDA(cudaEventCreateWithFlags(&d.slot_ready[i], cudaEventDisableTiming));
      UPIPE_CUDA(cudaEventCreateWithFlags(&d.slot_free[i], cudaEventDisableTiming));
      UPIPE_CUDA(cudaEventCreateWithFlags(&d.dkdv_done[i], cudaEventDisableTiming));
      UPIPE_CUDA(cudaEventCreateWithFlags(&d.dkdv_free[i], cudaEventDisableTiming));
      UPIPE_CUDA(cudaEventCreateWithFlags(&d.act_ready[i], cudaEventDisableTiming));
      UPIPE_CUDA(cudaEventCreateWithFlags(&d.act_free[i], cudaEventDisableTiming));
      UPIPE_CUDA(cudaEventCreateWithFlags(&d.out_done[i], cudaEventDisableTiming));
      UPIPE_CUDA(cudaEventCreateWithFlags(&d.out_free[i], cudaEventDisableTiming));
    }
    UPIPE_CUDA(cudaEventCreateWithFlags(&d.entry, cudaEventDisableTiming));
    UPIPE_CUDA(cudaEventCreateWithFlags(&d.copy_done, cudaEventDisableTiming));
    UPIPE_CUDA(cudaEventCreateWithFlags(&d.act_done, cudaEventDisableTiming));
    UPIPE_CUDA(cudaMalloc(&d.err, 256));
    UPIPE_CUDA(cudaMemset(d.err, 0, 256));
    UPIPE_CUDA(cudaDeviceSynchronize());
    d.ready = true;
  }
  *out = &d;
  return UPIPE_OK;
}

// ---- launch accounting / profiling ----------------------------------------------------------
std::atomic<uint64_t> g_launches{0};
std::atomic<bool> g_profile{false};
struct ProfRec {
  int kclass;
  cudaEvent_t e0, e1;
};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;
thread_local cudaEvent_t g_pending_e0 = nullptr;

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

void launch_begin(int kclass, cudaStream_t stream) {
  (void)kclass;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_profile.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_pending_e0 = pool_event();
  if (g_pending_e0) cudaEventRecord(g_pending_e0, stream);
}

void copy_begin(cudaStream_t stream) {
  if (!g_profile.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_pending_e0 = pool_event();
  if (g_pending_e0) cudaEventRecord(g_pending_e0, stream);
}

void copy_end(int kclass, cudaStream_t stream) { launch_end(kclass, stream); }

void launch_end(int kclass, cudaStream_t stream) {
  if (!g_profile.load(std::memory_order_relaxed) || !g_pending_e0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t e1 = pool_event();
  if (!e1) return;
  cudaEventRecord(e1, stream);
  g_prof.push_back({kclass, g_pending_e0, e1});
  g_pending_e0 = nullptr;
}

// ---- per-device kernel attributes --------------------------------------------------------
cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;  // (kernel, device) already set
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& d : done)
    if (d.first == kernel && d.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  done.emplace_back(kernel, dev);
  return cudaSuccess;
}

// ---- tensor maps ----------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// The driver's tensor-map encoder, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}
}  // namespace

int launch_band(int64_t units_per_lane, int lanes) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  if (units_per_lane < 1 || lanes < 1) return 1;
  // at least eight waves of units per band, and bands of equal size (a short last band would
  // start its heavy units late and end alone)
  const int64_t min_band = (8 * static_cast<int64_t>(sms) + units_per_lane - 1) / units_per_lane;
  const int64_t n_bands = std::max<int64_t>(1, lanes / std::max<int64_t>(1, min_band));
  return static_cast<int>((lanes + n_bands - 1) / n_bands);
}

cudaError_t make_tmap_bf16(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                           int64_t depth, int box_rows) {
  tensor_map_encoder();
  if (!g_encode) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(depth)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols * 2),
                                 static_cast<cuuint64_t>(cols * rows * 2)};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// ---- workspace plan ---------------------------------------------------------------------------
constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

using Plan = AttnPlan;

}  // namespace

// Validates shapes (no device access). Returns UPIPE_OK and fills the plan.
int make_attn_plan(int B, int64_t S, int Hq, int Hkv, int D, int causal, int head_chunk,
                   int64_t seq_trunk, int host_mask, AttnPlan* p) {
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || D < 1)
    return fail(UPIPE_ERR_INVALID_ARG, "sizes must be positive (B=%d S=%lld Hq=%d Hkv=%d D=%d)",
                B, static_cast<long long>(S), Hq, Hkv, D);
  if (Hq % Hkv) return fail(UPIPE_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  const int G = Hq / Hkv;
  if (head_chunk < 1 || Hq % head_chunk)
    return fail(UPIPE_ERR_INVALID_ARG, "head_chunk=%d must divide Hq=%d", head_chunk, Hq);
  if (head_chunk % G)
    return fail(UPIPE_ERR_INVALID_ARG,
                "head_chunk=%d must be a multiple of Hq/Hkv=%d (a group owns whole kv-heads)",
                head_chunk, G);
  if (causal != 0 && causal != 1) return fail(UPIPE_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (seq_trunk < 1) return fail(UPIPE_ERR_INVALID_ARG, "seq_trunk must be >= 1");
  if (D != 64 && D != 128) return fail(UPIPE_ERR_UNSUPPORTED, "D=%d (supported: 64, 128)", D);
  if (S > (int64_t(1) << 30)) return fail(UPIPE_ERR_UNSUPPORTED, "S=%lld > 2^30", (long long)S);
  const int64_t T = seq_trunk >= S ? S : seq_trunk;
  if (T < S && T % 128)
    return fail(UPIPE_ERR_INVALID_ARG, "seq_trunk=%lld must be a multiple of 128 when < S",
                static_cast<long long>(seq_trunk));
  p->B = B; p->Hq = Hq; p->Hkv = Hkv; p->D = D; p->G = G; p->hc = head_chunk;
  p->kc = head_chunk / G; p->causal = causal; p->S = S; p->T = T;
  p->S_pad = (S + 127) / 128 * 128;
  p->T_pad = (T + 127) / 128 * 128;
  p->n_trunks = static_cast<int>((S + T - 1) / T);
  p->kv_host = (host_mask & UPIPE_HOST_KV) != 0;
  p->act_host = (host_mask & UPIPE_HOST_ACT) != 0;

  const size_t hcB = static_cast<size_t>(B) * p->hc, kcB = static_cast<size_t>(B) * p->kc;
  const size_t qw = hcB * S * D * 2, kvw = kcB * S * D * 2, slot = kcB * T * D * 2;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  // forward
  p->f_qw = take(qw);
  if (p->act_host) {
    // host q: a second head-major Q buffer so the next group's Q is staged during this one;
    // host o: two [B, S, hc, D] staging buffers, copied out while the next group computes
    p->f_qw2 = take(qw);
    for (int i = 0; i < 2; ++i) p->f_ostg[i] = take(qw);
  }
  if (p->kv_host) {
    for (int i = 0; i < 2; ++i) { p->f_slot_k[i] = take(slot); p->f_slot_v[i] = take(slot); }
  } else {
    p->f_kw = take(kvw);
    p->f_vw = take(kvw);
  }
  if (p->kv_host && p->n_trunks > 1) {
    // Host K/V: the forward walks key/value trunks outermost (each trunk is staged once), so
    // the running state of every query trunk is kept between launches: S_pad rows. Device
    // K/V need none: one launch walks every trunk with the state on chip.
    p->f_state_o = take(hcB * p->S_pad * D * 4);
    p->f_state_ml = take(hcB * p->S_pad * 2 * 4);
  }
  p->f_total = off;
  // backward
  off = 0;
  p->b_qw = take(qw);
  p->b_dow = take(qw);
  if (p->kv_host) {
    for (int i = 0; i < 2; ++i) { p->b_slot_k[i] = take(slot); p->b_slot_v[i] = take(slot); }
    // dK/dV of a trunk land here when dk/dv are pinned host memory too
    for (int i = 0; i < 2; ++i) { p->b_slot_dk[i] = take(slot); p->b_slot_dv[i] = take(slot); }
  } else {
    p->b_kw = take(kvw);
    p->b_vw = take(kvw);
  }
  if (p->act_host) {
    p->b_qw2 = take(qw);
    p->b_dow2 = take(qw);
    for (int i = 0; i < 2; ++i) p->b_ow[i] = take(qw);
    for (int i = 0; i < 2; ++i) p->b_dqs[i] = take(qw);
  }
  p->b_dqacc = take(hcB * p->S_pad * D * 4);
  p->b_lse2 = take(hcB * p->S_pad * 4);
  p->b_dvec = take(hcB * p->S_pad * 4);
  // Short causal sequences: a key tile's backward walk covers the query tiles of all G q-heads
  // of its kv-head, and the earliest key tiles walk the most, so with few key tiles per launch
  // the first CTAs set the launch time (at S = 8K and 2 kv-heads: 128 CTAs, the longest 64
  // times the shortest). Up to S = 16K the walk is shared by G CTAs, one q-head each, whose
  // fp32 dK/dV shares a reduce kernel adds in a fixed order. The rule depends on the shape
  // only (not on head_chunk), so the workspace stays proportional to head_chunk.
  // The same holds per launch with host K/V, where each key/value trunk is one launch: up to
  // 512 key tiles per launch (T <= 64K) split too.
  const int64_t kt_launch = (p->kv_host ? p->T_pad : p->S_pad) / 128 * B;
  if (causal && D == 128 && G > 1 && kt_launch <= (p->kv_host ? 512 : 128)) {
    p->bwd_split = G;
    p->part_rows = p->kv_host ? p->T_pad : p->S_pad;
    p->b_dkv_part = take(static_cast<size_t>(G) * kcB * p->part_rows * 2 * D * 4);
  }
  p->b_total = off;
  return UPIPE_OK;
}

namespace {

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Where a pointer lives. kind: 0 device (of *dev), 1 pinned host, -1 pageable/unknown.
int pointer_kind(const void* ptr, int* dev) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (at.type == cudaMemoryTypeDevice) {
    *dev = at.device;
    return 0;
  }
  if (at.type == cudaMemoryTypeHost) return 1;
  return -1;
}

// Checks placement of the token-major tensors; selects the device. kv_host out.
int check_placement(const void* const* dev_ptrs, int n_dev, const char* const* names,
                    const void* k, const void* v, bool* kv_host, int* device) {
  int dev0 = -1;
  for (int i = 0; i < n_dev; ++i) {
    int d = -1;
    if (pointer_kind(dev_ptrs[i], &d) != 0)
      return fail(UPIPE_ERR_INVALID_ARG, "%s must be device memory", names[i]);
    if (dev0 < 0) dev0 = d;
    if (d != dev0) return fail(UPIPE_ERR_INVALID_ARG, "%s is on device %d, not %d", names[i], d, dev0);
  }
  int dk = -1, dv = -1;
  const int kk = pointer_kind(k, &dk), kv = pointer_kind(v, &dv);
  if (kk < 0 || kv < 0)
    return fail(UPIPE_ERR_INVALID_ARG, "k and v must be device memory or pinned host memory");
  if (kk != kv) return fail(UPIPE_ERR_INVALID_ARG, "k and v must both be on the device or both pinned on the host");
  if (kk == 0 && (dk != dev0 || dv != dev0))
    return fail(UPIPE_ERR_INVALID_ARG, "k/v are on another device");
  *kv_host = (kk == 1);
  *device = dev0;
  return UPIPE_OK;
}

// Host -> device copy of one key/value trunk [n*T, n*T+Tn) of kv-heads kvh0..kvh0+kc into a
// slot laid out [B*kc][Tn][D]. The 2-D copy does the head gather.
int stage_trunk(const Plan& p, const void* src, uint8_t* slot, int kvh0, int64_t t0, int64_t Tn,
                cudaStream_t copy) {
  const size_t row = static_cast<size_t>(p.D) * 2;
  for (int b = 0; b < p.B; ++b)
    for (int c = 0; c < p.kc; ++c) {
      const uint8_t* s = static_cast<const uint8_t*>(src) +
                         ((static_cast<size_t>(b) * p.S + t0) * p.Hkv + kvh0 + c) * row;
      uint8_t* d = slot + (static_cast<size_t>(b) * p.kc + c) * Tn * row;
      if (staging_copy_fails()) return fail(UPIPE_ERR_CUDA, "injected staging copy failure");
      UPIPE_CUDA(cudaMemcpy2DAsync(d, row, s, static_cast<size_t>(p.Hkv) * row, row,
                                   static_cast<size_t>(Tn), cudaMemcpyHostToDevice, copy));
    }
  return UPIPE_OK;
}

// Device -> host copy of one trunk's dK or dV, slot [B][Tn][kc][D] -> token-major rows
// [t0, t0+Tn) of kv-heads kvh0..kvh0+kc of dst [B,S,Hkv,D]: one 2-D copy per batch row.
int unstage_trunk(const Plan& p, const uint8_t* slot, void* dst, int kvh0, int64_t t0, int64_t Tn,
                  cudaStream_t copy) {
  const size_t row = static_cast<size_t>(p.D) * 2, w = row * p.kc;
  for (int b = 0; b < p.B; ++b) {
    uint8_t* d = static_cast<uint8_t*>(dst) + ((static_cast<size_t>(b) * p.S + t0) * p.Hkv + kvh0) * row;
    const uint8_t* s = slot + static_cast<size_t>(b) * Tn * w;
    if (staging_copy_fails()) return fail(UPIPE_ERR_CUDA, "injected staging copy failure");
    UPIPE_CUDA(cudaMemcpy2DAsync(d, static_cast<size_t>(p.Hkv) * row, s, w, w,
                                 static_cast<size_t>(Tn), cudaMemcpyDeviceToHost, copy));
  }
  return UPIPE_OK;
}

// Host -> device copy of heads [h0, h0+hc) of a token-major [B,S,H,D] tensor into a head-major
// [B*hc][S][D] buffer: one 2-D copy (rows of D elements) per (batch row, head).
int stage_heads(const void* src, void* dst, int B, int64_t S, int H, int D, int h0, int hc,
                cudaStream_t copy) {
  const size_t row = static_cast<size_t>(D) * 2;
  for (int b = 0; b < B; ++b)
    for (int c = 0; c < hc; ++c) {
      const uint8_t* s = static_cast<const uint8_t*>(src) +
                         (static_cast<size_t>(b) * S * H + h0 + c) * row;
      uint8_t* d = static_cast<uint8_t*>(dst) + (static_cast<size_t>(b) * hc + c) * S * row;
      if (staging_copy_fails()) return fail(UPIPE_ERR_CUDA, "injected staging copy failure");
      UPIPE_CUDA(cudaMemcpy2DAsync(d, row, s, static_cast<size_t>(H) * row, row,
                                   static_cast<size_t>(S), cudaMemcpyHostToDevice, copy));
    }
  return UPIPE_OK;
}

// Device -> host copy of a group staging [B,S,hc,D] into heads [h0, h0+hc) of a token-major
// [B,S,H,D] tensor: one 2-D copy per batch row.
int unstage_heads(const void* stg, void* dst, int B, int64_t S, int H, int D, int h0, int hc,
                  cudaStream_t copy) {
  const size_t row = static_cast<size_t>(D) * 2, w = row * hc;
  for (int b = 0; b < B; ++b) {
    uint8_t* d = static_cast<uint8_t*>(dst) + (static_cast<size_t>(b) * S * H + h0) * row;
    const uint8_t* s = static_cast<const uint8_t*>(stg) + static_cast<size_t>(b) * S * w;
    if (staging_copy_fails()) return fail(UPIPE_ERR_CUDA, "injected staging copy failure");
    UPIPE_CUDA(cudaMemcpy2DAsync(d, static_cast<size_t>(H) * row, s, w, w,
                                 static_cast<size_t>(S), cudaMemcpyDeviceToHost, copy));
  }
  return UPIPE_OK;
}

// Up to three head-group gathers, issued as one launch.
struct GatherList {
  const void* src[3];
  void* dst[3];
  int H[3], h0[3], count[3];
  int n = 0;
  void add(const void* s, void* d, int heads, int first, int cnt) {
    src[n] = s; dst[n] = d; H[n] = heads; h0[n] = first; count[n] = cnt;
    ++n;
  }
  cudaError_t launch(int B, int64_t S, int D, cudaStream_t stream) const {
    if (n == 0) return cudaSuccess;
    return launch_gather_group(src, dst, H, h0, count, n, B, S, D, stream);
  }
};

// Double-buffered trunk stager shared by forward and backward.
struct Stager {
  const Plan& p;
  DevState* ds;
  cudaStream_t compute;
  const void* k;
  const void* v;
  uint8_t* slot_k[2];
  uint8_t* slot_v[2];
  struct Job { int kvh0; int n; };
  std::vector<Job> jobs;
  int staged = 0;  // jobs whose copies are enqueued

  int enqueue_copy(int i) {
    const Job& j = jobs[i];
    const int s = i & 1;
    const int64_t t0 = static_cast<int64_t>(j.n) * p.T;
    const int64_t Tn = std::min<int64_t>(p.T, p.S - t0);
    UPIPE_CUDA(cudaStreamWaitEvent(ds->copy, ds->slot_free[s], 0));
    copy_begin(ds->copy);
    int st = stage_trunk(p, k, slot_k[s], j.kvh0, t0, Tn, ds->copy);
    if (st == UPIPE_OK) st = stage_trunk(p, v, slot_v[s], j.kvh0, t0, Tn, ds->copy);
    copy_end(UPIPE_K_KV_H2D, ds->copy);
    if (st != UPIPE_OK) return st;
    UPIPE_CUDA(cudaEventRecord(ds->slot_ready[s], ds->copy));
    return UPIPE_OK;
  }
  // Before the kernel of job i: its copy (and the next one, as prefetch) are enqueued and the
  // compute stream waits for slot i%2.
  int before(int i) {
    while (staged <= i + 1 && staged < static_cast<int>(jobs.size())) {
      const int st = enqueue_copy(staged);
      if (st != UPIPE_OK) return st;
      ++staged;
    }
    // bracketed when profiling: the gap is the time the compute stream stalled for the copy
    copy_begin(compute);
    UPIPE_CUDA(cudaStreamWaitEvent(compute, ds->slot_ready[i & 1], 0));
    copy_end(UPIPE_K_KV_WAIT, compute);
    return UPIPE_OK;
  }
  int after(int i) {
    UPIPE_CUDA(cudaEventRecord(ds->slot_free[i & 1], compute));
    return UPIPE_OK;
  }
};

}  // namespace

namespace {
std::atomic<int> g_fail_copy_after{0};  // 0: disarmed; n: the n-th staging copy from now fails
}  // namespace

bool staging_copy_fails() {
  int n = g_fail_copy_after.load(std::memory_order_relaxed);
  while (n > 0) {
    if (g_fail_copy_after.compare_exchange_weak(n, n - 1)) return n == 1;
  }
  return false;
}

int upipe_debug_arm_copy_failure(int n) {
  g_fail_copy_after.store(n);
  return UPIPE_OK;
}

int device_status_word(int dev, uint32_t** err) {
  if (dev < 0 || dev >= kMaxDev) return fail(UPIPE_ERR_INVALID_ARG, "device %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DevState* ds = nullptr;
  const int st = dev_state(dev, &ds);
  if (st != UPIPE_OK) return st;
  *err = ds->err;
  return UPIPE_OK;
}

cudaError_t launch_fwd_resident(const AttnPlan& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, int h0, void* o, int o_heads, float* lse,
                                uint32_t* err, cudaStream_t stream) {
  FwdArgs a{};
  a.q_lo = 0;
  a.q_hi = p.S;
  a.kv_row_lo = 0;
  a.kv_row_hi = p.S;
  a.kv_pos0 = 0;
  a.S = p.S;
  a.hc = p.hc; a.kc = p.kc; a.G = p.G; a.Hq = p.Hq; a.h0 = h0;
  a.causal = p.causal; a.first = 1; a.last = 1;
  const float scale = 1.0f / std::sqrt(static_cast<float>(p.D));
  a.scale_log2 = scale * 1.4426950408889634f;
  a.o = o; a.lse = lse;
  a.o_heads = o_heads; a.o_head0 = 0;
  a.state_o = nullptr; a.state_ml = nullptr;
  a.state_rows = 0; a.state_stride = 0;
  a.err = err;
  return launch_attn_fwd(p.D, p.B, tq, tk, tv, a, stream);
}

}  // namespace upipe

using namespace upipe;

extern "C" {

size_t upipe_workspace_bytes(int B, int64_t S, int Hq, int Hkv, int D, int causal,
                             int head_chunk, int64_t seq_trunk, int pass, int host_mask) {
  Plan p;
  if (make_attn_plan(B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk, host_mask, &p) != UPIPE_OK)
    return 0;
  if (pass == UPIPE_PASS_FWD) return p.f_total;
  if (pass == UPIPE_PASS_BWD) return p.b_total;
  if (pass == UPIPE_PASS_BOTH) return std::max(p.f_total, p.b_total);
  return 0;
}

int upipe_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int64_t S, int Hq, int Hkv, int D, int causal, int head_chunk,
                   int64_t seq_trunk, void* workspace, size_t workspace_bytes, void* stream_) {
  const NvtxRange range("upipe_attn_fwd");
  g_last_error.clear();
  // lse may be NULL: a prefill (inference) forward that keeps no statistics for a backward
  if (!q || !k || !v || !o || !workspace)
    return fail(UPIPE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(UPIPE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign)
    return fail(UPIPE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  Plan p0;
  int st = make_attn_plan(B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk, 0, &p0);
  if (st != UPIPE_OK) return st;
  // q and o: device memory of the call's device, or pinned host memory (each on its own)
  int dq_dev = -1, do_dev = -1;
  const int kq = pointer_kind(q, &dq_dev), ko = pointer_kind(o, &do_dev);
  if (kq < 0 || ko < 0)
    return fail(UPIPE_ERR_INVALID_ARG, "q and o must be device memory or pinned host memory");
  const bool q_host = kq == 1, o_host = ko == 1;
  const void* dptrs[4] = {workspace, lse, q, o};
  const char* names[4] = {"workspace", "lse", "q", "o"};
  const void* dlist[4];
  const char* nlist[4];
  int nd = 0;
  for (int i = 0; i < 4; ++i) {
    if (!dptrs[i] || (i == 2 && q_host) || (i == 3 && o_host)) continue;
    dlist[nd] = dptrs[i];
    nlist[nd++] = names[i];
  }
  bool kv_host = false;
  int dev = 0;
  st = check_placement(dlist, nd, nlist, k, v, &kv_host, &dev);
  if (st != UPIPE_OK) return st;
  Plan p;
  make_attn_plan(B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk,
            (kv_host ? UPIPE_HOST_KV : 0) | (q_host || o_host ? UPIPE_HOST_ACT : 0), &p);
  if (workspace_bytes < p.f_total)
    return fail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                p.f_total);

  std::lock_guard<std::mutex> lk(g_mu);
  const DeviceGuard dguard;
  UPIPE_CUDA(cudaSetDevice(dev));
  DevState* ds = nullptr;
  st = dev_state(dev, &ds);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool carried = kv_host && p.n_trunks > 1;  // running state kept between launches
  float* state_o = carried ? reinterpret_cast<float*>(ws + p.f_state_o) : nullptr;
  float* state_ml = carried ? reinterpret_cast<float*>(ws + p.f_state_ml) : nullptr;
  const float scale = 1.0f / std::sqrt(static_cast<float>(D));

  Stager stg{p, ds, stream, k, v, {ws + p.f_slot_k[0], ws + p.f_slot_k[1]},
             {ws + p.f_slot_v[0], ws + p.f_slot_v[1]}, {}, 0};
  if (kv_host) {
    // one staging job per (group, key/value trunk): the trunk serves every query trunk
    for (int g = 0; g < Hq / p.hc; ++g)
      for (int n = 0; n < p.n_trunks; ++n) stg.jobs.push_back({g * p.kc, n});
  }
  if (kv_host || q_host || o_host) {
    // The copy stream must not touch the workspace before earlier work on `stream` is done.
    UPIPE_CUDA(cudaEventRecord(ds->entry, stream));
    UPIPE_CUDA(cudaStreamWaitEvent(ds->copy, ds->entry, 0));
    UPIPE_CUDA(cudaStreamWaitEvent(ds->act_copy, ds->entry, 0));
  }
  const int n_groups = Hq / p.hc;
  auto q_buf = [&](int g) -> uint8_t* { return ws + ((q_host && (g & 1)) ? p.f_qw2 : p.f_qw); };
  // host q: group g's heads go into Q buffer g%2 once group g-2 no longer reads it
  auto stage_q = [&](int g) -> int {
    const int s = g & 1;
    if (g >= 2) UPIPE_CUDA(cudaStreamWaitEvent(ds->act_copy, ds->act_free[s], 0));
    const int r = stage_heads(q, q_buf(g), B, S, Hq, D, g * p.hc, p.hc, ds->act_copy);
    if (r != UPIPE_OK) return r;
    UPIPE_CUDA(cudaEventRecord(ds->act_ready[s], ds->act_copy));
    return UPIPE_OK;
  };
  if (q_host) {
    st = stage_q(0);
    if (st != UPIPE_OK) return st;
  }
  // host o: group g's kernels write a [B, S, hc, D] staging buffer, copied out afterwards
  void* o_out = o;
  // Host K/V: one launch per key/value trunk n over every query row that sees it (rows from
  // n*T on when causal, all rows otherwise). Each query trunk's running state sits in the
  // S-row arena state; a tile finalises when n is its last trunk (its diagonal one when
  // causal), the others store their state for trunk n+1.
  auto launch_trunk = [&](const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          int h0, int n, int64_t Tn) -> int {
    const int64_t t0 = static_cast<int64_t>(n) * p.T;
    FwdArgs a{};
    a.q_lo = causal ? t0 : 0;
    a.q_hi = S;
    a.S = S;
    a.hc = p.hc; a.kc = p.kc; a.G = p.G; a.Hq = Hq; a.h0 = h0;
    a.causal = causal; a.first = (n == 0);
    a.last = causal || n == p.n_trunks - 1;
    a.last_q_end = causal ? std::min<int64_t>(S, t0 + p.T) : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.o = o_out; a.lse = lse;
    if (o_host) { a.o_heads = p.hc; a.o_head0 = 0; }
    // the state rows of this launch start q_lo rows into the S_pad-row state
    a.state_o = state_o ? state_o + a.q_lo * D : nullptr;
    a.state_ml = state_ml ? state_ml + a.q_lo * 2 : nullptr;
    a.state_rows = p.S_pad - a.q_lo;
    a.state_stride = p.S_pad;
    a.err = ds->err;
    a.kv_row_lo = 0; a.kv_row_hi = Tn; a.kv_pos0 = t0;
    UPIPE_CUDA(launch_attn_fwd(D, B, tq, tk, tv, a, stream));
    return UPIPE_OK;
  };
  int job = 0;
  for (int g = 0; g < n_groups; ++g) {
    const NvtxRange range("upipe fwd head group %lld", g);
    const int h0 = g * p.hc, kvh0 = g * p.kc;
    const int gs = g & 1;
    uint8_t* qwg = q_buf(g);
    if (q_host) {
      if (g + 1 < n_groups) {  // prefetch the next group's Q while this group computes
        st = stage_q(g + 1);
        if (st != UPIPE_OK) return st;
      }
      UPIPE_CUDA(cudaStreamWaitEvent(stream, ds->act_ready[gs], 0));
    }
    if (o_host) {
      // the staging this group writes must have reached the host from group g-2
      if (g >= 2) UPIPE_CUDA(cudaStreamWaitEvent(stream, ds->out_free[gs], 0));
      o_out = ws + p.f_ostg[gs];
    }
    {
      // the group's device-resident Q, K and V gathered head-major in one launch
      GatherList gl;
      if (!q_host) gl.add(q, qwg, Hq, h0, p.hc);
      if (!kv_host) {
        gl.add(k, ws + p.f_kw, Hkv, kvh0, p.kc);
        gl.add(v, ws + p.f_vw, Hkv, kvh0, p.kc);
      }
      UPIPE_CUDA(gl.launch(B, S, D, stream));
    }
    CUtensorMap tq, tk, tv;
    UPIPE_CUDA(make_tmap_bf16(&tq, qwg, D, S, static_cast<int64_t>(B) * p.hc));
    if (!kv_host) {
      // Device-resident K/V: one launch folds every key/value trunk into every query row, the
      // running softmax state of each query tile staying in TMEM and registers from the first
      // key tile to the last (FPDT's trunk loop, run inside the kernel).
      UPIPE_CUDA(make_tmap_bf16(&tk, ws + p.f_kw, D, S, static_cast<int64_t>(B) * p.kc));
      UPIPE_CUDA(make_tmap_bf16(&tv, ws + p.f_vw, D, S, static_cast<int64_t>(B) * p.kc));
      UPIPE_CUDA(launch_fwd_resident(p, tq, tk, tv, h0, o_out, o_host ? p.hc : 0, lse, ds->err,
                                     stream));
    } else {
      // Host K/V: key/value trunk n is staged once and then met, in one launch, by every
      // query trunk that sees it (m >= n when causal).
      for (int n = 0; n < p.n_trunks; ++n, ++job) {
        const int64_t t0 = static_cast<int64_t>(n) * p.T;
        const int64_t Tn = std::min<int64_t>(p.T, S - t0);
        st = stg.before(job);
        if (st != UPIPE_OK) return st;
        const int s = job & 1;
        UPIPE_CUDA(make_tmap_bf16(&tk, stg.slot_k[s], D, Tn, static_cast<int64_t>(B) * p.kc));
        UPIPE_CUDA(make_tmap_bf16(&tv, stg.slot_v[s], D, Tn, static_cast<int64_t>(B) * p.kc));
        st = launch_trunk(tq, tk, tv, h0, n, Tn);
        if (st != UPIPE_OK) return st;
        st = stg.after(job);
        if (st != UPIPE_OK) return st;
      }
    }
    // end of group g: its Q buffer is free again; its O staging goes to the host
    if (q_host) UPIPE_CUDA(cudaEventRecord(ds->act_free[gs], stream));
    if (o_host) {
      UPIPE_CUDA(cudaEventRecord(ds->out_done[gs], stream));
      UPIPE_CUDA(cudaStreamWaitEvent(ds->act_copy, ds->out_done[gs], 0));
      st = unstage_heads(ws + p.f_ostg[gs], o, B, S, Hq, D, h0, p.hc, ds->act_copy);
      if (st != UPIPE_OK) return st;
      UPIPE_CUDA(cudaEventRecord(ds->out_free[gs], ds->act_copy));
    }
  }
  if (o_host) {
    // the caller's stream completes only after the last group's O reached the host
    UPIPE_CUDA(cudaEventRecord(ds->act_done, ds->act_copy));
    UPIPE_CUDA(cudaStreamWaitEvent(stream, ds->act_done, 0));
  }
  return UPIPE_OK;
}

int upipe_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, int B, int64_t S, int Hq,
                   int Hkv, int D, int causal, int head_chunk, int64_t seq_trunk,
                   void* workspace, size_t workspace_bytes, void* stream_) {
  const NvtxRange range("upipe_attn_bwd");
  g_last_error.clear();
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return fail(UPIPE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(UPIPE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign)
    return fail(UPIPE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  Plan p0;
  int st = make_attn_plan(B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk, 0, &p0);
  if (st != UPIPE_OK) return st;
  // q, o, dout, dq: device memory of the call's device, or pinned host memory (each on its own)
  const void* act[4] = {q, o, dout, dq};
  const char* act_names[4] = {"q", "o", "dout", "dq"};
  bool act_host[4];
  const void* dlist[6] = {lse, workspace};
  const char* nlist[6] = {"lse", "workspace"};
  int nd = 2;
  for (int i = 0; i < 4; ++i) {
    int d = -1;
    const int kind = pointer_kind(act[i], &d);
    if (kind < 0)
      return fail(UPIPE_ERR_INVALID_ARG, "%s must be device memory or pinned host memory",
                  act_names[i]);
    act_host[i] = kind == 1;
    if (!act_host[i]) {
      dlist[nd] = act[i];
      nlist[nd++] = act_names[i];
    }
  }
  const bool q_host = act_host[0], o_host = act_host[1], dout_host = act_host[2],
             dq_host = act_host[3];
  const bool any_act = q_host || o_host || dout_host || dq_host;
  // with a host o or dout the pre-pass reads head-major copies of both
  const bool hm_pre = o_host || dout_host;
  bool kv_host = false;
  int dev = 0;
  st = check_placement(dlist, nd, nlist, k, v, &kv_host, &dev);
  if (st != UPIPE_OK) return st;
  // dk/dv: device memory, or (with host k/v) both pinned host memory, written trunk by trunk
  int ddk = -1, ddv = -1;
  const int kdk = pointer_kind(dk, &ddk), kdv = pointer_kind(dv, &ddv);
  if (kdk != kdv || kdk < 0)
    return fail(UPIPE_ERR_INVALID_ARG, "dk and dv must both be device memory or both pinned host memory");
  if (kdk == 0 && (ddk != dev || ddv != dev))
    return fail(UPIPE_ERR_INVALID_ARG, "dk/dv are on another device");
  const bool dkdv_host = kdk == 1;
  if (dkdv_host && !kv_host)
    return fail(UPIPE_ERR_INVALID_ARG, "dk/dv may be pinned host memory only when k/v are too");
  Plan p;
  make_attn_plan(B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk,
            (kv_host ? UPIPE_HOST_KV : 0) | (any_act ? UPIPE_HOST_ACT : 0), &p);
  if (workspace_bytes < p.b_total)
    return fail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                p.b_total);

  std::lock_guard<std::mutex> lk(g_mu);
  const DeviceGuard dguard;
  UPIPE_CUDA(cudaSetDevice(dev));
  DevState* ds = nullptr;
  st = dev_state(dev, &ds);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* dqacc = reinterpret_cast<float*>(ws + p.b_dqacc);
  float* lse2 = reinterpret_cast<float*>(ws + p.b_lse2);
  float* dvec = reinterpret_cast<float*>(ws + p.b_dvec);
  const float scale = 1.0f / std::sqrt(static_cast<float>(D));

  Stager stg{p, ds, stream, k, v, {ws + p.b_slot_k[0], ws + p.b_slot_k[1]},
             {ws + p.b_slot_v[0], ws + p.b_slot_v[1]}, {}, 0};
  if (kv_host) {
    for (int g = 0; g < Hq / p.hc; ++g)
      for (int n = 0; n < p.n_trunks; ++n) stg.jobs.push_back({g * p.kc, n});
  }
  if (kv_host || any_act) {
    // The copy stream must not touch the workspace before earlier work on `stream` is done.
    UPIPE_CUDA(cudaEventRecord(ds->entry, stream));
    UPIPE_CUDA(cudaStreamWaitEvent(ds->copy, ds->entry, 0));
    UPIPE_CUDA(cudaStreamWaitEvent(ds->act_copy, ds->entry, 0));
  }
  const int n_groups = Hq / p.hc;
  // Per head group g, buffers g%2 when host activations rotate through them.
  auto qw_of = [&](int g) -> uint8_t* { return ws + ((q_host && (g & 1)) ? p.b_qw2 : p.b_qw); };
  auto dow_of = [&](int g) -> uint8_t* {
    return ws + ((hm_pre && (g & 1)) ? p.b_dow2 : p.b_dow);
  };
  auto ow_of = [&](int g) -> uint8_t* { return ws + p.b_ow[g & 1]; };
  const bool stage_any = q_host || o_host || dout_host;
  // host q / o / dout: group g's heads are copied head-major once group g-2 is done with them
  auto stage_act = [&](int g) -> int {
    const int s = g & 1, h0 = g * p.hc;
    if (g >= 2) UPIPE_CUDA(cudaStreamWaitEvent(ds->act_copy, ds->act_free[s], 0));
    int r = UPIPE_OK;
    if (q_host) r = stage_heads(q, qw_of(g), B, S, Hq, D, h0, p.hc, ds->act_copy);
    if (r == UPIPE_OK && o_host)
      r = stage_heads(o, ow_of(g), B, S, Hq, D, h0, p.hc, ds->act_copy);
    if (r == UPIPE_OK && dout_host)
      r = stage_heads(dout, dow_of(g), B, S, Hq, D, h0, p.hc, ds->act_copy);
    if (r != UPIPE_OK) return r;
    UPIPE_CUDA(cudaEventRecord(ds->act_ready[s], ds->act_copy));
    return UPIPE_OK;
  };
  if (stage_any) {
    st = stage_act(0);
    if (st != UPIPE_OK) return st;
  }
  int job = 0;
  for (int g = 0; g < n_groups; ++g) {
    const NvtxRange range("upipe bwd head group %lld", g);
    const int h0 = g * p.hc, kvh0 = g * p.kc;
    const int gs = g & 1;
    void* qw = qw_of(g);
    void* dow = dow_of(g);
    if (stage_any) {
      if (g + 1 < n_groups) {  // prefetch the next group's activations
        st = stage_act(g + 1);
        if (st != UPIPE_OK) return st;
      }
      UPIPE_CUDA(cudaStreamWaitEvent(stream, ds->act_ready[gs], 0));
    }
    {
      GatherList gl;
      if (!q_host) gl.add(q, qw, Hq, h0, p.hc);
      if (!kv_host) {
        gl.add(k, ws + p.b_kw, Hkv, kvh0, p.kc);
        gl.add(v, ws + p.b_vw, Hkv, kvh0, p.kc);
      }
      UPIPE_CUDA(gl.launch(B, S, D, stream));
    }
    if (hm_pre) {
      void* ow = ow_of(g);
      if (!o_host) UPIPE_CUDA(launch_seq_to_head(o, ow, B, S, Hq, D, h0, p.hc, stream));
      if (!dout_host) UPIPE_CUDA(launch_seq_to_head(dout, dow, B, S, Hq, D, h0, p.hc, stream));
      UPIPE_CUDA(launch_bwd_pre(ow, dow, lse, dow, dvec, lse2, dqacc, B, S, p.S_pad, Hq, D, h0,
                                p.hc, scale, 1, stream));
    } else {
      UPIPE_CUDA(launch_bwd_pre(o, dout, lse, dow, dvec, lse2, dqacc, B, S, p.S_pad, Hq, D, h0,
                                p.hc, scale, 0, stream));
    }
    CUtensorMap tq, tdo, tk, tv;
    UPIPE_CUDA(make_tmap_bf16(&tq, qw, D, S, static_cast<int64_t>(B) * p.hc, bwd_q_box_rows(D)));
    UPIPE_CUDA(make_tmap_bf16(&tdo, dow, D, S, static_cast<int64_t>(B) * p.hc, bwd_q_box_rows(D)));
    if (!kv_host) {
      UPIPE_CUDA(make_tmap_bf16(&tk, ws + p.b_kw, D, S, static_cast<int64_t>(B) * p.kc));
      UPIPE_CUDA(make_tmap_bf16(&tv, ws + p.b_vw, D, S, static_cast<int64_t>(B) * p.kc));
    }
    // Host K/V: one launch per key/value trunk (each staged once). Device-resident K/V: one
    // launch over every key tile; each CTA's walk over the query tiles that see its key tile
    // is the same either way, so only the number of launches differs.
    const int n_launch = kv_host ? p.n_trunks : 1;
    const int64_t T_launch = kv_host ? p.T : S;
    for (int n = 0; n < n_launch; ++n, ++job) {
      const int64_t t0 = static_cast<int64_t>(n) * T_launch;
      const int64_t Tn = std::min<int64_t>(T_launch, S - t0);
      BwdArgs a{};
      a.S = S; a.S_pad = p.S_pad;
      a.hc = p.hc; a.kc = p.kc; a.G = p.G; a.Hkv = Hkv; a.kvh0 = kvh0;
      a.causal = causal; a.scale = scale; a.scale_log2 = scale * 1.4426950408889634f;
      a.lse2 = lse2; a.dvec = dvec; a.dqacc = dqacc; a.err = ds->err;
      const int s = job & 1;
      if (dkdv_host) {
        // the slot's previous trunk must have reached the host before it is overwritten
        if (job >= 2) UPIPE_CUDA(cudaStreamWaitEvent(stream, ds->dkdv_free[s], 0));
        a.dk = ws + p.b_slot_dk[s]; a.dv = ws + p.b_slot_dv[s];
        a.dkv_rows = Tn; a.dkv_row0 = t0; a.dkv_heads = p.kc; a.dkv_head0 = 0;
      } else {
        a.dk = dk; a.dv = dv;
        a.dkv_rows = S; a.dkv_row0 = 0; a.dkv_heads = Hkv; a.dkv_head0 = kvh0;
      }
      if (kv_host) {
        st = stg.before(job);
        if (st != UPIPE_OK) return st;
        UPIPE_CUDA(make_tmap_bf16(&tk, stg.slot_k[s], D, Tn, static_cast<int64_t>(B) * p.kc));
        UPIPE_CUDA(make_tmap_bf16(&tv, stg.slot_v[s], D, Tn, static_cast<int64_t>(B) * p.kc));
        a.kv_row_lo = 0; a.kv_row_hi = Tn; a.kv_pos0 = t0;
      } else {
        a.kv_row_lo = t0; a.kv_row_hi = t0 + Tn; a.kv_pos0 = 0;
      }
      a.split = p.bwd_split;
      a.dkv_part = p.bwd_split > 1 ? reinterpret_cast<float*>(ws + p.b_dkv_part) : nullptr;
      a.part_rows = p.part_rows;
      UPIPE_CUDA(launch_attn_bwd(D, B, tq, tdo, tk, tv, a, stream));
      if (p.bwd_split > 1)
        UPIPE_CUDA(launch_dkdv_reduce(a.dkv_part, p.bwd_split, p.part_rows, Tn, t0, B, p.kc, D,
                                      S, a.dk, a.dv, a.dkv_rows, a.dkv_row0, a.dkv_heads,
                                      a.dkv_head0, stream));
      if (kv_host) {
        st = stg.after(job);
        if (st != UPIPE_OK) return st;
      }
      if (dkdv_host) {
        // this trunk's dK/dV are final: copy them out on the copy stream
        UPIPE_CUDA(cudaEventRecord(ds->dkdv_done[s], stream));
        UPIPE_CUDA(cudaStreamWaitEvent(ds->copy, ds->dkdv_done[s], 0));
        copy_begin(ds->copy);
        st = unstage_trunk(p, ws + p.b_slot_dk[s], dk, kvh0, t0, Tn, ds->copy);
        if (st == UPIPE_OK) st = unstage_trunk(p, ws + p.b_slot_dv[s], dv, kvh0, t0, Tn, ds->copy);
        copy_end(UPIPE_K_DKDV_D2H, ds->copy);
        if (st != UPIPE_OK) return st;
        UPIPE_CUDA(cudaEventRecord(ds->dkdv_free[s], ds->copy));
      }
    }
    if (stage_any) UPIPE_CUDA(cudaEventRecord(ds->act_free[gs], stream));
    if (dq_host) {
      // this group's dQ goes to staging g%2 (free once group g-2's copy-out is done), then out
      if (g >= 2) UPIPE_CUDA(cudaStreamWaitEvent(stream, ds->out_free[gs], 0));
      UPIPE_CUDA(launch_dq_convert(dqacc, ws + p.b_dqs[gs], B, S, p.S_pad, p.hc, D, 0, p.hc,
                                   stream));
      UPIPE_CUDA(cudaEventRecord(ds->out_done[gs], stream));
      UPIPE_CUDA(cudaStreamWaitEvent(ds->act_copy, ds->out_done[gs], 0));
      st = unstage_heads(ws + p.b_dqs[gs], dq, B, S, Hq, D, h0, p.hc, ds->act_copy);
      if (st != UPIPE_OK) return st;
      UPIPE_CUDA(cudaEventRecord(ds->out_free[gs], ds->act_copy));
    } else {
      UPIPE_CUDA(launch_dq_convert(dqacc, dq, B, S, p.S_pad, Hq, D, h0, p.hc, stream));
    }
  }
  // the caller's stream completes only after the last copy to the host
  if (dkdv_host) {
    UPIPE_CUDA(cudaEventRecord(ds->copy_done, ds->copy));
    UPIPE_CUDA(cudaStreamWaitEvent(stream, ds->copy_done, 0));
  }
  if (dq_host) {
    UPIPE_CUDA(cudaEventRecord(ds->act_done, ds->act_copy));
    UPIPE_CUDA(cudaStreamWaitEvent(stream, ds->act_done, 0));
  }
  return UPIPE_OK;
}

static int layout_args(const void* src, const void* dst, int B, int64_t S, int H, int D,
                       int h_begin, int h_count, int* dev) {
  if (!src || !dst) return fail(UPIPE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(src) || !aligned16(dst))
    return fail(UPIPE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (B < 1 || S < 1 || H < 1 || D < 8 || D % 8)
    return fail(UPIPE_ERR_INVALID_ARG, "bad sizes (B=%d S=%lld H=%d D=%d; D %% 8 == 0)", B,
                static_cast<long long>(S), H, D);
  if (h_begin < 0 || h_count < 1 || h_begin + h_count > H)
    return fail(UPIPE_ERR_INVALID_ARG, "head range [%d, %d) outside [0, %d)", h_begin,
                h_begin + h_count, H);
  int d1 = -1, d2 = -1;
  if (pointer_kind(src, &d1) != 0 || pointer_kind(dst, &d2) != 0 || d1 != d2)
    return fail(UPIPE_ERR_INVALID_ARG, "src and dst must be memory of one device");
  *dev = d1;
  return UPIPE_OK;
}

int upipe_seq_to_head_major(const void* src, void* dst, int B, int64_t S, int H, int D,
                            int h_begin, int h_count, void* stream) {
  g_last_error.clear();
  int dev = 0;
  const int st = layout_args(src, dst, B, S, H, D, h_begin, h_count, &dev);
  if (st != UPIPE_OK) return st;
  const DeviceGuard dguard;
  UPIPE_CUDA(cudaSetDevice(dev));
  UPIPE_CUDA(launch_seq_to_head(src, dst, B, S, H, D, h_begin, h_count,
                                static_cast<cudaStream_t>(stream)));
  return UPIPE_OK;
}

int upipe_head_to_seq_major(const void* src, void* dst, int B, int64_t S, int H, int D,
                            int h_begin, int h_count, void* stream) {
  g_last_error.clear();
  int dev = 0;
  const int st = layout_args(src, dst, B, S, H, D, h_begin, h_count, &dev);
  if (st != UPIPE_OK) return st;
  const DeviceGuard dguard;
  UPIPE_CUDA(cudaSetDevice(dev));
  UPIPE_CUDA(launch_head_to_seq(src, dst, B, S, H, D, h_begin, h_count,
                                static_cast<cudaStream_t>(stream)));
  return UPIPE_OK;
}

int upipe_sync_status(void* stream) {
  g_last_error.clear();
  UPIPE_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int dev = 0;
  UPIPE_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev < 0 || dev >= kMaxDev || !g_dev[dev].ready) return UPIPE_OK;
  uint32_t w = 0;
  UPIPE_CUDA(cudaMemcpy(&w, g_dev[dev].err, sizeof(w), cudaMemcpyDeviceToHost));
  if (w) {
    UPIPE_CUDA(cudaMemset(g_dev[dev].err, 0, sizeof(w)));
    return fail(UPIPE_ERR_TIMEOUT, "device status word 0x%x: a bounded wait expired", w);
  }
  return UPIPE_OK;
}

const char* upipe_status_string(int status) {
  switch (status) {
    case UPIPE_OK: return "UPIPE_OK";
    case UPIPE_ERR_INVALID_ARG: return "UPIPE_ERR_INVALID_ARG";
    case UPIPE_ERR_UNSUPPORTED: return "UPIPE_ERR_UNSUPPORTED";
    case UPIPE_ERR_WORKSPACE_TOO_SMALL: return "UPIPE_ERR_WORKSPACE_TOO_SMALL";
    case UPIPE_ERR_CUDA: return "UPIPE_ERR_CUDA";
    case UPIPE_ERR_TIMEOUT: return "UPIPE_ERR_TIMEOUT";
    default: return "UPIPE_ERR_UNKNOWN";
  }
}

const char* upipe_last_error_message(void) { return g_last_error.c_str(); }

void upipe_shutdown(void) {
  const DeviceGuard dguard;
  upipe::seqtile_shutdown();
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < kMaxDev; ++i) {
    DevState& d = g_dev[i];
    if (!d.ready) continue;
    cudaSetDevice(i);
    cudaStreamSynchronize(d.copy);
    cudaStreamDestroy(d.copy);
    cudaStreamSynchronize(d.act_copy);
    cudaStreamDestroy(d.act_copy);
    for (int s = 0; s < 2; ++s) {
      cudaEventDestroy(d.slot_ready[s]);
      cudaEventDestroy(d.slot_free[s]);
      cudaEventDestroy(d.dkdv_done[s]);
      cudaEventDestroy(d.dkdv_free[s]);
      cudaEventDestroy(d.act_ready[s]);
      cudaEventDestroy(d.act_free[s]);
      cudaEventDestroy(d.out_done[s]);
      cudaEventDestroy(d.out_free[s]);
    }
    cudaEventDestroy(d.entry);
    cudaEventDestroy(d.copy_done);
    cudaEventDestroy(d.act_done);
    cudaFree(d.err);
    d = DevState{};
  }
}

uint64_t upipe_launch_count(void) { return g_launches.load(); }

int upipe_debug_fail_copy_after(int n) {
  g_last_error.clear();
  if (n < 0) return fail(UPIPE_ERR_INVALID_ARG, "n must be >= 0");
  return upipe::upipe_debug_arm_copy_failure(n);
}

int upipe_profile_enable(int on) {
  g_profile.store(on != 0);
  return UPIPE_OK;
}

int upipe_profile_read(upipe_kernel_stat* out, int n) {
  g_last_error.clear();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (const ProfRec& r : g_prof) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(r.e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.e0, r.e1);
    if (e != cudaSuccess) return cuda_fail(e, "profile event");
    if (out && r.kclass >= 0 && r.kclass < n) {
      out[r.kclass].total_ms += ms;
      out[r.kclass].launches += 1;
    }
    g_event_pool.push_back(r.e0);
    g_event_pool.push_back(r.e1);
  }
  g_prof.clear();
  return UPIPE_OK;
}

int upipe_selftest_umma(const void* a, const void* b, float* c, int N, int K, int a_mn_major,
                        int b_mn_major, int a_manual, int lbo, int sbo, void* stream) {
  g_last_error.clear();
  if (!a || !b || !c || !aligned16(a) || !aligned16(b) || !aligned16(c))
    return fail(UPIPE_ERR_INVALID_ARG, "null or unaligned pointer");
  if ((N != 64 && N != 128) || (K != 64 && K != 128))
    return fail(UPIPE_ERR_INVALID_ARG, "N and K must be 64 or 128");
  if (a_manual < 0 || a_manual > 2) return fail(UPIPE_ERR_INVALID_ARG, "a_manual must be 0, 1 or 2");
  if (a_manual && a_mn_major) return fail(UPIPE_ERR_INVALID_ARG, "a_manual needs a K-major A");
  if (lbo < 16 || lbo > 65536 || sbo < 16 || sbo > 65536 || lbo % 16 || sbo % 16)
    return fail(UPIPE_ERR_INVALID_ARG, "lbo/sbo must be multiples of 16 in [16, 65536]");
  // The descriptors may only address the two 32 KiB operand tiles.
  if ((a_mn_major || b_mn_major) && 7 * 2048 + lbo + sbo + 1024 > 32768)
    return fail(UPIPE_ERR_INVALID_ARG, "lbo/sbo would address outside the operand tile");
  int dev = -1, d2 = -1, d3 = -1;
  if (pointer_kind(a, &dev) != 0 || pointer_kind(b, &d2) != 0 || pointer_kind(c, &d3) != 0 ||
      dev != d2 || dev != d3)
    return fail(UPIPE_ERR_INVALID_ARG, "a, b, c must be memory of one device");
  std::lock_guard<std::mutex> lk(g_mu);
  const DeviceGuard dguard;
  UPIPE_CUDA(cudaSetDevice(dev));
  DevState* ds = nullptr;
  const int st = dev_state(dev, &ds);
  if (st != UPIPE_OK) return st;
  UPIPE_CUDA(launch_selftest_umma(a, b, c, N, K, a_mn_major, b_mn_major, a_manual, lbo, sbo,
                                  ds->err, static_cast<cudaStream_t>(stream)));
  return UPIPE_OK;
}

int upipe_selftest_wait_timeout(int limit_us, void* stream) {
  g_last_error.clear();
  if (limit_us < 1 || limit_us > 2000000)
    return fail(UPIPE_ERR_INVALID_ARG, "limit_us must be in [1, 2000000]");
  int dev = 0;
  UPIPE_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_mu);
  DevState* ds = nullptr;
  const int st = dev_state(dev, &ds);
  if (st != UPIPE_OK) return st;
  UPIPE_CUDA(launch_selftest_wait(limit_us, ds->err, static_cast<cudaStream_t>(stream)));
  return UPIPE_OK;
}

}  // extern "C"
