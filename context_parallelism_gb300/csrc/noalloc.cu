// Forward attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs under an allocator that owns every
// device byte (a framework's caching allocator or a fixed memory pool that must not be bypassed),
// real-time or embedded code that forbids allocation after start-up, or plugins that are handed
// only their input and output buffers. For them this file holds the forward's scratch in a
// file-scope static device array: it is created when the library's device code is loaded on a
// GPU and stays there until the process exits; no call allocates or frees anything.
//
// The set-up (once per device, on the first call with that device current) asks the runtime
// for the device address of the array with cudaGetSymbolAddress: in host code the array's name
// is only a host-side stand-in, never a device address, so it is never passed to a kernel.
//
// Every call shares the one array, which keeps the last call's contents. The forward needs no
// zeroed scratch: each call writes every byte it later reads (the gathers fill Q/K/V before
// the attention launch reads them; the running softmax state stays on chip). Calls
// whose work overlaps on the GPU (on different streams, or from different host threads without
// ordering) race on the array and must be serialised by the caller.
#include <mutex>

#include "upipe.h"
#include "internal.h"

namespace upipe {
namespace {

// 32 MiB: enough for the Llama3-8B-shaped layer at S = 8192 with head_chunk 8 (24 MiB) and
// everything smaller.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
static __device__ __align__(256) uint32_t g_noalloc_status[64];

struct NoAllocDevice {
  bool ready = false;
  uint8_t* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  uint32_t* status = nullptr;   // device address of g_noalloc_status on this device
};
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[64];

int na_fail(int status, const char* msg) {
  set_last_error(msg);
  return status;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" int upipe_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int64_t S, int Hq, int Hkv, int D,
                                      int causal, int head_chunk, int64_t seq_trunk,
                                      int check_status, void* stream_) {
  const NvtxRange range("upipe_attn_fwd_noalloc");
  set_last_error("");
  if (!q || !k || !v || !o || !lse) return na_fail(UPIPE_ERR_INVALID_ARG, "null pointer argument");
  for (const void* p : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)})
    if (reinterpret_cast<uintptr_t>(p) & 15u)
      return na_fail(UPIPE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  // The shape rules, status codes and arena layout of upipe_attn_fwd with device-resident K/V:
  // the same plan places the segments, here inside the static array.
  AttnPlan p;
  const int plan_st = make_attn_plan(B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk, 0, &p);
  if (plan_st != UPIPE_OK) return plan_st;  // the plan recorded the reason
  if (p.f_total > kNoAllocScratchBytes)
    return na_fail(UPIPE_ERR_WORKSPACE_TOO_SMALL,
                   "problem needs more forward scratch than the 32 MiB static array");
  int dev = -1;
  for (const void* ptr : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)}) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess || at.type != cudaMemoryTypeDevice) {
      cudaGetLastError();
      return na_fail(UPIPE_ERR_INVALID_ARG, "q, k, v, o and lse must all be device memory");
    }
    if (dev < 0) dev = at.device;
    if (at.device != dev) return na_fail(UPIPE_ERR_INVALID_ARG, "tensors on different devices");
  }
  if (dev >= 64) return na_fail(UPIPE_ERR_UNSUPPORTED, "device index >= 64");

  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  const DeviceGuard dguard;
  if (cudaSetDevice(dev) != cudaSuccess) return na_fail(UPIPE_ERR_CUDA, "cudaSetDevice failed");
  NoAllocDevice& nd = g_noalloc_dev[dev];
  if (!nd.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return na_fail(UPIPE_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed");
    nd.scratch = static_cast<uint8_t*>(ptr);
    if (cudaGetSymbolAddress(&ptr, g_noalloc_status) != cudaSuccess || !ptr)
      return na_fail(UPIPE_ERR_CUDA, "cudaGetSymbolAddress(status) failed");
    nd.status = static_cast<uint32_t*>(ptr);
    if (cudaMemset(nd.status, 0, sizeof(g_noalloc_status)) != cudaSuccess)
      return na_fail(UPIPE_ERR_CUDA, "clearing the status word failed");
    nd.ready = true;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (check_status) {
    // Opt-in, blocking: reports a bounded wait that expired in an earlier call's kernels.
    uint32_t w = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess ||
        cudaMemcpy(&w, nd.status, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess)
      return na_fail(UPIPE_ERR_CUDA, "reading the status word failed");
    if (w) {
      cudaMemset(nd.status, 0, sizeof(w));
      return na_fail(UPIPE_ERR_TIMEOUT, "a bounded wait expired in an earlier call");
    }
  }

  uint8_t* qw = nd.scratch + p.f_qw;
  uint8_t* kw = nd.scratch + p.f_kw;
  uint8_t* vw = nd.scratch + p.f_vw;
  for (int g = 0; g < Hq / p.hc; ++g) {
    const int h0 = g * p.hc, kvh0 = g * p.kc;
    const void* src[3] = {q, k, v};
    void* dst[3] = {qw, kw, vw};
    const int H[3] = {Hq, Hkv, Hkv}, first[3] = {h0, kvh0, kvh0}, cnt[3] = {p.hc, p.kc, p.kc};
    if (launch_gather_group(src, dst, H, first, cnt, 3, B, S, D, stream) != cudaSuccess)
      return na_fail(UPIPE_ERR_CUDA, "gather launch failed");
    CUtensorMap tq, tk, tv;
    if (make_tmap_bf16(&tq, qw, D, S, int64_t(B) * p.hc) != cudaSuccess ||
        make_tmap_bf16(&tk, kw, D, S, int64_t(B) * p.kc) != cudaSuccess ||
        make_tmap_bf16(&tv, vw, D, S, int64_t(B) * p.kc) != cudaSuccess)
      return na_fail(UPIPE_ERR_CUDA, "tensor map encoding failed");
    // the launch upipe_attn_fwd makes for device-resident tensors
    if (launch_fwd_resident(p, tq, tk, tv, h0, o, 0, lse, nd.status, stream) != cudaSuccess)
      return na_fail(UPIPE_ERR_CUDA, "attention launch failed");
  }
  return UPIPE_OK;
}
