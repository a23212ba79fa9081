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
// zeroed scratch: each call writes every byte it later reads (the gathers fill Q/K/V, and the
// first key/value trunk writes the carried softmax state before later trunks read it). Calls
// whose work overlaps on the GPU (on different streams, or from different host threads without
// ordering) race on the array and must be serialised by the caller.
#include <cmath>
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

constexpr size_t na_align(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" int upipe_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int64_t S, int Hq, int Hkv, int D,
                                      int causal, int head_chunk, int64_t seq_trunk,
                                      int check_status, void* stream_) {
  if (!q || !k || !v || !o || !lse) return na_fail(UPIPE_ERR_INVALID_ARG, "null pointer argument");
  for (const void* p : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)})
    if (reinterpret_cast<uintptr_t>(p) & 15u)
      return na_fail(UPIPE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  // The same shape rules and arena layout as upipe_attn_fwd with device-resident K/V.
  const size_t need = upipe_workspace_bytes(B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk,
                                            UPIPE_PASS_FWD, 0);
  if (need == 0) return UPIPE_ERR_INVALID_ARG;  // the sizing call recorded the reason
  if (need > kNoAllocScratchBytes)
    return na_fail(UPIPE_ERR_WORKSPACE_TOO_SMALL,
                   "problem needs more forward scratch than the 32 MiB static array");
  int dev = -1;
  for (const void* p : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)}) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess || at.type != cudaMemoryTypeDevice) {
      cudaGetLastError();
      return na_fail(UPIPE_ERR_INVALID_ARG, "q, k, v, o and lse must all be device memory");
    }
    if (dev < 0) dev = at.device;
    if (at.device != dev) return na_fail(UPIPE_ERR_INVALID_ARG, "tensors on different devices");
  }
  if (dev >= 64) return na_fail(UPIPE_ERR_UNSUPPORTED, "device index >= 64");

  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (cudaSetDevice(dev) != cudaSuccess) return na_fail(UPIPE_ERR_CUDA, "cudaSetDevice failed");
  NoAllocDevice& nd = g_noalloc_dev[dev];
  if (!nd.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
      return na_fail(UPIPE_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed");
    nd.scratch = static_cast<uint8_t*>(p);
    if (cudaGetSymbolAddress(&p, g_noalloc_status) != cudaSuccess || !p)
      return na_fail(UPIPE_ERR_CUDA, "cudaGetSymbolAddress(status) failed");
    nd.status = static_cast<uint32_t*>(p);
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

  // Arena: Qw [B*hc][S][D], Kw and Vw [B*kc][S][D], then the trunk state when T < S.
  const int G = Hq / Hkv, hc = head_chunk, kc = head_chunk / G;
  const int64_t T = seq_trunk >= S ? S : seq_trunk;
  const int64_t T_pad = (T + 127) / 128 * 128;
  const int n_trunks = static_cast<int>((S + T - 1) / T);
  const size_t qw_b = size_t(B) * hc * S * D * 2, kv_b = size_t(B) * kc * S * D * 2;
  uint8_t* qw = nd.scratch;
  uint8_t* kw = qw + na_align(qw_b);
  uint8_t* vw = kw + na_align(kv_b);
  float* state_o = reinterpret_cast<float*>(vw + na_align(kv_b));
  float* state_ml =
      reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(state_o) +
                               na_align(size_t(B) * hc * T_pad * D * 4));
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));

  for (int g = 0; g < Hq / hc; ++g) {
    const int h0 = g * hc, kvh0 = g * kc;
    if (launch_seq_to_head(q, qw, B, S, Hq, D, h0, hc, stream) != cudaSuccess ||
        launch_seq_to_head(k, kw, B, S, Hkv, D, kvh0, kc, stream) != cudaSuccess ||
        launch_seq_to_head(v, vw, B, S, Hkv, D, kvh0, kc, stream) != cudaSuccess)
      return na_fail(UPIPE_ERR_CUDA, "gather launch failed");
    CUtensorMap tq, tk, tv;
    if (make_tmap_bf16(&tq, qw, D, S, int64_t(B) * hc) != cudaSuccess ||
        make_tmap_bf16(&tk, kw, D, S, int64_t(B) * kc) != cudaSuccess ||
        make_tmap_bf16(&tv, vw, D, S, int64_t(B) * kc) != cudaSuccess)
      return na_fail(UPIPE_ERR_CUDA, "tensor map encoding failed");
    for (int m = 0; m < n_trunks; ++m) {
      const int n_last = causal ? m : n_trunks - 1;
      for (int n = 0; n <= n_last; ++n) {
        FwdArgs a{};
        a.q_lo = int64_t(m) * T;
        a.q_hi = a.q_lo + T < S ? a.q_lo + T : S;
        a.kv_row_lo = int64_t(n) * T;
        a.kv_row_hi = a.kv_row_lo + T < S ? a.kv_row_lo + T : S;
        a.kv_pos0 = 0;
        a.S = S; a.hc = hc; a.kc = kc; a.G = G; a.Hq = Hq; a.h0 = h0;
        a.causal = causal; a.first = (n == 0); a.last = (n == n_last);
        a.scale_log2 = scale_log2;
        a.o = o; a.lse = lse;
        a.state_o = n_trunks > 1 ? state_o : nullptr;
        a.state_ml = n_trunks > 1 ? state_ml : nullptr;
        a.state_rows = T_pad;
        a.err = nd.status;
        if (launch_attn_fwd(D, B, tq, tk, tv, a, stream) != cudaSuccess)
          return na_fail(UPIPE_ERR_CUDA, "attention launch failed");
      }
    }
  }
  return UPIPE_OK;
}
