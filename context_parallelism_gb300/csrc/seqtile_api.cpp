// C ABI of the sequence-tiled per-token computations - the readout + cross-entropy loss and the
// gated (SwiGLU) MLP: validation, workspace plans, host staging and the per-tile launch
// sequences.
//
// Sequence tiling chunks the per-token computations along the sequence so that no buffer has
// the whole sequence along one dimension ("Road to 5 million sequence length" talk notes,
// Arctic sequence-tiling passage; "Road to 5 Million Tokens" summary, section 2 item 5). Per
// tile of seq_tile tokens:
//   loss forward:  logits GEMM with the CE_FWD epilogue (a (max, sum) pair per token and
//                  256-column vocabulary tile, the target's logit), then one merge launch;
//   loss backward: logits GEMM again with the CE_BWD epilogue -> dlogits (bf16, seq_tile x V,
//                  the only large buffer), dh_tile = dlogits w, dw += dlogits^T h_tile;
//   MLP forward:   gate/up GEMM with the SWIGLU epilogue -> a (bf16, seq_tile x F), y = a Wd^T;
//   MLP backward:  the gate/up GEMM again (a, and g | u), da = dy Wd with the DSWIGLU epilogue
//                  -> dg | du, dWd += dy^T a, dWgu += (dg | du)^T x, dx = (dg | du) [Wg; Wu].
//
// Token-indexed activations (h, dh; x, y, dy, dx) may be pinned host memory instead: the
// inputs of tile i + 2 are then copied into one of two device slots on an inbound copy stream
// while tile i computes, and each tile's outputs are copied out on an outbound copy stream
// while the next tile computes (the block-input offload the talk lists before sequence
// tiling: activations live on the host and are brought in when needed).
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "upipe.h"
#include "internal.h"

namespace upipe {
namespace {

int lfail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  set_last_error(buf);
  return status;
}

#define LOSS_CUDA(call)                                                          \
  do {                                                                           \
    cudaError_t e_ = (call);                                                     \
    if (e_ != cudaSuccess)                                                       \
      return lfail(UPIPE_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_));     \
  } while (0)

// M tiles (128 tokens each) walked together by the GEMMs whose B operand is a weight matrix
// streamed past the token rows: the token rows of one group (group x 128 x Dm x 2 bytes:
// 32 MiB at Dm 4096) stay in L2 while the weights stream past them once per group.
#ifndef UPIPE_CE_GROUP_M
#define UPIPE_CE_GROUP_M 32
#endif
// N tiles (256 output columns each) walked together by the weight-gradient GEMMs (dw of the
// loss, dWgu of the MLP), whose B operand is the token tile: 8 column strips of it (8 x 256 x
// T x 2 bytes: 32 MiB at T = 8192) stay in L2 while the A strips stream past them.
#ifndef UPIPE_WG_GROUP_N
#define UPIPE_WG_GROUP_N 8
#endif
// N tiles walked together by the output GEMMs with a long reduction (dh = dlogits w, y = a Wd^T,
// dx = (dg | du) [Wg; Wu]): each wave of CTAs streams its A strips (128 token rows each) and
// its B strips (256 output columns each) along the whole reduction, so a wave of 19 x 8 tiles
// moves fewer bytes than one of 9.5 x 16 when a B strip is twice an A strip.
#ifndef UPIPE_ST_GROUP_N
#define UPIPE_ST_GROUP_N 8
#endif

constexpr size_t kAl = 256;
inline size_t al(size_t x) { return (x + kAl - 1) / kAl * kAl; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// 0 = device memory (*dev set), 1 = pinned host memory, -1 = anything else.
int placement(const void* p, int* dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (at.type == cudaMemoryTypeDevice) {
    *dev = at.device;
    return 0;
  }
  return at.type == cudaMemoryTypeHost ? 1 : -1;
}

// Every pointer non-null and 16-byte aligned; those with may_host[i] may be pinned host memory
// (host[i] set), every other one device memory of one device (*dev).
int check_ptrs(const void* const* ptrs, const char* const* names, const bool* may_host, int n,
               bool* host, int* dev) {
  int d0 = -1;
  for (int i = 0; i < n; ++i) {
    if (!ptrs[i]) return lfail(UPIPE_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return lfail(UPIPE_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    int d = -1;
    const int kind = placement(ptrs[i], &d);
    host[i] = kind == 1;
    if (kind < 0 || (kind == 1 && !may_host[i]))
      return lfail(UPIPE_ERR_INVALID_ARG, may_host[i] ? "%s must be device or pinned host memory"
                                                      : "%s must be device memory",
                   names[i]);
    if (kind == 1) continue;
    if (d0 < 0) d0 = d;
    if (d != d0) return lfail(UPIPE_ERR_INVALID_ARG, "%s is on device %d, not %d", names[i], d, d0);
  }
  if (d0 < 0) return lfail(UPIPE_ERR_INVALID_ARG, "no device buffer among the arguments");
  *dev = d0;
  return UPIPE_OK;
}

int sm_count(int dev) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  return n;
}

// ---- host staging of token-indexed activations ------------------------------------------------
// Per device: an inbound and an outbound copy stream and the events that order the two slots.
struct Staging {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t in_ready[2], in_free[2], out_done[2], out_free[2], entry, in_join, out_join;
};
constexpr int kMaxDev = 64;
std::mutex g_stage_mu;
Staging g_stage[kMaxDev];

int staging(int dev, Staging** out) {
  if (dev < 0 || dev >= kMaxDev) return lfail(UPIPE_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lk(g_stage_mu);
  Staging& s = g_stage[dev];
  if (!s.ready) {
    LOSS_CUDA(cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking));
    LOSS_CUDA(cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
      LOSS_CUDA(cudaEventCreateWithFlags(&s.in_ready[i], cudaEventDisableTiming));
      LOSS_CUDA(cudaEventCreateWithFlags(&s.in_free[i], cudaEventDisableTiming));
      LOSS_CUDA(cudaEventCreateWithFlags(&s.out_done[i], cudaEventDisableTiming));
      LOSS_CUDA(cudaEventCreateWithFlags(&s.out_free[i], cudaEventDisableTiming));
    }
    LOSS_CUDA(cudaEventCreateWithFlags(&s.entry, cudaEventDisableTiming));
    LOSS_CUDA(cudaEventCreateWithFlags(&s.in_join, cudaEventDisableTiming));
    LOSS_CUDA(cudaEventCreateWithFlags(&s.out_join, cudaEventDisableTiming));
    s.ready = true;
  }
  *out = &s;
  return UPIPE_OK;
}

// One token-indexed activation of a tiled call: its caller buffer, bytes per token row, and,
// when it is pinned host memory, the two device slots it is staged through.
struct Act {
  const void* base = nullptr;
  int64_t row_bytes = 0;
  bool host = false;
  uint8_t* slot[2] = {nullptr, nullptr};
  // device address of row r0 of this activation for tile slot s
  uint8_t* rows(int s, int64_t r0) const {
    return host ? slot[s]
                : const_cast<uint8_t*>(static_cast<const uint8_t*>(base)) + r0 * row_bytes;
  }
};

// Runs body(r0, Mc, slot) for every tile, staging host inputs in and host outputs out around
// it. body launches the tile's kernels on `stream` and returns a status.
template <typename Body>
int run_tiles(int64_t S, int64_t T, const Act* ins, int n_in, const Act* outs, int n_out,
              int dev, cudaStream_t stream, Body body) {
  bool any_in = false, any_out = false;
  for (int k = 0; k < n_in; ++k) any_in |= ins[k].host;
  for (int k = 0; k < n_out; ++k) any_out |= outs[k].host;
  const int64_t n_tiles = (S + T - 1) / T;
  Staging* sg = nullptr;
  if (any_in || any_out) {
    const int st = staging(dev, &sg);
    if (st != UPIPE_OK) return st;
    // the slots live in the workspace: earlier work on the caller's stream may still use it
    LOSS_CUDA(cudaEventRecord(sg->entry, stream));
    LOSS_CUDA(cudaStreamWaitEvent(sg->in, sg->entry, 0));
    LOSS_CUDA(cudaStreamWaitEvent(sg->out, sg->entry, 0));
  }
  auto issue_in = [&](int64_t i) -> int {
    const int s = static_cast<int>(i & 1);
    const int64_t r0 = i * T, Mc = (S - r0) < T ? (S - r0) : T;
    if (i >= 2) LOSS_CUDA(cudaStreamWaitEvent(sg->in, sg->in_free[s], 0));
    for (int k = 0; k < n_in; ++k)
      if (ins[k].host) {
        if (staging_copy_fails()) return lfail(UPIPE_ERR_CUDA, "injected staging copy failure");
        LOSS_CUDA(cudaMemcpyAsync(ins[k].slot[s],
                                  static_cast<const uint8_t*>(ins[k].base) + r0 * ins[k].row_bytes,
                                  Mc * ins[k].row_bytes, cudaMemcpyHostToDevice, sg->in));
      }
    LOSS_CUDA(cudaEventRecord(sg->in_ready[s], sg->in));
    return UPIPE_OK;
  };
  int st = UPIPE_OK;
  if (any_in)
    for (int64_t i = 0; i < 2 && i < n_tiles; ++i)
      if ((st = issue_in(i)) != UPIPE_OK) return st;
  for (int64_t i = 0; i < n_tiles; ++i) {
    const int s = static_cast<int>(i & 1);
    const int64_t r0 = i * T, Mc = (S - r0) < T ? (S - r0) : T;
    if (any_in) LOSS_CUDA(cudaStreamWaitEvent(stream, sg->in_ready[s], 0));
    // the slot's outputs from tile i - 2 must have left before this tile overwrites them
    if (any_out && i >= 2) LOSS_CUDA(cudaStreamWaitEvent(stream, sg->out_free[s], 0));
    {
      const NvtxRange range("upipe tile %lld", static_cast<long long>(i));
      if ((st = body(r0, Mc, s)) != UPIPE_OK) return st;
    }
    if (any_in) {
      LOSS_CUDA(cudaEventRecord(sg->in_free[s], stream));
      if (i + 2 < n_tiles && (st = issue_in(i + 2)) != UPIPE_OK) return st;
    }
    if (any_out) {
      LOSS_CUDA(cudaEventRecord(sg->out_done[s], stream));
      LOSS_CUDA(cudaStreamWaitEvent(sg->out, sg->out_done[s], 0));
      for (int k = 0; k < n_out; ++k)
        if (outs[k].host) {
          if (staging_copy_fails()) return lfail(UPIPE_ERR_CUDA, "injected staging copy failure");
          LOSS_CUDA(cudaMemcpyAsync(const_cast<uint8_t*>(static_cast<const uint8_t*>(outs[k].base)) +
                                        r0 * outs[k].row_bytes,
                                    outs[k].slot[s], Mc * outs[k].row_bytes,
                                    cudaMemcpyDeviceToHost, sg->out));
        }
      LOSS_CUDA(cudaEventRecord(sg->out_free[s], sg->out));
    }
  }
  // the caller's stream completes after the last copies
  if (any_in) {
    LOSS_CUDA(cudaEventRecord(sg->in_join, sg->in));
    LOSS_CUDA(cudaStreamWaitEvent(stream, sg->in_join, 0));
  }
  if (any_out) {
    LOSS_CUDA(cudaEventRecord(sg->out_join, sg->out));
    LOSS_CUDA(cudaStreamWaitEvent(stream, sg->out_join, 0));
  }
  return UPIPE_OK;
}

// Two staging slots of T token rows each, appended to a workspace plan at *off.
void plan_slots(size_t* off, int64_t T, int64_t row_bytes, size_t slot[2]) {
  for (int s = 0; s < 2; ++s) {
    slot[s] = *off;
    *off += al(static_cast<size_t>(T) * row_bytes);
  }
}

Act make_act(const void* base, int64_t row_bytes, bool host, uint8_t* ws, const size_t slot[2]) {
  Act a;
  a.base = base;
  a.row_bytes = row_bytes;
  a.host = host;
  if (host) {
    a.slot[0] = ws + slot[0];
    a.slot[1] = ws + slot[1];
  }
  return a;
}

// ---- loss plan ----------------------------------------------------------------------------
struct CePlan {
  int64_t T = 0;      // tokens per tile (min(seq_tile, S))
  int64_t T_pad = 0;  // T rounded up to 128 rows (partials row pitch)
  int n_vt = 0;       // 256-column vocabulary tiles
  size_t f_part = 0, f_tl = 0, f_h[2] = {0, 0}, f_total = 0;
  size_t b_dl = 0, b_h[2] = {0, 0}, b_dh[2] = {0, 0}, b_total = 0;
  // fused forward + backward: partials, target logits, fp32 logits, bf16 dlogits
  size_t x_part = 0, x_tl = 0, x_L = 0, x_dl = 0, x_h[2] = {0, 0}, x_dh[2] = {0, 0}, x_total = 0;
};

// 0 if the shape is accepted, else a status (message set).
int check_shape(int64_t S, int Dm, int64_t V, int64_t seq_tile) {
  if (S < 1 || Dm < 1 || V < 1 || seq_tile < 1)
    return lfail(UPIPE_ERR_INVALID_ARG, "S, Dm, V, seq_tile must be positive");
  if (Dm % 64 != 0 || V % 64 != 0 || seq_tile % 128 != 0)
    return lfail(UPIPE_ERR_UNSUPPORTED, "need Dm %% 64 == 0, V %% 64 == 0, seq_tile %% 128 == 0");
  if (V >= (int64_t(1) << 31)) return lfail(UPIPE_ERR_UNSUPPORTED, "V must be below 2^31");
  return UPIPE_OK;
}

CePlan make_plan(int64_t S, int Dm, int64_t V, int64_t seq_tile, bool host_act) {
  CePlan p;
  p.T = seq_tile < S ? seq_tile : S;
  p.T_pad = (p.T + 127) / 128 * 128;
  p.n_vt = static_cast<int>((V + 255) / 256);
  const int64_t row = int64_t(Dm) * 2;
  size_t off = 0;
  p.f_part = off;
  off += al(static_cast<size_t>(p.n_vt) * p.T_pad * 8);
  p.f_tl = off;
  off += al(static_cast<size_t>(p.T_pad) * 4);
  if (host_act) plan_slots(&off, p.T, row, p.f_h);
  p.f_total = off;
  off = 0;
  p.b_dl = off;
  off += al(static_cast<size_t>(p.T) * V * 2);
  if (host_act) {
    plan_slots(&off, p.T, row, p.b_h);
    plan_slots(&off, p.T, row, p.b_dh);
  }
  p.b_total = off;
  off = 0;
  p.x_part = off;
  off += al(static_cast<size_t>(p.n_vt) * p.T_pad * 8);
  p.x_tl = off;
  off += al(static_cast<size_t>(p.T_pad) * 4);
  p.x_L = off;
  off += al(static_cast<size_t>(p.T) * V * 4);
  p.x_dl = off;
  off += al(static_cast<size_t>(p.T) * V * 2);
  if (host_act) {
    plan_slots(&off, p.T, row, p.x_h);
    plan_slots(&off, p.T, row, p.x_dh);
  }
  p.x_total = off;
  return p;
}

// ---- MLP plan -----------------------------------------------------------------------------
struct MlpPlan {
  int64_t T = 0;
  size_t a = 0, gu = 0, dgu = 0;
  size_t f_x[2] = {0, 0}, f_y[2] = {0, 0}, f_total = 0;
  size_t b_x[2] = {0, 0}, b_dy[2] = {0, 0}, b_dx[2] = {0, 0}, b_total = 0;
};

int check_mlp_shape(int64_t S, int Dm, int F, int64_t seq_tile) {
  if (S < 1 || Dm < 1 || F < 1 || seq_tile < 1)
    return lfail(UPIPE_ERR_INVALID_ARG, "S, Dm, F, seq_tile must be positive");
  if (Dm % 64 != 0 || F % 128 != 0 || seq_tile % 128 != 0)
    return lfail(UPIPE_ERR_UNSUPPORTED, "need Dm %% 64 == 0, F %% 128 == 0, seq_tile %% 128 == 0");
  if (2 * static_cast<int64_t>(F) >= (int64_t(1) << 31))
    return lfail(UPIPE_ERR_UNSUPPORTED, "2F must be below 2^31");
  return UPIPE_OK;
}

MlpPlan make_mlp_plan(int64_t S, int Dm, int F, int64_t seq_tile, bool host_act) {
  MlpPlan p;
  p.T = seq_tile < S ? seq_tile : S;
  const size_t tf = static_cast<size_t>(p.T) * F * 2;  // one [T][F] bf16 buffer
  const int64_t row = int64_t(Dm) * 2;
  size_t off = 0;
  p.a = off;
  off += al(tf);
  const size_t after_a = off;
  if (host_act) {
    plan_slots(&off, p.T, row, p.f_x);
    plan_slots(&off, p.T, row, p.f_y);
  }
  p.f_total = off;
  off = after_a;
  p.gu = off;
  off += al(2 * tf);
  p.dgu = off;
  off += al(2 * tf);
  if (host_act) {
    plan_slots(&off, p.T, row, p.b_x);
    plan_slots(&off, p.T, row, p.b_dy);
    plan_slots(&off, p.T, row, p.b_dx);
  }
  p.b_total = off;
  return p;
}

}  // namespace

void seqtile_shutdown() {
  std::lock_guard<std::mutex> lk(g_stage_mu);
  for (int d = 0; d < kMaxDev; ++d) {
    Staging& s = g_stage[d];
    if (!s.ready) continue;
    cudaSetDevice(d);
    cudaStreamSynchronize(s.in);
    cudaStreamSynchronize(s.out);
    cudaStreamDestroy(s.in);
    cudaStreamDestroy(s.out);
    for (int i = 0; i < 2; ++i) {
      cudaEventDestroy(s.in_ready[i]);
      cudaEventDestroy(s.in_free[i]);
      cudaEventDestroy(s.out_done[i]);
      cudaEventDestroy(s.out_free[i]);
    }
    cudaEventDestroy(s.entry);
    cudaEventDestroy(s.in_join);
    cudaEventDestroy(s.out_join);
    s = Staging{};
  }
}

}  // namespace upipe

using namespace upipe;

extern "C" {

// ---- sequence-tiled readout + cross-entropy loss -----------------------------------------------

size_t upipe_ce_workspace_bytes(int64_t S, int Dm, int64_t V, int64_t seq_tile, int pass,
                                int host_mask) {
  if (check_shape(S, Dm, V, seq_tile) != UPIPE_OK) return 0;
  if (pass < UPIPE_PASS_FWD || pass > UPIPE_PASS_FUSED) return 0;
  if (host_mask & ~UPIPE_HOST_ACT) return 0;
  const CePlan p = make_plan(S, Dm, V, seq_tile, (host_mask & UPIPE_HOST_ACT) != 0);
  if (pass == UPIPE_PASS_FWD) return p.f_total;
  if (pass == UPIPE_PASS_BWD) return p.b_total;
  if (pass == UPIPE_PASS_FUSED) return p.x_total;
  return p.f_total > p.b_total ? p.f_total : p.b_total;
}

int upipe_ce_fwd(const void* h, const void* w, const int64_t* target, float* loss, float* lse,
                 int64_t S, int Dm, int64_t V, int64_t seq_tile, void* workspace,
                 size_t workspace_bytes, void* stream_) {
  const NvtxRange range("upipe_ce_fwd");
  set_last_error("");
  int st = check_shape(S, Dm, V, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[6] = {h, w, target, loss, lse, workspace};
  const char* names[6] = {"h", "w", "target", "loss", "lse", "workspace"};
  const bool may_host[6] = {true, false, false, false, false, false};
  bool host[6];
  int dev = -1;
  st = check_ptrs(ptrs, names, may_host, 6, host, &dev);
  if (st != UPIPE_OK) return st;
  const CePlan p = make_plan(S, Dm, V, seq_tile, host[0]);
  if (workspace_bytes < p.f_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.f_total);
  const DeviceGuard dguard;
  LOSS_CUDA(cudaSetDevice(dev));
  uint32_t* err = nullptr;
  st = device_status_word(dev, &err);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* part = reinterpret_cast<float*>(ws + p.f_part);
  float* tl = reinterpret_cast<float*>(ws + p.f_tl);
  const int cap = sm_count(dev);

  const Act in[1] = {make_act(h, int64_t(Dm) * 2, host[0], ws, p.f_h)};
  CUtensorMap tw;
  LOSS_CUDA(make_tmap_bf16(&tw, w, Dm, V, 1, 256));
  return run_tiles(S, p.T, in, 1, nullptr, 0, dev, stream,
                   [&](int64_t r0, int64_t Mc, int s) -> int {
    CUtensorMap th;
    LOSS_CUDA(make_tmap_bf16(&th, in[0].rows(s, r0), Dm, Mc, 1, 128));
    GemmArgs a{};
    a.M = static_cast<int>(Mc);
    a.N = static_cast<int>(V);
    a.K = Dm;
    a.m_fastest = 1;
    a.group_m = UPIPE_CE_GROUP_M;
    a.target = target + r0;
    a.part = part;
    a.part_stride = p.T_pad;
    a.tlogit = tl;
    a.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiCeFwd, false, false, th, tw, a, cap, stream));
    LOSS_CUDA(launch_ce_merge(part, p.T_pad, p.n_vt, tl, target + r0, loss + r0, lse + r0, Mc,
                              V, stream));
    return UPIPE_OK;
  });
}

int upipe_ce_bwd(const void* h, const void* w, const int64_t* target, const float* lse,
                 const float* dloss, void* dh, float* dw, int64_t S, int Dm, int64_t V,
                 int64_t seq_tile, void* workspace, size_t workspace_bytes, void* stream_) {
  const NvtxRange range("upipe_ce_bwd");
  set_last_error("");
  int st = check_shape(S, Dm, V, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[8] = {h, w, target, lse, dloss, dh, dw, workspace};
  const char* names[8] = {"h", "w", "target", "lse", "dloss", "dh", "dw", "workspace"};
  const bool may_host[8] = {true, false, false, false, false, true, false, false};
  bool host[8];
  int dev = -1;
  st = check_ptrs(ptrs, names, may_host, 8, host, &dev);
  if (st != UPIPE_OK) return st;
  const CePlan p = make_plan(S, Dm, V, seq_tile, host[0] || host[5]);
  if (workspace_bytes < p.b_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.b_total);
  const DeviceGuard dguard;
  LOSS_CUDA(cudaSetDevice(dev));
  uint32_t* err = nullptr;
  st = device_status_word(dev, &err);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* dl = ws + p.b_dl;
  const int cap = sm_count(dev);

  const Act in[1] = {make_act(h, int64_t(Dm) * 2, host[0], ws, p.b_h)};
  const Act out[1] = {make_act(dh, int64_t(Dm) * 2, host[5], ws, p.b_dh)};
  CUtensorMap tw_k, tw_mn;
  LOSS_CUDA(make_tmap_bf16(&tw_k, w, Dm, V, 1, 256));   // w as B [N = V][K = Dm]
  LOSS_CUDA(make_tmap_bf16(&tw_mn, w, Dm, V, 1, 64));   // w as B [K = V][N = Dm]
  return run_tiles(S, p.T, in, 1, out, 1, dev, stream,
                   [&](int64_t r0, int64_t Mc, int s) -> int {
    const uint8_t* hc = in[0].rows(s, r0);
    CUtensorMap th_k, th_mn, tdl_k, tdl_mn;
    LOSS_CUDA(make_tmap_bf16(&th_k, hc, Dm, Mc, 1, 128));  // h tile as A [M = Mc][K = Dm]
    LOSS_CUDA(make_tmap_bf16(&th_mn, hc, Dm, Mc, 1, 64));  // h tile as B [K = Mc][N = Dm]
    LOSS_CUDA(make_tmap_bf16(&tdl_k, dl, V, Mc, 1, 128));  // dlogits as A [M = Mc][K = V]
    LOSS_CUDA(make_tmap_bf16(&tdl_mn, dl, V, Mc, 1, 64));  // dlogits as A [K = Mc][M = V]

    GemmArgs g{};
    g.M = static_cast<int>(Mc);
    g.N = static_cast<int>(V);
    g.K = Dm;
    g.m_fastest = 1;
    g.group_m = UPIPE_CE_GROUP_M;
    g.c = dl;
    g.ldc = V;
    g.target = target + r0;
    g.lse = lse + r0;
    g.g = dloss + r0;
    g.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiCeBwd, false, false, th_k, tw_k, g, cap, stream));

    GemmArgs x{};
    x.M = static_cast<int>(Mc);
    x.N = Dm;
    x.K = static_cast<int>(V);
    x.m_fastest = 0;
    x.group_m = UPIPE_ST_GROUP_N;
    x.c = out[0].rows(s, r0);
    x.ldc = Dm;
    x.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiStoreBf16, false, true, tdl_k, tw_mn, x, cap, stream));

    GemmArgs y{};
    y.M = static_cast<int>(V);
    y.N = Dm;
    y.K = static_cast<int>(Mc);
    y.m_fastest = 0;
    y.group_m = UPIPE_WG_GROUP_N;
    y.c = dw;
    y.ldc = Dm;
    y.accumulate = r0 > 0 ? 1 : 0;
    y.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiAccF32, true, true, tdl_mn, th_mn, y, cap, stream));
    return UPIPE_OK;
  });
}

int upipe_ce_fwd_bwd(const void* h, const void* w, const int64_t* target, const float* dloss,
                     float* loss, float* lse, void* dh, float* dw, int64_t S, int Dm, int64_t V,
                     int64_t seq_tile, void* workspace, size_t workspace_bytes, void* stream_) {
  const NvtxRange range("upipe_ce_fwd_bwd");
  set_last_error("");
  int st = check_shape(S, Dm, V, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[9] = {h, w, target, dloss, loss, lse, dh, dw, workspace};
  const char* names[9] = {"h", "w", "target", "dloss", "loss", "lse", "dh", "dw", "workspace"};
  const bool may_host[9] = {true, false, false, false, false, false, true, false, false};
  bool host[9];
  int dev = -1;
  st = check_ptrs(ptrs, names, may_host, 9, host, &dev);
  if (st != UPIPE_OK) return st;
  const CePlan p = make_plan(S, Dm, V, seq_tile, host[0] || host[6]);
  if (workspace_bytes < p.x_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.x_total);
  const DeviceGuard dguard;
  LOSS_CUDA(cudaSetDevice(dev));
  uint32_t* err = nullptr;
  st = device_status_word(dev, &err);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* part = reinterpret_cast<float*>(ws + p.x_part);
  float* tl = reinterpret_cast<float*>(ws + p.x_tl);
  float* logits = reinterpret_cast<float*>(ws + p.x_L);
  void* dl = ws + p.x_dl;
  const int cap = sm_count(dev);

  const Act in[1] = {make_act(h, int64_t(Dm) * 2, host[0], ws, p.x_h)};
  const Act out[1] = {make_act(dh, int64_t(Dm) * 2, host[6], ws, p.x_dh)};
  CUtensorMap tw_k, tw_mn;
  LOSS_CUDA(make_tmap_bf16(&tw_k, w, Dm, V, 1, 256));   // w as B [N = V][K = Dm]
  LOSS_CUDA(make_tmap_bf16(&tw_mn, w, Dm, V, 1, 64));   // w as B [K = V][N = Dm]
  return run_tiles(S, p.T, in, 1, out, 1, dev, stream,
                   [&](int64_t r0, int64_t Mc, int s) -> int {
    const uint8_t* hc = in[0].rows(s, r0);
    CUtensorMap th_k, th_mn, tdl_k, tdl_mn;
    LOSS_CUDA(make_tmap_bf16(&th_k, hc, Dm, Mc, 1, 128));
    LOSS_CUDA(make_tmap_bf16(&th_mn, hc, Dm, Mc, 1, 64));
    LOSS_CUDA(make_tmap_bf16(&tdl_k, dl, V, Mc, 1, 128));
    LOSS_CUDA(make_tmap_bf16(&tdl_mn, dl, V, Mc, 1, 64));

    GemmArgs a{};  // logits: loss statistics, and the fp32 logits kept for the backward
    a.M = static_cast<int>(Mc);
    a.N = static_cast<int>(V);
    a.K = Dm;
    a.m_fastest = 1;
    a.group_m = UPIPE_CE_GROUP_M;
    a.c = logits;
    a.ldc = V;
    a.target = target + r0;
    a.part = part;
    a.part_stride = p.T_pad;
    a.tlogit = tl;
    a.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiCeFwd, false, false, th_k, tw_k, a, cap, stream));
    LOSS_CUDA(launch_ce_merge(part, p.T_pad, p.n_vt, tl, target + r0, loss + r0, lse + r0, Mc,
                              V, stream));
    LOSS_CUDA(launch_ce_dlogits(logits, lse + r0, target + r0, dloss + r0, dl, Mc, V, stream));

    GemmArgs x{};  // dh = dlogits w
    x.M = static_cast<int>(Mc);
    x.N = Dm;
    x.K = static_cast<int>(V);
    x.m_fastest = 0;
    x.group_m = UPIPE_ST_GROUP_N;
    x.c = out[0].rows(s, r0);
    x.ldc = Dm;
    x.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiStoreBf16, false, true, tdl_k, tw_mn, x, cap, stream));

    GemmArgs y{};  // dw += dlogits^T h
    y.M = static_cast<int>(V);
    y.N = Dm;
    y.K = static_cast<int>(Mc);
    y.m_fastest = 0;
    y.group_m = UPIPE_WG_GROUP_N;
    y.c = dw;
    y.ldc = Dm;
    y.accumulate = r0 > 0 ? 1 : 0;
    y.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiAccF32, true, true, tdl_mn, th_mn, y, cap, stream));
    return UPIPE_OK;
  });
}

// ---- sequence-tiled gated MLP -------------------------------------------------------------

size_t upipe_mlp_workspace_bytes(int64_t S, int Dm, int F, int64_t seq_tile, int pass,
                                 int host_mask) {
  if (check_mlp_shape(S, Dm, F, seq_tile) != UPIPE_OK) return 0;
  if (pass < UPIPE_PASS_FWD || pass > UPIPE_PASS_BOTH) return 0;
  if (host_mask & ~UPIPE_HOST_ACT) return 0;
  const MlpPlan p = make_mlp_plan(S, Dm, F, seq_tile, (host_mask & UPIPE_HOST_ACT) != 0);
  if (pass == UPIPE_PASS_FWD) return p.f_total;
  if (pass == UPIPE_PASS_BWD) return p.b_total;
  return p.f_total > p.b_total ? p.f_total : p.b_total;
}

int upipe_mlp_fwd(const void* x, const void* w_gu, const void* w_d, void* y, int64_t S, int Dm,
                  int F, int64_t seq_tile, void* workspace, size_t workspace_bytes,
                  void* stream_) {
  const NvtxRange range("upipe_mlp_fwd");
  set_last_error("");
  int st = check_mlp_shape(S, Dm, F, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[5] = {x, w_gu, w_d, y, workspace};
  const char* names[5] = {"x", "w_gu", "w_d", "y", "workspace"};
  const bool may_host[5] = {true, false, false, true, false};
  bool host[5];
  int dev = -1;
  st = check_ptrs(ptrs, names, may_host, 5, host, &dev);
  if (st != UPIPE_OK) return st;
  const MlpPlan p = make_mlp_plan(S, Dm, F, seq_tile, host[0] || host[3]);
  if (workspace_bytes < p.f_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.f_total);
  const DeviceGuard dguard;
  LOSS_CUDA(cudaSetDevice(dev));
  uint32_t* err = nullptr;
  st = device_status_word(dev, &err);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* a_ws = ws + p.a;
  const int cap = sm_count(dev);

  const Act in[1] = {make_act(x, int64_t(Dm) * 2, host[0], ws, p.f_x)};
  const Act out[1] = {make_act(y, int64_t(Dm) * 2, host[3], ws, p.f_y)};
  CUtensorMap t_wgu, t_wd;
  LOSS_CUDA(make_tmap_bf16(&t_wgu, w_gu, Dm, 2 * static_cast<int64_t>(F), 1, 128));
  LOSS_CUDA(make_tmap_bf16(&t_wd, w_d, F, Dm, 1, 256));  // Wd as B [N = Dm][K = F]
  return run_tiles(S, p.T, in, 1, out, 1, dev, stream,
                   [&](int64_t r0, int64_t Mc, int s) -> int {
    CUtensorMap t_x, t_a;
    LOSS_CUDA(make_tmap_bf16(&t_x, in[0].rows(s, r0), Dm, Mc, 1, 128));
    LOSS_CUDA(make_tmap_bf16(&t_a, a_ws, F, Mc, 1, 128));
    GemmArgs g{};
    g.M = static_cast<int>(Mc);
    g.N = F;
    g.K = Dm;
    g.m_fastest = 1;
    g.group_m = UPIPE_CE_GROUP_M;
    g.c = a_ws;
    g.ldc = F;
    g.split = F;
    g.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiSwiglu, false, false, t_x, t_wgu, g, cap, stream));
    GemmArgs o{};
    o.M = static_cast<int>(Mc);
    o.N = Dm;
    o.K = F;
    o.m_fastest = 0;
    o.group_m = UPIPE_ST_GROUP_N;
    o.c = out[0].rows(s, r0);
    o.ldc = Dm;
    o.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiStoreBf16, false, false, t_a, t_wd, o, cap, stream));
    return UPIPE_OK;
  });
}

int upipe_mlp_bwd(const void* x, const void* w_gu, const void* w_d, const void* dy, void* dx,
                  float* dw_gu, float* dw_d, int64_t S, int Dm, int F, int64_t seq_tile,
                  void* workspace, size_t workspace_bytes, void* stream_) {
  const NvtxRange range("upipe_mlp_bwd");
  set_last_error("");
  int st = check_mlp_shape(S, Dm, F, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[8] = {x, w_gu, w_d, dy, dx, dw_gu, dw_d, workspace};
  const char* names[8] = {"x", "w_gu", "w_d", "dy", "dx", "dw_gu", "dw_d", "workspace"};
  const bool may_host[8] = {true, false, false, true, true, false, false, false};
  bool host[8];
  int dev = -1;
  st = check_ptrs(ptrs, names, may_host, 8, host, &dev);
  if (st != UPIPE_OK) return st;
  const MlpPlan p = make_mlp_plan(S, Dm, F, seq_tile, host[0] || host[3] || host[4]);
  if (workspace_bytes < p.b_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.b_total);
  const DeviceGuard dguard;
  LOSS_CUDA(cudaSetDevice(dev));
  uint32_t* err = nullptr;
  st = device_status_word(dev, &err);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* a_ws = ws + p.a;
  void* gu_ws = ws + p.gu;
  void* dgu_ws = ws + p.dgu;
  const int64_t F2 = 2 * static_cast<int64_t>(F);
  const int cap = sm_count(dev);

  const Act in[2] = {make_act(x, int64_t(Dm) * 2, host[0], ws, p.b_x),
                     make_act(dy, int64_t(Dm) * 2, host[3], ws, p.b_dy)};
  const Act out[1] = {make_act(dx, int64_t(Dm) * 2, host[4], ws, p.b_dx)};
  CUtensorMap t_wgu_k, t_wgu_mn, t_wd_mn;
  LOSS_CUDA(make_tmap_bf16(&t_wgu_k, w_gu, Dm, F2, 1, 128));  // [Wg; Wu] as B [N][K = Dm]
  LOSS_CUDA(make_tmap_bf16(&t_wgu_mn, w_gu, Dm, F2, 1, 64));  // as B [K = 2F][N = Dm]
  LOSS_CUDA(make_tmap_bf16(&t_wd_mn, w_d, F, Dm, 1, 64));     // Wd as B [K = Dm][N = F]
  return run_tiles(S, p.T, in, 2, out, 1, dev, stream,
                   [&](int64_t r0, int64_t Mc, int s) -> int {
    const uint8_t* xt = in[0].rows(s, r0);
    const uint8_t* dyt = in[1].rows(s, r0);
    CUtensorMap t_x_k, t_x_mn, t_dy_k, t_dy_mn, t_a_mn, t_dgu_k, t_dgu_mn;
    LOSS_CUDA(make_tmap_bf16(&t_x_k, xt, Dm, Mc, 1, 128));
    LOSS_CUDA(make_tmap_bf16(&t_x_mn, xt, Dm, Mc, 1, 64));
    LOSS_CUDA(make_tmap_bf16(&t_dy_k, dyt, Dm, Mc, 1, 128));
    LOSS_CUDA(make_tmap_bf16(&t_dy_mn, dyt, Dm, Mc, 1, 64));
    LOSS_CUDA(make_tmap_bf16(&t_a_mn, a_ws, F, Mc, 1, 64));
    LOSS_CUDA(make_tmap_bf16(&t_dgu_k, dgu_ws, F2, Mc, 1, 128));
    LOSS_CUDA(make_tmap_bf16(&t_dgu_mn, dgu_ws, F2, Mc, 1, 64));

    GemmArgs r{};  // recompute: a, and g | u
    r.M = static_cast<int>(Mc);
    r.N = F;
    r.K = Dm;
    r.m_fastest = 1;
    r.group_m = UPIPE_CE_GROUP_M;
    r.c = a_ws;
    r.ldc = F;
    r.c2 = gu_ws;
    r.ldc2 = F2;
    r.split = F;
    r.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiSwiglu, false, false, t_x_k, t_wgu_k, r, cap, stream));

    GemmArgs d{};  // da = dy Wd -> dg | du
    d.M = static_cast<int>(Mc);
    d.N = F;
    d.K = Dm;
    d.m_fastest = 1;
    d.group_m = UPIPE_CE_GROUP_M;
    d.c = dgu_ws;
    d.ldc = F2;
    d.aux = gu_ws;
    d.ld_aux = F2;
    d.split = F;
    d.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiDSwiglu, false, true, t_dy_k, t_wd_mn, d, cap, stream));

    GemmArgs wd{};  // dWd += dy^T a
    wd.M = Dm;
    wd.N = F;
    wd.K = static_cast<int>(Mc);
    // M tiles first, 16 at a time: the CTAs in flight share 16 dy strips (32 MiB at 8192
    // tokens) and stream each strip of a about twice per tile, instead of all of a per wave
    wd.m_fastest = 1;
    wd.group_m = 16;
    wd.c = dw_d;
    wd.ldc = F;
    wd.accumulate = r0 > 0 ? 1 : 0;
    wd.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiAccF32, true, true, t_dy_mn, t_a_mn, wd, cap, stream));

    GemmArgs wg{};  // dWgu += (dg | du)^T x
    wg.M = static_cast<int>(F2);
    wg.N = Dm;
    wg.K = static_cast<int>(Mc);
    wg.m_fastest = 0;
    wg.group_m = UPIPE_WG_GROUP_N;
    wg.c = dw_gu;
    wg.ldc = Dm;
    wg.accumulate = r0 > 0 ? 1 : 0;
    wg.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiAccF32, true, true, t_dgu_mn, t_x_mn, wg, cap, stream));

    GemmArgs gx{};  // dx = (dg | du) [Wg; Wu]
    gx.M = static_cast<int>(Mc);
    gx.N = Dm;
    gx.K = static_cast<int>(F2);
    gx.m_fastest = 0;
    gx.group_m = UPIPE_ST_GROUP_N;
    gx.c = out[0].rows(s, r0);
    gx.ldc = Dm;
    gx.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiStoreBf16, false, true, t_dgu_k, t_wgu_mn, gx, cap, stream));
    return UPIPE_OK;
  });
}

}  // extern "C"
