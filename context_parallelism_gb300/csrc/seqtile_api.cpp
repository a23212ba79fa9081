// C ABI of the sequence-tiled per-token computations - the readout + cross-entropy loss and the
// gated (SwiGLU) MLP: validation, workspace plans and the per-tile launch sequences.
//
// Sequence tiling chunks the per-token computations along the sequence so that no buffer has
// the whole sequence along one dimension ("Road to 5 million sequence length" talk notes,
// Arctic sequence-tiling passage; "Road to 5 Million Tokens" summary, section 2 item 5). Per
// tile of seq_tile tokens:
//   forward:  logits GEMM with the CE_FWD epilogue (a (max, sum) pair per token and 256-column
//             vocabulary tile, the target's logit), then one merge launch -> loss, lse;
//   backward: logits GEMM again with the CE_BWD epilogue -> dlogits (bf16, seq_tile x V, the
//             only large buffer), dh_tile = dlogits w (stored), dw += dlogits^T h_tile.
// and for the MLP (y = (silu(x Wg^T) * x Wu^T) Wd^T), per tile:
//   forward:  gate/up GEMM with the SWIGLU epilogue -> a (bf16, seq_tile x F), y = a Wd^T;
//   backward: the gate/up GEMM again (a, and g | u for the gating derivative), da = dy Wd with
//             the DSWIGLU epilogue -> dg | du, dWd += dy^T a, dWgu += (dg | du)^T x,
//             dx = (dg | du) [Wg; Wu].
#include <cstdarg>
#include <cstdio>

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

// M tiles (128 tokens each) walked together by the two vocabulary GEMMs: the token rows of one
// group (group x 128 x Dm x 2 bytes: 32 MiB at Dm 4096) stay in L2 while the vocabulary streams
// past them once per group.
#ifndef UPIPE_CE_GROUP_M
#define UPIPE_CE_GROUP_M 32
#endif

constexpr size_t kAl = 256;
inline size_t al(size_t x) { return (x + kAl - 1) / kAl * kAl; }

struct CePlan {
  int64_t T = 0;      // tokens per tile (min(seq_tile, S))
  int64_t T_pad = 0;  // T rounded up to 128 rows (partials row pitch)
  int n_vt = 0;       // 256-column vocabulary tiles
  size_t f_part = 0, f_tl = 0, f_total = 0;
  size_t b_dl = 0, b_total = 0;
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

CePlan make_plan(int64_t S, int64_t V, int64_t seq_tile) {
  CePlan p;
  p.T = seq_tile < S ? seq_tile : S;
  p.T_pad = (p.T + 127) / 128 * 128;
  p.n_vt = static_cast<int>((V + 255) / 256);
  p.f_part = 0;
  p.f_tl = al(static_cast<size_t>(p.n_vt) * p.T_pad * 8);
  p.f_total = p.f_tl + al(static_cast<size_t>(p.T_pad) * 4);
  p.b_dl = 0;
  p.b_total = al(static_cast<size_t>(p.T) * V * 2);
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// All pointers non-null, 16-byte aligned device memory of one device; *dev gets it.
int check_device_ptrs(const void* const* ptrs, const char* const* names, int n, int* dev) {
  int d0 = -1;
  for (int i = 0; i < n; ++i) {
    if (!ptrs[i]) return lfail(UPIPE_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return lfail(UPIPE_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptrs[i]) != cudaSuccess) {
      cudaGetLastError();
      return lfail(UPIPE_ERR_INVALID_ARG, "%s is not device memory", names[i]);
    }
    if (at.type != cudaMemoryTypeDevice)
      return lfail(UPIPE_ERR_INVALID_ARG, "%s must be device memory", names[i]);
    if (d0 < 0) d0 = at.device;
    if (at.device != d0)
      return lfail(UPIPE_ERR_INVALID_ARG, "%s is on device %d, not %d", names[i], at.device, d0);
  }
  *dev = d0;
  return UPIPE_OK;
}

int sm_count(int dev) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  return n;
}

const uint8_t* bf16_rows(const void* base, int64_t row, int64_t cols) {
  return static_cast<const uint8_t*>(base) + row * cols * 2;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" {

size_t upipe_ce_workspace_bytes(int64_t S, int Dm, int64_t V, int64_t seq_tile, int pass) {
  if (check_shape(S, Dm, V, seq_tile) != UPIPE_OK) return 0;
  if (pass < UPIPE_PASS_FWD || pass > UPIPE_PASS_BOTH) return 0;
  const CePlan p = make_plan(S, V, seq_tile);
  if (pass == UPIPE_PASS_FWD) return p.f_total;
  if (pass == UPIPE_PASS_BWD) return p.b_total;
  return p.f_total > p.b_total ? p.f_total : p.b_total;
}

int upipe_ce_fwd(const void* h, const void* w, const int64_t* target, float* loss, float* lse,
                 int64_t S, int Dm, int64_t V, int64_t seq_tile, void* workspace,
                 size_t workspace_bytes, void* stream_) {
  set_last_error("");
  int st = check_shape(S, Dm, V, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[6] = {h, w, target, loss, lse, workspace};
  const char* names[6] = {"h", "w", "target", "loss", "lse", "workspace"};
  int dev = -1;
  st = check_device_ptrs(ptrs, names, 6, &dev);
  if (st != UPIPE_OK) return st;
  const CePlan p = make_plan(S, V, seq_tile);
  if (workspace_bytes < p.f_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.f_total);
  LOSS_CUDA(cudaSetDevice(dev));
  uint32_t* err = nullptr;
  st = device_status_word(dev, &err);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* part = reinterpret_cast<float*>(ws + p.f_part);
  float* tl = reinterpret_cast<float*>(ws + p.f_tl);
  const int cap = sm_count(dev);

  CUtensorMap tw, th;
  LOSS_CUDA(make_tmap_bf16(&tw, w, Dm, V, 1, 256));
  for (int64_t r0 = 0; r0 < S; r0 += p.T) {
    const int64_t Mc = (S - r0) < p.T ? (S - r0) : p.T;
    LOSS_CUDA(make_tmap_bf16(&th, bf16_rows(h, r0, Dm), Dm, Mc, 1, 128));
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
  }
  return UPIPE_OK;
}

int upipe_ce_bwd(const void* h, const void* w, const int64_t* target, const float* lse,
                 const float* dloss, void* dh, float* dw, int64_t S, int Dm, int64_t V,
                 int64_t seq_tile, void* workspace, size_t workspace_bytes, void* stream_) {
  set_last_error("");
  int st = check_shape(S, Dm, V, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[8] = {h, w, target, lse, dloss, dh, dw, workspace};
  const char* names[8] = {"h", "w", "target", "lse", "dloss", "dh", "dw", "workspace"};
  int dev = -1;
  st = check_device_ptrs(ptrs, names, 8, &dev);
  if (st != UPIPE_OK) return st;
  const CePlan p = make_plan(S, V, seq_tile);
  if (workspace_bytes < p.b_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.b_total);
  LOSS_CUDA(cudaSetDevice(dev));
  uint32_t* err = nullptr;
  st = device_status_word(dev, &err);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  void* dl = static_cast<uint8_t*>(workspace) + p.b_dl;
  const int cap = sm_count(dev);

  CUtensorMap tw_k, tw_mn, th_k, th_mn, tdl_k, tdl_mn;
  LOSS_CUDA(make_tmap_bf16(&tw_k, w, Dm, V, 1, 256));   // w as B [N = V][K = Dm]
  LOSS_CUDA(make_tmap_bf16(&tw_mn, w, Dm, V, 1, 64));   // w as B [K = V][N = Dm]
  for (int64_t r0 = 0; r0 < S; r0 += p.T) {
    const int64_t Mc = (S - r0) < p.T ? (S - r0) : p.T;
    const uint8_t* hc = bf16_rows(h, r0, Dm);
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
    x.c = static_cast<uint8_t*>(dh) + r0 * Dm * 2;
    x.ldc = Dm;
    x.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiStoreBf16, false, true, tdl_k, tw_mn, x, cap, stream));

    GemmArgs y{};
    y.M = static_cast<int>(V);
    y.N = Dm;
    y.K = static_cast<int>(Mc);
    y.m_fastest = 0;
    y.c = dw;
    y.ldc = Dm;
    y.accumulate = r0 > 0 ? 1 : 0;
    y.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiAccF32, true, true, tdl_mn, th_mn, y, cap, stream));
  }
  return UPIPE_OK;
}

}  // extern "C"

// ---- sequence-tiled gated MLP -------------------------------------------------------------

namespace upipe {
namespace {

struct MlpPlan {
  int64_t T = 0;
  size_t a = 0, gu = 0, dgu = 0, f_total = 0, b_total = 0;
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

MlpPlan make_mlp_plan(int64_t S, int F, int64_t seq_tile) {
  MlpPlan p;
  p.T = seq_tile < S ? seq_tile : S;
  const size_t tf = static_cast<size_t>(p.T) * F * 2;  // one [T][F] bf16 buffer
  p.a = 0;
  p.gu = al(tf);
  p.dgu = p.gu + al(2 * tf);
  p.f_total = al(tf);
  p.b_total = p.dgu + al(2 * tf);
  return p;
}

}  // namespace
}  // namespace upipe

extern "C" {

size_t upipe_mlp_workspace_bytes(int64_t S, int Dm, int F, int64_t seq_tile, int pass) {
  if (check_mlp_shape(S, Dm, F, seq_tile) != UPIPE_OK) return 0;
  if (pass < UPIPE_PASS_FWD || pass > UPIPE_PASS_BOTH) return 0;
  const MlpPlan p = make_mlp_plan(S, F, seq_tile);
  if (pass == UPIPE_PASS_FWD) return p.f_total;
  return p.b_total;  // the backward's buffers include the forward's
}

int upipe_mlp_fwd(const void* x, const void* w_gu, const void* w_d, void* y, int64_t S, int Dm,
                  int F, int64_t seq_tile, void* workspace, size_t workspace_bytes,
                  void* stream_) {
  set_last_error("");
  int st = check_mlp_shape(S, Dm, F, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[5] = {x, w_gu, w_d, y, workspace};
  const char* names[5] = {"x", "w_gu", "w_d", "y", "workspace"};
  int dev = -1;
  st = check_device_ptrs(ptrs, names, 5, &dev);
  if (st != UPIPE_OK) return st;
  const MlpPlan p = make_mlp_plan(S, F, seq_tile);
  if (workspace_bytes < p.f_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.f_total);
  LOSS_CUDA(cudaSetDevice(dev));
  uint32_t* err = nullptr;
  st = device_status_word(dev, &err);
  if (st != UPIPE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  void* a_ws = static_cast<uint8_t*>(workspace) + p.a;
  const int cap = sm_count(dev);

  CUtensorMap t_wgu, t_wd, t_x, t_a;
  LOSS_CUDA(make_tmap_bf16(&t_wgu, w_gu, Dm, 2 * static_cast<int64_t>(F), 1, 128));
  LOSS_CUDA(make_tmap_bf16(&t_wd, w_d, F, Dm, 1, 256));  // Wd as B [N = Dm][K = F]
  for (int64_t r0 = 0; r0 < S; r0 += p.T) {
    const int64_t Mc = (S - r0) < p.T ? (S - r0) : p.T;
    LOSS_CUDA(make_tmap_bf16(&t_x, bf16_rows(x, r0, Dm), Dm, Mc, 1, 128));
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
    o.c = static_cast<uint8_t*>(y) + r0 * Dm * 2;
    o.ldc = Dm;
    o.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiStoreBf16, false, false, t_a, t_wd, o, cap, stream));
  }
  return UPIPE_OK;
}

int upipe_mlp_bwd(const void* x, const void* w_gu, const void* w_d, const void* dy, void* dx,
                  float* dw_gu, float* dw_d, int64_t S, int Dm, int F, int64_t seq_tile,
                  void* workspace, size_t workspace_bytes, void* stream_) {
  set_last_error("");
  int st = check_mlp_shape(S, Dm, F, seq_tile);
  if (st != UPIPE_OK) return st;
  const void* ptrs[8] = {x, w_gu, w_d, dy, dx, dw_gu, dw_d, workspace};
  const char* names[8] = {"x", "w_gu", "w_d", "dy", "dx", "dw_gu", "dw_d", "workspace"};
  int dev = -1;
  st = check_device_ptrs(ptrs, names, 8, &dev);
  if (st != UPIPE_OK) return st;
  const MlpPlan p = make_mlp_plan(S, F, seq_tile);
  if (workspace_bytes < p.b_total)
    return lfail(UPIPE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes,
                 p.b_total);
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

  CUtensorMap t_wgu_k, t_wgu_mn, t_wd_mn, t_x_k, t_x_mn, t_dy_k, t_dy_mn, t_a_mn, t_dgu_k,
      t_dgu_mn;
  LOSS_CUDA(make_tmap_bf16(&t_wgu_k, w_gu, Dm, F2, 1, 128));  // [Wg; Wu] as B [N][K = Dm]
  LOSS_CUDA(make_tmap_bf16(&t_wgu_mn, w_gu, Dm, F2, 1, 64));  // as B [K = 2F][N = Dm]
  LOSS_CUDA(make_tmap_bf16(&t_wd_mn, w_d, F, Dm, 1, 64));     // Wd as B [K = Dm][N = F]
  for (int64_t r0 = 0; r0 < S; r0 += p.T) {
    const int64_t Mc = (S - r0) < p.T ? (S - r0) : p.T;
    const uint8_t* xt = bf16_rows(x, r0, Dm);
    const uint8_t* dyt = bf16_rows(dy, r0, Dm);
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
    gx.c = static_cast<uint8_t*>(dx) + r0 * Dm * 2;
    gx.ldc = Dm;
    gx.err = err;
    LOSS_CUDA(launch_gemm_tc(kEpiStoreBf16, false, true, t_dgu_k, t_wgu_mn, gx, cap, stream));
  }
  return UPIPE_OK;
}

}  // extern "C"
