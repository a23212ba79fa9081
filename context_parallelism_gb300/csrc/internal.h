// Interface between the host-side scheduler (api.cpp) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cstdio>

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

namespace upipe {

// NVTX range for the lifetime of a scope (a call, a head group, a tile), visible in profilers
// that record NVTX; without one attached, a push/pop pair is a few nanoseconds of host time.
class NvtxRange {
 public:
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  NvtxRange(const char* fmt, long long i) {
    char buf[64];
    snprintf(buf, sizeof(buf), fmt, i);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---- attention workspace plan (api.cpp) ----------------------------------------------------
// Byte offsets of every arena segment of the attention calls, each 256-byte aligned. f_* are
// the forward's segments, b_* the backward's; *_total is each pass's size.
struct AttnPlan {
  int B = 0, Hq = 0, Hkv = 0, D = 0, G = 0, hc = 0, kc = 0, causal = 1;
  int64_t S = 0, T = 0, S_pad = 0, T_pad = 0;
  int n_trunks = 0;
  bool kv_host = false;
  bool act_host = false;  // q/o (and dout/dq) may be pinned host memory: staging reserved
  // forward segments
  size_t f_qw = 0, f_kw = 0, f_vw = 0, f_slot_k[2] = {0, 0}, f_slot_v[2] = {0, 0};
  size_t f_qw2 = 0, f_ostg[2] = {0, 0};  // host activations: second Q buffer, O staging
  size_t f_state_o = 0, f_state_ml = 0, f_total = 0;
  // backward segments
  size_t b_qw = 0, b_dow = 0, b_kw = 0, b_vw = 0, b_slot_k[2] = {0, 0}, b_slot_v[2] = {0, 0};
  size_t b_slot_dk[2] = {0, 0}, b_slot_dv[2] = {0, 0};  // host-K/V mode: dK/dV trunk slots
  // host activations: second Q and dO buffers, head-major O copies, dQ output stagings
  size_t b_qw2 = 0, b_dow2 = 0, b_ow[2] = {0, 0}, b_dqs[2] = {0, 0};
  size_t b_dqacc = 0, b_lse2 = 0, b_dvec = 0, b_total = 0;
  // Split backward (short causal sequences, see make_attn_plan): each key tile's walk is shared
  // by bwd_split CTAs, whose fp32 dK/dV shares of part_rows key rows live at b_dkv_part.
  int bwd_split = 1;
  int64_t part_rows = 0;
  size_t b_dkv_part = 0;
};


// Validates the shape arguments of the attention calls (no device access) and fills the plan.
// host_mask: UPIPE_HOST_KV / UPIPE_HOST_ACT reserve the staging segments of pinned-host tensors.
// Returns UPIPE_OK, or UPIPE_ERR_INVALID_ARG / UPIPE_ERR_UNSUPPORTED with the reason recorded
// for upipe_last_error_message().
int make_attn_plan(int B, int64_t S, int Hq, int Hkv, int D, int causal, int head_chunk,
                   int64_t seq_trunk, int host_mask, AttnPlan* p);

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device, once per
// (kernel, device): the attribute is per device, so a process that drives several GPUs sets it
// on each. Thread-safe.
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

// Restores the caller's current device when the scope ends (the entry points select the
// device their tensors live on, and must not leave it changed).
class DeviceGuard {
 public:
  DeviceGuard() {
    if (cudaGetDevice(&prev_) != cudaSuccess) {
      cudaGetLastError();
      prev_ = -1;
    }
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev_) cudaSetDevice(prev_);
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;

 private:
  int prev_ = -1;
};

// ---- launch bookkeeping (api.cpp) ---------------------------------------------------------
// Every kernel launch goes through begin/end so the library can count launches and, when
// profiling is on, bracket each one with CUDA events on its own stream.
void launch_begin(int kclass, cudaStream_t stream);
void launch_end(int kclass, cudaStream_t stream);
// The same bracketing for a host<->device copy (profiling only; not a launch).
void copy_begin(cudaStream_t stream);
void copy_end(int kclass, cudaStream_t stream);

// Records the message upipe_last_error_message() returns on this thread.
void set_last_error(const char* msg);

// Builds a 3-D bf16 tensor map over a dense [depth][rows][cols] array with a box of
// box_rows rows x 64 columns and 128-byte swizzle (cols % 64 == 0). Returns cudaSuccess or an
// error if the driver refused the map.
cudaError_t make_tmap_bf16(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                           int64_t depth, int box_rows = 128);

// ---- forward attention (attn_fwd.cu) -------------------------------------------------------
struct FwdArgs {
  int64_t q_lo, q_hi;            // global query rows covered by this launch (one Q trunk)
  int64_t kv_row_lo, kv_row_hi;  // rows of the K/V map used by this launch (one KV trunk)
  int64_t kv_pos0;               // global token position of K/V map row 0
  int64_t S;                     // sequence length
  int hc, kc, G, Hq, h0;         // group q-heads, group kv-heads, Hq/Hkv, total q-heads, first q-head
  int causal, first, last;       // first: no carried state; last: finalise O and LSE
  int64_t last_q_end;            // with last: only query tiles starting below it are final
                                 // (the rest store their state); 0 = every tile
  float scale_log2;              // softmax scale * log2(e)
  void* o;                       // bf16, written when last: [B,S,Hq,D], or a staging [B,S,o_heads,D]
  int o_heads, o_head0;          // heads per row of o and this group's first; 0 means Hq and h0
  float* lse;                    // [B,Hq,S], written when last
  float* state_o;                // [B*hc][state_stride][D] fp32 running numerator (rows from q_lo)
  float* state_ml;               // [B*hc][state_stride][2] fp32 running max (log2 units), sum
  int64_t state_rows;            // rows of this launch's state (rows past it are never stored)
  int64_t state_stride;          // rows per head in the state buffers; 0 means state_rows
  int band;                      // launch order, set by launch_attn_fwd (see launch_band)
  uint32_t* err;                 // device status word
};

// Launch order of the attention kernels. A launch is `lanes` independent sequences of work
// units (a head's query-tile pairs, a kv-head's key tiles), each ordered heaviest first. Lanes
// go in bands of `band` lanes: inside a band the units interleave across lanes, heaviest of
// every lane first; bands run one after the other. A band holds at least eight waves of units
// on the current device and the bands are of equal size, so long launches run a lane or two at
// a time (their CTAs share Q/dO or K/V tiles in L2: interleaving the eight kv-heads of a 256K,
// 64-head backward ran at two thirds of the speed) and short ones interleave every lane (no
// lane's heavy units start last).
int launch_band(int64_t units_per_lane, int lanes);

// q_map: Q workspace [B*hc][S][D]; k_map / v_map: [B*kc][kv_rows][D].
cudaError_t launch_attn_fwd_generic(int D, int B, const CUtensorMap& q_map,
                                    const CUtensorMap& k_map, const CUtensorMap& v_map,
                                    const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_attn_fwd(int D, int B, const CUtensorMap& q_map, const CUtensorMap& k_map,
                            const CUtensorMap& v_map, const FwdArgs& a, cudaStream_t stream);

// One forward launch over the whole sequence of head group h0..h0+hc-1 with device-resident,
// head-major Q/K/V maps: every key/value trunk folded in with the running state on chip, O and
// LSE finalised. o: token-major [B,S,Hq,D] (o_heads = 0) or a group staging [B,S,o_heads,D];
// lse may be NULL (prefill). Used by upipe_attn_fwd and the no-allocation forward.
cudaError_t launch_fwd_resident(const AttnPlan& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, int h0, void* o, int o_heads, float* lse,
                                uint32_t* err, cudaStream_t stream);

// ---- backward attention (attn_bwd.cu) ------------------------------------------------------
struct BwdArgs {
  int64_t kv_row_lo, kv_row_hi;  // K/V map rows of this launch (one KV trunk)
  int64_t kv_pos0;               // global token position of K/V map row 0
  int64_t S, S_pad;              // sequence length, per-head row pitch of lse2/dvec/dqacc
  int hc, kc, G, Hkv, kvh0;      // group sizes, total kv-heads, first kv-head of the group
  int causal;
  float scale, scale_log2;
  const float* lse2;             // [B*hc][S_pad] -LSE * log2(e)
  const float* dvec;             // [B*hc][S_pad] -scale * D_i,  D_i = <dO_i, O_i>
  float* dqacc;                  // [B*hc][S_pad][D] fp32 dQ accumulator
  // dK / dV rows: element (b, key position p, kv-head kvl of the group, d) is written at
  // ((b * dkv_rows + p - dkv_row0) * dkv_heads + dkv_head0 + kvl) * D: the token-major outputs
  // [B,S,Hkv,D] (rows S, row0 0, heads Hkv, head0 kvh0) or a trunk slot [B,Tn,kc,D].
  void* dk;
  void* dv;
  int64_t dkv_rows, dkv_row0;
  int dkv_heads, dkv_head0;
  // split > 1 (a divisor of G): each key tile's walk is shared by `split` CTAs, CTA sp taking
  // q-heads [sp*G/split, (sp+1)*G/split) of the group; each writes its fp32 dK, dV share of
  // key row r (launch-relative, r = p - kv_pos0 - kv_row_lo) to
  // dkv_part + (((sp * B + b) * kc + kvl) * part_rows + r) * 2 * D, dK in the first D floats,
  // dV in the next, and launch_dkdv_reduce adds the shares up. split = 1: dk, dv as above.
  int split;
  float* dkv_part;
  int64_t part_rows;
  int band;                      // launch order, set by launch_attn_bwd (see launch_band)
  uint32_t* err;
};

// q_map / do_map: [B*hc][S][D] with boxes of bwd_q_box_rows(D) rows; k_map / v_map:
// [B*kc][kv_rows][D] with 128-row boxes.
int bwd_q_box_rows(int D);
cudaError_t launch_attn_bwd_generic(int D, int B, const CUtensorMap& q_map,
                                    const CUtensorMap& do_map, const CUtensorMap& k_map,
                                    const CUtensorMap& v_map, const BwdArgs& a,
                                    cudaStream_t stream);
cudaError_t launch_attn_bwd(int D, int B, const CUtensorMap& q_map, const CUtensorMap& do_map,
                            const CUtensorMap& k_map, const CUtensorMap& v_map,
                            const BwdArgs& a, cudaStream_t stream);

// ---- HBM-bound helpers (layout.cu) ---------------------------------------------------------
// dst[b][h][s][:] = src[b][s][h_begin + h][:]  for h < h_count   (bf16, D % 8 == 0)
cudaError_t launch_seq_to_head(const void* src, void* dst, int B, int64_t S, int H, int D,
                               int h_begin, int h_count, cudaStream_t stream);
// Up to three gathers in one launch: job i copies heads [h0[i], h0[i] + count[i]) of the
// token-major [B,S,H[i],D] tensor src[i] into the head-major [B,count[i],S,D] buffer dst[i].
cudaError_t launch_gather_group(const void* const* src, void* const* dst, const int* H,
                                const int* h0, const int* count, int n, int B, int64_t S, int D,
                                cudaStream_t stream);
// dst[b][s][h_begin + h][:] = src[b][h][s][:]
cudaError_t launch_head_to_seq(const void* src, void* dst, int B, int64_t S, int H, int D,
                               int h_begin, int h_count, cudaStream_t stream);

// Backward pre-pass for one head group (q-heads h0 .. h0+hc-1):
//   dow[b*hc+h][s][:] = dout[b][s][h0+h][:]
//   dvec[(b*hc+h)*S_pad + s] = -scale * sum_d dout*o (fp32), lse2[...] = -lse[b][h0+h][s]*log2(e)
//   (stored negated: the kernels add them with one fused multiply-add)
//   dqacc[(b*hc+h)*S_pad + s][:] = 0
// rows s in [S, S_pad) get dvec = lse2 = 0 and zeroed dqacc.
// head_major_in: o and dout are this group's head-major [B*hc][S][D] copies (dout == dow,
// not rewritten) instead of the token-major tensors.
cudaError_t launch_bwd_pre(const void* o, const void* dout, const float* lse, void* dow,
                           float* dvec, float* lse2, float* dqacc, int B, int64_t S,
                           int64_t S_pad, int Hq, int D, int h0, int hc, float scale,
                           int head_major_in, cudaStream_t stream);

// Sums the split backward's shares (BwdArgs::split, dkv_part) of key rows [0, rows) in order
// sp = 0, 1, ... and writes them as bf16 with the epilogue's addressing: element (b, row r,
// kv-head kvl, d) of dK goes to dk[((b * dkv_rows + row0_pos + r - dkv_row0) * dkv_heads +
// dkv_head0 + kvl) * D + d], dV likewise; rows with row0_pos + r >= S are skipped.
cudaError_t launch_dkdv_reduce(const float* part, int split, int64_t part_rows, int64_t rows,
                               int64_t row0_pos, int B, int kc, int D, int64_t S, void* dk,
                               void* dv, int64_t dkv_rows, int64_t dkv_row0, int dkv_heads,
                               int dkv_head0, cudaStream_t stream);

// dq[b][s][h0+h][:] = bf16(dqacc[(b*hc+h)*S_pad + s][:])
// dq rows of out_heads heads, this group's at [out_head0, out_head0 + hc): (Hq, h0) for the
// token-major output, (hc, 0) for a group staging [B,S,hc,D].
cudaError_t launch_dq_convert(const float* dqacc, void* dq, int B, int64_t S, int64_t S_pad,
                              int out_heads, int D, int out_head0, int hc, cudaStream_t stream);

// ---- sequence-tiled loss (gemm_tc.cu) ------------------------------------------------------
// C[m, n] = sum_k A(m, k) B(n, k) over 128 x 256 tiles, with the epilogue chosen by `epi`.
enum : int {
  kEpiCeFwd = 0,
  kEpiCeBwd = 1,
  kEpiStoreBf16 = 2,
  kEpiAccF32 = 3,
  kEpiSwiglu = 4,   // N = F outputs per row; B = w_gu [2F][K] with the up block at row `split`
  kEpiDSwiglu = 5,  // c = dgu [M][2F]: dg at column j, du at split + j; aux = gu likewise
};

struct GemmArgs {
  int M, N, K;            // N % 64 == 0; M, K any (tensor maps zero-fill past the edges)
  int m_fastest;          // tile order: 1 walks M tiles first (shares a B strip), 0 N tiles first
  int group_m;            // tiles of the fast dimension per group (<= 0: all), see tile_coords
  void* c;                // STORE: bf16 [M][ldc]; ACC_F32: fp32 [M][ldc]; CE_BWD: bf16 dlogits;
                          // CE_FWD: optional fp32 logits [M][ldc] (NULL: not stored)
  int64_t ldc;
  int accumulate;         // ACC_F32: add into c instead of overwriting
  const int64_t* target;  // CE: [M] vocabulary index of each row's target, < 0 = ignored
  const float* lse;       // CE_BWD: [M] natural-log log-sum-exp of each row's logits
  const float* g;         // CE_BWD: [M] upstream gradient of each row's loss
  float* part;            // CE_FWD: float2 [ceil(N/256)][part_stride] (max in log2 units, sum)
  int64_t part_stride;
  float* tlogit;          // CE_FWD: [M] logit at the target
  void* c2;               // SWIGLU: optional bf16 g | u store [M][ldc2] (u at column split + j)
  int64_t ldc2;
  const void* aux;        // DSWIGLU: bf16 g | u [M][ld_aux]
  int64_t ld_aux;
  int split;              // SWIGLU / DSWIGLU: F, the offset of the up half
  uint32_t* err;
};

// Supported (epi, A MN-major, B MN-major): (CE_FWD, 0, 0), (CE_BWD, 0, 0), (STORE, 0, 1),
// (STORE, 0, 0), (ACC_F32, 1, 1), (SWIGLU, 0, 0), (DSWIGLU, 0, 1). K-major maps have 128-row
// (A) / 256-row (B; 128-row for SWIGLU, loaded twice) boxes; MN-major maps 64-row boxes; all
// 64 columns wide with 128-byte swizzle. The grid is min(tiles, grid_cap) CTAs.
cudaError_t launch_gemm_tc(int epi, bool a_mn, bool b_mn, const CUtensorMap& ta,
                           const CUtensorMap& tb, const GemmArgs& a, int grid_cap,
                           cudaStream_t stream);

// dl[r][j] (bf16 [M][V]) = g_r (exp(logits[r][j] - lse_r) - [j == target_r]) from stored fp32
// logits [M][V]: bitwise what the CE_BWD epilogue gives on recomputed logits.
cudaError_t launch_ce_dlogits(const float* logits, const float* lse, const int64_t* target,
                              const float* g, void* dl, int64_t M, int64_t V, cudaStream_t stream);

// loss[r], lse[r] for r < M from the CE_FWD partials of n_parts column tiles (V: vocabulary
// size, for the out-of-range target check).
cudaError_t launch_ce_merge(const float* part, int64_t part_stride, int n_parts,
                            const float* tlogit, const int64_t* target, float* loss, float* lse,
                            int64_t M, int64_t V, cudaStream_t stream);

// ---- services of api.cpp to the other entry points -----------------------------------------
// Per-device state (streams, status word) for `dev`, created on first use; a upipe status.
int device_status_word(int dev, uint32_t** err);

// Releases the sequence-tiled calls' copy streams and events (seqtile_api.cpp); part of
// upipe_shutdown.
void seqtile_shutdown();

// Test hook (upipe_debug_fail_copy_after): true when the staging copy about to be issued is the
// one armed to fail; the caller then returns UPIPE_ERR_CUDA without issuing it. Counts every
// host<->device staging copy of every call while armed.
bool staging_copy_fails();

// ---- self-tests (selftest.cu) --------------------------------------------------------------
cudaError_t launch_selftest_umma(const void* a, const void* b, float* c, int N, int K,
                                 int a_mn, int b_mn, int a_manual, int lbo, int sbo,
                                 uint32_t* err, cudaStream_t stream);
cudaError_t launch_selftest_wait(int limit_us, uint32_t* err, cudaStream_t stream);

}  // namespace upipe
