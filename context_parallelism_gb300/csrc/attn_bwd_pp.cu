// Backward causal (GQA) attention for D = 128 on sm_103a: 128-row query tiles, every tcgen05
// MMA at M = 128, N = 128, with two compute warpgroups splitting each tile's columns.
//
// One CTA owns a 128-row key/value tile of one kv-head (K and V stay in shared memory) and walks
// the 128-row query tiles of every q-head of its group that can see the tile; the probabilities
// are recomputed from the saved log-sum-exp, never stored ("Training Ultra Long Context LM with
// Fully Pipelined Distributed Transformer", Background: the attention backward pass is the memory
// peak; "Road to 5 million sequence length" talk, UPipe passage: each head group is recomputed).
//
// Per query tile i (key row j = TMEM lane of S^T and dP^T, query row q):
//   S^T  = K Q^T                 tcgen05 (M 128, N 128, K 128)  -> TMEM S
//   dP^T = V dO^T                tcgen05                         -> TMEM dP
//   P^T  = exp2(S^T*scale*log2e - LSE*log2e), masked; bf16 back into TMEM S
//   dS^T = P^T * (scale*dP^T - scale*D)                bf16 -> shared memory (two boxes)
//   (the pre-pass stores -LSE*log2e and -scale*D, so each is one fused multiply-add)
//   dV  += P^T dO                tcgen05 with A read from TMEM
//   dK  += dS^T Q                tcgen05 (A K-major, B MN-major)
//   dQ^T = K^T dS^T              tcgen05 (M 128 = head dim, N 128)  -> TMEM dP (dP is consumed)
//   dQ  += dQ^T read back with lanes = head dim: one contiguous 128-byte line per query row and
//          warp, added with fire-and-forget fp32 reductions.
// Compute group w in {0, 1} owns query columns [64w, 64w+64) of every tile. Its packed P^T goes
// to S columns [64w, 64w+32) (inside the columns it alone reads), and its dS^T to shared box w.
// A third warpgroup drains dQ^T(i) from TMEM into the fp32 accumulator, off the groups' path.
//
// MMA issue order: S(0), dP(0), dV(0), then per tile i: S(i+1), dQ(i), dK(i), dP(i+1), dV(i+1).
// Each group runs dS(i) then P(i+1): its dS(i) overlaps S(i+1), and its P(i+1) overlaps dQ(i),
// dK(i) and dP(i+1), so dP(i+1) is ready when the group turns to dS(i+1) (issued before dV(i+1),
// which must wait for P(i+1)). The drain reads dQ(i) while dK(i) runs (dQ goes first for that)
// and releases the columns dP(i+1) reuses. One thread's MMAs execute in order, so S(i+1)
// overwrites S only after dV(i) has read P^T(i); the commit that publishes dP(i+1) also covers
// dK(i) and dQ(i), which read the single dS^T buffer the groups then overwrite; and the commit
// that frees the dO stage (after dV(i+1)) covers dP(i+1), its other reader. Q has three stages
// and dO one: Q(i+1) must be resident when S(i+1) is issued, at the top of the tile, and a
// third stage lets its load start a whole tile earlier (Q(i+1) overwrites Q(i-2)); dO(i+1) is
// needed only by dP(i+1), after S(i+1), dQ(i) and dK(i), which leaves its load time enough.
//
// Threads (512): warps 0-3 compute group 0, warps 4-7 compute group 1, warps 8-11 dQ drain,
// warp 12 TMEM + MMA issue, warp 13 TMA producer, warps 14-15 idle. Registers move from the
// MMA/TMA warpgroup to the compute groups and the drain (152 / 152 / 152 / 56 per thread).
// TMEM: dV [0,128), dK [128,256), S [256,384), dP/dQ [384,512).
// Shared memory (226 KB, no alignment slack to spare: the dynamic window must start 1 KiB-
// aligned, which is checked): K, V, three Q stages, one dO stage, dS^T, two LSE/D vector
// stages (each freed by both groups' dS of its tile), barriers.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr int kTile = 128 * kD * 2;  // 32 KiB

struct BppLayout {
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;         // 3 stages
  static constexpr int kDO = kQ + 3 * kTile;    // 1 stage
  static constexpr int kDS = kDO + kTile;       // 2 boxes: query columns 0-63, 64-127
  static constexpr int kVec = kDS + kTile;      // 2 stages x (128 LSE2 + 128 D) fp32
  static constexpr int kBar = kVec + 2 * 1024;
  static constexpr int kNumBars = 19;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 4;
  static constexpr int kBytes = kAbort + 4;
};
static_assert(BppLayout::kBytes <= 232448, "shared memory budget");

// A CTA walks the query tiles q-head outer (of its kv-head's group), tile inner. Each role
// steps its own cursor through that walk one tile at a time: no division per tile.
struct Cursor {
  int head = 0, qt = 0;
  __device__ void next(int n) {
    if (++qt == n) {
      qt = 0;
      ++head;
    }
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_pp_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const BwdArgs a) {
  using L = BppLayout;
  extern __shared__ __align__(1024) uint8_t smem[];
  // TMA 128-byte swizzle needs 1 KiB-aligned tiles; refuse to run otherwise (no fault).
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrWaitTimeout | 0x10000u);
    return;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bar;
  uint64_t* qf = bar + 1;        // [3] Q stage (and its tile's LSE/D vectors) landed
  uint64_t* qe = bar + 4;        // [3] Q stage free (after dK)
  uint64_t* df = bar + 7;        // dO landed
  uint64_t* de = bar + 8;        // dO free (after dV)
  uint64_t* s_full = bar + 9;
  uint64_t* dp_full = bar + 10;
  uint64_t* dq_full = bar + 11;
  uint64_t* p_ready = bar + 12;  // 8 warp arrivals
  uint64_t* ds_ready = bar + 13; // 8
  uint64_t* dq_free = bar + 14;  // 4 drain-warp arrivals
  uint64_t* done = bar + 15;
  uint64_t* drain = bar + 16;
  uint64_t* vfree = bar + 17;    // [2] LSE/D vector stage read by both groups (8 warp arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // One-dimensional grid over (key tile, lane), lane = (batch, kv-head, share) and the
  // smallest key positions (the longest causal walks) first, in bands of a.band lanes: inside
  // a band the lanes' key tiles interleave, the band's longest walks first; bands follow one
  // another.
  const int split = a.split > 1 ? a.split : 1;
  const int ny = a.kc * split;
  const int n_kt = static_cast<int>((a.kv_row_hi - a.kv_row_lo + 127) / 128);
  const int nb = static_cast<int>(gridDim.x) / (n_kt * ny);  // batch
  int kt, yb;
  {
    const int L = static_cast<int>(blockIdx.x), lanes = ny * nb;
    const int band = L / (a.band * n_kt);
    const int lane0 = band * a.band;
    const int bl = min(a.band, lanes - lane0);  // lanes of this band
    const int u = L - lane0 * n_kt;
    kt = u / bl;
    yb = lane0 + (u - kt * bl);
  }
  const int yy = yb % ny;
  const int b = yb / ny;
  const int kvl = yy / split;
  const int sp = yy - kvl * split;  // share of the group's q-heads
  const int gh = a.G / split;       // q-heads this CTA walks
  const int64_t r0 = a.kv_row_lo + static_cast<int64_t>(kt) * 128;  // K/V map row
  const int64_t p0 = a.kv_pos0 + r0;                                // global key position
  const int zk = b * a.kc + kvl;
  const int qt_lo = a.causal ? static_cast<int>(p0 / 128) : 0;
  const int qt_hi = static_cast<int>((a.S + 127) / 128);
  const int nq = qt_hi > qt_lo ? qt_hi - qt_lo : 0;
  const int n_it = gh * nq;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(qf + s, 1);
      mbar_init(qe + s, 1);
    }
    mbar_init(df, 1);
    mbar_init(de, 1);
    mbar_init(vfree, 8);
    mbar_init(vfree + 1, 8);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(dq_full, 1);
    mbar_init(p_ready, 8);
    mbar_init(ds_ready, 8);
    mbar_init(dq_free, 4);
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tDV = tmem, tDK = tmem + 128, tS = tmem + 256, tDP = tmem + 384;

  // Bounded wait: the clock and the abort flag are checked every 32 failed polls.
  auto wait = [&](uint64_t* br, uint32_t parity) -> bool {
    if (mbar_try_wait(br, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
      if (mbar_try_wait(br, parity)) return true;
      if ((n & 31) == 0) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          *abort_flag = 1;
          atomicOr(a.err, kErrWaitTimeout | 0x4000u);
          return false;
        }
      }
    }
  };
  auto decode = [&](const Cursor& c, int& zq, int64_t& q0) {
    zq = b * a.hc + kvl * a.G + sp * gh + c.head;
    q0 = static_cast<int64_t>(qt_lo + c.qt) * 128;
  };

  // Launched with 512 x 128 registers. The MMA/TMA warpgroup gives up 72, the dQ drain and each
  // compute group take 24 more: 128 * (56 + 3 * 152) = 65536, exactly the launch's pool. Each
  // role's code sits inside the branch that sets its count, so the compiler allocates that code
  // for it.
  if (warp >= 12) {
  setmaxnreg_dec<56>();
  if (warp == 13) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(kv_full, 2 * kTile);
      for (int x = 0; x < 2; ++x) {
        tma_load_3d(smem + L::kK + x * kBoxBytes, &tm_k, x * 64, static_cast<int>(r0), zk, kv_full);
        tma_load_3d(smem + L::kV + x * kBoxBytes, &tm_v, x * 64, static_cast<int>(r0), zk, kv_full);
      }
      int q_issued = 0, d_issued = 0;
      bool ok = true;
      Cursor cur;
      int st = 0, sq = 0;  // Q stage it % 3 and its use count it / 3
      for (int it = 0; it < n_it; ++it, cur.next(nq)) {
        int zq;
        int64_t q0;
        decode(cur, zq, q0);
        // Q(it) overwrites Q(it - 3), last read by dK(it - 3); its LSE/D vectors overwrite
        // tile it - 2's, last read by the groups' dS(it - 2)
        if (it >= 3 && !wait(qe + st, (sq - 1) & 1)) { ok = false; break; }
        if (it >= 2 && !wait(vfree + (it & 1), ((it >> 1) - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(qf + st, kTile + 1024);
        for (int x = 0; x < 2; ++x)
          tma_load_3d(smem + L::kQ + st * kTile + x * kBoxBytes, &tm_q, x * 64,
                      static_cast<int>(q0), zq, qf + st);
        const int64_t vo = static_cast<int64_t>(zq) * a.S_pad + q0;
        uint8_t* vec = smem + L::kVec + (it & 1) * 1024;
        bulk_load(vec, a.lse2 + vo, 512, qf + st);
        bulk_load(vec + 512, a.dvec + vo, 512, qf + st);
        q_issued = it + 1;
        // dO(it) goes into the single dO stage once dV(it - 1) has read it
        if (it >= 1 && !wait(de, (it - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(df, kTile);
        for (int x = 0; x < 2; ++x)
          tma_load_3d(smem + L::kDO + x * kBoxBytes, &tm_do, x * 64, static_cast<int>(q0), zq, df);
        d_issued = it + 1;
        if (++st == 3) {
          st = 0;
          ++sq;
        }
      }
      mbar_wait(kv_full, 0, ok ? kWaitLimitNs : 100000000ull);
      if (!ok) {  // let every load already issued land before the CTA can exit
        for (int it = (q_issued > 3 ? q_issued - 3 : 0); it < q_issued; ++it)
          mbar_wait(qf + it % 3, (it / 3) & 1, 100000000ull);
        if (d_issued > 0) mbar_wait(df, (d_issued - 1) & 1, 100000000ull);
      }
    }
  } else if (warp == 12) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_kk = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      const uint32_t id_kmn = idesc_bf16(128, 128, false, true);  // dV (A in TMEM), dK
      const uint32_t id_mnmn = idesc_bf16(128, 128, true, true);  // dQ^T = K^T dS^T
      // Every descriptor is one base descriptor (K-major or MN-major, at the start of shared
      // memory) plus a compile-time offset in 16-byte units. The base goes through an opaque
      // move at each use, so the compiler cannot precompute the 40 per-step descriptors of a
      // tile into registers: this warpgroup runs on 56 registers.
      const uint64_t base_k = kdesc0(smem_u32(smem));
      const uint64_t base_mn = mndesc0(smem_u32(smem));
      constexpr uint32_t kStageU = kTile >> 4;
      constexpr uint32_t uK = L::kK >> 4, uV = L::kV >> 4, uQ = L::kQ >> 4, uDO = L::kDO >> 4,
                         uDS = L::kDS >> 4;
      bool ok = wait(kv_full, 0);

      auto issue_s = [&](int i) -> bool {
        const int st = i % 3;
        if (!wait(qf + st, (i / 3) & 1)) return false;
        tc_fence_after();
        const uint64_t bk = opaque_u64(base_k);
        const uint32_t uq = uQ + st * kStageU;
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tS, bk + (uK + kstep(k16)), bk + (uq + kstep(k16)), id_kk,
                      k16 > 0 ? 1u : 0u);
        umma_commit(s_full);
        return true;
      };
      auto issue_dv = [&](int i) -> bool {
        if (!wait(p_ready, i & 1)) return false;
        if (!wait(df, i & 1)) return false;
        tc_fence_after();
        const uint64_t bmn = opaque_u64(base_mn);
        const uint32_t udo = uDO;
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)  // group 0's P^T at S+0, group 1's at S+64
          umma_f16_ts(tDV, tS + (k16 >> 2) * 64 + (k16 & 3) * 8, bmn + (udo + mnstep(k16)),
                      id_kmn, k16 > 0 ? 1u : acc0);
        umma_commit(de);
        return true;
      };
      auto issue_dp = [&](int i) -> bool {
        if (i >= 1 && !wait(dq_free, (i - 1) & 1)) return false;
        if (!wait(df, i & 1)) return false;
        tc_fence_after();
        const uint64_t bk = opaque_u64(base_k);
        const uint32_t udo = uDO;
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tDP, bk + (uV + kstep(k16)), bk + (udo + kstep(k16)), id_kk,
                      k16 > 0 ? 1u : 0u);
        umma_commit(dp_full);
        return true;
      };
      auto issue_dk_dq = [&](int i) -> bool {
        const int st = i % 3;
        if (!wait(ds_ready, i & 1)) return false;
        tc_fence_after();
        const uint64_t bmn = opaque_u64(base_mn);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tDP, bmn + (uK + mnstep(k16)), bmn + (uDS + mnstep(k16)), id_mnmn,
                      k16 > 0 ? 1u : 0u);
        umma_commit(dq_full);
        const uint64_t bk = opaque_u64(base_k);
        const uint64_t bmn2 = opaque_u64(base_mn);
        const uint32_t uq = uQ + st * kStageU;
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tDK, bk + (uDS + kstep(k16)), bmn2 + (uq + mnstep(k16)), id_kmn,
                      k16 > 0 ? 1u : acc0);
        umma_commit(qe + st);
        return true;
      };

      if (ok && n_it > 0) ok = issue_s(0) && issue_dp(0) && issue_dv(0);
      for (int i = 0; ok && i < n_it; ++i) {
        if (i + 1 < n_it && !issue_s(i + 1)) { ok = false; break; }
        if (!issue_dk_dq(i)) { ok = false; break; }
        if (i + 1 < n_it && !(issue_dp(i + 1) && issue_dv(i + 1))) { ok = false; break; }
      }
      if (ok) {
        umma_commit(done);
      } else {
        umma_commit(drain);
        mbar_wait(drain, 0, 100000000ull);
      }
    }
  }  // warps 14-15: idle, they only complete the warpgroup of the MMA and TMA warps
  } else if (warp >= 8) {
    setmaxnreg_inc<152>();
    // ---------------- dQ drain ----------------
    // dQ^T(i): lane t = head-dim index d, column c = query row q0 + c. The drain reads all 128
    // columns into registers and releases them at once (dP(i+1) reuses them), then adds each
    // query row's 128 floats as one contiguous 128-byte line per warp, fire-and-forget, while
    // the tensor pipe already runs the next tile. Query rows past S fall in the accumulator's
    // padding (S_pad rows per head, a multiple of 128) and add exact zeros there (their P is
    // masked to 0), so no bound check.
    const int t = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    Cursor cur;
    for (int i = 0; i < n_it; ++i, cur.next(nq)) {
      if (!__all_sync(0xffffffffu, wait(dq_full, i & 1))) break;
      tc_fence_after();
      int zq;
      int64_t q0;
      decode(cur, zq, q0);
      float* dq_col = a.dqacc + (static_cast<int64_t>(zq) * a.S_pad + q0) * kD + t;
      uint32_t ra[64], rb[64];
      tmem_ld64_nowait(tDP + lane_off, ra);
      tmem_ld64_nowait(tDP + lane_off + 64, rb);
      tmem_wait_ld_dep64(ra);
      tmem_reg_dep64(rb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
#pragma unroll
      for (int x = 0; x < 64; ++x) red_add_f32(dq_col + x * kD, __uint_as_float(ra[x]));
#pragma unroll
      for (int x = 0; x < 64; ++x) red_add_f32(dq_col + (64 + x) * kD, __uint_as_float(rb[x]));
    }
  } else {
    setmaxnreg_inc<152>();
    // ---------------- compute groups ----------------
    const int w = warp >> 2;              // owns query columns [64w, 64w+64)
    const int t = threadIdx.x & 127;      // key row (S^T/dP^T lanes)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t sDS = smem_u32(smem + L::kDS + w * kBoxBytes);
    const int64_t pj = p0 + t;
    const bool key_ok = (r0 + t) < a.kv_row_hi;
    const uint64_t sl2 = f2_pack(a.scale_log2, a.scale_log2);
    const uint64_t sc2 = f2_pack(a.scale, a.scale);
    float p[64];  // this group's P^T row of the tile in flight
    Cursor cur_p;  // the tile do_p handles next
    // P^T(i) of this group's columns: S^T -> exp2 -> bf16 back into its own S columns.
    auto do_p = [&](int i) -> bool {
      const int st = i & 1;  // LSE/D vector stage
      int zq;
      int64_t q0;
      decode(cur_p, zq, q0);
      cur_p.next(nq);
      const int64_t qc0 = q0 + 64 * w;  // first query row of this group's columns
      const float* lse_s = reinterpret_cast<const float*>(smem + L::kVec + st * 1024) + 64 * w;
      // qf: the LSE/D vectors of this tile landed (the stage is refilled only after dK(i),
      // which needs this group's ds_ready).
      if (!__all_sync(0xffffffffu, wait(qf + i % 3, (i / 3) & 1) && wait(s_full, i & 1)))
        return false;
      tc_fence_after();
      const bool need_mask = (a.causal && qc0 < p0 + 127) || (qc0 + 64 > a.S) ||
                             (r0 + 128 > a.kv_row_hi);
      uint32_t r[64];
      tmem_ld64_sync(tS + lane_off + 64 * w, r);
      // Two 32-column halves: the first half's bf16 P^T is stored while the second half is
      // exponentiated, so the store's latency is hidden behind MUFU work.
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int x = 32 * hh; x < 32 * hh + 32; x += 4) {
          // -LSE*log2e pairs straight from shared memory as packed fp32x2 operands
          const ulonglong2 l4 = *reinterpret_cast<const ulonglong2*>(lse_s + x);
          float y0, y1, y2, y3;
          f2_unpack(ffma2(f2_pack_u(r[x], r[x + 1]), sl2, l4.x), y0, y1);
          f2_unpack(ffma2(f2_pack_u(r[x + 2], r[x + 3]), sl2, l4.y), y2, y3);
          p[x + 0] = ex2_approx(y0);
          p[x + 1] = ex2_approx(y1);
          p[x + 2] = ex2_approx(y2);
          p[x + 3] = ex2_approx(y3);
        }
        if (need_mask) {
#pragma unroll
          for (int c = 32 * hh; c < 32 * hh + 32; ++c) {
            const int64_t q = qc0 + c;
            if (!(key_ok && q < a.S && (!a.causal || q >= pj))) p[c] = 0.f;
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) pk[x] = pack_bf16(p[32 * hh + 2 * x], p[32 * hh + 2 * x + 1]);
        tmem_st16(tS + lane_off + 64 * w + 16 * hh, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
      return true;
    };
    // dS^T(i) of this group's columns -> shared box w.
    auto do_ds = [&](int i) -> bool {
      const float* dv_s =
          reinterpret_cast<const float*>(smem + L::kVec + (i & 1) * 1024) + 128 + 64 * w;
      if (!__all_sync(0xffffffffu, wait(dp_full, i & 1))) return false;
      tc_fence_after();
      uint32_t r[64];
      tmem_ld64_sync(tDP + lane_off + 64 * w, r);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        // -scale*D pairs straight from shared memory as packed fp32x2 operands
        const ulonglong2 da = *reinterpret_cast<const ulonglong2*>(dv_s + u * 8);
        const ulonglong2 db = *reinterpret_cast<const ulonglong2*>(dv_s + u * 8 + 4);
        const uint64_t dvv[4] = {da.x, da.y, db.x, db.y};
        uint32_t pk[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int col = u * 8 + 2 * x;
          const uint64_t t2 = ffma2(f2_pack_u(r[col], r[col + 1]), sc2, dvv[x]);
          float d0, d1;
          f2_unpack(fmul2(t2, f2_pack(p[col], p[col + 1])), d0, d1);
          pk[x] = pack_bf16(d0, d1);
        }
        st_shared_v4(sDS + swz_offset(t, u * 8), pk[0], pk[1], pk[2], pk[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(ds_ready);
        mbar_arrive(vfree + (i & 1));
      }
      return true;
    };
    // Software-pipelined per group: dS(i), then P(i+1), which overlaps dK(i) and dQ(i) on the
    // tensor pipe. P(i+1) overwrites p[] only after dS(i) has consumed it.
    bool good = n_it == 0 || do_p(0);
    for (int i = 0; good && i < n_it; ++i) {
      good = do_ds(i);
      if (good && i + 1 < n_it) good = do_p(i + 1);
    }
    if (good && n_it > 0) {
      good = __all_sync(0xffffffffu, wait(done, 0));
      if (good) tc_fence_after();
    }
    if (good && split > 1) {
      // this CTA's fp32 share of dV (group 0) or dK (group 1) for its key rows; the reduce
      // kernel adds the shares of the key tile's CTAs in a fixed order
      const uint32_t tAcc = w == 0 ? tDV : tDK;
      float* part = a.dkv_part +
                    (((static_cast<int64_t>(sp) * nb + b) * a.kc + kvl) * a.part_rows +
                     (r0 - a.kv_row_lo) + t) * (2 * kD) + (w == 0 ? kD : 0);
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t r[32];
        if (n_it > 0) {
          tmem_ld32_sync(tAcc + lane_off + c * 32, r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(part + c * 32 + i) =
              make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                          __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
      }
    } else if (good) {
      // group 0 writes dV, group 1 writes dK (both already carry their final scaling)
      const uint32_t tAcc = w == 0 ? tDV : tDK;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(w == 0 ? a.dv : a.dk) +
                           ((static_cast<int64_t>(b) * a.dkv_rows + pj - a.dkv_row0) * a.dkv_heads +
                            a.dkv_head0 + kvl) * kD;
      const bool store = key_ok && pj < a.S;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t r[32];
        if (n_it > 0) {
          tmem_ld32_sync(tAcc + lane_off + c * 32, r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (store) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(out + c * 32 + i * 8) = make_uint4(
                pack_bf16(__uint_as_float(r[8 * i + 0]), __uint_as_float(r[8 * i + 1])),
                pack_bf16(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                pack_bf16(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                pack_bf16(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int bwd_q_box_rows(int D) {
  (void)D;
  return 128;
}

cudaError_t launch_attn_bwd(int D, int B, const CUtensorMap& q_map, const CUtensorMap& do_map,
                            const CUtensorMap& k_map, const CUtensorMap& v_map,
                            const BwdArgs& a, cudaStream_t stream) {
  if (D != kD) return launch_attn_bwd_generic(D, B, q_map, do_map, k_map, v_map, a, stream);
  {
    const cudaError_t e =
        ensure_smem_attr(reinterpret_cast<const void*>(&attn_bwd_pp_kernel), BppLayout::kBytes);
    if (e != cudaSuccess) return e;
  }
  const int64_t n_kt = (a.kv_row_hi - a.kv_row_lo + 127) / 128;
  const int split = a.split > 1 ? a.split : 1;
  if (a.G % split || (split > 1 && (!a.dkv_part || a.part_rows < n_kt * 128)))
    return cudaErrorInvalidValue;
  const int64_t n_cta = n_kt * a.kc * split * B;
  if (n_cta <= 0) return cudaSuccess;
  if (n_cta > 0x7fffffff) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(n_cta));
  BwdArgs args = a;
  args.band = launch_band(n_kt, a.kc * split * B);
  launch_begin(3, stream);
  attn_bwd_pp_kernel<<<grid, kThreads, BppLayout::kBytes, stream>>>(q_map, do_map, k_map, v_map,
                                                                     args);
  cudaError_t e = cudaGetLastError();
  launch_end(3, stream);
  return e;
}

}  // namespace upipe
