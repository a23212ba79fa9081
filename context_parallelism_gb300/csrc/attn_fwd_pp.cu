// Forward causal (GQA) attention for D = 128 on sm_103a: two 128-row query tiles per CTA with
// two softmax warpgroups ping-ponging, so one tile's softmax overlaps the other tile's MMAs.
//
// Method: exact attention computed block by block with running maximum / sum statistics (the
// partial-output-plus-statistics fold of "Training Ultra Long Context LM with Fully Pipelined
// Distributed Transformer", Technical Deep Dive), across 128-row key tiles inside one launch and
// across key/value trunks between launches (state in/out exactly as the single-tile kernel).
//
// Per key tile j, for query tile w in {0, 1}:
//   S_w = Q_w K_j^T            tcgen05 (M 128, N 128, K 128) -> TMEM S[w]
//   P_w = exp2(S_w*scale*log2e - m_w), masked; bf16, written back over S[w]'s first 64 columns
//         (from the scores held in registers: one TMEM read of S per tile)
//   O_w += P_w V_j             tcgen05 with A read from TMEM
// MMA issue order: S0_0, S1_0, then per j: PV0_j, S0_{j+1}, PV1_j, S1_{j+1}. The tcgen05 pipe
// executes one thread's MMAs in order, so S0_{j+1} overwrites S[0] only after PV0_j has read
// P0_j from it, and the commit that publishes S_w(j+1) also covers PV_w(j): when a softmax group
// sees its next S, its O accumulator is settled and may be rescaled in place.
//
// Threads (320): warps 0-3 softmax for tile 0, warps 4-7 for tile 1 (thread = query row = TMEM
// lane), warp 8 TMEM + MMA issue, warp 9 TMA producer. A softmax thread reads its row's 128
// scores from TMEM once and keeps them in registers (168 per thread: ten warps share an SM's
// four 16K-register partitions three, three, two and two). Shared memory: Q0, Q1, two K and two
// V stages. TMEM: S[0] 0, S[1] 128, O[0] 256, O[1] 384.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 320;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kTile = 128 * kD * 2;  // 32 KiB

struct FppLayout {
  static constexpr int kQ = 0;                  // 2 query tiles
  static constexpr int kK = kQ + 2 * kTile;     // 2 stages
  static constexpr int kV = kK + 2 * kTile;     // 2 stages
  static constexpr int kBar = kV + 2 * kTile;
  static constexpr int kNumBars = 1 + 6 + 6 + 1;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 4;
  static constexpr int kBytes = kAbort + 4 + 1024;
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_pp_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = FppLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bar;
  uint64_t* k_full = bar + 1;     // [2] stages
  uint64_t* v_full = bar + 3;     // [2]
  uint64_t* kv_empty = bar + 5;   // [2]
  uint64_t* s_full = bar + 7;     // [2] query tiles
  uint64_t* p_full = bar + 9;     // [2]
  uint64_t* o_done = bar + 11;    // [2]
  uint64_t* drain = bar + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // One-dimensional grid over (query-tile pair, lane), lane = (batch, head) and the heaviest
  // causal pairs (largest query index) first, in bands of a.band lanes: inside a band the
  // lanes' pairs interleave, the band's heaviest first; bands follow one another.
  const int n_pairs = static_cast<int>((a.q_hi - a.q_lo + 255) / 256);
  const int nh = static_cast<int>(gridDim.x) / n_pairs;  // hc * B
  int pr, hb;
  {
    const int L = static_cast<int>(blockIdx.x);
    const int band = L / (a.band * n_pairs);
    const int lane0 = band * a.band;
    const int bl = min(a.band, nh - lane0);  // lanes of this band
    const int u = L - lane0 * n_pairs;
    pr = n_pairs - 1 - u / bl;
    hb = lane0 + (u - (n_pairs - 1 - pr) * bl);
  }
  const int64_t q0 = a.q_lo + static_cast<int64_t>(pr) * 256;
  const int hl = hb % a.hc;
  const int b = hb / a.hc;
  const int zq = b * a.hc + hl;
  const int zk = b * a.kc + hl / a.G;
  int64_t kv_end = a.kv_row_hi;
  if (a.causal) kv_end = min(kv_end, q0 + 256 - a.kv_pos0);
  const int n_kv = kv_end > a.kv_row_lo ? static_cast<int>((kv_end - a.kv_row_lo + 127) / 128) : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(v_full + i, 1);
      mbar_init(kv_empty + i, 1);
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 4);
      mbar_init(o_done + i, 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

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
          atomicOr(a.err, kErrWaitTimeout | 0x8000u);
          return false;
        }
      }
    }
  };

  if (warp >= 8) {
  if (warp == 9) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, 2 * kTile);
      for (int w = 0; w < 2; ++w)
        for (int x = 0; x < 2; ++x)
          tma_load_3d(smem + L::kQ + w * kTile + x * kBoxBytes, &tm_q, x * 64,
                      static_cast<int>(q0 + 128 * w), zq, q_full);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        if (j >= 2 && !wait(kv_empty + s, ((j - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        const int row = static_cast<int>(a.kv_row_lo + static_cast<int64_t>(j) * 128);
        mbar_arrive_expect_tx(k_full + s, kTile);
        for (int x = 0; x < 2; ++x)
          tma_load_3d(smem + L::kK + s * kTile + x * kBoxBytes, &tm_k, x * 64, row, zk, k_full + s);
        mbar_arrive_expect_tx(v_full + s, kTile);
        for (int x = 0; x < 2; ++x)
          tma_load_3d(smem + L::kV + s * kTile + x * kBoxBytes, &tm_v, x * 64, row, zk, v_full + s);
        issued = j + 1;
      }
      if (!ok) {
        mbar_wait(q_full, 0, 100000000ull);
        for (int j = (issued >= 2 ? issued - 2 : 0); j < issued; ++j) {
          mbar_wait(k_full + (j & 1), (j >> 1) & 1, 100000000ull);
          mbar_wait(v_full + (j & 1), (j >> 1) & 1, 100000000ull);
        }
      }
    }
  } else if (warp == 8) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false, false);
      const uint32_t id_o = idesc_bf16(128, kD, false, true);
      // One base descriptor per operand form; stages and steps are compile-time offsets (in
      // 16-byte units), the base made opaque at each use so that no per-step descriptor is
      // held in a register across the loop.
      const uint64_t base_k = kdesc0(smem_u32(smem));
      const uint64_t base_mn = mndesc0(smem_u32(smem));
      constexpr uint32_t kTileU = kTile >> 4;
      constexpr uint32_t uQ = L::kQ >> 4, uK = L::kK >> 4, uV = L::kV >> 4;
      bool ok = wait(q_full, 0);
      auto issue_s = [&](int w, int j) -> bool {
        if (w == 0 && !wait(k_full + (j & 1), (j >> 1) & 1)) return false;
        tc_fence_after();
        const uint64_t bk = opaque_u64(base_k);
        const uint32_t uq = uQ + w * kTileU, uk = uK + (j & 1) * kTileU;
        const uint32_t tS = tmem + 128 * w;
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16)
          umma_f16_ss(tS, bk + (uq + kstep(k16)), bk + (uk + kstep(k16)), id_s,
                      k16 > 0 ? 1u : 0u);
        umma_commit(s_full + w);
        return true;
      };
      auto issue_pv = [&](int w, int j) -> bool {
        if (!wait(p_full + w, j & 1)) return false;
        if (w == 0 && !wait(v_full + (j & 1), (j >> 1) & 1)) return false;
        tc_fence_after();
        const uint64_t bmn = opaque_u64(base_mn);
        const uint32_t uv = uV + (j & 1) * kTileU;
        const uint32_t acc0 = (j > 0 || !a.first) ? 1u : 0u;
        const uint32_t tP = tmem + 128 * w, tO = tmem + 256 + 128 * w;
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ts(tO, tP + k16 * 8, bmn + (uv + mnstep(k16)), id_o, k16 > 0 ? 1u : acc0);
        if (j == n_kv - 1) umma_commit(o_done + w);
        return true;
      };
      if (ok && n_kv > 0) ok = issue_s(0, 0) && issue_s(1, 0);
      for (int j = 0; ok && j < n_kv; ++j) {
        ok = issue_pv(0, j);
        if (ok && j + 1 < n_kv) ok = issue_s(0, j + 1);
        if (ok) ok = issue_pv(1, j);
        if (ok) umma_commit(kv_empty + (j & 1));
        if (ok && j + 1 < n_kv) ok = issue_s(1, j + 1);
      }
      if (!ok) {
        umma_commit(drain);
        mbar_wait(drain, 0, 100000000ull);
      }
    }
  }
  } else {
    // ---------------- softmax groups ----------------
    const int w = warp >> 2;
    const int t = threadIdx.x & 127;  // query row within tile w
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 128 * w, tO = tmem + 256 + 128 * w;
    const int64_t qw0 = q0 + 128 * w;
    const int64_t qrow = qw0 + t;
    const int64_t srow = (qw0 - a.q_lo) + t;  // row inside the carried state
    const int64_t sstride = a.state_stride ? a.state_stride : a.state_rows;
    float m_used = -INFINITY;  // log2 units
    float l_sum = 0.f;
    // Rows past the carried state (the second tile of a trunk with an odd tile count) belong
    // to no output; they compute on whatever TMEM holds and are never stored.
    if (!a.first && srow < a.state_rows) {
      const float* so = a.state_o + (static_cast<int64_t>(zq) * sstride + srow) * kD;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 f = *reinterpret_cast<const float4*>(so + c * 32 + i);
          r[i] = __float_as_uint(f.x);
          r[i + 1] = __float_as_uint(f.y);
          r[i + 2] = __float_as_uint(f.z);
          r[i + 3] = __float_as_uint(f.w);
        }
        tmem_st32(tO + lane_off + c * 32, r);
      }
      tmem_wait_st();
      const float2 ml = *reinterpret_cast<const float2*>(
          a.state_ml + (static_cast<int64_t>(zq) * sstride + srow) * 2);
      m_used = ml.x;
      l_sum = ml.y;
    }
    bool good = true;
    for (int j = 0; j < n_kv; ++j) {
      good = __all_sync(0xffffffffu, wait(s_full + w, j & 1));
      if (!good) break;
      tc_fence_after();
      const int64_t r0 = a.kv_row_lo + static_cast<int64_t>(j) * 128;
      const int64_t p0 = a.kv_pos0 + r0;
      const bool need_mask = (r0 + 128 > a.kv_row_hi) || (a.causal && p0 + 127 > qw0);
      int64_t lim = 128;
      if (need_mask) {
        lim = a.kv_row_hi - r0;
        if (a.causal) lim = min(lim, qrow - p0 + 1);
      }
      // The row's 128 scores are read from TMEM once, both 64-column halves in flight together,
      // and stay in registers: the maximum, the exponentials and the bf16 packing all work on
      // them (P packed in place into the low half of each array). Only tiles that straddle the
      // diagonal or an end pay for the mask. Four independent running maxima keep the dependent
      // chain short.
      uint32_t ra[64], rb[64];
      tmem_ld64_nowait(tS + lane_off, ra);
      tmem_ld64_nowait(tS + lane_off + 64, rb);
      tmem_wait_ld_dep64(ra);
      tmem_reg_dep64(rb);
      if (need_mask) {
        const int lim32 = static_cast<int>(lim < 0 ? 0 : lim);  // visible columns, <= 128
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          if (i >= lim32) ra[i] = __float_as_uint(-INFINITY);
          if (64 + i >= lim32) rb[i] = __float_as_uint(-INFINITY);
        }
      }
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        mq[(i >> 1) & 3] = fmax3(mq[(i >> 1) & 3], __uint_as_float(ra[i]), __uint_as_float(ra[i + 1]));
        mq[((i >> 1) + 2) & 3] =
            fmax3(mq[((i >> 1) + 2) & 3], __uint_as_float(rb[i]), __uint_as_float(rb[i + 1]));
      }
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      const float m_new = fmaxf(m_used, mx * a.scale_log2);
      float alpha = 1.f;
      const bool upd = m_new > m_used + kRescaleLog2;
      if (upd) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      l_sum *= alpha;
      const float mb = (m_used == -INFINITY) ? 0.f : m_used;
      // P rounded to bf16 once, written over S's first 64 columns (P of key columns c..c+63
      // goes to TMEM columns c/2..c/2+31; every score is already in registers). The row sum adds
      // the same bf16 weights the P.V MMA multiplies, in four independent chains, so that O's
      // numerator and denominator agree: a row dominated by one key then gives that key's V
      // up to the output's own rounding, whatever the weight's rounding.
      const uint64_t sl2 = f2_pack(a.scale_log2, a.scale_log2);
      const uint64_t nm2 = f2_pack(-mb, -mb);
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float x0, x1;
        f2_unpack(ffma2(f2_pack_u(ra[2 * i], ra[2 * i + 1]), sl2, nm2), x0, x1);
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
        ra[i] = pack_bf16(e0, e1);  // reads 2i, 2i+1 >= i first
        add_bf16x2(s0, s1, ra[i]);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float x0, x1;
        f2_unpack(ffma2(f2_pack_u(rb[2 * i], rb[2 * i + 1]), sl2, nm2), x0, x1);
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
        rb[i] = pack_bf16(e0, e1);
        add_bf16x2(s2, s3, rb[i]);
      }
      {
        uint32_t pa[32], pb[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          pa[i] = ra[i];
          pb[i] = rb[i];
        }
        tmem_st32(tS + lane_off, pa);
        tmem_st32(tS + lane_off + 32, pb);
      }
      // O_w is settled (the commit that published S_w(j) covers PV_w(j-1)): rescale it in place
      // now that the scores are consumed (their registers free), before P_w(j) is published.
      const bool o_has = (j >= 1) || !a.first;
      if (o_has && __any_sync(0xffffffffu, upd)) {
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(tO + lane_off + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tO + lane_off + c * 32, r);
        }
      }
      l_sum += (s0 + s1) + (s2 + s3);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + w);
    }
    if (good && n_kv > 0) {
      good = __all_sync(0xffffffffu, wait(o_done + w, 0));
      if (good) tc_fence_after();
    }
    if (good) {
      const bool row_ok = qrow < a.q_hi;
      // a launch that walks one key/value trunk for several query trunks finalises only the
      // tiles of the trunk it is the last for
      const bool last = a.last && (a.last_q_end == 0 || qw0 < a.last_q_end);
      if (last) {
        const float inv_l = 1.f / l_sum;
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) +
                              ((static_cast<int64_t>(b) * a.S + qrow) * (a.o_heads ? a.o_heads : a.Hq) +
                               (a.o_heads ? a.o_head0 : a.h0) + hl) * kD;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(tO + lane_off + c * 32, r);
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(orow + c * 32 + i * 8) = make_uint4(
                  pack_bf16(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l),
                  pack_bf16(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l),
                  pack_bf16(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l),
                  pack_bf16(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l));
          }
        }
        if (row_ok && a.lse)  // no LSE in prefill (inference) calls
          a.lse[(static_cast<int64_t>(b) * a.Hq + a.h0 + hl) * a.S + qrow] =
              (m_used + __log2f(l_sum)) * 0.69314718055994530942f;
      } else if (srow < a.state_rows) {
        float* so = a.state_o + (static_cast<int64_t>(zq) * sstride + srow) * kD;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(tO + lane_off + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(so + c * 32 + i) =
                make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                            __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
        }
        *reinterpret_cast<float2*>(a.state_ml + (static_cast<int64_t>(zq) * sstride + srow) * 2) =
            make_float2(m_used, l_sum);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attn_fwd(int D, int B, const CUtensorMap& q_map, const CUtensorMap& k_map,
                            const CUtensorMap& v_map, const FwdArgs& a, cudaStream_t stream) {
  if (D != kD) return launch_attn_fwd_generic(D, B, q_map, k_map, v_map, a, stream);
  {
    const cudaError_t e =
        ensure_smem_attr(reinterpret_cast<const void*>(&attn_fwd_pp_kernel), FppLayout::kBytes);
    if (e != cudaSuccess) return e;
  }
  const int64_t n_pairs = (a.q_hi - a.q_lo + 255) / 256;
  const int64_t n_cta = n_pairs * a.hc * B;
  if (n_cta <= 0) return cudaSuccess;
  if (n_cta > 0x7fffffff) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(n_cta));
  FwdArgs args = a;
  args.band = launch_band(n_pairs, a.hc * B);
  launch_begin(1, stream);
  attn_fwd_pp_kernel<<<grid, kThreads, FppLayout::kBytes, stream>>>(q_map, k_map, v_map, args);
  cudaError_t e = cudaGetLastError();
  launch_end(1, stream);
  return e;
}

}  // namespace upipe
