// Forward causal (GQA) attention on sm_103a, one 128-row query tile per CTA (used for D = 64;
// D = 128 runs the two-tile ping-pong kernel in attn_fwd_pp.cu): TMA-staged Q/K/V tiles, tcgen05 MMAs with TMEM
// accumulators for S = Q K^T and O += P V, online softmax in registers (one query row per
// thread), causal tile skipping, and optional carried state so that a query trunk can fold
// key/value trunks in over several launches.
//
// Method: exact attention computed block by block with running maximum / sum statistics, the
// way the FPDT talk's Technical Deep Dive describes folding trunks into "partial attention
// output plus statistics (like maximum logits)" ("Training Ultra Long Context LM with Fully
// Pipelined Distributed Transformer", Technical Deep Dive), applied both across 128-row key
// tiles inside one launch and across key/value trunks between launches.
//
// CTA layout (192 threads, one CTA per SM):
//   warps 0-3  softmax: thread t owns query row t of the tile (TMEM lane t)
//   warp 4     TMEM allocation + MMA issue (lane 0)
//   warp 5     TMA producer (lane 0)
// Shared memory: Q tile, two K and two V stages, one P tile (all 128-byte swizzled bf16).
// TMEM columns: S buffer 0 at 0, S buffer 1 at 128, O accumulator at 256 (D columns).
//
// Softmax statistics are kept in log2 units of the scaled score. The running maximum is only
// moved when the new row maximum exceeds it by more than kRescaleLog2 (exact: numerator and
// denominator always share the same reference), which skips most O rescaling passes.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {
namespace {

constexpr int kThreads = 192;
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct FwdLayout {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;        // 2 stages
  static constexpr int kV = kK + 2 * kTile;    // 2 stages
  static constexpr int kP = kV + 2 * kTile;    // 128 x 128 bf16
  static constexpr int kBar = kP + 128 * 128 * 2;
  static constexpr int kNumBars = 14;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 4;
  static constexpr int kBytes = kAbort + 4 + 1024;  // + slack for 1024-byte alignment
};

struct Bars {
  uint64_t* q_full;
  uint64_t* k_full;    // [2]
  uint64_t* v_full;    // [2]
  uint64_t* kv_empty;  // [2]
  uint64_t* s_full;    // [2]
  uint64_t* s_free;    // [2]
  uint64_t* p_full;
  uint64_t* o_done;
  uint64_t* drain;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  const Bars B{bar + 0, bar + 1, bar + 3, bar + 5, bar + 7, bar + 9, bar + 11, bar + 12, bar + 13};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heaviest causal tiles (largest query index) are scheduled first.
  const int qt = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);
  const int64_t q0 = a.q_lo + static_cast<int64_t>(qt) * 128;
  const int hl = blockIdx.y;
  const int b = blockIdx.z;
  const int zq = b * a.hc + hl;
  const int zk = b * a.kc + hl / a.G;
  int64_t kv_end = a.kv_row_hi;
  if (a.causal) kv_end = min(kv_end, q0 + 128 - a.kv_pos0);
  const int n_kv = kv_end > a.kv_row_lo ? static_cast<int>((kv_end - a.kv_row_lo + 127) / 128) : 0;

  if (threadIdx.x == 0) {
    mbar_init(B.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(B.k_full + i, 1);
      mbar_init(B.v_full + i, 1);
      mbar_init(B.kv_empty + i, 1);
      mbar_init(B.s_full + i, 1);
      mbar_init(B.s_free + i, 128);
    }
    mbar_init(B.p_full, 128);
    mbar_init(B.o_done, 1);
    mbar_init(B.drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 256;

  // Bounded wait shared by all roles: gives up when the limit passes or another role gave up.
  auto wait = [&](uint64_t* br, uint32_t parity) -> bool {
    if (mbar_try_wait(br, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (mbar_try_wait(br, parity)) return true;
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(a.err, kErrWaitTimeout | 0x1000u);
        return false;
      }
    }
  };

  if (warp == 5) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint8_t* sQ = smem + L::kQ;
      mbar_arrive_expect_tx(B.q_full, L::kTile);
      for (int x = 0; x < D / 64; ++x)
        tma_load_3d(sQ + x * kBoxBytes, &tm_q, x * 64, static_cast<int>(q0), zq, B.q_full);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        if (j >= 2 && !wait(B.kv_empty + s, ((j - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        const int row = static_cast<int>(a.kv_row_lo + static_cast<int64_t>(j) * 128);
        uint8_t* sK = smem + L::kK + s * L::kTile;
        uint8_t* sV = smem + L::kV + s * L::kTile;
        mbar_arrive_expect_tx(B.k_full + s, L::kTile);
        for (int x = 0; x < D / 64; ++x)
          tma_load_3d(sK + x * kBoxBytes, &tm_k, x * 64, row, zk, B.k_full + s);
        mbar_arrive_expect_tx(B.v_full + s, L::kTile);
        for (int x = 0; x < D / 64; ++x)
          tma_load_3d(sV + x * kBoxBytes, &tm_v, x * 64, row, zk, B.v_full + s);
        issued = j + 1;
      }
      if (!ok) {
        // Let every load already issued land before the CTA can exit.
        mbar_wait(B.q_full, 0, 100000000ull);
        for (int j = (issued >= 2 ? issued - 2 : 0); j < issued; ++j) {
          mbar_wait(B.k_full + (j & 1), (j >> 1) & 1, 100000000ull);
          mbar_wait(B.v_full + (j & 1), (j >> 1) & 1, 100000000ull);
        }
      }
    }
  } else if (warp == 4) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false, false);
      const uint32_t id_o = idesc_bf16(128, D, false, true);
      const uint32_t sQ = smem_u32(smem + L::kQ);
      const uint32_t sP = smem_u32(smem + L::kP);
      bool ok = wait(B.q_full, 0);
      auto issue_pv = [&](int i) -> bool {
        if (!wait(B.p_full, i & 1)) return false;
        if (!wait(B.v_full + (i & 1), (i >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + L::kV + (i & 1) * L::kTile);
        const uint32_t acc0 = (i > 0 || !a.first) ? 1u : 0u;
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tO, desc_kmajor(sP, k16), desc_mnmajor(sV, k16), id_o,
                      k16 > 0 ? 1u : acc0);
        umma_commit(B.o_done);
        umma_commit(B.kv_empty + (i & 1));
        return true;
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j & 1;
        if (!wait(B.k_full + s, (j >> 1) & 1)) { ok = false; break; }
        if (j >= 2 && !wait(B.s_free + s, ((j - 2) >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + L::kK + s * L::kTile);
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          umma_f16_ss(tmem + s * 128, desc_kmajor(sQ, k16), desc_kmajor(sK, k16), id_s,
                      k16 > 0 ? 1u : 0u);
        umma_commit(B.s_full + s);
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok && n_kv > 0) ok = issue_pv(n_kv - 1);
      if (!ok) {
        umma_commit(B.drain);
        mbar_wait(B.drain, 0, 100000000ull);
      }
    }
  } else {
    // ---------------- softmax warps ----------------
    const int t = threadIdx.x;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int64_t qrow = q0 + t;
    const int64_t srow = (q0 - a.q_lo) + t;  // row inside the carried state
    const int64_t sstride = a.state_stride ? a.state_stride : a.state_rows;
    float m_used = -INFINITY;  // log2 units
    float l_sum = 0.f;
    if (!a.first) {
      const float* so = a.state_o + (static_cast<int64_t>(zq) * sstride + srow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
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
      const float2 ml =
          *reinterpret_cast<const float2*>(a.state_ml + (static_cast<int64_t>(zq) * sstride + srow) * 2);
      m_used = ml.x;
      l_sum = ml.y;
    }
    const uint32_t sP = smem_u32(smem + L::kP);
    bool good = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      good = __all_sync(0xffffffffu, wait(B.s_full + sb, (j >> 1) & 1));
      if (!good) break;
      tc_fence_after();
      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32_sync(tmem + sb * 128 + lane_off + c * 32, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      mbar_arrive(B.s_free + sb);

      const int64_t r0 = a.kv_row_lo + static_cast<int64_t>(j) * 128;
      const int64_t p0 = a.kv_pos0 + r0;
      const bool need_mask = (r0 + 128 > a.kv_row_hi) || (a.causal && p0 + 127 > q0);
      if (need_mask) {
        int64_t lim = a.kv_row_hi - r0;
        if (a.causal) lim = min(lim, qrow - p0 + 1);
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) sv[c] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) mx = fmaxf(mx, sv[c]);
      const float m_new = fmaxf(m_used, mx * a.scale_log2);
      float alpha = 1.f;
      const bool upd = m_new > m_used + kRescaleLog2;
      if (upd) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      l_sum *= alpha;
      const float mb = (m_used == -INFINITY) ? 0.f : m_used;
      // P is rounded to bf16 here, once; the row sum adds exactly the rounded weights the
      // P.V MMA consumes, so O stays a convex combination of V rows (a dominant weight's
      // rounding cancels) and LSE moves by at most one bf16 rounding (2^-9 relative).
      uint32_t pk[64];
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const uint32_t w = pack_bf16(ex2_approx(fmaf(sv[c], a.scale_log2, -mb)),
                                     ex2_approx(fmaf(sv[c + 1], a.scale_log2, -mb)));
        pk[c >> 1] = w;
        sum += __uint_as_float(w << 16) + __uint_as_float(w & 0xFFFF0000u);
      }
      l_sum += sum;

      // P_{j-1} must have been consumed (and O updated) before P_j and any rescale land.
      if (j >= 1) {
        good = __all_sync(0xffffffffu, wait(B.o_done, (j - 1) & 1));
        if (!good) break;
        tc_fence_after();
      }
      const bool o_has = (j >= 1) || !a.first;
      if (o_has && __any_sync(0xffffffffu, upd)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(tO + lane_off + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tO + lane_off + c * 32, r);
        }
        tmem_wait_st();
      }
#pragma unroll
      for (int cc = 0; cc < 16; ++cc)
        st_shared_v4(sP + swz_offset(t, cc * 8), pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2],
                     pk[4 * cc + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(B.p_full);
    }
    if (good && n_kv > 0) {
      good = __all_sync(0xffffffffu, wait(B.o_done, (n_kv - 1) & 1));
      if (good) tc_fence_after();
    }
    if (good) {
      const bool row_ok = qrow < a.q_hi;
      const bool last = a.last && (a.last_q_end == 0 || q0 < a.last_q_end);
      if (last) {
        const float inv_l = 1.f / l_sum;
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) +
                              ((static_cast<int64_t>(b) * a.S + qrow) * (a.o_heads ? a.o_heads : a.Hq) +
                               (a.o_heads ? a.o_head0 : a.h0) + hl) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(tO + lane_off + c * 32, r);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(orow + c * 32 + i * 8) =
                  make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
        if (row_ok && a.lse)  // no LSE in prefill (inference) calls
          a.lse[(static_cast<int64_t>(b) * a.Hq + a.h0 + hl) * a.S + qrow] =
              (m_used + __log2f(l_sum)) * 0.69314718055994530942f;
      } else {
        float* so = a.state_o + (static_cast<int64_t>(zq) * sstride + srow) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
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
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_impl(int B, const CUtensorMap& q_map, const CUtensorMap& k_map,
                        const CUtensorMap& v_map, const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  {
    const cudaError_t e =
        ensure_smem_attr(reinterpret_cast<const void*>(&attn_fwd_kernel<D>), L::kBytes);
    if (e != cudaSuccess) return e;
  }
  const int64_t n_qt = (a.q_hi - a.q_lo + 127) / 128;
  dim3 grid(static_cast<unsigned>(n_qt), static_cast<unsigned>(a.hc), static_cast<unsigned>(B));
  launch_begin(1, stream);
  attn_fwd_kernel<D><<<grid, kThreads, L::kBytes, stream>>>(q_map, k_map, v_map, a);
  cudaError_t e = cudaGetLastError();
  launch_end(1, stream);
  return e;
}

}  // namespace

cudaError_t launch_attn_fwd_generic(int D, int B, const CUtensorMap& q_map,
                                    const CUtensorMap& k_map, const CUtensorMap& v_map,
                                    const FwdArgs& a, cudaStream_t stream) {
  if (D == 128) return launch_impl<128>(B, q_map, k_map, v_map, a, stream);
  if (D == 64) return launch_impl<64>(B, q_map, k_map, v_map, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace upipe
