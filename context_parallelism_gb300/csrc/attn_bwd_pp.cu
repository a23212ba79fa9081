// Backward causal (GQA) attention for D = 128 on sm_103a: two compute warpgroups ping-pong
// over 64-row query subtiles while one thread keeps the tensor core fed.
//
// One CTA owns a 128-row key/value tile of one kv-head (K and V stay in shared memory) and walks
// the 64-row query subtiles of every q-head of its group that can see the tile; the probabilities
// are recomputed from the saved log-sum-exp, never stored ("Training Ultra Long Context LM with
// Fully Pipelined Distributed Transformer", Background: the attention backward pass is the memory
// peak; "Road to 5 million sequence length" talk, UPipe passage: each head group is recomputed).
//
// Per subtile it (kv row j = TMEM lane of the S^T / dP^T accumulators, query row i):
//   S^T  = K Q^T                 tcgen05 (M 128, N 64, K 128) -> TMEM S[w]
//   dP^T = V dO^T                tcgen05 -> TMEM dP[w]
//   P^T  = exp2(S^T*scale*log2e - LSE_i*log2e), masked; bf16 back into TMEM S[w]
//   dS^T = P^T * (scale*dP^T - scale*D_i)                  bf16 -> shared memory (one box)
//   dV  += P^T dO                tcgen05 with A read from TMEM (M 128, N 128, K 64)
//   dK  += dS^T Q                tcgen05 (A K-major, B MN-major)
//   dQ^T = K^T dS^T              tcgen05 (M 128 = head dim, N 64) -> TMEM dP[w]
//   dQ  += dQ^T read back with lanes = head dim, so each warp adds one contiguous 128-byte
//          line per query row with fire-and-forget fp32 reductions
// Warpgroup w = it % 2 handles subtile it, so one warpgroup's exp/pack/reduction work overlaps
// the other's MMAs; Q/dO/LSE/D stream through three shared-memory stages (stage = it % 3).
//
// Threads (320): warps 0-3 compute group 0, warps 4-7 compute group 1, warp 8 TMEM + MMA issue,
// warp 9 TMA producer. TMEM (512 columns): dV [0,128), dK [128,256), S[w] at 256+128w (64),
// dP[w] at 320+128w (64).
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {
namespace {

constexpr int kD = 128;
constexpr int kSub = 64;          // query rows per subtile
constexpr int kStages = 3;
constexpr int kThreads = 320;
constexpr uint32_t kQBox = kSub * 128;  // one 64-row x 64-column bf16 box (8 KiB)

struct PPLayout {
  static constexpr int kK = 0;                              // 2 boxes of 128 x 64
  static constexpr int kV = kK + 2 * kBoxBytes;
  static constexpr int kQ = kV + 2 * kBoxBytes;             // kStages x (2 boxes of 64 x 64)
  static constexpr int kDO = kQ + kStages * 2 * kQBox;
  static constexpr int kDS = kDO + kStages * 2 * kQBox;     // 2 groups x (one 128 x 64 box)
  static constexpr int kVec = kDS + 2 * kBoxBytes;          // kStages x (64 LSE2 + 64 D) fp32
  static constexpr int kBar = kVec + kStages * 512;
  static constexpr int kNumBars = 1 + 2 * kStages + 6 * 2 + 2;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 4;
  static constexpr int kBytes = kAbort + 4 + 1024;
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_pp_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const BwdArgs a) {
  using L = PPLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bar;
  uint64_t* q_full = bar + 1;                  // [kStages]
  uint64_t* q_empty = bar + 1 + kStages;       // [kStages]
  uint64_t* s_full = bar + 1 + 2 * kStages;    // [2] per compute group
  uint64_t* dp_full = s_full + 2;
  uint64_t* ds_full = s_full + 4;
  uint64_t* dq_full = s_full + 6;
  uint64_t* dq_free = s_full + 8;
  uint64_t* pt_done = s_full + 10;
  uint64_t* done = s_full + 12;
  uint64_t* drain = s_full + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kt = blockIdx.x;  // smallest key positions (most query subtiles) first
  const int kvl = blockIdx.y;
  const int b = blockIdx.z;
  const int64_t r0 = a.kv_row_lo + static_cast<int64_t>(kt) * 128;  // K/V map row
  const int64_t p0 = a.kv_pos0 + r0;                                // global key position
  const int zk = b * a.kc + kvl;
  const int qs_lo = a.causal ? static_cast<int>(p0 / kSub) : 0;
  const int qs_hi = static_cast<int>((a.S + kSub - 1) / kSub);
  const int nq = qs_hi > qs_lo ? qs_hi - qs_lo : 0;
  const int n_it = a.G * nq;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(q_full + s, 1);
      mbar_init(q_empty + s, 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(s_full + w, 1);
      mbar_init(dp_full + w, 1);
      mbar_init(ds_full + w, 4);
      mbar_init(dq_full + w, 1);
      mbar_init(dq_free + w, 4);
      mbar_init(pt_done + w, 1);
    }
    mbar_init(done, 1);
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
  const uint32_t tDV = tmem, tDK = tmem + 128;

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
  auto decode = [&](int it, int& zq, int64_t& q0) {
    const int hl = kvl * a.G + it / nq;
    zq = b * a.hc + hl;
    q0 = static_cast<int64_t>(qs_lo + it % nq) * kSub;
  };

  if (warp == 9) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(kv_full, 4 * kBoxBytes);
      for (int x = 0; x < 2; ++x) {
        tma_load_3d(smem + L::kK + x * kBoxBytes, &tm_k, x * 64, static_cast<int>(r0), zk, kv_full);
        tma_load_3d(smem + L::kV + x * kBoxBytes, &tm_v, x * 64, static_cast<int>(r0), zk, kv_full);
      }
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        const int st = it % kStages;
        if (it >= kStages && !wait(q_empty + st, ((it / kStages) - 1) & 1)) {
          ok = false;
          break;
        }
        int zq;
        int64_t q0;
        decode(it, zq, q0);
        mbar_arrive_expect_tx(q_full + st, 4 * kQBox + 512);
        for (int x = 0; x < 2; ++x) {
          tma_load_3d(smem + L::kQ + st * 2 * kQBox + x * kQBox, &tm_q, x * 64,
                      static_cast<int>(q0), zq, q_full + st);
          tma_load_3d(smem + L::kDO + st * 2 * kQBox + x * kQBox, &tm_do, x * 64,
                      static_cast<int>(q0), zq, q_full + st);
        }
        const int64_t vo = static_cast<int64_t>(zq) * a.S_pad + q0;
        uint8_t* vec = smem + L::kVec + st * 512;
        bulk_load(vec, a.lse2 + vo, 256, q_full + st);
        bulk_load(vec + 256, a.dvec + vo, 256, q_full + st);
        issued = it + 1;
      }
      mbar_wait(kv_full, 0, ok ? kWaitLimitNs : 100000000ull);
      if (!ok)
        for (int it = (issued > kStages ? issued - kStages : 0); it < issued; ++it)
          mbar_wait(q_full + it % kStages, (it / kStages) & 1, 100000000ull);
    }
  } else if (warp == 8) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_sdp = idesc_bf16(128, kSub, false, false);  // S^T, dP^T
      const uint32_t id_dvdk = idesc_bf16(128, kD, false, true);    // dV (A in TMEM), dK
      const uint32_t id_dq = idesc_bf16(128, kSub, true, true);     // dQ^T = K^T dS^T
      const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
      bool ok = wait(kv_full, 0);

      auto finish = [&](int i) -> bool {
        const int st = i % kStages, w = i & 1, j = i >> 1;
        if (!wait(ds_full + w, j & 1)) return false;
        tc_fence_after();
        const uint32_t sQ = smem_u32(smem + L::kQ + st * 2 * kQBox);
        const uint32_t sDO = smem_u32(smem + L::kDO + st * 2 * kQBox);
        const uint32_t sDS = smem_u32(smem + L::kDS + w * kBoxBytes);
        const uint32_t tS = tmem + 256 + 128 * w, tDP = tS + 64;
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int k16 = 0; k16 < kSub / 16; ++k16)
          umma_f16_ts(tDV, tS + k16 * 8, desc_mnmajor(sDO, k16, kQBox), id_dvdk,
                      k16 > 0 ? 1u : acc0);
        umma_commit(pt_done + w);
#pragma unroll
        for (int k16 = 0; k16 < kSub / 16; ++k16)
          umma_f16_ss(tDK, desc_kmajor(sDS, k16), desc_mnmajor(sQ, k16, kQBox), id_dvdk,
                      k16 > 0 ? 1u : acc0);
        umma_commit(q_empty + st);
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tDP, desc_mnmajor(sK, k16), desc_mnmajor(sDS, k16), id_dq,
                      k16 > 0 ? 1u : 0u);
        umma_commit(dq_full + w);
        return true;
      };

      // Issue order S(it), dV/dK/dQ(it-1), dP(it): five MMA blocks separate dQ(it-2) from
      // dP(it), which reuses its TMEM columns, so the read-out of dQ hides behind them; the
      // group's P(it) overlaps dV/dK/dQ(it-1) and its dS(it) overlaps S(it+1).
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it % kStages, w = it & 1, j = it >> 1;
        const uint32_t tS = tmem + 256 + 128 * w, tDP = tS + 64;
        if (!wait(q_full + st, (it / kStages) & 1)) { ok = false; break; }
        // S[w] last held P^T of subtile it-2, which dV(it-2) reads.
        if (j >= 1 && !wait(pt_done + w, (j - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sQ = smem_u32(smem + L::kQ + st * 2 * kQBox);
        const uint32_t sDO = smem_u32(smem + L::kDO + st * 2 * kQBox);
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16)
          umma_f16_ss(tS, desc_kmajor(sK, k16), desc_kmajor(sQ, k16, kQBox), id_sdp,
                      k16 > 0 ? 1u : 0u);
        umma_commit(s_full + w);
        if (it >= 1 && !finish(it - 1)) { ok = false; break; }
        // dP[w] last held dQ^T of subtile it-2 until the group read it out.
        if (j >= 1 && !wait(dq_free + w, (j - 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16)
          umma_f16_ss(tDP, desc_kmajor(sV, k16), desc_kmajor(sDO, k16, kQBox), id_sdp,
                      k16 > 0 ? 1u : 0u);
        umma_commit(dp_full + w);
      }
      if (ok && n_it > 0) ok = finish(n_it - 1);
      if (ok) {
        umma_commit(done);
      } else {
        umma_commit(drain);
        mbar_wait(drain, 0, 100000000ull);
      }
    }
  } else {
    // ---------------- compute groups ----------------
    const int w = warp >> 2;                  // compute group
    const int t = threadIdx.x & 127;          // key row (S^T/dP^T lanes) / head dim (dQ^T lanes)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 256 + 128 * w, tDP = tS + 64;
    const uint32_t sDS = smem_u32(smem + L::kDS + w * kBoxBytes);
    const int64_t pj = p0 + t;
    const bool key_ok = (r0 + t) < a.kv_row_hi;
    bool good = true;
    for (int it = w; it < n_it; it += 2) {
      const int st = it % kStages, j = it >> 1;
      int zq;
      int64_t q0;
      decode(it, zq, q0);
      const float* lse_s = reinterpret_cast<const float*>(smem + L::kVec + st * 512);
      const float* dv_s = lse_s + 64;
      // q_full: LSE/D of this subtile landed (the stage cannot be refilled before this group
      // signals ds_full for it).
      good = __all_sync(0xffffffffu, wait(q_full + st, (it / kStages) & 1) &&
                                         wait(s_full + w, j & 1));
      if (!good) break;
      tc_fence_after();
      const bool need_mask = (a.causal && q0 < p0 + 127) || (q0 + kSub > a.S) ||
                             (r0 + 128 > a.kv_row_hi);
      float p[64];
      {
        uint32_t r[64];
        tmem_ld64_sync(tS + lane_off, r);
        const uint64_t sl2 = f2_pack(a.scale_log2, a.scale_log2);
#pragma unroll
        for (int x = 0; x < 64; x += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(lse_s + x);
          float y0, y1, y2, y3;
          f2_unpack(ffma2(f2_pack_u(r[x], r[x + 1]), sl2, f2_pack(-l4.x, -l4.y)), y0, y1);
          f2_unpack(ffma2(f2_pack_u(r[x + 2], r[x + 3]), sl2, f2_pack(-l4.z, -l4.w)), y2, y3);
          p[x + 0] = ex2_approx(y0);
          p[x + 1] = ex2_approx(y1);
          p[x + 2] = ex2_approx(y2);
          p[x + 3] = ex2_approx(y3);
        }
      }
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int64_t i = q0 + c;
          if (!(key_ok && i < a.S && (!a.causal || i >= pj))) p[c] = 0.f;
        }
      }
      // P^T (bf16) back into this group's S columns: the A operand of dV.
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) pk[x] = pack_bf16(p[c * 32 + 2 * x], p[c * 32 + 2 * x + 1]);
        tmem_st16(tS + lane_off + c * 16, pk);
      }
      good = __all_sync(0xffffffffu, wait(dp_full + w, j & 1));
      if (!good) break;
      tc_fence_after();
      {
        uint32_t r[64];
        tmem_ld64_sync(tDP + lane_off, r);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 da = *reinterpret_cast<const float4*>(dv_s + u * 8);
          const float4 db = *reinterpret_cast<const float4*>(dv_s + u * 8 + 4);
          const float dvv[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
          uint32_t pk[4];
          const uint64_t sc2 = f2_pack(a.scale, a.scale);
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int col = u * 8 + 2 * x;
            const uint64_t t2 = ffma2(f2_pack_u(r[col], r[col + 1]), sc2,
                                      f2_pack(-dvv[2 * x], -dvv[2 * x + 1]));
            float d0, d1;
            f2_unpack(fmul2(t2, f2_pack(p[col], p[col + 1])), d0, d1);
            pk[x] = pack_bf16(d0, d1);
          }
          st_shared_v4(sDS + swz_offset(t, u * 8), pk[0], pk[1], pk[2], pk[3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full + w);

      good = __all_sync(0xffffffffu, wait(dq_full + w, j & 1));
      if (!good) break;
      tc_fence_after();
      // dQ^T: lane t = head-dim index d, column c = query row q0 + c. The TMEM region is
      // released as soon as it is in registers; the reductions drain behind the next MMAs.
      uint32_t r[64];
      tmem_ld64_sync(tDP + lane_off, r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free + w);
      float* dq_col = a.dqacc + (static_cast<int64_t>(zq) * a.S_pad + q0) * kD + t;
      const int64_t n_rows = a.S - q0;
#pragma unroll
      for (int x = 0; x < 64; ++x)
        if (x < n_rows) red_add_f32(dq_col + x * kD, __uint_as_float(r[x]));
    }
    if (good && n_it > 0) {
      good = __all_sync(0xffffffffu, wait(done, 0));
      if (good) tc_fence_after();
    }
    if (good) {
      // group 0 writes dV, group 1 writes dK (both already carry their final scaling)
      const uint32_t tAcc = w == 0 ? tDV : tDK;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(w == 0 ? a.dv : a.dk) +
                           ((static_cast<int64_t>(b) * a.S + pj) * a.Hkv + a.kvh0 + kvl) * kD;
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
  if (warp == 8) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int bwd_q_box_rows(int D) { return D == kD ? kSub : 128; }

cudaError_t launch_attn_bwd(int D, int B, const CUtensorMap& q_map, const CUtensorMap& do_map,
                            const CUtensorMap& k_map, const CUtensorMap& v_map,
                            const BwdArgs& a, cudaStream_t stream) {
  if (D != kD) return launch_attn_bwd_generic(D, B, q_map, do_map, k_map, v_map, a, stream);
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_pp_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PPLayout::kBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int64_t n_kt = (a.kv_row_hi - a.kv_row_lo + 127) / 128;
  dim3 grid(static_cast<unsigned>(n_kt), static_cast<unsigned>(a.kc), static_cast<unsigned>(B));
  launch_begin(3, stream);
  attn_bwd_pp_kernel<<<grid, kThreads, PPLayout::kBytes, stream>>>(q_map, do_map, k_map, v_map, a);
  cudaError_t e = cudaGetLastError();
  launch_end(3, stream);
  return e;
}

}  // namespace upipe
