// Backward causal (GQA) attention on sm_103a, one 128-row query tile per step (used for
// D = 64; D = 128 runs the ping-pong kernel in attn_bwd_pp.cu).
//
// One CTA owns a 128-row key/value tile of one kv-head and walks the query tiles of every
// q-head of its group that can see it (query rows >= the tile's first key when causal). Per
// query tile it recomputes the probabilities from the saved log-sum-exp instead of storing
// the S x S matrix, which is the recompute that makes the attention backward pass fit
// ("Training Ultra Long Context LM with Fully Pipelined Distributed Transformer",
// Background: the backward pass of attention is the memory peak; the "Road to 5 million
// sequence length" talk's UPipe passage: each head group is recomputed, then attended).
//
// Per (key tile, query tile), with j the key row (TMEM lane / thread) and i the query row:
//   S^T  = K Q^T                (tcgen05, TMEM cols [0,128))
//   dP^T = V dO^T               (tcgen05, TMEM cols [128,256))
//   P^T  = exp2(S^T * scale*log2e - LSE_i*log2e), masked   (registers -> smem, bf16)
//   dS^T = P^T * (scale*dP^T - scale*D_i)                 (registers -> smem, bf16)
//   dV  += P^T dO               (tcgen05, TMEM cols [256,256+D))
//   dK  += dS^T Q               (tcgen05, TMEM cols [256+D,256+2D))
//   dQ   = dS K                 (tcgen05, TMEM cols [0,D), reusing S^T), added to the fp32
//                               dQ accumulator with vector atomics
// (the softmax scale rides in dS, so dK and dQ need no scaling afterwards)
//
// CTA layout (192 threads): warps 0-3 compute (thread t = key row t), warp 4 TMEM + MMA
// issue, warp 5 TMA producer. Shared memory: K, V (resident), Q, dO (one stage), P^T, dS^T,
// and the 128-entry LSE and D vectors of the current query tile.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {
namespace {

constexpr int kThreads = 192;

template <int D>
struct BwdLayout {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;
  static constexpr int kDO = kQ + kTile;
  static constexpr int kPT = kDO + kTile;       // 128 x 128 bf16
  static constexpr int kDST = kPT + 32768;      // 128 x 128 bf16
  static constexpr int kLse = kDST + 32768;     // 128 fp32
  static constexpr int kDv = kLse + 512;        // 128 fp32
  static constexpr int kBar = kDv + 512;
  static constexpr int kNumBars = 9;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 4;
  static constexpr int kBytes = kAbort + 4 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const BwdArgs a) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bar + 0;
  uint64_t* q_full = bar + 1;
  uint64_t* q_empty = bar + 2;
  uint64_t* s_full = bar + 3;
  uint64_t* ds_full = bar + 4;
  uint64_t* dq_full = bar + 5;
  uint64_t* dq_free = bar + 6;
  uint64_t* done = bar + 7;
  uint64_t* drain = bar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  float* lse_s = reinterpret_cast<float*>(smem + L::kLse);
  float* dv_s = reinterpret_cast<float*>(smem + L::kDv);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kt = blockIdx.x;  // smallest key positions (most query tiles) first
  const int kvl = blockIdx.y;
  const int b = blockIdx.z;
  const int64_t r0 = a.kv_row_lo + static_cast<int64_t>(kt) * 128;  // K/V map row
  const int64_t p0 = a.kv_pos0 + r0;                                // global key position
  const int zk = b * a.kc + kvl;
  const int qt_lo = a.causal ? static_cast<int>(p0 / 128) : 0;
  const int qt_hi = static_cast<int>((a.S + 127) / 128);
  const int nq = qt_hi > qt_lo ? qt_hi - qt_lo : 0;
  const int n_it = a.G * nq;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(ds_full, 128);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 128);
    mbar_init(done, 1);
    mbar_init(drain, 1);
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
  const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 256 + D;
  const uint32_t tDQ = tmem;

  auto wait = [&](uint64_t* br, uint32_t parity) -> bool {
    if (mbar_try_wait(br, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (mbar_try_wait(br, parity)) return true;
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(a.err, kErrWaitTimeout | 0x2000u);
        return false;
      }
    }
  };
  auto decode = [&](int it, int& zq, int64_t& q0) {
    const int hl = kvl * a.G + it / nq;
    zq = b * a.hc + hl;
    q0 = static_cast<int64_t>(qt_lo + it % nq) * 128;
  };

  if (warp == 5) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(kv_full, 2 * L::kTile);
      for (int x = 0; x < D / 64; ++x) {
        tma_load_3d(smem + L::kK + x * kBoxBytes, &tm_k, x * 64, static_cast<int>(r0), zk, kv_full);
        tma_load_3d(smem + L::kV + x * kBoxBytes, &tm_v, x * 64, static_cast<int>(r0), zk, kv_full);
      }
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        if (it >= 1 && !wait(q_empty, (it - 1) & 1)) {
          ok = false;
          break;
        }
        int zq;
        int64_t q0;
        decode(it, zq, q0);
        mbar_arrive_expect_tx(q_full, 2 * L::kTile + 1024);
        for (int x = 0; x < D / 64; ++x) {
          tma_load_3d(smem + L::kQ + x * kBoxBytes, &tm_q, x * 64, static_cast<int>(q0), zq, q_full);
          tma_load_3d(smem + L::kDO + x * kBoxBytes, &tm_do, x * 64, static_cast<int>(q0), zq, q_full);
        }
        const int64_t vo = static_cast<int64_t>(zq) * a.S_pad + q0;
        bulk_load(lse_s, a.lse2 + vo, 512, q_full);
        bulk_load(dv_s, a.dvec + vo, 512, q_full);
        issued = it + 1;
      }
      mbar_wait(kv_full, 0, ok ? kWaitLimitNs : 100000000ull);
      if (!ok && issued > 0) mbar_wait(q_full, (issued - 1) & 1, 100000000ull);
    }
  } else if (warp == 4) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_ss = idesc_bf16(128, 128, false, false);
      const uint32_t id_kmn = idesc_bf16(128, D, false, true);  // A K-major, B MN-major
      const uint32_t id_mnmn = idesc_bf16(128, D, true, true);  // A MN-major, B MN-major
      const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
      const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
      const uint32_t sPT = smem_u32(smem + L::kPT), sDST = smem_u32(smem + L::kDST);
      bool ok = wait(kv_full, 0);
      for (int it = 0; ok && it < n_it; ++it) {
        if (!wait(q_full, it & 1)) { ok = false; break; }
        if (it >= 1 && !wait(dq_free, (it - 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          umma_f16_ss(tS, desc_kmajor(sK, k16), desc_kmajor(sQ, k16), id_ss, k16 > 0 ? 1u : 0u);
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          umma_f16_ss(tDP, desc_kmajor(sV, k16), desc_kmajor(sDO, k16), id_ss, k16 > 0 ? 1u : 0u);
        umma_commit(s_full);
        if (!wait(ds_full, it & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tDV, desc_kmajor(sPT, k16), desc_mnmajor(sDO, k16), id_kmn,
                      k16 > 0 ? 1u : acc0);
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tDK, desc_kmajor(sDST, k16), desc_mnmajor(sQ, k16), id_kmn,
                      k16 > 0 ? 1u : acc0);
        umma_commit(q_empty);
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)
          umma_f16_ss(tDQ, desc_mnmajor(sDST, k16), desc_mnmajor(sK, k16), id_mnmn,
                      k16 > 0 ? 1u : 0u);
        umma_commit(dq_full);
      }
      if (ok) {
        umma_commit(done);
      } else {
        umma_commit(drain);
        mbar_wait(drain, 0, 100000000ull);
      }
    }
  } else {
    // ---------------- compute warps ----------------
    const int t = threadIdx.x;  // key row within the tile (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int64_t pj = p0 + t;                    // this thread's key position
    const bool key_ok = (r0 + t) < a.kv_row_hi;   // inside this trunk
    const uint32_t sPT = smem_u32(smem + L::kPT), sDST = smem_u32(smem + L::kDST);
    bool good = true;
    for (int it = 0; it < n_it; ++it) {
      int zq;
      int64_t q0;
      decode(it, zq, q0);
      // q_full: the LSE / D vectors of this tile landed (its next phase needs this
      // iteration's ds_full, so the parity cannot have moved on).
      good = __all_sync(0xffffffffu, wait(q_full, it & 1) && wait(s_full, it & 1));
      if (!good) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t rs[32], rd[32];
        tmem_ld32_sync(tS + lane_off + c * 32, rs);
        tmem_ld32_sync(tDP + lane_off + c * 32, rd);
        float p[32], ds[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int col = c * 32 + x;
          const int64_t i = q0 + col;
          const bool vis = key_ok && (i < a.S) && (!a.causal || i >= pj);
          const float pv = vis ? ex2_approx(fmaf(__uint_as_float(rs[x]), a.scale_log2, lse_s[col])) : 0.f;
          p[x] = pv;
          ds[x] = pv * fmaf(__uint_as_float(rd[x]), a.scale, dv_s[col]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t off = swz_offset(t, c * 32 + u * 8);
          st_shared_v4(sPT + off, pack_bf16(p[u * 8 + 0], p[u * 8 + 1]),
                       pack_bf16(p[u * 8 + 2], p[u * 8 + 3]), pack_bf16(p[u * 8 + 4], p[u * 8 + 5]),
                       pack_bf16(p[u * 8 + 6], p[u * 8 + 7]));
          st_shared_v4(sDST + off, pack_bf16(ds[u * 8 + 0], ds[u * 8 + 1]),
                       pack_bf16(ds[u * 8 + 2], ds[u * 8 + 3]),
                       pack_bf16(ds[u * 8 + 4], ds[u * 8 + 5]),
                       pack_bf16(ds[u * 8 + 6], ds[u * 8 + 7]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_full);

      good = __all_sync(0xffffffffu, wait(dq_full, it & 1));
      if (!good) break;
      tc_fence_after();
      const int64_t qrow = q0 + t;  // for dQ the TMEM lane is the query row
      float* dqrow = a.dqacc + (static_cast<int64_t>(zq) * a.S_pad + qrow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_sync(tDQ + lane_off + c * 32, r);
        if (qrow < a.S) {
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            atomicAdd(reinterpret_cast<float4*>(dqrow + c * 32 + x),
                      make_float4(__uint_as_float(r[x]), __uint_as_float(r[x + 1]),
                                  __uint_as_float(r[x + 2]), __uint_as_float(r[x + 3])));
        }
      }
      tc_fence_before();
      mbar_arrive(dq_free);
    }
    if (good && n_it > 0) {
      good = __all_sync(0xffffffffu, wait(done, 0));
      if (good) tc_fence_after();
    }
    if (good) {
      const int64_t off =
          ((static_cast<int64_t>(b) * a.dkv_rows + pj - a.dkv_row0) * a.dkv_heads + a.dkv_head0 +
           kvl) * D;
      __nv_bfloat16* dvrow = static_cast<__nv_bfloat16*>(a.dv) + off;
      __nv_bfloat16* dkrow = static_cast<__nv_bfloat16*>(a.dk) + off;
      const bool store = key_ok && pj < a.S;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        uint32_t w[16];
        if (n_it > 0) {
          tmem_ld32_sync(tDV + lane_off + c * 32, r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        if (store) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(dvrow + c * 32 + i * 8) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
        if (n_it > 0) {
          tmem_ld32_sync(tDK + lane_off + c * 32, r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        if (store) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(dkrow + c * 32 + i * 8) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
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
cudaError_t launch_impl(int B, const CUtensorMap& q_map, const CUtensorMap& do_map,
                        const CUtensorMap& k_map, const CUtensorMap& v_map, const BwdArgs& a,
                        cudaStream_t stream) {
  using L = BwdLayout<D>;
  {
    const cudaError_t e =
        ensure_smem_attr(reinterpret_cast<const void*>(&attn_bwd_kernel<D>), L::kBytes);
    if (e != cudaSuccess) return e;
  }
  const int64_t n_kt = (a.kv_row_hi - a.kv_row_lo + 127) / 128;
  dim3 grid(static_cast<unsigned>(n_kt), static_cast<unsigned>(a.kc), static_cast<unsigned>(B));
  launch_begin(3, stream);
  attn_bwd_kernel<D><<<grid, kThreads, L::kBytes, stream>>>(q_map, do_map, k_map, v_map, a);
  cudaError_t e = cudaGetLastError();
  launch_end(3, stream);
  return e;
}

}  // namespace

cudaError_t launch_attn_bwd_generic(int D, int B, const CUtensorMap& q_map,
                                    const CUtensorMap& do_map, const CUtensorMap& k_map,
                                    const CUtensorMap& v_map, const BwdArgs& a,
                                    cudaStream_t stream) {
  if (D == 128) return launch_impl<128>(B, q_map, do_map, k_map, v_map, a, stream);
  if (D == 64) return launch_impl<64>(B, q_map, do_map, k_map, v_map, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace upipe
