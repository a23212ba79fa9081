// Persistent tcgen05 GEMM for the sequence-tiled readout + cross-entropy loss, and the
// loss's own reduction kernel.
//
//   C[m, n] = sum_k A(m, k) B(n, k),   bf16 operands, fp32 accumulation in TMEM
//
// Tiles are 128 x 256 (one cta_group::1 MMA of M = 128, N = 256 per 16-element k step), the
// reduction advances 64 elements per pipeline stage. A and B are each either K-major (the
// reduction index is contiguous: A stored [M][K], B stored [N][K]) or MN-major (A stored
// [K][M], B stored [K][N]); TMA loads them with 128-byte swizzle into the canonical layouts the
// shared-memory descriptors describe (K-major: one 64-element box per stage; MN-major: 64-wide
// boxes of 64 reduction rows). Anything past the edge of a tensor map is zero-filled by TMA, so
// ragged M, N and K need no special path in the main loop.
//
// One CTA per SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...; warp 0 issues TMA loads
// into a 4-stage ring, warp 1 owns TMEM and issues the MMAs, warps 2-5 run the epilogue (warp w
// reads TMEM lanes 32*(w%4)..+31, i.e. one row of the tile per thread). Two 256-column fp32
// accumulators alternate between tiles, so a tile's epilogue overlaps the next tile's MMAs.
//
// Epilogues (the per-token loss, "Road to 5 million sequence length" talk notes, Arctic
// sequence-tiling passage; "Road to 5 Million Tokens" summary, section 2 item 5):
//   CE_FWD    logits -> per (row, 256-column tile): running max (log2 units) and sum of
//             2^(x log2e - max); the logit at the row's target when it falls in the tile;
//             optionally the fp32 logits themselves (the fused forward + backward)
//   CE_BWD    logits -> dlogits = g_row * (exp(logit - lse_row) - [col == target]) as bf16
//   STORE     C -> bf16
//   ACC_F32   C -> fp32, added to what is there when accumulating, else stored
// and those of the sequence-tiled gated MLP (same passages: "all the MLPs" are chunked):
//   SWIGLU    gate and up projections in one tile: the B stage holds 128 rows of the gate
//             block and the matching 128 rows of the up block (two TMA boxes), so one
//             accumulator holds g (columns 0-127) and u (128-255) of the same 128 outputs;
//             a = silu(g) * u -> bf16, and optionally g, u -> bf16 for the backward
//   DSWIGLU   da = dy Wd -> dg = da * u * silu'(g), du = da * silu(g) -> bf16, reading the
//             stored g, u
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kAStage = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kBStage = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kMnBox = 64 * kBK * 2;    // one 64-wide, 64-row MN-major box: 8 KiB
constexpr float kLog2e = 1.4426950408889634f;

// Output columns of one tile: the gated epilogue spends the 256 accumulator columns on 128
// outputs (their gate and up halves).
template <int EPI>
constexpr int out_cols() { return EPI == kEpiSwiglu ? kBN / 2 : kBN; }

struct GLayout {
  static constexpr int kA = 0;
  static constexpr int kB = kStages * kAStage;
  static constexpr int kBar = kB + kStages * kBStage;  // full[S] empty[S] acc_full[2] acc_empty[2] drain
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 4;
  static constexpr int kBytes = kAbort + 4 + 1024;
};

// Tile order. m_fastest: groups of `group` M tiles (all of them when group <= 0) are walked
// M tile first, then N tile, group after group - the CTAs in flight then share a few B strips
// and at most `group` A strips, which bounds the set of operand bytes that has to stay in L2.
// Otherwise the same with the roles of M and N exchanged (groups of N tiles, N tile first).
__device__ __forceinline__ void tile_coords(int t, int mt_n, int nt_n, int m_fastest, int group,
                                            int& mt, int& nt) {
  const int fast_n = m_fastest ? mt_n : nt_n;  // tiles along the fast dimension
  const int slow_n = m_fastest ? nt_n : mt_n;
  const int g = (group > 0 && group < fast_n) ? group : fast_n;
  const int per_group = g * slow_n;
  const int grp = t / per_group;
  const int rem = t - grp * per_group;
  const int f0 = grp * g;
  const int width = min(g, fast_n - f0);
  const int f = f0 + rem % width;
  const int sl = rem / width;
  mt = m_fastest ? f : sl;
  nt = m_fastest ? sl : f;
}

__device__ __forceinline__ uint4 pack8(const float* x) {
  return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                    pack_bf16(x[6], x[7]));
}

// One 32-column slice of the tile for this thread's row (x: the fp32 accumulators).
template <int EPI>
struct Epi;

template <>
struct Epi<kEpiCeFwd> {
  float mx = -INFINITY, sm = 0.f, tl = 0.f;
  int64_t tg = -1;
  __device__ void begin(const GemmArgs& a, int64_t row, bool row_ok) {
    mx = -INFINITY;
    sm = 0.f;
    tl = 0.f;
    tg = row_ok ? a.target[row] : -1;
  }
  __device__ void slice(const GemmArgs& a, int64_t row, bool row_ok, int col0, const float* x) {
    if (a.c && row_ok) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.c) + row * a.ldc + col0);
#pragma unroll
      for (int v = 0; v < 8; ++v)
        dst[v] = make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
    }
    float cm = x[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) cm = fmaxf(cm, x[j]);
    const float mn = fmaxf(mx, cm * kLog2e);
    float cs = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) cs += ex2_approx(fmaf(x[j], kLog2e, -mn));
    sm = fmaf(sm, ex2_approx(mx - mn), cs);
    mx = mn;
    const int64_t off = tg - col0;
    if (off >= 0 && off < 32) {
      // a multiply-add per column keeps x in registers (a select would become an indexed
      // load from a local-memory copy)
      const int o = static_cast<int>(off);
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) acc = fmaf(x[j], j == o ? 1.f : 0.f, acc);
      tl = acc;
    }
  }
  __device__ void end(const GemmArgs& a, int64_t row, bool row_ok, int nt, int n0) {
    if (!row_ok) return;
    reinterpret_cast<float2*>(a.part)[static_cast<int64_t>(nt) * a.part_stride + row] =
        make_float2(mx, sm);
    if (tg >= n0 && tg < n0 + kBN && tg < a.N) a.tlogit[row] = tl;
  }
};

template <>
struct Epi<kEpiCeBwd> {
  float lse2 = 0.f, gi = 0.f;
  int64_t tg = -1;
  __device__ void begin(const GemmArgs& a, int64_t row, bool row_ok) {
    tg = row_ok ? a.target[row] : -1;
    lse2 = row_ok ? a.lse[row] * kLog2e : 0.f;
    gi = (row_ok && tg >= 0) ? a.g[row] : 0.f;
    if (tg >= a.N) gi = __int_as_float(0x7fc00000);  // target outside the vocabulary: NaN
  }
  __device__ void slice(const GemmArgs& a, int64_t row, bool row_ok, int col0, const float* x) {
    float d[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float p = ex2_approx(fmaf(x[j], kLog2e, -lse2));
      d[j] = gi * (p - (static_cast<int64_t>(col0 + j) == tg ? 1.f : 0.f));
    }
    if (!row_ok) return;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.c) + row * a.ldc + col0);
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = pack8(d + 8 * v);
  }
  __device__ void end(const GemmArgs&, int64_t, bool, int, int) {}
};

template <>
struct Epi<kEpiStoreBf16> {
  __device__ void begin(const GemmArgs&, int64_t, bool) {}
  __device__ void slice(const GemmArgs& a, int64_t row, bool row_ok, int col0, const float* x) {
    if (!row_ok) return;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.c) + row * a.ldc + col0);
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = pack8(x + 8 * v);
  }
  __device__ void end(const GemmArgs&, int64_t, bool, int, int) {}
};

// silu(g) = g / (1 + e^-g) and silu'(g) = s (1 + g (1 - s)), s = 1 / (1 + e^-g); __expf and
// __fdividef saturate cleanly at both ends (e^-g = inf gives silu = -0, s = 0).
__device__ __forceinline__ void silu_parts(float g, float& sg, float& dsg) {
  const float s = __fdividef(1.f, 1.f + __expf(-g));
  sg = g * s;
  dsg = s * fmaf(g, 1.f - s, 1.f);
}

template <>
struct Epi<kEpiSwiglu> {
  __device__ void begin(const GemmArgs&, int64_t, bool) {}
  // g, u: the gate and up accumulators of output columns col0 .. col0+31
  __device__ void slice2(const GemmArgs& a, int64_t row, bool row_ok, int col0, const float* g,
                         const float* u) {
    float o[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float s = __fdividef(1.f, 1.f + __expf(-g[j]));
      o[j] = g[j] * s * u[j];
    }
    if (!row_ok) return;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.c) + row * a.ldc + col0);
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = pack8(o + 8 * v);
    if (a.c2) {
      __nv_bfloat16* base = static_cast<__nv_bfloat16*>(a.c2) + row * a.ldc2;
      uint4* dg = reinterpret_cast<uint4*>(base + col0);
      uint4* du = reinterpret_cast<uint4*>(base + a.split + col0);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        dg[v] = pack8(g + 8 * v);
        du[v] = pack8(u + 8 * v);
      }
    }
  }
  __device__ void end(const GemmArgs&, int64_t, bool, int, int) {}
};

__device__ __forceinline__ void unpack8(uint4 v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <>
struct Epi<kEpiDSwiglu> {
  __device__ void begin(const GemmArgs&, int64_t, bool) {}
  __device__ void slice(const GemmArgs& a, int64_t row, bool row_ok, int col0, const float* da) {
    if (!row_ok) return;
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.aux) + row * a.ld_aux;
    const uint4* pg = reinterpret_cast<const uint4*>(src + col0);
    const uint4* pu = reinterpret_cast<const uint4*>(src + a.split + col0);
    float dg[32], du[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      float g[8], u[8];
      unpack8(pg[v], g);
      unpack8(pu[v], u);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float sg, dsg;
        silu_parts(g[i], sg, dsg);
        dg[8 * v + i] = da[8 * v + i] * u[i] * dsg;
        du[8 * v + i] = da[8 * v + i] * sg;
      }
    }
    __nv_bfloat16* base = static_cast<__nv_bfloat16*>(a.c) + row * a.ldc;
    uint4* og = reinterpret_cast<uint4*>(base + col0);
    uint4* ou = reinterpret_cast<uint4*>(base + a.split + col0);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      og[v] = pack8(dg + 8 * v);
      ou[v] = pack8(du + 8 * v);
    }
  }
  __device__ void end(const GemmArgs&, int64_t, bool, int, int) {}
};

template <>
struct Epi<kEpiAccF32> {
  __device__ void begin(const GemmArgs&, int64_t, bool) {}
  __device__ void slice(const GemmArgs& a, int64_t row, bool row_ok, int col0, const float* x) {
    if (!row_ok) return;
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.c) + row * a.ldc + col0);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      float4 r = make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
      if (a.accumulate) {
        const float4 o = dst[v];
        r.x += o.x;
        r.y += o.y;
        r.z += o.z;
        r.w += o.w;
      }
      dst[v] = r;
    }
  }
  __device__ void end(const GemmArgs&, int64_t, bool, int, int) {}
};

template <int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_b, const GemmArgs a) {
  using L = GLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* full = bar;
  uint64_t* empty = bar + kStages;
  uint64_t* acc_full = bar + 2 * kStages;
  uint64_t* acc_empty = bar + 2 * kStages + 2;
  uint64_t* drain = bar + 2 * kStages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int mt_n = (a.M + kBM - 1) / kBM;
  constexpr int kOut = out_cols<EPI>();
  const int nt_n = (a.N + kOut - 1) / kOut;
  const int nk = (a.K + kBK - 1) / kBK;
  const int n_tiles = mt_n * nt_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

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

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      int s = 0;
      uint32_t ph = 0;
      int64_t fills = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        int mt, nt;
        tile_coords(t, mt_n, nt_n, a.m_fastest, a.group_m, mt, nt);
        for (int kb = 0; kb < nk; ++kb) {
          if (!wait(empty + s, ph ^ 1)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + L::kA + s * kAStage;
          uint8_t* sb = smem + L::kB + s * kBStage;
          mbar_arrive_expect_tx(full + s, kAStage + kBStage);
          if (A_MN) {
#pragma unroll
            for (int i = 0; i < kBM / 64; ++i)
              tma_load_3d(sa + i * kMnBox, &tm_a, mt * kBM + 64 * i, kb * kBK, 0, full + s);
          } else {
            tma_load_3d(sa, &tm_a, kb * kBK, mt * kBM, 0, full + s);
          }
          if (EPI == kEpiSwiglu) {
            // 128 gate rows, then the 128 up rows of the same outputs (128-row boxes)
            tma_load_3d(sb, &tm_b, kb * kBK, nt * kOut, 0, full + s);
            tma_load_3d(sb + kBStage / 2, &tm_b, kb * kBK, a.split + nt * kOut, 0, full + s);
          } else if (B_MN) {
#pragma unroll
            for (int i = 0; i < kBN / 64; ++i)
              tma_load_3d(sb + i * kMnBox, &tm_b, nt * kBN + 64 * i, kb * kBK, 0, full + s);
          } else {
            tma_load_3d(sb, &tm_b, kb * kBK, nt * kBN, 0, full + s);
          }
          ++fills;
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok) {
        // let the loads still in flight land before the CTA exits
        const int64_t first = fills > kStages ? fills - kStages : 0;
        for (int64_t f = first; f < fills; ++f)
          mbar_wait(full + (f % kStages), static_cast<uint32_t>((f / kStages) & 1), 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kBM, kBN, A_MN, B_MN);
      const uint32_t sa0 = smem_u32(smem + L::kA), sb0 = smem_u32(smem + L::kB);
      const uint64_t dA0 = A_MN ? mndesc0(sa0, kMnBox, 1024u) : kdesc0(sa0);
      const uint64_t dB0 = B_MN ? mndesc0(sb0, kMnBox, 1024u) : kdesc0(sb0);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++it) {
        const int acc = it & 1;
        if (!wait(acc_empty + acc, ((it >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tD = tmem + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!wait(full + s, ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dA = dA0 + s * (kAStage >> 4);
          const uint64_t dB = dB0 + s * (kBStage >> 4);
#pragma unroll
          for (int k16 = 0; k16 < kBK / 16; ++k16)
            umma_f16_ss(tD, dA + (A_MN ? mnstep(k16) : kstep(k16)),
                        dB + (B_MN ? mnstep(k16) : kstep(k16)), idesc,
                        (kb > 0 || k16 > 0) ? 1u : 0u);
          umma_commit(empty + s);
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(acc_full + acc);
      }
      if (!ok) {
        umma_commit(drain);
        mbar_wait(drain, 0, 100000000ull);
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5, one tile row per thread ----------------
    const int quarter = warp & 3;
    const int r_in = 32 * quarter + lane;
    int it = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
      int mt, nt;
      tile_coords(t, mt_n, nt_n, a.m_fastest, a.group_m, mt, nt);
      const int acc = it & 1;
      if (!wait(acc_full + acc, (it >> 1) & 1)) break;
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(mt) * kBM + r_in;
      const bool row_ok = row < a.M;
      const int n0 = nt * kOut;
      const uint32_t tD = tmem + (static_cast<uint32_t>(32 * quarter) << 16) +
                          static_cast<uint32_t>(acc * kBN);
      Epi<EPI> e;
      e.begin(a, row, row_ok);
      if constexpr (EPI == kEpiSwiglu) {
        for (int c = 0; c < kOut; c += 32) {  // N % 128 == 0: every slice is inside
          uint32_t rg[32], ru[32];
          tmem_ld32_sync(tD + static_cast<uint32_t>(c), rg);
          tmem_ld32_sync(tD + static_cast<uint32_t>(kOut + c), ru);
          float xg[32], xu[32];  // explicit bit casts: no float access through the uint32 array
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            xg[j] = __uint_as_float(rg[j]);
            xu[j] = __uint_as_float(ru[j]);
          }
          e.slice2(a, row, row_ok, n0 + c, xg, xu);
        }
      } else {
        for (int c = 0; c < kBN; c += 32) {
          if (n0 + c >= a.N) break;  // N % 64 == 0: a slice is wholly inside or outside
          uint32_t r[32];
          tmem_ld32_sync(tD + static_cast<uint32_t>(c), r);
          float x[32];  // explicit bit casts: no float access through the uint32 array
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
          e.slice(a, row, row_ok, n0 + c, x);
        }
      }
      e.end(a, row, row_ok, nt, n0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// One thread per token row: merge the per-tile (max, sum) pairs of the row into its
// log-sum-exp, and the loss lse - logit[target] (0 for an ignored token, NaN for a target
// outside the vocabulary).
__global__ void ce_merge_kernel(const float2* __restrict__ part, int64_t part_stride, int n_parts,
                                const float* __restrict__ tlogit, const int64_t* __restrict__ target,
                                float* __restrict__ loss, float* __restrict__ lse, int64_t M,
                                int64_t V) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= M) return;
  float mx = -INFINITY;
  for (int k = 0; k < n_parts; ++k) mx = fmaxf(mx, part[k * part_stride + row].x);
  float sm = 0.f;
  for (int k = 0; k < n_parts; ++k) {
    const float2 p = part[k * part_stride + row];
    sm += p.y * exp2f(p.x - mx);
  }
  const float l = (mx + log2f(sm)) * 0.6931471805599453f;
  lse[row] = l;
  const int64_t tg = target[row];
  loss[row] = tg < 0 ? 0.f : (tg < V ? l - tlogit[row] : __int_as_float(0x7fc00000));
}

// One block per token row: dl[r][j] = g_r (exp(L[r][j] - lse_r) - [j == target_r]) as bf16,
// from the fp32 logits the CE_FWD epilogue stored - the same arithmetic, in the same order, as
// the CE_BWD epilogue applies to recomputed logits, so both give the same bits. Rows of ignored
// tokens are zero; a target outside the vocabulary makes its row NaN. V % 8 == 0.
__global__ void ce_dlogits_kernel(const float* __restrict__ L, const float* __restrict__ lse,
                                  const int64_t* __restrict__ target, const float* __restrict__ g,
                                  __nv_bfloat16* __restrict__ dl, int64_t V) {
  const int64_t r = blockIdx.x;
  const int64_t tg = target[r];
  float gi = tg >= 0 ? g[r] : 0.f;
  if (tg >= V) gi = __int_as_float(0x7fc00000);
  const float lse2 = lse[r] * kLog2e;
  const float4* src = reinterpret_cast<const float4*>(L + r * V);
  uint4* dst = reinterpret_cast<uint4*>(dl + r * V);
  for (int64_t q = threadIdx.x; q < V / 8; q += blockDim.x) {
    const float4 u = src[2 * q], w = src[2 * q + 1];
    const float x[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
    float d[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float p = ex2_approx(fmaf(x[k], kLog2e, -lse2));
      d[k] = gi * (p - (8 * q + k == tg ? 1.f : 0.f));
    }
    dst[q] = pack8(d);
  }
}

template <int EPI, bool A_MN, bool B_MN>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                       int grid_cap, cudaStream_t stream) {
  {
    const cudaError_t e = ensure_smem_attr(
        reinterpret_cast<const void*>(&gemm_tc_kernel<EPI, A_MN, B_MN>), GLayout::kBytes);
    if (e != cudaSuccess) return e;
  }
  constexpr int kOut = out_cols<EPI>();
  const int64_t tiles = static_cast<int64_t>((a.M + kBM - 1) / kBM) * ((a.N + kOut - 1) / kOut);
  const int grid = static_cast<int>(tiles < grid_cap ? tiles : grid_cap);
  if (grid <= 0) return cudaSuccess;
  launch_begin(6, stream);
  gemm_tc_kernel<EPI, A_MN, B_MN><<<grid, kThreads, GLayout::kBytes, stream>>>(ta, tb, a);
  cudaError_t e = cudaGetLastError();
  launch_end(6, stream);
  return e;
}

}  // namespace

cudaError_t launch_gemm_tc(int epi, bool a_mn, bool b_mn, const CUtensorMap& ta,
                           const CUtensorMap& tb, const GemmArgs& a, int grid_cap,
                           cudaStream_t stream) {
  if (epi == kEpiCeFwd && !a_mn && !b_mn) return launch_one<kEpiCeFwd, false, false>(ta, tb, a, grid_cap, stream);
  if (epi == kEpiCeBwd && !a_mn && !b_mn) return launch_one<kEpiCeBwd, false, false>(ta, tb, a, grid_cap, stream);
  if (epi == kEpiStoreBf16 && !a_mn && b_mn) return launch_one<kEpiStoreBf16, false, true>(ta, tb, a, grid_cap, stream);
  if (epi == kEpiAccF32 && a_mn && b_mn) return launch_one<kEpiAccF32, true, true>(ta, tb, a, grid_cap, stream);
  if (epi == kEpiStoreBf16 && !a_mn && !b_mn) return launch_one<kEpiStoreBf16, false, false>(ta, tb, a, grid_cap, stream);
  if (epi == kEpiSwiglu && !a_mn && !b_mn) return launch_one<kEpiSwiglu, false, false>(ta, tb, a, grid_cap, stream);
  if (epi == kEpiDSwiglu && !a_mn && b_mn) return launch_one<kEpiDSwiglu, false, true>(ta, tb, a, grid_cap, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_ce_dlogits(const float* logits, const float* lse, const int64_t* target,
                              const float* g, void* dl, int64_t M, int64_t V, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  launch_begin(7, stream);
  ce_dlogits_kernel<<<static_cast<unsigned>(M), 256, 0, stream>>>(
      logits, lse, target, g, static_cast<__nv_bfloat16*>(dl), V);
  cudaError_t e = cudaGetLastError();
  launch_end(7, stream);
  return e;
}

cudaError_t launch_ce_merge(const float* part, int64_t part_stride, int n_parts,
                            const float* tlogit, const int64_t* target, float* loss, float* lse,
                            int64_t M, int64_t V, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = static_cast<int>((M + threads - 1) / threads);
  launch_begin(7, stream);
  ce_merge_kernel<<<blocks, threads, 0, stream>>>(reinterpret_cast<const float2*>(part),
                                                  part_stride, n_parts, tlogit, target, loss,
                                                  lse, M, V);
  cudaError_t e = cudaGetLastError();
  launch_end(7, stream);
  return e;
}

}  // namespace upipe
