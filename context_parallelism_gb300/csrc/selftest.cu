// Self-tests of the building blocks the attention kernels rely on:
//   * one 128 x N x K bf16 tcgen05 MMA tile with TMA-loaded (or hand-swizzled) operands in
//     K-major or MN-major shared-memory layouts, read back from TMEM;
//   * the bounded mbarrier wait, made to expire on purpose on a barrier nothing completes.
#include "internal.h"
#include "ptx.cuh"

namespace upipe {
namespace {

constexpr int kStThreads = 128;

struct StSmemLayout {
  static constexpr int kA = 0;                 // up to 2 boxes (32 KiB)
  static constexpr int kB = 2 * kBoxBytes;     // up to 2 boxes (32 KiB)
  static constexpr int kBar = 4 * kBoxBytes;   // 2 barriers
  static constexpr int kSlot = kBar + 16;
  static constexpr int kBytes = kSlot + 16 + 1024;
};

__global__ void __launch_bounds__(kStThreads, 1)
    selftest_umma_kernel(const __grid_constant__ CUtensorMap ta,
                         const __grid_constant__ CUtensorMap tb, const __nv_bfloat16* a_raw,
                         float* c, int N, int K, int a_mn, int b_mn, int a_manual, int lbo,
                         int sbo, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(smem + StSmemLayout::kBar);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + StSmemLayout::kSlot);
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;

  if (t == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(slot, 256);  // accumulator at column 0, a TMEM-resident A at column 128
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  uint8_t* sA = smem + StSmemLayout::kA;
  uint8_t* sB = smem + StSmemLayout::kB;

  if (a_manual == 2) {
    // Row t of A into TMEM lane t, two bf16 per 32-bit column (the MMA's TMEM A layout).
    uint32_t r[32];
    for (int half = 0; half < 2; ++half) {
      for (int i = 0; i < 32; ++i) {
        const uint32_t lo = reinterpret_cast<const uint16_t*>(a_raw)[t * 128 + half * 64 + 2 * i];
        const uint32_t hi = reinterpret_cast<const uint16_t*>(a_raw)[t * 128 + half * 64 + 2 * i + 1];
        r[i] = lo | (hi << 16);
      }
      tmem_st32(tmem + 128 + (static_cast<uint32_t>(warp * 32) << 16) + half * 32, r);
    }
    tmem_wait_st();
    tc_fence_before();
  } else if (a_manual) {
    // Row t of A ([128][128] row-major) into the swizzled K-major image.
    for (int col = 0; col < 128; col += 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(a_raw + static_cast<size_t>(t) * 128 + col);
      st_shared_v4(smem_u32(sA) + swz_offset(t, col), v.x, v.y, v.z, v.w);
    }
    fence_proxy_async_smem();
  }
  __syncthreads();

  bool ok = true;
  if (t == 0) {
    // Both operands are 128 x 128 buffers: two 64-column boxes each.
    const int a_boxes = a_manual ? 0 : 2;
    mbar_arrive_expect_tx(bar_load, static_cast<uint32_t>((a_boxes + 2) * kBoxBytes));
    for (int x = 0; x < a_boxes; ++x) tma_load_3d(sA + x * kBoxBytes, &ta, x * 64, 0, 0, bar_load);
    for (int x = 0; x < 2; ++x) tma_load_3d(sB + x * kBoxBytes, &tb, x * 64, 0, 0, bar_load);
    ok = mbar_wait(bar_load, 0);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, N, a_mn != 0, b_mn != 0);
      for (int k16 = 0; k16 < K / 16; ++k16) {
        const uint64_t db = b_mn ? desc_mnmajor(smem_u32(sB), k16, lbo, sbo)
                                 : desc_kmajor(smem_u32(sB), k16);
        if (a_manual == 2) {
          umma_f16_ts(tmem, tmem + 128 + k16 * 8, db, idesc, k16 > 0);
        } else {
          const uint64_t da = a_mn ? desc_mnmajor(smem_u32(sA), k16, lbo, sbo)
                                   : desc_kmajor(smem_u32(sA), k16);
          umma_f16_ss(tmem, da, db, idesc, k16 > 0);
        }
      }
      umma_commit(bar_mma);
      ok = mbar_wait(bar_mma, 0);
    }
    if (!ok) atomicOr(err, kErrWaitTimeout);
  }
  __syncthreads();
  tc_fence_after();
  // Every warp reads its 32 lanes (rows) of the accumulator.
  for (int col = 0; col < N; col += 32) {
    uint32_t r[32];
    tmem_ld32_sync(tmem + (static_cast<uint32_t>(warp * 32) << 16) + col, r);
    for (int i = 0; i < 32; ++i) c[static_cast<size_t>(t) * N + col + i] = __uint_as_float(r[i]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

__global__ void selftest_wait_kernel(uint64_t limit_ns, uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the wait must expire and report, not hang.
    if (!mbar_wait(&bar, 0, limit_ns)) atomicOr(err, kErrWaitTimeout | 0x100u);
  }
}

}  // namespace

cudaError_t launch_selftest_umma(const void* a, const void* b, float* c, int N, int K, int a_mn,
                                 int b_mn, int a_manual, int lbo, int sbo, uint32_t* err,
                                 cudaStream_t stream) {
  CUtensorMap ta, tb;
  cudaError_t e = make_tmap_bf16(&ta, a, 128, 128, 1);
  if (e != cudaSuccess) return e;
  e = make_tmap_bf16(&tb, b, 128, 128, 1);
  if (e != cudaSuccess) return e;
  e = ensure_smem_attr(reinterpret_cast<const void*>(&selftest_umma_kernel),
                       StSmemLayout::kBytes);
  if (e != cudaSuccess) return e;
  launch_begin(5, stream);
  selftest_umma_kernel<<<1, kStThreads, StSmemLayout::kBytes, stream>>>(
      ta, tb, static_cast<const __nv_bfloat16*>(a), c, N, K, a_mn, b_mn, a_manual, lbo, sbo,
      err);
  e = cudaGetLastError();
  launch_end(5, stream);
  return e;
}

cudaError_t launch_selftest_wait(int limit_us, uint32_t* err, cudaStream_t stream) {
  launch_begin(5, stream);
  selftest_wait_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(limit_us) * 1000ull, err);
  cudaError_t e = cudaGetLastError();
  launch_end(5, stream);
  return e;
}

}  // namespace upipe
