// HBM-bound kernels around the attention kernels:
//   * seq_to_head_major / head_to_seq_major: the single-GPU stand-in for DeepSpeed Ulysses'
//     head<->sequence all-to-all, which gathers the whole sequence for a subset of heads
//     ("Training Ultra Long Context LM with Fully Pipelined Distributed Transformer",
//     Technical Deep Dive, first paragraph). Here it copies one head group of a token-major
//     [B,S,H,D] tensor into a head-major [B,h,S,D] workspace (and back).
//   * the backward pre-pass: scale * D_i, D_i = <dO_i, O_i> in fp32, the dO gather, the LSE prescale by
//     log2(e) and the zeroing of the fp32 dQ accumulator, fused in one pass;
//   * the dQ conversion: fp32 accumulator -> bf16 token-major dq.
// Each thread moves 16-byte vectors. Blocks cover fixed runs of sequence positions of one batch
// row and head, so no 64-bit division is done per element; the gathers of a head group's Q, K
// and V go in one launch.
#include <cuda_bf16.h>

#include "internal.h"

namespace upipe {
namespace {

constexpr int kLayoutThreads = 256;
// A block task of the gather / scatter kernels moves 16 KiB: 4 16-byte vectors per thread, all
// loaded before any is stored.
constexpr int kVecPerThread = 4;
constexpr int kBlockVecs = kLayoutThreads * kVecPerThread;

// Up to three head-group copies in one launch. Job j moves heads [h0, h0 + count) of a
// token-major [B, S, H, D] tensor to (or, for the scatter, from) a head-major
// [B, count, S, D] buffer. A block task is one run of `rows` consecutive sequence positions of
// one (batch row, head): its head-major side is one contiguous 16 KiB run, its token-major side
// `rows` pieces of D * 2 bytes, one per position. Tasks are numbered job, then (batch, head),
// then position run fastest, so neighbouring blocks stream neighbouring positions of a head.
struct LayoutJobs {
  const uint4* src[3];
  uint4* dst[3];
  int H[3], h0[3], count[3];
  int first_block[4];  // prefix sums of the jobs' task counts (B * count * seq_blocks)
  int seq_blocks;      // position runs per (batch row, head): ceil(S / rows)
  int rows;            // positions per run: kBlockVecs / Dc
  int lg_dc;           // log2 of the 16-byte vectors per position (Dc = D / 8)
  int n_jobs;
};

template <bool kToHead>
__global__ void __launch_bounds__(kLayoutThreads)
    layout_kernel(const LayoutJobs J, int64_t S) {
  const int task = static_cast<int>(blockIdx.x);
  // the job's fields picked by selects, not by a runtime index into the parameter block
  const int j = (task >= J.first_block[1]) + (J.n_jobs > 2 && task >= J.first_block[2]);
  auto pick = [j](auto x0, auto x1, auto x2) { return j == 0 ? x0 : (j == 1 ? x1 : x2); };
  const int bt = task - pick(J.first_block[0], J.first_block[1], J.first_block[2]);
  const int hb = bt / J.seq_blocks;
  const int sb = bt - hb * J.seq_blocks;
  const int count = pick(J.count[0], J.count[1], J.count[2]);
  const int H = pick(J.H[0], J.H[1], J.H[2]);
  const int hj0 = pick(J.h0[0], J.h0[1], J.h0[2]);
  const int b = hb / count, h = hb - b * count;
  const int64_t s0 = static_cast<int64_t>(sb) * J.rows;
  const int nrows = static_cast<int>(S - s0 < J.rows ? S - s0 : J.rows);
  const int n = nrows << J.lg_dc;
  const int Dc = 1 << J.lg_dc;
  // head-major run: ((b * count + h) * S + s0) * Dc + i; token-major vector i of the run:
  // ((b * S + s0 + r) * H + h0 + h) * Dc + c with r = i / Dc, c = i % Dc
  const int64_t hm0 = ((static_cast<int64_t>(b) * count + h) * S + s0) << J.lg_dc;
  const int64_t tok0 = ((static_cast<int64_t>(b) * S + s0) * H + hj0 + h) << J.lg_dc;
  const int64_t tokStride = static_cast<int64_t>(H) << J.lg_dc;
  const uint4* __restrict__ src = pick(J.src[0], J.src[1], J.src[2]);
  uint4* __restrict__ dst = pick(J.dst[0], J.dst[1], J.dst[2]);
  uint4 v[kVecPerThread];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int i = static_cast<int>(threadIdx.x) + u * kLayoutThreads;
    if (i < n) {
      const int64_t tok = tok0 + (i >> J.lg_dc) * tokStride + (i & (Dc - 1));
      v[u] = __ldg(src + (kToHead ? tok : hm0 + i));
    }
  }
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int i = static_cast<int>(threadIdx.x) + u * kLayoutThreads;
    if (i < n) {
      const int64_t tok = tok0 + (i >> J.lg_dc) * tokStride + (i & (Dc - 1));
      dst[kToHead ? hm0 + i : tok] = v[u];
    }
  }
}

cudaError_t launch_layout(bool to_head, const void* const* src, void* const* dst, const int* H,
                          const int* h0, const int* count, int n_jobs, int B, int64_t S, int D,
                          cudaStream_t stream) {
  const int Dc = D / 8;
  if (Dc != 8 && Dc != 16) return cudaErrorInvalidValue;
  LayoutJobs J{};
  J.n_jobs = n_jobs;
  J.lg_dc = Dc == 16 ? 4 : 3;
  J.rows = kBlockVecs / Dc;
  const int64_t sb = (S + J.rows - 1) / J.rows;
  if (sb > (int64_t(1) << 30)) return cudaErrorInvalidValue;
  J.seq_blocks = static_cast<int>(sb);
  int64_t total = 0;
  for (int j = 0; j < n_jobs; ++j) {
    J.src[j] = static_cast<const uint4*>(src[j]);
    J.dst[j] = static_cast<uint4*>(dst[j]);
    J.H[j] = H[j];
    J.h0[j] = h0[j];
    J.count[j] = count[j];
    J.first_block[j] = static_cast<int>(total);
    total += sb * B * count[j];
    if (total > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  }
  J.first_block[n_jobs] = static_cast<int>(total);
  if (total == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(total);
  launch_begin(0, stream);
  if (to_head)
    layout_kernel<true><<<grid, kLayoutThreads, 0, stream>>>(J, S);
  else
    layout_kernel<false><<<grid, kLayoutThreads, 0, stream>>>(J, S);
  cudaError_t e = cudaGetLastError();
  launch_end(0, stream);
  return e;
}

// The backward pre-pass. A block covers kPreRows sequence positions of one (batch, head) of
// the group (grid: position blocks x hc x B); one group of Dc = D/8 consecutive lanes handles
// one position, so the row reduction stays inside a warp (Dc is 8 or 16). o and dout are
// token-major [B,S,Hq,D] (dout is gathered into dow on the way), or, with head_major_in, this
// group's head-major [B*hc][S][D] copies (dout then already is dow, which is not written).
constexpr int kPreRows = 64;

__global__ void __launch_bounds__(kLayoutThreads)
    bwd_pre_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                   const float* __restrict__ lse, uint4* __restrict__ dow,
                   float* __restrict__ dvec, float* __restrict__ lse2,
                   float4* __restrict__ dqacc, int64_t S, int64_t S_pad, int Hq, int Dc, int h0,
                   int hc, float scale, int head_major_in) {
  const int h = blockIdx.y, b = blockIdx.z;
  const int per_pass = kLayoutThreads / Dc;  // positions per pass of the block
  const int c = static_cast<int>(threadIdx.x) % Dc;
  const int64_t zbase = (static_cast<int64_t>(b) * hc + h) * S_pad;  // dvec / lse2 / dqacc rows
  const float kLog2e = 1.4426950408889634f;
  // S_pad is a multiple of 128 and the grid covers it exactly, so every lane of a warp runs
  // every pass (the shuffles below need all 32).
  for (int r = static_cast<int>(threadIdx.x) / Dc; r < kPreRows; r += per_pass) {
    const int64_t s = static_cast<int64_t>(blockIdx.x) * kPreRows + r;
    float dot = 0.f;
    if (s < S) {
      const int64_t hm = ((static_cast<int64_t>(b) * hc + h) * S + s) * Dc + c;
      const int64_t tok =
          head_major_in ? hm : ((static_cast<int64_t>(b) * S + s) * Hq + h0 + h) * Dc + c;
      const uint4 ov = __ldg(o + tok);
      const uint4 dv = __ldg(dout + tok);
      if (!head_major_in) dow[hm] = dv;
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(o2[i]);
        const float2 g = __bfloat1622float2(d2[i]);
        dot = fmaf(a.x, g.x, dot);
        dot = fmaf(a.y, g.y, dot);
      }
    }
    // zero this chunk's share of the dQ accumulator row (D floats = 2*Dc float4)
    const int64_t zrow = zbase + s;
    dqacc[zrow * 2 * Dc + 2 * c] = make_float4(0.f, 0.f, 0.f, 0.f);
    dqacc[zrow * 2 * Dc + 2 * c + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int off = Dc / 2; off > 0; off >>= 1)
      dot += __shfl_xor_sync(0xffffffffu, dot, off, Dc);
    if (c == 0) {
      dvec[zrow] = (s < S) ? -(dot * scale) : 0.f;
      lse2[zrow] =
          (s < S) ? -(lse[(static_cast<int64_t>(b) * Hq + h0 + h) * S + s] * kLog2e) : 0.f;
    }
  }
}

// dq rows hold out_heads heads; this group's go to heads [out_head0, out_head0 + hc): the
// token-major [B,S,Hq,D] output (Hq, h0) or a group staging [B,S,hc,D] (hc, 0). A block covers
// kConvRows positions of one (batch, head) (grid: position blocks x hc x B).
constexpr int kConvRows = 128;

__global__ void __launch_bounds__(kLayoutThreads)
    dq_convert_kernel(const float4* __restrict__ dqacc, uint4* __restrict__ dq, int64_t S,
                      int64_t S_pad, int out_heads, int Dc, int out_head0, int hc) {
  const int h = blockIdx.y, b = blockIdx.z;
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kConvRows;
  const int64_t zbase = (static_cast<int64_t>(b) * hc + h) * S_pad + s0;
  const int64_t obase = (static_cast<int64_t>(b) * S + s0) * out_heads + out_head0 + h;
  const int n = static_cast<int>((S - s0 < kConvRows ? S - s0 : kConvRows) * Dc);
  for (int i = static_cast<int>(threadIdx.x); i < n; i += kLayoutThreads) {
    const int r = i / Dc, c = i - r * Dc;
    const int64_t z = (zbase + r) * 2 * Dc + 2 * c;
    const float4 x = dqacc[z];
    const float4 y = dqacc[z + 1];
    __nv_bfloat162 w[4] = {__floats2bfloat162_rn(x.x, x.y), __floats2bfloat162_rn(x.z, x.w),
                           __floats2bfloat162_rn(y.x, y.y), __floats2bfloat162_rn(y.z, y.w)};
    dq[(obase + static_cast<int64_t>(r) * out_heads) * Dc + c] =
        *reinterpret_cast<const uint4*>(w);
  }
}

// Split backward: the shares of `split` CTAs per key tile, added in a fixed order. One thread
// per 16-byte output vector (8 bf16 of dK or dV); a block covers kRedRows key rows of one
// (batch, kv-head) (grid: row blocks x kc x B).
constexpr int kRedRows = 64;

__global__ void __launch_bounds__(kLayoutThreads)
    dkdv_reduce_kernel(const float4* __restrict__ part, int split, int64_t part_rows,
                       int64_t rows, int64_t row0_pos, int B, int kc, int Dc, int64_t S,
                       uint4* __restrict__ dk, uint4* __restrict__ dv, int64_t dkv_rows,
                       int64_t dkv_row0, int dkv_heads, int dkv_head0) {
  const int kvl = blockIdx.y, b = blockIdx.z;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kRedRows;
  const int per_row = 2 * Dc;  // dK's Dc vectors, then dV's
  const int n = static_cast<int>((rows - r0 < kRedRows ? rows - r0 : kRedRows) * per_row);
  const int64_t slot = static_cast<int64_t>(B) * kc * part_rows * 2 * Dc * 2;  // float4s
  for (int i = static_cast<int>(threadIdx.x); i < n; i += kLayoutThreads) {
    const int rr = i / per_row, v = i - rr * per_row;
    const int64_t r = r0 + rr;
    const int64_t pos = row0_pos + r;
    if (pos >= S) continue;
    // float4 index of the share's 8 floats: row (b, kvl, r), vector v of its 2D floats
    const int64_t f = ((static_cast<int64_t>(b) * kc + kvl) * part_rows + r) * (4 * Dc) + 2 * v;
    float4 x = part[f], y = part[f + 1];
    for (int sp = 1; sp < split; ++sp) {
      const float4 x2 = part[sp * slot + f], y2 = part[sp * slot + f + 1];
      x.x += x2.x; x.y += x2.y; x.z += x2.z; x.w += x2.w;
      y.x += y2.x; y.y += y2.y; y.z += y2.z; y.w += y2.w;
    }
    __nv_bfloat162 o[4] = {__floats2bfloat162_rn(x.x, x.y), __floats2bfloat162_rn(x.z, x.w),
                           __floats2bfloat162_rn(y.x, y.y), __floats2bfloat162_rn(y.z, y.w)};
    const bool is_v = v >= Dc;
    const int c = is_v ? v - Dc : v;
    uint4* out = is_v ? dv : dk;
    out[((static_cast<int64_t>(b) * dkv_rows + pos - dkv_row0) * dkv_heads + dkv_head0 + kvl) *
            Dc + c] = *reinterpret_cast<const uint4*>(o);
  }
}

}  // namespace

cudaError_t launch_seq_to_head(const void* src, void* dst, int B, int64_t S, int H, int D,
                               int h_begin, int h_count, cudaStream_t stream) {
  return launch_layout(true, &src, &dst, &H, &h_begin, &h_count, 1, B, S, D, stream);
}

cudaError_t launch_gather_group(const void* const* src, void* const* dst, const int* H,
                                const int* h0, const int* count, int n, int B, int64_t S, int D,
                                cudaStream_t stream) {
  if (n < 1 || n > 3) return cudaErrorInvalidValue;
  return launch_layout(true, src, dst, H, h0, count, n, B, S, D, stream);
}

cudaError_t launch_head_to_seq(const void* src, void* dst, int B, int64_t S, int H, int D,
                               int h_begin, int h_count, cudaStream_t stream) {
  void* dsts[1] = {dst};
  const void* srcs[1] = {src};
  // the same job description, read the other way: head-major source, token-major destination
  return launch_layout(false, srcs, dsts, &H, &h_begin, &h_count, 1, B, S, D, stream);
}

cudaError_t launch_bwd_pre(const void* o, const void* dout, const float* lse, void* dow,
                           float* dvec, float* lse2, float* dqacc, int B, int64_t S,
                           int64_t S_pad, int Hq, int D, int h0, int hc, float scale,
                           int head_major_in, cudaStream_t stream) {
  const int Dc = D / 8;
  const dim3 grid(static_cast<unsigned>((S_pad + kPreRows - 1) / kPreRows),
                  static_cast<unsigned>(hc), static_cast<unsigned>(B));
  launch_begin(2, stream);
  bwd_pre_kernel<<<grid, kLayoutThreads, 0, stream>>>(
      static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse,
      static_cast<uint4*>(dow), dvec, lse2, reinterpret_cast<float4*>(dqacc), S, S_pad, Hq, Dc,
      h0, hc, scale, head_major_in);
  cudaError_t e = cudaGetLastError();
  launch_end(2, stream);
  return e;
}

cudaError_t launch_dq_convert(const float* dqacc, void* dq, int B, int64_t S, int64_t S_pad,
                              int out_heads, int D, int out_head0, int hc, cudaStream_t stream) {
  const int Dc = D / 8;
  const dim3 grid(static_cast<unsigned>((S + kConvRows - 1) / kConvRows),
                  static_cast<unsigned>(hc), static_cast<unsigned>(B));
  launch_begin(4, stream);
  dq_convert_kernel<<<grid, kLayoutThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(dqacc), static_cast<uint4*>(dq), S, S_pad, out_heads, Dc,
      out_head0, hc);
  cudaError_t e = cudaGetLastError();
  launch_end(4, stream);
  return e;
}

cudaError_t launch_dkdv_reduce(const float* part, int split, int64_t part_rows, int64_t rows,
                               int64_t row0_pos, int B, int kc, int D, int64_t S, void* dk,
                               void* dv, int64_t dkv_rows, int64_t dkv_row0, int dkv_heads,
                               int dkv_head0, cudaStream_t stream) {
  const int Dc = D / 8;
  const dim3 grid(static_cast<unsigned>((rows + kRedRows - 1) / kRedRows),
                  static_cast<unsigned>(kc), static_cast<unsigned>(B));
  launch_begin(4, stream);
  dkdv_reduce_kernel<<<grid, kLayoutThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(part), split, part_rows, rows, row0_pos, B, kc, Dc, S,
      static_cast<uint4*>(dk), static_cast<uint4*>(dv), dkv_rows, dkv_row0, dkv_heads,
      dkv_head0);
  cudaError_t e = cudaGetLastError();
  launch_end(4, stream);
  return e;
}

}  // namespace upipe
