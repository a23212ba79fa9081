// HBM-bound kernels around the attention kernels:
//   * seq_to_head_major / head_to_seq_major: the single-GPU stand-in for DeepSpeed Ulysses'
//     head<->sequence all-to-all, which gathers the whole sequence for a subset of heads
//     ("Training Ultra Long Context LM with Fully Pipelined Distributed Transformer",
//     Technical Deep Dive, first paragraph). Here it copies one head group of a token-major
//     [B,S,H,D] tensor into a head-major [B,h,S,D] workspace (and back).
//   * the backward pre-pass: scale * D_i, D_i = <dO_i, O_i> in fp32, the dO gather, the LSE prescale by
//     log2(e) and the zeroing of the fp32 dQ accumulator, fused in one pass;
//   * the dQ conversion: fp32 accumulator -> bf16 token-major dq.
// Each thread moves 16-byte vectors; grids are sized as a multiple of the SM count and loop.
#include <cuda_bf16.h>

#include "internal.h"

namespace upipe {
namespace {

constexpr int kLayoutThreads = 256;

inline unsigned grid_for(int64_t work, int threads) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sms = v;
  }
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

// One work item = one 16-byte chunk (8 bf16). Items are ordered (b, s, h, chunk) so that the
// token-major side is read/written contiguously.
__global__ void seq_to_head_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int B,
                                   int64_t S, int H, int Dc, int h_begin, int h_count) {
  const int64_t total = static_cast<int64_t>(B) * S * h_count * Dc;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % Dc);
    int64_t r = idx / Dc;
    const int h = static_cast<int>(r % h_count);
    r /= h_count;
    const int64_t s = r % S;
    const int64_t b = r / S;
    const uint4 v = __ldg(src + ((b * S + s) * H + h_begin + h) * Dc + c);
    dst[((b * h_count + h) * S + s) * Dc + c] = v;
  }
}

__global__ void head_to_seq_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int B,
                                   int64_t S, int H, int Dc, int h_begin, int h_count) {
  const int64_t total = static_cast<int64_t>(B) * S * h_count * Dc;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % Dc);
    int64_t r = idx / Dc;
    const int h = static_cast<int>(r % h_count);
    r /= h_count;
    const int64_t s = r % S;
    const int64_t b = r / S;
    dst[((b * S + s) * H + h_begin + h) * Dc + c] = __ldg(src + ((b * h_count + h) * S + s) * Dc + c);
  }
}

// One group of Dc = D/8 consecutive lanes handles one (b, s, h) row; Dc is 8 or 16 and
// divides the warp, so the row reduction stays inside a warp. o and dout are token-major
// [B,S,Hq,D] (dout is gathered into dow on the way), or, with head_major_in, this group's
// head-major [B*hc][S][D] copies (dout then already is dow, which is not written).
__global__ void bwd_pre_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                               const float* __restrict__ lse, uint4* __restrict__ dow,
                               float* __restrict__ dvec, float* __restrict__ lse2,
                               float4* __restrict__ dqacc, int B, int64_t S, int64_t S_pad, int Hq,
                               int Dc, int h0, int hc, float scale, int head_major_in) {
  const int64_t rows = static_cast<int64_t>(B) * S_pad * hc;
  const int64_t total = rows * Dc;
  const float kLog2e = 1.4426950408889634f;
  for (int64_t base = blockIdx.x * static_cast<int64_t>(blockDim.x);
       base < total; base += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t idx = base + threadIdx.x;
    const bool live = idx < total;
    const int c = static_cast<int>(idx % Dc);
    int64_t r = idx / Dc;
    const int h = static_cast<int>(r % hc);
    r /= hc;
    const int64_t s = r % S_pad;
    const int64_t b = r / S_pad;
    float dot = 0.f;
    const int64_t zrow = (b * hc + h) * S_pad + s;  // row of dvec / lse2 / dqacc
    if (live) {
      if (s < S) {
        const int64_t hm = ((b * hc + h) * S + s) * Dc + c;
        const int64_t tok = head_major_in ? hm : ((b * S + s) * Hq + h0 + h) * Dc + c;
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
      dqacc[zrow * 2 * Dc + 2 * c] = make_float4(0.f, 0.f, 0.f, 0.f);
      dqacc[zrow * 2 * Dc + 2 * c + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int off = Dc / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (live && c == 0) {
      dvec[zrow] = (s < S) ? -(dot * scale) : 0.f;
      lse2[zrow] = (s < S) ? -(lse[(b * Hq + h0 + h) * S + s] * kLog2e) : 0.f;
    }
  }
}

// dq rows hold out_heads heads; this group's go to heads [out_head0, out_head0 + hc): the
// token-major [B,S,Hq,D] output (Hq, h0) or a group staging [B,S,hc,D] (hc, 0).
__global__ void dq_convert_kernel(const float4* __restrict__ dqacc, uint4* __restrict__ dq, int B,
                                  int64_t S, int64_t S_pad, int out_heads, int Dc, int out_head0,
                                  int hc) {
  const int64_t total = static_cast<int64_t>(B) * S * hc * Dc;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % Dc);
    int64_t r = idx / Dc;
    const int h = static_cast<int>(r % hc);
    r /= hc;
    const int64_t s = r % S;
    const int64_t b = r / S;
    const int64_t zrow = (b * hc + h) * S_pad + s;
    const float4 x = dqacc[zrow * 2 * Dc + 2 * c];
    const float4 y = dqacc[zrow * 2 * Dc + 2 * c + 1];
    __nv_bfloat162 w[4] = {__floats2bfloat162_rn(x.x, x.y), __floats2bfloat162_rn(x.z, x.w),
                           __floats2bfloat162_rn(y.x, y.y), __floats2bfloat162_rn(y.z, y.w)};
    dq[((b * S + s) * out_heads + out_head0 + h) * Dc + c] = *reinterpret_cast<const uint4*>(w);
  }
}

}  // namespace

cudaError_t launch_seq_to_head(const void* src, void* dst, int B, int64_t S, int H, int D,
                               int h_begin, int h_count, cudaStream_t stream) {
  const int Dc = D / 8;
  const int64_t work = static_cast<int64_t>(B) * S * h_count * Dc;
  launch_begin(0, stream);
  seq_to_head_kernel<<<grid_for(work, kLayoutThreads), kLayoutThreads, 0, stream>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), B, S, H, Dc, h_begin, h_count);
  cudaError_t e = cudaGetLastError();
  launch_end(0, stream);
  return e;
}

cudaError_t launch_head_to_seq(const void* src, void* dst, int B, int64_t S, int H, int D,
                               int h_begin, int h_count, cudaStream_t stream) {
  const int Dc = D / 8;
  const int64_t work = static_cast<int64_t>(B) * S * h_count * Dc;
  launch_begin(0, stream);
  head_to_seq_kernel<<<grid_for(work, kLayoutThreads), kLayoutThreads, 0, stream>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), B, S, H, Dc, h_begin, h_count);
  cudaError_t e = cudaGetLastError();
  launch_end(0, stream);
  return e;
}

cudaError_t launch_bwd_pre(const void* o, const void* dout, const float* lse, void* dow,
                           float* dvec, float* lse2, float* dqacc, int B, int64_t S,
                           int64_t S_pad, int Hq, int D, int h0, int hc, float scale,
                           int head_major_in, cudaStream_t stream) {
  const int Dc = D / 8;
  const int64_t work = static_cast<int64_t>(B) * S_pad * hc * Dc;
  launch_begin(2, stream);
  bwd_pre_kernel<<<grid_for(work, kLayoutThreads), kLayoutThreads, 0, stream>>>(
      static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse,
      static_cast<uint4*>(dow), dvec, lse2, reinterpret_cast<float4*>(dqacc), B, S, S_pad, Hq, Dc,
      h0, hc, scale, head_major_in);
  cudaError_t e = cudaGetLastError();
  launch_end(2, stream);
  return e;
}

cudaError_t launch_dq_convert(const float* dqacc, void* dq, int B, int64_t S, int64_t S_pad,
                              int out_heads, int D, int out_head0, int hc, cudaStream_t stream) {
  const int Dc = D / 8;
  const int64_t work = static_cast<int64_t>(B) * S * hc * Dc;
  launch_begin(4, stream);
  dq_convert_kernel<<<grid_for(work, kLayoutThreads), kLayoutThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(dqacc), static_cast<uint4*>(dq), B, S, S_pad, out_heads, Dc,
      out_head0, hc);
  cudaError_t e = cudaGetLastError();
  launch_end(4, stream);
  return e;
}

}  // namespace upipe
