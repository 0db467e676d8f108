// E4M3 block quantization for the FP8 forward (triton-tutorial "8. FlashAttention 实战",
// §8.9.4: one scale per 128-row block of Q, K or V; scale = max|x| / 448, E4M3's largest
// finite value).  One CTA per (block, b*h): it finds the block's max |x|, writes the scale and
// the codes round(x / scale) (nearest, ties to even, saturating).  The scale and the division
// are IEEE fp32 operations (they decide byte codes).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int kBlockRows = 128;
constexpr int kThreads = 256;

template <int D>
__global__ void __launch_bounds__(kThreads) quant_e4m3_kernel(const __nv_bfloat16* __restrict__ x,
                                                              uint8_t* __restrict__ codes, float* __restrict__ scales,
                                                              int N) {
  constexpr int kVec = 8;                               // bf16 per 16-byte load
  constexpr int kPerRow = D / kVec;
  const int nb = (N + kBlockRows - 1) / kBlockRows;
  const int blk = static_cast<int>(blockIdx.x) % nb, bh = static_cast<int>(blockIdx.x) / nb;
  const int r0 = blk * kBlockRows;
  const int rows = min(kBlockRows, N - r0);
  const size_t base = (static_cast<size_t>(bh) * N + r0) * D;
  const int n_vec = rows * kPerRow;
  __shared__ float red[kThreads / 32];
  float amax = 0.f;
  for (int i = threadIdx.x; i < n_vec; i += kThreads) {
    const uint4 v = reinterpret_cast<const uint4*>(x + base)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(w[k])), fabsf(bf16hi(w[k]))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (threadIdx.x == 0) scales[blockIdx.x] = sc;  // = scales[bh][blk]
  for (int i = threadIdx.x; i < n_vec; i += kThreads) {
    const uint4 v = reinterpret_cast<const uint4*>(x + base)[i];
    uint2 out;
    out.x = pack_e4m3x4(__fdiv_rn(bf16lo(v.x), sc), __fdiv_rn(bf16hi(v.x), sc), __fdiv_rn(bf16lo(v.y), sc),
                        __fdiv_rn(bf16hi(v.y), sc));
    out.y = pack_e4m3x4(__fdiv_rn(bf16lo(v.z), sc), __fdiv_rn(bf16hi(v.z), sc), __fdiv_rn(bf16lo(v.w), sc),
                        __fdiv_rn(bf16hi(v.w), sc));
    reinterpret_cast<uint2*>(codes + base)[i] = out;
  }
}

}  // namespace

cudaError_t launch_quant_e4m3(const void* x, void* codes, float* scales, int BH, int N, int d, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(BH) * static_cast<unsigned>((N + kBlockRows - 1) / kBlockRows);
  if (d == 64)
    quant_e4m3_kernel<64><<<grid, kThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                         static_cast<uint8_t*>(codes), scales, N);
  else
    quant_e4m3_kernel<128><<<grid, kThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                          static_cast<uint8_t*>(codes), scales, N);
  return cudaGetLastError();
}

}  // namespace fattn
