// Output tiles leave the CTA through shared memory and one TMA tile store per 128-row x 128-byte
// box, instead of each thread writing its half row straight to global memory (16-byte stores
// that touch a different row in every lane).
#pragma once
#include <cstdint>

#include "ptx.cuh"
#include "tmem_io.cuh"

namespace fattn {

// This thread's half of row r of a 128-row fp32 tile in TMEM (D/2 columns from taddr: columns
// 32h .. at D = 64, 64h .. at D = 128), times `mult`, as bf16 into the staged tile.  The tile is
// D/64 boxes (at box0, box1) of 128 rows x 128 bytes with the 128-byte swizzle of the tensor
// maps (16-byte chunk c of row r at chunk c ^ (r & 7)): the thread's chunks are 4h .. 4h + 3 of
// the one box at D = 64 and all 8 chunks of box h at D = 128.  Every lane must call it (the TMEM
// load is warp-collective).  Ends with the proxy fence the TMA store's read needs.
template <int D>
__device__ __forceinline__ void stage_half_row_bf16(uint32_t box0, uint32_t box1, int r, int h, uint32_t taddr,
                                                    float mult) {
  static_assert(D == 64 || D == 128, "d = 64 or 128");
  uint32_t ur[D / 2];
  if constexpr (D == 128) tmem_ld2_x64<64>(taddr, ur); else tmem_ld2_x32<32>(taddr, ur);
  const uint32_t srow = (D == 128 && h ? box1 : box0) + static_cast<uint32_t>(r) * 128u;
  const int c0 = D == 128 ? 0 : 4 * h;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    const uint32_t* u = ur + 8 * i;
    sts128(srow + ((static_cast<uint32_t>(c0 + i) ^ static_cast<uint32_t>(r & 7)) << 4),
           pack_bf16(__uint_as_float(u[0]) * mult, __uint_as_float(u[1]) * mult),
           pack_bf16(__uint_as_float(u[2]) * mult, __uint_as_float(u[3]) * mult),
           pack_bf16(__uint_as_float(u[4]) * mult, __uint_as_float(u[5]) * mult),
           pack_bf16(__uint_as_float(u[6]) * mult, __uint_as_float(u[7]) * mult));
  }
  fence_proxy_async_smem();  // the TMA store reads the staging through the async proxy
}

}  // namespace fattn
