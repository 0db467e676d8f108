// Attention backward for sm_103a: gradients dQ, dK, dV from Q, K, V, O, dO and
// the forward's lse, recomputing P blockwise instead of storing it
// (triton-tutorial "8. FlashAttention 实战", §8.8.2-§8.8.4; operatorworld
// "反向传播：用重算换显存"; xuesongtap.github.io "flash-attention", §3).
//
//   D_i    = rowsum(O_i * dO_i)                                   bwd_delta_kernel
//   P_ij   = exp(S_ij * scale - lse_i)      S = Q K^T (recomputed)
//   dP_ij  = dO_i V_j^T
//   dS_ij  = P_ij (dP_ij - D_i)
//   dV_j  += P_ij^T dO_i,   dK_j += scale dS_ij^T Q_i             bwd_dkdv_kernel (one CTA per key tile)
//   dQ_i  += scale dS_ij K_j                                      bwd_dq_kernel   (one CTA per query tile)
// Two passes instead of atomics on dQ: the tutorial's two-phase kernel
// (§8.8.4) splits the same way; every output tile has one owner.
//
// Both main kernels keep their own tile resident in shared memory, stream the
// other side through a TMA ring, compute the two products of a step with
// tcgen05.mma into TMEM, let the elementwise warps (one thread per row at
// d = 128, two at d = 64) turn them into bf16 P^T and dS^T (or dS) in TMEM,
// chunk by chunk, and accumulate the gradient MMAs (A operand from TMEM) into
// TMEM, each chunk's as soon as it is ready.  The gradient
// MMAs of step i and the products of step i+1 are issued back to back; the
// tensor core runs them in order, so the products may overwrite the TMEM
// columns the gradient MMAs read.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "stage_io.cuh"
#include "tmem_io.cuh"

namespace fattn {

__device__ unsigned int g_bwd_status = 0;

namespace {

constexpr int kTile = 128;                // rows per tile on either side
constexpr uint32_t kBox = 128u * 128u;    // bytes of a 128-row x 64-column bf16 box
constexpr uint32_t kTmemCols = 512;
// Elementwise warps of the dK/dV and dQ kernels: at d = 128 one thread per (key or query) row (4
// warps, .32x32b TMEM access, the row's 128 columns in four chunks of 32); at d = 64 8 warps, two
// threads a row (.16x32bx2, two chunks; the dK/dV kernel takes each query tile in two halves).
template <int D>
struct BwdWarps {
  static constexpr bool ONE = D == 128;
  static constexpr int EW = ONE ? 4 : 8;
  static constexpr int CHUNKS = ONE ? 4 : 2;
  static constexpr int MMA = EW, TMA = EW + 1, THREADS = (EW + 2) * 32;
};
constexpr uint32_t kColA = 0, kColB = 128, kColG1 = 256;  // products at 0 / 128, gradients from 256
constexpr uint32_t kColS1 = 384;  // dQ kernel: second S buffer (S(j) at kColA for even j, here for odd j)
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      unsigned long long budget) {
  return mbar_wait(bar, parity, abort_flag, budget, &g_bwd_status);
}
__device__ __forceinline__ bool bwait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long budget) {
  return __all_sync(0xffffffffu, bwait(bar, parity, abort_flag, budget));
}
__device__ __forceinline__ void bdrain(uint32_t bar, uint32_t parity, unsigned long long budget) {
  if (budget < kDrainBudget) budget = kDrainBudget;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<unsigned long long>(clock64() - t0) > budget) {
      atomicOr(&g_bwd_status, kStatusTimeout);
      return;
    }
  }
}

__device__ __forceinline__ void tmem_st1_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                  "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
}

// --------------------------------------------------------------------- D = rowsum(O * dO)
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta, long long rows) {
  constexpr int TPR = D / 8;  // threads per row, 8 elements (16 bytes) each
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = gt / TPR;
  const int part = static_cast<int>(gt % TPR);
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = reinterpret_cast<const uint4*>(o + row * D)[part];
    const uint4 b = reinterpret_cast<const uint4*>(dout + row * D)[part];
    acc = fmaf(bf16lo(a.x), bf16lo(b.x), acc);
    acc = fmaf(bf16hi(a.x), bf16hi(b.x), acc);
    acc = fmaf(bf16lo(a.y), bf16lo(b.y), acc);
    acc = fmaf(bf16hi(a.y), bf16hi(b.y), acc);
    acc = fmaf(bf16lo(a.z), bf16lo(b.z), acc);
    acc = fmaf(bf16hi(a.z), bf16hi(b.z), acc);
    acc = fmaf(bf16lo(a.w), bf16lo(b.w), acc);
    acc = fmaf(bf16hi(a.w), bf16hi(b.w), acc);
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) delta[row] = acc;
}

// --------------------------------------------------------------------- shared pieces
template <int D>
struct BwdCfg {
  static constexpr int NH = D / 64;
  static constexpr uint32_t TB = NH * kBox;   // bytes of one 128 x d bf16 tile
  static constexpr int ST = (D == 128) ? 2 : 4;
  static constexpr uint32_t VEC = 2 * kTile * 4;  // per stage (dkdv only): {-lse2, -D} of 128 rows, see OFF_VEC
  static constexpr uint32_t COL_G2 = kColG1 + D;  // second gradient accumulator (dK)
};

// Gradient tile (TMEM, fp32, D columns) * scale -> global rows < N (bf16 or fp32), this thread's half row.
template <int D>
__device__ __forceinline__ void store_grad_half_row(void* out, size_t row_off, int h, bool valid, bool fp32,
                                                    uint32_t taddr, float scale) {
  uint32_t ur[D / 2];
  if constexpr (D == 128) tmem_ld2_x64<64>(taddr, ur); else tmem_ld2_x32<32>(taddr, ur);
  if (!valid) return;
  if (fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row_off * D + h * (D / 2));
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      dst[i] = make_float4(__uint_as_float(ur[4 * i]) * scale, __uint_as_float(ur[4 * i + 1]) * scale,
                           __uint_as_float(ur[4 * i + 2]) * scale, __uint_as_float(ur[4 * i + 3]) * scale);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row_off * D + h * (D / 2));
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      uint4 w;
      w.x = pack_bf16(__uint_as_float(ur[8 * i + 0]) * scale, __uint_as_float(ur[8 * i + 1]) * scale);
      w.y = pack_bf16(__uint_as_float(ur[8 * i + 2]) * scale, __uint_as_float(ur[8 * i + 3]) * scale);
      w.z = pack_bf16(__uint_as_float(ur[8 * i + 4]) * scale, __uint_as_float(ur[8 * i + 5]) * scale);
      w.w = pack_bf16(__uint_as_float(ur[8 * i + 6]) * scale, __uint_as_float(ur[8 * i + 7]) * scale);
      dst[i] = w;
    }
  }
}

// d = 128, one thread per row: a 128-column fp32 tile row in TMEM * scale -> global (fp32), or as
// bf16 into the staged tile (box0: columns 0..63, box1: 64..127, 128-byte swizzle).
__device__ __forceinline__ void store_grad_row128(void* out, size_t row_off, bool valid, uint32_t taddr, float scale) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t ur[64];
    tmem_ld_x64(taddr + 64u * half, ur);
    if (!valid) continue;
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row_off * 128 + 64 * half);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      dst[i] = make_float4(__uint_as_float(ur[4 * i]) * scale, __uint_as_float(ur[4 * i + 1]) * scale,
                           __uint_as_float(ur[4 * i + 2]) * scale, __uint_as_float(ur[4 * i + 3]) * scale);
  }
}
__device__ __forceinline__ void stage_row128_bf16(uint32_t box0, uint32_t box1, int r, uint32_t taddr, float scale) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t ur[64];
    tmem_ld_x64(taddr + 64u * half, ur);
    const uint32_t srow = (half ? box1 : box0) + static_cast<uint32_t>(r) * 128u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t* u = ur + 8 * i;
      sts128(srow + ((static_cast<uint32_t>(i) ^ static_cast<uint32_t>(r & 7)) << 4),
             pack_bf16(__uint_as_float(u[0]) * scale, __uint_as_float(u[1]) * scale),
             pack_bf16(__uint_as_float(u[2]) * scale, __uint_as_float(u[3]) * scale),
             pack_bf16(__uint_as_float(u[4]) * scale, __uint_as_float(u[5]) * scale),
             pack_bf16(__uint_as_float(u[6]) * scale, __uint_as_float(u[7]) * scale));
    }
  }
  fence_proxy_async_smem();
}

// S = A B^T into TMEM: A and B are resident/streamed 128 x d K-major tiles.
template <int D>
__device__ __forceinline__ void issue_product(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>(kk >> 2) * kBox + static_cast<uint32_t>(kk & 3) * 32u;
    if (kk == 0) mma_ss_c<0>(d_tmem, sdesc_add(da, off), sdesc_add(db, off), idesc);
    else mma_ss_c<1>(d_tmem, sdesc_add(da, off), sdesc_add(db, off), idesc);
  }
}
// Packed bf16 operands in TMEM keep each half of the 128-wide K dimension in its own half of
// the 128 columns it was computed in: elements 0..63 at packed columns 0..31, elements 64..127 at
// 64..95.  The elementwise threads that produce a half then only overwrite columns they have
// already read.  Column of the k-th 16-element K block:
__device__ __forceinline__ uint32_t packed_col(int kk) { return kk < 4 ? 8u * kk : 64u + 8u * (kk - 4); }

// G (+)= X Y with X (128 x 128) packed bf16 in TMEM (layout above) and Y a 128 x d MN-major
// tile, half at a time: the K blocks that the elementwise threads' chunk `part` produced (chunk c
// of the thread holding elements 64h.. writes elements 64h + 32c .. +31, i.e. K blocks
// {0, 1, 4, 5} for c = 0 and {2, 3, 6, 7} for c = 1), so the MMAs of the first chunk run while
// the second is computed.
template <int D>
__device__ __forceinline__ void issue_grad_part(uint32_t d_tmem, uint32_t a_tmem, uint64_t db, uint32_t idesc,
                                                bool accumulate, int part) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int kk = 2 * part + (q & 1) + 4 * (q >> 1);
    const uint32_t a = a_tmem + packed_col(kk);
    const uint64_t b = sdesc_add(db, static_cast<uint32_t>(kk) * 2048u);
    if (q == 0 && !accumulate) mma_ts_c<0>(d_tmem, a, b, idesc);
    else mma_ts_c<1>(d_tmem, a, b, idesc);
  }
}

// G (+)= X Y for chunk c of the one-thread-per-row kernels (d = 128: dK, dV from P^T, dS^T; dQ from
// dS): K blocks 2c, 2c + 1, packed at columns 8kk (each thread packs its chunk c into columns
// 16c .., which it has read).
__device__ __forceinline__ void issue_grad_chunk(uint32_t d_tmem, uint32_t a_tmem, uint64_t db, uint32_t idesc,
                                                 bool accumulate, int c) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int kk = 2 * c + q;
    const uint32_t a = a_tmem + 8u * static_cast<uint32_t>(kk);
    const uint64_t b = sdesc_add(db, static_cast<uint32_t>(kk) * 2048u);
    if (q == 0 && !accumulate) mma_ts_c<0>(d_tmem, a, b, idesc);
    else mma_ts_c<1>(d_tmem, a, b, idesc);
  }
}

// G (+)= X_q Y_q for query half q of the dK/dV kernel: X_q is the packed bf16 half of the 128 x
// 128 TMEM tile (columns 64q .. 64q + 63; the thread holding queries 64q + 32h .. writes them
// packed at columns 64q + 32h .. + 15, so K block 4q + m, m < 2 from h = 0 and m >= 2 from
// h = 1, is at column 64q + 32(m / 2) + 8(m % 2)), Y_q rows 64q .. 64q + 63 of a 128 x d MN-major
// tile.  Four MMAs of 16 queries each.
template <int D>
__device__ __forceinline__ void issue_grad_half(uint32_t d_tmem, uint32_t a_tmem, uint64_t db, uint32_t idesc,
                                                bool accumulate, int q) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int kk = 4 * q + m;
    const uint32_t a = a_tmem + 64u * q + 32u * (m >> 1) + 8u * (m & 1);
    const uint64_t b = sdesc_add(db, static_cast<uint32_t>(kk) * 2048u);
    if (m == 0 && !accumulate) mma_ts_c<0>(d_tmem, a, b, idesc);
    else mma_ts_c<1>(d_tmem, a, b, idesc);
  }
}

// Elementwise step of the dK/dV kernel on 32 query columns of one key row (column pairs packed
// as f32x2): P^T = 2^(S^T c - lse2), dS^T = P^T (dP^T - D), both rounded to bf16 pairs.  MASK
// (the diagonal tile only) zeroes P^T where the query precedes the key.
template <bool MASK>
__device__ __forceinline__ void ew_pairs_dkdv(const uint32_t (&sv)[32], const uint32_t (&pv)[32], const float4* nv,
                                              uint64_t c2, int col0, int qrow0, int key, uint32_t (&pp)[16],
                                              uint32_t (&dp)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const int col = col0 + e;  // query row within the tile
    const float4 x = nv[col >> 1];
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, f2_pack(x.x, x.y)), x0, x1);
    float p0 = ex2(x0), p1 = ex2(x1);
    if (MASK) {
      if (qrow0 + col < key) p0 = 0.f;
      if (qrow0 + col + 1 < key) p1 = 0.f;
    }
    const uint64_t p2 = f2_pack(p0, p1);
    float s0, s1;
    f2_unpack(f2_mul(p2, f2_add(f2_pack(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), f2_pack(x.z, x.w))),
              s0, s1);
    pp[e / 2] = pack_bf16(p0, p1);
    dp[e / 2] = pack_bf16(s0, s1);
  }
}

// Elementwise step of the dQ kernel on 32 key columns of one query row: dS = P (dP - D) with
// P = 2^(S c - lse2), rounded to bf16 pairs.  MASK zeroes keys past the row's last key.
template <bool MASK>
__device__ __forceinline__ void ew_pairs_dq(const uint32_t (&sv)[32], const uint32_t (&pv)[32], uint64_t c2,
                                            uint64_t nl2, uint64_t nd2, int key0, int lim, uint32_t (&dp)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nl2), x0, x1);
    float p0 = ex2(x0), p1 = ex2(x1);
    if (MASK) {
      if (key0 + e > lim) p0 = 0.f;
      if (key0 + e + 1 > lim) p1 = 0.f;
    }
    float s0, s1;
    f2_unpack(f2_mul(f2_pack(p0, p1), f2_add(f2_pack(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), nd2)), s0,
              s1);
    dp[e / 2] = pack_bf16(s0, s1);
  }
}

// --------------------------------------------------------------------- dK, dV: one CTA per key tile
// TMEM: S^T at 0 (P^T packed into it), dP^T at 128 (dS^T packed into it), dV at 256, dK at 256 + d.
template <int D>
struct DkdvCfg : BwdCfg<D> {
  using B = BwdCfg<D>;
  static constexpr uint32_t OFF_K = 0, OFF_V = B::TB;
  static constexpr uint32_t OFF_RING = 2 * B::TB;                   // stage: Q_i, dO_i
  static constexpr uint32_t STAGE = 2 * B::TB;
  // stage: float4 per query-row pair {-lse2[2p], -lse2[2p+1], -D[2p], -D[2p+1]}, lse2 = lse * log2(e)
  static constexpr uint32_t OFF_VEC = OFF_RING + B::ST * STAGE;
  static constexpr uint32_t OFF_BAR = OFF_VEC + B::ST * B::VEC;
  // d = 64 takes each query tile in two halves of 64 queries (see the MMA issuer); d = 128 whole.
  static constexpr bool HALVES = D == 64;
  // B_SF (+ q): products (of query half q) ready; B_PF + c: elementwise chunk c done (d = 128:
  // four 32-query chunks; d = 64: the two query halves); B_GF: gradients final
  static constexpr int B_KV = 0, B_FULL = 1, B_EMPTY = B_FULL + B::ST, B_SF = B_EMPTY + B::ST, B_PF = B_SF + 2,
                       B_GF = B_PF + 4, B_DRAIN = B_GF + 1, B_OW = B_DRAIN + 1, NBAR = B_OW + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8u * NBAR;
  static constexpr uint32_t SMEM = OFF_MISC + 16u + 1024u;
};
static_assert(DkdvCfg<128>::SMEM <= 232448, "dK/dV kernel shared memory");

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(BwdWarps<D>::THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const float* __restrict__ lse, const float* __restrict__ delta, void* __restrict__ dk,
                    void* __restrict__ dv, int N, float sl2, float scale, int grad_fp32,
                    unsigned long long budget, const __grid_constant__ CUtensorMap tdk,
                    const __grid_constant__ CUtensorMap tdv, int ng) {
  using C = DkdvCfg<D>;
  using W = BwdWarps<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sRing = base + C::OFF_RING, sBar = base + C::OFF_BAR;
  float* vec = reinterpret_cast<float*>(gbase + C::OFF_VEC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);
#define BAR(i) (sBar + 8u * static_cast<uint32_t>(i))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int bh, kt;  // key tile; small kt has the most causal work and is scheduled first (within a head group)
  grouped_block(ng, bh, kt);
  const int n_tiles = (N + kTile - 1) / kTile;
  const int i0 = CAUSAL ? kt : 0;  // first query tile that sees this key tile
  const int n_i = n_tiles - i0;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_KV), 1);
    for (int s = 0; s < C::ST; ++s) {
      mbar_init(BAR(C::B_FULL + s), 1 + 32);  // TMA bytes + the producer warp's lse/D stores
      mbar_init(BAR(C::B_EMPTY + s), 1);
    }
    mbar_init(BAR(C::B_SF), 1);
    mbar_init(BAR(C::B_SF + 1), 1);
    for (int c = 0; c < W::CHUNKS; ++c) mbar_init(BAR(C::B_PF + c), W::EW * 32);
    mbar_init(BAR(C::B_GF), 1);
    mbar_init(BAR(C::B_DRAIN), 1);
    mbar_init(BAR(C::B_OW), W::EW * 32);  // bf16 gradients staged
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == W::MMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == W::TMA) {
    // ------------------------------------------------------------ producer (whole warp)
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      mbar_arrive_expect_tx(BAR(C::B_KV), 2 * C::TB);
      for (int h = 0; h < C::NH; ++h) {
        tma_load_3d(sK + h * kBox, &tk, BAR(C::B_KV), h * 64, kt * kTile, bh);
        tma_load_3d(sV + h * kBox, &tv, BAR(C::B_KV), h * 64, kt * kTile, bh);
      }
    }
    int issued = 0;
    for (int i = 0; i < n_i; ++i) {
      const int s = i % C::ST;
      if (i >= C::ST && !bwait_all(BAR(C::B_EMPTY + s), ((i / C::ST) - 1) & 1, abort_flag, budget)) break;
      const int qt = i0 + i;
      if (lane == 0) {
        mbar_arrive_expect_tx(BAR(C::B_FULL + s), 2 * C::TB);
        const uint32_t st = sRing + s * C::STAGE;
        for (int h = 0; h < C::NH; ++h) {
          tma_load_3d(st + h * kBox, &tq, BAR(C::B_FULL + s), h * 64, qt * kTile, bh);
          tma_load_3d(st + C::TB + h * kBox, &tdo, BAR(C::B_FULL + s), h * 64, qt * kTile, bh);
        }
      }
      // -lse (log2 units) and -D of the tile's 128 query rows, pairs of rows in one float4 (the
      // elementwise warps add them with packed f32x2 operations); rows past N get -lse = -inf, so P = 0.
      float* vs = vec + s * (2 * kTile);
#pragma unroll
      for (int c = 0; c < kTile / 32; ++c) {
        const int col = 32 * c + lane;
        const int r = qt * kTile + col;
        const bool in = r < N;
        vs[4 * (col >> 1) + (col & 1)] = in ? -lse[static_cast<size_t>(bh) * N + r] * kLog2e : -INFINITY;
        vs[4 * (col >> 1) + 2 + (col & 1)] = in ? -delta[static_cast<size_t>(bh) * N + r] : 0.f;
      }
      mbar_arrive(BAR(C::B_FULL + s));
      issued = i + 1;
    }
    if (lane == 0) {
      bdrain(BAR(C::B_KV), 0, budget);
      for (int i = max(0, issued - C::ST); i < issued; ++i) bdrain(BAR(C::B_FULL + i % C::ST), (i / C::ST) & 1, budget);
    }
  } else if (warp == W::MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      if constexpr (C::HALVES) {
        // Each query tile is taken in two halves of 64 queries, so that the products of one half run
        // on the tensor core while the elementwise warps work on the other: S^T_q and dP^T_q are
        // columns 64q .. 64q + 63 of the S^T and dP^T accumulators.
        constexpr uint32_t idesc_p = idesc_bf16_f32(kTile, kTile / 2, 0);  // K Q_q^T, V dO_q^T: both K-major
        constexpr uint32_t idesc_g = idesc_bf16_f32(kTile, D, 1);          // P^T dO, dS^T Q: MN-major B
        const uint64_t dK = sdesc_sw128(sK, 16, 1024), dV = sdesc_sw128(sV, 16, 1024);
        const uint64_t dR = sdesc_sw128(sRing, 16, 1024), dRmn = sdesc_sw128(sRing, kBox, 1024);
        auto products = [&](int i, int q) {  // rows 64q .. 64q + 63 of Q_i and dO_i are N
          const uint32_t st = (i % C::ST) * C::STAGE + static_cast<uint32_t>(q) * (kTile / 2) * 128u;
          issue_product<D>(tmem + kColA + 64u * q, dK, sdesc_add(dR, st), idesc_p);          // S^T_q = K Q_q^T
          issue_product<D>(tmem + kColB + 64u * q, dV, sdesc_add(dR, st + C::TB), idesc_p);  // dP^T_q = V dO_q^T
        };
        bool ok = bwait(BAR(C::B_KV), 0, abort_flag, budget) && bwait(BAR(C::B_FULL), 0, abort_flag, budget);
        if (ok) {
          tc_fence_after();
          products(0, 0);
          tc_commit(BAR(C::B_SF));
          products(0, 1);
          tc_commit(BAR(C::B_SF + 1));
        }
        for (int i = 0; ok && i < n_i; ++i) {
          const uint32_t st = (i % C::ST) * C::STAGE;
          for (int q = 0; ok && q < 2; ++q) {
            if (!bwait(BAR(C::B_PF + q), i & 1, abort_flag, budget)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_grad_half<D>(tmem + kColG1, tmem + kColA, sdesc_add(dRmn, st + C::TB), idesc_g, i > 0 || q > 0,
                               q);  // dV += P^T_q dO_q
            issue_grad_half<D>(tmem + C::COL_G2, tmem + kColB, sdesc_add(dRmn, st), idesc_g, i > 0 || q > 0,
                               q);  // dK += dS^T_q Q_q
            if (q == 1) tc_commit(BAR(C::B_EMPTY + i % C::ST));  // Q_i, dO_i fully read
            if (i + 1 < n_i) {
              // half q of the next tile into the columns the gradient MMAs above read: they were
              // issued first, and MMAs complete in issue order
              if (q == 0 && !bwait(BAR(C::B_FULL + (i + 1) % C::ST), ((i + 1) / C::ST) & 1, abort_flag, budget)) {
                ok = false;
                break;
              }
              tc_fence_after();
              products(i + 1, q);
              tc_commit(BAR(C::B_SF + q));
            }
          }
        }
        tc_commit(BAR(C::B_GF));  // the gradients final (when every MMA above is complete)
      } else {
        // d = 128: TMEM holds S^T, dP^T, dV and dK (4 x 128 columns), so the products of the
        // next query tile start only after this tile's elementwise step; the gradient MMAs of
        // each 32-column chunk start as soon as the elementwise warps finish it.
        constexpr uint32_t idesc_p = idesc_bf16_f32(kTile, kTile, 0);  // K Q^T, V dO^T: both K-major
        constexpr uint32_t idesc_g = idesc_bf16_f32(kTile, D, 1);      // P^T dO, dS^T Q: MN-major B
        const uint64_t dK = sdesc_sw128(sK, 16, 1024), dV = sdesc_sw128(sV, 16, 1024);
        const uint64_t dR = sdesc_sw128(sRing, 16, 1024), dRmn = sdesc_sw128(sRing, kBox, 1024);
        auto products = [&](int i) {
          const uint32_t st = (i % C::ST) * C::STAGE;
          issue_product<D>(tmem + kColA, dK, sdesc_add(dR, st), idesc_p);           // S^T = K Q^T
          issue_product<D>(tmem + kColB, dV, sdesc_add(dR, st + C::TB), idesc_p);   // dP^T = V dO^T
        };
        bool ok = bwait(BAR(C::B_KV), 0, abort_flag, budget) && bwait(BAR(C::B_FULL), 0, abort_flag, budget);
        if (ok) {
          tc_fence_after();
          products(0);
          tc_commit(BAR(C::B_SF));
        }
        for (int i = 0; ok && i < n_i; ++i) {
          const uint32_t st = (i % C::ST) * C::STAGE;
          bool part_ok = true;
          for (int part = 0; part < W::CHUNKS; ++part) {  // each chunk as soon as the elementwise warps finish it
            if (!bwait(BAR(C::B_PF + part), i & 1, abort_flag, budget)) {
              part_ok = false;
              break;
            }
            tc_fence_after();
            issue_grad_chunk(tmem + kColG1, tmem + kColA, sdesc_add(dRmn, st + C::TB), idesc_g, i > 0 || part > 0,
                             part);  // dV += P^T dO
            issue_grad_chunk(tmem + C::COL_G2, tmem + kColB, sdesc_add(dRmn, st), idesc_g, i > 0 || part > 0,
                             part);  // dK += dS^T Q
          }
          if (!part_ok) break;
          tc_commit(BAR(C::B_EMPTY + i % C::ST));
          if (i + 1 < n_i) {
            if (!bwait(BAR(C::B_FULL + (i + 1) % C::ST), ((i + 1) / C::ST) & 1, abort_flag, budget)) break;
            tc_fence_after();
            products(i + 1);
          }
          if (i + 1 < n_i) tc_commit(BAR(C::B_SF));  // next products ready
        }
        tc_commit(BAR(C::B_GF));  // the gradients final (when every MMA above is complete)
      }
      tc_commit(BAR(C::B_DRAIN));
      bdrain(BAR(C::B_DRAIN), 0, budget);
    }
  } else {
    // ------------------------------------------------------------ elementwise warps: thread = key row
    const int quarter = warp & 3, sub = W::ONE ? 0 : warp >> 2, h = W::ONE ? 0 : lane >> 4;
    const int r = W::ONE ? 32 * quarter + lane : 32 * quarter + 16 * sub + (lane & 15);  // TMEM lane = key row
    const int key = kt * kTile + r;
    const uint32_t lane_addr = static_cast<uint32_t>(W::ONE ? 32 * quarter : 32 * quarter + 16 * sub) << 16;
    const uint32_t tA = tmem + lane_addr + kColA, tB = tmem + lane_addr + kColB;
    const uint64_t c2 = f2_pack(sl2, sl2);
    bool ok = true;
    if constexpr (C::HALVES) {
      for (int i = 0; ok && i < n_i; ++i) {
        const int s = i % C::ST;
        ok = bwait_all(BAR(C::B_FULL + s), (i / C::ST) & 1, abort_flag, budget);  // the tile's -lse, -D
        const int qt = i0 + i;
        const float4* nv = reinterpret_cast<const float4*>(vec + s * (2 * kTile));
        // Causal: only the diagonal query tile (qt == kt) holds pairs with query < key.
        const bool diag = CAUSAL && qt == kt;
        // query half q: this thread's 32 queries 64q + 32h .. (columns of S^T_q, dP^T_q)
        for (int q = 0; ok && q < 2; ++q) {
          ok = bwait_all(BAR(C::B_SF + q), i & 1, abort_flag, budget);
          if (!ok) break;
          tc_fence_after();
          uint32_t sv[32], pv[32];
          tmem_ld2_x32<32>(tA + 64 * q, sv);
          tmem_ld2_x32<32>(tB + 64 * q, pv);
          uint32_t pp[16], dp[16];
          if (diag) ew_pairs_dkdv<true>(sv, pv, nv, c2, 64 * q + 32 * h, qt * kTile, key, pp, dp);
          else ew_pairs_dkdv<false>(sv, pv, nv, c2, 64 * q + 32 * h, qt * kTile, key, pp, dp);
          tmem_st2_x16<32>(tA + 64 * q, pp);  // P^T packed: columns 64q + 32h .. + 15
          tmem_st2_x16<32>(tB + 64 * q, dp);  // dS^T packed
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(BAR(C::B_PF + q));  // half q ready: its gradient MMAs may start
        }
      }
    } else {
      for (int i = 0; ok && i < n_i; ++i) {
        const int s = i % C::ST;
        ok = bwait_all(BAR(C::B_SF), i & 1, abort_flag, budget) &&
             bwait_all(BAR(C::B_FULL + s), (i / C::ST) & 1, abort_flag, budget);
        if (!ok) break;
        tc_fence_after();
        const int qt = i0 + i;
        const float4* nv = reinterpret_cast<const float4*>(vec + s * (2 * kTile));
        // Causal: only the diagonal query tile (qt == kt) holds pairs with query < key.
        const bool diag = CAUSAL && qt == kt;
        // this thread's row: its 128 query columns in four chunks of 32, chunk c packed into
        // columns 16c .. 16c + 15 (all read by this thread already)
  #pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t sv[32], pv[32];
          tmem_ld_x32(tA + 32 * c, sv);
          tmem_ld_x32(tB + 32 * c, pv);
          uint32_t pp[16], dp[16];
          if (diag) ew_pairs_dkdv<true>(sv, pv, nv, c2, 32 * c, qt * kTile, key, pp, dp);
          else ew_pairs_dkdv<false>(sv, pv, nv, c2, 32 * c, qt * kTile, key, pp, dp);
          tmem_st1_x16(tA + 16 * c, pp);  // P^T packed
          tmem_st1_x16(tB + 16 * c, dp);  // dS^T packed
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(BAR(C::B_PF + c));  // chunk c ready: its gradient MMAs may start
        }
      }
    }
    if (ok) ok = bwait_all(BAR(C::B_GF), 0, abort_flag, budget);  // gradients final
    if (ok) {
      tc_fence_after();
      const size_t row_off = static_cast<size_t>(bh) * N + key;
      if (grad_fp32) {
        if constexpr (W::ONE) {
          store_grad_row128(dv, row_off, key < N, tmem + lane_addr + kColG1, 1.f);
          store_grad_row128(dk, row_off, key < N, tmem + lane_addr + C::COL_G2, scale);
        } else {
          store_grad_half_row<D>(dv, row_off, h, key < N, true, tmem + lane_addr + kColG1, 1.f);
          store_grad_half_row<D>(dk, row_off, h, key < N, true, tmem + lane_addr + C::COL_G2, scale);
        }
      } else {
        // bf16 dV and dK through shared memory: the V and K tiles have their shape and are no
        // longer read (every product MMA is complete); one thread stores them with TMA.
        if constexpr (W::ONE) {
          stage_row128_bf16(sV, sV + kBox, r, tmem + lane_addr + kColG1, 1.f);
          stage_row128_bf16(sK, sK + kBox, r, tmem + lane_addr + C::COL_G2, scale);
        } else {
          stage_half_row_bf16<D>(sV, sV + kBox, r, h, tmem + lane_addr + kColG1, 1.f);
          stage_half_row_bf16<D>(sK, sK + kBox, r, h, tmem + lane_addr + C::COL_G2, scale);
        }
        mbar_arrive(BAR(C::B_OW));
        if (warp == 0 && lane == 0 && bwait(BAR(C::B_OW), 0, abort_flag, budget)) {
          for (int hb = 0; hb < C::NH; ++hb) {
            tma_store_3d(&tdv, sV + static_cast<uint32_t>(hb) * kBox, hb * 64, kt * kTile, bh);
            tma_store_3d(&tdk, sK + static_cast<uint32_t>(hb) * kBox, hb * 64, kt * kTile, bh);
          }
          bulk_commit();
          bulk_wait_all();  // complete before the CTA exits
        }
      }
    }
    tmem_wait_st();
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == W::MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------------- dQ: one CTA per query tile
// TMEM: S at 0, dP at 128 (dS packed into it), dQ at 256.
template <int D>
struct DqCfg : BwdCfg<D> {
  using B = BwdCfg<D>;
  static constexpr uint32_t OFF_Q = 0, OFF_DO = B::TB;
  static constexpr uint32_t OFF_RING = 2 * B::TB;  // stage: K_j, V_j
  static constexpr uint32_t STAGE = 2 * B::TB;
  static constexpr uint32_t OFF_BAR = OFF_RING + B::ST * STAGE;
  static constexpr int B_QD = 0, B_FULL = 1, B_EMPTY = B_FULL + B::ST, B_SF = B_EMPTY + B::ST, B_PF = B_SF + 1,
                       B_DRAIN = B_PF + 4, B_OW = B_DRAIN + 1, NBAR = B_OW + 1;  // B_PF + c: chunk c of the
                                                                               // elementwise step
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8u * NBAR;
  static constexpr uint32_t SMEM = OFF_MISC + 16u + 1024u;
};
static_assert(DqCfg<128>::SMEM <= 232448, "dQ kernel shared memory");

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(BwdWarps<D>::THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const float* __restrict__ lse, const float* __restrict__ delta, void* __restrict__ dq, int N,
                  float sl2, float scale, int grad_fp32, unsigned long long budget,
                  const __grid_constant__ CUtensorMap tdq, int ng) {
  using C = DqCfg<D>;
  using W = BwdWarps<D>;  // thread = query row here
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + C::OFF_Q, sDO = base + C::OFF_DO, sRing = base + C::OFF_RING, sBar = base + C::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);
#define BAR(i) (sBar + 8u * static_cast<uint32_t>(i))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int bh, qt;
  grouped_block(ng, bh, qt);
  const int n_tiles = (N + kTile - 1) / kTile;
  qt = n_tiles - 1 - qt;  // most causal work first (within a head group)
  const int n_j = CAUSAL ? qt + 1 : n_tiles;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_QD), 1);
    for (int s = 0; s < C::ST; ++s) {
      mbar_init(BAR(C::B_FULL + s), 1);
      mbar_init(BAR(C::B_EMPTY + s), 1);
    }
    mbar_init(BAR(C::B_SF), 1);
    for (int c = 0; c < W::CHUNKS; ++c) mbar_init(BAR(C::B_PF + c), W::EW * 32);
    mbar_init(BAR(C::B_DRAIN), 1);
    mbar_init(BAR(C::B_OW), W::EW * 32);  // bf16 gradients staged
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == W::MMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == W::TMA) {
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      mbar_arrive_expect_tx(BAR(C::B_QD), 2 * C::TB);
      for (int h = 0; h < C::NH; ++h) {
        tma_load_3d(sQ + h * kBox, &tq, BAR(C::B_QD), h * 64, qt * kTile, bh);
        tma_load_3d(sDO + h * kBox, &tdo, BAR(C::B_QD), h * 64, qt * kTile, bh);
      }
      int issued = 0;
      for (int j = 0; j < n_j; ++j) {
        const int s = j % C::ST;
        if (j >= C::ST && !bwait(BAR(C::B_EMPTY + s), ((j / C::ST) - 1) & 1, abort_flag, budget)) break;
        mbar_arrive_expect_tx(BAR(C::B_FULL + s), 2 * C::TB);
        const uint32_t st = sRing + s * C::STAGE;
        for (int h = 0; h < C::NH; ++h) {
          tma_load_3d(st + h * kBox, &tk, BAR(C::B_FULL + s), h * 64, j * kTile, bh);
          tma_load_3d(st + C::TB + h * kBox, &tv, BAR(C::B_FULL + s), h * 64, j * kTile, bh);
        }
        issued = j + 1;
      }
      bdrain(BAR(C::B_QD), 0, budget);
      for (int j = max(0, issued - C::ST); j < issued; ++j) bdrain(BAR(C::B_FULL + j % C::ST), (j / C::ST) & 1, budget);
    }
  } else if (warp == W::MMA) {
    if (lane == 0) {
      constexpr uint32_t idesc_p = idesc_bf16_f32(kTile, kTile, 0);  // Q K^T, dO V^T: both K-major
      constexpr uint32_t idesc_g = idesc_bf16_f32(kTile, D, 1);      // dS K: K MN-major
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024), dDO = sdesc_sw128(sDO, 16, 1024);
      const uint64_t dR = sdesc_sw128(sRing, 16, 1024), dRmn = sdesc_sw128(sRing, kBox, 1024);
      // S(j) alternates between two TMEM buffers, so S(j+1) can run while the elementwise warps
      // still work on step j; dP(j+1) has one buffer (dS(j) is packed into it) and follows the
      // dQ MMAs of step j.
      auto issue_s = [&](int j) {
        const uint32_t st = (j % C::ST) * C::STAGE;
        issue_product<D>(tmem + ((j & 1) ? kColS1 : kColA), dQ, sdesc_add(dR, st), idesc_p);  // S = Q K^T
      };
      auto issue_dp = [&](int j) {
        const uint32_t st = (j % C::ST) * C::STAGE;
        issue_product<D>(tmem + kColB, dDO, sdesc_add(dR, st + C::TB), idesc_p);  // dP = dO V^T
      };
      bool ok = bwait(BAR(C::B_QD), 0, abort_flag, budget) && bwait(BAR(C::B_FULL), 0, abort_flag, budget);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
        tc_commit(BAR(C::B_SF));
      }
      for (int j = 0; ok && j < n_j; ++j) {
        // dQ += dS K for the first chunk, then S(j+1) (under the elementwise warps' second chunk),
        // then the second chunk's dQ MMAs and dP(j+1).
        if (!bwait(BAR(C::B_PF), j & 1, abort_flag, budget)) break;
        tc_fence_after();
        if constexpr (W::ONE)
          issue_grad_chunk(tmem + kColG1, tmem + kColB, sdesc_add(dRmn, (j % C::ST) * C::STAGE), idesc_g, j > 0, 0);
        else
          issue_grad_part<D>(tmem + kColG1, tmem + kColB, sdesc_add(dRmn, (j % C::ST) * C::STAGE), idesc_g, j > 0,
                             0);
        if (j + 1 < n_j) {
          if (!bwait(BAR(C::B_FULL + (j + 1) % C::ST), ((j + 1) / C::ST) & 1, abort_flag, budget)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        bool chunks_ok = true;
        for (int c = 1; c < W::CHUNKS; ++c) {
          if (!bwait(BAR(C::B_PF + c), j & 1, abort_flag, budget)) {
            chunks_ok = false;
            break;
          }
          tc_fence_after();
          if constexpr (W::ONE)
            issue_grad_chunk(tmem + kColG1, tmem + kColB, sdesc_add(dRmn, (j % C::ST) * C::STAGE), idesc_g, true, c);
          else
            issue_grad_part<D>(tmem + kColG1, tmem + kColB, sdesc_add(dRmn, (j % C::ST) * C::STAGE), idesc_g, true,
                               c);
        }
        if (!chunks_ok) break;
        tc_commit(BAR(C::B_EMPTY + j % C::ST));
        if (j + 1 < n_j) issue_dp(j + 1);
        tc_commit(BAR(C::B_SF));
      }
      tc_commit(BAR(C::B_DRAIN));
      bdrain(BAR(C::B_DRAIN), 0, budget);
    }
  } else {
    // ------------------------------------------------------------ elementwise warps: thread = query row
    const int quarter = warp & 3, sub = W::ONE ? 0 : warp >> 2, h = W::ONE ? 0 : lane >> 4;
    const int r = W::ONE ? 32 * quarter + lane : 32 * quarter + 16 * sub + (lane & 15);
    const int row = qt * kTile + r;
    const uint32_t lane_addr = static_cast<uint32_t>(W::ONE ? 32 * quarter : 32 * quarter + 16 * sub) << 16;
    const uint32_t tB = tmem + lane_addr + kColB;  // dP; S(j) is in buffer j % 2 (kColA, kColS1)
    const bool in = row < N;
    const float lse2 = in ? lse[static_cast<size_t>(bh) * N + row] * kLog2e : INFINITY;
    const float dd = in ? delta[static_cast<size_t>(bh) * N + row] : 0.f;
    const int lim = CAUSAL ? min(row, N - 1) : N - 1;  // last key this row attends
    const uint64_t c2 = f2_pack(sl2, sl2), nl2 = f2_pack(-lse2, -lse2), nd2 = f2_pack(-dd, -dd);
    bool ok = true;
    for (int j = 0; ok && j < n_j; ++j) {
      ok = bwait_all(BAR(C::B_SF), j & 1, abort_flag, budget);
      if (!ok) break;
      tc_fence_after();
      if constexpr (W::ONE) {
        // this thread's row: 128 keys in four chunks of 32, chunk c's dS packed into dP's columns
        // 16c .. 16c + 15 (read by this thread already)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t sv[32], pv[32];
          tmem_ld_x32(tmem + lane_addr + ((j & 1) ? kColS1 : kColA) + 32 * c, sv);
          tmem_ld_x32(tB + 32 * c, pv);
          uint32_t dp[16];
          const int key0 = j * kTile + 32 * c;
          if (key0 + 31 > lim) ew_pairs_dq<true>(sv, pv, c2, nl2, nd2, key0, lim, dp);
          else ew_pairs_dq<false>(sv, pv, c2, nl2, nd2, key0, lim, dp);
          tmem_st1_x16(tB + 16 * c, dp);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(BAR(C::B_PF + c));  // chunk c ready: its gradient MMAs may start
        }
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sv[32], pv[32];
          tmem_ld2_x32<64>(tmem + lane_addr + ((j & 1) ? kColS1 : kColA) + 32 * c, sv);
          tmem_ld2_x32<64>(tB + 32 * c, pv);
          uint32_t dp[16];
          const int key0 = j * kTile + 64 * h + 32 * c;
          // only the diagonal and the ragged last key tile reach past this row's last key
          if (key0 + 31 > lim) ew_pairs_dq<true>(sv, pv, c2, nl2, nd2, key0, lim, dp);
          else ew_pairs_dq<false>(sv, pv, c2, nl2, nd2, key0, lim, dp);
          tmem_st2_x16<64>(tB + 16 * c, dp);  // dS packed into dP's columns 64h + 16c ..
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(BAR(C::B_PF + c));  // chunk c ready: its gradient MMAs may start
        }
      }
    }
    if (ok) ok = bwait_all(BAR(C::B_SF), n_j & 1, abort_flag, budget);
    if (ok) {
      tc_fence_after();
      if (grad_fp32) {
        if constexpr (W::ONE) store_grad_row128(dq, static_cast<size_t>(bh) * N + row, in, tmem + lane_addr + kColG1, scale);
        else store_grad_half_row<D>(dq, static_cast<size_t>(bh) * N + row, h, in, true, tmem + lane_addr + kColG1, scale);
      } else {
        // bf16 dQ through shared memory: the Q tile has its shape and is no longer read
        if constexpr (W::ONE) stage_row128_bf16(sQ, sQ + kBox, r, tmem + lane_addr + kColG1, scale);
        else stage_half_row_bf16<D>(sQ, sQ + kBox, r, h, tmem + lane_addr + kColG1, scale);
        mbar_arrive(BAR(C::B_OW));
        if (warp == 0 && lane == 0 && bwait(BAR(C::B_OW), 0, abort_flag, budget)) {
          for (int hb = 0; hb < C::NH; ++hb)
            tma_store_3d(&tdq, sQ + static_cast<uint32_t>(hb) * kBox, hb * 64, qt * kTile, bh);
          bulk_commit();
          bulk_wait_all();  // complete before the CTA exits
        }
      }
    }
    tmem_wait_st();
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == W::MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_t(const BwdLaunch& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.BH) * a.N;
  const long long threads = rows * (D / 8);
  bwd_delta_kernel<D><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.delta, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const int ng = head_groups(a.BH, n_tiles, CAUSAL, a.sms);
  dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>(n_tiles));
  auto k1 = bwd_dkdv_kernel<D, CAUSAL>;
  if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvCfg<D>::SMEM)) != cudaSuccess)
    return e;
  k1<<<grid, BwdWarps<D>::THREADS, DkdvCfg<D>::SMEM, stream>>>(a.tq, a.tk, a.tv, a.tdo, a.lse, a.delta, a.dk, a.dv, a.N,
                                                   a.scale_log2, a.scale, a.grad_fp32, a.budget, a.tdk, a.tdv, ng);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto k2 = bwd_dq_kernel<D, CAUSAL>;
  if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM)) != cudaSuccess)
    return e;
  k2<<<grid, BwdWarps<D>::THREADS, DqCfg<D>::SMEM, stream>>>(a.tq, a.tk, a.tv, a.tdo, a.lse, a.delta, a.dq, a.N, a.scale_log2,
                                                 a.scale, a.grad_fp32, a.budget, a.tdq, ng);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_bwd_t<64, true>(a, stream) : launch_bwd_t<64, false>(a, stream);
  return a.causal ? launch_bwd_t<128, true>(a, stream) : launch_bwd_t<128, false>(a, stream);
}

unsigned int bwd_read_and_clear_status() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_bwd_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(zero));
  return v;
}

}  // namespace fattn
