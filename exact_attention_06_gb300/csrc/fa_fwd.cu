// Fused exact attention forward (prefill) for sm_103a.
//
// One CTA owns two 128-row query tiles Q_0, Q_1 (rows 256p .. 256p+255) of one
// (batch, head) and scans the 128-key tiles K_j, V_j once, FA-2 order
// (xuesongtap.github.io "flash-attention" page, §2.1; triton-tutorial
// "8. FlashAttention 实战", §8.4.1: Q outer and resident, K/V inner and
// streamed).  Per tile and query tile t:
//   S_t = Q_t K_j^T                    tcgen05.mma, bf16 x bf16 -> fp32 in TMEM
//   m_new = max(m, rowmax(S_t) * c)    c = scale * log2(e)  (exp2 trick, §8.7.3)
//   alpha = 2^(m - m_new),  P~ = 2^(S_t*c - m_new)  (online softmax, §8.3.3)
//   l = alpha * l + rowsum(P~)         fp32, from the unrounded P~
//   U_t = alpha * U_t + bf16(P~) V_j   P~ written back to TMEM as the A operand
// and after the scan O = U / l, lse = (m + log2 l) * ln 2.
//
// Warp roles (the producer/consumer split and the two-consumer "ping-pong" of
// triton-tutorial §8.10.2-§8.10.3, re-done with TMA + tcgen05 + TMEM):
//   softmax of Q_0, then the same number of warps for Q_1: bf16 at d = 128 (P~
//              aliasing S), 4 warps a tile, one thread per query row with all of
//              its 128 key columns (.32x32b TMEM access, two 64-column loads, so
//              that the max of the first half overlaps the second load); the
//              separate-P~ schedules 8 warps a tile, two threads per row, each
//              with half of the columns (.16x32bx2: a warp holds 16 rows x both
//              halves), the row max joined with one shuffle and l kept per half
//              until the epilogue.  Whole rows stay inside one warp, so there is
//              no cross-warp softmax merge (iceferryling "FlashAttention 1 和
//              FlashAttention 2 的区别", §7-8 split-Q).  They also apply the alpha
//              rescale of U_t and write O_t, lse.
//   MMA warp(s) one issuing thread each; the first also owns TMEM.
//   last warp  TMA producer: Q_0, Q_1 once, then K_j and V_j into two rings.
// Three schedules, by where P~ lives:
//   bf16, d = 128: TMEM holds S_0, S_1 (columns 0, 128) and U_0, U_1 (256, 384), so
//     P~ is written as packed bf16 into the first 64 columns of its own S.  One MMA
//     warp alternates between the tiles: [PV_0(j-1), S_0(j)] runs while the Q_1
//     softmax works on S_1(j-1) and vice versa; the commit after S_t(j) also covers
//     PV_t(j-1), so the softmax that sees S_t(j) may rescale U_t in place.
//   bf16, d = 64: U_t takes 64 columns, so P~_t gets its own TMEM columns
//     (384 + 64t) and one MMA warp per tile issues S_t(j+1) as soon as the softmax
//     has read S_t(j) ("separate P~"); the softmax waits for PV_t(j-1) only before
//     overwriting P~_t and rescaling U_t.
//   E4M3, d = 128: as bf16 d = 128, with P~ packed four keys a column into its S
//     (32 columns a row) and the PV MMA kind::f8f6f4 reading it from TMEM.
//
// Two kernels share these schedules.  fwd_kernel runs one CTA per block of 256 query rows
// (causal launches order the blocks longest first).  fwd_persist_kernel (non-causal bf16,
// d = 64) runs one CTA per SM that walks a list of blocks, keeping TMEM, barriers and the K/V
// ring between them, so that a block's Q load and first S overlap the previous block's last
// steps and epilogue; it also runs the split last round of fa_fwd_ex (key pieces or single query
// tiles).  It has three MMA-issuing threads: the S products of both tiles, the PV products of
// tile 0, those of tile 1 (an issuing thread keeps about one batch of MMAs in flight, so PV_0 and
// PV_1 from threads of their own overlap).
//
// Causal: key tiles above a query tile's diagonal are never computed for it
// (Q_0 stops one tile before Q_1); only the diagonal tile masks (col > row ->
// -inf), and the ragged last tile masks col >= N (triton-tutorial §8.7.1
// STAGE split; xuesongtap §2.2 last paragraph).
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>

#include "internal.h"
#include "ptx.cuh"
#include "stage_io.cuh"
#include "tmem_io.cuh"

namespace fattn {

__device__ unsigned int g_fwd_status = 0;

namespace {

constexpr int kBr = 128;                 // query rows per tile (TMEM lanes, MMA M)
constexpr int kBc = 128;                 // keys per tile
constexpr int kRowsPerCta = 2 * kBr;
constexpr uint32_t kBox = 128u * 128u;   // bytes of a 128-row x 128-byte box (64 bf16 or 128 E4M3 columns)
constexpr int kSoftmaxWarps = 8;          // per query tile
constexpr int kWarpMma = 2 * kSoftmaxWarps;  // first MMA warp; also allocates TMEM
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, bool FP8 = false>
struct FwdCfg {
  static constexpr int ESZ = FP8 ? 1 : 2;           // bytes per element (E4M3 or bf16)
  static constexpr int ROW = D * ESZ;               // bytes per row
  static constexpr int NH = ROW / 128;              // 128-byte boxes per row
  static constexpr int BOX_X = 128 / ESZ;           // elements per box row (TMA x step)
  static constexpr int K_MMA = 32 / ESZ;            // K elements per MMA instruction (32 bytes)
  static constexpr int KST = FP8 ? 4 : ((D == 128) ? 3 : 4);  // K ring stages
  static constexpr int VST = FP8 ? 4 : ((D == 128) ? 2 : 4);  // V ring stages
  static constexpr uint32_t QB = NH * kBox;         // bytes of one Q tile
  static constexpr uint32_t KVB = NH * kBox;        // bytes of one K (or V) tile
  static constexpr int B_Q = 0, B_QE = B_Q + 1, B_KF = B_QE + 1, B_KE = B_KF + KST, B_VF = B_KE + KST, B_VE = B_VF + VST,
                       B_SF = B_VE + VST, B_PF = B_SF + 2, B_SC = B_PF + 2, B_OF = B_SC + 2, B_DRAIN = B_OF + 2,
                       B_OSF = B_DRAIN + 2, B_OW = B_OSF + 2, NBAR = B_OW + 2;
  // d = 64 leaves 128 TMEM columns free: P~_t gets its own columns there, so S_t(j+1) can be
  // computed while the softmax of tile j still runs ("separate P~").  At d = 128 P~ aliases S,
  // for bf16 (two keys a column) and E4M3 (four keys a column) alike.
  static constexpr bool SEP = D == 64;
  // E4M3: a second 16 KB box per tile, which with the Q tile's stages O in bf16 (128 x 256 bytes)
  static constexpr bool P_SMEM = FP8;
  static constexpr uint32_t COL_P = SEP ? 384u : 0u;        // separate P~ columns (+ 64 t)
  static constexpr uint32_t PB = P_SMEM ? kBr * 128u : 0u;  // bytes of one tile's second O staging box (E4M3)
  // With separate P~ each tile gets its own MMA warp (at d = 64 the PV MMAs, N = 64, are also too
  // short for one issuing thread); with P~ aliasing S (bf16, d = 128) one MMA warp alternating
  // between the tiles measured faster.
  static constexpr bool TWO_ISSUERS = SEP;
  // Softmax warps per query tile: with P~ aliasing S (d = 128) one thread per row (4 warps,
  // .32x32b TMEM access); the separate-P~ schedule (d = 64) two threads per row (8 warps, .16x32bx2).
  static constexpr bool ONE = !SEP;
  static constexpr int SMW = ONE ? 4 : 8;
  static constexpr int WARP_MMA = 2 * SMW;
  static constexpr int WARP_TMA = WARP_MMA + (TWO_ISSUERS ? 2 : 1);
  static constexpr int THREADS = (WARP_TMA + 1) * 32;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = 2 * QB;
  static constexpr uint32_t OFF_V = OFF_K + KST * KVB;
  static constexpr uint32_t OFF_P = OFF_V + VST * KVB;       // E4M3 only: O staging boxes of both tiles
  static constexpr uint32_t OFF_BAR = OFF_P + 2 * PB;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8u * NBAR;  // TMEM address slot, abort flag
  static constexpr uint32_t SMEM = OFF_MISC + 16u + 1024u;   // + slack to align the base to 1 KB
};
// The persistent kernel (bf16 d = 64): the d = 64 layout with three MMA-issuing warps (the S
// products of both tiles, the PV products of tile 0, those of tile 1) before the producer, a
// drain barrier for each, and O of both tiles staged in shared memory for the TMA store (128
// bytes a row).  20 warps are five per SMSP: 96 registers a thread.
struct PersistCfg : FwdCfg<64> {
  static constexpr int N_ISSUERS = 3;
  static constexpr int WARP_TMA = kWarpMma + N_ISSUERS;
  static constexpr int THREADS = (WARP_TMA + 1) * 32;
  static constexpr int B_Q = 0, B_QE = B_Q + 1, B_KF = B_QE + 1, B_KE = B_KF + KST, B_VF = B_KE + KST, B_VE = B_VF + VST,
                       B_SF = B_VE + VST, B_PF = B_SF + 2, B_SC = B_PF + 2, B_OF = B_SC + 2, B_DRAIN = B_OF + 2,
                       B_OSF = B_DRAIN + N_ISSUERS, B_OW = B_OSF + 2, NBAR = B_OW + 2;
  static constexpr uint32_t OFF_BAR = OFF_V + VST * KVB;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8u * NBAR;
  static constexpr uint32_t OFF_O = (OFF_MISC + 16u + 1023u) & ~1023u;
  static constexpr uint32_t SMEM = OFF_O + 2u * kBr * 128u + 1024u;
};
static_assert(FwdCfg<128>::SMEM <= 232448, "shared memory of the d=128 kernel exceeds 227 KB");
static_assert(FwdCfg<128, true>::SMEM <= 232448, "shared memory of the FP8 kernel exceeds 227 KB");
static_assert(PersistCfg::SMEM <= 232448, "shared memory of the persistent kernel exceeds 227 KB");

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget, &g_fwd_status);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag: used to drain in-flight copies
// and MMAs before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long budget) {
  // A drain never gets less than the default budget, however short the caller's wait budget is.
  if (budget < kDrainBudget) budget = kDrainBudget;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<unsigned long long>(clock64() - t0) > budget) {
      atomicOr(&g_fwd_status, kStatusTimeout);
      return;
    }
  }
}

// This thread's half of a U_t row (D/2 columns) *= alpha, in one TMEM round trip.
template <int D>
__device__ __forceinline__ void rescale_half_row(uint32_t taddr, float alpha) {
  const uint64_t a2 = f2_pack(alpha, alpha);
  uint32_t ur[D / 2];
  if constexpr (D == 128) tmem_ld2_x64<64>(taddr, ur); else tmem_ld2_x32<32>(taddr, ur);
#pragma unroll
  for (int i = 0; i < D / 4; ++i) {
    float lo, hi;
    f2_unpack(f2_mul(f2_pack(__uint_as_float(ur[2 * i]), __uint_as_float(ur[2 * i + 1])), a2), lo, hi);
    ur[2 * i] = __float_as_uint(lo);
    ur[2 * i + 1] = __float_as_uint(hi);
  }
  if constexpr (D == 128) tmem_st2_x64<64>(taddr, ur); else tmem_st2_x32<32>(taddr, ur);
}

// This thread's half of an O row = U / l to global memory (columns h*D/2 ..), and
// lse from the h = 0 thread.  Every lane runs the TMEM load (it is warp-collective);
// only rows < N are stored.
template <int D>
__device__ __forceinline__ void store_half_row(void* o, float* lse, size_t row_off, int h, bool valid, bool o_fp32,
                                               uint32_t taddr, float l, float m2, float o_mult) {
  uint32_t ur[D / 2];
  if constexpr (D == 128) tmem_ld2_x64<64>(taddr, ur); else tmem_ld2_x32<32>(taddr, ur);
  if (!valid) return;
  const float inv = (l > 0.f) ? o_mult / l : 0.f;
  if (o_fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(o) + row_off * D + h * (D / 2));
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      dst[i] = make_float4(__uint_as_float(ur[4 * i]) * inv, __uint_as_float(ur[4 * i + 1]) * inv,
                           __uint_as_float(ur[4 * i + 2]) * inv, __uint_as_float(ur[4 * i + 3]) * inv);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + row_off * D + h * (D / 2));
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      uint4 w;
      w.x = pack_bf16(__uint_as_float(ur[8 * i + 0]) * inv, __uint_as_float(ur[8 * i + 1]) * inv);
      w.y = pack_bf16(__uint_as_float(ur[8 * i + 2]) * inv, __uint_as_float(ur[8 * i + 3]) * inv);
      w.z = pack_bf16(__uint_as_float(ur[8 * i + 4]) * inv, __uint_as_float(ur[8 * i + 5]) * inv);
      w.w = pack_bf16(__uint_as_float(ur[8 * i + 6]) * inv, __uint_as_float(ur[8 * i + 7]) * inv);
      dst[i] = w;
    }
  }
  if (h == 0) lse[row_off] = (l > 0.f) ? (m2 + log2f(l)) * kLn2 : -INFINITY;
}

// This thread's half of a partial (U, m, l) row for a key shard: U unnormalised (relative to
// exp(s - m)), m in natural-log units, l; an empty row (no admissible key) gets m = -inf,
// l = 0 and no U.
template <int D>
__device__ __forceinline__ void store_half_partial(const FwdAux& aux, size_t slot, int h, bool valid, uint32_t taddr,
                                                   float l, float m2, bool have_u) {
  uint32_t ur[D / 2];
  if (have_u) {
    if constexpr (D == 128) tmem_ld2_x64<64>(taddr, ur); else tmem_ld2_x32<32>(taddr, ur);
  }
  if (!valid) return;
  const bool empty = !(l > 0.f);
  if (!empty) {  // an empty partial's U is never read (the combine skips m = -inf)
    float4* dst = reinterpret_cast<float4*>(aux.u_part + slot * D + h * (D / 2));
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      dst[i] = make_float4(__uint_as_float(ur[4 * i]), __uint_as_float(ur[4 * i + 1]),
                           __uint_as_float(ur[4 * i + 2]), __uint_as_float(ur[4 * i + 3]));
  }
  if (h == 0) {
    aux.m_part[slot] = empty ? -INFINITY : m2 * kLn2;
    aux.l_part[slot] = empty ? 0.f : l;
  }
}

// The new running row max, in exponent units (scores x c), from this thread's 64 scores of
// the row (sr, raw fp32 bits; those from index `nvalid` on are masked to -inf in place) joined
// with the other half of the row held by lane ^ 16.
__device__ __forceinline__ float row_max_update(uint32_t (&sr)[64], int nvalid, float m2, float c) {
  if (nvalid < 64) {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i >= nvalid) sr[i] = __float_as_uint(-INFINITY);
  }
  float a0 = __uint_as_float(sr[0]), a1 = __uint_as_float(sr[1]);
  float a2 = __uint_as_float(sr[2]), a3 = __uint_as_float(sr[3]);
#pragma unroll
  for (int i = 4; i < 60; i += 8) {
    a0 = fmax3(a0, __uint_as_float(sr[i]), __uint_as_float(sr[i + 1]));
    a1 = fmax3(a1, __uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3]));
    a2 = fmax3(a2, __uint_as_float(sr[i + 4]), __uint_as_float(sr[i + 5]));
    a3 = fmax3(a3, __uint_as_float(sr[i + 6]), __uint_as_float(sr[i + 7]));
  }
  a0 = fmax3(a0, __uint_as_float(sr[60]), __uint_as_float(sr[61]));
  a1 = fmax3(a1, __uint_as_float(sr[62]), __uint_as_float(sr[63]));
  float mx = fmax3(a0, a1, fmaxf(a2, a3));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));  // join the two halves of the row
  return fmaxf(m2, mx * c);
}

// P~ = 2^(s c - m) of this thread's 64 scores as packed bf16 pairs, in place into sr[0..31]
// (entry i holds keys 2i, 2i + 1 of the half row); their fp32 sum goes to rs_a + rs_b.
__device__ __forceinline__ void exp_pack_bf16(uint32_t (&sr)[64], uint64_t c2, uint64_t nmb2, uint64_t& rs_a,
                                              uint64_t& rs_b) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float x0, x1, x2, x3;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), c2, nmb2), x0, x1);
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i + 2]), __uint_as_float(sr[2 * i + 3])), c2, nmb2), x2, x3);
    const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
    rs_a = f2_add(rs_a, f2_pack(p0, p1));
    rs_b = f2_add(rs_b, f2_pack(p2, p3));
    sr[i] = pack_bf16(p0, p1);
    sr[i + 1] = pack_bf16(p2, p3);
  }
}

// One thread per row (d = 128): the row max over its 128 scores (sr: columns 0..63, sr2: 64..127,
// raw fp32 bits; those from index `nvalid` on masked to -inf in place), in exponent units.
__device__ __forceinline__ float row_max_full(uint32_t (&sr)[64], uint32_t (&sr2)[64], int nvalid, float m2, float c) {
  if (nvalid < 128) {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      if (i >= nvalid) sr[i] = __float_as_uint(-INFINITY);
      if (64 + i >= nvalid) sr2[i] = __float_as_uint(-INFINITY);
    }
  }
  float a[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a[k] = fmax3(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1]), __uint_as_float(sr[8 + 2 * k]));
    a[4 + k] = fmax3(__uint_as_float(sr2[2 * k]), __uint_as_float(sr2[2 * k + 1]), __uint_as_float(sr2[8 + 2 * k]));
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a[k] = fmaxf(a[k], __uint_as_float(sr[9 + 2 * k]));
    a[4 + k] = fmaxf(a[4 + k], __uint_as_float(sr2[9 + 2 * k]));
  }
#pragma unroll
  for (int i = 16; i < 64; i += 8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      a[k] = fmax3(a[k], __uint_as_float(sr[i + 2 * k]), __uint_as_float(sr[i + 2 * k + 1]));
      a[4 + k] = fmax3(a[4 + k], __uint_as_float(sr2[i + 2 * k]), __uint_as_float(sr2[i + 2 * k + 1]));
    }
  }
  const float mx = fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
  return fmaxf(m2, mx * c);
}

// One thread per row (d = 128): U_t row *= alpha in two TMEM round trips of 64 columns.
__device__ __forceinline__ void rescale_row128(uint32_t taddr, float alpha) {
  const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t ur[64];
    tmem_ld_x64(taddr + 64u * half, ur);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(ur[2 * i]), __uint_as_float(ur[2 * i + 1])), a2), lo, hi);
      ur[2 * i] = __float_as_uint(lo);
      ur[2 * i + 1] = __float_as_uint(hi);
    }
    tmem_st_x64(taddr + 64u * half, ur);
  }
}

// One thread per row (d = 128): O row = U / l as bf16 into the staged tile (box0: columns 0..63,
// box1: 64..127, 128-byte swizzle), with the proxy fence the TMA store needs.
__device__ __forceinline__ void stage_full_row_bf16(uint32_t box0, uint32_t box1, int r, uint32_t taddr, float mult) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t ur[64];
    tmem_ld_x64(taddr + 64u * half, ur);
    const uint32_t srow = (half ? box1 : box0) + static_cast<uint32_t>(r) * 128u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t* u = ur + 8 * i;
      sts128(srow + ((static_cast<uint32_t>(i) ^ static_cast<uint32_t>(r & 7)) << 4),
             pack_bf16(__uint_as_float(u[0]) * mult, __uint_as_float(u[1]) * mult),
             pack_bf16(__uint_as_float(u[2]) * mult, __uint_as_float(u[3]) * mult),
             pack_bf16(__uint_as_float(u[4]) * mult, __uint_as_float(u[5]) * mult),
             pack_bf16(__uint_as_float(u[6]) * mult, __uint_as_float(u[7]) * mult));
    }
  }
  fence_proxy_async_smem();
}

// One thread per row (d = 128): O row = U * o_mult / l (fp32 or bf16; o_mult carries the E4M3 V
// scale) and lse to global memory, rows < N.
__device__ __forceinline__ void store_full_row(void* o, float* lse, size_t row_off, bool valid, bool o_fp32,
                                               uint32_t taddr, float l, float m2, float o_mult) {
  const float inv = (l > 0.f) ? o_mult / l : 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t ur[64];
    tmem_ld_x64(taddr + 64u * half, ur);
    if (!valid) continue;
    if (o_fp32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(o) + row_off * 128 + 64 * half);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        dst[i] = make_float4(__uint_as_float(ur[4 * i]) * inv, __uint_as_float(ur[4 * i + 1]) * inv,
                             __uint_as_float(ur[4 * i + 2]) * inv, __uint_as_float(ur[4 * i + 3]) * inv);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + row_off * 128 + 64 * half);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint4 w;
        w.x = pack_bf16(__uint_as_float(ur[8 * i + 0]) * inv, __uint_as_float(ur[8 * i + 1]) * inv);
        w.y = pack_bf16(__uint_as_float(ur[8 * i + 2]) * inv, __uint_as_float(ur[8 * i + 3]) * inv);
        w.z = pack_bf16(__uint_as_float(ur[8 * i + 4]) * inv, __uint_as_float(ur[8 * i + 5]) * inv);
        w.w = pack_bf16(__uint_as_float(ur[8 * i + 6]) * inv, __uint_as_float(ur[8 * i + 7]) * inv);
        dst[i] = w;
      }
    }
  }
  if (valid) lse[row_off] = (l > 0.f) ? (m2 + log2f(l)) * kLn2 : -INFINITY;
}

// One thread per row (d = 128): the key shard's partial (U, m, l) of the row, as store_half_partial.
__device__ __forceinline__ void store_full_partial(const FwdAux& aux, size_t slot, bool valid, uint32_t taddr, float l,
                                                   float m2) {
  const bool empty = !(l > 0.f);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t ur[64];
    tmem_ld_x64(taddr + 64u * half, ur);
    if (!valid || empty) continue;
    float4* dst = reinterpret_cast<float4*>(aux.u_part + slot * 128 + 64 * half);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      dst[i] = make_float4(__uint_as_float(ur[4 * i]), __uint_as_float(ur[4 * i + 1]), __uint_as_float(ur[4 * i + 2]),
                           __uint_as_float(ur[4 * i + 3]));
  }
  if (valid) {
    aux.m_part[slot] = empty ? -INFINITY : m2 * kLn2;
    aux.l_part[slot] = empty ? 0.f : l;
  }
}

// lse of this thread's row from the h = 0 thread, rows < N only.
__device__ __forceinline__ void store_lse(float* lse, size_t row_off, int h, bool valid, float l, float m2) {
  if (h == 0 && valid) lse[row_off] = (l > 0.f) ? (m2 + log2f(l)) * kLn2 : -INFINITY;
}

template <int D, bool CAUSAL, bool FP8>
__global__ void __launch_bounds__(FwdCfg<D, FP8>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, void* __restrict__ o, float* __restrict__ lse, int N,
               float sl2, int o_fp32, unsigned long long budget, const FwdAux aux,
               const __grid_constant__ CUtensorMap to) {
  using C = FwdCfg<D, FP8>;
  const float* __restrict__ sq = aux.sq;
  const float* __restrict__ sk = aux.sk;
  const float* __restrict__ sv = aux.sv;
  const int Nk = aux.Nk, koff = aux.koff;  // this launch's keys: global indices koff .. koff + Nk - 1
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
  const uint32_t sBar = base + C::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);
  float* sv_max_slot = reinterpret_cast<float*>(gbase + C::OFF_MISC + 8);
#define BAR(i) (sBar + 8u * static_cast<uint32_t>(i))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();  // a dependent kernel may launch once every CTA has started
  // Heads in aux.ng groups, the longest causal blocks of a group first: the blocks of a head read
  // its K/V prefixes close together in time, from L2.
  int bh, pair;
  grouped_block(aux.ng, bh, pair);
  pair = static_cast<int>(gridDim.y) - 1 - pair;
  const int n_tiles = (Nk + kBc - 1) / kBc;
  // KV steps of each query tile: all key tiles, or (causal) those holding a key at or before
  // its last row; 0 if the tile is past N.
  auto steps_of = [&](int t) {
    const int row0 = pair * kRowsPerCta + t * kBr;
    if (row0 >= N) return 0;
    if (!CAUSAL) return n_tiles;
    const int keys = min(row0 + kBr, N) - koff;  // admissible keys of the tile's last row
    return keys <= 0 ? 0 : min((keys + kBc - 1) / kBc, n_tiles);
  };
  const int n_t0 = steps_of(0), n_t1 = steps_of(1);
  const int n_max = max(n_t0, n_t1);
  if (aux.u_part && n_max == 0) {
    // A key shard that starts after every row of this block: each of the block's rows gets the
    // empty partial (m = -inf, l = 0; U is never read for it), without setting up the pipeline.
    grid_dep_wait();
    for (int i = threadIdx.x; i < kRowsPerCta; i += blockDim.x) {
      const int row = pair * kRowsPerCta + i;
      if (row < N) {
        const size_t slot = (static_cast<size_t>(bh) * N + row) * aux.S + aux.shard;
        aux.m_part[slot] = -INFINITY;
        aux.l_part[slot] = 0.f;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_Q), 1);
    // With an MMA warp per tile, each K (V) stage is released once by every tile that reads it.
    const uint32_t users = C::TWO_ISSUERS ? (n_t0 > 0 ? 1u : 0u) + (n_t1 > 0 ? 1u : 0u) : 1u;
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_KE + s), users);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(BAR(C::B_VF + s), 1);
      mbar_init(BAR(C::B_VE + s), users);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(C::B_SF + t), 1);
      mbar_init(BAR(C::B_PF + t), C::SMW * 32);
      mbar_init(BAR(C::B_SC + t), C::SMW * 32);
      mbar_init(BAR(C::B_OF + t), 1);
    }
    mbar_init(BAR(C::B_DRAIN), 1);
    mbar_init(BAR(C::B_DRAIN + 1), 1);
    mbar_init(BAR(C::B_OW), C::SMW * 32);  // O of tile t staged (bf16 O)
    mbar_init(BAR(C::B_OW + 1), C::SMW * 32);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // Set-up above may overlap the previous kernel in the stream (programmatic launch); every
  // global access below comes after it has completed.
  grid_dep_wait();
  if constexpr (FP8) {
    if (warp == 1) {  // the head's largest V block scale (P~ is quantized relative to it)
      float mv = 0.f;
      for (int i = lane; i < n_tiles; i += 32) mv = fmaxf(mv, sv[static_cast<size_t>(bh) * n_tiles + i]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
      if (lane == 0) *sv_max_slot = mv;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == C::WARP_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(BAR(C::B_Q), 2 * C::QB);
      for (int t = 0; t < 2; ++t)
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(sQ + t * C::QB + h * kBox, &tq, BAR(C::B_Q), h * C::BOX_X, pair * kRowsPerCta + t * kBr, bh);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_max; ++j) {
        const int ks = j % C::KST;
        if (j >= C::KST &&
            !mbar_wait(BAR(C::B_KE + ks), ((j / C::KST) - 1) & 1, abort_flag, budget, &g_fwd_status))
          break;
        mbar_arrive_expect_tx(BAR(C::B_KF + ks), C::KVB);
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(sK + ks * C::KVB + h * kBox, &tk, BAR(C::B_KF + ks), h * C::BOX_X, aux.kload0 + j * kBc, bh);
        k_issued = j + 1;
        const int vs = j % C::VST;
        if (j >= C::VST &&
            !mbar_wait(BAR(C::B_VE + vs), ((j / C::VST) - 1) & 1, abort_flag, budget, &g_fwd_status))
          break;
        mbar_arrive_expect_tx(BAR(C::B_VF + vs), C::KVB);
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(sV + vs * C::KVB + h * kBox, &tv, BAR(C::B_VF + vs), h * C::BOX_X, aux.kload0 + j * kBc, bh);
        v_issued = j + 1;
      }
      // Every copy this CTA started must land before its shared memory is released.
      drain_wait(BAR(C::B_Q), 0, budget);
      for (int j = max(0, k_issued - C::KST); j < k_issued; ++j)
        drain_wait(BAR(C::B_KF + j % C::KST), (j / C::KST) & 1, budget);
      for (int j = max(0, v_issued - C::VST); j < v_issued; ++j)
        drain_wait(BAR(C::B_VF + j % C::VST), (j / C::VST) & 1, budget);
    }
  } else if (C::TWO_ISSUERS && (warp == C::WARP_MMA || warp == C::WARP_MMA + 1)) {
    // ------------------------------------------------------------ MMA issuer of one tile
    if (lane == 0) {
      // bf16 (the separate-P~ schedule is d = 64 only)
      static_assert(!(FP8 && C::TWO_ISSUERS), "E4M3 runs the schedule with P~ aliasing S");
      const int t = warp - C::WARP_MMA;
      const int n = t ? n_t1 : n_t0;
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBr, kBc, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBr, D, 1);
      const uint64_t dq = sdesc_add(sdesc_sw128(sQ, 16, 1024), t * C::QB);
      const uint64_t dk0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sV, kBox, 1024);
      const uint32_t d_s = tmem + t * kBc;
      const uint32_t d_o = tmem + kColO + t * D;
      const uint32_t a_p = tmem + (C::SEP ? C::COL_P + 64u * t : static_cast<uint32_t>(t * kBc));
      auto issue_s = [&](int j) {
        const uint64_t dk = sdesc_add(dk0, (j % C::KST) * C::KVB);
#pragma unroll
        for (int kk = 0; kk < C::ROW / 32; ++kk) {  // 32 bytes of K per MMA
          const uint32_t off = static_cast<uint32_t>(kk >> 2) * kBox + static_cast<uint32_t>(kk & 3) * 32u;
          if (kk == 0) mma_ss_c<0>(d_s, sdesc_add(dq, off), sdesc_add(dk, off), idesc_s);
          else mma_ss_c<1>(d_s, sdesc_add(dq, off), sdesc_add(dk, off), idesc_s);
        }
      };
      auto issue_pv = [&](int j) {
        const uint64_t dv = sdesc_add(dv0, (j % C::VST) * C::KVB);
#pragma unroll
        for (int kk = 0; kk < kBc / C::K_MMA; ++kk) {
          // K_MMA keys per MMA: K_MMA rows x 128 B of each V box; A = P~ in TMEM, 8 columns (16
          // bf16 keys) per MMA
          const uint64_t b = sdesc_add(dv, static_cast<uint32_t>(kk * C::K_MMA) * 128u);
          if (j > 0 || kk > 0) mma_ts_c<1>(d_o, a_p + 8u * kk, b, idesc_o);
          else mma_ts_c<0>(d_o, a_p + 8u * kk, b, idesc_o);
        }
      };
      auto wait = [&](uint32_t bar, uint32_t parity) {
        return mbar_wait(bar, parity, abort_flag, budget, &g_fwd_status);
      };
      bool ok = n > 0 && wait(BAR(C::B_Q), 0) && wait(BAR(C::B_KF), 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        tc_commit(BAR(C::B_SF + t));
        tc_commit(BAR(C::B_KE));
      }
      if constexpr (C::SEP) {
        for (int j = 0; ok && j < n; ++j) {
          if (j + 1 < n) {
            ok = wait(BAR(C::B_SC + t), j & 1) &&
                 wait(BAR(C::B_KF + (j + 1) % C::KST), ((j + 1) / C::KST) & 1);
            if (!ok) break;
            tc_fence_after();
            issue_s(j + 1);
            tc_commit(BAR(C::B_SF + t));
            tc_commit(BAR(C::B_KE + (j + 1) % C::KST));
          }
          ok = wait(BAR(C::B_PF + t), j & 1) && wait(BAR(C::B_VF + j % C::VST), (j / C::VST) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(j);
          tc_commit(BAR(C::B_OF + t));
          tc_commit(BAR(C::B_VE + j % C::VST));
        }
      } else {
        for (int j = 1; ok && j <= n; ++j) {
          ok = wait(BAR(C::B_PF + t), (j - 1) & 1) && wait(BAR(C::B_VF + (j - 1) % C::VST), ((j - 1) / C::VST) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(j - 1);
          if (j < n) {
            ok = wait(BAR(C::B_KF + j % C::KST), (j / C::KST) & 1);
            if (!ok) break;
            tc_fence_after();
            issue_s(j);
          }
          tc_commit(BAR(C::B_SF + t));
          tc_commit(BAR(C::B_VE + (j - 1) % C::VST));
          if (j < n) tc_commit(BAR(C::B_KE + j % C::KST));
        }
      }
      if (n > 0) {
        tc_commit(BAR(C::B_DRAIN + t));
        drain_wait(BAR(C::B_DRAIN + t), 0, budget);
      }
    }
  } else if (!C::TWO_ISSUERS && warp == C::WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer for both tiles
    if constexpr (!C::TWO_ISSUERS) if (lane == 0) {
      // d = 128 (P~ aliasing S), bf16 or E4M3.  S = Q K^T (both K-major); U += P~ V (V MN-major).
      static_assert(!C::SEP, "one MMA warp for both tiles only with P~ aliasing S");
      constexpr uint32_t idesc_s = FP8 ? idesc_e4m3_f32(kBr, kBc, 0) : idesc_bf16_f32(kBr, kBc, 0);
      constexpr uint32_t idesc_o = FP8 ? idesc_e4m3_f32(kBr, D, 1) : idesc_bf16_f32(kBr, D, 1);
      // Descriptors computed once; each MMA below is one 32-bit add plus the tcgen05.mma.
      const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sV, kBox, 1024);
      auto mma_s = [&](bool acc, uint32_t d, uint64_t a, uint64_t b) {
        if constexpr (FP8) {
          if (acc) mma_ss_f8_c<1>(d, a, b, idesc_s); else mma_ss_f8_c<0>(d, a, b, idesc_s);
        } else {
          if (acc) mma_ss_c<1>(d, a, b, idesc_s); else mma_ss_c<0>(d, a, b, idesc_s);
        }
      };
      auto mma_o = [&](bool acc, uint32_t d, uint32_t a, uint64_t b) {
        if constexpr (FP8) {
          if (acc) mma_ts_f8_c<1>(d, a, b, idesc_o); else mma_ts_f8_c<0>(d, a, b, idesc_o);
        } else {
          if (acc) mma_ts_c<1>(d, a, b, idesc_o); else mma_ts_c<0>(d, a, b, idesc_o);
        }
      };
      auto issue_s = [&](int t, int j) {
        const uint64_t dq = sdesc_add(dq0, t * C::QB);
        const uint64_t dk = sdesc_add(dk0, (j % C::KST) * C::KVB);
        const uint32_t d_s = tmem + t * kBc;
#pragma unroll
        for (int kk = 0; kk < C::ROW / 32; ++kk) {  // 32 bytes of K per MMA
          const uint32_t off = static_cast<uint32_t>(kk >> 2) * kBox + static_cast<uint32_t>(kk & 3) * 32u;
          mma_s(kk > 0, d_s, sdesc_add(dq, off), sdesc_add(dk, off));
        }
      };
      auto issue_pv = [&](int t, int j) {
        const uint64_t dv = sdesc_add(dv0, (j % C::VST) * C::KVB);
        const uint32_t a_p = tmem + static_cast<uint32_t>(t * kBc);
        const uint32_t d_o = tmem + kColO + t * D;
        // K_MMA keys per MMA: K_MMA rows x 128 B of each V box (boxes kBox apart along d);
        // the P~ operand advances 8 TMEM columns (32 bytes of each row) per MMA.
#pragma unroll
        for (int kk = 0; kk < kBc / C::K_MMA; ++kk)
          mma_o(j > 0 || kk > 0, d_o, a_p + static_cast<uint32_t>(kk) * 8u,
                sdesc_add(dv, static_cast<uint32_t>(kk * C::K_MMA) * 128u));
      };
      // n_max = 0 (a key shard after both tiles' rows): no K/V is loaded and nothing is issued
      bool ok = n_max > 0 && mbar_wait(BAR(C::B_Q), 0, abort_flag, budget, &g_fwd_status) &&
                mbar_wait(BAR(C::B_KF), 0, abort_flag, budget, &g_fwd_status);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if ((t ? n_t1 : n_t0) > 0) {
            issue_s(t, 0);
            tc_commit(BAR(C::B_SF + t));
          }
        tc_commit(BAR(C::B_KE));
      }
      for (int j = 1; ok && j <= n_max; ++j) {
        // This iteration's operands first (V_{j-1} for the PVs, K_j for the next S; both are
        // normally loaded long before), so that once a tile's P~ is ready its 2x(ROW/32) MMAs
        // issue back to back: a wait between them lets the tensor pipe drain.
        ok = mbar_wait(BAR(C::B_VF + (j - 1) % C::VST), ((j - 1) / C::VST) & 1, abort_flag, budget,
                       &g_fwd_status) &&
             (j >= n_max ||
              mbar_wait(BAR(C::B_KF + j % C::KST), (j / C::KST) & 1, abort_flag, budget, &g_fwd_status));
        if (!ok) break;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nt = t ? n_t1 : n_t0;
          if (!ok || j - 1 >= nt) continue;
          if (!mbar_wait(BAR(C::B_PF + t), (j - 1) & 1, abort_flag, budget, &g_fwd_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(t, j - 1);
          if (j < nt) issue_s(t, j);
          tc_commit(BAR(C::B_SF + t));  // S_t(j) ready, and PV_t(j-1) done: U_t may be rescaled
        }
        if (!ok) break;
        tc_commit(BAR(C::B_VE + (j - 1) % C::VST));
        if (j < n_max) tc_commit(BAR(C::B_KE + j % C::KST));
      }
      // All MMAs must be complete before TMEM is released.
      tc_commit(BAR(C::B_DRAIN));
      drain_wait(BAR(C::B_DRAIN), 0, budget);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = warp / C::SMW;                 // query tile of this warp
    const int quarter = warp & 3;                // TMEM lane quarter this warp may access
    const int sub = C::ONE ? 0 : (warp % C::SMW) >> 2;  // which 16 lanes of the quarter (two threads a row)
    const int h = C::ONE ? 0 : lane >> 4;        // which half of the row's columns (two threads a row)
    const int r = C::ONE ? 32 * quarter + lane : 32 * quarter + 16 * sub + (lane & 15);  // TMEM lane = row
    const int row = pair * kRowsPerCta + t * kBr + r;
    const int n = t ? n_t1 : n_t0;
    const uint32_t lane_addr = static_cast<uint32_t>(C::ONE ? 32 * quarter : 32 * quarter + 16 * sub) << 16;
    const uint32_t t_s = tmem + lane_addr + static_cast<uint32_t>(t * kBc);
    const uint32_t t_o = tmem + lane_addr + kColO + static_cast<uint32_t>(t * D);
    const uint32_t t_p = tmem + lane_addr + C::COL_P + 64u * t;  // separate P~ columns (d = 64)
    const int lim = CAUSAL ? min(row - koff, Nk - 1) : Nk - 1;  // last admissible key of this row (local index)
    const int n_kt = (N + kBc - 1) / kBc;  // FP8 scale blocks per head (FP8 launches have Nk = N, koff = 0)
    // Q block scale (read only for a tile inside N: the scale array has ceil(N/128) entries per head)
    const float sq_t = (FP8 && n > 0) ? sq[static_cast<size_t>(bh) * n_kt + pair * 2 + t] : 1.f;
    const float sv_max = FP8 ? *sv_max_slot : 1.f;
    float m2 = -INFINITY, l = 0.f;  // l: this thread's part of the row sum (all of it, one thread a row)
    bool ok = n > 0;
    // FP8: key tile j's K and V block scales, loaded one step ahead
    const float* sk_h = FP8 ? sk + static_cast<size_t>(bh) * n_kt : nullptr;
    const float* sv_h = FP8 ? sv + static_cast<size_t>(bh) * n_kt : nullptr;
    float sk_next = (FP8 && n > 0) ? sk_h[0] : 1.f, sv_next = (FP8 && n > 0) ? sv_h[0] : 1.f;
    for (int j = 0; ok && j < n; ++j) {
      const float sk_j = sk_next, sv_j = sv_next;
      if (FP8 && j + 1 < n) {
        sk_next = sk_h[j + 1];
        sv_next = sv_h[j + 1];
      }
      ok = wait_all(BAR(C::B_SF + t), j & 1, abort_flag, budget);
      if (!ok) break;
      tc_fence_after();
      // exponent multiplier of this key tile: scale * log2(e), times the dequantization scales (FP8)
      const float cj = FP8 ? sq_t * sk_j * sl2 : sl2;
      const uint64_t c2 = f2_pack(cj, cj);
      uint32_t sr[64], sr2[C::ONE ? 64 : 1];  // one thread a row: columns 0..63 in sr, 64..127 in sr2
      if constexpr (C::ONE) {
        tmem_ld_x64(t_s, sr);
        tmem_ld_x64(t_s + 64, sr2);
      } else {
        tmem_ld2_x64<64>(t_s, sr);  // columns 64h .. 64h+63 of the row
      }
      if constexpr (C::SEP) {
        tc_fence_before();
        mbar_arrive(BAR(C::B_SC + t));  // S_t(j) is in registers: the MMA may overwrite it
      }
      // admissible keys among this thread's 64 (128) columns
      float m_new;
      if constexpr (C::ONE) m_new = row_max_full(sr, sr2, lim - j * kBc + 1, m2, cj);
      else m_new = row_max_update(sr, lim - j * kBc - 64 * h + 1, m2, cj);
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;  // fully-masked guard: alpha = p = 0
      const float alpha = ex2(m2 - mb);
      const uint64_t nmb2 = f2_pack(-mb, -mb);
      uint64_t rs_a = f2_pack(0.f, 0.f), rs_b = rs_a;
      float inv_ps = 1.f;  // FP8: the row sum below is of p * ps; l takes p
      if constexpr (C::SEP) {
        exp_pack_bf16(sr, c2, nmb2, rs_a, rs_b);  // P~ packed in place into sr[0..31]
        // PV_t(j-1) must be done before P~_t(j) overwrites P~_t(j-1) and before U_t is rescaled.
        if (j > 0) {
          ok = wait_all(BAR(C::B_OF + t), (j - 1) & 1, abort_flag, budget);
          if (!ok) break;
          tc_fence_after();
          if (!__all_sync(0xffffffffu, alpha == 1.f)) rescale_half_row<D>(t_o, alpha);
        }
        uint32_t pr[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pr[i] = sr[i];
        tmem_st2_x32<32>(t_p, pr);
      }
      if constexpr (!C::SEP && FP8) {
        // P~ as E4M3 of p * ps, ps = 256 * sv_j / sv_max (<= 256): the V block scale rides on P~ so
        // that U accumulates in one unit for every key tile; ps is folded into the exponent,
        // p * ps = 2^(s c - m + log2 ps).  Four keys a column: the row's 32 packed columns of S_t
        // (K block kk of 32 keys at column 8kk), which its thread has read.
        const float ps = 256.f * sv_j / sv_max;
        inv_ps = sv_max / (256.f * sv_j);
        const uint64_t nmp2 = f2_pack(log2f(ps) - mb, log2f(ps) - mb);
        uint32_t p8[32];
        auto pack4 = [&](const uint32_t* src4) {
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(src4[0]), __uint_as_float(src4[1])), c2, nmp2), x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(src4[2]), __uint_as_float(src4[3])), c2, nmp2), x2, x3);
          const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
          rs_a = f2_add(rs_a, f2_pack(p0, p1));
          rs_b = f2_add(rs_b, f2_pack(p2, p3));
          return pack_e4m3x4(p0, p1, p2, p3);
        };
#pragma unroll
        for (int i = 0; i < 16; ++i) p8[i] = pack4(sr + 4 * i);        // keys 4i .. 4i + 3
#pragma unroll
        for (int i = 0; i < 16; ++i) p8[16 + i] = pack4(sr2 + 4 * i);  // keys 64 + 4i ..
        tmem_st_x32(t_s, p8);
      } else if constexpr (!C::SEP) {
        // P~ packed in place into sr[0..31] and sr2[0..31], then the row's 64 packed columns of
        // S_t (keys 2i, 2i + 1 at column i), which its thread has read
        exp_pack_bf16(sr, c2, nmb2, rs_a, rs_b);
        exp_pack_bf16(sr2, c2, nmb2, rs_a, rs_b);
        tmem_st_x32(t_s, *reinterpret_cast<const uint32_t(*)[32]>(sr));         // keys 0..63
        tmem_st_x32(t_s + 32, *reinterpret_cast<const uint32_t(*)[32]>(sr2));   // keys 64..127
      }
      float s0, s1, s2, s3;
      f2_unpack(rs_a, s0, s1);
      f2_unpack(rs_b, s2, s3);
      l = fmaf(alpha, l, ((s0 + s1) + (s2 + s3)) * inv_ps);
      // PV_t(j-1) is complete (the commit that announced S_t(j) covers it): rescale U_t in place.
      if constexpr (!C::SEP) {
        if (j > 0 && !__all_sync(0xffffffffu, alpha == 1.f)) rescale_row128(t_o, alpha);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR(C::B_PF + t));
      m2 = m_new;
    }
    if (ok) {  // U_t final
      if constexpr (C::SEP) ok = wait_all(BAR(C::B_OF + t), (n - 1) & 1, abort_flag, budget);
      else ok = wait_all(BAR(C::B_SF + t), n & 1, abort_flag, budget);
    }
    if (ok) {
      tc_fence_after();
      const float l_row = C::ONE ? l : l + __shfl_xor_sync(0xffffffffu, l, 16);
      if (aux.u_part) {
        if constexpr (C::ONE)
          store_full_partial(aux, (static_cast<size_t>(bh) * N + row) * aux.S + aux.shard, row < N, t_o, l_row, m2);
        else
          store_half_partial<D>(aux, (static_cast<size_t>(bh) * N + row) * aux.S + aux.shard, h, row < N, t_o, l_row,
                                m2, true);
      } else if (!o_fp32) {
        // bf16 O through shared memory, in buffers this tile no longer reads: Q_t (its S MMAs are
        // complete), which has the O tile's shape for bf16 inputs; for E4M3 inputs Q_t and P~_t
        // (its PV MMAs are complete) hold one 128-row x 128-byte box each.  The tile's first
        // thread stores it with TMA once all 256 threads have written.
        const uint32_t box0 = sQ + static_cast<uint32_t>(t) * C::QB;
        const uint32_t box1 = FP8 ? base + C::OFF_P + static_cast<uint32_t>(t) * C::PB : box0 + kBox;
        store_lse(lse, static_cast<size_t>(bh) * N + row, h, row < N, l_row, m2);
        const float o_mul = (l_row > 0.f) ? (FP8 ? sv_max * (1.f / 256.f) : 1.f) / l_row : 0.f;
        if constexpr (C::ONE) stage_full_row_bf16(box0, box1, r, t_o, o_mul);
        else stage_half_row_bf16<D>(box0, box1, r, h, t_o, o_mul);
        mbar_arrive(BAR(C::B_OW + t));
        if ((warp % C::SMW) == 0 && lane == 0 &&
            mbar_wait(BAR(C::B_OW + t), 0, abort_flag, budget, &g_fwd_status)) {
          for (int hb = 0; hb < D / 64; ++hb)
            tma_store_3d(&to, hb ? box1 : box0, hb * 64, pair * kRowsPerCta + t * kBr, bh);
          bulk_commit();
          bulk_wait_all();  // complete before the CTA exits
        }
      } else {
        if constexpr (C::ONE)
          store_full_row(o, lse, static_cast<size_t>(bh) * N + row, row < N, o_fp32 != 0, t_o, l_row, m2,
                         FP8 ? sv_max * (1.f / 256.f) : 1.f);
        else
          store_half_row<D>(o, lse, static_cast<size_t>(bh) * N + row, h, row < N, o_fp32 != 0, t_o, l_row, m2,
                            FP8 ? sv_max * (1.f / 256.f) : 1.f);
      }
    } else if (aux.u_part && n == 0) {
      // no key of this shard is admissible for the tile: an empty partial, U never touched
      store_half_partial<D>(aux, (static_cast<size_t>(bh) * N + row) * aux.S + aux.shard, h, row < N, t_o, 0.f,
                            -INFINITY, false);
    }
    tmem_wait_st();
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// Persistent forward for non-causal bf16 at d = 64: one CTA per SM walks its work items
// (blockIdx.x, + gridDim.x, ...).  An item is a block of 256 query rows (two tiles) of one (b, h)
// against the keys koff .. koff + Nk - 1, loaded from key row kload; the blocks run in
// (b*h, block) order.  The blocks from n_full on (a partly filled last round) may be cut: into
// ksplit key pieces that leave partial (U, m, l) rows for the combine kernel (aux.lin, the key
// split), or into their two query tiles, each an item of its own (aux.qsplit).  Between items a
// CTA keeps its TMEM, barriers and K/V ring: the next Q is loaded as soon as the last S MMAs of
// the current item have read Q, and the next item's S(0) is issued as soon as the softmax has
// read the current item's last S, under its last steps and epilogue.  The step itself is the
// separate-P~ schedule of fwd_kernel at d = 64, with the S products issued by one thread and
// each tile's PV products by a thread of its own.
struct FwdItem {
  int bh, pair, koff, kload, Nk, n0, n1;
  bool to_part;
  long long srow0;  // partial slot of flat row r (= b*h*N + n): (r - srow0) * smul + sadd
  int smul, sadd;
};

__device__ __forceinline__ FwdItem item_at(int w, const FwdAux& aux, int N) {
  FwdItem I;
  I.koff = aux.koff;
  I.kload = aux.kload0;
  I.Nk = aux.Nk;
  I.to_part = aux.u_part != nullptr && !aux.lin;
  I.srow0 = 0;
  I.smul = aux.S;
  I.sadd = aux.shard;
  const int n_pairs = (N + kRowsPerCta - 1) / kRowsPerCta;
  int u = w, tile = -1;  // tile: the one query tile of a query-split item (-1: both)
  if (aux.qsplit && w >= aux.n_full) {
    u = aux.n_full + (w - aux.n_full) / 2;
    tile = (w - aux.n_full) % 2;
  }
  if (aux.lin && w >= aux.n_full) {
    const int piece = w - aux.n_full;
    u = aux.n_full + piece / aux.ksplit;
    I.sadd = piece % aux.ksplit;
    I.koff = I.sadd * aux.kchunk;
    I.kload = aux.kload0 + I.koff;
    I.Nk = min(aux.kchunk, N - I.koff);
    I.to_part = true;
    I.srow0 = aux.prow0;
    I.smul = aux.ksplit;
  }
  I.bh = u / n_pairs;
  I.pair = u % n_pairs;
  const int n_tiles = (I.Nk + kBc - 1) / kBc;
  I.n0 = tile == 1 ? 0 : n_tiles;  // tile 0 of a block is inside N; a query-split item runs one of the two
  I.n1 = (tile != 0 && I.pair * kRowsPerCta + kBr < N) ? n_tiles : 0;
  return I;
}

template <int D>
__global__ void __launch_bounds__(PersistCfg::THREADS, 1)
    fwd_persist_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, void* __restrict__ o, float* __restrict__ lse,
                       int N, float sl2, int o_fp32, unsigned long long budget, const FwdAux aux,
                       const __grid_constant__ CUtensorMap to) {
  using C = PersistCfg;
  static_assert(D == 64 && C::SEP && !C::P_SMEM, "the persistent forward is the d = 64 schedule");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
  const uint32_t sBar = base + C::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);
#define BAR(i) (sBar + 8u * static_cast<uint32_t>(i))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();  // a dependent kernel (a key split's combine) may launch once every CTA has started
  const int w0 = static_cast<int>(blockIdx.x), w_step = static_cast<int>(gridDim.x), n_items = aux.n_items;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_Q), 1);
    mbar_init(BAR(C::B_QE), 2);
    // Each K (V) stage is released once per tile, by the S issuer (the tile's PV issuer); for a
    // tile with no rows in an item the issuer releases the item's stages without reading them.
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_KE + s), 2);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(BAR(C::B_VF + s), 1);
      mbar_init(BAR(C::B_VE + s), 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(C::B_SF + t), 1);
      mbar_init(BAR(C::B_PF + t), kSoftmaxWarps * 32);
      mbar_init(BAR(C::B_SC + t), kSoftmaxWarps * 32);
      mbar_init(BAR(C::B_OF + t), 1);
    }
    for (int i = 0; i < C::N_ISSUERS; ++i) mbar_init(BAR(C::B_DRAIN + i), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(C::B_OSF + t), 1);                 // O staging of tile t free again
      mbar_init(BAR(C::B_OW + t), kSoftmaxWarps * 32);  // O staging of tile t written
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  grid_dep_wait();  // as in fwd_kernel: global accesses only after the previous kernel completed
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // Barrier phases run on across a CTA's items: K/V stage g of the ring is the CTA's g-th key
  // tile, the per-tile barriers count that tile's steps over all items, and Q's the items.

  if (warp == C::WARP_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int k_issued = 0, v_issued = 0, q_issued = 0, kc = 0;
      bool ok = true;
      for (int w = w0, it = 0; ok && w < n_items; w += w_step, ++it) {
        const FwdItem I = item_at(w, aux, N);
        const int n_max = max(I.n0, I.n1);
        // The previous item's Q is free once both tiles' last S MMAs have completed.
        if (it > 0 && !mbar_wait(BAR(C::B_QE), (it - 1) & 1, abort_flag, budget, &g_fwd_status)) break;
        mbar_arrive_expect_tx(BAR(C::B_Q), 2 * C::QB);
        for (int t = 0; t < 2; ++t)
          for (int h = 0; h < C::NH; ++h)
            tma_load_3d(sQ + t * C::QB + h * kBox, &tq, BAR(C::B_Q), h * C::BOX_X, I.pair * kRowsPerCta + t * kBr,
                        I.bh);
        q_issued = it + 1;
        for (int j = 0; j < n_max; ++j) {
          const int g = kc + j;
          const int ks = g % C::KST;
          if (g >= C::KST &&
              !mbar_wait(BAR(C::B_KE + ks), ((g / C::KST) - 1) & 1, abort_flag, budget, &g_fwd_status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(BAR(C::B_KF + ks), C::KVB);
          for (int h = 0; h < C::NH; ++h)
            tma_load_3d(sK + ks * C::KVB + h * kBox, &tk, BAR(C::B_KF + ks), h * C::BOX_X, I.kload + j * kBc, I.bh);
          k_issued = g + 1;
          const int vs = g % C::VST;
          if (g >= C::VST &&
              !mbar_wait(BAR(C::B_VE + vs), ((g / C::VST) - 1) & 1, abort_flag, budget, &g_fwd_status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(BAR(C::B_VF + vs), C::KVB);
          for (int h = 0; h < C::NH; ++h)
            tma_load_3d(sV + vs * C::KVB + h * kBox, &tv, BAR(C::B_VF + vs), h * C::BOX_X, I.kload + j * kBc, I.bh);
          v_issued = g + 1;
        }
        kc += n_max;
      }
      // Every copy this CTA started must land before its shared memory is released (a Q load is
      // issued only after the previous one was consumed, so only the last can be in flight).
      if (q_issued > 0) drain_wait(BAR(C::B_Q), (q_issued - 1) & 1, budget);
      for (int g = max(0, k_issued - C::KST); g < k_issued; ++g)
        drain_wait(BAR(C::B_KF + g % C::KST), (g / C::KST) & 1, budget);
      for (int g = max(0, v_issued - C::VST); g < v_issued; ++g)
        drain_wait(BAR(C::B_VF + g % C::VST), (g / C::VST) & 1, budget);
    }
  } else if (warp >= kWarpMma && warp < kWarpMma + C::N_ISSUERS) {
    // ------------------------------------------------------------ MMA issuers
    // Three threads: the S products of both tiles (tile 0's step before tile 1's), the PV
    // products of tile 0, those of tile 1, so that no PV issue waits behind the other tile's.
    // S_t(j+1) goes out as soon as the softmax has read S_t(j); PV_t(j) as soon as P~_t(j) is
    // stored.
    if (lane == 0) {
      const int role = warp - kWarpMma;
      const bool s_issuer = role == 0;
      const int t_pv = role - 1;  // the PV issuer's tile
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBr, kBc, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBr, D, 1);
      const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sV, kBox, 1024);
      auto issue_s = [&](int t, int g) {  // S_t = Q_t K^T with K from ring stage g
        const uint64_t dq = sdesc_add(dq0, t * C::QB);
        const uint64_t dk = sdesc_add(dk0, (g % C::KST) * C::KVB);
        const uint32_t d_s = tmem + t * kBc;
#pragma unroll
        for (int kk = 0; kk < C::ROW / 32; ++kk) {  // 32 bytes of K per MMA
          const uint32_t off = static_cast<uint32_t>(kk & 3) * 32u;
          if (kk == 0) mma_ss_c<0>(d_s, sdesc_add(dq, off), sdesc_add(dk, off), idesc_s);
          else mma_ss_c<1>(d_s, sdesc_add(dq, off), sdesc_add(dk, off), idesc_s);
        }
      };
      auto issue_pv = [&](int t, int g, bool first) {  // U_t (+)= P~_t V with V from ring stage g
        const uint64_t dv = sdesc_add(dv0, (g % C::VST) * C::KVB);
        const uint32_t d_o = tmem + kColO + t * D;
        const uint32_t a_p = tmem + C::COL_P + 64u * t;
#pragma unroll
        for (int kk = 0; kk < kBc / C::K_MMA; ++kk) {  // 16 keys per MMA: 8 TMEM columns of P~
          const uint64_t b = sdesc_add(dv, static_cast<uint32_t>(kk * C::K_MMA) * 128u);
          if (!first || kk > 0) mma_ts_c<1>(d_o, a_p + 8u * kk, b, idesc_o);
          else mma_ts_c<0>(d_o, a_p + 8u * kk, b, idesc_o);
        }
      };
      auto wait = [&](uint32_t bar, uint32_t parity) {
        return mbar_wait(bar, parity, abort_flag, budget, &g_fwd_status);
      };
      int g0 = 0, g1 = 0, kc = 0;  // each tile's steps and the CTA's key tiles over the items so far
      bool ok = true, issued = false;
      for (int w = w0, it = 0; ok && w < n_items; w += w_step, ++it) {
        const FwdItem I = item_at(w, aux, N);
        const int n_max = max(I.n0, I.n1);
        if (s_issuer) {
          // This item's Q; a tile with no rows in the item releases its share of Q at once and
          // each K stage of the item unread.
          ok = wait(BAR(C::B_Q), it & 1);
          if (!ok) break;
          if (I.n0 == 0) mbar_arrive(BAR(C::B_QE));
          if (I.n1 == 0) mbar_arrive(BAR(C::B_QE));
          for (int j = 0; ok && j < n_max; ++j) {
            const int gk = kc + j;
            ok = wait(BAR(C::B_KF + gk % C::KST), (gk / C::KST) & 1);
            for (int t = 0; ok && t < 2; ++t) {
              const int n = t ? I.n1 : I.n0, gt = (t ? g1 : g0) + j;
              if (n == 0) {
                mbar_arrive(BAR(C::B_KE + gk % C::KST));
                continue;
              }
              // S_t(j) overwrites S_t(j-1) (over items: the previous item's last S): read first
              ok = gt == 0 || wait(BAR(C::B_SC + t), (gt - 1) & 1);
              if (!ok) break;
              tc_fence_after();
              issue_s(t, gk);
              issued = true;
              tc_commit(BAR(C::B_SF + t));
              tc_commit(BAR(C::B_KE + gk % C::KST));
              if (j + 1 == n) tc_commit(BAR(C::B_QE));  // the tile's last S of the item
            }
          }
        } else {
          const int t = t_pv, n = t ? I.n1 : I.n0, g = t ? g1 : g0;
          for (int j = 0; ok && j < n_max; ++j) {
            const int gv = kc + j;
            ok = wait(BAR(C::B_VF + gv % C::VST), (gv / C::VST) & 1);
            if (!ok) break;
            if (n == 0) {
              mbar_arrive(BAR(C::B_VE + gv % C::VST));
              continue;
            }
            ok = wait(BAR(C::B_PF + t), (g + j) & 1);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, gv, j == 0);
            issued = true;
            tc_commit(BAR(C::B_OF + t));
            tc_commit(BAR(C::B_VE + gv % C::VST));
          }
        }
        g0 += I.n0;
        g1 += I.n1;
        kc += n_max;
      }
      if (issued) {  // all MMAs complete before TMEM is released
        tc_commit(BAR(C::B_DRAIN + role));
        drain_wait(BAR(C::B_DRAIN + role), 0, budget);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps 0-15
    const int t = warp / kSoftmaxWarps;           // query tile of this warp
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int sub = (warp % kSoftmaxWarps) >> 2;  // which 16 lanes of the quarter
    const int h = lane >> 4;                      // which half of the row's columns
    const int r = 32 * quarter + 16 * sub + (lane & 15);  // TMEM lane = row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(32 * quarter + 16 * sub) << 16;
    const uint32_t t_s = tmem + lane_addr + static_cast<uint32_t>(t * kBc);
    const uint32_t t_o = tmem + lane_addr + kColO + static_cast<uint32_t>(t * D);
    const uint32_t t_p = tmem + lane_addr + C::COL_P + 64u * t;
    const uint64_t c2 = f2_pack(sl2, sl2);
    // bf16 O leaves through shared memory and one TMA store per tile and item, issued by the
    // tile's first thread; fp32 O and partials are stored by each thread.
    const bool o_issuer = (warp % kSoftmaxWarps) == 0 && lane == 0;
    const uint32_t o_stage = base + C::OFF_O + static_cast<uint32_t>(t) * (kBr * 128u);
    int g = 0;   // this tile's steps over the items so far: the phases of its SF and OF barriers
    int gi = 0;  // this tile's O tiles staged so far: the phases of its OSF and OW barriers
    bool ok = true;
    for (int w = w0; ok && w < n_items; w += w_step) {
      const FwdItem I = item_at(w, aux, N);
      const int n = t ? I.n1 : I.n0;
      // The staging is free once the previous store has read it (long done by now); one phase
      // per item whose O is staged.
      if (o_issuer && n > 0 && !o_fp32 && !I.to_part) {
        bulk_wait_read_all();
        mbar_arrive(BAR(C::B_OSF + t));
      }
      const int row = I.pair * kRowsPerCta + t * kBr + r;
      const int lim = I.Nk - 1;  // last key of the item (local index)
      float m2 = -INFINITY, l = 0.f;  // l: this thread's half of the row
      for (int j = 0; ok && j < n; ++j) {
        ok = wait_all(BAR(C::B_SF + t), (g + j) & 1, abort_flag, budget);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld2_x64<64>(t_s, sr);  // columns 64h .. 64h+63 of the row
        tc_fence_before();
        mbar_arrive(BAR(C::B_SC + t));  // S_t(j) is in registers: the MMA may overwrite it
        // keys of the item among this thread's 64 columns
        const float m_new = row_max_update(sr, lim - j * kBc - 64 * h + 1, m2, sl2);
        const float mb = (m_new == -INFINITY) ? 0.f : m_new;  // fully-masked guard: alpha = p = 0
        const float alpha = ex2(m2 - mb);
        const uint64_t nmb2 = f2_pack(-mb, -mb);
        uint64_t rs_a = f2_pack(0.f, 0.f), rs_b = rs_a;
        exp_pack_bf16(sr, c2, nmb2, rs_a, rs_b);  // P~ packed in place into sr[0..31]
        // PV_t(j-1) must be done before P~_t(j) overwrites P~_t(j-1) and before U_t is rescaled
        // (for j = 0 the previous item's epilogue waited for its last PV).
        if (j > 0) {
          ok = wait_all(BAR(C::B_OF + t), (g + j - 1) & 1, abort_flag, budget);
          if (!ok) break;
          tc_fence_after();
          if (!__all_sync(0xffffffffu, alpha == 1.f)) rescale_half_row<D>(t_o, alpha);
        }
        {
          uint32_t pr[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pr[i] = sr[i];
          tmem_st2_x32<32>(t_p, pr);
        }
        float s0, s1, s2, s3;
        f2_unpack(rs_a, s0, s1);
        f2_unpack(rs_b, s2, s3);
        l = fmaf(alpha, l, (s0 + s1) + (s2 + s3));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(BAR(C::B_PF + t));
        m2 = m_new;
      }
      if (!ok) break;
      if (n == 0) continue;  // the tile is past N: nothing to write
      ok = wait_all(BAR(C::B_OF + t), (g + n - 1) & 1, abort_flag, budget);  // U_t final
      if (!ok) break;
      g += n;
      tc_fence_after();
      const float l_row = l + __shfl_xor_sync(0xffffffffu, l, 16);
      // (the item is decoded again here rather than kept live through the steps)
      const FwdItem E = item_at(w, aux, N);
      const long long frow = static_cast<long long>(E.bh) * N + row;
      if (E.to_part) {
        store_half_partial<D>(aux, static_cast<size_t>(frow - E.srow0) * E.smul + E.sadd, h, row < N, t_o, l_row, m2,
                              true);
      } else if (o_fp32) {
        store_half_row<D>(o, lse, static_cast<size_t>(frow), h, row < N, true, t_o, l_row, m2, 1.f);
      } else {
        // The staging is free (the previous store has read it); stage this thread's half row.
        ok = wait_all(BAR(C::B_OSF + t), gi & 1, abort_flag, budget);
        if (!ok) break;
        store_lse(lse, static_cast<size_t>(frow), h, row < N, l_row, m2);
        stage_half_row_bf16<D>(o_stage, o_stage, r, h, t_o, (l_row > 0.f) ? 1.f / l_row : 0.f);
        mbar_arrive(BAR(C::B_OW + t));
        if (o_issuer) {
          ok = mbar_wait(BAR(C::B_OW + t), gi & 1, abort_flag, budget, &g_fwd_status);
          if (ok) {
            tma_store_3d(&to, o_stage, 0, E.pair * kRowsPerCta + t * kBr, E.bh);
            bulk_commit();
          }
        }
        ++gi;
      }
      // The U_t loads above complete (tcgen05.wait::ld) before this thread's first P~-ready
      // arrival of the next item, after which PV_t(0) of that item may overwrite U_t.
    }
    if (o_issuer) bulk_wait_all();  // the stores complete before the CTA exits
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One launch of `kern` (a forward kernel) with programmatic stream serialization: its set-up may
// overlap the previous kernel in the stream.
template <typename Kern, typename... Args>
cudaError_t launch_kernel(Kern kern, dim3 grid, int threads, uint32_t smem, cudaStream_t stream, Args... args) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D, bool CAUSAL, bool FP8 = false>
cudaError_t launch_t(const FwdLaunch& a, cudaStream_t stream) {
  using C = FwdCfg<D, FP8>;
  const int n_pairs = (a.N + kRowsPerCta - 1) / kRowsPerCta;
  FwdAux aux = a.aux;
  if constexpr (!CAUSAL && !FP8 && D == 64) {
    // the persistent kernel: one CTA per SM over the work items
    const long long units = static_cast<long long>(a.BH) * n_pairs;
    const long long items = aux.lin      ? aux.n_full + (units - aux.n_full) * aux.ksplit
                            : aux.qsplit ? aux.n_full + (units - aux.n_full) * 2
                                         : units;
    if (items > INT_MAX) return cudaErrorInvalidValue;
    aux.n_items = static_cast<int>(items);
    const dim3 grid(static_cast<unsigned>(a.sms > 0 ? std::min<long long>(items, a.sms) : items));
    return launch_kernel(fwd_persist_kernel<D>, grid, PersistCfg::THREADS, PersistCfg::SMEM, stream, a.tq, a.tk, a.tv, a.o,
                         a.lse, a.N, a.scale_log2, a.o_fp32, a.budget, aux, a.to);
  } else {
    // one CTA per block of 256 query rows (a split last round is planned for the persistent kernel only)
    if (aux.lin) return cudaErrorInvalidValue;
    aux.ng = head_groups(a.BH, n_pairs, CAUSAL, a.sms);
    const dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>(n_pairs));
    return launch_kernel(fwd_kernel<D, CAUSAL, FP8>, grid, C::THREADS, C::SMEM, stream, a.tq, a.tk, a.tv, a.o, a.lse,
                         a.N, a.scale_log2, a.o_fp32, a.budget, aux, a.to);
  }
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
  if (a.fp8) return a.causal ? launch_t<128, true, true>(a, stream) : launch_t<128, false, true>(a, stream);
  if (a.d == 64) return a.causal ? launch_t<64, true>(a, stream) : launch_t<64, false>(a, stream);
  return a.causal ? launch_t<128, true>(a, stream) : launch_t<128, false>(a, stream);
}

unsigned int fwd_read_and_clear_status() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(zero));
  return v;
}

}  // namespace fattn
