// Fused exact attention forward (prefill) for sm_103a.
//
// One CTA owns one 128-row query tile Q_i of one (batch, head) and scans the
// 128-key tiles K_j, V_j once, FA-2 order (xuesongtap.github.io
// "flash-attention" page, §2.1; triton-tutorial "8. FlashAttention 实战",
// §8.4.1: Q outer and resident, K/V inner and streamed).  Per tile:
//   S_ij = Q_i K_j^T                   tcgen05.mma, bf16 x bf16 -> fp32 in TMEM
//   m_new = max(m, rowmax(S) * c)      c = scale * log2(e)  (exp2 trick, §8.7.3)
//   alpha = 2^(m - m_new),  P~ = 2^(S*c - m_new)  (online softmax, §8.3.3)
//   l = alpha * l + rowsum(P~)         fp32, from the unrounded P~
//   U = alpha * U + bf16(P~) V_j       P~ written back to TMEM as the A operand
// and after the scan O = U / l, lse = (m + log2 l) * ln 2.
//
// Warp roles (FA-3 style producer/consumer split, triton-tutorial §8.10.2,
// re-done with Blackwell's TMA + tcgen05 + TMEM):
//   warps 0-3  softmax: thread t owns query row t of the tile (TMEM lane t),
//              so no cross-thread row reduction is needed (iceferryling
//              "FlashAttention 1 和 FlashAttention 2 的区别", §7-8 split-Q);
//              they also apply the alpha rescale of U and the epilogue.
//   warp 4     TMA producer: Q once, then K_j / V_j into an ST-stage ring.
//   warp 5     MMA issuer (one thread) and TMEM owner.
// TMEM columns: S/P double buffer at 0 and 128 (P~ as packed bf16 in the
// first 64 columns of its S buffer), U at 256..256+d.
//
// Causal: key tiles above the diagonal are never loaded; only the diagonal
// tile masks (col > row -> -inf), and the ragged last tile masks col >= N
// (triton-tutorial §8.7.1 STAGE split; xuesongtap §2.2 last paragraph).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tmem_io.cuh"

namespace fattn {

__device__ unsigned int g_fwd_status = 0;

namespace {

constexpr int kBr = 128;                 // query rows per tile (TMEM lanes, MMA M)
constexpr int kBc = 128;                 // keys per tile
constexpr uint32_t kBox = 128u * 128u;   // bytes of a 128-row x 64-column bf16 box
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static constexpr int NH = D / 64;                // 64-column boxes per row
  static constexpr int ST = (D == 128) ? 2 : 4;    // K/V ring stages
  static constexpr uint32_t QB = NH * kBox;        // bytes of the Q tile
  static constexpr uint32_t KVB = NH * kBox;       // bytes of one K (or V) tile
  static constexpr int B_Q = 0, B_KF = 1, B_VF = B_KF + ST, B_EMPTY = B_VF + ST, B_SF = B_EMPTY + ST,
                       B_PF = B_SF + 2, B_OD = B_PF + 2, B_DRAIN = B_OD + 1, NBAR = B_DRAIN + 1;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = QB;
  static constexpr uint32_t OFF_V = OFF_K + ST * KVB;
  static constexpr uint32_t OFF_BAR = OFF_V + ST * KVB;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8u * NBAR;  // TMEM address slot, abort flag
  static constexpr uint32_t SMEM = OFF_MISC + 16u + 1024u;   // + slack to align the base to 1 KB
};

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget, &g_fwd_status);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag: used to drain in-flight copies
// and MMAs before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long budget) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<unsigned long long>(clock64() - t0) > budget) {
      atomicOr(&g_fwd_status, kStatusTimeout);
      return;
    }
  }
}

template <int D>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[D]);
template <>
__device__ __forceinline__ void tmem_ld_row<64>(uint32_t taddr, uint32_t (&r)[64]) { tmem_ld_x64(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ld_row<128>(uint32_t taddr, uint32_t (&r)[128]) { tmem_ld_x128(taddr, r); }
template <int D>
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const uint32_t (&r)[D]);
template <>
__device__ __forceinline__ void tmem_st_row<64>(uint32_t taddr, const uint32_t (&r)[64]) { tmem_st_x64(taddr, r); }
template <>
__device__ __forceinline__ void tmem_st_row<128>(uint32_t taddr, const uint32_t (&r)[128]) {
  tmem_st_x128(taddr, r);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, void* __restrict__ o, float* __restrict__ lse, int N,
               float sl2, int o_fp32, unsigned long long budget) {
  using C = FwdCfg<D>;
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
  const int bh = blockIdx.x;
  const int qt = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);  // longest causal tiles first
  const int n_tiles = (N + kBc - 1) / kBc;
  const int n_kv = CAUSAL ? min(qt + 1, n_tiles) : n_tiles;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_Q), 1);
    for (int s = 0; s < C::ST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_VF + s), 1);
      mbar_init(BAR(C::B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(C::B_SF + b), 1);
      mbar_init(BAR(C::B_PF + b), kBr);
    }
    mbar_init(BAR(C::B_OD), 1);
    mbar_init(BAR(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(BAR(C::B_Q), C::QB);
      for (int h = 0; h < C::NH; ++h) tma_load_3d(sQ + h * kBox, &tq, BAR(C::B_Q), h * 64, qt * kBr, bh);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % C::ST;
        if (j >= C::ST &&
            !mbar_wait(BAR(C::B_EMPTY + s), ((j / C::ST) - 1) & 1, abort_flag, budget, &g_fwd_status))
          break;
        mbar_arrive_expect_tx(BAR(C::B_KF + s), C::KVB);
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(sK + s * C::KVB + h * kBox, &tk, BAR(C::B_KF + s), h * 64, j * kBc, bh);
        mbar_arrive_expect_tx(BAR(C::B_VF + s), C::KVB);
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(sV + s * C::KVB + h * kBox, &tv, BAR(C::B_VF + s), h * 64, j * kBc, bh);
        issued = j + 1;
      }
      // Every copy this CTA started must land before its shared memory is released.
      drain_wait(BAR(C::B_Q), 0, budget);
      for (int j = issued - C::ST < 0 ? 0 : issued - C::ST; j < issued; ++j) {
        drain_wait(BAR(C::B_KF + j % C::ST), (j / C::ST) & 1, budget);
        drain_wait(BAR(C::B_VF + j % C::ST), (j / C::ST) & 1, budget);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBr, kBc, 0);  // S = Q K^T, both K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBr, D, 1);    // U += P V, V is MN-major
      bool ok = mbar_wait(BAR(C::B_Q), 0, abort_flag, budget, &g_fwd_status);
      tc_fence_after();
      auto issue_s = [&](int j) -> bool {
        const int s = j % C::ST;
        if (!mbar_wait(BAR(C::B_KF + s), (j / C::ST) & 1, abort_flag, budget, &g_fwd_status)) return false;
        tc_fence_after();
        const uint32_t d_s = tmem + ((j & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>(kk >> 2) * kBox + static_cast<uint32_t>(kk & 3) * 32u;
          mma_ss(d_s, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + s * C::KVB + off, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        tc_commit(BAR(C::B_SF + (j & 1)));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv && !issue_s(j + 1)) break;
        if (!mbar_wait(BAR(C::B_PF + (j & 1)), (j >> 1) & 1, abort_flag, budget, &g_fwd_status)) break;
        const int s = j % C::ST;
        if (!mbar_wait(BAR(C::B_VF + s), (j / C::ST) & 1, abort_flag, budget, &g_fwd_status)) break;
        tc_fence_after();
        const uint32_t a_p = tmem + ((j & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < kBc / 16; ++kk) {
          // 16 keys per MMA: 16 rows x 128 B of each 64-column V box; boxes kBox apart along d.
          const uint64_t b_desc = sdesc_sw128(sV + s * C::KVB + static_cast<uint32_t>(kk) * 2048u, kBox, 1024);
          mma_ts(tmem + kColO, a_p + static_cast<uint32_t>(kk) * 8u, b_desc, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(BAR(C::B_OD));
        tc_commit(BAR(C::B_EMPTY + s));
      }
      // All MMAs must be complete before TMEM is released.
      tc_commit(BAR(C::B_DRAIN));
      drain_wait(BAR(C::B_DRAIN), 0, budget);
    }
  } else {
    // ------------------------------------------------------------ softmax warps 0-3
    const int t = threadIdx.x;  // TMEM lane = row within the tile
    const int row = qt * kBr + t;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const int lim = CAUSAL ? min(row, N - 1) : N - 1;  // last admissible key of this row
    float m2 = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      const uint32_t col_s = b ? kColS1 : kColS0;
      ok = wait_all(BAR(C::B_SF + b), (j >> 1) & 1, abort_flag, budget);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld_x128(tmem + lane_addr + col_s, sr);
      const int nvalid = lim - j * kBc + 1;  // admissible keys of this tile for this row
      if (nvalid < kBc) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= nvalid) sr[i] = __float_as_uint(-INFINITY);
      }
      float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
      float mx2 = __uint_as_float(sr[2]), mx3 = __uint_as_float(sr[3]);
#pragma unroll
      for (int i = 4; i < 128; i += 4) {
        mx0 = fmaxf(mx0, __uint_as_float(sr[i]));
        mx1 = fmaxf(mx1, __uint_as_float(sr[i + 1]));
        mx2 = fmaxf(mx2, __uint_as_float(sr[i + 2]));
        mx3 = fmaxf(mx3, __uint_as_float(sr[i + 3]));
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float m_new = fmaxf(m2, mx * sl2);
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;  // fully-masked guard: alpha = p = 0
      const float alpha = ex2(m2 - mb);
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pr[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), sl2, -mb));
        const float p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), sl2, -mb));
        rs0 += p0;
        rs1 += p1;
        pr[i] = pack_bf16(p0, p1);
      }
      l = fmaf(alpha, l, rs0 + rs1);
      tmem_st_x64(tmem + lane_addr + col_s, pr);
      if (j > 0) {
        // U must hold the previous tile's contribution before it is rescaled.
        ok = wait_all(BAR(C::B_OD), (j - 1) & 1, abort_flag, budget);
        if (!ok) break;
        tc_fence_after();
        if (!__all_sync(0xffffffffu, alpha == 1.f)) {
          uint32_t ur[D];
          tmem_ld_row<D>(tmem + lane_addr + kColO, ur);
#pragma unroll
          for (int i = 0; i < D; ++i) ur[i] = __float_as_uint(__uint_as_float(ur[i]) * alpha);
          tmem_st_row<D>(tmem + lane_addr + kColO, ur);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR(C::B_PF + b));
      m2 = m_new;
    }
    if (ok) ok = wait_all(BAR(C::B_OD), (n_kv - 1) & 1, abort_flag, budget);
    if (ok) {
      tc_fence_after();
      uint32_t ur[D];
      tmem_ld_row<D>(tmem + lane_addr + kColO, ur);
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      if (row < N) {
        const size_t off = (static_cast<size_t>(bh) * N + row) * D;
        if (o_fp32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(o) + off);
#pragma unroll
          for (int i = 0; i < D / 4; ++i)
            dst[i] = make_float4(__uint_as_float(ur[4 * i]) * inv, __uint_as_float(ur[4 * i + 1]) * inv,
                                 __uint_as_float(ur[4 * i + 2]) * inv, __uint_as_float(ur[4 * i + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + off);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(ur[8 * i + 0]) * inv, __uint_as_float(ur[8 * i + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(ur[8 * i + 2]) * inv, __uint_as_float(ur[8 * i + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(ur[8 * i + 4]) * inv, __uint_as_float(ur[8 * i + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(ur[8 * i + 6]) * inv, __uint_as_float(ur[8 * i + 7]) * inv);
            dst[i] = w;
          }
        }
        lse[static_cast<size_t>(bh) * N + row] = (l > 0.f) ? (m2 + log2f(l)) * kLn2 : -INFINITY;
      }
    }
    tmem_wait_st();
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const FwdLaunch& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.N + kBr - 1) / kBr;
  dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>(n_tiles));
  kern<<<grid, kThreads, C::SMEM, stream>>>(a.tq, a.tk, a.tv, a.o, a.lse, a.N, a.scale_log2, a.o_fp32, a.budget);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
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
