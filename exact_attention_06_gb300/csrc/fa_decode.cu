// Split-KV single-token decode and the log-sum-exp combine, for sm_103a.
//
// FlashDecoding split-K (cnblogs jzssuanfa FlashAttention page, §三 场景 B):
// the query row of each (batch, head) is broadcast to every split of its KV
// cache; each CTA streams one split, keeps an online-softmax state and writes
// one partial (U, m, l); a second kernel merges the partials with the rule
// m = max m_s, l = sum e^(m_s - m) l_s, O = sum e^(m_s - m) U_s / l
// (iceferryling "FlashAttention 1 和 FlashAttention 2 的区别", §6).
//
// Decode moves 2 * L * d * 2 bytes of K/V per row for 4 * L * d flops, so it
// is bound by HBM bandwidth (iceferryling §13).  The split kernel therefore
// only has to keep enough bytes in flight: one producer thread issues 2-D TMA
// tile loads (64 keys x 64 dims, 128-byte swizzle) into a 3-stage shared
// memory ring; four compute warps consume it.  Within a stage, warp w owns
// keys 16w..16w+15:
//   scores: lane l takes key (l & 15) and half (l >> 4) of d; the swizzle puts
//           the 8 rows a quarter-warp reads in distinct banks; one shuffle
//           joins the halves.  q is pre-scaled by scale * log2(e).
//   values: lane l takes 16-byte column chunk (l % (d/8)) and every
//           (32/(d/8))-th key; p comes from the owning lane by shuffle.
// Each warp keeps its own (m, l, U); the four are merged through shared
// memory at the end with the same rule as the combine kernel.
//
// Paged KV cache (iceferryling §13: decode kernels read the cache through a
// paged block table): K and V live in pools of pages [P, H, page_size, d];
// sequence b's logical page i is pool page block_table[b][i], and its length
// is seq_lens[b].  The split kernel then copies the split's page ids into
// shared memory once and points each 64-key TMA tile at (page * H + head,
// key % page_size); a page id outside [0, P) reads as zero rows (the TMA
// out-of-bounds fill).  Keys at or past seq_lens[b] are masked and their V
// rows skipped, so whatever a partly filled page holds there never reaches O.
#include <cuda_bf16.h>

#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace fattn {

__device__ unsigned int g_dec_status = 0;

namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr int kNw = 4;                        // compute warps
constexpr int kSk = kDecodeStageKeys;         // keys per stage (16 per compute warp)
constexpr int kSt = 3;                        // ring stages
constexpr int kThreads = (kNw + 1) * 32;      // + one producer warp
static_assert(kSk == 16 * kNw, "each compute warp owns 16 keys of a stage");

template <int D>
struct DecCfg {
  static constexpr int NH = D / 64;
  static constexpr uint32_t BOX = kSk * 128u;   // bytes of one [kSk keys x 64 dims] box
  static constexpr uint32_t TB = NH * BOX;      // bytes of K (or V) per stage
  static constexpr int B_KF = 0, B_VF = kSt, B_EMPTY = 2 * kSt, NBAR = 3 * kSt;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = kSt * TB;
  static constexpr uint32_t OFF_BAR = 2 * kSt * TB;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8u * NBAR;       // abort flag
  static constexpr uint32_t OFF_RED = OFF_MISC + 16u;              // m_w[kNw], l_w[kNw], U_w[kNw][D]
  static constexpr uint32_t OFF_PAGES = OFF_RED + 4u * (2 * kNw + kNw * D);  // paged: the split's page ids
  static constexpr uint32_t SMEM = OFF_PAGES + 1024u;
  static constexpr uint32_t SMEM_PAGED = OFF_PAGES + 4u * kMaxSplitPages + 1024u;
};

__device__ __forceinline__ bool dwait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget, &g_dec_status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void ddrain_wait(uint32_t bar, uint32_t parity, unsigned long long budget) {
  // A drain never gets less than the default budget, however short the caller's wait budget is.
  if (budget < kDrainBudget) budget = kDrainBudget;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<unsigned long long>(clock64() - t0) > budget) {
      atomicOr(&g_dec_status, kStatusTimeout);
      return;
    }
  }
}

__device__ __forceinline__ float dot8(const uint4& x, const float* q, float acc) {
  acc = fmaf(bf16lo(x.x), q[0], acc);
  acc = fmaf(bf16hi(x.x), q[1], acc);
  acc = fmaf(bf16lo(x.y), q[2], acc);
  acc = fmaf(bf16hi(x.y), q[3], acc);
  acc = fmaf(bf16lo(x.z), q[4], acc);
  acc = fmaf(bf16hi(x.z), q[5], acc);
  acc = fmaf(bf16lo(x.w), q[6], acc);
  acc = fmaf(bf16hi(x.w), q[7], acc);
  return acc;
}

struct PagedArgs {
  const int* block_table;  // [B, max_pages]
  const int* seq_lens;     // [B]
  int H, page_size, max_pages, num_pages;
};

template <int D, bool PAGED>
__global__ void __launch_bounds__(kThreads)
    decode_split_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                        const __nv_bfloat16* __restrict__ q, float* __restrict__ u_part, float* __restrict__ m_part,
                        float* __restrict__ l_part, int L, int splits, int keys_per_split, float sl2,
                        unsigned long long budget, const PagedArgs pg) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sBar = base + C::OFF_BAR;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC);
  float* red = reinterpret_cast<float*>(gbase + C::OFF_RED);
#define BAR(i) (sBar + 8u * static_cast<uint32_t>(i))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();  // the combine may launch once every split CTA has started
  const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(splits));
  const int sp = static_cast<int>(blockIdx.x % static_cast<unsigned>(splits));
  int* page_ids = reinterpret_cast<int*>(gbase + C::OFF_PAGES);
  int Lr = L;  // keys of this row
  int b = 0, head = 0;
  if constexpr (PAGED) {
    b = bh / pg.H;
    head = bh - b * pg.H;
    Lr = min(max(pg.seq_lens[b], 0), L);  // L = the longest sequence the caller planned for
  }
  const long long k0ll = static_cast<long long>(sp) * keys_per_split;
  const int k0 = static_cast<int>(k0ll < Lr ? k0ll : Lr);
  const int k1 = static_cast<int>(k0ll + keys_per_split < Lr ? k0ll + keys_per_split : Lr);
  const int n_st = (k1 - k0 + kSk - 1) / kSk;
  if constexpr (PAGED) {
    // pool page of each logical page this split touches (the host keeps the count <= kMaxSplitPages)
    const int pg0 = k0 / pg.page_size;
    const int npg = k1 > k0 ? (k1 - 1) / pg.page_size - pg0 + 1 : 0;
    for (int i = threadIdx.x; i < npg; i += kThreads) {
      const int id = pg.block_table[static_cast<size_t>(b) * pg.max_pages + pg0 + i];
      page_ids[i] = (id >= 0 && id < pg.num_pages) ? id * pg.H + head : -1;  // -1: outside the pool, reads zeros
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_VF + s), 1);
      mbar_init(BAR(C::B_EMPTY + s), kNw);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kNw) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int issued = 0;
      for (int st = 0; st < n_st; ++st) {
        const int s = st % kSt;
        if (st >= kSt &&
            !mbar_wait(BAR(C::B_EMPTY + s), ((st / kSt) - 1) & 1, abort_flag, budget, &g_dec_status))
          break;
        const int key = k0 + st * kSk;
        int row = key, z = bh;  // contiguous cache: tensor [BH, L, d]
        if constexpr (PAGED) {  // pool [P * H, page_size, d]; a 64-key stage never straddles a page
          row = key % pg.page_size;
          z = page_ids[key / pg.page_size - k0 / pg.page_size];
        }
        mbar_arrive_expect_tx(BAR(C::B_KF + s), C::TB);
        for (int h = 0; h < C::NH; ++h) tma_load_3d(sK + s * C::TB + h * C::BOX, &tk, BAR(C::B_KF + s), h * 64, row, z);
        mbar_arrive_expect_tx(BAR(C::B_VF + s), C::TB);
        for (int h = 0; h < C::NH; ++h) tma_load_3d(sV + s * C::TB + h * C::BOX, &tv, BAR(C::B_VF + s), h * 64, row, z);
        issued = st + 1;
      }
      for (int st = issued - kSt < 0 ? 0 : issued - kSt; st < issued; ++st) {
        ddrain_wait(BAR(C::B_KF + st % kSt), (st / kSt) & 1, budget);
        ddrain_wait(BAR(C::B_VF + st % kSt), (st / kSt) & 1, budget);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    constexpr int CPL = D / 16;  // 16-byte chunks per lane in the score step (half a row)
    constexpr int DC = D / 8;    // 16-byte chunks per row
    constexpr int KG = 32 / DC;  // key groups in the value step
    const int hf = lane >> 4;
    float qf[CPL * 8];
    {
      const uint4* qv = reinterpret_cast<const uint4*>(q + static_cast<size_t>(bh) * D + hf * (D / 2));
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const uint4 x = qv[c];
        qf[8 * c + 0] = bf16lo(x.x) * sl2;
        qf[8 * c + 1] = bf16hi(x.x) * sl2;
        qf[8 * c + 2] = bf16lo(x.y) * sl2;
        qf[8 * c + 3] = bf16hi(x.y) * sl2;
        qf[8 * c + 4] = bf16lo(x.z) * sl2;
        qf[8 * c + 5] = bf16hi(x.z) * sl2;
        qf[8 * c + 6] = bf16lo(x.w) * sl2;
        qf[8 * c + 7] = bf16hi(x.w) * sl2;
      }
    }
    const int kk = warp * 16 + (lane & 15);  // this lane's key in the score step
    const int dc = lane % DC, kg = lane / DC;
    float m = -INFINITY, lsum = 0.f;
    float u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = 0.f;
    bool ok = true;
    for (int st = 0; st < n_st; ++st) {
      const int s = st % kSt;
      const uint32_t par = (st / kSt) & 1;
      ok = dwait_all(BAR(C::B_KF + s), par, abort_flag, budget);
      if (!ok) break;
      const uint32_t kb = sK + s * C::TB;
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; c += 2) {
        const int g0 = hf * CPL + c, g1 = g0 + 1;
        const uint4 x0 = lds128(kb + (g0 >> 3) * C::BOX + kk * 128 + (((g0 & 7) ^ (kk & 7)) << 4));
        const uint4 x1 = lds128(kb + (g1 >> 3) * C::BOX + kk * 128 + (((g1 & 7) ^ (kk & 7)) << 4));
        a0 = dot8(x0, &qf[8 * c], a0);
        a1 = dot8(x1, &qf[8 * c + 8], a1);
      }
      float acc = a0 + a1;
      acc += __shfl_xor_sync(0xffffffffu, acc, 16);
      const float s2 = (k0 + st * kSk + kk < k1) ? acc : -INFINITY;
      float mx = s2;
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      const float m_new = fmaxf(m, mx);
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m - mb);
      const float p = ex2(s2 - mb);
      lsum = fmaf(alpha, lsum, p);
      m = m_new;
      ok = dwait_all(BAR(C::B_VF + s), par, abort_flag, budget);
      if (!ok) break;
      const uint32_t vb = sV + s * C::TB + (dc >> 3) * C::BOX;
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] *= alpha;
#pragma unroll
      for (int i = 0; i < 16 / KG; ++i) {
        const int r = kg + i * KG;  // key within this warp's 16
        const float pk = __shfl_sync(0xffffffffu, p, r);
        const int vk = warp * 16 + r;
        // paged: rows past the sequence hold whatever the page holds; they must not reach U (0 * NaN)
        if (PAGED && k0 + st * kSk + vk >= k1) continue;
        const uint4 x = lds128(vb + vk * 128 + (((dc & 7) ^ (vk & 7)) << 4));
        u[0] = fmaf(pk, bf16lo(x.x), u[0]);
        u[1] = fmaf(pk, bf16hi(x.x), u[1]);
        u[2] = fmaf(pk, bf16lo(x.y), u[2]);
        u[3] = fmaf(pk, bf16hi(x.y), u[3]);
        u[4] = fmaf(pk, bf16lo(x.z), u[4]);
        u[5] = fmaf(pk, bf16hi(x.z), u[5]);
        u[6] = fmaf(pk, bf16lo(x.w), u[6]);
        u[7] = fmaf(pk, bf16hi(x.w), u[7]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::B_EMPTY + s));
    }
    // Warp partial: l over the 16 key lanes, U over the key groups.
    float lt = lsum;
    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 4);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
#pragma unroll
    for (int off = DC; off < 32; off <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] += __shfl_xor_sync(0xffffffffu, u[i], off);
    }
    if (lane == 0) {
      red[warp] = m;
      red[kNw + warp] = lt;
    }
    if (kg == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) red[2 * kNw + warp * D + dc * 8 + i] = u[i];
    }
    named_bar_sync(1, kNw * 32);
    if (threadIdx.x < D) {
      const int t = threadIdx.x;
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kNw; ++w) mm = fmaxf(mm, red[w]);
      const float mb = (mm == -INFINITY) ? 0.f : mm;
      float lw = 0.f, uw = 0.f;
#pragma unroll
      for (int w = 0; w < kNw; ++w) {
        const float wt = ex2(red[w] - mb);
        lw = fmaf(wt, red[kNw + w], lw);
        uw = fmaf(wt, red[2 * kNw + w * D + t], uw);
      }
      const size_t pidx = static_cast<size_t>(bh) * splits + sp;
      u_part[pidx * D + t] = uw;
      if (t == 0) {
        m_part[pidx] = mm * kLn2;  // natural-log units; -inf stays -inf
        l_part[pidx] = lw;
      }
    }
  }
#undef BAR
  __syncthreads();
}

// One warp per row, kCombineRows rows per CTA: lane l holds columns [l*D/32, (l+1)*D/32).
// With at most kCombineFast partials (every split-KV decode of a few splits, the forward's tail
// split) each lane issues all its loads at once -- the row's m and l (the same address in every
// lane) and one vector of each partial's U -- and then merges; an empty partial (m = -inf) gets
// weight 0 and its U and l, whatever they hold, are not used.  More partials: the maxima are
// read 32 at a time (one per lane) and reduced by shuffles, then the partials are merged one by
// one, an empty one without reading its U or l.
constexpr int kCombineRows = 8;
constexpr int kCombineFast = 8;

template <int D, bool OF32>
__global__ void __launch_bounds__(32 * kCombineRows)
    combine_kernel(const float* __restrict__ u_part, const float* __restrict__ m_part,
                   const float* __restrict__ l_part, void* __restrict__ o, float* __restrict__ lse, int R, int S) {
  constexpr int C = D / 32;  // columns per lane: 2 or 4
  using VecC = typename std::conditional<C == 4, float4, float2>::type;
  const int lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kCombineRows + (threadIdx.x >> 5);
  grid_dep_wait();  // launched programmatically after the kernel that writes the partials
  if (r >= R) return;
  const float* mr = m_part + r * S;
  const float* lr = l_part + r * S;
  const float* ur = u_part + r * S * D + lane * C;
  float mm = -INFINITY, lt = 0.f, acc[C];
#pragma unroll
  for (int i = 0; i < C; ++i) acc[i] = 0.f;
  auto add = [&](float w, const VecC& x) {
    acc[0] = fmaf(w, x.x, acc[0]);
    acc[1] = fmaf(w, x.y, acc[1]);
    if constexpr (C == 4) {
      acc[2] = fmaf(w, x.z, acc[2]);
      acc[3] = fmaf(w, x.w, acc[3]);
    }
  };
  if (S <= kCombineFast) {
    float ms[kCombineFast], ls[kCombineFast];
    VecC us[kCombineFast];
#pragma unroll
    for (int s = 0; s < kCombineFast; ++s)
      if (s < S) {
        ms[s] = mr[s];
        ls[s] = lr[s];
        us[s] = *reinterpret_cast<const VecC*>(ur + static_cast<size_t>(s) * D);
        mm = fmaxf(mm, ms[s]);
      }
    if (mm != -INFINITY) {
#pragma unroll
      for (int s = 0; s < kCombineFast; ++s)
        if (s < S && ms[s] != -INFINITY) {
          const float w = expf(ms[s] - mm);
          lt = fmaf(w, ls[s], lt);
          add(w, us[s]);
        }
    }
  } else {
    for (int s = lane; s < S; s += 32) mm = fmaxf(mm, mr[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
    if (mm != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        const float ms = mr[s];
        if (ms == -INFINITY) continue;  // empty partial: weight 0, U and l not read
        const float w = expf(ms - mm);
        lt = fmaf(w, lr[s], lt);
        add(w, *reinterpret_cast<const VecC*>(ur + static_cast<size_t>(s) * D));
      }
    }
  }
  const float inv = lt > 0.f ? 1.f / lt : 0.f;
  if constexpr (OF32) {
    float* orow = static_cast<float*>(o) + r * D + lane * C;
    if constexpr (C == 4)
      *reinterpret_cast<float4*>(orow) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    else
      *reinterpret_cast<float2*>(orow) = make_float2(acc[0] * inv, acc[1] * inv);
  } else if constexpr (C == 4) {
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(o) + r * D + lane * C;
    uint2 w2;
    w2.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    w2.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(orow) = w2;
  } else {
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(o) + r * D + lane * C;
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) lse[r] = lt > 0.f ? mm + logf(lt) : -INFINITY;
}

template <int D, bool PAGED>
cudaError_t launch_split_t(const DecodeLaunch& a, cudaStream_t stream) {
  using C = DecCfg<D>;
  auto kern = decode_split_kernel<D, PAGED>;
  const uint32_t smem = PAGED ? C::SMEM_PAGED : C::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(a.BH) * a.splits);
  const PagedArgs pg{a.block_table, a.seq_lens, a.H, a.page_size, a.max_pages, a.num_pages};
  kern<<<grid, kThreads, smem, stream>>>(a.tk, a.tv, static_cast<const __nv_bfloat16*>(a.q), a.u_part, a.m_part,
                                         a.l_part, a.L, a.splits, a.keys_per_split, a.scale_log2, a.budget, pg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_split(const DecodeLaunch& a, cudaStream_t stream) {
  if (a.block_table) return a.d == 64 ? launch_split_t<64, true>(a, stream) : launch_split_t<128, true>(a, stream);
  return a.d == 64 ? launch_split_t<64, false>(a, stream) : launch_split_t<128, false>(a, stream);
}

cudaError_t launch_combine(const float* u_part, const float* m_part, const float* l_part, void* o, float* lse, int R,
                           int S, int d, int o_fp32, cudaStream_t stream) {
  // Programmatic launch: the combine's CTAs may be scheduled while the kernel before it finishes
  // (they wait in grid_dep_wait), which hides its launch latency.
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>((R + kCombineRows - 1) / kCombineRows));
  cfg.blockDim = dim3(32 * kCombineRows);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (d == 64)
    return o_fp32 ? cudaLaunchKernelEx(&cfg, combine_kernel<64, true>, u_part, m_part, l_part, o, lse, R, S)
                  : cudaLaunchKernelEx(&cfg, combine_kernel<64, false>, u_part, m_part, l_part, o, lse, R, S);
  return o_fp32 ? cudaLaunchKernelEx(&cfg, combine_kernel<128, true>, u_part, m_part, l_part, o, lse, R, S)
                : cudaLaunchKernelEx(&cfg, combine_kernel<128, false>, u_part, m_part, l_part, o, lse, R, S);
}

// Scratch for fa_decode_splitkv_noalloc: the per-split partials live here
// instead of in a caller-provided workspace.  It is a file-scope device array,
// so every GPU that loads this code keeps kNoAllocScratchBytes of it until the
// process exits.  In host code `g_noalloc_scratch` only names a host-side
// stand-in; its device address comes from cudaGetSymbolAddress, once per
// device, with that device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

cudaError_t decode_noalloc_scratch(void** ptr) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

unsigned int decode_read_and_clear_status() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_dec_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_dec_status, &zero, sizeof(zero));
  return v;
}

}  // namespace fattn
