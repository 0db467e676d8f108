// Host side of the libfattn C ABI: argument validation, TMA tensor-map
// encoding, kernel launches and the status word.  Declared in fattn.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "fattn.h"
#include "internal.h"

namespace {

thread_local char g_last_error[512] = "";

fa_status_t fail(fa_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

fa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------- device info
struct DevInfo {
  bool known = false;
  int major = 0, minor = 0, sms = 0;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

fa_status_t check_device(int* sms) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) return fail(FA_ERR_ARCH, "no CUDA device: %s", cudaGetErrorString(e));
  if (dev >= kMaxDevices) return fail(FA_ERR_ARCH, "device ordinal %d out of range", dev);
  DevInfo info;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_dev[dev].known) {
      DevInfo d;
      if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(FA_ERR_ARCH, "cannot query device %d", dev);
      d.known = true;
      g_dev[dev] = d;
    }
    info = g_dev[dev];
  }
  if (info.major != 10 || info.minor != 3)
    return fail(FA_ERR_ARCH, "device %d has compute capability %d.%d; libfattn is built for sm_103a (10.3)", dev,
                info.major, info.minor);
  if (sms) *sms = info.sms;
  return FA_OK;
}

// ---------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A tensor [batches, rows, d] (d innermost) of bf16 (esz = 2) or bytes (esz = 1, E4M3
// codes) seen as 3-D {d, rows, batches}, loaded in boxes of 128 bytes (64 bf16 or 128
// E4M3 columns) x box_rows rows with 128-byte swizzle.  Rows past `rows` read as zeros.
fa_status_t make_map(CUtensorMap* map, const void* base, int d, long long rows, long long batches, int box_rows,
                     int esz = 2) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batches)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esz, static_cast<cuuint64_t>(rows) * d * esz};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult %d", static_cast<int>(r));
  return FA_OK;
}

using fattn::kDefaultBudget;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct DecodePlan {
  int splits = 0;
  int keys_per_split = 0;
  size_t u_bytes = 0, m_bytes = 0, l_bytes = 0;
  size_t total() const { return u_bytes + m_bytes + l_bytes; }
};

// Splits per (b, h) when the caller passes 0: the fewest that fill the GPU's
// resident split-CTA slots to within 3% in the last wave (or, when even one
// partial per chunk cannot fill one wave, one partial per chunk).
int auto_splits(long long bh, int n_chunks, int sms) {
  const double slots = static_cast<double>(sms) * fattn::kDecodeCtasPerSm;
  int best = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= n_chunks; ++s) {
    const int cps = (n_chunks + s - 1) / s;
    if ((n_chunks + cps - 1) / cps != s) continue;  // would leave a split empty
    const double waves = static_cast<double>(bh) * s / slots;
    const double eff = waves < 1.0 ? waves : waves / std::ceil(waves);
    if (eff >= 0.97) return s;
    if (eff > best_eff + 1e-12) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

fa_status_t plan_decode(int B, int H, int L, int d, int chunk, int splits, int sms, DecodePlan* plan) {
  if (B < 1 || H < 1 || L < 1) return fail(FA_ERR_INVALID_ARG, "B, H and L must be >= 1 (got %d, %d, %d)", B, H, L);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d is not supported (64 or 128)", d);
  if (chunk != 128) return fail(FA_ERR_UNSUPPORTED, "chunk=%d is not supported (128)", chunk);
  const long long bh = static_cast<long long>(B) * H;
  const int n_chunks = (L + chunk - 1) / chunk;
  if (splits < 0 || splits > n_chunks)
    return fail(FA_ERR_INVALID_ARG, "splits=%d must be in [0, %d] for L=%d", splits, n_chunks, L);
  const int s = splits == 0 ? auto_splits(bh, n_chunks, sms) : splits;
  if (bh * s > INT_MAX) return fail(FA_ERR_UNSUPPORTED, "B*H*splits=%lld exceeds the grid limit", bh * s);
  plan->splits = s;
  plan->keys_per_split = ((n_chunks + s - 1) / s) * chunk;
  plan->u_bytes = round256(static_cast<size_t>(bh) * s * d * sizeof(float));
  plan->m_bytes = round256(static_cast<size_t>(bh) * s * sizeof(float));
  plan->l_bytes = round256(static_cast<size_t>(bh) * s * sizeof(float));
  return FA_OK;
}


// Splits for the paged decode: as for the contiguous cache, then raised if a split would
// touch more than kMaxSplitPages pages (only for very long sequences with small pages).
fa_status_t plan_paged(int B, int H, int L, int d, int page_size, int splits, int sms, DecodePlan* plan) {
  fa_status_t st = plan_decode(B, H, L, d, 128, splits, sms, plan);
  if (st != FA_OK) return st;
  auto pages_of = [&](const DecodePlan& p) { return p.keys_per_split / page_size + 1; };
  if (pages_of(*plan) <= fattn::kMaxSplitPages) return FA_OK;
  if (splits != 0)
    return fail(FA_ERR_UNSUPPORTED, "splits=%d gives %d keys per split, more than %d pages of %d keys", splits,
                plan->keys_per_split, fattn::kMaxSplitPages - 1, page_size);
  const int n_chunks = (L + 127) / 128;
  const int chunks_per_split = ((fattn::kMaxSplitPages - 1) * page_size) / 128;
  return plan_decode(B, H, L, d, 128, (n_chunks + chunks_per_split - 1) / chunks_per_split, 0, plan);
}

// The last round of the non-causal d = 64 forward.  With one resident CTA per SM, U blocks of 256
// query rows run in ceil(U / sms) rounds, the last holding rem blocks.  Two ways to spread that
// round over more SMs:
//   key split: each of the rem blocks becomes k key pieces (>= 2 key tiles each) that leave
//     partial (U, m, l) rows, merged by the combine kernel (needs a workspace);
//   query split: each becomes two single-tile items (when 2 * rem <= sms; no workspace).
// Costs are counted in key-tile steps of a whole block: a block costs its n key tiles plus ~2
// of set-up and epilogue, a piece its share plus 2, the combine (with its launch) ~3; a
// single-tile item runs alone on its SM at ~0.72 of a whole block (both measured on GB300).
// The cheapest wins if it saves at least 5 % of the launch; ties go to the query split.
struct TailPlan {
  int ksplit = 1;  // > 1: key split into ksplit pieces
  int qsplit = 0;  // 1: query split (used when there is no key split, with or without a workspace)
  int n_full = 0, kchunk = 0;
  long long prow0 = 0, rows = 0;
  size_t u_bytes = 0, m_bytes = 0, l_bytes = 0;
  size_t total() const { return u_bytes + m_bytes + l_bytes; }
};

TailPlan plan_tail(long long bh, int N, int d, int causal, int sms) {
  TailPlan p;
  if (causal || d != 64 || sms < 1) return p;  // the persistent d = 64 kernel runs the split rounds
  const long long n_pairs = (N + 255) / 256;
  const long long U = bh * n_pairs;
  const int n_tiles = (N + 127) / 128;
  const long long waves = (U + sms - 1) / sms;
  const long long rem = U - (waves - 1) * sms;
  constexpr double kFixed = 2.0, kCombine = 3.0, kSingleTile = 0.72;
  const double t_whole = n_tiles + kFixed;
  const double t_q = 2 * rem <= sms ? kSingleTile * t_whole : t_whole;
  double best_t = t_whole;
  int best_k = 1, best_tpp = n_tiles;
  for (int k = 2; k <= 8 && 2 * k <= n_tiles; ++k) {
    const int tpp = (n_tiles + k - 1) / k;  // key tiles per piece
    if ((n_tiles + tpp - 1) / tpp != k) continue;
    const double t = std::ceil(static_cast<double>(k * rem) / sms) * (tpp + kFixed) + kCombine;
    if (t < best_t - 1e-9) {
      best_t = t;
      best_k = k;
      best_tpp = tpp;
    }
  }
  const double margin = 0.05 * waves * t_whole;
  if (U - rem + 2 * rem > INT_MAX || U - rem + rem * best_k > INT_MAX) return p;
  p.n_full = static_cast<int>(U - rem);
  if (t_q < t_whole - margin) p.qsplit = 1;  // the fallback whenever there is no key split
  if (best_k == 1 || best_t >= t_q || t_whole - best_t < margin) return p;
  p.ksplit = best_k;
  p.kchunk = best_tpp * 128;
  p.prow0 = (p.n_full / n_pairs) * N + (p.n_full % n_pairs) * 256;
  p.rows = bh * N - p.prow0;
  p.u_bytes = round256(static_cast<size_t>(p.rows) * best_k * d * sizeof(float));
  p.m_bytes = round256(static_cast<size_t>(p.rows) * best_k * sizeof(float));
  p.l_bytes = p.m_bytes;
  return p;
}

fa_status_t check_paged_args(int B, int H, int d, int page_size, int max_pages, int num_pages, int max_seq_len) {
  if (B < 1 || H < 1) return fail(FA_ERR_INVALID_ARG, "B and H must be >= 1 (got %d, %d)", B, H);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d is not supported (64 or 128)", d);
  if (page_size < 64 || page_size % 64 != 0)
    return fail(FA_ERR_UNSUPPORTED, "page_size=%d must be a positive multiple of 64", page_size);
  if (max_pages < 1 || num_pages < 1)
    return fail(FA_ERR_INVALID_ARG, "max_pages and num_pages must be >= 1 (got %d, %d)", max_pages, num_pages);
  if (max_seq_len < 1 || static_cast<long long>(max_seq_len) > static_cast<long long>(max_pages) * page_size)
    return fail(FA_ERR_INVALID_ARG, "max_seq_len=%d must be in [1, max_pages * page_size]", max_seq_len);
  if (static_cast<long long>(num_pages) * H > INT_MAX)
    return fail(FA_ERR_UNSUPPORTED, "num_pages*H=%lld exceeds the page index range",
                static_cast<long long>(num_pages) * H);
  return FA_OK;
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status_t status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_ARCH: return "FA_ERR_ARCH";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
  }
  return "FA_ERR_UNKNOWN";
}

const char* fa_last_error(void) { return g_last_error; }

fa_status_t fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                      float scale, int causal, void* stream, const fa_fwd_opts* opts) {
  g_last_error[0] = '\0';
  if (!q || !k || !v || !o || !lse) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (B < 1 || H < 1 || N < 1) return fail(FA_ERR_INVALID_ARG, "B, H and N must be >= 1 (got %d, %d, %d)", B, H, N);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d is not supported (64 or 128)", d);
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const int o_fp32 = opts ? opts->o_fp32 : 0;
  if (o_fp32 != 0 && o_fp32 != 1) return fail(FA_ERR_INVALID_ARG, "opts->o_fp32 must be 0 or 1");
  const long long bh = static_cast<long long>(B) * H;
  if (bh > INT_MAX) return fail(FA_ERR_UNSUPPORTED, "B*H=%lld exceeds the grid limit", bh);
  if ((N + 127) / 128 > 65535) return fail(FA_ERR_UNSUPPORTED, "N=%d exceeds the 65535 query-tile grid limit", N);
  int sms = 0;
  fa_status_t st = check_device(&sms);
  if (st != FA_OK) return st;
  void* ws = opts ? opts->workspace : nullptr;
  TailPlan tail = plan_tail(bh, N, d, causal, sms);
  if (!ws) tail.ksplit = 1;  // no workspace: no key split (the query split still applies)
  if (tail.ksplit > 1) {
    if (opts->workspace_bytes < tail.total())
      return fail(FA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes fa_fwd_workspace_bytes gives",
                  opts->workspace_bytes, tail.total());
    if (!aligned(ws, 256)) return fail(FA_ERR_INVALID_ARG, "opts->workspace must be 256-byte aligned");
  }

  fattn::FwdLaunch a{};
  if ((st = make_map(&a.tq, q, d, N, bh, 128)) != FA_OK) return st;
  if ((st = make_map(&a.tk, k, d, N, bh, 128)) != FA_OK) return st;
  if ((st = make_map(&a.tv, v, d, N, bh, 128)) != FA_OK) return st;
  if (!o_fp32 && (st = make_map(&a.to, o, d, N, bh, 128)) != FA_OK) return st;
  a.o = o;
  a.lse = lse;
  a.N = N;
  a.BH = static_cast<int>(bh);
  a.d = d;
  a.causal = causal;
  a.o_fp32 = o_fp32;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.budget = (opts && opts->wait_budget_cycles) ? opts->wait_budget_cycles : kDefaultBudget;
  a.aux.Nk = N;
  a.sms = sms;
  if (tail.ksplit == 1 && tail.qsplit) {  // the last round's blocks as single query tiles
    a.aux.qsplit = 1;
    a.aux.n_full = tail.n_full;
  }
  if (tail.ksplit > 1) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    a.aux.lin = 1;
    a.aux.n_full = tail.n_full;
    a.aux.ksplit = tail.ksplit;
    a.aux.kchunk = tail.kchunk;
    a.aux.prow0 = tail.prow0;
    a.aux.u_part = reinterpret_cast<float*>(w);
    a.aux.m_part = reinterpret_cast<float*>(w + tail.u_bytes);
    a.aux.l_part = reinterpret_cast<float*>(w + tail.u_bytes + tail.m_bytes);
  }
  cudaGetLastError();  // clear a stale, non-sticky error so that it is not blamed on this launch
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fattn::launch_fwd(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd launch");
  if (tail.ksplit > 1) {
    uint8_t* o_tail = static_cast<uint8_t*>(o) + static_cast<size_t>(tail.prow0) * d * (o_fp32 ? 4 : 2);
    e = fattn::launch_combine(a.aux.u_part, a.aux.m_part, a.aux.l_part, o_tail, lse + tail.prow0,
                              static_cast<int>(tail.rows), tail.ksplit, d, o_fp32, s);
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd tail combine launch");
  }
  return FA_OK;
}

size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int causal) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || (causal != 0 && causal != 1)) return 0;
  int sms = 0;
  if (check_device(&sms) != FA_OK) return 0;
  return plan_tail(static_cast<long long>(B) * H, N, d, causal, sms).total();
}

fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   float scale, int causal, void* stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, stream, nullptr);
}

fa_status_t fa_fwd_partial_ex(const void* q, const void* k, const void* v, float* u_part, float* m_part,
                              float* l_part, int B, int H, int N, int Nk, int key_offset, int kv_rows, int d,
                              float scale, int causal, int shard, int S, void* stream) {
  g_last_error[0] = '\0';
  if (!q || !k || !v || !u_part || !m_part || !l_part) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (B < 1 || H < 1 || N < 1 || Nk < 1)
    return fail(FA_ERR_INVALID_ARG, "B, H, N and Nk must be >= 1 (got %d, %d, %d, %d)", B, H, N, Nk);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d is not supported (64 or 128)", d);
  if (key_offset < 0) return fail(FA_ERR_INVALID_ARG, "key_offset=%d must be >= 0", key_offset);
  if (kv_rows < 0 || (kv_rows > 0 && static_cast<long long>(key_offset) + Nk > kv_rows))
    return fail(FA_ERR_INVALID_ARG, "kv_rows=%d must be 0 or >= key_offset + Nk = %lld", kv_rows,
                static_cast<long long>(key_offset) + Nk);
  if (S < 1 || shard < 0 || shard >= S) return fail(FA_ERR_INVALID_ARG, "shard=%d must be in [0, S=%d)", shard, S);
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(u_part, 16))
    return fail(FA_ERR_INVALID_ARG, "q, k, v and u_part must be 16-byte aligned");
  if (!aligned(m_part, 4) || !aligned(l_part, 4)) return fail(FA_ERR_INVALID_ARG, "m_part, l_part must be 4-byte aligned");
  const long long bh = static_cast<long long>(B) * H;
  if (bh > INT_MAX) return fail(FA_ERR_UNSUPPORTED, "B*H=%lld exceeds the grid limit", bh);
  if ((N + 127) / 128 > 65535) return fail(FA_ERR_UNSUPPORTED, "N=%d exceeds the 65535 query-tile grid limit", N);
  int sms = 0;
  fa_status_t st = check_device(&sms);
  if (st != FA_OK) return st;
  fattn::FwdLaunch a{};
  a.sms = sms;
  if ((st = make_map(&a.tq, q, d, N, bh, 128)) != FA_OK) return st;
  // The shard's own buffers ([B, H, Nk, d]), or the whole key tensors ([B, H, kv_rows, d]) read
  // from row key_offset on.
  const int rows = kv_rows > 0 ? kv_rows : Nk;
  if ((st = make_map(&a.tk, k, d, rows, bh, 128)) != FA_OK) return st;
  if ((st = make_map(&a.tv, v, d, rows, bh, 128)) != FA_OK) return st;
  a.aux.kload0 = kv_rows > 0 ? key_offset : 0;
  a.N = N;
  a.BH = static_cast<int>(bh);
  a.d = d;
  a.causal = causal;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.budget = kDefaultBudget;
  a.aux.Nk = Nk;
  a.aux.koff = key_offset;
  a.aux.u_part = u_part;
  a.aux.m_part = m_part;
  a.aux.l_part = l_part;
  a.aux.shard = shard;
  a.aux.S = S;
  cudaGetLastError();
  cudaError_t e = fattn::launch_fwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_partial launch");
  return FA_OK;
}

fa_status_t fa_fwd_partial(const void* q, const void* k, const void* v, float* u_part, float* m_part,
                           float* l_part, int B, int H, int N, int Nk, int key_offset, int d, float scale, int causal,
                           int shard, int S, void* stream) {
  return fa_fwd_partial_ex(q, k, v, u_part, m_part, l_part, B, H, N, Nk, key_offset, 0, d, scale, causal, shard, S,
                           stream);
}

fa_status_t fa_quantize_e4m3(const void* x, void* codes, float* scales, int B, int H, int N, int d, void* stream) {
  g_last_error[0] = '\0';
  if (!x || !codes || !scales) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (B < 1 || H < 1 || N < 1) return fail(FA_ERR_INVALID_ARG, "B, H and N must be >= 1 (got %d, %d, %d)", B, H, N);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d is not supported (64 or 128)", d);
  if (!aligned(x, 16) || !aligned(codes, 16)) return fail(FA_ERR_INVALID_ARG, "x and codes must be 16-byte aligned");
  if (!aligned(scales, 4)) return fail(FA_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  const long long grid = static_cast<long long>(B) * H * ((N + 127) / 128);
  if (grid > INT_MAX) return fail(FA_ERR_UNSUPPORTED, "B*H*ceil(N/128)=%lld exceeds the grid limit", grid);
  fa_status_t st = check_device(nullptr);
  if (st != FA_OK) return st;
  cudaGetLastError();
  cudaError_t e = fattn::launch_quant_e4m3(x, codes, scales, B * H, N, d, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_quantize_e4m3 launch");
  return FA_OK;
}

fa_status_t fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* sq, const float* sk,
                       const float* sv, void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
                       void* stream, const fa_fwd_opts* opts) {
  g_last_error[0] = '\0';
  if (!q8 || !k8 || !v8 || !sq || !sk || !sv || !o || !lse) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (B < 1 || H < 1 || N < 1) return fail(FA_ERR_INVALID_ARG, "B, H and N must be >= 1 (got %d, %d, %d)", B, H, N);
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "the FP8 forward supports d=128 only (got d=%d)", d);
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(v8, 16) || !aligned(o, 16))
    return fail(FA_ERR_INVALID_ARG, "q8, k8, v8 and o must be 16-byte aligned");
  if (!aligned(lse, 4) || !aligned(sq, 4) || !aligned(sk, 4) || !aligned(sv, 4))
    return fail(FA_ERR_INVALID_ARG, "lse and the scale arrays must be 4-byte aligned");
  const int o_fp32 = opts ? opts->o_fp32 : 0;
  if (o_fp32 != 0 && o_fp32 != 1) return fail(FA_ERR_INVALID_ARG, "opts->o_fp32 must be 0 or 1");
  const long long bh = static_cast<long long>(B) * H;
  if (bh > INT_MAX) return fail(FA_ERR_UNSUPPORTED, "B*H=%lld exceeds the grid limit", bh);
  if ((N + 127) / 128 > 65535) return fail(FA_ERR_UNSUPPORTED, "N=%d exceeds the 65535 query-tile grid limit", N);
  int sms = 0;
  fa_status_t st = check_device(&sms);
  if (st != FA_OK) return st;

  fattn::FwdLaunch a{};
  a.sms = sms;
  if ((st = make_map(&a.tq, q8, d, N, bh, 128, 1)) != FA_OK) return st;
  if ((st = make_map(&a.tk, k8, d, N, bh, 128, 1)) != FA_OK) return st;
  if ((st = make_map(&a.tv, v8, d, N, bh, 128, 1)) != FA_OK) return st;
  if (!o_fp32 && (st = make_map(&a.to, o, d, N, bh, 128)) != FA_OK) return st;
  a.o = o;
  a.lse = lse;
  a.N = N;
  a.BH = static_cast<int>(bh);
  a.d = d;
  a.causal = causal;
  a.o_fp32 = o_fp32;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.budget = (opts && opts->wait_budget_cycles) ? opts->wait_budget_cycles : kDefaultBudget;
  a.fp8 = 1;
  a.aux.sq = sq;
  a.aux.sk = sk;
  a.aux.sv = sv;
  a.aux.Nk = N;
  cudaGetLastError();
  cudaError_t e = fattn::launch_fwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_fp8 launch");
  return FA_OK;
}

size_t fa_decode_workspace_bytes(int B, int H, int L, int d, int chunk, int splits) {
  int sms = 0;
  if (splits == 0) {
    if (check_device(&sms) != FA_OK) return 0;
  }
  DecodePlan plan;
  if (plan_decode(B, H, L, d, chunk, splits, sms, &plan) != FA_OK) return 0;
  return plan.total();
}

fa_status_t fa_decode_splitkv_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                 int L, int d, float scale, int chunk, int splits, void* workspace, size_t ws_bytes,
                                 void* stream, const fa_decode_opts* opts) {
  g_last_error[0] = '\0';
  if (!q || !k || !v || !o || !lse) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  const int o_fp32 = opts ? opts->o_fp32 : 0;
  if (o_fp32 != 0 && o_fp32 != 1) return fail(FA_ERR_INVALID_ARG, "opts->o_fp32 must be 0 or 1");
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (workspace && !aligned(workspace, 256)) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  DecodePlan plan;
  fa_status_t st;
  if (splits != 0) {
    if ((st = plan_decode(B, H, L, d, chunk, splits, 0, &plan)) != FA_OK) return st;
    if (!workspace || ws_bytes < plan.total())
      return fail(FA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes,
                  plan.total());
    if ((st = check_device(nullptr)) != FA_OK) return st;
  } else {
    int sms = 0;
    if ((st = plan_decode(B, H, L, d, chunk, 1, 0, &plan)) != FA_OK) return st;  // argument checks first
    if ((st = check_device(&sms)) != FA_OK) return st;
    if ((st = plan_decode(B, H, L, d, chunk, 0, sms, &plan)) != FA_OK) return st;
  }
  if (!workspace || ws_bytes < plan.total())
    return fail(FA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes,
                plan.total());
  const long long bh = static_cast<long long>(B) * H;
  fattn::DecodeLaunch a{};
  if ((st = make_map(&a.tk, k, d, L, bh, fattn::kDecodeStageKeys)) != FA_OK) return st;
  if ((st = make_map(&a.tv, v, d, L, bh, fattn::kDecodeStageKeys)) != FA_OK) return st;
  char* ws = static_cast<char*>(workspace);
  a.q = q;
  a.u_part = reinterpret_cast<float*>(ws);
  a.m_part = reinterpret_cast<float*>(ws + plan.u_bytes);
  a.l_part = reinterpret_cast<float*>(ws + plan.u_bytes + plan.m_bytes);
  a.o = o;
  a.lse = lse;
  a.L = L;
  a.BH = static_cast<int>(bh);
  a.d = d;
  a.splits = plan.splits;
  a.keys_per_split = plan.keys_per_split;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.budget = (opts && opts->wait_budget_cycles) ? opts->wait_budget_cycles : kDefaultBudget;
  cudaGetLastError();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fattn::launch_decode_split(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv split launch");
  e = fattn::launch_combine(a.u_part, a.m_part, a.l_part, o, lse, a.BH, a.splits, d, o_fp32, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv combine launch");
  return FA_OK;
}

fa_status_t fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int L,
                              int d, float scale, int chunk, int splits, void* workspace, size_t ws_bytes,
                              void* stream) {
  return fa_decode_splitkv_ex(q, k, v, o, lse, B, H, L, d, scale, chunk, splits, workspace, ws_bytes, stream,
                              nullptr);
}

fa_status_t fa_decode_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                      int L, int d, float scale, int chunk, int splits, void* stream) {
  g_last_error[0] = '\0';
  // Size the partials exactly as fa_decode_splitkv would, and refuse what the
  // fixed scratch cannot hold (argument errors are reported as such first).
  DecodePlan plan;
  fa_status_t st;
  if (splits != 0) {
    if ((st = plan_decode(B, H, L, d, chunk, splits, 0, &plan)) != FA_OK) return st;
  } else {
    int sms = 0;
    if ((st = plan_decode(B, H, L, d, chunk, 1, 0, &plan)) != FA_OK) return st;
    if ((st = check_device(&sms)) != FA_OK) return st;
    if ((st = plan_decode(B, H, L, d, chunk, 0, sms, &plan)) != FA_OK) return st;
  }
  if (splits == 0 && plan.total() > fattn::kNoAllocScratchBytes) {
    // The automatic plan does not fit: take the largest smaller split count (that leaves no split
    // empty) whose partials fit.
    const int n_chunks = (L + chunk - 1) / chunk;
    for (int s = plan.splits - 1; s >= 1; --s) {
      const int cps = (n_chunks + s - 1) / s;
      if ((n_chunks + cps - 1) / cps != s) continue;
      DecodePlan p2;
      if ((st = plan_decode(B, H, L, d, chunk, s, 0, &p2)) != FA_OK) return st;
      if (p2.total() <= fattn::kNoAllocScratchBytes) {
        plan = p2;
        break;
      }
    }
  }
  if (plan.total() > fattn::kNoAllocScratchBytes)
    return fail(FA_ERR_WORKSPACE,
                "fa_decode_splitkv_noalloc: B=%d H=%d with %d splits needs %zu bytes of partials, more than its "
                "fixed scratch of %zu bytes; use fewer splits or fa_decode_splitkv with a workspace",
                B, H, plan.splits, plan.total(), fattn::kNoAllocScratchBytes);
  if ((st = check_device(nullptr)) != FA_OK) return st;
  void* scratch = nullptr;
  cudaError_t e = fattn::decode_noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv_noalloc scratch address");
  return fa_decode_splitkv(q, k, v, o, lse, B, H, L, d, scale, chunk, plan.splits, scratch,
                           fattn::kNoAllocScratchBytes, stream);
}


size_t fa_decode_paged_workspace_bytes(int B, int H, int max_seq_len, int d, int page_size, int max_pages,
                                       int splits) {
  const int saved = g_last_error[0];
  DecodePlan plan;
  fa_status_t st = check_paged_args(B, H, d, page_size, max_pages, 1, max_seq_len);
  int sms = 0;
  if (st == FA_OK && splits == 0) st = check_device(&sms);
  if (st == FA_OK) st = plan_paged(B, H, max_seq_len, d, page_size, splits, sms, &plan);
  if (!saved) g_last_error[0] = '\0';
  return st == FA_OK ? plan.total() : 0;
}

fa_status_t fa_decode_paged_ex(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                               const int* seq_lens, void* o, float* lse, int B, int H, int d, int page_size,
                               int max_pages, int num_pages, int max_seq_len, float scale, int splits,
                               void* workspace, size_t ws_bytes, void* stream, const fa_decode_opts* opts) {
  g_last_error[0] = '\0';
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !o || !lse)
    return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  const int o_fp32 = opts ? opts->o_fp32 : 0;
  if (o_fp32 != 0 && o_fp32 != 1) return fail(FA_ERR_INVALID_ARG, "opts->o_fp32 must be 0 or 1");
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(o, 16))
    return fail(FA_ERR_INVALID_ARG, "q, k_pages, v_pages and o must be 16-byte aligned");
  if (!aligned(lse, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return fail(FA_ERR_INVALID_ARG, "lse, block_table and seq_lens must be 4-byte aligned");
  if (workspace && !aligned(workspace, 256)) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  fa_status_t st = check_paged_args(B, H, d, page_size, max_pages, num_pages, max_seq_len);
  if (st != FA_OK) return st;
  if (splits < 0) return fail(FA_ERR_INVALID_ARG, "splits=%d must be >= 0", splits);
  DecodePlan plan;
  int sms = 0;
  if (splits != 0) {
    if ((st = plan_paged(B, H, max_seq_len, d, page_size, splits, 0, &plan)) != FA_OK) return st;
    if (!workspace || ws_bytes < plan.total())
      return fail(FA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes,
                  plan.total());
    if ((st = check_device(nullptr)) != FA_OK) return st;
  } else {
    if ((st = check_device(&sms)) != FA_OK) return st;
    if ((st = plan_paged(B, H, max_seq_len, d, page_size, 0, sms, &plan)) != FA_OK) return st;
  }
  if (!workspace || ws_bytes < plan.total())
    return fail(FA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes,
                plan.total());
  const long long bh = static_cast<long long>(B) * H;
  fattn::DecodeLaunch a{};
  const long long planes = static_cast<long long>(num_pages) * H;
  if ((st = make_map(&a.tk, k_pages, d, page_size, planes, fattn::kDecodeStageKeys)) != FA_OK) return st;
  if ((st = make_map(&a.tv, v_pages, d, page_size, planes, fattn::kDecodeStageKeys)) != FA_OK) return st;
  char* ws = static_cast<char*>(workspace);
  a.q = q;
  a.u_part = reinterpret_cast<float*>(ws);
  a.m_part = reinterpret_cast<float*>(ws + plan.u_bytes);
  a.l_part = reinterpret_cast<float*>(ws + plan.u_bytes + plan.m_bytes);
  a.o = o;
  a.lse = lse;
  a.L = max_seq_len;
  a.BH = static_cast<int>(bh);
  a.d = d;
  a.splits = plan.splits;
  a.keys_per_split = plan.keys_per_split;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.budget = (opts && opts->wait_budget_cycles) ? opts->wait_budget_cycles : kDefaultBudget;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.H = H;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  cudaGetLastError();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fattn::launch_decode_split(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_paged split launch");
  e = fattn::launch_combine(a.u_part, a.m_part, a.l_part, o, lse, a.BH, a.splits, d, o_fp32, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_paged combine launch");
  return FA_OK;
}

fa_status_t fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                            const int* seq_lens, void* o, float* lse, int B, int H, int d, int page_size,
                            int max_pages, int num_pages, int max_seq_len, float scale, int splits, void* workspace,
                            size_t ws_bytes, void* stream) {
  return fa_decode_paged_ex(q, k_pages, v_pages, block_table, seq_lens, o, lse, B, H, d, page_size, max_pages,
                            num_pages, max_seq_len, scale, splits, workspace, ws_bytes, stream, nullptr);
}

fa_status_t fa_combine_ex(const float* u_part, const float* m_part, const float* l_part, void* o, float* lse, int R,
                          int S, int d, int o_fp32, void* stream) {
  g_last_error[0] = '\0';
  if (!u_part || !m_part || !l_part || !o || !lse) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (o_fp32 != 0 && o_fp32 != 1) return fail(FA_ERR_INVALID_ARG, "o_fp32 must be 0 or 1");
  if (R < 1 || S < 1) return fail(FA_ERR_INVALID_ARG, "R and S must be >= 1 (got %d, %d)", R, S);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d is not supported (64 or 128)", d);
  if (!aligned(u_part, 16) || !aligned(o, 16)) return fail(FA_ERR_INVALID_ARG, "u_part and o must be 16-byte aligned");
  if (!aligned(m_part, 4) || !aligned(l_part, 4) || !aligned(lse, 4))
    return fail(FA_ERR_INVALID_ARG, "m_part, l_part and lse must be 4-byte aligned");
  fa_status_t st = check_device(nullptr);
  if (st != FA_OK) return st;
  cudaGetLastError();
  cudaError_t e =
      fattn::launch_combine(u_part, m_part, l_part, o, lse, R, S, d, o_fp32, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_combine launch");
  return FA_OK;
}

fa_status_t fa_combine(const float* u_part, const float* m_part, const float* l_part, void* o, float* lse, int R,
                       int S, int d, void* stream) {
  return fa_combine_ex(u_part, m_part, l_part, o, lse, R, S, d, 0, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  return round256(static_cast<size_t>(B) * H * N * sizeof(float));
}

fa_status_t fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int grad_fp32,
                   void* workspace, size_t ws_bytes, void* stream) {
  return fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, grad_fp32, workspace, ws_bytes,
                   stream, nullptr);
}

fa_status_t fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                      void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int grad_fp32,
                      void* workspace, size_t ws_bytes, void* stream, const fa_bwd_opts* opts) {
  g_last_error[0] = '\0';
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (B < 1 || H < 1 || N < 1) return fail(FA_ERR_INVALID_ARG, "B, H and N must be >= 1 (got %d, %d, %d)", B, H, N);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d is not supported (64 or 128)", d);
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (grad_fp32 != 0 && grad_fp32 != 1) return fail(FA_ERR_INVALID_ARG, "grad_fp32 must be 0 or 1");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return fail(FA_ERR_INVALID_ARG, "q, k, v, o, dout, dq, dk and dv must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const long long bh = static_cast<long long>(B) * H;
  if (bh > INT_MAX) return fail(FA_ERR_UNSUPPORTED, "B*H=%lld exceeds the grid limit", bh);
  if ((N + 127) / 128 > 65535) return fail(FA_ERR_UNSUPPORTED, "N=%d exceeds the 65535 tile grid limit", N);
  const size_t need = fa_bwd_workspace_bytes(B, H, N);
  if (!workspace || ws_bytes < need)
    return fail(FA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes, need);
  if (!aligned(workspace, 256)) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  int sms = 0;
  fa_status_t st = check_device(&sms);
  if (st != FA_OK) return st;
  fattn::BwdLaunch a{};
  a.sms = sms;
  if ((st = make_map(&a.tq, q, d, N, bh, 128)) != FA_OK) return st;
  if ((st = make_map(&a.tk, k, d, N, bh, 128)) != FA_OK) return st;
  if ((st = make_map(&a.tv, v, d, N, bh, 128)) != FA_OK) return st;
  if ((st = make_map(&a.tdo, dout, d, N, bh, 128)) != FA_OK) return st;
  if (!grad_fp32) {
    if ((st = make_map(&a.tdq, dq, d, N, bh, 128)) != FA_OK) return st;
    if ((st = make_map(&a.tdk, dk, d, N, bh, 128)) != FA_OK) return st;
    if ((st = make_map(&a.tdv, dv, d, N, bh, 128)) != FA_OK) return st;
  }
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.delta = static_cast<float*>(workspace);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.N = N;
  a.BH = static_cast<int>(bh);
  a.d = d;
  a.causal = causal;
  a.grad_fp32 = grad_fp32;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.budget = (opts && opts->wait_budget_cycles) ? opts->wait_budget_cycles : kDefaultBudget;
  cudaGetLastError();
  cudaError_t e = fattn::launch_bwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_bwd launch");
  return FA_OK;
}

fa_status_t fa_get_status(void* stream) {
  g_last_error[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_get_status synchronize");
  const unsigned int bits = fattn::fwd_read_and_clear_status() | fattn::decode_read_and_clear_status() |
                            fattn::bwd_read_and_clear_status();
  if (bits & fattn::kStatusTimeout) return fail(FA_ERR_TIMEOUT, "a kernel wait exceeded its budget");
  return FA_OK;
}

}  // extern "C"
