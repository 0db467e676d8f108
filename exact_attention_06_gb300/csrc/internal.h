// Internal interface between the C-ABI host code and the kernel translation
// units.  Not installed; callers use include/fattn.h.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fattn {

// Bits of the per-device status word that kernels raise.
constexpr unsigned int kStatusTimeout = 1u;
// Default per-wait budget in SM cycles (about 2 s), and the least any drain of in-flight copies
// and MMAs gets before a CTA releases its shared memory and TMEM.
constexpr unsigned long long kDefaultBudget = 4000000000ull;
constexpr unsigned long long kDrainBudget = kDefaultBudget;

// Forward (prefill) launch description.  The tensor maps describe q, k, v as
// 3-D tensors {d, N, B*H} (innermost first) with 64 x 128 boxes and 128-byte
// swizzle.
// Per-launch extras of the forward kernel, passed by value.
struct FwdAux {
  const float* sq;  // FP8: block scales [BH, ceil(N/128)] of q, k, v
  const float* sk;
  const float* sv;
  int Nk;           // keys of this launch (= N unless a key shard)
  int koff;         // global index of key 0 (causal masking of a key shard)
  int kload0;       // row of the k, v tensors (as mapped) that holds key 0 of this launch
  float* u_part;    // key shard: partials [BH*N, S, d], [BH*N, S], [BH*N, S]; null = write O, lse
  float* m_part;
  float* l_part;
  int shard, S;
  // Key split of the last round (lin = 1; work items over 256-row query blocks in (b*h, block)
  // order): items [0, n_full) are whole blocks writing O and lse; each later block is split
  // into ksplit key pieces of kchunk keys (items n_full + ksplit*(block - n_full) + piece),
  // and piece s of flat row r (= b*h*N + n) writes partial slot (r - prow0) * ksplit + s.
  int lin;
  int n_full;
  int ksplit;
  int kchunk;
  long long prow0;
  // Query split (persistent kernel, lin = 0): the blocks from n_full on run as two single-tile
  // items each (items n_full + 2*(block - n_full) + tile).
  int qsplit;
  // Persistent CTAs (non-causal bf16 d = 64): the number of work items; set by launch_fwd.
  int n_items;
  // One-block-per-CTA kernel: the heads are dispatched in ng groups (each group's blocks
  // longest first) so that the blocks of a head run close together in time; set by launch_fwd.
  int ng;
};

// Number of head groups for a grid (B*H, P) whose CTAs are ordered by grouped_block.  Causal:
// every group needs enough heads that its work, spread over the SMs, outlasts its longest block
// (about 2P tile steps against P^2 + P per head), or that block runs alone at the end of the
// launch: at least 2 * sms / (P + 1) heads per group.  Non-causal blocks are all alike: about one
// wave of CTAs per group.  Groups of near-equal size, so that no small group is left over.
inline int head_groups(int bh, int n_ranks, bool causal, int sms) {
  if (sms < 1 || n_ranks < 1 || bh < 1) return 1;
  long long min_heads = causal ? (2LL * sms + n_ranks) / (n_ranks + 1) : (sms + n_ranks - 1) / n_ranks;
  if (min_heads < 1) min_heads = 1;
  const long long ng = bh / min_heads;
  return static_cast<int>(ng < 1 ? 1 : ng);
}

struct FwdLaunch {
  CUtensorMap tq, tk, tv;
  CUtensorMap to;  // bf16 O as {d, N, B*H} (persistent kernel's TMA store; unused for fp32 O and partials)
  void* o;
  float* lse;
  int N;
  int BH;
  int d;
  int causal;
  int o_fp32;
  float scale_log2;  // scale * log2(e)
  unsigned long long budget;
  int fp8;            // 1: q, k, v are E4M3 with per-128-row block scales in aux (d = 128)
  int sms;            // SMs of the device: the persistent grid size (0: one CTA per work item)
  FwdAux aux;
};
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream);
unsigned int fwd_read_and_clear_status();

// Split-KV decode launch description.  The tensor maps describe k, v as 3-D
// tensors {d, L, B*H} with 64 x kDecodeStageKeys boxes and 128-byte swizzle.
struct DecodeLaunch {
  CUtensorMap tk, tv;
  const void* q;
  float* u_part;  // [BH, splits, d]
  float* m_part;  // [BH, splits]
  float* l_part;  // [BH, splits]
  void* o;        // [BH, d] bf16
  float* lse;     // [BH]
  int L;
  int BH;
  int d;
  int splits;
  int keys_per_split;  // multiple of 128
  float scale_log2;
  unsigned long long budget;
  // paged KV cache (block_table != nullptr): tk/tv map pools [P * H, page_size, d]
  const int* block_table;  // [B, max_pages]
  const int* seq_lens;     // [B]; L above is the longest length planned for
  int H, page_size, max_pages, num_pages;
};
constexpr int kDecodeStageKeys = 64;  // keys per pipeline stage of the split kernel
constexpr int kMaxSplitPages = 1024;  // page ids one split of the paged decode may touch
constexpr int kDecodeCtasPerSm = 2;   // resident split CTAs per SM (shared-memory bound)
cudaError_t launch_decode_split(const DecodeLaunch& a, cudaStream_t stream);
cudaError_t launch_combine(const float* u_part, const float* m_part, const float* l_part, void* o, float* lse,
                           int R, int S, int d, int o_fp32, cudaStream_t stream);
unsigned int decode_read_and_clear_status();

// Backward launch description: q, k, v, dO as 3-D tensors {d, N, B*H} with
// 64 x 128 boxes and 128-byte swizzle; delta is the caller's [B*H, N] fp32 scratch.
struct BwdLaunch {
  CUtensorMap tq, tk, tv, tdo;
  CUtensorMap tdq, tdk, tdv;  // bf16 gradients as {d, N, B*H} for the TMA stores (unused for fp32)
  const void* o;
  const void* dout;
  const float* lse;
  float* delta;
  void* dq;
  void* dk;
  void* dv;
  int N;
  int BH;
  int d;
  int causal;
  int grad_fp32;
  float scale;
  float scale_log2;
  unsigned long long budget;
  int sms;  // SMs of the device (block order of the dK/dV and dQ kernels)
};
cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t stream);
unsigned int bwd_read_and_clear_status();

// E4M3 block quantization: x [BH, N, d] bf16 -> codes [BH, N, d] bytes, scales [BH, ceil(N/128)].
cudaError_t launch_quant_e4m3(const void* x, void* codes, float* scales, int BH, int N, int d, cudaStream_t stream);

// Fixed device scratch used by fa_decode_splitkv_noalloc in place of a
// caller-provided workspace.  Size limit of that entry point.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
// Device address of that scratch on the current device (looked up once per device).
cudaError_t decode_noalloc_scratch(void** ptr);

}  // namespace fattn
