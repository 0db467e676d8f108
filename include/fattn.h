/*
 * libfattn -- exact fused attention for GB300 (sm_103a): the fused forward
 * (bf16, or E4M3 inputs with block scales), its backward, a split-KV decode
 * (contiguous or paged KV cache), the log-sum-exp combine of partials and a
 * forward over one key shard.  C ABI: plain pointers, sizes and a stream
 * handle.
 *
 * What is computed (per batch b and head h, scores scaled by `scale`):
 *     S = scale * Q K^T,   P = softmax(S) row-wise,   O = P V,
 *     lse_i = m_i + ln(l_i)   (natural log of the scaled scores),
 * in a single tiled pass with online softmax, so that the N x N score and
 * probability matrices never reach device memory (xuesongtap.github.io
 * "flash-attention" page, §1 equation for S, P, O, §2.1 tiling, §2.2 online
 * softmax, §3 saved log-sum-exp; triton-tutorial "8. FlashAttention 实战",
 * §8.3.3 incremental formula and §8.4 kernel walk-through).
 *
 * Conventions shared by every entry point
 *   - Device pointers only (memory the caller allocated with the CUDA runtime
 *     on the current device).  The library allocates nothing, frees nothing
 *     and keeps no state beyond a cached per-device query (arch, SM count),
 *     a per-device status word read by fa_get_status() and the fixed scratch
 *     array of fa_decode_splitkv_noalloc.
 *   - All tensors are contiguous, row-major in the head dimension d.
 *   - `stream` is a cudaStream_t (CUstream) handle; NULL is the legacy
 *     default stream.  Every call is asynchronous on that stream.
 *   - Arguments are checked before anything is launched; a rejected call
 *     returns an error status, writes nothing and launches nothing.  No C++
 *     exception crosses this boundary.  There is no CPU fallback and no
 *     other backend: an unsupported request is an error.
 *   - Supported head dimensions: d = 64 and d = 128 (the FP8 forward: 128).
 *   - Device: compute capability 10.3 (GB300).  Anything else gives
 *     FA_ERR_ARCH.
 */
#ifndef FATTN_H
#define FATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, non-finite or non-positive scale */
  FA_ERR_UNSUPPORTED = 2, /* valid request this library does not implement (e.g. d not in {64, 128}) */
  FA_ERR_ARCH = 3,        /* current device is not compute capability 10.3, or no device */
  FA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
  FA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait expired; its outputs are undefined */
  FA_ERR_WORKSPACE = 6    /* workspace missing or smaller than fa_decode_workspace_bytes() */
} fa_status_t;

/* Options for fa_fwd_ex.  A zero-initialised struct gives fa_fwd's behaviour. */
typedef struct {
  int o_fp32;                            /* 0: O is bf16 (round to nearest even); 1: O is fp32 */
  unsigned long long wait_budget_cycles; /* per-wait spin budget in SM clock cycles; 0 = default (about 2 s) */
  void* workspace;                       /* optional device scratch, 256-byte aligned, for the key split
                                            (fa_fwd_workspace_bytes); NULL: one launch, no split */
  size_t workspace_bytes;                /* its size in bytes */
} fa_fwd_opts;

/*
 * fa_fwd -- fused attention forward (prefill).
 *
 * Follows the FA-2 scan order: a 128-row query tile Q_i stays on chip while
 * the 128-key tiles K_j, V_j stream past it; per tile the running row max m,
 * the denominator l and the unnormalised output U are updated with
 * alpha = exp(m_old - m_new), and O = U / l is formed once after the scan
 * (xuesongtap §2.1-§2.2; triton-tutorial §8.4.1-§8.4.5).
 *
 *   q, k, v  [B, H, N, d] bf16, 16-byte aligned.
 *   o        [B, H, N, d] bf16, 16-byte aligned (written).
 *   lse      [B, H, N] fp32, 4-byte aligned (written): m + ln(l) of the
 *            scaled scores, the statistic a backward pass recomputes P from.
 *   B, H, N  >= 1.   d in {64, 128}.
 *   scale    finite and > 0 (callers usually pass 1/sqrt(d)).
 *   causal   0: every key; 1: query i attends keys j <= i (top-left aligned,
 *            square), masked scores are -inf and tiles above the diagonal
 *            are skipped (triton-tutorial §8.7.1).
 * Returns FA_OK once the kernel is queued.  Kernel-side timeouts are reported
 * by fa_get_status().
 */
fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, float scale, int causal, void* stream);

/* fa_fwd with options (opts may be NULL).  With opts->o_fp32 = 1, `o` is an
 * fp32 [B, H, N, d] tensor.
 *
 * The last round (non-causal, d = 64): the forward works on blocks of 256
 * query rows of a (b, h), one block per SM at a time, so when the last round
 * of blocks only partly fills the SMs most of them idle through it.  Such a
 * round is split, whichever of two ways the plan (by the device's SM count)
 * finds cheaper: its blocks run as their two 128-row query tiles, each on an
 * SM of its own (no workspace); or, given a workspace of
 * fa_fwd_workspace_bytes() bytes, they are cut along the keys into pieces that
 * each leave a partial (U, m, l) per row, which a second kernel merges by the
 * online-softmax rule, as the split-KV decode does (FlashDecoding split-K,
 * cnblogs jzssuanfa page, §三 场景 B).  O and lse are the same function of
 * q, k, v up to rounding order.  With a workspace too small for the plan:
 * FA_ERR_WORKSPACE. */
fa_status_t fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int N, int d, float scale, int causal, void* stream,
                      const fa_fwd_opts* opts);

/* fa_fwd_workspace_bytes -- scratch bytes the key split of fa_fwd_ex's last
 * round needs on the current device for this problem, or 0 when it plans no
 * key split (causal launches, d = 128, last rounds that are nearly full or
 * that the query split serves as well, fewer than 4 key tiles, invalid sizes,
 * no sm_103a device).  The plan depends on the device's SM count. */
size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int causal);

/*
 * fa_fwd_partial -- the forward over one shard of the keys, leaving a partial
 * (U, m, l) per query row for fa_combine instead of O and lse.  This is the
 * sequence-sharded prefill of Ring Attention without the ring: each KV shard
 * is one pass of the forward kernel, and the partials merge by the
 * online-softmax rule (cnblogs jzssuanfa page, §三 场景 A; xuesongtap §5).
 *
 *   q        [B, H, N, d] bf16, 16-byte aligned: every query row.
 *   k, v     [B, H, Nk, d] bf16, 16-byte aligned: the shard's keys, whose
 *            global indices are key_offset .. key_offset + Nk - 1.
 *   u_part   [B*H*N, S, d] fp32, 16-byte aligned: slot `shard` of each row is
 *            written with U = sum_j exp(s_j - m) v_j over the row's admissible
 *            keys of the shard.
 *   m_part,  [B*H*N, S] fp32, 4-byte aligned: slot `shard` gets m (the row max
 *   l_part   of the scaled scores, natural-log units) and l = sum_j exp(s_j - m).
 *            A row with no admissible key in the shard gets m = -inf and
 *            l = 0; its U slot is left as it was (fa_combine does not use it).
 *   causal   1: query i attends global keys j <= i (top-left aligned).
 *   d in {64, 128}; 0 <= shard < S; key_offset >= 0; other arguments as fa_fwd.
 * After one call per shard (any order, any stream order that completes them
 * first), fa_combine(u_part, m_part, l_part, o, lse, B*H*N, S, d) gives the
 * forward over all the shards' keys.
 */
fa_status_t fa_fwd_partial(const void* q, const void* k, const void* v, float* u_part, float* m_part,
                           float* l_part, int B, int H, int N, int Nk, int key_offset, int d,
                           float scale, int causal, int shard, int S, void* stream);

/* fa_fwd_partial reading the shard straight from the whole key tensors, with no per-shard copy:
 *   k, v     [B, H, kv_rows, d] bf16, 16-byte aligned: the full key sequence of every head; the
 *            shard is rows key_offset .. key_offset + Nk - 1 of each head (its global key
 *            indices, as for fa_fwd_partial).  kv_rows >= key_offset + Nk.  Keys of the tensor
 *            outside the shard may be read (a tile that ends inside the shard) and are masked
 *            as inadmissible.
 *   kv_rows  0: k, v are the shard's own [B, H, Nk, d] buffers, exactly fa_fwd_partial.
 * Other arguments, results and errors as fa_fwd_partial (FA_ERR_INVALID_ARG for kv_rows < 0 or
 * kv_rows < key_offset + Nk). */
fa_status_t fa_fwd_partial_ex(const void* q, const void* k, const void* v, float* u_part, float* m_part,
                              float* l_part, int B, int H, int N, int Nk, int key_offset, int kv_rows,
                              int d, float scale, int causal, int shard, int S, void* stream);

/*
 * fa_quantize_e4m3 -- block quantization of Q, K or V for fa_fwd_fp8
 * (triton-tutorial "8. FlashAttention 实战", §8.9.4: one scale per block of
 * 128 rows x d; scale = max|x| / 448, 448 being E4M3's largest finite value).
 *
 *   x        [B, H, N, d] bf16, 16-byte aligned (read).
 *   codes    [B, H, N, d] bytes, 16-byte aligned (written): the E4M3 code
 *            (OCP FP8 E4M3, bias 7, no infinities) of x / scale, rounded to
 *            nearest, ties to even, saturating at +-448; the sign of x is kept.
 *   scales   [B, H, ceil(N/128)] fp32, 4-byte aligned (written): the block's
 *            scale, fp32(max|x| / 448), or 1 for an all-zero block.
 *   B, H, N  >= 1;  d in {64, 128}.
 * The scale and the division are IEEE fp32 operations, so the codes are a
 * deterministic function of x.  Returns FA_OK once the kernel is queued.
 */
fa_status_t fa_quantize_e4m3(const void* x, void* codes, float* scales,
                             int B, int H, int N, int d, void* stream);

/*
 * fa_fwd_fp8 -- fused attention forward on E4M3 inputs (triton-tutorial
 * §8.9.3: both GEMMs in FP8 with fp32 accumulation, the softmax in fp32,
 * P quantized to FP8 before the second GEMM).
 *
 *   q8, k8, v8  [B, H, N, d] E4M3 codes (fa_quantize_e4m3), 16-byte aligned.
 *   sq, sk, sv  [B, H, ceil(N/128)] fp32 block scales, 4-byte aligned:
 *               row r of a head dequantizes as code * s[r / 128].
 *   o           [B, H, N, d] bf16 (fp32 with opts->o_fp32), 16-byte aligned.
 *   lse         [B, H, N] fp32 (written), as for fa_fwd.
 *   d           must be 128 (FA_ERR_UNSUPPORTED otherwise).
 *   scale, causal, opts: as for fa_fwd_ex (opts may be NULL; no split last round:
 *               opts->workspace is not used).
 * Scores are S = (q8 k8^T) * sq_i * sk_j * scale in fp32; P~ of key tile j
 * is stored as E4M3 of p * 256 * sv_j / max_j(sv_j) (p <= 1 after the row
 * max is subtracted), so that P~ V8 accumulates in one unit for every key
 * tile and O = U * max(sv) / 256 / l.  l sums the fp32 p.
 */
fa_status_t fa_fwd_fp8(const void* q8, const void* k8, const void* v8,
                       const float* sq, const float* sk, const float* sv,
                       void* o, float* lse, int B, int H, int N, int d, float scale,
                       int causal, void* stream, const fa_fwd_opts* opts);

/* Options of fa_decode_splitkv_ex and fa_decode_paged_ex.  A zero-initialised
 * struct (or NULL) gives the behaviour of the entry points without _ex. */
typedef struct {
  int o_fp32;                            /* 0: O is bf16 (round to nearest even); 1: O is fp32 [B, H, d] */
  unsigned long long wait_budget_cycles; /* per-wait spin budget of the split kernel in SM clock
                                            cycles; 0 = default (about 2 s).  A wait that runs out
                                            ends the kernel and fa_get_status() reports
                                            FA_ERR_TIMEOUT; O and lse are then undefined. */
} fa_decode_opts;

/*
 * fa_decode_workspace_bytes -- bytes of scratch that fa_decode_splitkv needs.
 *
 * The workspace holds one partial (U [d] fp32, m fp32, l fp32) per (b, h, split).
 * `chunk` is the key granularity of a split (must be 128); `splits` is the
 * number of partials per (b, h), or 0 to let the library choose from L and the
 * current device's SM count.  Returns 0 for invalid arguments.
 */
size_t fa_decode_workspace_bytes(int B, int H, int L, int d, int chunk, int splits);

/*
 * fa_decode_splitkv -- single-token decode with the KV sequence split
 * (FlashDecoding split-K: the query row is broadcast, each split of the KV
 * cache yields a partial (O_partial, m, l), and the partials are merged by
 * the online-softmax rule; cnblogs jzssuanfa page, §三 场景 B; iceferryling
 * "FlashAttention 1 和 FlashAttention 2 的区别", §13 decode is KV-bandwidth
 * bound).
 *
 *   q        [B, H, d] bf16, 16-byte aligned.
 *   k, v     [B, H, L, d] bf16, 16-byte aligned (the KV cache, every key
 *            admissible: no mask).
 *   o        [B, H, d] bf16 (written).   lse [B, H] fp32 (written).
 *   L >= 1.  chunk = 128.  splits in [0, ceil(L/128)], 0 = automatic; each
 *   split covers a whole number of 128-key chunks.  splits = ceil(L/128)
 *   gives one partial per chunk.
 *   workspace, ws_bytes: caller-owned device scratch of at least
 *   fa_decode_workspace_bytes(B, H, L, d, chunk, splits) bytes, 256-byte
 *   aligned; FA_ERR_WORKSPACE if smaller or NULL.  Its contents on return
 *   are the partials in fa_combine's layout (u_part, then m_part, then
 *   l_part, each 256-byte aligned).
 * Two kernels run on `stream`: the split kernel, then the combine kernel.
 */
fa_status_t fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int L, int d, float scale, int chunk, int splits,
                              void* workspace, size_t ws_bytes, void* stream);

/* fa_decode_splitkv with options (opts may be NULL): opts->o_fp32 = 1 makes `o`
 * an fp32 [B, H, d] tensor (16-byte aligned); opts->wait_budget_cycles bounds
 * each wait of the split kernel. */
fa_status_t fa_decode_splitkv_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int L, int d, float scale, int chunk, int splits,
                                 void* workspace, size_t ws_bytes, void* stream, const fa_decode_opts* opts);

/*
 * fa_decode_splitkv_noalloc -- fa_decode_splitkv for callers that cannot
 * allocate device memory.  (The pages have no counterpart to this entry
 * point: it exists for embedding, not for the method.)
 *
 * Some callers are handed only their input and output buffers and may not
 * call cudaMalloc themselves: plugins inside inference runtimes that own all
 * device memory through their own allocator, and request paths that must not
 * pay for, or risk the device-wide synchronisation of, an allocation or a
 * free.  They have no workspace to pass, so this entry point keeps the
 * per-split partials in a fixed array of device memory compiled into the
 * library (FA_NOALLOC_SCRATCH_BYTES, 8 MiB) instead.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 *   Arguments as fa_decode_splitkv, without workspace and ws_bytes.
 *   The partials of B*H rows with S splits take
 *   fa_decode_workspace_bytes(B, H, L, d, chunk, S) bytes; B*H*S*(d+2)*4 bytes
 *   is about the need: e.g. B*H = 2048 rows at d = 128 fit up to 7 splits.
 *   With splits = 0 the split count is the automatic one of fa_decode_splitkv
 *   when its partials fit, else the largest smaller count whose partials fit
 *   (O and lse are the same function of q, k, v either way, up to rounding
 *   order).  An explicit split count whose partials do not fit, or B*H rows
 *   that do not fit even with one split (more than 16131 rows at d = 128),
 *   return FA_ERR_WORKSPACE (fa_last_error() says by how much) and launch
 *   nothing.
 *   Every GPU that loads the library's decode code holds the 8 MiB array until
 *   the process exits.  The first call on each device looks up the array's
 *   device address (cudaGetSymbolAddress) with that device current; make that
 *   first call before any stream capture.
 *   All calls share the one array and it keeps the last call's partials:
 *   nothing in it needs to start at zero (every partial is written before it
 *   is read), but calls whose kernels overlap on the GPU -- on different
 *   streams, or from different host threads -- race on it and give undefined
 *   results.  Serialise them (one stream, or events).
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
fa_status_t fa_decode_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                      int B, int H, int L, int d, float scale, int chunk, int splits,
                                      void* stream);

/*
 * fa_decode_paged -- fa_decode_splitkv over a paged KV cache (iceferryling
 * "FlashAttention 1 和 FlashAttention 2 的区别", §13: decode kernels read the
 * cache through a paged block table).  Same split and combine; only the
 * address of each key changes.
 *
 *   q            [B, H, d] bf16, 16-byte aligned.
 *   k_pages,     [num_pages, H, page_size, d] bf16 pools, 16-byte aligned:
 *   v_pages      page p holds page_size consecutive keys of one sequence for
 *                every head.
 *   block_table  [B, max_pages] int32, 4-byte aligned: logical page i of
 *                sequence b (keys i*page_size .. +page_size-1) is pool page
 *                block_table[b*max_pages + i].  Only the entries covering
 *                seq_lens[b] keys are read.  An id outside [0, num_pages)
 *                reads as zero keys and values (no fault).
 *   seq_lens     [B] int32, 4-byte aligned: keys of sequence b.  Values are
 *                clamped to [0, max_seq_len]; a length of 0 gives O = 0 and
 *                lse = -inf for that sequence.
 *   o [B, H, d] bf16, lse [B, H] fp32 (written), as for fa_decode_splitkv.
 *   page_size    a positive multiple of 64.  max_pages, num_pages >= 1.
 *   max_seq_len  the longest seq_lens value, 1 .. max_pages*page_size: the
 *                host plans the splits for it (the lengths are device data).
 *   splits       partials per (b, h), 0 = chosen from max_seq_len and the SM
 *                count, as for fa_decode_splitkv; a split covers at most
 *                1023 pages (FA_ERR_UNSUPPORTED beyond).
 *   workspace    >= fa_decode_paged_workspace_bytes(...) bytes, 256-byte aligned.
 * Keys at or past seq_lens[b] are masked and their rows never read into O,
 * whatever the page holds there.  Returns FA_OK once both kernels are queued.
 */
size_t fa_decode_paged_workspace_bytes(int B, int H, int max_seq_len, int d, int page_size, int max_pages,
                                       int splits);
fa_status_t fa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                            const int* block_table, const int* seq_lens, void* o, float* lse,
                            int B, int H, int d, int page_size, int max_pages, int num_pages,
                            int max_seq_len, float scale, int splits, void* workspace,
                            size_t ws_bytes, void* stream);
/* fa_decode_paged with options (opts may be NULL), as for fa_decode_splitkv_ex. */
fa_status_t fa_decode_paged_ex(const void* q, const void* k_pages, const void* v_pages,
                               const int* block_table, const int* seq_lens, void* o, float* lse,
                               int B, int H, int d, int page_size, int max_pages, int num_pages,
                               int max_seq_len, float scale, int splits, void* workspace,
                               size_t ws_bytes, void* stream, const fa_decode_opts* opts);

/*
 * fa_combine -- merge S partial (U, m, l) triples per row into O and lse:
 *     m = max_s m_s,  w_s = exp(m_s - m),  l = sum_s w_s l_s,
 *     O = sum_s w_s U_s / l,  lse = m + ln(l)
 * (iceferryling page §6, cross-warp merge formula; the same rule is the
 * FlashDecoding tree reduction and the Ring Attention merge).
 *
 *   u_part [R, S, d] fp32, unnormalised numerators (relative to exp(s - m_s)).
 *   m_part [R, S] fp32, row maxima in natural-log units of scaled scores.
 *   l_part [R, S] fp32, denominators.
 *   An empty partial (m = -inf) has weight 0 and its U and l are not used;
 *   a row whose partials are all empty gets O = 0 and lse = -inf.
 *   o [R, d] bf16 (written), lse [R] fp32 (written).  R, S >= 1, d in {64, 128}.
 *   u_part 16-byte aligned; m_part, l_part, lse 4-byte aligned; o 16-byte aligned.
 */
fa_status_t fa_combine(const float* u_part, const float* m_part, const float* l_part,
                       void* o, float* lse, int R, int S, int d, void* stream);
/* fa_combine with the output type chosen: o_fp32 = 0 writes o [R, d] bf16
 * (round to nearest even), o_fp32 = 1 writes o [R, d] fp32 (16-byte aligned). */
fa_status_t fa_combine_ex(const float* u_part, const float* m_part, const float* l_part,
                          void* o, float* lse, int R, int S, int d, int o_fp32, void* stream);

/*
 * fa_bwd_workspace_bytes -- scratch bytes fa_bwd needs: the per-row
 * D_i = rowsum(O_i * dO_i), B*H*N fp32, rounded up to 256 bytes.  0 for
 * invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N);

/*
 * fa_bwd -- attention backward with recomputation: from Q, K, V, the
 * forward's O and lse, and dO, compute
 *     D  = rowsum(O * dO),   P = exp(scale Q K^T - lse)  (recomputed per tile),
 *     dV = P^T dO,   dS = P * (dO V^T - D),   dQ = scale dS K,   dK = scale dS^T Q
 * (triton-tutorial "8. FlashAttention 实战", §8.8.1-§8.8.4; operatorworld,
 * "反向传播：用重算换显存").  P is never stored: one kernel owns a key tile
 * and produces its dK, dV; another owns a query tile and produces its dQ
 * (no atomics: every output is written by one CTA in a fixed order, so the
 * gradients are bitwise repeatable).
 *
 *   q, k, v, o, dout  [B, H, N, d] bf16, 16-byte aligned; o and lse must be the
 *                     forward's outputs for the same q, k, v, scale, causal.
 *   lse               [B, H, N] fp32 (natural log of scaled scores).
 *   dq, dk, dv        [B, H, N, d], written: bf16, or fp32 when grad_fp32 = 1.
 *   d in {64, 128}; scale finite > 0; causal 0/1 as for fa_fwd.
 *   workspace         >= fa_bwd_workspace_bytes(B, H, N) bytes, 256-byte
 *                     aligned, caller-owned (holds D); FA_ERR_WORKSPACE if
 *                     smaller or NULL.
 * Three kernels run on `stream`: D, then dK/dV, then dQ.
 */
fa_status_t fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   float scale, int causal, int grad_fp32, void* workspace, size_t ws_bytes,
                   void* stream);

/* Options of fa_bwd_ex.  wait_budget_cycles: per-wait budget in SM cycles of
 * the dK/dV and dQ kernels, as in fa_fwd_opts (0 = the default, about 2 s);
 * a wait that runs out ends the kernel, and fa_get_status then reports
 * FA_ERR_TIMEOUT (the gradients are undefined). */
typedef struct fa_bwd_opts {
  unsigned long long wait_budget_cycles;
} fa_bwd_opts;

/* fa_bwd with options; opts may be NULL (then it is fa_bwd).  Arguments,
 * results and errors otherwise as fa_bwd. */
fa_status_t fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                      float scale, int causal, int grad_fp32, void* workspace, size_t ws_bytes,
                      void* stream, const fa_bwd_opts* opts);

/*
 * fa_get_status -- synchronise `stream`, then read and clear the current
 * device's kernel status word.  Returns FA_ERR_TIMEOUT if any kernel of this
 * library ran out of its wait budget since the last call, FA_ERR_CUDA if the
 * synchronisation itself failed, else FA_OK.
 */
fa_status_t fa_get_status(void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* fa_status_string(fa_status_t status);

/* Detail of the most recent error on the calling thread (static thread-local
 * storage, "" if none). */
const char* fa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H */
