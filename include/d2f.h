/*
 * d2f.h -- C ABI of libd2f, the GB300 (sm_103a) hot path of Discrete Diffusion
 * Forcing (D2F) block-diffusion decoding.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀 모델보다 2.5배 빨라지는
 *        방법 (arXiv:2508.09192)"
 *   [P2] "D2F 논문 리뷰: 확산 LLM이 자기회귀 모델보다 빠른 추론을 처음으로
 *        달성한 방식"
 *   [P3] "확산 언어 모델(Diffusion LLM)이란 무엇인가"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named as device buffers are CUDA device (or managed) memory owned
 *   by the caller. The library never allocates, frees or copies between host
 *   and device; it only enqueues kernels.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream). Every call is asynchronous: it validates its host-side arguments,
 *   enqueues its kernel(s) on `stream` and returns without synchronising.
 * - Return value: a d2f_status. D2F_ERR_INVALID_ARG, D2F_ERR_UNSUPPORTED and
 *   D2F_ERR_WORKSPACE are detected on the host before anything is enqueued;
 *   D2F_ERR_CUDA means a launch failed. d2f_last_error_string() gives a
 *   one-line reason for the last non-OK return in the calling thread.
 * - `err_word` (nullable) is a device int32 the caller zeroes. Problems found
 *   on the device (a page id outside [0, num_pages), window metadata that
 *   contradicts the host sizes, a bounded wait that gave up) store the first
 *   error code there with an atomic compare-and-swap; the offending work is
 *   skipped without any out-of-range access, and the caller reads the word
 *   after its own synchronisation. Kernels never trap or assert.
 * - Window metadata: sequence b owns window rows q_start[b] .. q_start[b+1]-1
 *   (n_b rows; q_start[0] = 0, q_start[batch] <= total_q, every q_start value a
 *   multiple of block_size). Row i of sequence b lies in window block i / B.
 *   Global window block jb covers rows jb*B .. jb*B+B-1. total_q may exceed
 *   q_start[batch] (a launch sized for a capacity while the layout is written on
 *   the device, as d2f_window_step does): the rows past q_start[batch] belong to
 *   no sequence, the attention writes nothing for them, and the commit wants them
 *   not masked (masked = 0) and leaves them as they are.
 * - K/V pool layout: [num_pages][num_heads_kv][block_size][head_dim], one page
 *   = one block of B tokens of one sequence ([P1] §운영 관점: block completion
 *   is the cache-persistence signal, so a page holds exactly one block). Token t
 *   of sequence b lives in page page_table[b*max_pages_per_seq + t/B], slot t%B.
 * - GQA: query head h reads KV head h / (num_heads_q / num_heads_kv).
 * - Workspace: caller-provided device memory of at least the size the matching
 *   *_workspace_size query returns. It must be zero-filled before its first use
 *   (e.g. cudaMemsetAsync); every call leaves it ready for the next call on the
 *   same stream. Calls that share one workspace must not overlap in time.
 *
 * Size limits (a call beyond one returns D2F_ERR_UNSUPPORTED before anything is
 * enqueued):
 * - attention: batch * num_heads_kv <= 65535 (one grid dimension); head_dim 64
 *   or 128 with bf16 on the tensor-core path (block_size 8, 16 or 32), any other
 *   case on the CUDA-core path, block_size <= 256;
 * - commit: total_q <= 65535 window rows, block_size 1..32, num_splits <= 64;
 * - window step: one CTA holds the whole window state in shared memory
 *   (block_size <= 128; about 5 bytes per window row of capacity plus per-
 *   sequence state against 227 KB: some 45,000 rows for a small batch);
 * - the no-allocation commit: the scratch bound stated at d2f_commit_noalloc.
 * The workloads this library is measured on (up to 512 window rows, batch 16,
 * 32 KV heads, 32,768 cached tokens) are far inside all of them.
 */
#ifndef D2F_H
#define D2F_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum d2f_status {
  D2F_OK = 0,
  D2F_ERR_INVALID_ARG = 1, /* bad sizes, null required pointer, bad metadata */
  D2F_ERR_UNSUPPORTED = 2, /* valid request this build does not implement      */
  D2F_ERR_CUDA = 3,        /* a CUDA runtime / launch error                      */
  D2F_ERR_BAD_INDEX = 4,   /* device: page id / row index out of range          */
  D2F_ERR_TIMEOUT = 5,     /* device: a bounded wait gave up                     */
  D2F_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required         */
  D2F_ERR_NO_PAGE = 7      /* device: a finished block got no page (free list    */
                           /* empty or its page-table row full); it stays put    */
} d2f_status;

typedef enum d2f_dtype { D2F_BF16 = 0, D2F_F32 = 1 } d2f_dtype;

/* Block phases ([P2] §쉽게 이해하기). */
enum { D2F_PHASE_CONSERVATIVE = 0, D2F_PHASE_AGGRESSIVE = 1 };
/* Keys attended by d2f_block_attn_part (d2f_block_attn attends to all). */
enum { D2F_ATTN_ALL = 0, D2F_ATTN_CACHED = 1, D2F_ATTN_WINDOW = 2 };
/* Confidence metrics of d2f_commit_metric (d2f_commit uses D2F_CONF_PMAX). */
enum {
  D2F_CONF_PMAX = 0,         /* largest softmax probability */
  D2F_CONF_NEG_ENTROPY = 1,  /* sum_v p_v ln p_v */
  D2F_CONF_MARGIN = 2,       /* largest minus second largest probability */
  D2F_CONF_LOGIT_GAP = 3     /* largest minus second largest logit */
};

/* Library version, e.g. 100 for 0.1.0. */
int d2f_version(void);

/* Static description of a status code. */
const char *d2f_status_string(int status);

/* One-line reason for the last non-OK status returned in this thread
 * (empty string if none). The pointer stays valid until the next call. */
const char *d2f_last_error_string(void);

/* ------------------------------------------------------------------------- */
/* Block-causal attention over [paged cache ; window]                        */
/* ------------------------------------------------------------------------- */

/*
 * Workspace bytes for d2f_block_attn with the same size arguments. num_splits
 * = 0 selects the automatic split count for the current CUDA device (the same
 * one d2f_block_attn picks for num_splits = 0 on that device).
 */
int d2f_block_attn_workspace_size(int batch, int total_q, int max_q_per_seq, int max_ctx,
                                  int num_heads_q, int num_heads_kv, int head_dim,
                                  int block_size, int dtype, int num_splits, size_t *bytes);

/*
 * d2f_block_attn -- one layer's attention for the active window.
 *
 * [P1] §블록 단위 인과 어텐션, [P2] §쉽게 이해하기: query head h of window row i
 * of sequence b attends to
 *   (a) every cached token t < ctx_len[b] (prompt and committed blocks, read
 *       through the page table), and
 *   (b) every window row i2 of the same sequence with i2/B <= i/B (its own
 *       block in both directions, earlier window blocks, no later ones);
 * scores = softmax_scale * <q, k>, out = softmax(scores) . v. The cached part
 * is split over several CTAs whose partial (O, max, sum) are composed in log
 * space ([P3] §FlashBlock: log-space composition of attention parts).
 *
 *   q           device [total_q][num_heads_q][head_dim], dtype
 *   k_win,v_win device [total_q][num_heads_kv][head_dim], dtype (this step's
 *               window K/V)
 *   k_pool,
 *   v_pool      device [num_pages][num_heads_kv][block_size][head_dim], dtype
 *   page_table  device int32 [batch][max_pages_per_seq]; entries at or past
 *               ceil(ctx_len[b]/B) are not read
 *   ctx_len     device int32 [batch], 0 <= ctx_len[b] <= max_pages_per_seq*B;
 *               need not be a multiple of B (slots past it are masked)
 *   q_start     device int32 [batch+1]
 *   out         device [total_q][num_heads_q][head_dim], dtype
 *   lse_out     device float [total_q][num_heads_q] natural-log normaliser, or NULL
 *   max_q_per_seq  host upper bound on n_b (rows past it are reported through
 *               err_word as D2F_ERR_INVALID_ARG and left unwritten)
 *   max_ctx     host hint used only to pick the split count
 *   dtype       D2F_BF16 with head_dim 64 or 128 and block_size 8, 16 or 32 takes
 *               the tensor-core path; everything else (D2F_F32, other bf16 shapes)
 *               takes the CUDA-core path, head_dim 32, 64 or 128, block_size 1..256
 *   softmax_scale  > 0, typically 1/sqrt(head_dim)
 *   num_splits  0 = automatic, else the number of CTAs sharing one row tile's keys.
 *               Tensor-core path: 1..8, the CTAs of one thread-block cluster, whose
 *               partials are composed in distributed shared memory (larger requests
 *               are clamped to 8). CUDA-core path: any count; partials go through
 *               the workspace.
 *   workspace   device, >= d2f_block_attn_workspace_size(...) bytes, zeroed once
 *               (and again after a device error). The tensor-core path needs none
 *               (NULL is accepted), except its stream-K form: the one-CTA-per-SM
 *               variant with fewer (sequence, KV head) pairs than SMs takes a
 *               counter per pair and two 33 KB partial slots per CTA (~10 MB on
 *               GB300).
 *
 * Alignment: every device buffer 16-byte aligned.
 */
int d2f_block_attn(const void *q, const void *k_win, const void *v_win, const void *k_pool,
                   const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
                   const int32_t *ctx_len, const int32_t *q_start, void *out, float *lse_out,
                   int batch, int total_q, int max_q_per_seq, int max_ctx, int num_heads_q,
                   int num_heads_kv, int head_dim, int block_size, int num_pages, int dtype,
                   float softmax_scale, int num_splits, void *workspace, size_t workspace_bytes,
                   int32_t *err_word, void *stream);

/*
 * d2f_block_attn_flags -- d2f_block_attn with launch flags.
 *
 *   flags  0 or D2F_ATTN_CACHE_READY. D2F_ATTN_CACHE_READY is the caller's promise
 *          that page_table, ctx_len, q_start and the cached K/V pages those name
 *          are final before the kernel that precedes this call in `stream`
 *          starts: that kernel writes none of them. Q, the window K/V and the
 *          outputs carry no such promise. The attention may then load its first
 *          cached tiles before it waits for the preceding kernel. Under
 *          programmatic dependent launch, its CTAs start while that kernel
 *          finishes, so the first tiles land sooner. Results are those of
 *          d2f_block_attn. Do not pass it when the preceding kernel writes the
 *          cache or the window layout: a d2f_kv_append, or d2f_window_step, as in
 *          a device-driven decode. Unknown bits give D2F_ERR_INVALID_ARG.
 */
#define D2F_ATTN_CACHE_READY 1u
int d2f_block_attn_flags(const void *q, const void *k_win, const void *v_win, const void *k_pool,
                         const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
                         const int32_t *ctx_len, const int32_t *q_start, void *out,
                         float *lse_out, int batch, int total_q, int max_q_per_seq, int max_ctx,
                         int num_heads_q, int num_heads_kv, int head_dim, int block_size,
                         int num_pages, int dtype, float softmax_scale, int num_splits,
                         void *workspace, size_t workspace_bytes, unsigned flags,
                         int32_t *err_word, void *stream);

/*
 * d2f_block_attn_append -- d2f_block_attn, then d2f_kv_append of finished
 * window blocks, in one launch where the attention runs on tensor cores.
 *
 * [P1] §블록 단위 인과 어텐션 and §운영 관점: a completed block's K/V are final
 * and persisted into the paged cache. The attention already streams every
 * window block's K/V into shared memory; there the CTA that holds a block
 * listed in src_row stores it to its page (one tensor copy per page and
 * tensor) instead of a separate kernel reading the window again. The result is
 * that of d2f_block_attn followed by d2f_kv_append with the same arguments.
 *
 * Arguments as d2f_block_attn, plus src_row / dst_page / n_append as for
 * d2f_kv_append (src_row[a] a window row starting a block: a multiple of
 * block_size below total_q). Additional requirement: no dst_page is a page the
 * attention reads in this call (a cached page of any sequence); the append
 * writes while the attention reads. Out-of-range pages set err_word =
 * D2F_ERR_BAD_INDEX and are skipped. On the CUDA-core path (float32, or shapes
 * outside the tensor-core variants) the append runs as its own kernel after the
 * attention.
 */
int d2f_block_attn_append(const void *q, const void *k_win, const void *v_win, const void *k_pool,
                          const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
                          const int32_t *ctx_len, const int32_t *q_start, void *out,
                          float *lse_out, int batch, int total_q, int max_q_per_seq, int max_ctx,
                          int num_heads_q, int num_heads_kv, int head_dim, int block_size,
                          int num_pages, int dtype, float softmax_scale, int num_splits,
                          void *workspace, size_t workspace_bytes, const int32_t *src_row,
                          const int32_t *dst_page, int n_append, int32_t *err_word,
                          void *stream);

/*
 * d2f_block_attn_part -- the attention over one part of the keys, and the reuse
 * of a kept cached part.
 *
 * "확산 언어 모델(Diffusion LLM)이란 무엇인가", §FlashBlock: 블록 외부 어텐션 캐싱:
 * the attention output and normaliser over the tokens outside the blocks being
 * decoded are kept from one step; at the next step only the attention inside
 * is recomputed and the two are recombined in log space; when more tokens than
 * a threshold have changed, the kept part is recomputed instead (the caller's
 * choice: it calls D2F_ATTN_CACHED again).
 *
 *   part D2F_ATTN_ALL     d2f_block_attn.
 *   part D2F_ATTN_CACHED  only the cached tokens (lse_out required); a row of a
 *                         sequence without cached tokens gets out 0, lse -inf.
 *                         out / lse_out are the part to keep.
 *   part D2F_ATTN_WINDOW  only the window keys (no cached page is read:
 *                         k_pool / v_pool / page_table may be NULL, max_ctx is
 *                         ignored); with prev_out / prev_lse (a kept
 *                         D2F_ATTN_CACHED result, of this step or an earlier
 *                         one) the output is the composition
 *                           out = (e^{lse_p} prev + e^{lse_w} out_w) / (e^{lse_p} + e^{lse_w}),
 *                           lse = ln(e^{lse_p} + e^{lse_w}).
 *                         With the same queries this is the full attention (up
 *                         to the kept part's bf16 rounding); with the kept part of
 *                         earlier queries it is the softmax whose cached scores use
 *                         those.
 * Other arguments as d2f_block_attn; prev_out is laid out as out, prev_lse as
 * lse_out. Tensor-core path only (bf16, head_dim 64/128, block_size 8/16/32):
 * D2F_ERR_UNSUPPORTED otherwise.
 */
int d2f_block_attn_part(const void *q, const void *k_win, const void *v_win, const void *k_pool,
                        const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
                        const int32_t *ctx_len, const int32_t *q_start, void *out, float *lse_out,
                        int batch, int total_q, int max_q_per_seq, int max_ctx, int num_heads_q,
                        int num_heads_kv, int head_dim, int block_size, int num_pages, int dtype,
                        float softmax_scale, int num_splits, void *workspace,
                        size_t workspace_bytes, int part, const void *prev_out,
                        const float *prev_lse, int32_t *err_word, void *stream);

/* ------------------------------------------------------------------------- */
/* Confidence commit over the vocabulary                                    */
/* ------------------------------------------------------------------------- */

/* Workspace bytes for d2f_commit (num_splits 0 = automatic for the current device). */
int d2f_commit_workspace_size(int total_q, int vocab, int dtype, int block_size, int num_splits,
                              size_t *bytes);

/*
 * d2f_commit -- confidence, greedy token, commit and remask for every
 * still-masked window position.
 *
 * [P3] §양방향 어텐션과 사라진 KV 캐시, §토큰 순서의 이론: confidence is the largest
 * softmax probability of the position's prediction (LLaDA low-confidence
 * remasking). [P2] §쉽게 이해하기: a conservative block commits the positions
 * whose confidence is above the threshold; an aggressive block also commits its
 * relatively most confident position; every position not committed is masked
 * again for the next step.
 *
 * For each row r with masked[r] != 0, with l = the logit row logit_row[r]
 * (or r when logit_row is NULL):
 *   m = max_v l_v, a = lowest v with l_v = m (bf16 widened exactly to float),
 *   p = 1 / sum_v exp(l_v - m) (float accumulation).
 * For each window block jb of sequence b (tau[b], block_phase[jb]):
 *   commit {r masked : p_r > tau[b]} (strict, in float); if aggressive and the
 *   block has a masked row, also the masked row with the largest p (lowest row
 *   on ties). Committed rows: tokens[r] = a, masked[r] = 0. Other masked rows:
 *   tokens[r] = mask_id. Rows not masked on entry are left unchanged.
 *
 *   logits          device [num_logit_rows][row_stride] dtype; columns >= vocab are not read
 *   row_stride      elements between logit rows (>= vocab)
 *   logit_row       device int32 [total_q] or NULL (e.g. Dream's one-position shift)
 *   tokens, masked  device int32 / uint8 [total_q], in/out
 *   q_start         device int32 [batch+1]
 *   block_phase     device uint8 [total_q / block_size] (D2F_PHASE_*)
 *   tau             device float [batch]
 *   conf_out        device float [total_q] or NULL: p for rows masked on entry, -1 otherwise
 *   argmax_out      device int32 [total_q] or NULL: a for rows masked on entry, -1 otherwise
 *   block_remaining device int32 [total_q / block_size] or NULL: masked rows left per block
 *   block_size      1..32
 */
int d2f_commit(const void *logits, int64_t row_stride, int dtype, int vocab, int num_logit_rows,
               const int32_t *logit_row, int32_t *tokens, uint8_t *masked,
               const int32_t *q_start, const uint8_t *block_phase, const float *tau, int batch,
               int total_q, int block_size, int32_t mask_id, float *conf_out,
               int32_t *argmax_out, int32_t *block_remaining, int num_splits, void *workspace,
               size_t workspace_bytes, int32_t *err_word, void *stream);

/*
 * d2f_commit_metric -- d2f_commit with another confidence, in the same single
 * pass over each masked position's logits.
 *
 * "확산 언어 모델(Diffusion LLM)이란 무엇인가", §토큰 순서의 이론: Dream ranks
 * positions by negative entropy rather than the largest probability, and the
 * top-probability-margin ordering ranks them by the difference between the
 * largest and the second largest probability; §답을 미리 안다: 조기 확정
 * 디코딩(Prophet): the confidence gap is the largest logit minus the second
 * largest. With m, a and S = sum_v exp(l_v - m) as for d2f_commit,
 * E = sum_v exp(l_v - m) (l_v - m) and l2 the second largest logit counted with
 * multiplicity (l2 = m when the maximum occurs twice):
 *   D2F_CONF_PMAX         c = 1 / S                   (d2f_commit)
 *   D2F_CONF_NEG_ENTROPY  c = E / S - ln S  (= sum_v p_v ln p_v, <= 0)
 *   D2F_CONF_MARGIN       c = (1 - exp(l2 - m)) / S  (= p_1 - p_2)
 *   D2F_CONF_LOGIT_GAP    c = m - l2
 * in float arithmetic (the gap is exact for bf16 logits). The commit rule is
 * d2f_commit's with c in place of p: conservative blocks commit c > tau[b]
 * (tau in the metric's units), aggressive blocks also their largest c;
 * conf_out receives c. A logit of -inf adds nothing to S or E.
 *
 * Early commit (same passage on Prophet: once the gap between the largest and
 * the second largest logit over the answer region exceeds a threshold, every
 * remaining mask is filled with its argmax; the threshold is lowered in stages,
 * 7.5 / 5.0 / 2.5, as decoding progresses): with early_gap non-NULL (device
 * float [batch], the caller's current thresholds), sequence b -- reading taken:
 * its window is the region, its gap the smallest m - l2 over the rows masked on
 * entry -- stops when that gap exceeds early_gap[b] (strict): after the block
 * rules every row of b still masked is committed with its greedy token, its
 * blocks' block_remaining become 0 and stopped[b] = 1 (device uint8 [batch], or
 * NULL); otherwise stopped[b] = 0, also for a sequence with nothing masked.
 * It combines with D2F_CONF_PMAX, _MARGIN and _LOGIT_GAP (D2F_ERR_UNSUPPORTED
 * with _NEG_ENTROPY).
 *
 * Arguments as d2f_commit, plus metric (D2F_CONF_*; other values return
 * D2F_ERR_INVALID_ARG), early_gap and stopped. The workspace is
 * d2f_commit_workspace_size's for the same sizes.
 */
int d2f_commit_metric(const void *logits, int64_t row_stride, int dtype, int vocab,
                      int num_logit_rows, const int32_t *logit_row, int32_t *tokens,
                      uint8_t *masked, const int32_t *q_start, const uint8_t *block_phase,
                      const float *tau, int batch, int total_q, int block_size, int32_t mask_id,
                      int metric, const float *early_gap, uint8_t *stopped, float *conf_out,
                      int32_t *argmax_out, int32_t *block_remaining, int num_splits,
                      void *workspace, size_t workspace_bytes, int32_t *err_word, void *stream);

/*
 * d2f_commit_noalloc -- d2f_commit without a caller workspace, for callers that
 * cannot allocate device memory (a plugin or callback that may only use the
 * buffers its host framework passes in, a runtime that must not allocate once it
 * serves, a caller with no allocator at hand). The pages describe no such entry
 * point; it exists only for those callers.
 *
 * Same arguments and result as d2f_commit, minus workspace / workspace_bytes.
 * Its scratch is a fixed 2 MiB array in the library's device image, held by
 * every GPU that loads the library until the process exits. Requests whose
 * d2f_commit_workspace_size exceeds 2 MiB return D2F_ERR_WORKSPACE (use
 * d2f_commit instead): at block size 16 that is more than 2,032 window rows at
 * 64 vocabulary slices per row, 15,792 at 8, 57,056 at 2. The array's device
 * address is looked up (cudaGetSymbolAddress) by the first call in each CUDA
 * context and cached under the context's unique id, so calls from another
 * context, or from a context re-created after a reset, get their own; make the
 * first call in a context before any stream capture. Each call clears the
 * scratch's arrival counters with cudaMemsetAsync on `stream` (the rest is
 * written before it is read); nothing is allocated or freed. All calls share
 * the one array: calls that may overlap on the GPU race and must be serialised.
 */
int d2f_commit_noalloc(const void *logits, int64_t row_stride, int dtype, int vocab,
                       int num_logit_rows, const int32_t *logit_row, int32_t *tokens,
                       uint8_t *masked, const int32_t *q_start, const uint8_t *block_phase,
                       const float *tau, int batch, int total_q, int block_size, int32_t mask_id,
                       float *conf_out, int32_t *argmax_out, int32_t *block_remaining,
                       int num_splits, int32_t *err_word, void *stream);

/* ------------------------------------------------------------------------- */
/* KV append of finished blocks                                             */
/* ------------------------------------------------------------------------- */

/*
 * d2f_kv_append -- copy finished blocks from the window K/V into their pages.
 *
 * [P1] §블록 단위 인과 어텐션 and §운영 관점: a completed block's K/V never change
 * and are stored permanently; with pages of one block, completion is the signal
 * to persist. For append a: k_pool[dst_page[a]][g][s][:] = k_win[src_row[a]+s][g][:]
 * for every KV head g and slot s < block_size (same for V); a bitwise copy.
 * The caller then extends page_table / ctx_len.
 *
 *   src_row, dst_page  device int32 [n_append]; src_row[a] + block_size <= total_q,
 *                      0 <= dst_page[a] < num_pages (else err_word = D2F_ERR_BAD_INDEX
 *                      and that append is skipped). Destination pages must be distinct.
 */
int d2f_kv_append(const void *k_win, const void *v_win, const int32_t *src_row,
                  const int32_t *dst_page, int n_append, int total_q, void *k_pool,
                  void *v_pool, int num_heads_kv, int head_dim, int block_size, int num_pages,
                  int dtype, int32_t *err_word, void *stream);

/*
 * d2f_kv_append_dev -- d2f_kv_append whose list length lives in device memory
 * (written by d2f_window_step), so that no host readback sits between steps.
 *
 *   n_append_dev  device int32 [1]: entries of src_row / dst_page to apply, read
 *                 on the device; values above max_append are taken as max_append,
 *                 negative ones as 0. max_append >= 0 sizes the launch.
 * Everything else as d2f_kv_append.
 */
int d2f_kv_append_dev(const void *k_win, const void *v_win, const int32_t *src_row,
                      const int32_t *dst_page, const int32_t *n_append_dev, int max_append,
                      int total_q, void *k_pool, void *v_pool, int num_heads_kv, int head_dim,
                      int block_size, int num_pages, int dtype, int32_t *err_word, void *stream);

/*
 * d2f_block_attn_append_dev -- d2f_block_attn_append whose list length lives in
 * device memory (n_append_dev, at most max_append entries, as d2f_kv_append_dev).
 */
int d2f_block_attn_append_dev(const void *q, const void *k_win, const void *v_win,
                              const void *k_pool, const void *v_pool, const int32_t *page_table,
                              int max_pages_per_seq, const int32_t *ctx_len,
                              const int32_t *q_start, void *out, float *lse_out, int batch,
                              int total_q, int max_q_per_seq, int max_ctx, int num_heads_q,
                              int num_heads_kv, int head_dim, int block_size, int num_pages,
                              int dtype, float softmax_scale, int num_splits, void *workspace,
                              size_t workspace_bytes, const int32_t *src_row,
                              const int32_t *dst_page, const int32_t *n_append_dev,
                              int max_append, int32_t *err_word, void *stream);

/* ------------------------------------------------------------------------- */
/* Pipelined window scheduler                                               */
/* ------------------------------------------------------------------------- */

/*
 * d2f_window_step -- between two decode steps, on the device: turn the state the
 * commit left into the window, phases, append list and cache bookkeeping of the
 * next step, so a whole step (attention with its appends, commit, scheduler)
 * replays from one CUDA graph with no host readback.
 *
 * [P2] §쉽게 이해하기 (pipelined parallel decoding): an active window of blocks;
 * once the last block's progress passes a threshold a new block enters behind
 * it; a new block is conservative and turns aggressive once the block before it
 * has progressed enough; uncommitted positions stay masked. [P1] §운영 관점: a
 * completed block is persisted to the paged cache (completion is the signal).
 *
 * Rule (readings of the pages, which give no values and no order):
 *  - progress of a block = its committed positions c out of B. A new block
 *    enters a sequence's window when c(last block) > tau_add * B, or the window is
 *    empty, and next_block < gen_blocks, the window holds fewer than max_blocks
 *    blocks and the sequence is not stopped; at most one per step.
 *  - block k of the new window is aggressive (phase 1) when the block before it
 *    has c >= tau_act * B; the block before the oldest is the cache (c = B).
 *  - complete blocks forming the oldest prefix of the window are listed for the
 *    next step's append (its forward pass computes their K/V from final tokens);
 *    they stay in the window for that step and leave at the next call (their
 *    count is n_leaving), when ctx_len grows by B each.
 *  - pages come from the top of the free list, free_pages[*free_count - 1] first,
 *    in (sequence, block) order; the page of the i-th listed block of sequence b
 *    is written to page_table[b][ctx_len[b] / B + i] at once. A block that gets no
 *    page (list empty or page-table row full) stays in the window, listed again
 *    later, and err_word takes D2F_ERR_NO_PAGE.
 *  - the products tau * B and the comparisons are float.
 *
 * Layout: the window rows of sequence b are q_start[b] .. q_start[b+1]-1, block by
 * block, oldest first, as every other entry point takes them. capacity rows are
 * allocated; capacity % block_size == 0 and capacity >= batch * max_blocks *
 * block_size, so the window always fits. All pointers are device memory owned by
 * the caller; in/out unless said:
 *   q_start      int32 [batch+1]
 *   tokens       int32 [capacity];  masked uint8 [capacity]
 *   block_phase  uint8 [capacity / block_size] (out)
 *   row_pos      int32 [capacity] (out): position of the row's token in its
 *                sequence (ctx_len + offset in the window), -1 past the window
 *   ctx_len      int32 [batch]; page_table int32 [batch][max_pages_per_seq]
 *   next_block   int32 [batch]: generation blocks that have entered so far
 *   gen_blocks   int32 [batch] (in): generation blocks of each sequence
 *   n_leaving    int32 [batch]: blocks listed for append by the previous call
 *   stopped      uint8 [batch] (in, may be NULL): the early commit's flags
 *   free_pages   int32 [>= *free_count] (in); free_count int32 [1]
 *   app_src, app_dst  int32 [capacity / block_size] (out); n_append int32 [1] (out):
 *                the next step's append list (first window row of the block in the
 *                new layout, its page), for d2f_block_attn_append_dev or
 *                d2f_kv_append_dev
 * Rows past the new window read tokens = mask_id, masked = 0, row_pos = -1 and
 * their blocks phase 0, so the commit skips them. A sequence is finished when its
 * window is empty after a call. ctx_len must be a multiple of block_size (pad the
 * prompt).
 *
 * Errors: D2F_ERR_INVALID_ARG for bad sizes (host), or, in err_word, for a state
 * that is not consistent (a window not made of whole blocks, beyond capacity or
 * longer than max_blocks, n_leaving larger than the window, ctx_len negative or
 * not a multiple of block_size, q_start[0] != 0, *free_count < 0): then nothing is
 * written. D2F_ERR_UNSUPPORTED when the state does not fit one CTA's shared
 * memory (about 5 bytes per capacity row + 36 per sequence, 227 KB in all) or
 * block_size > 128.
 */
int d2f_window_step(int batch, int block_size, int max_blocks, int capacity,
                    int max_pages_per_seq, int32_t mask_id, float tau_add, float tau_act,
                    int32_t *q_start, int32_t *tokens, uint8_t *masked, uint8_t *block_phase,
                    int32_t *row_pos, int32_t *ctx_len, int32_t *page_table, int32_t *next_block,
                    const int32_t *gen_blocks, int32_t *n_leaving, const uint8_t *stopped,
                    const int32_t *free_pages, int32_t *free_count, int32_t *app_src,
                    int32_t *app_dst, int32_t *n_append, int32_t *err_word, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* D2F_H */
