/*
 * dspark.h -- C ABI of libdspark.so: DSpark's confidence-scheduled ragged
 * verification step on one GB300 (sm_103a).
 *
 * The step, in the order a caller runs it on one CUDA stream:
 *
 *   dspark_schedule     calibrated prefix survival -> per-request verify windows
 *   dspark_pack         head-to-tail packing, cu_seqlens, captured tier, row indices
 *   dspark_verify_attn  varlen verify attention of the packed rows over paged KV
 *   dspark_accept       prefix speculative-sampling acceptance, bonus/correction, c*
 *   dspark_compact      scatter of accepted KV rows + page-table append
 *
 * Sources, cited by short name:
 *   [lesson] "DFlash 到 DSpark in SGLang：解码提速 4.3×，以及 DeepSeek-V4 支持"
 *            (AI Infra Visualized lesson on DSpark)
 *   [csdn]   DevPress/CSDN article on DSpark in SGLang (sections 2-5)
 *   [notes]  "DSpark：投机解码与生产级 Serving 学习笔记" (sections 02, 05, 07, 08, 09)
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless the
 *     argument's comment says "host".  Tensors are dense row-major, no strides.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is enqueued
 *     on it; no call synchronises, allocates or frees memory.  Each of the five
 *     step calls launches a fixed sequence of kernels whose grid does not depend
 *     on device data, so the step can be captured in a CUDA graph.
 *   - Return value: a dspark_status.  Arguments are checked on the host before
 *     anything is launched; a non-OK return means nothing was enqueued (except
 *     DSPARK_ECUDA, which reports a failed launch).  Nothing throws or aborts.
 *   - Conditions only the device can see (a packed batch larger than the row
 *     capacity, an exhausted free-page stack, a wait that ran out) set bits of a
 *     per-device error word (DSPARK_DEVERR_*); the kernel that sees them skips
 *     the offending writes.  dspark_read_device_error() returns and clears it.
 *   - The library must have been built for sm_103a; on any other device the
 *     first call returns DSPARK_EUNSUPPORTED.
 *   - Per-device set-up (kernel attributes, the address of the error word and of
 *     fixed scratch) is done once per device on the first call made with that
 *     device current, and is safe when several host threads make that first call
 *     at once.  It is kept for the life of the process: the library is not usable
 *     after a cudaDeviceReset in the same process.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSPARK_OK = 0,
  DSPARK_EINVAL = -1,        /* bad argument: NULL pointer, size, alignment      */
  DSPARK_EUNSUPPORTED = -2,  /* shape or device outside what the kernels handle  */
  DSPARK_ECUDA = -3,         /* a CUDA runtime call or launch failed             */
  DSPARK_ENOSPACE = -4,      /* workspace smaller than *_workspace_size()        */
  DSPARK_EDEVICE = -5        /* device error word non-zero (read_device_error)   */
} dspark_status;

/* Verify modes ([lesson] "Confidence scheduler 与 verify 模式"; [csdn] 2.):
 * COMPACT verifies only each request's window (the production path); STATIC
 * verifies the whole block; CAP_ACCEPT verifies the whole block but commits
 * only up to the window (identical commits to COMPACT) and records the cap. */
typedef enum { DSPARK_COMPACT = 0, DSPARK_STATIC = 1, DSPARK_CAP_ACCEPT = 2 } dspark_mode;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

/* Bits of the device error word. */
#define DSPARK_DEVERR_ROWS_OVERFLOW 0x1u   /* packed tier > max_rows               */
#define DSPARK_DEVERR_NO_FREE_PAGE  0x2u   /* free-page stack exhausted (compact)  */
#define DSPARK_DEVERR_PAGE_ROW_FULL 0x4u   /* page-table row too short (compact)   */
#define DSPARK_DEVERR_WAIT_TIMEOUT  0x8u   /* a bounded in-kernel wait ran out     */
#define DSPARK_DEVERR_BAD_INPUT     0x10u  /* index input out of range (token, page) */
#define DSPARK_DEVERR_WORK_OVERFLOW 0x20u  /* attention work list larger than ws   */

/* Limits checked on the host. */
#define DSPARK_MAX_B        1024   /* requests per step                          */
#define DSPARK_MAX_GAMMA    32     /* draft block length                         */
#define DSPARK_MAX_CANDS    4096   /* B * gamma for the scheduler's sort          */
#define DSPARK_MAX_TIERS    64
#define DSPARK_MAX_ECE_BINS 256

const char* dspark_status_string(int status);

/* Reads and clears the device error word of the current device.  Synchronises
 * `stream`.  Returns the word (>= 0) or DSPARK_ECUDA. */
int dspark_read_device_error(void* stream);

/* Number of SMs the persistent kernels size their grids by (current device). */
int dspark_num_sms(void);

/* Time limit of each bounded in-kernel wait of the acceptance pass on the current
 * device, for calls enqueued after this one (ns; 0 restores the default, 2 s).  A
 * wait that runs past it sets DSPARK_DEVERR_WAIT_TIMEOUT and makes its kernel stop:
 * every role leaves its loop, the copies already issued are waited for (always on
 * the 2 s limit), and the kernel returns; the outputs of that call are undefined
 * and the next call is unaffected.  (The attention kernels keep their fixed 2 s
 * limit.)  A calibration of failure handling, not a tuning knob. */
int dspark_set_wait_limit_ns(unsigned long long ns);
/* Failure-detection test hook: while on (for calls enqueued after it, on the
 * current device), the acceptance pass first waits on a barrier nothing arrives at,
 * so that its bounded wait must run out (after the limit above) and the timeout
 * path runs: DSPARK_DEVERR_WAIT_TIMEOUT, every role stops, nothing is left in
 * flight.  Off by default; it never faults or hangs the device. */
int dspark_set_wait_probe(int on);

/* ---------------------------------------------------------------------------
 * dspark_schedule -- per-request verify windows.
 * [notes] 07 (c_k, a_j = prod_{i<=j} c_i, STS), [notes] 08.3 (global greedy:
 * sort candidates by survival, add while expected throughput rises, stop at the
 * first drop), [csdn] 4. (T(bs,K) = bias + alpha(bs) + theta(M), M = bs + K).
 *
 *   conf        fp32 [B, gamma]  confidence logits (conf_is_logit = 1) or c
 *   sts_temp    fp32 [gamma]     per-position STS temperature T_j > 0
 *   cost_table  fp32 [cost_len]  step cost T[M] (any unit, > 0) for M = 0..cost_len-1;
 *                                cost_len >= min(max_tokens, B*(gamma+1)) + 1
 *   max_tokens  largest verify row count the step may use (largest captured tier)
 *   mode        dspark_mode; STATIC sets every window to gamma
 *   windows     int32 [B]  out: verified drafts w_r in [0, gamma]
 *   a_hat       fp32 [B, gamma]  out: calibrated survival (non-increasing in j)
 *   survival    fp32 [B, gamma]  out, nullable: the uncalibrated prefix survival
 *               a_j (what dspark_calib_collect records for a temperature refit)
 *   M_out       int32 [1]  out: B + sum w_r
 *   E_out       fp64 [1]   out: expected committed tokens B + sum of chosen a_hat
 *
 * Arithmetic: c = fp32(1/(1+exp(-z))) in fp64; a_j = fp32 running product;
 * a_hat_j = fp32(1/(1+exp(-(log a - log1p(-a))/T_j))) in fp64, then the running
 * minimum over j.  Candidates sort by a_hat descending, ties by request then
 * position ascending.  E starts at B and M at B; candidate k is accepted iff
 * B + k + 1 <= max_tokens and (E_k + a_k)/T[M_k+1] > E_k/T[M_k], evaluated in
 * fp64 cross-multiplied: (E_k + a_k) * T[M_k] > E_k * T[M_k+1] (T > 0).
 * Limits: 1 <= B <= 1024, 1 <= gamma <= 32, B*gamma <= 4096.
 * ------------------------------------------------------------------------- */
int dspark_schedule(const float* conf, int conf_is_logit, const float* sts_temp,
                    const float* cost_table, int cost_len, int B, int gamma, int max_tokens,
                    int mode, int32_t* windows, float* a_hat, float* survival, int32_t* M_out,
                    double* E_out, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_pack -- head-to-tail ragged packing ([lesson] "Ragged verify under full
 * CUDA graphs"; [csdn] 3.).
 *
 * Request r occupies n_r = 1 + v_r consecutive rows, v_r = windows[r] (COMPACT,
 * STATIC) or gamma (CAP_ACCEPT): the anchor token then drafts d_1..d_{v_r}.
 *   cu_seqlens  int32 [B+1] out: exclusive prefix sum of n_r
 *   M_out       int32 [1]   out: cu_seqlens[B]
 *   tier_out    int32 [1]   out: smallest entry of `tiers` >= M, or M if none is
 *   tier_host   int32 [1]   out, nullable, HOST: pinned memory mapped into the
 *               device (cudaHostAlloc with cudaHostAllocMapped, or registered
 *               with cudaHostRegisterMapped); the kernel also stores the tier
 *               there, so a host-side engine can read it once the pack kernel
 *               has finished (an event after this call) without synchronising
 *               the stream, and pick the target forward captured for that tier
 *               ([lesson] "Ragged verify under full CUDA graphs").
 *   row_req     int32 [max_rows] out: request of each packed row, -1 on padding
 *   row_pos     int32 [max_rows] out: absolute position ctx_len[r] + i, -1 on padding
 *                                     (its page is page_table[r][pos / page_size])
 *   row_tok     int32 [max_rows] out: token of the row (anchor or d_i), -1 on padding
 *   tiers       int32 [n_tiers] ascending captured tier sizes (device)
 * Rows tier..max_rows-1 are left untouched.  If tier > max_rows the device sets
 * DSPARK_DEVERR_ROWS_OVERFLOW and writes only the first max_rows rows.
 * ------------------------------------------------------------------------- */
int dspark_pack(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out, int32_t* tier_out,
                int32_t* tier_host, int32_t* row_req, int32_t* row_pos, int32_t* row_tok,
                void* stream);

/* ---------------------------------------------------------------------------
 * dspark_verify_attn -- variable-length verify attention over the paged cache
 * ([lesson] "Ragged verify under full CUDA graphs": every packed token attends
 * only to its own request's KV; causal inside the block).
 *
 * Packed row cu_seqlens[r] + i (block index i) of request r, query head h, sees
 * the ctx_len[r] committed keys (through page_table) followed by block rows
 * 0..i of its own segment:  o = softmax(scale q.K^T) V,  lse = log sum exp.
 *
 * Two shapes:
 *   GQA  d_qk = d_v = 128, Hq % Hkv == 0, Hq/Hkv <= 128.
 *        q       bf16 [max_rows, Hq, 128]
 *        k_new   bf16 [max_rows, Hkv, 128],  v_new   the same
 *        k_cache bf16 [n_pages, page_size, Hkv, 128], v_cache the same
 *   MLA  d_qk = 576, d_v = 512, Hkv = 1, Hq = 128, v_new = v_cache = NULL.
 *        q       bf16 [max_rows, 128, 576]
 *        k_new   bf16 [max_rows, 576]   (latent of the block rows)
 *        k_cache bf16 [n_pages, page_size, 576]; values are the first 512 dims.
 *   page_table  int32 [B, max_pages]; entries past ceil(ctx/page_size) unused
 *   out         fp32 [max_rows, Hq, d_v]  out (rows >= M not written)
 *   lse         fp32 [max_rows, Hq]       out, natural log
 *   workspace   >= dspark_verify_attn_workspace_size(...) bytes, 256-B aligned
 * page_size must be a power of two >= 16.  All base pointers 16-byte aligned.
 * Work is divided stream-K style: the key tiles of all (request, row tile, KV
 * head) groups are cut into equal per-CTA ranges; a group cut by a range
 * boundary (into at most max_splits pieces, 2..32) is merged by a log-sum-exp
 * combine.  If cu_seqlens[B] > max_rows the device sets
 * DSPARK_DEVERR_ROWS_OVERFLOW and nothing is computed.  max_block_rows is a
 * hint: the rows of one request's segment the query tile of the GQA kernel is
 * sized for (32, 64 or 128 columns for max_block_rows x Hq/Hkv query rows; <= 0
 * counts as 1).  Any segment length is handled correctly
 * whatever its value: a longer segment runs as several row tiles, each over all
 * of its keys.  The whole block (gamma + 1) suits segments that are all long
 * (static and cap-accept verification); a compact step's short windows run
 * fastest on the smallest tile that holds a few rows (floor(32 / G) rows, the
 * 32-column tile, for G <= 8).  The workspace size
 * depends on it: a smaller hint needs more work items.
 * ------------------------------------------------------------------------- */
size_t dspark_verify_attn_workspace_size(int B, int max_rows, int Hq, int Hkv, int d_qk, int d_v,
                                         int max_splits, int max_block_rows);
int dspark_verify_attn(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                       const void* v_cache, int n_pages, const int32_t* page_table, int max_pages,
                       const int32_t* ctx_len, const int32_t* cu_seqlens, int B, int max_rows,
                       int Hq, int Hkv, int d_qk, int d_v, int page_size, float scale,
                       int max_splits, int max_block_rows, float* out, float* lse,
                       void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_pack_plan + dspark_verify_attn_planned -- the same two steps with the
 * attention's work list built inside the pack kernel (one kernel fewer between
 * the schedule and the attention of a step).
 *
 * dspark_pack_plan takes dspark_pack's arguments (same meaning, same outputs)
 * followed by the shape of the dspark_verify_attn_planned call that will use
 * the plan: Hq, Hkv, d_qk, d_v, its max_rows (attn_max_rows), max_splits and
 * max_block_rows, and that call's workspace (attn_workspace, at least
 * dspark_verify_attn_workspace_size(B, attn_max_rows, ...) bytes, 256-B
 * aligned).  It writes the work list for the cu_seqlens it computes and the
 * given ctx_len into attn_workspace.
 * dspark_verify_attn_planned has dspark_verify_attn's arguments and result, and
 * uses that work list: the caller passes the same workspace, shape, B, ctx_len
 * and cu_seqlens, on the same stream after the pack, with nothing writing the
 * workspace in between.  Errors: as dspark_pack and dspark_verify_attn; an
 * unsupported head shape gives DSPARK_EUNSUPPORTED from either call.
 * ------------------------------------------------------------------------- */
int dspark_pack_plan(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                     const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                     int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out,
                     int32_t* tier_out, int32_t* tier_host, int32_t* row_req, int32_t* row_pos,
                     int32_t* row_tok, int Hq, int Hkv, int d_qk, int d_v, int attn_max_rows,
                     int max_splits,
                     int max_block_rows, void* attn_workspace, size_t attn_ws_bytes,
                     void* stream);
int dspark_verify_attn_planned(const void* q, const void* k_new, const void* v_new,
                               const void* k_cache, const void* v_cache, int n_pages,
                               const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                               const int32_t* cu_seqlens, int B, int max_rows, int Hq, int Hkv,
                               int d_qk, int d_v, int page_size, float scale, int max_splits,
                               int max_block_rows, float* out, float* lse, void* workspace,
                               size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_accept -- prefix speculative sampling ([notes] 02; [lesson]
 * "Background" and "Confidence scheduler 与 verify 模式"; c* label [notes] 07).
 *
 *   p_target   [max_rows, V] packed target rows (fp32 or bf16 per pdt); row
 *              cu_seqlens[r] + i is the target distribution for position i + 1
 *   p_draft    [B, gamma, V] drafter distribution for positions 1..gamma
 *   draft_tok  int32 [B, gamma]
 *   uniforms   fp32 [B, gamma]  u in (0, 1) for the test at each position
 *   exp_noise  fp32 [B, V]      e ~ Exp(1) (Gumbel noise in exponential form,
 *                               G = -log e), used for the one sampled row
 *   windows    int32 [B]        the scheduler's windows (commit limit)
 *   accept_len int32 [B] out: committed drafts L_r
 *   cap_len    int32 [B] out: accepted prefix over the verified positions
 *   out_tok    int32 [B] out: correction (after a rejection) or bonus token
 *   cstar      fp32 [B, gamma] out: 1 - 0.5 ||p_d - p_t||_1 where a target row
 *              exists for the position, NaN elsewhere
 *   fallback   int32 [B] out (nullable): 1 if an all-zero residual forced the
 *              draw from p_target
 * If cu_seqlens[B] > max_rows the device sets DSPARK_DEVERR_ROWS_OVERFLOW and no
 * output is written.
 * Test: accept d_j iff fp32(u_j * p_d(d_j)) <= p_t(d_j).  Draws: argmax over v of
 * w_v / e_v in fp32 (w = max(0, p_t - p_d) after a rejection, p_t for the bonus),
 * lowest index on ties.
 * ------------------------------------------------------------------------- */
size_t dspark_accept_workspace_size(int B, int gamma, int max_rows, int V);
int dspark_accept(const void* p_target, const void* p_draft, int pdt, int V,
                  const int32_t* draft_tok, const float* uniforms, const float* exp_noise,
                  const int32_t* windows, const int32_t* cu_seqlens, int mode, int B, int gamma,
                  int max_rows, int32_t* accept_len, int32_t* cap_len, int32_t* out_tok,
                  float* cstar, int32_t* fallback, void* workspace, size_t ws_bytes,
                  void* stream);

/* ---------------------------------------------------------------------------
 * dspark_accept_noalloc -- dspark_accept without a caller-provided workspace.
 *
 * The paper has no counterpart: this is a library convenience.  It is meant for
 * callers that cannot hand over device memory of their own -- a plain C host that
 * links only this library and owns no CUDA allocator, or a serving engine whose
 * device memory pool is sized and frozen before serving starts, so that no
 * allocation may happen while it runs.  The call allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine); its scratch is one fixed array of
 * DSPARK_ACCEPT_NOALLOC_SCRATCH_BYTES compiled into the library, one per device.
 *
 * Arguments, outputs, error handling and results are those of dspark_accept.
 * Limit: the call returns DSPARK_ENOSPACE, launching nothing, when
 * dspark_accept_workspace_size(B, gamma, max_rows, V) exceeds the scratch size
 * (about max_rows * ceil(V / 8192) * 32 bytes; the 8 MiB hold max_rows = 8192,
 * i.e. B = 256 requests of 32 rows, at V = 151936).  No part of the scratch needs to start at zero: every entry read
 * is written earlier in the same call.
 * The first call on a device looks up the scratch address with that device
 * current (DSPARK_ECUDA if the lookup fails); make that first call before any
 * stream capture begins.  The address is kept for the life of the process: after
 * a cudaDeviceReset it would be stale, so this call (like the rest of the
 * library, whose per-device set-up is cached the same way) must not be used
 * after a device reset in the same process.  All calls on one device share the one array, so two
 * calls that may run at the same time (on different streams, or from host threads
 * without ordering between them) race on it and give undefined results: order
 * them on one stream.
 * ------------------------------------------------------------------------- */
#define DSPARK_ACCEPT_NOALLOC_SCRATCH_BYTES (8u << 20)
int dspark_accept_noalloc(const void* p_target, const void* p_draft, int pdt, int V,
                          const int32_t* draft_tok, const float* uniforms,
                          const float* exp_noise, const int32_t* windows,
                          const int32_t* cu_seqlens, int mode, int B, int gamma, int max_rows,
                          int32_t* accept_len, int32_t* cap_len, int32_t* out_tok, float* cstar,
                          int32_t* fallback, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_block_accept_estimate -- the uncut cap from inside a compact run
 * ([csdn] 5 "可观测性": compact verifies only the scheduler's window, so how many
 * drafts a full-block verification would have accepted is censored; the block-
 * accept estimator recovers an interval for it inside the compact run, without a
 * companion cap-accept run).  Run after dspark_accept on the same step's tensors.
 *
 * For request r (compact mode), window w, accepted length L = accept_len[r]:
 *   L < w          -> cap_lo = cap_hi = L   (a draft inside the window was rejected)
 *   L = w = gamma  -> cap_lo = cap_hi = gamma
 *   L = w < gamma  -> the step holds the target row of position w + 1 (the bonus
 *                     row, packed row cu_seqlens[r] + w) and the drafter's row of
 *                     that position, so the full-block test at w + 1 is made here
 *                     with the same operands: u_{w+1} p_d(d_{w+1}) <= p_t(d_{w+1})
 *                     (fp32) rejected -> cap_lo = cap_hi = w; accepted ->
 *                     cap_lo = w + 1, cap_hi = gamma.
 * Static and cap-accept modes verified the whole block: cap_lo = cap_hi = cap_len[r].
 * Arguments as dspark_accept's (p_target packed [max_rows, V], p_draft [B, gamma, V]
 * of type pdt; draft_tok, uniforms [B, gamma]; windows [B]; cu_seqlens [B+1]) plus
 * accept_len, cap_len [B] from dspark_accept; cap_lo, cap_hi int32 [B] out.  A bonus
 * row outside the request's segment or past max_rows, or a draft token outside
 * [0, V), sets DSPARK_DEVERR_BAD_INPUT and gives cap_lo = cap_hi = L.
 * ------------------------------------------------------------------------- */
int dspark_block_accept_estimate(const void* p_target, const void* p_draft, int pdt, int V,
                                 const int32_t* draft_tok, const float* uniforms,
                                 const int32_t* windows, const int32_t* cu_seqlens,
                                 const int32_t* accept_len, const int32_t* cap_len, int mode,
                                 int B, int gamma, int max_rows, int32_t* cap_lo, int32_t* cap_hi,
                                 void* stream);

/* ---------------------------------------------------------------------------
 * dspark_compact -- commit the step ([lesson] "Zero-overhead scheduling 与
 * kernel": compact scatter, device-resident page table).
 *
 * For each request in order: rows 0..L_r of its packed segment (anchor and
 * accepted drafts) are copied to cache positions ctx_r..ctx_r+L_r; pages are
 * popped from the top of free_pages (free_pages[*free_top-1] first, requests in
 * order) when a position opens a new page and appended to page_table[r];
 * ctx_len[r] += L_r + 1; anchor[r] = out_tok[r]; committed[r] = d_1..d_L, out_tok
 * (-1 beyond), n_committed[r] = L_r + 1.  Rejected rows are never written.
 *   row_bytes   bytes of one K row (GQA: Hkv*128*2, MLA: 576*2); V rows the same
 *   max_rows    rows of k_new/v_new
 *   k_new/v_new [max_rows, row] packed block rows; v_new/v_cache NULL for MLA
 *   k_cache/v_cache [n_pages, page_size, row]
 *   page_table  int32 [B, max_pages] in/out; ctx_len, anchor int32 [B] in/out
 *   free_pages  int32 [n_free]; free_top int32 [1] in/out
 *   committed   int32 [B, gamma+1] out; n_committed int32 [B] out
 * If the free stack or a page-table row is too short the device sets
 * DSPARK_DEVERR_NO_FREE_PAGE / _PAGE_ROW_FULL, if cu_seqlens[B] > max_rows it sets
 * DSPARK_DEVERR_ROWS_OVERFLOW, and if accept_len[r] is outside 0..gamma or keeps
 * more rows than request r's packed segment holds it sets DSPARK_DEVERR_BAD_INPUT;
 * in each of these cases it changes nothing.
 * ------------------------------------------------------------------------- */
size_t dspark_compact_workspace_size(int B);
int dspark_compact(const void* k_new, const void* v_new, int row_bytes, int max_rows,
                   const int32_t* cu_seqlens,
                   const int32_t* accept_len, const int32_t* out_tok, const int32_t* draft_tok,
                   int B, int gamma, int page_size, int max_pages, int n_pages,
                   int32_t* page_table, int32_t* ctx_len, int32_t* anchor,
                   const int32_t* free_pages, int32_t* free_top, void* k_cache, void* v_cache,
                   int32_t* committed, int32_t* n_committed, void* workspace, size_t ws_bytes,
                   void* stream);

/* ---------------------------------------------------------------------------
 * Calibration of the confidence head from the step's own accept outcomes
 * ([csdn] 5. "可观测性": per-request confidence and calibration metrics such as
 * ECE; [notes] 07: a_j predicts that prefix 1..j is accepted, and Sequential
 * Temperature Scaling a_hat_j = sigmoid(logit(a_j) / T_j) calibrates it).
 *
 * Sample store (device, caller-owned, per draft position j = 0..gamma-1, each
 * region `capacity` entries): s_a, s_ahat fp32 [gamma, capacity], s_y int8
 * [gamma, capacity], count int32 [gamma] (the caller zeroes count once).
 *
 * dspark_calib_collect appends one step's samples: every verified position j of
 * request r (j < windows[r], or j < gamma in CAP_ACCEPT mode; in request order)
 * adds (survival[r][j], a_hat[r][j], y = [j + 1 <= cap_len[r]]) at index count[j]
 * of position j's region (dropped once the region is full; count keeps counting).
 * survival/a_hat are dspark_schedule's outputs, cap_len dspark_accept's.  One CTA;
 * B <= 1024.  CAP_ACCEPT steps give unbiased samples (every position verified).
 *
 * dspark_calib_ece: expected calibration error of the stored a_hat against y over
 * all stored samples: equal-width bins b = min(floor(a_hat * n_bins), n_bins - 1),
 * bin_n int32 / bin_p fp64 (sum of a_hat) / bin_y fp64 (sum of y) [n_bins], and
 * ece fp64 [1] = (1/N) sum_b |bin_y - bin_p| (0 with no sample).  n_bins <= 256.
 * The bin sums of a_hat add each a_hat rounded to a multiple of 2^-32, exactly
 * (fixed point within a CTA, fp64 across CTAs while a bin's sum stays below 2^21):
 * the result does not depend on the order of the atomics.
 *
 * dspark_sts_fit: per position, the temperature T_j minimising the binary
 * cross-entropy of sigmoid(logit(a) / T) against y over the stored samples (those
 * with 0 < a < 1): `iters` bisections of log(1/T) in [log 1/64, log 64] on the
 * sign of the derivative sum (sigmoid(z/T) - y) z, z = logit(a) (evaluated in fp64,
 * kept as fp32; the sigmoid in fp32, the sum in fp32 per thread and fp64 across
 * threads); temps fp32 [gamma] out (1 for a position with no usable sample).
 * Workspace: at least dspark_sts_fit_workspace_size(gamma, capacity) bytes,
 * 4-byte aligned.
 * ------------------------------------------------------------------------- */
int dspark_calib_collect(const float* survival, const float* a_hat, const int32_t* windows,
                         const int32_t* cap_len, int mode, int B, int gamma, float* s_a,
                         float* s_ahat, int8_t* s_y, int32_t* count, int capacity, void* stream);
int dspark_calib_ece(const float* s_ahat, const int8_t* s_y, const int32_t* count, int capacity,
                     int gamma, int n_bins, int32_t* bin_n, double* bin_p, double* bin_y,
                     double* ece, void* stream);
size_t dspark_sts_fit_workspace_size(int gamma, int capacity);
int dspark_sts_fit(const float* s_a, const int8_t* s_y, const int32_t* count, int capacity,
                   int gamma, int iters, float* temps, void* workspace, size_t ws_bytes,
                   void* stream);

/* ---------------------------------------------------------------------------
 * dspark_markov_draft -- draft-side sampling of one block with a Markov head
 * ([notes] 05 "Core Innovation A", 5.1-5.3: the parallel backbone gives base
 * logits U_1..U_gamma for the whole block, the sequential head adds the bias
 * B(x_{k-1}, v) ~ (W1 W2)[x_{k-1}, v] of the previous token, rank 256; [lesson]
 * "Zero-overhead scheduling 与 kernel": the drafter's sampling folded into fused
 * kernels).  For k = 0..gamma-1, every request r:
 *     logit[v] = U[r, k, v] + sum_j W1[x, j] W2[j, v]     x = anchor[r] (k = 0)
 *                                                          or draft_tok[r, k-1]
 *     p_draft[r, k, :] = softmax(logit)
 *     draft_tok[r, k]  = argmax_v p_draft[r, k, v] / exp_noise[r, k, v]
 * (the exponential race, lowest index on ties; decided on logit - ln(noise), the
 * same order up to rounding).  p_draft and exp_noise then feed dspark_accept.
 *
 *   U          fp32 [B, gamma, V]  the backbone's base logits
 *   W1         bf16 [V, rank]      token embedding of the head (row x = token x)
 *   W2         bf16 [rank, V]      projection of the head
 *   rank       must be 256 (DSPARK_EUNSUPPORTED otherwise)
 *   anchor     int32 [B]           the last committed token of each request
 *   exp_noise  fp32 [B, gamma, V]  Exp(1) draws, > 0
 *   draft_tok  int32 [B, gamma]    out
 *   p_draft    fp32 [B, gamma, V]  out
 * V a multiple of 128 with V / 128 <= 16 x (SM count) (311,296 on GB300);
 * B <= DSPARK_MAX_B (one launch per 32 requests, or per 16 when V / 128 is above
 * 8 x the SM count); gamma <= DSPARK_MAX_GAMMA; U, W1, W2, exp_noise, p_draft
 * 16-byte aligned.  An anchor outside [0, V) sets DSPARK_DEVERR_BAD_INPUT and
 * reads row 0.  Computation: bf16 products with fp32 accumulation, the softmax
 * and race in fp32.
 *
 * Each launch is a cooperative grid of one CTA per SM that meets at one grid
 * barrier per position; all of its waits are bounded (DSPARK_DEVERR_WAIT_TIMEOUT).
 * Workspace: dspark_markov_draft_workspace_size(V) bytes, 256-byte aligned, ZEROED
 * by the caller before its first use and again after any device error; calls on
 * one stream may share it, calls that may run at once may not.
 * ------------------------------------------------------------------------- */
size_t dspark_markov_draft_workspace_size(int V);
int dspark_markov_draft(const float* U, const void* W1, const void* W2, int rank,
                        const int32_t* anchor, const float* exp_noise, int B, int gamma, int V,
                        int32_t* draft_tok, float* p_draft, void* workspace, size_t ws_bytes,
                        void* stream);

/* ---------------------------------------------------------------------------
 * dspark_step_graph -- the whole verification step as one CUDA graph, with the
 * captured tier chosen on the device ([lesson] "Ragged verify under full CUDA
 * graphs": the packed batch is rounded up to a captured tier and that tier's
 * graph runs; [lesson] "Zero-overhead scheduling 与 kernel": the step runs from
 * device-resident state with no host synchronisation).
 *
 * The graph runs dspark_schedule, dspark_pack_plan and then a switch node with
 * one body per captured tier: body i holds dspark_verify_attn_planned,
 * dspark_accept and dspark_compact with their row counts (max_rows) set to
 * tiers[i], and body n_tiers the same with max_rows for a batch above every tier.
 * The pack kernel selects the body from the M it computes, so consecutive
 * launches may run different tiers without the host reading anything; a batch
 * larger than max_rows sets DSPARK_DEVERR_ROWS_OVERFLOW and runs no body.
 *
 * Every pointer in the descriptor is a device pointer that stays valid (and keeps
 * its meaning) for the life of the graph: a launch reads the buffers' current
 * contents, so the caller refills the input buffers between launches (on the
 * launch stream) and the state (page_table, ctx_len, anchor, free_top, caches)
 * carries over from one step to the next.  Field meanings, layouts and sizes are
 * those of the five calls; workspaces as their *_workspace_size functions give for
 * (B, gamma, max_rows, ...).  Optional:
 *   tier_host  nullable HOST pinned, mapped int32 word: receives each step's tier
 *   body_log   nullable device int32 [1 + log_len]: body_log[0] counts launches
 *              (the caller zeroes it) and body_log[1 + k] receives the body index
 *              run by launch k < log_len (observability of the device's choice)
 * dspark_step_graph_create captures and instantiates the graph on the current
 * device (it launches nothing, and allocates only the graph); it returns
 * DSPARK_EINVAL / DSPARK_EUNSUPPORTED for descriptors the five calls would refuse
 * and DSPARK_ECUDA if graph construction fails.  dspark_step_graph_launch enqueues
 * one step on `stream`; a graph must not run on two streams at once.  The graph
 * cannot be captured into another graph (it holds a conditional node).
 * ------------------------------------------------------------------------- */
typedef struct dspark_step_desc {
  /* shapes */
  int B, gamma, mode;
  int Hq, Hkv, d_qk, d_v, page_size, max_pages, n_pages;
  int V, pdt;
  int max_rows;               /* rows of q, k_new, v_new, p_target, out, lse, row_* */
  int n_tiers;                /* <= DSPARK_MAX_TIERS, ascending, each <= max_rows */
  const int32_t* tiers_host;  /* HOST [n_tiers] */
  const int32_t* tiers;       /* device copy of the same tiers */
  int conf_is_logit, cost_len, max_tokens, max_splits, max_block_rows;
  float scale;
  /* inputs */
  const float* conf;
  const float* sts_temp;
  const float* cost_table;
  const int32_t* draft_tok;
  const void* q;
  const void* k_new;
  const void* v_new;          /* NULL for the latent-KV shape */
  const void* p_target;
  const void* p_draft;
  const float* uniforms;
  const float* exp_noise;
  const int32_t* free_pages;
  /* state, updated in place by every step */
  int32_t* page_table;
  int32_t* ctx_len;
  int32_t* anchor;
  int32_t* free_top;
  void* k_cache;
  void* v_cache;              /* NULL for the latent-KV shape */
  /* outputs */
  int32_t* windows;
  float* a_hat;
  float* survival;            /* nullable */
  int32_t* M;
  double* E;
  int32_t* cu_seqlens;
  int32_t* M_pack;
  int32_t* tier;
  int32_t* row_req;
  int32_t* row_pos;
  int32_t* row_tok;
  float* out;
  float* lse;
  int32_t* accept_len;
  int32_t* cap_len;
  int32_t* out_tok;
  float* cstar;
  int32_t* fallback;
  int32_t* committed;
  int32_t* n_committed;
  int32_t* tier_host;
  int32_t* body_log;
  int log_len;
  /* workspaces */
  void* ws_attn;
  size_t ws_attn_bytes;
  void* ws_accept;
  size_t ws_accept_bytes;
  void* ws_compact;
  size_t ws_compact_bytes;
} dspark_step_desc;

typedef struct dspark_step_graph dspark_step_graph;
int dspark_step_graph_create(const dspark_step_desc* desc, dspark_step_graph** graph_out);
int dspark_step_graph_launch(dspark_step_graph* graph, void* stream);
/* How the graph was captured: DSPARK_STEP_GRAPH_PDL if its kernels keep their
 * programmatic dependencies (each may start while the one before it finishes);
 * otherwise they are plainly stream-ordered. */
#define DSPARK_STEP_GRAPH_PDL 1
int dspark_step_graph_flags(const dspark_step_graph* graph);
/* Frees the graph (NULL is ignored); the caller makes sure no launch is running. */
int dspark_step_graph_destroy(dspark_step_graph* graph);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_H */
