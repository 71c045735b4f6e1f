// Internal launchers of the step kernels (host side).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dspark {

// Where the pack kernel publishes the tier besides its device outputs: a pinned,
// mapped host word (nullable), and the switch handle of a step graph (use = 0: none).
struct TierSel {
  int32_t* host;
  unsigned long long handle;
  int use;
};

int launch_schedule(const float* conf, int conf_is_logit, const float* sts_temp,
                    const float* cost_table, int B, int gamma, int max_tokens, int mode,
                    int32_t* windows, float* a_hat, float* survival, int32_t* M_out,
                    double* E_out, cudaStream_t stream);

int launch_pack(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out, int32_t* tier_out,
                int32_t* row_req, int32_t* row_pos, int32_t* row_tok, const TierSel& ts,
                cudaStream_t stream);

namespace attn {
struct Plan;
}
// launch_pack and, in the same kernel, the attention work list of plan `pl` into the
// attention workspace `attn_ws` (the rest of the attention call then skips it).
int launch_pack_plan(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                     const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                     int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out,
                     int32_t* tier_out, int32_t* row_req, int32_t* row_pos, int32_t* row_tok,
                     int attn_max_rows, int Hkv, int max_splits, const attn::Plan& pl,
                     void* attn_ws, const TierSel& ts, cudaStream_t stream);

// dspark_pack_plan's host checks, then the launch, with the tier also published
// through `ts` (the step graph passes its switch handle).
int pack_plan_checked(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                      const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                      int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out,
                      int32_t* tier_out, int32_t* row_req, int32_t* row_pos, int32_t* row_tok,
                      int Hq, int Hkv, int d_qk, int d_v, int attn_max_rows, int max_splits,
                      int max_block_rows, void* attn_workspace, size_t attn_ws_bytes,
                      const TierSel& ts, cudaStream_t stream);

size_t accept_workspace(int B, int max_rows, int V);
// Wait limit of the acceptance pass's bounded waits on the current device (ns).
uint64_t accept_wait_limit_ns();
int set_accept_wait_limit_ns(unsigned long long ns);
// The wait probe: while on, the acceptance pass first waits on a barrier nothing
// arrives at (its limit must run out).
int accept_wait_probe();
int set_accept_wait_probe(int on);
int launch_accept(const void* p_t, const void* p_d, int pdt, int V, const int32_t* draft_tok,
                  const float* uniforms, const float* exp_noise, const int32_t* windows,
                  const int32_t* cu, int mode, int B, int gamma, int max_rows, int32_t* accept_len,
                  int32_t* cap_len, int32_t* out_tok, float* cstar, int32_t* fallback, void* ws,
                  cudaStream_t stream);

int launch_accept_estimate(const void* p_t, const void* p_d, int pdt, int V,
                           const int32_t* draft_tok, const float* uniforms, const int32_t* windows,
                           const int32_t* cu, const int32_t* accept_len, const int32_t* cap_len,
                           int mode, int B, int gamma, int max_rows, int32_t* cap_lo,
                           int32_t* cap_hi, cudaStream_t stream);

// Address of the fixed scratch array on the current device (looked up once per
// device); nullptr if the lookup fails.
void* accept_fixed_scratch();

int launch_calib_collect(const float* survival, const float* a_hat, const int32_t* windows,
                         const int32_t* cap_len, int mode, int B, int gamma, float* s_a,
                         float* s_ahat, int8_t* s_y, int32_t* count, int cap,
                         cudaStream_t stream);
int launch_calib_ece(const float* s_ahat, const int8_t* s_y, const int32_t* count, int cap,
                     int gamma, int n_bins, int32_t* bin_n, double* bin_p, double* bin_y,
                     double* ece, cudaStream_t stream);
int launch_sts_fit(const float* s_a, const int8_t* s_y, const int32_t* count, int cap, int gamma,
                   int iters, float* zbuf, float* temps, cudaStream_t stream);

// Markov-head draft sampling (markov_draft.cu).  markov_supported: whether a vocabulary
// of V fits the kernel on the current device, and the requests one launch takes.
bool markov_supported(int V, int* group);
size_t markov_workspace(int V);
int launch_markov_draft(const float* U, const void* W1, const void* W2, const int32_t* anchor,
                        const float* exp_noise, int B, int gamma, int V, int32_t* draft_tok,
                        float* p_draft, void* ws, cudaStream_t stream);

size_t compact_workspace(int B);
int launch_compact(const void* k_new, const void* v_new, int row_bytes, int max_rows,
                   const int32_t* cu,
                   const int32_t* accept_len, const int32_t* out_tok, const int32_t* draft_tok,
                   int B, int gamma, int page_size, int max_pages, int n_pages, int32_t* page_table,
                   int32_t* ctx_len, int32_t* anchor, const int32_t* free_pages, int32_t* free_top,
                   void* k_cache, void* v_cache, int32_t* committed, int32_t* n_committed, void* ws,
                   cudaStream_t stream);

}  // namespace dspark
