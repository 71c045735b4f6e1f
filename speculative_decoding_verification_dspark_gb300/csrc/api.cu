// C ABI of libdspark.so: argument checks on the host, then the launches.
// Every entry point returns a dspark_status and launches nothing on a bad argument.

#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"
#include "common.cuh"
#include "dspark.h"
#include "kernels.h"

namespace dspark {

__device__ unsigned int g_device_error;

namespace {

struct DeviceState {
  bool ok = false;  // the state below was read
  bool supported = false;
  int sms = 0;
  unsigned int* err = nullptr;
};

// The current device's state, read once per device (thread-safe); nullptr when
// the current device cannot be read.
DeviceState* state() {
  static PerDevice<DeviceState> st;
  static DeviceState none;
  DeviceState s = once_per_device(st, none, [] {
    DeviceState d;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return d;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    void* p = nullptr;
    const bool sym = cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess;
    d.err = static_cast<unsigned int*>(p);
    d.supported = sym && major == 10 && minor == 3 && d.sms > 0;
    d.ok = true;
    return d;
  });
  if (!s.ok) return nullptr;
  int dev = 0;
  cudaGetDevice(&dev);
  return &st.value[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

unsigned int* device_error_word() {
  DeviceState* s = state();
  return s ? s->err : nullptr;
}

int num_sms_cached() {
  DeviceState* s = state();
  return (s && s->sms > 0) ? s->sms : 1;
}

}  // namespace dspark

using namespace dspark;

#define CHECK(cond, code) \
  do {                    \
    if (!(cond)) return (code); \
  } while (0)

static int device_ok() {
  DeviceState* s = state();
  if (!s) return DSPARK_ECUDA;
  return s->supported ? DSPARK_OK : DSPARK_EUNSUPPORTED;
}

static bool attn_shape_ok(int Hq, int Hkv, int d_qk, int d_v, int page_size) {
  if (page_size < 16 || (page_size & (page_size - 1)) != 0) return false;  // power of two
  if (d_qk == 128 && d_v == 128) {
    if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || Hq / Hkv > 128) return false;
    if (page_size < 16 || page_size % 16 != 0) return false;
    return page_size <= 64 ? (64 % page_size == 0) : (page_size % 64 == 0);
  }
  if (d_qk == 576 && d_v == 512) {
    if (Hkv != 1 || Hq != 128) return false;
    if (page_size < 16 || page_size % 16 != 0) return false;
    return page_size <= 32 ? (32 % page_size == 0) : (page_size % 32 == 0);
  }
  return false;
}

namespace dspark {

int pack_plan_checked(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                      const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                      int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out,
                      int32_t* tier_out, int32_t* row_req, int32_t* row_pos, int32_t* row_tok,
                      int Hq, int Hkv, int d_qk, int d_v, int attn_max_rows, int max_splits,
                      int max_block_rows, void* attn_workspace, size_t attn_ws_bytes,
                      const TierSel& ts, cudaStream_t stream) {
  CHECK(windows && ctx_len && anchor && draft_tok && cu_seqlens && M_out && tier_out && row_req &&
            row_pos && row_tok && attn_workspace,
        DSPARK_EINVAL);
  CHECK(n_tiers >= 0 && n_tiers <= DSPARK_MAX_TIERS && (n_tiers == 0 || tiers), DSPARK_EINVAL);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(mode >= DSPARK_COMPACT && mode <= DSPARK_CAP_ACCEPT, DSPARK_EINVAL);
  CHECK(max_rows >= 1 && attn_max_rows >= 1, DSPARK_EINVAL);
  CHECK(attn_shape_ok(Hq, Hkv, d_qk, d_v, 16), DSPARK_EUNSUPPORTED);  // the plan has no page size
  CHECK(max_splits >= 1 && max_splits <= 32, DSPARK_EINVAL);
  CHECK((reinterpret_cast<uintptr_t>(attn_workspace) & 255u) == 0, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  const attn::Plan pl =
      attn::plan(B, attn_max_rows, Hq, Hkv, d_qk, d_v, max_splits, max_block_rows);
  CHECK(attn_ws_bytes >= pl.bytes, DSPARK_ENOSPACE);
  return launch_pack_plan(windows, ctx_len, anchor, draft_tok, tiers, n_tiers, B, gamma, mode,
                          max_rows, cu_seqlens, M_out, tier_out, row_req, row_pos, row_tok,
                          attn_max_rows, Hkv, max_splits, pl, attn_workspace, ts, stream);
}

}  // namespace dspark

extern "C" {

const char* dspark_status_string(int status) {
  switch (status) {
    case DSPARK_OK: return "ok";
    case DSPARK_EINVAL: return "invalid argument";
    case DSPARK_EUNSUPPORTED: return "unsupported shape or device";
    case DSPARK_ECUDA: return "CUDA runtime error";
    case DSPARK_ENOSPACE: return "workspace too small";
    case DSPARK_EDEVICE: return "device error word set";
    default: return "unknown status";
  }
}

int dspark_num_sms(void) { return num_sms_cached(); }

int dspark_set_wait_limit_ns(unsigned long long ns) { return set_accept_wait_limit_ns(ns); }

int dspark_set_wait_probe(int on) { return set_accept_wait_probe(on); }

int dspark_read_device_error(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int* w = device_error_word();
  if (!w) return DSPARK_ECUDA;
  unsigned int h = 0;
  if (cudaMemcpyAsync(&h, w, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return DSPARK_ECUDA;
  if (cudaMemsetAsync(w, 0, sizeof(h), st) != cudaSuccess) return DSPARK_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DSPARK_ECUDA;
  return static_cast<int>(h & 0x7fffffffu);
}

int dspark_schedule(const float* conf, int conf_is_logit, const float* sts_temp,
                    const float* cost_table, int cost_len, int B, int gamma, int max_tokens,
                    int mode, int32_t* windows, float* a_hat, float* survival, int32_t* M_out,
                    double* E_out, void* stream) {
  CHECK(conf && sts_temp && cost_table && windows && a_hat && M_out && E_out, DSPARK_EINVAL);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(B * gamma <= DSPARK_MAX_CANDS, DSPARK_EINVAL);
  CHECK(mode >= DSPARK_COMPACT && mode <= DSPARK_CAP_ACCEPT, DSPARK_EINVAL);
  CHECK(max_tokens >= 1, DSPARK_EINVAL);
  if (mode != DSPARK_STATIC) {
    const long long need = (max_tokens < B * (gamma + 1) ? max_tokens : B * (gamma + 1)) + 1LL;
    CHECK(cost_len >= need, DSPARK_EINVAL);
  }
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  return launch_schedule(conf, conf_is_logit ? 1 : 0, sts_temp, cost_table, B, gamma, max_tokens,
                         mode, windows, a_hat, survival, M_out, E_out,
                         static_cast<cudaStream_t>(stream));
}

int dspark_pack(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out, int32_t* tier_out,
                int32_t* tier_host, int32_t* row_req, int32_t* row_pos, int32_t* row_tok,
                void* stream) {
  CHECK(windows && ctx_len && anchor && draft_tok && cu_seqlens && M_out && tier_out && row_req &&
            row_pos && row_tok,
        DSPARK_EINVAL);
  CHECK(n_tiers >= 0 && n_tiers <= DSPARK_MAX_TIERS && (n_tiers == 0 || tiers), DSPARK_EINVAL);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(mode >= DSPARK_COMPACT && mode <= DSPARK_CAP_ACCEPT, DSPARK_EINVAL);
  CHECK(max_rows >= 1, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  const TierSel ts{tier_host, 0ull, 0};
  return launch_pack(windows, ctx_len, anchor, draft_tok, tiers, n_tiers, B, gamma, mode, max_rows,
                     cu_seqlens, M_out, tier_out, row_req, row_pos, row_tok, ts,
                     static_cast<cudaStream_t>(stream));
}


size_t dspark_verify_attn_workspace_size(int B, int max_rows, int Hq, int Hkv, int d_qk, int d_v,
                                         int max_splits, int max_block_rows) {
  if (B < 1 || max_rows < 1 || max_splits < 1 || max_splits > 32) return 0;
  if (!attn_shape_ok(Hq, Hkv, d_qk, d_v, 16)) return 0;
  return attn::plan(B, max_rows, Hq, Hkv, d_qk, d_v, max_splits, max_block_rows).bytes;
}

static int verify_attn_impl(const void* q, const void* k_new, const void* v_new,
                            const void* k_cache, const void* v_cache, int n_pages,
                            const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                            const int32_t* cu_seqlens, int B, int max_rows, int Hq, int Hkv,
                            int d_qk, int d_v, int page_size, float scale, int max_splits,
                            int max_block_rows, float* out, float* lse, void* workspace,
                            size_t ws_bytes, void* stream, bool planned) {
  CHECK(attn_shape_ok(Hq, Hkv, d_qk, d_v, page_size), DSPARK_EUNSUPPORTED);
  const bool mla = d_qk == 576;
  CHECK(q && k_new && k_cache && page_table && ctx_len && cu_seqlens && out && lse && workspace,
        DSPARK_EINVAL);
  CHECK(mla || (v_new && v_cache), DSPARK_EINVAL);
  CHECK(aligned16(q) && aligned16(k_new) && aligned16(k_cache) && aligned16(out) &&
            (mla || (aligned16(v_new) && aligned16(v_cache))),
        DSPARK_EINVAL);
  CHECK((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, DSPARK_EINVAL);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && max_rows >= 1 && n_pages >= 1 && max_pages >= 1,
        DSPARK_EINVAL);
  CHECK(max_splits >= 1 && max_splits <= 32, DSPARK_EINVAL);
  CHECK(scale > 0.f, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  const attn::Plan pl = attn::plan(B, max_rows, Hq, Hkv, d_qk, d_v, max_splits, max_block_rows);
  CHECK(ws_bytes >= pl.bytes, DSPARK_ENOSPACE);
  return attn::launch(q, k_new, v_new, k_cache, v_cache, n_pages, page_table, max_pages, ctx_len,
                      cu_seqlens, B, max_rows, Hq, Hkv, d_qk, d_v, page_size, scale, max_splits,
                      out, lse, workspace, pl, static_cast<cudaStream_t>(stream), planned);
}

int dspark_verify_attn(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                       const void* v_cache, int n_pages, const int32_t* page_table, int max_pages,
                       const int32_t* ctx_len, const int32_t* cu_seqlens, int B, int max_rows,
                       int Hq, int Hkv, int d_qk, int d_v, int page_size, float scale,
                       int max_splits, int max_block_rows, float* out, float* lse, void* workspace,
                       size_t ws_bytes, void* stream) {
  return verify_attn_impl(q, k_new, v_new, k_cache, v_cache, n_pages, page_table, max_pages,
                          ctx_len, cu_seqlens, B, max_rows, Hq, Hkv, d_qk, d_v, page_size, scale,
                          max_splits, max_block_rows, out, lse, workspace, ws_bytes, stream, false);
}

int dspark_verify_attn_planned(const void* q, const void* k_new, const void* v_new,
                               const void* k_cache, const void* v_cache, int n_pages,
                               const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                               const int32_t* cu_seqlens, int B, int max_rows, int Hq, int Hkv,
                               int d_qk, int d_v, int page_size, float scale, int max_splits,
                               int max_block_rows, float* out, float* lse, void* workspace,
                               size_t ws_bytes, void* stream) {
  return verify_attn_impl(q, k_new, v_new, k_cache, v_cache, n_pages, page_table, max_pages,
                          ctx_len, cu_seqlens, B, max_rows, Hq, Hkv, d_qk, d_v, page_size, scale,
                          max_splits, max_block_rows, out, lse, workspace, ws_bytes, stream, true);
}

int dspark_pack_plan(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                     const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                     int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out,
                     int32_t* tier_out, int32_t* tier_host, int32_t* row_req, int32_t* row_pos,
                     int32_t* row_tok, int Hq, int Hkv, int d_qk, int d_v, int attn_max_rows,
                     int max_splits, int max_block_rows, void* attn_workspace, size_t attn_ws_bytes,
                     void* stream) {
  const TierSel ts{tier_host, 0ull, 0};
  return pack_plan_checked(windows, ctx_len, anchor, draft_tok, tiers, n_tiers, B, gamma, mode,
                           max_rows, cu_seqlens, M_out, tier_out, row_req, row_pos, row_tok, Hq,
                           Hkv, d_qk, d_v, attn_max_rows, max_splits, max_block_rows,
                           attn_workspace, attn_ws_bytes, ts, static_cast<cudaStream_t>(stream));
}

size_t dspark_accept_workspace_size(int B, int gamma, int max_rows, int V) {
  if (B < 1 || gamma < 1 || max_rows < 1 || V < 8) return 0;
  return accept_workspace(B, max_rows, V);
}

int dspark_accept(const void* p_target, const void* p_draft, int pdt, int V,
                  const int32_t* draft_tok, const float* uniforms, const float* exp_noise,
                  const int32_t* windows, const int32_t* cu_seqlens, int mode, int B, int gamma,
                  int max_rows, int32_t* accept_len, int32_t* cap_len, int32_t* out_tok,
                  float* cstar, int32_t* fallback, void* workspace, size_t ws_bytes,
                  void* stream) {
  CHECK(p_target && p_draft && draft_tok && uniforms && exp_noise && windows && cu_seqlens &&
            accept_len && cap_len && out_tok && cstar && workspace,
        DSPARK_EINVAL);
  CHECK(pdt == DSPARK_F32 || pdt == DSPARK_BF16, DSPARK_EINVAL);
  CHECK(V >= 8 && V % 8 == 0, DSPARK_EUNSUPPORTED);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(mode >= DSPARK_COMPACT && mode <= DSPARK_CAP_ACCEPT, DSPARK_EINVAL);
  CHECK(max_rows >= 1, DSPARK_EINVAL);
  CHECK(aligned16(p_target) && aligned16(p_draft) && aligned16(exp_noise), DSPARK_EINVAL);
  CHECK((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  CHECK(ws_bytes >= accept_workspace(B, max_rows, V), DSPARK_ENOSPACE);
  return launch_accept(p_target, p_draft, pdt, V, draft_tok, uniforms, exp_noise, windows,
                       cu_seqlens, mode, B, gamma, max_rows, accept_len, cap_len, out_tok, cstar,
                       fallback, workspace, static_cast<cudaStream_t>(stream));
}

int dspark_accept_noalloc(const void* p_target, const void* p_draft, int pdt, int V,
                          const int32_t* draft_tok, const float* uniforms,
                          const float* exp_noise, const int32_t* windows,
                          const int32_t* cu_seqlens, int mode, int B, int gamma, int max_rows,
                          int32_t* accept_len, int32_t* cap_len, int32_t* out_tok, float* cstar,
                          int32_t* fallback, void* stream) {
  CHECK(p_target && p_draft && draft_tok && uniforms && exp_noise && windows && cu_seqlens &&
            accept_len && cap_len && out_tok && cstar,
        DSPARK_EINVAL);
  CHECK(pdt == DSPARK_F32 || pdt == DSPARK_BF16, DSPARK_EINVAL);
  CHECK(V >= 8 && V % 8 == 0, DSPARK_EUNSUPPORTED);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(mode >= DSPARK_COMPACT && mode <= DSPARK_CAP_ACCEPT, DSPARK_EINVAL);
  CHECK(max_rows >= 1, DSPARK_EINVAL);
  CHECK(aligned16(p_target) && aligned16(p_draft) && aligned16(exp_noise), DSPARK_EINVAL);
  CHECK(accept_workspace(B, max_rows, V) <= DSPARK_ACCEPT_NOALLOC_SCRATCH_BYTES, DSPARK_ENOSPACE);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  void* scratch = accept_fixed_scratch();
  CHECK(scratch != nullptr, DSPARK_ECUDA);
  return launch_accept(p_target, p_draft, pdt, V, draft_tok, uniforms, exp_noise, windows,
                       cu_seqlens, mode, B, gamma, max_rows, accept_len, cap_len, out_tok, cstar,
                       fallback, scratch, static_cast<cudaStream_t>(stream));
}

int dspark_block_accept_estimate(const void* p_target, const void* p_draft, int pdt, int V,
                                 const int32_t* draft_tok, const float* uniforms,
                                 const int32_t* windows, const int32_t* cu_seqlens,
                                 const int32_t* accept_len, const int32_t* cap_len, int mode,
                                 int B, int gamma, int max_rows, int32_t* cap_lo, int32_t* cap_hi,
                                 void* stream) {
  CHECK(p_target && p_draft && draft_tok && uniforms && windows && cu_seqlens && accept_len &&
            cap_len && cap_lo && cap_hi,
        DSPARK_EINVAL);
  CHECK(pdt == DSPARK_F32 || pdt == DSPARK_BF16, DSPARK_EINVAL);
  CHECK(V >= 1, DSPARK_EINVAL);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(mode >= DSPARK_COMPACT && mode <= DSPARK_CAP_ACCEPT, DSPARK_EINVAL);
  CHECK(max_rows >= 1, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  return launch_accept_estimate(p_target, p_draft, pdt, V, draft_tok, uniforms, windows,
                                cu_seqlens, accept_len, cap_len, mode, B, gamma, max_rows, cap_lo,
                                cap_hi, static_cast<cudaStream_t>(stream));
}

size_t dspark_compact_workspace_size(int B) {
  if (B < 1) return 0;
  return compact_workspace(B);
}

int dspark_compact(const void* k_new, const void* v_new, int row_bytes, int max_rows,
                   const int32_t* cu_seqlens,
                   const int32_t* accept_len, const int32_t* out_tok, const int32_t* draft_tok,
                   int B, int gamma, int page_size, int max_pages, int n_pages,
                   int32_t* page_table, int32_t* ctx_len, int32_t* anchor,
                   const int32_t* free_pages, int32_t* free_top, void* k_cache, void* v_cache,
                   int32_t* committed, int32_t* n_committed, void* workspace, size_t ws_bytes,
                   void* stream) {
  CHECK(k_new && cu_seqlens && accept_len && out_tok && draft_tok && page_table && ctx_len &&
            anchor && free_pages && free_top && k_cache && committed && n_committed && workspace,
        DSPARK_EINVAL);
  CHECK((v_new == nullptr) == (v_cache == nullptr), DSPARK_EINVAL);
  CHECK(row_bytes >= 16 && row_bytes % 16 == 0, DSPARK_EINVAL);
  CHECK(max_rows >= 1, DSPARK_EINVAL);
  CHECK(aligned16(k_new) && aligned16(k_cache) && (!v_new || (aligned16(v_new) && aligned16(v_cache))),
        DSPARK_EINVAL);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(page_size >= 1 && max_pages >= 1 && n_pages >= 1, DSPARK_EINVAL);
  CHECK((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  CHECK(ws_bytes >= compact_workspace(B), DSPARK_ENOSPACE);
  return launch_compact(k_new, v_new, row_bytes, max_rows, cu_seqlens, accept_len, out_tok, draft_tok, B,
                        gamma, page_size, max_pages, n_pages, page_table, ctx_len, anchor,
                        free_pages, free_top, k_cache, v_cache, committed, n_committed, workspace,
                        static_cast<cudaStream_t>(stream));
}

int dspark_calib_collect(const float* survival, const float* a_hat, const int32_t* windows,
                         const int32_t* cap_len, int mode, int B, int gamma, float* s_a,
                         float* s_ahat, int8_t* s_y, int32_t* count, int capacity, void* stream) {
  CHECK(survival && a_hat && windows && cap_len && s_a && s_ahat && s_y && count, DSPARK_EINVAL);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(mode >= DSPARK_COMPACT && mode <= DSPARK_CAP_ACCEPT, DSPARK_EINVAL);
  CHECK(capacity >= 1, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  return launch_calib_collect(survival, a_hat, windows, cap_len, mode, B, gamma, s_a, s_ahat, s_y,
                              count, capacity, static_cast<cudaStream_t>(stream));
}

int dspark_calib_ece(const float* s_ahat, const int8_t* s_y, const int32_t* count, int capacity,
                     int gamma, int n_bins, int32_t* bin_n, double* bin_p, double* bin_y,
                     double* ece, void* stream) {
  CHECK(s_ahat && s_y && count && bin_n && bin_p && bin_y && ece, DSPARK_EINVAL);
  CHECK(gamma >= 1 && gamma <= DSPARK_MAX_GAMMA && capacity >= 1, DSPARK_EINVAL);
  CHECK(n_bins >= 1 && n_bins <= DSPARK_MAX_ECE_BINS, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  return launch_calib_ece(s_ahat, s_y, count, capacity, gamma, n_bins, bin_n, bin_p, bin_y, ece,
                          static_cast<cudaStream_t>(stream));
}

size_t dspark_sts_fit_workspace_size(int gamma, int capacity) {
  if (gamma < 1 || capacity < 1) return 0;
  return static_cast<size_t>(gamma) * static_cast<size_t>(capacity) * sizeof(float);
}

int dspark_sts_fit(const float* s_a, const int8_t* s_y, const int32_t* count, int capacity,
                   int gamma, int iters, float* temps, void* workspace, size_t ws_bytes,
                   void* stream) {
  CHECK(s_a && s_y && count && temps && workspace, DSPARK_EINVAL);
  CHECK(gamma >= 1 && gamma <= DSPARK_MAX_GAMMA && capacity >= 1, DSPARK_EINVAL);
  CHECK(iters >= 0 && iters <= 1000, DSPARK_EINVAL);
  CHECK((reinterpret_cast<uintptr_t>(workspace) & 3u) == 0, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  CHECK(ws_bytes >= dspark_sts_fit_workspace_size(gamma, capacity), DSPARK_ENOSPACE);
  return launch_sts_fit(s_a, s_y, count, capacity, gamma, iters, static_cast<float*>(workspace),
                        temps, static_cast<cudaStream_t>(stream));
}

size_t dspark_markov_draft_workspace_size(int V) {
  if (V < 128 || V % 128 != 0) return 0;
  return markov_workspace(V);
}

int dspark_markov_draft(const float* U, const void* W1, const void* W2, int rank,
                        const int32_t* anchor, const float* exp_noise, int B, int gamma, int V,
                        int32_t* draft_tok, float* p_draft, void* workspace, size_t ws_bytes,
                        void* stream) {
  CHECK(U && W1 && W2 && anchor && exp_noise && draft_tok && p_draft && workspace, DSPARK_EINVAL);
  CHECK(rank == 256, DSPARK_EUNSUPPORTED);
  CHECK(V >= 128 && V % 128 == 0, DSPARK_EUNSUPPORTED);
  CHECK(B >= 1 && B <= DSPARK_MAX_B && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA, DSPARK_EINVAL);
  CHECK(aligned16(U) && aligned16(W1) && aligned16(W2) && aligned16(exp_noise) && aligned16(p_draft),
        DSPARK_EINVAL);
  CHECK((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, DSPARK_EINVAL);
  int rc = device_ok();
  if (rc != DSPARK_OK) return rc;
  CHECK(markov_supported(V, nullptr), DSPARK_EUNSUPPORTED);
  CHECK(ws_bytes >= markov_workspace(V), DSPARK_ENOSPACE);
  return launch_markov_draft(U, W1, W2, anchor, exp_noise, B, gamma, V, draft_tok, p_draft,
                             workspace, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
