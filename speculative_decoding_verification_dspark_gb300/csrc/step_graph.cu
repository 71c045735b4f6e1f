// The verification step as one CUDA graph whose captured tier is chosen on the
// device ("DFlash 到 DSpark in SGLang", section "Ragged verify under full CUDA
// graphs": the packed batch is rounded up to a captured tier and that tier's graph
// runs; section "Zero-overhead scheduling 与 kernel": the step runs from
// device-resident state with no host synchronisation).
//
// Graph:  schedule -> pack (+ work list) -> switch(body index) -> body[i]
//   body[i] (i < n_tiers):  verify attention, acceptance and compaction with their
//                           row counts set to tiers[i];
//   body[n_tiers]:          the same with max_rows (a batch above every tier).
// The pack kernel computes M, its tier and the body index, and sets the switch's
// condition (cudaGraphSetConditional); a batch beyond max_rows selects no body.
// The host builds the graph once; each launch is one step, and launches may follow
// one another on a stream with nothing read back in between.

#include <cuda_runtime.h>
#include <stdint.h>

#include <new>
#include <vector>

#include "common.cuh"
#include "dspark.h"
#include "kernels.h"

struct dspark_step_graph {
  int device = -1;
  int flags = 0;  // DSPARK_STEP_GRAPH_PDL: captured with programmatic dependencies
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

namespace dspark {
namespace {

// First node of every body when a log is requested: the body index of this launch.
__global__ void body_mark_kernel(int body, int32_t* __restrict__ log, int log_len) {
  if (threadIdx.x == 0) {
    const int n = log[0];
    if (n < log_len) log[1 + n] = body;
    log[0] = n + 1;
  }
}

struct Capture {  // ends a capture on every exit path
  cudaStream_t s;
  bool on = false;
  ~Capture() {
    if (on) {
      cudaGraph_t g = nullptr;
      cudaStreamEndCapture(s, &g);
      cudaGetLastError();
    }
  }
};

int valid(const dspark_step_desc& d) {
  if (d.B < 1 || d.B > DSPARK_MAX_B || d.gamma < 1 || d.gamma > DSPARK_MAX_GAMMA)
    return DSPARK_EINVAL;
  if (d.n_tiers < 0 || d.n_tiers > DSPARK_MAX_TIERS) return DSPARK_EINVAL;
  if (d.n_tiers > 0 && (!d.tiers_host || !d.tiers)) return DSPARK_EINVAL;
  if (d.max_rows < 1) return DSPARK_EINVAL;
  for (int i = 0; i < d.n_tiers; ++i) {
    if (d.tiers_host[i] < 1 || d.tiers_host[i] > d.max_rows) return DSPARK_EINVAL;
    if (i > 0 && d.tiers_host[i] <= d.tiers_host[i - 1]) return DSPARK_EINVAL;
  }
  if (d.body_log && d.log_len < 0) return DSPARK_EINVAL;
  return DSPARK_OK;
}

// The graph's kernels, captured on `cs` into `g` (head) and the switch bodies.
int build(const dspark_step_desc& d, cudaStream_t cs, cudaGraph_t g) {
  cudaGraphConditionalHandle sel;
  const int n_bodies = d.n_tiers + 1;
  // default value at every launch: no body, unless the pack kernel selects one
  if (cudaGraphConditionalHandleCreate(&sel, g, static_cast<unsigned>(n_bodies),
                                       cudaGraphCondAssignDefault) != cudaSuccess)
    return DSPARK_ECUDA;
  Capture cap{cs};
  if (cudaStreamBeginCaptureToGraph(cs, g, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal) !=
      cudaSuccess)
    return DSPARK_ECUDA;
  cap.on = true;
  int rc = dspark_schedule(d.conf, d.conf_is_logit, d.sts_temp, d.cost_table, d.cost_len, d.B,
                           d.gamma, d.max_tokens, d.mode, d.windows, d.a_hat, d.survival, d.M,
                           d.E, cs);
  if (rc != DSPARK_OK) return rc;
  const TierSel ts{d.tier_host, static_cast<unsigned long long>(sel), 1};
  rc = pack_plan_checked(d.windows, d.ctx_len, d.anchor, d.draft_tok, d.tiers, d.n_tiers, d.B,
                         d.gamma, d.mode, d.max_rows, d.cu_seqlens, d.M_pack, d.tier, d.row_req,
                         d.row_pos, d.row_tok, d.Hq, d.Hkv, d.d_qk, d.d_v, d.max_rows,
                         d.max_splits, d.max_block_rows, d.ws_attn, d.ws_attn_bytes, ts, cs);
  if (rc != DSPARK_OK) return rc;
  // the switch node, appended to the capture after the pack kernel
  cudaStreamCaptureStatus st;
  cudaGraph_t cg = nullptr;
  const cudaGraphNode_t* deps = nullptr;
  size_t ndeps = 0;
  if (cudaStreamGetCaptureInfo(cs, &st, nullptr, &cg, &deps, nullptr, &ndeps) != cudaSuccess ||
      st != cudaStreamCaptureStatusActive)
    return DSPARK_ECUDA;
  cudaGraphNodeParams np = {};
  np.type = cudaGraphNodeTypeConditional;
  np.conditional.handle = sel;
  np.conditional.type = cudaGraphCondTypeSwitch;
  np.conditional.size = static_cast<unsigned>(n_bodies);
  cudaGraphNode_t cnode;
  if (cudaGraphAddNode(&cnode, cg, deps, nullptr, ndeps, &np) != cudaSuccess) return DSPARK_ECUDA;
  if (cudaStreamUpdateCaptureDependencies(cs, &cnode, nullptr, 1,
                                          cudaStreamSetCaptureDependencies) != cudaSuccess)
    return DSPARK_ECUDA;
  cap.on = false;
  cudaGraph_t done = nullptr;
  if (cudaStreamEndCapture(cs, &done) != cudaSuccess) return DSPARK_ECUDA;
  // the bodies (phGraph_out is owned by the node and valid while it exists)
  std::vector<cudaGraph_t> bodies(np.conditional.phGraph_out,
                                  np.conditional.phGraph_out + n_bodies);
  for (int b = 0; b < n_bodies; ++b) {
    const int rows = b < d.n_tiers ? d.tiers_host[b] : d.max_rows;
    Capture bc{cs};
    if (cudaStreamBeginCaptureToGraph(cs, bodies[b], nullptr, nullptr, 0,
                                      cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return DSPARK_ECUDA;
    bc.on = true;
    if (d.body_log) {
      body_mark_kernel<<<1, 32, 0, cs>>>(b, d.body_log, d.log_len);
      if (cudaGetLastError() != cudaSuccess) return DSPARK_ECUDA;
    }
    rc = dspark_verify_attn_planned(d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.n_pages,
                                    d.page_table, d.max_pages, d.ctx_len, d.cu_seqlens, d.B,
                                    d.max_rows, d.Hq, d.Hkv, d.d_qk, d.d_v, d.page_size, d.scale,
                                    d.max_splits, d.max_block_rows, d.out, d.lse, d.ws_attn,
                                    d.ws_attn_bytes, cs);
    if (rc != DSPARK_OK) return rc;
    rc = dspark_accept(d.p_target, d.p_draft, d.pdt, d.V, d.draft_tok, d.uniforms, d.exp_noise,
                       d.windows, d.cu_seqlens, d.mode, d.B, d.gamma, rows, d.accept_len,
                       d.cap_len, d.out_tok, d.cstar, d.fallback, d.ws_accept, d.ws_accept_bytes,
                       cs);
    if (rc != DSPARK_OK) return rc;
    const int row_bytes = d.d_qk == 576 ? 576 * 2 : d.Hkv * d.d_qk * 2;
    rc = dspark_compact(d.k_new, d.v_new, row_bytes, rows, d.cu_seqlens, d.accept_len, d.out_tok,
                        d.draft_tok, d.B, d.gamma, d.page_size, d.max_pages, d.n_pages,
                        d.page_table, d.ctx_len, d.anchor, d.free_pages, d.free_top, d.k_cache,
                        d.v_cache, d.committed, d.n_committed, d.ws_compact, d.ws_compact_bytes,
                        cs);
    if (rc != DSPARK_OK) return rc;
    bc.on = false;
    cudaGraph_t bd = nullptr;
    if (cudaStreamEndCapture(cs, &bd) != cudaSuccess) return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" {

int dspark_step_graph_create(const dspark_step_desc* desc, dspark_step_graph** graph_out) {
  if (!desc || !graph_out) return DSPARK_EINVAL;
  *graph_out = nullptr;
  int rc = valid(*desc);
  if (rc != DSPARK_OK) return rc;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ECUDA;
  cudaStream_t cs;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return DSPARK_ECUDA;
  // Kernels are captured with programmatic dependencies (each may start while the
  // one before it finishes); should the graph not instantiate that way, it is
  // captured again with plain stream ordering.
  dspark_step_graph* out = nullptr;
  for (int attempt = 0; attempt < 2 && rc == DSPARK_OK && !out; ++attempt) {
    g_no_pdl = attempt == 1;
    cudaGraph_t g = nullptr;
    if (cudaGraphCreate(&g, 0) != cudaSuccess) {
      rc = DSPARK_ECUDA;
      break;
    }
    rc = build(*desc, cs, g);
    cudaGraphExec_t exec = nullptr;
    if (rc == DSPARK_OK) {
      if (cudaGraphInstantiate(&exec, g, 0) == cudaSuccess) {
        out = new (std::nothrow) dspark_step_graph;
        if (out) {
          out->device = dev;
          out->flags = attempt == 0 ? DSPARK_STEP_GRAPH_PDL : 0;
          out->graph = g;
          out->exec = exec;
          break;
        }
        cudaGraphExecDestroy(exec);
        rc = DSPARK_ECUDA;
      } else {
        cudaGetLastError();  // try the plain-ordered capture
      }
    }
    cudaGraphDestroy(g);
    if (rc != DSPARK_OK) break;
  }
  g_no_pdl = false;
  cudaStreamDestroy(cs);
  if (rc != DSPARK_OK) return rc;
  if (!out) return DSPARK_ECUDA;
  *graph_out = out;
  return DSPARK_OK;
}

int dspark_step_graph_launch(dspark_step_graph* graph, void* stream) {
  if (!graph || !graph->exec) return DSPARK_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != graph->device) return DSPARK_EINVAL;
  return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_ECUDA;
}

int dspark_step_graph_flags(const dspark_step_graph* graph) { return graph ? graph->flags : 0; }

int dspark_step_graph_destroy(dspark_step_graph* graph) {
  if (!graph) return DSPARK_OK;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
  return DSPARK_OK;
}

}  // extern "C"
