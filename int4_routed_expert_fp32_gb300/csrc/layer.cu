// The whole routed int4 MoE layer on one stream (Kimi K3 latent up-projection
// page, KimiSparseMoeBlock.forward listing): the router sees the full-width x;
// the latent down-projection (if any) feeds the dispatch; experts; combine
// (+ RMSNorm and up-projection on the latent path); then, when configured,
// the shared expert on the full-width x is added to the output.
#include "combine.cuh"
#include "common.cuh"
#include "dispatch.cuh"

namespace moe {

struct LayerWs {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* row_slot;
  int32_t* inv_row;
  uint16_t* x_lat;     // [T, L] (latent)
  void* x_sorted;      // [T*k, D] fp16 or int8, pair order
  float* x_scale;      // [T*k] (act_bits 8)
  void* y_sorted;      // [T*k, D] bf16, or fp32 on the latent path
  bool y_f32;
  uint16_t* comb;      // [T, L] (latent)
  uint16_t* x_dev;     // [T, H] staging of the host-buffer variant
  uint16_t* out_dev;   // [T, H]
  void* scratch;       // shared by router, dispatch and experts (used one after another)
  size_t scratch_bytes;
  size_t total;
};

static size_t scratch_need(const moe_config& c) {
  const int D = c.L > 0 ? c.L : c.H;
  const int R = c.T * c.k;
  size_t a = moe_route_workspace_size(c.T, c.H, c.E);
  size_t b = moe_dispatch_workspace_size(c.T, c.E, c.k);
  size_t f = expert_ffn_ws_bytes(c.E, D, c.I, R, c.act_bits);
  size_t m = a > b ? a : b;
  m = m > f ? m : f;
  // the shared expert runs last and reuses the scratch
  const size_t sh = c.I_shared > 0 ? shared_expert_ws_bytes(c.T, c.H, c.I_shared) : 0;
  return m > sh ? m : sh;
}

// Carve the workspace; with base == nullptr only the total size is computed.
static LayerWs carve(const moe_config& c, void* base) {
  const size_t T = c.T, k = c.k, E = c.E, H = c.H;
  const size_t L = c.L > 0 ? c.L : 0;
  const size_t D = L ? L : H;
  const size_t R = T * k;
  LayerWs w{};
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? static_cast<char*>(base) + off : nullptr;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return p;
  };
  w.topk_idx = static_cast<int32_t*>(take(R * 4));
  w.topk_w = static_cast<float*>(take(R * 4));
  w.counts = static_cast<int32_t*>(take(E * 4));
  w.offsets = static_cast<int32_t*>(take((E + 1) * 4));
  w.row_token = static_cast<int32_t*>(take(R * 4));
  w.row_slot = static_cast<int32_t*>(take(R * 4));
  w.inv_row = static_cast<int32_t*>(take(R * 4));
  w.x_lat = L ? static_cast<uint16_t*>(take(T * L * 2)) : nullptr;
  w.x_sorted = take(R * D * (c.act_bits == 8 ? 1 : 2));
  w.x_scale = c.act_bits == 8 ? static_cast<float*>(take(R * 4)) : nullptr;
  w.y_f32 = L > 0;  // keeps the expert outputs unrounded before the latent RMSNorm
  w.y_sorted = take(R * D * (w.y_f32 ? 4 : 2));
  w.comb = L ? static_cast<uint16_t*>(take(T * L * 2)) : nullptr;
  w.x_dev = static_cast<uint16_t*>(take(T * H * 2));
  w.out_dev = static_cast<uint16_t*>(take(T * H * 2));
  w.scratch_bytes = scratch_need(c);
  w.scratch = take(w.scratch_bytes);
  w.total = off;
  return w;
}

static int validate(const moe_config* c, const moe_weights* w) {
  if (!c || !w) return MOE_ERR_INVALID;
  if (c->T < 0 || c->H <= 0 || c->E <= 0 || c->k <= 0 || c->I <= 0 || c->L < 0)
    return MOE_ERR_INVALID;
  if (c->H % 64 || c->I % 64 || (c->L > 0 && c->L % 64)) return MOE_ERR_UNSUPPORTED;
  if (c->E > kMaxExperts || c->k > c->E || c->k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (c->act_bits != 16 && c->act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (!(c->eps >= 0.f)) return MOE_ERR_INVALID;
  if (!w->router_w || !w->router_bias || !w->gate_packed || !w->gate_scale || !w->up_packed ||
      !w->up_scale || !w->down_packed || !w->down_scale)
    return MOE_ERR_INVALID;
  if (c->L > 0 && (!w->lat_down || !w->lat_up)) return MOE_ERR_INVALID;
  if (!aligned(w->gate_packed, 16) || !aligned(w->up_packed, 16) || !aligned(w->down_packed, 16) ||
      !aligned(w->gate_scale, 4) || !aligned(w->up_scale, 4) || !aligned(w->down_scale, 4))
    return MOE_ERR_INVALID;
  if (c->L > 0 && (!aligned(w->lat_down, 16) || !aligned(w->lat_up, 16) ||
                   (w->lat_norm && !aligned(w->lat_norm, 16))))
    return MOE_ERR_INVALID;
  if (c->I_shared < 0) return MOE_ERR_INVALID;
  if (c->I_shared > 0) {
    if (c->I_shared % 64) return MOE_ERR_UNSUPPORTED;
    if (!w->shared_gate || !w->shared_up || !w->shared_down || !aligned(w->shared_gate, 16) ||
        !aligned(w->shared_up, 16) || !aligned(w->shared_down, 16))
      return MOE_ERR_INVALID;
  }
  return MOE_OK;
}

static int routed(const moe_config& c, const moe_weights& w, const uint16_t* x, uint16_t* out,
                  const LayerWs& ws, cudaStream_t s) {
  const int D = c.L > 0 ? c.L : c.H;
  const int R = c.T * c.k;
  int rc = route_with_terms(x, w.router_w, w.router_w_terms, w.router_bias, c.T, c.H, c.E, c.k,
                            c.renorm, ws.topk_idx, ws.topk_w, ws.scratch, ws.scratch_bytes, s);
  if (rc) return rc;
  const uint16_t* u = x;
  if (c.L > 0) {
    Range r("latent_down");
    rc = launch_linear_bf16(x, w.lat_down, c.T, c.L, c.H, ws.x_lat, s);
    if (rc) return rc;
    u = ws.x_lat;
  }
  // expert-sorted rows in the expert kernels' pair order (fp16 / int8)
  {
    Range r("dispatch");
    rc = launch_dispatch_pairs(ws.topk_idx, u, c.T, D, c.E, c.k, c.act_bits, ws.counts,
                               ws.offsets, ws.row_token, ws.row_slot, ws.inv_row, ws.x_sorted,
                               ws.x_scale, ws.scratch, s);
  }
  if (rc) return rc;
  {
    Range r("expert_ffn");
    rc = launch_expert_ffn(ws.x_sorted, ws.x_scale, ws.offsets, c.E, D, c.I, R, c.T,
                           w.gate_packed, w.gate_scale, w.up_packed, w.up_scale, w.down_packed,
                           w.down_scale, c.act_bits, ws.y_sorted, ws.y_f32, ws.scratch, s);
  }
  if (rc) return rc;
  if (c.L > 0) {
    {
      Range r("combine_rmsnorm");
      rc = launch_combine(ws.y_sorted, ws.y_f32, ws.inv_row, ws.topk_w, c.T, c.L, c.k, w.lat_norm,
                          c.eps, ws.comb, s);
    }
    if (rc) return rc;
    Range r("latent_up");
    return launch_linear_bf16(ws.comb, w.lat_up, c.T, c.H, c.L, out, s);
  }
  Range r("combine");
  return launch_combine(ws.y_sorted, ws.y_f32, ws.inv_row, ws.topk_w, c.T, c.H, c.k, nullptr, 0.f,
                        out, s);
}

static int forward(const moe_config& c, const moe_weights& w, const uint16_t* x, uint16_t* out,
                   const LayerWs& ws, cudaStream_t s) {
  const int rc = routed(c, w, x, out, ws, s);
  if (rc || c.I_shared == 0) return rc;
  Range r("shared_expert");
  return launch_shared_expert(x, c.T, c.H, c.I_shared, w.shared_gate, w.shared_up, w.shared_down,
                              1, out, ws.scratch, s);
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_workspace_size(const moe_config* cfg) {
  if (!cfg || cfg->T < 0 || cfg->k <= 0 || cfg->E <= 0 || cfg->H <= 0 || cfg->I <= 0) return 0;
  return carve(*cfg, nullptr).total;
}

extern "C" int moe_layer_forward(const moe_config* cfg, const moe_weights* w, const uint16_t* x,
                                 uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  moe::Range range_("moe_layer_forward");
  int rc = validate(cfg, w);
  if (rc) return rc;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !out || !ws) return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(ws, 256)) return MOE_ERR_INVALID;
  const LayerWs lw = carve(*cfg, ws);
  if (ws_bytes < lw.total) return MOE_ERR_WORKSPACE;
  return forward(*cfg, *w, x, out, lw, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_layer_forward_host(const moe_config* cfg, const moe_weights* w,
                                      const uint16_t* x_host, uint16_t* out_host, void* ws,
                                      size_t ws_bytes, void* stream) {
  moe::Range range_("moe_layer_forward_host");
  int rc = validate(cfg, w);
  if (rc) return rc;
  if (cfg->T == 0) return MOE_OK;
  if (!x_host || !out_host || !ws || !aligned(ws, 256)) return MOE_ERR_INVALID;
  const LayerWs lw = carve(*cfg, ws);
  if (ws_bytes < lw.total) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)cfg->T * cfg->H * sizeof(uint16_t);
  MOE_TRY_CUDA(cudaMemcpyAsync(lw.x_dev, x_host, bytes, cudaMemcpyHostToDevice, s));
  rc = forward(*cfg, *w, lw.x_dev, lw.out_dev, lw, s);
  if (rc) return rc;
  MOE_TRY_CUDA(cudaMemcpyAsync(out_host, lw.out_dev, bytes, cudaMemcpyDeviceToHost, s));
  return MOE_OK;
}

// ---- captured layer calls (CUDA graphs) -----------------------------------

struct moe_layer_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  uint64_t launches;  // library kernels in the captured call
};

extern "C" int moe_layer_graph_create(const moe_config* cfg, const moe_weights* w, const void* x,
                                      void* out, int host, void* ws, size_t ws_bytes,
                                      void* stream, moe_layer_graph** graph) {
  moe::Range range_("moe_layer_graph_create");
  if (!graph) return MOE_ERR_INVALID;
  *graph = nullptr;
  // the argument checks of the captured call, before any capture begins
  int rc = validate(cfg, w);
  if (rc) return rc;
  if (!x || !out || !ws || !aligned(ws, 256)) return MOE_ERR_INVALID;
  if (!host && (!aligned(x, 16) || !aligned(out, 16))) return MOE_ERR_INVALID;
  if (ws_bytes < carve(*cfg, nullptr).total) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  MOE_TRY_CUDA(cudaStreamIsCapturing(s, &cs));
  if (cs != cudaStreamCaptureStatusNone) return MOE_ERR_INVALID;
  const uint64_t n0 = moe_launch_count();
  MOE_TRY_CUDA(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  rc = host ? moe_layer_forward_host(cfg, w, static_cast<const uint16_t*>(x),
                                     static_cast<uint16_t*>(out), ws, ws_bytes, stream)
            : moe_layer_forward(cfg, w, static_cast<const uint16_t*>(x),
                                static_cast<uint16_t*>(out), ws, ws_bytes, stream);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(s, &g);  // ends the capture on every path
  if (rc || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    if (rc) return rc;
    note_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, g, 0);
  if (ei != cudaSuccess) {
    cudaGraphDestroy(g);
    note_cuda_error(ei);
    return MOE_ERR_CUDA;
  }
  *graph = new moe_layer_graph{g, exec, moe_launch_count() - n0};
  return MOE_OK;
}

extern "C" int moe_layer_graph_launch(const moe_layer_graph* graph, void* stream) {
  if (!graph) return MOE_ERR_INVALID;
  MOE_TRY_CUDA(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)));
  for (uint64_t i = 0; i < graph->launches; ++i) count_launch();
  return MOE_OK;
}

extern "C" void moe_layer_graph_destroy(moe_layer_graph* graph) {
  if (!graph) return;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
}

// ---- pipelined calls on host buffers ---------------------------------------
//
// Two device slots for x and out; call n uses slot n % 2.  Its input copy
// (own stream) waits until call n - 2's compute has read the slot, its
// compute (the caller's stream, a captured graph per slot) waits for the
// input copy and for call n - 2's output copy, and its output copy (own
// stream) waits for the compute.  So the copies of one call overlap the
// compute of its neighbours.

struct moe_layer_pipe {
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t in_done[2] = {}, comp_done[2] = {}, out_done[2] = {}, join = nullptr;
  moe_layer_graph* g[2] = {};
  uint16_t* x_dev[2] = {};
  uint16_t* out_dev[2] = {};
  size_t bytes = 0;  // T * H * 2
  uint64_t n = 0;    // calls submitted
};

static size_t pipe_slot_bytes(const moe_config& c) {
  return align_up((size_t)c.T * c.H * sizeof(uint16_t), 256);
}

extern "C" size_t moe_layer_pipe_workspace_size(const moe_config* cfg) {
  const size_t layer = moe_workspace_size(cfg);
  if (!layer) return 0;
  return layer + 4 * pipe_slot_bytes(*cfg);
}

static void pipe_free(moe_layer_pipe* p) {
  if (!p) return;
  // the last calls' compute (on the caller's stream) and copies finish first
  for (int j = 0; j < 2; ++j)
    if (p->comp_done[j]) cudaEventSynchronize(p->comp_done[j]);
  if (p->s_in) cudaStreamSynchronize(p->s_in);
  if (p->s_out) cudaStreamSynchronize(p->s_out);
  for (int j = 0; j < 2; ++j) {
    moe_layer_graph_destroy(p->g[j]);
    if (p->in_done[j]) cudaEventDestroy(p->in_done[j]);
    if (p->comp_done[j]) cudaEventDestroy(p->comp_done[j]);
    if (p->out_done[j]) cudaEventDestroy(p->out_done[j]);
  }
  if (p->join) cudaEventDestroy(p->join);
  if (p->s_in) cudaStreamDestroy(p->s_in);
  if (p->s_out) cudaStreamDestroy(p->s_out);
  delete p;
}

extern "C" int moe_layer_pipe_create(const moe_config* cfg, const moe_weights* w, void* ws,
                                     size_t ws_bytes, void* stream, moe_layer_pipe** pipe) {
  moe::Range range_("moe_layer_pipe_create");
  if (!pipe) return MOE_ERR_INVALID;
  *pipe = nullptr;
  int rc = validate(cfg, w);
  if (rc) return rc;
  if (cfg->T == 0) return MOE_ERR_INVALID;
  if (!ws || !aligned(ws, 256)) return MOE_ERR_INVALID;
  const size_t layer = carve(*cfg, nullptr).total;
  if (ws_bytes < moe_layer_pipe_workspace_size(cfg)) return MOE_ERR_WORKSPACE;
  moe_layer_pipe* p = new moe_layer_pipe;
  p->bytes = (size_t)cfg->T * cfg->H * sizeof(uint16_t);
  char* slots = static_cast<char*>(ws) + layer;
  for (int j = 0; j < 2; ++j) {
    p->x_dev[j] = reinterpret_cast<uint16_t*>(slots + (2 * j) * pipe_slot_bytes(*cfg));
    p->out_dev[j] = reinterpret_cast<uint16_t*>(slots + (2 * j + 1) * pipe_slot_bytes(*cfg));
  }
  cudaError_t e = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking);
  for (int j = 0; j < 2 && e == cudaSuccess; ++j) {
    e = cudaEventCreateWithFlags(&p->in_done[j], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->comp_done[j], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->out_done[j], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    pipe_free(p);
    return MOE_ERR_CUDA;
  }
  for (int j = 0; j < 2; ++j) {
    rc = moe_layer_graph_create(cfg, w, p->x_dev[j], p->out_dev[j], 0, ws, layer, stream, &p->g[j]);
    if (rc) {
      pipe_free(p);
      return rc;
    }
  }
  *pipe = p;
  return MOE_OK;
}

extern "C" int moe_layer_pipe_submit(moe_layer_pipe* p, const uint16_t* x_host, uint16_t* out_host,
                                     void* stream) {
  if (!p || !x_host || !out_host) return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int j = static_cast<int>(p->n & 1);
  // input: slot j's x is free once call n - 2's compute has read it
  MOE_TRY_CUDA(cudaStreamWaitEvent(p->s_in, p->comp_done[j], 0));
  MOE_TRY_CUDA(cudaMemcpyAsync(p->x_dev[j], x_host, p->bytes, cudaMemcpyHostToDevice, p->s_in));
  MOE_TRY_CUDA(cudaEventRecord(p->in_done[j], p->s_in));
  // compute: the input has landed and call n - 2's output has been copied out
  MOE_TRY_CUDA(cudaStreamWaitEvent(s, p->in_done[j], 0));
  MOE_TRY_CUDA(cudaStreamWaitEvent(s, p->out_done[j], 0));
  const int rc = moe_layer_graph_launch(p->g[j], stream);
  if (rc) return rc;
  MOE_TRY_CUDA(cudaEventRecord(p->comp_done[j], s));
  // output
  MOE_TRY_CUDA(cudaStreamWaitEvent(p->s_out, p->comp_done[j], 0));
  MOE_TRY_CUDA(cudaMemcpyAsync(out_host, p->out_dev[j], p->bytes, cudaMemcpyDeviceToHost,
                               p->s_out));
  MOE_TRY_CUDA(cudaEventRecord(p->out_done[j], p->s_out));
  ++p->n;
  return MOE_OK;
}

extern "C" int moe_layer_pipe_join(moe_layer_pipe* p, void* stream) {
  if (!p) return MOE_ERR_INVALID;
  MOE_TRY_CUDA(cudaEventRecord(p->join, p->s_out));
  MOE_TRY_CUDA(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), p->join, 0));
  return MOE_OK;
}

extern "C" void moe_layer_pipe_destroy(moe_layer_pipe* p) { pipe_free(p); }
