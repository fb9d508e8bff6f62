// pa_graph.cu -- one decode step over L layers, captured once into a CUDA graph.
//
// A transformer's decode step runs the same KV write and paged decode in every
// layer, over the same block tables and slots (the block manager is layer
// agnostic: block p is the same slot range in every layer's cache).  Capturing
// the L x (pa_write_kv, pa_decode) launches into one graph and replaying it
// removes the host's per-launch cost from the step; the launches keep their
// programmatic-dependent edges inside the graph.  The decode work list depends
// only on the tables and lengths, which all layers share, so the graph runs the
// plan kernel once per step and each layer only its decode and merge kernels.
// ("Paged Attention and vLLM",
// "Continuous Batching and Scheduler": a new batch decision every iteration;
// "KV Cache Optimization and Management", recap: the cache grows by one token
// per layer per generated token.)
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "../../include/pa.h"
#include "pa_internal.h"

struct pa_step_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

namespace {

const char *at(const void *base, int64_t off) { return static_cast<const char *>(base) + off; }

}  // namespace

extern "C" {

pa_step_graph *pa_step_graph_create(const pa_dims *dims, int32_t num_layers, void *k_caches, void *v_caches,
                                    int64_t cache_layer_stride, const void *q, int64_t q_layer_stride,
                                    const void *k_new, const void *v_new, int64_t kv_new_layer_stride,
                                    const int64_t *slot_mapping, int32_t num_tokens, const int32_t *block_tables,
                                    const int32_t *context_lens, float scale, float *out, int64_t out_layer_stride,
                                    void *workspace, size_t workspace_bytes, int32_t *status) {
    int32_t dummy;
    if (!status) status = &dummy;
    *status = PA_ERR_INVALID;
    if (!dims || num_layers <= 0 || cache_layer_stride < 0 || q_layer_stride < 0 || kv_new_layer_stride < 0 ||
        out_layer_stride < 0)
        return nullptr;
    if (num_layers > 1) {
        // layers must not overlap: each stride covers one layer's tensor (sizes in
        // double, so that absurd dims cannot overflow before they are rejected)
        const double eb = dims->kv_dtype == PA_F32 ? 4.0 : 2.0;
        const double row = (double)dims->num_seqs * dims->num_q_heads * dims->head_dim;
        const double pool = (double)dims->num_blocks * dims->num_kv_heads * dims->block_size * dims->head_dim * eb;
        const double kv_new = (double)num_tokens * dims->num_kv_heads * dims->head_dim * eb;
        if ((double)cache_layer_stride < pool || (double)q_layer_stride < row * eb ||
            (double)kv_new_layer_stride < kv_new || (double)out_layer_stride < row * 4.0)
            return nullptr;
    }
    pa_step_graph *g = new (std::nothrow) pa_step_graph();
    if (!g) return nullptr;
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
        delete g;
        *status = PA_ERR_CUDA;
        return nullptr;
    }
    // Relaxed mode: the launch paths may make first-use set-up calls (kernel
    // attributes, symbol lookups, tensor-map encoding) that are not stream work.
    int32_t rc = PA_OK;
    if (out_layer_stride % 16 != 0) rc = PA_ERR_INVALID;
    if (rc == PA_OK && cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed) != cudaSuccess) rc = PA_ERR_CUDA;
    auto out_l = [&](int32_t l) { return reinterpret_cast<float *>(const_cast<char *>(at(out, l * out_layer_stride))); };
    if (rc == PA_OK)  // the work list (and every layer's zero rows) once for the step
        rc = pa::decode_call(dims, q, k_caches, v_caches, block_tables, context_lens, scale, out_l(0), workspace,
                             workspace_bytes, st, pa::DecodePhase::kPlanOnly, num_layers, out_layer_stride / 4);
    for (int32_t l = 0; l < num_layers && rc == PA_OK; ++l) {
        void *kc = const_cast<char *>(at(k_caches, l * cache_layer_stride));
        void *vc = const_cast<char *>(at(v_caches, l * cache_layer_stride));
        rc = pa_write_kv(dims, at(k_new, l * kv_new_layer_stride), at(v_new, l * kv_new_layer_stride),
                         slot_mapping, num_tokens, kc, vc, st);
        if (rc != PA_OK) break;
        rc = pa::decode_call(dims, at(q, l * q_layer_stride), kc, vc, block_tables, context_lens, scale, out_l(l),
                             workspace, workspace_bytes, st, pa::DecodePhase::kRunOnly, 1, 0);
    }
    cudaGraph_t graph = nullptr;
    const cudaError_t end = cudaStreamEndCapture(st, &graph);
    if (rc == PA_OK && (end != cudaSuccess || !graph)) rc = PA_ERR_CUDA;
    if (rc == PA_OK && cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess) rc = PA_ERR_CUDA;
    cudaStreamDestroy(st);
    if (rc != PA_OK) {
        if (g->exec) cudaGraphExecDestroy(g->exec);
        if (graph) cudaGraphDestroy(graph);
        delete g;
        *status = rc;
        return nullptr;
    }
    g->graph = graph;
    *status = PA_OK;
    return g;
}

int32_t pa_step_graph_launch(pa_step_graph *graph, void *stream) {
    if (!graph || !graph->exec) return PA_ERR_INVALID;
    return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

void pa_step_graph_destroy(pa_step_graph *graph) {
    if (!graph) return;
    if (graph->exec) cudaGraphExecDestroy(graph->exec);
    if (graph->graph) cudaGraphDestroy(graph->graph);
    delete graph;
}

}  // extern "C"
