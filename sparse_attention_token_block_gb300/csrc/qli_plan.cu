// qli_plan.cu -- execution plans: the metadata, score and top-k launches of one indexer call
// captured into a CUDA graph once and replayed (the launch path is paid at capture time).  The
// launches keep their programmatic-dependent-launch attribute, which the capture turns into
// programmatic graph edges, so the replayed kernels overlap their prologues as on a stream.
#include <cuda_runtime.h>

#include <new>

#include "qli.h"

struct qli_plan {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" qli_status qli_plan_create(const qli_problem* p, int with_metadata, const void* query,
                                      const void* key, const void* weights, const void* q_scale,
                                      const void* k_scale, const int32_t* seq_lens_q,
                                      const int32_t* seq_lens_k, const int32_t* block_table,
                                      int32_t* metadata, size_t metadata_words, void* workspace,
                                      size_t workspace_bytes, int32_t* sparse_indices, float* sparse_values,
                                      qli_plan** plan)
{
    if (!plan) return QLI_ERR_INVALID_ARG;
    *plan = nullptr;
    qli_status s = qli_validate(p, nullptr);
    if (s != QLI_OK) return s;
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return QLI_ERR_CUDA;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(cs);
        return QLI_ERR_CUDA;
    }
    if (with_metadata) s = qli_metadata(p, seq_lens_q, seq_lens_k, metadata, metadata_words, cs);
    if (s == QLI_OK)
        s = qli_score_topk(p, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table,
                           metadata, metadata_words, workspace, workspace_bytes, sparse_indices, sparse_values, cs);
    cudaGraph_t graph = nullptr;
    const cudaError_t end = cudaStreamEndCapture(cs, &graph);   // always ends the capture
    cudaStreamDestroy(cs);
    if (s != QLI_OK || end != cudaSuccess || !graph) {
        if (graph) cudaGraphDestroy(graph);
        (void)cudaGetLastError();
        return s != QLI_OK ? s : QLI_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
        cudaGraphDestroy(graph);
        (void)cudaGetLastError();
        return QLI_ERR_CUDA;
    }
    qli_plan* q = new (std::nothrow) qli_plan{graph, exec};
    if (!q) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
        return QLI_ERR_CUDA;
    }
    *plan = q;
    return QLI_OK;
}

extern "C" qli_status qli_plan_launch(const qli_plan* plan, void* stream)
{
    if (!plan) return QLI_ERR_INVALID_ARG;
    return cudaGraphLaunch(plan->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

extern "C" void qli_plan_destroy(qli_plan* plan)
{
    if (!plan) return;
    cudaGraphExecDestroy(plan->exec);
    cudaGraphDestroy(plan->graph);
    delete plan;
}
