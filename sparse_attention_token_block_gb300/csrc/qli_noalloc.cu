// qli_noalloc.cu -- qli_score_topk_static: the indexer for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain scratch memory: a plugin inside a host framework that owns
// every device allocation and forbids its plugins from calling cudaMalloc, a runtime with a fixed
// memory budget carved out at start-up, or latency-critical code that must not call cudaMalloc
// because it can synchronise the device.  For them this entry point keeps the scratch the
// indexer needs (the workspace: a device error word and one score line per query row) in one
// file-scope __device__ array instead of a caller-provided buffer.
//
// Rules of use:
//   * The array holds kStaticScratchBytes (16 MiB).  Every GPU that loads this library reserves
//     it until the process exits.  A problem whose workspace (qli_workspace_size) is larger is
//     rejected with QLI_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
//   * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
//     that device current; make that first call before any stream capture.
//   * All calls share the one array and it keeps the last call's contents.  Each call clears the
//     error word at its start; the score lines are fully rewritten for every visible key before
//     they are read.  Calls that overlap on the GPU (different streams, or concurrent host
//     threads) race on the array and give undefined results: order them on one stream.
//   * Nothing here calls cudaMalloc, cudaFree or any allocating library routine.
#include <cuda_runtime.h>

#include <mutex>

#include "qli_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is a host-side stand-in, not a device address: only the
// address returned by cudaGetSymbolAddress may be handed to kernels.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the array on the current device (looked up once per device)
qli_status static_scratch(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QLI_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return QLI_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return QLI_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return QLI_OK;
}

}  // namespace

extern "C" qli_status qli_score_topk_static(const qli_problem* p, const void* query, const void* key,
                                            const void* weights, const void* q_scale, const void* k_scale,
                                            const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                                            const int32_t* block_table, const int32_t* metadata,
                                            size_t metadata_words, int32_t* sparse_indices,
                                            uint32_t* device_error, void* stream)
{
    const char* why = nullptr;
    qli_status s = qli_validate(p, &why);
    if (s != QLI_OK) return s;
    const size_t need = qli_workspace_size(p);
    if (need == 0 || need > kStaticScratchBytes) return QLI_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    s = static_scratch(&scratch);
    if (s != QLI_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the error word must start at zero for this call
    if (cudaMemsetAsync(scratch, 0, qli::kWsHeaderBytes, st) != cudaSuccess) return QLI_ERR_CUDA;
    s = qli_score_topk(p, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table, metadata,
                       metadata_words, scratch, kStaticScratchBytes, sparse_indices, nullptr, stream);
    if (s != QLI_OK) return s;
    if (device_error &&
        cudaMemcpyAsync(device_error, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return QLI_ERR_CUDA;
    return QLI_OK;
}
