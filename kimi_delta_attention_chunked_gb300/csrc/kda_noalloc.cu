// kda_noalloc.cu -- kda_prefill_noalloc: prefill whose scratch lives in a
// fixed, file-scope device array instead of caller-provided memory.
//
// Some callers cannot allocate device memory for a workspace: runtimes that
// hand out all device memory from their own pre-sized pool and forbid
// libraries from calling cudaMalloc, plugin interfaces that pass a library
// only its input and output buffers, and deployments that fix their memory
// footprint at start-up.  This entry point serves them: it takes the same
// inputs and outputs as kda_prefill, and uses the array below as the
// workspace.  It allocates nothing.
//
// Limits and sharing: the array is KDA_NOALLOC_SCRATCH_BYTES (64 MiB) and is
// held by every GPU that loads the library until the process exits.  All
// calls on a device share it, and it keeps the previous call's contents (the
// prefill writes every byte it reads, so nothing needs clearing).  Calls that
// overlap on the GPU (different streams, or different host threads, without
// ordering) race on it.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (host code cannot use the array's name as a device address).
kda_status scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_prefill_noalloc(const void* q, const void* k, const void* v, const float* log_alpha,
                               const float* beta, const float* S0, const int32_t* cu_seqlens,
                               const int32_t* cu_seqlens_host, int n_seq, int T_total, int H, int dk,
                               int dv, int chunk, kda_dtype dtype, void* O, float* S_final,
                               cudaStream_t stream) {
    const size_t need = kda_prefill_workspace_size(n_seq, T_total, H, dk, dv, chunk, dtype);
    if (need > kScratchBytes) return KDA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        const kda_status st = scratch_for_current_device(&scratch);
        if (st != KDA_OK) return st;
    }
    return kda_prefill(q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, n_seq, T_total, H, dk,
                       dv, chunk, dtype, O, S_final, scratch, need > 0 ? kScratchBytes : 0, stream);
}

}  // extern "C"
