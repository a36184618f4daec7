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
// Limits and sharing: the array is KDA_NOALLOC_SCRATCH_BYTES (64 MiB).  With
// CUDA's lazy module loading (the default) it is reserved on a device when the
// first call there loads this file's module, and it is then held until the
// process exits; a caller with a fixed memory budget should make one call at
// start-up, before its runtime takes its pool.  All calls on a device share
// the array, and it keeps the previous call's contents (the prefill writes
// every byte it reads, so nothing needs clearing).  Calls that overlap on the
// GPU (different streams, or different host threads, without ordering) race
// on it.
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the array on the current device.  Host code cannot use
// the array's name as a device address, so it is looked up, with the device
// current, on every call: a cached address would go stale if the device's
// primary context were torn down and created again (the module, and with it
// the array, is then loaded anew).
kda_status scratch_for_current_device(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    *out = p;
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
