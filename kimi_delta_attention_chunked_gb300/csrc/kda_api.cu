// kda_api.cu -- the exported C ABI: argument checks, path selection, launches.
//
// Nothing here computes any part of KDA; it validates the call, chooses the
// kernel for the (dtype, d_k, d_v, chunk) combination and enqueues it on the
// caller's stream.  See include/kda.h for the contract of each entry point.
#include <algorithm>
#include <cstdint>
#include <cstdio>

#include "common.cuh"
#include "umma.cuh"

namespace {

// Per-device status word, set by kernels that give up waiting.
__device__ int g_kda_status = 0;

int* status_ptr() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_status) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return static_cast<int*>(p);
}

// Failure-detection check: one mbarrier that nothing arrives at, waited on with
// the kernels' own bounded wait; running out records KDA_ERR_TIMEOUT.
__global__ void kda_wait_check_kernel(int* status, long long limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        kda::mbar_init(&bar, 1);
        kda::fence_barrier_init();
        if (!kda::mbar_wait(&bar, 0, limit)) kda::record_status(status, kda::kDevTimeout);
    }
}

#ifdef KDA_DEBUG
// Debug-build precondition: every log-decay value inside [-5, 0] (the bound
// of "LLM architecture at trillion scale", section "The KDA update, in plain
// words"); the first one outside (or a NaN) records KDA_ERR_PRECONDITION.
__global__ void kda_check_log_alpha_kernel(const float* __restrict__ la, long long n, int* status) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float x = la[i];
        if (!(x >= -5.f && x <= 0.f)) {
            kda::record_status(status, KDA_ERR_PRECONDITION);
            return;
        }
    }
}
#endif

// Launches the precondition check of the debug library (nothing in release).
cudaError_t check_log_alpha(const float* la, long long n, cudaStream_t stream, int* status) {
#ifdef KDA_DEBUG
    if (n <= 0 || !la) return cudaSuccess;
    const long long blocks = std::min<long long>((n + 255) / 256, 1216);
    kda_check_log_alpha_kernel<<<(unsigned)blocks, 256, 0, stream>>>(la, n, status);
    return cudaGetLastError();
#else
    (void)la; (void)n; (void)stream; (void)status;
    return cudaSuccess;
#endif
}

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }
bool chunk_ok(int c) { return c == 16 || c == 32 || c == 64; }
bool dtype_ok(kda_dtype t) { return t == KDA_FP32 || t == KDA_BF16; }

kda_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
    return KDA_ERR_CUDA;
}

// Tracing hook state (per host thread).
thread_local void* const* t_events = nullptr;
thread_local int t_n_events = 0;
thread_local int t_next = 0;

// Maximum number of chunks any cu_seqlens with these sizes can produce.
long long chunk_upper_bound(int n_seq, int T_total, int chunk) {
    return (long long)T_total / chunk + (long long)n_seq;
}

}  // namespace

namespace kda_host {
void trace_reset() { t_next = 0; }
void trace_mark(cudaStream_t stream) {
    if (t_events && t_next < t_n_events) {
        (void)cudaEventRecord(static_cast<cudaEvent_t>(t_events[t_next]), stream);
    }
    ++t_next;
}
}  // namespace kda_host

extern "C" {

kda_status kda_set_trace_events(void* const* events, int n_events) {
    if (n_events < 0 || (n_events > 0 && !events)) return KDA_ERR_INVALID_ARG;
    t_events = n_events > 0 ? events : nullptr;
    t_n_events = n_events;
    t_next = 0;
    return KDA_OK;
}

size_t kda_prefill_workspace_size(int n_seq, int T_total, int H, int dk, int dv, int chunk,
                                  kda_dtype dtype) {
    if (n_seq < 0 || T_total < 0 || H <= 0 || !chunk_ok(chunk)) return 0;
    if (!kda_host::tc_supported(dk, dv, chunk, dtype)) return 0;
    return kda_host::tc_workspace_bytes(n_seq, T_total, H, chunk);
}

}  // extern "C"

namespace {

kda_status prefill_impl(const void* q, const void* k, const void* v, const float* log_alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens,
                        const int32_t* cu_seqlens_host, int n_seq, int T_total, int H, int dk, int dv,
                        int chunk, kda_dtype dtype, void* O, float* S_final, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream, int ckpt_every, float* ckpt,
                        int ckpt_cap, int prologue) {
    if (n_seq < 0 || T_total < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk)) return KDA_ERR_UNSUPPORTED;
    if ((long long)T_total * H * (dk > dv ? dk : dv) >= (1LL << 40)) return KDA_ERR_UNSUPPORTED;
    if (T_total > 0 && (!q || !k || !v || !log_alpha || !beta || !O)) return KDA_ERR_INVALID_ARG;
    if (n_seq == 0) return T_total == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (!cu_seqlens) {
        if (cu_seqlens_host) return KDA_ERR_INVALID_ARG;       // host copy of nothing
        if (T_total % n_seq != 0) return KDA_ERR_INVALID_ARG;
    }
    int total_chunks = 0, max_chunks = 0;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[n_seq] != T_total) return KDA_ERR_INVALID_ARG;
        long long tc = 0;
        for (int n = 0; n < n_seq; ++n) {
            const int len = cu_seqlens_host[n + 1] - cu_seqlens_host[n];
            if (len < 0) return KDA_ERR_INVALID_ARG;
            tc += (len + chunk - 1) / chunk;
            max_chunks = std::max(max_chunks, (len + chunk - 1) / chunk);
        }
        total_chunks = (int)tc;
    } else if (!cu_seqlens) {
        const int len = T_total / n_seq;
        total_chunks = n_seq * ((len + chunk - 1) / chunk);
    } else {
        const long long ub = chunk_upper_bound(n_seq, T_total, chunk);
        if (ub > INT32_MAX) return KDA_ERR_UNSUPPORTED;
        total_chunks = (int)ub;
    }
    // O must not overlap any input (S0 == S_final is the one allowed alias).
    if (O && (O == q || O == k || O == v || O == (const void*)log_alpha || O == (const void*)beta))
        return KDA_ERR_INVALID_ARG;

    kda_host::PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.S0 = S0;
    a.cu_seqlens = cu_seqlens; a.n_seq = n_seq; a.T_total = T_total; a.H = H; a.dk = dk;
    a.dv = dv; a.chunk = chunk; a.total_chunks = total_chunks; a.max_chunks = max_chunks; a.dtype = dtype;
    a.O = O;
    a.S_final = S_final; a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.stream = stream; a.ckpt_every = ckpt_every; a.ckpt = ckpt; a.ckpt_cap = ckpt_cap;
    a.prologue = prologue;

    if (kda_host::tc_supported(dk, dv, chunk, dtype)) {
        // the tensor-core kernels move whole 16-byte vectors of every token row
        for (const void* p : {q, k, v, (const void*)log_alpha, (const void*)O})
            if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return KDA_ERR_INVALID_ARG;
        const size_t need = kda_host::tc_workspace_bytes(n_seq, T_total, H, chunk);
        if (workspace_bytes < need || (need && !workspace)) return KDA_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return KDA_ERR_WORKSPACE;
        a.status = status_ptr();
        if (!prologue) {
            const cudaError_t e = check_log_alpha(log_alpha, (long long)T_total * H * dk, stream, a.status);
            if (e != cudaSuccess) return from_cuda(e);
        }
        kda_host::trace_reset();
        kda_host::trace_mark(stream);
        return from_cuda(kda_host::launch_prefill_tc(a));
    }
    a.status = status_ptr();
    if (!prologue) {
        const cudaError_t e = check_log_alpha(log_alpha, (long long)T_total * H * dk, stream, a.status);
        if (e != cudaSuccess) return from_cuda(e);
    }
    kda_host::trace_reset();
    kda_host::trace_mark(stream);
    using L = cudaError_t (*)(const kda_host::PrefillArgs&);
    static const L simt[2][3] = {
        {kda_host::launch_prefill_simt_fp32_c16, kda_host::launch_prefill_simt_fp32_c32,
         kda_host::launch_prefill_simt_fp32_c64},
        {kda_host::launch_prefill_simt_bf16_c16, kda_host::launch_prefill_simt_bf16_c32,
         kda_host::launch_prefill_simt_bf16_c64}};
    const int ci = chunk == 16 ? 0 : (chunk == 32 ? 1 : 2);
    return from_cuda(simt[dtype == KDA_BF16 ? 1 : 0][ci](a));
}


kda_status decode_impl(const void* q, const void* k, const void* v, const float* log_alpha,
                       const float* beta, float* S, int N, int H, int dk, int dv, kda_dtype dtype,
                       void* o, cudaStream_t stream, int prologue) {
    if (N < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if ((long long)N * H >= (1LL << 31)) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !S || !o) return KDA_ERR_INVALID_ARG;
    if (o == q || o == k || o == v || o == (void*)S) return KDA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(S) % 16 != 0) return KDA_ERR_INVALID_ARG;
    kda_host::DecodeArgs a{q, k, v, log_alpha, beta, S, N, H, dk, dv, dtype, o, stream, prologue};
    if (!prologue) {
        const cudaError_t e = check_log_alpha(log_alpha, (long long)N * H * dk, stream, status_ptr());
        if (e != cudaSuccess) return from_cuda(e);
    }
    kda_host::trace_reset();
    kda_host::trace_mark(stream);
    const cudaError_t e = kda_host::launch_decode(a);
    kda_host::trace_mark(stream);
    return from_cuda(e);
}
}  // namespace

extern "C" {

kda_status kda_prefill(const void* q, const void* k, const void* v, const float* log_alpha,
                       const float* beta, const float* S0, const int32_t* cu_seqlens,
                       const int32_t* cu_seqlens_host, int n_seq, int T_total, int H, int dk,
                       int dv, int chunk, kda_dtype dtype, void* O, float* S_final,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return prefill_impl(q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, n_seq, T_total, H, dk, dv,
                        chunk, dtype, O, S_final, workspace, workspace_bytes, stream, 0, nullptr, 0, 0);
}

kda_status kda_prefill_fused(const void* q, const void* k, const void* v, const float* gate,
                             const float* beta_logit, const float* S0, const int32_t* cu_seqlens,
                             const int32_t* cu_seqlens_host, int n_seq, int T_total, int H, int dk, int dv,
                             int chunk, kda_dtype dtype, void* O, float* S_final, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    return prefill_impl(q, k, v, gate, beta_logit, S0, cu_seqlens, cu_seqlens_host, n_seq, T_total, H, dk, dv,
                        chunk, dtype, O, S_final, workspace, workspace_bytes, stream, 0, nullptr, 0, 1);
}

kda_status kda_prefill_ckpt(const void* q, const void* k, const void* v, const float* log_alpha,
                            const float* beta, const float* S0, const int32_t* cu_seqlens,
                            const int32_t* cu_seqlens_host, int n_seq, int T_total, int H, int dk, int dv,
                            int chunk, kda_dtype dtype, void* O, float* S_final, int ckpt_every,
                            float* ckpt, int ckpt_capacity, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
    if (!chunk_ok(chunk)) return KDA_ERR_UNSUPPORTED;
    if (ckpt_every <= 0 || ckpt_every % chunk != 0 || ckpt_capacity < 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_capacity > 0 && !ckpt) return KDA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ckpt) % 16 != 0) return KDA_ERR_INVALID_ARG;   // vector stores
    if (cu_seqlens_host && n_seq > 0) {                 // the caller's buffer must hold every checkpoint
        long long need = 0;
        for (int n = 0; n < n_seq; ++n)
            need += (long long)std::max(0, cu_seqlens_host[n + 1] - cu_seqlens_host[n]) / ckpt_every;
        if (need > ckpt_capacity) return KDA_ERR_INVALID_ARG;
    } else if (!cu_seqlens && n_seq > 0) {
        if ((long long)n_seq * ((T_total / n_seq) / ckpt_every) > ckpt_capacity) return KDA_ERR_INVALID_ARG;
    }
    return prefill_impl(q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, n_seq, T_total, H, dk, dv,
                        chunk, dtype, O, S_final, workspace, workspace_bytes, stream, ckpt_every, ckpt,
                        ckpt_capacity, 0);
}


kda_status kda_decode(const void* q, const void* k, const void* v, const float* log_alpha,
                      const float* beta, float* S, int N, int H, int dk, int dv, kda_dtype dtype,
                      void* o, cudaStream_t stream) {
    return decode_impl(q, k, v, log_alpha, beta, S, N, H, dk, dv, dtype, o, stream, 0);
}

kda_status kda_decode_fused(const void* q, const void* k, const void* v, const float* gate,
                            const float* beta_logit, float* S, int N, int H, int dk, int dv, kda_dtype dtype,
                            void* o, cudaStream_t stream) {
    return decode_impl(q, k, v, gate, beta_logit, S, N, H, dk, dv, dtype, o, stream, 1);
}

kda_status kda_decode_multi(const void* q, const void* k, const void* v, const float* log_alpha,
                            const float* beta, float* S, const int32_t* commit_len, int N, int K, int H, int dk,
                            int dv, kda_dtype dtype, void* o, cudaStream_t stream) {
    if (N < 0 || H <= 0 || K < 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (K > kda_host::decode_multi_max_tokens()) return KDA_ERR_UNSUPPORTED;
    if ((long long)N * H >= (1LL << 31)) return KDA_ERR_UNSUPPORTED;
    if (N == 0 || K == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !S) return KDA_ERR_INVALID_ARG;
    if (o && (o == q || o == k || o == v || o == (void*)S)) return KDA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(S) % 16 != 0) return KDA_ERR_INVALID_ARG;
    kda_host::DecodeArgs a{q, k, v, log_alpha, beta, S, N, H, dk, dv, dtype, o, stream, 0};
    const cudaError_t ec = check_log_alpha(log_alpha, (long long)N * K * H * dk, stream, status_ptr());
    if (ec != cudaSuccess) return from_cuda(ec);
    kda_host::trace_reset();
    kda_host::trace_mark(stream);
    const cudaError_t e = kda_host::launch_decode_multi(a, K, commit_len);
    kda_host::trace_mark(stream);
    return from_cuda(e);
}

kda_status kda_check_wait_timeout(long long limit_cycles, cudaStream_t stream) {
    if (limit_cycles < 0 || limit_cycles > kda::kWaitCycles) return KDA_ERR_INVALID_ARG;
    kda_wait_check_kernel<<<1, 32, 0, stream>>>(status_ptr(), limit_cycles);
    return from_cuda(cudaGetLastError());
}

kda_status kda_get_last_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_kda_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_kda_status, &zero, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return h == 0 ? KDA_OK : static_cast<kda_status>(h);
}

int kda_debug_build(void) {
#ifdef KDA_DEBUG
    return 1;
#else
    return 0;
#endif
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK: success";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: shape, dtype or chunk not supported";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing, too small or misaligned";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime or launch error";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a kernel gave up waiting; outputs incomplete";
        case KDA_ERR_PRECONDITION: return "KDA_ERR_PRECONDITION: log_alpha outside [-5, 0] (debug library check)";
        case KDA_ERR_DEVICE_CHECK:
            return "KDA_ERR_DEVICE_CHECK: a kernel index left its buffer; access skipped (debug library check)";
    }
    return "KDA: unknown status";
}

}  // extern "C"
