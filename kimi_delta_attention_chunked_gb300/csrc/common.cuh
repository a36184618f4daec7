// common.cuh -- small device helpers shared by the KDA kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Device-side status codes (written into the status word by a kernel).
enum : int { kDevOk = 0, kDevTimeout = 5 };

// Upper bound on how long a kernel waits for an asynchronous event (an
// mbarrier phase) before it records KDA_ERR_TIMEOUT and gives up: ~2 s at the
// GB300 boost clock.  A correct launch never gets close.
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, kDevOk, code);
}

// Debug-build device checks (compiled with KDA_DEBUG): a condition that fails
// records KDA_ERR_DEVICE_CHECK in the status word and evaluates to false, so
// that the caller skips the access it guards.  In release builds the check is
// not compiled and evaluates to true.
#ifdef KDA_DEBUG
#define KDA_DCHECK(status, cond) ((cond) ? true : (::kda::record_status((status), KDA_ERR_DEVICE_CHECK), false))
#else
#define KDA_DCHECK(status, cond) true
#endif

template <typename T> struct io;
template <> struct io<float> {
    static __device__ __forceinline__ float ld(const float* p) { return *p; }
    static __device__ __forceinline__ void st(float* p, float x) { *p = x; }
};
template <> struct io<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}

// Index of the first checkpoint of sequence n: sum over earlier sequences of
// floor(len / every).  Block-wide sum; every thread of the block must call it.
// lens_of(m) returns the length of sequence m.
template <typename LenFn>
__device__ __forceinline__ int ckpt_base(int n, int every, LenFn lens_of) {
    __shared__ int red[32];
    int part = 0;
    for (int m = threadIdx.x; m < n; m += blockDim.x) part += lens_of(m) / every;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = part;
    __syncthreads();
    int tot = 0;
    for (int i = 0; i < nw; ++i) tot += red[i];
    __syncthreads();
    return tot;
}

// ---- fused parameter-free prologue of the Kimi Linear layer ("Kimi K3: the
// manos, the mythos, the legendos", section "Kimi Linear": q and k are L2
// normalised; the log-decay is kept inside (-5, 0) per the "LLM architecture at
// trillion scale" page, section "The KDA update, in plain words").
//   log_alpha = clamp(-softplus(a), -5, -1e-4),  beta = sigmoid(b),
//   x_hat = x / sqrt(sum x^2 + kNormEps)  over d_k, per (token, head).
constexpr float kNormEps = 1e-6f;
__device__ __forceinline__ float prologue_log_alpha(float a) {
    const float sp = a > 20.f ? a : log1pf(__expf(a));
    return fminf(fmaxf(-sp, -5.f), -1e-4f);
}
__device__ __forceinline__ float prologue_beta(float b) { return 1.f / (1.f + __expf(-b)); }

}  // namespace kda

// Host-side launchers implemented by the kernel translation units.
namespace kda_host {

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* beta;
    const float* S0;
    const int32_t* cu_seqlens;   // device, or nullptr (equal lengths)
    int n_seq, T_total, H, dk, dv, chunk;
    int total_chunks;            // exact when the host knows cu_seqlens, else an upper bound
    int max_chunks;              // chunks of the longest sequence (host-known lengths), else 0
    kda_dtype dtype;
    void* O;
    float* S_final;
    void* workspace;
    size_t workspace_bytes;
    cudaStream_t stream;
    int* status;                 // device status word
    int ckpt_every;              // 0: no checkpoints; else a multiple of chunk (tokens)
    float* ckpt;                 // [ckpt_cap, H, dk, dv]
    int ckpt_cap;
    int prologue;                // 1: q, k unnormalised, log_alpha / beta are pre-activations
};

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* beta;
    float* S;
    int N, H, dk, dv;
    kda_dtype dtype;
    void* o;
    cudaStream_t stream;
    int prologue;                // as in PrefillArgs
};

// Records the next trace event (see kda_set_trace_events) on `stream`.
void trace_mark(cudaStream_t stream);
void trace_reset();

cudaError_t launch_decode(const DecodeArgs& a);
int decode_multi_max_tokens();
cudaError_t launch_decode_multi(const DecodeArgs& a, int K, const int32_t* commit_len);
cudaError_t launch_prefill_simt_fp32_c16(const PrefillArgs& a);
cudaError_t launch_prefill_simt_fp32_c32(const PrefillArgs& a);
cudaError_t launch_prefill_simt_fp32_c64(const PrefillArgs& a);
cudaError_t launch_prefill_simt_bf16_c16(const PrefillArgs& a);
cudaError_t launch_prefill_simt_bf16_c32(const PrefillArgs& a);
cudaError_t launch_prefill_simt_bf16_c64(const PrefillArgs& a);
bool tc_supported(int dk, int dv, int chunk, kda_dtype dt);
size_t tc_workspace_bytes(int n_seq, int T_total, int H, int chunk);
cudaError_t launch_prefill_tc(const PrefillArgs& a);

}  // namespace kda_host
