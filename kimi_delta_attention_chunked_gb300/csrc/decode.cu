// decode.cu -- fused single-token KDA decode step, fp32 state updated in place.
//
// Per (sequence, head) the step is the per-token form of "Kimi K3: the manos,
// the mythos, the legendos", section "FlashKDA Algorithm":
//     Sbar = Diag(alpha) S            (alpha = exp(log_alpha), one per key row)
//     x    = Sbar^T k,   y = Sbar^T q (reductions over the d_k rows)
//     u    = beta (v - x)
//     S    = Sbar + k u^T             (written back in place)
//     o    = S^T q = y + (k^T q) u
// The pages count ~7 d^2 flops and ~8 d^2 bytes (fp32 state read + write) per
// head-step (section "Complexity Analysis"), so the step is HBM-bound: the
// kernel streams each 64 KiB state exactly once, with 16-byte loads and
// stores marked evict-first, and keeps the whole state tile in registers
// between the read and the write.
//
// Layout: one CTA of 256 threads per (sequence, head).  A row of S (d_v
// floats) is covered by d_v/4 consecutive threads holding one float4 each;
// the CTA covers 256/(d_v/4) rows per pass and d_k/(rows per pass) passes.
// All state loads are issued before anything else so that ~64 KiB per CTA is
// in flight.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kThreads, 2)
kda_decode_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                  const TIn* __restrict__ v, const float* __restrict__ log_alpha,
                  const float* __restrict__ beta, float* __restrict__ S,
                  TIn* __restrict__ o, int prologue) {
    constexpr int LPR = DV / 4;                       // threads per state row
    constexpr int RPP = kThreads / LPR;               // rows per pass
    constexpr int NPASS = (DK + RPP - 1) / RPP;
    static_assert(DV % 4 == 0 && kThreads % LPR == 0, "bad tile");

    __shared__ float s_k[DK], s_q[DK], s_a[DK];
    __shared__ float4 s_x[RPP][LPR];
    __shared__ float4 s_y[RPP][LPR];

    const size_t unit = blockIdx.x;                   // n * H + h
    const int tid = threadIdx.x;
    const int c4 = tid % LPR;                         // float4 column group
    const int r0 = tid / LPR;                         // first row of this thread
    float* Su = S + unit * (size_t)DK * DV;

    // 1. issue every state load first
    float4 s[NPASS];
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
        const int i = r0 + p * RPP;
        if (i < DK) s[p] = __ldcs(reinterpret_cast<const float4*>(Su + (size_t)i * DV) + c4);
    }
    // 2. the token's key, query and gate
    for (int i = tid; i < DK; i += kThreads) {
        s_k[i] = kda::io<TIn>::ld(k + unit * DK + i);
        s_q[i] = kda::io<TIn>::ld(q + unit * DK + i);
        const float la = log_alpha[unit * DK + i];
        s_a[i] = __expf(prologue ? kda::prologue_log_alpha(la) : la);
    }
    float4 vv;
    vv.x = kda::io<TIn>::ld(v + unit * DV + 4 * c4 + 0);
    vv.y = kda::io<TIn>::ld(v + unit * DV + 4 * c4 + 1);
    vv.z = kda::io<TIn>::ld(v + unit * DV + 4 * c4 + 2);
    vv.w = kda::io<TIn>::ld(v + unit * DV + 4 * c4 + 3);
    const float bt = prologue ? kda::prologue_beta(beta[unit]) : beta[unit];
    __syncthreads();
    // fused prologue: k and q scaled to unit length (1 / norms from warp 0)
    float nk = 1.f, nq = 1.f;
    if (prologue) {
        __shared__ float s_n[2];
        if (tid < 32) {
            float sk = 0.f, sq = 0.f;
            for (int i = tid; i < DK; i += 32) { sk = fmaf(s_k[i], s_k[i], sk); sq = fmaf(s_q[i], s_q[i], sq); }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) {
                sk += __shfl_xor_sync(0xffffffffu, sk, o2);
                sq += __shfl_xor_sync(0xffffffffu, sq, o2);
            }
            if (tid == 0) { s_n[0] = rsqrtf(sk + kda::kNormEps); s_n[1] = rsqrtf(sq + kda::kNormEps); }
        }
        __syncthreads();
        nk = s_n[0];
        nq = s_n[1];
    }

    // 3. decay the rows and form the partial reductions x = Sbar^T k, y = Sbar^T q
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
        const int i = r0 + p * RPP;
        if (i < DK) {
            const float a = s_a[i], ki = s_k[i] * nk, qi = s_q[i] * nq;
            s[p].x *= a; s[p].y *= a; s[p].z *= a; s[p].w *= a;
            x.x = fmaf(s[p].x, ki, x.x); x.y = fmaf(s[p].y, ki, x.y);
            x.z = fmaf(s[p].z, ki, x.z); x.w = fmaf(s[p].w, ki, x.w);
            y.x = fmaf(s[p].x, qi, y.x); y.y = fmaf(s[p].y, qi, y.y);
            y.z = fmaf(s[p].z, qi, y.z); y.w = fmaf(s[p].w, qi, y.w);
        }
    }
    s_x[r0][c4] = x;
    s_y[r0][c4] = y;
    __syncthreads();

    // 4. finish the reductions for this thread's 4 columns; u = beta (v - x)
    float4 X = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int r = 0; r < RPP; ++r) {
        const float4 t = s_x[r][c4];
        X.x += t.x; X.y += t.y; X.z += t.z; X.w += t.w;
    }
    float4 u;
    u.x = bt * (vv.x - X.x); u.y = bt * (vv.y - X.y);
    u.z = bt * (vv.z - X.z); u.w = bt * (vv.w - X.w);

    // 5. write the new state S = Sbar + k u^T
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
        const int i = r0 + p * RPP;
        if (i < DK) {
            const float ki = s_k[i] * nk;
            float4 w;
            w.x = fmaf(ki, u.x, s[p].x); w.y = fmaf(ki, u.y, s[p].y);
            w.z = fmaf(ki, u.z, s[p].z); w.w = fmaf(ki, u.w, s[p].w);
            __stcs(reinterpret_cast<float4*>(Su + (size_t)i * DV) + c4, w);
        }
    }

    // 6. read-out o = Sbar^T q + (k^T q) u  (one row of threads writes it)
    if (r0 == 0) {
        float4 Y = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < RPP; ++r) {
            const float4 t = s_y[r][c4];
            Y.x += t.x; Y.y += t.y; Y.z += t.z; Y.w += t.w;
        }
        float kq = 0.f;
        for (int i = 0; i < DK; ++i) kq = fmaf(s_k[i], s_q[i], kq);
        kq *= nk * nq;
        TIn* ou = o + unit * DV + 4 * c4;
        kda::io<TIn>::st(ou + 0, fmaf(kq, u.x, Y.x));
        kda::io<TIn>::st(ou + 1, fmaf(kq, u.y, Y.y));
        kda::io<TIn>::st(ou + 2, fmaf(kq, u.z, Y.z));
        kda::io<TIn>::st(ou + 3, fmaf(kq, u.w, Y.w));
    }
}

// Multi-token verify step: K tokens per sequence applied to a register-resident
// state, every o_t produced, the state written back after commit_len[n] of them.
// Same thread layout as the single-token kernel; the K tokens' q, k, v, gates
// are staged in shared memory first.
constexpr int kMaxVerify = 16;

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kThreads, 2)
kda_decode_multi_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                        const float* __restrict__ log_alpha, const float* __restrict__ beta,
                        float* __restrict__ S, const int32_t* __restrict__ commit_len, int K, int H,
                        TIn* __restrict__ o) {
    constexpr int LPR = DV / 4;
    constexpr int RPP = kThreads / LPR;
    constexpr int NPASS = (DK + RPP - 1) / RPP;
    __shared__ float s_k[kMaxVerify][DK], s_q[kMaxVerify][DK], s_a[kMaxVerify][DK];
    __shared__ float s_v[kMaxVerify][DV];
    __shared__ float s_b[kMaxVerify], s_kq[kMaxVerify];
    __shared__ float4 s_x[2][RPP][LPR];               // partial reductions, alternating by token
    __shared__ float4 s_y[2][RPP][LPR];

    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const size_t unit = blockIdx.x;                   // n * H + h
    const int tid = threadIdx.x;
    const int c4 = tid % LPR, r0 = tid / LPR;
    float* Su = S + unit * (size_t)DK * DV;
    int commit = commit_len ? commit_len[n] : K;
    commit = min(max(commit, 0), K);

    float4 s[NPASS];
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
        const int i = r0 + p * RPP;
        if (i < DK) s[p] = __ldcs(reinterpret_cast<const float4*>(Su + (size_t)i * DV) + c4);
    }
    for (int e = tid; e < K * DK; e += kThreads) {
        const int t = e / DK, i = e % DK;
        const size_t off = (((size_t)n * K + t) * H + h) * DK + i;
        s_k[t][i] = kda::io<TIn>::ld(k + off);
        s_q[t][i] = kda::io<TIn>::ld(q + off);
        s_a[t][i] = __expf(log_alpha[off]);
    }
    for (int e = tid; e < K * DV; e += kThreads) {
        const int t = e / DV, j = e % DV;
        s_v[t][j] = kda::io<TIn>::ld(v + (((size_t)n * K + t) * H + h) * DV + j);
    }
    for (int t = tid; t < K; t += kThreads) s_b[t] = beta[((size_t)n * K + t) * H + h];
    __syncthreads();
    // k_t . q_t of every token, one warp per token
    {
        const int w = tid >> 5, lane = tid & 31;
        for (int t = w; t < K; t += kThreads / 32) {
            float kq = 0.f;
            for (int i = lane; i < DK; i += 32) kq = fmaf(s_k[t][i], s_q[t][i], kq);
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o2);
            if (lane == 0) s_kq[t] = kq;
        }
    }
    __syncthreads();

    for (int t = 0; t < K; ++t) {
        const int pb = t & 1;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
        for (int p = 0; p < NPASS; ++p) {
            const int i = r0 + p * RPP;
            if (i < DK) {
                const float a = s_a[t][i], ki = s_k[t][i], qi = s_q[t][i];
                s[p].x *= a; s[p].y *= a; s[p].z *= a; s[p].w *= a;
                x.x = fmaf(s[p].x, ki, x.x); x.y = fmaf(s[p].y, ki, x.y);
                x.z = fmaf(s[p].z, ki, x.z); x.w = fmaf(s[p].w, ki, x.w);
                y.x = fmaf(s[p].x, qi, y.x); y.y = fmaf(s[p].y, qi, y.y);
                y.z = fmaf(s[p].z, qi, y.z); y.w = fmaf(s[p].w, qi, y.w);
            }
        }
        s_x[pb][r0][c4] = x;
        s_y[pb][r0][c4] = y;
        // one barrier per token: token t + 1 fills the other buffer, and token
        // t + 2 reuses this one only after every thread passed token t + 1's barrier
        __syncthreads();
        float4 X = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int r = 0; r < RPP; ++r) {
            const float4 a = s_x[pb][r][c4];
            X.x += a.x; X.y += a.y; X.z += a.z; X.w += a.w;
        }
        const float bt = s_b[t];
        float4 u;
        u.x = bt * (s_v[t][4 * c4 + 0] - X.x); u.y = bt * (s_v[t][4 * c4 + 1] - X.y);
        u.z = bt * (s_v[t][4 * c4 + 2] - X.z); u.w = bt * (s_v[t][4 * c4 + 3] - X.w);
#pragma unroll
        for (int p = 0; p < NPASS; ++p) {
            const int i = r0 + p * RPP;
            if (i < DK) {
                const float ki = s_k[t][i];
                s[p].x = fmaf(ki, u.x, s[p].x); s[p].y = fmaf(ki, u.y, s[p].y);
                s[p].z = fmaf(ki, u.z, s[p].z); s[p].w = fmaf(ki, u.w, s[p].w);
            }
        }
        if (o && r0 == 0) {
            float4 Y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
            for (int r = 0; r < RPP; ++r) {
                const float4 b = s_y[pb][r][c4];
                Y.x += b.x; Y.y += b.y; Y.z += b.z; Y.w += b.w;
            }
            const float kq = s_kq[t];
            TIn* ou = o + (((size_t)n * K + t) * H + h) * DV + 4 * c4;
            kda::io<TIn>::st(ou + 0, fmaf(kq, u.x, Y.x));
            kda::io<TIn>::st(ou + 1, fmaf(kq, u.y, Y.y));
            kda::io<TIn>::st(ou + 2, fmaf(kq, u.z, Y.z));
            kda::io<TIn>::st(ou + 3, fmaf(kq, u.w, Y.w));
        }
        if (t + 1 == commit) {                         // the accepted prefix ends here
#pragma unroll
            for (int p = 0; p < NPASS; ++p) {
                const int i = r0 + p * RPP;
                if (i < DK) __stcs(reinterpret_cast<float4*>(Su + (size_t)i * DV) + c4, s[p]);
            }
        }
    }
}

template <int DK, int DV, typename TIn>
cudaError_t launch_multi(const kda_host::DecodeArgs& a, int K, const int32_t* commit_len) {
    const unsigned units = (unsigned)((size_t)a.N * a.H);
    if (units == 0 || K == 0) return cudaSuccess;
    kda_decode_multi_kernel<DK, DV, TIn><<<units, kThreads, 0, a.stream>>>(
        static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v), a.log_alpha,
        a.beta, a.S, commit_len, K, a.H, static_cast<TIn*>(a.o));
    return cudaGetLastError();
}

template <int DK, int DV, typename TIn>
cudaError_t launch(const kda_host::DecodeArgs& a) {
    const unsigned units = (unsigned)((size_t)a.N * a.H);
    if (units == 0) return cudaSuccess;
    kda_decode_kernel<DK, DV, TIn><<<units, kThreads, 0, a.stream>>>(
        static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v),
        a.log_alpha, a.beta, a.S, static_cast<TIn*>(a.o), a.prologue);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t dispatch_dims(const kda_host::DecodeArgs& a) {
#define KDA_DECODE_CASE(DK_, DV_) \
    if (a.dk == DK_ && a.dv == DV_) return launch<DK_, DV_, TIn>(a);
    KDA_DECODE_CASE(32, 32) KDA_DECODE_CASE(32, 64) KDA_DECODE_CASE(32, 128)
    KDA_DECODE_CASE(64, 32) KDA_DECODE_CASE(64, 64) KDA_DECODE_CASE(64, 128)
    KDA_DECODE_CASE(128, 32) KDA_DECODE_CASE(128, 64) KDA_DECODE_CASE(128, 128)
#undef KDA_DECODE_CASE
    return cudaErrorNotSupported;
}

template <typename TIn>
cudaError_t dispatch_multi(const kda_host::DecodeArgs& a, int K, const int32_t* cl) {
#define KDA_MULTI_CASE(DK_, DV_) \
    if (a.dk == DK_ && a.dv == DV_) return launch_multi<DK_, DV_, TIn>(a, K, cl);
    KDA_MULTI_CASE(32, 32) KDA_MULTI_CASE(32, 64) KDA_MULTI_CASE(32, 128)
    KDA_MULTI_CASE(64, 32) KDA_MULTI_CASE(64, 64) KDA_MULTI_CASE(64, 128)
    KDA_MULTI_CASE(128, 32) KDA_MULTI_CASE(128, 64) KDA_MULTI_CASE(128, 128)
#undef KDA_MULTI_CASE
    return cudaErrorNotSupported;
}

}  // namespace

namespace kda_host {

cudaError_t launch_decode(const DecodeArgs& a) {
    if (a.dtype == KDA_BF16) return dispatch_dims<__nv_bfloat16>(a);
    return dispatch_dims<float>(a);
}

int decode_multi_max_tokens() { return kMaxVerify; }

cudaError_t launch_decode_multi(const DecodeArgs& a, int K, const int32_t* commit_len) {
    if (a.dtype == KDA_BF16) return dispatch_multi<__nv_bfloat16>(a, K, commit_len);
    return dispatch_multi<float>(a, K, commit_len);
}

}  // namespace kda_host
