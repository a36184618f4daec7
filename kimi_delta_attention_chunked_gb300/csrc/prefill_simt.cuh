// prefill_simt.cuh -- chunked KDA prefill on CUDA cores, fp32 throughout.
//
// This is the path for fp32 inputs (whose 1e-4 accuracy target bf16 or TF32
// tensor-core operands cannot meet) and for the shapes the tensor-core path is
// not built for.  It evaluates the same chunked form as the tensor-core path
// ("Kimi K3: the manos, the mythos, the legendos", section "FlashKDA
// Algorithm") with one CTA per (sequence, head, 32-column slice of d_v):
//
//   per chunk of n <= C tokens, with G the inclusive cumulative log-decay:
//     M_qk[r,t] = sum_i q_r,i k_t,i exp(G_r,i - G_t,i)           (t <= r)
//     L[r,t]    = beta_r sum_i k_r,i k_t,i exp(G_r,i - G_t,i)    (t <  r)
//     INV       = (I + L)^-1                  (forward substitution)
//     W         = INV Diag(beta) K_decay,  U0 = INV Diag(beta) V
//     U         = U0 - W S_in
//     O         = Q_decay S_in + M_qk U
//     S_out     = Diag(a_last) S_in + K_restore^T U
//
// The Gram entries are formed pair by pair with exp(G_r - G_t) <= 1, so no
// factor ever overflows (the factorised K_inv = K / a of the page would
// overflow fp32 for chunks longer than 16 under the (-5, 0) gate bound).
// Rows past the end of a sequence are zero (k = v = q = 0, beta = 0,
// log-decay 0), which leaves every result of the valid rows unchanged.
#include "common.cuh"

// Compiled once per (input dtype, chunk) by the prefill_simt_*.cu files, which
// define KDA_SIMT_BF16 (0/1) and KDA_SIMT_CHUNK, so the instantiations build in
// parallel.
#if !defined(KDA_SIMT_BF16) || !defined(KDA_SIMT_CHUNK)
#error "define KDA_SIMT_BF16 and KDA_SIMT_CHUNK"
#endif

namespace {

constexpr int kThreads = 256;

template <int DK, int DVT, int C>
struct SimtSmem {
    float q[C][DK];       // q, later Q_decay
    float k[C][DK];       // k, later K_restore
    float g[C][DK];       // log-decay, then G, later beta*K_decay, then W
    float v[C][DVT];      // v, then U0, then U
    float m[C][C];        // M_qk
    float l[C][C];        // L
    float inv[C][C];      // (I + L)^-1
    float s[DK][DVT];     // state slice
    float beta[C];
    float a_last[DK];
    float g_last[DK];
};

template <int DK, int DV, int C, typename TIn>
__global__ void __launch_bounds__(kThreads)
kda_prefill_simt_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                        const TIn* __restrict__ v, const float* __restrict__ log_alpha,
                        const float* __restrict__ beta, const float* __restrict__ S0,
                        const int32_t* __restrict__ cu_seqlens, int T_total, int H,
                        int seq_len_fixed, TIn* __restrict__ O, float* __restrict__ S_final,
                        int ckpt_every, float* __restrict__ ckpt, int ckpt_cap, int prologue) {
    constexpr int DVT = DV < 32 ? DV : 32;
    using Sm = SimtSmem<DK, DVT, C>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);

    constexpr int NTILE = DV / DVT;
    const int tile = blockIdx.x % NTILE;         // d_v slice
    const int n = blockIdx.x / NTILE;            // sequence
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int j0 = tile * DVT;

    int bos, eos;
    if (cu_seqlens) {
        bos = cu_seqlens[n];
        eos = cu_seqlens[n + 1];
        bos = min(max(bos, 0), T_total);
        eos = min(max(eos, bos), T_total);
    } else {
        bos = n * seq_len_fixed;
        eos = bos + seq_len_fixed;
    }

    // state checkpoints: index of this sequence's first one (block-wide sum)
    int ck_base = 0;
    if (ckpt_every > 0) {
        ck_base = cu_seqlens ? kda::ckpt_base(n, ckpt_every,
                                              [&](int m) {
                                                  const int b0 = min(max(cu_seqlens[m], 0), T_total);
                                                  return min(max(cu_seqlens[m + 1], b0), T_total) - b0;
                                              })
                             : n * (seq_len_fixed / ckpt_every);
    }
    auto put_ckpt = [&](int idx) {             // every thread stores its elements of the slice
        if (idx < 0 || idx >= ckpt_cap) return;
        for (int e = tid; e < DK * DVT; e += kThreads) {
            const int i = e / DVT, j = e % DVT;
            ckpt[(((size_t)idx * H + h) * DK + i) * DV + j0 + j] = sm.s[i][j];
        }
    };
    // initial state slice
    for (int e = tid; e < DK * DVT; e += kThreads) {
        const int i = e / DVT, j = e % DVT;
        sm.s[i][j] = S0 ? S0[(((size_t)n * H + h) * DK + i) * DV + j0 + j] : 0.f;
    }

    for (int c0 = bos; c0 < eos; c0 += C) {
        const int nr = min(C, eos - c0);         // valid rows of this chunk
        __syncthreads();                         // previous chunk fully consumed
        if (ckpt_every > 0 && c0 > bos && (c0 - bos) % ckpt_every == 0) put_ckpt(ck_base + (c0 - bos) / ckpt_every - 1);
        // ---- load q, k, log-decay, the v slice and beta (rows >= nr zero)
        for (int e = tid; e < C * DK; e += kThreads) {
            const int r = e / DK, i = e % DK;
            const bool ok = r < nr;
            const size_t off = ((size_t)(c0 + r) * H + h) * DK + i;
            sm.q[r][i] = ok ? kda::io<TIn>::ld(q + off) : 0.f;
            sm.k[r][i] = ok ? kda::io<TIn>::ld(k + off) : 0.f;
            sm.g[r][i] = ok ? (prologue ? kda::prologue_log_alpha(log_alpha[off]) : log_alpha[off]) : 0.f;
        }
        for (int e = tid; e < C * DVT; e += kThreads) {
            const int r = e / DVT, j = e % DVT;
            sm.v[r][j] = r < nr ? kda::io<TIn>::ld(v + ((size_t)(c0 + r) * H + h) * DV + j0 + j) : 0.f;
        }
        for (int r = tid; r < C; r += kThreads) {
            const float bl = r < nr ? beta[(size_t)(c0 + r) * H + h] : 0.f;
            sm.beta[r] = r < nr ? (prologue ? kda::prologue_beta(bl) : bl) : 0.f;
        }
        __syncthreads();
        if (prologue) {                          // fused prologue: unit-length q and k rows
            for (int e = tid >> 5; e < 2 * C; e += kThreads / 32) {   // one warp per row
                float* x = e < C ? sm.q[e] : sm.k[e - C];
                float ss = 0.f;
                for (int i = tid & 31; i < DK; i += 32) ss = fmaf(x[i], x[i], ss);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float sc = rsqrtf(ss + kda::kNormEps);
                for (int i = tid & 31; i < DK; i += 32) x[i] *= sc;
            }
            __syncthreads();
        }

        // ---- inclusive cumulative log-decay per key channel
        for (int i = tid; i < DK; i += kThreads) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) { acc += sm.g[r][i]; sm.g[r][i] = acc; }
            sm.g_last[i] = acc;
            sm.a_last[i] = __expf(acc);
        }
        __syncthreads();

        // ---- intra-chunk Gram matrices, pair by pair
        for (int e = tid; e < C * C; e += kThreads) {
            const int r = e / C, t = e % C;
            float mq = 0.f, lk = 0.f;
            if (t <= r) {
                for (int i = 0; i < DK; ++i) {
                    const float d = __expf(sm.g[r][i] - sm.g[t][i]) * sm.k[t][i];
                    mq = fmaf(sm.q[r][i], d, mq);
                    lk = fmaf(sm.k[r][i], d, lk);
                }
            }
            sm.m[r][t] = mq;
            sm.l[r][t] = t < r ? sm.beta[r] * lk : 0.f;
        }
        __syncthreads();

        // ---- INV = (I + L)^-1, one column per thread, by forward substitution
        if (tid < C) {
            const int jc = tid;
            for (int r = 0; r < C; ++r) {
                float acc = (r == jc) ? 1.f : 0.f;
                for (int t = jc; t < r; ++t) acc = fmaf(-sm.l[r][t], sm.inv[t][jc], acc);
                sm.inv[r][jc] = (r < jc) ? 0.f : acc;
            }
        }
        // ---- Q_decay and K_restore in place; beta * K_decay into g
        for (int e = tid; e < C * DK; e += kThreads) {
            const int r = e / DK, i = e % DK;
            const float G = sm.g[r][i];
            sm.q[r][i] *= __expf(G);
            const float kk = sm.k[r][i];
            sm.k[r][i] = kk * __expf(sm.g_last[i] - G);
            sm.g[r][i] = sm.beta[r] * kk * __expf(G);
        }
        __syncthreads();

        // ---- W = INV (beta K_decay), U0 = INV (beta V)
        constexpr int WPT = (C * DK + kThreads - 1) / kThreads;
        constexpr int UPT = (C * DVT + kThreads - 1) / kThreads;
        float w_reg[WPT], u_reg[UPT];
#pragma unroll
        for (int p = 0; p < WPT; ++p) {
            const int e = tid + p * kThreads;
            float acc = 0.f;
            if (e < C * DK) {
                const int r = e / DK, i = e % DK;
                for (int t = 0; t <= r; ++t) acc = fmaf(sm.inv[r][t], sm.g[t][i], acc);
            }
            w_reg[p] = acc;
        }
#pragma unroll
        for (int p = 0; p < UPT; ++p) {
            const int e = tid + p * kThreads;
            float acc = 0.f;
            if (e < C * DVT) {
                const int r = e / DVT, j = e % DVT;
                for (int t = 0; t <= r; ++t) acc = fmaf(sm.inv[r][t] * sm.beta[t], sm.v[t][j], acc);
            }
            u_reg[p] = acc;
        }
        __syncthreads();
#pragma unroll
        for (int p = 0; p < WPT; ++p) {
            const int e = tid + p * kThreads;
            if (e < C * DK) sm.g[e / DK][e % DK] = w_reg[p];
        }
        __syncthreads();

        // ---- U = U0 - W S_in ; P_q = Q_decay S_in
        float pq[UPT];
#pragma unroll
        for (int p = 0; p < UPT; ++p) {
            const int e = tid + p * kThreads;
            pq[p] = 0.f;
            if (e < C * DVT) {
                const int r = e / DVT, j = e % DVT;
                float pw = 0.f, acc_q = 0.f;
                for (int i = 0; i < DK; ++i) {
                    pw = fmaf(sm.g[r][i], sm.s[i][j], pw);
                    acc_q = fmaf(sm.q[r][i], sm.s[i][j], acc_q);
                }
                u_reg[p] -= pw;
                pq[p] = acc_q;
            }
        }
        __syncthreads();
#pragma unroll
        for (int p = 0; p < UPT; ++p) {
            const int e = tid + p * kThreads;
            if (e < C * DVT) sm.v[e / DVT][e % DVT] = u_reg[p];
        }
        __syncthreads();

        // ---- O = P_q + M_qk U  (valid rows only)
#pragma unroll
        for (int p = 0; p < UPT; ++p) {
            const int e = tid + p * kThreads;
            if (e < C * DVT) {
                const int r = e / DVT, j = e % DVT;
                float acc = pq[p];
                for (int t = 0; t <= r; ++t) acc = fmaf(sm.m[r][t], sm.v[t][j], acc);
                if (r < nr) kda::io<TIn>::st(O + ((size_t)(c0 + r) * H + h) * DV + j0 + j, acc);
            }
        }
        // ---- S_out = Diag(a_last) S_in + K_restore^T U  (each thread owns its elements)
        for (int e = tid; e < DK * DVT; e += kThreads) {
            const int i = e / DVT, j = e % DVT;
            float acc = sm.a_last[i] * sm.s[i][j];
            for (int t = 0; t < C; ++t) acc = fmaf(sm.k[t][i], sm.v[t][j], acc);
            sm.s[i][j] = acc;
        }
    }
    __syncthreads();
    if (ckpt_every > 0 && eos > bos && (eos - bos) % ckpt_every == 0) put_ckpt(ck_base + (eos - bos) / ckpt_every - 1);
    if (S_final) {
        for (int e = tid; e < DK * DVT; e += kThreads) {
            const int i = e / DVT, j = e % DVT;
            S_final[(((size_t)n * H + h) * DK + i) * DV + j0 + j] = sm.s[i][j];
        }
    }
}

template <int DK, int DV, int C, typename TIn>
cudaError_t launch(const kda_host::PrefillArgs& a) {
    constexpr int DVT = DV < 32 ? DV : 32;
    const size_t smem = sizeof(SimtSmem<DK, DVT, C>);
    auto kern = kda_prefill_simt_kernel<DK, DV, C, TIn>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((DV / DVT) * a.n_seq, a.H);
    if (a.n_seq == 0) return cudaSuccess;
    const int fixed = a.cu_seqlens ? 0 : a.T_total / a.n_seq;
    kern<<<grid, kThreads, smem, a.stream>>>(
        static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v),
        a.log_alpha, a.beta, a.S0, a.cu_seqlens, a.T_total, a.H, fixed,
        static_cast<TIn*>(a.O), a.S_final, a.ckpt_every, a.ckpt, a.ckpt_cap, a.prologue);
    const cudaError_t err = cudaGetLastError();
    kda_host::trace_mark(a.stream);
    return err;
}

template <typename TIn, int C>
cudaError_t dispatch_dims(const kda_host::PrefillArgs& a) {
#define KDA_SIMT_CASE(DK_, DV_) \
    if (a.dk == DK_ && a.dv == DV_) return launch<DK_, DV_, C, TIn>(a);
    KDA_SIMT_CASE(32, 32) KDA_SIMT_CASE(32, 64) KDA_SIMT_CASE(32, 128)
    KDA_SIMT_CASE(64, 32) KDA_SIMT_CASE(64, 64) KDA_SIMT_CASE(64, 128)
    KDA_SIMT_CASE(128, 32) KDA_SIMT_CASE(128, 64) KDA_SIMT_CASE(128, 128)
#undef KDA_SIMT_CASE
    return cudaErrorNotSupported;
}

#define KDA_SIMT_NAME2(dt, c) launch_prefill_simt_##dt##_c##c
#define KDA_SIMT_NAME(dt, c) KDA_SIMT_NAME2(dt, c)

}  // namespace

namespace kda_host {

#if KDA_SIMT_BF16
cudaError_t KDA_SIMT_NAME(bf16, KDA_SIMT_CHUNK)(const PrefillArgs& a) {
    return dispatch_dims<__nv_bfloat16, KDA_SIMT_CHUNK>(a);
}
#else
cudaError_t KDA_SIMT_NAME(fp32, KDA_SIMT_CHUNK)(const PrefillArgs& a) {
    return dispatch_dims<float, KDA_SIMT_CHUNK>(a);
}
#endif

}  // namespace kda_host
