// prefill_tc.cu -- chunked KDA prefill on tcgen05 tensor cores (bf16 inputs,
// d_k = d_v = 128, chunk C = 64, fp32 state).
//
// The chunked form is the one of "Kimi K3: the manos, the mythos, the
// legendos", section "FlashKDA Algorithm":
//     B = Diag(beta)(V - K_decay S_in),  L = StrictTril(Diag(beta) K_decay K_inv^T)
//     U = (I + L)^-1 B,  M_qk = tril(Q_decay K_inv^T)
//     O = Q_decay S_in + M_qk U,  S_out = Diag(a_last) S_in + K_restore^T U
// with a = exp(cumsum(log_alpha)) the inclusive cumulative decay of the chunk.
// Everything that does not depend on S_in is computed for all chunks in
// parallel; only the state pass is sequential.  Two kernels:
//
//  kda_tc_prep   persistent, two CTAs per SM, one (chunk, head) item at a time.
//      a1  gate prep: fp32 cumulative log-decay, then the MMA operands.
//          K_inv = k / a would overflow (|cumsum| reaches 5 * 64 = 320 under
//          the (-5, 0) log-decay bound of the "LLM architecture at trillion
//          scale" page), so the Gram matrices are built per 16-row block b with
//          a reference point p_b = first row of the block:
//             row factor  q_r exp(G_r - G_pb), k_r exp(G_r - G_pb)   (<= 1)
//             col factor  k_t exp(G_pb - G_t)  for t < p_b + 16      (<= e^75)
//          so every exponent stays inside [-75, 75] (fp32/bf16 range) and the
//          product equals the exact exp(G_r - G_t) weight.  Where no block
//          decays by more than e^10 the Gram operands are f16 instead of bf16.
//      a2  Gram MMAs (tcgen05, M = 128 stacked q/k rows; the four blocks'
//          column operands stacked along N = 160): M_qk (diagonal included)
//          and L (strict, beta folded in).
//      a3  INV = (I + L)^-1 in fp32 (16x16 diagonal blocks by substitution,
//          then the off-diagonal blocks from products of L blocks with those
//          inverses, warp by warp) and X = M_qk INV; then one MMA with
//          M = 128 stacked rows
//             [INV Diag(beta); X Diag(beta)] [K_decay | V]
//          gives W = INV Diag(beta) K_decay, U0 = INV Diag(beta) V and, in the
//          same instruction, M_qk W and O0 = M_qk U0.  Since U = U0 - W S_in,
//             O = Q_decay S_in + M_qk U = Q' S_in + O0,  Q' = Q_decay - M_qk W,
//          so the state pass needs no product for M_qk U.
//      Writes, per (chunk, head), the MMA-ready operand images the chain
//      needs: [Q'; W], K_restore^T, U0, O0, a_last.
//
//  kda_tc_chain  one CTA per (sequence, head, 64- or 32-column slice of d_v);
//      a4/a5  for each chunk in order (operands streamed by bulk copies into
//          two rings of two stages, U0 / O0 tiles one chunk at a time), with
//          S kept in TMEM in fp32:
//             P  = [Q'; W] S_in                         (MMA, M = 128)
//             U  = U0 - P_w                             (W S_in = K_decay part)
//             O  = P_q + O0
//             S  = Diag(a_last) S_in + K_restore^T U    (MMA, accumulate)
//
// With few chains and long sequences the state pass runs as a segment scan
// instead (kda_tc_segments, two passes of kda_tc_chain around kda_tc_seg_scan;
// see the section "segment scan" below); with many chains and long sequences
// the prep of later chunk slices runs beside the state pass (launch_prefill_tc).
//
// Precision: MMA operands are bf16 (or f16) with fp32 accumulation.  The
// operands whose rounding mattered -- X, [INV; X] Diag(beta), and in the
// state pass S_in, U and K_restore -- are carried as a high and a low bf16
// part, and U0 and O0 stay fp32, which leaves the bf16 output rounding as the
// largest single error term.
//
// Every wait on an asynchronous event is bounded; a wait that runs out records
// KDA_ERR_TIMEOUT in the status word and sets the CTA's abort flag: the CTA
// issues no further copy or MMA, waits (bounded) for what is in flight, and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "umma.cuh"

namespace {

using bf16 = __nv_bfloat16;

constexpr int DK = 128, DV = 128, C = 64;
constexpr int NT = 64;                       // d_v columns of a workspace U0 / O0 tile (ChainCfg: of a CTA)
constexpr int NTILES = DV / NT;

// ---- per (chunk, head) workspace block: images of shared-memory operands
constexpr uint32_t WS_A1 = 0;                // [Q'; W]       K-major SW128, 128 rows, K = 128 (2 panels)
constexpr uint32_t WS_KR = 32768;            // K_restore^T high part, MN-major SW128, K = 64 rows, M = 128 (2 panels)
constexpr uint32_t WS_KRL = 49152;           //   ... low part, same layout, right after it
constexpr uint32_t TILE_F32 = C * NT * 4;    // one d_v slice of U0 or O0, fp32, in the order the chain loads it
constexpr uint32_t WS_UO = 65536;            // per d_v slice t: U0 at WS_UO + 2 t TILE_F32, O0 right after it
constexpr uint32_t WS_AL = WS_UO + NTILES * 2 * TILE_F32;   // a_last fp32 [DK]
constexpr uint32_t WS_BLOCK = 132096;        // 129 KiB
// Byte offset of element (r, c) (row r < 64, column c < 64 of one d_v slice)
// in a U0 / O0 tile: the 16 columns [16 g, 16 g + 16) of a row are the four
// 16-byte pieces one state-pass thread loads, piece j of all 64 rows stored
// together, so that the 32 lanes of a warp load 512 contiguous bytes.
__host__ __device__ constexpr uint32_t uo_off(uint32_t r, uint32_t c) {
    return ((((c >> 4) * 4u + ((c >> 2) & 3u)) * 64u + r) * 4u + (c & 3u)) * 4u;
}

// ---- prep kernel shared memory
constexpr uint32_t K1_BG = 0;                // Gram B: tiles b = 0..3 (16(b+1) rows each) stacked along N
                                             // at row 8b(b+1): one 160-row K-major tile, K = 128
constexpr uint32_t K1_AG = 40960;            // Gram A: 128 rows [q~ b0 | k^ b0 | q~ b1 | ...], K = 128
constexpr uint32_t K1_BWU = 73728;           // [K_decay | V]: MN-major, K = 64 rows, N = 256 (4 panels)
constexpr uint32_t K1_TOT = 106496;          // float [4][128] block totals of log-decay
constexpr uint32_t K1_FIRST = 108544;        // float [4][128] first-row log-decay of each block
constexpr uint32_t K1_BETA = 110592;         // float [64]
constexpr uint32_t K1_BAR = 110848;          // MMA mbarrier (8 B), TMEM address (4 B), Q_decay copy mbarrier at +16,
                                             // log-decay and V copy mbarrier at +24, abort flag (4 B) at +32,
                                             // drain mbarrier at +40, q and k copy mbarrier at +48
constexpr uint32_t K1_NRM = 110912;          // fused prologue: float [q, k][channel half][64 rows] sums of squares
constexpr uint32_t K1_BYTES = 111936;
// aliases, valid once the Gram MMAs have completed
constexpr int LDS_ = 68;                     // row stride (floats) of the fp32 64x64 matrices
constexpr uint32_t K1_LS = 0;                // L   fp32 [64][68]
constexpr uint32_t K1_IS = 17408;            // INV fp32 [64][68]
constexpr uint32_t K1_XS = 34816;            // 4 x 16x16 fp32 scratch blocks (dense), slots 0-3
constexpr uint32_t K1_XS2 = 55296;           // 4 more (slots 4-7), in the dead Gram A operand (the
                                             //   [INV; X] low part lands there after the inverse)
constexpr uint32_t K1_MH = 38912;            // M_qk high / low bf16 parts, K-major SW128, 64 rows, K = 64
constexpr uint32_t K1_ML = 47104;            //   (the M = 128 product reads 64 rows past each: still in the tile)
constexpr uint32_t K1_IH = 0;                // INV high / low bf16 parts, MN-major SW128, K = 64 rows, N = 64
constexpr uint32_t K1_IL = 8192;             //   (over L, once the inverse no longer needs it)
constexpr uint32_t K1_AI = 38912;            // [INV; X] Diag(beta), high bf16 part, K-major SW128, 128 rows, K = 64
constexpr uint32_t K1_AIL = 55296;           // ... low bf16 part (both written once the X product is done)
constexpr uint32_t K1_TMEM_COLS = 256;
constexpr uint32_t K1_TX = 160;              // TMEM columns of X = M_qk INV (lanes 0..63)
// input tiles of an item, copied by TMA over the Gram operands' space.  The
// log-decay tile (under the Gram A operand, read into registers before that is
// written) and V (straight into its operand slot) of the next item are copied
// while this item's epilogue runs; q and k (under the Gram B operand, which is
// written after every thread has read its rows) once this item's [Q'; W] image
// has been read out, behind the cumulative sum of the next item.
constexpr uint32_t K1_SG = 40960;            // log-decay fp32 [64 tokens][128]
constexpr uint32_t K1_SQ = 0;                // q bf16 [64][128]
constexpr uint32_t K1_SK = 16384;            // k bf16 [64][128]
constexpr uint32_t K1_GV_BYTES = 32768 + 16384;   // log-decay and V
constexpr uint32_t K1_QK_BYTES = 2 * 16384;       // q and k
// output image, assembled once the last MMA has completed and written to the
// workspace by one bulk copy (U0 and O0 go from registers straight to the workspace)
constexpr uint32_t K1_OUT_A1 = 0;            // [Q'; W] image (rows 0..63 arrive as Q_decay from the workspace)

// ---- chain kernel shared memory
constexpr int K2_NA = 2;                     // [Q'; W] stages (released as soon as the P product is done)
constexpr int K2_NB = 2;                     // K_restore^T stages, high and low part (released after the state update)
constexpr uint32_t K2_ASTAGE = 32768;
constexpr uint32_t K2_BSTAGE = 32768;
constexpr uint32_t K2_B0 = K2_NA * K2_ASTAGE;            // B ring: high part at +0, low part at +16384
// The rest depends on NTC, the d_v columns of one state-pass CTA (64, or 32
// when the whole pass fits one wave of CTAs):
template <int NTC>
struct ChainCfg {
    static constexpr int NTL = DV / NTC;                   // CTAs (slices) per (sequence, head)
    static constexpr int CW = NTC / 4;                     // state columns per conversion thread
    static constexpr uint32_t TILE = C * NTC * 4;          // one slice's U0 or O0 tile, fp32
    static constexpr uint32_t SB = K2_B0 + K2_NB * K2_BSTAGE;   // [S_hi | S_lo] bf16, MN-major SW128, K = 128 rows, N = 2 NTC
    static constexpr uint32_t UB = SB + 128 * 4 * NTC;     // [U_hi | U_lo] bf16, MN-major SW128, K = 64 rows, N = 2 NTC
    static constexpr uint32_t OS = UB + 64 * 4 * NTC;      // one chunk's bf16 output rows [64][NTC], 16-byte pieces swizzled
    static constexpr uint32_t U0 = OS + 64 * 2 * NTC;      // U0 tile of this slice (workspace order), one chunk
    static constexpr uint32_t O0 = U0 + TILE;              // O0 tile of this slice, one chunk
    static constexpr uint32_t BAR = O0 + TILE;             // full / empty A, B; p; s; drain; full / empty U0, O0;
                                                           // TMEM address; abort flag
    static constexpr uint32_t BYTES = BAR + 192;
    // TMEM: S [0, NTC), X [NTC, 2 NTC), P of even chunks [2 NTC, 4 NTC), of odd [4 NTC, 6 NTC)
    static constexpr uint32_t TMEM_COLS = NTC == 64 ? 512 : 256;
    static_assert(NTC == 64 || NTC == 32, "state-pass slice width");
    static_assert(SB % 1024 == 0 && UB % 1024 == 0 && OS % 1024 == 0, "SW128 operands / swizzled output tile");
    static_assert(BYTES + 1024 + 256 <= 232448, "chain smem");
    static_assert(BAR + 15 * 8 + 8 <= BYTES, "chain barriers and flags");
};
static_assert(K2_B0 % 1024 == 0, "SW128 operands are 1024-byte aligned");
static_assert(WS_KRL == WS_KR + 16384, "both parts of K_restore^T are one contiguous copy");
static_assert(K1_AIL + 16384 <= K1_BWU, "[INV; X] must stay inside the alias region");
static_assert(K1_ML + 16384 <= K1_BWU && K1_IL + 8192 <= K1_IS, "X operands stay inside the alias region");
static_assert(K1_OUT_A1 + 32768 <= K1_SG, "the next log-decay tile does not touch the [Q'; W] image");
static_assert(K1_BAR + 64 <= K1_NRM, "prep barriers and flags");
static_assert(K1_BG + 160 * 256 <= K1_AG && K1_AG + 32768 == K1_BWU && K1_AG % 1024 == 0, "Gram operands");
static_assert(K1_SK + 16384 <= K1_AG && K1_SG + 32768 <= K1_BWU && (K1_BWU + 16384) % 1024 == 0, "input tiles");
static_assert(K1_AIL + 16384 <= K1_SG + 32768 && K1_ML + 16384 <= K1_SG + 32768,
              "the next log-decay tile lands where only the last MMA's A operand was");
static_assert(K1_XS2 >= K1_ML + 8192 && K1_XS2 + 4096 <= K1_AG + 32768, "inverse scratch slots 4-7");
static_assert(K1_IS + 64 * LDS_ * 4 <= K1_XS && K1_XS + 4096 <= K1_MH && 16384 + 8192 <= K1_XS,
              "Q_decay rows land in the free L / INV region while the last MMA runs");
static_assert(WS_BLOCK % 1024 == 0 && WS_AL + DK * 4 <= WS_BLOCK, "workspace block");
static_assert(2 * (K1_BYTES + 1024 + 1024) <= 233472, "prep must fit two CTAs per SM");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// x = hi + lo with hi = x truncated to bf16 and lo = bf16(x - hi): the pair
// carries ~16 significant bits (|x - hi| < 2^-7 |x|, and lo is rounded to
// nearest), enough to keep an MMA operand's rounding out of the error budget.
// Eight values -> two packed bf16 x 8; hi needs no conversion instruction.
__device__ __forceinline__ void split_pack8(const float* x, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t a = __float_as_uint(x[2 * j]), b = __float_as_uint(x[2 * j + 1]);
        h[j] = __byte_perm(a, b, 0x7632);              // upper halves of a (low 16 bits) and b
        const __nv_bfloat162 lb = __floats2bfloat162_rn(x[2 * j] - __uint_as_float(a & 0xFFFF0000u),
                                                        x[2 * j + 1] - __uint_as_float(b & 0xFFFF0000u));
        l[j] = *reinterpret_cast<const uint32_t*>(&lb);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// One warp: acc (+)= A * B for 16x16 fp32 blocks in shared memory (row-major,
// leading dimensions lda / ldb), on the tensor cores with mma.sync m16n8k8
// TF32 and a three-product big/small split of every operand (x = big + small,
// big = tf32(x), small = tf32(x - big); big*big + big*small + small*big), which
// keeps the product at about fp32 accuracy.  The accumulator is the m16n8
// fragment of the two 8-column halves: acc[4 h + i] holds row
// (lane / 4) + 8 (i / 2), column 8 h + 2 (lane % 4) + (i % 2).
__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t& big, uint32_t& small) {
    big = tf32_rna(x);
    small = tf32_rna(x - __uint_as_float(big));
}
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mm16(float (&acc)[8], const float* A, int lda, const float* B, int ldb, int lane,
                                     bool accumulate) {
    const int g = lane >> 2, t = lane & 3;
    if (!accumulate) {
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    }
#pragma unroll 1
    for (int kk = 0; kk < 16; kk += 8) {      // rolled: this code is inlined at eight call sites
        uint32_t ab[4], as[4];
        split_tf32(A[g * lda + kk + t], ab[0], as[0]);
        split_tf32(A[(g + 8) * lda + kk + t], ab[1], as[1]);
        split_tf32(A[g * lda + kk + t + 4], ab[2], as[2]);
        split_tf32(A[(g + 8) * lda + kk + t + 4], ab[3], as[3]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t bb[2], bs[2];
            split_tf32(B[(kk + t) * ldb + 8 * h + g], bb[0], bs[0]);
            split_tf32(B[(kk + t + 4) * ldb + 8 * h + g], bb[1], bs[1]);
            mma_tf32(acc + 4 * h, as, bb);
            mma_tf32(acc + 4 * h, ab, bs);
            mma_tf32(acc + 4 * h, ab, bb);
        }
    }
}

// acc <- the 16x16 block C in the accumulator layout that st16 stores
__device__ __forceinline__ void ld16(float (&acc)[8], const float* C, int ldc, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float2 a = *reinterpret_cast<const float2*>(C + g * ldc + 8 * h + 2 * t);
        const float2 b = *reinterpret_cast<const float2*>(C + (g + 8) * ldc + 8 * h + 2 * t);
        acc[4 * h] = a.x; acc[4 * h + 1] = a.y; acc[4 * h + 2] = b.x; acc[4 * h + 3] = b.y;
    }
}

__device__ __forceinline__ void st16(float* D, int ldd, const float (&acc)[8], int lane, float scale) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        *reinterpret_cast<float2*>(D + g * ldd + 8 * h + 2 * t) =
            make_float2(scale * acc[4 * h], scale * acc[4 * h + 1]);
        *reinterpret_cast<float2*>(D + (g + 8) * ldd + 8 * h + 2 * t) =
            make_float2(scale * acc[4 * h + 2], scale * acc[4 * h + 3]);
    }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    return make_uint4(kda::pack_bf16x2(f[0], f[1]), kda::pack_bf16x2(f[2], f[3]),
                      kda::pack_bf16x2(f[4], f[5]), kda::pack_bf16x2(f[6], f[7]));
}

// Eight values as packed bf16, or as f16 (nearest even) when f16 != 0: three
// more mantissa bits for a Gram operand whose values the chunk's decay range
// keeps inside f16.  The type is a run-time choice: the bf16 conversions are
// overwritten by predicated f16 ones, so that one copy of the operand code
// serves both types without a branch (two copies, one per type, made the
// kernel's code a quarter larger and every phase slower).
__device__ __forceinline__ uint4 pack8g(const float* f, uint32_t f16) {
    uint4 r;
    asm("{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %12, 0;\n\t"
        "cvt.rn.bf16x2.f32 %0, %5, %4;\n\t"
        "cvt.rn.bf16x2.f32 %1, %7, %6;\n\t"
        "cvt.rn.bf16x2.f32 %2, %9, %8;\n\t"
        "cvt.rn.bf16x2.f32 %3, %11, %10;\n\t"
        "@p cvt.rn.f16x2.f32 %0, %5, %4;\n\t"
        "@p cvt.rn.f16x2.f32 %1, %7, %6;\n\t"
        "@p cvt.rn.f16x2.f32 %2, %9, %8;\n\t"
        "@p cvt.rn.f16x2.f32 %3, %11, %10;\n\t}"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]), "r"(f16));
    return r;
}
// Largest log-decay across one 16-row block (over every channel) for which
// the Gram operands go to the tensor cores as f16: the column factors are at
// most e^10 = 22026 (below f16's 65504; |k| <= 1 for unit-length keys, and
// the factor itself is what the bound limits), the row factors at least e^-10.
constexpr float kF16GramLog = 10.f;

// ============================================================== schedule
// cu_seqlens -> per-chunk (token start, rows, sequence) and per-sequence
// (bos, len, first chunk, chunks).  One block; lengths are clamped so that no
// later access leaves the arrays even for an inconsistent device cu_seqlens.
__global__ void __launch_bounds__(1024)
kda_tc_schedule(const int32_t* __restrict__ cu, int n_seq, int T_total, int slots,
                int4* __restrict__ chunk_info, int4* __restrict__ seq_info, int* __restrict__ seq_order,
                int* status) {
    __shared__ int part[1024];
    __shared__ int total;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (n_seq + nt - 1) / nt;
    const int s0 = min(tid * per, n_seq), s1 = min(s0 + per, n_seq);
    int cnt = 0;
    for (int n = s0; n < s1; ++n) {
        const int bos = min(max(cu[n], 0), T_total);
        const int eos = min(max(cu[n + 1], bos), T_total);
        cnt += (eos - bos + C - 1) / C;
    }
    part[tid] = cnt;
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int i = 0; i < nt; ++i) { const int c = part[i]; part[i] = acc; acc += c; }
        total = min(acc, slots);
        if (acc > slots) kda::record_status(status, KDA_ERR_INVALID_ARG);
    }
    __syncthreads();
    int first = part[tid];
    for (int n = s0; n < s1; ++n) {
        const int bos = min(max(cu[n], 0), T_total);
        const int eos = min(max(cu[n + 1], bos), T_total);
        int len = eos - bos;
        int nch = (len + C - 1) / C;
        if (first + nch > slots) { nch = max(0, slots - first); len = min(len, nch * C); }
        seq_info[n] = make_int4(bos, len, first, nch);
        for (int j = 0; j < nch; ++j) chunk_info[first + j] = make_int4(bos + j * C, min(C, len - j * C), n, 0);
        first += nch;
    }
    for (int s = total + tid; s < slots; s += nt) chunk_info[s] = make_int4(0, 0, -1, 0);
    // the sequences by chunk count, longest first (ties by index), for the
    // order of the state pass's CTAs (few sequences only: one rank a thread)
    if (seq_order != nullptr && n_seq <= nt) {
        __syncthreads();                          // seq_info of every sequence is written
        if (tid < n_seq) {
            const int mine = seq_info[tid].w;
            int rank = 0;
            for (int m = 0; m < n_seq; ++m) {
                const int other = seq_info[m].w;
                rank += (other > mine || (other == mine && m < tid)) ? 1 : 0;
            }
            seq_order[rank] = tid;
        }
    }
}

// ============================================================== prep (a1-a3)
// Two warps per row block B (0..3), one per 32-column half: TMEM lanes
// 32 B .. 32 B + 31 hold the block's q~ rows (lanes 0..15) and k^ rows (lanes
// 16..31) against the first 16 (B + 1) tokens, at columns 8 B (B + 1) ...
// Writes the M_qk rows (diagonal included) as high / low bf16 operand parts and
// the L rows (beta folded in, strict) as fp32, both zero past the row's last
// kept column.  One rolled copy for all four blocks.
__device__ __forceinline__ void gram_epilogue(uint32_t tmem, int B, int half, int lane, uint8_t* mh, uint8_t* ml,
                                              float* LS) {
    const int N = 16 * (B + 1), OFF = 8 * B * (B + 1);
    const bool is_m = lane < 16;
    const int r = 16 * B + (lane & 15);
    const int lim = is_m ? r + 1 : r;             // columns t < lim are kept (lim <= N)
#pragma unroll 1
    for (int c = 32 * half; c < 32 * half + 32; c += 16) {
        float v[16];
        if (c < N) {                              // warp-uniform
            kda::tmem_ld16(tmem + ((uint32_t)(32 * B) << 16) + OFF + c, v);
            kda::tmem_wait_ld();
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = (c + u < lim) ? v[u] : 0.f;
        if (is_m) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint4 hi, lo;
                split_pack8(v + 8 * j, hi, lo);
                *reinterpret_cast<uint4*>(mh + kda::sw128(r, c + 8 * j, 64)) = hi;
                *reinterpret_cast<uint4*>(ml + kda::sw128(r, c + 8 * j, 64)) = lo;
            }
        } else {
            float* row = LS + r * LDS_ + c;
#pragma unroll
            for (int u = 0; u < 16; u += 4) *reinterpret_cast<float4*>(row + u) = make_float4(v[u], v[u + 1], v[u + 2], v[u + 3]);
        }
    }
}

template <bool PROLOGUE>
__global__ void __launch_bounds__(256, 2)
kda_tc_prep(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
            const float* __restrict__ beta, int H, int use_table,
            int fixed_len, int nch_per_seq, const int4* __restrict__ chunk_info,
            const int4* __restrict__ seq_info, int j_begin, int j_count, int n_x, int n_slots,
            uint8_t* __restrict__ ws_blocks, int* status, unsigned long long* item_ctr, int reserve_sm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    // Persistent over the n_x * H (chunk, head) items, head fastest.  The launch
    // covers chunks j_begin .. j_begin + j_count - 1 of every sequence: equal
    // lengths -> n_x = n_seq * j_count; chunk table -> n_x = chunk slots.
    // Static schedule (item_ctr null): this CTA takes items blockIdx.x,
    // blockIdx.x + gridDim.x, ...  Dynamic schedule: the CTAs draw items from
    // the counter *item_ctr (zero at launch), and a CTA that finds itself on an
    // SM whose id is below reserve_sm leaves at once, so that a state pass
    // launched beside this kernel finds those SMs free.
    if (item_ctr != nullptr && reserve_sm > 0) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        if ((int)smid < reserve_sm) return;        // nothing allocated or initialised yet
    }
    auto item = [&](long long it, int& tok0, int& nrows, int& slot, int& h) -> bool {
        const int x = (int)(it / H);
        h = (int)(it % H);
        if (!use_table) {
            const int n = x / j_count, j = j_begin + x % j_count;
            if (j >= nch_per_seq) return false;
            slot = n * nch_per_seq + j;
            tok0 = n * fixed_len + j * C;
            nrows = min(C, fixed_len - j * C);
        } else {
            slot = x;
            const int4 ci = chunk_info[slot];
            if (ci.z < 0) return false;
            const int j = slot - seq_info[ci.z].z;
            if (j < j_begin || j >= j_begin + j_count) return false;
            tok0 = ci.x;
            nrows = ci.y;
        }
        if (!KDA_DCHECK(status, slot >= 0 && slot < n_slots)) return false;    // workspace block of the item
        return nrows > 0;
    };
    const long long n_items = (long long)n_x * H;
    // dynamic schedule (thread 0): the next item that exists, or n_items
    auto draw = [&]() -> long long {
        for (;;) {
            const long long x = (long long)atomicAdd(item_ctr, 1ull);
            if (x >= n_items) return n_items;
            int t_, r_, s_, h_;
            if (item(x, t_, r_, s_, h_)) return x;
        }
    };

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + K1_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + K1_BAR + 8);
    uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + K1_BAR + 16);
    uint64_t* bar_gv = reinterpret_cast<uint64_t*>(sm + K1_BAR + 24);
    volatile int* abort_f = reinterpret_cast<volatile int*>(sm + K1_BAR + 32);
    uint64_t* bar_drain = reinterpret_cast<uint64_t*>(sm + K1_BAR + 40);
    uint64_t* bar_qk = reinterpret_cast<uint64_t*>(sm + K1_BAR + 48);
    volatile long long* next_it = reinterpret_cast<volatile long long*>(sm + K1_BAR + 56);   // dynamic schedule
    if (w == 0) {
        kda::tmem_alloc(tmem_slot, K1_TMEM_COLS);
        kda::tmem_relinquish();
    }
    if (tid == 0) {
        kda::mbar_init(bar, 1);
        kda::mbar_init(bar_q, 1);
        kda::mbar_init(bar_gv, 1);
        kda::mbar_init(bar_qk, 1);
        kda::mbar_init(bar_drain, 1);
        kda::fence_barrier_init();
        *abort_f = 0;
        if (item_ctr != nullptr) *next_it = draw();
    }
    uint32_t n_done = 0;                          // items finished by this CTA (bar_q parity)
    uint32_t bar_phase = 0;                       // completed phases of bar (three per item)
    uint32_t n_gv = 0, n_qk = 0, n_qloads = 0;    // copy phases issued (thread 0): log-decay and V, q and k, Q_decay
    // log-decay tile and V of item `it` into shared memory (thread 0)
    auto load_gv = [&](int t0, int hh) {
        kda::mbar_arrive_expect_tx(bar_gv, K1_GV_BYTES);
        kda::tma_load_3d(sm + K1_SG, &tm_g, 0, hh, t0, bar_gv);
        kda::tma_load_3d(sm + K1_BWU + 16384, &tm_v, 0, hh, t0, bar_gv);
        kda::tma_load_3d(sm + K1_BWU + 16384 + 8192, &tm_v, 64, hh, t0, bar_gv);
        ++n_gv;
    };
    bool gv_ready = false;                        // thread 0: this item's log-decay and V already issued
    // Bounded wait.  Once one runs out (or another thread's did) the CTA
    // issues no further copy or MMA: the remaining items run through without
    // waiting, and what is in flight is drained before the CTA exits.
    auto wait = [&](uint64_t* b, uint32_t parity) {
        if (!kda::mbar_wait_or_abort(b, parity, kda::kWaitCycles, abort_f)) {
            kda::record_status(status, kda::kDevTimeout);
            *abort_f = 1;
        }
    };
    kda::tc_fence_before();
    __syncthreads();
    kda::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const bool dyn = item_ctr != nullptr;
    for (long long it = dyn ? *next_it : blockIdx.x; it < n_items; it = dyn ? *next_it : it + gridDim.x) {
        int tok0, nrows, slot, h;
        if (!item(it, tok0, nrows, slot, h)) {
            if (dyn) break;                        // (drawn items exist: not reached)
            continue;
        }
        uint8_t* blk = ws_blocks + ((size_t)slot * H + h) * WS_BLOCK;

        // ---------------- a1: loads and per-block cumulative log-decay
        // Thread tile: rows r0 .. r0 + 3 of row block b (r0 = 16 b + 4 rq) and
        // the eight channels c0 .. c0 + 7 (c0 = 64 p + 8 cg), so that every load
        // and store of a row piece is one 16-byte vector; the four row quads of
        // a block are lanes 8 apart, and the cumulative sum crosses them by
        // shuffles.
        const int b = w >> 1, p = w & 1, cg = lane & 7, rq = lane >> 3;
        const int c0 = 64 * p + 8 * cg, r0 = 16 * b + 4 * rq;
        // inputs: one TMA copy per tensor, rows past the end of the tensor read
        // as zero.  The log-decay tile and V were copied during the previous
        // item's epilogue (the first item's are copied here); q and k once the
        // previous item's [Q'; W] image has left shared memory (they land where
        // it was staged): thread 0 waits for that after the first barrier, not
        // before it, unless the fused prologue needs q and k right away.
        auto issue_qk = [&]() {
            kda::bulk_wait_read_all();
            kda::mbar_arrive_expect_tx(bar_qk, K1_QK_BYTES);
            kda::tma_load_3d(sm + K1_SQ, &tm_q, 0, h, tok0, bar_qk);
            kda::tma_load_3d(sm + K1_SK, &tm_k, 0, h, tok0, bar_qk);
            ++n_qk;
        };
        if (tid == 0 && !*abort_f) {
            if (!gv_ready) load_gv(tok0, h);
            if (PROLOGUE) issue_qk();
        }
        gv_ready = false;
        float bt[4];                               // beta of this thread's rows (used after the cumulative sum)
#pragma unroll
        for (int i = 0; i < 4; ++i) bt[i] = beta[((size_t)tok0 + min(r0 + i, nrows - 1)) * H + h];
        wait(bar_gv, n_done & 1);
        float e[4][8];                             // log-decay, then its cumulative sum, then staged factors
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + i;
            const float4 g0 = *reinterpret_cast<const float4*>(sm + K1_SG + r * 512 + c0 * 4);
            const float4 g1 = *reinterpret_cast<const float4*>(sm + K1_SG + r * 512 + c0 * 4 + 16);
            e[i][0] = g0.x; e[i][1] = g0.y; e[i][2] = g0.z; e[i][3] = g0.w;
            e[i][4] = g1.x; e[i][5] = g1.y; e[i][6] = g1.z; e[i][7] = g1.w;
            // rows past the chunk's end (another sequence's tokens, or zeros): zero
            // inputs (log-decay 0, beta 0, and q = k = v = 0 below)
            if (r >= nrows) {
#pragma unroll
                for (int j = 0; j < 8; ++j) e[i][j] = 0.f;
            }
        }
        // this thread's q and k row pieces (zero past the chunk's end)
        auto load_qk = [&](int i, float* q, float* k) {
            const int r = r0 + i;
            uint4 qv = *reinterpret_cast<const uint4*>(sm + K1_SQ + r * 256 + c0 * 2);
            uint4 kv = *reinterpret_cast<const uint4*>(sm + K1_SK + r * 256 + c0 * 2);
            if (r >= nrows) { qv = make_uint4(0u, 0u, 0u, 0u); kv = qv; }
            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
            const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 qf = kda::unpack_bf16x2(qw[j]), kf = kda::unpack_bf16x2(kw[j]);
                q[2 * j] = qf.x; q[2 * j + 1] = qf.y; k[2 * j] = kf.x; k[2 * j + 1] = kf.y;
            }
        };
        for (int el = tid; el < (C - nrows) * (DV / 8); el += 256) {
            const int t = nrows + (el >> 4), cc = el & 15;
            *reinterpret_cast<uint4*>(sm + K1_BWU + 16384 + kda::sw128(t, 8 * cc, 64)) = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncthreads();                           // the log-decay tile is in registers
        if (!PROLOGUE && tid == 0 && !*abort_f) issue_qk();
        float* nrm = reinterpret_cast<float*>(sm + K1_NRM);
        if (PROLOGUE) {
            wait(bar_qk, n_done & 1);
            // fused prologue: gates from their pre-activations; squared norms of
            // the q and k rows over this panel's 64 channels
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float sq = 0.f, sk = 0.f;
                {
                    float q[8], k[8];
                    load_qk(i, q, k);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        sq = fmaf(q[j], q[j], sq);
                        sk = fmaf(k[j], k[j], sk);
                    }
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    sq += __shfl_xor_sync(0xffffffffu, sq, o);
                    sk += __shfl_xor_sync(0xffffffffu, sk, o);
                }
                if (cg == 0) {
                    nrm[p * 64 + r0 + i] = sq;
                    nrm[128 + p * 64 + r0 + i] = sk;
                }
                if (r0 + i < nrows) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) e[i][j] = kda::prologue_log_alpha(e[i][j]);
                }
            }
        }
        // inclusive cumulative sum within the 16-row block: over this thread's
        // four rows, then across the block's four row quads
#pragma unroll
        for (int i = 1; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 8; ++j) e[i][j] += e[i - 1][j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float t = e[3][j];
            float x = t;
            float y = __shfl_up_sync(0xffffffffu, x, 8);
            if (rq >= 1) x += y;
            y = __shfl_up_sync(0xffffffffu, x, 16);
            if (rq >= 2) x += y;
            const float excl = x - t;
#pragma unroll
            for (int i = 0; i < 4; ++i) e[i][j] += excl;
        }
        float* tot = reinterpret_cast<float*>(sm + K1_TOT);
        float* first = reinterpret_cast<float*>(sm + K1_FIRST);
        float* beta_s = reinterpret_cast<float*>(sm + K1_BETA);
        if (rq == 3) {
            *reinterpret_cast<float4*>(tot + b * 128 + c0) = make_float4(e[3][0], e[3][1], e[3][2], e[3][3]);
            *reinterpret_cast<float4*>(tot + b * 128 + c0 + 4) = make_float4(e[3][4], e[3][5], e[3][6], e[3][7]);
        }
        if (rq == 0) {
            *reinterpret_cast<float4*>(first + b * 128 + c0) = make_float4(e[0][0], e[0][1], e[0][2], e[0][3]);
            *reinterpret_cast<float4*>(first + b * 128 + c0 + 4) = make_float4(e[0][4], e[0][5], e[0][6], e[0][7]);
        }
        // beta: zero past the chunk's end (the loads were issued at the item's start)
#pragma unroll
        for (int i = 0; i < 4; ++i) bt[i] = r0 + i >= nrows ? 0.f : (PROLOGUE ? kda::prologue_beta(bt[i]) : bt[i]);
        if (p == 0 && cg == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) beta_s[r0 + i] = bt[i];
        }
        __syncthreads();

        // chunk-wide cumulative log-decay at this block's first row (myG) and at
        // the chunk's end (acc), per channel
        float myG[8], acc[8], fb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) { acc[j] = 0.f; myG[j] = 0.f; fb[j] = 0.f; }
        // the largest decay across a block, G(block start) - G(block end) =
        // first - tot, decides the Gram operands' type for the whole item
        bool wide = false;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 f0 = *reinterpret_cast<const float4*>(first + m * 128 + c0);
            const float4 f1 = *reinterpret_cast<const float4*>(first + m * 128 + c0 + 4);
            const float4 t0 = *reinterpret_cast<const float4*>(tot + m * 128 + c0);
            const float4 t1 = *reinterpret_cast<const float4*>(tot + m * 128 + c0 + 4);
            const float fm[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
            const float tm[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (m == b) { myG[j] = acc[j] + fm[j]; fb[j] = fm[j]; }
                acc[j] += tm[j];
                wide |= !(fm[j] - tm[j] <= kF16GramLog);   // (a NaN counts as wide)
            }
        }
        // Gram operands as f16 when every block's decay allows it (the weak-decay
        // end of the gate range, where the rounding of q~ and k^ is carried
        // through the most chunks), else bf16
        const bool gram_f16 = !__syncthreads_or(wide);
        float ap[8], R[8];                         // a at the block start; a_last / a(block start)
#pragma unroll
        for (int j = 0; j < 8; ++j) { ap[j] = __expf(myG[j]); R[j] = __expf(acc[j] - myG[j]); }
        if (b == 0 && rq == 0) {
            float al[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) al[j] = __expf(acc[j]);
            *reinterpret_cast<float4*>(blk + WS_AL + 4 * c0) = make_float4(al[0], al[1], al[2], al[3]);
            *reinterpret_cast<float4*>(blk + WS_AL + 4 * c0 + 16) = make_float4(al[4], al[5], al[6], al[7]);
        }

        if (!PROLOGUE) wait(bar_qk, n_done & 1);   // q and k (copied behind the cumulative sum)
        // ---------------- a1: operands, row by row.  Row factors exp(G_r - G_pb) <= 1,
        // column factors exp(G_pb - G_t) >= 1 (<= e^75), with p_b the block's first row
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 8; ++j) e[i][j] = __expf(e[i][j] - fb[j]);
        }
        // the row operands and the Gram column tiles
        auto operands = [&](uint32_t F16) {
    #pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = r0 + i;
                float q[8], k[8];
                load_qk(i, q, k);
                if (PROLOGUE) {                        // unit-length q and k rows
                    const float iq = rsqrtf(nrm[r] + nrm[64 + r] + kda::kNormEps);
                    const float ik = rsqrtf(nrm[128 + r] + nrm[192 + r] + kda::kNormEps);
    #pragma unroll
                    for (int j = 0; j < 8; ++j) { q[j] *= iq; k[j] *= ik; }
                }
                // each operand row is formed and stored before the next one is formed
                // (few values live at a time)
                {
                    float t[8];
    #pragma unroll
                    for (int j = 0; j < 8; ++j) t[j] = q[j] * e[i][j];            // q~ (row factor)
                    *reinterpret_cast<uint4*>(sm + K1_AG + kda::sw128(32 * b + 4 * rq + i, c0, 128)) = pack8g(t, F16);
    #pragma unroll
                    for (int j = 0; j < 8; ++j) t[j] *= ap[j];                    // Q_decay
                    // -> rows 0..63 of the [Q_decay; W] image (read back for Q')
                    *reinterpret_cast<uint4*>(blk + WS_A1 + kda::sw128(r, c0, 128)) = pack8(t);
    #pragma unroll
                    for (int j = 0; j < 8; ++j) t[j] = bt[i] * k[j] * e[i][j];    // k^ = beta k (row factor)
                    *reinterpret_cast<uint4*>(sm + K1_AG + kda::sw128(32 * b + 16 + 4 * rq + i, c0, 128)) = pack8g(t, F16);
    #pragma unroll
                    for (int j = 0; j < 8; ++j) t[j] = k[j] * e[i][j] * ap[j];    // K_decay
                    *reinterpret_cast<uint4*>(sm + K1_BWU + kda::sw128(r, c0, 64)) = pack8(t);
                }
                float kt[8];
    #pragma unroll
                for (int j = 0; j < 8; ++j) kt[j] = k[j] * __fdividef(1.f, e[i][j]);   // k (column factor, own block)
                // K_restore -> K_restore^T images, high and low bf16 parts (MN-major:
                // row = token, contiguous = channel)
                {
                    float kr[8];
    #pragma unroll
                    for (int j = 0; j < 8; ++j) kr[j] = kt[j] * R[j];
                    uint4 hi, lo;
                    split_pack8(kr, hi, lo);
                    const uint32_t off = kda::sw128(r, c0, 64);
                    *reinterpret_cast<uint4*>(blk + WS_KR + off) = hi;
                    *reinterpret_cast<uint4*>(blk + WS_KRL + off) = lo;
                }
    #pragma unroll
                for (int j = 0; j < 8; ++j) e[i][j] = kt[j];           // kept for the later tiles
            }
            // the column operands overlay the q / k input tiles: every thread has read its rows
            __syncthreads();
            // own block's column operand (block b of tile b)
    #pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(sm + K1_BG + kda::sw128(8 * b * (b + 1) + r0 + i, c0, 160)) = pack8g(e[i], F16);
            // tiles m > b hold this block's column factors times a(p_m) / a(p_b) <= 1
            // (a rolled loop keeps this replicated part of the code small)
    #pragma unroll 1
            for (int m = b + 1; m < 4; ++m) {
                float sc[8], gm[8];
    #pragma unroll
                for (int j = 0; j < 8; ++j) gm[j] = 0.f;
                for (int mm = 0; mm < m; ++mm) {
    #pragma unroll
                    for (int j = 0; j < 8; ++j) gm[j] += tot[mm * 128 + c0 + j];
                }
                float gb[8];                           // this block's reference G_pb
    #pragma unroll
                for (int j = 0; j < 8; ++j) gb[j] = 0.f;
                for (int mm = 0; mm < b; ++mm) {
    #pragma unroll
                    for (int j = 0; j < 8; ++j) gb[j] += tot[mm * 128 + c0 + j];
                }
    #pragma unroll
                for (int j = 0; j < 8; ++j)
                    sc[j] = __expf((gm[j] + first[m * 128 + c0 + j]) - (gb[j] + first[b * 128 + c0 + j]));
                uint8_t* tile = sm + K1_BG + 1024 * m * (m + 1);        // row 8 m (m + 1), an 8-row atom boundary
    #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float f[8];
    #pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] = e[i][j] * sc[j];
                    *reinterpret_cast<uint4*>(tile + kda::sw128(16 * b + 4 * rq + i, c0, 160)) = pack8g(f, F16);
                }
            }
        };
        operands(gram_f16 ? 1u : 0u);
        kda::fence_proxy_async_all();              // shared operands and the Q_decay rows read back later
        kda::tc_fence_before();
        __syncthreads();

        // ---------------- a2: Gram MMAs: all 128 rows against the 160 stacked B rows
        // (row block b's products sit in columns [8b(b+1), 8b(b+1) + 16(b+1)))
        if (tid == 0 && !*abort_f) {
            kda::tc_fence_after();
            const uint32_t sAG = kda::smem_u32(sm + K1_AG), sBG = kda::smem_u32(sm + K1_BG);
            const uint32_t idesc = gram_f16 ? kda::idesc_f16(128, 160, 0, 0) : kda::idesc_bf16(128, 160, 0, 0);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t ad = kda::sw128_desc(sAG + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
                const uint64_t bd = kda::sw128_desc(sBG + (s >> 2) * 20480 + (s & 3) * 32, 16, 1024);
                kda::umma_bf16(tmem, ad, bd, idesc, s > 0 ? 1u : 0u);
            }
            kda::umma_commit(bar);
        }
        wait(bar, bar_phase & 1);
        ++bar_phase;
        kda::tc_fence_after();

        float* LS = reinterpret_cast<float*>(sm + K1_LS);
        float* IS = reinterpret_cast<float*>(sm + K1_IS);
        gram_epilogue(tmem, w & 3, w >> 2, lane, sm + K1_MH, sm + K1_ML, LS);
        kda::tc_fence_before();
        __syncthreads();

        // ---------------- a3: INV = (I + L)^-1, by 16x16 blocks
        // (1) diagonal blocks D_b by forward substitution (warps 0-3); zero the blocks above
        if (w < 4) {
            if (lane < 16) {                       // diagonal block w, column `lane`
                const int o = 16 * w, j = lane;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {              // four partial sums shorten the FMA chain
                    float a[4] = {(r == j) ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int t = 0; t < r; ++t) a[t & 3] = fmaf(-LS[(o + r) * LDS_ + o + t], x[t], a[t & 3]);
                    x[r] = (a[0] + a[1]) + (a[2] + a[3]);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) IS[(o + r) * LDS_ + o + j] = x[r];
            }
        } else {
            for (int e = tid - 128; e < 6 * 256; e += 128) {
                const int pb = e >> 8, idx = e & 255;
                const int bi = pb < 3 ? 0 : (pb < 5 ? 1 : 2);
                const int bj = pb < 3 ? pb + 1 : (pb < 5 ? pb - 1 : 3);
                IS[(16 * bi + (idx >> 4)) * LDS_ + 16 * bj + (idx & 15)] = 0.f;
            }
        }
        __syncthreads();
        auto blkL = [&](int bi, int bj) { return LS + (16 * bi) * LDS_ + 16 * bj; };
        auto blkI = [&](int bi, int bj) { return IS + (16 * bi) * LDS_ + 16 * bj; };
        // scratch slots (dense 16x16): 0 F = L10 D0, 1 E = L32 D2, 2 -L21 D1, 3 -L31 D1,
        // 4 L20 D0, 5 L30 D0, 6 Z00, 7 Z10
        auto xs = [&](int i) { return reinterpret_cast<float*>(sm + (i < 4 ? K1_XS : K1_XS2)) + 256 * (i & 3); };
        // The lower-left 2x2 block of INV is -INV_bottom Z with Z = L_[23][01] INV_top,
        // INV_top / INV_bottom the inverses of the top-left / bottom-right 2x2 blocks;
        // Z's blocks L20 D0 + L21 INV_10 (INV_10 = -D1 L10 D0) etc. are formed from
        // products that need only the diagonal inverses, so the chain of dependent
        // 16x16 products is four long (instead of six).
        // (2) the products of L blocks with diagonal inverses (warps 0-5)
        if (w < 6) {
            // warp w: L block (bi, bj) times D_bj, with (bi, bj) = (1,0) (3,2) (2,1) (3,1) (2,0) (3,0),
            // 4 bits per warp in one constant (no per-thread table in local memory)
            const uint32_t code = (0x3276B1u >> (4 * w)) & 15u;    // warp 0 in the low nibble
            const int bi = (int)(code & 3u), bj = (int)(code >> 2);
            float acc[8];
            mm16(acc, blkL(bi, bj), LDS_, blkI(bj, bj), LDS_, lane, false);
            st16(xs(w), 16, acc, lane, (w == 2 || w == 3) ? -1.f : 1.f);
        }
        __syncthreads();
        // (3) INV_10 = -D1 F, INV_32 = -D3 E, Z00 = L20 D0 - (L21 D1) F, Z10 = L30 D0 - (L31 D1) F  (warps 0-3)
        if (w < 4) {
            float acc[8];
            if (w < 2) {
                mm16(acc, blkI(2 * w + 1, 2 * w + 1), LDS_, xs(w), 16, lane, false);
                st16(blkI(2 * w + 1, 2 * w), LDS_, acc, lane, -1.f);
            } else {
                ld16(acc, xs(w + 2), 16, lane);
                mm16(acc, xs(w), 16, xs(0), 16, lane, true);
                st16(xs(w + 4), 16, acc, lane, 1.f);
            }
        }
        __syncthreads();
        // (4) INV_20 = -D2 Z00, INV_21 = D2 (-Z01), INV_30 = -(INV_32 Z00 + D3 Z10),
        //     INV_31 = INV_32 (-Z01) + D3 (-Z11)   (Z01 = L21 D1, Z11 = L31 D1; warps 0-3)
        if (w < 4) {
            const int yi = w >> 1, yj = w & 1;
            float acc[8];
            const float* z0 = xs(yj ? 2 : 6);            // Z0j (negated for j = 1)
            if (yi == 0) {
                mm16(acc, blkI(2, 2), LDS_, z0, 16, lane, false);
            } else {
                mm16(acc, blkI(3, 2), LDS_, z0, 16, lane, false);
                mm16(acc, blkI(3, 3), LDS_, xs(yj ? 3 : 7), 16, lane, true);
            }
            st16(blkI(2 + yi, yj), LDS_, acc, lane, yj ? 1.f : -1.f);
        }
        __syncthreads();
        // (5) X = M_qk INV on the tensor cores: INV -> high / low bf16 operand parts
        // (over L), then X = M_hi I_hi + M_hi I_lo + M_lo I_hi into TMEM
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int e = tid + 256 * half;
            const int t = e >> 3, cc = e & 7;
            uint4 hi, lo;
            split_pack8(IS + t * LDS_ + 8 * cc, hi, lo);
            *reinterpret_cast<uint4*>(sm + K1_IH + kda::sw128(t, 8 * cc, 64)) = hi;
            *reinterpret_cast<uint4*>(sm + K1_IL + kda::sw128(t, 8 * cc, 64)) = lo;
        }
        kda::fence_proxy_async_smem();
        kda::tc_fence_before();
        __syncthreads();
        if (tid == 0 && !*abort_f) {
            kda::tc_fence_after();
            const uint32_t idesc = kda::idesc_bf16(128, 64, 0, 1);
            const uint32_t sA[3] = {kda::smem_u32(sm + K1_MH), kda::smem_u32(sm + K1_MH), kda::smem_u32(sm + K1_ML)};
            const uint32_t sB[3] = {kda::smem_u32(sm + K1_IH), kda::smem_u32(sm + K1_IL), kda::smem_u32(sm + K1_IH)};
#pragma unroll
            for (int pr = 0; pr < 3; ++pr) {
#pragma unroll
                for (int st = 0; st < 4; ++st) {
                    const uint64_t ad = kda::sw128_desc(sA[pr] + st * 32, 16, 1024);
                    const uint64_t bd = kda::sw128_desc(sB[pr] + st * 2048, 8192, 1024);
                    kda::umma_bf16(tmem + K1_TX, ad, bd, idesc, (pr | st) ? 1u : 0u);
                }
            }
            kda::umma_commit(bar);
        }
        wait(bar, bar_phase & 1);
        ++bar_phase;
        kda::tc_fence_after();
        // [INV; X] Diag(beta) -> 128-row K-major A operand as high + low bf16 parts
        // (the operand overlays the M_qk parts, which the X product has finished reading)
        if ((w & 2) == 0) {                        // warps 0, 1, 4, 5: X rows from TMEM lanes 0..63
            const int r = 32 * (w & 1) + lane, c0 = 32 * (w >> 2);
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                float f[8];
                kda::tmem_ld8(tmem + ((uint32_t)(32 * (w & 1)) << 16) + K1_TX + c0 + 8 * cc, f);
                kda::tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] *= beta_s[c0 + 8 * cc + u];
                uint4 hi, lo;
                split_pack8(f, hi, lo);
                *reinterpret_cast<uint4*>(sm + K1_AI + kda::sw128(64 + r, c0 + 8 * cc, 64)) = hi;
                *reinterpret_cast<uint4*>(sm + K1_AIL + kda::sw128(64 + r, c0 + 8 * cc, 64)) = lo;
            }
        } else {                                   // warps 2, 3, 6, 7: INV rows from shared memory
            const int li = 32 * (((w >> 2) << 1) | (w & 1)) + lane;
            const int r = li >> 1, c0 = 32 * (li & 1);
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                float f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] = IS[r * LDS_ + c0 + 8 * cc + u] * beta_s[c0 + 8 * cc + u];
                uint4 hi, lo;
                split_pack8(f, hi, lo);
                *reinterpret_cast<uint4*>(sm + K1_AI + kda::sw128(r, c0 + 8 * cc, 64)) = hi;
                *reinterpret_cast<uint4*>(sm + K1_AIL + kda::sw128(r, c0 + 8 * cc, 64)) = lo;
            }
        }
        kda::fence_proxy_async_smem();
        kda::tc_fence_before();
        __syncthreads();

        // ---------------- a3: [W | U0] = INV Diag(beta) [K_decay | V]  (INV in two bf16 parts)
        if (tid == 0 && !*abort_f) {
            kda::tc_fence_after();
            const uint32_t sB = kda::smem_u32(sm + K1_BWU);
            const uint32_t idesc = kda::idesc_bf16(128, 256, 0, 1);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint32_t sAI = kda::smem_u32(sm + (part ? K1_AIL : K1_AI));
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ad = kda::sw128_desc(sAI + s * 32, 16, 1024);
                    const uint64_t bd = kda::sw128_desc(sB + s * 2048, 8192, 1024);
                    kda::umma_bf16(tmem, ad, bd, idesc, (part | s) ? 1u : 0u);
                }
            }
            kda::umma_commit(bar);
            // meanwhile, the Q_decay rows (both 64-channel panels) back into the [Q'; W] image
            kda::mbar_arrive_expect_tx(bar_q, 16384);
            kda::bulk_g2s(sm + K1_OUT_A1, blk + WS_A1, 8192, bar_q);
            kda::bulk_g2s(sm + K1_OUT_A1 + 16384, blk + WS_A1 + 16384, 8192, bar_q);
            ++n_qloads;
        }
        wait(bar, bar_phase & 1);
        ++bar_phase;
        kda::tc_fence_after();

        // the last MMA is done with its operands: the next item's log-decay tile
        // (over the [INV; X] operand) and V (over this item's V) can come in
        if (tid == 0) {
            if (dyn) {
                // the next item is drawn even after an abort (the loop runs out the items)
                const long long nx = draw();
                *next_it = nx;                     // read by every thread after the item's last barrier
                int t1, r1, s1, h1;
                if (!*abort_f && nx < n_items && item(nx, t1, r1, s1, h1)) {
                    load_gv(t1, h1);
                    gv_ready = true;
                }
            } else if (!*abort_f) {
                for (long long nx = it + gridDim.x; nx < n_items; nx += gridDim.x) {
                    int t1, r1, s1, h1;
                    if (!item(nx, t1, r1, s1, h1)) continue;
                    load_gv(t1, h1);
                    gv_ready = true;
                    break;
                }
            }
        }
        // TMEM lanes 0..63 hold [W | U0], lanes 64..127 hold [M_qk W | O0] (columns
        // 0..127 | 128..255).  The two warps of a TMEM lane quarter (w and w + 4)
        // each take two of the four 32-column blocks of both halves: first the fp32
        // U0 / O0 rows, straight to the workspace (512 contiguous bytes a warp), then
        // the W rows or, once Q_decay is back, the Q' rows of the [Q'; W] image.
        const int quad = w & 3, r = 32 * (quad & 1) + lane, cb0 = 2 * (w >> 2);
        const uint32_t t_lane = tmem + ((uint32_t)(32 * quad) << 16);
        {
            const uint32_t part = quad < 2 ? 0u : TILE_F32;    // U0 (lanes 0..63) or O0 (lanes 64..127)
#pragma unroll 1
            for (int cb = cb0; cb < cb0 + 2; ++cb) {
                float x[32];
                kda::tmem_ld32(t_lane + 128 + 32 * cb, x);
                kda::tmem_wait_ld();
                const int tile = (32 * cb) / NT, c0 = (32 * cb) % NT;
                uint8_t* dst = blk + WS_UO + 2 * TILE_F32 * tile + part;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<float4*>(dst + uo_off(r, c0 + 4 * u)) =
                        make_float4(x[4 * u], x[4 * u + 1], x[4 * u + 2], x[4 * u + 3]);
            }
        }
        if (quad < 2) {                            // W rows -> rows 64..127 of [Q'; W]
#pragma unroll 1
            for (int cb = cb0; cb < cb0 + 2; ++cb) {
                float x[32];
                kda::tmem_ld32(t_lane + 32 * cb, x);
                kda::tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4*>(sm + K1_OUT_A1 + kda::sw128(64 + r, 32 * cb + 8 * u, 128)) = pack8(x + 8 * u);
            }
        } else {                                   // Q' = Q_decay - M_qk W -> rows 0..63 of [Q'; W]
            wait(bar_q, n_done & 1);
#pragma unroll 1
            for (int cb = cb0; cb < cb0 + 2; ++cb) {
                float x[32];
                kda::tmem_ld32(t_lane + 32 * cb, x);
                kda::tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4* qp = reinterpret_cast<uint4*>(sm + K1_OUT_A1 + kda::sw128(r, 32 * cb + 8 * u, 128));
                    const uint4 qd = *qp;
                    const uint32_t qs[4] = {qd.x, qd.y, qd.z, qd.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 f = kda::unpack_bf16x2(qs[j]);
                        x[8 * u + 2 * j] = f.x - x[8 * u + 2 * j];
                        x[8 * u + 2 * j + 1] = f.y - x[8 * u + 2 * j + 1];
                    }
                    *qp = pack8(x + 8 * u);
                }
            }
        }
        kda::fence_proxy_async_smem();
        kda::tc_fence_before();
        __syncthreads();                           // shared memory and TMEM are reused by the next item
        kda::tc_fence_after();
        if (tid == 0 && !*abort_f) {
            kda::bulk_s2g(blk + WS_A1, sm + K1_OUT_A1, 32768);
            kda::bulk_commit();
        }
        ++n_done;
    }
    if (tid == 0) {
        if (*abort_f) {
            // a wait ran out: let the copies and MMAs already issued finish
            // (bounded again) before the shared memory and TMEM are released
            if (n_gv) (void)kda::mbar_wait(bar_gv, (n_gv - 1) & 1, kda::kWaitCycles);
            if (n_qk) (void)kda::mbar_wait(bar_qk, (n_qk - 1) & 1, kda::kWaitCycles);
            if (n_qloads) (void)kda::mbar_wait(bar_q, (n_qloads - 1) & 1, kda::kWaitCycles);
            kda::umma_commit(bar_drain);           // arrives once every MMA issued so far is done
            (void)kda::mbar_wait(bar_drain, 0, kda::kWaitCycles);
        }
        kda::bulk_wait_all();                      // the workspace is complete when the kernel ends
    }
    kda::tc_fence_before();
    __syncthreads();
    kda::tc_fence_after();
    if (w == 0) kda::tmem_dealloc(tmem, K1_TMEM_COLS);
}

// ============================================================== chain (a4, a5)
// Per CTA: one (sequence, head) pair and NTC columns of d_v (64; or 32, with
// four CTAs per pair, when the whole pass fits one wave: each conversion
// thread then moves half as many values on the sequential path, while the
// MMAs, issue-bound at this size, take as long).  TMEM columns:
//   [0, NTC)          S, the fp32 state slice (TMEM lane = key channel)
//   [NTC, 2 NTC)      X, the low-part share K_restore^T U_lo of the state
//                     update, folded into S when the state is next read
//   [2 NTC, 4 NTC)    P of even chunks, [4 NTC, 6 NTC) P of odd chunks:
//                     P = [Q'; W] [S_hi | S_lo]: columns 0..NTC-1 against the
//                     high part of S_in, the next NTC against its low part;
//                     lanes 0..63 Q' S_in, lanes 64..127 W S_in
// MMAs per chunk (16 instructions):
//   P        = [Q'; W] [S_hi | S_lo]                        K = 128, N = 2 NTC -> commit(p)
//   [S | X] += K_hi^T [U_hi | U_lo] + K_lo^T [U_hi | U_lo]  K = 64,  N = 2 NTC -> commit(s)
// with U = U0 - W S_in, O = Q' S_in + O0, and S_in, K_restore and U each
// carried as a high and a low bf16 part (x = hi + lo, |lo| <= 2^-8 |x|), so
// that no operand of the sequential pass is rounded to a single bf16: the
// pass carries its error from chunk to chunk, and at the no-decay end of the
// gate range it would otherwise add up over the sequence.  Q' = Q_decay -
// M_qk W and O0 = M_qk U0 come from the prep kernel, so O = Q_decay S_in +
// M_qk U needs no product of its own here.
// [Q'; W] and K_restore^T stream through two rings filled by bulk copies;
// the U0 and O0 tiles of the slice arrive by bulk copy too (one chunk each),
// and the output rows leave by a tensor store, so that the conversion warps
// have no global loads or stores in flight at their proxy fences.  P
// alternates between two TMEM buffers, so the output rows of chunk c are
// formed while chunk c + 1 runs, off the sequential path.
// Warp roles:
//   warps 0-15 conversion warps; warp w reads TMEM lanes 32 (w % 4) .. +31 and
//              columns CW (w / 4) .. +CW-1 (CW = NTC / 4) of each NTC-wide
//              block (four warps per sub-partition, so that their latencies
//              overlap).
//              - all 16: S_in = S + X -> high/low bf16 operand; then
//                S <- Diag(a_last) S_in, X <- 0
//              - lanes 64..127 (w % 4 = 2, 3): U = U0 - W S_in -> high/low bf16 operand
//              - lanes 0..63 (w % 4 = 0, 1): O rows of the previous chunk =
//                Q' S_in + O0, staged in shared memory and stored row by row
//   warp 16    lane 0 issues the MMAs
//   warp 17    lane 0 issues the bulk copies of the two rings
//   warp 18    lane 0 issues the bulk copies of the U0 and O0 tiles
// Named barriers (warps 0-16): 1 = S_in ready; 2 = conversion warps arrive, the
// issuer waits (U ready, state rescaled); 3 = the eight O warps (output staging).
// A wait that runs out sets the CTA's abort flag: from then on no copy or MMA
// is issued, every other wait returns at once, and before the CTA exits the
// copies and MMAs already in flight are waited for (bounded again).
constexpr int K2_CONV_WARPS = 16;
constexpr int K2_THREADS = 32 * (K2_CONV_WARPS + 3);
constexpr int K2_SYNC = 32 * (K2_CONV_WARPS + 1);  // conversion warps + the MMA issuer
constexpr int K2_ISSUER_WARP = K2_CONV_WARPS;
constexpr int K2_PRODUCER_WARP = K2_CONV_WARPS + 1;
constexpr int K2_TILE_WARP = K2_CONV_WARPS + 2;

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int NTC>
__global__ void __launch_bounds__(K2_THREADS, 1)
kda_tc_chain(const int4* __restrict__ seq_info, int use_table, int fixed_len, int nch_per_seq,
             int c_begin, int c_end, const uint8_t* __restrict__ ws_blocks, const float* __restrict__ S0, int H,
             bf16* __restrict__ O, float* __restrict__ S_final, int ckpt_every, float* __restrict__ ckpt,
             int ckpt_cap, int* status, int seg_pass1, float* __restrict__ S_final_map, int n_slots,
             const __grid_constant__ CUtensorMap tm_o, int o_tma, const int* __restrict__ seq_order) {
    // seg_pass1 (segment scan, first pass): blockIdx.z = 0 runs each segment
    // from a zero state (its affine offset, into S_final), blockIdx.z = 1 from
    // the identity with U0 taken as zero (its linear map, into S_final_map);
    // neither writes O.
    using Cfg = ChainCfg<NTC>;
    constexpr int K2_CW = Cfg::CW;
    constexpr uint32_t K2_SB = Cfg::SB, K2_UB = Cfg::UB, K2_OS = Cfg::OS, K2_U0 = Cfg::U0, K2_O0 = Cfg::O0;
    const bool run_map = seg_pass1 && blockIdx.z == 1;
    const bool write_o = !seg_pass1;
    if (run_map) S_final = S_final_map;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    // CTA -> (slice, sequence, head): grid (slices x sequences, heads), or with
    // seq_order grid (slices x heads, sequences) with y the sequence's rank by length
    const int tile = blockIdx.x % Cfg::NTL;
    const int n = seq_order ? seq_order[blockIdx.y] : (int)(blockIdx.x / Cfg::NTL);
    const int h = seq_order ? (int)(blockIdx.x / Cfg::NTL) : (int)blockIdx.y;
    // this slice's U0 / O0 tiles in a workspace block: the prep stores them per
    // 64-column slice, and a 32-column slice is one half of such a tile
    const uint32_t ws_u0 = WS_UO + 2 * TILE_F32 * (uint32_t)((tile * NTC) / 64) + (uint32_t)((tile * NTC) % 64) * C * 4;
    int bos, len, first, nch;
    if (!use_table) {
        bos = n * fixed_len; len = fixed_len; first = n * nch_per_seq; nch = nch_per_seq;
    } else {
        const int4 si = seq_info[n];
        bos = si.x; len = si.y; first = si.z; nch = si.w;
    }
    // this launch runs chunks [c_begin, c_end) of the sequence; locally they are
    // numbered 0 .. nloc - 1 (stage and barrier parities use the local number)
    const int cb = min(c_begin, nch);
    int nloc = max(0, min(c_end, nch) - cb);
    // the chunks' workspace blocks must exist (debug builds check; none is read otherwise)
    if (!KDA_DCHECK(status, nloc == 0 || (first + cb >= 0 && first + cb + nloc <= n_slots))) nloc = 0;
    // state checkpoints: index of this sequence's first one (block-wide sum)
    int ck_base = 0;
    if (ckpt_every > 0)
        ck_base = use_table ? kda::ckpt_base(n, ckpt_every, [&](int m) { return seq_info[m].y; })
                            : n * (fixed_len / ckpt_every);
    // store this thread's K2_CW state values as checkpoint `idx` (if it fits)
    auto put_ckpt = [&](int idx, const float* vals, int row_, int col0) {
        if (idx < 0 || idx >= ckpt_cap) return;
        float4* dst = reinterpret_cast<float4*>(ckpt + (((size_t)idx * H + h) * DK + row_) * DV + tile * NTC + col0);
#pragma unroll
        for (int u = 0; u < K2_CW / 4; ++u)
            dst[u] = make_float4(vals[4 * u], vals[4 * u + 1], vals[4 * u + 2], vals[4 * u + 3]);
    };
    auto block_of = [&](int c) { return ws_blocks + ((size_t)(first + cb + c) * H + h) * WS_BLOCK; };
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    uint64_t* fullA = reinterpret_cast<uint64_t*>(sm + Cfg::BAR);
    uint64_t* emptyA = fullA + K2_NA;
    uint64_t* fullB = emptyA + K2_NA;
    uint64_t* emptyB = fullB + K2_NB;
    uint64_t* bar_p = emptyB + K2_NB;
    uint64_t* bar_s = bar_p + 1;
    uint64_t* bar_drain = bar_s + 1;
    uint64_t* fullU = bar_drain + 1;                // U0 tile: landed / read by the eight U warps
    uint64_t* emptyU = fullU + 1;
    uint64_t* fullO = emptyU + 1;                   // O0 tile: landed / read by the eight O warps
    uint64_t* emptyO = fullO + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(emptyO + 1);
    volatile int* abort_f = reinterpret_cast<volatile int*>(tmem_slot + 1);
    if (w == 0) {
        kda::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        kda::tmem_relinquish();
    }
    if (tid == 0) {
        // a stage is free once the MMAs that read it are done (one commit each)
        for (int s = 0; s < K2_NA; ++s) { kda::mbar_init(fullA + s, 1); kda::mbar_init(emptyA + s, 1); }
        for (int s = 0; s < K2_NB; ++s) { kda::mbar_init(fullB + s, 1); kda::mbar_init(emptyB + s, 1); }
        kda::mbar_init(bar_p, 1);
        kda::mbar_init(bar_s, 1);
        kda::mbar_init(bar_drain, 1);
        kda::mbar_init(fullU, 1);
        kda::mbar_init(emptyU, K2_CONV_WARPS / 2);
        kda::mbar_init(fullO, 1);
        kda::mbar_init(emptyO, K2_CONV_WARPS / 2);
        kda::fence_barrier_init();
        *abort_f = 0;
    }
    kda::tc_fence_before();
    __syncthreads();
    kda::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto wait = [&](uint64_t* b, uint32_t parity) {
        if (!kda::mbar_wait_or_abort(b, parity, kda::kWaitCycles, abort_f)) {
            kda::record_status(status, kda::kDevTimeout);
            *abort_f = 1;
        }
    };

    if (w == K2_PRODUCER_WARP) {
        // ---------------- bulk copies, in the order the chunks need them
        if (lane == 0) {
            int nA = 0, nB = 0;                             // copies issued into each ring
            for (int k = 0; k < nloc && !*abort_f; ++k) {
                const int sa = k % K2_NA;
                if (k >= K2_NA) wait(emptyA + sa, (uint32_t)(((k - K2_NA) / K2_NA) & 1));
                if (*abort_f) break;
                kda::mbar_arrive_expect_tx(fullA + sa, K2_ASTAGE);
                kda::bulk_g2s(sm + sa * K2_ASTAGE, block_of(k) + WS_A1, K2_ASTAGE, fullA + sa);
                ++nA;
                // this chunk's U0 / O0 tiles (copied by the tile warp when their
                // buffers come free) and a_last (loaded by every conversion thread) into L2
                kda::bulk_prefetch_l2(block_of(k) + ws_u0, Cfg::TILE);
                kda::bulk_prefetch_l2(block_of(k) + ws_u0 + TILE_F32, Cfg::TILE);
                kda::bulk_prefetch_l2(block_of(k) + WS_AL, DK * 4);
                const int sb = k % K2_NB;
                if (k >= K2_NB) wait(emptyB + sb, (uint32_t)(((k - K2_NB) / K2_NB) & 1));
                if (*abort_f) break;
                kda::mbar_arrive_expect_tx(fullB + sb, K2_BSTAGE);
                kda::bulk_g2s(sm + K2_B0 + sb * K2_BSTAGE, block_of(k) + WS_KR, K2_BSTAGE, fullB + sb);
                ++nB;
            }
            if (*abort_f) {
                // the last copy into each stage completes that stage's newest phase
                for (int k = max(0, nA - K2_NA); k < nA; ++k)
                    (void)kda::mbar_wait(fullA + k % K2_NA, (uint32_t)((k / K2_NA) & 1), kda::kWaitCycles);
                for (int k = max(0, nB - K2_NB); k < nB; ++k)
                    (void)kda::mbar_wait(fullB + k % K2_NB, (uint32_t)((k / K2_NB) & 1), kda::kWaitCycles);
            }
        }
    } else if (w == K2_TILE_WARP) {
        // ---------------- U0 / O0 tiles of this slice, one chunk of each at a time
        if (lane == 0) {
            int nU = 0, nO = 0;                             // copies issued into each tile
            for (int k = 0; k < nloc && !*abort_f; ++k) {
                const uint8_t* uo = block_of(k) + ws_u0;
                if (k > 0) wait(emptyU, (uint32_t)((k - 1) & 1));
                if (*abort_f) break;
                kda::mbar_arrive_expect_tx(fullU, Cfg::TILE);
                kda::bulk_g2s(sm + K2_U0, uo, Cfg::TILE, fullU);
                ++nU;
                if (!write_o) continue;                     // no output rows: O0 is not needed
                if (k > 0) wait(emptyO, (uint32_t)((k - 1) & 1));
                if (*abort_f) break;
                kda::mbar_arrive_expect_tx(fullO, Cfg::TILE);
                kda::bulk_g2s(sm + K2_O0, uo + TILE_F32, Cfg::TILE, fullO);
                ++nO;
            }
            if (*abort_f) {                                 // the newest copy into each tile
                if (nU > 0) (void)kda::mbar_wait(fullU, (uint32_t)((nU - 1) & 1), kda::kWaitCycles);
                if (nO > 0) (void)kda::mbar_wait(fullO, (uint32_t)((nO - 1) & 1), kda::kWaitCycles);
            }
        }
    } else if (w == K2_ISSUER_WARP) {
        // ---------------- MMAs
        // operand descriptors: one per operand base; each MMA's start is a constant step from it
        const uint64_t sb0 = kda::sw128_desc(kda::smem_u32(sm + K2_SB), 16384, 1024);
        const uint64_t ub0 = kda::sw128_desc(kda::smem_u32(sm + K2_UB), 8192, 1024);
        named_bar_sync(1, K2_SYNC);                        // initial state in TMEM
        for (int c = 0; c < nloc; ++c) {
            const int sa = c % K2_NA, sb = c % K2_NB;
            if (lane == 0) wait(fullA + sa, (uint32_t)((c / K2_NA) & 1));
            __syncwarp();
            named_bar_sync(1, K2_SYNC);
            if (lane == 0 && !*abort_f) {                   // P = [Q'; W] [S_hi | S_lo]
                kda::tc_fence_after();
                const uint64_t ad0 = kda::sw128_desc(kda::smem_u32(sm + sa * K2_ASTAGE), 16, 1024);
                const uint32_t idesc = kda::idesc_bf16(128, 2 * NTC, 0, 1);
                const uint32_t tP = tmem + 2 * NTC + 2 * NTC * (c & 1);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    kda::umma_bf16(tP, ad0 + kda::desc_step((s >> 2) * 16384 + (s & 3) * 32),
                                   sb0 + kda::desc_step(s * 2048), idesc, s > 0 ? 1u : 0u);
                kda::umma_commit(bar_p);
                kda::umma_commit(emptyA + sa);
            }
            if (lane == 0) wait(fullB + sb, (uint32_t)((c / K2_NB) & 1));
            __syncwarp();
            named_bar_sync(2, K2_SYNC);
            if (lane == 0 && !*abort_f) {                   // [S | X] += K_hi^T [U_hi | U_lo] + K_lo^T [U_hi | U_lo]
                kda::tc_fence_after();
                const uint64_t ad0 = kda::sw128_desc(kda::smem_u32(sm + K2_B0 + sb * K2_BSTAGE), 8192, 1024);
                const uint32_t id_s = kda::idesc_bf16(128, 2 * NTC, 1, 1);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    kda::umma_bf16(tmem, ad0 + kda::desc_step((s >> 2) * 16384 + (s & 3) * 2048),
                                   ub0 + kda::desc_step((s & 3) * 2048), id_s, 1u);
                kda::umma_commit(bar_s);
                kda::umma_commit(emptyB + sb);
            }
            __syncwarp();
        }
        if (lane == 0) {                                    // every MMA done before TMEM is released
            kda::umma_commit(bar_drain);
            (void)kda::mbar_wait(bar_drain, 0, kda::kWaitCycles);
        }
        __syncwarp();
    } else {
        // ---------------- conversion warps
        const int quad = w & 3, grp = w >> 2;
        const int row = 32 * quad + lane;                       // TMEM lane = state row / P row
        const int col0 = K2_CW * grp;                           // this warp's first column of the slice
        const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
        const uint32_t tS = tmem + lane_off + col0;             // this warp's state columns (X at +NTC)
        const uint32_t tP = tmem + lane_off + 2 * NTC + col0;   // ... of P (buffer of chunk parity at +2 NTC)
        auto tld = [&](uint32_t ta, float* r) {
            if constexpr (K2_CW == 16) kda::tmem_ld16(ta, r); else kda::tmem_ld8(ta, r);
        };
        auto tst = [&](uint32_t ta, const float* r) {
            if constexpr (K2_CW == 16) kda::tmem_st16(ta, r); else kda::tmem_st8(ta, r);
        };
        const bool u_rows = quad >= 2;                          // lanes 64..127: U; lanes 0..63: O
        // this thread's 16 values of a U0 or O0 tile in shared memory (row r of the chunk)
        auto read_tile = [&](uint32_t off, int r, float* dst) {
#pragma unroll
            for (int j = 0; j < K2_CW / 4; ++j) {
                const float4 x = *reinterpret_cast<const float4*>(sm + off + uo_off(r, col0 + 4 * j));
                dst[4 * j] = x.x; dst[4 * j + 1] = x.y; dst[4 * j + 2] = x.z; dst[4 * j + 3] = x.w;
            }
        };
        const bool o_issuer = w == 0 && lane == 0;           // issues the output tensor stores
        // 16-byte piece k of output row r in the staging tile: the 128-byte
        // (NTC = 64) or 64-byte (NTC = 32) swizzle of the tensor store
        auto o_swz = [](int r, int k) -> int { return NTC == 64 ? (k ^ (r & 7)) : (k ^ ((r >> 1) & 3)); };
        // O rows of chunk co (lanes 0..63 warps): P of that chunk is complete (the
        // state update issued after it is); staged in shared memory and stored
        auto out_rows = [&](int co) {
            float o0[K2_CW];
            wait(fullO, (uint32_t)(co & 1));
            read_tile(K2_O0, row, o0);
            __syncwarp();
            if (lane == 0) kda::mbar_arrive(emptyO);
            kda::tc_fence_after();
            float ph[K2_CW], pl[K2_CW];
            tld(tP + 2 * NTC * (co & 1), ph);
            tld(tP + 2 * NTC * (co & 1) + NTC, pl);
            kda::tmem_wait_ld();
            uint4 ov[K2_CW / 8];
#pragma unroll
            for (int cc = 0; cc < K2_CW / 8; ++cc) {
                float f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] = o0[8 * cc + u] + (ph[8 * cc + u] + pl[8 * cc + u]);
                ov[cc] = pack8(f);
            }
            uint8_t* ost = sm + K2_OS;
            if (o_issuer) kda::bulk_wait_read_all();             // the previous tile has left shared memory
            named_bar_sync(3, K2_CONV_WARPS * 16);             // every O warp is done with the last staged rows
#pragma unroll
            for (int cc = 0; cc < K2_CW / 8; ++cc) {
                const int k = (col0 + 8 * cc) / 8;               // 16-byte piece of the row
                *reinterpret_cast<uint4*>(ost + row * (2 * NTC) + (o_swz(row, k) << 4)) = ov[cc];
            }
            const int valid = len - (cb + co) * C;
            // a full chunk leaves by one tensor store (the staging order is the
            // store's 128-byte swizzle); the last rows of a sequence row by row,
            // since the rows past them belong to the next sequence
            const bool whole = o_tma && valid >= C;
            if (whole) kda::fence_proxy_async_smem();
            named_bar_sync(3, K2_CONV_WARPS * 16);             // the staged tile is complete
            if (whole) {
                if (o_issuer && !*abort_f) {
                    kda::tma_store_3d(&tm_o, tile * NTC, h, bos + (cb + co) * C, ost);
                    kda::bulk_commit();
                }
            } else {
                const int wo = (grp << 1) | quad;                // 0..7: rows 8 wo .. 8 wo + 7
                constexpr int LR = NTC / 2;                      // lanes per row (4 bytes each)
#pragma unroll
                for (int i = 0; i < 8 * LR / 32; ++i) {
                    const int rr = 8 * wo + (32 / LR) * i + lane / LR, pc = lane % LR;
                    if (rr < valid) {
                        const uint32_t x = *reinterpret_cast<const uint32_t*>(
                            ost + rr * (2 * NTC) + (o_swz(rr, pc >> 2) << 4) + 4 * (pc & 3));
                        *reinterpret_cast<uint32_t*>(O + ((size_t)(bos + (cb + co) * C + rr) * H + h) * DV +
                                                     tile * NTC + 2 * pc) = x;
                    }
                }
            }
            kda::tc_fence_before();
        };
        {
            // initial state slice -> TMEM (X = 0)
            float s[K2_CW];
            if (run_map) {
#pragma unroll
                for (int u = 0; u < K2_CW; ++u) s[u] = (row == tile * NTC + col0 + u) ? 1.f : 0.f;
            } else if (S0 && !seg_pass1) {
                const float4* src = reinterpret_cast<const float4*>(S0 + (((size_t)n * H + h) * DK + row) * DV +
                                                                    tile * NTC + col0);
#pragma unroll
                for (int u = 0; u < K2_CW / 4; ++u) {
                    const float4 x = src[u];
                    s[4 * u] = x.x; s[4 * u + 1] = x.y; s[4 * u + 2] = x.z; s[4 * u + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int u = 0; u < K2_CW; ++u) s[u] = 0.f;
            }
            tst(tS, s);
#pragma unroll
            for (int u = 0; u < K2_CW; ++u) s[u] = 0.f;
            tst(tS + NTC, s);
            kda::tmem_wait_st();
            kda::tc_fence_before();
            named_bar_sync(1, K2_SYNC);
        }
        float al_next = nloc > 0 ? reinterpret_cast<const float*>(block_of(0) + WS_AL)[row] : 1.f;
        for (int c = 0; c < nloc; ++c) {
            const float al = al_next;
            // ---- S_in = S + X -> high/low bf16 operand
            if (c > 0) wait(bar_s, (uint32_t)((c - 1) & 1));
            kda::tc_fence_after();
            float s[K2_CW], x[K2_CW];
            tld(tS, s);
            tld(tS + NTC, x);
            kda::tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < K2_CW; ++u) s[u] += x[u];
#pragma unroll
            for (int cc = 0; cc < K2_CW / 8; ++cc) {
                uint4 hi, lo;
                split_pack8(s + 8 * cc, hi, lo);
                *reinterpret_cast<uint4*>(sm + K2_SB + kda::sw128(row, col0 + 8 * cc, 128)) = hi;
                *reinterpret_cast<uint4*>(sm + K2_SB + kda::sw128(row, NTC + col0 + 8 * cc, 128)) = lo;
            }
            kda::fence_proxy_async_smem();
            kda::tc_fence_before();
            named_bar_sync(1, K2_SYNC);
            // the next chunk's a_last, loaded after the proxy fence (which would wait for it)
            if (c + 1 < nloc) al_next = reinterpret_cast<const float*>(block_of(c + 1) + WS_AL)[row];
            if (ckpt_every > 0 && cb + c > 0 && ((cb + c) * C) % ckpt_every == 0)   // state after (cb + c) chunks
                put_ckpt(ck_base + (cb + c) * C / ckpt_every - 1, s, row, col0);
            // ---- S <- Diag(a_last) S_in, X <- 0 while the P product runs
#pragma unroll
            for (int u = 0; u < K2_CW; ++u) { s[u] *= al; x[u] = 0.f; }
            tst(tS, s);
            tst(tS + NTC, x);
            kda::tmem_wait_st();
            if (u_rows) {
                // ---- U = U0 - W S_in -> high/low bf16 operand
                float uo[K2_CW];                                // U0 of this chunk
                wait(fullU, (uint32_t)(c & 1));
                read_tile(K2_U0, row - 64, uo);
                __syncwarp();
                if (lane == 0) kda::mbar_arrive(emptyU);
                wait(bar_p, (uint32_t)(c & 1));
                kda::tc_fence_after();
                const int r = row - 64;
                float ph[K2_CW], pl[K2_CW];
                tld(tP + 2 * NTC * (c & 1), ph);
                tld(tP + 2 * NTC * (c & 1) + NTC, pl);
                kda::tmem_wait_ld();
#pragma unroll
                for (int cc = 0; cc < K2_CW / 8; ++cc) {
                    float f[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        f[u] = (run_map ? 0.f : uo[8 * cc + u]) - (ph[8 * cc + u] + pl[8 * cc + u]);
                    uint4 hi, lo;
                    split_pack8(f, hi, lo);
                    *reinterpret_cast<uint4*>(sm + K2_UB + kda::sw128(r, col0 + 8 * cc, 64)) = hi;
                    *reinterpret_cast<uint4*>(sm + K2_UB + kda::sw128(r, NTC + col0 + 8 * cc, 64)) = lo;
                }
                kda::fence_proxy_async_smem();
                kda::tc_fence_before();
                named_bar_arrive(2, K2_SYNC);
            } else {
                kda::tc_fence_before();
                named_bar_arrive(2, K2_SYNC);
                if (write_o && c > 0) out_rows(c - 1);          // the previous chunk's output
            }
        }
        if (nloc > 0) wait(bar_s, (uint32_t)((nloc - 1) & 1));
        kda::tc_fence_after();
        if (write_o && !u_rows && nloc > 0) out_rows(nloc - 1);
        if (o_issuer) kda::bulk_wait_all();                     // the output stores are complete
        const bool end_ckpt = ckpt_every > 0 && nloc > 0 && cb + nloc == nch && len % ckpt_every == 0;
        if (S_final || end_ckpt) {
            float s[K2_CW], x[K2_CW];
            tld(tS, s);
            tld(tS + NTC, x);
            kda::tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < K2_CW; ++u) s[u] += x[u];
            if (end_ckpt) put_ckpt(ck_base + len / ckpt_every - 1, s, row, col0);
            if (S_final) {
                float4* dst = reinterpret_cast<float4*>(S_final + (((size_t)n * H + h) * DK + row) * DV +
                                                        tile * NTC + col0);
#pragma unroll
                for (int u = 0; u < K2_CW / 4; ++u)
                    dst[u] = make_float4(s[4 * u], s[4 * u + 1], s[4 * u + 2], s[4 * u + 3]);
            }
        }
    }
    kda::tc_fence_before();
    __syncthreads();
    if (w == 0) kda::tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// ============================================================== segment scan
// For few (sequence, head) chains and long sequences the state pass leaves most
// SMs idle.  The chunk-level map S -> A_c S + B_c (A_c = Diag(a_last) -
// K_restore^T W, B_c = K_restore^T U0) composes over a segment of chunks into
// S -> A_p S + B_p, so each sequence is cut into segments of at most L chunks:
// pass 1 runs the state pass on every segment twice in one launch (from zero:
// B_p; from the identity with U0 taken as zero: A_p), a scan forms each
// segment's true starting state, and pass 3 runs the state pass again from it,
// writing O.  Each pass is short; the scan is sequential only over segments.

// Segment tables: seg_info[s] = (token start, length, first chunk slot, chunks)
// for the segments of every sequence in order; seq_seg[n] = (first segment,
// segments).  Entries up to s_max that no sequence uses get zero chunks.
__global__ void __launch_bounds__(1024)
kda_tc_segments(const int4* __restrict__ seq_info, int use_table, int fixed_len, int nch_per_seq, int n_seq,
                int L, int s_max, int4* __restrict__ seg_info, int2* __restrict__ seq_seg, int* status) {
    __shared__ int part[1024];
    __shared__ int total;
    const int tid = threadIdx.x, nt = blockDim.x;
    auto info = [&](int n) {
        return use_table ? seq_info[n] : make_int4(n * fixed_len, fixed_len, n * nch_per_seq, nch_per_seq);
    };
    const int per = (n_seq + nt - 1) / nt;
    const int s0 = min(tid * per, n_seq), s1 = min(s0 + per, n_seq);
    int cnt = 0;
    for (int n = s0; n < s1; ++n) cnt += (info(n).w + L - 1) / L;
    part[tid] = cnt;
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int i = 0; i < nt; ++i) { const int c = part[i]; part[i] = acc; acc += c; }
        total = min(acc, s_max);
        if (acc > s_max) kda::record_status(status, KDA_ERR_INVALID_ARG);
    }
    __syncthreads();
    int sidx = part[tid];
    for (int n = s0; n < s1; ++n) {
        const int4 si = info(n);
        const int nseg = min((si.w + L - 1) / L, max(0, s_max - sidx));
        seq_seg[n] = make_int2(sidx, nseg);
        for (int j = 0; j < nseg; ++j) {
            const int c0 = j * L;
            seg_info[sidx + j] = make_int4(si.x + c0 * C, min(si.y - c0 * C, L * C), si.z + c0, min(L, si.w - c0));
        }
        sidx += nseg;
    }
    for (int e = total + tid; e < s_max; e += nt) seg_info[e] = make_int4(0, 0, 0, 0);
}

// Scan over the segments of one sequence, for one head and 32 state columns:
// S_start[first] = S0, S_start[p + 1] = A_p S_start[p] + B_p, S_final = the
// state after the last segment.  fp32 on CUDA cores (A_p in shared memory).
constexpr int SC_COLS = 32;
constexpr int SC_LDA = DK + 1;                   // padded row of A: conflict-free column reads
constexpr uint32_t SC_SMEM = (DK * SC_LDA + DK * SC_COLS) * 4;

__global__ void __launch_bounds__(256)
kda_tc_seg_scan(const int2* __restrict__ seq_seg, const float* __restrict__ A, const float* __restrict__ B,
                const float* __restrict__ S0, float* __restrict__ S_start, float* __restrict__ S_final, int H,
                int s_max, int* status) {
    extern __shared__ float sc_smem[];
    float* As = sc_smem;                         // [DK][SC_LDA]
    float* Ss = sc_smem + DK * SC_LDA;           // [DK][SC_COLS]
    const int n = blockIdx.x, h = blockIdx.y, c0 = SC_COLS * blockIdx.z;
    const int tid = threadIdx.x, i = tid >> 1, j0 = 16 * (tid & 1);   // this thread's row and 16 columns
    auto mat = [&](const float* base, int idx) { return base + ((size_t)idx * H + h) * DK * DV; };
    auto matw = [&](float* base, int idx) { return base + ((size_t)idx * H + h) * DK * DV; };
    {
        float4* srow = reinterpret_cast<float4*>(Ss + i * SC_COLS + j0);
        const float4* src = S0 ? reinterpret_cast<const float4*>(mat(S0, n) + (size_t)i * DV + c0 + j0) : nullptr;
#pragma unroll
        for (int u = 0; u < 4; ++u) srow[u] = src ? src[u] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    int2 ss = seq_seg[n];
    if (!KDA_DCHECK(status, ss.x >= 0 && ss.y >= 0 && ss.x + ss.y <= s_max)) ss.y = 0;
    for (int p = 0; p < ss.y; ++p) {
        const int sg = ss.x + p;
        // this segment's starting state; then its map A_p into shared memory
        const float4* srow = reinterpret_cast<const float4*>(Ss + i * SC_COLS + j0);
        float4* dst = reinterpret_cast<float4*>(matw(S_start, sg) + (size_t)i * DV + c0 + j0);
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u] = srow[u];
        const float4* a4 = reinterpret_cast<const float4*>(mat(A, sg));
        for (int e = tid; e < DK * DK / 4; e += 256) {
            const float4 x = a4[e];
            const int r = (4 * e) / DK, k = (4 * e) % DK;
            As[r * SC_LDA + k] = x.x; As[r * SC_LDA + k + 1] = x.y; As[r * SC_LDA + k + 2] = x.z;
            As[r * SC_LDA + k + 3] = x.w;
        }
        float acc[16];
        const float4* b4 = reinterpret_cast<const float4*>(mat(B, sg) + (size_t)i * DV + c0 + j0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float4 x = b4[u];
            acc[4 * u] = x.x; acc[4 * u + 1] = x.y; acc[4 * u + 2] = x.z; acc[4 * u + 3] = x.w;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < DK; ++k) {
            const float a = As[i * SC_LDA + k];
            const float4* sk = reinterpret_cast<const float4*>(Ss + k * SC_COLS + j0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 x = sk[u];
                acc[4 * u] = fmaf(a, x.x, acc[4 * u]); acc[4 * u + 1] = fmaf(a, x.y, acc[4 * u + 1]);
                acc[4 * u + 2] = fmaf(a, x.z, acc[4 * u + 2]); acc[4 * u + 3] = fmaf(a, x.w, acc[4 * u + 3]);
            }
        }
        __syncthreads();
        float4* sw = reinterpret_cast<float4*>(Ss + i * SC_COLS + j0);
#pragma unroll
        for (int u = 0; u < 4; ++u) sw[u] = make_float4(acc[4 * u], acc[4 * u + 1], acc[4 * u + 2], acc[4 * u + 3]);
        __syncthreads();
    }
    if (S_final) {
        const float4* srow = reinterpret_cast<const float4*>(Ss + i * SC_COLS + j0);
        float4* dst = reinterpret_cast<float4*>(matw(S_final, n) + (size_t)i * DV + c0 + j0);
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u] = srow[u];
    }
}

// Workspace header: chunk table (16 B a slot), sequence table (16 B a
// sequence), then kSliceWords 8-byte words: the item counters of the chunk-prep
// slices that run beside the state pass (and, once per device, the SM-id mask),
// then the sequences' order by length (4 B a sequence, up to kMaxOrdered).
constexpr int kSliceWords = 16;
constexpr int kMaxOrdered = 1024;            // the schedule kernel's block size
size_t header_bytes(int n_seq, long long slots) {
    const size_t raw = 16u * (size_t)slots + 16u * (size_t)n_seq + 8u * kSliceWords +
                       4u * (size_t)std::min(n_seq, kMaxOrdered);
    return (raw + 1023) & ~size_t(1023);
}

size_t state_bytes(int n_seq, int H) { return (size_t)n_seq * H * DK * DV * sizeof(float); }

long long slot_bound(int n_seq, int T_total) { return (long long)T_total / C + n_seq; }

// Segment-scan plan, a function of the problem's shape only (so that the
// workspace size is too): possible when one state pass has at most 32 CTAs;
// the segments are sized so that the first pass (two runs per segment) has at
// most 128 CTAs, and are at least 16 chunks long.
struct SegPlan {
    bool possible = false;
    int s_target = 0;                            // segments aimed at
    int s_max = 0;                               // table / buffer capacity
};
SegPlan seg_plan(int n_seq, int H) {
    SegPlan p;
    if ((long long)NTILES * n_seq * H > 32) return p;
    p.possible = true;
    p.s_target = std::max(n_seq, 128 / (2 * NTILES * H));
    p.s_max = p.s_target + n_seq;
    return p;
}
constexpr int kMinSegChunks = 16;
size_t seg_table_bytes(const SegPlan& p, int n_seq) {
    return p.possible ? ((16u * (size_t)p.s_max + 8u * (size_t)n_seq + 1023) & ~size_t(1023)) : 0;
}
size_t seg_state_bytes(const SegPlan& p, int H) {
    return p.possible ? 3u * (size_t)p.s_max * H * DK * DV * sizeof(float) : 0;
}

// ---- TMA descriptors for the [T, H, 128] input tensors.  cuTensorMapEncodeTiled
// is a driver entry point, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// Tensor [T, H, 128] of `esize`-byte elements at `base`; box = `box_x` channels
// of one head for 64 tokens, 128-byte swizzled when `swizzle` (box_x * esize = 128).
cudaError_t make_input_map(CUtensorMap* m, const void* base, int esize, int H, int T, int box_x, bool swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)128 * esize, (cuuint64_t)H * 128 * esize};
    const cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                           const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of the output O [T][H][d_v] bf16 for the state pass's stores: one
// box = 64 tokens x one head x ntc channels, swizzled in shared memory by the
// row's byte width (128 bytes for ntc = 64, 64 for ntc = 32).
cudaError_t make_output_map(CUtensorMap* m, void* base, int H, int T, int ntc) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)DV, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)DV * 2, (cuuint64_t)H * DV * 2};
    const cuuint32_t box[3] = {(cuuint32_t)ntc, 1, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           ntc == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// ---- stream overlap: the prep of a later slice of chunks runs while the
// state pass works through the previous slice, for long sequences whose state
// pass (one CTA per SM) leaves at least half of the SMs free.  (At a few
// thousand tokens the prep on the remaining SMs takes longer than the state
// pass saves: 0.56 against 0.49 ms at 8192 tokens and 32 heads.)  The state pass is
// launched on a high-priority stream, but a prep slice launched first would
// still take every SM; so the preps that run beside it draw their items from
// a counter, and their CTAs that land on the SMs kept for the state pass (the
// ones with the lowest ids) leave at once.  The whole call is bound by the
// prep, which runs 1.7x slower per item beside the state pass than on the
// whole GPU; so the first slice, prepared on the whole GPU, is made as large
// as lets the prep of the rest (beside the state pass) still end about when
// the state pass has caught up with it.  Per device: the state-pass stream, a
// pool of events and the sorted SM ids, found on first use and kept for the
// life of the process.
constexpr int kMaxSlices = 16;
// cycles of one chunk step of the state pass (64 columns) and of one (chunk,
// head) item of the prep per SM beside it (two CTAs share an SM), measured on
// GB300 at 1M tokens x 32 heads
constexpr double kChainStepCycles = 3.56e3;
constexpr double kPrepItemSmCycles = 17.0e3;
static_assert(kMaxSlices <= kSliceWords, "one item counter per prep slice");
constexpr int kSliceChunks = 16;                 // fewest chunks in a slice
constexpr int kOverlapMinChunks = 1024;          // "long": chunks of the longest sequence
constexpr int kMaxDevices = 64;
constexpr int kMaxSmIds = 256;
struct OverlapRes {
    cudaStream_t chain = nullptr;
    cudaEvent_t ev[kMaxSlices + 2] = {};
    int n_ids = 0;                               // SM ids seen (0: not known)
    int ids[kMaxSmIds] = {};                     // ... sorted
    bool ok = false;
};

// One bit per SM id that a CTA ran on; the CTAs stay resident for ~10 us so
// that they spread over every SM.
__global__ void kda_sm_ids(unsigned int* mask) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    if (threadIdx.x == 0 && smid < kMaxSmIds) atomicOr(mask + (smid >> 5), 1u << (smid & 31));
    const long long t0 = clock64();
    while (clock64() - t0 < 20000) {
    }
}

// SM-id bound below which `count` SMs lie (the ids need not be contiguous);
// with the ids not known, `count` itself.
int reserve_bound(const OverlapRes& r, long long count) {
    if (count <= 0) return 0;
    if (r.n_ids < count) return (int)count;
    return r.ids[count - 1] + 1;
}

// Finds the device's SM ids once (not while the stream is being captured),
// using 32 bytes of the caller's workspace.
cudaError_t probe_sm_ids(OverlapRes& r, int n_sm, void* scratch, cudaStream_t st) {
    if (r.n_ids > 0) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess || cs != cudaStreamCaptureStatusNone) return e;
    unsigned int* mask = static_cast<unsigned int*>(scratch);
    if ((e = cudaMemsetAsync(mask, 0, kMaxSmIds / 8, st)) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_sm_ids, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
    if (e != cudaSuccess) return e;
    kda_sm_ids<<<4 * n_sm, 32, 100 * 1024, st>>>(mask);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    unsigned int h[kMaxSmIds / 32];
    if ((e = cudaMemcpyAsync(h, mask, sizeof(h), cudaMemcpyDeviceToHost, st)) != cudaSuccess) return e;
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return e;
    int n = 0;
    for (int i = 0; i < kMaxSmIds; ++i)
        if (h[i >> 5] >> (i & 31) & 1u) r.ids[n++] = i;
    r.n_ids = n;
    return cudaSuccess;
}
std::mutex g_overlap_mutex;
OverlapRes g_overlap[kMaxDevices];

cudaError_t overlap_resources(OverlapRes** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorNotSupported;
    OverlapRes& r = g_overlap[dev];
    if (!r.ok) {
        int lo = 0, hi = 0;
        e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
        if (e != cudaSuccess) return e;
        e = cudaStreamCreateWithPriority(&r.chain, cudaStreamNonBlocking, hi);
        if (e != cudaSuccess) return e;
        for (auto& ev : r.ev) {
            e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        r.ok = true;
    }
    *out = &r;
    return cudaSuccess;
}

}  // namespace

namespace kda_host {

bool tc_supported(int dk, int dv, int chunk, kda_dtype dt) {
    return dt == KDA_BF16 && dk == DK && dv == DV && chunk == C;
}

size_t tc_workspace_bytes(int n_seq, int T_total, int H, int chunk) {
    (void)chunk;
    const long long ub = slot_bound(n_seq, T_total);
    const SegPlan sp = seg_plan(n_seq, H);
    return header_bytes(n_seq, ub) + state_bytes(n_seq, H) + (size_t)ub * H * WS_BLOCK + seg_table_bytes(sp, n_seq) +
           seg_state_bytes(sp, H);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a) {
    if (a.n_seq == 0) return cudaSuccess;
    const long long ub = slot_bound(a.n_seq, a.T_total);
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    int4* chunk_info = reinterpret_cast<int4*>(ws);
    int4* seq_info = reinterpret_cast<int4*>(ws + 16 * (size_t)ub);
    // item counters of the prep slices that run beside the state pass
    unsigned long long* slice_ctr = reinterpret_cast<unsigned long long*>(ws + 16 * (size_t)ub + 16 * (size_t)a.n_seq);
    int* seq_order = reinterpret_cast<int*>(ws + 16 * (size_t)ub + 16 * (size_t)a.n_seq + 8 * kSliceWords);
    float* S_mid = reinterpret_cast<float*>(ws + header_bytes(a.n_seq, ub));
    uint8_t* blocks = ws + header_bytes(a.n_seq, ub) + state_bytes(a.n_seq, a.H);

    // Equal-length batches map chunks to sequences arithmetically; packed
    // varlen batches go through the chunk table built on the device.
    const int use_table = a.cu_seqlens != nullptr;
    const int fixed_len = use_table ? 0 : a.T_total / a.n_seq;
    const int nch_per = use_table ? 0 : (fixed_len + C - 1) / C;
    // longest sequence in chunks (the device-only cu_seqlens case is not sliced)
    const int max_chunks = use_table ? (a.max_chunks > 0 ? a.max_chunks : (int)min(ub, (long long)INT32_MAX))
                                     : nch_per;
    // Overlap only pays when the state pass is the long pole, i.e. when its
    // CTAs leave most SMs to the chunk preps (few sequences x heads).
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess)
        return cudaGetLastError();
    const long long chain_ctas = (long long)NTILES * a.n_seq * a.H;
    // segment scan: few chains, long sequences, no checkpoints
    const SegPlan sp = seg_plan(a.n_seq, a.H);
    const int seg_L = sp.possible ? std::max(kMinSegChunks, (a.total_chunks + sp.s_target - 1) / std::max(1, sp.s_target))
                                  : 0;
    const bool use_seg = sp.possible && a.ckpt_every == 0 && a.total_chunks > 0 && seg_L < max_chunks;
    uint8_t* seg_base = blocks + (size_t)ub * a.H * WS_BLOCK;
    int4* seg_info = reinterpret_cast<int4*>(seg_base);
    int2* seq_seg = reinterpret_cast<int2*>(seg_base + 16u * (size_t)sp.s_max);
    float* seg_B = reinterpret_cast<float*>(seg_base + seg_table_bytes(sp, a.n_seq));
    float* seg_A = seg_B + (size_t)sp.s_max * a.H * DK * DV;
    float* seg_S = seg_A + (size_t)sp.s_max * a.H * DK * DV;
    const bool overlap = !use_seg && chain_ctas * 2 <= n_sm && max_chunks >= kOverlapMinChunks &&
                         !(use_table && a.max_chunks <= 0);
    const int n_slices = overlap ? std::min(kMaxSlices, max_chunks / kSliceChunks) : 1;
    // slice borders (chunk index within a sequence): slice 0 takes the share f
    // for which the state pass's time over all chunks equals the prep's time
    // over the rest on the SMs it leaves, f = 1 - t_chain / t_prep_beside
    // (kept between one slice's and nine tenths); the others split the rest
    auto slice_begin = [&](int k) -> int {
        if (n_slices == 1) return k == 0 ? 0 : max_chunks;
        const double t_chain = kChainStepCycles * max_chunks;
        const double t_side = kPrepItemSmCycles * (double)a.total_chunks * a.H /
                              (double)std::max<long long>(1, n_sm - chain_ctas);
        const double f = std::min(0.9, std::max(1.0 / n_slices, 1.0 - t_chain / std::max(1.0, t_side)));
        const int first = std::min(max_chunks - (n_slices - 1), std::max(1, (int)(f * max_chunks)));
        if (k == 0) return 0;
        const long long rest = max_chunks - first;
        return first + (int)((rest * (k - 1) + (n_slices - 2)) / (n_slices - 1));
    };
    // the state pass over 32-column slices when that still fits one wave of CTAs
    // (one per SM) and runs alone (no segment scan, no prep beside it)
    const bool narrow = !use_seg && n_slices == 1 && 4LL * a.n_seq * a.H <= n_sm;
    // more than one wave of state-pass CTAs over sequences of different
    // lengths: the CTAs of the longest sequences go first (grid y = the
    // sequence's rank by length), so that no long chain starts late
    const bool ordered = use_table && !use_seg && !narrow && n_slices == 1 && chain_ctas > n_sm && a.n_seq > 1 &&
                         a.n_seq <= kMaxOrdered;

    if (use_table) {
        kda_tc_schedule<<<1, kMaxOrdered, 0, a.stream>>>(a.cu_seqlens, a.n_seq, a.T_total, (int)ub, chunk_info,
                                                         seq_info, ordered ? seq_order : nullptr, a.status);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int prep_smem = (int)(K1_BYTES + 1024);
    const int chain_smem = (int)(ChainCfg<64>::BYTES + 1024);
    const int narrow_smem = (int)(ChainCfg<32>::BYTES + 1024);
    auto prep_kernel = a.prologue ? kda_tc_prep<true> : kda_tc_prep<false>;
    cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, prep_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_tc_chain<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, chain_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_tc_chain<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, narrow_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_tc_seg_scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SC_SMEM);
    if (e != cudaSuccess) return e;

    CUtensorMap tm_q, tm_k, tm_v, tm_g, tm_o, tm_o32;
    std::memset(&tm_o, 0, sizeof(tm_o));
    std::memset(&tm_o32, 0, sizeof(tm_o32));
    // full output chunks leave the state pass by tensor stores when O is 16-byte aligned
    const int o_tma = a.T_total > 0 && a.O != nullptr && (reinterpret_cast<uintptr_t>(a.O) & 15) == 0;
    // the segment scan's last pass (one CTA per segment, head and slice) over
    // 32-column slices too when they fit one wave; likewise the last state-pass
    // slice of an overlapped launch (nothing runs beside it)
    const bool seg_narrow = use_seg && 4LL * sp.s_max * a.H <= n_sm;
    const bool last_narrow = n_slices > 1 && 4LL * a.n_seq * a.H <= n_sm;
    if (o_tma && (e = make_output_map(&tm_o, a.O, a.H, a.T_total, 64)) != cudaSuccess) return e;
    if (o_tma && (e = make_output_map(&tm_o32, a.O, a.H, a.T_total, 32)) != cudaSuccess) return e;
    if (a.T_total > 0) {
        if ((e = make_input_map(&tm_q, a.q, 2, a.H, a.T_total, 128, false)) != cudaSuccess) return e;
        if ((e = make_input_map(&tm_k, a.k, 2, a.H, a.T_total, 128, false)) != cudaSuccess) return e;
        if ((e = make_input_map(&tm_v, a.v, 2, a.H, a.T_total, 64, true)) != cudaSuccess) return e;
        if ((e = make_input_map(&tm_g, a.log_alpha, 4, a.H, a.T_total, 128, false)) != cudaSuccess) return e;
    }
    // chunks [j0, j0 + jn) of every sequence; beside a running state pass
    // (reserve > 0) the CTAs draw items from `ctr` and leave the SMs below `reserve`
    auto prep = [&](int j0, int jn, cudaStream_t st, unsigned long long* ctr, int reserve) {
        if (jn <= 0 || a.total_chunks <= 0 || a.T_total <= 0) return cudaSuccess;
        const int gx = use_table ? a.total_chunks : a.n_seq * jn;
        const long long items = (long long)gx * a.H;
        const unsigned grid = (unsigned)std::min<long long>(items + (ctr ? 2LL * n_sm : 0), 2LL * n_sm);
        prep_kernel<<<grid, 256, prep_smem, st>>>(tm_q, tm_k, tm_v, tm_g, a.beta, a.H, use_table, fixed_len,
                                                  nch_per, chunk_info, seq_info, j0, jn, gx, (int)ub, blocks,
                                                  a.status, ctr, reserve);
        return cudaGetLastError();
    };
    auto chain = [&](int c0, int c1, const float* s_in, float* s_out, cudaStream_t st, bool nar) {
        if (nar)
            kda_tc_chain<32><<<dim3(ChainCfg<32>::NTL * a.n_seq, a.H), K2_THREADS, narrow_smem, st>>>(
                seq_info, use_table, fixed_len, nch_per, c0, c1, blocks, s_in, a.H, static_cast<bf16*>(a.O), s_out,
                a.ckpt_every, a.ckpt, a.ckpt_cap, a.status, 0, nullptr, (int)ub, tm_o32, o_tma, nullptr);
        else if (ordered)
            kda_tc_chain<64><<<dim3(NTILES * a.H, a.n_seq), K2_THREADS, chain_smem, st>>>(
                seq_info, use_table, fixed_len, nch_per, c0, c1, blocks, s_in, a.H, static_cast<bf16*>(a.O), s_out,
                a.ckpt_every, a.ckpt, a.ckpt_cap, a.status, 0, nullptr, (int)ub, tm_o, o_tma, seq_order);
        else
            kda_tc_chain<64><<<dim3(NTILES * a.n_seq, a.H), K2_THREADS, chain_smem, st>>>(
                seq_info, use_table, fixed_len, nch_per, c0, c1, blocks, s_in, a.H, static_cast<bf16*>(a.O), s_out,
                a.ckpt_every, a.ckpt, a.ckpt_cap, a.status, 0, nullptr, (int)ub, tm_o, o_tma, nullptr);
        return cudaGetLastError();
    };

    if (use_seg) {
        if ((e = prep(0, max_chunks, a.stream, nullptr, 0)) != cudaSuccess) return e;
        trace_mark(a.stream);
        kda_tc_segments<<<1, 1024, 0, a.stream>>>(seq_info, use_table, fixed_len, nch_per, a.n_seq, seg_L, sp.s_max,
                                                  seg_info, seq_seg, a.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // pass 1: every segment from zero (-> seg_B) and as a map from the identity (-> seg_A)
        kda_tc_chain<64><<<dim3(NTILES * sp.s_max, a.H, 2), K2_THREADS, chain_smem, a.stream>>>(
            seg_info, 1, 0, 0, 0, INT32_MAX, blocks, nullptr, a.H, static_cast<bf16*>(a.O), seg_B, 0, nullptr, 0,
            a.status, 1, seg_A, (int)ub, tm_o, o_tma, nullptr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // pass 2: starting state of every segment, and the final states
        kda_tc_seg_scan<<<dim3(a.n_seq, a.H, DV / SC_COLS), 256, SC_SMEM, a.stream>>>(seq_seg, seg_A, seg_B, a.S0,
                                                                                       seg_S, a.S_final, a.H,
                                                                                       sp.s_max, a.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // pass 3: every segment from its starting state, writing O
        if (seg_narrow)
            kda_tc_chain<32><<<dim3(ChainCfg<32>::NTL * sp.s_max, a.H), K2_THREADS, narrow_smem, a.stream>>>(
                seg_info, 1, 0, 0, 0, INT32_MAX, blocks, seg_S, a.H, static_cast<bf16*>(a.O), nullptr, 0, nullptr, 0,
                a.status, 0, nullptr, (int)ub, tm_o32, o_tma, nullptr);
        else
            kda_tc_chain<64><<<dim3(NTILES * sp.s_max, a.H), K2_THREADS, chain_smem, a.stream>>>(
                seg_info, 1, 0, 0, 0, INT32_MAX, blocks, seg_S, a.H, static_cast<bf16*>(a.O), nullptr, 0, nullptr, 0,
                a.status, 0, nullptr, (int)ub, tm_o, o_tma, nullptr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        trace_mark(a.stream);
        return cudaSuccess;
    }

    if (n_slices == 1) {
        if ((e = prep(0, max_chunks, a.stream, nullptr, 0)) != cudaSuccess) return e;
        trace_mark(a.stream);
        if ((e = chain(0, max_chunks, a.S0, a.S_final, a.stream, narrow)) != cudaSuccess) return e;
        trace_mark(a.stream);
        return cudaSuccess;
    }
    // prep slices on the caller's stream, state-pass slices on the internal
    // stream, slice k of the state pass waiting for slice k of the prep; the
    // state is carried between slices in S_mid; the caller's stream joins at the end.
    std::lock_guard<std::mutex> lock(g_overlap_mutex);
    OverlapRes* r = nullptr;
    if ((e = overlap_resources(&r)) != cudaSuccess) return e;
    if ((e = probe_sm_ids(*r, n_sm, slice_ctr, a.stream)) != cudaSuccess) return e;
    const int reserve = reserve_bound(*r, chain_ctas);
    if ((e = cudaMemsetAsync(slice_ctr, 0, 8u * kMaxSlices, a.stream)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(r->ev[n_slices], a.stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(r->chain, r->ev[n_slices], 0)) != cudaSuccess) return e;
    for (int k = 0; k < n_slices; ++k) {
        const int c0 = slice_begin(k), c1 = k + 1 < n_slices ? slice_begin(k + 1) : max_chunks;
        // the first slice has the GPU to itself; the others run beside the state pass
        if ((e = prep(c0, c1 - c0, a.stream, k > 0 ? slice_ctr + k : nullptr, k > 0 ? reserve : 0)) != cudaSuccess)
            return e;
        if ((e = cudaEventRecord(r->ev[k], a.stream)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(r->chain, r->ev[k], 0)) != cudaSuccess) return e;
        const bool last = (k == n_slices - 1);
        if ((e = chain(c0, c1, k == 0 ? a.S0 : S_mid, last ? a.S_final : S_mid, r->chain, last && last_narrow)) !=
            cudaSuccess)
            return e;
    }
    trace_mark(a.stream);                       // every prep slice enqueued
    if ((e = cudaEventRecord(r->ev[n_slices + 1], r->chain)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(a.stream, r->ev[n_slices + 1], 0)) != cudaSuccess) return e;
    trace_mark(a.stream);
    return cudaSuccess;
}

}  // namespace kda_host
