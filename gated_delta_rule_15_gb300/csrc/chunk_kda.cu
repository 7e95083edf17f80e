// chunk_kda.cu -- chunkwise forward of the gated delta rule with a per-channel gate (KDA),
// bf16 inputs, d_k = d_v = 128, chunk C = 64, on the tensor cores, in two kernels.
//
// With a per-channel gate (page "NLP: linear attention summary", KDA section: S_t =
// (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T, a_t in (0, 1)^{d_k}) the decay no
// longer factors out of the chunk's k.k and q.k products, so every operand that meets the
// state carries its own per-channel scaling.  With g_r = sum_{u <= r} log a_u (a d_k-vector),
// G_r = exp(g_r) and the chunk form of chunk_simt.cu:
//
//   A_rs = b_r sum_c k_rc k_sc exp(g_rc - g_sc)  (s < r),   P_rs = sum_c q_rc k_sc exp(...)
//   T = (I + A)^-1,  U = T diag(b) V,  W = T diag(b) (K*G),  E = U - W S
//   S <- Diag(G_C) S + (K * G_C/G)^T E,   O = (Q*G) S + P E
//
// kda_prep_kernel (one CTA per (b, h, chunk), all chunks in parallel) computes everything
// that does not depend on S and stores it, ready for the tensor core, in the workspace:
// W (bf16), U (fp32), Q*G (a bf16 high/low pair), P and (K*G_C/G)^T (TF32-rounded fp32, the
// B operands of two kind::tf32 products) and G_C.  The exponentials
// inside A and P are split per 16-token block j of the column index s, against the
// reference g_ref = g at the block's last token: exp(g_ref - g_s) <= 1 for s in the block and
// exp(g_r - g_ref) <= 1 for every row r below it, so the off-diagonal blocks take no factor
// above one whatever the decay strength (the log-space, two-level remedy that the page
// "Transformer notes (5): linear attention optimisations" names for this gate).  Inside the
// diagonal blocks exp(g_r - g_ref) is bounded by the block's own decay; a chunk where some
// channel decays by more than exp(64) inside one block recomputes those entries on the CUDA
// cores instead.  The four blocks are four tcgen05 products [Q; K]_j R_j^T (M = 128,
// N = 16) on high/low bf16 pairs.
//
// kda_state_kernel (one CTA per (b, h), chunks in sequence) keeps S^T in TMEM and, per
// chunk, TMA-loads the stored operands: D = S^T [W; Q*G]^T, E^T = U^T - (W S)^T (fp32 in
// TMEM, the A operand of the next two products), S^T <- S^T Diag(G_C) + E^T (K*G_C/G) and
// O^T = (Q*G S)^T + E^T P^T as kind::tf32 products, with the operand buffers of the next
// chunk refilled as soon as each is consumed.
//
// Fused neighbours (DR_FUSE_* of include/dr.h; page "linear-attention gated-deltanet
// guide", section 4): the prep kernel computes 1 / |q_r| and 1 / |k_r| from the bf16 tiles
// (threads 128..255, while threads 0..127 scan the gates) and scales every q and k value
// as it converts it to fp32, so all the stored operands are those of the normalised rows;
// it takes beta = sigmoid(logit) rounded to bf16 (beta's storage dtype).  The state kernel
// multiplies each output by silu(z), z's tile arriving by TMA one chunk ahead.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "chunk_layout.h"
#include "common.cuh"
#include "tc_common.cuh"
#include "umma.cuh"

namespace dr {
namespace {

using namespace umma;
using namespace tc;

constexpr int kThreads = 256;

// ---------------------------------------------------------------- workspace (per chunk n)
// W [64][128] bf16, U [64][128] fp32, P [64][64] fp32 (TF32-rounded), QH/QL [64][128] bf16,
// KT = (K*G_C/G)^T [128][64] fp32 (TF32-rounded), GAM [128]
struct KdaWorkspace {
    __nv_bfloat16 *W, *QH, *QL;
    float *U, *P, *KT, *GAM;
};
constexpr size_t kKdaBytesPerChunk = 16384 + 32768 + 2 * 8192 + 4 * 16384 + 512;

KdaWorkspace kda_carve(void *base, int64_t nch) {
    char *p = (char *)base;
    KdaWorkspace w;
    w.W = (__nv_bfloat16 *)p;   p += nch * 16384;
    w.U = (float *)p;           p += nch * 32768;
    w.P = (float *)p;           p += nch * 16384;
    w.QH = (__nv_bfloat16 *)p;  p += nch * 16384;
    w.QL = (__nv_bfloat16 *)p;  p += nch * 16384;
    w.KT = (float *)p;          p += nch * 32768;
    w.GAM = (float *)p;
    return w;
}

// ---------------------------------------------------------------- prep kernel layout
// Sized for two CTAs per SM (<= 113 KB each): the left factors of the intra-chunk products
// live in tensor memory (A operand of tcgen05.mma), the right factors in shared memory.
constexpr uint32_t P1_Q = 0, P1_K = 16384;    // 64 x 128 bf16 tiles, 2 K-blocks, 128B swizzle
constexpr uint32_t P1_LA = 32768;   // log alpha -> g log2(e): 4 boxes [64][32] fp32, 128B swizzle
constexpr uint32_t P1_V = 65536, P1_KG = 81920;
constexpr uint32_t P1_R = 98304;              // right factors: high [kb][16][64], low at +4096
constexpr uint32_t P1_SMALL = 106496;         // beta[64], solve scratch[1024]
constexpr uint32_t P1_TOTAL = P1_SMALL + 256 + 4096 + 512 + 512;   // + G_C[128], row norms[128]
// after the products: A over Q, T over K (and the first KB of g), T diag(beta) inside g,
// the exact diagonal blocks over the right factors; staging of W and U at the end
constexpr uint32_t P1_A = 0, P1_T = 16384, P1_TB = 34816, P1_XD = P1_R;
constexpr uint32_t P1_WST = 0, P1_UST = 16384;
// one-product chunks: the right factor as a K-major tf32 B operand (64 token rows, four
// 8 KB blocks of 32 channels) over V and K*G
constexpr uint32_t P1_R1 = P1_V;
// tensor memory: X = [Q; K] R^T (64 columns), the left factor (one product: fp32, 128
// columns; four rounds: high and low bf16 halves); U^T, W^T afterwards
constexpr uint32_t P1_TM_X = 0, P1_TM_LH = 128, P1_TM_LL = 192, P1_TM_U = 128, P1_TM_W = 192;
// (one-product chunks) the left factor as fp32, the tf32 A operand: 128 columns
constexpr uint32_t P1_TM_L1 = 128;
static_assert(P1_T + 64 * kTs * 4 <= P1_TB && P1_TB + 8192 <= P1_V, "prep layout");
static_assert(P1_UST + 32768 <= P1_V && P1_TOTAL + 1024 <= 113 * 1024, "prep layout");

constexpr uint32_t ID_KK_N16 = idesc_bf16(128, 16, false, false);
constexpr uint32_t ID_TF_N128 = idesc_tf32(128, 128);
constexpr uint32_t ID_TF_N64 = idesc_tf32(128, 64);
constexpr uint32_t ID_KK_N64 = idesc_bf16(128, 64, false, false);
// Largest per-channel decay (natural log) inside one 16-token block that the tensor-core
// products of the diagonal blocks take; beyond it the chunk recomputes those entries.
constexpr float kDiagLimit = 64.f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kDiagLimit2 = kDiagLimit * kLog2e;   // the same bound in base-2 units

// 2^x (PTX ex2.approx.ftz: relative error about 2^-22; results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr uint32_t ID_MK_N64 = idesc_bf16(128, 64, true, false);

struct PrepArgs {
    const __nv_bfloat16 *beta;
    KdaWorkspace ws;
    int *status;
    int T, H, NC;
    uint32_t fuse;   // DR_FUSE_* bits
};

// Float index of element (t, c) of the [64][128] fp32 tile held as four 128-byte-swizzled
// [64][32] boxes: 16-byte groups of a row permuted by t % 8.
__device__ __forceinline__ int la_idx(int t, int c) {
    return (c >> 5) * 2048 + t * 32 + ((((c & 31) >> 2) ^ (t & 7)) << 2) + (c & 3);
}
// Eight consecutive bf16 values (columns 8 c8 .. 8 c8 + 7) of row r of a swizzled tile.
__device__ __forceinline__ void load8_bf16(const unsigned char *tile, int r, int c8, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(tile + (c8 >> 3) * 8192 + sw128_off(r, (8 * c8) & 63));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
// g at token t, channels c .. c + 7 (c a multiple of 8).
__device__ __forceinline__ void load8_g(const float *LA, int t, int c, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(LA + la_idx(t, c));
    const float4 b = *reinterpret_cast<const float4 *>(LA + la_idx(t, c + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__global__ void __launch_bounds__(kThreads, 2)
kda_prep_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tla,
                const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
                const PrepArgs a) {
    extern __shared__ unsigned char dsm_raw[];
    unsigned char *sm = align1024(dsm_raw);
    __shared__ uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s, diag_exact_s, four_rounds_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;   // TMEM lane: row of [Q; K], or channel
    const int64_t n = blockIdx.x;
    const int c = (int)(n % a.NC);
    const int64_t bh = n / a.NC;
    const int h = (int)(bh % a.H), b = (int)(bh / a.H);
    const int t0 = c * 64;
    const int Lc = min(64, a.T - t0);
    float *sBeta = reinterpret_cast<float *>(sm + P1_SMALL);
    float *sM = sBeta + 64;
    float *sGamC = sM + 1024;   // G_C per channel
    float *sInv = sGamC + 128;  // 1 / |x| of the rows of [Q; K] (1 unless normalised)
    float *LA = reinterpret_cast<float *>(sm + P1_LA);
    float *const Xd = reinterpret_cast<float *>(sm + P1_XD);   // exact diagonal blocks
    const int t_row = row & 63, blk = t_row >> 4;   // this thread's row of [Q; K]: token, block
    const bool qrow = quarter < 2;
    const unsigned char *xt = sm + (qrow ? P1_Q : P1_K);
    float *const sF = reinterpret_cast<float *>(sm + P1_V);        // [8][128] block factors
    float *const sExpRef = sF + 8 * 128;                           // [4][128] exp(ref_i)
    bool diag_exact = false;
    float rinv = 1.f;   // 1 / |x| of this thread's row of [Q; K] (after the norms)

    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        abort_s = 0;
        diag_exact_s = 0;
        four_rounds_s = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmb = tmem_base_s;
    const uint32_t tm = tmb + ((uint32_t)(32 * quarter) << 16);
    uint32_t mma_phase = 0;
    // operand descriptors of the shared-memory base: K-major and MN-major (two 64-wide atoms)
    const uint64_t dK0 = smem_desc_sw128(smem_u32(sm), 16, 1024), dM0 = smem_desc_sw128(smem_u32(sm), 8192, 1024);
    auto fail = [&]() {
        abort_s = 1;
        atomicExch(a.status, kErrTimeout);
    };

    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_ld, 32768 + 32768);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sm + P1_Q + kb * 8192, &tq, &bar_ld, 64 * kb, h, t0, b);
            tma_load_4d(sm + P1_K + kb * 8192, &tk, &bar_ld, 64 * kb, h, t0, b);
        }
        for (int bx = 0; bx < 4; ++bx)
            tma_load_4d(sm + P1_LA + bx * 8192, &tla, &bar_ld, 32 * bx, h, t0, b);
    }
    if (tid < 64) {
        float bt = tid < Lc ? __bfloat162float(a.beta[((size_t)b * a.T + t0 + tid) * a.H + h]) : 0.f;
        if ((a.fuse & kFuseSigmoid) && tid < Lc) bt = round_bf16(sigmoid_f(bt));
        sBeta[tid] = bt;
    }
    if (!wait_cycles(&bar_ld, 0)) fail();
    __syncthreads();
    if (abort_s) goto done;

    // ---- cumulative log decay g (in place, stored as g log2(e) so that every factor below
    //      is one ex2; one channel per thread, held in registers),
    //      G_C = exp(g_63); flag the chunk if a channel decays by more than kDiagLimit
    //      inside one 16-token block.  With ref_i = g at the last token of block i, the
    //      per-channel factors exp(ref_i) and F_ij = exp(ref_i - ref_j) (i > j, both <= 1)
    //      go to the V buffer, which is loaded only after the products.
    if (tid < 128) {
        float v[64];
#pragma unroll
        for (int t = 0; t < 64; ++t) v[t] = LA[la_idx(t, tid)];
#pragma unroll
        for (int t = 1; t < 64; ++t) v[t] += v[t - 1];
#pragma unroll
        for (int t = 0; t < 64; ++t) LA[la_idx(t, tid)] = v[t] * kLog2e;   // g in base-2 units
        bool steep = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) steep |= v[16 * j] - v[16 * j + 15] > kDiagLimit;
        if (steep) diag_exact_s = 1;
        if (v[0] - v[63] > kDiagLimit) four_rounds_s = 1;
        const float gc = __expf(v[63]);
        a.ws.GAM[n * 128 + tid] = gc;
        sGamC[tid] = gc;
#pragma unroll
        for (int i = 0; i < 4; ++i) sExpRef[i * 128 + tid] = __expf(v[16 * i + 15]);
#pragma unroll
        for (int i = 1; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < i; ++j)
                sF[(i * (i - 1) / 2 + j) * 128 + tid] = __expf(v[16 * i + 15] - v[16 * j + 15]);
        sF[6 * 128 + tid] = 1.f;   // same block
        sF[7 * 128 + tid] = 0.f;   // row above the column block (entry masked)
    } else {
        // row norms of [Q; K] (thread 128 + i: row i; a quarter-warp's 16-byte loads of one
        // logical group fall in eight different bank groups)
        const int i = tid - 128;
        float inv = 1.f;
        if (a.fuse & kFuseL2) {
            const unsigned char *src = sm + (i < 64 ? P1_Q : P1_K) + (i & 63) * 128;
            float ss = 0.f;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(src + kb * 8192 + 16 * (j ^ (i & 7)));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
                        ss = fmaf(f.x, f.x, ss);
                        ss = fmaf(f.y, f.y, ss);
                    }
                }
            inv = rsqrtf(ss + kL2NormEps);
        }
        sInv[i] = inv;
    }
    __syncthreads();
    diag_exact = diag_exact_s != 0;
    rinv = sInv[row];

    if (!four_rounds_s) {
        // ---- one product for the whole chunk against ref = g_63 (no channel decays by more
        //      than kDiagLimit across the chunk): left factor xE_t = x_t exp(g_t - g_63) in
        //      [|x|, |x| e^kDiagLimit] (tensor memory), right factor k_s exp(g_63 - g_s) =
        //      (K*G_C/G)_s <= |k_s| (shared memory, and the workspace's transposed copy), both
        //      TF32-rounded fp32 for one kind::tf32 product.  Q rows also write Q*G = xE G_C;
        //      K rows keep K*G = xE G_C for the W operand.
        uint32_t kg_keep[32];
        {
            const size_t go = ((size_t)n * 64 + t_row) * 128 + 64 * half;
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                float lf[32];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = 64 * half + 32 * p + 8 * i, w = 4 * (4 * p + i);
                    float x8[8], g8[8], gl[8], e8[8];
                    load8_bf16(xt, t_row, c >> 3, x8);
#pragma unroll
                    for (int u = 0; u < 8; ++u) x8[u] *= rinv;
                    load8_g(LA, t_row, c, g8);
                    load8_g(LA, 63, c, gl);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        e8[u] = x8[u] * ex2(g8[u] - gl[u]);
                        lf[8 * i + u] = round_tf32(e8[u]);
                    }
                    uint32_t oh[4], ol[4];
                    if (qrow) {
#pragma unroll
                        for (int u = 0; u < 8; u += 2)
                            pack_hi_lo(e8[u] * sGamC[c + u], e8[u + 1] * sGamC[c + u + 1], oh[u >> 1], ol[u >> 1]);
                        *reinterpret_cast<uint4 *>(a.ws.QH + go + 32 * p + 8 * i) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
                        *reinterpret_cast<uint4 *>(a.ws.QL + go + 32 * p + 8 * i) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
                    } else {
                        float kt[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) kt[u] = x8[u] * ex2(gl[u] - g8[u]);
#pragma unroll
                        for (int u = 0; u < 8; u += 2)
                            kg_keep[w + (u >> 1)] = pack_bf16(e8[u] * sGamC[c + u], e8[u + 1] * sGamC[c + u + 1]);
#pragma unroll
                        for (int u = 0; u < 8; ++u) kt[u] = round_tf32(kt[u]);
                        // the right factor, row t_row of a K-major tf32 tile (32 channels per
                        // 128-byte row, four channel blocks 8 KB apart)
                        const uint32_t sb = P1_R1 + (c >> 5) * 8192;
                        *reinterpret_cast<float4 *>(sm + sb + sw128_off32(t_row, c & 31)) =
                            make_float4(kt[0], kt[1], kt[2], kt[3]);
                        *reinterpret_cast<float4 *>(sm + sb + sw128_off32(t_row, (c & 31) + 4)) =
                            make_float4(kt[4], kt[5], kt[6], kt[7]);
                        // row c + u of K*G_C/G transposed (a warp's 32 tokens: 128 contiguous bytes)
#pragma unroll
                        for (int u = 0; u < 8; ++u) a.ws.KT[(n * 128 + c + u) * 64 + t_row] = kt[u];
                    }
                }
                tmem_st32(tm + P1_TM_L1 + 64 * half + 32 * p, lf);
            }
            tmem_wait_st();
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // X = L R^T: one N = 64 kind::tf32 product over the 128 channels
#pragma unroll
            for (int ks = 0; ks < 16; ++ks)
                mma_tf32_ts(tmb + P1_TM_X, tmb + P1_TM_L1 + 8 * ks,
                            desc_add(dK0, P1_R1 + (ks >> 2) * 8192 + (ks & 3) * 32), ID_TF_N64, ks > 0);
            mma_commit(&bar_mma);
        }
        if (!wait_cycles(&bar_mma, mma_phase)) fail();
        mma_phase ^= 1;
        tc_fence_after();
        __syncthreads();   // the right factors are dead: K*G takes their place
        if (!qrow) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = 64 * half + 8 * i;
                *reinterpret_cast<uint4 *>(sm + P1_KG + (c >> 6) * 8192 + sw128_off(t_row, c & 63)) =
                    make_uint4(kg_keep[4 * i], kg_keep[4 * i + 1], kg_keep[4 * i + 2], kg_keep[4 * i + 3]);
            }
        }
        if (abort_s) goto done;
    } else {
        // ---- per row (this thread: row t of Q or K, channels 64 half .. 64 half + 63):
        //      xE_c = x_tc exp(g_tc - ref_i(t)) in [|x|, |x| e^kDiagLimit], kept in registers for
        //      the products below; Q rows write Q*G = xE exp(ref_i) (pair) to the workspace, K rows
        //      write K*G = xE exp(ref_i) (the W operand) and K*G_C/G = k exp(g_63 - g_t) (pair).
        //      A flagged chunk takes every factor directly from its own exponent instead.
        float xE[64];
        {
            const size_t go = ((size_t)n * 64 + t_row) * 128 + 64 * half;
    #pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = 64 * half + 8 * i;
                float x8[8], g8[8], r8[8], e8[8];
                load8_bf16(xt, t_row, c >> 3, x8);
    #pragma unroll
                for (int u = 0; u < 8; ++u) x8[u] *= rinv;
                load8_g(LA, t_row, c, g8);
                load8_g(LA, 16 * blk + 15, c, r8);
    #pragma unroll
                for (int u = 0; u < 8; ++u) {
                    xE[8 * i + u] = x8[u] * ex2(fminf(g8[u] - r8[u], kDiagLimit2));
                    e8[u] = diag_exact ? x8[u] * ex2(g8[u]) : xE[8 * i + u] * sExpRef[blk * 128 + c + u];
                }
                if (qrow) {
                    uint32_t hi[4], lo[4];
    #pragma unroll
                    for (int u = 0; u < 8; u += 2) pack_hi_lo(e8[u], e8[u + 1], hi[u >> 1], lo[u >> 1]);
                    *reinterpret_cast<uint4 *>(a.ws.QH + go + 8 * i) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(a.ws.QL + go + 8 * i) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                } else {
                    float gl[8];
                    load8_g(LA, 63, c, gl);
                    uint32_t kg[4];
    #pragma unroll
                    for (int u = 0; u < 8; u += 2) kg[u >> 1] = pack_bf16(e8[u], e8[u + 1]);
                    *reinterpret_cast<uint4 *>(sm + P1_KG + (c >> 6) * 8192 + sw128_off(t_row, c & 63)) =
                        make_uint4(kg[0], kg[1], kg[2], kg[3]);
    #pragma unroll
                    for (int u = 0; u < 8; ++u)
                        a.ws.KT[(n * 128 + c + u) * 64 + t_row] = round_tf32(x8[u] * ex2(gl[u] - g8[u]));
                }
            }
        }

        // ---- X = [Q; K] K^T with per-channel decays, by column block j (tokens 16 j .. 16 j + 15),
        //      against ref_j: the right factor k_s exp(ref_j - g_s) (shared memory) is <= |k_s|;
        //      the left factor x_t exp(g_t - ref_j) = xE_t F_{i(t) j} (tensor memory, one [Q; K]
        //      row per lane, 64 channels per warp) is <= |x_t| below the block and at most
        //      |x_t| e^kDiagLimit inside it (a flagged chunk clamps it there, takes it directly
        //      from its exponent, and recomputes the diagonal blocks below).  Rows above the
        //      block get zeros: their entries are masked.
        for (int j = 0; j < 4; ++j) {
            const int ref = 16 * j + 15;
            {
                const int rr = tid >> 4, c8 = tid & 15, s = 16 * j + rr;
                float k8[8], g8[8], rf[8];
                load8_bf16(sm + P1_K, s, c8, k8);
                const float ks = sInv[64 + s];
    #pragma unroll
                for (int u = 0; u < 8; ++u) k8[u] *= ks;
                load8_g(LA, s, 8 * c8, g8);
                load8_g(LA, ref, 8 * c8, rf);
                uint32_t hi[4], lo[4];
    #pragma unroll
                for (int u = 0; u < 8; u += 2)
                    pack_hi_lo(k8[u] * ex2(rf[u] - g8[u]), k8[u + 1] * ex2(rf[u + 1] - g8[u + 1]),
                               hi[u >> 1], lo[u >> 1]);
                const uint32_t off = (c8 >> 3) * 2048 + sw128_off(rr, (8 * c8) & 63);
                *reinterpret_cast<uint4 *>(sm + P1_R + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(sm + P1_R + 4096 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            if ((quarter & 1) || j < 2) {   // some row of this warp is at or below the block
                const int fr = blk < j ? 7 : (blk == j ? 6 : blk * (blk - 1) / 2 + j);
                const float *Fr = sF + fr * 128;
    #pragma unroll
                for (int p = 0; p < 2; ++p) {
                    uint32_t hi[16], lo[16];
    #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int cl = 32 * p + 8 * i, c = 64 * half + cl;
                        float f8[8];
                        if (!diag_exact) {
                            const float4 f0 = *reinterpret_cast<const float4 *>(Fr + c);
                            const float4 f1 = *reinterpret_cast<const float4 *>(Fr + c + 4);
                            f8[0] = xE[cl] * f0.x;     f8[1] = xE[cl + 1] * f0.y;
                            f8[2] = xE[cl + 2] * f0.z; f8[3] = xE[cl + 3] * f0.w;
                            f8[4] = xE[cl + 4] * f1.x; f8[5] = xE[cl + 5] * f1.y;
                            f8[6] = xE[cl + 6] * f1.z; f8[7] = xE[cl + 7] * f1.w;
                        } else {
                            float x8[8], g8[8], r8[8];
                            load8_bf16(xt, t_row, c >> 3, x8);
    #pragma unroll
                            for (int u = 0; u < 8; ++u) x8[u] *= rinv;
                            load8_g(LA, t_row, c, g8);
                            load8_g(LA, ref, c, r8);
    #pragma unroll
                            for (int u = 0; u < 8; ++u)
                                f8[u] = blk < j ? 0.f : x8[u] * ex2(fminf(g8[u] - r8[u], kDiagLimit2));
                        }
    #pragma unroll
                        for (int u = 0; u < 8; u += 2)
                            pack_hi_lo(f8[u], f8[u + 1], hi[4 * i + (u >> 1)], lo[4 * i + (u >> 1)]);
                    }
                    tmem_st16u(tm + P1_TM_LH + 32 * half + 16 * p, hi);
                    tmem_st16u(tm + P1_TM_LL + 32 * half + 16 * p, lo);
                }
                tmem_wait_st();
            }
            fence_proxy_async();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
    #pragma unroll
                for (int part = 0; part < 3; ++part)
    #pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ts(tmb + P1_TM_X + 16 * j, tmb + (part == 2 ? P1_TM_LL : P1_TM_LH) + 8 * ks,
                                    desc_add(dK0, P1_R + (part == 1 ? 4096 : 0) +
                                                             (ks >> 2) * 2048 + (ks & 3) * 32),
                                    ID_KK_N16, (part | ks) != 0);
                mma_commit(&bar_mma);
            }
            if (!wait_cycles(&bar_mma, mma_phase)) fail();
            mma_phase ^= 1;
            tc_fence_after();
            __syncthreads();
            if (abort_s) goto done;
        }
    }
    if (tid == 0) {   // the factors in the V buffer are dead: load V (U operand)
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar_ld, 16384);
        for (int kb = 0; kb < 2; ++kb) tma_load_4d(sm + P1_V + kb * 8192, &tv, &bar_ld, 64 * kb, h, t0, b);
    }

    // ---- flagged chunk: entries of the four diagonal 16 x 16 blocks in fp32, one exponential
    //      per channel, into Xd[2][64][16] (rows of P, then rows of A before beta)
    if (diag_exact) {
        for (int task = tid; task < 2 * 64 * 16; task += kThreads) {
            const int part = task >> 10, r = (task >> 4) & 63, s = (r & ~15) + (task & 15);
            const unsigned char *xs = sm + (part ? P1_K : P1_Q);
            float acc = 0.f;
            if (s <= r)
                for (int ch = 0; ch < 128; ++ch) {
                    const uint32_t o = (ch >> 6) * 8192;
                    const float xr = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16 *>(xs + o + sw128_off(r, ch & 63)));
                    const float ks = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16 *>(sm + P1_K + o + sw128_off(s, ch & 63)));
                    acc = fmaf(xr * ks, ex2(LA[la_idx(r, ch)] - LA[la_idx(s, ch)]), acc);
                }
            Xd[task] = acc * sInv[part * 64 + r] * sInv[64 + s];
        }
    }
    __syncthreads();   // Q, K and g are dead from here on

    // ---- P (rows 0..63 of X) to the workspace, TF32-rounded; A (rows 64..127) in fp32
    {
        float x[32];
        tmem_ld32(tm + P1_TM_X + 32 * half, x);
        tmem_wait_ld();
        const int c0 = 32 * half;
        if (diag_exact) {
            const int part = quarter >> 1, r = row & 63;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                if (((c0 + u) >> 4) == (r >> 4)) x[u] = Xd[part * 1024 + r * 16 + ((c0 + u) & 15)];
        }
        if (quarter < 2) {   // P row r, TF32-rounded, zero above the diagonal
            const int r = row;
            float4 *dp = reinterpret_cast<float4 *>(a.ws.P + (n * 64 + r) * 64 + c0);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = c0 + 4 * q4 + e <= r ? round_tf32(x[4 * q4 + e]) : 0.f;
                dp[q4] = make_float4(v[0], v[1], v[2], v[3]);
            }
        } else {
            const int r = row - 64;
            const float br = sBeta[r];
            float *sA = reinterpret_cast<float *>(sm + P1_A);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const int s0 = c0 + 4 * q4;
                float4 v4;
                v4.x = s0 < r ? br * x[4 * q4] : 0.f;
                v4.y = s0 + 1 < r ? br * x[4 * q4 + 1] : 0.f;
                v4.z = s0 + 2 < r ? br * x[4 * q4 + 2] : 0.f;
                v4.w = s0 + 3 < r ? br * x[4 * q4 + 3] : 0.f;
                *reinterpret_cast<float4 *>(sA + a_index(r, s0)) = v4;
            }
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---- T = (I + A)^-1 and its bf16 operand T diag(beta)
    solve_unit_lower64<false>(reinterpret_cast<const float *>(sm + P1_A), reinterpret_cast<float *>(sm + P1_T),
                              sM, sm + P1_TB, sBeta, nullptr, tid);

    // ---- U^T = V^T (T diag beta)^T,  W^T = (K*G)^T (T diag beta)^T
    if (tid == 0) {
        if (!wait_cycles(&bar_ld, 1)) fail();
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmb + P1_TM_U, desc_add(dM0, P1_V + ks * 2048),
                     desc_add(dK0, P1_TB + ks * 32), ID_MK_N64, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmb + P1_TM_W, desc_add(dM0, P1_KG + ks * 2048),
                     desc_add(dK0, P1_TB + ks * 32), ID_MK_N64, ks > 0);
        mma_commit(&bar_mma);
    }
    if (!wait_cycles(&bar_mma, mma_phase)) fail();
    tc_fence_after();
    // ---- W (bf16) and U (fp32) staged row-major (lane = channel, column = token) and
    //      written by TMA
    {
        float w[32], u32[32];
        tmem_ld32(tm + P1_TM_W + 32 * half, w);
        tmem_ld32(tm + P1_TM_U + 32 * half, u32);
        tmem_wait_ld();
        const int j = row;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int r = 32 * half + u;
            *reinterpret_cast<__nv_bfloat16 *>(sm + P1_WST + (j >> 6) * 8192 + sw128_off(r, j & 63)) =
                __float2bfloat16_rn(w[u]);
            *reinterpret_cast<float *>(sm + P1_UST + (j >> 5) * 8192 + r * 128 + (j & 31) * 4) = u32[u];
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
        const int y = (int)(n * 64);
        tma_store_2d(&mw, sm + P1_WST, 0, y);
        tma_store_2d(&mw, sm + P1_WST + 8192, 64, y);
#pragma unroll
        for (int bx = 0; bx < 4; ++bx) tma_store_2d(&mu, sm + P1_UST + bx * 8192, 32 * bx, y);
        bulk_commit();
        bulk_wait_read_all();
    }
done:
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmb, 256);
}

// ---------------------------------------------------------------- state kernel layout
// [W; Q*G high; Q*G low] as one 192-row K-major B operand: per K-block of 64 channels
// [W (8 KB) | QH (8 KB) | QL (8 KB)], the two K-blocks 24 KB apart
constexpr uint32_t S2_WQ = 0, S2_WQ_KB = 24576;
constexpr uint32_t S2_KT = 49152;   // (K*G_C/G)^T, tf32 K-major: [2 token blocks][128 ch][32 tok]
constexpr uint32_t S2_P = 81920;    // 2 buffers of P, tf32 K-major: [2 token blocks][64][32]
constexpr uint32_t S2_U = 114688;                            // [64][128] fp32, 4 boxes of 32
constexpr uint32_t S2_ST = 147456;                           // S^T bf16 [128][128]; output staging
constexpr uint32_t S2_SMALL = 212992;                        // G_C of two chunks
constexpr uint32_t S2_TOTAL = S2_SMALL + 1024;
constexpr uint32_t S2_Z = S2_TOTAL;                          // output gate: z tile [64][128] bf16
constexpr uint32_t S2_TOTAL_Z = S2_Z + 16384;
static_assert(S2_TOTAL_Z + 1024 <= 227 * 1024, "state layout");
// tensor memory: S^T, then two buffers of [(W S)^T, then E^T | (QH S)^T + E^T P^T | (QL S)^T]
constexpr uint32_t S2_TM_S = 0, S2_TM_D = 128, S2_TM_DSTRIDE = 192;

constexpr uint32_t ID_KK_N192 = idesc_bf16(128, 192, false, false);

struct StateArgs {
    const float *init_state;
    float *final_state;
    const float *gam;
    int *status;
    int T, H, NC;
    bool zgate;   // multiply the outputs by silu(z)
    // Sequence segments (few long chains, chain_segments of chunk_layout.h): role 0 runs whole
    // sequences; role 1 runs each segment twice without outputs, CTA 2i from S_0 = 0 (end
    // state to ws_s0) and CTA 2i + 1 from S_0 = I with no value term (U = 0: the segment's
    // transition, to ws_phi); role 2 runs each segment from its start state (ws_start),
    // writing outputs.  [B*H][nseg][128][128] fp32, element [i][j] as in the state.
    int role, nseg, seg_len;
    float *ws_phi, *ws_s0;
    const float *ws_start;
};

// Per chunk c, in order (thread 0 issues the MMAs, thread 224 the TMA loads):
//   1. S^T -> bf16 operand (ST), S^T <- S^T Diag(G_C)
//   2. D[c % 2] = S^T [W; QH; QL]^T, one N = 192 product [bar_dw]
//   3. refill W and Q for c + 1; refill P for c + 1 (its buffer was read by chunk c - 1)
//   4. E^T = U^T - (W S)^T in place of (W S)^T (TF32-rounded fp32); refill U
//   5. S^T += E^T (K*G_C/G), kind::tf32 [bar_s]
//   6. output of chunk c - 1 = the sum of its D buffer's two (Q*G S)^T halves, staged in ST
//      (free: D[c % 2] is done reading it) and stored by TMA (overlaps step 5's MMAs); then
//      E^T P^T accumulated onto (QH S)^T in D[c % 2], kind::tf32 [bar_pe]
//   7. wait for the state update; refill K
// Every parity wait is placed where its barrier can be at most one phase ahead.
template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
kda_state_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mqh,
                 const __grid_constant__ CUtensorMap mql, const __grid_constant__ CUtensorMap mkt,
                 const __grid_constant__ CUtensorMap mp, const __grid_constant__ CUtensorMap mu,
                 const __grid_constant__ CUtensorMap to, const __grid_constant__ CUtensorMap tz,
                 const StateArgs a) {
    extern __shared__ unsigned char dsm_raw[];
    unsigned char *sm = align1024(dsm_raw);
    __shared__ uint64_t bar_w, bar_q, bar_u, bar_k, bar_p[2], bar_dw, bar_s, bar_pe, bar_z;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;
    // this CTA's chain and chunk range [c_begin, c_begin + nc), its start state (NULL: zero;
    // `identity`: I) and where its end state goes
    int bh = blockIdx.x, c_begin = 0, nc = a.NC;
    const float *s_init = a.init_state ? a.init_state + (size_t)bh * 16384 : nullptr;
    float *s_fin = a.final_state ? a.final_state + (size_t)bh * 16384 : nullptr;
    bool identity = false, use_u = true, outputs = true;
    if (a.role != 0) {
        const int idx = a.role == 1 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
        const int seg = idx % a.nseg;
        bh = idx / a.nseg;
        c_begin = seg * a.seg_len;
        nc = min(a.NC, c_begin + a.seg_len) - c_begin;
        const size_t slot = ((size_t)bh * a.nseg + seg) * 16384;
        if (a.role == 1) {
            outputs = false;
            s_init = nullptr;
            identity = (blockIdx.x & 1) != 0;
            use_u = !identity;
            s_fin = (identity ? a.ws_phi : a.ws_s0) + slot;
        } else {
            s_init = a.ws_start + slot;
            s_fin = (seg == a.nseg - 1 && a.final_state) ? a.final_state + (size_t)bh * 16384 : nullptr;
        }
    }
    const int h = bh % a.H, b = bh / a.H;
    constexpr int kTmaThread = 224;
    constexpr int kOutBoxes = sizeof(Tout) == 2 ? 2 : 4;
    float *sGam = reinterpret_cast<float *>(sm + S2_SMALL);   // [2][128]

    if (tid == 0) {
        uint64_t *bars[] = {&bar_w, &bar_q, &bar_u, &bar_k, &bar_p[0], &bar_p[1],
                            &bar_dw, &bar_s, &bar_pe, &bar_z};
        for (uint64_t *bb : bars) mbar_init(bb, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmb = tmem_base_s;
    const uint32_t tm = tmb + ((uint32_t)(32 * quarter) << 16);
    // operand descriptor of the shared-memory base: K-major, 128-byte swizzle
    const uint64_t dK0 = smem_desc_sw128(smem_u32(sm), 16, 1024);
    auto fail = [&]() {
        abort_s = 1;
        atomicExch(a.status, kErrTimeout);
    };
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
        if (!wait_cycles(bar, parity)) fail();
        tc_fence_after();
    };

    {   // S^T[j][i] = S_0[i][j]
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                v[u] = s_init ? s_init[(size_t)(i0 + u) * 128 + row] : (identity && i0 + u == row ? 1.f : 0.f);
            tmem_st32(tm + S2_TM_S + i0, v);
        }
        tmem_wait_st();
    }

    // first chunk of this CTA's range in the workspace; loads and buffers are indexed by the
    // step `it` within the range (chunk c_begin + it)
    const int64_t n0 = (int64_t)bh * a.NC + c_begin;
    auto rowc = [&](int it) { return (int)((n0 + it) * 64); };
    // (TMA thread) loads issued per barrier: w, q, u, k, p[0], p[1], z -- on an abort it
    // waits (bounded) for the last phase of each
    int issued[7] = {0, 0, 0, 0, 0, 0, 0};
    auto load_z = [&](int it) {
        ++issued[6];
        mbar_arrive_expect_tx(&bar_z, 16384);
        for (int kb = 0; kb < 2; ++kb)
            tma_load_4d(sm + S2_Z + kb * 8192, &tz, &bar_z, 64 * kb, h, (c_begin + it) * 64, b);
    };
    auto load_w = [&](int c) {
        ++issued[0];
        mbar_arrive_expect_tx(&bar_w, 16384);
        for (int kb = 0; kb < 2; ++kb) tma_load_2d(sm + S2_WQ + kb * S2_WQ_KB, &mw, &bar_w, 64 * kb, rowc(c));
    };
    auto load_q = [&](int c) {
        ++issued[1];
        mbar_arrive_expect_tx(&bar_q, 32768);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_2d(sm + S2_WQ + kb * S2_WQ_KB + 8192, &mqh, &bar_q, 64 * kb, rowc(c));
            tma_load_2d(sm + S2_WQ + kb * S2_WQ_KB + 16384, &mql, &bar_q, 64 * kb, rowc(c));
        }
    };
    auto load_u = [&](int c) {
        ++issued[2];
        mbar_arrive_expect_tx(&bar_u, 32768);
        for (int bx = 0; bx < 4; ++bx) tma_load_2d(sm + S2_U + bx * 8192, &mu, &bar_u, 32 * bx, rowc(c));
    };
    auto load_k = [&](int c) {   // four boxes: token block kb, channel half hf
        ++issued[3];
        mbar_arrive_expect_tx(&bar_k, 32768);
        for (int kb = 0; kb < 2; ++kb)
            for (int hf = 0; hf < 2; ++hf)
                tma_load_2d(sm + S2_KT + kb * 16384 + hf * 8192, &mkt, &bar_k, 32 * kb,
                            (int)((n0 + c) * 128 + 64 * hf));
    };
    auto load_p = [&](int c) {
        uint64_t *bb = &bar_p[c & 1];
        ++issued[4 + (c & 1)];
        unsigned char *dst = sm + S2_P + (c & 1) * 16384;
        mbar_arrive_expect_tx(bb, 16384);
        for (int kb = 0; kb < 2; ++kb) tma_load_2d(dst + kb * 8192, &mp, bb, 32 * kb, rowc(c));
    };
    if (tid == kTmaThread && nc > 0) {
        load_w(0);
        if (outputs) load_q(0);
        if (use_u) load_u(0);
        load_k(0);
        if (outputs) {
            load_p(0);
            if (nc > 1) load_p(1);
            if (a.zgate) load_z(0);
        }
    }
    if (tid < 128 && nc > 0) cp_async4(sGam + tid, a.gam + n0 * 128 + tid, 4);
    cp_async_commit();

    bool store_outstanding = false;   // thread 0: a TMA store from ST may still be reading it
    // output of chunk c from its DQ / PE buffers, staged in ST (free: see the callers)
    auto emit = [&](int c) {   // c: the step within the range
        float o[32], pe[32];   // (QH S)^T + E^T P^T, and (QL S)^T
        tmem_ld32(tm + S2_TM_D + S2_TM_DSTRIDE * (c & 1) + 64 + 32 * half, o);
        tmem_ld32(tm + S2_TM_D + S2_TM_DSTRIDE * (c & 1) + 128 + 32 * half, pe);
        tmem_wait_ld();
        const int j = row;
#pragma unroll
        for (int u = 0; u < 32; ++u) o[u] += pe[u];
        if (a.zgate) {
            if (!wait_cycles(&bar_z, c & 1)) fail();
            const unsigned char *zt = sm + S2_Z + (j >> 6) * 8192;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                o[u] *= silu_tanh(__bfloat162float(
                    *reinterpret_cast<const __nv_bfloat16 *>(zt + sw128_off(32 * half + u, j & 63))));
        }
        if (sizeof(Tout) == 2) {
            unsigned char *dst = sm + S2_ST + (j >> 6) * 8192;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                *reinterpret_cast<__nv_bfloat16 *>(dst + sw128_off(32 * half + u, j & 63)) =
                    __float2bfloat16_rn(o[u]);
        } else {
            unsigned char *dst = sm + S2_ST + (j >> 5) * 8192;
            const int cj = j & 31;
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int r = 32 * half + u;
                *reinterpret_cast<float *>(dst + r * 128 + ((((cj >> 2) ^ (r & 7)) & 7) << 4) +
                                           ((cj & 3) << 2)) = o[u];
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == kTmaThread && a.zgate && c + 1 < nc) load_z(c + 1);   // the z tile is read
        if (tid == 0) {
            constexpr int cols = sizeof(Tout) == 2 ? 64 : 32;
#pragma unroll
            for (int kb = 0; kb < kOutBoxes; ++kb)
                tma_store_4d(&to, sm + S2_ST + kb * 8192, cols * kb, h, (c_begin + c) * 64, b);
            bulk_commit();
            store_outstanding = true;
        }
    };

    for (int c = 0; c < nc; ++c) {   // step c: chunk c_begin + c
        const uint32_t par = c & 1;
        // ---- 1. S^T to bf16 (ST, free once the previous output's store has read it);
        //         S^T <- S^T Diag(G_C)
        if (tid == 0 && store_outstanding) {
            bulk_wait_read_all();
            store_outstanding = false;
        }
        cp_async_wait_all();
        __syncthreads();   // G_C of this chunk visible; ST free
        if (tid < 128 && c + 1 < nc)   // prefetch the next chunk's G_C
            cp_async4(sGam + ((c + 1) & 1) * 128 + tid, a.gam + (n0 + c + 1) * 128 + tid, 4);
        cp_async_commit();
        {
            const float *gam = sGam + (c & 1) * 128;
            float v[32];
            unsigned char *dst = sm + S2_ST + half * 16384;
            for (int part = 0; part < 2; ++part) {
                const int i0 = 64 * half + 32 * part;
                tmem_ld32(tm + S2_TM_S + i0, v);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float *f = v + 8 * q4;
                    *reinterpret_cast<uint4 *>(dst + sw128_off(row, 32 * part + 8 * q4)) =
                        make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]),
                                   pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
                }
#pragma unroll
                for (int u = 0; u < 32; ++u) v[u] *= gam[i0 + u];
                tmem_st32(tm + S2_TM_S + i0, v);
            }
            tmem_wait_st();
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (abort_s) break;

        // ---- 2. D[c % 2] = S^T [W; QH; QL]^T in one N = 192 product (without outputs:
        //         (W S)^T alone)
        if (tid == 0) {
            if (!wait_cycles(&bar_w, par)) fail();
            if (outputs && !wait_cycles(&bar_q, par)) fail();
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kk = (ks & 3) * 32;
                mma_bf16(tmb + S2_TM_D + S2_TM_DSTRIDE * par, desc_add(dK0, S2_ST + (ks >> 2) * 16384 + kk),
                         desc_add(dK0, S2_WQ + (ks >> 2) * S2_WQ_KB + kk), outputs ? ID_KK_N192 : ID_KK_N64,
                         ks > 0);
            }
            mma_commit(&bar_dw);
        }
        wait_bar(&bar_dw, par);
        // ---- 3. refills: W and Q for c + 1; P for c + 1 into the buffer chunk c - 1 read
        if (tid == kTmaThread && c + 1 < nc) {
            load_w(c + 1);
            if (outputs) {
                load_q(c + 1);
                if (c >= 1) {
                    if (!wait_cycles(&bar_pe, (c - 1) & 1)) fail();
                    load_p(c + 1);
                }
            }
        }

        // ---- 4. E^T = U^T - (W S)^T in place of (W S)^T, TF32-rounded (lane j = value channel,
        //         columns = tokens; U = 0 for a segment's transition): the A operand, in tensor
        //         memory, of the state update and of E^T P^T.  (E^T P^T of chunk c - 1 must be
        //         done before the next D product reuses its buffer.)
        if (outputs && c >= 1) wait_bar(&bar_pe, (c - 1) & 1);
        if (use_u && !wait_cycles(&bar_u, par)) fail();
        {
            const uint32_t te = tm + S2_TM_D + S2_TM_DSTRIDE * par + 32 * half;
            float ws[32];
            tmem_ld32(te, ws);
            tmem_wait_ld();
            const float *U = reinterpret_cast<const float *>(sm + S2_U);
            const int j = row;
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int r = 32 * half + u;
                ws[u] = round_tf32((use_u ? U[(j >> 5) * 2048 + r * 32 + (j & 31)] : 0.f) - ws[u]);
            }
            tmem_st32(te, ws);
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        if (tid == kTmaThread && use_u && c + 1 < nc) load_u(c + 1);   // U buffer is free

        // ---- 5. S^T += E^T (K*G_C/G) [bar_s]: kind::tf32, A = E^T in tensor memory, B the
        //         TF32 (K*G_C/G)^T tile (K-major: channels x tokens)
        const uint32_t tE = tmb + S2_TM_D + S2_TM_DSTRIDE * par;
        if (tid == 0) {
            if (!wait_cycles(&bar_k, par)) fail();
            if (outputs && !wait_cycles(&bar_p[par], (c >> 1) & 1)) fail();
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_tf32_ts(tmb + S2_TM_S, tE + 8 * ks, desc_add(dK0, S2_KT + (ks >> 2) * 16384 + (ks & 3) * 32),
                            ID_TF_N128, true);
            mma_commit(&bar_s);
        }

        // ---- 6. output of chunk c - 1 (ST is free: this chunk's D product has completed)
        if (outputs && c >= 1) emit(c - 1);

        // ---- 6b. E^T P^T -> PE[c % 2] [bar_pe], after the output: issuing blocks the issuing
        //          thread while the pipe drains the state update, which would hold the
        //          output's barriers
        if (tid == 0 && outputs) {   // (kind::tf32, A = E^T in tensor memory, B = P)
            tc_fence_after();
            const uint32_t pb = S2_P + par * 16384;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_tf32_ts(tE + 64, tE + 8 * ks, desc_add(dK0, pb + (ks >> 2) * 8192 + (ks & 3) * 32), ID_TF_N64,
                            true);   // onto (QH S)^T
            mma_commit(&bar_pe);
        }

        // ---- 7. state update done; K buffer is free
        wait_bar(&bar_s, par);
        if (tid == kTmaThread && c + 1 < nc) load_k(c + 1);
    }
    if (!abort_s && outputs && nc > 0) {   // output of the last chunk
        wait_bar(&bar_pe, (nc - 1) & 1);
        if (tid == 0 && store_outstanding) {
            bulk_wait_read_all();
            store_outstanding = false;
        }
        __syncthreads();
        emit(nc - 1);
    }
    if (!abort_s && s_fin) {
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
            tmem_ld32(tm + S2_TM_S + i0, v);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) s_fin[(size_t)(i0 + u) * 128 + row] = v[u];
        }
    }
    cp_async_wait_all();
    if (tid == 0 && store_outstanding) bulk_wait_all();
    if (abort_s && tid == kTmaThread) {
        uint64_t *lbars[7] = {&bar_w, &bar_q, &bar_u, &bar_k, &bar_p[0], &bar_p[1], &bar_z};
        for (int i = 0; i < 7; ++i)
            if (issued[i] > 0) wait_cycles(lbars[i], (uint32_t)(issued[i] - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmb, 512);
}

// ---------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// [B, T, H, 128] viewed as 4-D (128, H, T, B): box (128-byte row) x 1 x 64 x 1.
bool map4(CUtensorMap *m, const void *base, int64_t B, int64_t T, int64_t H, int esize, bool swz) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t e = (cuuint64_t)esize;
    cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {128 * e, (cuuint64_t)H * 128 * e, (cuuint64_t)(T * H) * 128 * e};
    cuuint32_t box[4] = {(cuuint32_t)(128 / e), 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [rows][cols] row-major workspace array: box (128-byte row) x 64 rows.
bool map2(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int esize, bool swz) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t e = (cuuint64_t)esize;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * e};
    cuuint32_t box[2] = {(cuuint32_t)(128 / e), 64};
    cuuint32_t es[2] = {1, 1};
    return enc(m, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_kda_supported(const ChunkProblem &p) {
    return p.in_bf16 && p.dk == 128 && p.dv == 128 && p.C == 64 && p.T > 0 && p.gate == 2;
}

// The per-chunk operand slabs, then (few long chains split into segments) the segments'
// transitions, zero-start end states and start states, [B*H][nseg][128][128] fp32 each.
size_t chunk_kda_workspace_bytes(const ChunkProblem &p) {
    int nseg, len;
    chain_segments(p.B * p.H, p.NC, &nseg, &len);
    const size_t seg = nseg > 1 ? (size_t)3 * p.B * p.H * nseg * 16384 * sizeof(float) : 0;
    return (size_t)(p.B * p.H * p.NC) * kKdaBytesPerChunk + seg;
}

int launch_chunk_kda(const ChunkProblem &p, void *workspace, int *status_word, cudaStream_t stream) {
    const int64_t nch = p.B * p.H * p.NC;
    const KdaWorkspace ws = kda_carve(workspace, nch);
    CUtensorMap tq, tk, tv, tla, to, tz;
    const bool zgate = (p.fuse & kFuseGate) != 0;
    if (!map4(&tq, p.q, p.B, p.T, p.H, 2, true) || !map4(&tk, p.k, p.B, p.T, p.H, 2, true) ||
        !map4(&tv, p.v, p.B, p.T, p.H, 2, true) || !map4(&tla, p.log_alpha, p.B, p.T, p.H, 4, true) ||
        !map4(&to, p.out, p.B, p.T, p.H, p.out_bf16 ? 2 : 4, true) ||
        !map4(&tz, zgate ? p.z : p.q, p.B, p.T, p.H, 2, true))   // (unused unless gated)
        return kErrCuda;
    CUtensorMap mw, mqh, mql, mkt, mp, mu;
    const int64_t rows = nch * 64;
    if (!map2(&mw, ws.W, rows, 128, 2, true) || !map2(&mqh, ws.QH, rows, 128, 2, true) ||
        !map2(&mql, ws.QL, rows, 128, 2, true) || !map2(&mkt, ws.KT, nch * 128, 64, 4, true) ||
        !map2(&mp, ws.P, rows, 64, 4, true) || !map2(&mu, ws.U, rows, 128, 4, false))
        return kErrCuda;

    const int s1 = (int)P1_TOTAL + 1024, s2 = (int)(zgate ? S2_TOTAL_Z : S2_TOTAL) + 1024;
    const int s2max = (int)S2_TOTAL_Z + 1024;
    if (cudaFuncSetAttribute(kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, s1) != cudaSuccess)
        return kErrCuda;
    PrepArgs pa{(const __nv_bfloat16 *)p.beta, ws, status_word, (int)p.T, (int)p.H, p.NC, p.fuse};
    kda_prep_kernel<<<(unsigned)nch, kThreads, s1, stream>>>(tq, tk, tv, tla, mw, mu, pa);
    if (cudaGetLastError() != cudaSuccess) return kErrCuda;

    StateArgs sa{p.init_state, p.final_state, ws.GAM, status_word, (int)p.T, (int)p.H, p.NC, zgate,
                 0, 1, p.NC, nullptr, nullptr, nullptr};
    auto state = [&](const StateArgs &sa_, unsigned grid) {
        auto kern = p.out_bf16 ? kda_state_kernel<__nv_bfloat16> : kda_state_kernel<float>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s2max) != cudaSuccess)
            return (int)kErrCuda;
        kern<<<grid, kThreads, s2, stream>>>(mw, mqh, mql, mkt, mp, mu, to, tz, sa_);
        return cudaGetLastError() == cudaSuccess ? (int)kOk : (int)kErrCuda;
    };
    const unsigned bh = (unsigned)(p.B * p.H);
    int nseg, seg_len;
    chain_segments(bh, p.NC, &nseg, &seg_len);
    if (nseg <= 1) return state(sa, bh);
    // segments: end states (two runs per segment), chaining, then outputs
    float *seg = reinterpret_cast<float *>(reinterpret_cast<char *>(workspace) + (size_t)nch * kKdaBytesPerChunk);
    const size_t per = (size_t)bh * nseg * 16384;
    sa.nseg = nseg;
    sa.seg_len = seg_len;
    sa.ws_phi = seg;
    sa.ws_s0 = seg + per;
    sa.ws_start = seg + 2 * per;
    sa.role = 1;
    int rc = state(sa, bh * nseg * 2);
    if (rc != kOk) return rc;
    rc = tc_launch_seg_combine(p.init_state, sa.ws_phi, sa.ws_s0, seg + 2 * per, bh, nseg, stream);
    if (rc != kOk) return rc;
    sa.role = 2;
    return state(sa, bh * nseg);
}

}  // namespace dr
