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
// W (bf16), U (fp32), P, Q*G and K*G_C/G (bf16 high/low pairs) and G_C.  The exponentials
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
// chunk, TMA-loads the stored operands: D = S^T [W; Q*G]^T, E^T = U^T - (W S)^T,
// S^T <- S^T Diag(G_C) + E^T (K*G_C/G), O^T = (Q*G S)^T + E^T P^T, with the operand
// buffers of the next chunk refilled as soon as each is consumed.
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
// W [64][128] bf16, U [64][128] fp32, PH/PL [64][64] bf16, QH/QL/KH/KL [64][128] bf16, GAM [128]
struct KdaWorkspace {
    __nv_bfloat16 *W, *PH, *PL, *QH, *QL, *KH, *KL;
    float *U, *GAM;
};
constexpr size_t kKdaBytesPerChunk = 16384 + 32768 + 2 * 8192 + 4 * 16384 + 512;

KdaWorkspace kda_carve(void *base, int64_t nch) {
    char *p = (char *)base;
    KdaWorkspace w;
    w.W = (__nv_bfloat16 *)p;   p += nch * 16384;
    w.U = (float *)p;           p += nch * 32768;
    w.PH = (__nv_bfloat16 *)p;  p += nch * 8192;
    w.PL = (__nv_bfloat16 *)p;  p += nch * 8192;
    w.QH = (__nv_bfloat16 *)p;  p += nch * 16384;
    w.QL = (__nv_bfloat16 *)p;  p += nch * 16384;
    w.KH = (__nv_bfloat16 *)p;  p += nch * 16384;
    w.KL = (__nv_bfloat16 *)p;  p += nch * 16384;
    w.GAM = (float *)p;
    return w;
}

// ---------------------------------------------------------------- prep kernel layout
constexpr uint32_t P1_Q = 0, P1_K = 16384, P1_V = 32768;   // 64 x 128 bf16 tiles, 2 K-blocks
constexpr uint32_t P1_LA = 49152;    // log alpha, then g: 4 boxes [64][32] fp32 (no swizzle)
constexpr uint32_t P1_OPS = 81920;   // round operands; after them A, T, T diag(beta), K*G
constexpr uint32_t P1_LH = P1_OPS, P1_LL = P1_OPS + 32768;   // [L_Q kb0|L_K kb0|L_Q kb1|L_K kb1]
constexpr uint32_t P1_RH = P1_OPS + 65536, P1_RL = P1_OPS + 69632;   // [R kb0 | R kb1], 2 KB each
constexpr uint32_t P1_A = P1_OPS, P1_T = P1_OPS + 16384, P1_TB = P1_OPS + 34816,
                   P1_KG = P1_OPS + 51200;
constexpr uint32_t P1_SMALL = P1_OPS + 73728;   // beta[64], ones[64], solve scratch[1024]
constexpr uint32_t P1_TOTAL = P1_SMALL + 8192;
constexpr uint32_t P1_TM_X = 0, P1_TM_U = 64, P1_TM_W = 128;

constexpr uint32_t ID_KK_N16 = idesc_bf16(128, 16, false, false);
// Largest per-channel decay (natural log) inside one 16-token block that the tensor-core
// products of the diagonal blocks take; beyond it the chunk recomputes those entries.
constexpr float kDiagLimit = 64.f;
constexpr uint32_t ID_MK_N64 = idesc_bf16(128, 64, true, false);

struct PrepArgs {
    const __nv_bfloat16 *beta;
    KdaWorkspace ws;
    int *status;
    int T, H, NC;
};

// Element (t, c) of the [64][128] fp32 tile loaded as four [64][32] boxes.
__device__ __forceinline__ uint32_t la_off(int t, int c) {
    return (uint32_t)((c >> 5) * 8192 + t * 128 + (c & 31) * 4);
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
__device__ __forceinline__ void load8_f32(const float *p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__global__ void __launch_bounds__(kThreads, 1)
kda_prep_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tla,
                const PrepArgs a) {
    extern __shared__ unsigned char dsm_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)dsm_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s, diag_exact_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;
    const int64_t n = blockIdx.x;
    const int c = (int)(n % a.NC);
    const int64_t bh = n / a.NC;
    const int h = (int)(bh % a.H), b = (int)(bh / a.H);
    const int t0 = c * 64;
    const int Lc = min(64, a.T - t0);
    float *sBeta = reinterpret_cast<float *>(sm + P1_SMALL);
    float *sOnes = sBeta + 64;
    float *sM = sBeta + 128;
    const float *LA = reinterpret_cast<const float *>(sm + P1_LA);
    float *const Xd = reinterpret_cast<float *>(sm + P1_KG);   // exact diagonal blocks
    bool diag_exact = false;

    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        abort_s = 0;
        diag_exact_s = 0;
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
    auto fail = [&]() {
        abort_s = 1;
        atomicExch(a.status, kErrTimeout);
    };

    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_ld, 49152 + 32768);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sm + P1_Q + kb * 8192, &tq, &bar_ld, 64 * kb, h, t0, b);
            tma_load_4d(sm + P1_K + kb * 8192, &tk, &bar_ld, 64 * kb, h, t0, b);
            tma_load_4d(sm + P1_V + kb * 8192, &tv, &bar_ld, 64 * kb, h, t0, b);
        }
        for (int bx = 0; bx < 4; ++bx)
            tma_load_4d(sm + P1_LA + bx * 8192, &tla, &bar_ld, 32 * bx, h, t0, b);
    }
    if (tid < 64) {
        sBeta[tid] = tid < Lc ? __bfloat162float(a.beta[((size_t)b * a.T + t0 + tid) * a.H + h]) : 0.f;
        sOnes[tid] = 1.f;
    }
    if (!wait_cycles(&bar_ld, 0)) fail();
    __syncthreads();
    if (abort_s) goto done;

    // ---- cumulative log decay g (in place) and G_C = exp(g_63) per channel; flag the chunk
    //      if some channel decays by more than kDiagLimit inside one 16-token block
    if (tid < 128) {
        float *la = reinterpret_cast<float *>(sm + P1_LA);
        float acc = 0.f;
        bool steep = false;
        for (int t = 0; t < 64; ++t) {
            acc += la[la_off(t, tid) / 4];
            la[la_off(t, tid) / 4] = acc;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            steep |= la[la_off(16 * j, tid) / 4] - la[la_off(16 * j + 15, tid) / 4] > kDiagLimit;
        if (steep) diag_exact_s = 1;
        a.ws.GAM[n * 128 + tid] = __expf(acc);
    }
    __syncthreads();

    // ---- X = [Q; K] K^T with per-channel decays, by column block j (tokens 16 j .. 16 j + 15),
    //      against the reference g_ref = g at the block's last token: the right factor
    //      k_s exp(g_ref - g_s) is <= |k_s|, the left factor exp(g_r - g_ref) is <= 1 below
    //      the block and at most exp(kDiagLimit) inside it (clamped there; a flagged chunk
    //      recomputes those entries below)
    for (int j = 0; j < 4; ++j) {
        const int ref = 16 * j + 15;
        for (int task = tid; task < (64 - 16 * j) * 16; task += kThreads) {
            const int r = 16 * j + (task >> 4), c8 = task & 15;
            float q8[8], k8[8], g8[8], rf[8];
            load8_bf16(sm + P1_Q, r, c8, q8);
            load8_bf16(sm + P1_K, r, c8, k8);
            load8_f32(LA + la_off(r, 8 * c8) / 4, g8);
            load8_f32(LA + la_off(ref, 8 * c8) / 4, rf);
            uint32_t qh[4], ql[4], kh[4], kl[4];
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
                const float f0 = __expf(fminf(g8[u] - rf[u], kDiagLimit));
                const float f1 = __expf(fminf(g8[u + 1] - rf[u + 1], kDiagLimit));
                pack_hi_lo(q8[u] * f0, q8[u + 1] * f1, qh[u >> 1], ql[u >> 1]);
                pack_hi_lo(k8[u] * f0, k8[u + 1] * f1, kh[u >> 1], kl[u >> 1]);
            }
            const uint32_t off = (c8 >> 3) * 16384 + sw128_off(r, (8 * c8) & 63);
            *reinterpret_cast<uint4 *>(sm + P1_LH + off) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
            *reinterpret_cast<uint4 *>(sm + P1_LL + off) = make_uint4(ql[0], ql[1], ql[2], ql[3]);
            *reinterpret_cast<uint4 *>(sm + P1_LH + 8192 + off) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
            *reinterpret_cast<uint4 *>(sm + P1_LL + 8192 + off) = make_uint4(kl[0], kl[1], kl[2], kl[3]);
        }
        {
            const int rr = tid >> 4, c8 = tid & 15, s = 16 * j + rr;
            float k8[8], g8[8], rf[8];
            load8_bf16(sm + P1_K, s, c8, k8);
            load8_f32(LA + la_off(s, 8 * c8) / 4, g8);
            load8_f32(LA + la_off(ref, 8 * c8) / 4, rf);
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int u = 0; u < 8; u += 2)
                pack_hi_lo(k8[u] * __expf(rf[u] - g8[u]), k8[u + 1] * __expf(rf[u + 1] - g8[u + 1]),
                           hi[u >> 1], lo[u >> 1]);
            const uint32_t off = (c8 >> 3) * 2048 + sw128_off(rr, (8 * c8) & 63);
            *reinterpret_cast<uint4 *>(sm + P1_RH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sm + P1_RL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t la_[3] = {P1_LH, P1_LH, P1_LL}, ra_[3] = {P1_RH, P1_RL, P1_RH};
#pragma unroll
            for (int part = 0; part < 3; ++part)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, kk = (ks & 3) * 32;
                    mma_bf16(tmb + P1_TM_X + 16 * j,
                             smem_desc_sw128(smem_u32(sm + la_[part] + kb * 16384 + kk), 16, 1024),
                             smem_desc_sw128(smem_u32(sm + ra_[part] + kb * 2048 + kk), 16, 1024),
                             ID_KK_N16, (part | ks) != 0);
                }
            mma_commit(&bar_mma);
        }
        if (!wait_cycles(&bar_mma, j & 1)) fail();
        tc_fence_after();
        __syncthreads();
        if (abort_s) goto done;
    }

    // ---- flagged chunk: entries of the four diagonal 16 x 16 blocks in fp32, one exponential
    //      per channel, into Xd[2][64][16] (rows of P, then rows of A before beta)
    diag_exact = diag_exact_s != 0;
    if (diag_exact) {
        for (int task = tid; task < 2 * 64 * 16; task += kThreads) {
            const int part = task >> 10, r = (task >> 4) & 63, s = (r & ~15) + (task & 15);
            const unsigned char *xt = sm + (part ? P1_K : P1_Q);
            float acc = 0.f;
            if (s <= r)
                for (int ch = 0; ch < 128; ++ch) {
                    const uint32_t o = (ch >> 6) * 8192;
                    const float xr = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16 *>(xt + o + sw128_off(r, ch & 63)));
                    const float ks = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16 *>(sm + P1_K + o + sw128_off(s, ch & 63)));
                    acc = fmaf(xr * ks, __expf(LA[la_off(r, ch) / 4] - LA[la_off(s, ch) / 4]), acc);
                }
            Xd[task] = acc;
        }
        __syncthreads();
    }

    // ---- P (rows 0..63 of X) to the workspace as a bf16 pair; A (rows 64..127) in fp32
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
        if (quarter < 2) {
            const int r = row;
            uint32_t ph[16], pl[16];
#pragma unroll
            for (int u = 0; u < 32; u += 2)
                pack_hi_lo(c0 + u <= r ? x[u] : 0.f, c0 + u + 1 <= r ? x[u + 1] : 0.f, ph[u >> 1], pl[u >> 1]);
            uint4 *dh = reinterpret_cast<uint4 *>(a.ws.PH + (n * 64 + r) * 64 + c0);
            uint4 *dl = reinterpret_cast<uint4 *>(a.ws.PL + (n * 64 + r) * 64 + c0);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                dh[q4] = make_uint4(ph[4 * q4], ph[4 * q4 + 1], ph[4 * q4 + 2], ph[4 * q4 + 3]);
                dl[q4] = make_uint4(pl[4 * q4], pl[4 * q4 + 1], pl[4 * q4 + 2], pl[4 * q4 + 3]);
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

    // ---- T = (I + A)^-1 with T diag(beta) in bf16 (the second operand, T diag(beta)
    //      diag(ones), is not used here)
    solve_unit_lower64(reinterpret_cast<const float *>(sm + P1_A), reinterpret_cast<float *>(sm + P1_T),
                       sM, sm + P1_TB, sBeta, sOnes, tid);

    // ---- K*G (MMA operand), and Q*G, K*G_C/G (bf16 pairs) to the workspace
    for (int task = tid; task < 64 * 16; task += kThreads) {
        const int r = task >> 4, c8 = task & 15;
        float q8[8], k8[8], g8[8], gl[8];
        load8_bf16(sm + P1_Q, r, c8, q8);
        load8_bf16(sm + P1_K, r, c8, k8);
        load8_f32(LA + la_off(r, 8 * c8) / 4, g8);
        load8_f32(LA + la_off(63, 8 * c8) / 4, gl);
        uint32_t kg[4], qh[4], ql[4], dh[4], dl[4];
#pragma unroll
        for (int u = 0; u < 8; u += 2) {
            const float e0 = __expf(g8[u]), e1 = __expf(g8[u + 1]);
            kg[u >> 1] = pack_bf16(k8[u] * e0, k8[u + 1] * e1);
            pack_hi_lo(q8[u] * e0, q8[u + 1] * e1, qh[u >> 1], ql[u >> 1]);
            pack_hi_lo(k8[u] * __expf(gl[u] - g8[u]), k8[u + 1] * __expf(gl[u + 1] - g8[u + 1]),
                       dh[u >> 1], dl[u >> 1]);
        }
        *reinterpret_cast<uint4 *>(sm + P1_KG + (c8 >> 3) * 8192 + sw128_off(r, (8 * c8) & 63)) =
            make_uint4(kg[0], kg[1], kg[2], kg[3]);
        const size_t go = ((size_t)n * 64 + r) * 128 + 8 * c8;
        *reinterpret_cast<uint4 *>(a.ws.QH + go) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
        *reinterpret_cast<uint4 *>(a.ws.QL + go) = make_uint4(ql[0], ql[1], ql[2], ql[3]);
        *reinterpret_cast<uint4 *>(a.ws.KH + go) = make_uint4(dh[0], dh[1], dh[2], dh[3]);
        *reinterpret_cast<uint4 *>(a.ws.KL + go) = make_uint4(dl[0], dl[1], dl[2], dl[3]);
    }
    fence_proxy_async();
    __syncthreads();

    // ---- U^T = V^T (T diag beta)^T,  W^T = (K*G)^T (T diag beta)^T
    if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmb + P1_TM_U, smem_desc_sw128(smem_u32(sm + P1_V + ks * 2048), 8192, 1024),
                     smem_desc_sw128(smem_u32(sm + P1_TB + ks * 32), 16, 1024), ID_MK_N64, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmb + P1_TM_W, smem_desc_sw128(smem_u32(sm + P1_KG + ks * 2048), 8192, 1024),
                     smem_desc_sw128(smem_u32(sm + P1_TB + ks * 32), 16, 1024), ID_MK_N64, ks > 0);
        mma_commit(&bar_mma);
    }
    if (!wait_cycles(&bar_mma, 0)) fail();   // fifth completion of bar_mma: parity 0
    tc_fence_after();
    // W[r][i] and U[r][j] from the transposed TMEM tiles (lane = channel, column = token)
    {
        float w[32], u32[32];
        tmem_ld32(tm + P1_TM_W + 32 * half, w);
        tmem_ld32(tm + P1_TM_U + 32 * half, u32);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const size_t rr = (size_t)n * 64 + 32 * half + u;
            a.ws.W[rr * 128 + row] = __float2bfloat16_rn(w[u]);
            a.ws.U[rr * 128 + row] = u32[u];
        }
    }
done:
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmb, 256);
}

// ---------------------------------------------------------------- state kernel layout
constexpr uint32_t S2_W = 0, S2_QH = 16384, S2_QL = 32768;   // K-major [64][128], 2 K-blocks
constexpr uint32_t S2_KH = 49152, S2_KL = 65536;             // MN-major [64 tok][128 ch]
constexpr uint32_t S2_PH = 81920, S2_PL = 90112;             // K-major [64][64]
constexpr uint32_t S2_U = 98304;                             // [64][128] fp32, 4 boxes of 32
constexpr uint32_t S2_ST = 131072;                           // S^T bf16 [128][128], 2 K-blocks
constexpr uint32_t S2_EH = 163840, S2_EL = 180224;           // E^T bf16 pair [128][64]
constexpr uint32_t S2_OUT = S2_EH;                           // output tile after the MMAs
constexpr uint32_t S2_SMALL = 196608;                        // G_C of two chunks
constexpr uint32_t S2_TOTAL = S2_SMALL + 1024;
constexpr uint32_t S2_TM_S = 0, S2_TM_D = 128, S2_TM_PE = 256;

constexpr uint32_t ID_KK_N64 = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_KM_N128 = idesc_bf16(128, 128, false, true);

struct StateArgs {
    const float *init_state;
    float *final_state;
    const float *gam;
    int *status;
    int T, H, NC;
};

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
kda_state_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mqh,
                 const __grid_constant__ CUtensorMap mql, const __grid_constant__ CUtensorMap mkh,
                 const __grid_constant__ CUtensorMap mkl, const __grid_constant__ CUtensorMap mph,
                 const __grid_constant__ CUtensorMap mpl, const __grid_constant__ CUtensorMap mu,
                 const __grid_constant__ CUtensorMap to, const StateArgs a) {
    extern __shared__ unsigned char dsm_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)dsm_raw + 1023) & ~(uintptr_t)1023);
    // operand groups (each completes once per chunk): W + Q pair, U, K pair + P pair
    __shared__ uint64_t bar_wq, bar_u, bar_kp, bar_d, bar_s;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;
    const int bh = blockIdx.x, h = bh % a.H, b = bh / a.H;
    constexpr int kTmaThread = 224;
    constexpr int kOutBoxes = sizeof(Tout) == 2 ? 2 : 4;
    float *sGam = reinterpret_cast<float *>(sm + S2_SMALL);   // [2][128]

    if (tid == 0) {
        mbar_init(&bar_wq, 1);
        mbar_init(&bar_u, 1);
        mbar_init(&bar_kp, 1);
        mbar_init(&bar_d, 1);
        mbar_init(&bar_s, 1);
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
                v[u] = a.init_state ? a.init_state[((size_t)bh * 128 + i0 + u) * 128 + row] : 0.f;
            tmem_st32(tm + S2_TM_S + i0, v);
        }
        tmem_wait_st();
    }

    const int64_t n0 = (int64_t)bh * a.NC;   // first chunk of this chain in the workspace
    auto load_wq = [&](int c) {
        const int y = (int)((n0 + c) * 64);
        mbar_arrive_expect_tx(&bar_wq, 3 * 16384);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_2d(sm + S2_W + kb * 8192, &mw, &bar_wq, 64 * kb, y);
            tma_load_2d(sm + S2_QH + kb * 8192, &mqh, &bar_wq, 64 * kb, y);
            tma_load_2d(sm + S2_QL + kb * 8192, &mql, &bar_wq, 64 * kb, y);
        }
    };
    auto load_u = [&](int c) {
        const int y = (int)((n0 + c) * 64);
        mbar_arrive_expect_tx(&bar_u, 32768);
        for (int bx = 0; bx < 4; ++bx) tma_load_2d(sm + S2_U + bx * 8192, &mu, &bar_u, 32 * bx, y);
    };
    auto load_kp = [&](int c) {
        const int y = (int)((n0 + c) * 64);
        mbar_arrive_expect_tx(&bar_kp, 2 * 16384 + 2 * 8192);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_2d(sm + S2_KH + kb * 8192, &mkh, &bar_kp, 64 * kb, y);
            tma_load_2d(sm + S2_KL + kb * 8192, &mkl, &bar_kp, 64 * kb, y);
        }
        tma_load_2d(sm + S2_PH, &mph, &bar_kp, 0, y);
        tma_load_2d(sm + S2_PL, &mpl, &bar_kp, 0, y);
    };
    if (tid == kTmaThread && a.NC > 0) {
        load_wq(0);
        load_u(0);
        load_kp(0);
    }
    if (tid < 128 && a.NC > 0) cp_async4(sGam + tid, a.gam + n0 * 128 + tid, 4);
    cp_async_commit();

    bool store_outstanding = false;
    for (int c = 0; c < a.NC; ++c) {
        const uint32_t par = c & 1;
        const int t0 = c * 64;
        // ---- S^T to bf16 (MMA operand); S^T <- S^T Diag(G_C)
        cp_async_wait_all();
        __syncthreads();   // G_C of this chunk visible
        if (tid < 128 && c + 1 < a.NC)   // prefetch the next chunk's G_C
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

        // ---- D = S^T [W; Q*G]^T  (the Q*G half as a high/low pair)
        if (tid == 0) {
            if (store_outstanding) {   // the previous output tile must have left S2_OUT
                bulk_wait_read_all();
                store_outstanding = false;
            }
            if (!wait_cycles(&bar_wq, par)) fail();
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32, ob = (ks >> 2) * 8192 + (ks & 3) * 32;
                const uint64_t ad = smem_desc_sw128(smem_u32(sm + S2_ST + o), 16, 1024);
                mma_bf16(tmb + S2_TM_D, ad, smem_desc_sw128(smem_u32(sm + S2_W + ob), 16, 1024), ID_KK_N64, ks > 0);
                mma_bf16(tmb + S2_TM_D + 64, ad, smem_desc_sw128(smem_u32(sm + S2_QH + ob), 16, 1024), ID_KK_N64, ks > 0);
                mma_bf16(tmb + S2_TM_D + 64, ad, smem_desc_sw128(smem_u32(sm + S2_QL + ob), 16, 1024), ID_KK_N64, 1);
            }
            mma_commit(&bar_d);
        }
        wait_bar(&bar_d, par);
        if (tid == kTmaThread && c + 1 < a.NC) load_wq(c + 1);   // W, Q*G buffers are free

        // ---- E^T = U^T - (W S)^T as a bf16 pair (lane j = value channel, columns = tokens)
        if (!wait_cycles(&bar_u, par)) fail();
        {
            float ws[32];
            tmem_ld32(tm + S2_TM_D + 32 * half, ws);
            tmem_wait_ld();
            const float *U = reinterpret_cast<const float *>(sm + S2_U);
            const int j = row;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float e[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int r = 32 * half + 8 * q4 + u;
                    e[u] = U[(j >> 5) * 2048 + r * 32 + (j & 31)] - ws[8 * q4 + u];
                }
                uint32_t eh[4], el[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) pack_hi_lo(e[2 * u], e[2 * u + 1], eh[u], el[u]);
                const uint32_t off = sw128_off(row, 32 * half + 8 * q4);
                *reinterpret_cast<uint4 *>(sm + S2_EH + off) = make_uint4(eh[0], eh[1], eh[2], eh[3]);
                *reinterpret_cast<uint4 *>(sm + S2_EL + off) = make_uint4(el[0], el[1], el[2], el[3]);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == kTmaThread && c + 1 < a.NC) load_u(c + 1);    // U buffer is free

        // ---- S^T += E^T (K*G_C/G);  PE = E^T P^T   (bf16 pairs: hi.hi + hi.lo + lo.hi)
        if (tid == 0) {
            if (!wait_cycles(&bar_kp, par)) fail();
            tc_fence_after();
            const uint32_t ea[3] = {S2_EH, S2_EH, S2_EL}, kbuf[3] = {S2_KH, S2_KL, S2_KH},
                           pbuf[3] = {S2_PH, S2_PL, S2_PH};
#pragma unroll
            for (int part = 0; part < 3; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t ad = smem_desc_sw128(smem_u32(sm + ea[part] + ks * 32), 16, 1024);
                    mma_bf16(tmb + S2_TM_S, ad,
                             smem_desc_sw128(smem_u32(sm + kbuf[part] + ks * 2048), 8192, 1024), ID_KM_N128, 1);
                    mma_bf16(tmb + S2_TM_PE, ad, smem_desc_sw128(smem_u32(sm + pbuf[part] + ks * 32), 16, 1024),
                             ID_KK_N64, (part | ks) != 0);
                }
            mma_commit(&bar_s);
        }
        wait_bar(&bar_s, par);
        if (tid == kTmaThread && c + 1 < a.NC) load_kp(c + 1);   // K, P buffers are free

        // ---- outputs o = (Q*G S)^T + E^T P^T, staged row-major and written by TMA
        {
            float o[32], pe[32];
            tmem_ld32(tm + S2_TM_D + 64 + 32 * half, o);
            tmem_ld32(tm + S2_TM_PE + 32 * half, pe);
            tmem_wait_ld();
            const int j = row;
            if (sizeof(Tout) == 2) {
                unsigned char *dst = sm + S2_OUT + (j >> 6) * 8192;
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    *reinterpret_cast<__nv_bfloat16 *>(dst + sw128_off(32 * half + u, j & 63)) =
                        __float2bfloat16_rn(o[u] + pe[u]);
            } else {
                unsigned char *dst = sm + S2_OUT + (j >> 5) * 8192;
                const int cj = j & 31;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int r = 32 * half + u;
                    *reinterpret_cast<float *>(dst + r * 128 + ((((cj >> 2) ^ (r & 7)) & 7) << 4) +
                                               ((cj & 3) << 2)) = o[u] + pe[u];
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            constexpr int cols = sizeof(Tout) == 2 ? 64 : 32;
#pragma unroll
            for (int kb = 0; kb < kOutBoxes; ++kb)
                tma_store_4d(&to, sm + S2_OUT + kb * 8192, cols * kb, h, t0, b);
            bulk_commit();
            store_outstanding = true;
        }
    }
    if (!abort_s && a.final_state) {
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
            tmem_ld32(tm + S2_TM_S + i0, v);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) a.final_state[((size_t)bh * 128 + i0 + u) * 128 + row] = v[u];
        }
    }
    cp_async_wait_all();
    if (tid == 0 && store_outstanding) bulk_wait_all();
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

size_t chunk_kda_workspace_bytes(const ChunkProblem &p) {
    return (size_t)(p.B * p.H * p.NC) * kKdaBytesPerChunk;
}

int launch_chunk_kda(const ChunkProblem &p, void *workspace, int *status_word, cudaStream_t stream) {
    const int64_t nch = p.B * p.H * p.NC;
    const KdaWorkspace ws = kda_carve(workspace, nch);
    CUtensorMap tq, tk, tv, tla, to;
    if (!map4(&tq, p.q, p.B, p.T, p.H, 2, true) || !map4(&tk, p.k, p.B, p.T, p.H, 2, true) ||
        !map4(&tv, p.v, p.B, p.T, p.H, 2, true) || !map4(&tla, p.log_alpha, p.B, p.T, p.H, 4, false) ||
        !map4(&to, p.out, p.B, p.T, p.H, p.out_bf16 ? 2 : 4, true))
        return kErrCuda;
    CUtensorMap mw, mqh, mql, mkh, mkl, mph, mpl, mu;
    const int64_t rows = nch * 64;
    if (!map2(&mw, ws.W, rows, 128, 2, true) || !map2(&mqh, ws.QH, rows, 128, 2, true) ||
        !map2(&mql, ws.QL, rows, 128, 2, true) || !map2(&mkh, ws.KH, rows, 128, 2, true) ||
        !map2(&mkl, ws.KL, rows, 128, 2, true) || !map2(&mph, ws.PH, rows, 64, 2, true) ||
        !map2(&mpl, ws.PL, rows, 64, 2, true) || !map2(&mu, ws.U, rows, 128, 4, false))
        return kErrCuda;

    const int s1 = (int)P1_TOTAL + 1024, s2 = (int)S2_TOTAL + 1024;
    if (cudaFuncSetAttribute(kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, s1) != cudaSuccess)
        return kErrCuda;
    PrepArgs pa{(const __nv_bfloat16 *)p.beta, ws, status_word, (int)p.T, (int)p.H, p.NC};
    kda_prep_kernel<<<(unsigned)nch, kThreads, s1, stream>>>(tq, tk, tv, tla, pa);
    if (cudaGetLastError() != cudaSuccess) return kErrCuda;

    StateArgs sa{p.init_state, p.final_state, ws.GAM, status_word, (int)p.T, (int)p.H, p.NC};
    const unsigned grid = (unsigned)(p.B * p.H);
    if (p.out_bf16) {
        if (cudaFuncSetAttribute(kda_state_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 s2) != cudaSuccess)
            return kErrCuda;
        kda_state_kernel<__nv_bfloat16><<<grid, kThreads, s2, stream>>>(mw, mqh, mql, mkh, mkl, mph, mpl, mu, to, sa);
    } else {
        if (cudaFuncSetAttribute(kda_state_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, s2) !=
            cudaSuccess)
            return kErrCuda;
        kda_state_kernel<float><<<grid, kThreads, s2, stream>>>(mw, mqh, mql, mkh, mkl, mph, mpl, mu, to, sa);
    }
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace dr
