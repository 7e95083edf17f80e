// chunk_simt.cu -- chunkwise forward of the gated delta rule with fp32 sums: the path for every
// configuration the tensor-core kernels do not take, and the backward's operand recompute.
//
// Chunk form (derived from the recurrence S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} +
// b_t k_t v_t^T, o_t = S_t^T q_t of the page "NLP: linear attention summary", KDA section;
// the pages name the technique -- chunks computed in parallel inside, state carried
// between them, WY representation and a triangular solve -- on the pages "Transformer
// notes (5): linear attention optimisations" and "linear-attention gated-deltanet guide",
// section 5, but print no chunk equations).  Inside a chunk of C tokens started from
// S_0, with g_r = sum_{u<=r} log a_u (scalar or per key channel) and G_r = exp(g_r):
//
//   e_r = b_r (v_r - (Diag(a_r) S_{r-1})^T k_r)               (written residual)
//   (I + A) E = diag(b) (V - (K*G) S_0),  A_rs = b_r (k_r*G_r).(k_s/G_s), s < r
//   T = (I + A)^{-1},  W = T diag(b) (K*G),  U = T diag(b) V,  E = U - W S_0
//   O = (Q*G) S_0 + P E,  P_rs = (q_r*G_r).(k_s/G_s) for s <= r, else 0
//   S_C = Diag(G_C) S_0 + (K * G_C/G)^T E
//
// Two kernels:
//   chunk_prep_kernel   one CTA per (b, h, chunk), all chunks in parallel: cumulative log
//                       decay, A and P, the forward substitution for T, W and U; writes
//                       W, U, P, Q*G, K*G_C/G and G_C to the workspace (fp32).  For the
//                       scalar gate and no gate, A, P, W and U are TF32 warp tiles
//                       (tc_common.cuh: three split products at fp32 accuracy for fp32
//                       inputs, one for bf16 inputs); the per-channel gate's A and P stay
//                       per-thread fp32 dot products around the sub-chunk references.
//   chunk_state_kernel  one CTA per (b, h, 32 state columns), sequential over chunks:
//                       E = U - W S, O = (Q*G) S + P E, S <- Diag(G_C) S + (K*G_C/G)^T E.
//
// Exponents: every factor exp(x) taken here has x <= 0, except inside one 16-token
// sub-chunk, where x is bounded by 16 max|log a|.  For the per-channel gate the pair term
// exp(g_r - g_s) of A and P is split at the last position p of the sub-chunk before the
// one holding s (s <= p < r):  exp(g_r - ref_i) * exp(ref_i - ref_j) * exp(ref_j - g_s),
// ref_j = g_{16 j - 1} (0 for j = 0), so no product divides by a tiny cumulative decay
// (the log-space, two-level chunking remedy named on the "Transformer notes (5)" page).
//
// Fused neighbours (DR_FUSE_* of include/dr.h): the prep kernel takes beta = sigmoid(logit)
// (stored in beta's dtype) and divides each q and k row by its norm as soon as the rows are
// in shared memory (fp32); the state kernel multiplies each output by silu(z).
#include <algorithm>

#include "common.cuh"
#include "chunk_layout.h"
#include "tc_common.cuh"

namespace dr {

namespace {

constexpr int kThreads = 256;
constexpr int kLd = 132;   // padded fp32 row stride of [64][<=128] smem tiles
constexpr int kLdA = 65;   // padded row stride of [64][64] smem tiles
constexpr int kSub = 16;   // sub-chunk length of the exponent reference points

struct PrepArgs {
    const void *q, *k, *v;
    const float *log_alpha;
    const void *beta;
    int64_t B, T, H;
    int dv, C, NC, gate;
    uint32_t fuse;
    ChunkWorkspace ws;
    float *T_out;    // backward only: T = (I + A)^-1 per chunk, [n][C][C] (NULL otherwise)
};

struct StateArgs {
    const float *init_state;
    void *out;
    float *final_state;
    const void *z;   // output gate input (in_bf16 ? bf16 : fp32), NULL when not fused
    bool z_bf16;
    int64_t B, T, H;
    int dv, C, NC;
    ChunkWorkspace ws;
    float *ckpt;     // backward only: the state at each chunk's start, [n][dk][dv] (NULL
                     // otherwise); with it, `out` may be NULL (no outputs written)
    // Sequence segments (few long chains): role 0 runs whole sequences; role 1 runs each
    // segment without outputs, its first dv/32 CTAs from S_0 = 0 (end state to ws_s0,
    // [chains][nseg][dk][dv]) and its next dk/32 CTAs as the transition, from S_0 = I with
    // no value term (U = 0; end state to ws_phi, [chains][nseg][dk][dk]); role 2 runs each
    // segment from its start state (ws_start, [chains][nseg][dk][dv]), writing outputs.
    int role, nseg, seg_len;
    float *ws_phi, *ws_s0;
    const float *ws_start;
};

// The per-channel gate needs its [64][dk] cumulative decays, the sub-chunk pair factors and
// a separate right-factor tile; the scalar gate and no gate take the right factors over q's
// tile (dead once P is formed), which lets two CTAs share an SM.
size_t prep_smem_bytes(int dk, int gate) {
    const size_t tiles = gate == 2 ? 3 * 64 * kLd + 64 * dk + 16 * dk : 2 * 64 * kLd;
    return sizeof(float) * (tiles + 2 * 64 * kLdA + 64 + 64 + 1024 + 64);
}

// out(r, n) (r, n < 16) = sum_{k < 16 nk} L(r, k) R(k, n) by one warp in fp32; lane owns row
// lane / 2 and columns 8 (lane % 2) .. + 7; result written through st(r, n, v).
template <class FL, class FR, class FS>
__device__ __forceinline__ void warp_tile16(FL L, FR R, int nk, FS st, int lane) {
    const int r = lane >> 1, n0 = 8 * (lane & 1);
    float acc[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m] = 0.f;
    for (int k = 0; k < 16 * nk; ++k) {
        const float l = L(r, k);
#pragma unroll
        for (int m = 0; m < 8; ++m) acc[m] = fmaf(l, R(k, n0 + m), acc[m]);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) st(r, n0 + m, acc[m]);
}

// T = (I + A)^{-1} for C = 64 in fp32 by 16 x 16 blocks (A, T: [64][kLdA]; M: 1024 floats):
// the diagonal blocks by right-looking substitution (four threads per column, the pivot
// value broadcast by a shuffle), then T_ij = -T_ii sum_{j <= k < i} A_ik T_kj: T_10 and
// T_32, then the lower-left 32 x 32 quarter through M = A[32:64, 0:32] T[0:32, 0:32].
// Only the lower triangle of T (diagonal included) is written.  All 256 threads; ends with a
// barrier.
__device__ __forceinline__ void solve64_blocked(const float *sA, float *sT, float *sM, int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    {
        const int o = 16 * (tid >> 6), c = (tid >> 2) & 15, part = tid & 3, owner = lane & ~3;
        float ar[4][16];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int q = 0; q < 16; ++q) ar[m][q] = sA[(o + part + 4 * m) * kLdA + o + q];
        float y[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) y[m] = (part + 4 * m == c) ? 1.f : 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 15; ++s2) {
            const float xs = __shfl_sync(0xffffffffu, y[s2 >> 2], owner | (s2 & 3));
#pragma unroll
            for (int m = 0; m < 4; ++m)
                if (part + 4 * m > s2) y[m] = fmaf(-ar[m][s2], xs, y[m]);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) sT[(o + part + 4 * m) * kLdA + o + c] = y[m];
    }
    __syncthreads();
    if (warp < 2) {
        const int i = 2 * warp + 1, j = 2 * warp;
        float *Ms = sM + 256 * warp;
        warp_tile16([&](int r, int k) { return sA[(16 * i + r) * kLdA + 16 * j + k]; },
                    [&](int k, int n) { return sT[(16 * j + k) * kLdA + 16 * j + n]; }, 1,
                    [&](int r, int n, float v) { Ms[r * 16 + n] = v; }, lane);
        __syncwarp();
        warp_tile16([&](int r, int k) { return sT[(16 * i + r) * kLdA + 16 * i + k]; },
                    [&](int k, int n) { return Ms[k * 16 + n]; }, 1,
                    [&](int r, int n, float v) { sT[(16 * i + r) * kLdA + 16 * j + n] = -v; }, lane);
    }
    __syncthreads();
    if (warp < 4) {   // M tile (rb, cb) = sum_{k = cb}^{1} A_{rb,k} T_{k,cb}
        const int rb = 2 + (warp >> 1), cb = warp & 1;
        float *Mt = sM + 256 * warp;
        warp_tile16([&](int r, int k) { return sA[(16 * rb + r) * kLdA + 16 * cb + k]; },
                    [&](int k, int n) { return sT[(16 * cb + k) * kLdA + 16 * cb + n]; }, 2 - cb,
                    [&](int r, int n, float v) { Mt[r * 16 + n] = v; }, lane);
    }
    __syncthreads();
    if (warp < 4) {   // T_{rb,cb} = -sum_{k = 2}^{rb} T_{rb,k} M_{k,cb}
        const int rb = 2 + (warp >> 1), cb = warp & 1;
        warp_tile16([&](int r, int k) { return sT[(16 * rb + r) * kLdA + 32 + k]; },
                    [&](int k, int n) { return sM[256 * (((k >> 4) << 1) | cb) + (k & 15) * 16 + n]; },
                    rb - 1,
                    [&](int r, int n, float v) { sT[(16 * rb + r) * kLdA + 16 * cb + n] = -v; }, lane);
    }
    __syncthreads();
}

template <int DK, typename Tin>
__global__ void __launch_bounds__(kThreads) chunk_prep_kernel(PrepArgs a) {
    // fp32 inputs: products at fp32 accuracy (three split-TF32 products); bf16 inputs, whose
    // results are held to the bf16 bound: one TF32 product (~2^-11 relative)
    constexpr bool kSplit = sizeof(Tin) == 4;
    extern __shared__ float4 smem4[];
    const bool chan = a.gate == 2;
    float *sK = reinterpret_cast<float *>(smem4);  // k, then left factor of A
    float *sQ = sK + 64 * kLd;                     // q, then left factor of P
    float *sR = chan ? sQ + 64 * kLd : sQ;         // right factor, then b*K*G, then b*V
    float *sG = sR + 64 * kLd;                     // [64][DK] cumulative log decay (channel)
    float *sF = sG + 64 * DK;                      // [16][DK] sub-chunk pair factors
    float *sA = chan ? sF + 16 * DK : sQ + 64 * kLd;   // [64][kLdA] A
    float *sT = sA + 64 * kLdA;                    // [64][kLdA] T = (I + A)^-1
    float *sB = sT + 64 * kLdA;                    // [64] beta
    float *sg = sB + 64;                           // [64] cumulative log decay (scalar)
    float *sM = sg + 64;                           // [1024] scratch of the blocked solve
    float *sNk = sM + 1024;                        // [64] 1 / |k_r| (1 unless normalised)

    const Tin *q = (const Tin *)a.q, *k = (const Tin *)a.k, *v = (const Tin *)a.v;
    const Tin *beta = (const Tin *)a.beta;
    const int C = a.C, NC = a.NC, dv = a.dv, tid = threadIdx.x;
    const int gate = a.gate;
    const int64_t n = blockIdx.x;            // (b*H + h)*NC + c
    const int c = (int)(n % NC);
    const int64_t bh = n / NC;
    const int64_t h = bh % a.H, b = bh / a.H;
    const int64_t t0 = (int64_t)c * C;
    const int Lc = (int)(a.T - t0 < (int64_t)C ? a.T - t0 : (int64_t)C);
    auto tok = [&](int r) -> int64_t { return (b * a.T + t0 + r) * a.H + h; };

    // 1. beta and the cumulative log decay (padded rows: beta = 0, log a = 0).
    const bool l2 = (a.fuse & kFuseL2) != 0;
    for (int r = tid; r < C; r += kThreads) {
        float br = r < Lc ? to_f32(beta[tok(r)]) : 0.f;
        if ((a.fuse & kFuseSigmoid) && r < Lc) br = to_f32(from_f32<Tin>(sigmoid_f(br)));
        sB[r] = br;
    }
    if (gate == 2) {
        // stage the chunk's log alpha rows (coalesced, all loads in flight), then scan
        for (int idx = tid; idx < C * (DK / 4); idx += kThreads) {
            const int r = idx / (DK / 4), c4 = 4 * (idx % (DK / 4));
            *reinterpret_cast<float4 *>(sG + r * DK + c4) =
                r < Lc ? *reinterpret_cast<const float4 *>(a.log_alpha + tok(r) * DK + c4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
        for (int ch = tid; ch < DK; ch += kThreads) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) {
                acc += sG[r * DK + ch];
                sG[r * DK + ch] = acc;
            }
        }
    } else if (tid < 32) {   // scalar gate: warp 0, two tokens per lane, one scan
        const int lane = tid, r = 2 * lane;
        const float l0 = (gate == 1 && r < Lc) ? a.log_alpha[tok(r)] : 0.f;
        const float l1 = (gate == 1 && r + 1 < Lc) ? a.log_alpha[tok(r + 1)] : 0.f;
        float p = l0 + l1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, p, o);
            if (lane >= o) p += y;
        }
        if (r < C) sg[r] = p - l1;
        if (r + 1 < C) sg[r + 1] = p;
    }
    // 2. k and q rows as fp32.
    for (int idx = tid; idx < C * (DK / 4); idx += kThreads) {
        const int r = idx / (DK / 4), c4 = 4 * (idx % (DK / 4));
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), qq = kk;
        if (r < Lc) {
            kk = load4(k + tok(r) * DK + c4);
            qq = load4(q + tok(r) * DK + c4);
        }
        *reinterpret_cast<float4 *>(sK + r * kLd + c4) = kk;
        *reinterpret_cast<float4 *>(sQ + r * kLd + c4) = qq;
    }
    __syncthreads();
    //    L2-normalised rows: four threads per row, each a quarter of the channels.
    {
        const int r = tid >> 2, part = tid & 3;
        float nk = 1.f;
        if (l2) {
            float sk2 = 0.f, sq2 = 0.f;
            for (int ch = part * (DK / 4); ch < (part + 1) * (DK / 4); ++ch) {
                sk2 = fmaf(sK[r * kLd + ch], sK[r * kLd + ch], sk2);
                sq2 = fmaf(sQ[r * kLd + ch], sQ[r * kLd + ch], sq2);
            }
            sk2 += __shfl_xor_sync(0xffffffffu, sk2, 1);
            sq2 += __shfl_xor_sync(0xffffffffu, sq2, 1);
            sk2 += __shfl_xor_sync(0xffffffffu, sk2, 2);
            sq2 += __shfl_xor_sync(0xffffffffu, sq2, 2);
            nk = rsqrtf(sk2 + kL2NormEps);
            const float nq = rsqrtf(sq2 + kL2NormEps);
            if (r < C)
                for (int ch = part * (DK / 4); ch < (part + 1) * (DK / 4); ++ch) {
                    sK[r * kLd + ch] *= nk;
                    sQ[r * kLd + ch] *= nq;
                }
        }
        if (part == 0 && r < C) sNk[r] = nk;
        if (l2) __syncthreads();
    }

    auto G = [&](int r, int ch) -> float { return gate == 2 ? sG[r * DK + ch] : sg[r]; };

    // 3. G_C, K*G_C/G and Q*G to the workspace.
    const int64_t wofs = n * (int64_t)C * DK;
    for (int ch = tid; ch < DK; ch += kThreads) a.ws.gam[n * DK + ch] = expf(G(C - 1, ch));
    if (gate == 2) {
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int r = idx / DK, ch = idx % DK;
            const float gr = G(r, ch);
            a.ws.Kd[wofs + idx] = sK[r * kLd + ch] * expf(G(C - 1, ch) - gr);
            a.ws.Qg[wofs + idx] = sQ[r * kLd + ch] * expf(gr);
        }
    } else {   // one decay per row: two exponentials per row, four channels per store
#pragma unroll 4
        for (int idx = tid; idx < C * (DK / 4); idx += kThreads) {
            const int r = idx / (DK / 4), c4 = 4 * (idx % (DK / 4));
            const float fk = expf(sg[C - 1] - sg[r]), fq = expf(sg[r]);
            const float4 kk = *reinterpret_cast<const float4 *>(sK + r * kLd + c4);
            const float4 qq = *reinterpret_cast<const float4 *>(sQ + r * kLd + c4);
            *reinterpret_cast<float4 *>(a.ws.Kd + wofs + r * DK + c4) =
                make_float4(kk.x * fk, kk.y * fk, kk.z * fk, kk.w * fk);
            *reinterpret_cast<float4 *>(a.ws.Qg + wofs + r * DK + c4) =
                make_float4(qq.x * fq, qq.y * fq, qq.z * fq, qq.w * fq);
        }
    }
    __syncthreads();

    // 4. A (strictly lower) and P (lower, diagonal included).
    const int nsub = C / kSub;
    if (gate == 2) {
        auto ref = [&](int j, int ch) -> float { return j == 0 ? 0.f : sG[(kSub * j - 1) * DK + ch]; };
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int r = idx / DK, ch = idx % DK, i = r / kSub;
            const float gr = sG[r * DK + ch], ri = ref(i, ch);
            sR[r * kLd + ch] = sK[r * kLd + ch] * expf(ri - gr);  // exponent in [0, 16 max|log a|]
        }
        for (int idx = tid; idx < 16 * DK; idx += kThreads) {
            const int pr = idx / DK, ch = idx % DK, i = pr / 4, j = pr % 4;
            sF[idx] = (j < i && i < nsub) ? expf(ref(i, ch) - ref(j, ch)) : 1.f;
        }
        __syncthreads();
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int r = idx / DK, ch = idx % DK;
            const float f = expf(sG[r * DK + ch] - ref(r / kSub, ch));   // exponent <= 0
            sK[r * kLd + ch] *= f;
            sQ[r * kLd + ch] *= f;
        }
        __syncthreads();
    }
    const int64_t pofs = n * (int64_t)C * C;
    const int warp = tid >> 5, lane = tid & 31;
    if (gate != 2) {
        // X = K K^T and Q K^T on the lower tiles (split-TF32 warp tiles, about fp32
        // accuracy), then the decay exp(g_r - g_s) (exponent <= 0) and beta_r
        auto upper = [](int r0, int n0) { return n0 > r0 + 15; };
        tc::rows_dot_rows<kSplit>(sK, kLd, sK, kLd, C, C, DK, warp, kThreads / 32, lane, upper,
                          [&](int r, int s2, float v) {
                              sA[r * kLdA + s2] = s2 < r ? sB[r] * v * expf(sg[r] - sg[s2]) : 0.f;
                          });
        tc::rows_dot_rows<kSplit>(sQ, kLd, sK, kLd, C, C, DK, warp, kThreads / 32, lane, upper,
                          [&](int r, int s2, float v) {
                              a.ws.P[pofs + r * C + s2] = s2 <= r ? v * expf(sg[r] - sg[s2]) : 0.f;
                          });
        for (int idx = tid; idx < C * C; idx += kThreads) {   // the skipped tiles: zeros
            const int r = idx / C, s2 = idx % C;
            if ((s2 & ~7) > (r | 15)) {
                sA[r * kLdA + s2] = 0.f;
                a.ws.P[pofs + idx] = 0.f;   // zero above the diagonal
            }
        }
    } else {
        const int r = tid >> 2;
        for (int m = 0; m < 16; ++m) {
            const int s = (tid & 3) + 4 * m;
            if (r >= C || s >= C) continue;
            float ak = 0.f, aq = 0.f;
            if (s <= r) {
                const float *lk = sK + r * kLd, *lq = sQ + r * kLd;
                {   // per-channel gate: factors around the sub-chunk references
                    const float *rs = sR + s * kLd;
                    const int i = r / kSub, j = s / kSub;
                    if (i == j) {
                        for (int ch = 0; ch < DK; ch += 4) {
                            const float4 x = *reinterpret_cast<const float4 *>(lk + ch);
                            const float4 y = *reinterpret_cast<const float4 *>(lq + ch);
                            const float4 z = *reinterpret_cast<const float4 *>(rs + ch);
                            ak += x.x * z.x + x.y * z.y + x.z * z.z + x.w * z.w;
                            aq += y.x * z.x + y.y * z.y + y.z * z.z + y.w * z.w;
                        }
                    } else {
                        const float *f = sF + (i * 4 + j) * DK;
                        for (int ch = 0; ch < DK; ch += 4) {
                            const float4 x = *reinterpret_cast<const float4 *>(lk + ch);
                            const float4 y = *reinterpret_cast<const float4 *>(lq + ch);
                            const float4 z = *reinterpret_cast<const float4 *>(rs + ch);
                            const float4 w = *reinterpret_cast<const float4 *>(f + ch);
                            const float4 zw = make_float4(z.x * w.x, z.y * w.y, z.z * w.z, z.w * w.w);
                            ak += x.x * zw.x + x.y * zw.y + x.z * zw.z + x.w * zw.w;
                            aq += y.x * zw.x + y.y * zw.y + y.z * zw.z + y.w * zw.w;
                        }
                    }
                }
            }
            sA[r * kLdA + s] = (s < r) ? sB[r] * ak : 0.f;
            a.ws.P[pofs + r * C + s] = aq;   // zero above the diagonal
        }
    }
    __syncthreads();

    // 5. T = (I + A)^{-1}: blocked for C = 64; otherwise by forward substitution, column j
    //    by the 4 lanes tid/4 == j: T_rj = delta_rj - sum_{j <= s < r} A_rs T_sj.
    if (C == 64) {
        solve64_blocked(sA, sT, sM, tid);
    } else {
        const int j = tid >> 2, part = tid & 3;
        for (int r = part; r < C; r += 4)
            if (j < C) sT[r * kLdA + j] = (r == j) ? 1.f : 0.f;
        __syncwarp();
        for (int r = 1; r < C; ++r) {
            float acc = 0.f;
            if (j < r)
                for (int s = j + part; s < r; s += 4) acc += sA[r * kLdA + s] * sT[s * kLdA + j];
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0 && j < r) sT[r * kLdA + j] = -acc;
            __syncwarp();
        }
    }
    if (a.T_out) {   // T for the backward (lower triangle, diagonal included)
        __syncthreads();
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int r = idx / C, s2 = idx % C;
            a.T_out[n * (int64_t)C * C + idx] = s2 <= r ? sT[r * kLdA + s2] : 0.f;
        }
    }
    // 6. W = T diag(b) (K*G):  rows b_s k_s exp(g_s) (exponent <= 0), four channels per
    //    step; k as held (scalar gate or none) or reloaded raw (the per-channel gate has
    //    rescaled sK)
#pragma unroll 4
    for (int idx = tid; idx < C * (DK / 4); idx += kThreads) {
        const int s = idx / (DK / 4), c4 = 4 * (idx % (DK / 4));
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s < Lc) {
            if (gate == 2) {
                kk = load4(k + tok(s) * DK + c4);
                const float f = sNk[s];
                kk = make_float4(kk.x * f, kk.y * f, kk.z * f, kk.w * f);
            } else {
                kk = *reinterpret_cast<const float4 *>(sK + s * kLd + c4);
            }
        }
        const float b = sB[s];
        *reinterpret_cast<float4 *>(sR + s * kLd + c4) =
            make_float4(b * kk.x * expf(G(s, c4)), b * kk.y * expf(G(s, c4 + 1)),
                        b * kk.z * expf(G(s, c4 + 2)), b * kk.w * expf(G(s, c4 + 3)));
    }
    __syncthreads();
    // the [C][N] product T (lower triangular, as stored: entries above the diagonal are
    // not read) times sR, written to `dst` with row stride N: warp tiles of 16 rows x
    // N / (8 warps / (C / 16)) columns
    auto t_times_r = [&](int N, float *dst) {
        const int rbs = C / 16, groups = (kThreads / 32) / rbs, ncol = N / groups;
        const int r0 = 16 * (warp % rbs), n0 = (warp / rbs) * ncol, g8 = lane >> 2, t4 = lane & 3;
        float acc[8][4];
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[t][u] = 0.f;
        tc::rows_times_cols<kSplit>(acc, ncol / 8, [&](int rr, int kk) { return kk <= rr ? sT[rr * kLdA + kk] : 0.f; },
                            [&](int kk, int nn) { return sR[kk * kLd + nn]; }, r0, n0, C, g8, t4);
#pragma unroll
        for (int t = 0; t < 8; ++t)
            if (8 * t < ncol)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    dst[(r0 + g8 + 8 * (u >> 1)) * N + n0 + 8 * t + 2 * t4 + (u & 1)] = acc[t][u];
    };
    t_times_r(DK, a.ws.W + wofs);
    __syncthreads();
    //    U = T diag(b) V.
#pragma unroll 4
    for (int idx = tid; idx < C * (dv / 4); idx += kThreads) {
        const int s = idx / (dv / 4), j4 = 4 * (idx % (dv / 4));
        float4 vv = s < Lc ? load4(v + tok(s) * dv + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float b = sB[s];
        *reinterpret_cast<float4 *>(sR + s * kLd + j4) = make_float4(b * vv.x, b * vv.y, b * vv.z, b * vv.w);
    }
    __syncthreads();
    const int64_t uofs = n * (int64_t)C * dv;
    t_times_r(dv, a.ws.U + uofs);
}

constexpr int kDvt = 32;   // state columns per CTA of the state pass

size_t state_smem_bytes(int dk) {
    return sizeof(float) * (size_t)(dk * kDvt + 3 * 64 * (dk + 4) + 2 * 64 * kDvt + 64 * kLdA + dk);
}

template <int DK, typename Tout>
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(StateArgs a) {
    constexpr int LD = DK + 4;
    extern __shared__ float4 smem4[];
    float *sS = reinterpret_cast<float *>(smem4);  // [DK][32] state columns
    float *sW = sS + DK * kDvt;                    // [64][LD]
    float *sQg = sW + 64 * LD;                     // [64][LD]
    float *sKd = sQg + 64 * LD;                    // [64][LD]
    float *sU = sKd + 64 * LD;                     // [64][32]
    float *sE = sU + 64 * kDvt;                    // [64][32]
    float *sP = sE + 64 * kDvt;                    // [64][kLdA]
    float *sGam = sP + 64 * kLdA;                  // [DK]

    const int tiles = a.dv / kDvt;
    const int C = a.C, NC = a.NC, dv = a.dv, tid = threadIdx.x;
    const int j = tid & 31, rg = tid >> 5;  // column in tile, row group (8 groups)
    Tout *out = (Tout *)a.out;
    // this CTA's chain, column tile and chunk range [c_begin, c_end); its start state (NULL:
    // zero; `identity`: I) and end state, both with row stride `ld`
    int64_t bh = blockIdx.x / tiles;
    int jt = blockIdx.x % tiles, c_begin = 0, c_end = NC, ld = dv;
    const float *s_init = a.init_state ? a.init_state + bh * DK * dv : nullptr;
    float *s_fin = a.final_state ? a.final_state + bh * DK * dv : nullptr;
    bool identity = false, use_u = true;
    if (a.role != 0) {
        const int per = a.role == 1 ? tiles + DK / kDvt : tiles;
        const int64_t idx = blockIdx.x / per;
        const int seg = (int)(idx % a.nseg);
        jt = blockIdx.x % per;
        bh = idx / a.nseg;
        c_begin = seg * a.seg_len;
        c_end = min(NC, c_begin + a.seg_len);
        const size_t slot = (size_t)(bh * a.nseg + seg);
        if (a.role == 1) {
            out = nullptr;
            s_init = nullptr;
            if (jt >= tiles) {   // the transition: DK columns
                jt -= tiles;
                identity = true;
                use_u = false;
                ld = DK;
                s_fin = a.ws_phi + slot * DK * DK;
            } else {
                s_fin = a.ws_s0 + slot * DK * dv;
            }
        } else {
            s_init = a.ws_start + slot * DK * dv;
            s_fin = (seg == a.nseg - 1 && a.final_state) ? a.final_state + bh * DK * dv : nullptr;
        }
    }
    const int64_t h = bh % a.H, b = bh / a.H;
    const int col = jt * kDvt + j;

    for (int i = rg; i < DK; i += 8)
        sS[i * kDvt + j] = s_init ? s_init[(int64_t)i * ld + col] : (identity && i == col ? 1.f : 0.f);

    for (int c = c_begin; c < c_end; ++c) {
        const int64_t n = bh * NC + c;
        const int64_t t0 = (int64_t)c * C;
        const int Lc = (int)(a.T - t0 < (int64_t)C ? a.T - t0 : (int64_t)C);
        const float *W = a.ws.W + n * (int64_t)C * DK;
        const float *Qg = a.ws.Qg + n * (int64_t)C * DK;
        const float *Kd = a.ws.Kd + n * (int64_t)C * DK;
        const float *U = a.ws.U + n * (int64_t)C * dv;
        const float *P = a.ws.P + n * (int64_t)C * C;
        __syncthreads();   // previous chunk's readers of the staged tiles are done
        for (int idx = tid; idx < C * (DK / 4); idx += kThreads) {
            const int r = idx / (DK / 4), c4 = 4 * (idx % (DK / 4));
            *reinterpret_cast<float4 *>(sW + r * LD + c4) = load4(W + r * DK + c4);
            *reinterpret_cast<float4 *>(sQg + r * LD + c4) = load4(Qg + r * DK + c4);
            *reinterpret_cast<float4 *>(sKd + r * LD + c4) = load4(Kd + r * DK + c4);
        }
        for (int idx = tid; idx < C * kDvt; idx += kThreads)
            sU[idx] = use_u ? U[(idx / kDvt) * dv + jt * kDvt + idx % kDvt] : 0.f;
        for (int idx = tid; idx < C * C; idx += kThreads) sP[(idx / C) * kLdA + idx % C] = P[idx];
        for (int i = tid; i < DK; i += kThreads) sGam[i] = a.ws.gam[n * DK + i];
        if (a.ckpt)   // the state at this chunk's start (sS is final after the barrier above)
            for (int i = rg; i < DK; i += 8) a.ckpt[(n * DK + i) * dv + col] = sS[i * kDvt + j];
        __syncthreads();

        // E = U - W S and the inter-chunk read (Q*G) S, rows r = rg + 8m.
        float e[8], o[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) { e[m] = 0.f; o[m] = 0.f; }
        for (int i = 0; i < DK; i += 4) {
            const float s0 = sS[(i + 0) * kDvt + j], s1 = sS[(i + 1) * kDvt + j];
            const float s2 = sS[(i + 2) * kDvt + j], s3 = sS[(i + 3) * kDvt + j];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = rg + 8 * m;
                if (r < C) {
                    const float4 w = *reinterpret_cast<const float4 *>(sW + r * LD + i);
                    const float4 qg = *reinterpret_cast<const float4 *>(sQg + r * LD + i);
                    e[m] += w.x * s0 + w.y * s1 + w.z * s2 + w.w * s3;
                    o[m] += qg.x * s0 + qg.y * s1 + qg.z * s2 + qg.w * s3;
                }
            }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int r = rg + 8 * m;
            if (r < C) sE[r * kDvt + j] = sU[r * kDvt + j] - e[m];
        }
        __syncthreads();
        // O = (Q*G) S + P E  (P lower triangular, diagonal included): eight rows at once;
        // skipped when the outputs are not wanted (the backward's recompute)
        if (out) {
#pragma unroll 4
            for (int s = 0; s < C; ++s) {
                const float es = sE[s * kDvt + j];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int r = rg + 8 * m;
                    if (r < C && s <= r) o[m] = fmaf(sP[r * kLdA + s], es, o[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = rg + 8 * m;
                if (r < Lc) {
                    float acc = o[m];
                    const int64_t oi = ((b * a.T + t0 + r) * a.H + h) * dv + col;
                    if (a.z)
                        acc *= silu_f(a.z_bf16 ? to_f32(((const __nv_bfloat16 *)a.z)[oi])
                                               : ((const float *)a.z)[oi]);
                    out[oi] = from_f32<Tout>(acc);
                }
            }
        }
        // S <- Diag(G_C) S + (K*G_C/G)^T E: DK / 8 independent sums per thread
        {
            constexpr int NR = DK / 8;
            float acc[NR];
#pragma unroll
            for (int m = 0; m < NR; ++m) acc[m] = sGam[rg + 8 * m] * sS[(rg + 8 * m) * kDvt + j];
            for (int r = 0; r < C; ++r) {
                const float e = sE[r * kDvt + j];
#pragma unroll
                for (int m = 0; m < NR; ++m) acc[m] = fmaf(sKd[r * LD + rg + 8 * m], e, acc[m]);
            }
#pragma unroll
            for (int m = 0; m < NR; ++m) sS[(rg + 8 * m) * kDvt + j] = acc[m];
        }
    }
    if (s_fin) {
        __syncthreads();
        for (int i = rg; i < DK; i += 8) s_fin[(int64_t)i * ld + col] = sS[i * kDvt + j];
    }
}

// Segment chaining: per chain, S_start(0) = S_0 and S_start(p + 1) = Phi_p S_start(p) + S0_p
// (Phi_p [DK][DK], S0_p and S_start [DK][dv], fp32).  One CTA per (chain, 32 state columns);
// each Phi_p is staged in shared memory (combine_smem_bytes), each thread keeping DK / 8 rows
// of one column.
constexpr size_t combine_smem_bytes(int dk) { return sizeof(float) * (size_t)dk * (dk + 1); }
template <int DK>
__global__ void __launch_bounds__(kThreads) seg_combine_simt_kernel(const float *__restrict__ init_state,
                                                                    const float *__restrict__ phi,
                                                                    const float *__restrict__ s0,
                                                                    float *__restrict__ start, int dv,
                                                                    int nseg) {
    __shared__ float S[DK][kDvt + 1];
    extern __shared__ float4 phi_s4[];
    float (*P)[DK + 1] = reinterpret_cast<float (*)[DK + 1]>(phi_s4);
    constexpr int NR = DK / 8;
    const int tiles = dv / kDvt;
    const int jt = blockIdx.x % tiles;
    const int64_t bh = blockIdx.x / tiles;
    const int tid = threadIdx.x, j = tid & 31, rg = tid >> 5;
    const int col = jt * kDvt + j;
    for (int i = rg; i < DK; i += 8) S[i][j] = init_state ? init_state[(bh * DK + i) * dv + col] : 0.f;
    for (int p = 0; p < nseg; ++p) {
        const int64_t slot = bh * nseg + p;
        __syncthreads();   // S is complete; the previous Phi's readers are done
        for (int i = rg; i < DK; i += 8) start[(slot * DK + i) * dv + col] = S[i][j];
        if (p + 1 == nseg) break;
        for (int idx = tid; idx < DK * DK; idx += kThreads) P[idx / DK][idx % DK] = phi[slot * DK * DK + idx];
        float acc[NR];
#pragma unroll
        for (int m = 0; m < NR; ++m) acc[m] = s0[(slot * DK + rg + 8 * m) * dv + col];
        __syncthreads();
        for (int k = 0; k < DK; ++k) {
            const float sk = S[k][j];
#pragma unroll
            for (int m = 0; m < NR; ++m) acc[m] = fmaf(P[rg + 8 * m][k], sk, acc[m]);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < NR; ++m) S[rg + 8 * m][j] = acc[m];
    }
}

template <int DK, typename Tin, typename Tout>
int launch_simt_t(const PrepArgs &pa, StateArgs sa, cudaStream_t stream, bool prep_only, float *seg_ws) {
    const size_t ps = prep_smem_bytes(DK, pa.gate), ss = state_smem_bytes(DK);
    if (cudaFuncSetAttribute(chunk_prep_kernel<DK, Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)prep_smem_bytes(DK, 2)) != cudaSuccess ||
        cudaFuncSetAttribute(chunk_prep_kernel<DK, Tin>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             100) != cudaSuccess)
        return kErrCuda;
    if (cudaFuncSetAttribute(chunk_state_kernel<DK, Tout>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss) != cudaSuccess)
        return kErrCuda;
    const int64_t nprep = pa.B * pa.H * pa.NC;
    const int64_t bh = sa.B * sa.H, tiles = sa.dv / kDvt;
    if (nprep > 0) chunk_prep_kernel<DK, Tin><<<(unsigned)nprep, kThreads, ps, stream>>>(pa);
    if (prep_only) return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
    int nseg = 1, seg_len = sa.NC;
    if (seg_ws) simt_segments(bh, DK, sa.dv, sa.NC, &nseg, &seg_len);
    if (nseg <= 1) {
        chunk_state_kernel<DK, Tout><<<(unsigned)(bh * tiles), kThreads, ss, stream>>>(sa);
        return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
    }
    // segments: end states and transitions, chaining, then outputs
    const size_t ns = (size_t)bh * nseg;
    sa.nseg = nseg;
    sa.seg_len = seg_len;
    sa.ws_phi = seg_ws;
    sa.ws_s0 = seg_ws + ns * DK * DK;
    float *start = sa.ws_s0 + ns * DK * sa.dv;
    sa.ws_start = start;
    sa.role = 1;
    chunk_state_kernel<DK, Tout><<<(unsigned)(ns * (tiles + DK / kDvt)), kThreads, ss, stream>>>(sa);
    constexpr int cs = (int)combine_smem_bytes(DK);
    if (cudaFuncSetAttribute(seg_combine_simt_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, cs) !=
        cudaSuccess)
        return kErrCuda;
    seg_combine_simt_kernel<DK><<<(unsigned)(bh * tiles), kThreads, cs, stream>>>(
        sa.init_state, sa.ws_phi, sa.ws_s0, start, sa.dv, nseg);
    sa.role = 2;
    chunk_state_kernel<DK, Tout><<<(unsigned)(ns * tiles), kThreads, ss, stream>>>(sa);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

// Few long chains: segments of at least 16 chunks, as many as let the first segment pass (one
// CTA per 32 columns of the end state and of the transition, per segment) fill the 152 SMs
// once.  nseg = 1: not split.
void simt_segments(int64_t chains, int dk, int dv, int NC, int *nseg, int *seg_len) {
    constexpr int64_t kGpuSms = 152;
    *nseg = 1;
    *seg_len = NC;
    const int64_t per = chains * ((dv + dk) / kDvt);
    if (NC < 32 || per > kGpuSms / 2) return;
    const int n = (int)std::min<int64_t>(NC / 16, kGpuSms / per);
    if (n < 2) return;
    const int len = (NC + n - 1) / n;
    *seg_len = len;
    *nseg = (NC + len - 1) / len;
}

size_t simt_segment_floats(const ChunkProblem &p) {
    int nseg, len;
    simt_segments(p.B * p.H, p.dk, p.dv, p.NC, &nseg, &len);
    if (nseg <= 1) return 0;
    const size_t ns = (size_t)(p.B * p.H) * nseg;
    return ns * p.dk * p.dk + 2 * ns * p.dk * p.dv;
}

int launch_chunk_simt(const ChunkProblem &p, const ChunkWorkspace &ws, cudaStream_t stream,
                      float *T_out, float *ckpt, bool prep_only, float *seg_ws) {
    PrepArgs pa{p.q, p.k, p.v, p.log_alpha, p.beta, p.B, p.T, p.H, p.dv, p.C, p.NC, p.gate, p.fuse, ws,
                T_out};
    StateArgs sa{p.init_state, p.out, p.final_state, (p.fuse & kFuseGate) ? p.z : nullptr, p.in_bf16,
                 p.B, p.T, p.H, p.dv, p.C, p.NC, ws, ckpt, 0, 1, p.NC, nullptr, nullptr, nullptr};
    if (ckpt) seg_ws = nullptr;   // the backward's recompute walks whole chains
    using bf = __nv_bfloat16;
    const bool ib = p.in_bf16, ob = p.out_bf16;
    if (p.dk == 128) {
        if (ib && ob) return launch_simt_t<128, bf, bf>(pa, sa, stream, prep_only, seg_ws);
        if (ib) return launch_simt_t<128, bf, float>(pa, sa, stream, prep_only, seg_ws);
        if (ob) return launch_simt_t<128, float, bf>(pa, sa, stream, prep_only, seg_ws);
        return launch_simt_t<128, float, float>(pa, sa, stream, prep_only, seg_ws);
    }
    if (p.dk == 64) {
        if (ib && ob) return launch_simt_t<64, bf, bf>(pa, sa, stream, prep_only, seg_ws);
        if (ib) return launch_simt_t<64, bf, float>(pa, sa, stream, prep_only, seg_ws);
        if (ob) return launch_simt_t<64, float, bf>(pa, sa, stream, prep_only, seg_ws);
        return launch_simt_t<64, float, float>(pa, sa, stream, prep_only, seg_ws);
    }
    return kErrUnsupported;
}

}  // namespace dr
