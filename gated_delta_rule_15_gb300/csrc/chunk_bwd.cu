// chunk_bwd.cu -- backward of the chunkwise forward: the gradients of
// L = <d_out, out> + <d_final, final_state> with respect to q, k, v, log alpha, beta and the
// initial state, with fp32 sums and every contraction as a TF32 warp tile (tc_common.cuh:
// three split products at fp32 accuracy for fp32 inputs, one for bf16 inputs).
//
// The pages ask for chunkwise kernels for training (page "linear-attention gated-deltanet
// guide", section 5) and print no backward; this one differentiates the chunk form of
// chunk_simt.cu.  Per chunk, started from S0, with g_r the cumulative log decay, G = exp(g),
// gamma = G at the chunk's last token and the pair factor D_rs = exp(g_r - g_s) (s <= r, per
// key channel, <= 1):
//
//   A_rs = b_r sum_i k_ri k_si D_rs,i (s < r),  T = (I + A)^-1,  R = diag(b) (V - (K*G) S0),
//   E = T R,  P_rs = sum_i q_ri k_si D_rs,i (s <= r),  O = (Q*G) S0 + P E,
//   S_C = Diag(gamma) S0 + Kd^T E,  Kd_r = k_r * exp(g_C - g_r).
//
// Given dO and dS_C:
//   dE = P^T dO + Kd dS_C,   dR = T^T dE,   dP = tril(dO E^T),   dA = -stril(dR E^T)
//   dS0 = Diag(gamma) dS_C + (Q*G)^T dO - W^T dE          (W = T diag(b) (K*G))
//   dv_r = b_r dR_r,   db_r = dR_r . (v_r - ((K*G) S0)_r) + sum_{s<r} dA_rs A_rs / b_r
//   and dq, dk, dg from the products holding q, k and g (chunk_grad_kernel, phase by phase);
//   d log alpha_t = sum_{r >= t} dg_r, the last token's dg also taking the terms of gamma.
//
// Three steps after the CUDA-core forward has recomputed W, U, Q*G, Kd, P, gamma and T, and
// a forward pass (the tensor-core kernel where it serves the problem, else the CUDA-core
// state pass) the state at every chunk's start (the checkpoints):
//   chunk_dstate_kernel  one CTA per (b, h, 64 state columns), chunks in reverse: stores
//                        dS_C of every chunk and returns dS0 of the first;
//   chunk_grad_kernel    one CTA per (b, h, chunk), all chunks in parallel: every gradient
//                        of the chunk's tokens.
#include "chunk_layout.h"
#include "common.cuh"
#include "tc_common.cuh"

namespace dr {
namespace {

constexpr int kThreads = 256;
constexpr int kLdA = 65;   // padded row stride of [64][64] tiles
constexpr int kLdP = 68;   // row stride of the reverse pass's P tile (16-byte rows)
constexpr int kDvt = 64;   // state columns per CTA of the reverse pass
constexpr int kLdC = kDvt + 8;   // row stride of the reverse pass's column tiles (conflict-free
                                 // tensor-core fragments)
constexpr int kSlice = 32; // rows of a [dk][dv] state matrix staged at a time
constexpr int kGThreads = 512;   // per-chunk gradient kernel: 8 threads per token row
constexpr int kParts = 8;
constexpr int kLdM = kSlice + 4;   // row stride of the gradient kernel's product slices

// 16-byte asynchronous global -> shared copy (both addresses 16-byte aligned)
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_all;" ::: "memory");
}
// Prefetch of `bytes` (a multiple of 16, 16-byte-aligned address) into L2, no completion
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Workspace of the backward, in floats, after the forward's slabs: T [n][C][C], checkpoints
// [n][dk][dv], dS_C [n][dk][dv].
struct BwdWorkspace {
    ChunkWorkspace fw;
    float *T, *ckpt, *dsc;
    float *tc;   // the tensor-core forward's workspace (checkpoint recompute)
};

// The tensor-core forward's own workspace (segments of few long chains) when it writes the
// checkpoints, in floats.
size_t tc_ws_floats(const ChunkProblem &p) {
    return chunk_tc_supported(p) ? (chunk_tc_workspace_bytes(p, true) + 3) / 4 : 0;
}

size_t bwd_floats(const ChunkProblem &p) {
    const int64_t n = p.B * p.H * p.NC;
    return simt_workspace_floats(p.B, p.H, p.NC, p.C, p.dk, p.dv) +
           (size_t)(n * ((int64_t)p.C * p.C + 2 * (int64_t)p.dk * p.dv)) + tc_ws_floats(p);
}

BwdWorkspace bwd_carve(void *base, const ChunkProblem &p) {
    BwdWorkspace w;
    w.fw = simt_workspace_carve(base, p.B, p.H, p.NC, p.C, p.dk, p.dv);
    const int64_t n = p.B * p.H * p.NC;
    float *f = (float *)base + simt_workspace_floats(p.B, p.H, p.NC, p.C, p.dk, p.dv);
    w.T = f;     f += n * p.C * p.C;
    w.ckpt = f;  f += n * (int64_t)p.dk * p.dv;
    w.dsc = f;   f += n * (int64_t)p.dk * p.dv;
    w.tc = f;
    return w;
}

struct DStateArgs {
    const void *d_out;
    const float *d_final;
    float *d_init;
    BwdWorkspace ws;
    int64_t B, T, H;
    int dv, C, NC;
};

size_t dstate_smem_bytes(int dk) {
    return sizeof(float) * (size_t)(dk * kLdC + 3 * 64 * (dk + 4) + 2 * 64 * kLdC + 64 * kLdP + dk);
}

// Reverse state-gradient pass: dS starts as d_final; for each chunk, last first, it is
// stored as that chunk's dS_C, then  dE = P^T dO + Kd dS,  dS <- Diag(gamma) dS + (Q*G)^T dO
// - W^T dE.  Column j of dS only meets column j of dO, so a CTA owns 64 columns (every
// (b, h) in at most two rounds of CTAs over the GPU, each reading the chunk's operands
// once for its 64 columns).  A chunk's
// operands arrive by 16-byte asynchronous copies behind one wait, and the next chunk's are
// prefetched into L2 meanwhile: one CTA fits an SM, so the chain of chunks is otherwise
// paced by global-load latency.  Both products run as TF32 warp tiles (kSplit: three split
// products at fp32 accuracy, for fp32 inputs).
template <int DK, typename Tg, bool kSplit>
__global__ void __launch_bounds__(kThreads) chunk_dstate_kernel(DStateArgs a) {
    constexpr int LD = DK + 4;
    extern __shared__ float4 smem4[];
    float *sDS = reinterpret_cast<float *>(smem4);  // [DK][kLdC]
    float *sW = sDS + DK * kLdC;                    // [64][LD]
    float *sQg = sW + 64 * LD;                      // [64][LD]
    float *sKd = sQg + 64 * LD;                     // [64][LD]
    float *sDO = sKd + 64 * LD;                     // [64][kLdC]
    float *sDE = sDO + 64 * kLdC;                   // [64][kLdC]
    float *sP = sDE + 64 * kLdC;                    // [64][kLdP]
    float *sGam = sP + 64 * kLdP;                   // [DK]

    const int tiles = a.dv / kDvt;
    const int jt = blockIdx.x % tiles;
    const int64_t bh = blockIdx.x / tiles;
    const int64_t h = bh % a.H, b = bh / a.H;
    const int C = a.C, NC = a.NC, dv = a.dv, tid = threadIdx.x;
    const int j = tid & 31, rg = tid >> 5;
    const int col = jt * kDvt + j;
    const Tg *dout = (const Tg *)a.d_out;

    for (int i = rg; i < DK; i += 8)
        for (int jj = j; jj < kDvt; jj += 32)
            sDS[i * kLdC + jj] = a.d_final ? a.d_final[(bh * DK + i) * dv + col + jj - j] : 0.f;

    for (int c = NC - 1; c >= 0; --c) {
        const int64_t n = bh * NC + c;
        const int64_t t0 = (int64_t)c * C;
        const int Lc = (int)(a.T - t0 < (int64_t)C ? a.T - t0 : (int64_t)C);
        const float *W = a.ws.fw.W + n * (int64_t)C * DK;
        const float *Qg = a.ws.fw.Qg + n * (int64_t)C * DK;
        const float *Kd = a.ws.fw.Kd + n * (int64_t)C * DK;
        const float *P = a.ws.fw.P + n * (int64_t)C * C;
        const float *gam = a.ws.fw.gam + n * DK;
        __syncthreads();   // the previous chunk's readers are done
        for (int idx = tid; idx < C * (DK / 4); idx += kThreads) {
            const int r = idx / (DK / 4), c4 = 4 * (idx % (DK / 4));
            cp_async16(sW + r * LD + c4, W + r * DK + c4);
            cp_async16(sQg + r * LD + c4, Qg + r * DK + c4);
            cp_async16(sKd + r * LD + c4, Kd + r * DK + c4);
        }
        for (int idx = tid; idx < C * (C / 4); idx += kThreads) {
            const int r = idx / (C / 4), c4 = 4 * (idx % (C / 4));
            cp_async16(sP + r * kLdP + c4, P + r * C + c4);
        }
        for (int idx = tid; idx < DK / 4; idx += kThreads) cp_async16(sGam + 4 * idx, gam + 4 * idx);
        {   // dO's kDvt columns: every load of this thread issued before its stores
            constexpr int kPer = 64 * kDvt / kThreads;   // >= C * kDvt / kThreads
            float dov[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int idx = tid + u * kThreads, r = idx / kDvt, jj = idx % kDvt;
                dov[u] = (idx < C * kDvt && r < Lc)
                             ? to_f32(dout[((b * a.T + t0 + r) * a.H + h) * dv + jt * kDvt + jj]) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u)
                if (tid + u * kThreads < C * kDvt) sDO[((tid + u * kThreads) / kDvt) * kLdC + (tid + u * kThreads) % kDvt] = dov[u];
        }
        for (int i = rg; i < DK; i += 8)
            for (int jj = j; jj < kDvt; jj += 32) a.ws.dsc[(n * DK + i) * dv + col + jj - j] = sDS[i * kLdC + jj];
        cp_async_commit_wait_all();
        __syncthreads();
        if (c > 0) {   // the next chunk's operands into L2 while this one computes
            if (tid == 0) {
                prefetch_l2(W - C * DK, (uint32_t)(C * DK * 4));
                prefetch_l2(Qg - C * DK, (uint32_t)(C * DK * 4));
                prefetch_l2(Kd - C * DK, (uint32_t)(C * DK * 4));
                prefetch_l2(P - C * C, (uint32_t)(C * C * 4));
            } else if (tid > 32 && tid <= 32 + C && t0 - C + (tid - 33) < a.T) {
                const int r = tid - 33;   // dO rows of the next chunk (this CTA's columns)
                const Tg *row = dout + ((b * a.T + t0 - C + r) * a.H + h) * dv + jt * kDvt;
                for (int e = 0; e < kDvt; e += 128 / (int)sizeof(Tg))
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + e));
            }
        }
        // dE [C][kDvt] = P^T dO + Kd dS (P lower triangular): warp w, rows 16 (w % 4) ..,
        // columns kDvt/2 (w / 4) .. (four tiles of 8)
        const int g8 = j >> 2, t4 = j & 3;
        {
            constexpr int NT = kDvt / 16;
            const int r0 = 16 * (rg & 3), n0 = (kDvt / 2) * (rg >> 2);
            float acc[NT][4];
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u) acc[t][u] = 0.f;
            if (r0 < C) {
                tc::rows_times_cols<kSplit>(acc, NT, [&](int rr, int kk) { return sP[kk * kLdP + rr]; },
                                            [&](int kk, int nn) { return sDO[kk * kLdC + nn]; }, r0, n0, C, g8, t4);
                tc::rows_times_cols<kSplit>(acc, NT, [&](int rr, int kk) { return sKd[rr * LD + kk]; },
                                            [&](int kk, int nn) { return sDS[kk * kLdC + nn]; }, r0, n0, DK, g8, t4);
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        sDE[(r0 + g8 + 8 * (u >> 1)) * kLdC + n0 + 8 * t + 2 * t4 + (u & 1)] = acc[t][u];
            }
        }
        __syncthreads();
        // dS <- Diag(gamma) dS + (Q*G)^T dO - W^T dE  [DK][kDvt] (its own entries only, in
        // place): DK = 128, warp w owns row block w and all 8 column tiles; DK = 64, row block
        // w % 4 and the column half w / 4
        {
            constexpr int RB = DK / 16, NTS = RB * (kDvt / 8) / 8;   // tiles per warp
            const int i0 = 16 * (rg % RB), n0 = 8 * NTS * (rg / RB);
            float acc[NTS][4];
#pragma unroll
            for (int t = 0; t < NTS; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + g8 + 8 * (u >> 1), jj = n0 + 8 * t + 2 * t4 + (u & 1);
                    acc[t][u] = sGam[i] * sDS[i * kLdC + jj];
                }
            tc::rows_times_cols<kSplit>(acc, NTS, [&](int ii, int kk) { return sQg[kk * LD + ii]; },
                                        [&](int kk, int nn) { return sDO[kk * kLdC + nn]; }, i0, n0, C, g8, t4);
            tc::rows_times_cols<kSplit>(acc, NTS, [&](int ii, int kk) { return -sW[kk * LD + ii]; },
                                        [&](int kk, int nn) { return sDE[kk * kLdC + nn]; }, i0, n0, C, g8, t4);
#pragma unroll
            for (int t = 0; t < NTS; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    sDS[(i0 + g8 + 8 * (u >> 1)) * kLdC + n0 + 8 * t + 2 * t4 + (u & 1)] = acc[t][u];
        }
    }
    if (a.d_init) {
        __syncthreads();
        for (int i = rg; i < DK; i += 8)
            for (int jj = j; jj < kDvt; jj += 32) a.d_init[(bh * DK + i) * dv + col + jj - j] = sDS[i * kLdC + jj];
    }
}

struct GradArgs {
    const void *q, *k, *v;
    const float *log_alpha;
    const void *beta;
    const void *d_out;
    BwdWorkspace ws;
    void *dq, *dk, *dv;
    float *d_log_alpha;
    void *d_beta;
    int64_t B, T, H;
    int dv_, C, NC, gate;
};

size_t grad_smem_bytes(int dk, int dv) {
    const int ldw = (dk > dv ? dk : dv) + 4;
    return sizeof(float) * (size_t)(3 * 64 * (dk + 8) + 2 * 64 * ldw + 2 * 64 * kLdA + 64 + dk + 64 +
                                    kSlice * (dv + 4) + 64 * kLdM);
}

// Every gradient of one chunk's tokens.  Thread (row r = tid / 8, part = tid % 8) owns key
// channels i = part + 8m and value columns j = part + 8m of row r; its dq, dk and dg entries
// accumulate in registers over the phases:
//   0. q, k, beta, g (cumulative, per channel; a scalar gate is broadcast), T, P, dO;
//   1. E = U - W S0;  dO S0^T  -> dq, dg;
//   2. dE = P^T dO + Kd dS_C;  dP = tril(dO E^T) (over P);
//   3. dR = T^T dE (over dE);
//   4. dA = -stril(dR E^T) (over T);  dv = b dR;  db, part 1;  dR S0^T -> dk, dg;
//      E dS_C^T -> dk, dg and the last token's dg;
//   5. the pair products of P and A -> dq, dk, dg, db part 2;
//   6. db, dq, dk out; dg summed from the last token back -> d log alpha.
template <int DK, typename Tin, typename Tg>
__global__ void __launch_bounds__(kGThreads) chunk_grad_kernel(GradArgs a) {
    // fp32 inputs: products at fp32 accuracy (three split-TF32 products); bf16 inputs, whose
    // results are held to the bf16 bound: one TF32 product (~2^-11 relative)
    constexpr bool kSplit = sizeof(Tin) == 4;
    constexpr int LDK = DK + 8;
    constexpr int NI = DK / kParts;   // key channels per thread
    extern __shared__ float4 smem4[];
    const int dv = a.dv_;
    const int ldw = (DK > dv ? DK : dv) + 4;
    float *sQ = reinterpret_cast<float *>(smem4);  // [64][LDK] q (then dg)
    float *sK = sQ + 64 * LDK;                     // [64][LDK] k
    float *sG = sK + 64 * LDK;                     // [64][LDK] g per channel
    float *sE = sG + 64 * LDK;                     // [64][ldw] E
    float *sX = sE + 64 * ldw;                     // [64][ldw] dO -> dE -> dR -> E dS_C^T terms
    float *sT = sX + 64 * ldw;                     // [64][kLdA] T -> dA
    float *sP = sT + 64 * kLdA;                    // [64][kLdA] P -> dP
    float *sB = sP + 64 * kLdA;                    // [64] beta
    float *sDgC = sB + 64;                         // [DK] d g of the last token (gamma terms)
    float *sRed = sDgC + DK;                       // [64] row sums
    float *sS = sRed + 64;                         // [kSlice][dv + 4] rows of S0 or dS_C
    float *sM = sS + kSlice * (dv + 4);            // [64][kLdM] a product against a staged slice

    const Tin *q = (const Tin *)a.q, *k = (const Tin *)a.k, *v = (const Tin *)a.v;
    const Tin *beta = (const Tin *)a.beta;
    const Tg *dout = (const Tg *)a.d_out;
    const int C = a.C, NC = a.NC, tid = threadIdx.x;
    const int64_t n = blockIdx.x;
    const int c = (int)(n % NC);
    const int64_t bh = n / NC;
    const int64_t h = bh % a.H, b = bh / a.H;
    const int64_t t0 = (int64_t)c * C;
    const int Lc = (int)(a.T - t0 < (int64_t)C ? a.T - t0 : (int64_t)C);
    auto tok = [&](int r) -> int64_t { return (b * a.T + t0 + r) * a.H + h; };
    const float *S0 = a.ws.ckpt + n * (int64_t)DK * dv;
    const float *dSC = a.ws.dsc + n * (int64_t)DK * dv;
    const float *Wn = a.ws.fw.W + n * (int64_t)C * DK;
    const float *Un = a.ws.fw.U + n * (int64_t)C * dv;
    const int r = tid / kParts, part = tid % kParts;
    const bool row_ok = r < C;
    const int lds = dv + 4;
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int kWarps = kGThreads / 32;
    auto none = [](int, int) { return false; };
    // sM[r][n] = X_r . S_n over the staged slice (rows r < C of X, row stride ldx); ends
    // with a barrier
    // [C][dv] products (E, dE, dR, (K*G) S0): warp w owns rows 16 (w % 4) .. + 15 and the
    // dv / 4 columns from (w / 4) dv / 4, as nt tiles of 8; the fragment element (u of tile
    // t) is row orow(u), column ocol(t, u)
    const int g8 = lane >> 2, t4 = lane & 3;
    const int orb = 16 * (warp & 3), ocn = (warp >> 2) * (dv / 4), ont = dv / 32;
    const bool own = orb < C;
    auto orow = [&](int u) { return orb + g8 + 8 * (u >> 1); };
    auto ocol = [&](int t, int u) { return ocn + 8 * t + 2 * t4 + (u & 1); };
    float acc[4][4];
    auto acc_zero = [&]() {
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[t][u] = 0.f;
    };
    auto slice_products = [&](const float *X, int ldx) {
        tc::rows_dot_rows<kSplit>(X, ldx, sS, lds, C, kSlice, dv, warp, kWarps, lane, none,
                      [&](int rr, int nn, float v) { sM[rr * kLdM + nn] = v; });
        __syncthreads();
    };
    // rows i0 .. i0 + kSlice - 1 of a [DK][dv] matrix into sS (all threads; barriers around)
    // The stages follow one fixed sequence: the slices of S0, of dS_C, of S0, of dS_C (phases
    // 1, 2, 4, 4b).  Each stage stores the slice that the previous one loaded into registers
    // and starts the loads of the next, which run while this slice is computed on.
    const int nsl = DK / kSlice, nstages = 4 * nsl;
    constexpr int kPf = kSlice * 128 / 4 / kGThreads;   // float4 per thread per slice (dv <= 128)
    float4 pf[kPf];
    int sn = 0;
    auto load_slice = [&](int k) {
        const float *M = ((k / nsl) & 1) ? dSC : S0;
        const int i0 = (k % nsl) * kSlice;
#pragma unroll
        for (int u = 0; u < kPf; ++u) {
            const int idx = tid + u * kGThreads, ii = idx / (dv / 4), j4 = 4 * (idx % (dv / 4));
            if (idx < kSlice * (dv / 4)) pf[u] = load4(M + (i0 + ii) * dv + j4);
        }
    };
    auto stage = [&](const float *M, int i0) {   // (M, i0): the sequence's next slice
        (void)M;
        (void)i0;
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kPf; ++u) {
            const int idx = tid + u * kGThreads, ii = idx / (dv / 4), j4 = 4 * (idx % (dv / 4));
            if (idx < kSlice * (dv / 4)) *reinterpret_cast<float4 *>(sS + ii * lds + j4) = pf[u];
        }
        if (++sn < nstages) load_slice(sn);
        __syncthreads();
    };

    // the chunk's S0 and dS_C (staged later by slices), U (phase 1) and v rows (phase 4)
    // into L2
    if (tid == 0) {
        prefetch_l2(S0, (uint32_t)(DK * dv * 4));
        prefetch_l2(dSC, (uint32_t)(DK * dv * 4));
        prefetch_l2(Un, (uint32_t)(C * dv * 4));
    } else if (tid >= 32 && tid < 32 + Lc) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(v + tok(tid - 32) * dv));
    }
    load_slice(0);
    // ---- 0. inputs (rows past the sequence: zero, log alpha 0)
    //      (four elements per load, several loads in flight per thread)
#pragma unroll 4
    for (int idx = tid; idx < C * (DK / 4); idx += kGThreads) {
        const int rr = idx / (DK / 4), i4 = 4 * (idx % (DK / 4));
        const bool ok = rr < Lc;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(sQ + rr * LDK + i4) = ok ? load4(q + tok(rr) * DK + i4) : z4;
        *reinterpret_cast<float4 *>(sK + rr * LDK + i4) = ok ? load4(k + tok(rr) * DK + i4) : z4;
        float4 la = z4;
        if (ok && a.gate == 2) la = *reinterpret_cast<const float4 *>(a.log_alpha + tok(rr) * DK + i4);
        if (ok && a.gate == 1) {
            const float l = a.log_alpha[tok(rr)];
            la = make_float4(l, l, l, l);
        }
        *reinterpret_cast<float4 *>(sG + rr * LDK + i4) = la;
    }
    for (int rr = tid; rr < C; rr += kGThreads) sB[rr] = rr < Lc ? to_f32(beta[tok(rr)]) : 0.f;
#pragma unroll 2
    for (int idx = tid; idx < C * C / 4; idx += kGThreads) {
        const int rr = (4 * idx) / C, c0 = (4 * idx) % C;
        const float4 t4v = *reinterpret_cast<const float4 *>(a.ws.T + n * (int64_t)C * C + 4 * idx);
        const float4 p4v = *reinterpret_cast<const float4 *>(a.ws.fw.P + n * (int64_t)C * C + 4 * idx);
        float *tr = sT + rr * kLdA + c0, *pr = sP + rr * kLdA + c0;
        tr[0] = t4v.x; tr[1] = t4v.y; tr[2] = t4v.z; tr[3] = t4v.w;
        pr[0] = p4v.x; pr[1] = p4v.y; pr[2] = p4v.z; pr[3] = p4v.w;
    }
#pragma unroll 4
    for (int idx = tid; idx < C * (dv / 4); idx += kGThreads) {
        const int rr = idx / (dv / 4), j4 = 4 * (idx % (dv / 4));
        *reinterpret_cast<float4 *>(sX + rr * ldw + j4) =
            rr < Lc ? load4(dout + tok(rr) * dv + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i = tid; i < DK; i += kGThreads) sDgC[i] = 0.f;
    for (int rr = tid; rr < 64; rr += kGThreads) sRed[rr] = 0.f;   // db terms of phase 4
    __syncthreads();
    for (int i = tid; i < DK; i += kGThreads) {   // cumulative log decay down each channel
        float acc = 0.f;
        for (int rr = 0; rr < C; ++rr) {
            acc += sG[rr * LDK + i];
            sG[rr * LDK + i] = acc;
        }
    }
    __syncthreads();

    float aq[NI], ak[NI], ag[NI];
#pragma unroll
    for (int m = 0; m < NI; ++m) { aq[m] = 0.f; ak[m] = 0.f; ag[m] = 0.f; }

    // ---- 1. E = U - W S0 (tiles, W read from the workspace); dq, dg from (dO S0^T)_ri;
    //         S0 staged by slices of kSlice rows
    acc_zero();
    for (int idx = tid; idx < C * (DK / 4); idx += kGThreads) {   // W over sE until E is formed
        const int rr = idx / (DK / 4), c4 = 4 * (idx % (DK / 4));
        cp_async16(sE + rr * ldw + c4, Wn + rr * DK + c4);
    }
    cp_async_commit_wait_all();
    for (int i0 = 0; i0 < DK; i0 += kSlice) {
        stage(S0, i0);
        slice_products(sX, ldw);   // (dO S0^T) over the slice
        if (own)
            tc::rows_times_cols<kSplit>(acc, ont, [&](int rr, int kk) { return sE[rr * ldw + i0 + kk]; },
                            [&](int kk, int nn) { return sS[kk * lds + nn]; }, orb, ocn, kSlice, g8, t4);
        if (!row_ok) continue;
#pragma unroll
        for (int m = 0; m < NI; ++m) {
            const int i = part + kParts * m;
            if (i < i0 || i >= i0 + kSlice) continue;
            const float acc = sM[r * kLdM + i - i0];
            const float e = __expf(sG[r * LDK + i]);
            aq[m] = fmaf(e, acc, aq[m]);
            ag[m] = fmaf(sQ[r * LDK + i] * e, acc, ag[m]);
        }
    }
    __syncthreads();   // every tile has read W
    if (own)
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (t < ont) sE[orow(u) * ldw + ocol(t, u)] = Un[orow(u) * dv + ocol(t, u)] - acc[t][u];
    __syncthreads();

    // ---- 2. dE = P^T dO + Kd dS_C (tiles; P lower triangular, dS_C by slices), dP =
    //         tril(dO E^T) over P, then dE over dO
    acc_zero();
    if (own)
        tc::rows_times_cols<kSplit>(acc, ont, [&](int rr, int kk) { return sP[kk * kLdA + rr]; },
                        [&](int kk, int nn) { return sX[kk * ldw + nn]; }, orb, ocn, C, g8, t4);
    for (int i0 = 0; i0 < DK; i0 += kSlice) {
        stage(dSC, i0);
        if (own)
            tc::rows_times_cols<kSplit>(acc, ont, [&](int rr, int kk) {   // Kd = k exp(g_C - g)
                                    const int i = i0 + kk;
                                    return sK[rr * LDK + i] * __expf(sG[(C - 1) * LDK + i] - sG[rr * LDK + i]); },
                            [&](int kk, int nn) { return sS[kk * lds + nn]; }, orb, ocn, kSlice, g8, t4);
    }
    __syncthreads();
    tc::rows_dot_rows<kSplit>(sX, ldw, sE, ldw, C, C, dv, warp, kWarps, lane,
                  [](int r0, int n0) { return n0 > r0 + 15; },   // tiles above the diagonal
                  [&](int rr, int nn, float v) { sP[rr * kLdA + nn] = nn <= rr ? v : 0.f; });
    for (int idx = tid; idx < C * C; idx += kGThreads) {          // their zeros
        const int rr = idx / C, nn = idx % C;
        if ((nn & ~7) > (rr | 15)) sP[rr * kLdA + nn] = 0.f;
    }
    __syncthreads();
    auto acc_to_x = [&]() {   // the tiles over sX (rows < C)
        if (own)
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (t < ont) sX[orow(u) * ldw + ocol(t, u)] = acc[t][u];
    };
    acc_to_x();
    __syncthreads();

    // ---- 3. dR = T^T dE (T lower triangular), over dE
    acc_zero();
    if (own)
        tc::rows_times_cols<kSplit>(acc, ont, [&](int rr, int kk) { return sT[kk * kLdA + rr]; },
                        [&](int kk, int nn) { return sX[kk * ldw + nn]; }, orb, ocn, C, g8, t4);
    __syncthreads();
    acc_to_x();
    __syncthreads();

    // ---- 4. dA over T; dv; db part 1 (with (K*G) S0); (dR S0^T) -> dk, dg; S0 by slices
    const float br = row_ok ? sB[r] : 0.f;
    float db = 0.f;
    tc::rows_dot_rows<kSplit>(sX, ldw, sE, ldw, C, C, dv, warp, kWarps, lane,
                  [](int r0, int n0) { return n0 > r0 + 15; },
                  [&](int rr, int nn, float v) { sT[rr * kLdA + nn] = nn < rr ? -v : 0.f; });
    for (int idx = tid; idx < C * C; idx += kGThreads) {
        const int rr = idx / C, nn = idx % C;
        if ((nn & ~7) > (rr | 15)) sT[rr * kLdA + nn] = 0.f;
    }
    if (row_ok) {
        if (r < Lc) {
            Tin *gv = (Tin *)a.dv;
            for (int j = part; j < dv; j += kParts) gv[tok(r) * dv + j] = from_f32<Tin>(br * sX[r * ldw + j]);
        }
    }
    acc_zero();   // ((K*G) S0)_rj
    for (int i0 = 0; i0 < DK; i0 += kSlice) {
        stage(S0, i0);
        slice_products(sX, ldw);   // (dR S0^T) over the slice
        if (own)
            tc::rows_times_cols<kSplit>(acc, ont,
                            [&](int rr, int kk) { return sK[rr * LDK + i0 + kk] * __expf(sG[rr * LDK + i0 + kk]); },
                            [&](int kk, int nn) { return sS[kk * lds + nn]; }, orb, ocn, kSlice, g8, t4);
        if (!row_ok) continue;
#pragma unroll
        for (int m = 0; m < NI; ++m) {
            const int i = part + kParts * m;
            if (i < i0 || i >= i0 + kSlice) continue;
            const float acc = sM[r * kLdM + i - i0];
            const float w = br * __expf(sG[r * LDK + i]) * acc;
            ak[m] -= w;
            ag[m] = fmaf(-w, sK[r * LDK + i], ag[m]);
        }
    }
    if (own) {   // db_r, part 1: sum_j dR_rj (v_rj - ((K*G) S0)_rj), into sRed[r]
        float d2[2] = {0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int rr = orow(u), j = ocol(t, u);
                if (t < ont) {
                    const float u0 = (rr < Lc ? to_f32(v[tok(rr) * dv + j]) : 0.f) - acc[t][u];
                    d2[u >> 1] = fmaf(sX[rr * ldw + j], u0, d2[u >> 1]);
                }
            }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            d2[h2] += __shfl_xor_sync(0xffffffffu, d2[h2], 1);
            d2[h2] += __shfl_xor_sync(0xffffffffu, d2[h2], 2);
        }
        if (t4 == 0) {
            atomicAdd(&sRed[orb + g8], d2[0]);
            atomicAdd(&sRed[orb + g8 + 8], d2[1]);
        }
    }

    // ---- 4b. Y = E dS_C^T -> dk, dg; Y k exp(g_C - g) -> sX (dR is dead after the first
    //          staging barrier) for the last token's dg; dS_C by slices
    for (int i0 = 0; i0 < DK; i0 += kSlice) {
        stage(dSC, i0);
        slice_products(sE, ldw);   // (E dS_C^T) over the slice
        if (!row_ok) continue;
#pragma unroll
        for (int m = 0; m < NI; ++m) {
            const int i = part + kParts * m;
            if (i < i0 || i >= i0 + kSlice) continue;
            const float y = sM[r * kLdM + i - i0];
            const float f = __expf(sG[(C - 1) * LDK + i] - sG[r * LDK + i]);
            const float z = y * sK[r * LDK + i] * f;
            ak[m] = fmaf(y, f, ak[m]);
            ag[m] -= z;
            sX[r * ldw + i] = z;
        }
    }
    __syncthreads();
    {   // d g_C,i = sum_r z_ri + gamma_i sum_j dS_C,ij S0_ij: four threads per key channel
        const int i = tid >> 2, q4 = tid & 3;
        float acc = 0.f;
        if (i < DK) {
            for (int rr = q4; rr < C; rr += 4) acc += sX[rr * ldw + i];
            const float4 *a4 = reinterpret_cast<const float4 *>(dSC + i * dv);
            const float4 *b4 = reinterpret_cast<const float4 *>(S0 + i * dv);
            float sd = 0.f;
            for (int j4 = q4; j4 < dv / 4; j4 += 4) {
                const float4 x = a4[j4], y = b4[j4];
                sd = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, sd))));
            }
            acc = fmaf(sd, __expf(sG[(C - 1) * LDK + i]), acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        if (i < DK && q4 == 0) sDgC[i] = acc;
    }

    // ---- 5. pair products: P_rs = sum_i q_ri k_si D_rs,i (s <= r) and A_rs = b_r sum_i
    //         k_ri k_si D_rs,i (s < r), D = exp(g_r - g_s) <= 1; row r as the row, then as
    //         the column
    float db2 = 0.f;
    if (a.gate != 2) {
        // Scalar gate or none: D_rs is one number per (r, s), so with Pd = dP * D and Ad =
        // dA * D (in place over dP and dA) the pair terms are three [C][DK] products,
        //   dq += Pd K,   dk += diag(b) Ad K + Pd^T Q + (diag(b) Ad)^T K,
        //   dg += Q * (Pd K) + diag(b) K * (Ad K) - K * (Pd^T Q + (diag(b) Ad)^T K),
        //   db_r += sum_i k_ri (Ad K)_ri,
        // as split-TF32 tiles.  The accumulators go through shared memory (dq over E, dk over
        // the z values, dg over g, whose column 0 is kept in sM first).
        __syncthreads();   // the z values in sX have been read
        if (tid < C) sM[tid] = sG[tid * LDK];
        __syncthreads();
        if (row_ok)
#pragma unroll
            for (int m = 0; m < NI; ++m) {
                const int i = part + kParts * m;
                sE[r * ldw + i] = aq[m];
                sX[r * ldw + i] = ak[m];
                sG[r * LDK + i] = ag[m];
            }
        for (int idx = tid; idx < C * C; idx += kGThreads) {
            const int rr = idx / C, ss = idx % C;
            const float d = ss <= rr ? __expf(sM[rr] - sM[ss]) : 0.f;   // exponent <= 0
            sP[rr * kLdA + ss] *= d;
            sT[rr * kLdA + ss] *= d;
        }
        __syncthreads();
        if (own) {
            const int kcn = (warp >> 2) * (DK / 4), knt = DK / 32;
            auto kcol = [&](int t, int u) { return kcn + 8 * t + 2 * t4 + (u & 1); };
            auto Kat = [&](int kk, int nn) { return sK[kk * LDK + nn]; };
            // Pd K
            acc_zero();
            tc::rows_times_cols<kSplit>(acc, knt, [&](int rr, int kk) { return sP[rr * kLdA + kk]; }, Kat, orb, kcn, C,
                                g8, t4);
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (t < knt) {
                        const int rr = orow(u), i = kcol(t, u);
                        sE[rr * ldw + i] += acc[t][u];
                        sG[rr * LDK + i] = fmaf(sQ[rr * LDK + i], acc[t][u], sG[rr * LDK + i]);
                    }
            // Ad K
            acc_zero();
            tc::rows_times_cols<kSplit>(acc, knt, [&](int rr, int kk) { return sT[rr * kLdA + kk]; }, Kat, orb, kcn, C,
                                g8, t4);
            float d2[2] = {0.f, 0.f};
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (t < knt) {
                        const int rr = orow(u), i = kcol(t, u);
                        const float kri = sK[rr * LDK + i], bm = sB[rr] * acc[t][u];
                        sX[rr * ldw + i] += bm;
                        sG[rr * LDK + i] = fmaf(kri, bm, sG[rr * LDK + i]);
                        d2[u >> 1] = fmaf(kri, acc[t][u], d2[u >> 1]);
                    }
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                d2[h2] += __shfl_xor_sync(0xffffffffu, d2[h2], 1);
                d2[h2] += __shfl_xor_sync(0xffffffffu, d2[h2], 2);
            }
            if (t4 == 0) {
                atomicAdd(&sRed[orb + g8], d2[0]);
                atomicAdd(&sRed[orb + g8 + 8], d2[1]);
            }
            // Pd^T Q + (diag(b) Ad)^T K
            acc_zero();
            tc::rows_times_cols<kSplit>(acc, knt, [&](int rr, int kk) { return sP[kk * kLdA + rr]; },
                                [&](int kk, int nn) { return sQ[kk * LDK + nn]; }, orb, kcn, C, g8, t4);
            tc::rows_times_cols<kSplit>(acc, knt, [&](int rr, int kk) { return sB[kk] * sT[kk * kLdA + rr]; }, Kat, orb,
                                kcn, C, g8, t4);
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (t < knt) {
                        const int rr = orow(u), i = kcol(t, u);
                        sX[rr * ldw + i] += acc[t][u];
                        sG[rr * LDK + i] = fmaf(-sK[rr * LDK + i], acc[t][u], sG[rr * LDK + i]);
                    }
        }
        __syncthreads();
        if (row_ok)
#pragma unroll
            for (int m = 0; m < NI; ++m) {
                const int i = part + kParts * m;
                aq[m] = sE[r * ldw + i];
                ak[m] = sX[r * ldw + i];
                ag[m] = sG[r * LDK + i];
            }
    } else if (row_ok) {
        for (int s = 0; s <= r; ++s) {
            const float dp = sP[r * kLdA + s];
            const float da = s < r ? sT[r * kLdA + s] : 0.f;
#pragma unroll
            for (int m = 0; m < NI; ++m) {
                const int i = part + kParts * m;
                const float kd = sK[s * LDK + i] * __expf(sG[r * LDK + i] - sG[s * LDK + i]);
                const float kr = sK[r * LDK + i];
                const float tq = dp * kd, ta = da * br * kd;
                aq[m] += tq;
                ak[m] += ta;
                ag[m] = fmaf(sQ[r * LDK + i], tq, fmaf(kr, ta, ag[m]));
                db2 = fmaf(da * kr, kd, db2);
            }
        }
        for (int s2 = r; s2 < C; ++s2) {
            const float dp = sP[s2 * kLdA + r];
            const float da = s2 > r ? sT[s2 * kLdA + r] * sB[s2] : 0.f;
#pragma unroll
            for (int m = 0; m < NI; ++m) {
                const int i = part + kParts * m;
                const float d = __expf(sG[s2 * LDK + i] - sG[r * LDK + i]);
                const float t = (dp * sQ[s2 * LDK + i] + da * sK[s2 * LDK + i]) * d;
                ak[m] += t;
                ag[m] = fmaf(-sK[r * LDK + i], t, ag[m]);
            }
        }
    }
    db += db2;
    if (row_ok && part == 0) db += sRed[r];   // complete since the staging barriers of 4b
    db += __shfl_xor_sync(0xffffffffu, db, 1);
    db += __shfl_xor_sync(0xffffffffu, db, 2);
    db += __shfl_xor_sync(0xffffffffu, db, 4);

    // ---- 6. outputs; d log alpha_t = sum_{r >= t} dg_r (+ the last token's gamma terms)
    if (row_ok && r < Lc) {
        Tin *gq = (Tin *)a.dq, *gk = (Tin *)a.dk;
        if (part == 0) ((Tin *)a.d_beta)[tok(r)] = from_f32<Tin>(db);
#pragma unroll
        for (int m = 0; m < NI; ++m) {
            gq[tok(r) * DK + part + kParts * m] = from_f32<Tin>(aq[m]);
            gk[tok(r) * DK + part + kParts * m] = from_f32<Tin>(ak[m]);
        }
    }
    if (a.gate == 0) return;
    __syncthreads();   // sQ is dead
    if (row_ok)
#pragma unroll
        for (int m = 0; m < NI; ++m) sQ[r * LDK + part + kParts * m] = ag[m];
    __syncthreads();
    if (a.gate == 2) {
        for (int i = tid; i < DK; i += kGThreads) {
            float run = sDgC[i];
            for (int rr = C - 1; rr >= 0; --rr) {
                run += sQ[rr * LDK + i];
                if (rr < Lc) a.d_log_alpha[tok(rr) * DK + i] = run;
            }
        }
    } else {
        {   // row sums of dg: eight threads per row
            const int rr = tid >> 3, p8 = tid & 7;
            float acc = 0.f;
            if (rr < C)
                for (int i = p8; i < DK; i += 8) acc += sQ[rr * LDK + i];
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            if (rr < C && p8 == 0) sRed[rr] = acc;
        }
        __syncthreads();
        if (warp == 0) {   // d log alpha_t = sum_i dg_C,i + sum_{r >= t} (row sum)_r: one warp
            float tg = 0.f;
            for (int i = lane; i < DK; i += 32) tg += sDgC[i];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) tg += __shfl_xor_sync(0xffffffffu, tg, o);
            const int r0 = 2 * lane;   // rows r0, r0 + 1 (C <= 64)
            const float v0 = r0 < C ? sRed[r0] : 0.f, v1 = r0 + 1 < C ? sRed[r0 + 1] : 0.f;
            float suf = v0 + v1;   // suffix sums over lanes >= this one
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += y;
            }
            if (r0 < Lc) a.d_log_alpha[tok(r0)] = tg + suf;
            if (r0 + 1 < Lc) a.d_log_alpha[tok(r0 + 1)] = tg + suf - v0;
        }
    }
}

template <int DK, typename Tin, typename Tg>
int launch_bwd_t(const DStateArgs &da, const GradArgs &ga, int64_t nstate, int64_t ngrad,
                 cudaStream_t stream) {
    const size_t ds = dstate_smem_bytes(DK), gs = grad_smem_bytes(DK, ga.dv_);
    constexpr bool kSplit = sizeof(Tin) == 4;
    if (cudaFuncSetAttribute(chunk_dstate_kernel<DK, Tg, kSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ds) != cudaSuccess ||
        cudaFuncSetAttribute(chunk_grad_kernel<DK, Tin, Tg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gs) != cudaSuccess)
        return kErrCuda;
    chunk_dstate_kernel<DK, Tg, kSplit><<<(unsigned)nstate, kThreads, ds, stream>>>(da);
    if (ngrad > 0) chunk_grad_kernel<DK, Tin, Tg><<<(unsigned)ngrad, kGThreads, gs, stream>>>(ga);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

size_t bwd_workspace_bytes(const ChunkProblem &p) { return sizeof(float) * bwd_floats(p); }

int launch_chunk_bwd(const ChunkProblem &p, const BwdIo &g, void *workspace, int *status_word,
                     cudaStream_t stream) {
    const BwdWorkspace ws = bwd_carve(workspace, p);
    if (p.NC > 0) {
        // the forward's per-chunk operands and T (CUDA cores), and the chunk-start states,
        // without outputs: from the tensor-core forward where it serves the problem
        ChunkProblem f = p;
        f.out = nullptr;
        f.final_state = nullptr;
        f.fuse = 0;
        f.z = nullptr;
        const bool tc = chunk_tc_supported(f);
        int rc = launch_chunk_simt(f, ws.fw, stream, ws.T, tc ? nullptr : ws.ckpt, tc);
        if (rc != kOk) return rc;
        if (tc) {
            rc = launch_chunk_tc(f, ws.tc, tc_ws_floats(f) * sizeof(float), status_word, stream, ws.ckpt);
            if (rc != kOk) return rc;
        }
    }
    DStateArgs da{g.d_out, g.d_final, g.d_init, ws, p.B, p.T, p.H, p.dv, p.C, p.NC};
    GradArgs ga{p.q, p.k, p.v, p.log_alpha, p.beta, g.d_out, ws, g.dq, g.dk, g.dv, g.d_log_alpha,
                g.d_beta, p.B, p.T, p.H, p.dv, p.C, p.NC, p.gate};
    const int64_t nstate = p.B * p.H * (p.dv / kDvt), ngrad = p.B * p.H * p.NC;
    using bf = __nv_bfloat16;
    const bool ib = p.in_bf16, ob = p.out_bf16;
    if (p.dk == 128) {
        if (ib && ob) return launch_bwd_t<128, bf, bf>(da, ga, nstate, ngrad, stream);
        if (ib) return launch_bwd_t<128, bf, float>(da, ga, nstate, ngrad, stream);
        if (ob) return launch_bwd_t<128, float, bf>(da, ga, nstate, ngrad, stream);
        return launch_bwd_t<128, float, float>(da, ga, nstate, ngrad, stream);
    }
    if (p.dk == 64) {
        if (ib && ob) return launch_bwd_t<64, bf, bf>(da, ga, nstate, ngrad, stream);
        if (ib) return launch_bwd_t<64, bf, float>(da, ga, nstate, ngrad, stream);
        if (ob) return launch_bwd_t<64, float, bf>(da, ga, nstate, ngrad, stream);
        return launch_bwd_t<64, float, float>(da, ga, nstate, ngrad, stream);
    }
    return kErrUnsupported;
}

}  // namespace dr
