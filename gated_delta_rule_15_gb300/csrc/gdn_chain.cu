// gdn_chain.cu -- chunkwise forward of the gated delta rule as two tensor-core kernels: a
// chunk-parallel prep kernel and a per-chain kernel whose per-chunk products are a few wide
// tcgen05 MMAs.  bf16 inputs, d_k = d_v = 128, chunk C = 64, scalar gate or no gate.
//
// The chunk form is the one of chunk_simt.cu and chunk_tc.cu (derived from the recurrence of
// the page "NLP: linear attention summary", KDA section, in the order of the
// `gated_delta_rule` loop of the page "linear-attention gated-deltanet guide", section 4;
// chunks are processed in parallel inside and carried sequentially between them, page
// "Transformer notes (5): linear attention optimisations", paragraph on chunked
// computation).  Per chunk, with g the cumulative log decay, G = exp(g), gamma = G_63 and
// delta_r = exp(g_63 - g_r):
//
//   A   = stril(beta_r exp(g_r - g_s) K K^T),  T = (I + A)^-1          (prep kernel)
//   U^T = V^T (T diag beta)^T,   W^T = K^T (T diag(beta G))^T
//   [(W S)^T | (Q S)^T] = S^T [W; Q]^T                                  (one N = 128 product)
//   E^T = U^T - (W S)^T
//   [O^T | S^T] <- [G (Q S)^T | gamma S^T] + E^T [P; Kt^T]^T             (one N = 192 product)
//   with P = tril(exp(g_r - g_s) Q K^T) and Kt = diag(delta) K.
//
// The only step that depends on the previous chunk is the state: S^T -> [W S, Q S] -> E ->
// S^T.  The triangular solve T = (I + A)^-1 depends on the chunk's own k, beta and gates
// only, so gdn_prep_kernel forms it for every chunk at once (one CTA per chunk) and writes
// the two bf16 operands T diag(beta) | T diag(beta G) (16 KB per chunk, already in the
// swizzled layout of the tensor core's B operand) to the workspace.  gdn_chain_kernel then
// walks each chain's chunks with nine or ten warps, each group with one duty:
//
//   warp 0       TMA: each chunk's q, k tiles (two stages) and its v tile and T operands
//   warp 1       issues every tcgen05.mma and commits it to an mbarrier
//   warp 2       the gates: beta and log alpha by cp.async, cumulative decays per chunk
//   warps 3..6   the state: S^T -> bf16 (an A operand in tensor memory) and S^T <- gamma S^T,
//                P from X = [Q; K] K^T, E^T = U^T - (W S)^T (fp32, in tensor memory: the
//                tf32 A operand of the state update) and G (Q S)^T
//   warps 7..10  W^T (tensor memory) -> W (bf16, the B operand of the next product), Kt^T
//                (tf32) from the k tile, and the chunk's output (TMA store)
//
// Precision: S and W enter (W S, Q S) as bf16 (Q exactly), the state update and the output's
// intra-chunk term take E, P and Kt as tf32 (10 explicit mantissa bits); T's operands are
// bf16, as in chunk_tc.cu.  Every wait is bounded by a cycle budget: on expiry the kernel
// records DR_ERR_TIMEOUT in the status word, stops, drains its own copies and MMAs with the
// same bound, frees tensor memory and returns.
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "chunk_layout.h"
#include "common.cuh"
#include "tc_common.cuh"
#include "umma.cuh"

namespace dr {

// chunk_tc.cu: the tensor map of a [B, T, H, 128] tensor (64-token boxes, 128-byte swizzle)
// and the segment split of few long chains.
bool tc_make_map(CUtensorMap *m, const void *base, int64_t B, int64_t T, int64_t H, bool fp32);
void tc_segment_split(const ChunkProblem &p, int *nseg, int *seg_len);

namespace {

using namespace umma;
using namespace tc;

// Largest in-chunk log-decay span for which exp(g_r - g_s) is formed as a product of two
// exponentials around the chunk's middle token (both factors stay within fp32 range).
constexpr float kSpan = 80.f;

// ============================================================ prep kernel
// Persistent CTAs of four warps walk the (chain, chunk) pairs; per chunk, all independent:
// the k tile arrives by TMA (128-byte swizzle; the next chunk's tile is prefetched into L2
// meanwhile), X = K K^T on the lower 16 x 16 blocks (mma.sync, bf16 in, fp32 out, fragments
// by ldmatrix; warp w takes row block w), A_rs = beta_r exp(g_r - g_s) X_rs for s < r
// (off-diagonal blocks TF32-rounded), then the blocked solve of tc_common.cuh, which writes
// T diag(beta) | T diag(beta G) in bf16; the 16 KB image leaves by one bulk store.  Tokens
// past T are zero rows of K (the TMA fill) with beta = 0, T being the identity there, as the
// chain kernel's loads make them.
// Fused neighbours (DR_FUSE_* of include/dr.h): beta = sigmoid(logit) rounded to beta's bf16;
// with the L2 norm the q tile arrives too (over A's buffer, free until the A build), each
// thread takes 1 / |x| of one row of [Q; K]
// (written to the workspace's norm vectors for the chain kernel), A takes the normalised
// rows' products n_r n_s (k_r . k_s), and the second operand becomes T diag(beta G n), so
// that W = T diag(beta G) diag(n) K is formed from the raw k tile.
constexpr int kPrepThreads = 128;
constexpr uint32_t PR_K = 0;                       // k tile (two 64-channel halves, swizzled);
                                                   // then the fp32 T (swizzled)
constexpr uint32_t PR_A = 16384;                   // (fused L2 norm) the q tile, until the norms;
                                                   // then fp32 A (a_index)
constexpr uint32_t PR_TB = PR_A + 16384;           // the operand image
constexpr uint32_t PR_M = PR_TB + 16384;           // solve scratch
constexpr uint32_t PR_V = PR_M + 4096;             // g, G, beta, exp(g - g_31), exp(g_31 - g),
                                                   // 1/|q|, 1/|k|, G/|k|
constexpr uint32_t PR_TOTAL = PR_V + 8 * 256;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}


template <int GATE>
__global__ void __launch_bounds__(kPrepThreads, 4)
gdn_prep_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tq,
                const __nv_bfloat16 *__restrict__ beta, const float *__restrict__ log_alpha,
                unsigned char *__restrict__ tops, float *__restrict__ norms, int T, int H, int NC,
                unsigned nchunks, uint32_t fuse, int *status) {
    extern __shared__ unsigned char prep_sm[];
    unsigned char *sm = align1024(prep_sm);
    __shared__ uint64_t bar_k;
    __shared__ int fac_s, abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *sA = reinterpret_cast<float *>(sm + PR_A);
    float *sV = reinterpret_cast<float *>(sm + PR_V);
    float *sG = sV, *sGam = sV + 64, *sBeta = sV + 128, *sE = sV + 192, *sF = sV + 256;
    float *sNq = sV + 320, *sNk = sV + 384, *sGn = sV + 448;
    const bool l2 = (fuse & kFuseL2) != 0, sig = (fuse & kFuseSigmoid) != 0;
    if (tid == 0) {
        mbar_init(&bar_k, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto coords = [&](unsigned n, int &h, int &b, int &t0) {
        const int c = (int)(n % (unsigned)NC), bh = (int)(n / (unsigned)NC);
        h = bh % H; b = bh / H; t0 = c * 64;
    };
    uint32_t phase = 0;
    for (unsigned n = blockIdx.x; n < nchunks; n += gridDim.x, phase ^= 1) {
        int h, b, t0;
        coords(n, h, b, t0);
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_k, l2 ? 32768 : 16384);
            for (int kb = 0; kb < 2; ++kb) tma_load_4d(sm + PR_K + kb * 8192, &tk, &bar_k, 64 * kb, h, t0, b);
            if (l2)
                for (int kb = 0; kb < 2; ++kb) tma_load_4d(sm + PR_A + kb * 8192, &tq, &bar_k, 64 * kb, h, t0, b);
            const unsigned nn = n + gridDim.x;
            if (nn < nchunks) {
                int h2, b2, t2;
                coords(nn, h2, b2, t2);
                for (int kb = 0; kb < 2; ++kb) {
                    tma_prefetch_4d(&tk, 64 * kb, h2, t2, b2);
                    if (l2) tma_prefetch_4d(&tq, 64 * kb, h2, t2, b2);
                }
            }
        }
        if (warp == 1) {   // the next chunk's gates into L2 (two tokens per lane)
            const unsigned nn = n + gridDim.x;
            if (nn < nchunks) {
                int h2, b2, t2;
                coords(nn, h2, b2, t2);
                const int t = t2 + 2 * lane;
                if (t < T) {
                    const size_t tok = ((size_t)b2 * T + t) * H + h2;
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(beta + tok));
                    if (GATE == 1) asm volatile("prefetch.global.L2 [%0];" ::"l"(log_alpha + tok));
                }
            }
        }
        if (warp == 0) {   // the chunk's gates, two tokens per lane
            float l[2], bt[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = t0 + 2 * lane + e;
                const size_t tok = ((size_t)b * T + t) * H + h;
                bt[e] = t < T ? __bfloat162float(beta[tok]) : 0.f;
                if (sig && t < T) bt[e] = round_bf16(sigmoid_f(bt[e]));
                l[e] = (GATE == 1 && t < T) ? log_alpha[tok] : 0.f;
            }
            float p = l[0] + l[1];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, p, o);
                if (lane >= o) p += y;
            }
            const float g1 = p, g0 = p - l[1];
            const float glast = __shfl_sync(0xffffffffu, g1, 31);
            const float gmid = __shfl_sync(0xffffffffu, g1, 15);
            const float gfirst = __shfl_sync(0xffffffffu, g0, 0);
            const int r = 2 * lane;
            sG[r] = g0; sG[r + 1] = g1;
            sBeta[r] = bt[0]; sBeta[r + 1] = bt[1];
            sGam[r] = __expf(g0); sGam[r + 1] = __expf(g1);
            const bool fac = gfirst - glast < kSpan;
            if (fac) {
                sE[r] = __expf(g0 - gmid); sE[r + 1] = __expf(g1 - gmid);
                sF[r] = __expf(gmid - g0); sF[r + 1] = __expf(gmid - g1);
            }
            if (lane == 0) fac_s = fac;
        }
        if (!wait_cycles(&bar_k, phase)) {
            abort_s = 1;
            atomicExch(status, kErrTimeout);
        }
        __syncthreads();
        if (abort_s) break;
        if (l2) {   // 1 / |x| of row tid of [Q; K] (zero rows past T give 1 / sqrt(eps), unused)
            const unsigned char *src = sm + (tid < 64 ? PR_A : PR_K) + (tid & 63) * 128;
            float ss = 0.f;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(src + kb * 8192 + 16 * (j ^ (tid & 7)));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
                        ss = fmaf(f.x, f.x, ss);
                        ss = fmaf(f.y, f.y, ss);
                    }
                }
            const float inv = rsqrtf(ss + kL2NormEps);
            if (tid < 64) {
                sNq[tid] = inv;
            } else {
                sNk[tid - 64] = inv;
                sGn[tid - 64] = sGam[tid - 64] * inv;
            }
            norms[(size_t)n * 128 + tid] = inv;
            __syncthreads();
        }

        // X on the lower blocks and A from it: warp w owns rows 16 w .. 16 w + 15
        {
            const int g = lane >> 2, t4 = lane & 3, r0 = 16 * warp;
            const bool fac = fac_s != 0;
            const uint32_t kbase = smem_u32(sm + PR_K);
            // ldmatrix row address: tile row `row`, 8-element chunk `kc` (of 16 per row)
            auto addr = [&](int row, int kc) {
                return kbase + (uint32_t)((kc >> 3) * 8192 + row * 128 + (((kc & 7) ^ (row & 7)) << 4));
            };
            const int mi = lane >> 3, mr = lane & 7;
            uint32_t af[8][4];
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) ldsm_x4(addr(r0 + mr + 8 * (mi & 1), 2 * ks + (mi >> 1)), af[ks]);
            for (int cb = 0; cb <= warp; ++cb) {
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t bf[4];
                    ldsm_x4(addr(16 * cb + mr + 8 * (mi >> 1), 2 * ks + (mi & 1)), bf);
                    mma_bf16_16x8x16(acc[0], af[ks], bf[0], bf[1]);
                    mma_bf16_16x8x16(acc[1], af[ks], bf[2], bf[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int r = r0 + g + 8 * hf, s0 = 16 * cb + 8 * nt + 2 * t4;
                        float v[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int s = s0 + e;
                            float dec = fac ? sE[r] * sF[s] : __expf(fminf(sG[r] - sG[s], 0.f));
                            if (l2) dec *= sNk[r] * sNk[s];
                            v[e] = s < r ? sBeta[r] * dec * acc[nt][2 * hf + e] : 0.f;
                            if (cb != warp) v[e] = round_tf32(v[e]);
                        }
                        *reinterpret_cast<float2 *>(sA + a_index(r, s0)) = make_float2(v[0], v[1]);
                    }
            }
        }
        // the previous chunk's image has been read out by its store before the solve rewrites it
        if (tid == 0) bulk_wait_read_all();
        __syncthreads();   // the k tile is dead: T goes over it

        const SolveOut<true, true, true> out{reinterpret_cast<float *>(sm + PR_K), sm + PR_TB, sBeta,
                                             l2 ? sGn : sGam, nullptr};
        solve_diag64(sA, out, tid);          // diagonal blocks 0, 1 (and operand zero blocks)
        solve_diag64(sA, out, tid + 128);    // diagonal blocks 2, 3
        __syncthreads();
        solve_merge64(sA, out, reinterpret_cast<float *>(sm + PR_M), tid, 1);
        __syncthreads();   // (the merge ends with the operands' proxy fence)
        if (tid == 0) {
            bulk_store(tops + (size_t)n * 16384, sm + PR_TB, 16384);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait_all();
}

// ============================================================ chain kernel
constexpr int kChainThreads = 352;             // 11 warps
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpGate = 2, kWarpO0 = 7;   // state warps: 3..6
// shared memory (offsets from the 1024-byte-aligned base)
// One stage: two K-blocks (64 of the 128 key channels each) of [W | Q | K], every part 64
// rows (tokens) x 128 bytes, K-major with the 128-byte swizzle, so that [W; Q] is one
// 128-row B operand ((W S)^T and (Q S)^T in one product) and [Q; K] one 128-row A operand.
constexpr uint32_t C_STAGE = 49152;
constexpr uint32_t C_KB = 24576;
constexpr uint32_t C_OFF_W = 0, C_OFF_Q = 8192, C_OFF_K = 16384;
constexpr uint32_t C_VU = 2 * C_STAGE;         // v tile (two 64-channel halves) and T diag(beta)
constexpr uint32_t C_TB = C_VU + 16384;        //   T diag(beta) (bf16, 8 KB)
constexpr uint32_t C_WT = C_VU + 24576;        // T diag(beta G) of two chunks (8 KB each)
constexpr uint32_t C_BU = C_WT + 16384;        // tf32 [P; Kt^T]: two K-blocks of 32 tokens
constexpr uint32_t C_BU_KB = 24576;            // 192 rows x 128 bytes
constexpr uint32_t C_OUT = C_BU + 2 * C_BU_KB; // output staging (bf16: 2 boxes, fp32: 4 boxes)
constexpr uint32_t C_Z = C_OUT + 16384;        // (bf16 outputs, fused output gate) the z tile
constexpr uint32_t C_SMALL = C_OUT + 32768;    // gate vectors [2][8][64], raw gates [2][128],
                                               // row norms [2][128]
constexpr uint32_t C_GATE = C_SMALL + 4096, C_NORM = C_SMALL + 5120;
constexpr uint32_t C_TOTAL = C_SMALL + 6144;
static_assert(C_TOTAL + 1024 <= 227 * 1024, "layout");
// tensor memory columns
constexpr uint32_t TM_WE = 0;     // (W S)^T, then E^T (fp32)
constexpr uint32_t TM_QO = 64;    // (Q S)^T, then G (Q S)^T, then O^T
constexpr uint32_t TM_S = 128;    // S^T (fp32)
constexpr uint32_t TM_SB = 256;   // S^T as bf16 pairs (the A operand of [W S | Q S])
constexpr uint32_t TM_X = 320;    // [Q; K] K^T
constexpr uint32_t TM_W = 384;    // W^T
constexpr uint32_t TM_U = 448;    // U^T
// gate vector slots of one set: g, G, delta/|k|, G/|q|, exp(g - g_31)/|q|, exp(g_31 - g)/|k|,
// 1/|q|, 1/|k| (the norms are 1 without the fused L2 norm)
enum { GV_G = 0, GV_GAM = 1, GV_DEL = 2, GV_GQ = 3, GV_E = 4, GV_F = 5, GV_NQ = 6, GV_NK = 7 };
constexpr int kGvSet = 8 * 64;

constexpr uint32_t ID_X = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_UW = idesc_bf16(128, 64, true, false);
constexpr uint32_t ID_D = idesc_bf16(128, 128, false, false);  // B = [W; Q] rows (K-major)
constexpr uint32_t ID_DW = idesc_bf16(128, 64, false, false);  // B = W rows alone (no outputs)
constexpr uint32_t ID_UPD = idesc_tf32(128, 192);
constexpr uint32_t ID_UPD_S = idesc_tf32(128, 128);

struct ChainArgs {
    const float *log_alpha;
    const float *init_state;
    float *final_state;
    const unsigned char *tops;   // [B*H][NC][16384]: T diag(beta) | T diag(beta G) per chunk
    int *status;
    int B, T, H, NC;
    // Sequence segments (few long chains), as in chunk_tc.cu: role 0 runs whole sequences;
    // role 1 runs each segment twice without outputs -- from S_0 = 0 (end state to ws_s0)
    // and as the transition from S_0 = I with no value term (to ws_phi); role 2 reruns each
    // segment from its true start state (ws_start) writing outputs.
    int role, nseg, seg_len;
    float *ws_phi, *ws_s0, *ws_start;
    // fused neighbours (DR_FUSE_*): the prep kernel has applied beta = sigmoid(logit) and the
    // L2 norm's effect on A and W; with the L2 norm the chain scales P, Kt and Q S by the row
    // norms the prep kernel wrote to `norms` ([B*H][NC][1/|q| x 64, 1/|k| x 64]); with the
    // output gate (bf16 outputs) each output is multiplied by silu(z), z's tile by TMA
    uint32_t fuse;
    const float *norms;
};


// Per chunk it (period: from the state update of it - 1 to that of it), the MMA warp issues
//   [W S | Q S](it)  W(it + 1)  update(it)  X(it + 1)  U(it + 1)
// so that only the state's own steps sit between two updates: S^T -> bf16 (warps 3..6),
// [W S | Q S], E (warps 3..6), update.  Everything else is formed a chunk ahead or behind:
// W(it + 1) and its conversion during chunk it (its T operand has a double buffer), P and
// Kt^T of chunk it by warps 7..10 while S^T converts, the output of it - 1 by them first.
template <typename Tout, int GATE>
__global__ void __launch_bounds__(kChainThreads, 1)
gdn_chain_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                 const __grid_constant__ CUtensorMap tz, const ChainArgs a) {
    extern __shared__ unsigned char dsm_raw[];
    unsigned char *sm = align1024(dsm_raw);
    // Completed by TMA transactions or tcgen05.commit (count 1) ...
    __shared__ uint64_t qkw_full[2], wt_full[2], wt_free[2], vu_full, x_done, w_done, uu_done, d_done, u_done;
    // ... or by every thread of a group (stage_free: the commit of [W S | Q S] and warps
    // 7..10 after Kt^T; gset_free: warps 3..10 after their last use of a gate set).
    __shared__ uint64_t sb_ready, p_ready, e_ready, w_ready, kt_ready, o_read;
    __shared__ uint64_t stage_free[2], g_ready[2], gset_free[2], z_full;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s, fac_s[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = 32 * (warp & 3) + lane;   // the TMEM lane this thread reads and writes
    // this CTA's chain, chunk range, initial/final state and duties
    int bh = blockIdx.x, c_begin = 0, c_end = a.NC;
    const float *init_ptr = a.init_state ? a.init_state + (size_t)blockIdx.x * 16384 : nullptr;
    float *fin_ptr = a.final_state ? a.final_state + (size_t)blockIdx.x * 16384 : nullptr;
    bool init_identity = false, zero_u = false, outputs = true;
    if (a.role != 0) {
        const int idx = a.role == 1 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
        const int seg = idx % a.nseg;
        bh = idx / a.nseg;
        c_begin = seg * a.seg_len;
        c_end = min(a.NC, c_begin + a.seg_len);
        const size_t slot = ((size_t)bh * a.nseg + seg) * 16384;
        if (a.role == 1) {
            outputs = false;
            init_ptr = nullptr;
            if (blockIdx.x & 1) {   // transition: S_0 = I, no value term
                init_identity = true;
                zero_u = true;
                fin_ptr = a.ws_phi + slot;
            } else {
                fin_ptr = a.ws_s0 + slot;
            }
        } else {
            init_ptr = a.ws_start + slot;
            fin_ptr = (seg == a.nseg - 1 && a.final_state) ? a.final_state + (size_t)bh * 16384 : nullptr;
        }
    }
    const int h = bh % a.H, b = bh / a.H;
    const int n_it = c_end - c_begin;
    auto tops = [&](int it) { return a.tops + ((size_t)bh * a.NC + c_begin + it) * 16384; };

    float *sVec = reinterpret_cast<float *>(sm + C_SMALL);   // [2][8][64]
    const uint32_t sm_s = smem_u32(sm);                      // the same bytes by shared address
    auto vec_s = [&](int it, int k) { return sm_s + C_SMALL + 4u * ((it & 1) * kGvSet + 64 * k); };
    auto vec = [&](int it, int k) { return sVec + (it & 1) * kGvSet + 64 * k; };
    uint32_t *sGate = reinterpret_cast<uint32_t *>(sm + C_GATE);   // [2][(unused) | log alpha][64]
    float *sNorm = reinterpret_cast<float *>(sm + C_NORM);         // [2][1/|q| | 1/|k|][64]
    const bool l2 = (a.fuse & kFuseL2) != 0;
    const bool zgate = (a.fuse & kFuseGate) != 0 && outputs;

    if (tid == 0) {
        uint64_t *ones[] = {&qkw_full[0], &qkw_full[1], &wt_full[0], &wt_full[1], &wt_free[0], &wt_free[1],
                            &vu_full,     &x_done,      &w_done,     &uu_done,    &d_done,     &u_done};
        for (uint64_t *bb : ones) mbar_init(bb, 1);
        mbar_init(&z_full, 1);
        uint64_t *groups[] = {&sb_ready, &e_ready, &w_ready, &kt_ready, &o_read};
        for (uint64_t *bb : groups) mbar_init(bb, 128);
        mbar_init(&p_ready, 256);   // warps 3..10 (P is built by warps 4, 5, 8, 9)
        for (int s = 0; s < 2; ++s) {
            mbar_init(&stage_free[s], 129);
            mbar_init(&g_ready[s], 32);
            mbar_init(&gset_free[s], 256);
        }
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
    const uint32_t tm = tmb + ((uint32_t)(32 * (warp & 3)) << 16);   // + this warp's lanes
    const uint64_t dK0 = smem_desc_sw128(smem_u32(sm), 16, 1024);
    const uint64_t dMv = smem_desc_sw128(smem_u32(sm), 8192, 1024);    // MN-major, v halves
    const uint64_t dMk = smem_desc_sw128(smem_u32(sm), C_KB, 1024);    // MN-major, k halves
    auto stage = [&](int it) { return sm + (it & 1) * C_STAGE; };
    volatile int *abort_v = &abort_s;
    auto fail = [&]() {
        *abort_v = 1;
        atomicExch(a.status, kErrTimeout);
    };
    // bounded wait; false (and nothing further to do) once the CTA has failed
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) {   // already complete: the common case, no further reads
            tc_fence_after();
            return true;
        }
        if (*abort_v) return false;
        if (!wait_cycles(bar, parity)) {
            fail();
            return false;
        }
        tc_fence_after();
        return true;
    };

    // P(it), columns 32 hh .. 32 hh + 31 (K-block hh of [P; Kt^T]), from the Q K^T rows of X
    // (TMEM lanes 0..63: this thread's row r), tf32: P_rs = exp(g_r - g_s) (q_r . k_s), s <= r
    auto build_p_half = [&](int it, int hh) {
        const int r = row;
        const uint32_t sG = vec_s(it, GV_G), sF = vec_s(it, GV_F);
        const bool fac = fac_s[it & 1] != 0;
        const float er = lds32f(vec_s(it, GV_E) + 4 * r), gr = lds32f(sG + 4 * r);
        float x[32];
        tmem_ld32(tm + TM_X + 32 * hh, x);
        tmem_wait_ld();
        if (fac) {   // exp(g_r - g_s) = exp(g_r - g_31) exp(g_31 - g_s)
            float4 f4[8];   // all factor loads first
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) f4[c4] = lds128f(sF + 4 * (32 * hh + 4 * c4));
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const int s0 = 32 * hh + 4 * c4;
                const float fs[4] = {f4[c4].x, f4[c4].y, f4[c4].z, f4[c4].w};
                float pv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) pv[e] = s0 + e <= r ? round_tf32(er * fs[e] * x[4 * c4 + e]) : 0.f;
                sts128f(sm_s + C_BU + hh * C_BU_KB + sw128_off32(r, 4 * c4), pv[0], pv[1], pv[2], pv[3]);
            }
        } else {   // with the row norms 1/|q_r| and 1/|k_s|
            const uint32_t sNk = vec_s(it, GV_NK);
            const float nqr = lds32f(vec_s(it, GV_NQ) + 4 * r);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const int s0 = 32 * hh + 4 * c4;
                float pv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    pv[e] = s0 + e <= r ? round_tf32(__expf(fminf(gr - lds32f(sG + 4 * (s0 + e)), 0.f)) * x[4 * c4 + e] *
                                                     nqr * lds32f(sNk + 4 * (s0 + e)))
                                        : 0.f;
                sts128f(sm_s + C_BU + hh * C_BU_KB + sw128_off32(r, 4 * c4), pv[0], pv[1], pv[2], pv[3]);
            }
        }
    };

    if (warp == kWarpTma) {
        // ---------------- TMA.  Chunk it's q, k into stage it % 2 and its T diag(beta G) into
        // its slot once chunk it - 2 has left them; its v and T diag(beta) once U(it - 1) has
        // read the previous ones.
        if (lane == 0) {
            int q_last[2] = {-1, -1}, w_last[2] = {-1, -1}, v_last = -1;
            // chunk `it`'s tiles into L2 ahead of their loads (kPrefetch chunks ahead: the
            // loads themselves run about one chunk ahead, less than the memory latency of a
            // GPU full of chains)
            constexpr int kPrefetch = 2;
            auto prefetch = [&](int it) {
                if (it >= n_it) return;
                const int t0 = (c_begin + it) * 64;
                for (int kb = 0; kb < 2; ++kb) {
                    tma_prefetch_4d(&tq, 64 * kb, h, t0, b);
                    tma_prefetch_4d(&tk, 64 * kb, h, t0, b);
                    if (!zero_u) tma_prefetch_4d(&tv, 64 * kb, h, t0, b);
                    if (zgate) tma_prefetch_4d(&tz, 64 * kb, h, t0, b);
                }
                bulk_prefetch_l2(tops(it), 16384);
            };
            for (int it = 1; it < kPrefetch; ++it) prefetch(it);
            for (int it = 0; it < n_it; ++it) {
                const int s = it & 1, t0 = (c_begin + it) * 64;
                prefetch(it + kPrefetch);
                if (it >= 2 && !wait_bar(&stage_free[s], ((it - 2) >> 1) & 1)) break;
                unsigned char *st = stage(it);
                mbar_arrive_expect_tx(&qkw_full[s], 32768);
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_4d(st + kb * C_KB + C_OFF_Q, &tq, &qkw_full[s], 64 * kb, h, t0, b);
                    tma_load_4d(st + kb * C_KB + C_OFF_K, &tk, &qkw_full[s], 64 * kb, h, t0, b);
                }
                q_last[s] = it;
                if (it >= 2 && !wait_bar(&wt_free[s], ((it - 2) >> 1) & 1)) break;
                mbar_arrive_expect_tx(&wt_full[s], 8192);
                bulk_load(sm + C_WT + s * 8192, tops(it) + 8192, 8192, &wt_full[s]);
                w_last[s] = it;
                if (it >= 1 && !wait_bar(&uu_done, (it - 1) & 1)) break;
                if (!zero_u) {
                    mbar_arrive_expect_tx(&vu_full, 24576);
                    for (int kb = 0; kb < 2; ++kb) tma_load_4d(sm + C_VU + kb * 8192, &tv, &vu_full, 64 * kb, h, t0, b);
                    bulk_load(sm + C_TB, tops(it), 8192, &vu_full);
                    v_last = it;
                }
            }
            if (*abort_v) {   // loads this thread issued may still be in flight (bounded waits)
                for (int s = 0; s < 2; ++s) {
                    if (q_last[s] >= 0) wait_cycles(&qkw_full[s], (q_last[s] >> 1) & 1);
                    if (w_last[s] >= 0) wait_cycles(&wt_full[s], (w_last[s] >> 1) & 1);
                }
                if (v_last >= 0) wait_cycles(&vu_full, v_last & 1);
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------- MMA issue
        if (lane == 0 && n_it > 0) {
            // waits without the tcgen05 fence (about 250 cycles each in this thread, whose
            // own MMAs are in flight); one fence before each group of MMAs orders it after
            // the waits before it
            auto wait_m = [&](uint64_t *bar, uint32_t parity) -> bool {
                if (mbar_try_wait(bar, parity)) return true;
                if (*abort_v) return false;
                if (!wait_cycles(bar, parity)) {
                    fail();
                    return false;
                }
                return true;
            };
            uint64_t *last = nullptr;
            uint32_t last_par = 0;
            auto issue_x = [&](int it) {   // X = [Q; K] K^T (rows 0..63: Q K^T)
                tc_fence_after();
                unsigned char *st = stage(it);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t o = (uint32_t)((st - sm) + (ks >> 2) * C_KB + (ks & 3) * 32);
                    mma_bf16(tmb + TM_X, desc_add(dK0, o + C_OFF_Q), desc_add(dK0, o + C_OFF_K), ID_X, ks > 0);
                }
                mma_commit(&x_done);
                last = &x_done; last_par = it & 1;
            };
            auto issue_w = [&](int it) {   // W^T = K^T (T diag(beta G))^T
                tc_fence_after();
                const uint32_t sk = (uint32_t)(stage(it) - sm) + C_OFF_K, wt = C_WT + (it & 1) * 8192;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmb + TM_W, desc_add(dMk, sk + ks * 2048), desc_add(dK0, wt + ks * 32), ID_UW, ks > 0);
                mma_commit(&w_done);
                mma_commit(&wt_free[it & 1]);
                last = &w_done; last_par = it & 1;
            };
            auto issue_u = [&](int it) {   // U^T = V^T (T diag beta)^T
                tc_fence_after();
                if (!zero_u)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmb + TM_U, desc_add(dMv, C_VU + ks * 2048), desc_add(dK0, C_TB + ks * 32), ID_UW,
                                 ks > 0);
                mma_commit(&uu_done);
                last = &uu_done; last_par = it & 1;
            };
            bool ok = true;
            if (outputs) {
                ok = wait_m(&qkw_full[0], 0);
                if (ok) issue_x(0);
            }
            ok = ok && wait_m(&qkw_full[0], 0) && wait_m(&wt_full[0], 0);
            if (ok) issue_w(0);
            ok = ok && (zero_u || wait_m(&vu_full, 0));
            if (ok) issue_u(0);
            for (int it = 0; ok && it < n_it; ++it) {
                const uint32_t par = it & 1;
                const int s = it & 1;
                const bool next = it + 1 < n_it;
                // [(W S)^T | (Q S)^T] in one N = 128 product: A = S^T (bf16 pairs in tensor
                // memory), B = [W; Q] (W written by warps 7..10 above Q in the stage); without
                // outputs (W S)^T alone
                if (!wait_m(&sb_ready, par) || !wait_m(&w_ready, par)) break;
                if (outputs && it >= 1 && !wait_m(&o_read, par ^ 1)) break;
                tc_fence_after();
                const uint32_t sw = (uint32_t)(stage(it) - sm);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ts(tmb + TM_WE, tmb + TM_SB + 8 * ks,
                                desc_add(dK0, sw + C_OFF_W + (ks >> 2) * C_KB + (ks & 3) * 32), outputs ? ID_D : ID_DW,
                                ks > 0);
                mma_commit(&d_done);
                mma_commit(&stage_free[s]);
                last = &d_done; last_par = par;
                // The tensor pipe runs one CTA's MMAs in issue order, and issuing blocks this
                // thread while earlier MMAs drain, so the order below keeps the state's own
                // products (D, the update) from queueing behind work for the next chunk that
                // can wait: W(it + 1) (its conversion by warps 7..10 feeds D(it + 1)) runs
                // while E(it) forms; X(it + 1) and U(it + 1) follow the update and run while
                // the next S^T operand forms.
                if (next) {
                    if (!wait_m(&qkw_full[(it + 1) & 1], ((it + 1) >> 1) & 1) ||
                        !wait_m(&wt_full[(it + 1) & 1], ((it + 1) >> 1) & 1))
                        break;
                    issue_w(it + 1);
                }
                // [O^T | S^T] += E^T [P; Kt^T]^T  (tf32; E^T from tensor memory)
                if (!wait_m(&e_ready, par) || !wait_m(&kt_ready, par)) break;
                if (outputs && !wait_m(&p_ready, par)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_tf32_ts(tmb + (outputs ? TM_QO : TM_S), tmb + TM_WE + 8 * ks,
                                desc_add(dK0, C_BU + (outputs ? 0u : 8192u) + (ks >> 2) * C_BU_KB + (ks & 3) * 32),
                                outputs ? ID_UPD : ID_UPD_S, true);
                mma_commit(&u_done);
                last = &u_done; last_par = par;
                // X(it + 1): P(it) has been read out of TM_X (p_ready above)
                if (outputs && next) issue_x(it + 1);
                // U(it + 1) (E(it) has read U(it))
                if (next) {
                    if (!zero_u && !wait_m(&vu_full, (it + 1) & 1)) break;
                    issue_u(it + 1);
                }
            }
            if (*abort_v && last) wait_cycles(last, last_par);   // drain (bounded)
        }
        __syncwarp();
    } else if (warp == kWarpGate) {
        // ---------------- gates: log alpha two chunks ahead (cp.async; beta enters through the
        // prep kernel's T operands only), the scan of chunk it into set it % 2 once the chunk
        // two back has been consumed
        auto issue_gate = [&](int it) {
            if (it < n_it) {
                uint32_t *dst = sGate + (it & 1) * 128;
                if (GATE == 1)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int r = 2 * lane + e, t = (c_begin + it) * 64 + r;
                        const bool valid = t < a.T;
                        const size_t tok = valid ? ((size_t)b * a.T + t) * a.H + h : 0;
                        cp_async4(dst + 64 + r, a.log_alpha + tok, valid ? 4 : 0);   // zeros past T
                    }
                if (l2)   // the chunk's 128 row norms, 16 bytes per lane
                    cp_async16(sNorm + (it & 1) * 128 + 4 * lane,
                               a.norms + ((size_t)bh * a.NC + c_begin + it) * 128 + 4 * lane);
            }
            cp_async_commit();
        };
        issue_gate(0);
        issue_gate(1);
        for (int it = 0; it < n_it; ++it) {
            if (it >= 2 && !wait_bar(&gset_free[it & 1], ((it - 2) >> 1) & 1)) break;
            cp_async_wait_group1();
            __syncwarp();
            const uint32_t *gw = sGate + (it & 1) * 128;
            float l[2] = {0.f, 0.f};
            if (GATE == 1) {
                l[0] = __uint_as_float(gw[64 + 2 * lane]);
                l[1] = __uint_as_float(gw[64 + 2 * lane + 1]);
            }
            // the row norms of the fused L2 norm (1 otherwise), read before the set is refilled
            float nq[2] = {1.f, 1.f}, nk[2] = {1.f, 1.f};
            if (l2) {
                const float *nv = sNorm + (it & 1) * 128;
                nq[0] = nv[2 * lane]; nq[1] = nv[2 * lane + 1];
                nk[0] = nv[64 + 2 * lane]; nk[1] = nv[64 + 2 * lane + 1];
            }
            __syncwarp();
            issue_gate(it + 2);
            float p = l[0] + l[1];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, p, o);
                if (lane >= o) p += y;
            }
            const float g1 = p, g0 = p - l[1];
            const float glast = __shfl_sync(0xffffffffu, g1, 31);
            const float gmid = __shfl_sync(0xffffffffu, g1, 15);
            const float gfirst = __shfl_sync(0xffffffffu, g0, 0);
            const int r = 2 * lane;
            float *sG = vec(it, GV_G), *sGam = vec(it, GV_GAM), *sDel = vec(it, GV_DEL), *sGq = vec(it, GV_GQ),
                  *sE = vec(it, GV_E), *sF = vec(it, GV_F), *sNq = vec(it, GV_NQ), *sNk = vec(it, GV_NK);
            sG[r] = g0; sG[r + 1] = g1;
            sNq[r] = nq[0]; sNq[r + 1] = nq[1];
            sNk[r] = nk[0]; sNk[r + 1] = nk[1];
            const float G0 = __expf(g0), G1 = __expf(g1);
            sGam[r] = G0; sGam[r + 1] = G1;
            sGq[r] = G0 * nq[0]; sGq[r + 1] = G1 * nq[1];
            sDel[r] = __expf(glast - g0) * nk[0]; sDel[r + 1] = __expf(glast - g1) * nk[1];
            const bool fac = gfirst - glast < kSpan;
            if (fac) {
                sE[r] = __expf(g0 - gmid) * nq[0]; sE[r + 1] = __expf(g1 - gmid) * nq[1];
                sF[r] = __expf(gmid - g0) * nk[0]; sF[r + 1] = __expf(gmid - g1) * nk[1];
            }
            if (lane == 0) fac_s[it & 1] = fac;
            mbar_arrive(&g_ready[it & 1]);
        }
        cp_async_wait_all();
    } else if (warp < kWarpO0) {
        // ---------------- state warps (TMEM lane j = row of S^T, value channel j): the two
        // steps of the state's own chain
        {
            float v[32];
            for (int part = 0; part < 4; ++part) {
                const int i0 = 32 * part;
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    v[u] = init_identity ? (i0 + u == row ? 1.f : 0.f)
                                         : (init_ptr ? init_ptr[(size_t)(i0 + u) * 128 + row] : 0.f);
                tmem_st32(tm + TM_S + i0, v);
            }
            tmem_wait_st();
        }
        for (int it = 0; it < n_it; ++it) {
            const uint32_t par = it & 1;
            if (it >= 1 && !wait_bar(&u_done, par ^ 1)) break;
            if (!wait_bar(&g_ready[it & 1], (it >> 1) & 1)) break;
            // S^T -> bf16 pairs (the A operand of [W S | Q S]) and S^T <- gamma S^T, two
            // 32-column parts per TMEM round trip
            {
                const float gamma = lds32f(vec_s(it, GV_GAM) + 4 * 63);
#pragma unroll 1
                for (int pp = 0; pp < 2; ++pp) {
                    float v[2][32];
                    tmem_ld32(tm + TM_S + 64 * pp, v[0]);
                    tmem_ld32(tm + TM_S + 64 * pp + 32, v[1]);
                    tmem_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t pk[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) pk[u] = pack_bf16(v[hh][2 * u], v[hh][2 * u + 1]);
                        tmem_st16u(tm + TM_SB + 32 * pp + 16 * hh, pk);
#pragma unroll
                        for (int u = 0; u < 32; ++u) v[hh][u] *= gamma;
                        tmem_st32(tm + TM_S + 64 * pp + 32 * hh, v[hh]);
                    }
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&sb_ready);
            // P(it), columns 32..63 (warps 4, 5: TMEM lanes 0..63), while [W S | Q S](it) runs
            if (outputs) {
                if ((warp & 3) < 2) {
                    if (!wait_bar(&x_done, par)) break;
                    build_p_half(it, 1);
                    fence_proxy_async();
                }
                tc_fence_before();
                mbar_arrive(&p_ready);
            }
            // E^T = U^T - (W S)^T in place of (W S)^T (fp32: the next product's A operand,
            // read as tf32) and G (Q S)^T in place of (Q S)^T
            if (!wait_bar(&d_done, par)) break;
            {
                const uint32_t sGam = vec_s(it, GV_GQ);
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float ws[32], uu[32], qs[32];
                    tmem_ld32(tm + TM_WE + 32 * hh, ws);
                    if (!zero_u) tmem_ld32(tm + TM_U + 32 * hh, uu);
                    if (outputs) tmem_ld32(tm + TM_QO + 32 * hh, qs);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 32; ++u) ws[u] = round_tf32((zero_u ? 0.f : uu[u]) - ws[u]);
                    tmem_st32(tm + TM_WE + 32 * hh, ws);
                    if (outputs) {
#pragma unroll
                        for (int u4 = 0; u4 < 8; ++u4) {
                            const float4 g4 = lds128f(sGam + 4 * (32 * hh + 4 * u4));
                            qs[4 * u4] *= g4.x; qs[4 * u4 + 1] *= g4.y; qs[4 * u4 + 2] *= g4.z; qs[4 * u4 + 3] *= g4.w;
                        }
                        tmem_st32(tm + TM_QO + 32 * hh, qs);
                    }
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&e_ready);
            mbar_arrive(&gset_free[it & 1]);
        }
        if (n_it > 0 && wait_bar(&u_done, (n_it - 1) & 1) && fin_ptr) {
            float v[32];
            for (int part = 0; part < 4; ++part) {
                const int i0 = 32 * part;
                tmem_ld32(tm + TM_S + i0, v);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 32; ++u) fin_ptr[(size_t)(i0 + u) * 128 + row] = v[u];
            }
        }
    } else {
        // ---------------- operand / output warps
        const int to_ = tid - 32 * kWarpO0;   // 0..127
        constexpr int kOutBoxes = sizeof(Tout) == 2 ? 2 : 4;
        const bool prows = (warp & 3) < 2;    // TMEM lanes 0..63: the Q K^T rows of X
        // W^T (lane i = key channel, 64 tokens) -> W (bf16, K-major) in the W slot of stage it:
        // column i of the 64 token rows (a warp's 32 channels fill 64 contiguous bytes of a row)
        auto convert_w = [&](int it) -> bool {
            if (!wait_bar(&w_done, it & 1)) return false;
            const uint32_t dst = smem_u32(stage(it)) + C_OFF_W + (row >> 6) * C_KB;
            const uint32_t ci = row & 63;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float w[32];
                tmem_ld32(tm + TM_W + 32 * hh, w);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    sts16(dst + sw128_off(32 * hh + u, ci), __bfloat16_as_ushort(__float2bfloat16_rn(w[u])));
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&w_ready);
            return true;
        };
        // (thread 0 of these warps) chunk it's z tile into the z slot
        int z_last = -1;
        auto load_z = [&](int it) {
            mbar_arrive_expect_tx(&z_full, 16384);
            for (int kb = 0; kb < 2; ++kb)
                tma_load_4d(sm + C_Z + kb * 8192, &tz, &z_full, 64 * kb, h, (c_begin + it) * 64, b);
            z_last = it;
        };
        // chunk it's output O^T (lane j = value channel, 64 tokens) -> staging -> TMA store
        auto emit = [&](int it) {
            float o[2][32];
            tmem_ld32(tm + TM_QO, o[0]);
            tmem_ld32(tm + TM_QO + 32, o[1]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&o_read);
            if (to_ == 0) bulk_wait_read_all();   // the previous store has read the staging
            named_sync(1, 128);
            const int j = row;
            if (sizeof(Tout) == 2 && zgate) {   // out = o silu(z); z(r, j) from the z tile
                if (!wait_bar(&z_full, it & 1)) return;
                const uint32_t zt = sm_s + C_Z + (j >> 6) * 8192;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int r = 0; r < 32; ++r)
                        o[hh][r] *= silu_tanh(__bfloat162float(__ushort_as_bfloat16(lds16(zt + sw128_off(32 * hh + r, j & 63)))));
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (sizeof(Tout) == 2) {
                    const uint32_t dst = sm_s + C_OUT + (j >> 6) * 8192;
#pragma unroll
                    for (int r = 0; r < 32; ++r)
                        sts16(dst + sw128_off(32 * hh + r, j & 63), __bfloat16_as_ushort(__float2bfloat16_rn(o[hh][r])));
                } else {
                    const uint32_t dst = sm_s + C_OUT + (j >> 5) * 8192;
                    const int cj = j & 31;
#pragma unroll
                    for (int r = 0; r < 32; ++r) {
                        const int rr = 32 * hh + r;
                        sts32f(dst + rr * 128 + ((((cj >> 2) ^ (rr & 7)) & 7) << 4) + ((cj & 3) << 2), o[hh][r]);
                    }
                }
            }
            fence_proxy_async();
            named_sync(1, 128);
            if (to_ == 0) {
                constexpr int cols = sizeof(Tout) == 2 ? 64 : 32;
                const int t0 = (c_begin + it) * 64;
#pragma unroll
                for (int kb = 0; kb < kOutBoxes; ++kb)
                    tma_store_4d(&to, sm + C_OUT + kb * 8192, cols * kb, h, t0, b);
                bulk_commit();
                if (sizeof(Tout) == 2 && zgate && it + 1 < n_it) load_z(it + 1);   // the z tile is read
            }
        };
        // Kt^T of channel blocks [ib0, ib0 + nib) (8 key channels each): ldmatrix.trans of the
        // k tile gives each thread channel i and two consecutive tokens r, r + 1 of one 8 x 8
        // block; Kt^T[i][r] = delta_r k_r[i], tf32, into row 64 + i of [P; Kt^T]
        auto kt_blocks = [&](int it, int ib0, int nib) {
            const uint32_t kbase = smem_u32(stage(it)) + C_OFF_K;
            const uint32_t sDel = vec_s(it, GV_DEL);
            const int m = lane >> 3;
            // this lane's eight token pairs r = 8 q + 2 (lane % 4), q = 0..7: their decays once
            float2 d[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) d[q] = lds64f(sDel + 4 * (8 * q + 2 * (lane & 3)));
#pragma unroll 1
            for (int ib = ib0; ib < ib0 + nib; ++ib) {
                const int kb = ib >> 3, c8 = ib & 7, i = 8 * ib + (lane >> 2);
                uint32_t v[2][4];   // all loads first, then the products and stores
#pragma unroll
                for (int rq = 0; rq < 2; ++rq) {
                    const int rr = 8 * (4 * rq + m) + (lane & 7);   // the token row this lane addresses
                    ldsm_x4_trans(kbase + kb * C_KB + rr * 128 + ((c8 ^ (rr & 7)) << 4), v[rq]);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int r = 8 * q + 2 * (lane & 3);
                    const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v[q >> 2][q & 3]));
                    sts64f(sm_s + C_BU + (r >> 5) * C_BU_KB + sw128_off32(64 + i, r & 31), round_tf32(d[q].x * kv.x),
                           round_tf32(d[q].y * kv.y));
                }
            }
        };
        if (sizeof(Tout) == 2 && zgate && to_ == 0 && n_it > 0) load_z(0);
        bool ok = n_it > 0 && convert_w(0);
        for (int it = 0; ok && it < n_it; ++it) {
            const uint32_t par = it & 1;
            // the previous chunk's output first: its TMEM read releases TM_QO to [W S | Q S](it)
            if (it >= 1) {
                if (!wait_bar(&u_done, par ^ 1)) break;
                if (outputs) emit(it - 1);
            }
            if (!wait_bar(&qkw_full[it & 1], (it >> 1) & 1) || !wait_bar(&g_ready[it & 1], (it >> 1) & 1)) break;
            if (outputs && prows) {
                // P(it), columns 0..31 (the state warps take 32..63)
                if (!wait_bar(&x_done, par)) break;
                build_p_half(it, 0);
                kt_blocks(it, 3 * (warp - 8) + 10, 3);   // warps 8, 9: channel blocks 10..15
            } else if (outputs) {
                kt_blocks(it, warp == kWarpO0 ? 0 : 5, 5);   // warps 7, 10: blocks 0..4, 5..9
            } else {
                kt_blocks(it, 4 * (warp - kWarpO0), 4);     // no P: four blocks per warp
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&p_ready);
            mbar_arrive(&kt_ready);
            mbar_arrive(&stage_free[it & 1]);
            mbar_arrive(&gset_free[it & 1]);
            // W(it + 1), issued after [W S | Q S](it)
            if (it + 1 < n_it && !convert_w(it + 1)) break;
        }
        if (outputs && n_it > 0 && !*abort_v && wait_bar(&u_done, (n_it - 1) & 1)) emit(n_it - 1);
        if (to_ == 0) {
            bulk_wait_all();   // the output stores' global writes
            if (z_last >= 0) wait_cycles(&z_full, (uint32_t)z_last & 1);   // (bounded) a z load in flight
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmb, 512);
}
template <typename Tout, int GATE>
int launch_chain(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
                 const CUtensorMap &mz, const ChainArgs &ca, unsigned grid, cudaStream_t stream) {
    const int smem = (int)C_TOTAL + 1024;
    if (cudaFuncSetAttribute(gdn_chain_kernel<Tout, GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return kErrCuda;
    gdn_chain_kernel<Tout, GATE><<<grid, kChainThreads, smem, stream>>>(mq, mk, mv, mo, mz, ca);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

// Workspace of the two-kernel path: the segments' states [3][B*H][nseg][128][128] fp32 (when
// few long chains are split), then the T operands [B*H][NC][16 KB], then the row norms of the
// fused L2 norm [B*H][NC][128] fp32.
size_t gdn_split_workspace_bytes(const ChunkProblem &p) {
    int nseg, len;
    tc_segment_split(p, &nseg, &len);
    const size_t seg = nseg > 1 ? (size_t)3 * p.B * p.H * nseg * 16384 * sizeof(float) : 0;
    return seg + (size_t)p.B * p.H * p.NC * (16384 + 512);
}

// The output gate's z tile takes the free half of the bf16 output staging.
bool gdn_split_fuse_supported(const ChunkProblem &p) { return !(p.fuse & kFuseGate) || p.out_bf16; }

int launch_gdn_split(const ChunkProblem &p, void *workspace, int *status_word, cudaStream_t stream) {
    int nseg, seg_len;
    tc_segment_split(p, &nseg, &seg_len);
    const unsigned bh = (unsigned)(p.B * p.H);
    const size_t seg_bytes = nseg > 1 ? (size_t)3 * bh * nseg * 16384 * sizeof(float) : 0;
    unsigned char *tops = reinterpret_cast<unsigned char *>(workspace) + seg_bytes;
    const unsigned nchunks = bh * (unsigned)p.NC;
    float *norms = reinterpret_cast<float *>(tops + (size_t)nchunks * 16384);
    const bool zgate = (p.fuse & kFuseGate) != 0;
    CUtensorMap mq, mk, mv, mo, mz;
    if (!tc_make_map(&mq, p.q, p.B, p.T, p.H, false) || !tc_make_map(&mk, p.k, p.B, p.T, p.H, false) ||
        !tc_make_map(&mv, p.v, p.B, p.T, p.H, false) ||
        !tc_make_map(&mo, p.out ? p.out : p.q, p.B, p.T, p.H, p.out ? !p.out_bf16 : false) ||
        !tc_make_map(&mz, zgate ? p.z : p.q, p.B, p.T, p.H, false))   // (unused unless gated)
        return kErrCuda;
    {   // every chunk's T operands: persistent CTAs, four per SM
        auto kern = p.gate == 1 ? gdn_prep_kernel<1> : gdn_prep_kernel<0>;
        const int smem = (int)PR_TOTAL + 1024;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return kErrCuda;
        const unsigned grid = std::min<unsigned>(nchunks, 4u * 152u);
        kern<<<grid, kPrepThreads, smem, stream>>>(mk, mq, (const __nv_bfloat16 *)p.beta, p.log_alpha, tops, norms,
                                                   (int)p.T, (int)p.H, p.NC, nchunks, p.fuse, status_word);
        if (cudaGetLastError() != cudaSuccess) return kErrCuda;
    }
    ChainArgs ca{p.log_alpha, p.init_state, p.final_state, tops, status_word,
                 (int)p.B, (int)p.T, (int)p.H, p.NC, 0, 1, p.NC, nullptr, nullptr, nullptr, p.fuse, norms};
    auto launch = [&](const ChainArgs &c, unsigned grid) {
        if (p.out_bf16)
            return p.gate == 1 ? launch_chain<__nv_bfloat16, 1>(mq, mk, mv, mo, mz, c, grid, stream)
                               : launch_chain<__nv_bfloat16, 0>(mq, mk, mv, mo, mz, c, grid, stream);
        return p.gate == 1 ? launch_chain<float, 1>(mq, mk, mv, mo, mz, c, grid, stream)
                           : launch_chain<float, 0>(mq, mk, mv, mo, mz, c, grid, stream);
    };
    if (nseg <= 1) return launch(ca, bh);
    // segments: end states (two runs per segment), chaining, then outputs
    float *ws = reinterpret_cast<float *>(workspace);
    const size_t per = (size_t)bh * nseg * 16384;
    ca.nseg = nseg;
    ca.seg_len = seg_len;
    ca.ws_phi = ws;
    ca.ws_s0 = ws + per;
    ca.ws_start = ws + 2 * per;
    ca.role = 1;
    int rc = launch(ca, bh * nseg * 2);
    if (rc != kOk) return rc;
    rc = tc_launch_seg_combine(p.init_state, ca.ws_phi, ca.ws_s0, ca.ws_start, bh, nseg, stream);
    if (rc != kOk) return rc;
    ca.role = 2;
    return launch(ca, bh * nseg);
}

}  // namespace dr
