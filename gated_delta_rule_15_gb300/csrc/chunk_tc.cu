// chunk_tc.cu -- fused chunkwise forward of the gated delta rule on the 5th-generation
// tensor cores (tcgen05, TMEM, TMA), bf16 inputs, d_k = d_v = 128, chunk C = 64, scalar
// gate or no gate.
//
// The chunk form is the one of chunk_simt.cu (see there for its derivation from the
// recurrence of the page "NLP: linear attention summary", KDA section, taken in the order
// of the `gated_delta_rule` loop of the page "linear-attention gated-deltanet guide").
// Here every product is arranged so that the tensor core's M dimension is 128 and the
// state never leaves the SM: the kernel keeps S^T (d_v x d_k, fp32) in tensor memory and,
// per chunk, with g the cumulative log decay, G = exp(g), delta_r = exp(g_C - g_r):
//
//   X   = [Q; K] K^T                     (128 x 64)  raw q.k and k.k products
//   P   = tril(exp(g_r - g_s) Q K^T)     (64 x 64)   read matrix, diagonal included
//   A   = stril(beta_r exp(g_r - g_s) K K^T),  T = (I + A)^-1   (fp32, blocked, see below)
//   U^T = V^T (T diag beta)^T            (128 x 64)  = (T diag(beta) V)^T
//   W^T = K^T (T diag(beta G))^T         (128 x 64)  = (T diag(beta) (K*G))^T
//   D   = S^T [W; Q]^T                   (128 x 128) = [(W S)^T | (Q S)^T]
//   E^T = U^T - (W S)^T
//   S^T <- gamma S^T + (E^T diag(delta)) K                 (state carried to the next chunk)
//   O^T = (Q S)^T diag(G) + E^T P^T                        (chunk output)
//
// Precision: P, E^T and E^T diag(delta) enter their products as a bf16 pair (high part and
// the bf16 rounding of the remainder), so those products carry ~2^-16 relative error
// instead of bf16's 2^-8; S^T, W and the T factors enter as single bf16 operands, Q exactly
// (its decay G is applied to Q S in fp32).  A
// rounding model of this arithmetic against the fp64 oracle puts the output error at
// ~1e-2 x RMS (about 3e-2 without the pairs).
//
// One CTA per (b, h), 256 threads, the whole TMEM (512 columns): S^T [0,128), D [128,256),
// X [256,320) (later E^T P^T), U^T [320,384), W^T [384,448).  T = (I + A)^-1 is built by
// 16 x 16 blocks: the diagonal blocks by right-looking substitution (one thread per column),
// the blocks below them by warp-level TF32 mma.sync chains, T_ij = -T_ii sum_k A_ik T_kj,
// one warp per block column (no cross-warp dependence).  q, k, v tiles (64 tokens x 128, bf16) arrive
// by TMA with 128-byte swizzle into a double-buffered stage; the next chunk's tiles load
// while the current chunk computes.  Operands written by the CUDA cores (P, T diag beta,
// W, Q*G, S^T, E^T) use the same swizzled K-major layout; V and K tiles also serve as
// MN-major operands directly.  One thread issues the MMAs; completion is tracked with
// tcgen05.commit on an mbarrier.  Every wait is bounded by a cycle budget: on expiry the
// kernel records DR_ERR_TIMEOUT in the status word, drains its own copies and MMAs (with
// the same bound), frees TMEM and returns.
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

constexpr int kThreads = 256;                  // compute warps 0..7
constexpr int kMmaWarp = 8;                    // warp 8 only issues the tcgen05 MMAs
constexpr int kCtaThreads = kThreads + 32;
constexpr uint32_t kStageBytes = 49152;
// stage layout: [Q kb0 | K kb0 | Q kb1 | K kb1 | V kb0 | V kb1], 8 KB each (64 x 64 bf16)
constexpr uint32_t OFF_K0 = 8192, OFF_V0 = 32768;
constexpr uint32_t SM_W = 2 * kStageBytes;    // T diag beta (+G) for the U/W products, then
                                              // [W kb0 | Q kb0 | W kb1 | Q kb1]: the 128-row
                                              // B operand [W; Q] of D (W 64 x 128 K-major and
                                              // a copy of the chunk's Q), then the low part
                                              // of E^T
constexpr uint32_t SM_ST = SM_W + 32768;      // S^T 128 x 128 K-major; fp32 T during the solve
constexpr uint32_t SM_ET = SM_ST + 32768;     // E^T (high) 128 x 64
constexpr uint32_t SM_ET2 = SM_ET + 16384;    // E^T diag(delta) (high); fp32 A during the solve
                                              // SM_ET..SM_ET2 + 16 KB: the output tile at the end
constexpr uint32_t SM_P = SM_ET2 + 16384;     // P (high part) 64 x 64 K-major
constexpr uint32_t SM_PLO = SM_P + 8192;      // P (low part)
// The low part of E^T diag(delta) goes to the current stage's V tile, which is free from the
// completion of the U/W products until the stage is reloaded after the state update.
constexpr uint32_t SM_ETLO = SM_W, SM_OUT = SM_ET;
constexpr uint32_t SM_SMALL = SM_PLO + 8192;  // per-token vectors and solve scratch
constexpr uint32_t SM_A = SM_ET2;   // fp32 A during the solve
constexpr uint32_t SM_TB = SM_W;    // T diag(beta), T diag(beta G) until the U/W products
constexpr uint32_t SM_TOTAL = SM_SMALL + 8192;
static_assert(SM_TOTAL + 1024 <= 227 * 1024, "layout");
constexpr uint32_t TM_S = 0, TM_D = 128, TM_X = 256, TM_U = 320, TM_W = 384, TM_PE = 448;
// TM_D: [ (W S)^T | (Q S)^T ];  TM_X: [Q; K] K^T;  TM_PE: E^T P^T
// Largest in-chunk log-decay span for which exp(g_r - g_s) is formed as a product of two
// exponentials around the chunk's middle token (both factors stay within fp32 range).
constexpr float kFactorSpan = 80.f;

constexpr uint32_t ID_KK_N64 = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_MK_N64 = idesc_bf16(128, 64, true, false);
constexpr uint32_t ID_KM_N128 = idesc_bf16(128, 128, false, true);
constexpr uint32_t ID_KK_N128 = idesc_bf16(128, 128, false, false);

struct TcArgs {
    const float *log_alpha;
    const __nv_bfloat16 *beta;
    const float *init_state;
    float *final_state;
    int *status;
    int T, H, NC;
    // Sequence segments (few long chains): role 0 runs whole sequences; role 1 runs each
    // segment twice without outputs -- from S_0 = 0 (end state to ws_s0) and as the
    // transition from S_0 = I with no value term (to ws_phi); role 2 reruns each segment
    // from its true start state (ws_start) writing outputs.  [B*H][nseg][128][128] fp32.
    int role, nseg, seg_len;
    float *ws_phi, *ws_s0, *ws_start;
};

template <typename Tout, int GATE>
__global__ void __launch_bounds__(kCtaThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                const TcArgs a) {
    extern __shared__ unsigned char dsm_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)dsm_raw + 1023) & ~(uintptr_t)1023);
    // mbarriers: TMA stages; per MMA group its completion (committed by the MMA warp) and,
    // for the groups whose operands the compute warps write, "operands ready" (full_*,
    // arrived by thread 0 after the compute warps' barrier).  Each completes once per chunk.
    __shared__ uint64_t bar_tma[2], bar_x, bar_uw, bar_d, bar_s, full_uw, full_d, full_s;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s, factored_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;        // the TMEM lane this thread reads and writes
    // this CTA's chain, token-chunk range, initial/final state and duties
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
    constexpr int kTmaThread = 224;              // lane 0 of warp 7 issues the TMA loads
    constexpr int kGateWarp = 1;                 // warp 1 scans the gates
    float *sG = reinterpret_cast<float *>(sm + SM_SMALL);   // g_r (cumulative log decay)
    float *sGam = sG + 64;     // exp(g_r)
    float *sDel = sG + 128;    // exp(g_63 - g_r)
    float *sBeta = sG + 192;   // beta_r
    float *sE = sG + 256;      // exp(g_r - g_31)
    float *sF = sG + 320;      // exp(g_31 - g_r)
    float *sM = sG + 384;      // 1024 floats of solve scratch
    // raw gate words of two chunks: [slot][beta word | log alpha][64 tokens]
    uint32_t *sGate = reinterpret_cast<uint32_t *>(sG + 1408);
    float *sGamOut = sG + 1664;   // exp(g_r) of the chunk whose outputs are pending
    constexpr int kOutBoxes = sizeof(Tout) == 2 ? 2 : 4;   // 128-byte rows per output box
    constexpr bool kWideOut = sizeof(Tout) == 4;           // fp32 tile covers SM_ET and SM_ET2

    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(&bar_x, 1);
        mbar_init(&bar_uw, 1);
        mbar_init(&bar_d, 1);
        mbar_init(&bar_s, 1);
        mbar_init(&full_uw, 1);
        mbar_init(&full_d, 1);
        mbar_init(&full_s, 1);
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
    const uint32_t tm = tmem_base_s + ((uint32_t)(32 * quarter) << 16);   // + this warp's lanes
    // operand descriptors of the shared-memory base: K-major, and MN-major with the two
    // 64-wide atoms 8192 or 16384 bytes apart
    const uint64_t dK0 = smem_desc_sw128(smem_u32(sm), 16, 1024);
    const uint64_t dM8 = smem_desc_sw128(smem_u32(sm), 8192, 1024), dM16 = smem_desc_sw128(smem_u32(sm), 16384, 1024);

    // S^T[j][i] = S_0[i][j]: this thread owns j = row and i in [64 half, 64 half + 64).
    if (warp < kMmaWarp) {
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                v[u] = init_identity ? (i0 + u == row ? 1.f : 0.f)
                                     : (init_ptr ? init_ptr[(size_t)(i0 + u) * 128 + row] : 0.f);
            tmem_st32(tm + TM_S + i0, v);
        }
        tmem_wait_st();
    }

    // `it` counts this CTA's chunks (stage, barrier phases); `c` is the global chunk index
    auto issue_tma = [&](int it, int c) {
        const int s = it & 1;
        unsigned char *st = sm + s * kStageBytes;
        mbar_arrive_expect_tx(&bar_tma[s], kStageBytes);
        const int t0 = c * 64;
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(st + kb * 16384, &tq, &bar_tma[s], 64 * kb, h, t0, b);
            tma_load_4d(st + kb * 16384 + OFF_K0, &tk, &bar_tma[s], 64 * kb, h, t0, b);
            tma_load_4d(st + OFF_V0 + kb * 8192, &tv, &bar_tma[s], 64 * kb, h, t0, b);
        }
    };
    // beta (the aligned 32-bit word holding it) and log alpha of chunk c, two tokens per
    // lane of warp 1 (warp 0 issues the MMAs), copied asynchronously one chunk ahead
    const size_t ntok = (size_t)(gridDim.x / (a.role == 0 ? 1 : (a.role == 1 ? 2 * a.nseg : a.nseg))) * a.T;
    auto issue_gate = [&](int it, int c) {
        uint32_t *dst = sGate + (it & 1) * 128;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * lane + e, t = c * 64 + r;
            const bool valid = t < a.T;
            const size_t tok = valid ? ((size_t)b * a.T + t) * a.H + h : 0;
            if (valid && tok + 1 == ntok && ((2 * tok) & 3) == 0) {
                // the 32-bit word would run past the end of beta: load this value alone
                dst[r] = (uint32_t)__bfloat16_as_ushort(a.beta[tok]);
            } else {
                cp_async4(dst + r, reinterpret_cast<const char *>(a.beta) + ((2 * tok) & ~(size_t)3),
                          valid ? 4 : 0);
            }
            cp_async4(dst + 64 + r, GATE == 1 ? (const void *)(a.log_alpha + tok) : (const void *)a.beta,
                      (GATE == 1 && valid) ? 4 : 0);
        }
        cp_async_commit();
    };
    const int n_it = c_end - c_begin;
    if (tid == kTmaThread && n_it > 0) issue_tma(0, c_begin);
    if (warp == kGateWarp && n_it > 0) issue_gate(0, c_begin);

    bool out_pending = false;       // chunk whose outputs wait in TMEM for the write-out
    bool store_outstanding = false; // a TMA store may still be reading SM_OUT
    int last_tma_it = 0;            // iteration of the most recent TMA load (TMA thread)
    bool s_outstanding = false;     // MMA group S (state update, E^T P^T) committed, not waited
    int cur_t0 = 0;                 // t0 of the chunk whose outputs are pending
    auto fail = [&]() {
        abort_s = 1;
        atomicExch(a.status, kErrTimeout);
    };
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
        if (!wait_cycles(bar, parity)) fail();
        tc_fence_after();
    };
    // (MMA warp) wait for chunk c's tiles, then X = [Q; K] K^T into TM_X
    auto issue_x = [&](int it) {
        if (!wait_cycles(&bar_tma[it & 1], (it >> 1) & 1)) fail();
        unsigned char *st = sm + (it & 1) * kStageBytes;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
            mma_bf16(tmem_base_s + TM_X, desc_add(dK0, (uint32_t)((st + o) - sm)),
                     desc_add(dK0, (uint32_t)((st + OFF_K0 + o) - sm)), ID_KK_N64, ks > 0);
        }
        mma_commit(&bar_x);
    };

    // Output of the chunk at t0: o = G_r (Q S)^T + E^T P^T, staged row-major at SM_OUT in
    // 128-byte swizzled boxes and written by TMA (rows past T are skipped).  Needs group S.
    auto write_out = [&](int t0) {
        float o[32], pe[32];
        tmem_ld32(tm + TM_D + 64 + 32 * half, o);
        tmem_ld32(tm + TM_PE + 32 * half, pe);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) o[u] = fmaf(sGamOut[32 * half + u], o[u], pe[u]);
        const int j = row;
        if (sizeof(Tout) == 2) {
            unsigned char *dst = sm + SM_OUT + (j >> 6) * 8192;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                *reinterpret_cast<__nv_bfloat16 *>(dst + sw128_off(32 * half + u, j & 63)) =
                    __float2bfloat16_rn(o[u]);
        } else {
            unsigned char *dst = sm + SM_OUT + (j >> 5) * 8192;
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
        named_sync(1, kThreads);
        if (tid == 0) {
            constexpr int cols = sizeof(Tout) == 2 ? 64 : 32;
#pragma unroll
            for (int kb = 0; kb < kOutBoxes; ++kb)
                tma_store_4d(&to, sm + SM_OUT + kb * 8192, cols * kb, h, t0, b);
            bulk_commit();
            store_outstanding = true;
            if (kWideOut) {   // the fp32 tile also covers SM_A, written next by P/A
                bulk_wait_read_all();
                store_outstanding = false;
            }
        }
        if (kWideOut) named_sync(1, kThreads);
    };

    // ---------------- MMA warp: issues every tcgen05.mma group in chunk order, each once its
    // operands are ready, and commits it to the barrier the compute warps wait on.
    if (warp == kMmaWarp) {
        if (lane == 0 && n_it > 0) {
            uint64_t *last = &bar_x;   // most recent commit (drained on abort)
            uint32_t last_par = 0;
            issue_x(0);
            for (int it = 0; it < n_it && !abort_s; ++it) {
                const uint32_t par = it & 1;
                unsigned char *st = sm + (it & 1) * kStageBytes;
                // U^T = V^T (T diag beta)^T,  W^T = K^T (T diag(beta G))^T
                if (!wait_cycles(&full_uw, par)) { fail(); break; }
                tc_fence_after();
                if (!zero_u)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem_base_s + TM_U, desc_add(dM8, (uint32_t)((st + OFF_V0 + ks * 2048) - sm)),
                             desc_add(dK0, (uint32_t)(SM_TB + ks * 32)), ID_MK_N64, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem_base_s + TM_W, desc_add(dM16, (uint32_t)((st + OFF_K0 + ks * 2048) - sm)),
                             desc_add(dK0, (uint32_t)(SM_TB + 8192 + ks * 32)), ID_MK_N64, ks > 0);
                mma_commit(&bar_uw);
                last = &bar_uw; last_par = par;
                // D = S^T [W; Q]^T in one N = 128 product: (W S)^T | (Q S)^T
                if (!wait_cycles(&full_d, par)) { fail(); break; }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tmem_base_s + TM_D, desc_add(dK0, SM_ST + o), desc_add(dK0, SM_W + o),
                             outputs ? ID_KK_N128 : ID_KK_N64, ks > 0);
                }
                mma_commit(&bar_d);
                last = &bar_d; last_par = par;
                // S^T += (E^T diag delta) K ;  PE = E^T P^T  (high/low pairs); then the next X
                if (!wait_cycles(&full_s, par)) { fail(); break; }
                tc_fence_after();
                unsigned char *e2[2] = {sm + SM_ET2, st + OFF_V0};
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmem_base_s + TM_S, desc_add(dK0, (uint32_t)((e2[part] + ks * 32) - sm)),
                                 desc_add(dM16, (uint32_t)((st + OFF_K0 + ks * 2048) - sm)), ID_KM_N128, 1);
                const uint32_t ea[3] = {SM_ET, SM_ET, SM_ETLO}, pb[3] = {SM_P, SM_PLO, SM_P};
                if (outputs)
#pragma unroll
                for (int part = 0; part < 3; ++part)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmem_base_s + TM_PE, desc_add(dK0, ea[part] + ks * 32),
                                 desc_add(dK0, pb[part] + ks * 32), ID_KK_N64, (part | ks) != 0);
                mma_commit(&bar_s);
                last = &bar_s; last_par = par;
                if (it + 1 < n_it) {
                    issue_x(it + 1);
                    last = &bar_x; last_par = (it + 1) & 1;
                }
            }
            if (abort_s) wait_cycles(last, last_par);   // drain this warp's MMAs (bounded)
        }
        __syncwarp();
    } else {

    for (int it = 0; it < n_it; ++it) {
        const int c = c_begin + it;
        const int s = it & 1;
        const uint32_t par = it & 1;              // parity of this chunk's MMA barriers
        unsigned char *st = sm + s * kStageBytes;
        const int t0 = c * 64;

        // ---- 1. X = [Q; K] K^T of this chunk: issued by the MMA warp (the first chunk's at
        //         once, later ones right after the previous chunk's state update)
        // ---- 2. cumulative log decay of this chunk (gate warp; its gates arrived by cp.async)
        if (warp == kGateWarp) {
            cp_async_wait_all();
            __syncwarp();
            const uint32_t *gw = sGate + s * 128;
            float l[2], bt[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 2 * lane + e, t = t0 + r;
                const size_t tok = t < a.T ? ((size_t)b * a.T + t) * a.H + h : 0;
                const uint32_t wd = gw[r];
                const uint16_t hb = (uint16_t)(((2 * tok) & 2) ? (wd >> 16) : (wd & 0xffffu));
                bt[e] = __bfloat162float(__ushort_as_bfloat16(hb));
                l[e] = __uint_as_float(gw[64 + r]);
            }
            __syncwarp();
            if (it + 1 < n_it) issue_gate(it + 1, c + 1);
            float p = l[0] + l[1];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, p, o);
                if (lane >= o) p += y;
            }
            const float g1 = p, g0 = p - l[1];                     // g_{2l}, g_{2l+1}
            const float glast = __shfl_sync(0xffffffffu, g1, 31);  // g_63
            const float gmid = __shfl_sync(0xffffffffu, g1, 15);   // g_31
            const float gfirst = __shfl_sync(0xffffffffu, g0, 0);  // g_0
            const int r = 2 * lane;
            sG[r] = g0; sG[r + 1] = g1;
            sBeta[r] = bt[0]; sBeta[r + 1] = bt[1];
            sGam[r] = __expf(g0); sGam[r + 1] = __expf(g1);
            sDel[r] = __expf(glast - g0); sDel[r + 1] = __expf(glast - g1);
            const bool fac = gfirst - glast < kFactorSpan;
            if (fac) {
                sE[r] = __expf(g0 - gmid); sE[r + 1] = __expf(g1 - gmid);
                sF[r] = __expf(gmid - g0); sF[r + 1] = __expf(gmid - g1);
            }
            if (lane == 0) factored_s = fac;
        }
        // ---- 3. previous chunk: wait for its state update, write its outputs; then the
        //         stage it used is free for the next chunk's tiles
        if (s_outstanding) {
            wait_bar(&bar_s, par ^ 1);
            s_outstanding = false;
        }
        named_sync(1, kThreads);    // gate vectors published; previous chunk's MMAs done
        if (abort_s) break;
        if (out_pending && outputs) write_out(cur_t0);
        if (tid == kTmaThread && it + 1 < n_it) {
            issue_tma(it + 1, c + 1);
            last_tma_it = it + 1;
        }
        // keep this chunk's exp(g_r) for its deferred write-out (write_out above ended with
        // a barrier, so no thread still reads the previous values)
        if (tid < 64) sGamOut[tid] = sGam[tid];

        // ---- 4. P (rows 0..63 of X, bf16 high/low) and A (rows 64..127 of X, fp32)
        wait_bar(&bar_x, par);
        {
            float x[32];
            tmem_ld32(tm + TM_X + 32 * half, x);
            tmem_wait_ld();
            const int c0 = 32 * half;
            const bool fac = factored_s;
            const int r = quarter < 2 ? row : row - 64;
            float dec[32];   // exp(g_r - g_s), s = c0 + u
            if (fac) {
                const float er = sE[r];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 f4 = *reinterpret_cast<const float4 *>(sF + c0 + 4 * q);
                    dec[4 * q] = er * f4.x; dec[4 * q + 1] = er * f4.y;
                    dec[4 * q + 2] = er * f4.z; dec[4 * q + 3] = er * f4.w;
                }
            } else {
                const float gr = sG[r];
#pragma unroll
                for (int u = 0; u < 32; ++u) dec[u] = __expf(fminf(gr - sG[c0 + u], 0.f));
            }
            if (quarter < 2) {
                uint32_t pk[16], pl[16];
#pragma unroll
                for (int u = 0; u < 32; u += 2) {
                    const int s0 = c0 + u;
                    const float p0 = s0 <= r ? dec[u] * x[u] : 0.f;
                    const float p1 = s0 + 1 <= r ? dec[u + 1] * x[u + 1] : 0.f;
                    pack_hi_lo(p0, p1, pk[u >> 1], pl[u >> 1]);
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const uint32_t off = sw128_off(r, c0 + 8 * q4);
                    *reinterpret_cast<uint4 *>(sm + SM_P + off) =
                        make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    *reinterpret_cast<uint4 *>(sm + SM_PLO + off) =
                        make_uint4(pl[4 * q4], pl[4 * q4 + 1], pl[4 * q4 + 2], pl[4 * q4 + 3]);
                }
            } else {
                const float br = sBeta[r];
                float *sA = reinterpret_cast<float *>(sm + SM_A);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    float4 v4;
                    const int s0 = c0 + 4 * q4;
                    v4.x = s0 < r ? br * dec[4 * q4] * x[4 * q4] : 0.f;
                    v4.y = s0 + 1 < r ? br * dec[4 * q4 + 1] * x[4 * q4 + 1] : 0.f;
                    v4.z = s0 + 2 < r ? br * dec[4 * q4 + 2] * x[4 * q4 + 2] : 0.f;
                    v4.w = s0 + 3 < r ? br * dec[4 * q4 + 3] * x[4 * q4 + 3] : 0.f;
                    *reinterpret_cast<float4 *>(sA + a_index(r, s0)) = v4;
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(1, kThreads);

        // ---- 5-6. T = (I + A)^-1 (fp32, [64][kTs] at SM_ST), with T diag(beta) and
        //           T diag(beta G) in bf16 at SM_TB
        solve_unit_lower64(reinterpret_cast<const float *>(sm + SM_A),
                           reinterpret_cast<float *>(sm + SM_ST), sM, sm + SM_TB, sBeta, sGam, tid);

        // ---- 7. U^T = V^T (T diag beta)^T,  W^T = K^T (T diag(beta G))^T (MMA warp)
        if (tid == 0) mbar_arrive(&full_uw);
        // ---- 8. meanwhile: S^T to bf16 (MMA operand at SM_ST); S^T <- gamma S^T in TMEM
        {
            const float gamma = sGam[63];
            float v[32];
            unsigned char *dst = sm + SM_ST + half * 16384;
            for (int part = 0; part < 2; ++part) {
                const int i0 = 64 * half + 32 * part;
                tmem_ld32(tm + TM_S + i0, v);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float *f = v + 8 * q4;
                    *reinterpret_cast<uint4 *>(dst + sw128_off(row, 32 * part + 8 * q4)) =
                        make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]),
                                   pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
                }
#pragma unroll
                for (int u = 0; u < 32; ++u) v[u] *= gamma;
                tmem_st32(tm + TM_S + i0, v);
            }
            tmem_wait_st();
        }
        // ---- 9. W from W^T (lane i = key channel, columns = tokens r) into the B operand
        //         [W; Q] of D, and the chunk's Q tiles copied beside it
        wait_bar(&bar_uw, par);
        {
            float w[32];
            tmem_ld32(tm + TM_W + 32 * half, w);
            tmem_wait_ld();
            const int i = row, kb = i >> 6, ci = i & 63;
            unsigned char *dst = sm + SM_W + kb * 16384;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                *reinterpret_cast<__nv_bfloat16 *>(dst + sw128_off(32 * half + u, ci)) =
                    __float2bfloat16_rn(w[u]);
            if (outputs) {   // 16 KB of swizzled tiles: the copy keeps the pattern (1 KB aligned)
                // the tiles arrived by TMA (seen so far by the MMA warp only); this stage's
                // next load is issued after the next chunk's step 3
                if (!wait_cycles(&bar_tma[it & 1], (it >> 1) & 1)) fail();
                const uint4 *qs = reinterpret_cast<const uint4 *>(st);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = tid + 256 * k, kbq = e >> 9, off = e & 511;   // 512 x 16 B per kb
                    reinterpret_cast<uint4 *>(sm + SM_W + kbq * 16384 + 8192)[off] = qs[kbq * 1024 + off];
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(1, kThreads);
        if (abort_s) break;

        // ---- 10. D = S^T [W; Q]^T  (MMA warp)
        if (tid == 0) {
            mbar_arrive(&full_d);
            if (store_outstanding) {   // the previous output tile must have left SM_OUT
                bulk_wait_read_all();  // before E^T is written there
                store_outstanding = false;
            }
        }
        named_sync(1, kThreads);
        wait_bar(&bar_d, par);

        // ---- 11. E^T = U^T - (W S)^T, and E^T diag(delta)  (bf16 high/low pairs); the (Q S)^T
        //          half is read by the deferred write-out
        {
            float ws[32], uu[32];
            tmem_ld32(tm + TM_D + 32 * half, ws);
            tmem_ld32(tm + TM_U + 32 * half, uu);
            tmem_wait_ld();
            if (zero_u)
#pragma unroll
                for (int u = 0; u < 32; ++u) uu[u] = 0.f;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float e[8], ed[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int r = 32 * half + 8 * q4 + u;
                    e[u] = uu[8 * q4 + u] - ws[8 * q4 + u];
                    ed[u] = e[u] * sDel[r];
                }
                const uint32_t off = sw128_off(row, 32 * half + 8 * q4);
                uint32_t eh[4], el[4], dh[4], dlo[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    pack_hi_lo(e[2 * u], e[2 * u + 1], eh[u], el[u]);
                    pack_hi_lo(ed[2 * u], ed[2 * u + 1], dh[u], dlo[u]);
                }
                *reinterpret_cast<uint4 *>(sm + SM_ET + off) = make_uint4(eh[0], eh[1], eh[2], eh[3]);
                *reinterpret_cast<uint4 *>(sm + SM_ETLO + off) = make_uint4(el[0], el[1], el[2], el[3]);
                *reinterpret_cast<uint4 *>(sm + SM_ET2 + off) = make_uint4(dh[0], dh[1], dh[2], dh[3]);
                *reinterpret_cast<uint4 *>(st + OFF_V0 + off) =
                    make_uint4(dlo[0], dlo[1], dlo[2], dlo[3]);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(1, kThreads);

        // ---- 12. S^T += (E^T diag delta) K ;  PE = E^T P^T  (high/low pairs; MMA warp, which
        //          then issues the next chunk's X); completes while the next chunk starts,
        //          whose step 3 waits for it
        if (tid == 0) mbar_arrive(&full_s);
        s_outstanding = true;
        out_pending = true;
        cur_t0 = t0;
    }

    if (!abort_s && s_outstanding) {
        wait_bar(&bar_s, (n_it - 1) & 1);
        s_outstanding = false;
        named_sync(1, kThreads);
        if (!abort_s && out_pending && outputs) write_out(cur_t0);
    }
    if (abort_s) {
        // Drain this CTA's own asynchronous work (bounded) before TMEM is freed; the MMA
        // warp drains its own MMAs.
        if (tid == kTmaThread)   // the last load may still be in flight (bounded wait)
            wait_cycles(&bar_tma[last_tma_it & 1], (last_tma_it >> 1) & 1);
    } else if (fin_ptr) {
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
            tmem_ld32(tm + TM_S + i0, v);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) fin_ptr[(size_t)(i0 + u) * 128 + row] = v[u];
        }
    }
    if (warp == kGateWarp) cp_async_wait_all();
    if (tid == 0 && store_outstanding) bulk_wait_all();
    }   // compute warps
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base_s, 512);
}

// Segment chaining (between the two segment passes): per chain, S_start(0) = S_0 and
// S_start(p + 1) = Phi_p S_start(p) + S0_p, where Phi_p and S0_p are segment p's transition
// and zero-start end state.  One CTA per (chain, block of 32 state columns), fp32.
__global__ void __launch_bounds__(256) seg_combine_kernel(const float *__restrict__ init_state,
                                                           const float *__restrict__ phi,
                                                           const float *__restrict__ s0,
                                                           float *__restrict__ start, int nseg) {
    __shared__ float S[128][33];
    const int cb = blockIdx.x & 3, bh = blockIdx.x >> 2;
    const int tid = threadIdx.x, j = tid & 31, rg = tid >> 5;
    const int col = 32 * cb + j;
    for (int i = rg; i < 128; i += 8)
        S[i][j] = init_state ? init_state[((size_t)bh * 128 + i) * 128 + col] : 0.f;
    __syncthreads();
    for (int p = 0; p < nseg; ++p) {
        const size_t slot = ((size_t)bh * nseg + p) * 16384;
        for (int i = rg; i < 128; i += 8) start[slot + i * 128 + col] = S[i][j];
        if (p + 1 == nseg) break;
        float acc[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) acc[m] = s0[slot + (size_t)(rg + 8 * m) * 128 + col];
        for (int k = 0; k < 128; ++k) {
            const float sk = S[k][j];
#pragma unroll
            for (int m = 0; m < 16; ++m) acc[m] = fmaf(phi[slot + (size_t)(rg + 8 * m) * 128 + k], sk, acc[m]);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 16; ++m) S[rg + 8 * m][j] = acc[m];
        __syncthreads();
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// [B, T, H, 128] viewed as 4-D (128, H, T, B); box of 128-byte rows x 1 x 64 tokens x 1,
// 128-byte swizzle; loads read rows past T as zeros, stores skip them.
bool make_map(CUtensorMap *m, const void *base, int64_t B, int64_t T, int64_t H, bool fp32) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t e = fp32 ? 4 : 2;
    cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {128 * e, (cuuint64_t)H * 128 * e, (cuuint64_t)(T * H) * 128 * e};
    cuuint32_t box[4] = {(cuuint32_t)(128 / e), 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tout, int GATE>
int launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
             const CUtensorMap &mo, const TcArgs &ta, unsigned grid, cudaStream_t stream) {
    const int smem = (int)SM_TOTAL + 1024;
    if (cudaFuncSetAttribute(chunk_tc_kernel<Tout, GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return kErrCuda;
    chunk_tc_kernel<Tout, GATE><<<grid, kCtaThreads, smem, stream>>>(mq, mk, mv, mo, ta);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

bool chunk_tc_supported(const ChunkProblem &p) {
    return p.in_bf16 && p.dk == 128 && p.dv == 128 && p.C == 64 && p.T > 0 &&
           (p.gate == 0 || p.gate == 1);
}

// Few long chains leave most of the GPU's 152 SMs idle while each chain walks its chunks
// one after another; such problems are split into `nseg` segments per chain (at least 16
// chunks each) so that about 152 CTAs work at once.
static constexpr int kGpuSms = 152;
static void tc_segments(const ChunkProblem &p, int *nseg, int *seg_len) {
    *nseg = 1;
    *seg_len = p.NC;
    const int64_t bh = p.B * p.H;
    if (!chunk_tc_supported(p) || bh > kGpuSms / 2 || p.NC < 32) return;
    int n = (int)std::min<int64_t>(p.NC / 16, kGpuSms / bh);
    if (n < 2) return;
    const int len = (p.NC + n - 1) / n;
    *seg_len = len;
    *nseg = (p.NC + len - 1) / len;
}

size_t chunk_tc_workspace_bytes(const ChunkProblem &p) {
    int nseg, len;
    tc_segments(p, &nseg, &len);
    return nseg > 1 ? (size_t)3 * p.B * p.H * nseg * 16384 * sizeof(float) : 0;
}

int launch_chunk_tc(const ChunkProblem &p, void *workspace, int *status_word, cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, p.q, p.B, p.T, p.H, false) || !make_map(&mk, p.k, p.B, p.T, p.H, false) ||
        !make_map(&mv, p.v, p.B, p.T, p.H, false) ||
        !make_map(&mo, p.out, p.B, p.T, p.H, !p.out_bf16))
        return kErrCuda;
    TcArgs ta{p.log_alpha, (const __nv_bfloat16 *)p.beta, p.init_state, p.final_state,
              status_word, (int)p.T, (int)p.H, p.NC, 0, 1, p.NC, nullptr, nullptr, nullptr};
    auto launch = [&](const TcArgs &t, unsigned grid) {
        if (p.out_bf16)
            return p.gate == 1 ? launch_t<__nv_bfloat16, 1>(mq, mk, mv, mo, t, grid, stream)
                               : launch_t<__nv_bfloat16, 0>(mq, mk, mv, mo, t, grid, stream);
        return p.gate == 1 ? launch_t<float, 1>(mq, mk, mv, mo, t, grid, stream)
                           : launch_t<float, 0>(mq, mk, mv, mo, t, grid, stream);
    };
    const unsigned bh = (unsigned)(p.B * p.H);
    int nseg, seg_len;
    tc_segments(p, &nseg, &seg_len);
    if (nseg <= 1) return launch(ta, bh);
    // segments: end states (two runs per segment), chaining, then outputs
    float *ws = reinterpret_cast<float *>(workspace);
    const size_t per = (size_t)bh * nseg * 16384;
    ta.nseg = nseg;
    ta.seg_len = seg_len;
    ta.ws_phi = ws;
    ta.ws_s0 = ws + per;
    ta.ws_start = ws + 2 * per;
    ta.role = 1;
    int rc = launch(ta, bh * nseg * 2);
    if (rc != kOk) return rc;
    seg_combine_kernel<<<bh * 4, 256, 0, stream>>>(p.init_state, ta.ws_phi, ta.ws_s0, ta.ws_start, nseg);
    if (cudaGetLastError() != cudaSuccess) return kErrCuda;
    ta.role = 2;
    return launch(ta, bh * nseg);
}

}  // namespace dr
