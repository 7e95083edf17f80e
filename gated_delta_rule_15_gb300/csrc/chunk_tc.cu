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
//   A   = stril(beta_r exp(g_r - g_s) K K^T),  T = (I + A)^-1   (fp32, blocked)
//   U^T = V^T (T diag beta)^T            (128 x 64)  = (T diag(beta) V)^T
//   W^T = K^T (T diag(beta G))^T         (128 x 64)  = (T diag(beta) (K*G))^T
//   D   = S^T [W; Q]^T                   (128 x 128) = [(W S)^T | (Q S)^T]
//   E^T = U^T - (W S)^T
//   [O^T | S^T] <- [(Q S)^T diag(G) | gamma S^T] + E^T [P; Kt^T]^T,  Kt = diag(delta) K
//
// Precision: the state update and the output's intra-chunk term take E, P and Kt as tf32
// (10 explicit mantissa bits): E^T stays fp32 in tensor memory, where it is the A operand,
// and [P; Kt^T] is one K-major fp32 B operand; S^T (a bf16 A operand in tensor memory), W
// and the T factors enter as single bf16 operands, Q exactly (its decay G is applied to Q S
// in fp32).
//
// One CTA per (b, h): eight compute warps and one warp that only issues the tcgen05 MMAs.
// The chunk steps are software-pipelined across two chunks, so that the MMA groups of one
// run while the CUDA cores work on the other.  In the iteration of chunk c the compute warps
//   1. convert S^T to the bf16 operand of D (in TMEM) and decay S^T,
//   2. write W (from TMEM) as the B operand of D            -> MMA warp: D(c)
//   3. build this chunk's Kt^T and the next chunk's A from its X (already in TMEM), and
//      solve the diagonal blocks of the next chunk's T = (I + A)^-1 while D runs,
//   4. form E^T and G (Q S)^T in TMEM                        -> MMA warp: [O^T | S^T] (c)
//   5. merge the next chunk's T (warps 0..3) while warps 4..7 build the next chunk's P
//                                                           -> MMA warp: X(c+2)
//      and write chunk c's output,
//   6. hand off                                             -> MMA warp: U/W(c+1), stage of
//                                                              c takes c + 2
// and the gate warp scans the gates two chunks ahead.  T = (I + A)^-1 is built by 16 x 16
// blocks (tc_common.cuh).  q, k, v tiles (64 tokens x 128, bf16) arrive by TMA with 128-byte
// swizzle into two stages; operands written by the CUDA cores use the same swizzled K-major
// layout, and the V and K tiles also serve as MN-major operands directly.  Every wait is
// bounded by a cycle budget: on expiry the kernel records DR_ERR_TIMEOUT in the status
// word, drains its own copies and MMAs (with the same bound), frees TMEM and returns.
//
// Fused neighbours (DR_FUSE_* of include/dr.h: L2-normalised q and k, beta from logits, the
// SiLU output gate of the Gated DeltaNet layer, page "linear-attention gated-deltanet
// guide", section 4).  With N = diag(nk), nk_r = 1 / |k_r|, and nq_r = 1 / |q_r|, every
// product is bilinear in the rows of Q and K, so the tiles stay as loaded and the norms
// enter scalings the kernel applies in fp32 anyway: P_rs gets nq_r nk_s, the state update's
// diag(delta) becomes diag(delta nk), the output's G_r becomes G_r nq_r, and the U and W
// operands are T diag(beta) and T diag(beta G nk).  Only A_rs = beta_r nk_r nk_s (...) would
// need every norm while A is built; the kernel builds instead the similar B = N A N^-1,
// B_rs = beta_r nk_r^2 (...), whose row r needs only |k_r| (summed by the row's own
// thread), solves T_B = (I + B)^-1 and writes the operands of T = N^-1 T_B N:
// (T diag beta)_rs = |k_r| T_B,rs nk_s beta_s.  So no extra barrier is needed; the four
// warps that build no A rows compute the norm vectors meanwhile.  The diagonal of the U
// operand stays exact: T_rr = 1 and the gate warp takes beta = sigmoid(logit) rounded to
// bf16, beta's storage dtype, as a stored beta would be.  The output warps multiply by
// silu(z).  z's tile is prefetched into L2 with the chunk's q, k, v and copied by TMA into
// the stage's Q tiles as soon as (Q S)^T has read them (the MMA warp waits for it), two MMA
// groups before the output step needs it; the output is then staged in the V slot (and the
// K tiles for fp32).
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
// Beyond the two stages (lifetimes within the iteration of chunk c, steps as above):
constexpr uint32_t SM_T = 2 * kStageBytes;    // the next chunk's fp32 T (16 KB, swizzled; step 3
constexpr uint32_t SM_TB = SM_T + 16384;      // on) and T diag beta | T diag beta G (16 KB,
                                              // until U/W(c+1))
constexpr uint32_t SM_W = SM_T + 32768;       // 16 KB: W^T 128 x 64 (MN-major B operand of
                                              // (W S)^T; step 2 -> D(c))
constexpr uint32_t SM_A = SM_W + 16384;       // the next chunk's fp32 A (step 3)
constexpr uint32_t SM_BU = SM_A + 16384;      // [P; Kt^T] (tf32, K-major): two K-blocks of 32
constexpr uint32_t BU_KB = 24576;             // tokens, 192 rows x 128 bytes each; P rows
                                              // (step 5 of the chunk before), Kt^T rows (step 3)
constexpr uint32_t SM_SMALL = SM_BU + 2 * BU_KB;   // gate vectors of two chunks, solve scratch
constexpr uint32_t SM_TOTAL = SM_SMALL + 8192;
// fused neighbours only: norm vectors of two chunks [2][7][64]: nq, nk, G nq, beta nk,
// G nk, |k| (1 / nk) and delta nk
constexpr uint32_t SM_NRM = SM_TOTAL;
constexpr uint32_t SM_TOTAL_FUSED = SM_NRM + 3584;
static_assert(SM_TOTAL_FUSED + 1024 <= 227 * 1024, "layout");
// 128-byte-swizzled operands and TMA boxes start on 1024-byte boundaries; [P; Kt^T] holds
// 192 rows of 128 bytes per K-block, the bf16 output staging its rows 128..191 of each
static_assert(SM_T % 1024 == 0 && SM_TB % 1024 == 0 && SM_W % 1024 == 0 && SM_BU % 1024 == 0 &&
              BU_KB % 1024 == 0 && BU_KB == 192 * 128, "layout");
static_assert(16384 + BU_KB + 8192 <= 2 * BU_KB, "output staging inside [P; Kt^T]");
enum { NV_NQ = 0, NV_NK = 1, NV_GQ = 2, NV_BK = 3, NV_GK = 4, NV_RK = 5, NV_DK = 6 };
constexpr uint32_t TM_WE = 0, TM_QO = 64, TM_S = 128, TM_SB = 256, TM_X = 320, TM_U = 384, TM_W = 448;
static_assert(TM_QO == TM_WE + 64 && TM_S == TM_QO + 64 && TM_SB == TM_S + 128 && TM_X == TM_SB + 64 &&
              TM_U == TM_X + 64 && TM_W == TM_U + 64 && TM_W + 64 == 512,
              "TMEM: [O^T | S^T] contiguous (one N = 192 accumulator), 512 columns in all");
// TM_WE: (W S)^T, then E^T (fp32, the A operand of the state update);  TM_QO: (Q S)^T, then
// G (Q S)^T, then O^T: [TM_QO | TM_S] is the accumulator of the state update;  TM_SB: S^T as
// bf16 pairs (the A operand of D);  TM_X: [Q; K] K^T
// Largest in-chunk log-decay span for which exp(g_r - g_s) is formed as a product of two
// exponentials around the chunk's middle token (both factors stay within fp32 range).
constexpr float kFactorSpan = 80.f;

constexpr uint32_t ID_KK_N64 = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_MK_N64 = idesc_bf16(128, 64, true, false);
constexpr uint32_t ID_UPD = idesc_tf32(128, 192);     // [O^T | S^T]: B = [P; Kt^T]
constexpr uint32_t ID_UPD_S = idesc_tf32(128, 128);   // S^T alone (no outputs): B = Kt^T
constexpr uint32_t ID_KM_N64 = idesc_bf16(128, 64, false, true);

struct TcArgs {
    const float *log_alpha;
    const __nv_bfloat16 *beta;
    const float *init_state;
    float *final_state;
    int *status;
    int T, H, NC;
    uint32_t fuse;   // DR_FUSE_* bits
    // Sequence segments (few long chains): role 0 runs whole sequences; role 1 runs each
    // segment twice without outputs -- from S_0 = 0 (end state to ws_s0) and as the
    // transition from S_0 = I with no value term (to ws_phi); role 2 reruns each segment
    // from its true start state (ws_start) writing outputs.  [B*H][nseg][128][128] fp32.
    int role, nseg, seg_len;
    float *ws_phi, *ws_s0, *ws_start;
    // (fused instantiation) the state at every chunk's start, [B*H][NC][dk][dv] fp32, for
    // the backward's recompute: written by roles 0 and 2, which then write no outputs
    float *ckpt;
};

// MODE 0: plain.  MODE 1 (FUSED): the fused neighbours' code is compiled in (each still
// switched by a.fuse).  MODE 2 (CKPT): no outputs; the state at every chunk's start goes to
// a.ckpt (the backward's recompute).  Each instantiation carries only its own code, which
// keeps the register pressure of the others down.
template <typename Tout, int GATE, int MODE>
__global__ void __launch_bounds__(kCtaThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                const __grid_constant__ CUtensorMap tz, const TcArgs a) {
    constexpr bool FUSED = MODE == 1, CKPT = MODE == 2;
    extern __shared__ unsigned char dsm_raw[];
    unsigned char *sm = align1024(dsm_raw);
    // mbarriers: TMA stages; per MMA group its completion (committed by the MMA warp) and,
    // for the groups whose operands the compute warps write, "operands ready" (full_*,
    // arrived by thread 0 after the compute warps' barrier).  Each completes once per chunk.
    __shared__ uint64_t bar_tma[2], bar_x, bar_uw, bar_d, bar_q, bar_s;
    __shared__ uint64_t full_x, full_uw, full_d, full_s, bar_z;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s, factored_s[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;        // the TMEM lane this thread reads and writes
    // this CTA's chain, token-chunk range, initial/final state and duties
    int bh = blockIdx.x, c_begin = 0, c_end = a.NC;
    const float *init_ptr = a.init_state ? a.init_state + (size_t)blockIdx.x * 16384 : nullptr;
    float *fin_ptr = a.final_state ? a.final_state + (size_t)blockIdx.x * 16384 : nullptr;
    bool init_identity = false, zero_u = false, outputs = !CKPT;
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
            if (blockIdx.x & 1) {   // transition: S_0 = I, no value term (no checkpoints)
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
    const int n_it = c_end - c_begin;            // this CTA's chunks, indexed 0 .. n_it - 1
    constexpr int kTmaThread = 224;              // lane 0 of warp 7 issues the TMA loads
    constexpr int kGateWarp = 6;                 // warp 6 scans the gates (idle after its output)
    // gate vectors of two chunks (chunk `it` in set it % 2): g_r, exp(g_r), exp(g_63 - g_r),
    // beta_r, and the factors exp(g_r - g_31), exp(g_31 - g_r)
    float *sVec = reinterpret_cast<float *>(sm + SM_SMALL);   // [2][6][64]
    auto vec = [&](int it, int k) { return sVec + (it & 1) * 384 + 64 * k; };
    float *sM = sVec + 768;    // 1024 floats of solve scratch
    // raw gate words of two chunks: [slot][beta word | log alpha][64 tokens]
    uint32_t *sGate = reinterpret_cast<uint32_t *>(sVec + 1792);
    constexpr int kOutBoxes = sizeof(Tout) == 2 ? 2 : 4;   // 128-byte rows per output box
    const bool l2 = FUSED && (a.fuse & kFuseL2) != 0;
    const bool zgate = FUSED && (a.fuse & kFuseGate) != 0 && outputs;
    // norm vectors of chunk `it` (set it % 2)
    auto nvec = [&](int it, int k) { return reinterpret_cast<float *>(sm + SM_NRM) + (it & 1) * 448 + 64 * k; };

    if (tid == 0) {
        uint64_t *bars[] = {&bar_tma[0], &bar_tma[1], &bar_x, &bar_uw, &bar_d, &bar_q, &bar_s,
                            &full_x, &full_uw, &full_d, &full_s, &bar_z};
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
    const uint32_t tm = tmb + ((uint32_t)(32 * quarter) << 16);   // + this warp's lanes
    // operand descriptors of the shared-memory base: K-major, and MN-major with the two
    // 64-wide atoms 8192 or 16384 bytes apart
    const uint64_t dK0 = smem_desc_sw128(smem_u32(sm), 16, 1024);
    const uint64_t dM8 = smem_desc_sw128(smem_u32(sm), 8192, 1024), dM16 = smem_desc_sw128(smem_u32(sm), 16384, 1024);
    auto stage = [&](int it) { return sm + (it & 1) * kStageBytes; };
    auto fail = [&]() {
        abort_s = 1;
        atomicExch(a.status, kErrTimeout);
    };
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
        if (!wait_cycles(bar, parity)) fail();
        tc_fence_after();
    };

    auto issue_tma = [&](int it) {   // chunk `it`'s q, k, v tiles into stage it % 2
        const int s = it & 1;
        unsigned char *st = stage(it);
        mbar_arrive_expect_tx(&bar_tma[s], kStageBytes);
        const int t0 = (c_begin + it) * 64;
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(st + kb * 16384, &tq, &bar_tma[s], 64 * kb, h, t0, b);
            tma_load_4d(st + kb * 16384 + OFF_K0, &tk, &bar_tma[s], 64 * kb, h, t0, b);
            tma_load_4d(st + OFF_V0 + kb * 8192, &tv, &bar_tma[s], 64 * kb, h, t0, b);
            if (zgate) tma_prefetch_4d(&tz, 64 * kb, h, t0, b);
        }
    };
    auto prefetch_tiles = [&](int it) {   // chunk `it`'s q, k, v tiles into L2
        const int t0 = (c_begin + it) * 64;
        for (int kb = 0; kb < 2; ++kb) {
            tma_prefetch_4d(&tq, 64 * kb, h, t0, b);
            tma_prefetch_4d(&tk, 64 * kb, h, t0, b);
            tma_prefetch_4d(&tv, 64 * kb, h, t0, b);
        }
    };
    // Without the output gate the stage of chunk c is free once (Q S)^T(c) has read it (step 4)
    // and takes chunk c + 2 then (X(c + 2) may then be issued once P(c + 1) has read TM_X);
    // with the gate the stage is released after the output (step 6).
    const bool early = !zgate;
    // (MMA warp) chunk `it`'s output gate input into its stage's Q tiles (dead once (Q S)^T
    // has read them)
    auto issue_z = [&](int it) {
        mbar_arrive_expect_tx(&bar_z, 16384);
        const int t0 = (c_begin + it) * 64;
        for (int kb = 0; kb < 2; ++kb)
            tma_load_4d(stage(it) + kb * 16384, &tz, &bar_z, 64 * kb, h, t0, b);
    };
    // Output box kb (8 KB: 64 tokens x 64 bf16 or 32 fp32 channels) of chunk `it`.  Without the
    // output gate: Kt^T rows of [P; Kt^T] (free once the state update has read them), so that
    // the stage is released after (Q S)^T and takes the chunk after next early -- for bf16 the
    // rows of key channels 64..127 (two 8 KB runs), which the next chunk's Kt^T build
    // rewrites only in its step 3, for fp32 all four.  With the gate, whose z holds the
    // stage's Q tiles: the V slot (bf16) or the K tiles and the V slot (fp32) of the stage,
    // which then takes the chunk after next once the output has left.
    auto obox = [&](int it, int kb) -> unsigned char * {
        if (!zgate && sizeof(Tout) == 2) return sm + SM_BU + 16384u + kb * BU_KB;
        if (!zgate) return sm + SM_BU + (kb >> 1) * BU_KB + 8192u * (1 + (kb & 1));
        if (sizeof(Tout) == 2) return stage(it) + OFF_V0 + 8192u * kb;
        return stage(it) + (kb < 2 ? OFF_K0 + 16384u * kb : OFF_V0 + 8192u * (kb - 2));
    };
    // beta (the aligned 32-bit word holding it) and log alpha of chunk `it`, two tokens per
    // lane of the gate warp, copied asynchronously two chunks ahead; one commit group per
    // chunk (empty past the end), so that waiting for all but the newest group finds the
    // chunk about to be scanned complete
    const size_t ntok = (size_t)(gridDim.x / (a.role == 0 ? 1 : (a.role == 1 ? 2 * a.nseg : a.nseg))) * a.T;
    auto issue_gate = [&](int it) {
        if (it < n_it) {
            uint32_t *dst = sGate + (it & 1) * 128;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 2 * lane + e, t = (c_begin + it) * 64 + r;
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
        }
        cp_async_commit();
    };
    // (gate warp) chunk `it`'s cumulative log decay and factors into set it % 2; its raw
    // gate slot then takes chunk it + 2
    auto scan_gates = [&](int it) {
        cp_async_wait_group1();
        __syncwarp();
        const uint32_t *gw = sGate + (it & 1) * 128;
        const int t0 = (c_begin + it) * 64;
        float l[2], bt[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * lane + e, t = t0 + r;
            const size_t tok = t < a.T ? ((size_t)b * a.T + t) * a.H + h : 0;
            const uint32_t wd = gw[r];
            const uint16_t hb = (uint16_t)(((2 * tok) & 2) ? (wd >> 16) : (wd & 0xffffu));
            bt[e] = __bfloat162float(__ushort_as_bfloat16(hb));
            if (FUSED && (a.fuse & kFuseSigmoid)) bt[e] = t < a.T ? round_bf16(sigmoid_f(bt[e])) : 0.f;
            l[e] = __uint_as_float(gw[64 + r]);
        }
        __syncwarp();
        issue_gate(it + 2);
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
        float *sG = vec(it, 0), *sGam = vec(it, 1), *sDel = vec(it, 2), *sBeta = vec(it, 3),
              *sE = vec(it, 4), *sF = vec(it, 5);
        sG[r] = g0; sG[r + 1] = g1;
        sBeta[r] = bt[0]; sBeta[r + 1] = bt[1];
        sGam[r] = __expf(g0); sGam[r + 1] = __expf(g1);
        sDel[r] = __expf(glast - g0); sDel[r + 1] = __expf(glast - g1);
        const bool fac = gfirst - glast < kFactorSpan;
        if (fac) {
            sE[r] = __expf(g0 - gmid); sE[r + 1] = __expf(g1 - gmid);
            sF[r] = __expf(gmid - g0); sF[r + 1] = __expf(gmid - g1);
        }
        if (lane == 0) factored_s[it & 1] = fac;
    };
    // (fused L2 norm) 1 / sqrt(|x|^2 + eps) of row r of chunk `it`'s Q (rows_k false) or K
    // tile, after waiting for the tiles: the row's 128 values are 128 bytes of each K-block
    // tile (a quarter-warp's 16-byte loads of consecutive rows hit eight bank groups)
    auto inv_norm = [&](int it, bool rows_k, int r) {
        wait_bar(&bar_tma[it & 1], (it >> 1) & 1);
        const unsigned char *src = stage(it) + (rows_k ? OFF_K0 : 0) + r * 128;
        float ss = 0.f;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll 4
            for (int j = 0; j < 8; ++j) {
                const uint4 u = *reinterpret_cast<const uint4 *>(src + kb * 16384 + 16 * (j ^ (r & 7)));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
                    ss = fmaf(f.x, f.x, ss);
                    ss = fmaf(f.y, f.y, ss);
                }
            }
        return rsqrtf(ss + kL2NormEps);
    };
    // (the four warps that build no A rows: quarters 0 and 1) chunk `it`'s norm vectors, one
    // row of Q or K per thread
    auto norm_vecs = [&](int it) {
        const int i = 64 * half + row;   // 0..127: Q rows, then K rows
        const int r = i & 63;
        const float inv = inv_norm(it, i >= 64, r);
        const float gr = vec(it, 1)[r];
        if (i < 64) {
            nvec(it, NV_NQ)[r] = inv;
            nvec(it, NV_GQ)[r] = gr * inv;
        } else {
            nvec(it, NV_NK)[r] = inv;
            nvec(it, NV_BK)[r] = vec(it, 3)[r] * inv;
            nvec(it, NV_GK)[r] = gr * inv;
            nvec(it, NV_RK)[r] = 1.f / inv;
            nvec(it, NV_DK)[r] = vec(it, 2)[r] * inv;
        }
    };
    // (MMA warp) wait for chunk `it`'s tiles, then X = [Q; K] K^T into TM_X
    auto issue_x = [&](int it) {
        if (!wait_cycles(&bar_tma[it & 1], (it >> 1) & 1)) fail();
        unsigned char *st = stage(it);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
            mma_bf16(tmb + TM_X, desc_add(dK0, (uint32_t)((st + o) - sm)),
                     desc_add(dK0, (uint32_t)((st + OFF_K0 + o) - sm)), ID_KK_N64, ks > 0);
        }
        mma_commit(&bar_x);
    };
    // (compute warps) rows of X for chunk `it` (whose X is in TMEM, gate set it % 2): the
    // A rows (64..127, fp32, at SM_A; warps of lane quarters 2 and 3) or the P rows (0..63,
    // tf32, rows 0..63 of [P; Kt^T], K-block col_half; quarters 0 and 1)
    auto build_pa = [&](int it, bool rows_a, int col_half) {
        if ((quarter >= 2) != rows_a) return;
        const int r = quarter < 2 ? row : row - 64;
        float nk2 = 1.f;   // A rows of B (fused norm): nk_r^2, summed before X is held
        if (l2 && rows_a) {
            const float nk = inv_norm(it, true, r);
            nk2 = nk * nk;
        }
        float x[32];
        tmem_ld32(tm + TM_X + 32 * col_half, x);
        tmem_wait_ld();
        const int c0 = 32 * col_half;
        const float *sG = vec(it, 0), *sBeta = vec(it, 3), *sE = vec(it, 4), *sF = vec(it, 5);
        if (l2 && !rows_a) {   // P_rs nq_r nk_s
            const float *nk = nvec(it, NV_NK);
            const float nq = nvec(it, NV_NQ)[r];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 n4 = *reinterpret_cast<const float4 *>(nk + c0 + 4 * q);
                x[4 * q] *= nq * n4.x; x[4 * q + 1] *= nq * n4.y;
                x[4 * q + 2] *= nq * n4.z; x[4 * q + 3] *= nq * n4.w;
            }
        }

        float dec[32];   // exp(g_r - g_s), s = c0 + u
        if (factored_s[it & 1]) {
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
        if (!rows_a) {
            const uint32_t pb = smem_u32(sm + SM_BU + col_half * BU_KB);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                float pv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    pv[e] = c0 + 4 * q4 + e <= r ? round_tf32(dec[4 * q4 + e] * x[4 * q4 + e]) : 0.f;
                sts128f(pb + sw128_off32(r, 4 * q4), pv[0], pv[1], pv[2], pv[3]);
            }
        } else {
            const float br = sBeta[r] * nk2;   // B_rs = beta_r nk_r^2 ... with the fused norm
            float *sA = reinterpret_cast<float *>(sm + SM_A);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                float4 v4;
                const int s0 = c0 + 4 * q4;
                v4.x = s0 < r ? br * dec[4 * q4] * x[4 * q4] : 0.f;
                v4.y = s0 + 1 < r ? br * dec[4 * q4 + 1] * x[4 * q4 + 1] : 0.f;
                v4.z = s0 + 2 < r ? br * dec[4 * q4 + 2] * x[4 * q4 + 2] : 0.f;
                v4.w = s0 + 3 < r ? br * dec[4 * q4 + 3] * x[4 * q4 + 3] : 0.f;
                if ((s0 >> 4) != (r >> 4)) {   // off-diagonal blocks: read only as TF32 operands
                    v4.x = round_tf32(v4.x); v4.y = round_tf32(v4.y);
                    v4.z = round_tf32(v4.z); v4.w = round_tf32(v4.w);
                }
                *reinterpret_cast<float4 *>(sA + a_index(r, s0)) = v4;
            }
        }
    };
    // (compute warps) Kt^T of chunk `it` into rows 64..191 of [P; Kt^T]: Kt^T[i][r] =
    // delta_r k_r[i] (tf32; delta_r / |k_r| with the fused norm), key-channel blocks ib and
    // ib + nb - 1 (eight channels each; nb = 1 or 2): ldmatrix.trans of the k tile gives
    // each lane channel i and the tokens r, r + 1 of one 8 x 8 block.
    auto kt_build = [&](int it, int ib0, int nb) {
        wait_bar(&bar_tma[it & 1], (it >> 1) & 1);
        const uint32_t kbase = smem_u32(stage(it) + OFF_K0);
        const uint32_t bu = smem_u32(sm + SM_BU);
        const uint32_t sDel = smem_u32(l2 ? nvec(it, NV_DK) : vec(it, 2));
        uint32_t v[2][2][4];   // [block][token half][matrix]: all loads first
#pragma unroll
        for (int bq = 0; bq < 2; ++bq) {
            const int ib = ib0 + (bq < nb ? bq : 0), kb = ib >> 3, c8 = ib & 7;
#pragma unroll
            for (int rq = 0; rq < 2; ++rq) {
                const int rr = 8 * (4 * rq + (lane >> 3)) + (lane & 7);   // the token row this lane addresses
                ldsm_x4_trans(kbase + kb * 16384 + rr * 128 + ((c8 ^ (rr & 7)) << 4), v[bq][rq]);
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {   // this lane's token pair r, r + 1 of token block q
            const int r = 8 * q + 2 * (lane & 3);
            const float2 dq = lds64f(sDel + 4 * r);
#pragma unroll
            for (int bq = 0; bq < 2; ++bq) {
                if (bq >= nb) break;
                const int i = 8 * (ib0 + bq) + (lane >> 2);
                const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v[bq][q >> 2][q & 3]));
                sts64f(bu + (r >> 5) * BU_KB + sw128_off32(64 + i, r & 31), round_tf32(dq.x * kv.x),
                       round_tf32(dq.y * kv.y));
            }
        }
    };
    // (compute warps) T = (I + A)^-1 of chunk `it` (fp32, swizzled, over the S^T operand's
    // first half) with T diag(beta) and T diag(beta G) in bf16 at SM_TB; with the fused
    // norm, the operands of N^-1 (I + B)^-1 N
    const float *sA_c = reinterpret_cast<const float *>(sm + SM_A);
    auto solve_out = [&](int it) {
        return SolveOut<true, true, true>{reinterpret_cast<float *>(sm + SM_T), sm + SM_TB, vec(it, 3),
                                          vec(it, 1), nullptr};
    };
    auto solve_out_l2 = [&](int it) {
        return SolveOut<true, true, true, true>{reinterpret_cast<float *>(sm + SM_T), sm + SM_TB,
                                                nvec(it, NV_BK), nvec(it, NV_GK), nvec(it, NV_RK)};
    };
    auto solve_diag = [&](int it) {
        if (l2) solve_diag64(sA_c, solve_out_l2(it), tid);
        else solve_diag64(sA_c, solve_out(it), tid);
    };
    auto solve_merge = [&](int it) {   // warps 0..3
        if (l2) solve_merge64(sA_c, solve_out_l2(it), sM, tid, 2);
        else solve_merge64(sA_c, solve_out(it), sM, tid, 2);
    };
    auto solve = [&](int it) {   // all compute warps; starts after and ends with a barrier
        solve_diag(it);
        named_sync(1, kThreads);
        if (warp < 4) solve_merge(it);
        named_sync(1, kThreads);
    };

    // prologue loads: stages 0 and 1, raw gates of chunks 0 and 1
    if (tid == kTmaThread) {
        if (n_it > 0) issue_tma(0);
        if (n_it > 1) issue_tma(1);
    }
    if (warp == kGateWarp) {
        issue_gate(0);
        issue_gate(1);
    }

    // ---------------- MMA warp: issues every tcgen05.mma group, each once its operands are
    // ready, in the order the compute warps produce them, and commits it to the barrier
    // they wait on.  Chunk c's D and [O^T | S^T]; then chunk c + 2's X and chunk c + 1's U/W.
    if (warp == kMmaWarp) {
        if (lane == 0 && n_it > 0) {
            uint64_t *last = &bar_x;   // most recent commit (drained on abort)
            uint32_t last_par = 0;
            int z_last = -1;           // chunk of the most recent z copy
            auto issue_uw = [&](int it) {   // U^T = V^T (T diag beta)^T, W^T = K^T (T diag(beta G))^T
                unsigned char *st = stage(it);
                if (!zero_u)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmb + TM_U, desc_add(dM8, (uint32_t)((st + OFF_V0 + ks * 2048) - sm)),
                             desc_add(dK0, SM_TB + ks * 32), ID_MK_N64, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmb + TM_W, desc_add(dM16, (uint32_t)((st + OFF_K0 + ks * 2048) - sm)),
                             desc_add(dK0, SM_TB + 8192 + ks * 32), ID_MK_N64, ks > 0);
                mma_commit(&bar_uw);
            };
            issue_x(0);
            if (!wait_cycles(&full_uw, 0)) fail();
            tc_fence_after();
            issue_uw(0);
            last = &bar_uw;
            if (n_it > 1) {
                if (!wait_cycles(&full_x, 0)) fail();
                tc_fence_after();
                issue_x(1);
                last = &bar_x; last_par = 1;
            }
            for (int it = 0; it < n_it && !abort_s; ++it) {
                const uint32_t par = it & 1;
                unsigned char *st = stage(it);
                // D = S^T [W; Q]^T: (W S)^T first (W^T MN-major; the E^T build waits for it),
                // then (Q S)^T (Q straight from the stage)
                if (!wait_cycles(&full_d, par)) { fail(); break; }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ts(tmb + TM_WE, tmb + TM_SB + 8 * ks, desc_add(dM8, SM_W + ks * 2048), ID_KM_N64, ks > 0);
                mma_commit(&bar_d);
                if (outputs)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16_ts(tmb + TM_QO, tmb + TM_SB + 8 * ks, desc_add(dK0, (uint32_t)((st + o) - sm)),
                                    ID_KK_N64, ks > 0);
                    }
                mma_commit(&bar_q);
                last = &bar_q; last_par = par;
                if (zgate) {   // the Q tiles are dead once (Q S)^T has read them
                    if (!wait_cycles(&bar_q, par)) { fail(); break; }
                    issue_z(it);
                    z_last = it;
                }
                // [O^T | S^T] += E^T [P; Kt^T]^T  (tf32; E^T from tensor memory); without
                // outputs S^T += E^T Kt
                if (!wait_cycles(&full_s, par)) { fail(); break; }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_tf32_ts(tmb + (outputs ? TM_QO : TM_S), tmb + TM_WE + 8 * ks,
                                desc_add(dK0, SM_BU + (outputs ? 0u : 8192u) + (ks >> 2) * BU_KB + (ks & 3) * 32),
                                outputs ? ID_UPD : ID_UPD_S, true);
                mma_commit(&bar_s);
                last = &bar_s; last_par = par;
                // the next chunk's U/W (the next D waits for it), then the chunk after next's X
                bool ok = true;
                for (int g = 0; g < 2 && ok; ++g) {
                    if (g == 1) {
                        if (it + 2 < n_it) {
                            if (!wait_cycles(&full_x, (it + 1) & 1)) { fail(); ok = false; break; }
                            tc_fence_after();
                            issue_x(it + 2);
                            last = &bar_x; last_par = it & 1;
                        }
                    } else if (it + 1 < n_it) {
                        if (!wait_cycles(&full_uw, (it + 1) & 1)) { fail(); ok = false; break; }
                        tc_fence_after();
                        issue_uw(it + 1);
                        last = &bar_uw; last_par = (it + 1) & 1;
                    }
                }
                if (!ok) break;
            }
            if (abort_s) {   // drain this warp's MMAs and copies (bounded)
                wait_cycles(last, last_par);
                if (z_last >= 0) wait_cycles(&bar_z, (uint32_t)z_last & 1);
            }
        }
        __syncwarp();
    } else {
    // ---------------- compute warps
    // S^T[j][i] = S_0[i][j]: this thread owns j = row and i in [64 half, 64 half + 64).
    {
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
    if (n_it > 0) {
        // prologue: chunk 0's gates, A and P, solve; chunk 1's gates
        if (warp == kGateWarp) scan_gates(0);
        named_sync(1, kThreads);
        if (l2) {   // the P build reads every norm
            if (quarter < 2) norm_vecs(0);
            named_sync(1, kThreads);
        }
        wait_bar(&bar_x, 0);
        build_pa(0, true, half);
        if (outputs) build_pa(0, false, half);
        fence_proxy_async();
        tc_fence_before();
        named_sync(1, kThreads);
        if (tid == 0 && n_it > 1) mbar_arrive(&full_x);   // X(1) may overwrite TM_X
        solve(0);
        if (tid == 0) mbar_arrive(&full_uw);
        if (warp == kGateWarp && n_it > 1) scan_gates(1);
    }

    for (int it = 0; it < n_it; ++it) {
        const uint32_t par = it & 1;
        unsigned char *st = stage(it);
        const int t0 = (c_begin + it) * 64;
        const bool next = it + 1 < n_it;
        if (tid == kTmaThread && it + 2 < n_it) prefetch_tiles(it + 2);

        // ---- 1. S^T to bf16 pairs (TM_SB: 32-bit column c holds S^T columns 2c, 2c + 1) and
        //         S^T <- gamma S^T: after the previous state update (D(c - 1), which read
        //         TM_SB, completed before it)
        if (it >= 1) wait_bar(&bar_s, par ^ 1);
        {
            const float gamma = vec(it, 1)[63];
            float v[32];
            for (int part = 0; part < 2; ++part) {
                const int i0 = 64 * half + 32 * part;
                tmem_ld32(tm + TM_S + i0, v);
                tmem_wait_ld();
                if (CKPT && a.role != 1) {   // S[i][j] at this chunk's start
                    float *ck = a.ckpt + ((size_t)bh * a.NC + c_begin + it) * 16384 + (size_t)i0 * 128 + row;
#pragma unroll
                    for (int u = 0; u < 32; ++u) ck[(size_t)u * 128] = v[u];
                }
                {
                    uint32_t pk[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) pk[u] = pack_bf16(v[2 * u], v[2 * u + 1]);
                    tmem_st16u(tm + TM_SB + i0 / 2, pk);
                }
#pragma unroll
                for (int u = 0; u < 32; ++u) v[u] *= gamma;
                tmem_st32(tm + TM_S + i0, v);
            }
            tmem_wait_st();
        }
        // ---- 1b. this chunk's Kt^T, key channels 0..63 (the previous state update has read
        //          [P; Kt^T], and the output staged over its rows has left), while U/W(c) runs
        kt_build(it, warp, 1);
        // ---- 2. W^T (lane i = key channel, columns = tokens r) as the MN-major B operand of
        //         (W S)^T: this lane's row of 64 tokens, 16 bytes at a time
        wait_bar(&bar_uw, par);
        {
            float w[32];
            tmem_ld32(tm + TM_W + 32 * half, w);
            tmem_wait_ld();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float *f = w + 8 * q4;
                *reinterpret_cast<uint4 *>(sm + SM_W + sw128_off(row, 32 * half + 8 * q4)) =
                    make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                               pack_bf16(f[6], f[7]));
            }
        }
        fence_proxy_async();   // W and Kt^T for the tensor core
        // (bf16, no gate) the previous output's store has read its staging before step 3
        // rewrites those rows
        if (early && sizeof(Tout) == 2 && tid == kTmaThread) bulk_wait_read_all();
        tc_fence_before();
        named_sync(1, kThreads);
        if (abort_s) break;
        if (tid == 0) mbar_arrive(&full_d);   // D = S^T [W; Q]^T (MMA warp)

        // ---- 3. Kt^T, key channels 64..127 (lane quarters 0 and 1), while the other warps build
        //         the next chunk's A (its X arrived before D was issued); then the diagonal
        //         blocks of the next chunk's T (U/W(c) has read SM_TB), all while D runs
        if (quarter < 2) kt_build(it, 8 + 2 * ((warp & 1) + 2 * half), 2);
        if (next) {
            if (l2 && quarter < 2) norm_vecs(it + 1);   // read by the solve
            wait_bar(&bar_x, (it + 1) & 1);
            build_pa(it + 1, true, half);
            tc_fence_before();
            named_sync(1, kThreads);
            // without outputs X(c + 1) has no other reader: X(c + 2) may overwrite TM_X
            if (!outputs && tid == 0 && it + 2 < n_it) mbar_arrive(&full_x);
            solve_diag(it + 1);
        }

        // ---- 4. E^T = U^T - (W S)^T in place of (W S)^T (fp32, TF32-rounded: the A operand of
        //         the state update) and G (Q S)^T in place of (Q S)^T (the update accumulates
        //         the output onto it)
        wait_bar(&bar_d, par);
        {
            float ws[32], uu[32];
            tmem_ld32(tm + TM_WE + 32 * half, ws);
            if (!zero_u) tmem_ld32(tm + TM_U + 32 * half, uu);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) ws[u] = round_tf32((zero_u ? 0.f : uu[u]) - ws[u]);
            tmem_st32(tm + TM_WE + 32 * half, ws);
        }
        if (outputs) {
            wait_bar(&bar_q, par);
            const float *sGam = (l2 ? nvec(it, NV_GQ) : vec(it, 1)) + 32 * half;
            float qs[32];
            tmem_ld32(tm + TM_QO + 32 * half, qs);
            tmem_wait_ld();
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4) {
                const float4 g4 = *reinterpret_cast<const float4 *>(sGam + 4 * u4);
                qs[4 * u4] *= g4.x; qs[4 * u4 + 1] *= g4.y; qs[4 * u4 + 2] *= g4.z; qs[4 * u4 + 3] *= g4.w;
            }
            tmem_st32(tm + TM_QO + 32 * half, qs);
        }
        tmem_wait_st();
        fence_proxy_async();   // Kt^T (step 3) for the tensor core
        tc_fence_before();
        named_sync(1, kThreads);
        if (tid == 0) mbar_arrive(&full_s);   // [O^T | S^T] (MMA warp)
        // the stage's last readers, (Q S)^T and the Kt^T build, are done: it takes the chunk
        // after next
        if (early && tid == kTmaThread && it + 2 < n_it) issue_tma(it + 2);

        // ---- 5. the merges of the next chunk's T on warps 0..3, while warps 4..7 build the
        //         next chunk's P (the update has read [P; Kt^T]; then X(c + 2) may overwrite
        //         TM_X) and write this chunk's output O^T (staged as obox() places it)
        if (warp < 4) {
            if (next) solve_merge(it + 1);
        } else {
            wait_bar(&bar_s, par);
            if (outputs) {
                if (next && quarter < 2) {   // P rows: lanes 0..63 (warps 4 and 5), both column halves
                    // (one copy of the build for both column halves: the loop body's code
                    // size, not its instruction count, limits this kernel -- see below)
#pragma unroll 1
                    for (int ch = 0; ch < 2; ++ch) build_pa(it + 1, false, ch);
                    tc_fence_before();
                    named_sync(4, 64);
                    if (early && warp == 4 && lane == 0 && it + 2 < n_it) mbar_arrive(&full_x);
                }
                const int j = row;   // value channel; all 64 tokens of this lane
                if (zgate) wait_bar(&bar_z, it & 1);
                // The two 32-token halves share one copy of the code.  Nine warps run
                // different parts of a ~155 KB kernel at once, and instruction fetch is the
                // largest stall ("no instruction"): keeping this loop and the P build above
                // rolled (7 KB less code) cut the call by 6.5 %.
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float o[32];
                    tmem_ld32(tm + TM_QO + 32 * hh, o);
                    tmem_wait_ld();
                    if (zgate) {
                        const unsigned char *zt = st + (j >> 6) * 16384;
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            o[u] *= silu_tanh(__bfloat162float(
                                *reinterpret_cast<const __nv_bfloat16 *>(zt + sw128_off(32 * hh + u, j & 63))));
                    }
                    if (sizeof(Tout) == 2) {
                        unsigned char *dst = obox(it, j >> 6);
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            *reinterpret_cast<__nv_bfloat16 *>(dst + sw128_off(32 * hh + u, j & 63)) =
                                __float2bfloat16_rn(o[u]);
                    } else {
                        unsigned char *dst = obox(it, j >> 5);
                        const int cj = j & 31;
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            const int r = 32 * hh + u;
                            *reinterpret_cast<float *>(dst + r * 128 + ((((cj >> 2) ^ (r & 7)) & 7) << 4) +
                                                       ((cj & 3) << 2)) = o[u];
                        }
                    }
                }
                fence_proxy_async();
                // the gates of the chunk after next (into this chunk's set, which no later step
                // of this chunk reads), while warps 4 and 5 are still busy with P
                if (warp == kGateWarp && it + 2 < n_it) scan_gates(it + 2);
                named_sync(3, 128);
                if (tid == kTmaThread) {
                    constexpr int cols = sizeof(Tout) == 2 ? 64 : 32;
#pragma unroll
                    for (int kb = 0; kb < kOutBoxes; ++kb)
                        tma_store_4d(&to, obox(it, kb), cols * kb, h, t0, b);
                    bulk_commit();
                    if (early && sizeof(Tout) == 4) bulk_wait_read_all();   // step 1b rewrites the staging
                }
            }
            if (!outputs && warp == kGateWarp && it + 2 < n_it) scan_gates(it + 2);
        }
        tc_fence_before();
        named_sync(1, kThreads);

        // ---- 6. hand-offs: the next chunk's U/W (MMA warp); with the output gate, the chunk
        //         after next's X and that chunk's tiles into this chunk's stage
        if (tid == 0 && next) mbar_arrive(&full_uw);
        if (!early && tid == 0 && it + 2 < n_it) mbar_arrive(&full_x);
        if (!early && tid == kTmaThread && it + 2 < n_it) {
            bulk_wait_read_all();   // the output has left the stage
            issue_tma(it + 2);
        }
    }

    if (!abort_s && n_it > 0) {
        wait_bar(&bar_s, (n_it - 1) & 1);
        if (fin_ptr) {
            float v[32];
            for (int part = 0; part < 2; ++part) {
                const int i0 = 64 * half + 32 * part;
                tmem_ld32(tm + TM_S + i0, v);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 32; ++u) fin_ptr[(size_t)(i0 + u) * 128 + row] = v[u];
            }
        }
    } else if (abort_s && tid == kTmaThread) {
        // the stage loads this thread issued may still be in flight (bounded waits)
        for (int i = 0; i < min(n_it, 2); ++i) wait_cycles(&bar_tma[i], 0);
    }
    if (warp == kGateWarp) cp_async_wait_all();
    if (tid == kTmaThread) bulk_wait_all();   // the output stores' global writes
    }   // compute warps
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmb, 512);
}

// Segment chaining (between the two segment passes): per chain, S_start(0) = S_0 and
// S_start(p + 1) = Phi_p S_start(p) + S0_p, where Phi_p and S0_p are segment p's transition
// and zero-start end state.  One CTA per (chain, block of 16 state columns), fp32: each
// Phi_p is staged in shared memory (64 KB, coalesced; the next one is prefetched into L2
// meanwhile) before its product, each thread taking 8 rows of one column.
constexpr int kCombineSmem = 128 * 128 * 4;
constexpr int kCombineCols = 16;
__global__ void __launch_bounds__(256) seg_combine_kernel(const float *__restrict__ init_state,
                                                           const float *__restrict__ phi,
                                                           const float *__restrict__ s0,
                                                           float *__restrict__ start, int nseg) {
    __shared__ float S[128][kCombineCols + 1];
    extern __shared__ float4 phi_s4[];
    const float *phi_s = reinterpret_cast<const float *>(phi_s4);   // [128][128]
    constexpr int kBlocks = 128 / kCombineCols;
    const int cb = blockIdx.x % kBlocks, bh = blockIdx.x / kBlocks;
    const int tid = threadIdx.x, j = tid % kCombineCols, rg = tid / kCombineCols;   // rg 0..15
    const int col = kCombineCols * cb + j;
    for (int i = rg; i < 128; i += 16)
        S[i][j] = init_state ? init_state[((size_t)bh * 128 + i) * 128 + col] : 0.f;
    for (int p = 0; p < nseg; ++p) {
        const size_t slot = ((size_t)bh * nseg + p) * 16384;
        __syncthreads();   // S is complete; the previous Phi's readers are done
        for (int i = rg; i < 128; i += 16) start[slot + i * 128 + col] = S[i][j];
        if (p + 1 == nseg) break;
        if (tid == 0 && p + 2 < nseg) umma::bulk_prefetch_l2(phi + slot + 16384, 65536);
        for (int idx = tid; idx < 4096; idx += 256)
            phi_s4[idx] = reinterpret_cast<const float4 *>(phi + slot)[idx];
        float acc[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) acc[m] = s0[slot + (size_t)(rg + 16 * m) * 128 + col];
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < 128; ++k) {
            const float sk = S[k][j];
#pragma unroll
            for (int m = 0; m < 8; ++m) acc[m] = fmaf(phi_s[(rg + 16 * m) * 128 + k], sk, acc[m]);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 8; ++m) S[rg + 16 * m][j] = acc[m];
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

template <typename Tout, int GATE, int MODE>
int launch_f(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
             const CUtensorMap &mo, const CUtensorMap &mz, const TcArgs &ta, unsigned grid,
             cudaStream_t stream) {
    const int smem = (int)(MODE == 1 ? SM_TOTAL_FUSED : SM_TOTAL) + 1024;
    if (cudaFuncSetAttribute(chunk_tc_kernel<Tout, GATE, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return kErrCuda;
    chunk_tc_kernel<Tout, GATE, MODE><<<grid, kCtaThreads, smem, stream>>>(mq, mk, mv, mo, mz, ta);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

template <typename Tout, int GATE>
int launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
             const CUtensorMap &mo, const CUtensorMap &mz, const TcArgs &ta, unsigned grid,
             cudaStream_t stream) {
    if (ta.ckpt) return launch_f<Tout, GATE, 2>(mq, mk, mv, mo, mz, ta, grid, stream);
    return ta.fuse ? launch_f<Tout, GATE, 1>(mq, mk, mv, mo, mz, ta, grid, stream)
                   : launch_f<Tout, GATE, 0>(mq, mk, mv, mo, mz, ta, grid, stream);
}

}  // namespace

bool tc_make_map(CUtensorMap *m, const void *base, int64_t B, int64_t T, int64_t H, bool fp32) {
    return make_map(m, base, B, T, H, fp32);
}

int tc_launch_seg_combine(const float *init_state, const float *phi, const float *s0, float *start,
                          unsigned chains, int nseg, cudaStream_t stream) {
    if (cudaFuncSetAttribute(seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCombineSmem) !=
        cudaSuccess)
        return kErrCuda;
    seg_combine_kernel<<<chains * (128 / kCombineCols), 256, kCombineSmem, stream>>>(init_state, phi, s0, start, nseg);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

bool chunk_tc_supported(const ChunkProblem &p) {
    return p.in_bf16 && p.dk == 128 && p.dv == 128 && p.C == 64 && p.T > 0 &&
           (p.gate == 0 || p.gate == 1);
}

void tc_segment_split(const ChunkProblem &p, int *nseg, int *seg_len) {
    *nseg = 1;
    *seg_len = p.NC;
    if (chunk_tc_supported(p)) chain_segments(p.B * p.H, p.NC, nseg, seg_len);
}

size_t gdn_split_workspace_bytes(const ChunkProblem &p);
bool gdn_split_fuse_supported(const ChunkProblem &p);
int launch_gdn_split(const ChunkProblem &p, void *workspace, int *status_word, cudaStream_t stream);

// Few long chains split into segments take the two-kernel path of gdn_chain.cu when the
// workspace holds every chunk's T operands: its chunk-parallel solve keeps all SMs busy and
// its chain kernel is lighter per chunk (measured on B1 H16 T65536: 1.43 ms against 1.73 ms).
// Many chains keep the single kernel below for the plain forward, which solves inside the
// chain (B8 H16 T4096: 0.373 ms against 0.398 ms) and needs only the segments' states.  The
// fused neighbours cost the two-kernel path little (its prep kernel applies the L2 norm and
// the sigmoid; the chain folds the norms into factors it applies anyway), so they take it
// whenever the workspace allows; otherwise the single kernel serves them, as it serves the
// backward's checkpoints.
static bool split_path(const ChunkProblem &p) {
    int nseg, len;
    tc_segment_split(p, &nseg, &len);
    return nseg > 1;
}

size_t chunk_tc_workspace_bytes(const ChunkProblem &p, bool least) {
    if (!least && split_path(p)) return gdn_split_workspace_bytes(p);
    int nseg, len;
    tc_segment_split(p, &nseg, &len);
    return nseg > 1 ? (size_t)3 * p.B * p.H * nseg * 16384 * sizeof(float) : 0;
}

size_t chunk_tc_fused_workspace_bytes(const ChunkProblem &p) {
    return gdn_split_fuse_supported(p) ? gdn_split_workspace_bytes(p) : chunk_tc_workspace_bytes(p, true);
}

int launch_chunk_tc(const ChunkProblem &p, void *workspace, size_t workspace_bytes, int *status_word,
                    cudaStream_t stream, float *ckpt) {
    if (!ckpt && (p.fuse ? gdn_split_fuse_supported(p) : split_path(p)) && workspace &&
        workspace_bytes >= gdn_split_workspace_bytes(p))
        return launch_gdn_split(p, workspace, status_word, stream);
    CUtensorMap mq, mk, mv, mo, mz;
    const bool zgate = (p.fuse & kFuseGate) != 0;
    if (!make_map(&mq, p.q, p.B, p.T, p.H, false) || !make_map(&mk, p.k, p.B, p.T, p.H, false) ||
        !make_map(&mv, p.v, p.B, p.T, p.H, false) ||
        !make_map(&mo, p.out ? p.out : p.q, p.B, p.T, p.H, p.out ? !p.out_bf16 : false) ||
        !make_map(&mz, zgate ? p.z : p.q, p.B, p.T, p.H, false))   // (unused unless gated)
        return kErrCuda;
    TcArgs ta{p.log_alpha, (const __nv_bfloat16 *)p.beta, p.init_state, p.final_state,
              status_word, (int)p.T, (int)p.H, p.NC, p.fuse, 0, 1, p.NC, nullptr, nullptr, nullptr, ckpt};
    auto launch = [&](const TcArgs &t, unsigned grid) {
        if (p.out_bf16)
            return p.gate == 1 ? launch_t<__nv_bfloat16, 1>(mq, mk, mv, mo, mz, t, grid, stream)
                               : launch_t<__nv_bfloat16, 0>(mq, mk, mv, mo, mz, t, grid, stream);
        return p.gate == 1 ? launch_t<float, 1>(mq, mk, mv, mo, mz, t, grid, stream)
                           : launch_t<float, 0>(mq, mk, mv, mo, mz, t, grid, stream);
    };
    const unsigned bh = (unsigned)(p.B * p.H);
    int nseg, seg_len;
    tc_segment_split(p, &nseg, &seg_len);
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
    rc = tc_launch_seg_combine(p.init_state, ta.ws_phi, ta.ws_s0, ta.ws_start, bh, nseg, stream);
    if (rc != kOk) return rc;
    ta.role = 2;
    return launch(ta, bh * nseg);
}

}  // namespace dr
