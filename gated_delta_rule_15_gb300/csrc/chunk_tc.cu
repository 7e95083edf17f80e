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
//   A   = stril(beta_r exp(g_r - g_s) K K^T),  T = (I + A)^-1   (fp32 forward substitution)
//   U^T = V^T (T diag beta)^T            (128 x 64)  = (T diag(beta) V)^T
//   W^T = K^T (T diag(beta G))^T         (128 x 64)  = (T diag(beta) (K*G))^T
//   D   = S^T [W; Q*G]^T                 (128 x 128) = [(W S)^T | (Q*G S)^T]
//   E^T = U^T - (W S)^T
//   S^T <- gamma S^T + (E^T diag(delta)) K                 (state carried to the next chunk)
//   O^T = (Q*G S)^T + E^T P^T                              (chunk output)
//
// Precision: P, E^T and E^T diag(delta) enter their products as a bf16 pair (high part and
// the bf16 rounding of the remainder), so those products carry ~2^-16 relative error
// instead of bf16's 2^-8; S^T, W, Q*G and the T factors enter as single bf16 operands.  A
// rounding model of this arithmetic against the fp64 oracle puts the output error at
// ~1e-2 x RMS (about 3e-2 without the pairs).
//
// One CTA per (b, h), 256 threads, the whole TMEM (512 columns): S^T [0,128), D [128,256),
// X [256,320), U^T [320,384), W^T [384,448).  q, k, v tiles (64 tokens x 128, bf16) arrive
// by TMA with 128-byte swizzle into a double-buffered stage; the next chunk's tiles load
// while the current chunk computes.  Operands written by the CUDA cores (P, T diag beta,
// W, Q*G, S^T, E^T) use the same swizzled K-major layout; V and K tiles also serve as
// MN-major operands directly.  One thread issues the MMAs; completion is tracked with
// tcgen05.commit on an mbarrier.  Every wait is bounded by a cycle budget: on expiry the
// kernel records DR_ERR_TIMEOUT in the status word, drains its own copies and MMAs (with
// the same bound), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "chunk_layout.h"
#include "common.cuh"
#include "umma.cuh"

namespace dr {
namespace {

using namespace umma;

constexpr int kThreads = 256;
constexpr uint32_t kStageBytes = 49152;
// stage layout: [Q kb0 | K kb0 | Q kb1 | K kb1 | V kb0 | V kb1], 8 KB each (64 x 64 bf16)
constexpr uint32_t OFF_K0 = 8192, OFF_V0 = 32768;
constexpr uint32_t SM_B2 = 2 * kStageBytes;   // [W; Q*G] 128 x 128 K-major, 2 K-blocks;
                                              // after its MMA: low parts of E^T, E^T diag(delta)
constexpr uint32_t SM_ST = SM_B2 + 32768;     // S^T 128 x 128 K-major; fp32 T during the solve
constexpr uint32_t SM_ET = SM_ST + 32768;     // E^T (high part) 128 x 64; fp32 A during the solve
constexpr uint32_t SM_ET2 = SM_ET + 16384;    // E^T diag(delta) (high); T diag beta (+G) before
constexpr uint32_t SM_P = SM_ET2 + 16384;     // P (high part) 64 x 64 K-major
constexpr uint32_t SM_PLO = SM_P + 8192;      // P (low part)
constexpr uint32_t SM_ETLO = SM_B2, SM_ET2LO = SM_B2 + 16384;
constexpr uint32_t SM_SMALL = SM_PLO + 8192;  // g, G, delta, beta: fp32 [64] each
constexpr uint32_t SM_TOTAL = SM_SMALL + 1024;
constexpr uint32_t TM_S = 0, TM_D = 128, TM_X = 256, TM_U = 320, TM_W = 384;
constexpr long long kWaitCycles = 2000000000LL;   // ~1 s at the loaded SM clock

constexpr uint32_t ID_KK_N64 = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_KK_N128 = idesc_bf16(128, 128, false, false);
constexpr uint32_t ID_MK_N64 = idesc_bf16(128, 64, true, false);
constexpr uint32_t ID_KM_N128 = idesc_bf16(128, 128, false, true);

struct TcArgs {
    const float *log_alpha;
    const __nv_bfloat16 *beta;
    const float *init_state;
    void *out;
    float *final_state;
    int *status;
    int T, H, NC;
};

__device__ __forceinline__ bool wait_cycles(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi); packs two such pairs.
__device__ __forceinline__ void pack_hi_lo(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat16 ha = __float2bfloat16_rn(a), hb = __float2bfloat16_rn(b);
    __nv_bfloat162 h2;
    h2.x = ha;
    h2.y = hb;
    hi = *reinterpret_cast<uint32_t *>(&h2);
    lo = pack_bf16(a - __bfloat162float(ha), b - __bfloat162float(hb));
}

__device__ __forceinline__ uint4 scale_bf16x8(uint4 raw, float s) {
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&w[i]));
        w[i] = pack_bf16(f.x * s, f.y * s);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename Tout, int GATE>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const TcArgs a) {
    extern __shared__ unsigned char dsm_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)dsm_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar_tma[2], bar_mma;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;        // the TMEM lane this thread reads and writes
    const int bh = blockIdx.x;
    const int h = bh % a.H, b = bh / a.H;
    float *sG = reinterpret_cast<float *>(sm + SM_SMALL);
    float *sGam = sG + 64, *sDel = sG + 128, *sBeta = sG + 192;

    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(&bar_mma, 1);
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

    // S^T[j][i] = S_0[i][j]: this thread owns j = row and i in [64 half, 64 half + 64).
    {
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                v[u] = a.init_state ? a.init_state[((size_t)bh * 128 + i0 + u) * 128 + row] : 0.f;
            tmem_st32(tm + TM_S + i0, v);
        }
        tmem_wait_st();
    }

    auto issue_tma = [&](int c, int s) {
        unsigned char *st = sm + s * kStageBytes;
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar_tma[s], kStageBytes);
        const int t0 = c * 64;
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(st + kb * 16384, &tq, &bar_tma[s], 64 * kb, h, t0, b);
            tma_load_4d(st + kb * 16384 + OFF_K0, &tk, &bar_tma[s], 64 * kb, h, t0, b);
            tma_load_4d(st + OFF_V0 + kb * 8192, &tv, &bar_tma[s], 64 * kb, h, t0, b);
        }
    };
    if (tid == 0) issue_tma(0, 0);

    uint32_t mma_phase = 0;
    int last_c = -1;                       // chunk whose prefetch may still be in flight
    bool mma_outstanding = false;
    auto fail = [&]() {
        abort_s = 1;
        atomicExch(a.status, kErrTimeout);
    };
    auto wait_mma = [&]() {
        const bool ok = wait_cycles(&bar_mma, mma_phase);
        mma_phase ^= 1;
        if (ok) mma_outstanding = false; else fail();
        tc_fence_after();
    };

    for (int c = 0; c < a.NC; ++c) {
        const int s = c & 1;
        unsigned char *st = sm + s * kStageBytes;
        const int t0 = c * 64;
        const int Lc = min(64, a.T - t0);
        last_c = c;

        // ---- next chunk's tiles; beta and the cumulative log decay of this chunk
        if (tid == 0 && c + 1 < a.NC) issue_tma(c + 1, s ^ 1);
        if (tid < 64) {
            const bool valid = tid < Lc;
            const size_t tok = ((size_t)b * a.T + t0 + tid) * a.H + h;
            float g = (GATE == 1 && valid) ? a.log_alpha[tok] : 0.f;
            sBeta[tid] = valid ? __bfloat162float(a.beta[tok]) : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, g, o);
                if (lane >= o) g += y;
            }
            sG[tid] = g;
        }
        __syncthreads();
        if (tid >= 32 && tid < 64) sG[tid] += sG[31];
        __syncthreads();
        if (tid < 64) {
            const float g = sG[tid];
            sGam[tid] = __expf(g);
            sDel[tid] = __expf(sG[63] - g);
        }
        const float gamma = __expf(sG[63]);
        if (!wait_cycles(&bar_tma[s], (c >> 1) & 1)) fail();
        __syncthreads();
        if (abort_s) break;

        // ---- X = [Q; K] K^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_bf16(tmem_base_s + TM_X, smem_desc_sw128(smem_u32(st + o), 16, 1024),
                         smem_desc_sw128(smem_u32(st + OFF_K0 + o), 16, 1024), ID_KK_N64, ks > 0);
            }
            mma_commit(&bar_mma);
        }
        mma_outstanding = true;
        // Q*G into rows 64..127 of [W; Q*G] (same swizzle phase: (64 + r) % 8 == r % 8)
        for (int task = tid; task < 1024; task += kThreads) {
            const int r = task >> 4, kb = (task >> 3) & 1, ch = task & 7;
            const uint32_t off = kb * 16384 + r * 128 + (ch << 4);
            const uint4 raw = *reinterpret_cast<const uint4 *>(st + off);
            *reinterpret_cast<uint4 *>(sm + SM_B2 + 64 * 128 + off) = scale_bf16x8(raw, sGam[r]);
        }
        wait_mma();

        // ---- P (bf16, rows 0..63 of X) and A (fp32, rows 64..127 of X)
        {
            float x[32];
            tmem_ld32(tm + TM_X + 32 * half, x);
            tmem_wait_ld();
            const int c0 = 32 * half;
            if (quarter < 2) {
                const int r = row;
                const float gr = sG[r];
                uint32_t pk[16], pl[16];
#pragma unroll
                for (int u = 0; u < 32; u += 2) {
                    const int s0 = c0 + u;
                    const float p0 = s0 <= r ? __expf(gr - sG[s0]) * x[u] : 0.f;
                    const float p1 = s0 + 1 <= r ? __expf(gr - sG[s0 + 1]) * x[u + 1] : 0.f;
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
                const int r = row - 64;
                const float gr = sG[r], br = sBeta[r];
                float *sA = reinterpret_cast<float *>(sm + SM_ET);
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int s2 = c0 + u;
                    sA[r * 64 + (s2 ^ (r & 31))] = s2 < r ? br * __expf(gr - sG[s2]) * x[u] : 0.f;
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---- T = (I + A)^-1: column j by the 4 lanes tid/4 == j,
        //      T_rj = delta_rj - sum_{j <= s < r} A_rs T_sj  (fp32, stride 65)
        {
            const float *sA = reinterpret_cast<const float *>(sm + SM_ET);
            float *sT = reinterpret_cast<float *>(sm + SM_ST);
            const int j = tid >> 2, part = tid & 3;
            for (int r = part; r < 64; r += 4) sT[r * 65 + j] = (r == j) ? 1.f : 0.f;
            __syncwarp();
            for (int r = 1; r < 64; ++r) {
                float acc = 0.f;
                if (j < r)
                    for (int s2 = j + part; s2 < r; s2 += 4)
                        acc += sA[r * 64 + (s2 ^ (r & 31))] * sT[s2 * 65 + j];
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                if (part == 0 && j < r) sT[r * 65 + j] = -acc;
                __syncwarp();
            }
        }
        __syncthreads();

        // ---- T diag(beta) and T diag(beta G) as bf16 K-major operands (64 x 64)
        {
            const float *sT = reinterpret_cast<const float *>(sm + SM_ST);
            for (int task = tid; task < 512; task += kThreads) {
                const int r = task >> 3, ch = task & 7;
                uint32_t p1[4], p2[4];
#pragma unroll
                for (int u = 0; u < 8; u += 2) {
                    const int s0 = 8 * ch + u;
                    const float t0v = sT[r * 65 + s0] * sBeta[s0];
                    const float t1v = sT[r * 65 + s0 + 1] * sBeta[s0 + 1];
                    p1[u >> 1] = pack_bf16(t0v, t1v);
                    p2[u >> 1] = pack_bf16(t0v * sGam[s0], t1v * sGam[s0 + 1]);
                }
                const uint32_t off = sw128_off(r, 8 * ch);
                *reinterpret_cast<uint4 *>(sm + SM_ET2 + off) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
                *reinterpret_cast<uint4 *>(sm + SM_ET2 + 8192 + off) =
                    make_uint4(p2[0], p2[1], p2[2], p2[3]);
            }
        }
        fence_proxy_async();
        __syncthreads();

        // ---- U^T = V^T (T diag beta)^T,  W^T = K^T (T diag(beta G))^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem_base_s + TM_U, smem_desc_sw128(smem_u32(st + OFF_V0 + ks * 2048), 8192, 1024),
                         smem_desc_sw128(smem_u32(sm + SM_ET2 + ks * 32), 16, 1024), ID_MK_N64, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem_base_s + TM_W, smem_desc_sw128(smem_u32(st + OFF_K0 + ks * 2048), 16384, 1024),
                         smem_desc_sw128(smem_u32(sm + SM_ET2 + 8192 + ks * 32), 16, 1024), ID_MK_N64, ks > 0);
            mma_commit(&bar_mma);
        }
        mma_outstanding = true;
        wait_mma();
        // W (rows 0..63 of [W; Q*G]) from W^T: lane i = key channel, columns = tokens r
        {
            float w[32];
            tmem_ld32(tm + TM_W + 32 * half, w);
            tmem_wait_ld();
            const int i = row, kb = i >> 6, ci = i & 63;
            unsigned char *dst = sm + SM_B2 + kb * 16384;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                *reinterpret_cast<__nv_bfloat16 *>(dst + sw128_off(32 * half + u, ci)) =
                    __float2bfloat16_rn(w[u]);
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (abort_s) break;

        // ---- S^T to bf16 (MMA operand); S^T <- gamma S^T in TMEM
        {
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
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---- D = S^T [W; Q*G]^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_bf16(tmem_base_s + TM_D, smem_desc_sw128(smem_u32(sm + SM_ST + o), 16, 1024),
                         smem_desc_sw128(smem_u32(sm + SM_B2 + o), 16, 1024), ID_KK_N128, ks > 0);
            }
            mma_commit(&bar_mma);
        }
        mma_outstanding = true;
        wait_mma();

        // ---- E^T = U^T - (W S)^T, and E^T diag(delta)
        {
            float ws[32], uu[32];
            tmem_ld32(tm + TM_D + 32 * half, ws);
            tmem_ld32(tm + TM_U + 32 * half, uu);
            tmem_wait_ld();
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
                *reinterpret_cast<uint4 *>(sm + SM_ET2LO + off) =
                    make_uint4(dlo[0], dlo[1], dlo[2], dlo[3]);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---- S^T += (E^T diag delta) K ;  O^T = (Q*G S)^T + E^T P^T  (high/low pairs)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t e2[2] = {SM_ET2, SM_ET2LO};
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem_base_s + TM_S, smem_desc_sw128(smem_u32(sm + e2[part] + ks * 32), 16, 1024),
                             smem_desc_sw128(smem_u32(st + OFF_K0 + ks * 2048), 16384, 1024), ID_KM_N128, 1);
            const uint32_t ea[3] = {SM_ET, SM_ET, SM_ETLO}, pb[3] = {SM_P, SM_PLO, SM_P};
#pragma unroll
            for (int part = 0; part < 3; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem_base_s + TM_D + 64, smem_desc_sw128(smem_u32(sm + ea[part] + ks * 32), 16, 1024),
                             smem_desc_sw128(smem_u32(sm + pb[part] + ks * 32), 16, 1024), ID_KK_N64, 1);
            mma_commit(&bar_mma);
        }
        mma_outstanding = true;
        wait_mma();

        // ---- outputs: lane j = value channel, columns = tokens
        {
            float o[32];
            tmem_ld32(tm + TM_D + 64 + 32 * half, o);
            tmem_wait_ld();
            Tout *out = reinterpret_cast<Tout *>(a.out);
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int r = 32 * half + u;
                if (r < Lc) out[(((size_t)b * a.T + t0 + r) * a.H + h) * 128 + row] = from_f32<Tout>(o[u]);
            }
        }
        tc_fence_before();
        __syncthreads();
        if (abort_s) break;
    }

    if (abort_s) {
        // Drain this CTA's own asynchronous work (bounded) before TMEM is freed.
        if (tid == 0) {
            if (last_c >= 0 && last_c + 1 < a.NC)
                wait_cycles(&bar_tma[(last_c + 1) & 1], ((last_c + 1) >> 1) & 1);
            if (mma_outstanding) wait_cycles(&bar_mma, mma_phase);
        }
    } else if (a.final_state) {
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
            tmem_ld32(tm + TM_S + i0, v);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) a.final_state[((size_t)bh * 128 + i0 + u) * 128 + row] = v[u];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base_s, 512);
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

// [B, T, H, 128] bf16 viewed as 4-D (128, H, T, B); box 64 x 1 x 64 x 1, 128-byte swizzle,
// rows past T read as zeros.
bool make_map(CUtensorMap *m, const void *base, int64_t B, int64_t T, int64_t H) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {256, (cuuint64_t)H * 256, (cuuint64_t)(T * H) * 256};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tout, int GATE>
int launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const TcArgs &ta,
             unsigned grid, cudaStream_t stream) {
    const int smem = (int)SM_TOTAL + 1024;
    if (cudaFuncSetAttribute(chunk_tc_kernel<Tout, GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return kErrCuda;
    chunk_tc_kernel<Tout, GATE><<<grid, kThreads, smem, stream>>>(mq, mk, mv, ta);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

bool chunk_tc_supported(const ChunkProblem &p) {
    return p.in_bf16 && p.dk == 128 && p.dv == 128 && p.C == 64 && p.T > 0 &&
           (p.gate == 0 || p.gate == 1);
}

int launch_chunk_tc(const ChunkProblem &p, int *status_word, cudaStream_t stream) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, p.q, p.B, p.T, p.H) || !make_map(&mk, p.k, p.B, p.T, p.H) ||
        !make_map(&mv, p.v, p.B, p.T, p.H))
        return kErrCuda;
    TcArgs ta{p.log_alpha, (const __nv_bfloat16 *)p.beta, p.init_state, p.out, p.final_state,
              status_word, (int)p.T, (int)p.H, p.NC};
    const unsigned grid = (unsigned)(p.B * p.H);
    if (p.out_bf16)
        return p.gate == 1 ? launch_t<__nv_bfloat16, 1>(mq, mk, mv, ta, grid, stream)
                           : launch_t<__nv_bfloat16, 0>(mq, mk, mv, ta, grid, stream);
    return p.gate == 1 ? launch_t<float, 1>(mq, mk, mv, ta, grid, stream)
                       : launch_t<float, 0>(mq, mk, mv, ta, grid, stream);
}

}  // namespace dr
