// tc_common.cuh -- device helpers shared by the tensor-core chunk kernels: bounded mbarrier
// waits, bf16 packing (single and high/low pairs), warp-level TF32 16 x 16 products and the
// blocked 64 x 64 unit-lower-triangular inverse, and split-TF32 warp tiles of row products.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "umma.cuh"

namespace dr {
namespace tc {

using namespace umma;

constexpr long long kWaitCycles = 2000000000LL;   // ~1 s at the loaded SM clock

// Waits for the phase with the given parity; false once about kWaitCycles have passed
// without it.  (try_wait with a suspend-time hint was measured slower here: the waiting
// thread's wake-up lengthens every hand-off between warps.)
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
    hi = pack_bf16(a, b);
    lo = pack_bf16(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}

// x rounded to the nearest TF32 value (ties away from zero, as cvt.rna.tf32.f32), as its bit
// pattern with the low 13 mantissa bits clear: half a TF32 unit added to the magnitude bits,
// then the low bits cleared -- two integer operations on the full-rate ALU (infinities and
// NaNs stay what they are; values within half a unit of the largest float become infinite,
// as the conversion's rounding makes them).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
}
// d += a (16 x 8, row) * b (8 x 8, col), TF32 operands, fp32 accumulate (one warp).
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d += a (16 x 16, row) * b (16 x 8, col), bf16 operands, fp32 accumulate (one warp).
__device__ __forceinline__ void mma_bf16_16x8x16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// fp32 element as a TF32 operand: rounded here (kCvt), or already rounded when stored
template <bool kCvt>
__device__ __forceinline__ uint32_t tf32_op(float x) { return kCvt ? to_tf32(x) : __float_as_uint(x); }
// x rounded to TF32 (its low 13 mantissa bits cleared), as a float
__device__ __forceinline__ float round_tf32(float x) { return __uint_as_float(to_tf32(x)); }

// acc (16 x 16, mma.sync C fragment) += L (16 x 16 nk) * R (16 nk x 16); one warp.
// L(r, k) and R(k, n) return fp32 elements, rounded to TF32 here unless kCvt is false
// (then they must have been stored rounded).
template <bool kCvt = true, class FL, class FR>
__device__ __forceinline__ void warp_mm16(float (&acc)[2][4], FL L, FR R, int nk, int g, int t4) {
    for (int kt = 0; kt < 2 * nk; ++kt) {
        const int kc = 8 * kt;
        const uint32_t af[4] = {tf32_op<kCvt>(L(g, kc + t4)), tf32_op<kCvt>(L(g + 8, kc + t4)),
                                tf32_op<kCvt>(L(g, kc + t4 + 4)), tf32_op<kCvt>(L(g + 8, kc + t4 + 4))};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
            mma_tf32_16x8x8(acc[nt], af, tf32_op<kCvt>(R(kc + t4, 8 * nt + g)),
                            tf32_op<kCvt>(R(kc + t4 + 4, 8 * nt + g)));
    }
}
// acc (16 x 8) += L (16 x 16 nk) * R (16 nk x 8); one warp, one n-tile.
template <bool kCvt = true, class FL, class FR>
__device__ __forceinline__ void warp_mm16x8(float (&acc)[4], FL L, FR R, int nk, int g, int t4) {
    for (int kt = 0; kt < 2 * nk; ++kt) {
        const int kc = 8 * kt;
        const uint32_t af[4] = {tf32_op<kCvt>(L(g, kc + t4)), tf32_op<kCvt>(L(g + 8, kc + t4)),
                                tf32_op<kCvt>(L(g, kc + t4 + 4)), tf32_op<kCvt>(L(g + 8, kc + t4 + 4))};
        mma_tf32_16x8x8(acc, af, tf32_op<kCvt>(R(kc + t4, g)), tf32_op<kCvt>(R(kc + t4 + 4, g)));
    }
}
// Writes sign * acc through st(r, n, v0, v1): elements (r, n) and (r, n + 1), n even.
template <class FS>
__device__ __forceinline__ void warp_store16(const float (&acc)[2][4], float sign, FS st, int g, int t4) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n = 8 * nt + 2 * t4;
        st(g, n, sign * acc[nt][0], sign * acc[nt][1]);
        st(g + 8, n, sign * acc[nt][2], sign * acc[nt][3]);
    }
}

constexpr int kTs = 68;   // row stride (floats) of the padded fp32 T matrix: 16-byte aligned rows

// Element (r, s) of the fp32 T matrix: padded rows of kTs floats (kSwizzledT false), or dense
// rows of 64 with 16-byte groups XOR-swizzled by r % 16 (16 KB; pairs and quads stay whole).
template <bool kSwizzledT>
__device__ __forceinline__ int t_index(int r, int s) {
    return kSwizzledT ? r * 64 + (s ^ ((r & 15) << 2)) : r * kTs + s;
}

// Element (r, s) of the fp32 A matrix: rows of 64, 16-byte groups XOR-swizzled by r % 16.
__device__ __forceinline__ int a_index(int r, int s) {
    return r * 64 + ((((s >> 2) ^ (r & 15)) << 2) | (s & 3));
}

// T = (I + A)^-1 for a strictly lower-triangular 64 x 64 A (fp32), T stored as t_index says.
//   1. the four diagonal 16 x 16 blocks by right-looking substitution, four threads per
//      column (each owns four rows; the pivot row's value is broadcast by a shuffle);
//   2. T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32 T_22 (two warps);
//   3. lower-left 32 x 32 quarter: M = A[32:64, 0:32] T[0:32, 0:32], then
//      T[32:64, 0:32] = -T[32:64, 32:64] M (four warps, one 16 x 16 tile each).
// Each element is written, once final, also as T diag(beta) in bf16 (a 128-byte-swizzled
// K-major 64 x 64 tile at TB) and, with kPair, as T diag(beta G) at TB + 8192: the U and W
// operands.  With kRow the operands are diag(rowf) T diag(beta) and diag(rowf) T diag(beta G)
// (a similarity of T, the fp32 copy staying T).  Products use TF32 mma.sync with fp32 accumulation.  M needs 1024 floats.
// Step 1 is solve_diag64 (256 threads); steps 2 and 3 are solve_merge64 (warps 0..3 only,
// synchronising on their own named barrier), so that warps 4..7 are free meanwhile.
template <bool kPair, bool kSwizzledT, bool kPreRound = false, bool kRow = false>
struct SolveOut {
    float *T;
    unsigned char *TB;
    const float *beta, *gam;
    const float *rowf;   // kRow only
    // final element (r, s) of T: fp32 copy for the later levels, and the bf16 MMA operands
    __device__ __forceinline__ void fin(int r, int s, float v) const {
        T[t_index<kSwizzledT>(r, s)] = kPreRound ? round_tf32(v) : v;
        const float vb = kRow ? v * beta[s] * rowf[r] : v * beta[s];
        const uint32_t off = sw128_off(r, s);
        *reinterpret_cast<__nv_bfloat16 *>(TB + off) = __float2bfloat16_rn(vb);
        if constexpr (kPair)
            *reinterpret_cast<__nv_bfloat16 *>(TB + 8192 + off) = __float2bfloat16_rn(vb * gam[s]);
    }
    // final elements (r, s) and (r, s + 1), s even: one 32-bit store per operand
    __device__ __forceinline__ void fin2(int r, int s, float v0, float v1) const {
        *reinterpret_cast<float2 *>(T + t_index<kSwizzledT>(r, s)) =
            kPreRound ? make_float2(round_tf32(v0), round_tf32(v1)) : make_float2(v0, v1);
        float b0 = v0 * beta[s], b1 = v1 * beta[s + 1];
        if constexpr (kRow) {
            const float f = rowf[r];
            b0 *= f;
            b1 *= f;
        }
        const uint32_t off = sw128_off(r, s);
        *reinterpret_cast<uint32_t *>(TB + off) = pack_bf16(b0, b1);
        if constexpr (kPair)
            *reinterpret_cast<uint32_t *>(TB + 8192 + off) = pack_bf16(b0 * gam[s], b1 * gam[s + 1]);
    }
};

// Step 1 (256 threads, tid 0..255): the diagonal blocks and the zero blocks of the operands.
template <bool kPair, bool kSwizzledT, bool kPreRound, bool kRow>
__device__ __forceinline__ void solve_diag64(const float *A,
                                             const SolveOut<kPair, kSwizzledT, kPreRound, kRow> &out,
                                             int tid) {
    const int lane = tid & 31;
    const int o = 16 * (tid >> 6), c = (tid >> 2) & 15, part = tid & 3;
    const int owner = lane & ~3;
    // this thread's four rows of the diagonal block, o + part + 4m, columns o .. o + 15
    float ar[4][16];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int r = o + part + 4 * m;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v4 = *reinterpret_cast<const float4 *>(A + a_index(r, o + 4 * q));
            ar[m][4 * q] = v4.x; ar[m][4 * q + 1] = v4.y;
            ar[m][4 * q + 2] = v4.z; ar[m][4 * q + 3] = v4.w;
        }
    }
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
    for (int m = 0; m < 4; ++m) out.fin(o + part + 4 * m, o + c, y[m]);
    // the six blocks above the diagonal are zero in the bf16 operands (the fp32 copy of
    // those blocks is never read): (0,1) (0,2) (0,3) (1,2) (1,3) (2,3), 8 per task
    if (tid < 6 * 32) {
        const int blk = tid >> 5, e = tid & 31;
        const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        const uint32_t off = sw128_off(16 * bi + (e >> 1), 16 * bj + 8 * (e & 1));
        *reinterpret_cast<uint4 *>(out.TB + off) = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (kPair)
            *reinterpret_cast<uint4 *>(out.TB + 8192 + off) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();   // these operand entries are read by the tensor core later
}

// Steps 2 and 3 (warps 0..3, tid 0..127; starts after a barrier that follows step 1 and
// ends with the operands' proxy fence, without a final barrier).  With kPreRound, T, M and
// the off-diagonal blocks of A hold TF32-rounded values (the products take them as they are;
// the result is the same as rounding at each load), and level 2 runs on four warps, one
// 8-column half of a block each (the second product needs only its own half of the first).
template <bool kPair, bool kSwizzledT, bool kPreRound, bool kRow>
__device__ __forceinline__ void solve_merge64(const float *A,
                                              const SolveOut<kPair, kSwizzledT, kPreRound, kRow> &out,
                                              float *M, int tid, uint32_t bar_id) {
    constexpr bool kCvt = !kPreRound;
    const float *T = out.T;
    auto a = [&](int r, int s) { return A[a_index(r, s)]; };
    auto tt = [&](int r, int s) { return T[t_index<kSwizzledT>(r, s)]; };
    auto rnd = [&](float x) { return kPreRound ? round_tf32(x) : x; };
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    if constexpr (kPreRound) {
        // T_10 (warps 0, 1) and T_32 (warps 2, 3), columns 8 nh .. 8 nh + 7
        const int bp = warp >> 1, nh = warp & 1, i = 2 * bp + 1, j = 2 * bp;
        float *Ms = M + 256 * bp;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        warp_mm16x8<false>(acc, [&](int r, int k) { return a(16 * i + r, 16 * j + k); },
                           [&](int k, int n) { return tt(16 * j + k, 16 * j + 8 * nh + n); }, 1, g, t4);
        const int n0 = 8 * nh + 2 * t4;
        *reinterpret_cast<float2 *>(Ms + g * 16 + n0) = make_float2(rnd(acc[0]), rnd(acc[1]));
        *reinterpret_cast<float2 *>(Ms + (g + 8) * 16 + n0) = make_float2(rnd(acc[2]), rnd(acc[3]));
        __syncwarp();
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};
        warp_mm16x8<false>(acc2, [&](int r, int k) { return tt(16 * i + r, 16 * i + k); },
                           [&](int k, int n) { return Ms[k * 16 + 8 * nh + n]; }, 1, g, t4);
        out.fin2(16 * i + g, 16 * j + n0, -acc2[0], -acc2[1]);
        out.fin2(16 * i + g + 8, 16 * j + n0, -acc2[2], -acc2[3]);
    } else if (warp < 2) {
        const int i = 2 * warp + 1, j = 2 * warp;
        float *Ms = M + 256 * warp;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        warp_mm16<kCvt>(acc, [&](int r, int k) { return a(16 * i + r, 16 * j + k); },
                        [&](int k, int n) { return tt(16 * j + k, 16 * j + n); }, 1, g, t4);
        warp_store16(acc, 1.f, [&](int r, int n, float v0, float v1) {
            *reinterpret_cast<float2 *>(Ms + r * 16 + n) = make_float2(v0, v1); }, g, t4);
        __syncwarp();
        float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        warp_mm16<kCvt>(acc2, [&](int r, int k) { return tt(16 * i + r, 16 * i + k); },
                        [&](int k, int n) { return Ms[k * 16 + n]; }, 1, g, t4);
        warp_store16(acc2, -1.f, [&](int r, int n, float v0, float v1) {
            out.fin2(16 * i + r, 16 * j + n, v0, v1); }, g, t4);
    }
    named_sync(bar_id, 128);
    {   // M tile (rb, cb) = sum_{k = cb}^{1} A_{rb,k} T_{k,cb},  rb = 2 + w/2, cb = w%2
        const int rb = 2 + (warp >> 1), cb = warp & 1;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        warp_mm16<kCvt>(acc, [&](int r, int k) { return a(16 * rb + r, 16 * cb + k); },
                        [&](int k, int n) { return tt(16 * cb + k, 16 * cb + n); }, 2 - cb, g, t4);
        float *Mt = M + 256 * warp;
        warp_store16(acc, 1.f, [&](int r, int n, float v0, float v1) {
            *reinterpret_cast<float2 *>(Mt + r * 16 + n) = make_float2(rnd(v0), rnd(v1)); }, g, t4);
    }
    named_sync(bar_id, 128);
    {   // T_{rb,cb} = -sum_{k = 2}^{rb} T_{rb,k} M_{k,cb}
        const int rb = 2 + (warp >> 1), cb = warp & 1;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        warp_mm16<kCvt>(acc, [&](int r, int k) { return tt(16 * rb + r, 32 + k); },
                        [&](int k, int n) { return M[256 * (((k >> 4) << 1) | cb) + (k & 15) * 16 + n]; },
                        rb - 1, g, t4);
        warp_store16(acc, -1.f, [&](int r, int n, float v0, float v1) {
            out.fin2(16 * rb + r, 16 * cb + n, v0, v1); }, g, t4);
    }
    fence_proxy_async();   // the bf16 operands are read next by the tensor core
}

// The whole solve by 256 threads (the CTA's compute warps, which synchronise on named
// barriers 1 (all) and 2 (warps 0..3)); starts after and ends with a barrier.
template <bool kPair = true, bool kSwizzledT = false>
__device__ __forceinline__ void solve_unit_lower64(const float *A, float *T, float *M,
                                                   unsigned char *TB, const float *beta,
                                                   const float *gam, int tid) {
    const SolveOut<kPair, kSwizzledT> out{T, TB, beta, gam, nullptr};
    solve_diag64(A, out, tid);
    named_sync(1, 256);
    if (tid < 128) solve_merge64(A, out, M, tid, 2);
    named_sync(1, 256);
}

// out(r, n) = sum_{k < K} A[r][k] B[n][k] for r < R, n < N (R, N multiples of 16 and 8, K of
// 8): fp32 rows in shared memory, A row r at A + r lda, B row n at B + n ldb.  Each warp of
// the CTA takes 16 x 8 tiles (the mma.sync fragment shapes) in turn; a tile skipped by
// `skip(r0, n0)` is not computed.  kSplit: three TF32 products of split operands (x = hi + lo,
// hi and lo TF32: hi.hi + hi.lo + lo.hi) give about fp32 accuracy, the dropped lo.lo term
// being ~2^-22 of the product; otherwise one product of the TF32-rounded operands (~2^-11
// relative).  st(r, n, v) receives each element once.
template <bool kSplit, class FSkip, class FS>
__device__ __forceinline__ void rows_dot_rows(const float *A, int lda, const float *B, int ldb, int R, int N,
                                              int K, int warp, int nwarps, int lane, FSkip skip, FS st) {
    const int g = lane >> 2, t4 = lane & 3;
    const int nrb = R / 16, ntiles = nrb * (N / 8);
    for (int tile = warp; tile < ntiles; tile += nwarps) {
        const int r0 = 16 * (tile % nrb), n0 = 8 * (tile / nrb);
        if (skip(r0, n0)) continue;
        const float *a = A + (r0 + g) * lda + t4, *b = B + (n0 + g) * ldb + t4;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; k0 < K; k0 += 8) {
            const float av[4] = {a[k0], a[8 * lda + k0], a[k0 + 4], a[8 * lda + k0 + 4]};
            const float bv[2] = {b[k0], b[k0 + 4]};
            uint32_t ah[4], bh[2];
#pragma unroll
            for (int u = 0; u < 4; ++u) ah[u] = to_tf32(av[u]);
#pragma unroll
            for (int u = 0; u < 2; ++u) bh[u] = to_tf32(bv[u]);
            if constexpr (kSplit) {
                uint32_t al[4], bl[2];
#pragma unroll
                for (int u = 0; u < 4; ++u) al[u] = to_tf32(av[u] - __uint_as_float(ah[u]));
#pragma unroll
                for (int u = 0; u < 2; ++u) bl[u] = to_tf32(bv[u] - __uint_as_float(bh[u]));
                mma_tf32_16x8x8(acc, al, bh[0], bh[1]);
                mma_tf32_16x8x8(acc, ah, bl[0], bl[1]);
            }
            mma_tf32_16x8x8(acc, ah, bh[0], bh[1]);
        }
        st(r0 + g, n0 + 2 * t4, acc[0]);
        st(r0 + g, n0 + 2 * t4 + 1, acc[1]);
        st(r0 + g + 8, n0 + 2 * t4, acc[2]);
        st(r0 + g + 8, n0 + 2 * t4 + 1, acc[3]);
    }
}

// acc[t] (t < nt <= NT: the 16 x 8 C fragments at rows r0 .. r0 + 15, columns n0 + 8t ..)
// += sum_{k < K} A(r, k) B(k, n), K a multiple of 8; A(r, k) and B(k, n) return fp32
// elements.  The same TF32 products as rows_dot_rows (kSplit as there); one warp.
template <bool kSplit, int NT, class FA, class FB>
__device__ __forceinline__ void rows_times_cols(float (&acc)[NT][4], int nt, FA A, FB B, int r0, int n0, int K,
                                                int g, int t4) {
    for (int k0 = 0; k0 < K; k0 += 8) {
        const float av[4] = {A(r0 + g, k0 + t4), A(r0 + g + 8, k0 + t4), A(r0 + g, k0 + t4 + 4),
                             A(r0 + g + 8, k0 + t4 + 4)};
        uint32_t ah[4], al[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            ah[u] = to_tf32(av[u]);
            if constexpr (kSplit) al[u] = to_tf32(av[u] - __uint_as_float(ah[u]));
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t >= nt) break;
            const float bv[2] = {B(k0 + t4, n0 + 8 * t + g), B(k0 + t4 + 4, n0 + 8 * t + g)};
            uint32_t bh[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) bh[u] = to_tf32(bv[u]);
            if constexpr (kSplit) {
                uint32_t bl[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) bl[u] = to_tf32(bv[u] - __uint_as_float(bh[u]));
                mma_tf32_16x8x8(acc[t], al, bh[0], bh[1]);
                mma_tf32_16x8x8(acc[t], ah, bl[0], bl[1]);
            }
            mma_tf32_16x8x8(acc[t], ah, bh[0], bh[1]);
        }
    }
}

}  // namespace tc
}  // namespace dr
