// decode.cu -- single-token recurrent decode step of the gated delta rule.
//
// Per chain (b, h), with the state S in R^{dk x dv} resident in HBM (fp32, row i = key
// channel):  S <- Diag(alpha) S;  p = S^T k;  S <- S + beta k (v - p)^T;  o = S^T q.
// (loop body of `gated_delta_rule`, page "linear-attention gated-deltanet guide",
// section 4; the per-step cost is independent of the sequence length, section 1 table.)
//
// The step is a pure stream of S through HBM: every element is read once and written
// once, so the kernel is bound by HBM bandwidth.  Column j of S only meets v_j, p_j and
// o_j, so one pass suffices: with S held in registers,
//     p_j = sum_i alpha_i k_i S_ij,   r_j = sum_i alpha_i q_i S_ij,
//     e_j = beta (v_j - p_j),         S'_ij = alpha_i S_ij + k_i e_j,
//     o_j = sum_i q_i S'_ij = r_j + (q . k) e_j.
//
// Mapping: one CTA per chain, dv/16 warps, warp w owns columns [16w, 16w + 16).  Lane
// (rr, cq) = (lane / 4, lane % 4) owns the float4 at columns 16w + 4cq of rows
// i = rr + 8m, m < dk/8.  A warp's load instruction touches 8 rows x 64 contiguous bytes
// (two full 32-byte sectors each); the column reductions are register sums over m
// followed by three xor-shuffles across rr.  No shared-memory reduction, one barrier.
//
// Fused neighbours (DR_FUSE_* of include/dr.h; the write gate, the SiLU output gate and
// L2-normalised q, k of the Gated DeltaNet layer, page "linear-attention gated-deltanet
// guide", section 4), all on values the kernel already holds: with the raw q, k and
// nq = 1 / |q|, nk = 1 / |k| (each warp reduces the two sums of squares itself),
// p_j = nk sum_i alpha_i k_i S_ij, r_j = nq sum_i alpha_i q_i S_ij, q.k scaled by nq nk,
// and the write k_i (nk e_j); beta = sigmoid(logit) stored in beta's dtype; out_j = o_j
// silu(z_j).
#include "chunk_layout.h"
#include "common.cuh"

namespace dr {

// FUSED: the fused neighbours' code is compiled in (each switched by `fuse_flags`); the
// plain instantiation carries none of it.
template <int DK, int DV, int GATE, bool FUSED, typename Tin, typename Tout>
__global__ void __launch_bounds__(DV * 2)
decode_step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                   const Tin *__restrict__ v, const float *__restrict__ log_alpha,
                   const Tin *__restrict__ beta, const Tin *__restrict__ z, uint32_t fuse_flags,
                   float *__restrict__ state, Tout *__restrict__ out) {
    const uint32_t fuse = FUSED ? fuse_flags : 0u;
    constexpr int NT = DV * 2;     // threads: DV/16 warps
    constexpr int RPL = DK / 8;    // rows per lane
    const int bh = blockIdx.x;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int cq = lane & 3, rr = lane >> 2;
    const int col = warp * 16 + cq * 4;

    // Issue the whole state tile's loads first: they are the only long-latency work.
    float *S = state + (size_t)bh * DK * DV;
    float4 s[RPL];
#pragma unroll
    for (int m = 0; m < RPL; ++m)
        s[m] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(rr + 8 * m) * DV + col));

    __shared__ float sk[DK], sq[DK], sa[DK];
    for (int i = tid; i < DK; i += NT) {
        sk[i] = to_f32(k[(size_t)bh * DK + i]);
        sq[i] = to_f32(q[(size_t)bh * DK + i]);
        float a = 1.f;
        if (GATE == 2) a = __expf(log_alpha[(size_t)bh * DK + i]);
        if (GATE == 1) a = __expf(log_alpha[bh]);
        sa[i] = a;
    }
    float bt = to_f32(beta[bh]);
    if (fuse & kFuseSigmoid) bt = to_f32(from_f32<Tin>(sigmoid_f(bt)));   // stored as beta
    const float4 vv = load4(v + (size_t)bh * DV + col);
    float4 zz = make_float4(0.f, 0.f, 0.f, 0.f);
    if ((fuse & kFuseGate) && rr == 0) zz = load4(z + (size_t)bh * DV + col);
    __syncthreads();
    // 1 / |k| and 1 / |q| (every warp reduces both sums of squares from shared memory)
    float nk = 1.f, nq = 1.f;
    if (fuse & kFuseL2) {
        float sk2 = 0.f, sq2 = 0.f;
#pragma unroll
        for (int i = lane; i < DK; i += 32) {
            sk2 = fmaf(sk[i], sk[i], sk2);
            sq2 = fmaf(sq[i], sq[i], sq2);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sk2 += __shfl_xor_sync(0xffffffffu, sk2, off);
            sq2 += __shfl_xor_sync(0xffffffffu, sq2, off);
        }
        nk = rsqrtf(sk2 + kL2NormEps);
        nq = rsqrtf(sq2 + kL2NormEps);
    }

    float4 p = make_float4(0.f, 0.f, 0.f, 0.f), r = p;
    float qk = 0.f;
#pragma unroll
    for (int m = 0; m < RPL; ++m) {
        const int i = rr + 8 * m;
        const float a = sa[i], ki = sk[i], qi = sq[i];
        const float ka = a * ki, qa = a * qi;
        p.x = fmaf(ka, s[m].x, p.x); p.y = fmaf(ka, s[m].y, p.y);
        p.z = fmaf(ka, s[m].z, p.z); p.w = fmaf(ka, s[m].w, p.w);
        r.x = fmaf(qa, s[m].x, r.x); r.y = fmaf(qa, s[m].y, r.y);
        r.z = fmaf(qa, s[m].z, r.z); r.w = fmaf(qa, s[m].w, r.w);
        qk = fmaf(qi, ki, qk);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        p.x += __shfl_xor_sync(0xffffffffu, p.x, off);
        p.y += __shfl_xor_sync(0xffffffffu, p.y, off);
        p.z += __shfl_xor_sync(0xffffffffu, p.z, off);
        p.w += __shfl_xor_sync(0xffffffffu, p.w, off);
        r.x += __shfl_xor_sync(0xffffffffu, r.x, off);
        r.y += __shfl_xor_sync(0xffffffffu, r.y, off);
        r.z += __shfl_xor_sync(0xffffffffu, r.z, off);
        r.w += __shfl_xor_sync(0xffffffffu, r.w, off);
        qk += __shfl_xor_sync(0xffffffffu, qk, off);
    }
    if (fuse & kFuseL2) {
        p.x *= nk; p.y *= nk; p.z *= nk; p.w *= nk;
        r.x *= nq; r.y *= nq; r.z *= nq; r.w *= nq;
        qk *= nq * nk;
    }
    const float4 e = make_float4(bt * (vv.x - p.x), bt * (vv.y - p.y),
                                 bt * (vv.z - p.z), bt * (vv.w - p.w));
    const float4 ek = make_float4(nk * e.x, nk * e.y, nk * e.z, nk * e.w);   // the write k e^T
#pragma unroll
    for (int m = 0; m < RPL; ++m) {
        const int i = rr + 8 * m;
        const float a = sa[i], ki = sk[i];
        float4 n;
        n.x = fmaf(a, s[m].x, ki * ek.x);
        n.y = fmaf(a, s[m].y, ki * ek.y);
        n.z = fmaf(a, s[m].z, ki * ek.z);
        n.w = fmaf(a, s[m].w, ki * ek.w);
        __stcs(reinterpret_cast<float4 *>(S + (size_t)i * DV + col), n);
    }
    if (rr == 0) {
        float4 o = make_float4(fmaf(qk, e.x, r.x), fmaf(qk, e.y, r.y),
                               fmaf(qk, e.z, r.z), fmaf(qk, e.w, r.w));
        if (fuse & kFuseGate) {
            o.x *= silu_f(zz.x); o.y *= silu_f(zz.y); o.z *= silu_f(zz.z); o.w *= silu_f(zz.w);
        }
        store4(out + (size_t)bh * DV + col, o);
    }
}

struct DecodeIo {
    const void *q, *k, *v;
    const float *la;
    const void *beta, *z;
    uint32_t fuse;
    float *state;
    void *out;
};

template <int DK, int DV, int GATE, typename Tin, typename Tout>
static int launch_decode_t(int64_t BH, const DecodeIo &io, cudaStream_t stream) {
    if (io.fuse)
        decode_step_kernel<DK, DV, GATE, true, Tin, Tout><<<(unsigned)BH, DV * 2, 0, stream>>>(
            (const Tin *)io.q, (const Tin *)io.k, (const Tin *)io.v, io.la, (const Tin *)io.beta,
            (const Tin *)io.z, io.fuse, io.state, (Tout *)io.out);
    else
        decode_step_kernel<DK, DV, GATE, false, Tin, Tout><<<(unsigned)BH, DV * 2, 0, stream>>>(
            (const Tin *)io.q, (const Tin *)io.k, (const Tin *)io.v, io.la, (const Tin *)io.beta,
            nullptr, 0u, io.state, (Tout *)io.out);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

template <int DK, int DV, typename Tin, typename Tout>
static int launch_decode_g(int gate, int64_t BH, const DecodeIo &io, cudaStream_t s) {
    switch (gate) {
        case 0: return launch_decode_t<DK, DV, 0, Tin, Tout>(BH, io, s);
        case 1: return launch_decode_t<DK, DV, 1, Tin, Tout>(BH, io, s);
        default: return launch_decode_t<DK, DV, 2, Tin, Tout>(BH, io, s);
    }
}

template <int DK, int DV>
static int launch_decode_d(int in_bf16, int out_bf16, int gate, int64_t BH, const DecodeIo &io,
                           cudaStream_t s) {
    using bf = __nv_bfloat16;
    if (in_bf16 && out_bf16) return launch_decode_g<DK, DV, bf, bf>(gate, BH, io, s);
    if (in_bf16) return launch_decode_g<DK, DV, bf, float>(gate, BH, io, s);
    if (out_bf16) return launch_decode_g<DK, DV, float, bf>(gate, BH, io, s);
    return launch_decode_g<DK, DV, float, float>(gate, BH, io, s);
}

// Host launcher: arguments already validated by the C-ABI layer.
int launch_decode(int64_t BH, int dk, int dv, int in_bf16, int out_bf16, int gate,
                  uint32_t fuse, const void *q, const void *k, const void *v, const float *la,
                  const void *beta, const void *z, float *state, void *out, cudaStream_t s) {
    const DecodeIo io{q, k, v, la, beta, z, fuse, state, out};
    if (dk == 128 && dv == 128) return launch_decode_d<128, 128>(in_bf16, out_bf16, gate, BH, io, s);
    if (dk == 128 && dv == 64) return launch_decode_d<128, 64>(in_bf16, out_bf16, gate, BH, io, s);
    if (dk == 64 && dv == 128) return launch_decode_d<64, 128>(in_bf16, out_bf16, gate, BH, io, s);
    if (dk == 64 && dv == 64) return launch_decode_d<64, 64>(in_bf16, out_bf16, gate, BH, io, s);
    return kErrUnsupported;
}

}  // namespace dr
