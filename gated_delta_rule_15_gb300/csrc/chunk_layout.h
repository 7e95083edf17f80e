// chunk_layout.h -- problem record and workspace layout of the chunkwise forward.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dr.h"

namespace dr {

// A validated chunk-forward problem (all pointers are device pointers).
struct ChunkProblem {
    const void *q, *k, *v;
    const float *log_alpha;
    const void *beta;
    const float *init_state;
    void *out;
    float *final_state;
    int64_t B, T, H;
    int dk, dv, C, NC, gate;
    bool in_bf16, out_bf16;
    // fused neighbours (DR_FUSE_* bits of include/dr.h) and the output gate's input
    // [B, T, H, dv] in the input dtype (NULL unless the output gate is fused)
    uint32_t fuse;
    const void *z;
};

// DR_FUSE_* bits (include/dr.h)
constexpr uint32_t kFuseL2 = 1, kFuseSigmoid = 2, kFuseGate = 4;

// fp32 intermediates of the two-kernel CUDA-core path, one slab per (b, h, chunk) n:
//   W  [n][C][dk]   T diag(beta) (K*G)
//   U  [n][C][dv]   T diag(beta) V
//   Qg [n][C][dk]   Q*G
//   Kd [n][C][dk]   K*G_C/G
//   P  [n][C][C]    lower-triangular intra-chunk read matrix
//   gam [n][dk]     G_C
struct ChunkWorkspace {
    float *W, *U, *Qg, *Kd, *P, *gam;
};

inline size_t simt_workspace_floats(int64_t B, int64_t H, int64_t NC, int64_t C, int64_t dk,
                                    int64_t dv) {
    const int64_t n = B * H * NC;
    return (size_t)(n * (C * dk * 3 + C * dv + C * C + dk));
}

// Carve the workspace; every slab starts on a 16-byte boundary because each slab size is
// a multiple of 4 floats (C, dk, dv are multiples of 16).
inline ChunkWorkspace simt_workspace_carve(void *base, int64_t B, int64_t H, int64_t NC,
                                           int64_t C, int64_t dk, int64_t dv) {
    const int64_t n = B * H * NC;
    float *p = (float *)base;
    ChunkWorkspace w;
    w.W = p;   p += n * C * dk;
    w.U = p;   p += n * C * dv;
    w.Qg = p;  p += n * C * dk;
    w.Kd = p;  p += n * C * dk;
    w.P = p;   p += n * C * C;
    w.gam = p;
    return w;
}

// CUDA-core path (chunk_simt.cu).  For the backward, `T_out` ([n][C][C]) and `ckpt`
// ([n][dk][dv], the state at each chunk's start) are also written; `p.out` may then be NULL.
// With `seg_ws` (simt_segment_floats(p) floats; NULL: whole chains) few long chains are split
// into segments (the split rule is simt_segments).
int launch_chunk_simt(const ChunkProblem &p, const ChunkWorkspace &ws, cudaStream_t stream,
                      float *T_out = nullptr, float *ckpt = nullptr, bool prep_only = false,
                      float *seg_ws = nullptr);
void simt_segments(int64_t chains, int dk, int dv, int NC, int *nseg, int *seg_len);
size_t simt_segment_floats(const ChunkProblem &p);
// Backward of the chunk forward on the CUDA cores (chunk_bwd.cu): gradients of
// <d_out, out> + <d_final, final_state>.  Workspace: bwd_workspace_bytes(p).
struct BwdIo {
    const void *d_out;          // [B,T,H,dv] out dtype
    const float *d_final;       // [B,H,dk,dv] or NULL (zero)
    void *dq, *dk, *dv;         // in dtype
    float *d_log_alpha;         // shape of log_alpha (NULL iff no gate)
    void *d_beta;               // [B,T,H] in dtype
    float *d_init;              // [B,H,dk,dv] or NULL (not returned)
};
size_t bwd_workspace_bytes(const ChunkProblem &p);
int launch_chunk_bwd(const ChunkProblem &p, const BwdIo &g, void *workspace, int *status_word,
                     cudaStream_t stream);

// Tensor-core path for bf16 inputs, dk = dv = 128, C = 64, scalar gate or none, T > 0
// (chunk_tc.cu, gdn_chain.cu).  With a workspace of chunk_tc_workspace_bytes(p) (every
// chunk's 16 KB T operands, plus the segments' states when few long chains are split) the
// plain forward runs as two kernels (chunk-parallel solve, then the chains); with at least
// chunk_tc_workspace_bytes(p, true) (the segments' states only) a single kernel solves inside
// each chain, which also serves the fused neighbours and the backward's checkpoints.
// `status_word` is the device status word of the library (bounded waits record
// DR_ERR_TIMEOUT there).
bool chunk_tc_supported(const ChunkProblem &p);
size_t chunk_tc_workspace_bytes(const ChunkProblem &p, bool least = false);
// The workspace of the fastest path for the fused neighbours p.fuse (the two-kernel path).
size_t chunk_tc_fused_workspace_bytes(const ChunkProblem &p);
// With `ckpt` ([B*H][NC][dk][dv] fp32), it writes the state at every chunk's start instead of
// the outputs (the backward's recompute).
int launch_chunk_tc(const ChunkProblem &p, void *workspace, size_t workspace_bytes, int *status_word,
                    cudaStream_t stream, float *ckpt = nullptr);
// Few long chains leave most of the GPU's 152 SMs idle while each chain walks its chunks one
// after another; the tensor-core paths then split every chain into `nseg` segments of
// `seg_len` chunks (at least 16 each) so that about 152 CTAs work at once.  A segment's end
// state is affine in its start state, S_end = Phi S_start + S0 (S0: the end state from a zero
// start; Phi: the run from the identity with no value term), so the segments run in three
// passes: end states of every segment in parallel, the chaining of the affine maps along each
// chain (tc_launch_seg_combine), then every segment again from its true start, writing outputs.
// nseg = 1 when the problem is not split.
inline void chain_segments(int64_t chains, int NC, int *nseg, int *seg_len) {
    constexpr int kGpuSms = 152;
    *nseg = 1;
    *seg_len = NC;
    if (chains > kGpuSms / 2 || NC < 32) return;
    const int n = (int)(NC / 16 < kGpuSms / chains ? NC / 16 : kGpuSms / chains);
    if (n < 2) return;
    const int len = (NC + n - 1) / n;
    *seg_len = len;
    *nseg = (NC + len - 1) / len;
}
// Per chain, S_start(0) = S_0 (NULL: zero) and S_start(p + 1) = Phi_p S_start(p) + S0_p over
// the [chains][nseg][128][128] fp32 arrays phi, s0 and start (chunk_tc.cu).
int tc_launch_seg_combine(const float *init_state, const float *phi, const float *s0, float *start,
                          unsigned chains, int nseg, cudaStream_t stream);
// The least workspace dr_chunk_fwd accepts for *desc (dr_api.cu).
int chunk_fwd_least_workspace(const dr_chunk_desc *desc, size_t *bytes);
// Two-kernel tensor-core path for the per-channel gate (chunk_kda.cu): bf16 inputs,
// dk = dv = 128, C = 64, T > 0.  Its workspace holds the per-chunk operands that the
// prep kernel writes and the state kernel reads (chunk_kda_workspace_bytes).
bool chunk_kda_supported(const ChunkProblem &p);
size_t chunk_kda_workspace_bytes(const ChunkProblem &p);
int launch_chunk_kda(const ChunkProblem &p, void *workspace, int *status_word, cudaStream_t stream);
int launch_decode(int64_t BH, int dk, int dv, int in_bf16, int out_bf16, int gate,
                  uint32_t fuse, const void *q, const void *k, const void *v, const float *la,
                  const void *beta, const void *z, float *state, void *out, cudaStream_t s);

}  // namespace dr
