// dr_api.cu -- the C ABI of libdr.so (declared in include/dr.h): argument validation,
// workspace sizing and dispatch to the kernels.  Nothing here allocates device memory or
// synchronises, except dr_get_device_status.
#include "../../include/dr.h"
#include "chunk_layout.h"
#include "common.cuh"
#include "umma.cuh"

namespace dr {

// Sticky device status word written by kernels whose waits are bounded.
__device__ int g_device_status = 0;

namespace {

// Device address of g_device_status on the current device (looked up once per device).
int *device_status_ptr() {
    static int *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        addr[dev] = (int *)p;
    }
    return addr[dev];
}

// dr_selftest_bounded_wait's kernel: one thread waits, with the chunk kernels' bounded loop
// (try_wait until a clock64 budget is spent), on an mbarrier that nothing completes; on
// expiry it records DR_ERR_TIMEOUT in the status word, as an expired wait in a chunk
// kernel does, and returns.
__global__ void bounded_wait_kernel(long long budget, int *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    umma::mbar_init(&bar, 1);
    umma::fence_mbar_init();
    const long long t0 = clock64();
    bool done = false;
    while (!(done = umma::mbar_try_wait(&bar, 0)))
        if (clock64() - t0 > budget) break;
    if (!done) atomicExch(status, kErrTimeout);
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool dim_ok(int64_t d) { return d == 64 || d == 128; }
bool dtype_ok(int32_t t) { return t == DR_F32 || t == DR_BF16; }

// Common checks of a chunk descriptor; fills the problem's sizes.
int check_chunk_desc(const dr_chunk_desc *d, ChunkProblem *p) {
    if (!d) return kErrInvalid;
    if (d->B < 1 || d->H < 1 || d->T < 0 || d->dk < 1 || d->dv < 1) return kErrInvalid;
    if (!dtype_ok(d->in_dtype) || !dtype_ok(d->out_dtype)) return kErrInvalid;
    if (d->gate < DR_GATE_NONE || d->gate > DR_GATE_CHANNEL) return kErrInvalid;
    if (d->chunk != 0 && d->chunk != 16 && d->chunk != 32 && d->chunk != 64) {
        return d->chunk < 0 ? kErrInvalid : kErrUnsupported;
    }
    if (!dim_ok(d->dk) || !dim_ok(d->dv)) return kErrUnsupported;
    // Grid sizes are 1-D 32-bit; B*H*ceil(T/16) must fit.
    if (d->B > (1 << 20) || d->H > (1 << 16) || d->T > ((int64_t)1 << 31)) return kErrUnsupported;
    const int C = d->chunk == 0 ? 64 : d->chunk;
    const int64_t NC = (d->T + C - 1) / C;
    if (d->B * d->H * NC > 0x7fffffffLL) return kErrUnsupported;
    p->B = d->B; p->T = d->T; p->H = d->H;
    p->dk = (int)d->dk; p->dv = (int)d->dv; p->C = C; p->NC = (int)NC; p->gate = d->gate;
    p->in_bf16 = d->in_dtype == DR_BF16;
    p->out_bf16 = d->out_dtype == DR_BF16;
    return kOk;
}

}  // namespace
}  // namespace dr

using namespace dr;

extern "C" int dr_version(void) { return (0 << 16) | 1; }

extern "C" int dr_chunk_fwd_workspace_bytes(const dr_chunk_desc *desc, size_t *bytes) {
    if (!bytes) return kErrInvalid;
    ChunkProblem p{};
    const int rc = check_chunk_desc(desc, &p);
    if (rc != kOk) return rc;
    if (chunk_tc_supported(p))
        *bytes = chunk_tc_workspace_bytes(p);
    else if (chunk_kda_supported(p))
        *bytes = chunk_kda_workspace_bytes(p);
    else
        *bytes = sizeof(float) * (simt_workspace_floats(p.B, p.H, p.NC, p.C, p.dk, p.dv) +
                                  simt_segment_floats(p));
    return kOk;
}

namespace dr {
int chunk_fwd_least_workspace(const dr_chunk_desc *desc, size_t *bytes) {
    if (!bytes) return kErrInvalid;
    ChunkProblem p{};
    const int rc = check_chunk_desc(desc, &p);
    if (rc != kOk) return rc;
    if (chunk_tc_supported(p)) {
        *bytes = chunk_tc_workspace_bytes(p, true);
        return kOk;
    }
    return dr_chunk_fwd_workspace_bytes(desc, bytes);
}
}  // namespace dr

extern "C" int dr_chunk_fwd_min_workspace_bytes(const dr_chunk_desc *desc, size_t *bytes) {
    return chunk_fwd_least_workspace(desc, bytes);
}

extern "C" int dr_chunk_fwd_ex_workspace_bytes(const dr_chunk_desc *desc, uint32_t fuse, size_t *bytes) {
    if (!bytes || (fuse & ~DR_FUSE_ALL)) return kErrInvalid;
    ChunkProblem p{};
    const int rc = check_chunk_desc(desc, &p);
    if (rc != kOk) return rc;
    p.fuse = fuse;
    if (fuse && chunk_tc_supported(p)) {
        *bytes = chunk_tc_fused_workspace_bytes(p);
        return kOk;
    }
    return dr_chunk_fwd_workspace_bytes(desc, bytes);
}

// Whether byte ranges [a, a + na) and [b, b + nb) overlap.
static bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const char *a0 = (const char *)a, *b0 = (const char *)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

extern "C" int dr_chunk_fwd_ex(const dr_chunk_desc *desc, uint32_t fuse, const void *q,
                               const void *k, const void *v, const float *log_alpha,
                               const void *beta, const void *z, const float *init_state,
                               void *out, float *final_state, void *workspace,
                               size_t workspace_bytes, dr_stream_t stream) {
    ChunkProblem p{};
    int rc = check_chunk_desc(desc, &p);
    if (rc != kOk) return rc;
    if (fuse & ~DR_FUSE_ALL) return kErrInvalid;
    if (!(fuse & kFuseGate)) z = nullptr;
    if (p.T > 0 && (!q || !k || !v || !beta || !out)) return kErrInvalid;
    if (p.gate != DR_GATE_NONE && p.T > 0 && !log_alpha) return kErrInvalid;
    if ((fuse & kFuseGate) && p.T > 0 && !z) return kErrInvalid;
    const void *ptrs[] = {q, k, v, log_alpha, beta, z, init_state, out, final_state, workspace};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return kErrInvalid;
    if (final_state && init_state && final_state != init_state) {
        const size_t sb = sizeof(float) * (size_t)(p.B * p.H * p.dk * p.dv);
        if (overlaps(init_state, sb, final_state, sb)) return kErrInvalid;   // partial overlap
    }
    if (z && p.T > 0) {
        const size_t n = (size_t)(p.B * p.T * p.H * p.dv);
        if (overlaps(z, n * (p.in_bf16 ? 2 : 4), out, n * (p.out_bf16 ? 2 : 4))) return kErrInvalid;
    }
    size_t need = 0;
    chunk_fwd_least_workspace(desc, &need);
    if (need > 0 && p.NC > 0 && (!workspace || workspace_bytes < need)) return kErrWorkspace;

    p.q = q; p.k = k; p.v = v; p.log_alpha = p.gate == DR_GATE_NONE ? nullptr : log_alpha;
    p.beta = beta; p.init_state = init_state; p.out = out; p.final_state = final_state;
    p.fuse = fuse; p.z = z;
    if (p.NC == 0 && !final_state) return kOk;
    if (chunk_tc_supported(p)) {
        int *status = device_status_ptr();
        if (!status) return kErrCuda;
        return launch_chunk_tc(p, workspace, workspace ? workspace_bytes : 0, status, (cudaStream_t)stream);
    }
    if (chunk_kda_supported(p)) {
        int *status = device_status_ptr();
        if (!status) return kErrCuda;
        return launch_chunk_kda(p, workspace, status, (cudaStream_t)stream);
    }
    const ChunkWorkspace ws = simt_workspace_carve(workspace, p.B, p.H, p.NC, p.C, p.dk, p.dv);
    float *seg = simt_segment_floats(p) > 0
                     ? (float *)workspace + simt_workspace_floats(p.B, p.H, p.NC, p.C, p.dk, p.dv)
                     : nullptr;
    return launch_chunk_simt(p, ws, (cudaStream_t)stream, nullptr, nullptr, false, seg);
}

extern "C" int dr_chunk_bwd_workspace_bytes(const dr_chunk_desc *desc, size_t *bytes) {
    if (!bytes) return kErrInvalid;
    ChunkProblem p{};
    const int rc = check_chunk_desc(desc, &p);
    if (rc != kOk) return rc;
    *bytes = bwd_workspace_bytes(p);
    return kOk;
}

extern "C" int dr_chunk_bwd(const dr_chunk_desc *desc, const void *q, const void *k,
                            const void *v, const float *log_alpha, const void *beta,
                            const float *init_state, const void *d_out,
                            const float *d_final_state, void *dq, void *dk, void *dv,
                            float *d_log_alpha, void *d_beta, float *d_init_state,
                            void *workspace, size_t workspace_bytes, dr_stream_t stream) {
    ChunkProblem p{};
    const int rc = check_chunk_desc(desc, &p);
    if (rc != kOk) return rc;
    if (p.T > 0 && (!q || !k || !v || !beta || !d_out || !dq || !dk || !dv || !d_beta))
        return kErrInvalid;
    if (p.gate != DR_GATE_NONE && p.T > 0 && (!log_alpha || !d_log_alpha)) return kErrInvalid;
    if (p.gate == DR_GATE_NONE && d_log_alpha) return kErrInvalid;
    const void *ptrs[] = {q, k, v, log_alpha, beta, init_state, d_out, d_final_state, dq, dk, dv,
                          d_log_alpha, d_beta, d_init_state, workspace};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return kErrInvalid;
    const size_t need = bwd_workspace_bytes(p);
    if (need > 0 && (!workspace || workspace_bytes < need)) return kErrWorkspace;
    if (p.NC == 0 && !d_init_state) return kOk;
    p.q = q; p.k = k; p.v = v; p.log_alpha = p.gate == DR_GATE_NONE ? nullptr : log_alpha;
    p.beta = beta; p.init_state = init_state; p.out = nullptr; p.final_state = nullptr;
    const BwdIo g{d_out, d_final_state, dq, dk, dv, d_log_alpha, d_beta, d_init_state};
    int *status = device_status_ptr();
    if (!status) return kErrCuda;
    return launch_chunk_bwd(p, g, workspace, status, (cudaStream_t)stream);
}

extern "C" int dr_chunk_fwd(const dr_chunk_desc *desc, const void *q, const void *k,
                            const void *v, const float *log_alpha, const void *beta,
                            const float *init_state, void *out, float *final_state,
                            void *workspace, size_t workspace_bytes, dr_stream_t stream) {
    return dr_chunk_fwd_ex(desc, 0u, q, k, v, log_alpha, beta, nullptr, init_state, out,
                           final_state, workspace, workspace_bytes, stream);
}

extern "C" int dr_recurrent_step_ex(const dr_step_desc *d, uint32_t fuse, const void *q,
                                    const void *k, const void *v, const float *log_alpha,
                                    const void *beta, const void *z, float *state, void *out,
                                    dr_stream_t stream) {
    if (!d) return kErrInvalid;
    if (d->B < 1 || d->H < 1 || d->dk < 1 || d->dv < 1 || d->reserved != 0) return kErrInvalid;
    if (!dtype_ok(d->in_dtype) || !dtype_ok(d->out_dtype)) return kErrInvalid;
    if (d->gate < DR_GATE_NONE || d->gate > DR_GATE_CHANNEL) return kErrInvalid;
    if (fuse & ~DR_FUSE_ALL) return kErrInvalid;
    if (!dim_ok(d->dk) || !dim_ok(d->dv)) return kErrUnsupported;
    if (d->B * d->H > 0x7fffffffLL) return kErrUnsupported;
    if (!(fuse & kFuseGate)) z = nullptr;
    if (!q || !k || !v || !beta || !state || !out) return kErrInvalid;
    if (d->gate != DR_GATE_NONE && !log_alpha) return kErrInvalid;
    if ((fuse & kFuseGate) && !z) return kErrInvalid;
    const void *ptrs[] = {q, k, v, log_alpha, beta, z, state, out};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return kErrInvalid;
    const size_t sb = sizeof(float) * (size_t)(d->B * d->H * d->dk * d->dv);
    const size_t ob = (size_t)(d->B * d->H * d->dv) * (d->out_dtype == DR_BF16 ? 2 : 4);
    if (overlaps(state, sb, out, ob)) return kErrInvalid;
    if (z) {
        const size_t zb = (size_t)(d->B * d->H * d->dv) * (d->in_dtype == DR_BF16 ? 2 : 4);
        if (overlaps(z, zb, state, sb) || overlaps(z, zb, out, ob)) return kErrInvalid;
    }
    return launch_decode(d->B * d->H, (int)d->dk, (int)d->dv, d->in_dtype == DR_BF16,
                         d->out_dtype == DR_BF16, d->gate, fuse, q, k, v,
                         d->gate == DR_GATE_NONE ? nullptr : log_alpha, beta, z, state, out,
                         (cudaStream_t)stream);
}

extern "C" int dr_recurrent_step(const dr_step_desc *d, const void *q, const void *k,
                                 const void *v, const float *log_alpha, const void *beta,
                                 float *state, void *out, dr_stream_t stream) {
    return dr_recurrent_step_ex(d, 0u, q, k, v, log_alpha, beta, nullptr, state, out, stream);
}

extern "C" int dr_selftest_bounded_wait(long long cycles, dr_stream_t stream) {
    if (cycles < 1 || cycles > 4000000000LL) return kErrInvalid;
    int *status = device_status_ptr();
    if (!status) return kErrCuda;
    bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(cycles, status);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

extern "C" int dr_get_device_status(dr_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return kErrCuda;
    int st = 0;
    if (cudaMemcpyFromSymbol(&st, g_device_status, sizeof(int)) != cudaSuccess) return kErrCuda;
    const int zero = 0;
    if (st != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess)
        return kErrCuda;
    return st;
}

extern "C" const char *dr_strerror(int status) {
    switch (status) {
        case DR_OK: return "ok";
        case DR_ERR_INVALID: return "invalid argument (null, size, alignment, overlap or enum)";
        case DR_ERR_UNSUPPORTED: return "unsupported configuration (dk, dv in {64,128}; chunk in {16,32,64})";
        case DR_ERR_CUDA: return "CUDA runtime or launch error";
        case DR_ERR_TIMEOUT: return "a bounded device-side wait expired";
        case DR_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}
