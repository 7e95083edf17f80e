// host_api.cu -- dr_chunk_fwd_host: the chunk forward for callers holding HOST buffers.
//
// Copies the inputs host -> device, runs dr_chunk_fwd and copies out and final_state
// device -> host, all enqueued asynchronously behind `stream`.  The sequence is split into
// `pieces` time ranges (whole chunks): piece p's forward starts, from the state piece p - 1
// left (carried in place in one device state buffer), as soon as its inputs have arrived,
// while the inputs of piece p + 1 are still on their way in and the outputs of piece p - 1
// on their way out (the two copy directions use different copy engines and overlap on the
// link).  After the last input copy only the last piece's kernels and output copy remain.
// Each time range of a [B, T, H, w] tensor is B rows of contiguous bytes: one 2-D copy.
// Streams and events are created per call and released behind the work; the only device
// memory used is the caller's buffer `dev`.
#include <algorithm>

#include "../../include/dr.h"
#include "chunk_layout.h"
#include "common.cuh"

namespace dr {
namespace {

constexpr int kMaxPieces = 16;

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// Per piece, one 256-byte-aligned region per tensor: [q | k | v | beta | log alpha | out |
// ws]; then the state buffer [B, H, dk, dv] fp32 (initial state in, carried, final out).
struct HostLayout {
    int pieces;
    int64_t t[kMaxPieces + 1];   // token boundaries of the pieces (multiples of the chunk)
    size_t in_isz, out_isz, la_w;
    size_t base[kMaxPieces][7];  // byte offsets in `dev`, piece p, tensor i
    size_t ws_bytes[kMaxPieces];
    size_t state, total;
};
enum { HQ, HK, HV, HB, HLA, HOUT, HWS };

bool host_layout(const dr_chunk_desc *d, int pieces, HostLayout *L) {
    if (!d || pieces < 1) return false;
    const int64_t C = d->chunk == 0 ? 64 : d->chunk;
    const int64_t nch = (d->T + C - 1) / C;
    const int P = (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(pieces, kMaxPieces), nch));
    L->pieces = P;
    for (int p = 0; p <= P; ++p) L->t[p] = std::min<int64_t>(d->T, (nch * p / P) * C);
    L->t[P] = d->T;
    L->in_isz = d->in_dtype == DR_BF16 ? 2 : 4;
    L->out_isz = d->out_dtype == DR_BF16 ? 2 : 4;
    L->la_w = d->gate == DR_GATE_NONE ? 0 : (d->gate == DR_GATE_CHANNEL ? (size_t)d->dk : 1);
    const size_t bh = (size_t)(d->B * d->H);
    size_t off = 0;
    for (int p = 0; p < P; ++p) {
        const size_t tp = (size_t)(L->t[p + 1] - L->t[p]);
        dr_chunk_desc dp = *d;
        dp.T = (int64_t)tp;
        size_t w = 0;
        if (dr_chunk_fwd_workspace_bytes(&dp, &w) != DR_OK) return false;
        const size_t sizes[7] = {bh * tp * d->dk * L->in_isz, bh * tp * d->dk * L->in_isz,
                                 bh * tp * d->dv * L->in_isz, bh * tp * L->in_isz, bh * tp * 4 * L->la_w,
                                 bh * tp * d->dv * L->out_isz, w};
        for (int i = 0; i < 7; ++i) {
            L->base[p][i] = off;
            off += align256(sizes[i]);
        }
        L->ws_bytes[p] = w;
    }
    L->state = off;
    off += align256(bh * (size_t)(d->dk * d->dv) * 4);
    L->total = off;
    return true;
}

}  // namespace
}  // namespace dr

using namespace dr;

extern "C" int dr_chunk_fwd_host_dev_bytes(const dr_chunk_desc *desc, int pieces, size_t *bytes) {
    if (!bytes || !desc) return kErrInvalid;
    size_t w = 0;
    const int rc = dr_chunk_fwd_workspace_bytes(desc, &w);   // validates the descriptor
    if (rc != kOk) return rc;
    HostLayout L;
    if (!host_layout(desc, pieces, &L)) return kErrInvalid;
    *bytes = L.total;
    return kOk;
}

extern "C" int dr_chunk_fwd_host(const dr_chunk_desc *desc, int pieces, const void *q, const void *k,
                                 const void *v, const float *log_alpha, const void *beta,
                                 const float *init_state, void *out, float *final_state, void *dev,
                                 size_t dev_bytes, dr_stream_t stream) {
    size_t w = 0;
    int rc = dr_chunk_fwd_workspace_bytes(desc, &w);
    if (rc != kOk) return rc;
    if (desc->T > 0 && (!q || !k || !v || !beta || !out)) return kErrInvalid;
    if (desc->gate != DR_GATE_NONE && desc->T > 0 && !log_alpha) return kErrInvalid;
    HostLayout L;
    if (!host_layout(desc, pieces, &L)) return kErrInvalid;
    if (!dev || dev_bytes < L.total || ((uintptr_t)dev & 255u) != 0) return kErrWorkspace;

    cudaStream_t main = (cudaStream_t)stream;
    cudaStream_t s_in = nullptr, s_out = nullptr, s_comp = nullptr;
    cudaEvent_t e_start = nullptr, e_in[kMaxPieces] = {}, e_comp[kMaxPieces] = {}, e_done = nullptr;
    auto cleanup = [&]() {   // released once the enqueued work has finished
        for (int p = 0; p < kMaxPieces; ++p) {
            if (e_in[p]) cudaEventDestroy(e_in[p]);
            if (e_comp[p]) cudaEventDestroy(e_comp[p]);
        }
        if (s_in) cudaStreamDestroy(s_in);
        if (s_out) cudaStreamDestroy(s_out);
        if (s_comp) cudaStreamDestroy(s_comp);
        if (e_start) cudaEventDestroy(e_start);
        if (e_done) cudaEventDestroy(e_done);
    };
    const int P = L.pieces;
    bool ok = cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&s_comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&e_start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&e_done, cudaEventDisableTiming) == cudaSuccess;
    for (int p = 0; ok && p < P; ++p)
        ok = cudaEventCreateWithFlags(&e_in[p], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&e_comp[p], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cleanup();
        return kErrCuda;
    }

    char *d = (char *)dev;
    const int64_t B = desc->B, T = desc->T, H = desc->H;
    const size_t st_bytes = (size_t)(B * H * desc->dk * desc->dv) * 4;
    // tokens [t0, t1) of a [B, T, H, w] host tensor (w elements of `isz` bytes per (b, t, h))
    // <-> the piece's contiguous [B, t1 - t0, H, w] region at `off` of `dev`
    auto h2d = [&](size_t off, const void *src, size_t w_bytes, int64_t t0, int64_t t1) {
        const size_t row = (size_t)((t1 - t0) * H) * w_bytes;
        if (row == 0 || !src) return cudaSuccess;
        return cudaMemcpy2DAsync(d + off, row, (const char *)src + (size_t)(t0 * H) * w_bytes,
                                 (size_t)(T * H) * w_bytes, row, (size_t)B, cudaMemcpyHostToDevice, s_in);
    };
    auto d2h = [&](void *dst, size_t off, size_t w_bytes, int64_t t0, int64_t t1) {
        const size_t row = (size_t)((t1 - t0) * H) * w_bytes;
        if (row == 0 || !dst) return cudaSuccess;
        return cudaMemcpy2DAsync((char *)dst + (size_t)(t0 * H) * w_bytes, (size_t)(T * H) * w_bytes, d + off,
                                 row, row, (size_t)B, cudaMemcpyDeviceToHost, s_out);
    };
    ok = cudaEventRecord(e_start, main) == cudaSuccess && cudaStreamWaitEvent(s_in, e_start, 0) == cudaSuccess &&
         cudaStreamWaitEvent(s_out, e_start, 0) == cudaSuccess;
    if (ok && init_state)
        ok = cudaMemcpyAsync(d + L.state, init_state, st_bytes, cudaMemcpyHostToDevice, s_in) == cudaSuccess;
    float *state = (float *)(d + L.state);
    for (int p = 0; ok && p < P; ++p) {
        const int64_t t0 = L.t[p], t1 = L.t[p + 1];
        const size_t *O = L.base[p];
        ok = h2d(O[HQ], q, desc->dk * L.in_isz, t0, t1) == cudaSuccess &&
             h2d(O[HK], k, desc->dk * L.in_isz, t0, t1) == cudaSuccess &&
             h2d(O[HV], v, desc->dv * L.in_isz, t0, t1) == cudaSuccess &&
             h2d(O[HB], beta, L.in_isz, t0, t1) == cudaSuccess &&
             (desc->gate == DR_GATE_NONE || h2d(O[HLA], log_alpha, 4 * L.la_w, t0, t1) == cudaSuccess) &&
             cudaEventRecord(e_in[p], s_in) == cudaSuccess && cudaStreamWaitEvent(s_comp, e_in[p], 0) == cudaSuccess;
        if (!ok) break;
        dr_chunk_desc dp = *desc;
        dp.T = t1 - t0;
        // the state: from the host (or zero) into piece 0, then carried in place
        const float *s_in_ptr = (p == 0 && !init_state) ? nullptr : state;
        rc = dr_chunk_fwd(&dp, d + O[HQ], d + O[HK], d + O[HV],
                          desc->gate == DR_GATE_NONE ? nullptr : (const float *)(d + O[HLA]), d + O[HB],
                          s_in_ptr, d + O[HOUT], state, L.ws_bytes[p] ? d + O[HWS] : nullptr,
                          L.ws_bytes[p], (dr_stream_t)s_comp);
        if (rc != kOk) {
            ok = false;
            break;
        }
        ok = cudaEventRecord(e_comp[p], s_comp) == cudaSuccess &&
             cudaStreamWaitEvent(s_out, e_comp[p], 0) == cudaSuccess &&
             d2h(out, O[HOUT], desc->dv * L.out_isz, t0, t1) == cudaSuccess;
    }
    if (ok && final_state)
        ok = cudaMemcpyAsync(final_state, state, st_bytes, cudaMemcpyDeviceToHost, s_out) == cudaSuccess;
    if (ok) ok = cudaEventRecord(e_done, s_out) == cudaSuccess && cudaStreamWaitEvent(main, e_done, 0) == cudaSuccess;
    if (!ok) {
        // part of the work may be enqueued: `main` still waits for all of it, so that a
        // caller who synchronises `stream` after the error may free or reuse the buffers
        // (a stream whose event cannot be recorded is synchronised instead)
        for (cudaStream_t s : {s_in, s_comp, s_out})
            if (cudaEventRecord(e_done, s) != cudaSuccess || cudaStreamWaitEvent(main, e_done, 0) != cudaSuccess)
                cudaStreamSynchronize(s);
    }
    cleanup();
    if (!ok) return rc != kOk ? rc : kErrCuda;
    return kOk;
}
