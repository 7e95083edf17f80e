// host_api.cu -- dr_chunk_fwd_host: the chunk forward for callers holding HOST buffers.
//
// Copies the inputs host -> device, runs dr_chunk_fwd and copies out and final_state
// device -> host, all enqueued asynchronously behind `stream`.  Every (b, h) chain is
// independent, so the batch is split into `pieces` groups of batch rows; piece p's
// kernels run on their own stream as soon as its inputs have arrived, while the inputs of
// piece p + 1 are still on their way in and the outputs of piece p - 1 on their way out
// (the two copy directions use different copy engines and overlap on the link).  Streams
// and events are created per call and released behind the work; the only device memory
// used is the caller's buffer `dev`.
#include <algorithm>

#include "../../include/dr.h"
#include "chunk_layout.h"
#include "common.cuh"

namespace dr {
namespace {

constexpr int kMaxPieces = 16;

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// Per piece, one 256-byte-aligned region per tensor (so every slice the kernels get is
// aligned whatever the row sizes): [q | k | v | beta | log alpha | S0 | out | final | ws].
struct HostLayout {
    int pieces;
    int64_t rows[kMaxPieces + 1];          // batch-row boundaries of the pieces
    size_t in_isz, out_isz;
    size_t base[kMaxPieces][9];            // byte offsets in `dev`, piece p, tensor i
    size_t ws_bytes[kMaxPieces];
    size_t total;
};
enum { HQ, HK, HV, HB, HLA, HS0, HOUT, HFIN, HWS };

bool host_layout(const dr_chunk_desc *d, int pieces, bool has_s0, bool has_fin, HostLayout *L) {
    if (!d || d->B < 1 || pieces < 1) return false;
    const int P = (int)std::min<int64_t>(std::min<int64_t>(pieces, kMaxPieces), d->B);
    L->pieces = P;
    for (int p = 0; p <= P; ++p) L->rows[p] = d->B * p / P;
    L->in_isz = d->in_dtype == DR_BF16 ? 2 : 4;
    L->out_isz = d->out_dtype == DR_BF16 ? 2 : 4;
    const size_t th = (size_t)(d->T * d->H);
    const size_t st = (size_t)(d->H * d->dk * d->dv) * 4;
    const size_t la_w = d->gate == DR_GATE_NONE ? 0 : (d->gate == DR_GATE_CHANNEL ? (size_t)d->dk : 1);
    size_t off = 0;
    for (int p = 0; p < P; ++p) {
        const size_t nb = (size_t)(L->rows[p + 1] - L->rows[p]);
        dr_chunk_desc dp = *d;
        dp.B = (int64_t)nb;
        size_t w = 0;
        if (dr_chunk_fwd_workspace_bytes(&dp, &w) != DR_OK) return false;
        const size_t sizes[9] = {nb * th * d->dk * L->in_isz, nb * th * d->dk * L->in_isz,
                                 nb * th * d->dv * L->in_isz, nb * th * L->in_isz, nb * th * 4 * la_w,
                                 has_s0 ? nb * st : 0, nb * th * d->dv * L->out_isz, has_fin ? nb * st : 0, w};
        for (int i = 0; i < 9; ++i) {
            L->base[p][i] = off;
            off += align256(sizes[i]);
        }
        L->ws_bytes[p] = w;
    }
    L->total = off;
    return true;
}

}  // namespace
}  // namespace dr

using namespace dr;

extern "C" int dr_chunk_fwd_host_dev_bytes(const dr_chunk_desc *desc, int pieces, int with_init_state,
                                           int with_final_state, size_t *bytes) {
    if (!bytes || !desc) return kErrInvalid;
    size_t w = 0;
    const int rc = dr_chunk_fwd_workspace_bytes(desc, &w);   // validates the descriptor
    if (rc != kOk) return rc;
    if (pieces < 1) return kErrInvalid;
    HostLayout L;
    if (!host_layout(desc, pieces, with_init_state != 0, with_final_state != 0, &L)) return kErrInvalid;
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
    if (pieces < 1) return kErrInvalid;
    if (desc->T > 0 && (!q || !k || !v || !beta || !out)) return kErrInvalid;
    if (desc->gate != DR_GATE_NONE && desc->T > 0 && !log_alpha) return kErrInvalid;
    HostLayout L;
    if (!host_layout(desc, pieces, init_state != nullptr, final_state != nullptr, &L)) return kErrInvalid;
    if (!dev || dev_bytes < L.total || ((uintptr_t)dev & 255u) != 0) return kErrWorkspace;

    cudaStream_t main = (cudaStream_t)stream;
    cudaStream_t s_in = nullptr, s_out = nullptr, s_comp[kMaxPieces] = {};
    cudaEvent_t e_start = nullptr, e_in[kMaxPieces] = {}, e_comp[kMaxPieces] = {}, e_done = nullptr;
    auto cleanup = [&]() {   // released once the enqueued work has finished
        for (int p = 0; p < kMaxPieces; ++p) {
            if (s_comp[p]) cudaStreamDestroy(s_comp[p]);
            if (e_in[p]) cudaEventDestroy(e_in[p]);
            if (e_comp[p]) cudaEventDestroy(e_comp[p]);
        }
        if (s_in) cudaStreamDestroy(s_in);
        if (s_out) cudaStreamDestroy(s_out);
        if (e_start) cudaEventDestroy(e_start);
        if (e_done) cudaEventDestroy(e_done);
    };
    const int P = L.pieces;
    bool ok = cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&e_start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&e_done, cudaEventDisableTiming) == cudaSuccess;
    for (int p = 0; ok && p < P; ++p)
        ok = cudaStreamCreateWithFlags(&s_comp[p], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&e_in[p], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&e_comp[p], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cleanup();
        return kErrCuda;
    }

    char *d = (char *)dev;
    const size_t TH = (size_t)(desc->T * desc->H);
    const size_t st_row = (size_t)(desc->H * desc->dk * desc->dv) * 4;   // one batch row of a state
    const size_t la_w = desc->gate == DR_GATE_CHANNEL ? (size_t)desc->dk : 1;
    // rows [r0, r1) of a host tensor of `row_bytes` per batch row <-> region `dst` of piece p
    auto h2d = [&](size_t dst, const void *src, size_t row_bytes, int64_t r0, int64_t r1) {
        const size_t n = row_bytes * (size_t)(r1 - r0);
        if (n == 0 || !src) return cudaSuccess;
        return cudaMemcpyAsync(d + dst, (const char *)src + row_bytes * r0, n, cudaMemcpyHostToDevice, s_in);
    };
    auto d2h = [&](void *dst, size_t src, size_t row_bytes, int64_t r0, int64_t r1) {
        const size_t n = row_bytes * (size_t)(r1 - r0);
        if (n == 0 || !dst) return cudaSuccess;
        return cudaMemcpyAsync((char *)dst + row_bytes * r0, d + src, n, cudaMemcpyDeviceToHost, s_out);
    };
    ok = cudaEventRecord(e_start, main) == cudaSuccess && cudaStreamWaitEvent(s_in, e_start, 0) == cudaSuccess &&
         cudaStreamWaitEvent(s_out, e_start, 0) == cudaSuccess;
    for (int p = 0; ok && p < P; ++p) {
        const int64_t r0 = L.rows[p], r1 = L.rows[p + 1];
        const size_t *B0 = L.base[p];
        ok = h2d(B0[HQ], q, TH * desc->dk * L.in_isz, r0, r1) == cudaSuccess &&
             h2d(B0[HK], k, TH * desc->dk * L.in_isz, r0, r1) == cudaSuccess &&
             h2d(B0[HV], v, TH * desc->dv * L.in_isz, r0, r1) == cudaSuccess &&
             h2d(B0[HB], beta, TH * L.in_isz, r0, r1) == cudaSuccess &&
             (desc->gate == DR_GATE_NONE || h2d(B0[HLA], log_alpha, TH * 4 * la_w, r0, r1) == cudaSuccess) &&
             h2d(B0[HS0], init_state, st_row, r0, r1) == cudaSuccess &&
             cudaEventRecord(e_in[p], s_in) == cudaSuccess &&
             cudaStreamWaitEvent(s_comp[p], e_in[p], 0) == cudaSuccess;
        if (!ok) break;
        dr_chunk_desc dp = *desc;
        dp.B = r1 - r0;
        rc = dr_chunk_fwd(&dp, d + B0[HQ], d + B0[HK], d + B0[HV],
                          desc->gate == DR_GATE_NONE ? nullptr : (const float *)(d + B0[HLA]), d + B0[HB],
                          init_state ? (const float *)(d + B0[HS0]) : nullptr, d + B0[HOUT],
                          final_state ? (float *)(d + B0[HFIN]) : nullptr,
                          L.ws_bytes[p] ? d + B0[HWS] : nullptr, L.ws_bytes[p], (dr_stream_t)s_comp[p]);
        if (rc != kOk) {
            ok = false;
            break;
        }
        ok = cudaEventRecord(e_comp[p], s_comp[p]) == cudaSuccess &&
             cudaStreamWaitEvent(s_out, e_comp[p], 0) == cudaSuccess &&
             d2h(out, B0[HOUT], TH * desc->dv * L.out_isz, r0, r1) == cudaSuccess &&
             d2h(final_state, B0[HFIN], st_row, r0, r1) == cudaSuccess;
    }
    if (ok) ok = cudaEventRecord(e_done, s_out) == cudaSuccess && cudaStreamWaitEvent(main, e_done, 0) == cudaSuccess;
    cleanup();
    if (!ok) return rc != kOk ? rc : kErrCuda;
    return kOk;
}
