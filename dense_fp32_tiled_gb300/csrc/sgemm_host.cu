// sgemm_host.cu -- the FP32 product for operands that live in host memory.
//
// The product itself is sgemm_f32_ws (the tiled CUDA-core kernel).  This
// file adds the transfers around it.  B is copied to the device first, since
// every row of C needs all of B.  A is then copied in row panels on a copy
// stream, and the product of each panel starts, on the caller's stream, as
// soon as that panel has landed.  Each finished panel of C is copied back on
// a second copy stream while the next panel computes.  Host memory should be
// pinned (page-locked) for the copies to run asynchronously at full speed;
// pageable memory works, but the CUDA runtime then stages it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sgemm_f32.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxPanels = 4;
constexpr int kPanelRows = 1024;  // rows per panel when M allows several (a multiple of the 128-row tile)

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Row panels: P panels of `rows` rows (the last may be shorter).
void panels_of(int M, int &P, int &rows) {
    P = M / kPanelRows;
    P = P < 1 ? 1 : (P > kMaxPanels ? kMaxPanels : P);
    rows = (M + P - 1) / P;
    rows = (rows + 127) / 128 * 128;
    P = (M + rows - 1) / rows;
}

struct HostLayout {
    size_t b, a, c, ws, ws_bytes, bytes;
};
HostLayout host_layout(int M, int N, int K) {
    int P = 0, rows = 0;
    panels_of(M, P, rows);
    HostLayout l;
    l.b = 0;
    l.a = round256(static_cast<size_t>(K) * N * 4);
    l.c = l.a + round256(static_cast<size_t>(M) * K * 4);
    l.ws = l.c + round256(static_cast<size_t>(M) * N * 4);
    const int last = M - (P - 1) * rows;  // the last panel's rows (its schedule may differ)
    const size_t w_full = sgemm_f32_workspace_size(rows < M ? rows : M, N, K);
    const size_t w_last = sgemm_f32_workspace_size(last, N, K);
    l.ws_bytes = round256(w_full > w_last ? w_full : w_last);
    l.bytes = l.ws + l.ws_bytes;
    return l;
}

// One pair of non-blocking copy streams per device, made on first use.
std::mutex g_stream_mutex;
cudaStream_t g_h2d[kMaxDevices], g_d2h[kMaxDevices];

int copy_streams(int dev, cudaStream_t &h2d, cudaStream_t &d2h) {
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_stream_mutex);
    if (g_h2d[dev] == nullptr) {
        cudaStream_t a = nullptr, b = nullptr;
        if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
            (void)cudaGetLastError();
            if (a != nullptr) (void)cudaStreamDestroy(a);
            return SGEMM_ERR_DEVICE;
        }
        g_h2d[dev] = a;
        g_d2h[dev] = b;
    }
    h2d = g_h2d[dev];
    d2h = g_d2h[dev];
    return SGEMM_OK;
}

bool overlap(const void *a, long long an, const void *b, long long bn) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return an > 0 && bn > 0 && x < y + static_cast<uintptr_t>(bn) && y < x + static_cast<uintptr_t>(an);
}
long long extent(int rows, int cols, int ld) {
    return rows > 0 && cols > 0 ? (static_cast<long long>(rows) - 1) * ld + cols : 0;
}

}  // namespace

extern "C" size_t sgemm_f32_host_workspace_size(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K < 0) return 0;
    return host_layout(M, N, K).bytes;
}

extern "C" int sgemm_f32_host(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C,
                              int ldc, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return SGEMM_ERR_INVALID_LD;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr)) || workspace == nullptr) return SGEMM_ERR_NULL_PTR;
    const uintptr_t host_bits =
        reinterpret_cast<uintptr_t>(C) | (K > 0 ? reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) : 0);
    if (host_bits % 4 != 0 || reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SGEMM_ERR_INVALID_ARG;
    const long long c_bytes = 4 * extent(M, N, ldc);
    if (K > 0 && (overlap(C, c_bytes, A, 4 * extent(M, K, lda)) || overlap(C, c_bytes, B, 4 * extent(K, N, ldb))))
        return SGEMM_ERR_ALIAS;
    const HostLayout l = host_layout(M, N, K);
    if (workspace_bytes < l.bytes) return SGEMM_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    cudaStream_t h2d = nullptr, d2h = nullptr;
    int st = copy_streams(dev, h2d, d2h);
    if (st != SGEMM_OK) return st;

    char *ws = static_cast<char *>(workspace);
    float *dB = reinterpret_cast<float *>(ws + l.b);
    float *dA = reinterpret_cast<float *>(ws + l.a);
    float *dC = reinterpret_cast<float *>(ws + l.c);
    void *dW = ws + l.ws;
    int P = 0, rows = 0;
    panels_of(M, P, rows);

    // events: start, B landed, A panel p landed, C panel p computed, all copied back
    cudaEvent_t ev[3 + 2 * kMaxPanels] = {};
    const int n_ev = 3 + 2 * P;
    for (int i = 0; i < n_ev; ++i) {
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            for (int j = 0; j < i; ++j) (void)cudaEventDestroy(ev[j]);
            return SGEMM_ERR_DEVICE;
        }
    }
    cudaEvent_t &e_start = ev[0], &e_b = ev[1], &e_done = ev[2];
    cudaEvent_t *e_a = ev + 3, *e_c = ev + 3 + P;

    auto fail = [&](int code) {
        (void)cudaGetLastError();
        for (int i = 0; i < n_ev; ++i) (void)cudaEventDestroy(ev[i]);
        return code;
    };
    // the workspace may still be in use by work queued earlier on `stream`
    if (cudaEventRecord(e_start, stream) != cudaSuccess || cudaStreamWaitEvent(h2d, e_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(d2h, e_start, 0) != cudaSuccess)
        return fail(SGEMM_ERR_LAUNCH);
    if (K > 0 && cudaMemcpy2DAsync(dB, static_cast<size_t>(N) * 4, B, static_cast<size_t>(ldb) * 4,
                                   static_cast<size_t>(N) * 4, K, cudaMemcpyHostToDevice, h2d) != cudaSuccess)
        return fail(SGEMM_ERR_LAUNCH);
    if (cudaEventRecord(e_b, h2d) != cudaSuccess) return fail(SGEMM_ERR_LAUNCH);
    for (int p = 0; p < P; ++p) {
        const int r0 = p * rows, nr = (M - r0) < rows ? (M - r0) : rows;
        if (K > 0 && cudaMemcpy2DAsync(dA + static_cast<size_t>(r0) * K, static_cast<size_t>(K) * 4,
                                       A + static_cast<size_t>(r0) * lda, static_cast<size_t>(lda) * 4,
                                       static_cast<size_t>(K) * 4, nr, cudaMemcpyHostToDevice, h2d) != cudaSuccess)
            return fail(SGEMM_ERR_LAUNCH);
        if (cudaEventRecord(e_a[p], h2d) != cudaSuccess) return fail(SGEMM_ERR_LAUNCH);
    }
    if (cudaStreamWaitEvent(stream, e_b, 0) != cudaSuccess) return fail(SGEMM_ERR_LAUNCH);
    for (int p = 0; p < P; ++p) {
        const int r0 = p * rows, nr = (M - r0) < rows ? (M - r0) : rows;
        if (cudaStreamWaitEvent(stream, e_a[p], 0) != cudaSuccess) return fail(SGEMM_ERR_LAUNCH);
        st = sgemm_f32_ws(nr, N, K, dA + static_cast<size_t>(r0) * K, K > 0 ? K : 1, dB, N,
                          dC + static_cast<size_t>(r0) * N, N, dW, l.ws_bytes, stream);
        if (st != SGEMM_OK) return fail(st);
        if (cudaEventRecord(e_c[p], stream) != cudaSuccess || cudaStreamWaitEvent(d2h, e_c[p], 0) != cudaSuccess)
            return fail(SGEMM_ERR_LAUNCH);
        if (cudaMemcpy2DAsync(C + static_cast<size_t>(r0) * ldc, static_cast<size_t>(ldc) * 4,
                              dC + static_cast<size_t>(r0) * N, static_cast<size_t>(N) * 4,
                              static_cast<size_t>(N) * 4, nr, cudaMemcpyDeviceToHost, d2h) != cudaSuccess)
            return fail(SGEMM_ERR_LAUNCH);
    }
    // later work on `stream` sees C complete in host memory
    if (cudaEventRecord(e_done, d2h) != cudaSuccess || cudaStreamWaitEvent(stream, e_done, 0) != cudaSuccess)
        return fail(SGEMM_ERR_LAUNCH);
    for (int i = 0; i < n_ev; ++i) (void)cudaEventDestroy(ev[i]);  // released once they complete
    return SGEMM_OK;
}
