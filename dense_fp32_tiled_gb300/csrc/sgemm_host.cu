// sgemm_host.cu -- the FP32 product for operands that live in host memory.
//
// The product itself is sgemm_f32_ws (the tiled CUDA-core kernel).  This
// file adds the transfers around it.  A is copied in row panels on a copy
// stream, and the product of each panel starts, on the caller's stream, as
// soon as that panel and B have landed.  Each finished panel of C is copied
// back on a second copy stream while the next panel computes; the last panel
// is cut in two so that the final copy back, which nothing hides, is short.
//
// Every row of C needs all of B, so B's copy would otherwise stall the first
// product.  When there are several panels and N >= 512, the first panel's
// product is cut into column blocks instead (4 when N >= 1024, else 2): the
// copy order is A's first panel, B's column blocks one by one, then A's
// other panels, and each block of the first panel computes while the next
// block of B is still in flight.
//
// The device copies of A, B and C have 16-byte aligned rows (leading
// dimensions rounded up to 4 floats), whatever the host leading dimensions.
//
// Host memory should be pinned (page-locked) for the copies to run
// asynchronously at full speed; pageable memory works, but the CUDA runtime
// then stages it.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "ctx_key.cuh"
#include "nvtx_range.cuh"
#include "sgemm_f32.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxPanels = 4;
constexpr int kPanelRows = 1024;  // rows per panel when M allows several (a multiple of the 128-row tile)

size_t round256(size_t b) { return (b + 255) / 256 * 256; }
// Device copies keep rows 16-byte aligned (leading dimension rounded up to
// 4 floats), so the products always run on the tensor-copy kernels.
long long pad4(long long n) { return (n + 3) / 4 * 4; }

// Row panels, panel p holding rows [start[p], start[p + 1]).
//   Wide products (N >= 2048, M >= 3 kPanelRows): a first panel of
//   kPanelRows rows, one panel up to the last 512 rows, and a last panel of
//   512 rows.  The product of a row of A takes several times longer than its
//   copy here (the ratio grows with N), so the middle panel's rows have
//   landed before the first panel's product ends, and one large product runs
//   on the whole-wave schedules instead of several panel products of fewer
//   tiles than the GPU holds at once.  Measured on GB300 against the plan
//   below (TFLOP/s, pinned buffers): 4096^3 56.6 -> 58.8, 8192^3 68.0 ->
//   69.2, 4096 x 2048 x 4096 49.2 -> 50.6; first / last panels of 768 / 512,
//   1280 / 512, 1024 / 256 and 1024 / 1024 rows did no better overall.
//   Otherwise: up to kMaxPanels panels of `rows` rows (the last may be
//   shorter); with several panels, a last panel of at least 512 rows is cut
//   in two (on the 128-row tile), so that the copy back of the last panel of
//   C, which nothing hides, is half as long.
struct Panels {
    int P;
    int start[kMaxPanels + 2];
    int rows(int p) const { return start[p + 1] - start[p]; }
};
Panels panels_of(int M, int N) {
    if (N >= 2048 && M >= 3 * kPanelRows) {
        Panels pn;
        pn.start[0] = 0;
        pn.start[1] = kPanelRows;
        pn.start[2] = M - 512;
        pn.start[3] = M;
        pn.P = 3;
        return pn;
    }
    int P = M / kPanelRows;
    P = P < 1 ? 1 : (P > kMaxPanels ? kMaxPanels : P);
    int rows = (M + P - 1) / P;
    rows = (rows + 127) / 128 * 128;
    P = (M + rows - 1) / rows;
    Panels pn;
    for (int p = 0; p < P; ++p) pn.start[p] = p * rows;
    pn.start[P] = M;
    pn.P = P;
    const int last = M - (P - 1) * rows;
    if (P >= 2 && last >= 512) {
        pn.start[P] = (P - 1) * rows + (last / 2 + 127) / 128 * 128;
        pn.start[P + 1] = M;
        pn.P = P + 1;
    }
    return pn;
}

// Column blocks of the first panel's product: with several panels, B is
// copied and the first panel computed in NB blocks of columns (4 when
// N >= 1024, 2 when N >= 512, else 1), block j covering [col_start(j),
// col_start(j + 1)) with boundaries on the 128-column tile.
constexpr int kMaxColBlocks = 4;
int col_blocks(int P, int N) { return P >= 2 ? (N >= 1024 ? 4 : (N >= 512 ? 2 : 1)) : 1; }
int col_start(int j, int NB, int N) {
    return j >= NB ? N : static_cast<int>(static_cast<long long>(N) * j / NB) / 128 * 128;
}

struct HostLayout {
    size_t b, a, c, ws, ws_bytes, bytes;
};
HostLayout host_layout(int M, int N, int K) {
    const Panels pn = panels_of(M, N);
    HostLayout l;
    l.b = 0;
    l.a = round256(static_cast<size_t>(K) * pad4(N) * 4);
    l.c = l.a + round256(static_cast<size_t>(M) * pad4(K) * 4);
    l.ws = l.c + round256(static_cast<size_t>(M) * pad4(N) * 4);
    // the products run one after another on one stream, so they share one
    // workspace sized for the largest need among the shapes they take: the
    // schedule's words and, where it pays, the k-major copy of the panel of
    // A (the device copies have 16-byte aligned rows, which is all the size
    // query inspects of its pointers, so any 16-byte aligned stand-in will do)
    const int NB = col_blocks(pn.P, N);
    const float *aligned = reinterpret_cast<const float *>(static_cast<uintptr_t>(256));
    const int K4 = static_cast<int>(pad4(K > 0 ? K : 1)), N4 = static_cast<int>(pad4(N));
    auto need_for = [&](int m, int n) { return sgemm_f32_workspace_size_for(m, n, K, aligned, K4, aligned, N4); };
    size_t w = 0;
    for (int p = 0; p < pn.P; ++p) {
        const size_t x = need_for(pn.rows(p), N);
        w = x > w ? x : w;
    }
    for (int j = 0; j < NB; ++j) {
        const size_t x = need_for(pn.rows(0), col_start(j + 1, NB, N) - col_start(j, NB, N));
        w = x > w ? x : w;
    }
    l.ws_bytes = round256(w);
    l.bytes = l.ws + l.ws_bytes;
    return l;
}

// One pair of non-blocking copy streams per device, made on first use.
// A new context of the device (e.g. after cudaDeviceReset, which destroys
// the streams with the old one) gets a new pair.
std::mutex g_stream_mutex;
cudaStream_t g_h2d[kMaxDevices], g_d2h[kMaxDevices];
unsigned long long g_stream_ctx[kMaxDevices];

int copy_streams(int dev, cudaStream_t &h2d, cudaStream_t &d2h) {
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    unsigned long long ctx = 0;
    const bool known = sg_ctx::current_id(dev, &ctx);
    std::lock_guard<std::mutex> lock(g_stream_mutex);
    if (known && g_h2d[dev] != nullptr && g_stream_ctx[dev] != ctx) g_h2d[dev] = g_d2h[dev] = nullptr;
    if (g_h2d[dev] == nullptr) {
        g_stream_ctx[dev] = ctx;
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
    if (K > INT_MAX - 3 || N > INT_MAX - 3) return SGEMM_ERR_INVALID_DIM;  // padded leading dimensions
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
    const Panels pn = panels_of(M, N);
    const int P = pn.P;
    const int NB = col_blocks(P, N);
    const int K4 = static_cast<int>(pad4(K)), N4 = static_cast<int>(pad4(N));  // fit: checked above

    // events: start, all copied back, B's column block j landed, A panel p
    // landed, C panel p computed
    cudaEvent_t ev[2 + kMaxColBlocks + 2 * (kMaxPanels + 1)] = {};
    const int n_ev = 2 + NB + 2 * P;
    for (int i = 0; i < n_ev; ++i) {
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            for (int j = 0; j < i; ++j) (void)cudaEventDestroy(ev[j]);
            return SGEMM_ERR_DEVICE;
        }
    }
    cudaEvent_t &e_start = ev[0], &e_done = ev[1];
    cudaEvent_t *e_b = ev + 2, *e_a = ev + 2 + NB, *e_c = ev + 2 + NB + P;

    auto fail = [&](int code) {
        (void)cudaGetLastError();
        for (int i = 0; i < n_ev; ++i) (void)cudaEventDestroy(ev[i]);
        return code;
    };
    // columns [c0, c0 + nc) of B, all K rows
    auto copy_b = [&](int c0, int nc) {
        sg_nvtx::Range r("sgemm_f32_host: copy in B block");
        return K == 0 || cudaMemcpy2DAsync(dB + c0, static_cast<size_t>(N4) * 4, B + c0, static_cast<size_t>(ldb) * 4,
                                           static_cast<size_t>(nc) * 4, K, cudaMemcpyHostToDevice, h2d) == cudaSuccess;
    };
    auto copy_a = [&](int p) {
        sg_nvtx::Range r("sgemm_f32_host: copy in A panel");
        const int r0 = pn.start[p], nr = pn.rows(p);
        return (K == 0 || cudaMemcpy2DAsync(dA + static_cast<size_t>(r0) * K4, static_cast<size_t>(K4) * 4,
                                            A + static_cast<size_t>(r0) * lda, static_cast<size_t>(lda) * 4,
                                            static_cast<size_t>(K) * 4, nr, cudaMemcpyHostToDevice,
                                            h2d) == cudaSuccess) &&
               cudaEventRecord(e_a[p], h2d) == cudaSuccess;
    };
    // columns [c0, c0 + nc) of panel p's product
    auto product = [&](int p, int c0, int nc) {
        const int r0 = pn.start[p], nr = pn.rows(p);
        return sgemm_f32_ws(nr, nc, K, dA + static_cast<size_t>(r0) * K4, K4 > 0 ? K4 : 1, dB + c0, N4,
                            dC + static_cast<size_t>(r0) * N4 + c0, N4, dW, l.ws_bytes, stream);
    };
    // the workspace may still be in use by work queued earlier on `stream`
    if (cudaEventRecord(e_start, stream) != cudaSuccess || cudaStreamWaitEvent(h2d, e_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(d2h, e_start, 0) != cudaSuccess)
        return fail(SGEMM_ERR_LAUNCH);
    // copy order: A panel 0, B's column blocks, A panels 1..
    if (!copy_a(0)) return fail(SGEMM_ERR_LAUNCH);
    for (int j = 0; j < NB; ++j) {
        const int c0 = col_start(j, NB, N), c1 = col_start(j + 1, NB, N);
        if (!copy_b(c0, c1 - c0) || cudaEventRecord(e_b[j], h2d) != cudaSuccess) return fail(SGEMM_ERR_LAUNCH);
    }
    for (int p = 1; p < P; ++p)
        if (!copy_a(p)) return fail(SGEMM_ERR_LAUNCH);
    for (int p = 0; p < P; ++p) {
        const int r0 = pn.start[p], nr = pn.rows(p);
        if (cudaStreamWaitEvent(stream, e_a[p], 0) != cudaSuccess) return fail(SGEMM_ERR_LAUNCH);
        if (p == 0) {  // block by block, each while the next block of B lands
            for (int j = 0; j < NB; ++j) {
                const int c0 = col_start(j, NB, N), c1 = col_start(j + 1, NB, N);
                if (cudaStreamWaitEvent(stream, e_b[j], 0) != cudaSuccess) return fail(SGEMM_ERR_LAUNCH);
                st = product(0, c0, c1 - c0);
                if (st != SGEMM_OK) return fail(st);
            }
        } else {
            st = product(p, 0, N);
        }
        if (st != SGEMM_OK) return fail(st);
        if (cudaEventRecord(e_c[p], stream) != cudaSuccess || cudaStreamWaitEvent(d2h, e_c[p], 0) != cudaSuccess)
            return fail(SGEMM_ERR_LAUNCH);
        sg_nvtx::Range r("sgemm_f32_host: copy out C panel");
        if (cudaMemcpy2DAsync(C + static_cast<size_t>(r0) * ldc, static_cast<size_t>(ldc) * 4,
                              dC + static_cast<size_t>(r0) * N4, static_cast<size_t>(N4) * 4,
                              static_cast<size_t>(N) * 4, nr, cudaMemcpyDeviceToHost, d2h) != cudaSuccess)
            return fail(SGEMM_ERR_LAUNCH);
    }
    // later work on `stream` sees C complete in host memory
    if (cudaEventRecord(e_done, d2h) != cudaSuccess || cudaStreamWaitEvent(stream, e_done, 0) != cudaSuccess)
        return fail(SGEMM_ERR_LAUNCH);
    for (int i = 0; i < n_ev; ++i) (void)cudaEventDestroy(ev[i]);  // released once they complete
    return SGEMM_OK;
}
