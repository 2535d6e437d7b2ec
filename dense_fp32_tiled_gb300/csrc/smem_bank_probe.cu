// smem_bank_probe.cu -- the shared-memory stride sweep (declared in
// include/smem_bank_probe.h): measures, on the running GPU, how many passes a
// warp-wide 32-bit shared-memory access with a given lane stride needs (bank
// page, "四种访问，四种结果" and "把推导变成测量").
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "smem_bank_probe.h"

namespace {

constexpr int kWords = 4096;

// Access U of a group: one 32-bit shared load (OP 0, added into acc in the
// same asm block, so the value is consumed at once) or store (OP 1) of word
// lane_word + 32 U at address lane_addr + 128 U; the offset is an immediate
// of the instruction.
template <int OP, int U>
__device__ __forceinline__ void access(uint32_t lane_addr, int lane_word, unsigned &acc) {
    if constexpr (OP == 0) {
        asm volatile("{\n .reg .b32 t;\n ld.volatile.shared.b32 t, [%1+%2];\n add.u32 %0, %0, t;\n}\n"
                     : "+r"(acc)
                     : "r"(lane_addr), "n"(128 * U)
                     : "memory");
    } else {
        asm volatile("st.volatile.shared.b32 [%0+%1], %2;" ::"r"(lane_addr), "n"(128 * U), "r"(lane_word + 32 * U)
                     : "memory");
    }
}
template <int OP, int... U>
__device__ __forceinline__ void access_group(uint32_t lane_addr, int lane_word, unsigned &acc,
                                             std::integer_sequence<int, U...>) {
    (access<OP, U>(lane_addr, lane_word, acc), ...);
}

// One CTA.  Lane l of every warp touches word l * stride + 32 u in access u
// of each group of 64 (u = 0 .. 63): at most 31 * 64 + 32 * 63 = 4000 < 4096,
// so every access stays inside the array.  The accesses are inline PTX with
// immediate offsets, so each one is exactly one 32-bit shared load (op 0) or
// store (op 1) per lane with little else around it, and the shared-memory
// pipe, not instruction issue, bounds the loop.  result[0] = cycles of the
// timed loop (thread 0), result[1] = the checksum.
template <int OP>
__global__ void __launch_bounds__(256) bank_stride_kernel(int stride, int iters, long long *result) {
    __shared__ int s[kWords];
    for (int i = threadIdx.x; i < kWords; i += blockDim.x) s[i] = OP == 0 ? i : -1;
    const int l = threadIdx.x & 31;
    const int lane_word = l * stride;
    const uint32_t lane_addr = static_cast<uint32_t>(__cvta_generic_to_shared(s)) + 4u * lane_word;
    unsigned acc = 0u;
    __syncthreads();
    const long long t0 = clock64();
    for (int j = 0; j < iters; j += 64)
        access_group<OP>(lane_addr, lane_word, acc, std::make_integer_sequence<int, 64>{});
    __syncthreads();
    const long long t1 = clock64();
    long long sum = acc;
    if (OP == 1)
        for (int i = threadIdx.x; i < kWords; i += blockDim.x) sum += s[i];
    if (threadIdx.x == 0) result[0] = t1 - t0;
    atomicAdd(reinterpret_cast<unsigned long long *>(result + 1), static_cast<unsigned long long>(sum));
}

// One warp-wide access pattern: lane l reads W bytes at word lane_word[l] +
// 32 u in access u of each group of 64 (a shift by 32 words keeps every bank;
// every word stays below 2048 + 32 * 63 + 4 < 4096).  The loads are volatile,
// so none is merged with another or moved out of the loop, and only the
// first word of each is added into acc (one add per load keeps instruction
// issue below the pipe's rate for all but the cheapest patterns).
struct LaneWords {
    int w[32];
};
template <int W, int U>
__device__ __forceinline__ void vload(uint32_t lane_addr, unsigned &acc) {
    constexpr int off = 128 * U;
    if constexpr (W == 4) {
        asm volatile("{\n .reg .b32 t;\n ld.volatile.shared.b32 t, [%1+%2];\n add.u32 %0, %0, t;\n}\n"
                     : "+r"(acc) : "r"(lane_addr), "n"(off) : "memory");
    } else if constexpr (W == 8) {
        asm volatile("{\n .reg .b32 t0, t1;\n ld.volatile.shared.v2.b32 {t0, t1}, [%1+%2];\n add.u32 %0, %0, t0;\n}\n"
                     : "+r"(acc) : "r"(lane_addr), "n"(off) : "memory");
    } else {
        asm volatile("{\n .reg .b32 t0, t1, t2, t3;\n ld.volatile.shared.v4.b32 {t0, t1, t2, t3}, [%1+%2];\n"
                     " add.u32 %0, %0, t0;\n}\n"
                     : "+r"(acc) : "r"(lane_addr), "n"(off) : "memory");
    }
}
template <int W, int... U>
__device__ __forceinline__ void vload_group(uint32_t lane_addr, unsigned &acc, std::integer_sequence<int, U...>) {
    (vload<W, U>(lane_addr, acc), ...);
}
template <int W>
__global__ void __launch_bounds__(256) bank_pattern_kernel(const LaneWords lw, int iters, long long *result) {
    __shared__ __align__(16) int s[kWords];
    for (int i = threadIdx.x; i < kWords; i += blockDim.x) s[i] = i;
    const uint32_t lane_addr = static_cast<uint32_t>(__cvta_generic_to_shared(s)) + 4u * lw.w[threadIdx.x & 31];
    unsigned acc = 0u;
    __syncthreads();
    const long long t0 = clock64();
    for (int j = 0; j < iters; j += 64) vload_group<W>(lane_addr, acc, std::make_integer_sequence<int, 64>{});
    __syncthreads();
    const long long t1 = clock64();
    if (threadIdx.x == 0) result[0] = t1 - t0;
    atomicAdd(reinterpret_cast<unsigned long long *>(result + 1), static_cast<unsigned long long>(acc));
}

// Runs one probe launch and copies back (cycles, checksum).
template <class Launch>
int run_probe(Launch launch, int warps, int iters, double *cycles_per_access, long long *checksum) {
    long long *d = nullptr;
    if (cudaMalloc(&d, 2 * sizeof(long long)) != cudaSuccess) {
        (void)cudaGetLastError();
        return -5;
    }
    int rc = 0;
    long long h[2] = {0, 0};
    if (cudaMemset(d, 0, 2 * sizeof(long long)) != cudaSuccess) {
        rc = -5;
    } else {
        launch(d);
        if (cudaGetLastError() != cudaSuccess || cudaMemcpy(h, d, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
            rc = -5;
    }
    (void)cudaGetLastError();
    (void)cudaFree(d);
    if (rc == 0) {
        *cycles_per_access = static_cast<double>(h[0]) / (static_cast<double>(warps) * iters);
        *checksum = h[1];
    }
    return rc;
}

}  // namespace

extern "C" int smem_bank_pattern_probe(int width_bytes, const int *lane_word, int warps, int iters,
                                       double *cycles_per_access, long long *checksum) {
    if (cycles_per_access == nullptr || checksum == nullptr || lane_word == nullptr) return -3;
    if ((width_bytes != 4 && width_bytes != 8 && width_bytes != 16) || warps < 1 || warps > 8 || iters < 64 ||
        iters > 65536 || iters % 64 != 0)
        return -7;
    LaneWords lw;
    for (int l = 0; l < 32; ++l) {
        if (lane_word[l] < 0 || lane_word[l] >= 2048 || lane_word[l] % (width_bytes / 4) != 0) return -7;
        lw.w[l] = lane_word[l];
    }
    return run_probe(
        [&](long long *d) {
            if (width_bytes == 4) bank_pattern_kernel<4><<<1, 32 * warps>>>(lw, iters, d);
            else if (width_bytes == 8) bank_pattern_kernel<8><<<1, 32 * warps>>>(lw, iters, d);
            else bank_pattern_kernel<16><<<1, 32 * warps>>>(lw, iters, d);
        },
        warps, iters, cycles_per_access, checksum);
}

extern "C" int smem_bank_stride_probe(int stride, int op, int warps, int iters, double *cycles_per_access,
                                      long long *checksum) {
    if (cycles_per_access == nullptr || checksum == nullptr) return -3;
    if (stride < 1 || stride > 64 || (op != 0 && op != 1) || warps < 1 || warps > 8 || iters < 64 ||
        iters > 65536 || iters % 64 != 0)
        return -7;
    return run_probe(
        [&](long long *d) {
            if (op == 0) bank_stride_kernel<0><<<1, 32 * warps>>>(stride, iters, d);
            else bank_stride_kernel<1><<<1, 32 * warps>>>(stride, iters, d);
        },
        warps, iters, cycles_per_access, checksum);
}
