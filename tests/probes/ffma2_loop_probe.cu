// ffma2_loop_probe.cu -- throughput ceiling of the CUDA-core inner loop on
// GB300 (sm_103a): packed FP32 FMAs (fma.rn.f32x2) alone, and with the
// 128-bit shared-memory fragment reads that feed them, for three per-thread
// register tiles.  No global traffic, no barrier in the loop: what is left
// is the FMA pipe, the issue slots and the shared-memory reads.
//
// Build and run (GB300):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 tests/probes/ffma2_loop_probe.cu -o _build_probe/ffma2_loop_probe
//   _build_probe/ffma2_loop_probe
//
// Every shared-memory index stays below the allocation (16384 floats) and
// every output index below blocks x threads; see the bounds noted per kernel.
#include <cuda_runtime.h>

#include <cstdio>

constexpr int kFloats = 16384;  // dynamic shared memory of every probe: 64 KiB

// TM x TN register tile per thread, NT threads.  Per k step a thread reads
// TM/4 + TN/4 float4 fragments (LOADS) or none, then issues TM * TN / 2
// packed FMAs, column pair by column pair.
//   A reads: index (it&1)*4096 + k*256 + ra + 32q + c <= 4096 + 3840 + 28 + 96 + 3 = 8063
//   B reads: 8192 + (it&1)*4096 + k*256 + cb + 32q + c <= 12288 + 3840 + 28 + 96 + 3 = 16255
template <int TM, int TN, int NT, bool LOADS>
__global__ void __launch_bounds__(NT) probe(float *out, int iters) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x, l = tid & 31;
    for (int i = tid; i < kFloats; i += NT) sm[i] = 1.0f + 1e-7f * static_cast<float>(i);
    __syncthreads();
    float2 acc[TM][TN / 2];
#pragma unroll
    for (int r = 0; r < TM; ++r)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[r][j] = make_float2(0.0f, 0.0f);
    // quads of lanes share A (rows) or B (cols) fragments, as in the kernel's 4 x 8 lane grid
    const int ra = 4 * (l & 7), cb = 4 * (l >> 2);
    float a[TM], b[TN];
#pragma unroll
    for (int i = 0; i < TM; ++i) a[i] = 1.0f + 1e-6f * static_cast<float>(tid + i);
#pragma unroll
    for (int i = 0; i < TN; ++i) b[i] = 1.0f - 1e-6f * static_cast<float>(tid + i);
    for (int it = 0; it < iters; ++it) {
        const float *A = sm + (it & 1) * 4096;
        const float *B = sm + 8192 + (it & 1) * 4096;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (LOADS) {
#pragma unroll
                for (int q = 0; q < TM / 4; ++q) {
                    const float4 v = *reinterpret_cast<const float4 *>(A + k * 256 + ra + 32 * q);
                    a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
                }
#pragma unroll
                for (int q = 0; q < TN / 4; ++q) {
                    const float4 v = *reinterpret_cast<const float4 *>(B + k * 256 + cb + 32 * q);
                    b[4 * q] = v.x; b[4 * q + 1] = v.y; b[4 * q + 2] = v.z; b[4 * q + 3] = v.w;
                }
            }
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) {
                const float2 bp = make_float2(b[2 * j], b[2 * j + 1]);
#pragma unroll
                for (int r = 0; r < TM; ++r) acc[r][j] = __ffma2_rn(make_float2(a[r], a[r]), bp, acc[r][j]);
            }
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int r = 0; r < TM; ++r)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) s += acc[r][j].x + acc[r][j].y;
    out[blockIdx.x * NT + tid] = s;
}

template <int TM, int TN, int NT, bool LOADS>
void measure(const char *name, int sms, int per_sm, float *out, size_t out_floats) {
    auto kern = probe<TM, TN, NT, LOADS>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kFloats * 4);
    const int blocks = sms * per_sm * 4, iters = 2000;
    if (static_cast<size_t>(blocks) * NT > out_floats) {
        printf("%s: output buffer too small, skipped\n", name);
        return;
    }
    kern<<<blocks, NT, kFloats * 4>>>(out, iters);  // warm-up
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    float ms = 1e30f;
    for (int rep = 0; rep < 5; ++rep) {  // best of 5
        cudaEventRecord(e0);
        kern<<<blocks, NT, kFloats * 4>>>(out, iters);
        cudaEventRecord(e1);
        if (cudaEventSynchronize(e1) != cudaSuccess) {
            printf("%s: %s\n", name, cudaGetErrorString(cudaGetLastError()));
            return;
        }
        float t = 0.0f;
        cudaEventElapsedTime(&t, e0, e1);
        ms = t < ms ? t : ms;
    }
    const double flop = 2.0 * blocks * NT * static_cast<double>(iters) * 16 * TM * TN;
    const double tflops = flop / (ms * 1e-3) / 1e12;
    const double peak = sms * 128.0 * 2 * 2.07e9 / 1e12;
    printf("%-44s %d CTAs/SM requested: %6.2f TFLOP/s = %5.1f %% of %.2f (2070 MHz), best of 5\n", name, per_sm, tflops,
           100.0 * tflops / peak, peak);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
}

int main() {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    const size_t out_floats = static_cast<size_t>(sms) * 3 * 4 * 256;  // largest grid: 3 per SM x 4 waves x 256 threads
    float *out = nullptr;
    if (cudaMalloc(&out, out_floats * sizeof(float)) != cudaSuccess) return 1;
    // bring the SM clock up before the first measurement (about half a second of FMA work)
    cudaFuncSetAttribute(probe<8, 8, 256, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFloats * 4);
    for (int i = 0; i < 20; ++i) probe<8, 8, 256, false><<<sms * 8, 256, kFloats * 4>>>(out, 2000);
    cudaDeviceSynchronize();
    measure<8, 8, 256, false>("8x8 tile, 256 threads, FFMA2 only", sms, 2, out, out_floats);
    measure<8, 8, 256, true>("8x8 tile, 256 threads, 4 LDS.128 + 32 FFMA2", sms, 2, out, out_floats);
    measure<8, 16, 128, true>("8x16 tile, 128 threads, 6 LDS.128 + 64 FFMA2", sms, 3, out, out_floats);
    measure<16, 8, 128, true>("16x8 tile, 128 threads, 6 LDS.128 + 64 FFMA2", sms, 3, out, out_floats);
    cudaFree(out);
    return 0;
}
