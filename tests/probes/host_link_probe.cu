// Host<->device link probe (test infrastructure): how fast 64 MiB moves
// between pinned host memory and the device by each available route --
// cudaMemcpyAsync split over 1, 2 or 4 streams in each direction, both
// directions at once, and a grid-stride copy kernel that reads or writes the
// pinned buffer through its mapped device pointer.  Best of 5 timed
// repetitions after one warm-up, CUDA events.  Indices stay below the 64 MiB
// of every buffer (grid-stride loop over bytes / 16 float4 elements).
#include <cstdio>
#include <cuda_runtime.h>
#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("%s failed: %s\n", #x, cudaGetErrorString(e)); return 1; } } while (0)
__global__ void copy_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) dst[i] = src[i];
}
int main() {
  const size_t bytes = 64ull << 20;
  float *h_src, *h_dst, *d_a, *d_b;
  CK(cudaHostAlloc(&h_src, bytes, cudaHostAllocMapped));
  CK(cudaHostAlloc(&h_dst, bytes, cudaHostAllocMapped));
  CK(cudaMalloc(&d_a, bytes));
  CK(cudaMalloc(&d_b, bytes));
  for (size_t i = 0; i < bytes / 4; ++i) h_src[i] = (float)(i & 1023);
  float *h_src_dev, *h_dst_dev;
  CK(cudaHostGetDevicePointer(&h_src_dev, h_src, 0));
  CK(cudaHostGetDevicePointer(&h_dst_dev, h_dst, 0));
  cudaStream_t st[4];
  for (int i = 0; i < 4; ++i) CK(cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking));
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
  auto run_ce = [&](int nstreams, cudaMemcpyKind kind, const char *name) -> int {
    float best = 1e9;
    for (int rep = 0; rep < 6; ++rep) {
      CK(cudaDeviceSynchronize());
      CK(cudaEventRecord(e0, 0));
      for (int i = 0; i < nstreams; ++i) {
        CK(cudaStreamWaitEvent(st[i], e0, 0));
        size_t off = bytes / nstreams * i;
        if (kind == cudaMemcpyHostToDevice) CK(cudaMemcpyAsync((char *)d_a + off, (char *)h_src + off, bytes / nstreams, kind, st[i]));
        else CK(cudaMemcpyAsync((char *)h_dst + off, (char *)d_a + off, bytes / nstreams, kind, st[i]));
      }
      for (int i = 0; i < nstreams; ++i) { cudaEvent_t ev; CK(cudaEventCreate(&ev)); CK(cudaEventRecord(ev, st[i])); CK(cudaStreamWaitEvent(0, ev, 0)); CK(cudaEventDestroy(ev)); }
      CK(cudaEventRecord(e1, 0));
      CK(cudaEventSynchronize(e1));
      float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
      if (rep > 0 && ms < best) best = ms;
    }
    printf("%-34s %d streams: %.1f GB/s\n", name, nstreams, bytes / best / 1e6);
    return 0;
  };
  for (int n : {1, 2, 4}) if (run_ce(n, cudaMemcpyHostToDevice, "copy engine H2D")) return 1;
  for (int n : {1, 2, 4}) if (run_ce(n, cudaMemcpyDeviceToHost, "copy engine D2H")) return 1;
  // both directions at once, 2 streams each
  {
    float best = 1e9;
    for (int rep = 0; rep < 6; ++rep) {
      CK(cudaDeviceSynchronize());
      CK(cudaEventRecord(e0, 0));
      for (int i = 0; i < 4; ++i) CK(cudaStreamWaitEvent(st[i], e0, 0));
      CK(cudaMemcpyAsync(d_a, h_src, bytes / 2, cudaMemcpyHostToDevice, st[0]));
      CK(cudaMemcpyAsync((char *)d_a + bytes / 2, (char *)h_src + bytes / 2, bytes / 2, cudaMemcpyHostToDevice, st[1]));
      CK(cudaMemcpyAsync(h_dst, d_b, bytes / 2, cudaMemcpyDeviceToHost, st[2]));
      CK(cudaMemcpyAsync((char *)h_dst + bytes / 2, (char *)d_b + bytes / 2, bytes / 2, cudaMemcpyDeviceToHost, st[3]));
      for (int i = 0; i < 4; ++i) { cudaEvent_t ev; CK(cudaEventCreate(&ev)); CK(cudaEventRecord(ev, st[i])); CK(cudaStreamWaitEvent(0, ev, 0)); CK(cudaEventDestroy(ev)); }
      CK(cudaEventRecord(e1, 0));
      CK(cudaEventSynchronize(e1));
      float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
      if (rep > 0 && ms < best) best = ms;
    }
    printf("%-34s both ways, 2+2 streams: %.1f GB/s total\n", "copy engines", 2 * bytes / best / 1e6);
  }
  // SM-driven copies through the mapped pointers
  for (int blocks : {152, 304, 608, 1216}) {
    for (int dir = 0; dir < 2; ++dir) {
      float best = 1e9;
      for (int rep = 0; rep < 6; ++rep) {
        CK(cudaEventRecord(e0, 0));
        if (dir == 0) copy_kernel<<<blocks, 256>>>((const float4 *)h_src_dev, (float4 *)d_a, bytes / 16);
        else copy_kernel<<<blocks, 256>>>((const float4 *)d_a, (float4 *)h_dst_dev, bytes / 16);
        CK(cudaGetLastError());
        CK(cudaEventRecord(e1, 0));
        CK(cudaEventSynchronize(e1));
        float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
        if (rep > 0 && ms < best) best = ms;
      }
      printf("SM copy kernel %s, %4d blocks x 256: %.1f GB/s\n", dir == 0 ? "H2D" : "D2H", blocks, bytes / best / 1e6);
    }
  }
  CK(cudaMemcpy(h_dst, d_a, 64, cudaMemcpyDeviceToHost));
  printf("check %f %f\n", h_dst[5], h_dst[15]);
  return 0;
}
