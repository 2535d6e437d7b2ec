// Shared-store contention probe (test infrastructure): runs the tiled FP32
// matrix multiply's A transpose (32 consecutive rows read from the 64-byte
// swizzled raw tile, four 32-bit stores of 32 consecutive words each to the
// k-major tile; one wavefront per store by the bank rule) in warps 0-7,
// while warp 8 keeps a second client of shared memory busy on a separate
// region:
//   mode 0  nothing (the transpose alone);
//   mode 1  bulk tensor-engine copies (cp.async.bulk, 8 KiB each, from L2);
//   mode 2  per-lane 16-byte cp.async copies (8 KiB per round);
//   mode 3  128-bit loads of 32 distinct chunks (4 wavefronts each).
// ncu then shows whether the store counters (wavefronts and "bank
// conflicts") of the same conflict-free stores change with the other client.
//
// frag_contention_probe does the same for the kernel's fragment loads: warps
// 0-7 read a k-major 16 x 128 A tile and a 16 x 128 B tile with the kernel's
// lane grid (per k step two 128-bit A reads at rows 4*lr and 16 + 4*lr of the
// warp's 32 rows, two 128-bit B reads at columns 4*lc and 32 + 4*lc of its
// 64 columns; lr = 2*(lane/16) + lane%2, lc = 2*((lane/4)%4) + (lane%4)/2),
// 2 wavefronts per load by the measured bank model, while warp 8 runs mode
// 0, 1 or 2 above.
//
// Bounds: raw, kmaj and fill are indexed below their sizes (row m < 128,
// k + 3 < 16, fill offsets < 2048 floats; fragment reads: k < 16, row + 3 <
// 128, column + 3 < 128); the source buffer holds 2048 floats.  Warp 8 stops when warps 0-7 have all finished or after
// kFillLimit rounds; every mbarrier wait gives up after kPollLimit polls and
// records it in the status word.
#include <cstdio>
#include <cuda_runtime.h>

constexpr int kFillFloats = 2048;  // 8 KiB
constexpr unsigned kFillLimit = 1u << 20;
constexpr unsigned kPollLimit = 1u << 20;

__device__ unsigned g_status;

__device__ __forceinline__ unsigned smem_addr(const void *p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

// Warp 8's work: keeps the second client of shared memory busy until
// *done reaches 8 (or kFillLimit rounds).
template <int MODE>
__device__ __forceinline__ float fill_until_done(const float *src, float *fill, unsigned long long *bar,
                                                 unsigned *done, int l) {
  float acc = 0.0f;
  unsigned rounds = 0, phase = 0;
  for (;;) {
    // one decision per warp (lane 0's view of the counter), so the
    // warp-wide shuffle below is reached by every lane or by none
    unsigned go = *static_cast<volatile unsigned *>(done) < 8u && rounds < kFillLimit;
    if (!__shfl_sync(0xffffffffu, go, 0)) break;
    ++rounds;
    if constexpr (MODE == 1) {
      if (l == 0) {
        const unsigned b = smem_addr(bar);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(kFillFloats * 4)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_addr(fill)),
            "l"(src), "r"(kFillFloats * 4), "r"(b)
            : "memory");
        unsigned polls = 0, ok = 0;
        while (!ok) {
          asm volatile(
              "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, "
              "p;\n}\n"
              : "=r"(ok)
              : "r"(b), "r"(phase)
              : "memory");
          if (!ok && ++polls > kPollLimit) {
            atomicOr(&g_status, 1u);
            break;
          }
        }
        phase ^= 1u;
        if (!ok) rounds = kFillLimit;  // stop filling after a lost wait
      }
      rounds = __shfl_sync(0xffffffffu, rounds, 0);
    } else if constexpr (MODE == 2) {
#pragma unroll
      for (int c = 0; c < kFillFloats / 128; ++c) {
        const int off = 128 * c + 4 * l;  // < 2048
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(&fill[off])), "l"(src + off)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    } else if constexpr (MODE == 3) {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const unsigned s = smem_addr(&fill[(128 * c + 4 * l) & (kFillFloats - 1)]);
        float x, y, z, v;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x), "=f"(y), "=f"(z), "=f"(v) : "r"(s));
        acc += x + y + z + v;
      }
    }
  }
  return acc;
}

template <int MODE>
__global__ void __launch_bounds__(288) xpose_contention_probe(const float *src, float *out, int iters) {
  __shared__ __align__(128) float raw[2][128 * 16];
  __shared__ __align__(128) float kmaj[2][16 * 128];
  __shared__ __align__(128) float fill[kFillFloats];
  __shared__ __align__(8) unsigned long long bar;
  __shared__ unsigned done;
  for (int i = threadIdx.x; i < 2 * 2048; i += blockDim.x) (&raw[0][0])[i] = i;
  for (int i = threadIdx.x; i < kFillFloats; i += blockDim.x) fill[i] = 0.0f;
  if (threadIdx.x == 0) {
    done = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  float acc = 0.0f;
  if (w < 8) {
    const int m = 32 * (w & 3) + l;
    for (int it = 0; it < iters; ++it) {
      const int k = 8 * (w >> 2) + 4 * (it & 1);
      const unsigned s = smem_addr(&raw[(it >> 1) & 1][m * 16 + 4 * ((k >> 2) ^ ((m >> 1) & 3))]);
      float x, y, z, v;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x), "=f"(y), "=f"(z), "=f"(v) : "r"(s));
      const unsigned d = smem_addr(&kmaj[(it >> 2) & 1][k * 128 + m]);
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(d), "f"(x) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(d + 512), "f"(y) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(d + 1024), "f"(z) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(d + 1536), "f"(v) : "memory");
      acc += x;
    }
    __syncwarp();
    if (l == 0) atomicAdd(&done, 1u);
  } else if (MODE != 0) {
    acc += fill_until_done<MODE>(src, fill, &bar, &done, l);
  }
  __syncthreads();
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc + kmaj[0][threadIdx.x & 2047] + fill[threadIdx.x];
}

template <int MODE>
__global__ void __launch_bounds__(288) frag_contention_probe(const float *src, float *out, int iters) {
  __shared__ __align__(128) float at[16 * 128];  // k-major A tile: (k, m) at k*128 + m
  __shared__ __align__(128) float bt[16 * 128];  // B tile: (k, n) at k*128 + n
  __shared__ __align__(128) float fill[kFillFloats];
  __shared__ __align__(8) unsigned long long bar;
  __shared__ unsigned done;
  for (int i = threadIdx.x; i < 2048; i += blockDim.x) {
    at[i] = i;
    bt[i] = -i;
  }
  for (int i = threadIdx.x; i < kFillFloats; i += blockDim.x) fill[i] = 0.0f;
  if (threadIdx.x == 0) {
    done = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  float acc = 0.0f;
  if (w < 8) {
    const int lr = 2 * (l >> 4) + (l & 1), lc = 2 * ((l >> 2) & 3) + ((l & 3) >> 1);
    const int r0 = 32 * (w / 2) + 4 * lr;   // < 128 - 19
    const int c0 = 64 * (w % 2) + 4 * lc;   // < 128 - 35
    for (int it = 0; it < iters; ++it) {
      const int k = it & 15;
      float x0, y0, z0, v0, x1, y1, z1, v1, x2, y2, z2, v2, x3, y3, z3, v3;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x0), "=f"(y0), "=f"(z0), "=f"(v0)
                   : "r"(smem_addr(&at[k * 128 + r0])));
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x1), "=f"(y1), "=f"(z1), "=f"(v1)
                   : "r"(smem_addr(&at[k * 128 + r0 + 16])));
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x2), "=f"(y2), "=f"(z2), "=f"(v2)
                   : "r"(smem_addr(&bt[k * 128 + c0])));
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x3), "=f"(y3), "=f"(z3), "=f"(v3)
                   : "r"(smem_addr(&bt[k * 128 + c0 + 32])));
      acc += x0 * x2 + y0 * y2 + z0 * z2 + v0 * v2 + x1 * x3 + y1 * y3 + z1 * z3 + v1 * v3;
    }
    __syncwarp();
    if (l == 0) atomicAdd(&done, 1u);
  } else if (MODE != 0) {
    acc += fill_until_done<MODE>(src, fill, &bar, &done, l);
  }
  __syncthreads();
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc + fill[threadIdx.x];
}

int main() {
  float *src = nullptr, *out = nullptr;
  if (cudaMalloc(&src, kFillFloats * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&out, 152 * 288 * sizeof(float)) != cudaSuccess) {
    printf("allocation failed\n");
    return 1;
  }
  cudaMemset(src, 0, kFillFloats * sizeof(float));
  const int iters = 4096;
  xpose_contention_probe<0><<<152, 288>>>(src, out, iters);
  xpose_contention_probe<1><<<152, 288>>>(src, out, iters);
  xpose_contention_probe<2><<<152, 288>>>(src, out, iters);
  xpose_contention_probe<3><<<152, 288>>>(src, out, iters);
  frag_contention_probe<0><<<152, 288>>>(src, out, iters);
  frag_contention_probe<1><<<152, 288>>>(src, out, iters);
  frag_contention_probe<2><<<152, 288>>>(src, out, iters);
  cudaError_t e = cudaDeviceSynchronize();
  unsigned status = 0;
  cudaMemcpyFromSymbol(&status, g_status, sizeof(status));
  printf("probe done: %s, wait status %u\n", cudaGetErrorString(e), status);
  cudaFree(src);
  cudaFree(out);
  return (e == cudaSuccess && status == 0) ? 0 : 1;
}
