// Shared-memory access-pattern probe (test infrastructure): launches one small
// kernel per lane->address pattern so ncu can count the wavefronts each
// 64-bit and 128-bit shared load needs.  The measured counts pin the oracle's
// bank model (tests/golden/lds_wavefronts_sm103.txt).  Every index is masked
// into the 16 KB shared array.
#include <cstdio>
#include <cuda_runtime.h>
__device__ __forceinline__ int pat(int P, int l) {
  switch (P) {
    case 0: return 0;            // all lanes one chunk
    case 1: return l;            // 32 distinct consecutive
    case 2: return l & 7;        // 8 distinct, repeated per quarter (B-read)
    case 3: return l >> 3;       // 4 distinct, quarter-uniform (A-read)
    case 4: return l & 3;        // 4 distinct, repeated
    case 5: return l >> 4;       // 2 distinct, half-uniform
    case 6: return l & 15;       // 16 distinct, repeated per half
    case 7: return l >> 2;       // 8 distinct, groups of 4 lanes
    case 8: return (l >> 3) * 8; // 4 distinct chunks 128 B apart (same banks)
    case 9: return (l & 1) * 8 + (l >> 3); // mixed
    // quarter-pairing discriminators: quarters q = l / 8 read chunk sets
    case 10: return (l >> 4) * 4 + (l & 3);                      // q0=q1, q2=q3
    case 11: return ((l >> 3) & 1) * 4 + (l & 3);                // q0=q2, q1=q3
    case 12: return (((l >> 3) & 1) ^ (l >> 4)) * 4 + (l & 3);   // q0=q3, q1=q2
    case 13: return 2 * ((l >> 3) & 1) + ((l & 7) >> 2);         // a lane-grid row map
    case 14: return 4 * (((l >> 3) & 1) ^ (l >> 4)) + (l & 3);   // a lane-grid column map
    case 15: return l >> 1;                                      // 16 distinct, lane pairs
    case 16: return (l >> 4) * 8 + (l & 7);                      // halves on different chunk octets
    case 17: return ((l >> 3) & 1) * 8 + (l & 7);                // q0=q2, q1=q3 (8 chunks each)
    case 18: return (l & 3) + 4 * ((l >> 4) & 1) + 8 * ((l >> 2) & 1);  // mixed low bits
    case 19: return (l >> 2) & 3;                                // 4 distinct, groups of 4, repeating per half
    // 2 x 2 lane quads: rows paired / cols alternating, and the reverse
    case 20: return (l & 1) + 2 * (l >> 2);                      // alternating inside each quad
    case 21: return 2 * (l >> 4) + ((l & 3) >> 1);               // grid G2 row read
    case 22: return 2 * ((l >> 2) & 3) + (l & 1);                // grid G2 column read
    case 23: return 2 * (l >> 4) + (l & 1);                      // grid G3 row read
    case 24: return 2 * ((l >> 2) & 3) + ((l & 3) >> 1);         // grid G3 column read
    case 25: return ((l >> 1) & 1) + 2 * (l >> 3) + 8 * (l & 1); // pairs split across octets
    default: return 0;
  }
}
template <int P>
__global__ void lds128_probe(float *out, int iters) {
  __shared__ float4 s[1024];
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) s[i] = make_float4(i, i + 1, i + 2, i + 3);
  __syncthreads();
  const int l = threadIdx.x & 31;
  const int idx = pat(P, l);
  float4 acc = make_float4(0, 0, 0, 0);
  for (int it = 0; it < iters; ++it) {
    const float4 v = s[(idx + 32 * it) & 1023];
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc.x + acc.y + acc.z + acc.w;
}
template <int P>
__global__ void lds64_probe(float *out, int iters) {
  __shared__ float2 s[2048];
  for (int i = threadIdx.x; i < 2048; i += blockDim.x) s[i] = make_float2(i, i + 1);
  __syncthreads();
  const int l = threadIdx.x & 31;
  const int idx = pat(P, l);
  float2 acc = make_float2(0, 0);
  for (int it = 0; it < iters; ++it) {
    const float2 v = s[(idx + 32 * it) & 2047];
    acc.x += v.x; acc.y += v.y;
  }
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc.x + acc.y;
}
// 32-bit accesses s[lane * STRIDE] (the bank page's stride law: a full warp
// touches 32/gcd(stride,32) banks, conflict degree gcd(stride,32)).
template <int STRIDE>
__global__ void lds32_stride_probe(float *out, int iters) {
  __shared__ float s[4096];
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) s[i] = i;
  __syncthreads();
  const int l = threadIdx.x & 31;
  float acc = 0.0f;
  for (int it = 0; it < iters; ++it) acc += s[(l * STRIDE + 32 * (it & 63)) & 4095];
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}
template <int STRIDE>
__global__ void sts32_stride_probe(float *out, int iters) {
  __shared__ float s[4096];
  const int l = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  for (int it = 0; it < iters; ++it) s[(l * STRIDE + 32 * ((it + w) & 63)) & 4095] = float(it);
  __syncthreads();
  out[blockIdx.x * blockDim.x + threadIdx.x] = s[threadIdx.x];
}
// The sgemm kernel's A transpose, in isolation: each warp reads 32 consecutive
// rows of a 128 x 16 tile stored with the 64-byte XOR swizzle (16-byte
// groups g at g ^ ((row >> 1) & 3)) and writes the 4 components to a k-major
// 16 x 128 tile (32 consecutive words per store).  Two raw tiles and two
// k-major tiles rotate; the accesses are inline PTX so none is merged or
// hoisted.
__global__ void xpose_probe(float *out, int iters) {
  __shared__ __align__(16) float raw[2][128 * 16];
  __shared__ __align__(16) float kmaj[2][16 * 128];
  for (int i = threadIdx.x; i < 2 * 2048; i += blockDim.x) (&raw[0][0])[i] = i;
  __syncthreads();
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int m = 32 * (w & 3) + l;
  float acc = 0.0f;
  for (int it = 0; it < iters; ++it) {
    const int k = 8 * (w >> 2) + 4 * (it & 1);
    const unsigned src = static_cast<unsigned>(__cvta_generic_to_shared(
        &raw[(it >> 1) & 1][m * 16 + 4 * ((k >> 2) ^ ((m >> 1) & 3))]));
    float x, y, z, v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x), "=f"(y), "=f"(z), "=f"(v) : "r"(src));
    const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(&kmaj[(it >> 2) & 1][k * 128 + m]));
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst), "f"(x) : "memory");
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + 512), "f"(y) : "memory");
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + 1024), "f"(z) : "memory");
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + 1536), "f"(v) : "memory");
    acc += x;
  }
  __syncthreads();
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc + kmaj[0][threadIdx.x];
}

template <int S>
void run_strides(float *out, int iters) {
  if constexpr (S <= 33) {
    lds32_stride_probe<S><<<152, 256>>>(out, iters);
    sts32_stride_probe<S><<<152, 256>>>(out, iters);
    run_strides<S + 1>(out, iters);
  }
}

int main() {
  float *out;
  cudaMalloc(&out, 1024 * 256 * sizeof(float));
  const int iters = 4096;
#define RUN(P) lds128_probe<P><<<152, 256>>>(out, iters); lds64_probe<P><<<152, 256>>>(out, iters);
  RUN(0) RUN(1) RUN(2) RUN(3) RUN(4) RUN(5) RUN(6) RUN(7) RUN(8) RUN(9)
  RUN(10) RUN(11) RUN(12) RUN(13) RUN(14) RUN(15) RUN(16) RUN(17) RUN(18) RUN(19)
  RUN(20) RUN(21) RUN(22) RUN(23) RUN(24) RUN(25)
  run_strides<1>(out, iters);
  xpose_probe<<<152, 256>>>(out, iters);
  cudaError_t e = cudaDeviceSynchronize();
  printf("probe done: %s\n", cudaGetErrorString(e));
  cudaFree(out);
  return e == cudaSuccess ? 0 : 1;
}
