// alu_throughput.cu -- per-SM throughput probes for the arithmetic of the
// decode inner loops on GB300 (run: nvcc -gencode arch=compute_103a,code=sm_103a
// -O3 -o alu_throughput alu_throughput.cu && ./alu_throughput).
//
// Each kernel runs one CTA of 1024 threads per SM; thread 0 reads clock64()
// around an unrolled loop of independent chains, so the result is lane-ops
// (or half2 units) per SM clock:
//   A/B/C  fp16->fp32 conversion then 7 packed / scalar / mixed-precision FMAs
//   D/E    packed fma.rn.f32x2 vs scalar FFMA alone
//   F/H    broadcast vs per-lane-distinct 16-byte shared-memory loads
//   conv<> conversion variants inside a 7-head packed-FMA loop
//   shfl   warp shuffles; int: shift/xor/and chains
#include <cuda_fp16.h>
#include <cstdio>
#include <cstdint>
#define G 7

#define ITERS1 2048


__device__ __forceinline__ unsigned long long f2u(float2 v) { return *reinterpret_cast<unsigned long long*>(&v); }
__device__ __forceinline__ float2 u2f(unsigned long long v) { return *reinterpret_cast<float2*>(&v); }
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)), "l"(f2u(c)));
  return u2f(d);
}

// A: cvt half2->float2 then G packed FMAs (q pair in registers)
__global__ void kA(const __half2* __restrict__ kin, const float2* __restrict__ qin, float* out, long long* cyc) {
  float2 q[G], acc[G];
  for (int h = 0; h < G; ++h) { q[h] = qin[h]; acc[h] = make_float2(0.f, 0.f); }
  __half2 kv[8];
  for (int i = 0; i < 8; ++i) kv[i] = kin[(threadIdx.x + i) & 255];
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS1; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 kf = __half22float2(kv[i]);
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = ffma2(q[h], kf, acc[h]);
    }
    kv[it & 7] = __hadd2(kv[it & 7], kv[(it + 1) & 7]);
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int h = 0; h < G; ++h) s += acc[h].x + acc[h].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// B: cvt then scalar FFMA (2 per head per half2)
__global__ void kB(const __half2* __restrict__ kin, const float2* __restrict__ qin, float* out, long long* cyc) {
  float2 q[G], acc[G];
  for (int h = 0; h < G; ++h) { q[h] = qin[h]; acc[h] = make_float2(0.f, 0.f); }
  __half2 kv[8];
  for (int i = 0; i < 8; ++i) kv[i] = kin[(threadIdx.x + i) & 255];
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS1; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 kf = __half22float2(kv[i]);
#pragma unroll
      for (int h = 0; h < G; ++h) { acc[h].x = fmaf(q[h].x, kf.x, acc[h].x); acc[h].y = fmaf(q[h].y, kf.y, acc[h].y); }
    }
    kv[it & 7] = __hadd2(kv[it & 7], kv[(it + 1) & 7]);
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int h = 0; h < G; ++h) s += acc[h].x + acc[h].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// C: mixed-precision scalar fma (f16 x f16 + f32), no conversion
__global__ void kC(const __half2* __restrict__ kin, const __half2* __restrict__ qin, float* out, long long* cyc) {
  __half2 q[G]; float2 acc[G];
  for (int h = 0; h < G; ++h) { q[h] = qin[h]; acc[h] = make_float2(0.f, 0.f); }
  __half2 kv[8];
  for (int i = 0; i < 8; ++i) kv[i] = kin[(threadIdx.x + i) & 255];
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS1; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      unsigned ku = *reinterpret_cast<unsigned*>(&kv[i]);
      unsigned short klo = ku & 0xffff, khi = ku >> 16;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        unsigned qu = *reinterpret_cast<unsigned*>(&q[h]);
        unsigned short qlo = qu & 0xffff, qhi = qu >> 16;
        asm volatile("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc[h].x) : "h"(qlo), "h"(klo));
        asm volatile("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc[h].y) : "h"(qhi), "h"(khi));
      }
    }
    kv[it & 7] = __hadd2(kv[it & 7], kv[(it + 1) & 7]);
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int h = 0; h < G; ++h) s += acc[h].x + acc[h].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// D: pure FFMA2 (no cvt) and E: pure FFMA
__global__ void kD(const float2* __restrict__ qin, float* out, long long* cyc) {
  float2 q[8], acc[8];
  for (int h = 0; h < 8; ++h) { q[h] = qin[h]; acc[h] = make_float2(0.f, 0.f); }
  float2 x = qin[threadIdx.x & 7];
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS1 * 8; ++it) {
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[h] = ffma2(q[h], x, acc[h]);
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int h = 0; h < 8; ++h) s += acc[h].x + acc[h].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}
__global__ void kE(const float2* __restrict__ qin, float* out, long long* cyc) {
  float q[16], acc[16];
  for (int h = 0; h < 16; ++h) { q[h] = qin[h / 2].x + h; acc[h] = 0.f; }
  float x = qin[threadIdx.x & 7].y;
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS1 * 8; ++it) {
#pragma unroll
    for (int h = 0; h < 16; ++h) acc[h] = fmaf(q[h], x, acc[h]);
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int h = 0; h < 16; ++h) s += acc[h];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// F: broadcast LDS.128 (all lanes same address) feeding 2 FFMA2 each
__global__ void kF(const float4* __restrict__ qin, float* out, long long* cyc) {
  __shared__ float4 sq[512];
  for (int i = threadIdx.x; i < 512; i += blockDim.x) sq[i] = qin[i];
  float2 acc[4] = {};
  float2 x = make_float2(1.0f + threadIdx.x, 2.0f);
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS1; ++it) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float4 v = sq[(it * 16 + j) & 511];
      acc[j & 3] = ffma2(make_float2(v.x, v.y), x, acc[j & 3]);
      acc[(j + 1) & 3] = ffma2(make_float2(v.z, v.w), x, acc[(j + 1) & 3]);
    }
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int h = 0; h < 4; ++h) s += acc[h].x + acc[h].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}
// H: per-lane-distinct LDS.128 (row stride 16 B, conflict-free), 2 FFMA2 each
__global__ void kH(const float4* __restrict__ qin, float* out, long long* cyc) {
  __shared__ float4 sq[2048];
  for (int i = threadIdx.x; i < 2048; i += blockDim.x) sq[i] = qin[i & 511];
  float2 acc[4] = {};
  float2 x = make_float2(1.0f + threadIdx.x, 2.0f);
  int lane = threadIdx.x & 31;
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS1; ++it) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float4 v = sq[((it * 16 + j) * 32 + lane) & 2047];
      acc[j & 3] = ffma2(make_float2(v.x, v.y), x, acc[j & 3]);
      acc[(j + 1) & 3] = ffma2(make_float2(v.z, v.w), x, acc[(j + 1) & 3]);
    }
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int h = 0; h < 4; ++h) s += acc[h].x + acc[h].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

int main_part1() {
  int nsm = 0; cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  const int threads = 1024;
  __half2* kin; float2* qin; float* out; long long* cyc;
  cudaMalloc(&kin, 256 * sizeof(__half2));
  cudaMalloc(&qin, 4096 * sizeof(float2));
  cudaMalloc(&out, (size_t)nsm * threads * sizeof(float));
  cudaMalloc(&cyc, nsm * sizeof(long long));
  cudaMemset(kin, 0x3c, 256 * sizeof(__half2));
  cudaMemset(qin, 0, 4096 * sizeof(float2));
  long long h[1024];
  auto report = [&](const char* name, double ops_per_thread) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("%s: error %s\n", name, cudaGetErrorString(e)); return; }
    cudaMemcpy(h, cyc, nsm * sizeof(long long), cudaMemcpyDeviceToHost);
    double mx = 0; for (int i = 0; i < nsm; ++i) mx = h[i] > mx ? h[i] : mx;
    printf("%-44s cycles %10.0f  ops/clk/SM %8.2f\n", name, mx, ops_per_thread * threads / mx);
  };
  for (int rep = 0; rep < 2; ++rep) {
    kA<<<nsm, threads>>>(kin, qin, out, cyc); report("A cvt+ffma2 (FMA lane-ops, G=7)", (double)ITERS1 * 8 * G * 2);
    kB<<<nsm, threads>>>(kin, qin, out, cyc); report("B cvt+ffma  (FMA lane-ops, G=7)", (double)ITERS1 * 8 * G * 2);
    kC<<<nsm, threads>>>(kin, (const __half2*)qin, out, cyc); report("C mixed f32.f16 fma (FMA lane-ops, G=7)", (double)ITERS1 * 8 * G * 2);
    kD<<<nsm, threads>>>(qin, out, cyc); report("D pure ffma2 (FMA lane-ops)", (double)ITERS1 * 8 * 8 * 2);
    kE<<<nsm, threads>>>(qin, out, cyc); report("E pure ffma (FMA lane-ops)", (double)ITERS1 * 8 * 16);
    kF<<<nsm, threads>>>((const float4*)qin, out, cyc); report("F bcast LDS.128 (LDS per clk/SM x32)", (double)ITERS1 * 16);
    kH<<<nsm, threads>>>((const float4*)qin, out, cyc); report("H distinct LDS.128 (LDS per clk/SM x32)", (double)ITERS1 * 16);
  }
  return 0;
}


#define ITERS2 1024


__device__ __forceinline__ unsigned long long f2u_b(float2 v) { return *reinterpret_cast<unsigned long long*>(&v); }
__device__ __forceinline__ float2 u2f_b(unsigned long long v) { return *reinterpret_cast<float2*>(&v); }

template <int MODE>
__device__ __forceinline__ float2 conv(uint32_t x) {
  if (MODE == 0) {  // __half22float2
    __half2 h = *reinterpret_cast<__half2*>(&x);
    return __half22float2(h);
  } else if (MODE == 1) {  // two scalar cvt
    __half2 h = *reinterpret_cast<__half2*>(&x);
    return make_float2(__low2float(h), __high2float(h));
  } else if (MODE == 2) {  // integer bit trick (value * 2^-112)
    uint32_t lo = ((x << 13) & 0x0FFFE000u) | ((x << 16) & 0x80000000u);
    uint32_t hi = ((x >> 3) & 0x0FFFE000u) | (x & 0x80000000u);
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
  } else if (MODE == 3) {  // mixed-precision add with -0
    float a, b;
    unsigned short l = x & 0xffff, h = x >> 16;
    asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(a) : "h"(l), "f"(-0.0f));
    asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(b) : "h"(h), "f"(-0.0f));
    return make_float2(a, b);
  } else {  // integer trick, sign-less magnitude only (lower bound on cost)
    uint32_t lo = (x << 13) & 0x0FFFE000u;
    uint32_t hi = (x >> 3) & 0x0FFFE000u;
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
  }
}

template <int MODE, int NG>
__global__ void kconv(const uint32_t* __restrict__ kin, const float2* __restrict__ qin, float* out, long long* cyc) {
  float2 q[NG > 0 ? NG : 1], acc[NG > 0 ? NG : 1];
  for (int h = 0; h < (NG > 0 ? NG : 1); ++h) { q[h] = qin[h]; acc[h] = make_float2(0.f, 0.f); }
  uint32_t kv[8];
  for (int i = 0; i < 8; ++i) kv[i] = kin[(threadIdx.x + i) & 255];
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS2; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 kf = conv<MODE>(kv[i]);
      if (NG > 0) {
#pragma unroll
        for (int h = 0; h < NG; ++h) acc[h] = ffma2(q[h], kf, acc[h]);
      } else {
        acc[0].x += kf.x; acc[0].y += kf.y;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) kv[i] += 0x00010001u;
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int h = 0; h < (NG > 0 ? NG : 1); ++h) s += acc[h].x + acc[h].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// SHFL throughput: 8 independent butterfly-adds per iteration
__global__ void kshfl(const float* __restrict__ in, float* out, long long* cyc) {
  float v[8];
  for (int i = 0; i < 8; ++i) v[i] = in[(threadIdx.x + i) & 255];
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS2; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], 1 << (i & 3));
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
  for (int i = 0; i < 8; ++i) s += v[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// integer LOP3/SHF throughput: 8 independent chains
__global__ void kint(const uint32_t* __restrict__ in, float* out, long long* cyc) {
  uint32_t v[8];
  for (int i = 0; i < 8; ++i) v[i] = in[(threadIdx.x + i) & 255];
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < ITERS2; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ((v[i] << 3) ^ (v[i] >> 5)) & (0x0FFFE000u | i);
  }
  __syncthreads();
  long long t1 = clock64();
  uint32_t s = 0;
  for (int i = 0; i < 8; ++i) s ^= v[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (float)s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

int main_part2() {
  int nsm = 0; cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  const int threads = 1024;
  uint32_t* kin; float2* qin; float* out; long long* cyc;
  cudaMalloc(&kin, 256 * sizeof(uint32_t));
  cudaMalloc(&qin, 4096 * sizeof(float2));
  cudaMalloc(&out, (size_t)nsm * threads * sizeof(float));
  cudaMalloc(&cyc, nsm * sizeof(long long));
  cudaMemset(kin, 0x3c, 256 * sizeof(uint32_t));
  cudaMemset(qin, 0, 4096 * sizeof(float2));
  long long h[1024];
  auto report = [&](const char* name, double per_thread, const char* unit) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("%s: error %s\n", name, cudaGetErrorString(e)); return; }
    cudaMemcpy(h, cyc, nsm * sizeof(long long), cudaMemcpyDeviceToHost);
    double mx = 0; for (int i = 0; i < nsm; ++i) mx = h[i] > mx ? h[i] : mx;
    double per_sm_clk = per_thread * threads / mx;
    printf("%-40s %8.2f %s/clk/SM   (SMSP clk per warp-unit %6.2f)\n", name, per_sm_clk, unit, 32.0 * 4.0 / per_sm_clk);
  };
  const double H2 = (double)ITERS2 * 8;  // half2 units per thread
  for (int rep = 0; rep < 2; ++rep) {
    kconv<0, G><<<nsm, threads>>>(kin, qin, out, cyc); report("cvt half22float2 + 7 ffma2", H2, "half2");
    kconv<1, G><<<nsm, threads>>>(kin, qin, out, cyc); report("cvt 2x scalar + 7 ffma2", H2, "half2");
    kconv<2, G><<<nsm, threads>>>(kin, qin, out, cyc); report("int trick + 7 ffma2", H2, "half2");
    kconv<3, G><<<nsm, threads>>>(kin, qin, out, cyc); report("mixed add + 7 ffma2", H2, "half2");
    kconv<4, G><<<nsm, threads>>>(kin, qin, out, cyc); report("int trick nosign + 7 ffma2", H2, "half2");
    kconv<0, 0><<<nsm, threads>>>(kin, qin, out, cyc); report("cvt half22float2 alone (+fadd)", H2, "half2");
    kconv<2, 0><<<nsm, threads>>>(kin, qin, out, cyc); report("int trick alone (+fadd)", H2, "half2");
    kconv<3, 0><<<nsm, threads>>>(kin, qin, out, cyc); report("mixed add alone (+fadd)", H2, "half2");
    kconv<0, 1><<<nsm, threads>>>(kin, qin, out, cyc); report("cvt half22float2 + 1 ffma2", H2, "half2");
    kconv<2, 1><<<nsm, threads>>>(kin, qin, out, cyc); report("int trick + 1 ffma2", H2, "half2");
    kconv<2, 4><<<nsm, threads>>>(kin, qin, out, cyc); report("int trick + 4 ffma2", H2, "half2");
    kconv<0, 4><<<nsm, threads>>>(kin, qin, out, cyc); report("cvt half22float2 + 4 ffma2", H2, "half2");
    kshfl<<<nsm, threads>>>((const float*)qin, out, cyc); report("shfl+fadd", (double)ITERS2 * 8, "shfl");
    kint<<<nsm, threads>>>(kin, out, cyc); report("shl/shr/xor/and chain (4 ops)", (double)ITERS2 * 8 * 4, "intop");
  }
  return 0;
}

int main() {
  main_part1();
  main_part2();
  return 0;
}
