// h2d_transport.cu -- host->device bandwidth on a Grace-Blackwell node, for the
// end-to-end leg (inputs copied from pinned host memory every step).  Measures
// cudaMemcpyAsync from pinned memory on 1 and on 4 streams, a kernel reading
// pinned mapped host memory directly (zero-copy, 16-byte loads) and a kernel
// copying it into device memory.  2 GiB per transfer, CUDA events.
// Run: nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o h2d_transport
//      h2d_transport.cu && ./h2d_transport
#include <cstdio>
#include <cstring>
#include <cstdint>
#include <vector>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("err %s line %d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

__global__ void read_sum(const uint4* __restrict__ src, size_t n16, uint4* __restrict__ dst) {
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  size_t stride = (size_t)gridDim.x * blockDim.x;
  uint4 acc = make_uint4(0, 0, 0, 0);
  for (; i < n16; i += stride) {
    uint4 v = src[i];
    acc.x ^= v.x; acc.y ^= v.y; acc.z ^= v.z; acc.w ^= v.w;
  }
  if (acc.x == 0x12345678u) dst[0] = acc;  // keep the loads alive
}

__global__ void copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16) {
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n16; i += stride) dst[i] = src[i];
}

int main() {
  const size_t bytes = (size_t)2 << 30;  // 2 GiB
  void *h = nullptr, *d = nullptr, *dd = nullptr;
  CK(cudaHostAlloc(&h, bytes, cudaHostAllocMapped));
  CK(cudaMalloc(&d, bytes));
  CK(cudaMalloc(&dd, 64));
  memset(h, 1, bytes);
  cudaStream_t s[4];
  for (int i = 0; i < 4; ++i) CK(cudaStreamCreateWithFlags(&s[i], cudaStreamNonBlocking));
  cudaEvent_t a, b;
  CK(cudaEventCreate(&a)); CK(cudaEventCreate(&b));
  float ms;
  // 1 stream
  for (int rep = 0; rep < 3; ++rep) {
    CK(cudaEventRecord(a, s[0]));
    CK(cudaMemcpyAsync(d, h, bytes, cudaMemcpyHostToDevice, s[0]));
    CK(cudaEventRecord(b, s[0]));
    CK(cudaEventSynchronize(b));
    CK(cudaEventElapsedTime(&ms, a, b));
    printf("memcpy 1 stream: %.1f GB/s\n", bytes / (ms * 1e-3) / 1e9);
  }
  // 4 streams, quarter each
  for (int rep = 0; rep < 3; ++rep) {
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(a, 0));
    for (int i = 0; i < 4; ++i)
      CK(cudaMemcpyAsync((char*)d + i * (bytes / 4), (char*)h + i * (bytes / 4), bytes / 4,
                         cudaMemcpyHostToDevice, s[i]));
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(b, 0));
    CK(cudaEventSynchronize(b));
    CK(cudaEventElapsedTime(&ms, a, b));
    printf("memcpy 4 streams: %.1f GB/s\n", bytes / (ms * 1e-3) / 1e9);
  }
  void* hd = nullptr;
  CK(cudaHostGetDevicePointer(&hd, h, 0));
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  for (int blocks_per_sm : {4, 8, 16}) {
    for (int rep = 0; rep < 2; ++rep) {
      CK(cudaEventRecord(a, s[0]));
      read_sum<<<sms * blocks_per_sm, 256, 0, s[0]>>>((const uint4*)hd, bytes / 16, (uint4*)dd);
      CK(cudaGetLastError());
      CK(cudaEventRecord(b, s[0]));
      CK(cudaEventSynchronize(b));
      CK(cudaEventElapsedTime(&ms, a, b));
      printf("zero-copy read (%d CTAs/SM x 256): %.1f GB/s\n", blocks_per_sm, bytes / (ms * 1e-3) / 1e9);
    }
  }
  for (int rep = 0; rep < 2; ++rep) {
    CK(cudaEventRecord(a, s[0]));
    copy_kernel<<<sms * 8, 256, 0, s[0]>>>((const uint4*)hd, (uint4*)d, bytes / 16);
    CK(cudaGetLastError());
    CK(cudaEventRecord(b, s[0]));
    CK(cudaEventSynchronize(b));
    CK(cudaEventElapsedTime(&ms, a, b));
    printf("copy kernel host->device: %.1f GB/s\n", bytes / (ms * 1e-3) / 1e9);
  }
  printf("done\n");
  return 0;
}
