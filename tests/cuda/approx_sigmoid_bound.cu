// Test program: the largest |approx_sigmoid(x) - spec_sigmoid(x)| over every FP32 bit
// pattern, and the number of inputs where exactly one of the two is NaN. The top-K
// candidate search assumes the former stays below kApproxErr. Prints one line:
// "<max error> <kApproxErr> <nan mismatches>".
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "topk.cuh"

using namespace moe::topk_impl;

__global__ void sweep(unsigned long long base, unsigned int* max_bits, unsigned int* nan_mismatch) {
  const unsigned long long i = base + (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i > 0xFFFFFFFFull) return;
  const float x = __uint_as_float((unsigned int)i);
  const float a = approx_sigmoid(x), s = spec_sigmoid(x);
  if ((a != a) != (s != s)) {
    atomicAdd(nan_mismatch, 1u);
    return;
  }
  if (s != s) return;
  atomicMax(max_bits, __float_as_uint(fabsf(a - s)));
}

int main() {
  unsigned int* d = nullptr;
  if (cudaMalloc(&d, 8) != cudaSuccess || cudaMemset(d, 0, 8) != cudaSuccess) return 2;
  const unsigned long long per = 1ull << 30;
  for (unsigned long long b = 0; b < (1ull << 32); b += per) sweep<<<(unsigned)(per / 256), 256>>>(b, d, d + 1);
  unsigned int h[2];
  if (cudaMemcpy(h, d, 8, cudaMemcpyDeviceToHost) != cudaSuccess) return 3;
  float err;
  std::memcpy(&err, &h[0], sizeof(err));
  printf("%.9g %.9g %u\n", (double)err, (double)kApproxErr, h[1]);
  return 0;
}
