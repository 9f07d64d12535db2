// Seeded synthetic inputs, GPU side: the same draws as synth_host.c, bit for bit.
//
// Only random numbers live here (no MoE arithmetic).  The definition is
// repeated from synth_host.c: SplitMix64 as a counter-based generator, twelve
// 24-bit uniforms per element summed and centred (Irwin-Hall, n = 12), one
// rounded double multiply by the column scale, one rounding to the storage
// type (nearest-even).  Used to create multi-gigabyte expert weights directly
// in device memory.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ULL;

__host__ __device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + kGolden;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__global__ void fill_kernel(void* out, int dtype, uint64_t first, uint64_t n, uint64_t key,
                            double sigma, const double* __restrict__ scale, uint64_t ncols) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n; q += stride) {
    uint64_t i = first + q;
    uint64_t base = key + 12ULL * i;
    int64_t acc = 0;
#pragma unroll
    for (int j = 0; j < 12; ++j) acc += (int64_t)(splitmix64(base + (uint64_t)j) >> 40);
    double z = (double)(acc - 6LL * 16777216LL) * (1.0 / 16777216.0);
    double s = scale ? scale[i % ncols] : sigma;
    double v = __dmul_rn(z, s);
    if (dtype == 0) static_cast<float*>(out)[q] = __double2float_rn(v);
    else static_cast<__half*>(out)[q] = __double2half(v);
  }
}

}  // namespace

extern "C" int synth_cuda_fill(void* out, int dtype, uint64_t first, uint64_t n, uint64_t seed,
                               uint64_t tid, double sigma, const double* scale_dev, uint64_t ncols,
                               cudaStream_t stream) {
  if (n == 0) return 0;
  if (!out || (dtype != 0 && dtype != 1) || (scale_dev && ncols == 0)) return 1;
  uint64_t key = splitmix64(splitmix64(seed) ^ (tid * kGolden));
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (n + 255) / 256;
  uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(out, dtype, first, n, key, sigma, scale_dev, ncols);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
