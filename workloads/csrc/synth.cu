// Seeded synthetic inputs for the paged-attention workloads.
//
// This file is the input generator only.  It knows nothing of attention,
// block tables or slots: it writes pseudo-random fp16 values into flat arrays
// indexed by their plain linear element index.  The same function is
// provided twice, once for the host (OpenMP loop) and once for the device
// (a CUDA kernel), so that a CPU checker and the GPU see bit-identical
// inputs without a host copy of a 100 GB pool.
//
// Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014; the 64-bit finaliser
// constants are S. Vigna's published `splitmix64.c`).  The i-th output of a
// SplitMix64 stream whose state starts at `x0` is mix(x0 + (i+1)*GAMMA).
//
// Element value: element i of stream `base` is bank[out_i >> (64 - bits)],
// where bank is a table of 2^bits fp16 values (normal deviates produced by
// synth_bank_normal below and rounded to fp16 by the caller).
#include <cstdint>
#include <cmath>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// i-th output (0-based) of the SplitMix64 stream with initial state x0.
__host__ __device__ __forceinline__ uint64_t splitmix_at(uint64_t x0, uint64_t i) {
  return mix64(x0 + (i + 1) * kGamma);
}

__global__ void fill_kernel(uint16_t* __restrict__ dst, const uint16_t* __restrict__ bank,
                            int shift, uint64_t base, uint64_t start, uint64_t n) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    dst[i] = bank[splitmix_at(base, start + i) >> shift];
  }
}

// Eight consecutive elements per thread, written as one 16-byte store.
__global__ void fill_kernel_vec8(uint4* __restrict__ dst, const uint16_t* __restrict__ bank,
                                 int shift, uint64_t base, uint64_t start, uint64_t nvec) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t v = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const uint64_t e0 = start + v * 8;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = bank[splitmix_at(base, e0 + 2 * j) >> shift];
      const uint32_t hi = bank[splitmix_at(base, e0 + 2 * j + 1) >> shift];
      w[j] = lo | (hi << 16);
    }
    dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

extern "C" {

// i-th output of the SplitMix64 stream with initial state x0 (exposed so a
// test can check it against the generator's published definition).
uint64_t synth_splitmix64_at(uint64_t x0, uint64_t i) { return splitmix_at(x0, i); }

// Stream base for (seed, stream id): the first output of the SplitMix64
// stream whose state starts at seed * 2^32 + stream.
uint64_t synth_stream_base(uint64_t seed, uint64_t stream) {
  return splitmix_at((seed << 32) + stream, 0);
}

// n standard normal deviates in double via the Box-Muller transform
// (G. Box, M. Muller, Ann. Math. Statist. 29(2), 1958) from SplitMix64
// uniforms u = (x >> 11) * 2^-53.  Pairs (2j, 2j+1) share one (u1, u2).
void synth_bank_normal(double* out, uint64_t n, uint64_t seed) {
  const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
  for (long long j = 0; j < (long long)((n + 1) / 2); ++j) {
    const double u1 = (double)(splitmix_at(seed, 2 * (uint64_t)j) >> 11) * 0x1.0p-53;
    const double u2 = (double)(splitmix_at(seed, 2 * (uint64_t)j + 1) >> 11) * 0x1.0p-53;
    const double r = std::sqrt(-2.0 * std::log(1.0 - u1));
    const double t = two_pi * u2;
    out[2 * j] = r * std::cos(t);
    if ((uint64_t)(2 * j + 1) < n) out[2 * j + 1] = r * std::sin(t);
  }
}

// n uniform draws in [0, 2^64) (raw SplitMix64 outputs start .. start+n-1).
void synth_raw(uint64_t* out, uint64_t x0, uint64_t start, uint64_t n) {
  for (uint64_t i = 0; i < n; ++i) out[i] = splitmix_at(x0, start + i);
}

// Host fill: dst[i] = bank[splitmix_at(base, start + i) >> (64 - bank_bits)].
void synth_fill_host(uint16_t* dst, const uint16_t* bank, int bank_bits, uint64_t base,
                     uint64_t start, uint64_t n) {
  const int shift = 64 - bank_bits;
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i) {
    dst[i] = bank[splitmix_at(base, start + (uint64_t)i) >> shift];
  }
}

// Device fill of the same values.  `dst` and `bank` are device pointers;
// returns 0 on success or the cudaError_t of the launch.
int synth_fill_device(void* dst, const void* bank, int bank_bits, uint64_t base, uint64_t start,
                      uint64_t n, void* stream) {
  if (n == 0) return 0;
  const int shift = 64 - bank_bits;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0 && (n % 8) == 0) {
    const uint64_t nvec = n / 8;
    uint64_t blocks = (nvec + threads - 1) / threads;
    if (blocks > (uint64_t)sms * 64) blocks = (uint64_t)sms * 64;
    fill_kernel_vec8<<<(unsigned)blocks, threads, 0, st>>>(
        static_cast<uint4*>(dst), static_cast<const uint16_t*>(bank), shift, base, start, nvec);
  } else {
    uint64_t blocks = (n + threads - 1) / threads;
    if (blocks > (uint64_t)sms * 64) blocks = (uint64_t)sms * 64;
    fill_kernel<<<(unsigned)blocks, threads, 0, st>>>(
        static_cast<uint16_t*>(dst), static_cast<const uint16_t*>(bank), shift, base, start, n);
  }
  return (int)cudaGetLastError();
}

}  // extern "C"
