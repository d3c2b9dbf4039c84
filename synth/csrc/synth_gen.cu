// synth_gen.cu - device fill of the seeded synthetic byte streams.
//
// Produces exactly the bytes of synth.byte_stream / synth.int4_scales_bits (host,
// numpy): draw i of the stream with key k is mix64(k + (i + 1) * GAMMA), mix64 being
// the SplitMix64 output function (Steele, Lea, Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014); byte p of a byte stream is byte p % 8 (little
// endian) of draw p / 8; a scale is the fp16 bit pattern (7 << 10) | (draw >> 54).
// Input generation only: nothing here is arithmetic of the expert layer.
#include <cstdint>
#include <cuda_runtime.h>

namespace {
constexpr uint64_t GAMMA = 0x9E3779B97F4A7C15ull;
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__global__ void fill_bytes_kernel(uint64_t key, uint8_t* dst, size_t nbytes) {
  const size_t ndraw = (nbytes + 7) / 8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < ndraw;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint64_t d = mix64(key + (i + 1) * GAMMA);
    const size_t b0 = i * 8;
    if (b0 + 8 <= nbytes && ((reinterpret_cast<uintptr_t>(dst) + b0) & 7) == 0) {
      *reinterpret_cast<uint64_t*>(dst + b0) = d;
    } else {
      for (int b = 0; b < 8 && b0 + b < nbytes; ++b) dst[b0 + b] = (uint8_t)(d >> (8 * b));
    }
  }
}
__global__ void fill_scales_kernel(uint64_t key, uint16_t* dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint64_t d = mix64(key + (i + 1) * GAMMA);
    dst[i] = (uint16_t)((7u << 10) | (uint32_t)(d >> 54));
  }
}
}  // namespace

extern "C" int synth_fill_bytes(uint64_t key, void* dst, size_t nbytes, void* stream) {
  if (!nbytes) return 0;
  const size_t ndraw = (nbytes + 7) / 8;
  const int blocks = (int)((ndraw + 255) / 256 < 65536 ? (ndraw + 255) / 256 : 65536);
  fill_bytes_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(key, (uint8_t*)dst, nbytes);
  return (int)cudaGetLastError();
}

extern "C" int synth_fill_scales(uint64_t key, void* dst, size_t n, void* stream) {
  if (!n) return 0;
  const int blocks = (int)((n + 255) / 256 < 65536 ? (n + 255) / 256 : 65536);
  fill_scales_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(key, (uint16_t*)dst, n);
  return (int)cudaGetLastError();
}
