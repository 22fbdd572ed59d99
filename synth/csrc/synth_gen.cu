// Device twin of synth/generate.py: the same SplitMix64 counter streams and the
// same value derivations, so that large weight sets can be generated in device
// memory.  Holds no arithmetic of the MoE method; both the oracle tests and the
// CUDA path read what this (or the host twin) writes.  Every fp64 step uses an
// explicitly rounded intrinsic, so no multiply-add is contracted and the bits
// match the host twin exactly.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kKey0 = 0x243F6A8885A308D3ull;
enum { P_CODES = 1, P_SCALES = 2, P_BIASES = 3 };

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t stream_key(const uint64_t* f, int n) {
  uint64_t k = kKey0;
  for (int i = 0; i < n; ++i) k = mix64((k ^ f[i]) + kGamma);
  return k;
}

__device__ inline uint64_t out64(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * kGamma); }
__device__ inline double uni(uint64_t r) { return __dmul_rn((double)(r >> 11), 0x1.0p-53); }
__device__ inline uint16_t f32_to_bf16(float x) {
  const uint32_t b = __float_as_uint(x);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

__global__ void codes_kernel(uint64_t key, uint8_t* dst, size_t nbytes) {
  const size_t n64 = (nbytes + 7) / 8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n64; i += (size_t)gridDim.x * blockDim.x) {
    const uint64_t r = out64(key, i);
    if (8 * i + 8 <= nbytes) {
      reinterpret_cast<uint2*>(dst)[i] = make_uint2((uint32_t)r, (uint32_t)(r >> 32));
    } else {
      for (size_t b = 8 * i; b < nbytes; ++b) dst[b] = (uint8_t)(r >> (8 * (b - 8 * i)));
    }
  }
}

__global__ void scale_bias_kernel(uint64_t kscale, uint64_t kbias, double c, uint16_t* s_out, uint16_t* b_out,
                                  size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const double s = __dadd_rn(0.005, __dmul_rn(0.015, uni(out64(kscale, i))));
    const uint16_t sb = f32_to_bf16(__double2float_rn(s));
    const double s64 = (double)__uint_as_float((uint32_t)sb << 16);
    const double v = __dadd_rn(0.9, __dmul_rn(0.2, uni(out64(kbias, i))));
    const double b = __dmul_rn(__dmul_rn(-c, s64), v);
    s_out[i] = sb;
    b_out[i] = f32_to_bf16(__double2float_rn(b));
  }
}

}  // namespace

extern "C" {

// One canonical matrix (codes uint8 [rows, cols*bits/8], bf16 scales and biases
// [rows, cols/group]) of stream fields (seed, layer, expert, tensor).
int synth_matrix(uint64_t seed, uint64_t layer, uint64_t expert, uint64_t tensor, int rows, int cols, int bits,
                 int group, uint8_t* codes, uint16_t* scales, uint16_t* biases, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t fc[5] = {seed, layer, expert, tensor, P_CODES};
  const uint64_t fs[5] = {seed, layer, expert, tensor, P_SCALES};
  const uint64_t fb[5] = {seed, layer, expert, tensor, P_BIASES};
  const size_t nbytes = (size_t)rows * cols * bits / 8;
  const size_t ng = (size_t)rows * (cols / group);
  codes_kernel<<<1184, 256, 0, s>>>(stream_key(fc, 5), codes, nbytes);
  scale_bias_kernel<<<296, 256, 0, s>>>(stream_key(fs, 5), stream_key(fb, 5), bits == 4 ? 8.0 : 1.5, scales, biases,
                                        ng);
  return (int)cudaGetLastError();
}

uint64_t synth_stream_key(const uint64_t* fields, int n) { return stream_key(fields, n); }

}  // extern "C"
