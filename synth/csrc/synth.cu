// Device-side fill of the seeded synthetic inputs.
//
// This is the CUDA twin of the numpy generator in synth/__init__.py: Philox-4x32-10
// (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11) followed by
// a Box-Muller deviate whose log and cos use only correctly rounded fp32
// +, -, *, / and sqrt in the same order as the numpy code.  Every operation is an
// explicitly rounded intrinsic and the file is compiled with -fmad=false, so no
// multiply-add is contracted and the two sides agree bit for bit.  It holds none
// of the Muon method's arithmetic and is used only to make test and bench inputs.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;

__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += kW0; k1 += kW1; }
    const uint32_t hi0 = __umulhi(kM0, c[0]), lo0 = kM0 * c[0];
    const uint32_t hi1 = __umulhi(kM1, c[2]), lo1 = kM1 * c[2];
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
  }
}

__device__ __forceinline__ float bits(uint32_t b) { return __uint_as_float(b); }

__device__ __forceinline__ float unit(uint32_t x) {
  return __fmul_rn(__fadd_rn((float)(x >> 8), 0.5f), bits(0x33800000u));
}

__device__ __forceinline__ float ln32(float u) {
  const uint32_t b = __float_as_uint(u);
  int e = (int)(b >> 23) - 127;
  float f = bits((b & 0x7FFFFFu) | 0x3F800000u);
  if (f > bits(0x3fb504f3u)) { f = __fmul_rn(f, 0.5f); e += 1; }
  const float t = __fdiv_rn(__fsub_rn(f, 1.0f), __fadd_rn(f, 1.0f));
  const float t2 = __fmul_rn(t, t);
  float p = bits(0x3dba2e8cu);                       // 1/11
  p = __fadd_rn(__fmul_rn(p, t2), bits(0x3de38e39u)); // 1/9
  p = __fadd_rn(__fmul_rn(p, t2), bits(0x3e124925u)); // 1/7
  p = __fadd_rn(__fmul_rn(p, t2), bits(0x3e4ccccdu)); // 1/5
  p = __fadd_rn(__fmul_rn(p, t2), bits(0x3eaaaaabu)); // 1/3
  p = __fadd_rn(__fmul_rn(p, t2), 1.0f);
  const float lnf = __fmul_rn(__fmul_rn(t, p), 2.0f);
  return __fadd_rn(__fmul_rn((float)e, bits(0x3f317218u)), lnf);
}

__device__ __forceinline__ float cos2pi32(float u) {
  float w = fabsf(__fsub_rn(u, 0.5f));
  const bool far = w > 0.25f;
  if (far) w = __fsub_rn(0.5f, w);
  const float sign = far ? 1.0f : -1.0f;
  const float x = __fmul_rn(w, bits(0x40c90fdbu));
  const float y = __fmul_rn(x, x);
  const uint32_t k[7] = {0xbf000000u, 0x3d2aaaabu, 0xbab60b61u, 0x37d00d01u,
                         0xb493f27eu, 0x310f76c7u, 0xad49cba5u};
  float c = bits(k[6]);
#pragma unroll
  for (int i = 5; i >= 0; --i) c = __fadd_rn(__fmul_rn(c, y), bits(k[i]));
  c = __fadd_rn(__fmul_rn(c, y), 1.0f);
  return __fmul_rn(sign, c);
}

__device__ __forceinline__ float box_muller(uint32_t a, uint32_t b, float sigma) {
  const float r = __fsqrt_rn(__fmul_rn(ln32(unit(a)), -2.0f));
  return __fmul_rn(__fmul_rn(r, cos2pi32(unit(b))), sigma);
}

// One thread per Philox block = two consecutive elements [2*blk, 2*blk+1].
__global__ void fill_normal_kernel(void* out, int64_t start, int64_t n, uint32_t seed,
                                   uint32_t stream, uint32_t step, float sigma, int dtype) {
  const int64_t first_blk = start >> 1;
  const int64_t last_blk = (start + n - 1) >> 1;
  for (int64_t blk = first_blk + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
       blk <= last_blk; blk += (int64_t)gridDim.x * blockDim.x) {
    uint32_t c[4] = {(uint32_t)(blk & 0xFFFFFFFFll), (uint32_t)((uint64_t)blk >> 32), step, 0u};
    philox4x32_10(c, seed, stream);
    const float z0 = box_muller(c[0], c[1], sigma);
    const float z1 = box_muller(c[2], c[3], sigma);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int64_t e = 2 * blk + j;           // element index in the tensor
      const int64_t i = e - start;             // index in the output buffer
      if (i < 0 || i >= n) continue;
      const float z = j ? z1 : z0;
      if (dtype == 1) reinterpret_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(z);
      else reinterpret_cast<float*>(out)[i] = z;
    }
  }
}

__global__ void philox_kernel(uint32_t* out, const uint32_t* ctr, const uint32_t* key, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  uint32_t c[4] = {ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]};
  philox4x32_10(c, key[2 * i], key[2 * i + 1]);
  for (int j = 0; j < 4; ++j) out[4 * i + j] = c[j];
}

}  // namespace

extern "C" {

// Fill out[0..n) with element values [start, start+n) of the seeded N(0, sigma^2)
// tensor (seed, stream, step); dtype 0 = fp32, 1 = bf16 (round to nearest even).
// out is a device pointer; stream_handle a cudaStream_t (NULL = default stream).
// Returns 0, or the cudaError_t of the launch.
int synth_fill_normal(void* out, int64_t start, int64_t n, uint32_t seed, uint32_t stream,
                      uint32_t step, float sigma, int32_t dtype, void* stream_handle) {
  if (n <= 0) return 0;
  if (out == nullptr || start < 0 || (dtype != 0 && dtype != 1)) return (int)cudaErrorInvalidValue;
  const int64_t blocks_needed = (((start + n - 1) >> 1) - (start >> 1) + 1 + 255) / 256;
  const int grid = (int)(blocks_needed < 152 * 32 ? blocks_needed : 152 * 32);
  fill_normal_kernel<<<grid, 256, 0, (cudaStream_t)stream_handle>>>(out, start, n, seed, stream,
                                                                    step, sigma, dtype);
  return (int)cudaGetLastError();
}

// Raw Philox-4x32-10 on n (counter, key) pairs, all device pointers: ctr[4n], key[2n], out[4n].
int synth_philox(uint32_t* out, const uint32_t* ctr, const uint32_t* key, int64_t n,
                 void* stream_handle) {
  if (n <= 0) return 0;
  if (!out || !ctr || !key) return (int)cudaErrorInvalidValue;
  philox_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream_handle>>>(out, ctr, key, n);
  return (int)cudaGetLastError();
}

}  // extern "C"
