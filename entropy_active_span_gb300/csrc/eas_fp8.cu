// Per-row e4m3 quantisation of hidden states or weights for the FP8 forward.
//   amax = max |x|, scale = amax / 448, inv = 448 / amax (IEEE round to
//   nearest), q = e4m3(x * inv) rounded to nearest-even, saturating at 448;
//   an all-zero row uses scale = inv = 1.  Dequantised value: e4m3(q) * scale.
#include <cuda_fp8.h>

#include "eas_device.cuh"
#include "eas_kernels.h"

namespace eas {

namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename In>
__global__ void __launch_bounds__(256)
quantize_rows_e4m3_kernel(const In* __restrict__ src, long long R, long long H,
                          uint8_t* __restrict__ dst, float* __restrict__ scale) {
  __shared__ float red[8];
  for (long long r = blockIdx.x; r < R; r += gridDim.x) {
    const In* x = src + r * H;
    float amax = 0.f;
    for (long long i = threadIdx.x; i < H; i += blockDim.x) amax = fmaxf(amax, fabsf(to_f32(x[i])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();
    float sc = 1.f, inv = 1.f;
    if (amax > 0.f) {
      sc = __fdiv_rn(amax, 448.f);
      inv = __fdiv_rn(448.f, amax);
    }
    if (threadIdx.x == 0) scale[r] = sc;
    uint8_t* d = dst + r * H;
    for (long long i = threadIdx.x; i < H; i += blockDim.x)
      d[i] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fmul_rn(to_f32(x[i]), inv),
                                                        __NV_SATFINITE, __NV_E4M3));
  }
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const void* src, int src_is_bf16, long long R, long long H,
                                      uint8_t* dst, float* scale, int num_sms, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const long long grid = R < 16LL * num_sms ? R : 16LL * num_sms;
  if (src_is_bf16)
    quantize_rows_e4m3_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(src), R, H, dst, scale);
  else
    quantize_rows_e4m3_kernel<float><<<static_cast<unsigned>(grid), 256, 0, s>>>(
        static_cast<const float*>(src), R, H, dst, scale);
  return cudaGetLastError();
}

}  // namespace eas
