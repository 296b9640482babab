// Per-row E4M3 quantisation for the FP8 expert GEMMs.
//
// The pages only say that MoE is the most FP8-sensitive architecture ("Expert
// Parallelism (EP)", "See also"); the recipe here is the plainest one.  Each row of an
// operand gets one fp32 scale: amax = max |row|, inv = 448 / amax, code = E4M3(row * inv)
// (round to nearest even, saturating at +-448), scale = amax / 448; a zero row gets zero
// codes and scale 0.  The GEMM multiplies its fp32 accumulator by the A row's and the B
// row's scales.  Every step is one correctly rounded fp32 operation, so the codes are a
// fixed function of the input values.
//
// One warp per row: a pass for the amax, then a pass that scales, converts and stores
// (16-byte loads; the second pass re-reads the row, mostly from L1/L2).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

template <typename T> struct QIn;
template <> struct QIn<float> {
  static constexpr int PER16 = 4;
  __device__ static void unpack(const uint4& v, float* f) { Elem<float>::unpack(v, f); }
};
template <> struct QIn<__nv_bfloat16> {
  static constexpr int PER16 = 8;
  __device__ static void unpack(const uint4& v, float* f) { Elem<__nv_bfloat16>::unpack(v, f); }
};
template <> struct QIn<__half> {
  static constexpr int PER16 = 8;
  __device__ static void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
};

template <typename T>
__global__ void __launch_bounds__(256)
quantize_rows_e4m3_kernel(const T* __restrict__ src, int64_t rows, int cols,
                          const int32_t* __restrict__ rows_dev, uint8_t* __restrict__ codes,
                          float* __restrict__ scales) {
  constexpr int P = QIn<T>::PER16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (rows_dev != nullptr) {
    const int64_t rd = *rows_dev;
    if (rd < rows) rows = rd < 0 ? 0 : rd;
  }
  const int nvec = cols / P;
  for (int64_t r = (int64_t)blockIdx.x * 8 + warp; r < rows; r += (int64_t)gridDim.x * 8) {
    const uint4* in = reinterpret_cast<const uint4*>(src + r * cols);
    float amax = 0.f;
    for (int j = lane; j < nvec; j += 32) {
      float f[P];
      QIn<T>::unpack(ld_nc_v4(in + j), f);
#pragma unroll
      for (int i = 0; i < P; ++i) amax = fmaxf(amax, fabsf(f[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 0.f;
    if (lane == 0) scales[r] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 0.f;
    uint8_t* out = codes + r * cols;
    for (int j = lane; j < nvec; j += 32) {
      float f[P];
      QIn<T>::unpack(ld_nc_v4(in + j), f);
      uint16_t pk[P / 2];
#pragma unroll
      for (int i = 0; i < P / 2; ++i)
        pk[i] = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv)), __NV_SATFINITE,
            __NV_E4M3);
      // element 2i in the low byte of pk[i]; codes stored in element order
      if constexpr (P == 8) {
        *reinterpret_cast<uint2*>(out + (size_t)j * 8) =
            make_uint2(pk[0] | ((uint32_t)pk[1] << 16), pk[2] | ((uint32_t)pk[3] << 16));
      } else {
        *reinterpret_cast<uint32_t*>(out + (size_t)j * 4) = pk[0] | ((uint32_t)pk[1] << 16);
      }
    }
  }
}

// src dtype: MOE_F32, MOE_BF16 or MOE_F16; cols a multiple of 16.
cudaError_t launch_quantize_e4m3(int dtype, const void* src, int64_t rows, int cols,
                                 const int32_t* rows_dev, void* codes, float* scales, int num_sms,
                                 cudaStream_t st) {
  const int64_t want = (rows + 7) / 8;
  const int grid = (int)(want < num_sms * 16 ? (want > 0 ? want : 1) : num_sms * 16);
  uint8_t* c = (uint8_t*)codes;
  if (dtype == MOE_F32)
    quantize_rows_e4m3_kernel<float><<<grid, 256, 0, st>>>((const float*)src, rows, cols, rows_dev, c, scales);
  else if (dtype == MOE_BF16)
    quantize_rows_e4m3_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)src, rows, cols,
                                                                    rows_dev, c, scales);
  else
    quantize_rows_e4m3_kernel<__half><<<grid, 256, 0, st>>>((const __half*)src, rows, cols, rows_dev, c,
                                                             scales);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
