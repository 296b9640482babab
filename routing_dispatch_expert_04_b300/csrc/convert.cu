// bf16 -> fp16 conversion of expert weights for the fp16 down-projection.
//
// The intermediate activation h between the two expert Linears is kept in fp16 (11
// significant bits against bf16's 8), so the second Linear runs with fp16 operands and
// its weights W2 need an fp16 copy.  Every bf16 value with magnitude in [2^-17, 65504]
// converts exactly; smaller magnitudes round at 2^-25 (fp16 subnormals); larger ones
// cannot be represented and are reported as a range error in the status word.
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

__global__ void __launch_bounds__(256)
bf16_to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n8,
                   uint32_t* hdr) {
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = ld_nc_v4(src + i);
    float f[8];
    Elem<__nv_bfloat16>::unpack(v, f);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      bad |= !(fabsf(f[2 * j]) <= 65504.f) || !(fabsf(f[2 * j + 1]) <= 65504.f);
      __half2 h = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    st_v4(dst + i, make_uint4(w[0], w[1], w[2], w[3]));
  }
  if (bad) raise_error(hdr, DEV_ERR_RANGE);
}

cudaError_t launch_bf16_to_f16(const void* src, void* dst, int64_t n, uint32_t* hdr, int num_sms,
                               cudaStream_t st) {
  const int64_t n8 = n / 8;
  int64_t grid = (n8 + 255) / 256;
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  if (grid < 1) grid = 1;
  bf16_to_f16_kernel<<<(unsigned)grid, 256, 0, st>>>((const uint4*)src, (uint4*)dst, n8, hdr);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
