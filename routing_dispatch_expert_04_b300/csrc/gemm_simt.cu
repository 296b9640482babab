// CUDA-core (FFMA) grouped GEMM: C[r, n] = epi( sum_k A[r, k] * B[g, n, k] ) for the rows
// r of group g, rows [offsets[g], offsets[g+1]).
//
// This is the fp32 path ("Expert Parallelism (MoE)", "MoE Layer Structure": each expert
// applies Linear(d -> 4d) -> GELU -> Linear(4d -> d); the router is Linear d -> E).
// fp32 operands need fp32 products to hold a 1e-4 relative error, which TF32 tensor
// cores do not give, so fp32 stays on the CUDA cores; bf16 contractions run on the
// tcgen05 engine.  Epilogues: none, exact-erf GELU, or + fp32 bias with fp32 output.
//
// The (group, m-tile) of a block is found on the device from `offsets`, so the launch
// needs no host synchronisation; blocks past the last tile exit at once.
#include <math.h>

#include "common.cuh"

namespace moe {

enum { EPI_NONE = 0, EPI_GELU = 1, EPI_BIAS = 2 };

__device__ __forceinline__ float gelu_erf(float v) {
  return 0.5f * v * (1.0f + erff(v * 0.70710678118654752440f));
}

template <typename Tin, typename Tout, int EPI>
__global__ void __launch_bounds__(256)
simt_gemm_kernel(const Tin* __restrict__ A, const int32_t* __restrict__ gather_src, int gather_k,
                 int64_t gather_rows, const Tin* __restrict__ B, Tout* __restrict__ Cout,
                 const int32_t* __restrict__ offsets, int G, int M, int N, int Kd,
                 int64_t rows_cap, const float* __restrict__ bias, uint32_t* hdr) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ int s_g;
  __shared__ int64_t s_row0, s_rowend;
  if (threadIdx.x == 0) {
    int g = -1;
    int64_t row0 = 0, rowend = 0;
    const int y = blockIdx.x;
    if (offsets == nullptr) {
      if ((int64_t)y * BM < M) {
        g = 0;
        row0 = (int64_t)y * BM;
        rowend = M;
      }
    } else {
      int64_t acc = 0;
      for (int gg = 0; gg < G; ++gg) {
        int64_t lo = offsets[gg], hi = offsets[gg + 1];
        if (hi > rows_cap) {
          raise_error(hdr, DEV_ERR_OVERFLOW);
          hi = rows_cap;
        }
        if (lo < 0) lo = 0;
        if (lo > hi) lo = hi;
        const int64_t nt = (hi - lo + BM - 1) / BM;
        if (y < acc + nt) {
          g = gg;
          row0 = lo + (y - acc) * BM;
          rowend = hi;
          break;
        }
        acc += nt;
      }
    }
    s_g = g;
    s_row0 = row0;
    s_rowend = rowend;
  }
  __syncthreads();
  const int g = s_g;
  if (g < 0) return;
  const int64_t row0 = s_row0, rowend = s_rowend;
  const int n0 = blockIdx.y * BN;
  const Tin* Bg = B + (size_t)g * N * Kd;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < Kd; k0 += BK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = threadIdx.x + i * 256;
      const int r = idx / BK, kk = idx % BK;
      const int64_t row = row0 + r;
      const int k = k0 + kk;
      int64_t arow = row;  // A row: the packed row, or the token row it was gathered from
      if (gather_src != nullptr && row < rowend) {
        arow = gather_src[row] / gather_k;
        if (arow < 0 || arow >= gather_rows) {
          raise_error(hdr, DEV_ERR_BAD_ID);
          arow = 0;
        }
      }
      As[kk][r] = (row < rowend && k < Kd) ? Elem<Tin>::to_f(A[arow * Kd + k]) : 0.f;
      const int n = n0 + r;
      Bs[kk][r] = (n < N && k < Kd) ? Elem<Tin>::to_f(Bg[(size_t)n * Kd + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = row0 + ty * 4 + i;
    if (row >= rowend) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx * 4 + j;
      if (col >= N) continue;
      float v = acc[i][j];
      if (EPI == EPI_GELU) v = gelu_erf(v);
      if (EPI == EPI_BIAS && bias != nullptr) v += bias[col];
      Cout[row * N + col] = Elem<Tout>::from_f(v);
    }
  }
}

// Grouped expert GEMM on CUDA cores.  gelu: GELU epilogue and dtype output (first
// Linear); otherwise plain fp32 output (second Linear).
cudaError_t launch_simt_grouped(int dtype, const void* A, const int32_t* gather_src, int gather_k,
                                int64_t gather_rows, const void* B, void* C,
                                const int32_t* offsets, int G, int N, int Kd, int64_t rows_cap,
                                bool gelu, uint32_t* hdr, cudaStream_t st) {
  const int64_t mt = (rows_cap + 63) / 64 + G;
  const dim3 grid((unsigned)mt, (unsigned)((N + 63) / 64));
  if (dtype == MOE_BF16) {
    using T = __nv_bfloat16;
    if (gelu)
      simt_gemm_kernel<T, T, EPI_GELU><<<grid, 256, 0, st>>>((const T*)A, gather_src, gather_k, gather_rows,
                                                             (const T*)B, (T*)C, offsets, G, 0, N,
                                                             Kd, rows_cap, nullptr, hdr);
    else
      simt_gemm_kernel<T, float, EPI_NONE><<<grid, 256, 0, st>>>(
          (const T*)A, gather_src, gather_k, gather_rows, (const T*)B, (float*)C, offsets, G, 0, N,
          Kd, rows_cap, nullptr, hdr);
  } else {
    if (gelu)
      simt_gemm_kernel<float, float, EPI_GELU><<<grid, 256, 0, st>>>(
          (const float*)A, gather_src, gather_k, gather_rows, (const float*)B, (float*)C, offsets,
          G, 0, N, Kd, rows_cap, nullptr, hdr);
    else
      simt_gemm_kernel<float, float, EPI_NONE><<<grid, 256, 0, st>>>(
          (const float*)A, gather_src, gather_k, gather_rows, (const float*)B, (float*)C, offsets,
          G, 0, N, Kd, rows_cap, nullptr, hdr);
  }
  count_launch();
  return cudaGetLastError();
}

// Router Linear on CUDA cores: logits[T, E] (fp32) = x . W_r^T + b_r.
cudaError_t launch_simt_router(int dtype, const void* x, const void* w_r, const float* b_r,
                               float* logits, int T, int E, int d, uint32_t* hdr, cudaStream_t st) {
  const dim3 grid((unsigned)((T + 63) / 64), (unsigned)((E + 63) / 64));
  if (dtype == MOE_BF16) {
    using Tb = __nv_bfloat16;
    simt_gemm_kernel<Tb, float, EPI_BIAS><<<grid, 256, 0, st>>>(
        (const Tb*)x, nullptr, 1, 0, (const Tb*)w_r, logits, nullptr, 1, T, E, d, T, b_r, hdr);
  } else {
    simt_gemm_kernel<float, float, EPI_BIAS><<<grid, 256, 0, st>>>(
        (const float*)x, nullptr, 1, 0, (const float*)w_r, logits, nullptr, 1, T, E, d, T, b_r,
        hdr);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
