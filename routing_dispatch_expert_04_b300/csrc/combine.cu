// Combine back to token order, and the auxiliary load-balancing statistics.
//
// Combine -- "Expert Parallelism (MoE)", "MoE Layer Structure": Y = sum over the selected
// experts of expert_output[token] * routing_weight[token]; "Expert Parallelism (EP)",
// step 4 (all-to-all COMBINE sends outputs back to each token's home position).  On one
// GPU this is a gather: one warp per token reads the token's kept packed rows (fp32
// expert outputs) with 16-byte loads, accumulates w * y in fp32 in ascending k (then the shared expert's row),
// and stores the token's row once.  Each output element is written by exactly one
// thread, so there are no atomics and the result is deterministic.  A dropped
// assignment (slot -1) contributes exactly 0.
//
// Aux statistics -- "Load Balancing: The Auxiliary Loss": L_aux = alpha * sum_i f_i P_i
// with f_i the fraction of the T*K assignments routed to expert i (counted before
// dropping) and P_i the mean softmax probability of expert i.  P_i is the fixed-order
// fp64 sum of the per-block partial sums the routing kernel left in the workspace.
#include "common.cuh"

namespace moe {

// Expert outputs (yp, ys) are fp32; each thread handles 4 consecutive columns.
template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ yp, const int32_t* __restrict__ slot,
               const float* __restrict__ w, const float* __restrict__ ys, T* __restrict__ y,
               int Tn, int d, int K) {
  constexpr int P = 4;
  __shared__ int s_slot[8][32];
  __shared__ float s_w[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = d / P;
  for (int t = blockIdx.x * 8 + warp; t < Tn; t += gridDim.x * 8) {
    if (lane < K) {
      s_slot[warp][lane] = slot[(size_t)t * K + lane];
      s_w[warp][lane] = w[(size_t)t * K + lane];
    }
    __syncwarp();
    for (int j = lane; j < nvec; j += 32) {
      float acc[P];
#pragma unroll
      for (int i = 0; i < P; ++i) acc[i] = 0.f;
      for (int k0 = 0; k0 < K; k0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int k = k0 + u;
          const int s = (k < K) ? s_slot[warp][k] : -1;
          v[u] = (s >= 0) ? ld_nc_v4(reinterpret_cast<const uint4*>(yp + (size_t)s * d) + j)
                          : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int k = k0 + u;
          if (k < K && s_slot[warp][k] >= 0) {
            float f[P];
            Elem<float>::unpack(v[u], f);
            const float wk = s_w[warp][k];
#pragma unroll
            for (int i = 0; i < P; ++i) acc[i] = fmaf(wk, f[i], acc[i]);
          }
        }
      }
      if (ys != nullptr) {
        float f[P];
        Elem<float>::unpack(ld_nc_v4(reinterpret_cast<const uint4*>(ys + (size_t)t * d) + j), f);
#pragma unroll
        for (int i = 0; i < P; ++i) acc[i] += f[i];
      }
      T* out = y + (size_t)t * d + (size_t)j * P;
      if (sizeof(T) == 4) {
        st_v4(out, Elem<float>::pack(acc));
      } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2], acc[3]);
        uint2 v2 = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        *reinterpret_cast<uint2*>(out) = v2;
      }
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(256)
aux_kernel(const int32_t* __restrict__ counts, const float* __restrict__ ppart, int nblk, int E,
           int Tn, int K, float alpha, float* __restrict__ f, float* __restrict__ P,
           float* __restrict__ l_aux) {
  __shared__ double s_fp[256];
  const int e = threadIdx.x;
  if (e < E) {
    double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
    int b = 0;
    for (; b + 3 < nblk; b += 4) {
      a0 += (double)ppart[(size_t)(b + 0) * E + e];
      a1 += (double)ppart[(size_t)(b + 1) * E + e];
      a2 += (double)ppart[(size_t)(b + 2) * E + e];
      a3 += (double)ppart[(size_t)(b + 3) * E + e];
    }
    for (; b < nblk; ++b) a0 += (double)ppart[(size_t)b * E + e];
    const double psum = (a0 + a1) + (a2 + a3);
    double fe = 0.0, pe = 0.0;
    if (Tn > 0) {
      fe = (double)counts[e] / ((double)Tn * (double)K);
      pe = psum / (double)Tn;
    }
    f[e] = (float)fe;
    P[e] = (float)pe;
    s_fp[e] = fe * pe;
  }
  __syncthreads();
  if (e == 0) {
    double acc = 0.0;
    for (int i = 0; i < E; ++i) acc += s_fp[i];
    l_aux[0] = (float)((double)alpha * acc);
  }
}

cudaError_t launch_combine(int dtype, const void* yp, const int32_t* slot, const float* w,
                           const void* ys, void* y, int Tn, int d, int K, int num_sms,
                           cudaStream_t st) {
  const int want = (Tn + 7) / 8;
  const int grid = want < num_sms * 16 ? want : num_sms * 16;
  if (dtype == MOE_BF16)
    combine_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const float*)yp, slot, w,
                                                        (const float*)ys, (__nv_bfloat16*)y, Tn, d, K);
  else
    combine_kernel<float><<<grid, 256, 0, st>>>((const float*)yp, slot, w, (const float*)ys,
                                                (float*)y, Tn, d, K);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_aux(const int32_t* counts, const float* ppart, int nblk, int E, int Tn, int K,
                       float alpha, float* f, float* P, float* l_aux, cudaStream_t st) {
  aux_kernel<<<1, 256, 0, st>>>(counts, ppart, nblk, E, Tn, K, alpha, f, P, l_aux);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
