// Combine back to token order, and the auxiliary load-balancing statistics.
//
// Combine -- "Expert Parallelism (MoE)", "MoE Layer Structure": Y = sum over the selected
// experts of expert_output[token] * routing_weight[token]; "Expert Parallelism (EP)",
// step 4 (all-to-all COMBINE sends outputs back to each token's home position).  On one
// GPU this is a gather: one warp per token reads the token's kept packed rows (expert
// outputs: fp16 for bf16 layers, fp32 for fp32 layers) with 16-byte loads, accumulates
// w * y in fp32 in ascending k (then the shared expert's row), and stores the token's
// row once.  Each output element is written by exactly one
// thread, so there are no atomics and the result is deterministic.  A dropped
// assignment (slot -1) contributes exactly 0.
//
// Aux statistics -- "Load Balancing: The Auxiliary Loss": L_aux = alpha * sum_i f_i P_i
// with f_i the fraction of the T*K assignments routed to expert i (counted before
// dropping) and P_i the mean softmax probability of expert i.  P_i is a fixed-order
// fp64 reduction of the per-block partial sums the routing kernel left in the workspace,
// and the sum over experts is taken in expert order, so the result is deterministic.
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

// Expert outputs (yp, ys) are fp16 for bf16 layers and fp32 for fp32 layers.  Each
// lane handles JV 16-byte slots of a row per pass (j, j + 32, ...: 8 fp16 or 4 fp32
// columns each) for 8 / JV rows at a time, so that 8 row loads are in flight per lane; k
// is summed in order, in fp32.
template <typename Tin> struct CombineIn;
template <> struct CombineIn<float> {
  static constexpr int P = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    Elem<float>::unpack(v, f);
  }
};
template <> struct CombineIn<__half> {
  static constexpr int P = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
};

// One 16-byte slot of P output columns, rounded once to the output type.
template <typename Tout, int P>
__device__ __forceinline__ void store_slot(Tout* out, const float* acc);
template <>
__device__ __forceinline__ void store_slot<float, 4>(float* out, const float* acc) {
  st_v4(out, Elem<float>::pack(acc));
}
template <>
__device__ __forceinline__ void store_slot<__nv_bfloat16, 8>(__nv_bfloat16* out, const float* acc) {
  st_v4(out, Elem<__nv_bfloat16>::pack(acc));
}

template <typename Tout, typename Tin, int JV>
__global__ void __launch_bounds__(256, JV == 2 ? 4 : 3)  // two slots: four blocks per SM
combine_kernel(const Tin* __restrict__ yp, const int32_t* __restrict__ slot,
               const float* __restrict__ w, const Tin* __restrict__ ys, Tout* __restrict__ y,
               int Tn, int d, int K) {
  // JV 16-byte slots of each row per lane and pass, KC rows per batch of loads: 8 loads
  // in flight per lane either way
  constexpr int P = CombineIn<Tin>::P, KC = 8 / JV;
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
    for (int j0 = lane; j0 < nvec; j0 += 32 * JV) {
      float acc[JV][P];
#pragma unroll
      for (int v = 0; v < JV; ++v)
#pragma unroll
        for (int i = 0; i < P; ++i) acc[v][i] = 0.f;
      for (int k0 = 0; k0 < K; k0 += KC) {
        uint4 ld[KC][JV];
#pragma unroll
        for (int u = 0; u < KC; ++u) {
          const int k = k0 + u;
          const int s = (k < K) ? s_slot[warp][k] : -1;
          const uint4* rowp = reinterpret_cast<const uint4*>(yp + (size_t)(s < 0 ? 0 : s) * d);
#pragma unroll
          for (int v = 0; v < JV; ++v) {
            const int j = j0 + 32 * v;
            ld[u][v] = (s >= 0 && j < nvec) ? ld_nc_v4(rowp + j) : make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int u = 0; u < KC; ++u) {
          const int k = k0 + u;
          if (k < K && s_slot[warp][k] >= 0) {
            const float wk = s_w[warp][k];
#pragma unroll
            for (int v = 0; v < JV; ++v) {
              float f[P];
              CombineIn<Tin>::unpack(ld[u][v], f);
#pragma unroll
              for (int i = 0; i < P; ++i) acc[v][i] = fmaf(wk, f[i], acc[v][i]);
            }
          }
        }
      }
      if (ys != nullptr) {
        const uint4* rs = reinterpret_cast<const uint4*>(ys + (size_t)t * d);
#pragma unroll
        for (int v = 0; v < JV; ++v) {
          const int j = j0 + 32 * v;
          float f[P];
          CombineIn<Tin>::unpack(j < nvec ? ld_nc_v4(rs + j) : make_uint4(0u, 0u, 0u, 0u), f);
#pragma unroll
          for (int i = 0; i < P; ++i) acc[v][i] += f[i];
        }
      }
      Tout* out = y + (size_t)t * d;
#pragma unroll
      for (int v = 0; v < JV; ++v) {
        const int j = j0 + 32 * v;
        if (j < nvec) store_slot<Tout, P>(out + (size_t)j * P, acc[v]);
      }
    }
    __syncwarp();
  }
}

// One block per expert: P_i from the per-route-block partial sums (layout [E][nblk]),
// f_i from the pre-drop counts; the last block to finish sums f_i * P_i over i in order.
constexpr int AUX_THREADS = 128;

__global__ void __launch_bounds__(AUX_THREADS)
aux_kernel(const int32_t* __restrict__ counts, const float* __restrict__ ppart, int E,
           int Tn, int K, float alpha, float* __restrict__ f, float* __restrict__ P,
           float* __restrict__ l_aux, double* auxfp, uint32_t* hdr) {
  __shared__ double s_red[AUX_THREADS];
  __shared__ bool s_last;
  const int e = blockIdx.x, tid = threadIdx.x;
  // the partial sums' layout [E][nblk] follows the routing grid the routing call recorded
  const int nblk = Tn > 0 ? (int)*(volatile uint32_t*)&hdr[HDR_ROUTE_NBLK] : 0;
  const float* row = ppart + (size_t)e * nblk;
  double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
  int b = tid;
  for (; b + 3 * AUX_THREADS < nblk; b += 4 * AUX_THREADS) {
    a0 += (double)row[b];
    a1 += (double)row[b + AUX_THREADS];
    a2 += (double)row[b + 2 * AUX_THREADS];
    a3 += (double)row[b + 3 * AUX_THREADS];
  }
  for (; b < nblk; b += AUX_THREADS) a0 += (double)row[b];
  s_red[tid] = (a0 + a1) + (a2 + a3);
  __syncthreads();
  for (int w = AUX_THREADS / 2; w > 0; w >>= 1) {
    if (tid < w) s_red[tid] += s_red[tid + w];
    __syncthreads();
  }
  if (tid == 0) {
    double fe = 0.0, pe = 0.0;
    if (Tn > 0) {
      fe = (double)counts[e] / ((double)Tn * (double)K);
      pe = s_red[0] / (double)Tn;
    }
    f[e] = (float)fe;
    P[e] = (float)pe;
    auxfp[e] = fe * pe;
    __threadfence();
    s_last = (atomicAdd(&hdr[2], 1u) == (uint32_t)(E - 1));
  }
  __syncthreads();
  if (s_last && tid == 0) {
    __threadfence();
    const volatile double* v = auxfp;
    double acc = 0.0;
    for (int i = 0; i < E; ++i) acc += v[i];
    l_aux[0] = (float)((double)alpha * acc);
    hdr[2] = 0u;  // ready for the next call
  }
}

// Backward of the auxiliary loss ("Load Balancing: The Auxiliary Loss": the loss is
// added to the task loss and backpropagated).  f_i counts top-K choices and is a step
// function of the logits (zero derivative away from ties), so only P_i carries gradient:
//   grad[t,j] = (alpha / T) * p[t,j] * (f_j - sum_i f_i p[t,i]),  p = softmax(logits[t]).
// One warp per token; the softmax is recomputed in fp32 as in the routing kernel.
template <int VPT>
__global__ void __launch_bounds__(256)
aux_grad_kernel(const float* __restrict__ logits, const float* __restrict__ f, int Tn, int E,
                float scale, float* __restrict__ grad) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float fv[VPT];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int e = lane + 32 * j;
    fv[j] = e < E ? f[e] : 0.f;
  }
  for (int t = blockIdx.x * 8 + warp; t < Tn; t += gridDim.x * 8) {
    float v[VPT];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e = lane + 32 * j;
      v[j] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
      m = fmaxf(m, v[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e = lane + 32 * j;
      v[j] = e < E ? expf(v[j] - m) : 0.f;
      s += v[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    float mf = 0.f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      v[j] = v[j] / s;
      mf = fmaf(fv[j], v[j], mf);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mf += __shfl_xor_sync(0xffffffffu, mf, o);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e = lane + 32 * j;
      if (e < E) grad[(size_t)t * E + e] = scale * v[j] * (fv[j] - mf);
    }
  }
}

cudaError_t launch_aux_grad(const float* logits, const float* f, int Tn, int E, float alpha,
                            float* grad, int num_sms, cudaStream_t st) {
  const int want = (Tn + 7) / 8;
  const int grid = want < num_sms * 16 ? want : num_sms * 16;
  const float scale = Tn > 0 ? alpha / (float)Tn : 0.f;
  if (E <= 32)
    aux_grad_kernel<1><<<grid, 256, 0, st>>>(logits, f, Tn, E, scale, grad);
  else if (E <= 64)
    aux_grad_kernel<2><<<grid, 256, 0, st>>>(logits, f, Tn, E, scale, grad);
  else if (E <= 128)
    aux_grad_kernel<4><<<grid, 256, 0, st>>>(logits, f, Tn, E, scale, grad);
  else
    aux_grad_kernel<8><<<grid, 256, 0, st>>>(logits, f, Tn, E, scale, grad);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine(int dtype, const void* yp, const int32_t* slot, const float* w,
                           const void* ys, void* y, int Tn, int d, int K, int num_sms,
                           cudaStream_t st) {
  const int want = (Tn + 7) / 8;
  const int grid = want < num_sms * 16 ? want : num_sms * 16;
  // with one or two rows per token, four slots of each row per lane keep 8 loads in
  // flight; with more rows, two slots of four rows
  const bool wide = K <= 2;
  if (dtype == MOE_BF16) {
    if (wide)
      combine_kernel<__nv_bfloat16, __half, 4><<<grid, 256, 0, st>>>(
          (const __half*)yp, slot, w, (const __half*)ys, (__nv_bfloat16*)y, Tn, d, K);
    else
      combine_kernel<__nv_bfloat16, __half, 2><<<grid, 256, 0, st>>>(
          (const __half*)yp, slot, w, (const __half*)ys, (__nv_bfloat16*)y, Tn, d, K);
  } else {
    if (wide)
      combine_kernel<float, float, 4><<<grid, 256, 0, st>>>((const float*)yp, slot, w,
                                                            (const float*)ys, (float*)y, Tn, d, K);
    else
      combine_kernel<float, float, 2><<<grid, 256, 0, st>>>((const float*)yp, slot, w,
                                                            (const float*)ys, (float*)y, Tn, d, K);
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_aux(const int32_t* counts, const float* ppart, int E, int Tn, int K,
                       float alpha, float* f, float* P, float* l_aux, double* auxfp, uint32_t* hdr,
                       cudaStream_t st) {
  aux_kernel<<<E, AUX_THREADS, 0, st>>>(counts, ppart, E, Tn, K, alpha, f, P, l_aux, auxfp, hdr);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
