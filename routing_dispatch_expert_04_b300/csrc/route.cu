// Softmax over the experts and top-K selection, one warp per token.
//
// "Expert Parallelism (MoE)", section "MoE Layer Structure": for each token the
// top-K experts are activated; the routing weight is the softmax probability of the
// chosen expert ("Load Balancing: The Auxiliary Loss" speaks of the probability after
// softmax).  Selection compares the fp32 logits: higher first, equal values go to the
// lower expert id, so the picks are a deterministic function of the fp32 logits.
//
// With a selection-only bias (DeepSeek-V3's auxiliary-loss-free balancing, "Expert
// Parallelism (EP)", "Load balancing") the choice compares logit + bias, while the
// weights and the probability sums stay those of the unbiased softmax.
//
// The kernel also leaves, per block, the sum over its tokens of every expert's
// probability; the aux-statistics kernel reduces those partial sums in a fixed order
// to P_i, so the result is deterministic without floating-point atomics.
//
// With the dispatch plan (moe_route_plan) it also takes the capacity rule's first step
// ("Top-K Routing and Capacity Factor": an expert keeps the first C assignments in
// arrival order): every assignment's rank among its block's assignments to the same
// expert, and the block's count per expert.  The plan scan (one block per expert) turns
// the counts into each block's count in all earlier blocks and writes counts and
// offsets; the dispatch adds the two.  No block waits for another.
#include <math.h>
#include <limits.h>

#include "common.cuh"

namespace moe {

// Integer key whose unsigned order is the fp32 order of the score (-0 and +0 map to
// the same key, as they compare equal); never 0 for a finite or infinite score.
__device__ __forceinline__ uint32_t score_key(float f) {
  if (f == 0.f) f = 0.f;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int VPT, int TPW, bool PLAN>
__global__ void __launch_bounds__(ROUTE_WARPS * 32)
softmax_topk_kernel(float* __restrict__ logits, int T, int E, int K, int renorm,
                    int32_t* __restrict__ ids, float* __restrict__ wout,
                    float* __restrict__ ppart, const float* __restrict__ lpart, int nsplit,
                    const float* __restrict__ bias, const float* __restrict__ sel_bias,
                    const RoutePlan plan) {
  __shared__ float s_p[ROUTE_WARPS][VPT * 32];
  __shared__ int s_wcnt[PLAN ? ROUTE_WARPS : 1][PLAN ? 256 : 1];  // per-warp running counts
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the dispatch scan, launched as a programmatic dependent, may be scheduled as soon as
  // every block of this grid has started; it waits for this grid's results
  griddep_launch();
  // the aux statistics read the layout of the partial sums (this grid's size) from here
  if (blockIdx.x == 0 && threadIdx.x == 0) plan.hdr[HDR_ROUTE_NBLK] = gridDim.x;
  const int blk = blockIdx.x;
  if (PLAN) {
    for (int i = threadIdx.x; i < ROUTE_WARPS * 256; i += blockDim.x) (&s_wcnt[0][0])[i] = 0;
    __syncthreads();
  }
  int my_rank[TPW];  // PLAN: rank of this lane's assignment among the warp's earlier ones
  int my_pick[TPW];  //   and its expert (-1: no assignment)
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    my_rank[i] = 0;
    my_pick[i] = -1;
  }
  float pacc[VPT];
  float sb[VPT];  // selection-only bias of this lane's experts (0 without one)
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int e = lane + 32 * j;
    pacc[j] = 0.f;
    sb[j] = (sel_bias != nullptr && e < E) ? sel_bias[e] : 0.f;
  }

  const int t0 = (blk * ROUTE_WARPS + warp) * TPW;
  // the warp's token rows are loaded up front: one memory latency for all of them.  With
  // a split-K router the logits are the partial slices summed in slice order, plus the
  // bias; they are written back to `logits`.
  float vv[TPW][VPT];
  const size_t stride = (size_t)T * E;
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int t = t0 + i;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e = lane + 32 * j;
      float v = -INFINITY;
      if (t < T && e < E) {
        const size_t o = (size_t)t * E + e;
        if (lpart == nullptr) {
          v = logits[o];
        } else {
          v = lpart[o];
          for (int sp = 1; sp < nsplit; ++sp) v += lpart[sp * stride + o];
          if (bias != nullptr) v += bias[e];
          logits[o] = v;
        }
      }
      vv[i][j] = v;
    }
  }
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int t = t0 + i;
    if (t >= T) break;  // warp-uniform
    float v[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) v[j] = vv[i][j];
    // softmax: max, sum of exp, normalise
    float m = v[0];
#pragma unroll
    for (int j = 1; j < VPT; ++j) m = fmaxf(m, v[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float p[VPT];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e = lane + 32 * j;
      p[j] = (e < E) ? expf(v[j] - m) : 0.f;
      s += p[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      p[j] = p[j] / s;
      pacc[j] += p[j];
    }
    // top-K: K rounds of a warp arg-max under (score desc, id asc); the score is the
    // logit, plus the selection-only bias when there is one (one fp32 addition)
    float sc[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) sc[j] = (sel_bias != nullptr) ? __fadd_rn(v[j], sb[j]) : v[j];
    int my_id = 0;
    float my_w = 0.f, wsum = 0.f;
    if constexpr (VPT <= 4) {
      // this lane's candidates, sorted once by (score desc, id asc): key = order-preserving
      // integer image of the score (0: no candidate), with the expert's probability and j;
      // each round the warp picks the largest head key and, among the lanes holding it,
      // the lowest id, and the pick's owner drops its head (measured faster than a fresh
      // scan of the lane's candidates per round up to 4 candidates per lane)
      uint32_t ck[VPT];
      float cp[VPT];
      int cj[VPT];
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        ck[j] = (lane + 32 * j < E) ? score_key(sc[j]) : 0u;
        cp[j] = p[j];
        cj[j] = j;
      }
#pragma unroll
      for (int pass = 0; pass < VPT; ++pass) {  // odd-even transposition sort
#pragma unroll
        for (int a = pass & 1; a + 1 < VPT; a += 2) {
          const bool sw = ck[a + 1] > ck[a] || (ck[a + 1] == ck[a] && cj[a + 1] < cj[a]);
          if (sw) {
            const uint32_t tk = ck[a]; ck[a] = ck[a + 1]; ck[a + 1] = tk;
            const float tp = cp[a]; cp[a] = cp[a + 1]; cp[a + 1] = tp;
            const int tj = cj[a]; cj[a] = cj[a + 1]; cj[a + 1] = tj;
          }
        }
      }
      for (int k = 0; k < K; ++k) {
        const uint32_t top = __reduce_max_sync(0xffffffffu, ck[0]);
        const int bi = (int)__reduce_min_sync(
            0xffffffffu, ck[0] == top ? (uint32_t)(lane + 32 * cj[0]) : 0xffffffffu);
        const int owner = bi & 31;
        const float pw = __shfl_sync(0xffffffffu, cp[0], owner);
        if (lane == owner) {
#pragma unroll
          for (int j = 0; j + 1 < VPT; ++j) {
            ck[j] = ck[j + 1];
            cp[j] = cp[j + 1];
            cj[j] = cj[j + 1];
          }
          ck[VPT - 1] = 0u;
        }
        if (lane == k) {
          my_id = bi;
          my_w = pw;
        }
        wsum += pw;
      }
    } else {
      // eight candidates per lane: each round every lane rescans its untaken candidates
      // (equal scores: the lower j, i.e. the lower id), then the warp's largest key and,
      // among the lanes holding it, the lowest id
      uint32_t taken = 0;
      uint32_t key[VPT];  // order-preserving integer image of each score (0: no candidate)
#pragma unroll
      for (int j = 0; j < VPT; ++j) key[j] = (lane + 32 * j < E) ? score_key(sc[j]) : 0u;
      for (int k = 0; k < K; ++k) {
        uint32_t bk = 0;
        int be = INT_MAX;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
          const uint32_t kj = ((taken >> j) & 1u) ? 0u : key[j];
          if (kj > bk) {
            bk = kj;
            be = lane + 32 * j;
          }
        }
        const uint32_t top = __reduce_max_sync(0xffffffffu, bk);
        const int bi = (int)__reduce_min_sync(0xffffffffu, bk == top ? (uint32_t)be : 0xffffffffu);
        const int owner = bi & 31, jw = bi >> 5;
        float mine = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
          if (j == jw) mine = p[j];
        if (lane == owner) taken |= 1u << jw;
        const float pw = __shfl_sync(0xffffffffu, mine, owner);
        if (lane == k) {
          my_id = bi;
          my_w = pw;
        }
        wsum += pw;
      }
    }
    if (renorm) my_w = my_w / wsum;
    if (lane < K) {
      ids[(size_t)t * K + lane] = my_id;
      wout[(size_t)t * K + lane] = my_w;
    }
    if (PLAN) {
      // a token's K experts are distinct, so lane k's expert is counted once per token;
      // the warp's tokens are ranked in order
      my_pick[i] = lane < K ? my_id : -1;
      my_rank[i] = 0;
      if (lane < K) {
        my_rank[i] = s_wcnt[warp][my_id];
        s_wcnt[warp][my_id] = my_rank[i] + 1;
      }
      __syncwarp();
    }
  }
#pragma unroll
  for (int j = 0; j < VPT; ++j) s_p[warp][lane + 32 * j] = pacc[j];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < ROUTE_WARPS; ++w) acc += s_p[w][e];
    ppart[(size_t)e * gridDim.x + blk] = acc;
  }
  if (!PLAN) return;

  // ---- dispatch plan: exclusive prefix of the warps' counts per expert (the warps hold
  // consecutive tokens), the block's count per expert, and each assignment's rank in
  // the block
  const int nblk = gridDim.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int agg = 0;
#pragma unroll
    for (int w = 0; w < ROUTE_WARPS; ++w) {
      const int c = s_wcnt[w][e];
      s_wcnt[w][e] = agg;
      agg += c;
    }
    plan.pcnt[(size_t)e * nblk + blk] = agg;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int t = t0 + i;
    if (t < T && my_pick[i] >= 0)
      plan.pos[(size_t)t * K + lane] = s_wcnt[warp][my_pick[i]] + my_rank[i];
  }
}

// Plan scan: block e replaces the counts of expert e in the routing blocks (pcnt row e)
// by their exclusive prefix sums and records the total; the last block to finish writes
// counts (the totals, before dropping) and offsets (the exclusive scan over the experts
// of min(total, C), or of the totals when C < 0), and resets the finished counter.
constexpr int PLAN_SCAN_THREADS = 256;
constexpr int PLAN_SCAN_PER = 8;  // consecutive counts per thread in one pass

__global__ void __launch_bounds__(PLAN_SCAN_THREADS)
plan_scan_kernel(int32_t* __restrict__ pcnt, int nblk, int E, int C, int32_t* __restrict__ ptot,
                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets, uint32_t* hdr) {
  __shared__ int s_warp[PLAN_SCAN_THREADS / 32];
  __shared__ bool s_last;
  griddep_wait();    // the counts come from the routing kernel
  griddep_launch();  // the dispatch may be scheduled; it waits for this grid
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* row = pcnt + (size_t)e * nblk;
  int carry = 0;
  for (int b0 = 0; b0 < nblk; b0 += PLAN_SCAN_THREADS * PLAN_SCAN_PER) {
    const int first = b0 + tid * PLAN_SCAN_PER;
    int v[PLAN_SCAN_PER];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < PLAN_SCAN_PER; ++j) {
      v[j] = first + j < nblk ? row[first + j] : 0;
      sum += v[j];
    }
    // exclusive scan of the threads' sums: within the warp, then over the warps
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = carry;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    int chunk = 0;
    for (int w = 0; w < PLAN_SCAN_THREADS / 32; ++w) chunk += s_warp[w];
    __syncthreads();  // s_warp is rewritten by the next pass
    int run = before + incl - sum;
#pragma unroll
    for (int j = 0; j < PLAN_SCAN_PER; ++j) {
      if (first + j < nblk) row[first + j] = run;
      run += v[j];
    }
    carry += chunk;
  }
  if (tid == 0) {
    ptot[e] = carry;
    __threadfence();
    s_last = atomicAdd(&hdr[HDR_PLAN_DONE], 1u) == (uint32_t)(gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;  // block-uniform
  __threadfence();
  int total = 0;
  if (tid < E) total = *(volatile int32_t*)&ptot[tid];
  // E <= 256 = blockDim: one thread per expert
  int kept = tid < E ? ((C < 0) ? total : min(total, C)) : 0;
  if (tid < E) counts[tid] = total;
  int incl = kept;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += s_warp[w];
  if (tid < E) offsets[tid + 1] = before + incl;
  if (tid == 0) {
    offsets[0] = 0;
    hdr[HDR_PLAN_DONE] = 0u;
  }
}

cudaError_t launch_plan_scan(int32_t* pcnt, int nblk, int E, int C, int32_t* ptot, int32_t* counts,
                             int32_t* offsets, uint32_t* hdr, cudaStream_t st) {
  const cudaError_t e = launch_dependent(plan_scan_kernel, dim3(E), dim3(PLAN_SCAN_THREADS), 0,
                                         st, pcnt, nblk, E, C, ptot, counts, offsets, hdr);
  count_launch();
  return e;
}

// lpart == nullptr: `logits` is the input.  Otherwise the logits are the sum of nsplit
// partial slices of lpart (+ bias), and are also written to `logits`.  `plan` carries the
// workspace header (always) and, for the dispatch plan, its buffers (plan->pos != null).
cudaError_t launch_softmax_topk(float* logits, int T, int E, int K, int renorm, int32_t* ids,
                                float* w, float* ppart, const float* lpart, int nsplit,
                                const float* bias, const float* sel_bias, const RoutePlan& plan,
                                cudaStream_t st) {
  const bool planned = plan.pos != nullptr;
  const int tpw = planned ? route_plan_tpw(T) : route_tpw(T);
  const dim3 grid(route_blocks(T, tpw)), block(ROUTE_WARPS * 32);
#define MOE_SOFTMAX_TOPK(V, P, PL)                                                                \
  softmax_topk_kernel<V, P, PL><<<grid, block, 0, st>>>(logits, T, E, K, renorm, ids, w, ppart,    \
                                                         lpart, nsplit, bias, sel_bias, plan)
#define MOE_SOFTMAX_TOPK_TPW(V)                                                                  \
  do {                                                                                           \
    if (!planned) {                                                                              \
      if (tpw == 4) MOE_SOFTMAX_TOPK(V, 4, false); else MOE_SOFTMAX_TOPK(V, 1, false);           \
    } else {                                                                                     \
      if (tpw == 4) MOE_SOFTMAX_TOPK(V, 4, true); else MOE_SOFTMAX_TOPK(V, 1, true);             \
    }                                                                                            \
  } while (0)
  if (E <= 32) MOE_SOFTMAX_TOPK_TPW(1);
  else if (E <= 64) MOE_SOFTMAX_TOPK_TPW(2);
  else if (E <= 128) MOE_SOFTMAX_TOPK_TPW(4);
  else MOE_SOFTMAX_TOPK_TPW(8);
#undef MOE_SOFTMAX_TOPK_TPW
#undef MOE_SOFTMAX_TOPK
  count_launch();
  return cudaGetLastError();
}

// Selection-bias adjustment after a step: b_i += gamma * sign(T*K/E - count_i), the
// comparison with the mean load done exactly in integers, the sum rounded once to fp32.
__global__ void adjust_select_bias_kernel(const int32_t* __restrict__ counts,
                                          float* __restrict__ sel_bias, int E, int64_t A,
                                          float gamma) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int64_t diff = A - (int64_t)counts[e] * E;
  const float step = diff > 0 ? gamma : (diff < 0 ? -gamma : 0.f);
  sel_bias[e] = __fadd_rn(sel_bias[e], step);
}

cudaError_t launch_adjust_select_bias(const int32_t* counts, float* sel_bias, int E, int64_t A,
                                      float gamma, cudaStream_t st) {
  adjust_select_bias_kernel<<<(E + 255) / 256, 256, 0, st>>>(counts, sel_bias, E, A, gamma);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
