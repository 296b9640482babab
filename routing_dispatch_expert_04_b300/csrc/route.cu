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
#include <math.h>
#include <limits.h>

#include "common.cuh"
#include "lookback.cuh"

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
  __shared__ int s_excl[PLAN ? 256 : 1];
  __shared__ int s_blk;
  __shared__ uint32_t s_epoch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the dispatch scan, launched as a programmatic dependent, may be scheduled as soon as
  // every block of this grid has started; it waits for this grid's results
  griddep_launch();
  // the aux statistics read the layout of the partial sums (this grid's size) from here
  if (blockIdx.x == 0 && threadIdx.x == 0) plan.hdr[HDR_ROUTE_NBLK] = gridDim.x;
  int blk = blockIdx.x;
  if (PLAN) {
    // tokens go to blocks in ticket order, so every chunk the look-back waits for belongs
    // to a block that has started
    if (threadIdx.x == 0) {
      s_blk = (int)atomicAdd(&plan.hdr[HDR_PLAN_TICKET], 1u);
      s_epoch = *(volatile uint32_t*)&plan.hdr[HDR_PLAN_EPOCH];
    }
    for (int i = threadIdx.x; i < ROUTE_WARPS * 256; i += blockDim.x) (&s_wcnt[0][0])[i] = 0;
    __syncthreads();
    blk = s_blk;
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
  // consecutive tokens), the block's count, then the two-level look-back over the blocks
  // (groups of PLAN_GROUP blocks, then the groups)
  const int nblk = gridDim.x;
  const unsigned long long tag = epoch_tag(s_epoch);
  const int e = threadIdx.x;  // E <= 256 = blockDim
  int agg = 0;
  if (e < E) {
#pragma unroll
    for (int w = 0; w < ROUTE_WARPS; ++w) {
      const int c = s_wcnt[w][e];
      s_wcnt[w][e] = agg;
      agg += c;
    }
    s_excl[e] = grouped_lookback_exclusive<PLAN_GROUP, 16>(
        plan.desc + e, plan.desc + (size_t)nblk * E + e, E, blk, nblk, agg, tag,
        blk != plan.skip_block, plan.spin_limit, plan.hdr);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int t = t0 + i;
    if (t < T && my_pick[i] >= 0)
      plan.pos[(size_t)t * K + lane] = s_excl[my_pick[i]] + s_wcnt[warp][my_pick[i]] + my_rank[i];
  }
  if (blk == nblk - 1) {  // block-uniform
    __syncthreads();
    write_counts_offsets(e < E ? s_excl[e] + agg : 0, E, plan.C, plan.counts, plan.offsets,
                         &s_wcnt[0][0]);
  }
  finish_lookback_call(plan.hdr, HDR_PLAN_TICKET, HDR_PLAN_DONE, HDR_PLAN_EPOCH, s_epoch, nblk);
}

// lpart == nullptr: `logits` is the input.  Otherwise the logits are the sum of nsplit
// partial slices of lpart (+ bias), and are also written to `logits`.  `plan` carries the
// workspace header (always) and, for the dispatch plan, its buffers (plan->pos != null).
cudaError_t launch_softmax_topk(float* logits, int T, int E, int K, int renorm, int32_t* ids,
                                float* w, float* ppart, const float* lpart, int nsplit,
                                const float* bias, const float* sel_bias, const RoutePlan& plan,
                                cudaStream_t st) {
  const bool planned = plan.pos != nullptr;
  const int tpw = planned ? route_plan_tpw(T, E) : route_tpw(T);
  const dim3 grid(route_blocks(T, tpw)), block(ROUTE_WARPS * 32);
#define MOE_SOFTMAX_TOPK(V, P, PL)                                                                \
  softmax_topk_kernel<V, P, PL><<<grid, block, 0, st>>>(logits, T, E, K, renorm, ids, w, ppart,    \
                                                         lpart, nsplit, bias, sel_bias, plan)
#define MOE_SOFTMAX_TOPK_TPW(V)                                                                  \
  do {                                                                                           \
    if (!planned) {                                                                              \
      if (tpw == 4) MOE_SOFTMAX_TOPK(V, 4, false); else MOE_SOFTMAX_TOPK(V, 1, false);           \
    } else if (tpw == 16) {                                                                      \
      if constexpr (V <= 2) MOE_SOFTMAX_TOPK(V, 16, true);                                       \
    } else if (tpw == 8) {                                                                       \
      if constexpr (V <= 4) MOE_SOFTMAX_TOPK(V, 8, true);                                        \
    } else if (tpw == 4) {                                                                       \
      MOE_SOFTMAX_TOPK(V, 4, true);                                                              \
    } else {                                                                                     \
      MOE_SOFTMAX_TOPK(V, 1, true);                                                              \
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
