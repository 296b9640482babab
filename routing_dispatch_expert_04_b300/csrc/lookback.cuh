// The per-expert running count behind the capacity rule ("Top-K Routing and Capacity
// Factor": an assignment is dropped when its expert already holds C assignments that
// arrived before it), computed over chunks of the arrival-ordered assignment stream by
// a single-pass decoupled look-back (the dispatch scan, scan.cu).
//
// Every chunk, in the order of an atomic ticket (so each chunk a block waits for is held
// by a block that has already started), publishes per expert one descriptor word:
//   flag (2 bits: own count, or inclusive total of chunks 0..b) | epoch (30 bits) | count.
// A descriptor counts as published only with the current call's epoch; the block that
// finishes a call last resets the ticket and starts the next epoch, so no call has to
// clear the previous call's descriptors.  Every wait is bounded: past `spin_limit` polls
// the block records a timeout in the status word and carries on.
#pragma once

#include "common.cuh"

namespace moe {

constexpr unsigned long long FLAG_AGG = 1ull << 62;   // this chunk's own count
constexpr unsigned long long FLAG_INCL = 2ull << 62;  // total of chunks 0..this one
constexpr unsigned long long FLAG_MASK = 3ull << 62;
constexpr uint32_t EPOCH_MASK = 0x3FFFFFFFu;

__device__ __forceinline__ unsigned long long epoch_tag(uint32_t epoch) {
  return (unsigned long long)(epoch & EPOCH_MASK) << 32;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// One thread per expert e: publishes chunk b's count `agg` of expert e, returns the
// count of e in chunks 0..b-1, and publishes the inclusive total.  desc_e points at
// chunk 0's descriptor of expert e; consecutive chunks are E words apart.  The next W
// predecessors' descriptors are loaded together, then walked from the nearest:
// their counts add up until an inclusive total ends the walk; an unpublished one is
// polled again.  Flag and count share one 64-bit word, so relaxed loads suffice (acquire
// loads would serialise).  `publish` = false withholds this chunk's descriptors (the
// bounded-wait test hook).
template <int W>
__device__ __forceinline__ int lookback_exclusive(unsigned long long* desc_e, int E, int b, int agg,
                                                  unsigned long long tag, bool publish,
                                                  int spin_limit, uint32_t* hdr) {
  unsigned long long* mine = desc_e + (size_t)b * E;
  if (b == 0) {
    if (publish) st_release_u64(mine, FLAG_INCL | tag | (uint32_t)agg);
    return 0;
  }
  if (publish) st_release_u64(mine, FLAG_AGG | tag | (uint32_t)agg);
  int excl = 0;
  int j = b - 1, spins = 0;
  while (j >= 0) {
    unsigned long long v[W];
#pragma unroll
    for (int i = 0; i < W; ++i)
      v[i] = (j - i >= 0) ? ld_relaxed_u64(desc_e + (size_t)(j - i) * E) : (FLAG_INCL | tag);
    int used = 0;
    bool stop = false, blocked = false;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      if (!stop && !blocked) {
        const unsigned long long flag = v[i] & FLAG_MASK;
        if (flag == 0 || (v[i] & ~FLAG_MASK & ~0xffffffffull) != tag) {  // not yet published
          blocked = true;
        } else {
          excl += (int)(uint32_t)v[i];
          ++used;
          stop = (flag == FLAG_INCL);
        }
      }
    }
    if (stop) break;
    j -= used;
    if (blocked) {
      if (++spins > spin_limit) {
        raise_error(hdr, DEV_ERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
  }
  if (publish) st_release_u64(mine, FLAG_INCL | tag | (uint32_t)(excl + agg));
  return excl;
}

// The last chunk's block: grand totals (counts, before dropping), kept = min(total, C)
// (C < 0: all), and offsets = their exclusive scan over the experts (a warp scan of each
// 32 experts, then the sums of the earlier warps).  `total` is expert tid's grand total
// for tid < E; s_warp is shared scratch of at least blockDim/32 ints.  Block-uniform.
__device__ __forceinline__ void write_counts_offsets(int total, int E, int C, int32_t* counts,
                                                     int32_t* offsets, int* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int kept = 0;
  if (tid < E) {
    counts[tid] = total;
    kept = (C < 0) ? total : min(total, C);
  }
  int incl = kept;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += s_warp[w];
  if (tid < E) offsets[tid + 1] = before + incl;
  if (tid == 0) offsets[0] = 0;
}

// Called by every block once it is done with the descriptors (block-uniform): the last
// of the call's nblk blocks resets the ticket (hdr[ticket]) and the finished counter
// (hdr[finished]) and starts the next epoch (hdr[epoch]).
__device__ __forceinline__ void finish_lookback_call(uint32_t* hdr, int ticket, int finished,
                                                     int epoch_word, uint32_t epoch, int nblk) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&hdr[finished], 1u) == (uint32_t)(nblk - 1)) {
      hdr[ticket] = 0u;
      hdr[finished] = 0u;
      hdr[epoch_word] = (epoch + 1u) & EPOCH_MASK;
      __threadfence();
    }
  }
}

// Workspace header words of the dispatch scan's look-back.
constexpr int HDR_SCAN_TICKET = 1, HDR_SCAN_DONE = 3, HDR_SCAN_EPOCH = 4;

}  // namespace moe
