// Per-expert histogram, capacity, drop mask and the dispatch permutation.
//
// "Expert Parallelism (MoE)", "Top-K Routing and Capacity Factor": each expert accepts
// at most C assignments; assignments that would push an expert over capacity are
// dropped and their routing weight is zeroed.  "The All-to-All Communication": after
// routing, every token is sent to the holder of each chosen expert; on one GPU the
// all-to-all becomes a permutation that packs each expert's rows contiguously.
//
// Order fixed here: assignments arrive in flat order a = t*K + k (or, with the
// slot-major drop priority, every token's k-th choice before any (k+1)-th).  An
// assignment's position in its expert is the number of assignments to the same expert
// that arrived before it; it is kept iff that position is below C, and kept rows of
// expert e are packed at offsets[e] + position.  The result is unique, so it can be
// compared bit for bit.
//
// scan_kernel -- one pass over the flat id stream.  Each block takes a chunk of
// SCAN_ITEMS assignments (chunk index drawn from an atomic ticket, so every block it
// waits for has already started).  Each warp ranks a contiguous segment of the chunk
// per expert with warp match/popc and a warp-private running count in shared memory;
// one prefix over the warps turns those into chunk ranks.  The block publishes its
// per-expert totals, and obtains the totals of all earlier chunks by a decoupled look-back with
// one descriptor per (chunk, expert), reading up to 32 of them per round.  The
// descriptors carry the call's epoch and the last block to finish resets the ticket, so
// consecutive calls need no clearing of the workspace in between.  Both kernels are
// launched as programmatic dependents of their predecessor on the stream: they are
// scheduled while it finishes and wait for its results (griddepcontrol) before reading them.  Every wait is bounded: past `spin_limit` polls
// the block records a timeout in the status word and carries on, so the kernel always
// terminates.  The last chunk knows the grand totals and writes counts and offsets.
//
// dispatch_kernel -- one warp per token: turns positions into packed rows (slot, src)
// and copies the token's row once from HBM into each of its kept packed rows with
// 16-byte loads and stores (a token with no kept row is not read).
#include "common.cuh"
#include "lookback.cuh"

namespace moe {

// Flat assignment index (t*K + k) of the i-th assignment in arrival order: token-major
// (the identity) or slot-major (every token's k-th choice before any (k+1)-th).
__device__ __forceinline__ int64_t arrival_to_flat(int64_t i, int slot_major, int Tn, int K) {
  return slot_major ? (i % Tn) * K + i / Tn : i;
}

// Lanes of the warp whose expert id equals this lane's: the ids compared bit plane by bit
// plane with ballots (one per bit of E - 1, plus one separating invalid ids, -1), which
// takes far fewer cycles than a match instruction when a warp holds many distinct ids.
__device__ __forceinline__ uint32_t same_id_lanes(int e, int nbits) {
  const uint32_t valid = __ballot_sync(0xffffffffu, e >= 0);
  uint32_t m = e >= 0 ? valid : ~valid;
#pragma unroll
  for (int bit = 0; bit < 8; ++bit) {
    if (bit < nbits) {
      const bool on = (e >> bit) & 1;
      const uint32_t plane = __ballot_sync(0xffffffffu, on);
      m &= on ? plane : ~plane;
    }
  }
  return m;
}

__global__ void __launch_bounds__(SCAN_THREADS)
scan_kernel(const int32_t* __restrict__ ids, int A, int E, int C, int nblk,
            unsigned long long* desc, int32_t* __restrict__ pos, int32_t* __restrict__ counts,
            int32_t* __restrict__ offsets, uint32_t* hdr, int skip_block, int spin_limit,
            int slot_major, int Tn, int K) {
  constexpr int NW = SCAN_THREADS / 32;
  constexpr int WITEMS = SCAN_IPT * 32;  // each warp ranks one contiguous segment
  __shared__ int s_wrun[NW][256];        // per-warp running count of e, then warp base
  __shared__ int s_run[256];             // count of e in this chunk
  __shared__ int s_excl[256];            // count of e in all earlier chunks
  __shared__ int s_b;
  __shared__ uint32_t s_epoch;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  griddep_wait();    // the ids come from the routing kernel
  griddep_launch();  // the row copy may be scheduled once every chunk has started
  if (tid == 0) {
    s_b = (int)atomicAdd(&hdr[HDR_SCAN_TICKET], 1u);
    s_epoch = *(volatile uint32_t*)&hdr[HDR_SCAN_EPOCH];
  }
  for (int i = tid; i < NW * 256; i += SCAN_THREADS) (&s_wrun[0][0])[i] = 0;
  __syncthreads();
  const int b = s_b;
  const unsigned long long tag = epoch_tag(s_epoch);
  const int64_t base = (int64_t)b * SCAN_ITEMS;
  const int64_t wbase = base + (int64_t)warp * WITEMS;
  uint32_t lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));

  // this lane's ids, loaded up front: one memory latency for the whole segment
  int my_e[SCAN_IPT], my_r[SCAN_IPT];
#pragma unroll
  for (int r = 0; r < SCAN_IPT; ++r) {
    const int64_t a = wbase + r * 32 + lane;
    my_e[r] = (a < A) ? ids[arrival_to_flat(a, slot_major, Tn, K)] : -1;
  }
#pragma unroll
  for (int r = 0; r < SCAN_IPT; ++r) {
    const int64_t a = wbase + r * 32 + lane;
    if (a < A && (my_e[r] < 0 || my_e[r] >= E)) {
      raise_error(hdr, DEV_ERR_BAD_ID);
      my_e[r] = -1;
    }
  }
  // rank inside the warp's segment, 32 assignments at a time, in flat order
  const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;
#pragma unroll
  for (int r = 0; r < SCAN_IPT; ++r) {
    const int e = my_e[r];
    const uint32_t peers = same_id_lanes(e, nbits);
    const int run = (e >= 0) ? s_wrun[warp][e] : 0;
    my_r[r] = run + __popc(peers & lt);
    __syncwarp();
    if (e >= 0 && (31 - __clz(peers)) == lane) s_wrun[warp][e] = run + __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // exclusive prefix of the per-warp counts (earlier warps hold earlier assignments)
  for (int e = tid; e < E; e += SCAN_THREADS) {
    int acc = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int c = s_wrun[w][e];
      s_wrun[w][e] = acc;
      acc += c;
    }
    s_run[e] = acc;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < SCAN_IPT; ++r)
    if (my_e[r] >= 0) my_r[r] += s_wrun[warp][my_e[r]];

  // decoupled look-back, one thread per expert
  if (tid < E)
    s_excl[tid] = lookback_exclusive<32>(desc + tid, E, b, s_run[tid], tag, b != skip_block, spin_limit,
                                     hdr);
  __syncthreads();

#pragma unroll
  for (int r = 0; r < SCAN_IPT; ++r) {
    if (my_e[r] >= 0)
      pos[arrival_to_flat(wbase + r * 32 + lane, slot_major, Tn, K)] = s_excl[my_e[r]] + my_r[r];
  }

  if (b == nblk - 1) {  // block-uniform
    __syncthreads();  // every thread has read its chunk counts from s_run
    write_counts_offsets(tid < E ? s_excl[tid] + s_run[tid] : 0, E, C, counts, offsets, s_run);
  }
  finish_lookback_call(hdr, HDR_SCAN_TICKET, HDR_SCAN_DONE, HDR_SCAN_EPOCH, s_epoch, nblk);
}

template <typename T>
__global__ void __launch_bounds__(256)
dispatch_kernel(const T* __restrict__ x, const int32_t* __restrict__ ids,
                const int32_t* __restrict__ pos, const int32_t* __restrict__ base, int nbase,
                int tpb, const int32_t* __restrict__ offsets, int Tn, int d, int E, int K, int C,
                int32_t* __restrict__ slot, int32_t* __restrict__ src, T* __restrict__ xp,
                int64_t rows_cap, uint32_t* hdr) {
  __shared__ int s_slot[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = d / Elem<T>::PER16;
  griddep_wait();  // positions and offsets come from the scan
  for (int t = blockIdx.x * 8 + warp; t < Tn; t += gridDim.x * 8) {
    if (lane < K) {
      const int64_t a = (int64_t)t * K + lane;
      const int e = ids[a];
      int s = -1;
      if (e >= 0 && e < E) {
        // with a per-block base (the plan from the routing kernel), pos is the rank inside
        // the token's routing block of tpb tokens
        const int p = pos[a] + (base != nullptr ? base[(size_t)e * nbase + t / tpb] : 0);
        if (C < 0 || p < C) s = offsets[e] + p;
      }
      if (s >= rows_cap) {
        raise_error(hdr, DEV_ERR_OVERFLOW);
        s = -1;
      }
      slot[a] = s;
      if (s >= 0) src[s] = (int32_t)a;
      s_slot[warp][lane] = s;
    }
    // a token whose assignments were all dropped is not read at all
    const bool kept_any = __any_sync(0xffffffffu, lane < K && s_slot[warp][lane < K ? lane : 0] >= 0);
    __syncwarp();
    if (xp != nullptr && kept_any) {
      const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
      int j = lane;
      for (; j + 96 < nvec; j += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = ld_nc_v4(xr + j + 32 * u);
        for (int k = 0; k < K; ++k) {
          const int s = s_slot[warp][k];
          if (s < 0) continue;
          uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)s * d) + j;
#pragma unroll
          for (int u = 0; u < 4; ++u) st_v4(dst + 32 * u, v[u]);
        }
      }
      for (; j < nvec; j += 32) {
        const uint4 v = ld_nc_v4(xr + j);
        for (int k = 0; k < K; ++k) {
          const int s = s_slot[warp][k];
          if (s >= 0) st_v4(reinterpret_cast<uint4*>(xp + (size_t)s * d) + j, v);
        }
      }
    }
    __syncwarp();
  }
}

cudaError_t launch_scan(const int32_t* ids, int A, int E, int C, int nblk, unsigned long long* desc,
                        int32_t* pos, int32_t* counts, int32_t* offsets, uint32_t* hdr,
                        int skip_block, int spin_limit, int slot_major, int Tn, int K,
                        cudaStream_t st) {
  const cudaError_t e = launch_dependent(scan_kernel, dim3(nblk), dim3(SCAN_THREADS), 0, st, ids, A,
                                         E, C, nblk, desc, pos, counts, offsets, hdr, skip_block,
                                         spin_limit, slot_major, Tn, K);
  count_launch();
  return e;
}

cudaError_t launch_dispatch(int dtype, const void* x, const int32_t* ids, const int32_t* pos,
                            const int32_t* base, int nbase, int tpb, const int32_t* offsets,
                            int Tn, int d, int E, int K, int C, int32_t* slot, int32_t* src,
                            void* xp, int64_t rows_cap, uint32_t* hdr, int num_sms,
                            cudaStream_t st) {
  const int want = (Tn + 7) / 8;
  const int grid = want < num_sms * 16 ? want : num_sms * 16;
  cudaError_t e;
  if (dtype == MOE_BF16)
    e = launch_dependent(dispatch_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st,
                         (const __nv_bfloat16*)x, ids, pos, base, nbase, tpb, offsets, Tn, d, E,
                         K, C, slot, src, (__nv_bfloat16*)xp, rows_cap, hdr);
  else
    e = launch_dependent(dispatch_kernel<float>, dim3(grid), dim3(256), 0, st, (const float*)x, ids,
                         pos, base, nbase, tpb, offsets, Tn, d, E, K, C, slot, src, (float*)xp,
                         rows_cap, hdr);
  count_launch();
  return e;
}

}  // namespace moe
