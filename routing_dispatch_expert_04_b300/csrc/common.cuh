// Shared device helpers, workspace layout and launch bookkeeping of the MoE layer library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------------------ device status word
// Bits OR-ed into ws header word 0 by kernels; moe_sync_status maps them to a status.
constexpr uint32_t DEV_ERR_TIMEOUT = 1u;   // a bounded spin-wait gave up
constexpr uint32_t DEV_ERR_BAD_ID = 2u;    // expert id outside [0, E)
constexpr uint32_t DEV_ERR_OVERFLOW = 4u;  // offsets[G] larger than the row buffer
constexpr uint32_t DEV_ERR_RANGE = 8u;     // a value outside the fp16 range was stored

__device__ __forceinline__ void raise_error(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

// ------------------------------------------------------------------ workspace layout
// [0, 256)        header: u32 status, u32 scan ticket, u32 aux ticket, u32 scan blocks
//                 finished, u32 scan epoch (the look-back descriptors of one dispatch call
//                 carry its epoch, so no call has to clear those of the previous one), two
//                 unused words, u32 plan-scan blocks finished, u32 routing blocks of the
//                 last routing call; bytes 64..79 clock telemetry
// desc            scan descriptors, nblk_scan * E * u64 (flag << 32 | value)
// pos             A * i32, position of each assignment inside its expert (pre-drop); with
//                 the plan in the routing kernel, its rank inside its routing block
// ppart           E * nblk * f32, per-block sums of softmax probabilities (nblk = the
//                 routing grid of the last routing call, which it records in header word 8)
// auxfp           E * f64, per-expert f_i * P_i for the final fixed-order sum
// lpart           router_splits * T * E * f32, partial router logits (split-K router only)
// pcnt            E * nblk * i32, the routing kernel's plan: each routing block's count per
//                 expert, replaced by the plan scan with the count in all earlier blocks
// ptot            E * i32, each expert's total (plan scan)
constexpr int SCAN_THREADS = 256;
constexpr int SCAN_IPT = 16;
constexpr int SCAN_ITEMS = SCAN_THREADS * SCAN_IPT;  // assignments per scan block
constexpr int ROUTE_WARPS = 8;

// Tokens per warp of the softmax/top-K kernel: four (more loads in flight per warp)
// when the batch has enough tokens to keep every SM busy with a quarter as many warps,
// one otherwise (measured on B300, routing stage: T=65536 E=8 0.130 vs 0.135 ms with 4;
// T=16384 E=128 0.045 vs 0.049 ms and T=8192 E=256 0.074 vs 0.115 ms with 1).
inline int route_tpw(int T) { return T >= 32768 ? 4 : 1; }

// Tokens per warp of the routing kernel when it also computes the dispatch plan: the same
// as without, so both paths sum the probabilities over the same token groups.
inline int route_plan_tpw(int T) { return route_tpw(T); }
inline int route_blocks(int T, int tpw) {
  const int per = ROUTE_WARPS * tpw;
  return (int)(((int64_t)T + per - 1) / per);
}

// Workspace header word holding the routing grid (blocks) of the last routing call: the
// layout of the probability partial sums the aux statistics reduce.
constexpr int HDR_ROUTE_NBLK = 8;
// Header word counting the plan scan's finished blocks (reset by the last one).
constexpr int HDR_PLAN_DONE = 7;

struct WsLayout {
  size_t desc, pos, ppart, auxfp, lpart, pcnt, ptot, total;
  int nblk_scan, nblk_route, nblk_plan, router_splits;
};

// CTAs of the tensor-core router that share one SM: its E <= 64 variants stage in at
// most 100 KB of shared memory and hold at most 128 TMEM columns, so two fit (measured
// faster on the 64K-token layer); the wider variants take a whole SM (for E = 128, two
// 3-stage CTAs per SM measured slower than one 6-stage CTA).
inline int router_ctas_per_sm(int E) { return E <= 64 ? 2 : 1; }

// K splits of the tensor-core router: enough CTAs to fill the SMs' CTA slots when T/128
// row tiles alone would not (planned for 148 SMs; a smaller GPU just runs more waves),
// at most 8.  Every slice keeps at least one 64-wide k-block.
inline int router_splits(const moe_config& c) {
  if (c.dtype != MOE_BF16 || c.T <= 0) return 1;
  const int mt = (c.T + 127) / 128;
  const int nkb = (c.d + 63) / 64;
  int s = 148 * router_ctas_per_sm(c.E) / mt;
  if (s > 8) s = 8;
  if (s > nkb) s = nkb;
  if (s < 2) return 1;
  const int kpb = (nkb + s - 1) / s;
  return (nkb + kpb - 1) / kpb;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(const moe_config& c) {
  WsLayout L;
  int64_t A = (int64_t)c.T * c.K;
  L.nblk_scan = (int)((A + SCAN_ITEMS - 1) / SCAN_ITEMS);
  // the routing kernel runs route_blocks(T, route_tpw(T)) blocks, or with the dispatch plan
  // route_blocks(T, route_plan_tpw(T)); the per-block buffers hold the larger count
  L.nblk_route = route_blocks(c.T, route_tpw(c.T));
  L.nblk_plan = route_blocks(c.T, route_plan_tpw(c.T));
  const int nblk_rmax = L.nblk_route > L.nblk_plan ? L.nblk_route : L.nblk_plan;
  size_t off = 256;
  L.desc = off;
  off = align_up(off + (size_t)L.nblk_scan * c.E * 8, 256);
  L.pos = off;
  off = align_up(off + (size_t)A * 4, 256);
  L.ppart = off;
  off = align_up(off + (size_t)nblk_rmax * c.E * 4, 256);
  L.auxfp = off;
  off = align_up(off + (size_t)c.E * 8, 256);
  L.router_splits = router_splits(c);
  L.lpart = off;
  if (L.router_splits > 1) off = align_up(off + (size_t)L.router_splits * c.T * c.E * 4, 256);
  L.pcnt = off;
  off = align_up(off + (size_t)L.nblk_plan * c.E * 4, 256);
  L.ptot = off;
  off = align_up(off + (size_t)c.E * 4, 256);
  L.total = off;
  return L;
}

// The dispatch plan computed with the routing (token-major arrival order, moe_route_plan):
// the routing kernel ranks each block's assignments per expert in arrival order and
// writes the block's count per expert; the plan scan turns the counts into each block's
// count in all earlier blocks, and writes counts and offsets.  The dispatch adds the two.
struct RoutePlan {
  int32_t* pos;   // [T*K] rank of each assignment among its routing block's ones to its expert
  int32_t* pcnt;  // [E, nblk] count of each expert in each routing block
  uint32_t* hdr;  // workspace header
};

// ------------------------------------------------------------------ launch bookkeeping
void count_launch();

// Argument checks and sizes shared by the entry points (api.cu): the config's validity
// (MOE_OK or the error status), the rows of the packed buffers, and the scan test hook.
moe_status_t check_cfg(const moe_config* c);
int64_t rows_capacity(const moe_config& c);
void take_scan_test_hook(int* skip_block, int* spin_limit);

// ------------------------------------------------------------------ element helpers
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int PER16 = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                      __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  __device__ __forceinline__ static float to_f(float x) { return x; }
  __device__ __forceinline__ static float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int PER16 = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);  // .x = low half
      w[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while its predecessor on the stream is still running;
// griddep_wait() blocks until that predecessor has completed and its memory operations
// are visible (a no-op for a kernel launched the ordinary way), and griddep_launch() lets
// the successor be scheduled once every block of this grid has issued it.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// Launch with programmatic stream serialisation (see griddep_wait).
template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

}  // namespace moe
