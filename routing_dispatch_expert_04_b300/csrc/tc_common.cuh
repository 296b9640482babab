// Pieces shared by the one-CTA and the CTA-pair tcgen05 grouped GEMMs: the argument
// block, bounded mbarrier waits, the ragged (group, n-tile, m-tile) tile list built on
// the device from `offsets`, the fused epilogues and the TMA descriptor encoding.
//
// The GEMM is the expert FFN of "Expert Parallelism (MoE)", "MoE Layer Structure" (each
// expert applies Linear(d -> 4d) -> GELU -> Linear(4d -> d)) run for all experts in one
// launch ("Expert Parallelism (EP)", step 3: expert GEMMs compute locally):
//   C[r, n] = epi( sum_k A[r, k] * B[g*N + n, k] ),  r in [offsets[g], offsets[g+1]).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {

constexpr int TC_BK = 64;  // 64 bf16/fp16 = one 128-byte swizzle row
constexpr int TC_ROW_BYTES = 128;  // bytes of K per stage row (a 128-byte swizzle row)

// Operand kinds of the expert GEMMs.
enum { OP_BF16 = 0, OP_F16 = 1, OP_E4M3 = 2 };
template <int KIND> struct OpKind {
  static constexpr int BYTES = KIND == OP_E4M3 ? 1 : 2;
  static constexpr int BK = TC_ROW_BYTES / BYTES;  // K elements per stage
};
constexpr int TC_THREADS = 192;
constexpr int TC_THREADS_GATED = 224;  // + the watcher warp (warp 6)
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;
constexpr int TC_MAX_GROUPS = 256;

enum { TC_EPI_GELU_F16 = 0, TC_EPI_F32 = 1, TC_EPI_BIAS_F32 = 2, TC_EPI_F16 = 3 };

struct TcArgs {
  const int32_t* offsets;  // [G+1] device, or nullptr: one group of M rows
  int G, M, N, Kd;
  int64_t rows_cap;
  void* out;               // [rows_cap, ldo] (times ksplit partial slices)
  int ldo;
  const float* bias;       // [N] or nullptr (added only when ksplit == 1)
  uint32_t* hdr;           // status word
  int ksplit;              // K split across CTAs: slice s holds the partial sum of k-blocks
  int kpb;                 //   [s*kpb, min(nkb, (s+1)*kpb)); ksplit*kpb covers nkb, no slice empty
  int64_t split_stride;    // elements between the partial slices of `out`
  int row_part;            // rows of each group this launch covers: 0 all; 1 the leading
                           //   whole 256-row tiles; 2 the rest (fewer than 256 rows)
  const int32_t* gather_src;  // non-null: A row r is row gather_src[r] / gather_k of the
  int gather_k;               //   gathered matrix (token rows of X), which has
  int64_t gather_rows;        //   gather_rows rows
  const float* a_scale;    // E4M3 operands: per-row scale of A (per token row when gathered)
  const float* b_scale;    //   and of B (per row of the stacked weights, g*N + n)
};

// Token row of packed row r of a gathered A operand (row 0 for rows past the group,
// whose results are never stored; an out-of-range index is reported and replaced by 0).
__device__ __forceinline__ int gather_row(const TcArgs& args, int r, int rowend) {
  if (r >= rowend) return 0;
  const int tok = args.gather_src[r] / args.gather_k;
  if (tok < 0 || (int64_t)tok >= args.gather_rows) {
    raise_error(args.hdr, DEV_ERR_BAD_ID);
    return 0;
  }
  return tok;
}

constexpr int TC_ROWS_ALL = 0, TC_ROWS_FULL256 = 1, TC_ROWS_REST256 = 2;

// Group table in shared memory: row range, m-tile count and tile prefix per group.
struct GroupTable {
  int lo[TC_MAX_GROUPS + 1];
  int hi[TC_MAX_GROUPS + 1];
  int mt[TC_MAX_GROUPS + 1];
  int tpre[TC_MAX_GROUPS + 1];
};

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           uint32_t* hdr) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::globaltimer_ns();
  while (true) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (tc::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      raise_error(hdr, DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Stage gate between a watcher warp and the MMA warp: named barrier TC_GATE_BAR0 + s means
// "stage s holds its data".  A shared-memory access by the thread that issues the MMAs
// stalls while its MMAs are in flight (an mbarrier wait or a plain load, about 230 cycles
// each on B300), so the MMA warp waits on a named barrier and the watcher warp, which
// issues no MMAs, does the mbarrier waits.  The watcher arrives exactly once per stage
// the MMA warp syncs, in the same order, and never more than one round ahead of it: it
// waits for the stage's data, or, after a wait has given up, for the MMA warp's commit of
// the stage's previous round (or for the MMA warp to have left its loop, after which it
// stops arriving).
constexpr int TC_GATE_BAR0 = 1;
constexpr int TC_GATE_THREADS = 64;  // watcher warp + MMA warp

__device__ __forceinline__ bool gate_arrive(int s, uint64_t* full, uint64_t* empty, uint32_t ph,
                                            bool& gave_up, volatile int* abort_flag,
                                            volatile int* mma_left, uint32_t* hdr, int lane) {
  if (lane == 0) {
    if (!gave_up && !wait_phase(&full[s], ph, abort_flag, hdr)) gave_up = true;
    if (gave_up) {
      const uint64_t t0 = tc::globaltimer_ns();
      while (!tc::mbar_try_wait(&empty[s], ph ^ 1u) && !*mma_left) {
        if (tc::globaltimer_ns() - t0 > DRAIN_LIMIT_NS) break;
      }
    }
  }
  __syncwarp();
  if (*mma_left) return false;
  tc::named_arrive(TC_GATE_BAR0 + s, TC_GATE_THREADS);
  return true;
}

// Wait used only while draining after an abort: ignores the abort flag, shorter limit.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = tc::globaltimer_ns();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (tc::globaltimer_ns() - t0 > DRAIN_LIMIT_NS) return;
  }
}

// Clock telemetry: thread 0 of every CTA of the tensor-core kernels adds the SM cycles and
// the nanoseconds it ran to two 64-bit counters at byte offset 64 of the workspace header,
// so a caller can read the mean SM clock these kernels ran at (a power-limited GPU lowers
// it under load, which no sampling from the host resolves at kernel time scales).
__device__ __forceinline__ void clock_telemetry_add(uint32_t* hdr, long long c0, uint64_t t0) {
  unsigned long long* acc = reinterpret_cast<unsigned long long*>(hdr + 16);
  atomicAdd(&acc[0], (unsigned long long)(clock64() - c0));
  atomicAdd(&acc[1], (unsigned long long)(tc::globaltimer_ns() - t0));
}

// One warp fills the group table: rows clamped to the buffer, m-tiles of BM rows, and
// the exclusive prefix of tiles (mt * n_tiles) over the groups.
template <int BM>
__device__ __forceinline__ void build_group_table(GroupTable* tab, const TcArgs& args, int n_tiles,
                                                  int lane) {
  int carry = 0;
  for (int base = 0; base < args.G; base += 32) {
    const int g = base + lane;
    int lo = 0, hi = 0, mt = 0;
    if (g < args.G) {
      if (args.offsets == nullptr) {
        lo = 0;
        hi = args.M;
      } else {
        lo = args.offsets[g];
        hi = args.offsets[g + 1];
      }
      if (hi > args.rows_cap) {
        raise_error(args.hdr, DEV_ERR_OVERFLOW);
        hi = (int)args.rows_cap;
      }
      if (lo < 0) lo = 0;
      if (lo > hi) lo = hi;
      if (args.row_part != TC_ROWS_ALL) {
        const int whole = ((hi - lo) / 256) * 256;
        if (args.row_part == TC_ROWS_FULL256) hi = lo + whole;
        else lo += whole;
      }
      mt = (hi - lo + BM - 1) / BM;
      tab->lo[g] = lo;
      tab->hi[g] = hi;
      tab->mt[g] = mt;
    }
    int v = mt * n_tiles;  // inclusive warp scan of tiles
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (g < args.G) tab->tpre[g + 1] = carry + v;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) tab->tpre[0] = 0;
}

struct TileInfo {
  int g;
  int row0;
  int rowend;
  int n0;
};

// Tile t of the list: groups in order, inside a group n-tiles in order, inside an
// n-tile m-tiles in order (m fastest, so CTAs that run together share the weight box).
template <int BM>
__device__ __forceinline__ TileInfo decode_tile(int t, int G, const GroupTable* tab, int BN) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tab->tpre[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int g = lo;
  const int local = t - tab->tpre[g];
  const int mt = tab->mt[g];
  TileInfo ti;
  ti.g = g;
  ti.row0 = tab->lo[g] + (local % mt) * BM;
  ti.rowend = tab->hi[g];
  ti.n0 = (local / mt) * BN;
  return ti;
}

// GELU for the tensor-core epilogues.  GELU(v) = v Phi(v) = max(v, 0) - t Phi(-t) with
// t = |v|, and the normal tail Phi(-t) from Abramowitz & Stegun 26.2.17 (after Zelen &
// Severo): Phi(-t) = Z(t) (b1 k + b2 k^2 + b3 k^3 + b4 k^4 + b5 k^5) + eps(t), k = 1/(1 + p t),
// Z(t) = exp(-t^2/2) / sqrt(2 pi), |eps| < 7.5e-8.  The factor -1/sqrt(2 pi) is folded into
// the coefficients (GELU_B*), exp(-t^2/2) is 2^(GELU_C t^2), and the reciprocal and the
// power of two are the hardware's approximate instructions.  Evaluated in fp32 the result
// is within 3.4e-7 of GELU(v) in absolute terms (for every fp32 v; the tests check it on
// a dense sweep), far below the fp16 rounding of the stored h.  It takes about a third of
// the instructions of an erf-based form, and the epilogue's arithmetic competes with the
// MMAs of the next tile: on the Mixtral-shaped GEMM the tensor pipe idles measurably less.
// gelu() and gelu2() perform the same correctly rounded operations in the same order (the
// packed form two lanes at a time), so every kernel stores identical h.
constexpr float GELU_P = 0.2316419f;
constexpr float GELU_B1 = -0.127414796f;  // -b1 / sqrt(2 pi), b1 = 0.319381530
constexpr float GELU_B2 = 0.142248368f;   // -b2 / sqrt(2 pi), b2 = -0.356563782
constexpr float GELU_B3 = -0.710706871f;  // -b3 / sqrt(2 pi), b3 = 1.781477937
constexpr float GELU_B4 = 0.726576013f;   // -b4 / sqrt(2 pi), b4 = -1.821255978
constexpr float GELU_B5 = -0.530702714f;  // -b5 / sqrt(2 pi), b5 = 1.330274429
constexpr float GELU_C = -0.72134752044448170368f;  // -1 / (2 ln 2)

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float gelu(float v) {
  const float t = fabsf(v);
  const float k = rcp_approx(__fmaf_rn(t, GELU_P, 1.0f));
  float p = __fmaf_rn(k, GELU_B5, GELU_B4);
  p = __fmaf_rn(k, p, GELU_B3);
  p = __fmaf_rn(k, p, GELU_B2);
  p = __fmaf_rn(k, p, GELU_B1);
  p = __fmul_rn(p, k);                                // -Phi(-t) / Z(t) * (1/sqrt(2 pi))
  const float e = ex2_approx(__fmul_rn(t, __fmul_rn(t, GELU_C)));  // exp(-t^2/2)
  return __fmaf_rn(__fmul_rn(t, p), e, fmaxf(v, 0.0f));
}

// Two fp32 values packed in a 64-bit register, and the packed fp32 FMA and multiply
// (two correctly rounded operations per instruction).
__device__ __forceinline__ uint64_t f32x2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_splat(float a) { return f32x2_pack(a, a); }

// gelu() of two values at once: (gelu(va), gelu(vb)).
__device__ __forceinline__ void gelu2(float va, float vb, float& ga, float& gb) {
  const float ta = fabsf(va), tb = fabsf(vb);
  const uint64_t t = f32x2_pack(ta, tb);
  float da, db;
  f32x2_unpack(f32x2_fma(t, f32x2_splat(GELU_P), f32x2_splat(1.0f)), da, db);
  const uint64_t k = f32x2_pack(rcp_approx(da), rcp_approx(db));
  uint64_t p = f32x2_fma(k, f32x2_splat(GELU_B5), f32x2_splat(GELU_B4));
  p = f32x2_fma(k, p, f32x2_splat(GELU_B3));
  p = f32x2_fma(k, p, f32x2_splat(GELU_B2));
  p = f32x2_fma(k, p, f32x2_splat(GELU_B1));
  p = f32x2_mul(p, k);
  float sa, sb;
  f32x2_unpack(f32x2_mul(t, f32x2_mul(t, f32x2_splat(GELU_C))), sa, sb);
  const uint64_t e = f32x2_pack(ex2_approx(sa), ex2_approx(sb));
  const uint64_t m = f32x2_pack(fmaxf(va, 0.0f), fmaxf(vb, 0.0f));
  f32x2_unpack(f32x2_fma(f32x2_mul(t, p), e, m), ga, gb);
}

// Packs two fp32 values into fp16x2 (round to nearest even) and folds their magnitudes
// into `amax` (NaN-propagating), so one test per chunk catches any value outside the
// fp16 range (an overflow rounds to infinity).
__device__ __forceinline__ uint32_t pack_f16x2_track(float a, float b, __half2& amax) {
  const __half2 h2 = __floats2half2_rn(a, b);
  amax = __hmax2_nan(amax, __habs2(h2));
  return *reinterpret_cast<const uint32_t*>(&h2);
}
__device__ __forceinline__ bool f16x2_out_of_range(__half2 amax) {
  const float2 m = __half22float2(amax);
  return !(m.x <= 65504.f) || !(m.y <= 65504.f);
}

// E4M3 operands: the accumulator holds sum_k qa*qb; the real product is that times the
// row's A scale and the column's B scale.
// (r * sa) * sb for each column, rounded twice in that order; a whole aligned chunk loads
// the column scales as four-float vectors and multiplies two columns per instruction.
__device__ __forceinline__ void apply_scales(uint32_t (&r)[32], float sa, const float* sb_row,
                                             int col0, int N) {
  const float* sb = sb_row + col0;
  if (col0 + 32 <= N && ((uintptr_t)sb & 15u) == 0) {
    const uint64_t sa2 = f32x2_splat(sa);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 b = __ldg(reinterpret_cast<const float4*>(sb) + v);
      float x0, x1, x2, x3;
      f32x2_unpack(f32x2_mul(f32x2_mul(f32x2_pack(__uint_as_float(r[4 * v]),
                                                  __uint_as_float(r[4 * v + 1])), sa2),
                             f32x2_pack(b.x, b.y)), x0, x1);
      f32x2_unpack(f32x2_mul(f32x2_mul(f32x2_pack(__uint_as_float(r[4 * v + 2]),
                                                  __uint_as_float(r[4 * v + 3])), sa2),
                             f32x2_pack(b.z, b.w)), x2, x3);
      r[4 * v] = __float_as_uint(x0);
      r[4 * v + 1] = __float_as_uint(x1);
      r[4 * v + 2] = __float_as_uint(x2);
      r[4 * v + 3] = __float_as_uint(x3);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float s = (col0 + i < N) ? sb[i] : 0.f;
    r[i] = __float_as_uint(__fmul_rn(__fmul_rn(__uint_as_float(r[i]), sa), s));
  }
}

// Epilogue for 32 accumulator columns [col0, col0+32) of one output row, held by this
// thread in r[] (fp32 bit patterns).  Returns true if an fp16 output left the fp16 range.
template <int EPI>
__device__ __forceinline__ bool epilogue_chunk(const uint32_t (&r)[32], int row, int col0,
                                               const TcArgs& args, int64_t slice,
                                               const float* bias) {
  bool bad = false;
  if (EPI == TC_EPI_F16 || EPI == TC_EPI_GELU_F16) {
    __half* out = (__half*)args.out + (size_t)row * args.ldo + col0;
    __half2 amax = __float2half2_rn(0.f);
#pragma unroll
    for (int v8 = 0; v8 < 4; ++v8) {
      if (col0 + v8 * 8 >= args.N) break;
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a = __uint_as_float(r[v8 * 8 + 2 * i]);
        float b = __uint_as_float(r[v8 * 8 + 2 * i + 1]);
        if (EPI == TC_EPI_GELU_F16) gelu2(a, b, a, b);
        w[i] = pack_f16x2_track(a, b, amax);
      }
      st_v4(out + v8 * 8, make_uint4(w[0], w[1], w[2], w[3]));
    }
    bad = f16x2_out_of_range(amax);
  } else if (EPI == TC_EPI_F32) {
    float* out = (float*)args.out + slice + (size_t)row * args.ldo + col0;
#pragma unroll
    for (int v4 = 0; v4 < 8; ++v4) {
      if (col0 + v4 * 4 >= args.N) break;
      st_v4(out + v4 * 4, make_uint4(r[v4 * 4], r[v4 * 4 + 1], r[v4 * 4 + 2], r[v4 * 4 + 3]));
    }
  } else {
    float* out = (float*)args.out + slice + (size_t)row * args.ldo;
    const bool vec = col0 + 32 <= args.N && ((uintptr_t)(out + col0) & 15u) == 0 &&
                     (bias == nullptr || ((uintptr_t)(bias + col0) & 15u) == 0);
    if (vec) {  // 16-byte stores of the 32 columns (one fp32 addition each, as below)
#pragma unroll
      for (int v4 = 0; v4 < 8; ++v4) {
        float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
        if (bias != nullptr) b = __ldg(reinterpret_cast<const float4*>(bias + col0) + v4);
        st_v4(out + col0 + v4 * 4,
              make_uint4(__float_as_uint(__uint_as_float(r[v4 * 4]) + b.x),
                         __float_as_uint(__uint_as_float(r[v4 * 4 + 1]) + b.y),
                         __float_as_uint(__uint_as_float(r[v4 * 4 + 2]) + b.z),
                         __float_as_uint(__uint_as_float(r[v4 * 4 + 3]) + b.w)));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int col = col0 + i;
        if (col < args.N) out[col] = __uint_as_float(r[i]) + (bias != nullptr ? bias[col] : 0.f);
      }
    }
  }
  return bad;
}

// Epilogues of a transposed tile (output columns on the TMEM lanes, the tile's rows on
// its columns), shared by the transposed-pair and the mixed-pair kernels.
// Epilogue of the transposed tile: r[j] = C[tok0 + c0 + j, col] for j < 32.  E4M3
// operands: the accumulator times the token row's scale, then the column's scale (the
// order of the other kernels' epilogues, so every plan stores the same values).
template <int EPI, int KIND>
__device__ __forceinline__ bool epilogue_chunk_t(const uint32_t (&r)[32], int col, int tok_first,
                                                 int tok_end, const TcArgs& args, float sb) {
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int tok = tok_first + j;
    if (tok >= tok_end) break;
    float v = __uint_as_float(r[j]);
    if (KIND == OP_E4M3) v = __fmul_rn(__fmul_rn(v, args.a_scale[tok]), sb);
    if (EPI == TC_EPI_GELU_F16 || EPI == TC_EPI_F16) {
      const float a = EPI == TC_EPI_GELU_F16 ? gelu(v) : v;
      bad |= !(fabsf(a) <= 65504.f);
      ((__half*)args.out)[(size_t)tok * args.ldo + col] = __float2half_rn(a);
    } else {
      ((float*)args.out)[(size_t)tok * args.ldo + col] = v;
    }
  }
  return bad;
}

// 16-bit outputs of the transposed tile: lane l holds column colbase + l of 32 tokens.
// The warp's 32 x 32 block goes through its shared-memory buffer (token-major), so that
// each lane then stores 16 contiguous bytes of one token row (four 16-byte stores per lane
// instead of 32 two-byte ones).  Same values and range test as epilogue_chunk_t.
template <int EPI, int KIND>
__device__ __forceinline__ bool epilogue_chunk_t16(const uint32_t (&r)[32], int colbase, int lane,
                                                   int tok_first, int tok_end, const TcArgs& args,
                                                   float sb, __half* sbuf) {
  const bool valid = colbase + lane < args.N;
  float sa_l = 0.f;  // E4M3: the scale of token tok_first + lane
  if (KIND == OP_E4M3 && tok_first + lane < tok_end) sa_l = args.a_scale[tok_first + lane];
  bool bad = false;
  __syncwarp();  // the previous chunk's reads of the buffer are done
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float a = __uint_as_float(r[j]), b = __uint_as_float(r[j + 1]);
    if (KIND == OP_E4M3) {
      a = __fmul_rn(__fmul_rn(a, __shfl_sync(0xffffffffu, sa_l, j)), sb);
      b = __fmul_rn(__fmul_rn(b, __shfl_sync(0xffffffffu, sa_l, j + 1)), sb);
    }
    if (EPI == TC_EPI_GELU_F16) gelu2(a, b, a, b);
    bad |= valid && ((tok_first + j < tok_end && !(fabsf(a) <= 65504.f)) ||
                     (tok_first + j + 1 < tok_end && !(fabsf(b) <= 65504.f)));
    sbuf[j * 32 + lane] = __float2half_rn(a);
    sbuf[(j + 1) * 32 + lane] = __float2half_rn(b);
  }
  __syncwarp();
  const int cg = (lane & 3) * 8;  // this lane's 8 columns of a token row
  if (colbase + cg < args.N) {    // N is a multiple of 8: a group is all in or all out
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = (lane >> 2) + 8 * i;
      if (tok_first + row < tok_end)
        st_v4((__half*)args.out + (size_t)(tok_first + row) * args.ldo + colbase + cg,
              *reinterpret_cast<const uint4*>(sbuf + row * 32 + cg));
    }
  }
  return bad;
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn();

// 2-D tensor map of a row-major [outer, inner] matrix of operand kind `kind`, box
// [box_outer rows, 128 bytes], 128-byte swizzle.
bool tc_make_map(CUtensorMap* m, const void* base, int kind, uint64_t inner, uint64_t outer,
                 uint32_t box_outer);

}  // namespace moe
