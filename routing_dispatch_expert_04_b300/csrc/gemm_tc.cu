// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// C[r, n] = epi( sum_k A[r, k] * B[g*N + n, k] ) for the rows r of group g,
// r in [offsets[g], offsets[g+1]).  A is the packed expert input (K-major, row pitch Kd),
// B the stacked expert weights in Linear layout [G*N, Kd].  This is the expert FFN of
// "Expert Parallelism (MoE)", "MoE Layer Structure" (each expert applies Linear(d -> 4d)
// -> GELU -> Linear(4d -> d)) run for all experts in one launch ("Expert Parallelism
// (EP)", step 3: expert GEMMs compute locally).
//
// Design (one CTA per SM, persistent):
//   warp 0      TMA producer: per k-block, one A box of 128 rows and one B box of BN rows,
//               128 bytes of K each (64 bf16/fp16 or 128 E4M3 values), into a
//               STAGES-deep ring of 128-byte-swizzled shared-memory stages;
//   warp 1      owns TMEM (2 x BN fp32 columns: double-buffered accumulators) and one
//               elected thread issues tcgen05.mma (M=128, N=BN; kind::f16 with K=16 or
//               kind::f8f6f4 with K=32) and commits; the warp learns that a stage holds
//               its data from a named barrier, not from the stage's mbarrier;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows, E4M3 row/column scales,
//               fused GELU (the normal-tail form in tc_common.cuh) or plain/bias,
//               conversion and masked stores.  Overlaps the next tile's main loop through
//               the second accumulator;
//   warp 6      stage watcher: waits on each stage's mbarrier and arrives on its named
//               barrier (the stage gate in tc_common.cuh), so the MMA thread touches no
//               shared memory per k-block.
// Tiles are (group, n-tile, m-tile) with m fastest, so CTAs running at the same time
// share one weight box through L2.  The per-group row ranges are read from `offsets` on
// the device (no host synchronisation); the last m-tile of a group may run past the
// group's rows (those rows are loaded but never stored) and past the buffer (TMA fills
// zeros).  Every mbarrier wait is bounded: after WAIT_LIMIT_NS the CTA records a timeout
// in the status word, every role leaves its loop, in-flight copies and MMAs are awaited
// (bounded), TMEM is freed and the CTA exits.
#include <mutex>

#include "tc_common.cuh"

namespace moe {
using namespace tc;

constexpr int TC_BM = 128;

template <int BN, int STAGES>
struct TcLayout {
  static constexpr int A_BYTES = TC_BM * TC_ROW_BYTES;
  static constexpr int B_BYTES = BN * TC_ROW_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int B_OFF = STAGES * A_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NBAR = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], done
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int GRP_OFF = MISC_OFF + 16;
  static constexpr int TOTAL = GRP_OFF + (int)sizeof(GroupTable);
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr uint32_t TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64
                                       : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
};

template <int BN, int STAGES, int EPI, int KIND, bool GATHER>
__global__ void __launch_bounds__(TC_THREADS_GATED, 1)
tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_b, const TcArgs args) {
  using Lay = TcLayout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + Lay::BAR_OFF);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* done = bars + 2 * STAGES + 4;
  uint32_t* s_tmem = (uint32_t*)(smem + Lay::MISC_OFF);
  volatile int* s_abort = (volatile int*)(smem + Lay::MISC_OFF + 4);
  volatile int* s_mma_left = (volatile int*)(smem + Lay::MISC_OFF + 8);
  GroupTable* tab = (GroupTable*)(smem + Lay::GRP_OFF);

  const long long clk0 = clock64();
  const uint64_t ns0 = globaltimer_ns();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.G;
  const int n_tiles = (args.N + BN - 1) / BN;
  constexpr int BKE = OpKind<KIND>::BK;  // K elements per stage
  const int nkb = (args.Kd + BKE - 1) / BKE;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(done, 1);
    *s_abort = 0;
    *s_mma_left = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 0) {
    build_group_table<TC_BM>(tab, args, n_tiles, lane);
  } else if (warp == 1) {
    tmem_alloc(s_tmem, Lay::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int ksplit = args.ksplit;
  const int total = tab->tpre[G] * ksplit;

  if (warp == 0) {
    if (GATHER || lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      // Plain A: lane 0 issues one box per k-block.  Gathered A: every lane gathers four
      // of the tile's 128 rows (tile::gather4) into their place in the stage.
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile<TC_BM>(t / ksplit, G, tab, BN);
        const int brow = ti.g * args.N + ti.n0;
        const int kb0 = (t % ksplit) * args.kpb;
        const int kb1 = min(nkb, kb0 + args.kpb);
        int tok[4] = {0, 0, 0, 0};
        if (GATHER) {
#pragma unroll
          for (int i = 0; i < 4; ++i) tok[i] = gather_row(args, ti.row0 + 4 * lane + i, ti.rowend);
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          bool got = true;
          if (lane == 0) got = wait_phase(&empty[s], ph ^ 1u, s_abort, args.hdr);
          if (GATHER) got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * Lay::A_BYTES;
          uint8_t* sb = smem + Lay::B_OFF + s * Lay::B_BYTES;
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], Lay::STAGE_BYTES);
            if (!GATHER) tma_load_2d(sa, &tmap_a, &full[s], kb * BKE, ti.row0);
            tma_load_2d(sb, &tmap_b, &full[s], kb * BKE, brow);
          }
          if (GATHER) {
            __syncwarp();
            tma_gather4(sa + lane * 4 * TC_ROW_BYTES, &tmap_a, &full[s], kb * BKE, tok[0], tok[1],
                        tok[2], tok[3]);
          }
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && lane == 0) {  // let the copies already in flight land before shared memory goes away
        for (int i = 0; i < STAGES && i < issued; ++i) {
          if (--s < 0) {
            s = STAGES - 1;
            ph ^= 1u;
          }
          drain_wait(&full[s], ph);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // lane 0 issues; the whole warp waits on the stage gate (named barriers)
    constexpr uint32_t IDESC = KIND == OP_BF16 ? idesc_bf16_f32(TC_BM, BN)
                                              : idesc_fmt0_f32(TC_BM, BN);
    int s = 0;
    uint32_t acc = 0, aph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int ok = 1;
      if (lane == 0) ok = wait_phase(&tempty[acc], aph ^ 1u, s_abort, args.hdr) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const uint32_t d_tmem = tmem_base + acc * BN;
      const int kb0 = (t % ksplit) * args.kpb;
      const int kb1 = min(nkb, kb0 + args.kpb);
      for (int kb = kb0; kb < kb1; ++kb) {
        named_sync(TC_GATE_BAR0 + s, TC_GATE_THREADS);
        if (lane == 0) {
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * Lay::A_BYTES);
          const uint32_t b_addr = smem_u32(smem + Lay::B_OFF + s * Lay::B_BYTES);
#pragma unroll
          for (int k = 0; k < TC_ROW_BYTES / 32; ++k) {  // 32 bytes of K per MMA
            if (KIND == OP_E4M3)
              mma_e4m3(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32), IDESC,
                       (kb != kb0 || k != 0) ? 1u : 0u);
            else
              mma_bf16(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32), IDESC,
                       (kb != kb0 || k != 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == STAGES) s = 0;
      }
      if (lane == 0) mma_commit(&tfull[acc]);
      __syncwarp();
      acc ^= 1u;
      if (acc == 0) aph ^= 1u;
    }
    if (lane == 0) {
      *s_mma_left = 1;  // the watcher stops arriving
      // every MMA issued by this thread has completed once `done` flips
      mma_commit(done);
      drain_wait(done, 0);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ---------------------------------------------------------------- stage watcher
    int s = 0;
    uint32_t ph = 0;
    bool gave_up = false, go = true;
    for (int t = blockIdx.x; t < total && go; t += gridDim.x) {
      const int kb0 = (t % ksplit) * args.kpb;
      const int kb1 = min(nkb, kb0 + args.kpb);
      for (int kb = kb0; kb < kb1 && go; ++kb) {
        go = gate_arrive(s, full, empty, ph, gave_up, s_abort, s_mma_left, args.hdr, lane);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in_tile = q * 32 + lane;
    uint32_t acc = 0, aph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = decode_tile<TC_BM>(t / ksplit, G, tab, BN);
      const int64_t slice = (int64_t)(t % ksplit) * args.split_stride;
      const float* bias = ksplit == 1 ? args.bias : nullptr;
      if (!wait_phase(&tfull[acc], aph, s_abort, args.hdr)) break;
      tc_fence_after();
      const int row = ti.row0 + r_in_tile;
      const bool valid = row < ti.rowend;
      float sa = 0.f;  // E4M3: this row's A scale (of its token row when gathered)
      if (KIND == OP_E4M3 && valid) sa = args.a_scale[GATHER ? gather_row(args, row, ti.rowend) : row];
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int col0 = ti.n0 + c * 32;
        if (col0 >= args.N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + c * 32, r);
        tmem_ld_wait();
        if (!valid) continue;
        if (KIND == OP_E4M3) apply_scales(r, sa, args.b_scale + (size_t)ti.g * args.N, col0, args.N);
        if (epilogue_chunk<EPI>(r, row, col0, args, slice, bias)) raise_error(args.hdr, DEV_ERR_RANGE);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1u;
      if (acc == 0) aph ^= 1u;
    }
  }

  if (threadIdx.x == 0) clock_telemetry_add(args.hdr, clk0, ns0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Lay::TMEM_COLS);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

bool tc_make_map(CUtensorMap* m, const void* base, int kind, uint64_t inner, uint64_t outer,
                 uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tc_encode_fn();
  if (fn == nullptr) return false;
  const uint64_t esize = kind == OP_E4M3 ? 1 : 2;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {(cuuint32_t)(TC_ROW_BYTES / esize), box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = kind == OP_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : kind == OP_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int STAGES, int EPI, int KIND, bool GATHER = false>
static cudaError_t launch_tc(const void* A, const void* B, const TcArgs& a, int num_sms,
                             cudaStream_t st, int ctas_per_sm = 1) {
  using Lay = TcLayout<BN, STAGES>;
  static bool attr_set = false;
  auto kern = tc_grouped_gemm_kernel<BN, STAGES, EPI, KIND, GATHER>;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC);
    if (e != cudaSuccess) return e;
    if (ctas_per_sm > 1) {  // room for several CTAs' stages on one SM
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  CUtensorMap ma, mb;
  const int64_t a_rows = a.rows_cap > 0 ? a.rows_cap : 1;
  const bool ok_a = GATHER ? tc_make_map(&ma, A, KIND, (uint64_t)a.Kd, (uint64_t)a.gather_rows, 1)
                           : tc_make_map(&ma, A, KIND, (uint64_t)a.Kd, (uint64_t)a_rows, TC_BM);
  if (!ok_a) return cudaErrorInvalidValue;
  if (!tc_make_map(&mb, B, KIND, (uint64_t)a.Kd, (uint64_t)a.G * a.N, BN)) return cudaErrorInvalidValue;
  const int64_t n_tiles = (a.N + BN - 1) / BN;
  const int64_t m_bound = (a.rows_cap + TC_BM - 1) / TC_BM + (a.offsets ? a.G : 0);
  int64_t grid = m_bound * n_tiles * a.ksplit;
  if (grid > (int64_t)num_sms * ctas_per_sm) grid = (int64_t)num_sms * ctas_per_sm;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, TC_THREADS_GATED, Lay::ALLOC, st>>>(ma, mb, a);
  count_launch();
  return cudaGetLastError();
}

// N tile of an expert GEMM: 256, or 192 when 256-wide tiles would leave the last wave
// of the persistent grid much emptier or waste columns.  The m-tile count (tiles of `bm`
// rows) is estimated on the host from the row capacity (each group holds at most
// `cap_per_group` rows when that is known); `slots` = tiles that run at once (CTAs, or
// CTA pairs).  Qwen3 shape on pairs (B300): GEMM1 (F = 768: 384 tiles of 256 on 74 pairs,
// 5.2 waves) 0.115 -> 0.109 ms with 192-wide tiles (512 tiles, 6.9 waves).
static int pick_bn(int64_t rows_cap, int G, int64_t cap_per_group, int N, int slots, int bm) {
  int64_t m_tiles;
  if (cap_per_group > 0) {
    const int64_t per = cap_per_group < rows_cap ? cap_per_group : rows_cap;
    m_tiles = (int64_t)G * ((per + bm - 1) / bm);
    const int64_t bound = (rows_cap + bm - 1) / bm + G;
    if (m_tiles > bound) m_tiles = bound;
  } else {
    m_tiles = (rows_cap + bm - 1) / bm + G / 2;
  }
  double best = -1.0;
  int best_bn = 256;
  for (int bn : {256, 192}) {
    const int64_t nt = (N + bn - 1) / bn;
    const double waves = (double)(m_tiles * nt) / slots;
    const double full_waves = (double)(int64_t)(waves + 0.999999);
    const double eff = waves / full_waves * ((double)N / (double)(nt * bn));
    if (eff > best + 0.02) {
      best = eff;
      best_bn = bn;
    }
  }
  return best_bn;
}

cudaError_t launch_tc2_up(const void* a_in, const int32_t* gather_src, int gather_k,
                          int64_t gather_rows, const void* w1, void* h, const int32_t* offsets,
                          int G, int N, int Kd, int64_t rows_cap, int row_part, int bn,
                          uint32_t* hdr, int num_sms, cudaStream_t st);
cudaError_t launch_tc2_down(const void* h, const void* w2h, void* y_perm, const int32_t* offsets,
                            int G, int N, int Kd, int64_t rows_cap, int row_part, int bn,
                            uint32_t* hdr, int num_sms, cudaStream_t st);

// How the expert GEMM's rows are split between the kernels: one CTA per 128-row tile
// for all rows, CTA pairs per 256-row tile for all rows, or pairs for each group's whole
// 256-row tiles and one CTA per 128-row tile for the rest.  Measured on B300, the
// one-CTA 128x256 tiles keep the tensor pipe about two thirds busy and the pair tiles
// (which stage and read half of B per SM) 85-93%.  But pairs pad a group to a multiple
// of 256 rows.  The split runs pairs on each group's whole 256-row tiles and, at the same
// time on the remaining SMs, one CTA per tile on the rest.  Measured on the layer shapes
// (B300), MOE_GEMM_AUTO takes pairs when their padding is at most 5% (judged from the
// per-group row bound, and with N filling 256-wide tiles), the split when groups are
// known to reach 256 rows (Mixtral shape: 0.50 -> 0.47-0.48 ms per GEMM), one CTA
// otherwise, and for groups of unknown size (no capacity) the transposed pairs, which
// size the token side of each tile to the group (DeepSeek-V3 shape).
enum { PLAN_SINGLE = 0, PLAN_PAIR = 1, PLAN_SPLIT = 2, PLAN_PAIR_T = 3, PLAN_MIXED = 4 };

cudaError_t launch_tc2m_up(const void* x_perm, const void* w1, void* h, const int32_t* offsets,
                           int G, int N, int Kd, int64_t rows_cap, uint32_t* hdr, int num_sms,
                           cudaStream_t st);
cudaError_t launch_tc2m_down(const void* h, const void* w2h, void* y_perm, const int32_t* offsets,
                             int G, int N, int Kd, int64_t rows_cap, uint32_t* hdr, int num_sms,
                             cudaStream_t st);

cudaError_t launch_tc2t_up(const void* x_perm, const void* w1, void* h, const int32_t* offsets,
                           int G, int N, int Kd, int64_t rows_cap, uint32_t* hdr, int num_sms,
                           cudaStream_t st);
cudaError_t launch_tc2t_down(const void* h, const void* w2h, void* y_perm, const int32_t* offsets,
                             int G, int N, int Kd, int64_t rows_cap, uint32_t* hdr, int num_sms,
                             cudaStream_t st);

static int gemm_plan(int mode, int64_t rows_cap, int G, int64_t cap_per_group, int N) {
  if (mode == MOE_GEMM_SINGLE) return PLAN_SINGLE;
  if (mode == MOE_GEMM_PAIR) return PLAN_PAIR;
  if (mode == MOE_GEMM_SPLIT) return PLAN_SPLIT;
  if (mode == MOE_GEMM_PAIR_T) return PLAN_PAIR_T;
  if (mode == MOE_GEMM_MIXED) return PLAN_MIXED;
  if (N % 256 != 0) return PLAN_SINGLE;
  // groups of unknown size (no capacity): the transposed pairs size each token tile to
  // the group, so ragged groups pad to 32 rows, not 128 or 256
  if (cap_per_group <= 0) return PLAN_PAIR_T;
  const int64_t per = cap_per_group < rows_cap ? cap_per_group : rows_cap;
  const int64_t rows128 = (int64_t)G * ((per + 127) / 128) * 128;
  const int64_t rows256 = (int64_t)G * ((per + 255) / 256) * 256;
  if (rows256 * 100 <= rows128 * 105) return PLAN_PAIR;
  return per >= 256 ? PLAN_SPLIT : PLAN_SINGLE;
}

// The split plan runs the CTA-pair kernel (whole 256-row tiles) and the one-CTA kernel
// (the rest of each group) at the same time on disjoint SM shares: the second kernel
// goes on a library-owned side stream, forked from and joined back into the caller's
// stream with events (which also works inside stream capture).  One side stream and
// one event pair per device, created on first use.
struct SplitStreams {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

static cudaError_t split_streams(SplitStreams** out) {
  static std::mutex mu;
  static SplitStreams per_dev[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  SplitStreams& s = per_dev[dev];
  if (s.side == nullptr) {
    if ((e = cudaStreamCreateWithFlags(&s.side, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &s;
  return cudaSuccess;
}

// SMs given to the pair kernel in the split plan: its share of the rows, weighted by
// the one-CTA kernel taking ~1.4x as long per row, so that both finish together; an even
// count (whole pairs), leaving the one-CTA kernel some.  Measured on the Mixtral shape
// (640-row groups: 512 on pairs, 128 on one CTA), GEMM1 / GEMM2 ms by pair SMs: 106
// 0.471 / 0.477, 108 0.451 / 0.473, 112 0.512 / 0.473, 114+ 0.51 / 0.55; the weighting
// gives 108.  Past the optimum the one-CTA kernel's share of the tiles finishes last, and
// the time rises steeply.
static int split_pair_sms(int64_t cap_per_group, int num_sms) {
  double frac = 0.75;  // groups of unknown size
  if (cap_per_group > 0) {
    const double whole = (double)(cap_per_group / 256 * 256);
    const double rest = (double)(cap_per_group - cap_per_group / 256 * 256);
    frac = whole / (whole + 1.4 * rest);
  }
  int sp = ((int)(num_sms * frac)) & ~1;
  if (sp > num_sms - 2) sp = (num_sms - 2) & ~1;
  if (sp < 2) sp = 2;
  return sp;
}

// Runs `pair(st)` on the caller's stream and, at the same time, `rest(side)` on the side
// stream, forked from and joined back into `st`.
template <class PairFn, class RestFn>
static cudaError_t run_split(cudaStream_t st, PairFn pair, RestFn rest) {
  SplitStreams* ss = nullptr;
  cudaError_t e = split_streams(&ss);
  if (e != cudaSuccess) return e;
  if ((e = cudaEventRecord(ss->fork, st)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(ss->side, ss->fork, 0)) != cudaSuccess) return e;
  if ((e = pair(st)) != cudaSuccess) return e;
  if ((e = rest(ss->side)) != cudaSuccess) return e;
  if ((e = cudaEventRecord(ss->join, ss->side)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(st, ss->join, 0);
}

template <int EPI, int KIND, bool GATHER>
static cudaError_t launch_tc_single(const void* A, const void* B, const TcArgs& a,
                                    int64_t cap_per_group, int num_sms, cudaStream_t st) {
  if (pick_bn(a.rows_cap, a.G, cap_per_group, a.N, num_sms, TC_BM) == 192)
    return launch_tc<192, 5, EPI, KIND, GATHER>(A, B, a, num_sms, st);
  return launch_tc<256, 4, EPI, KIND, GATHER>(A, B, a, num_sms, st);
}

// First expert Linear, bf16 in, GELU fused, fp16 out: h[r] = GELU(A[r] . W1[g]^T), with
// A = x_perm, or with `gather_src` A[r] = x[gather_src[r] / gather_k] gathered from the
// token matrix x ([gather_rows, Kd]) while the tile is loaded.
cudaError_t launch_tc_up(const void* a_in, const int32_t* gather_src, int gather_k,
                         int64_t gather_rows, const void* w1, void* h, const int32_t* offsets,
                         int G, int N, int Kd, int64_t rows_cap, int64_t cap_per_group,
                         int pair_mode, uint32_t* hdr, int num_sms, cudaStream_t st) {
  int plan = gemm_plan(pair_mode, rows_cap, G, cap_per_group, N);
  const bool gather = gather_src != nullptr;
  if (plan == PLAN_PAIR_T && gather) plan = PLAN_PAIR;  // row gathers need rows on the M side
  if (plan == PLAN_MIXED && gather) plan = PLAN_SPLIT;
  if (plan == PLAN_PAIR_T)
    return launch_tc2t_up(a_in, w1, h, offsets, G, N, Kd, rows_cap, hdr, num_sms, st);
  if (plan == PLAN_MIXED)
    return launch_tc2m_up(a_in, w1, h, offsets, G, N, Kd, rows_cap, hdr, num_sms, st);
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, h, N, nullptr, hdr, 1, (Kd + TC_BK - 1) / TC_BK, 0,
           TC_ROWS_ALL, gather_src, gather_k, gather_rows};
  if (plan == PLAN_SINGLE)
    return gather ? launch_tc_single<TC_EPI_GELU_F16, OP_BF16, true>(a_in, w1, a, cap_per_group,
                                                                  num_sms, st)
                  : launch_tc_single<TC_EPI_GELU_F16, OP_BF16, false>(a_in, w1, a, cap_per_group,
                                                                   num_sms, st);
  if (plan == PLAN_PAIR)
    return launch_tc2_up(a_in, gather_src, gather_k, gather_rows, w1, h, offsets, G, N, Kd,
                         rows_cap, TC_ROWS_ALL,
                         pick_bn(rows_cap, G, cap_per_group, N, num_sms / 2, 256), hdr, num_sms,
                         st);
  const int sp = split_pair_sms(cap_per_group, num_sms);
  a.row_part = TC_ROWS_REST256;
  return run_split(
      st,
      [&](cudaStream_t s) {
        return launch_tc2_up(a_in, gather_src, gather_k, gather_rows, w1, h, offsets, G, N, Kd,
                             rows_cap, TC_ROWS_FULL256, 256, hdr, sp, s);
      },
      [&](cudaStream_t s) {
        return gather ? launch_tc_single<TC_EPI_GELU_F16, OP_BF16, true>(a_in, w1, a, 255,
                                                                      num_sms - sp, s)
                      : launch_tc_single<TC_EPI_GELU_F16, OP_BF16, false>(a_in, w1, a, 255,
                                                                       num_sms - sp, s);
      });
}

// Second expert Linear, fp16 in, fp16 out: y_perm[r] = h[r] . W2[g]^T.
cudaError_t launch_tc_down(const void* h, const void* w2h, void* y_perm, const int32_t* offsets,
                           int G, int N, int Kd, int64_t rows_cap, int64_t cap_per_group,
                           int pair_mode, uint32_t* hdr, int num_sms, cudaStream_t st) {
  const int plan = gemm_plan(pair_mode, rows_cap, G, cap_per_group, N);
  if (plan == PLAN_PAIR_T)
    return launch_tc2t_down(h, w2h, y_perm, offsets, G, N, Kd, rows_cap, hdr, num_sms, st);
  if (plan == PLAN_MIXED)
    return launch_tc2m_down(h, w2h, y_perm, offsets, G, N, Kd, rows_cap, hdr, num_sms, st);
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, y_perm, N, nullptr, hdr, 1, (Kd + TC_BK - 1) / TC_BK, 0,
           TC_ROWS_ALL};
  if (plan == PLAN_SINGLE)
    return launch_tc_single<TC_EPI_F16, OP_F16, false>(h, w2h, a, cap_per_group, num_sms, st);
  if (plan == PLAN_PAIR)
    return launch_tc2_down(h, w2h, y_perm, offsets, G, N, Kd, rows_cap, TC_ROWS_ALL,
                           pick_bn(rows_cap, G, cap_per_group, N, num_sms / 2, 256), hdr,
                           num_sms, st);
  const int sp = split_pair_sms(cap_per_group, num_sms);
  a.row_part = TC_ROWS_REST256;
  return run_split(
      st,
      [&](cudaStream_t s) {
        return launch_tc2_down(h, w2h, y_perm, offsets, G, N, Kd, rows_cap, TC_ROWS_FULL256, 256,
                               hdr, sp, s);
      },
      [&](cudaStream_t s) {
        return launch_tc_single<TC_EPI_F16, OP_F16, false>(h, w2h, a, 255, num_sms - sp, s);
      });
}

cudaError_t launch_tc2_up_e4m3(const void* xq, const float* sx, const int32_t* gather_src,
                               int gather_k, int64_t gather_rows, const void* w1q, const float* sw1,
                               void* h, const int32_t* offsets, int G, int N, int Kd,
                               int64_t rows_cap, int row_part, uint32_t* hdr, int num_sms,
                               cudaStream_t st);
cudaError_t launch_tc2_down_e4m3(const void* hq, const float* sh, const void* w2q, const float* sw2,
                                 void* y_perm, const int32_t* offsets, int G, int N, int Kd,
                                 int64_t rows_cap, int row_part, uint32_t* hdr, int num_sms,
                                 cudaStream_t st);

cudaError_t launch_tc2t_up_e4m3(const void* xq, const float* sx, const void* w1q, const float* sw1,
                                void* h, const int32_t* offsets, int G, int N, int Kd,
                                int64_t rows_cap, uint32_t* hdr, int num_sms, cudaStream_t st);
cudaError_t launch_tc2t_down_e4m3(const void* hq, const float* sh, const void* w2q, const float* sw2,
                                  void* y_perm, const int32_t* offsets, int G, int N, int Kd,
                                  int64_t rows_cap, uint32_t* hdr, int num_sms, cudaStream_t st);

// Plan for the E4M3 GEMMs: as for 16-bit operands, except that E4M3 halves the weight
// bytes but doubles the tensor rate, so small groups stay HBM-bound (2 x rows flops per
// weight byte against a ridge near 550): there the pair's halved shared-memory traffic
// buys nothing and its longer tiles lose to the one-CTA kernel (measured on B300:
// 192-row groups 0.111 vs 0.123 ms per GEMM; 8192-row groups pairs 2.62 vs 2.68 ms).
// AUTO takes pairs for E4M3 only from 512 rows per group on.  Nor does AUTO take the
// transposed pairs for E4M3: with half as many k-blocks per tile their transposed
// epilogue weighs more (DeepSeek-V3 shape, B300: GEMM2 1.71 vs 1.26 ms on one CTA per
// tile; GEMM1 1.44 vs 1.49 ms).
static int gemm_plan_e4m3(int mode, int64_t rows_cap, int G, int64_t cap_per_group, int N) {
  int plan = gemm_plan(mode, rows_cap, G, cap_per_group, N);
  if (plan == PLAN_MIXED) plan = PLAN_SPLIT;  // the mixed-tile kernel takes 16-bit operands
  if (mode != MOE_GEMM_AUTO) return plan;
  if (plan == PLAN_PAIR && cap_per_group < 512) return PLAN_SINGLE;
  if (plan == PLAN_PAIR_T) return PLAN_SINGLE;
  return plan;
}

// First expert Linear on E4M3 operands (codes + per-row scales), GELU fused, fp16 out:
// h[r] = GELU(sx[a(r)] * sw1[g*N + n] * sum_k xq[a(r), k] w1q[g*N + n, k]) with
// a(r) = gather_src[r] / gather_k (the token row) when gather_src is given, else r.
cudaError_t launch_tc_up_e4m3(const void* xq, const float* sx, const int32_t* gather_src,
                              int gather_k, int64_t gather_rows, const void* w1q, const float* sw1,
                              void* h, const int32_t* offsets, int G, int N, int Kd,
                              int64_t rows_cap, int64_t cap_per_group, int pair_mode,
                              uint32_t* hdr, int num_sms, cudaStream_t st) {
  int plan = gemm_plan_e4m3(pair_mode, rows_cap, G, cap_per_group, N);
  if (plan == PLAN_PAIR_T && gather_src != nullptr) plan = PLAN_PAIR;  // gathers: rows on M
  if (plan == PLAN_PAIR_T)
    return launch_tc2t_up_e4m3(xq, sx, w1q, sw1, h, offsets, G, N, Kd, rows_cap, hdr, num_sms, st);
  if (plan == PLAN_PAIR)
    return launch_tc2_up_e4m3(xq, sx, gather_src, gather_k, gather_rows, w1q, sw1, h, offsets, G,
                              N, Kd, rows_cap, TC_ROWS_ALL, hdr, num_sms, st);
  constexpr int BKE = OpKind<OP_E4M3>::BK;
  const bool gather = gather_src != nullptr;
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, h, N, nullptr, hdr, 1, (Kd + BKE - 1) / BKE, 0,
           TC_ROWS_ALL, gather_src, gather_k, gather_rows, sx, sw1};
  if (plan == PLAN_SINGLE)
    return gather ? launch_tc_single<TC_EPI_GELU_F16, OP_E4M3, true>(xq, w1q, a, cap_per_group,
                                                                  num_sms, st)
                  : launch_tc_single<TC_EPI_GELU_F16, OP_E4M3, false>(xq, w1q, a, cap_per_group,
                                                                   num_sms, st);
  const int sp = split_pair_sms(cap_per_group, num_sms);
  a.row_part = TC_ROWS_REST256;
  return run_split(
      st,
      [&](cudaStream_t s) {
        return launch_tc2_up_e4m3(xq, sx, gather_src, gather_k, gather_rows, w1q, sw1, h, offsets,
                                  G, N, Kd, rows_cap, TC_ROWS_FULL256, hdr, sp, s);
      },
      [&](cudaStream_t s) {
        return gather ? launch_tc_single<TC_EPI_GELU_F16, OP_E4M3, true>(xq, w1q, a, 255,
                                                                      num_sms - sp, s)
                      : launch_tc_single<TC_EPI_GELU_F16, OP_E4M3, false>(xq, w1q, a, 255,
                                                                       num_sms - sp, s);
      });
}

// Second expert Linear on E4M3 operands, fp16 out:
// y_perm[r] = sh[r] * sw2[g*N + n] * sum_k hq[r, k] w2q[g*N + n, k].
cudaError_t launch_tc_down_e4m3(const void* hq, const float* sh, const void* w2q, const float* sw2,
                                void* y_perm, const int32_t* offsets, int G, int N, int Kd,
                                int64_t rows_cap, int64_t cap_per_group, int pair_mode,
                                uint32_t* hdr, int num_sms, cudaStream_t st) {
  const int plan = gemm_plan_e4m3(pair_mode, rows_cap, G, cap_per_group, N);
  if (plan == PLAN_PAIR_T)
    return launch_tc2t_down_e4m3(hq, sh, w2q, sw2, y_perm, offsets, G, N, Kd, rows_cap, hdr,
                                 num_sms, st);
  if (plan == PLAN_PAIR)
    return launch_tc2_down_e4m3(hq, sh, w2q, sw2, y_perm, offsets, G, N, Kd, rows_cap,
                                TC_ROWS_ALL, hdr, num_sms, st);
  constexpr int BKE = OpKind<OP_E4M3>::BK;
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, y_perm, N, nullptr, hdr, 1, (Kd + BKE - 1) / BKE, 0,
           TC_ROWS_ALL, nullptr, 1, 0, sh, sw2};
  if (plan == PLAN_SINGLE)
    return launch_tc_single<TC_EPI_F16, OP_E4M3, false>(hq, w2q, a, cap_per_group, num_sms, st);
  const int sp = split_pair_sms(cap_per_group, num_sms);
  a.row_part = TC_ROWS_REST256;
  return run_split(
      st,
      [&](cudaStream_t s) {
        return launch_tc2_down_e4m3(hq, sh, w2q, sw2, y_perm, offsets, G, N, Kd, rows_cap,
                                    TC_ROWS_FULL256, hdr, sp, s);
      },
      [&](cudaStream_t s) {
        return launch_tc_single<TC_EPI_F16, OP_E4M3, false>(hq, w2q, a, 255, num_sms - sp, s);
      });
}

// Router Linear, bf16 in, fp32 logits: logits[t] = x[t] . W_r^T + b_r.  With nsplit > 1
// the K dimension is split over CTAs and `out` receives nsplit partial slices of
// T*E floats (no bias); the softmax kernel sums them in slice order and adds the bias.
cudaError_t launch_tc_router(const void* x, const void* w_r, const float* b_r, float* out, int T,
                             int E, int d, int nsplit, uint32_t* hdr, int num_sms, cudaStream_t st) {
  const int nkb = (d + TC_BK - 1) / TC_BK;
  const int kpb = (nkb + nsplit - 1) / nsplit;
  const int ks = (nkb + kpb - 1) / kpb;
  TcArgs a{nullptr, 1, T, E, d, (int64_t)T, out, E, b_r, hdr, ks, kpb, (int64_t)T * E,
           TC_ROWS_ALL};
  // the epilogue reads TMEM 32 columns at a time, so the narrowest tile is 32 wide; the
  // E <= 64 variants keep their stages within 100 KB so that two CTAs share an SM
  const int per_sm = router_ctas_per_sm(E);
  if (E <= 32) return launch_tc<32, 4, TC_EPI_BIAS_F32, OP_BF16>(x, w_r, a, num_sms, st, per_sm);
  if (E <= 64) return launch_tc<64, 4, TC_EPI_BIAS_F32, OP_BF16>(x, w_r, a, num_sms, st, per_sm);
  if (E <= 128) return launch_tc<128, 6, TC_EPI_BIAS_F32, OP_BF16>(x, w_r, a, num_sms, st);
  return launch_tc<256, 4, TC_EPI_BIAS_F32, OP_BF16>(x, w_r, a, num_sms, st);
}

}  // namespace moe
