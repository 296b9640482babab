// Grouped GEMM on CTA pairs: tcgen05.mma.cta_group::2 over two SMs, sm_103a.
//
// Same computation and tile list as the one-CTA kernel (gemm_tc.cu) -- the expert FFN
// of "Expert Parallelism (MoE)", "MoE Layer Structure", for all experts in one launch --
// with 256-row tiles computed by a cluster of two CTAs:
//   - each CTA TMA-loads its own 128 rows of the A tile and its own half (BN/2 rows) of
//     the B tile into its shared memory, so a CTA streams 32 KB per 64-deep k-block
//     instead of 48 KB, and six stages fit where the one-CTA kernel holds four;
//   - the even CTA issues one M=256 x N=BN MMA that reads both CTAs' stages; each CTA's
//     TMEM receives its 128 rows of the accumulator (two accumulators of BN columns);
//   - both CTAs' copies signal the even CTA's "full" barrier (it expects both CTAs'
//     bytes); its MMA commits arrive on the "empty" and "accumulator full" barriers of
//     both CTAs; both CTAs' epilogue warps arrive on the even CTA's "accumulator empty"
//     barrier, which therefore counts 8 warps.
// Roles per CTA: warp 0 TMA producer, warp 1 TMEM owner (+ MMA issuer in the even CTA),
// warps 2..5 epilogue (same fused GELU / fp32 epilogues as the one-CTA kernel), warp 6
// (even CTA) the stage watcher of the one-CTA kernel's stage gate.
// Every mbarrier wait is bounded (the CTA records a timeout and leaves its loops); the
// pair meets at a cluster barrier before TMEM is freed, so neither CTA exits while the
// other's MMAs or copies may still touch its shared memory or TMEM.
#include "tc_common.cuh"

namespace moe {
using namespace tc;

constexpr int TC2_BM = 256;      // rows per pair tile
constexpr int TC2_CTA_ROWS = 128;

template <int BN, int STAGES>
struct Tc2Layout {
  static constexpr int A_BYTES = TC2_CTA_ROWS * TC_ROW_BYTES;
  static constexpr int B_BYTES = (BN / 2) * TC_ROW_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int B_OFF = STAGES * A_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NBAR = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], done
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int GRP_OFF = MISC_OFF + 16;
  static constexpr int TOTAL = GRP_OFF + (int)sizeof(GroupTable);
  static constexpr int ALLOC = TOTAL + 1024;
  // two accumulators of BN columns in a power-of-two allocation
  static constexpr uint32_t TMEM_COLS = BN == 192 ? 512 : 2 * BN;
  static_assert(BN == 128 || BN == 192 || BN == 256, "pair tiles are 128, 192 or 256 wide");
};

// Time an aborting CTA gives copies it cannot observe (they signal the other CTA's
// barrier) to land before its shared memory is released.
constexpr uint64_t PAIR_ABORT_SETTLE_NS = 200000ull;

template <int BN, int STAGES, int EPI, int KIND, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS_GATED, 1)
tc2_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const TcArgs args) {
  using Lay = Tc2Layout<BN, STAGES>;
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
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
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
      mbar_init(&tempty[i], 8);
    }
    mbar_init(done, 1);
    *s_abort = 0;
    *s_mma_left = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 0) {
    build_group_table<TC2_BM>(tab, args, n_tiles, lane);
  } else if (warp == 1) {
    tmem_alloc_pair(s_tmem, Lay::TMEM_COLS);
    tmem_relinquish_pair();
  }
  // barriers of both CTAs initialised and TMEM allocated before anyone uses them
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total = tab->tpre[G];

  if (warp == 0) {
    if (GATHER || lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      // Plain A: lane 0 issues one box per k-block.  Gathered A: every lane gathers four
      // of this CTA's 128 rows (tile::gather4) into their place in the stage.
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = true;
      for (int t = cluster; t < total && ok; t += n_clusters) {
        const TileInfo ti = decode_tile<TC2_BM>(t, G, tab, BN);
        const int arow = ti.row0 + (int)rank * TC2_CTA_ROWS;
        const int brow = ti.g * args.N + ti.n0 + (int)rank * (BN / 2);
        int tok[4] = {0, 0, 0, 0};
        if (GATHER) {
#pragma unroll
          for (int i = 0; i < 4; ++i) tok[i] = gather_row(args, arow + 4 * lane + i, ti.rowend);
        }
        for (int kb = 0; kb < nkb; ++kb) {
          bool got = true;
          if (lane == 0) got = wait_phase(&empty[s], ph ^ 1u, s_abort, args.hdr);
          if (GATHER) got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * Lay::A_BYTES;
          uint8_t* sb = smem + Lay::B_OFF + s * Lay::B_BYTES;
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);  // the even CTA's full[s]
          if (lane == 0) {
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * Lay::STAGE_BYTES);
            if (!GATHER) tma_load_2d_pair(sa, &tmap_a, fb, kb * BKE, arow);
            tma_load_2d_pair(sb, &tmap_b, fb, kb * BKE, brow);
          }
          if (GATHER) {
            __syncwarp();
            tma_gather4_pair(sa + lane * 4 * TC_ROW_BYTES, &tmap_a, fb, kb * BKE, tok[0], tok[1],
                             tok[2], tok[3]);
          }
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && lane == 0) {
        if (rank == 0) {  // the even CTA can see its stages complete
          for (int i = 0; i < STAGES && i < issued; ++i) {
            if (--s < 0) {
              s = STAGES - 1;
              ph ^= 1u;
            }
            drain_wait(&full[s], ph);
          }
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < PAIR_ABORT_SETTLE_NS) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------------------------------------------------------- MMA issuer
      // lane 0 issues; the whole warp waits on the stage gate (named barriers)
      constexpr uint32_t IDESC = KIND == OP_BF16 ? idesc_bf16_f32(TC2_BM, BN)
                                                : idesc_fmt0_f32(TC2_BM, BN);
      int s = 0;
      uint32_t acc = 0, aph = 0;
      for (int t = cluster; t < total; t += n_clusters) {
        int ok = 1;
        if (lane == 0) ok = wait_phase(&tempty[acc], aph ^ 1u, s_abort, args.hdr) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          named_sync(TC_GATE_BAR0 + s, TC_GATE_THREADS);
          if (lane == 0) {
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + s * Lay::A_BYTES);
            const uint32_t b_addr = smem_u32(smem + Lay::B_OFF + s * Lay::B_BYTES);
#pragma unroll
            for (int k = 0; k < TC_ROW_BYTES / 32; ++k) {  // 32 bytes of K per MMA
              if (KIND == OP_E4M3)
                mma_e4m3_pair(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32),
                              IDESC, (kb != 0 || k != 0) ? 1u : 0u);
              else
                mma_f16_pair(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32),
                             IDESC, (kb != 0 || k != 0) ? 1u : 0u);
            }
            mma_commit_pair_mc(&empty[s], (uint16_t)3);
          }
          __syncwarp();
          if (++s == STAGES) s = 0;
        }
        if (lane == 0) mma_commit_pair_mc(&tfull[acc], (uint16_t)3);
        __syncwarp();
        acc ^= 1u;
        if (acc == 0) aph ^= 1u;
      }
      if (lane == 0) {
        *s_mma_left = 1;  // the watcher stops arriving
        // every MMA issued by this thread has completed once `done` flips
        mma_commit_pair_local(done);
        drain_wait(done, 0);
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    if (rank == 0) {
      // -------------------------------------------------------------- stage watcher
      int s = 0;
      uint32_t ph = 0;
      bool gave_up = false, go = true;
      for (int t = cluster; t < total && go; t += n_clusters) {
        for (int kb = 0; kb < nkb && go; ++kb) {
          go = gate_arrive(s, full, empty, ph, gave_up, s_abort, s_mma_left, args.hdr, lane);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in_tile = (int)rank * TC2_CTA_ROWS + q * 32 + lane;
    uint32_t acc = 0, aph = 0;
    for (int t = cluster; t < total; t += n_clusters) {
      const TileInfo ti = decode_tile<TC2_BM>(t, G, tab, BN);
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
        if (epilogue_chunk<EPI>(r, row, col0, args, 0, nullptr)) raise_error(args.hdr, DEV_ERR_RANGE);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      acc ^= 1u;
      if (acc == 0) aph ^= 1u;
    }
  }

  __syncwarp();
  if (threadIdx.x == 0) clock_telemetry_add(args.hdr, clk0, ns0);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, Lay::TMEM_COLS);
}

template <int BN, int STAGES, int EPI, int KIND, bool GATHER>
static cudaError_t launch_tc2(const void* A, const void* B, const TcArgs& a, int num_sms,
                              cudaStream_t st) {
  using Lay = Tc2Layout<BN, STAGES>;
  static bool attr_set = false;
  auto kern = tc2_grouped_gemm_kernel<BN, STAGES, EPI, KIND, GATHER>;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap ma, mb;
  const int64_t a_rows = a.rows_cap > 0 ? a.rows_cap : 1;
  const bool ok_a = GATHER ? tc_make_map(&ma, A, KIND, (uint64_t)a.Kd, (uint64_t)a.gather_rows, 1)
                           : tc_make_map(&ma, A, KIND, (uint64_t)a.Kd, (uint64_t)a_rows,
                                         TC2_CTA_ROWS);
  if (!ok_a) return cudaErrorInvalidValue;
  if (!tc_make_map(&mb, B, KIND, (uint64_t)a.Kd, (uint64_t)a.G * a.N, BN / 2))
    return cudaErrorInvalidValue;
  const int64_t n_tiles = (a.N + BN - 1) / BN;
  const int64_t m_bound = (a.rows_cap + TC2_BM - 1) / TC2_BM + (a.offsets ? a.G : 0);
  int64_t clusters = m_bound * n_tiles;
  if (clusters > num_sms / 2) clusters = num_sms / 2;
  if (clusters < 1) clusters = 1;
  kern<<<(unsigned)(2 * clusters), TC_THREADS_GATED, Lay::ALLOC, st>>>(ma, mb, a);
  count_launch();
  return cudaGetLastError();
}

// First expert Linear on CTA pairs, bf16 in, GELU fused, fp16 out, over the rows that
// `row_part` selects; with `gather_src` the A rows are gathered from the token matrix.
// `bn`: tile width, 256 or (without a gather) 192.
cudaError_t launch_tc2_up(const void* a_in, const int32_t* gather_src, int gather_k,
                          int64_t gather_rows, const void* w1, void* h, const int32_t* offsets,
                          int G, int N, int Kd, int64_t rows_cap, int row_part, int bn,
                          uint32_t* hdr, int num_sms, cudaStream_t st) {
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, h, N, nullptr, hdr, 1, (Kd + TC_BK - 1) / TC_BK, 0,
           row_part, gather_src, gather_k, gather_rows};
  if (gather_src != nullptr)
    return launch_tc2<256, 6, TC_EPI_GELU_F16, OP_BF16, true>(a_in, w1, a, num_sms, st);
  if (bn == 192)
    return launch_tc2<192, 7, TC_EPI_GELU_F16, OP_BF16, false>(a_in, w1, a, num_sms, st);
  return launch_tc2<256, 6, TC_EPI_GELU_F16, OP_BF16, false>(a_in, w1, a, num_sms, st);
}

// Expert Linears on CTA pairs with E4M3 operands (codes + per-row scales applied in the
// epilogue): the first with GELU (rows optionally gathered), the second with fp16 out.
cudaError_t launch_tc2_up_e4m3(const void* xq, const float* sx, const int32_t* gather_src,
                               int gather_k, int64_t gather_rows, const void* w1q, const float* sw1,
                               void* h, const int32_t* offsets, int G, int N, int Kd,
                               int64_t rows_cap, int row_part, uint32_t* hdr, int num_sms,
                               cudaStream_t st) {
  constexpr int BKE = OpKind<OP_E4M3>::BK;
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, h, N, nullptr, hdr, 1, (Kd + BKE - 1) / BKE, 0,
           row_part, gather_src, gather_k, gather_rows, sx, sw1};
  if (gather_src != nullptr)
    return launch_tc2<256, 6, TC_EPI_GELU_F16, OP_E4M3, true>(xq, w1q, a, num_sms, st);
  return launch_tc2<256, 6, TC_EPI_GELU_F16, OP_E4M3, false>(xq, w1q, a, num_sms, st);
}

cudaError_t launch_tc2_down_e4m3(const void* hq, const float* sh, const void* w2q, const float* sw2,
                                 void* y_perm, const int32_t* offsets, int G, int N, int Kd,
                                 int64_t rows_cap, int row_part, uint32_t* hdr, int num_sms,
                                 cudaStream_t st) {
  constexpr int BKE = OpKind<OP_E4M3>::BK;
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, y_perm, N, nullptr, hdr, 1, (Kd + BKE - 1) / BKE, 0,
           row_part, nullptr, 1, 0, sh, sw2};
  return launch_tc2<256, 6, TC_EPI_F16, OP_E4M3, false>(hq, w2q, a, num_sms, st);
}

// Second expert Linear on CTA pairs, fp16 in, fp16 out; `bn` as for the first.
cudaError_t launch_tc2_down(const void* h, const void* w2h, void* y_perm, const int32_t* offsets,
                            int G, int N, int Kd, int64_t rows_cap, int row_part, int bn,
                            uint32_t* hdr, int num_sms, cudaStream_t st) {
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, y_perm, N, nullptr, hdr, 1, (Kd + TC_BK - 1) / TC_BK, 0,
           row_part};
  if (bn == 192) return launch_tc2<192, 7, TC_EPI_F16, OP_F16, false>(h, w2h, a, num_sms, st);
  return launch_tc2<256, 6, TC_EPI_F16, OP_F16, false>(h, w2h, a, num_sms, st);
}

}  // namespace moe
