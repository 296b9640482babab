// Grouped GEMM on CTA pairs with mixed tiles: whole 256-row tiles and, for each group's
// remainder, one transposed tile -- all in one persistent launch, sm_103a.
//
// Same computation as the other expert-GEMM kernels -- the expert FFN of "Expert
// Parallelism (MoE)", "MoE Layer Structure", for all experts in one launch:
//   C[r, n] = epi( sum_k A[r, k] * B[g*N + n, k] ),  r in [offsets[g], offsets[g+1]).
// A group of R rows is covered, per 256-wide slab of output columns, by floor(R/256)
// tiles of 256 rows computed as in gemm_tc2.cu (tcgen05.mma.cta_group::2, M=256 rows
// with 128 per CTA, N=256 columns with each CTA staging half of the weight rows) and, if
// R is not a multiple of 256, by one tile of the remaining R mod 256 rows computed as in
// gemm_tc2t.cu: the transpose C^T = B . A^T with the slab's 256 weight rows on the MMA's M
// side (128 per CTA) and the remaining rows on its N side, sized to them (rounded up to
// 32), so no group is padded to 256 rows.  Both kinds of tile stage exactly the same
// weight box -- the slab's 256 weight rows, 128 per CTA -- so they share one shared-memory
// layout and one pipeline, and only the operand roles of the MMA, the instruction's N and
// the epilogue differ.  Tiles are (group, slab, m-tile) with the remainder tile the last
// m-tile of its slab, so the pairs that run together walk each weight slab once between
// them (the split plan instead ran the remainders as a second kernel on other SMs).
// Pipeline, barriers, bounded waits and teardown as in gemm_tc2.cu: warp 0 TMA producer,
// warp 1 TMEM owner + MMA issuer (even CTA), warps 2..5 epilogue, warp 6 stage watcher
// (even CTA; the stage gate of tc_common.cuh); both CTAs' copies
// signal the even CTA's "full" barrier, its commits arrive on both CTAs' "empty" and
// "accumulator full" barriers, both CTAs' epilogues arrive on its "accumulator empty".
#include "tc_common.cuh"

namespace moe {
using namespace tc;

constexpr int TM_TILE = 256;      // rows of a whole tile; weight rows (columns) of every tile
constexpr int TM_CTA_ROWS = 128;

template <int STAGES>
struct Tc2mLayout {
  static constexpr int A_BYTES = TM_CTA_ROWS * TC_ROW_BYTES;  // this CTA's token rows (<= 128)
  static constexpr int B_BYTES = TM_CTA_ROWS * TC_ROW_BYTES;  // this CTA's weight rows
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int B_OFF = STAGES * A_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NBAR = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], done
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int GRP_OFF = MISC_OFF + 16;
  static constexpr int EPI_OFF = (GRP_OFF + (int)sizeof(GroupTable) + 15) / 16 * 16;
  static constexpr int EPI_BYTES = 32 * 32 * 2;  // per epilogue warp: a 32 x 32 fp16 block
  static constexpr int TOTAL = EPI_OFF + 4 * EPI_BYTES;
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * TM_TILE;
};

constexpr uint64_t T2M_ABORT_SETTLE_NS = 200000ull;

// Group table: mt[g] = whole 256-row tiles of group g plus one for a remainder; tiles per
// group = mt[g] * slabs.
__device__ __forceinline__ void build_mixed_tiles(GroupTable* tab, const TcArgs& args, int slabs,
                                                  int lane) {
  int carry = 0;
  for (int base = 0; base < args.G; base += 32) {
    const int g = base + lane;
    int lo = 0, hi = 0, mt = 0;
    if (g < args.G) {
      lo = args.offsets[g];
      hi = args.offsets[g + 1];
      if (hi > args.rows_cap) {
        raise_error(args.hdr, DEV_ERR_OVERFLOW);
        hi = (int)args.rows_cap;
      }
      if (lo < 0) lo = 0;
      if (lo > hi) lo = hi;
      mt = (hi - lo + TM_TILE - 1) / TM_TILE;
      tab->lo[g] = lo;
      tab->hi[g] = hi;
      tab->mt[g] = mt;
    }
    int v = mt * slabs;  // inclusive warp scan of tiles
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

struct MTile {
  int g;
  int row0;     // first row of the tile
  int rowend;   // end of the tile's valid rows (the group's end)
  int n0;       // first output column (weight row within the group)
  bool tr;      // transposed remainder tile
  int ninst;    // transposed: instruction N (rows rounded up to 32)
  int box;      // transposed: row box of each CTA, 0 (128 rows), 1 (64) or 2 (32)
};

__device__ __forceinline__ MTile decode_mtile(int t, int G, const GroupTable* tab) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tab->tpre[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int g = lo;
  const int local = t - tab->tpre[g];
  const int mt = tab->mt[g];
  const int m = local % mt;
  MTile ti;
  ti.g = g;
  ti.row0 = tab->lo[g] + m * TM_TILE;
  ti.rowend = tab->hi[g];
  ti.n0 = (local / mt) * TM_TILE;
  const int rows = ti.rowend - ti.row0;
  ti.tr = rows < TM_TILE;
  ti.ninst = (rows + 31) & ~31;
  const int half = ti.ninst >> 1;
  ti.box = half > 64 ? 0 : (half > 32 ? 1 : 2);
  return ti;
}

template <int STAGES, int EPI, int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS_GATED, 1)
tc2m_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a128,
                         const __grid_constant__ CUtensorMap tmap_a64,
                         const __grid_constant__ CUtensorMap tmap_a32,
                         const __grid_constant__ CUtensorMap tmap_b, const TcArgs args) {
  static_assert(KIND != OP_E4M3, "the mixed-tile kernel takes 16-bit operands");
  static_assert(EPI == TC_EPI_GELU_F16 || EPI == TC_EPI_F16, "fp16 outputs only");
  using Lay = Tc2mLayout<STAGES>;
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
  const int slabs = (args.N + TM_TILE - 1) / TM_TILE;
  constexpr int BKE = OpKind<KIND>::BK;
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
    tma_prefetch_desc(&tmap_a128);
    tma_prefetch_desc(&tmap_a64);
    tma_prefetch_desc(&tmap_a32);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 0) {
    build_mixed_tiles(tab, args, slabs, lane);
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
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      // Every tile stages the slab's weight rows (128 per CTA); a whole tile 128 of its
      // rows per CTA, a remainder tile half of its instruction N per CTA, with the
      // smallest box that covers it.
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = true;
      for (int t = cluster; t < total && ok; t += n_clusters) {
        const MTile ti = decode_mtile(t, G, tab);
        const int brow = ti.g * args.N + ti.n0 + (int)rank * TM_CTA_ROWS;
        int arow = ti.row0 + (int)rank * TM_CTA_ROWS;
        const CUtensorMap* amap = &tmap_a128;
        uint32_t a_bytes = Lay::A_BYTES;
        if (ti.tr) {
          arow = ti.row0 + (int)rank * (ti.ninst >> 1);
          amap = ti.box == 0 ? &tmap_a128 : (ti.box == 1 ? &tmap_a64 : &tmap_a32);
          a_bytes = ((uint32_t)TM_CTA_ROWS >> ti.box) * TC_ROW_BYTES;
        }
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_phase(&empty[s], ph ^ 1u, s_abort, args.hdr)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * Lay::A_BYTES;
          uint8_t* sb = smem + Lay::B_OFF + s * Lay::B_BYTES;
          // both CTAs' bytes land on the even CTA's full[s]
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (Lay::B_BYTES + a_bytes));
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
          tma_load_2d_pair(sa, amap, fb, kb * BKE, arow);
          tma_load_2d_pair(sb, &tmap_b, fb, kb * BKE, brow);
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
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
          while (globaltimer_ns() - t0 < T2M_ABORT_SETTLE_NS) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------------------------------------------------------- MMA issuer
      // Whole tile: D[rows, cols] += A(rows) . B(cols)^T, M=256, N=256.
      // Remainder tile: D[cols, rows] += B(cols) . A(rows)^T, M=256, N = its rows.
      // lane 0 issues; the whole warp waits on the stage gate (named barriers)
      const uint32_t idesc_whole =
          KIND == OP_BF16 ? idesc_bf16_f32(TM_TILE, TM_TILE) : idesc_fmt0_f32(TM_TILE, TM_TILE);
      const uint32_t idesc_tr0 =
          KIND == OP_BF16 ? idesc_bf16_f32(TM_TILE, 0) : idesc_fmt0_f32(TM_TILE, 0);
      int s = 0;
      uint32_t acc = 0, aph = 0;
      for (int t = cluster; t < total; t += n_clusters) {
        const MTile ti = decode_mtile(t, G, tab);
        const uint32_t idesc = ti.tr ? (idesc_tr0 | ((uint32_t)(ti.ninst >> 3) << 17)) : idesc_whole;
        int ok = 1;
        if (lane == 0) ok = wait_phase(&tempty[acc], aph ^ 1u, s_abort, args.hdr) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const uint32_t d_tmem = tmem_base + acc * TM_TILE;
        for (int kb = 0; kb < nkb; ++kb) {
          named_sync(TC_GATE_BAR0 + s, TC_GATE_THREADS);
          if (lane == 0) {
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + s * Lay::A_BYTES);
            const uint32_t b_addr = smem_u32(smem + Lay::B_OFF + s * Lay::B_BYTES);
            const uint32_t m_addr = ti.tr ? b_addr : a_addr;  // operand on the MMA's M side
            const uint32_t n_addr = ti.tr ? a_addr : b_addr;  // and on its N side
#pragma unroll
            for (int k = 0; k < TC_ROW_BYTES / 32; ++k)  // 32 bytes of K per MMA
              mma_f16_pair(d_tmem, sdesc_sw128(m_addr + k * 32), sdesc_sw128(n_addr + k * 32),
                           idesc, (kb != 0 || k != 0) ? 1u : 0u);
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
    const int lrow = (int)rank * TM_CTA_ROWS + q * 32 + lane;  // this thread's TMEM lane in the tile
    __half* epi_buf = (__half*)(smem + Lay::EPI_OFF + (warp - 2) * Lay::EPI_BYTES);
    uint32_t acc = 0, aph = 0;
    for (int t = cluster; t < total; t += n_clusters) {
      const MTile ti = decode_mtile(t, G, tab);
      if (!wait_phase(&tfull[acc], aph, s_abort, args.hdr)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * TM_TILE;
      if (!ti.tr) {
        // whole tile: this lane holds output row row0 + lrow, 32 columns per load
        const int row = ti.row0 + lrow;
        const bool valid = row < ti.rowend;
#pragma unroll 1
        for (int c = 0; c < TM_TILE / 32; ++c) {
          const int col0 = ti.n0 + c * 32;
          if (col0 >= args.N) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + c * 32, r);
          tmem_ld_wait();
          if (!valid) continue;
          if (epilogue_chunk<EPI>(r, row, col0, args, 0, nullptr)) raise_error(args.hdr, DEV_ERR_RANGE);
        }
      } else {
        // remainder tile: this lane holds output column n0 + lrow, 32 rows per load
        const int col = ti.n0 + lrow;
#pragma unroll 1
        for (int c = 0; c < ti.ninst; c += 32) {  // warp-uniform
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + c, r);
          tmem_ld_wait();
          if (epilogue_chunk_t16<EPI, KIND>(r, col - lane, lane, ti.row0 + c, ti.rowend, args, 0.f,
                                             epi_buf))
            raise_error(args.hdr, DEV_ERR_RANGE);
        }
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

template <int STAGES, int EPI, int KIND>
static cudaError_t launch_tc2m(const void* X, const void* W, const TcArgs& a, int num_sms,
                               cudaStream_t st) {
  using Lay = Tc2mLayout<STAGES>;
  static bool attr_set = false;
  auto kern = tc2m_grouped_gemm_kernel<STAGES, EPI, KIND>;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap m128, m64, m32, mw;
  const int64_t x_rows = a.rows_cap > 0 ? a.rows_cap : 1;
  if (!tc_make_map(&m128, X, KIND, (uint64_t)a.Kd, (uint64_t)x_rows, 128) ||
      !tc_make_map(&m64, X, KIND, (uint64_t)a.Kd, (uint64_t)x_rows, 64) ||
      !tc_make_map(&m32, X, KIND, (uint64_t)a.Kd, (uint64_t)x_rows, 32))
    return cudaErrorInvalidValue;
  if (!tc_make_map(&mw, W, KIND, (uint64_t)a.Kd, (uint64_t)a.G * a.N, TM_CTA_ROWS))
    return cudaErrorInvalidValue;
  const int64_t slabs = (a.N + TM_TILE - 1) / TM_TILE;
  const int64_t t_bound = (a.rows_cap + TM_TILE - 1) / TM_TILE + a.G;
  int64_t clusters = slabs * t_bound;
  if (clusters > num_sms / 2) clusters = num_sms / 2;
  if (clusters < 1) clusters = 1;
  kern<<<(unsigned)(2 * clusters), TC_THREADS_GATED, Lay::ALLOC, st>>>(m128, m64, m32, mw, a);
  count_launch();
  return cudaGetLastError();
}

// First expert Linear with mixed tiles: h = GELU(x_perm . W1[g]^T), bf16 in, fp16 out.
cudaError_t launch_tc2m_up(const void* x_perm, const void* w1, void* h, const int32_t* offsets,
                           int G, int N, int Kd, int64_t rows_cap, uint32_t* hdr, int num_sms,
                           cudaStream_t st) {
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, h, N, nullptr, hdr, 1, 0, 0, TC_ROWS_ALL};
  return launch_tc2m<6, TC_EPI_GELU_F16, OP_BF16>(x_perm, w1, a, num_sms, st);
}

// Second expert Linear with mixed tiles: y_perm = h . W2[g]^T, fp16 in, fp16 out.
cudaError_t launch_tc2m_down(const void* h, const void* w2h, void* y_perm, const int32_t* offsets,
                             int G, int N, int Kd, int64_t rows_cap, uint32_t* hdr, int num_sms,
                             cudaStream_t st) {
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, y_perm, N, nullptr, hdr, 1, 0, 0, TC_ROWS_ALL};
  return launch_tc2m<6, TC_EPI_F16, OP_F16>(h, w2h, a, num_sms, st);
}

}  // namespace moe
