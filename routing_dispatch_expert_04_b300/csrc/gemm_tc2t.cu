// Grouped GEMM on CTA pairs with the tokens on the MMA's N side, sm_103a.
//
// Same computation as the other expert-GEMM kernels -- the expert FFN of "Expert
// Parallelism (MoE)", "MoE Layer Structure", for all experts in one launch:
//   C[r, n] = epi( sum_k A[r, k] * B[g*N + n, k] ),  r in [offsets[g], offsets[g+1]) --
// computed as its transpose, C^T = B . A^T, on CTA pairs (tcgen05.mma.cta_group::2):
//   - the MMA's M side (256 rows, 128 per CTA) is a tile of 256 weight rows (output
//     columns n), which always fills it when N is a multiple of 256;
//   - the N side is a tile of up to 256 of the group's rows (tokens), each CTA staging
//     half of them; the instruction's N is the tile's row count rounded up to 32, so a
//     group of 640 rows runs as 256 + 256 + 128 columns instead of three 256-row tiles
//     (cutting a group into equal tiles, 224 + 224 + 192, measured no faster: the tensor
//     pipe appears to spend a 256-column instruction's time on 192 or 224 columns);
//     each CTA loads its half of the tile with the smallest of three boxes (128, 64 or
//     32 rows) that covers it, so the bytes staged follow the tile;
//   - each CTA's TMEM holds its 128 weight rows x the tile's tokens, and the epilogue
//     writes the transpose: lane l of a warp owns output column n of a chunk of 32
//     tokens; for fp16 outputs the warp's 32 x 32 block goes through a shared-memory
//     buffer, token-major, and each lane then stores 16 contiguous bytes of a token row.
// Pipeline, barriers, bounded waits and teardown as in gemm_tc2.cu: warp 0 TMA producer,
// warp 1 TMEM owner + MMA issuer (even CTA), warps 2..5 epilogue, warp 6 stage watcher
// (even CTA; the stage gate of tc_common.cuh); both CTAs' copies
// signal the even CTA's "full" barrier, its commits arrive on both CTAs' "empty" and
// "accumulator full" barriers, both CTAs' epilogues arrive on its "accumulator empty".
// Tiles are (group, weight tile, token tile) with token tiles fastest, so the pairs that
// run together share the weight tile through L2.
#include "tc_common.cuh"

namespace moe {
using namespace tc;

constexpr int T2T_TILE = 256;    // weight rows per tile (M) and most tokens per tile (N)
constexpr int T2T_CTA_ROWS = 128;

template <int STAGES>
struct Tc2tLayout {
  static constexpr int W_BYTES = T2T_CTA_ROWS * TC_ROW_BYTES;  // this CTA's weight rows
  static constexpr int X_BYTES = T2T_CTA_ROWS * TC_ROW_BYTES;  // this CTA's token rows
  static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr int X_OFF = STAGES * W_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NBAR = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], done
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int GRP_OFF = MISC_OFF + 16;
  static constexpr int EPI_OFF = (GRP_OFF + (int)sizeof(GroupTable) + 15) / 16 * 16;
  static constexpr int EPI_BYTES = 32 * 32 * 2;  // per epilogue warp: 32 tokens x 32 columns, fp16
  static constexpr int TOTAL = EPI_OFF + 4 * EPI_BYTES;
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * T2T_TILE;
};

constexpr uint64_t T2T_ABORT_SETTLE_NS = 200000ull;

// Group table for this kernel: mt[g] = token tiles of group g; tiles per group =
// mt[g] * weight tiles.
__device__ __forceinline__ void build_token_tiles(GroupTable* tab, const TcArgs& args, int w_tiles,
                                                  int lane) {
  int carry = 0;
  for (int base = 0; base < args.G; base += 32) {
    const int g = base + lane;
    int lo = 0, hi = 0, nt = 0;
    if (g < args.G) {
      lo = args.offsets[g];
      hi = args.offsets[g + 1];
      if (hi > args.rows_cap) {
        raise_error(args.hdr, DEV_ERR_OVERFLOW);
        hi = (int)args.rows_cap;
      }
      if (lo < 0) lo = 0;
      if (lo > hi) lo = hi;
      nt = (hi - lo + T2T_TILE - 1) / T2T_TILE;
      tab->lo[g] = lo;
      tab->hi[g] = hi;
      tab->mt[g] = nt;
    }
    int v = nt * w_tiles;
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

struct TTile {
  int g;
  int tok0;   // first token row of the tile
  int ntok;   // token rows in the tile (<= 256)
  int ninst;  // instruction N: ntok rounded up to 32
  int w0;     // first weight row (output column) of the tile within the group
  int box;    // token box of each CTA: 0 (128 rows), 1 (64) or 2 (32) -- covers ninst/2
};

__device__ __forceinline__ TTile decode_ttile(int t, int G, const GroupTable* tab) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tab->tpre[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int g = lo;
  const int local = t - tab->tpre[g];
  const int nt = tab->mt[g];
  TTile ti;
  ti.g = g;
  ti.tok0 = tab->lo[g] + (local % nt) * T2T_TILE;
  ti.ntok = min(T2T_TILE, tab->hi[g] - ti.tok0);
  ti.ninst = (ti.ntok + 31) & ~31;
  ti.w0 = (local / nt) * T2T_TILE;
  const int half = ti.ninst >> 1;
  ti.box = half > 64 ? 0 : (half > 32 ? 1 : 2);
  return ti;
}

template <int STAGES, int EPI, int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS_GATED, 1)
tc2t_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x128,
                         const __grid_constant__ CUtensorMap tmap_x64,
                         const __grid_constant__ CUtensorMap tmap_x32,
                         const __grid_constant__ CUtensorMap tmap_w, const TcArgs args) {
  using Lay = Tc2tLayout<STAGES>;
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
  const int w_tiles = (args.N + T2T_TILE - 1) / T2T_TILE;
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
    tma_prefetch_desc(&tmap_x128);
    tma_prefetch_desc(&tmap_x64);
    tma_prefetch_desc(&tmap_x32);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 0) {
    build_token_tiles(tab, args, w_tiles, lane);
  } else if (warp == 1) {
    tmem_alloc_pair(s_tmem, Lay::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total = tab->tpre[G];

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = true;
      for (int t = cluster; t < total && ok; t += n_clusters) {
        const TTile ti = decode_ttile(t, G, tab);
        const int wrow = ti.g * args.N + ti.w0 + (int)rank * T2T_CTA_ROWS;
        const int xrow = ti.tok0 + (int)rank * (ti.ninst >> 1);
        const CUtensorMap* xmap = ti.box == 0 ? &tmap_x128 : (ti.box == 1 ? &tmap_x64 : &tmap_x32);
        const uint32_t stage_bytes = Lay::W_BYTES + ((uint32_t)T2T_CTA_ROWS >> ti.box) * TC_ROW_BYTES;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_phase(&empty[s], ph ^ 1u, s_abort, args.hdr)) {
            ok = false;
            break;
          }
          uint8_t* sw = smem + s * Lay::W_BYTES;
          uint8_t* sx = smem + Lay::X_OFF + s * Lay::X_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * stage_bytes);
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);  // the even CTA's full[s]
          tma_load_2d_pair(sw, &tmap_w, fb, kb * BKE, wrow);
          tma_load_2d_pair(sx, xmap, fb, kb * BKE, xrow);
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        if (rank == 0) {
          for (int i = 0; i < STAGES && i < issued; ++i) {
            if (--s < 0) {
              s = STAGES - 1;
              ph ^= 1u;
            }
            drain_wait(&full[s], ph);
          }
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < T2T_ABORT_SETTLE_NS) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------------------------------------------------------- MMA issuer
      // lane 0 issues; the whole warp waits on the stage gate (named barriers)
      const uint32_t idesc0 =
          KIND == OP_BF16 ? idesc_bf16_f32(T2T_TILE, 0) : idesc_fmt0_f32(T2T_TILE, 0);
      int s = 0;
      uint32_t acc = 0, aph = 0;
      for (int t = cluster; t < total; t += n_clusters) {
        const TTile ti = decode_ttile(t, G, tab);
        const uint32_t idesc = idesc0 | ((uint32_t)(ti.ninst >> 3) << 17);
        int ok = 1;
        if (lane == 0) ok = wait_phase(&tempty[acc], aph ^ 1u, s_abort, args.hdr) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const uint32_t d_tmem = tmem_base + acc * T2T_TILE;
        for (int kb = 0; kb < nkb; ++kb) {
          named_sync(TC_GATE_BAR0 + s, TC_GATE_THREADS);
          if (lane == 0) {
            tc_fence_after();
            const uint32_t w_addr = smem_u32(smem + s * Lay::W_BYTES);
            const uint32_t x_addr = smem_u32(smem + Lay::X_OFF + s * Lay::X_BYTES);
#pragma unroll
            for (int k = 0; k < TC_ROW_BYTES / 32; ++k) {  // 32 bytes of K per MMA
              if (KIND == OP_E4M3)
                mma_e4m3_pair(d_tmem, sdesc_sw128(w_addr + k * 32), sdesc_sw128(x_addr + k * 32),
                              idesc, (kb != 0 || k != 0) ? 1u : 0u);
              else
                mma_f16_pair(d_tmem, sdesc_sw128(w_addr + k * 32), sdesc_sw128(x_addr + k * 32),
                             idesc, (kb != 0 || k != 0) ? 1u : 0u);
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
    const int wl = (int)rank * T2T_CTA_ROWS + q * 32 + lane;  // weight row within the tile
    __half* epi_buf = (__half*)(smem + Lay::EPI_OFF + (warp - 2) * Lay::EPI_BYTES);
    uint32_t acc = 0, aph = 0;
    for (int t = cluster; t < total; t += n_clusters) {
      const TTile ti = decode_ttile(t, G, tab);
      if (!wait_phase(&tfull[acc], aph, s_abort, args.hdr)) break;
      tc_fence_after();
      const int col = ti.w0 + wl;
      const bool valid = col < args.N;
      const int tok_end = ti.tok0 + ti.ntok;
      const float sb = (KIND == OP_E4M3 && valid) ? args.b_scale[(size_t)ti.g * args.N + col] : 0.f;
#pragma unroll 1
      for (int c = 0; c < ti.ninst; c += 32) {  // warp-uniform
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + acc * T2T_TILE + c, r);
        tmem_ld_wait();
        if (EPI == TC_EPI_GELU_F16 || EPI == TC_EPI_F16) {  // whole warp, staged stores
          if (epilogue_chunk_t16<EPI, KIND>(r, col - lane, lane, ti.tok0 + c, tok_end, args, sb,
                                             epi_buf))
            raise_error(args.hdr, DEV_ERR_RANGE);
          continue;
        }
        if (!valid) continue;
        if (epilogue_chunk_t<EPI, KIND>(r, col, ti.tok0 + c, tok_end, args, sb))
          raise_error(args.hdr, DEV_ERR_RANGE);
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
static cudaError_t launch_tc2t(const void* X, const void* W, const TcArgs& a, int num_sms,
                               cudaStream_t st) {
  using Lay = Tc2tLayout<STAGES>;
  static bool attr_set = false;
  auto kern = tc2t_grouped_gemm_kernel<STAGES, EPI, KIND>;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap mx128, mx64, mx32, mw;
  const int64_t x_rows = a.rows_cap > 0 ? a.rows_cap : 1;
  if (!tc_make_map(&mx128, X, KIND, (uint64_t)a.Kd, (uint64_t)x_rows, 128) ||
      !tc_make_map(&mx64, X, KIND, (uint64_t)a.Kd, (uint64_t)x_rows, 64) ||
      !tc_make_map(&mx32, X, KIND, (uint64_t)a.Kd, (uint64_t)x_rows, 32))
    return cudaErrorInvalidValue;
  if (!tc_make_map(&mw, W, KIND, (uint64_t)a.Kd, (uint64_t)a.G * a.N, T2T_CTA_ROWS))
    return cudaErrorInvalidValue;
  const int64_t w_tiles = (a.N + T2T_TILE - 1) / T2T_TILE;
  const int64_t t_bound = (a.rows_cap + T2T_TILE - 1) / T2T_TILE + a.G;
  int64_t clusters = w_tiles * t_bound;
  if (clusters > num_sms / 2) clusters = num_sms / 2;
  if (clusters < 1) clusters = 1;
  kern<<<(unsigned)(2 * clusters), TC_THREADS_GATED, Lay::ALLOC, st>>>(mx128, mx64, mx32, mw, a);
  count_launch();
  return cudaGetLastError();
}

// First expert Linear, tokens on the N side: h = GELU(x_perm . W1[g]^T), fp16 out.
cudaError_t launch_tc2t_up(const void* x_perm, const void* w1, void* h, const int32_t* offsets,
                           int G, int N, int Kd, int64_t rows_cap, uint32_t* hdr, int num_sms,
                           cudaStream_t st) {
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, h, N, nullptr, hdr, 1, 0, 0, TC_ROWS_ALL};
  return launch_tc2t<6, TC_EPI_GELU_F16, OP_BF16>(x_perm, w1, a, num_sms, st);
}

// Second expert Linear, tokens on the N side: y_perm = h . W2[g]^T, fp16 out.
cudaError_t launch_tc2t_down(const void* h, const void* w2h, void* y_perm, const int32_t* offsets,
                             int G, int N, int Kd, int64_t rows_cap, uint32_t* hdr, int num_sms,
                             cudaStream_t st) {
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, y_perm, N, nullptr, hdr, 1, 0, 0, TC_ROWS_ALL};
  return launch_tc2t<6, TC_EPI_F16, OP_F16>(h, w2h, a, num_sms, st);
}

// The same two Linears on E4M3 operands (codes + per-row scales of the packed rows and of
// the stacked weight rows, applied in the epilogue).
cudaError_t launch_tc2t_up_e4m3(const void* xq, const float* sx, const void* w1q, const float* sw1,
                                void* h, const int32_t* offsets, int G, int N, int Kd,
                                int64_t rows_cap, uint32_t* hdr, int num_sms, cudaStream_t st) {
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, h, N, nullptr, hdr, 1, 0, 0, TC_ROWS_ALL,
           nullptr, 1, 0, sx, sw1};
  return launch_tc2t<6, TC_EPI_GELU_F16, OP_E4M3>(xq, w1q, a, num_sms, st);
}

cudaError_t launch_tc2t_down_e4m3(const void* hq, const float* sh, const void* w2q, const float* sw2,
                                  void* y_perm, const int32_t* offsets, int G, int N, int Kd,
                                  int64_t rows_cap, uint32_t* hdr, int num_sms, cudaStream_t st) {
  TcArgs a{offsets, G, 0, N, Kd, rows_cap, y_perm, N, nullptr, hdr, 1, 0, 0, TC_ROWS_ALL,
           nullptr, 1, 0, sh, sw2};
  return launch_tc2t<6, TC_EPI_F16, OP_E4M3>(hq, w2q, a, num_sms, st);
}

}  // namespace moe
