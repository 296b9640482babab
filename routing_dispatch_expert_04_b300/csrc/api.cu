// C-ABI entry points: argument validation, workspace carving and kernel launches.
// Every call only enqueues work on the caller's stream; nothing here synchronises the
// host except moe_sync_status.
#include <atomic>
#include <stdio.h>

#include "common.cuh"

namespace moe {

cudaError_t launch_softmax_topk(float* logits, int T, int E, int K, int renorm, int32_t* ids,
                                float* w, float* ppart, const float* lpart, int nsplit,
                                const float* bias, const float* sel_bias, const RoutePlan& plan,
                                cudaStream_t st);
cudaError_t launch_adjust_select_bias(const int32_t* counts, float* sel_bias, int E, int64_t A,
                                      float gamma, cudaStream_t st);
cudaError_t launch_scan(const int32_t* ids, int A, int E, int C, int nblk, unsigned long long* desc,
                        int32_t* pos, int32_t* counts, int32_t* offsets, uint32_t* hdr,
                        int skip_block, int spin_limit, int slot_major, int Tn, int K,
                        cudaStream_t st);
cudaError_t launch_dispatch(int dtype, const void* x, const int32_t* ids, const int32_t* pos,
                            const int32_t* base, int nbase, int tpb, const int32_t* offsets,
                            int Tn, int d, int E, int K, int C, int32_t* slot, int32_t* src,
                            void* xp, int64_t rows_cap, uint32_t* hdr, int num_sms,
                            cudaStream_t st);
cudaError_t launch_plan_scan(int32_t* pcnt, int nblk, int E, int C, int32_t* ptot, int32_t* counts,
                             int32_t* offsets, uint32_t* hdr, cudaStream_t st);
cudaError_t launch_combine(int dtype, const void* yp, const int32_t* slot, const float* w,
                           const void* ys, void* y, int Tn, int d, int K, int num_sms,
                           cudaStream_t st);
cudaError_t launch_aux(const int32_t* counts, const float* ppart, int E, int Tn, int K,
                       float alpha, float* f, float* P, float* l_aux, double* auxfp, uint32_t* hdr,
                       cudaStream_t st);
cudaError_t launch_aux_grad(const float* logits, const float* f, int Tn, int E, float alpha,
                            float* grad, int num_sms, cudaStream_t st);
cudaError_t launch_simt_grouped(int dtype, const void* A, const int32_t* gather_src, int gather_k,
                                int64_t gather_rows, const void* B, void* C,
                                const int32_t* offsets, int G, int N, int Kd, int64_t rows_cap,
                                bool gelu, uint32_t* hdr, cudaStream_t st);
cudaError_t launch_simt_router(int dtype, const void* x, const void* w_r, const float* b_r,
                               float* logits, int T, int E, int d, uint32_t* hdr, cudaStream_t st);
cudaError_t launch_tc_up(const void* a_in, const int32_t* gather_src, int gather_k,
                         int64_t gather_rows, const void* w1, void* h, const int32_t* offsets,
                         int G, int N, int Kd, int64_t rows_cap, int64_t cap_per_group,
                         int pair_mode, uint32_t* hdr, int num_sms, cudaStream_t st);
cudaError_t launch_tc_down(const void* h, const void* w2h, void* y_perm, const int32_t* offsets,
                           int G, int N, int Kd, int64_t rows_cap, int64_t cap_per_group,
                           int pair_mode, uint32_t* hdr, int num_sms, cudaStream_t st);
cudaError_t launch_tc_up_e4m3(const void* xq, const float* sx, const int32_t* gather_src,
                              int gather_k, int64_t gather_rows, const void* w1q, const float* sw1,
                              void* h, const int32_t* offsets, int G, int N, int Kd,
                              int64_t rows_cap, int64_t cap_per_group, int pair_mode,
                              uint32_t* hdr, int num_sms, cudaStream_t st);
cudaError_t launch_tc_down_e4m3(const void* hq, const float* sh, const void* w2q, const float* sw2,
                                void* y_perm, const int32_t* offsets, int G, int N, int Kd,
                                int64_t rows_cap, int64_t cap_per_group, int pair_mode,
                                uint32_t* hdr, int num_sms, cudaStream_t st);
cudaError_t launch_quantize_e4m3(int dtype, const void* src, int64_t rows, int cols,
                                 const int32_t* rows_dev, void* codes, float* scales, int num_sms,
                                 cudaStream_t st);
cudaError_t launch_tc_router(const void* x, const void* w_r, const float* b_r, float* out, int T,
                             int E, int d, int nsplit, uint32_t* hdr, int num_sms, cudaStream_t st);
cudaError_t launch_bf16_to_f16(const void* src, void* dst, int64_t n, uint32_t* hdr, int num_sms,
                               cudaStream_t st);

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<int> g_skip_block{-1};
static std::atomic<int> g_spin_limit{1 << 21};
static std::atomic<int> g_gemm_pairing{MOE_GEMM_AUTO};
static std::atomic<int> g_gemm_sms{0};  // SM budget of the expert GEMMs (0: all)

// The scan test hook (moe_test_arm_scan_timeout) for the next dispatch call, disarmed as
// it is taken: the block that withholds its counts (-1: none) and the spin limit.
void take_scan_test_hook(int* skip_block, int* spin_limit) {
  const int skip = g_skip_block.exchange(-1);
  *skip_block = skip;
  *spin_limit = skip >= 0 ? g_spin_limit.load() : (1 << 21);
}

static int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

// SMs the persistent expert GEMMs may occupy: the budget set by moe_set_gemm_sms, capped
// at the device's count, or all of them.
static int gemm_sms() {
  const int all = num_sms();
  const int n = g_gemm_sms.load();
  return (n > 0 && n < all) ? n : all;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

moe_status_t check_cfg(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID;
  if (c->T < 0 || c->d <= 0 || c->E <= 0 || c->K <= 0 || c->F <= 0) return MOE_ERR_INVALID;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID;
  if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID;
  if (c->drop_order != MOE_DROP_TOKEN_MAJOR && c->drop_order != MOE_DROP_SLOT_MAJOR)
    return MOE_ERR_INVALID;
  if (c->K > c->E) return MOE_ERR_INVALID;
  if (c->E > 256 || c->K > 32) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->K >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  const int vec = c->dtype == MOE_BF16 ? 8 : 4;
  if (c->d % vec != 0 || c->F % vec != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static moe_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  fprintf(stderr, "moe: CUDA error: %s\n", cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

// Most rows one group can hold (for tile planning only): C for the routed experts of a
// layer with dropping, the whole buffer for a single group; <= 0 when unknown.
static int64_t group_row_bound(const moe_config& c, int n_groups, int64_t rows_cap) {
  if (n_groups == 1) return rows_cap;
  if (n_groups == c.E && c.capacity >= 0) return c.capacity;
  return 0;
}

int64_t rows_capacity(const moe_config& c) {
  const int64_t A = (int64_t)c.T * c.K;
  if (c.capacity < 0) return A;
  const int64_t ec = (int64_t)c.E * c.capacity;
  return A < ec ? A : ec;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return ws_layout(*cfg).total;
}

int64_t moe_rows_capacity(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return -1;
  return rows_capacity(*cfg);
}

static moe_status_t route_impl(const moe_config* cfg, const void* x, const void* w_r,
                               const float* b_r, const float* sel_bias, float* logits,
                               int32_t* topk_ids, float* topk_w, void* ws, void* stream,
                               int32_t* counts = nullptr, int32_t* offsets = nullptr) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  const bool planned = counts != nullptr;
  if (c.T == 0) {  // nothing is read; a plan is empty
    if (!planned) return MOE_OK;
    s = cuda_status(cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, (cudaStream_t)stream));
    if (s != MOE_OK) return s;
    return cuda_status(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), (cudaStream_t)stream));
  }
  if (!logits || !topk_ids || !topk_w || !ws) return MOE_ERR_INVALID;
  if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(ws))
    return MOE_ERR_INVALID;
  if (x != nullptr && (w_r == nullptr || !aligned16(x) || !aligned16(w_r))) return MOE_ERR_INVALID;
  if (b_r != nullptr && !aligned16(b_r)) return MOE_ERR_INVALID;
  if (sel_bias != nullptr && ((uintptr_t)sel_bias & 3u)) return MOE_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(c);
  uint32_t* hdr = (uint32_t*)ws;
  const float* lpart = nullptr;
  if (x != nullptr) {
    if (c.dtype == MOE_BF16) {
      float* out = logits;
      if (L.router_splits > 1) {
        out = (float*)((char*)ws + L.lpart);
        lpart = out;
      }
      s = cuda_status(launch_tc_router(x, w_r, b_r, out, c.T, c.E, c.d, L.router_splits, hdr,
                                       num_sms(), st));
    } else {
      s = cuda_status(launch_simt_router(c.dtype, x, w_r, b_r, logits, c.T, c.E, c.d, hdr, st));
    }
    if (s != MOE_OK) return s;
  }
  RoutePlan plan{};
  plan.hdr = hdr;
  if (planned) plan = RoutePlan{(int32_t*)((char*)ws + L.pos), (int32_t*)((char*)ws + L.pcnt), hdr};
  s = cuda_status(launch_softmax_topk(logits, c.T, c.E, c.K, c.renormalize, topk_ids, topk_w,
                                      (float*)((char*)ws + L.ppart), lpart, L.router_splits, b_r,
                                      sel_bias, plan, st));
  if (s != MOE_OK || !planned) return s;
  return cuda_status(launch_plan_scan(plan.pcnt, L.nblk_plan, c.E, c.capacity,
                                      (int32_t*)((char*)ws + L.ptot), counts, offsets, hdr, st));
}

moe_status_t moe_route(const moe_config* cfg, const void* x, const void* w_r, const float* b_r,
                       float* logits, int32_t* topk_ids, float* topk_w, void* ws, void* stream) {
  return route_impl(cfg, x, w_r, b_r, nullptr, logits, topk_ids, topk_w, ws, stream);
}

moe_status_t moe_route_select_bias(const moe_config* cfg, const void* x, const void* w_r,
                                   const float* b_r, const float* sel_bias, float* logits,
                                   int32_t* topk_ids, float* topk_w, void* ws, void* stream) {
  if (sel_bias == nullptr) return MOE_ERR_INVALID;
  return route_impl(cfg, x, w_r, b_r, sel_bias, logits, topk_ids, topk_w, ws, stream);
}

moe_status_t moe_route_plan(const moe_config* cfg, const void* x, const void* w_r, const float* b_r,
                            const float* sel_bias, float* logits, int32_t* topk_ids, float* topk_w,
                            int32_t* counts, int32_t* offsets, void* ws, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (cfg->drop_order != MOE_DROP_TOKEN_MAJOR) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !aligned16(counts) || !aligned16(offsets)) return MOE_ERR_INVALID;
  if (sel_bias != nullptr && ((uintptr_t)sel_bias & 3u)) return MOE_ERR_INVALID;
  return route_impl(cfg, x, w_r, b_r, sel_bias, logits, topk_ids, topk_w, ws, stream, counts,
                    offsets);
}

moe_status_t moe_dispatch_planned(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                                  const int32_t* offsets, int32_t* slot, int32_t* src,
                                  void* x_perm, void* ws, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (c.drop_order != MOE_DROP_TOKEN_MAJOR) return MOE_ERR_UNSUPPORTED;
  const int A = c.T * c.K;
  if (A == 0) return MOE_OK;  // nothing is read or written
  if (!topk_ids || !offsets || !slot || !src || !ws) return MOE_ERR_INVALID;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID;
  if (!aligned16(topk_ids) || !aligned16(offsets) || !aligned16(slot) || !aligned16(src) ||
      !aligned16(ws))
    return MOE_ERR_INVALID;
  if (x != nullptr && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID;
  const WsLayout L = ws_layout(c);
  return cuda_status(launch_dispatch(c.dtype, x, topk_ids, (const int32_t*)((char*)ws + L.pos),
                                     (const int32_t*)((char*)ws + L.pcnt), L.nblk_plan,
                                     ROUTE_WARPS * route_plan_tpw(c.T), offsets, c.T, c.d, c.E,
                                     c.K, c.capacity, slot, src, x_perm, rows_capacity(c),
                                     (uint32_t*)ws, num_sms(), (cudaStream_t)stream));
}

moe_status_t moe_adjust_select_bias(const moe_config* cfg, const int32_t* counts, float* sel_bias,
                                    float gamma, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!counts || !sel_bias || ((uintptr_t)counts & 3u) || ((uintptr_t)sel_bias & 3u))
    return MOE_ERR_INVALID;
  if (!(gamma >= 0.0f) || isinf(gamma)) return MOE_ERR_INVALID;
  return cuda_status(launch_adjust_select_bias(counts, sel_bias, cfg->E,
                                               (int64_t)cfg->T * cfg->K, gamma,
                                               (cudaStream_t)stream));
}

moe_status_t moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                          int32_t* counts, int32_t* offsets, int32_t* slot, int32_t* src,
                          void* x_perm, void* ws, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  cudaStream_t st = (cudaStream_t)stream;
  const int A = c.T * c.K;
  if (!counts || !offsets || !aligned16(counts) || !aligned16(offsets)) return MOE_ERR_INVALID;
  if (A > 0) {
    if (!topk_ids || !slot || !src || !ws) return MOE_ERR_INVALID;
    if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID;
    if (!aligned16(topk_ids) || !aligned16(slot) || !aligned16(src) || !aligned16(ws))
      return MOE_ERR_INVALID;
    if (x != nullptr && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID;
  }
  if (A == 0) {
    s = cuda_status(cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, st));
    if (s != MOE_OK) return s;
    return cuda_status(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), st));
  }
  const WsLayout L = ws_layout(c);
  uint32_t* hdr = (uint32_t*)ws;
  int skip = -1, spin = 0;
  take_scan_test_hook(&skip, &spin);
  int32_t* pos = (int32_t*)((char*)ws + L.pos);
  s = cuda_status(launch_scan(topk_ids, A, c.E, c.capacity, L.nblk_scan,
                              (unsigned long long*)((char*)ws + L.desc), pos, counts, offsets, hdr,
                              skip, spin, c.drop_order, c.T, c.K, st));
  if (s != MOE_OK) return s;
  return cuda_status(launch_dispatch(c.dtype, x, topk_ids, pos, nullptr, 0, 1, offsets, c.T, c.d,
                                     c.E, c.K, c.capacity, slot, src, x_perm, rows_capacity(c),
                                     hdr, num_sms(), st));
}

static moe_status_t check_ffn_args(const moe_config* cfg, const void* in, const int32_t* offsets,
                                   int32_t n_groups, int64_t rows_cap, const void* w,
                                   const void* out, const void* ws) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (n_groups < 1 || n_groups > 256 || rows_cap < 0) return MOE_ERR_INVALID;
  if (rows_cap == 0) return MOE_OK;  // nothing is read or written
  if (rows_cap >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (!in || !offsets || !w || !out || !ws) return MOE_ERR_INVALID;
  if (!aligned16(in) || !aligned16(w) || !aligned16(out) || !aligned16(ws) || ((uintptr_t)offsets & 3))
    return MOE_ERR_INVALID;
  return MOE_OK;
}

static moe_status_t expert_up_impl(const moe_config& c, const void* a_in, const int32_t* gather_src,
                                   const int32_t* offsets, int32_t n_groups, int64_t rows_cap,
                                   const void* w1, void* h, void* ws, void* stream) {
  const int64_t gather_rows = gather_src != nullptr ? c.T : 0;
  if (c.dtype == MOE_BF16)
    return cuda_status(launch_tc_up(a_in, gather_src, c.K, gather_rows, w1, h, offsets, n_groups,
                                    c.F, c.d, rows_cap, group_row_bound(c, n_groups, rows_cap),
                                    g_gemm_pairing.load(), (uint32_t*)ws, gemm_sms(),
                                    (cudaStream_t)stream));
  return cuda_status(launch_simt_grouped(c.dtype, a_in, gather_src, c.K, gather_rows, w1, h, offsets,
                                         n_groups, c.F, c.d, rows_cap, true, (uint32_t*)ws,
                                         (cudaStream_t)stream));
}

moe_status_t moe_expert_up(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                           int32_t n_groups, int64_t rows_cap, const void* w1, void* h, void* ws,
                           void* stream) {
  moe_status_t s = check_ffn_args(cfg, x_perm, offsets, n_groups, rows_cap, w1, h, ws);
  if (s != MOE_OK) return s;
  if (rows_cap == 0) return MOE_OK;
  return expert_up_impl(*cfg, x_perm, nullptr, offsets, n_groups, rows_cap, w1, h, ws, stream);
}

moe_status_t moe_expert_up_gather(const moe_config* cfg, const void* x, const int32_t* src,
                                  const int32_t* offsets, int32_t n_groups, int64_t rows_cap,
                                  const void* w1, void* h, void* ws, void* stream) {
  moe_status_t s = check_ffn_args(cfg, x, offsets, n_groups, rows_cap, w1, h, ws);
  if (s != MOE_OK) return s;
  if (rows_cap == 0) return MOE_OK;
  if (src == nullptr || ((uintptr_t)src & 3u)) return MOE_ERR_INVALID;
  if (cfg->T == 0) return MOE_OK;  // no token rows: every group is empty
  return expert_up_impl(*cfg, x, src, offsets, n_groups, rows_cap, w1, h, ws, stream);
}

// E4M3 expert GEMMs: bf16 layers only; the K and N extents must be multiples of 16 (the
// E4M3 rows are TMA-loaded in 16-byte units).
static moe_status_t check_e4m3(const moe_config* cfg, const void* scale_a, const void* scale_b) {
  if (cfg->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (cfg->d % 16 != 0 || cfg->F % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (!scale_a || !scale_b || ((uintptr_t)scale_a & 3u) || ((uintptr_t)scale_b & 3u))
    return MOE_ERR_INVALID;
  return MOE_OK;
}

moe_status_t moe_expert_up_e4m3(const moe_config* cfg, const void* xq, const float* x_scale,
                                const int32_t* src, const int32_t* offsets, int32_t n_groups,
                                int64_t rows_cap, const void* w1q, const float* w1_scale, void* h,
                                void* ws, void* stream) {
  moe_status_t s = check_ffn_args(cfg, xq, offsets, n_groups, rows_cap, w1q, h, ws);
  if (s != MOE_OK || rows_cap == 0) return s;
  s = check_e4m3(cfg, x_scale, w1_scale);
  if (s != MOE_OK) return s;
  if (src != nullptr && ((uintptr_t)src & 3u)) return MOE_ERR_INVALID;
  const moe_config& c = *cfg;
  if (src != nullptr && c.T == 0) return MOE_OK;
  return cuda_status(launch_tc_up_e4m3(xq, x_scale, src, c.K, src != nullptr ? c.T : 0, w1q,
                                       w1_scale, h, offsets, n_groups, c.F, c.d, rows_cap,
                                       group_row_bound(c, n_groups, rows_cap),
                                       g_gemm_pairing.load(), (uint32_t*)ws, gemm_sms(),
                                       (cudaStream_t)stream));
}

moe_status_t moe_expert_down_e4m3(const moe_config* cfg, const void* hq, const float* h_scale,
                                  const int32_t* offsets, int32_t n_groups, int64_t rows_cap,
                                  const void* w2q, const float* w2_scale, void* y_perm, void* ws,
                                  void* stream) {
  moe_status_t s = check_ffn_args(cfg, hq, offsets, n_groups, rows_cap, w2q, y_perm, ws);
  if (s != MOE_OK || rows_cap == 0) return s;
  s = check_e4m3(cfg, h_scale, w2_scale);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  return cuda_status(launch_tc_down_e4m3(hq, h_scale, w2q, w2_scale, y_perm, offsets, n_groups,
                                         c.d, c.F, rows_cap, group_row_bound(c, n_groups, rows_cap),
                                         g_gemm_pairing.load(), (uint32_t*)ws, gemm_sms(),
                                         (cudaStream_t)stream));
}

moe_status_t moe_quantize_e4m3(const void* src, int32_t dtype, int64_t rows, int32_t cols,
                               const int32_t* rows_dev, void* codes, float* scales, void* stream) {
  if (dtype != MOE_F32 && dtype != MOE_BF16 && dtype != MOE_F16) return MOE_ERR_INVALID;
  if (rows < 0 || cols <= 0 || cols % 16 != 0) return MOE_ERR_INVALID;
  if (rows == 0) return MOE_OK;
  if (!src || !codes || !scales || !aligned16(src) || !aligned16(codes) || ((uintptr_t)scales & 3u))
    return MOE_ERR_INVALID;
  if (rows_dev != nullptr && ((uintptr_t)rows_dev & 3u)) return MOE_ERR_INVALID;
  return cuda_status(launch_quantize_e4m3(dtype, src, rows, cols, rows_dev, codes, scales,
                                          num_sms(), (cudaStream_t)stream));
}

moe_status_t moe_expert_down(const moe_config* cfg, const void* h, const int32_t* offsets,
                             int32_t n_groups, int64_t rows_cap, const void* w2, void* y_perm,
                             void* ws, void* stream) {
  moe_status_t s = check_ffn_args(cfg, h, offsets, n_groups, rows_cap, w2, y_perm, ws);
  if (s != MOE_OK) return s;
  if (rows_cap == 0) return MOE_OK;
  const moe_config& c = *cfg;
  if (c.dtype == MOE_BF16)
    return cuda_status(launch_tc_down(h, w2, y_perm, offsets, n_groups, c.d, c.F, rows_cap,
                                      group_row_bound(c, n_groups, rows_cap), g_gemm_pairing.load(),
                                      (uint32_t*)ws, gemm_sms(), (cudaStream_t)stream));
  return cuda_status(launch_simt_grouped(c.dtype, h, nullptr, 1, 0, w2, y_perm, offsets, n_groups,
                                         c.d, c.F, rows_cap, false, (uint32_t*)ws,
                                         (cudaStream_t)stream));
}

moe_status_t moe_grouped_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                             int32_t n_groups, int64_t rows_cap, const void* w1, const void* w2,
                             void* h, void* y_perm, void* ws, void* stream) {
  moe_status_t s = moe_expert_up(cfg, x_perm, offsets, n_groups, rows_cap, w1, h, ws, stream);
  if (s != MOE_OK) return s;
  return moe_expert_down(cfg, h, offsets, n_groups, rows_cap, w2, y_perm, ws, stream);
}

moe_status_t moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* slot,
                         const float* topk_w, const void* y_shared, void* y, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (c.T == 0) return MOE_OK;  // nothing is read or written
  if (!y_perm || !slot || !topk_w || !y) return MOE_ERR_INVALID;
  if (!aligned16(y_perm) || !aligned16(slot) || !aligned16(topk_w) || !aligned16(y)) return MOE_ERR_INVALID;
  if (y_shared != nullptr && !aligned16(y_shared)) return MOE_ERR_INVALID;
  return cuda_status(launch_combine(c.dtype, y_perm, slot, topk_w, y_shared, y, c.T, c.d, c.K,
                                    num_sms(), (cudaStream_t)stream));
}

moe_status_t moe_aux_stats(const moe_config* cfg, const int32_t* counts, const void* ws, float* f,
                           float* P, float* l_aux, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!counts || !ws || !f || !P || !l_aux) return MOE_ERR_INVALID;
  if (!aligned16(ws) || ((uintptr_t)counts & 3) || ((uintptr_t)f & 3) || ((uintptr_t)P & 3) ||
      ((uintptr_t)l_aux & 3))
    return MOE_ERR_INVALID;
  const WsLayout L = ws_layout(c);
  char* w = (char*)const_cast<void*>(ws);
  return cuda_status(launch_aux(counts, (const float*)(w + L.ppart), c.E, c.T, c.K,
                                c.alpha, f, P, l_aux, (double*)(w + L.auxfp), (uint32_t*)w,
                                (cudaStream_t)stream));
}

moe_status_t moe_aux_loss_grad(const moe_config* cfg, const float* logits, const float* f,
                               float* grad_logits, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (c.T == 0) return MOE_OK;
  if (!logits || !f || !grad_logits) return MOE_ERR_INVALID;
  if (((uintptr_t)logits & 3u) || ((uintptr_t)f & 3u) || ((uintptr_t)grad_logits & 3u))
    return MOE_ERR_INVALID;
  return cuda_status(launch_aux_grad(logits, f, c.T, c.E, c.alpha, grad_logits, num_sms(),
                                     (cudaStream_t)stream));
}

moe_status_t moe_bf16_to_f16(const void* src, void* dst, int64_t n, void* ws, void* stream) {
  if (n < 0 || (n % 8) != 0) return MOE_ERR_INVALID;
  if (n == 0) return MOE_OK;
  if (!src || !dst || !ws || !aligned16(src) || !aligned16(dst) || !aligned16(ws)) return MOE_ERR_INVALID;
  return cuda_status(launch_bf16_to_f16(src, dst, n, (uint32_t*)ws, num_sms(), (cudaStream_t)stream));
}

moe_status_t moe_sync_status(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  moe_status_t s = cuda_status(cudaStreamSynchronize(st));
  if (s != MOE_OK) return s;
  uint32_t word = 0;
  s = cuda_status(cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost));
  if (s != MOE_OK) return s;
  if (word != 0) {
    s = cuda_status(cudaMemset(ws, 0, sizeof(word)));
    if (s != MOE_OK) return s;
  }
  if (word & DEV_ERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (word & (DEV_ERR_BAD_ID | DEV_ERR_OVERFLOW | DEV_ERR_RANGE)) return MOE_ERR_DEVICE;
  return MOE_OK;
}

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID: return "MOE_ERR_INVALID";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

moe_status_t moe_set_gemm_sms(int32_t n) {
  if (n < 0 || n == 1) return MOE_ERR_INVALID;
  g_gemm_sms.store(n);
  return MOE_OK;
}

moe_status_t moe_set_gemm_pairing(int32_t mode) {
  if (mode != MOE_GEMM_AUTO && mode != MOE_GEMM_SINGLE && mode != MOE_GEMM_PAIR &&
      mode != MOE_GEMM_SPLIT && mode != MOE_GEMM_PAIR_T && mode != MOE_GEMM_MIXED)
    return MOE_ERR_INVALID;
  g_gemm_pairing.store(mode);
  return MOE_OK;
}

void moe_test_arm_scan_timeout(int32_t skip_block, int32_t spin_limit) {
  g_spin_limit.store(spin_limit > 0 ? spin_limit : 1);
  g_skip_block.store(skip_block);
}

}  // extern "C"
