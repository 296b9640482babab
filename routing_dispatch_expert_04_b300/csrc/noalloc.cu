// moe_dispatch_noalloc: the dispatch step with its scratch in a static device array.
//
// Some callers cannot allocate device memory at the point where they run the layer:
// code that runs inside a framework's custom allocator or memory pool, a plugin that is
// not allowed to call cudaMalloc, or an embedded runtime that reserved its memory up
// front.  moe_dispatch needs a caller-allocated workspace for its scan (per-chunk
// look-back descriptors, a chunk ticket, each assignment's position in its expert);
// this variant keeps that scratch in `g_dispatch_scratch` below instead, so the caller
// passes only the inputs and outputs.
//
// The array is a fixed NOALLOC_SCRATCH_BYTES (4 MiB) that every GPU which loads this
// library holds until the process exits.  Its device address is looked up once per
// device (cudaGetSymbolAddress, on the first call with that device current) -- in host
// code the symbol names a host-side stand-in, never a device address.  Its first word is
// the status word the kernels record device-side errors in; it keeps them, across calls,
// until moe_dispatch_noalloc_status reads and clears it.
#include <mutex>
#include <stdio.h>

#include "common.cuh"

namespace moe {

cudaError_t launch_scan(const int32_t* ids, int A, int E, int C, int nblk, unsigned long long* desc,
                        int32_t* pos, int32_t* counts, int32_t* offsets, uint32_t* hdr,
                        int skip_block, int spin_limit, int slot_major, int Tn, int K,
                        cudaStream_t st);
cudaError_t launch_dispatch(int dtype, const void* x, const int32_t* ids, const int32_t* pos,
                            const int32_t* base, int nbase, int tpb, const int32_t* offsets,
                            int Tn, int d, int E, int K, int C, int32_t* slot, int32_t* src,
                            void* xp, int64_t rows_cap, uint32_t* hdr, int num_sms,
                            cudaStream_t st);

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_dispatch_scratch[NOALLOC_SCRATCH_BYTES];

static std::mutex g_scratch_mu;
static void* g_scratch_addr[64] = {nullptr};
static int g_scratch_sms[64] = {0};

// Device address of g_dispatch_scratch (and the SM count) on the current device.
static cudaError_t scratch_for_current_device(void** addr, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
    g_scratch_sms[dev] = n > 0 ? n : 148;
  }
  *addr = g_scratch_addr[dev];
  *sms = g_scratch_sms[dev];
  return cudaSuccess;
}

static bool aligned16_na(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_noalloc(const moe_config* cfg, const void* x,
                                             const int32_t* topk_ids, int32_t* counts,
                                             int32_t* offsets, int32_t* slot, int32_t* src,
                                             void* x_perm, void* stream) {
  // the same configurations are accepted and rejected as by moe_dispatch
  const moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!counts || !offsets || !aligned16_na(counts) || !aligned16_na(offsets)) return MOE_ERR_INVALID;
  const int A = c.T * c.K;
  if (A > 0) {
    if (!topk_ids || !slot || !src) return MOE_ERR_INVALID;
    if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID;
    if (!aligned16_na(topk_ids) || !aligned16_na(slot) || !aligned16_na(src)) return MOE_ERR_INVALID;
    if (x != nullptr && (!aligned16_na(x) || !aligned16_na(x_perm))) return MOE_ERR_INVALID;
  }
  // scratch this call needs: header, look-back descriptors, positions
  const WsLayout L = ws_layout(c);
  const size_t need = L.ppart;
  if (need > NOALLOC_SCRATCH_BYTES) {
    fprintf(stderr,
            "moe_dispatch_noalloc: T*K=%d assignments over E=%d experts need %zu bytes of "
            "scratch; the static scratch holds %zu bytes (use moe_dispatch with a workspace)\n",
            A, c.E, need, NOALLOC_SCRATCH_BYTES);
    return MOE_ERR_UNSUPPORTED;
  }
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  if (A == 0) {
    e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), st);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  void* scratch = nullptr;
  int sms = 148;
  e = scratch_for_current_device(&scratch, &sms);
  if (e != cudaSuccess) {
    fprintf(stderr, "moe_dispatch_noalloc: %s\n", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  char* base = (char*)scratch;
  // the array keeps the previous call's contents: the scan's ticket is reset by the block
  // that finishes a call last and its descriptors carry the call's epoch, so none of it
  // needs clearing; the status word at offset 0 keeps an error until
  // moe_dispatch_noalloc_status reads it
  uint32_t* hdr = (uint32_t*)base;
  int32_t* pos = (int32_t*)(base + L.pos);
  int skip = -1, spin = 0;
  take_scan_test_hook(&skip, &spin);
  e = launch_scan(topk_ids, A, c.E, c.capacity, L.nblk_scan, (unsigned long long*)(base + L.desc),
                  pos, counts, offsets, hdr, skip, spin, c.drop_order, c.T, c.K, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_dispatch(c.dtype, x, topk_ids, pos, nullptr, 0, 1, offsets, c.T, c.d, c.E, c.K,
                      c.capacity, slot, src, x_perm, rows_capacity(c), hdr, sms, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_dispatch_noalloc_status(void* stream) {
  void* scratch = nullptr;
  int sms = 0;
  cudaError_t e = scratch_for_current_device(&scratch, &sms);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  uint32_t word = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word != 0) e = cudaMemset(scratch, 0, sizeof(word));
  if (e != cudaSuccess) {
    fprintf(stderr, "moe_dispatch_noalloc_status: %s\n", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (word & DEV_ERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (word & (DEV_ERR_BAD_ID | DEV_ERR_OVERFLOW | DEV_ERR_RANGE)) return MOE_ERR_DEVICE;
  return MOE_OK;
}
