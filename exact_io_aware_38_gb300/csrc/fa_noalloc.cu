// Backward pass for callers that cannot allocate device memory.
//
// fa_bwd needs a caller-supplied workspace (the fp32 row vector D and the fp32 dQ accumulator).
// Some callers have no way to provide one: a custom operator or plugin running inside another
// framework gets only its input and output buffers, and that framework owns the device memory
// pool, so a cudaMalloc of its own would bypass the host's memory accounting (or fail when the
// pool holds the whole device) and may synchronise the device in the middle of the host's
// stream work. fa_bwd_noalloc serves them: its workspace is a fixed array in the library's own
// device image, so the call allocates nothing.
//
// The array is a file-scope __device__ object of FA_NOALLOC_SCRATCH_BYTES bytes. Every GPU on
// which the library is loaded holds it until the process exits. Host code cannot use the
// array's name as a device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it with the context it belongs to;
// after a device reset the next call looks it up again in the new context. Make the first call on
// a device (and the first after a reset) before any stream capture. All calls share the one array and it keeps the previous call's contents;
// the backward kernels overwrite D and clear the dQ accumulator themselves on every call, so no
// extra clearing is needed. Two calls whose work overlaps on the GPU (e.g. on two streams) race
// on the array.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "fa_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_fa_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_fa_scratch per device ordinal
CUcontext g_scratch_ctx[kMaxDevices];  // the context that address belongs to

// The current context (through the driver entry point; null if it cannot be queried). A device
// reset gives the device a new primary context, in which the array has a new address.
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Same shape rules as fa_bwd, checked before any CUDA call.
int check_shape_noalloc(int B, int H, int N, int d, int causal, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((double)B * H * N * d >= 2147483648.0) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  const CUcontext ctx = current_context();
  if (g_scratch_addr[dev] == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = current_context();  // the runtime has made the primary context current by now
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                              const uint8_t* block_mask, const int32_t* seqlens_k, float scale, int* dev_status,
                              void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  const int rc = check_shape_noalloc(B, H, N, d, causal, scale);
  if (rc != FA_OK) return rc;
  if (fa_bwd_workspace_bytes(B, H, N, d) > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int s = scratch_address(&scratch);
  if (s != FA_OK) return s;
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, block_mask, seqlens_k, scale, scratch,
                (size_t)FA_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
