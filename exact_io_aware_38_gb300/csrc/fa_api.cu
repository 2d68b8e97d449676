// C ABI of the attention library: argument validation, workspace layout and kernel launches.
// Every check runs on the host before any CUDA call, so invalid arguments never reach a GPU.
#include <math.h>

#include "fa_common.cuh"

namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int B, int H, int N, int d, int causal, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const double elems = (double)B * H * N * d;
  if (elems >= 2147483648.0) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// K/V heads: each must serve the same number of query heads.
inline bool check_kv_heads(int H, int Hkv) { return Hkv >= 1 && Hkv <= H && H % Hkv == 0; }

fa::AttnShape make_shape(int B, int H, int Hkv, int N, int d, int causal, const uint8_t* bm, const int32_t* sl) {
  fa::AttnShape s;
  s.B = B;
  s.H = H;
  s.Hkv = Hkv;
  s.N = N;
  s.d = d;
  s.nb = (N + fa::kTile - 1) / fa::kTile;
  s.causal = causal;
  s.block_mask = bm;
  s.seqlens_k = sl;
  return s;
}

}  // namespace

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument (null pointer, size, flag or scale)";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dimension or tensor size";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: tensor pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA call or kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a bounded in-kernel wait ran out";
    case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS: an in-kernel index check failed";
    case FA_ERR_SCRATCH_LIMIT: return "FA_ERR_SCRATCH_LIMIT: problem exceeds the fixed scratch of fa_bwd_noalloc";
    default: return "unknown fa status";
  }
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N, int d,
               int causal, const uint8_t* block_mask, const int32_t* seqlens_k, float scale, int32_t* tile_visits,
               int* dev_status, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  const int rc = check_shape(B, H, N, d, causal, scale);
  if (rc != FA_OK) return rc;
  if (!check_kv_heads(H, Hkv)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(seqlens_k, 4) || !aligned(tile_visits, 4) || !aligned(dev_status, 4))
    return FA_ERR_MISALIGNED;
  FaFwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.s = make_shape(B, H, Hkv, N, d, causal, block_mask, seqlens_k);
  a.scale = scale;
  a.tile_visits = tile_visits;
  a.status = dev_status;
  const cudaError_t e = fa_launch_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d, int causal,
           const uint8_t* block_mask, const int32_t* seqlens_k, float scale, int32_t* tile_visits, int* dev_status,
           void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, block_mask, seqlens_k, scale, tile_visits, dev_status,
                    stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d, 0, 1.f) != FA_OK) return 0;
  const size_t rows = (size_t)B * H * N;
  return round_up(rows * sizeof(float)) + round_up(rows * d * sizeof(float));
}

int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
               void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, int causal,
               const uint8_t* block_mask, const int32_t* seqlens_k, float scale, void* workspace,
               size_t workspace_bytes, int* dev_status, void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  const int rc = check_shape(B, H, N, d, causal, scale);
  if (rc != FA_OK) return rc;
  if (!check_kv_heads(H, Hkv)) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(workspace, kAlign) ||
      !aligned(seqlens_k, 4) || !aligned(dev_status, 4))
    return FA_ERR_MISALIGNED;
  const size_t rows = (size_t)B * H * N;
  FaBwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dvec = static_cast<float*>(workspace);
  a.dqacc = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(rows * sizeof(float)));
  a.s = make_shape(B, H, Hkv, N, d, causal, block_mask, seqlens_k);
  a.scale = scale;
  a.status = dev_status;
  const cudaError_t e = fa_launch_bwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int N, int d, int causal, const uint8_t* block_mask,
           const int32_t* seqlens_k, float scale, void* workspace, size_t workspace_bytes, int* dev_status,
           void* stream) {
  return fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, H, N, d, causal, block_mask, seqlens_k, scale, workspace,
                    workspace_bytes, dev_status, stream);
}

}  // extern "C"
