// Shared device/host definitions of the attention kernels (sm_103a).
//
// The mask predicate here is the one every kernel applies; it follows the readings stated in
// include/fa.h: key j is valid for query i iff (!causal || j <= i) && j < L_b && the 128 x 128
// block (i/128, j/128) is kept by the block mask. Whole 128 x 128 tiles with no valid pair are
// skipped; only diagonal and tail tiles apply the element predicate.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

constexpr int kTile = 128;  // mask granularity and tile size (query rows x keys)

struct AttnShape {
  int B, H, N, d;
  int Hkv;     // K/V heads; query head h reads K/V head h / (H / Hkv) (grouped-query attention)
  int nb;      // ceil(N / 128)
  int causal;  // 0/1
  const uint8_t* block_mask;  // [nb * nb] or null
  const int32_t* seqlens_k;   // [B] or null
};

// Effective key length of sequence b: min(max(L_b, 0), N).
__device__ __forceinline__ int key_len(const AttnShape& s, int b) {
  int L = s.N;
  if (s.seqlens_k != nullptr) {
    L = __ldg(s.seqlens_k + b);
    L = L < 0 ? 0 : (L > s.N ? s.N : L);
  }
  return L;
}

// Is the (query tile qt, key tile kt) block visited? True iff it holds at least one valid pair.
__device__ __forceinline__ bool tile_visited(const AttnShape& s, int qt, int kt, int L) {
  if (s.causal && kt > qt) return false;
  if (kt * kTile >= L) return false;
  if (s.block_mask != nullptr && __ldg(s.block_mask + (size_t)qt * s.nb + kt) == 0) return false;
  return true;
}

// Record an in-kernel error (first writer wins); never traps.
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace fa

// Host-side launch entry points of the kernel translation units (called by fa_api.cu).
struct FaFwdArgs {
  const void *q, *k, *v;
  void* o;
  float* lse;
  fa::AttnShape s;
  float scale;
  int32_t* tile_visits;
  int* status;
};

struct FaBwdArgs {
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float* dvec;   // D, fp32 [B,H,N]
  float* dqacc;  // fp32 [B,H,N,d]
  fa::AttnShape s;
  float scale;
  int* status;
};

cudaError_t fa_launch_fwd(const FaFwdArgs& a, cudaStream_t st);
cudaError_t fa_launch_bwd(const FaBwdArgs& a, cudaStream_t st);
