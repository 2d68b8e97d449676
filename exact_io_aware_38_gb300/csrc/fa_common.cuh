// Shared device/host definitions of the attention kernels (sm_103a).
//
// The mask predicate here is the one every kernel applies; it follows the readings stated in
// include/fa.h. Sequence b has L_q query rows and L_k keys (fixed-length batches: L_q = N_q and
// L_k = N_k, or the key length of seqlens_k; packed batches: from cu_seqlens). Key j is valid for
// query i iff j < L_k, (!causal || j <= i + L_k - L_q) (causal aligned to the bottom-right corner;
// the square case is j <= i) and the 128 x 128 block (i/128, j/128) is kept by the block mask.
// Whole 128 x 128 tiles with no valid pair are skipped; only tiles that straddle the diagonal or
// the key end apply the element predicate.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

constexpr int kTile = 128;  // mask granularity and tile size (query rows x keys)

struct AttnShape {
  int B, H, d;
  int Hkv;     // K/V heads; query head h reads K/V head h / (H / Hkv) (grouped-query attention)
  int Nq, Nk;  // fixed length: the lengths; packed: the maximum lengths (the grid covers these)
  int nbq, nbk;  // ceil(Nq / 128), ceil(Nk / 128)
  int causal;    // 0/1, bottom-right aligned
  const uint8_t* block_mask;  // [nbq * nbk] or null (fixed length only)
  const int32_t* seqlens_k;   // [B] or null (fixed length only)
  const int32_t* cu_q;        // [B + 1] or null: packed query rows of sequence b are cu_q[b] .. cu_q[b+1]
  const int32_t* cu_k;        // [B + 1], set exactly when cu_q is
  int rows_q, rows_k;         // packed: rows of the packed Q/O/dO/dQ and K/V/dK/dV tensors
};

// One sequence of the batch, resolved once per CTA.
struct SeqInfo {
  int Lq, Lk;  // query rows and valid keys
  int q0, k0;  // first row of the sequence in the tensor's row dimension (packed), else 0
  int bb;      // batch coordinate of the tensor maps (fixed length), else 0
  int off;     // causal offset (keys - queries of the sequence): key j visible to query i iff j <= i + off
  int krows;   // key rows that exist in the tensor for this sequence (dK/dV rows to write)
};

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

__device__ __forceinline__ SeqInfo seq_info(const AttnShape& s, int b) {
  SeqInfo r;
  if (s.cu_q != nullptr) {
    // Lengths are clamped to the maxima the grid covers and rows to the tensors' extents, so a
    // malformed cu_seqlens can never index outside the buffers.
    r.q0 = clampi(__ldg(s.cu_q + b), 0, s.rows_q);
    r.k0 = clampi(__ldg(s.cu_k + b), 0, s.rows_k);
    r.Lq = clampi(__ldg(s.cu_q + b + 1) - r.q0, 0, min(s.Nq, s.rows_q - r.q0));
    r.Lk = clampi(__ldg(s.cu_k + b + 1) - r.k0, 0, min(s.Nk, s.rows_k - r.k0));
    r.bb = 0;
    r.krows = r.Lk;
  } else {
    r.q0 = r.k0 = 0;
    r.Lq = s.Nq;
    r.Lk = s.Nk;
    if (s.seqlens_k != nullptr) r.Lk = clampi(__ldg(s.seqlens_k + b), 0, s.Nk);
    r.bb = b;
    r.krows = s.Nk;
  }
  // Causal alignment uses the sequence's key count; key padding (seqlens_k) is a separate mask.
  r.off = (s.cu_q != nullptr ? r.Lk : s.Nk) - r.Lq;
  return r;
}

// Is the (query tile qt, key tile kt) block visited? True iff it holds at least one valid pair.
__device__ __forceinline__ bool tile_visited(const AttnShape& s, const SeqInfo& q, int qt, int kt) {
  if (qt * kTile >= q.Lq || kt * kTile >= q.Lk) return false;
  if (s.causal && kt * kTile > qt * kTile + (kTile - 1) + q.off) return false;
  if (s.block_mask != nullptr && __ldg(s.block_mask + (size_t)qt * s.nbk + kt) == 0) return false;
  return true;
}

// First index of (b, h)'s rows in the per-row arrays (LSE, and the backward's D and fp32 dQ
// accumulator): fixed length [B][H][Nq]; packed [H][rows_q] (a sequence's rows are contiguous).
__device__ __forceinline__ size_t row_base(const AttnShape& s, const SeqInfo& q, int b, int h) {
  return s.cu_q != nullptr ? (size_t)h * s.rows_q + q.q0 : ((size_t)b * s.H + h) * s.Nq;
}

// Per-row arrays (D, the fp32 dQ accumulator, split partials) use the LSE's row order: fixed length
// [B][H][Nq], packed [H][rows_q]. Row R of that order sits at these coordinates of the
// [batch][row][head][d] tensors.
__device__ __forceinline__ void row_coords(const AttnShape& s, size_t R, int& b, int& row, int& h) {
  if (s.cu_q != nullptr) {
    b = 0;
    h = (int)(R / s.rows_q);
    row = (int)(R % s.rows_q);
  } else {
    b = (int)(R / ((size_t)s.H * s.Nq));
    const size_t rem = R % ((size_t)s.H * s.Nq);
    h = (int)(rem / s.Nq);
    row = (int)(rem % s.Nq);
  }
}

__host__ __device__ inline size_t per_row_count(const AttnShape& s) {
  return s.cu_q != nullptr ? (size_t)s.H * s.rows_q : (size_t)s.B * s.H * s.Nq;
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

// Element strides of a bf16 tensor addressed as [batch][row][head][d] (d contiguous).
struct FaStrides {
  long long row, head, batch;
};

__device__ __forceinline__ size_t elem_offset(const FaStrides& t, int b, int row, int h) {
  return (size_t)b * t.batch + (size_t)row * t.row + (size_t)h * t.head;
}

// Host-side launch entry points of the kernel translation units (called by fa_api.cu).
struct FaFwdArgs {
  const void *q, *k, *v;
  void* o;
  float* lse;
  FaStrides sq, sk, sv, so;
  fa::AttnShape s;
  float scale;
  int32_t* tile_visits;
  int* status;
  // Split over keys: CTA split s covers key tiles [s * kt_chunk, (s + 1) * kt_chunk) and, when
  // part_o is set, writes its normalised fp32 partial O [split][row][d] and LSE [split][row]
  // (rows in the LSE order, part_rows per split) for the merge pass instead of O and LSE.
  int splits, kt_chunk;
  float *part_o, *part_lse;
  size_t part_rows;
  // e4m3 operands (fp8 != 0): q, k are [B][H or Hkv][N][d] bytes, v is V^T [B][Hkv][d][N] bytes, and
  // the true inputs are q_descale[b * H + h] * q (k, v likewise with [b * Hkv + hk]).
  int fp8;
  const float *q_descale, *k_descale, *v_descale;
};

struct FaBwdArgs {
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  FaStrides sq, sk, sv, so, sdo, sdq, sdk, sdv;
  float* dvec;   // D, fp32, one per query row (laid out like the LSE)
  float* dqacc;  // fp32 dQ accumulator, d per query row (laid out like the LSE)
  int* tile_counter;  // key tiles handed out so far by the persistent main kernel (workspace)
  fa::AttnShape s;
  float scale;
  int* status;
  // Accumulate mode (all three set): fp32 dQ, dK, dV shares are added into these caller tensors
  // (element strides sdq, sdk, sdv) instead of writing bf16 dq, dk, dv.
  float *dq_acc, *dk_acc, *dv_acc;
  int32_t* step_visits;       // nullable: query steps visited per (b, K/V head, key tile)
  cudaEvent_t ev_main_begin;  // nullable (host side): recorded around the main launch
  cudaEvent_t ev_main_end;
};

cudaError_t fa_launch_fwd(const FaFwdArgs& a, cudaStream_t st);
// A launch that may begin while the previous kernel on the stream finishes: the kernel waits on
// the grid dependency (griddepcontrol.wait) before its first global-memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
cudaError_t fa_launch_splitkv_merge(const FaFwdArgs& a, cudaStream_t st);
cudaError_t fa_launch_merge_two(float* acc_o, float* acc_lse, const float* part_o, const float* part_lse, size_t rows,
                                int d, cudaStream_t st);
cudaError_t fa_launch_bwd(const FaBwdArgs& a, cudaStream_t st);
