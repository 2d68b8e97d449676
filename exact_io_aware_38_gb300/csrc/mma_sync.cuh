// Warp-level tensor-core helpers (mma.sync m16n8k16 bf16, ldmatrix, cp.async) and the
// 128-byte XOR swizzle used for shared-memory tiles of row-major [rows][D] bf16 data.
#pragma once

#include "fa_common.cuh"

namespace fa {

// Byte offset of 16-byte chunk c of row r in a [rows][D] bf16 tile: chunk index XOR (r % 8),
// which makes 8 consecutive rows at the same logical chunk land in 8 distinct bank groups.
template <int D>
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int n>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(n) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// c[4] += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Copy `rows` rows of a [*, D] bf16 matrix starting at global row g0 into a swizzled smem tile;
// rows at or beyond `nvalid` are zero-filled (no global read).
template <int D, int NT>
__device__ __forceinline__ void load_tile_async(uint32_t s_base, const __nv_bfloat16* g, int g0, int rows, int nvalid,
                                                int tid) {
  constexpr int CH = D / 8;
  for (int idx = tid; idx < rows * CH; idx += NT) {
    const int r = idx / CH, c = idx % CH;
    const bool ok = g0 + r < nvalid;
    const __nv_bfloat16* src = g + (size_t)(ok ? g0 + r : 0) * D + c * 8;
    cp_async16(s_base + sw_off<D>(r, c), src, ok);
  }
}

}  // namespace fa
