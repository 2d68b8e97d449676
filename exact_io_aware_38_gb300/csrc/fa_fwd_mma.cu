// Forward attention kernel on the warp-level tensor-core path (mma.sync m16n8k16).
//
// One CTA per (128-row query tile, head, batch); 8 warps, each owning 16 query rows. Key/value
// tiles of 64 rows stream through a 2-stage cp.async ring; scores stay in registers; the online
// softmax keeps a running row max and sum per row and rescales the partial output
// ("FlashAttention." plate, intro; "Flash Attention: IO-Aware Attention Computation", para. 4);
// row statistics are reduced across the 4 lanes sharing a row with warp shuffles.
#include "mma_sync.cuh"

namespace fa {
namespace {

template <int D>
__global__ void __launch_bounds__(256, 1) fwd_mma_kernel(const FaFwdArgs a) {
  constexpr int BM = 128, BN = 64, NT = 256, CH = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + BM * D * 2;
  const uint32_t sV = sK + 2 * BN * D * 2;

  const AttnShape& s = a.s;
  const int qt = s.causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;  // longest first
  const int h = blockIdx.y, b = blockIdx.z;
  const size_t head = ((size_t)b * s.H + h) * (size_t)s.N;
  const __nv_bfloat16* Q = reinterpret_cast<const __nv_bfloat16*>(a.q) + head * D;
  const __nv_bfloat16* K = reinterpret_cast<const __nv_bfloat16*>(a.k) + head * D;
  const __nv_bfloat16* V = reinterpret_cast<const __nv_bfloat16*>(a.v) + head * D;
  const int L = key_len(s, b);
  const int q0 = qt * BM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const float sl2 = a.scale * kLog2e;

  // Steps are (key tile, half) pairs e = 2*kt + half over visited tiles, halves starting below L.
  auto next_step = [&](int e) -> int {
    for (; e < 2 * s.nb; ++e) {
      const int kt = e >> 1;
      if (!tile_visited(s, qt, kt, L)) {
        e |= 1;
        continue;
      }
      if (kt * kTile + (e & 1) * BN < L) return e;
    }
    return -1;
  };

  load_tile_async<D, NT>(sQ, Q, q0, BM, s.N, tid);
  int cur = next_step(0);
  if (cur >= 0) {
    const int k0 = (cur >> 1) * kTile + (cur & 1) * BN;
    load_tile_async<D, NT>(sK, K, k0, BN, s.N, tid);
    load_tile_async<D, NT>(sV, V, k0, BN, s.N, tid);
  }
  cp_async_commit();

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  uint32_t qf[D / 16][4];
  bool have_q = false;
  int stage = 0;
  const int row0 = q0 + warp * 16 + g, row1 = row0 + 8;

  while (cur >= 0) {
    const int nxt = next_step(cur + 1);
    if (nxt >= 0) {
      const int k1 = (nxt >> 1) * kTile + (nxt & 1) * BN;
      load_tile_async<D, NT>(sK + (stage ^ 1) * BN * D * 2, K, k1, BN, s.N, tid);
      load_tile_async<D, NT>(sV + (stage ^ 1) * BN * D * 2, V, k1, BN, s.N, tid);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (!have_q) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(sQ + sw_off<D>(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), qf[kk][0], qf[kk][1], qf[kk][2],
                qf[kk][3]);
      have_q = true;
    }
    const int k0 = (cur >> 1) * kTile + (cur & 1) * BN;
    const uint32_t sKs = sK + stage * BN * D * 2, sVs = sV + stage * BN * D * 2;

    // S = Q K^T for this warp's 16 rows x 64 keys.
    float sc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sKs + sw_off<D>(np * 16 + (lane & 7) + ((lane >> 4) << 3), kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma16816(sc[2 * np], qf[kk], b0, b1);
        mma16816(sc[2 * np + 1], qf[kk], b2, b3);
      }
    }

    // Scale into the log2 domain and apply the element mask on diagonal / tail steps.
    const bool need_mask = (s.causal && k0 + BN - 1 > q0) || (k0 + BN > L);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = sc[nt][e] * sl2;
        if (need_mask) {
          const int key = k0 + nt * 8 + 2 * t + (e & 1);
          const int row = (e < 2) ? row0 : row1;
          if ((s.causal && key > row) || key >= L) x = -INFINITY;
        }
        sc[nt][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    }
    float alpha[2], muse[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(m[r], mx[r]);
      muse[r] = (mn == -INFINITY) ? 0.f : mn;
      alpha[r] = ex2_approx(m[r] - muse[r]);
      m[r] = mn;
    }
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = ex2_approx(sc[nt][e] - muse[e >> 1]);
        sc[nt][e] = p;
        ls[e >> 1] += p;
      }
    }
    l[0] = l[0] * alpha[0] + ls[0];
    l[1] = l[1] * alpha[1] + ls[1];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }

    // O += P V: P fragments come straight from the score accumulators.
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
      pa[1] = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
      pa[2] = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sVs + sw_off<D>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), np * 2 + (lane >> 4)), b0, b1, b2, b3);
        mma16816(o[2 * np], pa, b0, b1);
        mma16816(o[2 * np + 1], pa, b2, b3);
      }
    }
    __syncthreads();
    stage ^= 1;
    cur = nxt;
  }
  cp_async_wait<0>();
  __syncthreads();

  // Epilogue: O / l in bf16 through shared memory (Q's tile), LSE = (m + log2 l) ln 2.
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  const float inv0 = l[0] > 0.f ? 1.f / l[0] : 0.f, inv1 = l[1] > 0.f ? 1.f / l[1] : 0.f;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const uint32_t v0 = pack_bf16x2(o[dt][0] * inv0, o[dt][1] * inv0);
    const uint32_t v1 = pack_bf16x2(o[dt][2] * inv1, o[dt][3] * inv1);
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + sw_off<D>(warp * 16 + g, dt) + 4 * t), "r"(v0));
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + sw_off<D>(warp * 16 + g + 8, dt) + 4 * t), "r"(v1));
  }
  if (t == 0) {
    if (row0 < s.N) a.lse[head + row0] = l[0] > 0.f ? (m[0] + log2f(l[0])) * kLn2 : -INFINITY;
    if (row1 < s.N) a.lse[head + row1] = l[1] > 0.f ? (m[1] + log2f(l[1])) * kLn2 : -INFINITY;
  }
  __syncthreads();
  __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(a.o) + head * D;
  for (int idx = tid; idx < BM * CH; idx += NT) {
    const int r = idx / CH, c = idx % CH;
    if (q0 + r < s.N) {
      uint4 val;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                   : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                   : "r"(sQ + sw_off<D>(r, c)));
      *reinterpret_cast<uint4*>(O + (size_t)(q0 + r) * D + c * 8) = val;
    }
  }
  if (a.tile_visits != nullptr && tid == 0) {
    int cnt = 0;
    for (int kt = 0; kt < s.nb; ++kt) cnt += tile_visited(s, qt, kt, L) ? 1 : 0;
    a.tile_visits[((size_t)b * s.H + h) * s.nb + qt] = cnt;
  }
}

template <int D>
cudaError_t launch(const FaFwdArgs& a, cudaStream_t st) {
  constexpr int smem = (128 + 4 * 64) * D * 2;
  cudaError_t e = cudaFuncSetAttribute(fwd_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.s.nb, a.s.H, a.s.B);
  fwd_mma_kernel<D><<<grid, 256, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fa

cudaError_t fa_launch_fwd(const FaFwdArgs& a, cudaStream_t st) {
  return a.s.d == 64 ? fa::launch<64>(a, st) : fa::launch<128>(a, st);
}
