// Backward attention kernels on the warp-level tensor-core path (mma.sync m16n8k16).
//
// Three launches: (1) pre-pass D_i = sum_k dO_ik O_ik and a cleared fp32 dQ accumulator;
// (2) main pass, one CTA per 64-key block: it keeps K_j, V_j in shared memory, loops over the
// 64-row query blocks that can see them, recomputes S^T = K Q^T and P^T = exp(c S^T - LSE) (the
// scores are recomputed, never stored: "FlashAttention." plate, "Never write the scores"), forms
// dP^T = V dO^T and dS^T = P^T (dP^T - D), accumulates dV += P^T dO and dK += dS^T Q in registers
// and adds dQ += dS K into the accumulator with fp32 atomics; (3) post-pass dQ = bf16(c dQacc).
#include "mma_sync.cuh"

namespace fa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const FaBwdArgs a) {
  constexpr int PER = D / 32;  // elements per lane
  const size_t rows = (size_t)a.s.B * a.s.H * a.s.N;
  const int lane = threadIdx.x & 31;
  const size_t warp0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
  const __nv_bfloat16* O = reinterpret_cast<const __nv_bfloat16*>(a.o);
  const __nv_bfloat16* dO = reinterpret_cast<const __nv_bfloat16*>(a.dout);
  for (size_t r = warp0; r < rows; r += nwarps) {
    const size_t base = r * D + lane * PER;
    float acc = 0.f;
    if constexpr (PER == 2) {
      const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(O + base);
      const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(dO + base);
      acc = __bfloat162float(x.x) * __bfloat162float(y.x) + __bfloat162float(x.y) * __bfloat162float(y.y);
      *reinterpret_cast<float2*>(a.dqacc + base) = make_float2(0.f, 0.f);
    } else {
      const uint2 xs = *reinterpret_cast<const uint2*>(O + base);
      const uint2 ys = *reinterpret_cast<const uint2*>(dO + base);
      const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&xs);
      const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&ys);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        acc += __bfloat162float(x[i].x) * __bfloat162float(y[i].x) + __bfloat162float(x[i].y) * __bfloat162float(y[i].y);
      *reinterpret_cast<float4*>(a.dqacc + base) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) a.dvec[r] = acc;
  }
}

template <int D>
__global__ void __launch_bounds__(128, 1) bwd_mma_kernel(const FaBwdArgs a) {
  constexpr int BK = 64, BQ = 64, NT = 128, CH = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + BK * D * 2;
  const uint32_t sQ = sV + BK * D * 2;          // 2 stages
  const uint32_t sdO = sQ + 2 * BQ * D * 2;     // 2 stages
  const uint32_t sdS = sdO + 2 * BQ * D * 2;    // [BK][BQ] bf16, swizzled as D = 64
  float* sL = reinterpret_cast<float*>(smem + (sdS - sK) + BK * BQ * 2);  // 2 x BQ (LSE, natural log)
  float* sD = sL + 2 * BQ;                                                 // 2 x BQ

  const AttnShape& s = a.s;
  const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const size_t head = ((size_t)b * s.H + h) * (size_t)s.N;
  const __nv_bfloat16* Q = reinterpret_cast<const __nv_bfloat16*>(a.q) + head * D;
  const __nv_bfloat16* K = reinterpret_cast<const __nv_bfloat16*>(a.k) + head * D;
  const __nv_bfloat16* V = reinterpret_cast<const __nv_bfloat16*>(a.v) + head * D;
  const __nv_bfloat16* dO = reinterpret_cast<const __nv_bfloat16*>(a.dout) + head * D;
  const float* LSE = a.lse + head;
  const float* Dv = a.dvec + head;
  float* dQa = a.dqacc + head * D;
  const int L = key_len(s, b);
  const int k0 = kb * BK, kt = k0 / kTile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const float sl2 = a.scale * kLog2e;
  const int nqb = (s.N + BQ - 1) / BQ;

  auto q_ok = [&](int qb) -> bool {
    if (!tile_visited(s, qb * BQ / kTile, kt, L)) return false;
    if (s.causal && qb * BQ + BQ - 1 < k0) return false;
    return true;
  };
  auto next_qb = [&](int qb) -> int {
    if (k0 >= L) return -1;
    for (; qb < nqb; ++qb)
      if (q_ok(qb)) return qb;
    return -1;
  };
  auto load_q = [&](int qb, int st) {
    load_tile_async<D, NT>(sQ + st * BQ * D * 2, Q, qb * BQ, BQ, s.N, tid);
    load_tile_async<D, NT>(sdO + st * BQ * D * 2, dO, qb * BQ, BQ, s.N, tid);
    if (tid < 32) {
      const int half = tid >> 4, c = tid & 15;  // 16 x 16 B of LSE, then of D
      const int r = qb * BQ + c * 4;
      const bool ok = r < s.N;  // N is not a multiple of 4 only in ragged tails: handled below
      const float* src = half ? Dv : LSE;
      float* dst = (half ? sD : sL) + st * BQ + c * 4;
      if (ok && r + 4 <= s.N && ((reinterpret_cast<uintptr_t>(src + r) & 15) == 0)) {
        cp_async16(smem_u32(dst), src + r, true);
      } else {
        for (int u = 0; u < 4; ++u) dst[u] = (r + u < s.N) ? src[r + u] : 0.f;
      }
    }
  };

  float dv[D / 8][4], dk[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dv[i][e] = dk[i][e] = 0.f;

  int cur = next_qb(0);
  if (cur >= 0) {
    load_tile_async<D, NT>(sK, K, k0, BK, s.N, tid);
    load_tile_async<D, NT>(sV, V, k0, BK, s.N, tid);
    load_q(cur, 0);
  }
  cp_async_commit();
  int stage = 0;
  const int key0 = k0 + warp * 16 + g, key1 = key0 + 8;

  while (cur >= 0) {
    const int nxt = next_qb(cur + 1);
    if (nxt >= 0) load_q(nxt, stage ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int q0 = cur * BQ;
    const uint32_t sQs = sQ + stage * BQ * D * 2, sdOs = sdO + stage * BQ * D * 2;
    const float* sLs = sL + stage * BQ;
    const float* sDs = sD + stage * BQ;

    // S^T = K Q^T and dP^T = V dO^T for this warp's 16 keys x 64 queries.
    float st[8][4], dpt[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[i][e] = dpt[i][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t ka[4], va[4];
      ldsm_x4(sK + sw_off<D>(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), ka[0], ka[1], ka[2], ka[3]);
      ldsm_x4(sV + sw_off<D>(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), va[0], va[1], va[2], va[3]);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int rr = np * 16 + (lane & 7) + ((lane >> 4) << 3), cc = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sQs + sw_off<D>(rr, cc), b0, b1, b2, b3);
        mma16816(st[2 * np], ka, b0, b1);
        mma16816(st[2 * np + 1], ka, b2, b3);
        ldsm_x4(sdOs + sw_off<D>(rr, cc), b0, b1, b2, b3);
        mma16816(dpt[2 * np], va, b0, b1);
        mma16816(dpt[2 * np + 1], va, b2, b3);
      }
    }

    // P^T and dS^T (element mask: query in range, causal, key length).
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qc = nt * 8 + 2 * t + (e & 1);
        const int q = q0 + qc;
        const int key = (e < 2) ? key0 : key1;
        const bool ok = q < s.N && key < L && !(s.causal && key > q);
        const float p = ok ? ex2_approx(st[nt][e] * sl2 - sLs[qc] * kLog2e) : 0.f;
        st[nt][e] = p;
        dpt[nt][e] = p * (dpt[nt][e] - sDs[qc]);
      }
    }

    // dV += P^T dO, dK += dS^T Q (A from the accumulators, B via transposed ldmatrix).
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4], da[4];
      pa[0] = pack_bf16x2(st[2 * kk][0], st[2 * kk][1]);
      pa[1] = pack_bf16x2(st[2 * kk][2], st[2 * kk][3]);
      pa[2] = pack_bf16x2(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(st[2 * kk + 1][2], st[2 * kk + 1][3]);
      da[0] = pack_bf16x2(dpt[2 * kk][0], dpt[2 * kk][1]);
      da[1] = pack_bf16x2(dpt[2 * kk][2], dpt[2 * kk][3]);
      da[2] = pack_bf16x2(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
      da[3] = pack_bf16x2(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        const int rr = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), cc = np * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sdOs + sw_off<D>(rr, cc), b0, b1, b2, b3);
        mma16816(dv[2 * np], pa, b0, b1);
        mma16816(dv[2 * np + 1], pa, b2, b3);
        ldsm_x4_t(sQs + sw_off<D>(rr, cc), b0, b1, b2, b3);
        mma16816(dk[2 * np], da, b0, b1);
        mma16816(dk[2 * np + 1], da, b2, b3);
      }
      // dS^T (bf16) to shared memory for the dQ product.
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + sw_off<64>(warp * 16 + g, 2 * kk) + 4 * t), "r"(da[0]));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + sw_off<64>(warp * 16 + g + 8, 2 * kk) + 4 * t), "r"(da[1]));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + sw_off<64>(warp * 16 + g, 2 * kk + 1) + 4 * t), "r"(da[2]));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + sw_off<64>(warp * 16 + g + 8, 2 * kk + 1) + 4 * t), "r"(da[3]));
    }
    __syncthreads();

    // dQ (this warp's 16 queries x D) += dS K, in 64-wide halves, added with fp32 atomics.
    const int qr0 = q0 + warp * 16 + g, qr1 = qr0 + 8;
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) {
      float dq[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t aa[4];
        ldsm_x4_t(sdS + sw_off<64>(kk * 16 + (lane & 7) + ((lane >> 4) << 3), 2 * warp + ((lane >> 3) & 1)), aa[0], aa[1],
                  aa[2], aa[3]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sK + sw_off<D>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), hf * 8 + np * 2 + (lane >> 4)), b0, b1,
                    b2, b3);
          mma16816(dq[2 * np], aa, b0, b1);
          mma16816(dq[2 * np + 1], aa, b2, b3);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = hf * 64 + nt * 8 + 2 * t;
        if (qr0 < s.N) atomicAdd(reinterpret_cast<float2*>(dQa + (size_t)qr0 * D + col), make_float2(dq[nt][0], dq[nt][1]));
        if (qr1 < s.N) atomicAdd(reinterpret_cast<float2*>(dQa + (size_t)qr1 * D + col), make_float2(dq[nt][2], dq[nt][3]));
      }
    }
    __syncthreads();
    stage ^= 1;
    cur = nxt;
  }
  cp_async_wait<0>();
  __syncthreads();

  // Epilogue: dK = c * acc, dV = acc, bf16 through shared memory (the two Q stages).
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const uint32_t k0v = pack_bf16x2(dk[dt][0] * a.scale, dk[dt][1] * a.scale);
    const uint32_t k1v = pack_bf16x2(dk[dt][2] * a.scale, dk[dt][3] * a.scale);
    const uint32_t v0v = pack_bf16x2(dv[dt][0], dv[dt][1]);
    const uint32_t v1v = pack_bf16x2(dv[dt][2], dv[dt][3]);
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + sw_off<D>(warp * 16 + g, dt) + 4 * t), "r"(k0v));
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + sw_off<D>(warp * 16 + g + 8, dt) + 4 * t), "r"(k1v));
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + BQ * D * 2 + sw_off<D>(warp * 16 + g, dt) + 4 * t), "r"(v0v));
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + BQ * D * 2 + sw_off<D>(warp * 16 + g + 8, dt) + 4 * t), "r"(v1v));
  }
  __syncthreads();
  __nv_bfloat16* dK = reinterpret_cast<__nv_bfloat16*>(a.dk) + head * D;
  __nv_bfloat16* dV = reinterpret_cast<__nv_bfloat16*>(a.dv) + head * D;
  for (int idx = tid; idx < 2 * BK * CH; idx += NT) {
    const int which = idx / (BK * CH), rem = idx % (BK * CH);
    const int r = rem / CH, c = rem % CH;
    if (k0 + r < s.N) {
      uint4 val;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                   : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                   : "r"(sQ + which * BQ * D * 2 + sw_off<D>(r, c)));
      __nv_bfloat16* dst = (which ? dV : dK) + (size_t)(k0 + r) * D + c * 8;
      *reinterpret_cast<uint4*>(dst) = val;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256) bwd_post_kernel(const FaBwdArgs a) {
  const size_t n4 = (size_t)a.s.B * a.s.H * a.s.N * D / 4;
  __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(a.dq);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const float4 x = reinterpret_cast<const float4*>(a.dqacc)[i];
    uint2 out;
    out.x = pack_bf16x2(x.x * a.scale, x.y * a.scale);
    out.y = pack_bf16x2(x.z * a.scale, x.w * a.scale);
    reinterpret_cast<uint2*>(dq)[i] = out;
  }
}

template <int D>
cudaError_t launch(const FaBwdArgs& a, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid_ew = sms * 8;
  bwd_pre_kernel<D><<<grid_ew, 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int smem = (2 * 64 * D + 4 * 64 * D + 64 * 64) * 2 + 4 * 64 * 4;
  e = cudaFuncSetAttribute(bwd_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.s.N + 63) / 64, a.s.H, a.s.B);
  bwd_mma_kernel<D><<<grid, 128, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_post_kernel<D><<<grid_ew, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fa

cudaError_t fa_launch_bwd(const FaBwdArgs& a, cudaStream_t st) {
  return a.s.d == 64 ? fa::launch<64>(a, st) : fa::launch<128>(a, st);
}
