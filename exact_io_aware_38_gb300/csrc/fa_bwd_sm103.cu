// Backward attention on the 5th-generation tensor cores (sm_103a).
//
// Three launches on the caller's stream:
//   pre   D_i = sum_k dO_ik O_ik (fp32, from the stored bf16 O) and a cleared fp32 dQ accumulator;
//   main  one CTA per (128-key tile j, head): K_j and V_j stay in shared memory while the 128-row
//         query tiles i that can see them stream through a TMA ring. The score tile is recomputed
//         from Q, K and the saved log-sum-exp instead of being stored ("FlashAttention." plate,
//         "Never write the scores"), and the softmax gradient is applied tile by tile:
//           S^T = K_j Q_i^T,  dP^T = V_j dO_i^T                  (tcgen05, into tensor memory)
//           P^T = exp(c S^T - LSE_i),  dS^T = P^T * (dP^T - D_i)  (one thread per key row)
//           dV_j += P^T dO_i,  dK_j += dS^T Q_i                  (A operand from tensor memory)
//           dQ_i += dS K_j                                       (fp32 atomics into the accumulator)
//         dK_j = c * acc and dV_j leave through shared memory and TMA stores.
//   post  dQ = bf16(c * accumulator).
// For d = 128 the dQ product is formed transposed, dQ_i^T = K_j^T dS_i^T, so the tensor-memory
// lane is the head dimension and each warp's atomics cover 128 contiguous bytes of one dQ row.
// For d = 64 it is formed as dS_i K_j (lane = query row), with 16-byte vector atomics.
//
// CTA layout (256 threads): warp 0 TMA producer, warp 1 MMA issuer and tensor-memory owner,
// warps 4-7 the elementwise warpgroup (thread = key row of the tile; lane quadrant = warp % 4).
// Tensor memory: d = 128: dK [0,128) dV [128,256) S^T and dQ^T [256,384) dP^T [384,512);
//                d = 64:  dK [0,64) dV [64,128) S^T [128,256) dP^T [256,384) dQ [384,448).
// P^T and dS^T (bf16) are written over the first 64 columns of S^T and dP^T.
#include "fa_tmap.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace tc;

constexpr int kBwdThreads = 256;

template <int D>
struct BwdCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kStages = D == 128 ? 2 : 3;
  static constexpr int kDsBytes = 128 * 128 * 2;
  static constexpr int kSmem = (2 + 2 * kStages) * kTileBytes + kDsBytes + 1024;
  static constexpr uint32_t kTdK = 0, kTdV = D, kTS = 2 * D, kTdP = 2 * D + 128;
  static constexpr uint32_t kTdQ = D == 128 ? kTS : 2 * D + 256;
  static constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t kIdG = idesc_bf16(128, D, false, true);
  static constexpr uint32_t kIdQ = D == 128 ? idesc_bf16(128, 128, true, true) : idesc_bf16(128, D, true, true);
};

struct BwdSmemCtl {
  uint64_t kv_full;
  uint64_t full[3];
  uint64_t empty[3];
  uint64_t s_full, p_ready, dq_full, dq_free, done, drain;
  uint32_t tmem_base;
  int abort_flag;
  float lse2[128];  // LSE * log2(e) of the current query tile
  float dvec[128];  // D of the current query tile
};

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const FaBwdArgs a) {
  constexpr int PER = D / 32;
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
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                  const FaBwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + C::kTileBytes;
  const uint32_t sStage0 = sV + C::kTileBytes;  // stage s: Q at +2s tiles, dO at +2s+1 tiles
  const uint32_t sDs = sK + (2 + 2 * C::kStages) * C::kTileBytes;
  volatile int* abort_flag = &ctl.abort_flag;

  const AttnShape& s = a.s;
  const int BH = s.B * s.H;
  const int kt = blockIdx.x / BH;  // key tile: small kt (most causal work) first
  const int bh = blockIdx.x % BH;
  const int b = bh / s.H;
  const int L = key_len(s, b);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  auto next_q = [&](int qt) -> int {
    for (; qt < s.nb; ++qt)
      if (tile_visited(s, qt, kt, L)) return qt;
    return s.nb;
  };
  auto sQs = [&](int st) { return sStage0 + (2 * st) * C::kTileBytes; };
  auto sdOs = [&](int st) { return sStage0 + (2 * st + 1) * C::kTileBytes; };

  const uint32_t b_kv = smem_u32(&ctl.kv_full);
  auto b_full = [&](int i) { return smem_u32(&ctl.full[i]); };
  auto b_empty = [&](int i) { return smem_u32(&ctl.empty[i]); };
  const uint32_t b_sfull = smem_u32(&ctl.s_full), b_pready = smem_u32(&ctl.p_ready);
  const uint32_t b_dqfull = smem_u32(&ctl.dq_full), b_dqfree = smem_u32(&ctl.dq_free);
  const uint32_t b_done = smem_u32(&ctl.done), b_drain = smem_u32(&ctl.drain);

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(b_kv, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(b_full(i), 1);
      mbar_init(b_empty(i), 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_pready, 128);
    mbar_init(b_dqfull, 1);
    mbar_init(b_dqfree, 128);
    mbar_init(b_done, 1);
    mbar_init(b_drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;
  const bool any_work = next_q(0) < s.nb;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && any_work) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmdO);
      mbar_expect_tx(b_kv, 2 * C::kTileBytes);
      for (int c = 0; c < C::kBoxes; ++c) {
        tma_load_3d(sK + c * 16384, &tmK, c * 64, kt * 128, bh, b_kv);
        tma_load_3d(sV + c * 16384, &tmV, c * 64, kt * 128, bh, b_kv);
      }
      int st = 0;
      uint32_t ph = 0;
      uint32_t last_par[3];
      bool issued[3] = {false, false, false};
      for (int qt = next_q(0); qt < s.nb; qt = next_q(qt + 1)) {
        if (mbar_wait(b_empty(st), ph ^ 1, abort_flag, a.status)) {
          mbar_expect_tx(b_full(st), 2 * C::kTileBytes);
          for (int c = 0; c < C::kBoxes; ++c) {
            tma_load_3d(sQs(st) + c * 16384, &tmQ, c * 64, qt * 128, bh, b_full(st));
            tma_load_3d(sdOs(st) + c * 16384, &tmdO, c * 64, qt * 128, bh, b_full(st));
          }
          issued[st] = true;
          last_par[st] = ph;
        }
        if (++st == C::kStages) {
          st = 0;
          ph ^= 1;
        }
      }
      if (*abort_flag) {
        mbar_wait_drain(b_kv, 0);
        for (int i = 0; i < C::kStages; ++i)
          if (issued[i]) mbar_wait_drain(b_full(i), last_par[i]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      if (any_work) {
        mbar_wait(b_kv, 0, abort_flag, a.status);
        int st = 0;
        uint32_t ph = 0;
        uint32_t it = 0;
        for (int qt = next_q(0); qt < s.nb; qt = next_q(qt + 1), ++it) {
          mbar_wait(b_full(st), ph, abort_flag, a.status);
          if (it > 0) mbar_wait(b_dqfree, (it - 1) & 1, abort_flag, a.status);
          fence_after_sync();
          const uint32_t q_s = sQs(st), do_s = sdOs(st);
          if (!*abort_flag) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_ss(tmem + C::kTS, desc_kmajor_sw128(sK + off), desc_kmajor_sw128(q_s + off), C::kIdS, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_ss(tmem + C::kTdP, desc_kmajor_sw128(sV + off), desc_kmajor_sw128(do_s + off), C::kIdS, kk > 0);
            }
            mma_commit(b_sfull);
          }
          mbar_wait(b_pready, it & 1, abort_flag, a.status);
          fence_after_sync();
          if (!*abort_flag) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kTdV, tmem + C::kTS + kk * 8, desc_mnmajor_sw128(do_s + kk * 2048, 16384), C::kIdG,
                     (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kTdK, tmem + C::kTdP + kk * 8, desc_mnmajor_sw128(q_s + kk * 2048, 16384), C::kIdG,
                     (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              if constexpr (D == 128) {
                mma_ss(tmem + C::kTdQ, desc_mnmajor_sw128(sK + kk * 2048, 16384),
                       desc_mnmajor_sw128(sDs + kk * 2048, 16384), C::kIdQ, kk > 0);
              } else {
                mma_ss(tmem + C::kTdQ, desc_mnmajor_sw128(sDs + kk * 2048, 16384),
                       desc_mnmajor_sw128(sK + kk * 2048, 16384), C::kIdQ, kk > 0);
              }
            }
            mma_commit(b_dqfull);
            mma_commit(b_empty(st));
          }
          if (++st == C::kStages) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!*abort_flag) mma_commit(b_done);
      }
      mma_commit(b_drain);
      mbar_wait_drain(b_drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ elementwise warpgroup
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // key row of the tile (and head-dimension lane of dQ^T)
    const int key = kt * 128 + r;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kTS, tdP = tmem + lane_off + C::kTdP;
    const uint32_t tdQ = tmem + lane_off + C::kTdQ;
    const float sl2 = a.scale * kLog2e;
    const float* LSE = a.lse + (size_t)bh * s.N;
    const float* Dv = a.dvec + (size_t)bh * s.N;
    float* dQa = a.dqacc + (size_t)bh * s.N * D;
    const bool key_ok = key < L;
    uint32_t it = 0;
    for (int qt = next_q(0); qt < s.nb; qt = next_q(qt + 1), ++it) {
      const int q0 = qt * 128;
      named_bar_sync(1, 128);  // every thread is done with the previous tile's LSE and D
      {
        const int q = q0 + r;
        ctl.lse2[r] = q < s.N ? LSE[q] * kLog2e : 0.f;
        ctl.dvec[r] = q < s.N ? Dv[q] : 0.f;
      }
      named_bar_sync(1, 128);
      mbar_wait(b_sfull, it & 1, abort_flag, a.status);
      fence_after_sync();
      const bool need_mask = (s.causal && qt == kt) || (kt * 128 + 128 > L) || (q0 + 128 > s.N);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tS + c * 32, sr);
        tmem_ld32(tdP + c * 32, dr);
        tmem_ld_wait();
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          float pp[2], dd[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qq = c * 32 + t + u;
            float p = ex2_approx(fmaf(__uint_as_float(sr[t + u]), sl2, -ctl.lse2[qq]));
            if (need_mask) {
              const int q = q0 + qq;
              const bool ok = key_ok && q < s.N && !(s.causal && key > q);
              p = ok ? p : 0.f;
            }
            pp[u] = p;
            dd[u] = p * (__uint_as_float(dr[t + u]) - ctl.dvec[qq]);
          }
          pk[t >> 1] = pack_bf16x2(pp[0], pp[1]);
          dk[t >> 1] = pack_bf16x2(dd[0], dd[1]);
        }
        tmem_st16(tS + c * 16, pk);
        tmem_st16(tdP + c * 16, dk);
        const uint32_t box = sDs + (c >> 1) * 16384 + r * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int chunk = (c & 1) * 4 + j;
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(box + ((chunk ^ (r & 7)) << 4)), "r"(dk[4 * j]),
                       "r"(dk[4 * j + 1]), "r"(dk[4 * j + 2]), "r"(dk[4 * j + 3])
                       : "memory");
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      fence_before_sync();
      mbar_arrive(b_pready);

      mbar_wait(b_dqfull, it & 1, abort_flag, a.status);
      fence_after_sync();
      if constexpr (D == 128) {
        // dQ^T: this thread holds head-dimension r of dQ for the tile's 128 queries.
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tdQ + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const int q = q0 + c * 32 + t;
            if (q < s.N) atomicAdd(dQa + (size_t)q * D + r, __uint_as_float(v[t]));
          }
        }
      } else {
        // dQ: this thread holds query row r of the tile.
        const int q = q0 + r;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tdQ + c * 32, v);
          tmem_ld_wait();
          if (q < s.N) {
#pragma unroll
            for (int t = 0; t < 32; t += 4)
              atomicAdd(reinterpret_cast<float4*>(dQa + (size_t)q * D + c * 32 + t),
                        make_float4(__uint_as_float(v[t]), __uint_as_float(v[t + 1]), __uint_as_float(v[t + 2]),
                                    __uint_as_float(v[t + 3])));
          }
        }
      }
      fence_before_sync();
      mbar_arrive(b_dqfree);
    }

    // ---------------------------------------------------------------- epilogue: dK, dV
    if (it > 0) {
      mbar_wait(b_done, 0, abort_flag, a.status);
      fence_after_sync();
    }
    const uint32_t stgK = sStage0, stgV = sStage0 + C::kTileBytes;  // stage 0 Q / dO buffers
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t tacc = tmem + lane_off + (which ? C::kTdV : C::kTdK);
      const float mul = which ? 1.f : a.scale;
      const uint32_t stg = which ? stgV : stgK;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        if (it > 0) {
          tmem_ld32(tacc + c * 32, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
        const uint32_t box = stg + (c >> 1) * 16384 + r * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int chunk = (c & 1) * 4 + j;
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(box + ((chunk ^ (r & 7)) << 4)), "r"(pk[4 * j]),
                       "r"(pk[4 * j + 1]), "r"(pk[4 * j + 2]), "r"(pk[4 * j + 3])
                       : "memory");
        }
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (warp == 4 && lane == 0) {
      for (int c = 0; c < C::kBoxes; ++c) {
        tma_store_3d(&tmdK, stgK + c * 16384, c * 64, kt * 128, bh);
        tma_store_3d(&tmdV, stgV + c * 16384, c * 64, kt * 128, bh);
      }
      tma_store_commit();
      tma_store_wait0();
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch(const FaBwdArgs& a, cudaStream_t st) {
  using C = BwdCfg<D>;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid_ew = sms * 8;
  const int BH = a.s.B * a.s.H;
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  if (!fa_make_tmap_bf16(&tq, a.q, a.s.N, D, BH) || !fa_make_tmap_bf16(&tk, a.k, a.s.N, D, BH) ||
      !fa_make_tmap_bf16(&tv, a.v, a.s.N, D, BH) || !fa_make_tmap_bf16(&tdo, a.dout, a.s.N, D, BH) ||
      !fa_make_tmap_bf16(&tdk, a.dk, a.s.N, D, BH) || !fa_make_tmap_bf16(&tdv, a.dv, a.s.N, D, BH))
    return cudaErrorInvalidValue;
  bwd_pre_kernel<D><<<grid_ew, 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)a.s.nb * BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  bwd_tc_kernel<D><<<(unsigned)grid, kBwdThreads, C::kSmem, st>>>(tq, tk, tv, tdo, tdk, tdv, a);
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
