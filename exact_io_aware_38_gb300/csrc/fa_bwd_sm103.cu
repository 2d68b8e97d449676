// Backward attention on the 5th-generation tensor cores (sm_103a).
//
// Three launches on the caller's stream, each a programmatic dependent of the kernel before it
// (its launch overlaps that kernel's tail; it waits on the grid dependency before touching memory):
//   pre   D_i = sum_k dO_ik O_ik (fp32, from the stored bf16 O), a cleared fp32 dQ accumulator and
//         a cleared key-tile counter;
//   main  persistent, one CTA per SM, taking (128-key tile j, K/V head) pairs from the counter,
//         heavy tiles first: K_j and V_j stay in shared memory while the query rows that can see
//         them stream through a TMA ring, 64 rows per step. The score tile
//         is recomputed from Q, K and the saved log-sum-exp instead of being stored
//         ("FlashAttention." plate, "Never write the scores"), and the softmax gradient is applied
//         tile by tile:
//           S^T = K_j Q_i^T,  dP^T = V_j dO_i^T                  (tcgen05, into tensor memory)
//           P^T = exp(c S^T - LSE_i),  dS^T = P^T * (dP^T - D_i)  (one thread per key row)
//           dV_j += P^T dO_i,  dK_j += dS^T Q_i                  (A operand from tensor memory)
//           dQ_i^T = K_j^T dS_i^T                                (added into the fp32 accumulator)
//         dK_j = c * acc and dV_j are read out of tensor memory and stored from registers while
//         the next tile's K, V and first Q/dO steps load; the ring and the step counters run on
//         across tiles, so only the next tile's first gradient products wait for that read-out.
//   post  dQ = bf16(c * accumulator).
// dQ_i is formed transposed (tensor-memory lane = head dimension; at d = 64 the product keeps
// M = 128 and its upper rows are unused), staged row-major in shared memory and added into the
// accumulator by one bulk reduce-add of the bulk-copy engine per step. Two tensor-memory buffers
// [S^T | dP^T] alternate between steps; dQ^T accumulates over its buffer's dP^T columns once dK
// has read dS^T there, so S^T of step i+2 waits only for dV of step i and dP^T for the read-out
// of step i's dQ^T.
//
// d = 64 runs a single mode (192 threads, two CTAs per SM): one tensor-memory buffer, one issuer
// for the whole step chain, and one warpgroup for the elementwise step, the dQ read-out and dK, dV.
// There dQ^T accumulates over the S^T columns instead (free once dV has read P^T) and is issued
// before dK, so the step's dQ^T completes earlier and the next dP^T runs during its read-out.
// CTA layout (384 threads): warp 0 TMA producer; warp 1 S^T/dP^T MMA issuer and tensor-memory owner;
// warp 2 gradient MMA issuer;
// warps 4-7 elementwise warpgroup (thread = key row; lane quadrant = warp % 4), which also writes
// dK; warps 8-11 dQ warpgroup (reads dQ out of tensor memory, adds it into the accumulator), which
// also writes dV. The two warpgroups run concurrently on different steps.
// Tensor memory: dK [0,d) dV [d,2d), buffer b: S^T [2d+128b, +64), dP^T / dQ^T [+64, +128).
// P^T and dS^T (bf16) are written over the first 32 columns of S^T and dP^T.
#include <type_traits>

#include "fa_tmap.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace tc;

constexpr int kBwdThreads = 384;

// SINGLE (d = 64): one [S^T | dP^T] buffer, a 2-stage Q/dO ring and one K/V pair (97 KB of shared
// memory, 256 tensor-memory columns), 192 threads (producer, one issuer, one warpgroup), so two
// CTAs share an SM and one CTA's step chain runs while the other's waits.
template <int D, bool SINGLE = false>
struct BwdCfg {
  // Steps of 64 queries through two [S^T | dP^T] tensor-memory buffers; dQ^T = K^T dS^T (lanes =
  // head dimension) accumulates over its buffer's dP^T columns. At d = 64 that product keeps
  // M = 128: its upper 64 rows read the next shared-memory tile and are never read out (half of
  // one small product wasted for the known 128-lane layout and the double buffering).
  static constexpr int BM = 64;                      // query rows per step
  static constexpr int kBufs = SINGLE ? 1 : 2;       // tensor-memory [S^T | dP^T] buffers
  static constexpr int kBoxes = D / 64;              // 64-column boxes per row
  static constexpr int kKVBytes = 128 * D * 2;       // K or V tile (128 rows)
  static constexpr int kQBox = BM * 128;             // one 64-column box of a Q or dO tile
  static constexpr int kQBytes = BM * D * 2;         // Q or dO tile (BM rows)
  static constexpr int kStages = SINGLE ? 2 : 3;     // Q/dO ring depth
  // dS^T tile [128 keys][BM queries] per buffer, in 128-byte-swizzled rows of 64 queries (a step
  // of 32 queries uses the first half of each row).
  static constexpr int kDsBytes = 128 * BM * 2;
  static constexpr int kDqBytes = BM * D * 4;        // fp32 dQ staging for the bulk add
  static constexpr int kSmem = 2 * kKVBytes + kStages * 2 * kQBytes + kBufs * kDsBytes + kDqBytes + 1024;
  static constexpr int kThreadsCta = SINGLE ? 192 : kBwdThreads;
  static constexpr uint32_t kTmemCols = SINGLE ? 256 : 512;
  static_assert(!SINGLE || D == 64, "the single mode fits tensor memory at d = 64");
  static constexpr uint32_t kTdK = 0, kTdV = D;
  static constexpr uint32_t kTS0 = 2 * D;            // S^T of buffer b at kTS0 + b * 2 * BM
  static constexpr uint32_t kIdS = idesc_bf16(128, BM, false, false);
  static constexpr uint32_t kIdG = idesc_bf16(128, D, false, true);
  static constexpr uint32_t kIdQ = idesc_bf16(128, BM, true, true);
  static_assert(kSmem <= 232448 - 1536, "shared memory budget");
  static_assert(kStages <= 4 && kBufs <= 4, "barrier arrays of the control block");
};

constexpr int kMaxStages = 4;
constexpr int kMaxBufs = 4;

struct alignas(16) BwdSmemCtl {
  uint64_t kv_full;
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t s_full[kMaxBufs], p_ready[kMaxBufs], dq_full[kMaxBufs], dq_free[kMaxBufs], s_free[kMaxBufs];
  uint64_t done, acc_free, drain;
  uint64_t tq_full[2], tq_empty[2];  // key-tile queue
  uint32_t tmem_base;
  int abort_flag;
  int tile_q[2];      // key-tile queue slots
  int tile_bc[2][2];  // the tile index shared within each warpgroup, two slots each
  alignas(16) float lse2[128];  // LSE * log2(e) per query of the step: [buffer][BM]
  alignas(16) float dvec[128];  // D per query of the step: [buffer][BM]
  // Single mode: the queue item's visited steps per query head and first step, and the first step
  // as shared within the warpgroup (after the fields above, which keep their places).
  int tile_n[2], tile_vf[2];
  int tile_bcv[2];
};

template <int D>
__device__ __forceinline__ float* lse_row(BwdSmemCtl& c, int buf) {
  return c.lse2 + buf * BwdCfg<D>::BM;
}
template <int D>
__device__ __forceinline__ float* dvec_row(BwdSmemCtl& c, int buf) {
  return c.dvec + buf * BwdCfg<D>::BM;
}

// The pre and post passes walk the per-row arrays (D, the fp32 dQ accumulator) in their LSE order:
// runs of rows, one per (b, h) for fixed-length batches or per h for packed ones. A CTA takes 64
// rows of one run, so a row's tensor coordinates need no division, and moves 16 bytes per thread.
constexpr int kRowTile = 64;
struct RowTile {
  int b, h, row0, rows;  // rows [row0, row0 + rows) of run (b, h)
  size_t r0;             // LSE-order index of the run's row 0
};
__device__ __forceinline__ RowTile row_tile(const AttnShape& s) {
  const bool packed = s.cu_q != nullptr;
  const int nrows = packed ? s.rows_q : s.Nq;
  const int tiles = (nrows + kRowTile - 1) / kRowTile;
  const int run = blockIdx.x / tiles;
  RowTile t;
  t.b = packed ? 0 : run / s.H;
  t.h = packed ? run : run % s.H;
  t.row0 = (blockIdx.x % tiles) * kRowTile;
  t.rows = min(kRowTile, nrows - t.row0);
  t.r0 = (size_t)run * nrows;
  return t;
}
__host__ inline long long row_tile_grid(const AttnShape& s) {
  const bool packed = s.cu_q != nullptr;
  const long long nrows = packed ? s.rows_q : s.Nq;
  return (packed ? (long long)s.H : (long long)s.B * s.H) * ((nrows + kRowTile - 1) / kRowTile);
}

// D = rowsum(dO * O) per query row and a cleared dQ accumulator. A row of O (d bf16) is read by
// d / 8 lanes, 16 bytes each, and summed over them with shuffles.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const FaBwdArgs a) {
  grid_dependency_wait();  // a programmatic dependent of the previous kernel on the stream
  constexpr int LPR = D / 8, RPW = 32 / LPR;  // lanes per row, rows per warp
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.tile_counter = 0;  // the main kernel's key-tile counter
  if ((a.s.cu_q != nullptr ? a.s.rows_q : a.s.Nq) <= 0) return;   // (then a one-CTA launch)
  const RowTile T = row_tile(a.s);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, part = lane % LPR;
  const __nv_bfloat16* O = reinterpret_cast<const __nv_bfloat16*>(a.o);
  const __nv_bfloat16* dO = reinterpret_cast<const __nv_bfloat16*>(a.dout);
#pragma unroll
  for (int i = warp * RPW + lane / LPR; i < kRowTile; i += 8 * RPW) {
    const bool live = i < T.rows;
    float acc = 0.f;
    if (live) {
      const int row = T.row0 + i;
      const uint4 xs = *reinterpret_cast<const uint4*>(O + elem_offset(a.so, T.b, row, T.h) + part * 8);
      const uint4 ys = *reinterpret_cast<const uint4*>(dO + elem_offset(a.sdo, T.b, row, T.h) + part * 8);
      const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&xs);
      const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&ys);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc += __bfloat162float(x[e].x) * __bfloat162float(y[e].x) + __bfloat162float(x[e].y) * __bfloat162float(y[e].y);
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && part == 0) a.dvec[T.r0 + T.row0 + i] = acc;
  }
  float4* z = reinterpret_cast<float4*>(a.dqacc + (T.r0 + T.row0) * D);
  const int n4 = T.rows * (D / 4);
  for (int i = threadIdx.x; i < n4; i += 256) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = scale * accumulator in bf16 (or, accumulating, the caller's fp32 dQ += scale * accumulator).
// A row of the accumulator (d fp32) is read by d / 4 lanes, 16 bytes each.
template <int D>
__global__ void __launch_bounds__(256) bwd_post_kernel(const FaBwdArgs a) {
  grid_dependency_wait();  // the main pass has completed
  constexpr int LPR = D / 4, RPW = 32 / LPR;
  const RowTile T = row_tile(a.s);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, part = lane % LPR;
  __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(a.dq);
#pragma unroll
  for (int i = warp * RPW + lane / LPR; i < kRowTile; i += 8 * RPW) {
    if (i >= T.rows) continue;
    const int row = T.row0 + i;
    const float4 x = *reinterpret_cast<const float4*>(a.dqacc + (T.r0 + row) * D + part * 4);
    if (a.dq_acc != nullptr) {
      float4* dst = reinterpret_cast<float4*>(a.dq_acc + elem_offset(a.sdq, T.b, row, T.h) + part * 4);
      float4 y = *dst;
      y.x += x.x * a.scale;
      y.y += x.y * a.scale;
      y.z += x.z * a.scale;
      y.w += x.w * a.scale;
      *dst = y;
    } else {
      *reinterpret_cast<uint2*>(dq + elem_offset(a.sdq, T.b, row, T.h) + part * 4) =
          make_uint2(pack_bf16x2(x.x * a.scale, x.y * a.scale), pack_bf16x2(x.z * a.scale, x.w * a.scale));
    }
  }
}

// One key tile of the persistent backward kernel: the (key tile, K/V head) pair whose dK, dV it
// owns and the query steps that can see it. Every role derives the same values from the tile index.
struct BwdTile {
  int kt, b, hk, h0;
  SeqInfo seq;
  int nv;    // 64-row query steps of the sequence
  int v_lo;  // first candidate step (the key tile's diagonal step with the causal mask)
  bool live;  // the key tile has rows in this sequence (packed sequences end early)
};

__device__ __forceinline__ BwdTile bwd_tile(const AttnShape& s, int tile, int BM) {
  BwdTile t;
  const int BHkv = s.B * s.Hkv;
  t.kt = tile / BHkv;  // key tile: small kt (most causal work) first
  const int bkv = tile % BHkv;
  t.b = bkv / s.Hkv;
  t.hk = bkv % s.Hkv;
  t.h0 = t.hk * (s.H / s.Hkv);  // the group's first query head
  t.seq = seq_info(s, t.b);
  t.live = t.kt * 128 < t.seq.krows;
  t.nv = (t.seq.Lq + BM - 1) / BM;
  // No step is visited when the key tile lies past the key length; with the causal mask the first
  // candidate is the key tile's own diagonal step. Scans start there.
  t.v_lo = t.kt * 128 >= t.seq.Lk ? t.nv : (s.causal ? max(t.kt * 128 - t.seq.off, 0) / BM : 0);
  return t;
}

// Query steps v (rows v*BM ..) are visited iff their 128-row tile is visited for the key tile. The
// pattern is the same for every query head of the group; a step is a (group head gi, v) pair, heads
// outer, so dK and dV sum over the group in tensor memory. Without a block mask every step from
// v_lo on is visited (tile_visited in closed form). The next visited step is found by a whole warp
// with the same v, 32 candidates per block-mask probe (a serial scan would put one dependent load
// per skipped step on the path of the thread that waits on it).
__device__ __forceinline__ int bwd_next_v_warp(const AttnShape& s, const BwdTile& t, int v, int BM) {
  v = v < t.v_lo ? t.v_lo : v;
  if (s.block_mask == nullptr) return v < t.nv ? v : t.nv;
  const int lane_id = threadIdx.x & 31;
  for (; v < t.nv; v += 32) {
    const int c = v + lane_id;
    const unsigned hit = __ballot_sync(0xffffffffu, c < t.nv && tile_visited(s, t.seq, (c * BM) / 128, t.kt));
    if (hit) return v + __ffs(hit) - 1;
  }
  return t.nv;
}

// Visited steps of the tile for one query head and the first of them (nv if none), found by a
// whole warp: every step from v_lo on without a block mask; with one, each lane first loads its
// eight mask bytes unconditionally (the candidate is clamped to the last step, whose 128-row tile
// is inside the mask), so the eight loads are in flight together, and only then applies the
// bounds and the causal test. With the tests guarding each load, the loads went out one after
// another (~12,600 cycles per key tile on a 128 x 128 mask).
__device__ __forceinline__ int bwd_scan_steps(const AttnShape& s, const BwdTile& t, int BM, int& v_first) {
  if (!t.live) {
    v_first = t.nv;
    return 0;
  }
  if (s.block_mask == nullptr) {
    v_first = min(t.v_lo, t.nv);
    return t.nv - v_first;
  }
  const int lane_id = threadIdx.x & 31;
  int n = 0;
  v_first = t.nv;
  for (int v0 = t.v_lo; v0 < t.nv; v0 += 8 * 32) {
    uint32_t m[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = min(v0 + u * 32 + lane_id, t.nv - 1);
      m[u] = __ldg(s.block_mask + (size_t)((v * BM) / 128) * s.nbk + t.kt);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = v0 + u * 32 + lane_id;
      const int qt = (v * BM) / 128;
      const unsigned hit = __ballot_sync(
          0xffffffffu, v < t.nv && m[u] != 0 && !(s.causal && t.kt * 128 > qt * 128 + 127 + t.seq.off));
      if (v_first == t.nv && hit) v_first = v0 + u * 32 + __ffs(hit) - 1;
      n += __popc(hit);
    }
  }
  return n;
}

// ACC: accumulate mode (dK and dV added in fp32 into the caller's accumulators); a separate
// instantiation keeps the bf16-output kernel's code as it is.
template <int D, bool ACC = false, bool SINGLE = false>
__global__ void __launch_bounds__(SINGLE ? 192 : kBwdThreads, SINGLE ? 2 : 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const FaBwdArgs a) {
  using C = BwdCfg<D, SINGLE>;
  grid_dependency_wait();  // the pre pass has completed (D, the cleared accumulator, the counter)
  constexpr int BM = C::BM;
  constexpr int NB = C::kBufs;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_u32(smem), sV = sK + C::kKVBytes;  // the key tile's K and V
  const uint32_t sStage0 = sV + C::kKVBytes;                    // stage s: Q at +2s, dO at +2s+1
  const uint32_t sDs0 = sStage0 + C::kStages * 2 * C::kQBytes;
  const uint32_t sDq = sDs0 + NB * C::kDsBytes;
  volatile int* abort_flag = &ctl.abort_flag;
  volatile int* tile_q = ctl.tile_q;

  const AttnShape& s = a.s;
  const int G = s.H / s.Hkv;  // query heads sharing a K/V head
  const int ntiles = s.nbk * s.B * s.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  auto sQs = [&](int st) { return sStage0 + (2 * st) * C::kQBytes; };
  auto sdOs = [&](int st) { return sStage0 + (2 * st + 1) * C::kQBytes; };
  auto sDs = [&](int buf) { return sDs0 + buf * C::kDsBytes; };
  auto tS = [&](int buf) { return C::kTS0 + buf * 2 * BM; };
  auto tdP = [&](int buf) { return C::kTS0 + buf * 2 * BM + BM; };
  // dQ^T of a step accumulates over its buffer's dP^T columns (free once dK has read dS^T there),
  // so the next S^T into the buffer waits only for dV's read of P^T. The single mode puts it over
  // the S^T columns (free once dV has read P^T), issued ahead of dK (see the issuer).
  auto tdQ = [&](int buf) { return SINGLE ? tS(buf) : tdP(buf); };

  const uint32_t b_kv = smem_u32(&ctl.kv_full);
  auto b_full = [&](int i) { return smem_u32(&ctl.full[i]); };
  auto b_empty = [&](int i) { return smem_u32(&ctl.empty[i]); };
  auto b_sfull = [&](int i) { return smem_u32(&ctl.s_full[i]); };
  auto b_pready = [&](int i) { return smem_u32(&ctl.p_ready[i]); };
  auto b_dqfull = [&](int i) { return smem_u32(&ctl.dq_full[i]); };
  auto b_dqfree = [&](int i) { return smem_u32(&ctl.dq_free[i]); };
  auto b_sfree = [&](int i) { return smem_u32(&ctl.s_free[i]); };
  auto b_tqfull = [&](int i) { return smem_u32(&ctl.tq_full[i]); };
  auto b_tqempty = [&](int i) { return smem_u32(&ctl.tq_empty[i]); };
  const uint32_t b_done = smem_u32(&ctl.done);
  const uint32_t b_accfree = smem_u32(&ctl.acc_free), b_drain = smem_u32(&ctl.drain);

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(b_kv, 1);
    mbar_init(b_done, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(b_full(i), 1);
      mbar_init(b_empty(i), 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(b_sfull(i), 1);
      mbar_init(b_pready(i), 128);
      mbar_init(b_dqfull(i), 1);
      mbar_init(b_dqfree(i), 128);
      mbar_init(b_sfree(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_tqfull(i), 1);
      mbar_init(b_tqempty(i), SINGLE ? 2 : 4);  // the issuers and the warpgroups' leaders
    }
    mbar_init(b_accfree, SINGLE ? 128 : 256);  // every warpgroup thread, after reading dK or dV
    mbar_init(b_drain, SINGLE ? 1 : 2);        // one commit per MMA issuer
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  // Key tiles come from a counter shared by all CTAs (the first one is the CTA's own index), in
  // the heavy-first order of the tile index. The producer takes each one and publishes it through
  // a two-slot queue; every other role reads the same sequence from there. In the single mode the
  // producer also counts the tile's visited steps and finds the first before publishing, so the
  // issuer and the warpgroup scan nothing at a tile's start, where two CTAs with short key tiles
  // (d = 64) wait on it. With one CTA per SM (d = 128) each role scans for itself: the published
  // form measured 2-6% slower there, with identical outputs. Item w's phase of a
  // slot's full barrier cannot be confused with item w + 2's: that one is published only after all
  // four readers of item w have arrived on the slot's empty barrier.
  auto take_tile = [&](int w) -> int {  // one reader thread per role
    int tile = ntiles;  // an abandoned wait ends the loop
    if (mbar_wait(b_tqfull(w & 1), (w >> 1) & 1, abort_flag, a.status)) tile = tile_q[w & 1];
    mbar_arrive(b_tqempty(w & 1));
    return tile;
  };
  // Single mode: the same, also returning the item's step count and first step (read before the
  // arrival that lets the producer rewrite the slot).
  auto take_item = [&](int w, int& nsteps, int& v_first) -> int {
    int tile = ntiles;
    nsteps = 0;
    v_first = 0;
    if (mbar_wait(b_tqfull(w & 1), (w >> 1) & 1, abort_flag, a.status)) {
      tile = tile_q[w & 1];
      nsteps = ((volatile int*)ctl.tile_n)[w & 1];
      v_first = ((volatile int*)ctl.tile_vf)[w & 1];
    }
    mbar_arrive(b_tqempty(w & 1));
    return tile;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // Lane 0 takes the tiles, waits and issues the copies; with a block mask the whole warp walks
    // the steps with it (the mask is scanned 32 candidates per load).
    const bool walk = lane == 0 || s.block_mask != nullptr;
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmdO);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
    }
    uint32_t last_par[kMaxStages];
    bool issued[kMaxStages] = {};
    bool kv_any = false;
    uint32_t kv_par = 1;  // parity of the last K/V phase issued (flips before each issue)
    uint32_t i = 0;  // Q/dO ring position, continued across key tiles
    int wt = 0;      // key tiles with work so far
    for (int w = 0;; ++w) {
      int tile = ntiles;
      bool publish = false;
      if (lane == 0 && (w < 2 || mbar_wait(b_tqempty(w & 1), ((w - 2) >> 1) & 1, abort_flag, a.status))) {
        // After an abort the end marker is published, so every reader leaves its tile loop.
        tile = *abort_flag ? ntiles : (w == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(a.tile_counter, 1));
        if constexpr (!SINGLE) {
          tile_q[w & 1] = tile;
          mbar_arrive(b_tqfull(w & 1));  // release: the index is visible to every waiter of the phase
        }
        publish = true;
      }
      tile = __shfl_sync(0xffffffffu, tile, 0);
      int v_first = 0;
      BwdTile T;
      if constexpr (SINGLE) {  // scan first, then publish the item (the whole warp scans)
        int nsteps = 0;
        if (tile < ntiles) {
          T = bwd_tile(s, tile, BM);
          nsteps = bwd_scan_steps(s, T, BM, v_first);
        }
        if (publish) {
          tile_q[w & 1] = tile;
          ctl.tile_n[w & 1] = nsteps;
          ctl.tile_vf[w & 1] = v_first;
          mbar_arrive(b_tqfull(w & 1));  // release: the item is visible to every waiter of the phase
        }
        if (tile >= ntiles) break;
      } else {
        if (tile >= ntiles) break;
        T = bwd_tile(s, tile, BM);
        v_first = T.live ? bwd_next_v_warp(s, T, 0, BM) : T.nv;
      }
      if (v_first >= T.nv) continue;
      // K and V of this tile load once every MMA of the previous tile has completed (its done
      // commit), so the first two Q/dO steps are requested before that wait (their stages are
      // released earlier).
      bool kv_issued = false;
      auto issue_kv = [&]() {  // lane 0
        kv_issued = true;
        if (wt > 0 && !mbar_wait(b_done, (wt - 1) & 1, abort_flag, a.status)) return;
        // The previous K/V copy has landed (only the producer arrives on this barrier, so the
        // parity test cannot alias), and no copy is issued after an abort.
        if ((kv_any && !mbar_wait(b_kv, kv_par, abort_flag, a.status)) || *abort_flag) return;
#ifndef FA_TEST_WITHHOLD_KV  // a test-only build never loads K/V: every wait on them must run out
        mbar_expect_tx(b_kv, 2 * C::kKVBytes);
        for (int c = 0; c < C::kBoxes; ++c) {
          tma_load_4d(sK + c * 16384, &tmK, c * 64, T.seq.k0 + T.kt * 128, T.hk, T.seq.bb, b_kv);
          tma_load_4d(sV + c * 16384, &tmV, c * 64, T.seq.k0 + T.kt * 128, T.hk, T.seq.bb, b_kv);
        }
        kv_any = true;
        kv_par ^= 1u;
#endif
      };
      if (lane == 0 && wt == 0) issue_kv();
      int l = 0;
      for (int gi = 0, v = v_first; walk && gi < G && v < T.nv; ++i, ++l) {
        if (lane == 0) {
          if (l == 2 && !kv_issued) issue_kv();
          const int st = i % C::kStages;
          const uint32_t par = (i / C::kStages) & 1;
          // The stage is free once dV and dK of step j = i - kStages have read it (its S^T/dP^T
          // finished before them), which the gradient issuer commits to the stage's own barrier.
          // One barrier per stage keeps the parity test unambiguous: its next phase belongs to
          // step i, not loaded yet. The producer also checks that step j's own copy has landed (in
          // the normal path long since; after an abort the issuers' releases no longer prove it),
          // so a stage barrier never gets a second arrive.expect_tx while a phase is open, and it
          // issues no copy after an abort.
          const int j = (int)i - C::kStages;
          if ((j < 0 || (mbar_wait(b_empty(j % C::kStages), (j / C::kStages) & 1, abort_flag, a.status) &&
                         mbar_wait(b_full(j % C::kStages), (j / C::kStages) & 1, abort_flag, a.status))) &&
              !*abort_flag) {
            mbar_expect_tx(b_full(st), 2 * C::kQBytes);
            for (int c = 0; c < C::kBoxes; ++c) {
              tma_load_4d(sQs(st) + c * C::kQBox, &tmQ, c * 64, T.seq.q0 + v * BM, T.h0 + gi, T.seq.bb, b_full(st));
              tma_load_4d(sdOs(st) + c * C::kQBox, &tmdO, c * 64, T.seq.q0 + v * BM, T.h0 + gi, T.seq.bb, b_full(st));
            }
            issued[st] = true;
            last_par[st] = par;
          }
        }
        v = bwd_next_v_warp(s, T, v + 1, BM);
        if (v >= T.nv) {
          ++gi;
          v = v_first;
        }
      }
      if (lane == 0 && !kv_issued) issue_kv();
      ++wt;
    }
    // Let copies still in flight land before the CTA exits. A stage (and the K/V buffer) is
    // reloaded only once its previous copy has landed, so each of these barriers has at most one
    // phase in flight: the last one issued, whose only arrival is the producer's own.
    if (lane == 0 && *abort_flag) {
      if (kv_any) mbar_wait_drain(b_kv, kv_par);
      for (int k = 0; k < C::kStages; ++k)
        if (issued[k]) mbar_wait_drain(b_full(k), last_par[k]);
    }
  } else if (SINGLE ? warp == 1 : (warp == 1 || warp == 2)) {
    // ------------------------------------------------------------------ MMA issuers
    // Two issuing threads, one per dependency chain: a thread issuing tcgen05 MMAs blocks while
    // the tensor core's queue is full, so one issuer could not react to the other chain.
    //   warp 1: S^T/dP^T of step sn into buffer sn % NB, once its Q/dO tile has landed: S^T once
    //           dV of step sn - NB has read P^T (the s_free commit), dP^T once that step's dQ^T,
    //           accumulated over the dP^T columns after dK read dS^T there, has been read out;
    //   warp 2: dV, dK and dQ of step g, once P^T/dS^T of step g are in place (which follows the
    //           completion of step g's S^T/dP^T); a tile's first dV and dK (which overwrite the
    //           accumulators) once the previous tile's dK and dV have been read out.
    // Step counters run on across key tiles, so the ring and the buffers never drain between them.
    // Descriptors of the resident K and V tiles, advanced by constant byte offsets per k-step.
    const uint64_t dK0 = desc_kmajor_sw128(sK), dV0 = desc_kmajor_sw128(sV), mK0 = desc_mnmajor_sw128(sK, 16384);
    uint32_t sn = 0;  // global step counter (lane 0)
    int wt = 0;
    for (int w = 0;; ++w) {
      int tile = 0, n = 0;
      if constexpr (SINGLE) {  // the producer's count
        int vf_unused;
        if (lane == 0) tile = take_item(w, n, vf_unused);
        tile = __shfl_sync(0xffffffffu, tile, 0);
        if (tile >= ntiles) break;
        n = __shfl_sync(0xffffffffu, n, 0) * G;
      } else {
        if (lane == 0) tile = take_tile(w);
        tile = __shfl_sync(0xffffffffu, tile, 0);
        if (tile >= ntiles) break;
        const BwdTile T = bwd_tile(s, tile, BM);
        if (!T.live) continue;
        int vf_unused;
        n = bwd_scan_steps(s, T, BM, vf_unused) * G;
      }
      if (n == 0) continue;
      if (lane == 0 && SINGLE) {
        // One issuer, one buffer: per step dP^T and S^T, then (after the warpgroup's P^T, dS^T)
        // dV, dQ^T and dK. In the one in-order queue dQ^T overwrites P^T only after dV has read
        // it, and the next step's dP^T overwrites dS^T only after dK has read it, so dP^T issues
        // at once; the next S^T waits for the read-out of dQ^T, held in the S^T columns. With dK
        // after dQ^T the read-out starts one product earlier, and the next dP^T runs during it
        // (block-sparse d = 64 backward 0.4585 -> 0.4366 ms side by side, against dV, dK, dQ^T
        // over the dP^T columns).
        mbar_wait_spin(b_kv, wt & 1, abort_flag, a.status);
        fence_after_sync();
        for (int l = 0; l < n; ++l, ++sn) {
          const int st = sn % C::kStages;
          mbar_wait_spin(b_full(st), (sn / C::kStages) & 1, abort_flag, a.status);
          fence_after_sync();
          const uint64_t dq = desc_kmajor_sw128(sQs(st)), ddo = desc_kmajor_sw128(sdOs(st));
          // dP^T first: its columns are free once the previous step's dK has read dS^T (earlier in
          // this queue); S^T waits for the read-out of the previous dQ^T, held in its columns.
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t okk = (kk >> 2) * 16384 + (kk & 3) * 32, oq = (kk >> 2) * C::kQBox + (kk & 3) * 32;
            mma_ss(tmem + tdP(0), desc_add(dV0, okk), desc_add(ddo, oq), C::kIdS, kk > 0);
          }
          if (sn > 0) {  // dQ^T of the previous step has been read out of the S^T columns
            mbar_wait_spin(b_dqfree(0), (sn - 1) & 1, abort_flag, a.status);
            fence_after_sync();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t okk = (kk >> 2) * 16384 + (kk & 3) * 32, oq = (kk >> 2) * C::kQBox + (kk & 3) * 32;
            mma_ss(tmem + tS(0), desc_add(dK0, okk), desc_add(dq, oq), C::kIdS, kk > 0);
          }
          mma_commit(b_sfull(0));
          if (l == 0 && wt > 0) {  // the previous tile's dK and dV have left tensor memory
            mbar_wait_spin(b_accfree, (wt - 1) & 1, abort_flag, a.status);
            fence_after_sync();
          }
          mbar_wait_spin(b_pready(0), sn & 1, abort_flag, a.status);
          fence_after_sync();
          const uint64_t mq = desc_mnmajor_sw128(sQs(st), C::kQBox), mdo = desc_mnmajor_sw128(sdOs(st), C::kQBox);
          const uint64_t mds = desc_mnmajor_sw128(sDs(0), 16384);
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_ts(tmem + C::kTdV, tmem + tS(0) + kk * 8, desc_add(mdo, kk * 2048), C::kIdG, (l > 0 || kk > 0) ? 1u : 0u);
          // dQ^T over the S^T columns (after dV has read P^T there), ahead of dK.
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + tdQ(0), desc_add(mK0, kk * 2048), desc_add(mds, kk * 2048), C::kIdQ, kk > 0);
          mma_commit(b_dqfull(0));
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_ts(tmem + C::kTdK, tmem + tdP(0) + kk * 8, desc_add(mq, kk * 2048), C::kIdG, (l > 0 || kk > 0) ? 1u : 0u);
          mma_commit(b_empty(st));  // dV and dK have read the step's Q/dO stage
        }
        mma_commit(b_done);  // the tile's last MMAs complete after every product of it
      } else if (lane == 0) {
        if (warp == 1) {
          mbar_wait_spin(b_kv, wt & 1, abort_flag, a.status);
          fence_after_sync();
          for (int l = 0; l < n; ++l, ++sn) {
            const int st = sn % C::kStages, buf = sn % NB;
            mbar_wait_spin(b_full(st), (sn / C::kStages) & 1, abort_flag, a.status);
            if (sn >= NB) {  // dV of step sn - NB has read P^T from these columns
              mbar_wait_spin(b_sfree(buf), ((sn - NB) / NB) & 1, abort_flag, a.status);
              fence_after_sync();
            }
            const uint64_t dq = desc_kmajor_sw128(sQs(st)), ddo = desc_kmajor_sw128(sdOs(st));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t okk = (kk >> 2) * 16384 + (kk & 3) * 32, oq = (kk >> 2) * C::kQBox + (kk & 3) * 32;
              mma_ss(tmem + tS(buf), desc_add(dK0, okk), desc_add(dq, oq), C::kIdS, kk > 0);
            }
            if (sn >= NB) {  // dQ^T of step sn - NB has been read out of these columns
              mbar_wait_spin(b_dqfree(buf), ((sn - NB) / NB) & 1, abort_flag, a.status);
              fence_after_sync();
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t okk = (kk >> 2) * 16384 + (kk & 3) * 32, oq = (kk >> 2) * C::kQBox + (kk & 3) * 32;
              mma_ss(tmem + tdP(buf), desc_add(dV0, okk), desc_add(ddo, oq), C::kIdS, kk > 0);
            }
            mma_commit(b_sfull(buf));
          }
        } else {
          if (wt > 0) {  // the previous tile's dK and dV have left tensor memory
            mbar_wait_spin(b_accfree, (wt - 1) & 1, abort_flag, a.status);
            fence_after_sync();
          }
          for (int l = 0; l < n; ++l, ++sn) {
            const int st = sn % C::kStages, buf = sn % NB;
            mbar_wait_spin(b_pready(buf), (sn / NB) & 1, abort_flag, a.status);
            fence_after_sync();
            const uint64_t mq = desc_mnmajor_sw128(sQs(st), C::kQBox), mdo = desc_mnmajor_sw128(sdOs(st), C::kQBox);
            const uint64_t mds = desc_mnmajor_sw128(sDs(buf), 16384);
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              mma_ts(tmem + C::kTdV, tmem + tS(buf) + kk * 8, desc_add(mdo, kk * 2048), C::kIdG,
                     (l > 0 || kk > 0) ? 1u : 0u);
            mma_commit(b_sfree(buf));  // P^T read: the S^T columns are free
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              mma_ts(tmem + C::kTdK, tmem + tdP(buf) + kk * 8, desc_add(mq, kk * 2048), C::kIdG,
                     (l > 0 || kk > 0) ? 1u : 0u);
            mma_commit(b_empty(st));  // dV and dK have read the step's Q/dO stage
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + tdQ(buf), desc_add(mK0, kk * 2048), desc_add(mds, kk * 2048), C::kIdQ, kk > 0);
            mma_commit(b_dqfull(buf));
          }
          mma_commit(b_done);  // the tile's last MMAs complete after every S^T/dP^T of it
        }
      }
      ++wt;
    }
    if (lane == 0) {
      mma_commit(b_drain);
      mbar_wait_drain(b_drain, 0);
    }
  } else if (SINGLE ? warp >= 2 : warp >= 4) {
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // tensor-memory lane: key row (and head dimension of dQ^T)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // SINGLE: one warpgroup (warps 2-5) does the elementwise step, the dQ read-out and both dK, dV.
    const bool elementwise = SINGLE || warp < 8;
    const int grp_bar = elementwise ? 1 : 2;                     // the warpgroup's named barrier
    const int leader = SINGLE ? 64 : (elementwise ? 128 : 256);  // its reader of the tile queue
    const int dq_leader = SINGLE ? 64 : 256;                     // issues the dQ bulk adds
    volatile int* tile_bc = ctl.tile_bc[elementwise ? 0 : 1];
    const float sl2 = a.scale * kLog2e;
    uint32_t it = 0;  // global step counter
    int wt = 0;
    for (int w = 0;; ++w) {
      // The warpgroup agrees on the tile: its leader reads the queue and shares the index (and in
      // the single mode the first visited step; two slots, so a slot is rewritten only after the
      // next iteration's barrier).
      if (threadIdx.x == leader) {
        if constexpr (SINGLE) {
          int n_unused, vf;
          tile_bc[w & 1] = take_item(w, n_unused, vf);
          ctl.tile_bcv[w & 1] = vf;
        } else {
          tile_bc[w & 1] = take_tile(w);
        }
      }
      named_bar_sync(grp_bar, 128);
      const int tile = tile_bc[w & 1];
      if (tile >= ntiles) break;
      const BwdTile T = bwd_tile(s, tile, BM);
      int32_t* visits = (a.step_visits != nullptr && threadIdx.x == (SINGLE ? 64 : 128))
                            ? a.step_visits + ((size_t)T.b * s.Hkv + T.hk) * s.nbk + T.kt
                            : nullptr;
      if (!T.live) {
        if (visits) *visits = 0;
        continue;
      }
      const SeqInfo& seq = T.seq;
      const int kt = T.kt;
      int v_first;
      if constexpr (SINGLE) {
        v_first = ((volatile int*)ctl.tile_bcv)[w & 1];  // the producer's scan
      } else {
        v_first = bwd_next_v_warp(s, T, 0, BM);
      }
      const bool any_work = v_first < T.nv;
      const uint32_t it_first = it;
      // dQ^T of step it_ (query head gi_, rows q0_..): read out of tensor memory, staged row-major
      // and added into the fp32 accumulator by one bulk reduce-add.
      auto dq_out = [&](uint32_t it_, int gi_, int q0_) {
        const int buf = it_ % NB;
        float* dQa = a.dqacc + row_base(s, seq, T.b, T.h0 + gi_) * D;
        mbar_wait(b_dqfull(buf), (it_ / NB) & 1, abort_flag, a.status);
        fence_after_sync();
        const uint32_t tq = tmem + lane_off + tdQ(buf);
        // dQ^T: lane r = head dimension, columns = the step's BM queries (lanes r >= d hold the
        // unused rows of the d = 64 product).
        uint32_t vals[BM];
#pragma unroll
        for (int c = 0; c < BM / 32; ++c) tmem_ld32(tq + c * 32, *reinterpret_cast<uint32_t(*)[32]>(vals + c * 32));
        tmem_ld_wait();
        fence_before_sync();
        mbar_arrive(b_dqfree(buf));  // tensor-memory columns free for step it_ + NB
        if (threadIdx.x == dq_leader) tma_store_wait_read0();  // the previous bulk add has read the staging
        named_bar_sync(2, 128);
        if (r < D) {
#pragma unroll
          for (int qq = 0; qq < BM; ++qq)
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(sDq + (uint32_t)(qq * D + r) * 4u), "r"(vals[qq]) : "memory");
        }
        fence_proxy_async_smem();
        named_bar_sync(2, 128);
        if (threadIdx.x == dq_leader && !*abort_flag) {
          const int rows = min(BM, seq.Lq - q0_);
          bulk_reduce_add_f32(dQa + (size_t)q0_ * D, sDq, (uint32_t)(rows * D * 4));
          tma_store_commit();
        }
      };
      if (elementwise) {
        // -------------------------------------------------------------- P^T and dS^T
        const int key = kt * 128 + r;
        const bool key_ok = key < seq.Lk;
        // LSE and D of a step are loaded one step ahead and consumed only when they are stored
        // for the next step, so the load latency overlaps a whole step.
        auto fetch = [&](int gi, int v, float& lv, float& dv) {
          const int q = v * BM + r;
          const bool ok = gi < G && v < T.nv && r < BM && q < seq.Lq;
          const size_t row = row_base(s, seq, T.b, T.h0 + gi) + q;
          lv = ok ? a.lse[row] : 0.f;
          dv = ok ? a.dvec[row] : 0.f;
        };
        float next_l, next_d;
        fetch(0, v_first, next_l, next_d);
        for (int gi = 0, v = v_first; gi < G && v < T.nv; ++it) {
          const int q0 = v * BM;
          const int buf = it % NB;
          float* lrow = lse_row<D>(ctl, it & 1);
          float* drow = dvec_row<D>(ctl, it & 1);
          // With two row buffers, every thread finished reading this one (step it - 2) before the
          // barrier of step it - 1, so only one barrier per step is needed.
          if (r < BM) {
            lrow[r] = next_l * kLog2e;
            drow[r] = next_d;
          }
          named_bar_sync(1, 128);  // the rows are written before anyone reads them
          int gn = gi, vn = bwd_next_v_warp(s, T, v + 1, BM);
          if (vn >= T.nv) {
            ++gn;
            vn = v_first;
          }
          fetch(gn, vn, next_l, next_d);
          mbar_wait_spin(b_sfull(buf), (it / NB) & 1, abort_flag, a.status);  // on the critical path
          fence_after_sync();
          const bool need_mask =
              (s.causal && kt * 128 + 127 > q0 + seq.off) || (kt * 128 + 128 > seq.Lk) || (q0 + BM > seq.Lq);
          const uint32_t ts = tmem + lane_off + tS(buf), tdp = tmem + lane_off + tdP(buf);
          // P^T, dS^T for the step's BM queries, 32 at a time; the mask is resolved per step so
          // the unmasked body has no branches.
          auto step = [&](auto mask_tag) {
            constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
              uint32_t sr[32], dr[32];
              tmem_ld32(ts + c * 32, sr);
              tmem_ld32(tdp + c * 32, dr);
              tmem_ld_wait();
              uint32_t pk[16], dk[16];
#pragma unroll
              for (int t = 0; t < 32; t += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(lrow + c * 32 + t);
                const float4 d4 = *reinterpret_cast<const float4*>(drow + c * 32 + t);
                const float2 sc2 = make_float2(sl2, sl2);
#pragma unroll
                for (int u = 0; u < 4; u += 2) {
                  const float2 lv = u == 0 ? make_float2(-l4.x, -l4.y) : make_float2(-l4.z, -l4.w);
                  const float2 dv2 = u == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);
                  const float2 x =
                      fma2(make_float2(__uint_as_float(sr[t + u]), __uint_as_float(sr[t + u + 1])), sc2, lv);
                  float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                  if constexpr (MASK) {
                    const int q = q0 + c * 32 + t + u;
                    p.x = (key_ok && q < seq.Lq && !(s.causal && key > q + seq.off)) ? p.x : 0.f;
                    p.y = (key_ok && q + 1 < seq.Lq && !(s.causal && key > q + 1 + seq.off)) ? p.y : 0.f;
                  }
                  const float2 dd =
                      mul2(p, sub2(make_float2(__uint_as_float(dr[t + u]), __uint_as_float(dr[t + u + 1])), dv2));
                  pk[(t + u) >> 1] = pack_bf16x2(p.x, p.y);
                  dk[(t + u) >> 1] = pack_bf16x2(dd.x, dd.y);
                }
              }
              tmem_st16(ts + c * 16, pk);
              tmem_st16(tdp + c * 16, dk);
              const uint32_t box = sDs(buf) + (c >> 1) * 16384 + r * 128;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int chunk = (c & 1) * 4 + j;
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(box + ((chunk ^ (r & 7)) << 4)),
                             "r"(dk[4 * j]), "r"(dk[4 * j + 1]), "r"(dk[4 * j + 2]), "r"(dk[4 * j + 3])
                             : "memory");
              }
            }
          };
          if (need_mask)
            step(std::true_type{});
          else
            step(std::false_type{});
          tmem_st_wait();
          fence_proxy_async_smem();
          fence_before_sync();
          mbar_arrive(b_pready(buf));
          if constexpr (SINGLE) dq_out(it, gi, q0);  // the same warpgroup reads out the step's dQ
          gi = gn;
          v = vn;
        }
        if (visits) *visits = (int32_t)(it - it_first);  // the steps this warpgroup walked
      } else {
        // -------------------------------------------------------------- dQ into the accumulator
        for (int gi = 0, v = v_first; gi < G && v < T.nv; ++it) {
          dq_out(it, gi, v * BM);
          v = bwd_next_v_warp(s, T, v + 1, BM);
          if (v >= T.nv) {
            ++gi;
            v = v_first;
          }
        }
      }

      // -------------------------------------------------------------- dK (warps 4-7), dV (8-11)
      // Read out of tensor memory, released for the next tile's first products, then stored
      // straight from registers (no shared-memory staging competes with the next tile's loads).
      // SINGLE: the one warpgroup writes both, staged through shared memory (below); with ACC
      // it adds dK, then dV, into the caller's fp32 accumulators.
      const int key = kt * 128 + r;
      const bool store = key < seq.krows;
      if (any_work) {
        mbar_wait(b_done, wt & 1, abort_flag, a.status);
        fence_after_sync();
      }
      if constexpr (SINGLE && !ACC) {
        // Both accumulators are read out first (the next tile's first products may then start),
        // staged as bf16 rows in 128-byte-swizzled shared memory (dK in the dS^T tile, which the
        // tile's last dQ^T product has finished reading, dV in the dQ staging once its last bulk
        // add has read it), and copied out eight threads per 128-byte row: a warp's store covers
        // four rows instead of 32 (the row-per-thread stores took ~3,200 cycles per key tile).
        uint32_t pk[2][D / 2];
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          const float mul = pass == 0 ? a.scale : 1.f;
          const uint32_t tacc = tmem + lane_off + (pass == 0 ? C::kTdK : C::kTdV);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t vv[32];
            if (any_work) {
              tmem_ld32(tacc + c * 32, vv);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) vv[i] = 0u;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[pass][c * 16 + i] = pack_bf16x2(__uint_as_float(vv[2 * i]) * mul, __uint_as_float(vv[2 * i + 1]) * mul);
          }
        }
        if (any_work) {  // the accumulators may be overwritten by the next tile's first products
          fence_before_sync();
          mbar_arrive(b_accfree);
          ++wt;
        }
        if (threadIdx.x == dq_leader) tma_store_wait_read0();  // the last dQ bulk add has read its staging
        named_bar_sync(1, 128);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          const uint32_t row = (pass == 0 ? sDs(0) : sDq) + (uint32_t)r * 128u;
#pragma unroll
          for (int j = 0; j < D / 8; ++j)
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(row + ((j ^ (r & 7)) << 4)),
                         "r"(pk[pass][4 * j]), "r"(pk[pass][4 * j + 1]), "r"(pk[pass][4 * j + 2]), "r"(pk[pass][4 * j + 3])
                         : "memory");
        }
        named_bar_sync(1, 128);
        const int t = threadIdx.x - 64;  // 0..127 within the warpgroup
#pragma unroll 4
        for (int k = 0; k < 2 * 128 * (D / 8) / 128; ++k) {
          const int idx = k * 128 + t;
          const int pass = idx / (128 * (D / 8));
          const int rr = (idx / (D / 8)) % 128, chunk = idx % (D / 8);
          uint4 x;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                       : "r"((pass == 0 ? sDs(0) : sDq) + (uint32_t)rr * 128u + ((chunk ^ (rr & 7)) << 4))
                       : "memory");
          const int krow = kt * 128 + rr;
          if (krow < seq.krows)
            *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(pass == 0 ? a.dk : a.dv) +
                                      elem_offset(pass == 0 ? a.sdk : a.sdv, seq.bb, seq.k0 + krow, T.hk) +
                                      chunk * 8) = x;
        }
        // The staging buffers are next written after the next tile's first barrier.
        continue;
      }
#pragma unroll 1
      for (int pass = 0; pass < (SINGLE ? 2 : 1); ++pass) {
      const bool is_dk = SINGLE ? pass == 0 : elementwise;
      const float mul = is_dk ? a.scale : 1.f;
      __nv_bfloat16* grow = reinterpret_cast<__nv_bfloat16*>(is_dk ? a.dk : a.dv) +
                            elem_offset(is_dk ? a.sdk : a.sdv, seq.bb, seq.k0 + (store ? key : 0), T.hk);
      const uint32_t tacc = tmem + lane_off + (is_dk ? C::kTdK : C::kTdV);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t vv[32];
        if (any_work) {
          tmem_ld32(tacc + c * 32, vv);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) vv[i] = 0u;
        }
        if constexpr (ACC) {  // fp32 shares added into the caller's accumulators (this CTA owns the rows)
          if (store) {
            float4* arow = reinterpret_cast<float4*>((is_dk ? a.dk_acc : a.dv_acc) +
                                                     elem_offset(is_dk ? a.sdk : a.sdv, seq.bb, seq.k0 + key, T.hk)) +
                           c * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float4 x = arow[j];
              x.x += __uint_as_float(vv[4 * j]) * mul;
              x.y += __uint_as_float(vv[4 * j + 1]) * mul;
              x.z += __uint_as_float(vv[4 * j + 2]) * mul;
              x.w += __uint_as_float(vv[4 * j + 3]) * mul;
              arow[j] = x;
            }
          }
        } else {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(vv[2 * i]) * mul, __uint_as_float(vv[2 * i + 1]) * mul);
        if (store) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(grow + c * 32 + j * 8) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
        }
      }
      }
      if (any_work) {  // the accumulators may be overwritten by the next tile's first products
        fence_before_sync();
        mbar_arrive(b_accfree);
        ++wt;
      }
    }
    if (threadIdx.x == dq_leader) tma_store_wait_read0();  // the staging is read before the CTA exits
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch(const FaBwdArgs& a, cudaStream_t st) {
  // d = 64 runs the single mode: two CTAs per SM, so one CTA's step chain runs while the other's
  // waits on its softmax or dQ read-out.
  constexpr bool SG = D == 64;
  using C = BwdCfg<D, SG>;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long grid_rows = row_tile_grid(a.s);
  if (grid_rows > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const AttnShape& s = a.s;
  const bool packed = s.cu_q != nullptr;
  const int rq = packed ? s.rows_q : s.Nq, rk = packed ? s.rows_k : s.Nk, nbatch = packed ? 1 : s.B;
  CUtensorMap tq, tk, tv, tdo;
  if (!fa_make_tmap_bf16(&tq, a.q, D, rq, s.H, nbatch, a.sq.row, a.sq.head, a.sq.batch, C::BM) ||
      !fa_make_tmap_bf16(&tk, a.k, D, rk, s.Hkv, nbatch, a.sk.row, a.sk.head, a.sk.batch) ||
      !fa_make_tmap_bf16(&tv, a.v, D, rk, s.Hkv, nbatch, a.sv.row, a.sv.head, a.sv.batch) ||
      !fa_make_tmap_bf16(&tdo, a.dout, D, rq, s.H, nbatch, a.sdo.row, a.sdo.head, a.sdo.batch, C::BM))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_dependent(bwd_pre_kernel<D>, dim3((unsigned)(grid_rows > 0 ? grid_rows : 1)), dim3(256), 0, st, a);
  if (e != cudaSuccess) return e;
  auto main_kernel = a.dk_acc != nullptr ? bwd_tc_kernel<D, true, SG> : bwd_tc_kernel<D, false, SG>;
  e = cudaFuncSetAttribute(main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  if (SG && (e = cudaFuncSetAttribute(main_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100)) != cudaSuccess)
    return e;
  // Persistent: one CTA per SM (two in the single mode), key tiles handed out by the counter.
  const long long ntiles = (long long)s.nbk * s.B * s.Hkv;
  if (ntiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (a.ev_main_begin != nullptr && (e = cudaEventRecord(a.ev_main_begin, st)) != cudaSuccess) return e;
  if (ntiles > 0) {
    const long long slots = (long long)sms * (SG ? 2 : 1);
    const unsigned grid = (unsigned)(ntiles < slots ? ntiles : slots);
    e = launch_dependent(main_kernel, dim3(grid), dim3(C::kThreadsCta), C::kSmem, st, tq, tk, tv, tdo, a);
    if (e != cudaSuccess) return e;
  }
  if (a.ev_main_end != nullptr && (e = cudaEventRecord(a.ev_main_end, st)) != cudaSuccess) return e;
  if (grid_rows > 0) return launch_dependent(bwd_post_kernel<D>, dim3((unsigned)grid_rows), dim3(256), 0, st, a);
  return cudaSuccess;
}

}  // namespace
}  // namespace fa

cudaError_t fa_launch_bwd(const FaBwdArgs& a, cudaStream_t st) {
  return a.s.d == 64 ? fa::launch<64>(a, st) : fa::launch<128>(a, st);
}
