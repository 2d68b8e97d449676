// Forward attention on the 5th-generation tensor cores (sm_103a): TMA + mbarrier pipeline,
// tcgen05 MMAs accumulating in tensor memory, warp-specialised roles.
//
// What it computes ("FlashAttention." plate, intro and "Never write the scores"; essay "Flash
// Attention: IO-Aware Attention Computation", paragraphs 3-5): for each 128-row query tile, the
// key/value tiles it can see are streamed through shared memory; each score tile S = Q K^T is
// folded into a running output with the online softmax (running row max m and row sum l; the
// partial output is rescaled when m grows), and O = acc / l and LSE = m + ln l are written at
// the end. Scores never leave the chip. Tiles with no valid (query, key) pair are skipped whole.
//
// CTA layout (320 threads, one CTA per SM): two 128-row query tiles Q0, Q1 share every K/V tile.
//   warp 0      TMA producer: Q0, Q1 once, the first K tile alone, then one ring stage per visited
//               key tile j: V_j and K_j+1 in one buffer (kStages buffers).
//   warp 1      MMA issuer (one thread) and tensor-memory owner: S_x = Q_x K_j^T (both operands
//               K-major in smem) and O_x += P_x V_j (P_x from tensor memory, V_j MN-major in smem).
//   warps 2-5   softmax for Q0; warps 6-9 softmax for Q1. Thread t of a warpgroup owns one query
//               row (its tensor-memory lane), so row max and row sum are thread-local (the row is
//               never split across threads in the 32x32b tensor-memory access shape).
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+d), O1 [256+d,256+2d).
// P_x is written as bf16 over the first 64 columns of S_x.
// MMA issue order per key tile j: PV0(j), S0(j+1), PV1(j), S1(j+1), so the tensor core computes
// one tile's products while the other tile's softmax runs.
// The single mode at d = 64 (256 columns: S [0,128), O [128,192)) writes P to the last 64 columns
// [192,256) instead, and issues S(j+1) ahead of PV(j): the next scores need only the softmax's
// read of S, and P V leaves the tile's chain. The softmax waits for PV(j) (a commit of its own)
// before it rescales O or writes P(j+1) (block-sparse d = 64 forward 0.1687 -> 0.1629 ms side by
// side, outputs identical).
// The tensor core's instruction queue is shallow: the issuing thread runs nearly in step with the
// pipe, and every barrier wait or commit it executes between MMA groups is time the pipe idles.
// So the issuer waits twice per key tile: once on the stage barrier, which completes when the
// stage's copies have landed AND tile 0's softmax has written P0 (the producer stands in with
// 128 arrivals when tile 0 skips the key tile), and once on P1. It polls without suspending.
// The partial output is rescaled only when a row max grows by more than 2^8 (lazy rescaling;
// exact, since l and O always share the same reference max).
#include <type_traits>

#include "fa_tmap.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace tc;

constexpr int kThreads = 320;        // pair mode: producer, issuer, two softmax warpgroups
constexpr int kThreadsSingle = 192;  // single mode: producer, issuer, one softmax warpgroup
constexpr int kVisWords = 64;  // key tiles covered by the per-CTA visibility bitmap: 2048

// F8: e4m3 operands (Q, K and V^T with per-head descales; d = 128), the two products as
// kind::f8f6f4 MMAs and P rounded to e4m3 as 2^8 P; otherwise bf16 operands (kind::f16).
template <int D, bool F8 = false, bool SINGLE = false>
struct FwdCfg {
  static constexpr int kBoxCols = F8 ? 128 : 64;        // columns of one 128-byte TMA box
  static constexpr int kBoxes = D / kBoxCols;           // boxes per operand row
  static constexpr int kOBoxes = D / 64;                // boxes per bf16 output row
  static constexpr int kTileBytes = 128 * D * (F8 ? 1 : 2);  // one 128-row operand tile (Q, K, V or V^T)
  static constexpr int kQSlot = 128 * D * 2;            // a query tile's slot: Q, later its bf16 O staging
  static constexpr int kTiles = SINGLE ? 1 : 2;         // query tiles per CTA
  // K/V ring: stage t holds V_t, K_t+1. The bf16 single mode at d = 128 (one query tile: decode
  // shapes) keeps one stage, so two CTAs fit an SM and each hides the other's loads.
  static constexpr int kStages = SINGLE ? ((D == 128 && !F8) ? 1 : 2) : ((D == 128 && !F8) ? 2 : 4);
  static constexpr int kSmem = kTiles * kQSlot + 2 * kStages * kTileBytes + 1024;
  static constexpr int kThreadsCta = SINGLE ? kThreadsSingle : kThreads;
  static constexpr uint32_t kTmemCols = SINGLE ? 256 : 512;
  static constexpr int kSSteps = D / (F8 ? 32 : 16);    // MMAs of one S = Q K^T (K = 16 bf16 / 32 e4m3 each)
  static constexpr int kPVSteps = 128 / (F8 ? 32 : 16);  // MMAs of one O += P V
  static constexpr uint32_t kIdS = F8 ? idesc_e4m3(128, 128) : idesc_bf16(128, 128, false, false);
  static constexpr uint32_t kIdPV = F8 ? idesc_e4m3(128, D) : idesc_bf16(128, D, false, true);
  static constexpr uint32_t kTmemS0 = 0, kTmemO0 = SINGLE ? 128 : 256;
  // d = 64 single mode: P gets the last 64 of the 256 columns instead of S's first ones, so the
  // next S may be issued once the softmax has read S, ahead of this tile's P V.
  static constexpr bool kSepP = SINGLE && D == 64 && !F8;
  static constexpr uint32_t kTmemP0 = kSepP ? 192 : kTmemS0;
  // O is rescaled only when a row max grows by more than kRescale in log2 units (lazy; exact since
  // l and O share the stale max). The e4m3 P is 2^8 exp2(s - m): with m at most 0.8 below the
  // true max it stays <= 2^8.8 < 448, the largest e4m3 value, so it never saturates (measured:
  // the e4m3 forward 4% faster than with an exact running max).
  static constexpr float kRescale = F8 ? 0.8f : 8.0f;
  static constexpr float kPExp = F8 ? 8.0f : 0.0f;      // P is computed as 2^kPExp exp2(s - m)
  // Chunks of 32 columns of S a softmax thread loads from tensor memory per wait: two in the
  // single mode (measured 2% faster there), one in the pair mode (two measured 1.5% slower).
  static constexpr int kLdBatch = SINGLE ? 2 : 1;
};

struct FwdSmemCtl {
  uint64_t q_full;
  uint64_t k0_full;   // the first key tile (loaded alone, before any stage)
  uint64_t full[4];   // stage landed and P of query tile 0 written (or stood in for)
  uint64_t empty[4];
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  uint32_t vis[2][kVisWords];  // block mask: bit kt of query tile x's word kt / 32 = tile visited
  // Abort-path drain (read only after an abort): per ring buffer the last stage the producer issued
  // into it (-1: none) and whether tile 0's softmax arrives on that stage; per row of query tile 0
  // the last stage its thread arrived on.
  int last_stage[4];
  int last_needs_p0[4];
  int k0_issued;
  int p0_last[128];
};

// One key tile of the online softmax for the query row this thread owns (its tensor-memory
// lane): S is read at tS, O (at tO) is rescaled when the row max grows by more than a factor 2^kRescale,
// P is written over the first columns of S and m, l are updated. With `masked`, the keys at
// columns >= lim are excluded. first: the row's first key tile. Called by whole warps.
template <int D, bool F8, bool SINGLE, typename PreWrite>
__device__ __forceinline__ void softmax_tile(uint32_t tS, uint32_t tO, uint32_t tP, bool masked, int lim, float sl2,
                                             bool first, float& m, float& l, PreWrite&& pre_write) {
  using C = FwdCfg<D, F8, SINGLE>;
  // Columns [32c, 32c + 32) of the row of S: the loads of kLdBatch chunks share one wait.
  uint32_t sr[C::kLdBatch * 32];
  auto chunk = [&](int c, uint32_t(&rr)[32]) {
    constexpr int NB = C::kLdBatch;
    if (c % NB == 0) {
#pragma unroll
      for (int j = 0; j < NB; ++j) tmem_ld32(tS + (c + j) * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + j * 32));
      tmem_ld_wait();
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) rr[i] = sr[(c % NB) * 32 + i];
  };
  // Pass 1: row max of the (masked) scores, 32 columns at a time.
  auto row_max = [&](auto mask_tag) -> float {
    constexpr bool MASK = decltype(mask_tag)::value;
    float pm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t rr[32];
      chunk(c, rr);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float v0 = __uint_as_float(rr[i]), v1 = __uint_as_float(rr[i + 1]);
        if constexpr (MASK) {
          v0 = (c * 32 + i < lim) ? v0 : -INFINITY;
          v1 = (c * 32 + i + 1 < lim) ? v1 : -INFINITY;
        }
        pm[(i >> 1) & 3] = fmax3(pm[(i >> 1) & 3], v0, v1);
      }
    }
    return fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
  };
  const float mx = masked ? row_max(std::true_type{}) : row_max(std::false_type{});
  const float mc = mx * sl2;
  pre_write();  // O and P may be written once the previous P V has completed
  if (first) {
    m = mc;
  } else if (__any_sync(0xffffffffu, mc > m + C::kRescale)) {
    const float mn = fmaxf(m, mc);
    const float alpha = (mn == -INFINITY) ? 1.f : ex2_approx(m - mn);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t rr[32];
      tmem_ld32(tO + c * 32, rr);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
      tmem_st32(tO + c * 32, rr);
    }
    l *= alpha;
    m = mn;
  }
  const float mu = (m == -INFINITY) ? 0.f : m;
  // Pass 2: P = exp2(c log2(e) s - m) over the first columns of S (bf16: 64 columns; e4m3,
  // as 2^8 P: 32 columns; each chunk is written only over columns already read), and the
  // row sum of P.
  auto exp_pass = [&](auto mask_tag) -> float {
    constexpr bool MASK = decltype(mask_tag)::value;
    const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(C::kPExp - mu, C::kPExp - mu);
    float2 ps[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t rr[32];
      chunk(c, rr);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 x = fma2(make_float2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1])), sc2, nm2);
        float p0 = ex2_approx(x.x);
        float p1 = ex2_approx(x.y);
        if constexpr (MASK) {
          p0 = (c * 32 + 2 * i < lim) ? p0 : 0.f;
          p1 = (c * 32 + 2 * i + 1 < lim) ? p1 : 0.f;
        }
        ps[i & 1] = add2(ps[i & 1], make_float2(p0, p1));
        if constexpr (F8) {  // four e4m3 values per column, key 4w + j in byte j of column w
          const uint32_t pair = pack_e4m3x2(p0, p1);
          pk[i >> 1] = (i & 1) ? (pk[i >> 1] | (pair << 16)) : pair;
        } else {
          pk[i] = pack_bf16x2(p0, p1);
        }
      }
      if constexpr (F8) {
        tmem_st8(tP + c * 8, *reinterpret_cast<const uint32_t(*)[8]>(pk));
      } else {
        tmem_st16(tP + c * 16, pk);
      }
    }
    return (ps[0].x + ps[0].y) + (ps[1].x + ps[1].y);
  };
  const float sum = masked ? exp_pass(std::true_type{}) : exp_pass(std::false_type{});
  tmem_st_wait();
  l += sum;
}

// SPLIT: the CTA covers one split of the key tiles and writes fp32 partials (see FaFwdArgs).
// MASKED: a block mask is given (never with SPLIT); without one, visibility is in closed form.
// F8: e4m3 operands (see FwdCfg; never with SPLIT).
// SINGLE: one query tile per CTA (d = 64, and e4m3 at d = 128), small enough that two CTAs share
// an SM: one CTA's softmax runs while the other's products do. A pair of query tiles instead
// walks the union of their key tiles, and under a block mask one tile's softmax is then often idle.
template <int D, bool SPLIT, bool MASKED, bool F8 = false, bool SINGLE = false>
__global__ void __launch_bounds__(SINGLE ? kThreadsSingle : kThreads, SINGLE ? 2 : 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const FaFwdArgs a) {
  using C = FwdCfg<D, F8, SINGLE>;
  grid_dependency_wait();  // launched as a programmatic dependent of the previous kernel
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);                       // Q0, Q1 (later O staging), kQSlot each
  const uint32_t sKV = sQ + C::kTiles * C::kQSlot;         // ring: stage buffer b = V (V^T) then K
  volatile int* abort_flag = &ctl.abort_flag;

  const AttnShape& s = a.s;
  const int BH = s.B * s.H;
  const int npairs = (s.nbq + C::kTiles - 1) / C::kTiles;  // CTAs per head (pairs of query tiles, or tiles)
  const int split = SPLIT ? (int)(blockIdx.x / (npairs * BH)) : 0;  // key range [kt_lo, kt_hi) of this CTA
  const int pidx = (blockIdx.x % (npairs * BH)) / BH;
  const int bh = blockIdx.x % BH;
  const int kt_lo = SPLIT ? split * a.kt_chunk : 0, kt_hi = SPLIT ? kt_lo + a.kt_chunk : s.nbk;
  const int pair = s.causal ? (npairs - 1 - pidx) : pidx;  // longest causal work first
  const int b = bh / s.H, h = bh % s.H;
  const int hk = h / (s.H / s.Hkv);  // K/V head of this query head
  const SeqInfo seq = seq_info(s, b);
  const int qt0 = C::kTiles * pair, qt1 = qt0 + 1;
  if (qt0 * 128 >= seq.Lq) return;  // a packed sequence shorter than the grid's maximum
  const bool has1 = !SINGLE && qt1 * 128 < seq.Lq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Without a block mask a query tile sees exactly the key tiles 0 .. last_kt (the predicate of
  // tile_visited in closed form); with one, each tile is looked up.
  auto last_kt = [&](int qt) -> int {
    if (qt * 128 >= seq.Lq || seq.Lk <= 0) return -1;
    int l = (seq.Lk - 1) / 128;
    if (s.causal) {
      const int key = qt * 128 + 127 + seq.off;
      l = key < 0 ? -1 : min(l, key / 128);
    }
    return l;
  };
  const int lim0 = min(last_kt(qt0), kt_hi - 1), lim1 = has1 ? min(last_kt(qt1), kt_hi - 1) : -1;
  // Key tiles past both query tiles' last visible key tile (or past the split's range) are never
  // visited; scans stop there, and start at the split's first key tile.
  const int kt_end = max(lim0, lim1) + 1;
  // With a block mask the CTA first turns its two mask rows into a bitmap in shared memory, so
  // finding the next visited key tile is a word read and a bit scan instead of one dependent
  // mask load per skipped tile (longer rows than the bitmap holds are looked up tile by tile).
  const bool bitmap = MASKED && kt_end <= 32 * kVisWords;
  auto vis = [&](int x, int kt) -> bool {
    if constexpr (!MASKED) return kt <= (x ? lim1 : lim0);
    if (bitmap) return (ctl.vis[x][kt >> 5] >> (kt & 31)) & 1u;
    return (x == 0 || has1) && tile_visited(s, seq, x ? qt1 : qt0, kt);
  };
  auto next_union = [&](int kt) -> int {
    if (MASKED && bitmap) {
      for (; kt < kt_end; kt = (kt | 31) + 1) {
        const uint32_t m = (ctl.vis[0][kt >> 5] | ctl.vis[1][kt >> 5]) >> (kt & 31);
        if (m) return kt + __ffs(m) - 1;
      }
      return s.nbk;
    }
    for (; kt < kt_end; ++kt)
      if (vis(0, kt) || vis(1, kt)) return kt;
    return s.nbk;
  };
  // The same scan, also reporting which query tiles see the key tile found (for the issuer, whose
  // every instruction between MMA groups is time the tensor pipe idles).
  auto next_union_vis = [&](int kt, bool& v0, bool& v1) -> int {
    if (MASKED && bitmap) {
      kt = next_union(kt);
      v0 = kt < s.nbk && vis(0, kt);
      v1 = kt < s.nbk && vis(1, kt);
      return kt;
    }
    for (; kt < kt_end; ++kt) {
      v0 = vis(0, kt);
      v1 = vis(1, kt);
      if (v0 || v1) return kt;
    }
    v0 = v1 = false;
    return s.nbk;
  };

  const uint32_t b_q = smem_u32(&ctl.q_full), b_k0 = smem_u32(&ctl.k0_full);
  auto b_full = [&](int i) { return smem_u32(&ctl.full[i]); };
  auto sV = [&](int b) { return sKV + (2 * b) * C::kTileBytes; };
  auto sK = [&](int b) { return sKV + (2 * b + 1) * C::kTileBytes; };
  auto b_empty = [&](int i) { return smem_u32(&ctl.empty[i]); };
  const uint32_t b_sfull[2] = {smem_u32(&ctl.s_full[0]), smem_u32(&ctl.s_full[1])};
  const uint32_t b_pready[2] = {smem_u32(&ctl.p_ready[0]), smem_u32(&ctl.p_ready[1])};
  const uint32_t b_odone[2] = {smem_u32(&ctl.o_done[0]), smem_u32(&ctl.o_done[1])};

  // The producer's first copies: Q0, Q1 and the first key tile alone, into the K half of the last
  // buffer. Without a block mask the first key tile is known before the CTA-wide barrier, so they
  // are issued right after the barrier set-up and their latency overlaps the rest of the prologue.
  // The query tiles' copy does not depend on the mask: with one it is issued before the bitmap is
  // built, and only the first K copy waits for the bitmap.
  auto load_q = [&]() {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    mbar_expect_tx(b_q, (has1 ? 2 : 1) * C::kTileBytes);
    for (int x = 0; x < (has1 ? 2 : 1); ++x)
      for (int c = 0; c < C::kBoxes; ++c)
        tma_load_4d(sQ + x * C::kQSlot + c * 16384, &tmQ, c * C::kBoxCols, seq.q0 + (x ? qt1 : qt0) * 128, h, seq.bb,
                    b_q);
  };
  auto load_k0 = [&]() {
    const int kt = next_union(kt_lo);
#ifndef FA_TEST_WITHHOLD_KV
    if (kt < s.nbk) {
      mbar_expect_tx(b_k0, C::kTileBytes);
      for (int c = 0; c < C::kBoxes; ++c)
        tma_load_4d(sK(C::kStages - 1) + c * 16384, &tmK, c * C::kBoxCols, seq.k0 + kt * 128, hk, seq.bb, b_k0);
      ctl.k0_issued = 1;
    }
#endif
  };
  if (threadIdx.x < 4) ctl.last_stage[threadIdx.x] = -1;
  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    ctl.k0_issued = 0;
    mbar_init(b_q, 1);
    mbar_init(b_k0, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(b_full(i), 1 + 128);  // the producer's arrival with the byte count, tile 0's softmax
      mbar_init(b_empty(i), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(b_sfull[x], 1);
      mbar_init(b_pready[x], (C::kSepP && x == 1) ? 1 : 128);  // sepP: [1] = P V of tile 0 complete
      mbar_init(b_odone[x], 1);
    }
    mbar_init(smem_u32(&ctl.drain), 1);
    fence_mbar_init();
    load_q();  // thread 0 is the producer
    if constexpr (!MASKED) load_k0();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  if (MASKED && bitmap) {  // one vote per 32 key tiles of a query tile; only [kt_lo, kt_end) is ever read
    // Items (query tile x, word wd) are dealt to the warps; without a second query tile its row is
    // all zeros and takes no warp's turn, so no warp waits on two mask loads in a row.
    const int words = (kt_end + 31) >> 5;
    const int nx = has1 ? 2 : 1;
    if (!has1 && warp == 0) {
      for (int wd = lane; wd < words; wd += 32) ctl.vis[1][wd] = 0u;
    }
    for (int idx = warp; idx < nx * words; idx += C::kThreadsCta / 32) {
      const int x = idx % nx, wd = idx / nx, kt = wd * 32 + lane;
      const bool bit = kt >= kt_lo && kt < kt_end && tile_visited(s, seq, x ? qt1 : qt0, kt);
      const uint32_t m = __ballot_sync(0xffffffffu, bit);
      if (lane == 0) ctl.vis[x][wd] = m;
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      if constexpr (MASKED) load_k0();
      // Stage t (the t-th key tile u_t the pair visits) lands V_{u_t} and K_{u_t+1} in buffer
      // t % kStages. A buffer is reloaded once the MMAs of its previous stage have completed. No
      // copy is issued after an abort; the copies already issued are drained at the CTA's exit.
      int kt = next_union(kt_lo);
      for (int t = 0; kt < s.nbk; ++t) {
        const int b = t % C::kStages;
        const int ktn = next_union(kt + 1);
        const int uses = t / C::kStages + (b == C::kStages - 1 ? 1 : 0);  // earlier users of buffer b
        // FA_TEST_WITHHOLD_KV (a test-only build) never loads K/V, so every consumer's bounded
        // wait must run out and the kernel must return FA_ERR_DEVICE_TIMEOUT cleanly.
#ifndef FA_TEST_WITHHOLD_KV
        // Besides the release, the buffer's previous stage barrier phase must have completed (in the
        // normal path long since: the issuer waited for it before releasing the buffer), so a stage
        // barrier never gets a second arrive.expect_tx while a phase is open.
        if ((uses == 0 || mbar_wait(b_empty(b), (uses - 1) & 1, abort_flag, a.status)) &&
            (t < C::kStages || mbar_wait(b_full(b), ((t - C::kStages) / C::kStages) & 1, abort_flag, a.status)) &&
            !*abort_flag) {
#else
        if (false) {
#endif
          mbar_expect_tx(b_full(b), (ktn < s.nbk ? 2 : 1) * C::kTileBytes);
          if constexpr (F8) {  // V^T: rows are the d dimensions, keys along the row
            tma_load_4d(sV(b), &tmV, kt * 128, 0, hk, seq.bb, b_full(b));
          } else {
            for (int c = 0; c < C::kBoxes; ++c)
              tma_load_4d(sV(b) + c * 16384, &tmV, c * 64, seq.k0 + kt * 128, hk, seq.bb, b_full(b));
          }
          if (ktn < s.nbk)
            for (int c = 0; c < C::kBoxes; ++c)
              tma_load_4d(sK(b) + c * 16384, &tmK, c * C::kBoxCols, seq.k0 + ktn * 128, hk, seq.bb, b_full(b));
          const bool p0 = vis(0, kt);
          if (!p0) mbar_arrive_cnt(b_full(b), 128);  // tile 0 has no P for this key tile
          ctl.last_stage[b] = t;
          ctl.last_needs_p0[b] = p0;
        }
        kt = ktn;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool first[2] = {true, true};
      bool any[2] = {false, false};
      uint32_t np[2] = {0, 0};
      // No abort-flag reads on the issue path (see mbar_wait): after an abort the remaining MMAs
      // run on stale data and complete normally.
      // Descriptors are built once per operand tile and advanced by constant byte offsets per k-step.
      const uint64_t dQ[2] = {desc_kmajor_sw128(sQ), desc_kmajor_sw128(sQ + C::kQSlot)};
      // Each K step is 32 bytes of the 128-byte rows (16 bf16 or 32 e4m3 elements).
      auto issue_s = [&](int x, uint32_t ka) {
        const uint64_t dq = dQ[x], dk = desc_kmajor_sw128(ka);
#pragma unroll
        for (int kk = 0; kk < C::kSSteps; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if constexpr (F8)
            mma_ss_f8(tmem + C::kTmemS0 + x * 128, desc_add(dq, off), desc_add(dk, off), C::kIdS, kk > 0);
          else
            mma_ss(tmem + C::kTmemS0 + x * 128, desc_add(dq, off), desc_add(dk, off), C::kIdS, kk > 0);
        }
        mma_commit(b_sfull[x]);
      };
      // P (8 tensor-memory columns per K step) times V: bf16 V is MN-major (d contiguous); e4m3 V^T
      // is K-major (keys contiguous).
      auto issue_pv = [&](int x, uint32_t va) {
        const uint64_t dv = F8 ? desc_kmajor_sw128(va) : desc_mnmajor_sw128(va, 16384);
#pragma unroll
        for (int kk = 0; kk < C::kPVSteps; ++kk) {
          if constexpr (F8)
            mma_ts_f8(tmem + C::kTmemO0 + x * D, tmem + C::kTmemP0 + x * 128 + kk * 8, desc_add(dv, kk * 32),
                      C::kIdPV, (first[x] && kk == 0) ? 0u : 1u);
          else
            mma_ts(tmem + C::kTmemO0 + x * D, tmem + C::kTmemP0 + x * 128 + kk * 8, desc_add(dv, kk * 2048),
                   C::kIdPV, (first[x] && kk == 0) ? 0u : 1u);
        }
        first[x] = false;
      };

      // Per key tile two waits: the stage barrier (V_t and K_t+1 landed, P0 written) and P1.
      // After its first wait that fails (a timeout, or the CTA's abort flag) the issuer issues no
      // MMA and no commit: a buffer release committed for a stage it did not see land would let
      // the producer reload the buffer while a copy into it is still in flight.
      bool run = mbar_wait_spin(b_q, 0, abort_flag, a.status);
      bool v0, v1;  // which query tiles see key tile kt
      int kt = next_union_vis(kt_lo, v0, v1);
      if (kt < s.nbk && run) {
        run = mbar_wait_spin(b_k0, 0, abort_flag, a.status);
        fence_after_sync();
        if (run) {
          if (v0) issue_s(0, sK(C::kStages - 1));
          if (v1) issue_s(1, sK(C::kStages - 1));
          any[0] = v0;
          any[1] = v1;
          mma_commit(b_empty(C::kStages - 1));
        }
        for (int t = 0; run; ++t) {
          const int b = t % C::kStages;
          bool n0, n1;
          const int ktn = next_union_vis(kt + 1, n0, n1);  // n0 = n1 = false past the last tile
          run = mbar_wait_spin(b_full(b), (t / C::kStages) & 1, abort_flag, a.status);
          fence_after_sync();
          if (!run) break;
          if constexpr (C::kSepP) {  // the next S first: the softmax has read this S (P is written)
            if (n0) {
              issue_s(0, sK(b));
              any[0] = true;
            }
            if (v0) {
              issue_pv(0, sV(b));
              mma_commit(b_pready[1]);  // this P V has read P and updated O
            }
          } else {
          if (v0) issue_pv(0, sV(b));
          if (n0) {
            issue_s(0, sK(b));
            any[0] = true;
          }
          }
          if (v1) {
            run = mbar_wait_spin(b_pready[1], np[1] & 1, abort_flag, a.status);
            ++np[1];
            fence_after_sync();
            if (!run) break;
            issue_pv(1, sV(b));
          }
          if (n1) {
            issue_s(1, sK(b));
            any[1] = true;
          }
          mma_commit(b_empty(b));
          if (ktn >= s.nbk) break;
          kt = ktn;
          v0 = n0;
          v1 = n1;
        }
      }
      for (int x = 0; x < 2; ++x)
        if (any[x] && run) mma_commit(b_odone[x]);
      mma_commit(smem_u32(&ctl.drain));  // every MMA of this CTA has finished when this arrives
      mbar_wait_drain(smem_u32(&ctl.drain), 0);
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int x = (warp - 2) >> 2;
    const bool active = (x == 0) || has1;
    const int qt = x ? qt1 : qt0;
    const int quad = warp & 3;                    // tensor-memory lane quadrant of this warp
    const int r = quad * 32 + lane;               // row within the tile
    const int row = qt * 128 + r;                 // row within the head
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kTmemS0 + x * 128;
    const uint32_t tO = tmem + lane_off + C::kTmemO0 + x * D;
    const uint32_t tP = tmem + lane_off + C::kTmemP0 + x * 128;
    // e4m3 operands: the per-head descales of Q and K enter the scores, V's the output.
    const float qk_descale = F8 ? a.q_descale[(size_t)b * s.H + h] * a.k_descale[(size_t)b * s.Hkv + hk] : 1.f;
    const float sl2 = a.scale * kLog2e * qk_descale;
    float m = -INFINITY, l = 0.f;  // l: row sum of 2^kPExp exp2(s - m)
    int cnt = 0;
    // After its first wait that fails, a thread makes no more arrivals; its warp keeps the same
    // control flow (the tensor-memory accesses are warp-collective). Tile 0's threads record the
    // last stage they arrived on, for the producer's drain at exit.
    bool run = mbar_wait(b_q, 0, abort_flag, a.status);
    if (x == 0) ctl.p0_last[r] = -1;
    if (active) {
      int t = -1;  // union index of the key tile (tile 0 reports P on stage t's barrier)
      for (int kt = next_union(kt_lo); kt < s.nbk; kt = next_union(kt + 1)) {
        ++t;
        if (!vis(x, kt)) continue;
        if (run) run = mbar_wait(b_sfull[x], cnt & 1, abort_flag, a.status);
        fence_after_sync();
        const int k0 = kt * 128;
        const bool masked = (s.causal && k0 + 127 > qt * 128 + seq.off) || k0 + 128 > seq.Lk;
        const int lim = min(seq.Lk - k0, s.causal ? row + seq.off - k0 + 1 : 128);  // keys [k0, k0 + lim) valid
        softmax_tile<D, F8, SINGLE>(tS, tO, tP, masked, lim, sl2, cnt == 0, m, l, [&]() {
          if constexpr (C::kSepP) {
            if (cnt > 0) {  // the previous tile's P V has completed (it reads P, writes O)
              if (run) run = mbar_wait(b_pready[1], (cnt - 1) & 1, abort_flag, a.status);
              fence_after_sync();
            }
          }
        });
        fence_before_sync();
        if (run) {
          mbar_arrive(x == 0 ? b_full(t % C::kStages) : b_pready[1]);
          if (x == 0) ctl.p0_last[r] = t;
        }
        ++cnt;
      }
      // ---------------------------------------------------------------- epilogue
      if (cnt > 0) {
        if (run) run = mbar_wait(b_odone[x], 0, abort_flag, a.status);
        fence_after_sync();
      }
      // l sums 2^kPExp exp2(s - m); with e4m3 operands V's descale scales the output.
      const float inv = l > 0.f ? (F8 ? a.v_descale[(size_t)b * s.Hkv + hk] : 1.f) / l : 0.f;
      const float lse2 = l > 0.f ? m + log2f(l) - C::kPExp : -INFINITY;  // log2-domain LSE
      if constexpr (SPLIT) {  // split over keys: normalised fp32 partials for the merge pass
        // The tensor-memory loads are warp-collective: every lane loads, only valid rows store.
        const bool live = row < seq.Lq;
        const size_t R = (size_t)split * a.part_rows + row_base(s, seq, b, h) + row;
        float* po = a.part_o + R * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          if (cnt > 0) {
            tmem_ld32(tO + c * 32, rr);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = 0u;
          }
          if (live) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(po + c * 32 + i) =
                  make_float4(__uint_as_float(rr[i]) * inv, __uint_as_float(rr[i + 1]) * inv,
                              __uint_as_float(rr[i + 2]) * inv, __uint_as_float(rr[i + 3]) * inv);
          }
        }
        if (live) a.part_lse[R] = lse2 * kLn2;
        // The merge pass may be scheduled now; it still waits for this grid to complete.
        asm volatile("griddepcontrol.launch_dependents;");
      } else {
        const uint32_t stg = sQ + x * C::kQSlot;
        // A packed sequence's last tile is stored row by row: a tile-wide copy would write the next
        // sequence's rows.
        const bool direct = s.cu_q != nullptr && qt * 128 + 128 > seq.Lq;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + elem_offset(a.so, seq.bb, seq.q0 + row, h);
  #pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          if (cnt > 0) {
            tmem_ld32(tO + c * 32, rr);
            tmem_ld_wait();
          } else {
  #pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = 0u;
          }
          uint32_t pk[16];
  #pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv);
          if (direct) {
            if (row < seq.Lq) {
  #pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(orow + c * 32 + j * 8) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
            continue;
          }
          const uint32_t box = stg + (c >> 1) * 16384 + r * 128;
  #pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int chunk = (c & 1) * 4 + j;
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(box + ((chunk ^ (r & 7)) << 4)), "r"(pk[4 * j]),
                         "r"(pk[4 * j + 1]), "r"(pk[4 * j + 2]), "r"(pk[4 * j + 3])
                         : "memory");
          }
        }
        if (row < seq.Lq) a.lse[row_base(s, seq, b, h) + row] = lse2 * kLn2;
        fence_proxy_async_smem();
        named_bar_sync(1 + x, 128);
        if (warp == 2 + 4 * x && lane == 0) {
          if (!direct)
            for (int c = 0; c < C::kOBoxes; ++c) tma_store_4d(&tmO, stg + c * 16384, c * 64, seq.q0 + qt * 128, h, seq.bb);
          tma_store_commit();
          tma_store_wait_read0();  // the staging is read; the writes land before the grid completes
          if (a.tile_visits != nullptr) a.tile_visits[(size_t)bh * s.nbq + qt] = cnt;
        }
      }  // normal epilogue
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) {
    // Every role has finished, so no arrival is still to come: let the copies still in flight
    // land before the CTA exits. A buffer is reloaded only after the issuer released it, which it
    // does only for a stage it saw complete (a role issues and arrives only while all its waits
    // have succeeded), so each stage barrier has at most one phase in flight, the last one issued.
    // That phase also counts tile 0's 128 softmax arrivals: the ones that will never come are made
    // here (a thread arrived on stage t iff its last arrival was on a stage >= t, since threads
    // arrive in stage order and stop at their first failed wait), then the copies' bytes
    // complete the phase.
    mbar_wait_drain(b_q, 0);
    if (ctl.k0_issued) mbar_wait_drain(b_k0, 0);
    for (int b = 0; b < C::kStages; ++b) {
      const int t = ctl.last_stage[b];
      if (t < 0) continue;
      const uint32_t par = (t / C::kStages) & 1;
      if (mbar_test(b_full(b), par)) continue;
      if (ctl.last_needs_p0[b]) {
        int arrived = 0;
        for (int i = 0; i < 128; ++i) arrived += ctl.p0_last[i] >= t;
        if (arrived < 128) mbar_arrive_cnt(b_full(b), 128 - arrived);
      }
      mbar_wait_drain(b_full(b), par);
    }
  }
}


template <int D>
cudaError_t launch(const FaFwdArgs& a, cudaStream_t st) {
  using C = FwdCfg<D>;
  const AttnShape& s = a.s;
  const bool packed = s.cu_q != nullptr;
  const int rq = packed ? s.rows_q : s.Nq, rk = packed ? s.rows_k : s.Nk, nbatch = packed ? 1 : s.B;
  CUtensorMap tq, tk, tv, to;
  if (!fa_make_tmap_bf16(&tq, a.q, D, rq, s.H, nbatch, a.sq.row, a.sq.head, a.sq.batch) ||
      !fa_make_tmap_bf16(&tk, a.k, D, rk, s.Hkv, nbatch, a.sk.row, a.sk.head, a.sk.batch) ||
      !fa_make_tmap_bf16(&tv, a.v, D, rk, s.Hkv, nbatch, a.sv.row, a.sv.head, a.sv.batch) ||
      // (the partial pass writes no O; its map is then built over Q and never used)
      !fa_make_tmap_bf16(&to, a.o ? a.o : a.q, D, rq, s.H, nbatch, a.o ? a.so.row : a.sq.row,
                         a.o ? a.so.head : a.sq.head, a.o ? a.so.batch : a.sq.batch))
    return cudaErrorInvalidValue;
  const int BH = s.B * s.H;
  const bool split = a.part_o != nullptr;
  if (split && s.block_mask != nullptr) return cudaErrorInvalidValue;  // no split path takes a mask
  // A split over keys with one query tile per (batch, head) (decode shapes): the single mode, two
  // CTAs per SM, instead of a pair whose second tile would be empty (measured on the decode shape:
  // 4.73 TB/s of K/V read at 4 splits against 4.42 at the pair's best count; without a split the
  // pair's two-stage ring stays ahead, and so it does for one split: 64 CTAs, 2.7 against 2.2).
  if (split && s.nbq == 1 && a.splits > 1) {
    using CS = FwdCfg<D, false, true>;
    auto ks = fwd_tc_kernel<D, true, false, false, true>;
    cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, CS::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(ks, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)BH * a.splits;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_dependent(ks, dim3((unsigned)grid), dim3(CS::kThreadsCta), CS::kSmem, st, tq, tk, tv, to, a);
  }
  // d = 64 without a split: one query tile per CTA, two CTAs per SM (measured faster than the pair
  // of query tiles on block-sparse and causal problems, equal on the rest).
  if constexpr (D == 64) {
    if (!split) {
      using CS = FwdCfg<D, false, true>;
      auto ks = s.block_mask != nullptr ? fwd_tc_kernel<D, false, true, false, true>
                                        : fwd_tc_kernel<D, false, false, false, true>;
      cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, CS::kSmem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(ks, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return e;
      const long long grid = (long long)s.nbq * BH;
      if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
      return launch_dependent(ks, dim3((unsigned)grid), dim3(CS::kThreadsCta), CS::kSmem, st, tq, tk, tv, to, a);
    }
  }
  auto kern = split ? fwd_tc_kernel<D, true, false>
                    : (s.block_mask != nullptr ? fwd_tc_kernel<D, false, true> : fwd_tc_kernel<D, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)((s.nbq + 1) / 2) * BH * (split ? a.splits : 1);
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_dependent(kern, dim3((unsigned)grid), dim3(kThreads), C::kSmem, st, tq, tk, tv, to, a);
}

// e4m3 operands (d = 128, fixed-length [B, H, N, d] Q and K, [B, Hkv, d, N] V^T, no split). The
// 8-bit operand tiles are small enough for the single mode (one query tile per CTA, a 2-stage
// ring, 97 KB of shared memory): two CTAs share an SM and hide each other's softmax.
cudaError_t launch_f8(const FaFwdArgs& a, cudaStream_t st) {
  constexpr int D = 128;
  using C = FwdCfg<D, true, true>;
  const AttnShape& s = a.s;
  if (s.cu_q != nullptr || a.part_o != nullptr || s.d != D) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv, to;
  const long long nq = s.Nq, nk = s.Nk;
  if (!fa_make_tmap_u8(&tq, a.q, D, s.Nq, s.H, s.B, D, nq * D, (long long)s.H * nq * D, 128, 128) ||
      !fa_make_tmap_u8(&tk, a.k, D, s.Nk, s.Hkv, s.B, D, nk * D, (long long)s.Hkv * nk * D, 128, 128) ||
      !fa_make_tmap_u8(&tv, a.v, s.Nk, D, s.Hkv, s.B, nk, nk * D, (long long)s.Hkv * nk * D, 128, 128) ||
      !fa_make_tmap_bf16(&to, a.o, D, s.Nq, s.H, s.B, a.so.row, a.so.head, a.so.batch))
    return cudaErrorInvalidValue;
  auto kern = s.block_mask != nullptr ? fwd_tc_kernel<D, false, true, true, true>
                                      : fwd_tc_kernel<D, false, false, true, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)s.nbq * s.B * s.H;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_dependent(kern, dim3((unsigned)grid), dim3(C::kThreadsCta), C::kSmem, st, tq, tk, tv, to, a);
}

}  // namespace
}  // namespace fa

cudaError_t fa_launch_fwd(const FaFwdArgs& a, cudaStream_t st) {
  if (a.fp8) return fa::launch_f8(a, st);
  return a.s.d == 64 ? fa::launch<64>(a, st) : fa::launch<128>(a, st);
}

namespace fa {
namespace {

// Merge of the split partials (one warp per query row): with M = max_s LSE_s and
// w_s = exp(LSE_s - M), O = sum_s w_s O_s / sum_s w_s and LSE = M + ln sum_s w_s; a row with no
// visible key in any split gets O = 0 and LSE = -inf.
template <int D>
__global__ void __launch_bounds__(256) splitkv_merge_kernel(const FaFwdArgs a) {
  // Launched as a programmatic dependent of the split pass: wait until that grid has completed and
  // its partials are visible (no effect when launched without the dependency).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int PER = D / 32;
  const AttnShape& s = a.s;
  const size_t rows = (size_t)s.B * s.H * s.Nq;  // (b, h, i) with i below the longest length
  const int lane = threadIdx.x & 31;
  const size_t warp0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
  for (size_t w = warp0; w < rows; w += nwarps) {
    const int i = (int)(w % s.Nq);
    const int h = (int)((w / s.Nq) % s.H);
    const int b = (int)(w / ((size_t)s.Nq * s.H));
    const SeqInfo seq = seq_info(s, b);
    if (i >= seq.Lq) continue;
    const size_t R = row_base(s, seq, b, h) + i;
    float M = -INFINITY;
    for (int sp = 0; sp < a.splits; ++sp) M = fmaxf(M, a.part_lse[(size_t)sp * a.part_rows + R]);
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float W = 0.f;
    if (M != -INFINITY) {
      for (int sp = 0; sp < a.splits; ++sp) {
        const size_t P = (size_t)sp * a.part_rows + R;
        const float wt = expf(a.part_lse[P] - M);
        W += wt;
        const float* po = a.part_o + P * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] += wt * po[e];
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o) + elem_offset(a.so, seq.bb, seq.q0 + i, h) + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2)
      *reinterpret_cast<uint32_t*>(out + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0) a.lse[R] = W > 0.f ? M + logf(W) : -INFINITY;
  }
}

}  // namespace
}  // namespace fa

namespace fa {
namespace {

// acc <- merge(acc, part) for every row of the partial layout (one warp per row):
// M = max(L_a, L_p), w = exp(L - M), O = (w_a O_a + w_p O_p) / (w_a + w_p), L = M + ln(w_a + w_p).
template <int D>
__global__ void __launch_bounds__(256) merge_two_kernel(float* acc_o, float* acc_lse, const float* part_o,
                                                        const float* part_lse, size_t rows) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const size_t warp0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
  for (size_t r = warp0; r < rows; r += nwarps) {
    const float la = acc_lse[r], lp = part_lse[r];
    const float M = fmaxf(la, lp);
    if (M == -INFINITY) continue;  // neither saw a key: stays O = 0, LSE = -inf
    const float wa = la == -INFINITY ? 0.f : expf(la - M), wp = lp == -INFINITY ? 0.f : expf(lp - M);
    const float inv = 1.f / (wa + wp);
    float* oa = acc_o + r * D + lane * PER;
    const float* op = part_o + r * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) oa[e] = (wa * oa[e] + wp * op[e]) * inv;
    if (lane == 0) acc_lse[r] = M + logf(wa + wp);
  }
}

}  // namespace
}  // namespace fa

cudaError_t fa_launch_merge_two(float* acc_o, float* acc_lse, const float* part_o, const float* part_lse, size_t rows,
                                int d, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (d == 64)
    fa::merge_two_kernel<64><<<sms * 4, 256, 0, st>>>(acc_o, acc_lse, part_o, part_lse, rows);
  else
    fa::merge_two_kernel<128><<<sms * 4, 256, 0, st>>>(acc_o, acc_lse, part_o, part_lse, rows);
  return cudaGetLastError();
}

cudaError_t fa_launch_splitkv_merge(const FaFwdArgs& a, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // One warp per row. A programmatic dependent launch: the merge's CTAs are scheduled while the
  // split pass's last CTAs finish (decode shape: 55.2 -> 52.6 us per split + merge).
  const long long rows = (long long)a.s.B * a.s.H * a.s.Nq;
  long long ctas = (rows + 7) / 8;
  if (ctas > (long long)sms * 4) ctas = (long long)sms * 4;
  if (ctas < 1) ctas = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.s.d == 64) return cudaLaunchKernelEx(&cfg, fa::splitkv_merge_kernel<64>, a);
  return cudaLaunchKernelEx(&cfg, fa::splitkv_merge_kernel<128>, a);
}
