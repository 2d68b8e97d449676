// C ABI of the attention library: argument validation, workspace layout and kernel launches.
// Every check runs on the host before any CUDA call, so invalid arguments never reach a GPU.
#include <math.h>

#include "fa_common.cuh"

namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Tensors are limited to 2^31 elements (int element offsets inside the kernels' tile math).
constexpr double kMaxElems = 2147483648.0;
constexpr int kMaxSplits = 256;  // splits over keys in fa_fwd_splitkv

int check_common(int B, int H, int Hkv, int d, int causal, float scale) {
  if (B < 1 || H < 1) return FA_ERR_INVALID_ARG;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int check_shape(int B, int H, int N, int d, int causal, float scale) {
  if (N < 1) return FA_ERR_INVALID_ARG;
  const int rc = check_common(B, H, H, d, causal, scale);
  if (rc != FA_OK) return rc;
  if ((double)B * H * N * d >= kMaxElems) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

FaStrides contiguous(int heads, int N, int d) {
  FaStrides t;
  t.row = d;
  t.head = (long long)N * d;
  t.batch = (long long)heads * N * d;
  return t;
}

fa::AttnShape fixed_shape(int B, int H, int Hkv, int N, int d, int causal, const uint8_t* bm, const int32_t* sl) {
  fa::AttnShape s{};
  s.B = B;
  s.H = H;
  s.Hkv = Hkv;
  s.d = d;
  s.Nq = s.Nk = N;
  s.nbq = s.nbk = (N + fa::kTile - 1) / fa::kTile;
  s.causal = causal;
  s.block_mask = bm;
  s.seqlens_k = sl;
  return s;
}

// Varlen problem -> shape; FA_OK or an error code.
int varlen_shape(const fa_varlen_problem* p, fa::AttnShape* out) {
  if (p == nullptr) return FA_ERR_INVALID_ARG;
  const int rc = check_common(p->B, p->H, p->Hkv, p->d, p->causal, p->scale);
  if (rc != FA_OK) return rc;
  if (p->seqlen_q < 1 || p->seqlen_k < 1) return FA_ERR_INVALID_ARG;
  const bool packed = p->cu_seqlens_q != nullptr;
  if (packed != (p->cu_seqlens_k != nullptr)) return FA_ERR_INVALID_ARG;
  if (packed && (p->rows_q < 1 || p->rows_k < 1)) return FA_ERR_INVALID_ARG;
  if (!aligned(p->cu_seqlens_q, 4) || !aligned(p->cu_seqlens_k, 4)) return FA_ERR_MISALIGNED;
  fa::AttnShape s{};
  s.B = p->B;
  s.H = p->H;
  s.Hkv = p->Hkv;
  s.d = p->d;
  s.Nq = p->seqlen_q;
  s.Nk = p->seqlen_k;
  s.nbq = (s.Nq + fa::kTile - 1) / fa::kTile;
  s.nbk = (s.Nk + fa::kTile - 1) / fa::kTile;
  s.causal = p->causal;
  s.cu_q = p->cu_seqlens_q;
  s.cu_k = p->cu_seqlens_k;
  s.rows_q = packed ? p->rows_q : 0;
  s.rows_k = packed ? p->rows_k : 0;
  const double rq = packed ? (double)p->rows_q : (double)p->B * p->seqlen_q;
  const double rk = packed ? (double)p->rows_k : (double)p->B * p->seqlen_k;
  if (rq * p->H * p->d >= kMaxElems || rk * p->Hkv * p->d >= kMaxElems) return FA_ERR_UNSUPPORTED;
  *out = s;
  return FA_OK;
}

// Strides of a caller tensor: positive multiples of 8 elements (16 bytes, the TMA rule); the
// batch stride is unused (and replaced by a valid one) for packed batches and single sequences.
int take_strides(const fa_strides& in, bool packed, int B, int rows, int heads, FaStrides* out) {
  if (in.row <= 0 || in.head <= 0 || in.row % 8 || in.head % 8) return FA_ERR_INVALID_ARG;
  FaStrides t;
  t.row = in.row;
  t.head = in.head;
  t.batch = in.batch;
  if (packed || B == 1) {
    const long long span = (long long)in.row * rows + (long long)in.head * heads;
    t.batch = (span + 7) / 8 * 8;
  } else if (in.batch <= 0 || in.batch % 8) {
    return FA_ERR_INVALID_ARG;
  }
  *out = t;
  return FA_OK;
}

size_t per_row(const fa::AttnShape& s) { return s.cu_q != nullptr ? (size_t)s.H * s.rows_q : (size_t)s.B * s.H * s.Nq; }

// Backward workspace: D, the fp32 dQ accumulator, then one aligned block holding the main kernel's
// key-tile counter.
size_t workspace_for(const fa::AttnShape& s) {
  const size_t rows = per_row(s);
  return round_up(rows * sizeof(float)) + round_up(rows * s.d * sizeof(float)) + kAlign;
}

// The masks and sequence arrays are read by the kernels, so they must be device-accessible
// (device, managed, or mapped host memory). A plain host array would fault the kernel; it is
// rejected here instead, after every other check, with FA_ERR_INVALID_ARG.
bool device_accessible(const void* p) {
  if (p == nullptr) return true;
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged ||
         (attr.type == cudaMemoryTypeHost && attr.devicePointer != nullptr);
}
bool aux_on_device(const fa::AttnShape& s) {
  return device_accessible(s.block_mask) && device_accessible(s.seqlens_k) && device_accessible(s.cu_q) &&
         device_accessible(s.cu_k);
}

// Decode with grouped K/V heads: one query row per head (fixed length, no block mask). The G query
// heads of a K/V head are viewed as G query rows of one head: the head stride becomes the row stride
// (the row stride is unused with one row), so one query tile carries all G and each K/V tile is
// streamed once for them instead of G times. A single query row sees every key under the
// bottom-right causal reading, so the view is non-causal. Its LSE and per-row order, [B][Hkv][G],
// is the problem's [B][H] for one row, so outputs, partials and merges are unchanged.
bool decode_view(fa::AttnShape& s, FaStrides* sq, FaStrides* so) {
  if (s.cu_q != nullptr || s.Nq != 1 || s.H == s.Hkv || s.block_mask != nullptr) return false;
  const int G = s.H / s.Hkv;
  for (FaStrides* t : {sq, so})
    if (t != nullptr) {
      t->row = t->head;
      t->head *= G;
    }
  s.H = s.Hkv;
  s.Nq = G;
  s.nbq = (G + fa::kTile - 1) / fa::kTile;
  s.causal = 0;
  return true;
}

int launch_fwd(fa::AttnShape s, const void* q, FaStrides sq, const void* k, FaStrides sk, const void* v,
               FaStrides sv, void* o, FaStrides so, float* lse, float scale, int32_t* tile_visits, int* dev_status,
               void* stream) {
  if (tile_visits == nullptr) decode_view(s, &sq, &so);  // (tile visits are recorded per query head)
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(tile_visits, 4) || !aligned(dev_status, 4))
    return FA_ERR_MISALIGNED;
  if (!aux_on_device(s)) return FA_ERR_INVALID_ARG;
  FaFwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.so = so;
  a.s = s;
  a.scale = scale;
  a.tile_visits = tile_visits;
  a.status = dev_status;
  a.splits = 1;
  a.kt_chunk = s.nbk;
  a.part_o = a.part_lse = nullptr;
  a.part_rows = 0;
  const cudaError_t e = fa_launch_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Split over keys: partial launches then the merge; workspace = partial LSE, then partial O.
size_t splitkv_bytes(const fa::AttnShape& s, int splits) {
  const size_t rows = per_row(s) * (size_t)splits;
  return round_up(rows * sizeof(float)) + round_up(rows * s.d * sizeof(float));
}

struct BwdTensors {
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;  // bf16 outputs, or (accumulate) the fp32 accumulators
  FaStrides sq, sk, sv, so, sdo, sdq, sdk, sdv;
  bool accumulate = false;
};

int launch_bwd(const fa::AttnShape& s, const BwdTensors& t, float scale, void* workspace, size_t workspace_bytes,
               int* dev_status, void* stream, const fa_bwd_extras* extras = nullptr) {
  if (!t.q || !t.k || !t.v || !t.o || !t.dout || !t.lse || !t.dq || !t.dk || !t.dv || !workspace)
    return FA_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_for(s)) return FA_ERR_INVALID_ARG;
  if (!aligned(t.q, 16) || !aligned(t.k, 16) || !aligned(t.v, 16) || !aligned(t.o, 16) || !aligned(t.dout, 16) ||
      !aligned(t.dq, 16) || !aligned(t.dk, 16) || !aligned(t.dv, 16) || !aligned(t.lse, 4) ||
      !aligned(workspace, kAlign) || !aligned(dev_status, 4) || (extras && !aligned(extras->step_visits, 4)))
    return FA_ERR_MISALIGNED;
  if (!aux_on_device(s)) return FA_ERR_INVALID_ARG;
  FaBwdArgs a{};
  a.q = t.q;
  a.k = t.k;
  a.v = t.v;
  a.o = t.o;
  a.dout = t.dout;
  a.lse = t.lse;
  a.dq = t.dq;
  a.dk = t.dk;
  a.dv = t.dv;
  a.sq = t.sq;
  a.sk = t.sk;
  a.sv = t.sv;
  a.so = t.so;
  a.sdo = t.sdo;
  a.sdq = t.sdq;
  a.sdk = t.sdk;
  a.sdv = t.sdv;
  const size_t rows = per_row(s);
  a.dvec = static_cast<float*>(workspace);
  a.dqacc = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(rows * sizeof(float)));
  a.tile_counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + round_up(rows * sizeof(float)) +
                                          round_up(rows * s.d * sizeof(float)));
  a.s = s;
  a.scale = scale;
  a.status = dev_status;
  if (t.accumulate) {
    a.dq_acc = static_cast<float*>(t.dq);
    a.dk_acc = static_cast<float*>(t.dk);
    a.dv_acc = static_cast<float*>(t.dv);
  }
  a.step_visits = extras ? extras->step_visits : nullptr;
  a.ev_main_begin = extras ? static_cast<cudaEvent_t>(extras->main_begin_event) : nullptr;
  a.ev_main_end = extras ? static_cast<cudaEvent_t>(extras->main_end_event) : nullptr;
  const cudaError_t e = fa_launch_bwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Shared by fa_fwd_splitkv and fa_fwd_partial: the split-mode forward into partial buffers, then
// (merge) the pass that combines them into O and LSE.
int launch_partial(const fa::AttnShape& s, const fa_varlen_problem* p, int splits, const void* q, fa_strides sq,
                   const void* k, fa_strides sk, const void* v, fa_strides sv, void* o, fa_strides so, float* lse,
                   float* part_o, float* part_lse, int* dev_status, cudaStream_t st, bool merge) {
  int rc;
  const bool packed = s.cu_q != nullptr;
  const int rq = packed ? s.rows_q : s.Nq, rk = packed ? s.rows_k : s.Nk;
  FaStrides tq, tk, tv, to{};
  if ((rc = take_strides(sq, packed, s.B, rq, s.H, &tq)) != FA_OK ||
      (rc = take_strides(sk, packed, s.B, rk, s.Hkv, &tk)) != FA_OK ||
      (rc = take_strides(sv, packed, s.B, rk, s.Hkv, &tv)) != FA_OK)
    return rc;
  if (merge && (rc = take_strides(so, packed, s.B, rq, s.H, &to)) != FA_OK) return rc;
  if (!q || !k || !v || !part_o || !part_lse || (merge && (!o || !lse))) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(part_o, 16) || !aligned(part_lse, 4) || !aligned(dev_status, 4))
    return FA_ERR_MISALIGNED;
  if (!aux_on_device(s)) return FA_ERR_INVALID_ARG;
  fa::AttnShape sv_ = s;
  decode_view(sv_, &tq, merge ? &to : nullptr);
  FaFwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = merge ? o : nullptr;
  a.lse = merge ? lse : nullptr;
  a.sq = tq;
  a.sk = tk;
  a.sv = tv;
  a.so = to;
  a.s = sv_;
  a.scale = p->scale;
  a.tile_visits = nullptr;
  a.status = dev_status;
  a.splits = splits;
  a.kt_chunk = (sv_.nbk + splits - 1) / splits;
  a.part_rows = per_row(sv_);
  a.part_o = part_o;
  a.part_lse = part_lse;
  cudaError_t e = fa_launch_fwd(a, st);
  if (e == cudaSuccess && merge) e = fa_launch_splitkv_merge(a, st);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument (null pointer, size, flag, stride or scale)";
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
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!aligned(seqlens_k, 4)) return FA_ERR_MISALIGNED;
  const fa::AttnShape s = fixed_shape(B, H, Hkv, N, d, causal, block_mask, seqlens_k);
  return launch_fwd(s, q, contiguous(H, N, d), k, contiguous(Hkv, N, d), v, contiguous(Hkv, N, d), o,
                    contiguous(H, N, d), lse, scale, tile_visits, dev_status, stream);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d, int causal,
           const uint8_t* block_mask, const int32_t* seqlens_k, float scale, int32_t* tile_visits, int* dev_status,
           void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, block_mask, seqlens_k, scale, tile_visits, dev_status,
                    stream);
}

int fa_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int H, int Hkv, int N, int d,
               int causal, const uint8_t* block_mask, const int32_t* seqlens_k, const float* q_descale,
               const float* k_descale, const float* v_descale, float scale, int32_t* tile_visits, int* dev_status,
               void* stream) {
  if (!q || !k || !vt || !o || !lse || !q_descale || !k_descale || !v_descale) return FA_ERR_INVALID_ARG;
  const int rc = check_shape(B, H, N, d, causal, scale);
  if (rc != FA_OK) return rc;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (d != 128 || N % 16 != 0) return FA_ERR_UNSUPPORTED;  // 128-byte operand rows; V^T rows on 16-byte boundaries
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(vt, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(q_descale, 4) || !aligned(k_descale, 4) || !aligned(v_descale, 4) || !aligned(seqlens_k, 4) ||
      !aligned(tile_visits, 4) || !aligned(dev_status, 4))
    return FA_ERR_MISALIGNED;
  FaFwdArgs a{};
  a.s = fixed_shape(B, H, Hkv, N, d, causal, block_mask, seqlens_k);
  if (!aux_on_device(a.s)) return FA_ERR_INVALID_ARG;
  a.q = q;
  a.k = k;
  a.v = vt;
  a.o = o;
  a.lse = lse;
  a.so = contiguous(H, N, d);
  a.scale = scale;
  a.tile_visits = tile_visits;
  a.status = dev_status;
  a.splits = 1;
  a.kt_chunk = a.s.nbk;
  a.fp8 = 1;
  a.q_descale = q_descale;
  a.k_descale = k_descale;
  a.v_descale = v_descale;
  const cudaError_t e = fa_launch_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d, 0, 1.f) != FA_OK) return 0;
  return workspace_for(fixed_shape(B, H, H, N, d, 0, nullptr, nullptr));
}

int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
               void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, int causal,
               const uint8_t* block_mask, const int32_t* seqlens_k, float scale, void* workspace,
               size_t workspace_bytes, int* dev_status, void* stream) {
  return fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, block_mask, seqlens_k, scale,
                   workspace, workspace_bytes, nullptr, dev_status, stream);
}

int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
              void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, int causal,
              const uint8_t* block_mask, const int32_t* seqlens_k, float scale, void* workspace,
              size_t workspace_bytes, const fa_bwd_extras* extras, int* dev_status, void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  const int rc = check_shape(B, H, N, d, causal, scale);
  if (rc != FA_OK) return rc;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!aligned(seqlens_k, 4)) return FA_ERR_MISALIGNED;
  const fa::AttnShape s = fixed_shape(B, H, Hkv, N, d, causal, block_mask, seqlens_k);
  BwdTensors t;
  t.q = q;
  t.k = k;
  t.v = v;
  t.o = o;
  t.dout = dout;
  t.lse = lse;
  t.dq = dq;
  t.dk = dk;
  t.dv = dv;
  t.sq = t.so = t.sdo = t.sdq = contiguous(H, N, d);
  t.sk = t.sv = t.sdk = t.sdv = contiguous(Hkv, N, d);
  return launch_bwd(s, t, scale, workspace, workspace_bytes, dev_status, stream, extras);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int N, int d, int causal, const uint8_t* block_mask,
           const int32_t* seqlens_k, float scale, void* workspace, size_t workspace_bytes, int* dev_status,
           void* stream) {
  return fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, H, N, d, causal, block_mask, seqlens_k, scale, workspace,
                    workspace_bytes, dev_status, stream);
}

int fa_fwd_splitkv_splits(const fa_varlen_problem* p, int num_sms) {
  fa::AttnShape s;
  if (varlen_shape(p, &s) != FA_OK || num_sms < 1) return 1;
  decode_view(s, nullptr, nullptr);  // the shape the kernels run
  // The count with the least estimated time, in key-tile units: the CTAs' waves times (a CTA's
  // fixed cost, measured at about 6 key tiles: start-up, pipeline fill and drain, epilogue, plus
  // its key tiles), and for a split the merge pass (about 3). At least four key tiles per split.
  // With one query tile per (batch, head) a split runs two CTAs per SM (the single mode).
  constexpr long long kFixedTiles = 6, kMergeTiles = 3;
  const long long units = (long long)s.B * s.H * ((s.nbq + 1) / 2);  // CTAs without a split
  const long long slots = (long long)num_sms * (s.nbq == 1 ? 2 : 1);
  long long cap = s.nbk / 4;
  if (cap > kMaxSplits) cap = kMaxSplits;
  int best = 1;
  long long best_cost = -1;
  for (long long n = 1; n <= (cap < 1 ? 1 : cap); ++n) {
    const long long waves = (n * units + (n > 1 ? slots : num_sms) - 1) / (n > 1 ? slots : num_sms);
    const long long cost = waves * (kFixedTiles + (s.nbk + n - 1) / n) + (n > 1 ? kMergeTiles : 0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = (int)n;
    }
  }
  return best;
}

size_t fa_fwd_splitkv_workspace_bytes(const fa_varlen_problem* p, int num_splits) {
  fa::AttnShape s;
  if (varlen_shape(p, &s) != FA_OK || num_splits < 1 || num_splits > kMaxSplits) return 0;
  return splitkv_bytes(s, num_splits);
}

int fa_fwd_splitkv(const fa_varlen_problem* p, int num_splits, const void* q, fa_strides sq, const void* k,
                   fa_strides sk, const void* v, fa_strides sv, void* o, fa_strides so, float* lse, void* workspace,
                   size_t workspace_bytes, int* dev_status, void* stream) {
  fa::AttnShape s;
  int rc = varlen_shape(p, &s);
  if (rc != FA_OK) return rc;
  if (num_splits < 1 || num_splits > kMaxSplits || !workspace) return FA_ERR_INVALID_ARG;
  if (workspace_bytes < splitkv_bytes(s, num_splits)) return FA_ERR_INVALID_ARG;
  if (!aligned(workspace, kAlign)) return FA_ERR_MISALIGNED;
  float* part_lse = static_cast<float*>(workspace);
  float* part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           round_up(per_row(s) * num_splits * sizeof(float)));
  return launch_partial(s, p, num_splits, q, sq, k, sk, v, sv, o, so, lse, part_o, part_lse, dev_status,
                        static_cast<cudaStream_t>(stream), true);
}

size_t fa_partial_rows(const fa_varlen_problem* p) {
  fa::AttnShape s;
  if (varlen_shape(p, &s) != FA_OK) return 0;
  return per_row(s);
}

int fa_fwd_partial(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                   const void* v, fa_strides sv, float* part_o, float* part_lse, int* dev_status, void* stream) {
  fa::AttnShape s;
  const int rc = varlen_shape(p, &s);
  if (rc != FA_OK) return rc;
  fa_strides none{8, 8, 8};
  return launch_partial(s, p, 1, q, sq, k, sk, v, sv, nullptr, none, nullptr, part_o, part_lse, dev_status,
                        static_cast<cudaStream_t>(stream), false);
}

int fa_merge_partials(const fa_varlen_problem* p, float* acc_o, float* acc_lse, const float* part_o,
                      const float* part_lse, void* stream) {
  fa::AttnShape s;
  const int rc = varlen_shape(p, &s);
  if (rc != FA_OK) return rc;
  if (!acc_o || !acc_lse || !part_o || !part_lse) return FA_ERR_INVALID_ARG;
  if (!aligned(acc_o, 16) || !aligned(part_o, 16) || !aligned(acc_lse, 4) || !aligned(part_lse, 4))
    return FA_ERR_MISALIGNED;
  const cudaError_t e = fa_launch_merge_two(acc_o, acc_lse, part_o, part_lse, per_row(s), s.d,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_finalize_partials(const fa_varlen_problem* p, const float* acc_o, const float* acc_lse, void* o, fa_strides so,
                         float* lse, void* stream) {
  fa::AttnShape s;
  int rc = varlen_shape(p, &s);
  if (rc != FA_OK) return rc;
  const bool packed = s.cu_q != nullptr;
  FaStrides to;
  if ((rc = take_strides(so, packed, s.B, packed ? s.rows_q : s.Nq, s.H, &to)) != FA_OK) return rc;
  if (!acc_o || !acc_lse || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(acc_o, 16) || !aligned(o, 16) || !aligned(acc_lse, 4) || !aligned(lse, 4)) return FA_ERR_MISALIGNED;
  if (!aux_on_device(s)) return FA_ERR_INVALID_ARG;
  FaFwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.so = to;
  a.s = s;
  a.splits = 1;
  a.part_rows = per_row(s);
  a.part_o = const_cast<float*>(acc_o);
  a.part_lse = const_cast<float*>(acc_lse);
  const cudaError_t e = fa_launch_splitkv_merge(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_varlen(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                  const void* v, fa_strides sv, void* o, fa_strides so, float* lse, int* dev_status, void* stream) {
  fa::AttnShape s;
  int rc = varlen_shape(p, &s);
  if (rc != FA_OK) return rc;
  const bool packed = s.cu_q != nullptr;
  const int rq = packed ? s.rows_q : s.Nq, rk = packed ? s.rows_k : s.Nk;
  FaStrides tq, tk, tv, to;
  if ((rc = take_strides(sq, packed, s.B, rq, s.H, &tq)) != FA_OK ||
      (rc = take_strides(sk, packed, s.B, rk, s.Hkv, &tk)) != FA_OK ||
      (rc = take_strides(sv, packed, s.B, rk, s.Hkv, &tv)) != FA_OK ||
      (rc = take_strides(so, packed, s.B, rq, s.H, &to)) != FA_OK)
    return rc;
  return launch_fwd(s, q, tq, k, tk, v, tv, o, to, lse, p->scale, nullptr, dev_status, stream);
}

size_t fa_bwd_varlen_workspace_bytes(const fa_varlen_problem* p) {
  fa::AttnShape s;
  if (varlen_shape(p, &s) != FA_OK) return 0;
  return workspace_for(s);
}

static int bwd_varlen_impl(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                           const void* v, fa_strides sv, const void* o, fa_strides so, const void* dout,
                           fa_strides sdo, const float* lse, void* dq, fa_strides sdq, void* dk, fa_strides sdk,
                           void* dv, fa_strides sdv, void* workspace, size_t workspace_bytes, int* dev_status,
                           void* stream, bool accumulate);

int fa_bwd_varlen(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                  const void* v, fa_strides sv, const void* o, fa_strides so, const void* dout, fa_strides sdo,
                  const float* lse, void* dq, fa_strides sdq, void* dk, fa_strides sdk, void* dv, fa_strides sdv,
                  void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
  return bwd_varlen_impl(p, q, sq, k, sk, v, sv, o, so, dout, sdo, lse, dq, sdq, dk, sdk, dv, sdv, workspace,
                         workspace_bytes, dev_status, stream, false);
}

int fa_bwd_varlen_accumulate(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                             const void* v, fa_strides sv, const void* o, fa_strides so, const void* dout,
                             fa_strides sdo, const float* lse, float* dq_acc, fa_strides sdq, float* dk_acc,
                             fa_strides sdk, float* dv_acc, fa_strides sdv, void* workspace, size_t workspace_bytes,
                             int* dev_status, void* stream) {
  return bwd_varlen_impl(p, q, sq, k, sk, v, sv, o, so, dout, sdo, lse, dq_acc, sdq, dk_acc, sdk, dv_acc, sdv,
                         workspace, workspace_bytes, dev_status, stream, true);
}

static int bwd_varlen_impl(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                           const void* v, fa_strides sv, const void* o, fa_strides so, const void* dout,
                           fa_strides sdo, const float* lse, void* dq, fa_strides sdq, void* dk, fa_strides sdk,
                           void* dv, fa_strides sdv, void* workspace, size_t workspace_bytes, int* dev_status,
                           void* stream, bool accumulate) {
  fa::AttnShape s;
  int rc = varlen_shape(p, &s);
  if (rc != FA_OK) return rc;
  const bool packed = s.cu_q != nullptr;
  const int rq = packed ? s.rows_q : s.Nq, rk = packed ? s.rows_k : s.Nk;
  BwdTensors t;
  t.q = q;
  t.k = k;
  t.v = v;
  t.o = o;
  t.dout = dout;
  t.lse = lse;
  t.dq = dq;
  t.dk = dk;
  t.dv = dv;
  t.accumulate = accumulate;
  if ((rc = take_strides(sq, packed, s.B, rq, s.H, &t.sq)) != FA_OK ||
      (rc = take_strides(sk, packed, s.B, rk, s.Hkv, &t.sk)) != FA_OK ||
      (rc = take_strides(sv, packed, s.B, rk, s.Hkv, &t.sv)) != FA_OK ||
      (rc = take_strides(so, packed, s.B, rq, s.H, &t.so)) != FA_OK ||
      (rc = take_strides(sdo, packed, s.B, rq, s.H, &t.sdo)) != FA_OK ||
      (rc = take_strides(sdq, packed, s.B, rq, s.H, &t.sdq)) != FA_OK ||
      (rc = take_strides(sdk, packed, s.B, rk, s.Hkv, &t.sdk)) != FA_OK ||
      (rc = take_strides(sdv, packed, s.B, rk, s.Hkv, &t.sdv)) != FA_OK)
    return rc;
  return launch_bwd(s, t, p->scale, workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"
