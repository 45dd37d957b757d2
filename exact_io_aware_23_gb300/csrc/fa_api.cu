// C-ABI layer of libfa: argument validation, dispatch to the kernels, the per-device error
// word and the failure-detection test hooks.  See include/fa.h for the contract.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "fa_internal.cuh"
#include "fa_sm103.cuh"

namespace {

// Per-device error word written by kernels whose bounded waits ran out.
__device__ int g_fa_error_word;

fa::SymbolCache g_err_cache;
// Test hooks of the failure-detection path (process-wide; see fa_debug_set_fault_injection).
std::atomic<int> g_inject{0};
std::atomic<uint32_t> g_wait_limit_ms{2000};

// The error word of the current context (looked up once per context).
fa_status device_error_word(int** out) {
  void* p = nullptr;
  if (fa::symbol_address(g_err_cache, (const void*)&g_fa_error_word, &p) != cudaSuccess) return FA_ERR_CUDA;
  *out = static_cast<int*>(p);
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_common(int B, int H, int N, int d, float scale, fa_dtype dtype) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (!isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP32 && dtype != FA_FP16) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (H > 65535 || B > 65535) return FA_ERR_UNSUPPORTED;
  // one CTA per (b, h, 128-row tile) must fit a 1-D grid
  if ((size_t)B * (size_t)H * (size_t)((N + 127) / 128) > (size_t)0x7fffffff) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Grouped heads: Hkv key/value heads shared by H query heads.  Hkv must divide H (Hkv = H is
// plain multi-head attention); the fp32 SIMT path takes one key/value head per query head.
fa_status check_heads(int H, int Hkv, fa_dtype dtype) {
  if (Hkv < 0 || (H > 0 && Hkv == 0)) return FA_ERR_INVALID_ARG;
  if (H == 0) return FA_OK;
  if (Hkv > H || H % Hkv != 0) return FA_ERR_UNSUPPORTED;
  if (Hkv != H && dtype == FA_FP32) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// A block-sparse mask is kept as a one-bit-per-tile list in shared memory: N <= 786432.
constexpr int kMaxBlockSparseN = 786432;

fa::DebugKnobs knobs() {
  fa::DebugKnobs k;
  k.inject = g_inject.load();
  k.wait_limit_ms = g_wait_limit_ms.load();
  return k;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" {

int fa_version(void) { return 201; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_UNKNOWN_STATUS";
}

void fa_debug_set_fault_injection(int mode) { g_inject.store(mode); }

void fa_debug_set_wait_limit_ms(uint32_t ms) { g_wait_limit_ms.store(ms == 0 ? 2000u : ms); }

}  // extern "C"

namespace {

// Packed sequences (cu_seqlens != null): B sequences, N the longest, `total` tokens per head.
struct Packing {
  const int32_t* cu_seqlens;
  int total;
};

// Host form of the dropout arguments (validated; disabled when nothing is dropped).
fa_status make_dropout(const fa_dropout* in, fa::DropoutArgs* out) {
  *out = fa::DropoutArgs{};
  if (in == nullptr) return FA_ERR_INVALID_ARG;
  if (!isfinite(in->p) || in->p < 0.f || in->p > 1.f) return FA_ERR_INVALID_ARG;
  long long k8 = llrint((1.0 - (double)in->p) * 256.0);
  k8 = k8 < 0 ? 0 : (k8 > 256 ? 256 : k8);
  out->enabled = k8 < 256 ? 1 : 0;
  out->seed_lo = (uint32_t)(in->seed & 0xFFFFFFFFull);
  out->seed_hi = (uint32_t)(in->seed >> 32);
  out->offset = in->offset;
  out->k8 = (int)k8;
  out->scale = k8 > 0 ? 256.f / (float)k8 : 0.f;
  // Philox4x32-10's key schedule: round r uses the key plus r times the two Weyl increments
  for (int r = 0; r < 10; ++r) {
    out->rk0[r] = out->seed_lo + (uint32_t)r * 0x9E3779B9u;
    out->rk1[r] = out->seed_hi + (uint32_t)r * 0xBB67AE85u;
  }
  return FA_OK;
}

// Balanced block-sparse forward: the caller's workspace, carved into the plan's buffers.
struct Balance {
  void* workspace;
  size_t bytes;
};

constexpr int kPlanExtra = 16;                 // extra CTAs per (b, h) slice for split pairs
constexpr int kPlanSlots = 2 * kPlanExtra;     // partial slots per slice (split ranges <= 2 x extra)

// Byte offsets of the plan's buffers in the workspace: counts, plan, merge counters (and the
// persistent forward's unit counter after them), partial O, partial LSE, the pairs' live-tile
// bitmaps (each 256-byte aligned), and the total.
struct PlanLayout {
  size_t counts, plan, merge, next_unit, o_part, lse_part, bits, total;
  int words;
};

PlanLayout plan_layout(int B, int H, int N, int d) {
  const size_t pairs = (size_t)(N + 255) / 256, bh = (size_t)B * H;
  const int T = (N + fa::kMaskTile - 1) / fa::kMaskTile;
  PlanLayout L;
  L.words = (T + 31) / 32;
  L.counts = 0;
  L.plan = round_up(pairs * sizeof(int), 256);
  L.merge = L.plan + round_up((pairs + kPlanExtra) * 4 * sizeof(int), 256);
  L.next_unit = L.merge + bh * kPlanSlots * sizeof(int);
  L.o_part = L.merge + round_up(bh * kPlanSlots * sizeof(int) + sizeof(int), 256);
  L.lse_part = L.o_part + round_up(bh * kPlanSlots * 256 * (size_t)d * sizeof(float), 256);
  L.bits = L.lse_part + round_up(bh * kPlanSlots * 256 * sizeof(float), 256);
  L.total = L.bits + round_up(pairs * (size_t)L.words * sizeof(uint32_t), 256);
  return L;
}

fa_status forward_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int Hkv, int N, int d, float scale, int causal,
                       const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                       void* stream, Packing pk = {nullptr, 0}, fa::DropoutArgs drop = {},
                       Balance bal = {nullptr, 0}) {
  fa_status st = check_common(B, H, N, d, scale, dtype);
  if (st != FA_OK) return st;
  st = check_heads(H, Hkv, dtype);
  if (st != FA_OK) return st;
  if ((pk.cu_seqlens != nullptr || drop.enabled) && dtype == FA_FP32) return FA_ERR_UNSUPPORTED;
  if (pk.cu_seqlens != nullptr && drop.enabled) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0 || (pk.cu_seqlens != nullptr && pk.total == 0)) return FA_OK;
  if (block_mask != nullptr && N > kMaxBlockSparseN) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  fa::FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = B; a.H = H; a.Hkv = Hkv; a.N = N; a.d = d; a.scale = scale; a.causal = causal != 0;
  a.block_mask = block_mask; a.n_tiles = (N + fa::kMaskTile - 1) / fa::kMaskTile;
  a.kv_lens = kv_lens; a.dbg = knobs();
  // Masks make the work per tile unequal: then every slice's heaviest tiles go first.  Without
  // them, the tiles of one slice run together so its K/V (or Q/dO) stream is shared in L2.
  a.heads_fastest = (a.causal || block_mask != nullptr || kv_lens != nullptr) ? 1 : 0;
  a.Nk = N; a.n_splits = 1; a.tiles_per_split = 0; a.o_part = nullptr; a.lse_part = nullptr;
  a.cu_seqlens = pk.cu_seqlens;
  a.rows = pk.cu_seqlens != nullptr ? pk.total : N;
  if (pk.cu_seqlens != nullptr) a.heads_fastest = 1;     // sequences of unequal length
  a.drop = drop;
  a.plan = nullptr;
  a.plan_entries = 0;
  a.n_slots = 0;
  a.merge_count = nullptr;
  a.next_unit = nullptr;
  a.pair_bits = nullptr;
  a.bit_words = 0;
  if (device_error_word(&a.err) != FA_OK) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (bal.workspace != nullptr && block_mask != nullptr && dtype != FA_FP32) {
    const PlanLayout L = plan_layout(B, H, N, d);
    if (bal.bytes < L.total) return FA_ERR_INVALID_ARG;
    char* w = static_cast<char*>(bal.workspace);
    fa::PlanArgs p{};
    p.block_mask = block_mask;
    p.T = a.n_tiles;
    p.n_pairs = (N + 255) / 256;
    p.causal = a.causal;
    p.extra = kPlanExtra;
    p.n_slots = kPlanSlots;
    p.BH = B * H;
    p.sms = 152;                               // GB300's SM count when no device can be asked
    int sms = 0;
    if (fa::sm_count(&sms) == cudaSuccess && sms > 0) p.sms = sms;
    p.counts = reinterpret_cast<int*>(w + L.counts);
    p.plan = reinterpret_cast<int4*>(w + L.plan);
    p.merge_count = reinterpret_cast<int*>(w + L.merge);
    p.pair_bits = reinterpret_cast<uint32_t*>(w + L.bits);
    p.words = L.words;
    p.next_unit = reinterpret_cast<int*>(w + L.next_unit);
    cudaError_t e = fa::launch_blocksparse_plan(p, s);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    a.plan = p.plan;
    a.plan_entries = p.n_pairs + kPlanExtra;
    a.n_slots = kPlanSlots;
    a.merge_count = p.merge_count;
    a.next_unit = p.next_unit;
    a.pair_bits = p.pair_bits;
    a.bit_words = p.words;
    a.o_part = reinterpret_cast<float*>(w + L.o_part);
    a.lse_part = reinterpret_cast<float*>(w + L.lse_part);
  }
  cudaError_t e = dtype == FA_FP32 ? fa::launch_fwd_simt(a, dtype, s) : fa::launch_fwd_sm103(a, dtype, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int N, int d, float scale, int causal,
                     const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                     void* stream) {
  return forward_impl(q, k, v, o, lse, B, H, H, N, d, scale, causal, block_mask, dtype, kv_lens,
                      stream);
}

fa_status fa_forward_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int Hkv, int N, int d, float scale, int causal,
                         const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                         void* stream) {
  return forward_impl(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, block_mask, dtype, kv_lens,
                      stream);
}

size_t fa_forward_blocksparse_workspace_size(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
  return plan_layout(B, H, N, d).total;
}

fa_status fa_forward_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int Hkv, int N, int d, float scale, int causal,
                                 const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (block_mask != nullptr && B > 0 && H > 0 && N > 0) {
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return FA_ERR_INVALID_ARG;
  }
  return forward_impl(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, block_mask, dtype, kv_lens,
                      stream, Packing{nullptr, 0}, fa::DropoutArgs{}, Balance{workspace, workspace_bytes});
}

int fa_forward_splitkv_auto_splits(int B, int H, int Nq, int Nk) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return 1;
  int sms = 152;                            // GB300's SM count when no device can be asked
  int n = 0;
  if (fa::sm_count(&n) == cudaSuccess && n > 0) sms = n;
  const long long units = (long long)B * H * ((Nq + 255) / 256);   // CTAs without splitting
  const int kv_tiles = (Nk + 127) / 128;
  long long want = (2LL * sms + units - 1) / units;                 // about two CTAs per SM
  want = want < 1 ? 1 : want;
  const long long cap = (kv_tiles + 1) / 2 < 64 ? (kv_tiles + 1) / 2 : 64;   // >= 2 tiles each
  if (want > cap) want = cap < 1 ? 1 : cap;
  // From there, the fewest ranges whose CTAs fill their last wave of one-CTA-per-SM launches to
  // at least 95 % (a ragged last wave left most of the SMs idle at the end: on a 32K-key decode
  // the best count measured 1.1-1.3x faster than the first count above it); else the fullest
  // last wave among up to four times as many ranges.
  long long best = want;
  double best_fill = 0.0;
  for (long long s = want; s <= cap && s <= 4 * want; ++s) {
    const long long ctas = units * s, waves = (ctas + sms - 1) / sms;
    const double fill = (double)ctas / (double)(waves * sms);
    if (fill >= 0.95) return (int)s;
    if (fill > best_fill + 1e-9) { best_fill = fill; best = s; }
  }
  return (int)best;
}

size_t fa_forward_splitkv_workspace_size(int B, int H, int Nq, int d, int n_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || d <= 0 || n_splits <= 0) return 0;
  const size_t rows = (size_t)n_splits * B * H * Nq;
  return round_up(rows * (size_t)d * sizeof(float), 256) + round_up(rows * sizeof(float), 256);
}

fa_status fa_forward_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int Nq, int Nk, int d, float scale,
                             const int32_t* kv_lens, fa_dtype dtype, int n_splits,
                             void* workspace, size_t workspace_bytes, void* stream) {
  fa_status st = check_common(B, H, Nq, d, scale, dtype);
  if (st != FA_OK) return st;
  if (Nk < 0 || n_splits < 0) return FA_ERR_INVALID_ARG;
  if (dtype == FA_FP32) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || Nq == 0) return FA_OK;
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
  const int kv_tiles = (Nk + 127) / 128;
  if (n_splits == 0) n_splits = fa_forward_splitkv_auto_splits(B, H, Nq, Nk);
  if (n_splits > kv_tiles) n_splits = kv_tiles > 0 ? kv_tiles : 1;
  if ((size_t)B * H * ((Nq + 255) / 256) * (size_t)n_splits > (size_t)0x7fffffff) return FA_ERR_UNSUPPORTED;
  if (workspace_bytes < fa_forward_splitkv_workspace_size(B, H, Nq, d, n_splits)) return FA_ERR_INVALID_ARG;
  fa::FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = B; a.H = H; a.Hkv = H; a.N = Nq; a.d = d; a.scale = scale; a.causal = 0;
  a.block_mask = nullptr; a.n_tiles = (Nq + fa::kMaskTile - 1) / fa::kMaskTile;
  a.kv_lens = kv_lens; a.dbg = knobs(); a.heads_fastest = kv_lens != nullptr ? 1 : 0;
  a.Nk = Nk; a.n_splits = n_splits; a.tiles_per_split = (kv_tiles + n_splits - 1) / n_splits;
  a.cu_seqlens = nullptr; a.rows = Nq;
  const size_t rows = (size_t)B * H * Nq;
  a.o_part = static_cast<float*>(workspace);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        round_up((size_t)n_splits * rows * d * sizeof(float), 256));
  if (device_error_word(&a.err) != FA_OK) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_fwd_sm103(a, dtype, s);
  if (e == cudaSuccess) {
    fa::SplitMergeArgs m{};
    m.o_part = a.o_part; m.lse_part = a.lse_part; m.o = o; m.lse = lse;
    m.rows = (int)rows; m.d = d; m.n_splits = n_splits;
    e = fa::launch_splitkv_merge(m, dtype, s);
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_backward_workspace_size(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
  return fa_backward_deterministic_workspace_size(B, H, N);
}

size_t fa_backward_deterministic_workspace_size(int B, int H, int N) {
  if (B <= 0 || H <= 0 || N <= 0) return 0;
  // D (no dQ accumulator), then the unit order used under a tile mask (1/64 of D's size)
  return round_up((size_t)B * H * N * sizeof(float), 256) + fa::backward_order_bytes((size_t)B * H, N);
}

size_t fa_backward_fused_workspace_size(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
  const size_t rows = (size_t)B * H * N;
  return round_up(rows * (size_t)d * sizeof(float), 256) + round_up(rows * sizeof(float), 256);
}

}  // extern "C"

namespace {

// Which backward runs: kAuto = the two-pass kernel for 16-bit inputs and the CUDA-core kernel
// for fp32; kTwoPass = the two-pass kernel only (fp32 unsupported); kFused = the key-stationary
// kernel that adds dQ into an fp32 workspace (16-bit only).
enum class BwdPath { kAuto, kTwoPass, kFused };

fa_status backward_impl(const void* q, const void* k, const void* v, const void* o,
                        const void* dO, const float* lse, void* dq, void* dk, void* dv,
                        int B, int H, int Hkv, int N, int d, float scale, int causal,
                        const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                        void* workspace, size_t workspace_bytes, void* stream,
                        BwdPath path, Packing pk = {nullptr, 0}, fa::DropoutArgs drop = {}) {
  fa_status st = check_common(B, H, N, d, scale, dtype);
  if (st != FA_OK) return st;
  st = check_heads(H, Hkv, dtype);
  if (st != FA_OK) return st;
  if ((path != BwdPath::kAuto || pk.cu_seqlens != nullptr || drop.enabled) && dtype == FA_FP32)
    return FA_ERR_UNSUPPORTED;
  if (pk.cu_seqlens != nullptr && drop.enabled) return FA_ERR_UNSUPPORTED;
  // 16-bit inputs run the two-pass backward unless the fused one was asked for; fp32 always runs
  // the CUDA-core backward, which adds dQ from several blocks into the fp32 dQ output itself.
  const bool fused = path == BwdPath::kFused;
  const bool two_pass = !fused && dtype != FA_FP32;
  // workspace sizes count the query rows of all slices: B*H*N, or H*total when packed
  const int wB = pk.cu_seqlens != nullptr ? 1 : B, wN = pk.cu_seqlens != nullptr ? pk.total : N;
  if (B == 0 || H == 0 || N == 0 || (pk.cu_seqlens != nullptr && pk.total == 0)) return FA_OK;
  if (block_mask != nullptr && N > kMaxBlockSparseN) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
  const size_t need = fused ? fa_backward_fused_workspace_size(wB, H, wN, d)
                            : fa_backward_workspace_size(wB, H, wN, d);
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.dO = dO; a.lse = lse; a.dq = dq; a.dk = dk; a.dv = dv;
  const size_t rows = (size_t)wB * H * wN;
  a.perm = nullptr;
  if (two_pass) {                      // D only: dQ is written once, no accumulator
    a.dq_acc = nullptr;
    a.delta = static_cast<float*>(workspace);
  } else if (!fused) {                 // fp32: the fp32 dQ output is its own accumulator
    a.dq_acc = static_cast<float*>(dq);
    a.delta = static_cast<float*>(workspace);
  } else {
    a.dq_acc = static_cast<float*>(workspace);
    a.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       round_up(rows * (size_t)d * sizeof(float), 256));
  }
  a.B = B; a.H = H; a.Hkv = Hkv; a.N = N; a.d = d; a.scale = scale; a.causal = causal != 0;
  a.block_mask = block_mask; a.n_tiles = (N + fa::kMaskTile - 1) / fa::kMaskTile;
  a.kv_lens = kv_lens; a.dbg = knobs();
  // Masks make the work per tile unequal: then every slice's heaviest tiles go first.  Without
  // them, the tiles of one slice run together so its K/V (or Q/dO) stream is shared in L2.
  a.heads_fastest = (a.causal || block_mask != nullptr || kv_lens != nullptr) ? 1 : 0;
  a.cu_seqlens = pk.cu_seqlens;
  a.rows = pk.cu_seqlens != nullptr ? pk.total : N;
  if (pk.cu_seqlens != nullptr) a.heads_fastest = 1;     // sequences of unequal length
  a.drop = drop;
  if (device_error_word(&a.err) != FA_OK) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (two_pass && block_mask != nullptr) {
    // the units' order under the tile mask: the longest first (after D in the workspace)
    int* w = reinterpret_cast<int*>(static_cast<char*>(workspace) + round_up(rows * sizeof(float), 256));
    const int T = a.n_tiles;
    fa::OrderArgs p{};
    p.block_mask = block_mask;
    p.T = T;
    p.causal = a.causal;
    p.BH = B * H;
    p.BHkv = B * Hkv;
    p.counts = w;
    p.rank = p.counts + 2 * T;
    p.order = reinterpret_cast<int2*>(p.rank + 2 * T);
    p.order_off = reinterpret_cast<int*>(p.order + 2 * T);
    p.perm = p.order_off + 2 * T + 1;
    if (fa::launch_backward_order(p, s) != cudaSuccess) return FA_ERR_CUDA;
    a.perm = p.perm;
  }
  cudaError_t e = fa::launch_bwd_preprocess(a, dtype, s);
  if (e == cudaSuccess) {
    if (two_pass) {
      e = fa::launch_bwd_split_sm103(a, dtype, s);
    } else {
      e = dtype == FA_FP32 ? fa::launch_bwd_simt(a, dtype, s) : fa::launch_bwd_sm103(a, dtype, s);
      if (e == cudaSuccess) e = fa::launch_bwd_dq_convert(a, dtype, s);
    }
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

fa_status fa_backward(const void* q, const void* k, const void* v, const void* o,
                      const void* dO, const float* lse, void* dq, void* dk, void* dv,
                      int B, int H, int N, int d, float scale, int causal,
                      const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d, scale, causal, block_mask,
                       dtype, kv_lens, workspace, workspace_bytes, stream, BwdPath::kAuto);
}

fa_status fa_backward_gqa(const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv,
                          int B, int H, int Hkv, int N, int d, float scale, int causal,
                          const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                          void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal, block_mask,
                       dtype, kv_lens, workspace, workspace_bytes, stream, BwdPath::kAuto);
}

fa_status fa_backward_fused(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv,
                            int B, int H, int Hkv, int N, int d, float scale, int causal,
                            const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal, block_mask,
                       dtype, kv_lens, workspace, workspace_bytes, stream, BwdPath::kFused);
}

fa_status fa_backward_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                    int B, int H, int Hkv, int N, int d, float scale, int causal,
                                    const uint8_t* block_mask, fa_dtype dtype,
                                    const int32_t* kv_lens, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal, block_mask,
                       dtype, kv_lens, workspace, workspace_bytes, stream, BwdPath::kTwoPass);
}

fa_status fa_forward_splitkv_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                                 const int32_t* kv_lens, fa_dtype dtype, int n_splits,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || Nq < 0) return FA_ERR_INVALID_ARG;
  const fa_status st = check_heads(H, Hkv, dtype);
  if (st != FA_OK) return st;
  if (B == 0 || H == 0 || Nq == 0) return fa_forward_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale,
                                                             kv_lens, dtype, n_splits, workspace,
                                                             workspace_bytes, stream);
  const long long rows = (long long)(H / Hkv) * Nq;     // a group's queries, contiguous
  if (rows > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return fa_forward_splitkv(q, k, v, o, lse, B, Hkv, (int)rows, Nk, d, scale, kv_lens, dtype,
                            n_splits, workspace, workspace_bytes, stream);
}

fa_status fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int Hkv, int N, int d, float scale, int causal,
                             const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                             const fa_dropout* dropout, void* stream) {
  fa::DropoutArgs drop;
  const fa_status st = make_dropout(dropout, &drop);
  if (st != FA_OK) return st;
  return forward_impl(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, block_mask, dtype, kv_lens,
                      stream, Packing{nullptr, 0}, drop);
}

fa_status fa_backward_dropout(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int Hkv, int N, int d, float scale, int causal,
                              const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                              const fa_dropout* dropout, void* workspace, size_t workspace_bytes,
                              void* stream) {
  fa::DropoutArgs drop;
  const fa_status st = make_dropout(dropout, &drop);
  if (st != FA_OK) return st;
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal, block_mask,
                       dtype, kv_lens, workspace, workspace_bytes, stream, BwdPath::kTwoPass,
                       Packing{nullptr, 0}, drop);
}

fa_status fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens, int n_seqs, int max_seqlen, int total,
                            int H, int Hkv, int d, float scale, int causal, fa_dtype dtype,
                            void* stream) {
  if (n_seqs < 0 || max_seqlen < 0 || total < 0) return FA_ERR_INVALID_ARG;
  if (n_seqs > 0 && total > 0 && cu_seqlens == nullptr) return FA_ERR_INVALID_ARG;
  return forward_impl(q, k, v, o, lse, n_seqs, H, Hkv, max_seqlen, d, scale, causal, nullptr,
                      dtype, nullptr, stream, Packing{cu_seqlens, total});
}

fa_status fa_backward_varlen(const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse, void* dq, void* dk, void* dv,
                             const int32_t* cu_seqlens, int n_seqs, int max_seqlen, int total,
                             int H, int Hkv, int d, float scale, int causal, fa_dtype dtype,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (n_seqs < 0 || max_seqlen < 0 || total < 0) return FA_ERR_INVALID_ARG;
  if (n_seqs > 0 && total > 0 && cu_seqlens == nullptr) return FA_ERR_INVALID_ARG;
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, n_seqs, H, Hkv, max_seqlen, d, scale,
                       causal, nullptr, dtype, nullptr, workspace, workspace_bytes, stream,
                       BwdPath::kTwoPass, Packing{cu_seqlens, total});
}

fa_status fa_check_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  int* p = nullptr;
  if (device_error_word(&p) != FA_OK) return FA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    return word == fa::kDevBadOffsets ? FA_ERR_INVALID_ARG : FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

}  // extern "C"
