// mla_decode_noalloc: one decode step, like mla_decode, for callers that cannot allocate GPU
// memory.
//
// Some hosts of this library cannot call cudaMalloc, or any allocator, at the point where a
// decode step runs: a serving loop that owns all device memory through a fixed arena, an
// embedding runtime that forbids driver allocations after start-up, or a caller running
// under a memory budget that must not move.  mla_decode asks them for a workspace; this entry
// point needs none.  Its scratch (every intermediate of the step and the split-KV partial
// outputs of the attention) lives in one file-scope device array of kScratchBytes, which
// every GPU that loads the library holds until the process exits.
//
// Limits and rules (also stated in include/mla.h):
//   * at most kMaxBatch sequences per call; the attention uses at most kMaxItems partial slots
//     (sequences + shares), so long contexts are cut into fewer, longer shares than mla_decode
//     would use;
//   * every call shares the one array: calls whose work overlaps on the GPU (two streams, two
//     threads, two contexts on one device) race with each other;
//   * the array keeps the last call's contents; this path writes every scratch byte it reads
//     before reading it, so nothing needs clearing between calls;
//   * mla_create looks up the array's device address on the context's device (with that
//     device current) and keeps it in the context, so the address lives and dies with the
//     context; a call made with another device current is refused.
#include "mla_internal.h"

using namespace mla;

namespace {

constexpr int kMaxBatch = 8;
constexpr int kMaxItems = 48;
constexpr size_t kScratchBytes = size_t(12) << 20;
constexpr size_t kGemmScratch = size_t(29) << 18;  // 7.25 MiB: tensor-core GEMM scratch
constexpr int kMaxSms = 1024;                       // SM counts the GEMM scratch is sized for

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// The largest scratch the tensor-core projections of this path (kGemvMaxM < B <= kMaxBatch)
// plan for, over every SM count up to kMaxSms: the split-K partials grow when few SMs make the
// planner cut the reduction finer (on 5 SMs o_proj takes 32 splits, 7.1 MiB for 8 tokens).
constexpr size_t max_gemm_scratch() {
  size_t worst = 0;
  for (int sms = 1; sms <= kMaxSms; ++sms)
    for (int b = kGemvMaxM + 1; b <= kMaxBatch; ++b) {
      const size_t v[3] = {gemm_partial_bytes(b, Q_LORA + KVA_N, HIDDEN, sms),
                           gemm_partial_bytes(b, QB_N, Q_LORA, sms),
                           gemm_partial_bytes(b, HIDDEN, O_IN, sms)};
      for (size_t x : v) worst = x > worst ? x : worst;
    }
  return worst;
}
static_assert(max_gemm_scratch() <= kGemmScratch, "GEMM scratch too small for some SM count");

struct Regions {
  size_t g1, cq, q, qfull, opart, ml, olat, attn, gpart, total;
};

constexpr Regions regions(int B) {
  Regions r{};
  size_t off = 0;
  r.g1 = off;    off += up256((size_t)B * G1_N * 4);
  r.cq = off;    off += up256((size_t)B * Q_LORA * 2);
  r.q = off;     off += up256((size_t)B * QB_N * 2);
  r.qfull = off; off += up256((size_t)B * HEADS * LAT * 2);
  r.opart = off; off += up256((size_t)kMaxItems * HEADS * KV_LORA * 2);
  r.ml = off;    off += up256((size_t)kMaxItems * HEADS * 2 * 4);
  r.olat = off;  off += up256((size_t)B * HEADS * KV_LORA * 2);
  r.attn = off;  off += up256((size_t)B * O_IN * 2);
  r.gpart = off; off += kGemmScratch;
  r.total = off;
  return r;
}
static_assert(regions(kMaxBatch).total <= kScratchBytes, "scratch too small for kMaxBatch");

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace mla {

// Host code holds only a stand-in for g_decode_scratch; this is its address on the current
// device.
cudaError_t noalloc_scratch_address(void** out) {
  return cudaGetSymbolAddress(out, g_decode_scratch);
}

}  // namespace mla

extern "C" mla_status mla_decode_noalloc(mla_ctx* c, const void* x, int B, void* cache, int cap,
                                         int* lens_dev, const int* lens_host, void* out,
                                         void* stream) {
  if (!c || B < 0 || cap < 0) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (B > kMaxBatch) return MLA_ERR_CAPACITY;  // beyond the static scratch
  if (c->cfg.block) return MLA_ERR_UNSUPPORTED;  // no room for the block's normalised input
  if (!x || !cache || !lens_dev || !lens_host || !out || out == x) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(cache) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i)
    if (!c->W[i] || !c->S[i]) return MLA_ERR_STATE;
  if (!c->gain[0] || !c->gain[1]) return MLA_ERR_STATE;
  long total = 0;
  for (int b = 0; b < B; ++b) {
    if (lens_host[b] < 0) return MLA_ERR_INVALID_ARG;
    if ((long)lens_host[b] + 1 > cap || (long)lens_host[b] + 1 > c->cfg.max_positions)
      return MLA_ERR_CAPACITY;
    total += (long)lens_host[b] + 1;
  }
  // Split-KV schedule with at most kMaxItems partial slots (B + shares).
  const DecodePlan plan = make_decode_plan(B, total, c->num_sms, kMaxItems);
  // The tensor-core projections' scratch (more than kGemvMaxM sequences) fits its region on
  // every SM count up to kMaxSms (checked at compile time); beyond that, check here.
  if (c->num_sms > kMaxSms &&
      (gemm_partial_bytes(B, Q_LORA + KVA_N, HIDDEN, c->num_sms) > kGemmScratch ||
       gemm_partial_bytes(B, QB_N, Q_LORA, c->num_sms) > kGemmScratch ||
       gemm_partial_bytes(B, HIDDEN, O_IN, c->num_sms) > kGemmScratch))
    return MLA_ERR_CAPACITY;
  // The scratch address belongs to the context's device.
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev != c->device || !c->noalloc_scratch) return MLA_ERR_INVALID_ARG;
  void* scratch = c->noalloc_scratch;
  const Regions R = regions(B);
  char* w = static_cast<char*>(scratch);
  float* g1 = reinterpret_cast<float*>(w + R.g1);
  __nv_bfloat16* cq = reinterpret_cast<__nv_bfloat16*>(w + R.cq);
  __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(w + R.q);
  __nv_bfloat16* qfull = reinterpret_cast<__nv_bfloat16*>(w + R.qfull);
  __half* opart = reinterpret_cast<__half*>(w + R.opart);
  float* ml = reinterpret_cast<float*>(w + R.ml);
  __nv_bfloat16* olat = reinterpret_cast<__nv_bfloat16*>(w + R.olat);
  __nv_bfloat16* attn = reinterpret_cast<__nv_bfloat16*>(w + R.attn);
  float* gpart = reinterpret_cast<float*>(w + R.gpart);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->n_launch = 0;  // this call keeps no launch log
  c->last_profiled = false;
  const int limit = cap < c->cfg.max_positions ? cap : c->cfg.max_positions;
  const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(x);
  __nv_bfloat16* C = static_cast<__nv_bfloat16*>(cache);

#define NA_RUN(expr)                              \
  do {                                            \
    if ((expr) != cudaSuccess) return MLA_ERR_CUDA; \
  } while (0)
  Proj p1[2] = {{c->W[MLA_W_Q_A], c->S[MLA_W_Q_A], Q_LORA, g1, G1_N, 1},
                {c->W[MLA_W_KV_A], c->S[MLA_W_KV_A], KVA_N, g1 + Q_LORA, G1_N, 1}};
  NA_RUN(launch_gemm(X, HIDDEN, B, HIDDEN, p1, 2, gpart, c->num_sms, c->d_err, s));
  const CacheRef CR = dense_cache(C, cap);
  NA_RUN(launch_norm_rope_cache(g1, B, 1, c->gain[0], c->gain[1], c->cfg.eps, c->rope_tab,
                                c->cfg.rope_pairing, lens_dev, CR, limit, cq, nullptr,
                                c->d_err, s));
  Proj p2{c->W[MLA_W_Q_B], c->S[MLA_W_Q_B], QB_N, q, QB_N, 0};
  NA_RUN(launch_gemm(cq, Q_LORA, B, Q_LORA, &p2, 1, gpart, c->num_sms, c->d_err, s));
  NA_RUN(launch_absorb_q(q, B, c->W[MLA_W_KV_B], c->S[MLA_W_KV_B], c->rope_tab,
                         c->cfg.rope_pairing, lens_dev, limit, qfull, s));
  NA_RUN(launch_decode_attention_tc(qfull, CR, lens_dev, plan, c->cfg.softmax_scale, opart,
                                    ml, c->d_err, s));
  NA_RUN(launch_decode_combine(lens_dev, plan, opart, ml, olat, c->d_err, s));
  NA_RUN(launch_absorb_out(olat, B, c->W[MLA_W_KV_B], c->S[MLA_W_KV_B], attn, s));
  Proj p4{c->W[MLA_W_O], c->S[MLA_W_O], HIDDEN, out, HIDDEN, 0};
  NA_RUN(launch_gemm(attn, O_IN, B, O_IN, &p4, 1, gpart, c->num_sms, c->d_err, s));
  NA_RUN(launch_advance_lens(lens_dev, B, 1, s));
#undef NA_RUN
  return MLA_OK;
}
