// C ABI of libmla (declared in include/mla.h): argument checks, workspace layout and the
// launch sequence of each call.  Every step of the layer runs in this library's kernels.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/mla.h"
#include "mla_internal.h"

using namespace mla;

namespace {

const int kRows[5] = {Q_LORA, QB_N, KVA_N, KVB_N, HIDDEN};
const int kCols[5] = {HIDDEN, Q_LORA, HIDDEN, KV_LORA, O_IN};
const int kNorm[3] = {Q_LORA, KV_LORA, HIDDEN};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

bool ready(const mla_ctx* c) {
  for (int i = 0; i < 5; ++i)
    if (!c->W[i] || !c->S[i]) return false;
  return c->gain[0] && c->gain[1] && (!c->cfg.block || c->gain[2]);
}

// Workspace regions (byte offsets into the caller's buffer).
struct Layout {
  size_t g1 = 0, cq = 0, cq_sx = 0, ckv = 0, ckv_sx = 0, q = 0, kv = 0, attn = 0, attn_sx = 0,
         qfull = 0, opart = 0, ml = 0, olat = 0, gpart = 0, gather = 0, xn = 0, total = 0;
};

// Largest split-K partial buffer of the projections of one call with M token rows.
size_t gemm_partials(long M, int num_sms) {
  const int m = (int)M;
  size_t b = gemm_partial_bytes(m, Q_LORA + KVA_N, HIDDEN, num_sms);
  const size_t o[3] = {gemm_partial_bytes(m, QB_N, Q_LORA, num_sms),
                       gemm_partial_bytes(m, KVB_N, KV_LORA, num_sms),
                       gemm_partial_bytes(m, HIDDEN, O_IN, num_sms)};
  for (size_t v : o) b = v > b ? v : b;
  return b;
}

int items_max(const mla_ctx* c, int B) { return 2 * c->num_sms + B; }

// Prefill / cache-append workspace for M new tokens.  kv_rows: rows of the rebuilt keys and
// values (M over an empty cache; the sum of L_b + T with cached positions); kvb_M: the largest
// per-sequence kv_b_proj over cache rows (0 when the cache is empty).  With cached positions
// the layout also holds the latents of all kv_rows gathered from a paged cache (and the
// GEMM scratch of one kv_b_proj over all of them).
Layout prefill_layout(long M, int num_sms, long kv_rows = -1, long kvb_M = 0, bool block = false) {
  Layout L;
  if (kv_rows < 0) kv_rows = M;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += up256(bytes); return o; };
  if (block) L.xn = take((size_t)M * HIDDEN * 2);  // the block's normalised input
  L.g1 = take((size_t)M * G1_N * 4);
  L.cq = take((size_t)M * Q_LORA * 2);    // bf16, or its two e4m3 terms
  L.cq_sx = take((size_t)M * 4);
  L.ckv = take((size_t)M * KV_LORA * 2);  // bf16, or its two e4m3 terms
  L.ckv_sx = take((size_t)M * 4);
  L.q = take((size_t)M * QB_N * 2);
  L.kv = take((size_t)kv_rows * KVB_N * 2);
  L.attn = take((size_t)M * O_IN * 2);  // bf16, or its two e4m3 terms (M * O_IN bytes each)
  L.attn_sx = take((size_t)M * HEADS * 4);
  size_t gp = gemm_partials(M, num_sms);
  if (kvb_M > 0) {
    size_t k = gemm_partial_bytes((int)kvb_M, KVB_N, KV_LORA, num_sms);
    gp = k > gp ? k : gp;
    k = gemm_partial_bytes((int)kv_rows, KVB_N, KV_LORA, num_sms);
    gp = k > gp ? k : gp;
    L.gather = take((size_t)kv_rows * KV_LORA * 2);
  }
  L.gpart = take(gp);
  L.total = off;
  return L;
}

Layout decode_layout(const mla_ctx* c, int B) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += up256(bytes); return o; };
  const size_t items = (size_t)items_max(c, B);
  if (c->cfg.block) L.xn = take((size_t)B * HIDDEN * 2);  // the block's normalised input
  L.g1 = take((size_t)B * G1_N * 4);
  L.cq = take((size_t)B * Q_LORA * 2);
  L.q = take((size_t)B * QB_N * 2);
  L.qfull = take((size_t)B * HEADS * LAT * 2);
  L.opart = take(items * HEADS * KV_LORA * 2);
  L.ml = take(items * HEADS * 2 * 4);
  L.olat = take((size_t)B * HEADS * KV_LORA * 2);
  L.attn = take((size_t)B * O_IN * 2);
  size_t gp = gemm_partials(B, c->num_sms);
  if (B >= kAbsorbTcMinB) {  // the batched absorptions' e4m3 split of o_lat (the larger one)
    const size_t ab = absorb_split_bytes(B, KV_LORA);
    gp = ab > gp ? ab : gp;
  }
  L.gpart = take(gp);
  L.total = off;
  return L;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

void log_reset(mla_ctx* c) {
  c->n_launch = 0;
  c->last_profiled = c->profiling;
}

// Records one kernel launch of the current call; with profiling on, brackets it with events
// recorded on the launching stream.
// A context created with MLA_TEST_FAIL_AFTER=n fails at launch n of every call, before it is
// enqueued, exactly as a failed CUDA launch returns.
#define MLA_LAUNCH(name, expr)                                                          \
  do {                                                                                  \
    if (c->fail_at >= 0 && c->n_launch == c->fail_at) return MLA_ERR_CUDA;             \
    const int _k = c->n_launch < mla_ctx::kMaxLaunch ? c->n_launch : mla_ctx::kMaxLaunch - 1; \
    if (c->profiling && cudaEventRecord(c->ev[2 * _k], s) != cudaSuccess) return MLA_ERR_CUDA; \
    cudaError_t _e = (expr);                                                            \
    if (_e != cudaSuccess) return MLA_ERR_CUDA;                                         \
    if (c->profiling && cudaEventRecord(c->ev[2 * _k + 1], s) != cudaSuccess) return MLA_ERR_CUDA; \
    c->names[_k] = name;                                                                \
    if (c->n_launch < mla_ctx::kMaxLaunch) ++c->n_launch;                               \
  } while (0)

// Common checks of the token calls.  Lengths come from the host copy.
mla_status check_tokens(const mla_ctx* c, const void* x, int B, int T, const void* cache,
                        long long cap, const int* lens_dev, const int* lens_host, void* ws,
                        size_t ws_bytes, size_t need) {
  if (!c) return MLA_ERR_INVALID_ARG;
  if (B < 0 || T < 0 || cap < 0) return MLA_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return MLA_OK;
  if (!x || !cache || !lens_dev || !lens_host || !ws) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(cache) || !aligned16(ws)) return MLA_ERR_INVALID_ARG;
  if (!ready(c)) return MLA_ERR_STATE;
  if (ws_bytes < need) return MLA_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    if (lens_host[b] < 0) return MLA_ERR_INVALID_ARG;
    if ((long long)lens_host[b] + T > cap || (long)lens_host[b] + T > c->cfg.max_positions)
      return MLA_ERR_CAPACITY;
  }
  return MLA_OK;
}

// YaRN's attention temperature m(s, mu) = 0.1 mu ln s + 1 (s > 1), else 1.
double yarn_temperature(double s, double mu) { return s > 1.0 ? 0.1 * mu * std::log(s) + 1.0 : 1.0; }

// Angular frequency of each rotary pair and the cos/sin gain.  Plain RoPE: theta^(-2j/64).
// YaRN (Peng et al., 2023, in the parametrisation of config.json's rope_scaling keys): the
// pair whose wavelength turns r times over the original context is
// j(r) = 64 ln(original / (2 pi r)) / (2 ln theta); pairs up to floor(j(beta_fast)) keep their
// frequency, pairs from ceil(j(beta_slow)) on run `factor` times slower, and the frequency
// ramps linearly in j between the two (bounds clamped to [0, 63]; a zero-width ramp is one
// thousandth of a pair wide).  The gain is m(factor, mscale) / m(factor, mscale_all_dim).
void rope_frequencies(const mla_config& cfg, double* w, double* gain) {
  const double theta = cfg.rope_theta;
  for (int j = 0; j < ROPE / 2; ++j) w[j] = std::pow(theta, -2.0 * j / ROPE);
  *gain = 1.0;
  if (cfg.rope_scaling != MLA_ROPE_YARN) return;
  const double pi = 3.14159265358979323846;
  auto pair_of = [&](double r) {
    return ROPE * std::log((double)cfg.yarn_original_max_positions / (2.0 * pi * r)) /
           (2.0 * std::log(theta));
  };
  double lo = std::floor(pair_of(cfg.yarn_beta_fast)), hi = std::ceil(pair_of(cfg.yarn_beta_slow));
  lo = lo < 0.0 ? 0.0 : lo;
  hi = hi > ROPE - 1.0 ? ROPE - 1.0 : hi;
  const double width = hi > lo ? hi - lo : 1e-3;
  for (int j = 0; j < ROPE / 2; ++j) {
    double t = (j - lo) / width;
    t = t < 0.0 ? 0.0 : (t > 1.0 ? 1.0 : t);
    w[j] = w[j] * (1.0 - t) + (w[j] / cfg.yarn_factor) * t;
  }
  *gain = yarn_temperature(cfg.yarn_factor, cfg.yarn_mscale) /
          yarn_temperature(cfg.yarn_factor, cfg.yarn_mscale_all_dim);
}

// Positions allowed in a call: inside the cache and the RoPE table.
int limit_of(const mla_ctx* c, const CacheRef& CR) {
  const long long cap = CR.capacity();
  return cap < c->cfg.max_positions ? (int)cap : c->cfg.max_positions;
}

// The paged cache descriptor as a CacheRef, or MLA_ERR_INVALID_ARG.
mla_status paged_ref(const mla_paged_cache* pc, CacheRef* out) {
  if (!pc || !pc->pool || !pc->block_table || !aligned16(pc->pool) ||
      (reinterpret_cast<uintptr_t>(pc->block_table) & 3u))
    return MLA_ERR_INVALID_ARG;
  if (pc->page_size <= 0 || pc->page_size % 64 != 0 || pc->num_pages <= 0 || pc->max_pages <= 0)
    return MLA_ERR_INVALID_ARG;
  // Pool rows and positions must stay within the 32-bit coordinates of the tile copies.
  if ((long long)pc->num_pages * pc->page_size > 0x7FFFFFFFll - 256 ||
      (long long)pc->max_pages * pc->page_size > 0x7FFFFFFFll)
    return MLA_ERR_INVALID_ARG;
  *out = CacheRef{static_cast<__nv_bfloat16*>(pc->pool), pc->page_size, pc->block_table,
                  pc->max_pages, pc->num_pages};
  return MLA_OK;
}

// Whether a projection of M token rows takes the FP8-activation option's single-term path.
bool fp8_path(const mla_ctx* c, long M) { return c->cfg.fp8_activations && gemm_takes_split_blocks((int)M); }

// Y = X W^T of bf16 activations X [M, K] (row stride ldx): launch_gemm, or with the
// FP8-activation option the group quantisation of X into the scratch (q, then its scales
// where the second activation term would go) and the single-term GEMM.
cudaError_t proj_bf16(const mla_ctx* c, const __nv_bfloat16* X, int ldx, int M, int K,
                      const Proj* p, int np, float* scratch, cudaStream_t s, int* adv = nullptr,
                      int adv_n = 0, int adv_by = 0, bool pdl = false) {
  if (!fp8_path(c, M))
    return launch_gemm(X, ldx, M, K, p, np, scratch, c->num_sms, c->d_err, s, adv, adv_n, adv_by,
                       pdl);
  uint8_t* q = reinterpret_cast<uint8_t*>(scratch);
  float* sx = reinterpret_cast<float*>(q + up256((size_t)M * K));
  float* partial = reinterpret_cast<float*>(q + 2 * up256((size_t)M * K) + up256((size_t)M * 4));
  cudaError_t e = launch_quant_e4m3_groups(X, ldx, M, K, q, sx, s, pdl);
  if (e != cudaSuccess) return e;
  return launch_gemm_tc_split(q, nullptr, sx, true, M, K, p, np, partial, c->num_sms, c->d_err, s,
                              adv, adv_n, adv_by, true, pdl);
}

// The norm kernel's e4m3 output for q_b / kv_b over M token rows of n values, in the
// workspace region at `off` (sized for bf16): hi, then lo (the default pair, with one scale per
// token at sx_off), or with the FP8-activation option hi alone, its per-(token, 128-group)
// scales taking lo's place.
E4m3Split latent_split(const mla_ctx* c, void* ws, size_t off, size_t sx_off, long M, int n) {
  uint8_t* hi = at<uint8_t>(ws, off);
  if (fp8_path(c, M)) return E4m3Split{hi, nullptr, reinterpret_cast<float*>(hi + (size_t)M * n), 1};
  return E4m3Split{hi, hi + (size_t)M * n, at<float>(ws, sx_off), 0};
}

// The layer's input: x itself, or with block = 1 its input RMSNorm, written to the workspace by
// a first kernel (recorded in the call's launch log).  nullptr if that launch fails.
const __nv_bfloat16* block_input(mla_ctx* c, const void* x, int M, void* ws, const Layout& L,
                                 cudaStream_t s) {
  const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(x);
  if (!c->cfg.block) return X;
  __nv_bfloat16* xn = at<__nv_bfloat16>(ws, L.xn);
  auto launch = [&]() -> mla_status {
    MLA_LAUNCH("input_norm", launch_input_norm(X, M, c->gain[2], c->cfg.eps, xn, s));
    return MLA_OK;
  };
  return launch() == MLA_OK ? xn : nullptr;
}

mla_status cache_append_impl(mla_ctx* c, const void* x, int B, int T, const CacheRef& CR,
                             int* lens_dev, const int* lens_host, void* ws, size_t ws_bytes,
                             void* stream) {
  const Layout L = prefill_layout((long)B * T, c ? c->num_sms : 0, -1, 0, c && c->cfg.block);
  mla_status st = check_tokens(c, x, B, T, CR.base, CR.capacity(), lens_dev, lens_host, ws,
                               ws_bytes, L.total);
  if (st != MLA_OK || B == 0 || T == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  log_reset(c);
  const int M = B * T, limit = limit_of(c, CR);
  const __nv_bfloat16* X = block_input(c, x, M, ws, L, s);
  if (!X) return MLA_ERR_CUDA;
  float* g1 = at<float>(ws, L.g1);
  Proj p{c->W[MLA_W_KV_A], c->S[MLA_W_KV_A], KVA_N, g1 + Q_LORA, G1_N, 1};
  MLA_LAUNCH("gemm_kv_a", proj_bf16(c, X, HIDDEN, M, HIDDEN, &p, 1, at<float>(ws, L.gpart), s, nullptr, 0, 0, c->cfg.block != 0));
  MLA_LAUNCH("norm_rope_cache", launch_norm_rope_cache(g1, B, T, c->gain[0], c->gain[1], c->cfg.eps, c->rope_tab,
                                    c->cfg.rope_pairing, lens_dev, CR, limit, nullptr,
                                    nullptr, c->d_err, s));
  MLA_LAUNCH("advance_lens", launch_advance_lens(lens_dev, B, T, s));
  return MLA_OK;
}

mla_status prefill_impl(mla_ctx* c, const void* x, int B, int T, const CacheRef& CR,
                        int* lens_dev, const int* lens_host, void* out, void* ws,
                        size_t ws_bytes, void* stream) {
  // Cached positions before the call (chunked prefill when any is non-zero): the rebuilt keys
  // and values then cover L_b + T rows per sequence.
  long kv_rows = 0, kvb_M = 0;
  bool chunked = false;
  for (int b = 0; lens_host && b < B && B > 0 && T > 0; ++b) {
    if (lens_host[b] < 0) break;  // rejected by check_tokens below
    kv_rows += (long)lens_host[b] + T;
    kvb_M = (long)lens_host[b] + T > kvb_M ? (long)lens_host[b] + T : kvb_M;
    chunked = chunked || lens_host[b] != 0;
  }
  const Layout L = prefill_layout((long)B * T, c ? c->num_sms : 0, chunked ? kv_rows : -1,
                                  chunked ? kvb_M : 0, c && c->cfg.block);
  mla_status st = check_tokens(c, x, B, T, CR.base, CR.capacity(), lens_dev, lens_host, ws,
                               ws_bytes, L.total);
  if (st != MLA_OK || B == 0 || T == 0) return st;
  if (!out || !aligned16(out) || out == x) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  log_reset(c);
  const int M = B * T, limit = limit_of(c, CR);
  const __nv_bfloat16* X = block_input(c, x, M, ws, L, s);
  if (!X) return MLA_ERR_CUDA;
  const __nv_bfloat16* residual = c->cfg.block ? static_cast<const __nv_bfloat16*>(x) : nullptr;
  // Every kernel after the first is launched with programmatic dependent launch for few
  // tokens (the projections then stream their weights while the small kernels before them
  // run); with many tokens the early GEMM CTAs would only take SMs from their predecessors.
  const bool pdl = M <= kPrefillPdlMaxM;
  float* g1 = at<float>(ws, L.g1);
  __nv_bfloat16* cq = at<__nv_bfloat16>(ws, L.cq);
  __nv_bfloat16* ckv = at<__nv_bfloat16>(ws, L.ckv);
  __nv_bfloat16* q = at<__nv_bfloat16>(ws, L.q);
  __nv_bfloat16* kv = at<__nv_bfloat16>(ws, L.kv);
  __nv_bfloat16* attn = at<__nv_bfloat16>(ws, L.attn);

  Proj p1[2] = {{c->W[MLA_W_Q_A], c->S[MLA_W_Q_A], Q_LORA, g1, G1_N, 1},
                {c->W[MLA_W_KV_A], c->S[MLA_W_KV_A], KVA_N, g1 + Q_LORA, G1_N, 1}};
  MLA_LAUNCH("gemm_q_a_kv_a", proj_bf16(c, X, HIDDEN, M, HIDDEN, p1, 2, at<float>(ws, L.gpart), s, nullptr, 0, 0, pdl && c->cfg.block != 0));
  Proj p2{c->W[MLA_W_Q_B], c->S[MLA_W_Q_B], QB_N, q, QB_N, 0};
  Proj p3{c->W[MLA_W_KV_B], c->S[MLA_W_KV_B], KVB_N, kv, KVB_N, 0};
  if (chunked) {
    // Keys and values of the cached and the new positions: kv_b_proj over each sequence's
    // cache rows 0 .. L_b + T - 1 (the first 512 values of a row are its normalised latent),
    // after the norm kernel has appended the new rows.
    const E4m3Split qsp = latent_split(c, ws, L.cq, L.cq_sx, M, Q_LORA);
    MLA_LAUNCH("norm_rope_cache", launch_norm_rope_cache(g1, B, T, c->gain[0], c->gain[1], c->cfg.eps, c->rope_tab,
                                      c->cfg.rope_pairing, lens_dev, CR, limit, M > kGemvMaxM ? nullptr : cq,
                                      nullptr, c->d_err, s, pdl, M > kGemvMaxM ? &qsp : nullptr, nullptr));
    if (M > kGemvMaxM) {
      MLA_LAUNCH("gemm_q_b", launch_gemm_tc_split(qsp.hi, qsp.lo, qsp.sx, qsp.groups != 0, M, Q_LORA, &p2, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s,
                                                  nullptr, 0, 0, qsp.groups != 0, pdl));
    } else {
      MLA_LAUNCH("gemm_q_b", launch_gemm(cq, Q_LORA, M, Q_LORA, &p2, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s, nullptr, 0, 0, pdl));
    }
    MLA_LAUNCH("rope_q", launch_rope_q(q, B, T, c->rope_tab, c->cfg.rope_pairing, lens_dev, limit, s, pdl));
    if (CR.paged()) {
      // The cached latents are scattered over pages: gather all sequences' rows 0..L_b+T-1
      // back to back, then one kv_b_proj over them.
      __nv_bfloat16* lat = at<__nv_bfloat16>(ws, L.gather);
      MLA_LAUNCH("gather_latent", launch_gather_latent(CR, lens_dev, B, T, (int)kvb_M, kv_rows, lat,
                                                       c->d_err, s, pdl));
      MLA_LAUNCH("gemm_kv_b", proj_bf16(c, lat, KV_LORA, (int)kv_rows, KV_LORA, &p3, 1, at<float>(ws, L.gpart), s, nullptr, 0, 0, pdl));
    } else {
      long r0 = 0;
      for (int b = 0; b < B; ++b) {
        const int Mb = lens_host[b] + T;
        const Proj pb{c->W[MLA_W_KV_B], c->S[MLA_W_KV_B], KVB_N, kv + (size_t)r0 * KVB_N, KVB_N, 0};
        MLA_LAUNCH("gemm_kv_b", proj_bf16(c, CR.base + (size_t)b * CR.page * LAT, LAT, Mb, KV_LORA, &pb, 1, at<float>(ws, L.gpart), s, nullptr, 0, 0, pdl));
        r0 += Mb;
      }
    }
  } else if (M > kGemvMaxM) {
    // Tensor-core projections: the norm kernel writes q_b's and kv_b's e4m3 inputs itself (the
    // two terms share the bf16 latents' regions; one scale per token).
    const E4m3Split qsp = latent_split(c, ws, L.cq, L.cq_sx, M, Q_LORA);
    const E4m3Split kvsp = latent_split(c, ws, L.ckv, L.ckv_sx, M, KV_LORA);
    const bool one = qsp.groups != 0;
    MLA_LAUNCH("norm_rope_cache", launch_norm_rope_cache(g1, B, T, c->gain[0], c->gain[1], c->cfg.eps, c->rope_tab,
                                      c->cfg.rope_pairing, lens_dev, CR, limit, nullptr, nullptr,
                                      c->d_err, s, pdl, &qsp, &kvsp));
    MLA_LAUNCH("gemm_q_b", launch_gemm_tc_split(qsp.hi, qsp.lo, qsp.sx, one, M, Q_LORA, &p2, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s,
                                                nullptr, 0, 0, one, pdl));
    MLA_LAUNCH("rope_q", launch_rope_q(q, B, T, c->rope_tab, c->cfg.rope_pairing, lens_dev, limit, s, pdl));
    MLA_LAUNCH("gemm_kv_b", launch_gemm_tc_split(kvsp.hi, kvsp.lo, kvsp.sx, one, M, KV_LORA, &p3, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s,
                                                 nullptr, 0, 0, one, pdl));
  } else {
    MLA_LAUNCH("norm_rope_cache", launch_norm_rope_cache(g1, B, T, c->gain[0], c->gain[1], c->cfg.eps, c->rope_tab,
                                      c->cfg.rope_pairing, lens_dev, CR, limit, cq, ckv,
                                      c->d_err, s, pdl));
    MLA_LAUNCH("gemm_q_b", launch_gemm(cq, Q_LORA, M, Q_LORA, &p2, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s, nullptr, 0, 0, pdl));
    MLA_LAUNCH("rope_q", launch_rope_q(q, B, T, c->rope_tab, c->cfg.rope_pairing, lens_dev, limit, s, pdl));
    MLA_LAUNCH("gemm_kv_b", launch_gemm(ckv, KV_LORA, M, KV_LORA, &p3, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s, nullptr, 0, 0, pdl));
  }
  Proj p4{c->W[MLA_W_O], c->S[MLA_W_O], HIDDEN, out, HIDDEN, 0, residual};
  if (gemm_takes_split_blocks(M)) {
    // The attention writes o_proj's e4m3 input itself (one scale per token and head).
    uint8_t* a_hi = at<uint8_t>(ws, L.attn);
    uint8_t* a_lo = a_hi + (size_t)M * O_IN;
    float* a_sx = at<float>(ws, L.attn_sx);
    MLA_LAUNCH("prefill_attention", launch_prefill_attention_tc(q, kv, CR, B, T, chunked ? lens_dev : nullptr,
                                                              chunked ? kv_rows : M, c->cfg.softmax_scale, nullptr,
                                                              a_hi, a_lo, a_sx, c->num_sms, c->d_err, s, pdl));
    // With the FP8-activation option o_proj multiplies the high term alone: e4m3 of the
    // attention output over its own per-(token, head) scale, a head being one 128-wide group.
    MLA_LAUNCH("gemm_o", launch_gemm_tc_split(a_hi, a_lo, a_sx, true, M, O_IN, &p4, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s,
                                              lens_dev, B, T, fp8_path(c, M), pdl));
  } else {
    MLA_LAUNCH("prefill_attention", launch_prefill_attention_tc(q, kv, CR, B, T, chunked ? lens_dev : nullptr,
                                                              chunked ? kv_rows : M, c->cfg.softmax_scale, attn,
                                                              nullptr, nullptr, nullptr, c->num_sms, c->d_err, s, pdl));
    if (gemm_can_advance(M) && B <= 128) {  // the length update rides on o_proj
      MLA_LAUNCH("gemm_o", launch_gemm(attn, O_IN, M, O_IN, &p4, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s,
                                       lens_dev, B, T, pdl));
    } else {
      MLA_LAUNCH("gemm_o", launch_gemm(attn, O_IN, M, O_IN, &p4, 1, at<float>(ws, L.gpart), c->num_sms, c->d_err, s, nullptr, 0, 0, pdl));
      MLA_LAUNCH("advance_lens", launch_advance_lens(lens_dev, B, T, s, pdl));
    }
  }
  return MLA_OK;
}

// input_chained: the caller has already launched (and logged) a kernel that writes x, so the
// first projection is launched under programmatic dependent launch behind it.
mla_status decode_impl(mla_ctx* c, const void* x, int B, const CacheRef& CR, int* lens_dev,
                       const int* lens_host, void* out, void* ws, size_t ws_bytes, void* stream,
                       bool input_chained = false) {
  if (!c) return MLA_ERR_INVALID_ARG;
  const Layout L = decode_layout(c, B < 0 ? 0 : B);
  mla_status st = check_tokens(c, x, B, 1, CR.base, CR.capacity(), lens_dev, lens_host, ws,
                               ws_bytes, L.total);
  if (st != MLA_OK || B == 0) return st;
  if (!out || !aligned16(out) || out == x) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!input_chained) log_reset(c);
  const int limit = limit_of(c, CR);
  const __nv_bfloat16* X = block_input(c, x, B, ws, L, s);
  if (!X) return MLA_ERR_CUDA;
  const __nv_bfloat16* residual = c->cfg.block ? static_cast<const __nv_bfloat16*>(x) : nullptr;

  // Every kernel after the first is launched with programmatic dependent launch: it may start
  // (and fetch its weights) while its predecessor finishes, and waits for the predecessor's
  // results before reading them.
  // Split-KV schedule: the positions of all sequences cut into about one equal share per SM.
  long long total = 0;
  for (int b = 0; b < B; ++b) total += (long long)lens_host[b] + 1;
  const DecodePlan plan = make_decode_plan(B, total, c->num_sms, items_max(c, B));

  float* g1 = at<float>(ws, L.g1);
  __nv_bfloat16* cq = at<__nv_bfloat16>(ws, L.cq);
  __nv_bfloat16* q = at<__nv_bfloat16>(ws, L.q);
  __nv_bfloat16* qfull = at<__nv_bfloat16>(ws, L.qfull);
  __half* opart = at<__half>(ws, L.opart);
  float* ml = at<float>(ws, L.ml);
  __nv_bfloat16* olat = at<__nv_bfloat16>(ws, L.olat);
  __nv_bfloat16* attn = at<__nv_bfloat16>(ws, L.attn);

  Proj p1[2] = {{c->W[MLA_W_Q_A], c->S[MLA_W_Q_A], Q_LORA, g1, G1_N, 1},
                {c->W[MLA_W_KV_A], c->S[MLA_W_KV_A], KVA_N, g1 + Q_LORA, G1_N, 1}};
  MLA_LAUNCH("gemm_q_a_kv_a", launch_gemm(X, HIDDEN, B, HIDDEN, p1, 2, at<float>(ws, L.gpart), c->num_sms, c->d_err, s, nullptr, 0, 0, c->cfg.block != 0 || input_chained));
  if (B <= 2) {
    // One or two sequences: six kernels.  q_b_proj normalises the q latent itself (and one of
    // its CTAs appends the cache rows); the combine is fused with the W_UV absorption; the
    // length update rides on o_proj.  (Every q_b CTA normalises every token, and every
    // (head, sequence) CTA reads its head's W_UV: both pay only for very few sequences.)
    Proj p2{c->W[MLA_W_Q_B], c->S[MLA_W_Q_B], QB_N, q, QB_N, 0};
    MLA_LAUNCH("gemm_q_b_norm", launch_qb_norm(g1, B, p2, c->gain[0], c->gain[1], c->cfg.eps,
                                               c->rope_tab, c->cfg.rope_pairing, lens_dev, CR,
                                               limit, c->d_err, c->num_sms, s, true));
    MLA_LAUNCH("absorb_q", launch_absorb_q(q, B, c->W[MLA_W_KV_B], c->S[MLA_W_KV_B], c->rope_tab,
                                           c->cfg.rope_pairing, lens_dev, limit, qfull, s, true));
    MLA_LAUNCH("decode_attention", launch_decode_attention_tc(qfull, CR, lens_dev, plan,
                                                              c->cfg.softmax_scale, opart, ml,
                                                              c->d_err, s, true, true));
    MLA_LAUNCH("combine_absorb_out",
               launch_combine_absorb_out(lens_dev, lens_host, plan, opart, ml, c->W[MLA_W_KV_B],
                                         c->S[MLA_W_KV_B], attn, c->d_err, s, true));
    Proj p4{c->W[MLA_W_O], c->S[MLA_W_O], HIDDEN, out, HIDDEN, 0, residual};
    MLA_LAUNCH("gemm_o", launch_gemm(attn, O_IN, B, O_IN, &p4, 1, at<float>(ws, L.gpart),
                                     c->num_sms, c->d_err, s, lens_dev, B, 1, true));
    return MLA_OK;
  }
  MLA_LAUNCH("norm_rope_cache", launch_norm_rope_cache(g1, B, 1, c->gain[0], c->gain[1], c->cfg.eps, c->rope_tab,
                                    c->cfg.rope_pairing, lens_dev, CR, limit, cq, nullptr,
                                    c->d_err, s, true));
  Proj p2{c->W[MLA_W_Q_B], c->S[MLA_W_Q_B], QB_N, q, QB_N, 0};
  MLA_LAUNCH("gemm_q_b", launch_gemm(cq, Q_LORA, B, Q_LORA, &p2, 1, at<float>(ws, L.gpart),
                                     c->num_sms, c->d_err, s, nullptr, 0, 0, true));
  // Many sequences: both absorptions as batched tcgen05 GEMMs over the heads (W_UK through its
  // transposed copy, K-major; W_UV as stored), each after a head-major e4m3 split of its input
  // (the query's split also writes RoPE(q_pe)).  Fewer: the CUDA-core kernels.
  const bool absorb_tc = B >= kAbsorbTcMinB;
  const float* skvb = c->S[MLA_W_KV_B];
  if (absorb_tc) {
    if (c->wuk_t_stale) {
      MLA_LAUNCH("transpose_w_uk", launch_transpose_wuk(c->W[MLA_W_KV_B], c->wuk_t, s));
      c->wuk_t_stale = false;
    }
    MLA_LAUNCH("absorb_q", launch_absorb_tc(q, QB_N, QHEAD, B, NOPE, c->wuk_t,
                                            (long long)HEADS * KV_LORA, 0, KV_LORA, skvb,
                                            2 * (KV_LORA / BLK), KV_LORA, qfull, HEADS * LAT, LAT,
                                            qfull + KV_LORA, c->rope_tab, c->cfg.rope_pairing,
                                            lens_dev, limit, at<void>(ws, L.gpart), c->num_sms,
                                            c->d_err, s));
  } else {
    MLA_LAUNCH("absorb_q", launch_absorb_q(q, B, c->W[MLA_W_KV_B], skvb, c->rope_tab,
                                           c->cfg.rope_pairing, lens_dev, limit, qfull, s, true));
  }
  MLA_LAUNCH("decode_attention", launch_decode_attention_tc(qfull, CR, lens_dev, plan,
                                                            c->cfg.softmax_scale, opart, ml,
                                                            c->d_err, s, true));
  MLA_LAUNCH("decode_combine", launch_decode_combine(lens_dev, plan, opart, ml, olat, c->d_err, s,
                                                         true));
  if (absorb_tc) {
    MLA_LAUNCH("absorb_out", launch_absorb_tc(olat, (long long)HEADS * KV_LORA, KV_LORA, B,
                                              KV_LORA, c->W[MLA_W_KV_B], KVB_N, NOPE,
                                              KVB_PER_HEAD, skvb + KV_LORA / BLK,
                                              2 * (KV_LORA / BLK), VDIM, attn, O_IN, VDIM,
                                              nullptr, nullptr, 0, nullptr, 0,
                                              at<void>(ws, L.gpart), c->num_sms, c->d_err, s));
  } else {
    MLA_LAUNCH("absorb_out", launch_absorb_out(olat, B, c->W[MLA_W_KV_B], skvb, attn, s, true));
  }
  Proj p4{c->W[MLA_W_O], c->S[MLA_W_O], HIDDEN, out, HIDDEN, 0, residual};
  if (gemm_can_advance(B)) {  // the length update rides on the last kernel
    MLA_LAUNCH("gemm_o", launch_gemm(attn, O_IN, B, O_IN, &p4, 1, at<float>(ws, L.gpart),
                                     c->num_sms, c->d_err, s, lens_dev, B, 1, true));
  } else {
    MLA_LAUNCH("gemm_o", launch_gemm(attn, O_IN, B, O_IN, &p4, 1, at<float>(ws, L.gpart),
                                     c->num_sms, c->d_err, s, nullptr, 0, 0, true));
    MLA_LAUNCH("advance_lens", launch_advance_lens(lens_dev, B, 1, s));
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

void mla_default_config(mla_config* cfg) {
  if (!cfg) return;
  cfg->hidden = HIDDEN;
  cfg->q_lora = Q_LORA;
  cfg->kv_lora = KV_LORA;
  cfg->heads = HEADS;
  cfg->nope = NOPE;
  cfg->rope = ROPE;
  cfg->vdim = VDIM;
  cfg->eps = 1e-6f;
  cfg->rope_theta = 50000.0f;
  cfg->softmax_scale = (float)(1.0 / std::sqrt((double)(NOPE + ROPE)));
  cfg->max_positions = 131073;
  cfg->rope_pairing = MLA_ROPE_ADJACENT;
  cfg->rope_scaling = MLA_ROPE_PLAIN;
  cfg->yarn_factor = 32.0f;
  cfg->yarn_original_max_positions = 4096;
  cfg->yarn_beta_fast = 1.0f;
  cfg->yarn_beta_slow = 1.0f;
  cfg->yarn_mscale = 1.0f;
  cfg->yarn_mscale_all_dim = 1.0f;
  cfg->block = 0;
  cfg->fp8_activations = 0;
}

mla_status mla_create(const mla_config* cfg, mla_ctx** out) {
  if (!cfg || !out) return MLA_ERR_INVALID_ARG;
  if (cfg->hidden != HIDDEN || cfg->q_lora != Q_LORA || cfg->kv_lora != KV_LORA ||
      cfg->heads != HEADS || cfg->nope != NOPE || cfg->rope != ROPE || cfg->vdim != VDIM)
    return MLA_ERR_UNSUPPORTED;
  if (cfg->rope_pairing != MLA_ROPE_ADJACENT && cfg->rope_pairing != MLA_ROPE_HALF)
    return MLA_ERR_INVALID_ARG;
  if (cfg->max_positions <= 0 || !(cfg->eps >= 0.f) || !(cfg->rope_theta > 0.f) ||
      !(cfg->softmax_scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (cfg->rope_scaling != MLA_ROPE_PLAIN && cfg->rope_scaling != MLA_ROPE_YARN)
    return MLA_ERR_INVALID_ARG;
  if (cfg->block != 0 && cfg->block != 1) return MLA_ERR_INVALID_ARG;
  if (cfg->fp8_activations != 0 && cfg->fp8_activations != 1) return MLA_ERR_INVALID_ARG;
  if (cfg->rope_scaling == MLA_ROPE_YARN &&
      (!(cfg->yarn_factor >= 1.f) || cfg->yarn_original_max_positions <= 0 ||
       !(cfg->yarn_beta_fast > 0.f) || !(cfg->yarn_beta_slow > 0.f) ||
       !(cfg->yarn_mscale >= 0.f) || !(cfg->yarn_mscale_all_dim >= 0.f)))
    return MLA_ERR_INVALID_ARG;
  mla_ctx* c = new (std::nothrow) mla_ctx();
  if (!c) return MLA_ERR_INVALID_ARG;
  c->cfg = *cfg;
  if (const char* f = std::getenv("MLA_TEST_FAIL_AFTER")) {
    char* end = nullptr;
    const long v = std::strtol(f, &end, 10);
    if (end != f && *end == '\0' && v >= 0 && v < 1000) c->fail_at = (int)v;
  }
  if (init_kernels() != cudaSuccess || cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess ||
      noalloc_scratch_address(&c->noalloc_scratch) != cudaSuccess) {
    delete c;
    return MLA_ERR_CUDA;
  }
  // RoPE table in double precision: angle = pos * w_j, stored as float (g cos, g sin).
  // Plain: w_j = theta^(-2j/64), g = 1.  YaRN: see rope_frequencies.
  double w[ROPE / 2], g = 1.0;
  rope_frequencies(*cfg, w, &g);
  if (cfg->rope_scaling == MLA_ROPE_YARN) {
    const double m = yarn_temperature(cfg->yarn_factor, cfg->yarn_mscale_all_dim);
    c->cfg.softmax_scale = (float)((double)cfg->softmax_scale * m * m);
  }
  const size_t n = (size_t)cfg->max_positions * (ROPE / 2);
  std::vector<float2> tab(n);
  for (int j = 0; j < ROPE / 2; ++j) {
    for (int p = 0; p < cfg->max_positions; ++p) {
      const double a = (double)p * w[j];
      tab[(size_t)p * (ROPE / 2) + j] = make_float2((float)(g * std::cos(a)), (float)(g * std::sin(a)));
    }
  }
  if (cudaMalloc(&c->rope_tab, n * sizeof(float2)) != cudaSuccess) {
    delete c;
    return MLA_ERR_CUDA;
  }
  if (cudaMalloc(&c->d_err, sizeof(int)) != cudaSuccess ||
      cudaMemcpy(c->rope_tab, tab.data(), n * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess) {
    cudaFree(c->rope_tab);
    if (c->d_err) cudaFree(c->d_err);
    delete c;
    return MLA_ERR_CUDA;
  }
  *out = c;
  return MLA_OK;
}

void mla_destroy(mla_ctx* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  cudaFree(c->rope_tab);
  cudaFree(c->d_err);
  if (c->wuk_t) cudaFree(c->wuk_t);
  for (cudaEvent_t e : c->ev)
    if (e) cudaEventDestroy(e);
  delete c;
}

mla_status mla_set_profiling(mla_ctx* c, int on) {
  if (!c) return MLA_ERR_INVALID_ARG;
  if (on && !c->ev[0]) {
    for (cudaEvent_t& e : c->ev)
      if (cudaEventCreate(&e) != cudaSuccess) return MLA_ERR_CUDA;
  }
  c->profiling = on != 0;
  return MLA_OK;
}

int mla_last_launches(mla_ctx* c, int max, const char** names, float* ms) {
  if (!c) return -1;
  const int n = c->n_launch;
  for (int k = 0; k < n && k < max; ++k) {
    if (names) names[k] = c->names[k];
    if (ms) {
      // Events captured into a graph that has not been replayed yet are not recorded: they
      // report -1.  Failed queries must not leave an error behind for the caller's next check.
      ms[k] = -1.f;
      if (c->last_profiled && cudaEventSynchronize(c->ev[2 * k + 1]) == cudaSuccess &&
          cudaEventQuery(c->ev[2 * k]) == cudaSuccess &&
          cudaEventElapsedTime(&ms[k], c->ev[2 * k], c->ev[2 * k + 1]) != cudaSuccess)
        ms[k] = -1.f;
    }
  }
  cudaGetLastError();
  return n;
}

mla_status mla_upload_weights(mla_ctx* c, int which, const void* q, const float* s, int rows,
                              int cols) {
  if (!c || which < 0 || which > 4 || !q || !s) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(s) & 3u)) return MLA_ERR_INVALID_ARG;
  if (rows != kRows[which] || cols != kCols[which]) return MLA_ERR_SHAPE;
  if (which == MLA_W_KV_B) {
    if (!c->wuk_t && cudaMalloc(&c->wuk_t, (size_t)HEADS * KV_LORA * NOPE) != cudaSuccess) {
      c->wuk_t = nullptr;
      return MLA_ERR_CUDA;
    }
    c->wuk_t_stale = true;
  }
  c->W[which] = static_cast<const uint8_t*>(q);
  c->S[which] = s;
  return MLA_OK;
}

mla_status mla_upload_norm(mla_ctx* c, int which, const void* g, int n) {
  if (!c || which < 0 || which > 2 || !g || !aligned16(g)) return MLA_ERR_INVALID_ARG;
  if (n != kNorm[which]) return MLA_ERR_SHAPE;
  c->gain[which] = static_cast<const __nv_bfloat16*>(g);
  return MLA_OK;
}

size_t mla_workspace_bytes_len(const mla_ctx* c, int B, int T, int max_len) {
  if (!c || B < 0 || T < 0 || max_len < T) return 0;
  const size_t p = prefill_layout((long)B * T, c->num_sms, (long)B * max_len,
                                  max_len > T ? max_len : 0, c->cfg.block != 0).total;
  const size_t d = decode_layout(c, B).total;
  return p > d ? p : d;
}

size_t mla_workspace_bytes(const mla_ctx* c, int B, int T) {
  return mla_workspace_bytes_len(c, B, T, T);
}

mla_status mla_cache_append(mla_ctx* c, const void* x, int B, int T, void* cache, int cap,
                            int* lens_dev, const int* lens_host, void* ws, size_t ws_bytes,
                            void* stream) {
  return cache_append_impl(c, x, B, T, dense_cache(cache, cap), lens_dev, lens_host, ws, ws_bytes,
                           stream);
}

mla_status mla_prefill(mla_ctx* c, const void* x, int B, int T, void* cache, int cap,
                       int* lens_dev, const int* lens_host, void* out, void* ws,
                       size_t ws_bytes, void* stream) {
  return prefill_impl(c, x, B, T, dense_cache(cache, cap), lens_dev, lens_host, out, ws,
                      ws_bytes, stream);
}

mla_status mla_decode(mla_ctx* c, const void* x, int B, void* cache, int cap, int* lens_dev,
                      const int* lens_host, void* out, void* ws, size_t ws_bytes, void* stream) {
  return decode_impl(c, x, B, dense_cache(cache, cap), lens_dev, lens_host, out, ws, ws_bytes,
                     stream);
}

namespace {
// The device address of page-locked host memory that the device can address directly (16-byte
// aligned), else null.
void* mapped_host(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer || !aligned16(a.devicePointer))
    return nullptr;
  return a.devicePointer;
}
}  // namespace

size_t mla_decode_host_workspace_bytes(const mla_ctx* c, int B) {
  if (!c || B <= 0) return 0;
  return up256(mla_workspace_bytes(c, B, 1)) + 2 * up256((size_t)B * HIDDEN * 2);
}

mla_status mla_decode_host(mla_ctx* c, const void* x_host, int B, void* cache, int cap,
                           int* lens_dev, const int* lens_host, void* out_host, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!c || B < 0) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!x_host || !out_host || x_host == out_host) return MLA_ERR_INVALID_ARG;
  const size_t base = up256(mla_workspace_bytes(c, B, 1));
  const size_t io = up256((size_t)B * HIDDEN * 2);
  if (!ws || ws_bytes < base + 2 * io) return MLA_ERR_INVALID_ARG;
  const CacheRef CR = dense_cache(cache, cap);
  // Everything the step checks, before anything is enqueued.
  mla_status st = check_tokens(c, ws, B, 1, CR.base, CR.capacity(), lens_dev, lens_host, ws,
                               base, decode_layout(c, B).total);
  if (st != MLA_OK) return st;
  uint8_t* x_dev = static_cast<uint8_t*>(ws) + base;  // staged input, then output
  uint8_t* out_dev = x_dev + io;
  const size_t bytes = (size_t)B * HIDDEN * 2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* xm = mapped_host(x_host);
  void* om = mapped_host(out_host);
  log_reset(c);
  if (xm) {
    MLA_LAUNCH("copy_in", launch_copy16(xm, x_dev, bytes, false, s, false));
  } else if (cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyDefault, s) != cudaSuccess) {
    return MLA_ERR_CUDA;
  }
  st = decode_impl(c, x_dev, B, CR, lens_dev, lens_host, out_dev, ws, base, stream, xm != nullptr);
  if (st != MLA_OK) return st;
  if (om) {
    MLA_LAUNCH("copy_out", launch_copy16(out_dev, om, bytes, true, s, true));
  } else if (cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDefault, s) != cudaSuccess) {
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status mla_cache_append_paged(mla_ctx* c, const void* x, int B, int T,
                                  const mla_paged_cache* cache, int* lens_dev,
                                  const int* lens_host, void* ws, size_t ws_bytes, void* stream) {
  CacheRef cr;
  const mla_status st = paged_ref(cache, &cr);
  if (st != MLA_OK) return st;
  return cache_append_impl(c, x, B, T, cr, lens_dev, lens_host, ws, ws_bytes, stream);
}

mla_status mla_prefill_paged(mla_ctx* c, const void* x, int B, int T, const mla_paged_cache* cache,
                             int* lens_dev, const int* lens_host, void* out, void* ws,
                             size_t ws_bytes, void* stream) {
  CacheRef cr;
  const mla_status st = paged_ref(cache, &cr);
  if (st != MLA_OK) return st;
  return prefill_impl(c, x, B, T, cr, lens_dev, lens_host, out, ws, ws_bytes, stream);
}

mla_status mla_decode_paged(mla_ctx* c, const void* x, int B, const mla_paged_cache* cache,
                            int* lens_dev, const int* lens_host, void* out, void* ws,
                            size_t ws_bytes, void* stream) {
  CacheRef cr;
  const mla_status st = paged_ref(cache, &cr);
  if (st != MLA_OK) return st;
  return decode_impl(c, x, B, cr, lens_dev, lens_host, out, ws, ws_bytes, stream);
}
mla_status mla_dequant_weight(mla_ctx* c, int which, float* out, void* stream) {
  if (!c || which < 0 || which > 4 || !out) return MLA_ERR_INVALID_ARG;
  if (!c->W[which]) return MLA_ERR_STATE;
  return cuda_status(launch_dequant(c->W[which], c->S[which], kRows[which], kCols[which], out,
                                    static_cast<cudaStream_t>(stream)));
}

mla_status mla_get_device_status(mla_ctx* c, void* stream) {
  if (!c) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaMemcpy(&h, c->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
  if (h == DEV_ERR_NONE) return MLA_OK;
  return h == DEV_ERR_TIMEOUT ? MLA_ERR_TIMEOUT : MLA_ERR_STATE;
}

mla_status mla_selftest_wait_timeout(mla_ctx* c, unsigned long long limit_ns, void* stream) {
  if (!c || limit_ns > 2000000000ull) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_wait_selftest(c->d_err, limit_ns, static_cast<cudaStream_t>(stream)));
}

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_SHAPE: return "MLA_ERR_SHAPE";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CAPACITY: return "MLA_ERR_CAPACITY";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_STATE: return "MLA_ERR_STATE";
  }
  return "MLA_ERR_UNKNOWN";
}

}  // extern "C"
