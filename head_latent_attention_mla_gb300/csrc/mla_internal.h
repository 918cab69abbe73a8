// Internal declarations shared by the libmla translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

// Kimi-K2 MLA dimensions (config.json on the "KV cache" page).
constexpr int HIDDEN = 7168;
constexpr int Q_LORA = 1536;
constexpr int KV_LORA = 512;
constexpr int HEADS = 64;
constexpr int NOPE = 128;
constexpr int ROPE = 64;
constexpr int VDIM = 128;
constexpr int QHEAD = NOPE + ROPE;         // 192
constexpr int LAT = KV_LORA + ROPE;        // 576 values per cached position
constexpr int KVA_N = KV_LORA + ROPE;      // 576 rows of kv_a_proj_with_mqa
constexpr int QB_N = HEADS * QHEAD;        // 12288
constexpr int KVB_PER_HEAD = NOPE + VDIM;  // 256
constexpr int KVB_N = HEADS * KVB_PER_HEAD;  // 16384
constexpr int O_IN = HEADS * VDIM;         // 8192
constexpr int G1_N = Q_LORA + KVA_N;       // 2112: q_a and kv_a outputs side by side
constexpr int BLK = 128;                   // FP8 weight block (weight_block_size)

// Programmatic dependent launch.  A kernel launched with pdl=true may start while the previous
// kernel in the stream is still running; it must call pdl_wait() before touching anything that
// kernel (or an earlier one) writes.  pdl_wait() is a no-op for a normal launch, and every
// kernel calls pdl_launch_dependents() early so that its successor can be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Loads of data that an earlier kernel of the stream writes, in kernels launched with pdl=true.
// They are coherent loads (never ld.global.nc: a non-coherent load promises that the data stay
// unchanged for the whole life of the kernel, which is not so before pdl_wait() returns, and
// lets the compiler hoist it above the wait), issued as volatile asm so that they stay after
// pdl_wait() in program order.  `p` must be aligned to the access size.
__device__ __forceinline__ uint4 ld_dep_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_dep_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_dep_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ld_dep_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_dep_f32(const float* p) { return __uint_as_float(ld_dep_u32(p)); }
__device__ __forceinline__ float2 ld_dep_f32x2(const float* p) {
  const uint2 v = ld_dep_v2(p);
  return make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
}
__device__ __forceinline__ float ld_dep_bf16(const __nv_bfloat16* p) {
  return __uint_as_float((uint32_t)ld_dep_u16(p) << 16);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Device error word values (read back by mla_get_device_status).
constexpr int DEV_ERR_NONE = 0;
constexpr int DEV_ERR_RANGE = 1;    // a cache position outside the cache (or an invalid page)
constexpr int DEV_ERR_TIMEOUT = 2;  // a bounded wait gave up
constexpr int DEV_ERR_PLAN = 3;     // device lengths disagree with the host schedule

// Where position `pos` of sequence `b` lives in the latent cache (rows of LAT bf16 values).
//   dense (table == nullptr): an array [B, page, LAT]; row b * page + pos.
//   paged: a pool [num_pages, page, LAT] of pages of `page` positions (a multiple of 64, so a
//          64-position tile never crosses a page) and a block table [B, max_pages] of pool
//          pages; row table[b][pos / page] * page + pos % page.
// row() returns -1 for a logical page outside the table or a pool page outside the pool.
struct CacheRef {
  __nv_bfloat16* base;
  int page;              // dense: positions per sequence (the capacity); paged: per page
  const int* table;      // paged: device int32 [B, max_pages]; dense: nullptr
  int max_pages;
  int num_pages;
  __host__ __device__ bool paged() const { return table != nullptr; }
  __host__ __device__ long long capacity() const {
    return paged() ? (long long)page * max_pages : (long long)page;
  }
  // Rows of the array a tensor map covers (B sequences of a dense cache, or the pool).
  __host__ __device__ long long rows(int B) const {
    return paged() ? (long long)num_pages * page : (long long)B * page;
  }
  __device__ __forceinline__ long long row(int b, int pos) const {
    if (!paged()) return (long long)b * page + pos;
    const int lp = pos / page;
    if (pos < 0 || lp >= max_pages) return -1;
    const int pg = __ldg(table + (size_t)b * max_pages + lp);
    if (pg < 0 || pg >= num_pages) return -1;
    return (long long)pg * page + pos % page;
  }
};
inline CacheRef dense_cache(void* base, int cap) {
  return CacheRef{static_cast<__nv_bfloat16*>(base), cap, nullptr, 0, 0};
}

// One FP8 block-scaled projection: Y[m, n] = sum_k X[m, k] * W[n, k] * S[n/128][k/128].
struct Proj {
  const uint8_t* W;  // e4m3 [N, K]
  const float* S;    // [ceil(N/128), K/128]
  int N;
  void* Y;           // fp32 or bf16 output, row stride ldy elements
  int ldy;
  int y_fp32;        // 1: float32 output, 0: bf16 output
  // bf16 output only: a residual [M, ldy] added to the bf16-rounded product,
  // Y = bf16(R + bf16(XW^T)) (the decoder block's residual connection); nullptr: none.
  const __nv_bfloat16* R = nullptr;
};

// Two-term e4m3 split of two values already divided by their scale: hi = e4m3(f),
// lo = e4m3(f - hi), both rounded to nearest even with saturation; f ~ hi + lo to a relative
// 2^-8.  Returns the hi pair in bits 0..15 and the lo pair in bits 16..31 (first value in the
// low byte of each).
__device__ __forceinline__ uint32_t e4m3_split2(float2 f) {
  const __nv_fp8x2_storage_t hp = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hh = __nv_cvt_fp8x2_to_halfraw2(hp, __NV_E4M3);
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hh));
  const __nv_fp8x2_storage_t lp =
      __nv_cvt_float2_to_fp8x2(make_float2(f.x - hf.x, f.y - hf.y), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)hp | ((uint32_t)lp << 16);
}

// Projections of at most kGemvMaxM token rows run as weight-streaming GEMVs (k_gemv.cu: the
// CUDA cores for one or two tokens, mma.sync for three or four); larger ones run on the tcgen05
// GEMM.  Measured decode steps with 1,000 cached positions per sequence: 80.5 / 84.0 / 103.5 us
// with the GEMVs against 79.8 / 91.7 / 99.2 us with the tcgen05 GEMM for 3 / 4 / 8 sequences.
constexpr int kGemvMaxM = 4;

// Token-tile width of the tensor-core GEMM for M token rows.
constexpr int gemm_bn(int M) { return M <= 32 ? 32 : (M <= 64 ? 64 : 128); }

// Split-K factor of the tensor-core GEMM: 1 for large token counts (the tiles alone fill the
// SMs and fp32 partials would cost more than they save); for few tokens the one that minimises
// the k blocks of the busiest CTA, ceil(units / SMs) * ceil(k blocks / splits), the smaller on
// ties.
constexpr int gemm_splits(int M, int N_total, int K, int num_sms) {
  // K <= 1536 (q_b, kv_b): one split.  Their few k blocks per unit gain less from splitting
  // than the reduce launch and the fp32 partials cost (measured: decode B=64 168.5 -> 165.0 us,
  // prefill T=16 74.3 -> 72.3 us).
  if (M <= kGemvMaxM || M > 128 || K <= 1536) return 1;
  const int bn = gemm_bn(M);
  const long tiles = (long)((N_total + 127) / 128) * ((M + bn - 1) / bn);
  const int nkb = K / BLK;
  int best = 1;
  long best_cost = -1;
  for (int s = 1; s <= nkb / 2 || s == 1; ++s) {
    const long cost = ((tiles * s + num_sms - 1) / num_sms) * ((nkb + s - 1) / s);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// Scratch of one tensor-core GEMM: hi and lo e4m3 copies of X [M, K], sx [M], and the split-K
// partials (none for M <= kGemvMaxM, which runs as a GEMV).
constexpr size_t gemm_partial_bytes(int M, int N_total, int K, int num_sms) {
  if (M <= kGemvMaxM) return 0;
  const int s = gemm_splits(M, N_total, K, num_sms);
  const size_t mk = ((size_t)M * K + 255) & ~size_t(255);
  return 2 * mk + (((size_t)M * 4 + 255) & ~size_t(255)) +
         (s > 1 ? (size_t)s * M * N_total * sizeof(float) : 0);
}

// ---- launchers (each returns the launch's cudaError_t) ----------------------------------

// Y = X W^T for up to two projections sharing X [M, K] (row stride ldx elements).
// M <= kGemvMaxM runs as a weight-streaming GEMV; larger M runs on the tcgen05 tensor
// cores, split over K when the grid would be small, with fp32 partials in `partial`
// (gemm_partial_bytes bytes).  Block 0 of the launch also adds adv_by to adv[0..adv_n) (the
// call's length bookkeeping, riding on its last kernel; adv_n <= 128 with M <= kGemvMaxM).
cudaError_t launch_gemm(const __nv_bfloat16* X, int ldx, int M, int K, const Proj* p, int np,
                        float* partial, int num_sms, int* err, cudaStream_t st,
                        int* adv = nullptr, int adv_n = 0, int adv_by = 0, bool pdl = false);
bool gemm_can_advance(int M);  // whether launch_gemm honours adv for this M
// pdl: launch the split, GEMM and reduce kernels with programmatic dependent launch (each
// waits for its predecessor before touching its data; the GEMM requests its first weight
// tiles before that wait).
cudaError_t launch_gemm_tc(const __nv_bfloat16* X, int ldx, int M, int K, const Proj* p, int np,
                           float* partial, int num_sms, int* err, cudaStream_t st,
                           int* adv = nullptr, int adv_n = 0, int adv_by = 0, bool pdl = false);
// The same GEMM (M > kGemvMaxM) on activations already split into two e4m3 terms, hi and
// lo [M, K], with one scale per token, sx [M] (X[m, k] ~ sx[m] (hi + lo)), or with block_scales one per
// (token, 128-wide k block), sx [M, K/128] (X[m, k] ~ sx[m][k/128] (hi + lo)); block scales
// are accepted when gemm_takes_split_blocks(M).  `partial` as for launch_gemm_tc.
bool gemm_takes_split_blocks(int M);
// one_term (the FP8-activation option, with block_scales): the activations are the single
// e4m3 term hi (lo is not read), X[m, k] ~ sx[m][k/128] hi[m, k]: one MMA per k step.
cudaError_t launch_gemm_tc_split(const uint8_t* hi, const uint8_t* lo, const float* sx,
                                 bool block_scales, int M, int K, const Proj* p, int np,
                                 float* partial, int num_sms, int* err, cudaStream_t st,
                                 int* adv = nullptr, int adv_n = 0, int adv_by = 0,
                                 bool one_term = false, bool pdl = false);
// The FP8-activation option's input quantisation: q [M, K] = e4m3(X / sx) with one scale per
// (token, 128-wide group), sx [M, K/128] = amax / 448 (K a multiple of 128, at most 8192).
// The decode absorptions for many sequences as one batched tcgen05 GEMM over the 64 heads
// ("Key content up-projection" page; W_UK / W_UV are the two 128-row halves of each head's
// 256 rows of kv_b_proj): for head h and sequence b,
//   Y[b, h-th output block] = sum_k X[b, h, k] * W[w_row_base + h w_row_step + n, k] * scale,
// with X[b, h, 0 .. K) at X + b sb + h sh (bf16, written by the previous kernel), the weight's
// block scales at S + h s_step (row block of the head's rows, K / 128 columns), and output row
// b of head h at Y + h y_step + b ldy (bf16, N values).  The activations are split into two
// e4m3 terms per (sequence, head) row first (as launch_gemm_tc does per token).  With
// rope_out set, the split launch also writes RoPE of X[b, h, K .. K + 64) at position
// seq_lens[b] to rope_out[(b H + h) 576 .. + 64).  scratch: absorb_split_bytes(B, K) bytes.
size_t absorb_split_bytes(int B, int K);
cudaError_t launch_absorb_tc(const __nv_bfloat16* X, long long sb, int sh, int B, int K,
                             const uint8_t* W, long long w_rows, int w_row_base, int w_row_step,
                             const float* S, int s_step, int N, __nv_bfloat16* Y, int ldy,
                             long long y_step, __nv_bfloat16* rope_out, const float2* rope_tab,
                             int pairing, const int* seq_lens, int limit, void* scratch,
                             int num_sms, int* err, cudaStream_t st);
cudaError_t launch_quant_e4m3_groups(const __nv_bfloat16* X, int ldx, int M, int K, uint8_t* q,
                                     float* sx, cudaStream_t st, bool pdl = false);
cudaError_t init_gemm_tc_kernels();
cudaError_t init_gemv_kernels();

// RMSNorm of the q latent and kv latent, RoPE of k_pe, cache row store.  Positions at or
// past `limit` (min of cache capacity and RoPE table rows) are skipped and flagged in *err.
//   g1: fp32 [M, G1_N] (q_a | kv_a outputs), token m = b*T + t at position seq_lens[b] + t.
//   cq_out: bf16 [M, Q_LORA] normalised q latent (skipped if null).
//   ckv_out: bf16 [M, KV_LORA] normalised kv latent, the same values as the cache rows
//   (skipped if null).
//   q_split / kv_split (optional, instead of cq_out / ckv_out): those bf16 latents as the two
//   e4m3 terms and per-token scale that launch_gemm_tc_split reads (block_scales = false).
struct E4m3Split {
  uint8_t* hi;  // [M, n]
  uint8_t* lo;  // [M, n]
  float* sx;    // [M]
  // 1: the FP8-activation option's single term instead: hi = e4m3(v / s) with one scale per
  // (token, 128-wide group), sx [M, n/128]; lo is not written.
  int groups = 0;
};
cudaError_t launch_norm_rope_cache(const float* g1, int B, int T, const __nv_bfloat16* gq,
                                   const __nv_bfloat16* gkv, float eps, const float2* rope_tab,
                                   int rope_pairing, const int* seq_lens, const CacheRef& cache,
                                   int limit, __nv_bfloat16* cq_out,
                                   __nv_bfloat16* ckv_out, int* err, cudaStream_t st,
                                   bool pdl = false, const E4m3Split* q_split = nullptr,
                                   const E4m3Split* kv_split = nullptr);

// In-place RoPE of the rotary slice of q [M, HEADS, QHEAD] (prefill).
cudaError_t launch_rope_q(__nv_bfloat16* q, int B, int T, const float2* rope_tab,
                          int rope_pairing, const int* seq_lens, int limit, cudaStream_t st,
                          bool pdl = false);

// Decode query absorption: qfull[b, h] = [W_UK,h^T q_nope | RoPE(q_pe)] as bf16 [B, HEADS, LAT].
cudaError_t launch_absorb_q(const __nv_bfloat16* q, int B, const uint8_t* Wkvb,
                            const float* Skvb, const float2* rope_tab, int rope_pairing,
                            const int* seq_lens, int limit, __nv_bfloat16* qfull,
                            cudaStream_t st, bool pdl = false);

// Split-KV decode attention over the latent cache, then the log-sum-exp combine.
// The shares are cut from a line on which sequence b occupies K positions that hold no work
// (they stand for the cost of a segment: a query reload, a partial tile and an epilogue)
// followed by its seq_lens[b] + 1 real positions; K = 0 for a single sequence.
struct DecodePlan {
  int B;
  int G;            // CTAs: the line is cut into G equal shares
  long long P;      // length of the line, sum over b of (K + seq_lens[b] + 1)
  int K;            // positions charged per sequence
};
constexpr int kDecodeSeqCost = 96;
// First position (in the concatenation of all sequences) of CTA c's share.
__host__ __device__ inline long long decode_share_start(int c, int G, long long P) {
  return (long long)c * P / G;
}
// The CTA whose share holds position pos.
__host__ __device__ inline int decode_share_of(long long pos, int G, long long P) {
  int c = (int)((pos * G) / P);
  while (c + 1 < G && decode_share_start(c + 1, G, P) <= pos) ++c;
  while (c > 0 && decode_share_start(c, G, P) > pos) --c;
  return c;
}
// Partial slots used by a plan: sequence b's share in CTA c goes to slot b + c.
inline int decode_slots(const DecodePlan& p) { return p.B + p.G; }
// The plan for B sequences holding P positions in total, on num_sms SMs, with at most
// max_slots partial slots: about one share per SM (at most kMaxDecodeShares), at least 64
// positions per share.
constexpr int kMaxDecodeShares = 160;  // the combine kernel's bound on shares per sequence
inline DecodePlan make_decode_plan(int B, long long P, int num_sms, int max_slots) {
  long long G = (P + 63) / 64;
  if (G > num_sms) G = num_sms;
  if (G > kMaxDecodeShares) G = kMaxDecodeShares;
  if (G > max_slots - B) G = max_slots - B;
  if (G < 1) G = 1;
  const int K = B > 1 ? kDecodeSeqCost : 0;
  return DecodePlan{B, (int)G, P + (long long)B * K, K};
}
cudaError_t launch_decode_combine(const int* seq_lens, DecodePlan plan, const __half* o_part,
                                  const float* ml_part, __nv_bfloat16* o_lat, int* err,
                                  cudaStream_t st, bool pdl = false);

// Decode for a few sequences: the combine fused with the output absorption (one CTA per
// head and sequence), and q_b_proj fused with the q-latent norm plus the kv cache-row append.
cudaError_t launch_qb_norm(const float* g1, int M, const Proj& p, const __nv_bfloat16* gq,
                           const __nv_bfloat16* gkv, float eps, const float2* rope_tab,
                           int rope_pairing, const int* seq_lens, const CacheRef& cache,
                           int limit, int* err, int num_sms, cudaStream_t st, bool pdl = false);
cudaError_t launch_combine_absorb_out(const int* seq_lens, const int* lens_host,
                                      DecodePlan plan, const __half* o_part,
                                      const float* ml_part, const uint8_t* Wkvb,
                                      const float* Skvb, __nv_bfloat16* attn, int* err,
                                      cudaStream_t st, bool pdl = false);

// Split-KV decode attention over the latent cache on the tcgen05 tensor cores (TMA-fed,
// accumulators in tensor memory): per work item, unnormalised partial outputs and (m, l).
// Each sequence's share is read in 64-position tiles from the share's first position; with a
// paged cache the tiles start at multiples of 64 within the sequence instead (positions
// before the share's start are masked), so a tile never crosses a page.
// head_major: partials laid out [slot][head][dim] (read by the combine fused with W_UV)
// instead of [slot][dim][head] (read by the stand-alone combine).
cudaError_t launch_decode_attention_tc(const __nv_bfloat16* qfull, const CacheRef& cache,
                                       const int* seq_lens, DecodePlan plan,
                                       float scale, __half* o_part, float* ml_part, int* err,
                                       cudaStream_t st, bool pdl = false, bool head_major = false);
cudaError_t init_decode_tc_kernel();

// Device address of mla_decode_noalloc's static scratch array on the current device.
cudaError_t noalloc_scratch_address(void** out);

// One CTA waits on an mbarrier that nothing arrives at, with the library's bounded wait and
// the given limit; it records DEV_ERR_TIMEOUT in *err when the limit runs out.
cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t st);

// One-time kernel attributes (dynamic shared memory opt-in); called by mla_create so that
// later calls only enqueue work and can be captured into CUDA graphs.
cudaError_t init_kernels();

// Decode output absorption: out[b, h*VDIM + v] = sum_c W_UV,h[v, c] o_lat[b, h, c].
// W_UK^T: out[h][c][i] = Wkvb[256 h + i][c] (e4m3 bytes) for the batched query absorption.
cudaError_t launch_transpose_wuk(const uint8_t* Wkvb, uint8_t* out, cudaStream_t st);
// Decode with at least kAbsorbTcMinB sequences runs both absorptions as batched tcgen05 GEMMs
// (launch_absorb_tc); fewer keep the CUDA-core kernels.
constexpr int kAbsorbTcMinB = 9;
// Prefill calls with at most this many tokens launch every kernel after the first with
// programmatic dependent launch.  Measured: T=16 78.6 -> 74.3 us, a 16-token chunk after 300
// positions 92.8 -> 85.2 us, a 1024-token chunk after 4096 0.503 -> 0.497 ms; T=4096 1.033 ->
// 1.038 ms (slower: the early GEMM CTAs take SMs from the large kernels before them).
constexpr int kPrefillPdlMaxM = 2048;
cudaError_t launch_absorb_out(const __nv_bfloat16* o_lat, int B, const uint8_t* Wkvb,
                              const float* Skvb, __nv_bfloat16* out, cudaStream_t st,
                              bool pdl = false);

// Causal prefill attention on the tcgen05 tensor cores: q [M, HEADS, QHEAD] (rotated),
// kv [M, HEADS, 256] (k_nope | v), rotated k_pe from the cache rows; writes attn_out
// [M, HEADS*VDIM] bf16.
// The output goes to attn_out as bf16 [B*T, HEADS*VDIM], or, when o_hi/o_lo/o_sx are given
// (attn_out may then be null), as the two e4m3 terms of those bf16 values, [B*T, HEADS*VDIM]
// each, with one scale per (token, head) in o_sx [B*T, HEADS] (the input of
// launch_gemm_tc_split).
// Queries: q [B*T, HEADS, QHEAD]; sequence b has seq_lens[b] cached positions before this call
// (seq_lens null: none), and its keys/values are rows kvr0(b) .. kvr0(b) + L_b + T - 1 of kv
// [kv_rows, HEADS, KVB_PER_HEAD] with kvr0(b) = sum over b' < b of (L_b' + T); the rotary keys
// come from the cache rows.  Query t of sequence b sees positions 0 .. L_b + t.
cudaError_t launch_prefill_attention_tc(const __nv_bfloat16* q, const __nv_bfloat16* kv,
                                        const CacheRef& cache, int B, int T,
                                        const int* seq_lens, long kv_rows, float scale,
                                        __nv_bfloat16* attn_out, uint8_t* o_hi, uint8_t* o_lo,
                                        float* o_sx, int num_sms, int* err, cudaStream_t st,
                                        bool pdl = false);
cudaError_t init_prefill_tc_kernel();

// Chunked prefill over a paged cache: the normalised latents (the first KV_LORA values) of
// every sequence's cache rows 0 .. seq_lens[b] + T - 1, packed sequence after sequence into
// out [kv_rows, KV_LORA] bf16 (the layout the kv_b_proj of launch_prefill_attention_tc's keys
// and values expects).  max_len >= seq_lens[b] + T bounds the grid; a layout that does not
// fit kv_rows, or an invalid page, is flagged in *err and its rows are skipped.
cudaError_t launch_gather_latent(const CacheRef& cache, const int* seq_lens, int B, int T,
                                 int max_len, long kv_rows, __nv_bfloat16* out, int* err,
                                 cudaStream_t st, bool pdl = false);

// The decoder block's input RMSNorm: xn[m] = bf16(g * bf16(x[m] * rsqrt(mean(x[m]^2) + eps)))
// for M rows of HIDDEN bf16 values.
cudaError_t launch_input_norm(const __nv_bfloat16* x, int M, const __nv_bfloat16* g, float eps,
                              __nv_bfloat16* xn, cudaStream_t st, bool pdl = false);

// seq_lens[b] += T.
cudaError_t launch_advance_lens(int* seq_lens, int B, int T, cudaStream_t st, bool pdl = false);
// bytes (a multiple of 16, both addresses 16-byte aligned) from src to dst by a kernel, for
// copies to or from page-locked host memory that the device addresses directly.  wait_prev:
// the source is the previous kernel's output (read after programmatic launch's wait).
cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, bool wait_prev,
                          cudaStream_t st, bool pdl);

// out[r][c] = float(e4m3(W[r][c])) * S[r/128][c/128].
cudaError_t launch_dequant(const uint8_t* W, const float* S, int rows, int cols, float* out,
                           cudaStream_t st);

}  // namespace mla

// Host-side state of one context (the opaque mla_ctx of the C ABI).
struct mla_ctx {
  mla_config cfg;
  int device = 0;
  int num_sms = 0;
  const uint8_t* W[5] = {};
  const float* S[5] = {};
  const __nv_bfloat16* gain[3] = {};  // q_a_layernorm, kv_a_layernorm, input_layernorm
  float2* rope_tab = nullptr;  // [max_positions][32] (cos, sin)
  int* d_err = nullptr;
  // W_UK of every head transposed, [64][512][128] e4m3 (the batched query absorption's weight
  // operand, K-major), allocated when kv_b_proj is registered and rebuilt on the stream of the
  // first call that needs it after each registration.
  uint8_t* wuk_t = nullptr;
  bool wuk_t_stale = true;
  // Device address, on this context's device, of the static scratch array that
  // mla_decode_noalloc uses (looked up by mla_create, with the device current).
  void* noalloc_scratch = nullptr;
  // Testing aid, from the environment variable MLA_TEST_FAIL_AFTER at creation: when >= 0,
  // every token call fails at its launch with this index, as if that CUDA launch had failed
  // (the launches before it are enqueued; it and the rest are not).  -1: off.
  int fail_at = -1;
  // Launch log of the most recent token call (names, and device timings when profiling).
  static constexpr int kMaxLaunch = 32;
  bool profiling = false;
  bool last_profiled = false;
  int n_launch = 0;
  const char* names[kMaxLaunch] = {};
  cudaEvent_t ev[2 * kMaxLaunch] = {};
};
