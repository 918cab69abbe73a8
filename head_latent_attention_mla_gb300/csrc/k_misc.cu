// Elementwise and small kernels of the MLA layer: latent RMSNorms with RoPE and the cache
// store, query RoPE, decode-side W_UK / W_UV absorption, length bookkeeping and the FP8
// dequantisation export.
#include "mla_internal.h"

namespace mla {

namespace {

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t v) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
  return __half2float(__half(h));
}

// Block-wide sum of two values (256 threads).
__device__ __forceinline__ float2 block_max2(float a, float b, float2* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, off));
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = make_float2(a, b);
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  if (threadIdx.x < 32) {
    t = (l < (int)(blockDim.x >> 5)) ? red[l] : make_float2(0.f, 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      t.x = fmaxf(t.x, __shfl_xor_sync(0xffffffffu, t.x, off));
      t.y = fmaxf(t.y, __shfl_xor_sync(0xffffffffu, t.y, off));
    }
    if (l == 0) red[8] = t;
  }
  __syncthreads();
  return red[8];
}

// Eight consecutive values v of one token, starting at element `at` of the split rows, as two
// e4m3 terms with the token's scale s = amax / 448 (1 for an all-zero row): hi = e4m3(v / s),
// lo = e4m3(v / s - hi), the split the tensor-core GEMM's own activation pass would make.
__device__ __forceinline__ void store_e4m3_split8(const float (&v)[8], float amax, size_t at,
                                                  const E4m3Split& o) {
  const float s = amax > 0.f ? amax / 448.f : 1.f;
  const float inv = 1.f / s;
  uint32_t h[2] = {0u, 0u}, l[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t hl = e4m3_split2(make_float2(v[2 * i] * inv, v[2 * i + 1] * inv));
    h[i >> 1] |= (hl & 0xFFFFu) << (16 * (i & 1));
    l[i >> 1] |= (hl >> 16) << (16 * (i & 1));
  }
  *reinterpret_cast<uint2*>(o.hi + at) = make_uint2(h[0], h[1]);
  *reinterpret_cast<uint2*>(o.lo + at) = make_uint2(l[0], l[1]);
}

__device__ __forceinline__ float2 block_sum2(float a, float b, float2* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    b += __shfl_xor_sync(0xffffffffu, b, off);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = make_float2(a, b);
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  if (threadIdx.x < 32) {
    t = (l < (int)(blockDim.x >> 5)) ? red[l] : make_float2(0.f, 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      t.x += __shfl_xor_sync(0xffffffffu, t.x, off);
      t.y += __shfl_xor_sync(0xffffffffu, t.y, off);
    }
    if (l == 0) red[8] = t;
  }
  __syncthreads();
  return red[8];
}

// RoPE of one pair (a, b) by the table entry (cos, sin): (a c - b s, b c + a s).
__device__ __forceinline__ float2 rotate(float a, float b, float2 cs) {
  return make_float2(a * cs.x - b * cs.y, b * cs.x + a * cs.y);
}

// Element indices of pair j in a 64-wide rotary slice.
__device__ __forceinline__ int2 pair_idx(int j, int pairing) {
  return pairing == 0 ? make_int2(2 * j, 2 * j + 1) : make_int2(j, j + ROPE / 2);
}

// One CTA (256 threads) per token; threads 0..191 own eight consecutive q-latent values each,
// threads 192..255 eight kv-latent values (16-byte loads and stores).
// RMSNorm ("rmsnorm" excerpt): y = g * bf16(x * rsqrt(mean(x^2) + eps)), rounded to bf16,
// for the q latent (1536) and the kv latent (512); the kv latent and the rotated shared
// rotary key form the token's cache row [c_hat (512) | RoPE(k_pe) (64)].
constexpr int NRC_QT = Q_LORA / 8;  // q threads
static_assert(NRC_QT + KV_LORA / 8 == 256, "one 8-value run per thread");
__global__ void __launch_bounds__(256) norm_rope_cache_kernel(
    const float* g1, int T, const __nv_bfloat16* __restrict__ gq,
    const __nv_bfloat16* __restrict__ gkv, float eps, const float2* __restrict__ rope_tab,
    int pairing, const int* __restrict__ seq_lens, const CacheRef cache, int limit, __nv_bfloat16* __restrict__ cq_out, __nv_bfloat16* __restrict__ ckv_out, int* err,
    E4m3Split q_split, E4m3Split kv_split) {
  __shared__ float2 red[9], red2[9];
  __shared__ __align__(16) __nv_bfloat16 row[LAT];
  pdl_launch_dependents();
  pdl_wait();
  const int token = blockIdx.x, b = token / T, t = token % T;
  const int tid = threadIdx.x;
  const float* in = g1 + (size_t)token * G1_N;
  const bool do_q = cq_out != nullptr || q_split.hi != nullptr;
  const bool is_q = tid < NRC_QT;
  const int c0 = is_q ? 8 * tid : 8 * (tid - NRC_QT);  // first element within its latent

  float x[8] = {};
  float sq = 0.f, sk = 0.f;
  if (!is_q || do_q) {
    const float* src = in + (is_q ? 0 : Q_LORA) + c0;
    const uint4 a = ld_dep_v4(src), b4 = ld_dep_v4(src + 4);
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b4.x); x[5] = __uint_as_float(b4.y);
    x[6] = __uint_as_float(b4.z); x[7] = __uint_as_float(b4.w);
    float s2 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s2 += x[i] * x[i];
    (is_q ? sq : sk) = s2;
  }
  const float2 ss = block_sum2(sq, sk, red);
  const float rs = is_q ? rsqrtf(ss.x / Q_LORA + eps) : rsqrtf(ss.y / KV_LORA + eps);
  float y[8];  // the bf16 outputs, as floats
  float am = 0.f;
  if (!is_q || do_q) {
    const uint4 gv = *reinterpret_cast<const uint4*>((is_q ? gq : gkv) + c0);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t ow[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat16 y0 =
          __float2bfloat16_rn(__uint_as_float(gw[i] << 16) * bf16_round(x[2 * i] * rs));
      const __nv_bfloat16 y1 =
          __float2bfloat16_rn(__uint_as_float(gw[i] & 0xFFFF0000u) * bf16_round(x[2 * i + 1] * rs));
      y[2 * i] = __bfloat162float(y0);
      y[2 * i + 1] = __bfloat162float(y1);
      am = fmaxf(am, fmaxf(fabsf(y[2 * i]), fabsf(y[2 * i + 1])));
      ow[i] = (uint32_t)__bfloat16_as_ushort(y0) | ((uint32_t)__bfloat16_as_ushort(y1) << 16);
    }
    const uint4 o4 = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    if (is_q) {
      if (cq_out) *reinterpret_cast<uint4*>(cq_out + (size_t)token * Q_LORA + c0) = o4;
    } else {
      *reinterpret_cast<uint4*>(row + c0) = o4;
      if (ckv_out) *reinterpret_cast<uint4*>(ckv_out + (size_t)token * KV_LORA + c0) = o4;
    }
  }
  const bool grouped = q_split.hi != nullptr ? q_split.groups != 0 : kv_split.groups != 0;
  if ((q_split.hi != nullptr || kv_split.hi != nullptr) && grouped) {  // the same for every CTA
    // Single e4m3 term with one scale per 128-wide group: the group is 16 consecutive threads.
    float g = am;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, off));
    const E4m3Split& o = is_q ? q_split : kv_split;
    if ((!is_q || do_q) && o.hi != nullptr) {
      const float sg = g > 0.f ? g / 448.f : 1.f, inv = 1.f / sg;
      const int n = is_q ? Q_LORA : KV_LORA;
      uint32_t h[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_fp8x2_storage_t pk = __nv_cvt_float2_to_fp8x2(
            make_float2(y[2 * i] * inv, y[2 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
        h[i >> 1] |= (uint32_t)pk << (16 * (i & 1));
      }
      *reinterpret_cast<uint2*>(o.hi + (size_t)token * n + c0) = make_uint2(h[0], h[1]);
      if ((tid & 15) == 0) o.sx[(size_t)token * (n / BLK) + c0 / BLK] = sg;
    }
  } else if (q_split.hi != nullptr || kv_split.hi != nullptr) {  // the same for every CTA
    const float2 m2 = block_max2(is_q ? am : 0.f, is_q ? 0.f : am, red2);
    if (is_q && do_q && q_split.hi != nullptr) {
      store_e4m3_split8(y, m2.x, (size_t)token * Q_LORA + c0, q_split);
      if (tid == 0) q_split.sx[token] = m2.x > 0.f ? m2.x / 448.f : 1.f;
    }
    if (!is_q && kv_split.hi != nullptr) {
      store_e4m3_split8(y, m2.y, (size_t)token * KV_LORA + c0, kv_split);
      if (tid == NRC_QT) kv_split.sx[token] = m2.y > 0.f ? m2.y / 448.f : 1.f;
    }
  }
  const int pos = seq_lens[b] + t;
  // Device lengths past the cache or the RoPE table, or an invalid page: skipped and flagged.
  const long long crow = (pos < 0 || pos >= limit) ? -1 : cache.row(b, pos);
  if (crow < 0) {
    if (tid == 0) atomicExch(err, DEV_ERR_RANGE);
    return;
  }
  if (tid < ROPE / 2) {
    const int2 ij = pair_idx(tid, pairing);
    const float* kr = in + Q_LORA + KV_LORA;
    const float2 r = rotate(ld_dep_f32(kr + ij.x), ld_dep_f32(kr + ij.y),
                            rope_tab[(size_t)pos * (ROPE / 2) + tid]);
    row[KV_LORA + ij.x] = __float2bfloat16_rn(r.x);
    row[KV_LORA + ij.y] = __float2bfloat16_rn(r.y);
  }
  __syncthreads();
  if (tid < LAT / 8) {
    uint4* dst = reinterpret_cast<uint4*>(cache.base + (size_t)crow * LAT);
    dst[tid] = reinterpret_cast<const uint4*>(row)[tid];
  }
}

// The decoder block's input RMSNorm ("rmsnorm" excerpt over the hidden size): one CTA of 224
// threads per token, each with four 16-byte runs of 8 values.
constexpr int IN_THREADS = HIDDEN / 32;
__global__ void __launch_bounds__(IN_THREADS) input_norm_kernel(const __nv_bfloat16* __restrict__ x,
                                                                const __nv_bfloat16* __restrict__ g,
                                                                float eps,
                                                                __nv_bfloat16* __restrict__ xn) {
  __shared__ float red[IN_THREADS / 32];
  pdl_launch_dependents();
  pdl_wait();
  const int m = blockIdx.x, tid = threadIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)m * HIDDEN);
  uint4 v[4];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = src[tid + IN_THREADS * i];
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = __uint_as_float(w[e] << 16), b = __uint_as_float(w[e] & 0xFFFF0000u);
      ss += a * a + b * b;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < IN_THREADS / 32; ++w) tot += red[w];
  const float rs = rsqrtf(tot / HIDDEN + eps);
  uint4* dst = reinterpret_cast<uint4*>(xn + (size_t)m * HIDDEN);
  const uint4* gs = reinterpret_cast<const uint4*>(g);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 gv = gs[tid + IN_THREADS * i];
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16 y0 = __float2bfloat16_rn(__uint_as_float(gw[e] << 16) *
                                                   bf16_round(__uint_as_float(w[e] << 16) * rs));
      const __nv_bfloat16 y1 = __float2bfloat16_rn(
          __uint_as_float(gw[e] & 0xFFFF0000u) * bf16_round(__uint_as_float(w[e] & 0xFFFF0000u) * rs));
      o[e] = (uint32_t)__bfloat16_as_ushort(y0) | ((uint32_t)__bfloat16_as_ushort(y1) << 16);
    }
    dst[tid + IN_THREADS * i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Row t of sequence b's latents (its first KV_LORA cache values) to row r0(b) + t of out, with
// r0(b) = sum over b' < b of (seq_lens[b'] + T): one CTA (64 threads, 16 bytes each) per row.
__global__ void __launch_bounds__(KV_LORA / 8) gather_latent_kernel(
    const CacheRef cache, const int* __restrict__ seq_lens, int T, long kv_rows,
    __nv_bfloat16* __restrict__ out, int* err) {
  pdl_launch_dependents();
  pdl_wait();  // the cache rows of this call come from the norm kernel
  const int t = blockIdx.x, b = blockIdx.y;
  const int n = seq_lens[b] + T;
  if (t >= n) return;
  long r0 = 0;
  for (int bb = 0; bb < b; ++bb) r0 += seq_lens[bb] + T;
  const long long crow = cache.row(b, t);
  if (r0 + n > kv_rows || crow < 0) {  // the host's layout or the block table is wrong
    if (threadIdx.x == 0) atomicExch(err, crow < 0 ? DEV_ERR_RANGE : DEV_ERR_PLAN);
    return;
  }
  const uint4 v = ld_dep_v4(cache.base + (size_t)crow * LAT + 8 * threadIdx.x);
  reinterpret_cast<uint4*>(out + (size_t)(r0 + t) * KV_LORA)[threadIdx.x] = v;
}

// In-place RoPE of q's rotary slices.  One CTA per RQ_TOK tokens; eight threads per head,
// each with one 16-byte chunk (8 values) of the head's 64 rotary values in every token, so a
// warp reads and writes four whole 128-byte slices per token and each thread keeps RQ_TOK
// loads in flight.  Adjacent pairs lie inside a chunk; half pairs (j, j + 32) join chunk c and
// chunk c + 4, which swap values with a shuffle.  The tokens' angles are staged once in
// shared memory; tokens whose position lies outside [0, limit) are left as they are.
constexpr int RQ_TOK = 4;
__global__ void __launch_bounds__(HEADS * 8) rope_q_kernel(__nv_bfloat16* __restrict__ q, int M,
                                                           int T,
                                                           const float2* __restrict__ rope_tab,
                                                           int pairing,
                                                           const int* __restrict__ seq_lens,
                                                           int limit) {
  __shared__ float2 cs[RQ_TOK][ROPE / 2];
  __shared__ int live[RQ_TOK];
  pdl_launch_dependents();
  pdl_wait();  // q comes from the q_b projection
  const int tok0 = blockIdx.x * RQ_TOK;
  if (threadIdx.x < RQ_TOK * (ROPE / 2)) {
    const int k = threadIdx.x / (ROPE / 2), j = threadIdx.x % (ROPE / 2), token = tok0 + k;
    int pos = -1;
    if (token < M) pos = seq_lens[token / T] + token % T;
    const bool ok = pos >= 0 && pos < limit;
    cs[k][j] = ok ? rope_tab[(size_t)pos * (ROPE / 2) + j] : make_float2(1.f, 0.f);
    if (j == 0) live[k] = ok;
  }
  __syncthreads();
  const int h = threadIdx.x >> 3, c = threadIdx.x & 7;
  uint4 v[RQ_TOK];
#pragma unroll
  for (int k = 0; k < RQ_TOK; ++k)
    if (live[k])
      v[k] = reinterpret_cast<const uint4*>(q + ((size_t)(tok0 + k) * HEADS + h) * QHEAD + NOPE)[c];
#pragma unroll
  for (int k = 0; k < RQ_TOK; ++k) {
    if (!live[k]) continue;  // the same for the whole CTA
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    float f[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(w[e] << 16);
      f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
    if (pairing == 0) {  // pair j = 4c + e is (f[2e], f[2e + 1])
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 r = rotate(f[2 * e], f[2 * e + 1], cs[k][4 * c + e]);
        f[2 * e] = r.x;
        f[2 * e + 1] = r.y;
      }
    } else {  // pair j = 8 (c % 4) + i is (value i of chunk c % 4, value i of chunk c % 4 + 4)
      float g[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = __shfl_xor_sync(0xffffffffu, f[i], 4);
      const bool first = c < 4;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 a = cs[k][8 * (c & 3) + i];
        f[i] = first ? f[i] * a.x - g[i] * a.y : f[i] * a.x + g[i] * a.y;
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 v2 = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
      o[e] = *reinterpret_cast<const uint32_t*>(&v2);
    }
    reinterpret_cast<uint4*>(q + ((size_t)(tok0 + k) * HEADS + h) * QHEAD + NOPE)[c] =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* f) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFF), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
  float2 c = __half22float2(*reinterpret_cast<__half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = c.x; f[3] = c.y;
}

// Decode query absorption, q~_h = W_UK,h^T q_nope,h with W_UK,h = rows 0..127 of head h's 256
// in kv_b_proj ("Key content up-projection" page, Explanation):
//   qfull[b, h, c] = bf16( s[2h][c/128] * sum_i q_nope[b, h, i] * e4m3(W_kvb[256 h + i, c]) ).
// CTA (h, cb, z) owns latent columns [128 cb, 128 cb + 128) (one scale) of sequences
// [8 z, 8 z + 8); warp w sums rows i in [32 w, 32 w + 32) for 4 columns per lane, and the 4
// warps' partials meet in shared memory.  The cb == 0 CTAs also write RoPE(q_pe) to columns
// [512, 576).
constexpr int ABQ_B = 8;
__global__ void __launch_bounds__(128) absorb_q_kernel(
    const __nv_bfloat16* q, int B, const uint8_t* __restrict__ Wkvb,
    const float* __restrict__ Skvb, const float2* __restrict__ rope_tab, int pairing,
    const int* __restrict__ seq_lens, int limit, __nv_bfloat16* __restrict__ qfull) {
  __shared__ float qn[ABQ_B][NOPE];
  __shared__ float4 part[4][ABQ_B][32];
  const int h = blockIdx.x, cb = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float sc = Skvb[(size_t)(2 * h) * (KV_LORA / BLK) + cb];
  // This lane's 32 rows x 4 columns of W_UK,h, kept in registers across the batch.
  float w[32][4];
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(
        Wkvb + (size_t)(h * KVB_PER_HEAD + warp * 32 + r) * KV_LORA + cb * BLK + lane * 4));
    e4m3x4_to_f32(v, w[r]);
  }
  pdl_launch_dependents();
  pdl_wait();  // the weights above do not depend on earlier kernels; q does
  {
    const int b0 = blockIdx.z * ABQ_B;  // this CTA's batch of sequences
    const int nb = min(ABQ_B, B - b0);
    for (int e = threadIdx.x; e < nb * NOPE; e += blockDim.x) {
      const int bb = e / NOPE, i = e % NOPE;
      qn[bb][i] = ld_dep_bf16(q + ((size_t)(b0 + bb) * HEADS + h) * QHEAD + i);
    }
    __syncthreads();
    for (int bb = 0; bb < nb; ++bb) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const float x = qn[bb][warp * 32 + r];
        acc.x = fmaf(x, w[r][0], acc.x);
        acc.y = fmaf(x, w[r][1], acc.y);
        acc.z = fmaf(x, w[r][2], acc.z);
        acc.w = fmaf(x, w[r][3], acc.w);
      }
      part[warp][bb][lane] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nb * 32; e += blockDim.x) {
      const int bb = e / 32, l = e % 32;
      float4 t = part[0][bb][l];
#pragma unroll
      for (int ww = 1; ww < 4; ++ww) {
        const float4 u = part[ww][bb][l];
        t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
      }
      __nv_bfloat162 lo = __floats2bfloat162_rn(sc * t.x, sc * t.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(sc * t.z, sc * t.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(qfull + ((size_t)(b0 + bb) * HEADS + h) * LAT + cb * BLK + l * 4) = pk;
    }
  }
  if (cb == 0) {
    for (int e = threadIdx.x; e < min(ABQ_B, B - (int)blockIdx.z * ABQ_B) * (ROPE / 2);
         e += blockDim.x) {
      const int bb = blockIdx.z * ABQ_B + e / (ROPE / 2), j = e % (ROPE / 2);
      const int pos = seq_lens[bb];
      if (pos < 0 || pos >= limit) continue;
      const int2 ij = pair_idx(j, pairing);
      const __nv_bfloat16* qp = q + ((size_t)bb * HEADS + h) * QHEAD + NOPE;
      const float2 r = rotate(ld_dep_bf16(qp + ij.x), ld_dep_bf16(qp + ij.y),
                              rope_tab[(size_t)pos * (ROPE / 2) + j]);
      __nv_bfloat16* dst = qfull + ((size_t)bb * HEADS + h) * LAT + KV_LORA;
      dst[ij.x] = __float2bfloat16_rn(r.x);
      dst[ij.y] = __float2bfloat16_rn(r.y);
    }
  }
}

// Decode output absorption, one warp per output row (h, v):
//   out[b, 128 h + v] = bf16( sum_c s[2h+1][c/128] * e4m3(W_kvb[256 h + 128 + v, c]) * o_lat[b, h, c] )
// (W_UV,h = rows 128..255 of head h's 256).  Lane l holds columns [16 l, 16 l + 16).  The
// CTA's 8 rows belong to one head, whose o_lat rows it stages in shared memory 32 sequences at
// a time (each row of o_lat is then read from L2 once per CTA, not once per warp).
constexpr int ABO_B = 8;
constexpr int ABO_CH = 32;  // sequences staged in shared memory at a time (32 KB)
__global__ void __launch_bounds__(256) absorb_out_kernel(
    const __nv_bfloat16* o_lat, int B, const uint8_t* __restrict__ Wkvb,
    const float* __restrict__ Skvb, __nv_bfloat16* __restrict__ out) {
  __shared__ __align__(16) __nv_bfloat16 xs[ABO_CH][KV_LORA];  // o_lat of this head
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;   // h * 128 + v
  const int lane = threadIdx.x & 31;
  const int h = row / VDIM, v = row % VDIM;  // h: the same for the CTA's 8 rows
  const uint4 wv = __ldg(reinterpret_cast<const uint4*>(
      Wkvb + (size_t)(h * KVB_PER_HEAD + NOPE + v) * KV_LORA + lane * 16));
  float w[16];
  e4m3x4_to_f32(wv.x, w);
  e4m3x4_to_f32(wv.y, w + 4);
  e4m3x4_to_f32(wv.z, w + 8);
  e4m3x4_to_f32(wv.w, w + 12);
  const float sc = Skvb[(size_t)(2 * h + 1) * (KV_LORA / BLK) + lane / 8];
  pdl_launch_dependents();
  pdl_wait();  // the weights above do not depend on earlier kernels; o_lat does
  for (int c0 = 0; c0 < B; c0 += ABO_CH) {
    // The head's o_lat rows of sequences [c0, c0 + nc), read once for the CTA's 8 rows.
    const int nc = min(ABO_CH, B - c0);
    __syncthreads();
    for (int e = threadIdx.x; e < nc * (KV_LORA / 8); e += blockDim.x) {
      const int bb = e / (KV_LORA / 8), k = e % (KV_LORA / 8);
      reinterpret_cast<uint4*>(xs[bb])[k] =
          ld_dep_v4(o_lat + ((size_t)(c0 + bb) * HEADS + h) * KV_LORA + 8 * k);
    }
    __syncthreads();
    for (int b0 = 0; b0 < nc; b0 += ABO_B) {
      float acc[ABO_B];
#pragma unroll
      for (int bb = 0; bb < ABO_B; ++bb) {
        acc[bb] = 0.f;
        if (b0 + bb < nc) {
          const uint4* xp = reinterpret_cast<const uint4*>(xs[b0 + bb] + lane * 16);
          const uint4 x0 = xp[0], x1 = xp[1];
          const uint32_t u[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          float p = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            p = fmaf(w[2 * i], __uint_as_float(u[i] << 16), p);
            p = fmaf(w[2 * i + 1], __uint_as_float(u[i] & 0xFFFF0000u), p);
          }
          acc[bb] = sc * p;
        }
      }
#pragma unroll
      for (int bb = 0; bb < ABO_B; ++bb) {
        float t = acc[bb];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if (lane == 0 && b0 + bb < nc)
          out[(size_t)(c0 + b0 + bb) * O_IN + row] = __float2bfloat16_rn(t);
      }
    }
  }
}

__global__ void advance_lens_kernel(int* seq_lens, int B, int T) {
  pdl_launch_dependents();
  pdl_wait();  // every reader of the lengths in this call is done
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) seq_lens[b] += T;
}

// n 16-byte words from src to dst, one of them page-locked host memory that the device
// addresses directly (the input and output copies of a decode call with host buffers).  The
// next kernel may start at once; with wait_prev the source is the previous kernel's output,
// read after it has finished.
__global__ void copy16_kernel(const uint4* src, uint4* dst, size_t n, int wait_prev) {
  pdl_launch_dependents();
  if (wait_prev) pdl_wait();
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = ld_dep_v4(src + i);
}

__global__ void dequant_kernel(const uint8_t* __restrict__ W, const float* __restrict__ S,
                               int rows, int cols, float* __restrict__ out) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)rows * cols) return;
  const int r = (int)(i / cols), c = (int)(i % cols);
  const int kb = (cols + BLK - 1) / BLK;
  out[i] = __fmul_rn(e4m3_to_f32(W[i]), S[(size_t)(r / BLK) * kb + c / BLK]);
}

}  // namespace

cudaError_t launch_norm_rope_cache(const float* g1, int B, int T, const __nv_bfloat16* gq,
                                   const __nv_bfloat16* gkv, float eps, const float2* rope_tab,
                                   int rope_pairing, const int* seq_lens, const CacheRef& cache,
                                   int limit, __nv_bfloat16* cq_out,
                                   __nv_bfloat16* ckv_out, int* err, cudaStream_t st, bool pdl,
                                   const E4m3Split* q_split, const E4m3Split* kv_split) {
  if (B * T == 0) return cudaSuccess;
  const E4m3Split none{nullptr, nullptr, nullptr, 0};
  return launch_kernel(norm_rope_cache_kernel, dim3(B * T), dim3(256), 0, st, pdl, g1, T, gq, gkv,
                       eps, rope_tab, rope_pairing, seq_lens, cache, limit, cq_out, ckv_out,
                       err, q_split ? *q_split : none, kv_split ? *kv_split : none);
}

cudaError_t launch_input_norm(const __nv_bfloat16* x, int M, const __nv_bfloat16* g, float eps,
                              __nv_bfloat16* xn, cudaStream_t st, bool pdl) {
  if (M <= 0) return cudaSuccess;
  return launch_kernel(input_norm_kernel, dim3(M), dim3(IN_THREADS), 0, st, pdl, x, g, eps, xn);
}

cudaError_t launch_gather_latent(const CacheRef& cache, const int* seq_lens, int B, int T,
                                 int max_len, long kv_rows, __nv_bfloat16* out, int* err,
                                 cudaStream_t st, bool pdl) {
  if (B * T == 0 || max_len <= 0) return cudaSuccess;
  return launch_kernel(gather_latent_kernel, dim3(max_len, B), dim3(KV_LORA / 8), 0, st, pdl,
                       cache, seq_lens, T, kv_rows, out, err);
}

cudaError_t launch_rope_q(__nv_bfloat16* q, int B, int T, const float2* rope_tab,
                          int rope_pairing, const int* seq_lens, int limit, cudaStream_t st,
                          bool pdl) {
  if (B * T == 0) return cudaSuccess;
  const int M = B * T;
  return launch_kernel(rope_q_kernel, dim3((M + RQ_TOK - 1) / RQ_TOK), dim3(HEADS * 8), 0, st, pdl,
                       q, M, T, rope_tab, rope_pairing, seq_lens, limit);
}

// The same output absorption for many sequences (B > 8) as a small tiled product per head:
// CTA (h, vb) computes out[b, 128 h + v] for the 32 rows v in [32 vb, 32 vb + 32) and every
// sequence.  It stages W_UV,h's 32 rows as fp32 with their block scale folded in, transposed
// to [512 c][32 v], and the head's o_lat rows of up to 64 sequences transposed to
// [512 c][64 b] (bf16); thread (r, s) then accumulates a 4-row x 2-sequence tile over the 512
// latent columns (one 16-byte and one 4-byte shared load per 8 FMAs).
constexpr int ABT_V = 32;    // output rows per CTA
constexpr int ABT_S = 64;    // sequences per staged chunk
constexpr int ABT_THREADS = (ABT_V / 4) * (ABT_S / 2);  // 256
constexpr size_t ABT_SMEM = (size_t)KV_LORA * ABT_V * 4 + (size_t)KV_LORA * ABT_S * 2;
__global__ void __launch_bounds__(ABT_THREADS) absorb_out_tiled_kernel(
    const __nv_bfloat16* o_lat, int B, const uint8_t* __restrict__ Wkvb,
    const float* __restrict__ Skvb, __nv_bfloat16* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t abt_smem[];
  float* ws = reinterpret_cast<float*>(abt_smem);                              // [512][32]
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(abt_smem + KV_LORA * ABT_V * 4);  // [512][64]
  const int h = blockIdx.x, v0 = blockIdx.y * ABT_V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {  // W_UV rows (lane = row), 16 columns per chunk, 4 chunks per thread
    const uint8_t* wrow = Wkvb + (size_t)(h * KVB_PER_HEAD + NOPE + v0 + lane) * KV_LORA;
    for (int k = 0; k < KV_LORA / 16 / (ABT_THREADS / 32); ++k) {
      const int c0 = (warp * (KV_LORA / 16 / (ABT_THREADS / 32)) + k) * 16;
      const float sc = Skvb[(size_t)(2 * h + 1) * (KV_LORA / BLK) + c0 / BLK];
      const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wrow + c0));
      float f[16];
      e4m3x4_to_f32(wv.x, f);
      e4m3x4_to_f32(wv.y, f + 4);
      e4m3x4_to_f32(wv.z, f + 8);
      e4m3x4_to_f32(wv.w, f + 12);
#pragma unroll
      for (int i = 0; i < 16; ++i) ws[(c0 + i) * ABT_V + lane] = f[i] * sc;
    }
  }
  pdl_launch_dependents();
  pdl_wait();  // the weights above do not depend on earlier kernels; o_lat does
  const int r0 = (threadIdx.x % (ABT_V / 4)) * 4, s0 = (threadIdx.x / (ABT_V / 4)) * 2;
  for (int b0 = 0; b0 < B; b0 += ABT_S) {
    const int nb = min(ABT_S, B - b0);
    __syncthreads();  // the previous chunk's reads of xs are done (and ws is written)
    // o_lat rows of this head: 8 columns per 16-byte load, written transposed.
    for (int e = threadIdx.x; e < nb * (KV_LORA / 8); e += ABT_THREADS) {
      const int sb = e % nb, c0 = (e / nb) * 8;
      const uint4 x = ld_dep_v4(o_lat + ((size_t)(b0 + sb) * HEADS + h) * KV_LORA + c0);
      const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&x);
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[(c0 + i) * ABT_S + sb] = xb[i];
    }
    __syncthreads();
    if (s0 < nb) {
      float acc[4][2] = {};
#pragma unroll 4
      for (int c = 0; c < KV_LORA; ++c) {
        const float4 w = *reinterpret_cast<const float4*>(ws + c * ABT_V + r0);
        const uint32_t xp = *reinterpret_cast<const uint32_t*>(xs + c * ABT_S + s0);
        const float x0 = __uint_as_float(xp << 16), x1 = __uint_as_float(xp & 0xFFFF0000u);
        acc[0][0] = fmaf(w.x, x0, acc[0][0]);
        acc[1][0] = fmaf(w.y, x0, acc[1][0]);
        acc[2][0] = fmaf(w.z, x0, acc[2][0]);
        acc[3][0] = fmaf(w.w, x0, acc[3][0]);
        acc[0][1] = fmaf(w.x, x1, acc[0][1]);
        acc[1][1] = fmaf(w.y, x1, acc[1][1]);
        acc[2][1] = fmaf(w.z, x1, acc[2][1]);
        acc[3][1] = fmaf(w.w, x1, acc[3][1]);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (s0 + j >= nb) break;
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0][j], acc[1][j]);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2][j], acc[3][j]);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out + (size_t)(b0 + s0 + j) * O_IN + h * VDIM + v0 + r0) = pk;
      }
    }
  }
}

namespace {
// out[h][c][i] = W[256 h + i][c]: a 64 x 64-byte tile per CTA through shared memory.
__global__ void __launch_bounds__(256) transpose_wuk_kernel(const uint8_t* __restrict__ W,
                                                            uint8_t* __restrict__ out) {
  __shared__ uint8_t t[64][65];
  const int h = blockIdx.z, i0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  for (int e = threadIdx.x; e < 64 * 64; e += 256) {
    const int i = e / 64, c = e % 64;
    t[i][c] = W[((size_t)h * KVB_PER_HEAD + i0 + i) * KV_LORA + c0 + c];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 64 * 64; e += 256) {
    const int c = e / 64, i = e % 64;
    out[((size_t)h * KV_LORA + c0 + c) * NOPE + i0 + i] = t[i][c];
  }
}
}  // namespace

cudaError_t launch_transpose_wuk(const uint8_t* Wkvb, uint8_t* out, cudaStream_t st) {
  transpose_wuk_kernel<<<dim3(KV_LORA / 64, NOPE / 64, HEADS), 256, 0, st>>>(Wkvb, out);
  return cudaGetLastError();
}

cudaError_t launch_absorb_q(const __nv_bfloat16* q, int B, const uint8_t* Wkvb,
                            const float* Skvb, const float2* rope_tab, int rope_pairing,
                            const int* seq_lens, int limit, __nv_bfloat16* qfull,
                            cudaStream_t st, bool pdl) {
  if (B <= 0) return cudaSuccess;
  return launch_kernel(absorb_q_kernel, dim3(HEADS, KV_LORA / BLK, (B + ABQ_B - 1) / ABQ_B),
                       dim3(128), 0, st, pdl, q, B,
                       Wkvb, Skvb, rope_tab, rope_pairing, seq_lens, limit, qfull);
}

cudaError_t launch_absorb_out(const __nv_bfloat16* o_lat, int B, const uint8_t* Wkvb,
                              const float* Skvb, __nv_bfloat16* out, cudaStream_t st, bool pdl) {
  if (B > 8)
    return launch_kernel(absorb_out_tiled_kernel, dim3(HEADS, VDIM / ABT_V), dim3(ABT_THREADS),
                         ABT_SMEM, st, pdl, o_lat, B, Wkvb, Skvb, out);
  return launch_kernel(absorb_out_kernel, dim3(HEADS * VDIM / 8), dim3(256), 0, st, pdl, o_lat, B,
                       Wkvb, Skvb, out);
}

cudaError_t init_kernels() {
  cudaError_t e = cudaFuncSetAttribute(absorb_out_tiled_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ABT_SMEM);
  if (e == cudaSuccess) e = init_decode_tc_kernel();
  if (e == cudaSuccess) e = init_prefill_tc_kernel();
  if (e == cudaSuccess) e = init_gemv_kernels();
  return e != cudaSuccess ? e : init_gemm_tc_kernels();
}

cudaError_t launch_advance_lens(int* seq_lens, int B, int T, cudaStream_t st, bool pdl) {
  return launch_kernel(advance_lens_kernel, dim3((B + 255) / 256), dim3(256), 0, st, pdl, seq_lens,
                       B, T);
}

cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, bool wait_prev,
                          cudaStream_t st, bool pdl) {
  if (bytes == 0) return cudaSuccess;
  if (bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(src) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(dst) & 15) != 0)
    return cudaErrorInvalidValue;
  const size_t n = bytes / 16;
  const size_t blocks = (n + 255) / 256;
  return launch_kernel(copy16_kernel, dim3((unsigned)(blocks < 1024 ? blocks : 1024)), dim3(256),
                       0, st, pdl, static_cast<const uint4*>(src), static_cast<uint4*>(dst), n,
                       wait_prev ? 1 : 0);
}

cudaError_t launch_dequant(const uint8_t* W, const float* S, int rows, int cols, float* out,
                           cudaStream_t st) {
  const size_t n = (size_t)rows * cols;
  dequant_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(W, S, rows, cols, out);
  return cudaGetLastError();
}

}  // namespace mla
