// FP8 block-scaled projections for a few tokens (M <= kGemvMaxM), weight-streaming GEMVs
// (larger token counts go to the tcgen05 GEMM in k_gemm_tc.cu):
//
// Y[m, n] = sum_k X[m, k] * e4m3(W[n, k]) * S[n/128][k/128]  ("linear" excerpt of the
// "Key-value latent" page: fmt e4m3, weight_block_size [128, 128]; nn.Linear without bias).
// Every 128-wide k block is summed in fp32 and multiplied by its block scale once, so the
// dequantised weight is never rounded.
//
// One or two tokens: gemv_f8w_kernel, one warp per weight row on the CUDA cores, the whole row
// requested before the kernel waits for its input.  Its CTAs are small (4 warps), so under
// programmatic dependent launch they start beside the previous kernel's CTAs and hold a first
// wave of rows in registers when that kernel finishes.  Each 512-byte piece of the row is
// dequantised four values at a time (the sum in the same order), which keeps the long rows
// (K = 7168, 8192) within 96 registers: five CTAs per SM, a quarter more rows in that first
// wave (B=1 step 46.7-47.0 -> 45.8-46.0 us).
//
// Three or four tokens: gemv_mma_kernel, on the tensor cores (mma.sync m16n8k16, f16 x f16 ->
// f32), where the row GEMV's CUDA-core work would grow with the tokens.  A CTA owns TPC tiles of
// 16 weight rows; warp w of a tile owns the k-slice [512 s, 512 s + 512), s = w % NCH,
// NCH = K / 512.  Per 64-wide k step j, thread (g, t) of the warp (g = lane / 4, t = lane % 4)
// holds 16 contiguous e4m3 bytes of rows g and g + 8 at k = 512 s + 64 j + 16 t, converts them
// exactly to f16 pairs and issues four MMAs.  The MMA's k order is permuted identically in A
// (weights) and B (activations): MMA q of a step takes k = base + 4 q + {0, 1} as its k-slots
// 2t, 2t+1 and base + 4 q + {2, 3} as slots 8 + 2t, 9 + 2t (base = 512 s + 64 j + 16 t), so
// every thread reads whole 16-byte runs of its rows.  B's eight columns are the tokens (columns
// >= M read token 0 and are discarded; the kernel is written for up to eight).  The NCH warps' partial sums of a tile meet in shared
// memory.  e4m3 -> f16 is exact and the MMA's products are exact; the activations enter as
// f16, each token scaled by a power of two that puts its largest magnitude below 2^15 (exact
// for every value within 2^32 of that maximum), and the outputs are scaled back.  The grid is
// at most the CTAs that fit at once: each CTA loops over its tile groups, and asks L2 for its
// later groups' rows (cp.async.bulk.prefetch.L2) before the wait.
#include "mla_internal.h"

namespace mla {

namespace {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Starts the DRAM reads of `bytes` (a multiple of 16; address 16-byte aligned) into L2: no
// destination, no completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Two e4m3 values (the low 16 bits of `pair`) -> an f16 pair (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(pair & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// D += A . B for one m16n8k16 tile, f16 inputs, f32 accumulators.
__device__ __forceinline__ void mma_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Four e4m3 bytes of one 32-bit word -> four floats (exact).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* f) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFF), __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float* f) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

struct ProjSet {
  Proj p[2];
  int np;
  int rows0;  // rows of p[0] (a multiple of 16)
  int* adv;   // optional: adv[i] += adv_by for i < adv_n, by block 0 (lengths bookkeeping)
  int adv_n, adv_by;
};

// ---------------------------------------------------------------- one or two tokens
template <int M, int NCH>
__global__ void __launch_bounds__(128, NCH >= 14 ? 5 : 4) gemv_f8w_kernel(const __nv_bfloat16* X, int ldx,
                                                          ProjSet ps) {
  constexpr int K = NCH * 512;
  pdl_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int total = ps.p[0].N + (ps.np > 1 ? ps.p[1].N : 0);
  if (warp >= total) {
    if (ps.adv && blockIdx.x == 0 && (int)threadIdx.x < ps.adv_n) {
      pdl_wait();
      ps.adv[threadIdx.x] += ps.adv_by;
    }
    return;
  }
  const Proj& P = (warp < ps.rows0) ? ps.p[0] : ps.p[1];
  const int n = (warp < ps.rows0) ? warp : warp - ps.rows0;
  const uint8_t* wrow = P.W + (size_t)n * K;
  const float* srow = P.S + (size_t)(n / BLK) * (K / BLK);

  uint4 w[NCH];
#pragma unroll
  for (int u = 0; u < NCH; ++u) w[u] = ld_stream(wrow + u * 512 + lane * 16);
  // The weights do not depend on earlier kernels; the activations do.
  pdl_wait();
  if (ps.adv && blockIdx.x == 0 && (int)threadIdx.x < ps.adv_n) ps.adv[threadIdx.x] += ps.adv_by;

  float acc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) acc[m] = 0.f;
#pragma unroll
  for (int u = 0; u < NCH; ++u) {
    const int k = u * 512 + lane * 16;
    const float sc = __ldg(srow + k / BLK);
    const uint32_t wv[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const __nv_bfloat16* xp = X + (size_t)m * ldx + k;  // written by the previous kernel
      float part = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 xv = ld_dep_v4(xp + 8 * h);
        const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float wf[4];
          e4m3x4_to_f32(wv[2 * h + q], wf);
          part = fmaf(wf[0], __uint_as_float(xu[2 * q] << 16), part);
          part = fmaf(wf[1], __uint_as_float(xu[2 * q] & 0xFFFF0000u), part);
          part = fmaf(wf[2], __uint_as_float(xu[2 * q + 1] << 16), part);
          part = fmaf(wf[3], __uint_as_float(xu[2 * q + 1] & 0xFFFF0000u), part);
        }
      }
      acc[m] = fmaf(sc, part, acc[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float v = acc[m];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) {
      if (P.y_fp32) {
        reinterpret_cast<float*>(P.Y)[(size_t)m * P.ldy + n] = v;
      } else {
        if (P.R)  // residual: bf16(R + bf16(product))
          v = bf16r(v) + __bfloat162float(P.R[(size_t)m * P.ldy + n]);
        reinterpret_cast<__nv_bfloat16*>(P.Y)[(size_t)m * P.ldy + n] = __float2bfloat16_rn(v);
      }
    }
  }
}

// q_b_proj for one or two decode tokens with the q-latent RMSNorm done on the fly ("rmsnorm"
// excerpt: cq = g * bf16(x * rsqrt(mean(x^2) + eps))): every CTA normalises the tokens' fp32
// q_a outputs (g1[m][0:1536], 6 KB each from L2) into shared memory and then streams its
// weight rows like gemv_f8w_kernel, QB_RW consecutive rows per warp (all of them requested
// before the wait on the previous kernel), so the norm is shared by 4 QB_RW rows.  One extra CTA
// at the end normalises the kv latent, rotates the shared rotary key and appends each token's
// cache row, the other half of the norm kernel of the prefill path.
struct NormArgs {
  const float* g1;               // [M][2112] fp32 q_a | kv_a outputs
  const __nv_bfloat16* gq;       // q_a_layernorm gain [1536]
  const __nv_bfloat16* gkv;      // kv_a_layernorm gain [512]
  float eps;
  const float2* rope_tab;
  int pairing;
  const int* seq_lens;
  CacheRef cache;
  int limit;
  int* err;
};
constexpr int QB_RW = 4;
static_assert(QB_N % (4 * QB_RW) == 0, "whole CTAs of q_b rows");

// Sum over the 128 threads of a CTA (red: 4 floats of shared memory).
__device__ __forceinline__ float cta_sum128(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  return (red[0] + red[1]) + (red[2] + red[3]);
}

template <int M>
__global__ void __launch_bounds__(128, 4) gemv_norm_qb_kernel(Proj P, NormArgs na) {
  constexpr int K = Q_LORA, NCH = K / 512;
  __shared__ __align__(16) __nv_bfloat16 xs[M][K];
  __shared__ float red[4];
  __shared__ __align__(16) __nv_bfloat16 row[LAT];
  pdl_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, tid = threadIdx.x;
  const bool kv_cta = blockIdx.x == gridDim.x - 1;
  const int n0 = warp * QB_RW;  // rows n0 .. n0 + QB_RW - 1
  uint4 w[QB_RW][NCH];
  if (!kv_cta) {
#pragma unroll
    for (int j = 0; j < QB_RW; ++j)
#pragma unroll
      for (int u = 0; u < NCH; ++u)
        w[j][u] = ld_stream(P.W + (size_t)(n0 + j) * K + u * 512 + lane * 16);
  }
  pdl_wait();  // g1 comes from the previous kernel
  if (kv_cta) {
    // kv latent norm, rotary key and the cache row of every token.
    for (int m = 0; m < M; ++m) {
      const float* in = na.g1 + (size_t)m * G1_N + Q_LORA;
      float xk[KV_LORA / 128];
      float sk = 0.f;
#pragma unroll
      for (int i = 0; i < KV_LORA / 128; ++i) {
        xk[i] = ld_dep_f32(in + tid + 128 * i);
        sk += xk[i] * xk[i];
      }
      const float rk = rsqrtf(cta_sum128(sk, red) / KV_LORA + na.eps);
#pragma unroll
      for (int i = 0; i < KV_LORA / 128; ++i) {
        const int c = tid + 128 * i;
        row[c] = __float2bfloat16_rn(__bfloat162float(na.gkv[c]) * bf16r(xk[i] * rk));
      }
      const int pos = na.seq_lens[m];
      // positions past the cache or the RoPE table, or an invalid page: skipped and flagged
      const long long crow = (pos < 0 || pos >= na.limit) ? -1 : na.cache.row(m, pos);
      const bool bad = crow < 0;
      if (bad && tid == 0) atomicExch(na.err, DEV_ERR_RANGE);
      if (!bad && tid < ROPE / 2) {
        const int2 ij = na.pairing == 0 ? make_int2(2 * tid, 2 * tid + 1)
                                        : make_int2(tid, tid + ROPE / 2);
        const float2 cs = na.rope_tab[(size_t)pos * (ROPE / 2) + tid];
        const float a = ld_dep_f32(in + KV_LORA + ij.x), b = ld_dep_f32(in + KV_LORA + ij.y);
        row[KV_LORA + ij.x] = __float2bfloat16_rn(a * cs.x - b * cs.y);
        row[KV_LORA + ij.y] = __float2bfloat16_rn(b * cs.x + a * cs.y);
      }
      __syncthreads();
      if (!bad && tid < LAT / 8)
        reinterpret_cast<uint4*>(na.cache.base + (size_t)crow * LAT)[tid] =
            reinterpret_cast<const uint4*>(row)[tid];
      __syncthreads();
    }
    return;
  }
  // q latent norm of every token into shared memory.
  for (int m = 0; m < M; ++m) {
    const float* in = na.g1 + (size_t)m * G1_N;
    float xq[K / 128];
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < K / 128; ++i) {
      xq[i] = ld_dep_f32(in + tid + 128 * i);
      sq += xq[i] * xq[i];
    }
    const float rq = rsqrtf(cta_sum128(sq, red) / K + na.eps);
#pragma unroll
    for (int i = 0; i < K / 128; ++i) {
      const int c = tid + 128 * i;
      xs[m][c] = __float2bfloat16_rn(__bfloat162float(na.gq[c]) * bf16r(xq[i] * rq));
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < QB_RW; ++j) {
    const int n = n0 + j;
    const float* srow = P.S + (size_t)(n / BLK) * (K / BLK);
    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.f;
#pragma unroll
    for (int u = 0; u < NCH; ++u) {
      const int k = u * 512 + lane * 16;
      float wf[16];
      e4m3x4_to_f32(w[j][u].x, wf);
      e4m3x4_to_f32(w[j][u].y, wf + 4);
      e4m3x4_to_f32(w[j][u].z, wf + 8);
      e4m3x4_to_f32(w[j][u].w, wf + 12);
      const float sc = __ldg(srow + k / BLK);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint4* xp = reinterpret_cast<const uint4*>(&xs[m][k]);
        float xf[16];
        bf16x8_to_f32(xp[0], xf);
        bf16x8_to_f32(xp[1], xf + 8);
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) part = fmaf(wf[i], xf[i], part);
        acc[m] = fmaf(sc, part, acc[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = acc[m];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0)
        reinterpret_cast<__nv_bfloat16*>(P.Y)[(size_t)m * P.ldy + n] = __float2bfloat16_rn(v);
    }
  }
}

// ---------------------------------------------------------------- three to eight tokens
// Tiles of 16 rows per CTA for a k-extent of NCH slices of 512.
constexpr int gemv_tpc(int nch) { return nch >= 14 ? 1 : (nch >= 3 ? 2 : 4); }
constexpr int gemv_threads(int nch) { return 32 * nch * gemv_tpc(nch); }
constexpr int kXPad = 8;  // halfs of padding per activation row in shared memory

// Shared memory of a CTA: the activations (f16, M rows of K + kXPad), the tiles' partial sums
// [TPC][NCH][16 rows][8 tokens] (f32) and the tokens' scale exponents.
constexpr int gemv_smem(int M, int nch) {
  return M * (nch * 512 + kXPad) * 2 + gemv_tpc(nch) * nch * 16 * 8 * 4 + 8 * 4;
}


// Sum (or maximum) over the CTA's NT threads; red holds NT / 32 floats.  Every thread gets the
// result.
template <int NT, bool MAX>
__device__ __forceinline__ float cta_reduce(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = MAX ? fmaxf(v, o) : v + o;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = MAX ? fmaxf(r, red[w]) : r + red[w];
  return r;
}

// Exponent e >= 0 with amax * 2^-e < 2^15 (0 for amax < 2^15, NaN or Inf).
__device__ __forceinline__ int f16_shift(float amax) {
  if (!(amax >= 32768.f) || isinf(amax)) return 0;
  int e;
  frexpf(amax, &e);  // amax < 2^e
  return e - 15;
}

// The weight loads of one thread: rows g and g + 8 of its tile, k-slice s.
template <int NCH>
__device__ __forceinline__ void gemv_load(const uint8_t* tile_w, int s, int lane, uint4 (&wa)[8],
                                          uint4 (&wb)[8]) {
  constexpr int K = NCH * 512;
  const uint8_t* pa = tile_w + (size_t)(lane >> 2) * K + 512 * s + 16 * (lane & 3);
  const uint8_t* pb = pa + (size_t)8 * K;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    wa[j] = ld_stream(pa + 64 * j);
    wb[j] = ld_stream(pb + 64 * j);
  }
}

// The tensor-core work of one thread's slice and its partial sums into red: d = sum over the
// slice's four k blocks of scale * block sum, for rows g, g + 8 and tokens 2t, 2t + 1.
template <int M, int NCH>
__device__ __forceinline__ void gemv_mma(const __half* xs, int s, int lane, const uint4 (&wa)[8],
                                         const uint4 (&wb)[8], const float* srow, float* red_tile) {
  constexpr int XS = NCH * 512 + kXPad;
  const int g = lane >> 2, t = lane & 3;
  const __half* xr = xs + (size_t)(g < M ? g : 0) * XS + 512 * s + 16 * t;
  float acc[4][4];
#pragma unroll
  for (int b = 0; b < 4; ++b)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[b][i] = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 x0 = *reinterpret_cast<const uint4*>(xr + 64 * j);
    const uint4 x1 = *reinterpret_cast<const uint4*>(xr + 64 * j + 8);
    const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const uint32_t ua[4] = {wa[j].x, wa[j].y, wa[j].z, wa[j].w};
    const uint32_t ub[4] = {wb[j].x, wb[j].y, wb[j].z, wb[j].w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      mma_16816(acc[j / 2], e4m3x2_to_f16x2(ua[q]), e4m3x2_to_f16x2(ub[q]),
                e4m3x2_to_f16x2(ua[q] >> 16), e4m3x2_to_f16x2(ub[q] >> 16), xb[2 * q],
                xb[2 * q + 1]);
  }
  float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const float sc = __ldg(srow + 4 * s + b);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = fmaf(sc, acc[b][i], d[i]);
  }
  float* r = red_tile + (size_t)s * 128;
  r[g * 8 + 2 * t] = d[0];
  r[g * 8 + 2 * t + 1] = d[1];
  r[(g + 8) * 8 + 2 * t] = d[2];
  r[(g + 8) * 8 + 2 * t + 1] = d[3];
}

// Activations X[m][0:K] (written by the previous kernel) -> xs as f16, each token scaled by
// 2^-xexp[m].
template <int M, int NCH>
__device__ __forceinline__ void gemv_stage_x(const __nv_bfloat16* X, int ldx, __half* xs,
                                             int* xexp, float* red) {
  constexpr int K = NCH * 512, NT = gemv_threads(NCH), XS = K + kXPad;
#pragma unroll 1
  for (int m = 0; m < M; ++m) {
    const __nv_bfloat16* xm = X + (size_t)m * ldx;
    float amax = 0.f;
    for (int e = threadIdx.x; e < K / 8; e += NT) {
      const uint4 v = ld_dep_v4(xm + 8 * e);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(u[i] << 16)),
                                 fabsf(__uint_as_float(u[i] & 0xFFFF0000u))));
    }
    const int sh = f16_shift(cta_reduce<NT, true>(amax, red));
    const float mul = ldexpf(1.f, -sh);
    if (threadIdx.x == 0) xexp[m] = sh;
    for (int e = threadIdx.x; e < K / 8; e += NT) {
      const uint4 v = ld_dep_v4(xm + 8 * e);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 p = __floats2half2_rn(__uint_as_float(u[i] << 16) * mul,
                                            __uint_as_float(u[i] & 0xFFFF0000u) * mul);
        h[i] = *reinterpret_cast<const uint32_t*>(&p);
      }
      *reinterpret_cast<uint4*>(xs + (size_t)m * XS + 8 * e) = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
}

// Output of one tile group: the NCH partial sums of each (row, token) from red, scaled back by
// the token's exponent, into Y (fp32, or bf16 with the optional residual).
template <int M, int NCH>
__device__ __forceinline__ void gemv_store(const ProjSet& ps, int total, int grp, const float* red,
                                           const int* xexp) {
  constexpr int TPC = gemv_tpc(NCH), NT = gemv_threads(NCH);
  for (int e = threadIdx.x; e < TPC * 16 * M; e += NT) {
    const int t2 = e / (16 * M), r = (e / M) % 16, m = e % M;
    const int row = (grp * TPC + t2) * 16 + r;
    if (row >= total) continue;
    float v = 0.f;
#pragma unroll 4
    for (int k = 0; k < NCH; ++k) v += red[((t2 * NCH + k) * 16 + r) * 8 + m];
    v = ldexpf(v, xexp[m]);
    const Proj& P = row < ps.rows0 ? ps.p[0] : ps.p[1];
    const int n = row < ps.rows0 ? row : row - ps.rows0;
    if (P.y_fp32) {
      reinterpret_cast<float*>(P.Y)[(size_t)m * P.ldy + n] = v;
    } else {
      if (P.R)  // residual: bf16(R + bf16(product))
        v = bf16r(v) + __bfloat162float(P.R[(size_t)m * P.ldy + n]);
      reinterpret_cast<__nv_bfloat16*>(P.Y)[(size_t)m * P.ldy + n] = __float2bfloat16_rn(v);
    }
  }
}

// Persistent: CTA c takes the tile groups c, c + G, c + 2G, ... (G = gridDim.x, at most the
// CTAs that fit at once).  Its first group's weights are in registers and the later groups'
// rows on their way into L2 before the wait on the previous kernel.
template <int M, int NCH>
__global__ void __launch_bounds__(gemv_threads(NCH), 1) gemv_mma_kernel(const __nv_bfloat16* X,
                                                                        int ldx, ProjSet ps) {
  constexpr int K = NCH * 512, TPC = gemv_tpc(NCH), XS = K + kXPad;
  extern __shared__ __align__(16) uint8_t smem[];
  __half* xs = reinterpret_cast<__half*>(smem);
  float* red = reinterpret_cast<float*>(smem + (size_t)M * XS * 2);  // [TPC][NCH][16][8]
  int* xexp = reinterpret_cast<int*>(red + TPC * NCH * 128);
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tl = warp / NCH, s = warp % NCH;
  const int total = ps.p[0].N + (ps.np > 1 ? ps.p[1].N : 0);
  const int groups = (total + 16 * TPC - 1) / (16 * TPC);
  auto tile_rows = [&](int r0) -> const uint8_t* {
    return r0 < ps.rows0 ? ps.p[0].W + (size_t)r0 * K : ps.p[1].W + (size_t)(r0 - ps.rows0) * K;
  };
  uint4 wa[8], wb[8];
  {
    const int r0 = (blockIdx.x * TPC + tl) * 16;
    if (r0 < total) gemv_load<NCH>(tile_rows(r0), s, lane, wa, wb);
  }
  if (threadIdx.x == 0)  // the later groups' rows into L2 while this kernel waits
    for (int grp = blockIdx.x + gridDim.x; grp < groups; grp += gridDim.x)
      for (int r = grp * TPC * 16; r < (grp + 1) * TPC * 16 && r < total; r += 16)
        prefetch_l2(tile_rows(r), 16 * K);
  // The weights do not depend on earlier kernels; the activations do.
  pdl_wait();
  if (ps.adv && blockIdx.x == 0 && (int)threadIdx.x < ps.adv_n) ps.adv[threadIdx.x] += ps.adv_by;
  gemv_stage_x<M, NCH>(X, ldx, xs, xexp, red);
  __syncthreads();
  for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    const int r0 = (grp * TPC + tl) * 16;
    if (grp != (int)blockIdx.x && r0 < total) gemv_load<NCH>(tile_rows(r0), s, lane, wa, wb);
    if (r0 < total) {
      const Proj& P = r0 < ps.rows0 ? ps.p[0] : ps.p[1];
      const int n0 = r0 < ps.rows0 ? r0 : r0 - ps.rows0;
      gemv_mma<M, NCH>(xs, s, lane, wa, wb, P.S + (size_t)(n0 / BLK) * (K / BLK),
                       red + tl * NCH * 128);
    }
    __syncthreads();
    gemv_store<M, NCH>(ps, total, grp, red, xexp);
    __syncthreads();  // red is rewritten by the next group
  }
}

// CTAs of a tensor-core GEMV instantiation that fit on one SM at its dynamic shared memory
// (the same on every GB300; queried once, after init_gemv_kernels has raised the limit).
template <int M, int NCH>
int mma_per_sm() {
  static const int n = [] {
    int r = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, gemv_mma_kernel<M, NCH>,
                                                         gemv_threads(NCH), gemv_smem(M, NCH)) ==
                   cudaSuccess
               ? r
               : 0;
  }();
  return n;
}

template <int M, int NCH>
cudaError_t launch_rows_k(const __nv_bfloat16* X, int ldx, const ProjSet& ps, int rows,
                          cudaStream_t st, bool pdl) {
  return launch_kernel(gemv_f8w_kernel<M, NCH>, dim3((rows + 3) / 4), dim3(128), 0, st, pdl, X,
                       ldx, ps);
}

template <int M, int NCH>
cudaError_t launch_mma_k(const __nv_bfloat16* X, int ldx, const ProjSet& ps, int rows,
                         int num_sms, cudaStream_t st, bool pdl) {
  constexpr int per_cta = 16 * gemv_tpc(NCH);
  const int groups = (rows + per_cta - 1) / per_cta, resident = mma_per_sm<M, NCH>() * num_sms;
  const int grid = resident > 0 && groups > resident ? resident : groups;
  return launch_kernel(gemv_mma_kernel<M, NCH>, dim3(grid), dim3(gemv_threads(NCH)),
                       gemv_smem(M, NCH), st, pdl, X, ldx, ps);
}

template <int M>
cudaError_t launch_gemv(const __nv_bfloat16* X, int ldx, int K, const ProjSet& ps, int rows,
                        int num_sms, cudaStream_t st, bool pdl) {
  if constexpr (M <= 2) {
    switch (K) {
      case 512: return launch_rows_k<M, 1>(X, ldx, ps, rows, st, pdl);
      case 1536: return launch_rows_k<M, 3>(X, ldx, ps, rows, st, pdl);
      case 7168: return launch_rows_k<M, 14>(X, ldx, ps, rows, st, pdl);
      case 8192: return launch_rows_k<M, 16>(X, ldx, ps, rows, st, pdl);
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (K) {
      case 512: return launch_mma_k<M, 1>(X, ldx, ps, rows, num_sms, st, pdl);
      case 1536: return launch_mma_k<M, 3>(X, ldx, ps, rows, num_sms, st, pdl);
      case 7168: return launch_mma_k<M, 14>(X, ldx, ps, rows, num_sms, st, pdl);
      case 8192: return launch_mma_k<M, 16>(X, ldx, ps, rows, num_sms, st, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
}

// Raises every tensor-core instantiation's dynamic shared memory limit (current device).
template <int M>
cudaError_t init_gemv_m() {
  constexpr auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<M, 1>, attr, gemv_smem(M, 1));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_mma_kernel<M, 3>, attr, gemv_smem(M, 3));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_mma_kernel<M, 14>, attr, gemv_smem(M, 14));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_mma_kernel<M, 16>, attr, gemv_smem(M, 16));
  return e;
}

}  // namespace

cudaError_t init_gemv_kernels() {
  static_assert(kGemvMaxM == 4, "instantiations below cover M <= 4");
  cudaError_t e = init_gemv_m<3>();
  if (e == cudaSuccess) e = init_gemv_m<4>();
  return e;
}

cudaError_t launch_gemm(const __nv_bfloat16* X, int ldx, int M, int K, const Proj* p, int np,
                        float* partial, int num_sms, int* err, cudaStream_t st, int* adv,
                        int adv_n, int adv_by, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (M > kGemvMaxM)
    return launch_gemm_tc(X, ldx, M, K, p, np, partial, num_sms, err, st, adv, adv_n, adv_by, pdl);
  if (p[0].N % 16 != 0 || (np > 1 && p[1].N % 16 != 0)) return cudaErrorInvalidValue;
  ProjSet ps{};
  ps.np = np;
  ps.adv = adv;
  ps.adv_n = adv_n;
  ps.adv_by = adv_by;
  ps.p[0] = p[0];
  if (np > 1) ps.p[1] = p[1];
  ps.rows0 = p[0].N;
  const int rows = p[0].N + (np > 1 ? p[1].N : 0);
  switch (M) {
    case 1: return launch_gemv<1>(X, ldx, K, ps, rows, num_sms, st, pdl);
    case 2: return launch_gemv<2>(X, ldx, K, ps, rows, num_sms, st, pdl);
    case 3: return launch_gemv<3>(X, ldx, K, ps, rows, num_sms, st, pdl);
    default: return launch_gemv<4>(X, ldx, K, ps, rows, num_sms, st, pdl);
  }
}

bool gemm_can_advance(int M) { return M > 0; }

cudaError_t launch_qb_norm(const float* g1, int M, const Proj& p, const __nv_bfloat16* gq,
                           const __nv_bfloat16* gkv, float eps, const float2* rope_tab,
                           int rope_pairing, const int* seq_lens, const CacheRef& cache,
                           int limit, int* err, int num_sms, cudaStream_t st, bool pdl) {
  (void)num_sms;
  if (M < 1 || M > 2 || p.N != QB_N || p.y_fp32) return cudaErrorInvalidValue;
  const NormArgs na{g1, gq, gkv, eps, rope_tab, rope_pairing, seq_lens, cache, limit, err};
  const dim3 grid(QB_N / (4 * QB_RW) + 1), block(128);  // + the kv-cache CTA
  return M == 1 ? launch_kernel(gemv_norm_qb_kernel<1>, grid, block, 0, st, pdl, p, na)
                : launch_kernel(gemv_norm_qb_kernel<2>, grid, block, 0, st, pdl, p, na);
}

}  // namespace mla
