// FP8 block-scaled projections for a few tokens: a weight-streaming GEMV on the CUDA cores
// (larger token counts go to the tensor-core kernel in k_gemm_tc.cu).
//
// Y[m, n] = sum_k X[m, k] * e4m3(W[n, k]) * S[n/128][k/128]  ("linear" excerpt of the
// "Key-value latent" page: fmt e4m3, weight_block_size [128, 128]; nn.Linear without bias).
// Every 128-wide k block is summed in float32 with the raw e4m3 values and then multiplied by
// its block scale once, so the dequantised weight is never rounded.
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

// Four e4m3 bytes of one 32-bit word -> four floats (exact).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* f) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFF), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
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
  int rows0;    // rows of p[0]
  int* adv;     // optional: adv[i] += adv_by for i < adv_n, by block 0 (lengths bookkeeping)
  int adv_n, adv_by;
};

template <int M, int NCH>
__global__ void __launch_bounds__(128) gemv_f8w_kernel(const __nv_bfloat16* __restrict__ X,
                                                       int ldx, ProjSet ps) {
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
    float wf[16];
    e4m3x4_to_f32(w[u].x, wf);
    e4m3x4_to_f32(w[u].y, wf + 4);
    e4m3x4_to_f32(w[u].z, wf + 8);
    e4m3x4_to_f32(w[u].w, wf + 12);
    const float sc = __ldg(srow + k / BLK);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const uint4* xp = reinterpret_cast<const uint4*>(X + (size_t)m * ldx + k);
      float xf[16];
      bf16x8_to_f32(__ldg(xp), xf);
      bf16x8_to_f32(__ldg(xp + 1), xf + 8);
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
    if (lane == 0) {
      if (P.y_fp32) {
        reinterpret_cast<float*>(P.Y)[(size_t)m * P.ldy + n] = v;
      } else {
        if (P.R)  // residual: bf16(R + bf16(product))
          v = __bfloat162float(__float2bfloat16_rn(v)) +
              __bfloat162float(P.R[(size_t)m * P.ldy + n]);
        reinterpret_cast<__nv_bfloat16*>(P.Y)[(size_t)m * P.ldy + n] = __float2bfloat16_rn(v);
      }
    }
  }
}

// q_b_proj for a few decode tokens with the q-latent RMSNorm done on the fly ("rmsnorm"
// excerpt: cq = g * bf16(x * rsqrt(mean(x^2) + eps))): every CTA normalises the tokens' fp32
// q_a outputs (g1[m][0:1536], 6 KB each from L2) into shared memory and then streams its four
// weight rows like gemv_f8w_kernel.  One extra CTA at the end normalises the kv latent,
// rotates the shared rotary key and appends each token's cache row, the other half of the
// norm kernel of the prefill path.
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

__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

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
__global__ void __launch_bounds__(128) gemv_norm_qb_kernel(Proj P, NormArgs na) {
  constexpr int K = Q_LORA, NCH = K / 512;
  __shared__ __align__(16) __nv_bfloat16 xs[M][K];
  __shared__ float red[4];
  __shared__ __align__(16) __nv_bfloat16 row[LAT];
  pdl_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, tid = threadIdx.x;
  const bool kv_cta = blockIdx.x == gridDim.x - 1;
  const int n = warp;
  uint4 w[NCH];
  if (!kv_cta) {
    const uint8_t* wrow = P.W + (size_t)n * K;
#pragma unroll
    for (int u = 0; u < NCH; ++u) w[u] = ld_stream(wrow + u * 512 + lane * 16);
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
        xk[i] = in[tid + 128 * i];
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
        const float a = in[KV_LORA + ij.x], b = in[KV_LORA + ij.y];
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
      xq[i] = in[tid + 128 * i];
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
  if (n >= P.N) return;
  const float* srow = P.S + (size_t)(n / BLK) * (K / BLK);
  float acc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) acc[m] = 0.f;
#pragma unroll
  for (int u = 0; u < NCH; ++u) {
    const int k = u * 512 + lane * 16;
    float wf[16];
    e4m3x4_to_f32(w[u].x, wf);
    e4m3x4_to_f32(w[u].y, wf + 4);
    e4m3x4_to_f32(w[u].z, wf + 8);
    e4m3x4_to_f32(w[u].w, wf + 12);
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

template <int M>
cudaError_t launch_gemv(const __nv_bfloat16* X, int ldx, int K, const ProjSet& ps, int rows,
                        cudaStream_t st, bool pdl) {
  const dim3 grid((rows + 3) / 4), block(128);
  switch (K) {
    case 512: return launch_kernel(gemv_f8w_kernel<M, 1>, grid, block, 0, st, pdl, X, ldx, ps);
    case 1536: return launch_kernel(gemv_f8w_kernel<M, 3>, grid, block, 0, st, pdl, X, ldx, ps);
    case 7168: return launch_kernel(gemv_f8w_kernel<M, 14>, grid, block, 0, st, pdl, X, ldx, ps);
    case 8192: return launch_kernel(gemv_f8w_kernel<M, 16>, grid, block, 0, st, pdl, X, ldx, ps);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm(const __nv_bfloat16* X, int ldx, int M, int K, const Proj* p, int np,
                        float* partial, int num_sms, int* err, cudaStream_t st, int* adv,
                        int adv_n, int adv_by, bool pdl) {
  if (M <= 0) return cudaSuccess;
  ProjSet ps{};
  ps.np = np;
  ps.adv = adv;
  ps.adv_n = adv_n;
  ps.adv_by = adv_by;
  ps.p[0] = p[0];
  if (np > 1) ps.p[1] = p[1];
  ps.rows0 = p[0].N;
  const int rows = p[0].N + (np > 1 ? p[1].N : 0);
  if (M <= kGemvMaxM) {
    switch (M) {
      case 1: return launch_gemv<1>(X, ldx, K, ps, rows, st, pdl);
      case 2: return launch_gemv<2>(X, ldx, K, ps, rows, st, pdl);
      case 3: return launch_gemv<3>(X, ldx, K, ps, rows, st, pdl);
      case 4: return launch_gemv<4>(X, ldx, K, ps, rows, st, pdl);
      case 5: return launch_gemv<5>(X, ldx, K, ps, rows, st, pdl);
      case 6: return launch_gemv<6>(X, ldx, K, ps, rows, st, pdl);
      case 7: return launch_gemv<7>(X, ldx, K, ps, rows, st, pdl);
      default: return launch_gemv<8>(X, ldx, K, ps, rows, st, pdl);
    }
  }
  return launch_gemm_tc(X, ldx, M, K, p, np, partial, num_sms, err, st, adv, adv_n, adv_by);
}

bool gemm_can_advance(int M) { return M > 0; }

cudaError_t launch_qb_norm(const float* g1, int M, const Proj& p, const __nv_bfloat16* gq,
                           const __nv_bfloat16* gkv, float eps, const float2* rope_tab,
                           int rope_pairing, const int* seq_lens, const CacheRef& cache,
                           int limit, int* err, cudaStream_t st, bool pdl) {
  if (M < 1 || M > 8 || p.N != QB_N || p.y_fp32) return cudaErrorInvalidValue;
  const NormArgs na{g1, gq, gkv, eps, rope_tab, rope_pairing, seq_lens, cache, limit, err};
  const dim3 grid(p.N / 4 + 1), block(128);  // + the kv-cache CTA
  switch (M) {
    case 1: return launch_kernel(gemv_norm_qb_kernel<1>, grid, block, 0, st, pdl, p, na);
    case 2: return launch_kernel(gemv_norm_qb_kernel<2>, grid, block, 0, st, pdl, p, na);
    case 3: return launch_kernel(gemv_norm_qb_kernel<3>, grid, block, 0, st, pdl, p, na);
    case 4: return launch_kernel(gemv_norm_qb_kernel<4>, grid, block, 0, st, pdl, p, na);
    case 5: return launch_kernel(gemv_norm_qb_kernel<5>, grid, block, 0, st, pdl, p, na);
    case 6: return launch_kernel(gemv_norm_qb_kernel<6>, grid, block, 0, st, pdl, p, na);
    case 7: return launch_kernel(gemv_norm_qb_kernel<7>, grid, block, 0, st, pdl, p, na);
    default: return launch_kernel(gemv_norm_qb_kernel<8>, grid, block, 0, st, pdl, p, na);
  }
}

}  // namespace mla
