// FP8 block-scaled projections for a few tokens with K = 512 (kv_b_proj over a chunk's first
// cached rows): a GEMV on the CUDA cores, one warp per weight row.  The other shapes of one to
// three rows stream their weights in k_gemv_stream.cu; larger token counts run on the
// tensor-core kernel in k_gemm_tc.cu.
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
      if (P.y_fp32)
        reinterpret_cast<float*>(P.Y)[(size_t)m * P.ldy + n] = v;
      else
        reinterpret_cast<__nv_bfloat16*>(P.Y)[(size_t)m * P.ldy + n] = __float2bfloat16_rn(v);
    }
  }
}

template <int M>
cudaError_t launch_gemv(const __nv_bfloat16* X, int ldx, int K, const ProjSet& ps, int rows,
                        cudaStream_t st, bool pdl) {
  const dim3 grid((rows + 3) / 4), block(128);
  if (K != KV_LORA) return cudaErrorInvalidValue;
  return launch_kernel(gemv_f8w_kernel<M, 1>, grid, block, 0, st, pdl, X, ldx, ps);
}

}  // namespace

cudaError_t launch_gemm(const __nv_bfloat16* X, int ldx, int M, int K, const Proj* p, int np,
                        float* partial, int num_sms, int* err, cudaStream_t st, int* adv,
                        int adv_n, int adv_by, bool pdl, const L2Region* pf, int npf) {
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
    if (gemv_stream_supports(M, K))
      return launch_gemv_stream(X, ldx, M, K, p, np, num_sms, err, st, pdl, adv, adv_n, adv_by,
                                pf, npf);
    switch (M) {
      case 1: return launch_gemv<1>(X, ldx, K, ps, rows, st, pdl);
      case 2: return launch_gemv<2>(X, ldx, K, ps, rows, st, pdl);
      default: return launch_gemv<3>(X, ldx, K, ps, rows, st, pdl);
    }
  }
  return launch_gemm_tc(X, ldx, M, K, p, np, partial, num_sms, err, st, adv, adv_n, adv_by);
}

bool gemm_can_advance(int M) { return M > 0; }

}  // namespace mla
