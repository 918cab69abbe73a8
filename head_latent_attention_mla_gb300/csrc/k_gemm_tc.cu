// FP8 block-scaled projection GEMM on the tcgen05 tensor cores.
//
// Y[m, n] = sum_kb s[n/128][kb] * sum_{k in kb} X[m, k] * e4m3(W[n, k])   ("linear" excerpt of
// the "Key-value latent" page: e4m3 weights with one scale per 128x128 block; the config's
// activation_scheme is dynamic).
//
// The bf16 activations are first split, per token row, into two e4m3 terms,
//   X[m, k] ~= sx[m] * (hi[m, k] + lo[m, k]),  sx[m] = amax_k |X[m, k]| / 448,
//   hi = e4m3(X / sx), lo = e4m3(X / sx - hi)            (relative error <= 2^-8),
// so that both MMA operands are e4m3 and the weights feed the tensor cores exactly as stored:
// two kind::f8f6f4 MMAs (hi, then lo) cost what one bf16 MMA would, and no weight conversion
// is needed.  The weight is the 128-row MMA operand (D^T[n, m] = W . X^T), so any token count
// works with N = BN tokens per MMA.  One CTA owns 128 output features (one scale row block) and
// BN tokens over a run of 128-wide k blocks (split-K when the grid would otherwise be small):
//   warp 0      TMA producer: weight tile [128 x 128] and hi/lo token tiles [BN x 128] into a
//               four-stage ring (128-byte swizzle);
//   warp 1      allocates tensor memory; one thread issues 4 x 2 MMAs (K=32) per k block into
//               one of two accumulators;
//   warps 2..5  epilogue: per k block, read the accumulator (lane = feature n) and add it,
//               times that block's scale, to fp32 registers; finally multiply by the token's
//               sx and store Y[m, n] (or an fp32 split-K partial).
// Each k block starts a fresh accumulator, so the weight's block scales are applied exactly.
#include "tc_common.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int GT_THREADS = 192;
constexpr int GT_STAGES = 4;
constexpr int W_TILE = 128 * 128;              // e4m3 bytes of one weight tile
constexpr float E4M3_MAX = 448.f;

template <int BN>
struct GemmSmem {
  static constexpr int X_TILE = BN * 128;      // e4m3 token tile [BN x 128]
  static constexpr int STAGE = W_TILE + 2 * X_TILE;
  static constexpr int OFF_IN = 0;
  static constexpr int OFF_BAR = OFF_IN + GT_STAGES * STAGE;
  static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
  static constexpr int OFF_SCALE = OFF_MISC + 16;
  static constexpr int OFF_SX = OFF_SCALE + 64 * 4;
  static constexpr int BYTES = OFF_SX + BN * 4 + 1024;
};

struct GemmTcArgs {
  int M, K;
  int n_tiles0;          // n tiles of problem 0
  int N[2];
  const float* S[2];     // weight block scales
  void* Y[2];
  int ldy[2];
  int y_fp32[2];
  const float* sx;       // [M] per-token activation scales
  int splits;            // k-block ranges per (n tile, m tile)
  float* partial;        // [splits][M][ldp] fp32 when splits > 1
  int ldp;               // total N of both problems (partial row stride)
  int* err;
};

// One CTA per token row: sx = amax/448 (1 for an all-zero row), hi = e4m3(x/sx),
// lo = e4m3(x/sx - hi), both rounded to nearest even with saturation.
__global__ void __launch_bounds__(256) split_e4m3_kernel(const __nv_bfloat16* __restrict__ X,
                                                         int ldx, int K, uint8_t* __restrict__ hi,
                                                         uint8_t* __restrict__ lo,
                                                         float* __restrict__ sx) {
  __shared__ float red[8];
  const int m = blockIdx.x, tid = threadIdx.x;
  const __nv_bfloat16* row = X + (size_t)m * ldx;
  float amax = 0.f;
  for (int k = tid * 8; k < K; k += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + k);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(u[i] << 16)),
                               fabsf(__uint_as_float(u[i] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid < 32) {
    float a = tid < 8 ? red[tid] : 0.f;
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if (tid == 0) red[0] = a;
  }
  __syncthreads();
  const float s = red[0] > 0.f ? red[0] / E4M3_MAX : 1.f;
  const float inv = 1.f / s;
  if (tid == 0) sx[m] = s;
  for (int k = tid * 8; k < K; k += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + k);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[2] = {0u, 0u}, l[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = make_float2(__uint_as_float(u[i] << 16) * inv,
                                   __uint_as_float(u[i] & 0xFFFF0000u) * inv);
      const __nv_fp8x2_storage_t hp = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      const __half2_raw hh = __nv_cvt_fp8x2_to_halfraw2(hp, __NV_E4M3);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hh));
      const __nv_fp8x2_storage_t lp =
          __nv_cvt_float2_to_fp8x2(make_float2(f.x - hf.x, f.y - hf.y), __NV_SATFINITE, __NV_E4M3);
      h[i >> 1] |= (uint32_t)hp << (16 * (i & 1));
      l[i >> 1] |= (uint32_t)lp << (16 * (i & 1));
    }
    *reinterpret_cast<uint2*>(hi + (size_t)m * K + k) = make_uint2(h[0], h[1]);
    *reinterpret_cast<uint2*>(lo + (size_t)m * K + k) = make_uint2(l[0], l[1]);
  }
}

template <int BN>
__global__ void __launch_bounds__(GT_THREADS, 1) gemm_f8w_tc_kernel(
    const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
    const __grid_constant__ CUtensorMap map_hi, const __grid_constant__ CUtensorMap map_lo,
    GemmTcArgs args) {
  using L = GemmSmem<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* in_full = bars;                    // [4]  TMA transaction bytes
  uint64_t* in_empty = bars + GT_STAGES;       // [4]  MMA commit
  uint64_t* acc_full = bars + 2 * GT_STAGES;   // [2]  MMA commit
  uint64_t* acc_empty = acc_full + 2;          // [2]  128 epilogue threads
  uint64_t* mma_idle = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  float* s_scale = reinterpret_cast<float*>(smem + L::OFF_SCALE);
  float* s_sx = reinterpret_cast<float*>(smem + L::OFF_SX);
  constexpr uint32_t TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int nt = blockIdx.x;
  const int prob = nt < args.n_tiles0 ? 0 : 1;
  if (prob) nt -= args.n_tiles0;
  const int n0 = nt * 128, m0 = blockIdx.y * BN;
  const int nkb_all = args.K / BLK;
  const int split = blockIdx.z;
  const int kb_begin = (int)((long)nkb_all * split / args.splits);
  const int kb_end = (int)((long)nkb_all * (split + 1) / args.splits);
  const int nkb = kb_end - kb_begin;
  const CUtensorMap* map_w = prob ? &map_w1 : &map_w0;
  const float* scales = prob ? args.S[1] : args.S[0];

  if (threadIdx.x == 0) {
    for (int i = 0; i < GT_STAGES; ++i) {
      mbar_init(&in_full[i], 1);
      mbar_init(&in_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
    }
    mbar_init(mma_idle, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 64 && threadIdx.x < nkb)
    s_scale[threadIdx.x] = scales[(size_t)(n0 / BLK) * nkb_all + kb_begin + threadIdx.x];
  for (int j = threadIdx.x; j < BN; j += GT_THREADS)
    s_sx[j] = (m0 + j < args.M) ? args.sx[m0 + j] : 0.f;
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  int* err = args.err;

  if (nkb > 0) {
    if (warp == 0) {
      // ------------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(map_w);
        tma_prefetch_desc(&map_hi);
        tma_prefetch_desc(&map_lo);
        int issued = 0;
        for (int i = 0; i < nkb; ++i) {
          const int st = i % GT_STAGES;
          if (i >= GT_STAGES &&
              !mbar_wait(&in_empty[st], ((i - GT_STAGES) / GT_STAGES) & 1, err, abort_flag))
            break;
          uint8_t* stg = smem + L::OFF_IN + st * L::STAGE;
          const int k0 = (kb_begin + i) * BLK;
          mbar_expect_tx(&in_full[st], L::STAGE);
          tma_load_2d(stg, map_w, &in_full[st], k0, n0);
          tma_load_2d(stg + W_TILE, &map_hi, &in_full[st], k0, m0);
          tma_load_2d(stg + W_TILE + L::X_TILE, &map_lo, &in_full[st], k0, m0);
          issued = i + 1;
        }
        volatile int no_abort = 0;
        for (int i = max(0, issued - GT_STAGES); i < issued; ++i)
          mbar_wait(&in_full[i % GT_STAGES], (i / GT_STAGES) & 1, err, &no_abort);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3(128, BN);
        for (int i = 0; i < nkb; ++i) {
          const int st = i % GT_STAGES, ab = i & 1;
          if (!mbar_wait(&in_full[st], (i / GT_STAGES) & 1, err, abort_flag)) break;
          if (i >= 2 && !mbar_wait(&acc_empty[ab], ((i - 2) >> 1) & 1, err, abort_flag)) break;
          fence_after();
          const uint32_t w_base = sbase + L::OFF_IN + st * L::STAGE;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = sdesc_sw128(w_base + k * 32, 16, 1024);
            const uint64_t bh = sdesc_sw128(w_base + W_TILE + k * 32, 16, 1024);
            const uint64_t bl = sdesc_sw128(w_base + W_TILE + L::X_TILE + k * 32, 16, 1024);
            mma_e4m3(tmem + ab * BN, a, bh, idesc, k > 0);
            mma_e4m3(tmem + ab * BN, a, bl, idesc, true);
          }
          mma_commit(&acc_full[ab]);
          mma_commit(&in_empty[st]);
        }
        mma_commit(mma_idle);
        volatile int no_abort = 0;
        mbar_wait(mma_idle, 0, err, &no_abort);
      }
    } else {
      // ------------------------------------------------------------------ epilogue
      const int q = warp & 3;
      const int n = n0 + 32 * q + lane;
      const uint32_t lane_off = (uint32_t)(32 * q) << 16;
      float acc[BN];
#pragma unroll
      for (int j = 0; j < BN; ++j) acc[j] = 0.f;
      bool ok = true;
      for (int i = 0; i < nkb; ++i) {
        const int ab = i & 1;
        if (!(ok = mbar_wait(&acc_full[ab], (i >> 1) & 1, err, abort_flag))) break;
        fence_after();
        const float sc = s_scale[i];
#pragma unroll
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + ab * BN + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[c + j] = fmaf(sc, __uint_as_float(v[j]), acc[c + j]);
        }
        fence_before();
        mbar_arrive(&acc_empty[ab]);
      }
      if (ok && n < (prob ? args.N[1] : args.N[0])) {
        const int mend = min(BN, args.M - m0);
        const int ldy = prob ? args.ldy[1] : args.ldy[0];
        if (args.splits > 1) {
          float* p = args.partial + ((size_t)split * args.M + m0) * args.ldp +
                     (prob ? args.N[0] : 0) + n;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j < mend) p[(size_t)j * args.ldp] = acc[j] * s_sx[j];
        } else if (prob ? args.y_fp32[1] : args.y_fp32[0]) {
          float* y = reinterpret_cast<float*>(prob ? args.Y[1] : args.Y[0]) + (size_t)m0 * ldy + n;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j < mend) y[(size_t)j * ldy] = acc[j] * s_sx[j];
        } else {
          __nv_bfloat16* y =
              reinterpret_cast<__nv_bfloat16*>(prob ? args.Y[1] : args.Y[0]) + (size_t)m0 * ldy + n;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j < mend) y[(size_t)j * ldy] = __float2bfloat16_rn(acc[j] * s_sx[j]);
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Y = sum over splits of the fp32 partials, in split order (deterministic).
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, int M, int ldp,
                                     int n_off, int N, void* Y, int ldy, int y_fp32) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)M * N) return;
  const int m = (int)(i / N), n = (int)(i % N);
  float s = 0.f;
  for (int k = 0; k < splits; ++k) s += part[((size_t)k * M + m) * ldp + n_off + n];
  if (y_fp32)
    reinterpret_cast<float*>(Y)[(size_t)m * ldy + n] = s;
  else
    reinterpret_cast<__nv_bfloat16*>(Y)[(size_t)m * ldy + n] = __float2bfloat16_rn(s);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap* w, const CUtensorMap& hi, const CUtensorMap& lo,
                      const GemmTcArgs& a, int n_tiles, cudaStream_t st) {
  const dim3 grid(n_tiles, (a.M + BN - 1) / BN, a.splits);
  gemm_f8w_tc_kernel<BN><<<grid, GT_THREADS, GemmSmem<BN>::BYTES, st>>>(w[0], w[1], hi, lo, a);
  return cudaGetLastError();
}

constexpr size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

bool make_tmap_2d(CUtensorMap* m, bool bf16, const void* base, uint64_t cols, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows);

int gemm_bn(int M) { return M <= 32 ? 32 : (M <= 64 ? 64 : 128); }

int gemm_splits(int M, int N_total, int K, int num_sms) {
  if (M <= 8) return 1;
  const int bn = gemm_bn(M);
  const int tiles = ((N_total + 127) / 128) * ((M + bn - 1) / bn);
  const int nkb = K / BLK;
  int s = (num_sms + tiles - 1) / tiles;
  if (s > nkb / 4) s = nkb / 4;
  return s < 1 ? 1 : s;
}

// Scratch of one tensor-core GEMM: hi and lo e4m3 copies of X [M, K], sx [M], and the split-K
// partials.
size_t gemm_partial_bytes(int M, int N_total, int K, int num_sms) {
  if (M <= 8) return 0;
  const int s = gemm_splits(M, N_total, K, num_sms);
  return 2 * up256((size_t)M * K) + up256((size_t)M * 4) +
         (s > 1 ? (size_t)s * M * N_total * sizeof(float) : 0);
}

cudaError_t init_gemm_tc_kernels() {
  cudaError_t e = cudaFuncSetAttribute(gemm_f8w_tc_kernel<32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       GemmSmem<32>::BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_f8w_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GemmSmem<64>::BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_f8w_tc_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, GemmSmem<128>::BYTES);
  return e;
}

cudaError_t launch_gemm_tc(const __nv_bfloat16* X, int ldx, int M, int K, const Proj* p, int np,
                           float* scratch, int num_sms, int* err, cudaStream_t st) {
  if (!scratch) return cudaErrorInvalidValue;
  const int bn = gemm_bn(M);
  uint8_t* base = reinterpret_cast<uint8_t*>(scratch);
  uint8_t* hi = base;
  uint8_t* lo = hi + up256((size_t)M * K);
  float* sx = reinterpret_cast<float*>(lo + up256((size_t)M * K));
  float* partial = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sx) + up256((size_t)M * 4));

  split_e4m3_kernel<<<M, 256, 0, st>>>(X, ldx, K, hi, lo, sx);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  GemmTcArgs a{};
  a.M = M;
  a.K = K;
  a.err = err;
  a.sx = sx;
  CUtensorMap mw[2], mh, ml;
  int n_total = 0;
  for (int i = 0; i < 2; ++i) {
    const Proj& P = p[i < np ? i : 0];
    if (!make_tmap_2d(&mw[i], false, P.W, (uint64_t)K, (uint64_t)P.N, (uint64_t)K, 128, 128))
      return cudaErrorInvalidValue;
    if (i < np) {
      a.N[i] = P.N;
      a.S[i] = P.S;
      a.Y[i] = P.Y;
      a.ldy[i] = P.ldy;
      a.y_fp32[i] = P.y_fp32;
      n_total += P.N;
    }
  }
  if (!make_tmap_2d(&mh, false, hi, (uint64_t)K, (uint64_t)M, (uint64_t)K, 128, bn) ||
      !make_tmap_2d(&ml, false, lo, (uint64_t)K, (uint64_t)M, (uint64_t)K, 128, bn))
    return cudaErrorInvalidValue;
  a.n_tiles0 = (p[0].N + 127) / 128;
  const int n_tiles = a.n_tiles0 + (np > 1 ? (p[1].N + 127) / 128 : 0);
  a.splits = gemm_splits(M, n_total, K, num_sms);
  a.partial = partial;
  a.ldp = n_total;
  switch (bn) {
    case 32: e = launch_bn<32>(mw, mh, ml, a, n_tiles, st); break;
    case 64: e = launch_bn<64>(mw, mh, ml, a, n_tiles, st); break;
    default: e = launch_bn<128>(mw, mh, ml, a, n_tiles, st); break;
  }
  if (e != cudaSuccess || a.splits == 1) return e;
  for (int i = 0; i < np; ++i) {
    const size_t cnt = (size_t)M * p[i].N;
    splitk_reduce_kernel<<<(unsigned)((cnt + 255) / 256), 256, 0, st>>>(
        partial, a.splits, M, n_total, i ? p[0].N : 0, p[i].N, p[i].Y, p[i].ldy, p[i].y_fp32);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace mla
