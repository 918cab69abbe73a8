// FP8 block-scaled projection GEMM on the tcgen05 tensor cores.
//
// Y[m, n] = sum_kb s[n/128][kb] * sum_{k in kb} X[m, k] * e4m3(W[n, k])   ("linear" excerpt of
// the "Key-value latent" page: e4m3 weights with one scale per 128x128 block).
//
// The weight is the 128-row MMA operand (D^T[n, m] = W . X^T), so any token count m works
// with N = BN tokens per MMA.  One CTA owns 128 output features (one scale row block) and BN
// tokens, over a run of 128-wide k blocks (split-K when the grid would otherwise be small):
//   warp 0      TMA producer: e4m3 weight tile [128 x 128] and bf16 token tile [BN x 128]
//               into a three-stage ring (128-byte swizzle);
//   warp 1      allocates tensor memory; one thread issues 8 MMAs (K=16) per k block into one
//               of two accumulators, A = converted weight tile, B = token tile;
//   warps 2..5  convert the e4m3 tile to bf16 in the MMA's swizzled K-major layout (exact:
//               every e4m3 value is a bf16 value; integer bit operations, a slower path for the
//               rare subnormal codes);
//   warps 6..9  epilogue: per k block, read the accumulator (lane = feature n) and add it,
//               times that block's scale, to fp32 registers; finally store Y[m, n] (or an
//               fp32 split-K partial).
// Each k block starts a fresh accumulator, so the dequantised weight is never rounded.
#include "tc_common.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int GT_THREADS = 320;
constexpr int GT_STAGES = 3;
constexpr int W_TILE = 128 * 128;              // e4m3 bytes of one weight tile
constexpr int A_TILE = 128 * 128 * 2;          // bf16 bytes of the converted tile (2 atoms)

template <int BN>
struct GemmSmem {
  static constexpr int X_TILE = BN * 128 * 2;  // bf16 token tile, 2 boxes of [BN x 64]
  static constexpr int STAGE = W_TILE + X_TILE;
  static constexpr int OFF_IN = 0;
  static constexpr int OFF_A = OFF_IN + GT_STAGES * STAGE;
  static constexpr int OFF_BAR = OFF_A + 2 * A_TILE;
  static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
  static constexpr int OFF_SCALE = OFF_MISC + 16;
  static constexpr int BYTES = OFF_SCALE + 64 * 4 + 1024;
};

struct GemmTcArgs {
  int M, K;
  int n_tiles0;          // n tiles of problem 0
  int N[2];
  const float* S[2];     // block scales
  void* Y[2];
  int ldy[2];
  int y_fp32[2];
  int splits;            // k-block ranges per (n tile, m tile)
  float* partial;        // [splits][M][ldp] fp32 when splits > 1
  int ldp;               // total N of both problems (partial row stride)
  int* err;
};

// bf16 bits of the e4m3 subnormal magnitude m * 2^-9 (m = 0..7): exact in float, and with at
// most 3 significant bits the upper half of the float is the bf16 value.
__device__ __forceinline__ uint32_t e4m3_sub_bf16(uint32_t m) {
  return __float_as_uint((float)m * 0x1p-9f) >> 16;
}

// Four e4m3 bytes -> four bf16 (two words), exact.  Normal codes: the 7 exponent/mantissa
// bits move up by 4 and the exponent bias grows by 120; zero and subnormal codes (exponent
// field 0, value m * 2^-9) are rare and take a slower path.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t v) {  // v = (b0 << 8) | (b1 << 24)
  uint32_t r = (((v & 0x7F007F00u) >> 4) + 0x3C003C00u) | (v & 0x80008000u);
  if (__vcmpeq2(v & 0x78007800u, 0u)) {
    if ((v & 0x00007800u) == 0)
      r = (r & 0xFFFF0000u) | (v & 0x8000u) | e4m3_sub_bf16((v >> 8) & 7);
    if ((v & 0x78000000u) == 0)
      r = (r & 0x0000FFFFu) | (v & 0x80000000u) | (e4m3_sub_bf16((v >> 24) & 7) << 16);
  }
  return r;
}

template <int BN>
__global__ void __launch_bounds__(GT_THREADS, 1) gemm_f8w_tc_kernel(
    const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
    const __grid_constant__ CUtensorMap map_x, GemmTcArgs args) {
  using L = GemmSmem<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* in_full = bars;        // [3]
  uint64_t* in_empty = bars + 3;   // [3]  converter leader + MMA commit
  uint64_t* a_full = bars + 6;     // [2]  128 converter threads
  uint64_t* a_empty = bars + 8;    // [2]  MMA commit
  uint64_t* acc_full = bars + 10;  // [2]  MMA commit
  uint64_t* acc_empty = bars + 12; // [2]  128 epilogue threads
  uint64_t* mma_idle = bars + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  float* s_scale = reinterpret_cast<float*>(smem + L::OFF_SCALE);
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < GT_STAGES; ++i) {
      mbar_init(&in_full[i], 1);
      mbar_init(&in_empty[i], 2);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 128);
      mbar_init(&a_empty[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
    }
    mbar_init(mma_idle, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 64 && threadIdx.x < nkb)
    s_scale[threadIdx.x] = args.S[prob][(size_t)(n0 / BLK) * nkb_all + kb_begin + threadIdx.x];
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
        tma_prefetch_desc(&map_x);
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
          tma_load_2d(stg + W_TILE, &map_x, &in_full[st], k0, m0);
          tma_load_2d(stg + W_TILE + BN * 128, &map_x, &in_full[st], k0 + 64, m0);
          issued = i + 1;
        }
        volatile int no_abort = 0;
        for (int i = max(0, issued - GT_STAGES); i < issued; ++i)
          mbar_wait(&in_full[i % GT_STAGES], (i / GT_STAGES) & 1, err, &no_abort);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16(128, BN, false, false);
        for (int i = 0; i < nkb; ++i) {
          const int st = i % GT_STAGES, ab = i & 1;
          if (!mbar_wait(&in_full[st], (i / GT_STAGES) & 1, err, abort_flag)) break;
          if (!mbar_wait(&a_full[ab], (i >> 1) & 1, err, abort_flag)) break;
          if (i >= 2 && !mbar_wait(&acc_empty[ab], ((i - 2) >> 1) & 1, err, abort_flag)) break;
          fence_after();
          const uint32_t a_base = sbase + L::OFF_A + ab * A_TILE;
          const uint32_t x_base = sbase + L::OFF_IN + st * L::STAGE + W_TILE;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t a = sdesc_sw128(a_base + (k >> 2) * (A_TILE / 2) + (k & 3) * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(x_base + (k >> 2) * (BN * 128) + (k & 3) * 32, 16, 1024);
            mma_bf16(tmem + ab * BN, a, b, idesc, k > 0);
          }
          mma_commit(&acc_full[ab]);
          mma_commit(&a_empty[ab]);
          mma_commit(&in_empty[st]);
        }
        mma_commit(mma_idle);
        volatile int no_abort = 0;
        mbar_wait(mma_idle, 0, err, &no_abort);
      }
    } else if (warp >= 2 && warp <= 5) {
      // ------------------------------------------------------------------ converters
      const int r = threadIdx.x - 64;  // weight row of this thread, 0..127
      for (int i = 0; i < nkb; ++i) {
        const int st = i % GT_STAGES, ab = i & 1;
        if (!mbar_wait(&in_full[st], (i / GT_STAGES) & 1, err, abort_flag)) break;
        if (i >= 2 && !mbar_wait(&a_empty[ab], ((i - 2) >> 1) & 1, err, abort_flag)) break;
        const uint8_t* wrow = smem + L::OFF_IN + st * L::STAGE + r * 128;
        uint8_t* arow = smem + L::OFF_A + ab * A_TILE + r * 128;
        const int sw = r & 7;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // e4m3 chunk c: k = 16c .. 16c+15
          const uint4 q = *reinterpret_cast<const uint4*>(wrow + ((c ^ sw) << 4));
          const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
          uint32_t o[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            o[2 * j] = e4m3x2_to_bf16x2(__byte_perm(w4[j], 0, 0x1404));
            o[2 * j + 1] = e4m3x2_to_bf16x2(__byte_perm(w4[j], 0, 0x3424));
          }
          uint8_t* atom = arow + (c >> 2) * (A_TILE / 2);
          const int j0 = 2 * (c & 3);
          *reinterpret_cast<uint4*>(atom + (((j0) ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(atom + (((j0 + 1) ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async();
        mbar_arrive(&a_full[ab]);
        named_bar(2, 128);  // every converter is done reading this stage's weight tile
        if (r == 0) mbar_arrive(&in_empty[st]);
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
      if (ok && n < n0 + 128 && n < args.N[prob]) {
        const int mend = min(BN, args.M - m0);
        if (args.splits > 1) {
          float* p = args.partial + ((size_t)split * args.M + m0) * args.ldp +
                     (prob ? args.N[0] : 0) + n;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j < mend) p[(size_t)j * args.ldp] = acc[j];
        } else if (args.y_fp32[prob]) {
          float* y = reinterpret_cast<float*>(args.Y[prob]) + (size_t)m0 * args.ldy[prob] + n;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j < mend) y[(size_t)j * args.ldy[prob]] = acc[j];
        } else {
          __nv_bfloat16* y =
              reinterpret_cast<__nv_bfloat16*>(args.Y[prob]) + (size_t)m0 * args.ldy[prob] + n;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j < mend) y[(size_t)j * args.ldy[prob]] = __float2bfloat16_rn(acc[j]);
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
cudaError_t launch_bn(const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap& x,
                      const GemmTcArgs& a, int n_tiles, cudaStream_t st) {
  const dim3 grid(n_tiles, (a.M + BN - 1) / BN, a.splits);
  gemm_f8w_tc_kernel<BN><<<grid, GT_THREADS, GemmSmem<BN>::BYTES, st>>>(w0, w1, x, a);
  return cudaGetLastError();
}

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

size_t gemm_partial_bytes(int M, int N_total, int K, int num_sms) {
  const int s = gemm_splits(M, N_total, K, num_sms);
  return s > 1 ? (size_t)s * M * N_total * sizeof(float) : 0;
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
                           float* partial, int num_sms, int* err, cudaStream_t st) {
  const int bn = gemm_bn(M);
  GemmTcArgs a{};
  a.M = M;
  a.K = K;
  a.err = err;
  CUtensorMap mw[2], mx;
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
  if (!make_tmap_2d(&mx, true, X, (uint64_t)K, (uint64_t)M, (uint64_t)ldx * 2, 64, bn))
    return cudaErrorInvalidValue;
  a.n_tiles0 = (p[0].N + 127) / 128;
  const int n_tiles = a.n_tiles0 + (np > 1 ? (p[1].N + 127) / 128 : 0);
  a.splits = gemm_splits(M, n_total, K, num_sms);
  a.partial = partial;
  a.ldp = n_total;
  if (a.splits > 1 && !partial) return cudaErrorInvalidValue;
  cudaError_t e;
  switch (bn) {
    case 32: e = launch_bn<32>(mw[0], mw[1], mx, a, n_tiles, st); break;
    case 64: e = launch_bn<64>(mw[0], mw[1], mx, a, n_tiles, st); break;
    default: e = launch_bn<128>(mw[0], mw[1], mx, a, n_tiles, st); break;
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
