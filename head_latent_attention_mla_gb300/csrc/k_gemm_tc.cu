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
// works with N = BN tokens per MMA.
//
// Persistent kernel, one CTA per SM.  The work is cut into units (128 output features = one
// scale row block) x (BN tokens) x (a run of 128-wide k blocks; split-K when there are few
// tiles), and each CTA walks units c, c + G, ... with its pipelines running across unit
// boundaries:
//   warp 0      TMA producer: weight tile [128 x 128] and hi/lo token tiles [BN x 128] into a
//               four-stage ring (128-byte swizzle);
//   warp 1      allocates tensor memory; one thread issues 4 x 2 MMAs (K=32) per k block into
//               one of four accumulators;
//   warps 2..9  epilogue, two warpgroups each owning half of the BN token columns: per k
//               block, read the accumulator (lane = feature n), release it, and add it, times
//               that block's scale, to fp32 registers; at the end of a unit multiply by the
//               token's sx and store Y[m, n] (or an fp32 split-K partial) while the MMAs of the
//               next unit already run.
// Each k block starts a fresh accumulator, so the weight's block scales are applied exactly.
#include "tc_common.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int GT_THREADS = 320;
constexpr float E4M3_MAX = 448.f;
constexpr int W_TILE = 128 * 128;              // e4m3 bytes of one weight tile
// Bytes of the stage ring.  The loads, not the tensor cores, set the pace: a stage is busy for
// its load latency (about 2 us under full load) plus its MMAs, so the ring is as large as
// shared memory allows.  Stages of 128-byte rows: halving them to 64-byte rows (twice the
// stages, twice the copy requests) measured slower.
constexpr int GT_RING = 192 * 1024;

// BN tokens per unit; WT weight tiles (of 128 features) per unit.  WT = 2 reads the token
// tile once for 256 features: 1.5x the MMA work per staged byte.
//
// Orientation of the accumulator.  With BN = 128 the token tile is the MMA's A operand
// (M = 128 tokens) and the weight tiles its B operand (N = 128 WT features): tensor-memory
// lane = token, column = feature, so each epilogue thread ends a unit holding a run of one
// output row and writes it as 16-byte vectors.  With fewer tokens (BN = 32, 64) the weight
// tile is the A operand (M = 128 features, N = BN tokens): lane = feature, column = token.
// ONE: the activations are a single e4m3 term (the FP8-activation option) instead of the
// hi/lo pair: one MMA per k step, and a stage holds one token tile.
template <int BN, int WT, bool ONE = false>
struct GemmSmem {
  static constexpr bool TR = BN == 128;          // lane = token (else lane = feature)
  static constexpr int NACC = WT == 2 ? 2 : 4;   // tensor-memory accumulators
  static constexpr int ACC_COLS = WT * BN;       // columns of one accumulator (WT halves)
  static constexpr int X_TILE = BN * 128;        // e4m3 token tile [BN x 128]
  static constexpr int W_BYTES = WT * W_TILE;
  static constexpr int NX = ONE ? 1 : 2;         // activation terms per stage
  static constexpr int STAGE = W_BYTES + NX * X_TILE;
  static constexpr int STAGES = GT_RING / STAGE;
  static constexpr int OFF_IN = 0;
  static constexpr int OFF_BAR = OFF_IN + STAGES * STAGE;
  static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  // Epilogue warpgroups: one per weight half when WT = 2 (each holds the 128 accumulator
  // columns of its 128 features), else two (one) splitting the accumulator's columns.
  static constexpr int NGRP = WT == 2 ? 2 : (BN >= 64 ? 2 : 1);
  static constexpr int CW = WT == 2 ? 128 : BN / NGRP;  // accumulator columns per thread
  static constexpr int CH = WT == 2 ? 16 : CW;    // columns read from TMEM at once
  static constexpr uint32_t TMEM_COLS = NACC * ACC_COLS < 32 ? 32 : NACC * ACC_COLS;
  static_assert(2 * STAGES + 2 * NACC + 1 <= 32, "barrier space");
  static_assert(WT == 1 || TR, "two weight tiles only with the token-lane orientation");
  static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte alignment of the ring");
  static_assert(TMEM_COLS <= 512, "tensor memory");
  static_assert(BYTES <= 227 * 1024, "shared memory");
  static_assert(CW % 32 == 0 && CW % CH == 0 && (CH == 16 || CH % 32 == 0), "epilogue columns");
};

struct GemmTcArgs {
  int M, K;
  int n_tiles0;          // n tiles of problem 0
  int n_tiles;           // n tiles of both problems
  int m_tiles;
  int units;             // n_tiles * m_tiles * splits
  int N[2];
  const float* S[2];     // weight block scales
  void* Y[2];
  int ldy[2];
  int y_fp32[2];
  const __nv_bfloat16* R[2];  // bf16 outputs: residual added after rounding (or nullptr)
  const float* sx;       // per-token activation scales [M], or [M][K/128] (SXB kernels)
  int splits;            // k-block ranges per (n tile, m tile)
  float* partial;        // [splits][M][ldp] fp32 when splits > 1
  int ldp;               // total N of both problems (partial row stride)
  int* err;
  int* adv;              // CTA 0 adds adv_by to adv[0..adv_n) (the call's length update)
  int adv_n, adv_by;
  // Batched GEMMs (batches > 1; one problem, no split-K): batch b multiplies weight rows
  // w_row_base + b w_row_step + [0, N), token rows b x_row_step + [0, M) of the hi/lo maps and
  // sx, block scales S[0] + b s_step, and writes Y[0] + b y_step (elements).
  int batches;
  int w_row_base, w_row_step, x_row_step, s_step;
  long long y_step;
};

// Unit u: split fastest, then m tile, then n tile (CTAs running at the same time share weight
// tiles through L2).
struct Unit {
  int prob, n0, m0, split, kb_begin, kb_end, batch;
};
template <bool BATCH>
__device__ __forceinline__ Unit unit_of(const GemmTcArgs& a, int u, int BN, int WT) {
  Unit r;
  r.batch = 0;
  if constexpr (BATCH) {
    const int per_batch = a.units / a.batches;
    r.batch = u / per_batch;
    u -= r.batch * per_batch;
  }
  r.split = u % a.splits;
  const int t = u / a.splits;
  const int mt = t % a.m_tiles;
  int nt = t / a.m_tiles;
  r.prob = nt < a.n_tiles0 ? 0 : 1;
  if (r.prob) nt -= a.n_tiles0;
  r.n0 = nt * 128 * WT;
  r.m0 = mt * BN;
  const int nkb = a.K / BLK;
  r.kb_begin = (int)((long)nkb * r.split / a.splits);
  r.kb_end = (int)((long)nkb * (r.split + 1) / a.splits);
  return r;
}

// One CTA per token row: sx = amax/448 (1 for an all-zero row), hi = e4m3(x/sx),
// lo = e4m3(x/sx - hi), both rounded to nearest even with saturation.  Safe under
// programmatic dependent launch (X comes from the previous kernel; hi, lo and sx may still be
// read by an earlier GEMM until the wait returns).
__global__ void __launch_bounds__(256) split_e4m3_kernel(const __nv_bfloat16* X, int ldx, int K,
                                                         uint8_t* __restrict__ hi,
                                                         uint8_t* __restrict__ lo,
                                                         float* __restrict__ sx) {
  __shared__ float red[8];
  const int m = blockIdx.x, tid = threadIdx.x;
  const __nv_bfloat16* row = X + (size_t)m * ldx;
  pdl_launch_dependents();
  pdl_wait();
  float amax = 0.f;
  for (int k = tid * 8; k < K; k += 256 * 8) {
    const uint4 v = ld_dep_v4(row + k);
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
    const uint4 v = ld_dep_v4(row + k);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[2] = {0u, 0u}, l[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t hl = e4m3_split2(make_float2(__uint_as_float(u[i] << 16) * inv,
                                                  __uint_as_float(u[i] & 0xFFFF0000u) * inv));
      h[i >> 1] |= (hl & 0xFFFFu) << (16 * (i & 1));
      l[i >> 1] |= (hl >> 16) << (16 * (i & 1));
    }
    *reinterpret_cast<uint2*>(hi + (size_t)m * K + k) = make_uint2(h[0], h[1]);
    *reinterpret_cast<uint2*>(lo + (size_t)m * K + k) = make_uint2(l[0], l[1]);
  }
}

// The two-term split of per-(sequence, head) rows for the batched absorption GEMMs, written
// head-major: CTA (b, h) splits X[b * sb + h * sh + 0 .. K) (as split_e4m3_kernel does) into row
// h * B + b of hi / lo / sx, so that head h's B token rows are contiguous.  With rope_out set
// (the query absorption), it also writes RoPE of the head's rotary slice X[.. + K .. + K + 64)
// at position seq_lens[b] into rope_out[(b * H + h) * rope_ld + 0 .. 64), as a plain rotation
// of pairs (pairing 0: (2j, 2j+1); 1: (j, j+32)).  max(32, K / 8) threads, eight values each
// (K <= 512); launched under programmatic dependent launch (X comes from an earlier kernel).
__global__ void __launch_bounds__(64) split_heads_e4m3_kernel(
    const __nv_bfloat16* X, int B, int H, long long sb, int sh, int K, uint8_t* __restrict__ hi,
    uint8_t* __restrict__ lo, float* __restrict__ sx, __nv_bfloat16* rope_out, int rope_ld,
    const float2* __restrict__ rope_tab, int pairing, const int* __restrict__ seq_lens,
    int limit) {
  __shared__ float red[2];
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const __nv_bfloat16* row = X + (size_t)b * sb + (size_t)h * sh;
  const size_t r = (size_t)h * B + b;
  pdl_launch_dependents();
  pdl_wait();
  const bool act = 8 * tid < K;
  const uint4 v = act ? ld_dep_v4(row + 8 * tid) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = blockDim.x > 32 ? fmaxf(red[0], red[1]) : red[0];
  const float sc = amax > 0.f ? amax / E4M3_MAX : 1.f;
  const float inv = 1.f / sc;
  if (tid == 0) sx[r] = sc;
  uint32_t hw[2] = {0u, 0u}, lw[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t hl = e4m3_split2(make_float2(f[2 * i] * inv, f[2 * i + 1] * inv));
    hw[i >> 1] |= (hl & 0xFFFFu) << (16 * (i & 1));
    lw[i >> 1] |= (hl >> 16) << (16 * (i & 1));
  }
  if (act) {
    *reinterpret_cast<uint2*>(hi + r * K + 8 * tid) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(lo + r * K + 8 * tid) = make_uint2(lw[0], lw[1]);
  }
  if (rope_out && tid < ROPE / 2) {
    const int pos = seq_lens[b];
    if (pos >= 0 && pos < limit) {
      const int2 ij = pairing == 0 ? make_int2(2 * tid, 2 * tid + 1) : make_int2(tid, tid + ROPE / 2);
      const float x0 = ld_dep_bf16(row + K + ij.x), x1 = ld_dep_bf16(row + K + ij.y);
      const float2 cs = rope_tab[(size_t)pos * (ROPE / 2) + tid];
      __nv_bfloat16* dst = rope_out + ((size_t)b * H + h) * rope_ld;
      dst[ij.x] = __float2bfloat16_rn(x0 * cs.x - x1 * cs.y);
      dst[ij.y] = __float2bfloat16_rn(x1 * cs.x + x0 * cs.y);
    }
  }
}

// The FP8-activation option's input quantisation ("linear" excerpt: activation_scheme dynamic):
// one e4m3 term per value with one scale per (token, 128-wide group), s = amax / 448 (1 for an
// all-zero group), q = e4m3(x / s) rounded to nearest even with saturation.  One CTA per token,
// K/8 threads of eight values; the sixteen threads of a group find its maximum by shuffles.
__global__ void __launch_bounds__(1024) quant_e4m3_groups_kernel(const __nv_bfloat16* X,
                                                                 int ldx, int K,
                                                                 uint8_t* __restrict__ q,
                                                                 float* __restrict__ sx) {
  pdl_launch_dependents();
  pdl_wait();  // X may come from the previous kernel
  const int m = blockIdx.x, tid = threadIdx.x, k = 8 * tid;
  const uint4 v = ld_dep_v4(X + (size_t)m * ldx + k);
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  float f[8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = amax > 0.f ? amax / E4M3_MAX : 1.f;
  const float inv = 1.f / s;
  uint32_t h[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t p =
        __nv_cvt_float2_to_fp8x2(make_float2(f[2 * i] * inv, f[2 * i + 1] * inv), __NV_SATFINITE,
                                 __NV_E4M3);
    h[i >> 1] |= (uint32_t)p << (16 * (i & 1));
  }
  *reinterpret_cast<uint2*>(q + (size_t)m * K + k) = make_uint2(h[0], h[1]);
  if ((tid & 15) == 0) sx[(size_t)m * (K / BLK) + k / BLK] = s;
}

// Two floats as bf16 (round to nearest even), the first in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// SXB: the activations carry one scale per (token, 128-wide k block), sx[m][kb], applied with
// the weight's block scale to each k block's partial product (token-lane orientation only).
// ONE: the activations are one e4m3 term (map_lo is not read).
template <int BN, int WT, bool SXB, bool ONE = false, bool BATCH = false>
__global__ void __launch_bounds__(GT_THREADS, 1) gemm_f8w_tc_kernel(
    const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
    const __grid_constant__ CUtensorMap map_hi, const __grid_constant__ CUtensorMap map_lo,
    const __grid_constant__ GemmTcArgs args) {
  using L = GemmSmem<BN, WT, ONE>;
  static_assert(!SXB || L::TR, "block-scaled activations need the token-lane orientation");
  static_assert(!ONE || SXB, "single-term activations come with per-block scales");
  constexpr int GT_STAGES = L::STAGES;
  constexpr int GT_NACC = L::NACC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* in_full = bars;                        // [GT_STAGES]  TMA transaction bytes
  uint64_t* in_empty = bars + GT_STAGES;           // [GT_STAGES]  MMA commit
  uint64_t* acc_full = bars + 2 * GT_STAGES;       // [GT_NACC]    MMA commit
  uint64_t* acc_empty = acc_full + GT_NACC;        // [GT_NACC]    epilogue threads
  uint64_t* mma_idle = acc_empty + GT_NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb_all = args.K / BLK;
  int* err = args.err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < GT_STAGES; ++i) {
      mbar_init(&in_full[i], 1);
      mbar_init(&in_empty[i], 1);
    }
    for (int i = 0; i < GT_NACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128 * L::NGRP);
    }
    mbar_init(mma_idle, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  // Under programmatic dependent launch this kernel may start while the previous one runs:
  // the weight tiles of the first stages are requested before the wait (the weights do not
  // depend on it); everything that reads or writes the previous kernels' data comes after.
  pdl_launch_dependents();
  if (warp == 0) {
    // -------------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_w0);
      tma_prefetch_desc(&map_w1);
      tma_prefetch_desc(&map_hi);
      tma_prefetch_desc(&map_lo);
      int npre = 0;  // stages whose weight tiles are issued before the wait
      for (int u = blockIdx.x; npre < GT_STAGES && u < args.units; u += gridDim.x) {
        const Unit U = unit_of<BATCH>(args, u, BN, WT);
        const CUtensorMap* map_w = U.prob ? &map_w1 : &map_w0;
        const int wt = (WT == 2 && U.n0 + 128 >= args.N[U.prob]) ? 1 : WT;
        const int wrow = args.w_row_base + U.batch * args.w_row_step + U.n0;
        for (int kb = U.kb_begin; npre < GT_STAGES && kb < U.kb_end; ++kb, ++npre) {
          uint8_t* stg = smem + L::OFF_IN + npre * L::STAGE;
          mbar_expect_tx(&in_full[npre], L::STAGE - (WT - wt) * W_TILE);
          for (int h = 0; h < wt; ++h)
            tma_load_2d(stg + h * W_TILE, map_w, &in_full[npre], kb * BLK, wrow + 128 * h);
        }
      }
      pdl_wait();
      int i = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < args.units; u += gridDim.x) {
        const Unit U = unit_of<BATCH>(args, u, BN, WT);
        const CUtensorMap* map_w = U.prob ? &map_w1 : &map_w0;
        for (int kb = U.kb_begin; ok && kb < U.kb_end; ++kb, ++i) {
          const int st = i % GT_STAGES;
          if (i >= GT_STAGES &&
              !(ok = mbar_wait(&in_empty[st], ((i / GT_STAGES) - 1) & 1, err, abort_flag)))
            break;
          uint8_t* stg = smem + L::OFF_IN + st * L::STAGE;
          const int k0 = kb * BLK;
          // A weight half that lies wholly past N is neither loaded nor multiplied.
          const int wt = (WT == 2 && U.n0 + 128 >= args.N[U.prob]) ? 1 : WT;
          const int wrow = args.w_row_base + U.batch * args.w_row_step + U.n0;
          const int xrow = U.batch * args.x_row_step + U.m0;
          if (i >= npre) {  // (the first npre stages' weight tiles are already on their way)
            mbar_expect_tx(&in_full[st], L::STAGE - (WT - wt) * W_TILE);
            for (int h = 0; h < wt; ++h)
              tma_load_2d(stg + h * W_TILE, map_w, &in_full[st], k0, wrow + 128 * h);
          }
          tma_load_2d(stg + L::W_BYTES, &map_hi, &in_full[st], k0, xrow);
          if constexpr (!ONE) tma_load_2d(stg + L::W_BYTES + L::X_TILE, &map_lo, &in_full[st], k0, xrow);
        }
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the last ones.
      volatile int no_abort = 0;
      for (int j = max(0, i - GT_STAGES); j < i; ++j)
        mbar_wait(&in_full[j % GT_STAGES], (j / GT_STAGES) & 1, err, &no_abort);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(128, L::TR ? 128 : BN);
      constexpr uint32_t idesc2 = idesc_e4m3(128, 256);  // token-lane, two weight tiles
      int i = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < args.units; u += gridDim.x) {
        const Unit U = unit_of<BATCH>(args, u, BN, WT);
        const int wt = (WT == 2 && U.n0 + 128 >= args.N[U.prob]) ? 1 : WT;
        for (int kb = U.kb_begin; ok && kb < U.kb_end; ++kb, ++i) {
          const int st = i % GT_STAGES, ab = i % GT_NACC;
          if (!(ok = mbar_wait(&in_full[st], (i / GT_STAGES) & 1, err, abort_flag))) break;
          if (i >= GT_NACC &&
              !(ok = mbar_wait(&acc_empty[ab], ((i / GT_NACC) - 1) & 1, err, abort_flag)))
            break;
          fence_after();
          const uint32_t w_base = sbase + L::OFF_IN + st * L::STAGE;
          const uint64_t h0 = sdesc_sw128(w_base + L::W_BYTES, 16, 1024);
          const uint64_t l0 = sdesc_sw128(w_base + L::W_BYTES + L::X_TILE, 16, 1024);
          if constexpr (L::TR) {
            // D[token, feature]: A = token tile (hi, then lo), B = the wt weight tiles, which
            // sit back to back as one operand of 128 wt rows.
            const uint64_t b0 = sdesc_sw128(w_base, 16, 1024);
            const uint32_t id = wt == 2 ? idesc2 : idesc;
            const uint32_t d = tmem + ab * L::ACC_COLS;
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // descriptor address field counts 16-byte units
              mma_e4m3(d, h0 + 2 * k, b0 + 2 * k, id, k > 0);
              if constexpr (!ONE) mma_e4m3(d, l0 + 2 * k, b0 + 2 * k, id, true);
            }
          } else {
            // D[feature, token]: A = the weight tile, B = token tile (hi, then lo).
            const uint64_t a0 = sdesc_sw128(w_base, 16, 1024);
            const uint32_t d = tmem + ab * L::ACC_COLS;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              mma_e4m3(d, a0 + 2 * k, h0 + 2 * k, idesc, k > 0);
              mma_e4m3(d, a0 + 2 * k, l0 + 2 * k, idesc, true);
            }
          }
          mma_commit(&acc_full[ab]);
          mma_commit(&in_empty[st]);
        }
      }
      mma_commit(mma_idle);
      volatile int no_abort = 0;
      mbar_wait(mma_idle, 0, err, &no_abort);
    }
  } else if ((warp - 2) / 4 < L::NGRP) {
    // -------------------------------------------------------------------- epilogue
    constexpr int CW = L::CW, CH = L::CH;
    pdl_wait();  // the token scales and outputs belong to the previous kernels' data
    if (blockIdx.x == 0 && args.adv != nullptr && warp == 2)  // every earlier kernel is done
      for (int j = lane; j < args.adv_n; j += 32) args.adv[j] += args.adv_by;
    const int grp = (warp - 2) / 4, q = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const int half = WT == 2 ? grp : 0;       // weight half (128 features) of this warpgroup
    const int col0 = WT == 2 ? 0 : grp * CW;  // first accumulator column within the half
    int i = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < args.units; u += gridDim.x) {
      const Unit U = unit_of<BATCH>(args, u, BN, WT);
      const int nh = U.n0 + 128 * half;       // first feature of this warpgroup's half
      const bool live = nh < args.N[U.prob];  // a half wholly past N was not multiplied
      const float* scales = args.S[U.prob] + (size_t)U.batch * args.s_step + (size_t)(nh / BLK) * nkb_all;
      // This batch's token scales and output (evaluated where used, so that unbatched
      // instantiations keep reading them from the parameter space).
#define GT_SXP (BATCH ? args.sx + (size_t)U.batch * args.x_row_step : args.sx)
#define GT_YBASE                                                                          \
  (BATCH ? reinterpret_cast<char*>(args.Y[U.prob]) +                                      \
               (size_t)U.batch * args.y_step * (args.y_fp32[U.prob] ? 4 : 2)               \
         : reinterpret_cast<char*>(args.Y[U.prob]))
      // SXB: this thread's token (lane = token) and its block scales, one k block ahead.
      const int mt = U.m0 + 32 * q + lane;
      const int sxoff = (mt < args.M ? mt : -1) * nkb_all;  // < 0: token past M
      float sx_next = 0.f;
      if constexpr (SXB) sx_next = sxoff >= 0 ? ld_dep_f32(GT_SXP + sxoff + U.kb_begin) : 0.f;
      // The unit's first block scale and (token-lane orientation, per-token scales) this
      // thread's token scale are requested now, not when first needed: a unit of a few k
      // blocks would otherwise wait an L2 round trip for each.
      float sc_next = live ? __ldg(scales + U.kb_begin) : 0.f;
      float sxm_pre = 1.f;
      if constexpr (L::TR && !SXB) sxm_pre = mt < args.M ? ld_dep_f32(GT_SXP + mt) : 0.f;
      float acc[CW];
#pragma unroll
      for (int j = 0; j < CW; ++j) acc[j] = 0.f;
      for (int kb = U.kb_begin; kb < U.kb_end; ++kb, ++i) {
        const int ab = i % GT_NACC;
        ok = mbar_wait(&acc_full[ab], (i / GT_NACC) & 1, err, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {  // the warp leaves together (loads are warp-wide)
          ok = false;
          break;
        }
        fence_after();
        float sc = sc_next;
        if (kb + 1 < U.kb_end) sc_next = live ? __ldg(scales + kb + 1) : 0.f;
        if constexpr (SXB) {
          sc *= sx_next;
          sx_next = (sxoff >= 0 && kb + 1 < U.kb_end) ? ld_dep_f32(GT_SXP + sxoff + kb + 1) : 0.f;
        }
        const uint32_t t0 = tmem + lane_off + ab * L::ACC_COLS + half * BN + col0;
#pragma unroll
        for (int c = 0; c < CW; c += CH) {
          uint32_t v[CH];
          if constexpr (CH == 16) {
            tmem_ld32x16(t0 + c, v);
          } else {
#pragma unroll
            for (int cc = 0; cc < CH; cc += 32)
              tmem_ld32(t0 + c + cc, *reinterpret_cast<uint32_t(*)[32]>(v + cc));
          }
          tmem_wait_ld();
          if (c + CH >= CW) {
            fence_before();
            mbar_arrive(&acc_empty[ab]);  // the values are in registers: the MMA may reuse it
          }
#pragma unroll
          for (int j = 0; j < CH; ++j) acc[c + j] = fmaf(sc, __uint_as_float(v[j]), acc[c + j]);
        }
      }
      if (!ok) break;
      if constexpr (L::TR) {
        // Thread = token m; acc[j] = feature nh + col0 + j.  16-byte stores along the row.
        const int m = U.m0 + 32 * q + lane;
        const int nb = nh + col0;
        const int nend = args.N[U.prob];
        if (m < args.M) {
          // Token scale, applied as each vector is formed (SXB: already in the block scales).
          const float sxm = sxm_pre;
          if (args.splits > 1 || args.y_fp32[U.prob]) {
            float* y = args.splits > 1
                           ? args.partial + ((size_t)U.split * args.M + m) * args.ldp +
                                 (U.prob ? args.N[0] : 0) + nb
                           : reinterpret_cast<float*>(GT_YBASE) + (size_t)m * args.ldy[U.prob] + nb;
#pragma unroll
            for (int j = 0; j < CW; j += 4)
              if (nb + j < nend)
                *reinterpret_cast<float4*>(y + j) = make_float4(
                    acc[j] * sxm, acc[j + 1] * sxm, acc[j + 2] * sxm, acc[j + 3] * sxm);
          } else {
            __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(GT_YBASE) +
                               (size_t)m * args.ldy[U.prob] + nb;
            const __nv_bfloat16* res = args.R[U.prob];
#pragma unroll
            for (int j = 0; j < CW; j += 8)
              if (nb + j < nend) {
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = acc[j + e] * sxm;
                if (res) {  // residual: bf16(R + bf16(product))
                  const uint4 r = *reinterpret_cast<const uint4*>(
                      res + (size_t)m * args.ldy[U.prob] + nb + j);
                  const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    o[2 * e] = __bfloat162float(__float2bfloat16_rn(o[2 * e])) +
                               __uint_as_float(rw[e] << 16);
                    o[2 * e + 1] = __bfloat162float(__float2bfloat16_rn(o[2 * e + 1])) +
                                   __uint_as_float(rw[e] & 0xFFFF0000u);
                  }
                }
                uint4 v;
                v.x = pack_bf16x2(o[0], o[1]);
                v.y = pack_bf16x2(o[2], o[3]);
                v.z = pack_bf16x2(o[4], o[5]);
                v.w = pack_bf16x2(o[6], o[7]);
                *reinterpret_cast<uint4*>(y + j) = v;
              }
          }
        }
        continue;
      }
      // Feature-lane orientation.
      // Token scales: lane l holds sx[m0 + l + 32c]; the warp passes them round by shuffles.
      const int m0 = U.m0 + col0;
      float sxr[CW / 32];
#pragma unroll
      for (int c = 0; c < CW / 32; ++c) {
        const int m = m0 + 32 * c + lane;
        sxr[c] = m < args.M ? ld_dep_f32(GT_SXP + m) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < CW; ++j) acc[j] *= __shfl_sync(0xffffffffu, sxr[j >> 5], j & 31);
      const int n = nh + 32 * q + lane;
      if (n < args.N[U.prob]) {
        const int mend = min(CW, args.M - m0);
        const int ldy = args.ldy[U.prob];
        if (args.splits > 1) {
          float* p = args.partial + ((size_t)U.split * args.M + m0) * args.ldp +
                     (U.prob ? args.N[0] : 0) + n;
#pragma unroll
          for (int j = 0; j < CW; ++j)
            if (j < mend) p[(size_t)j * args.ldp] = acc[j];
        } else if (args.y_fp32[U.prob]) {
          float* y = reinterpret_cast<float*>(GT_YBASE) + (size_t)m0 * ldy + n;
#pragma unroll
          for (int j = 0; j < CW; ++j)
            if (j < mend) y[(size_t)j * ldy] = acc[j];
        } else {
          __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(GT_YBASE) + (size_t)m0 * ldy + n;
          const __nv_bfloat16* res = args.R[U.prob];
#pragma unroll
          for (int j = 0; j < CW; ++j)
            if (j < mend) {
              float o = acc[j];
              if (res)  // residual: bf16(R + bf16(product))
                o = __bfloat162float(__float2bfloat16_rn(o)) +
                    __bfloat162float(res[(size_t)(m0 + j) * ldy + n]);
              y[(size_t)j * ldy] = __float2bfloat16_rn(o);
            }
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}
#undef GT_SXP
#undef GT_YBASE

// Y = sum over splits of the fp32 partials, in split order (deterministic), for both
// problems of the GEMM in one launch (partial columns [0, N[0]) and [N[0], N[0] + N[1])).
// Safe under programmatic dependent launch.
struct ReduceArgs {
  const float* part;
  int splits, M, ldp;  // ldp = N[0] + N[1]
  int N0;
  void* Y[2];
  int ldy[2], y_fp32[2];
  const __nv_bfloat16* R[2];
};
__global__ void splitk_reduce_kernel(const __grid_constant__ ReduceArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)a.M * a.ldp) return;
  const int m = (int)(i / a.ldp), c = (int)(i % a.ldp);
  const int pb = c < a.N0 ? 0 : 1, n = pb ? c - a.N0 : c;
  float s = 0.f;
  for (int k = 0; k < a.splits; ++k) s += ld_dep_f32(a.part + ((size_t)k * a.M + m) * a.ldp + c);
  if (a.y_fp32[pb]) {
    reinterpret_cast<float*>(a.Y[pb])[(size_t)m * a.ldy[pb] + n] = s;
  } else {
    if (a.R[pb])  // residual: bf16(R + bf16(product))
      s = __bfloat162float(__float2bfloat16_rn(s)) +
          __bfloat162float(a.R[pb][(size_t)m * a.ldy[pb] + n]);
    reinterpret_cast<__nv_bfloat16*>(a.Y[pb])[(size_t)m * a.ldy[pb] + n] = __float2bfloat16_rn(s);
  }
}

template <int BN, int WT, bool SXB, bool ONE = false, bool BATCH = false>
cudaError_t launch_bn(const CUtensorMap* w, const CUtensorMap& hi, const CUtensorMap& lo,
                      const GemmTcArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  const int grid = a.units < num_sms ? a.units : num_sms;
  return launch_kernel(gemm_f8w_tc_kernel<BN, WT, SXB, ONE, BATCH>, dim3(grid), dim3(GT_THREADS),
                       GemmSmem<BN, WT, ONE>::BYTES, st, pdl, w[0], w[1], hi, lo, a);
}

template <int BN, int WT, bool SXB, bool ONE = false, bool BATCH = false>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gemm_f8w_tc_kernel<BN, WT, SXB, ONE, BATCH>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              GemmSmem<BN, WT, ONE>::BYTES);
}

constexpr size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

bool make_tmap_2d(CUtensorMap* m, bool bf16, const void* base, uint64_t cols, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows);

// Weight tiles per unit for a token count M: 2 (256 features against one token tile) when
// there are more than 128 tokens, the reduction spans at least 8 k blocks, and the rounds of
// units over the SMs, weighted by the wide unit's cost (kWideCost x a narrow unit, for twice
// the work), come out lower; else 1.  Measured wide/narrow unit costs on GB300: 1.3-1.5 for
// K = 1536..8192, 2.0 for K = 512 (too few k blocks to gain).
constexpr double kWideCost = 1.45;
int gemm_weight_tiles(int M, int K, const Proj* p, int np, int num_sms) {
  if (M <= 128 || K < 1024) return 1;
  const long m_tiles = (M + 127) / 128;
  long t1 = 0, t2 = 0;
  for (int i = 0; i < np; ++i) {
    t1 += (p[i].N + 127) / 128;
    t2 += (p[i].N + 255) / 256;
  }
  const long r1 = (t1 * m_tiles + num_sms - 1) / num_sms;
  const long r2 = (t2 * m_tiles + num_sms - 1) / num_sms;
  return kWideCost * (double)r2 < (double)r1 ? 2 : 1;
}

cudaError_t init_gemm_tc_kernels() {
  cudaError_t e = set_smem_attr<32, 1, false>();
  if (e == cudaSuccess) e = set_smem_attr<64, 1, false>();
  if (e == cudaSuccess) e = set_smem_attr<128, 1, false>();
  if (e == cudaSuccess) e = set_smem_attr<128, 2, false>();
  if (e == cudaSuccess) e = set_smem_attr<128, 1, true>();
  if (e == cudaSuccess) e = set_smem_attr<128, 2, true>();
  if (e == cudaSuccess) e = set_smem_attr<128, 1, true, true>();
  if (e == cudaSuccess) e = set_smem_attr<128, 2, true, true>();
  if (e == cudaSuccess) e = set_smem_attr<32, 1, false, false, true>();
  if (e == cudaSuccess) e = set_smem_attr<64, 1, false, false, true>();
  if (e == cudaSuccess) e = set_smem_attr<128, 1, false, false, true>();
  return e;
}

namespace {

// The GEMM proper on e4m3 hi/lo activations [M, K] with per-token (sxb = false) or per-(token,
// k block) (sxb = true) scales; split-K partials in `partial`.
cudaError_t gemm_tc_core(const uint8_t* hi, const uint8_t* lo, const float* sx, bool sxb, int M,
                         int K, const Proj* p, int np, float* partial, int num_sms, int* err,
                         cudaStream_t st, int* adv, int adv_n, int adv_by, bool one, bool pdl) {
  const int bn = gemm_bn(M);
  if (sxb && bn != 128) return cudaErrorInvalidValue;
  if (one && !sxb) return cudaErrorInvalidValue;
  if (one) lo = hi;  // not read; the tensor map only needs a valid address
  cudaError_t e = cudaSuccess;
  GemmTcArgs a{};
  a.M = M;
  a.K = K;
  a.batches = 1;
  a.err = err;
  a.sx = sx;
  a.adv = adv;
  a.adv_n = adv_n;
  a.adv_by = adv_by;
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
      a.R[i] = P.R;
      n_total += P.N;
    }
  }
  if (!make_tmap_2d(&mh, false, hi, (uint64_t)K, (uint64_t)M, (uint64_t)K, 128, bn) ||
      !make_tmap_2d(&ml, false, lo, (uint64_t)K, (uint64_t)M, (uint64_t)K, 128, bn))
    return cudaErrorInvalidValue;
  a.m_tiles = (M + bn - 1) / bn;
  a.splits = gemm_splits(M, n_total, K, num_sms);
  const int wt = gemm_weight_tiles(M, K, p, np, num_sms);
  a.n_tiles0 = (p[0].N + 128 * wt - 1) / (128 * wt);
  a.n_tiles = a.n_tiles0 + (np > 1 ? (p[1].N + 128 * wt - 1) / (128 * wt) : 0);
  a.units = a.n_tiles * a.m_tiles * a.splits;
  a.partial = partial;
  a.ldp = n_total;
  switch (bn) {
    case 32: e = launch_bn<32, 1, false>(mw, mh, ml, a, num_sms, st, pdl); break;
    case 64: e = launch_bn<64, 1, false>(mw, mh, ml, a, num_sms, st, pdl); break;
    default:
      if (one)
        e = wt == 2 ? launch_bn<128, 2, true, true>(mw, mh, ml, a, num_sms, st, pdl)
                    : launch_bn<128, 1, true, true>(mw, mh, ml, a, num_sms, st, pdl);
      else if (sxb)
        e = wt == 2 ? launch_bn<128, 2, true>(mw, mh, ml, a, num_sms, st, pdl)
                    : launch_bn<128, 1, true>(mw, mh, ml, a, num_sms, st, pdl);
      else
        e = wt == 2 ? launch_bn<128, 2, false>(mw, mh, ml, a, num_sms, st, pdl)
                    : launch_bn<128, 1, false>(mw, mh, ml, a, num_sms, st, pdl);
      break;
  }
  if (e != cudaSuccess || a.splits == 1) return e;
  ReduceArgs r{};
  r.part = partial;
  r.splits = a.splits;
  r.M = M;
  r.ldp = n_total;
  r.N0 = p[0].N;
  for (int i = 0; i < np; ++i) {
    r.Y[i] = p[i].Y;
    r.ldy[i] = p[i].ldy;
    r.y_fp32[i] = p[i].y_fp32;
    r.R[i] = p[i].R;
  }
  const size_t cnt = (size_t)M * n_total;
  return launch_kernel(splitk_reduce_kernel, dim3((unsigned)((cnt + 255) / 256)), dim3(256), 0, st,
                       pdl, r);
}

}  // namespace

cudaError_t launch_gemm_tc(const __nv_bfloat16* X, int ldx, int M, int K, const Proj* p, int np,
                           float* scratch, int num_sms, int* err, cudaStream_t st, int* adv,
                           int adv_n, int adv_by, bool pdl) {
  if (!scratch) return cudaErrorInvalidValue;
  uint8_t* base = reinterpret_cast<uint8_t*>(scratch);
  uint8_t* hi = base;
  uint8_t* lo = hi + up256((size_t)M * K);
  float* sx = reinterpret_cast<float*>(lo + up256((size_t)M * K));
  float* partial = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sx) + up256((size_t)M * 4));
  const cudaError_t e =
      launch_kernel(split_e4m3_kernel, dim3(M), dim3(256), 0, st, pdl, X, ldx, K, hi, lo, sx);
  if (e != cudaSuccess) return e;
  return gemm_tc_core(hi, lo, sx, false, M, K, p, np, partial, num_sms, err, st, adv, adv_n,
                      adv_by, false, pdl);
}

bool gemm_takes_split_blocks(int M) { return gemm_bn(M) == 128; }

cudaError_t launch_gemm_tc_split(const uint8_t* hi, const uint8_t* lo, const float* sx,
                                 bool block_scales, int M, int K, const Proj* p, int np,
                                 float* scratch, int num_sms, int* err, cudaStream_t st, int* adv,
                                 int adv_n, int adv_by, bool one_term, bool pdl) {
  if (!scratch || !hi || (!lo && !one_term) || !sx || M <= kGemvMaxM ||
      (block_scales && !gemm_takes_split_blocks(M)) || (one_term && !block_scales))
    return cudaErrorInvalidValue;
  return gemm_tc_core(hi, lo, sx, block_scales, M, K, p, np, scratch, num_sms, err, st, adv,
                      adv_n, adv_by, one_term, pdl);
}

size_t absorb_split_bytes(int B, int K) {
  return 2 * up256((size_t)B * HEADS * K) + up256((size_t)B * HEADS * 4);
}

cudaError_t launch_absorb_tc(const __nv_bfloat16* X, long long sb, int sh, int B, int K,
                             const uint8_t* W, long long w_rows, int w_row_base, int w_row_step,
                             const float* S, int s_step, int N, __nv_bfloat16* Y, int ldy,
                             long long y_step, __nv_bfloat16* rope_out, const float2* rope_tab,
                             int pairing, const int* seq_lens, int limit, void* scratch,
                             int num_sms, int* err, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  if ((K != NOPE && K != KV_LORA) || N % 128 != 0 || !scratch) return cudaErrorInvalidValue;
  uint8_t* hi = reinterpret_cast<uint8_t*>(scratch);
  uint8_t* lo = hi + up256((size_t)B * HEADS * K);
  float* sx = reinterpret_cast<float*>(lo + up256((size_t)B * HEADS * K));
  cudaError_t e = launch_kernel(split_heads_e4m3_kernel, dim3(B, HEADS), dim3(K / 8 < 32 ? 32 : K / 8), 0, st, true,
                                X, B, HEADS, sb, sh, K, hi, lo, sx, rope_out, LAT, rope_tab,
                                pairing, seq_lens, limit);
  if (e != cudaSuccess) return e;
  const int bn = gemm_bn(B);
  CUtensorMap mw[2], mh, ml;
  if (!make_tmap_2d(&mw[0], false, W, (uint64_t)K, (uint64_t)w_rows, (uint64_t)K, 128, 128) ||
      !make_tmap_2d(&mh, false, hi, (uint64_t)K, (uint64_t)B * HEADS, (uint64_t)K, 128, bn) ||
      !make_tmap_2d(&ml, false, lo, (uint64_t)K, (uint64_t)B * HEADS, (uint64_t)K, 128, bn))
    return cudaErrorInvalidValue;
  mw[1] = mw[0];
  GemmTcArgs a{};
  a.M = B;
  a.K = K;
  a.N[0] = N;
  a.S[0] = S;
  a.Y[0] = Y;
  a.ldy[0] = ldy;
  a.y_fp32[0] = 0;
  a.R[0] = nullptr;
  a.sx = sx;
  a.splits = 1;
  a.ldp = N;
  a.err = err;
  a.m_tiles = (B + bn - 1) / bn;
  a.n_tiles0 = a.n_tiles = N / 128;
  a.batches = HEADS;
  a.units = HEADS * a.n_tiles * a.m_tiles;
  a.w_row_base = w_row_base;
  a.w_row_step = w_row_step;
  a.x_row_step = B;
  a.s_step = s_step;
  a.y_step = y_step;
  switch (bn) {
    case 32: return launch_bn<32, 1, false, false, true>(mw, mh, ml, a, num_sms, st, true);
    case 64: return launch_bn<64, 1, false, false, true>(mw, mh, ml, a, num_sms, st, true);
    default: return launch_bn<128, 1, false, false, true>(mw, mh, ml, a, num_sms, st, true);
  }
}

cudaError_t launch_quant_e4m3_groups(const __nv_bfloat16* X, int ldx, int M, int K, uint8_t* q,
                                     float* sx, cudaStream_t st, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (K % BLK != 0 || K > 8192) return cudaErrorInvalidValue;
  return launch_kernel(quant_e4m3_groups_kernel, dim3(M), dim3(K / 8), 0, st, pdl, X, ldx, K, q,
                       sx);
}

}  // namespace mla
