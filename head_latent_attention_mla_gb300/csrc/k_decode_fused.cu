// One decode step for one or two sequences with short caches, as a single persistent kernel.
//
// The step is a chain of six dependent stages (q_a + kv_a; the q-latent norm and q_b; the W_UK
// absorption; the attention over the latent cache; the split combine and W_UV; o_proj) that
// together read 101 MB of FP8 weights and little else.  As separate kernels each stage waits
// for the previous one to finish before its reads start, and HBM idles in between.  Here one
// CTA per SM runs all six stages, separated by grid-wide barriers (the launch is cooperative,
// so every CTA is resident), and each CTA knows at its start which weights its later stages
// read: it queues them at once, the q_b rows as a bulk copy into its shared memory, the W_UK,
// W_UV and o_proj rows as L2 prefetches, so the whole step's weights stream from HBM while
// the first stages run.
//
// Stages (G CTAs, 16 warps each; rows of a projection split evenly over the CTAs):
//   1  q_a_proj and kv_a_proj_with_mqa -> g1 [M, 2112] fp32
//   2  q-latent RMSNorm (every CTA, from g1) and q_b_proj -> q [M, 12288] bf16; CTA G-1 also
//      the kv-latent RMSNorm, RoPE of the shared rotary key and the cache row append
//   3  W_UK absorption and RoPE of q_pe -> qfull [M, 64, 576] bf16
//   4  attention over the latent cache on the CUDA cores: unit (sequence, 8 heads, position
//      chunk) with an online softmax over 64-position sub-tiles -> fp32 partials (O, m, l)
//   5  combine of the partials (per head) and W_UV -> attn [M, 8192] bf16
//   6  o_proj -> out [M, 7168] bf16; CTA 0 advances the lengths
// The projections (stages 1, 2, 6) give each warp a fixed 512-wide k-slice of the input held in
// registers; a warp forms per-row partial sums over its slice (raw e4m3 times the activation,
// one weight block scale per lane's 16-value run) and the CTA adds the slices' partials.
// Arithmetic follows the per-stage kernels of the decode chain: fp32 sums, bf16 outputs where
// those kernels round, and the attention's softmax in base 2 with fp32 weights.
#include "tc_common.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int FD_THREADS = 512;
constexpr int FD_WARPS = FD_THREADS / 32;
constexpr int FD_QB_ROWS = 96;          // q_b rows a CTA holds: needs at least 128 CTAs
constexpr int FD_HG = 8;                // heads of one attention unit
constexpr int FD_TP = 64;               // positions of one attention sub-tile
constexpr int FD_RED = 56 * 16 * 2;     // floats of the k-slice partials (rows x slices x M)
// Region B (floats): the partials, then 1/rms per token, per-warp sums, an abort flag and the kv
// cache row being built (576 bf16).
constexpr int B_RS = FD_RED, B_WS = FD_RED + 4, B_FLAG = FD_RED + 40, B_ROW = FD_RED + 48;
constexpr int OFF_A = 0;                                   // q_b rows; later stage 4's tiles
constexpr int A_BYTES = FD_QB_ROWS * Q_LORA;               // 147,456
constexpr int OFF_B = OFF_A + A_BYTES;                     // partials and small arrays
constexpr int B_BYTES = 16 * 1024;
constexpr int OFF_BAR = OFF_B + B_BYTES;
constexpr int FD_SMEM = OFF_BAR + 64;
static_assert(FD_HG * LAT * 4 + FD_TP * LAT * 2 + FD_HG * FD_TP * 4 + 256 <= A_BYTES,
              "stage 4 tiles fit the q_b region");
static_assert((B_ROW + LAT / 2) * 4 <= B_BYTES, "region B");

struct FusedArgs {
  const uint8_t* W[5];          // q_a, q_b, kv_a, kv_b, o (e4m3, [out, in])
  const float* S[5];            // their block scales
  const __nv_bfloat16* gq;      // q_a_layernorm gain
  const __nv_bfloat16* gkv;     // kv_a_layernorm gain
  float eps;
  const float2* rope_tab;
  int pairing;
  const __nv_bfloat16* x;       // [M, 7168]
  CacheRef cache;
  int limit;                    // positions allowed (cache and RoPE table)
  int* seq_lens;                // [M], advanced by 1 at the end
  float scale_log2;             // softmax scale * log2(e)
  float* g1;                    // [M, 2112]
  __nv_bfloat16* q;             // [M, 12288]
  __nv_bfloat16* qfull;         // [M, 64, 576]
  float* opart;                 // [M, npc, 64, 512]
  float* ml;                    // [M, npc, 64, 2]
  __nv_bfloat16* attn;          // [M, 8192]
  __nv_bfloat16* out;           // [M, 7168]
  unsigned* bar;                // grid barrier: count, generation (0, any at rest)
  int* err;
  int npc;                      // position chunks per (sequence, head group)
};

__device__ __forceinline__ float bf16r(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* f) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFF), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  const float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
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

__device__ __forceinline__ uint4 ld_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Loads of data this kernel wrote earlier (in another CTA, before a grid barrier) go through
// L2 (ld.global.cg), never the read-only path.
__device__ __forceinline__ uint4 ld_cg(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// All CTAs of the cooperative launch meet.  The last to arrive resets the count and advances
// the generation; the others wait (bounded) for the generation to change.  Writes before the
// barrier are visible to every CTA after it.  Returns false after a timeout (recorded in err).
__device__ bool grid_sync(unsigned* bar, int* err) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned* gen = bar + 1;
    const unsigned g0 = *gen;
    __threadfence();
    int ok = 1;
    if (atomicAdd(bar, 1u) == gridDim.x - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const unsigned long long t0 = global_ns();
      while (*gen == g0) {
        if (global_ns() - t0 > kWaitLimitNs) {
          atomicExch(err, DEV_ERR_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Rows [r0, r1) of Y = X W^T for M token rows, K = 512 * KS, split into KS k-slices of 512: warp
// w works on slice w % KS for the rows r0 + (w / KS), r0 + (w / KS) + NG, ... (NG = 16 / KS
// warp groups), with its lane's 16 activation values of each token in xr.  row_ptr(r) gives a
// row's weights (in shared memory when SMEM, else global), scale(r, kb) its block scale.  The slices' partials
// meet in red [(r1 - r0) x KS x M] and emit(r, m, v) receives each output.
template <int M, int KS, bool SMEM, class RowPtr, class Scale, class Emit>
__device__ void gemv_rows(int r0, int r1, const float (&xr)[M][16], RowPtr row_ptr, Scale scale,
                          Emit emit, float* red) {
  constexpr int NG = FD_WARPS / KS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = warp % KS, grp = warp / KS;
  const int k0 = slice * 512 + lane * 16;
  constexpr int RB = 8;  // rows in flight per warp
  if (grp < NG) {
    for (int rb = r0 + grp; rb < r1; rb += NG * RB) {
      uint4 w[RB];
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        const int r = rb + j * NG;
        if (r >= r1)
          w[j] = make_uint4(0, 0, 0, 0);
        else if constexpr (SMEM)
          w[j] = *reinterpret_cast<const uint4*>(row_ptr(r) + k0);
        else
          w[j] = ld_nc(row_ptr(r) + k0);
      }
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        const int r = rb + j * NG;
        float wf[16];
        e4m3x4_to_f32(w[j].x, wf);
        e4m3x4_to_f32(w[j].y, wf + 4);
        e4m3x4_to_f32(w[j].z, wf + 8);
        e4m3x4_to_f32(w[j].w, wf + 12);
        const float sc = r < r1 ? scale(r, k0 / BLK) : 0.f;
        float p[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float a = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) a = fmaf(wf[i], xr[m][i], a);
          p[m] = a * sc;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
          for (int m = 0; m < M; ++m) p[m] += __shfl_xor_sync(0xffffffffu, p[m], off);
        if (lane == 0 && r < r1)
#pragma unroll
          for (int m = 0; m < M; ++m) red[((r - r0) * KS + slice) * M + m] = p[m];
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < (r1 - r0) * M; e += FD_THREADS) {
    const int r = e / M, m = e % M;
    float v = 0.f;
#pragma unroll
    for (int s = 0; s < KS; ++s) v += red[(r * KS + s) * M + m];
    emit(r0 + r, m, v);
  }
  __syncthreads();
}

// This lane's 16 bf16 activations of each token at column k0 as floats.
// (CG: the values were written earlier in this kernel.)
template <int M, bool CG>
__device__ __forceinline__ void load_x16(const __nv_bfloat16* x, int ld, int k0, float (&xr)[M][16]) {
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const __nv_bfloat16* p = x + (size_t)m * ld + k0;
    bf16x8_to_f32(CG ? ld_cg(p) : ld_nc(p), xr[m]);
    bf16x8_to_f32(CG ? ld_cg(p + 8) : ld_nc(p + 8), xr[m] + 8);
  }
}

template <int M>
__global__ void __launch_bounds__(FD_THREADS, 1) decode_fused_kernel(const __grid_constant__ FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sA = smem + OFF_A;
  float* sB = reinterpret_cast<float*>(smem + OFF_B);
  uint64_t* qb_bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  int* err = a.err;

  // Row ranges of this CTA in the three projections and its units in stages 3 and 5.
  const int r1a = G1_N * c / G, r1b = G1_N * (c + 1) / G;
  const int r2a = QB_N * c / G, r2b = QB_N * (c + 1) / G;
  const int r6a = HIDDEN * c / G, r6b = HIDDEN * (c + 1) / G;
  const int u3a = HEADS * 4 * c / G, u3b = HEADS * 4 * (c + 1) / G;
  const int n5 = M * HEADS * 4;
  const int u5a = n5 * c / G, u5b = n5 * (c + 1) / G;

  // ---- queue the later stages' weights ----------------------------------------------------
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sB + B_FLAG);
  if (tid == 0) {
    mbar_init(qb_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Leaving early (a barrier gave up): first wait (bounded) for this CTA's bulk copy, so that no
  // copy into its shared memory is in flight when it exits.
  bool qb_done = false;
  auto drain = [&]() {
    if (tid == 0 && !qb_done) {
      volatile int no_abort = 0;
      mbar_wait(qb_bar, 0, err, &no_abort);
    }
    __syncthreads();
  };
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)((r2b - r2a) * Q_LORA);
    mbar_expect_tx(qb_bar, bytes);
    const uint8_t* src = a.W[MLA_W_Q_B] + (size_t)r2a * Q_LORA;
    for (uint32_t o = 0; o < bytes; o += 32768u)
      bulk_load(sA + o, src + o, bytes - o < 32768u ? bytes - o : 32768u, qb_bar);
  } else if (warp == 1) {
    // W_UK of this CTA's stage-3 heads (rows 256h .. 256h+127 of kv_b, 64 KB each) and W_UV of
    // its stage-5 units (32 rows, 16 KB each).  (The o_proj rows follow after stage 1, whose
    // own reads would otherwise queue behind them.)
    const uint8_t* kvb = a.W[MLA_W_KV_B];
    for (int u = u3a + lane; u < u3b; u += 32)
      if (u == u3a || u % 4 == 0) prefetch_l2_bulk(kvb + (size_t)(u / 4) * KVB_PER_HEAD * KV_LORA, 65536u);
    for (int u = u5a + lane; u < u5b; u += 32) {
      const int h = (u / 4) % HEADS, vb = u % 4;
      prefetch_l2_bulk(kvb + ((size_t)h * KVB_PER_HEAD + NOPE + 32 * vb) * KV_LORA, 16384u);
    }
  }

  // ---- stage 1: q_a_proj | kv_a_proj_with_mqa -> g1 -------------------------------------------
  {
    float xr[M][16];
    if (warp < HIDDEN / 512) load_x16<M, false>(a.x, HIDDEN, warp * 512 + lane * 16, xr);
    auto rowp = [&](int r) -> const uint8_t* {
      return r < Q_LORA ? a.W[MLA_W_Q_A] + (size_t)r * HIDDEN
                        : a.W[MLA_W_KV_A] + (size_t)(r - Q_LORA) * HIDDEN;
    };
    auto scale = [&](int r, int kb) -> float {
      return r < Q_LORA ? __ldg(a.S[MLA_W_Q_A] + (size_t)(r / BLK) * (HIDDEN / BLK) + kb)
                        : __ldg(a.S[MLA_W_KV_A] + (size_t)((r - Q_LORA) / BLK) * (HIDDEN / BLK) + kb);
    };
    auto emit = [&](int r, int m, float v) { a.g1[(size_t)m * G1_N + r] = v; };
    gemv_rows<M, HIDDEN / 512, false>(r1a, r1b, xr, rowp, scale, emit, sB);
  }
  if (!grid_sync(a.bar, err)) {
    drain();
    return;
  }

  // ---- stage 2: q-latent norm, q_b_proj; kv-latent norm, RoPE(k_pe), cache row --------------
  if (warp == 1) {  // this CTA's o_proj rows, into L2 while stages 2-5 run
    const uint8_t* wo = a.W[MLA_W_O] + (size_t)r6a * O_IN;
    const size_t ob = (size_t)(r6b - r6a) * O_IN;
    for (size_t o = (size_t)lane * 65536u; o < ob; o += 32 * 65536u)
      prefetch_l2_bulk(wo + o, (uint32_t)(ob - o < 65536u ? ob - o : 65536u));
  }
  {
    float* rs = sB + B_RS;  // [M] 1 / rms of the q latent
    {
      float ss[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float v = 0.f;
        for (int i = tid; i < Q_LORA; i += FD_THREADS) {
          const float t = __ldcg(a.g1 + (size_t)m * G1_N + i);
          v += t * t;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        ss[m] = v;
      }
      if (lane == 0)
#pragma unroll
        for (int m = 0; m < M; ++m) sB[B_WS + m * FD_WARPS + warp] = ss[m];
      __syncthreads();
      if (tid < M) {
        float t = 0.f;
        for (int w = 0; w < FD_WARPS; ++w) t += sB[B_WS + tid * FD_WARPS + w];
        rs[tid] = rsqrtf(t / Q_LORA + a.eps);
      }
      __syncthreads();
    }
    float xr[M][16];
    const int k0 = (warp % (Q_LORA / 512)) * 512 + lane * 16;
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        xr[m][i] = bf16r(__bfloat162float(a.gq[k0 + i]) *
                         bf16r(__ldcg(a.g1 + (size_t)m * G1_N + k0 + i) * rs[m]));
    const bool got = mbar_wait(qb_bar, 0, err, abort_flag);
    qb_done = got;
    if (!__syncthreads_and(got)) {
      drain();
      return;
    }
    auto rowp = [&](int r) -> const uint8_t* { return sA + (size_t)(r - r2a) * Q_LORA; };
    auto scale = [&](int r, int kb) -> float {
      return __ldg(a.S[MLA_W_Q_B] + (size_t)(r / BLK) * (Q_LORA / BLK) + kb);
    };
    auto emit = [&](int r, int m, float v) { a.q[(size_t)m * QB_N + r] = __float2bfloat16_rn(v); };
    if (c == G - 1) {
      // kv latent of every token: RMSNorm, RoPE of the shared rotary key at its position, and
      // the cache row (the norm kernel's arithmetic).
      __nv_bfloat16* row = reinterpret_cast<__nv_bfloat16*>(sB + B_ROW);
      for (int m = 0; m < M; ++m) {
        const float* in = a.g1 + (size_t)m * G1_N + Q_LORA;
        float v = tid < KV_LORA ? __ldcg(in + tid) : 0.f;
        float sq = v * v;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
        if (lane == 0) sB[B_WS + warp] = sq;
        __syncthreads();
        float t = 0.f;
        for (int w = 0; w < FD_WARPS; ++w) t += sB[B_WS + w];
        const float rk = rsqrtf(t / KV_LORA + a.eps);
        if (tid < KV_LORA) row[tid] = __float2bfloat16_rn(__bfloat162float(a.gkv[tid]) * bf16r(v * rk));
        const int pos = a.seq_lens[m];
        const long long crow = (pos < 0 || pos >= a.limit) ? -1 : a.cache.row(m, pos);
        if (crow < 0 && tid == 0) atomicExch(err, DEV_ERR_RANGE);
        if (crow >= 0 && tid < ROPE / 2) {
          const int2 ij = a.pairing == 0 ? make_int2(2 * tid, 2 * tid + 1) : make_int2(tid, tid + ROPE / 2);
          const float2 cs = a.rope_tab[(size_t)pos * (ROPE / 2) + tid];
          const float x0 = __ldcg(in + KV_LORA + ij.x), x1 = __ldcg(in + KV_LORA + ij.y);
          row[KV_LORA + ij.x] = __float2bfloat16_rn(x0 * cs.x - x1 * cs.y);
          row[KV_LORA + ij.y] = __float2bfloat16_rn(x1 * cs.x + x0 * cs.y);
        }
        __syncthreads();
        if (crow >= 0 && tid < LAT / 8)
          reinterpret_cast<uint4*>(a.cache.base + (size_t)crow * LAT)[tid] =
              reinterpret_cast<const uint4*>(row)[tid];
        __syncthreads();
      }
    }
    gemv_rows<M, Q_LORA / 512, true>(r2a, r2b, xr, rowp, scale, emit, sB);
  }
  if (!grid_sync(a.bar, err)) return;  // the bulk copy has completed

  // ---- stage 3: W_UK absorption and RoPE(q_pe) -> qfull ----------------------------------------
  for (int u = u3a; u < u3b; ++u) {
    const int h = u / 4, cb = u % 4;
    float* qn = sB;                    // [M][128] q_nope of head h
    float* part = sB + M * NOPE;       // [16][128] partial sums of each 8-row group
    for (int e = tid; e < M * NOPE; e += FD_THREADS)
      qn[e] = __bfloat162float(__ldcg(a.q + (size_t)(e / NOPE) * QB_N + h * QHEAD + e % NOPE));
    __syncthreads();
    const int cg = tid % 32, ig = tid / 32;  // 4 columns, 8 rows
    float w[8][4];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(
          a.W[MLA_W_KV_B] + (size_t)(h * KVB_PER_HEAD + ig * 8 + r) * KV_LORA + cb * BLK + cg * 4));
      e4m3x4_to_f32(v, w[r]);
    }
    const float sc = __ldg(a.S[MLA_W_KV_B] + (size_t)(2 * h) * (KV_LORA / BLK) + cb);
    for (int m = 0; m < M; ++m) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float qv = qn[m * NOPE + ig * 8 + r];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = fmaf(qv, w[r][j], acc[j]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) part[ig * 128 + cg * 4 + j] = acc[j];
      __syncthreads();
      if (tid < 128) {
        float v = 0.f;
#pragma unroll
        for (int g = 0; g < 16; ++g) v += part[g * 128 + tid];
        a.qfull[((size_t)m * HEADS + h) * LAT + cb * BLK + tid] = __float2bfloat16_rn(sc * v);
      }
      __syncthreads();
    }
    if (cb == 0 && tid < M * (ROPE / 2)) {  // RoPE of this head's q_pe at each token's position
      const int m = tid / (ROPE / 2), j = tid % (ROPE / 2);
      const int pos = a.seq_lens[m];
      if (pos >= 0 && pos < a.limit) {
        const int2 ij = a.pairing == 0 ? make_int2(2 * j, 2 * j + 1) : make_int2(j, j + ROPE / 2);
        const __nv_bfloat16* qp = a.q + (size_t)m * QB_N + h * QHEAD + NOPE;
        const float x0 = __bfloat162float(__ldcg(qp + ij.x)), x1 = __bfloat162float(__ldcg(qp + ij.y));
        const float2 cs = a.rope_tab[(size_t)pos * (ROPE / 2) + j];
        __nv_bfloat16* dst = a.qfull + ((size_t)m * HEADS + h) * LAT + KV_LORA;
        dst[ij.x] = __float2bfloat16_rn(x0 * cs.x - x1 * cs.y);
        dst[ij.y] = __float2bfloat16_rn(x1 * cs.x + x0 * cs.y);
      }
    }
    __syncthreads();
  }
  if (!grid_sync(a.bar, err)) return;

  // ---- stage 4: attention of 8 heads over a chunk of positions --------------------------------
  {
    const int units = M * (HEADS / FD_HG) * a.npc;
    for (int u = c; u < units; u += G) {
      const int m = u / ((HEADS / FD_HG) * a.npc);
      const int hg = (u / a.npc) % (HEADS / FD_HG), pc = u % a.npc;
      float* q8 = reinterpret_cast<float*>(sA);                        // [8][576]
      __nv_bfloat16* ct = reinterpret_cast<__nv_bfloat16*>(sA + FD_HG * LAT * 4);  // [64][576]
      float* sp = reinterpret_cast<float*>(sA + FD_HG * LAT * 4 + FD_TP * LAT * 2);  // [8][64]
      float* alpha = sp + FD_HG * FD_TP;                               // [8]
      const int S = a.seq_lens[m] + 1;
      const int cs = (S + a.npc - 1) / a.npc;
      const int p0 = pc * cs, p1 = min(S, p0 + cs);
      for (int e = tid; e < FD_HG * LAT; e += FD_THREADS)
        q8[e] = __bfloat162float(__ldcg(a.qfull + ((size_t)m * HEADS + hg * FD_HG) * LAT + e));
      // This thread's 8 dims of O for head th (64 threads per head).
      const int th = tid / 64, d0 = (tid % 64) * 8;
      float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float mrun = -INFINITY, lrun = 0.f;  // (valid in the lane that owns head th's stats)
      for (int t0 = p0; t0 < p1; t0 += FD_TP) {
        const int nt = min(FD_TP, p1 - t0);
        __syncthreads();  // the previous sub-tile's rows and weights are consumed
        for (int e = tid; e < FD_TP * (LAT / 8); e += FD_THREADS) {
          const int j = e / (LAT / 8), ch = e % (LAT / 8);
          uint4 v = make_uint4(0, 0, 0, 0);
          if (j < nt) {
            const long long crow = a.cache.row(m, t0 + j);
            if (crow >= 0) v = ld_cg(a.cache.base + (size_t)crow * LAT + ch * 8);
            else if (ch == 0) atomicExch(err, DEV_ERR_RANGE);
          }
          reinterpret_cast<uint4*>(ct)[e] = v;
        }
        __syncthreads();
        // Scores: warp w takes pairs (head, position) w, w + 16, ...; lanes split the 576 dims.
        for (int pr = warp; pr < FD_HG * FD_TP; pr += FD_WARPS) {
          const int hh = pr / FD_TP, j = pr % FD_TP;
          float s = 0.f;
          if (j < nt) {
            const __nv_bfloat16* cr = ct + j * LAT;
            for (int d = lane * 2; d < LAT; d += 64) {
              const __nv_bfloat162 cv = *reinterpret_cast<const __nv_bfloat162*>(cr + d);
              s = fmaf(q8[hh * LAT + d], __low2float(cv), s);
              s = fmaf(q8[hh * LAT + d + 1], __high2float(cv), s);
            }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
          if (lane == 0) sp[hh * FD_TP + j] = j < nt ? s * a.scale_log2 : -INFINITY;
        }
        __syncthreads();
        // Online softmax: warp hh < 8 owns head hh's statistics, lane j positions j and j + 32.
        static_assert(FD_TP == 64, "two positions per lane");
        if (warp < FD_HG) {
          const float s0 = sp[warp * FD_TP + lane], s1 = sp[warp * FD_TP + lane + 32];
          float mx = fmaxf(s0, s1);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          const float mnew = fmaxf(mrun, mx);
          const float p0 = lane < nt ? exp2f(s0 - mnew) : 0.f;
          const float p1 = lane + 32 < nt ? exp2f(s1 - mnew) : 0.f;
          float ps = p0 + p1;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
          const float al = mrun == -INFINITY ? 0.f : exp2f(mrun - mnew);
          lrun = lrun * al + ps;
          mrun = mnew;
          sp[warp * FD_TP + lane] = p0;
          sp[warp * FD_TP + lane + 32] = p1;
          if (lane == 0) alpha[warp] = al;
        }
        __syncthreads();
        const float al = alpha[th];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] *= al;
        for (int j = 0; j < nt; ++j) {
          const float p = sp[th * FD_TP + j];
          const uint4 cv = *reinterpret_cast<const uint4*>(ct + j * LAT + d0);
          float cf[8];
          bf16x8_to_f32(cv, cf);
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = fmaf(p, cf[i], o[i]);
        }
      }
      // Partial of unit (m, pc) for heads hg*8 .. hg*8+7: O (relative to m), m and l.
      const size_t slot = (size_t)m * a.npc + pc;
      float* op = a.opart + ((slot * HEADS + hg * FD_HG + th) * KV_LORA + d0);
      *reinterpret_cast<float4*>(op) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(op + 4) = make_float4(o[4], o[5], o[6], o[7]);
      if (warp < FD_HG && lane == 0) {
        a.ml[(slot * HEADS + hg * FD_HG + warp) * 2] = mrun;
        a.ml[(slot * HEADS + hg * FD_HG + warp) * 2 + 1] = lrun;
      }
      __syncthreads();
    }
  }
  if (!grid_sync(a.bar, err)) return;

  // ---- stage 5: combine and W_UV -> attn -------------------------------------------------------
  for (int u = u5a; u < u5b; ++u) {
    const int m = u / (HEADS * 4), h = (u / 4) % HEADS, vb = u % 4;
    float* ol = sB;                     // [512] o_lat of head h (bf16 values)
    float* wts = sB + KV_LORA;          // [npc] chunk weights
    if (tid < 32) {
      float mx = -INFINITY;
      for (int pc = lane; pc < a.npc; pc += 32)
        mx = fmaxf(mx, __ldcg(a.ml + (((size_t)m * a.npc + pc) * HEADS + h) * 2));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      float L = 0.f;
      for (int pc = lane; pc < a.npc; pc += 32) {
        const float* v = a.ml + (((size_t)m * a.npc + pc) * HEADS + h) * 2;
        const float m0 = __ldcg(v), l0 = __ldcg(v + 1);
        const float wgt = m0 == -INFINITY ? 0.f : exp2f(m0 - mx);
        wts[pc] = wgt;
        L += wgt * l0;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
      if (lane == 0) wts[a.npc] = 1.f / L;
    }
    __syncthreads();
    {
      const int d = tid;  // 512 threads, one latent dim each
      float v = 0.f;
      for (int pc = 0; pc < a.npc; ++pc)
        v = fmaf(wts[pc], __ldcg(a.opart + (((size_t)m * a.npc + pc) * HEADS + h) * KV_LORA + d), v);
      ol[d] = bf16r(v * wts[a.npc]);
    }
    __syncthreads();
    // Rows 32 vb .. 32 vb + 31 of W_UV,h: two per warp, lanes over 16-value runs of c.
    for (int r = warp; r < 32; r += FD_WARPS) {
      const int row = 32 * vb + r;
      const uint4 wv = ld_nc(a.W[MLA_W_KV_B] + ((size_t)h * KVB_PER_HEAD + NOPE + row) * KV_LORA + lane * 16);
      float wf[16];
      e4m3x4_to_f32(wv.x, wf);
      e4m3x4_to_f32(wv.y, wf + 4);
      e4m3x4_to_f32(wv.z, wf + 8);
      e4m3x4_to_f32(wv.w, wf + 12);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) s = fmaf(wf[i], ol[lane * 16 + i], s);
      s *= __ldg(a.S[MLA_W_KV_B] + (size_t)(2 * h + 1) * (KV_LORA / BLK) + lane / 8);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane == 0) a.attn[(size_t)m * O_IN + h * VDIM + row] = __float2bfloat16_rn(s);
    }
    __syncthreads();
  }
  if (!grid_sync(a.bar, err)) return;

  // ---- stage 6: o_proj -> out; the lengths advance -------------------------------------------
  {
    float xr[M][16];
    load_x16<M, true>(a.attn, O_IN, warp * 512 + lane * 16, xr);
    auto rowp = [&](int r) -> const uint8_t* { return a.W[MLA_W_O] + (size_t)r * O_IN; };
    auto scale = [&](int r, int kb) -> float {
      return __ldg(a.S[MLA_W_O] + (size_t)(r / BLK) * (O_IN / BLK) + kb);
    };
    auto emit = [&](int r, int m, float v) { a.out[(size_t)m * HIDDEN + r] = __float2bfloat16_rn(v); };
    gemv_rows<M, O_IN / 512, false>(r6a, r6b, xr, rowp, scale, emit, sB);
  }
  if (c == 0 && tid < M) a.seq_lens[tid] += 1;  // every reader of the lengths is done
}

template <int M>
cudaError_t launch_m(const FusedArgs& a, int G, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(FD_THREADS);
  cfg.dynamicSmemBytes = FD_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_fused_kernel<M>, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool decode_fused_supports(int B, int max_len, int num_sms) {
  return B >= 1 && B <= 2 && max_len + 1 <= kFusedMaxPositions && num_sms >= 128 &&
         num_sms * FD_QB_ROWS >= QB_N;
}

int decode_fused_chunks(int B, int num_sms) { return num_sms / (B * (HEADS / FD_HG)); }

cudaError_t init_decode_fused_kernel() {
  cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, FD_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_fused_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             FD_SMEM);
  return e;
}

cudaError_t launch_decode_fused(const FusedDecode& d, cudaStream_t st) {
  if (!decode_fused_supports(d.B, 0, d.num_sms)) return cudaErrorInvalidValue;
  FusedArgs a{};
  for (int i = 0; i < 5; ++i) {
    a.W[i] = d.W[i];
    a.S[i] = d.S[i];
  }
  a.gq = d.gq;
  a.gkv = d.gkv;
  a.eps = d.eps;
  a.rope_tab = d.rope_tab;
  a.pairing = d.pairing;
  a.x = d.x;
  a.cache = d.cache;
  a.limit = d.limit;
  a.seq_lens = d.seq_lens;
  a.scale_log2 = d.scale * 1.4426950408889634f;
  a.g1 = d.g1;
  a.q = d.q;
  a.qfull = d.qfull;
  a.opart = d.opart;
  a.ml = d.ml;
  a.attn = d.attn;
  a.out = d.out;
  a.bar = d.bar;
  a.err = d.err;
  a.npc = decode_fused_chunks(d.B, d.num_sms);
  return d.B == 1 ? launch_m<1>(a, d.num_sms, st) : launch_m<2>(a, d.num_sms, st);
}

}  // namespace mla
