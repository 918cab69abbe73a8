// FP8 block-scaled projections of a few token rows (decode, tiny prefills): a persistent
// weight-streaming GEMV on the CUDA cores, fed by bulk copies.
//
// Y[m, n] = sum_kb S[n/128][kb] * sum_{k in kb} X[m, k] * e4m3(W[n, k])   ("linear" excerpt of
// the "Key-value latent" page: fmt e4m3, weight_block_size [128, 128]; nn.Linear without
// bias).  The raw e4m3 values times the bf16 activations are summed in float32 over each
// lane's run of one 128-wide k block, and that sum is multiplied by the block's scale once, so
// the dequantised weight is never rounded.
//
// With one to three token rows the projection only streams its weight once: the work is
// bandwidth, not arithmetic.  One CTA per SM owns a contiguous run of weight rows (rows of
// the row-major [N, K] weight are contiguous in memory) and streams it through a ring of
// shared-memory slots with cp.async.bulk, so every SM keeps about 100 KB of reads in flight
// from its first cycle to its last, with no waves of CTAs.  Roles:
//   warp NW (producer)  lane 0 issues one bulk copy per slot (RPS whole rows) as soon as the
//                       slot is free; lanes 1..31 start L2 prefetches of weights that later
//                       kernels of the call will read (their DRAM reads then overlap this
//                       kernel and the dependency chain in between);
//   warps 0..NW-1       each owns a fixed k-slice of CH bytes per lane (NW * 32 * CH = K),
//                       so its activations stay in registers (float32) for every row; per
//                       row it forms a scaled partial sum per token, reduces it over the
//                       warp and leaves it in shared memory; every GR rows the warps meet and
//                       each reduces a few rows over the warps and stores Y.
// The weights and the prefetches do not depend on earlier kernels, so they start before the
// programmatic-launch wait; the activations are read after it.
//
// With `norm` set (q_b_proj of a decode step), the activations are the q latent's RMSNorm
// ("rmsnorm" excerpt: x = g * bf16(c * rsqrt(mean(c^2) + eps)), rounded to bf16) computed on
// the fly from the fp32 q_a outputs, and one extra CTA normalises the kv latent, rotates the
// shared rotary key and appends each token's cache row [c_hat | RoPE(k_pe)].
#include "tc_common.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int GS_RING = 96 * 1024;  // bytes of the slot ring per CTA
constexpr int GS_PF_CHUNK = 32 * 1024;

struct L2Prefetch {
  const void* p[3];
  unsigned long long bytes[3];
  int n;
};

// The decode step's kv half of the norm kernel (q_b_proj with the fused norm): per token, the
// kv-latent RMSNorm, RoPE of the shared rotary key at the token's position and the cache row.
struct KvAppend {
  const float* g1;               // [M][2112] fp32 q_a | kv_a outputs
  const __nv_bfloat16* gq;       // q_a_layernorm gain [1536]
  const __nv_bfloat16* gkv;      // kv_a_layernorm gain [512]
  float eps;
  const float2* rope_tab;
  int pairing;
  const int* seq_lens;
  __nv_bfloat16* cache;
  int cap, limit;
};

struct GemvArgs {
  Proj p[2];
  int np, rows0, rows;           // rows of p[0]; rows of both
  const __nv_bfloat16* X;        // [M][ldx] bf16 activations (norm == 0)
  int ldx;
  int norm;                      // 1: X is the q-latent norm of kv.g1 (K = Q_LORA)
  KvAppend kv;
  L2Prefetch pf;
  int* adv;                      // CTA 0 adds adv_by to adv[0..adv_n) (length bookkeeping)
  int adv_n, adv_by;
  int* err;
  int ncta;                      // CTAs streaming rows (the kv-append CTA comes after them)
};

template <int M, int K>
struct GemvCfg {
  static constexpr int CH = K >= 4096 ? 16 : 8;        // bytes of a row per lane
  static constexpr int NW = K / (32 * CH);             // consumer warps
  static constexpr int RPS = K >= 4096 ? 1 : 8192 / K; // rows per slot
  static constexpr int SPB = K >= 4096 ? 4 : 1;        // slots a consumer batch takes
  static constexpr int RB = RPS * SPB;                 // rows per consumer batch
  static constexpr int GR = RB * 8;                    // rows per reduction group
  static constexpr int SLOT = RPS * K;
  static constexpr int NSLOT = (GS_RING / SLOT) / SPB * SPB;
  static constexpr int THREADS = (NW + 1) * 32;
  static constexpr int OFF_BAR = NSLOT * SLOT;
  static constexpr int OFF_RED = OFF_BAR + 2 * NSLOT * 8;
  static constexpr int RED_FLOATS = 2 * NW * GR * M;
  static constexpr int OFF_NSUM = OFF_RED + RED_FLOATS * 4;
  static constexpr int OFF_MISC = OFF_NSUM + NW * M * 4;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(NW * 32 * CH == K, "k slices cover a row");
  static_assert(128 % CH == 0, "a lane's run lies in one 128-wide k block");
  static_assert(SLOT % 16 == 0 && NSLOT >= 2 * SPB, "slot ring");
  static_assert(THREADS <= 1024 && NW <= 32, "block shape");
};

__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* f) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFF), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  const float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Sum over the first 128 threads of the CTA (named barrier 2; red: 4 floats).
__device__ __forceinline__ float sum128(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  named_bar(2, 128);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  named_bar(2, 128);
  return (red[0] + red[1]) + (red[2] + red[3]);
}

// kv-latent norm, rotary key and cache row of every token (threads 0..127 of the kv CTA).
template <int M>
__device__ void kv_append(const KvAppend& a, int* err, float* red, __nv_bfloat16* row) {
  const int tid = threadIdx.x;
  for (int m = 0; m < M; ++m) {
    const float* in = a.g1 + (size_t)m * G1_N + Q_LORA;
    float xk[KV_LORA / 128];
    float sk = 0.f;
#pragma unroll
    for (int i = 0; i < KV_LORA / 128; ++i) {
      xk[i] = in[tid + 128 * i];
      sk += xk[i] * xk[i];
    }
    const float rk = rsqrtf(sum128(sk, red) / KV_LORA + a.eps);
#pragma unroll
    for (int i = 0; i < KV_LORA / 128; ++i) {
      const int c = tid + 128 * i;
      row[c] = __float2bfloat16_rn(__bfloat162float(a.gkv[c]) * bf16r(xk[i] * rk));
    }
    const int pos = a.seq_lens[m];
    const bool bad = pos < 0 || pos >= a.limit;
    if (bad && tid == 0) atomicExch(err, DEV_ERR_RANGE);
    if (!bad && tid < ROPE / 2) {
      const int2 ij = a.pairing == 0 ? make_int2(2 * tid, 2 * tid + 1)
                                     : make_int2(tid, tid + ROPE / 2);
      const float2 cs = a.rope_tab[(size_t)pos * (ROPE / 2) + tid];
      const float x0 = in[KV_LORA + ij.x], x1 = in[KV_LORA + ij.y];
      row[KV_LORA + ij.x] = __float2bfloat16_rn(x0 * cs.x - x1 * cs.y);
      row[KV_LORA + ij.y] = __float2bfloat16_rn(x1 * cs.x + x0 * cs.y);
    }
    named_bar(2, 128);
    if (!bad && tid < LAT / 8)
      reinterpret_cast<uint4*>(a.cache + ((size_t)m * a.cap + pos) * LAT)[tid] =
          reinterpret_cast<const uint4*>(row)[tid];
    named_bar(2, 128);
  }
}

template <int M, int K>
__global__ void __launch_bounds__(GemvCfg<M, K>::THREADS, 1) gemv_stream_kernel(
    const __grid_constant__ GemvArgs args) {
  using C = GemvCfg<M, K>;
  constexpr int CH = C::CH, NW = C::NW, RPS = C::RPS, NSLOT = C::NSLOT;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NSLOT;
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);    // [2][NW][GR][M]
  float* nsum = reinterpret_cast<float*>(smem + C::OFF_NSUM);  // [M][NW]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = args.err;
  pdl_launch_dependents();

  if (blockIdx.x >= args.ncta) {  // the kv-append CTA of the fused q_b launch
    __shared__ float kred[4];
    __shared__ __align__(16) __nv_bfloat16 row[LAT];
    pdl_wait();                   // g1 comes from the previous kernel
    if (threadIdx.x < 128) kv_append<M>(args.kv, err, kred, row);
    return;
  }

  const int c = blockIdx.x;
  const int r0 = (int)((long)args.rows * c / args.ncta);
  const int r1 = (int)((long)args.rows * (c + 1) / args.ncta);
  const int nrows = r1 - r0;
  const int nslots = (nrows + RPS - 1) / RPS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ---------------------------------------------------------------- producer
    // Lane 0 fills the ring first; only then do lanes 1..31 queue the L2 prefetches (this
    // CTA's remaining rows, then later kernels' weights), so the first copies go out first.
    auto issue = [&](int s) {
      const int st = s % NSLOT;
      const int j0 = s * RPS, cnt = min(RPS, nrows - j0);
      mbar_expect_tx(&full[st], (uint32_t)(cnt * K));
      uint8_t* dst = smem + st * C::SLOT;
      // The slot's rows are contiguous in memory except where they cross from p[0] to p[1].
      int g = r0 + j0, left = cnt;
      while (left > 0) {
        const bool second = g >= args.rows0;
        const int n = second ? g - args.rows0 : g;
        const int run = second ? left : min(left, args.rows0 - g);
        const uint8_t* src = args.p[second ? 1 : 0].W + (size_t)n * K;
        bulk_load(dst, src, (uint32_t)(run * K), &full[st]);
        dst += run * K;
        g += run;
        left -= run;
      }
    };
    const int first = min(NSLOT, nslots);
    if (lane == 0)
      for (int s = 0; s < first; ++s) issue(s);
    __syncwarp();
    if (lane == 0) {
      int s = first;
      for (; s < nslots; ++s) {
        if (!mbar_wait(&empty[s % NSLOT], ((s / NSLOT) - 1) & 1, err, abort_flag)) break;
        issue(s);
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the last ones.
      volatile int no_abort = 0;
      for (int u = max(0, s - NSLOT); u < s; ++u)
        mbar_wait(&full[u % NSLOT], (u / NSLOT) & 1, err, &no_abort);
    } else {
      // First the rest of this CTA's own rows: the ring holds too few bytes to cover the DRAM
      // latency under full load, so every row's read starts now and its bulk copy later
      // finds it in L2.
      {
        const int g0 = r0 + first * RPS;
        const int lanes = 31;
        for (int part = 0; part < 2; ++part) {
          const int a = part ? max(g0, args.rows0) : g0;
          const int b = part ? r1 : min(r1, args.rows0);
          if (a >= b) continue;
          const uint8_t* base = args.p[part].W + (size_t)(a - (part ? args.rows0 : 0)) * K;
          const unsigned long long len = (unsigned long long)(b - a) * K;
          for (unsigned long long o = (unsigned long long)(lane - 1) * GS_PF_CHUNK; o < len;
               o += (unsigned long long)lanes * GS_PF_CHUNK)
            prefetch_l2_bulk(base + o, (uint32_t)min((unsigned long long)GS_PF_CHUNK, len - o));
        }
      }
      // Then the L2 prefetch of later kernels' weights: this CTA's share of each region.
      for (int i = 0; i < args.pf.n; ++i) {
        const unsigned long long len = args.pf.bytes[i] & ~15ull;
        const unsigned long long lo = (len * c / args.ncta) & ~15ull;
        const unsigned long long hi = c + 1 == args.ncta ? len : (len * (c + 1) / args.ncta) & ~15ull;
        const uint8_t* base = static_cast<const uint8_t*>(args.pf.p[i]);
        for (unsigned long long o = lo + (unsigned long long)(lane - 1) * GS_PF_CHUNK; o < hi;
             o += 31ull * GS_PF_CHUNK)
          prefetch_l2_bulk(base + o, (uint32_t)min((unsigned long long)GS_PF_CHUNK, hi - o));
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int k0 = (warp * 32 + lane) * CH;  // this lane's run of every row
  pdl_wait();                              // activations (and g1) come from earlier kernels
  if (c == 0 && args.adv != nullptr)       // every earlier kernel of the stream is done
    for (int j = threadIdx.x; j < args.adv_n; j += NW * 32) args.adv[j] += args.adv_by;

  float xr[M][CH];
  if (args.norm) {
    // q-latent RMSNorm of every token over the consumer threads (K = Q_LORA).
    float ss[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float4* src = reinterpret_cast<const float4*>(args.kv.g1 + (size_t)m * G1_N + k0);
#pragma unroll
      for (int i = 0; i < CH / 4; ++i) {
        const float4 v = src[i];
        xr[m][4 * i] = v.x; xr[m][4 * i + 1] = v.y; xr[m][4 * i + 2] = v.z; xr[m][4 * i + 3] = v.w;
      }
      float s2 = 0.f;
#pragma unroll
      for (int i = 0; i < CH; ++i) s2 += xr[m][i] * xr[m][i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
      ss[m] = s2;
    }
    if (lane == 0)
#pragma unroll
      for (int m = 0; m < M; ++m) nsum[m * NW + warp] = ss[m];
    named_bar(1, NW * 32);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float t = 0.f;
      for (int w = 0; w < NW; ++w) t += nsum[m * NW + w];
      const float rs = rsqrtf(t / K + args.kv.eps);
#pragma unroll
      for (int i = 0; i < CH; ++i)
        xr[m][i] = bf16r(__bfloat162float(args.kv.gq[k0 + i]) * bf16r(xr[m][i] * rs));
    }
  } else {
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const uint4* src = reinterpret_cast<const uint4*>(args.X + (size_t)m * args.ldx + k0);
#pragma unroll
      for (int i = 0; i < CH / 8; ++i) {
        const uint4 v = src[i];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xr[m][8 * i + 2 * e] = __uint_as_float(u[e] << 16);
          xr[m][8 * i + 2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
        }
      }
    }
  }

  // Rows go in batches of RB (SPB slots): the RB x M warp reductions are independent
  // shuffle chains, so their latencies overlap.
  constexpr int RB = C::RB, SPB = C::SPB, GR = C::GR;
  int cur_rb = -1, cur_prob = -1;
  float sc = 0.f;
  bool ok = true;
  for (int s0 = 0; s0 < nslots; s0 += SPB) {
#pragma unroll
    for (int q = 0; q < SPB; ++q)
      if (ok && s0 + q < nslots)
        ok = mbar_wait(&full[(s0 + q) % NSLOT], ((s0 + q) / NSLOT) & 1, err, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    const int jb = s0 * RPS;                 // first row of the batch
    const int nb = min(RB, nrows - jb);      // rows in the batch
    float part[RB][M];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int j = jb + r;
#pragma unroll
      for (int m = 0; m < M; ++m) part[r][m] = 0.f;
      if (r < nb) {
        const int g = r0 + j;
        const int prob = g >= args.rows0 ? 1 : 0;
        const int n = prob ? g - args.rows0 : g;
        if (n / BLK != cur_rb || prob != cur_prob) {
          cur_rb = n / BLK;
          cur_prob = prob;
          sc = __ldg(args.p[prob].S + (size_t)cur_rb * (K / BLK) + k0 / BLK);
        }
        // Row j sits in slot (j / RPS) % NSLOT at row j % RPS.
        const uint8_t* wrow = smem + ((j / RPS) % NSLOT) * C::SLOT + (j % RPS) * K + k0;
        float wf[CH];
        if constexpr (CH == 16) {
          const uint4 w = *reinterpret_cast<const uint4*>(wrow);
          e4m3x4_to_f32(w.x, wf);
          e4m3x4_to_f32(w.y, wf + 4);
          e4m3x4_to_f32(w.z, wf + 8);
          e4m3x4_to_f32(w.w, wf + 12);
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(wrow);
          e4m3x4_to_f32(w.x, wf);
          e4m3x4_to_f32(w.y, wf + 4);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float a = 0.f;
#pragma unroll
          for (int i = 0; i < CH; ++i) a = fmaf(wf[i], xr[m][i], a);
          part[r][m] = a * sc;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) part[r][m] += __shfl_xor_sync(0xffffffffu, part[r][m], off);
    if (lane == 0)
#pragma unroll
      for (int r = 0; r < RB; ++r)
        if (r < nb) {
          const int j = jb + r;
#pragma unroll
          for (int m = 0; m < M; ++m)
            red[((((j / GR) & 1) * NW + warp) * GR + j % GR) * M + m] = part[r][m];
        }
    __syncwarp();
    if (lane == 0)
#pragma unroll
      for (int q = 0; q < SPB; ++q)
        if (s0 + q < nslots) mbar_arrive(&empty[(s0 + q) % NSLOT]);
    // End of a group of rows (GR is a multiple of RB), or of the CTA's rows: the warps meet,
    // and each finishes a few rows: the sum over the warps' partials, then the store.
    const int jl = jb + nb - 1;
    if (jl % GR == GR - 1 || jl == nrows - 1) {
      named_bar(1, NW * 32);
      const int gb = (jl / GR) & 1, jg = jl - jl % GR;
      for (int i = warp; i <= jl % GR; i += NW) {
        const int gg = r0 + jg + i;
        const int pp = gg >= args.rows0 ? 1 : 0;
        const int nn = pp ? gg - args.rows0 : gg;
        const Proj& P = args.p[pp];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = lane < NW ? red[((gb * NW + lane) * GR + i) * M + m] : 0.f;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane == 0) {
            if (P.y_fp32)
              reinterpret_cast<float*>(P.Y)[(size_t)m * P.ldy + nn] = v;
            else
              reinterpret_cast<__nv_bfloat16*>(P.Y)[(size_t)m * P.ldy + nn] =
                  __float2bfloat16_rn(v);
          }
        }
      }
    }
  }
}

template <int M, int K>
cudaError_t launch_stream(const GemvArgs& a, cudaStream_t st, bool pdl) {
  using C = GemvCfg<M, K>;
  const int grid = a.ncta + (a.norm ? 1 : 0);
  return launch_kernel(gemv_stream_kernel<M, K>, dim3(grid), dim3(C::THREADS), (size_t)C::BYTES,
                       st, pdl, a);
}

template <int M, int K>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(gemv_stream_kernel<M, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              GemvCfg<M, K>::BYTES);
}

template <int M>
cudaError_t launch_m(const GemvArgs& a, int K, cudaStream_t st, bool pdl) {
  switch (K) {
    case Q_LORA: return launch_stream<M, Q_LORA>(a, st, pdl);
    case HIDDEN: return launch_stream<M, HIDDEN>(a, st, pdl);
    case O_IN: return launch_stream<M, O_IN>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_any(const GemvArgs& a, int M, int K, cudaStream_t st, bool pdl) {
  switch (M) {
    case 1: return launch_m<1>(a, K, st, pdl);
    case 2: return launch_m<2>(a, K, st, pdl);
    case 3: return launch_m<3>(a, K, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

void fill_prefetch(GemvArgs& a, const L2Region* pf, int npf) {
  a.pf.n = 0;
  for (int i = 0; i < npf && i < 3; ++i) {
    if (!pf[i].p || pf[i].bytes < 16) continue;
    a.pf.p[a.pf.n] = pf[i].p;
    a.pf.bytes[a.pf.n] = pf[i].bytes;
    ++a.pf.n;
  }
}

}  // namespace

bool gemv_stream_supports(int M, int K) {
  return M >= 1 && M <= kGemvMaxM && (K == Q_LORA || K == HIDDEN || K == O_IN);
}

cudaError_t init_gemv_stream_kernels() {
  cudaError_t e = cudaSuccess;
  e = e == cudaSuccess ? set_attr<1, Q_LORA>() : e;
  e = e == cudaSuccess ? set_attr<2, Q_LORA>() : e;
  e = e == cudaSuccess ? set_attr<3, Q_LORA>() : e;
  e = e == cudaSuccess ? set_attr<1, HIDDEN>() : e;
  e = e == cudaSuccess ? set_attr<2, HIDDEN>() : e;
  e = e == cudaSuccess ? set_attr<3, HIDDEN>() : e;
  e = e == cudaSuccess ? set_attr<1, O_IN>() : e;
  e = e == cudaSuccess ? set_attr<2, O_IN>() : e;
  e = e == cudaSuccess ? set_attr<3, O_IN>() : e;
  return e;
}

cudaError_t launch_gemv_stream(const __nv_bfloat16* X, int ldx, int M, int K, const Proj* p,
                               int np, int num_sms, int* err, cudaStream_t st, bool pdl,
                               int* adv, int adv_n, int adv_by, const L2Region* pf, int npf) {
  if (!gemv_stream_supports(M, K) || np < 1 || np > 2) return cudaErrorInvalidValue;
  GemvArgs a{};
  a.p[0] = p[0];
  if (np > 1) a.p[1] = p[1];
  a.np = np;
  a.rows0 = p[0].N;
  a.rows = p[0].N + (np > 1 ? p[1].N : 0);
  a.X = X;
  a.ldx = ldx;
  a.norm = 0;
  a.adv = adv;
  a.adv_n = adv_n;
  a.adv_by = adv_by;
  a.err = err;
  a.ncta = num_sms;
  fill_prefetch(a, pf, npf);
  return launch_any(a, M, K, st, pdl);
}

cudaError_t launch_qb_norm_stream(const float* g1, int M, const Proj& p, const __nv_bfloat16* gq,
                                  const __nv_bfloat16* gkv, float eps, const float2* rope_tab,
                                  int rope_pairing, const int* seq_lens, __nv_bfloat16* cache,
                                  int cap, int limit, int num_sms, int* err, cudaStream_t st,
                                  bool pdl, const L2Region* pf, int npf) {
  if (M < 1 || M > kGemvMaxM || p.N != QB_N || p.y_fp32) return cudaErrorInvalidValue;
  GemvArgs a{};
  a.p[0] = p;
  a.np = 1;
  a.rows0 = a.rows = p.N;
  a.norm = 1;
  a.kv = KvAppend{g1, gq, gkv, eps, rope_tab, rope_pairing, seq_lens, cache, cap, limit};
  a.err = err;
  a.ncta = num_sms;
  fill_prefetch(a, pf, npf);
  return launch_any(a, M, Q_LORA, st, pdl);
}

}  // namespace mla
