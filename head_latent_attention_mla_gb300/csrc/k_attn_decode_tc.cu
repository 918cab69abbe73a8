// Split-KV decode attention over the latent cache on the tcgen05 tensor cores.
//
// Absorbed form of the `mla-prefill` scores ("Key content up-projection" page): with
// q~_h = [W_UK,h^T q_nope,h | RoPE(q_pe,h)] (576 wide) and the cached row
// c_j = [c_hat_j | RoPE(k_pe)_j], the score of head h and position j is q~_h . c_j times the
// softmax scale, and the latent output is o_lat,h = sum_j p_h(j) c_hat_j.  Each 64-position
// latent tile is read from HBM once and serves as both key and value.
//
// Work split: the positions of all sequences, concatenated, are cut into G equal shares, one
// per CTA (G = the SM count, fewer for short caches), so ragged batches stay balanced.  A share
// can span several sequences; each piece ("segment") is attended with its own query block and
// softmax state, and leaves one partial output in slot b + c (b the sequence, c the CTA: along
// the staircase of (b, c) pairs this sum never repeats).  A combine kernel merges the slots.
//
// 7 warps per CTA:
//   warp 0      TMA producer: the query block once, then 64-position cache tiles into a
//               two-stage ring (9 boxes of 64 rows x 64 columns, 128-byte swizzle);
//   warp 1      allocates tensor memory and issues, from one thread,
//                 MMA1  S[64 heads, 64 pos]   = Q[64, 576] . C[64, 576]^T    (M=64,  N=64);
//   warp 6      issues, from one thread,
//                 MMA2  O^T[512, 64 heads]   += C[64 pos, 0:512]^T . P^T     (M=128, N=64, x4).
//               Two issuers keep MMA2 of a tile from queueing behind the next tile's load;
//   warps 2..5  softmax: one head per thread (rows of S), online softmax in base 2 with a
//               lazy rescale of O^T (only when a head's running maximum grows by more than
//               2^8), P written as bf16 into the tile's rotary box (box 8), which MMA1 no
//               longer needs; then the epilogue writes the unnormalised partial O, the
//               maximum m and the sum l of every head.
// Tensor memory: O^T in columns [0, 256) (lane = latent dim, column = head within each of the
// four 128-dim blocks), S in [256, 320) and [320, 384) (double buffer).
#include "tc_common.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int DA_TILE = 64;                     // positions per tile
constexpr int DA_BOX = 64 * 128;                // one [64 rows x 64 bf16] box, bytes
constexpr int DA_NBOX = LAT / 64;               // 9 boxes per 576-wide row block
constexpr int DA_TILE_BYTES = DA_NBOX * DA_BOX;  // 73728
constexpr int DA_THREADS = 224;
constexpr int OFF_Q = 0;
constexpr int OFF_C = OFF_Q + DA_TILE_BYTES;    // two stages
constexpr int OFF_BAR = OFF_C + 2 * DA_TILE_BYTES;
constexpr int OFF_MISC = OFF_BAR + 16 * 8;  // 13 barriers used
constexpr int OFF_ALPHA = OFF_MISC + 16;
constexpr int MAX_SEG = 96;                     // segments one CTA can hold
constexpr int OFF_SEG = OFF_ALPHA + HEADS * 4;
constexpr int DA_SMEM = OFF_SEG + MAX_SEG * 12 + 16 + 1024;  // + slack for 1024-byte alignment
constexpr uint32_t TM_O = 0, TM_S = 256;
constexpr float RESCALE_LOG2 = 8.f;             // tolerated growth of p before rescaling O

__global__ void __launch_bounds__(DA_THREADS, 1) decode_attn_tc_kernel(
    const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_c,
    const int* __restrict__ seq_lens, int B, int cap, int G, long long P, float scale_log2,
    float* __restrict__ o_part, float* __restrict__ ml_part, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* c_full = bars + 1;   // [2]
  uint64_t* c_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;   // [2]
  uint64_t* s_free = bars + 7;   // [2]
  uint64_t* p_full = bars + 9;
  uint64_t* o_done = bars + 10;
  uint64_t* mma_idle = bars + 11;  // [2]: one per MMA-issuing thread
  uint64_t* q_free = bars + 13;    // MMA1 finished with the segment's query block
  uint64_t* o_free = bars + 14;    // the epilogue has read the segment's O^T
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* s_nseg = reinterpret_cast<int*>(smem + OFF_MISC + 8);
  float* s_alpha = reinterpret_cast<float*>(smem + OFF_ALPHA);
  int* seg = reinterpret_cast<int*>(smem + OFF_SEG);  // [MAX_SEG][3]: b, first, end

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();  // the query and the new cache row come from earlier kernels
  if (threadIdx.x == 0) {
    const long long r0 = decode_share_start(cta, G, P), r1 = decode_share_start(cta + 1, G, P);
    long long acc = 0;
    int nseg = 0;
    bool bad = false;
    for (int b = 0; b < B; ++b) {
      const long long S = (long long)seq_lens[b] + 1;
      if (S > cap) bad = true;
      const long long lo = max(acc, r0), hi = min(acc + S, r1);
      if (lo < hi) {
        if (nseg < MAX_SEG) {
          seg[3 * nseg] = b;
          seg[3 * nseg + 1] = (int)(lo - acc);
          seg[3 * nseg + 2] = (int)(hi - acc);
        }
        ++nseg;
      }
      acc += S;
    }
    if (bad) atomicExch(err, DEV_ERR_RANGE);
    if (acc != P || nseg > MAX_SEG) atomicExch(err, DEV_ERR_PLAN);
    *s_nseg = (bad || acc != P || nseg > MAX_SEG) ? 0 : nseg;
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c_full[i], 1);
      mbar_init(&c_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(&mma_idle[0], 1);
    mbar_init(&mma_idle[1], 1);
    mbar_init(q_free, 1);
    mbar_init(o_free, 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nseg = *s_nseg;
  auto seg_tiles = [&](int sg) { return (seg[3 * sg + 2] - seg[3 * sg + 1] + DA_TILE - 1) / DA_TILE; };

  if (nseg > 0) {
    if (warp == 0) {
      // ---------------------------------------------------------------- TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_c);
        int t = 0, issued = 0, qloads = 0;
        bool ok = true;
        for (int sg = 0; ok && sg < nseg; ++sg) {
          const int b = seg[3 * sg], p0 = seg[3 * sg + 1], nt = seg_tiles(sg);
          if (sg > 0 && !(ok = mbar_wait(q_free, (sg - 1) & 1, err, abort_flag))) break;
          mbar_expect_tx(q_full, DA_TILE_BYTES);
          for (int c = 0; c < DA_NBOX; ++c)
            tma_load_2d(smem + OFF_Q + c * DA_BOX, &map_q, q_full, 64 * c, HEADS * b);
          qloads = sg + 1;
          for (int i = 0; i < nt; ++i, ++t) {
            const int st = t & 1;
            if (t >= 2 && !(ok = mbar_wait(&c_empty[st], ((t - 2) >> 1) & 1, err, abort_flag)))
              break;
            mbar_expect_tx(&c_full[st], DA_TILE_BYTES);
            const int row = b * cap + p0 + DA_TILE * i;
            for (int c = 0; c < DA_NBOX; ++c)
              tma_load_2d(smem + OFF_C + st * DA_TILE_BYTES + c * DA_BOX, &map_c, &c_full[st],
                          64 * c, row);
            issued = t + 1;
          }
        }
        // Never leave the CTA with copies in flight: wait (bounded) for the last ones.
        volatile int no_abort = 0;
        if (qloads > 0) mbar_wait(q_full, (qloads - 1) & 1, err, &no_abort);
        for (int u = max(0, issued - 2); u < issued; ++u)
          mbar_wait(&c_full[u & 1], (u >> 1) & 1, err, &no_abort);
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA1 issuer
      if (lane == 0) {
        constexpr uint32_t idesc_s = idesc_bf16(64, 64, false, false);
        const uint32_t qb = sbase + OFF_Q;
        bool ok = true;
        int t = 0;
        for (int sg = 0; ok && sg < nseg; ++sg) {
          const int nt = seg_tiles(sg);
          if (!(ok = mbar_wait(q_full, sg & 1, err, abort_flag))) break;
          for (int i = 0; i < nt; ++i, ++t) {
            const int st = t & 1;
            ok = mbar_wait(&c_full[st], (t >> 1) & 1, err, abort_flag);
            if (ok && t >= 2) ok = mbar_wait(&s_free[st], ((t - 2) >> 1) & 1, err, abort_flag);
            if (!ok) break;
            fence_after();
            const uint32_t cb = sbase + OFF_C + st * DA_TILE_BYTES;
#pragma unroll
            for (int c = 0; c < DA_NBOX; ++c)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t a = sdesc_sw128(qb + c * DA_BOX + k * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(cb + c * DA_BOX + k * 32, 16, 1024);
                mma_bf16(tmem + TM_S + 64 * st, a, bd, idesc_s, (c | k) != 0);
              }
            mma_commit(&s_full[st]);
          }
          mma_commit(q_free);  // the query block may be replaced once these MMAs are done
        }
        // All issued MMAs must finish before tensor memory is released.
        mma_commit(&mma_idle[0]);
        volatile int no_abort = 0;
        mbar_wait(&mma_idle[0], 0, err, &no_abort);
      }
    } else if (warp == 6) {
      // ---------------------------------------------------------------- MMA2 issuer
      if (lane == 0) {
        constexpr uint32_t idesc_o = idesc_bf16(128, 64, true, false);
        bool ok = true;
        int t = 0;
        for (int sg = 0; ok && sg < nseg; ++sg) {
          const int nt = seg_tiles(sg);
          if (sg > 0 && !(ok = mbar_wait(o_free, (sg - 1) & 1, err, abort_flag))) break;
          for (int i = 0; i < nt; ++i, ++t) {
            const int st = t & 1;
            if (!(ok = mbar_wait(p_full, t & 1, err, abort_flag))) break;
            fence_after();
            const uint32_t cb = sbase + OFF_C + st * DA_TILE_BYTES;
#pragma unroll
            for (int d = 0; d < 4; ++d)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                // A = C^T: MN-major, 128 latent dims (2 boxes, DA_BOX apart) x 16 positions.
                const uint64_t a = sdesc_sw128(cb + 2 * d * DA_BOX + k * 2048, DA_BOX, 1024);
                const uint64_t bd = sdesc_sw128(cb + 8 * DA_BOX + k * 32, 16, 1024);
                mma_bf16(tmem + TM_O + 64 * d, a, bd, idesc_o, (i > 0) || (k > 0));
              }
            mma_commit(o_done);
            mma_commit(&c_empty[st]);
          }
        }
        mma_commit(&mma_idle[1]);
        volatile int no_abort = 0;
        mbar_wait(&mma_idle[1], 0, err, &no_abort);
      }
    } else if (warp >= 2 && warp <= 5) {
      // ---------------------------------------------------------------- softmax warps
      const int q = warp & 3;                 // tensor-memory lane quarter of this warp
      const int h = 16 * q + lane;            // head of this thread's S row (lanes 0..15)
      const bool own = lane < 16;
      const int tid = threadIdx.x - 64;       // 0..127
      const uint32_t lane_off = (uint32_t)(32 * q) << 16;
      bool ok = true;
      int t = 0;
      for (int sg = 0; ok && sg < nseg; ++sg) {
        const int b = seg[3 * sg], p0 = seg[3 * sg + 1], p1 = seg[3 * sg + 2];
        const int nt = seg_tiles(sg);
        float m = -INFINITY, l = 0.f;
        for (int i = 0; i < nt; ++i, ++t) {
          const int st = t & 1;
          if (!(ok = mbar_wait(&s_full[st], (t >> 1) & 1, err, abort_flag))) break;
          fence_after();
          uint32_t r[2][32];
          tmem_ld32(tmem + lane_off + TM_S + 64 * st, r[0]);
          tmem_ld32(tmem + lane_off + TM_S + 64 * st + 32, r[1]);
          tmem_wait_ld();
          fence_before();
          mbar_arrive(&s_free[st]);
          const int n = min(DA_TILE, p1 - (p0 + DA_TILE * i));
          float tmax = -INFINITY;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float sc = (j < n) ? __uint_as_float(r[j >> 5][j & 31]) * scale_log2 : -INFINITY;
            r[j >> 5][j & 31] = __float_as_uint(sc);
            tmax = fmaxf(tmax, sc);
          }
          bool need = false;
          if (own) {
            float alpha = 1.f;
            if (tmax > m + RESCALE_LOG2) {
              if (m != -INFINITY) {
                alpha = exp2f(m - tmax);
                need = true;
              }
              l *= alpha;
              m = tmax;
            }
            s_alpha[h] = alpha;
          }
          uint32_t pk[32];
          float lsum = 0.f;
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float a = exp2f(__uint_as_float(r[j >> 5][j & 31]) - m);
            const float c = exp2f(__uint_as_float(r[(j + 1) >> 5][(j + 1) & 31]) - m);
            __nv_bfloat162 pr = __floats2bfloat162_rn(a, c);
            lsum += __low2float(pr) + __high2float(pr);
            pk[j >> 1] = *reinterpret_cast<uint32_t*>(&pr);
          }
          l += lsum;
          // Box 8 (rotary dims) of this stage was last read by this tile's MMA1 and by MMA2 of
          // tile t-2, both complete (the stage was refilled for tile t after the latter).
          uint8_t* cst = smem + OFF_C + st * DA_TILE_BYTES;
          if (own) {  // P row h: 64 bf16 = 8 chunks of 16 B, 128-byte swizzle, in box 8
            uint8_t* prow = cst + 8 * DA_BOX + h * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(prow + ((c ^ (h & 7)) * 16)) =
                  make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          }
          if (n < DA_TILE) {  // rows past the segment end must not reach MMA2 as NaN/Inf
            const int chunks = (DA_TILE - n) * 8 * 8;
            for (int e = tid; e < chunks; e += 128) {
              const int row = n + e / 64, box = (e / 8) % 8, c16 = e % 8;
              *reinterpret_cast<uint4*>(cst + box * DA_BOX + row * 128 + c16 * 16) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          // MMA2 of the previous tile must be complete before O^T may be rescaled, and every
          // o_done phase is consumed here, in order, before this tile's MMA2 can be issued.
          if (t >= 1 && !(ok = mbar_wait(o_done, (t - 1) & 1, err, abort_flag))) break;
          if (named_bar_or(1, 128, need)) {
            fence_after();
#pragma unroll
            for (int d = 0; d < 4; ++d)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                uint32_t o[32];
                const uint32_t ta = tmem + lane_off + TM_O + 64 * d + 32 * hh;
                tmem_ld32(ta, o);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  o[e] = __float_as_uint(__uint_as_float(o[e]) * s_alpha[32 * hh + e]);
                tmem_st32(ta, o);
              }
            tmem_wait_st();
          }
          fence_proxy_async();
          fence_before();
          mbar_arrive(p_full);
        }
        if (!ok || !(ok = mbar_wait(o_done, (t - 1) & 1, err, abort_flag))) break;
        // Segment epilogue: unnormalised O^T, m and l of every head into slot b + cta.
        fence_after();
        const size_t slot = (size_t)b + cta;
        float* op = o_part + slot * HEADS * KV_LORA;
#pragma unroll
        for (int d = 0; d < 4; ++d) {
          const int dim = 128 * d + 32 * q + lane;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + TM_O + 64 * d + 32 * hh, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              op[(size_t)(32 * hh + e) * KV_LORA + dim] = __uint_as_float(o[e]);
          }
        }
        if (own) {
          ml_part[(slot * HEADS + h) * 2] = m;
          ml_part[(slot * HEADS + h) * 2 + 1] = l;
        }
        fence_before();
        mbar_arrive(o_free);
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

// 2-D bf16 / uint8 tensor map with 128-byte swizzle: rows x cols, row pitch in bytes.
bool make_tmap_2d(CUtensorMap* m, bool bf16, const void* base, uint64_t cols, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t init_decode_tc_kernel() {
  return cudaFuncSetAttribute(decode_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DA_SMEM);
}

cudaError_t launch_decode_attention_tc(const __nv_bfloat16* qfull, const __nv_bfloat16* cache,
                                       int cap, const int* seq_lens, DecodePlan plan,
                                       float scale, float* o_part, float* ml_part, int* err,
                                       cudaStream_t st, bool pdl) {
  if (plan.B == 0) return cudaSuccess;
  CUtensorMap mq, mc;
  if (!make_tmap_2d(&mq, true, qfull, LAT, (uint64_t)plan.B * HEADS, LAT * 2, 64, 64) ||
      !make_tmap_2d(&mc, true, cache, LAT, (uint64_t)plan.B * cap, LAT * 2, 64, 64))
    return cudaErrorInvalidValue;
  return launch_kernel(decode_attn_tc_kernel, dim3(plan.G), dim3(DA_THREADS), DA_SMEM, st, pdl,
                       mq, mc, seq_lens, plan.B, cap, plan.G, plan.P,
                       scale * 1.4426950408889634f, o_part, ml_part, err);
}

}  // namespace mla
