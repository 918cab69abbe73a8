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
//   warp 0      computes the CTA's segments (a warp-wide prefix sum of the lengths), then, as
//               TMA producer, loads the query block once per segment and 64-position cache
//               tiles into a two-stage ring (9 boxes of 64 rows x 64 columns, 128-byte swizzle);
//   warp 1      allocates tensor memory and issues, from one thread,
//                 MMA1  S[64 heads, 64 pos]   = Q[64, 576] . C[64, 576]^T    (M=64,  N=64);
//   warp 6      issues, from one thread,
//                 MMA2  O^T[512, 64 heads]   += C[64 pos, 0:512]^T . P^T     (M=128, N=64, x4).
//               Two issuers keep MMA2 of a tile from queueing behind the next tile's load;
//   warps 2..5  softmax: two threads per head (a row of S, 32 scores each), online softmax in
//               base 2 with a lazy rescale of O^T (only when a head's running maximum grows by
//               more than 2^8), P written as bf16 into the tile's rotary box (box 8), which
//               MMA1 no longer needs; then the epilogue writes the unnormalised partial O, the
//               maximum m and the sum l of every head.
// A tile's MMA2 does not wait for the previous tile's: only a rescale of O^T needs the previous
// MMA2 to be complete, and it is rare once a head's maximum has settled.
// Partial outputs: o_part[slot][dim][head] = O / l (fp16), or [slot][head][dim] when
// head_major is set; ml_part[slot][head] = (m, l).
// Tensor memory: O^T in columns [0, 256) (lane = latent dim, column = head within each of the
// four 128-dim blocks), S in [256, 320) and [320, 384) (double buffer).
#include "tc_common.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int DA_TILE = 64;                     // positions per tile
constexpr int DA_STAGES = 2;                    // tiles in flight
constexpr int DA_QBOX = 64 * 128;               // one [64 heads x 64 bf16] query box, bytes
constexpr int DA_BOX = DA_TILE * 128;           // one [64 rows x 64 bf16] cache box, bytes
constexpr int DA_NBOX = LAT / 64;               // 9 boxes per 576-wide row block
constexpr int DA_Q_BYTES = DA_NBOX * DA_QBOX;    // 73728
// 73728 per tile: two stages and the query block (221 KB) fill shared memory.
constexpr int DA_TILE_BYTES = DA_NBOX * DA_BOX;
constexpr int DA_THREADS = 224;
constexpr int OFF_Q = 0;
constexpr int OFF_C = OFF_Q + DA_Q_BYTES;
constexpr int OFF_BAR = OFF_C + DA_STAGES * DA_TILE_BYTES;
constexpr int DA_NBAR = 21;                     // mbarriers (bars[0..20], with gaps)
constexpr int OFF_MISC = OFF_BAR + 24 * 8;
static_assert(DA_NBAR * 8 <= OFF_MISC - OFF_BAR, "the barriers must not reach the misc words");
constexpr int OFF_ALPHA = OFF_MISC + 16;   // [2][HEADS] rescale factors, by tile parity
constexpr int OFF_INVL = OFF_ALPHA + 2 * HEADS * 4;  // [HEADS] 1 / l of the finished segment
constexpr int MAX_SEG = 96;                     // segments one CTA can hold
constexpr int DA_L2_AHEAD = 1;                  // tiles prefetched into L2 ahead of the ring
constexpr int OFF_SEG = OFF_INVL + HEADS * 4;
constexpr int DA_SMEM = OFF_SEG + MAX_SEG * 12 + 16 + 1024;  // + slack for 1024-byte alignment
constexpr uint32_t TM_O = 0, TM_S = 256;
static_assert(DA_BOX == HEADS * DA_TILE * 2, "P (64 heads x DA_TILE bf16) must fill box 8");
constexpr float RESCALE_LOG2 = 8.f;             // tolerated growth of p before rescaling O

// Eight consecutive 32-bit words to global memory in one 32-byte store (dst 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__global__ void __launch_bounds__(DA_THREADS, 1) decode_attn_tc_kernel(
    const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_c,
    const int* __restrict__ seq_lens, int B, const CacheRef cache, int G, long long P, int K,
    float scale_log2,
    __half* __restrict__ o_part, float* __restrict__ ml_part, int* err, int head_major) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* c_full = bars + 1;   // [DA_STAGES]
  uint64_t* c_empty = bars + 5;  // [DA_STAGES]
  uint64_t* s_full = bars + 9;   // [2]
  uint64_t* s_free = bars + 11;  // [2]
  uint64_t* p_full = bars + 13;  // [DA_STAGES]: P of the stage's tile is in box 8
  uint64_t* mma_idle = bars + 17;  // [2]: one per MMA-issuing thread
  uint64_t* q_free = bars + 19;    // MMA1 finished with the segment's query block
  uint64_t* o_free = bars + 20;    // the epilogue has read the segment's O^T
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* s_nseg = reinterpret_cast<int*>(smem + OFF_MISC + 8);
  float* s_alpha = reinterpret_cast<float*>(smem + OFF_ALPHA);
  float* s_invl = reinterpret_cast<float*>(smem + OFF_INVL);
  int* seg = reinterpret_cast<int*>(smem + OFF_SEG);  // [MAX_SEG][3]: b, first, end

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  pdl_launch_dependents();
  // The set-up below reads only the lengths, which no kernel of this decode step changes before
  // the attention has finished, so it overlaps the tail of the previous kernel; the loads of
  // the query and of the cache (whose new row an earlier kernel wrote) wait for it.
  if (warp == 0) {
    // This CTA's segments: the pieces of [r0, r1) in the concatenation of all sequences, found
    // with a warp-wide prefix sum of the lengths, 32 sequences at a time.
    const long long r0 = decode_share_start(cta, G, P), r1 = decode_share_start(cta + 1, G, P);
    long long base = 0;
    int nseg = 0;
    bool bad = false;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      const long long S = b < B ? (long long)seq_lens[b] + 1 + K : 0;
      long long inc = S;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += v;
      }
      const long long acc = base + inc - S + K;  // line position of sequence b's position 0
      const long long lo = max(acc, r0), hi = min(acc + S - K, r1);
      const bool has = b < B && lo < hi;
      const unsigned mask = __ballot_sync(0xffffffffu, has);
      const int idx = nseg + __popc(mask & ((1u << lane) - 1u));
      if (has && idx < MAX_SEG) {
        seg[3 * idx] = b;
        seg[3 * idx + 1] = (int)(lo - acc);
        seg[3 * idx + 2] = (int)(hi - acc);
      }
      nseg += __popc(mask);
      bad |= __any_sync(0xffffffffu, b < B && S - K > cache.capacity()) != 0;
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
      if (bad) atomicExch(err, DEV_ERR_RANGE);
      if (base != P || nseg > MAX_SEG) atomicExch(err, DEV_ERR_PLAN);
      *s_nseg = (bad || base != P || nseg > MAX_SEG) ? 0 : nseg;
    }
  }
  if (threadIdx.x == 32) {
    mbar_init(q_full, 1);
    for (int i = 0; i < DA_STAGES; ++i) {
      mbar_init(&c_full[i], 1);
      mbar_init(&c_empty[i], 1);
      mbar_init(&p_full[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
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
  // A segment [p0, p1) is read in tiles from a0 = p0.  With a paged cache the tiles start at
  // multiples of DA_TILE within the sequence instead (so a tile never crosses a page): a0 = p0
  // rounded down, and positions before p0 in the first tile are masked.
  const int align_mask = cache.paged() ? ~(DA_TILE - 1) : ~0;
  auto seg_a0 = [&](int sg) { return seg[3 * sg + 1] & align_mask; };
  auto seg_tiles = [&](int sg) { return (seg[3 * sg + 2] - seg_a0(sg) + DA_TILE - 1) / DA_TILE; };
  // Cache row of a tile's first position; an invalid page reads past the array (zero fill)
  // and is flagged.
  const long long c_rows = cache.rows(B);
  auto tile_row = [&](int b, int pos) -> int {
    const long long r = cache.row(b, pos);
    if (r < 0) {
      atomicExch(err, DEV_ERR_RANGE);
      return (int)c_rows;
    }
    return (int)r;
  };
  pdl_wait();  // the query and the new cache row come from earlier kernels

  if (nseg > 0) {
    if (warp == 0) {
      // ---------------------------------------------------------------- TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_c);
        int t = 0, issued = 0, qloads = 0;
        bool ok = true;
        for (int sg = 0; ok && sg < nseg; ++sg) {
          const int b = seg[3 * sg], a0 = seg_a0(sg), nt = seg_tiles(sg);
          if (sg > 0 && !(ok = mbar_wait(q_free, (sg - 1) & 1, err, abort_flag))) break;
          mbar_expect_tx(q_full, DA_Q_BYTES);
          for (int c = 0; c < DA_NBOX; ++c)
            tma_load_2d(smem + OFF_Q + c * DA_QBOX, &map_q, q_full, 64 * c, HEADS * b);
          qloads = sg + 1;
          for (int i = 0; i < nt; ++i, ++t) {
            const int st = t % DA_STAGES;
            if (t >= DA_STAGES &&
                !(ok = mbar_wait(&c_empty[st], ((t / DA_STAGES) - 1) & 1, err, abort_flag)))
              break;
            mbar_expect_tx(&c_full[st], DA_TILE_BYTES);
            const int row = tile_row(b, a0 + DA_TILE * i);
            for (int c = 0; c < DA_NBOX; ++c)
              tma_load_2d(smem + OFF_C + st * DA_TILE_BYTES + c * DA_BOX, &map_c, &c_full[st],
                          64 * c, row);
            // The two-stage ring holds few bytes in flight: start the DRAM reads of the tile
            // DA_L2_AHEAD later into L2, so its own load later finds it there.  At the last
            // tile of a segment, the next segment's query block and first tile instead.
            if (i + DA_L2_AHEAD < nt) {
              const int ra = tile_row(b, a0 + DA_TILE * (i + DA_L2_AHEAD));
              for (int c = 0; c < DA_NBOX; ++c)
                tma_prefetch_l2_2d(&map_c, 64 * c, ra);
            } else if (i == nt - 1 && sg + 1 < nseg) {
              const int bn = seg[3 * (sg + 1)], rn = tile_row(bn, seg_a0(sg + 1));
              for (int c = 0; c < DA_NBOX; ++c) {
                tma_prefetch_l2_2d(&map_q, 64 * c, HEADS * bn);
                tma_prefetch_l2_2d(&map_c, 64 * c, rn);
              }
            }
            issued = t + 1;
          }
        }
        // Never leave the CTA with copies in flight: wait (bounded) for the last ones.
        volatile int no_abort = 0;
        if (qloads > 0) mbar_wait(q_full, (qloads - 1) & 1, err, &no_abort);
        for (int u = max(0, issued - DA_STAGES); u < issued; ++u)
          mbar_wait(&c_full[u % DA_STAGES], (u / DA_STAGES) & 1, err, &no_abort);
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA1 issuer
      if (lane == 0) {
        constexpr uint32_t idesc_s = idesc_bf16(64, DA_TILE, false, false);
        const uint32_t qb = sbase + OFF_Q;
        bool ok = true;
        int t = 0;
        for (int sg = 0; ok && sg < nseg; ++sg) {
          const int nt = seg_tiles(sg);
          if (!(ok = mbar_wait(q_full, sg & 1, err, abort_flag))) break;
          for (int i = 0; i < nt; ++i, ++t) {
            const int st = t % DA_STAGES, sb = t & 1;
            ok = mbar_wait(&c_full[st], (t / DA_STAGES) & 1, err, abort_flag);
            if (ok && t >= 2) ok = mbar_wait(&s_free[sb], ((t - 2) >> 1) & 1, err, abort_flag);
            if (!ok) break;
            fence_after();
            const uint32_t cb = sbase + OFF_C + st * DA_TILE_BYTES;
#pragma unroll
            for (int c = 0; c < DA_NBOX; ++c)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t a = sdesc_sw128(qb + c * DA_QBOX + k * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(cb + c * DA_BOX + k * 32, 16, 1024);
                mma_bf16(tmem + TM_S + DA_TILE * sb, a, bd, idesc_s, (c | k) != 0);
              }
            mma_commit(&s_full[sb]);
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
            const int st = t % DA_STAGES;
            if (!(ok = mbar_wait(&p_full[st], (t / DA_STAGES) & 1, err, abort_flag))) break;
            fence_after();
            const uint32_t cb = sbase + OFF_C + st * DA_TILE_BYTES;
#pragma unroll
            for (int d = 0; d < 4; ++d)
#pragma unroll
              for (int k = 0; k < DA_TILE / 16; ++k) {
                // A = C^T: MN-major, 128 latent dims (2 boxes, DA_BOX apart) x 16 positions.
                const uint64_t a = sdesc_sw128(cb + 2 * d * DA_BOX + k * 2048, DA_BOX, 1024);
                // B = P: K-major, 64 heads x 16 positions (rows of 128 B, 128-byte swizzle).
                const uint64_t bd = sdesc_sw128(cb + 8 * DA_BOX + k * 32, 16, 1024);
                mma_bf16(tmem + TM_O + 64 * d, a, bd, idesc_o, (i > 0) || (k > 0));
              }
            mma_commit(&c_empty[st]);  // also tells the softmax warps that MMA2(t) is done
          }
        }
        mma_commit(&mma_idle[1]);
        volatile int no_abort = 0;
        mbar_wait(&mma_idle[1], 0, err, &no_abort);
      }
    } else if (warp >= 2 && warp <= 5) {
      // ---------------------------------------------------------------- softmax warps
      // S rows (heads) of an M=64 accumulator sit in lanes 0..15 of each 32-lane quarter.  The
      // 16x64b load spreads such a quarter over the whole warp: thread `lane` reads row
      // lane/4 + 8*(lane%2) of the quarter and the columns of parity (lane/2)%2, so every
      // head is shared by two threads (lanes l and l^2), each holding 32 of its 64 scores.
      const int q = warp & 3;                 // tensor-memory lane quarter of this warp
      const int h = 16 * q + (lane >> 2) + 8 * (lane & 1);  // head of this thread's S row
      const int par = (lane >> 1) & 1;        // this thread's column parity
      const int tid = threadIdx.x - 64;       // 0..127
      const uint32_t lane_off = (uint32_t)(32 * q) << 16;
      bool ok = true;
      int t = 0;
      for (int sg = 0; ok && sg < nseg; ++sg) {
        const int b = seg[3 * sg], p0 = seg[3 * sg + 1], p1 = seg[3 * sg + 2];
        const int nt = seg_tiles(sg);
        float m = -INFINITY, l = 0.f;         // running maximum; this thread's half of the sum
        for (int i = 0; i < nt; ++i, ++t) {
          const int st = t % DA_STAGES, sb = t & 1;
          if (!(ok = mbar_wait(&s_full[sb], (t >> 1) & 1, err, abort_flag))) break;
          fence_after();
          uint32_t r[32];                     // r[j] = S[h][2j + par]
          tmem_ld16x64b_x32(tmem + lane_off + TM_S + DA_TILE * sb, r);
          tmem_wait_ld();
          fence_before();
          mbar_arrive(&s_free[sb]);
          const int a0 = p0 & align_mask;
          const int n = min(DA_TILE, p1 - (a0 + DA_TILE * i));  // columns [lo, n) are valid
          const int lo = i == 0 ? p0 - a0 : 0;
          float tmax = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = 2 * j + par;
            const float sc = (col >= lo && col < n) ? __uint_as_float(r[j]) * scale_log2 : -INFINITY;
            r[j] = __float_as_uint(sc);
            tmax = fmaxf(tmax, sc);
          }
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
          bool need = false;
          {
            float alpha = 1.f;
            if (tmax > m + RESCALE_LOG2) {
              if (m != -INFINITY) {
                alpha = exp2f(m - tmax);
                need = true;
              }
              l *= alpha;
              m = tmax;
            }
            if (par == 0) s_alpha[HEADS * sb + h] = alpha;
          }
          // p = 2^(s - m) rounded to bf16 (the MMA's operand type; l sums the rounded values).
          uint32_t pb[16];                    // bf16 bits of this thread's 32 values, 2 per word
          float lsum = 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            __nv_bfloat162 pr = __floats2bfloat162_rn(fast_exp2(__uint_as_float(r[j]) - m),
                                                      fast_exp2(__uint_as_float(r[j + 1]) - m));
            lsum += __low2float(pr) + __high2float(pr);
            pb[j >> 1] = *reinterpret_cast<uint32_t*>(&pr);
          }
          l += lsum;
          // Trade halves with the partner so that the even-column thread owns columns 0..31 and
          // the odd-column thread columns 32..63: the even thread sends its values of columns
          // 32..62, the odd thread its values of columns 1..31.
          uint32_t pk[16];                    // bf16x2 of columns (2w, 2w+1) of this thread's half
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const uint32_t send = par ? pb[w] : pb[8 + w];
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
            // send/recv carry two values: word w holds elements 2w and 2w+1 of a half.
            const uint32_t mine = par ? pb[8 + w] : pb[w];
            const uint32_t ev = par ? recv : mine, od = par ? mine : recv;  // even / odd cols
            pk[2 * w] = (ev & 0xFFFFu) | (od << 16);
            pk[2 * w + 1] = (ev >> 16) | (od & 0xFFFF0000u);
          }
          // Box 8 (rotary dims) of this stage was last read by this tile's MMA1 and by MMA2 of
          // tile t-2, both complete (the stage was refilled for tile t after the latter).
          uint8_t* cst = smem + OFF_C + st * DA_TILE_BYTES;
          {  // P row h: 64 bf16 = 8 chunks of 16 B, 128-byte swizzle; this thread's 4 chunks
            uint8_t* prow = cst + 8 * DA_BOX + h * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(prow + (((4 * par + c) ^ (h & 7)) * 16)) =
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
          // O^T may only be rescaled once MMA2 of the previous tile is complete; its commit on
          // that tile's stage barrier says so.  Without a rescale, this tile's MMA2 simply
          // queues behind the previous one, so the tiles do not wait on each other.  (That
          // barrier's next phase needs this warpgroup's P of tile t+3, so it cannot run ahead.)
          if (named_bar_or(1, 128, need)) {
            if (!(ok = mbar_wait(&c_empty[(t - 1) % DA_STAGES], ((t - 1) / DA_STAGES) & 1, err,
                                 abort_flag)))
              break;
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
                  o[e] = __float_as_uint(__uint_as_float(o[e]) * s_alpha[HEADS * sb + 32 * hh + e]);
                tmem_st32(ta, o);
              }
            tmem_wait_st();
          }
          fence_proxy_async();
          fence_before();
          mbar_arrive(&p_full[st]);
        }
        if (!ok || !(ok = mbar_wait(&c_empty[(t - 1) % DA_STAGES], ((t - 1) / DA_STAGES) & 1, err,
                                    abort_flag)))
          break;
        // Segment epilogue: O / l, m and l of every head into slot b + cta.  The partial is
        // divided by its own sum, so its values are bounded by those of the cache rows, and
        // stored as fp16 (11-bit mantissa).  Head-minor ([dim][head]): a thread writes the 64
        // heads of its latent dimension (its TMEM lane) as four 32-byte vectors.  Head-major
        // ([head][dim]): lanes 2i and 2i+1 (consecutive dims) swap one value per head pair, so
        // each stores two dims of one head as a 4-byte pair.
        const float lrow = l + __shfl_xor_sync(0xffffffffu, l, 2);
        if (par == 0) {
          s_invl[h] = 1.f / lrow;
          ml_part[((size_t)b + cta) * HEADS * 2 + 2 * h] = m;
          ml_part[((size_t)b + cta) * HEADS * 2 + 2 * h + 1] = lrow;
        }
        named_bar(1, 128);
        fence_after();
        const size_t slot = (size_t)b + cta;
        __half* op = o_part + slot * HEADS * KV_LORA;
#pragma unroll 1
        for (int d = 0; d < 4; ++d) {
          const int dim = 128 * d + 32 * q + lane;
          uint32_t o[2][32];
          tmem_ld32(tmem + lane_off + TM_O + 64 * d, o[0]);
          tmem_ld32(tmem + lane_off + TM_O + 64 * d + 32, o[1]);
          tmem_wait_ld();
          if (head_major) {
            const int odd = lane & 1;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int hh = 2 * e;
              const float x0 = __uint_as_float(o[hh >> 5][hh & 31]) * s_invl[hh];
              const float x1 = __uint_as_float(o[(hh + 1) >> 5][(hh + 1) & 31]) * s_invl[hh + 1];
              // the even lane keeps head hh, the odd lane head hh + 1
              const float got = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
              const __half2 v = odd ? __floats2half2_rn(got, x1) : __floats2half2_rn(x0, got);
              *reinterpret_cast<__half2*>(op + (size_t)(hh + odd) * KV_LORA + (dim - odd)) = v;
            }
          } else {
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int hh = 2 * e;
              __half2 v = __floats2half2_rn(__uint_as_float(o[hh >> 5][hh & 31]) * s_invl[hh],
                                            __uint_as_float(o[(hh + 1) >> 5][(hh + 1) & 31]) *
                                                s_invl[hh + 1]);
              pk[e] = *reinterpret_cast<uint32_t*>(&v);
            }
            __half* dst = op + (size_t)dim * HEADS;
#pragma unroll
            for (int v = 0; v < 4; ++v) st_global_v8(dst + 16 * v, &pk[8 * v]);
          }
        }
        fence_before();
        mbar_arrive(o_free);
        // Every thread has read s_invl before the next segment's epilogue rewrites it: that
        // epilogue is at least one tile (and its named barrier) away.
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

cudaError_t launch_decode_attention_tc(const __nv_bfloat16* qfull, const CacheRef& cache,
                                       const int* seq_lens, DecodePlan plan,
                                       float scale, __half* o_part, float* ml_part, int* err,
                                       cudaStream_t st, bool pdl, bool head_major) {
  if (plan.B == 0) return cudaSuccess;
  const long long rows = cache.rows(plan.B);
  if (rows <= 0 || rows + DA_TILE > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  CUtensorMap mq, mc;
  if (!make_tmap_2d(&mq, true, qfull, LAT, (uint64_t)plan.B * HEADS, LAT * 2, 64, 64) ||
      !make_tmap_2d(&mc, true, cache.base, LAT, (uint64_t)rows, LAT * 2, 64, DA_TILE))
    return cudaErrorInvalidValue;
  return launch_kernel(decode_attn_tc_kernel, dim3(plan.G), dim3(DA_THREADS), DA_SMEM, st, pdl,
                       mq, mc, seq_lens, plan.B, cache, plan.G, plan.P, plan.K,
                       scale * 1.4426950408889634f, o_part, ml_part, err, head_major ? 1 : 0);
}

}  // namespace mla
