// Causal prefill attention on the tcgen05 tensor cores.
//
// `mla-prefill` excerpt ("Key content up-projection" page): per head, q = [q_nope | RoPE(q_pe)]
// (192), k = [k_nope | RoPE(k_pe)] with the rotary key shared by all heads, scores q.k times the
// softmax scale, key s visible from query t iff s <= t, fp32 softmax over keys, o = P v (128).
// The head dimensions stay 192 / 128 (no padding of v to 192).
//
// Work items are (head, 128-query tile, sequence), heaviest query tiles first.  One persistent
// CTA per SM takes its share of them in turn (rounds of one item per CTA, in alternating
// direction), and every role keeps its stage and barrier-phase counters across items, so that
// the next item's query and key loads and its first MMAs overlap the current item's epilogue.
// The query tile's buffer is reloaded once MMA1 of the item's last key tile is done (its commit
// on that key stage).  20 warps:
//   warp 0      TMA producer of the query tile (3 boxes of 64 columns) and, for every 128-key
//               tile, of k = [k_nope (2 boxes) | rotary key from the cache rows (1 box)] into
//               a two-stage ring that MMA1 releases (128-byte swizzle, 3-D maps over
//               [tokens, heads, dims]);
//   warp 7      TMA producer of v (2 boxes) into its own two-stage ring, which MMA2 releases,
//               so that k runs ahead of the softmax;
//   warp 1      allocates tensor memory and issues MMA1  S = Q K^T  (M=128, N=128, K=192);
//   warp 6      issues MMA2  O += P V  (M=128, N=128, K=128) with P read from tensor memory
//               and v read MN-major;
//   warps 2..5, 8..19  softmax, four threads per query row (32 columns each of S, P and O;
//               the four trade row maxima through shared memory): causal mask on the
//               diagonal tile, online softmax in base 2 with a lazy rescale of O (only when the
//               running maximum grows by more than 2^8), P written to tensor memory as packed
//               bf16; then the epilogue normalises O and stores it as bf16, or as the two
//               e4m3 terms and per-(token, head) scale that the o_proj GEMM reads.
// MMA2 of a tile does not wait for the previous tile's: only a rescale of O needs the previous
// MMA2 to be complete, and the softmax waits for it then.
// Tensor memory: O in columns [0,128), S in [128,256) and [256,384), P in [384,448) and
// [448,512).
#include "tc_common.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int PA_TILE = 128;
constexpr int PA_BOX = 128 * 128;                 // [128 rows x 64 bf16] box, bytes
constexpr int PA_Q_BYTES = 3 * PA_BOX;            // q tile: 192 columns
constexpr int PA_K_BYTES = 3 * PA_BOX;            // k tile: 128 nope + 64 rotary
constexpr int PA_V_BYTES = 2 * PA_BOX;            // v tile: 128 columns
constexpr int PA_NG = 4;                           // softmax threads per query row
constexpr int PA_GC = PA_TILE / PA_NG;             // columns of S, P and O per thread (32)
constexpr int PA_SM_THREADS = 128 * PA_NG;         // softmax threads
constexpr int PA_THREADS = 128 + PA_SM_THREADS;    // + 4 warps: TMA k, MMA1, MMA2, TMA v
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + PA_Q_BYTES;          // two k stages
constexpr int OFF_V = OFF_K + 2 * PA_K_BYTES;      // two v stages
constexpr int OFF_BAR = OFF_V + 2 * PA_V_BYTES;
constexpr int PA_NBAR = 17;                        // mbarriers (bars[0..16])
constexpr int OFF_MISC = OFF_BAR + 24 * 8;
static_assert(PA_NBAR * 8 <= OFF_MISC - OFF_BAR, "the barriers must not reach the misc words");
constexpr int OFF_QFAIL = OFF_MISC + 16;          // [4] failure flags, one per lane quarter
constexpr int OFF_XCH = OFF_QFAIL + 16;           // [2 tile parities][PA_NG groups][128 rows]
// [2 item parities][PA_NG groups][128 rows] row sums: apart from xch, which a slower warp of
// the quarter may still be reading for the last tile when a faster one stores its sum.
constexpr int OFF_LX = OFF_XCH + 2 * PA_NG * 128 * 4;
constexpr int OFF_AX = OFF_LX + 2 * PA_NG * 128 * 4;  // [2 item parities][PA_NG][128 rows]
constexpr int PA_SMEM = OFF_AX + 2 * PA_NG * 128 * 4 + 1024;
constexpr uint32_t TM_O = 0, TM_S = 128, TM_P = 384;
constexpr float RESCALE_LOG2 = 8.f;

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// A box of a 3-D tensor map into L2 (no shared-memory destination, no completion).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// D (+)= A * B^T with A read from tensor memory (kind::f16, bf16 operands).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Two fp32 values in one 64-bit register (lo, hi), and the packed element-wise fused
// multiply-add and add on them: each lane is rounded exactly as fmaf and the fp32 add round it,
// in half the instructions.
__device__ __forceinline__ uint64_t pack2f(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// The largest of three values (one instruction).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// The work item (head, query tile, sequence) of a given index: heads vary fastest, then the
// query tiles from the heaviest (latest) one, then the sequences.
struct PaItem {
  int h, b, q0, L, kvr0, nt;
};

__device__ __forceinline__ PaItem pa_item(int i, int T, int nq, const int* seq_lens) {
  PaItem it;
  it.h = i % HEADS;
  const int y = (i / HEADS) % nq;
  it.b = i / (HEADS * nq);
  it.q0 = (nq - 1 - y) * PA_TILE;
  // Cached positions before this call (0 for a prefill over an empty cache): query i sits at
  // position L + i and sees keys 0..L+i.  The sequence's keys are rows kvr0 .. kvr0+L+T-1 of
  // kv (each sequence's L + T rows back to back).
  it.L = 0;
  it.kvr0 = 0;
  if (seq_lens != nullptr) {
    it.L = seq_lens[it.b];
    for (int bb = 0; bb < it.b; ++bb) it.kvr0 += seq_lens[bb] + T;
  } else {
    it.kvr0 = it.b * T;
  }
  it.nt = (it.L + min(it.q0 + PA_TILE, T) - 1) / PA_TILE + 1;  // key tiles (causal)
  return it;
}

// The r-th work item of this CTA, or -1: rounds of gridDim.x items, taken in alternating
// directions so that each CTA's share of heavy and light items evens out.
__device__ __forceinline__ int pa_item_index(int r, int n_items) {
  const long long G = gridDim.x;
  const long long i = r * G + ((r & 1) ? G - 1 - (long long)blockIdx.x : (long long)blockIdx.x);
  return i < n_items ? (int)i : -1;
}

__global__ void __launch_bounds__(PA_THREADS, 1) prefill_attn_tc_kernel(
    const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
    const __grid_constant__ CUtensorMap map_c, int T, const CacheRef cache,
    const int* __restrict__ seq_lens,
    float scale_log2,
    __nv_bfloat16* __restrict__ attn_out, uint8_t* __restrict__ o_hi, uint8_t* __restrict__ o_lo,
    float* __restrict__ o_sx, long kv_rows, int n_items, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* k_empty = bars + 3;   // [2]  MMA1 of the stage's tile is done
  uint64_t* v_full = bars + 5;    // [2]
  uint64_t* v_empty = bars + 7;   // [2]  MMA2 of the stage's tile is done (also frees P)
  uint64_t* s_full = bars + 9;    // [2]
  uint64_t* s_free = bars + 11;   // [2]
  uint64_t* p_full = bars + 13;   // [2]  P of the buffer's tile is in tensor memory
  uint64_t* mma_idle = bars + 15; // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  // [2] softmax failure flags, by item parity
  volatile int* s_fail = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Under programmatic dependent launch: let the next kernel be scheduled, then wait for the
  // previous one (q, kv and the cache rows are its outputs).
  pdl_launch_dependents();
  pdl_wait();
  const int nq = (T + PA_TILE - 1) / PA_TILE;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], PA_SM_THREADS);
      mbar_init(&p_full[i], PA_SM_THREADS);
      mbar_init(&mma_idle[i], 1);
    }
    *abort_flag = 0;
    s_fail[0] = s_fail[1] = 0;
    for (int qq = 0; qq < 4; ++qq) reinterpret_cast<volatile int*>(smem + OFF_QFAIL)[qq] = 0;
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

  if (warp == 0) {
    // -------------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_kv);
      tma_prefetch_desc(&map_c);
      int u = 0, nql = 0;  // key tiles and query tiles issued
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int i = pa_item_index(r, n_items);
        if (i < 0) break;
        const PaItem it = pa_item(i, T, nq, seq_lens);
        if ((long)it.kvr0 + it.L + T > kv_rows)
          atomicExch(err, DEV_ERR_PLAN);  // device lengths disagree with the host's kv layout
        // The query buffer is free once MMA1 of the previous item's last tile is done.
        if (r > 0 && !mbar_wait(&k_empty[(u - 1) & 1], ((u - 1) >> 1) & 1, err, abort_flag)) break;
        mbar_expect_tx(q_full, PA_Q_BYTES);
        for (int c = 0; c < 3; ++c)
          tma_load_3d(smem + OFF_Q + c * PA_BOX, &map_q, q_full, 64 * c, it.h, it.b * T + it.q0);
        ++nql;
        // The next item's query tile, into L2 ahead of its load.
        const int inext = pa_item_index(r + 1, n_items);
        if (inext >= 0) {
          const PaItem nx = pa_item(inext, T, nq, seq_lens);
          for (int c = 0; c < 3; ++c) tma_prefetch_l2_3d(&map_q, 64 * c, nx.h, nx.b * T + nx.q0);
        }
        for (int j = 0; j < it.nt; ++j, ++u) {
          const int st = u & 1;
          if (u >= 2 && !mbar_wait(&k_empty[st], ((u - 2) >> 1) & 1, err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* stg = smem + OFF_K + st * PA_K_BYTES;
          mbar_expect_tx(&k_full[st], PA_K_BYTES);
          const int k0 = j * PA_TILE;
          tma_load_3d(stg, &map_kv, &k_full[st], 0, it.h, it.kvr0 + k0);
          tma_load_3d(stg + PA_BOX, &map_kv, &k_full[st], 64, it.h, it.kvr0 + k0);
          if (!cache.paged()) {
            tma_load_2d(stg + 2 * PA_BOX, &map_c, &k_full[st], KV_LORA, it.b * cache.page + k0);
          } else {
            // Two 64-position boxes, each inside one page.  A block of real keys (before
            // L + T) on an invalid page is flagged; every out-of-range block reads zeros past
            // the pool (its keys, if any, are masked).
            for (int hb = 0; hb < 2; ++hb) {
              const int pos = k0 + 64 * hb;
              long long rr = cache.row(it.b, pos);
              if (rr < 0) {
                if (pos < it.L + T) atomicExch(err, DEV_ERR_RANGE);
                rr = cache.rows(0);
              }
              tma_load_2d(stg + 2 * PA_BOX + hb * (PA_BOX / 2), &map_c, &k_full[st], KV_LORA,
                          (int)rr);
            }
          }
        }
      }
      // No copy may be in flight when the CTA exits.
      volatile int no_abort = 0;
      if (nql > 0) mbar_wait(q_full, (nql - 1) & 1, err, &no_abort);
      for (int v = max(0, u - 2); v < u; ++v) mbar_wait(&k_full[v & 1], (v >> 1) & 1, err, &no_abort);
    }
  } else if (warp == 7) {
    // -------------------------------------------------------------------- v producer
    if (lane == 0) {
      int u = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int i = pa_item_index(r, n_items);
        if (i < 0) break;
        const PaItem it = pa_item(i, T, nq, seq_lens);
        for (int j = 0; j < it.nt; ++j, ++u) {
          const int st = u & 1;
          if (u >= 2 && !mbar_wait(&v_empty[st], ((u - 2) >> 1) & 1, err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* stg = smem + OFF_V + st * PA_V_BYTES;
          mbar_expect_tx(&v_full[st], PA_V_BYTES);
          const int k0 = j * PA_TILE;
          tma_load_3d(stg, &map_kv, &v_full[st], 128, it.h, it.kvr0 + k0);
          tma_load_3d(stg + PA_BOX, &map_kv, &v_full[st], 192, it.h, it.kvr0 + k0);
        }
      }
      volatile int no_abort = 0;
      for (int v = max(0, u - 2); v < u; ++v) mbar_wait(&v_full[v & 1], (v >> 1) & 1, err, &no_abort);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------------- MMA1 issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
      int u = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int i = pa_item_index(r, n_items);
        if (i < 0) break;
        const int nt = pa_item(i, T, nq, seq_lens).nt;
        ok = mbar_wait(q_full, r & 1, err, abort_flag);
        for (int j = 0; ok && j < nt; ++j, ++u) {
          const int st = u & 1;
          ok = mbar_wait(&k_full[st], (u >> 1) & 1, err, abort_flag);
          if (ok && u >= 2) ok = mbar_wait(&s_free[st], ((u - 2) >> 1) & 1, err, abort_flag);
          if (!ok) break;
          fence_after();
          const uint32_t kb = sbase + OFF_K + st * PA_K_BYTES;
#pragma unroll
          for (int ks = 0; ks < 12; ++ks) {
            const uint64_t a =
                sdesc_sw128(sbase + OFF_Q + (ks >> 2) * PA_BOX + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(kb + (ks >> 2) * PA_BOX + (ks & 3) * 32, 16, 1024);
            mma_bf16(tmem + TM_S + 128 * st, a, bd, idesc, ks > 0);
          }
          mma_commit(&s_full[st]);
          mma_commit(&k_empty[st]);
        }
      }
      mma_commit(&mma_idle[0]);
      volatile int no_abort = 0;
      mbar_wait(&mma_idle[0], 0, err, &no_abort);
    }
  } else if (warp == 6) {
    // -------------------------------------------------------------------- MMA2 issuer
    // An item's first MMA2 overwrites O: every softmax thread has read the previous item's O
    // in its epilogue before it takes part in this tile's p_full.
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, 128, false, true);
      int u = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int i = pa_item_index(r, n_items);
        if (i < 0) break;
        const int nt = pa_item(i, T, nq, seq_lens).nt;
        for (int j = 0; j < nt; ++j, ++u) {
          const int st = u & 1;
          if (!mbar_wait(&p_full[st], (u >> 1) & 1, err, abort_flag) ||
              !mbar_wait(&v_full[st], (u >> 1) & 1, err, abort_flag)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t vb = sbase + OFF_V + st * PA_V_BYTES;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            // B = v: MN-major, 128 value dims (2 boxes, PA_BOX apart) x 16 keys.
            const uint64_t bd = sdesc_sw128(vb + ks * 2048, PA_BOX, 1024);
            mma_bf16_ts(tmem + TM_O, tmem + TM_P + 64 * st + 8 * ks, bd, idesc,
                        (j > 0) || (ks > 0));
          }
          mma_commit(&v_empty[st]);
        }
      }
      mma_commit(&mma_idle[1]);
      volatile int no_abort = 0;
      mbar_wait(&mma_idle[1], 0, err, &no_abort);
    }
  } else if ((warp >= 2 && warp <= 5) || warp >= 8) {
    static_assert(PA_GC == 32, "one 32-column chunk per softmax thread");
    // -------------------------------------------------------------------- softmax warps
    // The four threads of a row sit in the four softmax warps of one tensor-memory lane
    // quarter; they trade their maxima through shared memory at one barrier of those 128
    // threads per tile.  Every thread of a quarter reaches that barrier in every tile it
    // starts; a failed wait is published in the quarter's flag before it, and all four warps
    // leave together after it.  The epilogue's exchanges (row sums, output maxima) and its
    // failure flag alternate between two slots by item parity: a thread can only write an
    // item's slot after the epilogue barrier of the item in between, which every thread
    // reaches only after reading the slot's previous contents.
    const int qw = warp & 3;
    const int grp = warp < 8 ? 0 : (warp - 4) / 4;  // columns [32 grp, 32 grp + 32)
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    const int row = 32 * qw + lane;
    float* xch = reinterpret_cast<float*>(smem + OFF_XCH);
    float* lx = reinterpret_cast<float*>(smem + OFF_LX);  // [item parity][PA_NG][128] sums
    float* ax = reinterpret_cast<float*>(smem + OFF_AX);  // [item parity][PA_NG][128] maxima
    volatile int* q_fail = reinterpret_cast<volatile int*>(smem + OFF_QFAIL) + qw;
    int u = 0;  // key tiles of this CTA so far: their stages and barrier phases
    bool ok = true;
    for (int r = 0;; ++r) {
      const int i = pa_item_index(r, n_items);
      if (i < 0) break;
      const PaItem it = pa_item(i, T, nq, seq_lens);
      const int L = it.L, q0 = it.q0, nt = it.nt;
      const int qi = q0 + row;                      // query position of this thread's row
      float m = -INFINITY, l = 0.f;                 // running maximum; this group's sum
      for (int j = 0; j < nt; ++j, ++u) {
        const int st = u & 1;
        if (ok) ok = mbar_wait(&s_full[st], (u >> 1) & 1, err, abort_flag);
        fence_after();
        const uint32_t s_addr = tmem + lane_off + TM_S + 128 * st + PA_GC * grp;
        const int kbase = j * PA_TILE + PA_GC * grp;
        const int vis = min(L + qi - kbase + 1, L + T - kbase);  // columns [0, vis) visible
        // Tiles wholly at or before the tile's first query position are visible to every row:
        // no mask there.
        const bool full = (j + 1) * PA_TILE <= L + q0 + 1;
        // The thread's 32 scores, read once; masked ones become -inf.
        uint32_t rs[32];
        float tmax = -INFINITY;
        if (ok) {
          tmem_ld32(s_addr, rs);
          tmem_wait_ld();
          if (!full) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (e >= vis) rs[e] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            tmax = max3f(tmax, __uint_as_float(rs[e]), __uint_as_float(rs[e + 1]));
        }
        xch[(PA_NG * st + grp) * 128 + row] = tmax;
        if (!ok) *q_fail = 1;
        named_bar(2 + qw, 128);
        if (*q_fail) {
          ok = false;
          break;
        }
#pragma unroll
        for (int g = 0; g < PA_NG; ++g) tmax = fmaxf(tmax, xch[(PA_NG * st + g) * 128 + row]);
        tmax *= scale_log2;  // scale > 0
        // The row's maximum, and so this decision, is the same in all four threads of the row.
        float alpha = 1.f;
        bool need = false;
        if (tmax > m + RESCALE_LOG2) {
          if (m != -INFINITY) {
            alpha = exp2f(m - tmax);
            need = true;
          }
          l *= alpha;
          m = tmax;
        }
        const float mu = (m == -INFINITY) ? 0.f : m;   // rows past T see no key at all
        // P's buffer was last read by MMA2 two tiles back (its commit on the v stage says so).
        if (u >= 2) ok = mbar_wait(&v_empty[st], ((u - 2) >> 1) & 1, err, abort_flag);
        // p = 2^(s * scale - m) (masked scores give 0), rounded to bf16 into P (16 packed
        // columns); l sums the unrounded p.
        if (ok) {
          uint32_t pk[16];
          const uint64_t sc2 = pack2f(scale_log2, scale_log2), nmu2 = pack2f(-mu, -mu);
          uint64_t ls = 0;  // the sums of the even and of the odd columns
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t x = ffma2(((uint64_t)rs[e + 1] << 32) | rs[e], sc2, nmu2);
            const float e0 = fast_exp2(__uint_as_float((uint32_t)x));
            const float e1 = fast_exp2(__uint_as_float((uint32_t)(x >> 32)));
            ls = fadd2(ls, pack2f(e0, e1));
            __nv_bfloat162 pr = __floats2bfloat162_rn(e0, e1);
            pk[e >> 1] = *reinterpret_cast<uint32_t*>(&pr);
          }
          l += __uint_as_float((uint32_t)ls) + __uint_as_float((uint32_t)(ls >> 32));
          tmem_st16(tmem + lane_off + TM_P + 64 * st + (PA_GC / 2) * grp, pk);
          fence_before();
          mbar_arrive(&s_free[st]);  // S of this buffer has been read
        }
        // O may only be rescaled once the previous tile's MMA2 is done (its commit on the
        // other v stage); each thread rescales its own 32 columns of its row.  (j >= 1 here:
        // the first tile of an item starts from m = -inf.)
        if (ok && need) {
          ok = mbar_wait(&v_empty[st ^ 1], ((u - 1) >> 1) & 1, err, abort_flag);
          if (ok) {
            fence_after();
            uint32_t o[32];
            const uint32_t ta = tmem + lane_off + TM_O + PA_GC * grp;
            tmem_ld32(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(ta, o);
          }
        }
        if (ok) {
          tmem_wait_st();
          fence_before();
          mbar_arrive(&p_full[st]);
        }
      }
      // Epilogue: the row's sum from all groups, O / l as bf16, this group's 32 value dims.
      const int par = r & 1;
      if (ok) ok = mbar_wait(&v_empty[(u - 1) & 1], ((u - 1) >> 1) & 1, err, abort_flag);
      if (!ok) s_fail[par] = 1;
      lx[(par * PA_NG + grp) * 128 + row] = l;
      named_bar(1, PA_SM_THREADS);
      if (s_fail[par]) break;
      fence_after();
      float lrow = 0.f;
#pragma unroll
      for (int g = 0; g < PA_NG; ++g) lrow += lx[(par * PA_NG + g) * 128 + row];
      const float inv = (lrow > 0.f) ? 1.f / lrow : 0.f;
      uint32_t o[32];
      tmem_ld32(tmem + lane_off + TM_O + PA_GC * grp, o);
      tmem_wait_ld();  // the next item's first MMA2 may overwrite O once every thread is here
      const size_t at = (size_t)(it.b * T + qi) * O_IN + it.h * VDIM + PA_GC * grp;
      if (o_hi == nullptr) {
        if (qi < T) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v;
            uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int f = 0; f < 4; ++f) {
              __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(o[e + 2 * f]) * inv,
                                                        __uint_as_float(o[e + 2 * f + 1]) * inv);
              w[f] = *reinterpret_cast<uint32_t*>(&pr);
            }
            *reinterpret_cast<uint4*>(attn_out + at + e) = v;
          }
        }
      } else {
        // The bf16 output values, split into two e4m3 terms with one scale per (token, head):
        // s = amax over the head's 128 values / 448 (the four threads of the row trade their
        // maxima), hi = e4m3(v / s), lo = e4m3(v / s - hi).
        float v[32];
        float am = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          v[e] = __bfloat162float(__float2bfloat16_rn(__uint_as_float(o[e]) * inv));
          am = fmaxf(am, fabsf(v[e]));
        }
        ax[(par * PA_NG + grp) * 128 + row] = am;
        named_bar(1, PA_SM_THREADS);
        float amax = 0.f;
#pragma unroll
        for (int g = 0; g < PA_NG; ++g) amax = fmaxf(amax, ax[(par * PA_NG + g) * 128 + row]);
        const float sc = amax > 0.f ? amax / 448.f : 1.f;
        const float is = 1.f / sc;
        if (qi < T) {
          uint32_t hw[8] = {}, lw[8] = {};
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t hl = e4m3_split2(make_float2(v[2 * e] * is, v[2 * e + 1] * is));
            hw[e >> 1] |= (hl & 0xFFFFu) << (16 * (e & 1));
            lw[e >> 1] |= (hl >> 16) << (16 * (e & 1));
          }
          uint4* dh = reinterpret_cast<uint4*>(o_hi + at);
          uint4* dl = reinterpret_cast<uint4*>(o_lo + at);
          dh[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          dh[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          dl[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          dl[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
          if (grp == 0) o_sx[(size_t)(it.b * T + qi) * HEADS + it.h] = sc;
        }
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

bool make_tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_tmap_2d(CUtensorMap* m, bool bf16, const void* base, uint64_t cols, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows);

cudaError_t init_prefill_tc_kernel() {
  return cudaFuncSetAttribute(prefill_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PA_SMEM);
}

cudaError_t launch_prefill_attention_tc(const __nv_bfloat16* q, const __nv_bfloat16* kv,
                                        const CacheRef& cache, int B, int T,
                                        const int* seq_lens, long kv_rows, float scale,
                                        __nv_bfloat16* attn_out, uint8_t* o_hi, uint8_t* o_lo,
                                        float* o_sx, int num_sms, int* err, cudaStream_t st,
                                        bool pdl) {
  if ((o_hi == nullptr) != (o_lo == nullptr) || (o_hi == nullptr) != (o_sx == nullptr) ||
      (o_hi == nullptr && attn_out == nullptr))
    return cudaErrorInvalidValue;
  if (B * T == 0) return cudaSuccess;
  const uint64_t M = (uint64_t)B * T;
  CUtensorMap mq, mkv, mc;
  if (!make_tmap_3d(&mq, q, QHEAD, HEADS, M, QHEAD * 2, (uint64_t)HEADS * QHEAD * 2, 64, 1, 128) ||
      !make_tmap_3d(&mkv, kv, KVB_PER_HEAD, HEADS, (uint64_t)kv_rows, KVB_PER_HEAD * 2,
                    (uint64_t)HEADS * KVB_PER_HEAD * 2, 64, 1, 128) ||
      !make_tmap_2d(&mc, true, cache.base, LAT, (uint64_t)cache.rows(B), LAT * 2, 64,
                    cache.paged() ? 64 : 128))
    return cudaErrorInvalidValue;
  if (cache.rows(B) + PA_TILE > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  // One persistent CTA per SM (at most one per work item), each taking its share of the
  // (head, query tile, sequence) items in turn.
  const long long items = (long long)HEADS * ((T + PA_TILE - 1) / PA_TILE) * B;
  if (items > 0x7FFFFFFFll || num_sms <= 0) return cudaErrorInvalidValue;
  const int grid = (int)(items < num_sms ? items : num_sms);
  return launch_kernel(prefill_attn_tc_kernel, dim3(grid), dim3(PA_THREADS), PA_SMEM, st, pdl, mq,
                       mkv, mc, T, cache, seq_lens, scale * 1.4426950408889634f, attn_out, o_hi,
                       o_lo, o_sx, kv_rows, (int)items, err);
}

}  // namespace mla
