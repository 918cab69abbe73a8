// Log-sum-exp combine of the split-KV decode partials (the tensor-core decode attention writes
// one normalised partial output [dim][head] in fp16, maximum and sum per work item and head;
// maxima are in base 2, scores having been multiplied by scale*log2(e)).
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kMaxSplits = kMaxDecodeShares;  // shares one sequence can span

// A half2 partial written by the attention kernel, as two floats.
__device__ __forceinline__ float2 half2_dep(const __half2* p) {
  const uint32_t u = ld_dep_u32(p);
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}
constexpr int kDims = 32;                       // latent dims per CTA
constexpr int kThreads = 256;

// Combine of the partials of sequence b for latent dims [32 y, 32 y + 32) of all heads: the
// shares of CTAs c_first..c_last cover its positions and left, in slots b + c, the normalised
// partial o_i = O_i / l_i with its maximum m_i and sum l_i (per head); then
//   o = sum_i v_i o_i,  v_i = 2^(m_i - M) l_i / sum_j 2^(m_j - M) l_j,  M = max_i m_i.
// The weights v_i of every head are formed once in shared memory by four groups of 64 threads
// (one thread per head, each group every fourth share).  Partials are fp16 [slot][dim][head]:
// a thread then owns two heads and four dims, so a warp reads 128 contiguous bytes per dim.
__global__ void __launch_bounds__(kThreads) decode_combine_kernel(
    const int* __restrict__ seq_lens, int B, int G, long long P, int K,
    const __half* o_part, const float* ml_part,
    __nv_bfloat16* __restrict__ o_lat, int* err) {
  const int b = blockIdx.x, tid = threadIdx.x;
  __shared__ int s_first, s_n;
  __shared__ float s_w[kMaxSplits * HEADS];
  __shared__ float s_red[4][HEADS];
  pdl_launch_dependents();
  pdl_wait();
  if (tid == 0) {
    long long start = K;  // line position of sequence b's position 0
    for (int bb = 0; bb < b; ++bb) start += (long long)seq_lens[bb] + 1 + K;
    const long long end = start + seq_lens[b] + 1;
    int c0 = 0, n = 0;
    if (end <= P) {
      c0 = decode_share_of(start, G, P);
      n = decode_share_of(end - 1, G, P) - c0 + 1;
    }
    if (n < 1 || n > kMaxSplits) {  // device lengths disagree with the host schedule
      if (blockIdx.y == 0) atomicExch(err, DEV_ERR_PLAN);
      n = 0;
    }
    s_first = b + c0;  // slot of the first share
    s_n = n;
  }
  __syncthreads();
  const int first = s_first, n = s_n;
  if (n == 0) return;
  {
    const int h = tid & (HEADS - 1), g = tid >> 6;
    float M = -INFINITY;
    for (int i = g; i < n; i += 4) M = fmaxf(M, ld_dep_f32(ml_part + ((size_t)(first + i) * HEADS + h) * 2));
    s_red[g][h] = M;
    __syncthreads();
    M = fmaxf(fmaxf(s_red[0][h], s_red[1][h]), fmaxf(s_red[2][h], s_red[3][h]));
    __syncthreads();
    float L = 0.f;
    for (int i = g; i < n; i += 4) {
      const size_t it = (size_t)(first + i) * HEADS + h;
      const float2 v = ld_dep_f32x2(ml_part + it * 2);
      const float wl = exp2f(v.x - M) * v.y;
      s_w[i * HEADS + h] = wl;
      L += wl;
    }
    s_red[g][h] = L;
    __syncthreads();
    const float inv = 1.f / ((s_red[0][h] + s_red[1][h]) + (s_red[2][h] + s_red[3][h]));
    for (int i = g; i < n; i += 4) s_w[i * HEADS + h] *= inv;
    __syncthreads();
  }
  // This thread: heads 2 hp, 2 hp + 1 and dims d0 .. d0 + 3.
  const int hp = tid & 31, d0 = kDims * blockIdx.y + 4 * (tid >> 5);
  const __half2* op = reinterpret_cast<const __half2*>(o_part + (size_t)first * KV_LORA * HEADS +
                                                       (size_t)d0 * HEADS) + hp;
  const size_t step = (size_t)KV_LORA * HEADS / 2;  // one slot, in half2
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 2
  for (int i = 0; i < n; ++i) {
    const float w0 = s_w[i * HEADS + 2 * hp], w1 = s_w[i * HEADS + 2 * hp + 1];
    const __half2* oi = op + i * step;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t u = ld_dep_u32(oi + e * (HEADS / 2));
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&u));
      acc[0][e] = fmaf(w0, v.x, acc[0][e]);
      acc[1][e] = fmaf(w1, v.y, acc[1][e]);
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k][0], acc[k][1]);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k][2], acc[k][3]);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(o_lat + ((size_t)b * HEADS + 2 * hp + k) * KV_LORA + d0) = pk;
  }
}

// Combine and output absorption for a few decode sequences, CTA (h, vb, b) for head h, rows
// 32 vb .. 32 vb + 31 of W_UV,h and sequence b:
//   o_lat = sum_i v_i o_i as in decode_combine_kernel (rounded to bf16), then
//   attn[b][128 h + v] = sum_c s[2h+1][c/128] * e4m3(W_kvb[256 h + 128 + v][c]) * o_lat[c]
// ("Key content up-projection" page, W_UV,h = rows 128..255 of head h's 256).  The partials
// are head-major ([slot][head][dim], fp16), so the 1 KB of head h in each share is one
// contiguous read; each of the four CTAs of a head merges them again (from L2) rather than
// wait for one another.  Each warp owns 4 rows of W_UV,h, loaded into registers before the
// wait on the attention.  The share ranges come from the host's plan (and the device length is
// checked against it), and every load after the wait is issued at once: the work after the
// attention is one memory round trip.
struct ShareRanges {
  int first[8], n[8], len[8];  // slot of the first share, number of shares, length (host)
};
constexpr int CAO_BATCH = 16;  // shares per round of loads
constexpr int CAO_SPLIT = 4;   // CTAs per (head, sequence)
constexpr int CAO_ROWS = VDIM / CAO_SPLIT / 8;  // rows of W_UV,h per warp

__global__ void __launch_bounds__(256) combine_absorb_out_kernel(
    const int* __restrict__ seq_lens, const __grid_constant__ ShareRanges sr,
    const __half* o_part, const float* ml_part,
    const uint8_t* __restrict__ Wkvb, const float* __restrict__ Skvb,
    __nv_bfloat16* __restrict__ attn, int* err) {
  const int h = blockIdx.x, vb = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int v0 = VDIM / CAO_SPLIT * vb + CAO_ROWS * warp;  // this warp's first row
  __shared__ float s_w[kMaxSplits];
  __shared__ float s_red[8];
  __shared__ __align__(16) float ol[KV_LORA];
  uint4 wv[CAO_ROWS];
#pragma unroll
  for (int r = 0; r < CAO_ROWS; ++r) {
    const uint8_t* src =
        Wkvb + ((size_t)h * KVB_PER_HEAD + NOPE + v0 + r) * KV_LORA + lane * 16;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(wv[r].x), "=r"(wv[r].y), "=r"(wv[r].z), "=r"(wv[r].w)
                 : "l"(src));
  }
  const float sc = __ldg(Skvb + (size_t)(2 * h + 1) * (KV_LORA / BLK) + lane / 8);
  const int first = sr.first[b], n = sr.n[b];
  pdl_launch_dependents();
  pdl_wait();  // the attention's partials are complete
  // Loads first: (m, l) of share tid, and this thread's dims 2 tid, 2 tid + 1 of the first
  // shares.
  const bool own = tid < n;
  float mi = -INFINITY, li = 0.f;
  if (own) {
    const float2 v = ld_dep_f32x2(ml_part + ((size_t)(first + tid) * HEADS + h) * 2);
    mi = v.x;
    li = v.y;
  }
  const __half2* op = reinterpret_cast<const __half2*>(o_part + ((size_t)first * HEADS + h) * KV_LORA) + tid;
  constexpr size_t kSlot = (size_t)HEADS * KV_LORA / 2;  // one slot, in half2
  float2 pv[CAO_BATCH];
#pragma unroll
  for (int k = 0; k < CAO_BATCH; ++k)
    pv[k] = k < n ? half2_dep(op + k * kSlot) : make_float2(0.f, 0.f);
  if (tid == 0 && h == 0 && vb == 0 && seq_lens[b] != sr.len[b])  // lengths disagree with the plan
    atomicExch(err, DEV_ERR_PLAN);
  // v_i = 2^(m_i - M) l_i / sum_j 2^(m_j - M) l_j  (n <= 256: one share per thread)
  float M = mi;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();
  M = s_red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) M = fmaxf(M, s_red[w]);
  __syncthreads();
  const float wl = own ? exp2f(mi - M) * li : 0.f;
  float L = wl;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  if (lane == 0) s_red[warp] = L;
  __syncthreads();
  L = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) L += s_red[w];
  if (own) s_w[tid] = wl / L;
  __syncthreads();
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int k = 0; k < CAO_BATCH; ++k)
    if (k < n) {
      a0 = fmaf(s_w[k], pv[k].x, a0);
      a1 = fmaf(s_w[k], pv[k].y, a1);
    }
  for (int i0 = CAO_BATCH; i0 < n; i0 += CAO_BATCH) {  // long contexts: more rounds
#pragma unroll
    for (int k = 0; k < CAO_BATCH; ++k)
      pv[k] = i0 + k < n ? half2_dep(op + (i0 + k) * kSlot) : make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < CAO_BATCH; ++k)
      if (i0 + k < n) {
        a0 = fmaf(s_w[i0 + k], pv[k].x, a0);
        a1 = fmaf(s_w[i0 + k], pv[k].y, a1);
      }
  }
  ol[2 * tid] = __bfloat162float(__float2bfloat16_rn(a0));
  ol[2 * tid + 1] = __bfloat162float(__float2bfloat16_rn(a1));
  __syncthreads();
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = ol[lane * 16 + i];
#pragma unroll
  for (int r = 0; r < CAO_ROWS; ++r) {
    const uint32_t u[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
    float p = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(u[q] & 0xFFFF), __NV_E4M3);
      __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(u[q] >> 16), __NV_E4M3);
      const float2 fa = __half22float2(*reinterpret_cast<__half2*>(&lo));
      const float2 fb = __half22float2(*reinterpret_cast<__half2*>(&hi));
      p = fmaf(fa.x, x[4 * q], p);
      p = fmaf(fa.y, x[4 * q + 1], p);
      p = fmaf(fb.x, x[4 * q + 2], p);
      p = fmaf(fb.y, x[4 * q + 3], p);
    }
    float t = sc * p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    if (lane == 0) attn[(size_t)b * O_IN + h * VDIM + v0 + r] = __float2bfloat16_rn(t);
  }
}

}  // namespace

cudaError_t launch_combine_absorb_out(const int* seq_lens, const int* lens_host,
                                      DecodePlan plan, const __half* o_part,
                                      const float* ml_part, const uint8_t* Wkvb,
                                      const float* Skvb, __nv_bfloat16* attn, int* err,
                                      cudaStream_t st, bool pdl) {
  if (plan.B == 0) return cudaSuccess;
  if (plan.B > 8) return cudaErrorInvalidValue;
  ShareRanges sr{};
  long long start = plan.K;  // line position of sequence b's position 0
  for (int b = 0; b < plan.B; ++b) {
    const long long end = start + lens_host[b] + 1;
    const int c0 = decode_share_of(start, plan.G, plan.P);
    sr.first[b] = b + c0;
    sr.n[b] = decode_share_of(end - 1, plan.G, plan.P) - c0 + 1;
    sr.len[b] = lens_host[b];
    if (sr.n[b] < 1 || sr.n[b] > kMaxSplits) return cudaErrorInvalidValue;
    start = end + plan.K;
  }
  return launch_kernel(combine_absorb_out_kernel, dim3(HEADS, CAO_SPLIT, plan.B), dim3(256), 0, st, pdl,
                       seq_lens, sr, o_part, ml_part, Wkvb, Skvb, attn, err);
}

cudaError_t launch_decode_combine(const int* seq_lens, DecodePlan plan, const __half* o_part,
                                  const float* ml_part, __nv_bfloat16* o_lat, int* err,
                                  cudaStream_t st, bool pdl) {
  if (plan.B == 0) return cudaSuccess;
  return launch_kernel(decode_combine_kernel, dim3(plan.B, KV_LORA / kDims), dim3(kThreads), 0,
                       st, pdl, seq_lens, plan.B, plan.G, plan.P, plan.K, o_part, ml_part, o_lat,
                       err);
}

}  // namespace mla
