// Log-sum-exp combine of the split-KV decode partials (the tensor-core decode attention writes
// one normalised partial output [dim][head] in fp16, maximum and sum per work item and head;
// maxima are in base 2, scores having been multiplied by scale*log2(e)).
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kMaxSplits = kMaxDecodeShares;  // shares one sequence can span
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
    const int* __restrict__ seq_lens, int B, int G, long long P,
    const __half* __restrict__ o_part, const float* __restrict__ ml_part,
    __nv_bfloat16* __restrict__ o_lat, int* err) {
  const int b = blockIdx.x, tid = threadIdx.x;
  __shared__ int s_first, s_n;
  __shared__ float s_w[kMaxSplits * HEADS];
  __shared__ float s_red[4][HEADS];
  pdl_launch_dependents();
  pdl_wait();
  if (tid == 0) {
    long long start = 0;
    for (int bb = 0; bb < b; ++bb) start += (long long)seq_lens[bb] + 1;
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
    for (int i = g; i < n; i += 4) M = fmaxf(M, ml_part[((size_t)(first + i) * HEADS + h) * 2]);
    s_red[g][h] = M;
    __syncthreads();
    M = fmaxf(fmaxf(s_red[0][h], s_red[1][h]), fmaxf(s_red[2][h], s_red[3][h]));
    __syncthreads();
    float L = 0.f;
    for (int i = g; i < n; i += 4) {
      const size_t it = (size_t)(first + i) * HEADS + h;
      const float wl = exp2f(ml_part[it * 2] - M) * ml_part[it * 2 + 1];
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
      const float2 v = __half22float2(oi[e * (HEADS / 2)]);
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

}  // namespace

cudaError_t launch_decode_combine(const int* seq_lens, DecodePlan plan, const __half* o_part,
                                  const float* ml_part, __nv_bfloat16* o_lat, int* err,
                                  cudaStream_t st, bool pdl) {
  if (plan.B == 0) return cudaSuccess;
  return launch_kernel(decode_combine_kernel, dim3(plan.B, KV_LORA / kDims), dim3(kThreads), 0,
                       st, pdl, seq_lens, plan.B, plan.G, plan.P, o_part, ml_part, o_lat, err);
}

}  // namespace mla
