// Log-sum-exp combine of the split-KV decode partials (the tensor-core decode attention writes
// one unnormalised partial output, maximum and sum per work item and head; maxima are in base
// 2, scores having been multiplied by scale*log2(e)).
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kMaxSplits = 512;   // shares one sequence can span (at most the CTA count)

// Combine of the partial outputs of sequence b, head h: the shares of CTAs c_first..c_last
// cover its positions and left partials in slots b + c;
// o = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i, M = max_i m_i.
// The per-share weights are formed once in shared memory; each thread then sums 4 columns with
// independent loads.
__global__ void __launch_bounds__(128) decode_combine_kernel(
    const int* __restrict__ seq_lens, int B, int G, long long P, const float* __restrict__ o_part,
    const float* __restrict__ ml_part, __nv_bfloat16* __restrict__ o_lat, int* err) {
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  __shared__ int s_first, s_n;
  __shared__ float s_w[kMaxSplits];
  __shared__ float s_red[8];
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
      atomicExch(err, DEV_ERR_PLAN);
      n = 0;
    }
    s_first = b + c0;  // slot of the first share
    s_n = n;
  }
  __syncthreads();
  const int first = s_first, n = s_n;
  if (n == 0) return;
  const int warp = tid >> 5, lane = tid & 31;
  float M = -INFINITY;
  for (int i = tid; i < n; i += 128) M = fmaxf(M, ml_part[((size_t)(first + i) * HEADS + h) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));
  float L = 0.f;
  for (int i = tid; i < n; i += 128) {
    const size_t it = (size_t)(first + i) * HEADS + h;
    const float w = exp2f(ml_part[it * 2] - M);
    s_w[i] = w;
    L = fmaf(w, ml_part[it * 2 + 1], L);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  if (lane == 0) s_red[4 + warp] = L;
  __syncthreads();
  L = (s_red[4] + s_red[5]) + (s_red[6] + s_red[7]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const float* op = o_part + ((size_t)first * HEADS + h) * KV_LORA + tid * 4;
  const size_t step = (size_t)HEADS * KV_LORA;
  int i = 0;
  for (; i + 4 <= n; i += 4) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4*>(op + (i + u) * step);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = s_w[i + u];
      acc[0] = fmaf(w, v[u].x, acc[0]); acc[1] = fmaf(w, v[u].y, acc[1]);
      acc[2] = fmaf(w, v[u].z, acc[2]); acc[3] = fmaf(w, v[u].w, acc[3]);
    }
  }
  for (; i < n; ++i) {
    const float4 v = *reinterpret_cast<const float4*>(op + i * step);
    const float w = s_w[i];
    acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
    acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
  }
  const float inv = 1.f / L;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(o_lat + ((size_t)b * HEADS + h) * KV_LORA + tid * 4) = pk;
}

}  // namespace

cudaError_t launch_decode_combine(const int* seq_lens, DecodePlan plan, const float* o_part,
                                  const float* ml_part, __nv_bfloat16* o_lat, int* err,
                                  cudaStream_t st, bool pdl) {
  if (plan.B == 0) return cudaSuccess;
  return launch_kernel(decode_combine_kernel, dim3(plan.B, HEADS), dim3(128), 0, st, pdl,
                       seq_lens, plan.B, plan.G, plan.P, o_part, ml_part, o_lat, err);
}

}  // namespace mla
