// Log-sum-exp combine of the split-KV decode partials (the tensor-core decode attention writes
// one unnormalised partial output, maximum and sum per work item and head; maxima are in base
// 2, scores having been multiplied by scale*log2(e)).
#include "mla_internal.h"

namespace mla {

namespace {

// Combine of the split partials of sequence b, head h:
// o = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i, M = max_i m_i.
__global__ void __launch_bounds__(128) decode_combine_kernel(
    const int* __restrict__ seq_lens, int B, int chunk, int items, const float* __restrict__ o_part,
    const float* __restrict__ ml_part, __nv_bfloat16* __restrict__ o_lat, int* err) {
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  __shared__ int s_first, s_n;
  if (tid == 0) {
    int acc = 0;
    for (int bb = 0; bb < b; ++bb) acc += (seq_lens[bb] + 1 + chunk - 1) / chunk;
    int n = (seq_lens[b] + 1 + chunk - 1) / chunk;
    if (acc + n > items || n < 1) {  // device lengths disagree with the host schedule
      atomicExch(err, DEV_ERR_PLAN);
      n = 0;
    }
    s_first = acc;
    s_n = n;
  }
  __syncthreads();
  const int first = s_first, n = s_n;
  if (n == 0) return;
  float M = -INFINITY;
  for (int i = 0; i < n; ++i) M = fmaxf(M, ml_part[((size_t)(first + i) * HEADS + h) * 2]);
  float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int i = 0; i < n; ++i) {
    const size_t it = (size_t)(first + i) * HEADS + h;
    const float w = exp2f(ml_part[it * 2] - M);
    L = fmaf(w, ml_part[it * 2 + 1], L);
    const float4 v = *reinterpret_cast<const float4*>(o_part + it * KV_LORA + tid * 4);
    acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
    acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
  }
  const float inv = 1.f / L;
  __nv_bfloat16* dst = o_lat + ((size_t)b * HEADS + h) * KV_LORA + tid * 4;
#pragma unroll
  for (int c = 0; c < 4; ++c) dst[c] = __float2bfloat16_rn(acc[c] * inv);
}

}  // namespace

cudaError_t launch_decode_combine(const int* seq_lens, DecodePlan plan, const float* o_part,
                                  const float* ml_part, __nv_bfloat16* o_lat, int* err,
                                  cudaStream_t st) {
  if (plan.B == 0) return cudaSuccess;
  decode_combine_kernel<<<dim3(plan.B, HEADS), 128, 0, st>>>(seq_lens, plan.B, plan.chunk,
                                                             plan.items, o_part, ml_part, o_lat,
                                                             err);
  return cudaGetLastError();
}

}  // namespace mla
