// Attention on the CUDA cores: split-KV absorbed decode over the latent cache with its
// log-sum-exp combine, and causal flash-style prefill.
//
// Scores follow the `mla-prefill` excerpt ("Key content up-projection" page): q.k times the
// softmax scale, the causal mask, a float32 softmax over keys and the value contraction.
// Softmax runs online in base 2: scores are multiplied by scale*log2(e) and exponentiated with
// exp2f, which is the same softmax.
#include "mla_internal.h"

namespace mla {

namespace {

constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b, float acc) {
  const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(__uint_as_float(ua[i] << 16), __uint_as_float(ub[i] << 16), acc);
    acc = fmaf(__uint_as_float(ua[i] & 0xFFFF0000u), __uint_as_float(ub[i] & 0xFFFF0000u), acc);
  }
  return acc;
}

// Locates work item `item` in the concatenation of per-sequence splits: sequence b owns
// ceil((seq_lens[b] + 1) / chunk) consecutive items.  Returns b (or -1) and the item index
// within b; `first` receives b's first item.
__device__ int find_item(const int* seq_lens, int B, int chunk, int item, int* local, int* first) {
  int acc = 0;
  for (int b = 0; b < B; ++b) {
    const int n = (seq_lens[b] + 1 + chunk - 1) / chunk;
    if (item < acc + n) {
      *local = item - acc;
      *first = acc;
      return b;
    }
    acc += n;
  }
  return -1;
}

// ---------------------------------------------------------------------------- decode
constexpr int DT = 32;          // cached positions per tile
constexpr int QS = LAT + 8;     // padded smem row (bank spread)

constexpr int HG = 16;           // heads per CTA (4 CTAs share each work item)

// CTA (g, item): heads [16 g, 16 g + 16) over positions [i*chunk, min(S_b, (i+1)*chunk)) of
// sequence b, S_b = seq_lens[b] + 1 (the new token's row is already stored).  Thread
// t = 16 hl + u handles head 16 g + hl: scores of positions 2u, 2u+1 of each 32-position tile,
// and output columns [32 u, 32 u + 32).
// scores s_h(j) = qfull[b,h] . cache[b,j]  (576 = 512 latent + 64 rotary)
// partial o_h = sum_j exp2(s_h(j)*c - m_h) cache[b, j, 0:512],  l_h = sum_j exp2(...).
__global__ void __launch_bounds__(256) decode_attn_simt_kernel(
    const __nv_bfloat16* __restrict__ qfull, const __nv_bfloat16* __restrict__ cache, int cap,
    const int* __restrict__ seq_lens, int B, int chunk, float scale_log2,
    float* __restrict__ o_part, float* __restrict__ ml_part, int* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* Cs = Qs + HG * QS;
  float* Ps = reinterpret_cast<float*>(Cs + DT * QS);
  __shared__ int s_b, s_i;
  const int tid = threadIdx.x, hl = tid >> 4, u = tid & 15;
  const int g = blockIdx.x, item = blockIdx.y, h = g * HG + hl;
  if (tid == 0) {
    int first;
    s_b = find_item(seq_lens, B, chunk, item, &s_i, &first);
    if (s_b < 0) atomicExch(err, DEV_ERR_PLAN);
  }
  __syncthreads();
  const int b = s_b;
  if (b < 0) return;
  const int S = seq_lens[b] + 1;
  const int p0 = s_i * chunk, p1 = min(S, p0 + chunk);
  if (S > cap) {
    if (tid == 0) atomicExch(err, DEV_ERR_RANGE);
    return;
  }
  for (int e = tid; e < HG * (LAT / 8); e += 256) {
    const int r = e / (LAT / 8), c = e % (LAT / 8);
    reinterpret_cast<uint4*>(Qs + r * QS)[c] =
        reinterpret_cast<const uint4*>(qfull + ((size_t)b * HEADS + g * HG + r) * LAT)[c];
  }
  float o[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) o[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  const __nv_bfloat16* cb = cache + (size_t)b * cap * LAT;

  for (int p = p0; p < p1; p += DT) {
    const int n = min(DT, p1 - p);
    __syncthreads();
    for (int e = tid; e < DT * (LAT / 8); e += 256) {
      const int r = e / (LAT / 8), c = e % (LAT / 8);
      reinterpret_cast<uint4*>(Cs + r * QS)[c] =
          r < n ? reinterpret_cast<const uint4*>(cb + (size_t)(p + r) * LAT)[c] : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    float s0 = 0.f, s1 = 0.f;
    const uint4* qrow = reinterpret_cast<const uint4*>(Qs + hl * QS);
    const uint4* c0 = reinterpret_cast<const uint4*>(Cs + (2 * u) * QS);
    const uint4* c1 = reinterpret_cast<const uint4*>(Cs + (2 * u + 1) * QS);
#pragma unroll 4
    for (int k = 0; k < LAT / 8; ++k) {
      const uint4 qv = qrow[k];
      s0 = dot8_bf16(qv, c0[k], s0);
      s1 = dot8_bf16(qv, c1[k], s1);
    }
    s0 = (2 * u < n) ? s0 * scale_log2 : -INFINITY;
    s1 = (2 * u + 1 < n) ? s1 * scale_log2 : -INFINITY;
    float tmax = fmaxf(s0, s1);
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m, tmax);
    const float alpha = exp2f(m - m_new);
    const float p0v = exp2f(s0 - m_new), p1v = exp2f(s1 - m_new);
    float lsum = p0v + p1v;
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    Ps[hl * DT + 2 * u] = p0v;
    Ps[hl * DT + 2 * u + 1] = p1v;
    l = l * alpha + lsum;
    m = m_new;
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 32; ++c) o[c] *= alpha;
    for (int j = 0; j < n; ++j) {
      const float pj = Ps[hl * DT + j];
      const uint4* crow = reinterpret_cast<const uint4*>(Cs + j * QS + u * 32);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const uint4 v = crow[c8];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[c8 * 8 + 2 * i] = fmaf(pj, __uint_as_float(w[i] << 16), o[c8 * 8 + 2 * i]);
          o[c8 * 8 + 2 * i + 1] = fmaf(pj, __uint_as_float(w[i] & 0xFFFF0000u), o[c8 * 8 + 2 * i + 1]);
        }
      }
    }
  }
  float* op = o_part + ((size_t)item * HEADS + h) * KV_LORA + u * 32;
#pragma unroll
  for (int c = 0; c < 32; c += 4)
    *reinterpret_cast<float4*>(op + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
  if (u == 0) {
    ml_part[((size_t)item * HEADS + h) * 2] = m;
    ml_part[((size_t)item * HEADS + h) * 2 + 1] = l;
  }
}

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

// ---------------------------------------------------------------------------- prefill
constexpr int PT = 64;            // queries and keys per tile
constexpr int KS = QHEAD + 8;     // padded rows
constexpr int VS = VDIM + 8;

// One CTA (256 threads) per (query tile, head, sequence).  Thread t = 4r + q: query row r,
// score columns [16q, 16q + 16), output columns [32q, 32q + 32).
// Keys of head h: [k_nope (kv[., h, 0:128]) | rotated k_pe (cache row [512:576])];
// values kv[., h, 128:256].  Key s is visible from query t iff s <= t.
__global__ void __launch_bounds__(256) prefill_attn_simt_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv,
    const __nv_bfloat16* __restrict__ cache, int cap, int T, float scale_log2,
    __nv_bfloat16* __restrict__ attn_out) {
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* Ks = Qs + PT * KS;
  __nv_bfloat16* Vs = Ks + PT * KS;
  float (*Ps)[PT + 1] = reinterpret_cast<float (*)[PT + 1]>(Vs + PT * VS);
  const int q0 = blockIdx.x * PT, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, r = tid >> 2, qq = tid & 3;
  const size_t tok0 = (size_t)b * T;

  for (int e = tid; e < PT * (QHEAD / 8); e += 256) {
    const int rr = e / (QHEAD / 8), c = e % (QHEAD / 8);
    reinterpret_cast<uint4*>(Qs + rr * KS)[c] = (q0 + rr < T)
        ? reinterpret_cast<const uint4*>(q + ((tok0 + q0 + rr) * HEADS + h) * QHEAD)[c]
        : make_uint4(0, 0, 0, 0);
  }
  float o[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) o[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int qrow = q0 + r;
  const int kend = min(T, q0 + PT);

  for (int k0 = 0; k0 < kend; k0 += PT) {
    __syncthreads();
    for (int e = tid; e < PT * (QHEAD / 8); e += 256) {
      const int rr = e / (QHEAD / 8), c = e % (QHEAD / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (k0 + rr < T) {
        v = (c < NOPE / 8)
            ? reinterpret_cast<const uint4*>(kv + ((tok0 + k0 + rr) * HEADS + h) * KVB_PER_HEAD)[c]
            : reinterpret_cast<const uint4*>(cache + ((size_t)b * cap + k0 + rr) * LAT + KV_LORA)[c - NOPE / 8];
      }
      reinterpret_cast<uint4*>(Ks + rr * KS)[c] = v;
    }
    for (int e = tid; e < PT * (VDIM / 8); e += 256) {
      const int rr = e / (VDIM / 8), c = e % (VDIM / 8);
      reinterpret_cast<uint4*>(Vs + rr * VS)[c] = (k0 + rr < T)
          ? reinterpret_cast<const uint4*>(kv + ((tok0 + k0 + rr) * HEADS + h) * KVB_PER_HEAD + NOPE)[c]
          : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    float s[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) s[jj] = 0.f;
    for (int k = 0; k < QHEAD / 8; ++k) {
      const uint4 qv = reinterpret_cast<const uint4*>(Qs + r * KS)[k];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        s[jj] = dot8_bf16(qv, reinterpret_cast<const uint4*>(Ks + (qq * 16 + jj) * KS)[k], s[jj]);
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int key = k0 + qq * 16 + jj;
      s[jj] = (key <= qrow && key < T) ? s[jj] * scale_log2 : -INFINITY;
      tmax = fmaxf(tmax, s[jj]);
    }
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float m_new = fmaxf(m, tmax);
    // Rows past T see no key at all; keep them finite (they are not stored).
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = exp2f(m - m_use);
    float lsum = 0.f;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const float pj = exp2f(s[jj] - m_use);
      lsum += pj;
      Ps[r][qq * 16 + jj] = pj;
    }
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    l = l * alpha + lsum;
    m = m_new;
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 32; ++c) o[c] *= alpha;
    for (int j = 0; j < PT; ++j) {
      const float pj = Ps[r][j];
      const uint4* vrow = reinterpret_cast<const uint4*>(Vs + j * VS + qq * 32);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const uint4 v = vrow[c8];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[c8 * 8 + 2 * i] = fmaf(pj, __uint_as_float(u[i] << 16), o[c8 * 8 + 2 * i]);
          o[c8 * 8 + 2 * i + 1] = fmaf(pj, __uint_as_float(u[i] & 0xFFFF0000u), o[c8 * 8 + 2 * i + 1]);
        }
      }
    }
  }
  if (qrow < T) {
    const float inv = 1.f / l;
    __nv_bfloat16* dst = attn_out + (tok0 + qrow) * O_IN + h * VDIM + qq * 32;
#pragma unroll
    for (int c = 0; c < 32; c += 8) {
      uint4 v;
      uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 pr = __floats2bfloat162_rn(o[c + 2 * i] * inv, o[c + 2 * i + 1] * inv);
        u[i] = *reinterpret_cast<uint32_t*>(&pr);
      }
      *reinterpret_cast<uint4*>(dst + c) = v;
    }
  }
}

}  // namespace

constexpr size_t kDecodeSmem =
    (size_t)(HG + DT) * QS * sizeof(__nv_bfloat16) + HG * DT * sizeof(float);
constexpr size_t kPrefillSmem =
    (size_t)PT * (2 * KS + VS) * sizeof(__nv_bfloat16) + PT * (PT + 1) * sizeof(float);

cudaError_t init_attention_kernels() {
  cudaError_t e = cudaFuncSetAttribute(decode_attn_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecodeSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_attn_simt_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrefillSmem);
}

cudaError_t launch_decode_attention(const __nv_bfloat16* qfull, const __nv_bfloat16* cache,
                                    int cap, const int* seq_lens, DecodePlan plan, float scale,
                                    float* o_part, float* ml_part, int* err, cudaStream_t st) {
  if (plan.B == 0) return cudaSuccess;
  decode_attn_simt_kernel<<<dim3(HEADS / HG, plan.items), 256, kDecodeSmem, st>>>(
      qfull, cache, cap, seq_lens, plan.B, plan.chunk, scale * LOG2E, o_part, ml_part, err);
  return cudaGetLastError();
}

cudaError_t launch_decode_combine(const int* seq_lens, DecodePlan plan, const float* o_part,
                                  const float* ml_part, __nv_bfloat16* o_lat, int* err,
                                  cudaStream_t st) {
  if (plan.B == 0) return cudaSuccess;
  decode_combine_kernel<<<dim3(plan.B, HEADS), 128, 0, st>>>(seq_lens, plan.B, plan.chunk,
                                                             plan.items, o_part, ml_part, o_lat,
                                                             err);
  return cudaGetLastError();
}

cudaError_t launch_prefill_attention(const __nv_bfloat16* q, const __nv_bfloat16* kv,
                                     const __nv_bfloat16* cache, int cap, int B, int T,
                                     float scale, __nv_bfloat16* attn_out, cudaStream_t st) {
  if (B * T == 0) return cudaSuccess;
  const dim3 grid((T + PT - 1) / PT, HEADS, B);
  prefill_attn_simt_kernel<<<grid, 256, kPrefillSmem, st>>>(q, kv, cache, cap, T, scale * LOG2E,
                                                            attn_out);
  return cudaGetLastError();
}

}  // namespace mla
