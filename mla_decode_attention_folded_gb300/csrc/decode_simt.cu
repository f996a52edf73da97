// Split-KV decode on CUDA cores: one CTA per (work item, 32-row block).
//
// Same numerics contract as the header states for mla_folded_decode: FP32
// scores, base-2 online softmax whose running max is kept while a new score
// exceeds it by at most 8, P as the sum of two E4M3 terms, FP32 normaliser.
// Each key page (64 keys x 576 bytes) is staged in shared memory.
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace mlafold {
namespace {

constexpr int kRows = 32;
constexpr int kThreads = 256;

__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

__device__ __forceinline__ float round_e4m3(float x) {
  return e4m3_to_f32((uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

struct __align__(16) SimtSmem {
  uint8_t q[kRows][kDqk];
  uint8_t k[kPage][kDqk];
  float s[kRows][kPage + 1];
  float m[kRows], l[kRows], alpha[kRows];
};

__global__ void __launch_bounds__(kThreads)
decode_simt_kernel(const DecodeArgs a, int nb) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
  auto& s_q = sm.q;
  auto& s_k = sm.k;
  auto& s_s = sm.s;
  auto& s_m = sm.m;
  auto& s_l = sm.l;
  auto& s_alpha = sm.alpha;

  grid_dep_wait();
  const int item = blockIdx.x / nb, blk = blockIdx.x % nb;
  if (item >= a.list_len) return;
  const int e = a.work[item];
  if (e < 0) return;
  const int r = e >> kSplitBits, s = e & ((1 << kSplitBits) - 1);
  if (r >= a.R || s >= a.counts[r]) {
    if (a.status && threadIdx.x == 0) atomicOr(a.status, MLA_FAULT_WORK_ITEM);
    return;
  }
  const int n = a.counts[r];
  int L = max(a.seq_lens[r], 0);
  if (L > a.max_pages * kPage) {           // never read past the block-table row
    if (a.status && threadIdx.x == 0) atomicOr(a.status, MLA_FAULT_PAGE_RANGE);
    L = a.max_pages * kPage;
  }
  int j0, j1;
  split_range(L, n, s, j0, j1);
  const int m0 = blk * kRows;
  const int t = threadIdx.x;

  // Query rows of this block (rows past M are zero).
  for (int idx = t; idx < kRows * kDqk / 16; idx += kThreads) {
    const int row = idx / (kDqk / 16), c16 = idx % (kDqk / 16);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (m0 + row < a.M)
      v = reinterpret_cast<const uint4*>(a.q + ((long long)r * a.M + m0 + row) * kDqk)[c16];
    reinterpret_cast<uint4*>(&s_q[row][0])[c16] = v;
  }
  if (t < kRows) { s_m[t] = -INFINITY; s_l[t] = 0.f; }

  float acc[kRows][2];
#pragma unroll
  for (int i = 0; i < kRows; ++i) acc[i][0] = acc[i][1] = 0.f;
  const int d0 = 2 * t;                     // this thread's two value dims

  for (int pj = j0; pj < j1; pj += kPage) {
    int page = a.block_table[(long long)r * a.max_pages + pj / kPage];
    const bool bad = page < 0 || page >= a.num_pages;
    if (bad && a.status && t == 0) atomicOr(a.status, MLA_FAULT_PAGE_RANGE);
    __syncthreads();
    for (int idx = t; idx < kPage * kDqk / 16; idx += kThreads) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (!bad) v = reinterpret_cast<const uint4*>(a.kv + (long long)page * kPage * kDqk)[idx];
      reinterpret_cast<uint4*>(&s_k[0][0])[idx] = v;
    }
    __syncthreads();
    // Scores: thread -> row t%32, keys (t/32)*8 .. +7.
    {
      const int row = t & 31, kg = t >> 5;
      for (int kk = 0; kk < 8; ++kk) {
        const int key = kg * 8 + kk;
        float dot = 0.f;
        for (int d = 0; d < kDqk; ++d) dot += e4m3_to_f32(s_q[row][d]) * e4m3_to_f32(s_k[key][d]);
        s_s[row][key] = (pj + key < j1) ? dot * a.bmm1_log2 : -INFINITY;
      }
    }
    __syncthreads();
    // Online softmax per row (lazy max, two-term E4M3 P).
    if (t < kRows) {
      float tmax = -INFINITY;
      for (int key = 0; key < kPage; ++key) tmax = fmaxf(tmax, s_s[t][key]);
      float m = s_m[t], alpha = 1.f;
      if (tmax > m + 8.f) {
        alpha = (m == -INFINITY) ? 0.f : ex2(m - tmax);
        m = tmax;
      }
      float l = s_l[t] * alpha;
      for (int key = 0; key < kPage; ++key) {
        const float x = s_s[t][key];
        const float p = (x == -INFINITY) ? 0.f : ex2(x - m);
        l += p;
        const float hi = round_e4m3(p);
        const float lo = round_e4m3(p - hi);
        s_s[t][key] = hi + lo;
      }
      s_m[t] = m; s_l[t] = l; s_alpha[t] = alpha;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      acc[i][0] *= s_alpha[i];
      acc[i][1] *= s_alpha[i];
    }
    for (int key = 0; key < kPage; ++key) {
      const float v0 = e4m3_to_f32(s_k[key][d0]), v1 = e4m3_to_f32(s_k[key][d0 + 1]);
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const float p = s_s[i][key];
        acc[i][0] += p * v0;
        acc[i][1] += p * v1;
      }
    }
  }
  __syncthreads();
  const bool direct = n == 1;
  if (!direct && item >= a.slots) {
    if (a.status && t == 0) atomicOr(a.status, MLA_FAULT_WORK_ITEM);
    return;
  }
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int m = m0 + i;
    if (m >= a.M) break;
    const float l = s_l[i];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse2 = l > 0.f ? s_m[i] + __log2f(l) : -INFINITY;
    if (direct) {
      const uint32_t packed = (uint32_t)f32_to_bf16_bits(acc[i][0] * inv * a.bmm2) |
                              ((uint32_t)f32_to_bf16_bits(acc[i][1] * inv * a.bmm2) << 16);
      *reinterpret_cast<uint32_t*>(a.out + ((long long)r * a.M + m) * kDv + d0) = packed;
      if (t == 0) a.lse[(long long)r * a.M + m] = lse2;
    } else {
      float2 v = make_float2(acc[i][0] * inv, acc[i][1] * inv);
      *reinterpret_cast<float2*>(a.part_o + ((long long)item * a.M + m) * kDv + d0) = v;
      if (t == 0) a.part_lse[(long long)item * a.M + m] = lse2;
    }
  }
  grid_dep_launch();
}

}  // namespace

cudaError_t launch_decode(const mla_shape& s, const DecodeArgs& a, cudaStream_t st) {
  const int nb = (a.M + kRows - 1) / kRows;
  cudaError_t err = cudaFuncSetAttribute(decode_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(SimtSmem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.dynamicSmemBytes = sizeof(SimtSmem);
  cfg.gridDim = dim3((unsigned)(a.list_len * nb));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_simt_kernel, a, nb);
}

}  // namespace mlafold
