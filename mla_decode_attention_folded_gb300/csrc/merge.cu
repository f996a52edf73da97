// LSE merge of S partial decode results over disjoint key sets of the same
// rows: the combine the drafter-attention page's `DraftDcp` runs across decode-
// context-parallel shards (each shard decodes its local KV, then every row is
// merged over the shards by exp2(lse - max) / sum in FP32 with one BF16
// rounding). Here the S sources sit in one device buffer; moving them between
// GPUs is the caller's transport.
//   w_s = 2^(lse_s - max_s lse_s), out = sum_s w_s out_s / sum_s w_s,
//   lse = max + log2 sum_s w_s; rows whose sources are all empty: 0 and -inf.
// One warp per row; each lane owns 16 of the 512 dims; lanes hold 32 sources'
// LSEs at a time and share weights by shuffles.
#include "internal.h"
#include "ptx.cuh"

namespace mlafold {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(kWarps * 32)
lse_merge_kernel(int S, int rows, const uint16_t* __restrict__ parts_out,
                 const float* __restrict__ parts_lse, uint16_t* __restrict__ out,
                 float* __restrict__ lse) {
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  for (long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); row < rows;
       row += (long long)gridDim.x * kWarps) {
    float mx = -INFINITY;
    for (int c0 = 0; c0 < S; c0 += 32)
      if (c0 + lane < S) mx = fmaxf(mx, parts_lse[(long long)(c0 + lane) * rows + row]);
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    float z = 0.f;
    for (int c0 = 0; c0 < S; c0 += 32) {
      const float lc = c0 + lane < S ? parts_lse[(long long)(c0 + lane) * rows + row] : -INFINITY;
      const float wc = (mx == -INFINITY || lc == -INFINITY) ? 0.f : ex2(lc - mx);
      z += wc;
      const int cn = min(32, S - c0);
      for (int s = 0; s < cn; ++s) {
        const float w = __shfl_sync(0xffffffffu, wc, s);
        if (w == 0.f) continue;                      // warp-uniform
        const uint4* src = reinterpret_cast<const uint4*>(
            parts_out + ((long long)(c0 + s) * rows + row) * kDv + lane * 16);
        float f[16];
        bf16x8_to_f32(src[0], f);
        bf16x8_to_f32(src[1], f + 8);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] += w * f[i];
      }
    }
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv = z > 0.f ? 1.f / z : 0.f;
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      pk[i] = (uint32_t)f32_to_bf16_bits(acc[2 * i] * inv) |
              ((uint32_t)f32_to_bf16_bits(acc[2 * i + 1] * inv) << 16);
    uint4* dst = reinterpret_cast<uint4*>(out + row * kDv + lane * 16);
    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    if (lse && lane == 0) lse[row] = z > 0.f ? mx + __log2f(z) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_lse_merge(int S, int rows, const uint16_t* parts_out, const float* parts_lse,
                             uint16_t* out, float* lse, cudaStream_t st) {
  long long blocks = cdiv(rows, kWarps);
  if (blocks > 4096) blocks = 4096;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel, S, rows, parts_out, parts_lse, out, lse);
}

}  // namespace mlafold
