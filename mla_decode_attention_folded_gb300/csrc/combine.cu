// Split-KV LSE reduction: FP32 partials of the multi-split requests -> BF16 out
// and base-2 LSE.
//
// Math (drafter-attention page, `DraftDcp`: the head owner merges partial rows
// by exp2(lse - max) / sum in FP32 with one BF16 rounding; balanced-MLA page,
// module overview: FP32 split partials with a log2 LSE):
//   mx = max_s lse_s, w_s = 2^(lse_s - mx), out = bmm2 * sum_s w_s O_s / sum_s w_s,
//   lse = mx + log2(sum_s w_s).
// One warp reduces one (request, row, band) of 512 / bands dims; the band
// count follows the pages' `reducer_d_tiles` rule (two D bands when the rows
// fill at most half of the SMs). Multi-split requests sit at the front of the
// work list, so each CTA finds them by scanning the list's first `slots`
// entries for split 0 of a request with two or more splits.
#include "internal.h"
#include "ptx.cuh"

namespace mlafold {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxStarts = 2048;   // multi-split requests tracked per CTA

template <int BANDS>
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ work,
               int list_len, int slots, int R, int M, const float* __restrict__ part_o,
               const float* __restrict__ part_lse, float bmm2, uint16_t* __restrict__ out,
               float* __restrict__ lse) {
  __shared__ int s_req[kMaxStarts];
  __shared__ int s_start[kMaxStarts];
  __shared__ int s_warp[kWarps];
  __shared__ int s_nreq;
  // Ordered compaction of the multi-split requests' first items: every CTA
  // must see the same list, in work-list order, to agree on row ownership.
  // It runs before the wait for the decode, on SMs the decode has left: the
  // work list and counts are the plan's, and every decode CTA passed its own
  // wait for the plan's completion before this grid could launch (L2 reads,
  // so no stale L1 line of an earlier step is seen).
  const int lane = threadIdx.x & 31, warp_id = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_nreq = 0;
  __syncthreads();
  const int scan = min(list_len, slots);
  for (int base = 0; base < scan; base += blockDim.x) {
    const int e = base + threadIdx.x;
    bool first = false;
    int r = 0;
    if (e < scan) {
      const int w = __ldcg(work + e);
      if (w >= 0 && entry_split(w) == 0) {
        r = entry_request(w);
        first = r < R && __ldcg(counts + r) >= 2;
      }
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, first);
    if (lane == 0) s_warp[warp_id] = __popc(ballot);
    __syncthreads();
    int before = s_nreq;
    for (int w = 0; w < warp_id; ++w) before += s_warp[w];
    before += __popc(ballot & ((1u << lane) - 1u));
    if (first && before < kMaxStarts) { s_req[before] = r; s_start[before] = e; }
    __syncthreads();
    if (threadIdx.x == 0) {
      int add = 0;
      for (int w = 0; w < kWarps; ++w) add += s_warp[w];
      s_nreq += add;
    }
    __syncthreads();
  }
  const int nreq = min(s_nreq, kMaxStarts);
  grid_dep_wait();      // the decode's partials are complete
  grid_dep_launch();
  constexpr int kDims = kDv / BANDS;          // dims per warp
  constexpr int kVec = kDims / 32 / 4;        // float4 per lane
  const long long total = (long long)nreq * M * BANDS;
  for (long long t = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); t < total;
       t += (long long)gridDim.x * kWarps) {
    const int band = (int)(t % BANDS);
    const long long rm = t / BANDS;
    const int m = (int)(rm % M);
    const int qi = (int)(rm / M);
    const int r = s_req[qi], start = s_start[qi];
    const int n = counts[r];
    if (start + n > slots) continue;       // not a plan of this shape: nothing to read
    // Lanes hold 32 splits' LSEs at a time; the max, the weights and their sum
    // come from shuffles, so only the partial rows are loaded per split.
    const float* lrow = part_lse + (long long)start * M + m;
    float mx = -INFINITY;
    for (int c0 = 0; c0 < n; c0 += 32)
      if (c0 + lane < n) mx = fmaxf(mx, lrow[(long long)(c0 + lane) * M]);
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float z = 0.f;
    float4 acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* base = part_o + ((long long)start * M + m) * kDv + band * kDims;
    const long long split_stride = (long long)M * kDv;
    for (int c0 = 0; c0 < n; c0 += 32) {
      const float lc = c0 + lane < n ? lrow[(long long)(c0 + lane) * M] : -INFINITY;
      const float wc = (mx == -INFINITY || lc == -INFINITY) ? 0.f : ex2(lc - mx);
      z += wc;
      const int cn = min(32, n - c0);
      for (int s0 = 0; s0 < cn; s0 += 4) {
        float4 o[4][kVec];
        float w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {          // four splits' loads in flight together
          const int s = s0 + u;
          w[u] = __shfl_sync(0xffffffffu, wc, s & 31);
          const bool live = s < cn;
          const float4* src =
              reinterpret_cast<const float4*>(base + (live ? c0 + s : 0) * split_stride);
#pragma unroll
          for (int v = 0; v < kVec; ++v)
            o[u][v] = live ? src[v * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
          if (!live) w[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < kVec; ++v) {
            acc[v].x += w[u] * o[u][v].x; acc[v].y += w[u] * o[u][v].y;
            acc[v].z += w[u] * o[u][v].z; acc[v].w += w[u] * o[u][v].w;
          }
      }
    }
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float scale = z > 0.f ? bmm2 / z : 0.f;
    uint16_t* dst = out + ((long long)r * M + m) * kDv + band * kDims;
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      uint2 packed;
      packed.x = (uint32_t)f32_to_bf16_bits(acc[v].x * scale) |
                 ((uint32_t)f32_to_bf16_bits(acc[v].y * scale) << 16);
      packed.y = (uint32_t)f32_to_bf16_bits(acc[v].z * scale) |
                 ((uint32_t)f32_to_bf16_bits(acc[v].w * scale) << 16);
      *reinterpret_cast<uint2*>(dst + (v * 32 + lane) * 4) = packed;
    }
    if (lse && band == 0 && lane == 0)
      lse[(long long)r * M + m] = z > 0.f ? mx + __log2f(z) : -INFINITY;
  }
}

}  // namespace

// The pages' `reducer_d_tiles`: 2 D512 bands when ceil(2 rows / sms) <
// 2 ceil(rows / sms), i.e. when the rows fill at most half the SMs, else 1.
int reducer_bands(long long rows, int sms) {
  return cdiv(2 * rows, sms) < 2 * cdiv(rows, sms) ? 2 : 1;
}

cudaError_t launch_combine(const mla_shape& s, const int32_t* counts, const int32_t* work,
                           int list_len, const float* part_o, const float* part_lse, int slots,
                           float bmm2, uint16_t* out, float* lse, cudaStream_t st) {
  const int M = group_rows(s), R = plan_rows(s);
  const int bands = reducer_bands((long long)R * M, s.num_ctas);
  // Up to slots / 2 multi-split requests (each has two or more items).
  const long long rows = (long long)(slots / 2) * M * bands;
  long long blocks = cdiv(rows, kWarps);
  const long long cap = 4LL * s.num_ctas;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bands == 2)
    return cudaLaunchKernelEx(&cfg, combine_kernel<2>, counts, work, list_len, slots, R, M,
                              part_o, part_lse, bmm2, out, lse);
  return cudaLaunchKernelEx(&cfg, combine_kernel<1>, counts, work, list_len, slots, R, M,
                            part_o, part_lse, bmm2, out, lse);
}

}  // namespace mlafold
