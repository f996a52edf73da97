// The tiered launch's two helper kernels (drafter-attention page,
// `balanced_decode`, `_balanced_tables`, `_plan_kernel`, `_row_copy_kernel`):
//
// * tier_plan_kernel -- one CTA, one thread per decode row: rank the rows by
//   length (longest first, ties to the lower row); of the split_rows longest,
//   move those longer than move_num/move_den of a pair's share of the batch's
//   keys (len * move_den * pairs > move_num * total) out of the unsplit
//   launch and into the tiers.
// * row_copy_kernel -- whole-row gather or scatter of the rows whose target
//   index is in [0, bound): the tier rows' queries and block-table rows in,
//   their outputs and LSEs back out.
//
// Both are plain CUDA-core kernels: integer work and copies of a few MB.
#include <cstdint>

#include "internal.h"

namespace mlafold {
namespace {

constexpr int kTierThreads = 1024;            // rows <= kMaxR = 1024

__global__ void __launch_bounds__(kTierThreads)
tier_plan_kernel(const int32_t* __restrict__ seq_lens, int rows, int split_rows, int pairs,
                 int move_num, int move_den, int32_t* __restrict__ rest,
                 int32_t* __restrict__ tier_rows, int32_t* __restrict__ tier_lens) {
  __shared__ int s_len[kTierThreads];
  __shared__ unsigned long long s_part[kTierThreads / 32];
  const int i = threadIdx.x;
  const int len = i < rows ? max(seq_lens[i], 0) : 0;
  s_len[i] = len;
  unsigned long long v = (unsigned long long)len;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((i & 31) == 0) s_part[i >> 5] = v;
  __syncthreads();
  unsigned long long total = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += s_part[w];
  if (i >= rows) return;
  int rank = 0;                                // rows ahead of this one
  for (int j = 0; j < rows; ++j) {
    const int o = s_len[j];
    rank += (o > len) || (o == len && j < i);
  }
  if (rank >= split_rows) {
    rest[i] = len;
    return;
  }
  const bool move = (unsigned long long)len * (unsigned long long)move_den *
                        (unsigned long long)pairs >
                    (unsigned long long)move_num * total;
  rest[i] = move ? 0 : len;
  tier_rows[rank] = move ? i : rows;
  tier_lens[rank] = move ? len : 0;
}

// Row i of the target list: gather copies src row index[i] to dst row i,
// scatter copies src row i to dst row index[i]; rows whose index is outside
// [0, bound) are skipped. VEC: 16-byte pieces (row pitch and both bases
// 16-byte aligned), else 4-byte words.
template <bool VEC>
__global__ void row_copy_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                const int32_t* __restrict__ index, int bound,
                                long long row_bytes, int gather) {
  const int i = blockIdx.x;
  const int t = index[i];
  if (t < 0 || t >= bound) return;
  const long long s_row = gather ? t : i, d_row = gather ? i : t;
  const uint8_t* s = src + s_row * row_bytes;
  uint8_t* d = dst + d_row * row_bytes;
  const long long step = (long long)gridDim.y * blockDim.x;
  const long long first = (long long)blockIdx.y * blockDim.x + threadIdx.x;
  if constexpr (VEC) {
    const long long n = row_bytes / 16;
    for (long long c = first; c < n; c += step)
      reinterpret_cast<uint4*>(d)[c] = reinterpret_cast<const uint4*>(s)[c];
  } else {
    const long long n = row_bytes / 4;
    for (long long c = first; c < n; c += step)
      reinterpret_cast<uint32_t*>(d)[c] = reinterpret_cast<const uint32_t*>(s)[c];
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace mlafold

using namespace mlafold;

extern "C" int32_t mla_tier_plan(int32_t rows, int32_t split_rows, int32_t pairs,
                                 int32_t move_num, int32_t move_den, const int32_t* seq_lens,
                                 int32_t* rest_lens, int32_t* tier_rows, int32_t* tier_lens,
                                 mla_stream_t stream) {
  if (!seq_lens || !rest_lens || (split_rows > 0 && (!tier_rows || !tier_lens)))
    return MLA_ERR_NULL;
  if (rows < 1 || rows > kMaxR || split_rows < 0 || split_rows > rows || pairs < 1 ||
      pairs > 4096 || move_num < 1 || move_num > 65536 || move_den < 1 || move_den > 65536)
    return MLA_ERR_SHAPE;
  if (!aligned(seq_lens, 4) || !aligned(rest_lens, 4) ||
      (split_rows > 0 && (!aligned(tier_rows, 4) || !aligned(tier_lens, 4))))
    return MLA_ERR_ALIGN;
  tier_plan_kernel<<<1, kTierThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      seq_lens, rows, split_rows, pairs, move_num, move_den, rest_lens, tier_rows, tier_lens);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" int32_t mla_row_copy(const void* src, void* dst, const int32_t* index,
                                int32_t targets, int32_t bound, int64_t row_bytes,
                                int32_t gather, mla_stream_t stream) {
  if (targets < 0 || bound < 0 || row_bytes <= 0 || row_bytes % 4 != 0 ||
      (gather != 0 && gather != 1))
    return MLA_ERR_SHAPE;
  if (targets == 0) return MLA_OK;
  if (!src || !dst || !index) return MLA_ERR_NULL;
  if (!aligned(src, 4) || !aligned(dst, 4) || !aligned(index, 4)) return MLA_ERR_ALIGN;
  const bool vec = row_bytes % 16 == 0 && aligned(src, 16) && aligned(dst, 16);
  const long long pieces = row_bytes / (vec ? 16 : 4);
  const int threads = 256;
  long long chunks = (pieces + threads - 1) / threads;
  if (chunks > 64) chunks = 64;
  const dim3 grid((unsigned)targets, (unsigned)chunks);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* s = static_cast<const uint8_t*>(src);
  uint8_t* d = static_cast<uint8_t*>(dst);
  if (vec)
    row_copy_kernel<true><<<grid, threads, 0, st>>>(s, d, index, bound, row_bytes, gather);
  else
    row_copy_kernel<false><<<grid, threads, 0, st>>>(s, d, index, bound, row_bytes, gather);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
