// Device split planner: KV lengths -> split counts and work list, one CTA.
//
// The balanced-MLA page (module overview) plans each request's split count
// from the KV lengths on the device, once per decode step, and the persistent
// decode walks the resulting work list; `BalancedMla.require` pre-fills the
// list with -1. The ordering is the rank rule of the drafter-attention page's
// `_plan_kernel`: longest first, ties to the lower row. The split formula is
// this project's reading (the pages do not give it):
//
//   p_i = ceil(len_i / 64), T = sum p_i, U = max(1, num_ctas / row_blocks(M))
//   balanced: c0 = max(minp, ceil(T / U)); if every non-empty request fits in
//             one wave (Rn <= U) and c0 leaves more than U items, c is the
//             smallest chunk >= c0 with at most U items; n_i = min(ceil(p_i/c),
//             max_splits)
//   uniform:  n_i = min(clamp(ceil(U / R), 1, max_splits), p_i)
//   empty requests get one split in both policies.
//
// Integer arithmetic only, so the CPU planner reproduces it bit for bit.
#include "internal.h"
#include "ptx.cuh"

namespace mlafold {
namespace {

constexpr int kThreads = kMaxR;   // one thread per request

template <typename T>
__device__ T block_sum(T v, T* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (blockDim.x == 32) return v;        // one warp: no shared-memory round trip
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();                       // red[] may still be read by a previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  T t = lane < (blockDim.x >> 5) ? red[lane] : T(0);
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

__device__ int block_max(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (blockDim.x == 32) return v;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = lane < (blockDim.x >> 5) ? red[lane] : 0;
  for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

__global__ void __launch_bounds__(kThreads, 1)
plan_kernel(const int32_t* __restrict__ seq_lens, int R, int groups, int M, int num_ctas,
            int minp, int max_splits, int policy, int32_t* __restrict__ counts,
            int32_t* __restrict__ work, int items, int list_len) {
  __shared__ int s_len[kThreads];
  __shared__ int s_n_by_rank[kThreads];
  __shared__ long long s_red64[32];
  __shared__ int s_red[32];
  __shared__ int s_scan[32];

  grid_dep_wait();
  const int i = threadIdx.x;
  const bool live = i < R;
  int L = live ? seq_lens[i / groups] : 0;   // row group i reads request i / groups
  if (L < 0) L = 0;
  s_len[i] = live ? L : -1;               // dead slots rank after every request
  grid_dep_launch();                      // the decode may start its prologue
  const int p = (int)cdiv(L, kPage);

  const long long T = block_sum<long long>((long long)p, s_red64);
  const int Rn = block_sum<int>(live && L > 0 ? 1 : 0, s_red);
  const int maxp = block_max(p, s_red);
  const int U = plan_units(M, num_ctas);

  int n = 1;
  if (policy == MLA_POLICY_BALANCED) {
    long long c0 = cdiv(T, U);
    if (c0 < minp) c0 = minp;
    // A chunk above the longest request gives every request one split, as the
    // longest request's own length does: clamp so 32-bit division suffices.
    int c = (int)(c0 < maxp ? c0 : (maxp > 0 ? maxp : 1));
    auto count = [&](int cc) {
      int mine = p > 0 ? min(max_splits, (p + cc - 1) / cc) : 0;
      return block_sum<int>(mine, s_red);
    };
    if (Rn <= U && count(c) > U) {        // block-uniform branch
      // Smallest chunk in (c, maxp] with at most U items (count(maxp) = Rn <= U;
      // count never increases with the chunk). Gallop up from c, then bisect:
      // the answer is usually within a step or two of c.
      int lo = c + 1, hi = lo, step = 1;
      while (hi < maxp && count(hi) > U) {
        lo = hi + 1;
        step *= 2;
        hi = min(maxp, lo + step - 1);
      }
      while (lo < hi) {
        const int mid = (lo + hi) / 2;
        if (count(mid) <= U) hi = mid; else lo = mid + 1;
      }
      c = lo;
    }
    n = p > 0 ? min(max_splits, (p + c - 1) / c) : 1;
  } else {
    const int S = uniform_splits(R, M, num_ctas, max_splits);
    n = L > 0 ? min(S, p) : 1;
  }

  // Rank: longest first, ties to the lower index.
  __syncthreads();
  int rank = 0;
  if (live) {
    for (int j = 0; j < R; ++j) {
      const int o = s_len[j];
      rank += (o > L) || (o == L && j < i);
    }
    s_n_by_rank[rank] = n;
  } else {
    s_n_by_rank[i] = 0;                   // ranks R..blockDim-1 hold nothing
  }
  __syncthreads();

  // Exclusive scan of the split counts in rank order.
  const int lane = i & 31, warp = i >> 5;
  int v = s_n_by_rank[i];
  int incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (blockDim.x >> 5) ? s_scan[lane] : 0;
    int wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    s_scan[lane] = wi - w;                // exclusive warp offsets
  }
  __syncthreads();
  const int excl_by_rank = s_scan[warp] + incl - v;   // start of rank i's items
  __syncthreads();
  s_n_by_rank[i] = excl_by_rank;          // reuse: start offset per rank
  const int total = block_sum<int>(v, s_red);
  __syncthreads();

  if (live) {
    const int start = s_n_by_rank[rank];
    for (int s = 0; s < n; ++s)
      if (start + s < items) work[start + s] = (i << kSplitBits) | s;
    counts[i] = n;
  }
  for (int e = total + i; e < list_len; e += blockDim.x) work[e] = -1;
}

}  // namespace

cudaError_t launch_plan(const mla_shape& s, const int32_t* seq_lens, int32_t* counts,
                        int32_t* work, int list_len, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  const int R = plan_rows(s);
  cfg.blockDim = dim3((unsigned)((R + 31) / 32 * 32));   // one thread per row group
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int minp = (int)cdiv(s.min_split_tokens, kPage) < 1 ? 1 : (int)cdiv(s.min_split_tokens, kPage);
  return cudaLaunchKernelEx(&cfg, plan_kernel, seq_lens, R, shape_groups(s), group_rows(s),
                            s.num_ctas, minp, s.max_splits, s.policy, counts, work,
                            plan_items(s), list_len);
}

}  // namespace mlafold
