// Device split planner: KV lengths -> split counts and the plan buffer, one CTA.
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
//             max_splits), equal page-aligned splits
//   packed:   items of two or more row blocks, R <= U <= kMaxPackedUnits
//             (the decode launch knows from the shape that the plan may be
//             packed: plan_packable) and, with `big` that plan's
//             largest item and J = kJobPages (a piece's query load and
//             epilogue, in pages), 8 (c0 + 2J) <= 7 (big + J): the rank-ordered
//             pages cut into segments of c0 pages, unit u takes the pieces of
//             segment u; kept if every n_i <= max_splits, every unit holds
//             <= kUnitSlots pieces and max_u (pages of u + J * pieces of u) is
//             at most 7/8 of big + J
//   uniform:  n_i = min(clamp(ceil(U / R), 1, max_splits), p_i)
//   empty requests get one (empty) piece in every mode.
//
// Buffer: entries (multi-piece requests first, then the others, each in rank
// order; bit 30 set in every entry of a packed plan), two job counters, then,
// for a packed plan, each entry's page range and the unit table.
// Integer arithmetic only, so the CPU planner reproduces it bit for bit.
#include "internal.h"
#include "ptx.cuh"

namespace mlafold {
namespace {

constexpr int kThreads = kMaxR;   // one thread per request
constexpr int kJobPages = 4;      // overhead charged per piece of a packed plan

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

__device__ long long block_max64(long long v, long long* red) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (blockDim.x == 32) return v;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  long long t = lane < (blockDim.x >> 5) ? red[lane] : 0;
  for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

// Exclusive scan over the block of one value per thread (thread t's value is
// element t); also returns the total.
template <typename T>
__device__ T block_excl_scan(T v, T* warp_tot, T& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const T t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();                       // warp_tot may still be read by a previous call
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  T before = 0, all = 0;
  for (int w = 0; w < nw; ++w) {
    const T x = warp_tot[w];
    if (w < warp) before += x;
    all += x;
  }
  total = all;
  return before + incl - v;
}

// PACKABLE: the shape allows a packed plan (plan_packable); the other shapes
// run the per-request plan alone, without the packed plan's tables.
template <bool PACKABLE>
__global__ void __launch_bounds__(kThreads, 1)
plan_kernel(const int32_t* __restrict__ seq_lens, int R, int groups, int M, int num_ctas,
            int minp, int max_splits, int policy, int32_t* __restrict__ counts,
            int32_t* __restrict__ work, int items, int list_len) {
  __shared__ int s_len[kThreads];
  __shared__ int s_byrank[kThreads];
  __shared__ long long s_red64[32];
  __shared__ int s_red[32];
  // Packed plans only: dynamic shared memory, one 64-bit word per thread and
  // two words per unit.
  extern __shared__ long long s_dyn[];
  long long* s_byrank64 = s_dyn;                              // [blockDim]
  int* s_cnt = reinterpret_cast<int*>(s_byrank64 + blockDim.x);   // real pieces per segment
  int* s_first = s_cnt + plan_units(M, num_ctas);   // rank of a segment's first piece

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
  long long c0 = cdiv(T, U);
  if (c0 < minp) c0 = minp;

  int n = 1;
  if (policy == MLA_POLICY_BALANCED) {
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
  int rank = i;                           // dead slots keep ranks R..blockDim-1
  if (live) {
    rank = 0;
    for (int j = 0; j < R; ++j) {
      const int o = s_len[j];
      rank += (o > L) || (o == L && j < i);
    }
  }

  // Packed plan (block-uniform decision).
  bool packed = false;
  long long P = 0;                        // pages of the requests ranked before
  int u0 = 0;                             // first segment of this request
  int nseg = 1;
  const int big = PACKABLE ? block_max(p > 0 ? (p + n - 1) / n : 0, s_red) : 0;
  if (PACKABLE && T > 0 && 8 * (c0 + 2 * kJobPages) <= 7LL * (big + kJobPages)) {
    s_byrank64[rank] = live ? (long long)p : 0;
    __syncthreads();
    long long tot64;
    P = block_excl_scan<long long>(s_byrank64[i], s_red64, tot64);   // element i = rank i
    __syncthreads();
    s_byrank64[i] = P;                    // exclusive prefix at rank i
    for (int u = i; u < U; u += blockDim.x) s_cnt[u] = 0;
    __syncthreads();
    P = s_byrank64[rank];
    nseg = (int)cdiv(T, c0);
    int npk = 1, unit_of_empty = -1;
    if (live && p > 0) {
      u0 = (int)(P / c0);
      const int u1 = (int)((P + p - 1) / c0);
      npk = u1 - u0 + 1;
      for (int u = u0; u <= u1; ++u) {
        atomicAdd(&s_cnt[u], 1);
        if ((long long)u * c0 >= P) s_first[u] = rank;   // this request starts segment u
      }
    } else if (live) {
      unit_of_empty = (rank - Rn) % nseg;  // empty requests rank last
    }
    __syncthreads();
    const int ne = R - Rn;
    int worst = 0;
    long long cost = 0;                   // pages + kJobPages per piece, costliest unit
    for (int u = i; u < nseg; u += blockDim.x) {
      const int with_empty = s_cnt[u] + (ne > u ? (ne - 1 - u) / nseg + 1 : 0);
      worst = max(worst, with_empty);
      const long long pages = min(c0, T - (long long)u * c0);
      cost = max(cost, pages + (long long)kJobPages * with_empty);
    }
    worst = block_max(worst, s_red);
    const int most = block_max(live ? npk : 0, s_red);
    cost = block_max64(cost, s_red64);
    if (most <= max_splits && worst <= kUnitSlots && 8 * cost <= 7LL * (big + kJobPages)) {
      packed = true;
      n = npk;
      if (unit_of_empty >= 0) u0 = unit_of_empty;
    }
  }

  // Entry order: multi-piece requests in rank order, then the others. In the
  // per-request plans n never decreases with the length: that is rank order.
  int pos = rank;
  if (packed) {                           // block-uniform
    const int multi = live && n >= 2 ? 1 : 0;
    s_byrank[rank] = multi;
    __syncthreads();
    int nmulti;
    const int mbefore_i = block_excl_scan<int>(s_byrank[i], s_red, nmulti);
    __syncthreads();
    s_byrank[i] = mbefore_i;              // multi-piece requests ranked before rank i
    __syncthreads();
    const int mbefore = s_byrank[rank];
    pos = multi ? mbefore : nmulti + (rank - mbefore);
  }
  __syncthreads();
  s_byrank[pos] = live ? n : 0;           // dead slots: positions R..blockDim-1
  __syncthreads();
  int total;
  const int start_i = block_excl_scan<int>(s_byrank[i], s_red, total);
  __syncthreads();
  s_byrank[i] = start_i;
  // -1: the entries after the last one and the two job counters; a packed
  // plan's range words after the last entry's and its unit table.
  int32_t* rng = work + items + kSchedWords;
  int32_t* utab = work + 3 * items + kSchedWords;
  for (int e = total + i; e < items + kSchedWords; e += blockDim.x) work[e] = -1;
  if (packed) {
    for (int e = 2 * total + i; e < 2 * items; e += blockDim.x) rng[e] = -1;
    for (int e = i; e < kUnitSlots * U; e += blockDim.x) utab[e] = -1;
    __syncthreads();                      // the fills land before the pieces' words
  }

  if (live) {
    const int start = s_byrank[pos];
    for (int sp = 0; sp < n; ++sp) {
      const int e = start + sp;
      if (e >= items) break;
      work[e] = (packed ? kPackedBit : 0) | (i << kSplitBits) | sp;
      if (packed) {
        const long long u = u0 + sp;
        rng[2 * e] = p > 0 ? (int)(max(P, u * c0) - P) : 0;
        rng[2 * e + 1] = p > 0 ? (int)(min(P + p, (u + 1) * c0) - P) : 0;
        const int slot = p > 0 ? rank - s_first[u] : s_cnt[u] + (rank - Rn) / nseg;
        utab[slot * U + (int)u] = e;      // slot-major
      }
    }
    counts[i] = n;
  }
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
  const int U = plan_units(group_rows(s), s.num_ctas);
  if (!plan_packable(s))
    return cudaLaunchKernelEx(&cfg, plan_kernel<false>, seq_lens, R, shape_groups(s),
                              group_rows(s), s.num_ctas, minp, s.max_splits, s.policy, counts,
                              work, plan_items(s), list_len);
  cfg.dynamicSmemBytes = cfg.blockDim.x * sizeof(long long) + 2 * sizeof(int) * (size_t)U;
  return cudaLaunchKernelEx(&cfg, plan_kernel<true>, seq_lens, R, shape_groups(s),
                            group_rows(s), s.num_ctas, minp, s.max_splits, s.policy, counts,
                            work, plan_items(s), list_len);
}

}  // namespace mlafold
