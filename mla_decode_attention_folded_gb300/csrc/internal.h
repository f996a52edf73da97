// Shared constants, plan arithmetic and kernel entry declarations of libmlafold.
// Host and device code of the library include this; nothing outside it does.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/mlafold.h"

namespace mlafold {

constexpr int kPage = 64;          // tokens per cache page
constexpr int kDqk = 576;          // latent 512 + rope 64 (bytes per FP8 row)
constexpr int kDv = 512;           // value = latent slice
constexpr int kSplitBits = 12;     // work item = request << 12 | split
constexpr int kPackedBit = 1 << 30;   // set in every entry of a packed plan
__host__ __device__ inline int entry_request(int e) {
  return (e & ~kPackedBit) >> kSplitBits;
}
__host__ __device__ inline int entry_split(int e) { return e & ((1 << kSplitBits) - 1); }
constexpr int kMaxR = 1024;        // the planner runs one CTA with one thread per request
constexpr int kMaxM = 4096;

__host__ __device__ inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// Jobs per work item: blocks of the request's M query rows, processed with the
// query rows as the MMA's N dimension (decode_tc.cu): blocks of 32 rows when
// M <= 32, else of 64 rows.
__host__ __device__ inline int row_block(int M) { return M <= 32 ? 32 : 64; }
__host__ __device__ inline int row_blocks(int M) { return (M + row_block(M) - 1) / row_block(M); }
// Concurrent work items the plan targets.
__host__ __device__ inline int plan_units(int M, int num_ctas) {
  int u = num_ctas / row_blocks(M);
  return u < 1 ? 1 : u;
}
__host__ __device__ inline int uniform_splits(int R, int M, int num_ctas, int max_splits) {
  long long s = cdiv(plan_units(M, num_ctas), R > 0 ? R : 1);
  if (s < 1) s = 1;
  return (int)(s < max_splits ? s : max_splits);
}
// Decode row groups (the planned "requests") and query rows per group.
inline int shape_groups(const mla_shape& s) { return s.groups > 0 ? s.groups : 1; }
inline int plan_rows(const mla_shape& s) { return s.R * shape_groups(s); }
inline int group_rows(const mla_shape& s) { return (s.k / shape_groups(s)) * s.H; }
// Work-list entries for items (the plan's bound on their number).
inline int plan_items(const mla_shape& s) {
  const int R = plan_rows(s), M = group_rows(s);
  if (s.policy == MLA_POLICY_BALANCED) return plan_units(M, s.num_ctas) + R;
  return R * uniform_splits(R, M, s.num_ctas, s.max_splits);
}
// The plan buffer: the E entries, then the decode's two job counters (claimed
// jobs, finished CTAs: the plan sets them to -1 with the rest of the padding,
// they count down during a decode, and its last CTA sets them back to -1),
// then each entry's first and end page within its request, then the packed
// plan's per-unit piece table (kUnitSlots entries per unit, all -1 when the
// plan is not packed).
constexpr int kSchedWords = 2;
constexpr int kUnitSlots = 8;          // pieces a unit of a packed plan may hold
constexpr int kMaxPackedUnits = 1024;  // the planner's per-unit tables
// Whether the plan of this shape may be packed (the planner packs only then):
// items of several row blocks, at most one request per unit.
inline bool plan_packable(const mla_shape& s) {
  const int M = group_rows(s), U = plan_units(M, s.num_ctas);
  return s.policy == MLA_POLICY_BALANCED && row_blocks(M) >= 2 && plan_rows(s) <= U &&
         U <= kMaxPackedUnits;
}
inline int plan_ranges_offset(const mla_shape& s) { return plan_items(s) + kSchedWords; }
inline int plan_units_offset(const mla_shape& s) { return 3 * plan_items(s) + kSchedWords; }
inline int plan_list_len(const mla_shape& s) {
  return plan_units_offset(s) + kUnitSlots * plan_units(group_rows(s), s.num_ctas);
}
// Bound on items of multi-split requests; they occupy work-list slots [0, slots).
inline int partial_slots(const mla_shape& s) {
  const int R = plan_rows(s), M = group_rows(s);
  if (s.policy == MLA_POLICY_BALANCED) {
    int a = plan_items(s), b = 2 * plan_units(M, s.num_ctas);
    return a < b ? a : b;
  }
  int u = uniform_splits(R, M, s.num_ctas, s.max_splits);
  return u >= 2 ? R * u : 0;
}
// Keys [j0, j1) of split s of n of a request of L keys (page-aligned cuts).
__host__ __device__ inline void split_range(int L, int n, int s, int& j0, int& j1) {
  long long p = cdiv(L, kPage);
  long long p0 = (s * p) / n, p1 = ((s + 1) * p) / n;
  j0 = (int)(kPage * p0);
  long long e = kPage * p1;
  j1 = (int)(e < L ? e : L);
}
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
// Workspace: FP32 partial outputs [slots][M][512], then FP32 LSEs [slots][M].
inline size_t partial_out_bytes(int slots, int M) { return align256(size_t(slots) * M * kDv * 4); }
inline size_t workspace_bytes(const mla_shape& s) {
  int slots = partial_slots(s), M = group_rows(s);
  if (slots == 0) return 0;
  return partial_out_bytes(slots, M) + align256(size_t(slots) * M * 4);
}

struct DecodeArgs {
  const uint8_t* q;
  const uint8_t* kv;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* counts;
  const int32_t* work;
  int32_t* sched;    // work + items: the job counters
  const int32_t* ranges;   // each entry's first and end page within its request
  const int32_t* units;    // packed plan: unit u's entry k at k * nunits + u
  float* part_o;     // [slots][M][512]
  float* part_lse;   // [slots][M]
  uint16_t* out;     // [R][M][512] bf16 bits
  float* lse;        // [R][M]
  int32_t* status;   // may be null
  float bmm1_log2;   // bmm1_scale * log2(e)
  float bmm2;
  int R, M, max_pages, num_pages, items, slots;   // R, M: row groups, rows per group
  int nunits;          // units of the plan (its unit table's rows)
  int groups;          // row group g reads request g / groups
  unsigned long long wait_limit_ns;   // bound of every pipeline wait (drains keep their own)
  int withhold_first_copy;            // failure-detection test: CTA 0 never issues its
                                      // first KV tile's copy, so one wait must run out
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_plan(const mla_shape& s, const int32_t* seq_lens, int32_t* counts,
                        int32_t* work, int list_len, cudaStream_t st);
cudaError_t launch_combine(const mla_shape& s, const int32_t* counts, const int32_t* work,
                           int list_len, const float* part_o, const float* part_lse, int slots,
                           float bmm2, uint16_t* out, float* lse, cudaStream_t st);
cudaError_t launch_decode(const mla_shape& s, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_uv(const mla_shape& s, const int32_t* counts, const int32_t* work,
                      int list_len, const float* part_o, const float* part_lse, int slots,
                      float bmm2, const uint16_t* out, const uint16_t* w_uv, uint16_t* y,
                      int32_t* status, cudaStream_t st);
cudaError_t launch_lse_merge(int S, int rows, const uint16_t* parts_out, const float* parts_lse,
                             uint16_t* out, float* lse, cudaStream_t st);

}  // namespace mlafold
