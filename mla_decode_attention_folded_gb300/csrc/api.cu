// Host side of the C ABI declared in include/mlafold.h: argument validation,
// plan and workspace sizing, and the kernel launches. Nothing here allocates
// device memory or synchronises a stream.
#include <cmath>
#include <cstdint>

#include "internal.h"

using namespace mlafold;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(const mla_shape* s) {
  if (!s) return MLA_ERR_NULL;
  if (s->page_size != kPage) return MLA_ERR_UNSUPPORTED;
  if (s->R < 1 || s->k < 1 || s->H < 1 || s->groups < 0) return MLA_ERR_SHAPE;
  const int groups = s->groups > 0 ? s->groups : 1;
  if (s->k % groups != 0 || (long long)s->R * groups > kMaxR) return MLA_ERR_SHAPE;
  const long long M = (long long)s->k * s->H;
  if (M > kMaxM) return MLA_ERR_SHAPE;
  if (s->max_pages < 1 || s->max_pages >= (1 << 25) || s->num_pages < 1 ||
      s->num_pages >= (1 << 25))
    return MLA_ERR_SHAPE;
  if (s->num_ctas < 1 || s->num_ctas > 2048) return MLA_ERR_SHAPE;
  if (s->min_split_tokens < 1) return MLA_ERR_SHAPE;
  if (s->max_splits < 1 || s->max_splits > (1 << kSplitBits)) return MLA_ERR_SHAPE;
  if (s->policy != MLA_POLICY_BALANCED && s->policy != MLA_POLICY_UNIFORM) return MLA_ERR_SHAPE;
  return MLA_OK;
}

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (major != 10 || minor != 3) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

}  // namespace

extern "C" {

int32_t mla_plan_list_len(const mla_shape* shape) {
  int st = check_shape(shape);
  if (st != MLA_OK) return st;
  return plan_list_len(*shape);
}

int32_t mla_workspace_bytes(const mla_shape* shape, size_t* bytes) {
  int st = check_shape(shape);
  if (st != MLA_OK) return st;
  if (!bytes) return MLA_ERR_NULL;
  *bytes = workspace_bytes(*shape);
  return MLA_OK;
}

int32_t mla_plan_splits(const mla_shape* shape, const int32_t* seq_lens, int32_t* counts,
                        int32_t* work, int32_t list_len, mla_stream_t stream) {
  int st = check_shape(shape);
  if (st != MLA_OK) return st;
  if (!seq_lens || !counts || !work) return MLA_ERR_NULL;
  if (!aligned(seq_lens, 4) || !aligned(counts, 4) || !aligned(work, 4)) return MLA_ERR_ALIGN;
  if (list_len < plan_list_len(*shape)) return MLA_ERR_LIST;
  if ((st = check_device()) != MLA_OK) return st;
  cudaError_t e = launch_plan(*shape, seq_lens, counts, work, list_len,
                              reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"

namespace {

// mla_folded_decode with an explicit pipeline-wait bound and the
// failure-detection test's withheld copy.
int32_t decode_impl(const mla_shape* shape, const void* q, const void* kv,
                    const int32_t* block_table, const int32_t* seq_lens, float bmm1_scale,
                    float bmm2_scale, const int32_t* counts, int32_t* work, int32_t list_len,
                    void* workspace, size_t workspace_bytes_given, void* out, float* lse,
                    int32_t* status, mla_stream_t stream, unsigned long long wait_limit_ns,
                    int withhold_first_copy) {
  int st = check_shape(shape);
  if (st != MLA_OK) return st;
  if (!q || !kv || !block_table || !seq_lens || !counts || !work || !out) return MLA_ERR_NULL;
  const size_t need = workspace_bytes(*shape);
  if (need > 0 && !workspace) return MLA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4)) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(counts, 4) ||
      !aligned(work, 4) || (workspace && !aligned(workspace, 256)) ||
      (status && !aligned(status, 4)))
    return MLA_ERR_ALIGN;
  if (list_len < plan_list_len(*shape)) return MLA_ERR_LIST;
  if (workspace_bytes_given < need) return MLA_ERR_WORKSPACE;
  if (!std::isfinite(bmm1_scale) || !(bmm1_scale > 0.f) || !std::isfinite(bmm2_scale))
    return MLA_ERR_SHAPE;
  if ((st = check_device()) != MLA_OK) return st;
  const int M = group_rows(*shape);
  const int slots = partial_slots(*shape);
  DecodeArgs a;
  a.q = static_cast<const uint8_t*>(q);
  a.kv = static_cast<const uint8_t*>(kv);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.counts = counts;
  a.work = work;
  a.sched = work + plan_items(*shape);
  a.ranges = work + plan_ranges_offset(*shape);
  a.units = work + plan_units_offset(*shape);
  a.nunits = plan_units(M, shape->num_ctas);
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                    partial_out_bytes(slots, M))
                         : nullptr;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.status = status;
  a.bmm1_log2 = (float)((double)bmm1_scale * 1.4426950408889634);
  a.bmm2 = bmm2_scale;
  a.R = plan_rows(*shape);
  a.M = M;
  a.groups = shape_groups(*shape);
  a.max_pages = shape->max_pages;
  a.num_pages = shape->num_pages;
  a.items = plan_items(*shape);
  a.slots = slots;
  a.wait_limit_ns = wait_limit_ns;
  a.withhold_first_copy = withhold_first_copy;
  cudaError_t e = launch_decode(*shape, a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

constexpr unsigned long long kDecodeWaitLimitNs = 2000000000ull;   // 2 s

}  // namespace

extern "C" {

int32_t mla_folded_decode(const mla_shape* shape, const void* q, const void* kv,
                          const int32_t* block_table, const int32_t* seq_lens, float bmm1_scale,
                          float bmm2_scale, const int32_t* counts, int32_t* work,
                          int32_t list_len, void* workspace, size_t workspace_bytes_given,
                          void* out, float* lse, int32_t* status, mla_stream_t stream) {
  return decode_impl(shape, q, kv, block_table, seq_lens, bmm1_scale, bmm2_scale, counts, work,
                     list_len, workspace, workspace_bytes_given, out, lse, status, stream,
                     kDecodeWaitLimitNs, 0);
}

int32_t mla_folded_decode_wait_test(const mla_shape* shape, const void* q, const void* kv,
                                    const int32_t* block_table, const int32_t* seq_lens,
                                    float bmm1_scale, float bmm2_scale, const int32_t* counts,
                                    int32_t* work, int32_t list_len, void* workspace,
                                    size_t workspace_bytes_given, void* out, float* lse,
                                    int32_t* status, uint64_t wait_limit_ns,
                                    mla_stream_t stream) {
  if (!status) return MLA_ERR_NULL;
  if (wait_limit_ns < 1000000ull || wait_limit_ns > kDecodeWaitLimitNs) return MLA_ERR_SHAPE;
  return decode_impl(shape, q, kv, block_table, seq_lens, bmm1_scale, bmm2_scale, counts, work,
                     list_len, workspace, workspace_bytes_given, out, lse, status, stream,
                     wait_limit_ns, 1);
}

int32_t mla_split_combine(const mla_shape* shape, const int32_t* counts, const int32_t* work,
                          int32_t list_len, const void* workspace, size_t workspace_bytes_given,
                          float bmm2_scale, void* out, float* lse, mla_stream_t stream) {
  int st = check_shape(shape);
  if (st != MLA_OK) return st;
  if (!counts || !work || !out) return MLA_ERR_NULL;
  const size_t need = workspace_bytes(*shape);
  if (need > 0 && !workspace) return MLA_ERR_NULL;
  if (!aligned(out, 16) || (lse && !aligned(lse, 4)) || !aligned(counts, 4) || !aligned(work, 4) ||
      (workspace && !aligned(workspace, 256)))
    return MLA_ERR_ALIGN;
  if (list_len < plan_list_len(*shape)) return MLA_ERR_LIST;
  if (workspace_bytes_given < need) return MLA_ERR_WORKSPACE;
  if (!std::isfinite(bmm2_scale)) return MLA_ERR_SHAPE;
  if ((st = check_device()) != MLA_OK) return st;
  const int M = group_rows(*shape);
  const int slots = partial_slots(*shape);
  if (slots == 0) return MLA_OK;       // no request can have two splits
  const float* po = static_cast<const float*>(workspace);
  const float* pl = reinterpret_cast<const float*>(static_cast<const char*>(workspace) +
                                                   partial_out_bytes(slots, M));
  cudaError_t e = launch_combine(*shape, counts, work, list_len, po, pl, slots, bmm2_scale,
                                 static_cast<uint16_t*>(out), lse,
                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_uv_combine(const mla_shape* shape, const int32_t* counts, const int32_t* work,
                       int32_t list_len, const void* workspace, size_t workspace_bytes_given,
                       float bmm2_scale, const void* out, const void* w_uv, void* y,
                       int32_t* status, mla_stream_t stream) {
  int st = check_shape(shape);
  if (st != MLA_OK) return st;
  if (!counts || !work || !out || !w_uv || !y) return MLA_ERR_NULL;
  const size_t need = workspace_bytes(*shape);
  if (need > 0 && !workspace) return MLA_ERR_NULL;
  if (!aligned(out, 16) || !aligned(w_uv, 16) || !aligned(y, 16) || !aligned(counts, 4) ||
      !aligned(work, 4) || (workspace && !aligned(workspace, 256)) ||
      (status && !aligned(status, 4)))
    return MLA_ERR_ALIGN;
  if (list_len < plan_list_len(*shape)) return MLA_ERR_LIST;
  if (workspace_bytes_given < need) return MLA_ERR_WORKSPACE;
  if (!std::isfinite(bmm2_scale)) return MLA_ERR_SHAPE;
  if ((st = check_device()) != MLA_OK) return st;
  const int M = group_rows(*shape);
  const int slots = partial_slots(*shape);
  const float* po = static_cast<const float*>(workspace);
  const float* pl = workspace ? reinterpret_cast<const float*>(static_cast<const char*>(workspace) +
                                                               partial_out_bytes(slots, M))
                              : nullptr;
  cudaError_t e = launch_uv(*shape, counts, work, list_len, po, pl, slots, bmm2_scale,
                            static_cast<const uint16_t*>(out), static_cast<const uint16_t*>(w_uv),
                            static_cast<uint16_t*>(y), status,
                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_lse_merge(int32_t S, int32_t rows, const void* parts_out, const float* parts_lse,
                      void* out, float* lse, mla_stream_t stream) {
  if (!parts_out || !parts_lse || !out) return MLA_ERR_NULL;
  if (S < 1 || S > 4096 || rows < 1) return MLA_ERR_SHAPE;
  if (!aligned(parts_out, 16) || !aligned(out, 16) || !aligned(parts_lse, 4) ||
      (lse && !aligned(lse, 4)))
    return MLA_ERR_ALIGN;
  int st;
  if ((st = check_device()) != MLA_OK) return st;
  cudaError_t e = launch_lse_merge(S, rows, static_cast<const uint16_t*>(parts_out), parts_lse,
                                   static_cast<uint16_t*>(out), lse,
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"
