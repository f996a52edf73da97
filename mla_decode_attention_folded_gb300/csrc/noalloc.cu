// Decode entry point for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: code that runs while a
// memory pool is being sized and must not fragment it, plugins whose host
// application owns every device allocation, and runtimes whose allocator is
// forbidden on the decode path. mla_folded_decode_noalloc gives them the same
// decode as mla_folded_decode followed by mla_split_combine, with the split-KV
// partials kept in a fixed array of device memory that belongs to this
// library instead of a caller-provided workspace.
//
// The array is a file-scope __device__ object of MLA_NOALLOC_SCRATCH_BYTES
// (64 MiB); every GPU that loads the library's device code holds it until the
// process exits. In host code its name is only a host-side stand-in, so the
// device address is looked up with cudaGetSymbolAddress, with the device
// current, on the first call per device, and cached. All calls on a device
// share the array; nothing in it has to start at zero, because each call
// writes every partial it later reads.
#include <atomic>
#include <cstdint>

#include "internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes == (size_t(64) << 20), "the header states 64 MiB");
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the array per device; two host threads making their first
// call on one device at once both look it up and store the same value.
std::atomic<void*> g_scratch_addr[kMaxDevices];

// The scratch array's device address on the current device (looked up on the
// first call per device).
int32_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return MLA_OK;
}

}  // namespace

extern "C" int32_t mla_folded_decode_noalloc(const mla_shape* shape, const void* q,
                                             const void* kv, const int32_t* block_table,
                                             const int32_t* seq_lens, float bmm1_scale,
                                             float bmm2_scale, const int32_t* counts,
                                             int32_t* work, int32_t list_len, void* out,
                                             float* lse, int32_t* status, mla_stream_t stream) {
  size_t need = 0;
  int32_t st = mla_workspace_bytes(shape, &need);
  if (st != MLA_OK) return st;
  if (need > kNoallocScratchBytes) return MLA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != MLA_OK) return st;
  st = mla_folded_decode(shape, q, kv, block_table, seq_lens, bmm1_scale, bmm2_scale, counts,
                         work, list_len, scratch, kNoallocScratchBytes, out, lse, status, stream);
  if (st != MLA_OK) return st;
  return mla_split_combine(shape, counts, work, list_len, scratch, kNoallocScratchBytes,
                           bmm2_scale, out, lse, stream);
}
