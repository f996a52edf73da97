// The split-KV reduction fused with the W_UV up-projection: every (token,
// head) row's merged 512-dim latent output, rounded once to BF16, times that
// head's W_UV [512, 128] on the tensor cores (BF16 operands, FP32
// accumulation), rounded to BF16 (drafter-attention page, `DraftDcp`: the head
// owner merges its heads' rows by exp2(lse - max) / sum in FP32 with one BF16
// rounding and applies W_UV as a BF16 MMA; `latent_major`: W_UV stored
// latent-contiguous). The merged 512-dim rows never reach HBM.
//
// Persistent CTAs walk contiguous ranges of (head, 32-token block) tiles,
// head-major. The 128 W_UV output dims are the MMA's M and the 32 tokens its
// N ("swap-AB": 32 tokens keep even the smallest batches spread over SMs):
//     Y^T[128, 32] = W_UV[h]^T[128, 512] . X[32, 512]^T,  8 chunks x 4 MMAs (K = 16)
// W_UV[h] (128 KB) stays in shared memory while the CTA's tiles share a head.
// X, a tile's 32 merged BF16 rows, lands in shared memory by TMA from the
// decode's own BF16 rows (the rows of a request with one split; viewed as
// [token][head][512] they form one box per 64-dim chunk), issued one tile
// ahead; then 256 reducer threads (8 per token row, interleaved 16-byte
// pieces) overwrite the rows of requests with several splits with their merge
// of the FP32 split partials. X and the TMEM accumulator are double-buffered,
// so a tile's loads and merges overlap the previous tile's MMAs and the
// read-back of the one before; four of the reducer warps read the
// accumulator back and store Y.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace mlafold {
namespace {

constexpr int kTok = 32;                       // tokens per tile: the MMA's N
constexpr int kOut = 128;                      // W_UV output dims: the MMA's M
constexpr int kChunks = kDv / 64;              // 64 latent dims = 128 B of BF16 per chunk
constexpr int kRed = 256;                      // reducer threads: 8 per token row
constexpr int kThreads = 32 + kRed;            // warp 0: TMA + MMA + TMEM owner
constexpr int kWChunk = kOut * 128;            // one W chunk: 128 rows x 128 B
constexpr int kXChunk = kTok * 128;            // one X chunk: 32 rows x 128 B
constexpr int kXBytes = kChunks * kXChunk;     // one X buffer
constexpr int kOffW = 0;                       // W_UV[h], eight chunks
constexpr int kOffX = kChunks * kWChunk;       // two X buffers
constexpr int kOffStart = kOffX + 2 * kXBytes; // first slot of each multi-split row group
constexpr int kOffCount = kOffStart + kMaxR * 4;   // split count of every row group
constexpr int kOffBar = kOffCount + kMaxR * 4;
constexpr int kSmemBytes = kOffBar + 256 + 1024;        // + control block, + alignment slack
constexpr uint32_t kTmemCols = 2 * kTok;       // two FP32 accumulators of 32 columns
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kOut, kTok);
constexpr unsigned long long kTimeoutNs = 2000000000ull;
static_assert(kOffX % 1024 == 0 && kXChunk % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

struct UvCtl {
  uint64_t w_full[kChunks];   // TMA -> MMA: W chunk landed (one phase per head loaded)
  uint64_t x_full[2];         // reducers -> MMA: X buffer's merged rows written
  uint64_t x_tma[2];          // TMA -> reducers, MMA: X buffer's one-split rows landed
  uint64_t x_empty[2];        // MMA -> reducers (and W reload): the tile's MMAs finished
  uint64_t d_full[2];         // MMA -> read-back: accumulator final
  uint64_t d_empty[2];        // read-back -> MMA: accumulator read
  uint64_t drain;             // MMA issuer, on abort: every MMA it issued has finished
  uint32_t tmem_base;
  int abort_flag;
};

struct UvArgs {
  const int32_t* counts;
  const int32_t* work;
  const float* part_o;     // [slots][Mg][512]
  const float* part_lse;   // [slots][Mg]
  const uint16_t* out;     // [R][M][512] BF16: the decode's one-split rows
  uint16_t* y;             // [R*k][H][128] BF16
  int32_t* status;         // may be null
  float bmm2;
  int list_len, slots, plan_rows, k, H, groups, M, Mg, T;
};

__device__ __forceinline__ bool uv_wait(uint64_t* bar, uint32_t parity, UvCtl* ctl,
                                        int32_t* status) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = tc::globaltimer_ns();
  while (true) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl->abort_flag)) return false;
    if (tc::globaltimer_ns() - t0 > kTimeoutNs) {
      *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
      if (status) atomicOr(status, MLA_FAULT_WAIT_TIMEOUT);
      return false;
    }
  }
}

// X is K-major with the 128-byte swizzle: 64 latent dims (128 B of BF16) per
// chunk, 16-byte piece p of a row at ((p ^ (row & 7)) * 16) within the row.
// Byte offset in X of BF16 latent dims [8 i, 8 i + 8) of token row `row`:
__device__ __forceinline__ int x_piece(int row, int i) {
  return (i >> 3) * kXChunk + row * 128 + (((i & 7) ^ (row & 7)) << 4);
}

// Writes one token row's merged BF16 latent output into X when the row's
// request has several splits (the tile's TMA load brings the other rows). The
// 8 threads of the row (consecutive lanes; this one is `c`) cover it
// interleaved: thread c takes the float4s 8 v + c (v = 0..15) of an FP32
// partial row, so that each warp-wide load reads whole 128-byte lines.
// `ready()` is called once, after the row's global loads and before its first
// shared-memory write (it waits for the tile's TMA load); false = give up.
template <typename Ready>
__device__ __forceinline__ bool merged_row(const UvArgs& a, const int* s_start,
                                           const int* s_count, int tau, int h,
                                           int c, uint8_t* x, int row, Ready ready) {
  const uint4 zero = make_uint4(0, 0, 0, 0);
  int n = 0, r = 0, t = 0, i = 0, mg = 0;
  if (tau < a.T) {
    r = tau / a.k;
    t = tau - r * a.k;
    const int kg = a.k / a.groups;
    i = r * a.groups + t / kg;                  // the row group that decoded this token
    mg = (t % kg) * a.H + h;                    // its row within that group
    n = s_count[i];
  }
  // Rows past the batch (zero filled) and one-split rows come with the tile's
  // TMA load. Every thread still waits for it (ready()) before it arrives on
  // x_full: that load follows the MMAs of the tile two back, so no thread
  // arrives for a tile before the barrier's phase of the tile two back is
  // complete.
  if (tau >= a.T || n <= 1) return ready();
  const int start = s_start[i];
  if (start < 0 || start + n > a.slots) {       // not a plan of this shape: leave zeros
    if (a.status) atomicOr(a.status, MLA_FAULT_WORK_ITEM);
    if (!ready()) return false;
#pragma unroll
    for (int v = 0; v < 8; ++v) *reinterpret_cast<uint4*>(x + x_piece(row, 8 * v + c)) = zero;
    return true;
  }
  // LSEs of 8 splits at a time, one per thread of the row: max and weights by
  // shuffles within the 8.
  const unsigned grp = 0xFFu << (threadIdx.x & 24);
  const int base = threadIdx.x & 24;
  const float* lse = a.part_lse + (size_t)start * a.Mg + mg;
  float mx = -INFINITY;
  for (int g0 = 0; g0 < n; g0 += 8)
    if (g0 + c < n) mx = fmaxf(mx, lse[(size_t)(g0 + c) * a.Mg]);
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(grp, mx, o));
  const float4* po = reinterpret_cast<const float4*>(a.part_o + ((size_t)start * a.Mg + mg) * kDv);
  const size_t stride = (size_t)a.Mg * kDv / 4;  // float4s between splits
  float4 acc[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  for (int g0 = 0; g0 < n; g0 += 8) {
    const float l = g0 + c < n ? lse[(size_t)(g0 + c) * a.Mg] : -INFINITY;
    const float wc = (mx == -INFINITY || l == -INFINITY) ? 0.f : ex2(l - mx);
    z += wc;
    const int m = min(8, n - g0);
    // Two splits' partial rows in flight per round trip.
    for (int u = 0; u < m; u += 2) {
      const bool two = u + 1 < m;
      const float w0 = __shfl_sync(grp, wc, base + u);
      const float w1 = __shfl_sync(grp, wc, base + (two ? u + 1 : u));
      const float4* s0 = po + (size_t)(g0 + u) * stride;
      const float4* s1 = po + (size_t)(g0 + (two ? u + 1 : u)) * stride;
      float4 x0[16], x1[16];                   // x1 repeats x0 (weight 0) when m is odd
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        x0[v] = s0[8 * v + c];
        x1[v] = s1[8 * v + c];
      }
      const float v1 = two ? w1 : 0.f;
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        acc[v].x += w0 * x0[v].x + v1 * x1[v].x; acc[v].y += w0 * x0[v].y + v1 * x1[v].y;
        acc[v].z += w0 * x0[v].z + v1 * x1[v].z; acc[v].w += w0 * x0[v].w + v1 * x1[v].w;
      }
    }
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) z += __shfl_xor_sync(grp, z, o);
  const float sc = z > 0.f ? a.bmm2 / z : 0.f;
  // float4 8 v + c holds latent dims 4 (8 v + c) ..: half (c & 1) of the 16-byte
  // BF16 piece 4 v + c / 2.
  if (!ready()) return false;
#pragma unroll
  for (int v = 0; v < 16; ++v) {
    const float4 u = acc[v];
    const uint2 b = make_uint2((uint32_t)f32_to_bf16_bits(u.x * sc) |
                                   ((uint32_t)f32_to_bf16_bits(u.y * sc) << 16),
                               (uint32_t)f32_to_bf16_bits(u.z * sc) |
                                   ((uint32_t)f32_to_bf16_bits(u.w * sc) << 16));
    *reinterpret_cast<uint2*>(x + x_piece(row, 4 * v + (c >> 1)) + (c & 1) * 8) = b;
  }
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
uv_kernel(const UvArgs a, const __grid_constant__ CUtensorMap tm_w,
          const __grid_constant__ CUtensorMap tm_x) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  UvCtl* ctl = reinterpret_cast<UvCtl*>(smem + kOffBar);
  int* s_start = reinterpret_cast<int*>(smem + kOffStart);
  int* s_count = reinterpret_cast<int*>(smem + kOffCount);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This CTA's tiles: a contiguous, head-major range of (head, token block).
  const int nblk = (int)cdiv(a.T, kTok);
  const long long ntiles = (long long)nblk * a.H;
  const int t_begin = (int)(ntiles * blockIdx.x / gridDim.x);
  const int t_end = (int)(ntiles * (blockIdx.x + 1) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int c = 0; c < kChunks; ++c) tc::mbar_init(&ctl->w_full[c], 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->x_full[b], kRed);
      tc::mbar_init(&ctl->x_tma[b], 1);
      tc::mbar_init(&ctl->x_empty[b], 1);
      tc::mbar_init(&ctl->d_full[b], 1);
      tc::mbar_init(&ctl->d_empty[b], 128);
    }
    tc::mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tm_w);
      tc::prefetch_tmap(&tm_x);
    }
    tc::tmem_alloc(&ctl->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  for (int i = threadIdx.x; i < a.plan_rows; i += blockDim.x) s_start[i] = -1;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;

  // Before the wait for the decode, on SMs the decode has left: the first
  // head's W_UV (an input no kernel of the chain writes) and the scan of the
  // plan's work list (every decode CTA passed its own wait for the plan's
  // completion before this grid could launch; L2 reads, no stale L1 line).
  int cur_h = -1, loads = 0;   // the W_UV head in shared memory, loads issued
  if (warp == 0 && lane == 0 && t_begin < t_end) {
    cur_h = t_begin / nblk;
    for (int c = 0; c < kChunks; ++c) {
      tc::mbar_arrive_expect_tx(&ctl->w_full[c], kWChunk);
      tc::tma_load_2d(smem + kOffW + c * kWChunk, &tm_w, &ctl->w_full[c], c * 128,
                      cur_h * kOut);
    }
    loads = 1;
  }
  for (int i = threadIdx.x; i < a.plan_rows; i += blockDim.x) s_count[i] = __ldcg(a.counts + i);
  // First slot of every multi-split row group: split 0 followed by split 1 of
  // the same group at the head of the work list (multi-split items come first).
  const int scan = min(a.list_len, a.slots);
  for (int e = threadIdx.x; e + 1 < scan; e += blockDim.x) {
    const int w = __ldcg(a.work + e);
    if (w >= 0 && entry_split(w) == 0 && __ldcg(a.work + e + 1) == w + 1) {
      const int r = entry_request(w);
      if (r < a.plan_rows) s_start[r] = e;
    }
  }
  __syncthreads();

  grid_dep_wait();      // the decode's partials and one-split rows are complete
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      bool w_ready = false;
      int it = 0;
      // The one-split rows of tile `tile` into X buffer `b` (eight 64-dim chunks).
      auto load_x = [&](int tile, int b) {
        const int h = tile / nblk, tok0 = (tile % nblk) * kTok;
        tc::mbar_arrive_expect_tx(&ctl->x_tma[b], kXBytes);
        for (int c = 0; c < kChunks; ++c)
          tc::tma_load_3d(smem + kOffX + b * kXBytes + c * kXChunk, &tm_x, &ctl->x_tma[b],
                          c * 128, h, tok0);
      };
      int x_loads = 0;                         // tiles whose X load was issued
      if (t_begin < t_end) {
        load_x(t_begin, 0);
        x_loads = 1;
      }
      for (int tile = t_begin; ok && tile < t_end; ++tile, ++it) {
        const int h = tile / nblk, buf = it & 1;
        // The next tile's X goes to the other buffer once the MMAs of the
        // tile before this one (its last reader) are done.
        if (tile + 1 < t_end) {
          if (it >= 1 &&
              !(ok = uv_wait(&ctl->x_empty[(it - 1) & 1], ((it - 1) >> 1) & 1, ctl, a.status)))
            break;
          load_x(tile + 1, (it + 1) & 1);
          x_loads = it + 2;
        }
        if (h != cur_h) {
          // The previous tile's MMAs must be done reading W before it is replaced.
          if (it > 0 &&
              !(ok = uv_wait(&ctl->x_empty[(it - 1) & 1], ((it - 1) >> 1) & 1, ctl, a.status)))
            break;
          for (int c = 0; c < kChunks; ++c) {
            tc::mbar_arrive_expect_tx(&ctl->w_full[c], kWChunk);
            tc::tma_load_2d(smem + kOffW + c * kWChunk, &tm_w, &ctl->w_full[c], c * 128,
                            h * kOut);
          }
          ++loads;
          cur_h = h;
          w_ready = false;
        }
        if (!(ok = uv_wait(&ctl->x_tma[buf], (it >> 1) & 1, ctl, a.status))) break;
        if (!(ok = uv_wait(&ctl->x_full[buf], (it >> 1) & 1, ctl, a.status))) break;
        if (it >= 2 &&
            !(ok = uv_wait(&ctl->d_empty[buf], ((it - 2) >> 1) & 1, ctl, a.status)))
          break;
        tc::fence_after_sync();
        const uint32_t d = tmem + buf * kTok;
        for (int c = 0; ok && c < kChunks; ++c) {
          if (!w_ready && !(ok = uv_wait(&ctl->w_full[c], (loads - 1) & 1, ctl, a.status))) break;
          tc::fence_after_sync();
          const uint32_t wa = tc::smem_u32(smem + kOffW + c * kWChunk);
          const uint32_t xa = tc::smem_u32(smem + kOffX + buf * kXBytes + c * kXChunk);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16(d, tc::smem_desc(wa + kk * 32, 16, 1024, tc::kSw128),
                         tc::smem_desc(xa + kk * 32, 16, 1024, tc::kSw128), kIdesc,
                         (c | kk) != 0);
        }
        if (!ok) break;
        w_ready = true;
        tc::mma_commit(&ctl->x_empty[buf]);
        tc::mma_commit(&ctl->d_full[buf]);
      }
      if (!ok) {                               // never leave with copies or MMAs in flight
        tc::mma_commit(&ctl->drain);
        const unsigned long long t0 = tc::globaltimer_ns();
        if (loads > 0)
          for (int c = 0; c < kChunks; ++c)
            while (!tc::mbar_try_wait(&ctl->w_full[c], (loads - 1) & 1) &&
                   tc::globaltimer_ns() - t0 < kTimeoutNs) {
            }
        for (int j = x_loads - 2 < 0 ? 0 : x_loads - 2; j < x_loads; ++j)
          while (!tc::mbar_try_wait(&ctl->x_tma[j & 1], (j >> 1) & 1) &&
                 tc::globaltimer_ns() - t0 < kTimeoutNs) {
          }
        while (!tc::mbar_try_wait(&ctl->drain, 0) && tc::globaltimer_ns() - t0 < kTimeoutNs) {
        }
      }
    }
  } else {
    const int rt = threadIdx.x - 32;
    const int row = rt >> 3, c = rt & 7;        // token row of a tile, this thread's eighth
    const bool reads_back = warp <= 4;          // four warps: one TMEM lane quarter each
    const int q = warp & 3;
    bool ok = true;
    auto read_back = [&](int tile, int it) {
      const int h = tile / nblk, tok0 = (tile % nblk) * kTok, buf = it & 1;
      if (!(ok = uv_wait(&ctl->d_full[buf], (it >> 1) & 1, ctl, a.status))) return;
      tc::fence_after_sync();
      uint32_t raw[32];
      tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * kTok, raw);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      tc::mbar_arrive(&ctl->d_empty[buf]);
      const int j = q * 32 + lane;              // output dim = accumulator row = TMEM lane
#pragma unroll
      for (int col = 0; col < kTok; ++col) {
        const int tau = tok0 + col;
        if (tau < a.T)
          a.y[((size_t)tau * a.H + h) * kOut + j] = f32_to_bf16_bits(__uint_as_float(raw[col]));
      }
    };
    int it = 0;
    for (int tile = t_begin; tile < t_end; ++tile, ++it) {
      const int h = tile / nblk, tok0 = (tile % nblk) * kTok, buf = it & 1;
      // A merged row overwrites the tile's TMA-loaded one: wait for that load
      // (issued once X[buf] was free) only after the row's loads are in flight.
      const int it_now = it;
      auto x_free = [&]() {
        return uv_wait(&ctl->x_tma[it_now & 1], (it_now >> 1) & 1, ctl, a.status);
      };
      if (!(ok = merged_row(a, s_start, s_count, tok0 + row, h, c, smem + kOffX + buf * kXBytes, row,
                            x_free)))
        break;
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&ctl->x_full[buf]);
      if (reads_back && it > 0) {
        read_back(tile - 1, it - 1);
        if (!ok) break;
      }
    }
    if (ok && reads_back && it > 0) read_back(t_end - 1, it - 1);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 uv_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

cudaError_t launch_uv(const mla_shape& s, const int32_t* counts, const int32_t* work,
                      int list_len, const float* part_o, const float* part_lse, int slots,
                      float bmm2, const uint16_t* out, const uint16_t* w_uv, uint16_t* y,
                      int32_t* status, cudaStream_t st) {
  // W_UV as bytes: H * 128 rows of 1024 bytes (512 BF16 latent values each).
  CUtensorMap tm;
  auto fn = uv_encode_fn();
  if (!fn) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)kDv * 2, (cuuint64_t)s.H * kOut};
  const cuuint64_t strides[1] = {(cuuint64_t)kDv * 2};
  const cuuint32_t box[2] = {128, kOut}, es[2] = {1, 1};
  if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint16_t*>(w_uv), dims, strides, box,
         es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // The decode's BF16 rows as [token][head][512]: one box = 32 tokens x 64
  // dims (128 bytes) of one head, rows past the batch zero filled.
  CUtensorMap tmx;
  const cuuint64_t xdims[3] = {(cuuint64_t)kDv * 2, (cuuint64_t)s.H,
                               (cuuint64_t)s.R * s.k};
  const cuuint64_t xstrides[2] = {(cuuint64_t)kDv * 2, (cuuint64_t)s.H * kDv * 2};
  const cuuint32_t xbox[3] = {128, 1, kTok}, xes[3] = {1, 1, 1};
  if (fn(&tmx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint16_t*>(out), xdims, xstrides,
         xbox, xes, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(uv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  UvArgs a;
  a.counts = counts;
  a.work = work;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.out = out;
  a.y = y;
  a.status = status;
  a.bmm2 = bmm2;
  a.list_len = list_len;
  a.slots = slots;
  a.plan_rows = plan_rows(s);
  a.k = s.k;
  a.H = s.H;
  a.groups = shape_groups(s);
  a.M = s.k * s.H;
  a.Mg = group_rows(s);
  a.T = s.R * s.k;
  cudaLaunchConfig_t cfg = {};
  const long long ntiles = cdiv(a.T, kTok) * (long long)s.H;
  cfg.gridDim = dim3((unsigned)(ntiles < s.num_ctas ? ntiles : s.num_ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, uv_kernel, a, tm, tmx);
}

}  // namespace mlafold
