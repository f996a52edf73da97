// The split-KV reduction fused with the W_UV up-projection: every (token,
// head) row's merged 512-dim latent output, rounded once to BF16, times that
// head's W_UV [512, 128] on the tensor cores (BF16 operands, FP32
// accumulation), rounded to BF16 (drafter-attention page, `DraftDcp`: the head
// owner merges its heads' rows by exp2(lse - max) / sum in FP32 with one BF16
// rounding and applies W_UV as a BF16 MMA; `latent_major`: W_UV stored
// latent-contiguous). The merged 512-dim rows never reach HBM.
//
// One CTA per (32-token block, head). The 128 W_UV output dims are the MMA's
// M and the 32 tokens its N ("swap-AB": 32 tokens keep even the smallest
// batches spread over many SMs):
//     Y^T[128, 32] = W_UV[h]^T[128, 512] . X[32, 512]^T,  8 chunks x 4 MMAs (K = 16)
// X, the CTA's 32 merged BF16 rows, is built in shared memory by 256 reducer
// threads (8 per token row, 64 latent dims each): from the decode's own BF16
// row for a request with one split, else from the FP32 split partials and
// their LSEs. W_UV[h]'s eight 64-dim chunks stream in by TMA through two
// stages. The accumulator lives in 32 TMEM columns; four warps read it back
// and store Y.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace mlafold {
namespace {

constexpr int kTok = 32;                       // tokens per CTA: the MMA's N
constexpr int kOut = 128;                      // W_UV output dims: the MMA's M
constexpr int kChunks = kDv / 64;              // 64 latent dims = 128 B of BF16 per chunk
constexpr int kRed = 256;                      // reducer threads: 8 per token row
constexpr int kThreads = 32 + kRed;            // warp 0: TMA + MMA + TMEM owner
constexpr int kWStage = kOut * 128;            // one W chunk: 128 rows x 128 B
constexpr int kXChunk = kTok * 128;            // one X chunk: 32 rows x 128 B
constexpr int kOffW = 0;                       // two W stages
constexpr int kOffX = 2 * kWStage;             // X, eight chunks
constexpr int kOffStart = kOffX + kChunks * kXChunk;   // first slot of each multi-split row
constexpr int kOffBar = kOffStart + kMaxR * 4;
constexpr int kSmemBytes = kOffBar + 128 + 1024;        // + control block, + alignment slack
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kOut, kTok);
constexpr unsigned long long kTimeoutNs = 2000000000ull;
static_assert(kOffX % 1024 == 0 && kXChunk % 1024 == 0, "swizzle atoms need 1 KB alignment");

struct UvCtl {
  uint64_t w_full[2];   // TMA -> MMA: W chunk landed
  uint64_t w_free[2];   // MMA -> TMA: the chunk's MMAs finished reading the stage
  uint64_t x_full;      // reducers -> MMA: X written
  uint64_t d_full;      // MMA -> epilogue: accumulator final
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

// X chunk c, row `row`, is K-major with the 128-byte swizzle: its 16-byte
// piece p lives at ((p ^ (row & 7)) * 16) of the row's 128 bytes.
__device__ __forceinline__ void put_piece(uint8_t* xrow, int row, int p, uint4 v) {
  *reinterpret_cast<uint4*>(xrow + ((p ^ (row & 7)) * 16)) = v;
}

// Writes the BF16 values [64 c, 64 c + 64) of one token row's merged output
// into its row of X chunk c.
__device__ __forceinline__ void merged_chunk(const UvArgs& a, const int* s_start, int tau, int h,
                                             int c, uint8_t* xrow, int row) {
  const uint4 zero = make_uint4(0, 0, 0, 0);
  int n = 0, r = 0, t = 0, i = 0, mg = 0;
  if (tau < a.T) {
    r = tau / a.k;
    t = tau - r * a.k;
    const int kg = a.k / a.groups;
    i = r * a.groups + t / kg;                  // the row group that decoded this token
    mg = (t % kg) * a.H + h;                    // its row within that group
    n = a.counts[i];
  }
  if (tau >= a.T) {                             // rows past the batch stay zero
#pragma unroll
    for (int p = 0; p < 8; ++p) put_piece(xrow, row, p, zero);
    return;
  }
  if (n <= 1) {                                 // one split: the decode's BF16 row
    const uint4* src = reinterpret_cast<const uint4*>(
        a.out + ((size_t)r * a.M + (size_t)t * a.H + h) * kDv + c * 64);
    uint4 v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) v[p] = src[p];
#pragma unroll
    for (int p = 0; p < 8; ++p) put_piece(xrow, row, p, v[p]);
    return;
  }
  const int start = s_start[i];
  if (start < 0 || start + n > a.slots) {       // not a plan of this shape: leave zeros
    if (a.status) atomicOr(a.status, MLA_FAULT_WORK_ITEM);
#pragma unroll
    for (int p = 0; p < 8; ++p) put_piece(xrow, row, p, zero);
    return;
  }
  const float* lse = a.part_lse + (size_t)start * a.Mg + mg;
  float mx = -INFINITY;
  for (int s = 0; s < n; ++s) mx = fmaxf(mx, lse[(size_t)s * a.Mg]);
  const float* po = a.part_o + ((size_t)start * a.Mg + mg) * kDv + c * 64;
  const size_t stride = (size_t)a.Mg * kDv;
  float4 acc[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  for (int s = 0; s < n; ++s) {
    const float4* src = reinterpret_cast<const float4*>(po + s * stride);
    float4 x[16];
#pragma unroll
    for (int v = 0; v < 16; ++v) x[v] = src[v];
    const float l = lse[(size_t)s * a.Mg];
    const float w = (mx == -INFINITY || l == -INFINITY) ? 0.f : ex2(l - mx);
    z += w;
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      acc[v].x += w * x[v].x; acc[v].y += w * x[v].y;
      acc[v].z += w * x[v].z; acc[v].w += w * x[v].w;
    }
  }
  const float sc = z > 0.f ? a.bmm2 / z : 0.f;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const float4 u = acc[2 * p], w = acc[2 * p + 1];
    put_piece(xrow, row, p,
              make_uint4((uint32_t)f32_to_bf16_bits(u.x * sc) |
                             ((uint32_t)f32_to_bf16_bits(u.y * sc) << 16),
                         (uint32_t)f32_to_bf16_bits(u.z * sc) |
                             ((uint32_t)f32_to_bf16_bits(u.w * sc) << 16),
                         (uint32_t)f32_to_bf16_bits(w.x * sc) |
                             ((uint32_t)f32_to_bf16_bits(w.y * sc) << 16),
                         (uint32_t)f32_to_bf16_bits(w.z * sc) |
                             ((uint32_t)f32_to_bf16_bits(w.w * sc) << 16)));
  }
}

__global__ void __launch_bounds__(kThreads, 1)
uv_kernel(const UvArgs a, const __grid_constant__ CUtensorMap tm_w) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  UvCtl* ctl = reinterpret_cast<UvCtl*>(smem + kOffBar);
  int* s_start = reinterpret_cast<int*>(smem + kOffStart);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, tok0 = blockIdx.x * kTok;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&ctl->w_full[s], 1);
      tc::mbar_init(&ctl->w_free[s], 1);
    }
    tc::mbar_init(&ctl->x_full, kRed);
    tc::mbar_init(&ctl->d_full, 1);
    ctl->abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    if (lane == 0) tc::prefetch_tmap(&tm_w);
    tc::tmem_alloc(&ctl->tmem_base, 32);
    tc::tmem_relinquish();
  }
  for (int i = threadIdx.x; i < a.plan_rows; i += blockDim.x) s_start[i] = -1;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;

  grid_dep_wait();      // the decode's partials and one-split rows are complete
  grid_dep_launch();

  // First slot of every multi-split row group: split 0 followed by split 1 of
  // the same group at the head of the work list (multi-split items come first).
  const int scan = min(a.list_len, a.slots);
  for (int e = threadIdx.x; e + 1 < scan; e += blockDim.x) {
    const int w = a.work[e];
    if (w >= 0 && (w & ((1 << kSplitBits) - 1)) == 0 && a.work[e + 1] == w + 1) {
      const int r = w >> kSplitBits;
      if (r < a.plan_rows) s_start[r] = e;
    }
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int last_parity[2] = {-1, -1};
      auto load_w = [&](int c) {
        const int st = c & 1;
        tc::mbar_arrive_expect_tx(&ctl->w_full[st], kWStage);
        tc::tma_load_2d(smem + kOffW + st * kWStage, &tm_w, &ctl->w_full[st], c * 128, h * kOut);
        last_parity[st] = (c >> 1) & 1;
      };
      load_w(0);
      load_w(1);
      ok = uv_wait(&ctl->x_full, 0, ctl, a.status);
      for (int c = 0; ok && c < kChunks; ++c) {
        const int st = c & 1;
        if (!(ok = uv_wait(&ctl->w_full[st], (c >> 1) & 1, ctl, a.status))) break;
        tc::fence_after_sync();
        const uint32_t wa = tc::smem_u32(smem + kOffW + st * kWStage);
        const uint32_t xa = tc::smem_u32(smem + kOffX + c * kXChunk);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tmem, tc::smem_desc(wa + kk * 32, 16, 1024, tc::kSw128),
                       tc::smem_desc(xa + kk * 32, 16, 1024, tc::kSw128), kIdesc, (c | kk) != 0);
        tc::mma_commit(&ctl->w_free[st]);
        if (c + 2 < kChunks) {
          if (!(ok = uv_wait(&ctl->w_free[st], (c >> 1) & 1, ctl, a.status))) break;
          load_w(c + 2);
        }
      }
      tc::mma_commit(&ctl->d_full);            // once every MMA above has finished
      if (!ok) {                               // never leave with copies in flight
        const unsigned long long t0 = tc::globaltimer_ns();
        for (int st = 0; st < 2; ++st)
          while (last_parity[st] >= 0 && !tc::mbar_try_wait(&ctl->w_full[st], last_parity[st]) &&
                 tc::globaltimer_ns() - t0 < kTimeoutNs) {
          }
        while (!tc::mbar_try_wait(&ctl->d_full, 0) && tc::globaltimer_ns() - t0 < kTimeoutNs) {
        }
      }
    }
  } else {
    const int rt = threadIdx.x - 32;
    const int row = rt >> 3, c = rt & 7;        // token row of the tile, its 64-dim chunk
    merged_chunk(a, s_start, tok0 + row, h, c, smem + kOffX + c * kXChunk + row * 128, row);
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(&ctl->x_full);

    if (warp <= 4) {                            // four warps: one TMEM lane quarter each
      const bool ok = uv_wait(&ctl->d_full, 0, ctl, a.status);
      tc::fence_after_sync();
      const int q = warp & 3;
      const int j = q * 32 + lane;              // output dim = accumulator row = TMEM lane
      uint32_t raw[32];
      tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16), raw);
      tc::tmem_wait_ld();
      if (ok && !*reinterpret_cast<volatile int*>(&ctl->abort_flag)) {
#pragma unroll
        for (int col = 0; col < kTok; ++col) {
          const int tau = tok0 + col;
          if (tau < a.T)
            a.y[((size_t)tau * a.H + h) * kOut + j] = f32_to_bf16_bits(__uint_as_float(raw[col]));
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 32);
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
  cfg.gridDim = dim3((unsigned)cdiv(a.T, kTok), (unsigned)s.H);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, uv_kernel, a, tm);
}

}  // namespace mlafold
