// Split-KV FP8 MLA decode with the query rows as the tcgen05 M dimension, for
// requests of M = k*H >= 128 folded rows (the tensor-bound shapes).
//
// Same computation as decode_tc.cu (drafter-attention page, module overview
// and `folded_decode`; balanced-MLA page, module overview): each work item's
// split of the keys, softmax in base 2 with the +8 lazy max (moved to 2 below the
// tile's max), P as two E4M3
// terms, FP32 normaliser, BF16 out + log2 LSE or FP32 partial + LSE.
//
// Layout (ours): a job is (work item, 128-row block, half of the 512 output
// dims); the two halves of a row block run on two CTAs that read the same KV
// tiles (the second from L2). Per 128-key tile:
//     S[128 rows, 128 keys] = Q[128, 576] . K[128, 576]^T   18 MMAs, N = 128
//     O[128, 256 dims]     += P[128, 128] . V[128, 256]    8 MMAs, N = 256
// with P (hi and lo E4M3 terms) written by the softmax into tensor memory over
// the S buffer it came from and read from there as the A operand. TMEM: O half
// in columns 0..255, two S/P buffers of 128 columns. Two threads own a query
// row (64 keys and 128 output dims each), so the row max, the lazy rescale and
// the row sum need no reduction beyond exchanging the pair's tile maxima and
// row sums. Wide MMAs (N >= 128) run near the FP8 rate, where the N = 32/64
// MMAs of decode_tc.cu sit on the per-instruction floor.
#include "decode_common.cuh"

namespace mlafold {
namespace {

using namespace dec;

constexpr int kQRows = 128;
constexpr int kQChunk = kQRows * 128;
constexpr int kOffQ = kStages * kStageBytes;      // Q block after the KV ring
constexpr int kOffCtl = kOffQ + kQRows * kDqk;
constexpr int kHalfDims = 256;                    // output dims per CTA
constexpr int kSBuf = 256;                        // S/P buffers at TMEM columns 256, 384
constexpr uint32_t kIdescS = tc::idesc_e4m3_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = tc::idesc_e4m3_f32(128, 256, false, true);
constexpr int kRowsThreads = 320;                 // warp 0 TMA, warp 1 MMA, warps 2-9 softmax
constexpr int kGroup = 256;                       // two threads per query row

// Row-max exchange (double-buffered by tile parity) and row-sum halves of the
// two threads that share a query row; after the control block.
struct RowsXchg {
  float tmax[2][2][kQRows];
  float lsum[2][kQRows];
};

__device__ __forceinline__ void group256_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// ---------------------------------------------------------------- MMA issuer
__device__ void rows_mma_issuer(const DecodeArgs& a, uint8_t* smem, Ctl* ctl, uint32_t tmem,
                                int nb) {
  const uint32_t s_kv = tc::smem_u32(smem), s_q = tc::smem_u32(smem + kOffQ);
  uint32_t g = 0, x = 0;
  bool ok = true;

  auto issue_s = [&](uint32_t gg) {
    const int st = gg & 1;
    const uint32_t d = tmem + kSBuf + st * 128;
    const uint32_t kv = s_kv + st * kStageBytes;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_e4m3(d, tc::smem_desc(s_q + c * kQChunk + kk * 32, 16, 1024, tc::kSw128),
                     tc::smem_desc(kv + c * kChunkBytes + kk * 32, 16, 1024, tc::kSw128),
                     kIdescS, (c | kk) != 0);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
      tc::mma_e4m3(d, tc::smem_desc(s_q + 4 * kQChunk + kk * 32, 16, 512, tc::kSw64),
                   tc::smem_desc(kv + 4 * kChunkBytes + kk * 32, 16, 512, tc::kSw64), kIdescS,
                   true);
    tc::mma_commit(&ctl->s_full[st]);
  };
  auto issue_pv = [&](uint32_t gg, bool first, int half) {
    const int st = gg & 1;
    // V rows of this half: two 128-dim bands, 16 KB apart; 8-key groups 1 KB apart.
    const uint32_t v = s_kv + st * kStageBytes + 2 * half * kChunkBytes;
    const uint32_t p = tmem + kSBuf + st * 128;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t vb = tc::smem_desc(v + kk * 32 * 128, kChunkBytes, 1024, tc::kSw128);
      tc::mma_e4m3_ts(tmem, p + kk * 8, vb, kIdescPV, !(first && kk == 0));   // hi term
      tc::mma_e4m3_ts(tmem, p + 32 + kk * 8, vb, kIdescPV, true);             // lo term
    }
    tc::mma_commit(&ctl->pv_done[st]);
  };

  for (uint32_t seq = 0; ok; ++seq) {
    Job jb;
    if (!(ok = take_job(ctl, seq, a.status, jb)) || jb.item < 0) break;
    const int sub = jb.blk;
    if (jb.skip || jb.ntiles == 0) continue;
    const int half = sub & 1;
    if (!(ok = wait_bar(&ctl->q_full, x & 1, ctl, a.status))) break;
    int ns = 0, npv = 0;
    unsigned long long t0 = 0;
    while (npv < jb.ntiles) {
      bool progress = false;
      if (npv < ns) {                              // PV first: it frees a KV stage
        const uint32_t gg = g + npv;
        const int st = gg & 1;
        if (tc::mbar_test_wait(&ctl->p_full[st], (gg >> 1) & 1) &&
            (npv > 0 || x == 0 || tc::mbar_test_wait(&ctl->o_empty, (x - 1) & 1))) {
          tc::fence_after_sync();
          issue_pv(gg, npv == 0, half);
          ++npv;
          progress = true;
        }
      }
      if (ns < jb.ntiles && ns <= npv + 1) {
        const uint32_t gg = g + ns;
        const int st = gg & 1;
        // The S/P buffer is free once the PV that read its P (tile gg-2) is done.
        if (tc::mbar_test_wait(&ctl->kv_full[st], (gg >> 1) & 1) &&
            (gg < 2 || tc::mbar_test_wait(&ctl->pv_done[st], ((gg >> 1) - 1) & 1))) {
          tc::fence_after_sync();
          issue_s(gg);
          if (ns == jb.ntiles - 1) tc::mma_commit(&ctl->q_empty);
          ++ns;
          progress = true;
        }
      }
      if (progress) {
        t0 = 0;
      } else {
        const unsigned long long now = tc::globaltimer_ns();
        if (t0 == 0) t0 = now;
        const bool expired = now - t0 > ctl->wait_limit_ns;
        if (*reinterpret_cast<volatile int*>(&ctl->abort_flag) || expired) {
          *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
          if (expired && a.status) atomicOr(a.status, MLA_FAULT_WAIT_TIMEOUT);
          ok = false;
          break;
        }
      }
    }
    if (!ok) break;
    tc::mma_commit(&ctl->o_full);
    g += jb.ntiles;
    ++x;
  }
  tc::mma_commit(&ctl->drain);
  const unsigned long long t0 = tc::globaltimer_ns();
  while (!tc::mbar_try_wait(&ctl->drain, 0) && tc::globaltimer_ns() - t0 < kTimeoutNs) {
  }
}

// ---------------------------------------------------------------- softmax + epilogue
// Eight warps, two threads per query row: warps 2-5 take keys 0..63 of every
// tile and output dims 0..127 of the CTA's half, warps 6-9 keys 64..127 and
// dims 128..255 (a warp may only touch its lane quarter of TMEM: warp & 3).
__device__ void rows_softmax_epilogue(const DecodeArgs& a, uint8_t* smem, Ctl* ctl,
                                      RowsXchg* xg, uint32_t tmem, int nb) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int kh = (warp - 2) >> 2;                 // which half of the keys / of the dims
  const int tl = quarter * 32 + lane;             // this thread's query row (and key row)
  const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
  uint32_t g = 0, x = 0;
  bool ok = true;

  for (uint32_t seq = 0; ok; ++seq) {
    Job jb;
    if (!(ok = take_job(ctl, seq, a.status, jb)) || jb.item < 0) break;
    const int sub = jb.blk;
    if (jb.skip) continue;
    const int half = sub & 1;
    const int m0 = (sub >> 1) * kQRows;
    const bool mine = m0 + tl < a.M;               // a real query row
    const long long orow = jb.direct ? ((long long)jb.r * a.M + m0 + tl)
                                     : ((long long)jb.item * a.M + m0 + tl);
    const int dcol = half * kHalfDims + kh * 128;  // first output dim of this thread
    if (jb.ntiles == 0) {                          // empty split: out 0, lse -inf
      if (mine) {
        if (jb.direct) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kDv + dcol);
          for (int c = 0; c < 128 * 2 / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          if (a.lse && half == 0 && kh == 0) a.lse[orow] = -INFINITY;
        } else {
          uint4* dst = reinterpret_cast<uint4*>(a.part_o + orow * kDv + dcol);
          for (int c = 0; c < 128 * 4 / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          if (half == 0 && kh == 0) a.part_lse[orow] = -INFINITY;
        }
      }
      continue;
    }
    float m = -INFINITY, l = 0.f;
    for (int t = 0; t < jb.ntiles; ++t) {
      const uint32_t gg = g + t;
      const int st = gg & 1;
      const uint32_t sbuf = tmem + lane_addr + kSBuf + st * 128;
      if (!(ok = wait_bar(&ctl->s_full[st], (gg >> 1) & 1, ctl, a.status))) break;
      tc::fence_after_sync();
      float xv[64];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t raw[32];
        tc::tmem_ld32(sbuf + kh * 64 + h * 32, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) xv[h * 32 + i] = __uint_as_float(raw[i]);
      }
      const int nvalid = min(kTileKeys, jb.j1 - (jb.j0 + t * kTileKeys)) - kh * 64;
      // Raw scores (masked past the split); the scale (> 0) is applied inside
      // the exponent, so the max is taken on raw scores, then over both halves.
      float smax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        xv[i] = i < nvalid ? xv[i] : -INFINITY;
        smax = fmaxf(smax, xv[i]);
      }
      xg->tmax[t & 1][kh][tl] = smax;
      group256_sync();
      smax = fmaxf(xg->tmax[t & 1][0][tl], xg->tmax[t & 1][1][tl]);
      const float tmax = smax * a.bmm1_log2;
      float alpha = 1.f;
      if (tmax > m + 8.f) {                        // the row's max moved by more than 8
        const float mn = tmax - kMaxLead;
        alpha = m == -INFINITY ? 0.f : ex2(m - mn);
        m = mn;
        l *= alpha;
      }
      // O holds tiles < gg: rows whose max moved scale their dims (whole warps
      // take part in the TMEM traffic; rows that did not move scale by 1).
      if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const uint32_t gp = gg - 1;
        if (!(ok = wait_bar(&ctl->pv_done[gp & 1], (gp >> 1) & 1, ctl, a.status))) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t raw[32];
          const uint32_t addr = tmem + lane_addr + kh * 128 + c0;
          tc::tmem_ld32(addr, raw);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
          tc::tmem_st32(addr, raw);
        }
        tc::tmem_wait_st();
      }
      // P = 2^(x - m) as two E4M3 terms over this S buffer: hi in columns
      // 0..31, lo in 32..63, four codes per column in key order; this thread
      // writes its 64 keys' 16 columns of each.
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          float p[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            p[u] = ex2(fmaf(xv[c * 32 + w * 4 + u], a.bmm1_log2, -m));
            l += p[u];
          }
          const uint32_t h01 = f32x2_to_f16x2(p[0], p[1]), h23 = f32x2_to_f16x2(p[2], p[3]);
          const uint16_t e01 = f16x2_to_e4m3x2(h01), e23 = f16x2_to_e4m3x2(h23);
          const uint16_t l01 = f16x2_to_e4m3x2(f16x2_sub(h01, e4m3x2_to_f16x2(e01)));
          const uint16_t l23 = f16x2_to_e4m3x2(f16x2_sub(h23, e4m3x2_to_f16x2(e23)));
          hi[w] = (uint32_t)e01 | ((uint32_t)e23 << 16);
          lo[w] = (uint32_t)l01 | ((uint32_t)l23 << 16);
        }
        tc::tmem_st8(sbuf + kh * 16 + c * 8, hi);
        tc::tmem_st8(sbuf + 32 + kh * 16 + c * 8, lo);
      }
      // Keys past the split: their V rows must be 0 in the two bands this
      // CTA's PV reads.
      if (kh == 0 && tl >= nvalid) {
        uint8_t* stage = smem + st * kStageBytes;
#pragma unroll
        for (int c = 2 * half; c < 2 * half + 2; ++c) {
          uint4* vrow = reinterpret_cast<uint4*>(stage + c * kChunkBytes + tl * 128);
#pragma unroll
          for (int u = 0; u < 8; ++u) vrow[u] = make_uint4(0, 0, 0, 0);
        }
        tc::fence_proxy_async_smem();
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive(&ctl->p_full[st]);
    }
    if (!ok) break;

    xg->lsum[kh][tl] = l;
    group256_sync();
    l = xg->lsum[0][tl] + xg->lsum[1][tl];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse2 = l > 0.f ? m + __log2f(l) : -INFINITY;
    if (!(ok = wait_bar(&ctl->o_full, x & 1, ctl, a.status))) break;
    tc::fence_after_sync();
    const float sc = inv * (jb.direct ? a.bmm2 : 1.f);
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t raw[32];
      tc::tmem_ld32(tmem + lane_addr + kh * 128 + c0, raw);
      tc::tmem_wait_ld();
      if (!mine) continue;
      if (jb.direct) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = (uint32_t)f32_to_bf16_bits(__uint_as_float(raw[2 * i]) * sc) |
                  ((uint32_t)f32_to_bf16_bits(__uint_as_float(raw[2 * i + 1]) * sc) << 16);
        uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kDv + dcol + c0);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      } else {
        float4* dst = reinterpret_cast<float4*>(a.part_o + orow * kDv + dcol + c0);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          dst[v] = make_float4(__uint_as_float(raw[4 * v]) * sc,
                               __uint_as_float(raw[4 * v + 1]) * sc,
                               __uint_as_float(raw[4 * v + 2]) * sc,
                               __uint_as_float(raw[4 * v + 3]) * sc);
      }
    }
    tc::fence_before_sync();
    tc::mbar_arrive(&ctl->o_empty);
    if (mine && half == 0 && kh == 0) {
      if (jb.direct) {
        if (a.lse) a.lse[orow] = lse2;        // one-split rows have no partial slot
      } else {
        a.part_lse[orow] = lse2;
      }
    }
    g += jb.ntiles;
    ++x;
  }
}

__global__ void __launch_bounds__(kRowsThreads, 1)
decode_rows_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_kv,
                   const __grid_constant__ CUtensorMap tm_kvr,
                   const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_qr, int nb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  RowsXchg* xg = reinterpret_cast<RowsXchg*>(smem + kOffCtl + sizeof(Ctl));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&ctl->kv_full[s], 1);
      tc::mbar_init(&ctl->pv_done[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->s_full[b], 1);
      tc::mbar_init(&ctl->s_empty[b], kGroup);
      tc::mbar_init(&ctl->p_full[b], kGroup);
    }
    tc::mbar_init(&ctl->q_full, 1);
    tc::mbar_init(&ctl->q_empty, 1);
    tc::mbar_init(&ctl->o_full, 1);
    tc::mbar_init(&ctl->o_empty, kGroup);
    tc::mbar_init(&ctl->drain, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->job_full[b], 1);
      tc::mbar_init(&ctl->job_empty[b], 1 + kGroup);   // the MMA thread + the softmax group
    }
    ctl->abort_flag = 0;
    ctl->wait_limit_ns = a.wait_limit_ns;
    tc::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tm_kv);
    tc::prefetch_tmap(&tm_kvr);
    tc::prefetch_tmap(&tm_q);
    tc::prefetch_tmap(&tm_qr);
  }
  if (warp == 1) {
    tc::tmem_alloc(&ctl->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;

  grid_dep_wait();      // the plan is complete; earlier readers of out/workspace are done
  grid_dep_launch();    // the reducer may launch; it still waits for this grid to finish
  if (warp == 0) {
    producer<kQRows, 2, kOffQ, false, true>(a, smem, ctl, nb, &tm_kv, &tm_kvr, &tm_q, &tm_qr);
  } else if (warp == 1) {
    if (lane == 0) rows_mma_issuer(a, smem, ctl, tmem, nb);
  } else {
    rows_softmax_epilogue(a, smem, ctl, xg, tmem, nb);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_decode_rows(const mla_shape& s, const DecodeArgs& a, cudaStream_t st) {
  CUtensorMap tkv, tkvr, tq, tqr;
  const cuuint64_t kv_dims[2] = {(cuuint64_t)kDqk, (cuuint64_t)a.num_pages * kPage};
  const cuuint64_t kv_str[1] = {(cuuint64_t)kDqk};
  const cuuint32_t kv_box[2] = {128, kPage}, kvr_box[2] = {64, kPage};
  const cuuint64_t q_dims[3] = {(cuuint64_t)kDqk, (cuuint64_t)a.M, (cuuint64_t)a.R};
  const cuuint64_t q_str[2] = {(cuuint64_t)kDqk, (cuuint64_t)a.M * kDqk};
  const cuuint32_t q_box[3] = {128, kQRows, 1}, qr_box[3] = {64, kQRows, 1};
  if (!encode(&tkv, a.kv, 2, kv_dims, kv_str, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode(&tkvr, a.kv, 2, kv_dims, kv_str, kvr_box, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode(&tq, a.q, 3, q_dims, q_str, q_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode(&tqr, a.q, 3, q_dims, q_str, qr_box, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const int smem_bytes = kOffCtl + (int)sizeof(Ctl) + (int)sizeof(RowsXchg) + 1024;
  static bool attr_set[64] = {};
  cudaError_t e = set_smem(decode_rows_kernel, smem_bytes, attr_set);
  if (e != cudaSuccess) return e;
  const int nb = row_blocks(a.M);
  const long long jobs = (long long)a.items * nb;
  const int grid = (int)(jobs < s.num_ctas ? jobs : s.num_ctas);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(kRowsThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_rows_kernel, a, tkv, tkvr, tq, tqr, nb);
}

}  // namespace mlafold
