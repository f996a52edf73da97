// Split-KV FP8 MLA decode on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// What it computes (drafter-attention page, module overview and
// `folded_decode`; balanced-MLA page, module overview): for each work item of
// the plan (request r, split s: keys [j0, j1)) and each block of NR query rows
// of the request's M = k*H folded rows, the split's softmax attention over the
// 576-dim latent keys with the 512-dim latent slice as the value, written as
// BF16 out + base-2 LSE (one split) or as an FP32 partial + LSE (several).
//
// Design (ours; the pages' kernels are prior art only):
// * Persistent CTAs, one per SM: CTA b takes (item, row block) job b, then
//   claims further jobs in list order from a counter (longest requests
//   first), so CTAs that finish early take more of the list; warp 0 claims
//   and hands each job to the other roles through a two-slot ring.
// * Swap-AB: keys are the MMA's M dimension (128 per tile = two pages) and
//   query rows its N, so M = k*H of 32..448 needs no padding to 128 and the
//   whole O^T accumulator (512 dims x N rows) plus two S^T buffers fit TMEM.
//     S^T[128 keys, NR]  = K[128, 576] . Q[NR, 576]^T   (18 MMAs, K-major)
//     O^T[512, NR(x2)]  += V^T[512, 128] . P^T[128, NR] (V = latent slice of
//                          the same shared-memory tile, read MN-major)
// * Warp roles: warp 0 issues TMA (per-page gathers through the block table
//   into a 2-stage ring of 128-key tiles; Q block once per job); warp 1 issues
//   the MMAs and owns TMEM; warps 2-9 (two 128-thread halves) own one key of
//   the tile each for the softmax and one value dim per 128-dim band for the
//   epilogue, the first half for query rows 0 .. NR/2 - 1 and the second for
//   the rest (16 rows per thread for NR = 32, 32 for NR = 64).
// * Softmax in base 2 with a lazily updated row max: the max moves only when a
//   new score exceeds it by more than 8 (P <= 2^8, balanced-MLA page, module
//   overview), and then to 2 below the tile's max (kMaxLead). P enters the PV
//   MMA as FP8 E4M3, unscaled, split into two E4M3 terms hi = e4m3(p16),
//   lo = e4m3(p16 - hi), p16 = fp16(p) (both FP8 operands: one E4M3 term alone misses the
//   +-(2e-2 + 2e-2|ref|) bound on short requests). The normaliser is the FP32
//   sum of p.
// * Every mbarrier wait is bounded (2 s); on expiry the CTA sets
//   MLA_FAULT_WAIT_TIMEOUT in the status word, stops, drains its own copies and
//   MMAs, frees TMEM and returns. No trap, no unbounded spin.
#include "decode_common.cuh"

namespace mlafold {
namespace {

using namespace dec;

template <int NR>
struct Cfg {
  static constexpr int kHalves = 2;               // 128-thread softmax groups per row block
  static constexpr int kRowsPerThread = NR / kHalves;
  static constexpr int kGroup = 128 * kHalves;    // softmax threads
  static constexpr int kThreads = 64 + kGroup;    // + the TMA warp and the MMA warp
  static constexpr int kQChunk = NR * 128;
  static constexpr int kQBytes = 4 * kQChunk + NR * 64;
  // P^T of a tile: one row per key holding the hi codes of the NR query rows,
  // then their lo codes (2*NR bytes: 64-byte swizzle for NR = 32, 128-byte for
  // NR = 64).
  static constexpr int kPRow = 2 * NR;
  static constexpr int kPBytes = kTileKeys * kPRow;
  static constexpr tc::Swizzle kPSw = NR == 32 ? tc::kSw64 : tc::kSw128;
  static constexpr int kPAtom = 8 * kPRow;        // 8-key group stride of P^T
  // O^T in TMEM, one 128-dim value band after another. A "split" band keeps
  // the hi and lo products in separate accumulators side by side (NR columns
  // each) so that one MMA of N = 2*NR covers both terms; the others take the
  // two terms as two N = NR MMAs into one accumulator. NR = 32: all four bands
  // split (256 columns) beside two S^T buffers. NR = 64: bands 0-2 split and
  // band 3 not (448 columns) beside one S^T buffer, which the softmax frees as
  // soon as it has read S into registers, before the next tile's S is usually
  // ready to issue anyway.
  static constexpr int kSplitBands = NR == 32 ? 4 : 3;
  static constexpr int kSBufs = NR == 32 ? 2 : 1;
  __host__ __device__ static constexpr bool split(int dt) { return dt < kSplitBands; }
  __host__ __device__ static constexpr int band_col(int dt) {
    return dt < kSplitBands ? dt * 2 * NR : kSplitBands * 2 * NR + (dt - kSplitBands) * NR;
  }
  static constexpr int kSCol = band_col(4);       // S^T buffers after O^T
  __host__ __device__ static constexpr int s_col(uint32_t gg) {
    return kSCol + (int)(gg % kSBufs) * NR;
  }
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffP = kOffQ + kQBytes;
  static constexpr int kOffCtl = kOffP + 2 * kPBytes;
  static constexpr uint32_t kIdescS = tc::idesc_e4m3_f32(128, NR, false, false);
  static constexpr uint32_t kIdescPVSplit = tc::idesc_e4m3_f32(128, 2 * NR, true, true);
  static constexpr uint32_t kIdescPVOne = tc::idesc_e4m3_f32(128, NR, true, true);
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms need 1 KB alignment");
  static_assert(kSCol + kSBufs * NR <= (int)kTmemCols, "TMEM budget");
};

// Reduce v[32] across the 32 lanes by halving exchanges (31 shuffles per
// lane instead of 160); afterwards lane l holds the reduction of row l in v[0].
template <int LEN, bool MAX>
__device__ __forceinline__ void tr_step(float* v, int lane, int o) {
  const bool upper = (lane & o) != 0;
#pragma unroll
  for (int i = 0; i < LEN / 2; ++i) {
    const float send = upper ? v[i] : v[i + LEN / 2];
    const float keep = upper ? v[i + LEN / 2] : v[i];
    const float recv = __shfl_xor_sync(0xffffffffu, send, o);
    v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
  }
}
// The same for v[16] (16 rows per thread): after four halving steps v[0]
// holds row (lane >> 1) reduced over the 16 lanes that share bit 0 of the
// lane index; one more exchange with lane ^ 1 completes it.
template <bool MAX>
__device__ __forceinline__ void transpose_reduce16(float* v, int lane) {
  tr_step<16, MAX>(v, lane, 16);
  tr_step<8, MAX>(v, lane, 8);
  tr_step<4, MAX>(v, lane, 4);
  tr_step<2, MAX>(v, lane, 2);
  const float r = __shfl_xor_sync(0xffffffffu, v[0], 1);
  v[0] = MAX ? fmaxf(v[0], r) : v[0] + r;
}
template <bool MAX>
__device__ __forceinline__ void transpose_reduce32(float* v, int lane) {
  tr_step<32, MAX>(v, lane, 16);
  tr_step<16, MAX>(v, lane, 8);
  tr_step<8, MAX>(v, lane, 4);
  tr_step<4, MAX>(v, lane, 2);
  tr_step<2, MAX>(v, lane, 1);
}

// Reduce this thread's RT row values across the warp's 32 keys and store row
// results in red[r0 + row] (RT = 32: lane l holds row l; RT = 16: row l >> 1).
template <int RT, bool MAX>
__device__ __forceinline__ void reduce_rows(float* v, int lane, float* red_row0) {
  if constexpr (RT == 32) {
    transpose_reduce32<MAX>(v, lane);
    red_row0[lane] = v[0];
  } else {
    transpose_reduce16<MAX>(v, lane);
    if ((lane & 1) == 0) red_row0[lane >> 1] = v[0];
  }
}
// RT consecutive 32-bit TMEM columns of this thread's lane.
template <int RT>
__device__ __forceinline__ void tmem_ld_rows(uint32_t taddr, uint32_t (&r)[RT]) {
  if constexpr (RT == 32) tc::tmem_ld32(taddr, r); else tc::tmem_ld16(taddr, r);
}
template <int RT>
__device__ __forceinline__ void tmem_st_rows(uint32_t taddr, const uint32_t (&r)[RT]) {
  if constexpr (RT == 32) tc::tmem_st32(taddr, r); else tc::tmem_st16(taddr, r);
}

// ---------------------------------------------------------------- MMA issuer
template <int NR, bool HALVES>
__device__ void mma_issuer(const DecodeArgs& a, uint8_t* smem, Ctl* ctl, uint32_t tmem, int nb) {
  using C = Cfg<NR>;
  const uint32_t s_kv = tc::smem_u32(smem), s_q = tc::smem_u32(smem + C::kOffQ);
  const uint32_t s_p = tc::smem_u32(smem + C::kOffP);
  uint32_t g = 0, x = 0;
  bool ok = true;

  auto issue_s = [&](uint32_t gg) {
    const int st = gg & 1;
    const uint32_t d = tmem + C::s_col(gg);
    const uint32_t kv = s_kv + st * kStageBytes;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_e4m3(d, tc::smem_desc(kv + c * kChunkBytes + kk * 32, 16, 1024, tc::kSw128),
                     tc::smem_desc(s_q + c * C::kQChunk + kk * 32, 16, 1024, tc::kSw128),
                     C::kIdescS, (c | kk) != 0);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
      tc::mma_e4m3(d, tc::smem_desc(kv + 4 * kChunkBytes + kk * 32, 16, 512, tc::kSw64),
                   tc::smem_desc(s_q + 4 * C::kQChunk + kk * 32, 16, 512, tc::kSw64),
                   C::kIdescS, true);
    tc::mma_commit(&ctl->s_full[st]);
  };

  auto issue_pv = [&](uint32_t gg, bool first) {
    const int st = gg & 1;
    const uint32_t kv = s_kv + st * kStageBytes;
    const uint32_t p = s_p + st * C::kPBytes;
#pragma unroll
    for (int dt = 0; dt < 4; ++dt) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // V^T band dt, keys 32kk..32kk+31: MN-major, 8-key groups 1 KB apart.
        const uint64_t va = tc::smem_desc(kv + dt * kChunkBytes + kk * 32 * 128, kChunkBytes,
                                          1024, tc::kSw128);
        // P^T rows of these 32 keys: the hi codes, then the lo codes, of NR rows.
        const uint32_t pk = p + kk * 32 * C::kPRow;
        const bool acc = !(first && kk == 0);
        if (C::split(dt)) {          // one N = 2*NR MMA: hi and lo accumulate apart
          tc::mma_e4m3(tmem + C::band_col(dt), va,
                       tc::smem_desc(pk, C::kPBytes, C::kPAtom, C::kPSw), C::kIdescPVSplit, acc);
        } else {                     // two N = NR MMAs into one accumulator
          tc::mma_e4m3(tmem + C::band_col(dt), va,
                       tc::smem_desc(pk, C::kPBytes, C::kPAtom, C::kPSw), C::kIdescPVOne, acc);
          tc::mma_e4m3(tmem + C::band_col(dt), va,
                       tc::smem_desc(pk + NR, C::kPBytes, C::kPAtom, C::kPSw), C::kIdescPVOne,
                       true);
        }
      }
      // The producer refills bands 0-1 as soon as they are free (HALVES).
      if constexpr (HALVES) if (dt == 1) tc::mma_commit(&ctl->pv_half[st]);
    }
    tc::mma_commit(&ctl->pv_done[st]);
  };

  for (uint32_t seq = 0; ok; ++seq) {
    Job jb;
    if (!(ok = take_job(ctl, seq, a.status, jb)) || jb.item < 0) break;
    if (jb.skip || jb.ntiles == 0) continue;
    if (!(ok = wait_bar(&ctl->q_full, x & 1, ctl, a.status))) break;
    // Issue S(t) as soon as its tile landed and its S buffer is free, and PV(t)
    // as soon as P(t) is written: neither waits on the other's inputs. S runs
    // at most one tile ahead of PV (two S buffers).
    int ns = 0, npv = 0;
    unsigned long long t0 = 0;
    while (npv < jb.ntiles) {
      bool progress = false;
      // PV first: its completion frees a KV stage for the next TMA.
      if (npv < ns) {
        const uint32_t gg = g + npv;
        const int st = gg & 1;
        if (tc::mbar_test_wait(&ctl->p_full[st], (gg >> 1) & 1) &&
            (npv > 0 || x == 0 || tc::mbar_test_wait(&ctl->o_empty, (x - 1) & 1))) {
          tc::fence_after_sync();
          issue_pv(gg, npv == 0);
          ++npv;
          progress = true;
        }
      }
      if (ns < jb.ntiles && ns <= npv + 1) {
        const uint32_t gg = g + ns;
        const int st = gg & 1;
        // Its S^T buffer is free once the softmax read the S that used it last
        // (tile gg - kSBufs; s_empty is indexed by tile parity).
        const uint32_t gp = gg - C::kSBufs;
        if (tc::mbar_test_wait(&ctl->kv_full[st], (gg >> 1) & 1) &&
            (gg < (uint32_t)C::kSBufs ||
             tc::mbar_test_wait(&ctl->s_empty[gp & 1], (gp >> 1) & 1))) {
          tc::fence_after_sync();
          issue_s(gg);
          if (ns == jb.ntiles - 1) tc::mma_commit(&ctl->q_empty);   // every S of the job issued
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
  // Wait for every MMA this thread issued before TMEM is released.
  tc::mma_commit(&ctl->drain);
  const unsigned long long t0 = tc::globaltimer_ns();
  while (!tc::mbar_try_wait(&ctl->drain, 0) && tc::globaltimer_ns() - t0 < kTimeoutNs) {
  }
}

// ---------------------------------------------------------------- softmax + epilogue
// The softmax group: two 128-thread halves on the same keys, one thread per
// key of the tile and per NR/2 query rows (16 or 32 rows per thread).
template <int G>
__device__ __forceinline__ void group_sync_n() {
  asm volatile("bar.sync 1, %0;" ::"n"(G) : "memory");
}
template <int G>
__device__ __forceinline__ bool group_any_n(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 2, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(G)
      : "memory");
  return r != 0;
}

template <int NR>
__device__ void softmax_epilogue(const DecodeArgs& a, uint8_t* smem, Ctl* ctl, uint32_t tmem,
                                 int nb) {
  using C = Cfg<NR>;
  constexpr int G = C::kGroup;
  constexpr int RT = C::kRowsPerThread;           // 32 or 16
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;                   // TMEM lanes this warp may access
  const int tl = quarter * 32 + lane;             // key of the tile / dim of a band
  const int half = C::kHalves == 1 ? 0 : (warp - 2) >> 2;   // which RT query rows
  const int r0 = half * RT;
  const int gt = threadIdx.x - 64;                // 0..G-1 within the group
  const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
  uint32_t g = 0, x = 0;
  bool ok = true;
  float lp[RT];                                   // this key's share of its rows' sums

  for (uint32_t seq = 0; ok; ++seq) {
    Job jb;
    if (!(ok = take_job(ctl, seq, a.status, jb)) || jb.item < 0) break;
    const int blk = jb.blk;
    if (jb.skip) continue;
    const int m0 = blk * NR;
    const int rows = min(NR, a.M - m0);
    if (jb.ntiles == 0) {                          // empty split: out 0, lse -inf
      for (int i = 0; i < rows; ++i)
        for (int d = gt; d < kDv; d += G) {
          if (jb.direct)
            a.out[((long long)jb.r * a.M + m0 + i) * kDv + d] = 0;
          else
            a.part_o[((long long)jb.item * a.M + m0 + i) * kDv + d] = 0.f;
        }
      if (gt < rows) {
        // One-split rows have no partial slot: without an LSE output there is
        // nothing to write for them.
        if (jb.direct) {
          if (a.lse) a.lse[(long long)jb.r * a.M + m0 + gt] = -INFINITY;
        } else {
          a.part_lse[(long long)jb.item * a.M + m0 + gt] = -INFINITY;
        }
      }
      continue;
    }
    group_sync_n<G>();                             // previous job's readers are done
    if (gt < NR) ctl->m_run[gt] = -INFINITY;
#pragma unroll
    for (int i = 0; i < RT; ++i) lp[i] = 0.f;
    group_sync_n<G>();

    for (int t = 0; t < jb.ntiles; ++t) {
      const uint32_t gg = g + t;
      const int st = gg & 1;
      if (!(ok = wait_bar(&ctl->s_full[st], (gg >> 1) & 1, ctl, a.status))) break;
      tc::fence_after_sync();
      float xv[RT];
      {
        uint32_t raw[RT];
        tmem_ld_rows<RT>(tmem + lane_addr + C::s_col(gg) + r0, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < RT; ++i) xv[i] = __uint_as_float(raw[i]);
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&ctl->s_empty[st]);
      const bool valid = jb.j0 + t * kTileKeys + tl < jb.j1;
      bool exceed = false;
#pragma unroll
      for (int i = 0; i < RT; ++i) {
        xv[i] = valid ? xv[i] * a.bmm1_log2 : -INFINITY;
        exceed |= xv[i] > ctl->m_run[r0 + i] + 8.f;
      }
      if (group_any_n<G>(exceed)) {
        // Rows whose max grew by more than 8: the new max is kMaxLead below the tile's.
        {
          float v[RT];
#pragma unroll
          for (int i = 0; i < RT; ++i) v[i] = xv[i];
          reduce_rows<RT, true>(v, lane, &ctl->red[quarter][r0]);
        }
        group_sync_n<G>();
        if (gt < NR) {
          const float tm = fmaxf(fmaxf(ctl->red[0][gt], ctl->red[1][gt]),
                                 fmaxf(ctl->red[2][gt], ctl->red[3][gt]));
          const float mo = ctl->m_run[gt];
          const float mn = tm > mo + 8.f ? tm - kMaxLead : mo;
          ctl->vec[gt] = mo == -INFINITY ? 0.f : ex2(mo - mn);
          ctl->m_run[gt] = mn;
        }
        group_sync_n<G>();
#pragma unroll
        for (int i = 0; i < RT; ++i) lp[i] *= ctl->vec[r0 + i];
        if (t > 0) {
          // O^T holds tiles < gg: wait for the last PV, then scale this
          // thread's rows' columns (32-row kernel: in both the hi and the lo
          // columns).
          const uint32_t gp = gg - 1;
          if (!(ok = wait_bar(&ctl->pv_done[gp & 1], (gp >> 1) & 1, ctl, a.status))) break;
          tc::fence_after_sync();
#pragma unroll
          for (int dt = 0; dt < 4; ++dt) {
#pragma unroll
            for (int h = 0; h < (C::split(dt) ? 2 : 1); ++h) {
              uint32_t raw[RT];
              const uint32_t addr = tmem + lane_addr + C::band_col(dt) + h * NR + r0;
              tmem_ld_rows<RT>(addr, raw);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < RT; ++i)
                raw[i] = __float_as_uint(__uint_as_float(raw[i]) * ctl->vec[r0 + i]);
              tmem_st_rows<RT>(addr, raw);
            }
          }
          tc::tmem_wait_st();
        }
      }
      // P buffer st is free: PV(gg - 2), the last reader of this buffer and of
      // KV stage st, finished before the producer refilled that stage with
      // tile gg, whose S this thread has just read.
      uint32_t hi[RT / 4], lo[RT / 4];
#pragma unroll
      for (int i = 0; i < RT; i += 4) {
        float p[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          p[u] = ex2(xv[i + u] - ctl->m_run[r0 + i + u]);
          lp[i + u] += p[u];
        }
        const uint32_t h01 = f32x2_to_f16x2(p[0], p[1]), h23 = f32x2_to_f16x2(p[2], p[3]);
        const uint16_t e01 = f16x2_to_e4m3x2(h01), e23 = f16x2_to_e4m3x2(h23);
        const uint16_t l01 = f16x2_to_e4m3x2(f16x2_sub(h01, e4m3x2_to_f16x2(e01)));
        const uint16_t l23 = f16x2_to_e4m3x2(f16x2_sub(h23, e4m3x2_to_f16x2(e23)));
        hi[i / 4] = (uint32_t)e01 | ((uint32_t)e23 << 16);
        lo[i / 4] = (uint32_t)l01 | ((uint32_t)l23 << 16);
      }
      // P^T row of this key, MN-major: kPRow bytes (the hi codes of the NR query
      // rows, then their lo codes) in 16-byte chunks of 16 rows, swizzled: with
      // the 64-byte swizzle chunk c of key k lives at k*64 + ((c ^ ((k >> 1) & 3))
      // * 16), with the 128-byte swizzle at k*128 + ((c ^ (k & 7)) * 16). This
      // thread writes the chunks of its rows r0 .. r0 + RT - 1 in both halves.
      uint8_t* pbuf = smem + C::kOffP + st * C::kPBytes;
      const int sw = NR == 32 ? (tl >> 1) & 3 : tl & 7;
      const int cb = r0 / 16;
      uint4* row = reinterpret_cast<uint4*>(pbuf + tl * C::kPRow);
#pragma unroll
      for (int j = 0; j < RT / 16; ++j) {
        row[(cb + j) ^ sw] = make_uint4(hi[4 * j], hi[4 * j + 1], hi[4 * j + 2], hi[4 * j + 3]);
        row[(NR / 16 + cb + j) ^ sw] =
            make_uint4(lo[4 * j], lo[4 * j + 1], lo[4 * j + 2], lo[4 * j + 3]);
      }
      if (!valid) {                                // keys past the split: V rows must be 0
        uint8_t* stage = smem + st * kStageBytes;
        constexpr int kBands = 4 / C::kHalves;     // each half clears its share of the bands
#pragma unroll
        for (int c = 0; c < kBands; ++c) {
          uint4* vrow =
              reinterpret_cast<uint4*>(stage + (half * kBands + c) * kChunkBytes + tl * 128);
#pragma unroll
          for (int u = 0; u < 8; ++u) vrow[u] = make_uint4(0, 0, 0, 0);
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&ctl->p_full[st]);
    }
    if (!ok) break;

    // Row sums across the 128 keys of every tile, then 1/l and the LSE.
    reduce_rows<RT, false>(lp, lane, &ctl->red[quarter][r0]);
    group_sync_n<G>();
    if (gt < NR) {
      const float l = ctl->red[0][gt] + ctl->red[1][gt] + ctl->red[2][gt] + ctl->red[3][gt];
      ctl->vec[gt] = l > 0.f ? 1.f / l : 0.f;
      ctl->lse[gt] = l > 0.f ? ctl->m_run[gt] + __log2f(l) : -INFINITY;
    }
    group_sync_n<G>();
    if (!(ok = wait_bar(&ctl->o_full, x & 1, ctl, a.status))) break;
    tc::fence_after_sync();
    // Each thread holds one output dim of a 128-dim band (TMEM lane = dim) for
    // its RT rows, so for each row a warp's 32 lanes store 32 consecutive
    // values straight from registers.
    float sc[RT];                                  // per-row output scale
#pragma unroll
    for (int i = 0; i < RT; ++i) sc[i] = ctl->vec[r0 + i] * (jb.direct ? a.bmm2 : 1.f);
#pragma unroll 1
    for (int dt = 0; dt < 4; ++dt) {
      float o[RT];
      if (C::split(dt)) {                          // hi and lo accumulators side by side
        uint32_t rh[RT], rl[RT];
        tmem_ld_rows<RT>(tmem + lane_addr + C::band_col(dt) + r0, rh);
        tmem_ld_rows<RT>(tmem + lane_addr + C::band_col(dt) + NR + r0, rl);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < RT; ++i) o[i] = __uint_as_float(rh[i]) + __uint_as_float(rl[i]);
      } else {
        uint32_t raw[RT];
        tmem_ld_rows<RT>(tmem + lane_addr + C::band_col(dt) + r0, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < RT; ++i) o[i] = __uint_as_float(raw[i]);
      }
      if (jb.direct) {
        uint16_t* dst = a.out + ((long long)jb.r * a.M + m0 + r0) * kDv + dt * 128 + tl;
#pragma unroll
        for (int i = 0; i < RT; ++i)
          if (r0 + i < rows) dst[(long long)i * kDv] = f32_to_bf16_bits(o[i] * sc[i]);
      } else {
        float* dst = a.part_o + ((long long)jb.item * a.M + m0 + r0) * kDv + dt * 128 + tl;
#pragma unroll
        for (int i = 0; i < RT; ++i)
          if (r0 + i < rows) dst[(long long)i * kDv] = o[i] * sc[i];
      }
    }
    tc::fence_before_sync();
    tc::mbar_arrive(&ctl->o_empty);
    if (gt < rows) {
      if (jb.direct) {
        if (a.lse) a.lse[(long long)jb.r * a.M + m0 + gt] = ctl->lse[gt];
      } else {
        a.part_lse[(long long)jb.item * a.M + m0 + gt] = ctl->lse[gt];
      }
    }
    g += jb.ntiles;
    ++x;
  }
}

// HALVES: the work items have several row blocks, so sibling jobs share each
// tile through L2 and a stage is refilled in two halves (decode_common.cuh).
// PACKABLE: the shape allows a packed plan, so the kernel checks for one.
template <int NR, bool HALVES, bool PACKABLE>
__global__ void __launch_bounds__(Cfg<NR>::kThreads, 1)
decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_kv,
                 const __grid_constant__ CUtensorMap tm_kvr,
                 const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_qr, int nb) {
  using C = Cfg<NR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::kOffCtl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&ctl->kv_full[s], 1);
      tc::mbar_init(&ctl->pv_done[s], 1);
      if (HALVES) tc::mbar_init(&ctl->pv_half[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->s_full[b], 1);
      tc::mbar_init(&ctl->s_empty[b], C::kGroup);
      tc::mbar_init(&ctl->p_full[b], C::kGroup);
    }
    tc::mbar_init(&ctl->q_full, 1);
    tc::mbar_init(&ctl->q_empty, 1);
    tc::mbar_init(&ctl->o_full, 1);
    tc::mbar_init(&ctl->o_empty, C::kGroup);
    tc::mbar_init(&ctl->drain, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->job_full[b], 1);
      tc::mbar_init(&ctl->job_empty[b], 1 + C::kGroup);   // the MMA thread + the softmax group
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

  // While the plan runs, warm L2 with the block table (a prefetch returns no
  // data, so whatever an earlier kernel writes there is still what is read).
  // The short, latency-bound jobs of the 32-row kernel gain from it; the
  // 64-row kernel is at its register limit.
  if constexpr (NR == 32) {
    const long long lines = ((long long)(a.R / a.groups) * a.max_pages * 4 + 127) / 128;
    for (long long l = (long long)blockIdx.x * blockDim.x + threadIdx.x; l < lines;
         l += (long long)gridDim.x * blockDim.x)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a.block_table + l * 32));
  }
  grid_dep_wait();      // the plan is complete; earlier readers of out/workspace are done
  grid_dep_launch();    // the reducer may launch; it still waits for this grid to finish
  if (warp == 0) {
    // The entry of job blockIdx.x says whether the plan is packed.
    const int e0 =
        PACKABLE && (int)blockIdx.x < a.items * nb ? a.work[blockIdx.x / nb] : -1;
    if (PACKABLE && e0 >= 0 && (e0 & kPackedBit))
      producer_packed<NR, Cfg<NR>::kOffQ, NR == 32, NR != 32, HALVES>(a, smem, ctl, nb, &tm_kv,
                                                                      &tm_kvr, &tm_q, &tm_qr);
    else
      producer<NR, Cfg<NR>::kOffQ, NR == 32, NR != 32, HALVES, false, PACKABLE>(
          a, smem, ctl, nb, &tm_kv, &tm_kvr, &tm_q, &tm_qr, e0);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<NR, HALVES>(a, smem, ctl, tmem, nb);
  } else {
    softmax_epilogue<NR>(a, smem, ctl, tmem, nb);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
template <int NR, bool HALVES, bool PACKABLE>
cudaError_t launch_nr(const mla_shape& s, const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<NR>;
  CUtensorMap tkv, tkvr, tq, tqr;
  const cuuint64_t kv_dims[2] = {(cuuint64_t)kDqk, (cuuint64_t)a.num_pages * kPage};
  const cuuint64_t kv_str[1] = {(cuuint64_t)kDqk};
  const cuuint32_t kv_box[2] = {128, kPage}, kvr_box[2] = {64, kPage};
  const cuuint64_t q_dims[3] = {(cuuint64_t)kDqk, (cuuint64_t)a.M, (cuuint64_t)a.R};
  const cuuint64_t q_str[2] = {(cuuint64_t)kDqk, (cuuint64_t)a.M * kDqk};
  const cuuint32_t q_box[3] = {128, (cuuint32_t)NR, 1}, qr_box[3] = {64, (cuuint32_t)NR, 1};
  if (!encode(&tkv, a.kv, 2, kv_dims, kv_str, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode(&tkvr, a.kv, 2, kv_dims, kv_str, kvr_box, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode(&tq, a.q, 3, q_dims, q_str, q_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode(&tqr, a.q, 3, q_dims, q_str, qr_box, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const int smem_bytes = C::kOffCtl + (int)sizeof(Ctl) + 1024;
  static bool attr_set[64] = {};
  cudaError_t e = set_smem(decode_tc_kernel<NR, HALVES, PACKABLE>, smem_bytes, attr_set);
  if (e != cudaSuccess) return e;
  const int nb = row_blocks(a.M);
  const long long jobs = (long long)a.items * nb;
  const int grid = (int)(jobs < s.num_ctas ? jobs : s.num_ctas);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<NR, HALVES, PACKABLE>, a, tkv, tkvr, tq, tqr,
                            nb);
}

template <bool PACKABLE>
cudaError_t launch_kind(const mla_shape& s, const DecodeArgs& a, cudaStream_t st) {
  if (row_block(a.M) == 32) return launch_nr<32, false, PACKABLE>(s, a, st);
  return row_blocks(a.M) > 1 ? launch_nr<64, true, PACKABLE>(s, a, st)
                             : launch_nr<64, false, PACKABLE>(s, a, st);
}

}  // namespace

cudaError_t launch_decode(const mla_shape& s, const DecodeArgs& a, cudaStream_t st) {
  return plan_packable(s) ? launch_kind<true>(s, a, st) : launch_kind<false>(s, a, st);
}

}  // namespace mlafold
