// Pieces of the split-KV decode kernel (decode_tc.cu) kept apart from its MMA
// and softmax roles: tile geometry, the control block with its mbarriers,
// bounded waits, per-job facts, job claiming, the TMA producer warp, the P
// conversion helpers and tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace mlafold {
namespace dec {

constexpr int kTileKeys = 128;                    // keys per MMA tile (two pages)
constexpr int kStages = 2;                        // KV tiles in flight
constexpr int kChunkBytes = kTileKeys * 128;      // one 128-dim latent band of a tile
constexpr int kRopeBytes = kTileKeys * 64;        // the 64 rope dims of a tile
constexpr int kStageBytes = 4 * kChunkBytes + kRopeBytes;     // 73728
constexpr int kPageBytes = kPage * kDqk;          // 36864 bytes per page
constexpr uint32_t kTmemCols = 512;
// Bound of every pipeline wait (the decode's default) and of the drain of a
// CTA's own copies and MMAs when it stops early.
constexpr unsigned long long kTimeoutNs = 2000000000ull;
// When a row's lazy max moves (a score beyond the old max + 8, base 2), it is
// set kMaxLead below the tile's max instead of at it: P = 2^(x - max) then
// reaches 2^kMaxLead on that tile and at most 2^8 (< 448) later, and more of
// P's small values sit in E4M3's normal range (down to 2^-6) instead of its
// subnormals, whose absolute step of 2^-9 dominated the output error. A larger
// lead buys little more accuracy and moves the max (rescaling O) more often.
constexpr float kMaxLead = 2.f;

// Per-job facts, from the plan (read_job). item < 0: no more jobs.
struct Job {
  int r, blk, item, j0, j1, ntiles;
  bool direct, skip;
};

struct Ctl {
  uint64_t kv_full[kStages];   // TMA -> MMA: tile landed
  uint64_t pv_done[kStages];   // MMA -> TMA, softmax: PV of a tile finished (stage, P free)
  uint64_t s_full[2];          // MMA -> softmax: S^T ready
  uint64_t s_empty[2];         // softmax -> MMA: S^T read
  uint64_t p_full[2];          // softmax -> MMA: P^T written, masked V rows zeroed
  uint64_t q_full, q_empty;    // Q block of the job
  uint64_t o_full, o_empty;    // O^T of the job
  uint64_t drain;
  uint64_t job_full[2];        // producer -> other roles: the next job is in job[]
  uint64_t job_empty[2];       // other roles -> producer: job read
  Job job[2];
  uint32_t tmem_base;
  int abort_flag;
  unsigned long long wait_limit_ns;   // DecodeArgs::wait_limit_ns
  float m_run[64];             // running row max (base-2 scores)
  float vec[64];               // rescale factors, then 1/l
  float lse[64];
  float red[4][64];            // cross-warp reduction scratch
  uint64_t pv_half[kStages];   // MMA -> TMA: PV is done with value bands 0-1 (HALVES)
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Ctl* ctl,
                                         int32_t* status) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = tc::globaltimer_ns();
  while (true) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl->abort_flag)) return false;
    if (tc::globaltimer_ns() - t0 > ctl->wait_limit_ns) {
      *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
      if (status) atomicOr(status, MLA_FAULT_WAIT_TIMEOUT);
      return false;
    }
  }
}



// A job of work-list entry `item`: its request, rows and keys. A packed plan
// gives each entry's page range; the other plans split each request into
// equal, page-aligned parts.
__device__ __forceinline__ Job read_job(const DecodeArgs& a, int item, int blk, bool packed,
                                        bool report) {
  Job jb;
  jb.item = item;
  jb.blk = blk;
  jb.skip = false;
  const int e = a.work[item];
  // Only a packed plan's entries carry kPackedBit.
  const int r = packed ? entry_request(e) : e >> kSplitBits, s = entry_split(e);
  jb.r = r;
  if (r >= a.R || s >= a.counts[r]) {
    if (report && a.status) atomicOr(a.status, MLA_FAULT_WORK_ITEM);
    jb.skip = true;
    jb.j0 = jb.j1 = jb.ntiles = 0;
    jb.direct = false;
    return jb;
  }
  const int n = a.counts[r];
  int L = max(a.seq_lens[r / a.groups], 0);   // row group r reads request r / groups
  if (L > a.max_pages * kPage) {          // never read past the block-table row
    if (report && a.status) atomicOr(a.status, MLA_FAULT_PAGE_RANGE);
    L = a.max_pages * kPage;
  }
  if (!packed) {
    split_range(L, n, s, jb.j0, jb.j1);
  } else {
    const int pa = a.ranges[2 * item], pb = a.ranges[2 * item + 1];
    if (pa < 0 || pa > pb || (long long)pb > cdiv(L, kPage)) {
      if (report && a.status) atomicOr(a.status, MLA_FAULT_WORK_ITEM);
      jb.skip = true;
    }
    jb.j1 = min(L, max(pb, 0) * kPage);
    jb.j0 = min(max(pa, 0) * kPage, jb.j1);
  }
  jb.ntiles = (int)cdiv(jb.j1 - jb.j0, kTileKeys);
  jb.direct = n == 1;
  if (!jb.direct && item >= a.slots) {
    if (report && a.status) atomicOr(a.status, MLA_FAULT_WORK_ITEM);
    jb.skip = true;
  }
  return jb;
}

// ---------------------------------------------------------------- job claiming
// A CTA's first job is its index; after that its producer claims jobs in
// work-list order from a counter (the entry after the items), so a CTA that
// finishes early takes more of the list, which runs longest request first.
// The counter counts down from -1: claim k (from 0) is job gridDim.x + k.
__device__ __forceinline__ int claim_job(const DecodeArgs& a, int lane) {
  int k = 0;
  if (lane == 0) k = -1 - atomicAdd(a.sched, -1);
  return (int)gridDim.x + __shfl_sync(0xffffffffu, k, 0);
}

// The producer hands each job, or one with item -1 at the end, to the MMA and
// softmax roles through a two-slot ring (lane 0 of the producer).
__device__ __forceinline__ bool publish_job(Ctl* ctl, uint32_t seq, const Job& jb,
                                            int32_t* status) {
  const int b = seq & 1;
  if (seq >= 2 && !wait_bar(&ctl->job_empty[b], ((seq >> 1) - 1) & 1, ctl, status)) return false;
  volatile Job* slot = &ctl->job[b];
  slot->r = jb.r;
  slot->blk = jb.blk;
  slot->item = jb.item;
  slot->j0 = jb.j0;
  slot->j1 = jb.j1;
  slot->ntiles = jb.ntiles;
  slot->direct = jb.direct;
  slot->skip = jb.skip;
  tc::mbar_arrive(&ctl->job_full[b]);       // release: the job is visible to the waiters
  return true;
}
__device__ __forceinline__ bool take_job(Ctl* ctl, uint32_t seq, int32_t* status, Job& jb) {
  const int b = seq & 1;
  if (!wait_bar(&ctl->job_full[b], (seq >> 1) & 1, ctl, status)) return false;
  const volatile Job* slot = &ctl->job[b];
  jb.r = slot->r;
  jb.blk = slot->blk;
  jb.item = slot->item;
  jb.j0 = slot->j0;
  jb.j1 = slot->j1;
  jb.ntiles = slot->ntiles;
  jb.direct = slot->direct;
  jb.skip = slot->skip;
  tc::mbar_arrive(&ctl->job_empty[b]);
  return true;
}

// Lane 0 of the producer, after the CTA's last claim: count the CTA out; the
// last one resets both counters to -1 for the next decode of the same plan.
// The other roles are still finishing their last tiles meanwhile.
__device__ __forceinline__ void finish_jobs(const DecodeArgs& a) {
  __threadfence();
  const int done = -1 - atomicAdd(a.sched + 1, -1);
  if (done == (int)gridDim.x - 1) {
    __threadfence();
    atomicExch(a.sched, -1);
    atomicExch(a.sched + 1, -1);
  }
}

// ---------------------------------------------------------------- producer
// Runs on all 32 lanes of warp 0: the lanes fetch the job's block-table
// entries 32 at a time (lane i holds page i of the chunk, checked against the
// cache), lane 0 waits on the ring and issues the TMA copies.
// QROWS: query rows per Q block (the job's row block); OFFQ: shared-memory
// offset of the Q block; STAGGER: request the CTA's second tile only once its
// first has landed; PREFETCH: with each tile, warm L2 with the pages of the
// tile that will next use the same stage; HALVES: refill a stage in two
// halves (below); PACKED: the plan is packed (bit 30 of its entries); e0:
// the entry of job blockIdx.x when the caller loaded it (E0), used for the
// first job of a per-request plan instead of loading it again.
template <int QROWS, int OFFQ, bool STAGGER, bool PREFETCH, bool HALVES, bool PACKED,
          bool E0 = false>
__device__ __forceinline__ void producer(const DecodeArgs& a, uint8_t* smem, Ctl* ctl, int nb,
                                         const CUtensorMap* tm_kv, const CUtensorMap* tm_kvr,
                                         const CUtensorMap* tm_q, const CUtensorMap* tm_qr,
                                         int e0 = -1) {
  constexpr int kQChunk = QROWS * 128, kQBytes = QROWS * kDqk;
  const int lane = threadIdx.x & 31;
  uint32_t g = 0, x = 0;
  int last_q_parity = -1;
  int last_kv_parity[kStages] = {-1, -1};
  const int njobs = a.items * nb;
  bool ok = true;
  auto wait0 = [&](uint64_t* bar, uint32_t parity) {
    int r = 1;
    if (lane == 0) r = wait_bar(bar, parity, ctl, a.status) ? 1 : 0;
    return __shfl_sync(0xffffffffu, r, 0) != 0;
  };
  auto fetch = [&](const Job& jb, int chunk) {   // page ids of job pages 32*chunk + lane
    const int first = jb.j0 / kPage + chunk * 32 + lane;
    const int end = (int)cdiv(jb.j1, kPage);
    int p = -1;
    if (first < end) {
      p = a.block_table[(long long)(jb.r / a.groups) * a.max_pages + first];
      if (p < 0 || p >= a.num_pages) {
        if (a.status) atomicOr(a.status, MLA_FAULT_PAGE_RANGE);
        p = -1;
      }
    }
    return p;
  };
  int job = (int)blockIdx.x;
  // A packed plan (bit 30 of its entries) gives each unit a fixed list of
  // entries, slot-major in its unit table: CTA b, row block b % nb of unit
  // b / nb, takes jobs b, b + U nb, b + 2 U nb, ... through the table instead
  // of claiming.
  constexpr bool packed = PACKED;
  const int stride = a.nunits * nb;
  const int jobs_end = !packed ? njobs : (job < stride ? kUnitSlots * stride : 0);
  bool first = E0;
  for (uint32_t seq = 0; ok; ++seq) {
    Job jb;
    int blk = 0;
    bool have = false;
    while (job < jobs_end) {                     // the next job that is not malformed
      int item = job / nb;
      blk = job % nb;
      if (packed && ((item = a.units[item]) < 0 || item >= a.items)) break;   // list ended
      if ((first ? e0 : a.work[item]) < 0) break;   // past the last item (the list is compact)
      first = false;
      jb = read_job(a, item, blk, packed, lane == 0);
      if (!jb.skip) {
        have = true;
        break;
      }
      job = packed ? job + stride : claim_job(a, lane);
    }
    if (!have) jb.item = -1;
    int pub = 1;
    if (lane == 0) pub = publish_job(ctl, seq, jb, a.status) ? 1 : 0;
    if (!(ok = __shfl_sync(0xffffffffu, pub, 0) != 0) || !have) break;
    if (jb.ntiles == 0) {                        // an empty split: the softmax role writes it
      job = packed ? job + stride : claim_job(a, lane);
      continue;
    }
    int cur = fetch(jb, 0), nxt = fetch(jb, 1);
    if (x > 0 && !(ok = wait0(&ctl->q_empty, (x - 1) & 1))) break;
    if (lane == 0) {
      uint8_t* q = smem + OFFQ;
      const int qrow = blk * QROWS;
      tc::mbar_arrive_expect_tx(&ctl->q_full, kQBytes);
      for (int c = 0; c < 4; ++c)
        tc::tma_load_3d(q + c * kQChunk, tm_q, &ctl->q_full, c * 128, qrow, jb.r);
      tc::tma_load_3d(q + 4 * kQChunk, tm_qr, &ctl->q_full, 512, qrow, jb.r);
    }
    last_q_parity = x & 1;
    for (int t = 0; t < jb.ntiles; ++t, ++g) {
      if (t > 0 && (t & 15) == 0) {            // 16 tiles = 32 pages per chunk
        cur = nxt;
        nxt = fetch(jb, (t >> 4) + 1);
      }
      const int st = g & 1;
      if constexpr (!HALVES)
        if (g >= 2 && !(ok = wait0(&ctl->pv_done[st], ((g >> 1) - 1) & 1))) break;
      // Every CTA starts at once. With short, HBM-bound jobs it pays to ask
      // for the second tile only after the first has landed: the first tiles
      // then arrive first and the MMAs start while the second ones stream in,
      // instead of both arriving together.
      if (STAGGER && g == 1 && !(ok = wait0(&ctl->kv_full[0], 0))) break;
      const int kbase = jb.j0 + t * kTileKeys;
      const int pages = (kbase + kPage < jb.j1) ? 2 : 1;
      const int pid0 = __shfl_sync(0xffffffffu, cur, (2 * t) & 31);
      const int pid1 = __shfl_sync(0xffffffffu, cur, (2 * t + 1) & 31);
      // Failure-detection test only: CTA 0 issues no copy for its first tile,
      // so the waits on it run out (bounded) and the CTA stops early.
      const bool withhold = a.withhold_first_copy && blockIdx.x == 0 && g == 0;
      const int pid[2] = {pid0, pages == 2 ? pid1 : -1};
      uint8_t* stage = smem + st * kStageBytes;
      const int nbytes = ((pid[0] >= 0) + (pid[1] >= 0)) * kPageBytes;
      if constexpr (!HALVES) {
        // The stage is refilled, page by page, once PV of the tile two back is
        // done (waited for above; one row block per item: the tile streams
        // from HBM).
        if (lane == 0 && !withhold) {
          tc::mbar_arrive_expect_tx(&ctl->kv_full[st], nbytes);
          for (int h = 0; h < 2; ++h) {
            if (pid[h] < 0) continue;
            const int row = pid[h] * kPage;
            for (int c = 0; c < 4; ++c)
              tc::tma_load_2d(stage + c * kChunkBytes + h * (kChunkBytes / 2), tm_kv,
                              &ctl->kv_full[st], c * 128, row);
            tc::tma_load_2d(stage + 4 * kChunkBytes + h * (kRopeBytes / 2), tm_kvr,
                            &ctl->kv_full[st], 512, row);
          }
        }
        last_kv_parity[st] = withhold ? -1 : (int)((g >> 1) & 1);
      } else {
        // Several row blocks per item (their jobs share each tile through L2):
        // the stage is refilled in two halves, value bands 0-1 and the rope
        // (which only S reads) once PV of the tile two back is done with bands
        // 0-1, bands 2-3 once that PV is done. kv_full is armed for the whole
        // tile after the first wait, which proves the stage's previous phase
        // completed (that PV ran on its data).
        for (int part = 0; part < 2; ++part) {
          if (g >= 2 &&
              !(ok = wait0(part == 0 ? &ctl->pv_half[st] : &ctl->pv_done[st], ((g >> 1) - 1) & 1)))
            break;
          if (part == 0) {
            if (lane == 0 && !withhold) tc::mbar_arrive_expect_tx(&ctl->kv_full[st], nbytes);
            last_kv_parity[st] = withhold ? -1 : (int)((g >> 1) & 1);
          }
          if (lane == 0 && !withhold) {
            for (int h = 0; h < 2; ++h) {
              if (pid[h] < 0) continue;
              const int row = pid[h] * kPage;
              for (int c = 2 * part; c < 2 * part + 2; ++c)
                tc::tma_load_2d(stage + c * kChunkBytes + h * (kChunkBytes / 2), tm_kv,
                                &ctl->kv_full[st], c * 128, row);
              if (part == 0)
                tc::tma_load_2d(stage + 4 * kChunkBytes + h * (kRopeBytes / 2), tm_kvr,
                                &ctl->kv_full[st], 512, row);
            }
          }
        }
        if (!ok) break;
      }
      // Tile t + kStages is requested only once PV(t) frees this stage; warmed
      // in L2 now, its copy then skips most of the HBM latency.
      if (PREFETCH && t + kStages < jb.ntiles) {
        const int tp = t + kStages;
        const int src = (tp >> 4) == (t >> 4) ? cur : nxt;
        const int q0 = __shfl_sync(0xffffffffu, src, (2 * tp) & 31);
        const int q1 = __shfl_sync(0xffffffffu, src, (2 * tp + 1) & 31);
        if (lane == 0) {
          if (q0 >= 0) tc::prefetch_l2(a.kv + (size_t)q0 * kPageBytes, kPageBytes);
          if (q1 >= 0 && jb.j0 + tp * kTileKeys + kPage < jb.j1)
            tc::prefetch_l2(a.kv + (size_t)q1 * kPageBytes, kPageBytes);
        }
      }
    }
    if (!ok) break;
    ++x;
    job = packed ? job + stride : claim_job(a, lane);
  }
  if (lane == 0) finish_jobs(a);
  // Never leave with copies in flight into this CTA's shared memory.
  if (!ok && lane == 0) {
    const unsigned long long t0 = tc::globaltimer_ns();
    for (int st = 0; st < kStages; ++st)
      while (last_kv_parity[st] >= 0 &&
             !tc::mbar_try_wait(&ctl->kv_full[st], last_kv_parity[st]) &&
             tc::globaltimer_ns() - t0 < kTimeoutNs) {
      }
    while (last_q_parity >= 0 && !tc::mbar_try_wait(&ctl->q_full, last_q_parity) &&
           tc::globaltimer_ns() - t0 < kTimeoutNs) {
    }
  }
}

// The packed plan's producer, kept out of line: the per-request plans' producer
// (inlined into the kernel) stays as compact as it is without packing.
template <int QROWS, int OFFQ, bool STAGGER, bool PREFETCH, bool HALVES>
__device__ __noinline__ void producer_packed(const DecodeArgs& a, uint8_t* smem, Ctl* ctl,
                                             int nb, const CUtensorMap* tm_kv,
                                             const CUtensorMap* tm_kvr,
                                             const CUtensorMap* tm_q, const CUtensorMap* tm_qr) {
  producer<QROWS, OFFQ, STAGGER, PREFETCH, HALVES, true>(a, smem, ctl, nb, tm_kv, tm_kvr, tm_q,
                                                         tm_qr);
}

// ---------------------------------------------------------------- P conversion
// P (FP32, <= 2^8) enters the PV product as two E4M3 terms built in FP16:
// p16 = fp16(p) (round to nearest even, relative error <= 2^-11),
// hi = e4m3(p16), lo = e4m3(p16 - hi), all conversions round to nearest even
// with satfinite; p16 - hi is exact in FP16 (hi is p16 rounded to 4
// significant bits, so both lie within a factor of two). hi + lo is p to
// about 2^-8 relative; the FP16 step adds at most 2^-11. FP16 pairs keep the
// conversion at a few instructions per two values.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t f16x2_to_e4m3x2(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// ---------------------------------------------------------------- host side
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

inline bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// Opt a kernel into `bytes` of dynamic shared memory, once per device.
template <typename K>
inline cudaError_t set_smem(K kernel, int bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

}  // namespace dec
}  // namespace mlafold
