// Split decode-attention kernel, all-heads form (tensor cores, T = 1).
//
// The per-head kernels give each CTA one KV head, so a page of 16 positions
// is read as 2 KB boxes (16 rows x 128 bytes of one head, rows 2 KB apart)
// by eight CTAs on different SMs.  On GB300 that pattern streamed a page-16
// pool at 6.25 TB/s, while boxes holding all eight KV heads of 16 positions
// (the whole 32 KB slice of K or V, read in two 64-dim halves) streamed it
// at 7.1 TB/s.  This kernel reads the pool that way:
//
//  * one persistent CTA per SM takes work items (sequence b, shard s) from
//    an atomic counter in the workspace (items b-major; the shard grid is the
//    split plan's, so partials, slots and the merge are those of the grid
//    schedule);
//  * a producer warp streams each 16-position slice of all Hkv = 8 heads per
//    ring stage (one 4-D TMA box per 64-dim half of K and of V), and tags the
//    stage with its item (shared-memory metadata published by the barrier);
//  * consumer warp h owns KV head h for the whole item: its G query rows, the
//    q.k and p.v products of mma_block (the same arithmetic as the per-head
//    kernel) on rows 16h..16h+15 of the stage, its own online-softmax state,
//    so no cross-warp fold is needed;
//  * at the item's end each warp writes its head's partial to the slots of
//    the grid schedule; a sequence held by one shard is written to out
//    directly (the merge of one partial gives the same bits), otherwise the
//    warp that completes a (sequence, KV head) group (an atomic ticket) merges
//    its shards with merge_group in ascending order, as the standalone combine
//    does.
//
// Waits are bounded like every wait in these kernels.  After a timeout the
// kernel raises DECODE_ATTN_DEV_TIMEOUT and stops; the rows of that call are
// then unspecified and the workspace must be cleared before the next call.
#pragma once

#include "split_mma.cuh"

namespace pgd {

template <int D>
struct AhCfg {
  static constexpr int kHeads = 8;                  // KV heads per stage, one consumer warp each
  static constexpr int kWarps = kHeads;
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kStageTok = 16;              // positions per stage
  static constexpr int kRows = kStageTok * kHeads;  // 128-byte rows per 64-dim sub-tile
  static_assert(kRows == 128, "the consumers address the stage as one piece of 2^7 rows");
  static constexpr int kTileBytes = kRows * D * 2;  // K (or V) of one stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = (192 * 1024) / kStageBytes;  // 3 at D = 128, 6 at D = 64
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kMergeCap = 32;  // (m, l) pairs per row staged by a warp's merge
  static constexpr int kMergeBytes = (merge_smem_bytes(8, kMergeCap) + 15) & ~15;
  static constexpr int kSmemBytes = kRingBytes + kWarps * kMergeBytes + 1024;
  static constexpr int kMaxChunk = 1024;  // tokens per shard (the planner's bound)
  static constexpr int kMaxStagesPerItem = kMaxChunk / kStageTok + 1;
  static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");
};

// Stage metadata, written by the producer before it arrives on the stage's
// full barrier (release) and read by the consumers after their wait
// (acquire).
enum : int32_t { kAhFirst = 1, kAhLast = 2, kAhBad = 4, kAhZero = 8, kAhEnd = 16 };
struct AhStage {
  int32_t b, s;       // item: sequence and shard
  int32_t tok0;       // first position of the stage
  int32_t lo, hi;     // the item's attended positions
  int32_t cs, ce;     // the sequence's attended range [start, end)
  int32_t nsh;        // shards of the sequence
  int32_t flags;
};

// Zero output rows of KV head h of sequence b (a sequence with no attended
// position or an invalid length).
template <int D>
__device__ __forceinline__ void ah_zero_rows(const SplitArgs& a, int b, int h, int lane) {
  uint32_t* out = static_cast<uint32_t*>(a.out);  // +0.0 is all zero bits in both formats
  for (int e = lane; e < a.G * D / 2; e += 32) {
    const size_t i = (((size_t)b * a.Hq + (size_t)h * a.G) * D) / 2 + e;
    if (PGD_IN(i, (size_t)a.batch * a.Hq * D / 2, a.err)) out[i] = 0u;
  }
}

// The end of an item for one warp: its head's partial, then out directly
// (one shard) or the ticket and, for the last shard to finish, the merge.
template <int D, class E>
__device__ __forceinline__ void ah_finish(const SplitArgs& a, const AhStage& m, int h, int lane,
                                          const float (&acc)[D / 16][1][4],
                                          const float (&m_run)[1][2], const float (&l_part)[1][2],
                                          uint8_t* msm, int merge_cap) {
  constexpr int KS = D / 16;
  const int gid = lane >> 2, tig = lane & 3;
  const bool bad = (m.flags & kAhBad) != 0;
  float l[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float v = l_part[0][e];
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    l[e] = v;
  }
  // the fragment's column 2 * tig + e is query row h * G + 2 * tig + e;
  // its dims mi * 16 + gid (e) and mi * 16 + gid + 8 (e + 2)
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int rr = 2 * tig + e;
    if (rr >= a.G) continue;
    const size_t row = (size_t)m.b * a.Hq + (size_t)h * a.G + rr;
    const size_t slot = row * a.max_shards + m.s;
    if (!PGD_IN(slot, (size_t)a.batch * a.Hq * a.max_shards, a.err)) continue;
    float* dst = a.ws_acc + slot * D;
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) {
      dst[mi * 16 + gid] = acc[mi][0][e];
      dst[mi * 16 + gid + 8] = acc[mi][0][e + 2];
    }
    if (gid == 0) a.ws_ml[slot] = make_float2(m_run[0][e], bad ? -1.f : l[e]);
    if (m.nsh == 1 && PGD_IN(row, (size_t)a.batch * a.Hq, a.err)) {
      // one shard: out = fp16_rn(acc / l), what the merge of this one
      // partial computes (weight 2^0 = 1)
      uint16_t* o = static_cast<uint16_t*>(a.out) + row * D;
      const bool z = bad || l[e] == 0.f;
#pragma unroll
      for (int mi = 0; mi < KS; ++mi) {
        o[mi * 16 + gid] = z ? 0 : ElemOps<E>::round(__fdiv_rn(acc[mi][0][e], l[e]));
        o[mi * 16 + gid + 8] = z ? 0 : ElemOps<E>::round(__fdiv_rn(acc[mi][0][e + 2], l[e]));
      }
    }
  }
  if (m.nsh == 1) return;
  __threadfence();  // this lane's partial, visible GPU-wide before the ticket
  __syncwarp();
  const size_t ti = (size_t)m.b * a.Hkv + h;
  int last = 0;
  if (lane == 0 && PGD_IN(ti, (size_t)a.batch * a.Hkv, a.err)) {
    const int old = atomicAdd(a.counters + ti, 1);
    if (old < 0 || old >= m.nsh) raise_error(a.err, DECODE_ATTN_DEV_WORKSPACE);
    last = old == m.nsh - 1;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  CombineArgs c{};
  c.seq_lens = a.seq_lens;
  c.ws_acc = a.ws_acc;
  c.ws_ml = a.ws_ml;
  c.out = a.out;
  c.err = a.err;
  c.B = a.batch;
  c.Hq = a.Hq;
  c.G = a.G;
  c.T = 1;
  c.capacity = a.max_pages * a.page_size;
  c.window = a.window;
  c.chunk = a.chunk;
  c.max_shards = a.max_shards;
  merge_group<D, E>(c, m.b, h, m.nsh, false, lane, 32, msm, merge_cap, [] { __syncwarp(); },
                    GridSlots{m.b, h, 1, a.G, a.Hq, a.max_shards});
  __syncwarp();
  if (lane == 0) a.counters[ti] = 0;  // cleared for the next call
}

template <int D, class E>
__global__ void __launch_bounds__(AhCfg<D>::kThreads, 1)
    split_allheads_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
  using C = AhCfg<D>;
  constexpr int KS = D / 16;
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ AhStage meta_s[C::kStages];
  __shared__ int32_t coord_s[C::kMaxStagesPerItem];
  __shared__ volatile int32_t abort_s;

  // a programmatic dependent launch: nothing is read or written before the
  // preceding kernel has completed
  grid_dependency_wait();
  grid_launch_dependents();
  uint8_t* ring = ring_base();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(smem_u32(&full_bar[st]), 1);
      mbar_init(smem_u32(&empty_bar[st]), C::kWarps);
    }
    fence_mbar_init();
    abort_s = 0;
  }
  __syncthreads();
  // after the B * Hkv group tickets: [0] the next work item, [1] CTAs done
  int32_t* const work = a.counters + (size_t)a.batch * a.Hkv;
  const int num_items = a.batch * a.max_shards;
  const int capacity = a.max_pages * a.page_size;
  const int pool_rows = a.num_pages * a.page_size;

  if (warp == C::kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    int issued = 0;  // ring stages pushed (lane 0's count)
    bool dead = false;
    // lane 0: the ring slot of stage `issued` is free (bounded wait)
    auto slot_free = [&]() -> bool {
      if (abort_s) return false;
      if (issued < C::kStages) return true;
      const int st = issued % C::kStages;
      if (!mbar_wait(smem_u32(&empty_bar[st]), ((issued / C::kStages) & 1) ^ 1)) {
        abort_s = 1;
        raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
        return false;
      }
      return abort_s == 0;
    };
    // lane 0: a stage with metadata only (no copies)
    auto push_marker = [&](const AhStage& m) -> bool {
      if (!slot_free()) return false;
      const int st = issued % C::kStages;
      meta_s[st] = m;
      mbar_arrive(smem_u32(&full_bar[st]));
      ++issued;
      return true;
    };
    while (!dead) {
      int item = 0;
      if (lane == 0) item = atomicAdd(work, 1);
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item >= num_items) break;
      const int b = item / a.max_shards, s = item % a.max_shards;
      const SeqRange r = seq_range(a.seq_lens[b], a.window, capacity, a.chunk, a.max_shards, 1);
      if (r.status != 0 || r.nshards == 0) {
        if (s == 0) {  // one marker per such sequence: its rows are zero
          if (lane == 0) {
            if (r.status != 0) raise_error(a.err, r.status);
            dead = !push_marker(AhStage{b, 0, 0, 0, 0, 0, 0, 0, kAhZero});
          }
          dead = __shfl_sync(0xffffffffu, dead, 0);
        }
        continue;
      }
      if (s >= r.nshards) continue;
      const int shard_lo = r.base + s * a.chunk;
      const int lo = max(r.start, shard_lo);
      const int hi = min(r.end, shard_lo + a.chunk);
      const int t0 = lo & ~(C::kStageTok - 1);
      const int nst = (hi - t0 + C::kStageTok - 1) / C::kStageTok;
      // the item's page rows, all lanes (a page holds whole 16-position
      // slices: the page size is a multiple of 16)
      int bad = nst > C::kMaxStagesPerItem ? 1 : 0;
      for (int i = lane; i < nst && i < C::kMaxStagesPerItem; i += 32) {
        const int tok = t0 + i * C::kStageTok;
        const size_t pi = (size_t)b * a.max_pages + (tok >> a.page_shift);
        const int phys =
            PGD_IN(pi, (size_t)a.batch * a.max_pages, a.err) ? a.page_table[pi] : -1;
        int coord = pool_rows;
        if (phys < 0 || phys >= a.num_pages) {
          bad = 1;
        } else {
          coord = phys * a.page_size + (tok & (a.page_size - 1));
        }
        coord_s[i] = coord;
      }
      bad = __any_sync(0xffffffffu, bad);
      __syncwarp();
      if (lane == 0) {
        if (bad) {
          raise_error(a.err, DECODE_ATTN_DEV_BAD_PAGE);
          dead = !push_marker(
              AhStage{b, s, t0, lo, hi, r.start, r.end, r.nshards, kAhFirst | kAhLast | kAhBad});
        } else {
          for (int i = 0; i < nst; ++i) {
            if (!slot_free()) {
              dead = true;
              break;
            }
            const int st = issued % C::kStages;
            meta_s[st] = AhStage{b, s, t0 + i * C::kStageTok, lo, hi, r.start, r.end, r.nshards,
                                 (i == 0 ? kAhFirst : 0) | (i == nst - 1 ? kAhLast : 0)};
            const uint32_t fb = smem_u32(&full_bar[st]);
            // (stall_tx, a test's hook, is 0: the barrier expects the stage's bytes)
            mbar_arrive_expect_tx(fb, C::kStageBytes + (issued == 0 ? a.stall_tx : 0));
            const uint32_t kd = smem_u32(ring + st * C::kStageBytes);
            int coord = coord_s[i];
            // (checked build) the 16 rows lie inside the pool
            if (!PGD_IN((int64_t)coord + C::kStageTok - 1, (int64_t)pool_rows, a.err))
              coord = pool_rows;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
              tma_load_4d(kd + c * (C::kRows * 128), &tmap_k, 0, coord, 0, c, fb);
              tma_load_4d(kd + C::kTileBytes + c * (C::kRows * 128), &tmap_v, 0, coord, 0, c, fb);
            }
            ++issued;
          }
        }
      }
      dead = __shfl_sync(0xffffffffu, dead, 0);
    }
    if (lane == 0) {
      // the copies in flight land first (the end marker completes one more
      // phase of a full barrier, after which these waits could not tell)
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(smem_u32(&full_bar[i % C::kStages]), (i / C::kStages) & 1);
      if (!dead) push_marker(AhStage{0, 0, 0, 0, 0, 0, 0, 0, kAhEnd});
      // the last CTA to finish clears the work counter for the next call
      if (atomicAdd(work + 1, 1) == (int)gridDim.x - 1) {
        atomicExch(work, 0);
        atomicExch(work + 1, 0);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int h = warp;  // this warp's KV head
  const int gid = lane >> 2, tig = lane & 3;
  uint8_t* msm = ring + C::kRingBytes + warp * C::kMergeBytes;
  uint32_t qf[1][KS][2];
  float acc[KS][1][4];
  float m_run[1][2], l_part[1][2];
  int col_lo[1][2], col_hi[1][2];
  for (int i = 0;; ++i) {
    const int st = i % C::kStages;
    if (!mbar_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1)) {
      abort_s = 1;
      raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
      break;
    }
    const AhStage m = meta_s[st];
    if (m.flags & kAhEnd) break;
    if (m.flags & kAhZero) {
      ah_zero_rows<D>(a, m.b, h, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
      continue;
    }
    if (m.flags & kAhFirst) {
      const int rr = gid;  // this lane's q row of the B operand
      size_t qr = (size_t)m.b * a.Hq + (size_t)h * a.G + (rr < a.G ? rr : 0);
      if (!PGD_IN(qr, (size_t)a.batch * a.Hq, a.err)) qr = 0;
      const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + qr * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[0][ks][0] = rr < a.G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tig) : 0u;
        qf[0][ks][1] =
            rr < a.G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tig) : 0u;
      }
#pragma unroll
      for (int mi = 0; mi < KS; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mi][0][e] = 0.f;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        m_run[0][e] = -INFINITY;
        l_part[0][e] = 0.f;
        col_lo[0][e] = m.cs;  // one query position: every row attends [start, L)
        col_hi[0][e] = m.ce;
      }
    }
    // the warp's K and V rows go to registers and the stage is released
    // before the arithmetic: with three stages in the ring, the time a stage
    // is held is time the SM has a third less in flight
    const uint32_t eb = smem_u32(&empty_bar[st]);
    auto release = [eb, lane] {
      __syncwarp();
      if (lane == 0) mbar_arrive(eb);
    };
    if (!(m.flags & kAhBad)) {
      mma_block<D, 1, E, C::kRows, true>(ring + st * C::kStageBytes, h, lane, m.tok0, m.lo, m.hi,
                                         col_lo, col_hi, qf, a.scale_log2, acc, m_run, l_part,
                                         7, release);  // one piece of kRows = 128 rows
    } else {
      release();
    }
    if (m.flags & kAhLast) ah_finish<D, E>(a, m, h, lane, acc, m_run, l_part, msm, C::kMergeCap);
  }
}

}  // namespace pgd
