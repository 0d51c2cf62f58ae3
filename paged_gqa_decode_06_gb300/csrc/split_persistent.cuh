// Split decode-attention kernel, tensor-core variant on a persistent,
// balanced schedule.
//
// The grid schedule (split_mma.cuh) gives every (shard, KV head, sequence) a
// CTA of its own; with sequences of very different lengths many CTAs are short
// and each pays a prologue (lengths, page ids, the first TMA round trip).
// Here the grid is the resident CTA count.  For each KV head the work is the
// list of (sequence, 64-token tile) pairs, sequence-major, W tiles; it is cut
// into N equal ranges (N = CTAs / Hkv, at most W, so every range is
// non-empty) and CTA c = j * Hkv + h takes range j of head h, so every CTA
// streams the same number of tiles and the Hkv CTAs of range j read the same
// positions' rows of all heads at about the same time (the rows of one
// position are adjacent in the pool).  A range falls into segments, one per
// sequence it touches; the TMA producer runs straight across segment
// boundaries (one running stage counter), the consumers restart their
// online-softmax state per segment.
//
// A unit that lies inside one CTA's range is finished there (normalised
// output written directly).  A unit cut by range boundaries has one segment
// in each CTA it touches; each writes a partial (m, l, acc) to one of two
// slots of its CTA (slot 0: the CTA's first segment, slot 1: its last), and
// the last CTA of the unit to finish (an atomic ticket, nothing waits) merges
// the unit's partials in ascending range order, i.e. in token order.  The
// partition depends only on the lengths and the CTA count, so the bits of the
// result do not depend on timing.
//
// The four consumer warps of a CTA each hold a full online-softmax state for
// their 16 positions of every tile; at a segment's end they are folded into
// warp 0 one after another through a one-warp shared slot (fixed order).
#pragma once

#include "split_mma.cuh"

namespace pgd {

constexpr int kPersistMaxBatch = 1024;  // sequences whose tile prefix fits in shared memory
constexpr int kPersistPieces = 512;     // page coordinates staged per producer pass

struct PersistArgs {
  SplitArgs s;   // ws_ml / ws_acc hold the per-CTA slots: [N][2][R] (+ D floats)
  int32_t B;     // sequences
  int32_t nc;    // persistent CTAs (grid size)
};

// Bytes of the one-warp slot that folds the consumer warps' states.
template <int D, int NT8>
__host__ __device__ constexpr int persist_slot_bytes() {
  return 32 * ((D / 16) * NT8 * 4 + NT8 * 4) * 4;
}

template <int D, int NT8>
__host__ __device__ constexpr int persist_smem_bytes() {
  return MmaCfg<D>::kRingBytes + persist_slot_bytes<D, NT8>() + 1024;
}

// One (sequence, KV head) unit's piece of a CTA's tile range.
struct Segment {
  int b, h;        // unit
  int t0, nt;      // first tile within the unit, tiles in this segment
  int n;           // tiles of the unit
  int64_t u0;      // global index of the unit's first tile
};

// Walks one head's tile range [g, g_end) sequence by sequence; prefix[b] =
// tiles (per head) of the sequences before b.
struct SegWalker {
  const int32_t* prefix;
  int B, h;
  int64_t g, g_end;
  int b, off;  // current sequence and tile offset inside it

  __device__ void start(const int32_t* pre, int nb, int head, int64_t g0, int64_t g1) {
    prefix = pre;
    B = nb;
    h = head;
    g = g0;
    g_end = g1;
    if (g >= g_end) return;
    int lo = 0, hi = B;  // prefix[lo] <= g < prefix[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= g) lo = mid; else hi = mid;
    }
    b = lo;
    off = (int)(g - prefix[b]);
  }
  __device__ bool done() const { return g >= g_end; }
  __device__ Segment current() const {
    Segment sg;
    sg.b = b;
    sg.h = h;
    sg.n = prefix[b + 1] - prefix[b];
    sg.t0 = off;
    const int64_t left = g_end - g;
    sg.nt = (int)(left < (int64_t)(sg.n - off) ? left : (int64_t)(sg.n - off));
    sg.u0 = prefix[b];
    return sg;
  }
  __device__ void advance(const Segment& sg) {
    g += sg.nt;
    if (g >= g_end) return;
    off = 0;
    do { ++b; } while (prefix[b + 1] == prefix[b]);
  }
};

__device__ __forceinline__ int64_t range_start(int c, int64_t W, int N) {
  return (int64_t)c * W / N;
}
// CTA whose range holds global tile u.
__device__ __forceinline__ int cta_of_tile(int64_t u, int64_t W, int N) {
  return (int)(((u + 1) * N - 1) / W);
}

template <int D, int NT8, class E>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads)
    split_mma_persistent_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                const __grid_constant__ CUtensorMap tmap_v,
                                const PersistArgs pa) {
  using C = MmaCfg<D>;
  constexpr int GP = 8 * NT8;
  constexpr int KS = D / 16;
  constexpr int kWarps = C::kWarps;
  const SplitArgs& a = pa.s;
  const int c = blockIdx.x;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ int32_t prefix_s[kPersistMaxBatch + 1];
  __shared__ int32_t coord_s[kPersistPieces];
  __shared__ int32_t seg_bad_s[8];
  __shared__ float2 ml_s[GP];
  __shared__ int is_last_s;
  __shared__ volatile int32_t abort_s;

  // launched as a programmatic dependent: nothing is read or written before
  // the preceding grid on the stream has completed
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int capacity = a.max_pages * a.page_size;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* slot = ring + C::kRingBytes;  // one warp's folded state / merge scratch

  // ---- tiles per sequence, their prefix, this CTA's range ----------------
  for (int b = threadIdx.x; b < pa.B; b += blockDim.x) {
    const SeqRange r = seq_range(a.seq_lens[b], a.window, capacity, 1 << 30, 1, a.T);
    const int n = (r.status == 0 && r.nshards > 0) ? (r.end - r.base + kTile - 1) / kTile : 0;
    prefix_s[b + 1] = n;
  }
  if (threadIdx.x == 0) {
    prefix_s[0] = 0;
    abort_s = 0;
  }
  __syncthreads();
  if (warp == 0) {  // inclusive scan, 32 sequences at a time
    int carry = 0;
    for (int i0 = 0; i0 < pa.B; i0 += 32) {
      int v = (i0 + lane < pa.B) ? prefix_s[i0 + lane + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (i0 + lane < pa.B) prefix_s[i0 + lane + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  const int64_t W = prefix_s[pa.B];  // tiles per head
  // ranges per head: at most one per tile, so that every active CTA's range
  // holds at least one tile and a unit's segments sit in consecutive ranges
  const int per_head = pa.nc / a.Hkv;  // >= 1: the planner keeps Hkv <= CTAs
  const int N = (int)(W < per_head ? (W > 0 ? W : 1) : per_head);
  const int hh = c % a.Hkv, jr = c / a.Hkv;  // this CTA's head and range

  // sequences without tiles (empty or invalid): rows zeroed, errors raised
  for (int b = c; b < pa.B; b += pa.nc) {
    if (prefix_s[b + 1] != prefix_s[b]) continue;
    const SeqRange r = seq_range(a.seq_lens[b], a.window, capacity, 1 << 30, 1, a.T);
    if (r.status != 0 && threadIdx.x == 0) raise_error(a.err, r.status);
    for (int h = 0; h < a.Hkv; ++h) zero_group_rows<D, GP>(a, b, h);
  }
  if (jr >= N) return;
  const int64_t g0 = range_start(jr, W, N), g1 = range_start(jr + 1, W, N);
  if (g0 >= g1) return;

  if (threadIdx.x == 0) {
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(smem_u32(&full_bar[st]), 1);
      mbar_init(smem_u32(&empty_bar[st]), kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int box_t = a.box_tokens;
  const int ppt = kTile / box_t;  // TMA boxes per tile

  // =========================================================== producer
  if (warp == kWarps) {
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    const int oob = a.num_pages * a.page_size;  // past the pool: TMA writes zeros
    const uint32_t box_bytes = box_t * 128;  // one 64-dim slice of box_t rows
    SegWalker wk;
    wk.start(prefix_s, pa.B, hh, g0, g1);
    int it = 0, ord = 0;
    bool stop = false;
    while (!wk.done() && !stop) {
      const Segment sg = wk.current();
      const SeqRange r = seq_range(a.seq_lens[sg.b], a.window, capacity, 1 << 30, 1, a.T);
      const int seg_lo = r.base + sg.t0 * kTile;  // first position of the segment's tiles
      if (a.k_new != nullptr) {
        // new rows inside this segment: written before any of its TMA reads
        const int hi_pos = seg_lo + sg.nt * kTile;
        if (r.end - a.T < hi_pos && r.end > seg_lo) {
          SeqRange rr = r;
          SplitArgs aa = a;
          aa.chunk = sg.nt * kTile;
          append_new_rows<D>(aa, rr, sg.b, sg.h, seg_lo, lane);
        }
      }
      int bad = 0;
      const int n_pieces = sg.nt * ppt;
      for (int p0 = 0; p0 < n_pieces && !stop; p0 += kPersistPieces) {
        const int np = min(kPersistPieces, n_pieces - p0);
        __syncwarp();
        for (int i = lane; i < np; i += 32) {
          const int ptok = seg_lo + (p0 + i) * box_t;
          int coord = oob;
          if (ptok < r.end && ptok + box_t > r.start) {
            const int phys =
                a.page_table[(size_t)sg.b * a.max_pages + (ptok >> a.page_shift)];
            if (phys < 0 || phys >= a.num_pages) bad = 1;
            else coord = phys * a.page_size + (ptok & (a.page_size - 1));
          }
          coord_s[i] = coord;
        }
        bad = __any_sync(0xffffffffu, bad);
        __syncwarp();
        if (lane == 0) {
          for (int pt = 0; pt < np; pt += ppt, ++it) {
            const int st = it % C::kStages;
            if (it >= C::kStages &&
                !mbar_wait(smem_u32(&empty_bar[st]), ((it / C::kStages) & 1) ^ 1)) {
              abort_s = 1;
              raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
              stop = true;
              break;
            }
            if (abort_s) {
              stop = true;
              break;
            }
            // the segment's flag travels with its last tile's arrival
            if (p0 + pt + ppt >= n_pieces) seg_bad_s[ord & 7] = bad;
            const uint32_t fb = smem_u32(&full_bar[st]);
            mbar_arrive_expect_tx(fb, C::kStageBytes);
            const uint32_t kdst = smem_u32(ring + st * C::kStageBytes);
            const uint32_t vdst = kdst + C::kTileBytes;
            for (int pc = 0; pc < ppt; ++pc) {
              const int coord = coord_s[pt + pc];
#pragma unroll
              for (int dc = 0; dc < D / 64; ++dc) {  // one box per 64-dim chunk
                const uint32_t off = dc * (kTile * 128) + pc * box_bytes;
                tma_load_4d(kdst + off, &tmap_k, 0, coord, sg.h, dc, fb);
                tma_load_4d(vdst + off, &tmap_v, 0, coord, sg.h, dc, fb);
              }
            }
          }
        }
        stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
        it = __shfl_sync(0xffffffffu, it, 0);
      }
      if (bad && lane == 0) raise_error(a.err, DECODE_ATTN_DEV_BAD_PAGE);
      wk.advance(sg);
      ++ord;
    }
    if (lane == 0)  // leave no copy in flight into this CTA's shared memory
      for (int i = max(0, it - C::kStages); i < it; ++i)
        mbar_wait(smem_u32(&full_bar[i % C::kStages]), (i / C::kStages) & 1);
    return;
  }

  // ========================================================== consumers
  const int G = a.G;
  const int R = a.T * G;
  const int gid = lane >> 2, tig = lane & 3;
  const int nthreads = kWarps * 32;
  float* slot_f = reinterpret_cast<float*>(slot);
  SegWalker wk;
  wk.start(prefix_s, pa.B, hh, g0, g1);
  int it = 0, ord = 0;
  while (!wk.done()) {
    const Segment sg = wk.current();
    const int b = sg.b, h = sg.h;
    const SeqRange r = seq_range(a.seq_lens[b], a.window, capacity, 1 << 30, 1, a.T);
    const int seg_lo = r.base + sg.t0 * kTile;
    const int lo = max(r.start, seg_lo);
    const int hi = min(r.end, seg_lo + sg.nt * kTile);

    uint32_t qf[NT8][KS][2];
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
      const int rr = 8 * j + gid;
      const uint16_t* qrow =
          static_cast<const uint16_t*>(a.q) + group_row(b, h, rr < R ? rr : 0, a.T, G, a.Hq) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[j][ks][0] = rr < R ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tig) : 0u;
        qf[j][ks][1] =
            rr < R ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tig) : 0u;
      }
    }
    int col_lo[NT8][2], col_hi[NT8][2];
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int rr = 8 * j + 2 * tig + e;
        const int t = rr < R ? rr / G : a.T - 1;
        col_hi[j][e] = r.end - a.T + t + 1;
        col_lo[j][e] = a.window > 0 ? max(0, col_hi[j][e] - a.window) : 0;
      }
    float acc[KS][NT8][4];
    float m_run[NT8][2], l_part[NT8][2];
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
#pragma unroll
      for (int mi = 0; mi < KS; ++mi) acc[mi][j][0] = acc[mi][j][1] = acc[mi][j][2] =
          acc[mi][j][3] = 0.f;
      m_run[j][0] = m_run[j][1] = -INFINITY;
      l_part[j][0] = l_part[j][1] = 0.f;
    }

    bool timed_out = false;
    for (int k = 0; k < sg.nt; ++k, ++it) {
      const int st = it % C::kStages;
      if (!mbar_wait(smem_u32(&full_bar[st]), (it / C::kStages) & 1)) {
        abort_s = 1;
        raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
        timed_out = true;
        break;
      }
      if (abort_s) {
        timed_out = true;
        break;
      }
      const int tok0 = seg_lo + k * kTile + 16 * warp;
      if (tok0 + 16 > lo && tok0 < hi)
        // per-chunk boxes: the stage is one piece of 64 rows
        mma_block<D, NT8, E>(ring + st * C::kStageBytes, warp, lane, tok0, lo, hi, col_lo,
                             col_hi, qf, a.scale_log2, acc, m_run, l_part, 6);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    }
    // every consumer saw the same abort flag only once all are here
    named_barrier_sync(1, nthreads);
    if (timed_out || abort_s) return;  // all consumer warps leave together
    const bool dead = seg_bad_s[ord & 7] != 0;

    // ---- fold warps 1..3 into warp 0, in order, through the slot -------
    for (int w = 1; w < kWarps; ++w) {
      if (warp == w) {
        int q = 0;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi)
#pragma unroll
          for (int j = 0; j < NT8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) slot_f[(q++) * 32 + lane] = acc[mi][j][e];
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            slot_f[(q++) * 32 + lane] = m_run[j][e];
            slot_f[(q++) * 32 + lane] = l_part[j][e];
          }
      }
      named_barrier_sync(1, nthreads);
      if (warp == 0) {
        constexpr int kAcc = KS * NT8 * 4;
        float fa[NT8][2], fb[NT8][2];
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mw = slot_f[(kAcc + (j * 2 + e) * 2) * 32 + lane];
            const float lw = slot_f[(kAcc + (j * 2 + e) * 2 + 1) * 32 + lane];
            const float M = fmaxf(m_run[j][e], mw);
            fa[j][e] = (M == -INFINITY) ? 0.f : fast_exp2(m_run[j][e] - M);
            fb[j][e] = (M == -INFINITY) ? 0.f : fast_exp2(mw - M);
            l_part[j][e] = l_part[j][e] * fa[j][e] + lw * fb[j][e];
            m_run[j][e] = M;
          }
        int q = 0;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi)
#pragma unroll
          for (int j = 0; j < NT8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e, ++q)
              acc[mi][j][e] = acc[mi][j][e] * fa[j][e & 1] + slot_f[q * 32 + lane] * fb[j][e & 1];
      }
      named_barrier_sync(1, nthreads);
    }

    // ---- this segment's result: output rows or a partial slot ----------
    const bool complete = sg.u0 >= g0 && sg.u0 + sg.n <= g1;
    int c_first = jr, c_last = jr, jslot = 0;  // ranges of head h holding the unit
    if (!complete) {
      c_first = cta_of_tile(sg.u0, W, N);
      c_last = cta_of_tile(sg.u0 + sg.n - 1, W, N);
      jslot = (jr == c_first && range_start(jr, W, N) < sg.u0) ? 1 : 0;
    }
    if (warp == 0) {
#pragma unroll
      for (int j = 0; j < NT8; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float l = l_part[j][e];
          l += __shfl_xor_sync(0xffffffffu, l, 4);
          l += __shfl_xor_sync(0xffffffffu, l, 8);
          l += __shfl_xor_sync(0xffffffffu, l, 16);
          l_part[j][e] = l;
          if (gid == 0) ml_s[8 * j + 2 * tig + e] = make_float2(m_run[j][e], l);
        }
#pragma unroll
      for (int mi = 0; mi < KS; ++mi)
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int rr = 8 * j + 2 * tig + (e & 1);
            if (rr >= R) continue;
            const int d = 16 * mi + gid + ((e & 2) ? 8 : 0);
            const float L = l_part[j][e & 1];
            if (complete) {
              const size_t row = group_row(b, h, rr, a.T, G, a.Hq);
              static_cast<uint16_t*>(a.out)[row * D + d] =
                  ElemOps<E>::round((dead || L == 0.f) ? 0.f : acc[mi][j][e] / L);
            } else {
              const size_t sl = ((size_t)c * 2 + jslot) * R + rr;
              a.ws_acc[sl * D + d] = dead ? 0.f : acc[mi][j][e];
            }
          }
      if (!complete) {
        __syncwarp();
        for (int rr = lane; rr < R; rr += 32) {
          const size_t sl = ((size_t)c * 2 + jslot) * R + rr;
          const float2 ml = ml_s[rr];
          a.ws_ml[sl] = make_float2(ml.x, dead ? -1.f : ml.y);
        }
      }
    }
    if (!complete) {
      // the last of the unit's CTAs to finish merges its partials in order
      __threadfence();
      named_barrier_sync(1, nthreads);
      int32_t* ticket = a.counters + (size_t)b * a.Hkv + h;
      const int nseg = c_last - c_first + 1;
      if (threadIdx.x == 0) {
        const int old = atomicAdd(ticket, 1);
        if (old < 0 || old >= nseg) raise_error(a.err, DECODE_ATTN_DEV_WORKSPACE);
        is_last_s = old == nseg - 1;
      }
      named_barrier_sync(1, nthreads);
      if (is_last_s) {
        __threadfence();
        CombineArgs cm{};
        cm.seq_lens = a.seq_lens;
        cm.err = a.err;
        cm.ws_acc = a.ws_acc;
        cm.ws_ml = a.ws_ml;
        cm.out = a.out;
        cm.B = pa.B;
        cm.Hq = a.Hq;
        cm.G = G;
        cm.T = a.T;
        cm.capacity = capacity;
        cm.window = a.window;
        cm.chunk = 0;
        cm.max_shards = 0;
        const bool first_is_tail = range_start(c_first, W, N) < sg.u0;
        const int cap = (persist_slot_bytes<D, NT8>() - merge_smem_bytes(R, 0)) / (R * 8);
        const int hkv = a.Hkv;
        merge_group<D, E>(cm, b, h, nseg, false, threadIdx.x, nthreads, slot, cap,
                          [nthreads] { named_barrier_sync(1, nthreads); },
                          [=](int rr, int sidx) -> size_t {
                            const int cc = (c_first + sidx) * hkv + h;  // CTA of that range
                            const int jj = (sidx == 0 && first_is_tail) ? 1 : 0;
                            return ((size_t)cc * 2 + jj) * R + rr;
                          });
        if (threadIdx.x == 0) *ticket = 0;
      }
      named_barrier_sync(1, nthreads);  // the slot is reused by the next segment
    }
    wk.advance(sg);
    ++ord;
  }
}

}  // namespace pgd
