// Split decode-attention kernel, CUDA-core variant.
//
// One CTA owns (shard s, KV head h, batch entry b): it streams the shard's
// K/V rows of head h once and serves all G query heads of the group from
// each row (BackendStack21/mlx-runner pull request 3, commit "GQA-shared
// split attention").  The shard keeps an online-softmax state (running max,
// sum, fp32 accumulator; apache/tvm pull request 20426, sharded-nest commit)
// and either writes it as a partial for the ordered combine or, when the
// sequence is a single shard, normalises and writes the fp16 output.
//
// Data movement: one producer warp copies 64-token tiles of K and V from the
// paged pool into a ring of shared-memory stages with 3-D TMA boxes (one box
// per page, or per 64 tokens of a larger page), gated by full/empty
// mbarriers.  Positions outside the attended range are never loaded from a
// page: their boxes point past the pool and TMA fills them with zeros.
//
// Compute: each consumer warp takes groups of NT = 32/GP tokens; every lane
// holds D/32 dims of q for all GP heads, forms the GP*NT partial dot
// products, and one reduce-scatter over the 32 lanes (31 shuffles) leaves
// each lane with one complete score (token lane/GP, head lane%GP).  The max
// is a shuffle butterfly over the lanes of a head; p and the rescale factors
// go through a per-warp shared-memory slot, and each lane accumulates p*v
// for its dims and all heads.  Scores are scaled by scale*log2(e) in fp32
// and exponentiated with ex2.
#pragma once

#include "combine.cuh"  // CombineArgs, grid_launch_dependents
#include "device_common.cuh"

namespace pgd {

struct SplitArgs {
  const void* q;              // [B][T][Hq][D] 16-bit elements (fp16 or bf16)
  const int32_t* page_table;  // [B][max_pages]
  const int32_t* seq_lens;    // [B]
  void* out;                  // [B][T][Hq][D]       (single pass and merge)
  float* ws_acc;              // [B*Hq*S_max][D]     (split)
  float2* ws_ml;              // [B*Hq*S_max] (m, l) (split; l = -1 marks a bad row)
  int32_t* counters;          // [B*Hkv] shards finished per group (split; zero on entry)
  int32_t* err;               // nullable
  const void* k_new;          // [B][T][Hkv][D] rows to append at the last T positions, or null
  const void* v_new;
  void* k_pages_w;            // the pool, written only when appending
  void* v_pages_w;
  int32_t Hq, Hkv, G;
  int32_t max_pages, num_pages, page_size, page_shift, box_tokens;
  int32_t window, chunk, max_shards, split;
  int32_t balanced;           // shards of each sequence of near-equal length (seq_range)
  int32_t T;                  // query positions per sequence (1 for the CUDA-core variant)
  int32_t head_fastest;       // grid (Hkv, S, B) when set, else (S, Hkv, B)
  int32_t stall_tx;           // 0; a test sets extra bytes on the first stage's barrier
  int32_t batch;              // B (the checked build's bounds)
  int32_t len_hint;           // the plan's bound on seq_lens (the speculative page-id read)
  float scale_log2;           // scale * log2(e)
};

template <int D>
struct SimtCfg {
  static constexpr int kWarps = 4;  // consumer warps; one more warp produces
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kStages = (D == 64) ? 6 : 3;
  static constexpr int kTileBytes = kTile * D * 2;  // K or V of one stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kRingBytes + 1024;  // + alignment slack
};

// DPL consecutive fp16 values -> fp32.
template <int DPL>
__device__ __forceinline__ void load_f16_row(const __half* p, float (&f)[DPL]) {
  static_assert(DPL == 2 || DPL == 4 || DPL == 8, "dims per lane");
  if constexpr (DPL == 2) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(p));
    f[0] = v.x;
    f[1] = v.y;
  } else if constexpr (DPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = a.x;
      f[2 * i + 1] = a.y;
    }
  }
}

// v[0..31] per lane -> v[0] of lane L holds the sum over all lanes of v[L].
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  return v[0];
}

template <int D, int GP>
__device__ __forceinline__ void zero_group_rows(const SplitArgs& a, int b, int h) {
  uint16_t* out = static_cast<uint16_t*>(a.out);  // +0.0 is all zero bits in both formats
  for (int e = threadIdx.x; e < a.T * a.G * D; e += blockDim.x) {
    const int g = e / D, d = e % D;
    const size_t i = group_row(b, h, g, a.T, a.G, a.Hq) * D + d;
    if (PGD_IN(i, (size_t)a.batch * a.T * a.Hq * D, a.err)) out[i] = 0;
  }
}

// Fused append (producer warp, before any TMA of this CTA): the CTA holding
// a sequence's last position writes the step's new K/V rows of its head
// there, then fences the generic-proxy writes against the TMA reads that
// follow (the rows are read back through L2 like every other row).
template <int D>
__device__ __forceinline__ void append_new_rows(const SplitArgs& a, const SeqRange& r, int b,
                                                int h, int shard_lo, int lane) {
  for (int i = 0; i < a.T; ++i) {
    const int pos = r.end - a.T + i;  // position of the i-th new token
    if (pos < shard_lo || pos >= shard_lo + r.chunk || pos < 0) continue;
    const size_t pi = (size_t)b * a.max_pages + (pos >> a.page_shift);
    if (!PGD_IN(pi, (size_t)a.batch * a.max_pages, a.err)) continue;
    const int phys = a.page_table[pi];
    const size_t off =
        (((size_t)phys * a.page_size + (pos & (a.page_size - 1))) * a.Hkv + h) * D;
    const size_t src = (((size_t)b * a.T + i) * a.Hkv + h) * D;
    if (!PGD_IN(off + D - 1, (size_t)a.num_pages * a.page_size * a.Hkv * D, a.err) ||
        !PGD_IN(src + D - 1, (size_t)a.batch * a.T * a.Hkv * D, a.err))
      continue;
    const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.k_new) + src);
    const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.v_new) + src);
    uint4* kd = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.k_pages_w) + off);
    uint4* vd = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.v_pages_w) + off);
    for (int c = lane; c < D / 8; c += 32) {
      kd[c] = ks[c];
      vd[c] = vs[c];
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

// Split path epilogue, run by the consumer threads [0, nthreads) after this
// CTA's partial is written: the last CTA of the group to finish (an atomic
// ticket; no CTA ever waits on another) merges the group's partials into the
// output in ascending shard order and clears the ticket for the next call.
// The ticket is one acquire-release atomic of thread 0 after a barrier of
// the writing threads: its release publishes the whole CTA's partial (the
// barrier orders the other threads' writes before it), and in the last CTA
// its acquire, passed on by the next barrier, makes every other CTA's
// partial visible to the merge.
// kOneTrip: as merge_group's (0: the staged form for every group).
template <int D, class E = __half, int kOneTrip = 0>
__device__ __forceinline__ void merge_if_last(const SplitArgs& a, const SeqRange& r, int b, int h,
                                              uint8_t* smem, int nthreads) {
  __shared__ int is_last_s;
  named_barrier_sync(1, nthreads);  // every thread's partial writes are issued
  int32_t* ticket = a.counters + (size_t)b * a.Hkv + h;
  if (!PGD_IN((size_t)b * a.Hkv + h, (size_t)a.batch * a.Hkv, a.err)) return;
  if (threadIdx.x == 0) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(ticket)
                 : "memory");
    if (old < 0 || old >= r.nshards) raise_error(a.err, DECODE_ATTN_DEV_WORKSPACE);
    is_last_s = old == r.nshards - 1;
  }
  named_barrier_sync(1, nthreads);
  if (!is_last_s) return;
  CombineArgs c{};
  c.seq_lens = a.seq_lens;
  c.ws_acc = a.ws_acc;
  c.ws_ml = a.ws_ml;
  c.out = a.out;
  c.err = a.err;
  c.B = a.batch;
  c.Hq = a.Hq;
  c.G = a.G;
  c.T = a.T;
  c.capacity = a.max_pages * a.page_size;
  c.window = a.window;
  c.chunk = a.chunk;
  c.balanced = a.balanced;
  c.max_shards = a.max_shards;
  merge_group<D, E, kOneTrip>(c, b, h, r.nshards, false, threadIdx.x, nthreads, smem,
                              kShardBlock, [nthreads] { named_barrier_sync(1, nthreads); },
                              GridSlots{b, h, a.T, a.G, a.Hq, a.max_shards});
  if (threadIdx.x == 0) *ticket = 0;
}

template <int D, int GP>
__global__ void __launch_bounds__(SimtCfg<D>::kThreads)
    split_simt_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
  using C = SimtCfg<D>;
  constexpr int DPL = D / 32;  // dims per lane
  constexpr int NT = 32 / GP;  // tokens per reduce-scatter group
  constexpr int kWarps = C::kWarps;
  static_assert(kTile % NT == 0, "token groups tile the stage");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ int32_t coord_s[kMaxPieces];
  __shared__ float p_s[kWarps][32];
  __shared__ float alpha_s[kWarps][GP];
  __shared__ float2 ml_s[kWarps][GP];
  __shared__ int32_t bad_s;
  __shared__ volatile int32_t abort_s;

  // launched as a programmatic dependent of the preceding kernel: its CTAs
  // may become resident while that kernel drains, but nothing is read or
  // written before it has completed
  grid_dependency_wait();
  // a kernel launched after this one (a combine, the next step) may be
  // scheduled now; it waits the same way before touching memory
  grid_launch_dependents();
  // grid order: head fastest for plans of several waves (the Hkv CTAs of one
  // (sequence, shard) start together and read the rows of the same positions,
  // adjacent in the pool, side by side), shard fastest for one-wave plans
  // (a group's shards run on neighbouring SMs for its merge)
  const int h = a.head_fastest ? blockIdx.x : blockIdx.y;
  const int s = a.head_fastest ? blockIdx.y : blockIdx.x;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqRange r = seq_range(a.seq_lens[b], a.window, a.max_pages * a.page_size, a.chunk,
                               a.max_shards, a.T, a.balanced);
  if (r.status != 0 || s >= r.nshards) {
    // nothing to stream: report a bad length once; shard 0 owns the group's
    // output rows (zero for an empty or invalid range)
    if (s == 0) {
      if (r.status != 0 && threadIdx.x == 0) raise_error(a.err, r.status);
      zero_group_rows<D, GP>(a, b, h);
    }
    return;
  }

  const int shard_lo = r.base + s * r.chunk;  // tile-aligned absolute position
  const int lo = max(r.start, shard_lo);
  const int hi = min(r.end, shard_lo + r.chunk);
  const int n_tiles = (hi - shard_lo + kTile - 1) / kTile;
  const int box_t = a.box_tokens;
  const int pieces_per_tile = kTile / box_t;
  const int n_pieces = n_tiles * pieces_per_tile;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));

  if (warp == kWarps) {
    // producer warp: physical coordinates of every box of the shard
    int bad = 0;
    const int oob = a.num_pages * a.page_size;  // past the pool: TMA writes zeros
    for (int i = lane; i < n_pieces; i += 32) {
      const int ptok = shard_lo + i * box_t;
      int coord = oob;
      if (ptok < hi && ptok + box_t > lo) {
        const size_t pi = (size_t)b * a.max_pages + (ptok >> a.page_shift);
        const int phys =
            PGD_IN(pi, (size_t)a.batch * a.max_pages, a.err) ? a.page_table[pi] : -1;
        if (phys < 0 || phys >= a.num_pages) {
          bad = 1;
        } else {
          coord = phys * a.page_size + (ptok & (a.page_size - 1));
        }
      }
      coord_s[i] = coord;
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      bad_s = bad;
      abort_s = 0;
      for (int st = 0; st < C::kStages; ++st) {
        mbar_init(smem_u32(&full_bar[st]), 1);
        mbar_init(smem_u32(&empty_bar[st]), kWarps);
      }
      fence_mbar_init();
      if (bad) raise_error(a.err, DECODE_ATTN_DEV_BAD_PAGE);
    }
  }
  __syncthreads();
  const bool bad = bad_s != 0;

  if (warp == kWarps) {
    if (a.k_new != nullptr && !bad) {
      const int shard_lo_w = r.base + s * r.chunk;
      if (r.end - a.T < shard_lo_w + r.chunk && r.end > shard_lo_w)
        append_new_rows<D>(a, r, b, h, shard_lo_w, lane);
    }
    if (lane == 0 && !bad) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
      const uint32_t box_bytes = box_t * D * 2;
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % C::kStages;
        if (i >= C::kStages &&
            !mbar_wait(smem_u32(&empty_bar[st]), ((i / C::kStages) & 1) ^ 1)) {
          abort_s = 1;
          raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
          break;
        }
        if (abort_s) break;
        const uint32_t fb = smem_u32(&full_bar[st]);
        mbar_arrive_expect_tx(fb, C::kStageBytes);
        const uint32_t kdst = smem_u32(ring + st * C::kStageBytes);
        const uint32_t vdst = kdst + C::kTileBytes;
        for (int pc = 0; pc < pieces_per_tile; ++pc) {
          int coord = coord_s[i * pieces_per_tile + pc];
          const int pool_rows = a.num_pages * a.page_size;  // (checked build) see split_mma
          if (!PGD_IN(coord == pool_rows ? 0 : (int64_t)coord + box_t - 1, pool_rows, a.err))
            coord = pool_rows;
          tma_load_3d(kdst + pc * box_bytes, &tmap_k, 0, h, coord, fb);
          tma_load_3d(vdst + pc * box_bytes, &tmap_v, 0, h, coord, fb);
        }
        issued = i + 1;
      }
      // leave no copy in flight into this CTA's shared memory
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(smem_u32(&full_bar[i % C::kStages]), (i / C::kStages) & 1);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int G = a.G;
  float qf[GP][DPL];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    if (g < G && PGD_IN((size_t)b * a.Hq + h * G + g, (size_t)a.batch * a.Hq, a.err)) {
      load_f16_row<DPL>(static_cast<const __half*>(a.q) + ((size_t)b * a.Hq + h * G + g) * D +
                            lane * DPL,
                        qf[g]);
    } else {
#pragma unroll
      for (int i = 0; i < DPL; ++i) qf[g][i] = 0.f;
    }
  }
  float acc[GP][DPL];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[g][i] = 0.f;
  float m_run = -INFINITY;  // running max (log2 units) of head lane % GP
  float l_lane = 0.f;       // this lane's share of the running sum
  const int my_j = lane / GP;

  for (int i = 0; i < n_tiles && !bad; ++i) {
    const int st = i % C::kStages;
    if (!mbar_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1)) {
      abort_s = 1;
      raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
      break;
    }
    if (abort_s) break;
    const __half* Ks = reinterpret_cast<const __half*>(ring + st * C::kStageBytes);
    const __half* Vs = Ks + kTile * D;
    const int tok0 = shard_lo + i * kTile;
    for (int gi = warp; gi < kTile / NT; gi += kWarps) {
      const int g0 = tok0 + gi * NT;
      if (g0 + NT <= lo || g0 >= hi) continue;  // whole group outside the range
      float part[32];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float kf[DPL];
        load_f16_row<DPL>(Ks + (gi * NT + j) * D + lane * DPL, kf);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < DPL; ++e) dot = fmaf(qf[g][e], kf[e], dot);
          part[j * GP + g] = dot;
        }
      }
      const float sc = reduce_scatter32(part, lane);
      const int tok = g0 + my_j;
      const float sv = (tok >= lo && tok < hi) ? sc * a.scale_log2 : -INFINITY;
      float mx = sv;
#pragma unroll
      for (int o = GP; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
      const float p = (sv == -INFINITY) ? 0.f : fast_exp2(sv - m_new);
      l_lane = l_lane * alpha + p;
      m_run = m_new;
      p_s[warp][lane] = p;
      if (lane < GP) alpha_s[warp][lane] = alpha;
      __syncwarp();
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float al = alpha_s[warp][g];
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[g][e] *= al;
        }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int tj = g0 + j;
        if (tj < lo || tj >= hi) continue;  // same for the whole warp
        float vf[DPL];
        load_f16_row<DPL>(Vs + (gi * NT + j) * D + lane * DPL, vf);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float pj = p_s[warp][j * GP + g];
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[g][e] = fmaf(pj, vf[e], acc[g][e]);
        }
      }
      __syncwarp();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
  }

  // ---- merge the consumer warps in fixed order (deterministic) ----------
#pragma unroll
  for (int o = GP; o < 32; o <<= 1) l_lane += __shfl_xor_sync(0xffffffffu, l_lane, o);
  named_barrier_sync(1, kWarps * 32);  // every consumer is done with the ring
  float* acc_s = reinterpret_cast<float*>(ring);  // [kWarps][GP][D]
  if (lane < GP) ml_s[warp][lane] = make_float2(m_run, l_lane);
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc_s[(warp * GP + g) * D + lane * DPL + e] = acc[g][e];
  named_barrier_sync(1, kWarps * 32);
  const bool dead = bad || abort_s != 0;

  for (int e = threadIdx.x; e < G * D; e += kWarps * 32) {
    const int g = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml_s[w][g].x);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float2 ml = ml_s[w][g];
      if (ml.y == 0.f) continue;
      const float c = fast_exp2(ml.x - M);
      L += c * ml.y;
      O += c * acc_s[(w * GP + g) * D + d];
    }
    const size_t row = (size_t)b * a.Hq + h * G + g;
    if (!PGD_IN(row, (size_t)a.batch * a.Hq, a.err)) continue;
    if (!a.split) {
      static_cast<__half*>(a.out)[row * D + d] = __float2half_rn((dead || L == 0.f) ? 0.f : O / L);
    } else {
      const size_t slot = row * a.max_shards + s;
      if (!PGD_IN(slot, (size_t)a.batch * a.Hq * a.max_shards, a.err)) continue;
      a.ws_acc[slot * D + d] = dead ? 0.f : O;
      if (d == 0) a.ws_ml[slot] = make_float2(M, dead ? -1.f : L);
    }
  }
  if (a.split) merge_if_last<D>(a, r, b, h, ring, kWarps * 32);
}

}  // namespace pgd
