// Split decode-attention kernel, tensor-core variant.
//
// Same CTA shape, shard arithmetic, TMA producer and fixed-order epilogue as
// the CUDA-core variant (split_simt.cuh); only the q.k and p.v products move
// to mma.sync.m16n8k16 (fp16 x fp16 -> fp32), with tokens on the 16-row M
// side and the G query heads of the group on the N side (N = 8 per tile, two
// tiles for G up to 16):
//   scores^T [16 tok x 8 heads] = K [16 tok x D] . Q^T [D x 8 heads]
//   out^T    [D x 8 heads]     += V^T [D x 16 tok] . P^T [16 tok x 8 heads]
// The score accumulator's fragment is transposed into the P^T operand with
// movmatrix; P is split into an fp16 head and an fp16 remainder (two mma per
// tile) so the weights keep about twice the element format's bits (22 for
// fp16, 16 for bf16).  Templated on the element format E (fp16 or bf16).
//
// A stage's K (and V) tile is 64 tokens made of pieces of box_t = min(page,
// 64) rows, one TMA box each, every piece laid out [D/64][box_t rows][64
// dims] with the 128-byte TMA swizzle (16-byte chunk c of token row t lives
// at chunk c ^ (t % 8)), so every ldmatrix of 8 token rows touches 8
// distinct bank groups (swz_offset).
#pragma once

#include "split_simt.cuh"  // SplitArgs, zero_group_rows

namespace pgd {

// kShallow: the ring of plans made of many short shards, 2 stages (4 at
// D = 64) instead of 3 (6), so that 3 CTAs fit per SM and more CTAs' first
// round trips overlap.
template <int D, bool kShallow = false>
struct MmaCfg {
  static constexpr int kWarps = 4;  // consumer warps, 16 tokens of each stage apiece
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kStages = (D == 64) ? (kShallow ? 4 : 6) : (kShallow ? 2 : 3);
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kRingBytes + 1024;
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of (row t, dim d) inside a swizzled tile made of pieces of
// 2^ps rows, one TMA box each, laid out [D/64][2^ps rows][64 dims] (the
// 128-byte swizzle: 16-byte chunk c of row t at c ^ (t % 8)).  A tile that is
// one piece (2^ps = its rows) is [D/64][rows][64].
template <int D>
__device__ __forceinline__ uint32_t swz_offset(int t, int d, int ps) {
  const int bt = 1 << ps;
  return (uint32_t)((t >> ps) * (bt * D * 2) + (d >> 6) * (bt * 128) + (t & (bt - 1)) * 128 +
                    ((((d >> 3) & 7) ^ (t & 7)) << 4));
}

struct NoRelease {
  __device__ void operator()() const {}
};

// One consumer warp's 16 positions [tok0, tok0 + 16) of a staged tile:
// scores^T = K . Q^T, the per-column causal / window mask, the online
// softmax update and out^T += V^T . P^T.  kt points at the stage's K tile of
// kRows rows in pieces of 2^ps rows (swz_offset), the warp's 16 rows at
// 16 * warp (V follows at kRows * D * 2 bytes); [lo, hi) is the union of the
// columns' ranges clipped to the shard, and the block must overlap it.  kFetchFirst: all of
// the warp's K and V fragments are loaded into registers first and
// release() is called before any arithmetic, so the stage can be refilled
// while the warp computes (the same operations in the same order).
template <int D, int NT8, class E, int kRows = kTile, bool kFetchFirst = false,
          class Release = NoRelease>
__device__ __forceinline__ void mma_block(uint8_t* kt, int warp, int lane, int tok0, int lo,
                                          int hi, const int (&col_lo)[NT8][2],
                                          const int (&col_hi)[NT8][2],
                                          const uint32_t (&qf)[NT8][D / 16][2], float scale_log2,
                                          float (&acc)[D / 16][NT8][4], float (&m_run)[NT8][2],
                                          float (&l_part)[NT8][2], int ps,
                                          Release release = {}) {
  constexpr int kTileBytes = kRows * D * 2;
  constexpr int KS = D / 16;
  const int gid = lane >> 2;
  const int mat = lane >> 3, mrow = lane & 7;
  const int k_tok = 16 * warp + mrow + ((mat & 1) ? 8 : 0);  // K: matrix bit 0 -> +8 tokens
  const int k_dof = (mat & 2) ? 8 : 0;                       // K: matrix bit 1 -> +8 dims
  const int v_tok = 16 * warp + mrow + ((mat & 2) ? 8 : 0);  // V: matrix bit 1 -> +8 tokens
  const int v_dof = (mat & 1) ? 8 : 0;                       // V: matrix bit 0 -> +8 dims
  const uint32_t kbase = smem_u32(kt);
  const uint32_t vbase = kbase + kTileBytes;
  if (tok0 < lo || tok0 + 16 > hi) {
    // rows of this block outside the range: clear their V rows so a
    // zero weight never meets a non-finite cache value
    uint8_t* vt = kt + kTileBytes;
    for (int e = lane; e < 16 * (D / 8); e += 32) {
      const int t = e / (D / 8), c = e % (D / 8);
      const int tok = tok0 + t;
      if (tok < lo || tok >= hi)
        *reinterpret_cast<uint4*>(vt + swz_offset<D>(16 * warp + t, c * 8, ps)) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncwarp();
  }
  constexpr int kHeld = kFetchFirst ? KS : 1;
  uint32_t kf[kHeld][4], vf[kHeld][4];
  if constexpr (kFetchFirst) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldmatrix_x4(kf[ks], kbase + swz_offset<D>(k_tok, ks * 16 + k_dof, ps));
#pragma unroll
    for (int mi = 0; mi < KS; ++mi)
      ldmatrix_x4_trans(vf[mi], vbase + swz_offset<D>(v_tok, mi * 16 + v_dof, ps));
    release();
  }
  // scores^T = K . Q^T
  float sc[NT8][4];
#pragma unroll
  for (int j = 0; j < NT8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
  if constexpr (kFetchFirst) {
    // two independent accumulation chains (even and odd k-steps), added at
    // the end: half the dependent mma latency on the warp's critical path
    float sc1[NT8][4];
#pragma unroll
    for (int j = 0; j < NT8; ++j) sc1[j][0] = sc1[j][1] = sc1[j][2] = sc1[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ks += 2) {
#pragma unroll
      for (int j = 0; j < NT8; ++j) {
        ElemOps<E>::mma(sc[j], kf[ks], qf[j][ks][0], qf[j][ks][1]);
        ElemOps<E>::mma(sc1[j], kf[ks + 1], qf[j][ks + 1][0], qf[j][ks + 1][1]);
      }
    }
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[j][e] += sc1[j][e];
  } else {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t af[4];
      ldmatrix_x4(af, kbase + swz_offset<D>(k_tok, ks * 16 + k_dof, ps));
#pragma unroll
      for (int j = 0; j < NT8; ++j) ElemOps<E>::mma(sc[j], af, qf[j][ks][0], qf[j][ks][1]);
    }
  }
  // online softmax over this block's 16 positions
  const int tok_a = tok0 + gid, tok_b = tok0 + gid + 8;
  uint32_t pb_hi[NT8][2], pb_lo[NT8][2];
  bool rescale = false;
  float alpha[NT8][2];
#pragma unroll
  for (int j = 0; j < NT8; ++j) {
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = (e < 2) ? tok_a : tok_b;
      const bool ok = tok >= col_lo[j][e & 1] && tok < col_hi[j][e & 1];
      sc[j][e] = ok ? sc[j][e] * scale_log2 : -INFINITY;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mx = fmaxf(sc[j][e], sc[j][e + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run[j][e], mx);
      alpha[j][e] = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run[j][e] - m_new);
      rescale |= alpha[j][e] != 1.f;
      p[e] = (sc[j][e] == -INFINITY) ? 0.f : fast_exp2(sc[j][e] - m_new);
      p[e + 2] = (sc[j][e + 2] == -INFINITY) ? 0.f : fast_exp2(sc[j][e + 2] - m_new);
      l_part[j][e] = l_part[j][e] * alpha[j][e] + p[e] + p[e + 2];
      m_run[j][e] = m_new;
    }
    // P^T operand: fp16 head and fp16 remainder, transposed by movmatrix
    const uint32_t h0 = ElemOps<E>::pack2(p[0], p[1]);
    const uint32_t h1 = ElemOps<E>::pack2(p[2], p[3]);
    const float2 f0 = ElemOps<E>::unpack2(h0);
    const float2 f1 = ElemOps<E>::unpack2(h1);
    const uint32_t l0 = ElemOps<E>::pack2(p[0] - f0.x, p[1] - f0.y);
    const uint32_t l1 = ElemOps<E>::pack2(p[2] - f1.x, p[3] - f1.y);
    pb_hi[j][0] = movmatrix_trans(h0);
    pb_hi[j][1] = movmatrix_trans(h1);
    pb_lo[j][0] = movmatrix_trans(l0);
    pb_lo[j][1] = movmatrix_trans(l1);
  }
  if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
    for (int mi = 0; mi < KS; ++mi)
#pragma unroll
      for (int j = 0; j < NT8; ++j) {
        acc[mi][j][0] *= alpha[j][0];
        acc[mi][j][1] *= alpha[j][1];
        acc[mi][j][2] *= alpha[j][0];
        acc[mi][j][3] *= alpha[j][1];
      }
  }
  // out^T += V^T . P^T
#pragma unroll
  for (int mi = 0; mi < KS; ++mi) {
    uint32_t af[4];
    if constexpr (kFetchFirst) {
      af[0] = vf[mi][0], af[1] = vf[mi][1], af[2] = vf[mi][2], af[3] = vf[mi][3];
    } else {
      ldmatrix_x4_trans(af, vbase + swz_offset<D>(v_tok, mi * 16 + v_dof, ps));
    }
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
      ElemOps<E>::mma(acc[mi][j], af, pb_hi[j][0], pb_hi[j][1]);
      ElemOps<E>::mma(acc[mi][j], af, pb_lo[j][0], pb_lo[j][1]);
    }
  }
}

// Where a CTA of a cluster plan keeps its shard's partial for the cluster's
// merge: after the warps' states in the (by then idle) ring, out [GP][D]
// fp32, then (m, l) [GP] float2 (l = -1: a dead shard).
template <int D, int NT8>
struct ClusterPartial {
  static constexpr int kRowStride = D + 4;
  static constexpr int kOutOffset = ((MmaCfg<D>::kWarps * 8 * NT8 * kRowStride * 4) + 15) & ~15;
  static constexpr int kMlOffset = kOutOffset + 8 * NT8 * D * 4;
  static constexpr int kEnd = kMlOffset + 8 * NT8 * 8;
  static_assert(kEnd <= MmaCfg<D>::kRingBytes, "the partial fits in the ring");
};

__device__ __forceinline__ uint8_t* ring_base() {
  extern __shared__ uint8_t smem_raw[];
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                    ~uintptr_t(1023));
}

// The split kernel's body, shared by the kernels below.  CL: a cluster plan
// (one cluster per (KV head, sequence), one CTA per shard): the CTA leaves
// its partial in its shared memory (and in the workspace, for
// decode_attn_combine) and the kernel's cluster merge follows.
template <int D, int NT8, class E, bool SH, bool CL = false>
__device__ __forceinline__ void split_mma_body(const CUtensorMap& tmap_k,
                                               const CUtensorMap& tmap_v, const SplitArgs& a) {
  using C = MmaCfg<D, SH>;
  constexpr int GP = 8 * NT8;  // padded heads of the group
  constexpr int KS = D / 16;   // k-steps of q.k, m-tiles of p.v
  constexpr int kWarps = C::kWarps;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ int32_t coord_s[kMaxPieces];
  __shared__ float2 ml_s[kWarps][GP];
  __shared__ float cw_s[kWarps][GP];  // each warp's weight per row
  __shared__ float2 row_s[GP];        // (M, L) per row
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
                               a.max_shards, a.T);
  if (r.status != 0 || s >= r.nshards) {
    if constexpr (CL) {
      // an empty partial (no position of any row); the cluster merge zeroes
      // rows that no shard holds
      if (s == 0 && r.status != 0 && threadIdx.x == 0) raise_error(a.err, r.status);
      using P = ClusterPartial<D, NT8>;
      uint8_t* base = ring_base();
      float* po = reinterpret_cast<float*>(base + P::kOutOffset);
      float2* pml = reinterpret_cast<float2*>(base + P::kMlOffset);
      for (int e = threadIdx.x; e < GP * D; e += blockDim.x) po[e] = 0.f;
      for (int g = threadIdx.x; g < GP; g += blockDim.x) pml[g] = make_float2(-INFINITY, 0.f);
    } else {
      if (s == 0) {
        if (r.status != 0 && threadIdx.x == 0) raise_error(a.err, r.status);
        zero_group_rows<D, GP>(a, b, h);
      }
    }
    return;
  }

  const int shard_lo = r.base + s * a.chunk;
  const int lo = max(r.start, shard_lo);
  const int hi = min(r.end, shard_lo + a.chunk);
  const int n_tiles = (hi - shard_lo + kTile - 1) / kTile;
  const int box_t = a.box_tokens;
  const int pieces_per_tile = kTile / box_t;
  const int n_pieces = n_tiles * pieces_per_tile;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));

  if (warp == kWarps) {
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
      const int shard_lo_w = r.base + s * a.chunk;
      if (r.end - a.T < shard_lo_w + a.chunk && r.end > shard_lo_w)
        append_new_rows<D>(a, r, b, h, shard_lo_w, lane);
    }
    if (lane == 0 && !bad) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
      const uint32_t box_bytes = box_t * D * 2;  // one piece: box_t rows, all D dims
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
        // (stall_tx, a test's hook, is 0: the barrier expects the stage's bytes)
        mbar_arrive_expect_tx(fb, C::kStageBytes + (i == 0 ? a.stall_tx : 0));
        const uint32_t kdst = smem_u32(ring + st * C::kStageBytes);
        const uint32_t vdst = kdst + C::kTileBytes;
        for (int pc = 0; pc < pieces_per_tile; ++pc) {
          int coord = coord_s[i * pieces_per_tile + pc];
          // (checked build) a box must lie inside the pool or start at its
          // end, where TMA fills zeros
          const int pool_rows = a.num_pages * a.page_size;
          if (!PGD_IN(coord == pool_rows ? 0 : (int64_t)coord + box_t - 1, pool_rows, a.err))
            coord = pool_rows;
          if (box_t < kTile) {  // one box holds the piece's D dims
            tma_load_4d(kdst + pc * box_bytes, &tmap_k, 0, coord, h, 0, fb);
            tma_load_4d(vdst + pc * box_bytes, &tmap_v, 0, coord, h, 0, fb);
          } else {  // 64-row pieces: one box per 64-dim chunk
#pragma unroll
            for (int dc = 0; dc < D / 64; ++dc) {
              tma_load_4d(kdst + dc * (kTile * 128), &tmap_k, 0, coord, h, dc, fb);
              tma_load_4d(vdst + dc * (kTile * 128), &tmap_v, 0, coord, h, dc, fb);
            }
          }
        }
        issued = i + 1;
      }
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(smem_u32(&full_bar[i % C::kStages]), (i / C::kStages) & 1);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int G = a.G;
  const int gid = lane >> 2, tig = lane & 3;
  const int piece_shift = __ffs(box_t) - 1;  // a stage is pieces of box_t rows
  // Q^T operand fragments, held for the whole shard
  const int R = a.T * G;  // query rows of the group: r = t * G + g
  uint32_t qf[NT8][KS][2];
#pragma unroll
  for (int j = 0; j < NT8; ++j) {
    const int rr = 8 * j + gid;
    size_t qr = group_row(b, h, rr < R ? rr : 0, a.T, G, a.Hq);
    if (!PGD_IN(qr, (size_t)a.batch * a.T * a.Hq, a.err)) qr = 0;
    const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + qr * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (rr < R) {
        qf[j][ks][0] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tig);
        qf[j][ks][1] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tig);
      } else {
        qf[j][ks][0] = qf[j][ks][1] = 0u;
      }
    }
  }
  float acc[KS][NT8][4];
#pragma unroll
  for (int mi = 0; mi < KS; ++mi)
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mi][j][e] = 0.f;
  // attended range of each of this lane's score columns (query rows
  // 8j + 2*tig + e): causal up to the row's own position, window from there
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
  float m_run[NT8][2], l_part[NT8][2];
#pragma unroll
  for (int j = 0; j < NT8; ++j) {
    m_run[j][0] = m_run[j][1] = -INFINITY;
    l_part[j][0] = l_part[j][1] = 0.f;
  }

  for (int i = 0; i < n_tiles && !bad; ++i) {
    const int st = i % C::kStages;
    if (!mbar_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1)) {
      abort_s = 1;
      raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
      break;
    }
    if (abort_s) break;
    const int tok0 = shard_lo + i * kTile + 16 * warp;  // this warp's 16 positions
    if (tok0 + 16 > lo && tok0 < hi)
      mma_block<D, NT8, E>(ring + st * C::kStageBytes, warp, lane, tok0, lo, hi, col_lo, col_hi,
                           qf, a.scale_log2, acc, m_run, l_part, piece_shift);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
  }

  // ---- merge the consumer warps in fixed order (deterministic) ----------
#pragma unroll
  for (int j = 0; j < NT8; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = l_part[j][e];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      l_part[j][e] = l;
    }
  named_barrier_sync(1, kWarps * 32);  // every consumer is done with the ring
  // the warps' states in [kWarps][GP][D + 4] fp32: the padding sends a
  // fragment's 32 stores to 32 distinct banks and keeps rows 16-byte aligned
  constexpr int kRowStride = D + 4;
  static_assert(kWarps * GP * kRowStride * 4 <= C::kRingBytes, "warp states fit in the ring");
  float* acc_s = reinterpret_cast<float*>(ring);
  if (gid == 0) {
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        ml_s[warp][8 * j + 2 * tig + e] = make_float2(m_run[j][e], l_part[j][e]);
  }
#pragma unroll
  for (int mi = 0; mi < KS; ++mi)
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
      const int hd = 8 * j + 2 * tig, d = 16 * mi + gid;
      float* base = acc_s + (warp * GP) * kRowStride;
      base[hd * kRowStride + d] = acc[mi][j][0];
      base[(hd + 1) * kRowStride + d] = acc[mi][j][1];
      base[hd * kRowStride + d + 8] = acc[mi][j][2];
      base[(hd + 1) * kRowStride + d + 8] = acc[mi][j][3];
    }
  named_barrier_sync(1, kWarps * 32);
  // per row: M = max over warps, each warp's weight c_w = 2^(m_w - M) (none
  // for a warp that saw no position of the row), L = sum_w c_w l_w in warp
  // order
  if (threadIdx.x < R) {
    const int g = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml_s[w][g].x);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float2 ml = ml_s[w][g];
      const float c = ml.y == 0.f ? 0.f : fast_exp2(ml.x - M);
      if (ml.y != 0.f) L += c * ml.y;
      cw_s[w][g] = ml.y == 0.f ? 0.f : c;
    }
    row_s[g] = make_float2(M, L);
  }
  named_barrier_sync(1, kWarps * 32);
  const bool dead = bad || abort_s != 0;

  // fold the warps, 4 dims per thread and pass, in warp order
  constexpr int kQuads = D / 4;
  for (int e = threadIdx.x; e < R * kQuads; e += kWarps * 32) {
    const int g = e / kQuads, q = e % kQuads;
    const float2 ML = row_s[g];
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float c = cw_s[w][g];
      if (c == 0.f) continue;
      const float4 x =
          *reinterpret_cast<const float4*>(acc_s + (w * GP + g) * kRowStride + 4 * q);
      O.x += c * x.x;
      O.y += c * x.y;
      O.z += c * x.z;
      O.w += c * x.w;
    }
    const size_t row = group_row(b, h, g, a.T, G, a.Hq);
    if (!PGD_IN(row, (size_t)a.batch * a.T * a.Hq, a.err)) continue;
    if (!a.split) {
      const bool z = dead || ML.y == 0.f;
      const uint32_t lo = (uint32_t)ElemOps<E>::round(z ? 0.f : O.x / ML.y) |
                          ((uint32_t)ElemOps<E>::round(z ? 0.f : O.y / ML.y) << 16);
      const uint32_t hi = (uint32_t)ElemOps<E>::round(z ? 0.f : O.z / ML.y) |
                          ((uint32_t)ElemOps<E>::round(z ? 0.f : O.w / ML.y) << 16);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + row * D + 4 * q) =
          make_uint2(lo, hi);
    } else {
      const float4 Ow = dead ? make_float4(0.f, 0.f, 0.f, 0.f) : O;
      const float2 MLw = make_float2(ML.x, dead ? -1.f : ML.y);
      if constexpr (CL) {
        using P = ClusterPartial<D, NT8>;
        *reinterpret_cast<float4*>(ring + P::kOutOffset + (g * D + 4 * q) * 4) = Ow;
        if (q == 0) reinterpret_cast<float2*>(ring + P::kMlOffset)[g] = MLw;
      }
      const size_t slot = row * a.max_shards + s;
      if (!PGD_IN(slot, (size_t)a.batch * a.T * a.Hq * a.max_shards, a.err)) continue;
      *reinterpret_cast<float4*>(a.ws_acc + slot * D + 4 * q) = Ow;
      if (q == 0) a.ws_ml[slot] = MLw;
    }
  }
  if constexpr (!CL) {
    if (a.split) merge_if_last<D, E>(a, r, b, h, ring, kWarps * 32);
  }
}

// %cluster_ctarank / %cluster_nctarank, the cluster-wide barrier (every
// thread of every CTA of the cluster; the release / acquire pair orders the
// partials written before it with the reads after it) and loads from another
// CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_u32(local)), "r"(rank));
  return remote;
}
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// The cluster merge: every thread of the cluster's CTAs arrives here once the
// body has returned (on any path); after the barrier each CTA merges its
// slice of the group's (row, 4 dims) items from all the cluster's partials
// in ascending shard (= cluster rank) order with merge_group's arithmetic
// (max, then c_s = 2^(m_s - M) with fused multiply-adds), so the bits equal
// the workspace merge's; a second barrier keeps every CTA's shared memory
// alive until the last read.
template <int D, int NT8, class E>
__device__ __forceinline__ void cluster_merge(const SplitArgs& a) {
  using P = ClusterPartial<D, NT8>;
  constexpr int kQuads = D / 4;
  __syncwarp();
  cluster_sync_all();
  const uint32_t S = cluster_size(), rank = cluster_rank();
  const int h = blockIdx.y, b = blockIdx.z;
  const int R = a.T * a.G, total = R * kQuads;
  const int per = (total + (int)S - 1) / (int)S;
  const int e_end = min(total, ((int)rank + 1) * per);
  uint8_t* base = ring_base();
  for (int e = (int)rank * per + (int)threadIdx.x; e < e_end; e += (int)blockDim.x) {
    const int g = e / kQuads, q = e % kQuads;
    const float2* ml_local = reinterpret_cast<const float2*>(base + P::kMlOffset) + g;
    const float* o_local = reinterpret_cast<const float*>(base + P::kOutOffset) + g * D + 4 * q;
    float M = -INFINITY;
    bool z = false;
    for (uint32_t j = 0; j < S; ++j) {
      const float2 v = ld_dsmem_f2(dsmem_addr(ml_local, j));
      z |= v.y < 0.f;  // a shard saw a bad page or gave up waiting
      M = fmaxf(M, v.x);
    }
    z |= M == -INFINITY;  // no shard holds a position of this row
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (uint32_t j = 0; !z && j < S; ++j) {
      const float2 v = ld_dsmem_f2(dsmem_addr(ml_local, j));
      const float4 x = ld_dsmem_f4(dsmem_addr(o_local, j));
      const float c = fast_exp2(v.x - M);
      L = __fmaf_rn(c, v.y, L);
      o.x = __fmaf_rn(c, x.x, o.x);
      o.y = __fmaf_rn(c, x.y, o.y);
      o.z = __fmaf_rn(c, x.z, o.z);
      o.w = __fmaf_rn(c, x.w, o.w);
    }
    z |= L == 0.f;
    const uint32_t lo = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o.x, L), z ? 0.f : __fdiv_rn(o.y, L));
    const uint32_t hi = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o.z, L), z ? 0.f : __fdiv_rn(o.w, L));
    const size_t row = group_row(b, h, g, a.T, a.G, a.Hq);
    if (PGD_IN(row, (size_t)a.batch * a.T * a.Hq, a.err)) {
      uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + row * D + 4 * q);
      dst[0] = lo;
      dst[1] = hi;
    }
  }
  cluster_sync_all();
}

// The split kernel with the deep ring.  Its launch bounds name no CTA count:
// the register allocation it gets that way (128 at D = 128 with one n8 tile,
// 166 with two) leaves two CTAs per SM; naming one CTA per SM instead gave
// the two-tile kernel 205 registers, one CTA per SM and a 20 % slower T = 2
// long step.
template <int D, int NT8, class E>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads)
    split_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
  split_mma_body<D, NT8, E, false>(tmap_k, tmap_v, a);
}

// The split kernel of cluster plans (grid (S, Hkv, B), clusters of the S
// shards of one (KV head, sequence)): the merge goes through distributed
// shared memory instead of the workspace and a ticket.
template <int D, int NT8, class E>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads)
    split_mma_kernel_cluster(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
  split_mma_body<D, NT8, E, false, true>(tmap_k, tmap_v, a);
  cluster_merge<D, NT8, E>(a);
}

// The split kernel with the shallow ring: registers capped for 3 CTAs per SM.
template <int D, int NT8, class E>
__global__ void __launch_bounds__(MmaCfg<D, true>::kThreads, 3)
    split_mma_kernel_shallow(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
  split_mma_body<D, NT8, E, true>(tmap_k, tmap_v, a);
}

}  // namespace pgd
