// Split decode-attention kernel, tensor-core variant.
//
// One CTA owns (shard s, KV head h, sequence b): a producer warp streams the
// shard's K and V rows of head h through a shared-memory ring with TMA boxes,
// and every K/V row read serves all G query heads of the group
// (BackendStack21/mlx-runner pull request 3, commit "GQA-shared split
// attention").  The products run on the tensor cores with mma.sync.m16n8k16
// (16-bit inputs, fp32 accumulation), tokens on the 16-row M side and the
// group's query rows on the N side (one n8 tile, or two for up to 16 rows):
//   scores^T [16 tok x 8 rows] = K [16 tok x D] . Q^T [D x 8 rows]
//   out^T    [D x 8 rows]     += V^T [D x 16 tok] . P^T [16 tok x 8 rows]
// Each of the four consumer warps takes 16 positions of every 64-position
// stage; a shard's partial (running max, sum, fp32 accumulator; apache/tvm
// pull request 20426, sharded-nest commit) is the warps' states folded in
// fixed order.  The score fragment is transposed into the P^T operand with movmatrix; P is
// split into a 16-bit head and a 16-bit remainder (two mma per tile), so the
// weights keep about 22 (fp16) / 16 (bf16) bits.
//
// A stage's K (and V) tile is 64 tokens made of pieces of box_t = min(page,
// 64) rows, one TMA box each, every piece laid out [D/64][box_t rows][64
// dims] with the 128-byte TMA swizzle (16-byte chunk c of token row t lives
// at chunk c ^ (t % 8)), so every ldmatrix of 8 token rows touches 8
// distinct bank groups (swz_offset).
#pragma once

#include "split_simt.cuh"  // SplitArgs, zero_group_rows, append_new_rows, merge_if_last

namespace pgd {

// kShallow: the ring of plans made of many short shards, 2 stages (4 at
// D = 64) instead of 3 (6), so that 3 CTAs fit per SM and more CTAs' first
// round trips overlap.
template <int D, bool kShallow = false>
struct MmaCfg {
  static constexpr int kWarps = 4;  // consumer warps, 16 positions of each stage apiece
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kStages = (D == 64) ? (kShallow ? 4 : 6) : (kShallow ? 2 : 3);
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kRingBytes + 1024;
};

// Shared memory a cluster plan's CTA receives the group's partials in
// (after the ring): for each of the S CTAs of the cluster, its values of
// this CTA's slice of the (row, 4 dims) items, then its (m, l) per row.
struct ClusterRecv {
  int per;         // items of a slice: ceil(rows * D / 4 / S)
  int acc_bytes;   // S * per float4
  int bytes;       // + S * rows float2
  __host__ __device__ static ClusterRecv of(int rows, int D, int S) {
    ClusterRecv c;
    c.per = (rows * (D / 4) + S - 1) / S;
    c.acc_bytes = S * c.per * 16;
    c.bytes = c.acc_bytes + S * rows * 8;
    return c;
  }
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

// One consumer warp's 16 positions [tok0, tok0 + 16) of a staged tile:
// scores^T = K . Q^T, the per-column causal / window mask, the online
// softmax update and out^T += V^T . P^T.  kt points at the stage's K tile in
// pieces of 2^ps rows (swz_offset), the warp's 16 rows at 16 * warp (V
// follows at kTile * D * 2 bytes); [lo, hi) is the union of the columns'
// ranges clipped to the shard, and the block must overlap it.
template <int D, int NT8, class E>
__device__ __forceinline__ void mma_block(uint8_t* kt, int warp, int lane, int tok0, int lo,
                                          int hi, const int (&col_lo)[NT8][2],
                                          const int (&col_hi)[NT8][2],
                                          const uint32_t (&qf)[NT8][D / 16][2], float scale_log2,
                                          float (&acc)[D / 16][NT8][4], float (&m_run)[NT8][2],
                                          float (&l_part)[NT8][2], int ps) {
  constexpr int kTileBytes = kTile * D * 2;
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
  // scores^T = K . Q^T
  float sc[NT8][4];
#pragma unroll
  for (int j = 0; j < NT8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t af[4];
    ldmatrix_x4(af, kbase + swz_offset<D>(k_tok, ks * 16 + k_dof, ps));
#pragma unroll
    for (int j = 0; j < NT8; ++j) ElemOps<E>::mma(sc[j], af, qf[j][ks][0], qf[j][ks][1]);
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
    // P^T operand: 16-bit head and 16-bit remainder, transposed by movmatrix
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
    ldmatrix_x4_trans(af, vbase + swz_offset<D>(v_tok, mi * 16 + v_dof, ps));
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
      ElemOps<E>::mma(acc[mi][j], af, pb_hi[j][0], pb_hi[j][1]);
      ElemOps<E>::mma(acc[mi][j], af, pb_lo[j][0], pb_lo[j][1]);
    }
  }
}

__device__ __forceinline__ uint8_t* ring_base() {
  extern __shared__ uint8_t smem_raw[];
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                    ~uintptr_t(1023));
}

// %cluster_ctarank / %cluster_nctarank, the split cluster barrier (arrive
// right after the receive barrier's initialisation, wait only before the
// first access to another CTA's shared memory), stores to another CTA's
// shared memory and the remote release-arrive on its mbarrier.
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
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}
__device__ __forceinline__ void st_dsmem_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_dsmem_f2(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y)
               : "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded like mbar_wait, with cluster-scope acquire, but after about four
// seconds: twice the pipeline's bound.  A partner CTA reaches the exchange at
// most one pipeline give-up (about two seconds) after its own start, so a CTA
// that arrives first (one with an empty shard does at once) still waits for
// it, and no CTA exits while a partner may still store into its receive
// buffer.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (global_timer_ns() - t0 > 4000000000ull) return false;
  }
  return true;
}

// The cluster merge of a cluster plan (the S shards of one (KV head,
// sequence) form one thread-block cluster; cluster rank = shard index).
// Every CTA owns a slice of the group's (row, 4 dims) items: item
// e = row * D / 4 + quad belongs to CTA e / per.  Each CTA pushes its folded
// value of every item (cluster_push) and its (m, l) of every row
// (cluster_push_ml) into the owners' receive buffers in distributed shared
// memory; cluster_finish then has thread 0 arrive on every owner's receive
// barrier with release semantics, waits (bounded, acquire) for this CTA's S
// arrivals and merges its slice in ascending shard order with the workspace
// merge's arithmetic (max, then c_s = 2^(m_s - M) with fused multiply-adds),
// so both merges give the same bits.  Nothing is read from another CTA's
// shared memory, so no CTA waits for another to finish reading before it
// exits.  The receive buffer sits after the ring, so a CTA still streaming
// can already receive.
struct ClusterXchg {
  uint32_t recv_acc, recv_ml;  // this CTA's receive buffer (shared::cta addresses)
  int S, rank, R;
  ClusterRecv cr;
  __device__ ClusterXchg() {}
  __device__ ClusterXchg(uint8_t* recv, int rows, int D) {
    S = (int)cluster_size();
    rank = (int)cluster_rank();
    R = rows;
    cr = ClusterRecv::of(rows, D, S);
    recv_acc = smem_u32(recv);
    recv_ml = recv_acc + cr.acc_bytes;
  }
  __device__ void push(int e, float4 v) const {
    const int o = e / cr.per;
    const uint32_t at = recv_acc + (uint32_t)((rank * cr.per + (e - o * cr.per)) * 16);
    st_dsmem_f4(dsmem_addr(at, (uint32_t)o), v);
  }
  __device__ void push_ml(int r, float2 v) const {
    const uint32_t at = recv_ml + (uint32_t)((rank * R + r) * 8);
    for (int o = 0; o < S; ++o) st_dsmem_f2(dsmem_addr(at, (uint32_t)o), v);
  }
};

template <int D, class E>
__device__ __forceinline__ void cluster_finish(const SplitArgs& a, const ClusterXchg& x, int b,
                                               int h, uint32_t recv_bar, uint8_t* recv,
                                               int nthreads) {
  named_barrier_sync(1, nthreads);  // every consumer's stores are issued
  // thread o announces this CTA's partial to owner o: a cluster-scope release
  // fence (it orders the stores the barrier above ordered before it) and a
  // relaxed arrival on the owner's receive barrier
  if ((int)threadIdx.x < x.S) {
    fence_acq_rel_cluster();
    mbar_arrive_remote_relaxed(dsmem_addr(recv_bar, threadIdx.x));
  }
  // this CTA's slice: wait for the S partials, merge in shard order
  __shared__ int recv_ok_s;
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait_cluster(recv_bar, 0);
    if (!ok) raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
    recv_ok_s = ok ? 1 : 0;
  }
  named_barrier_sync(1, nthreads);
  // (every thread acquires as well; the phase is complete, so this returns)
  if (recv_ok_s) mbar_wait_cluster(recv_bar, 0);
  const int R = x.R, S = x.S, per = x.cr.per;
  const float4* racc = reinterpret_cast<const float4*>(recv);
  const float2* rml = reinterpret_cast<const float2*>(recv + x.cr.acc_bytes);
  const int total = R * (D / 4);
  const int e_end = min(total, (x.rank + 1) * per);
  for (int e = x.rank * per + (int)threadIdx.x; e < e_end; e += nthreads) {
    const int r = e / (D / 4), quad = e % (D / 4);
    const int slot = e - x.rank * per;
    float M = -INFINITY;
    bool z = !recv_ok_s;
    for (int j = 0; j < S; ++j) {
      const float2 v = rml[j * R + r];
      z |= v.y < 0.f;  // a shard saw a bad page or gave up waiting
      M = fmaxf(M, v.x);
    }
    z |= M == -INFINITY;  // no shard holds a position of this row
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; !z && j < S; ++j) {
      const float2 v = rml[j * R + r];
      const float4 xv = racc[j * per + slot];
      const float c = fast_exp2(v.x - M);
      L = __fmaf_rn(c, v.y, L);
      o.x = __fmaf_rn(c, xv.x, o.x);
      o.y = __fmaf_rn(c, xv.y, o.y);
      o.z = __fmaf_rn(c, xv.z, o.z);
      o.w = __fmaf_rn(c, xv.w, o.w);
    }
    z |= L == 0.f;
    const uint32_t lo = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o.x, L), z ? 0.f : __fdiv_rn(o.y, L));
    const uint32_t hi = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o.z, L), z ? 0.f : __fdiv_rn(o.w, L));
    const size_t row = group_row(b, h, r, a.T, a.G, a.Hq);
    if (PGD_IN(row, (size_t)a.batch * a.T * a.Hq, a.err))
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + row * D + 4 * quad) =
          make_uint2(lo, hi);
  }
}

// The split kernel's body.  SH: the shallow ring.  CL: a cluster plan (one
// cluster per (KV head, sequence), one CTA per shard, cluster rank = shard),
// merged through distributed shared memory (ClusterXchg, cluster_finish);
// other split plans write their partial to the workspace and the group's last
// CTA merges (merge_if_last; kOneTrip > 0: groups of at most that many shards
// in one L2 round trip, merge_group).
template <int D, int NT8, class E, bool SH, bool CL = false, int kOneTrip = 0>
__device__ __forceinline__ void split_mma_body(const CUtensorMap& tmap_k,
                                               const CUtensorMap& tmap_v, const SplitArgs& a) {
  using C = MmaCfg<D, SH>;
  constexpr int KS = D / 16;  // k-steps of q.k
  constexpr int kWarps = C::kWarps;
  constexpr int GP = 8 * NT8;  // padded query rows of the group

  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t recv_bar;
  __shared__ int32_t coord_s[kMaxPieces];
  __shared__ float2 ml_s[kWarps][GP];
  __shared__ float cw_s[kWarps][GP];  // each warp's weight per row
  __shared__ float2 row_s[GP];        // (M, L) per row
  __shared__ int32_t bad_s;
  __shared__ volatile int32_t abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = ring_base();

  // Before the dependency wait (nothing here touches global memory): the
  // pipeline's barriers, the tensor maps' prefetch and, for a cluster plan,
  // the receive barrier and this CTA's arrival at the cluster barrier that
  // the exchange waits on.
  if (threadIdx.x == kWarps * 32) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(smem_u32(&full_bar[st]), 1);
      mbar_init(smem_u32(&empty_bar[st]), kWarps);
    }
    if constexpr (CL) mbar_init(smem_u32(&recv_bar), cluster_size());
    fence_mbar_init();
    abort_s = 0;
    bad_s = 0;
  }
  __syncthreads();
  if constexpr (CL) cluster_arrive_relaxed();
  // launched as a programmatic dependent of the preceding kernel: nothing is
  // read or written before that kernel has completed
  grid_dependency_wait();
  // a kernel launched after this one (the next step) may be scheduled now;
  // it waits the same way before touching memory
  grid_launch_dependents();
  // grid order: head fastest for plans of several waves (the Hkv CTAs of one
  // (sequence, shard) start together and read the rows of the same positions,
  // adjacent in the pool, side by side), shard fastest for one-wave plans
  // (a group's shards run on neighbouring SMs, a cluster plan's in one
  // cluster)
  const int h = a.head_fastest ? blockIdx.x : blockIdx.y;
  const int s = a.head_fastest ? blockIdx.y : blockIdx.x;
  const int b = blockIdx.z;
  const int capacity = a.max_pages * a.page_size;
  const int box_t = a.box_tokens;
  // The producer reads the page ids of the shard's first 32 pieces together
  // with the length, under the guess that the sequence is as long as the
  // plan's bound: a shard's first position depends on the length only
  // through a window's start, so without a window the guess always holds
  // (with one, when the sequence is that long); otherwise they are read again.
  int spec_lo = -1, spec_phys = -1;
  if (warp == kWarps) {
    const SeqRange g =
        seq_range(a.len_hint, a.window, capacity, a.chunk, a.max_shards, a.T, a.balanced);
    if (g.status == 0 && s < g.nshards) {
      spec_lo = g.base + s * g.chunk;
      const int ptok = spec_lo + lane * box_t;
      const size_t pi = (size_t)b * a.max_pages + (ptok >> a.page_shift);
      if (ptok < capacity && PGD_IN(pi, (size_t)a.batch * a.max_pages, a.err))
        spec_phys = ld_global_s32(a.page_table + pi);
    }
  }
  // (ld_global_s32 keeps the two loads in this order, both in flight at once)
  const SeqRange r =
      seq_range(ld_global_s32(a.seq_lens + b), a.window, capacity, a.chunk, a.max_shards, a.T,
                a.balanced);
  const int R = a.T * a.G;  // query rows of the group: r = t * G + g
  const int gid = lane >> 2, tig = lane & 3;

  if (r.status != 0 || s >= r.nshards) {
    if (s == 0 && r.status != 0 && threadIdx.x == 0) raise_error(a.err, r.status);
    if constexpr (CL) {
      // an empty partial (no position of any row) still takes part in the
      // cluster's exchange; the merge zeroes rows that no shard holds
      if (warp < kWarps) {
        uint8_t* recv = ring + C::kRingBytes;
        const ClusterXchg x(recv, R, D);
        cluster_wait();  // every CTA of the cluster has initialised its barriers
        for (int e = threadIdx.x; e < R * (D / 4); e += kWarps * 32)
          x.push(e, make_float4(0.f, 0.f, 0.f, 0.f));
        for (int g = threadIdx.x; g < R; g += kWarps * 32)
          x.push_ml(g, make_float2(-INFINITY, 0.f));
        cluster_finish<D, E>(a, x, b, h, smem_u32(&recv_bar), recv, kWarps * 32);
      }
    } else if (s == 0) {
      zero_group_rows<D, 8 * NT8>(a, b, h);
    }
    return;
  }

  const int shard_lo = r.base + s * r.chunk;
  const int lo = max(r.start, shard_lo);
  const int hi = min(r.end, shard_lo + r.chunk);
  const int n_tiles = (hi - shard_lo + kTile - 1) / kTile;
  const int pieces_per_tile = kTile / box_t;
  const int n_pieces = n_tiles * pieces_per_tile;

  // Producer: the boxes of a stage are issued by several lanes at once
  // (lane j its j-th box) after lane 0 has armed the stage's full barrier
  // with its bytes; every box is read once, so it enters L2 with the
  // evict-first policy.  The first kStages stages go out at once, every later
  // one as soon as the consumers have released its slot.
  const uint32_t box_bytes = box_t * D * 2;  // one piece: box_t rows, all D dims
  const int per_piece = box_t < kTile ? 1 : D / 64;
  const int nbox = pieces_per_tile * per_piece * 2;
  const int pool_rows = a.num_pages * a.page_size;
  auto issue_stage = [&](int i, uint64_t policy) {
    const int st = i % C::kStages;
    if (lane == 0)
      // (stall_tx, a test's hook, is 0: the barrier expects the stage's bytes)
      mbar_arrive_expect_tx(smem_u32(&full_bar[st]), C::kStageBytes + (i == 0 ? a.stall_tx : 0));
    __syncwarp();
    const uint32_t fb = smem_u32(&full_bar[st]);
    const uint32_t kdst = smem_u32(ring + st * C::kStageBytes);
    const uint32_t vdst = kdst + C::kTileBytes;
    for (int jb = lane; jb < nbox; jb += 32) {
      const int is_v = jb & 1;
      const int pc = (jb >> 1) / per_piece, dc = (jb >> 1) % per_piece;
      int coord = coord_s[i * pieces_per_tile + pc];
      // (checked build) a box must lie inside the pool or start at its end,
      // where TMA fills zeros
      if (!PGD_IN(coord == pool_rows ? 0 : (int64_t)coord + box_t - 1, pool_rows, a.err))
        coord = pool_rows;
      const CUtensorMap* map = is_v ? &tmap_v : &tmap_k;
      const uint32_t dst = is_v ? vdst : kdst;
      if (box_t < kTile)  // one box holds the piece's D dims
        tma_load_4d_hint(dst + pc * box_bytes, map, 0, coord, h, 0, fb, policy);
      else  // 64-row pieces: one box per 64-dim chunk
        tma_load_4d_hint(dst + dc * (kTile * 128), map, 0, coord, h, dc, fb, policy);
    }
  };
  if (warp == kWarps) {
    // physical coordinates of every box of the shard
    int any_bad = 0;
    const int oob = pool_rows;  // past the pool: TMA writes zeros
#pragma unroll 4
    for (int i = lane; i < n_pieces; i += 32) {
      const int ptok = shard_lo + i * box_t;
      int coord = oob;
      if (ptok < hi && ptok + box_t > lo) {
        int phys;
        if (i == lane && shard_lo == spec_lo) {
          phys = spec_phys;
        } else {
          const size_t pi = (size_t)b * a.max_pages + (ptok >> a.page_shift);
          phys = PGD_IN(pi, (size_t)a.batch * a.max_pages, a.err) ? a.page_table[pi] : -1;
        }
        if (phys < 0 || phys >= a.num_pages) {
          any_bad = 1;
        } else {
          coord = phys * a.page_size + (ptok & (a.page_size - 1));
        }
      }
      coord_s[i] = coord;
    }
    const bool bad = __any_sync(0xffffffffu, any_bad) != 0;
    if (bad) {
      // no copy is issued; the consumers' first wait completes on a plain
      // arrival and they find the flag
      if (lane == 0) {
        bad_s = 1;
        raise_error(a.err, DECODE_ATTN_DEV_BAD_PAGE);
        mbar_arrive(smem_u32(&full_bar[0]));
      }
    } else {
      if (a.k_new != nullptr && r.end - a.T < shard_lo + r.chunk && r.end > shard_lo)
        append_new_rows<D>(a, r, b, h, shard_lo, lane);
      const uint64_t policy = l2_evict_first_policy();
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        if (i >= C::kStages) {
          const int st = i % C::kStages;
          int go = 1;
          if (lane == 0) {
            if (!mbar_wait(smem_u32(&empty_bar[st]), ((i / C::kStages) & 1) ^ 1)) {
              abort_s = 1;
              raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
              go = 0;
            }
            if (abort_s) go = 0;
          }
          if (!__shfl_sync(0xffffffffu, go, 0)) break;
        }
        issue_stage(i, policy);
        issued = i + 1;
      }
      // drain this CTA's copies in flight before the warp exits
      if (lane == 0)
        for (int i = max(0, issued - C::kStages); i < issued; ++i)
          mbar_wait(smem_u32(&full_bar[i % C::kStages]), (i / C::kStages) & 1);
    }
    return;
  }

  // ------------------------------------------------ consumers' set-up
  // Q^T operand fragments, held for the whole shard (loaded while the
  // producer reads the page ids)
  uint32_t qf[NT8][KS][2];
  float acc[KS][NT8][4];
  int col_lo[NT8][2], col_hi[NT8][2];
  float m_run[NT8][2], l_part[NT8][2];
  if (warp < kWarps) {
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
      const int rr = 8 * j + gid;
      size_t qr = group_row(b, h, rr < R ? rr : 0, a.T, a.G, a.Hq);
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
    // attended range of each of this lane's score columns (query rows
    // 8j + 2*tig + e): causal up to the row's own position, window from there
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int rr = 8 * j + 2 * tig + e;
        const int t = rr < R ? rr / a.G : a.T - 1;
        col_hi[j][e] = r.end - a.T + t + 1;
        col_lo[j][e] = a.window > 0 ? max(0, col_hi[j][e] - a.window) : 0;
        m_run[j][e] = -INFINITY;
        l_part[j][e] = 0.f;
      }
#pragma unroll
    for (int mi = 0; mi < KS; ++mi)
#pragma unroll
      for (int j = 0; j < NT8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mi][j][e] = 0.f;
  }
  // ------------------------------------------------------------ consumers
  const int piece_shift = __ffs(box_t) - 1;  // a stage is pieces of box_t rows
  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % C::kStages;
    if (!mbar_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1)) {
      abort_s = 1;
      raise_error(a.err, DECODE_ATTN_DEV_TIMEOUT);
      break;
    }
    if (bad_s || abort_s) break;
    const int tok0 = shard_lo + i * kTile + 16 * warp;  // this warp's 16 positions
    if (tok0 + 16 > lo && tok0 < hi)
      mma_block<D, NT8, E>(ring + st * C::kStageBytes, warp, lane, tok0, lo, hi, col_lo, col_hi,
                           qf, a.scale_log2, acc, m_run, l_part, piece_shift);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
  }

  // ---- fold the consumer warps in fixed order (deterministic) -----------
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
  const bool dead = bad_s != 0 || abort_s != 0;
  uint8_t* recv = ring + C::kRingBytes;  // a cluster plan's receive buffer
  ClusterXchg x;
  if constexpr (CL) {
    x = ClusterXchg(recv, R, D);
    cluster_wait();  // every CTA of the cluster has initialised its barriers
  }
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
      const float4 v =
          *reinterpret_cast<const float4*>(acc_s + (w * GP + g) * kRowStride + 4 * q);
      O.x += c * v.x;
      O.y += c * v.y;
      O.z += c * v.z;
      O.w += c * v.w;
    }
    const size_t row = group_row(b, h, g, a.T, a.G, a.Hq);
    if (!a.split) {
      if (!PGD_IN(row, (size_t)a.batch * a.T * a.Hq, a.err)) continue;
      const bool z = dead || ML.y == 0.f;
      const uint32_t lo = (uint32_t)ElemOps<E>::round(z ? 0.f : O.x / ML.y) |
                          ((uint32_t)ElemOps<E>::round(z ? 0.f : O.y / ML.y) << 16);
      const uint32_t hi = (uint32_t)ElemOps<E>::round(z ? 0.f : O.z / ML.y) |
                          ((uint32_t)ElemOps<E>::round(z ? 0.f : O.w / ML.y) << 16);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + row * D + 4 * q) =
          make_uint2(lo, hi);
      continue;
    }
    // split: this shard's partial (m, l, acc) to the workspace slots (read by
    // the group's merge, or later by decode_attn_combine; l = -1 marks a dead
    // shard) and, for a cluster plan, to the item's owner in the cluster
    const float4 Ow = dead ? make_float4(0.f, 0.f, 0.f, 0.f) : O;
    const float2 MLw = make_float2(ML.x, dead ? -1.f : ML.y);
    if constexpr (CL) {
      x.push(e, Ow);
      if (q == 0) x.push_ml(g, MLw);
    }
    const size_t slot = row * a.max_shards + s;
    if (!PGD_IN(slot, (size_t)a.batch * a.T * a.Hq * a.max_shards, a.err)) continue;
    *reinterpret_cast<float4*>(a.ws_acc + slot * D + 4 * q) = Ow;
    if (q == 0) a.ws_ml[slot] = MLw;
  }
  if (!a.split) return;
  if constexpr (CL) {
    cluster_finish<D, E>(a, x, b, h, smem_u32(&recv_bar), recv, kWarps * 32);
  } else {
    merge_if_last<D, E, kOneTrip>(a, r, b, h, ring, kWarps * 32);
  }
}

// The split kernel with the deep ring, for split plans: the last CTA of a
// group of up to 16 shards merges them in one L2 round trip.  Its launch
// bounds name no CTA count: the register allocation it gets that way leaves
// two CTAs per SM at D <= 128.
template <int D, int NT8, class E>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads)
    split_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
  split_mma_body<D, NT8, E, false, false, 16>(tmap_k, tmap_v, a);
}

// The deep-ring kernel of single-pass plans: the same body without the
// one-round-trip merge (a single-pass plan never merges).  Kept apart
// because the short single-CTA steps are sensitive to the code they run:
// with the merge form compiled in, or with the merge code compiled out,
// they measured 0.5-0.8 us slower on GB300.
template <int D, int NT8, class E>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads)
    split_mma_kernel_single(const __grid_constant__ CUtensorMap tmap_k,
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
}

// The split kernel with the shallow ring: registers capped for 3 CTAs per SM.
template <int D, int NT8, class E>
__global__ void __launch_bounds__(MmaCfg<D, true>::kThreads, 3)
    split_mma_kernel_shallow(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
  split_mma_body<D, NT8, E, true>(tmap_k, tmap_v, a);
}

}  // namespace pgd
