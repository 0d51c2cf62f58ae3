// Ordered combine of shard partials (apache/tvm pull request 20426: per-shard
// online-softmax states merged after the sharded pass; BackendStack21/
// mlx-runner pull request 3: the combine merges the partials in the same
// order every time, so results are bit-identical run to run).
//
// For one (sequence b, KV head h) group, each of its G query-head rows is
// merged strictly in ascending shard index:
//   M = max_s m_s,  c_s = 2^(m_s - M),  L = sum_s c_s l_s,
//   out = fp16_rn(sum_s c_s acc_s / L)
// with explicit fused multiply-adds, so the bits depend only on the inputs
// and the shard plan.  merge_group() is the one implementation: the split
// kernel's last CTA of a group runs it in its epilogue, and the standalone
// combine kernel (decode_attn_combine) runs it for every group, giving the
// same bits.
#pragma once

#include "device_common.cuh"
#include "elem.cuh"

namespace pgd {

struct CombineArgs {
  const int32_t* seq_lens;
  const float* ws_acc;   // [B*T*Hq*S_max][D]
  const float2* ws_ml;   // [B*T*Hq*S_max]
  void* out;             // [B][T][Hq][D] 16-bit elements
  int32_t* err;          // nullable; the checked build's bounds errors
  int32_t B, Hq, G, T, capacity, window, chunk, max_shards, balanced;
};

// Bounds of the partial slots (the checked build).
__device__ __forceinline__ size_t slot_bound(const CombineArgs& a) {
  return (size_t)a.B * a.T * a.Hq * a.max_shards;
}

// Output row of the group's r-th query row (r = t * G + g): query t of
// sequence b, query head h * G + g.
__device__ __forceinline__ size_t group_row(int b, int h, int r, int T, int G, int Hq) {
  return ((size_t)b * T + r / G) * Hq + (size_t)h * G + r % G;
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kShardBlock = 256;   // (m, l) entries of each row staged per pass
constexpr int kMaxMergeRows = 16;  // rows of one group (T * G <= 16)

// Shared memory merge_group needs when it stages `cap` (m, l) entries per
// row: the staged pairs plus a per-row max and flag.
__host__ __device__ constexpr int merge_smem_bytes(int rows, int cap = kShardBlock) {
  return rows * cap * 8 + kMaxMergeRows * 8;
}

// Partial slots of the grid schedule: row-major over (row, shard).
struct GridSlots {
  int b, h, T, G, Hq, max_shards;
  __device__ size_t operator()(int r, int s) const {
    return group_row(b, h, r, T, G, Hq) * (size_t)max_shards + s;
  }
};

// U consecutive shards [s, s + U) of one output item (row g, dims 4*quad ..
// 4*quad + 3): the U accumulator loads (and (m, l) reads) first, then the
// fused multiply-adds in shard order.
template <int D, int U, class SlotOf>
__device__ __forceinline__ void merge_batch(const CombineArgs& a, int g, int quad, int s, float M,
                                            bool staged, const float2* ml_s, int cap,
                                            SlotOf slot_of, float4& o, float& L) {
  float4 x[U];
  float2 v[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const size_t slot = slot_of(g, s + u);
    if (!PGD_IN(slot, slot_bound(a), a.err)) {
      x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      v[u] = make_float2(-INFINITY, 0.f);
      continue;
    }
    x[u] = __ldcg(reinterpret_cast<const float4*>(a.ws_acc + slot * D) + quad);
    v[u] = staged ? ml_s[g * cap + s + u] : __ldcg(a.ws_ml + slot);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const float c = fast_exp2(v[u].x - M);
    L = __fmaf_rn(c, v[u].y, L);
    o.x = __fmaf_rn(c, x[u].x, o.x);
    o.y = __fmaf_rn(c, x[u].y, o.y);
    o.z = __fmaf_rn(c, x[u].z, o.z);
    o.w = __fmaf_rn(c, x[u].w, o.w);
  }
}

// Merges the S shard partials of group (b, h) (its T*G query rows) into
// out, in ascending shard order, using threads [0, nthreads) (tid = this
// thread's index among them) and `smem` (merge_smem_bytes(rows, cap)
// bytes, 16-byte aligned; up to `cap` (m, l) pairs per row are staged there,
// more are read from global memory).  `sync` is a barrier over exactly those
// threads; slot_of(r, s) locates the partial of row r, shard s.  dead forces
// zero rows (an invalid range).  kOneTrip > 0: a group of at most kOneTrip
// shards with one output item per thread skips the staging and loads
// everything at once (below); the bits are the same either way.
template <int D, class E, int kOneTrip = 0, class Sync, class SlotOf>
__device__ __forceinline__ void merge_group(const CombineArgs& a, int b, int h, int S, bool dead,
                                            int tid, int nthreads, uint8_t* smem, int cap,
                                            Sync sync, SlotOf slot_of) {
  constexpr int kQuads = D / 4;
  const int G = a.T * a.G;  // rows of the group
  if constexpr (kOneTrip > 0) if (G * kQuads <= nthreads && S >= 1 && S <= kOneTrip) {
    // One L2 round trip for groups of at most kOneTrip shards and one item
    // per thread: every (m, l) and accumulator of the item is loaded at once
    // (shard indices clamped to the group's last, so no load sits behind a
    // branch), the row's maximum is taken in registers, then the same
    // multiply-adds in the same shard order as below: the same bits.
    const int e = tid;
    if (e >= G * kQuads) return;
    const int g = e / kQuads, quad = e % kQuads;
    float4 x[kOneTrip];
    float2 v[kOneTrip];
#pragma unroll
    for (int u = 0; u < kOneTrip; ++u) {
      const size_t slot = slot_of(g, min(u, S - 1));
      const bool in = PGD_IN(slot, slot_bound(a), a.err);
      x[u] = in ? __ldcg(reinterpret_cast<const float4*>(a.ws_acc + slot * D) + quad)
                : make_float4(0.f, 0.f, 0.f, 0.f);
      v[u] = in ? __ldcg(a.ws_ml + slot) : make_float2(-INFINITY, 0.f);
    }
    float M = -INFINITY;
    bool zero = dead;
#pragma unroll
    for (int u = 0; u < kOneTrip; ++u)
      if (u < S) {
        zero |= v[u].y < 0.f;  // a shard saw a bad page or gave up waiting
        M = fmaxf(M, v[u].x);
      }
    zero |= M == -INFINITY;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
#pragma unroll
    for (int u = 0; u < kOneTrip; ++u)
      if (!zero && u < S) {
        const float c = fast_exp2(v[u].x - M);
        L = __fmaf_rn(c, v[u].y, L);
        o.x = __fmaf_rn(c, x[u].x, o.x);
        o.y = __fmaf_rn(c, x[u].y, o.y);
        o.z = __fmaf_rn(c, x[u].z, o.z);
        o.w = __fmaf_rn(c, x[u].w, o.w);
      }
    const bool z = zero || L == 0.f;
    const uint32_t lo = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o.x, L), z ? 0.f : __fdiv_rn(o.y, L));
    const uint32_t hi = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o.z, L), z ? 0.f : __fdiv_rn(o.w, L));
    const size_t row = group_row(b, h, g, a.T, a.G, a.Hq);
    if (PGD_IN(row, (size_t)a.B * a.T * a.Hq, a.err)) {
      uint32_t* dst =
          reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + row * D + 4 * quad);
      dst[0] = lo;
      dst[1] = hi;
    }
    return;
  }
  float2* ml_s = reinterpret_cast<float2*>(smem);                // [G][cap]
  float* max_s = reinterpret_cast<float*>(smem + G * cap * 8);   // [G]
  int* zero_s = reinterpret_cast<int*>(max_s + kMaxMergeRows);   // [G]
  const bool staged = S <= cap;
  const int block = cap > 0 ? cap : 1;

  // per-row maximum and bad-partial flag, from (m, l) staged block by block
  sync();
  if (tid < G) {
    max_s[tid] = -INFINITY;
    zero_s[tid] = (dead || S == 0) ? 1 : 0;
  }
  for (int s0 = 0; s0 < S; s0 += block) {
    const int n = min(block, S - s0);
    sync();
    if (cap > 0)
      for (int e = tid; e < G * n; e += nthreads) {
        const int g = e / n, j = e % n;
        const size_t slot = slot_of(g, s0 + j);
        ml_s[g * cap + j] = PGD_IN(slot, slot_bound(a), a.err) ? __ldcg(a.ws_ml + slot)
                                                                : make_float2(-INFINITY, 0.f);
      }
    sync();
    if (tid < G) {
      float M = max_s[tid];
      int z = zero_s[tid];
      for (int j = 0; j < n; ++j) {
        const size_t slot = slot_of(tid, s0 + j);
        const float2 v = cap > 0 ? ml_s[tid * cap + j]
                         : PGD_IN(slot, slot_bound(a), a.err) ? __ldcg(a.ws_ml + slot)
                                                              : make_float2(-INFINITY, 0.f);
        z |= v.y < 0.f ? 1 : 0;  // a shard saw a bad page or gave up waiting
        M = fmaxf(M, v.x);
      }
      max_s[tid] = M;
      zero_s[tid] = z;
    }
  }
  sync();

  const int total = G * kQuads;
  if (total <= nthreads) {
    // at most one output item (row, 4 dims) per thread: its shard loads go
    // out 16 at a time (then 8, then one by one), so a batch of 16 shards
    // costs one L2 round trip
    const int e = tid;
    if (e < total) {
      const int g = e / kQuads, quad = e % kQuads;
      const float M = max_s[g];
      const bool zero = zero_s[g] != 0 || M == -INFINITY;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float L = 0.f;
      int s = 0;
      for (; !zero && s + 16 <= S; s += 16) merge_batch<D, 16>(a, g, quad, s, M, staged, ml_s, cap, slot_of, o, L);
      for (; !zero && s + 8 <= S; s += 8) merge_batch<D, 8>(a, g, quad, s, M, staged, ml_s, cap, slot_of, o, L);
      for (; !zero && s < S; ++s) merge_batch<D, 1>(a, g, quad, s, M, staged, ml_s, cap, slot_of, o, L);
      const bool z = zero || L == 0.f;
      const uint32_t lo = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o.x, L), z ? 0.f : __fdiv_rn(o.y, L));
      const uint32_t hi = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o.z, L), z ? 0.f : __fdiv_rn(o.w, L));
      const size_t row = group_row(b, h, g, a.T, a.G, a.Hq);
      if (PGD_IN(row, (size_t)a.B * a.T * a.Hq, a.err)) {
        uint32_t* dst =
            reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + row * D + 4 * quad);
        dst[0] = lo;
        dst[1] = hi;
      }
    }
    return;
  }
  // two output items (row, 4 dims) per thread and pass, their shard loads
  // issued together so several L2 round trips overlap
  for (int e0 = tid; e0 < total; e0 += 2 * nthreads) {
    int e[2] = {e0, e0 + nthreads};
    const int n_items = e[1] < total ? 2 : 1;
    if (n_items == 1) e[1] = e0;
    float4 o[2];
    float L[2], M[2];
    bool zero[2];
    int gg[2], quad[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      gg[k] = e[k] / kQuads;
      quad[k] = e[k] % kQuads;
      M[k] = max_s[gg[k]];
      // a row with no attended position in any shard (a query before the
      // first cached position) stays zero
      zero[k] = zero_s[gg[k]] != 0 || M[k] == -INFINITY;
      o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      L[k] = 0.f;
    }
    const bool any = !(zero[0] && zero[1]);
    int s = 0;
    for (; any && s + 8 <= S; s += 8) {
      float4 x[2][8];
      float2 v[2][8];
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const size_t slot = slot_of(gg[k], s + u);
          if (!PGD_IN(slot, slot_bound(a), a.err)) {
            x[k][u] = make_float4(0.f, 0.f, 0.f, 0.f);
            v[k][u] = make_float2(-INFINITY, 0.f);
            continue;
          }
          x[k][u] = __ldcg(reinterpret_cast<const float4*>(a.ws_acc + slot * D) + quad[k]);
          v[k][u] = staged ? ml_s[gg[k] * cap + s + u] : __ldcg(a.ws_ml + slot);
        }
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float c = fast_exp2(v[k][u].x - M[k]);
          L[k] = __fmaf_rn(c, v[k][u].y, L[k]);
          o[k].x = __fmaf_rn(c, x[k][u].x, o[k].x);
          o[k].y = __fmaf_rn(c, x[k][u].y, o[k].y);
          o[k].z = __fmaf_rn(c, x[k][u].z, o[k].z);
          o[k].w = __fmaf_rn(c, x[k][u].w, o[k].w);
        }
    }
    for (; any && s < S; ++s) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const size_t slot = slot_of(gg[k], s);
        if (!PGD_IN(slot, slot_bound(a), a.err)) continue;
        const float4 x = __ldcg(reinterpret_cast<const float4*>(a.ws_acc + slot * D) + quad[k]);
        const float2 v = staged ? ml_s[gg[k] * cap + s] : __ldcg(a.ws_ml + slot);
        const float c = fast_exp2(v.x - M[k]);
        L[k] = __fmaf_rn(c, v.y, L[k]);
        o[k].x = __fmaf_rn(c, x.x, o[k].x);
        o[k].y = __fmaf_rn(c, x.y, o[k].y);
        o[k].z = __fmaf_rn(c, x.z, o[k].z);
        o[k].w = __fmaf_rn(c, x.w, o[k].w);
      }
    }
    for (int k = 0; k < n_items; ++k) {
      const bool z = zero[k] || L[k] == 0.f;
      const float l_sum = L[k];
      const uint32_t lo = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o[k].x, l_sum),
                                            z ? 0.f : __fdiv_rn(o[k].y, l_sum));
      const uint32_t hi = ElemOps<E>::pack2(z ? 0.f : __fdiv_rn(o[k].z, l_sum),
                                            z ? 0.f : __fdiv_rn(o[k].w, l_sum));
      const size_t row = group_row(b, h, gg[k], a.T, a.G, a.Hq);
      if (!PGD_IN(row, (size_t)a.B * a.T * a.Hq, a.err)) continue;
      uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + row * D +
                                                  4 * quad[k]);
      dst[0] = lo;
      dst[1] = hi;
    }
  }
}

// Standalone combine: one CTA per (KV head, sequence).  Launched as a
// programmatic dependent of the split kernel: waits (griddepcontrol.wait) for
// the split grid's partials before reading them.
template <int D, class E>
__global__ void __launch_bounds__(512) combine_kernel(const CombineArgs a) {
  extern __shared__ __align__(16) uint8_t merge_smem[];
  const int h = blockIdx.x, b = blockIdx.y;
  grid_dependency_wait();  // the lengths and partials may come from the kernel before
  const SeqRange r =
      seq_range(a.seq_lens[b], a.window, a.capacity, a.chunk, a.max_shards, a.T, a.balanced);
  merge_group<D, E>(a, b, h, r.nshards, r.status != 0, threadIdx.x, blockDim.x, merge_smem,
                    kShardBlock, [] { __syncthreads(); },
                    GridSlots{b, h, a.T, a.G, a.Hq, a.max_shards});
}

}  // namespace pgd
