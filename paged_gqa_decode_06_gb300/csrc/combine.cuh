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
  int32_t B, Hq, G, T, capacity, window, chunk, max_shards;
};

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
constexpr int kMaxMergeRows = 16;  // rows of one group (G <= 16)

// Shared memory merge_group needs: staged (m, l) plus per-row max and flag.
__host__ __device__ constexpr int merge_smem_bytes(int G) {
  return G * kShardBlock * 8 + kMaxMergeRows * 8;
}

// Merges the S shards of group (b, h) (its T*G query rows) into out, using threads [0, nthreads)
// (tid = this thread's index among them) and `smem` (merge_smem_bytes(G)
// bytes, 16-byte aligned).  `sync` is a barrier over exactly those threads.
// dead forces zero rows (an invalid range).
template <int D, class E, class Sync>
__device__ __forceinline__ void merge_group(const CombineArgs& a, int b, int h, int S, bool dead,
                                            int tid, int nthreads, uint8_t* smem, Sync sync) {
  constexpr int kQuads = D / 4;
  const int G = a.T * a.G;  // rows of the group
  float2* ml_s = reinterpret_cast<float2*>(smem);                       // [G][kShardBlock]
  float* max_s = reinterpret_cast<float*>(smem + G * kShardBlock * 8);  // [G]
  int* zero_s = reinterpret_cast<int*>(max_s + kMaxMergeRows);          // [G]

  // per-row maximum and bad-partial flag, from (m, l) staged block by block
  sync();
  if (tid < G) {
    max_s[tid] = -INFINITY;
    zero_s[tid] = (dead || S == 0) ? 1 : 0;
  }
  for (int s0 = 0; s0 < S; s0 += kShardBlock) {
    const int n = min(kShardBlock, S - s0);
    sync();
    for (int e = tid; e < G * n; e += nthreads) {
      const int g = e / n, j = e % n;
      ml_s[g * kShardBlock + j] =
          __ldcg(a.ws_ml + group_row(b, h, g, a.T, a.G, a.Hq) * a.max_shards + s0 + j);
    }
    sync();
    if (tid < G) {
      float M = max_s[tid];
      int z = zero_s[tid];
      for (int j = 0; j < n; ++j) {
        const float2 v = ml_s[tid * kShardBlock + j];
        z |= v.y < 0.f ? 1 : 0;  // a shard saw a bad page or gave up waiting
        M = fmaxf(M, v.x);
      }
      max_s[tid] = M;
      zero_s[tid] = z;
    }
  }
  sync();

  // two output items (row, 4 dims) per thread and pass, their shard loads
  // issued together so several L2 round trips overlap
  const bool staged = S <= kShardBlock;
  const int total = G * kQuads;
  for (int e0 = tid; e0 < total; e0 += 2 * nthreads) {
    int e[2] = {e0, e0 + nthreads};
    const int n_items = e[1] < total ? 2 : 1;
    if (n_items == 1) e[1] = e0;
    float4 o[2];
    float L[2], M[2];
    bool zero[2];
    const float2* ml[2];
    const float4* acc[2];
    size_t row[2];
    int quad[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int g = e[k] / kQuads;
      quad[k] = e[k] % kQuads;
      row[k] = group_row(b, h, g, a.T, a.G, a.Hq);
      M[k] = max_s[g];
      // a row with no attended position in any shard (a query before the
      // first cached position) stays zero
      zero[k] = zero_s[g] != 0 || M[k] == -INFINITY;
      // (m, l) from shared memory when one block holds them all
      ml[k] = staged ? ml_s + g * kShardBlock : a.ws_ml + row[k] * a.max_shards;
      acc[k] = reinterpret_cast<const float4*>(a.ws_acc + row[k] * a.max_shards * D) + quad[k];
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
          x[k][u] = __ldcg(acc[k] + (size_t)(s + u) * kQuads);
          v[k][u] = staged ? ml[k][s + u] : __ldcg(ml[k] + s + u);
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
        const float4 x = __ldcg(acc[k] + (size_t)s * kQuads);
        const float2 v = staged ? ml[k][s] : __ldcg(ml[k] + s);
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
      uint32_t* dst =
          reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + row[k] * D + 4 * quad[k]);
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
  const SeqRange r =
      seq_range(a.seq_lens[b], a.window, a.capacity, a.chunk, a.max_shards, a.T);
  grid_dependency_wait();
  merge_group<D, E>(a, b, h, r.nshards, r.status != 0, threadIdx.x, blockDim.x, merge_smem,
                    [] { __syncthreads(); });
}

}  // namespace pgd
