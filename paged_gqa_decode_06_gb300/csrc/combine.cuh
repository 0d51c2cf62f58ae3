// Ordered combine of shard partials (apache/tvm pull request 20426: per-shard
// online-softmax states merged after the sharded pass; BackendStack21/
// mlx-runner pull request 3: the combine merges the partials in the same
// order every time, so results are bit-identical run to run).
//
// One warp per (b, hq) row; lane i owns dims [i*D/32, (i+1)*D/32).  Shards
// are merged strictly in ascending index:
//   M = max_s m_s,  c_s = 2^(m_s - M),  L = sum_s c_s l_s,
//   out = fp16_rn(sum_s c_s acc_s / L)
// No atomics, so the bits depend only on the inputs and the shard plan.
#pragma once

#include "device_common.cuh"

namespace pgd {

struct CombineArgs {
  const int32_t* seq_lens;
  const float* ws_acc;   // [B*Hq*S_max][D]
  const float2* ws_ml;   // [B*Hq*S_max]
  __half* out;           // [B][Hq][D]
  int32_t B, Hq, capacity, window, chunk, max_shards;
};

constexpr int kCombineWarps = 4;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineArgs a) {
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (row >= a.B * a.Hq) return;
  const int b = row / a.Hq;
  const SeqRange r = seq_range(a.seq_lens[b], a.window, a.capacity, a.chunk, a.max_shards);
  const float2* ml = a.ws_ml + (size_t)row * a.max_shards;
  const float* acc = a.ws_acc + (size_t)row * a.max_shards * D + lane * DPL;

  bool zero = r.status != 0 || r.nshards == 0;
  float M = -INFINITY;
  for (int s = 0; s < r.nshards && !zero; ++s) {
    const float2 v = ml[s];
    if (v.y < 0.f) zero = true;  // a shard saw a bad page or gave up waiting
    M = fmaxf(M, v.x);
  }
  float o[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) o[e] = 0.f;
  float L = 0.f;
  if (!zero) {
    for (int s = 0; s < r.nshards; ++s) {
      const float2 v = ml[s];
      if (v.y == 0.f) continue;
      const float c = fast_exp2(v.x - M);
      L += c * v.y;
      const float* src = acc + (size_t)s * D;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[e] += c * src[e];
    }
  }
  __half* dst = a.out + (size_t)row * D + lane * DPL;
#pragma unroll
  for (int e = 0; e < DPL; ++e)
    dst[e] = __float2half_rn((zero || L == 0.f) ? 0.f : o[e] / L);
}

}  // namespace pgd
