// Device helpers shared by the decode-attention kernels: inline PTX for
// mbarriers and TMA, bounded waits, and the shard arithmetic that the split
// and combine kernels must agree on.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through cudart)
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/decode_attn.h"

namespace pgd {

constexpr int kTile = 64;           // tokens per pipeline stage
constexpr int kMaxPieces = 1024;    // TMA boxes per shard (page-id table in smem)
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ PTX ---

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// A 32-bit global load the compiler keeps in program order with the other
// asm loads (so two independent loads go out back to back).
__device__ __forceinline__ int32_t ld_global_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase of `bar` with the given parity to complete, giving up
// after about two seconds (returns false then).  Every spin in these kernels
// goes through here, so a lost arrival cannot hang the GPU.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 2000000000ull) return false;
  }
  return true;
}

// 3-D tiled TMA load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, int32_t c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// An L2 cache policy that evicts the lines a load brings in first: every K/V
// byte of a step is read exactly once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 4-D tiled TMA load (the 128-byte swizzled view of the pool) into this
// CTA's shared memory, completing on `bar`, with an L2 cache policy
// (l2_evict_first_policy).
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                                 int32_t c1, int32_t c2, int32_t c3, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------- shard maths ---

// Attended range of one sequence and how it is cut into shards.  Shards are
// laid on a grid of kTile-aligned absolute positions starting at `base` (the
// window start rounded down), so every TMA box starts on a tile boundary.
struct SeqRange {
  int32_t start;    // first attended position
  int32_t end;      // one past the last attended position (= seq_len)
  int32_t base;     // start rounded down to a multiple of kTile
  int32_t chunk;    // positions per shard (a multiple of kTile)
  int32_t nshards;  // shards holding attended positions (0 for an empty range)
  int32_t status;   // 0 or DECODE_ATTN_DEV_* bits
};

// With T query positions per sequence (the last T positions), the range is
// the union of the queries' ranges: the first query's window start to L.
// balanced: the range is cut into max_shards near-equal shards (the planned
// chunk is then an upper bound), so that no shard of a sequence is much
// shorter than the others; otherwise every shard but the last has `chunk`
// positions.
__device__ __forceinline__ SeqRange seq_range(int32_t L, int32_t window, int32_t capacity,
                                              int32_t chunk, int32_t max_shards, int32_t T = 1,
                                              int32_t balanced = 0) {
  SeqRange r{0, 0, 0, chunk, 0, 0};
  if (L < 0 || L > capacity) {
    r.status = DECODE_ATTN_DEV_BAD_LEN;
    return r;
  }
  r.end = L;
  const int32_t first_end = L - T + 1;  // one past the first query's position
  r.start = (window > 0 && first_end > window) ? first_end - window : 0;
  r.base = r.start & ~(kTile - 1);
  if (balanced && L > r.base && max_shards > 0) {
    const int32_t even = (L - r.base + max_shards - 1) / max_shards;
    r.chunk = min(chunk, max(kTile, (even + kTile - 1) & ~(kTile - 1)));
  }
  r.nshards = (L > r.start) ? (L - r.base + r.chunk - 1) / r.chunk : 0;
  if (r.nshards > max_shards) {
    r.status = DECODE_ATTN_DEV_OVER_HINT;
    r.nshards = 0;
  }
  return r;
}

__device__ __forceinline__ void raise_error(int32_t* err, int32_t bits) {
  if (err) atomicOr(err, bits);
}

// Bounds checks of the checked build (compiled with PGD_CHECKED; the default
// build compiles them to `true` and evaluates nothing): an index outside
// [0, n) raises DECODE_ATTN_DEV_CHECK, and the caller skips the access or
// redirects it to a harmless one.  Stands in for a memory checker where none
// can run.
#ifdef PGD_CHECKED
__device__ __forceinline__ bool pgd_in_range(uint64_t i, uint64_t n, int32_t* err) {
  if (i < n) return true;
  raise_error(err, DECODE_ATTN_DEV_CHECK);
  return false;
}
#define PGD_IN(i, n, err) ::pgd::pgd_in_range((uint64_t)(i), (uint64_t)(n), (err))
#else
#define PGD_IN(i, n, err) true
#endif

}  // namespace pgd
