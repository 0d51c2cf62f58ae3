// Paged K/V append: writes the step's new K/V rows into their pages, the step
// before attention (idle-intelligence/llm-web pull request 8, suffix-prefill
// commit: new rows are scattered into the cache after the resident prefix).
// One thread per 16-byte chunk of a row; the copy is bit-exact.  A negative
// position means the sequence has no new row; a position past the page table
// or a page id outside the pool writes nothing and raises an error bit.
#include "launch.h"

namespace pgd {
namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(const KvAppendArgs a) {
  const int64_t per_seq = (int64_t)a.Hkv * a.chunks;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)a.B * per_seq) return;
  const int b = (int)(idx / per_seq);
  const int rem = (int)(idx % per_seq);
  const int h = rem / a.chunks, c = rem % a.chunks;
  const int pos = a.positions[b] + a.pos_offset;
  if (pos < 0) return;
  if (pos >= a.max_pages * a.page_size) {
    if (rem == 0) raise_error(a.err, DECODE_ATTN_DEV_BAD_LEN);
    return;
  }
  const size_t pi = (size_t)b * a.max_pages + pos / a.page_size;
  if (!PGD_IN(pi, (size_t)a.B * a.max_pages, a.err)) return;
  const int phys = a.page_table[pi];
  if (phys < 0 || phys >= a.num_pages) {
    if (rem == 0) raise_error(a.err, DECODE_ATTN_DEV_BAD_PAGE);
    return;
  }
  const size_t dst =
      (((size_t)phys * a.page_size + pos % a.page_size) * a.Hkv + h) * a.chunks + c;
  if (!PGD_IN(dst, (size_t)a.num_pages * a.page_size * a.Hkv * a.chunks, a.err)) return;
  a.k_pages[dst] = a.k_new[idx];
  a.v_pages[dst] = a.v_new[idx];
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendArgs& a, cudaStream_t stream) {
  const int64_t total = (int64_t)a.B * a.Hkv * a.chunks;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((total + threads - 1) / threads);
  kv_append_kernel<<<blocks, threads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pgd
