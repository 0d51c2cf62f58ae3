// Host-side interface between the C ABI (api.cu) and the per-head-dim
// translation units that instantiate the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "combine.cuh"
#include "split_mma.cuh"
#include "split_simt.cuh"

namespace pgd {

struct SplitLaunch {
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  SplitArgs args;
  dim3 grid;
  int group_pad;
  int variant;
  int dtype;
  int shallow;      // tensor-core kernel with the shallow ring (MmaCfg kShallow)
  int cluster;      // > 0: the cluster-merge kernel, clusters of this many CTAs along x
  cudaStream_t stream;
};

cudaError_t launch_split_d64(const SplitLaunch& L);
cudaError_t launch_split_d128(const SplitLaunch& L);
cudaError_t launch_split_d256(const SplitLaunch& L);
cudaError_t launch_combine_d64(const CombineArgs& a, int dtype, cudaStream_t stream);
cudaError_t launch_combine_d128(const CombineArgs& a, int dtype, cudaStream_t stream);
cudaError_t launch_combine_d256(const CombineArgs& a, int dtype, cudaStream_t stream);

struct KvAppendArgs {
  const uint4* k_new;   // [B][Hkv][D] as 16-byte chunks
  const uint4* v_new;
  const int32_t* positions;  // position of sequence b's new row: positions[b] + pos_offset
  const int32_t* page_table;
  uint4* k_pages;       // [P][PS][Hkv][D] as 16-byte chunks
  uint4* v_pages;
  int32_t* err;
  int32_t pos_offset;
  int32_t B, Hkv, chunks, page_size, max_pages, num_pages;
};
cudaError_t launch_kv_append(const KvAppendArgs& a, cudaStream_t stream);

// Resident CTAs per SM the kernels are sized for (shared-memory bound).
int simt_ctas_per_sm(int head_dim);
int mma_ctas_per_sm(int head_dim, bool shallow);
size_t simt_smem_bytes(int head_dim);

}  // namespace pgd
