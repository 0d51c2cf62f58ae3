// decode_attn_static_scratch: decode attention for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain scratch memory: a host program whose
// device memory is entirely held by another framework's caching allocator
// (the caller has no handle to it), a plugin interface that hands this code
// only the tensors of the call, or a latency-critical path that must not pay
// cudaMalloc's implicit synchronisation.  For them the shard partials live in
// a fixed array inside this library instead of a caller-provided workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds DECODE_ATTN_STATIC_SCRATCH_BYTES of it until the process
// exits.  Host code cannot use the variable's name as a device address (it
// is a host-side stand-in): the device address is looked up once per device
// with cudaGetSymbolAddress, with that device current, on the first call made
// on that device.  That first call should therefore come before any stream
// capture.  No call allocates: no cudaMalloc, cudaFree or allocating library
// routine is used here.
//
// Every call on a device shares the one array and leaves its contents behind.
// The only part that must start at zero, the per-group shard tickets, is
// cleared by each call itself: before its launch, an asynchronous memset on
// the call's stream zeroes the array's ticket region (a memset allocates
// nothing).  So a call that ended early (a pipeline wait that gave up) cannot
// leave a stale ticket for the next one.  Every partial the merge reads is
// written earlier in the same call.  Calls whose work overlaps on the GPU
// (different streams, or different host threads) race on the array and must
// be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/decode_attn.h"

namespace pgd {
// The argument checks decode_attn_make_plan starts with (api.cu): shapes,
// head dim, page size, group, dtype, schedule; no device call.
int validate_params(const decode_attn_params* p);
}  // namespace pgd

namespace {

__device__ __align__(256) unsigned char g_static_scratch[DECODE_ATTN_STATIC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
void* g_scratch_addr[kMaxScratchDevices];
std::mutex g_scratch_mu;

// Device address of the array on the current device (looked up once).
int scratch_address(int device, void** addr) {
  if (device < 0 || device >= kMaxScratchDevices) return DECODE_ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return DECODE_ATTN_ERR_CUDA;
    g_scratch_addr[device] = p;
  }
  *addr = g_scratch_addr[device];
  return DECODE_ATTN_OK;
}

}  // namespace

extern "C" int decode_attn_static_scratch(const decode_attn_params* p, const void* q,
                                          const void* k_pages, const void* v_pages,
                                          const int32_t* page_table, const int32_t* seq_lens,
                                          void* out, int32_t* err_flag, void* stream) {
  // argument errors first, without touching the device
  int st = pgd::validate_params(p);
  if (st) return st;
  int device = 0, sms = 0;
  if (cudaGetDevice(&device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return DECODE_ATTN_ERR_CUDA;
  void* scratch = nullptr;
  if ((st = scratch_address(device, &scratch))) return st;  // set-up on the first call
  decode_attn_plan plan;
  if ((st = decode_attn_make_plan(p, sms, &plan))) return st;
  if (plan.workspace_bytes > DECODE_ATTN_STATIC_SCRATCH_BYTES) return DECODE_ATTN_ERR_SCRATCH_LIMIT;
  // the tickets of this call start at zero whatever the last call left
  if ((st = decode_attn_workspace_clear(p, scratch, DECODE_ATTN_STATIC_SCRATCH_BYTES, stream)))
    return st;
  return decode_attn(p, q, k_pages, v_pages, page_table, seq_lens, out, scratch,
                     DECODE_ATTN_STATIC_SCRATCH_BYTES, err_flag, stream);
}
