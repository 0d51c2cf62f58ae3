// C ABI of the decode-attention library: argument checks, the host planner,
// TMA descriptors for the paged K/V pool, and the launches.
#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "launch.h"

using namespace pgd;

namespace {

constexpr int kDefaultSplitMin = 256;
constexpr int kMaxDevices = 64;
constexpr int kMinChunk = 128;        // shortest shard the planner picks, tokens
constexpr int kLargeChunkCap = 2048;  // longest shard for large work, unless span / 16
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kMaxCluster = 16;  // largest thread-block cluster (above 8: non-portable)
// Cost model of a one-wave split plan, calibrated on GB300 chunk sweeps (one,
// two and four sequences of 16 Ki..128 Ki tokens, the Llama-3.1-8B shape, the
// windowed long case):
constexpr double kStreamBytesPerS = 7.0e12;  // sustained K/V read rate of the split kernel
constexpr double kRoundTripS = 3.0e-6;       // loaded latency: a CTA moves its ring once per trip
// One-wave grids are kept to about this share of the CTA slots: with every
// slot filled, each SM runs two CTAs and the shared SMs' CTAs finish last
// (GB300: one 131072-token sequence 89.1 us at 256 CTAs against 94.3 us at
// 304; two of 65536 87.5 against 90.0; the long case 302.7 at 256).
constexpr double kOneWaveFill = 0.85;
// Clusters above the portable 8 CTAs only for grids this small: larger grids
// of 9..16-CTA clusters cannot be packed onto the GPCs (two 65536-token
// sequences in 16-CTA clusters: 133 us against 87.5 us merging through the
// workspace; the head_dim-256 sweep shape, 64 CTAs: 16.3 against 18.3 us).
constexpr int64_t kLargeClusterMaxCtas = 64;
constexpr double kMergeStepS = 1.2e-6;       // the last CTA's merge: one L2 round trip per 8 shards

std::atomic<int> g_sm_count[kMaxDevices];

int sm_count(int device, int* out) {
  if (device < 0 || device >= kMaxDevices) return DECODE_ATTN_ERR_CUDA;
  int n = g_sm_count[device].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        n <= 0)
      return DECODE_ATTN_ERR_CUDA;
    g_sm_count[device].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return DECODE_ATTN_OK;
}

// A positive integer from the environment, read once per process (0 when
// unset or not a positive number).
int env_positive(const char* name) {
  const char* v = std::getenv(name);
  if (!v || !*v) return 0;
  char* end = nullptr;
  const long x = std::strtol(v, &end, 10);
  return (end && *end == 0 && x > 0 && x < (1L << 30)) ? (int)x : 0;
}
int env_positive_now(const char* name) { return env_positive(name); }

// Process-wide defaults for the planner's two knobs, for A/B runs without
// code changes: DECODE_ATTN_SPLIT_MIN (the split threshold, default 256) and
// DECODE_ATTN_FORCE_CHUNK (a fixed shard length); a nonzero field of
// decode_attn_params takes precedence.
int env_split_min() {
  static const int v = env_positive("DECODE_ATTN_SPLIT_MIN");
  return v > 0 ? v : kDefaultSplitMin;
}
int env_force_chunk() {
  static const int v = env_positive("DECODE_ATTN_FORCE_CHUNK");
  return v;
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}
int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t ceil_div(int64_t x, int64_t m) { return (x + m - 1) / m; }

int check_params(const decode_attn_params* p) {
  if (!p) return DECODE_ATTN_ERR_NULL;
  if (p->batch < 0 || p->batch > 65535 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 ||
      p->num_kv_heads > 65535 || p->num_q_heads % p->num_kv_heads != 0 ||
      p->max_pages_per_seq <= 0 || p->num_pages <= 0)
    return DECODE_ATTN_ERR_SHAPE;
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256)
    return DECODE_ATTN_ERR_HEAD_DIM;
  if (!is_pow2(p->page_size) || p->page_size < 8 || p->page_size > 256)
    return DECODE_ATTN_ERR_PAGE_SIZE;
  if ((int64_t)p->max_pages_per_seq * p->page_size > INT32_MAX / 2 ||
      (int64_t)p->num_pages * p->page_size >= INT32_MAX)
    return DECODE_ATTN_ERR_SHAPE;
  if (p->num_q_heads / p->num_kv_heads > 16) return DECODE_ATTN_ERR_GROUP;
  if (!std::isfinite(p->scale) || p->num_queries > 4096) return DECODE_ATTN_ERR_SHAPE;
  if (p->dtype != DECODE_ATTN_DTYPE_FP16 && p->dtype != DECODE_ATTN_DTYPE_BF16)
    return DECODE_ATTN_ERR_SHAPE;
  if (p->schedule < 0 || p->schedule > DECODE_ATTN_SCHEDULE_CLUSTER) return DECODE_ATTN_ERR_SHAPE;
  return DECODE_ATTN_OK;
}

// The shard tickets (one int32 per (sequence, KV head)) sit in a region at
// the start of every workspace that partials never use, 64 KiB unless a plan
// has more groups: a zero-filled workspace therefore stays valid across calls
// with different shapes, since every completed call leaves its tickets zero.
constexpr size_t kTicketRegion = 64 * 1024;
// Group tickets [B*Hkv] (and 64 spare words).
size_t ticket_region_bytes(const decode_attn_params* p) {
  const size_t need = (((size_t)p->batch * p->num_kv_heads + 64) * 4 + 255) / 256 * 256;
  return need > kTicketRegion ? need : kTicketRegion;
}

int num_queries(const decode_attn_params* p) { return p->num_queries > 1 ? p->num_queries : 1; }

int next_pow2(int x) {
  int r = 1;
  while (r < x) r <<= 1;
  return r;
}

}  // namespace

namespace pgd {
int validate_params(const decode_attn_params* p) { return check_params(p); }
size_t simt_smem_bytes(int head_dim) {
  switch (head_dim) {
    case 64: return SimtCfg<64>::kSmemBytes;
    case 128: return SimtCfg<128>::kSmemBytes;
    default: return SimtCfg<256>::kSmemBytes;
  }
}
// Shards per sequence for plans whose grid fits in one wave of CTA slots
// (units = sequences x KV heads below the slot count): the S minimising
//   t(S) = bytes / min(stream rate, units * S * ring bytes / round trip)
//          + merge step * ceil(S / 8)          (no merge for S = 1)
// over chunks of kMinChunk..max_chunk tokens, at most `slots` CTAs and at
// least two shards (the length is above the split threshold); ties go to
// more CTAs.  Against the chunk sweeps it picks the measured best or a
// plan within 1 % of it (one 131072-token sequence: 32 shards, 89.1 us,
// against 92.0 at 24 and 94.3 at 38; the Llama shape: 16 shards, 14.3-14.4
// us, against 14.5-15.2 at 12 and 15.3 at 24).
int64_t one_wave_shards(int64_t units, int64_t slots, int64_t span, int head_dim,
                        int64_t max_chunk) {
  const int stages = head_dim == 64 ? 6 : 3;
  const double ring = (double)stages * 2 * kTile * head_dim * 2;  // K + V tiles in flight
  const double cta_rate = ring / kRoundTripS;
  const double bytes = (double)units * (double)span * 4.0 * head_dim;
  // above the split threshold the step is split: at least two shards
  const int64_t s_lo = std::max<int64_t>(2, ceil_div(span, max_chunk));
  const int64_t fill = std::max<int64_t>(1, (int64_t)(kOneWaveFill * (double)slots) / units);
  const int64_t s_hi = std::max<int64_t>(
      s_lo, std::min<int64_t>(std::min<int64_t>(slots / units, fill), ceil_div(span, kMinChunk)));
  int64_t best = s_lo;
  double best_t = 1e300;
  for (int64_t S = s_lo; S <= s_hi; ++S) {
    const int64_t chunk = round_up(ceil_div(span, S), kTile);
    if (chunk > max_chunk) continue;
    const int64_t se = ceil_div(span, chunk);  // shards this chunk really gives
    const double rate = std::min(kStreamBytesPerS, (double)(units * se) * cta_rate);
    const double t = bytes / rate + (se > 1 ? kMergeStepS * (double)ceil_div(se, 8) : 0.0);
    if (t < best_t * (1.0 - 1e-3) || (t <= best_t * (1.0 + 1e-3) && se > best)) {
      best = se;
      best_t = std::min(best_t, t);
    }
  }
  return best;
}

int simt_ctas_per_sm(int head_dim) {
  // dynamic ring + static smem (page coordinates, barriers, scratch) + 1 KB
  const size_t per_cta = simt_smem_bytes(head_dim) + kMaxPieces * 4 + 2048 + 1024;
  return std::max<int>(1, (int)(kSmemPerSm / per_cta));
}
int mma_ctas_per_sm(int head_dim, bool shallow) {
  size_t ring;
  switch (head_dim) {
    case 64: ring = shallow ? MmaCfg<64, true>::kSmemBytes : MmaCfg<64>::kSmemBytes; break;
    case 128: ring = shallow ? MmaCfg<128, true>::kSmemBytes : MmaCfg<128>::kSmemBytes; break;
    default: ring = MmaCfg<256>::kSmemBytes; break;
  }
  const size_t per_cta = ring + kMaxPieces * 4 + 2048 + 1024;
  return std::max<int>(1, (int)(kSmemPerSm / per_cta));
}
}  // namespace pgd

extern "C" int decode_attn_make_plan(const decode_attn_params* p, int32_t num_sms,
                                     decode_attn_plan* plan) {
  int st = check_params(p);
  if (st) return st;
  if (!plan) return DECODE_ATTN_ERR_NULL;
  if (num_sms <= 0) return DECODE_ATTN_ERR_SHAPE;
  std::memset(plan, 0, sizeof(*plan));
  const int G = p->num_q_heads / p->num_kv_heads;
  const int gp = next_pow2(G);
  const int T = p->num_queries > 1 ? p->num_queries : 1;
  int variant = p->variant;
  // the tensor-core variant measured faster on every shape (G = 4 and 8,
  // D = 64..256); the CUDA-core variant stays selectable
  if (variant == DECODE_ATTN_VARIANT_AUTO) variant = DECODE_ATTN_VARIANT_MMA;
  int group_pad = gp;
  if (variant == DECODE_ATTN_VARIANT_SIMT) {
    if (gp > 8 || T > 1 || p->dtype != DECODE_ATTN_DTYPE_FP16) return DECODE_ATTN_ERR_VARIANT;
  } else if (variant == DECODE_ATTN_VARIANT_MMA) {
    const int rows = T * G;  // query rows per KV head: one or two n8 tiles
    if (rows > 16) return DECODE_ATTN_ERR_VARIANT;
    group_pad = rows <= 8 ? 8 : 16;
  } else {
    return DECODE_ATTN_ERR_VARIANT;
  }

  const int64_t capacity = (int64_t)p->max_pages_per_seq * p->page_size;
  const int64_t max_len =
      p->max_seq_len > 0 ? std::min<int64_t>(p->max_seq_len, capacity) : capacity;
  // T queries: the first one's window starts T - 1 positions earlier
  const int64_t attended =
      p->window > 0 ? std::min<int64_t>(max_len, (int64_t)p->window + T - 1) : max_len;
  // positions from the tile-aligned base to the end of the longest sequence
  const int64_t span = std::max<int64_t>(1, p->window > 0 ? attended + kTile - 1 : max_len);
  const int box_t = std::min(p->page_size, kTile);
  const int64_t max_chunk = (int64_t)kMaxPieces * box_t;
  const int split_min = p->split_min > 0 ? p->split_min : env_split_min();
  const int ctas_per_sm = simt_ctas_per_sm(p->head_dim);

  int64_t chunk;
  const int force_chunk = p->force_chunk > 0 ? p->force_chunk : env_force_chunk();
  if (force_chunk > 0) {
    chunk = round_up(force_chunk, kTile);
    if (chunk > max_chunk) return DECODE_ATTN_ERR_SHAPE;
  } else if (attended <= split_min) {
    // one shard covers the whole range, unless the range is longer than one
    // shard can hold (kMaxPieces boxes): then the fewest shards that fit
    chunk = std::min(round_up(span, kTile), max_chunk);
  } else {
    // Shard count from the work bound (every (sequence, KV head) unit at the
    // longest length) and the CTA slots (SMs x resident CTAs), calibrated on
    // GB300 sweeps of the chunk size:
    //  * fewer units than slots: one wave, the shard count from the cost
    //    model above (stream rate against the merge's serial tail);
    //  * small work otherwise (up to 1 MiB per slot): one shard per unit;
    //  * large work: about 1.7 waves of CTAs, fewer prologues while DRAM stays
    //    saturated to the end; chunks capped at max(2048, span / 16) tokens
    //    so that batches of mixed lengths still cut into balanced pieces.
    const int64_t units = std::max<int64_t>(1, (int64_t)p->batch * p->num_kv_heads);
    const int64_t slots = (int64_t)num_sms * ctas_per_sm;
    const int64_t work_bytes = units * span * 4 * p->head_dim;
    int64_t S;
    if (units < slots) {
      S = one_wave_shards(units, slots, span, p->head_dim, max_chunk);
    } else if (work_bytes <= slots * (int64_t(1) << 20)) {
      S = std::max<int64_t>(1, std::min(slots / units, ceil_div(span, kMinChunk)));
    } else {
      const int64_t target = std::max<int64_t>(1, (17 * slots + 5 * units) / (10 * units));
      const int64_t cap = std::max<int64_t>(kLargeChunkCap, round_up(ceil_div(span, 16), kTile));
      S = std::max(target, ceil_div(span, cap));
    }
    chunk = std::min(round_up(ceil_div(span, S), kTile), max_chunk);
  }
  if (chunk > max_chunk) return DECODE_ATTN_ERR_SHAPE;
  const int64_t max_shards = ceil_div(span, chunk);
  if (max_shards > 65535) return DECODE_ATTN_ERR_SHAPE;

  plan->variant = variant;
  plan->group_pad = group_pad;
  plan->tile_tokens = kTile;
  plan->chunk_tokens = (int32_t)chunk;
  plan->max_shards = (int32_t)max_shards;
  plan->split = max_shards > 1 ? 1 : 0;
  // Shallow ring (tensor-core kernel, D <= 128): for grids of several waves
  // of short shards (at most 8 tiles each), 2 stages (4 at D = 64) fit 3
  // CTAs per SM, and more CTAs' first round trips overlap.  GB300: a
  // thousand sequences of U[1, 512] tokens 203.3 -> 178.4 us; long streams
  // lose by it (one 131072-token sequence 88.5 -> 95.6 us), so only short
  // shards take it.
  const int64_t ctas = (int64_t)p->batch * p->num_kv_heads * max_shards;
  const bool shallow = variant == DECODE_ATTN_VARIANT_MMA &&
                       (p->head_dim == 64 || (p->head_dim == 128 && group_pad == 8)) &&
                       chunk <= 8 * kTile && ctas > (int64_t)num_sms * ctas_per_sm;
  int cps = ctas_per_sm;
  if (variant == DECODE_ATTN_VARIANT_MMA) cps = mma_ctas_per_sm(p->head_dim, shallow);
  plan->ring_stages = variant == DECODE_ATTN_VARIANT_MMA
                          ? (p->head_dim == 64 ? (shallow ? 4 : 6) : (shallow ? 2 : 3))
                          : (p->head_dim == 64 ? 6 : 3);
  // several waves of CTAs: heads fastest; one wave: shards fastest (measured
  // on GB300: long context 303.0 vs 307.6 us, Llama-3.1-8B shape 18.1 vs 17.5 us)
  const int64_t slots_all = (int64_t)num_sms * cps;
  const bool head_fastest = ctas > slots_all;
  plan->head_fastest = head_fastest ? 1 : 0;
  // one-wave split plans cut each sequence into max_shards near-equal
  // shards: all CTAs run at once, so the step lasts as long as the longest
  // shard (a 4096-position window on 64-aligned lengths: 8 x 512 positions
  // instead of 7 x 576 + 64); a forced chunk is taken as given
  plan->balanced = (plan->split && !head_fastest && force_chunk <= 0) ? 1 : 0;
  plan->grid_x = head_fastest ? p->num_kv_heads : (int32_t)max_shards;
  plan->grid_y = head_fastest ? (int32_t)max_shards : p->num_kv_heads;
  plan->grid_z = p->batch;
  plan->ctas_per_sm = cps;
  // Cluster merge: the shards of a (KV head, sequence) as one thread-block
  // cluster (grid x = shards), merged through distributed shared memory
  // instead of the workspace and a ticket, for one-wave tensor-core split
  // plans of 2..16 shards.  The planner takes it when the grid fills at
  // least 4/5 of the CTA slots or the step is small: a cluster's CTAs are
  // packed onto neighbouring SMs of one GPC, so a sparse grid of clusters
  // leaves SMs idle.
  const bool cluster_ok = variant == DECODE_ATTN_VARIANT_MMA && plan->split && !head_fastest &&
                          !shallow && max_shards >= 2 &&
                          (max_shards <= 8 || (max_shards <= kMaxCluster &&
                                               ctas <= kLargeClusterMaxCtas));
  const int64_t step_bytes =
      (int64_t)p->batch * p->num_kv_heads * span * 4 * p->head_dim;
  if (p->schedule == DECODE_ATTN_SCHEDULE_CLUSTER) {
    if (!cluster_ok) return DECODE_ATTN_ERR_VARIANT;
    plan->cluster = (int32_t)max_shards;
  } else if (p->schedule == DECODE_ATTN_SCHEDULE_AUTO && cluster_ok &&
             (ctas * 5 >= slots_all * 4 || step_bytes <= (int64_t(32) << 20))) {
    plan->cluster = (int32_t)max_shards;
  }
  if (plan->split) {
    // shard tickets (a fixed region first), (m, l) pairs, fp32 accumulators
    const size_t rows = (size_t)p->batch * T * p->num_q_heads * (size_t)plan->max_shards;
    plan->workspace_bytes = ticket_region_bytes(p) + round_up(rows * sizeof(float2), 256) +
                            round_up(rows * p->head_dim * 4, 256);
  }
  return DECODE_ATTN_OK;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D view of a [P][PS][Hkv][D] fp16 pool: (d, kv head, P*PS token rows);
// one box = box_t consecutive rows of one KV head.
int encode_pool_map(CUtensorMap* map, const void* base, const decode_attn_params* p, int box_t) {
  auto fn = encode_fn();
  if (!fn) return DECODE_ATTN_ERR_TENSOR_MAP;
  const int D = p->head_dim;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p->num_kv_heads,
                        (cuuint64_t)p->num_pages * p->page_size};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p->num_kv_heads * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)box_t};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType et = p->dtype == DECODE_ATTN_DTYPE_BF16
                                    ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(map, et, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DECODE_ATTN_OK : DECODE_ATTN_ERR_TENSOR_MAP;
}

// 4-D view (64 dims, P*PS token rows, kv head, D/64 chunks) with the 128-byte
// swizzle, written to shared memory as [D/64][box_t][64] per box_t rows
// (16-byte chunk c of row t at c ^ (t % 8)).  Pieces shorter than 64 rows
// take one box for all D dims: on GB300 one CTA copying per-chunk boxes of
// 16 rows (2 KB) was capped near 45 GB/s, and the batched workload (pages
// of 16) went from 197.2 to 193-195 us with the whole piece in one box.
// 64-row pieces keep one box per 64-dim chunk (8 KB each), which measured
// faster there (one 131072-token sequence 89.1 against 90.2 us).
int encode_pool_map_swizzled(CUtensorMap* map, const void* base, const decode_attn_params* p,
                             int box_t) {
  auto fn = encode_fn();
  if (!fn) return DECODE_ATTN_ERR_TENSOR_MAP;
  const int D = p->head_dim;
  cuuint64_t dims[4] = {64, (cuuint64_t)p->num_pages * p->page_size,
                        (cuuint64_t)p->num_kv_heads, (cuuint64_t)D / 64};
  cuuint64_t strides[3] = {(cuuint64_t)p->num_kv_heads * D * 2, (cuuint64_t)D * 2, 128};
  cuuint32_t box[4] = {64, (cuuint32_t)box_t, 1, box_t < kTile ? (cuuint32_t)D / 64 : 1u};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType et = p->dtype == DECODE_ATTN_DTYPE_BF16
                                    ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(map, et, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DECODE_ATTN_OK : DECODE_ATTN_ERR_TENSOR_MAP;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

int plan_for_stream(const decode_attn_params* p, cudaStream_t stream, decode_attn_plan* plan) {
  (void)stream;
  int st = check_params(p);  // argument errors are reported before any CUDA call
  if (st) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DECODE_ATTN_ERR_CUDA;
  int n = 0;
  st = sm_count(dev, &n);
  if (st) return st;
  return decode_attn_make_plan(p, n, plan);
}

struct Workspace {
  float2* ml;
  float* acc;
  int32_t* counters;
  size_t counter_bytes;
};

int workspace_views(const decode_attn_params* p, const decode_attn_plan& plan, void* ws,
                    size_t ws_bytes, Workspace* out) {
  out->ml = nullptr;
  out->acc = nullptr;
  out->counters = nullptr;
  out->counter_bytes = 0;
  if (!plan.split) return DECODE_ATTN_OK;
  if (!ws || ws_bytes < plan.workspace_bytes || (reinterpret_cast<uintptr_t>(ws) & 255))
    return DECODE_ATTN_ERR_WORKSPACE;
  const size_t rows =
      (size_t)p->batch * num_queries(p) * p->num_q_heads * (size_t)plan.max_shards;
  char* base = static_cast<char*>(ws);
  const size_t tickets = ticket_region_bytes(p);
  const size_t ml_bytes = round_up(rows * sizeof(float2), 256);
  out->counters = reinterpret_cast<int32_t*>(base);
  out->counter_bytes = tickets;
  out->ml = reinterpret_cast<float2*>(base + tickets);
  out->acc = reinterpret_cast<float*>(base + tickets + ml_bytes);
  return DECODE_ATTN_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DECODE_ATTN_OK : DECODE_ATTN_ERR_CUDA; }

int run_split(const decode_attn_params* p, const decode_attn_plan& plan, const void* q,
              const void* k_pages, const void* v_pages, const int32_t* page_table,
              const int32_t* seq_lens, void* out, const Workspace& ws, int32_t* err_flag,
              cudaStream_t stream, const void* k_new = nullptr, const void* v_new = nullptr) {
  if (p->batch == 0) return DECODE_ATTN_OK;
  SplitLaunch L{};
  const int box_t = std::min(p->page_size, kTile);
  auto encode =
      plan.variant == DECODE_ATTN_VARIANT_MMA ? encode_pool_map_swizzled : encode_pool_map;
  int st = encode(&L.tmap_k, k_pages, p, box_t);
  if (!st) st = encode(&L.tmap_v, v_pages, p, box_t);
  if (st) return st;
  SplitArgs& a = L.args;
  a.q = q;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.ws_acc = ws.acc;
  a.ws_ml = ws.ml;
  a.counters = ws.counters;
  a.err = err_flag;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_pages_w = const_cast<void*>(k_pages);
  a.v_pages_w = const_cast<void*>(v_pages);
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.G = p->num_q_heads / p->num_kv_heads;
  a.max_pages = p->max_pages_per_seq;
  a.num_pages = p->num_pages;
  a.page_size = p->page_size;
  a.page_shift = ilog2(p->page_size);
  a.box_tokens = box_t;
  a.window = p->window > 0 ? p->window : 0;
  a.chunk = plan.chunk_tokens;
  a.max_shards = plan.max_shards;
  a.balanced = plan.balanced;
  a.split = plan.split;
  a.T = num_queries(p);
  a.head_fastest = plan.head_fastest;
  a.batch = p->batch;
  {
    const int64_t cap = (int64_t)p->max_pages_per_seq * p->page_size;
    a.len_hint = (int32_t)(p->max_seq_len > 0 ? std::min<int64_t>(p->max_seq_len, cap) : cap);
  }
  // Test hook (tensor-core kernel): DECODE_ATTN_TEST_STALL_TX=n makes the
  // first stage's barrier of every CTA expect n bytes more than the stage
  // brings, so its wait runs out (about 2 s) and the kernel must report
  // DECODE_ATTN_DEV_TIMEOUT, write zeros and leave the context usable.  Read
  // on every call, so a test can set and clear it; unset in normal use.
  a.stall_tx = env_positive_now("DECODE_ATTN_TEST_STALL_TX");
  a.scale_log2 = p->scale * kLog2e;
  L.grid = dim3(plan.grid_x, plan.grid_y, plan.grid_z);
  L.group_pad = plan.group_pad;
  L.variant = plan.variant;
  L.dtype = p->dtype;
  L.cluster = plan.cluster;
  L.shallow = (plan.variant == DECODE_ATTN_VARIANT_MMA && p->head_dim <= 128 &&
               plan.ring_stages == (p->head_dim == 64 ? 4 : 2))
                  ? 1
                  : 0;  // the launcher has the shallow kernels the planner picks from
  L.stream = stream;
  // the shard tickets are zero on entry: the last CTA of each group clears
  // its own, so a workspace cleared once stays clear across calls
  switch (p->head_dim) {
    case 64: return cuda_status(launch_split_d64(L));
    case 128: return cuda_status(launch_split_d128(L));
    default: return cuda_status(launch_split_d256(L));
  }
}

int run_combine(const decode_attn_params* p, const decode_attn_plan& plan,
                const int32_t* seq_lens, void* out, const Workspace& ws, int32_t* err_flag,
                cudaStream_t stream) {
  if (!plan.split || p->batch == 0) return DECODE_ATTN_OK;
  CombineArgs a{};
  a.seq_lens = seq_lens;
  a.err = err_flag;
  a.ws_acc = ws.acc;
  a.ws_ml = ws.ml;
  a.out = out;
  a.B = p->batch;
  a.Hq = p->num_q_heads;
  a.G = p->num_q_heads / p->num_kv_heads;
  a.T = num_queries(p);
  a.capacity = p->max_pages_per_seq * p->page_size;
  a.window = p->window > 0 ? p->window : 0;
  a.chunk = plan.chunk_tokens;
  a.max_shards = plan.max_shards;
  a.balanced = plan.balanced;
  switch (p->head_dim) {
    case 64: return cuda_status(launch_combine_d64(a, p->dtype, stream));
    case 128: return cuda_status(launch_combine_d128(a, p->dtype, stream));
    default: return cuda_status(launch_combine_d256(a, p->dtype, stream));
  }
}

int check_tensors(const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* page_table, const int32_t* seq_lens, const void* out) {
  if (!q || !k_pages || !v_pages || !page_table || !seq_lens || !out) return DECODE_ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return DECODE_ATTN_ERR_ALIGN;
  return DECODE_ATTN_OK;
}

}  // namespace

extern "C" size_t decode_attn_workspace_size(const decode_attn_params* p, int device) {
  int n = 0;
  if (sm_count(device, &n)) return 0;
  decode_attn_plan plan;
  if (decode_attn_make_plan(p, n, &plan)) return 0;
  return plan.workspace_bytes;
}

extern "C" int decode_attn_split(const decode_attn_params* p, const void* q, const void* k_pages,
                                 const void* v_pages, const int32_t* page_table,
                                 const int32_t* seq_lens, void* out, void* workspace,
                                 size_t workspace_bytes, int32_t* err_flag, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  decode_attn_plan plan;
  int st = plan_for_stream(p, s, &plan);
  if (st) return st;
  if ((st = check_tensors(q, k_pages, v_pages, page_table, seq_lens, out))) return st;
  Workspace ws;
  if ((st = workspace_views(p, plan, workspace, workspace_bytes, &ws))) return st;
  return run_split(p, plan, q, k_pages, v_pages, page_table, seq_lens, out, ws, err_flag, s);
}

extern "C" int decode_attn_combine(const decode_attn_params* p, const int32_t* seq_lens,
                                   void* out, void* workspace, size_t workspace_bytes,
                                   int32_t* err_flag, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  decode_attn_plan plan;
  int st = plan_for_stream(p, s, &plan);
  if (st) return st;
  if (!seq_lens || !out) return DECODE_ATTN_ERR_NULL;
  if (!aligned16(out)) return DECODE_ATTN_ERR_ALIGN;
  Workspace ws;
  if ((st = workspace_views(p, plan, workspace, workspace_bytes, &ws))) return st;
  return run_combine(p, plan, seq_lens, out, ws, err_flag, s);
}

extern "C" int decode_attn(const decode_attn_params* p, const void* q, const void* k_pages,
                           const void* v_pages, const int32_t* page_table,
                           const int32_t* seq_lens, void* out, void* workspace,
                           size_t workspace_bytes, int32_t* err_flag, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  decode_attn_plan plan;
  int st = plan_for_stream(p, s, &plan);
  if (st) return st;
  if ((st = check_tensors(q, k_pages, v_pages, page_table, seq_lens, out))) return st;
  Workspace ws;
  if ((st = workspace_views(p, plan, workspace, workspace_bytes, &ws))) return st;
  // the split kernel's last CTA per group merges the partials (no second launch)
  return run_split(p, plan, q, k_pages, v_pages, page_table, seq_lens, out, ws, err_flag, s);
}

extern "C" int decode_attn_append(const decode_attn_params* p, const void* q, const void* k_new,
                                  const void* v_new, void* k_pages, void* v_pages,
                                  const int32_t* page_table, const int32_t* seq_lens, void* out,
                                  void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                  void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  decode_attn_plan plan;
  int st = plan_for_stream(p, s, &plan);
  if (st) return st;
  if ((st = check_tensors(q, k_pages, v_pages, page_table, seq_lens, out))) return st;
  if (!k_new || !v_new) return DECODE_ATTN_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new)) return DECODE_ATTN_ERR_ALIGN;
  Workspace ws;
  if ((st = workspace_views(p, plan, workspace, workspace_bytes, &ws))) return st;
  return run_split(p, plan, q, k_pages, v_pages, page_table, seq_lens, out, ws, err_flag, s, k_new,
                   v_new);
}

extern "C" int decode_kv_append(const decode_attn_params* p, const void* k_new, const void* v_new,
                                const int32_t* positions, void* k_pages, void* v_pages,
                                const int32_t* page_table, int32_t* err_flag, void* stream) {
  int st = check_params(p);
  if (st) return st;
  if (!k_new || !v_new || !positions || !k_pages || !v_pages || !page_table)
    return DECODE_ATTN_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
    return DECODE_ATTN_ERR_ALIGN;
  if (p->batch == 0) return DECODE_ATTN_OK;
  KvAppendArgs a;
  a.k_new = static_cast<const uint4*>(k_new);
  a.v_new = static_cast<const uint4*>(v_new);
  a.positions = positions;
  a.pos_offset = 0;
  a.page_table = page_table;
  a.k_pages = static_cast<uint4*>(k_pages);
  a.v_pages = static_cast<uint4*>(v_pages);
  a.err = err_flag;
  a.B = p->batch;
  a.Hkv = p->num_kv_heads;
  a.chunks = p->head_dim / 8;
  a.page_size = p->page_size;
  a.max_pages = p->max_pages_per_seq;
  a.num_pages = p->num_pages;
  return cuda_status(launch_kv_append(a, static_cast<cudaStream_t>(stream)));
}

extern "C" int decode_attn_host(const decode_attn_params* p, const void* q_host,
                                const void* k_pages_host, const void* v_pages_host,
                                const int32_t* page_table_host, const int32_t* seq_lens_host,
                                void* out_host, void* d_q, void* d_k_pages, void* d_v_pages,
                                int32_t* d_page_table, int32_t* d_seq_lens, void* d_out,
                                size_t kv_bytes_to_copy, void* workspace,
                                size_t workspace_bytes, int32_t* err_flag, void* stream) {
  int st = check_params(p);
  if (st) return st;
  if (!q_host || !k_pages_host || !v_pages_host || !page_table_host || !seq_lens_host ||
      !out_host)
    return DECODE_ATTN_ERR_NULL;
  if ((st = check_tensors(d_q, d_k_pages, d_v_pages, d_page_table, d_seq_lens, d_out))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t D = p->head_dim;
  const size_t q_bytes = (size_t)p->batch * num_queries(p) * p->num_q_heads * D * 2;
  const size_t pool = (size_t)p->num_pages * p->page_size * p->num_kv_heads * D * 2;
  const size_t kv = (kv_bytes_to_copy == 0 || kv_bytes_to_copy > pool) ? pool : kv_bytes_to_copy;
  const size_t pt_bytes = (size_t)p->batch * p->max_pages_per_seq * 4;
  const size_t sl_bytes = (size_t)p->batch * 4;
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_q, q_host, q_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_k_pages, k_pages_host, kv, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_v_pages, v_pages_host, kv, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(d_page_table, page_table_host, pt_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(d_seq_lens, seq_lens_host, sl_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return DECODE_ATTN_ERR_CUDA;
  st = decode_attn(p, d_q, d_k_pages, d_v_pages, d_page_table, d_seq_lens, d_out, workspace,
                   workspace_bytes, err_flag, stream);
  if (st) return st;
  e = cudaMemcpyAsync(out_host, d_out, q_bytes, cudaMemcpyDeviceToHost, s);
  return cuda_status(e);
}

extern "C" int decode_attn_workspace_clear(const decode_attn_params* p, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  decode_attn_plan plan;
  int st = plan_for_stream(p, s, &plan);
  if (st) return st;
  if (!plan.split) return DECODE_ATTN_OK;
  Workspace ws;
  if ((st = workspace_views(p, plan, workspace, workspace_bytes, &ws))) return st;
  return cuda_status(cudaMemsetAsync(ws.counters, 0, ws.counter_bytes, s));
}

extern "C" const char* decode_attn_strerror(int status) {
  switch (status) {
    case DECODE_ATTN_OK: return "ok";
    case DECODE_ATTN_ERR_NULL: return "a required pointer is NULL";
    case DECODE_ATTN_ERR_SHAPE: return "invalid shape or size";
    case DECODE_ATTN_ERR_HEAD_DIM: return "head_dim must be 64, 128 or 256";
    case DECODE_ATTN_ERR_PAGE_SIZE: return "page_size must be a power of two in [8, 256]";
    case DECODE_ATTN_ERR_GROUP: return "num_q_heads / num_kv_heads must be at most 16";
    case DECODE_ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DECODE_ATTN_ERR_ALIGN: return "tensor pointers must be 16-byte aligned";
    case DECODE_ATTN_ERR_CUDA: return "CUDA runtime error";
    case DECODE_ATTN_ERR_TENSOR_MAP: return "TMA descriptor for the K/V pool rejected";
    case DECODE_ATTN_ERR_VARIANT: return "kernel variant unavailable for this shape";
    case DECODE_ATTN_ERR_SCRATCH_LIMIT:
      return "partials exceed the library's static scratch (8 MiB); use decode_attn with a "
             "workspace";
    default: return "unknown status";
  }
}
