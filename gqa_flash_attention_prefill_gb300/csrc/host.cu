// host.cu -- C ABI of libgqa_prefill.so: argument validation, the launch
// configuration cache, TMA tensor maps and the launch.  Declared in
// include/gqa_prefill.h, which states the operation, layouts and errors.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "gqa_prefill.h"
#include "launch.h"

namespace gqa {

// Device status word (GQA_DEV_* bits); kernels receive its address.
__device__ unsigned int g_device_status;

// Snapshots of the status word taken by status_take_kernel, one slot per
// concurrent reader (slots are handed out round-robin).
constexpr int kStatusSlots = 64;
__device__ unsigned int g_status_snapshot[kStatusSlots];

// Reads and clears the status word in one atomic step, in stream order.
__global__ void status_take_kernel(unsigned int* status, unsigned int* snapshot) {
  *snapshot = atomicExch(status, 0u);
}

// Failure-detection self-test: one thread waits on an mbarrier that nothing
// ever arrives on, through the same bounded wait the prefill kernel uses.  The
// wait runs out after `timeout_ns`, raises GQA_DEV_TIMEOUT and the kernel
// returns normally, so the context stays usable.
__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0u;
    mbar_init(smem_u32(&bar), 1u);
    fence_barrier_init();
    (void)wait_bounded(smem_u32(&bar), 0u, &abort_flag, status, timeout_ns);
  }
}

namespace {

// Per-host-thread call flags (gqa_prefill_set_call_flags), read at each launch.
thread_local unsigned int t_call_flags = 0u;

std::mutex g_mu;      // guards the configuration cache and the forced variant
std::mutex g_dev_mu;  // guards the per-device information
int g_forced_block_n = 0;
int g_forced_q_tiles = 0;  // query tiles per unit (0: the cache's choice)

struct DeviceInfo {
  int sms = 0;
  int smem_per_sm = 0;
  unsigned int* status = nullptr;
  void* ctx = nullptr;  // the CUDA context the entry belongs to
};
std::map<int, DeviceInfo> g_devices;

// Launch-configuration cache.  Keyed on what changes which tile shape wins
// (head dim, a power-of-two bucket of the query length, heads, group size,
// windowed or not, dtype) and never on the KV length: the KV length only
// scales every candidate's loop uniformly (hip-ep PR #622, config-cache
// commit), while a window caps the tiles walked and so may change the winner
// (same page, window commit).
using CfgKey = std::tuple<int, int, int, int, int, int>;
struct CfgEntry {
  int block_n;
  int q_tiles;  // 128-row query tiles per unit
  bool tuned;   // chosen by a timed sweep rather than the default
};
std::map<CfgKey, CfgEntry> g_cfg_cache;
int g_tune_mode = -1;  // -1: read GQA_PREFILL_TUNE on first use; 0 off; 1 on

bool env_flag(const char* name) {
  const char* v = std::getenv(name);
  return v != nullptr && v[0] != '\0' && v[0] != '0';
}
// Environment settings read once per process (a getenv per call would scan
// the environment on every launch).
bool debug_flag() {
  static const bool v = env_flag("GQA_PREFILL_DEBUG");
  return v;
}
unsigned long long timeout_ns() {
  static const unsigned long long v = [] {
    unsigned long long ns = 4000000000ull;  // 4 s
    if (const char* t = std::getenv("GQA_PREFILL_TIMEOUT_MS")) {
      const long long ms = std::atoll(t);
      if (ms > 0) ns = (unsigned long long)ms * 1000000ull;
    }
    return ns;
  }();
  return v;
}

}  // namespace

void* current_context() {
  typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
  static CtxGetCurrentFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(ptr);
    return static_cast<CtxGetCurrentFn>(nullptr);
  }();
  CUcontext ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

bool pdl_enabled() {
  static const bool v = [] {
    const char* e = std::getenv("GQA_PREFILL_PDL");
    return !(e != nullptr && e[0] == '0');
  }();
  return v;
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_dev_mu);
  auto itr = g_devices.find(dev);
  // A context other than the one the entry was made in (the device was reset
  // since) may have loaded the module elsewhere: look everything up again.
  if (itr != g_devices.end() && itr->second.ctx != ctx) {
    g_devices.erase(itr);
    itr = g_devices.end();
  }
  if (itr == g_devices.end()) {
    DeviceInfo di;
    di.ctx = ctx;
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GQA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                               dev) != cudaSuccess)
      return GQA_ERR_CUDA;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return GQA_ERR_CUDA;
    di.status = static_cast<unsigned int*>(ptr);
    // Load the status reader's module now: a kernel loaded lazily at its
    // first launch can wait for work already running on other streams,
    // which a stream-scoped status read must not do.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, status_take_kernel) != cudaSuccess) return GQA_ERR_CUDA;
    itr = g_devices.emplace(dev, di).first;
  }
  *out = itr->second;
  return GQA_OK;
}

int pow2_bucket(int x) {
  int b = 1;
  while (b < x && b < (1 << 30)) b <<= 1;
  return b;
}

// Measured on GB300 (gpt-oss layer pair and chunked-prefix workloads): a
// full-causal d=64 layer runs fastest with 128-key tiles; windowed layers with
// 64-key tiles, which waste fewer masked keys at the window's lower edge.
CfgEntry default_config(int d, bool windowed) {
  if (d == 64) return CfgEntry{windowed ? 64 : 128, 1, false};
  return CfgEntry{64, 1, false};
}

struct Plan {
  KernelShape shape;
  int rows;       // query positions per 128-row query tile (128 / G)
  int unit_rows;  // query positions per unit (q_tiles * rows)
  int G, ctas_per_sm, grid, max_units;
  int slots;      // CTAs resident at once (SMs x CTAs per SM)
  int groups;     // launches: sequences are taken kMaxSeqs at a time
  unsigned smem_launch;  // dynamic smem requested per CTA
};

// Split-KV: S splits per unit; partials live in a caller-provided workspace.
struct SplitArgs {
  int num_splits = 1;
  float* part_o = nullptr;
  float* part_ml = nullptr;
  int32_t* part_hdr = nullptr;
  bool balanced = false;  // balanced split: one kernel, cut units merged in it
  unsigned long long* sk_count = nullptr;
};
constexpr int kMaxSplits = 16;
constexpr int kBalanced = -1;  // num_splits value requesting the balanced split

// Paged KV: the page table and the pool geometry (indices == nullptr: the
// contiguous layout).
struct KvPaging {
  const int32_t* indices = nullptr;
  int page_size = 0, num_pages = 0;
};

// Custom mask: the per-sequence bitmaps over the extend keys (custom_mask
// == nullptr: none).
struct MaskArgs {
  const uint32_t* custom_mask = nullptr;
  const int32_t* mask_indptr = nullptr;
  long long total_words = 0;
};

struct SplitLayout {
  size_t o_off, ml_off, hdr_off, bytes;
};
// Workspace layout for S splits: partial O (fp32, d per row), (m, l) per row,
// and the unit headers, each 256-byte aligned.
SplitLayout split_layout(const Plan& pl, int d, int S) {
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t items = (size_t)pl.max_units * S;
  const size_t rows = (size_t)pl.shape.q_tiles * 128;
  SplitLayout L;
  L.o_off = 0;
  L.ml_off = al(items * rows * (size_t)d * 4u);
  L.hdr_off = L.ml_off + al(items * rows * 8u);
  L.bytes = L.hdr_off + al((4u + 4u * (size_t)pl.max_units) * 4u);
  return L;
}

// Workspace layout of the balanced split: two partial slots per resident CTA
// (O in fp32 and (m, l) per row of its first and its last piece), and four
// count words per unit, each 256-byte aligned.
struct BalancedLayout {
  size_t o_off, ml_off, cnt_off, bytes;
};
BalancedLayout balanced_layout(const Plan& pl, int d) {
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t slots = 2u * (size_t)pl.slots;
  BalancedLayout L;
  L.o_off = 0;
  L.ml_off = al(slots * 128u * (size_t)d * 4u);
  L.cnt_off = L.ml_off + al(slots * 128u * 8u);
  L.bytes = L.cnt_off + al((size_t)pl.max_units * 4u * 8u);
  return L;
}

// Launch epochs of the balanced split's count words: unique within the
// process (48 bits), from a per-process starting point so that words left in
// reused memory by another process are not taken for this one's.
unsigned long long next_epoch() {
  static std::atomic<unsigned long long> next{[] {
    unsigned long long x = (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
    static int anchor = 0;
    x ^= (unsigned long long)reinterpret_cast<uintptr_t>(&anchor) * 0x9E3779B97F4A7C15ull;
    return x;
  }()};
  return next.fetch_add(1ull, std::memory_order_relaxed) & ((1ull << 48) - 1ull);
}

// Split count when the caller leaves it to the library: only when the units
// fill less than half of the resident CTAs, the S in [2, 16] that minimises
// the waves of work items per split (ceil(units S / slots) / S) plus a small
// per-split cost for the partials and the merge.
int choose_splits(int units, int slots) {
  if (units <= 0 || 2 * units >= slots) return 1;
  int best = 1;
  double best_cost = 1.0;
  for (int S = 2; S <= kMaxSplits; ++S) {
    const double waves = std::ceil((double)units * S / slots);
    const double cost = waves / S + 0.01 * S;
    if (cost < best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

CfgKey cfg_key(int d, int total_q, int max_seqlen_q, int Hq, int G, int window, int dtype) {
  return CfgKey{d, pow2_bucket(max_seqlen_q > 0 ? max_seqlen_q : total_q), Hq, G,
                window > 0 ? 1 : 0, dtype};
}

// Plan for an explicit variant (block_n > 0, q_tiles > 0) or the cache's
// choice (0, 0).
int make_plan_bn(int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
                 int window, int force_bn, int force_qt, Plan* pl);

int make_plan(int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
              int window, Plan* pl) {
  return make_plan_bn(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, 0, 0, pl);
}

int make_plan_bn(int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
                 int window, int force_bn, int force_qt, Plan* pl) {
  if (num_seqs < 0 || total_q < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0)
    return GQA_ERR_INVALID;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return GQA_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return GQA_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G > 128 || 128 % G != 0) return GQA_ERR_UNSUPPORTED;
  // Calls with more sequences run as launches over groups of kMaxSeqs.
  const int seqs_per_launch = num_seqs < kMaxSeqs ? num_seqs : kMaxSeqs;
  pl->groups = num_seqs > kMaxSeqs ? (num_seqs + kMaxSeqs - 1) / kMaxSeqs : 1;
  DeviceInfo di;
  const bool have_dev = device_info(&di) == GQA_OK;
  int bn = force_bn, qt = force_qt;
  bool qt_pinned = force_qt != 0;
  if (bn == 0 || qt == 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    const CfgKey key = cfg_key(d, total_q, max_seqlen_q, Hq, G, window, dtype);
    auto itr = g_cfg_cache.find(key);
    if (itr == g_cfg_cache.end()) itr = g_cfg_cache.emplace(key, default_config(d, window > 0)).first;
    if (bn == 0) bn = g_forced_block_n != 0 ? g_forced_block_n : itr->second.block_n;
    if (qt == 0) {
      qt_pinned = g_forced_q_tiles != 0;
      qt = qt_pinned ? g_forced_q_tiles : itr->second.q_tiles;
    }
  }
  // A cached query-tile count that the tile size has no kernel for falls back
  // to one tile per unit; a pinned one is declined.
  if (!kernel_shape(d, bn, qt, &pl->shape) &&
      (qt_pinned || !kernel_shape(d, bn, 1, &pl->shape)))
    return GQA_ERR_UNSUPPORTED;
  pl->G = G;
  pl->rows = 128 / G;
  pl->unit_rows = pl->shape.q_tiles * pl->rows;
  const long long max_units =  // per launch
      (long long)Hkv * ((total_q + pl->unit_rows - 1) / pl->unit_rows + (long long)seqs_per_launch);
  if (max_units > (1ll << 30) || max_units * pl->groups > (1ll << 30)) return GQA_ERR_UNSUPPORTED;
  pl->max_units = (int)max_units;
  const int by_tmem = 512 / pl->shape.tmem_cols;
  int by_smem = pl->shape.min_blocks;
  if (have_dev && di.smem_per_sm > 0) by_smem = di.smem_per_sm / (int)(pl->shape.smem + 1024);
  int cps = by_tmem < by_smem ? by_tmem : by_smem;
  if (cps > pl->shape.min_blocks) cps = pl->shape.min_blocks;
  if (cps < 1) cps = 1;
  pl->ctas_per_sm = cps;
  pl->smem_launch = pl->shape.smem;
  if (have_dev && di.smem_per_sm > 0) {
    // Request enough that a (cps+1)-th CTA cannot fit next to the others.
    const unsigned pad = (unsigned)(di.smem_per_sm / (cps + 1)) + 1u;
    if (pad > pl->smem_launch) pl->smem_launch = pad;
  }
  const int sms = have_dev ? di.sms : 152;
  pl->slots = sms * cps;
  long long grid = (long long)sms * cps;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  pl->grid = (int)grid;
  return GQA_OK;
}

// Encodes a tensor map on a cache miss.  Calls that reuse buffers (layers of
// a model, benchmark loops, graph capture) hit a small direct-mapped cache
// keyed on everything the map encodes, which saves the driver call.
struct MapKey {
  const void* base;
  int dtype, d, heads, rows, box_heads, box_rows;
  bool operator==(const MapKey& o) const {
    return base == o.base && dtype == o.dtype && d == o.d && heads == o.heads && rows == o.rows &&
           box_heads == o.box_heads && box_rows == o.box_rows;
  }
};
struct MapSlot {
  MapKey key;
  CUtensorMap map;
  bool used = false;
};
constexpr int kMapSlots = 64;
MapSlot g_map_cache[kMapSlots];
std::mutex g_map_mu;

int encode_map_uncached(CUtensorMap* m, const void* base, int dtype, int d, int heads, int rows,
                        int box_heads, int box_rows);

int encode_map(CUtensorMap* m, const void* base, int dtype, int d, int heads, int rows,
               int box_heads, int box_rows) {
  const MapKey key{base, dtype, d, heads, rows, box_heads, box_rows};
  const uint64_t h = (reinterpret_cast<uintptr_t>(base) >> 8) * 0x9E3779B97F4A7C15ull ^
                     ((uint64_t)rows * 31u + (uint64_t)heads * 7u + (uint64_t)box_rows);
  MapSlot& slot = g_map_cache[(h >> 32) % kMapSlots];
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (slot.used && slot.key == key) {
      *m = slot.map;
      return GQA_OK;
    }
  }
  const int rc = encode_map_uncached(m, base, dtype, d, heads, rows, box_heads, box_rows);
  if (rc == GQA_OK) {
    std::lock_guard<std::mutex> lk(g_map_mu);
    slot.key = key;
    slot.map = *m;
    slot.used = true;
  }
  return rc;
}

int encode_map_uncached(CUtensorMap* m, const void* base, int dtype, int d, int heads, int rows,
                        int box_heads, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return GQA_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2u, (cuuint64_t)heads * d * 2u};
  const cuuint32_t box[3] = {64u, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = fn(m,
                        dtype == GQA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GQA_OK : GQA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Encodes the tensor maps and launches one planned kernel on `stream`.
int launch_planned(const Plan& pl, const void* q, const void* k, const void* v,
                   const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                   const int32_t* kv_indptr, int num_seqs, int total_q, int total_kv, int Hq,
                   int Hkv, int d, int dtype, float scale, int window, const float* sinks,
                   int smooth_softmax, void* out, float* lse, void* stream, int32_t* unit_log,
                   const SplitArgs& sp = SplitArgs(), const KvPaging& pg = KvPaging(),
                   int first_seq = 0, const MaskArgs& mk = MaskArgs()) {
  DeviceInfo di;
  if (device_info(&di) != GQA_OK) return GQA_ERR_CUDA;

  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  const bool paged = pg.indices != nullptr;
  const int bn = pl.shape.block_n;
  // K/V rows the maps cover and rows per box: the pool's page slots in boxes
  // of min(BN, page_size) rows, or the contiguous rows in boxes of BN.
  const int kv_rows = paged ? pg.num_pages * pg.page_size : total_kv;
  const int kv_box = paged ? (pg.page_size < bn ? pg.page_size : bn) : bn;
  int rc = encode_map(&p.tmap_q, q, dtype, d, Hq, total_q, pl.G, pl.rows);
  if (rc == GQA_OK) rc = encode_map(&p.tmap_k, k, dtype, d, Hkv, kv_rows, 1, kv_box);
  if (rc == GQA_OK) rc = encode_map(&p.tmap_v, v, dtype, d, Hkv, kv_rows, 1, kv_box);
  if (rc == GQA_OK) rc = encode_map(&p.tmap_o, out, dtype, d, Hq, total_q, pl.G, pl.rows);
  if (rc != GQA_OK) return rc;
  p.cu_seqlens_q = cu_seqlens_q;
  p.prefix_lens = prefix_lens;
  p.kv_indptr = kv_indptr;
  p.sinks = sinks;
  p.out = out;
  p.lse = lse;
  p.unit_log = unit_log;
  p.status = di.status;
  p.num_seqs = num_seqs;
  p.first_seq = first_seq;
  p.total_q = total_q;
  p.total_kv = total_kv;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = pl.G;
  p.rows = pl.rows;
  p.window = window > 0 ? window : 0;
  p.smooth = smooth_softmax != 0 ? 1 : 0;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = timeout_ns();
  p.kv_page_indices = pg.indices;
  p.page_size = pg.page_size;
  p.num_pages = pg.num_pages;
  p.page_rows = kv_box;
  p.custom_mask = mk.custom_mask;
  p.mask_indptr = mk.mask_indptr;
  p.total_mask_words = mk.total_words;
  p.num_splits = sp.num_splits > 1 ? sp.num_splits : 1;
  p.part_o = sp.part_o;
  p.part_ml = sp.part_ml;
  p.part_hdr = sp.part_hdr;
  p.sk_count = sp.sk_count;
  p.epoch = sp.balanced ? next_epoch() : 0ull;
  p.metadata_ready = (t_call_flags & GQA_FLAG_METADATA_READY) ? 1 : 0;
  int grid = pl.grid;
  if (p.num_splits > 1) {  // more work items than units: fill the resident slots
    const long long items = (long long)pl.max_units * p.num_splits;
    grid = (int)(items < pl.slots ? items : pl.slots);
  }
  if (sp.balanced) grid = pl.slots;  // one share per resident CTA
  const bool win = p.window > 0;
  const bool bf16 = dtype == GQA_BF16;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (mk.custom_mask != nullptr)
    e = launch_mask(p, pl.shape, d, win, bf16, grid, pl.smem_launch, st);
  else if (paged)
    e = launch_paged(p, pl.shape, d, win, bf16, grid, pl.smem_launch, st);
  else if (sp.balanced)
    e = launch_balanced(p, pl.shape, d, win, bf16, grid, pl.smem_launch, st);
  else if (p.num_splits > 1)
    e = launch_split(p, pl.shape, d, win, bf16, grid, pl.smem_launch, st);
  else if (d == 64)
    e = launch_d64(p, pl.shape, win, bf16, grid, pl.smem_launch, st);
  else if (d == 128)
    e = launch_d128(p, pl.shape, win, bf16, grid, pl.smem_launch, st);
  else
    e = launch_d256(p, pl.shape, win, bf16, grid, pl.smem_launch, st);
  if (e == cudaSuccess && p.num_splits > 1)
    e = launch_merge(p, d, bf16, pl.shape.q_tiles * 128, pl.max_units, st);
  if (debug_flag())
    std::fprintf(stderr,
                 "[gqa_prefill] B=%d total_q=%d total_kv=%d Hq=%d Hkv=%d d=%d %s window=%d "
                 "sink=%s block_n=%d q_tiles=%d stages=%d grid=%d (%d/SM) max_units=%d%s -> %s\n",
                 num_seqs, total_q, total_kv, Hq, Hkv, d, bf16 ? "bf16" : "f16", p.window,
                 sinks ? "head" : (p.smooth ? "smooth" : "none"), pl.shape.block_n,
                 pl.shape.q_tiles, pl.shape.kv_stages, grid, pl.ctas_per_sm, pl.max_units,
                 sp.balanced ? " balanced" : "",
                 e == cudaSuccess ? "launched" : cudaGetErrorString(e));
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// Launches a planned call group by group: group i takes sequences
// [i kMaxSeqs, (i+1) kMaxSeqs) through metadata pointers offset to its first
// sequence (row indices stay absolute), and its unit records start at record
// i * max_units.  Launches follow each other in stream order, so split-KV
// groups reuse one workspace.
int launch_groups(const Plan& pl, const void* q, const void* k, const void* v,
                  const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                  const int32_t* kv_indptr, int num_seqs, int total_q, int total_kv, int Hq,
                  int Hkv, int d, int dtype, float scale, int window, const float* sinks,
                  int smooth_softmax, void* out, float* lse, void* stream, int32_t* unit_log,
                  const SplitArgs& sp = SplitArgs(), const KvPaging& pg = KvPaging(),
                  const MaskArgs& mk = MaskArgs()) {
  for (int gi = 0; gi < pl.groups; ++gi) {
    const int b0 = gi * kMaxSeqs;
    const int nb = num_seqs - b0 < kMaxSeqs ? num_seqs - b0 : kMaxSeqs;
    int32_t* log = unit_log != nullptr ? unit_log + 8 * (size_t)gi * pl.max_units : nullptr;
    MaskArgs mg = mk;
    if (mg.mask_indptr != nullptr) mg.mask_indptr += b0;
    const int rc = launch_planned(pl, q, k, v, cu_seqlens_q + b0, prefix_lens + b0,
                                  kv_indptr + b0, nb, total_q, total_kv, Hq, Hkv, d, dtype, scale,
                                  window, sinks, smooth_softmax, out, lse, stream, log, sp, pg, b0,
                                  mg);
    if (rc != GQA_OK) return rc;
  }
  return GQA_OK;
}

int tune_mode() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_tune_mode < 0) g_tune_mode = env_flag("GQA_PREFILL_TUNE") ? 1 : 0;
  return g_tune_mode;
}

// The configuration cache's sweep ([HIPEP] config-cache commit: one sweep per
// key and process; tuning launches omit the sink, which cannot reorder the
// candidates): times every candidate variant (key-tile size x query tiles per
// unit) on the caller's stream and keeps the fastest.  Synchronises the
// stream; skipped while capturing.
int tune_key(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
             const int32_t* prefix_lens, const int32_t* kv_indptr, int num_seqs, int total_q,
             int total_kv, int max_seqlen_q, int Hq, int Hkv, int d, int dtype, float scale,
             int window, void* out, float* lse, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return GQA_OK;
  const int cands[5][2] = {{64, 1}, {96, 1}, {128, 1}, {64, 2}, {128, 2}};
  int best = 0, best_qt = 0;
  float best_ms = 0.f;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return GQA_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return GQA_ERR_CUDA;
  }
  int rc = GQA_OK;
  for (const auto& cand : cands) {
    const int bn = cand[0], qt = cand[1];
    Plan pl;
    KernelShape ks;
    if (!kernel_shape(d, bn, qt, &ks)) continue;
    rc = make_plan_bn(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, bn, qt, &pl);
    if (rc != GQA_OK) break;
    auto once = [&]() {
      return launch_groups(pl, q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q,
                           total_kv, Hq, Hkv, d, dtype, scale, window, nullptr, 0, out, lse,
                           stream, nullptr);
    };
    if ((rc = once()) != GQA_OK) break;
    cudaEventRecord(e0, st);
    for (int i = 0; i < 3 && rc == GQA_OK; ++i) rc = once();
    cudaEventRecord(e1, st);
    if (rc != GQA_OK || cudaEventSynchronize(e1) != cudaSuccess) {
      rc = rc != GQA_OK ? rc : GQA_ERR_CUDA;
      break;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    ms /= 3.f;
    if (env_flag("GQA_PREFILL_TUNE_DEBUG"))
      std::fprintf(stderr,
                   "[gqa_prefill tune] d=%d sq<=%d Hq=%d G=%d windowed=%d block_n=%d q_tiles=%d: "
                   "%.4f ms\n",
                   d, pow2_bucket(max_seqlen_q > 0 ? max_seqlen_q : total_q), Hq, Hq / Hkv,
                   window > 0 ? 1 : 0, bn, qt, ms);
    if (best == 0 || ms < best_ms) {
      best = bn;
      best_qt = qt;
      best_ms = ms;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (rc != GQA_OK) return rc;
  if (best != 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_cfg_cache[cfg_key(d, total_q, max_seqlen_q, Hq, Hq / Hkv, window, dtype)] =
        CfgEntry{best, best_qt, true};
  }
  return GQA_OK;
}

// Split count for a plan: `req` 0 = the library's choice, else 1..kMaxSplits.
// The unit count is estimated from below without reading device metadata:
// the tokens packed into units, and at least one unit per sequence and KV head
// (a decode step of many one-token sequences has many units).
int splits_for(const Plan& pl, int num_seqs, int total_q, int Hkv, int req) {
  if (req != 0) return req;
  const long long packed = (total_q + pl.unit_rows - 1) / pl.unit_rows;
  const long long units = (long long)Hkv * (packed > num_seqs ? packed : num_seqs);
  return choose_splits(units > (1ll << 30) ? (1 << 30) : (int)units, pl.slots);
}

// The plan of a split-KV call: the cached or forced plan when a split
// instantiation exists for its shape, else one query tile per unit with the
// key tile the split instantiations have for d.
int plan_split(int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
               int window, int req, Plan* pl, int* S) {
  int rc = make_plan(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, pl);
  if (rc != GQA_OK) return rc;
  *S = splits_for(*pl, num_seqs, total_q, Hkv, req);
  if (*S > 1 && !split_shape(d, pl->shape.block_n, pl->shape.q_tiles)) {
    const int bn = split_shape(d, pl->shape.block_n, 1) ? pl->shape.block_n : (d == 64 ? 128 : 64);
    rc = make_plan_bn(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, bn, 1, pl);
    if (rc != GQA_OK) return rc;
    *S = splits_for(*pl, num_seqs, total_q, Hkv, req);
  }
  return GQA_OK;
}

// The plan of a balanced-split call: as plan_split's, and declined when one
// launch's query tiles could overflow the shared-memory scratch the kernel
// computes the shares in (its K/V rings, one word per query tile plus one).
int plan_balanced(int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
                  int window, Plan* pl) {
  int rc = make_plan(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, pl);
  if (rc != GQA_OK) return rc;
  if (!split_shape(d, pl->shape.block_n, pl->shape.q_tiles)) {
    const int bn = split_shape(d, pl->shape.block_n, 1) ? pl->shape.block_n : (d == 64 ? 128 : 64);
    rc = make_plan_bn(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, bn, 1, pl);
    if (rc != GQA_OK) return rc;
  }
  const long long seqs = num_seqs < kMaxSeqs ? num_seqs : kMaxSeqs;
  const long long qtiles = (total_q + pl->unit_rows - 1) / pl->unit_rows + seqs;
  const long long ring_words = 2ll * pl->shape.kv_stages * pl->shape.block_n * d * 2 / 4;
  if (qtiles + 1 > ring_words) return GQA_ERR_UNSUPPORTED;
  // The kernel's share arithmetic is 32-bit for grids below 46341 CTAs.
  if (pl->slots >= 46341) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

int run(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
        const int32_t* prefix_lens, const int32_t* kv_indptr, int num_seqs, int total_q,
        int total_kv, int max_seqlen_q, int Hq, int Hkv, int d, int dtype, float scale,
        int window, const float* sinks, int smooth_softmax, void* out, float* lse, void* stream,
        int32_t* unit_log, int num_splits = 1, void* workspace = nullptr,
        size_t workspace_bytes = 0, ScratchFn scratch = nullptr) {
  if (num_splits < kBalanced || num_splits > kMaxSplits) return GQA_ERR_INVALID;
  if (num_seqs < 0 || total_q < 0 || total_kv < 0 || max_seqlen_q < 0) return GQA_ERR_INVALID;
  if (Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return GQA_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return GQA_ERR_INVALID;
  if (sinks != nullptr && smooth_softmax != 0) return GQA_ERR_INVALID;
  if (num_seqs == 0 || total_q == 0) return GQA_OK;  // no work, no launch
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
      cu_seqlens_q == nullptr || prefix_lens == nullptr || kv_indptr == nullptr)
    return GQA_ERR_INVALID;
  if (total_kv == 0) return GQA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return GQA_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return GQA_ERR_UNSUPPORTED;
  if (tune_mode() == 1) {
    bool need = false;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if (g_forced_block_n == 0 && g_forced_q_tiles == 0) {
        auto itr = g_cfg_cache.find(cfg_key(d, total_q, max_seqlen_q, Hq, Hq / Hkv, window, dtype));
        need = itr == g_cfg_cache.end() || !itr->second.tuned;
      }
    }
    if (need) {
      const int rc = tune_key(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q,
                              total_kv, max_seqlen_q, Hq, Hkv, d, dtype, scale, window, out, lse,
                              stream);
      if (rc != GQA_OK) return rc;
    }
  }
  Plan pl;
  SplitArgs sp;
  const int rc =
      (num_splits == 1)
          ? make_plan(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, &pl)
      : (num_splits == kBalanced)
          ? plan_balanced(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, &pl)
          : plan_split(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, num_splits,
                       &pl, &sp.num_splits);
  if (rc != GQA_OK) return rc;
  if (num_splits == kBalanced) {
    // The kernel counts key tiles in 32 bits: a unit walks at most
    // ceil(total_kv / block_n) + 1 tiles.
    const long long unit_tiles = (total_kv + pl.shape.block_n - 1) / pl.shape.block_n + 1;
    if ((long long)pl.max_units * unit_tiles >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
    const BalancedLayout L = balanced_layout(pl, d);
    if (workspace == nullptr && scratch != nullptr) {
      const int rs = scratch(L.bytes, &workspace, &workspace_bytes);
      if (rs != GQA_OK) return rs;
    }
    if (workspace == nullptr || workspace_bytes < L.bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return GQA_ERR_INVALID;
    char* base = static_cast<char*>(workspace);
    sp.balanced = true;
    sp.part_o = reinterpret_cast<float*>(base + L.o_off);
    sp.part_ml = reinterpret_cast<float*>(base + L.ml_off);
    sp.sk_count = reinterpret_cast<unsigned long long*>(base + L.cnt_off);
  } else if (sp.num_splits > 1) {
    const SplitLayout L = split_layout(pl, d, sp.num_splits);
    if (workspace == nullptr && scratch != nullptr) {
      // The library's own scratch, checked against this very plan's layout.
      const int rs = scratch(L.bytes, &workspace, &workspace_bytes);
      if (rs != GQA_OK) return rs;
    }
    if (workspace == nullptr || workspace_bytes < L.bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return GQA_ERR_INVALID;
    char* base = static_cast<char*>(workspace);
    sp.part_o = reinterpret_cast<float*>(base + L.o_off);
    sp.part_ml = reinterpret_cast<float*>(base + L.ml_off);
    sp.part_hdr = reinterpret_cast<int32_t*>(base + L.hdr_off);
  }
  return launch_groups(pl, q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q,
                       total_kv, Hq, Hkv, d, dtype, scale, window, sinks, smooth_softmax, out, lse,
                       stream, unit_log, sp);
}

// Paged KV: the same validation as run(), the pool geometry checks, and a
// plan whose key tile has a paged instantiation and tiles the pages.
int run_paged(const void* q, const void* k_pages, const void* v_pages,
              const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
              const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
              int num_page_entries, int page_size, int num_pages, int num_seqs, int total_q,
              int max_seqlen_q, int Hq, int Hkv, int d, int dtype, float scale, int window,
              const float* sinks, int smooth_softmax, void* out, float* lse, void* stream) {
  if (num_seqs < 0 || total_q < 0 || num_page_entries < 0 || max_seqlen_q < 0)
    return GQA_ERR_INVALID;
  if (Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return GQA_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return GQA_ERR_INVALID;
  if (sinks != nullptr && smooth_softmax != 0) return GQA_ERR_INVALID;
  if (page_size < 8 || page_size % 8 != 0 || num_pages <= 0 ||
      (long long)num_pages * page_size >= (1ll << 31))
    return GQA_ERR_INVALID;
  if (num_seqs == 0 || total_q == 0) return GQA_OK;  // no work, no launch
  if (q == nullptr || k_pages == nullptr || v_pages == nullptr || out == nullptr ||
      cu_seqlens_q == nullptr || prefix_lens == nullptr || kv_page_indptr == nullptr ||
      kv_page_indices == nullptr || num_page_entries == 0)
    return GQA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return GQA_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return GQA_ERR_UNSUPPORTED;
  Plan pl;
  int rc = make_plan(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, &pl);
  if (rc != GQA_OK) return rc;
  auto tiles_pages = [&](int bn) { return page_size % bn == 0 || bn % page_size == 0; };
  if (!split_shape(d, pl.shape.block_n, pl.shape.q_tiles) || !tiles_pages(pl.shape.block_n)) {
    int bn = 0;
    for (int cand : {128, 64})
      if (bn == 0 && split_shape(d, cand, 1) && tiles_pages(cand)) bn = cand;
    if (bn == 0) return GQA_ERR_UNSUPPORTED;
    rc = make_plan_bn(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, bn, 1, &pl);
    if (rc != GQA_OK) return rc;
  }
  KvPaging pg;
  pg.indices = kv_page_indices;
  pg.page_size = page_size;
  pg.num_pages = num_pages;
  return launch_groups(pl, q, k_pages, v_pages, cu_seqlens_q, prefix_lens, kv_page_indptr,
                       num_seqs, total_q, num_page_entries, Hq, Hkv, d, dtype, scale, window,
                       sinks, smooth_softmax, out, lse, stream, nullptr, SplitArgs(), pg);
}

// Custom mask: the same validation as run(), the mask arguments, and a plan
// whose shape has a custom-mask instantiation.
int run_masked(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
               const int32_t* prefix_lens, const int32_t* kv_indptr, int num_seqs, int total_q,
               int total_kv, int max_seqlen_q, int Hq, int Hkv, int d, int dtype, float scale,
               int window, const float* sinks, int smooth_softmax, const uint32_t* custom_mask,
               const int32_t* mask_indptr, long long total_mask_words, void* out, float* lse,
               void* stream) {
  if (num_seqs < 0 || total_q < 0 || total_kv < 0 || max_seqlen_q < 0 || total_mask_words < 0)
    return GQA_ERR_INVALID;
  if (Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return GQA_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return GQA_ERR_INVALID;
  if (sinks != nullptr && smooth_softmax != 0) return GQA_ERR_INVALID;
  if (num_seqs == 0 || total_q == 0) return GQA_OK;  // no work, no launch
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
      cu_seqlens_q == nullptr || prefix_lens == nullptr || kv_indptr == nullptr ||
      custom_mask == nullptr || mask_indptr == nullptr)
    return GQA_ERR_INVALID;
  if (total_kv == 0) return GQA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(custom_mask) & 3u) != 0)
    return GQA_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return GQA_ERR_UNSUPPORTED;
  Plan pl;
  int rc = make_plan(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, &pl);
  if (rc != GQA_OK) return rc;
  if (!split_shape(d, pl.shape.block_n, pl.shape.q_tiles)) {
    const int bn = split_shape(d, pl.shape.block_n, 1) ? pl.shape.block_n : (d == 64 ? 128 : 64);
    rc = make_plan_bn(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, bn, 1, &pl);
    if (rc != GQA_OK) return rc;
  }
  MaskArgs mk;
  mk.custom_mask = custom_mask;
  mk.mask_indptr = mask_indptr;
  mk.total_words = total_mask_words;
  return launch_groups(pl, q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q,
                       total_kv, Hq, Hkv, d, dtype, scale, window, sinks, smooth_softmax, out, lse,
                       stream, nullptr, SplitArgs(), KvPaging(), mk);
}

}  // namespace

int run_splitkv_scratch(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                        const int32_t* prefix_lens, const int32_t* kv_indptr, int num_seqs,
                        int total_q, int total_kv, int max_seqlen_q, int Hq, int Hkv, int d,
                        int dtype, float scale, int window, const float* sinks,
                        int smooth_softmax, void* out, float* lse, int num_splits, void* stream,
                        ScratchFn scratch) {
  return run(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q, total_kv,
             max_seqlen_q, Hq, Hkv, d, dtype, scale, window, sinks, smooth_softmax, out, lse,
             stream, nullptr, num_splits, nullptr, 0, scratch);
}

bool kernel_shape(int d, int block_n, int q_tiles, KernelShape* out) {
  KernelShape s;
  s.block_n = block_n;
  s.q_tiles = q_tiles;
  const int bn = block_n;
  if (q_tiles == 1) {
    if (d == 64 && bn == 128) { s.kv_stages = 2; s.min_blocks = 2; }
    else if (d == 64 && bn == 64) { s.kv_stages = 4; s.min_blocks = 2; }
    else if (d == 64 && bn == 96) { s.kv_stages = 2; s.min_blocks = 2; }
    else if (d == 128 && bn == 64) { s.kv_stages = 2; s.min_blocks = 2; }
    else if (d == 128 && bn == 128) { s.kv_stages = 2; s.min_blocks = 1; }
    else if (d == 256 && bn == 64) { s.kv_stages = 2; s.min_blocks = 1; }
    else return false;
  } else if (q_tiles == 2) {
    if (d == 64 && bn == 128) { s.kv_stages = 4; s.min_blocks = 1; }
    else if (d == 64 && bn == 64) { s.kv_stages = 8; s.min_blocks = 1; }
    else if (d == 128 && bn == 64) { s.kv_stages = 4; s.min_blocks = 1; }
    else return false;
  } else {
    return false;
  }
  s.smem = smem_bytes_for(d, block_n, s.kv_stages, q_tiles);
  s.tmem_cols = tmem_alloc_for(d, block_n, q_tiles);
  *out = s;
  return true;
}

}  // namespace gqa

extern "C" {

int gqa_flash_prefill(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                      const int32_t* prefix_lens, const int32_t* kv_indptr, int num_seqs,
                      int total_q, int total_kv, int max_seqlen_q, int Hq, int Hkv, int d,
                      int dtype, float scale, int window, const float* sinks, int smooth_softmax,
                      void* out, float* lse, void* stream) {
  return gqa::run(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q, total_kv,
                  max_seqlen_q, Hq, Hkv, d, dtype, scale, window, sinks, smooth_softmax, out, lse,
                  stream, nullptr);
}

int gqa_flash_prefill_debug(const void* q, const void* k, const void* v,
                            const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                            const int32_t* kv_indptr, int num_seqs, int total_q, int total_kv,
                            int max_seqlen_q, int Hq, int Hkv, int d, int dtype, float scale,
                            int window, const float* sinks, int smooth_softmax, void* out,
                            float* lse, void* stream, int32_t* unit_log) {
  if (unit_log == nullptr) return GQA_ERR_INVALID;
  return gqa::run(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q, total_kv,
                  max_seqlen_q, Hq, Hkv, d, dtype, scale, window, sinks, smooth_softmax, out, lse,
                  stream, unit_log);
}

int gqa_flash_prefill_splitkv(const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                              const int32_t* kv_indptr, int num_seqs, int total_q, int total_kv,
                              int max_seqlen_q, int Hq, int Hkv, int d, int dtype, float scale,
                              int window, const float* sinks, int smooth_softmax, void* out,
                              float* lse, int num_splits, void* workspace, size_t workspace_bytes,
                              void* stream) {
  return gqa::run(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q, total_kv,
                  max_seqlen_q, Hq, Hkv, d, dtype, scale, window, sinks, smooth_softmax, out, lse,
                  stream, nullptr, num_splits, workspace, workspace_bytes);
}

int gqa_flash_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                            const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                            const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
                            int num_page_entries, int page_size, int num_pages, int num_seqs,
                            int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
                            float scale, int window, const float* sinks, int smooth_softmax,
                            void* out, float* lse, void* stream) {
  return gqa::run_paged(q, k_pages, v_pages, cu_seqlens_q, prefix_lens, kv_page_indptr,
                        kv_page_indices, num_page_entries, page_size, num_pages, num_seqs,
                        total_q, max_seqlen_q, Hq, Hkv, d, dtype, scale, window, sinks,
                        smooth_softmax, out, lse, stream);
}

int gqa_flash_prefill_masked(const void* q, const void* k, const void* v,
                             const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                             const int32_t* kv_indptr, int num_seqs, int total_q, int total_kv,
                             int max_seqlen_q, int Hq, int Hkv, int d, int dtype, float scale,
                             int window, const float* sinks, int smooth_softmax,
                             const uint32_t* custom_mask, const int32_t* mask_indptr,
                             long long total_mask_words, void* out, float* lse, void* stream) {
  return gqa::run_masked(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs, total_q,
                         total_kv, max_seqlen_q, Hq, Hkv, d, dtype, scale, window, sinks,
                         smooth_softmax, custom_mask, mask_indptr, total_mask_words, out, lse,
                         stream);
}

int gqa_prefill_splitkv_workspace(int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv,
                                  int d, int dtype, int window, int num_splits, int* splits_used,
                                  size_t* bytes) {
  if (splits_used == nullptr || bytes == nullptr) return GQA_ERR_INVALID;
  if (num_splits < gqa::kBalanced || num_splits > gqa::kMaxSplits) return GQA_ERR_INVALID;
  gqa::Plan pl;
  if (num_splits == gqa::kBalanced) {
    const int rb = gqa::plan_balanced(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window,
                                      &pl);
    if (rb != GQA_OK) return rb;
    *splits_used = gqa::kBalanced;
    *bytes = gqa::balanced_layout(pl, d).bytes;
    return GQA_OK;
  }
  int S = 1;
  const int rc = gqa::plan_split(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window,
                                 num_splits, &pl, &S);
  if (rc != GQA_OK) return rc;
  *splits_used = S;
  *bytes = S > 1 ? gqa::split_layout(pl, d, S).bytes : 0;
  return GQA_OK;
}

int gqa_prefill_plan(int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int d,
                     int dtype, int window, gqa_prefill_plan_t* plan) {
  if (plan == nullptr) return GQA_ERR_INVALID;
  gqa::Plan pl;
  const int rc =
      gqa::make_plan(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype, window, &pl);
  if (rc != GQA_OK) return rc;
  plan->rows_per_unit = pl.unit_rows;
  plan->block_n = pl.shape.block_n;
  plan->q_tiles = pl.shape.q_tiles;
  plan->kv_stages = pl.shape.kv_stages;
  plan->ctas_per_sm = pl.ctas_per_sm;
  plan->grid = pl.grid;
  plan->max_units = pl.max_units * pl.groups;  // unit records over all launches
  return GQA_OK;
}

int gqa_prefill_set_tuning(int enable) {
  if (enable != 0 && enable != 1) return GQA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(gqa::g_mu);
  gqa::g_tune_mode = enable;
  return GQA_OK;
}

int gqa_prefill_clear_config_cache(void) {
  std::lock_guard<std::mutex> lk(gqa::g_mu);
  gqa::g_cfg_cache.clear();
  return GQA_OK;
}

int gqa_prefill_config_block_n(int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
                               int window, int* block_n, int* q_tiles, int* tuned) {
  if (block_n == nullptr || tuned == nullptr || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return GQA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(gqa::g_mu);
  auto itr = gqa::g_cfg_cache.find(
      gqa::cfg_key(d, total_q, max_seqlen_q, Hq, Hq / Hkv, window, dtype));
  if (itr == gqa::g_cfg_cache.end()) {
    *block_n = 0;
    *tuned = 0;
    if (q_tiles != nullptr) *q_tiles = 0;
  } else {
    *block_n = itr->second.block_n;
    *tuned = itr->second.tuned ? 1 : 0;
    if (q_tiles != nullptr) *q_tiles = itr->second.q_tiles;
  }
  return GQA_OK;
}

int gqa_prefill_selftest_timeout(int timeout_ms, void* stream, int* status) {
  if (status == nullptr || timeout_ms <= 0 || timeout_ms > 10000) return GQA_ERR_INVALID;
  gqa::DeviceInfo di;
  if (gqa::device_info(&di) != GQA_OK) return GQA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gqa::selftest_wait_kernel<<<1, 32, 0, st>>>(di.status,
                                              (unsigned long long)timeout_ms * 1000000ull);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GQA_ERR_CUDA;
  return gqa_prefill_get_device_status(status);
}

int gqa_prefill_force_block_n(int block_n) {
  if (block_n != 0 && block_n != 64 && block_n != 96 && block_n != 128) return GQA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(gqa::g_mu);
  gqa::g_forced_block_n = block_n;
  return GQA_OK;
}

int gqa_prefill_force_q_tiles(int q_tiles) {
  if (q_tiles < 0 || q_tiles > 2) return GQA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(gqa::g_mu);
  gqa::g_forced_q_tiles = q_tiles;
  return GQA_OK;
}

int gqa_prefill_get_device_status(int* status) {
  if (status == nullptr) return GQA_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, gqa::g_device_status, sizeof(v)) != cudaSuccess) return GQA_ERR_CUDA;
  if (cudaMemcpyToSymbol(gqa::g_device_status, &zero, sizeof(zero)) != cudaSuccess)
    return GQA_ERR_CUDA;
  *status = (int)v;
  return GQA_OK;
}

int gqa_prefill_get_stream_status(void* stream, int* status) {
  if (status == nullptr) return GQA_ERR_INVALID;
  gqa::DeviceInfo di;
  if (gqa::device_info(&di) != GQA_OK) return GQA_ERR_CUDA;
  static std::atomic<unsigned> next_slot{0};
  const unsigned slot = next_slot.fetch_add(1u, std::memory_order_relaxed) % gqa::kStatusSlots;
  void* snap_base = nullptr;
  if (cudaGetSymbolAddress(&snap_base, gqa::g_status_snapshot) != cudaSuccess) return GQA_ERR_CUDA;
  unsigned int* snap = static_cast<unsigned int*>(snap_base) + slot;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gqa::status_take_kernel<<<1, 1, 0, st>>>(di.status, snap);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyAsync(&v, snap, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GQA_ERR_CUDA;
  *status = (int)v;
  return GQA_OK;
}

int gqa_prefill_set_call_flags(unsigned int flags) {
  if ((flags & ~GQA_FLAG_METADATA_READY) != 0u) return GQA_ERR_INVALID;
  gqa::t_call_flags = flags;
  return GQA_OK;
}

unsigned int gqa_prefill_get_call_flags(void) { return gqa::t_call_flags; }

const char* gqa_prefill_status_string(int code) {
  switch (code) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported shape (declined)";
    case GQA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* gqa_prefill_version(void) { return "0.1.0"; }

}  // extern "C"
