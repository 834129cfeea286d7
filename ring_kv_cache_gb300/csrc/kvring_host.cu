// Host side of the kvring C ABI: argument checks, buffer carving, the RoPE
// table, TMA descriptors and kernel launches.  Every entry point only
// enqueues work on the caller's stream; none synchronises except
// kvring_create (which waits for its own upload) and none allocates device
// memory (the caller hands one buffer to kvring_create).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "kvring_internal.cuh"

struct kvring {
  kvring_config cfg;
  kvr::RingDev dev;
  CUtensorMap tmK;
  CUtensorMap tmV;
  int sm_count;
  int qtiles_max;
  int device;        // current at create; every call must run with it current
  bool calibrated;   // host mirror: a calibration has been enqueued
  unsigned long long attn_wait_ns;   // limit of the attention kernel's bounded waits
  int attn_debug_stall;              // test support: the next attention calls time out on purpose
  int attn_debug_guess;              // test support: the attention's position guess is wrong on purpose
};

namespace {

constexpr size_t kAlign = 256;
constexpr unsigned long long kDefaultWaitNs = 1000000000ull;   // one second

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool config_ok(const kvring_config* c) {
  if (!c) return false;
  if (c->num_heads < 1 || c->num_heads > 4096) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->capacity < 1 || c->capacity > (1 << 24)) return false;
  if (c->max_tokens < 1 || c->max_tokens > (1 << 24)) return false;
  if (c->max_position < 1 || c->max_position > (1 << 24)) return false;
  if (c->max_kv_splits < 1 || c->max_kv_splits > 32) return false;
  if (c->attn_precision < 0 || c->attn_precision > 4) return false;
  if (c->pinned_prefix < 0 || c->pinned_prefix >= c->capacity) return false;
  if (c->rope_pairs_t != 0 || c->rope_pairs_y != 0) {   // 3-D RoPE sections, in whole chunks of 8 pairs
    const int half = c->head_dim / 2, t = c->rope_pairs_t, y = c->rope_pairs_y;
    if (t < 8 || y < 0 || t % 8 != 0 || y % 8 != 0 || t + y > half || (half - t - y) % 8 != 0) return false;
  }
  if (!(c->rope_base > 0.0) || !std::isfinite(c->rope_base)) return false;
  return true;
}

struct Plan {
  size_t k, v, slot_pos, scales, state, amax, table, part_o, part_lse, tickets, levels, total;
  int qtiles;
};

Plan plan_for(const kvring_config* c) {
  Plan p{};
  const size_t H = (size_t)c->num_heads, D = (size_t)c->head_dim, C = (size_t)c->capacity;
  p.qtiles = (c->max_tokens + kvr::kTile - 1) / kvr::kTile;
  // split partials go through global memory only beyond 8 splits (up to 8
  // splits merge inside a thread-block cluster)
  const size_t Q = (size_t)p.qtiles, S = c->max_kv_splits > 8 ? (size_t)c->max_kv_splits : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  p.k = take(H * C * D);
  p.v = take(H * C * D);
  p.slot_pos = take(C * 4);
  p.scales = take(4 * H * 4);
  p.state = take(kvr::ST_WORDS_ALLOC * 4);
  p.amax = take(2 * H * 4);
  p.table = take((size_t)c->max_position * D * 4);
  p.part_o = take(S * Q * H * kvr::kTile * D * 4);
  p.part_lse = take(S * Q * H * kvr::kTile * 4);
  p.tickets = take(Q * H * 4);
  p.levels = take(Q * H * 4);
  p.total = off;
  return p;
}

kvring_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVRING_OK : KVRING_ERR_CUDA; }

// The ring's device is the current one (its kernels run on the current
// device, against the ring's memory).
bool on_device(const kvring* r) {
  int cur = -1;
  return cudaGetDevice(&cur) == cudaSuccess && cur == r->device;
}

// Split-KV count for one attention call: the grid has qtiles * H * nsplit
// CTAs of which one fits per SM; pick the split count with the fewest
// "waves x (tiles per CTA + fixed per-CTA cost)".  The fixed cost (prologue,
// epilogue and partial store, about four key/value tiles' time) was
// measured on GB300.
void choose_splits(const kvring* r, int n_q, int* nsplit, int* tiles_per_split) {
  const int ctiles = (r->cfg.capacity + kvr::kTile - 1) / kvr::kTile;
  const int qtiles = (n_q + kvr::kTile - 1) / kvr::kTile;
  const long long per_split = (long long)qtiles * r->cfg.num_heads;
  const int smax = r->cfg.max_kv_splits < ctiles ? r->cfg.max_kv_splits : ctiles;
  double best = 1e300;
  int best_ns = 1, best_tps = ctiles;
  for (int ns = 1; ns <= smax; ++ns) {
    const int tps = (ctiles + ns - 1) / ns;
    const int ns_eff = (ctiles + tps - 1) / tps;
    if (ns_eff != ns) continue;
    const long long ctas = per_split * ns_eff;
    const long long waves = (ctas + r->sm_count - 1) / r->sm_count;
    const double cost = (double)waves * (tps + 4.0) + (ns_eff > 1 ? 0.5 : 0.0);
    if (cost < best - 1e-9) {
      best = cost;
      best_ns = ns_eff;
      best_tps = tps;
    }
  }
  *nsplit = best_ns;
  *tiles_per_split = best_tps;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D map over a [H][C][D] byte cache: tiles of [1][128][D] with the
// swizzle the MMA descriptors expect (row bytes = D); rows past C read 0.
bool make_cache_map(CUtensorMap* m, void* base, int H, int C, int D) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)C, (cuuint64_t)H};
  const cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)C * (cuuint64_t)D};
  const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)kvr::kTile, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult res =
      fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS;
}

// 2-D map over a row-major bf16 matrix [rows][cols]: tiles of box_rows rows
// by 64 columns (128 bytes) with the 128-byte swizzle the MMA descriptors
// expect; rows past the end read 0.
bool make_bf16_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult res = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Which caller buffers kernels of this library that may still be running
// write, per stream.
//
// Every kernel here is launched as a programmatic dependent of the kernel
// before it on its stream.  The attention and the projection let their own
// dependents start only once their wait for their predecessor has returned,
// so after one of them, only that kernel itself may still be running.  The
// writes and delta rotations let theirs start at once, so a kernel after
// them may start while kernels before them still run -- but they write no
// caller buffer.  The attention reads its queries, and the write its frame,
// before its wait -- unless a kernel possibly still in flight writes them.
// So a library kernel that stores into caller buffers (attention output, the
// projection's queries and keys/values, the legacy window, the E4M3 test
// encoder) replaces its stream's record with those ranges; an attention or a
// projection with no such output clears it; a write or delta leaves it as it
// is (it lets older kernels stay in flight and adds nothing to them); and a
// call whose early inputs overlap the record reads them after the wait.  A
// caller kernel that does not use programmatic launch lets its successor
// start only at its end, so it needs no record.  The decision and the launch
// happen under one lock, in launch order, so calls from several threads on
// one stream see the record of the kernels that really precede theirs.
//
// The record also lists the rings that kernels possibly still in flight may
// read or write: a write or delta adds its rings (older kernels may still
// run); an attention or a projection leaves its own ring only (a projection
// that does not write, none); a kernel that lets no dependent start early
// (calibration, legacy upkeep, the test encoder) leaves none.  A single-ring
// write whose ring is not listed does its whole work before its wait.
struct Range {
  const void* p;
  size_t n;
};

struct OutRec {
  cudaStream_t s;
  std::thread::id tid;     // for the per-thread default stream, which each thread has its own of
  uint64_t used;           // LRU stamp; 0 = free entry
  uintptr_t lo[2], hi[2];  // written ranges [lo, hi); empty when lo == hi
  const kvring* touched[KVRING_MAX_BATCH];   // rings a kernel possibly in flight may read or write
  int ntouched;                              // -1: more than fit (every ring counts as listed)
};

constexpr int kOutRecs = 64;
std::mutex g_out_mu;
OutRec g_out[kOutRecs];
uint64_t g_out_clock = 0;
bool g_out_lost = false;   // a record was evicted: a stream without one reads late
long long g_late_reads = 0;

// Under g_out_mu.
OutRec* find_rec(cudaStream_t s, bool create) {
  const std::thread::id tid = s == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id();
  OutRec* oldest = &g_out[0];
  for (OutRec& e : g_out) {
    if (e.used && e.s == s && e.tid == tid) return &e;
    if (e.used < oldest->used) oldest = &e;
  }
  if (!create) return nullptr;
  if (oldest->used) g_out_lost = true;
  oldest->s = s;
  oldest->tid = tid;
  oldest->used = ++g_out_clock;
  oldest->lo[0] = oldest->hi[0] = oldest->lo[1] = oldest->hi[1] = 0;
  oldest->ntouched = 0;
  return oldest;
}

// Under g_out_mu: whether no kernel possibly in flight on s reads or writes
// the ring.
bool ring_idle(cudaStream_t s, const kvring* ring) {
  const OutRec* e = find_rec(s, false);
  if (!e) return !g_out_lost;
  if (e->ntouched < 0) return false;
  for (int i = 0; i < e->ntouched; ++i)
    if (e->touched[i] == ring) return false;
  return true;
}

// Under g_out_mu: whether the last library kernel on s may write any of the
// ranges (a call with these early inputs then reads them after its wait).
bool late_inputs(cudaStream_t s, std::initializer_list<Range> in) {
  const OutRec* e = find_rec(s, false);
  bool late = false;
  if (!e) {
    late = g_out_lost;
  } else {
    for (const Range& r : in) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(r.p), b = a + r.n;
      for (int i = 0; i < 2; ++i)
        if (e->lo[i] < e->hi[i] && a < e->hi[i] && e->lo[i] < b) late = true;
    }
  }
  if (late) ++g_late_reads;
  return late;
}

// Under g_out_mu, after a launch on s succeeded: its kernel is now the last
// one there, writing the given caller ranges (none for most calls).
void note_launch(cudaStream_t s, Range a, Range b, const kvring* touches) {
  OutRec* e = find_rec(s, true);
  e->used = ++g_out_clock;
  const Range rr[2] = {a, b};
  for (int i = 0; i < 2; ++i) {
    e->lo[i] = reinterpret_cast<uintptr_t>(rr[i].p);
    e->hi[i] = rr[i].p ? e->lo[i] + rr[i].n : e->lo[i];
  }
  e->ntouched = 0;
  if (touches) e->touched[e->ntouched++] = touches;
}

// Launches under the lock and records the launch when it succeeded (its
// kernel lets its dependents start only after its own wait, or not early at
// all; `touches`: the ring it reads or writes, if any).
template <typename F>
kvring_status tracked(cudaStream_t s, F launch, Range a = {nullptr, 0}, Range b = {nullptr, 0},
                      const kvring* touches = nullptr) {
  const cudaError_t e = launch();
  if (e == cudaSuccess) note_launch(s, a, b, touches);
  return cuda_status(e);
}

// A launch whose kernel lets its dependents start before its own wait and
// writes no caller buffer: the stream's written ranges stay as they are and
// its rings join the touched list.
template <typename F>
kvring_status passed_through(cudaStream_t s, F launch, kvring* const* rings, int count) {
  const cudaError_t e = launch();
  if (e == cudaSuccess) {
    OutRec* rec = find_rec(s, true);
    rec->used = ++g_out_clock;
    for (int i = 0; i < count && rec->ntouched >= 0; ++i) {
      bool listed = false;
      for (int j = 0; j < rec->ntouched; ++j) listed = listed || rec->touched[j] == rings[i];
      if (listed) continue;
      if (rec->ntouched == KVRING_MAX_BATCH) {
        rec->ntouched = -1;
      } else {
        rec->touched[rec->ntouched++] = rings[i];
      }
    }
  }
  return cuda_status(e);
}

}  // namespace

extern "C" {

size_t kvring_required_bytes(const kvring_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return plan_for(cfg).total;
}

kvring_status kvring_create(const kvring_config* cfg, void* dev_buf, size_t bytes, void* stream,
                            kvring_t** out) {
  if (!out) return KVRING_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config_ok(cfg) || !dev_buf || !aligned(dev_buf, kAlign)) return KVRING_ERR_INVALID_ARG;
  const Plan p = plan_for(cfg);
  if (bytes < p.total) return KVRING_ERR_CAPACITY;

  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVRING_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3) return KVRING_ERR_UNSUPPORTED;  // built for sm_103a only
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, dev_buf) != cudaSuccess || pa.type != cudaMemoryTypeDevice ||
      pa.device != dev)
    return KVRING_ERR_INVALID_ARG;

  kvring* r = new (std::nothrow) kvring();
  if (!r) return KVRING_ERR_INVALID_ARG;
  r->cfg = *cfg;
  r->sm_count = sms > 0 ? sms : 1;
  r->device = dev;
  r->qtiles_max = p.qtiles;
  r->calibrated = false;
  r->attn_wait_ns = kDefaultWaitNs;
  r->attn_debug_stall = 0;
  r->attn_debug_guess = 0;
  uint8_t* b = static_cast<uint8_t*>(dev_buf);
  kvr::RingDev& d = r->dev;
  d.k = b + p.k;
  d.v = b + p.v;
  d.slot_pos = reinterpret_cast<int32_t*>(b + p.slot_pos);
  d.scales = reinterpret_cast<float*>(b + p.scales);
  d.state = reinterpret_cast<int32_t*>(b + p.state);
  d.amax = reinterpret_cast<uint32_t*>(b + p.amax);
  d.table = reinterpret_cast<const float*>(b + p.table);
  // split partials exist only for rings allowing more than 8 splits
  d.part_o = cfg->max_kv_splits > 8 ? reinterpret_cast<float*>(b + p.part_o) : nullptr;
  d.part_lse = cfg->max_kv_splits > 8 ? reinterpret_cast<float*>(b + p.part_lse) : nullptr;
  d.tickets = reinterpret_cast<int32_t*>(b + p.tickets);
  d.levels = reinterpret_cast<int32_t*>(b + p.levels);
  d.H = cfg->num_heads;
  d.D = cfg->head_dim;
  d.C = cfg->capacity;
  d.max_pos = cfg->max_position;
  d.max_tokens = cfg->max_tokens;
  d.max_splits = cfg->max_kv_splits;
  d.qtiles_max = p.qtiles;
  d.P = cfg->pinned_prefix;
  d.pt = cfg->rope_pairs_t;
  d.py = cfg->rope_pairs_y;

  if (kvr::attention_prepare(d.D) != cudaSuccess || kvr::cache_prepare() != cudaSuccess ||
      kvr::project_prepare() != cudaSuccess) {
    delete r;
    return KVRING_ERR_CUDA;
  }
  if (!make_cache_map(&r->tmK, d.k, d.H, d.C, d.D) || !make_cache_map(&r->tmV, d.v, d.H, d.C, d.D)) {
    delete r;
    return KVRING_ERR_UNSUPPORTED;
  }

  // Host-built contents: empty positions, unit scales, the RoPE table
  // (theta_i = base^(-2i/d) and cos/sin of p*theta_i in double libm,
  // rounded to fp32; with 3-D RoPE each section has its own ladder:
  // local pair j of a section of m pairs gets base^(-2j/(2m))).
  const int H = d.H, D = d.D, C = d.C;
  std::vector<int32_t> slot_pos(C, kvr::kEmptyPos);
  std::vector<float> scales(4 * H, 1.0f);
  std::vector<float> table((size_t)cfg->max_position * D);
  std::vector<double> theta(D / 2);
  if (d.pt == 0) {
    for (int i = 0; i < D / 2; ++i) theta[i] = std::pow(cfg->rope_base, (-2.0 * i) / (double)D);
  } else {
    const int lo[3] = {0, d.pt, d.pt + d.py}, m[3] = {d.pt, d.py, D / 2 - d.pt - d.py};
    for (int a = 0; a < 3; ++a)
      for (int j = 0; j < m[a]; ++j) theta[lo[a] + j] = std::pow(cfg->rope_base, (-2.0 * j) / (double)(2 * m[a]));
  }
  for (int pos = 0; pos < cfg->max_position; ++pos) {
    float* row = table.data() + (size_t)pos * D;
    for (int i = 0; i < D / 2; ++i) {
      const double a = (double)pos * theta[i];
      row[2 * i] = (float)std::cos(a);
      row[2 * i + 1] = (float)std::sin(a);
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t x) {
    if (e == cudaSuccess) e = x;
  };
  chk(cudaMemsetAsync(b, 0, p.total, s));
  chk(cudaMemcpyAsync(d.slot_pos, slot_pos.data(), C * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  chk(cudaMemcpyAsync(d.scales, scales.data(), scales.size() * sizeof(float), cudaMemcpyHostToDevice, s));
  chk(cudaMemcpyAsync(b + p.table, table.data(), table.size() * sizeof(float), cudaMemcpyHostToDevice, s));
  chk(cudaStreamSynchronize(s));  // host vectors die at return
  if (e != cudaSuccess) {
    delete r;
    return KVRING_ERR_CUDA;
  }
  *out = r;
  return KVRING_OK;
}

kvring_status kvring_destroy(kvring_t* ring) {
  delete ring;
  return KVRING_OK;
}

kvring_status kvring_calibrate_scales(kvring_t* r, const void* k, const void* v, const int32_t* pos,
                                      int32_t n, void* stream) {
  if (!r || !k || !v || !aligned(k, 16) || !aligned(v, 16) || (pos && !aligned(pos, 4)) || n < 1)
    return KVRING_ERR_INVALID_ARG;
  if (r->dev.pt && !pos) return KVRING_ERR_INVALID_ARG;   // 3-D positions must be given
  if (!on_device(r)) return KVRING_ERR_INVALID_ARG;
  if (n > r->cfg.max_tokens) return KVRING_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_out_mu);
  const kvring_status st = tracked(s, [&] { return kvr::launch_calibrate(r->dev, k, v, pos, n, s); });
  if (st == KVRING_OK) r->calibrated = true;
  return st;
}

kvring_status kvring_write_frame(kvring_t* r, const void* k, const void* v, const int32_t* pos, int32_t n,
                                 void* stream) {
  if (!r || !k || !v || !aligned(k, 16) || !aligned(v, 16) || (pos && !aligned(pos, 4)) || n < 1)
    return KVRING_ERR_INVALID_ARG;
  if (r->dev.pt && !pos) return KVRING_ERR_INVALID_ARG;
  if (!on_device(r)) return KVRING_ERR_INVALID_ARG;
  if (!r->calibrated) return KVRING_ERR_NOT_CALIBRATED;
  if (n > r->cfg.capacity - r->cfg.pinned_prefix || n > r->cfg.max_tokens) return KVRING_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t frame = (size_t)n * r->dev.H * r->dev.D * 2;
  std::lock_guard<std::mutex> lk(g_out_mu);
  const bool late = late_inputs(s, {{k, frame}, {v, frame}});
  const bool idle = ring_idle(s, r);
  return passed_through(s, [&] { return kvr::launch_write(r->dev, k, v, pos, n, late, idle, s); }, &r, 1);
}

kvring_status kvring_delta_rotate(kvring_t* r, int32_t delta, void* stream) {
  if (!r || !on_device(r)) return KVRING_ERR_INVALID_ARG;
  if (delta != KVRING_DELTA_TO_OLDEST && (delta < 0 || delta >= r->cfg.max_position))
    return KVRING_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_out_mu);
  const bool idle = ring_idle(s, r);
  return passed_through(s, [&] { return kvr::launch_delta(r->dev, delta, idle, s); }, &r, 1);
}

namespace {
// Common checks of a batch: count, distinct non-NULL rings of one shape.
kvring_status check_batch(kvring_t* const* rings, int32_t count) {
  if (!rings || count < 1 || count > KVRING_MAX_BATCH || count > kvr::kMaxBatch) return KVRING_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    const kvring* r = rings[i];
    if (!r || !on_device(r)) return KVRING_ERR_INVALID_ARG;
    const kvring* r0 = rings[0];
    if (r->cfg.num_heads != r0->cfg.num_heads || r->cfg.head_dim != r0->cfg.head_dim ||
        r->cfg.capacity != r0->cfg.capacity || r->cfg.pinned_prefix != r0->cfg.pinned_prefix ||
        r->cfg.rope_pairs_t != r0->cfg.rope_pairs_t || r->cfg.rope_pairs_y != r0->cfg.rope_pairs_y)
      return KVRING_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (rings[j] == r) return KVRING_ERR_INVALID_ARG;
  }
  return KVRING_OK;
}
}  // namespace

kvring_status kvring_write_frames_many(kvring_t* const* rings, int32_t count, const void* const* k,
                                       const void* const* v, const int32_t* const* pos, int32_t n,
                                       void* stream) {
  kvring_status st = check_batch(rings, count);
  if (st != KVRING_OK) return st;
  if (!k || !v || n < 1) return KVRING_ERR_INVALID_ARG;
  static thread_local kvr::WriteMany b;   // ~10 KB: kernel parameters, not device memory
  for (int i = 0; i < count; ++i) {
    const kvring* r = rings[i];
    const int32_t* p = pos ? pos[i] : nullptr;
    if (!k[i] || !v[i] || !aligned(k[i], 16) || !aligned(v[i], 16) || (p && !aligned(p, 4)))
      return KVRING_ERR_INVALID_ARG;
    if (r->dev.pt && !p) return KVRING_ERR_INVALID_ARG;
    if (!r->calibrated) return KVRING_ERR_NOT_CALIBRATED;
    if (n > r->cfg.capacity - r->cfg.pinned_prefix || n > r->cfg.max_tokens) return KVRING_ERR_CAPACITY;
    b.r[i] = r->dev;
    b.k[i] = static_cast<const uint16_t*>(k[i]);
    b.v[i] = static_cast<const uint16_t*>(v[i]);
    b.pos[i] = p;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_out_mu);   // (frames are read after the wait: nothing to check)
  return passed_through(s, [&] { return kvr::launch_write_many(b, count, n, s); }, rings, count);
}

kvring_status kvring_delta_rotate_many(kvring_t* const* rings, int32_t count, int32_t delta, void* stream) {
  kvring_status st = check_batch(rings, count);
  if (st != KVRING_OK) return st;
  static thread_local kvr::DeltaMany b;
  for (int i = 0; i < count; ++i) {
    const kvring* r = rings[i];
    if (delta != KVRING_DELTA_TO_OLDEST && (delta < 0 || delta >= r->cfg.max_position))
      return KVRING_ERR_INVALID_ARG;
    b.r[i] = r->dev;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_out_mu);
  return passed_through(s, [&] { return kvr::launch_delta_many(b, count, delta, s); }, rings, count);
}

kvring_status kvring_project_write(kvring_t* r, const void* x, const void* w, int32_t d_model, const int32_t* pos,
                                   int32_t n, void* q_out, void* kv_out, int32_t flags, void* stream) {
  if (!r || !x || !w || !aligned(x, 16) || !aligned(w, 16) || n < 1) return KVRING_ERR_INVALID_ARG;
  if (flags & ~(KVRING_PROJECT_WRITE | KVRING_PROJECT_STORE_KV)) return KVRING_ERR_INVALID_ARG;
  if ((flags & KVRING_PROJECT_STORE_KV) && (!kv_out || !aligned(kv_out, 16))) return KVRING_ERR_INVALID_ARG;
  if ((q_out && !aligned(q_out, 16)) || (pos && !aligned(pos, 4))) return KVRING_ERR_INVALID_ARG;
  if (d_model < 64 || d_model % 64 != 0 || d_model > (1 << 20)) return KVRING_ERR_INVALID_ARG;
  const bool write = (flags & KVRING_PROJECT_WRITE) != 0;
  if (write && r->dev.pt && !pos) return KVRING_ERR_INVALID_ARG;   // 3-D positions must be given
  if (!on_device(r)) return KVRING_ERR_INVALID_ARG;
  if (write && !r->calibrated) return KVRING_ERR_NOT_CALIBRATED;
  if (n > r->cfg.max_tokens || (write && n > r->cfg.capacity - r->cfg.pinned_prefix)) return KVRING_ERR_CAPACITY;
  CUtensorMap tmX, tmW;
  if (!make_bf16_map(&tmX, x, n, d_model, 128) ||
      !make_bf16_map(&tmW, w, 3 * r->dev.H * r->dev.D, d_model, kvr::kProjTileN))
    return KVRING_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)n * r->dev.H * r->dev.D * 2;   // bytes of one bf16 [n][H][d] output
  const Range qr{q_out, q_out ? rows : 0};
  const bool kv = (flags & KVRING_PROJECT_STORE_KV) != 0;
  const Range kvo{kv ? kv_out : nullptr, kv ? 2 * rows : 0};
  std::lock_guard<std::mutex> lk(g_out_mu);
  return tracked(
      s, [&] { return kvr::launch_project(r->dev, &tmX, &tmW, pos, q_out, kv_out, n, d_model, flags, s); }, qr, kvo,
      write ? r : nullptr);
}

kvring_status kvring_legacy_upkeep(kvring_t* r, const void* wk_in, const void* wv_in, void* wk_out, void* wv_out,
                                   const void* k, const void* v, int32_t n, void* stream) {
  if (!r || !wk_in || !wv_in || !wk_out || !wv_out || !k || !v || n < 1 || !on_device(r))
    return KVRING_ERR_INVALID_ARG;
  const void* ptrs[6] = {wk_in, wv_in, wk_out, wv_out, k, v};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return KVRING_ERR_INVALID_ARG;
  if (wk_in == wk_out || wv_in == wv_out || wk_out == wv_out) return KVRING_ERR_INVALID_ARG;
  // the original upkeep had neither a prefix nor 3-D RoPE
  if (r->cfg.pinned_prefix != 0 || r->dev.pt != 0) return KVRING_ERR_UNSUPPORTED;
  if (n > r->cfg.capacity || n > r->cfg.max_tokens) return KVRING_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t window = (size_t)r->cfg.capacity * r->dev.H * r->dev.D * 2;
  std::lock_guard<std::mutex> lk(g_out_mu);
  const kvring_status st = tracked(
      s, [&] { return kvr::launch_legacy_upkeep(r->dev, wk_in, wv_in, wk_out, wv_out, k, v, n, s); },
      Range{wk_out, window}, Range{wv_out, window});
  if (st == KVRING_OK) r->calibrated = true;   // the path sets its own scales
  return st;
}

kvring_status kvring_attention(kvring_t* r, const void* q, const int32_t* qpos, int32_t n_q, void* out,
                               int32_t out_dtype, void* stream) {
  if (!r || !q || !out || !aligned(q, 16) || !aligned(out, 16) || (qpos && !aligned(qpos, 4)) || n_q < 1)
    return KVRING_ERR_INVALID_ARG;
  if (r->dev.pt && !qpos) return KVRING_ERR_INVALID_ARG;   // 3-D positions must be given
  if (out_dtype != KVRING_OUT_F32 && out_dtype != KVRING_OUT_BF16) return KVRING_ERR_INVALID_ARG;
  if (!on_device(r)) return KVRING_ERR_INVALID_ARG;
  if (!r->calibrated) return KVRING_ERR_NOT_CALIBRATED;
  if (n_q > r->cfg.max_tokens) return KVRING_ERR_CAPACITY;
  kvr::AttnLaunch a;
  a.q = q;
  a.qpos = qpos;
  a.out = out;
  a.n_q = n_q;
  a.out_bf16 = out_dtype == KVRING_OUT_BF16;
  a.forced_level = r->cfg.attn_precision;
  a.debug_stall = r->attn_debug_stall;
  a.debug_guess = r->attn_debug_guess;
  a.wait_ns = r->attn_wait_ns;
  choose_splits(r, n_q, &a.nsplit, &a.tiles_per_split);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)n_q * r->dev.H * r->dev.D;
  std::lock_guard<std::mutex> lk(g_out_mu);
  a.q_late = late_inputs(s, {{q, 2 * rows}}) ? 1 : 0;
  return tracked(s, [&] { return kvr::launch_attention(r->dev, &r->tmK, &r->tmV, a, s); },
                 Range{out, rows * (a.out_bf16 ? 2 : 4)}, Range{nullptr, 0}, r);
}

kvring_status kvring_attention_noalloc(kvring_t* r, const void* q, const int32_t* qpos, int32_t n_q,
                                       void* out, int32_t out_dtype, void* stream) {
  if (!r || !q || !out || !aligned(q, 16) || !aligned(out, 16) || (qpos && !aligned(qpos, 4)) || n_q < 1)
    return KVRING_ERR_INVALID_ARG;
  if (r->dev.pt && !qpos) return KVRING_ERR_INVALID_ARG;   // 3-D positions must be given
  if (out_dtype != KVRING_OUT_F32 && out_dtype != KVRING_OUT_BF16) return KVRING_ERR_INVALID_ARG;
  if (!on_device(r)) return KVRING_ERR_INVALID_ARG;
  if (!r->calibrated) return KVRING_ERR_NOT_CALIBRATED;
  if (n_q > r->cfg.max_tokens) return KVRING_ERR_CAPACITY;
  // Scratch for this call inside the static array: the precision level of
  // each (query tile, head).  At most 8 splits, which merge inside their
  // thread-block cluster, so no split partials or tickets are needed.
  const size_t H = (size_t)r->dev.H;
  const size_t qtiles = (size_t)((n_q + kvr::kTile - 1) / kvr::kTile);
  const size_t units = qtiles * H;
  if (units * 4 > kvr::static_scratch_bytes()) return KVRING_ERR_CAPACITY;
  kvr::AttnLaunch a;
  a.q = q;
  a.qpos = qpos;
  a.out = out;
  a.n_q = n_q;
  a.out_bf16 = out_dtype == KVRING_OUT_BF16;
  a.forced_level = r->cfg.attn_precision;
  a.debug_stall = r->attn_debug_stall;
  a.debug_guess = r->attn_debug_guess;
  a.wait_ns = r->attn_wait_ns;
  choose_splits(r, n_q, &a.nsplit, &a.tiles_per_split);
  const int ctiles = (r->cfg.capacity + kvr::kTile - 1) / kvr::kTile;
  if (a.nsplit > 8) {
    a.tiles_per_split = (ctiles + 7) / 8;
    a.nsplit = (ctiles + a.tiles_per_split - 1) / a.tiles_per_split;
  }
  void* base = nullptr;
  if (kvr::static_scratch_address(&base) != cudaSuccess) return KVRING_ERR_CUDA;
  kvr::RingDev d = r->dev;
  d.levels = static_cast<int32_t*>(base);
  d.tickets = nullptr;
  d.part_o = nullptr;
  d.part_lse = nullptr;
  d.qtiles_max = (int)qtiles;
  d.max_splits = a.nsplit;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)n_q * r->dev.H * r->dev.D;
  std::lock_guard<std::mutex> lk(g_out_mu);
  a.q_late = late_inputs(s, {{q, 2 * rows}}) ? 1 : 0;
  return tracked(s, [&] { return kvr::launch_attention(d, &r->tmK, &r->tmV, a, s); },
                 Range{out, rows * (a.out_bf16 ? 2 : 4)}, Range{nullptr, 0}, r);
}

kvring_status kvring_export(kvring_t* r, void* k_out, void* v_out, float* scales, int32_t* slot_pos,
                            int32_t* state, void* stream) {
  if (!r || !on_device(r)) return KVRING_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t cache = (size_t)r->dev.H * r->dev.C * r->dev.D;
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t x) {
    if (e == cudaSuccess) e = x;
  };
  if (k_out) chk(cudaMemcpyAsync(k_out, r->dev.k, cache, cudaMemcpyDefault, s));
  if (v_out) chk(cudaMemcpyAsync(v_out, r->dev.v, cache, cudaMemcpyDefault, s));
  if (scales) chk(cudaMemcpyAsync(scales, r->dev.scales, 4 * r->dev.H * sizeof(float), cudaMemcpyDefault, s));
  if (slot_pos) chk(cudaMemcpyAsync(slot_pos, r->dev.slot_pos, r->dev.C * sizeof(int32_t), cudaMemcpyDefault, s));
  if (state) chk(cudaMemcpyAsync(state, r->dev.state, KVRING_STATE_WORDS * sizeof(int32_t), cudaMemcpyDefault, s));
  return cuda_status(e);
}

kvring_status kvring_debug_encode_e4m3(const float* in, uint8_t* out, int64_t n, void* stream) {
  if ((!in || !out) && n > 0) return KVRING_ERR_INVALID_ARG;
  if (n < 0) return KVRING_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_out_mu);
  return tracked(s, [&] { return kvr::launch_encode_e4m3(in, out, n, s); }, Range{out, (size_t)n});
}

kvring_status kvring_debug_write_floor(kvring_t* r, int32_t n, void* stream) {
  if (!r || n < 1 || !on_device(r)) return KVRING_ERR_INVALID_ARG;
  if (n > r->cfg.capacity - r->cfg.pinned_prefix || n > r->cfg.max_tokens) return KVRING_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_out_mu);
  const bool idle = ring_idle(s, r);
  return passed_through(s, [&] { return kvr::launch_write_floor(r->dev, n, idle, s); }, &r, 1);
}

kvring_status kvring_debug_set_attention_wait(kvring_t* r, int64_t limit_ns, int32_t stall) {
  if (!r || limit_ns < 1000 || limit_ns > 60000000000ll || (stall != 0 && stall != 1))
    return KVRING_ERR_INVALID_ARG;
  r->attn_wait_ns = (unsigned long long)limit_ns;
  r->attn_debug_stall = stall;
  return KVRING_OK;
}

kvring_status kvring_debug_attention_guess(kvring_t* r, int32_t wrong) {
  if (!r || (wrong != 0 && wrong != 1)) return KVRING_ERR_INVALID_ARG;
  r->attn_debug_guess = wrong;
  return KVRING_OK;
}

kvring_status kvring_debug_attention_levels(kvring_t* r, int32_t* levels, void* stream) {
  if (!r || !levels || !on_device(r)) return KVRING_ERR_INVALID_ARG;
  const size_t bytes = (size_t)r->qtiles_max * r->dev.H * sizeof(int32_t);
  return cuda_status(cudaMemcpyAsync(levels, r->dev.levels, bytes, cudaMemcpyDefault, (cudaStream_t)stream));
}

int64_t kvring_debug_late_reads(void) {
  std::lock_guard<std::mutex> lk(g_out_mu);
  return g_late_reads;
}

const char* kvring_status_string(kvring_status s) {
  switch (s) {
    case KVRING_OK: return "ok";
    case KVRING_ERR_INVALID_ARG: return "invalid argument";
    case KVRING_ERR_NOT_CALIBRATED: return "ring not calibrated";
    case KVRING_ERR_CAPACITY: return "too many tokens for the ring or its config";
    case KVRING_ERR_UNSUPPORTED: return "unsupported head_dim or device";
    case KVRING_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

}  // extern "C"
