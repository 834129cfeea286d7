// Memory-bound kernels of the rolling FP8 cache: per-session scale
// calibration, the per-frame write (RoPE + E4M3 quantisation into the ring)
// and the in-place delta rotation at a position reset.  See the page
// "Runway Characters: Serving a 57B Video Diffusion Transformer for
// Real-Time Conversation", section "Do It Once, at Write Time".
//
// Work decomposition.  Calibration and the single-ring write: one thread
// owns 16 consecutive elements of one (token, head) row, i.e. one 16-byte
// chunk of FP8 output; consecutive threads walk a row, then the next head,
// then the next token, so bf16 input reads are fully contiguous and every
// cache row is written as whole 16-byte vectors.  The batched write and the
// delta rotation are bulk-copy pipelines: one block per SM, one producer
// thread streaming contiguous 16 KB units into shared-memory stages, sixteen
// consumer warps doing the arithmetic and storing whole 16-byte vectors.
// Completion work (ring state, scales, position map) is done by the last
// block (or warp) to finish, found with an atomic ticket; no block ever
// waits on another.
//
// Arithmetic is pinned so that cache bytes are reproducible: products and
// sums are rounded one at a time (__fmul_rn / __fadd_rn / __fsub_rn, no
// fused multiply-add), the cos/sin table is fp32 built on the host, and the
// E4M3 conversion is the hardware round-to-nearest-even saturating cvt.
#include "kvring_internal.cuh"
#include <cuda_bf16.h>

namespace kvr {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void unpack_bf16x16(const uint4& a, const uint4& b, float (&x)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack_e4m3x16(const float (&z)[16]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = f32x2_to_e4m3x2(z[4 * i], z[4 * i + 1]);
    const uint32_t hi = f32x2_to_e4m3x2(z[4 * i + 2], z[4 * i + 3]);
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Rotate 8 adjacent pairs by the angles whose fp32 cos/sin are in `cs`
// (c0, s0, c1, s1, ...): y0 = x0*c - x1*s, y1 = x0*s + x1*c, every step
// rounded to fp32.
__device__ __forceinline__ void rope_pinned(float (&x)[16], const float4 (&cs)[4]) {
  const float c[8] = {cs[0].x, cs[0].z, cs[1].x, cs[1].z, cs[2].x, cs[2].z, cs[3].x, cs[3].z};
  const float s[8] = {cs[0].y, cs[0].w, cs[1].y, cs[1].w, cs[2].y, cs[2].w, cs[3].y, cs[3].w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float x0 = x[2 * i], x1 = x[2 * i + 1];
    x[2 * i] = __fsub_rn(__fmul_rn(x0, c[i]), __fmul_rn(x1, s[i]));
    x[2 * i + 1] = __fadd_rn(__fmul_rn(x0, s[i]), __fmul_rn(x1, c[i]));
  }
}

__device__ __forceinline__ void load_table16(const float* table, int D, int p, int chunk,
                                             float4 (&cs)[4]) {
  const float4* t = reinterpret_cast<const float4*>(table + ((size_t)p * (D / 2) + chunk * 8) * 2);
#pragma unroll
  for (int i = 0; i < 4; ++i) cs[i] = __ldg(t + i);
}

// The same rotation for 2 adjacent pairs, cos/sin in `cs` as (c0, s0, c1, s1).
__device__ __forceinline__ void rope_pinned2(float (&x)[4], const float4& cs) {
  const float x0 = x[0], x1 = x[1], x2 = x[2], x3 = x[3];
  x[0] = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
  x[1] = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
  x[2] = __fsub_rn(__fmul_rn(x2, cs.z), __fmul_rn(x3, cs.w));
  x[3] = __fadd_rn(__fmul_rn(x2, cs.w), __fmul_rn(x3, cs.z));
}

// ------------------------------------------------------------ calibrate ---
template <int D>
__global__ void __launch_bounds__(kThreads) k_calibrate(RingDev r, const uint16_t* __restrict__ k,
                                                        const uint16_t* __restrict__ v,
                                                        const int32_t* __restrict__ pos, int n) {
  constexpr int CH = D / 16;
  __shared__ int s_next;
  __shared__ int s_last;
  if (threadIdx.x == 0) s_next = __ldcg(r.state + ST_NEXT_POS);
  __syncthreads();
  const int H = r.H;
  const long long per = (long long)n * H * CH;
  const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
  float m = 0.f;
  int isv = 0, h = 0, chunk = 0;
  if (gid < 2 * per) {
    isv = gid >= per;
    const long long w = isv ? gid - per : gid;
    chunk = (int)(w % CH);
    const long long th = w / CH;
    h = (int)(th % H);
    const int t = (int)(th / H);
    const uint4* src = reinterpret_cast<const uint4*>((isv ? v : k) + ((size_t)t * H + h) * D + chunk * 16);
    float x[16];
    unpack_bf16x16(__ldcs(src), __ldcs(src + 1), x);
    bool ok = true;
    if (!isv) {
      const int p = pos ? rope_pos(r, pos, t, 8 * chunk) : s_next + t;   // 3-D: the chunk's coordinate
      if (p < 0 || p >= r.max_pos) {
        ok = false;
        atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
      } else {
        float4 cs[4];
        load_table16(r.table, D, p, chunk, cs);
        rope_pinned(x, cs);
      }
    }
    if (ok) {
#pragma unroll
      for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(x[i]));
    }
  }
  // max over the CH lanes of one row (rows start at multiples of CH lanes)
#pragma unroll
  for (int off = CH / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if (gid < 2 * per && chunk == 0 && m > 0.f) atomicMax(r.amax + isv * H + h, __float_as_uint(m));

  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int tk = atomicAdd(r.state + ST_TICKET_CALIB, 1);
    s_last = tk == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int i = threadIdx.x; i < 2 * H; i += kThreads) {
      const float a = __uint_as_float(atomicExch(r.amax + i, 0u));
      float sc = __fdiv_rn(a, 448.0f);
      if (!(sc >= 0x1p-126f)) sc = 1.0f;
      r.scales[i] = sc;                         // scale_k then scale_v
      r.scales[2 * H + i] = __fdiv_rn(1.0f, sc);  // their reciprocals
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      r.state[ST_CALIBRATED] = 1;
      r.state[ST_TICKET_CALIB] = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------- write ---
// The single-ring write publishes its state from values every block's
// thread 0 gathers right after the wait, so the last block's publication is
// stores only.  token_of_slot: the index of this frame's token that goes to
// slot s (token t goes to head0 + t, wrapped past the prefix), or -1.
__device__ __forceinline__ int token_of_slot(const RingDev& r, int head0, int n, int s) {
  int t = s - head0;
  if (t < 0) {
    if (s < r.P) return -1;
    t += r.C - r.P;
  }
  return t < n ? t : -1;
}
struct WritePlan {
  int head, nv, tot_lo, tot_hi, next, oldest, prefix_end;
};
// From the state at the start of a write of n tokens (read after the wait):
// the state after it.  The position of the oldest rolling slot and of the
// prefix's last slot come from this frame's positions when this frame
// writes those slots, else from their current entries (which this write
// leaves alone), loaded here.
__device__ __forceinline__ WritePlan plan_write(const RingDev& r, const int32_t* pos, int head0, int nv0,
                                                unsigned long long total, int next0, int n) {
  const int C = r.C, P = r.P;
  WritePlan w;
  w.head = head0 + n;
  if (w.head >= C) w.head -= C - P;   // the wrap skips the pinned prefix
  w.nv = nv0 + n < C ? nv0 + n : C;
  const unsigned long long tot = total + (unsigned long long)n;
  w.tot_lo = (int)(unsigned)(tot & 0xFFFFFFFFull);
  w.tot_hi = (int)(unsigned)(tot >> 32);
  w.next = next0 + n;
  auto position = [&](int s) {
    const int t = token_of_slot(r, head0, n, s);
    return t >= 0 ? (pos ? rope_pos(r, pos, t, 0) : next0 + t) : __ldcg(r.slot_pos + s);
  };
  // oldest rolling slot: the next one to be overwritten once full, else slot P
  w.oldest = w.nv > P ? position(w.nv >= C ? w.head : P) : kEmptyPos;
  w.prefix_end = (P > 0 && w.nv >= P) ? position(P - 1) + 1 : 0;
  return w;
}

// Store a gathered plan as the ring's state (the publication of a write).
__device__ __forceinline__ void store_write_plan(const RingDev& r, const WritePlan& w) {
  r.state[ST_HEAD] = w.head;
  r.state[ST_NVALID] = w.nv;
  r.state[ST_TOTAL_LO] = w.tot_lo;
  r.state[ST_TOTAL_HI] = w.tot_hi;
  r.state[ST_NEXT_POS] = w.next;
  st_relaxed_gpu(r.state + ST_NEXT_POS_HINT, w.next);
  r.state[ST_OLDEST_POS] = w.oldest;
  if (r.P > 0 && w.nv >= r.P) r.state[ST_PREFIX_END] = w.prefix_end;
  r.state[ST_TICKET_WRITE] = 0;
}

// Each thread owns kWriteU chunks, (block * kWriteU + u) * 256 + tid, so a
// warp's accesses stay contiguous; all input loads are issued before the
// ring state is read, which hides one DRAM round trip.
constexpr int kWriteU = 2;

// One ring's share of a write: block `blk` of `nblk` blocks working on ring
// r, U chunks per thread (2 for one ring; batched launches are large enough
// to keep more in flight per thread).
template <int D, int U>
__device__ __forceinline__ void write_body(const RingDev& r, const uint16_t* __restrict__ k,
                                           const uint16_t* __restrict__ v, const int32_t* __restrict__ pos,
                                           int n, int blk, int nblk, bool late) {
  constexpr int CH = D / 16;
  __shared__ int s_head, s_next;
  // A following kernel launched as a programmatic dependent (an attention's
  // query preparation, or the next write) may start now: each waits for
  // this grid before it touches the ring.  (This kernel writes no caller
  // buffer; the host's record of which caller buffers kernels still in
  // flight may write carries over it to the next call.)  Block 0 first
  // leaves the next position this write will publish as a hint for them.
  if (blk == 0 && threadIdx.x == 0)
    st_relaxed_gpu(r.state + ST_NEXT_POS_HINT, ld_relaxed_gpu(r.state + ST_NEXT_POS) + n);
  griddep_launch_dependents();
  const int H = r.H, C = r.C;
  const long long per = (long long)n * H * CH;
  // The frame is loaded before the wait for the preceding kernel unless the
  // host found that a kernel still in flight may write it.
  if (late) griddep_wait();
  uint4 in[U][2];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const long long gid = ((long long)blk * U + u) * kThreads + threadIdx.x;
    if (gid < 2 * per) {
      const int isv = gid >= per;
      const long long w = isv ? gid - per : gid;
      const uint4* src = reinterpret_cast<const uint4*>((isv ? v : k) + (w / CH) * D + (w % CH) * 16);
      in[u][0] = __ldcs(src);
      in[u][1] = __ldcs(src + 1);
    }
  }
  // All table rows before any arithmetic or store, so their latencies overlap.
  float4 cs[U][4];
  int pp[U];
  auto load_rows = [&](int next) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long gid = ((long long)blk * U + u) * kThreads + threadIdx.x;
      pp[u] = -1;
      if (gid < per) {  // keys only
        const int chunk = (int)(gid % CH);
        const int t = (int)(gid / CH / H);
        const int p = pos ? rope_pos(r, pos, t, 8 * chunk) : next + t;   // chunk 0: t (3-D)
        pp[u] = p;
        if (p >= 0 && p < r.max_pos) load_table16(r.table, D, p, chunk, cs[u]);
      }
    }
  };
  // With default positions the rows depend only on next_pos, which nothing
  // but this ring's own calls changes: load them now for its current value
  // (a relaxed read that may race with a preceding call on this ring) and
  // reload after the wait only if it turned out different.
  __shared__ int s_guess;
  if (!pos) {
    if (threadIdx.x == 0) s_guess = ld_relaxed_gpu(r.state + ST_NEXT_POS);
    __syncthreads();
    load_rows(s_guess);
  }
  // This kernel is launched as a programmatic dependent of the preceding
  // kernel: the ring (state, cache, positions) is read and written only
  // after it is done.
  griddep_wait();
  int nv0 = 0;
  unsigned long long total0 = 0;
  if (threadIdx.x == 0) {
    const int4 st = __ldcg(reinterpret_cast<const int4*>(r.state));   // head, n_valid, total lo, hi
    s_head = st.x;
    nv0 = st.y;
    total0 = (unsigned long long)(unsigned)st.w << 32 | (unsigned)st.z;
    s_next = __ldcg(r.state + ST_NEXT_POS);
  }
  __syncthreads();
  // thread 0 gathers the state after this write while the block works
  WritePlan plan{};
  if (threadIdx.x == 0) plan = plan_write(r, pos, s_head, nv0, total0, s_next, n);
  if (pos || s_next != s_guess) load_rows(s_next);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const long long gid = ((long long)blk * U + u) * kThreads + threadIdx.x;
    if (gid >= 2 * per) continue;
    const int isv = gid >= per;
    const long long w = isv ? gid - per : gid;
    const int chunk = (int)(w % CH);
    const long long th = w / CH;
    const int h = (int)(th % H);
    const int t = (int)(th / H);
    // head < C and t < n <= C - P: at most one wrap, which skips the prefix
    int slot = s_head + t;
    if (slot >= C) slot -= C - r.P;
    float x[16];
    unpack_bf16x16(in[u][0], in[u][1], x);
    bool ok = true;
    if (!isv) {
      const int p = pp[u];
      if (p < 0 || p >= r.max_pos) {
        ok = false;
        atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
      } else {
        rope_pinned(x, cs[u]);
      }
      if (h == 0 && chunk == 0) r.slot_pos[slot] = p;
    }
    if (ok) {
      const float inv = r.scales[(isv ? 3 : 2) * H + h];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = __fmul_rn(x[i], inv);
      uint8_t* dst = (isv ? r.v : r.k) + ((size_t)h * C + slot) * D + chunk * 16;
      *reinterpret_cast<uint4*>(dst) = pack_e4m3x16(x);
    }
  }
  __syncthreads();
  // The last block to finish publishes the state.  No fence before the
  // ticket: the publication reads nothing another block wrote (the plan was
  // gathered at the start), every block read the old state before its
  // ticket, and the next kernel sees the cache through this grid's end.
  if (threadIdx.x == 0) {
    const int tk = atomicAdd(r.state + ST_TICKET_WRITE, 1);
    if (tk == nblk - 1) store_write_plan(r, plan);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 3) k_write(RingDev r, const uint16_t* __restrict__ k,
                                                    const uint16_t* __restrict__ v,
                                                    const int32_t* __restrict__ pos, int n, int late) {
  write_body<D, kWriteU>(r, k, v, pos, n, blockIdx.x, gridDim.x, late != 0);
}

// The write's fixed cost alone: the grid of an n-token write, the same
// programmatic-dependent launch, wait, ring-state read, completion ticket
// and state publication by the last block, with no data (zero tokens, so the
// published state equals the state read and the ring is unchanged).
template <int D>
__global__ void __launch_bounds__(kThreads, 3) k_write_floor(RingDev r) {
  write_body<D, kWriteU>(r, nullptr, nullptr, nullptr, 0, blockIdx.x, gridDim.x, false);
}

// One ring's write staged through shared memory.  Block b takes the tb
// whole tokens [b TB, b TB + tb) of the frame, keys and values of all heads,
// so a block is fat (about 28 KB of shared memory) and a production frame
// needs 152 of them, a few per SM: the grid fits on the SMs that the
// preceding attention leaves idle.  Before the wait for the preceding
// kernel the block copies the frame and the RoPE rows (for the ring's next
// position, read with a relaxed load) into shared memory with cp.async and
// encodes every chunk (rotation, scale, E4M3) in place; after the wait it
// only reads the ring state and copies the codes into their slots.  If the
// next position turned out different, or the positions are explicit (they
// are read only after the wait), the rows are staged again and the chunks
// encoded after the wait.  Shared memory: the frame, bf16 [2][tb][H][D] (a
// chunk's 16 codes land in the first half of its own 32 bytes), then one
// assembled table row per token, fp32 [tb][D] (chunk c's 16 values from the
// row of its section's position).  nodata: the fixed cost alone (same grid,
// launch, hint, wait, state read, plan, ticket and publication; nothing read
// from the frame, nothing written to the cache, 0 tokens published).
// idle: no kernel that may still run reads or writes this ring (the host
// keeps track); then, with default positions and early inputs, the ring
// state read before the wait is exact and the whole write -- codes into
// their slots, ticket, publication -- happens before it.  Block 0 then
// waits, so that the kernels of the stream still complete in order; the
// other blocks leave at once.
template <int D>
__global__ void __launch_bounds__(kThreads) k_write_tok(RingDev r, const uint16_t* __restrict__ k,
                                                       const uint16_t* __restrict__ v,
                                                       const int32_t* __restrict__ pos, int n, int TB, int late,
                                                       int nodata, int idle) {
  constexpr int CH = D / 16;
  extern __shared__ __align__(16) uint8_t wts_sm[];
  __shared__ int s_head, s_next, s_guess;
  const int H = r.H, C = r.C;
  const int t0 = blockIdx.x * TB;
  const int tb = nodata ? 0 : (n - t0 < TB ? n - t0 : TB);
  const int npub = nodata ? 0 : n;                       // tokens the publication accounts for
  const uint32_t fr = smem_u32(wts_sm);
  const size_t fbytes = (size_t)tb * H * D * 2;          // one tensor's bytes in this block
  const uint32_t rows = fr + (uint32_t)(2 * (size_t)TB * H * D * 2);
  const int per = tb * H * CH;                           // chunks of one tensor in this block
  // The next position this write will publish, as a hint for the kernels
  // after it; then they may start (this kernel writes no caller buffer: the
  // host's record of caller buffers written by kernels in flight carries
  // over it).
  if (blockIdx.x == 0 && threadIdx.x == 0)
    st_relaxed_gpu(r.state + ST_NEXT_POS_HINT, ld_relaxed_gpu(r.state + ST_NEXT_POS) + npub);
  griddep_launch_dependents();
  // The frame before the wait for the preceding kernel, unless the host
  // found that a kernel still in flight may write it.
  if (late) griddep_wait();
  const uint8_t* kb = reinterpret_cast<const uint8_t*>(k) + (size_t)t0 * H * D * 2;
  const uint8_t* vb = reinterpret_cast<const uint8_t*>(v) + (size_t)t0 * H * D * 2;
  for (size_t i = (size_t)threadIdx.x * 16; i < fbytes; i += kThreads * 16) {
    cp_async16(fr + (uint32_t)i, kb + i);
    cp_async16(fr + (uint32_t)(fbytes + i), vb + i);
  }
  // table rows: 16-byte piece q of chunk c of token tl
  auto stage_rows = [&](int next) {
    for (int i = threadIdx.x; i < tb * CH * 4; i += kThreads) {
      const int tl = i / (CH * 4), c = (i / 4) % CH, q = i % 4;
      const int p = pos ? rope_pos(r, pos, t0 + tl, 8 * c) : next + t0 + tl;
      if (p >= 0 && p < r.max_pos)
        cp_async16(rows + (uint32_t)((tl * D + 16 * c + 4 * q) * 4), r.table + (size_t)p * D + 16 * c + 4 * q);
    }
  };
  // Every chunk rotated (keys), scaled and converted, its codes written over
  // the first half of its own 32 bytes (each thread reads its chunks before
  // it writes them).  A key chunk whose position is outside the table keeps
  // whatever it holds: the copy below skips it.
  auto encode = [&](int next) {
    for (int i = threadIdx.x; i < 2 * per; i += kThreads) {
      const int isv = i >= per;
      const int w = isv ? i - per : i;
      const int chunk = w % CH, th = w / CH;
      const int h = th % H, tl = th / H;
      uint8_t* src = wts_sm + (size_t)isv * fbytes + ((size_t)th * D + 16 * chunk) * 2;
      float x[16];
      unpack_bf16x16(*reinterpret_cast<const uint4*>(src), *reinterpret_cast<const uint4*>(src + 16), x);
      if (!isv) {
        const int p = pos ? rope_pos(r, pos, t0 + tl, 8 * chunk) : next + t0 + tl;
        if (p < 0 || p >= r.max_pos) continue;
        const float4* rw = reinterpret_cast<const float4*>(wts_sm + (size_t)(rows - fr) + (size_t)(tl * D + 16 * chunk) * 4);
        const float4 cs[4] = {rw[0], rw[1], rw[2], rw[3]};
        rope_pinned(x, cs);
      }
      const float inv = r.scales[(isv ? 3 : 2) * H + h];
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] = __fmul_rn(x[e], inv);
      *reinterpret_cast<uint4*>(src) = pack_e4m3x16(x);
    }
  };
  const bool pre = idle && !pos && !late;
  int nv0 = 0;
  unsigned long long total0 = 0;
  if (!pos) {
    if (threadIdx.x == 0) {
      if (pre) {
        const int4 st = ld_relaxed_gpu_v4(r.state);   // head, n_valid, total lo, hi
        s_head = st.x;
        nv0 = st.y;
        total0 = (unsigned long long)(unsigned)st.w << 32 | (unsigned)st.z;
        s_next = ld_relaxed_gpu(r.state + ST_NEXT_POS);
        s_guess = s_next;
      } else {
        s_guess = ld_relaxed_gpu(r.state + ST_NEXT_POS);
      }
    }
    __syncthreads();
    stage_rows(s_guess);
  }
  cp_async_commit();
  if (!pos) {
    // (the scales are written only by a calibration, which never overlaps
    // a following kernel)
    cp_async_wait_all();
    __syncthreads();
    encode(s_guess);
  }
  if (!pre) {
    // The ring (state, cache, positions) only after the preceding kernel.
    griddep_wait();
    if (threadIdx.x == 0) {
      const int4 st = __ldcg(reinterpret_cast<const int4*>(r.state));   // head, n_valid, total lo, hi
      s_head = st.x;
      nv0 = st.y;
      total0 = (unsigned long long)(unsigned)st.w << 32 | (unsigned)st.z;
      s_next = __ldcg(r.state + ST_NEXT_POS);
    }
  }
  __syncthreads();
  if (pos || s_next != s_guess) {
    // explicit positions, or a wrong guess: rows and codes after the wait
    // (a wrong guess encoded the frame in place: load it again first)
    if (!pos) {
      for (size_t i = (size_t)threadIdx.x * 16; i < fbytes; i += kThreads * 16) {
        cp_async16(fr + (uint32_t)i, kb + i);
        cp_async16(fr + (uint32_t)(fbytes + i), vb + i);
      }
    }
    stage_rows(s_next);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    encode(s_next);
  }
  __syncthreads();
  // Thread 0 plans the state after this write (a slot-position load or two)
  // while the other threads copy the codes into their slots: thread c + 1
  // takes (tensor, head, chunk) c for every token of the block.
  WritePlan plan{};
  if (threadIdx.x == 0) plan = plan_write(r, pos, s_head, nv0, total0, s_next, npub);
  for (int c = (int)threadIdx.x - 1; threadIdx.x > 0 && c < 2 * H * CH; c += kThreads - 1) {
    const int isv = c >= H * CH;
    const int rem = isv ? c - H * CH : c;
    const int h = rem / CH, chunk = rem % CH;
    uint8_t* const base = (isv ? r.v : r.k) + (size_t)h * C * D + chunk * 16;
    const uint8_t* src = wts_sm + (size_t)isv * fbytes + ((size_t)h * D + 16 * chunk) * 2;
    for (int tl = 0; tl < tb; ++tl, src += (size_t)H * D * 2) {
      const int t = t0 + tl;
      // head < C and t < n <= C - P: at most one wrap, which skips the prefix
      int slot = s_head + t;
      if (slot >= C) slot -= C - r.P;
      if (!isv) {
        const int p = pos ? rope_pos(r, pos, t, 8 * chunk) : s_next + t;
        if (h == 0 && chunk == 0) r.slot_pos[slot] = p;
        if (p < 0 || p >= r.max_pos) {
          atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
          continue;
        }
      }
      *reinterpret_cast<uint4*>(base + (size_t)slot * D) = *reinterpret_cast<const uint4*>(src);
    }
  }
  __syncthreads();
  // The last block to finish publishes the state (planned at the start, so
  // it reads nothing another block wrote and no fence precedes the ticket).
  if (threadIdx.x == 0) {
    const int tk = atomicAdd(r.state + ST_TICKET_WRITE, 1);
    if (tk == (int)gridDim.x - 1) store_write_plan(r, plan);
  }
  // (one block waiting is enough to keep the grid from completing before
  // the preceding kernel; the others leave now and free their SMs)
  if (pre && blockIdx.x == 0) griddep_wait();
}

// Many rings of one shape in one launch, as a bulk-copy pipeline.  The work
// is cut into units of whole tokens (TU = RU / H tokens of all H heads, RU =
// 8192 / D rows, 16 KB of bf16) -- or, when one token's heads exceed RU rows,
// of one token's heads in groups of RU -- so every unit is a contiguous run of
// the frame; each ring's key and value units alternate, and block b of G
// takes the b-th G-th of the unit list.  One producer thread streams each
// unit into a shared-memory stage with cp.async.bulk: the rows, and for keys
// the RoPE rows of the unit's tokens (one copy when their positions are
// consecutive); sixteen consumer warps rotate, scale and quantise them (the
// single-ring write's arithmetic, byte for byte) and store the codes.
//
// A unit has RU x D/16 = 512 places of 16 values; consumer thread `tid`
// keeps place tid in every unit: row tid / CH (CH = D/16), lane k = tid % CH
// in the row, and of the row's D/8 runs of 8 values the runs k and k + CH.
// A quarter-warp then reads 128 contiguous input bytes and writes 64
// contiguous output bytes per run; all shared-memory offsets are constants of
// the thread, so a unit costs its arithmetic and little else.
//
// Stage layout: [TU][HU][D] bf16 | [TU][D] fp32 RoPE rows | the unit's token
// positions (explicit positions only), head and next_pos.
constexpr int kWmConsumerWarps = 16;
constexpr int kWmThreads = 32 * (kWmConsumerWarps + 1);  // one block per SM at 120 registers
constexpr int kWmStageBudget = 200 * 1024;               // bytes of stages per block
constexpr int kWmMaxStages = 16;
constexpr uint64_t kWmWaitLimitNs = 1000000000ull;       // one second
static_assert(32 * kWmConsumerWarps == 512, "one place per consumer thread and unit");

struct WmGeom {
  int HU, TU, NG, tab_off, pos_off, stage_bytes, stages;
};
__host__ __device__ inline WmGeom wm_geom(int H, int D) {
  WmGeom g;
  const int RU = 8192 / D;
  if (H <= RU) {
    g.HU = H;
    g.TU = RU / H;
    g.NG = 1;
  } else {
    g.HU = RU;
    g.TU = 1;
    g.NG = (H + RU - 1) / RU;
  }
  g.tab_off = g.TU * g.HU * D * 2;
  g.pos_off = g.tab_off + g.TU * D * 4;
  g.stage_bytes = (g.pos_off + (g.TU + 2) * 4 + 127) / 128 * 128;
  g.stages = kWmStageBudget / g.stage_bytes;
  if (g.stages > kWmMaxStages) g.stages = kWmMaxStages;
  if (g.stages < 2) g.stages = 2;
  return g;
}
// units per kind and ring
__host__ __device__ inline long long wm_units(const WmGeom& g, int n) {
  return (long long)((n + g.TU - 1) / g.TU) * g.NG;
}

// One consumer thread's place in one unit: read its two runs (and for keys
// their RoPE words) from the stage, hand the stage back (once per warp),
// then rotate, scale, quantise and store.
template <int D, bool KEY>
__device__ __forceinline__ void wm_place(const RingDev& r, const uint8_t* st, const int* hdr, bool act, bool expl,
                                         int in_off, int tab_off, int dt, int k, int h, int slot, int p_impl,
                                         float inv, uint32_t empty_bar, int lane) {
  constexpr int CH = D / 16;
  uint4 in[2];
  float4 cs[2][2];
  int p = 0;
  bool ok = act;
  if (act) {
#pragma unroll
    for (int j = 0; j < 2; ++j) in[j] = *reinterpret_cast<const uint4*>(st + in_off + 16 * CH * j);
    if (KEY) {
      p = expl ? hdr[dt] : p_impl;
      ok = p >= 0 && p < r.max_pos;
      if (ok) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          cs[j][0] = *reinterpret_cast<const float4*>(st + tab_off + 32 * CH * j);
          cs[j][1] = *reinterpret_cast<const float4*>(st + tab_off + 32 * CH * j + 16);
        }
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
  if (!act) return;
  if (KEY) {
    if (!ok) atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
    if (h == 0 && k == 0) r.slot_pos[slot] = p;
    if (!ok) return;
  }
  uint8_t* out = (KEY ? r.k : r.v) + ((size_t)h * r.C + slot) * D + 8 * k;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t wv[4] = {in[j].x, in[j].y, in[j].z, in[j].w};
    uint32_t code[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float x[4] = {__uint_as_float(wv[2 * i] << 16), __uint_as_float(wv[2 * i] & 0xFFFF0000u),
                    __uint_as_float(wv[2 * i + 1] << 16), __uint_as_float(wv[2 * i + 1] & 0xFFFF0000u)};
      if (KEY) rope_pinned2(x, cs[j][i]);
#pragma unroll
      for (int c = 0; c < 4; ++c) x[c] = __fmul_rn(x[c], inv);
      code[i] = (uint32_t)f32x2_to_e4m3x2(x[0], x[1]) | ((uint32_t)f32x2_to_e4m3x2(x[2], x[3]) << 16);
    }
    *reinterpret_cast<uint2*>(out + 8 * CH * j) = make_uint2(code[0], code[1]);
  }
}

template <int D>
__global__ void __maxnreg__(120) k_write_many(const __grid_constant__ WriteMany b, int count, int n) {
  constexpr int CH = D / 16;
  extern __shared__ __align__(128) uint8_t wsm[];
  __shared__ __align__(8) uint64_t full[kWmMaxStages], empty[kWmMaxStages];
  __shared__ int s_abort;
  __shared__ int s_warps_done[kMaxBatch];   // per ring: consumer warps of this block past their last unit of it
  const int H = b.r[0].H, C = b.r[0].C;
  const WmGeom g = wm_geom(H, D);
  const int S = g.stages;
  const long long ur = wm_units(g, n);
  const long long up = 2 * ur;  // units per ring: key and value units alternate
  const long long total = up * count;
  const long long u_begin = total * blockIdx.x / gridDim.x;
  const long long u_end = total * (blockIdx.x + 1) / gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kWmConsumerWarps);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  for (int i = threadIdx.x; i < kMaxBatch; i += blockDim.x) s_warps_done[i] = 0;
  // the next position each ring will have, as a hint for the kernels after
  if (blockIdx.x == 0 && threadIdx.x < count)
    st_relaxed_gpu(b.r[threadIdx.x].state + ST_NEXT_POS_HINT, ld_relaxed_gpu(b.r[threadIdx.x].state + ST_NEXT_POS) + n);
  griddep_launch_dependents();
  griddep_wait();  // the rings are touched only after the preceding kernel
  __syncthreads();
  if (u_begin >= u_end) return;
  volatile int* abort = &s_abort;
  const uint32_t base = smem_u32(wsm);
  // unit u = ring * up + jv; jv = 2 (tb NG + hg) + (1 for values)
  int ring = (int)(u_begin / up), jv = (int)(u_begin % up);
  int tb = (jv >> 1) / g.NG, hg = (jv >> 1) % g.NG;
  int s = 0;
  uint32_t ph = 0;

  if (warp == kWmConsumerWarps) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;
    int cur = -1, head = 0, next = 0;
    long long i = 0;
    for (long long u = u_begin; u < u_end; ++u, ++i) {
      if (i >= S && !mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1, abort, kWmWaitLimitNs)) break;
      const bool isv = jv & 1;
      const int t0 = tb * g.TU;
      const int ntok = min(g.TU, n - t0), nh = min(g.HU, H - hg * g.HU);
      const RingDev& r = b.r[ring];
      if (ring != cur) {
        cur = ring;
        head = __ldcg(r.state + ST_HEAD);
        next = __ldcg(r.state + ST_NEXT_POS);
      }
      int* hdr = reinterpret_cast<int*>(wsm + (size_t)s * g.stage_bytes + g.pos_off);
      hdr[g.TU] = head;
      hdr[g.TU + 1] = next;
      const uint32_t in_bytes = (uint32_t)(ntok * nh) * D * 2;
      uint32_t bytes = in_bytes;
      const int32_t* pos = b.pos[ring];
      const int p0 = next + t0;
      const bool one_copy = !isv && !pos && p0 >= 0 && p0 + ntok <= r.max_pos;
      if (!isv) {
        if (one_copy) {
          bytes += (uint32_t)ntok * D * 4;
        } else {
          for (int t = 0; t < ntok; ++t) {
            int p;
            if (r.pt) {   // 3-D: a token is valid when all three coordinates are
              const int32_t* q3 = pos + 3 * (t0 + t);
              const int a0 = __ldg(q3), a1 = __ldg(q3 + 1), a2 = __ldg(q3 + 2);
              const bool ok3 = a0 >= 0 && a0 < r.max_pos && a1 >= 0 && a1 < r.max_pos && a2 >= 0 && a2 < r.max_pos;
              p = ok3 ? a0 : -1;
            } else {
              p = pos ? __ldg(pos + t0 + t) : p0 + t;
            }
            hdr[t] = p;
            if (p >= 0 && p < r.max_pos) bytes += D * 4;
          }
        }
      }
      const uint32_t fb = smem_u32(&full[s]);
      const uint32_t sa = base + (uint32_t)s * g.stage_bytes;
      mbar_arrive_expect_tx(fb, bytes);
      bulk_load(sa, (isv ? b.v[ring] : b.k[ring]) + ((size_t)t0 * H + hg * g.HU) * D, in_bytes, fb);
      if (one_copy) {
        bulk_load(sa + g.tab_off, r.table + (size_t)p0 * D, (uint32_t)ntok * D * 4, fb);
      } else if (!isv) {
        for (int t = 0; t < ntok; ++t) {
          const int p = hdr[t];
          if (!(p >= 0 && p < r.max_pos)) continue;
          const uint32_t dst = sa + g.tab_off + t * D * 4;
          if (r.pt) {   // 3-D: each section's cos/sin from its own coordinate's row
            const int32_t* q3 = pos + 3 * (t0 + t);
            const int lo[3] = {0, r.pt, r.pt + r.py}, m[3] = {r.pt, r.py, D / 2 - r.pt - r.py};
            for (int a = 0; a < 3; ++a)
              if (m[a] > 0)
                bulk_load(dst + 8 * lo[a], r.table + (size_t)__ldg(q3 + a) * D + 2 * lo[a], (uint32_t)(8 * m[a]), fb);
          } else {
            bulk_load(dst, r.table + (size_t)p * D, D * 4, fb);
          }
        }
      }
      if (++s == S) {
        s = 0;
        ph ^= 1;
      }
      if (++jv == (int)up) {
        jv = 0;
        tb = hg = 0;
        ++ring;
      } else if (!(jv & 1) && ++hg == g.NG) {
        hg = 0;
        ++tb;
      }
    }
    if (*abort) {
      // leave no copy in flight: wait (bounded) for the stages issued last
      int no_abort = 0;
      for (long long q = i > S ? i - S : 0; q < i; ++q)
        mbar_wait_bounded(smem_u32(&full[q % S]), (uint32_t)((q / S) & 1), &no_abort, kWmWaitLimitNs);
      atomicOr(reinterpret_cast<unsigned*>(b.r[cur < 0 ? 0 : cur].state + ST_ERROR), KVRING_DEVERR_TIMEOUT);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int row = threadIdx.x / CH, k = threadIdx.x % CH;
  const int dt = row / g.HU, hl = row % g.HU;
  const int in_off = row * D * 2 + 16 * k;
  const int tab_off = g.tab_off + dt * D * 4 + 32 * k;
  float invk = 1.0f, invv = 1.0f;
  int done = 0, head = 0, next = 0, cur = -1, cur_hg = -1;
  for (long long u = u_begin; u < u_end; ++u) {
    if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abort, kWmWaitLimitNs)) {
      if (lane == 0) atomicOr(reinterpret_cast<unsigned*>(b.r[ring].state + ST_ERROR), KVRING_DEVERR_TIMEOUT);
      break;
    }
    const bool isv = jv & 1;
    const int t0 = tb * g.TU;
    const int ntok = min(g.TU, n - t0), nh = min(g.HU, H - hg * g.HU);
    const RingDev& r = b.r[ring];
    const int h = hg * g.HU + hl;
    if (ring != cur || hg != cur_hg) {
      cur = ring;
      cur_hg = hg;
      const int hc = min(h, H - 1);
      invk = r.scales[2 * H + hc];
      invv = r.scales[3 * H + hc];
    }
    const uint8_t* st = wsm + (size_t)s * g.stage_bytes;
    const int* hdr = reinterpret_cast<const int*>(st + g.pos_off);
    head = hdr[g.TU];
    next = hdr[g.TU + 1];
    const bool act = dt < ntok && hl < nh;
    int slot = head + t0 + dt;
    if (slot >= C) slot -= C - r.P;   // at most one wrap, which skips the prefix
    const uint32_t eb = smem_u32(&empty[s]);
    if (isv)
      wm_place<D, false>(r, st, hdr, act, false, in_off, tab_off, dt, k, h, slot, 0, invv, eb, lane);
    else
      wm_place<D, true>(r, st, hdr, act, b.pos[ring] != nullptr, in_off, tab_off, dt, k, h, slot, next + t0 + dt,
                        invk, eb, lane);
    ++done;
    if (++s == S) {
      s = 0;
      ph ^= 1;
    }
    // Ring done for this block: every consumer warp adds its units to the
    // ring's ticket; the warp that completes (consumer warps) x (units per
    // ring) publishes the new ring state, planned from the state as it still
    // stands and this frame's own positions for the slots this frame writes,
    // so it reads nothing another warp wrote and no fence precedes the
    // tickets (the next kernel sees the cache through this grid's end).
    const bool ring_end = jv + 1 == (int)up;
    if (ring_end || u + 1 == u_end) {
      __syncwarp();
      // (every consumer warp takes part in every unit, so the block's warps
      // count themselves in shared memory and its last one takes the ring's
      // ticket for all of them: one global atomic per block and ring, and
      // no warp ever waits for another)
      if (lane == 0 && atomicAdd(&s_warps_done[ring], 1) == kWmConsumerWarps - 1) {
        const int tk = atomicAdd(r.state + ST_TICKET_WRITE, done * kWmConsumerWarps);
        if (tk + done * kWmConsumerWarps == kWmConsumerWarps * (int)up) {
          const int4 st4 = __ldcg(reinterpret_cast<const int4*>(r.state));   // head, n_valid, total lo, hi
          const unsigned long long total0 = (unsigned long long)(unsigned)st4.w << 32 | (unsigned)st4.z;
          store_write_plan(r, plan_write(r, b.pos[ring], head, st4.y, total0, next, n));
        }
      }
      done = 0;
    }
    if (ring_end) {
      jv = 0;
      tb = hg = 0;
      ++ring;
    } else if (!(++jv & 1) && ++hg == g.NG) {
      hg = 0;
      ++tb;
    }
  }
}

// ---------------------------------------------------------------- delta ---
// Delta rotation of one or many rings as a bulk-copy pipeline.  A unit is
// RU = 16384 / D consecutive slots of one head of one ring, i.e. one
// contiguous 16 KB run of key codes; ring r contributes H x ceil(C / RU)
// units (sized for a full ring: rows at or past the fill level are neither
// copied nor written).  Block b of G takes the b-th G-th of the unit list.
// One producer thread resolves each ring's delta and fill level from its
// state and streams the unit's filled rows into a shared-memory stage with
// cp.async.bulk; sixteen consumer warps decode, rotate and re-encode them
// (the single-ring arithmetic, byte for byte) and store the codes back in
// place with 16-byte stores.  Consumer thread `tid` keeps chunk tid % CH of
// rows tid / CH + j * (512 / CH), so its table values are fixed per ring.
constexpr int kDpConsumerWarps = 16;
constexpr int kDpThreads = 32 * (kDpConsumerWarps + 1);
constexpr int kDpUnitBytes = 16384;
constexpr int kDpStages = 12;
constexpr int kDpSmemBytes = kDpStages * kDpUnitBytes;
static_assert(32 * kDpConsumerWarps == 512, "512 consumer threads");

template <int D>
__global__ void __launch_bounds__(kDpThreads, 1) k_delta_pipe(const __grid_constant__ DeltaMany b, int count,
                                                              int delta_arg) {
  constexpr int CH = D / 16;             // 16-byte chunks per row
  constexpr int RU = kDpUnitBytes / D;   // rows per unit
  constexpr int RSTEP = 512 / CH;        // rows between a thread's chunks
  constexpr int PASSES = RU / RSTEP;
  static_assert(PASSES * RSTEP == RU && RU <= 512, "unit shape");
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kDpStages], empty[kDpStages];
  __shared__ int hdr[kDpStages][2];  // filled rows of the unit, its ring's delta (-1: none)
  __shared__ int s_abort;
  __shared__ int s_warps_done[kMaxBatch];   // per ring: consumer warps of this block past their last unit of it
  const int H = b.r[0].H, C = b.r[0].C;
  const int P = b.r[0].P;                  // pinned prefix: never rotated
  const int runs = (C - P + RU - 1) / RU;  // runs of rolling slots per head
  const long long up = (long long)H * runs;  // units per ring
  const long long total = up * count;
  const long long u_begin = total * blockIdx.x / gridDim.x;
  const long long u_end = total * (blockIdx.x + 1) / gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDpStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kDpConsumerWarps);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  for (int i = threadIdx.x; i < kMaxBatch; i += blockDim.x) s_warps_done[i] = 0;
  griddep_launch_dependents();
  griddep_wait();  // the rings are touched only after the preceding kernel
  __syncthreads();
  if (u_begin >= u_end) return;
  volatile int* abort = &s_abort;
  const uint32_t base = smem_u32(dsm);
  // unit u = ring * up + h * runs + run
  int ring = (int)(u_begin / up);
  int h = (int)(u_begin % up) / runs, run = (int)(u_begin % up) % runs;
  int s = 0;
  uint32_t ph = 0;

  if (warp == kDpConsumerWarps) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;
    int cur = -1, nv = 0, d = -1;
    long long i = 0;
    for (long long u = u_begin; u < u_end; ++u, ++i) {
      if (i >= kDpStages && !mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1, abort, kWmWaitLimitNs)) break;
      const RingDev& r = b.r[ring];
      if (ring != cur) {
        cur = ring;
        nv = __ldcg(r.state + ST_NVALID);
        d = delta_arg;
        if (d == KVRING_DELTA_TO_OLDEST) {
          // the oldest rolling position, less the prefix's end with a prefix
          const int oldest = __ldcg(r.state + ST_OLDEST_POS);
          if (nv <= P || oldest == kEmptyPos) {
            d = 0;
          } else if (P == 0) {
            d = oldest;
          } else {
            const int gap = oldest - __ldcg(r.state + ST_PREFIX_END);
            d = gap > 0 ? gap : 0;
          }
        }
        if (d < 0 || d >= r.max_pos) {
          atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_DELTA);
          d = -1;  // skip the rotation entirely
        }
      }
      const int r0 = P + run * RU;
      int rows = d > 0 ? nv - r0 : 0;
      rows = rows < 0 ? 0 : (rows > RU ? RU : rows);
      hdr[s][0] = rows;
      hdr[s][1] = d;
      const uint32_t fb = smem_u32(&full[s]);
      mbar_arrive_expect_tx(fb, (uint32_t)rows * D);
      if (rows > 0)
        bulk_load(base + (uint32_t)s * kDpUnitBytes, r.k + ((size_t)h * C + r0) * D, (uint32_t)rows * D, fb);
      if (++s == kDpStages) {
        s = 0;
        ph ^= 1;
      }
      if (++run == runs) {
        run = 0;
        if (++h == H) {
          h = 0;
          ++ring;
        }
      }
    }
    if (*abort) {
      // leave no copy in flight: wait (bounded) for the stages issued last
      int no_abort = 0;
      for (long long q = i > kDpStages ? i - kDpStages : 0; q < i; ++q)
        mbar_wait_bounded(smem_u32(&full[q % kDpStages]), (uint32_t)((q / kDpStages) & 1), &no_abort,
                          kWmWaitLimitNs);
      atomicOr(reinterpret_cast<unsigned*>(b.r[cur < 0 ? 0 : cur].state + ST_ERROR), KVRING_DEVERR_TIMEOUT);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int k = threadIdx.x % CH, row0 = threadIdx.x / CH;
  // with 3-D RoPE only the temporal pairs turn: this thread's 8 pairs are
  // temporal or not for every row (sections are whole chunks of 8 pairs)
  const bool turns = b.r[0].pt == 0 || 8 * k < b.r[0].pt;
  float c[8], sn[8];  // cos / sin of this thread's 8 pairs at the ring's delta
  int cur_d = 0, done = 0, d = -1;
  for (long long u = u_begin; u < u_end; ++u) {
    if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abort, kWmWaitLimitNs)) {
      if (lane == 0) atomicOr(reinterpret_cast<unsigned*>(b.r[ring].state + ST_ERROR), KVRING_DEVERR_TIMEOUT);
      break;
    }
    const int rows = hdr[s][0];
    d = hdr[s][1];
    uint4 in[PASSES];
    const uint8_t* st = dsm + (size_t)s * kDpUnitBytes;
#pragma unroll
    for (int j = 0; j < PASSES; ++j)
      if (row0 + j * RSTEP < rows) in[j] = *reinterpret_cast<const uint4*>(st + (row0 + j * RSTEP) * D + 16 * k);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    const RingDev& r = b.r[ring];
    const int r0 = P + run * RU;
    if (rows > 0 && turns) {
      if (d != cur_d) {
        cur_d = d;
        const float4* t = reinterpret_cast<const float4*>(r.table + (size_t)d * D + 16 * k);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 cs = __ldg(t + i);  // (c, s) of pairs 8k + 2i and 8k + 2i + 1
          c[2 * i] = cs.x;
          sn[2 * i] = cs.y;
          c[2 * i + 1] = cs.z;
          sn[2 * i + 1] = cs.w;
        }
      }
#pragma unroll
      for (int j = 0; j < PASSES; ++j) {
        const int row = row0 + j * RSTEP;
        if (row >= rows) continue;
        const uint32_t w[4] = {in[j].x, in[j].y, in[j].z, in[j].w};
        float y[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 a = e4m3x2_to_f32x2((uint16_t)(w[i] & 0xFFFF));
          const float2 bb = e4m3x2_to_f32x2((uint16_t)(w[i] >> 16));
          y[4 * i + 0] = __fadd_rn(__fmul_rn(a.x, c[2 * i]), __fmul_rn(a.y, sn[2 * i]));
          y[4 * i + 1] = __fsub_rn(__fmul_rn(a.y, c[2 * i]), __fmul_rn(a.x, sn[2 * i]));
          y[4 * i + 2] = __fadd_rn(__fmul_rn(bb.x, c[2 * i + 1]), __fmul_rn(bb.y, sn[2 * i + 1]));
          y[4 * i + 3] = __fsub_rn(__fmul_rn(bb.y, c[2 * i + 1]), __fmul_rn(bb.x, sn[2 * i + 1]));
        }
        *reinterpret_cast<uint4*>(r.k + ((size_t)h * C + r0 + row) * D + 16 * k) = pack_e4m3x16(y);
      }
    }
    if (rows > 0 && h == 0 && (int)threadIdx.x < rows) r.slot_pos[r0 + threadIdx.x] -= d;
    ++done;
    if (++s == kDpStages) {
      s = 0;
      ph ^= 1;
    }
    // Ring done for this block: every consumer warp adds its units to the
    // ring's ticket; the warp that completes (consumer warps) x (units per
    // ring) publishes the new positions.
    const bool ring_end = h == H - 1 && run == runs - 1;
    if (ring_end || u + 1 == u_end) {
      __syncwarp();
      // No fence before the ticket: the publication reads nothing the
      // other warps wrote (every block's producer read this ring's state
      // before any of its units could finish), and the next kernel sees the
      // rotated keys and positions through this grid's end.  Every consumer
      // warp takes part in every unit, so the block's warps count themselves
      // in shared memory and its last one takes the ring's ticket for all of
      // them (no warp ever waits for another).
      if (lane == 0 && atomicAdd(&s_warps_done[ring], 1) == kDpConsumerWarps - 1) {
        const int tk = atomicAdd(r.state + ST_TICKET_DELTA, done * kDpConsumerWarps);
        if (tk + done * kDpConsumerWarps == kDpConsumerWarps * (int)up) {
          __threadfence();
          if (d >= 0) {
            r.state[ST_NEXT_POS] -= d;
            st_relaxed_gpu(r.state + ST_NEXT_POS_HINT, r.state[ST_NEXT_POS]);
            if (r.state[ST_OLDEST_POS] != kEmptyPos) r.state[ST_OLDEST_POS] -= d;
            r.state[ST_LAST_DELTA] = d;
          }
          r.state[ST_TICKET_DELTA] = 0;
          __threadfence();
        }
      }
      done = 0;
    }
    if (++run == runs) {
      run = 0;
      if (++h == H) {
        h = 0;
        ++ring;
        cur_d = 0;
      }
    }
  }
}

// The delta rotation of one ring: one block per (head, run of 128 rolling
// slots), each thread four (d = 128) or two (d = 64) 16-byte chunks of the
// run's key rows, all loaded before any arithmetic; the same rotation and
// re-encoding as the batched pipeline (decoded codes turned by -delta with
// the table row of delta, each product and sum rounded to fp32), the same
// delta rule and the same state publication by the last block.  One ring's
// key cache (7.4 MB at 10 heads x 5,788 slots x 128) is too small to fill a
// pipeline of one block per SM; independent blocks keep more rows in
// flight.  idle: no kernel that may still run reads or writes this ring
// (the host keeps track); then the state read before the wait is final and
// the whole rotation happens before it, block 0 then waiting so the
// stream's kernels still complete in order.
constexpr int kDeltaRows = 128;
template <int D>
__global__ void __launch_bounds__(kThreads) k_delta_one(RingDev r, int delta_arg, int idle) {
  constexpr int CH = D / 16;                         // 16-byte chunks per row
  constexpr int RSTEP = kThreads / CH;               // rows between a thread's chunks
  constexpr int PASSES = kDeltaRows / RSTEP;         // 4 (d = 128) or 2 (d = 64)
  static_assert(PASSES * RSTEP == kDeltaRows, "block shape");
  __shared__ int s_d, s_nv;
  const int C = r.C, P = r.P;
  const int runs = (C - P + kDeltaRows - 1) / kDeltaRows;
  const int h = (int)blockIdx.x / runs, run = (int)blockIdx.x % runs;
  const int r0 = P + run * kDeltaRows;
  griddep_launch_dependents();
  if (!idle) griddep_wait();   // the ring is touched only after the preceding kernel
  if (threadIdx.x == 0) {
    auto load = [&](int w) { return idle ? ld_relaxed_gpu(r.state + w) : __ldcg(r.state + w); };
    const int nv = load(ST_NVALID);
    int d = delta_arg;
    if (d == KVRING_DELTA_TO_OLDEST) {
      // the oldest rolling position, less the prefix's end with a prefix
      const int oldest = load(ST_OLDEST_POS);
      if (nv <= P || oldest == kEmptyPos) {
        d = 0;
      } else if (P == 0) {
        d = oldest;
      } else {
        const int gap = oldest - load(ST_PREFIX_END);
        d = gap > 0 ? gap : 0;
      }
    }
    if (d < 0 || d >= r.max_pos) {
      if (blockIdx.x == 0) atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_DELTA);
      d = -1;   // skip the rotation entirely
    }
    s_d = d;
    s_nv = nv;
  }
  __syncthreads();
  const int d = s_d;
  int rows = d > 0 ? s_nv - r0 : 0;
  rows = rows < 0 ? 0 : (rows > kDeltaRows ? kDeltaRows : rows);
  const int k = (int)threadIdx.x % CH, row0 = (int)threadIdx.x / CH;
  // with 3-D RoPE only the temporal pairs turn: this thread's 8 pairs are
  // temporal or not for every row (sections are whole chunks of 8 pairs)
  const bool turns = r.pt == 0 || 8 * k < r.pt;
  if (rows > 0 && turns) {
    uint8_t* base = r.k + ((size_t)h * C + r0) * D + 16 * k;
    uint4 in[PASSES];
#pragma unroll
    for (int j = 0; j < PASSES; ++j)
      if (row0 + j * RSTEP < rows) in[j] = __ldcg(reinterpret_cast<const uint4*>(base + (size_t)(row0 + j * RSTEP) * D));
    float c[8], sn[8];   // cos / sin of this thread's 8 pairs at delta
    const float4* t = reinterpret_cast<const float4*>(r.table + (size_t)d * D + 16 * k);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 cs = __ldg(t + i);   // (c, s) of pairs 8k + 2i and 8k + 2i + 1
      c[2 * i] = cs.x;
      sn[2 * i] = cs.y;
      c[2 * i + 1] = cs.z;
      sn[2 * i + 1] = cs.w;
    }
#pragma unroll
    for (int j = 0; j < PASSES; ++j) {
      const int row = row0 + j * RSTEP;
      if (row >= rows) continue;
      const uint32_t w[4] = {in[j].x, in[j].y, in[j].z, in[j].w};
      float y[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = e4m3x2_to_f32x2((uint16_t)(w[i] & 0xFFFF));
        const float2 bb = e4m3x2_to_f32x2((uint16_t)(w[i] >> 16));
        y[4 * i + 0] = __fadd_rn(__fmul_rn(a.x, c[2 * i]), __fmul_rn(a.y, sn[2 * i]));
        y[4 * i + 1] = __fsub_rn(__fmul_rn(a.y, c[2 * i]), __fmul_rn(a.x, sn[2 * i]));
        y[4 * i + 2] = __fadd_rn(__fmul_rn(bb.x, c[2 * i + 1]), __fmul_rn(bb.y, sn[2 * i + 1]));
        y[4 * i + 3] = __fsub_rn(__fmul_rn(bb.y, c[2 * i + 1]), __fmul_rn(bb.x, sn[2 * i + 1]));
      }
      *reinterpret_cast<uint4*>(base + (size_t)row * D) = pack_e4m3x16(y);
    }
  }
  if (rows > 0 && h == 0 && (int)threadIdx.x < rows) r.slot_pos[r0 + threadIdx.x] -= d;
  __syncthreads();
  // The last block publishes (no fence before the ticket: the publication
  // reads nothing another block wrote, and the next kernel sees the rotated
  // keys and positions through this grid's end).
  if (threadIdx.x == 0) {
    const int tk = atomicAdd(r.state + ST_TICKET_DELTA, 1);
    if (tk == (int)gridDim.x - 1) {
      __threadfence();
      if (d >= 0) {
        r.state[ST_NEXT_POS] -= d;
        st_relaxed_gpu(r.state + ST_NEXT_POS_HINT, r.state[ST_NEXT_POS]);
        if (r.state[ST_OLDEST_POS] != kEmptyPos) r.state[ST_OLDEST_POS] -= d;
        r.state[ST_LAST_DELTA] = d;
      }
      r.state[ST_TICKET_DELTA] = 0;
      __threadfence();
    }
  }
  if (idle && blockIdx.x == 0) griddep_wait();
}

// ------------------------------------------------------- legacy upkeep ---
// The upkeep the ring replaced ("Where the Time Went": every call re-applied
// RoPE to every cached key, re-quantised the cache and shifted the window by
// copying it), kept as the comparison path.  The window holds the unrotated
// bf16 keys and values of the last C tokens in time order ([C][H][d], token-
// major like the frames).  Ring state words reused: n_valid = tokens in the
// window, next_pos = tokens seen (the next token's position).
//
// Pass 1, one thread per 16-value chunk of every (window slot, head): copy
// the shifted window (the oldest tokens leave once it is full, the frame
// enters at its end) into the other window buffer, and take each head's
// maximum of the rotated keys (RoPE at position base + slot) and of the
// values; the last block turns the maxima into scales.
template <int D>
__global__ void __launch_bounds__(kThreads) k_legacy_shift(RingDev r, const uint16_t* __restrict__ wk_in,
                                                           const uint16_t* __restrict__ wv_in,
                                                           uint16_t* __restrict__ wk_out, uint16_t* __restrict__ wv_out,
                                                           const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                                           int n) {
  constexpr int CH = D / 16;
  __shared__ int s_fill, s_total, s_last;
  if (threadIdx.x == 0) {
    s_fill = __ldcg(r.state + ST_NVALID);
    s_total = __ldcg(r.state + ST_NEXT_POS);
  }
  __syncthreads();
  const int H = r.H, C = r.C;
  const int fill = s_fill, total = s_total;
  const int nf = fill + n < C ? fill + n : C;          // tokens in the new window
  const int keep = nf - n;                             // old tokens that stay
  const int base = total + n - nf;                     // position of window slot 0
  const long long per = (long long)nf * H * CH;
  const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
  float m = 0.f;
  int isv = 0, h = 0, chunk = 0;
  if (gid < 2 * per) {
    isv = gid >= per;
    const long long w = isv ? gid - per : gid;
    chunk = (int)(w % CH);
    const long long th = w / CH;
    h = (int)(th % H);
    const int i = (int)(th / H);                       // window slot
    const uint16_t* src = i < keep ? (isv ? wv_in : wk_in) + ((size_t)(fill - keep + i) * H + h) * D
                                   : (isv ? v : k) + ((size_t)(i - keep) * H + h) * D;
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(src) + 2 * chunk);
    const uint4 b = __ldcs(reinterpret_cast<const uint4*>(src) + 2 * chunk + 1);
    uint4* dst = reinterpret_cast<uint4*>((isv ? wv_out : wk_out) + ((size_t)i * H + h) * D) + 2 * chunk;
    dst[0] = a;
    dst[1] = b;
    float x[16];
    unpack_bf16x16(a, b, x);
    bool ok = true;
    if (!isv) {
      const int p = base + i;
      if (p < 0 || p >= r.max_pos) {
        ok = false;
        atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
      } else {
        float4 cs[4];
        load_table16(r.table, D, p, chunk, cs);
        rope_pinned(x, cs);
      }
    }
    if (ok) {
#pragma unroll
      for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(x[e]));
    }
  }
#pragma unroll
  for (int off = CH / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if (gid < 2 * per && chunk == 0 && m > 0.f) atomicMax(r.amax + isv * H + h, __float_as_uint(m));
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int tk = atomicAdd(r.state + ST_TICKET_CALIB, 1);
    s_last = tk == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int i = threadIdx.x; i < 2 * H; i += kThreads) {
      const float a = __uint_as_float(atomicExch(r.amax + i, 0u));
      float sc = __fdiv_rn(a, 448.0f);
      if (!(sc >= 0x1p-126f)) sc = 1.0f;
      r.scales[i] = sc;
      r.scales[2 * H + i] = __fdiv_rn(1.0f, sc);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      r.state[ST_TICKET_CALIB] = 0;
      __threadfence();
    }
  }
}

// Pass 2: the whole window rotated again and quantised with the new scales
// into the FP8 ring (slot = window slot), positions base + slot; the last
// block advances the state.
template <int D>
__global__ void __launch_bounds__(kThreads) k_legacy_quantise(RingDev r, const uint16_t* __restrict__ wk,
                                                              const uint16_t* __restrict__ wv, int n) {
  constexpr int CH = D / 16;
  __shared__ int s_fill, s_total;
  if (threadIdx.x == 0) {
    s_fill = __ldcg(r.state + ST_NVALID);
    s_total = __ldcg(r.state + ST_NEXT_POS);
  }
  __syncthreads();
  const int H = r.H, C = r.C;
  const int fill = s_fill, total = s_total;
  const int nf = fill + n < C ? fill + n : C;
  const int base = total + n - nf;
  const long long per = (long long)nf * H * CH;
  const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
  if (gid < 2 * per) {
    const int isv = gid >= per;
    const long long w = isv ? gid - per : gid;
    const int chunk = (int)(w % CH);
    const long long th = w / CH;
    const int h = (int)(th % H);
    const int i = (int)(th / H);
    const uint4* src = reinterpret_cast<const uint4*>((isv ? wv : wk) + ((size_t)i * H + h) * D) + 2 * chunk;
    float x[16];
    unpack_bf16x16(__ldcs(src), __ldcs(src + 1), x);
    bool ok = true;
    if (!isv) {
      const int p = base + i;
      if (p < 0 || p >= r.max_pos) {
        ok = false;
      } else {
        float4 cs[4];
        load_table16(r.table, D, p, chunk, cs);
        rope_pinned(x, cs);
      }
      if (h == 0 && chunk == 0) r.slot_pos[i] = p;
    }
    if (ok) {
      const float inv = r.scales[(isv ? 3 : 2) * H + h];
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] = __fmul_rn(x[e], inv);
      *reinterpret_cast<uint4*>((isv ? r.v : r.k) + ((size_t)h * C + i) * D + chunk * 16) = pack_e4m3x16(x);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int tk = atomicAdd(r.state + ST_TICKET_WRITE, 1);
    if (tk == (int)gridDim.x - 1) {
      __threadfence();
      r.state[ST_NVALID] = nf;
      r.state[ST_HEAD] = nf % C;
      r.state[ST_NEXT_POS] = total + n;
      st_relaxed_gpu(r.state + ST_NEXT_POS_HINT, (int)(total + n));
      const unsigned long long tot =
          ((unsigned long long)(unsigned)r.state[ST_TOTAL_HI] << 32 | (unsigned)r.state[ST_TOTAL_LO]) +
          (unsigned long long)n;
      r.state[ST_TOTAL_LO] = (int)(unsigned)(tot & 0xFFFFFFFFull);
      r.state[ST_TOTAL_HI] = (int)(unsigned)(tot >> 32);
      r.state[ST_OLDEST_POS] = base;
      r.state[ST_CALIBRATED] = 1;
      r.state[ST_TICKET_WRITE] = 0;
      __threadfence();
    }
  }
}

// -------------------------------------------------------- codec (tests) ---
__global__ void k_encode(const float* __restrict__ in, uint8_t* __restrict__ out, int64_t n) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2;
  if (i + 1 < n) {
    const uint16_t c = f32x2_to_e4m3x2(in[i], in[i + 1]);
    out[i] = (uint8_t)(c & 0xFF);
    out[i + 1] = (uint8_t)(c >> 8);
  } else if (i < n) {
    out[i] = (uint8_t)(f32x2_to_e4m3x2(in[i], 0.f) & 0xFF);
  }
}

// ------------------------------------------------------------ projection ---
// The QKV projection y = x W^T of one frame (bf16 activations [n][dm], bf16
// weights [3 H D][dm] in a linear layer's output-by-input layout), summed in
// fp32 on the tensor cores and rounded once to bf16, with the rest of the
// "fused pre-attention" work in its epilogue: query rows stored as bf16 for
// the attention call, key rows rotated (the write's pinned RoPE), scaled and
// quantised into their ring slots, value rows scaled and quantised, the slot
// positions set and the ring state advanced by the last CTA -- byte for byte
// what kvring_write_frame does with the same bf16 keys and values.
//
// One CTA per 128 tokens x 160 output columns (five 32-column chunks, each
// inside one head of one kind): 6 x 24 = 144 CTAs for a production frame
// (757 tokens, 3 x 10 heads of 128), nearly one per SM.  A 5-stage TMA
// pipeline of 64-wide reduction slices (A 16 KB + B 20 KB), one thread
// loading, one thread issuing M128 N160 K16 bf16 MMAs, the accumulator in
// TMEM (160 of 256 allocated columns), and all four warps in the epilogue
// with one token row per thread.
constexpr int kPjThreads = 128;
constexpr int kPjBM = 128, kPjBN = kProjTileN, kPjBK = 64;
constexpr int kPjStages = 5;
constexpr uint32_t kPjTmemCols = 256;   // a power of two >= kPjBN
static_assert(kPjBN % 32 == 0 && kPjBN % 16 == 0 && kPjBN <= 256, "tile of whole 32-column chunks");
constexpr int kPjABytes = kPjBM * kPjBK * 2;
constexpr int kPjBBytes = kPjBN * kPjBK * 2;
constexpr int kPjStageBytes = kPjABytes + kPjBBytes;
constexpr int kPjMiscBytes = 256;
constexpr int kPjSmem = kPjStages * kPjStageBytes + kPjMiscBytes + 1024;   // + alignment slack
constexpr uint64_t kPjWaitNs = 1000000000ull;
static_assert(kPjSmem <= 227 * 1024, "shared memory per CTA");

enum : int { PJ_WRITE = 1, PJ_STORE_KV = 2 };

struct ProjParams {
  RingDev r;
  const int32_t* pos;   // [n] or [n][3], or null (next position + t)
  uint16_t* q_out;      // [n][H][D] bf16, or null
  uint16_t* kv_out;     // [2][n][H][D] bf16 (keys, values), or null
  int n, dm, flags;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(mbar)
      : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], bf16 x bf16 -> fp32.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kind::f16 instruction descriptor with bf16 A and B (type code 1), both
// K-major, and an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t bf16_bits_rn(float f) {
  const __nv_bfloat16 b = __float2bfloat16_rn(f);
  return (uint32_t)(*reinterpret_cast<const uint16_t*>(&b));
}

template <int D>
__global__ void __launch_bounds__(kPjThreads, 1)
    k_project(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
              const ProjParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bars = sbase + kPjStages * kPjStageBytes;   // full[S], empty[S], accumulator
  auto full = [&](int s) -> uint32_t { return bars + 8u * (uint32_t)s; };
  auto empty = [&](int s) -> uint32_t { return bars + 8u * (uint32_t)(kPjStages + s); };
  const uint32_t acc_bar = bars + 8u * (2 * kPjStages);
  int* misc = reinterpret_cast<int*>(sm + kPjStages * kPjStageBytes + 8 * (2 * kPjStages + 1));
  // misc: [0] TMEM base, [1] abort, [2] head, [3] next position, [4] slices issued, [5] slices consumed,
  // [6..8] fill level and tokens written (lo, hi), [9..15] the ring state after this frame
  volatile int* abort = misc + 1;

  const RingDev& r = prm.r;
  const int warp = threadIdx.x >> 5;
  const int m0 = blockIdx.x * kPjBM, n0 = blockIdx.y * kPjBN;
  const int KB = prm.dm / kPjBK;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
    for (int s = 0; s < kPjStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(acc_bar, 1);
    misc[1] = 0;
    misc[4] = 0;
    misc[5] = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    __syncwarp();                                  // warp-collective allocation
    tmem_alloc(smem_u32(misc), kPjTmemCols);
    tmem_relinquish();
  }
  // the next position the write will publish, as a hint for the kernels after
  if ((prm.flags & PJ_WRITE) && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 32)
    st_relaxed_gpu(r.state + ST_NEXT_POS_HINT, ld_relaxed_gpu(r.state + ST_NEXT_POS) + prm.n);
  // The activations come from the preceding kernel; the ring as well.
  griddep_wait();
  if (threadIdx.x == 0) {
    const int4 st = __ldcg(reinterpret_cast<const int4*>(r.state));   // head, n_valid, total lo, hi
    misc[2] = st.x;
    misc[3] = __ldcg(r.state + ST_NEXT_POS);
    misc[6] = st.y;
    misc[7] = st.z;
    misc[8] = st.w;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = (uint32_t)misc[0];
  // With the write: a thread that idles through the main loop gathers the
  // ring state after this frame (misc[9..15]), so the last CTA's
  // publication is stores only.
  if ((prm.flags & PJ_WRITE) && threadIdx.x == 64) {
    const unsigned long long total0 = (unsigned long long)(unsigned)misc[8] << 32 | (unsigned)misc[7];
    const WritePlan w = plan_write(r, prm.pos, misc[2], misc[6], total0, misc[3], prm.n);
    misc[9] = w.head;
    misc[10] = w.nv;
    misc[11] = w.tot_lo;
    misc[12] = w.tot_hi;
    misc[13] = w.next;
    misc[14] = w.oldest;
    misc[15] = w.prefix_end;
  }

  if (threadIdx.x == 0) {
    // ------------------------------------------------------ TMA producer
    int kb = 0;
    for (; kb < KB; ++kb) {
      const int s = kb % kPjStages;
      if (kb >= kPjStages && !mbar_wait_bounded(empty(s), (uint32_t)((kb / kPjStages) - 1) & 1u, abort, kPjWaitNs))
        break;
      const uint32_t dst = sbase + (uint32_t)s * kPjStageBytes;
      mbar_arrive_expect_tx(full(s), (uint32_t)kPjStageBytes);
      tma_load_2d(dst, &tmX, kb * kPjBK, m0, full(s));
      tma_load_2d(dst + kPjABytes, &tmW, kb * kPjBK, n0, full(s));
    }
    misc[4] = kb;
  } else if (threadIdx.x == 32) {
    // ------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16(kPjBM, kPjBN);
    int kb = 0;
    for (; kb < KB; ++kb) {
      const int s = kb % kPjStages;
      if (!mbar_wait_bounded(full(s), (uint32_t)(kb / kPjStages) & 1u, abort, kPjWaitNs)) break;
      tc_fence_after();
      const uint32_t a = sbase + (uint32_t)s * kPjStageBytes;
      const uint64_t da = smem_desc(a, 16, 1024, 2u);
      const uint64_t db = smem_desc(a + kPjABytes, 16, 1024, 2u);
#pragma unroll
      for (int kk = 0; kk < kPjBK / 16; ++kk)          // 16 bf16 = 32 bytes per step
        mma_bf16(tmem, da + 2u * kk, db + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
      mma_commit(empty(s));
    }
    misc[5] = kb;
    mma_commit(acc_bar);   // arrives once every MMA issued above has completed
  }
  __syncwarp();

  // ------------------------------------------------------------ epilogue
  // every thread waits for the accumulator; the decision to run the epilogue
  // is taken after a CTA barrier, so it is the same in every warp (the TMEM
  // loads are warp-collective)
  mbar_wait_bounded(acc_bar, 0u, abort, kPjWaitNs);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool acc_ok = !*abort;
  const int H = r.H, C = r.C;
  const int tok = m0 + (int)threadIdx.x;          // TMEM lane = accumulator row = token
  const bool write = (prm.flags & PJ_WRITE) != 0, store_kv = (prm.flags & PJ_STORE_KV) != 0;
  const int head0 = misc[2], next0 = misc[3];
  if (acc_ok) {
    // 32-column chunk k of the tile is output column n0 + 32 k: kind (0 =
    // query, 1 = key, 2 = value), head h, chunk c of the head's D columns
#pragma unroll 1
    for (int k = 0; k < kPjBN / 32; ++k) {
      const int col = n0 + 32 * k;
      if (col >= 3 * H * D) break;                  // CTA-uniform
      const int kind = col / (H * D), h = (col % (H * D)) / D, c = (col % D) / 32;
      {
        uint32_t acc[32];
        __syncwarp();
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(32 * k), acc);
        tmem_wait_ld();
        if (tok >= prm.n) continue;
        // the projection's bf16 outputs, and their fp32 values
        uint32_t w16[16];
        float x[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          w16[i] = bf16_bits_rn(__uint_as_float(acc[2 * i])) | (bf16_bits_rn(__uint_as_float(acc[2 * i + 1])) << 16);
          x[2 * i] = __uint_as_float(w16[i] << 16);
          x[2 * i + 1] = __uint_as_float(w16[i] & 0xFFFF0000u);
        }
        const uint4 o[4] = {make_uint4(w16[0], w16[1], w16[2], w16[3]), make_uint4(w16[4], w16[5], w16[6], w16[7]),
                            make_uint4(w16[8], w16[9], w16[10], w16[11]),
                            make_uint4(w16[12], w16[13], w16[14], w16[15])};
        if (kind == 0) {
          if (prm.q_out) {
            uint4* dst = reinterpret_cast<uint4*>(prm.q_out + ((size_t)tok * H + h) * D + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = o[i];
          }
          continue;
        }
        if (store_kv) {
          uint4* dst = reinterpret_cast<uint4*>(prm.kv_out + (((size_t)(kind - 1) * prm.n + tok) * H + h) * D + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = o[i];
        }
        if (!write) continue;
        // the write's arithmetic on two 16-value chunks (a head's row is in slot
        // head0 + tok, past the prefix after a wrap)
        int slot = head0 + tok;
        if (slot >= C) slot -= C - r.P;
        const float inv = r.scales[(kind == 2 ? 3 : 2) * H + h];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int chunk = 2 * c + half;
          float y[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] = x[16 * half + i];
          bool ok = true;
          if (kind == 1) {
            const int p = prm.pos ? rope_pos(r, prm.pos, tok, 8 * chunk) : next0 + tok;
            if (p < 0 || p >= r.max_pos) {
              ok = false;
              atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
            } else {
              float4 cs[4];
              load_table16(r.table, D, p, chunk, cs);
              rope_pinned(y, cs);
            }
            if (h == 0 && chunk == 0) r.slot_pos[slot] = p;
          }
          if (ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(y[i], inv);
            *reinterpret_cast<uint4*>((kind == 2 ? r.v : r.k) + ((size_t)h * C + slot) * D + chunk * 16) =
                pack_e4m3x16(y);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort) {
    // a wait gave up: let every slice already requested land before the
    // CTA's shared memory is released (bounded, on a fresh flag)
    volatile int drain_abort = 0;
    for (int kb = misc[5]; kb < misc[4]; ++kb)
      if (!mbar_wait_bounded(full(kb % kPjStages), (uint32_t)(kb / kPjStages) & 1u, &drain_abort, kPjWaitNs)) break;
    drain_abort = 0;
    mbar_wait_bounded(acc_bar, 0u, &drain_abort, kPjWaitNs);   // the issued MMAs, before TMEM is freed
    atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_TIMEOUT);
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kPjTmemCols);
  }
  // The last CTA to finish publishes the gathered state (no fence before
  // the ticket: the publication reads nothing another CTA wrote).  The CTA
  // barrier above follows thread 64's gathering.
  if (write && threadIdx.x == 0) {
    const int tk = atomicAdd(r.state + ST_TICKET_WRITE, 1);
    if (tk == (int)(gridDim.x * gridDim.y) - 1) {
      r.state[ST_HEAD] = misc[9];
      r.state[ST_NVALID] = misc[10];
      r.state[ST_TOTAL_LO] = misc[11];
      r.state[ST_TOTAL_HI] = misc[12];
      r.state[ST_NEXT_POS] = misc[13];
      st_relaxed_gpu(r.state + ST_NEXT_POS_HINT, misc[13]);
      r.state[ST_OLDEST_POS] = misc[14];
      if (r.P > 0 && misc[10] >= r.P) r.state[ST_PREFIX_END] = misc[15];
      r.state[ST_TICKET_WRITE] = 0;
    }
  }
}

unsigned grid_for(long long items) { return (unsigned)((items + kThreads - 1) / kThreads); }

}  // namespace

cudaError_t launch_calibrate(const RingDev& r, const void* k, const void* v, const int32_t* pos,
                             int n, cudaStream_t s) {
  const long long items = 2LL * n * r.H * (r.D / 16);
  const unsigned g = grid_for(items);
  if (r.D == 128)
    k_calibrate<128><<<g, kThreads, 0, s>>>(r, (const uint16_t*)k, (const uint16_t*)v, pos, n);
  else
    k_calibrate<64><<<g, kThreads, 0, s>>>(r, (const uint16_t*)k, (const uint16_t*)v, pos, n);
  return cudaGetLastError();
}

// Writes launch as programmatic dependents of the preceding kernel (they
// load their inputs early and wait before touching the ring).
cudaLaunchConfig_t pdl_config(dim3 grid, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// The staged write takes whole tokens per block, up to this many bytes of
// shared memory (frame + table rows) per block: five tokens of a 10 x 128
// frame, 152 blocks for 757 tokens, about five per SM (measured against 8
// and 3 tokens per block: 8 made the writes of back-to-back calls slower,
// 3 lost the overlap).  A ring whose single token needs more (over 55 heads
// of 128) keeps the register-staged kernel.
constexpr int kWriteTokBudget = 28 * 1024;

// Tokens per block of the staged write, or 0 when a token does not fit.
int write_tok_tokens(const RingDev& r, int n) {
  const int per_token = 4 * r.H * r.D + 4 * r.D;
  if (per_token > kWriteTokBudget) return 0;
  const int tb = kWriteTokBudget / per_token;
  return tb < n ? tb : n;
}

cudaError_t launch_write_tok(const RingDev& r, const void* k, const void* v, const int32_t* pos, int n, int tb,
                             bool late, bool nodata, bool idle, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)((n + tb - 1) / tb)), s, attr);
  cfg.dynamicSmemBytes = (size_t)2 * tb * r.H * r.D * 2 + (size_t)tb * r.D * 4;
  const uint16_t* kk = static_cast<const uint16_t*>(k);
  const uint16_t* vv = static_cast<const uint16_t*>(v);
  const int lt = late ? 1 : 0, nd = nodata ? 1 : 0, id = idle ? 1 : 0;
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_write_tok<128>, r, kk, vv, pos, n, tb, lt, nd, id);
  return cudaLaunchKernelEx(&cfg, k_write_tok<64>, r, kk, vv, pos, n, tb, lt, nd, id);
}

cudaError_t launch_write(const RingDev& r, const void* k, const void* v, const int32_t* pos, int n,
                         bool late, bool idle, cudaStream_t s) {
  const int tb = write_tok_tokens(r, n);
  if (tb > 0) return launch_write_tok(r, k, v, pos, n, tb, late, false, idle, s);
  const long long items = 2LL * n * r.H * (r.D / 16);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid_for((items + kWriteU - 1) / kWriteU)), s, attr);
  const uint16_t* kk = static_cast<const uint16_t*>(k);
  const uint16_t* vv = static_cast<const uint16_t*>(v);
  const int lt = late ? 1 : 0;
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_write<128>, r, kk, vv, pos, n, lt);
  return cudaLaunchKernelEx(&cfg, k_write<64>, r, kk, vv, pos, n, lt);
}

cudaError_t launch_write_floor(const RingDev& r, int n, bool idle, cudaStream_t s) {
  const int tb = write_tok_tokens(r, n);
  if (tb > 0) return launch_write_tok(r, nullptr, nullptr, nullptr, n, tb, false, true, idle, s);
  const long long items = 2LL * n * r.H * (r.D / 16);   // the grid of an n-token write
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid_for((items + kWriteU - 1) / kWriteU)), s, attr);
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_write_floor<128>, r);
  return cudaLaunchKernelEx(&cfg, k_write_floor<64>, r);
}

cudaError_t launch_write_many(const WriteMany& b, int count, int n, cudaStream_t s) {
  // one block per SM, each streaming its share of the units
  const RingDev& r = b.r[0];
  const WmGeom g = wm_geom(r.H, r.D);
  const long long units = 2LL * count * wm_units(g, n);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long grid = sms;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)grid), s, attr);
  cfg.blockDim = dim3(kWmThreads);
  cfg.dynamicSmemBytes = (size_t)g.stages * g.stage_bytes;
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_write_many<128>, b, count, n);
  return cudaLaunchKernelEx(&cfg, k_write_many<64>, b, count, n);
}

// One block per SM (or per unit, if fewer), each streaming its share of the
// units; launched as a programmatic dependent like the writes.
cudaError_t launch_delta_pipe(const DeltaMany& b, int count, int delta, cudaStream_t s) {
  const RingDev& r = b.r[0];
  const int ru = kDpUnitBytes / r.D;
  const long long units = (long long)count * r.H * ((r.C - r.P + ru - 1) / ru);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long grid = sms;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)grid), s, attr);
  cfg.blockDim = dim3(kDpThreads);
  cfg.dynamicSmemBytes = kDpSmemBytes;
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_delta_pipe<128>, b, count, delta);
  return cudaLaunchKernelEx(&cfg, k_delta_pipe<64>, b, count, delta);
}

cudaError_t launch_delta_many(const DeltaMany& b, int count, int delta, cudaStream_t s) {
  return launch_delta_pipe(b, count, delta, s);
}

cudaError_t launch_delta(const RingDev& r, int delta, bool idle, cudaStream_t s) {
  const unsigned runs = (unsigned)((r.C - r.P + kDeltaRows - 1) / kDeltaRows);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(runs * (unsigned)r.H), s, attr);
  const int id = idle ? 1 : 0;
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_delta_one<128>, r, delta, id);
  return cudaLaunchKernelEx(&cfg, k_delta_one<64>, r, delta, id);
}

cudaError_t cache_prepare() {
  cudaError_t e = cudaFuncSetAttribute(k_write_many<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWmStageBudget);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_write_many<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWmStageBudget);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_delta_pipe<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDpSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_delta_pipe<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDpSmemBytes);
  return e;
}

cudaError_t launch_legacy_upkeep(const RingDev& r, const void* wk_in, const void* wv_in, void* wk_out,
                                 void* wv_out, const void* k, const void* v, int n, cudaStream_t s) {
  // sized for a full window; threads past the current fill exit at once
  const long long items = 2LL * r.C * r.H * (r.D / 16);
  const unsigned g = grid_for(items);
  const auto* ki = static_cast<const uint16_t*>(wk_in);
  const auto* vi = static_cast<const uint16_t*>(wv_in);
  auto* ko = static_cast<uint16_t*>(wk_out);
  auto* vo = static_cast<uint16_t*>(wv_out);
  const auto* kn = static_cast<const uint16_t*>(k);
  const auto* vn = static_cast<const uint16_t*>(v);
  if (r.D == 128) {
    k_legacy_shift<128><<<g, kThreads, 0, s>>>(r, ki, vi, ko, vo, kn, vn, n);
    k_legacy_quantise<128><<<g, kThreads, 0, s>>>(r, ko, vo, n);
  } else {
    k_legacy_shift<64><<<g, kThreads, 0, s>>>(r, ki, vi, ko, vo, kn, vn, n);
    k_legacy_quantise<64><<<g, kThreads, 0, s>>>(r, ko, vo, n);
  }
  return cudaGetLastError();
}

cudaError_t launch_encode_e4m3(const float* in, uint8_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t pairs = (n + 1) / 2;
  const unsigned g = (unsigned)((pairs + kThreads - 1) / kThreads);
  k_encode<<<g, kThreads, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

// the projection as a programmatic dependent.
cudaError_t launch_project(const RingDev& r, const CUtensorMap* tmX, const CUtensorMap* tmW, const int32_t* pos,
                           void* q_out, void* kv_out, int n, int dm, int flags, cudaStream_t s) {
  ProjParams p;
  p.r = r;
  p.pos = pos;
  p.q_out = static_cast<uint16_t*>(q_out);
  p.kv_out = static_cast<uint16_t*>(kv_out);
  p.n = n;
  p.dm = dm;
  p.flags = flags;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + kPjBM - 1) / kPjBM, (3 * r.H * r.D + kPjBN - 1) / kPjBN);
  cfg.blockDim = dim3(kPjThreads);
  cfg.dynamicSmemBytes = kPjSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_project<128>, *tmX, *tmW, p);
  return cudaLaunchKernelEx(&cfg, k_project<64>, *tmX, *tmW, p);
}

cudaError_t project_prepare() {
  cudaError_t e = cudaFuncSetAttribute(k_project<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPjSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_project<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPjSmem);
  return e;
}

}  // namespace kvr
