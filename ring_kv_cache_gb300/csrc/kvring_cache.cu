// Memory-bound kernels of the rolling FP8 cache: per-session scale
// calibration, the per-frame write (RoPE + E4M3 quantisation into the ring)
// and the in-place delta rotation at a position reset.  See the page
// "Runway Characters: Serving a 57B Video Diffusion Transformer for
// Real-Time Conversation", section "Do It Once, at Write Time".
//
// Work decomposition (all three kernels): one thread owns 16 consecutive
// elements of one (token or slot, head) row, i.e. one 16-byte chunk of FP8
// output; consecutive threads walk a row, then the next head, then the next
// token, so bf16 input reads are fully contiguous and every cache row is
// written as whole 16-byte vectors.  Completion work (ring state, scales,
// position map) is done by the last block to finish, found with an atomic
// ticket; no block ever waits on another.
//
// Arithmetic is pinned so that cache bytes are reproducible: products and
// sums are rounded one at a time (__fmul_rn / __fadd_rn / __fsub_rn, no
// fused multiply-add), the cos/sin table is fp32 built on the host, and the
// E4M3 conversion is the hardware round-to-nearest-even saturating cvt.
#include "kvring_internal.cuh"

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
      const int p = pos ? __ldg(pos + t) : s_next + t;
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
                                           int n, int blk, int nblk) {
  constexpr int CH = D / 16;
  __shared__ int s_head, s_next;
  // A following kernel launched as a programmatic dependent (an attention's
  // query preparation, or the next write) may start now: each waits for
  // this grid before it touches the ring.
  griddep_launch_dependents();
  const int H = r.H, C = r.C;
  const long long per = (long long)n * H * CH;
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
  // This kernel is launched as a programmatic dependent of the preceding
  // kernel: the inputs above were complete before that kernel started; the
  // ring (state, cache, positions) is read and written only after it is done.
  griddep_wait();
  if (threadIdx.x == 0) {
    s_head = __ldcg(r.state + ST_HEAD);
    s_next = __ldcg(r.state + ST_NEXT_POS);
  }
  __syncthreads();
  // all table rows before any arithmetic or store, so their latencies overlap
  float4 cs[U][4];
  int pp[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const long long gid = ((long long)blk * U + u) * kThreads + threadIdx.x;
    pp[u] = -1;
    if (gid < per) {  // keys only
      const int chunk = (int)(gid % CH);
      const int t = (int)(gid / CH / H);
      const int p = pos ? __ldg(pos + t) : s_next + t;
      pp[u] = p;
      if (p >= 0 && p < r.max_pos) load_table16(r.table, D, p, chunk, cs[u]);
    }
  }
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
    int slot = s_head + t;
    if (slot >= C) slot -= C;  // head < C and t < n <= C
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
  if (threadIdx.x == 0) {
    __threadfence();
    const int tk = atomicAdd(r.state + ST_TICKET_WRITE, 1);
    if (tk == nblk - 1) {
      __threadfence();
      int head = s_head + n;
      if (head >= C) head -= C;
      const int nv = r.state[ST_NVALID] + n;
      r.state[ST_HEAD] = head;
      r.state[ST_NVALID] = nv < C ? nv : C;
      const unsigned long long tot =
          ((unsigned long long)(unsigned)r.state[ST_TOTAL_HI] << 32 | (unsigned)r.state[ST_TOTAL_LO]) +
          (unsigned long long)n;
      r.state[ST_TOTAL_LO] = (int)(unsigned)(tot & 0xFFFFFFFFull);
      r.state[ST_TOTAL_HI] = (int)(unsigned)(tot >> 32);
      r.state[ST_NEXT_POS] = s_next + n;
      // oldest filled slot: the next one to be overwritten once full, else slot 0
      r.state[ST_OLDEST_POS] = __ldcg(r.slot_pos + (nv >= C ? head : 0));
      r.state[ST_TICKET_WRITE] = 0;
      __threadfence();
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) k_write(RingDev r, const uint16_t* __restrict__ k,
                                                    const uint16_t* __restrict__ v,
                                                    const int32_t* __restrict__ pos, int n) {
  write_body<D, kWriteU>(r, k, v, pos, n, blockIdx.x, gridDim.x);
}

// Many rings of one shape in one launch: ring blockIdx.y, the same blocks
// per ring as a single-ring write.
// Batched: two chunks per thread and four blocks per SM (a few registers
// spill); over 60 rings this measured 108.8 us against 152.8 us at three
// blocks per SM and 205 us at four chunks per thread.
constexpr int kWriteManyU = 2;
template <int D>
__global__ void __launch_bounds__(kThreads, 4) k_write_many(const __grid_constant__ WriteMany b, int n) {
  const int i = blockIdx.y;
  write_body<D, kWriteManyU>(b.r[i], b.k[i], b.v[i], b.pos[i], n, blockIdx.x, gridDim.x);
}

// ---------------------------------------------------------------- delta ---
// A few blocks per SM, each thread looping over 16-byte chunks of filled key
// rows (kDeltaU independent chunks in flight per iteration), so the number of
// completion tickets stays small.
constexpr int kDeltaU = 4;

// One ring's share of a delta rotation: block `blk` of `nblk`, U chunks in
// flight per thread and iteration.
template <int D, int U>
__device__ __forceinline__ void delta_body(const RingDev& r, int delta_arg, int blk, int nblk) {
  constexpr int CH = D / 16;
  __shared__ int s_delta, s_nv, s_last;
  __shared__ float4 s_cs[D / 4];  // table row of delta: D/2 (cos, sin) pairs
  if (threadIdx.x == 0) {
    const int nv = __ldcg(r.state + ST_NVALID);
    int d = delta_arg;
    if (d == KVRING_DELTA_TO_OLDEST) d = nv > 0 ? __ldcg(r.state + ST_OLDEST_POS) : 0;
    if (d < 0 || d >= r.max_pos) {
      if (blk == 0) atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_DELTA);
      d = -1;  // skip the rotation entirely
    }
    s_delta = d;
    s_nv = nv;
  }
  __syncthreads();
  const int delta = s_delta;
  const int nv = s_nv;
  // positions of the filled slots, spread over all blocks (nobody reads them here)
  if (delta > 0)
    for (int sl = blk * kThreads + threadIdx.x; sl < nv; sl += nblk * kThreads) r.slot_pos[sl] -= delta;
  if (delta > 0) {
    const float4* row = reinterpret_cast<const float4*>(r.table + (size_t)delta * D);
    for (int i = threadIdx.x; i < D / 4; i += kThreads) s_cs[i] = __ldg(row + i);
  }
  __syncthreads();
  if (delta > 0) {
    // items: (head, filled slot, chunk), slot-major within a head
    const long long per_head = (long long)nv * CH;
    const long long items = per_head * r.H;
    const long long stride = (long long)nblk * kThreads;
    for (long long base = (long long)blk * kThreads + threadIdx.x; base < items; base += stride * U) {
      uint4 in[U];
      uint4* ptr[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long it = base + u * stride;
        ptr[u] = nullptr;
        if (it < items) {
          const long long h = it / per_head, rem = it % per_head;
          ptr[u] = reinterpret_cast<uint4*>(r.k + ((size_t)h * r.C + rem / CH) * D + (rem % CH) * 16);
          in[u] = *ptr[u];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!ptr[u]) continue;
        const int chunk = (int)((base + u * stride) % per_head % CH);
        const uint32_t w[4] = {in[u].x, in[u].y, in[u].z, in[u].w};
        float y[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 a = e4m3x2_to_f32x2((uint16_t)(w[i] & 0xFFFF));
          const float2 b = e4m3x2_to_f32x2((uint16_t)(w[i] >> 16));
          // pairs (a.x, a.y) and (b.x, b.y); pair index chunk*8 + 2i (+1)
          const float4 cs = s_cs[chunk * 4 + i];  // (c, s) of both pairs
          y[4 * i + 0] = __fadd_rn(__fmul_rn(a.x, cs.x), __fmul_rn(a.y, cs.y));
          y[4 * i + 1] = __fsub_rn(__fmul_rn(a.y, cs.x), __fmul_rn(a.x, cs.y));
          y[4 * i + 2] = __fadd_rn(__fmul_rn(b.x, cs.z), __fmul_rn(b.y, cs.w));
          y[4 * i + 3] = __fsub_rn(__fmul_rn(b.y, cs.z), __fmul_rn(b.x, cs.w));
        }
        *ptr[u] = pack_e4m3x16(y);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int tk = atomicAdd(r.state + ST_TICKET_DELTA, 1);
    s_last = tk == nblk - 1;
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    if (delta >= 0) {
      r.state[ST_NEXT_POS] -= delta;
      r.state[ST_OLDEST_POS] -= delta;
      r.state[ST_LAST_DELTA] = delta;
    }
    r.state[ST_TICKET_DELTA] = 0;
    __threadfence();
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) k_delta(RingDev r, int delta_arg) {
  delta_body<D, kDeltaU>(r, delta_arg, blockIdx.x, gridDim.x);
}

// Batched: four chunks in flight per thread, about eight blocks per SM over
// the batch (measured best of 4/6/8/16 chunks and 4/8/12/16/32 blocks).
constexpr int kDeltaManyU = 4;
constexpr int kDeltaManyBlocksPerSm = 8;
template <int D>
__global__ void __launch_bounds__(kThreads) k_delta_many(const __grid_constant__ DeltaMany b, int delta_arg) {
  delta_body<D, kDeltaManyU>(b.r[blockIdx.y], delta_arg, blockIdx.x, gridDim.x);
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

cudaError_t launch_write(const RingDev& r, const void* k, const void* v, const int32_t* pos, int n,
                         cudaStream_t s) {
  const long long items = 2LL * n * r.H * (r.D / 16);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid_for((items + kWriteU - 1) / kWriteU)), s, attr);
  const uint16_t* kk = static_cast<const uint16_t*>(k);
  const uint16_t* vv = static_cast<const uint16_t*>(v);
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_write<128>, r, kk, vv, pos, n);
  return cudaLaunchKernelEx(&cfg, k_write<64>, r, kk, vv, pos, n);
}

cudaError_t launch_write_many(const WriteMany& b, int count, int n, cudaStream_t s) {
  const RingDev& r = b.r[0];
  const long long items = 2LL * n * r.H * (r.D / 16);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid_for((items + kWriteManyU - 1) / kWriteManyU), (unsigned)count), s, attr);
  if (r.D == 128) return cudaLaunchKernelEx(&cfg, k_write_many<128>, b, n);
  return cudaLaunchKernelEx(&cfg, k_write_many<64>, b, n);
}

cudaError_t launch_delta_many(const DeltaMany& b, int count, int delta, cudaStream_t s) {
  // per ring the single-ring grid capped so that the batch gives about
  // kDeltaManyBlocksPerSm blocks per SM, at least 8 per ring
  const RingDev& r = b.r[0];
  const long long items = (long long)r.H * r.C * (r.D / 16);
  unsigned g = grid_for((items + kDeltaManyU - 1) / kDeltaManyU);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  unsigned per = (unsigned)((kDeltaManyBlocksPerSm * sms + count - 1) / count);
  if (per < 8) per = 8;
  if (g > per) g = per;
  if (g < 1) g = 1;
  const dim3 grid(g, (unsigned)count);
  if (r.D == 128)
    k_delta_many<128><<<grid, kThreads, 0, s>>>(b, delta);
  else
    k_delta_many<64><<<grid, kThreads, 0, s>>>(b, delta);
  return cudaGetLastError();
}

cudaError_t launch_delta(const RingDev& r, int delta, cudaStream_t s) {
  // the fill level is device state: size for a full ring, at most ~2 blocks per SM
  const long long items = (long long)r.H * r.C * (r.D / 16);
  unsigned g = grid_for((items + kDeltaU - 1) / kDeltaU);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (g > (unsigned)(2 * sms)) g = (unsigned)(2 * sms);
  if (g < 1) g = 1;
  if (r.D == 128)
    k_delta<128><<<g, kThreads, 0, s>>>(r, delta);
  else
    k_delta<64><<<g, kThreads, 0, s>>>(r, delta);
  return cudaGetLastError();
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

}  // namespace kvr
