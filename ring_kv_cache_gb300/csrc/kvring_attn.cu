// FP8 attention of a frame's queries over the ring cache, on the sm_103a
// tensor cores (tcgen05, TMEM accumulators, TMA-fed shared memory).
//
// What it computes ("Where the Time Went" and "Blackwell and Beyond Four
// GPUs" on the page "Runway Characters: Serving a 57B Video Diffusion
// Transformer for Real-Time Conversation": FP8 attention over the cached
// window with per-head scales):
//   out[t,h,:] = sum_j softmax_j(rope(q[t,h], qpos[t]) . Kdeq[h,j] / sqrt(d)) Vdeq[h,j]
// over the filled slots j, Kdeq = code * scale_k[h], Vdeq = code * scale_v[h].
//
// CTA = one 128-query tile x one head x one range of key/value tiles
// (split-KV).  Twelve warps:
//   warps 0-7   Softmax, two groups of four warps that take the key/value
//               tiles in turn (group g: tiles g, g + 2, ...), each with its own
//               probability buffer P_g and O accumulator O_g in TMEM.  The one
//               S buffer passes from tile to tile: a group loads S(j) into
//               registers and hands the buffer back at once, so QK(j + 1) runs
//               while it exponentiates.  One thread per query row (row r =
//               TMEM lane r) holds all 128 scores of its row: no exchange
//               between threads.  Online softmax in log2 units with a lazily
//               raised running maximum; probabilities carry 2^7 and are
//               written into P_g as f16, and the thread sums its fp32
//               probabilities into the row's normaliser.  O is rescaled in TMEM when the maximum
//               rises by more than 8 (log2 units).  Epilogue: the two
//               groups' (m, l, O) merged, O / l, split partials and their merge.
//   warp 8      Copy producer: K and V tiles [128 slots][d] by TMA into a
//               3-stage ring (the third stage once the query prologue is done).
//   warp 9      TMEM allocation and the single MMA-issuing thread:
//               S = sum_t Q_t K^T (kind::f8f6f4, A and B from shared memory,
//               K-major), then O_g += P Vh (kind::f16, P read from TMEM, B = the
//               f16 copy of the V tile, MN-major).
//   warps 10-11 Value converters: each landed E4M3 V tile is widened, exactly,
//               into one of two f16 tiles (128B-swizzled MN-major atoms of 64
//               values), which frees the E4M3 stage for the next copy.
// MMA issue: QK(j) as soon as S(j - 1) is in its group's registers and the
// K/V stage has landed; PV(j) as soon as P(j) and its f16 V tile are written.
// A group waits for PV(j - 2) (its previous tile) before it rescales O_g or
// writes P_g for tile j.
//
// Query prologue, by the softmax threads at the start of every CTA: the
// tile's query rows and their RoPE-table rows are copied into shared memory
// (cp.async, into the third K/V stage and the f16 V tiles, unused until then),
// rotated in fp32, scaled per row by 448/amax(row), split into up to 3 E4M3
// terms written straight into the swizzled images the QK MMA reads; the
// per-row logit factor stays in the thread's register, and the tile's
// maximum picks the level.  Split CTAs of a tile each do their own.
//
// Precision level per query tile (from the tile's amax and the head's key
// range 448*scale_k and value range 448*scale_v): the number of E4M3 terms of
// the queries, 1 to 4.  Extra terms are residuals at the same scale,
// accumulated into the same TMEM accumulator.  Probabilities are f16; at
// level 4 they are carried as two f16 terms (p = hi + lo, lo = f16(p - hi)),
// each multiplied into O by its own PV MMA.  Level 4 has its own TMEM and
// shared-memory plan: each softmax group owns a 128-column S/P region (the
// group's scores, then its hi and lo probabilities in the same columns), so
// QK of a group's next tile waits for PV of its previous one instead of the
// shared S buffer's hand-over; the fourth query term lives in the third K
// stage, so the K tiles cycle through two stages.
//
// Every wait is bounded (one second of wall time unless the ring's debug
// setting shortens it); a wait that gives up sets KVRING_DEVERR_TIMEOUT in the
// ring's error word, the CTA drains its in-flight copies and MMAs, frees TMEM
// and returns.
#include <mutex>
#include <type_traits>

#include "kvring_internal.cuh"

namespace kvr {
namespace {

constexpr int kStages = 3;
constexpr int kSoftmaxThreads = 256;    // 2 groups x 4 warps, one thread per query row
constexpr int kGroupThreads = 128;
constexpr int kCvtThreads = 64;         // 2 value-converter warps
constexpr int kThreads = kSoftmaxThreads + 64 + kCvtThreads;
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpCvt = 10;
constexpr uint32_t kTmemCols = 512;
// The cluster merge moves each CTA's rows in chunks of kMergeRows, each on its
// own barrier, so that merging a chunk overlaps the copies of the next.
constexpr int kMergeChunks = 4;
constexpr int kMergeRows = kTile / 2 / kMergeChunks;   // a CTA owns at most 64 rows
// Probabilities carry a factor 2^kPShift relative to the running maximum,
// which is raised only when a tile's maximum exceeds it by more than kTau:
// the largest probability is 2^(kPShift + kTau) = 2^15, inside f16 (whose
// relative precision does not depend on the magnitude).  A raise costs a
// rescale of O in TMEM by every warp holding an affected row; with a
// threshold of 8 (a factor 256) rescales are rare after the first tiles.
constexpr float kTau = 8.0f;
constexpr float kPShift = 7.0f;
// Level rule: with L = max|q| * max|k| over the tile (rotated query units
// times 448 * scale_k) and V = 448 * scale_v (the largest value), level 1
// (one E4M3 query term, relative error up to 2^-4) only when both are small,
// level 2 while L * V <= 435, level 3 beyond.  The output error of level 2
// grows about as 2.3e-5 * L * V (measured against the float64 reference for
// L from 20 to 550), so level 2 stays within 1e-2 max-abs, half the 2e-2 bar;
// level 3 errs about 25 times less.
constexpr float kLevel1MaxL = 4.0f;
constexpr float kLevel1MaxV = 0.5f;
constexpr float kLevel2MaxLV = 435.0f;
// Level 4 (four query terms, probabilities as two f16 terms) once level 3
// would leave too much: its error grows about as 9e-7 * L * V on Gaussian
// heads (so L * V <= 4800 keeps it within 4.4e-3), and single f16
// probabilities err by up to about 1e-4 * V on heavy-tailed heads (so V <= 128
// keeps that near 1e-2 at worst).  Measured with the float64 emulation of the
// kernel on 40 Student-t heads with scales up to 10: level 3 + f16 reaches
// 7e-2 max-abs, level 4 stays within 3.7e-3.
constexpr float kLevel3MaxLV = 4800.0f;
constexpr float kLevel3MaxV = 128.0f;

template <int D>
struct Layout {
  static constexpr int kQTile = kTile * D;      // one Q term tile (bytes)
  static constexpr int kKVTile = kTile * D;     // one E4M3 K or V tile
  static constexpr int kVhTile = 2 * kTile * D; // one f16 V tile
  static constexpr int kVhAtom = kTile * 128;   // 64 f16 columns x 128 rows
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 3 * kQTile;
  static constexpr int kV = kK + kStages * kKVTile;
  static constexpr int kVh = kV + kStages * kKVTile;
  static constexpr int kEpi = kVh + 2 * kVhTile;        // float m[2][128], l[2][128], lse[128]
  static constexpr int kBars = kEpi + 5 * kTile * 4;
  // barrier slots (8 bytes each)
  static constexpr int kBarKFull = 0;                   // K tile of a stage landed
  static constexpr int kBarKEmpty = kStages;            // ... read by its QK
  static constexpr int kBarSFull = 2 * kStages;
  static constexpr int kBarPFull = 2 * kStages + 2;
  static constexpr int kBarPvDone = 2 * kStages + 4;
  static constexpr int kBarVhFull = 2 * kStages + 6;
  static constexpr int kBarMmaDone = 2 * kStages + 8;
  static constexpr int kBarSFree = 2 * kStages + 9;
  static constexpr int kBarPvIssuerDone = 2 * kStages + 10;  // every PV of the PV issuer has finished
  static constexpr int kBarVFull = 2 * kStages + 11;    // V tile of a stage landed
  static constexpr int kBarVEmpty = 3 * kStages + 11;   // ... widened to f16 by the converters
  static constexpr int kBarNever = 4 * kStages + 11;    // never arrived on: the debug stall waits here
  static constexpr int kBarRows = 4 * kStages + 12;     // the query prologue's RoPE rows have landed
  static constexpr int kBarMerge = 4 * kStages + 13;    // [kMergeChunks] a chunk of the peers' partial rows landed
  static constexpr int kNumBars = 4 * kStages + 13 + kMergeChunks;
  static constexpr int kMisc = kBars + 8 * kNumBars;
  static constexpr int kLseAll = kMisc + 64;             // float [8 splits][128]: the cluster's log2-sum-exps
  static constexpr int kBytes = kLseAll + 8 * kTile * 4;
  static constexpr uint32_t kSwz = D == 128 ? 2u : 4u;  // UMMA swizzle code of the E4M3 tiles
  static_assert(kVh % 1024 == 0, "128B-swizzled atoms need 1024-byte alignment");
  // TMEM columns (levels 1-3)
  static constexpr uint32_t kColS = 0;        // the S buffer (128 columns, one tile's scores)
  static constexpr uint32_t kColP = 128;      // f16 probabilities of group g at 128 + 64 g
  static constexpr uint32_t kColO = 256;      // O accumulator of group g at 256 + 128 g (D columns)
  // Level 4: group g's S/P region at 128 g (scores, then hi probabilities in
  // its first 64 columns and lo in the next 64); O as above.
  static constexpr uint32_t kColSP4 = 128;
  // Shared-memory byte offset of query term t (0..3): terms 0-2 in the Q
  // images, term 3 (level 4 only) in the third K stage.
  static constexpr int q_term(int t) { return t < 3 ? kQ + t * kQTile : kK + 2 * kKVTile; }
};

struct Misc {
  uint32_t tmem_base;
  int level;
  int abort;
  int last;
  int hint;      // the ring's next-position hint, read once before the wait
  int pos_bad;   // a speculative query position fell outside the table
  int nvalid_pre;   // the ring's fill level, read once before the wait
};

struct AttnParams {
  RingDev r;
  const uint16_t* q;
  const int32_t* qpos;
  void* out;
  int n_q;
  int out_bf16;
  int nsplit;
  int tiles_per_split;
  int forced_level;
  int cluster_merge;   // the splits of a query tile form one cluster (2..8 CTAs)
  int debug_stall;     // 1: the QK issuer first waits on a barrier nothing arrives on
  int q_late;          // 1: the preceding kernel may write the queries: read them after the wait
  int debug_guess;     // 1: guess the default positions wrong on purpose (test support)
  unsigned long long wait_ns;   // limit of every bounded wait
};

// 3-D RoPE: the (t, y, x) positions of a query tile's rows into qpos_s
// [128][3], a CTA barrier, then each row's table words into `dst` with
// cp.async, every 16-byte table chunk (2 pairs, one section: sections are
// whole chunks of 8 pairs) from the row of its section's coordinate.  Only
// the 3-D instantiation of the kernel contains it.
template <int D>
__device__ __forceinline__ void stage_rows_3d(const RingDev& r, const int32_t* qpos, int n_q, int qt, int rows_in,
                                           int* qpos_s, uint32_t dst) {
  constexpr int TPR = D / 4;
  if (threadIdx.x < 3 * kTile) {
    int p = 0;
    if (qt * kTile + (int)threadIdx.x / 3 < n_q) {
      p = __ldg(qpos + 3 * qt * kTile + threadIdx.x);
      if (p < 0 || p >= r.max_pos) {
        atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
        p = 0;
      }
    }
    qpos_s[threadIdx.x] = p;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < rows_in * TPR; k += blockDim.x) {
    const int rr = k / TPR, c = k % TPR;
    const int p = qpos_s[3 * rr + rope_axis(r, 2 * c)];
    cp_async16(dst + (uint32_t)(rr * TPR + c) * 16u, r.table + (size_t)p * D + 4 * c);
  }
}

// Named barriers: 0 = __syncthreads, 1 = the 256 softmax threads.
__device__ __forceinline__ void sync_softmax() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int D, bool R3>
__global__ void __launch_bounds__(kThreads, 1)
    k_attention(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const AttnParams prm) {
  using L = Layout<D>;
  constexpr int QD = D / 4;             // O columns per softmax thread
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base by pointer arithmetic on the shared array itself,
  // so the compiler keeps shared-memory (not generic) loads and stores
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  Misc* misc = reinterpret_cast<Misc*>(sm + L::kMisc);
  float* epi = reinterpret_cast<float*>(sm + L::kEpi);
  volatile int* abort = &misc->abort;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBars + 8u * (uint32_t)i; };

  const RingDev& r = prm.r;
  const uint64_t wait_ns = prm.wait_ns;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
  const int H = r.H;
  // Query rows of this tile that exist, and where they are staged in shared
  // memory until the query prologue has made E4M3 terms of them: the third
  // K and V stages (rows 0-63, 64-127), which hold no copy before then.
  const int rows_in = prm.n_q - qt * kTile < kTile ? prm.n_q - qt * kTile : kTile;
  auto q_stage = [&](int rr) -> uint32_t {
    return sbase + (rr < 64 ? L::kK : L::kV) + 2 * L::kKVTile + (uint32_t)(rr & 63) * (2 * D);
  };
  // The query rows: before the wait for the preceding kernel unless the
  // host found that a kernel possibly still in flight writes them.
  auto copy_queries = [&]() {
    for (int k = threadIdx.x; k < rows_in * (D / 8); k += kThreads) {
      const int rr = k / (D / 8), c = k % (D / 8);
      cp_async16(q_stage(rr) + 16u * c, prm.q + ((size_t)(qt * kTile + rr) * H + h) * D + 8 * c);
    }
    cp_async_commit();
  };
  // The ring's next-position hint, read first of all (its latency overlaps
  // the set-up below; see the query prologue).
  const int hint0 = (threadIdx.x == 0 && !prm.qpos) ? ld_relaxed_gpu(r.state + ST_NEXT_POS_HINT) : 0;
  // The fill level as well, for the producer: once it equals the capacity
  // it never changes again, so the first key/value copies can then be
  // issued as soon as the wait returns, without the state read after it.
  const int nvalid_pre = threadIdx.x == 32 ? ld_relaxed_gpu(r.state + ST_NVALID) : 0;
  if (!prm.q_late) copy_queries();
  // Set-up that touches nothing a preceding kernel writes runs before the
  // wait: barriers, TMEM, and (below) the query prologue.
  if (threadIdx.x == kWarpTma * 32) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    // K and V stages are loaded and freed separately: a K stage as soon as
    // its QK has read it, a V stage once the converters have widened it
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(L::kBarKFull + s), 1);
      mbar_init(bar(L::kBarKEmpty + s), 1);
      mbar_init(bar(L::kBarVFull + s), 1);
      mbar_init(bar(L::kBarVEmpty + s), kCvtThreads);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kBarSFull + b), 1);     // S of a group-b tile is in TMEM
      mbar_init(bar(L::kBarPFull + b), kGroupThreads);
      mbar_init(bar(L::kBarPvDone + b), 1);
      mbar_init(bar(L::kBarVhFull + b), kCvtThreads);
    }
    mbar_init(bar(L::kBarMmaDone), 1);
    mbar_init(bar(L::kBarSFree), kGroupThreads / 32);  // a tile's S is in its group's registers
    for (int c = 0; c < kMergeChunks; ++c) mbar_init(bar(L::kBarMerge + c), 1);
    mbar_init(bar(L::kBarPvIssuerDone), 1);
    mbar_init(bar(L::kBarNever), 1);
    mbar_init(bar(L::kBarRows), 1);
    misc->abort = 0;
    misc->last = 0;
    mbar_fence_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&misc->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  // The head's scales, read once here (the level choice, the softmax, the
  // epilogue and the split merge need them; a load there would sit on their
  // critical path).  Only a calibration or the legacy upkeep writes them,
  // and neither lets the kernel after it start early, so they may be read
  // before the wait.
  const float scale_k = r.scales[h], scale_v = r.scales[H + h];
  // ------------------------------------------------ query prologue
  // All twelve warps, before the roles split up (nothing can proceed without
  // the query terms anyway).  first_pos: the position of query 0 when the
  // positions are the default ones.
  int rows_phase = 0;   // completed phases of kBarRows (one per bulk row copy)
  auto query_prologue = [&](int first_pos, bool speculative) {
      // (1) one position per query row; (2) the RoPE-table rows of those
      // positions copied into the f16 V tiles' space with 16-byte cp.async
      // (the query rows are already on their way, see above); (3) one pass
      // over 8-value chunks: chunk task k = i * 384 + tid is query row
      // k / CPR, chunk k % CPR, so a warp holds every chunk of its rows and a
      // row's amax is a shuffle reduction; the chunk's first two E4M3 terms
      // go straight into the swizzled images the QK MMA reads; (4) the warps'
      // maxima give the tile's precision level, and levels 3 and 4 add their
      // terms from the residuals kept in registers.
      constexpr int CPR = D / 8;                           // 16-byte q chunks per row
      constexpr int TPR = D / 4;                           // 16-byte table chunks per row
      constexpr int PQ = (kTile * CPR + kThreads - 1) / kThreads;   // chunk tasks per thread
      int* qpos_s = reinterpret_cast<int*>(epi + 2 * kTile);   // [128] (1-D) or [128][3] (3-D)
      // Default positions that all lie in the table: the tile's rows are
      // consecutive table rows, one bulk copy (completing on kBarRows).
      const int p0 = first_pos + qt * kTile;
      const bool bulk_rows = !R3 && !prm.qpos && p0 >= 0 && p0 + rows_in <= r.max_pos;
      if (bulk_rows) {
        if (threadIdx.x == 0) {
          fence_proxy_async_smem();   // (a second pass rewrites rows the first one read)
          mbar_arrive_expect_tx(bar(L::kBarRows), (uint32_t)(rows_in * D * 4));
          bulk_load(sbase + L::kVh, r.table + (size_t)p0 * D, (uint32_t)(rows_in * D * 4), bar(L::kBarRows));
        }
      } else if (!R3 && threadIdx.x < kTile) {
        const int tq = qt * kTile + threadIdx.x;
        int p = 0;
        if (tq < prm.n_q) {
          p = prm.qpos ? __ldg(prm.qpos + tq) : first_pos + tq;
          if (p < 0 || p >= r.max_pos) {
            // (a guessed position is reported only once it proves right)
            if (speculative)
              misc->pos_bad = 1;
            else
              atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
            p = 0;
          }
        }
        qpos_s[threadIdx.x] = p;
      }
      if constexpr (R3) stage_rows_3d<D>(r, prm.qpos, prm.n_q, qt, rows_in, qpos_s, sbase + L::kVh);
      if (!bulk_rows) {
        __syncthreads();
        if constexpr (!R3) {
          for (int k = threadIdx.x; k < rows_in * TPR; k += kThreads) {
            const int rr = k / TPR, c = k % TPR;
            cp_async16(sbase + L::kVh + (uint32_t)(rr * TPR + c) * 16u, r.table + (size_t)qpos_s[rr] * D + 4 * c);
          }
        }
        cp_async_commit();
      }
      cp_async_wait_all();
      if (bulk_rows) {
        volatile int no_abort = 0;
        if (!mbar_wait_bounded(bar(L::kBarRows), (uint32_t)(rows_phase & 1), &no_abort, wait_ns))
          misc->abort = 1;
        ++rows_phase;
      }
      __syncthreads();
      auto rotate = [&](int rrow, int chunk, float (&u)[8]) -> float {
        float cmax = 0.f;
        if (rrow < rows_in) {
          const uint4 w = *reinterpret_cast<const uint4*>(sm + (q_stage(rrow) - sbase) + 16 * chunk);
          const float4* tb = reinterpret_cast<const float4*>(sm + L::kVh + (size_t)rrow * (4 * D)) + 2 * chunk;
          const float4 cs0 = tb[0], cs1 = tb[1];
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
          const float cc[4] = {cs0.x, cs0.z, cs1.x, cs1.z};
          const float ss[4] = {cs0.y, cs0.w, cs1.y, cs1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = __uint_as_float(ww[e] << 16), x1 = __uint_as_float(ww[e] & 0xFFFF0000u);
            u[2 * e] = x0 * cc[e] - x1 * ss[e];
            u[2 * e + 1] = x0 * ss[e] + x1 * cc[e];
            cmax = fmaxf(cmax, fmaxf(fabsf(u[2 * e]), fabsf(u[2 * e + 1])));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) u[e] = 0.f;          // rows past n_q: zero queries
        }
        return cmax;
      };
      // One pass rotates every chunk, takes its row's maximum (the CPR
      // consecutive lanes that hold the row), scales by it and writes the
      // first two E4M3 terms at once, keeping the exact fp32 residual in
      // registers (u[i]); after the CTA barrier that gives the tile's
      // maximum and level, the tiles whose level needs them get terms 3 and 4
      // from the residuals (term 4 goes to the third K stage, whose staged
      // query rows every thread has read by then).  Chunk tasks of one
      // iteration cover whole warps (rows x CPR is a multiple of 32), so
      // every shuffle has all lanes.
      float u[PQ][8];
      float wmax = 0.f;
      auto put_term = [&](int term, uint32_t off, float (&v)[8], bool residual) {
        uint16_t c4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) c4[e] = f32x2_to_e4m3x2(v[2 * e], v[2 * e + 1]);
        *reinterpret_cast<uint2*>(sm + L::q_term(term) + off) =
            make_uint2((uint32_t)c4[0] | ((uint32_t)c4[1] << 16), (uint32_t)c4[2] | ((uint32_t)c4[3] << 16));
        if (residual) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 dq = e4m3x2_to_f32x2(c4[e]);
            v[2 * e] -= dq.x;
            v[2 * e + 1] -= dq.y;
          }
        }
      };
#pragma unroll
      for (int i = 0; i < PQ; ++i) {
        const int k = i * kThreads + threadIdx.x;
        const int rrow = k / CPR, chunk = k % CPR;
        float cmax = 0.f;
        if (k < kTile * CPR) {
          cmax = rotate(rrow, chunk, u[i]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) u[i][e] = 0.f;
        }
#pragma unroll
        for (int off = CPR / 2; off > 0; off >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, off));
        wmax = fmaxf(wmax, cmax);
        if (k < kTile * CPR) {
          if (chunk == 0) epi[rrow] = cmax;
          // E4M3 terms of q / sigma_q (sigma_q = amax/448 of the row), exact
          // fp32 residuals; 8 bytes per chunk per term at the chunk's
          // swizzled place in the query images
          float sq = cmax / 448.0f;
          if (!(sq >= 0x1p-126f)) sq = 1.0f;
          // only invq * sq matters (the logit factor uses sq): a fast
          // reciprocal (a couple of ulp) leaves it 1 within 2^-21
          const float invq = __fdividef(1.0f, sq);
#pragma unroll
          for (int e = 0; e < 8; ++e) u[i][e] *= invq;
          const uint32_t off = swz_offset(rrow, chunk >> 1, D) + (chunk & 1) * 8;
          put_term(0, off, u[i], true);
          put_term(1, off, u[i], true);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xFFFFFFFFu, wmax, off));
      if (lane == 0) epi[kTile + warp] = wmax;
      __syncthreads();
      float qm = epi[kTile];
#pragma unroll
      for (int i = 1; i < kThreads / 32; ++i) qm = fmaxf(qm, epi[kTile + i]);
      int level = prm.forced_level;
      if (level == 0) {
        const float lg = qm * 448.0f * scale_k;
        const float vmax = 448.0f * scale_v;
        level = (vmax > kLevel3MaxV || lg * vmax > kLevel3MaxLV) ? 4
                : (lg <= kLevel1MaxL && vmax <= kLevel1MaxV)     ? 1
                : (lg * vmax <= kLevel2MaxLV)                   ? 2
                                                                : 3;
      }
      if (level >= 3) {
#pragma unroll
        for (int i = 0; i < PQ; ++i) {
          const int k = i * kThreads + threadIdx.x;
          if (k >= kTile * CPR) break;
          const int rrow = k / CPR, chunk = k % CPR;
          const uint32_t off = swz_offset(rrow, chunk >> 1, D) + (chunk & 1) * 8;
          put_term(2, off, u[i], level >= 4);
          if (level >= 4) put_term(3, off, u[i], false);
        }
      }
      if (threadIdx.x == 0) misc->level = level;
      fence_proxy_async_smem();   // generic writes -> tensor-core reads
      __syncthreads();
  };

  // The query prologue runs before the wait for the preceding kernel when
  // its inputs allow: the queries (and explicit positions) unless the host
  // found that a kernel still in flight writes them, and the default
  // positions from the ring's next-position hint, which a write sets as it
  // starts.  After the wait the guess is checked against the ring's next
  // position and the prologue repeated if it was wrong.
  const bool early = !prm.q_late;
  if (threadIdx.x == 0) {
    misc->hint = prm.qpos ? 0 : hint0 + (prm.debug_guess ? r.max_pos : 0);
    misc->pos_bad = 0;
  }
  if (threadIdx.x == 32) misc->nvalid_pre = nvalid_pre;
  __syncthreads();
  const int hint = misc->hint;
  if (early) query_prologue(hint - prm.n_q, prm.qpos == nullptr);
  const int tile0 = split * prm.tiles_per_split;
  auto first_copies = [&](int nv) {
    // The producer starts the first two key/value copies at once; the third
    // stage's space holds query rows until the query prologue is done.
    int nt = (nv + kTile - 1) / kTile - tile0;
    nt = nt < 0 ? 0 : (nt > prm.tiles_per_split ? prm.tiles_per_split : nt);
    const int first = nt < kStages - 1 ? nt : kStages - 1;
    for (int j = 0; j < first; ++j) {
      const int slot0 = (tile0 + j) * kTile;
      mbar_arrive_expect_tx(bar(L::kBarKFull + j), (uint32_t)(kTile * D));
      tma_load_3d(sbase + L::kK + j * L::kKVTile, &tmK, 0, slot0, h, bar(L::kBarKFull + j));
      mbar_arrive_expect_tx(bar(L::kBarVFull + j), (uint32_t)(kTile * D));
      tma_load_3d(sbase + L::kV + j * L::kKVTile, &tmV, 0, slot0, h, bar(L::kBarVFull + j));
    }
  };
  // This kernel is a programmatic dependent of the preceding kernel (a write,
  // or an earlier attention): the ring (state, cache) is read only after it.
  griddep_wait();
  if (threadIdx.x == kWarpTma * 32) first_copies(misc->nvalid_pre == r.C ? r.C : __ldcg(r.state + ST_NVALID));
  const int nvalid = __ldcg(r.state + ST_NVALID);
  const int next_pos = __ldcg(r.state + ST_NEXT_POS);
  const int ntile_total = (nvalid + kTile - 1) / kTile;
  int ntiles = ntile_total - tile0;
  ntiles = ntiles < 0 ? 0 : (ntiles > prm.tiles_per_split ? prm.tiles_per_split : ntiles);

  // ---------------------------------------------------------------- setup
  const size_t unit = (size_t)qt * H + h;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // A following write (or query preparation) launched as a programmatic
  // dependent may start on the idle SMs now: it loads its inputs and waits
  // for this grid before it touches the ring.
  griddep_launch_dependents();
  const uint32_t tmem = misc->tmem_base;
  if (!(early && (prm.qpos != nullptr || next_pos == hint))) {
    // (the staged query rows may have been overwritten by a fourth term)
    copy_queries();
    query_prologue(next_pos - prm.n_q, false);
  } else if (threadIdx.x == 0 && misc->pos_bad) {
    atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_POSITION);
  }
  if (threadIdx.x == 0 && split == 0) r.levels[unit] = misc->level;


  if (warp == kWarpTma) {
    // ------------------------------------------ TMA producer + PV issuer
    // One thread loads the key/value tiles and issues PV(j) = P_b(j) Vh_b(j)
    // into O_b (b = j & 1) as soon as P(j) and its f16 V tile are written;
    // the MMA warp issues only QK, so the two kinds of MMA are issued from
    // two warps and neither waits behind the other's issue (a single thread
    // needs longer to issue an M = 128, N = 128 MMA than the tensor core
    // needs to run it).
    // Level 4 cycles the K tiles through two stages (the third holds the
    // fourth query term) and issues two PV MMAs per tile (hi, then lo
    // probabilities, from the group's S/P region); the loop is instantiated
    // for levels 1-3 and for level 4 so that both keep constant stage math.
    auto producer = [&](auto level4) {
      constexpr bool l4 = decltype(level4)::value;
      constexpr int nks = l4 ? 2 : kStages;   // K stages in use
      auto kst = [](int j) { return j % nks; };
      auto kph = [](int j) { return (j / nks) & 1; };
      constexpr uint32_t idesc_pv = idesc_f16(128, D, true);
      // f16 V: 128B-swizzled MN-major atoms of 64 columns x 8 rows (1024 B
      // apart along the slots); the second 64 columns one atom column further
      const uint64_t dv = smem_desc(sbase + L::kVh, (uint32_t)L::kVhAtom, 1024, 2u);
      const uint32_t v_lo = (uint32_t)dv, v_hi = (uint32_t)(dv >> 32);
      constexpr uint32_t kVhStep = L::kVhTile >> 4;
      auto issue_pv = [&](int j) {
        const int b = j & 1;
        tc_fence_after();
        const uint32_t vl = v_lo + (uint32_t)b * kVhStep;
        if constexpr (!l4) {
          const uint32_t pa = tmem + L::kColP + 64u * b;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_f16_ts_w(tmem + L::kColO + b * 128, pa + kk * 8, vl + kk * (16 * 128 / 16), v_hi, idesc_pv,
                         (j > 1 || kk > 0) ? 1u : 0u);
        } else {
          // level 4: the block of slots 16 kk + [0, 16) has its f16 values at
          // columns 16 kk + [0, 8) of the group's region and the second terms
          // at 16 kk + [8, 16)
          const uint32_t pa = tmem + L::kColSP4 * b;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            mma_f16_ts_w(tmem + L::kColO + b * 128, pa + kk * 16, vl + kk * (16 * 128 / 16), v_hi, idesc_pv,
                         (j > 1 || kk > 0) ? 1u : 0u);
            mma_f16_ts_w(tmem + L::kColO + b * 128, pa + kk * 16 + 8, vl + kk * (16 * 128 / 16), v_hi, idesc_pv, 1u);
          }
        }
        mma_commit(bar(L::kBarPvDone + b));
      };
      const int first = ntiles < kStages - 1 ? ntiles : kStages - 1;
      int k_issued = first, v_issued = first, np = 0;
      uint32_t idle = 0;
      uint64_t t_idle = 0;
      while (np < ntiles) {
        bool prog = false;
        if (mbar_test_wait(bar(L::kBarPFull + (np & 1)), (np >> 1) & 1) &&
            mbar_test_wait(bar(L::kBarVhFull + (np & 1)), (np >> 1) & 1)) {
          issue_pv(np++);
          prog = true;
        }
        if (k_issued < ntiles && mbar_test_wait(bar(L::kBarKEmpty + kst(k_issued)), kph(k_issued) ^ 1)) {
          const int s = kst(k_issued);
          mbar_arrive_expect_tx(bar(L::kBarKFull + s), (uint32_t)(kTile * D));
          tma_load_3d(sbase + L::kK + s * L::kKVTile, &tmK, 0, (tile0 + k_issued) * kTile, h, bar(L::kBarKFull + s));
          ++k_issued;
          prog = true;
        }
        if (v_issued < ntiles &&
            mbar_test_wait(bar(L::kBarVEmpty + v_issued % kStages), ((v_issued / kStages) & 1) ^ 1)) {
          const int s = v_issued % kStages;
          mbar_arrive_expect_tx(bar(L::kBarVFull + s), (uint32_t)(kTile * D));
          tma_load_3d(sbase + L::kV + s * L::kKVTile, &tmV, 0, (tile0 + v_issued) * kTile, h, bar(L::kBarVFull + s));
          ++v_issued;
          prog = true;
        }
        if (prog) {
          idle = 0;
          continue;
        }
        if (idle++ == 0) {
          t_idle = globaltimer_ns();
        } else if ((idle & 15u) == 0) {
          if (*abort) break;
          if (globaltimer_ns() - t_idle > wait_ns) {
            *abort = 1;
            break;
          }
        }
      }
      // Drain: every issued copy must land before the CTA may exit.
      volatile int no_abort = 0;
      for (int j = k_issued - nks < 0 ? 0 : k_issued - nks; j < k_issued; ++j)
        mbar_wait_bounded(bar(L::kBarKFull + kst(j)), kph(j), &no_abort, wait_ns);
      for (int j = v_issued - kStages < 0 ? 0 : v_issued - kStages; j < v_issued; ++j)
        mbar_wait_bounded(bar(L::kBarVFull + j % kStages), (j / kStages) & 1, &no_abort, wait_ns);
      // and every PV this thread issued has finished before TMEM is freed
      mma_commit(bar(L::kBarPvIssuerDone));
      mbar_wait_bounded(bar(L::kBarPvIssuerDone), 0, &no_abort, wait_ns);
    };
    if (lane == 0) {   // the prologue ended with a CTA barrier: the level is known
      if (misc->level == 4) producer(std::true_type{});
      else producer(std::false_type{});
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- QK issuer
    auto qk_issuer = [&](auto level4) {
      constexpr bool l4 = decltype(level4)::value;
      constexpr uint32_t idesc_qk = idesc_e4m3(128, 128, false);
      // Descriptors are built once; per MMA only the low word (start address
      // in 16-byte units) moves: +2 per 32-byte k-step of a K-major tile.
      const uint64_t dq = smem_desc(sbase + L::kQ, 16, 8 * D, L::kSwz);
      const uint64_t dk = smem_desc(sbase + L::kK, 16, 8 * D, L::kSwz);
      const uint32_t q_lo = (uint32_t)dq, k_lo = (uint32_t)dk, kq_hi = (uint32_t)(dq >> 32);
      constexpr uint32_t kKVStep = L::kKVTile >> 4;
      const int n_qterms = misc->level;   // the prologue ended with a CTA barrier
      // The debug stall: a wait that nothing ends, so that the bounded wait
      // gives up and the whole CTA takes its abort path.
      const bool go = !prm.debug_stall || mbar_wait_bounded(bar(L::kBarNever), 0, abort, wait_ns);
      // Levels 1-3: S(j) into the one S buffer once its group has S(j - 1) in
      // registers and the K stage has landed.  Level 4: S(j) into group
      // (j & 1)'s S/P region once PV(j - 2) has read that group's previous
      // probabilities from it.  The K stage is freed by the commit.
      for (int j = 0; go && j < ntiles; ++j) {
        const int s = l4 ? (j & 1) : j % kStages;
        if constexpr (l4) {
          if (j > 1 && !mbar_wait_bounded(bar(L::kBarPvDone + (j & 1)), ((j - 2) >> 1) & 1, abort, wait_ns)) break;
        } else {
          if (j > 0 && !mbar_wait_bounded(bar(L::kBarSFree), (j - 1) & 1, abort, wait_ns)) break;
        }
        if (!mbar_wait_bounded(bar(L::kBarKFull + s), l4 ? (j >> 1) & 1 : (j / kStages) & 1, abort, wait_ns))
          break;
        tc_fence_after();
        const uint32_t kl = k_lo + s * kKVStep;
        const uint32_t dst = l4 ? tmem + L::kColSP4 * (j & 1) : tmem + L::kColS;
#pragma unroll
        for (int t = 0; t < (l4 ? 4 : 3); ++t) {
          if (l4 || t < n_qterms) {
            const uint32_t qt_lo = q_lo + (uint32_t)((L::q_term(t) - L::kQ) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk)
              mma_e4m3_w(dst, qt_lo + 2 * kk, kq_hi, kl + 2 * kk, kq_hi, idesc_qk, (t | kk) != 0);
          }
        }
        mma_commit(bar(L::kBarSFull + (j & 1)));
        mma_commit(bar(L::kBarKEmpty + s));   // the K stage is read
      }
    };
    if (lane == 0 && ntiles > 0) {
      if (misc->level == 4) qk_issuer(std::true_type{});
      else qk_issuer(std::false_type{});
    }
    if (lane == 0) {  // every MMA this thread issued has finished before TMEM is freed
      mma_commit(bar(L::kBarMmaDone));
      volatile int no_abort = 0;
      mbar_wait_bounded(bar(L::kBarMmaDone), 0, &no_abort, wait_ns);
    }
    __syncwarp();
  } else if (warp >= kWarpCvt) {
    // ------------------------------------------------- value converters
    // E4M3 V tile [128 slots][d] (TMA image, 128B or 64B swizzle) -> f16 tile
    // of d/64 atoms [128 slots][64 values] (128B swizzle).  Task i: slot
    // i / CPR, 16-value chunk i % CPR; each converter thread takes every
    // 64th task, a batch of loads first.
    constexpr int CPR = D / 16;
    constexpr int PER = kTile * CPR / kCvtThreads;   // 16 (d = 128) or 8
    constexpr int BATCH = PER < 8 ? PER : 8;
    const int ct = threadIdx.x - kWarpCvt * 32;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kStages, b = j & 1;
      bool ok = mbar_wait_bounded(bar(L::kBarVFull + s), (j / kStages) & 1, abort, wait_ns);
      if (ok && j >= 2) ok = mbar_wait_bounded(bar(L::kBarPvDone + b), ((j >> 1) & 1) ^ 1, abort, wait_ns);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      const uint8_t* src = sm + L::kV + s * L::kKVTile;
      uint8_t* dst = sm + L::kVh + b * L::kVhTile;
#pragma unroll
      for (int n0 = 0; n0 < PER; n0 += BATCH) {
        uint4 w[BATCH];
#pragma unroll
        for (int n = 0; n < BATCH; ++n) {
          const int i = ct + (n0 + n) * kCvtThreads;
          w[n] = *reinterpret_cast<const uint4*>(src + swz_offset(i / CPR, i % CPR, D));
        }
#pragma unroll
        for (int n = 0; n < BATCH; ++n) {
          const int i = ct + (n0 + n) * kCvtThreads;
          const int row = i / CPR, c = i % CPR;
          const uint32_t wi[4] = {w[n].x, w[n].y, w[n].z, w[n].w};
          uint32_t hv[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hv[2 * e] = e4m3x2_to_f16x2((uint16_t)(wi[e] & 0xFFFFu));
            hv[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(wi[e] >> 16));
          }
          uint8_t* atom = dst + (c >> 2) * L::kVhAtom;
          *reinterpret_cast<uint4*>(atom + swz_offset(row, 2 * (c & 3), 128)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<uint4*>(atom + swz_offset(row, 2 * (c & 3) + 1, 128)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
      }
      fence_proxy_async_smem();  // generic writes -> tensor-core reads
      mbar_arrive(bar(L::kBarVhFull + b));
      mbar_arrive(bar(L::kBarVEmpty + s));
    }
  } else {
    // ----------------------------------------------------------- softmax
    // thread = (group g, row): S columns [0, 128), P_g columns [0, 64),
    // O_g columns [0, d).
    const int g = warp >> 2;
    const int row = threadIdx.x & (kTile - 1);
    const int quarter = warp & 3;
    // the logit factor of this thread's query row (row amax from the prologue)
    float f_row;
    {
      float sq = epi[row] / 448.0f;
      if (!(sq >= 0x1p-126f)) sq = 1.0f;
      f_row = fmaxf(sq * scale_k * (1.4426950408889634f / sqrtf((float)D)), 1e-30f);
    }
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tO = trow + L::kColO + g * 128;
    float m_run = -INFINITY;
    float ell = 0.f;
    bool ok = true;
    // The tile loop, instantiated for levels 1-3 and for level 4.  Levels
    // 1-3 load a tile's 128 scores into registers at once and hand the S
    // buffer back.  Level 4 keeps its scores in the group's own S/P region
    // and streams them in 32-column chunks, twice (row maximum, then
    // probabilities): its probabilities go in place over the scores they
    // come from, each 16-slot block's 16 columns taking the block's f16
    // values (8 columns) and then the f16 roundings of what those left (8
    // columns), so no chunk overwrites a score not yet read.
    auto tile_loop = [&](auto level4) {
    constexpr bool l4 = decltype(level4)::value;
    const uint32_t tS = l4 ? trow + L::kColSP4 * g : trow + L::kColS;
    const uint32_t tP = l4 ? trow + L::kColSP4 * g : trow + L::kColP + 64 * g;
    for (int j = g; j < ntiles; j += 2) {
      const int n = j >> 1;
      ok = __all_sync(0xFFFFFFFFu, ok && mbar_wait_bounded(bar(L::kBarSFull + g), n & 1, abort, wait_ns));
      if (!ok) break;
      tc_fence_after();
      // slots past the fill level are masked (only the ring's last tile)
      const int valid = nvalid - (tile0 + j) * kTile;
      uint32_t sr[l4 ? 1 : 128];
      float smax;
      if constexpr (!l4) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
        tmem_wait_ld();
        // the scores are in registers: the S buffer may take the next tile
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kBarSFree));
        if (valid < kTile) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= valid) sr[c] = __float_as_uint(-INFINITY);
        }
        // row maximum: eight running three-way maxima, then a small tree
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmaxf(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1]));
#pragma unroll
        for (int i = 1; i < 8; ++i)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mx[k] = fmax3(mx[k], __uint_as_float(sr[16 * i + 2 * k]), __uint_as_float(sr[16 * i + 2 * k + 1]));
        smax = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
      } else {
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r32[32];
          tmem_ld32(tS + 32 * c, r32);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x = 32 * c + i < valid ? __uint_as_float(r32[i]) : -INFINITY;
            mx[i & 3] = fmaxf(mx[i & 3], x);
          }
        }
        smax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      }
      const float tmax = smax * f_row;          // f_row > 0
      const bool need = tmax > m_run + kTau;
      const float m_new = need ? tmax : m_run;
      // O_g and P_g are touched only once PV(j - 2), this group's previous
      // tile, has completed
      if (j > 1) {
        ok = __all_sync(0xFFFFFFFFu,
                        mbar_wait_bounded(bar(L::kBarPvDone + g), ((j - 2) >> 1) & 1, abort, wait_ns));
        if (!ok) break;
        tc_fence_after();
      }
      if (j > 1 && __any_sync(0xFFFFFFFFu, need)) {
        // O_g holds this group's earlier tiles: rescale it in chunks of 16
        // columns (the row's scores stay in registers meanwhile)
        const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t rr[16];
          tmem_ld_n<16>(tO + 16 * c, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 y = __fmul2_rn(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])),
                                        make_float2(alpha, alpha));
            rr[i] = __float_as_uint(y.x);
            rr[i + 1] = __float_as_uint(y.y);
          }
          tmem_st16(tO + 16 * c, rr);
        }
        ell *= alpha;
      }
      m_run = m_new;
      // probabilities 2^(x - m + 7) as f16 pairs, the lower slot in the low
      // half; the normaliser takes the fp32 values (pairs of scores through
      // the packed two-lane fp32 FMA and add)
      const float moff = kPShift - m_run;
      const float2 fr2 = make_float2(f_row, f_row), mo2 = make_float2(moff, moff);
      float2 lsum = make_float2(0.f, 0.f);
      if constexpr (l4) {
        // slots 16 b + [0, 16) -> columns 16 b + [0, 8) (f16 values) and
        // 16 b + [8, 16) (f16 roundings of what the values left; the fp32
        // difference is exact, both lying within 2^-11 of each other)
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r32[32];
          tmem_ld32(tS + 32 * c, r32);
          tmem_wait_ld();
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            float2 e[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int k = 16 * hb + 2 * i;
              const float2 x = __ffma2_rn(make_float2(__uint_as_float(r32[k]), __uint_as_float(r32[k + 1])), fr2, mo2);
              e[i] = make_float2(32 * c + k < valid ? ex2_approx(x.x) : 0.f,
                                 32 * c + k + 1 < valid ? ex2_approx(x.y) : 0.f);
            }
            uint32_t hv[8], lv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              hv[i] = f32x2_to_f16x2(e[i].x, e[i].y);
              const float2 hf = f16x2_to_f32x2(hv[i]);
              lv[i] = f32x2_to_f16x2(e[i].x - hf.x, e[i].y - hf.y);
            }
            tmem_st_n<8>(tP + 32 * c + 16 * hb, hv);
            tmem_st_n<8>(tP + 32 * c + 16 * hb + 8, lv);
#pragma unroll
            for (int w = 4; w > 0; w >>= 1)
#pragma unroll
              for (int i = 0; i < w; ++i) e[i] = __fadd2_rn(e[i], e[i + w]);
            lsum = __fadd2_rn(lsum, e[0]);
          }
        }
      } else {
        // slots 32 c + [0, 32) -> columns 16 c + [0, 16) of P_g
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float2 e[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(sr[32 * c + 2 * i]), __uint_as_float(sr[32 * c + 2 * i + 1])), fr2, mo2);
            e[i] = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          }
          uint32_t hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) hv[i] = f32x2_to_f16x2(e[i].x, e[i].y);
          tmem_st16(tP + 16 * c, hv);
#pragma unroll
          for (int w = 8; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) e[i] = __fadd2_rn(e[i], e[i + w]);
          lsum = __fadd2_rn(lsum, e[0]);
        }
      }
      ell += lsum.x + lsum.y;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::kBarPFull + g));
    }
    };
    if (misc->level == 4) tile_loop(std::true_type{});
    else tile_loop(std::false_type{});

    // ---------------------------------------------------------- epilogue
    // merge the two groups: m = max(m_0, m_1), w_g = 2^(m_g - m),
    // l = sum w_g l_g, O = sum w_g O_g.  After this barrier both groups are
    // done with their loops, so each PV-done barrier is at most one phase
    // short of the group's last PV.
    float* em = epi;                 // [2][128]
    float* el = epi + 2 * kTile;     // [2][128]
    float* lse_row = epi + 4 * kTile;
    em[g * kTile + row] = m_run;
    el[g * kTile + row] = ell;
    ok = __all_sync(0xFFFFFFFFu, ok);
    sync_softmax();
    const float m0 = em[row], m1 = em[kTile + row];
    const float m = fmaxf(m0, m1);
    const float w0 = m0 > -INFINITY ? ex2_approx(m0 - m) : 0.f;
    const float w1 = m1 > -INFINITY ? ex2_approx(m1 - m) : 0.f;
    const float l = w0 * el[row] + w1 * el[kTile + row];
    // the last tile of each group
    const int jl0 = ntiles > 0 ? ((ntiles - 1) & ~1) : -1;
    const int jl1 = ntiles > 1 ? (((ntiles - 2) & ~1) + 1) : -1;
    if (ok && jl0 >= 0)
      ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar(L::kBarPvDone + 0), (jl0 >> 1) & 1, abort, wait_ns));
    if (ok && jl1 >= 0)
      ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar(L::kBarPvDone + 1), (jl1 >> 1) & 1, abort, wait_ns));
    // Normalised rows go to shared memory (the key/value stages are free:
    // every copy landed, was converted and read by its MMAs), fp32
    // [128][d + 4]: group g's thread of the row writes columns [g d/2, (g+1) d/2)
    // from both accumulators.  Then the whole tile is stored, or merged
    // across splits, with coalesced 16-byte accesses.
    const float inv_l = l > 0.f ? 1.0f / l : 0.f;
    const bool single = prm.nsplit == 1;
    constexpr int SP = D + 4;                 // padded row stride (floats)
    constexpr int F4 = kTile * D / 4;         // float4 per tile
    constexpr int PER = F4 / kSoftmaxThreads; // float4 per thread
    float* stage = reinterpret_cast<float*>(sm + L::kK);
    {
      const float f = single ? inv_l * scale_v : inv_l;
      const float a0 = w0 * f, a1 = w1 * f;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const uint32_t col = g * (D / 2) + 32 * c;
        uint32_t r0[32], r1[32];
        if (ok && jl0 >= 0) tmem_ld32(trow + L::kColO + col, r0);
        if (ok && jl1 >= 0) tmem_ld32(trow + L::kColO + 128 + col, r1);
        tmem_wait_ld();
        float4* srow = reinterpret_cast<float4*>(stage + row * SP + col);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float x0 = (ok && jl0 >= 0) ? __uint_as_float(r0[4 * i + k]) * a0 : 0.f;
            const float x1 = (ok && jl1 >= 0) ? __uint_as_float(r1[4 * i + k]) * a1 : 0.f;
            v[k] = x0 + x1;
          }
          srow[i] = make_float4(v[0], v[1], v[2], v[3]);
        }
      }
      if (g == 0) lse_row[row] = (ok && l > 0.f) ? log2f(l) + m - kPShift : -INFINITY;
    }
    sync_softmax();
    const int rows_live = prm.n_q - qt * kTile < kTile ? prm.n_q - qt * kTile : kTile;
    auto store_out = [&](int f4, float4 v) {
      const int rrow = f4 / (D / 4), c4 = f4 % (D / 4);
      if (rrow >= rows_live) return;
      const size_t e = ((size_t)(qt * kTile + rrow) * H + h) * D + 4 * c4;
      if (prm.out_bf16) {
        const __nv_bfloat162 a0 = __floats2bfloat162_rn(v.x, v.y), a1 = __floats2bfloat162_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(prm.out) + e) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a0), *reinterpret_cast<const uint32_t*>(&a1));
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(prm.out) + e) = v;
      }
    };
    auto staged = [&](int f4) -> float4 {
      return *reinterpret_cast<const float4*>(stage + (f4 / (D / 4)) * SP + 4 * (f4 % (D / 4)));
    };
    if (single) {
#pragma unroll
      for (int i = 0; i < PER; ++i) store_out(threadIdx.x + i * kSoftmaxThreads, staged(threadIdx.x + i * kSoftmaxThreads));
    } else if (prm.cluster_merge) {
      // the staged partial stays here; the row's log2-sum-exp goes to every
      // CTA of the cluster now (a region nothing else uses), so the merge
      // after the cluster barrier reads the weights locally
      if (threadIdx.x < kTile) {
        const float v = lse_row[threadIdx.x];
        const uint32_t a = sbase + L::kLseAll + 4u * (uint32_t)(split * kTile + threadIdx.x);
        for (int s2 = 0; s2 < prm.nsplit; ++s2) st_dsmem_f32(dsmem_addr(a, (uint32_t)s2), v);
      }
      fence_proxy_async_smem();   // the staged rows are read by bulk copies
    } else {
      // partial (normalised) tile and its per-row log2-sum-exp
      const size_t pbase = ((size_t)split * r.qtiles_max + qt) * H + h;
      float4* dst = reinterpret_cast<float4*>(r.part_o + pbase * kTile * D);
#pragma unroll
      for (int i = 0; i < PER; ++i) __stcg(dst + threadIdx.x + i * kSoftmaxThreads, staged(threadIdx.x + i * kSoftmaxThreads));
      if (threadIdx.x < kTile) __stcg(r.part_lse + pbase * kTile + threadIdx.x, lse_row[threadIdx.x]);
      __threadfence();
      sync_softmax();
      if (threadIdx.x == 0) {
        const int tk = atomicAdd(r.tickets + qt * H + h, 1);
        misc->last = tk == prm.nsplit - 1;
      }
      sync_softmax();
      if (misc->last) {
        // last split of this tile: merge all splits
        __threadfence();
        float* wts = reinterpret_cast<float*>(sm + L::kQ);   // [nsplit][128]
        if (threadIdx.x < kTile) {
          const int rr = threadIdx.x;
          float mx = -INFINITY;
          for (int s2 = 0; s2 < prm.nsplit; ++s2)
            mx = fmaxf(mx, __ldcg(r.part_lse + (((size_t)s2 * r.qtiles_max + qt) * H + h) * kTile + rr));
          float sum = 0.f;
          for (int s2 = 0; s2 < prm.nsplit; ++s2) {
            const float lse = __ldcg(r.part_lse + (((size_t)s2 * r.qtiles_max + qt) * H + h) * kTile + rr);
            const float w = (mx > -INFINITY && lse > -INFINITY) ? ex2_approx(lse - mx) : 0.f;
            wts[s2 * kTile + rr] = w;
            sum += w;
          }
          const float g = sum > 0.f ? scale_v / sum : 0.f;
          for (int s2 = 0; s2 < prm.nsplit; ++s2) wts[s2 * kTile + rr] *= g;
        }
        sync_softmax();
        float4 acc[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s2 = 0; s2 < prm.nsplit; ++s2) {
          // a batch of this split's loads in flight before any use
          const float4* src = reinterpret_cast<const float4*>(
              r.part_o + (((size_t)s2 * r.qtiles_max + qt) * H + h) * kTile * D);
          constexpr int MB = PER < 8 ? PER : 8;
#pragma unroll
          for (int i0 = 0; i0 < PER; i0 += MB) {
            float4 v[MB];
#pragma unroll
            for (int i = 0; i < MB; ++i) v[i] = __ldcg(src + threadIdx.x + (i0 + i) * kSoftmaxThreads);
#pragma unroll
            for (int i = 0; i < MB; ++i) {
              const float w = wts[s2 * kTile + (threadIdx.x + (i0 + i) * kSoftmaxThreads) / (D / 4)];
              acc[i0 + i].x = fmaf(w, v[i].x, acc[i0 + i].x);
              acc[i0 + i].y = fmaf(w, v[i].y, acc[i0 + i].y);
              acc[i0 + i].z = fmaf(w, v[i].z, acc[i0 + i].z);
              acc[i0 + i].w = fmaf(w, v[i].w, acc[i0 + i].w);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < PER; ++i) store_out(threadIdx.x + i * kSoftmaxThreads, acc[i]);
        if (threadIdx.x == 0) r.tickets[qt * H + h] = 0;
      }
    }
  }

  // ------------------------------------------------------ cluster merge
  // The nsplit CTAs of this query tile form one cluster (rank = split); CTA
  // `split` owns output rows [split 128 / nsplit, (split + 1) 128 / nsplit).
  // After the cluster barrier every CTA's normalised partial is staged in
  // its shared memory, every CTA holds all log2-sum-exps (pushed to it
  // before the barrier), and no CTA needs its f16 V tiles any more: each CTA
  // bulk-copies the rows every peer owns into that peer's f16 V space (one
  // slot per sender), completing on the peer's merge barrier, then merges
  // its own rows from its own shared memory and stores them.  Rows travel in
  // chunks of kMergeRows, each completing on its own barrier, and a chunk is
  // merged and stored as soon as it has landed.  A CTA leaves once its
  // outgoing copies have read its rows and its incoming ones have landed, so
  // no second cluster barrier is needed.
  if (prm.cluster_merge) {
    __syncwarp();
    cluster_sync_all();
    constexpr int SP = D + 4;                      // staged row stride (floats)
    constexpr uint32_t SPB = SP * 4;               // ... in bytes
    const int ns = prm.nsplit;
    const int maxr = (kTile + ns - 1) / ns;        // rows of one slot
    const int r0 = split * kTile / ns, r1 = (split + 1) * kTile / ns, nr = r1 - r0;
    auto chunk_rows = [&](int c, int rows) {
      const int left = rows - c * kMergeRows;
      return left < 0 ? 0 : (left < kMergeRows ? left : kMergeRows);
    };
    if (threadIdx.x == kWarpTma * 32) {
      for (int c = 0; c < kMergeChunks; ++c)
        if (chunk_rows(c, nr) > 0)
          mbar_arrive_expect_tx(bar(L::kBarMerge + c), (uint32_t)((ns - 1) * chunk_rows(c, nr)) * SPB);
      // chunk-major, so that every peer's first chunk is on its way first
      for (int c = 0; c < kMergeChunks; ++c)
        for (int p = 0; p < ns; ++p) {
          if (p == split) continue;
          const int p0 = p * kTile / ns, p1 = (p + 1) * kTile / ns;
          const int rows = chunk_rows(c, p1 - p0);
          if (rows == 0) continue;
          const int slot = split < p ? split : split - 1;
          bulk_copy_to_cluster(
              dsmem_addr(sbase + L::kVh + (uint32_t)(slot * maxr + c * kMergeRows) * SPB, (uint32_t)p),
              sbase + L::kK + (uint32_t)(p0 + c * kMergeRows) * SPB, (uint32_t)rows * SPB,
              dsmem_addr(bar(L::kBarMerge + c), (uint32_t)p));
        }
      bulk_commit();
    }
    if (warp < kSoftmaxThreads / 32) {
      constexpr int MT = (kTile / 2) * (D / 4) / kSoftmaxThreads;  // float4 tasks per thread (nsplit >= 2)
      const float* lse_all = reinterpret_cast<const float*>(sm + L::kLseAll);   // [nsplit][128]
      float* wts = reinterpret_cast<float*>(sm + L::kQ);   // [nsplit][128]
      const int ntask = nr * (D / 4);
      if ((int)threadIdx.x < nr) {
        const int row = r0 + threadIdx.x;
        float lv[8];
        float mx = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2)
          if (s2 < ns) {
            lv[s2] = lse_all[s2 * kTile + row];
            mx = fmaxf(mx, lv[s2]);
          }
        float sum = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2)
          if (s2 < ns) {
            lv[s2] = (mx > -INFINITY && lv[s2] > -INFINITY) ? ex2_approx(lv[s2] - mx) : 0.f;
            sum += lv[s2];
          }
        const float gsc = sum > 0.f ? scale_v / sum : 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2)
          if (s2 < ns) wts[s2 * kTile + threadIdx.x] = lv[s2] * gsc;
      }
      sync_softmax();   // the weights
      // The peers' copies were issued unconditionally after the cluster
      // barrier, so they land even on an aborted call: wait for every chunk
      // whatever the abort flag says (a CTA must not exit while copies into
      // its shared memory are in flight); a chunk that never lands is a
      // timeout.
      const int rows_live = prm.n_q - qt * kTile < kTile ? prm.n_q - qt * kTile : kTile;
      // split s2's rows of this range: own staging, or the sender's slot
      auto rows_of = [&](int s2) -> const uint8_t* {
        return s2 == split ? sm + L::kK + (size_t)r0 * SPB
                           : sm + L::kVh + (size_t)((s2 < split ? s2 : s2 - 1) * maxr) * SPB;
      };
      constexpr int IPC = MT / kMergeChunks;   // float4 tasks of a thread in one chunk
      static_assert(MT % kMergeChunks == 0 && IPC * kSoftmaxThreads == kMergeRows * (D / 4),
                    "a chunk is a whole number of task rounds");
      bool landed = true;
#pragma unroll 1
      for (int c = 0; c < kMergeChunks && c * kMergeRows < nr; ++c) {
        volatile int no_abort = 0;
        landed = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar(L::kBarMerge + c), 0, &no_abort, wait_ns)) && landed;
        if (!landed) continue;
        float4 acc[IPC];
#pragma unroll
        for (int i = 0; i < IPC; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        // two splits at a time, all their loads issued before any use
        for (int s0 = 0; s0 < ns; s0 += 2) {
          float4 v[2][IPC];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint8_t* src = rows_of(s0 + q < ns ? s0 + q : s0);
#pragma unroll
            for (int i = 0; i < IPC; ++i) {
              const int idx = threadIdx.x + (c * IPC + i) * kSoftmaxThreads;
              const int lr = idx / (D / 4), c4 = idx % (D / 4);
              v[q][i] = idx < ntask ? *reinterpret_cast<const float4*>(src + (size_t)lr * SPB + 16 * c4)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            if (s0 + q >= ns) break;
#pragma unroll
            for (int i = 0; i < IPC; ++i) {
              const int idx = threadIdx.x + (c * IPC + i) * kSoftmaxThreads;
              const float w = idx < ntask ? wts[(s0 + q) * kTile + idx / (D / 4)] : 0.f;
              acc[i].x = fmaf(w, v[q][i].x, acc[i].x);
              acc[i].y = fmaf(w, v[q][i].y, acc[i].y);
              acc[i].z = fmaf(w, v[q][i].z, acc[i].z);
              acc[i].w = fmaf(w, v[q][i].w, acc[i].w);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < IPC; ++i) {
          const int idx = threadIdx.x + (c * IPC + i) * kSoftmaxThreads;
          const int row = r0 + idx / (D / 4), c4 = idx % (D / 4);
          if (idx >= ntask || row >= rows_live) continue;
          const size_t e = ((size_t)(qt * kTile + row) * H + h) * D + 4 * c4;
          if (prm.out_bf16) {
            const __nv_bfloat162 a0 = __floats2bfloat162_rn(acc[i].x, acc[i].y), a1 = __floats2bfloat162_rn(acc[i].z, acc[i].w);
            *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(prm.out) + e) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&a0), *reinterpret_cast<const uint32_t*>(&a1));
          } else {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(prm.out) + e) = acc[i];
          }
        }
      }
      if (!landed) misc->abort = 1;
    }
    // the outgoing copies have read this CTA's rows before it may leave
    if (threadIdx.x == kWarpTma * 32) bulk_wait_read();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && misc->abort)
    atomicOr(reinterpret_cast<unsigned*>(r.state + ST_ERROR), KVRING_DEVERR_TIMEOUT);
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t attention_prepare(int D) {
  const int smem = (int)attention_smem_bytes(D);
  cudaError_t e;
  if (D == 128) {
    e = cudaFuncSetAttribute(k_attention<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_attention<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  } else {
    e = cudaFuncSetAttribute(k_attention<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_attention<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  }
  return e;
}

size_t attention_smem_bytes(int D) {
  return (D == 128 ? Layout<128>::kBytes : Layout<64>::kBytes) + 1024;
}

cudaError_t launch_attention(const RingDev& r, const CUtensorMap* tmK, const CUtensorMap* tmV,
                             const AttnLaunch& a, cudaStream_t s) {
  AttnParams p;
  p.r = r;
  p.q = static_cast<const uint16_t*>(a.q);
  p.qpos = a.qpos;
  p.out = a.out;
  p.n_q = a.n_q;
  p.out_bf16 = a.out_bf16;
  p.nsplit = a.nsplit;
  p.tiles_per_split = a.tiles_per_split;
  p.forced_level = a.forced_level;
  p.cluster_merge = (a.nsplit >= 2 && a.nsplit <= 8) ? 1 : 0;
  p.debug_stall = a.debug_stall;
  p.q_late = a.q_late;
  p.debug_guess = a.debug_guess;
  p.wait_ns = a.wait_ns;
  const unsigned qtiles = (unsigned)((a.n_q + kTile - 1) / kTile);
  // A programmatic dependent of the preceding kernel: it may start while
  // that kernel still runs, copies its query rows (unless that kernel may
  // write them), and waits (griddepcontrol.wait) before it reads the ring.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(qtiles, (unsigned)r.H, (unsigned)a.nsplit);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = attention_smem_bytes(r.D);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.cluster_merge) {  // the splits of one query tile as one cluster
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = (unsigned)a.nsplit;
    cfg.numAttrs = 2;
  }
  // 3-D RoPE has its own instantiation (query positions from three rows)
  if (r.D == 128)
    return r.pt ? cudaLaunchKernelEx(&cfg, k_attention<128, true>, *tmK, *tmV, p)
                : cudaLaunchKernelEx(&cfg, k_attention<128, false>, *tmK, *tmV, p);
  return r.pt ? cudaLaunchKernelEx(&cfg, k_attention<64, true>, *tmK, *tmV, p)
              : cudaLaunchKernelEx(&cfg, k_attention<64, false>, *tmK, *tmV, p);
}

// ---------------------------------------------------------------------------
// Scratch for callers that cannot allocate device memory.
//
// kvring_attention_noalloc keeps its scratch (the precision level of every
// query tile and head; its splits merge in a cluster, so it needs no
// partials) in this file-scope array instead of the ring's buffer.  It is static device memory: every GPU that loads the
// library holds it until the process exits.  In host code the array's name
// is only a host-side stand-in, so its device address is looked up once per
// device (cudaGetSymbolAddress, with that device current) and then passed
// to the kernels like any other pointer.
namespace {
constexpr size_t kStaticScratchBytes = size_t(128) << 10;   // 32,768 units
__device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];
std::mutex g_scratch_mu;
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
}  // namespace

size_t static_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace kvr
