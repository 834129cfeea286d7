// Internal definitions shared by the kvring translation units: the device
// layout of one ring, the int32 state words, and thin inline-PTX wrappers
// for the sm_103a features the kernels use (E4M3 conversion, mbarrier,
// TMA tensor copies, tcgen05 MMA / TMEM).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvring.h"

namespace kvr {

// State words beyond the public ones (KVRING_STATE_*): completion tickets.
enum : int {
  ST_HEAD = KVRING_STATE_HEAD,
  ST_NVALID = KVRING_STATE_NVALID,
  ST_TOTAL_LO = KVRING_STATE_TOTAL_LO,
  ST_TOTAL_HI = KVRING_STATE_TOTAL_HI,
  ST_NEXT_POS = KVRING_STATE_NEXT_POS,
  ST_CALIBRATED = KVRING_STATE_CALIBRATED,
  ST_ERROR = KVRING_STATE_ERROR,
  ST_LAST_DELTA = KVRING_STATE_LAST_DELTA,
  ST_TICKET_WRITE = 8,
  ST_TICKET_CALIB = 9,
  ST_TICKET_DELTA = 10,
  ST_OLDEST_POS = 11,   // position of the oldest rolling slot (the default reset delta)
  ST_PREFIX_END = 12,   // with a pinned prefix: position of its last slot + 1
  // The next position as it will be once the write in flight is done: set
  // at the start of every write (from a relaxed read of ST_NEXT_POS plus the
  // frame's length) and with every change of ST_NEXT_POS.  Only a guess:
  // the attention prepares its queries for the positions it implies while
  // the preceding kernel still runs, and checks them against ST_NEXT_POS
  // once that kernel is done.
  ST_NEXT_POS_HINT = 13,
  ST_WORDS_ALLOC = 16,
};

constexpr int kTile = 128;          // slots per key/value tile, queries per query tile
constexpr int kProjTileN = 160;     // output columns per QKV-projection CTA (the weight tile's rows)
constexpr int kEmptyPos = INT32_MIN;

// Device-side view of one ring (plain pointers into the caller's buffer).
struct RingDev {
  uint8_t* k;          // [H][C][D] E4M3 codes, keys already rotated
  uint8_t* v;          // [H][C][D] E4M3 codes
  int32_t* slot_pos;   // [C] position of each slot, INT32_MIN when empty
  float* scales;       // [4H]: scale_k, scale_v, inv_scale_k, inv_scale_v
  int32_t* state;      // [ST_WORDS_ALLOC]
  uint32_t* amax;      // [2H] calibration maxima as float bits (0 between calls)
  const float* table;  // [max_position][D/2][2] fp32 (cos, sin)
  float* part_o;       // [max_splits][qtiles][H][128][D] attention partials (rings allowing more
                       // than 8 splits only; NULL otherwise)
  float* part_lse;     // [max_splits][qtiles][H][128]
  int32_t* tickets;    // [qtiles][H] split completion counters (0 between calls)
  int32_t* levels;     // [qtiles][H] precision level of each query tile
  int H, D, C, max_pos, max_tokens, max_splits, qtiles_max;
  int P;               // pinned prefix slots; tokens past it cycle over slots [P, C)
  int pt, py;          // 3-D RoPE: temporal and row pairs (pt = 0: 1-D RoPE)
};

// Coordinate (0 = t, 1 = y, 2 = x) a rotation pair takes its position from;
// 0 with 1-D RoPE, whose positions are one int32 per token.
__host__ __device__ inline int rope_axis(const RingDev& r, int pair) {
  return pair < r.pt || r.pt == 0 ? 0 : (pair < r.pt + r.py ? 1 : 2);
}
// Position of token t for pair `pair`: pos is [n] (1-D) or [n][3] (3-D).
__device__ __forceinline__ int rope_pos(const RingDev& r, const int32_t* pos, int t, int pair) {
  return r.pt == 0 ? __ldg(pos + t) : __ldg(pos + 3 * t + rope_axis(r, pair));
}

// ---------------------------------------------------------------- E4M3 ----
// Two fp32 values to two E4M3 codes (round to nearest even, saturating to
// +-448); `lo` lands in the low byte.  The PTX conversion puts its first
// source operand in the upper half of the result.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (low byte first) to two fp32 values, exactly (via f16).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  __half2 hh = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hh);
}

// Packed half-precision helpers (low element in the low half / low byte).
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// The two halves of an f16 pair (low half first) as fp32, exactly.
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h2) {
  float2 r;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(h2));
  return r;
}
__device__ __forceinline__ uint16_t f16x2_to_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Each half of h rounded to nearest with 4 significant bits (E4M3's normal
// precision) by Veltkamp splitting in f16 (11 bits) with C = 2^7 + 1:
// c = C h, hi = c - (c - h).  Valid for |h| < 65504 / 129.
__device__ __forceinline__ uint32_t f16x2_hi4(uint32_t h) {
  const uint32_t c = hmul2_u32(h, 0x58085808u);  // 129.0 in both halves
  return hsub2_u32(c, hsub2_u32(c, h));
}

// --------------------------------------------------------------- misc -----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// max(a, b, c) in one instruction (sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Programmatic dependent launch: let the next kernel in the stream start,
// and wait until the previous kernel's results are visible.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t addr) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(addr), "r"(tx)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// A relaxed load at device scope: a read of a word that a preceding kernel
// may still be writing, used only as a guess that is checked later.
__device__ __forceinline__ int ld_relaxed_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Four consecutive words by one relaxed load at device scope (16-byte aligned).
__device__ __forceinline__ int4 ld_relaxed_gpu_v4(const int32_t* p) {
  int4 v;
  asm volatile("ld.relaxed.gpu.global.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// The matching relaxed store, for a word that is only ever a guess.
__device__ __forceinline__ void st_relaxed_gpu(int32_t* p, int v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Non-blocking probe of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Gives up (returning
// false and raising *abort) after `limit_ns` of wall time, or at once when
// another thread of the CTA already raised *abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity,
                                                  volatile int* abort, uint64_t limit_ns) {
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// ------------------------------------------------------------ cp.async ---
// 16-byte global -> shared copy that bypasses registers (and L1); grouped by
// cp_async_commit, complete for the issuing thread after cp_async_wait_all.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Wait until at most N of this thread's most recent groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_stages() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// -------------------------------------------------------------- cluster ---
// Barrier over every thread of every CTA of the cluster (all warps
// converged), with release / acquire ordering of shared-memory accesses.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of the same variable in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ------------------------------------------------------------------ TMA ---
// Fetch a tensor map (a kernel parameter) into the descriptor cache ahead of
// its first copy.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}

// Contiguous global -> shared copy on the async proxy (16-byte aligned,
// size a multiple of 16), completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar)
      : "memory");
}

// Shared memory of this CTA -> shared memory of a CTA of the cluster (both
// addresses 16-byte aligned, size a multiple of 16); completes on the
// destination CTA's mbarrier (a shared::cluster address).  The issuing
// thread learns that the source has been read with bulk_wait_read().
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Prefetch a contiguous global range into L2 (16-byte aligned, size a
// multiple of 16); a hint with no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------- tcgen05 ---
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], E4M3 x E4M3 -> fp32.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every previously issued tcgen05 op of this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (warp quarter base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc], E4M3 x E4M3 -> fp32.  A occupies
// 128 lanes x (K / 4) columns, four E4M3 values per 32-bit column.
__device__ __forceinline__ void mma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same two MMAs with each shared-memory descriptor given as its low
// and high 32-bit words, so an issuing loop can step addresses with one
// 32-bit add (the start address lives in the low word, in 16-byte units).
__device__ __forceinline__ void mma_e4m3_w(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                           uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p, %7, 0;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(0), "r"(accumulate)
      : "memory");
}
// D (f32, TMEM) (+)= A (f16, TMEM, two values per 32-bit column, the lower
// k index in the low half) x B (f16, shared memory descriptor).
__device__ __forceinline__ void mma_f16_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_e4m3_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Round an fp32 value to 3 mantissa bits, nearest-even, in fp32 (the value
// an E4M3 code holds, for magnitudes in E4M3's normal range).
__device__ __forceinline__ float round_mant3(float x) {
  uint32_t b = __float_as_uint(x);
  b = (b + 0x7FFFFu + ((b >> 20) & 1u)) & 0xFFF00000u;
  return __uint_as_float(b);
}

// 32 lanes x N consecutive columns (N = 8, 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 8 || N == 16 || N == 32, "x8, x16 or x32");
  if constexpr (N == 32) {
    tmem_ld32(taddr, r);
  } else if constexpr (N == 16) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
  } else {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
  }
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 8 || N == 16 || N == 32, "x8, x16 or x32");
  if constexpr (N == 32) {
    tmem_st32(taddr, r);
  } else if constexpr (N == 16) {
    tmem_st16(taddr, r);
  } else {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
  }
}

__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  return r;
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (sm_100 family format):
// start address, leading / stride byte offsets (16-byte units), the fixed
// version field, and the swizzle mode (2 = 128-byte, 4 = 64-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle_mode & 7u) << 61;
  return d;
}

// Instruction descriptor for kind::f8f6f4, E4M3 x E4M3 with fp32
// accumulation; B either K-major (b_mn_major = false) or MN-major.
// Instruction descriptor of kind::f16 with f16 A and B and an f32
// accumulator (the same field layout as above; f16 is type code 0).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4)                                   // D format: f32
         | (0u << 7) | (0u << 10)                    // A, B: f16
         | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
         | ((uint32_t)(N >> 3) << 17)                // N / 8
         | ((uint32_t)(M >> 4) << 24);               // M / 16
}

__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool b_mn_major) {
  return (1u << 4)                                   // D format: f32
         | (0u << 7) | (0u << 10)                    // A, B: E4M3
         | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
         | ((uint32_t)(N >> 3) << 17)                // N / 8
         | ((uint32_t)(M >> 4) << 24);               // M / 16
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile of rows of
// `row_bytes` (64 or 128) stored with the matching TMA / UMMA swizzle
// (the chunk index is XOR-ed with address bits 7.. of the row start).
__device__ __forceinline__ uint32_t swz_offset(int row, int chunk, int row_bytes) {
  const uint32_t off = (uint32_t)row * row_bytes + (uint32_t)chunk * 16u;
  const uint32_t mask = row_bytes == 128 ? 7u : 3u;
  return off ^ (((off >> 7) & mask) << 4);
}

}  // namespace kvr

// Launchers implemented in the kernel translation units.
namespace kvr {
cudaError_t launch_calibrate(const RingDev& r, const void* k, const void* v, const int32_t* pos,
                             int n, cudaStream_t s);
// late: the preceding kernel may write k or v, so the frame is read only
// after the wait for it; idle: no kernel that may still run touches the
// ring, so (with default positions) the whole write happens before the wait
cudaError_t launch_write(const RingDev& r, const void* k, const void* v, const int32_t* pos, int n,
                         bool late, bool idle, cudaStream_t s);
cudaError_t launch_delta(const RingDev& r, int delta, bool idle, cudaStream_t s);
cudaError_t launch_write_floor(const RingDev& r, int n, bool idle, cudaStream_t s);
cudaError_t launch_encode_e4m3(const float* in, uint8_t* out, int64_t n, cudaStream_t s);
cudaError_t launch_project(const RingDev& r, const CUtensorMap* tmX, const CUtensorMap* tmW,
                           const int32_t* pos, void* q_out, void* kv_out, int n, int dm, int flags,
                           cudaStream_t s);
cudaError_t project_prepare();

struct AttnLaunch {
  const void* q;
  const int32_t* qpos;
  void* out;
  int n_q;
  int out_bf16;
  int nsplit;
  int tiles_per_split;
  int forced_level;
  int debug_stall;                 // test support: make the first QK wait time out
  int q_late;                      // the preceding kernel may write q: read it after the wait
  int debug_guess;                 // test support: speculate on wrong default positions
  unsigned long long wait_ns;      // limit of every bounded wait in the kernel
};
// Batched write / delta over rings of one shape (kernel parameters: no
// device memory is needed to describe the batch).
constexpr int kMaxBatch = 64;
struct WriteMany {
  RingDev r[kMaxBatch];
  const uint16_t* k[kMaxBatch];
  const uint16_t* v[kMaxBatch];
  const int32_t* pos[kMaxBatch];
};
struct DeltaMany {
  RingDev r[kMaxBatch];
};
cudaError_t cache_prepare();   // kernel attributes (shared-memory size) of the cache kernels
cudaError_t launch_write_many(const WriteMany& b, int count, int n, cudaStream_t s);
cudaError_t launch_delta_many(const DeltaMany& b, int count, int delta, cudaStream_t s);
cudaError_t launch_legacy_upkeep(const RingDev& r, const void* wk_in, const void* wv_in, void* wk_out,
                                 void* wv_out, const void* k, const void* v, int n, cudaStream_t s);
cudaError_t launch_attention(const RingDev& r, const CUtensorMap* tmK, const CUtensorMap* tmV,
                             const AttnLaunch& a, cudaStream_t s);
size_t attention_smem_bytes(int D);
// Fixed-size static device scratch used by kvring_attention_noalloc, and
// its device address on the current device (looked up once per device).
size_t static_scratch_bytes();
cudaError_t static_scratch_address(void** out);
// Once per process and head size, before the first launch (not capturable).
cudaError_t attention_prepare(int D);
}  // namespace kvr
