// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// (tiled tensor and plain bulk copies), Tensor Memory allocation and
// load/store, tcgen05.mma issue and commit, and the shared-memory and
// instruction descriptors those MMAs take.
//
// Every wait here is bounded: it gives up after a wall-clock limit, or as soon
// as another thread of the grid has raised the abort word, and reports failure
// so that the caller can drain its in-flight copies, free Tensor Memory and
// return.  No trap, no assert.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace bam {

// ---------------------------------------------------------------- basics
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async (TMA / tensor core) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware until the phase
// completes or about `hint_ns` nanoseconds have passed, instead of returning
// at once: a waiting warp then issues almost nothing.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Device status words shared by every CTA of a launch (in the caller's
// workspace).  The first error recorded stays until the host reads it
// (bam_attn_check_status): the first kernel of each call clears only the
// abort word, so that a later call on the same workspace neither erases nor
// overwrites an unread error.  `magic` marks a status area that has been
// initialised; a workspace whose magic does not match (fresh memory) has
// its status cleared by the first kernel of the call instead.
struct DevStatus {
  int abort;      // nonzero: some thread gave up; everyone else leaves early
  int code;       // first error code recorded (BAM_DEV_*)
  int site;       // where it happened (kernel-specific)
  int block;      // which block
  unsigned magic[2];
  // Debug builds (BAM_DEBUG) only: when positive, the bounded waits of the
  // call count it down and the wait that takes it to zero gives up as if its
  // time limit had passed (bam_attn_debug_arm_giveup).  Ignored otherwise.
  int giveup;
};

constexpr unsigned kStatusMagic0 = 0x4d414221u, kStatusMagic1 = 0x53544154u;

// Start of a call: one thread of the call's first kernel, before any other
// kernel of the call looks at the status.
__device__ __forceinline__ void status_begin_call(DevStatus* st) {
  if (st->magic[0] != kStatusMagic0 || st->magic[1] != kStatusMagic1) {
    st->code = 0;
    st->site = 0;
    st->block = 0;
    st->giveup = 0;
    st->magic[0] = kStatusMagic0;
    st->magic[1] = kStatusMagic1;
  }
  st->abort = 0;
}

// BAM_DEV_BAD_ARG: an argument only the device reads was out of range (a
// cache length of the ragged decode); the kernel clamped it and went on.
// BAM_DEV_BOUNDS: a debug build (BAM_DEBUG) found a bulk copy whose source
// left its buffer or broke the 16-byte rule; the copy was not issued.
enum : int {
  BAM_DEV_OK = 0,
  BAM_DEV_TIMEOUT = 1,
  BAM_DEV_ABORTED = 2,
  BAM_DEV_BAD_ARG = 3,
  BAM_DEV_BOUNDS = 4
};

// Wall-clock budget of one wait.  Normal waits last microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
// Longest hardware sleep of one try in the slow path: short enough that the
// abort words and the wall clock are still checked often.
constexpr uint32_t kWaitSleepNs = 20000;  // 20 us

// Records `code` (the first error of the call wins) and raises the CTA and
// grid abort words, so that every bounded wait of the grid gives up.
__device__ __forceinline__ void raise_error(DevStatus* st, volatile int* cta_abort, int site,
                                            int code) {
  *cta_abort = 1;
  if (atomicCAS(&st->code, BAM_DEV_OK, code) == BAM_DEV_OK) {
    st->site = site;
    st->block = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  }
  atomicExch(&st->abort, 1);
}
__device__ __forceinline__ void raise_abort(DevStatus* st, volatile int* cta_abort, int site) {
  raise_error(st, cta_abort, site, BAM_DEV_TIMEOUT);
}

// Slow path of mbar_wait: spins with a wall-clock limit.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, DevStatus* st,
                                            volatile int* cta_abort, int site) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if ((it & 3u) == 0) {
      if (*cta_abort) return false;
      if (*reinterpret_cast<volatile int*>(&st->abort)) {
        *cta_abort = 1;
        return false;
      }
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        raise_abort(st, cta_abort, site);
        return false;
      }
    }
  }
}

// Bounded wait on phase `parity`.  Returns false when the wait gave up (own
// timeout, a CTA-local abort, or the grid-wide abort word).  In a debug build
// an armed give-up count (DevStatus::giveup) makes the wait that exhausts it
// give up at once, as if its time limit had passed, so that tests can drive
// every kernel through its give-up and drain path.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, DevStatus* st,
                                          volatile int* cta_abort, int site) {
#ifdef BAM_DEBUG
  if (*reinterpret_cast<volatile int*>(&st->giveup) > 0 && atomicSub(&st->giveup, 1) == 1) {
    raise_abort(st, cta_abort, site);
    return false;
  }
#endif
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, st, cta_abort, site);
}

// Wait used on the error path only: bounded, ignores the abort words.
static __device__ __noinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled load (coordinates innermost first) completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Plain bulk copy global -> shared; both addresses 16-B aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Counts `bytes` of an expected transfer as arrived without copying them.
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// bulk_load with the checks of a debug build.  With BAM_DEBUG defined, the
// copy is issued only when its source [src, src + bytes) lies inside
// [lo, hi) and src, dst and bytes meet the 16-byte rule; otherwise the
// bytes are counted as arrived on `bar` (so no wait on it hangs), the error
// BAM_DEV_BOUNDS is recorded with `site`, the grid is aborted and false is
// returned.  Without BAM_DEBUG this is bulk_load and returns true; the
// bounds are then unused.
__device__ __forceinline__ bool bulk_load_checked(void* dst, const void* src, uint32_t bytes,
                                                  uint64_t* bar, const void* lo, const void* hi,
                                                  DevStatus* st, volatile int* cta_abort,
                                                  int site) {
#ifdef BAM_DEBUG
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src);
  const bool inside = s0 >= reinterpret_cast<uintptr_t>(lo) &&
                      s0 + bytes <= reinterpret_cast<uintptr_t>(hi);
  const bool aligned16 = ((s0 | smem_u32(dst) | bytes) & 15u) == 0;
  if (!inside || !aligned16 || bytes == 0) {
    mbar_complete_tx(bar, bytes);
    raise_error(st, cta_abort, site, BAM_DEV_BOUNDS);
    return false;
  }
#else
  (void)lo;
  (void)hi;
  (void)st;
  (void)cta_abort;
  (void)site;
#endif
  bulk_load(dst, src, bytes, bar);
  return true;
}

// Debug-build check of the row coordinate of a tiled store or reduction
// (which must not start at a negative coordinate): records BAM_DEV_BOUNDS
// and returns false when c1 is outside [0, rows).  Always true without
// BAM_DEBUG.
__device__ __forceinline__ bool store_row_ok(int c1, int rows, DevStatus* st,
                                             volatile int* cta_abort, int site) {
#ifdef BAM_DEBUG
  if (c1 < 0 || c1 >= rows) {
    raise_error(st, cta_abort, site, BAM_DEV_BOUNDS);
    return false;
  }
#else
  (void)c1;
  (void)rows;
  (void)st;
  (void)cta_abort;
  (void)site;
#endif
  return true;
}

// Element-wise add of a shared-memory tile into global memory through a 3-D
// tensor map (TMA reduction); coordinates innermost first, none negative.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, const void* src, int c0,
                                                  int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Tiled bulk store shared -> global (rows outside the tensor are not written).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk group has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Order generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- Tensor Memory
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
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
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// tcgen05.ld writes its destination registers asynchronously; they are
// valid only after tcgen05.wait::ld.  This empty statement, placed after the
// wait, makes the 32 registers depend on it so that no use is scheduled
// above the wait.
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile("" : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]),"+r"(r[8]),"+r"(r[9]),"+r"(r[10]),"+r"(r[11]),"+r"(r[12]),"+r"(r[13]),"+r"(r[14]),"+r"(r[15]),"+r"(r[16]),"+r"(r[17]),"+r"(r[18]),"+r"(r[19]),"+r"(r[20]),"+r"(r[21]),"+r"(r[22]),"+r"(r[23]),"+r"(r[24]),"+r"(r[25]),"+r"(r[26]),"+r"(r[27]),"+r"(r[28]),"+r"(r[29]),"+r"(r[30]),"+r"(r[31]));
}

__device__ __forceinline__ void reg_fence8(uint32_t* r) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]));
}
__device__ __forceinline__ void reg_fence16(uint32_t* r) {
  asm volatile("" : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]),"+r"(r[8]),"+r"(r[9]),"+r"(r[10]),"+r"(r[11]),"+r"(r[12]),"+r"(r[13]),"+r"(r[14]),"+r"(r[15]));
}

// Lane quarter of this warp: warp w may touch TMEM lanes [32*(w%4), 32*(w%4)+32).
__device__ __forceinline__ uint32_t tmem_lane_base(uint32_t warp) {
  return (32u * (warp & 3u)) << 16;
}

__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}

// ---------------------------------------------------------------- tcgen05.mma
// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format):
//   [0,14) start address >> 4, [16,30) leading byte offset >> 4,
//   [32,46) stride byte offset >> 4, [46,49) fixed 0b001, [61,64) swizzle (2 = 128B).
// K-major tile (rows of 128 B): SBO = 1024 (next 8-row group), LBO unused.
// MN-major tile: SBO = 1024 (next 8 rows along K), LBO = next 64-element
// block along M/N.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and an f32 accumulator:
//   [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format,
//   bit 15 A is MN-major, bit 16 B is MN-major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- register split
// Warpgroup-wide register budget changes; every warp of the warpgroup must
// execute the same one.
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// lo_acc += low bf16 half of w, hi_acc += high half: the widening to fp32 is
// exact, so this equals adding the unpacked values (sm_100+ mixed-type add).
__device__ __forceinline__ void add_bf16x2_f32(uint32_t w, float& lo_acc, float& hi_acc) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n add.rn.f32.bf16 %0, l, %0;\n"
      " add.rn.f32.bf16 %1, h, %1;\n}\n"
      : "+f"(lo_acc), "+f"(hi_acc)
      : "r"(w));
}

// Packed pairs of fp32 values in one 64-bit register pair (sm_100+ f32x2 ops).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Four consecutive fp32 values from a 16-byte aligned address as two f32x2
// pairs (values 0,1 and 2,3): one vector load.
__device__ __forceinline__ void ld_f2x2(const float* p, uint64_t& a, uint64_t& b) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  a = f2_pack(v.x, v.y);
  b = f2_pack(v.z, v.w);
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace bam
