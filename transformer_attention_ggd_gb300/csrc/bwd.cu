// Fused GGD-BAM attention backward for sm_103a (tcgen05 / TMEM / TMA).
//
// The pages give no backward; this is the chain rule of L = sum(O * dO)
// through the forward of fwd.cu:
//   P_ij  = exp(z_ij - LSE_i),  z_ij = c_i q_i.k_j + b_h(i - j)
//   dP_ij = dO_i . v_j,  Delta_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - Delta_i)
//   dV_j += sum_i P_ij dO_i,  dK_j += sum_i c_i dS_ij q_i,  dQ_i += sum_j c_i dS_ij k_j
//   dalpha_h = -(beta_h/alpha_h) sum dS b,  dbeta_h = sum dS db/dbeta,
//   dmu_h = sum dS db/dmu,  ds_h = sum dS ln(n_i) q_i.k_j / sqrt(D)   (SSMax)
// with db/dbeta and db/dmu read from the distance tables written by table.cu.
//
// Delta_i is taken from the forward's O, which carries the bf16 rounding of
// the weights in its PV product (or a bf16 output).  That error enters each
// scalar-gradient sum as -dDelta_i * sum_j P_ij X_ij without cancelling, so
// the kernel also accumulates, per row, B_i = sum_j P_ij X_ij and the exact
// C_i = sum_j P_ij dP_ij, and the final kernel adds sum_i (Delta_i - C_i) B_i:
//   sum_ij P_ij (dP_ij - C_i) X_ij = sum_ij dS_ij X_ij + sum_i (Delta_i - C_i) B_i.
//
// Persistent: one CTA per SM walks a list of work items, each a 128-key
// tile of one (b, h), and for each the 128-row query tiles that see it (the
// next item's K/V and first S/dP overlap the current item's last tile and
// its dK/dV epilogue):
//   warp 8     TMA producer: K, V once; per query tile Q, dO and the three
//              256-entry distance windows (b, db/dbeta, db/dmu, four shifted
//              reversed copies each for 16-byte loads), 2 stages.
//   warp 9     MMA issuer: S = Q K^T and dP = dO V^T (M = queries), then
//              dV += P^T dO and dK += (c dS)^T Q (A operands MN-major in shared
//              memory, M = keys) and dQ = (c dS) K (A = the same (c dS)^T
//              buffer read K-major: its layout is that of c dS, M = queries).
//              S and dP of the next query tile are issued as soon as every
//              element-wise warp has read its last S/dP columns of this one,
//              so they overlap the end of this tile's element-wise work.
//   warp 10    dQ reducer: issues the TMA reduction of each staged dQ tile
//              into the fp32 accumulator and frees the staging tile; at an
//              item's end, the TMA stores of its dK and dV.
//   warps 0-7  two warps per TMEM lane quarter; each thread owns one query
//              row and half (64 keys) of the tile, in 16-key chunks of two
//              passes (the derivative-table loads after P and dS): P, dS, the
//              scalar-gradient sums (as f32x2 pairs of partial sums), P and
//              c*dS to shared memory (each chunk stored one chunk later, so
//              the wait for the previous tile's products overlaps
//              arithmetic); the finished dQ tile goes to a shared
//              staging tile for warp 10.  At an item's end, its dK and dV rows
//              (TMEM lane = key) are staged as bf16 for warp 10.  Eight such
//              warps (168 registers, a few tens of bytes of spill stores)
//              measured as fast as sixteen (96 registers, more spills) and
//              leave the MMA issuer fewer busy warps on its scheduler.
// TMEM columns: S [0,128) dP [128,256) dQ [320,384) dK [384,448)
//               dV [448,512); [256,320) is unused.
#include <algorithm>
#include <climits>
#include <mutex>
#include <type_traits>
#include <vector>

#include "table_eval.cuh"

namespace bam {
namespace {

constexpr int kBStages = 2;
// Element-wise warps, a multiple of 4 (kBCompute / 4 per TMEM lane quarter).
constexpr int kBCompute = 8;
// + producer + MMA issuer + dQ reducer: 11 warps, at most 3 on one
// scheduler, so 168 registers per thread fit its share of the register file.
constexpr int kBThreads = 32 * (kBCompute + 3);
constexpr int kBProducerWarp = kBCompute;
constexpr int kBMmaWarp = kBCompute + 1;
constexpr int kBDqWarp = kBCompute + 2;
constexpr int kBKeysPerWarp = 128 / (kBCompute / 4);  // keys of the tile per thread
constexpr int kBDims = kHeadDim / (kBCompute / 4);     // dQ/dK/dV columns per warp
constexpr int kTile = 128 * 64 * 2;  // 16 KB bf16 tile
constexpr int kBWin = 256;            // window entries per query tile
constexpr int kBWinCopy = kBWin + 4;  // entries per reversed copy (shifts of 0..3)
constexpr int kBWinCopyStride = 288;
constexpr int kBWinPlane = kTabCopies * kBWinCopyStride;
static_assert(win_copy_off(kTabCopies - 1, kBWinCopyStride) + kBWinCopy <= kBWinPlane, "window");

struct __align__(1024) BwdSmem {
  uint8_t k[kTile];
  uint8_t v[kTile];
  uint8_t q[kBStages][kTile];
  uint8_t dO[kBStages][kTile];
  uint8_t pt[2 * kTile];   // P^T as an MN-major A operand: 2 atoms of 64 keys x 128 queries
  uint8_t dst[2 * kTile];  // (c dS)^T, same layout
  float dqs[2][128][32];   // dQ tile staged for the TMA reduction: two 128-B-swizzled boxes
  float win[kBStages][3][kBWinPlane];  // b, db/dbeta, db/dmu: four reversed copies each
  float red[2][kBCompute][4];  // per-item scalar sums, by item parity
  uint64_t kv_full;
  uint64_t k_empty;   // the item's K no longer read (after its last dQ product)
  uint64_t v_empty;   // the item's V no longer read (after its last dP product)
  uint64_t dqs_full;
  uint64_t dqs_free;
  uint64_t epi_full;   // dK/dV of an item staged (bf16) in the P^T buffer
  uint64_t epi_free;   // that staging read by its TMA stores
  uint64_t qd_full[kBStages];
  uint64_t qd_empty[kBStages];
  uint64_t s_full;
  uint64_t sdp_free;
  uint64_t ds_ready;
  uint64_t mma_done;
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort_flag;
};

enum : int {
  kSiteBProd = 50,
  kSiteBMmaKV = 60,
  kSiteBMmaQD = 61,
  kSiteBMmaDS = 62,
  kSiteBMmaFree = 63,
  kSiteBDq = 64,
  kSiteBWgS = 70,
  kSiteBWgQD = 71,
  kSiteBWgDone = 72,
  kSiteBWgDq = 73,
  // Debug-build bounds checks (BAM_DEV_BOUNDS)
  kSiteBWindowCopy = 74,
  kSiteBRow = 75
};

constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 320, kColDK = 384, kColDV = 448;

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, DevStatus* st,
                                          volatile int* ab, int site) {
  const bool ok = mbar_wait(bar, parity, st, ab, site);
  return __all_sync(0xffffffffu, ok);
}

// Barrier 1 over the element-wise warps, returning whether every thread
// passed ok != 0 (all of them reach it once per work item).
__device__ __forceinline__ int elementwise_barrier_and(int ok) {
  int all;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 q, %1, 0;\n bar.red.and.pred p, 1, %2, q;\n"
      " selp.s32 %0, 1, 0, p;\n}\n"
      : "=r"(all)
      : "r"(ok), "n"(32 * kBCompute)
      : "memory");
  return all;
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Adds v, a partial sum of scalar-gradient term x of head h (0: sum dS b in
// log2 units, 1: sum dS db/dbeta, 2: sum dS db/dmu, 3: the SSMax sum), to
// that head's output, which the preprocess zeroed.  Each output is a fixed
// multiple of its sum: d/dalpha = -(beta / alpha) ln 2 sum dS b (log2 units)
// since db/dalpha = -beta b / alpha, or ln 2 sum dS b with the theta prior
// (db/dtheta_alpha = b); the others are the sums themselves, and ds stays 0
// without SSMax.
__device__ __forceinline__ void add_head_grad(const BwdArgs& a, int x, int h, float v) {
  if (x == 0) {
    const float f = a.tab.prior == kPriorTheta
                        ? kLn2f
                        : -(__ldg(a.beta + h) / __ldg(a.alpha + h)) * kLn2f;
    atomicAdd(a.dalpha + h, f * v);
  } else if (x == 1) {
    atomicAdd(a.dbeta + h, v);
  } else if (x == 2) {
    atomicAdd(a.dmu + h, v);
  } else if (a.ssmax) {
    atomicAdd(a.ds + h, v);
  }
}

// Byte offset of element (m, k) of a 128 x 128 bf16 MN-major operand
// (m = key, contiguous; k = query) in the 128-byte-swizzled layout: atoms of
// 64 m-values; within an atom, row k at (k/8)*1024 + (k%8)*128 and the
// 16-byte chunk m/8 swizzled with k%8.
__device__ __forceinline__ uint32_t mn_chunk_offset(int m8, int k) {
  // m8: index of the 8-key chunk (0..15)
  return (m8 >> 3) * kTile + (k >> 3) * 1024 + (k & 7) * 128 + (((m8 & 7) ^ (k & 7)) << 4);
}

// Work item w of a persistent CTA: key tile kb of head bh (item index
// kb * B * H + bh; causal: kb = 0 sees every query tile).  With a schedule
// (BwdSched::n > 0) CTA c takes items item[start[c]] .. item[start[c+1]-1]
// in that order; otherwise items are taken longest first and dealt out in
// rounds, alternating direction ("snake") so that long and short items mix.
struct BwdItem {
  int kb, bh, h, j0, q_first, nq;
};

// Per-CTA item lists, passed by value as a kernel parameter (2.4 KB; larger
// problems keep the round-robin deal).
constexpr int kSchedMaxCtas = 160;
constexpr int kSchedMaxItems = 1024;
struct BwdSched {
  int n;  // scheduled items; 0: the kernel deals them out itself
  uint16_t start[kSchedMaxCtas + 1];
  uint16_t item[kSchedMaxItems];
};

__device__ __forceinline__ bool bwd_item(const BwdArgs& a, const BwdSched& sc, int round,
                                         BwdItem& it) {
  const int BH = a.B * a.H;
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  int idx;
  if (sc.n > 0) {
    const int p = sc.start[c] + round;
    if (p >= sc.start[c + 1]) return false;
    idx = sc.item[p];
  } else {
    idx = round * G + ((round & 1) ? (G - 1 - c) : c);
    if (idx >= a.nkb * BH) return false;
  }
  it.kb = idx / BH;
  it.bh = idx % BH;
  it.h = it.bh % a.H;
  it.j0 = it.kb * 128;
  it.q_first = a.causal ? it.kb : 0;
  it.nq = a.nkb - it.q_first;
  return true;
}

__global__ void __launch_bounds__(kBThreads, 1)
    bam_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
                   const __grid_constant__ CUtensorMap tdv, const BwdArgs a,
                   const __grid_constant__ BwdSched sc) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // Aligned by an offset from the shared array itself (not through an
  // integer cast), so that accesses stay in the shared address space.
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw + ((0u - smem_u32(smem_raw)) & 1023u));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* ab = &sm.abort_flag;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.k_empty, 1);
    mbar_init(&sm.v_empty, 1);
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&sm.qd_full[s], 1);
      mbar_init(&sm.qd_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.sdp_free, kBCompute);
    mbar_init(&sm.ds_ready, kBCompute);
    mbar_init(&sm.dqs_full, kBCompute);
    mbar_init(&sm.dqs_free, 1);
    mbar_init(&sm.epi_full, kBCompute);
    mbar_init(&sm.epi_free, 1);
    mbar_init(&sm.mma_done, 1);
    mbar_init(&sm.mma_final, 1);
    fence_barrier_init();
  }
  if (warp == kBMmaWarp) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Tables, Delta, the zeroed accumulators and the cleared status word come
  // from the preprocess.  Only the producer runs ahead of it (its K, V, Q
  // and dO loads need nothing from it); every other thread waits here,
  // before its first look at the status word.
  if (warp != kBProducerWarp) grid_dep_wait();
  const uint32_t tm = sm.tmem_base;
  const size_t copy_stride = static_cast<size_t>(a.H) * a.tab_len;  // floats between copies
  const size_t plane = kTabCopies * copy_stride;
  // End of the three tables and their padding: a window starts inside its
  // own row and may run past the row's end, never past this.
  const float* tab_end = a.table + 3 * plane + kTabPadFloats;

  // Barrier phases: per query tile g (counted over all items of this CTA)
  // for the Q/dO ring and the tile hand-offs; per item n for K/V.
  if (warp == kBProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = (*ab == 0);
      int g = 0, n = 0;
      int issued = 0;  // query tiles whose Q/dO/window copies were issued
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      BwdItem it;
      for (int round = 0; ok && bwd_item(a, sc, round, it); ++round) {
        for (int t = 0; ok && t < it.nq; ++t, ++g) {
          const int s = g % kBStages;
          const int i0 = (it.q_first + t) * 128;
          if (g >= kBStages) {
            ok = mbar_wait(&sm.qd_empty[s], ((g / kBStages) - 1) & 1, a.status, ab, kSiteBProd);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(&sm.qd_full[s], 2 * kTile + 3 * kTabCopies * kBWinCopy * 4);
          tma_load_3d(sm.q[s], &tq, &sm.qd_full[s], 0, i0, it.bh);
          tma_load_3d(sm.dO[s], &tdo, &sm.qd_full[s], 0, i0, it.bh);
          if (g == 0) grid_dep_wait();  // the windows come from the preprocess
          // Window: table indices tab_off + i0 - j0 - 128 + [0, kBWin), which
          // start at tab_len - kBWin minus that base in the reversed rows.
          const float* src = a.table + static_cast<size_t>(it.h) * a.tab_len +
                             (a.tab_len - kBWin - (a.tab_off + i0 - it.j0 - 128));
          for (int p = 0; p < 3; ++p)
            for (int k = 0; k < kTabCopies; ++k)
              ok &= bulk_load_checked(
                  sm.win[s][p] + win_copy_off(k, kBWinCopyStride), src + p * plane + k * copy_stride,
                  kBWinCopy * 4, &sm.qd_full[s],
                  a.table + p * plane + k * copy_stride + static_cast<size_t>(it.h) * a.tab_len,
                  tab_end, a.status, ab, kSiteBWindowCopy);
          issued = g + 1;
          if (!ok) break;
          if (t == 0) {
            // K and V of the item into the single K/V buffers: V as soon as
            // the previous item's last dP product is done, K after its last
            // dQ product (issued first among that tile's gradient products).
            // kv_full is armed only after v_empty: that product was issued
            // after the MMA warp saw the previous K/V phase complete, so the
            // barrier is never armed while that phase still has bytes in
            // flight (a one-tile item is followed at once by the next item,
            // before its own K/V loads need have landed).
            if (n > 0) {
              ok = mbar_wait(&sm.v_empty, (n - 1) & 1, a.status, ab, kSiteBProd);
              if (!ok) break;
            }
            mbar_arrive_expect_tx(&sm.kv_full, 2 * kTile);
            tma_load_3d(sm.v, &tv, &sm.kv_full, 0, it.j0, it.bh);
            // After a failed wait K is loaded all the same (the kernel is
            // giving up, so what K's buffer feeds no longer matters): the
            // phase then completes and the drain below sees both copies land.
            if (n > 0) ok = mbar_wait(&sm.k_empty, (n - 1) & 1, a.status, ab, kSiteBProd);
            tma_load_3d(sm.k, &tk, &sm.kv_full, 0, it.j0, it.bh);
            ++n;
            if (!ok) break;
          }
        }
      }
      // Copies still in flight land before this CTA leaves.
      if (n > 0) mbar_drain(&sm.kv_full, (n - 1) & 1);
      for (int x = max(0, issued - kBStages); x < issued; ++x)
        mbar_drain(&sm.qd_full[x % kBStages], (x / kBStages) & 1);
    }
  } else if (warp == kBMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = (*ab == 0);
      const uint32_t idSP = idesc_bf16(128, 128, false, false);
      const uint32_t idKV = idesc_bf16(128, 64, true, true);
      const uint32_t idQ = idesc_bf16(128, 64, false, true);
      // Shared-memory descriptors: K-major views (S, dP) and MN-major views
      // (the gradient products) of the tiles; stages and K-steps are fixed
      // offsets (16-byte units) from these, so each MMA costs an add or two.
      constexpr uint64_t kTileDesc = kTile >> 4;
      const uint64_t qK0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sm.dO[0]), 16, 1024);
      const uint64_t kK = sdesc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t vK = sdesc_sw128(smem_u32(sm.v), 16, 1024);
      const uint64_t qM0 = sdesc_sw128(smem_u32(sm.q[0]), kTile, 1024);
      const uint64_t dM0 = sdesc_sw128(smem_u32(sm.dO[0]), kTile, 1024);
      const uint64_t kM = sdesc_sw128(smem_u32(sm.k), kTile, 1024);
      const uint64_t ptM = sdesc_sw128(smem_u32(sm.pt), kTile, 1024);
      const uint64_t dsM = sdesc_sw128(smem_u32(sm.dst), kTile, 1024);
      // The same buffer read as c dS (M = queries, K = keys), K-major: its
      // 128-byte rows are queries holding 64 keys each, swizzled by query,
      // the second 64 keys one tile further on.
      const uint64_t dsK = sdesc_sw128(smem_u32(sm.dst), 16, 1024);
      // S and dP of global tile g (stage g % 2) once its Q/dO are in; the
      // caller has made sure the S/dP columns are free and K/V are in.
      auto issue_s_dp = [&](int g) -> bool {
        const int s = g % kBStages;
        if (!mbar_wait(&sm.qd_full[s], (g / kBStages) & 1, a.status, ab, kSiteBMmaQD)) return false;
        tc_fence_after();
        const uint64_t qd = qK0 + kTileDesc * s, dd = dK0 + kTileDesc * s;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ss(tm + kColS, qd + 2 * kk, kK + 2 * kk, idSP, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ss(tm + kColDP, dd + 2 * kk, vK + 2 * kk, idSP, kk > 0 ? 1u : 0u);
        umma_commit(&sm.s_full);
        return true;
      };
      int g = 0, n = 0;
      BwdItem it, nxt;
      bool have = bwd_item(a, sc, 0, it);
      if (ok && have) {
        ok = mbar_wait(&sm.kv_full, 0, a.status, ab, kSiteBMmaKV);
        if (ok) ok = issue_s_dp(0);
        if (ok && it.nq == 1) umma_commit(&sm.v_empty);  // that was the item's last dP
      }
      for (int round = 0; ok && have; ++round) {
        const bool have_next = bwd_item(a, sc, round + 1, nxt);
        for (int t = 0; ok && t < it.nq; ++t, ++g) {
          const int s = g % kBStages;
          // S and dP of the item's next tile once this tile's S/dP columns
          // are read (they overlap this tile's last element-wise chunk).
          if (t + 1 < it.nq) {
            ok = mbar_wait(&sm.sdp_free, g & 1, a.status, ab, kSiteBMmaFree);
            if (!ok) break;
            ok = issue_s_dp(g + 1);
            if (!ok) break;
            if (t + 2 == it.nq) umma_commit(&sm.v_empty);  // the item's last dP
          }
          ok = mbar_wait(&sm.ds_ready, g & 1, a.status, ab, kSiteBMmaDS);
          if (!ok) break;
          tc_fence_after();
          const uint64_t qd = qM0 + kTileDesc * s, dd = dM0 + kTileDesc * s;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dQ = (c dS) K
            umma_ss(tm + kColDQ, dsK + (kk >> 2) * kTileDesc + 2 * (kk & 3), kM + 128 * kk, idQ,
                    kk > 0 ? 1u : 0u);
          if (t + 1 == it.nq) umma_commit(&sm.k_empty);  // the item's last use of K
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dV += P^T dO
            umma_ss(tm + kColDV, ptM + 128 * kk, dd + 128 * kk, idKV, (t > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dK += (c dS)^T Q
            umma_ss(tm + kColDK, dsM + 128 * kk, qd + 128 * kk, idKV, (t > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&sm.mma_done);
          umma_commit(&sm.qd_empty[s]);
          if (t + 1 == it.nq) {
            ++n;
            if (have_next) {
              // First S/dP of the next item: its K/V in and this tile's
              // S/dP columns read.
              ok = mbar_wait(&sm.kv_full, n & 1, a.status, ab, kSiteBMmaKV);
              if (!ok) break;
              ok = mbar_wait(&sm.sdp_free, g & 1, a.status, ab, kSiteBMmaFree);
              if (!ok) break;
              ok = issue_s_dp(g + 1);
              if (!ok) break;
              if (nxt.nq == 1) umma_commit(&sm.v_empty);  // the next item's last dP
            }
          }
        }
        it = nxt;
        have = have_next;
      }
      umma_commit(&sm.mma_final);
      mbar_drain(&sm.mma_final, 0);
    }
  } else if (warp == kBDqWarp) {
    // ------------------------------------------------------------ dQ reducer
    if (lane == 0) {
      bool ok = (*ab == 0);
      int g = 0;
      BwdItem it;
      for (int round = 0; ok && bwd_item(a, sc, round, it); ++round) {
        for (int t = 0; ok && t < it.nq; ++t, ++g) {
          ok = mbar_wait(&sm.dqs_full, g & 1, a.status, ab, kSiteBDq);
          if (!ok) break;
          const int i0 = (it.q_first + t) * 128;
          ok = store_row_ok(i0, a.T, a.status, ab, kSiteBRow);
          if (!ok) break;
          tma_reduce_add_3d(&tdq, sm.dqs[0], 0, i0, it.bh);
          tma_reduce_add_3d(&tdq, sm.dqs[1], 32, i0, it.bh);
          bulk_commit();
          bulk_wait_read_all();  // staging tile read: it may be written again
          mbar_arrive(&sm.dqs_free);
        }
        if (!ok) break;
        // The item's dK and dV rows (bf16, staged in the P^T buffer).
        ok = mbar_wait(&sm.epi_full, round & 1, a.status, ab, kSiteBDq);
        if (!ok) break;
        ok = store_row_ok(it.j0, a.T, a.status, ab, kSiteBRow);
        if (!ok) break;
        tma_store_3d(&tdk, sm.pt, 0, it.j0, it.bh);
        tma_store_3d(&tdv, sm.pt + kTile, 0, it.j0, it.bh);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&sm.epi_free);
      }
      // The staging tile must stay valid until the last reduction has read
      // it; the writes themselves complete with the grid.
      bulk_wait_read_all();
    }
  } else {
    // ------------------------------------------------------------ element-wise
    const int r = 32 * (warp & 3) + lane;  // query row within the tile = TMEM lane
    const int hc = warp >> 2;              // which kBKeysPerWarp keys of the tile
    const uint32_t lb = tmem_lane_base(warp);
    const int kq = (r + 1) & 3;
    const int wrev = win_copy_off(kq, kBWinCopyStride) + (127 - r + kq);
    bool ok = (*ab == 0);
    // dQ of a finished query tile: TMEM -> shared staging tile (two
    // 128-byte-swizzled 32-column boxes) for the dQ warp's TMA reductions.
    // Hand-offs use bounded mbarrier waits: the staging tile is written once
    // the dQ warp has seen the previous reduction read it (dqs_free), and
    // every warp arrives on dqs_full when its part is written.
    int n_dq = 0;  // dQ tiles staged so far
    auto dq_epilogue = [&]() -> bool {
      uint32_t dv[kBDims];
#pragma unroll
      for (int u = 0; u < kBDims / 16; ++u)
        tmem_ld_32x32b_x16(tm + lb + kColDQ + kBDims * hc + 16 * u, dv + 16 * u);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < kBDims / 16; ++u) reg_fence16(dv + 16 * u);
      if (n_dq > 0 && !warp_wait(&sm.dqs_free, (n_dq - 1) & 1, a.status, ab, kSiteBWgDq))
        return false;
#pragma unroll
      for (int x = 0; x < kBDims / 4; ++x) {
        const int d0 = kBDims * hc + 4 * x;  // first of four dQ columns
        uint8_t* box = reinterpret_cast<uint8_t*>(sm.dqs[d0 >> 5]);
        const int cc = (d0 & 31) >> 2;       // 16-byte chunk of the 128-byte row
        *reinterpret_cast<uint4*>(box + r * 128 + ((cc ^ (r & 7)) << 4)) =
            make_uint4(dv[4 * x], dv[4 * x + 1], dv[4 * x + 2], dv[4 * x + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.dqs_full);
      ++n_dq;
      return true;
    };
    int g = 0;
    // The row data of a query tile (this thread's LSE and Delta) and the
    // item's SSMax scale are loaded one tile ahead, across item boundaries
    // too, so that no global load sits at the start of a tile.
    float lse_nx = 0.f, del_nx = 0.f, s_nx = 1.0f;
    auto prefetch_row = [&](int bh_, int i_, int h_) {
      if (i_ < a.T) {
        lse_nx = __ldg(a.lse + static_cast<size_t>(bh_) * a.T + i_);
        del_nx = __ldg(a.delta + static_cast<size_t>(bh_) * a.T + i_);
      }
      if (h_ >= 0) s_nx = a.ssmax ? __ldg(a.s + h_) : 1.0f;
    };
    BwdItem it;
    bool have = bwd_item(a, sc, 0, it);
    if (have) prefetch_row(it.bh, it.q_first * 128 + r, it.h);
    for (int round = 0; ok && have; ++round) {
      const int bh = it.bh, j0 = it.j0, q_first = it.q_first, nq = it.nq;
      const float s_h = s_nx;
      // Scalar-gradient sums of the item as f32x2 pairs (even / odd key
      // columns): sum dS b (log2 units), sum dS db/dbeta, sum dS db/dmu, and
      // sum over rows of w_i * sum_j dS S.
      uint64_t accB2 = 0ull, accBeta2 = 0ull, accMu2 = 0ull;
      float acc_s = 0.f;
      for (int t = 0; ok && t < nq; ++t, ++g) {
        const int s = g % kBStages;
        const int i0 = (q_first + t) * 128;
        const int i = i0 + r;
        const bool row_ok = i < a.T;
        const float lse_row = lse_nx, del_row = del_nx;
        if (t + 1 < nq) {
          prefetch_row(bh, i + 128, -1);
        } else {
          BwdItem nxt;
          if (bwd_item(a, sc, round + 1, nxt)) prefetch_row(nxt.bh, nxt.q_first * 128 + r, nxt.h);
        }
        // Per-row constants.
        const float n = a.causal ? static_cast<float>(i + 1) : static_cast<float>(a.T);
        const float w_ln = logf(n) * 0.125f;             // ln(n_i)/sqrt(D)
        const float cn = a.ssmax ? s_h * w_ln : 0.125f;   // c_i
        const float cr = cn * 1.44269504088896341f;      // c_i log2(e)
        const size_t ridx = static_cast<size_t>(bh) * a.T + i;
        const float lse2 = row_ok ? lse_row * 1.44269504088896341f : INFINITY;
        const float delta = row_ok ? del_row : 0.0f;
        int lim = a.T - 1 - j0;              // last visible key column
        if (a.causal) lim = min(lim, i - j0);
        const uint64_t cr2 = f2_pack(cr, cr), cn2 = f2_pack(cn, cn);
        const uint64_t nlse2 = f2_pack(-lse2, -lse2), ndel2 = f2_pack(-delta, -delta);

        ok = warp_wait(&sm.s_full, g & 1, a.status, ab, kSiteBWgS);
        if (!ok) break;
        ok = warp_wait(&sm.qd_full[s], (g / kBStages) & 1, a.status, ab, kSiteBWgQD);
        if (!ok) break;
        tc_fence_after();
        // Key c of row r reads window entry 128 + r - c, i.e. reversed entry
        // 127 - r + c; in copy kq the entries of c, c+1, c+2, c+3 (c % 4 == 0)
        // form one aligned 16-byte vector.
        const float* wv = sm.win[s][0] + wrev;
        // Row partial sums for the Delta correction and the SSMax sum.
        uint64_t pB2 = 0ull, pBeta2 = 0ull, pMu2 = 0ull, pS2 = 0ull, pDP2 = 0ull, rowSS2 = 0ull;
        // P and c*dS of keys [c0, c0+8) of query row r into the MN-major
        // operands (one 16-byte chunk each).
        auto store_chunk = [&](int c0, const uint32_t* pp, const uint32_t* dd) {
          const uint32_t off = mn_chunk_offset(c0 / 8, r);
          *reinterpret_cast<uint4*>(sm.pt + off) = make_uint4(pp[0], pp[1], pp[2], pp[3]);
          *reinterpret_cast<uint4*>(sm.dst + off) = make_uint4(dd[0], dd[1], dd[2], dd[3]);
        };
        // 16-key chunks of S and dP per thread (eight independent column
        // pairs per chunk: measured 5% faster than 8-key chunks with the next
        // chunk's columns prefetched).
        uint32_t pp_prev[8], dd_prev[8];  // chunk computed, not yet stored
        constexpr int kCW = 16;
        constexpr int kNC = kBKeysPerWarp / kCW;
#pragma unroll 1
        for (int ch = 0; ch < kNC; ++ch) {
          const int c0 = kBKeysPerWarp * hc + kCW * ch;
          uint32_t sv[16], dpv[16];
          tmem_ld_32x32b_x16(tm + lb + kColS + c0, sv);
          tmem_ld_32x32b_x16(tm + lb + kColDP + c0, dpv);
          uint64_t tb[8], tbeta[8], tmu[8];
          const float* wp = wv + c0;
#pragma unroll
          for (int q = 0; q < 4; ++q) ld_f2x2(wp + 4 * q, tb[2 * q], tb[2 * q + 1]);
          tmem_ld_wait();
          reg_fence16(sv);
          reg_fence16(dpv);
          if (ch == kNC - 1) {
            // This warp's last S/dP columns of the tile are in registers: the
            // next tile's S and dP may be written over them.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.sdp_free);
          }
          uint32_t pp[8], dd[8];
          // Masked keys (past the causal limit or T) only in chunks that reach
          // them; the test is warp-uniform so each warp takes one version.
          auto elementwise = [&](auto masked) {
            // Two passes: P, dS and the sums that need no derivative plane
            // from the bias plane alone, then the two derivative planes'
            // loads (so that a chunk's first arithmetic waits for a third of
            // its table loads) and their four sums.
            uint64_t p2v[8], ds2v[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const int c = c0 + 2 * x;
              const uint64_t s2 =
                  f2_pack(__uint_as_float(sv[2 * x]), __uint_as_float(sv[2 * x + 1]));
              const uint64_t dp2 =
                  f2_pack(__uint_as_float(dpv[2 * x]), __uint_as_float(dpv[2 * x + 1]));
              float z0, z1;
              f2_unpack(fadd2(ffma2(s2, cr2, tb[x]), nlse2), z0, z1);
              if constexpr (decltype(masked)::value) {
                if (c > lim) z0 = -INFINITY;
                if (c + 1 > lim) z1 = -INFINITY;
              }
              const float p0 = ex2_approx(z0), p1 = ex2_approx(z1);
              const uint64_t p2 = f2_pack(p0, p1);
              const uint64_t dS2 = fmul2(p2, fadd2(dp2, ndel2));
              p2v[x] = p2;
              ds2v[x] = dS2;
              accB2 = ffma2(dS2, tb[x], accB2);
              rowSS2 = ffma2(dS2, s2, rowSS2);
              pB2 = ffma2(p2, tb[x], pB2);
              pS2 = ffma2(p2, s2, pS2);
              pDP2 = ffma2(p2, dp2, pDP2);
              pp[x] = pack_bf16x2(p0, p1);
              float q0, q1;
              f2_unpack(fmul2(dS2, cn2), q0, q1);
              dd[x] = pack_bf16x2(q0, q1);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              ld_f2x2(wp + kBWinPlane + 4 * q, tbeta[2 * q], tbeta[2 * q + 1]);
              ld_f2x2(wp + 2 * kBWinPlane + 4 * q, tmu[2 * q], tmu[2 * q + 1]);
            }
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              accBeta2 = ffma2(ds2v[x], tbeta[x], accBeta2);
              accMu2 = ffma2(ds2v[x], tmu[x], accMu2);
              pBeta2 = ffma2(p2v[x], tbeta[x], pBeta2);
              pMu2 = ffma2(p2v[x], tmu[x], pMu2);
            }
          };
          if (__any_sync(0xffffffffu, c0 + kCW - 1 > lim))
            elementwise(std::true_type{});
          else
            elementwise(std::false_type{});
          if (ch == 1 && t > 0) {
            // The previous tile's gradient products must be done before its
            // P^T / dS^T buffers are overwritten; its dQ tile is drained
            // here, before this tile's dQ product is issued.  (The
            // previous item's last tile was drained at that item's end.)
            ok = warp_wait(&sm.mma_done, (g - 1) & 1, a.status, ab, kSiteBWgDone);
            if (!ok) break;
            tc_fence_after();
            if (!dq_epilogue()) {
              ok = false;
              break;
            }
          }
          if (ch == 1 && t == 0 && round > 0) {
            // The previous item's dK/dV staging in the P^T buffer is read.
            ok = warp_wait(&sm.epi_free, (round - 1) & 1, a.status, ab, kSiteBWgDq);
            if (!ok) break;
          }
          if (ch > 0) {
            store_chunk(c0 - kCW, pp_prev, dd_prev);
            store_chunk(c0 - kCW + 8, pp_prev + 4, dd_prev + 4);
          }
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            pp_prev[x] = pp[x];
            dd_prev[x] = dd[x];
          }
        }
        if (!ok) break;
        store_chunk(kBKeysPerWarp * hc + kBKeysPerWarp - 16, pp_prev, dd_prev);
        store_chunk(kBKeysPerWarp * hc + kBKeysPerWarp - 8, pp_prev + 4, dd_prev + 4);
        {
          float a0, a1;
          f2_unpack(rowSS2, a0, a1);
          acc_s = fmaf(a0 + a1, w_ln, acc_s);
        }
        if (row_ok) {
          float b0, b1, e0, e1, m0, m1, s0, s1, d0, d1;
          f2_unpack(pB2, b0, b1);
          f2_unpack(pBeta2, e0, e1);
          f2_unpack(pMu2, m0, m1);
          f2_unpack(pS2, s0, s1);
          f2_unpack(pDP2, d0, d1);
          float* ra = a.rowacc + ridx * 8;
          red_add_v4(ra, b0 + b1, e0 + e1, m0 + m1, (s0 + s1) * w_ln);
          atomicAdd(ra + 4, d0 + d1);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.ds_ready);
      }
      // Block reduction of the item's scalar-gradient sums, one atomic per
      // sum (while the item's last gradient products run).  Every
      // element-wise warp gets here once per item, also after giving up.
      float v4[4];
      {
        float a0, a1;
        f2_unpack(accB2, a0, a1);
        v4[0] = a0 + a1;
        f2_unpack(accBeta2, a0, a1);
        v4[1] = a0 + a1;
        f2_unpack(accMu2, a0, a1);
        v4[2] = a0 + a1;
        v4[3] = acc_s;
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v4[x] += __shfl_xor_sync(0xffffffffu, v4[x], off);
      if (lane == 0)
        for (int x = 0; x < 4; ++x) sm.red[round & 1][warp][x] = v4[x];
      const int all_ok = elementwise_barrier_and(ok ? 1 : 0);
      if (threadIdx.x < 4 && all_ok) {
        float tot = 0.f;
        for (int w = 0; w < kBCompute; ++w) tot += sm.red[round & 1][w][threadIdx.x];
        add_head_grad(a, threadIdx.x, it.h, tot);
      }
      ok = all_ok;
      if (ok) {
        // The item's last gradient products, then its dQ tile and the dK/dV
        // rows (TMEM lane = key j0 + r; this warp writes 16 of the 64
        // dimensions).  The next item's first dK/dV product comes after this
        // warp's next ds_ready arrival, so these TMEM reads are done by then.
        ok = warp_wait(&sm.mma_done, (g - 1) & 1, a.status, ab, kSiteBWgDone);
        if (ok) {
          tc_fence_after();
          ok = dq_epilogue();
        }
        if (ok) {
          // dK and dV rows as bf16 into the P^T buffer (free once the item's
          // last products are done), 128-byte rows with the 128-byte swizzle,
          // for the dQ warp's TMA stores: TMEM lane = key j0 + r; this warp
          // holds kBDims of the 64 dimensions (16-byte chunks of 8 columns).
          for (int which = 0; which < 2; ++which) {
            const uint32_t col = (which ? kColDV : kColDK) + kBDims * hc;
            uint32_t kvv[kBDims];
#pragma unroll
            for (int u = 0; u < kBDims / 16; ++u) tmem_ld_32x32b_x16(tm + lb + col + 16 * u, kvv + 16 * u);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < kBDims / 16; ++u) reg_fence16(kvv + 16 * u);
            uint8_t* rowp = sm.pt + which * kTile + r * 128;
#pragma unroll
            for (int x = 0; x < kBDims / 8; ++x) {
              const int cc = (kBDims / 8) * hc + x;
              *reinterpret_cast<uint4*>(rowp + ((cc ^ (r & 7)) << 4)) = make_uint4(
                  pack_bf16x2(__uint_as_float(kvv[8 * x]), __uint_as_float(kvv[8 * x + 1])),
                  pack_bf16x2(__uint_as_float(kvv[8 * x + 2]), __uint_as_float(kvv[8 * x + 3])),
                  pack_bf16x2(__uint_as_float(kvv[8 * x + 4]), __uint_as_float(kvv[8 * x + 5])),
                  pack_bf16x2(__uint_as_float(kvv[8 * x + 6]), __uint_as_float(kvv[8 * x + 7])));
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.epi_full);
        }
      }
      have = bwd_item(a, sc, round + 1, it);
    }
  }

  tc_fence_before();
  __syncthreads();
  grid_dep_trigger();
  if (warp == kBMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

// The three distance tables (first `table_blocks` blocks); Delta_i = dO_i .
// O_i; zero the dq accumulator, the row sums and the per-head gradient
// outputs (which the later kernels add into).
__global__ void __launch_bounds__(256) bam_bwd_prep_kernel(const BwdArgs a, int table_blocks) {
  grid_dep_trigger();
  if (static_cast<int>(blockIdx.x) < table_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_begin_call(a.status);  // the call starts here
    const size_t n = static_cast<size_t>(a.tab.H) * a.tab.len;
    for (size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
         e += static_cast<size_t>(table_blocks) * blockDim.x)
      table_entry(a.tab, static_cast<int>(e / a.tab.len), static_cast<int>(e % a.tab.len));
    return;
  }
  const size_t rows = static_cast<size_t>(a.B) * a.H * a.T;
  const size_t tid = static_cast<size_t>(blockIdx.x - table_blocks) * blockDim.x + threadIdx.x;
  const size_t nthreads = static_cast<size_t>(gridDim.x - table_blocks) * blockDim.x;
  grid_dep_wait();  // O comes from the forward
  // Delta: eight threads per row, eight elements each, shuffle reduction.
  // The loop bound is warp-uniform so that every lane reaches the shuffles.
  const int sub = threadIdx.x & 7;
  for (size_t wb = tid & ~static_cast<size_t>(31); wb < rows * 8; wb += nthreads) {
    const size_t row = (wb + (threadIdx.x & 31)) / 8;
    float acc = 0.f;
    if (row < rows) {
      const uint4 w = reinterpret_cast<const uint4*>(a.dO + row * kHeadDim)[sub];
      float o[8];
      if (a.o_fp32) {
        const float4* op = reinterpret_cast<const float4*>(static_cast<const float*>(a.o) +
                                                           row * kHeadDim) + 2 * sub;
        const float4 o0 = op[0], o1 = op[1];
        o[0] = o0.x; o[1] = o0.y; o[2] = o0.z; o[3] = o0.w;
        o[4] = o1.x; o[5] = o1.y; o[6] = o1.z; o[7] = o1.w;
      } else {
        const uint4 u = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.o) +
                                                       row * kHeadDim)[sub];
        o[0] = __uint_as_float(u.x << 16); o[1] = __uint_as_float(u.x & 0xFFFF0000u);
        o[2] = __uint_as_float(u.y << 16); o[3] = __uint_as_float(u.y & 0xFFFF0000u);
        o[4] = __uint_as_float(u.z << 16); o[5] = __uint_as_float(u.z & 0xFFFF0000u);
        o[6] = __uint_as_float(u.w << 16); o[7] = __uint_as_float(u.w & 0xFFFF0000u);
      }
      acc = __uint_as_float(w.x << 16) * o[0] + __uint_as_float(w.x & 0xFFFF0000u) * o[1] +
            __uint_as_float(w.y << 16) * o[2] + __uint_as_float(w.y & 0xFFFF0000u) * o[3] +
            __uint_as_float(w.z << 16) * o[4] + __uint_as_float(w.z & 0xFFFF0000u) * o[5] +
            __uint_as_float(w.w << 16) * o[6] + __uint_as_float(w.w & 0xFFFF0000u) * o[7];
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (sub == 0 && row < rows) a.delta[row] = acc;
  }
  float4* dq4 = reinterpret_cast<float4*>(a.dq_acc);
  const size_t n4 = rows * (kHeadDim / 4);
  for (size_t x = tid; x < n4; x += nthreads) dq4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
  float4* ra4 = reinterpret_cast<float4*>(a.rowacc);
  for (size_t x = tid; x < rows * 2; x += nthreads) ra4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (size_t x = tid; x < static_cast<size_t>(a.H); x += nthreads) {
    a.dalpha[x] = 0.f;
    a.dbeta[x] = 0.f;
    a.dmu[x] = 0.f;
    a.ds[x] = 0.f;
  }
}

// dq (bf16) from the fp32 accumulator; the Delta correction of the scalar
// sums (row blocks of one (b, h) per CTA), added straight into the per-head
// gradient outputs.
constexpr int kFinalRows = 256;  // = the block size: one row per thread

__global__ void __launch_bounds__(256) bam_bwd_final_kernel(const BwdArgs a) {
  grid_dep_wait();  // dq accumulator, row sums and scalar sums of the fused kernel
  const size_t n8 = static_cast<size_t>(a.B) * a.H * a.T * (kHeadDim / 8);
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  if (*reinterpret_cast<volatile int*>(&a.status->abort)) return;
  // Row blocks of kFinalRows rows (one per thread) for the Delta correction;
  // the inputs of this CTA's first block are loaded before the dq
  // conversion, so that their latency overlaps it.
  const int chunks = (a.T + kFinalRows - 1) / kFinalRows;
  const int items = a.B * a.H * chunks;
  float4 bsum = make_float4(0.f, 0.f, 0.f, 0.f);
  float dd = 0.f;
  auto load_rows = [&](int item) {
    const int i = (item % chunks) * kFinalRows + threadIdx.x;
    bsum = make_float4(0.f, 0.f, 0.f, 0.f);
    dd = 0.f;
    if (i < a.T) {
      const size_t row = static_cast<size_t>(item / chunks) * a.T + i;
      bsum = reinterpret_cast<const float4*>(a.rowacc + row * 8)[0];
      dd = a.delta[row] - a.rowacc[row * 8 + 4];
    }
  };
  if (static_cast<int>(blockIdx.x) < items) load_rows(blockIdx.x);
  const float4* src = reinterpret_cast<const float4*>(a.dq_acc);
  uint4* dst = reinterpret_cast<uint4*>(a.dq);
  // Four groups of eight values per thread and pass, all loads issued first.
  for (size_t x0 = tid; x0 < n8; x0 += 4 * nthreads) {
    float4 u[4], w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const size_t x = x0 + k * nthreads;
      if (x < n8) {
        u[k] = __ldcs(src + 2 * x);
        w[k] = __ldcs(src + 2 * x + 1);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const size_t x = x0 + k * nthreads;
      if (x < n8)
        dst[x] = make_uint4(pack_bf16x2(u[k].x, u[k].y), pack_bf16x2(u[k].z, u[k].w),
                            pack_bf16x2(w[k].x, w[k].y), pack_bf16x2(w[k].z, w[k].w));
    }
  }
  // Correction sum_i (Delta_i - C_i) B_i per row block, one atomic per sum.
  __shared__ float red[8][4];
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    if (item != static_cast<int>(blockIdx.x)) load_rows(item);
    float c4[4] = {dd * bsum.x, dd * bsum.y, dd * bsum.z, dd * bsum.w};
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) c4[x] += __shfl_xor_sync(0xffffffffu, c4[x], off);
    if ((threadIdx.x & 31) == 0)
      for (int x = 0; x < 4; ++x) red[threadIdx.x >> 5][x] = c4[x];
    __syncthreads();
    if (threadIdx.x < 4) {
      float tot = 0.f;
      for (int w2 = 0; w2 < 8; ++w2) tot += red[w2][threadIdx.x];
      add_head_grad(a, threadIdx.x, (item / chunks) % a.H, tot);
    }
    __syncthreads();
  }
}

// Host: per-CTA item lists for the causal backward.  Item costs in units of
// ~0.3 us: 11 per query tile, 8 per item boundary (~3.3 and ~2.4 us measured
// on the B=8 H=12 T=512 training workload).  First-fit decreasing packs the
// items, longest first, each into the first CTA where it fits under a
// makespan bound, and bisection finds the smallest bound that packs.  A local
// search then empties the makespan level CTA by CTA (moving one item, or
// swapping one item for one or two, between a CTA at the makespan and one
// below it, neither ending at or above it), which spreads the long CTAs: on
// the training workload first-fit leaves 96 CTAs with 4+3 query tiles and the
// search halves that (48 x 4+3, 48 x 4+1+1, 24 x 3+3, 32 x 2+2+2), which ran
// 1.5 us faster.  The lists are used when their makespan beats that of the
// round-robin snake (n = 0 otherwise).
constexpr long kTileCost = 11, kBoundaryCost = 8;

long list_cost(long tiles, size_t items) {
  return tiles * kTileCost + (items > 0 ? static_cast<long>(items - 1) * kBoundaryCost : 0);
}

long snake_makespan(int BH, int nkb, int G) {
  std::vector<long> tiles(G, 0);
  std::vector<size_t> items(G, 0);
  const int total = BH * nkb;
  for (int r = 0; r * G < total; ++r)
    for (int c = 0; c < G; ++c) {
      const int idx = r * G + ((r & 1) ? (G - 1 - c) : c);
      if (idx >= total) continue;
      tiles[c] += nkb - idx / BH;
      ++items[c];
    }
  long m = 0;
  for (int c = 0; c < G; ++c) m = std::max(m, list_cost(tiles[c], items[c]));
  return m;
}

// First-fit decreasing under makespan bound M: the sizes (query tiles) of the
// items each CTA runs.
bool pack_sizes(int BH, int nkb, int G, long M, std::vector<std::vector<int>>& per) {
  per.assign(G, {});
  std::vector<long> load(G, 0);
  for (int kb = 0; kb < nkb; ++kb) {
    const int size = nkb - kb;
    for (int bh = 0; bh < BH; ++bh) {
      int c = 0;
      for (; c < G; ++c) {
        const long add = size * kTileCost + (per[c].empty() ? 0 : kBoundaryCost);
        if (load[c] + add <= M) {
          load[c] += add;
          per[c].push_back(size);
          break;
        }
      }
      if (c == G) return false;
    }
  }
  return true;
}

// The local search described above, with at most `budget` candidate
// evaluations.  Each accepted change lowers the number of CTAs at the
// makespan, so the search ends.
void spread_makespan(std::vector<std::vector<int>>& per, long budget) {
  const int G = static_cast<int>(per.size());
  std::vector<long> tiles(G, 0);
  for (int c = 0; c < G; ++c)
    for (int x : per[c]) tiles[c] += x;
  while (budget > 0) {
    long m = 0;
    for (int c = 0; c < G; ++c) m = std::max(m, list_cost(tiles[c], per[c].size()));
    bool changed = false;
    for (int a = 0; a < G && !changed && budget > 0; ++a) {
      const size_t na = per[a].size();
      if (list_cost(tiles[a], na) != m) continue;
      long best = LONG_MAX;
      int kind = -1, bb = -1;
      size_t bi = 0, bj = 0, bk = 0;
      for (int b = 0; b < G; ++b) {
        if (b == a) continue;
        const size_t nb = per[b].size();
        const long lb = list_cost(tiles[b], nb);
        if (lb >= m) continue;
        const long base = m * m + lb * lb;
        auto consider = [&](long ca, long cb, int k, size_t i, size_t j, size_t l) {
          if (ca >= m || cb >= m) return;
          const long d = ca * ca + cb * cb - base;
          if (d < best) {
            best = d;
            kind = k;
            bb = b;
            bi = i;
            bj = j;
            bk = l;
          }
        };
        for (size_t i = 0; i < na; ++i) {
          const int si = per[a][i];
          consider(list_cost(tiles[a] - si, na - 1), list_cost(tiles[b] + si, nb + 1), 0, i, 0, 0);
          for (size_t j = 0; j < nb; ++j) {
            const int sj = per[b][j];
            if (sj != si)
              consider(list_cost(tiles[a] - si + sj, na), list_cost(tiles[b] - sj + si, nb), 1, i,
                       j, 0);
            if (nb > 12) continue;
            for (size_t l = j + 1; l < nb; ++l) {
              const int sl = per[b][l];
              consider(list_cost(tiles[a] - si + sj + sl, na + 1),
                       list_cost(tiles[b] - sj - sl + si, nb - 1), 2, i, j, l);
            }
          }
          budget -= static_cast<long>(nb * nb / 2 + nb + 1);
        }
      }
      if (kind < 0) continue;
      std::vector<int>& A = per[a];
      std::vector<int>& Bv = per[bb];
      const int si = A[bi];
      if (kind == 0) {
        A.erase(A.begin() + bi);
        Bv.push_back(si);
        tiles[a] -= si;
        tiles[bb] += si;
      } else if (kind == 1) {
        const int sj = Bv[bj];
        A[bi] = sj;
        Bv[bj] = si;
        tiles[a] += sj - si;
        tiles[bb] += si - sj;
      } else {
        const int sj = Bv[bj], sl = Bv[bk];
        A[bi] = sj;
        A.push_back(sl);
        Bv.erase(Bv.begin() + bk);  // bk > bj: erase the later one first
        Bv.erase(Bv.begin() + bj);
        Bv.push_back(si);
        tiles[a] += sj + sl - si;
        tiles[bb] += si - sj - sl;
      }
      changed = true;
    }
    if (!changed) return;
  }
}

bool build_schedule(int BH, int nkb, int G, BwdSched& sc) {
  const int total = BH * nkb;
  sc.n = 0;
  if (total > kSchedMaxItems || G > kSchedMaxCtas || G < 1 || total < G) return false;
  long sum = 0;
  for (int kb = 0; kb < nkb; ++kb) sum += static_cast<long>(nkb - kb) * BH * kTileCost;
  sum += static_cast<long>(total - G) * kBoundaryCost;
  long lo = std::max((sum + G - 1) / G, static_cast<long>(nkb) * kTileCost);
  long hi = snake_makespan(BH, nkb, G) - 1;  // only a strictly better bound is of use
  std::vector<std::vector<int>> per, best;
  while (lo <= hi) {
    const long mid = lo + (hi - lo) / 2;
    if (pack_sizes(BH, nkb, G, mid, per)) {
      best = per;
      hi = mid - 1;
    } else {
      lo = mid + 1;
    }
  }
  if (best.empty()) return false;
  spread_makespan(best, 50000000L);
  // Concrete items: within a size class, heads in CTA order; each CTA's items
  // longest first.
  std::vector<int> next_bh(nkb + 1, 0);
  int n = 0;
  for (int c = 0; c < G; ++c) {
    std::sort(best[c].begin(), best[c].end(), [](int x, int y) { return x > y; });
    sc.start[c] = static_cast<uint16_t>(n);
    for (int size : best[c]) sc.item[n++] = static_cast<uint16_t>((nkb - size) * BH + next_bh[size]++);
  }
  sc.start[G] = static_cast<uint16_t>(n);
  sc.n = n;
  return n == total;
}

// The schedule for this shape into `out` (n = 0: none).  Schedules of recent
// shapes are kept, so the host cost is paid once per shape.
void schedule_for(int BH, int nkb, int causal, int G, BwdSched& out) {
  struct Entry {
    int BH, nkb, G;
    BwdSched sc;
  };
  out.n = 0;
  if (!causal) return;
  static std::mutex mu;
  static std::vector<Entry> cache;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.BH == BH && e.nkb == nkb && e.G == G) {
      out = e.sc;
      return;
    }
  if (cache.size() >= 8) cache.erase(cache.begin());
  cache.push_back(Entry{BH, nkb, G, {}});
  build_schedule(BH, nkb, G, cache.back().sc);
  out = cache.back().sc;
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t st) {
  const size_t rows = static_cast<size_t>(a.B) * a.H * a.T;
  size_t want = (rows * 8 + 255) / 256;
  if (want < 1) want = 1;
  if (want > 152 * 7) want = 152 * 7;
  const size_t tab_entries = static_cast<size_t>(a.tab.H) * a.tab.len;
  size_t tb = (tab_entries + 255) / 256;
  if (tb > 152 * 2) tb = 152 * 2;
  const unsigned grid = static_cast<unsigned>(want + tb);
  return launch_k(bam_bwd_prep_kernel, dim3(grid), dim3(256), 0, st, false, a,
                  static_cast<int>(tb));
}

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(BwdSmem) + 1024;
  static bool limit_set[64] = {};
  cudaError_t e = smem_limit_once(bam_bwd_kernel, smem, limit_set);
  if (e != cudaSuccess) return e;
  // Persistent: one CTA per SM (at most one per work item).
  const int num_sms = sm_count();
  if (num_sms <= 0) return cudaErrorInvalidDevice;
  const long items = static_cast<long>(a.nkb) * a.B * a.H;
  const unsigned grid = static_cast<unsigned>(items < num_sms ? items : num_sms);
  BwdSched sc;
  schedule_for(a.B * a.H, a.nkb, a.causal, static_cast<int>(grid), sc);
  return launch_k(bam_bwd_kernel, dim3(grid), dim3(kBThreads), smem, st, true, tq, tk, tv, tdo,
                  tdq, tdk, tdv, a, sc);
}

cudaError_t launch_bwd_final(const BwdArgs& a, cudaStream_t st) {
  const size_t n8 = static_cast<size_t>(a.B) * a.H * a.T * (kHeadDim / 8);
  const size_t items = static_cast<size_t>(a.B) * a.H * ((a.T + kFinalRows - 1) / kFinalRows);
  // Enough threads that each converts about four groups; up to eight
  // 256-thread CTAs per SM.
  size_t want = (n8 + 1023) / 1024;
  if (want < items) want = items;
  if (want > 152 * 8) want = 152 * 8;
  const unsigned grid = static_cast<unsigned>(want);
  return launch_k(bam_bwd_final_kernel, dim3(grid), dim3(256), 0, st, true, a);
}

}  // namespace bam

extern "C" int bam_attn_bwd_schedule(int B, int H, int T, int causal, int grid, int* start,
                                     int* item, int max_items) {
  if (B < 1 || H < 1 || T < 1 || grid < 1 || !start || !item || max_items < 0) return -1;
  const int nkb = (T + 127) / 128;
  const long items = static_cast<long>(nkb) * B * H;
  if (items > 0x7fffffffL / 2) return -1;
  const int G = static_cast<int>(items < grid ? items : grid);
  bam::BwdSched sc;
  bam::schedule_for(B * H, nkb, causal, G, sc);
  if (sc.n == 0) return 0;
  if (sc.n > max_items) return -1;
  for (int c = 0; c <= G; ++c) start[c] = sc.start[c];
  for (int w = 0; w < sc.n; ++w) item[w] = sc.item[w];
  return sc.n;
}
