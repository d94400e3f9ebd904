// Fused GGD-BAM attention forward for sm_103a (tcgen05 / TMEM / TMA).
//
// Computes, per (b, h) and query row i,
//   z_ij = c_i * q_i . k_j + b_h(i - j),   O_i = softmax_j(z_ij) V,
//   LSE_i = log sum_j exp(z_ij),
// with c_i = 1/sqrt(D) or, with Scalable-Softmax, s_h ln(n_i)/sqrt(D)
// ("Bayesian Attention Mechanism" summary, "Solution Proposee : GGD-BAM" for
// the bias and SSMax; "ALiBi: Attention with Linear Biases", "Code" for
// scores -> softmax -> weights @ V).  The bias comes from the per-head
// distance table (table.cu), staged per key tile into shared memory by a
// bulk copy, so no power function runs per element.
//
// Long sequences (bam_fwd_kernel): one CTA owns 256 query rows of one (b, h)
// as two 128-row tiles A and B, and both walk every key/value tile of 128
// keys that they see, so each K/V tile loaded serves 256 rows.  Short
// sequences use a persistent single-tile form of the same pipeline, two
// CTAs per SM (bam_fwd_single_kernel, below).
// Warp roles:
//   warp 8      TMA producer: Q; per key tile K, V and the 384-entry
//               distance window (four shifted reversed copies, so that a
//               thread reads four keys' biases with one 16-byte load), into
//               a 3-stage ring.
//   warp 9      MMA issuer (one thread): S_t = Q K^T (128x128x64, both
//               operands K-major in shared memory) and O_t += P_t V (P from
//               Tensor Memory, V MN-major), accumulators in Tensor Memory.
//               Also allocates / frees the 512 TMEM columns.
//   warps 0-3   softmax group A, warps 4-7 softmax group B: one thread
//               per query row reads its S row from TMEM, adds c_i S + bias in
//               log2 units, runs the online softmax (exp2, rescaling O in
//               TMEM only when the running max grows by more than 8), writes
//               P (bf16) back to TMEM, and in the end normalises O.
// The two softmax groups are offset by one MMA so the tensor core works on
// one group's tile while the other is in its softmax.
//
// TMEM columns: S_A [0,128) S_B [128,256) P_A [256,320) P_B [320,384)
//               O_A [384,448) O_B [448,512)  (A, B: the two softmax groups).
#include "bam_common.cuh"

namespace bam {
namespace {

constexpr int kStages = 3;
constexpr int kThreads = 320;  // 10 warps: 168 registers per thread at most
constexpr int kTileBytes = 128 * 64 * 2;
constexpr int kWin = 384;          // window entries per key tile (two query tiles)
constexpr int kWinCopy = kWin + 4;  // entries per reversed copy (shifts of 0..3)
constexpr int kWinCopyStride = 416;
constexpr int kWinStage = kTabCopies * kWinCopyStride;
static_assert(win_copy_off(kTabCopies - 1, kWinCopyStride) + kWinCopy <= kWinStage, "window");
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct __align__(1024) FwdSmem {
  uint8_t q[2][kTileBytes];
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  // Normalised O of each query tile for its TMA store: fp32 as two
  // 128-byte-swizzled boxes of 32 columns, or bf16 as one of 64 columns.
  uint8_t ost[2][2 * kTileBytes];
  float win[kStages][kWinStage];
  uint64_t q_full[2];
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t o_full[2];      // the tile's four softmax warps have staged their O rows
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort_flag;
};

// Sites recorded in the status word when a wait gives up.
enum : int {
  kSiteProducer = 10,
  kSiteMmaQ = 20,
  kSiteMmaK = 21,
  kSiteMmaV = 22,
  kSiteMmaSFree = 23,
  kSiteMmaP = 24,
  kSiteSoftS = 30,
  kSiteSoftK = 31,
  kSiteSoftPV = 32,
  kSiteSoftEnd = 33,
  kSiteSoftStore = 34,
  // Debug-build bounds checks (BAM_DEV_BOUNDS)
  kSiteWindowCopy = 35,
  kSiteOutRow = 36
};

// All lanes wait; the result is made warp-uniform so that the collective
// tcgen05.ld/st that follow are executed by the whole warp or by none of it.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, DevStatus* st,
                                          volatile int* ab, int site) {
  const bool ok = mbar_wait(bar, parity, st, ab, site);
  return __all_sync(0xffffffffu, ok);
}

// Initialises the barriers and allocates Tensor Memory (whole CTA).
__device__ __forceinline__ uint32_t fwd_setup(FwdSmem& sm, int warp) {
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    for (int b = 0; b < 2; ++b) mbar_init(&sm.q_full[b], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.s_free[t], 4);
      mbar_init(&sm.p_full[t], 4);
      mbar_init(&sm.pv_done[t], 1);
      mbar_init(&sm.o_full[t], 4);
    }
    mbar_init(&sm.mma_final, 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return sm.tmem_base;
}

// Issues the K, window and V copies of key tile j of head bh (query rows
// from i0) into stage s, armed on k_full[s] and v_full[s].  `first` marks
// the CTA's first tile: the windows come from the table kernel, which the
// producer waits for there.  Windows hold W entries (384 for 256 query rows,
// 256 for 128), each reversed copy W + 4, copies WS floats apart.  Returns
// false when a debug bounds check refused a window copy.
template <int W = kWin, int WS = kWinCopyStride, class Sm>
__device__ __forceinline__ bool load_kv_tile(Sm& sm, const FwdArgs& a,
                                             const CUtensorMap* tk, const CUtensorMap* tv,
                                             int s, int j, int bh, int h, int i0, bool first,
                                             volatile int* ab, bool k_before_v = false) {
  // The window of key tile j covers table indices tab_off + i0 - 128 -
  // 128 j + [0, W); in the reversed rows it starts at tab_len - W minus
  // that base (a multiple of 4 entries).  A window starts inside its own row
  // and may run past the row's end into the padding after the last row,
  // never beyond it.
  const size_t copy_stride = static_cast<size_t>(a.H) * a.tab_len;
  const float* tab_h = a.table + static_cast<size_t>(h) * a.tab_len +
                       (a.tab_len - W - a.tab_off - i0 + 128);
  const float* tab_end = a.table + kTabCopies * copy_stride + kTabPadFloats;
  mbar_arrive_expect_tx(&sm.k_full[s], kTileBytes + kTabCopies * (W + 4) * 4);
  tma_load_3d(sm.k[s], tk, &sm.k_full[s], 0, 128 * j, bh);
  if (first) grid_dep_wait();
  bool ok = true;
  for (int k = 0; k < kTabCopies; ++k)
    ok &= bulk_load_checked(sm.win[s] + win_copy_off(k, WS),
                            tab_h + k * copy_stride + 128 * j, (W + 4) * 4, &sm.k_full[s],
                            a.table + k * copy_stride + static_cast<size_t>(h) * a.tab_len,
                            tab_end, a.status, ab, kSiteWindowCopy);
  // The CTA's first K tile lands before its V and the next stage are
  // requested, so that the first S product waits for Q and K only.
  if (ok && k_before_v) ok = mbar_wait(&sm.k_full[s], 0, a.status, ab, kSiteProducer);
  mbar_arrive_expect_tx(&sm.v_full[s], kTileBytes);
  tma_load_3d(sm.v[s], tv, &sm.v_full[s], 0, 128 * j, bh);
  return ok;
}

// S (TMEM columns at tS) = Q K^T from query buffer qb and the K tile in
// stage s; completion on `bar`.
template <class Sm>
__device__ __forceinline__ void issue_S(Sm& sm, uint32_t tS, int qb, int s, uint64_t* bar) {
  constexpr uint64_t kTileDesc = kTileBytes >> 4;  // descriptor units of 16 bytes
  const uint32_t idS = idesc_bf16(128, 128, false, false);
  const uint64_t qd = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024) + kTileDesc * qb;
  const uint64_t kd = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024) + kTileDesc * s;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    umma_ss(tS, qd + 2 * kk, kd + 2 * kk, idS, kk > 0 ? 1u : 0u);
  umma_commit(bar);
}

// O (TMEM columns at tO) (+)= P (at tP) V with the V tile in stage s
// (`first`: overwrite O); completion on `bar`.
template <class Sm>
__device__ __forceinline__ void issue_PV(Sm& sm, uint32_t tO, uint32_t tP, int s, bool first,
                                         uint64_t* bar) {
  constexpr uint64_t kTileDesc = kTileBytes >> 4;
  const uint32_t idO = idesc_bf16(128, 64, false, true);
  const uint64_t vd = sdesc_sw128(smem_u32(sm.v[0]), 16384, 1024) + kTileDesc * s;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_ts(tO, tP + 8 * kk, vd + 128 * kk, idO, (!first || kk > 0) ? 1u : 0u);
  umma_commit(bar);
}

// Running state of the online softmax of one query row.
struct SoftRow {
  float m, l, le;  // max (log2 units), sum of bf16-rounded weights, exact sum
};

// Barrier phases of one key tile of one softmax group.
struct TilePhases {
  uint32_t s;       // s_full phase of this group's tile
  uint32_t k;       // k_full phase of the tile's stage
  bool wait_pv;     // a previous PV of this group may still read P
  uint32_t pv;      // its pv_done phase
};

// One key tile of one softmax group; the thread owns one query row (its
// TMEM lane).  S row -> z = c_i S + bias (log2 units) -> mask -> running max
// (lazy rescale) -> P as bf16 to TMEM and the two row sums; O rescaled in
// TMEM when the max grew and `o_valid`.  Arrives on s_free once S is in
// registers and on p_full once P is written.  `lim`: last visible key column
// of the row within the tile (masking only when `masked`).  Returns false
// when a wait gave up.
template <class Sm>
__device__ __forceinline__ bool softmax_tile(Sm& sm, SoftRow& row, int t, int s,
                                             const TilePhases& ph, const float* wv, float cr,
                                             bool masked, int lim, bool o_valid, uint32_t tS,
                                             uint32_t tP, uint32_t tO, DevStatus* st,
                                             volatile int* ab, int lane) {
  if (!warp_wait(&sm.s_full[t], ph.s, st, ab, kSiteSoftS)) return false;
  if (!warp_wait(&sm.k_full[s], ph.k, st, ab, kSiteSoftK)) return false;
  tc_fence_after();
  // The S row comes from TMEM in two 64-column halves: the second half's
  // loads are in flight while the first half is turned into z = c_i S + bias
  // (column pairs as f32x2), so a tile waits on TMEM twice.
  const uint64_t cr2 = f2_pack(cr, cr);
  uint64_t z[64];
  uint32_t sv[128];
  tmem_ld_32x32b_x32(tS, sv);
  tmem_ld_32x32b_x32(tS + 32, sv + 32);
  tmem_ld_wait();
  reg_fence32(sv);
  reg_fence32(sv + 32);
  tmem_ld_32x32b_x32(tS + 64, sv + 64);
  tmem_ld_32x32b_x32(tS + 96, sv + 96);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    if (hf == 1) {
      tmem_ld_wait();
      reg_fence32(sv + 64);
      reg_fence32(sv + 96);
    }
#pragma unroll
    for (int x = 32 * hf; x < 32 * hf + 32; x += 2) {
      uint64_t t0, t1;
      ld_f2x2(wv + 2 * x, t0, t1);
      z[x] = ffma2(f2_pack(__uint_as_float(sv[2 * x]), __uint_as_float(sv[2 * x + 1])), cr2, t0);
      z[x + 1] = ffma2(f2_pack(__uint_as_float(sv[2 * x + 2]), __uint_as_float(sv[2 * x + 3])),
                       cr2, t1);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&sm.s_free[t]);

  if (masked) {
#pragma unroll
    for (int x = 0; x < 64; ++x) {
      float lo, hi;
      f2_unpack(z[x], lo, hi);
      if (2 * x > lim) lo = -INFINITY;
      if (2 * x + 1 > lim) hi = -INFINITY;
      z[x] = f2_pack(lo, hi);
    }
  }
  // Row max: four independent chains of 3-input max.
  float mq[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    float lo, hi;
    f2_unpack(z[x], lo, hi);
    mq[x] = fmaxf(lo, hi);
  }
#pragma unroll
  for (int x = 4; x < 64; ++x) {
    float lo, hi;
    f2_unpack(z[x], lo, hi);
    mq[x & 3] = fmax3(mq[x & 3], lo, hi);
  }
  const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
  const float m_new = fmaxf(row.m, mx);
  const bool resc = m_new > row.m + kRescaleThreshold;
  float scale = 1.0f;
  if (resc) {
    scale = ex2_approx(row.m - m_new);
    row.l *= scale;
    row.le *= scale;
    row.m = m_new;
  }
  if (ph.wait_pv) {
    // PV of this group's previous tile must be done: frees P, makes O stable.
    if (!warp_wait(&sm.pv_done[t], ph.pv, st, ab, kSiteSoftPV)) return false;
    tc_fence_after();
  }
  // Probabilities as bf16 pairs for the PV product, streamed to TMEM 16
  // columns at a time, and the two row sums (rounded weights for O,
  // unrounded for the LSE) in independent partial sums.
  const uint64_t negm2 = f2_pack(-row.m, -row.m);
  float lr[4] = {0.f, 0.f, 0.f, 0.f};
  uint64_t le2[2] = {0ull, 0ull};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pk[16];
#pragma unroll
    for (int y = 0; y < 16; ++y) {
      const int x = 16 * q + y;
      float a0, a1;
      f2_unpack(fadd2(z[x], negm2), a0, a1);
      const float p0 = ex2_approx(a0);
      const float p1 = ex2_approx(a1);
      const uint32_t w = pack_bf16x2(p0, p1);
      pk[y] = w;
      add_bf16x2_f32(w, lr[2 * (y & 1)], lr[2 * (y & 1) + 1]);
      le2[y & 1] = fadd2(le2[y & 1], f2_pack(p0, p1));
    }
    tmem_st_32x32b_x16(tP + 16 * q, pk);
  }
  {
    float b0, b1;
    f2_unpack(fadd2(le2[0], le2[1]), b0, b1);
    row.l += (lr[0] + lr[1]) + (lr[2] + lr[3]);
    row.le += b0 + b1;
  }
  if (o_valid && __any_sync(0xffffffffu, resc)) {
    uint32_t ov[64];
    tmem_ld_32x32b_x32(tO, ov);
    tmem_ld_32x32b_x32(tO + 32, ov + 32);
    tmem_ld_wait();
    reg_fence32(ov);
    reg_fence32(ov + 32);
#pragma unroll
    for (int x = 0; x < 64; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * scale);
    tmem_st_32x32b_x32(tO, ov);
    tmem_st_32x32b_x32(tO + 32, ov + 32);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&sm.p_full[t]);
  return true;
}

// Columns [32 hb, 32 hb + 32) of row r of a finished tile (32 fp32 values
// in ov), normalised, into the staging tile `ost` for its TMA store:
// 128-byte rows with 16-byte chunk c at (c ^ (r % 8)) * 16; fp32 as two boxes
// of 32 columns (box hb at hb * box_stride), bf16 as one box of 64 (chunks
// 4 hb .. 4 hb + 3).
__device__ __forceinline__ void stage_half(const FwdArgs& a, uint8_t* ost, const uint32_t* ov,
                                           int hb, float inv_l, int r,
                                           int box_stride = kTileBytes) {
  if (a.o_fp32) {
    uint8_t* rowp = ost + hb * box_stride + r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t* v4 = ov + 4 * c;
      *reinterpret_cast<float4*>(rowp + ((c ^ (r & 7)) << 4)) =
          make_float4(__uint_as_float(v4[0]) * inv_l, __uint_as_float(v4[1]) * inv_l,
                      __uint_as_float(v4[2]) * inv_l, __uint_as_float(v4[3]) * inv_l);
    }
  } else {
    uint8_t* rowp = ost + r * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t* v8 = ov + 8 * c;
      *reinterpret_cast<uint4*>(rowp + (((4 * hb + c) ^ (r & 7)) << 4)) = make_uint4(
          pack_bf16x2(__uint_as_float(v8[0]) * inv_l, __uint_as_float(v8[1]) * inv_l),
          pack_bf16x2(__uint_as_float(v8[2]) * inv_l, __uint_as_float(v8[3]) * inv_l),
          pack_bf16x2(__uint_as_float(v8[4]) * inv_l, __uint_as_float(v8[5]) * inv_l),
          pack_bf16x2(__uint_as_float(v8[6]) * inv_l, __uint_as_float(v8[7]) * inv_l));
    }
  }
}

// After stage_half of both halves: the row's LSE to global memory, then the
// tile's first warp stores the staged tile with TMA once all four warps have
// staged (o_full, phase `o_par`), clipped at T.
__device__ __forceinline__ void finish_store(const FwdArgs& a, const CUtensorMap* to,
                                             uint8_t* ost, uint64_t* o_full, uint32_t o_par,
                                             const SoftRow& row, int i, int row0, int bh,
                                             int warp, int lane, volatile int* ab) {
  if (i < a.T && a.lse)
    a.lse[static_cast<int64_t>(bh) * a.T + i] = (row.m + __log2f(row.le)) * kLn2f;
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(o_full);
  if ((warp & 3) == 0 && lane == 0) {
    if (mbar_wait(o_full, o_par, a.status, ab, kSiteSoftStore) &&
        store_row_ok(row0, a.T, a.status, ab, kSiteOutRow)) {
      if (a.o_fp32) {
        tma_store_3d(to, ost, 0, row0, bh);
        tma_store_3d(to, ost + kTileBytes, 32, row0, bh);
      } else {
        tma_store_3d(to, ost, 0, row0, bh);
      }
      bulk_commit();
      bulk_wait_read_all();  // the staging tile stays valid until read
    }
  }
}

// Logit scale c_i of query row i of head h, in log2 units.
__device__ __forceinline__ float logit_scale(const FwdArgs& a, int h, int i) {
  const float n = a.causal ? static_cast<float>(i + 1) : static_cast<float>(a.T);
  const float c = a.ssmax ? __ldg(a.s + h) * logf(n) * 0.125f : 0.125f;
  return c * 1.44269504088896341f;
}

// ================================================================ paired

__global__ void __launch_bounds__(kThreads, 1)
    bam_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                   const FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // Aligned by an offset from the shared array itself (not through an
  // integer cast), so that accesses stay in the shared address space.
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(smem_raw + ((0u - smem_u32(smem_raw)) & 1023u));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item (256 query rows of one head).
  const int BH = a.B * a.H;
  const int nqb = (a.T + 255) / 256;
  // Causal: the blocks with the most key tiles of every head first.
  // Non-causal (all blocks alike): head by head, so that the CTAs running at
  // the same time share their head's K and V in L2.
  const int qb = a.causal ? (nqb - 1 - static_cast<int>(blockIdx.x) / BH)
                          : static_cast<int>(blockIdx.x) % nqb;
  const int bh = a.causal ? static_cast<int>(blockIdx.x) % BH
                          : static_cast<int>(blockIdx.x) / nqb;
  const int h = bh % a.H;
  const int i0 = qb * 256;
  const int nkv = (a.T + 127) / 128;
  const int qt = i0 / 128;
  const bool hasB = i0 + 128 < a.T;
  const int nA = a.causal ? min(qt + 1, nkv) : nkv;
  const int nB = hasB ? (a.causal ? min(qt + 2, nkv) : nkv) : 0;
  const int nKV = max(nA, nB);
  volatile int* ab = &sm.abort_flag;

  const uint32_t tm = fwd_setup(sm, warp);
  // The distance table and the status word come from the previous kernel of
  // this call.  Only the producer runs ahead of it (its Q, K and V loads need
  // nothing from it); every other thread waits here, before its first look
  // at the status word.
  if (warp != 8) grid_dep_wait();

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = (*ab == 0);
      int issued = 0;
      bool q_issued = false;
      if (ok) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        mbar_arrive_expect_tx(&sm.q_full[0], kTileBytes * (hasB ? 2 : 1));
        tma_load_3d(sm.q[0], &tq, &sm.q_full[0], 0, i0, bh);
        if (hasB) tma_load_3d(sm.q[1], &tq, &sm.q_full[0], 0, i0 + 128, bh);
        q_issued = true;
      }
      for (int j = 0; ok && j < nKV; ++j) {
        const int s = j % kStages;
        if (j >= kStages) {
          ok = mbar_wait(&sm.kv_empty[s], ((j / kStages) - 1) & 1, a.status, ab, kSiteProducer);
          if (!ok) break;
        }
        ok = load_kv_tile(sm, a, &tk, &tv, s, j, bh, h, i0, j == 0, ab);
        issued = j + 1;
      }
      // Copies still in flight land before this CTA leaves.
      if (q_issued) mbar_drain(&sm.q_full[0], 0);
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        mbar_drain(&sm.k_full[j % kStages], (j / kStages) & 1);
        mbar_drain(&sm.v_full[j % kStages], (j / kStages) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = (*ab == 0);
      if (ok) ok = mbar_wait(&sm.q_full[0], 0, a.status, ab, kSiteMmaQ);
      if (ok) ok = mbar_wait(&sm.k_full[0], 0, a.status, ab, kSiteMmaK);
      if (ok) {
        tc_fence_after();
        if (nA > 0) issue_S(sm, tm, 0, 0, &sm.s_full[0]);
        if (nB > 0) issue_S(sm, tm + 128, 1, 0, &sm.s_full[1]);
      }
      for (int j = 0; ok && j < nKV; ++j) {
        const int s = j % kStages;
        if (j + 1 < nKV) {
          ok = mbar_wait(&sm.k_full[(j + 1) % kStages], ((j + 1) / kStages) & 1, a.status, ab,
                         kSiteMmaK);
          if (!ok) break;
        }
        ok = mbar_wait(&sm.v_full[s], (j / kStages) & 1, a.status, ab, kSiteMmaV);
        if (!ok) break;
        // Per query tile: S of the next key tile once the softmax has copied
        // the current S row, then PV once the probabilities are in, tile A's
        // pair before tile B's.  That order delays tile B by about half a
        // key tile at the start, after which the two softmax groups run
        // staggered (measured faster on long rows).  With only a few key
        // tiles the delay is not repaid, so there tile B's second S is
        // issued together with tile A's.
        const bool early_b = (j == 0 && nKV <= 8 && nB > 1);
        for (int t = 0; t < 2 && ok; ++t) {
          const int nt = t ? nB : nA;
          if (j >= nt) continue;
          if (j + 1 < nt && !(early_b && t == 1)) {
            ok = mbar_wait(&sm.s_free[t], j & 1, a.status, ab, kSiteMmaSFree);
            if (!ok) break;
            tc_fence_after();
            issue_S(sm, tm + 128 * t, t, (j + 1) % kStages, &sm.s_full[t]);
          }
          if (early_b && t == 0) {
            ok = mbar_wait(&sm.s_free[1], 0, a.status, ab, kSiteMmaSFree);
            if (!ok) break;
            tc_fence_after();
            issue_S(sm, tm + 128, 1, 1 % kStages, &sm.s_full[1]);
          }
          ok = mbar_wait(&sm.p_full[t], j & 1, a.status, ab, kSiteMmaP);
          if (!ok) break;
          tc_fence_after();
          issue_PV(sm, tm + 384 + 64 * t, tm + 256 + 64 * t, s, j == 0, &sm.pv_done[t]);
        }
        if (!ok) break;
        umma_commit(&sm.kv_empty[s]);
      }
      // Everything issued has completed before Tensor Memory is released.
      umma_commit(&sm.mma_final);
      mbar_drain(&sm.mma_final, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;              // 0: tile A, 1: tile B
    const int r = threadIdx.x - 128 * t;  // row within the tile = TMEM lane
    const int i = i0 + 128 * t + r;       // query position
    const int nt = t ? nB : nA;
    const uint32_t lb = tmem_lane_base(warp);
    const uint32_t tS = tm + lb + 128 * t;
    const uint32_t tP = tm + lb + 256 + 64 * t;
    const uint32_t tO = tm + lb + 384 + 64 * t;
    const float cr = logit_scale(a, h, i);
    SoftRow row{-INFINITY, 0.0f, 0.0f};
    bool ok = (*ab == 0);
    // Column c of this row reads window entry woff - c, i.e. reversed entry
    // kWin - 1 - woff + c; in copy kq those of c, c+1, c+2, c+3 (c % 4 == 0)
    // form one aligned 16-byte vector.
    const int woff = 128 * (t + 1) + r;
    const int kq = (r + 1) & 3;
    const int wrev = win_copy_off(kq, kWinCopyStride) + (kWin - 1 - woff + kq);
    for (int j = 0; ok && j < nt; ++j) {
      const int s = j % kStages;
      const int j0 = 128 * j;
      const bool masked = (a.causal && (j0 + 127 > i0 + 128 * t)) || (j0 + 128 > a.T);
      int lim = a.T - 1 - j0;
      if (a.causal) lim = min(lim, i - j0);
      const TilePhases ph{static_cast<uint32_t>(j & 1), static_cast<uint32_t>((j / kStages) & 1),
                          j > 0, static_cast<uint32_t>((j - 1) & 1)};
      ok = softmax_tile(sm, row, t, s, ph, sm.win[s] + wrev, cr, masked, lim, j > 0, tS, tP, tO,
                        a.status, ab, lane);
    }
    if (ok && nt > 0) {
      ok = warp_wait(&sm.pv_done[t], (nt - 1) & 1, a.status, ab, kSiteSoftEnd);
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / row.l;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t ov[32];
          tmem_ld_32x32b_x32(tO + 32 * hb, ov);
          tmem_ld_wait();
          reg_fence32(ov);
          stage_half(a, sm.ost[t], ov, hb, inv_l, r);
        }
        finish_store(a, &to, sm.ost[t], &sm.o_full[t], 0, row, i, i0 + 128 * t, bh, warp, lane,
                     ab);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

// ================================================================ single
// Short sequences: single-tile items (128 query rows of one (b, h)) on a
// persistent grid of two CTAs per SM.  Where paired CTAs would fill less than
// two waves of the SMs, a CTA per 256 rows leaves a ragged second wave of
// short tiles at the end; here each CTA walks a list of items (longest first,
// dealt in rounds of alternating direction, so that the short items of the
// last round go to the CTAs whose first items were short), one softmax group
// per CTA, 256 TMEM columns and ~107 KB of shared memory so that two CTAs
// share an SM and overlap each other's loads, first products and O stores.
// The K/V ring runs on across items; Q is reloaded once the item's last S
// product has read it; each softmax warp stages its own 32 rows of O in its
// quarter of a 16 KB staging tile and stores them itself (fp32 in two passes
// of 32 columns).
constexpr int kStages1 = 2;
constexpr int kThreads1 = 192;  // softmax warps 0-3, producer 4, MMA issuer 5
constexpr int kWin1 = 256;      // window entries per key tile (one query tile)
constexpr int kWin1CopyStride = 288;
constexpr int kWin1Stage = kTabCopies * kWin1CopyStride;
static_assert(win_copy_off(kTabCopies - 1, kWin1CopyStride) + kWin1 + 4 <= kWin1Stage, "window");

struct __align__(1024) Fwd1Smem {
  uint8_t q[1][kTileBytes];
  uint8_t k[kStages1][kTileBytes];
  uint8_t v[kStages1][kTileBytes];
  uint8_t ost[kTileBytes];  // per softmax warp, one 32-row 128-byte-swizzled box of O
  float win[kStages1][kWin1Stage];
  uint64_t q_full[1];
  uint64_t q_empty;   // the item's S products are done with its Q
  uint64_t k_full[kStages1];
  uint64_t v_full[kStages1];
  uint64_t kv_empty[kStages1];
  uint64_t s_full[1];
  uint64_t s_free[1];
  uint64_t p_full[1];
  uint64_t pv_done[1];
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Fwd1Smem) + 1024 <= 113 * 1024, "two CTAs per SM");

// Item n of this persistent CTA: query tile qt of head bh (nKV key tiles).
struct Item1 {
  int qt, bh, h, nKV;
};

__device__ __forceinline__ bool single_item(const FwdArgs& a, int n, Item1& it) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int BH = a.B * a.H, nqt = (a.T + 127) / 128;
  const int idx = n * G + ((n & 1) ? (G - 1 - c) : c);
  if (idx >= nqt * BH) return false;
  const int q = idx / BH;
  it.qt = a.causal ? nqt - 1 - q : q;
  it.bh = idx % BH;
  it.h = it.bh % a.H;
  it.nKV = a.causal ? it.qt + 1 : nqt;
  return true;
}

// TMEM columns (256): S [0,128) P [128,192) O [192,256).
__global__ void __launch_bounds__(kThreads1, 2)
    bam_fwd_single_kernel(const __grid_constant__ CUtensorMap tq,
                          const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv,
                          const __grid_constant__ CUtensorMap to, const FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Fwd1Smem& sm = *reinterpret_cast<Fwd1Smem*>(smem_raw + ((0u - smem_u32(smem_raw)) & 1023u));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* ab = &sm.abort_flag;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.q_full[0], 1);
    mbar_init(&sm.q_empty, 1);
    for (int s = 0; s < kStages1; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(&sm.s_full[0], 1);
    mbar_init(&sm.s_free[0], 4);
    mbar_init(&sm.p_full[0], 4);
    mbar_init(&sm.pv_done[0], 1);
    mbar_init(&sm.mma_final, 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&sm.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  // As in the paired kernel, only the producer runs ahead of the table
  // kernel; everyone else waits here before looking at the status word.
  if (warp != 4) grid_dep_wait();

  // Barrier phases run on over the CTA's items: Q by item, the K/V stages
  // and the per-tile barriers by the running key-tile count.
  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = (*ab == 0);
      int jg = 0, q_items = 0;
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      Item1 it;
      for (int n = 0; ok && single_item(a, n, it); ++n) {
        if (n > 0) {
          ok = mbar_wait(&sm.q_empty, (n - 1) & 1, a.status, ab, kSiteProducer);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(&sm.q_full[0], kTileBytes);
        tma_load_3d(sm.q[0], &tq, &sm.q_full[0], 0, 128 * it.qt, it.bh);
        q_items = n + 1;
        for (int j = 0; ok && j < it.nKV; ++j, ++jg) {
          const int s = jg % kStages1;
          if (jg >= kStages1) {
            ok = mbar_wait(&sm.kv_empty[s], ((jg / kStages1) - 1) & 1, a.status, ab,
                           kSiteProducer);
            if (!ok) break;
          }
          ok = load_kv_tile<kWin1, kWin1CopyStride>(sm, a, &tk, &tv, s, j, it.bh, it.h,
                                                     128 * it.qt, jg == 0, ab, jg == 0);
        }
      }
      // Copies still in flight land before this CTA leaves.
      if (q_items > 0) mbar_drain(&sm.q_full[0], (q_items - 1) & 1);
      for (int x = max(0, jg - kStages1); x < jg; ++x) {
        mbar_drain(&sm.k_full[x % kStages1], (x / kStages1) & 1);
        mbar_drain(&sm.v_full[x % kStages1], (x / kStages1) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = (*ab == 0);
      int jg = 0;
      Item1 it;
      for (int n = 0; ok && single_item(a, n, it); ++n) {
        ok = mbar_wait(&sm.q_full[0], n & 1, a.status, ab, kSiteMmaQ);
        if (!ok) break;
        // The S columns are free once the softmax has copied the previous S.
        if (jg > 0) {
          ok = mbar_wait(&sm.s_free[0], (jg - 1) & 1, a.status, ab, kSiteMmaSFree);
          if (!ok) break;
        }
        ok = mbar_wait(&sm.k_full[jg % kStages1], (jg / kStages1) & 1, a.status, ab, kSiteMmaK);
        if (!ok) break;
        tc_fence_after();
        issue_S(sm, tm, 0, jg % kStages1, &sm.s_full[0]);
        // Q is free for the next item once the item's last S is done.
        if (it.nKV == 1) umma_commit(&sm.q_empty);
        // Per key tile: S of the next tile once the softmax has copied this
        // S, then PV once its probabilities are in.
        for (int j = 0; ok && j < it.nKV; ++j) {
          const int g = jg + j, s = g % kStages1;
          if (j + 1 < it.nKV) {
            ok = mbar_wait(&sm.s_free[0], g & 1, a.status, ab, kSiteMmaSFree);
            if (!ok) break;
            ok = mbar_wait(&sm.k_full[(g + 1) % kStages1], ((g + 1) / kStages1) & 1, a.status,
                           ab, kSiteMmaK);
            if (!ok) break;
            tc_fence_after();
            issue_S(sm, tm, 0, (g + 1) % kStages1, &sm.s_full[0]);
            if (j + 2 == it.nKV) umma_commit(&sm.q_empty);
          }
          ok = mbar_wait(&sm.v_full[s], (g / kStages1) & 1, a.status, ab, kSiteMmaV);
          if (!ok) break;
          ok = mbar_wait(&sm.p_full[0], g & 1, a.status, ab, kSiteMmaP);
          if (!ok) break;
          tc_fence_after();
          issue_PV(sm, tm + 192, tm + 128, s, j == 0, &sm.pv_done[0]);
          umma_commit(&sm.kv_empty[s]);
        }
        if (!ok) break;
        jg += it.nKV;
      }
      umma_commit(&sm.mma_final);
      mbar_drain(&sm.mma_final, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // row within the tile = TMEM lane
    const uint32_t lb = tmem_lane_base(warp);
    const uint32_t tS = tm + lb, tP = tm + lb + 128, tO = tm + lb + 192;
    // Column c reads window entry 128 + r - c: reversed entry 127 - r + c, in
    // copy kq one aligned 16-byte vector per four columns.
    const int kq = (r + 1) & 3;
    const int wrev = win_copy_off(kq, kWin1CopyStride) + (kWin1 - 129 - r + kq);
    bool ok = (*ab == 0);
    int jg = 0, boxes = 0;
    Item1 it;
    for (int n = 0; ok && single_item(a, n, it); ++n) {
      const int i0 = 128 * it.qt, i = i0 + r;
      const float cr = logit_scale(a, it.h, i);
      SoftRow row{-INFINITY, 0.0f, 0.0f};
      for (int j = 0; ok && j < it.nKV; ++j) {
        const int g = jg + j, s = g % kStages1;
        const int j0 = 128 * j;
        const bool masked = (a.causal && (j0 + 127 > i0)) || (j0 + 128 > a.T);
        int lim = a.T - 1 - j0;
        if (a.causal) lim = min(lim, i - j0);
        const TilePhases ph{static_cast<uint32_t>(g & 1),
                            static_cast<uint32_t>((g / kStages1) & 1), j > 0,
                            static_cast<uint32_t>((g - 1) & 1)};
        ok = softmax_tile(sm, row, 0, s, ph, sm.win[s] + wrev, cr, masked, lim, j > 0, tS, tP, tO,
                          a.status, ab, lane);
      }
      jg += it.nKV;
      if (ok) ok = warp_wait(&sm.pv_done[0], (jg - 1) & 1, a.status, ab, kSiteSoftEnd);
      if (!ok) break;
      // O leaves through this warp's quarter of the staging tile, one
      // 32-row box per TMA store issued by the warp itself (no hand-off
      // between warps): fp32 as two boxes of 32 columns, bf16 as one of 64.
      // A box is staged once the warp's previous store has read the quarter.
      tc_fence_after();
      const float inv_l = 1.0f / row.l;
      const int nbox = a.o_fp32 ? 2 : 1;
      const int rw = i0 + 32 * warp;  // first row of this warp's box
      uint8_t* quarter = sm.ost + warp * (kTileBytes / 4);
      for (int bx = 0; bx < nbox; ++bx, ++boxes) {
        if (boxes > 0) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
        for (int hb = (a.o_fp32 ? bx : 0); hb < (a.o_fp32 ? bx + 1 : 2); ++hb) {
          uint32_t ov[32];
          tmem_ld_32x32b_x32(tO + 32 * hb, ov);
          tmem_ld_wait();
          reg_fence32(ov);
          stage_half(a, quarter, ov, hb, inv_l, r & 31, 0);
        }
        if (bx == 0 && i < a.T && a.lse)
          a.lse[static_cast<int64_t>(it.bh) * a.T + i] = (row.m + __log2f(row.le)) * kLn2f;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && rw < a.T && store_row_ok(rw, a.T, a.status, ab, kSiteOutRow)) {
          tma_store_3d(&to, quarter, a.o_fp32 ? 32 * bx : 0, rw, it.bh);
          bulk_commit();
        }
      }
    }
    // The staging quarter stays valid until this warp's last store has read it.
    if (lane == 0) bulk_wait_read_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tm, 256);
  }
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& to32, const FwdArgs& a,
                       cudaStream_t st) {
  const size_t smem = sizeof(FwdSmem) + 1024, smem1 = sizeof(Fwd1Smem) + 1024;
  static bool paired_set[64] = {}, single_set[64] = {};
  cudaError_t e = smem_limit_once(bam_fwd_kernel, smem, paired_set);
  if (e == cudaSuccess) e = smem_limit_once(bam_fwd_single_kernel, smem1, single_set);
  if (e != cudaSuccess) return e;
  // Paired CTAs (256 rows, one per SM) when they fill at least two waves of
  // the SMs; otherwise the persistent single-tile grid, two CTAs per SM.
  const long bh = static_cast<long>(a.B) * a.H;
  const long paired = static_cast<long>((a.T + 255) / 256) * bh;
  int sms = sm_count();
  if (sms <= 0) sms = 148;
  if (paired < 2L * sms) {
    const long items = static_cast<long>((a.T + 127) / 128) * bh;
    const unsigned grid = static_cast<unsigned>(items < 2L * sms ? items : 2L * sms);
    return launch_k(bam_fwd_single_kernel, dim3(grid), dim3(kThreads1), smem1, st, true, tq, tk,
                    tv, to32, a);
  }
  return launch_k(bam_fwd_kernel, dim3(static_cast<unsigned>(paired)), dim3(kThreads), smem, st,
                  true, tq, tk, tv, to, a);
}

}  // namespace bam
