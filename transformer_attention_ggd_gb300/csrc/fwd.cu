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
// One CTA owns 256 query rows of one (b, h) as two 128-row tiles A and B and
// walks the key/value tiles of 128 keys:
//   warp 8      TMA producer: Q once; per key tile K, V and the 384-entry
//               distance window (four shifted reversed copies, so that a
//               thread reads four keys' biases with one 16-byte load), into
//               a 3-stage ring.
//   warp 9      MMA issuer (one thread): S_t = Q_t K^T (128x128x64, both
//               operands K-major in shared memory) and O_t += P_t V (P from
//               Tensor Memory, V MN-major), accumulators in Tensor Memory.
//               Also allocates / frees the 512 TMEM columns.
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: one thread
//               per query row reads its S row from TMEM, adds c_i S + bias in
//               log2 units, runs the online softmax (exp2, rescaling O in
//               TMEM only when the running max grows by more than 8), writes
//               P (bf16) back to TMEM, and in the end normalises O.
// The two softmax groups are offset by one MMA so the tensor core works on
// one tile while the other is in its softmax.
//
// TMEM columns: S_A [0,128) S_B [128,256) P_A [256,320) P_B [320,384)
//               O_A [384,448) O_B [448,512).
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
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t o_full[2];  // the tile's four softmax warps have staged their O rows
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

  // Work item: causal blocks with the most key tiles go first.
  const int BH = a.B * a.H;
  const int qb = a.causal ? (a.nqb - 1 - static_cast<int>(blockIdx.x) / BH)
                          : static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int h = bh % a.H;
  const int i0 = qb * 256;
  const int nkv = (a.T + 127) / 128;
  const int qt = i0 / 128;
  const bool hasB = i0 + 128 < a.T;
  const int nA = a.causal ? min(qt + 1, nkv) : nkv;
  const int nB = hasB ? (a.causal ? min(qt + 2, nkv) : nkv) : 0;
  const int nKV = max(nA, nB);
  volatile int* ab = &sm.abort_flag;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.q_full, 1);
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
  const uint32_t tm = sm.tmem_base;
  // The distance table and the cleared status word come from the previous
  // kernel of this call.  Only the producer runs ahead of it (its Q, K and V
  // loads need nothing from it); every other thread waits here, before its
  // first look at the status word.
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
        mbar_arrive_expect_tx(&sm.q_full, kTileBytes * (hasB ? 2 : 1));
        tma_load_3d(sm.q[0], &tq, &sm.q_full, 0, i0, bh);
        if (hasB) tma_load_3d(sm.q[1], &tq, &sm.q_full, 0, i0 + 128, bh);
        q_issued = true;
      }
      // The window of key tile j covers table indices tab_off + i0 - 128 -
      // 128 j + [0, kWin); in the reversed rows it starts at tab_len - kWin
      // minus that base (a multiple of 4 entries).
      const size_t copy_stride = static_cast<size_t>(a.H) * a.tab_len;
      const float* tab_h = a.table + static_cast<size_t>(h) * a.tab_len +
                           (a.tab_len - kWin - a.tab_off - i0 + 128);
      // A window starts inside its own row and may run past the row's end
      // into the padding after the last row, never beyond it.
      const float* tab_end = a.table + kTabCopies * copy_stride + kTabPadFloats;
      for (int j = 0; ok && j < nKV; ++j) {
        const int s = j % kStages;
        if (j >= kStages) {
          ok = mbar_wait(&sm.kv_empty[s], ((j / kStages) - 1) & 1, a.status, ab, kSiteProducer);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(&sm.k_full[s], kTileBytes + kTabCopies * kWinCopy * 4);
        tma_load_3d(sm.k[s], &tk, &sm.k_full[s], 0, 128 * j, bh);
        if (j == 0) grid_dep_wait();  // the windows come from the table kernel
        for (int k = 0; k < kTabCopies; ++k)
          ok &= bulk_load_checked(sm.win[s] + win_copy_off(k, kWinCopyStride),
                                  tab_h + k * copy_stride + 128 * j, kWinCopy * 4, &sm.k_full[s],
                                  a.table + k * copy_stride + static_cast<size_t>(h) * a.tab_len,
                                  tab_end, a.status, ab, kSiteWindowCopy);
        mbar_arrive_expect_tx(&sm.v_full[s], kTileBytes);
        tma_load_3d(sm.v[s], &tv, &sm.v_full[s], 0, 128 * j, bh);
        issued = j + 1;
      }
      // Copies still in flight land before this CTA leaves.
      if (q_issued) mbar_drain(&sm.q_full, 0);
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        mbar_drain(&sm.k_full[j % kStages], (j / kStages) & 1);
        mbar_drain(&sm.v_full[j % kStages], (j / kStages) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = (*ab == 0);
      const uint32_t idS = idesc_bf16(128, 128, false, false);
      const uint32_t idO = idesc_bf16(128, 64, false, true);
      // Shared-memory descriptors of the first Q, K and V tiles; the others
      // (and the K-steps inside a tile) are fixed offsets from them, so each
      // MMA costs the issuing thread only an add or two.
      const uint64_t dq0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(sm.v[0]), 16384, 1024);
      constexpr uint64_t kTileDesc = kTileBytes >> 4;  // descriptor units of 16 bytes
      auto issue_S = [&](int t, int s) {
        const uint64_t qd = dq0 + kTileDesc * t, kd = dk0 + kTileDesc * s;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ss(tm + 128 * t, qd + 2 * kk, kd + 2 * kk, idS, kk > 0 ? 1u : 0u);
        umma_commit(&sm.s_full[t]);
      };
      auto issue_PV = [&](int t, int s, int j) {
        const uint64_t vd = dv0 + kTileDesc * s;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tm + 384 + 64 * t, tm + 256 + 64 * t + 8 * kk, vd + 128 * kk, idO,
                  (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&sm.pv_done[t]);
      };
      if (ok) ok = mbar_wait(&sm.q_full, 0, a.status, ab, kSiteMmaQ);
      if (ok) ok = mbar_wait(&sm.k_full[0], 0, a.status, ab, kSiteMmaK);
      if (ok) {
        tc_fence_after();
        if (nA > 0) issue_S(0, 0);
        if (nB > 0) issue_S(1, 0);
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
            issue_S(t, (j + 1) % kStages);
          }
          if (early_b && t == 0) {
            ok = mbar_wait(&sm.s_free[1], 0, a.status, ab, kSiteMmaSFree);
            if (!ok) break;
            tc_fence_after();
            issue_S(1, 1 % kStages);
          }
          ok = mbar_wait(&sm.p_full[t], j & 1, a.status, ab, kSiteMmaP);
          if (!ok) break;
          tc_fence_after();
          issue_PV(t, s, j);
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
    const int t = warp >> 2;                 // 0: tile A, 1: tile B
    const int r = threadIdx.x - 128 * t;     // row within the tile = TMEM lane
    const int i = i0 + 128 * t + r;          // query position
    const int nt = t ? nB : nA;
    const uint32_t lb = tmem_lane_base(warp);
    const uint32_t tS = tm + lb + 128 * t;
    const uint32_t tP = tm + lb + 256 + 64 * t;
    const uint32_t tO = tm + lb + 384 + 64 * t;
    float cr;  // logit scale in log2 units
    {
      const float n = a.causal ? static_cast<float>(i + 1) : static_cast<float>(a.T);
      const float c = a.ssmax ? __ldg(a.s + h) * logf(n) * 0.125f : 0.125f;
      cr = c * 1.44269504088896341f;
    }
    float m = -INFINITY, l = 0.0f, le = 0.0f;
    bool ok = (*ab == 0);
    // Column c of this row reads window entry woff - c, i.e. reversed entry
    // kWin - 1 - woff + c; in copy kq those of c, c+1, c+2, c+3 (c % 4 == 0)
    // form one aligned 16-byte vector.
    const int woff = 128 * (t + 1) + r;
    const int kq = (r + 1) & 3;
    const int wrev = win_copy_off(kq, kWinCopyStride) + (kWin - 1 - woff + kq);
    for (int j = 0; ok && j < nt; ++j) {
      const int s = j % kStages;
      ok = warp_wait(&sm.s_full[t], j & 1, a.status, ab, kSiteSoftS);
      if (!ok) break;
      ok = warp_wait(&sm.k_full[s], (j / kStages) & 1, a.status, ab, kSiteSoftK);
      if (!ok) break;
      tc_fence_after();
      // S row -> z = c_i S + bias (log2 units) as column pairs (f32x2), 8
      // columns at a time; the next chunk's TMEM load overlaps this chunk's
      // arithmetic.
      const float* wv = sm.win[s] + wrev;
      const uint64_t cr2 = f2_pack(cr, cr);
      uint64_t z[64];
      uint32_t sr[2][8];
      tmem_ld_32x32b_x8(tS, sr[0]);
      tmem_ld_wait();
      reg_fence8(sr[0]);
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        if (ch < 15) tmem_ld_32x32b_x8(tS + 8 * (ch + 1), sr[(ch + 1) & 1]);
#pragma unroll
        for (int x = 0; x < 4; x += 2) {
          uint64_t t0, t1;
          ld_f2x2(wv + 8 * ch + 2 * x, t0, t1);
          const uint64_t s0 = f2_pack(__uint_as_float(sr[ch & 1][2 * x]),
                                      __uint_as_float(sr[ch & 1][2 * x + 1]));
          const uint64_t s1 = f2_pack(__uint_as_float(sr[ch & 1][2 * x + 2]),
                                      __uint_as_float(sr[ch & 1][2 * x + 3]));
          z[4 * ch + x] = ffma2(s0, cr2, t0);
          z[4 * ch + x + 1] = ffma2(s1, cr2, t1);
        }
        if (ch < 15) {
          tmem_ld_wait();
          reg_fence8(sr[(ch + 1) & 1]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_free[t]);

      const int j0 = 128 * j;
      const bool tail = j0 + 128 > a.T;
      const bool diag = a.causal && (j0 + 127 > i0 + 128 * t);
      if (diag || tail) {
        int lim = a.T - 1 - j0;
        if (a.causal) lim = min(lim, i - j0);
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
      const float m_new = fmaxf(m, mx);
      const bool resc = m_new > m + kRescaleThreshold;
      float scale = 1.0f;
      if (resc) {
        scale = ex2_approx(m - m_new);
        l *= scale;
        le *= scale;
        m = m_new;
      }
      if (j > 0) {
        // PV of the previous tile must be done: frees P and makes O stable.
        ok = warp_wait(&sm.pv_done[t], (j - 1) & 1, a.status, ab, kSiteSoftPV);
        if (!ok) break;
        tc_fence_after();
      }
      // Probabilities as bf16 pairs for the PV product, streamed to TMEM 32
      // columns at a time, and the two row sums (rounded weights for O,
      // unrounded for the LSE) in independent partial sums.
      const uint64_t negm2 = f2_pack(-m, -m);
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
        l += (lr[0] + lr[1]) + (lr[2] + lr[3]);
        le += b0 + b1;
      }
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
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
    }
    if (ok && nt > 0) {
      ok = warp_wait(&sm.pv_done[t], (nt - 1) & 1, a.status, ab, kSiteSoftEnd);
      if (ok) {
        tc_fence_after();
        uint32_t ov[64];
        tmem_ld_32x32b_x32(tO, ov);
        tmem_ld_32x32b_x32(tO + 32, ov + 32);
        tmem_ld_wait();
        reg_fence32(ov);
        reg_fence32(ov + 32);
        // Row r of the tile into the staging tile (128-byte rows, 16-byte
        // chunk c at (c ^ (r % 8)) * 16); one TMA store per box writes the
        // tile, clipped at T.
        const float inv_l = 1.0f / l;
        if (a.o_fp32) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            uint8_t* rowp = sm.ost[t] + b * kTileBytes + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* v4 = ov + 32 * b + 4 * c;
              *reinterpret_cast<float4*>(rowp + ((c ^ (r & 7)) << 4)) =
                  make_float4(__uint_as_float(v4[0]) * inv_l, __uint_as_float(v4[1]) * inv_l,
                              __uint_as_float(v4[2]) * inv_l, __uint_as_float(v4[3]) * inv_l);
            }
          }
        } else {
          uint8_t* rowp = sm.ost[t] + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t* v8 = ov + 8 * c;
            *reinterpret_cast<uint4*>(rowp + ((c ^ (r & 7)) << 4)) = make_uint4(
                pack_bf16x2(__uint_as_float(v8[0]) * inv_l, __uint_as_float(v8[1]) * inv_l),
                pack_bf16x2(__uint_as_float(v8[2]) * inv_l, __uint_as_float(v8[3]) * inv_l),
                pack_bf16x2(__uint_as_float(v8[4]) * inv_l, __uint_as_float(v8[5]) * inv_l),
                pack_bf16x2(__uint_as_float(v8[6]) * inv_l, __uint_as_float(v8[7]) * inv_l));
          }
        }
        if (i < a.T && a.lse) a.lse[static_cast<int64_t>(bh) * a.T + i] = (m + __log2f(le)) * kLn2f;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.o_full[t]);
        if ((warp & 3) == 0 && lane == 0) {
          // The tile's first warp stores it once all four have staged.
          const int row0 = i0 + 128 * t;
          if (mbar_wait(&sm.o_full[t], 0, a.status, ab, kSiteSoftStore) &&
              store_row_ok(row0, a.T, a.status, ab, kSiteOutRow)) {
            if (a.o_fp32) {
              tma_store_3d(&to, sm.ost[t], 0, row0, bh);
              tma_store_3d(&to, sm.ost[t] + kTileBytes, 32, row0, bh);
            } else {
              tma_store_3d(&to, sm.ost[t], 0, row0, bh);
            }
            bulk_commit();
            bulk_wait_read_all();  // the staging tile stays valid until read
          }
        }
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

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(FwdSmem) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bam_fwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const unsigned grid = static_cast<unsigned>(a.nqb) * static_cast<unsigned>(a.B * a.H);
  return launch_k(bam_fwd_kernel, dim3(grid), dim3(kThreads), smem, st, true, tq, tk, tv, to, a);
}

}  // namespace bam
