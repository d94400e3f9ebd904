// Split-KV decode for GGD-BAM attention on sm_103a.
//
// One new query per (b, h) attends to a cache of Tkv keys that already holds
// its own key; the query sits at position Tkv-1, so key j is at distance
// d = Tkv-1-j and every key is visible (n = Tkv for Scalable-Softmax).  The
// long-context evaluation of the BAM README ("Evaluation", passkey retrieval
// up to 32k tokens) is the workload this serves.
//
// The work is a stream over the cache: 256 bytes of K and V per key against
// 256 multiply-adds, so it is bound by HBM bandwidth, not by math.  Each CTA
// takes one (b, h) and one contiguous chunk of keys; a producer warp streams
// 64-key stages of K, V and the matching 64 bias-table entries into a 4-deep
// shared-memory ring with plain bulk copies (each stage is one contiguous
// 8 KB run of K and of V), and four consumer warps reduce them:
// two lanes per key (32 dimensions each), dot product in fp32, lazy online
// softmax in log2 units, p * v accumulated in registers.  The partial
// (max, sum, unnormalised output) of each chunk goes to the workspace and a
// second kernel merges the chunks of each (b, h).
//
// Ragged decode: sequence b holds len_b <= Tkv cached keys (the cache keeps
// its [B, H, Tkv, 64] layout); its query sits at position len_b - 1 and
// n = len_b.  Key j then reads table entry j + (Tkv - len_b) of the table
// built for Tkv, so each stage copies an aligned 68-entry window and indexes
// it with the remainder; chunks past len_b hold no keys and leave an empty
// partial, which the merge skips.
//
// Paged cache: K and V live in pages of `page` keys (a multiple of 64), laid
// out [num_pages, H, page, 64]; a sequence's logical block i is the page its
// block-table row names, so a 64-key stage is one contiguous run of a page
// and only the producer's source address changes.
#include "bam_common.cuh"

namespace bam {
namespace {

constexpr int kDecStages = 4;
constexpr int kDecKeys = 64;                 // keys per stage
constexpr int kDecTab = kDecKeys + 4;        // table entries per stage (aligned window)
constexpr int kDecConsumerWarps = 4;
constexpr int kDecThreads = 32 * (kDecConsumerWarps + 1);
constexpr int kStageBytes = kDecKeys * kHeadDim * 2;  // 8 KB of K (and of V)
constexpr float kDecRescale = 8.0f;
constexpr int kPartStride = 2 + kHeadDim;   // m, l, o[64]

struct __align__(128) DecSmem {
  uint8_t k[kDecStages][kStageBytes];
  uint8_t v[kDecStages][kStageBytes];
  float tab[kDecStages][kDecTab];
  float red[kDecConsumerWarps][kPartStride];
  uint64_t full[kDecStages];
  uint64_t empty[kDecStages];
  int abort_flag;
};

enum : int {
  kSiteDecProducer = 40,
  kSiteDecConsumer = 41,
  // Debug-build bounds checks (BAM_DEV_BOUNDS)
  kSiteDecKV = 42,
  kSiteDecTable = 43
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& w, float* f) {
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  f[4] = __uint_as_float(w.z << 16);
  f[5] = __uint_as_float(w.z & 0xFFFF0000u);
  f[6] = __uint_as_float(w.w << 16);
  f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

// Merge (m2, l2, o2) into (m, l, o); m in log2 units.
__device__ __forceinline__ void merge_state(float& m, float& l, float* o, float m2, float l2,
                                            const float* o2, int n) {
  const float mn = fmaxf(m, m2);
  const float a = (m == -INFINITY) ? 0.0f : ex2_approx(m - mn);
  const float b = (m2 == -INFINITY) ? 0.0f : ex2_approx(m2 - mn);
  l = l * a + l2 * b;
  for (int x = 0; x < n; ++x) o[x] = o[x] * a + o2[x] * b;
  m = mn;
}

__global__ void __launch_bounds__(kDecThreads)
    bam_decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // Aligned by an offset from the shared array itself (not through an
  // integer cast), so that accesses stay in the shared address space.
  DecSmem& sm = *reinterpret_cast<DecSmem*>(smem_raw + ((0u - smem_u32(smem_raw)) & 127u));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sp = blockIdx.x;
  const int bh = blockIdx.y;
  const int h = bh % a.H;
  // Keys of this (b, h): all Tkv, or the sequence's own cache length.
  int len = a.Tkv;
  bool bad_len = false;
  if (a.lens) {
    const int raw = __ldg(a.lens + bh / a.H);
    len = min(max(raw, 1), a.Tkv);
    bad_len = raw != len;
  }
  const int kbeg = sp * a.chunk;
  const int kend = min(len, kbeg + a.chunk);
  const int nst = kend > kbeg ? (kend - kbeg + kDecKeys - 1) / kDecKeys : 0;
  const int tshift = a.Tkv - len;  // table entry of key j: j + tshift
  const int trem = tshift & 3;     // offset of key 0 of a stage in its window
  volatile int* ab = &sm.abort_flag;

  if (threadIdx.x == 0) {
    grid_dep_wait();  // the decode table comes from the previous kernel
    sm.abort_flag = *reinterpret_cast<volatile int*>(&a.status->abort);
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kDecConsumerWarps);
    }
    fence_barrier_init();
    // Recorded after the wait: the table kernel clears the status word.
    if (bad_len && sp == 0 && h == 0) atomicCAS(&a.status->code, BAM_DEV_OK, BAM_DEV_BAD_ARG);
  }
  __syncthreads();

  if (warp == kDecConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = (*ab == 0);
      int issued = 0;
      bool bad_page = false;
      const size_t row0 = static_cast<size_t>(bh) * a.Tkv;
      for (int it = 0; ok && it < nst; ++it) {
        const int s = it % kDecStages;
        if (it >= kDecStages) {
          ok = mbar_wait(&sm.empty[s], ((it / kDecStages) - 1) & 1, a.status, ab,
                         kSiteDecProducer);
          if (!ok) break;
        }
        const int kb = kbeg + it * kDecKeys;
        const int nk = min(kDecKeys, kend - kb);
        const uint32_t bytes = static_cast<uint32_t>(nk) * kHeadDim * 2;
        mbar_arrive_expect_tx(&sm.full[s], 2 * bytes + kDecTab * 4);
        size_t key0 = row0 + kb;  // first key of the stage, in keys of the cache
        size_t seg0 = row0, seg1 = row0 + a.Tkv;  // the keys a stage may read
        if (a.block_table) {
          int pg = __ldg(a.block_table + static_cast<size_t>(bh / a.H) * a.max_blocks +
                         kb / a.page);
          if (pg < 0 || pg >= a.num_pages) {
            bad_page = true;
            pg = 0;
          }
          seg0 = (static_cast<size_t>(pg) * a.H + h) * a.page;
          seg1 = seg0 + a.page;  // a stage never crosses a page
          key0 = seg0 + kb % a.page;
        }
        ok &= bulk_load_checked(sm.k[s], a.kc + key0 * kHeadDim, bytes, &sm.full[s],
                                a.kc + seg0 * kHeadDim, a.kc + seg1 * kHeadDim, a.status, ab,
                                kSiteDecKV);
        ok &= bulk_load_checked(sm.v[s], a.vc + key0 * kHeadDim, bytes, &sm.full[s],
                                a.vc + seg0 * kHeadDim, a.vc + seg1 * kHeadDim, a.status, ab,
                                kSiteDecKV);
        // 16-byte aligned window starting at or below entry kb + tshift
        const float* trow = a.table + static_cast<size_t>(h) * a.tab_len;
        ok &= bulk_load_checked(sm.tab[s], trow + ((kb + tshift) & ~3), kDecTab * 4, &sm.full[s],
                                trow, trow + a.tab_len, a.status, ab, kSiteDecTable);
        issued = it + 1;
      }
      for (int it = max(0, issued - kDecStages); it < issued; ++it)
        mbar_drain(&sm.full[it % kDecStages], (it / kDecStages) & 1);
      if (bad_page) atomicCAS(&a.status->code, BAM_DEV_OK, BAM_DEV_BAD_ARG);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int kk = 16 * warp + (lane >> 1);  // key slot within a stage
    const int hf = lane & 1;                 // which 32 dimensions
    float cr;
    {
      const float c = a.ssmax ? __ldg(a.s + h) * logf(static_cast<float>(len)) * 0.125f
                              : 0.125f;
      cr = c * 1.44269504088896341f;
    }
    float q[32];
    {
      const uint4* qp = reinterpret_cast<const uint4*>(a.q + static_cast<size_t>(bh) * kHeadDim +
                                                       32 * hf);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        bf16x8_to_f32(__ldg(qp + x), q + 8 * x);
      }
#pragma unroll
      for (int x = 0; x < 32; ++x) q[x] *= cr;
    }
    float m = -INFINITY, l = 0.0f, o[32];
#pragma unroll
    for (int x = 0; x < 32; ++x) o[x] = 0.0f;
    bool ok = (*ab == 0);
    for (int it = 0; ok && it < nst; ++it) {
      const int s = it % kDecStages;
      ok = mbar_wait(&sm.full[s], (it / kDecStages) & 1, a.status, ab, kSiteDecConsumer);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const bool valid = kbeg + it * kDecKeys + kk < kend;
      const uint4* kp = reinterpret_cast<const uint4*>(sm.k[s] + kk * 128 + 64 * hf);
      float dot = 0.0f;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        float kf[8];
        bf16x8_to_f32(kp[x], kf);
#pragma unroll
        for (int y = 0; y < 8; ++y) dot = fmaf(q[8 * x + y], kf[y], dot);
      }
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      if (valid) {
        const float z = dot + sm.tab[s][kk + trem];
        if (z > m + kDecRescale) {
          const float corr = ex2_approx(m - z);
          l *= corr;
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] *= corr;
          m = z;
        }
        const float p = ex2_approx(z - m);
        l += p;
        const uint4* vp = reinterpret_cast<const uint4*>(sm.v[s] + kk * 128 + 64 * hf);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          float vf[8];
          bf16x8_to_f32(vp[x], vf);
#pragma unroll
          for (int y = 0; y < 8; ++y) o[8 * x + y] = fmaf(p, vf[y], o[8 * x + y]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
    }
    // Merge the 16 key slots of each half within the warp.
#pragma unroll
    for (int off = 2; off < 32; off <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
      float o2[32];
#pragma unroll
      for (int x = 0; x < 32; ++x) o2[x] = __shfl_xor_sync(0xffffffffu, o[x], off);
      merge_state(m, l, o, m2, l2, o2, 32);
    }
    if (lane < 2) {
      if (lane == 0) {
        sm.red[warp][0] = m;
        sm.red[warp][1] = l;
      }
#pragma unroll
      for (int x = 0; x < 32; ++x) sm.red[warp][2 + 32 * hf + x] = o[x];
    }
  }
  __syncthreads();
  grid_dep_trigger();
  // Merge the four consumer warps and write this chunk's partial.
  if (threadIdx.x < kHeadDim && *ab == 0) {
    const int x = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < kDecConsumerWarps; ++w) M = fmaxf(M, sm.red[w][0]);
    float L = 0.0f, O = 0.0f;
    for (int w = 0; w < kDecConsumerWarps; ++w) {
      const float mw = sm.red[w][0];
      const float sc = (mw == -INFINITY) ? 0.0f : ex2_approx(mw - M);
      L += sm.red[w][1] * sc;
      O += sm.red[w][2 + x] * sc;
    }
    float* dst = a.part + (static_cast<size_t>(bh) * a.nsplit + sp) * kPartStride;
    dst[2 + x] = O;
    if (x == 0) {
      dst[0] = M;
      dst[1] = L;
    }
  }
}

// One warp per (b, h): merge the split partials, normalise, write O and LSE.
__global__ void __launch_bounds__(128) bam_decode_combine_kernel(const DecodeArgs a) {
  grid_dep_wait();  // partials of the decode kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x * 4 + warp;
  if (bh >= a.B * a.H) return;
  const size_t off = static_cast<size_t>(bh) * kHeadDim + 2 * lane;
  if (*reinterpret_cast<volatile int*>(&a.status->abort)) {
    // The call gave up: its partials are incomplete, so the outputs are
    // marked invalid (NaN) rather than left as they were.
    const float nan = __int_as_float(0x7fc00000);
    if (a.o_fp32) {
      reinterpret_cast<float2*>(static_cast<float*>(a.o) + off)[0] = make_float2(nan, nan);
    } else {
      reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.o) + off)[0] = 0x7fc07fc0u;
    }
    if (a.lse && lane == 0) a.lse[bh] = nan;
    return;
  }
  const float* part = a.part + static_cast<size_t>(bh) * a.nsplit * kPartStride;
  float M = -INFINITY;
  for (int sp = 0; sp < a.nsplit; ++sp) M = fmaxf(M, part[sp * kPartStride]);
  float L = 0.0f, o0 = 0.0f, o1 = 0.0f;
  for (int sp = 0; sp < a.nsplit; ++sp) {
    const float* p = part + sp * kPartStride;
    const float sc = (p[0] == -INFINITY) ? 0.0f : ex2_approx(p[0] - M);
    L += p[1] * sc;
    o0 += p[2 + 2 * lane] * sc;
    o1 += p[3 + 2 * lane] * sc;
  }
  const float inv = 1.0f / L;
  if (a.o_fp32) {
    reinterpret_cast<float2*>(static_cast<float*>(a.o) + off)[0] = make_float2(o0 * inv, o1 * inv);
  } else {
    reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.o) + off)[0] = pack_bf16x2(o0 * inv, o1 * inv);
  }
  if (a.lse && lane == 0) a.lse[bh] = (M + __log2f(L)) * kLn2f;
}

}  // namespace

void decode_split(int BH, int Tkv, int* nsplit, int* chunk) {
  // Aim for about 8 waves of 3 resident CTAs on 152 SMs; chunks are whole
  // 64-key stages.
  const int target = 152 * 3 * 8;
  const int max_split = (Tkv + 255) / 256;
  int ns = (target + BH - 1) / BH;
  if (ns > max_split) ns = max_split;
  if (ns < 1) ns = 1;
  int ch = (Tkv + ns - 1) / ns;
  ch = ((ch + kDecKeys - 1) / kDecKeys) * kDecKeys;
  *chunk = ch;
  *nsplit = (Tkv + ch - 1) / ch;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(DecSmem) + 128;
  static bool limit_set[64] = {};
  const cudaError_t e = smem_limit_once(bam_decode_kernel, smem, limit_set);
  if (e != cudaSuccess) return e;
  dim3 grid(a.nsplit, a.B * a.H);
  return launch_k(bam_decode_kernel, grid, dim3(kDecThreads), smem, st, true, a);
}

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t st) {
  const int BH = a.B * a.H;
  return launch_k(bam_decode_combine_kernel, dim3((BH + 3) / 4), dim3(128), 0, st, true, a);
}

}  // namespace bam
