// C ABI of the GGD-BAM attention library (declarations and contracts in
// include/bam_attn.h): argument validation, workspace layout, TMA tensor-map
// encoding and kernel launches.  No allocation, no host fallback: every step
// of the computation runs in the kernels of this library.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/bam_attn.h"
#include "bam_common.cuh"

static_assert(BAM_PRIOR_THETA == bam::kPriorTheta, "prior codes of the ABI and the kernels");

namespace bam {
namespace {

std::atomic<uint64_t> g_launches{0};
std::mutex g_prof_mu;
cudaEvent_t g_prof_before[BAM_KERNEL_COUNT] = {};
cudaEvent_t g_prof_after[BAM_KERNEL_COUNT] = {};

// Runs `launch` bracketed by the instrumentation events of kernel `which`.
template <class F>
cudaError_t launch_kernel(int which, cudaStream_t st, F launch) {
  cudaEvent_t before = nullptr, after = nullptr;
  {
    std::lock_guard<std::mutex> g(g_prof_mu);
    before = g_prof_before[which];
    after = g_prof_after[which];
  }
  // Under stream capture the records are external, so that they become
  // event-record nodes of the graph (timestamps on every replay) rather than
  // internal dependencies.
  unsigned flags = cudaEventRecordDefault;
  if (before || after) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    if (cs == cudaStreamCaptureStatusActive) flags = cudaEventRecordExternal;
  }
  if (before) {
    cudaError_t e = cudaEventRecordWithFlags(before, st, flags);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch();
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return e;
  if (after) e = cudaEventRecordWithFlags(after, st, flags);
  return e;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [BH, T, 64] bf16 viewed as a 3-D tensor (64, T, BH); boxes of `rows` x 64
// (128 by default) with the 128-byte swizzle that the tcgen05 K-major /
// MN-major operands expect.  Rows past T inside a head read as zeros.
bool encode_rows(CUtensorMap* m, const void* base, int BH, int T, unsigned rows = 128) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                           static_cast<cuuint64_t>(T) * kHeadDim * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 [BH, T, 64] accumulator as a 3-D tensor (64, T, BH) in boxes of 32
// columns x `rows` (128 by default; 128-byte rows, 128-byte swizzle) for TMA
// reductions and stores.
bool encode_acc_rows(CUtensorMap* m, void* base, int BH, int T, unsigned rows = 128) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 4,
                           static_cast<cuuint64_t>(T) * kHeadDim * 4};
  cuuint32_t box[3] = {32, rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bam_status check_sizes(int B, int H, int T, int D) {
  if (B < 1 || H < 1 || T < 1 || D < 1) return BAM_ERR_INVALID_ARG;
  if (D != kHeadDim) return BAM_ERR_UNSUPPORTED;
  if (T > (1 << 28)) return BAM_ERR_UNSUPPORTED;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t nqb = (T + 255) / 256;
  if (BH > (1 << 24) || BH * nqb >= (int64_t(1) << 31)) return BAM_ERR_UNSUPPORTED;
  if (H > 65535) return BAM_ERR_UNSUPPORTED;
  return BAM_OK;
}

bam_status check_params(const bam_params* p) {
  if (!p || !p->alpha || !p->beta || !p->mu) return BAM_ERR_INVALID_ARG;
  if (p->ssmax && !p->s) return BAM_ERR_INVALID_ARG;
  if (!(p->eps > 0.0f) || !std::isfinite(p->eps)) return BAM_ERR_INVALID_ARG;
  if ((p->causal != 0 && p->causal != 1) || (p->ssmax != 0 && p->ssmax != 1))
    return BAM_ERR_INVALID_ARG;
  if (p->prior != BAM_PRIOR_ALPHA && p->prior != BAM_PRIOR_THETA) return BAM_ERR_INVALID_ARG;
  return BAM_OK;
}

// Workspace layouts.
struct FwdWs {
  size_t table, total;
};
FwdWs fwd_ws(int H, int T, int causal) {
  const TableGeom g = table_geom(T, causal);
  FwdWs w;
  w.table = kStatusBytes;
  w.total = w.table + align256((kTabCopies * static_cast<size_t>(H) * g.len + kTabPadFloats) * 4);
  return w;
}

struct BwdWs {
  size_t table, delta, dq_acc, rowacc, total;
};
BwdWs bwd_ws(int B, int H, int T, int causal) {
  const TableGeom g = table_geom(T, causal);
  const size_t BH = static_cast<size_t>(B) * H;
  BwdWs w;
  w.table = kStatusBytes;
  w.delta =
      w.table + align256((3 * kTabCopies * static_cast<size_t>(H) * g.len + kTabPadFloats) * 4);
  w.dq_acc = w.delta + align256(BH * T * 4);
  w.rowacc = w.dq_acc + align256(BH * T * kHeadDim * 4);
  w.total = w.rowacc + align256(BH * T * 8 * 4);
  return w;
}

struct DecWs {
  size_t table, part, total;
  int nsplit, chunk, tab_len;
};
DecWs dec_ws(int B, int H, int Tkv) {
  DecWs w;
  decode_split(B * H, Tkv, &w.nsplit, &w.chunk);
  w.tab_len = decode_table_len(Tkv);
  w.table = kStatusBytes;
  w.part = w.table + align256(static_cast<size_t>(H) * w.tab_len * 4);
  w.total = w.part + align256(static_cast<size_t>(B) * H * w.nsplit * (2 + kHeadDim) * 4);
  return w;
}

bam_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || !aligned(ws, 256) || ws_bytes < need) return BAM_ERR_WORKSPACE;
  return BAM_OK;
}

inline bam_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BAM_OK : BAM_ERR_CUDA; }

}  // namespace
}  // namespace bam

namespace bam {
// Lets entry points defined in other files count their launches.
void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }
}  // namespace bam

namespace bam {
namespace {

// bam_attn_decode and its ragged form (lens: device int32 [B], or null).
// Paged form: block_table non-null, kc/vc [num_pages, H, page, D], Tkv the
// longest sequence a block-table row can hold (max_blocks * page).
struct Paging {
  const int* block_table = nullptr;
  int page = 0, max_blocks = 0, num_pages = 0;
};

bam_status decode_impl(const void* q, const void* kc, const void* vc, const int* lens, void* o,
                       int o_fp32, float* lse, int B, int H, int Tkv, int D,
                       const bam_params* p, void* ws, size_t ws_bytes, cudaStream_t stream,
                       const Paging& pg = Paging()) {
  bam_status s = check_sizes(B, H, Tkv, D);
  if (s != BAM_OK) return s;
  if ((s = check_params(p)) != BAM_OK) return s;
  if (!q || !kc || !vc || !o) return BAM_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kc, 16) || !aligned(vc, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)))
    return BAM_ERR_INVALID_ARG;
  const DecWs w = dec_ws(B, H, Tkv);
  if ((s = check_ws(ws, ws_bytes, w.total)) != BAM_OK) return s;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  DevStatus* status = reinterpret_cast<DevStatus*>(wsb);
  float* table = reinterpret_cast<float*>(wsb + w.table);

  TableArgs ta{table, p->alpha, p->beta, p->mu, status, p->eps, H, w.tab_len, 0, Tkv,
               kTableDecode, p->prior};
  cudaError_t e = launch_kernel(BAM_KERNEL_TABLE, stream, [&] { return launch_table(ta, stream); });
  if (e != cudaSuccess) return BAM_ERR_CUDA;

  DecodeArgs da;
  da.q = static_cast<const uint16_t*>(q);
  da.kc = static_cast<const uint16_t*>(kc);
  da.vc = static_cast<const uint16_t*>(vc);
  da.lens = lens;
  da.block_table = pg.block_table;
  da.page = pg.page;
  da.max_blocks = pg.max_blocks;
  da.num_pages = pg.num_pages;
  da.table = table;
  da.s = p->s;
  da.part = reinterpret_cast<float*>(wsb + w.part);
  da.o = o;
  da.lse = lse;
  da.status = status;
  da.B = B;
  da.H = H;
  da.Tkv = Tkv;
  da.nsplit = w.nsplit;
  da.chunk = w.chunk;
  da.tab_len = w.tab_len;
  da.ssmax = p->ssmax;
  da.o_fp32 = o_fp32 ? 1 : 0;
  e = launch_kernel(BAM_KERNEL_DECODE, stream, [&] { return launch_decode(da, stream); });
  if (e != cudaSuccess) return BAM_ERR_CUDA;
  e = launch_kernel(BAM_KERNEL_DECODE_COMBINE, stream,
                    [&] { return launch_decode_combine(da, stream); });
  return cuda_status(e);
}

}  // namespace

// For bam_attn_decode_noalloc (decode_noalloc.cu): the argument checks, the
// scratch size and the launches of bam_attn_decode, on caller-given scratch.
bam_status decode_args_ok(const void* q, const void* kc, const void* vc, void* o, float* lse,
                          int B, int H, int Tkv, int D, const bam_params* p) {
  bam_status s = check_sizes(B, H, Tkv, D);
  if (s != BAM_OK) return s;
  if ((s = check_params(p)) != BAM_OK) return s;
  if (!q || !kc || !vc || !o) return BAM_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kc, 16) || !aligned(vc, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)))
    return BAM_ERR_INVALID_ARG;
  return BAM_OK;
}
size_t decode_scratch_bytes(int B, int H, int Tkv) { return dec_ws(B, H, Tkv).total; }
bam_status decode_plain(const void* q, const void* kc, const void* vc, void* o, int o_fp32,
                        float* lse, int B, int H, int Tkv, int D, const bam_params* p,
                        void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  return decode_impl(q, kc, vc, nullptr, o, o_fp32, lse, B, H, Tkv, D, p, scratch, scratch_bytes,
                     stream);
}
// Reads and clears the status words at `st` (device memory) after
// synchronising `stream`; the sticky-error rules of bam_attn_check_status.
bam_status read_and_clear_status(void* st_dev, cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BAM_ERR_CUDA;
  DevStatus st;
  if (cudaMemcpy(&st, st_dev, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return BAM_ERR_CUDA;
  // A status area no call has initialised holds no error.
  if (st.magic[0] != kStatusMagic0 || st.magic[1] != kStatusMagic1) return BAM_OK;
  // Clears abort, code, site and block; the magic and the debug count stay.
  if (cudaMemset(st_dev, 0, 4 * sizeof(int)) != cudaSuccess) return BAM_ERR_CUDA;
  if (st.code == BAM_DEV_BAD_ARG && st.abort == 0) return BAM_ERR_INVALID_ARG;
  if (st.code == BAM_DEV_BOUNDS) return BAM_ERR_BOUNDS;
  if (st.code != BAM_DEV_OK || st.abort != 0) return BAM_ERR_TIMEOUT;
  return BAM_OK;
}
// Debug builds: arms the give-up count of the status words at `st_dev`.
bam_status arm_giveup(void* st_dev, int n) {
#ifdef BAM_DEBUG
  DevStatus st;
  if (cudaDeviceSynchronize() != cudaSuccess) return BAM_ERR_CUDA;
  if (cudaMemcpy(&st, st_dev, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return BAM_ERR_CUDA;
  if (st.magic[0] != kStatusMagic0 || st.magic[1] != kStatusMagic1) {
    std::memset(&st, 0, sizeof(st));
    st.magic[0] = kStatusMagic0;
    st.magic[1] = kStatusMagic1;
  }
  st.giveup = n;
  if (cudaMemcpy(st_dev, &st, sizeof(st), cudaMemcpyHostToDevice) != cudaSuccess)
    return BAM_ERR_CUDA;
  return BAM_OK;
#else
  (void)st_dev;
  (void)n;
  return BAM_ERR_UNSUPPORTED;
#endif
}
}  // namespace bam

using namespace bam;

extern "C" {

size_t bam_attn_workspace_size(int op, int B, int H, int T, int D) {
  if (check_sizes(B, H, T, D) != BAM_OK) return 0;
  switch (op) {
    case BAM_OP_FWD:
      // the larger of the causal and non-causal layouts
      return fwd_ws(H, T, 0).total;
    case BAM_OP_BWD:
      return bwd_ws(B, H, T, 0).total;
    case BAM_OP_DECODE:
      return dec_ws(B, H, T).total;
    default:
      return 0;
  }
}

bam_status bam_attn_fwd(const void* q, const void* k, const void* v, void* o, int o_fp32,
                        float* lse, int B, int H, int T, int D, const bam_params* p, void* ws,
                        size_t ws_bytes, cudaStream_t stream) {
  bam_status s = check_sizes(B, H, T, D);
  if (s != BAM_OK) return s;
  if ((s = check_params(p)) != BAM_OK) return s;
  if (!q || !k || !v || !o) return BAM_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)))
    return BAM_ERR_INVALID_ARG;
  const FwdWs w = fwd_ws(H, T, p->causal);
  if ((s = check_ws(ws, ws_bytes, w.total)) != BAM_OK) return s;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!encode_rows(&tq, q, BH, T) || !encode_rows(&tk, k, BH, T) || !encode_rows(&tv, v, BH, T))
    return BAM_ERR_CUDA;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  DevStatus* status = reinterpret_cast<DevStatus*>(wsb);
  float* table = reinterpret_cast<float*>(wsb + w.table);
  const TableGeom g = table_geom(T, p->causal);

  TableArgs ta{table, p->alpha, p->beta, p->mu, status, p->eps, H, g.len, g.off, 0,
               kTableByDistance, p->prior};
  cudaError_t e = launch_kernel(BAM_KERNEL_TABLE, stream, [&] { return launch_table(ta, stream); });
  if (e != cudaSuccess) return BAM_ERR_CUDA;

  FwdArgs fa;
  fa.o = o;
  fa.lse = lse;
  fa.table = table;
  fa.s = p->s;
  fa.status = status;
  fa.B = B;
  fa.H = H;
  fa.T = T;
  fa.causal = p->causal;
  fa.ssmax = p->ssmax;
  fa.o_fp32 = o_fp32 ? 1 : 0;
  fa.tab_len = g.len;
  fa.tab_off = g.off;
  // O by TMA stores: fp32 in 32-column boxes, bf16 in 64-column boxes; 128
  // rows a box for the paired kernel, 32 (one warp's rows) for the
  // single-tile kernel.
  CUtensorMap to, to32;
  if (!(o_fp32 ? encode_acc_rows(&to, o, BH, T) : encode_rows(&to, o, BH, T)) ||
      !(o_fp32 ? encode_acc_rows(&to32, o, BH, T, 32) : encode_rows(&to32, o, BH, T, 32)))
    return BAM_ERR_CUDA;
  e = launch_kernel(BAM_KERNEL_FWD, stream,
                    [&] { return launch_fwd(tq, tk, tv, to, to32, fa, stream); });
  return cuda_status(e);
}

bam_status bam_attn_decode(const void* q, const void* kc, const void* vc, void* o, int o_fp32,
                           float* lse, int B, int H, int Tkv, int D, const bam_params* p,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
  return decode_impl(q, kc, vc, nullptr, o, o_fp32, lse, B, H, Tkv, D, p, ws, ws_bytes, stream);
}

bam_status bam_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                 const int* block_table, const int* cache_lens, void* o,
                                 int o_fp32, float* lse, int B, int H, int page, int max_blocks,
                                 int num_pages, int D, const bam_params* p, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  if (!block_table || !aligned(block_table, 4) || !cache_lens || !aligned(cache_lens, 4))
    return BAM_ERR_INVALID_ARG;
  if (page < 64 || page % 64 != 0 || max_blocks < 1 || num_pages < 1) return BAM_ERR_INVALID_ARG;
  const int64_t tmax = static_cast<int64_t>(page) * max_blocks;
  if (tmax > (1 << 28)) return BAM_ERR_UNSUPPORTED;
  Paging pg;
  pg.block_table = block_table;
  pg.page = page;
  pg.max_blocks = max_blocks;
  pg.num_pages = num_pages;
  return decode_impl(q, k_pages, v_pages, cache_lens, o, o_fp32, lse, B, H,
                     static_cast<int>(tmax), D, p, ws, ws_bytes, stream, pg);
}

bam_status bam_attn_decode_varlen(const void* q, const void* kc, const void* vc,
                                  const int* cache_lens, void* o, int o_fp32, float* lse, int B,
                                  int H, int Tmax, int D, const bam_params* p, void* ws,
                                  size_t ws_bytes, cudaStream_t stream) {
  if (!cache_lens || !aligned(cache_lens, 4)) return BAM_ERR_INVALID_ARG;
  return decode_impl(q, kc, vc, cache_lens, o, o_fp32, lse, B, H, Tmax, D, p, ws, ws_bytes,
                     stream);
}

bam_status bam_attn_bwd(const void* q, const void* k, const void* v, const void* o, int o_fp32,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv,
                        float* dalpha, float* dbeta, float* dmu, float* ds, int B, int H, int T,
                        int D, const bam_params* p, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  bam_status s = check_sizes(B, H, T, D);
  if (s != BAM_OK) return s;
  if ((s = check_params(p)) != BAM_OK) return s;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !dalpha || !dbeta || !dmu ||
      !ds)
    return BAM_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dO, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 16))
    return BAM_ERR_INVALID_ARG;
  const BwdWs w = bwd_ws(B, H, T, p->causal);
  if ((s = check_ws(ws, ws_bytes, w.total)) != BAM_OK) return s;
  const int BH = B * H;
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_rows(&tq, q, BH, T) || !encode_rows(&tk, k, BH, T) ||
      !encode_rows(&tv, v, BH, T) || !encode_rows(&tdo, dO, BH, T))
    return BAM_ERR_CUDA;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  DevStatus* status = reinterpret_cast<DevStatus*>(wsb);
  float* table = reinterpret_cast<float*>(wsb + w.table);
  const TableGeom g = table_geom(T, p->causal);

  BwdArgs ba;
  ba.tab = TableArgs{table, p->alpha, p->beta, p->mu, status, p->eps, H, g.len, g.off, 0,
                     kTableBackward, p->prior};
  ba.o = o;
  ba.dO = static_cast<const uint16_t*>(dO);
  ba.lse = lse;
  ba.table = table;
  ba.alpha = p->alpha;
  ba.beta = p->beta;
  ba.s = p->s;
  ba.delta = reinterpret_cast<float*>(wsb + w.delta);
  ba.dq_acc = reinterpret_cast<float*>(wsb + w.dq_acc);
  ba.rowacc = reinterpret_cast<float*>(wsb + w.rowacc);
  ba.dq = static_cast<uint16_t*>(dq);
  ba.dk = static_cast<uint16_t*>(dk);
  ba.dv = static_cast<uint16_t*>(dv);
  ba.dalpha = dalpha;
  ba.dbeta = dbeta;
  ba.dmu = dmu;
  ba.ds = ds;
  ba.status = status;
  ba.B = B;
  ba.H = H;
  ba.T = T;
  ba.nkb = (T + 127) / 128;
  ba.causal = p->causal;
  ba.ssmax = p->ssmax;
  ba.o_fp32 = o_fp32 ? 1 : 0;
  ba.tab_len = g.len;
  ba.tab_off = g.off;
  cudaError_t e =
      launch_kernel(BAM_KERNEL_BWD_PREP, stream, [&] { return launch_bwd_prep(ba, stream); });
  if (e != cudaSuccess) return BAM_ERR_CUDA;
  CUtensorMap tdq, tdk, tdv;
  if (!encode_acc_rows(&tdq, ba.dq_acc, BH, T) || !encode_rows(&tdk, dk, BH, T) ||
      !encode_rows(&tdv, dv, BH, T))
    return BAM_ERR_CUDA;
  e = launch_kernel(BAM_KERNEL_BWD, stream,
                    [&] { return launch_bwd(tq, tk, tv, tdo, tdq, tdk, tdv, ba, stream); });
  if (e != cudaSuccess) return BAM_ERR_CUDA;
  e = launch_kernel(BAM_KERNEL_BWD_FINAL, stream, [&] { return launch_bwd_final(ba, stream); });
  return cuda_status(e);
}

bam_status bam_attn_check_status(void* ws, cudaStream_t stream) {
  if (!ws || !aligned(ws, 256)) return BAM_ERR_WORKSPACE;
  return read_and_clear_status(ws, stream);
}

bam_status bam_attn_debug_arm_giveup(void* ws, int n) {
  if (n < 0) return BAM_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return BAM_ERR_WORKSPACE;
  return arm_giveup(ws, n);
}

int bam_attn_debug_build(void) {
#ifdef BAM_DEBUG
  return 1;
#else
  return 0;
#endif
}

const char* bam_status_string(bam_status s) {
  switch (s) {
    case BAM_OK:
      return "ok";
    case BAM_ERR_INVALID_ARG:
      return "invalid argument";
    case BAM_ERR_UNSUPPORTED:
      return "unsupported size or option";
    case BAM_ERR_CUDA:
      return "CUDA error";
    case BAM_ERR_TIMEOUT:
      return "device-side wait gave up";
    case BAM_ERR_WORKSPACE:
      return "workspace missing, misaligned or too small";
    case BAM_ERR_BOUNDS:
      return "a bulk copy failed its bounds check (debug build)";
  }
  return "unknown status";
}

bam_status bam_attn_profile_events(int which, cudaEvent_t before, cudaEvent_t after) {
  if (which < 0 || which >= BAM_KERNEL_COUNT) return BAM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_prof_mu);
  g_prof_before[which] = before;
  g_prof_after[which] = after;
  return BAM_OK;
}

uint64_t bam_attn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
