// Decode without a caller workspace (bam_attn_decode_noalloc).
//
// Some callers cannot call cudaMalloc: plugin-style hosts (inference servers,
// framework extension points) hand a library only its input and output
// pointers and own every other byte of device memory through their own
// allocator, and cudaMalloc itself may synchronise the device, which a
// per-token decode loop cannot afford.  This entry point runs the same split-
// KV decode as bam_attn_decode (same table, decode and combine kernels) but
// takes its scratch from a fixed array in the library's device image instead
// of a workspace argument.  It allocates nothing.
//
// The array is `static __device__`: every GPU that loads the library holds
// kNoAllocScratchBytes of it until the process exits.  In host code the
// array's name is only a host-side stand-in, so the device address is looked
// up with cudaGetSymbolAddress, once per device, with that device current;
// the first call on each device does this set-up (make that first call
// before any stream capture on the device).  All calls share the array and it
// keeps the last call's contents: the table and every partial are fully
// rewritten by each call and the status word is cleared by the table kernel,
// so nothing else has to start at zero; calls that overlap on the GPU (for
// example on two streams) race on it.
#include <mutex>

#include "../../include/bam_attn.h"
#include "bam_common.cuh"

namespace bam {

// Launch counter of the library (defined with the other entry points).
void note_launches(int n);

namespace {

constexpr size_t kNoAllocScratchBytes = BAM_DECODE_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    if (!p || (reinterpret_cast<uintptr_t>(p) & 255) != 0) return cudaErrorInvalidValue;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace bam

using namespace bam;

extern "C" bam_status bam_attn_decode_noalloc(const void* q, const void* kc, const void* vc,
                                              void* o, int o_fp32, float* lse, int B, int H,
                                              int Tkv, int D, const bam_params* p,
                                              cudaStream_t stream) {
  if (B < 1 || H < 1 || Tkv < 1 || D < 1) return BAM_ERR_INVALID_ARG;
  if (D != kHeadDim) return BAM_ERR_UNSUPPORTED;
  if (Tkv > (1 << 28) || H > 65535 || static_cast<int64_t>(B) * H > (1 << 24))
    return BAM_ERR_UNSUPPORTED;
  if (!p || !p->alpha || !p->beta || !p->mu || (p->ssmax && !p->s)) return BAM_ERR_INVALID_ARG;
  if (!(p->eps > 0.0f) || !(p->eps < 3.0e38f)) return BAM_ERR_INVALID_ARG;
  if (p->ssmax != 0 && p->ssmax != 1) return BAM_ERR_INVALID_ARG;
  if (p->prior != BAM_PRIOR_ALPHA && p->prior != BAM_PRIOR_THETA) return BAM_ERR_INVALID_ARG;
  if (!q || !kc || !vc || !o) return BAM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3) != 0))
    return BAM_ERR_INVALID_ARG;

  // Scratch layout (same as the workspace of bam_attn_decode): status words,
  // the decode table, the split partials.
  int nsplit = 0, chunk = 0;
  decode_split(B * H, Tkv, &nsplit, &chunk);
  const int tab_len = decode_table_len(Tkv);
  const size_t table_off = kStatusBytes;
  const size_t part_off = table_off + align256(static_cast<size_t>(H) * tab_len * 4);
  const size_t need =
      part_off + align256(static_cast<size_t>(B) * H * nsplit * (2 + kHeadDim) * 4);
  if (need > kNoAllocScratchBytes) return BAM_ERR_WORKSPACE;

  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return BAM_ERR_CUDA;
  uint8_t* wsb = static_cast<uint8_t*>(scratch);
  DevStatus* status = reinterpret_cast<DevStatus*>(wsb);
  float* table = reinterpret_cast<float*>(wsb + table_off);

  TableArgs ta{table, p->alpha, p->beta, p->mu, status, p->eps, H, tab_len, 0, Tkv,
               kTableDecode, p->prior};
  cudaError_t e = launch_table(ta, stream);
  note_launches(1);
  if (e != cudaSuccess) return BAM_ERR_CUDA;

  DecodeArgs da;
  da.q = static_cast<const uint16_t*>(q);
  da.kc = static_cast<const uint16_t*>(kc);
  da.vc = static_cast<const uint16_t*>(vc);
  da.lens = nullptr;
  da.block_table = nullptr;
  da.page = da.max_blocks = da.num_pages = 0;
  da.table = table;
  da.s = p->s;
  da.part = reinterpret_cast<float*>(wsb + part_off);
  da.o = o;
  da.lse = lse;
  da.status = status;
  da.B = B;
  da.H = H;
  da.Tkv = Tkv;
  da.nsplit = nsplit;
  da.chunk = chunk;
  da.tab_len = tab_len;
  da.ssmax = p->ssmax;
  da.o_fp32 = o_fp32 ? 1 : 0;
  e = launch_decode(da, stream);
  note_launches(1);
  if (e != cudaSuccess) return BAM_ERR_CUDA;
  e = launch_decode_combine(da, stream);
  note_launches(1);
  return e == cudaSuccess ? BAM_OK : BAM_ERR_CUDA;
}
