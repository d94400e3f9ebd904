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
// rewritten by each call, and the status words at its start follow the
// workspace rules (the first kernel of a call clears the abort word; an
// error stays until bam_attn_decode_noalloc_check_status reads it), so
// nothing has to start at zero; calls that overlap on the GPU (for example on
// two streams) race on it.
//
// Argument checks, scratch layout and launches are those of bam_attn_decode
// (api.cu), on the array instead of a workspace.
#include <mutex>

#include "../../include/bam_attn.h"
#include "bam_common.cuh"

namespace bam {

// The decode path of bam_attn_decode (api.cu).
bam_status decode_args_ok(const void* q, const void* kc, const void* vc, void* o, float* lse,
                          int B, int H, int Tkv, int D, const bam_params* p);
size_t decode_scratch_bytes(int B, int H, int Tkv);
bam_status decode_plain(const void* q, const void* kc, const void* vc, void* o, int o_fp32,
                        float* lse, int B, int H, int Tkv, int D, const bam_params* p,
                        void* scratch, size_t scratch_bytes, cudaStream_t stream);
bam_status read_and_clear_status(void* st_dev, cudaStream_t stream);
bam_status arm_giveup(void* st_dev, int n);

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

}  // namespace
}  // namespace bam

using namespace bam;

extern "C" bam_status bam_attn_decode_noalloc(const void* q, const void* kc, const void* vc,
                                              void* o, int o_fp32, float* lse, int B, int H,
                                              int Tkv, int D, const bam_params* p,
                                              cudaStream_t stream) {
  // Every refusal comes before the array's address is looked up.
  bam_status s = decode_args_ok(q, kc, vc, o, lse, B, H, Tkv, D, p);
  if (s != BAM_OK) return s;
  if (decode_scratch_bytes(B, H, Tkv) > kNoAllocScratchBytes) return BAM_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return BAM_ERR_CUDA;
  return decode_plain(q, kc, vc, o, o_fp32, lse, B, H, Tkv, D, p, scratch, kNoAllocScratchBytes,
                      stream);
}

extern "C" bam_status bam_attn_decode_noalloc_check_status(cudaStream_t stream) {
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return BAM_ERR_CUDA;
  return read_and_clear_status(scratch, stream);
}

extern "C" bam_status bam_attn_debug_arm_giveup_noalloc(int n) {
  if (n < 0) return BAM_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return BAM_ERR_CUDA;
  return arm_giveup(scratch, n);
}
