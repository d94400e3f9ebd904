// Definitions shared by the kernels and the host entry points of the GGD-BAM
// attention library: workspace layout, distance-table geometry, kernel
// argument blocks and the internal launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bam_ptx.cuh"

namespace bam {

constexpr int kHeadDim = 64;
constexpr double kLog2e = 1.4426950408889634074;
constexpr float kLn2f = 0.69314718055994530942f;
// bam_params.prior value of the theta parameterisation (BAM_PRIOR_THETA).
constexpr int kPriorTheta = 1;

// Workspace: [0, 256) device status words, then op-specific regions, each
// 256-byte aligned.
constexpr size_t kStatusBytes = 256;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Per-head distance table (forward / backward): b_h(d) * log2(e) for every
// d that a tile window can touch, d = x - off for a table index x in
// [0, len).  In memory each row is stored reversed, in kTabCopies copies:
// entry y of copy k of head h holds index x = len - 1 - y + k (0 where that
// falls past the row).  A thread whose row meets key columns c, c+1, c+2,
// c+3 needs d, d-1, d-2, d-3, i.e. four consecutive reversed entries; in the
// copy k = (its row + 1) mod 4 they start on a 16-byte boundary, so one
// vector load fetches them.  Windows start at multiples of 128 entries.
constexpr int kTabCopies = 4;
// Window copies may read up to four entries past the end of a row (never
// used); the table region is padded so the last row stays inside it.
constexpr int kTabPadFloats = 16;

// Offset (floats) of window copy k in shared memory when copies are
// `stride` floats apart (stride a multiple of 32): extra shifts of 0, 4, 12
// and 20 floats spread the 16-byte loads of the eight lanes of each quarter
// warp over all 32 banks.
__host__ __device__ constexpr int win_copy_off(int k, int stride) {
  return k * stride + (k ? 8 * k - 4 : 0);
}

struct TableGeom {
  int off;  // index of d = 0
  int len;  // entries per head, multiple of 256
};

inline TableGeom table_geom(int T, int causal) {
  const int t256 = ((T + 255) / 256) * 256;
  const int off = causal ? 256 : t256 + 256;
  return TableGeom{off, off + t256 + 256};
}

// Decode table: entry j of head h holds b_h(Tkv - 1 - j) * log2(e) for the
// key at cache position j (0 beyond Tkv); rows padded to 64 entries.
// Entries of a decode table row: Tkv, plus room for the aligned 68-entry
// stage window of the last stage (ragged decode starts windows at any entry).
inline int decode_table_len(int Tkv) { return ((Tkv + 68 + 63) / 64) * 64; }

enum TableMode : int {
  kTableByDistance = 0,  // forward: b only
  kTableDecode = 1,      // decode: by key position
  kTableBackward = 2     // backward: b, db/dbeta, db/dmu (three tables)
};

struct TableArgs {
  float* tab;  // decode: [H][len]; by distance: [ntables][kTabCopies][H][len] reversed rows
  const float* alpha;
  const float* beta;
  const float* mu;
  DevStatus* status;  // the call's status words (status_begin_call in block 0)
  float eps;
  int H, len, off, Tkv, mode;
  int prior;  // BAM_PRIOR_ALPHA or BAM_PRIOR_THETA (alpha, beta, mu hold the thetas)
};

struct FwdArgs {
  void* o;
  float* lse;
  const float* table;
  const float* s;
  DevStatus* status;
  int B, H, T;
  int causal, ssmax, o_fp32;
  int tab_len, tab_off;
};

struct DecodeArgs {
  const uint16_t* q;   // [BH, 64]
  const uint16_t* kc;  // [BH, Tkv, 64]
  const uint16_t* vc;
  const int* lens;     // ragged decode: cache length of each sequence [B]; else null
  // Paged cache (block_table non-null): kc, vc are [num_pages, H, page, 64]
  // and logical block i of sequence b is page block_table[b * max_blocks + i].
  const int* block_table;
  int page, max_blocks, num_pages;
  const float* table;  // [H, tab_len]
  const float* s;
  float* part;         // [BH, nsplit, 2 + 64]: m (log2 units), l, o[64]
  void* o;
  float* lse;
  DevStatus* status;
  int B, H, Tkv, nsplit, chunk, tab_len;
  int ssmax, o_fp32;
};

struct BwdArgs {
  const void* o;        // forward output (fp32 or bf16)
  const uint16_t* dO;   // bf16
  const float* lse;     // natural-log LSE from the forward
  const float* table;   // [3][H][len]: b*log2e, db/dbeta, db/dmu
  const float* alpha;
  const float* beta;
  const float* s;
  float* delta;         // [BH, T]: rowsum(dO * O)
  float* dq_acc;        // [BH, T, 64] fp32
  float* rowacc;        // [BH, T, 8]: per row sum_j P*X for X = b, db/dbeta, db/dmu and
                        // ln(n) qk/sqrt(D), then sum_j P*dP
  uint16_t* dq;         // bf16 outputs
  uint16_t* dk;
  uint16_t* dv;
  float* dalpha;
  float* dbeta;
  float* dmu;
  float* ds;
  DevStatus* status;
  int B, H, T, nkb;
  int causal, ssmax, o_fp32;
  int tab_len, tab_off;
  TableArgs tab;        // the three distance tables, built by the preprocess
};

// Launch with an optional programmatic-dependent-launch attribute: the
// kernel may start while the previous kernel on the stream finishes, and must
// execute griddepcontrol.wait before touching anything that kernel writes.
// Only the second and later kernels of one entry point use it, so that two
// calls sharing a workspace never overlap.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Streaming multiprocessors of the current device (queried once per device).
inline int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (the attribute belongs to the device's context).
// `done` is the caller's per-kernel flag array.
template <typename F>
cudaError_t smem_limit_once(F* kernel, size_t bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < 64;
  if (cached && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e == cudaSuccess && cached) done[dev] = true;
  return e;
}

// Internal launchers (one per kernel).  Each returns the launch error.
cudaError_t launch_table(const TableArgs& a, cudaStream_t st);
// `to`: O in 128-row boxes (paired kernel); `to32`: O in 32-row boxes, one
// warp's rows (single-tile kernel).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& to32, const FwdArgs& a,
                       cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t st);
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t st);
cudaError_t launch_bwd_final(const BwdArgs& a, cudaStream_t st);

// Decode split geometry.
void decode_split(int BH, int Tkv, int* nsplit, int* chunk);

}  // namespace bam
