// qmv_internal.cuh -- declarations shared by the library's translation units.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "qmv.h"
#include "qmv_decode.cuh"

#define QMV_PACK_MAGIC 0x514D5650u

struct qmv_pack {
  uint32_t magic;
  int N, K, bits, group;
  int G;                      // scales per row: K / group
  size_t codes_bytes, scales_bytes;
  const uint32_t* d_codes;    // bound by qmv_pack_weights
  const uint16_t* d_scales;
  int bound;
};

namespace qmv {

// Arguments of one matvec launch (all device pointers).
struct GemvArgs {
  const uint4* codes;         // [N][row_u4] 16-byte units
  const __half* scales;       // [N][G]
  int N, K, G, row_u4;        // G = scales per row
  int perrow;                 // one scale per row (group == K)
  const __half* x;            // [M][K] activations (the normalised input when fused)
  const __half* r;            // [M][K] residual (fused only)
  const __half* gamma;        // [K] (fused only)
  float eps;
  __half* h_out;              // [M][K] nullable (fused only)
  void* y;                    // [M][N] fp32 or fp16
  int y_f16;
  int M;                      // columns (tokens)
  int fused;
  int folded;                 // fast mode's folded-offset form (see qmv_decode.cuh)
  // fused argmax epilogue (M = 1 pipeline only; null when off): workspace
  // {u64 key, u32 CTA count} (zero before a launch, left zero after it) and
  // the outputs
  unsigned long long* amax_ws;
  int* amax_index;
  float* amax_value;
  // expert gather (M = 1 pipeline only; gather_rows == 0 when off): the pack
  // holds gather_E experts of gather_rows rows each; output block j (rows
  // j*gather_rows ..) is expert gather_ids[j], j < gather_n
  const int* gather_ids;
  int gather_rows, gather_n, gather_E;
  // the caller's device scratch (256-byte aligned, ws_bytes long, nullable):
  // the tensor tiles' split-K partial tiles, or the fused prologue's
  // normalised activations for M >= 2 (workspace_bytes says how much)
  void* ws;
  size_t ws_bytes;
};

struct DevInfo {
  int sms;
  int max_smem_optin;
};
const DevInfo& dev_info();   // of the current device (cached)

cudaError_t launch_pack(int bits, const int8_t* in, uint32_t* out, int64_t nwords, cudaStream_t s);
cudaError_t launch_unpack(int bits, const uint32_t* in, int8_t* out, int64_t nwords, cudaStream_t s);

// Return a qmv_status; on QMV_ERR_CUDA, *err holds the CUDA error.
int launch_gemv_m1(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err);
int launch_gemm_small(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err);
// M = 1 through the bulk-copy pipeline; QMV_ERR_UNSUPPORTED if the shape does
// not fit it (the caller then uses launch_gemv_m1).
int launch_gemv_tma(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err);
// Whether the pipeline has a plan for this K (the fast mode's folded form is
// used by the M = 1 pipeline and the M-column tiles exactly when it does).
bool tma_fits(int K, int bits, bool perrow);
// tcgen05 tensor-core tiles for 1..128 token columns, int2 weights (fast
// mode); QMV_ERR_UNSUPPORTED for other widths or the fused prologue.
int launch_tc_gemm(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err);
// Scratch bytes launch_tc_gemm needs for up to 128 columns of M (split-K
// partial tiles; 0 when it needs none).
size_t tc_workspace_bytes(int M, int N, int K, bool y_f16);
// Scratch bytes launch_mtile needs: the segment tables of the M columns
// (per 512 codes, 8960 bytes per 4 columns or 17408 per 8, as the tile shape
// chosen for N, M, K and bits has them), with or without the fused prologue;
// 0 where it does not run (M < 2, K not a multiple of 256).
size_t mt_workspace_bytes(int M, int N, int K, int bits, bool fused);
// Programmatic dependent launch of the M = 1 kernels (off by default).
bool pdl_enabled();
void set_pdl(bool on);
// Read (and optionally clear) the device error word set by bounded waits.
int read_device_error(int clear, int* out);
// Record a CUDA error as the calling thread's last one; returns QMV_ERR_CUDA.
int record_cuda_error(cudaError_t e);
// M-column tiles on paired fp32 arithmetic (K a multiple of 64, M <= 32);
// QMV_ERR_UNSUPPORTED when the shape does not fit them.
int launch_tile(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err);
// M-column tiles on the bulk-copy pipeline (any M >= 2, K a multiple of 256,
// with or without the fused prologue), every column equal to the M = 1
// result, on a.ws of at least mt_workspace_bytes (QMV_ERR_WORKSPACE
// otherwise); QMV_ERR_UNSUPPORTED when the shape does not fit them.
int launch_mtile(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err);


// Per-kernel launch facts, cached per device: the dynamic shared-memory limit
// set so far and the occupancy for one (threads, smem) shape.  This keeps the
// host cost of a call to a few lookups after the first call.
struct KernCache {
  int dev = -1;
  size_t smem_set = 48 * 1024;
  int occ_threads = -1;
  size_t occ_smem = 0;
  int occ = 0;
};

template <typename Kern>
inline cudaError_t prep_kernel(Kern k, KernCache& c, int threads, size_t smem, int* occ) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (c.dev != dev) {
    c = KernCache();
    c.dev = dev;
  }
  if (smem > c.smem_set) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    c.smem_set = smem;
  }
  if (occ) {
    if (c.occ_threads != threads || c.occ_smem != smem) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c.occ, k, threads, smem);
      if (e != cudaSuccess) return e;
      c.occ_threads = threads;
      c.occ_smem = smem;
    }
    *occ = c.occ;
  }
  return cudaSuccess;
}

}  // namespace qmv
