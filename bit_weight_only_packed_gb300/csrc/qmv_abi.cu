// qmv_abi.cu -- the C ABI declared in include/qmv.h: argument validation on
// the host, pack descriptors, and dispatch to the kernels.  Nothing here
// computes on the host: every step of the matvec runs in the kernels.
#include <new>

#include "qmv_pipe.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return QMV_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool pack_ok(const qmv_pack* p) { return p && p->magic == QMV_PACK_MAGIC; }

bool shape_ok(int K, int bits) {
  if (K < 32 || K % 32 != 0) return false;
  return ((int64_t)K * bits) % 128 == 0;   // a row is a whole number of 16-byte units
}

}  // namespace

namespace qmv {

int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

static thread_local bool g_pdl = false;
bool pdl_enabled() { return g_pdl; }
void set_pdl(bool on) { g_pdl = on; }

const DevInfo& dev_info() {
  static thread_local int cached_dev = -1;
  static thread_local DevInfo info{152, 227 * 1024};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return info;
  if (dev != cached_dev) {
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
      info.sms = sms;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
        smem > 0)
      info.max_smem_optin = smem;
    cached_dev = dev;
  }
  return info;
}

}  // namespace qmv

extern "C" {

int qmv_create_pack(qmv_pack** out, int N, int K, int bits, int group, size_t* codes_bytes,
                    size_t* scales_bytes) {
  if (!out) return QMV_ERR_INVALID_ARG;
  *out = nullptr;
  if (bits != 2 && bits != 4 && bits != 8) return QMV_ERR_INVALID_ARG;
  if (N < 1 || !shape_ok(K, bits)) return QMV_ERR_SHAPE;
  if (group != 32 && group != K) return QMV_ERR_INVALID_ARG;
  qmv_pack* p = new (std::nothrow) qmv_pack;
  if (!p) return QMV_ERR_INVALID_ARG;
  memset(p, 0, sizeof(*p));
  p->magic = QMV_PACK_MAGIC;
  p->N = N;
  p->K = K;
  p->bits = bits;
  p->group = group;
  p->G = K / group;
  p->codes_bytes = (size_t)N * (size_t)K * (size_t)bits / 8;
  p->scales_bytes = (size_t)N * (size_t)p->G * 2;
  if (codes_bytes) *codes_bytes = p->codes_bytes;
  if (scales_bytes) *scales_bytes = p->scales_bytes;
  *out = p;
  return QMV_OK;
}

int qmv_pack_weights(qmv_pack* p, const int8_t* d_codes_in, const uint16_t* d_scales_in,
                     void* d_codes, void* d_scales, void* stream) {
  if (!pack_ok(p) || !d_codes_in || !d_scales_in || !d_codes || !d_scales)
    return QMV_ERR_INVALID_ARG;
  if (!aligned(d_codes_in, 16) || !aligned(d_codes, 16) || !aligned(d_scales, 16) ||
      !aligned(d_scales_in, 2))
    return QMV_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t nwords = (int64_t)p->codes_bytes / 4;
  cudaError_t e = qmv::launch_pack(p->bits, d_codes_in, (uint32_t*)d_codes, nwords, s);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpyAsync(d_scales, d_scales_in, p->scales_bytes, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e);
  p->d_codes = (const uint32_t*)d_codes;
  p->d_scales = (const uint16_t*)d_scales;
  p->bound = 1;
  return QMV_OK;
}

static int check_common(const qmv_pack* p, int M, const void* x, void* y, int y_dtype, int mode) {
  if (!pack_ok(p) || !x || !y) return QMV_ERR_INVALID_ARG;
  if (!p->bound) return QMV_ERR_INVALID_ARG;
  if (M < 1 || M > 4096) return QMV_ERR_INVALID_ARG;
  if (y_dtype != QMV_F32 && y_dtype != QMV_F16) return QMV_ERR_INVALID_ARG;
  if (mode != QMV_FAST && mode != QMV_EXACT) return QMV_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 4)) return QMV_ERR_ALIGNMENT;
  return QMV_OK;
}

static size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

// The scratch of a call, following run_cuda_core's dispatch: the tensor
// tiles' split-K partials (M > 32, fast mode, int2, no prologue), else the
// pipelined M-column tiles' segment tables and the fused prologue's
// activations (M >= 2, K % 256 == 0); nothing for M = 1 or for the 32-column
// tiles that take K not a multiple of 256.
static size_t workspace_need(const qmv_pack* p, int M, int y_dtype, int mode, int fused) {
  if (M < 2 || M > 4096 || p->K % 256 != 0) return 0;
  if (!fused && M > 32 && mode == QMV_FAST && p->bits == 2)
    return round256(qmv::tc_workspace_bytes(M, p->N, p->K, y_dtype == QMV_F16));
  return qmv::mt_workspace_bytes(M, p->N, p->K, p->bits, fused != 0);
}

static int check_workspace(const qmv_pack* p, int M, int y_dtype, int mode, int fused, void* ws,
                           size_t ws_bytes) {
  if (ws && !aligned(ws, 256)) return QMV_ERR_ALIGNMENT;
  const size_t need = workspace_need(p, M, y_dtype, mode, fused);
  if (need && (!ws || ws_bytes < need)) return QMV_ERR_WORKSPACE;
  return QMV_OK;
}

static qmv::GemvArgs base_args(const qmv_pack* p, int M, const void* x, void* y, int y_dtype) {
  qmv::GemvArgs a;
  memset(&a, 0, sizeof(a));
  a.codes = (const uint4*)p->d_codes;
  a.scales = (const __half*)p->d_scales;
  a.N = p->N;
  a.K = p->K;
  a.G = p->G;
  a.row_u4 = (int)((int64_t)p->K * p->bits / 128);
  a.perrow = (p->group == p->K && p->K != 32) ? 1 : 0;
  a.x = (const __half*)x;
  a.y = y;
  a.y_f16 = (y_dtype == QMV_F16);
  a.M = M;
  return a;
}

// Dispatch: M = 1 -> the bulk-copy pipeline kernel (or the generic one);
// M > 32 in fast mode with int2 weights -> tcgen05 tensor-core tiles, 128
// columns per launch; every other M >= 2 -> CUDA-core M-column tiles, each
// column equal to the M = 1 result: the pipelined tiles in one launch where
// they fit (K a multiple of 256, no fused prologue), else 32 columns per
// launch.
static int run_cuda_core(qmv::GemvArgs a, int bits, cudaStream_t s, int mode) {
  cudaError_t err = cudaSuccess;
  int rc;
  // fast mode: the folded-offset form, in the M = 1 pipeline and the
  // M-column tiles alike, for the shapes the pipeline runs (elsewhere both
  // keep the exact form, so a tile column always equals the M = 1 result)
  a.folded = (mode == QMV_FAST && qmv::tma_fits(a.K, bits, a.perrow != 0)) ? 1 : 0;
  if (a.M > 32 && mode == QMV_FAST && bits == 2 && !a.fused) {
    const int M = a.M;
    const size_t ysz = a.y_f16 ? 2 : 4;
    bool done = true;
    for (int m0 = 0; m0 < M; m0 += 128) {
      qmv::GemvArgs b = a;
      b.M = (M - m0 < 128) ? (M - m0) : 128;
      b.x = a.x + (int64_t)m0 * a.K;
      b.y = (char*)a.y + (size_t)m0 * (size_t)a.N * ysz;
      rc = qmv::launch_tc_gemm(b, bits, s, &err);
      if (rc == QMV_ERR_UNSUPPORTED && m0 == 0) {   // shape outside the tensor tiles:
        done = false;                                // the exact CUDA-core tiles below
        break;
      }
      if (rc != QMV_OK) return rc == QMV_ERR_CUDA ? cuda_fail(err) : rc;
    }
    if (done) return QMV_OK;
  }
  if (a.M == 1) {
    rc = qmv::launch_gemv_tma(a, bits, s, &err);
    if (rc == QMV_ERR_UNSUPPORTED) rc = qmv::launch_gemv_m1(a, bits, s, &err);
    return rc == QMV_ERR_CUDA ? cuda_fail(err) : rc;
  }
  rc = qmv::launch_mtile(a, bits, s, &err);
  if (rc != QMV_ERR_UNSUPPORTED) return rc == QMV_ERR_CUDA ? cuda_fail(err) : rc;
  const int M = a.M;
  const size_t ysz = a.y_f16 ? 2 : 4;
  for (int m0 = 0; m0 < M; m0 += 32) {
    qmv::GemvArgs b = a;
    b.M = (M - m0 < 32) ? (M - m0) : 32;
    b.x = a.x + (int64_t)m0 * a.K;
    if (a.r) b.r = a.r + (int64_t)m0 * a.K;
    if (a.h_out) b.h_out = a.h_out + (int64_t)m0 * a.K;
    b.y = (char*)a.y + (size_t)m0 * (size_t)a.N * ysz;
    rc = qmv::launch_gemm_small(b, bits, s, &err);
    if (rc != QMV_OK) return rc == QMV_ERR_CUDA ? cuda_fail(err) : rc;
  }
  return QMV_OK;
}

size_t qmv_workspace_bytes(const qmv_pack* p, int M, int y_dtype, int mode, int fused) {
  if (!pack_ok(p) || (y_dtype != QMV_F32 && y_dtype != QMV_F16) || (mode != QMV_FAST && mode != QMV_EXACT))
    return 0;
  return workspace_need(p, M, y_dtype, mode, fused != 0);
}

int qmv_gemv(const qmv_pack* p, int M, int N, int K, int bits, int group, const void* x, void* y,
             int y_dtype, int mode, void* d_workspace, size_t workspace_bytes, void* stream) {
  int rc = check_common(p, M, x, y, y_dtype, mode);
  if (rc != QMV_OK) return rc;
  if (N != p->N || K != p->K || bits != p->bits || group != p->group) return QMV_ERR_SHAPE;
  rc = check_workspace(p, M, y_dtype, mode, 0, d_workspace, workspace_bytes);
  if (rc != QMV_OK) return rc;
  qmv::GemvArgs a = base_args(p, M, x, y, y_dtype);
  a.ws = d_workspace;
  a.ws_bytes = workspace_bytes;
  return run_cuda_core(a, p->bits, (cudaStream_t)stream, mode);
}

int qmv_chunk_gemm(const qmv_pack* p, int M, const void* x, void* y, int y_dtype, int mode,
                   void* d_workspace, size_t workspace_bytes, void* stream) {
  int rc = check_common(p, M, x, y, y_dtype, mode);
  if (rc != QMV_OK) return rc;
  rc = check_workspace(p, M, y_dtype, mode, 0, d_workspace, workspace_bytes);
  if (rc != QMV_OK) return rc;
  qmv::GemvArgs a = base_args(p, M, x, y, y_dtype);
  a.ws = d_workspace;
  a.ws_bytes = workspace_bytes;
  return run_cuda_core(a, p->bits, (cudaStream_t)stream, mode);
}

int qmv_fused_rmsnorm_gemv(const qmv_pack* p, int M, const void* x, const void* residual,
                           const void* gamma, float eps, void* h_out, void* y, int y_dtype,
                           int mode, void* d_workspace, size_t workspace_bytes, void* stream) {
  int rc = check_common(p, M, x, y, y_dtype, mode);
  if (rc != QMV_OK) return rc;
  rc = check_workspace(p, M, y_dtype, mode, 1, d_workspace, workspace_bytes);
  if (rc != QMV_OK) return rc;
  if (!residual || !gamma) return QMV_ERR_INVALID_ARG;
  if (!(eps >= 0.0f)) return QMV_ERR_INVALID_ARG;
  if (!aligned(residual, 16) || !aligned(gamma, 16) || (h_out && !aligned(h_out, 16)))
    return QMV_ERR_ALIGNMENT;
  qmv::GemvArgs a = base_args(p, M, x, y, y_dtype);
  a.fused = 1;
  a.r = (const __half*)residual;
  a.gamma = (const __half*)gamma;
  a.eps = eps;
  a.h_out = (__half*)h_out;
  a.ws = d_workspace;
  a.ws_bytes = workspace_bytes;
  return run_cuda_core(a, p->bits, (cudaStream_t)stream, mode);
}

size_t qmv_argmax_workspace_bytes(void) { return 16; }

int qmv_gemv_argmax(const qmv_pack* p, const void* x, const void* residual, const void* gamma,
                    float eps, void* h_out, void* y, int y_dtype, int mode, int* d_index,
                    float* d_value, void* d_workspace, void* stream) {
  if (!pack_ok(p) || !p->bound || !x || !d_index || !d_workspace) return QMV_ERR_INVALID_ARG;
  if (y && y_dtype != QMV_F32 && y_dtype != QMV_F16) return QMV_ERR_INVALID_ARG;
  if (mode != QMV_FAST && mode != QMV_EXACT) return QMV_ERR_INVALID_ARG;
  if (residual && (!gamma || !(eps >= 0.0f))) return QMV_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (y && !aligned(y, 4)) || !aligned(d_index, 4) || (d_value && !aligned(d_value, 4)) ||
      !aligned(d_workspace, 8) || (residual && (!aligned(residual, 16) || !aligned(gamma, 16))) ||
      (h_out && !aligned(h_out, 16)))
    return QMV_ERR_ALIGNMENT;
  qmv::GemvArgs a = base_args(p, 1, x, y, y ? y_dtype : QMV_F32);
  if (residual) {
    a.fused = 1;
    a.r = (const __half*)residual;
    a.gamma = (const __half*)gamma;
    a.eps = eps;
    a.h_out = (__half*)h_out;
  }
  a.folded = (mode == QMV_FAST && qmv::tma_fits(a.K, p->bits, a.perrow != 0)) ? 1 : 0;
  a.amax_ws = (unsigned long long*)d_workspace;
  a.amax_index = d_index;
  a.amax_value = d_value;
  cudaError_t err = cudaSuccess;
  const int rc = qmv::launch_gemv_tma(a, p->bits, (cudaStream_t)stream, &err);
  return rc == QMV_ERR_CUDA ? cuda_fail(err) : rc;
}

int qmv_gemv_gather(const qmv_pack* p, int rows_per_expert, const int* d_expert_ids, int n_selected,
                    const void* x, void* y, int y_dtype, int mode, void* stream) {
  if (!pack_ok(p) || !p->bound || !x || !y || !d_expert_ids) return QMV_ERR_INVALID_ARG;
  if (y_dtype != QMV_F32 && y_dtype != QMV_F16) return QMV_ERR_INVALID_ARG;
  if (mode != QMV_FAST && mode != QMV_EXACT) return QMV_ERR_INVALID_ARG;
  if (rows_per_expert < 1 || p->N % rows_per_expert != 0) return QMV_ERR_SHAPE;
  if (n_selected < 1 || n_selected > qmv::pipe::GATHER_MAX) return QMV_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 4) || !aligned(d_expert_ids, 4)) return QMV_ERR_ALIGNMENT;
  qmv::GemvArgs a = base_args(p, 1, x, y, y_dtype);
  a.folded = (mode == QMV_FAST && qmv::tma_fits(a.K, p->bits, a.perrow != 0)) ? 1 : 0;
  a.gather_ids = d_expert_ids;
  a.gather_rows = rows_per_expert;
  a.gather_n = n_selected;
  a.gather_E = p->N / rows_per_expert;
  cudaError_t err = cudaSuccess;
  const int rc = qmv::launch_gemv_tma(a, p->bits, (cudaStream_t)stream, &err);
  return rc == QMV_ERR_CUDA ? cuda_fail(err) : rc;
}

int qmv_unpack_codes(const qmv_pack* p, int8_t* d_codes_out, void* stream) {
  if (!pack_ok(p) || !p->bound || !d_codes_out) return QMV_ERR_INVALID_ARG;
  if (!aligned(d_codes_out, 16)) return QMV_ERR_ALIGNMENT;
  cudaError_t e = qmv::launch_unpack(p->bits, p->d_codes, d_codes_out,
                                     (int64_t)p->codes_bytes / 4, (cudaStream_t)stream);
  return e == cudaSuccess ? QMV_OK : cuda_fail(e);
}

int qmv_pack_info(const qmv_pack* p, int* N, int* K, int* bits, int* group) {
  if (!pack_ok(p)) return QMV_ERR_INVALID_ARG;
  if (N) *N = p->N;
  if (K) *K = p->K;
  if (bits) *bits = p->bits;
  if (group) *group = p->group;
  return QMV_OK;
}

// The saved-pack header (layout in qmv.h): little-endian fields written
// byte by byte, so the format does not depend on the host's struct layout.
static void put32(unsigned char* b, uint32_t v) {
  for (int i = 0; i < 4; ++i) b[i] = (unsigned char)(v >> (8 * i));
}
static void put64(unsigned char* b, uint64_t v) {
  for (int i = 0; i < 8; ++i) b[i] = (unsigned char)(v >> (8 * i));
}
static uint32_t get32(const unsigned char* b) {
  uint32_t v = 0;
  for (int i = 0; i < 4; ++i) v |= (uint32_t)b[i] << (8 * i);
  return v;
}
static uint64_t get64(const unsigned char* b) {
  uint64_t v = 0;
  for (int i = 0; i < 8; ++i) v |= (uint64_t)b[i] << (8 * i);
  return v;
}
static const char k_pack_magic[8] = {'Q', 'M', 'V', 'P', 'A', 'C', 'K', 0};

int qmv_pack_header(const qmv_pack* p, void* header_out) {
  if (!pack_ok(p) || !header_out) return QMV_ERR_INVALID_ARG;
  unsigned char* b = (unsigned char*)header_out;
  memset(b, 0, QMV_PACK_HEADER_BYTES);
  memcpy(b, k_pack_magic, 8);
  put32(b + 8, QMV_PACK_VERSION);
  put32(b + 12, QMV_PACK_HEADER_BYTES);
  put32(b + 16, (uint32_t)p->N);
  put32(b + 20, (uint32_t)p->K);
  put32(b + 24, (uint32_t)p->bits);
  put32(b + 28, (uint32_t)p->group);
  put64(b + 32, (uint64_t)p->codes_bytes);
  put64(b + 40, (uint64_t)p->scales_bytes);
  return QMV_OK;
}

int qmv_create_pack_from_header(qmv_pack** out, const void* header, size_t* codes_bytes,
                                size_t* scales_bytes) {
  if (!out) return QMV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!header) return QMV_ERR_INVALID_ARG;
  const unsigned char* b = (const unsigned char*)header;
  if (memcmp(b, k_pack_magic, 8) != 0 || get32(b + 12) != QMV_PACK_HEADER_BYTES)
    return QMV_ERR_INVALID_ARG;
  for (int i = 48; i < QMV_PACK_HEADER_BYTES; ++i)
    if (b[i]) return QMV_ERR_INVALID_ARG;
  if (get32(b + 8) != QMV_PACK_VERSION) return QMV_ERR_UNSUPPORTED;
  const int N = (int)get32(b + 16), K = (int)get32(b + 20), bits = (int)get32(b + 24),
            group = (int)get32(b + 28);
  size_t cb = 0, sb = 0;
  qmv_pack* p = nullptr;
  const int st = qmv_create_pack(&p, N, K, bits, group, &cb, &sb);
  if (st != QMV_OK) return st;
  if (get64(b + 32) != (uint64_t)cb || get64(b + 40) != (uint64_t)sb) {
    qmv_destroy_pack(p);
    return QMV_ERR_SHAPE;
  }
  if (codes_bytes) *codes_bytes = cb;
  if (scales_bytes) *scales_bytes = sb;
  *out = p;
  return QMV_OK;
}

int qmv_bind_packed(qmv_pack* p, void* d_codes, void* d_scales) {
  if (!pack_ok(p) || !d_codes || !d_scales) return QMV_ERR_INVALID_ARG;
  if (!aligned(d_codes, 16) || !aligned(d_scales, 16)) return QMV_ERR_ALIGNMENT;
  p->d_codes = (const uint32_t*)d_codes;
  p->d_scales = (const uint16_t*)d_scales;
  p->bound = 1;
  return QMV_OK;
}

int qmv_destroy_pack(qmv_pack* p) {
  if (!pack_ok(p)) return QMV_ERR_INVALID_ARG;
  p->magic = 0;
  delete p;
  return QMV_OK;
}

const char* qmv_status_string(int status) {
  switch (status) {
    case QMV_OK: return "ok";
    case QMV_ERR_INVALID_ARG: return "invalid argument";
    case QMV_ERR_UNSUPPORTED: return "unsupported configuration";
    case QMV_ERR_ALIGNMENT: return "pointer not aligned as required";
    case QMV_ERR_SHAPE: return "shape does not match the pack or the layout rules";
    case QMV_ERR_CUDA: return "CUDA error (see qmv_last_cuda_error)";
    case QMV_ERR_TIMEOUT: return "device-side wait timed out";
    case QMV_ERR_WORKSPACE: return "workspace missing or smaller than qmv_workspace_bytes()";
    default: return "unknown status";
  }
}

int qmv_last_cuda_error(void) { return g_last_cuda_error; }

int qmv_set_pdl(int enable) {
  qmv::set_pdl(enable != 0);
  return QMV_OK;
}

int qmv_device_error(int* out, int clear) {
  if (!out) return QMV_ERR_INVALID_ARG;
  const int e = qmv::read_device_error(clear, out);
  if (e != 0) return cuda_fail((cudaError_t)e);
  return QMV_OK;
}

}  // extern "C"
