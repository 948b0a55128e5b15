// C ABI of the library (declared in include/falcon.h): argument checks, the
// zero-length cases, and dispatch to the kernels.  Nothing is launched when an
// argument is rejected.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace falcon {
// Device error word: set by a kernel whose bounded wait gave up, read and
// cleared by falcon_sync_check().
static __device__ int g_device_error = 0;
// Falcon-2 in chunk form on the tensor cores (bf16, m = dv = 64, chunk 64;
// falcon2_tc.cu): one CTA per head, no workspace.
bool tc_falcon2_applies(int dtype, int m, int dv, int C, int64_t BH, int64_t T);
cudaError_t launch_tc_falcon2(const ChunkArgs& a, int* err, cudaStream_t stream);
}  // namespace falcon

namespace {

using falcon::ChunkArgs;
using falcon::DecodeArgs;

bool misaligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// The kernels are built for sm_103a only.
int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FALCON_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FALCON_ERR_CUDA;
  return (major == 10 && minor == 3) ? FALCON_OK : FALCON_ERR_DEVICE;
}

int check_common(int dtype, int phi, int ridge, float eps, float eps_gamma) {
  if (dtype != FALCON_BF16 && dtype != FALCON_F32) return FALCON_ERR_BAD_DTYPE;
  if (phi != FALCON_PHI_IDENTITY && phi != FALCON_PHI_L2 && phi != FALCON_PHI_RMS)
    return FALCON_ERR_BAD_DTYPE;
  if (ridge != FALCON_RIDGE_GIVEN && ridge != FALCON_RIDGE_SCALED) return FALCON_ERR_BAD_ARG;
  if (!(eps >= 0.f) || !(eps_gamma > 0.f) || !(eps_gamma < 1.f)) return FALCON_ERR_BAD_ARG;
  return FALCON_OK;
}

int check_shape(const falcon_shape* s) {
  if (!s) return FALCON_ERR_NULL_PTR;
  if (s->B < 0 || s->H < 0 || s->T < 0) return FALCON_ERR_BAD_SHAPE;
  if (!dim_ok(s->m) || !dim_ok(s->dv)) return FALCON_ERR_BAD_SHAPE;
  if (s->chunk != 16 && s->chunk != 32 && s->chunk != 64) return FALCON_ERR_BAD_SHAPE;
  // Grid limits: B*H CTAs along y of the prep grid, chunks along x.
  if (s->B * s->H > 65535 || (s->T + s->chunk - 1) / s->chunk > 0x7fffffffLL)
    return FALCON_ERR_BAD_SHAPE;
  return check_common(s->dtype, s->phi, s->ridge, s->eps, s->eps_gamma);
}

int to_status(cudaError_t e) { return e == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA; }

// Device address of g_device_error on the current device (kernels with
// bounded waits set it); resolved once per device.
constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
int* g_err_ptr[kMaxDevices] = {};

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, falcon::g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

int fwd_chunked(int rule, const falcon_shape* s, const void* q, const void* k, const void* v,
                const float* beta, const float* lambda, const float* S0, const float* x_prev,
                void* o, float* S_out, float* x_last, void* workspace, size_t workspace_bytes,
                cudaStream_t stream, int window = 1, bool chunked_form = false,
                int (*resolve_workspace)(void**) = nullptr, float* norm_ws = nullptr) {
  int rc = check_shape(s);
  if (rc) return rc;
  const int64_t BH = s->B * s->H;
  if (BH == 0) return FALCON_OK;
  if (!S_out) return FALCON_ERR_NULL_PTR;
  if (s->T > 0 && (!q || !k || !v || !beta || !lambda || !o)) return FALCON_ERR_NULL_PTR;
  const void* ptrs[] = {q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last};
  for (const void* p : ptrs)
    if (misaligned(p)) return FALCON_ERR_MISALIGNED;
  // The per-column and windowed rules run in the token-recurrent form: no
  // workspace.  The window of Falcon-3A holds at most 32 pairs and does not
  // reach into a previous segment (no x_prev).
  const bool per_column = rule == falcon::kFalcon2 || rule == falcon::kFalcon2A;
  const bool windowed = rule == falcon::kFalcon3A;
  if (windowed && (window < 1 || window > 32 || x_prev)) return FALCON_ERR_BAD_ARG;
  // Falcon-3A in chunk form where the tensor-core path applies (it writes the
  // chunk maps to the workspace); otherwise the token-recurrent kernel.
  const bool window_tc = windowed && chunked_form &&
                         falcon::tc_falcon3a_applies(s->dtype, s->m, s->dv, s->chunk, BH, s->T);
  // Falcon-2A likewise (chunk maps in the workspace).  Falcon-2 in chunk form
  // runs one CTA per head and needs no workspace.
  const bool column_tc = rule == falcon::kFalcon2A && chunked_form &&
                         falcon::tc_falcon2a_applies(s->dtype, s->m, s->dv, s->chunk, BH, s->T);
  const bool column2_tc = rule == falcon::kFalcon2 && chunked_form &&
                          falcon::tc_falcon2_applies(s->dtype, s->m, s->dv, s->chunk, BH, s->T);
  const size_t need = ((per_column && !column_tc) || (windowed && !window_tc))
                          ? 0
                          : falcon_workspace_bytes(s);
  // A resolver stands for a workspace of workspace_bytes whose address is
  // only known once a device is current: it is asked after every argument
  // check, so that the codes are the same as for a caller-given workspace.
  if (need > 0 && ((!workspace && !resolve_workspace) || workspace_bytes < need))
    return FALCON_ERR_WORKSPACE;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FALCON_ERR_MISALIGNED;
  rc = check_device();
  if (rc) return rc;
  if (resolve_workspace) {
    rc = resolve_workspace(&workspace);
    if (rc) return rc;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FALCON_ERR_MISALIGNED;
  }

  const size_t state_bytes = sizeof(float) * (size_t)BH * s->m * s->dv;
  if (s->T == 0) {  // nothing to run: S_T = S0, x_last = x_prev
    cudaError_t e = cudaSuccess;
    if (S0 && S0 != S_out)
      e = cudaMemcpyAsync(S_out, S0, state_bytes, cudaMemcpyDeviceToDevice, stream);
    else if (!S0)
      e = cudaMemsetAsync(S_out, 0, state_bytes, stream);
    if (e == cudaSuccess && x_last && x_prev && x_last != x_prev)
      e = cudaMemcpyAsync(x_last, x_prev, sizeof(float) * (size_t)BH * s->m,
                          cudaMemcpyDeviceToDevice, stream);
    return to_status(e);
  }
  ChunkArgs a;
  a.rule = rule;
  a.BH = BH;
  a.T = s->T;
  a.m = s->m;
  a.dv = s->dv;
  a.C = s->chunk;
  a.dtype = s->dtype;
  a.phi = s->phi;
  a.ridge = s->ridge;
  a.eps = s->eps;
  a.eps_gamma = s->eps_gamma;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.lambda = lambda;
  a.S0 = S0;
  a.x_prev = x_prev;
  a.o = o;
  a.S_out = S_out;
  a.x_last = x_last;
  a.workspace = workspace;
  a.norm_ws = norm_ws;
  if (per_column || windowed) {
    int* err = device_error_word();
    if (!err) return FALCON_ERR_CUDA;
    if (window_tc) return to_status(falcon::launch_tc_falcon3a(a, window, err, stream));
    if (column_tc) return to_status(falcon::launch_tc_falcon2a(a, err, stream));
    if (column2_tc) return to_status(falcon::launch_tc_falcon2(a, err, stream));
    return to_status(windowed ? falcon::launch_falcon3a_recurrent(a, window, err, stream)
                              : falcon::launch_falcon2_recurrent(a, err, stream));
  }
  if (falcon::tc_path_applies(s->dtype, s->m, s->dv, s->chunk, s->B * s->H, s->T)) {
    int* err = device_error_word();
    if (!err) return FALCON_ERR_CUDA;
    return to_status(falcon::launch_tc_chunked(a, err, stream));
  }
  return to_status(falcon::launch_generic_chunked(a, stream));
}

int bwd_chunked(int rule, const falcon_shape* s, const void* q, const void* k, const void* v,
                const float* beta, const float* lambda, const float* S0, const float* x_prev,
                const void* dO, const float* dS_T, const float* dx_last, void* dq, void* dk,
                void* dv, float* dbeta, float* dlambda, float* dS0, float* dx_prev,
                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_shape(s);
  if (rc) return rc;
  const int64_t BH = s->B * s->H;
  if (BH == 0) return FALCON_OK;
  if (s->T > 0 && (!q || !k || !v || !beta || !lambda || !dO || !dq || !dk || !dv || !dbeta ||
                   !dlambda))
    return FALCON_ERR_NULL_PTR;
  const void* ptrs[] = {q,  k,  v,  beta,    lambda, S0,  x_prev,  dO,
                        dS_T, dx_last, dq, dk, dv, dbeta, dlambda, dS0, dx_prev};
  for (const void* p : ptrs)
    if (misaligned(p)) return FALCON_ERR_MISALIGNED;
  const size_t need = falcon_bwd_workspace_bytes(s);
  if (need > 0 && (!workspace || workspace_bytes < need)) return FALCON_ERR_WORKSPACE;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FALCON_ERR_MISALIGNED;
  rc = check_device();
  if (rc) return rc;
  if (s->T == 0) {  // S_T = S0 and x_last = x_prev: the cotangents pass through
    cudaError_t e = cudaSuccess;
    const size_t state_bytes = sizeof(float) * (size_t)BH * s->m * s->dv;
    const size_t feat_bytes = sizeof(float) * (size_t)BH * s->m;
    if (dS0 && dS_T && dS0 != dS_T)
      e = cudaMemcpyAsync(dS0, dS_T, state_bytes, cudaMemcpyDeviceToDevice, stream);
    else if (dS0 && !dS_T)
      e = cudaMemsetAsync(dS0, 0, state_bytes, stream);
    if (e == cudaSuccess && dx_prev) {
      if (x_prev && dx_last) {
        if (dx_prev != dx_last)
          e = cudaMemcpyAsync(dx_prev, dx_last, feat_bytes, cudaMemcpyDeviceToDevice, stream);
      } else {
        e = cudaMemsetAsync(dx_prev, 0, feat_bytes, stream);
      }
    }
    return to_status(e);
  }
  falcon::BwdArgs b;
  ChunkArgs& a = b.f;
  a.rule = rule;
  a.BH = BH;
  a.T = s->T;
  a.m = s->m;
  a.dv = s->dv;
  a.C = s->chunk;
  a.dtype = s->dtype;
  a.phi = s->phi;
  a.ridge = s->ridge;
  a.eps = s->eps;
  a.eps_gamma = s->eps_gamma;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.lambda = lambda;
  a.S0 = S0;
  a.x_prev = x_prev;
  a.o = nullptr;
  a.S_out = nullptr;
  a.x_last = nullptr;
  a.workspace = workspace;
  b.dO = dO;
  b.dS_T = dS_T;
  b.dx_last = dx_last;
  b.dq = dq;
  b.dk = dk;
  b.dv = dv;
  b.dbeta = dbeta;
  b.dlambda = dlambda;
  b.dS0 = dS0;
  b.dx_prev = dx_prev;
  int* err = device_error_word();
  if (!err) return FALCON_ERR_CUDA;
  return to_status(falcon::launch_bwd_chunked(b, err, stream));
}

// Failure-path diagnostic: every thread waits on an mbarrier that nothing
// completes, gives up after limit_ns and records the expiry in the device
// error word (the same path the tensor-core kernels take on a lost wait).
__global__ void wait_timeout_kernel(uint64_t limit_ns, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    falcon::tc::mbar_init(&bar, 1);
    falcon::tc::fence_mbar_init();
  }
  __syncthreads();
  const bool ok = falcon::tc::mbar_wait(&bar, 0, limit_ns);
  if (!__syncthreads_or(!ok)) return;
  if (threadIdx.x == 0) atomicExch(err, 1);
}

int decode(int rule, int64_t N, int32_t m, int32_t dv, int32_t dtype, int32_t phi, int32_t ridge,
           float eps, float eps_gamma, const void* q, const void* k, const void* v, const float* beta,
           const float* lambda, float* S, float* x_prev, const uint8_t* fresh, void* o,
           cudaStream_t stream) {
  if (N < 0 || N > 0x7fffffffLL || !dim_ok(m) || !dim_ok(dv)) return FALCON_ERR_BAD_SHAPE;
  int rc = check_common(dtype, phi, ridge, eps, eps_gamma);
  if (rc) return rc;
  if (N == 0) return FALCON_OK;
  if (!q || !k || !v || !beta || !lambda || !S || !x_prev || !o) return FALCON_ERR_NULL_PTR;
  const void* ptrs[] = {q, k, v, beta, lambda, S, x_prev, o};
  for (const void* p : ptrs)
    if (misaligned(p)) return FALCON_ERR_MISALIGNED;
  rc = check_device();
  if (rc) return rc;
  DecodeArgs a;
  a.rule = rule;
  a.N = N;
  a.m = m;
  a.dv = dv;
  a.dtype = dtype;
  a.phi = phi;
  a.ridge = ridge;
  a.eps = eps;
  a.eps_gamma = eps_gamma;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.lambda = lambda;
  a.S = S;
  a.x_prev = x_prev;
  a.fresh = fresh;
  a.o = o;
  a.err = device_error_word();
  if (!a.err) return FALCON_ERR_CUDA;
  return to_status(falcon::launch_decode(a, stream));
}

}  // namespace

namespace falcon {
// Falcon-1 chunked forward over a workspace of workspace_bytes whose device
// address `resolve` gives once the device check has passed.
int fwd_chunked_resolved(const falcon_shape* s, const void* q, const void* k, const void* v,
                         const float* beta, const float* lambda, const float* S0,
                         const float* x_prev, void* o, float* S_out, float* x_last,
                         int (*resolve)(void**), size_t workspace_bytes, cudaStream_t stream) {
  return fwd_chunked(kFalcon1, s, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last, nullptr,
                     workspace_bytes, stream, 1, false, resolve);
}
}  // namespace falcon

extern "C" {

size_t falcon_workspace_bytes(const falcon_shape* s) {
  if (check_shape(s) != FALCON_OK) return 0;
  if (falcon::tc_path_applies(s->dtype, s->m, s->dv, s->chunk, s->B * s->H, s->T)) {
    const size_t tc = falcon::tc_workspace_bytes(s->m, s->B * s->H, s->T);
    if (s->m != 64) return tc;
    // m = 64: room for the Falcon-2A chunk maps too (a little larger)
    const size_t c2a = falcon::tc_falcon2a_workspace_bytes(s->B * s->H, s->T);
    return tc > c2a ? tc : c2a;
  }
  return falcon::generic_workspace_bytes(s->B * s->H, s->T, s->m, s->dv, s->chunk);
}

int falcon1_fwd_chunked(const falcon_shape* s, const void* q, const void* k, const void* v,
                        const float* beta, const float* lambda, const float* S0,
                        const float* x_prev, void* o, float* S_out, float* x_last,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return fwd_chunked(falcon::kFalcon1, s, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last,
                     workspace, workspace_bytes, stream);
}

int falcon1a_fwd_chunked(const falcon_shape* s, const void* q, const void* k, const void* v,
                         const float* beta, const float* lambda, const float* S0,
                         const float* x_prev, void* o, float* S_out, float* x_last,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return fwd_chunked(falcon::kFalcon1A, s, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last,
                     workspace, workspace_bytes, stream);
}

// The normalised read's own workspace follows the forward's, 256-byte aligned.
static size_t norm_offset(const falcon_shape* s) {
  return (falcon_workspace_bytes(s) + 255) / 256 * 256;
}

size_t falcon_normalized_workspace_bytes(const falcon_shape* s) {
  if (check_shape(s) != FALCON_OK) return 0;
  if (s->B * s->H == 0 || s->T == 0) return falcon_workspace_bytes(s);
  return norm_offset(s) + falcon::norm_workspace_bytes(s->B * s->H, s->T, s->m, s->chunk);
}

int falcon1a_fwd_chunked_normalized(const falcon_shape* s, const void* q, const void* k,
                                    const void* v, const float* beta, const float* lambda,
                                    const float* S0, const float* z0, const float* x_prev,
                                    float eps_attn, void* o, float* S_out, float* z_out,
                                    float* x_last, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (!(eps_attn >= 0.f) || !(eps_attn < INFINITY)) return FALCON_ERR_BAD_ARG;
  const int64_t BH = s->B * s->H;
  if (BH == 0) return FALCON_OK;
  if (misaligned(z0) || misaligned(z_out)) return FALCON_ERR_MISALIGNED;
  const size_t need = falcon_normalized_workspace_bytes(s);
  if (s->T > 0 && need > 0 && (!workspace || workspace_bytes < need)) return FALCON_ERR_WORKSPACE;
  // The numerator: the Falcon-1A forward (every remaining check is its own;
  // nothing is launched when one fails).
  const size_t base = s->T > 0 ? norm_offset(s) : workspace_bytes;
  float* ws = s->T > 0
                  ? reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + base)
                  : nullptr;
  // On the tensor-core path with m = 64 the forward's map launch writes the
  // denominator's per-chunk terms as well.
  const bool terms_in_maps =
      ws && s->m == 64 && falcon::tc_path_applies(s->dtype, s->m, s->dv, s->chunk, BH, s->T);
  rc = fwd_chunked(falcon::kFalcon1A, s, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last,
                   workspace, base, stream, 1, false, nullptr, terms_in_maps ? ws : nullptr);
  if (rc) return rc;
  const size_t feat_bytes = sizeof(float) * (size_t)BH * s->m;
  if (s->T == 0) {  // z_T = z0
    cudaError_t e = cudaSuccess;
    if (z_out && z0 && z_out != z0)
      e = cudaMemcpyAsync(z_out, z0, feat_bytes, cudaMemcpyDeviceToDevice, stream);
    else if (z_out && !z0)
      e = cudaMemsetAsync(z_out, 0, feat_bytes, stream);
    return to_status(e);
  }
  ChunkArgs a;
  a.rule = falcon::kFalcon1A;
  a.BH = BH;
  a.T = s->T;
  a.m = s->m;
  a.dv = s->dv;
  a.C = s->chunk;
  a.dtype = s->dtype;
  a.phi = s->phi;
  a.ridge = s->ridge;
  a.eps = s->eps;
  a.eps_gamma = s->eps_gamma;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.lambda = lambda;
  a.S0 = S0;
  a.x_prev = x_prev;
  a.o = o;
  a.S_out = S_out;
  a.x_last = x_last;
  a.workspace = workspace;
  return to_status(falcon::launch_normalizer(a, z0, z_out, eps_attn, ws, terms_in_maps, stream));
}

size_t falcon_bwd_workspace_bytes(const falcon_shape* s) {
  if (check_shape(s) != FALCON_OK) return 0;
  return falcon::bwd_workspace_bytes(s->dtype, s->B * s->H, s->T, s->m, s->dv, s->chunk);
}

int falcon1_bwd_chunked(const falcon_shape* s, const void* q, const void* k, const void* v,
                        const float* beta, const float* lambda, const float* S0,
                        const float* x_prev, const void* dO, const float* dS_T,
                        const float* dx_last, void* dq, void* dk, void* dv, float* dbeta,
                        float* dlambda, float* dS0, float* dx_prev, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  return bwd_chunked(falcon::kFalcon1, s, q, k, v, beta, lambda, S0, x_prev, dO, dS_T, dx_last,
                     dq, dk, dv, dbeta, dlambda, dS0, dx_prev, workspace, workspace_bytes,
                     stream);
}

int falcon1a_bwd_chunked(const falcon_shape* s, const void* q, const void* k, const void* v,
                         const float* beta, const float* lambda, const float* S0,
                         const float* x_prev, const void* dO, const float* dS_T,
                         const float* dx_last, void* dq, void* dk, void* dv, float* dbeta,
                         float* dlambda, float* dS0, float* dx_prev, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  return bwd_chunked(falcon::kFalcon1A, s, q, k, v, beta, lambda, S0, x_prev, dO, dS_T, dx_last,
                     dq, dk, dv, dbeta, dlambda, dS0, dx_prev, workspace, workspace_bytes,
                     stream);
}

int falcon2_fwd_recurrent(const falcon_shape* s, const void* q, const void* k, const void* v,
                          const float* beta, const float* lambda, const float* S0,
                          const float* x_prev, void* o, float* S_out, float* x_last,
                          cudaStream_t stream) {
  return fwd_chunked(falcon::kFalcon2, s, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last,
                     nullptr, 0, stream);
}

int falcon2a_fwd_recurrent(const falcon_shape* s, const void* q, const void* k, const void* v,
                           const float* beta, const float* lambda, const float* S0,
                           const float* x_prev, void* o, float* S_out, float* x_last,
                           cudaStream_t stream) {
  return fwd_chunked(falcon::kFalcon2A, s, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last,
                     nullptr, 0, stream);
}

int falcon3a_fwd_recurrent(const falcon_shape* s, int32_t window, const void* q, const void* k,
                           const void* v, const float* beta, const float* lambda,
                           const float* S0, void* o, float* S_out, float* x_last,
                           cudaStream_t stream) {
  return fwd_chunked(falcon::kFalcon3A, s, q, k, v, beta, lambda, S0, nullptr, o, S_out, x_last,
                     nullptr, 0, stream, window);
}

int falcon2a_fwd_chunked(const falcon_shape* s, const void* q, const void* k, const void* v,
                         const float* beta, const float* lambda, const float* S0,
                         const float* x_prev, void* o, float* S_out, float* x_last,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return fwd_chunked(falcon::kFalcon2A, s, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last,
                     workspace, workspace_bytes, stream, 1, true);
}

int falcon2_fwd_chunked(const falcon_shape* s, const void* q, const void* k, const void* v,
                        const float* beta, const float* lambda, const float* S0,
                        const float* x_prev, void* o, float* S_out, float* x_last,
                        cudaStream_t stream) {
  return fwd_chunked(falcon::kFalcon2, s, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last,
                     nullptr, 0, stream, 1, true);
}

int falcon3a_fwd_chunked(const falcon_shape* s, int32_t window, const void* q, const void* k,
                         const void* v, const float* beta, const float* lambda, const float* S0,
                         void* o, float* S_out, float* x_last, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  return fwd_chunked(falcon::kFalcon3A, s, q, k, v, beta, lambda, S0, nullptr, o, S_out, x_last,
                     workspace, workspace_bytes, stream, window, true);
}

int falcon1_decode_step(int64_t N, int32_t m, int32_t dv, int32_t dtype, int32_t phi,
                        int32_t ridge, float eps, float eps_gamma, const void* q, const void* k,
                        const void* v, const float* beta, const float* lambda, float* S,
                        float* x_prev, const uint8_t* fresh, void* o, cudaStream_t stream) {
  return decode(falcon::kFalcon1, N, m, dv, dtype, phi, ridge, eps, eps_gamma, q, k, v, beta,
                lambda, S, x_prev, fresh, o, stream);
}

int falcon1a_decode_step(int64_t N, int32_t m, int32_t dv, int32_t dtype, int32_t phi,
                         int32_t ridge, float eps, float eps_gamma, const void* q, const void* k,
                         const void* v, const float* beta, const float* lambda, float* S,
                         float* x_prev, const uint8_t* fresh, void* o, cudaStream_t stream) {
  return decode(falcon::kFalcon1A, N, m, dv, dtype, phi, ridge, eps, eps_gamma, q, k, v, beta,
                lambda, S, x_prev, fresh, o, stream);
}

int falcon_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
  if (limit_us == 0 || limit_us > 10000000u) return FALCON_ERR_BAD_ARG;
  int rc = check_device();
  if (rc) return rc;
  int* err = device_error_word();
  if (!err) return FALCON_ERR_CUDA;
  wait_timeout_kernel<<<1, 64, 0, stream>>>((uint64_t)limit_us * 1000ull, err);
  return to_status(cudaGetLastError());
}

int falcon_sync_check(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FALCON_ERR_CUDA;
  int flag = 0;
  if (cudaMemcpyFromSymbol(&flag, falcon::g_device_error, sizeof(int)) != cudaSuccess)
    return FALCON_ERR_CUDA;
  if (flag) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(falcon::g_device_error, &zero, sizeof(int)) != cudaSuccess)
      return FALCON_ERR_CUDA;
    return FALCON_ERR_TIMEOUT;
  }
  return FALCON_OK;
}

const char* falcon_strerror(int code) {
  switch (code) {
    case FALCON_OK: return "ok";
    case FALCON_ERR_NULL_PTR: return "a required pointer is NULL";
    case FALCON_ERR_BAD_SHAPE: return "unsupported shape (m, dv in {16,32,64,128}; chunk in {16,32,64})";
    case FALCON_ERR_BAD_DTYPE: return "dtype or phi code out of range";
    case FALCON_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case FALCON_ERR_WORKSPACE: return "workspace missing or too small";
    case FALCON_ERR_CUDA: return "CUDA launch or query failed";
    case FALCON_ERR_TIMEOUT: return "a device-side wait hit its iteration limit";
    case FALCON_ERR_BAD_ARG:
      return "a scalar argument is out of range (eps >= 0, eps_gamma in (0, 1), eps_attn >= 0, "
             "window, wait limit)";
    case FALCON_ERR_DEVICE: return "current device is not sm_103 (GB300)";
    case FALCON_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the library's fixed array (FALCON_FIXED_SCRATCH_BYTES)";
  }
  return "unknown error code";
}

int falcon_version(void) { return 10200; }

}  // extern "C"
