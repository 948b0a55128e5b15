// Shared device helpers of the Falcon GB300 library (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "falcon.h"

namespace falcon {

// Rule selector shared by kernels: Falcon-1 writes the residual
// r_t = v_t - S_{t-1}^T x_t, Falcon-1A writes the target v_t; Falcon-2 and
// Falcon-2A are their per-column counterparts (one step size per column).
enum Rule : int { kFalcon1 = 1, kFalcon1A = 2, kFalcon2 = 3, kFalcon2A = 4, kFalcon3A = 5 };

__device__ __forceinline__ float load_elem(const void* p, int64_t i, int dtype) {
  if (dtype == FALCON_BF16)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ void store_elem(void* p, int64_t i, float x, int dtype) {
  if (dtype == FALCON_BF16)
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<float*>(p)[i] = x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// phi's scale for a row u of m values with squared norm ss: 1 for the
// identity, 1 / max(||u||, 1e-12) for the l2 map, 1 / sqrt(ss / m + eps_rms)
// for RMSNorm (eps_rms = 1e-6: the pages name the stabiliser without a value).
constexpr float kEpsRms = 1e-6f;
__device__ __forceinline__ float feature_scale(float ss, int m, int phi) {
  if (phi == FALCON_PHI_L2) return 1.f / fmaxf(sqrtf(ss), 1e-12f);
  if (phi == FALCON_PHI_RMS) return rsqrtf(ss / (float)m + kEpsRms);
  return 1.f;
}

// lambda_t used by the recurrence: as given, or the scale-coupled form
// lambda_bar_t * E_t with E_t = ||x_t||^2.
__device__ __forceinline__ float ridge_of(float lam, float E, int ridge) {
  return ridge == FALCON_RIDGE_SCALED ? lam * E : lam;
}

// Step size and decay of one token (Eq. (3.4) and the decay clamp).
// Returns eta; writes gamma = 1 - min(eta*lambda, 1 - eps_gamma) and its log.
// On the clamped branch gamma is exactly eps_gamma: forming 1 - (1 - eps_gamma)
// in fp32 would cancel (9.54e-7 instead of 1e-6).
__device__ __forceinline__ float step_eta_gamma(bool sentinel, float E, float beta,
                                                float lambda, float eps, float eps_gamma,
                                                float* gamma, float* log_gamma) {
  float eta = 0.f;
  if (!sentinel) {
    const float den = E + lambda + eps;
    eta = den > 0.f ? beta / den : 0.f;
  }
  const float a = eta * lambda;
  if (a >= 1.f - eps_gamma) {
    *gamma = eps_gamma;
    *log_gamma = logf(eps_gamma);
  } else {
    *gamma = 1.f - a;
    *log_gamma = log1pf(-a);
  }
  return eta;
}

}  // namespace falcon

// Host-side launchers (defined in the kernel translation units).
namespace falcon {
struct ChunkArgs {
  int rule;
  int64_t BH, T;
  int m, dv, C, dtype, phi, ridge;
  float eps, eps_gamma;
  const void *q, *k, *v;
  const float *beta, *lambda, *S0, *x_prev;
  void* o;
  float *S_out, *x_last;
  void* workspace;
  // Tensor-core path, m = 64: the state entering every chunk is also written
  // here when non-null ([B*H, chunks, m, dv] f32; for the backward pass).
  float* S_starts = nullptr;
  // Tensor-core path, m = 64: the normalised read's per-chunk terms (NormLayout
  // below) are also written here by the map launch when non-null.
  float* norm_ws = nullptr;
};

// Workspace of the normalised read's denominator, in floats, per (head,
// chunk) mi = bh * chunks + c: z entering the chunk (m), the chunk's increment
// y_C (m), its decay e^{g_C} (1, padded to 4), and per token e^{g_t}, phi's
// scale of q_t and the in-chunk read r_t = <phi(q_t), y_t> (C each).
struct NormLayout {
  int64_t maps, m, C;
  __host__ __device__ size_t zin() const { return 0; }
  __host__ __device__ size_t inc() const { return (size_t)(maps * m); }
  __host__ __device__ size_t dec() const { return (size_t)(2 * maps * m); }
  __host__ __device__ size_t eg() const { return dec() + (size_t)(maps * 4); }
  __host__ __device__ size_t nq() const { return eg() + (size_t)(maps * C); }
  __host__ __device__ size_t rd() const { return nq() + (size_t)(maps * C); }
  __host__ __device__ size_t floats() const { return rd() + (size_t)(maps * C); }
};
size_t generic_workspace_bytes(int64_t BH, int64_t T, int m, int dv, int C);
// a.o and a.S_out may be null (not written); S_starts (nullable) receives the
// state entering every chunk, [B*H, chunks, m, dv] f32.
cudaError_t launch_generic_chunked(const ChunkArgs& a, cudaStream_t stream,
                                   float* S_starts = nullptr);

// Falcon-2 / Falcon-2A, token-recurrent form (rule kFalcon2 or kFalcon2A;
// beta is [B*H, T, dv]: one gain per column and token).
cudaError_t launch_falcon2_recurrent(const ChunkArgs& a, int* err, cudaStream_t stream);

// Falcon-3A, token-recurrent form over fresh sequences, window 1 .. 32 pairs.
cudaError_t launch_falcon3a_recurrent(const ChunkArgs& a, int window, int* err,
                                      cudaStream_t stream);

// Tensor-core path (bf16, m = dv in {64, 128}, chunk = 64).
bool tc_path_applies(int dtype, int m, int dv, int C, int64_t BH, int64_t T);
size_t tc_workspace_bytes(int m, int64_t BH, int64_t T);
cudaError_t launch_tc_chunked(const ChunkArgs& a, int* err, cudaStream_t stream);
// The m = 64 tensor-core scan alone, over maps already in a.workspace.
cudaError_t launch_tc_scan64(const ChunkArgs& a, int* err, cudaStream_t stream);
// The map launch alone (m = d_v = 64), by programmatic dependent launch.
cudaError_t launch_tc_map64(const ChunkArgs& a, int* err, cudaStream_t stream);
// Falcon-2A in chunk form on the tensor cores (bf16, m = dv = 64, chunk 64).
bool tc_falcon2a_applies(int dtype, int m, int dv, int C, int64_t BH, int64_t T);
size_t tc_falcon2a_workspace_bytes(int64_t BH, int64_t T);
cudaError_t launch_tc_falcon2a(const ChunkArgs& a, int* err, cudaStream_t stream);
// Falcon-3A in chunk form on the tensor cores (bf16, m = dv = 64, chunk 64).
bool tc_falcon3a_applies(int dtype, int m, int dv, int C, int64_t BH, int64_t T);
cudaError_t launch_tc_falcon3a(const ChunkArgs& a, int window, int* err, cudaStream_t stream);

// Backward pass of Falcon-1 / Falcon-1A (chunk form).  Cotangents dO (dtype),
// dS_T and dx_last (f32, nullable = zero); gradients dq, dk, dv (dtype),
// dbeta, dlambda (f32), dS0 and dx_prev (f32, nullable = not written).
struct BwdArgs {
  ChunkArgs f;  // the forward problem (f.o, f.S_out, f.x_last unused)
  const void* dO;
  const float *dS_T, *dx_last;
  void *dq, *dk, *dv;
  float *dbeta, *dlambda, *dS0, *dx_prev;
};
size_t bwd_workspace_bytes(int dtype, int64_t BH, int64_t T, int m, int dv, int C);
cudaError_t launch_bwd_chunked(const BwdArgs& b, int* err, cudaStream_t stream);
// Tensor-core per-chunk gradients (bf16, m = dv = 64, chunk 64), dk included
// (edge: [B*H, chunks, 64] f32 scratch for row 0 of every chunk's dX).
bool tc_bwd_applies(int dtype, int m, int dv, int C);
cudaError_t launch_tc_bwd_grad(const BwdArgs& b, const float* S_starts, const float* dS_ends,
                               float* edge, int* err, cudaStream_t stream);
// Reverse scan of the state cotangent over the tensor-core forward's maps.
cudaError_t launch_tc_bwd_scan(const BwdArgs& b, const void* maps, float* dS_ends, int* err,
                               cudaStream_t stream);

// Falcon-1A's normalised read: the denominator z_t^T phi(q_t) + eps_attn
// (z_t = gamma_t z_{t-1} + eta_t x_t) and the division of o in place, after
// the Falcon-1A forward has written o.  ws: norm_workspace_bytes bytes.
// chunk_terms_written: the forward's map launch has already written the
// per-chunk terms (increment, decays, phi's scales of q, in-chunk reads) to ws
// (ChunkArgs::norm_ws), so the in-chunk kernel is not launched.
size_t norm_workspace_bytes(int64_t BH, int64_t T, int m, int C);
cudaError_t launch_normalizer(const ChunkArgs& a, const float* z0, float* z_out, float eps_attn,
                              float* ws, bool chunk_terms_written, cudaStream_t stream);

struct DecodeArgs {
  int rule;
  int64_t N;
  int m, dv, dtype, phi, ridge;
  float eps, eps_gamma;
  const void *q, *k, *v;
  const float *beta, *lambda;
  float *S, *x_prev;
  const uint8_t* fresh;
  void* o;
  int* err = nullptr;  // device error word (a bounded wait that gave up)
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
}  // namespace falcon
