// Single-token recurrent step (read after write) for N independent states.
//
// Per state: a = S^T x, b = S^T phi(q), r = v - a (Falcon-1) or v (Falcon-1A),
// o = gamma b + eta <x, phi(q)> r   (= S_t^T phi(q) with S_t below),
// S_t = gamma S + eta x r^T,  x_prev <- phi(k).
// The update order follows the one-step listing of page
// rcap.io/posts/fast-weight-attention-for-continual-learning-2026-08-27 and
// Eq. (3.3) of page hyper.ai/fr/papers/2608.27763.
//
// The step is HBM-bound: the fp32 state is read once and written once.  One
// CTA owns one state.  Each thread keeps its share of S in registers between
// the read pass and the write pass, as float4 (128-bit) loads and stores that
// cover whole rows per warp, so every access is coalesced.  The two column
// reductions (S^T x and S^T phi(q)) run over the rows a thread holds, then
// across row groups through shared memory.
#include "common.cuh"

namespace falcon {
namespace {

// The state streams through once per step (far larger than L2 at scale):
// evict-first loads and stores.
__device__ __forceinline__ float4 ld_stream(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void st_stream(float* p, float4 v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}

template <int M, int DV>
struct DecodeCfg {
  static constexpr int kLanesPerRow = DV / 4;                  // float4 per row
  static constexpr int kVec = M * DV / 4;                      // float4 per state
  static constexpr int kThreads = kVec < 256 ? kVec : 256;     // >= 32 for M,DV >= 16
  static constexpr int kRowsPerPass = kThreads / kLanesPerRow;
  static constexpr int kIters = M / kRowsPerPass;
};

template <int M, int DV>
__global__ void __launch_bounds__(DecodeCfg<M, DV>::kThreads)
    decode_kernel(DecodeArgs a) {
  using Cfg = DecodeCfg<M, DV>;
  constexpr int kT = Cfg::kThreads;
  const int64_t n = blockIdx.x;
  const int tid = threadIdx.x;
  const int col4 = tid % Cfg::kLanesPerRow;
  const int rgrp = tid / Cfg::kLanesPerRow;

  __shared__ float xs[M], qs[M];
  __shared__ float red[Cfg::kRowsPerPass][2][DV];
  __shared__ float scal[4];  // eta, gamma, <x,q>

  float* S = a.S + n * (int64_t)M * DV;
  // Issue the state loads first: they are the long-latency part.
  float4 s[Cfg::kIters];
#pragma unroll
  for (int it = 0; it < Cfg::kIters; ++it) {
    const int row = rgrp + it * Cfg::kRowsPerPass;
    s[it] = ld_stream(S + row * DV + col4 * 4);
  }

  // Features and scalars (warp 0): x, phi(q), phi(k).
  const bool fresh = a.fresh ? (a.fresh[n] != 0) : false;
  if (tid < 32) {
    float qv[(M + 31) / 32], kv[(M + 31) / 32], xv[(M + 31) / 32];
    float sq = 0.f, sk = 0.f, sx = 0.f;
#pragma unroll
    for (int e = 0; e < (M + 31) / 32; ++e) {
      const int i = tid + 32 * e;
      const bool in = i < M;
      qv[e] = in ? load_elem(a.q, n * M + i, a.dtype) : 0.f;
      kv[e] = in ? load_elem(a.k, n * M + i, a.dtype) : 0.f;
      xv[e] = (in && !fresh) ? a.x_prev[n * M + i] : 0.f;
      sq += qv[e] * qv[e];
      sk += kv[e] * kv[e];
      sx += xv[e] * xv[e];
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float E = warp_sum(sx);
    const float fq = feature_scale(sq, M, a.phi), fk = feature_scale(sk, M, a.phi);
    float xq = 0.f;
#pragma unroll
    for (int e = 0; e < (M + 31) / 32; ++e) {
      const int i = tid + 32 * e;
      if (i < M) {
        xs[i] = xv[e];
        qs[i] = qv[e] * fq;
        a.x_prev[n * M + i] = kv[e] * fk;  // write feature of the next token
      }
      xq += xv[e] * qv[e] * fq;
    }
    xq = warp_sum(xq);
    if (tid == 0) {
      float gamma, lg;
      const float eta = step_eta_gamma(fresh, E, a.beta[n], ridge_of(a.lambda[n], E, a.ridge),
                                       a.eps, a.eps_gamma, &gamma, &lg);
      scal[0] = eta;
      scal[1] = gamma;
      scal[2] = xq;
    }
  }
  __syncthreads();

  // Partial column sums over this thread's rows.
  float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int it = 0; it < Cfg::kIters; ++it) {
    const int row = rgrp + it * Cfg::kRowsPerPass;
    const float xr = xs[row], qr = qs[row];
    pa[0] += s[it].x * xr; pa[1] += s[it].y * xr; pa[2] += s[it].z * xr; pa[3] += s[it].w * xr;
    pb[0] += s[it].x * qr; pb[1] += s[it].y * qr; pb[2] += s[it].z * qr; pb[3] += s[it].w * qr;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    red[rgrp][0][col4 * 4 + e] = pa[e];
    red[rgrp][1][col4 * 4 + e] = pb[e];
  }
  __syncthreads();
  const float eta = scal[0], gamma = scal[1], xq = scal[2];
  // Column totals, residual and output; the residual goes to shared memory.
  __shared__ float rs[DV];
  for (int j = tid; j < DV; j += kT) {
    float ta = 0.f, tb = 0.f;
#pragma unroll
    for (int g = 0; g < Cfg::kRowsPerPass; ++g) {
      ta += red[g][0][j];
      tb += red[g][1][j];
    }
    const float vj = load_elem(a.v, n * DV + j, a.dtype);
    const float r = (a.rule == kFalcon1) ? vj - ta : vj;
    rs[j] = r;
    store_elem(a.o, n * DV + j, gamma * tb + eta * xq * r, a.dtype);
  }
  __syncthreads();

  // S_t = gamma S + eta x r^T, written back in place.
  const float4 r4 = make_float4(rs[col4 * 4 + 0], rs[col4 * 4 + 1], rs[col4 * 4 + 2],
                                rs[col4 * 4 + 3]);
#pragma unroll
  for (int it = 0; it < Cfg::kIters; ++it) {
    const int row = rgrp + it * Cfg::kRowsPerPass;
    const float ex = eta * xs[row];
    float4 w;
    w.x = gamma * s[it].x + ex * r4.x;
    w.y = gamma * s[it].y + ex * r4.y;
    w.z = gamma * s[it].z + ex * r4.z;
    w.w = gamma * s[it].w + ex * r4.w;
    st_stream(S + row * DV + col4 * 4, w);
  }
}

template <int M, int DV>
cudaError_t launch_mdv(const DecodeArgs& a, cudaStream_t stream) {
  decode_kernel<M, DV><<<(unsigned)a.N, DecodeCfg<M, DV>::kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int M>
cudaError_t launch_m(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.dv) {
    case 16: return launch_mdv<M, 16>(a, stream);
    case 32: return launch_mdv<M, 32>(a, stream);
    case 64: return launch_mdv<M, 64>(a, stream);
    case 128: return launch_mdv<M, 128>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.N == 0) return cudaSuccess;
  switch (a.m) {
    case 16: return launch_m<16>(a, stream);
    case 32: return launch_m<32>(a, stream);
    case 64: return launch_m<64>(a, stream);
    case 128: return launch_m<128>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace falcon
