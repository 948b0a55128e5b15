// Falcon-1A with the normalised read (page hyper.ai/fr/papers/2608.27763,
// Section 2.2, Eq. (2.1)-(2.3)):
//
//     o_t = S_t^T phi(q_t) / (z_t^T phi(q_t) + eps_attn),
//     z_t = gamma_t z_{t-1} + eta_t x_t,
//
// the normaliser z taking the numerator's gain eta_t and clamped decay gamma_t
// (the Falcon-1A version of Eq. (2.3) is deferred to an appendix the pages do
// not include; at lambda = 0 and unit gain this is Eq. (2.3) exactly).
//
// The numerator is the Falcon-1A chunked forward (the tensor-core or generic
// path).  The denominator runs beside it in three fp32 kernels, the chunk
// form of the z recurrence (z is the state column a constant unit target
// would write):
//   1. norm_chunk_kernel, one CTA per (head, chunk): the tokens' phi scales,
//      eta_t and log gamma_t; the in-chunk normaliser y_t (z started from 0
//      at the chunk), its read r_t = <phi(q_t), y_t>, the prefix decays
//      e^{g_t}, and the chunk's increment y_C and decay e^{g_C};
//   2. norm_chain_kernel, one CTA per head: z entering every chunk,
//      z_{c+1} = e^{g_C} z_c + y_C, and z_T;
//   3. norm_apply_kernel, one CTA per (head, chunk): den_t = e^{g_t}
//      <phi(q_t), z_c> + r_t and o_t <- o_t / (den_t + eps_attn) in place.
// Every exponential has a non-positive argument (decays only).
#include <cuda_bf16.h>

#include "common.cuh"

namespace falcon {
namespace {

constexpr int kNormThreads = 128;

// Workspace of the denominator, per (head, chunk): z entering the chunk (m),
// the chunk's increment y_C (m), its decay e^{g_C} (1, padded to 4), and per
// token e^{g_t}, phi's scale of q_t and r_t (C each).
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

// One CTA per (chunk, head).  Shared: the chunk's write features x (C x m,
// raw, row 0 = the token before the chunk) and raw q rows (C x m), then
// per-token scalars (eta, log gamma, phi's scales of x and q, gamma).
__global__ void __launch_bounds__(kNormThreads)
    norm_chunk_kernel(ChunkArgs a, int nchunks, NormLayout L, float* ws) {
  extern __shared__ float sh[];
  const int C = a.C, m = a.m;
  float* xs = sh;               // [C][m] raw write-feature rows
  float* qs = xs + C * m;       // [C][m] raw q rows, then the read products
  float* eta = qs + C * m;      // [C]
  float* lg = eta + C;          // [C] log gamma
  float* sx = lg + C;           // [C] phi's scale of x_t
  float* sq = sx + C;           // [C] phi's scale of q_t
  float* gm = sq + C;           // [C] gamma_t
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int64_t t0 = (int64_t)c * C;
  const int n = (int)min((int64_t)C, a.T - t0);
  const int64_t rowbase = bh * a.T;
  // rows: x_r = k_{t0 + r - 1} (r = 0: x_prev or the sentinel at the sequence
  // start), q_r = q_{t0 + r}
  for (int e = tid; e < C * m; e += blockDim.x) {
    const int r = e / m, i = e % m;
    float xv = 0.f, qv = 0.f;
    if (r < n) {
      const int64_t tk = t0 + r - 1;
      if (tk >= 0)
        xv = load_elem(a.k, (rowbase + tk) * m + i, a.dtype);
      else if (a.x_prev)
        xv = a.x_prev[bh * m + i];
      qv = load_elem(a.q, (rowbase + t0 + r) * m + i, a.dtype);
    }
    xs[e] = xv;
    qs[e] = qv;
  }
  __syncthreads();
  // per-token scalars: phi's scales (x_prev is already a feature), E_t, eta_t,
  // log gamma_t (the sentinel: eta = 0 at the sequence start without x_prev)
  for (int r = tid; r < C; r += blockDim.x) {
    float e_t = 0.f, lgt = 0.f, s_x = 1.f, s_q = 1.f, gam = 1.f;
    if (r < n) {
      float ssx = 0.f, ssq = 0.f;
      for (int i = 0; i < m; ++i) {
        ssx = fmaf(xs[r * m + i], xs[r * m + i], ssx);
        ssq = fmaf(qs[r * m + i], qs[r * m + i], ssq);
      }
      const bool carried = t0 + r == 0 && a.x_prev != nullptr;
      s_x = carried ? 1.f : feature_scale(ssx, m, a.phi);
      s_q = feature_scale(ssq, m, a.phi);
      const float E = ssx * s_x * s_x;
      const bool sentinel = t0 + r == 0 && a.x_prev == nullptr;
      e_t = step_eta_gamma(sentinel, E, a.beta[rowbase + t0 + r],
                           ridge_of(a.lambda[rowbase + t0 + r], E, a.ridge), a.eps, a.eps_gamma,
                           &gam, &lgt);
    }
    eta[r] = e_t;
    lg[r] = lgt;
    sx[r] = s_x;
    sq[r] = s_q;
    gm[r] = gam;
  }
  __syncthreads();
  const size_t mi = (size_t)(bh * nchunks + c);
  // in-chunk normaliser, one thread per feature dimension: y_t = gamma_t
  // y_{t-1} + eta_t x_t, and the products y_t[i] phi(q_t)[i] over q's rows
  if (tid < m) {
    float y = 0.f;
    for (int r = 0; r < n; ++r) {
      y = fmaf(gm[r], y, eta[r] * sx[r] * xs[r * m + tid]);
      qs[r * m + tid] = y * (sq[r] * qs[r * m + tid]);
    }
    ws[L.inc() + mi * m + tid] = y;
  }
  __syncthreads();
  // r_t, e^{g_t} (inclusive prefix of log gamma, one thread per token), e^{g_C}
  for (int r = tid; r < C; r += blockDim.x) {
    float acc = 0.f, g = 0.f;
    if (r < n) {
      for (int i = 0; i < m; ++i) acc += qs[r * m + i];
      for (int s = 0; s <= r; ++s) g += lg[s];
    }
    ws[L.rd() + mi * C + r] = acc;
    ws[L.eg() + mi * C + r] = __expf(g);
    ws[L.nq() + mi * C + r] = sq[r];
    if (r == n - 1) ws[L.dec() + mi * 4] = __expf(g);
  }
}

// One CTA per head: z entering every chunk, and z_T.
__global__ void __launch_bounds__(kNormThreads)
    norm_chain_kernel(int64_t BH, int m, int nchunks, NormLayout L, float* ws, const float* z0,
                      float* z_out) {
  const int64_t bh = blockIdx.x;
  const int i = threadIdx.x;
  if (i >= m) return;
  float z = z0 ? z0[bh * m + i] : 0.f;
  const size_t m0 = (size_t)(bh * nchunks);
  for (int c = 0; c < nchunks; ++c) {
    ws[L.zin() + (m0 + c) * m + i] = z;
    z = fmaf(ws[L.dec() + (m0 + c) * 4], z, ws[L.inc() + (m0 + c) * m + i]);
  }
  if (z_out) z_out[bh * m + i] = z;
}

// One CTA per (chunk, head), one warp per token at a time: den_t and o_t /= .
__global__ void __launch_bounds__(kNormThreads)
    norm_apply_kernel(ChunkArgs a, int nchunks, NormLayout L, const float* ws, float eps_attn) {
  const int C = a.C, m = a.m, dv = a.dv;
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = (int64_t)c * C;
  const int n = (int)min((int64_t)C, a.T - t0);
  const size_t mi = (size_t)(bh * nchunks + c);
  const float* zc = ws + L.zin() + mi * m;
  for (int r = warp; r < n; r += blockDim.x / 32) {
    const int64_t row = bh * a.T + t0 + r;
    float dot = 0.f;
    for (int i = lane; i < m; i += 32) dot = fmaf(load_elem(a.q, row * m + i, a.dtype), zc[i], dot);
    dot = warp_sum(dot);
    const float den = ws[L.eg() + mi * C + r] * ws[L.nq() + mi * C + r] * dot +
                      ws[L.rd() + mi * C + r] + eps_attn;
    for (int j = lane; j < dv; j += 32) {
      const int64_t e = row * dv + j;
      store_elem(a.o, e, load_elem(a.o, e, a.dtype) / den, a.dtype);
    }
  }
}

}  // namespace

size_t norm_workspace_bytes(int64_t BH, int64_t T, int m, int C) {
  const int64_t nch = (T + C - 1) / C;
  const NormLayout L{BH * nch, m, C};
  return ((L.floats() * sizeof(float) + 255) / 256) * 256;
}

cudaError_t launch_normalizer(const ChunkArgs& a, const float* z0, float* z_out, float eps_attn,
                              float* ws, cudaStream_t stream) {
  const int nchunks = (int)((a.T + a.C - 1) / a.C);
  const NormLayout L{a.BH * nchunks, a.m, a.C};
  const size_t smem = sizeof(float) * (size_t)(2 * a.C * a.m + 5 * a.C);
  cudaError_t e = cudaFuncSetAttribute(norm_chunk_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  norm_chunk_kernel<<<dim3(nchunks, (unsigned)a.BH), kNormThreads, smem, stream>>>(a, nchunks, L,
                                                                                   ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  norm_chain_kernel<<<(unsigned)a.BH, kNormThreads, 0, stream>>>(a.BH, a.m, nchunks, L, ws, z0,
                                                                   z_out);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  norm_apply_kernel<<<dim3(nchunks, (unsigned)a.BH), kNormThreads, 0, stream>>>(a, nchunks, L, ws,
                                                                                eps_attn);
  return cudaGetLastError();
}

}  // namespace falcon
