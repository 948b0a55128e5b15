// Generic chunk-parallel forward of Falcon-1 / Falcon-1A in fp32 (CUDA cores).
//
// This path takes every supported shape and dtype (it is the one that serves
// fp32 inputs, whose tolerance needs full fp32 products) and every ragged tail.
// It runs in two launches:
//
//   1. chunk_prep_kernel, one CTA per (head, chunk), all chunks in parallel:
//      builds the chunk's write features, step sizes and log-decays and turns
//      the chunk into an affine map of the entering state S,
//          [S'; O] = Mc S + Nc,   Mc = [e^{g_C} I - Xt^T W ; Diag(e^g) Q - P W],
//                                 Nc = [Xt^T U~ ; P U~],
//      with W = T Diag(eta e^{g_-}) X and U~ = T Diag(eta) V obtained by one
//      forward substitution with the unit lower-triangular I + A (the WY/UT
//      form: one multi-right-hand-side triangular solve per chunk, as the
//      complexity table of page juhoplayground.github.io describes).  Mc and
//      Nc go to the workspace.
//   2. chunk_scan_kernel, one CTA per (head, slice of dv columns): the
//      inter-chunk recurrence, sequential over chunks.  Columns of S evolve
//      independently, so slicing dv is exact.  For the backward pass it can
//      also record the state entering every chunk (and skip o).
//
// Only non-positive exponents are ever exponentiated (the chunk-local
// log-space form of the positive-decay renormalisation, page
// hyper.ai/fr/papers/2608.27763 Section 4.4 Eq. (4.15)-(4.16)), so decay
// products that underflow stay finite.
#include "common.cuh"

namespace falcon {

__host__ __device__ inline int64_t map_floats(int m, int dv, int C) {
  return (int64_t)(m + C) * (m + dv);
}

size_t generic_workspace_bytes(int64_t BH, int64_t T, int m, int dv, int C) {
  const int64_t nch = (T + C - 1) / C;
  return (size_t)(BH * nch * map_floats(m, dv, C) * (int64_t)sizeof(float));
}

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// phi of one m-vector held by a warp; lane handles elements lane, lane+32, ...
// Writes the feature to dst (may be nullptr) and returns ||phi(u)||^2.
__device__ float warp_feature(const void* src, int64_t off, int m, int dtype, int phi,
                              float* dst) {
  float u[4];
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = threadIdx.x % 32 + 32 * e;
    u[e] = (i < m) ? load_elem(src, off + i, dtype) : 0.f;
    ss += u[e] * u[e];
  }
  ss = warp_sum(ss);
  const float scale = feature_scale(ss, m, phi);
  float out_ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = threadIdx.x % 32 + 32 * e;
    const float f = u[e] * scale;
    out_ss += f * f;
    if (i < m && dst) dst[i] = f;
  }
  return warp_sum(out_ss);
}

__global__ void __launch_bounds__(kThreads) chunk_prep_kernel(ChunkArgs a, int nchunks) {
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int m = a.m, dv = a.dv, C = a.C;
  const int64_t t0 = (int64_t)c * C;
  const int n = (int)min((int64_t)C, a.T - t0);  // valid tokens of this chunk
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  extern __shared__ float sm[];
  // X and Qf rows are padded to m + 1 floats so that the Gram loop below,
  // where a warp walks down a column, hits 32 different banks.
  const int ld = m + 1;
  float* X = sm;               // (C+1) x ld : row i = write feature of token t0+i
  float* Qf = X + (C + 1) * ld;  // C x ld  : phi(q)
  float* V = Qf + C * ld;      // C x dv
  float* Am = V + C * dv;      // C x C     : strictly lower A of I + A
  float* P = Am + C * C;       // C x C     : masked, decayed Q X^T
  float* WU = P + C * C;       // C x (m+dv): [W | U~]
  float* eta = WU + C * (m + dv);
  float* g = eta + C;   // inclusive log prefix g_i
  float* gx = g + C;    // exclusive log prefix g_{i-1}
  float* E = gx + C;    // ||x_i||^2

  const int64_t rowbase = bh * a.T;
  // Write features: X[i] = phi(k_{t0+i-1}); X[n] = phi(k_{t0+n-1}) (the next
  // segment's x_prev when this is the last chunk).  Rows past n are zero.
  for (int i = warp; i <= C; i += kWarps) {
    const int64_t t = t0 + i;  // token whose write feature this row is
    float e = 0.f;
    if (i <= n) {
      if (t >= 1) {
        e = warp_feature(a.k, (rowbase + t - 1) * m, m, a.dtype, a.phi, X + i * ld);
      } else if (a.x_prev) {
        float ss = 0.f;
        for (int j = lane; j < m; j += 32) {
          const float xv = a.x_prev[bh * m + j];
          X[j] = xv;
          ss += xv * xv;
        }
        e = warp_sum(ss);
      } else {
        for (int j = lane; j < m; j += 32) X[j] = 0.f;
      }
    } else {
      for (int j = lane; j < m; j += 32) X[i * ld + j] = 0.f;
    }
    if (lane == 0 && i < C) E[i] = e;
    if (i < C) {
      if (i < n)
        warp_feature(a.q, (rowbase + t) * m, m, a.dtype, a.phi, Qf + i * ld);
      else
        for (int j = lane; j < m; j += 32) Qf[i * ld + j] = 0.f;
    }
  }
  for (int idx = threadIdx.x; idx < C * dv; idx += kThreads) {
    const int i = idx / dv, j = idx % dv;
    V[idx] = (i < n) ? load_elem(a.v, (rowbase + t0 + i) * dv + j, a.dtype) : 0.f;
  }
  __syncthreads();
  if (a.x_last && c == nchunks - 1)
    for (int j = threadIdx.x; j < m; j += kThreads) a.x_last[bh * m + j] = X[n * ld + j];

  // Per-token step size and log-decay, then the chunk-local prefix sums.
  if (threadIdx.x < C) {
    const int i = threadIdx.x;
    float lg = 0.f, e = 0.f, gam;
    if (i < n) {
      const bool sentinel = (t0 + i == 0) && (a.x_prev == nullptr);
      e = step_eta_gamma(sentinel, E[i], a.beta[rowbase + t0 + i],
                         ridge_of(a.lambda[rowbase + t0 + i], E[i], a.ridge), a.eps, a.eps_gamma,
                         &gam, &lg);
    }
    eta[i] = e;
    g[i] = lg;  // prefix below
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float run = 0.f;
    for (int i = 0; i < C; ++i) {
      gx[i] = run;
      run += g[i];
      g[i] = run;
    }
  }
  __syncthreads();

  // A_ij = eta_i e^{g_{i-1} - g_j} <x_i, x_j> (j < i);  P_ij = e^{g_i - g_j} <q_i, x_j> (j <= i).
  for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
    const int i = idx / C, j = idx % C;
    float aij = 0.f, pij = 0.f;
    if (j <= i) {
      float dq = 0.f, dx = 0.f;
      for (int r = 0; r < m; ++r) {
        dq += Qf[i * ld + r] * X[j * ld + r];
        dx += X[i * ld + r] * X[j * ld + r];
      }
      pij = __expf(fminf(g[i] - g[j], 0.f)) * dq;
      if (j < i && a.rule == kFalcon1) aij = eta[i] * __expf(fminf(gx[i] - g[j], 0.f)) * dx;
    }
    Am[idx] = aij;
    P[idx] = pij;
  }
  // Right-hand sides [Diag(eta e^{g_-}) X | Diag(eta) V].
  for (int idx = threadIdx.x; idx < C * (m + dv); idx += kThreads) {
    const int i = idx / (m + dv), j = idx % (m + dv);
    float rhs;
    if (j < m)
      rhs = (a.rule == kFalcon1) ? eta[i] * __expf(gx[i]) * X[i * ld + j] : 0.f;
    else
      rhs = eta[i] * V[i * dv + (j - m)];
    WU[idx] = rhs;
  }
  __syncthreads();

  // Forward substitution (I + A) [W | U~] = rhs, one thread per column.
  if (a.rule == kFalcon1) {
    for (int col = threadIdx.x; col < m + dv; col += kThreads) {
      for (int i = 1; i < C; ++i) {
        float acc = WU[i * (m + dv) + col];
        for (int j = 0; j < i; ++j) acc -= Am[i * C + j] * WU[j * (m + dv) + col];
        WU[i * (m + dv) + col] = acc;
      }
    }
  }
  __syncthreads();

  // Chunk map.  Rows 0..m-1 are the state rows, rows m..m+C-1 the outputs.
  const float gC = g[C - 1];
  float* Mc = reinterpret_cast<float*>(a.workspace) + (bh * nchunks + c) * map_floats(m, dv, C);
  float* Nc = Mc + (int64_t)(m + C) * m;
  for (int idx = threadIdx.x; idx < (m + C) * (m + dv); idx += kThreads) {
    const int r = idx / (m + dv), s = idx % (m + dv);
    float acc = 0.f;
    if (r < m) {  // Xt^T [W | U~] with Xt_j = e^{g_C - g_j} x_j
      for (int j = 0; j < C; ++j)
        acc += __expf(fminf(gC - g[j], 0.f)) * X[j * ld + r] * WU[j * (m + dv) + s];
      if (s < m) acc = ((r == s) ? __expf(gC) : 0.f) - acc;
    } else {  // P [W | U~]
      const int i = r - m;
      for (int j = 0; j <= i; ++j) acc += P[i * C + j] * WU[j * (m + dv) + s];
      if (s < m) acc = __expf(g[i]) * Qf[i * ld + s] - acc;
    }
    if (s < m)
      Mc[(int64_t)r * m + s] = acc;
    else
      Nc[(int64_t)r * dv + (s - m)] = acc;
  }
}

__global__ void __launch_bounds__(kThreads)
    chunk_scan_kernel(ChunkArgs a, int nchunks, int NV, float* S_starts) {
  const int64_t bh = blockIdx.x;
  const int j0 = blockIdx.y * NV;
  const int m = a.m, dv = a.dv, C = a.C;
  const int R = m + C;
  extern __shared__ float sm[];
  float* S = sm;             // m x NV
  float* Mc = S + m * NV;    // R x m
  float* Ns = Mc + R * m;    // R x NV
  for (int idx = threadIdx.x; idx < m * NV; idx += kThreads) {
    const int r = idx / NV, j = idx % NV;
    S[idx] = a.S0 ? a.S0[(bh * m + r) * dv + j0 + j] : 0.f;
  }
  for (int c = 0; c < nchunks; ++c) {
    const float* gM = reinterpret_cast<const float*>(a.workspace) +
                      (bh * nchunks + c) * map_floats(m, dv, C);
    const float* gN = gM + (int64_t)R * m;
    if (S_starts) {  // the state entering chunk c
      float* dst = S_starts + (bh * nchunks + c) * (int64_t)m * dv;
      for (int idx = threadIdx.x; idx < m * NV; idx += kThreads)
        dst[(idx / NV) * dv + j0 + idx % NV] = S[idx];
    }
    for (int idx = threadIdx.x; idx < R * m; idx += kThreads) Mc[idx] = gM[idx];
    for (int idx = threadIdx.x; idx < R * NV; idx += kThreads) {
      const int r = idx / NV, j = idx % NV;
      Ns[idx] = gN[(int64_t)r * dv + j0 + j];
    }
    __syncthreads();
    // [S'; O] = Mc S + Nc ; accumulate into Ns.
    for (int idx = threadIdx.x; idx < R * NV; idx += kThreads) {
      const int r = idx / NV, j = idx % NV;
      float acc = Ns[idx];
      for (int kk = 0; kk < m; ++kk) acc += Mc[r * m + kk] * S[kk * NV + j];
      Ns[idx] = acc;
    }
    __syncthreads();
    const int64_t t0 = (int64_t)c * C;
    for (int idx = threadIdx.x; idx < R * NV; idx += kThreads) {
      const int r = idx / NV, j = idx % NV;
      if (r < m) {
        S[idx] = Ns[idx];
      } else if (a.o) {
        const int64_t t = t0 + (r - m);
        if (t < a.T) store_elem(a.o, (bh * a.T + t) * dv + j0 + j, Ns[idx], a.dtype);
      }
    }
    __syncthreads();
  }
  if (a.S_out) {
    for (int idx = threadIdx.x; idx < m * NV; idx += kThreads) {
      const int r = idx / NV, j = idx % NV;
      a.S_out[(bh * m + r) * dv + j0 + j] = S[idx];
    }
  }
}

}  // namespace

cudaError_t launch_generic_chunked(const ChunkArgs& a, cudaStream_t stream, float* S_starts) {
  const int nchunks = (int)((a.T + a.C - 1) / a.C);
  const int m = a.m, dv = a.dv, C = a.C;
  const size_t prep_smem =
      sizeof(float) * ((size_t)(C + 1) * (m + 1) + (size_t)C * (m + 1) + (size_t)C * dv + 2 * (size_t)C * C +
                       (size_t)C * (m + dv) + 4 * (size_t)C);
  cudaError_t err = cudaFuncSetAttribute(chunk_prep_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)prep_smem);
  if (err != cudaSuccess) return err;
  dim3 g1(nchunks, (unsigned)a.BH);
  chunk_prep_kernel<<<g1, kThreads, prep_smem, stream>>>(a, nchunks);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  const int NV = dv < 32 ? dv : 32;
  const size_t scan_smem = sizeof(float) * ((size_t)m * NV + (size_t)(m + C) * m + (size_t)(m + C) * NV);
  err = cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)scan_smem);
  if (err != cudaSuccess) return err;
  dim3 g2((unsigned)a.BH, dv / NV);
  chunk_scan_kernel<<<g2, kThreads, scan_smem, stream>>>(a, nchunks, NV, S_starts);
  return cudaGetLastError();
}

}  // namespace falcon
