// Backward pass of the chunk-parallel Falcon-1 / Falcon-1A forward (fp32,
// CUDA cores).
//
// The pages say that training differentiates through the update, so that the
// slow weights producing q, k, v, beta and lambda learn (page
// hyper.ai/fr/papers/2608.27763, Section 3, "Implicit fast-memory
// objective"), through the log-decay renormalisation and the normalised step
// size (Section 4.6, "Backward pass"; its appendix is not on the pages).  This
// file computes the gradient of L = <dO, o> + <dS_T, S_T> + <dx_last, x_last>
// with respect to every input, in the chunk form:
//
//   1. the forward's chunk maps [S'; O] = Mc S + Nc (chunk_prep_kernel of the
//      generic path) and a forward scan that records the state S_c entering
//      every chunk (recomputation instead of storing per-token states);
//   2. bwd_scan_kernel, one CTA per (head, slice of dv columns): the reverse
//      scan of the state cotangent, dS_c = Mc^T [dS_{c+1}; dO_c] (the
//      transposed chunk map), newest chunk first, recording the cotangent of
//      the state leaving every chunk; dS0 is its final value;
//   3. bwd_grad_kernel, one CTA per (head, chunk), all chunks in parallel:
//      with S_c and the leaving cotangent dS', the chunk's own gradients
//        R  = Diag(eta) V - Diag(eta e^{g_-}) X S,  U = (I + A)^{-1} R,
//        dU = P^T dO + Diag(e^{g_C - g}) X dS',     dR = (I + A)^{-T} dU,
//        dA = -(dR U^T) (j < i),  dP = (dO U^T) (j <= i),  dV = Diag(eta) dR,
//        dQ = Diag(e^g) dO S^T + (dP o E) X,
//        dX = -Diag(eta e^{g_-}) dR S^T + (dP o E)^T Q + Diag(e^{g_C - g}) U dS'^T
//             + (dK + dK^T) X + 2 Diag(dE) X,
//      the log-prefix cotangent dg (every e^{...} factor), its suffix sums
//      d log gamma, and the chain through the clamp, eta = beta / (E +
//      lambda + eps) and the ridge (Falcon-1A: A = 0 and R = Diag(eta) V);
//      dq = J_phi(q)^T dQ is written here, dX goes to the workspace;
//   4. bwd_feature_kernel: dk_t = J_phi(k_t)^T dX_{t+1} (dx_last for the last
//      token), dx_prev = dX_1 when the call carried x_prev.
// The clamped branch of the decay is a constant (no gradient through alpha);
// the sentinel token passes no gradient to beta_1, lambda_1.
//
// For bf16 inputs with m = dv = 64 and chunk 64, steps 1-3 run on the
// tensor cores instead: the tensor-core forward (maps and scan, recording the
// chunk-start states), its reverse scan (chunk_tc_bwd.cu) and the tensor-core
// chunk kernel; step 4 is shared.
#include "common.cuh"

namespace falcon {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__host__ __device__ inline int64_t align_floats(int64_t n) { return (n + 63) & ~int64_t(63); }

struct BwdLayout {  // float offsets inside the workspace
  int64_t maps, S_starts, dS_ends, dX, o, S_out, total;
};

__host__ __device__ inline BwdLayout bwd_layout(int64_t BH, int64_t T, int m, int dv, int C) {
  const int64_t nch = (T + C - 1) / C;
  BwdLayout L;
  L.maps = 0;
  L.S_starts = align_floats(L.maps + BH * nch * (int64_t)(m + C) * (m + dv));
  L.dS_ends = align_floats(L.S_starts + BH * nch * (int64_t)m * dv);
  L.dX = align_floats(L.dS_ends + BH * nch * (int64_t)m * dv);
  L.total = align_floats(L.dX + BH * T * (int64_t)m);
  L.o = L.S_out = L.total;
  return L;
}

// Tensor-core path: the forward's bf16 maps, then the state and cotangent
// buffers, then room for the recomputed forward's o (its tensor map needs a
// buffer; the recording scan writes no o) and S_T (written, not used).
BwdLayout tc_bwd_layout(int64_t BH, int64_t T) {
  const int64_t nch = (T + 63) / 64;
  BwdLayout L;
  L.maps = 0;
  L.S_starts = align_floats((int64_t)((tc_workspace_bytes(64, BH, T) + 3) / 4));
  L.dS_ends = align_floats(L.S_starts + BH * nch * 4096);
  L.dX = align_floats(L.dS_ends + BH * nch * 4096);  // row 0 of every chunk's dX
  L.o = align_floats(L.dX + BH * nch * 64);
  L.S_out = align_floats(L.o + BH * T * 32);  // bf16 o: 32 floats per row
  L.total = align_floats(L.S_out + BH * 4096);
  return L;
}

bool use_tc_bwd(const ChunkArgs& a) {
  return tc_bwd_applies(a.dtype, a.m, a.dv, a.C) &&
         tc_path_applies(a.dtype, a.m, a.dv, a.C, a.BH, a.T);
}

// phi of one m-vector (m <= 128) held by a warp, lane owning elements lane +
// 32 e; writes it to dst and returns ||phi(u)||^2.  The scale is the
// forward's (feature_scale).
__device__ float row_feature(const void* src, int64_t off, int m, int dtype, int phi, float* dst) {
  const int lane = threadIdx.x % 32;
  float u[4], ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = lane + 32 * e;
    u[e] = i < m ? load_elem(src, off + i, dtype) : 0.f;
    ss += u[e] * u[e];
  }
  const float s = feature_scale(warp_sum(ss), m, phi);
  float out = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = lane + 32 * e;
    if (i < m) dst[i] = u[e] * s;
    out += u[e] * s * u[e] * s;
  }
  return warp_sum(out);
}

// J_phi(u)^T g for one m-vector held by a warp (u raw, g and the result in
// lane-strided registers).  l2: phi = u / n, n = max(||u||, 1e-12);
// RMSNorm: phi = u s, s = (||u||^2 / m + eps_rms)^(-1/2).
__device__ void feature_vjp(const float* u, const float* g, int m, int phi, float* out) {
  if (phi == FALCON_PHI_IDENTITY) {
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = g[e];
    return;
  }
  float ss = 0.f, ug = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    ss += u[e] * u[e];
    ug += u[e] * g[e];
  }
  ss = warp_sum(ss);
  ug = warp_sum(ug);
  if (phi == FALCON_PHI_L2) {
    const float nrm = sqrtf(ss);
    if (nrm < 1e-12f) {
#pragma unroll
      for (int e = 0; e < 4; ++e) out[e] = g[e] * 1e12f;
    } else {
      const float inv = 1.f / nrm;
      const float pg = ug * inv;  // <phi, g>
#pragma unroll
      for (int e = 0; e < 4; ++e) out[e] = (g[e] - u[e] * inv * pg) * inv;
    }
  } else {
    const float s = rsqrtf(ss / (float)m + kEpsRms);
    const float c = s * s * s * ug / (float)m;
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = s * g[e] - c * u[e];
  }
}

// ---- 2. reverse scan of the state cotangent -------------------------------
__global__ void __launch_bounds__(kThreads)
    bwd_scan_kernel(BwdArgs b, int nchunks, int NV, const float* maps, float* dS_ends) {
  const ChunkArgs& a = b.f;
  const int64_t bh = blockIdx.x;
  const int j0 = blockIdx.y * NV;
  const int m = a.m, dv = a.dv, C = a.C;
  const int R = m + C;
  extern __shared__ float sm[];
  float* dS = sm;            // m x NV
  float* Mc = dS + m * NV;   // R x m
  float* St = Mc + R * m;    // R x NV: [dS'; dO_c]
  for (int idx = threadIdx.x; idx < m * NV; idx += kThreads) {
    const int r = idx / NV, j = idx % NV;
    dS[idx] = b.dS_T ? b.dS_T[(bh * m + r) * dv + j0 + j] : 0.f;
  }
  __syncthreads();
  for (int c = nchunks - 1; c >= 0; --c) {
    float* dst = dS_ends + (bh * nchunks + c) * (int64_t)m * dv;
    const float* gM = maps + (bh * nchunks + c) * (int64_t)R * (m + dv);
    for (int idx = threadIdx.x; idx < m * NV; idx += kThreads) {
      dst[(idx / NV) * dv + j0 + idx % NV] = dS[idx];
      St[idx] = dS[idx];
    }
    for (int idx = threadIdx.x; idx < R * m; idx += kThreads) Mc[idx] = gM[idx];
    const int64_t t0 = (int64_t)c * C;
    for (int idx = threadIdx.x; idx < C * NV; idx += kThreads) {
      const int i = idx / NV, j = idx % NV;
      const int64_t t = t0 + i;
      St[m * NV + idx] = t < a.T ? load_elem(b.dO, (bh * a.T + t) * dv + j0 + j, a.dtype) : 0.f;
    }
    __syncthreads();
    // dS <- Mc^T [dS'; dO_c]
    for (int idx = threadIdx.x; idx < m * NV; idx += kThreads) {
      const int kk = idx / NV, j = idx % NV;
      float acc = 0.f;
      for (int r = 0; r < R; ++r) acc += Mc[r * m + kk] * St[r * NV + j];
      dS[idx] = acc;
    }
    __syncthreads();
  }
  if (b.dS0)
    for (int idx = threadIdx.x; idx < m * NV; idx += kThreads)
      b.dS0[(bh * m + idx / NV) * dv + j0 + idx % NV] = dS[idx];
}

// ---- 3. per-chunk gradients ------------------------------------------------
enum : int { kLive = 1, kClamped = 2 };

__global__ void __launch_bounds__(kThreads)
    bwd_grad_kernel(BwdArgs b, int nchunks, const float* S_starts, const float* dS_ends,
                    float* dXw) {
  const ChunkArgs& a = b.f;
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int m = a.m, dv = a.dv, C = a.C;
  const int64_t T = a.T, t0 = (int64_t)c * C, rowbase = bh * T;
  const int n = (int)min((int64_t)C, T - t0);
  const bool f1 = a.rule == kFalcon1;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float* S = S_starts + (bh * nchunks + c) * (int64_t)m * dv;  // state entering
  const float* dSp = dS_ends + (bh * nchunks + c) * (int64_t)m * dv;  // cotangent leaving

  extern __shared__ float sm[];
  const int ld = m + 1;
  float* X = sm;                 // C x ld   write features
  float* Q = X + C * ld;         // C x ld   phi(q)
  float* A = Q + C * ld;         // C x C    strictly lower A (Falcon-1)
  float* P = A + C * C;          // C x C    decayed, masked Q X^T
  float* dA = P + C * C;         // C x C
  float* dP = dA + C * C;        // C x C
  float* U = dP + C * C;         // C x dv   R, then U
  float* dR = U + C * dv;        // C x dv   dU, then dR
  float* eta = dR + C * dv;
  float* g = eta + C;            // inclusive log prefix
  float* gx = g + C;             // exclusive log prefix
  float* E = gx + C;             // ||x_i||^2
  float* lame = E + C;           // lambda_t used by the recurrence
  float* den = lame + C;
  float* gam = den + C;
  float* deta = gam + C;
  float* dg = deta + C;
  float* dE = dg + C;
  float* xy = dE + C;            // <x_i, S dR_i>
  float* xw = xy + C;            // <x_i, dS' U_i>
  float* sAr = xw + C;           // sum_j dA_ij A_ij
  float* sAc = sAr + C;          // sum_i dA_ij A_ij (column j)
  float* red = sAc + C;          // [0]: <dS', S>_F
  int* flag = reinterpret_cast<int*>(red + 4);

  // features: X_i = phi(k_{t-1}) (x_prev or the sentinel zero at t = 0)
  for (int i = warp; i < C; i += kWarps) {
    const int64_t t = t0 + i;
    float e = 0.f;
    if (i < n && t >= 1) {
      e = row_feature(a.k, (rowbase + t - 1) * m, m, a.dtype, a.phi, X + i * ld);
    } else if (i < n && a.x_prev) {
      float ss = 0.f;
      for (int r = lane; r < m; r += 32) {
        const float xv = a.x_prev[bh * m + r];
        X[i * ld + r] = xv;
        ss += xv * xv;
      }
      e = warp_sum(ss);
    } else {
      for (int r = lane; r < m; r += 32) X[i * ld + r] = 0.f;
    }
    if (i < n)
      row_feature(a.q, (rowbase + t) * m, m, a.dtype, a.phi, Q + i * ld);
    else
      for (int r = lane; r < m; r += 32) Q[i * ld + r] = 0.f;
    if (lane == 0) E[i] = e;
  }
  if (threadIdx.x == 0) red[0] = 0.f;
  __syncthreads();
  // per-token scalars exactly as the forward forms them
  if (threadIdx.x < C) {
    const int i = threadIdx.x;
    float et = 0.f, gm = 1.f, lg = 0.f, le = 0.f, d = 1.f;
    int fl = 0;
    if (i < n) {
      const int64_t t = t0 + i;
      const bool sentinel = (t == 0) && (a.x_prev == nullptr);
      le = ridge_of(a.lambda[rowbase + t], E[i], a.ridge);
      d = E[i] + le + a.eps;
      et = step_eta_gamma(sentinel, E[i], a.beta[rowbase + t], le, a.eps, a.eps_gamma, &gm, &lg);
      if (!sentinel && d > 0.f) fl |= kLive;
      if (et * le >= 1.f - a.eps_gamma) fl |= kClamped;
    }
    eta[i] = et;
    gam[i] = gm;
    g[i] = lg;
    lame[i] = le;
    den[i] = d;
    flag[i] = fl;
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
  const float gC = g[C - 1];

  // A and P, as the forward forms them
  for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
    const int i = idx / C, j = idx % C;
    float aij = 0.f, pij = 0.f;
    if (j <= i) {
      float dq = 0.f, dx = 0.f;
      for (int r = 0; r < m; ++r) {
        dq += Q[i * ld + r] * X[j * ld + r];
        dx += X[i * ld + r] * X[j * ld + r];
      }
      pij = __expf(fminf(g[i] - g[j], 0.f)) * dq;
      if (j < i && f1) aij = eta[i] * __expf(fminf(gx[i] - g[j], 0.f)) * dx;
    }
    A[idx] = aij;
    P[idx] = pij;
  }
  // R = Diag(eta) V - Diag(eta e^{g_-}) X S
  for (int idx = threadIdx.x; idx < C * dv; idx += kThreads) {
    const int i = idx / dv, col = idx % dv;
    float r = 0.f;
    if (i < n) {
      r = eta[i] * load_elem(a.v, (rowbase + t0 + i) * dv + col, a.dtype);
      if (f1) {
        float xs = 0.f;
        for (int kk = 0; kk < m; ++kk) xs += X[i * ld + kk] * S[kk * dv + col];
        r -= eta[i] * __expf(gx[i]) * xs;
      }
    }
    U[idx] = r;
  }
  __syncthreads();
  // U = (I + A)^{-1} R: forward substitution, one thread per column
  if (f1)
    for (int col = threadIdx.x; col < dv; col += kThreads)
      for (int i = 1; i < n; ++i) {
        float acc = U[i * dv + col];
        for (int j = 0; j < i; ++j) acc -= A[i * C + j] * U[j * dv + col];
        U[i * dv + col] = acc;
      }
  __syncthreads();
  // dU = P^T dO + Diag(e^{g_C - g}) X dS';  dP = dO U^T (j <= i)
  for (int idx = threadIdx.x; idx < C * dv; idx += kThreads) {
    const int i = idx / dv, col = idx % dv;
    float acc = 0.f;
    if (i < n) {
      for (int ip = i; ip < n; ++ip)
        acc += P[ip * C + i] * load_elem(b.dO, (rowbase + t0 + ip) * dv + col, a.dtype);
      float xd = 0.f;
      for (int kk = 0; kk < m; ++kk) xd += X[i * ld + kk] * dSp[kk * dv + col];
      acc += __expf(fminf(gC - g[i], 0.f)) * xd;
    }
    dR[idx] = acc;
  }
  for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
    const int i = idx / C, j = idx % C;
    float acc = 0.f;
    if (j <= i && i < n)
      for (int col = 0; col < dv; ++col)
        acc += load_elem(b.dO, (rowbase + t0 + i) * dv + col, a.dtype) * U[j * dv + col];
    dP[idx] = acc;
  }
  __syncthreads();
  // dR = (I + A)^{-T} dU: back substitution, one thread per column
  if (f1)
    for (int col = threadIdx.x; col < dv; col += kThreads)
      for (int i = n - 2; i >= 0; --i) {
        float acc = dR[i * dv + col];
        for (int j = i + 1; j < n; ++j) acc -= A[j * C + i] * dR[j * dv + col];
        dR[i * dv + col] = acc;
      }
  __syncthreads();
  // dA = -dR U^T (j < i);  dV = Diag(eta) dR
  for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
    const int i = idx / C, j = idx % C;
    float acc = 0.f;
    if (f1 && j < i && i < n)
      for (int col = 0; col < dv; ++col) acc -= dR[i * dv + col] * U[j * dv + col];
    dA[idx] = acc;
  }
  for (int idx = threadIdx.x; idx < n * dv; idx += kThreads) {
    const int i = idx / dv, col = idx % dv;
    store_elem(b.dv, (rowbase + t0 + i) * dv + col, eta[i] * dR[idx], a.dtype);
  }
  // <dS', S>_F
  {
    float acc = 0.f;
    for (int idx = threadIdx.x; idx < m * dv; idx += kThreads) acc += dSp[idx] * S[idx];
    acc = warp_sum(acc);
    if (lane == 0) atomicAdd(&red[0], acc);
  }
  __syncthreads();

  // Row quantities, one warp per row i: the step-size cotangent deta_i and
  // the pieces of the log-prefix cotangent.
  for (int i = warp; i < C; i += kWarps) {
    float rv = 0.f, xyi = 0.f, qz = 0.f, xwi = 0.f;
    if (i < n) {
      for (int col = lane; col < dv; col += 32) {
        float xs = 0.f, qs = 0.f, xd = 0.f;
        for (int kk = 0; kk < m; ++kk) {
          const float s = S[kk * dv + col];
          xs += X[i * ld + kk] * s;
          qs += Q[i * ld + kk] * s;
          xd += X[i * ld + kk] * dSp[kk * dv + col];
        }
        const float dRi = dR[i * dv + col];
        rv += dRi * load_elem(a.v, (rowbase + t0 + i) * dv + col, a.dtype);
        xyi += dRi * xs;
        qz += load_elem(b.dO, (rowbase + t0 + i) * dv + col, a.dtype) * qs;
        xwi += U[i * dv + col] * xd;
      }
    }
    float sar = 0.f, sac = 0.f, spr = 0.f, spc = 0.f;
    for (int j = lane; j < C; j += 32) {
      sar += dA[i * C + j] * A[i * C + j];
      sac += dA[j * C + i] * A[j * C + i];
      spr += dP[i * C + j] * P[i * C + j];
      spc += dP[j * C + i] * P[j * C + i];
    }
    rv = warp_sum(rv);
    xyi = warp_sum(xyi);
    qz = warp_sum(qz);
    xwi = warp_sum(xwi);
    sar = warp_sum(sar);
    sac = warp_sum(sac);
    spr = warp_sum(spr);
    spc = warp_sum(spc);
    if (lane == 0) {
      float de = rv;
      if (f1) {
        de -= __expf(gx[i]) * xyi;
        if (eta[i] != 0.f) de += sar / eta[i];  // sum_j dA_ij e^{g_{i-1} - g_j} <x_i, x_j>
      }
      deta[i] = de;
      xy[i] = xyi;
      xw[i] = __expf(fminf(gC - g[i], 0.f)) * xwi;
      sAr[i] = sar;
      sAc[i] = sac;
      // terms of dg that sit at index i itself
      dg[i] = __expf(g[i]) * qz + spr - spc - xw[i] - (f1 ? sac : 0.f);
    }
  }
  __syncthreads();
  // the rest of dg (terms at index i - 1 and at C - 1), then the suffix sums
  // d log gamma_r = sum_{i >= r} dg_i and the scalar chain of every token
  if (threadIdx.x == 0) {
    float tail = __expf(gC) * red[0];
    for (int j = 0; j < C; ++j) tail += xw[j];
    dg[C - 1] += tail;
    if (f1)
      for (int i = 1; i < C; ++i) dg[i - 1] += -eta[i] * __expf(gx[i]) * xy[i] + sAr[i];
    float run = 0.f;
    for (int i = C - 1; i >= 0; --i) {
      run += dg[i];
      dg[i] = run;
    }
  }
  __syncthreads();
  if (threadIdx.x < C) {
    const int i = threadIdx.x;
    float dEi = 0.f;
    if (i < n) {
      float db = 0.f, dl_in = 0.f;
      if (flag[i] & kLive) {
        float de = deta[i], dl = 0.f;
        if (!(flag[i] & kClamped)) {
          const float dal = -dg[i] / gam[i];
          de += lame[i] * dal;
          dl += eta[i] * dal;
        }
        db = de / den[i];
        const float dden = -de * eta[i] / den[i];
        dEi = dden;
        dl += dden;
        if (a.ridge == FALCON_RIDGE_SCALED) {
          dl_in = dl * E[i];
          dEi += dl * a.lambda[rowbase + t0 + i];
        } else {
          dl_in = dl;
        }
      }
      b.dbeta[rowbase + t0 + i] = db;
      b.dlambda[rowbase + t0 + i] = dl_in;
    }
    dE[i] = dEi;
  }
  __syncthreads();

  // dX (to the workspace; dk is formed from it by bwd_feature_kernel)
  for (int idx = threadIdx.x; idx < n * m; idx += kThreads) {
    const int i = idx / m, r = idx % m;
    float y = 0.f, w2 = 0.f;
    for (int col = 0; col < dv; ++col) {
      if (f1) y += S[r * dv + col] * dR[i * dv + col];
      w2 += dSp[r * dv + col] * U[i * dv + col];
    }
    float acc = __expf(fminf(gC - g[i], 0.f)) * w2 + 2.f * dE[i] * X[i * ld + r];
    if (f1) acc -= eta[i] * __expf(gx[i]) * y;
    for (int ip = i; ip < n; ++ip)
      acc += dP[ip * C + i] * __expf(fminf(g[ip] - g[i], 0.f)) * Q[ip * ld + r];
    if (f1) {
      for (int j = 0; j < i; ++j)  // dK_ij, j < i
        acc += dA[i * C + j] * eta[i] * __expf(fminf(gx[i] - g[j], 0.f)) * X[j * ld + r];
      for (int j = i + 1; j < n; ++j)  // dK_ji, i < j
        acc += dA[j * C + i] * eta[j] * __expf(fminf(gx[j] - g[i], 0.f)) * X[j * ld + r];
    }
    dXw[(rowbase + t0 + i) * m + r] = acc;
  }
  // dq = J_phi(q)^T dQ, dQ = Diag(e^g) dO S^T + (dP o E) X; one warp per row
  for (int i = warp; i < n; i += kWarps) {
    float gq[4], u[4], out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = lane + 32 * e;
      gq[e] = 0.f;
      u[e] = 0.f;
      if (r < m) {
        float z = 0.f;
        for (int col = 0; col < dv; ++col)
          z += S[r * dv + col] * load_elem(b.dO, (rowbase + t0 + i) * dv + col, a.dtype);
        float acc = __expf(g[i]) * z;
        for (int j = 0; j <= i; ++j)
          acc += dP[i * C + j] * __expf(fminf(g[i] - g[j], 0.f)) * X[j * ld + r];
        gq[e] = acc;
        u[e] = load_elem(a.q, (rowbase + t0 + i) * m + r, a.dtype);
      }
    }
    feature_vjp(u, gq, m, a.phi, out);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = lane + 32 * e;
      if (r < m) store_elem(b.dq, (rowbase + t0 + i) * m + r, out[e], a.dtype);
    }
  }
}

// ---- 4. dk and dx_prev -----------------------------------------------------
__global__ void __launch_bounds__(kThreads) bwd_feature_kernel(BwdArgs b, const float* dXw) {
  const ChunkArgs& a = b.f;
  const int m = a.m;
  const int lane = threadIdx.x % 32;
  const int64_t rows = a.BH * a.T;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32; row < rows;
       row += (int64_t)gridDim.x * kWarps) {
    const int64_t bh = row / a.T, t = row % a.T;
    float u[4], gk[4], out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = lane + 32 * e;
      u[e] = gk[e] = 0.f;
      if (r < m) {
        u[e] = load_elem(a.k, row * m + r, a.dtype);
        if (t + 1 < a.T)
          gk[e] = dXw[(row + 1) * m + r];
        else if (b.dx_last)
          gk[e] = b.dx_last[bh * m + r];
      }
    }
    feature_vjp(u, gk, m, a.phi, out);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = lane + 32 * e;
      if (r < m) store_elem(b.dk, row * m + r, out[e], a.dtype);
    }
    if (t == 0 && b.dx_prev)
      for (int r = lane; r < m; r += 32)
        b.dx_prev[bh * m + r] = a.x_prev ? dXw[row * m + r] : 0.f;
  }
}

}  // namespace

cudaError_t launch_generic_grad(const BwdArgs& b, int nchunks, const float* S_starts,
                                const float* dS_ends, float* dXw, cudaStream_t stream);

size_t bwd_workspace_bytes(int dtype, int64_t BH, int64_t T, int m, int dv, int C) {
  const bool tc = tc_bwd_applies(dtype, m, dv, C) && tc_path_applies(dtype, m, dv, C, BH, T);
  return (size_t)(tc ? tc_bwd_layout(BH, T) : bwd_layout(BH, T, m, dv, C)).total * sizeof(float);
}

cudaError_t launch_bwd_chunked(const BwdArgs& b, int* err, cudaStream_t stream) {
  const ChunkArgs& a = b.f;
  const int m = a.m, dv = a.dv, C = a.C;
  const int nchunks = (int)((a.T + C - 1) / C);
  const bool tc = use_tc_bwd(a);
  const BwdLayout L = tc ? tc_bwd_layout(a.BH, a.T) : bwd_layout(a.BH, a.T, m, dv, C);
  float* ws = reinterpret_cast<float*>(a.workspace);
  cudaError_t e;

  // 1. chunk maps and the state entering every chunk
  ChunkArgs f = a;
  f.x_last = nullptr;
  f.workspace = ws + L.maps;
  if (tc) {
    f.o = ws + L.o;
    f.S_out = ws + L.S_out;
    f.S_starts = ws + L.S_starts;
    // the maps, then the scan that records the state entering every chunk
    // (no o) and the reverse scan of the state cotangent over the same maps
    e = launch_tc_map64(f, err, stream);
    if (e == cudaSuccess) e = launch_tc_scan64(f, err, stream);
    if (e == cudaSuccess) e = launch_tc_bwd_scan(b, ws + L.maps, ws + L.dS_ends, err, stream);
  } else {
    f.o = nullptr;
    f.S_out = nullptr;
    e = launch_generic_chunked(f, stream, ws + L.S_starts);
  }
  if (e != cudaSuccess) return e;

  // 2. reverse scan of the state cotangent (tensor-core path: above),
  // 3. per-chunk gradients
  if (tc) {
    // dq, dv, dbeta, dlambda and dk (the chunk-end tokens by a small kernel)
    return launch_tc_bwd_grad(b, ws + L.S_starts, ws + L.dS_ends, ws + L.dX, err, stream);
  } else {
    const int NV = dv < 32 ? dv : 32;
    const size_t scan_smem =
        sizeof(float) * ((size_t)m * NV + (size_t)(m + C) * m + (size_t)(m + C) * NV);
    e = cudaFuncSetAttribute(bwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)scan_smem);
    if (e != cudaSuccess) return e;
    bwd_scan_kernel<<<dim3((unsigned)a.BH, dv / NV), kThreads, scan_smem, stream>>>(
        b, nchunks, NV, ws + L.maps, ws + L.dS_ends);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_generic_grad(b, nchunks, ws + L.S_starts, ws + L.dS_ends, ws + L.dX, stream);
  }
  if (e != cudaSuccess) return e;

  // 4. dk, dx_prev
  const int64_t rows = a.BH * a.T;
  const int64_t blocks = (rows + kWarps - 1) / kWarps;
  bwd_feature_kernel<<<(unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16), kThreads, 0,
                       stream>>>(b, ws + L.dX);
  return cudaGetLastError();
}

cudaError_t launch_generic_grad(const BwdArgs& b, int nchunks, const float* S_starts,
                                const float* dS_ends, float* dXw, cudaStream_t stream) {
  const ChunkArgs& a = b.f;
  const int m = a.m, dv = a.dv, C = a.C;
  const size_t grad_smem =
      sizeof(float) * (2 * (size_t)C * (m + 1) + 4 * (size_t)C * C + 2 * (size_t)C * dv +
                       16 * (size_t)C + 4) +
      sizeof(int) * (size_t)C;
  cudaError_t e = cudaFuncSetAttribute(bwd_grad_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)grad_smem);
  if (e != cudaSuccess) return e;
  bwd_grad_kernel<<<dim3(nchunks, (unsigned)a.BH), kThreads, grad_smem, stream>>>(
      b, nchunks, S_starts, dS_ends, dXw);
  return cudaGetLastError();
}

}  // namespace falcon
