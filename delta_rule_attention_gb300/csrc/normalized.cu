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
// would write); on the tensor-core path with m = 64 the forward's map launch
// writes the terms of kernel 1 (it holds the chunk's features, step sizes,
// decays and decayed Gram rows already), and only kernels 2 and 3 run:
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

// One CTA per (chunk, head), 128 threads.  Shared: the chunk's write features
// x (C x m, raw, row 0 = the token before the chunk) and raw q rows (C x m),
// then per-token scalars (eta, log gamma, phi's scales of x and q, gamma).
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
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t0 = (int64_t)c * C;
  const int n = (int)min((int64_t)C, a.T - t0);
  const int64_t rowbase = bh * a.T;
  // the token's gain and ridge (thread r), issued before the rows
  float beta_r = 0.f, lam_r = 0.f;
  if (tid < n) {
    beta_r = a.beta[rowbase + t0 + tid];
    lam_r = a.lambda[rowbase + t0 + tid];
  }
  // rows: x_r = k_{t0 + r - 1} (r = 0: x_prev or the sentinel at the sequence
  // start), q_r = q_{t0 + r}; 16-byte pieces (rows are contiguous in memory),
  // four pieces of each per thread in flight before any is stored
  const int es = a.dtype == FALCON_BF16 ? 2 : 4, vec = 16 / es;
  // the lanes that load one row (m / vec of them, a power of two <= 32, and
  // aligned in the warp) also form its squared norms
  const int lpr = m / vec;
  for (int e0 = tid * vec; e0 < C * m; e0 += 4 * kNormThreads * vec) {
    uint4 kv[4], qv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = e0 + k * kNormThreads * vec;
      const int r = e / m, i = e % m;
      kv[k] = qv[k] = make_uint4(0u, 0u, 0u, 0u);
      if (e < C * m && r < n) {
        const int64_t tk = t0 + r - 1;
        if (tk >= 0)
          kv[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(a.k) +
                                                  ((rowbase + tk) * m + i) * es);
        qv[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(a.q) +
                                                ((rowbase + t0 + r) * m + i) * es);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = e0 + k * kNormThreads * vec;
      if (e0 + k * kNormThreads * vec - tid * vec >= C * m) break;  // (uniform over the CTA)
      float xk[8], xq[8];
      if (a.dtype == FALCON_BF16) {
        const __nv_bfloat162* hk = reinterpret_cast<const __nv_bfloat162*>(&kv[k]);
        const __nv_bfloat162* hq = reinterpret_cast<const __nv_bfloat162*>(&qv[k]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 f = __bfloat1622float2(hk[u]), g = __bfloat1622float2(hq[u]);
          xk[2 * u] = f.x, xk[2 * u + 1] = f.y, xq[2 * u] = g.x, xq[2 * u + 1] = g.y;
        }
      } else {
        const float* fk = reinterpret_cast<const float*>(&kv[k]);
        const float* fq = reinterpret_cast<const float*>(&qv[k]);
#pragma unroll
        for (int u = 0; u < 4; ++u) xk[u] = fk[u], xq[u] = fq[u], xk[4 + u] = xq[4 + u] = 0.f;
      }
      float ssx = 0.f, ssq = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) ssx = fmaf(xk[u], xk[u], ssx), ssq = fmaf(xq[u], xq[u], ssq);
      for (int o = lpr >> 1; o > 0; o >>= 1) {
        ssx += __shfl_xor_sync(0xffffffffu, ssx, o);
        ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
      }
      if (e < C * m) {
        float* xd = xs + e;
        float* qd = qs + e;
        reinterpret_cast<float4*>(xd)[0] = make_float4(xk[0], xk[1], xk[2], xk[3]);
        reinterpret_cast<float4*>(qd)[0] = make_float4(xq[0], xq[1], xq[2], xq[3]);
        if (vec == 8) {
          reinterpret_cast<float4*>(xd)[1] = make_float4(xk[4], xk[5], xk[6], xk[7]);
          reinterpret_cast<float4*>(qd)[1] = make_float4(xq[4], xq[5], xq[6], xq[7]);
        }
        if (e % m == 0) {  // the row's first lane: its squared norms (in eta and lg for now)
          eta[e / m] = ssx;
          lg[e / m] = ssq;
        }
      }
    }
  }
  // x_1 = x_prev (already a feature) at the sequence start, over the zeros
  // stored for row 0 above
  if (t0 == 0 && a.x_prev) {
    __syncthreads();
    for (int i = tid; i < m; i += kNormThreads) xs[i] = a.x_prev[bh * m + i];
    __syncthreads();
    if (warp == 0) {  // (phi's scale of this row is 1; its squared norm enters E)
      float ss = 0.f;
      for (int i = lane; i < m; i += 32) ss = fmaf(xs[i], xs[i], ss);
      ss = warp_sum(ss);
      if (lane == 0) eta[0] = ss;
    }
  }
  __syncthreads();
  // per-token scalars, one thread per token: phi's scales (x_prev is already a
  // feature), E_t, eta_t, log gamma_t (the sentinel: eta = 0 at the sequence
  // start without x_prev)
  if (tid < C) {
    const int r = tid;
    const float ssx = eta[r], ssq = lg[r];
    float e_t = 0.f, lgt = 0.f, s_x = 1.f, s_q = 1.f, gam = 1.f;
    if (r < n) {
      const bool carried = t0 + r == 0 && a.x_prev != nullptr;
      s_x = carried ? 1.f : feature_scale(ssx, m, a.phi);
      s_q = feature_scale(ssq, m, a.phi);
      const float E = ssx * s_x * s_x;
      const bool sentinel = t0 + r == 0 && a.x_prev == nullptr;
      e_t = step_eta_gamma(sentinel, E, beta_r, ridge_of(lam_r, E, a.ridge), a.eps, a.eps_gamma,
                           &gam, &lgt);
    }
    eta[r] = e_t * s_x;  // the gain on the raw row
    lg[r] = lgt;
    sx[r] = s_x;
    sq[r] = s_q;
    gm[r] = gam;
  }
  __syncthreads();
  const size_t mi = (size_t)(bh * nchunks + c);
  // e^{g_t} (inclusive prefix of log gamma; warp 0, tokens lane and lane + 32)
  // and the chunk's decay e^{g_C}
  if (warp == 0) {
    float g0 = lane < C ? lg[lane] : 0.f, g1 = lane + 32 < C ? lg[lane + 32] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_up_sync(0xffffffffu, g0, o);
      const float y1 = __shfl_up_sync(0xffffffffu, g1, o);
      if (lane >= o) g0 += y0, g1 += y1;
    }
    g1 += __shfl_sync(0xffffffffu, g0, 31);
    if (lane < C) ws[L.eg() + mi * C + lane] = __expf(g0), lg[lane] = g0;
    if (lane + 32 < C) ws[L.eg() + mi * C + lane + 32] = __expf(g1), lg[lane + 32] = g1;
    const int last = n - 1;
    const float gl = __shfl_sync(0xffffffffu, last < 32 ? g0 : g1, last & 31);
    if (lane == 0) ws[L.dec() + mi * 4] = __expf(gl);
  }
  // in-chunk normaliser, one thread per feature dimension: y_t = gamma_t
  // y_{t-1} + eta_t x_t, and the products y_t[i] phi(q_t)[i] (over the x rows,
  // each read just before).  With m <= 64 the CTA's two halves take the two
  // halves of the chunk's tokens, each from y = 0; the second half's reads and
  // the chunk's increment then add the first half's last y, decayed by
  // e^{g_t - g_{H-1}}.
  __shared__ float yh[128], y1s[128];
  const bool split = 2 * m <= kNormThreads;
  const int H = split ? C / 2 : C;
  const int half = split ? tid / m : 0, fi = tid - half * m;
  float y = 0.f;  // (the prefix g written over lg above is read after the next barrier)
  if (tid < (split ? 2 * m : m)) {
    const int rs = half == 0 ? 0 : H, re = half == 0 ? min(n, H) : n;
    // (rows at and past n were loaded as zeros and have eta = 0, gamma = 1)
    for (int r = rs; r < re; r += 4) {
      float g4[4], w4[4], s4[4], q4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int rr = min(r + u, C - 1);
        g4[u] = r + u < re ? gm[rr] : 1.f;
        w4[u] = r + u < re ? eta[rr] * xs[rr * m + fi] : 0.f;
        s4[u] = sq[rr];
        q4[u] = qs[rr * m + fi];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        y = fmaf(g4[u], y, w4[u]);
        if (r + u < re) xs[(r + u) * m + fi] = y * (s4[u] * q4[u]);
      }
    }
    if (split) (half == 0 ? yh : y1s)[fi] = y;
  }
  __syncthreads();
  // the chunk's increment y_C
  if (tid < m) {
    float inc = y;
    if (split) inc = n > H ? fmaf(__expf(lg[n - 1] - lg[H - 1]), yh[tid], y1s[tid]) : yh[tid];
    ws[L.inc() + mi * m + tid] = inc;
  }
  // r_t = <phi(q_t), y_t>, one thread per token (element (r, (i + r) mod m):
  // the threads of a warp read different banks)
  if (tid < C) {
    const int r = tid;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < n) {
      for (int i = 0; i < m; i += 4)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] += xs[r * m + ((i + u + r) & (m - 1))];
      if (split && r >= H) {
        float dq[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < m; i += 4)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = (i + u + r) & (m - 1);
            dq[u] = fmaf(qs[r * m + e], yh[e], dq[u]);
          }
        acc[0] = fmaf(__expf(lg[r] - lg[H - 1]) * sq[r], (dq[0] + dq[1]) + (dq[2] + dq[3]),
                      acc[0]);
      }
    }
    ws[L.rd() + mi * C + r] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    ws[L.nq() + mi * C + r] = sq[r];
  }
}

// One CTA per head, one thread per feature: z entering every chunk, and z_T.
// The chunks' decays are staged in shared memory kStage at a time, and each
// thread loads its increments kBatch chunks ahead of the chain that uses them.
constexpr int kBatch = 32, kStage = 1024;
__global__ void __launch_bounds__(kNormThreads)
    norm_chain_kernel(int64_t BH, int m, int nchunks, NormLayout L, const float* __restrict__ wsr,
                      float* __restrict__ zin, const float* z0, float* z_out) {
  __shared__ float dsh[kStage];
  const int64_t bh = blockIdx.x;
  const int i = threadIdx.x;
  const size_t m0 = (size_t)(bh * nchunks);
  float z = (i < m && z0) ? z0[bh * m + i] : 0.f;
  for (int s0 = 0; s0 < nchunks; s0 += kStage) {
    const int ns = min(kStage, nchunks - s0);
    __syncthreads();
    for (int u = i; u < ns; u += kNormThreads) dsh[u] = wsr[L.dec() + (m0 + s0 + u) * 4];
    __syncthreads();
    if (i < m) {
      for (int c0 = 0; c0 < ns; c0 += kBatch) {
        float y[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          y[u] = c0 + u < ns ? wsr[L.inc() + (m0 + s0 + c0 + u) * m + i] : 0.f;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (c0 + u < ns) {
            zin[(m0 + s0 + c0 + u) * m + i] = z;
            z = fmaf(dsh[c0 + u], z, y[u]);
          }
        }
      }
    }
  }
  if (z_out && i < m) z_out[bh * m + i] = z;
}

// One CTA per (chunk, head): den_t and o_t /= den_t.  A group of G lanes takes
// one token: 16-byte pieces of its q row (the read of z) and of its o row,
// loaded before the read is formed.  own_chain (few chunks, and z_out not
// overlapping z0): the CTA runs the chain up to its chunk itself, with the
// chain kernel's operations in its order, and the last chunk's CTA writes z_T.
constexpr int kOwnChainChunks = 64;
constexpr int kOwnChainAhead = 8;
__global__ void __launch_bounds__(kNormThreads)
    norm_apply_kernel(ChunkArgs a, int nchunks, NormLayout L, const float* ws, float eps_attn,
                      bool own_chain, const float* z0, float* z_out) {
  __shared__ float zc[128], fq[64], fr[64];
  const int C = a.C, m = a.m, dv = a.dv;
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t0 = (int64_t)c * C;
  const int n = (int)min((int64_t)C, a.T - t0);
  const size_t mi = (size_t)(bh * nchunks + c);
  if (tid < m) {
    if (own_chain) {
      const size_t m0 = (size_t)(bh * nchunks);
      float z = z0 ? z0[bh * m + tid] : 0.f;
      for (int u0 = 0; u0 < c; u0 += kOwnChainAhead) {
        float d[kOwnChainAhead], y[kOwnChainAhead];
#pragma unroll
        for (int k = 0; k < kOwnChainAhead; ++k) {
          d[k] = u0 + k < c ? ws[L.dec() + (m0 + u0 + k) * 4] : 0.f;
          y[k] = u0 + k < c ? ws[L.inc() + (m0 + u0 + k) * m + tid] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kOwnChainAhead; ++k)
          if (u0 + k < c) z = fmaf(d[k], z, y[k]);
      }
      zc[tid] = z;
      if (z_out && c == nchunks - 1)
        z_out[bh * m + tid] = fmaf(ws[L.dec() + mi * 4], z, ws[L.inc() + mi * m + tid]);
    } else {
      zc[tid] = ws[L.zin() + mi * m + tid];
    }
  }
  if (tid < C) {
    fq[tid] = ws[L.eg() + mi * C + tid] * ws[L.nq() + mi * C + tid];  // e^{g_t} phi's scale of q_t
    fr[tid] = ws[L.rd() + mi * C + tid] + eps_attn;
  }
  const int es = a.dtype == FALCON_BF16 ? 2 : 4, vec = 16 / es;
  // 16-byte pieces per row (powers of two, at most 32): G = the larger count
  // of lanes per token, so a lane holds at most one piece of each row
  const int pq = m * es / 16, po = dv * es / 16;
  const int G = pq > po ? pq : po;
  const int per_warp = 32 / G, grp = lane / G, sub = lane % G;
  const int stride = (kNormThreads / 32) * per_warp;
  __syncthreads();
  // four tokens per lane group in flight: their q and o pieces are loaded
  // before any read is formed
  for (int rb = warp * per_warp; rb < n; rb += 4 * stride) {
    uint4 qv[4], ov[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = rb + k * stride + grp;
      const int64_t row = bh * a.T + t0 + r;
      qv[k] = ov[k] = make_uint4(0u, 0u, 0u, 0u);
      if (r < n) {
        if (sub < pq)
          qv[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(a.q) +
                                                  (row * m + sub * vec) * es);
        if (sub < po)
          ov[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(a.o) +
                                                  (row * dv + sub * vec) * es);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = rb + k * stride + grp;
      float dot = 0.f;
      if (sub < pq) {
        if (a.dtype == FALCON_BF16) {
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&qv[k]);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 f = __bfloat1622float2(h[u]);
            dot = fmaf(f.x, zc[sub * 8 + 2 * u], dot);
            dot = fmaf(f.y, zc[sub * 8 + 2 * u + 1], dot);
          }
        } else {
          const float* f = reinterpret_cast<const float*>(&qv[k]);
#pragma unroll
          for (int u = 0; u < 4; ++u) dot = fmaf(f[u], zc[sub * 4 + u], dot);
        }
      }
      for (int o = G >> 1; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (r >= n || sub >= po) continue;
      const float den = fq[r] * dot + fr[r];
      if (a.dtype == FALCON_BF16) {
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&ov[k]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 f = __bfloat1622float2(h[u]);
          h[u] = __floats2bfloat162_rn(f.x / den, f.y / den);
        }
      } else {
        float* f = reinterpret_cast<float*>(&ov[k]);
#pragma unroll
        for (int u = 0; u < 4; ++u) f[u] /= den;
      }
      const int64_t row = bh * a.T + t0 + r;
      unsigned char* op = reinterpret_cast<unsigned char*>(a.o) + (row * dv + sub * vec) * es;
      *reinterpret_cast<uint4*>(op) = ov[k];
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
                              float* ws, bool chunk_terms_written, cudaStream_t stream) {
  const int nchunks = (int)((a.T + a.C - 1) / a.C);
  const NormLayout L{a.BH * nchunks, a.m, a.C};
  cudaError_t e = cudaSuccess;
  if (!chunk_terms_written) {
    const size_t smem = sizeof(float) * (size_t)(2 * a.C * a.m + 5 * a.C);
    e = cudaFuncSetAttribute(norm_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    norm_chunk_kernel<<<dim3(nchunks, (unsigned)a.BH), kNormThreads, smem, stream>>>(a, nchunks,
                                                                                     L, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // Few chunks: every apply CTA runs the chain to its chunk (no chain launch),
  // unless z_out overlaps z0 (the last chunk's CTA would write z_T while
  // others still read z0).
  const size_t feat = (size_t)a.BH * a.m;
  const bool overlap = z0 && z_out && z_out < z0 + feat && z0 < z_out + feat;
  const bool own_chain = nchunks <= kOwnChainChunks && !overlap;
  if (!own_chain) {
    norm_chain_kernel<<<(unsigned)a.BH, kNormThreads, 0, stream>>>(a.BH, a.m, nchunks, L, ws,
                                                                     ws + L.zin(), z0, z_out);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  norm_apply_kernel<<<dim3(nchunks, (unsigned)a.BH), kNormThreads, 0, stream>>>(
      a, nchunks, L, ws, eps_attn, own_chain, z0, z_out);
  return cudaGetLastError();
}

}  // namespace falcon
