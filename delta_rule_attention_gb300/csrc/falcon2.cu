// Falcon-2 / Falcon-2A forward in the token-recurrent form.
//
// Per head, every column j of the state S (m x d_v) is its own scalar-step
// chain: eta_{j,t} = beta_{j,t} / (||x_t||^2 + lambda_t + eps), gamma_{j,t} =
// 1 - min(eta_{j,t} lambda_t, 1 - eps_gamma), and
//   Falcon-2:  s_j <- gamma_{j,t} s_j + eta_{j,t} x_t (v_{t,j} - s_j^T x_t)
//   Falcon-2A: s_j <- gamma_{j,t} s_j + eta_{j,t} x_t v_{t,j}
// with the shared write feature x_t = phi(k_{t-1}) (x_1 = 0 and eta_1 = 0 at a
// sequence start, or x_1 = x_prev), and the read after write
// o_{t,j} = s_j^T phi(q_t) = gamma_{j,t} (s_j^T phi(q_t))_{before} +
// eta_{j,t} r_{t,j} <x_t, phi(q_t)>.
// Page hyper.ai/fr/papers/2608.27763: the regression-family display of
// Section 3.1, the per-column NLMS step sizes of Section 4.2 and Falcon-2A of
// Section 4.3 (the loss separates over the columns of S).
//
// One CTA per (head, 32 columns); each column is held in fp32 registers by
// m / 16 threads (16 rows each), so the two column reductions per token need
// only log2(m / 16) shuffle steps.  Tokens go in blocks of 32: the raw k, q,
// v and beta rows of a block arrive by bulk async copies into a two-buffer
// ring (requested one block ahead), and are staged as phi(k) and phi(q) rows
// (fp32, with a 4-float gap after every 16 so that the row segments the
// threads of a warp read sit in distinct banks), <x_t, phi(q_t)>, and the step
// sizes and decays eta_{j,t}, gamma_{j,t}, which depend on the inputs only and
// are computed for the whole block in parallel.  The sequential part per token
// is then two dot products, a short shuffle reduction and the rank-1 update;
// o is collected in shared memory and stored once per block.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace falcon {
namespace {

using tc::bulk_g2s;
using tc::fence_mbar_init;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;

constexpr int kTB = 32;  // tokens per block

template <int M>
struct F2Cfg {
  static constexpr int kP = M / 16;         // threads per column (16 state rows each)
  static constexpr int kThreads = 32 * kP;  // 32 columns per CTA
  static constexpr int kLd = M / 16 * 20;   // fp32 row stride: 16 values + 4 gap per segment
};

// Position of row element i in a staged row (a 4-float gap after every 16):
// segment g of 16 values starts at float 20 g.
__device__ __forceinline__ int pad16(int i) { return i + 4 * (i >> 4); }

// Sixteen consecutive elements e0 .. e0 + 15 (e0 a multiple of 16) of a raw
// bf16 or fp32 row buffer in shared memory, by 16-byte loads; zeros if !ok.
__device__ __forceinline__ void load16(const unsigned char* p, int64_t e0, int dtype, bool ok,
                                       float* out) {
  if (!ok) {
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = 0.f;
  } else if (dtype == FALCON_BF16) {
    const uint4* v = reinterpret_cast<const uint4*>(p + 2 * e0);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 pk = v[c];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&pk);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        out[8 * c + 2 * e] = f.x;
        out[8 * c + 2 * e + 1] = f.y;
      }
    }
  } else {
    const float4* v = reinterpret_cast<const float4*>(p + 4 * e0);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 f = v[c];
      out[4 * c] = f.x;
      out[4 * c + 1] = f.y;
      out[4 * c + 2] = f.z;
      out[4 * c + 3] = f.w;
    }
  }
}

// Shared memory: fixed part, then the two raw buffers (dynamic size).
template <int M>
struct F2Smem {
  float xs[kTB + 1][F2Cfg<M>::kLd];  // row l: x_{t0+l}; row 0 carried in
  float qs[kTB][F2Cfg<M>::kLd];      // phi(q_{t0+l})
  float eta[kTB][32], gam[kTB][32], vs[kTB][32], os[kTB][32];
  float Es[kTB], xqs[kTB];
  uint64_t full[2];
  int fail;
};

struct RawLayout {  // byte offsets inside one raw buffer
  uint32_t k, q, v, b, bytes;
};

__host__ __device__ inline RawLayout raw_layout(int M, int dv, int es) {
  RawLayout L;
  L.k = 0;
  L.q = L.k + kTB * M * es;
  L.v = L.q + kTB * M * es;
  L.b = L.v + kTB * dv * es;
  L.bytes = L.b + kTB * dv * 4;
  return L;
}

template <int M>
__global__ void __launch_bounds__(F2Cfg<M>::kThreads)
    falcon2_recurrent_kernel(ChunkArgs a, int ncg, int* err) {
  using C = F2Cfg<M>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  F2Smem<M>& sm = *reinterpret_cast<F2Smem<M>*>(smem_raw);
  const int es = a.dtype == FALCON_BF16 ? 2 : 4;
  const RawLayout R = raw_layout(M, a.dv, es);
  unsigned char* raw0 = smem_raw + ((sizeof(F2Smem<M>) + 127) & ~size_t(127));

  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t bh = blockIdx.x / ncg;
  const int cg = blockIdx.x % ncg;
  const int cl = tid / C::kP;    // local column
  const int part = tid % C::kP;  // rows 16 part .. 16 part + 15
  const int col = cg * 32 + cl;
  const bool active = col < a.dv;
  const bool f2 = a.rule == kFalcon2;
  const int64_t T = a.T;
  const int64_t nblk = (T + kTB - 1) / kTB;
  volatile int* fail = &sm.fail;

  // Raw rows of block b (tokens b*32 .. ) into buffer b & 1.
  auto request = [&](int64_t b) {
    unsigned char* buf = raw0 + (b & 1) * R.bytes;
    const int64_t t0 = b * kTB;
    const int nb = (int)min((int64_t)kTB, T - t0);
    const int64_t row = bh * T + t0;
    const uint32_t kb = nb * M * es, vb = nb * a.dv * es, bb = nb * a.dv * 4;
    mbar_expect_tx(&sm.full[b & 1], 2 * kb + vb + bb);
    bulk_g2s(buf + R.k, reinterpret_cast<const unsigned char*>(a.k) + row * M * es, kb,
             &sm.full[b & 1]);
    bulk_g2s(buf + R.q, reinterpret_cast<const unsigned char*>(a.q) + row * M * es, kb,
             &sm.full[b & 1]);
    bulk_g2s(buf + R.v, reinterpret_cast<const unsigned char*>(a.v) + row * a.dv * es, vb,
             &sm.full[b & 1]);
    bulk_g2s(buf + R.b, a.beta + row * a.dv, bb, &sm.full[b & 1]);
  };

  float s[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    s[i] = (active && a.S0) ? a.S0[(bh * M + 16 * part + i) * a.dv + col] : 0.f;
  for (int i = tid; i < M; i += C::kThreads)
    sm.xs[0][pad16(i)] = a.x_prev ? a.x_prev[bh * M + i] : 0.f;
  const bool sentinel0 = a.x_prev == nullptr;
  if (tid == 0) {
    mbar_init(&sm.full[0], 1);
    mbar_init(&sm.full[1], 1);
    fence_mbar_init();
    sm.fail = 0;
    if (nblk > 0) request(0);
  }
  __syncthreads();

  for (int64_t b = 0; b < nblk; ++b) {
    const int64_t t0 = b * kTB;
    const int nb = (int)min((int64_t)kTB, T - t0);
    const unsigned char* buf = raw0 + (b & 1) * R.bytes;
    if (!mbar_wait(&sm.full[b & 1], (uint32_t)(b >> 1) & 1u)) *fail = 1;
    // Every thread has passed the wait; the other buffer (block b - 1) is
    // consumed: request block b + 1 into it.
    __syncthreads();
    if (*fail) break;
    if (tid == 0 && b + 1 < nblk) request(b + 1);
    const float lam_l = (lane < nb) ? a.lambda[bh * T + t0 + lane] : 0.f;
    // ---- phi(k) -> x of the next token, phi(q).  Thread (l, g) = (tid / kP,
    // tid % kP) takes elements 16g .. 16g + 15 of row l; the kP threads of a
    // row are adjacent lanes and combine their sums by shuffles.
    const int sl = tid / C::kP, sg = tid % C::kP;
    {
      float kk[16], qq[16];
      const int64_t e0 = (int64_t)sl * M + 16 * sg;
      load16(buf + R.k, e0, a.dtype, sl < nb, kk);
      load16(buf + R.q, e0, a.dtype, sl < nb, qq);
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        sk += kk[i] * kk[i];
        sq += qq[i] * qq[i];
      }
#pragma unroll
      for (int o = 1; o < C::kP; o <<= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
      }
      const float fk = feature_scale(sk, M, a.phi), fq = feature_scale(sq, M, a.phi);
      if (sl < nb) {
        float* xr = &sm.xs[sl + 1][20 * sg];
        float* qr = &sm.qs[sl][20 * sg];
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          *reinterpret_cast<float4*>(xr + 4 * i4) =
              make_float4(kk[4 * i4] * fk, kk[4 * i4 + 1] * fk, kk[4 * i4 + 2] * fk,
                          kk[4 * i4 + 3] * fk);
          *reinterpret_cast<float4*>(qr + 4 * i4) =
              make_float4(qq[4 * i4] * fq, qq[4 * i4 + 1] * fq, qq[4 * i4 + 2] * fq,
                          qq[4 * i4 + 3] * fq);
        }
      }
    }
    __syncthreads();
    // ---- ||x_t||^2 and <x_t, phi(q_t)> (x_t = row l of xs, written by row l - 1)
    {
      float se = 0.f, sxq = 0.f;
      if (sl < nb) {
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          const float4 xv = *reinterpret_cast<const float4*>(&sm.xs[sl][20 * sg + 4 * i4]);
          const float4 qv = *reinterpret_cast<const float4*>(&sm.qs[sl][20 * sg + 4 * i4]);
          se += xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w;
          sxq += xv.x * qv.x + xv.y * qv.y + xv.z * qv.z + xv.w * qv.w;
        }
      }
#pragma unroll
      for (int o = 1; o < C::kP; o <<= 1) {
        se += __shfl_xor_sync(0xffffffffu, se, o);
        sxq += __shfl_xor_sync(0xffffffffu, sxq, o);
      }
      if (sg == 0 && sl < nb) {
        sm.Es[sl] = se;
        sm.xqs[sl] = sxq;
      }
    }
    __syncthreads();
    // ---- eta, gamma and v of every (token, column) of the block
    // (a warp's 32 threads take the 32 columns of one token, so l is uniform
    // in the warp and lambda_l comes from lane l by one shuffle)
    for (int p = tid; p < kTB * 32; p += C::kThreads) {
      const int l = p >> 5, c = p & 31;
      const int gc = cg * 32 + c;
      const float lam = ridge_of(__shfl_sync(0xffffffffu, lam_l, l), sm.Es[l], a.ridge);
      if (l < nb && gc < a.dv) {
        // eta_{j,t} and the clamped decay (as step_eta_gamma, without the log)
        const bool sent = sentinel0 && (t0 + l == 0);
        const float beta = reinterpret_cast<const float*>(buf + R.b)[l * a.dv + gc];
        const float den = sm.Es[l] + lam + a.eps;
        const float eta = (!sent && den > 0.f) ? beta / den : 0.f;
        const float al = eta * lam;
        sm.eta[l][c] = eta;
        sm.gam[l][c] = (al >= 1.f - a.eps_gamma) ? a.eps_gamma : 1.f - al;
        sm.vs[l][c] = load_elem(buf + R.v, (int64_t)l * a.dv + gc, a.dtype);
      } else if (l < nb) {
        sm.eta[l][c] = 0.f;
        sm.gam[l][c] = 1.f;
        sm.vs[l][c] = 0.f;
      }
    }
    __syncthreads();

    // ---- the tokens of the block, in order
#pragma unroll 2
    for (int l = 0; l < nb; ++l) {
      float x[16], q[16];
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const float4 xv = *reinterpret_cast<const float4*>(&sm.xs[l][20 * part + 4 * i4]);
        const float4 qv = *reinterpret_cast<const float4*>(&sm.qs[l][20 * part + 4 * i4]);
        x[4 * i4] = xv.x; x[4 * i4 + 1] = xv.y; x[4 * i4 + 2] = xv.z; x[4 * i4 + 3] = xv.w;
        q[4 * i4] = qv.x; q[4 * i4 + 1] = qv.y; q[4 * i4 + 2] = qv.z; q[4 * i4 + 3] = qv.w;
      }
      float pa0 = 0.f, pa1 = 0.f, pb0 = 0.f, pb1 = 0.f;
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        pa0 += s[i] * x[i];
        pa1 += s[i + 1] * x[i + 1];
        pb0 += s[i] * q[i];
        pb1 += s[i + 1] * q[i + 1];
      }
      float pa = pa0 + pa1, pb = pb0 + pb1;  // s_j^T x_t, s_j^T phi(q_t) (before the write)
#pragma unroll
      for (int o = 1; o < C::kP; o <<= 1) {
        pa += __shfl_xor_sync(0xffffffffu, pa, o);
        pb += __shfl_xor_sync(0xffffffffu, pb, o);
      }
      const float eta = sm.eta[l][cl], gamma = sm.gam[l][cl];
      const float r = f2 ? sm.vs[l][cl] - pa : sm.vs[l][cl];
      const float er = eta * r;
#pragma unroll
      for (int i = 0; i < 16; ++i) s[i] = gamma * s[i] + er * x[i];
      // every thread of the column holds the full sums: all write o (one
      // address per column), which keeps the loop free of a divergent branch
      sm.os[l][cl] = gamma * pb + er * sm.xqs[l];
    }
    __syncthreads();
    // o of the block (coalesced), and x of the next block's first token
    for (int p = tid; p < nb * 32; p += C::kThreads) {
      const int l = p >> 5, c = p & 31;
      if (cg * 32 + c < a.dv)
        store_elem(a.o, (bh * T + t0 + l) * a.dv + cg * 32 + c, sm.os[l][c], a.dtype);
    }
    for (int i = tid; i < M; i += C::kThreads) sm.xs[0][pad16(i)] = sm.xs[nb][pad16(i)];
  }
  __syncthreads();
  if (*fail) {
    if (tid == 0 && err) atomicExch(err, 1);
    return;
  }
  if (active) {
#pragma unroll
    for (int i = 0; i < 16; ++i) a.S_out[(bh * M + 16 * part + i) * a.dv + col] = s[i];
  }
  if (a.x_last && cg == 0)
    for (int i = tid; i < M; i += C::kThreads) a.x_last[bh * M + i] = sm.xs[0][pad16(i)];
}

template <int M>
cudaError_t launch_m(const ChunkArgs& a, int* err, cudaStream_t stream) {
  const int ncg = (a.dv + 31) / 32;
  const int64_t grid = a.BH * ncg;
  const int es = a.dtype == FALCON_BF16 ? 2 : 4;
  const size_t smem = ((sizeof(F2Smem<M>) + 127) & ~size_t(127)) + 2 * raw_layout(M, a.dv, es).bytes;
  cudaError_t e = cudaFuncSetAttribute(falcon2_recurrent_kernel<M>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  falcon2_recurrent_kernel<M><<<(unsigned)grid, F2Cfg<M>::kThreads, smem, stream>>>(a, ncg, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_falcon2_recurrent(const ChunkArgs& a, int* err, cudaStream_t stream) {
  switch (a.m) {
    case 16: return launch_m<16>(a, err, stream);
    case 32: return launch_m<32>(a, err, stream);
    case 64: return launch_m<64>(a, err, stream);
    case 128: return launch_m<128>(a, err, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace falcon
