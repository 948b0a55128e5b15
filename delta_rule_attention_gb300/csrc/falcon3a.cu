// Falcon-3A forward (sliding-window inner-product rule) in the token-recurrent
// form, for fresh sequences.
//
// Page hyper.ai/fr/papers/2608.27763, Section 4.5: for t >= 2 the window I_t
// of the last B write pairs (x_j, v_j), x_j = phi(k_{j-1}), j >= 2, with
// B_t = |I_t|, gives N_bar_t = (1/B_t) sum x_j v_j^T and E_bar_t =
// (1/B_t) sum ||x_j||^2; eta_t = beta_t / (E_bar_t + lambda_t + eps)
// (lambda_t = lambda_bar_t E_bar_t with the scale-coupled ridge), gamma_t =
// 1 - min(eta_t lambda_t, 1 - eps_gamma), S_t = gamma_t S_{t-1} + eta_t N_bar_t;
// token 1 is the boundary (no update); o_t = S_t^T phi(q_t).
//
// One CTA per (head, 32 value columns); each column of S and of the window
// sum N (= B_t N_bar_t) is held in fp32 registers by m / 16 threads.  N is
// kept incrementally: the entering pair is added and the pair leaving the
// window subtracted, so a token costs two rank-1 terms, the decayed update and
// the read, whatever the window.  Tokens go in blocks of 32 as in the Falcon-2
// kernel (bulk async copies of the raw rows into a two-buffer ring); the
// staged x rows and v values keep the previous block's 32 as a tail, which
// bounds the window at 32 pairs.  The per-token scalars (E_bar_t, eta_t /
// B_t, gamma_t) are computed for the whole block before the token loop.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace falcon {
namespace {

using tc::bulk_g2s;
using tc::fence_mbar_init;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;

constexpr int kTB = 32;      // tokens per block
constexpr int kTail = 32;    // staged rows kept from the previous block (window <= 32)

template <int M>
struct F3Cfg {
  static constexpr int kP = M / 16;         // threads per column (16 state rows each)
  static constexpr int kThreads = 32 * kP;  // 32 columns per CTA
  static constexpr int kLd = M / 16 * 20;   // fp32 row stride: 16 values + 4 gap per segment
  static_assert(2 * kThreads > kTail, "two passes cover the kTail + 1 tail energies");
};

__device__ __forceinline__ int pad16(int i) { return i + 4 * (i >> 4); }

template <int M>
struct F3Smem {
  // Row kTail + l holds x_{t0+l} (l in [-kTail, kTB]): the tail, the carried
  // x of the block's first token, and the block's own x rows.
  float xs[kTail + kTB + 1][F3Cfg<M>::kLd];
  float qs[kTB][F3Cfg<M>::kLd];
  float vs[kTail + kTB][32];  // v of the CTA's columns, same row convention (no row kTB)
  float ex[kTail + kTB + 1];  // ||x||^2 of each staged x row
  float coef[kTB], gam[kTB];  // eta_t / B_t and gamma_t (0 and 1 at the boundary)
  float os[kTB][32];
  uint64_t full[2];
  int fail;
};

struct RawLayout3 {
  uint32_t k, q, v, bytes;
};

__host__ __device__ inline RawLayout3 raw_layout3(int M, int dv, int es) {
  RawLayout3 L;
  L.k = 0;
  L.q = L.k + kTB * M * es;
  L.v = L.q + kTB * M * es;
  L.bytes = L.v + kTB * dv * es;
  return L;
}

__device__ __forceinline__ void load16_raw(const unsigned char* p, int64_t e0, int dtype, bool ok,
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

__device__ __forceinline__ void ld_seg(const float* row, int part, float* out) {
#pragma unroll
  for (int i4 = 0; i4 < 4; ++i4) {
    const float4 v = *reinterpret_cast<const float4*>(row + 20 * part + 4 * i4);
    out[4 * i4] = v.x;
    out[4 * i4 + 1] = v.y;
    out[4 * i4 + 2] = v.z;
    out[4 * i4 + 3] = v.w;
  }
}

template <int M>
__global__ void __launch_bounds__(F3Cfg<M>::kThreads)
    falcon3a_recurrent_kernel(ChunkArgs a, int window, int ncg, int* err) {
  using C = F3Cfg<M>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  F3Smem<M>& sm = *reinterpret_cast<F3Smem<M>*>(smem_raw);
  const int es = a.dtype == FALCON_BF16 ? 2 : 4;
  const RawLayout3 R = raw_layout3(M, a.dv, es);
  unsigned char* raw0 = smem_raw + ((sizeof(F3Smem<M>) + 127) & ~size_t(127));

  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t bh = blockIdx.x / ncg;
  const int cg = blockIdx.x % ncg;
  const int cl = tid / C::kP;    // local column
  const int part = tid % C::kP;  // rows 16 part .. 16 part + 15
  const int col = cg * 32 + cl;
  const bool active = col < a.dv;
  const int64_t T = a.T;
  const int64_t nblk = (T + kTB - 1) / kTB;
  volatile int* fail = &sm.fail;

  auto request = [&](int64_t b) {
    unsigned char* buf = raw0 + (b & 1) * R.bytes;
    const int64_t t0 = b * kTB;
    const int nb = (int)min((int64_t)kTB, T - t0);
    const int64_t row = bh * T + t0;
    const uint32_t kb = nb * M * es, vb = nb * a.dv * es;
    mbar_expect_tx(&sm.full[b & 1], 2 * kb + vb);
    bulk_g2s(buf + R.k, reinterpret_cast<const unsigned char*>(a.k) + row * M * es, kb,
             &sm.full[b & 1]);
    bulk_g2s(buf + R.q, reinterpret_cast<const unsigned char*>(a.q) + row * M * es, kb,
             &sm.full[b & 1]);
    bulk_g2s(buf + R.v, reinterpret_cast<const unsigned char*>(a.v) + row * a.dv * es, vb,
             &sm.full[b & 1]);
  };

  float s[16], nw[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    s[i] = (active && a.S0) ? a.S0[(bh * M + 16 * part + i) * a.dv + col] : 0.f;
    nw[i] = 0.f;
  }
  // The tail and the first block's carried x (x_1 = 0): pairs before token 2
  // never enter a window, zeros keep the rows harmless.
  for (int p = tid; p < (kTail + 1) * C::kLd; p += C::kThreads) (&sm.xs[0][0])[p] = 0.f;
  for (int p = tid; p < kTail * 32; p += C::kThreads) (&sm.vs[0][0])[p] = 0.f;
  for (int p = tid; p <= kTail; p += C::kThreads) sm.ex[p] = 0.f;
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
    __syncthreads();
    if (*fail) break;
    if (tid == 0 && b + 1 < nblk) request(b + 1);
    const float lam_l = (lane < nb) ? a.lambda[bh * T + t0 + lane] : 0.f;
    const float beta_l = (lane < nb) ? a.beta[bh * T + t0 + lane] : 0.f;
    // ---- phi(k) -> x of the next token (row kTail + l + 1), phi(q), v
    const int sl = tid / C::kP, sg = tid % C::kP;
    {
      float kk[16], qq[16];
      const int64_t e0 = (int64_t)sl * M + 16 * sg;
      load16_raw(buf + R.k, e0, a.dtype, sl < nb, kk);
      load16_raw(buf + R.q, e0, a.dtype, sl < nb, qq);
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
        float* xr = &sm.xs[kTail + sl + 1][20 * sg];
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
        if (sg == 0) sm.ex[kTail + sl + 1] = sk * fk * fk;
      }
    }
    for (int p = tid; p < kTB * 32; p += C::kThreads) {
      const int l = p >> 5, c = p & 31;
      const int gc = cg * 32 + c;
      sm.vs[kTail + l][c] =
          (l < nb && gc < a.dv) ? load_elem(buf + R.v, (int64_t)l * a.dv + gc, a.dtype) : 0.f;
    }
    __syncthreads();
    // ---- per-token scalars: window energy, eta_t / B_t, gamma_t (warp 0)
    if (tid < 32) {
      const int l = tid;
      const int64_t t = t0 + l;  // 0-based token; t = 0 is the boundary
      float coef = 0.f, gamma = 1.f;
      if (l < nb && t >= 1) {
        const int64_t j0 = max(t - window + 1, (int64_t)1);
        const int Bt = (int)(t - j0 + 1);
        float e = 0.f;
        for (int j = 0; j < Bt; ++j) e += sm.ex[kTail + l - j];
        const float Ebar = e / (float)Bt;
        const float lam = ridge_of(lam_l, Ebar, a.ridge);
        const float den = Ebar + lam + a.eps;
        const float eta = den > 0.f ? beta_l / den : 0.f;
        const float al = eta * lam;
        gamma = (al >= 1.f - a.eps_gamma) ? a.eps_gamma : 1.f - al;
        coef = eta / (float)Bt;
      }
      sm.coef[l] = coef;
      sm.gam[l] = gamma;
    }
    __syncthreads();

    // ---- the tokens of the block, in order
#pragma unroll 2
    for (int l = 0; l < nb; ++l) {
      const int64_t t = t0 + l;
      float xin[16], q[16];
      ld_seg(&sm.xs[kTail + l][0], part, xin);
      ld_seg(&sm.qs[l][0], part, q);
      const float vin = t >= 1 ? sm.vs[kTail + l][cl] : 0.f;  // the boundary pair is never used
#pragma unroll
      for (int i = 0; i < 16; ++i) nw[i] += vin * xin[i];
      if (t - window >= 1) {  // the pair leaving the window
        float xout[16];
        ld_seg(&sm.xs[kTail + l - window][0], part, xout);
        const float vout = sm.vs[kTail + l - window][cl];
#pragma unroll
        for (int i = 0; i < 16; ++i) nw[i] -= vout * xout[i];
      }
      const float coef = sm.coef[l], gamma = sm.gam[l];
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        s[i] = gamma * s[i] + coef * nw[i];
        s[i + 1] = gamma * s[i + 1] + coef * nw[i + 1];
        p0 += s[i] * q[i];
        p1 += s[i + 1] * q[i + 1];
      }
      float o = p0 + p1;
#pragma unroll
      for (int k = 1; k < C::kP; k <<= 1) o += __shfl_xor_sync(0xffffffffu, o, k);
      sm.os[l][cl] = o;
    }
    __syncthreads();
    for (int p = tid; p < nb * 32; p += C::kThreads) {
      const int l = p >> 5, c = p & 31;
      if (cg * 32 + c < a.dv)
        store_elem(a.o, (bh * T + t0 + l) * a.dv + cg * 32 + c, sm.os[l][c], a.dtype);
    }
    // The last kTail x rows (and the carried one), their energies and v become
    // the tail of the next block.
    if (nb == kTB) {
      // Source rows kTB .. kTB + kTail and target rows 0 .. kTail overlap in
      // row kTB: read everything first, then write.
      constexpr int kPer = ((kTail + 1) * C::kLd + C::kThreads - 1) / C::kThreads;
      float tmp[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int p = tid + k * C::kThreads;
        tmp[k] = p < (kTail + 1) * C::kLd ? (&sm.xs[kTB][0])[p] : 0.f;
      }
      // (kTail + 1 = 33 energies: a CTA of 32 threads needs a second pass)
      const float etmp0 = tid <= kTail ? sm.ex[kTB + tid] : 0.f;
      const float etmp1 = tid + C::kThreads <= kTail ? sm.ex[kTB + tid + C::kThreads] : 0.f;
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int p = tid + k * C::kThreads;
        if (p < (kTail + 1) * C::kLd) (&sm.xs[0][0])[p] = tmp[k];
      }
      if (tid <= kTail) sm.ex[tid] = etmp0;
      if (tid + C::kThreads <= kTail) sm.ex[tid + C::kThreads] = etmp1;
      for (int p = tid; p < kTail * 32; p += C::kThreads)  // rows kTB.. -> 0..: disjoint
        (&sm.vs[0][0])[p] = (&sm.vs[kTB][0])[p];
    } else {
      for (int i = tid; i < M; i += C::kThreads)
        sm.xs[kTail][pad16(i)] = sm.xs[kTail + nb][pad16(i)];
    }
    __syncthreads();
  }
  if (*fail) {
    if (tid == 0 && err) atomicExch(err, 1);
    return;
  }
  if (active) {
#pragma unroll
    for (int i = 0; i < 16; ++i) a.S_out[(bh * M + 16 * part + i) * a.dv + col] = s[i];
  }
  if (a.x_last && cg == 0)
    for (int i = tid; i < M; i += C::kThreads) a.x_last[bh * M + i] = sm.xs[kTail][pad16(i)];
}

template <int M>
cudaError_t launch_m(const ChunkArgs& a, int window, int* err, cudaStream_t stream) {
  const int ncg = (a.dv + 31) / 32;
  const int64_t grid = a.BH * ncg;
  const int es = a.dtype == FALCON_BF16 ? 2 : 4;
  const size_t smem =
      ((sizeof(F3Smem<M>) + 127) & ~size_t(127)) + 2 * raw_layout3(M, a.dv, es).bytes;
  cudaError_t e = cudaFuncSetAttribute(falcon3a_recurrent_kernel<M>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  falcon3a_recurrent_kernel<M><<<(unsigned)grid, F3Cfg<M>::kThreads, smem, stream>>>(a, window,
                                                                                    ncg, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_falcon3a_recurrent(const ChunkArgs& a, int window, int* err,
                                      cudaStream_t stream) {
  switch (a.m) {
    case 16: return launch_m<16>(a, window, err, stream);
    case 32: return launch_m<32>(a, window, err, stream);
    case 64: return launch_m<64>(a, window, err, stream);
    case 128: return launch_m<128>(a, window, err, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace falcon
