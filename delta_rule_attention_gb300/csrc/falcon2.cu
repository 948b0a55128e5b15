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
// The residual's inner product is taken one token ahead, from the state
// before the previous write:
//   s_t^T x_{t+1} = gamma_t (s_{t-1}^T x_{t+1}) + eta_t r_t <x_t, x_{t+1}>,
// so that both reads of a token (s^T x_{t+1} and s^T phi(q_t)) and its write
// go in one pass over the state rows, all with the state before the write;
// the dependent chain from one token to the next is a few scalar operations.
// A column's state is held in fp32 registers by kP threads (kR = m / kP <= 32
// rows each, one shuffle step for m = 64).  Scalar fp32 multiply-adds: on
// sm_103 a lone warp issues one every ~1.2 cycles but the packed f32x2 form
// only every ~3 (measured), and a broadcast 16-byte shared-memory read costs
// it ~11 cycles, so the reads of the staged rows make up most of the cost of
// a token.
//
// One CTA of 64 threads per (head, group of 64 / kP columns).  Tokens arrive
// in blocks of 32: the raw k, q, v and beta rows of a block come by bulk
// async copies into a two-buffer ring (requested one block ahead) and are
// staged as phi(k) and phi(q) rows (fp32), with the per-token ||x_t||^2,
// <x_t, x_{t+1}>, <x_t, phi(q_t)>, lambda_t and 1 / (||x_t||^2 + lambda_t +
// eps) formed for the whole block in parallel.  o is collected in shared
// memory and stored once per block.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace falcon {
namespace {

using tc::bulk_g2s;
using tc::fence_mbar_init;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;

constexpr int kTB = 32;       // tokens per block
constexpr int kThreads = 64;  // threads per CTA

template <int M>
struct F2Cfg {
  static constexpr int kP = M >= 64 ? M / 32 : 1;  // threads per column
  static constexpr int kR = M / kP;            // state rows per thread
  static constexpr int kCols = kThreads / kP;  // columns per CTA
  static constexpr int kSeg = kR + 4;          // padded row segment (floats)
  static constexpr int kLd = kP * kSeg;        // staged row stride (floats)
};

// Position of row element i in a staged row.
template <int M>
__device__ __forceinline__ int padded(int i) {
  return i + 4 * (i / F2Cfg<M>::kR);
}

// Shared memory: fixed part, then the two raw buffers (dynamic size).
template <int M>
struct F2Smem {
  float xs[kTB + 1][F2Cfg<M>::kLd];  // row l: x_{t0+l}; row 0 carried in
  float qs[kTB][F2Cfg<M>::kLd];      // phi(q_{t0+l})
  float4 tok[kTB];  // 1 / (||x||^2 + lambda + eps) (0: no write), lambda, <x, x_next>, <x, phi(q)>
  float os[kTB][F2Cfg<M>::kCols];
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

// n consecutive elements (n a multiple of 8) of a raw bf16 or fp32 row buffer
// in shared memory, by 16-byte loads, as fp32.
template <int N>
__device__ __forceinline__ void load_raw(const unsigned char* p, int64_t e0, int dtype,
                                         float* out) {
  if (dtype == FALCON_BF16) {
    const uint4* v = reinterpret_cast<const uint4*>(p + 2 * e0);
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
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
    for (int c = 0; c < N / 4; ++c) {
      const float4 f = v[c];
      out[4 * c] = f.x;
      out[4 * c + 1] = f.y;
      out[4 * c + 2] = f.z;
      out[4 * c + 3] = f.w;
    }
  }
}

// Sum over the kP threads of a column (adjacent lanes).
template <int M>
__device__ __forceinline__ float column_sum(float v) {
#pragma unroll
  for (int o = 1; o < F2Cfg<M>::kP; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int M, bool kF2>
__global__ void __launch_bounds__(kThreads)
    falcon2_recurrent_kernel(ChunkArgs a, int ncg, int* err) {
  using C = F2Cfg<M>;
  constexpr int kR = C::kR, kP = C::kP, kCols = C::kCols, kH = M / 2;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  F2Smem<M>& sm = *reinterpret_cast<F2Smem<M>*>(smem_raw);
  const int es = a.dtype == FALCON_BF16 ? 2 : 4;
  const RawLayout R = raw_layout(M, a.dv, es);
  unsigned char* raw0 = smem_raw + ((sizeof(F2Smem<M>) + 127) & ~size_t(127));

  const int tid = threadIdx.x;
  const int64_t bh = blockIdx.x / ncg;
  const int cg = blockIdx.x % ncg;
  const int cl = tid / kP;    // local column
  const int part = tid % kP;  // rows kR part .. kR part + kR - 1
  const int col = cg * kCols + cl;
  const bool active = col < a.dv;
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

  float s[kR];  // rows kR part .. kR part + kR - 1 of this column
#pragma unroll
  for (int i = 0; i < kR; ++i)
    s[i] = (active && a.S0) ? a.S0[(bh * M + kR * part + i) * a.dv + col] : 0.f;
  for (int i = tid; i < M; i += kThreads)
    sm.xs[0][padded<M>(i)] = a.x_prev ? a.x_prev[bh * M + i] : 0.f;
  const bool sentinel0 = a.x_prev == nullptr;
  if (tid == 0) {
    mbar_init(&sm.full[0], 1);
    mbar_init(&sm.full[1], 1);
    fence_mbar_init();
    sm.fail = 0;
    if (nblk > 0) request(0);
  }
  __syncthreads();
  // x of the next token to write (this thread's rows, registers), and
  // p = s^T x for it.
  float xc[kR];
  {
    const float4* x4 = reinterpret_cast<const float4*>(sm.xs[0] + C::kSeg * part);
#pragma unroll
    for (int c = 0; c < kR / 4; ++c) {
      const float4 f = x4[c];
      xc[4 * c] = f.x;
      xc[4 * c + 1] = f.y;
      xc[4 * c + 2] = f.z;
      xc[4 * c + 3] = f.w;
    }
  }
  float p = 0.f;
  if constexpr (kF2) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kR; ++i) acc[i & 3] = fmaf(s[i], xc[i], acc[i & 3]);
    p = column_sum<M>((acc[0] + acc[1]) + (acc[2] + acc[3]));
  }

  const int hl = tid >> 1, hh = tid & 1;  // staging: row hl, half row hh
  for (int64_t b = 0; b < nblk; ++b) {
    const int64_t t0 = b * kTB;
    const int nb = (int)min((int64_t)kTB, T - t0);
    const unsigned char* buf = raw0 + (b & 1) * R.bytes;
    const float lam_raw = (hh == 0 && hl < nb) ? a.lambda[bh * T + t0 + hl] : 0.f;
    if (!mbar_wait(&sm.full[b & 1], (uint32_t)(b >> 1) & 1u)) *fail = 1;
    // Every thread has passed the wait; the other buffer (block b - 1) is
    // consumed: request block b + 1 into it.
    __syncthreads();
    if (*fail) break;
    if (tid == 0 && b + 1 < nblk) request(b + 1);
    // ---- phi(k) -> x of the next token, then phi(q): two threads per row
    //      (half rows of M / 2 elements), sums combined by one shuffle
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      float kk[kH];
      float sk = 0.f;
      if (hl < nb) {
        load_raw<kH>(buf + (which ? R.q : R.k), (int64_t)hl * M + kH * hh, a.dtype, kk);
#pragma unroll
        for (int i = 0; i < kH; ++i) sk = fmaf(kk[i], kk[i], sk);
      }
      sk += __shfl_xor_sync(0xffffffffu, sk, 1);
      if (hl < nb) {
        const float fk = feature_scale(sk, M, a.phi);
        float* xr = which ? sm.qs[hl] : sm.xs[hl + 1];
#pragma unroll
        for (int i4 = 0; i4 < kH / 4; ++i4)
          *reinterpret_cast<float4*>(xr + padded<M>(kH * hh + 4 * i4)) =
              make_float4(kk[4 * i4] * fk, kk[4 * i4 + 1] * fk, kk[4 * i4 + 2] * fk,
                          kk[4 * i4 + 3] * fk);
      }
    }
    __syncthreads();
    // ---- per token: ||x_t||^2, <x_t, x_{t+1}>, <x_t, phi(q_t)> (x_t = row l
    //      of xs, x_{t+1} = row l + 1), lambda_t and 1 / (||x_t||^2 + lambda_t + eps)
    {
      float se = 0.f, sg = 0.f, sxq = 0.f;
      if (hl < nb) {
#pragma unroll
        for (int i4 = 0; i4 < kH / 4; ++i4) {
          const int e = padded<M>(kH * hh + 4 * i4);
          const float4 x = *reinterpret_cast<const float4*>(sm.xs[hl] + e);
          const float4 xn = *reinterpret_cast<const float4*>(sm.xs[hl + 1] + e);
          const float4 qv = *reinterpret_cast<const float4*>(sm.qs[hl] + e);
          se = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, se))));
          sg = fmaf(x.x, xn.x, fmaf(x.y, xn.y, fmaf(x.z, xn.z, fmaf(x.w, xn.w, sg))));
          sxq = fmaf(x.x, qv.x, fmaf(x.y, qv.y, fmaf(x.z, qv.z, fmaf(x.w, qv.w, sxq))));
        }
      }
      se += __shfl_xor_sync(0xffffffffu, se, 1);
      sg += __shfl_xor_sync(0xffffffffu, sg, 1);
      sxq += __shfl_xor_sync(0xffffffffu, sxq, 1);
      if (hh == 0 && hl < nb) {
        const float lam = ridge_of(lam_raw, se, a.ridge);
        const float den = se + lam + a.eps;
        const bool sent = sentinel0 && t0 + hl == 0;  // x_1 = 0: no write
        sm.tok[hl] = make_float4((!sent && den > 0.f) ? 1.f / den : 0.f, lam, sg, sxq);
      }
    }
    __syncthreads();

    // ---- the tokens of the block, in order: both reads with the state before
    //      the write, and the write, in one pass over this thread's rows
    const float* braw = reinterpret_cast<const float*>(buf + R.b);
#pragma unroll 1
    for (int l = 0; l < nb; ++l) {
      const float4 tk = sm.tok[l];
      const float beta = active ? braw[l * a.dv + col] : 0.f;
      const float v = active ? load_elem(buf + R.v, (int64_t)l * a.dv + col, a.dtype) : 0.f;
      const float eta = beta * tk.x;
      const float al = eta * tk.y;
      const float gam = (al >= 1.f - a.eps_gamma) ? a.eps_gamma : 1.f - al;
      const float er = eta * (kF2 ? v - p : v);
      const float4* xn4 = reinterpret_cast<const float4*>(sm.xs[l + 1] + C::kSeg * part);
      const float4* q4 = reinterpret_cast<const float4*>(sm.qs[l] + C::kSeg * part);
      float aa[4] = {0.f, 0.f, 0.f, 0.f}, bb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kR / 4; ++c) {
        const float4 q = q4[c];
        bb[0] = fmaf(s[4 * c], q.x, bb[0]);
        bb[1] = fmaf(s[4 * c + 1], q.y, bb[1]);
        bb[2] = fmaf(s[4 * c + 2], q.z, bb[2]);
        bb[3] = fmaf(s[4 * c + 3], q.w, bb[3]);
        const float4 f = xn4[c];
        if constexpr (kF2) {
          aa[0] = fmaf(s[4 * c], f.x, aa[0]);
          aa[1] = fmaf(s[4 * c + 1], f.y, aa[1]);
          aa[2] = fmaf(s[4 * c + 2], f.z, aa[2]);
          aa[3] = fmaf(s[4 * c + 3], f.w, aa[3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s[4 * c + i] = fmaf(gam, s[4 * c + i], er * xc[4 * c + i]);
        xc[4 * c] = f.x;
        xc[4 * c + 1] = f.y;
        xc[4 * c + 2] = f.z;
        xc[4 * c + 3] = f.w;
      }
      const float bv = column_sum<M>((bb[0] + bb[1]) + (bb[2] + bb[3]));
      // s_t^T x_{t+1}, the next token's residual product
      if constexpr (kF2) p = fmaf(gam, column_sum<M>((aa[0] + aa[1]) + (aa[2] + aa[3])), er * tk.z);
      if (part == 0) sm.os[l][cl] = fmaf(gam, bv, er * tk.w);
    }
    __syncthreads();
    // o of the block (coalesced), and x of the next block's first token
    for (int p2 = tid; p2 < nb * kCols; p2 += kThreads) {
      const int l = p2 / kCols, c = p2 % kCols;
      if (cg * kCols + c < a.dv)
        store_elem(a.o, (bh * T + t0 + l) * a.dv + cg * kCols + c, sm.os[l][c], a.dtype);
    }
    for (int i = tid; i < M; i += kThreads) sm.xs[0][padded<M>(i)] = sm.xs[nb][padded<M>(i)];
  }
  __syncthreads();
  if (*fail) {
    if (tid == 0 && err) atomicExch(err, 1);
    return;
  }
  if (active) {
#pragma unroll
    for (int i = 0; i < kR; ++i) a.S_out[(bh * M + kR * part + i) * a.dv + col] = s[i];
  }
  if (a.x_last && cg == 0)
    for (int i = tid; i < M; i += kThreads) a.x_last[bh * M + i] = sm.xs[0][padded<M>(i)];
}

template <int M>
cudaError_t launch_m(const ChunkArgs& a, int* err, cudaStream_t stream) {
  const int ncg = (a.dv + F2Cfg<M>::kCols - 1) / F2Cfg<M>::kCols;
  const int64_t grid = a.BH * ncg;
  const int es = a.dtype == FALCON_BF16 ? 2 : 4;
  const size_t smem =
      ((sizeof(F2Smem<M>) + 127) & ~size_t(127)) + 2 * raw_layout(M, a.dv, es).bytes;
  auto kernel = a.rule == kFalcon2 ? falcon2_recurrent_kernel<M, true>
                                   : falcon2_recurrent_kernel<M, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<(unsigned)grid, kThreads, smem, stream>>>(a, ncg, err);
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
