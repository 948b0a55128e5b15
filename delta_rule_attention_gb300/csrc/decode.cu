// Single-token recurrent step (read after write) for N independent states.
//
// Per state: a = S^T x, b = S^T phi(q), r = v - a (Falcon-1) or v (Falcon-1A),
// o = gamma b + eta <x, phi(q)> r   (= S_t^T phi(q) with S_t below),
// S_t = gamma S + eta x r^T,  x_prev <- phi(k).
// The update order follows the one-step listing of page
// rcap.io/posts/fast-weight-attention-for-continual-learning-2026-08-27 and
// Eq. (3.3) of page hyper.ai/fr/papers/2608.27763.
//
// The step is HBM-bound: the fp32 state is read once and written once.
// Persistent CTAs (a few per SM, by state size) walk their share of the
// states through a ring of shared-memory stages filled by bulk async copies
// (state, q, k, x_prev and v of one state per stage), so the copies of the
// next states are in flight while a CTA reduces and writes back the current
// one.  A thread moves its share of the state (whole float4 groups of rows,
// so a warp covers contiguous rows) from the stage into registers before the
// reduction barrier, which frees the stage for the next copy at once; the
// two column reductions (S^T x and S^T q) run over the rows a thread holds,
// then across row groups through shared memory; the updated rows go from
// registers to global memory with evict-first stores.  Columns are
// independent given x, phi(q), eta and gamma, which one warp computes from
// the staged q, k and x_prev while the others reduce.

#include "common.cuh"
#include "tc_ptx.cuh"

namespace falcon {
namespace {

// The state streams through once per step (far larger than L2 at scale):
// evict-first stores.
__device__ __forceinline__ void st_stream(float* p, float4 v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}

// ---- streaming kernel ----------------------------------------------------
constexpr int kSmemPerSm = 233472;   // shared memory of one SM (bytes)
constexpr int kSmemPerCta = 232448;  // opt-in limit of one CTA
constexpr int kCtaReserve = 1024;    // reserved by the system per resident CTA

template <int M, int DV, int STAGES, int CTAS>
struct StreamCfg {
  static constexpr int kThreads = M * DV / 4 < 256 ? M * DV / 4 : 256;
  static constexpr int kLanesPerRow = DV / 4;
  static constexpr int kRowsPerPass = kThreads / kLanesPerRow;
  static constexpr int kIters = M / kRowsPerPass;
  // Stage layout (bytes): S [M][DV] fp32 | q [M] | k [M] | x_prev [M] | v [DV];
  // q, k, v are bf16 or fp32 and get room for fp32.  Every offset and every
  // copied size is a multiple of 16 bytes (M, DV >= 16).
  static constexpr uint32_t kSBytes = M * DV * 4;
  static constexpr uint32_t kQOff = kSBytes;
  static constexpr uint32_t kKOff = kQOff + M * 4;
  static constexpr uint32_t kXOff = kKOff + M * 4;
  static constexpr uint32_t kVOff = kXOff + M * 4;
  static constexpr uint32_t kStageBytes = kVOff + DV * 4;
  static constexpr int kStages = STAGES;
  static constexpr uint32_t kRedOff = kStages * kStageBytes;              // [kRowsPerPass][2][DV]
  static constexpr uint32_t kRsOff = kRedOff + kRowsPerPass * 2 * DV * 4;  // [DV]
  static constexpr uint32_t kScalOff = kRsOff + DV * 4;                    // 8 floats
  static constexpr uint32_t kBarOff = kScalOff + 32;
  static constexpr uint32_t kSmem = kBarOff + kStages * 8;
  static_assert(kThreads >= 64 && kThreads >= DV, "warp 0 and one thread per column");
  static_assert(kRowsPerPass * kIters == M, "rows per pass must divide M");
  static_assert(kStages >= 2, "at least two stages");
  static_assert(kSmem <= kSmemPerCta, "shared memory per CTA");
  static_assert(CTAS * (kSmem + kCtaReserve) <= kSmemPerSm, "resident CTAs per SM");
  static_assert(CTAS * kThreads <= 2048, "threads per SM");
};

template <int M, int DV, int STAGES, int CTAS>
__global__ void __launch_bounds__(StreamCfg<M, DV, STAGES, CTAS>::kThreads, CTAS)
    decode_stream_kernel(DecodeArgs a) {
  using Cfg = StreamCfg<M, DV, STAGES, CTAS>;
  constexpr int kStages = Cfg::kStages;
  extern __shared__ __align__(128) unsigned char smem[];
  float* red = reinterpret_cast<float*>(smem + Cfg::kRedOff);
  float* rs = reinterpret_cast<float*>(smem + Cfg::kRsOff);
  float* scal = reinterpret_cast<float*>(smem + Cfg::kScalOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);

  const int tid = threadIdx.x;
  const int col4 = tid % Cfg::kLanesPerRow;
  const int rgrp = tid / Cfg::kLanesPerRow;
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t count = first < a.N ? (a.N - 1 - first) / stride + 1 : 0;
  const bool bf16 = a.dtype == FALCON_BF16;
  const uint32_t esz = bf16 ? 2u : 4u;
  const uint32_t tx = Cfg::kSBytes + 2u * M * esz + M * 4u + DV * esz;

  // Copy the i-th state of this CTA (and its token's q, k, x_prev, v) into
  // stage i mod kStages.  One thread issues.
  auto issue = [&](int64_t i) {
    const int64_t n = first + i * stride;
    unsigned char* st = smem + (uint32_t)(i % kStages) * Cfg::kStageBytes;
    uint64_t* bar = &full[i % kStages];
    tc::mbar_expect_tx(bar, tx);
    tc::bulk_g2s(st, a.S + n * (int64_t)M * DV, Cfg::kSBytes, bar);
    tc::bulk_g2s(st + Cfg::kQOff, static_cast<const char*>(a.q) + n * M * esz, M * esz, bar);
    tc::bulk_g2s(st + Cfg::kKOff, static_cast<const char*>(a.k) + n * M * esz, M * esz, bar);
    tc::bulk_g2s(st + Cfg::kXOff, a.x_prev + n * M, M * 4u, bar);
    tc::bulk_g2s(st + Cfg::kVOff, static_cast<const char*>(a.v) + n * DV * esz, DV * esz, bar);
  };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) tc::mbar_init(&full[s], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t i = 0; i < count && i < kStages; ++i) issue(i);

  // Per-token scalars of the next state, loaded one state ahead (thread 0).
  float nb = 0.f, nl = 0.f;
  bool nf = false;
  if (tid == 0 && count > 0) {
    nb = a.beta[first];
    nl = a.lambda[first];
    nf = a.fresh ? a.fresh[first] != 0 : false;
  }

  for (int64_t i = 0; i < count; ++i) {
    const int64_t n = first + i * stride;
    const int s = (int)(i % kStages);
    const unsigned char* st = smem + (uint32_t)s * Cfg::kStageBytes;
    const float cb = nb, cl = nl;
    const bool cf = nf;
    if (tid == 0 && i + 1 < count) {
      const int64_t nn = n + stride;
      nb = a.beta[nn];
      nl = a.lambda[nn];
      nf = a.fresh ? a.fresh[nn] != 0 : false;
    }
    const bool ok = tc::mbar_wait(&full[s], (uint32_t)((i / kStages) & 1));

    // This thread's rows: state into registers, partial column sums of
    // S^T x and S^T q (q unscaled: phi(q) = f_q q with a scalar f_q).
    const float* Ss = reinterpret_cast<const float*>(st);
    const float* xs = reinterpret_cast<const float*>(st + Cfg::kXOff);
    float4 sv[Cfg::kIters];
    float xr[Cfg::kIters];
    float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
#pragma unroll
      for (int it = 0; it < Cfg::kIters; ++it) {
        const int row = rgrp + it * Cfg::kRowsPerPass;
        sv[it] = *reinterpret_cast<const float4*>(Ss + row * DV + col4 * 4);
        xr[it] = xs[row];
        const float qr = load_elem(st + Cfg::kQOff, row, a.dtype);
        pa[0] += sv[it].x * xr[it]; pa[1] += sv[it].y * xr[it];
        pa[2] += sv[it].z * xr[it]; pa[3] += sv[it].w * xr[it];
        pb[0] += sv[it].x * qr; pb[1] += sv[it].y * qr;
        pb[2] += sv[it].z * qr; pb[3] += sv[it].w * qr;
      }
    }
    *reinterpret_cast<float4*>(red + (rgrp * 2 + 0) * DV + col4 * 4) =
        make_float4(pa[0], pa[1], pa[2], pa[3]);
    *reinterpret_cast<float4*>(red + (rgrp * 2 + 1) * DV + col4 * 4) =
        make_float4(pb[0], pb[1], pb[2], pb[3]);
    const float vj = (ok && tid < DV) ? load_elem(st + Cfg::kVOff, tid, a.dtype) : 0.f;

    // Features and scalars (warp 0): ||q||, phi(k) (the next token's x),
    // E = ||x||^2, <x, phi(q)>, eta and gamma.
    if (tid < 32 && __all_sync(0xffffffffu, ok)) {
      const bool fr = __shfl_sync(0xffffffffu, cf ? 1 : 0, 0) != 0;
      float sq = 0.f, sk = 0.f, sx = 0.f, xq = 0.f;
      float kv[(M + 31) / 32];
#pragma unroll
      for (int e = 0; e < (M + 31) / 32; ++e) {
        const int r = tid + 32 * e;
        float qv = 0.f, xv = 0.f;
        kv[e] = 0.f;
        if (r < M) {
          qv = load_elem(st + Cfg::kQOff, r, a.dtype);
          kv[e] = load_elem(st + Cfg::kKOff, r, a.dtype);
          xv = fr ? 0.f : xs[r];
        }
        sq += qv * qv;
        sk += kv[e] * kv[e];
        sx += xv * xv;
        xq += xv * qv;
      }
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      const float E = warp_sum(sx);
      xq = warp_sum(xq);
      const float fq = feature_scale(sq, M, a.phi), fk = feature_scale(sk, M, a.phi);
#pragma unroll
      for (int e = 0; e < (M + 31) / 32; ++e) {
        const int r = tid + 32 * e;
        if (r < M) a.x_prev[n * M + r] = kv[e] * fk;
      }
      if (tid == 0) {
        float gamma, lg;
        const float eta = step_eta_gamma(cf, E, cb, ridge_of(cl, E, a.ridge), a.eps,
                                         a.eps_gamma, &gamma, &lg);
        scal[0] = eta;
        scal[1] = gamma;
        scal[2] = xq * fq;
        scal[3] = fq;
        scal[4] = cf ? 1.f : 0.f;
      }
    }
    // The stage is consumed: every read of it is above this barrier.
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        if (a.err) atomicExch(a.err, 1);
        // Let the copies still in flight land before the CTA leaves.
        for (int64_t j = i; j < count && j < i + kStages; ++j)
          tc::mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1));
      }
      return;
    }
    if (tid == 0 && i + kStages < count) issue(i + kStages);

    const float eta = scal[0], gamma = scal[1], xq = scal[2], fq = scal[3];
    const bool fr = scal[4] != 0.f;
    if (tid < DV) {
      float ta = 0.f, tb = 0.f;
#pragma unroll
      for (int g = 0; g < Cfg::kRowsPerPass; ++g) {
        ta += red[(g * 2 + 0) * DV + tid];
        tb += red[(g * 2 + 1) * DV + tid];
      }
      const float r = (a.rule == kFalcon1) ? vj - (fr ? 0.f : ta) : vj;
      rs[tid] = r;
      store_elem(a.o, n * DV + tid, gamma * (fq * tb) + eta * xq * r, a.dtype);
    }
    __syncthreads();

    // S_t = gamma S + eta x r^T, from registers to global memory.
    const float4 r4 = *reinterpret_cast<const float4*>(rs + col4 * 4);
    float* S = a.S + n * (int64_t)M * DV;
#pragma unroll
    for (int it = 0; it < Cfg::kIters; ++it) {
      const int row = rgrp + it * Cfg::kRowsPerPass;
      const float ex = fr ? 0.f : eta * xr[it];
      float4 w;
      w.x = gamma * sv[it].x + ex * r4.x;
      w.y = gamma * sv[it].y + ex * r4.y;
      w.z = gamma * sv[it].z + ex * r4.z;
      w.w = gamma * sv[it].w + ex * r4.w;
      st_stream(S + row * DV + col4 * 4, w);
    }
  }
}

template <int M, int DV, int STAGES, int CTAS>
cudaError_t launch_stream(const DecodeArgs& a, cudaStream_t stream) {
  using Cfg = StreamCfg<M, DV, STAGES, CTAS>;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_stream_kernel<M, DV, STAGES, CTAS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t slots = (int64_t)sms * CTAS;
  const int64_t grid = a.N < slots ? a.N : slots;
  decode_stream_kernel<M, DV, STAGES, CTAS>
      <<<(unsigned)grid, Cfg::kThreads, Cfg::kSmem, stream>>>(a);
  return cudaGetLastError();
}

// Stages and resident CTAs per SM by state size (measured on the decode step
// with bf16 q, k, v: fewer, larger states want deeper rings; smaller ones want
// more CTAs, so that one CTA's barriers overlap another's copies).
template <int M, int DV>
struct StreamChoice {
  static constexpr int kBytes = M * DV * 4;
  static constexpr int kStages = kBytes >= 65536 ? 3 : kBytes >= 32768 ? 2 : 3;
  static constexpr int kCtas = kBytes >= 65536   ? 1
                               : kBytes >= 16384 ? 2
                               : kBytes >= 8192  ? 4
                               : kBytes >= 4096  ? 8
                               : kBytes >= 2048  ? 16
                                                 : 24;
};

template <int M, int DV>
cudaError_t launch_mdv(const DecodeArgs& a, cudaStream_t stream) {
  return launch_stream<M, DV, StreamChoice<M, DV>::kStages, StreamChoice<M, DV>::kCtas>(a, stream);
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
