// Tensor-core (tcgen05) per-chunk gradients of the Falcon-1 / Falcon-1A
// backward pass, for bf16 inputs with m = d_v = 64 and chunk C = 64.
//
// It computes what bwd_grad_kernel of chunk_bwd.cu computes (the chunk form of
// the gradient; page hyper.ai/fr/papers/2608.27763, Section 3.1 Eq. (3.3),
// Section 4.3 Eq. (4.6), Section 4.4 Eq. (4.15)-(4.16)): with the state S
// entering the chunk and the cotangent dS' of the state leaving it,
//
//   R  = Diag(eta) V - Diag(eta e^{g_-}) X S,   U = T R,   T = (I + A)^{-1}
//   dU = P^T dO + Diag(e^{g_C - g}) X dS',       dR = T^T dU
//   dA = -(dR U^T) (j < i),  dP = (dO U^T) (j <= i),  dV = Diag(eta) dR
//   dQ = Diag(e^g) dO S^T + (dP o E) X
//   dX = -Diag(eta e^{g_-}) dR S^T + (dP o E)^T Q + Diag(e^{g_C - g}) U dS'^T
//        + (dK + dK^T) X + 2 Diag(dE) X
//
// and the step-size chain (log-prefix cotangent, clamp, eta, ridge).  Every
// contraction is a 64 x 64 x 64 tcgen05 MMA on bf16 operands in 128B-swizzled
// shared-memory tiles with fp32 accumulators in TMEM; two products that share
// an operand are stacked into one M = 128 MMA (the unused half of an M = 128
// operand reads a neighbouring tile and lands in accumulator lanes nobody
// reads).  Transposed operands are the same row-major tiles read MN-major.
// The unit-lower inverse T is the forward map kernel's solve (fp32 diagonal
// blocks, register-resident 8-column strips below them).  Epilogues run one
// accumulator row per thread (two threads per row, one per column half), so
// the per-row reductions of the step-size chain stay local; column sums go
// through shared-memory atomics.  Falcon-1A takes the same path with T = I
// and A = 0.
// The products that enter the residual r = v - S^T x (X S, and with them Q S
// and X dS') run as three bf16 MMAs on split operands, hi hi + hi lo + lo hi
// (v = hi + lo, hi = bf16(v)): the residual is a difference of nearly equal
// terms, and the step-size gradients are inner products with it.  P^T dO and
// T^T dU (the residual's cotangent) split P and dU the same way.  They and
// the other row sums of the step-size chain are formed from fp32 accumulator
// values.
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"
#include "tmap.cuh"

namespace falcon {

namespace {

using namespace tc;
using namespace tcu;

constexpr int kBC = 64;
constexpr int kBThreads = 256;
constexpr uint32_t kTile = 8192;  // 64 rows x 64 bf16, 128B-swizzled
// Shared memory: 13 tile slots of 8 KB from a 1024-aligned base, then the
// scalars.  Tiles whose lifetimes do not overlap share a slot (write -> last
// read):
//   0 X  1 Q  2 S  3 dS'  (the whole kernel)   6 dO (-> [dR; dO] U^T)
//   4 V (-> rv) | dPE                          5 dR (before dO: [dR; dO])
//   7 T (solve -> T^T dU) | dOs = Diag(e^g) dO
//   8 Xlo | A (bf16) | R | dU | dK              9 Qlo | A's diagonal blocks (fp32) | U
//   10 Slo | T's diagonal blocks (solve) | Us = Diag(e^{g_C-g}) U
//   11 dSlo | P | dUlo                          12 Plo | dRs = -Diag(eta e^{g_-}) dR
// The unused half of an M = 128 K-major operand reads the next slot (slot 13
// is the scalars: valid memory), that of an MN-major operand the slot LBO
// bytes on.  With 113 KB of shared memory and 256 TMEM columns two CTAs share
// an SM.
enum : int { kX = 0, kQt, kS, kdS, kV, kdR, kdO, kT, kW8, kW9, kW10, kW11, kW12, kSlots };
constexpr int kdPE = kV, kdOs = kT, kXlo = kW8, kSlo = kW10, kdSlo = kW11;  // Qlo = slot 9
constexpr int kR = kW8, kdU = kW8, kdK = kW8, kU = kW9, kUs = kW10, kP = kW11, kdUlo = kW11;
constexpr int kPlo = kW12, kdRs = kW12;
constexpr uint32_t kScOff = kSlots * kTile;
static_assert(64 * kLdD * 4 <= kTile, "A's diagonal blocks within one slot");

struct BwdScalars {
  float eta[64], g[64], gx[64], E[64], lame[64], den[64], gam[64];
  float deta[64], dg[64], dE[64], xwd[64];
  // accumulated with shared-memory atomics (zeroed first)
  float qz[64], rv[64], xy[64], xw[64], sAr[64], sAc[64], spr[64], spc[64];
  float ssk[64];      // ||k_{t0+i-1}||^2 of the raw write-feature rows
  float ssp[2][128];  // half-row partial sums
  float ugp[2][128];
  float fc[64];       // e^{r - g_j}, r = g_C / 2 (chunks with a log-decay span <= kBwdFactorSpan)
  float sds;          // <dS', S>_F
  int flag[64];
  int fail;
  uint64_t bar_in, bar_mma;
  uint32_t tmem_base;
};
// The scalars get a full slot: the unused half of the operands in slot 12
// reads it.  Two CTAs of kBwdSmem (+1 KB reserved each) fill an SM's 228 KB.
static_assert(sizeof(BwdScalars) <= kTile, "scalars within one slot");
constexpr size_t kBwdSmem = kScOff + kTile + 1024;
static_assert(2 * (kBwdSmem + 1024) <= 228 * 1024, "two CTAs per SM");
constexpr uint32_t kTmemCols = 256;
// TMEM columns of the accumulators (128 lanes each).
constexpr uint32_t kD1 = 0;     // [X; Q] X^T (until the dA, dP epilogue)
constexpr uint32_t kD2a = 64;   // [X; Q] S  -> dQ = [.; dPE] X + [.; dOs] S^T
constexpr uint32_t kD2b = 128;  // [X; Q] dS' -> dX - 2 Diag(dE) X
constexpr uint32_t kD3 = 192;   // T R, P^T dO, T^T dU, [dR; dO] U^T in turn
enum : int { kLive = 1, kClamped = 2 };

__device__ __forceinline__ float expn(float x) { return __expf(fminf(x, 0.f)); }

// A chunk whose log-decay spans at most this much factors every e^{a - b} of
// its decay tiles as e^{a - r} e^{r - b} with r = g_C / 2 (both factors stay
// within fp32 range): one exponential per row and per column instead of one
// per element.
constexpr float kBwdFactorSpan = 80.f;

// Half row (32 values) of a swizzled tile as bf16 hi parts, and the rounding
// remainders as the lo tile.
__device__ __forceinline__ void store_half_split(unsigned char* hi, unsigned char* lo, int r,
                                                 int h, const float* v) {
  float rest[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) rest[j] = v[j] - __bfloat162float(__float2bfloat16_rn(v[j]));
  store_half_sw(hi, r, h, v, 1.f);
  store_half_sw(lo, r, h, rest, 1.f);
}

// Wait for the MMA group committed last, with the CTA-wide failure agreement.
__device__ __forceinline__ bool wait_mma(BwdScalars& sc, uint32_t& phase) {
  if (!mbar_wait_backoff(&sc.bar_mma, phase)) sc.fail = 1;
  phase ^= 1u;
  tc_fence_after();
  return !__syncthreads_or(sc.fail);
}

// The same wait without the barrier: where the thread then only reads the
// accumulators and overwrites tiles the completed MMAs no longer need, it
// needs no other thread; a failed wait is agreed on at the next barrier.
__device__ __forceinline__ void wait_mma_own(BwdScalars& sc, uint32_t& phase) {
  if (!mbar_wait_backoff(&sc.bar_mma, phase)) sc.fail = 1;
  phase ^= 1u;
  tc_fence_after();
}

// Warp-wide scans of 64 values, two per lane.  Prefix: lane l takes elements
// 2l, 2l+1 and writes the exclusive and inclusive prefix sums.  Suffix: lane l
// takes elements 63-2l, 62-2l of v and writes sum_{j >= i} v_j to out.
__device__ __forceinline__ float warp_incl_scan(float s) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, s, o);
    if (lane >= o) s += t;
  }
  return s;
}
__device__ __forceinline__ void warp_prefix64(float* v, float* excl) {
  const int l = threadIdx.x & 31;
  const float a = v[2 * l], b = v[2 * l + 1];
  const float e = warp_incl_scan(a + b) - (a + b);
  excl[2 * l] = e;
  excl[2 * l + 1] = e + a;
  v[2 * l] = e + a;
  v[2 * l + 1] = (e + a) + b;
}
__device__ __forceinline__ void warp_suffix64(const float* v0, const float* v1, float* out) {
  const int l = threadIdx.x & 31;
  const float a = v0[0], b = v1[0];  // elements 63 - 2l and 62 - 2l
  const float e = warp_incl_scan(a + b) - (a + b);
  out[63 - 2 * l] = e + a;
  out[62 - 2 * l] = (e + a) + b;
}

// g <- J_phi(u)^T g for a half row (32 values) of a 64-wide feature row u,
// given the row's ||u||^2 and <u, g> (phi as in the forward: l2 u / ||u||,
// RMSNorm u / sqrt(||u||^2 / 64 + eps_rms), or the identity).
__device__ __forceinline__ void phi_vjp_half(float* g, const float* u, float ss, float ug,
                                             int phi) {
  if (phi == FALCON_PHI_L2) {
    const float nrm = sqrtf(ss);
    if (nrm < 1e-12f) {
#pragma unroll
      for (int j = 0; j < 32; ++j) g[j] *= 1e12f;
    } else {
      const float inv = 1.f / nrm, c2 = ug * inv * inv;
#pragma unroll
      for (int j = 0; j < 32; ++j) g[j] = (g[j] - u[j] * c2) * inv;
    }
  } else if (phi == FALCON_PHI_RMS) {
    const float sr = rsqrtf(ss / 64.f + kEpsRms), c3 = sr * sr * sr * ug / 64.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) g[j] = sr * g[j] - c3 * u[j];
  }
}

// 32 bf16 values (64 bytes) from global memory.
__device__ __forceinline__ void load_bf16x32(const void* p, float* v) {
  const uint4* src = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int q8 = 0; q8 < 4; ++q8) {
    const uint4 pk = src[q8];
    const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&pk);
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const float2 f = __bfloat1622float2(hv[e2]);
      v[8 * q8 + 2 * e2] = f.x;
      v[8 * q8 + 2 * e2 + 1] = f.y;
    }
  }
}

// Generic-proxy tile writes of this CTA become visible to the next MMA.
__device__ __forceinline__ void publish_tiles() {
  tc_fence_before();
  fence_async_smem();
  __syncthreads();
}

// The same, agreeing on a failed wait: false if any thread saw one.
__device__ __forceinline__ bool publish_tiles_ok(BwdScalars& sc) {
  tc_fence_before();
  fence_async_smem();
  return !__syncthreads_or(sc.fail);
}

// Column sums of a warp's 32 rows: v holds 32 consecutive columns of this
// lane's row; afterwards lane l returns the sum over the warp's rows of column
// l (recursive halving, 31 shuffles).
__device__ __forceinline__ float warp_col_sum32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int sh = 16; sh >= 1; sh >>= 1) {
    const bool up = (lane & sh) != 0;
#pragma unroll
    for (int k = 0; k < sh; ++k) {
      const float send = up ? v[k] : v[k + sh];
      const float keep = up ? v[k + sh] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
    }
  }
  return v[0];
}

__global__ void __launch_bounds__(kBThreads, 2)
    tc_bwd_grad_kernel(BwdArgs b, int nchunks, const float* S_starts, const float* dS_ends,
                       float* edge, int* err, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do) {
  const ChunkArgs& a = b.f;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = align1024(smem_raw);
  BwdScalars& sc = *reinterpret_cast<BwdScalars*>(base + kScOff);
  auto tile = [&](int i) { return base + i * kTile; };
  auto taddr = [&](int i) { return smem_addr(base + i * kTile); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, h = tid >> 7;  // accumulator lane, column half
  const int i = r & 63;                   // row of the 64-row tile this thread serves
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t T = a.T, t0 = (int64_t)c * kBC, rowbase = bh * T;
  const int n = (int)min((int64_t)kBC, T - t0);
  const bool f1 = a.rule == kFalcon1;
  const float* S = S_starts + (bh * nchunks + c) * 4096;
  const float* dSp = dS_ends + (bh * nchunks + c) * 4096;

  // The state entering the chunk and the cotangent leaving it are read only
  // after the feature phase: start bringing them into L2 now.
  if (tid == 0) {
    bulk_prefetch_l2(S, 4096 * 4);
    bulk_prefetch_l2(dSp, 4096 * 4);
  }
  // TMEM is allocated by warp 1, so that thread 0 issues the input tile copies
  // (the head of the CTA's chain) without waiting for the allocation.
  if (warp == 1) tmem_alloc(&sc.tmem_base, kTmemCols);
  if (tid == 0) {
    mbar_init(&sc.bar_in, 1);
    mbar_init(&sc.bar_mma, 1);
    fence_mbar_init();
    sc.fail = 0;
    sc.sds = 0.f;
    // raw k rows t0-1 .. t0+62 (row -1 reads zeros), q, v and dO rows t0 ..
    mbar_expect_tx(&sc.bar_in, 4 * kTile);
    tma_load_3d(tile(kX), &tm_k, 0, (int)(t0 - 1), (int)bh, &sc.bar_in);
    tma_load_3d(tile(kQt), &tm_q, 0, (int)t0, (int)bh, &sc.bar_in);
    tma_load_3d(tile(kV), &tm_v, 0, (int)t0, (int)bh, &sc.bar_in);
    tma_load_3d(tile(kdO), &tm_do, 0, (int)t0, (int)bh, &sc.bar_in);
  }
  // Per-token inputs of threads 0..63, loaded early (used after the features).
  float beta_t = 0.f, lam_t = 0.f;
  if (tid < n) {
    beta_t = a.beta[rowbase + t0 + tid];
    lam_t = a.lambda[rowbase + t0 + tid];
  }
  if (tid < 64) {
    sc.qz[tid] = sc.rv[tid] = sc.xy[tid] = sc.xw[tid] = 0.f;
    sc.sAr[tid] = sc.sAc[tid] = sc.spr[tid] = sc.spc[tid] = 0.f;
  }
  tc_fence_before();
  __syncthreads();  // barriers initialised, accumulators zeroed
  tc_fence_after();
  const uint32_t tmem = sc.tmem_base;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * h;  // + column
  uint32_t phase = 0;
  float gC = 0.f, rr = 0.f;
  bool factored = false;
  if (!mbar_wait_backoff(&sc.bar_in, 0)) sc.fail = 1;
  if (__syncthreads_or(sc.fail)) goto teardown;

  // ---- features: rows 0..63 of [X; Q] are x_i = phi(k_{t0+i-1}) (x_prev, or
  //      the sentinel zero, at t = 0), rows 64..127 are phi(q_{t0+i}); rows
  //      past the chunk's tokens are zero.
  {
    float v[32];
    load_half_sw(tile(kX), r, h, v);
    const bool xrow = r < 64;
    const bool given = xrow && t0 + i == 0 && a.x_prev != nullptr;
    const bool dead = i >= n || (xrow && t0 + i == 0 && a.x_prev == nullptr);
    if (given)
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = a.x_prev[bh * 64 + 32 * h + j];
    sc.ssp[h][r] = sumsq32(v);
    __syncthreads();
    const float ss = sc.ssp[0][r] + sc.ssp[1][r];
    const float s = dead ? 0.f : (given ? 1.f : phi_scale(ss, 64, a.phi));
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= s;
    store_half_split(tile(kX), tile(kXlo), r, h, v);
    if (xrow && h == 0) {
      sc.E[i] = ss * s * s;
      sc.ssk[i] = ss;
    }
  }
  __syncthreads();
  // The state row (or cotangent row) of this thread and, for the state rows,
  // the matching cotangent row: requested now, consumed after the scalars.
  float4 srow[8], drow[8];
  {
    const float4* src = reinterpret_cast<const float4*>(
        (r < 64 ? S + r * 64 : dSp + (r - 64) * 64) + 32 * h);
    const float4* d4 = reinterpret_cast<const float4*>(dSp + (r & 63) * 64 + 32 * h);
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) srow[q4] = src[q4];
    if (r < 64) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) drow[q4] = d4[q4];
    }
  }
  // ---- per-token scalars as the forward forms them, then the log prefixes
  if (tid < 64) {
    float et = 0.f, gm = 1.f, lg = 0.f, le = 0.f, d = 1.f;
    int fl = 0;
    if (tid < n) {
      const int64_t t = t0 + tid;
      const bool sentinel = (t == 0) && (a.x_prev == nullptr);
      le = ridge_of(lam_t, sc.E[tid], a.ridge);
      d = sc.E[tid] + le + a.eps;
      et = step_eta_gamma(sentinel, sc.E[tid], beta_t, le, a.eps, a.eps_gamma, &gm,
                          &lg);
      if (!sentinel && d > 0.f) fl |= kLive;
      if (et * le >= 1.f - a.eps_gamma) fl |= kClamped;
    }
    sc.eta[tid] = et;
    sc.gam[tid] = gm;
    sc.g[tid] = lg;
    sc.lame[tid] = le;
    sc.den[tid] = d;
    sc.flag[tid] = fl;
  }
  __syncthreads();
  if (warp == 0) warp_prefix64(sc.g, sc.gx);  // g: inclusive, gx: exclusive
  // [S; dS'] as split bf16 operand tiles (thread: row r of the pair, half h),
  // and <dS', S>_F from the state rows' threads.
  {
    float v[32];
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
      v[4 * q4] = srow[q4].x;
      v[4 * q4 + 1] = srow[q4].y;
      v[4 * q4 + 2] = srow[q4].z;
      v[4 * q4 + 3] = srow[q4].w;
    }
    float acc = 0.f;
    if (r < 64) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 y = drow[q4];
        acc += v[4 * q4] * y.x + v[4 * q4 + 1] * y.y + v[4 * q4 + 2] * y.z + v[4 * q4 + 3] * y.w;
      }
    }
    acc = warp_sum(acc);  // warps 2, 3, 6, 7 (rows of dS') add zeros
    if (lane == 0 && r < 64) atomicAdd(&sc.sds, acc);
    store_half_split(tile(kS), tile(kSlo), r, h, v);
  }
  publish_tiles();
  gC = sc.g[63];
  factored = -gC <= kBwdFactorSpan;
  rr = 0.5f * gC;

  // ---- MMA: [X; Q] X^T, [X; Q] S and [X; Q] dS' (split operands)
  if (tid == 0) {
    tc_fence_after();
    mma_k64(tmem + kD1, taddr(kX), false, 16, taddr(kX), false, 16,
            idesc_bf16(128, 64, false, false), false);
    const uint32_t id = idesc_bf16(128, 64, false, true);
    mma_k64(tmem + kD2a, taddr(kX), false, 16, taddr(kS), true, kTile, id, false);
    mma_k64(tmem + kD2a, taddr(kX), false, 16, taddr(kSlo), true, kTile, id, true);
    mma_k64(tmem + kD2a, taddr(kXlo), false, 16, taddr(kS), true, kTile, id, true);
    mma_k64(tmem + kD2b, taddr(kX), false, 16, taddr(kdS), true, kTile, id, false);
    mma_k64(tmem + kD2b, taddr(kX), false, 16, taddr(kdSlo), true, kTile, id, true);
    mma_k64(tmem + kD2b, taddr(kXlo), false, 16, taddr(kdS), true, kTile, id, true);
    mma_commit(&sc.bar_mma);
  }
  if (tid < 64 && factored) sc.fc[tid] = __expf(rr - sc.g[tid]);
  if (!wait_mma(sc, phase)) goto teardown;
  // A (for the solve, over the dead low parts: bf16 in slot 8, its fp32
  // diagonal blocks in slot 9), qz_i = <dO_i, (Q S)_i>
  {
    float d[32], w[32];
    if (r < 64) {
      const float ei = sc.eta[i], gxi = sc.gx[i];
      tmem_ld32(tl + kD1, d);
      if (factored) {
        const float ea = ei * __expf(gxi - rr);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * h + jj;
          d[jj] = (f1 && j < i) ? ea * sc.fc[j] * d[jj] : 0.f;
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * h + jj;
          d[jj] = (f1 && j < i) ? ei * expn(gxi - sc.g[j]) * d[jj] : 0.f;
        }
      }
      store_half_sw(tile(kW8), i, h, d, 1.f);
      if (h == (i >> 5)) {  // columns 16 (i / 16) .. +15 lie in this half
        float* drow = reinterpret_cast<float*>(tile(kW9)) + i * kLdD;
        if (i & 16) {
#pragma unroll
          for (int k = 0; k < 16; ++k) drow[k] = d[16 + k];
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) drow[k] = d[k];
        }
      }
    } else {
      tmem_ld32(tl + kD2a, d);
      load_half_sw(tile(kdO), i, h, w);
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) acc += w[jj] * d[jj];
      atomicAdd(&sc.qz[i], acc);
    }
  }
  __syncthreads();
  // ---- T = (I + A)^{-1} as a bf16 tile (T = I for Falcon-1A)
  if (f1) {
    solve_unit_lower_sw<false>(tile(kW8), reinterpret_cast<const float*>(tile(kW9)), tile(kT),
                               tile(kW10), nullptr);
  } else if (r < 64) {
    float v[32];
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) v[jj] = (32 * h + jj == i) ? 1.f : 0.f;
    store_half_sw(tile(kT), i, h, v, 1.f);
  }
  __syncthreads();
  // R = Diag(eta) (V - Diag(e^{g_-}) X S) (over A, now dead)
  if (r < 64) {
    float v[32], w[32];
    tmem_ld32(tl + kD2a, v);
    load_half_sw(tile(kV), i, h, w);
    const float bx = f1 ? __expf(sc.gx[i]) : 0.f;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) w[jj] = w[jj] - bx * v[jj];  // residual part
    store_half_sw(tile(kR), i, h, w, sc.eta[i]);
  }
  publish_tiles();
  // ---- U = T R
  if (tid == 0) {
    tc_fence_after();
    mma_k64(tmem + kD3, taddr(kT), false, 16, taddr(kR), true, kTile,
            idesc_bf16(128, 64, false, true), false);
    mma_commit(&sc.bar_mma);
  }
  wait_mma_own(sc, phase);
  // U and Us = Diag(e^{g_C - g}) U tiles, xw_i = <(X dS')_i, U_i>; P (split)
  {
    float d[32], e[32];
    if (r < 64) {
      tmem_ld32(tl + kD3, d);
      store_half_sw(tile(kU), i, h, d, 1.f);
      store_half_sw(tile(kUs), i, h, d, expn(gC - sc.g[i]));
      tmem_ld32(tl + kD2b, e);
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) acc += e[jj] * d[jj];
      atomicAdd(&sc.xw[i], acc);
    } else {
      const float gi = sc.g[i];
      tmem_ld32(tl + kD1, d);
      if (factored) {
        const float ep = __expf(gi - rr);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * h + jj;
          d[jj] = (j <= i) ? ep * sc.fc[j] * d[jj] : 0.f;
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * h + jj;
          d[jj] = (j <= i) ? expn(gi - sc.g[j]) * d[jj] : 0.f;
        }
      }
      store_half_split(tile(kP), tile(kPlo), i, h, d);
    }
  }
  if (!publish_tiles_ok(sc)) goto teardown;
  // ---- P^T dO (split P)
  if (tid == 0) {
    tc_fence_after();
    const uint32_t id = idesc_bf16(128, 64, true, true);
    mma_k64(tmem + kD3, taddr(kP), true, kTile, taddr(kdO), true, kTile, id, false);
    mma_k64(tmem + kD3, taddr(kPlo), true, kTile, taddr(kdO), true, kTile, id, true);
    mma_commit(&sc.bar_mma);
  }
  wait_mma_own(sc, phase);
  // dU = P^T dO + Diag(e^{g_C - g}) X dS' (split)
  if (r < 64) {
    float d[32], xd[32];
    tmem_ld32(tl + kD3, d);
    tmem_ld32(tl + kD2b, xd);
    const float f = expn(gC - sc.g[i]);
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) d[jj] += f * xd[jj];
    store_half_split(tile(kdU), tile(kdUlo), i, h, d);
  }
  if (!publish_tiles_ok(sc)) goto teardown;
  // ---- dR = T^T dU
  if (tid == 0) {
    tc_fence_after();
    const uint32_t id = idesc_bf16(128, 64, true, true);
    mma_k64(tmem + kD3, taddr(kT), true, kTile, taddr(kdU), true, kTile, id, false);
    mma_k64(tmem + kD3, taddr(kT), true, kTile, taddr(kdUlo), true, kTile, id, true);
    mma_commit(&sc.bar_mma);
  }
  wait_mma_own(sc, phase);
  // dR and dRs = -Diag(eta e^{g_-}) dR tiles; dv = Diag(eta) dR;
  // rv_i = <dR_i, v_i - e^{g_{i-1}} (X S)_i>, xy_i = <dR_i, (X S)_i>
  if (r < 64) {
    float d[32], w[32], xs[32];
    tmem_ld32(tl + kD3, d);
    store_half_sw(tile(kdR), i, h, d, 1.f);
    const float ei = sc.eta[i], bx = f1 ? __expf(sc.gx[i]) : 0.f;
    store_half_sw(tile(kdRs), i, h, d, -ei * bx);
    load_half_sw(tile(kV), i, h, w);
    tmem_ld32(tl + kD2a, xs);
    float acc = 0.f, axs = 0.f;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      acc += d[jj] * (w[jj] - bx * xs[jj]);
      axs += d[jj] * xs[jj];
    }
    atomicAdd(&sc.rv[i], acc);
    atomicAdd(&sc.xy[i], axs);
    if (i < n) {
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(b.dv) +
                                            (rowbase + t0 + i) * 64 + 32 * h);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) dst[q8] = pack8(d + 8 * q8, ei);
    }
  }
  if (!publish_tiles_ok(sc)) goto teardown;
  // ---- [dR; dO] U^T: rows 0..63 -dA (before masking), rows 64..127 dP
  if (tid == 0) {
    tc_fence_after();
    mma_k64(tmem + kD3, taddr(kdR), false, 16, taddr(kU), false, 16,
            idesc_bf16(128, 64, false, false), false);
    mma_commit(&sc.bar_mma);
  }
  wait_mma_own(sc, phase);
  {
    float d[32], e[32], pr[32];
    if (r < 64) {
      // dA (Falcon-1) with A recomputed from the Gram accumulator; dK tile
      const float ei = sc.eta[i], gxi = sc.gx[i];
      const float ea = factored ? ei * __expf(gxi - rr) : 0.f;
      tmem_ld32(tl + kD3, d);
      tmem_ld32(tl + kD1, e);
      float sar = 0.f;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = 32 * h + jj;
        const float fa = (f1 && j < i) ? (factored ? ea * sc.fc[j] : ei * expn(gxi - sc.g[j]))
                                       : 0.f;
        const float da = -d[jj];
        pr[jj] = da * fa * e[jj];  // dA_ij A_ij
        sar += pr[jj];
        d[jj] = da * fa;           // dK_ij
      }
      atomicAdd(&sc.sAr[i], sar);
      store_half_sw(tile(kdK), i, h, d, 1.f);
      atomicAdd(&sc.sAc[32 * h + lane], warp_col_sum32(pr));
    } else {
      // dP with P (fp32) from the Gram accumulator; dPE and dOs tiles
      const float gi = sc.g[i];
      const float ep = factored ? __expf(gi - rr) : 0.f;
      tmem_ld32(tl + kD3, d);
      tmem_ld32(tl + kD1, e);
      float spr = 0.f;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = 32 * h + jj;
        const float ef = (j <= i) ? (factored ? ep * sc.fc[j] : expn(gi - sc.g[j])) : 0.f;
        pr[jj] = d[jj] * ef * e[jj];  // dP_ij P_ij
        spr += pr[jj];
        d[jj] *= ef;
      }
      atomicAdd(&sc.spr[i], spr);
      store_half_sw(tile(kdPE), i, h, d, 1.f);
      load_half_sw(tile(kdO), i, h, e);
      store_half_sw(tile(kdOs), i, h, e, __expf(gi));
      atomicAdd(&sc.spc[32 * h + lane], warp_col_sum32(pr));
    }
  }
  if (__syncthreads_or(sc.fail)) goto teardown;
  // ---- the step-size cotangent, the log-prefix cotangent and its suffix sums,
  //      then dbeta, dlambda and dE per token
  if (tid < 64) {
    float de = sc.rv[tid];  // <dR_i, v_i - e^{g_{i-1}} (X S)_i>
    if (f1 && sc.eta[tid] != 0.f) de += sc.sAr[tid] / sc.eta[tid];
    sc.deta[tid] = de;
    const float xwd = expn(gC - sc.g[tid]) * sc.xw[tid];
    sc.xwd[tid] = xwd;
    sc.dg[tid] = __expf(sc.g[tid]) * sc.qz[tid] + sc.spr[tid] - sc.spc[tid] - xwd -
                 (f1 ? sc.sAc[tid] : 0.f);
  }
  __syncthreads();
  if (warp == 0) {
    // terms at index i - 1 (Falcon-1) and at C - 1, then the suffix sums
    const float tail = warp_sum(sc.xwd[2 * lane] + sc.xwd[2 * lane + 1]) + __expf(gC) * sc.sds;
    float v[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int k = 63 - 2 * lane - u;
      float x = sc.dg[k];
      if (f1 && k < 63)
        x += -sc.eta[k + 1] * __expf(sc.gx[k + 1]) * sc.xy[k + 1] + sc.sAr[k + 1];
      if (k == 63) x += tail;
      v[u] = x;
    }
    __syncwarp();
    warp_suffix64(&v[0], &v[1], sc.dg);
  }
  __syncthreads();
  if (tid < 64) {
    float dEi = 0.f;
    if (tid < n) {
      float db = 0.f, dl_in = 0.f;
      if (sc.flag[tid] & kLive) {
        float de = sc.deta[tid], dl = 0.f;
        if (!(sc.flag[tid] & kClamped)) {
          const float dal = -sc.dg[tid] / sc.gam[tid];
          de += sc.lame[tid] * dal;
          dl += sc.eta[tid] * dal;
        }
        db = de / sc.den[tid];
        const float dden = -de * sc.eta[tid] / sc.den[tid];
        dEi = dden;
        dl += dden;
        if (a.ridge == FALCON_RIDGE_SCALED) {
          dl_in = dl * sc.E[tid];
          dEi += dl * lam_t;
        } else {
          dl_in = dl;
        }
      }
      b.dbeta[rowbase + t0 + tid] = db;
      b.dlambda[rowbase + t0 + tid] = dl_in;
    }
    sc.dE[tid] = dEi;
  }
  publish_tiles();
  // ---- dQ = [.; dPE] X + [.; dOs] S^T (rows 64..127 of kD2a);
  //      dX - 2 Diag(dE) X = dPE^T Q + dK X + dK^T X + dRs S^T + Us dS'^T (rows 0..63 of kD2b)
  if (tid == 0) {
    tc_fence_after();
    mma_k64(tmem + kD2a, taddr(kdPE - 1), false, 16, taddr(kX), true, kTile,
            idesc_bf16(128, 64, false, true), false);
    mma_k64(tmem + kD2a, taddr(kdOs - 1), false, 16, taddr(kS), false, 16,
            idesc_bf16(128, 64, false, false), true);
    mma_k64(tmem + kD2b, taddr(kdPE), true, kTile, taddr(kQt), true, kTile,
            idesc_bf16(128, 64, true, true), false);
    mma_k64(tmem + kD2b, taddr(kdK), false, 16, taddr(kX), true, kTile,
            idesc_bf16(128, 64, false, true), true);
    mma_k64(tmem + kD2b, taddr(kdK), true, kTile, taddr(kX), true, kTile,
            idesc_bf16(128, 64, true, true), true);
    mma_k64(tmem + kD2b, taddr(kdRs), false, 16, taddr(kS), false, 16,
            idesc_bf16(128, 64, false, false), true);
    mma_k64(tmem + kD2b, taddr(kUs), false, 16, taddr(kdS), false, 16,
            idesc_bf16(128, 64, false, false), true);
    mma_commit(&sc.bar_mma);
  }
  if (!wait_mma(sc, phase)) goto teardown;
  {
    float d[32], u[32];
    float ss = 0.f, ug = 0.f;
    if (r < 64) {
      // dX_i; row i >= 1 is the cotangent of x_i = phi(k_{t0+i-1}), so dk of
      // that token follows here; row 0 (the previous chunk's last token, or
      // x_prev) goes to the edge buffer.
      tmem_ld32(tl + kD2b, d);
      load_half_sw(tile(kX), i, h, u);
      const float fe = 2.f * sc.dE[i];
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) d[jj] += fe * u[jj];
      if (i == 0) {
        float4* dst = reinterpret_cast<float4*>(edge + (bh * nchunks + c) * 64 + 32 * h);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          dst[q4] = make_float4(d[4 * q4], d[4 * q4 + 1], d[4 * q4 + 2], d[4 * q4 + 3]);
      } else if (i < n) {
        load_bf16x32(reinterpret_cast<const __nv_bfloat16*>(a.k) + (rowbase + t0 + i - 1) * 64 +
                         32 * h, u);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) ug += u[jj] * d[jj];
      }
    } else {
      tmem_ld32(tl + kD2a, d);  // dQ_i
      if (i < n) {
        load_bf16x32(reinterpret_cast<const __nv_bfloat16*>(a.q) + (rowbase + t0 + i) * 64 +
                         32 * h, u);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          ss += u[jj] * u[jj];
          ug += u[jj] * d[jj];
        }
      }
    }
    sc.ssp[h][r] = ss;
    sc.ugp[h][r] = ug;
    __syncthreads();
    // dk = J_phi(k)^T dX (rows 1 .. n-1), dq = J_phi(q)^T dQ (rows < n)
    const bool out = (r < 64) ? (i >= 1 && i < n) : (i < n);
    if (out) {
      const float ssr = (r < 64) ? sc.ssk[i] : sc.ssp[0][r] + sc.ssp[1][r];
      phi_vjp_half(d, u, ssr, sc.ugp[0][r] + sc.ugp[1][r], a.phi);
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(r < 64 ? b.dk : b.dq) +
                           (rowbase + t0 + i - (r < 64 ? 1 : 0)) * 64 + 32 * h;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) reinterpret_cast<uint4*>(dst)[q8] = pack8(d + 8 * q8, 1.f);
    }
  }

teardown:
  if (sc.fail && tid == 0) atomicExch(err, 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Reverse scan of the state cotangent over the tensor-core forward's maps,
// one CTA per head, newest chunk first:
//   dS_c = e^{g_C} dS' + Mc^T [dS'; dO_c]
// (Mc as stored: the state rows -Xt^T W without the e^{g_C} I part, the output
// rows Diag(e^g) Q - P W).  The MMAs read the stored Mc tile MN-major as Mc^T
// (K = 128: the state rows, then the output rows).  Per chunk two MMAs go into
// one of two TMEM accumulators: Mc_bot^T dO_c first (it does not depend on the
// chain, and is issued as soon as the chunk's stage has landed), then
// Mc_top^T dS' once the state threads have put dS' (bf16) in the operand tile;
// the e^{g_C} dS' part stays in fp32 registers.  Warps 0, 1, 4, 5 own state
// row 32 (w & 3) + lane and columns 32 (w >> 2) .. +31 (TMEM lanes 0..63);
// lane 0 of warp 2 issues the MMAs; lane 0 of warp 3 refills a ring of
// kRevStages stages (Mc, dO_c, e^{g_C}) as the MMAs and the state warps are
// done with one.  Every hand-off is an mbarrier; the chain per chunk is the
// state MMA, one accumulator read, the fp32 update and the operand write.
constexpr int kRevStages = 4;
constexpr int kRevThreads = 192;
constexpr uint32_t kRevStage = kMcBytes + kTile;  // Mc | dO_c

struct RevSmem {
  unsigned char stage[kRevStages][kRevStage];
  unsigned char op[kTile];  // dS' as the MN-major B operand
  float gc[kRevStages][4];
  uint64_t full[kRevStages];   // the stage has landed
  uint64_t empty[kRevStages];  // both MMAs and the state warps are done with the stage
  uint64_t mma_done[2];        // both MMAs into accumulator b have completed
  uint64_t s_ready;            // dS' of the next chunk is in op
  uint32_t tmem_base;
  int fail;
};

__device__ __forceinline__ void rev_issue_load(RevSmem& s, int st, const unsigned char* map,
                                               const CUtensorMap* tm_do, int t0, int bh) {
  mbar_expect_tx(&s.full[st], kMcBytes + 16 + kTile);
  bulk_g2s(s.stage[st], map, kMcBytes, &s.full[st]);
  bulk_g2s(s.gc[st], map + kMcBytes + kNcBytes, 16, &s.full[st]);
  tma_load_3d(s.stage[st] + kMcBytes, tm_do, 0, t0, bh, &s.full[st]);
}

__global__ void __launch_bounds__(kRevThreads)
    tc_bwd_scan_kernel(BwdArgs b, int nchunks, const unsigned char* maps, float* dS_ends,
                       int* err, const __grid_constant__ CUtensorMap tm_do) {
  extern __shared__ unsigned char smem_raw[];
  RevSmem& s = *reinterpret_cast<RevSmem*>(align1024(smem_raw));
  volatile int* fail = &s.fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bh = blockIdx.x;
  const bool state = (warp & 3) < 2;  // warps 0, 1, 4, 5
  const int row = 32 * (warp & 3) + lane, h = warp >> 2;
  const int n = nchunks;
  const unsigned char* hmaps = maps + (size_t)bh * nchunks * kMapBytes;
  if (warp == 0) tmem_alloc(&s.tmem_base, 128);
  if (tid == 0) {
    for (int st = 0; st < kRevStages; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], 1 + 4);  // the MMAs' commit, the four state warps
    }
    mbar_init(&s.mma_done[0], 1);
    mbar_init(&s.mma_done[1], 1);
    mbar_init(&s.s_ready, 4);
    fence_mbar_init();
    s.fail = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 2) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 64, true, true);
      for (int k = 0; k < n; ++k) {
        const int st = k % kRevStages, bb = k & 1;
        const uint32_t stg = smem_addr(s.stage[st]);
        // Accumulator bb was last read for chunk k - 2, before the state
        // threads signalled the operand of chunk k - 1 (waited for below in
        // the previous pass).
        if (!mbar_wait(&s.full[st], (uint32_t)(k / kRevStages) & 1u)) {
          *fail = 1;
          break;
        }
        tc_fence_after();
        // K rows 64..127: the output rows of Mc with dO_c.  A has two
        // M-atoms; the second (lanes 64..127, never read) is taken LBO = 8 KB
        // on, inside this stage, so that no MMA reads a stage the refill warp
        // may be writing.
        mma_k64(tmem + 64 * bb, stg + 8192, true, kTile, stg + kMcBytes, true, kTile, idesc,
                false);
        if (!mbar_wait(&s.s_ready, (uint32_t)k & 1u)) {
          *fail = 1;
          break;
        }
        tc_fence_after();
        // K rows 0..63: the state rows of Mc with dS' (unused M-atom: the
        // output rows of the same stage).
        mma_k64(tmem + 64 * bb, stg, true, kTile, smem_addr(s.op), true, kTile, idesc, true);
        mma_commit(&s.mma_done[bb]);
        mma_commit(&s.empty[st]);
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    if (lane == 0) {
      for (int k = 0; k < kRevStages && k < n; ++k) {
        const int c = n - 1 - k;
        rev_issue_load(s, k, hmaps + (size_t)c * kMapBytes, &tm_do, c * kBC, (int)bh);
      }
      for (int k = 0; k + kRevStages < n; ++k) {
        const int st = k % kRevStages;
        if (*fail || !mbar_wait(&s.empty[st], (uint32_t)(k / kRevStages) & 1u)) {
          *fail = 1;
          break;
        }
        const int c = n - 1 - (k + kRevStages);
        rev_issue_load(s, st, hmaps + (size_t)c * kMapBytes, &tm_do, c * kBC, (int)bh);
      }
    }
    __syncwarp();
  } else if (state) {
    float dS[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
      dS[j] = b.dS_T ? b.dS_T[(bh * 64 + row) * 64 + 32 * h + j] : 0.f;
    // The cotangent of the state leaving chunk c: out (fp32) and into the operand.
    auto publish = [&](int c) {
      float4* dst = reinterpret_cast<float4*>(dS_ends + ((size_t)(bh * nchunks + c) * 64 + row) *
                                                            64 + 32 * h);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        dst[q4] = make_float4(dS[4 * q4], dS[4 * q4 + 1], dS[4 * q4 + 2], dS[4 * q4 + 3]);
      store_half_sw(s.op, row, h, dS, 1.f);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.s_ready);
    };
    if (n > 0) publish(n - 1);
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * h;
    for (int k = 0; k < n; ++k) {
      const int c = n - 1 - k, st = k % kRevStages, bb = k & 1;
      bool ok = !*fail;
      ok = ok && mbar_wait(&s.full[st], (uint32_t)(k / kRevStages) & 1u);
      ok = ok && mbar_wait(&s.mma_done[bb], (uint32_t)(k >> 1) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        *fail = 1;
        break;
      }
      tc_fence_after();
      float d[32];
      tmem_ld32(tl + 64 * bb, d);
      tc_fence_before();
      const float gC = s.gc[st][0];
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[st]);
#pragma unroll
      for (int j = 0; j < 32; ++j) dS[j] = gC * dS[j] + d[j];
      if (c > 0) publish(c - 1);
    }
    if (!*fail && b.dS0) {
      float* dst = b.dS0 + (bh * 64 + row) * 64 + 32 * h;
#pragma unroll
      for (int j = 0; j < 32; ++j) dst[j] = dS[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s.fail && tid == 0) atomicExch(err, 1);
  if (warp == 0) tmem_dealloc(tmem, 128);
}

cudaError_t launch_tc_bwd_scan_impl(const BwdArgs& b, const void* maps, float* dS_ends,
                                    int* err, cudaStream_t stream) {
  const ChunkArgs& a = b.f;
  const int nchunks = (int)((a.T + kBC - 1) / kBC);
  CUtensorMap tm_do;
  if (!encode_rows_bf16(&tm_do, b.dO, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kBC))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(RevSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_scan_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_bwd_scan_kernel<<<(unsigned)a.BH, kRevThreads, smem, stream>>>(
      b, nchunks, reinterpret_cast<const unsigned char*>(maps), dS_ends, err, tm_do);
  return cudaGetLastError();
}

// dk of the tokens that end a chunk (from the next chunk's row 0) and of the
// last token (from dx_last), and dx_prev; one warp per item, items c = 1 ..
// nchunks-1 (token 64c - 1), nchunks (token T - 1) and 0 (dx_prev).
__global__ void __launch_bounds__(kBThreads) tc_bwd_edge_kernel(BwdArgs b, int nchunks,
                                                                const float* edge) {
  const ChunkArgs& a = b.f;
  const int lane = threadIdx.x & 31;
  const int64_t items = a.BH * (nchunks + 1);
  for (int64_t it = (int64_t)blockIdx.x * (kBThreads / 32) + threadIdx.x / 32; it < items;
       it += (int64_t)gridDim.x * (kBThreads / 32)) {
    const int64_t bh = it / (nchunks + 1);
    const int c = (int)(it % (nchunks + 1));
    if (c == 0) {
      if (b.dx_prev)
        for (int j = lane; j < 64; j += 32)
          b.dx_prev[bh * 64 + j] = a.x_prev ? edge[(bh * nchunks) * 64 + j] : 0.f;
      continue;
    }
    const int64_t t = (c < nchunks) ? (int64_t)c * kBC - 1 : a.T - 1;
    float u[2], g[2];
    float ss = 0.f, ug = 0.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = lane + 32 * e;
      u[e] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.k)[(bh * a.T + t) * 64 + j]);
      g[e] = (c < nchunks) ? edge[(bh * nchunks + c) * 64 + j] : (b.dx_last ? b.dx_last[bh * 64 + j] : 0.f);
      ss += u[e] * u[e];
      ug += u[e] * g[e];
    }
    ss = warp_sum(ss);
    ug = warp_sum(ug);
    float out[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) out[e] = g[e];
    if (a.phi == FALCON_PHI_L2) {
      const float nrm = sqrtf(ss);
      if (nrm < 1e-12f) {
        out[0] *= 1e12f;
        out[1] *= 1e12f;
      } else {
        const float inv = 1.f / nrm, c2 = ug * inv * inv;
#pragma unroll
        for (int e = 0; e < 2; ++e) out[e] = (g[e] - u[e] * c2) * inv;
      }
    } else if (a.phi == FALCON_PHI_RMS) {
      const float sr = rsqrtf(ss / 64.f + kEpsRms), c3 = sr * sr * sr * ug / 64.f;
#pragma unroll
      for (int e = 0; e < 2; ++e) out[e] = sr * g[e] - c3 * u[e];
    }
#pragma unroll
    for (int e = 0; e < 2; ++e)
      reinterpret_cast<__nv_bfloat16*>(b.dk)[(bh * a.T + t) * 64 + lane + 32 * e] =
          __float2bfloat16_rn(out[e]);
  }
}

}  // namespace

bool tc_bwd_applies(int dtype, int m, int dv, int C) {
  return dtype == FALCON_BF16 && m == 64 && dv == 64 && C == kBC;
}

cudaError_t launch_tc_bwd_scan(const BwdArgs& b, const void* maps, float* dS_ends, int* err,
                               cudaStream_t stream) {
  return launch_tc_bwd_scan_impl(b, maps, dS_ends, err, stream);
}

cudaError_t launch_tc_bwd_grad(const BwdArgs& b, const float* S_starts, const float* dS_ends,
                               float* edge, int* err, cudaStream_t stream) {
  const ChunkArgs& a = b.f;
  const int nchunks = (int)((a.T + kBC - 1) / kBC);
  CUtensorMap tm_k, tm_q, tm_v, tm_do;
  if (!encode_rows_bf16(&tm_k, a.k, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kBC) ||
      !encode_rows_bf16(&tm_q, a.q, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kBC) ||
      !encode_rows_bf16(&tm_v, a.v, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kBC) ||
      !encode_rows_bf16(&tm_do, b.dO, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kBC))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_grad_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBwdSmem);
  if (e != cudaSuccess) return e;
  tc_bwd_grad_kernel<<<dim3(nchunks, (unsigned)a.BH), kBThreads, kBwdSmem, stream>>>(
      b, nchunks, S_starts, dS_ends, edge, err, tm_k, tm_q, tm_v, tm_do);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t items = a.BH * (nchunks + 1);
  const int64_t blocks = (items + kBThreads / 32 - 1) / (kBThreads / 32);
  tc_bwd_edge_kernel<<<(unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16), kBThreads, 0,
                       stream>>>(b, nchunks, edge);
  return cudaGetLastError();
}

}  // namespace falcon
