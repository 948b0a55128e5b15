// Tensor-core (tcgen05) chunked forward for bf16 inputs with m = d_v = C = 64.
//
// Two launches:
//
//  1. tc_chunk_map_kernel -- one CTA (128 threads) per (head, chunk), all
//     chunks in parallel.  It turns the chunk into an affine map of the state
//     entering it (the chunk-local log-space form of the positive-decay
//     renormalisation of page hyper.ai/fr/papers/2608.27763, Section 4.4
//     Eq. (4.15)-(4.16); WY/UT form with one triangular solve per chunk, as
//     the complexity table of page juhoplayground.github.io describes):
//
//        S'  = e^{g_C} S + Mc_top S + Nc_top,   Mc_top = -Xt^T W,    Nc_top = Xt^T U~
//        O   =             Mc_bot S + Nc_bot,   Mc_bot = Diag(e^g) Q - P W,  Nc_bot = P U~
//
//     with W = T Diag(eta e^{g_-}) X, U~ = T Diag(eta) V, T = (I + A)^{-1}.
//     Three tcgen05 MMAs (bf16 operands from shared memory, fp32 accumulators
//     in TMEM) do the contractions:
//        MMA1  [X; Q] [X; Q]^T      -> G = X X^T and P^T (before masking)
//        MMA2  [Xh^T; Vh^T] T^T     -> [W^T; U~^T]
//        MMA3  [Xt^T; P] [W | U~]   -> [Xt^T W | Xt^T U~ ; P W | P U~]
//     The triangular solve runs in fp32 on the CUDA cores.  Mc is written to
//     the workspace as a ready-to-use swizzled bf16 operand tile, Nc in fp32.
//     Falcon-1A takes the same path with T = I and W = 0.
//
//  2. tc_chunk_scan_kernel -- one CTA per head, sequential over chunks: one
//     M=128 tcgen05 MMA per chunk, [Mc_top; Mc_bot] S, with the map of the
//     next chunks prefetched by bulk copies.  The e^{g_C} S part of the state
//     update stays in fp32 registers (only the correction goes through bf16
//     operands), so an undecayed state does not drift over long sequences.
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace falcon {

namespace {

using namespace tc;

constexpr int kC = 64;
constexpr uint32_t kMcBytes = 128 * 128;     // 128 rows x 64 bf16 (swizzled image)
constexpr uint32_t kNcBytes = 128 * 64 * 4;  // 128 rows x 64 fp32
constexpr uint32_t kMapBytes = kMcBytes + kNcBytes + 128;  // + e^{g_C} (padded)

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void flag_error(int* err) {
  if (err) atomicExch(err, 1);
}

// Load one 64-element bf16 row from global memory (16-byte vector loads).
__device__ __forceinline__ void load_row_global(const __nv_bfloat16* src, float* v) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 pk = __ldg(p + c);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&pk);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      v[8 * c + 2 * e] = f.x;
      v[8 * c + 2 * e + 1] = f.y;
    }
  }
}

// phi in place; returns ||phi(u)||^2.
__device__ __forceinline__ float apply_phi(float* v, int phi) {
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 64; ++j) ss += v[j] * v[j];
  if (phi == FALCON_PHI_L2) {
    const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
    ss = 0.f;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      v[j] *= inv;
      ss += v[j] * v[j];
    }
  }
  return ss;
}

__device__ __forceinline__ void store_row_scaled(unsigned char* tile, int r, const float* v,
                                                 float scale) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = scale * v[8 * c + e];
    uint4 pk;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(w[0], w[1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(w[2], w[3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(w[4], w[5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(w[6], w[7]);
    pk.x = *reinterpret_cast<uint32_t*>(&h0);
    pk.y = *reinterpret_cast<uint32_t*>(&h1);
    pk.z = *reinterpret_cast<uint32_t*>(&h2);
    pk.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(tile + r * 128 + ((c ^ (r & 7)) << 4)) = pk;
  }
}

// Shared memory of the map kernel.  Buffers with disjoint lifetimes share
// space: R1 holds the MMA1 operand [X; Q], then A (fp32), then MMA3's B
// operand; R2 holds the solve's fp32 scratch, then T as MMA2's B operand.
struct MapSmem {
  union {
    unsigned char xq[128 * 128];  // K-major: rows 0..63 X, 64..127 phi(Q) (MMA1 A and B)
    float As[64 * 65];            // strictly lower A of I + A (fp32), padded rows
    unsigned char b3[128 * 128];  // K-major B of MMA3: rows = [W^T; U~^T]
  } __align__(1024) r1;
  unsigned char a2[2 * 8192] __align__(1024);  // MN-major A of MMA2: atom 0 = Xh rows, atom 1 = Vh rows
  unsigned char a3[2 * 8192] __align__(1024);  // MN-major A of MMA3: atom 0 = Xt rows, atom 1 row j = P[:, j]
  union {
    struct {
      float Ts[64 * 65];    // T = (I + A)^{-1} during the solve
      float Rs[16 * 49];    // block-row right-hand sides
      float Dinv[64 * 17];  // inverses of the 16 x 16 diagonal blocks
    } sv;
    unsigned char tt[64 * 128];  // K-major B of MMA2: row i = T[i][:]
  } __align__(1024) r2;
  float eta[64], g[64], gx[64];
  float carry;
  int fail;
  uint64_t bar;
  uint32_t tmem_base;
};

// T = (I + A)^{-1} for the strictly lower 64 x 64 A in s.As (fp32, CUDA
// cores).  16 x 16 diagonal blocks are inverted by forward substitution with
// warp shuffles; block rows 1..3 follow T_b = Dinv_b (-A_b,<b T_<b).
__device__ void solve_unit_lower(MapSmem& s) {
  const int tid = threadIdx.x;
  if (tid < 64) {
    const int lane = tid & 31, r = tid & 15, b = tid >> 4;
    float dinv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) dinv[j] = (j == r) ? 1.f : 0.f;
#pragma unroll
    for (int k = 0; k < 15; ++k) {
      const float aik = s.r1.As[tid * 65 + 16 * b + k];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float tkj = __shfl_sync(0xffffffffu, dinv[j], (lane & 16) | k);
        if (r > k) dinv[j] -= aik * tkj;
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) s.r2.sv.Dinv[tid * 17 + j] = dinv[j];
    // T rows of block 0 are Dinv rows; every row is zero to the right of its
    // diagonal block.
    for (int j = 0; j < 64; ++j) {
      const int rel = j - 16 * b;
      s.r2.sv.Ts[tid * 65 + j] = (rel >= 0 && rel < 16) ? dinv[rel] : 0.f;
    }
  }
  __syncthreads();
  for (int b = 1; b < 4; ++b) {
    const int w = 16 * b;  // columns to the left of block b
    for (int idx = tid; idx < 16 * w; idx += 128) {
      const int ii = idx / w, cc = idx % w;
      const float* arow = s.r1.As + (w + ii) * 65;
      float acc = 0.f;
      for (int k = cc; k < w; ++k) acc -= arow[k] * s.r2.sv.Ts[k * 65 + cc];  // T[k][cc] = 0 for k < cc
      s.r2.sv.Rs[ii * 49 + cc] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < 16 * w; idx += 128) {
      const int ii = idx / w, cc = idx % w;
      const float* drow = s.r2.sv.Dinv + (w + ii) * 17;
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < 16; ++r) acc += drow[r] * s.r2.sv.Rs[r * 49 + cc];
      s.r2.sv.Ts[(w + ii) * 65 + cc] = acc;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(128) tc_chunk_map_kernel(ChunkArgs a, int nchunks, int* err) {
  extern __shared__ unsigned char smem_raw[];
  MapSmem& s = *reinterpret_cast<MapSmem*>(align1024(smem_raw));
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t0 = (int64_t)c * kC;
  const int n = (int)min((int64_t)kC, a.T - t0);
  const bool f1 = a.rule == kFalcon1;
  const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kg = reinterpret_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vg = reinterpret_cast<const __nv_bfloat16*>(a.v);
  const int64_t rowbase = bh * a.T;

  if (warp == 0) tmem_alloc(&s.tmem_base, 128);
  if (tid == 0) {
    mbar_init(&s.bar, 1);
    fence_mbar_init();
    s.fail = 0;
  }

  // ---- features: thread t < 64 builds the write feature x_t = phi(k_{t0+t-1});
  //      thread 64 + i builds phi(q_{t0+i}).  Rows past the sequence are zero.
  float x[64];
  float E = 0.f;
  if (tid < 64) {
    const int64_t tk = t0 + tid - 1;
    if (tid <= n && tk >= 0) {
      load_row_global(kg + (rowbase + tk) * 64, x);
      E = apply_phi(x, a.phi);
    } else if (tk < 0 && a.x_prev) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = a.x_prev[bh * 64 + j];
#pragma unroll
      for (int j = 0; j < 64; ++j) E += x[j] * x[j];
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = 0.f;
    }
    // phi(k_{T-1}) is x_n when the last chunk is partial.
    if (a.x_last && c == nchunks - 1 && n < kC && tid == n)
      for (int j = 0; j < 64; ++j) a.x_last[bh * 64 + j] = x[j];
  } else {
    const int i = tid - 64;
    if (i < n) {
      load_row_global(qg + (rowbase + t0 + i) * 64, x);
      apply_phi(x, a.phi);
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = 0.f;
    }
    if (a.x_last && c == nchunks - 1 && n == kC && tid == 64) {
      float kl[64];
      load_row_global(kg + (rowbase + a.T - 1) * 64, kl);
      apply_phi(kl, a.phi);
      for (int j = 0; j < 64; ++j) a.x_last[bh * 64 + j] = kl[j];
    }
  }
  store_row_bf16(s.r1.xq, tid, x);

  // ---- step sizes, log-decays, chunk-local inclusive prefix g ----
  float eta = 0.f, lg = 0.f;
  if (tid < 64 && tid < n) {
    float gam;
    const bool sentinel = (t0 + tid == 0) && (a.x_prev == nullptr);
    eta = step_eta_gamma(sentinel, E, a.beta[rowbase + t0 + tid], a.lambda[rowbase + t0 + tid],
                         a.eps, a.eps_gamma, &gam, &lg);
  }
  float incl = lg;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (tid == 31) s.carry = incl;
  fence_async_smem();
  __syncthreads();
  if (warp == 1) incl += s.carry;
  if (tid < 64) {
    s.eta[tid] = eta;
    s.g[tid] = incl;
    s.gx[tid] = incl - lg;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);

  // ---- MMA1: D[0:128) = [X; Q] [X; Q]^T ----
  if (tid == 0) {
    mma_k64(tmem, smem_addr(s.r1.xq), false, 16, smem_addr(s.r1.xq), false, 16,
            idesc_bf16(128, 128, false, false), false);
    mma_commit(&s.bar);
  }
  const float gC = s.g[kC - 1];
  // Meanwhile: Xh = Diag(eta e^{g_-}) X, Xt = Diag(e^{g_C - g}) X, Vh = Diag(eta) V.
  if (tid < 64) {
    store_row_scaled(s.a2, tid, x, f1 ? s.eta[tid] * __expf(s.gx[tid]) : 0.f);
    store_row_scaled(s.a3, tid, x, __expf(gC - s.g[tid]));
  } else {
    const int i = tid - 64;
    float v[64];
    if (i < n)
      load_row_global(vg + (rowbase + t0 + i) * 64, v);
    else
      for (int j = 0; j < 64; ++j) v[j] = 0.f;
    store_row_scaled(s.a2 + 8192, i, v, s.eta[i]);
  }
  if (!mbar_wait(&s.bar, 0)) s.fail = 1;
  tc_fence_after();
  if (tid < 64) {
    const int j = tid;  // row j of G, column j of P
    const float gxj = s.gx[j], gj = s.g[j], ej = s.eta[j];
    float d[32];
    for (int h = 0; h < 2; ++h) {
      tmem_ld32(tlane + 32 * h, d);
#pragma unroll
      for (int l = 0; l < 32; ++l) {
        const int col = 32 * h + l;
        s.r1.As[j * 65 + col] = (f1 && col < j) ? ej * __expf(gxj - s.g[col]) * d[l] : 0.f;
      }
    }
    float p[64];
    for (int h = 0; h < 2; ++h) {
      tmem_ld32(tlane + 64 + 32 * h, d);
#pragma unroll
      for (int l = 0; l < 32; ++l) {
        const int i = 32 * h + l;
        p[i] = (i >= j) ? __expf(fminf(s.g[i] - gj, 0.f)) * d[l] : 0.f;
      }
    }
    store_row_bf16(s.a3 + 8192, j, p);  // MN-major: row j holds P[:, j]
  }
  __syncthreads();
  if (__syncthreads_or(s.fail)) goto teardown;

  // ---- T = (I + A)^{-1} (identity for Falcon-1A) ----
  if (f1) {
    solve_unit_lower(s);
    float trow[64];
    if (tid < 64) {
#pragma unroll
      for (int j = 0; j < 64; ++j) trow[j] = s.r2.sv.Ts[tid * 65 + j];
    }
    __syncthreads();  // the bf16 T tile overwrites the fp32 scratch
    if (tid < 64) store_row_bf16(s.r2.tt, tid, trow);
  } else if (tid < 64) {
    float trow[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) trow[j] = (j == tid) ? 1.f : 0.f;
    store_row_bf16(s.r2.tt, tid, trow);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- MMA2: D[0:64) = [Xh^T; Vh^T] T^T = [W^T; U~^T] ----
  if (tid == 0) {
    mma_k64(tmem, smem_addr(s.a2), true, 8192, smem_addr(s.r2.tt), false, 16,
            idesc_bf16(128, 64, true, false), false);
    mma_commit(&s.bar);
  }
  if (!mbar_wait(&s.bar, 1)) s.fail = 1;
  tc_fence_after();
  {
    float d[64];
    tmem_ld32(tlane, d);
    tmem_ld32(tlane + 32, d + 32);
    store_row_bf16(s.r1.b3, tid, d);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (__syncthreads_or(s.fail)) goto teardown;

  // ---- MMA3: D[0:128) = [Xt^T; P] [W | U~] ----
  if (tid == 0) {
    mma_k64(tmem, smem_addr(s.a3), true, 8192, smem_addr(s.r1.b3), false, 16,
            idesc_bf16(128, 128, true, false), false);
    mma_commit(&s.bar);
  }
  if (!mbar_wait(&s.bar, 0)) s.fail = 1;
  tc_fence_after();
  if (!__syncthreads_or(s.fail)) {
    unsigned char* map = reinterpret_cast<unsigned char*>(a.workspace) +
                         (size_t)(bh * nchunks + c) * kMapBytes;
    float d[64];
    tmem_ld32(tlane, d);
    tmem_ld32(tlane + 32, d + 32);
    // Mc row: rows < 64 -> -Xt^T W ; rows >= 64 -> e^{g_i} q_i - P W
    const float eg = (tid >= 64) ? __expf(s.g[tid - 64]) : 0.f;
#pragma unroll
    for (int j = 0; j < 64; ++j) d[j] = (tid < 64) ? -d[j] : eg * x[j] - d[j];
    {
      // swizzled image of the K-major operand tile, row tid
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint4 pk;
        __nv_bfloat162 h0 = __floats2bfloat162_rn(d[8 * cc + 0], d[8 * cc + 1]);
        __nv_bfloat162 h1 = __floats2bfloat162_rn(d[8 * cc + 2], d[8 * cc + 3]);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(d[8 * cc + 4], d[8 * cc + 5]);
        __nv_bfloat162 h3 = __floats2bfloat162_rn(d[8 * cc + 6], d[8 * cc + 7]);
        pk.x = *reinterpret_cast<uint32_t*>(&h0);
        pk.y = *reinterpret_cast<uint32_t*>(&h1);
        pk.z = *reinterpret_cast<uint32_t*>(&h2);
        pk.w = *reinterpret_cast<uint32_t*>(&h3);
        *reinterpret_cast<uint4*>(map + tid * 128 + ((cc ^ (tid & 7)) << 4)) = pk;
      }
    }
    tmem_ld32(tlane + 64, d);
    tmem_ld32(tlane + 96, d + 32);
    float4* nc = reinterpret_cast<float4*>(map + kMcBytes + tid * 256);
#pragma unroll
    for (int j = 0; j < 16; ++j) nc[j] = make_float4(d[4 * j], d[4 * j + 1], d[4 * j + 2], d[4 * j + 3]);
    if (tid == 0) *reinterpret_cast<float*>(map + kMcBytes + kNcBytes) = __expf(gC);
  }

teardown:
  if (s.fail && tid == 0) flag_error(err);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
constexpr int kStages = 2;

struct ScanSmem {
  unsigned char mc[kStages][kMcBytes];  // A tiles of the state MMA (K-major)
  unsigned char sop[8192];              // S as MN-major B operand (rows = m, 64 bf16 along d_v)
  float nc[kStages][128 * 64];
  float gc[kStages][4];
  uint64_t full[kStages];
  uint64_t mbar;
  uint32_t tmem_base;
  int fail;
};

__global__ void __launch_bounds__(128) tc_chunk_scan_kernel(ChunkArgs a, int nchunks, int* err) {
  extern __shared__ unsigned char smem_raw[];
  ScanSmem& s = *reinterpret_cast<ScanSmem*>(align1024(smem_raw));
  const int64_t bh = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5;
  const unsigned char* ws = reinterpret_cast<const unsigned char*>(a.workspace) +
                            (size_t)bh * nchunks * kMapBytes;
  if (warp == 0) tmem_alloc(&s.tmem_base, 64);
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&s.full[st], 1);
    mbar_init(&s.mbar, 1);
    fence_mbar_init();
    s.fail = 0;
    for (int st = 0; st < kStages && st < nchunks; ++st) {
      const unsigned char* m = ws + (size_t)st * kMapBytes;
      mbar_expect_tx(&s.full[st], kMcBytes + kNcBytes + 16);
      bulk_g2s(s.mc[st], m, kMcBytes, &s.full[st]);
      bulk_g2s(s.nc[st], m + kMcBytes, kNcBytes, &s.full[st]);
      bulk_g2s(s.gc[st], m + kMcBytes + kNcBytes, 16, &s.full[st]);
    }
  }
  // State: thread t < 64 keeps row t of S in fp32 registers.
  float S[64];
  if (tid < 64) {
#pragma unroll
    for (int j = 0; j < 64; ++j) S[j] = a.S0 ? a.S0[(bh * 64 + tid) * 64 + j] : 0.f;
    store_row_bf16(s.sop, tid, S);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
  __nv_bfloat16* og = reinterpret_cast<__nv_bfloat16*>(a.o);

  for (int c = 0; c < nchunks; ++c) {
    const int st = c % kStages;
    const uint32_t par = (uint32_t)(c / kStages) & 1u;
    if (!mbar_wait(&s.full[st], par)) s.fail = 1;
    if (tid == 0 && !s.fail) {
      tc_fence_after();
      mma_k64(tmem, smem_addr(s.mc[st]), false, 16, smem_addr(s.sop), true, 8192,
              idesc_bf16(128, 64, false, true), false);
      mma_commit(&s.mbar);
    }
    if (!s.fail && !mbar_wait(&s.mbar, (uint32_t)c & 1u)) s.fail = 1;
    if (__syncthreads_or(s.fail)) break;
    tc_fence_after();
    float d[64];
    tmem_ld32(tlane, d);
    tmem_ld32(tlane + 32, d + 32);
    const float* nrow = s.nc[st] + tid * 64;
    if (tid < 64) {
      const float gC = s.gc[st][0];
#pragma unroll
      for (int j = 0; j < 64; ++j) S[j] = gC * S[j] + d[j] + nrow[j];
      store_row_bf16(s.sop, tid, S);  // the MMA of this chunk has completed
    } else {
      // o row t0 + i straight from registers (16-byte stores; rows past T skipped)
      const int i = tid - 64;
      const int64_t t = (int64_t)c * kC + i;
      if (t < a.T) {
        uint4* orow = reinterpret_cast<uint4*>(og + (bh * a.T + t) * 64);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint4 pk;
          __nv_bfloat162 h0 = __floats2bfloat162_rn(d[8 * cc + 0] + nrow[8 * cc + 0], d[8 * cc + 1] + nrow[8 * cc + 1]);
          __nv_bfloat162 h1 = __floats2bfloat162_rn(d[8 * cc + 2] + nrow[8 * cc + 2], d[8 * cc + 3] + nrow[8 * cc + 3]);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(d[8 * cc + 4] + nrow[8 * cc + 4], d[8 * cc + 5] + nrow[8 * cc + 5]);
          __nv_bfloat162 h3 = __floats2bfloat162_rn(d[8 * cc + 6] + nrow[8 * cc + 6], d[8 * cc + 7] + nrow[8 * cc + 7]);
          pk.x = *reinterpret_cast<uint32_t*>(&h0);
          pk.y = *reinterpret_cast<uint32_t*>(&h1);
          pk.z = *reinterpret_cast<uint32_t*>(&h2);
          pk.w = *reinterpret_cast<uint32_t*>(&h3);
          orow[cc] = pk;
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      const int nx = c + kStages;
      if (nx < nchunks) {
        const unsigned char* m = ws + (size_t)nx * kMapBytes;
        mbar_expect_tx(&s.full[st], kMcBytes + kNcBytes + 16);
        bulk_g2s(s.mc[st], m, kMcBytes, &s.full[st]);
        bulk_g2s(s.nc[st], m + kMcBytes, kNcBytes, &s.full[st]);
        bulk_g2s(s.gc[st], m + kMcBytes + kNcBytes, 16, &s.full[st]);
      }
    }
  }
  if (!s.fail && tid < 64)
#pragma unroll
    for (int j = 0; j < 64; ++j) a.S_out[(bh * 64 + tid) * 64 + j] = S[j];
  if (s.fail && tid == 0) flag_error(err);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace

bool tc_path_applies(int dtype, int m, int dv, int C) {
  return dtype == FALCON_BF16 && m == 64 && dv == 64 && C == 64;
}

size_t tc_workspace_bytes(int64_t BH, int64_t T) {
  const int64_t nch = (T + kC - 1) / kC;
  return (size_t)(BH * nch) * kMapBytes;
}

cudaError_t launch_tc_chunked(const ChunkArgs& a, int* err, cudaStream_t stream) {
  const int nchunks = (int)((a.T + kC - 1) / kC);
  const size_t map_smem = sizeof(MapSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(tc_chunk_map_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)map_smem);
  if (e != cudaSuccess) return e;
  tc_chunk_map_kernel<<<dim3(nchunks, (unsigned)a.BH), 128, map_smem, stream>>>(a, nchunks, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t scan_smem = sizeof(ScanSmem) + 1024;
  e = cudaFuncSetAttribute(tc_chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)scan_smem);
  if (e != cudaSuccess) return e;
  tc_chunk_scan_kernel<<<(unsigned)a.BH, 128, scan_smem, stream>>>(a, nchunks, err);
  return cudaGetLastError();
}

}  // namespace falcon
